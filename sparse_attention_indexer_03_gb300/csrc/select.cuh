// Exact top-k selection of one row of fp32 logits by a group of NT threads
// (a whole CTA, or a named-barrier group inside a larger CTA).  Used by the
// top-k kernels and by the fused logits + top-k kernel.
//
// Keys are order-preserving 32-bit images of the values (-0 and +0 equal).
// The k-th largest key is found by a radix select with digits of 8, 12 and 12
// bits, most significant first.  Pass 1 sees every key, and real logits share
// their top bits, so its histogram is kept per lane (256 bins x 32 lanes):
// the lanes of one atomic never hit the same word or bank.  Passes 2 and 3
// see only the keys of the chosen bin and use one plain 4096-bin histogram
// each.  The select stops as soon as every key of the chosen bin is taken.
// Output order is deterministic: the columns above the last bin the select
// examined, ascending, then the columns taken from that bin, ascending (the
// whole bin when the select stopped early; otherwise the bin is the ties at
// the k-th largest key, and the lowest of them are taken).
#pragma once

#include "common.cuh"

namespace sai {

constexpr int kSelBins1 = 256;
constexpr int kSelBins2 = 4096;
// Shared memory the radix select needs for its histograms (48 KB).
constexpr size_t kSelectSmem = (size_t)(kSelBins1 * 32 + kSelBins2) * sizeof(uint32_t);

// Shared-memory add of 1 under a predicate, as one predicated instruction:
// lanes whose key is outside the bin issue nothing and no branch is formed.
// No memory clobber: the compiler may issue later keys' loads before the
// adds; the group barrier that ends a count (a volatile asm with a memory
// clobber) keeps every add before every read of the bins.
__device__ __forceinline__ void count_if(uint32_t* word, bool pred) {
  const uint32_t a = (uint32_t)__cvta_generic_to_shared(word);
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\t@p red.shared.add.u32 [%0], 1;\n\t}"
      :: "r"(a), "r"((uint32_t)pred));
}

// Zero `words` words (a multiple of 4) at a 16-byte aligned shared address.
template <int NT>
__device__ __forceinline__ void zero_words(uint32_t* p, int words, int tid) {
  uint4* v = reinterpret_cast<uint4*>(p);
  for (int i = tid; i < words / 4; i += NT) v[i] = make_uint4(0u, 0u, 0u, 0u);
}

struct SelectResult {
  uint32_t prefix;     // digits chosen so far
  uint32_t mask;       // bits those digits cover
  uint32_t remaining;  // keys still to take from the chosen bin
};

template <int NT>
struct SelectShared {
  uint32_t wtot[NT / 32];         // per-warp totals of a pass's bins
  uint32_t warp_gt[NT / 32];      // compaction: per-warp counts
  uint32_t warp_eq[NT / 32];
  uint32_t digit, remaining, bin_count;
};

// A group that holds all of its row: its own histogram counts are the row's.
struct LocalCounts {
  template <int MP>
  __device__ __forceinline__ void operator()(int, uint32_t (&)[MP], int, int, int) const {}
};

// Radix select over the keys each thread visits through `for_each(f)`, which
// calls f(valid, key) for each of the thread's keys.  The counting adds are
// predicated instructions, so the loops carry no data-dependent branch.
// `tid` is the thread's
// index in the group (0 .. NT-1, whole warps), `bar()` a barrier of the group,
// `hist` kSelectSmem bytes of shared memory.  Three barriers per pass.
// `row_counts(pass, cnt, per, wbase, lane)` turns the counts of the bins a
// thread owns (bin wbase + 32 * i + lane in cnt[i], i < per) into the whole
// row's, for rows split over several groups; every group then takes the
// same digits.  With `first_counted` the caller has zeroed `hist` and
// counted pass 1 itself (count_first below), and a barrier has followed.
template <int NT, typename Bar, typename ForEach, typename RowCounts = LocalCounts>
__device__ __forceinline__ SelectResult radix_select(SelectShared<NT>& sh, uint32_t* hist, uint32_t k, int tid,
                                                     Bar bar, ForEach for_each, RowCounts row_counts = {},
                                                     bool first_counted = false) {
  constexpr int kW = NT / 32;
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t* h1 = hist;                              // pass 1: [bin][lane]; pass 3: plain, reused
  uint32_t* h2 = hist + kSelBins1 * 32;             // pass 2: plain
  if (!first_counted) {
    zero_words<NT>(hist, kSelBins1 * 32 + kSelBins2, tid);
    bar();
  }
  SelectResult s{0u, 0u, k};
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 24 : (pass == 1 ? 12 : 0);
    const int nb = pass == 0 ? kSelBins1 : kSelBins2;
    uint32_t* h = pass == 1 ? h2 : h1;
    if (pass == 1) zero_words<NT>(h1, kSelBins2, tid);   // pass 3 reuses h1, free since pass 1's search
    const uint32_t prefix = s.prefix, mask = s.mask;
    if (pass == 0) {
      if (!first_counted)
        for_each([&](bool valid, uint32_t key) { count_if(&h1[(key >> 24) * 32 + lane], valid); });
    } else {
      for_each([&](bool valid, uint32_t key) {
        count_if(&h[(key >> shift) & (uint32_t)(nb - 1)], valid && (key & mask) == prefix);
      });
    }
    if (pass != 0 || !first_counted) bar();
    // Thread (warp w, lane l) owns bins w * 32 * per + 32 * i + l, i < per:
    // a warp reads rows of 32 consecutive bins, one per bank.  Bins past nb
    // count zero.
    const int per = (nb + NT - 1) / NT;
    const int wbase = warp * 32 * per;
    auto count = [&](int bin) -> uint32_t {
      if (bin >= nb) return 0u;
      if (pass != 0) return h[bin];
      uint32_t c = 0;                               // sum of the 32 lane copies, staggered by bank
#pragma unroll 8
      for (int l = 0; l < 32; ++l) c += h1[bin * 32 + ((l + bin) & 31)];
      return c;
    };
    constexpr int kMaxPer = (kSelBins2 + NT - 1) / NT;
    uint32_t cnt[kMaxPer];
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) cnt[i] = i < per ? count(wbase + 32 * i + lane) : 0u;
    row_counts(pass, cnt, per, wbase, lane);
    uint32_t mine = 0;
#pragma unroll
    for (int i = 0; i < kMaxPer; ++i) mine += cnt[i];
    const uint32_t wsum = __reduce_add_sync(0xffffffffu, mine);
    if (lane == 0) sh.wtot[warp] = wsum;
    bar();
    // Keys in the warps above this one: lane l reads warp l's total, one
    // warp reduction sums them (no chain of dependent shared reads).
    uint32_t above = __reduce_add_sync(0xffffffffu, lane > warp && lane < kW ? sh.wtot[lane] : 0u);
    const uint32_t rem = s.remaining;
    if (above < rem && above + wsum >= rem) {       // warp-uniform: the bin is in this warp
#pragma unroll
      for (int i = kMaxPer - 1; i >= 0; --i) {
        if (i < per) {
          const uint32_t rt = __reduce_add_sync(0xffffffffu, cnt[i]);
          if (above + rt >= rem) {                  // warp-uniform: the bin is in this row
            uint32_t suf = cnt[i];                  // sum over lanes >= this one
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint32_t t = __shfl_down_sync(0xffffffffu, suf, o);
              if (lane + o < 32) suf += t;
            }
            const uint32_t ab = above + suf - cnt[i];
            if (ab < rem && ab + cnt[i] >= rem) {
              sh.digit = (uint32_t)(wbase + 32 * i + lane);
              sh.remaining = rem - ab;
              sh.bin_count = cnt[i];
            }
            break;
          }
          above += rt;
        }
      }
    }
    bar();
    s.prefix |= sh.digit << shift;
    s.mask |= (uint32_t)(nb - 1) << shift;
    s.remaining = sh.remaining;
    if (sh.bin_count == sh.remaining) break;        // every key of the chosen bin is selected
  }
  return s;
}

// Ordered compaction of the selection over keys key_at(i), i in [0, n): warp w
// owns columns [w * seg, (w + 1) * seg); two sweeps (count, then write), each
// reading kU chunks of 32 keys before using them so the reads overlap (16
// coalesced loads in flight per thread).
template <int NT, typename Bar, typename KeyAt>
__device__ __forceinline__ void compact_stream(SelectShared<NT>& sh, const SelectResult& s, int64_t n, int k,
                                               int32_t* out, int tid, Bar bar, KeyAt key_at) {
  constexpr int kW = NT / 32, kU = 16;
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t n_gt = (uint32_t)k - s.remaining;
  const int64_t seg = ((n + kW - 1) / kW + 31) / 32 * 32;
  const int64_t lo = warp * seg, hi = min(n, lo + seg);
  uint32_t c_gt = 0, c_eq = 0;
  for (int64_t base = lo; base < hi; base += 32 * kU) {
    uint32_t m[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) m[u] = key_at(min(base + u * 32 + lane, n - 1)) & s.mask;   // n > k >= 1
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const bool v = base + u * 32 + lane < hi;
      c_gt += (v && m[u] > s.prefix) ? 1u : 0u;
      c_eq += (v && m[u] == s.prefix) ? 1u : 0u;
    }
  }
  c_gt = __reduce_add_sync(0xffffffffu, c_gt);
  c_eq = __reduce_add_sync(0xffffffffu, c_eq);
  if (lane == 0) { sh.warp_gt[warp] = c_gt; sh.warp_eq[warp] = c_eq; }
  bar();
  uint32_t off_gt = __reduce_add_sync(0xffffffffu, lane < warp ? sh.warp_gt[lane] : 0u);   // the warps before
  uint32_t off_eq = __reduce_add_sync(0xffffffffu, lane < warp ? sh.warp_eq[lane] : 0u);
  const uint32_t lt = (1u << lane) - 1u;
  for (int64_t base = lo; base < hi; base += 32 * kU) {
    uint32_t m[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) m[u] = key_at(min(base + u * 32 + lane, n - 1)) & s.mask;
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t i = base + u * 32 + lane;
      const bool gt = i < hi && m[u] > s.prefix, eq = i < hi && m[u] == s.prefix;
      const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
      const uint32_t rank = off_eq + __popc(be & lt);
      const uint32_t pos = gt ? off_gt + __popc(bg & lt) : n_gt + rank;
      if (gt || (eq && rank < s.remaining)) out[pos] = (int32_t)i;
      off_gt += __popc(bg);
      off_eq += __popc(be);
    }
  }
  bar();                                            // warp_gt / warp_eq free for the next row
}

// A group that holds all of its row: nothing precedes it.
struct FirstGroup {
  template <int NT>
  __device__ __forceinline__ void operator()(const SelectShared<NT>&, uint32_t&, uint32_t&) const {}
};

// Ordered compaction by lanes.  Lane l of warp w owns the run of columns
// [base, base + len) with base = w * 32 * len + l * len (plus the group's
// first column), so column order is
// (warp, lane, slot): each lane counts its own selected keys, one packed
// warp scan gives every lane its offset, one barrier gives every warp its
// offset, and each lane then writes its keys in order with no warp-wide
// operation per key.  `key_at.for_each(f)` calls f(i, key) for the keys of
// columns base + i; only i < len and columns below n count.  For a row split
// over groups, `preceding(sh, pg, pe)` adds to a thread's offsets the keys
// above and at the threshold that the groups holding earlier columns select
// (sh.warp_gt / warp_eq hold this group's per-warp counts when it is called).
template <int NT, typename Bar, typename KeyAt, typename Preceding = FirstGroup>
__device__ __forceinline__ void compact_lanes(SelectShared<NT>& sh, const SelectResult& s, int n, int k,
                                              int32_t* out, int tid, Bar bar, int base, int len, KeyAt key_at,
                                              Preceding preceding = {}) {
  const int lane = tid & 31, warp = tid >> 5;
  const uint32_t n_gt = (uint32_t)k - s.remaining;
  uint32_t cg = 0, ce = 0;
  key_at.for_each([&](int i, uint32_t key) {
    const uint32_t m = key & s.mask;
    const bool v = i < len && base + i < n;
    cg += (v && m > s.prefix) ? 1u : 0u;
    ce += (v && m == s.prefix) ? 1u : 0u;
  });
  // Counts below 2^16 per warp (a warp owns at most 32 * len <= 65535 columns
  // for every caller), so both scans share one word.
  const uint32_t x = (cg << 16) | ce;
  uint32_t incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) { sh.warp_gt[warp] = incl >> 16; sh.warp_eq[warp] = incl & 0xffffu; }
  bar();
  const uint32_t excl = incl - x;
  // Plus the counts of the warps before this one (lane l reads warp l's).
  uint32_t pg = (excl >> 16) + __reduce_add_sync(0xffffffffu, lane < warp ? sh.warp_gt[lane] : 0u);
  uint32_t pe = (excl & 0xffffu) + __reduce_add_sync(0xffffffffu, lane < warp ? sh.warp_eq[lane] : 0u);
  preceding(sh, pg, pe);
  key_at.for_each([&](int i, uint32_t key) {
    const uint32_t m = key & s.mask;
    const int c = base + i;
    const bool v = i < len && c < n;
    const bool gt = v && m > s.prefix, eq = v && m == s.prefix;
    if (gt) out[pg] = c;
    if (eq && pe < s.remaining) out[n_gt + pe] = c;
    pg += gt ? 1u : 0u;
    pe += eq ? 1u : 0u;
  });
  bar();                                            // warp_gt / warp_eq free for the next row
}

// Keys of a lane's run held in registers: key[i], i < len <= KPT (len
// uniform across the group, so the slot test is a uniform branch).
template <int KPT>
struct RegRun {
  const uint32_t (&key)[KPT];
  int len;
  template <typename F>
  __device__ __forceinline__ void for_each(F&& f) const {
#pragma unroll
    for (int i = 0; i < KPT; ++i)
      if (i < len) f(i, key[i]);
  }
};

// Top-k of one row read from global memory (through L2: written by other
// CTAs of the same launch, or by an earlier kernel).  Row length n > k.
// The radix passes read the row as 16-byte vectors, consecutive threads on
// consecutive vectors, eight in flight per thread (a few scalar columns
// before the first 16-byte boundary and after the last).
template <int NT, typename Bar>
__device__ __forceinline__ void topk_row_stream(const float* row, int64_t n, int k, int32_t* out,
                                                SelectShared<NT>& sh, uint32_t* hist, int tid, Bar bar) {
  constexpr int kV = 8;
  const int64_t head = min(n, (int64_t)(((16u - (reinterpret_cast<uintptr_t>(row) & 15u)) & 15u) >> 2));
  const float4* vec = reinterpret_cast<const float4*>(row + head);
  const int64_t nv = (n - head) >> 2, tail0 = head + 4 * nv;
  auto for_each = [&](auto&& f) {
    if (tid < head) f(true, float_key(__ldcg(row + tid)));
    for (int64_t b = 0; b < nv; b += (int64_t)NT * kV) {
      float4 x[kV];
#pragma unroll
      for (int u = 0; u < kV; ++u) x[u] = __ldcg(vec + min(b + u * NT + tid, nv - 1));
#pragma unroll
      for (int u = 0; u < kV; ++u) {
        const bool v = b + u * NT + tid < nv;
        f(v, float_key(x[u].x));
        f(v, float_key(x[u].y));
        f(v, float_key(x[u].z));
        f(v, float_key(x[u].w));
      }
    }
    for (int64_t i = tail0 + tid; i < n; i += NT) f(true, float_key(__ldcg(row + i)));
  };
  const SelectResult s = radix_select<NT>(sh, hist, (uint32_t)k, tid, bar, for_each);
  compact_stream<NT>(sh, s, n, k, out, tid, bar, [&](int64_t i) { return float_key(__ldcg(row + i)); });
}

// A row's keys staged in shared memory: key of column c at keys[c]; keys +
// head is 16-byte aligned, so columns [head, head + 4 nv) are nv 16-byte
// vectors and [head + 4 nv, n) a scalar tail of at most 3 (head <= 3 too).
struct StagedRow {
  const uint32_t* keys;
  int n, head, nv;
  __device__ __forceinline__ const uint4* vec() const { return reinterpret_cast<const uint4*>(keys + head); }
  __device__ __forceinline__ int tail0() const { return head + 4 * nv; }
};

// Copies row[0, n) into shared memory as keys (16-byte loads from L2, eight
// in flight per thread, consecutive threads on consecutive vectors) and
// counts pass 1 of the radix select on the way: `hist` must be zero and a
// barrier must separate this from the select.  `base` needs room for n + 3
// words; the keys start 0..3 words past it so that 16-byte row segments
// land on 16-byte shared addresses.
template <int NT>
__device__ __forceinline__ StagedRow stage_and_count(const float* row, int n, uint32_t* base, uint32_t* hist,
                                                     int tid) {
  const int lane = tid & 31;
  const int head = min(n, (int)(((16u - (reinterpret_cast<uintptr_t>(row) & 15u)) & 15u) >> 2));
  uint32_t* keys = base + ((4 - head) & 3);
  auto put = [&](int c, uint32_t key) {
    keys[c] = key;
    count_if(&hist[(key >> 24) * 32 + lane], true);
  };
  if (tid < head) put(tid, float_key(__ldcg(row + tid)));
  const float4* v = reinterpret_cast<const float4*>(row + head);
  uint4* kv = reinterpret_cast<uint4*>(keys + head);
  const int nv = (n - head) >> 2;
  constexpr int kU = 8;
  for (int b = 0; b < nv; b += NT * kU) {
    float4 x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = b + u * NT + tid;
      if (i < nv) x[u] = __ldcg(v + i);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int i = b + u * NT + tid;
      if (i < nv) {
        const uint4 k4 = make_uint4(float_key(x[u].x), float_key(x[u].y), float_key(x[u].z), float_key(x[u].w));
        kv[i] = k4;
        count_if(&hist[(k4.x >> 24) * 32 + lane], true);
        count_if(&hist[(k4.y >> 24) * 32 + lane], true);
        count_if(&hist[(k4.z >> 24) * 32 + lane], true);
        count_if(&hist[(k4.w >> 24) * 32 + lane], true);
      }
    }
  }
  for (int i = head + nv * 4 + tid; i < n; i += NT) put(i, float_key(__ldcg(row + i)));
  return StagedRow{keys, n, head, nv};
}

// Every key of a staged row once, in no particular order (the radix passes'
// counts): thread t reads vectors t, t + NT, ... (consecutive threads on
// consecutive 16-byte vectors: four keys per load, no bank conflict), four
// loads ahead of their adds, then the scalar head and tail.
template <int NT, typename F>
__device__ __forceinline__ void staged_for_each(const StagedRow& r, int tid, F&& f) {
  const uint4* kv = r.vec();
  constexpr int kU = 4;
  for (int b = tid; b < r.nv; b += NT * kU) {
    uint4 x[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) x[u] = kv[min(b + u * NT, r.nv - 1)];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const bool v = b + u * NT < r.nv;
      f(v, x[u].x);
      f(v, x[u].y);
      f(v, x[u].z);
      f(v, x[u].w);
    }
  }
  if (tid < r.head) f(true, r.keys[tid]);
  if (tid < r.n - r.tail0()) f(true, r.keys[r.tail0() + tid]);
}

// Keys of a lane's run in shared memory: keys[base + i], i < len, read at
// min(base + i, n - 1) so the reads stay inside the n staged keys (the
// ordered compaction of a staged row).
struct SmemRun {
  const uint32_t* keys;
  int base, len, n;
  template <typename F>
  __device__ __forceinline__ void for_each(F&& f) const {
#pragma unroll 4
    for (int i = 0; i < len; ++i) f(i, keys[min(base + i, n - 1)]);
  }
};

// Top-k of row[0, n) (n > k), staged into shared memory at `key_base` (room
// for n + 3 words) with pass 1 counted on the way.
template <int NT, typename Bar>
__device__ __forceinline__ void topk_row_staged(const float* row, int n, int k, int32_t* out, SelectShared<NT>& sh,
                                                uint32_t* hist, uint32_t* key_base, int tid, Bar bar) {
  zero_words<NT>(hist, kSelBins1 * 32 + kSelBins2, tid);
  bar();
  const StagedRow r = stage_and_count<NT>(row, n, key_base, hist, tid);
  bar();
  auto for_each = [&](auto&& f) { staged_for_each<NT>(r, tid, f); };
  const SelectResult s = radix_select<NT>(sh, hist, (uint32_t)k, tid, bar, for_each, LocalCounts{}, true);
  // The compaction by lane runs: lane l of warp w owns about n / NT
  // consecutive columns from (w * 32 + l) * len (len odd: the 32 lanes'
  // reads fall in 32 banks).
  const int len = ((n + NT - 1) / NT) | 1;
  const int base = (tid >> 5) * 32 * len + (tid & 31) * len;
  compact_lanes<NT>(sh, s, n, k, out, tid, bar, base, len, SmemRun{r.keys, base, len, n});
}

}  // namespace sai
