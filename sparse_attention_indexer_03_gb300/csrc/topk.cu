// Per-row top-k of the indexer logits (`top_k_per_row_decode`, run right after
// the logits launch in aiter PR 4244, opening paragraph).
//
// One CTA per row runs the exact radix select of select.cuh
// and writes the row's indices in a deterministic order: the columns above
// the last bin the select examined, ascending, then the columns taken from
// that bin, ascending (ties at the k-th largest value: the lowest columns).
// Rows of a logical width up to 16384 are held in registers (each thread a
// run of KPT consecutive columns, read from global memory once).  Wider rows
// are copied into shared memory once their length is known (up to 40960
// columns, or 16384 on two CTAs of 512 threads per SM for logical widths
// beyond that), and longer ones re-read from global memory (mostly L2) on
// each pass.
//
// The kernel is launched as a programmatic dependent of the previous kernel
// in the stream (the logits launch): it may start while that kernel drains,
// and waits for it to complete before reading any logits.  It then lets its
// own dependents start at once: with one CTA per row, a decode batch leaves
// most SMs free, where the next launch can run its set-up.
//
// Few long rows (up to 131072 columns, too few rows to fill the GPU one CTA
// each) are split over a thread-block cluster of 2 to 8 CTAs, each holding
// 16384 columns in registers: each radix pass adds the CTAs' histograms
// through distributed shared memory, so every CTA takes the same digits, and
// the compaction offsets each CTA by the keys its predecessors select.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "select.cuh"

namespace sai {
namespace {

constexpr int kThreads = 1024;

__device__ __forceinline__ int64_t row_len(const TopKArgs& a, int64_t r) {
  const int b = (int)(r / a.next_n), j = (int)(r % a.next_n);
  return row_context(a.context_lens[b], a.next_n, j, a.width);
}

__device__ __forceinline__ void write_short_row(int32_t* out, int64_t n, int k) {
  for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
}

struct CtaBar {
  __device__ __forceinline__ void operator()() const { __syncthreads(); }
};

// Keys of columns [base, base + KPT) of a row (0 past the width).  A 16-byte
// aligned row is read as float4 vectors: a quarter of the load instructions
// of scalar reads, whose lanes, KPT words apart, each touch their own sector.
template <int KPT>
__device__ __forceinline__ void load_run(const float* row, int base, int64_t width, uint32_t (&key)[KPT]) {
  if ((reinterpret_cast<uintptr_t>(row) & 15u) == 0 && base + KPT <= width) {
#pragma unroll
    for (int v = 0; v < KPT / 4; ++v) {
      const float4 x = *reinterpret_cast<const float4*>(row + base + 4 * v);
      key[4 * v] = float_key(x.x);
      key[4 * v + 1] = float_key(x.y);
      key[4 * v + 2] = float_key(x.z);
      key[4 * v + 3] = float_key(x.w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < KPT; ++i) key[i] = base + i < width ? float_key(row[base + i]) : 0u;
  }
}

// ---- rows held in registers: lane l of warp w holds the KPT columns from
// w * 32 * KPT + l * KPT on, key[i] the i-th of them ---------------------------
template <int KPT>
__global__ void __launch_bounds__(kThreads)
topk_reg_kernel(TopKArgs a) {
  extern __shared__ uint32_t hist_smem[];
  __shared__ SelectShared<kThreads> sh;
  ptx::wait_prerequisites();
  ptx::launch_dependents();     // the next logits launch may take the SMs this grid leaves idle
  const int tid = threadIdx.x;
  const int64_t r = blockIdx.x;
  const float* row = a.logits + r * a.stride;              // 64-bit row base
  const int base = tid * KPT;
  // The keys are read before the row's length is known (columns below W
  // always exist), so the two loads overlap.
  uint32_t key[KPT];
  load_run<KPT>(row, base, a.width, key);
  const int64_t n64 = row_len(a, r);
  int32_t* out = a.indices + r * a.out_stride;             // 64-bit row base
  const int k = a.k;
  if (n64 <= k) {
    write_short_row(out, n64, k);
    return;
  }
  const int n = (int)n64;                                  // <= KPT * kThreads
  const bool warp_live = ((tid >> 5) * 32 * KPT) < n;     // warp-uniform
  auto for_each = [&](auto&& f) {
    if (warp_live) {
#pragma unroll
      for (int i = 0; i < KPT; ++i) f(base + i < n, key[i]);
    }
  };
  const SelectResult s = radix_select<kThreads>(sh, hist_smem, (uint32_t)k, tid, CtaBar{}, for_each);
  compact_lanes<kThreads>(sh, s, n, k, out, tid, CtaBar{}, base, KPT, RegRun<KPT>{key, KPT});
}

// ---- few long rows: CTA `rank` of a cluster of CL holds columns
// [rank * 16384, (rank + 1) * 16384) of the row, in registers as above --------
constexpr int kClusterKpt = 16;
constexpr int kClusterSlice = kClusterKpt * kThreads;     // 16384 columns per CTA

// Histogram counts of the whole row: each CTA publishes the counts of the
// bins its threads own in one of two exchange arrays (alternating passes, so
// a pass never overwrites an array another CTA may still be reading), and
// each thread sums its bins over the cluster.
template <int CL>
struct ClusterCounts {
  uint32_t* xch;                                           // 2 * kSelBins2 words
  template <int MP>
  __device__ __forceinline__ void operator()(int pass, uint32_t (&cnt)[MP], int per, int wbase, int lane) const {
    uint32_t* x = xch + (pass & 1) * kSelBins2;
#pragma unroll
    for (int i = 0; i < MP; ++i)
      if (i < per) x[wbase + 32 * i + lane] = cnt[i];
    ptx::cluster_sync();
#pragma unroll
    for (int i = 0; i < MP; ++i)
      if (i < per) {
        uint32_t v[CL];                                    // all CL loads in flight, then the sum
#pragma unroll
        for (int c = 0; c < CL; ++c) v[c] = ptx::ld_cluster_u32(x + wbase + 32 * i + lane, (uint32_t)c);
        uint32_t t = 0;
#pragma unroll
        for (int c = 0; c < CL; ++c) t += v[c];
        cnt[i] = t;
      }
  }
};

// Keys above and at the threshold selected by the CTAs of lower rank (which
// hold the earlier columns).  The second barrier keeps every CTA's shared
// memory alive until all the cluster's reads of it are done.
template <int CL>
struct ClusterPreceding {
  uint32_t* totals;                                        // 2 words
  uint32_t rank;
  template <int NT>
  __device__ __forceinline__ void operator()(const SelectShared<NT>& sh, uint32_t& pg, uint32_t& pe) const {
    if (threadIdx.x == 0) {
      uint32_t tg = 0, te = 0;
      for (int w = 0; w < NT / 32; ++w) { tg += sh.warp_gt[w]; te += sh.warp_eq[w]; }
      totals[0] = tg;
      totals[1] = te;
    }
    __syncwarp();                                          // the barrier is warp-aligned
    ptx::cluster_sync();
    uint32_t vg[CL], ve[CL];                               // all loads in flight, then the sums
#pragma unroll
    for (int c = 0; c < CL; ++c) {
      vg[c] = (uint32_t)c < rank ? ptx::ld_cluster_u32(totals, (uint32_t)c) : 0u;
      ve[c] = (uint32_t)c < rank ? ptx::ld_cluster_u32(totals + 1, (uint32_t)c) : 0u;
    }
#pragma unroll
    for (int c = 0; c < CL; ++c) { pg += vg[c]; pe += ve[c]; }
    ptx::cluster_sync();
  }
};

template <int CL>
__global__ void __launch_bounds__(kThreads)
topk_cluster_kernel(TopKArgs a) {
  constexpr int KPT = kClusterKpt, kSlice = kClusterSlice;
  extern __shared__ uint32_t hist_smem[];
  __shared__ SelectShared<kThreads> sh;
  __shared__ uint32_t xch[2 * kSelBins2];
  __shared__ uint32_t totals[2];
  ptx::wait_prerequisites();
  ptx::launch_dependents();
  const int tid = threadIdx.x;
  const uint32_t rank = ptx::cluster_rank();
  const int64_t r = blockIdx.x / CL;
  const float* row = a.logits + r * a.stride;              // 64-bit row base
  const int base = (int)rank * kSlice + tid * KPT;
  uint32_t key[KPT];
  load_run<KPT>(row, base, a.width, key);
  const int64_t n64 = row_len(a, r);
  int32_t* out = a.indices + r * a.out_stride;             // 64-bit row base
  const int k = a.k;
  if (n64 <= k) {                                          // the same for every CTA of the cluster
    if (rank == 0) write_short_row(out, n64, k);
    return;
  }
  const int n = (int)n64;                                  // <= CL * kSlice
  const bool warp_live = (int)rank * kSlice + (tid >> 5) * 32 * KPT < n;   // warp-uniform
  auto for_each = [&](auto&& f) {
    if (warp_live) {
#pragma unroll
      for (int i = 0; i < KPT; ++i) f(base + i < n, key[i]);
    }
  };
  // Every CTA of the cluster runs the same passes (the digits come from the
  // cluster's counts) and so the same cluster barriers.
  const SelectResult s =
      radix_select<kThreads>(sh, hist_smem, (uint32_t)k, tid, CtaBar{}, for_each, ClusterCounts<CL>{xch});
  compact_lanes<kThreads>(sh, s, n, k, out, tid, CtaBar{}, base, KPT, RegRun<KPT>{key, KPT},
                          ClusterPreceding<CL>{totals, rank});
}

// ---- wider rows: a row of up to KEYS columns has its keys copied into
// shared memory once its length is known (the radix passes then read them
// as 16-byte vectors; pass 1 is counted during the copy); a longer row is
// re-read from L2 on every pass.  For
// logical widths up to 40960, one CTA of 1024 threads per SM stages every
// row.  Wider rows (the wide outputs, whose rows hold far fewer context
// columns than their width) go to CTAs of 512 threads staging up to 16384
// keys (112 KB), two per SM: the select's phases are latency-bound, so two
// rows in flight overlap them.
// ---- longest rows first: when the grid is several waves, position p takes the
// row of rank p in an order by request length class (floor(log2) of the
// context, longest class first, request order within a class; a request's
// rows stay together), so the longest rows start in the first wave and the
// last waves hold short ones.  Every CTA derives its row from the context
// lengths: one coalesced read of all of them (the latency of its own row's
// length read, which it replaces), a 32-bin histogram, a warp scan, and one
// block-wide count of the chosen class.  Batches of at most NT requests.
template <int NT>
struct LongestFirst {
  uint32_t bins[32];
  uint32_t wcnt[NT / 32];
  int cls, off, b, ctx;
};

__device__ __forceinline__ int length_class(int64_t ctx, int64_t width) {
  const int64_t ce = ctx < 0 ? 0 : (ctx > width ? width : ctx);
  const uint32_t c = (uint32_t)(ce > 0x7fffffff ? 0x7fffffff : ce);
  return c <= 1 ? 31 : __clz(c);                         // 31 - floor(log2 c): the longest first
}

// Row of grid position p; *ctx its request's context length.
template <int NT>
__device__ __forceinline__ int64_t longest_first_row(const TopKArgs& a, int64_t p, LongestFirst<NT>& lf,
                                                     int64_t* ctx) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t q = p / a.next_n;                        // the request's rank
  const bool have = tid < a.batch;
  const int32_t c_me = have ? a.context_lens[tid] : 0;
  const int key = have ? length_class(c_me, a.width) : -1;
  if (tid < 32) lf.bins[tid] = 0u;
  __syncthreads();
  if (have) atomicAdd(&lf.bins[key], 1u);
  __syncthreads();
  if (warp == 0) {
    const uint32_t cnt = lf.bins[lane];
    uint32_t incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const uint32_t excl = incl - cnt;
    if (excl <= (uint64_t)q && (uint64_t)q < incl) {     // one lane: q < batch
      lf.cls = lane;
      lf.off = (int)(q - excl);
    }
  }
  __syncthreads();
  const bool mine = key == lf.cls;
  const uint32_t bal = __ballot_sync(0xffffffffu, mine);
  if (lane == 0) lf.wcnt[warp] = __popc(bal);
  __syncthreads();
  const uint32_t before = __reduce_add_sync(0xffffffffu, lane < warp ? lf.wcnt[lane] : 0u);
  if (mine && before + __popc(bal & ((1u << lane) - 1u)) == (uint32_t)lf.off) {
    lf.b = tid;
    lf.ctx = c_me;
  }
  __syncthreads();
  *ctx = lf.ctx;
  return (int64_t)lf.b * a.next_n + p % a.next_n;
}

// One row r of n columns by a CTA of NT threads: the histograms at the start
// of `topk_smem`, up to KEYS staged keys after them (longer rows, where
// STREAM, re-read from L2 per pass).  Ends with every thread done with the
// shared memory (a barrier), except for a row of at most k columns, which
// uses none.
template <int NT, int KEYS, bool STREAM = true>
__device__ __forceinline__ void smem_row(const TopKArgs& a, int64_t r, int64_t n, uint8_t* topk_smem,
                                         SelectShared<NT>& sh) {
  int32_t* out = a.indices + r * a.out_stride;             // 64-bit row base
  if (n <= a.k) {
    for (int i = threadIdx.x; i < a.k; i += NT) out[i] = i < n ? i : -1;
    return;
  }
  uint32_t* hist = reinterpret_cast<uint32_t*>(topk_smem);
  const float* row = a.logits + r * a.stride;
  if (!STREAM || n <= KEYS) {
    uint32_t* key_base = reinterpret_cast<uint32_t*>(topk_smem + kSelectSmem);
    topk_row_staged<NT>(row, (int)n, a.k, out, sh, hist, key_base, threadIdx.x, CtaBar{});
  } else {
    topk_row_stream<NT>(row, n, a.k, out, sh, hist, threadIdx.x, CtaBar{});
  }
}

template <int NT, int KEYS>
__global__ void __launch_bounds__(NT, NT == 512 ? 2 : 1)
topk_smem_kernel(TopKArgs a) {
  extern __shared__ __align__(16) uint8_t topk_smem[];
  __shared__ SelectShared<NT> sh;
  __shared__ LongestFirst<NT> lf;
  ptx::wait_prerequisites();
  ptx::launch_dependents();     // the next logits launch may take the SMs this grid leaves idle
  int64_t r = blockIdx.x, n;
  if (a.longest_first) {
    int64_t ctx;
    r = longest_first_row<NT>(a, blockIdx.x, lf, &ctx);
    n = row_context(ctx, a.next_n, (int)(r % a.next_n), a.width);
  } else {
    n = row_len(a, r);
  }
  smem_row<NT, KEYS>(a, r, n, topk_smem, sh);
}

// ---- many rows of up to KEYS staged keys, longest first, on one CTA per SM
// that keeps its shared memory across rows: the CTA ranks the batch's
// requests once in the order above (into a permutation kept after the key
// staging area: a request's rank is the start of its class plus the requests
// of its class in earlier warps and in earlier lanes of its warp, counted
// per warp by one match instruction), then takes the
// grid positions b, 2G - 1 - b, 2G + b, ... (alternating direction per wave
// of G positions, so each CTA takes one row of every length tier).  Saves the
// per-row ranking and CTA start of the one-row-per-CTA form, which most rows
// of a batch of short requests pay for a row of at most k columns.
template <int NT>
struct RowOrder {
  uint16_t perm[NT];              // request of each rank
  int32_t ctx[NT];                // each request's context length
};

// The permutation's place: after the histograms and a row's staged keys.
constexpr size_t row_order_offset(int64_t width) { return (kSelectSmem + 4 * ((size_t)width + 4) + 15) / 16 * 16; }

template <int KEYS>
__global__ void __launch_bounds__(kThreads, 1)
topk_smem_ordered_kernel(TopKArgs a) {
  constexpr int NT = kThreads, kW = NT / 32;
  extern __shared__ __align__(16) uint8_t topk_smem[];
  __shared__ SelectShared<NT> sh;
  ptx::wait_prerequisites();
  ptx::launch_dependents();     // the next logits launch may take the SMs this grid leaves idle
  RowOrder<NT>& ro = *reinterpret_cast<RowOrder<NT>*>(topk_smem + row_order_offset(a.width));
  {
    // Ranking scratch in the key staging area (no row staged yet).
    uint32_t(*wc)[32] = reinterpret_cast<uint32_t(*)[32]>(topk_smem + kSelectSmem);   // [warp][class]
    uint32_t* cpre = wc[kW];                                                             // [class]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const bool have = tid < a.batch;
    const int32_t c_me = have ? a.context_lens[tid] : 0;
    const int key = have ? length_class(c_me, a.width) : -1;
    if (have) ro.ctx[tid] = c_me;
    wc[warp][lane] = 0u;
    __syncwarp();
    const uint32_t same = __match_any_sync(0xffffffffu, key);
    const uint32_t lower = __popc(same & ((1u << lane) - 1u));   // equal keys in earlier lanes
    if (have && lower == 0) wc[warp][key] = __popc(same);
    __syncthreads();
    if (warp == 0) {                             // lane c: class c's prefix over warps, then over classes
      uint32_t run = 0;
      for (int w = 0; w < kW; ++w) {
        const uint32_t v = wc[w][lane];
        wc[w][lane] = run;
        run += v;
      }
      uint32_t incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      cpre[lane] = incl - run;
    }
    __syncthreads();
    if (have) ro.perm[cpre[key] + wc[warp][key] + lower] = (uint16_t)tid;
    __syncthreads();                             // the permutation is complete; the scratch is free
  }
  const int rows = a.batch * a.next_n, G = (int)gridDim.x;      // batch <= NT
  for (int t0 = 0, wave = 0; t0 < rows; t0 += G, ++wave) {
    const int p = t0 + ((wave & 1) ? G - 1 - (int)blockIdx.x : (int)blockIdx.x);
    if (p >= rows) continue;
    const int b = ro.perm[p / a.next_n], j = p % a.next_n;
    // (width <= KEYS: every row is staged)
    smem_row<NT, KEYS, false>(a, (int64_t)b * a.next_n + j, row_context(ro.ctx[b], a.next_n, j, a.width),
                              topk_smem, sh);
  }
}

constexpr int kSmemKeysWide = 40960;        // 1024 threads, one CTA per SM
constexpr int kSmemKeysPair = 16384;        // 512 threads, two CTAs per SM

template <int KEYS>
constexpr size_t smem_keys_bytes() { return kSelectSmem + 4 * ((size_t)KEYS + 4); }

template <typename Kern>
cudaError_t launch_pdl(Kern kern, unsigned grid, const TopKArgs& a, cudaStream_t stream, int* smem_set,
                       size_t smem, size_t smem_max, unsigned cluster = 1, unsigned threads = kThreads) {
  cudaError_t e = ensure_dynamic_smem(kern, smem_max, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = cluster > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

size_t topk_workspace_bytes(int, int64_t, int) { return 0; }

cudaError_t launch_topk(const TopKArgs& a, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.batch * a.next_n;
  if (rows == 0) return cudaSuccess;
  const unsigned g = (unsigned)rows;
  static int set4[64], set8[64], set16[64], set_smem[64], set_ord[64], set_pair[64], set_c2[64], set_c4[64], set_c8[64];
  // Rows wider than one CTA's registers go to a cluster (16384 columns per
  // CTA) while the grid stays within four CTAs per SM; more rows fill the
  // GPU one CTA each.  (Clusters of 16 CTAs of 8192 columns were slower on a
  // single 131072-column row: 37 us against 30 us.)
  const int sms = device_sm_count();
  const int64_t slices = (a.width + kClusterSlice - 1) / kClusterSlice;
  // More rows than one wave of the one-row-per-CTA kernels below: take them
  // longest first (for batches of at most one CTA's threads).
  auto lpt = [&](int ctas_per_sm, int nt) {
    TopKArgs b = a;
    b.longest_first = rows > (int64_t)ctas_per_sm * (sms > 0 ? sms : 152) && a.batch <= nt;
    return b;
  };
  const int cl = slices <= 2 ? 2 : (slices <= 4 ? 4 : 8);
  const bool clustered = a.width > kClusterSlice && slices <= 8 && rows * cl <= 4 * (int64_t)(sms > 0 ? sms : 152);
  cudaError_t e;
  if (clustered) {
    const unsigned gc = (unsigned)(rows * cl);
    if (cl == 2) e = launch_pdl(topk_cluster_kernel<2>, gc, a, stream, set_c2, kSelectSmem, kSelectSmem, 2);
    else if (cl == 4) e = launch_pdl(topk_cluster_kernel<4>, gc, a, stream, set_c4, kSelectSmem, kSelectSmem, 4);
    else e = launch_pdl(topk_cluster_kernel<8>, gc, a, stream, set_c8, kSelectSmem, kSelectSmem, 8);
  } else if (a.width <= 4 * kThreads) e = launch_pdl(topk_reg_kernel<4>, g, a, stream, set4, kSelectSmem, kSelectSmem);
  else if (a.width <= 8 * kThreads) e = launch_pdl(topk_reg_kernel<8>, g, a, stream, set8, kSelectSmem, kSelectSmem);
  else if (a.width <= 16 * kThreads) e = launch_pdl(topk_reg_kernel<16>, g, a, stream, set16, kSelectSmem, kSelectSmem);
  else if (a.width <= kSmemKeysWide && lpt(1, kThreads).longest_first)
    e = launch_pdl(topk_smem_ordered_kernel<kSmemKeysWide>, (unsigned)(sms > 0 ? sms : 152), a, stream, set_ord,
                   row_order_offset(a.width) + sizeof(RowOrder<kThreads>),
                   row_order_offset(kSmemKeysWide) + sizeof(RowOrder<kThreads>));
  else if (a.width <= kSmemKeysWide)
    e = launch_pdl(topk_smem_kernel<kThreads, kSmemKeysWide>, g, a, stream, set_smem,
                   kSelectSmem + 4 * (size_t)(a.width + 4), smem_keys_bytes<kSmemKeysWide>());
  else
    e = launch_pdl(topk_smem_kernel<512, kSmemKeysPair>, g, lpt(2, 512), stream, set_pair,
                   smem_keys_bytes<kSmemKeysPair>(), smem_keys_bytes<kSmemKeysPair>(), 1, 512);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sai
