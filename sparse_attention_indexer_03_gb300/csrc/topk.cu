// Per-row top-k of the indexer logits (`top_k_per_row_decode`, run right after
// the logits launch in aiter PR 4244, opening paragraph).
//
// One CTA of 512 threads per row.  The k-th largest value is found exactly by
// a radix select over order-preserving 32-bit keys: digits of 11, 11 and 10
// bits, most significant first, each counted in a shared-memory histogram.
// The select stops early once every key of the chosen bin is taken.  The indices
// are then written in a deterministic order: the columns strictly above the
// threshold, ascending, then the ties at the threshold, lowest columns first.
//
// Rows of a logical width up to 32768 are held in registers (KPT keys per
// thread, read from global memory once); longer rows are re-read from global
// memory (mostly L2) on each pass.
//
// The kernel is launched as a programmatic dependent of the previous kernel
// in the stream (the logits launch): it may start while that kernel drains,
// and waits for it to complete before reading any logits.
#include "common.cuh"
#include "ptx.cuh"

namespace sai {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;

struct Select {          // result of the radix select
  uint32_t prefix;       // digits chosen so far
  uint32_t mask;         // bits those digits cover
  uint32_t remaining;    // keys still to take from the chosen bin
};

// Inclusive prefix sum of one value per thread over the CTA, plus the total.
__device__ __forceinline__ uint32_t block_inclusive_scan(uint32_t v, uint32_t* scratch, uint32_t& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  if (warp == 0) {
    uint32_t w = lane < kWarps ? scratch[lane] : 0u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += n;
    }
    if (lane < kWarps) scratch[lane] = w;
  }
  __syncthreads();
  if (warp > 0) v += scratch[warp - 1];
  total = scratch[kWarps - 1];
  __syncthreads();
  return v;
}

struct Shared {
  uint32_t hist[kBins];
  uint32_t scan[kWarps];
  uint32_t digit, remaining, bin_count;
};

// Add one to bin `bin` for every lane with `take`.
__device__ __forceinline__ void hist_add(uint32_t* hist, bool take, uint32_t bin) {
  if (take) atomicAdd(&hist[bin], 1u);
}

// Choose the bin of this pass that holds the `remaining`-th largest key.
__device__ __forceinline__ void choose_digit(Shared& sh, int nb, uint32_t remaining) {
  const int tid = threadIdx.x;
  const int per = nb / kThreads;
  uint32_t mine = 0;
  for (int i = 0; i < per; ++i) mine += sh.hist[tid * per + i];
  uint32_t total;
  const uint32_t incl = block_inclusive_scan(mine, sh.scan, total);
  uint32_t above = total - incl;                  // keys in bins above this thread's
  for (int i = per - 1; i >= 0; --i) {
    const uint32_t c = sh.hist[tid * per + i];
    if (above < remaining && above + c >= remaining) {
      sh.digit = (uint32_t)(tid * per + i);
      sh.remaining = remaining - above;
      sh.bin_count = c;
    }
    above += c;
  }
  __syncthreads();
}

// Radix select over the keys each thread visits through `for_each`.
template <typename ForEach>
__device__ __forceinline__ Select radix_select(Shared& sh, uint32_t k, ForEach for_each) {
  Select s{0u, 0u, k};
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass < 2 ? 2048 : 1024;
    for (int i = threadIdx.x; i < nb; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s.prefix, mask = s.mask;
    for_each([&](bool valid, uint32_t key) {
      hist_add(sh.hist, valid && (key & mask) == prefix, (key >> shift) & (uint32_t)(nb - 1));
    });
    __syncthreads();
    choose_digit(sh, nb, s.remaining);
    s.prefix |= sh.digit << shift;
    s.mask |= (uint32_t)(nb - 1) << shift;
    s.remaining = sh.remaining;
    const bool all_taken = sh.bin_count == sh.remaining;
    __syncthreads();
    if (all_taken) break;                          // every key of the chosen bin is selected
  }
  return s;
}

__device__ __forceinline__ int64_t row_len(const TopKArgs& a, int64_t r) {
  const int b = (int)(r / a.next_n), j = (int)(r % a.next_n);
  return row_context(a.context_lens[b], a.next_n, j, a.width);
}

__device__ __forceinline__ void write_short_row(int32_t* out, int64_t n, int k) {
  for (int i = threadIdx.x; i < k; i += kThreads) out[i] = i < n ? i : -1;
}

// ---- rows held in registers: element i*512 + tid of the row is key[i] ------
template <int KPT>
__global__ void __launch_bounds__(kThreads)
topk_reg_kernel(TopKArgs a) {
  __shared__ Shared sh;
  __shared__ uint32_t seg_gt[KPT * kWarps], seg_eq[KPT * kWarps];
  ptx::wait_prerequisites();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r = blockIdx.x;
  const int64_t n = row_len(a, r);
  int32_t* out = a.indices + r * a.out_stride;             // 64-bit row base
  const int k = a.k;
  if (n <= k) {
    write_short_row(out, n, k);
    return;
  }
  const float* row = a.logits + r * a.stride;              // 64-bit row base
  const int live = (int)((n + kThreads - 1) / kThreads);   // slots that hold any key (CTA-uniform)
  uint32_t key[KPT];
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const int64_t idx = (int64_t)i * kThreads + tid;
    key[i] = (i < live && idx < n) ? float_key(row[idx]) : 0u;
  }
  auto for_each = [&](auto&& f) {
#pragma unroll
    for (int i = 0; i < KPT; ++i)
      if (i < live) f((int64_t)i * kThreads + tid < n, key[i]);
  };
  const Select s = radix_select(sh, (uint32_t)k, for_each);
  const uint32_t n_gt = (uint32_t)k - s.remaining;

  // Ordered compaction: element order (slot i, warp, lane) is column order.
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    if (i < live) {
      const bool v = (int64_t)i * kThreads + tid < n;
      const uint32_t m = key[i] & s.mask;
      const uint32_t bg = __ballot_sync(0xffffffffu, v && m > s.prefix);
      const uint32_t be = __ballot_sync(0xffffffffu, v && m == s.prefix);
      if (lane == 0) {
        seg_gt[i * kWarps + warp] = __popc(bg);
        seg_eq[i * kWarps + warp] = __popc(be);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {                                  // exclusive scan over (slot, warp) segments
    const int nseg = live * kWarps;
    const int per = (nseg + 31) / 32;
    uint32_t sg = 0, se = 0;
    for (int x = 0; x < per; ++x) {
      const int id = lane * per + x;
      if (id < nseg) { sg += seg_gt[id]; se += seg_eq[id]; }
    }
    uint32_t ig = sg, ie = se;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t g2 = __shfl_up_sync(0xffffffffu, ig, o), e2 = __shfl_up_sync(0xffffffffu, ie, o);
      if (lane >= o) { ig += g2; ie += e2; }
    }
    uint32_t og = ig - sg, oe = ie - se;
    for (int x = 0; x < per; ++x) {
      const int id = lane * per + x;
      if (id < nseg) {
        const uint32_t cg = seg_gt[id], cq = seg_eq[id];
        seg_gt[id] = og; seg_eq[id] = oe;
        og += cg; oe += cq;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    if (i < live) {
      const int64_t idx = (int64_t)i * kThreads + tid;
      const bool v = idx < n;
      const uint32_t m = key[i] & s.mask;
      const bool gt = v && m > s.prefix, eq = v && m == s.prefix;
      const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
      if (gt) out[seg_gt[i * kWarps + warp] + __popc(bg & lt)] = (int32_t)idx;
      if (eq) {
        const uint32_t rank = seg_eq[i * kWarps + warp] + __popc(be & lt);
        if (rank < s.remaining) out[n_gt + rank] = (int32_t)idx;
      }
    }
  }
}

// ---- long rows: keys re-read from global memory on every pass ----------------
__global__ void __launch_bounds__(kThreads)
topk_stream_kernel(TopKArgs a) {
  __shared__ Shared sh;
  __shared__ uint32_t warp_gt[kWarps], warp_eq[kWarps];
  ptx::wait_prerequisites();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r = blockIdx.x;
  const int64_t n = row_len(a, r);
  int32_t* out = a.indices + r * a.out_stride;
  const int k = a.k;
  if (n <= k) {
    write_short_row(out, n, k);
    return;
  }
  const float* row = a.logits + r * a.stride;
  auto for_each = [&](auto&& f) {
    for (int64_t base = 0; base < n; base += kThreads) {
      const int64_t idx = base + tid;
      const bool v = idx < n;
      f(v, v ? float_key(row[idx]) : 0u);
    }
  };
  const Select s = radix_select(sh, (uint32_t)k, for_each);
  const uint32_t n_gt = (uint32_t)k - s.remaining;

  // Ordered compaction: warp w owns columns [w * seg, (w + 1) * seg).
  const int64_t seg = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int64_t lo = warp * seg, hi = min(n, lo + seg);
  uint32_t c_gt = 0, c_eq = 0;
  for (int64_t base = lo; base < hi; base += 32) {
    const int64_t i = base + lane;
    const uint32_t m = (i < hi ? float_key(row[i]) : 0u) & s.mask;
    c_gt += __popc(__ballot_sync(0xffffffffu, i < hi && m > s.prefix));
    c_eq += __popc(__ballot_sync(0xffffffffu, i < hi && m == s.prefix));
  }
  if (lane == 0) { warp_gt[warp] = c_gt; warp_eq[warp] = c_eq; }
  __syncthreads();
  uint32_t off_gt = 0, off_eq = 0;
  for (int w = 0; w < warp; ++w) { off_gt += warp_gt[w]; off_eq += warp_eq[w]; }
  const uint32_t lt = (1u << lane) - 1u;
  for (int64_t base = lo; base < hi; base += 32) {
    const int64_t i = base + lane;
    const uint32_t m = (i < hi ? float_key(row[i]) : 0u) & s.mask;
    const bool gt = i < hi && m > s.prefix, eq = i < hi && m == s.prefix;
    const uint32_t bg = __ballot_sync(0xffffffffu, gt), be = __ballot_sync(0xffffffffu, eq);
    if (gt) out[off_gt + __popc(bg & lt)] = (int32_t)i;
    if (eq) {
      const uint32_t rank = off_eq + __popc(be & lt);
      if (rank < s.remaining) out[n_gt + rank] = (int32_t)i;
    }
    off_gt += __popc(bg);
    off_eq += __popc(be);
  }
}

template <typename Kern>
cudaError_t launch_pdl(Kern kern, unsigned grid, const TopKArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

size_t topk_workspace_bytes(int, int64_t, int) { return 0; }

cudaError_t launch_topk(const TopKArgs& a, cudaStream_t stream) {
  const int64_t rows = (int64_t)a.batch * a.next_n;
  if (rows == 0) return cudaSuccess;
  const unsigned g = (unsigned)rows;
  cudaError_t e;
  if (a.width <= 4 * kThreads) e = launch_pdl(topk_reg_kernel<4>, g, a, stream);
  else if (a.width <= 8 * kThreads) e = launch_pdl(topk_reg_kernel<8>, g, a, stream);
  else if (a.width <= 16 * kThreads) e = launch_pdl(topk_reg_kernel<16>, g, a, stream);
  else if (a.width <= 32 * kThreads) e = launch_pdl(topk_reg_kernel<32>, g, a, stream);
  else if (a.width <= 64 * kThreads) e = launch_pdl(topk_reg_kernel<64>, g, a, stream);
  else e = launch_pdl(topk_stream_kernel, g, a, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sai
