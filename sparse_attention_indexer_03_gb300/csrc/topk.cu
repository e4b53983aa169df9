// Per-row top-k of the indexer logits (`top_k_per_row_decode`, run right after
// the logits launch in aiter PR 4244, opening paragraph).
//
// One CTA of 512 threads per row runs the exact radix select of select.cuh
// and writes the row's indices in a deterministic order: the columns strictly
// above the threshold, ascending, then the ties at the threshold, lowest
// columns first.  Rows of a logical width up to 32768 are held in registers
// (KPT keys per thread, read from global memory once); longer rows are
// re-read from global memory (mostly L2) on each pass.
//
// The kernel is launched as a programmatic dependent of the previous kernel
// in the stream (the logits launch): it may start while that kernel drains,
// and waits for it to complete before reading any logits.
#include "common.cuh"
#include "ptx.cuh"
#include "select.cuh"

namespace sai {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

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

// ---- rows held in registers: element i*512 + tid of the row is key[i] ------
template <int KPT>
__global__ void __launch_bounds__(kThreads)
topk_reg_kernel(TopKArgs a) {
  extern __shared__ uint32_t hist_smem[];
  __shared__ SelectShared<kThreads> sh;
  __shared__ uint32_t seg_gt[KPT * kWarps], seg_eq[KPT * kWarps];
  ptx::wait_prerequisites();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r = blockIdx.x;
  const float* row = a.logits + r * a.stride;              // 64-bit row base
  // The first kSpec slots are read before the row's length is known (columns
  // below W always exist), so the two loads overlap; the rest after.
  constexpr int kSpec = KPT < 16 ? KPT : (KPT == 16 ? 16 : 8);
  uint32_t key[KPT];
#pragma unroll
  for (int i = 0; i < kSpec; ++i) {
    const int64_t idx = (int64_t)i * kThreads + tid;
    key[i] = idx < a.width ? float_key(row[idx]) : 0u;
  }
  const int64_t n = row_len(a, r);
  int32_t* out = a.indices + r * a.out_stride;             // 64-bit row base
  const int k = a.k;
  if (n <= k) {
    write_short_row(out, n, k);
    return;
  }
  const int live = (int)((n + kThreads - 1) / kThreads);   // slots that hold any key (CTA-uniform)
#pragma unroll
  for (int i = kSpec; i < KPT; ++i) {
    const int64_t idx = (int64_t)i * kThreads + tid;
    key[i] = (i < live && idx < n) ? float_key(row[idx]) : 0u;
  }
  auto for_each = [&](auto&& f) {
#pragma unroll
    for (int i = 0; i < KPT; ++i)
      if (i < live) f((int64_t)i * kThreads + tid < n, key[i]);
  };
  const SelectResult s = radix_select<kThreads>(sh, hist_smem, (uint32_t)k, tid, CtaBar{}, for_each);
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
  extern __shared__ uint32_t hist_smem[];
  __shared__ SelectShared<kThreads> sh;
  ptx::wait_prerequisites();
  const int64_t r = blockIdx.x;
  const int64_t n = row_len(a, r);
  int32_t* out = a.indices + r * a.out_stride;
  if (n <= a.k) {
    write_short_row(out, n, a.k);
    return;
  }
  topk_row_stream<kThreads>(a.logits + r * a.stride, n, a.k, out, sh, hist_smem, threadIdx.x, CtaBar{});
}

template <typename Kern>
cudaError_t launch_pdl(Kern kern, unsigned grid, const TopKArgs& a, cudaStream_t stream, int* smem_set) {
  cudaError_t e = ensure_dynamic_smem(kern, kSelectSmem, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSelectSmem;
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
  static int set4[64], set8[64], set16[64], set32[64], set64[64], set_stream[64];
  cudaError_t e;
  if (a.width <= 4 * kThreads) e = launch_pdl(topk_reg_kernel<4>, g, a, stream, set4);
  else if (a.width <= 8 * kThreads) e = launch_pdl(topk_reg_kernel<8>, g, a, stream, set8);
  else if (a.width <= 16 * kThreads) e = launch_pdl(topk_reg_kernel<16>, g, a, stream, set16);
  else if (a.width <= 32 * kThreads) e = launch_pdl(topk_reg_kernel<32>, g, a, stream, set32);
  else if (a.width <= 64 * kThreads) e = launch_pdl(topk_reg_kernel<64>, g, a, stream, set64);
  else e = launch_pdl(topk_stream_kernel, g, a, stream, set_stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sai
