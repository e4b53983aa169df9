// Per-row top-k of the indexer logits (`top_k_per_row_decode`, run right after
// the logits launch in aiter PR 4244, opening paragraph).
//
// One CTA of 512 threads per row runs the exact radix select of select.cuh
// and writes the row's indices in a deterministic order: the columns strictly
// above the threshold, ascending, then the ties at the threshold, lowest
// columns first.  Rows of a logical width up to 32768 are held in registers
// (KPT keys per thread, each warp a contiguous run of columns, read from
// global memory once); longer rows are re-read from global memory (mostly L2)
// on each pass.
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

// ---- rows held in registers: warp w holds columns [w * 32 * KPT, (w + 1) * 32 * KPT),
// lane l of it column w * 32 * KPT + 32 * i + l in key[i] ------------------------
template <int KPT>
__global__ void __launch_bounds__(kThreads)
topk_reg_kernel(TopKArgs a) {
  extern __shared__ uint32_t hist_smem[];
  __shared__ SelectShared<kThreads> sh;
  ptx::wait_prerequisites();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r = blockIdx.x;
  const float* row = a.logits + r * a.stride;              // 64-bit row base
  const int col0 = warp * 32 * KPT;
  // The first kSpec slots are read before the row's length is known (columns
  // below W always exist), so the two loads overlap; the rest after.
  constexpr int kSpec = KPT < 16 ? KPT : (KPT == 16 ? 16 : 8);
  uint32_t key[KPT];
#pragma unroll
  for (int i = 0; i < kSpec; ++i) {
    const int c = col0 + 32 * i + lane;
    key[i] = c < a.width ? float_key(row[c]) : 0u;
  }
  const int64_t n64 = row_len(a, r);
  int32_t* out = a.indices + r * a.out_stride;             // 64-bit row base
  const int k = a.k;
  if (n64 <= k) {
    write_short_row(out, n64, k);
    return;
  }
  const int n = (int)n64;                                  // <= 32 * KPT * kWarps
  const int live = max(0, min(KPT, (n - col0 + 31) / 32)); // slots holding any column < n (warp-uniform)
#pragma unroll
  for (int i = kSpec; i < KPT; ++i) {
    const int c = col0 + 32 * i + lane;
    key[i] = (i < live && c < n) ? float_key(row[c]) : 0u;
  }
  auto for_each = [&](auto&& f) {
#pragma unroll
    for (int i = 0; i < KPT; ++i)
      if (i < live) f(col0 + 32 * i + lane < n, key[i]);
  };
  const SelectResult s = radix_select<kThreads>(sh, hist_smem, (uint32_t)k, tid, CtaBar{}, for_each);
  compact_regs<kThreads, KPT>(sh, s, n, k, out, tid, CtaBar{}, key, col0, live);
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
