// Per-row top-k of the indexer logits (`top_k_per_row_decode`, run right after
// the logits launch in aiter PR 4244, opening paragraph).
//
// One CTA of 1024 threads per row runs the exact radix select of select.cuh
// and writes the row's indices in a deterministic order: the columns strictly
// above the threshold, ascending, then the ties at the threshold, lowest
// columns first.  Rows of a logical width up to 16384 are held in registers
// (each thread a run of KPT consecutive columns, read from global memory
// once); wider rows up to 40960 long are copied into shared memory once their
// length is known, and longer ones re-read from global memory (mostly L2) on
// each pass.
//
// The kernel is launched as a programmatic dependent of the previous kernel
// in the stream (the logits launch): it may start while that kernel drains,
// and waits for it to complete before reading any logits.  It then lets its
// own dependents start at once: with one CTA per row, a decode batch leaves
// most SMs free, where the next launch can run its set-up.
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"
#include "select.cuh"

namespace sai {
namespace {

constexpr int kThreads = 1024;
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
#pragma unroll
  for (int i = 0; i < KPT; ++i) {
    const int c = base + i;
    key[i] = c < a.width ? float_key(row[c]) : 0u;
  }
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

// ---- wider rows: a row of up to kSmemKeys columns has its keys copied into
// shared memory once its length is known (each lane then a run of about
// n / 512 columns); a longer row is re-read from L2 on every pass ------------
constexpr int kSmemKeys = 40960;
constexpr size_t kSmemKeysBytes = kSelectSmem + 4 * (kSmemKeys + 4);

__global__ void __launch_bounds__(kThreads)
topk_smem_kernel(TopKArgs a) {
  extern __shared__ __align__(16) uint8_t topk_smem[];
  __shared__ SelectShared<kThreads> sh;
  ptx::wait_prerequisites();
  ptx::launch_dependents();     // the next logits launch may take the SMs this grid leaves idle
  const int64_t r = blockIdx.x;
  const int64_t n = row_len(a, r);
  int32_t* out = a.indices + r * a.out_stride;             // 64-bit row base
  if (n <= a.k) {
    write_short_row(out, n, a.k);
    return;
  }
  uint32_t* hist = reinterpret_cast<uint32_t*>(topk_smem);
  const float* row = a.logits + r * a.stride;
  if (n <= kSmemKeys) {
    uint32_t* key_base = reinterpret_cast<uint32_t*>(topk_smem + kSelectSmem);
    const uint32_t* keys = stage_keys<kThreads>(row, (int)n, key_base, threadIdx.x);
    topk_row_smem<kThreads>(keys, (int)n, a.k, out, sh, hist, threadIdx.x, CtaBar{});
  } else {
    topk_row_stream<kThreads>(row, n, a.k, out, sh, hist, threadIdx.x, CtaBar{});
  }
}

template <typename Kern>
cudaError_t launch_pdl(Kern kern, unsigned grid, const TopKArgs& a, cudaStream_t stream, int* smem_set,
                       size_t smem, size_t smem_max) {
  cudaError_t e = ensure_dynamic_smem(kern, smem_max, smem_set);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
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
  static int set4[64], set8[64], set16[64], set_smem[64];
  cudaError_t e;
  if (a.width <= 4 * kThreads) e = launch_pdl(topk_reg_kernel<4>, g, a, stream, set4, kSelectSmem, kSelectSmem);
  else if (a.width <= 8 * kThreads) e = launch_pdl(topk_reg_kernel<8>, g, a, stream, set8, kSelectSmem, kSelectSmem);
  else if (a.width <= 16 * kThreads) e = launch_pdl(topk_reg_kernel<16>, g, a, stream, set16, kSelectSmem, kSelectSmem);
  else e = launch_pdl(topk_smem_kernel, g, a, stream, set_smem,
                     kSelectSmem + 4 * (size_t)(std::min<int64_t>(a.width, kSmemKeys) + 4), kSmemKeysBytes);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace sai
