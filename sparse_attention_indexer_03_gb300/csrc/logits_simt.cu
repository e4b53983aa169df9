// FP8 paged MQA logits on the CUDA cores: one thread per token, one CTA per
// (request, 128-column tile).  Full contract (64-bit addressing, MTP masks,
// -inf fill, status bits) with no tensor cores; used for layouts and shapes
// the tensor-core kernel does not take.
//
// Scoring rule (DeepSeek-style indexer, the op `deepgemm_fp8_paged_mqa_logits`
// of aiter PR 4244, "small reproducer"):
//   logits[r, t] = sum_h w[r, h] * ReLU(q[b, j, h] . k[t]) * scale[t],  t < ctx_r
//   logits[r, t] = -inf,                                               ctx_r <= t < W
#include <cuda_fp8.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace sai {
namespace {

constexpr int kSimtThreads = 128;

// Four e4m3fn bytes (little-endian in a word) to four floats; exact, since
// every e4m3fn value is an fp16 value.
__device__ __forceinline__ void fp8x4_to_float(uint32_t w, float& a, float& b, float& c, float& d) {
  __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w & 0xFFFFu), __NV_E4M3);
  __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(w >> 16), __NV_E4M3);
  float2 f0 = __half22float2(*reinterpret_cast<__half2*>(&lo));
  float2 f1 = __half22float2(*reinterpret_cast<__half2*>(&hi));
  a = f0.x; b = f0.y; c = f1.x; d = f1.y;
}

__global__ void __launch_bounds__(kSimtThreads)
logits_simt_kernel(LogitsArgs a) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int N = a.next_n * a.heads;
  const int b = blockIdx.y;
  const int tid = threadIdx.x;

  // Stage this request's q bytes [next_n * H, D] and weights [next_n * H].
  const uint4* qsrc = reinterpret_cast<const uint4*>(a.q + (int64_t)b * N * kHeadDim);
  uint4* qs = reinterpret_cast<uint4*>(smem);
  for (int i = tid; i < N * (kHeadDim / 16); i += kSimtThreads) qs[i] = qsrc[i];
  float* ws = reinterpret_cast<float*>(smem + (size_t)N * kHeadDim);
  for (int i = tid; i < N; i += kSimtThreads) ws[i] = a.weights[(int64_t)b * N + i];
  __syncthreads();

  const int64_t cap = min(a.width, a.bt_stride * (int64_t)a.page_size);
  const int64_t ctx_raw = a.context_lens[b];
  if ((ctx_raw < 0 || ctx_raw > cap) && blockIdx.x == 0 && tid == 0) raise_status(a.status, SAI_STATUS_CTX_CLAMPED);
  const int64_t t = (int64_t)blockIdx.x * kSimtThreads + tid;
  if (t >= a.width) return;
  const int64_t n_max = row_context(ctx_raw, a.next_n, a.next_n - 1, cap);

  float kf[kHeadDim];
  float scale = 0.f;
  bool bad = false;
  if (t < n_max) {
    const int64_t page = a.block_table[(int64_t)b * a.bt_stride + t / a.page_size];
    if (page < 0 || page >= a.num_pages) {
      bad = true;
      raise_status(a.status, SAI_STATUS_BAD_PAGE);
    } else {
      const int slot = (int)(t % a.page_size);
      const uint8_t* pg = a.kv + page * (int64_t)a.page_size * kTokenBytes;
      const uint8_t* vals;
      const uint8_t* sc;
      if (a.layout == SAI_KV_PAGE_SPLIT) {
        vals = pg + (int64_t)slot * kHeadDim;
        sc = pg + (int64_t)a.page_size * kHeadDim + slot * kScaleBytes;
      } else {
        vals = pg + (int64_t)slot * kTokenBytes;
        sc = vals + kHeadDim;
      }
      const uint32_t* v32 = reinterpret_cast<const uint32_t*>(vals);   // 4-byte aligned in both layouts
#pragma unroll
      for (int i = 0; i < kHeadDim / 4; ++i)
        fp8x4_to_float(v32[i], kf[4 * i], kf[4 * i + 1], kf[4 * i + 2], kf[4 * i + 3]);
      scale = *reinterpret_cast<const float*>(sc);
    }
  }

  const uint32_t* q32 = reinterpret_cast<const uint32_t*>(smem);
  for (int j = 0; j < a.next_n; ++j) {
    const int64_t r = (int64_t)b * a.next_n + j;
    const int64_t n_r = row_context(ctx_raw, a.next_n, j, cap);
    float out;
    if (t < n_r) {
      if (bad) {
        out = __int_as_float(0x7fc00000);
      } else {
        float acc = 0.f;
        for (int h = 0; h < a.heads; ++h) {
          const uint32_t* qh = q32 + (size_t)(j * a.heads + h) * (kHeadDim / 4);
          float s = 0.f;
#pragma unroll
          for (int i = 0; i < kHeadDim / 4; ++i) {
            float x0, x1, x2, x3;
            fp8x4_to_float(qh[i], x0, x1, x2, x3);
            s = fmaf(x0, kf[4 * i], s);
            s = fmaf(x1, kf[4 * i + 1], s);
            s = fmaf(x2, kf[4 * i + 2], s);
            s = fmaf(x3, kf[4 * i + 3], s);
          }
          acc = fmaf(ws[j * a.heads + h], fmaxf(s, 0.f), acc);
        }
        out = acc * scale;
      }
    } else {
      out = -INFINITY;
    }
    a.logits[r * a.stride + t] = out;     // 64-bit row base
  }
}

}  // namespace

cudaError_t launch_logits_simt(const LogitsArgs& a, cudaStream_t stream) {
  static int smem_set[64] = {0};
  const int N = a.next_n * a.heads;
  const size_t smem = (size_t)N * kHeadDim + (size_t)N * sizeof(float);
  cudaError_t e = ensure_dynamic_smem(logits_simt_kernel, (size_t)4 * 128 * kHeadDim + 4 * 128 * sizeof(float), smem_set);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (a.width + kSimtThreads - 1) / kSimtThreads;
  dim3 grid((unsigned)tiles, (unsigned)a.batch);
  logits_simt_kernel<<<grid, kSimtThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace sai
