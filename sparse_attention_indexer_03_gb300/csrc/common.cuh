// Shared definitions of the libsai kernels (device side and launch helpers).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "sai.h"

namespace sai {

constexpr int kHeadDim = 128;      // D: bytes of one token's FP8 values
constexpr int kScaleBytes = 4;     // one fp32 scale per token
constexpr int kTokenBytes = kHeadDim + kScaleBytes;

// Tokens row r = b * next_n + j sees: ctx_b - next_n + j + 1 clamped to [0, cap]
// (MTP row j sees one more token than row j - 1).
__host__ __device__ __forceinline__ int64_t row_context(int64_t ctx_b, int next_n, int j, int64_t cap) {
  int64_t n = ctx_b - next_n + j + 1;
  n = n < 0 ? 0 : n;
  return n > cap ? cap : n;
}

__device__ __forceinline__ void raise_status(uint32_t* status, uint32_t bits) {
  if (status != nullptr) atomicOr(status, bits);
}

// Order-preserving 32-bit key of an fp32 value: a > b  <=>  key(a) > key(b)
// for non-NaN values; -0.0 and +0.0 map to the same key.
__device__ __forceinline__ uint32_t float_key(float x) {
  uint32_t u = __float_as_uint(x);
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace sai

// Launchers implemented by the kernel files and called by api.cu after validation.
namespace sai {

struct LogitsArgs {
  const uint8_t* q;
  const uint8_t* kv;
  int64_t num_pages;
  int page_size;
  const float* weights;
  const int32_t* context_lens;
  const int32_t* block_table;
  int64_t bt_stride;
  int batch;
  int next_n;
  int heads;
  float* logits;
  int64_t stride;
  int64_t width;         // W = max_model_len
  int layout;
  uint32_t* status;
  // fused top-k (indices null: logits only)
  int32_t* indices = nullptr;
  int64_t idx_stride = 0;
  int k = 0;
  int32_t* req_counter = nullptr;
};

cudaError_t launch_logits_tc(const LogitsArgs& a, cudaStream_t stream);
cudaError_t launch_logits_tc_interleaved(const LogitsArgs& a, cudaStream_t stream);
cudaError_t launch_logits_tc_dual(const LogitsArgs& a, cudaStream_t stream);
cudaError_t launch_bounded_wait_selftest(int mode, long long cycles, uint32_t* status, cudaStream_t stream);

struct TopKArgs {
  const float* logits;
  int64_t stride;
  const int32_t* context_lens;
  int batch;
  int next_n;
  int64_t width;
  int k;
  int32_t* indices;
  int64_t out_stride;
  bool longest_first = false;   // set by launch_topk: CTAs take the rows longest first
};

cudaError_t launch_topk(const TopKArgs& a, cudaStream_t stream);
struct GatherArgs {
  const int32_t* indices;     // [rows, idx_stride]
  int64_t idx_stride;
  int32_t rows, k, next_n;
  const int32_t* block_table; // [rows / next_n, bt_stride]
  int64_t bt_stride;
  int32_t page_size;
  const uint8_t* pool;        // token-major rows of row_bytes
  int64_t num_pages;
  int32_t row_bytes;
  int64_t* row_ids;           // [rows, k] or null
  uint8_t* out;               // [rows, k, row_bytes] or null
  uint32_t* status;
};
cudaError_t launch_gather_rows(const GatherArgs& a, cudaStream_t stream);
cudaError_t launch_k_quant_insert(const uint16_t* k, int64_t num_tokens, const int64_t* slots, uint8_t* cache,
                                  int64_t num_pages, int page_size, int layout, uint32_t* status,
                                  cudaStream_t stream);
size_t topk_workspace_bytes(int rows, int64_t max_len, int k);

int device_sm_count();

// Raise a kernel's dynamic shared-memory limit to `bytes` once per device
// (a function attribute, not a stream operation; done before first use).
// `done` is a per-kernel array of 64 entries owned by the caller.
template <typename F>
cudaError_t ensure_dynamic_smem(F* func, size_t bytes, int* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && (size_t)done[dev] >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  // Every kernel of the library prefers the largest shared-memory carve-out,
  // so consecutive launches (logits, then top-k) keep one SM configuration
  // instead of reconfiguring the L1 / shared split between them.
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = (int)bytes;
  return e;
}

}  // namespace sai
