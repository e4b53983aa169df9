// Indexer K-cache write: per-token FP8 quantisation of new K rows and their
// insertion into the paged cache through int64 slots (the cache kernels'
// slot rule of ATOM PR 2533, "[MLA] Address Triton decode KV rows with int64
// ids", section "Problem"; the token format is the one the logits op reads:
// 128 e4m3fn bytes and one fp32 scale).
//
// A warp per token: lane l holds the token's values 4l .. 4l+3 (8 bytes of
// bf16), the warp's maximum magnitude gives scale = amax / 448 (1 for an
// all-zero row), each lane converts its four quotients value / scale with one
// round-to-nearest-even, saturating cvt per pair and stores 4 code bytes
// (the warp writes the token's 128 value bytes in one coalesced store); lane
// 0 stores the scale.  HBM-bound: 256 + 8 bytes read and 132 written per token.
#include "common.cuh"
#include "ptx.cuh"

namespace sai {
namespace {

constexpr int kQuantWarps = 8;

__device__ __forceinline__ uint32_t fp8x2(float hi, float lo) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Quantise and store one token whose row bits and slot have been read.
__device__ __forceinline__ void put_token(uint2 raw, int64_t s, int lane, uint8_t* cache, int64_t n_slots,
                                          int page_size, int64_t page_bytes, int layout, uint32_t* status) {
  if (s < 0) return;                                        // padding token (warp-uniform)
  if (s >= n_slots) {
    if (lane == 0) raise_status(status, SAI_STATUS_BAD_PAGE);
    return;
  }
  const float f0 = __uint_as_float(raw.x << 16), f1 = __uint_as_float(raw.x & 0xFFFF0000u);
  const float f2 = __uint_as_float(raw.y << 16), f3 = __uint_as_float(raw.y & 0xFFFF0000u);
  // Magnitudes of non-negative floats order like their bit patterns.
  const uint32_t m = max(max(__float_as_uint(fabsf(f0)), __float_as_uint(fabsf(f1))),
                         max(__float_as_uint(fabsf(f2)), __float_as_uint(fabsf(f3))));
  const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, m));
  const float scale = amax > 0.f ? amax / 448.f : 1.f;
  const uint32_t codes = fp8x2(f1 / scale, f0 / scale) | (fp8x2(f3 / scale, f2 / scale) << 16);
  const int64_t page = s / page_size, pos = s - page * page_size;
  uint8_t* base = cache + page * page_bytes;                // 64-bit offsets throughout
  uint8_t* vals;
  float* sc;
  if (layout == SAI_KV_PAGE_SPLIT) {
    vals = base + pos * kHeadDim;
    sc = reinterpret_cast<float*>(base + (int64_t)page_size * kHeadDim + pos * kScaleBytes);
  } else {
    vals = base + pos * kTokenBytes;
    sc = reinterpret_cast<float*>(vals + kHeadDim);
  }
  reinterpret_cast<uint32_t*>(vals)[lane] = codes;
  if (lane == 0) *sc = scale;
}

// Each warp takes two tokens at a time and reads both rows and both slots
// before using any, so one round of memory latency covers a 16K-token batch.
__global__ void __launch_bounds__(kQuantWarps * 32)
k_quant_insert_kernel(const uint16_t* __restrict__ k, int64_t num_tokens, const int64_t* __restrict__ slots,
                      uint8_t* __restrict__ cache, int64_t num_pages, int page_size, int layout, uint32_t* status) {
  ptx::wait_prerequisites();
  ptx::launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * kQuantWarps;
  const int64_t n_slots = num_pages * page_size;
  const int64_t page_bytes = (int64_t)page_size * kTokenBytes;
  for (int64_t t = 2 * ((int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5)); t < num_tokens; t += 2 * warps) {
    const bool two = t + 1 < num_tokens;                    // warp-uniform
    const int64_t s0 = __ldg(slots + t);
    const int64_t s1 = two ? __ldg(slots + t + 1) : -1;
    const uint2 r0 = __ldg(reinterpret_cast<const uint2*>(k + t * kHeadDim) + lane);
    const uint2 r1 = two ? __ldg(reinterpret_cast<const uint2*>(k + (t + 1) * kHeadDim) + lane) : make_uint2(0, 0);
    put_token(r0, s0, lane, cache, n_slots, page_size, page_bytes, layout, status);
    put_token(r1, s1, lane, cache, n_slots, page_size, page_bytes, layout, status);
  }
}

}  // namespace

cudaError_t launch_k_quant_insert(const uint16_t* k, int64_t num_tokens, const int64_t* slots, uint8_t* cache,
                                  int64_t num_pages, int page_size, int layout, uint32_t* status,
                                  cudaStream_t stream) {
  if (num_tokens == 0) return cudaSuccess;
  const int64_t blocks_needed = (num_tokens + 2 * kQuantWarps - 1) / (2 * kQuantWarps);
  const int sms = device_sm_count();
  const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 8;      // grid-stride beyond 8 CTAs per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks_needed < cap ? blocks_needed : cap));
  cfg.blockDim = dim3(kQuantWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // start while the previous kernel drains
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_quant_insert_kernel, k, num_tokens, slots, cache, num_pages, page_size, layout,
                            status);
}

}  // namespace sai
