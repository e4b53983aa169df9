// Per-row top-k of the indexer logits (`top_k_per_row_decode`, run right after
// the logits launch in aiter PR 4244, opening paragraph).
//
// One CTA per row.  The k-th largest value is found exactly by a radix select
// over order-preserving 32-bit keys (digits of 11, 11 and 10 bits, most
// significant first, each a shared-memory histogram).  The indices are then
// written in a deterministic order: the columns whose key is above the
// threshold, ascending, then the ties at the threshold, lowest columns first.
// Rows whose logical width fits in shared memory are read from global memory
// once; longer rows are re-read per pass.
#include "common.cuh"

namespace sai {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int64_t kCachedKeys = 16384;        // keys kept in shared memory (64 KB)

struct TopkShared {
  uint32_t hist[kBins];
  uint32_t scan[kWarps];
  uint32_t warp_gt[kWarps];
  uint32_t warp_eq[kWarps];
  uint32_t digit;
  uint32_t remaining;
};

// Inclusive prefix sum of one value per thread over the whole CTA; also
// returns the CTA total.
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

template <bool kCached>
__global__ void __launch_bounds__(kThreads)
topk_kernel(TopKArgs a) {
  extern __shared__ uint32_t cached_keys[];
  __shared__ TopkShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t r = blockIdx.x;
  const int b = (int)(r / a.next_n), j = (int)(r % a.next_n);
  const int64_t n = row_context(a.context_lens[b], a.next_n, j, a.width);
  int32_t* out = a.indices + r * a.out_stride;            // 64-bit row base
  const int k = a.k;

  if (n <= k) {                                            // whole row, then -1
    for (int i = tid; i < k; i += kThreads) out[i] = i < n ? i : -1;
    return;
  }
  const float* row = a.logits + r * a.stride;              // 64-bit row base
  if (kCached) {
    for (int64_t i = tid; i < n; i += kThreads) cached_keys[i] = float_key(row[i]);
  }
  auto key_at = [&](int64_t i) -> uint32_t { return kCached ? cached_keys[i] : float_key(row[i]); };

  // ---- radix select: the exact key T of the k-th largest value -------------
  uint32_t prefix = 0, mask = 0, remaining = (uint32_t)k;
#pragma unroll 1
  for (int pass = 0; pass < 3; ++pass) {
    const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
    const int nb = pass < 2 ? 2048 : 1024;
    for (int i = tid; i < nb; i += kThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int64_t i = tid; i < n; i += kThreads) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    // Thread t owns bins [t * per, (t + 1) * per); find the bin holding the
    // `remaining`-th largest key counting down from the top bin.
    const int per = nb / kThreads;
    uint32_t mine = 0;
    for (int i = 0; i < per; ++i) mine += sh.hist[tid * per + i];
    uint32_t total;
    const uint32_t incl = block_inclusive_scan(mine, sh.scan, total);
    uint32_t above = total - incl;                         // keys in bins above mine
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t c = sh.hist[tid * per + i];
      if (above < remaining && above + c >= remaining) {
        sh.digit = (uint32_t)(tid * per + i);
        sh.remaining = remaining - above;
      }
      above += c;
    }
    __syncthreads();
    prefix |= sh.digit << shift;
    mask |= (uint32_t)(nb - 1) << shift;
    remaining = sh.remaining;
    __syncthreads();
  }
  const uint32_t T = prefix;
  const uint32_t n_gt = (uint32_t)k - remaining;          // keys strictly above T

  // ---- ordered compaction: warp w owns columns [w * seg, (w + 1) * seg) -----
  const int64_t seg = ((n + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int64_t lo = warp * seg, hi = min(n, lo + seg);
  uint32_t c_gt = 0, c_eq = 0;
  for (int64_t base = lo; base < hi; base += 32) {
    const int64_t i = base + lane;
    const uint32_t key = i < hi ? key_at(i) : 0u;
    c_gt += __popc(__ballot_sync(0xffffffffu, i < hi && key > T));
    c_eq += __popc(__ballot_sync(0xffffffffu, i < hi && key == T));
  }
  if (lane == 0) { sh.warp_gt[warp] = c_gt; sh.warp_eq[warp] = c_eq; }
  __syncthreads();
  uint32_t off_gt = 0, off_eq = 0;
  for (int w = 0; w < warp; ++w) { off_gt += sh.warp_gt[w]; off_eq += sh.warp_eq[w]; }
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int64_t base = lo; base < hi; base += 32) {
    const int64_t i = base + lane;
    const uint32_t key = i < hi ? key_at(i) : 0u;
    const bool gt = i < hi && key > T, eq = i < hi && key == T;
    const uint32_t bgt = __ballot_sync(0xffffffffu, gt), beq = __ballot_sync(0xffffffffu, eq);
    if (gt) out[off_gt + __popc(bgt & lt_mask)] = (int32_t)i;
    if (eq) {
      const uint32_t rank = off_eq + __popc(beq & lt_mask);
      if (rank < remaining) out[n_gt + rank] = (int32_t)i;
    }
    off_gt += __popc(bgt);
    off_eq += __popc(beq);
  }
}

}  // namespace

size_t topk_workspace_bytes(int, int64_t, int) { return 0; }

cudaError_t launch_topk(const TopKArgs& a, cudaStream_t stream) {
  static int smem_set[64] = {0};
  const int64_t rows = (int64_t)a.batch * a.next_n;
  if (rows == 0) return cudaSuccess;
  if (a.width <= kCachedKeys) {
    const size_t smem = (size_t)a.width * sizeof(uint32_t);
    cudaError_t e = ensure_dynamic_smem(topk_kernel<true>, kCachedKeys * sizeof(uint32_t), smem_set);
    if (e != cudaSuccess) return e;
    topk_kernel<true><<<(unsigned)rows, kThreads, smem, stream>>>(a);
  } else {
    topk_kernel<false><<<(unsigned)rows, kThreads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace sai
