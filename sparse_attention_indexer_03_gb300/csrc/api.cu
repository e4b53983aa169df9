// C ABI of libsai: argument validation and kernel launch.  Every check runs
// before the first CUDA call, so a rejected call touches neither the device
// nor any output.
#include <climits>
#include <cstdint>

#include "common.cuh"

namespace sai {

int device_sm_count() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cached[dev] = n;
  return n;
}

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool supported_page_size(int p) {
  return p == 8 || p == 16 || p == 32 || p == 64 || p == 128 || p == 256;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? SAI_OK : SAI_ERR_CUDA; }

}  // namespace
}  // namespace sai

extern "C" {

int sai_version(void) { return 100; }

int sai_selftest_bounded_wait(int32_t mode, int64_t cycles, uint32_t* status, sai_stream_t stream) {
  if ((mode != 0 && mode != 1) || cycles < 1 || cycles > (int64_t{1} << 31) || status == nullptr)
    return SAI_ERR_INVALID_ARGUMENT;
  if (!sai::aligned(status, 4)) return SAI_ERR_MISALIGNED;
  return sai::from_cuda(sai::launch_bounded_wait_selftest(mode, (long long)cycles, status,
                                                          reinterpret_cast<cudaStream_t>(stream)));
}

const char* sai_error_string(int code) {
  switch (code) {
    case SAI_OK: return "ok";
    case SAI_ERR_INVALID_ARGUMENT: return "invalid argument";
    case SAI_ERR_UNSUPPORTED: return "unsupported shape or option";
    case SAI_ERR_MISALIGNED: return "misaligned pointer";
    case SAI_ERR_WORKSPACE: return "workspace missing or too small";
    case SAI_ERR_CUDA: return "CUDA runtime error";
    default: return "unknown error code";
  }
}

}  // extern "C"

namespace sai {
namespace {

// Checks shared by the logits entry points; fills `a` on success.
int check_logits(const uint8_t* q_fp8, const uint8_t* kv_cache, int64_t num_pages, int32_t page_size,
                 const float* weights, const int32_t* context_lens, const int32_t* block_table,
                 int64_t block_table_stride, int32_t batch, int32_t next_n, int32_t heads, int32_t head_dim,
                 float* logits, int64_t logits_stride, int64_t max_model_len, int32_t kv_layout,
                 uint32_t* status, LogitsArgs& a) {
  if (batch < 0 || next_n < 1 || heads < 1 || head_dim < 1 || page_size < 1 || num_pages < 1 ||
      block_table_stride < 1 || max_model_len < 1 || logits_stride < max_model_len)
    return SAI_ERR_INVALID_ARGUMENT;
  if (!q_fp8 || !kv_cache || !weights || !context_lens || !block_table || !logits) return SAI_ERR_INVALID_ARGUMENT;
  if (kv_layout != SAI_KV_PAGE_SPLIT && kv_layout != SAI_KV_INTERLEAVED) return SAI_ERR_INVALID_ARGUMENT;
  if (head_dim != kHeadDim || !supported_page_size(page_size) || next_n > 4 || (heads != 64 && heads != 128))
    return SAI_ERR_UNSUPPORTED;
  // Byte extents must stay far inside int64.
  if (num_pages > (INT64_MAX / 4) / ((int64_t)page_size * kTokenBytes)) return SAI_ERR_INVALID_ARGUMENT;
  if (logits_stride > (INT64_MAX / 8) / ((int64_t)batch * next_n + 1)) return SAI_ERR_INVALID_ARGUMENT;
  if (block_table_stride > (INT64_MAX / 8) / ((int64_t)batch + 1)) return SAI_ERR_INVALID_ARGUMENT;
  if (batch > 65535) return SAI_ERR_UNSUPPORTED;
  if (!aligned(q_fp8, 16) || !aligned(kv_cache, 16) || !aligned(weights, 16) || !aligned(context_lens, 4) ||
      !aligned(block_table, 4) || !aligned(logits, 4) || !aligned(status, 4))
    return SAI_ERR_MISALIGNED;
  a.q = q_fp8; a.kv = kv_cache; a.num_pages = num_pages; a.page_size = page_size;
  a.weights = weights; a.context_lens = context_lens; a.block_table = block_table;
  a.bt_stride = block_table_stride; a.batch = batch; a.next_n = next_n; a.heads = heads;
  a.logits = logits; a.stride = logits_stride; a.width = max_model_len; a.layout = kv_layout;
  a.status = status;
  return SAI_OK;
}

// Words of the fused launch's workspace for `batch` requests: a tile counter
// per request, a queue of up to 4 rows per request (next_n <= 4), its head,
// tail and done count, and the -inf fill's unit counter.
constexpr int64_t fused_workspace_words(int64_t batch) { return 5 * batch + 4; }

// The fused launch's workspace for sai_paged_mqa_logits_topk_static, for
// callers that cannot hand the library any memory of their own.  Zero when
// the module is loaded; every call that completes leaves it zero again.
constexpr int kStaticMaxBatch = 16384;
static __device__ __align__(256) int32_t g_static_counters[fused_workspace_words(kStaticMaxBatch)];

// Device address of the current device's counters, looked up on every call:
// a cached address would outlive a cudaDeviceReset, which unloads the module.
int static_counters(int32_t** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_counters) != cudaSuccess || p == nullptr) return SAI_ERR_CUDA;
  *out = static_cast<int32_t*>(p);
  return SAI_OK;
}

}  // namespace
}  // namespace sai

extern "C" {

int sai_paged_mqa_logits(const uint8_t* q_fp8, const uint8_t* kv_cache, int64_t num_pages, int32_t page_size,
                         const float* weights, const int32_t* context_lens, const int32_t* block_table,
                         int64_t block_table_stride, int32_t batch, int32_t next_n, int32_t heads,
                         int32_t head_dim, float* logits, int64_t logits_stride, int64_t max_model_len,
                         int32_t kv_layout, uint32_t* status, sai_stream_t stream) {
  using namespace sai;
  LogitsArgs a;
  const int rc = check_logits(q_fp8, kv_cache, num_pages, page_size, weights, context_lens, block_table,
                              block_table_stride, batch, next_n, heads, head_dim, logits, logits_stride,
                              max_model_len, kv_layout, status, a);
  if (rc != SAI_OK || batch == 0) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // The interleaved layout's 132-byte token pitch is no tensor-map stride:
  // its pages come in as bulk copies and are rewritten into the MMA layout.
  if (kv_layout == SAI_KV_PAGE_SPLIT) return from_cuda(launch_logits_tc(a, st));
  return from_cuda(launch_logits_tc_interleaved(a, st));
}

size_t sai_paged_mqa_logits_topk_workspace_bytes(int32_t batch) {
  return batch <= 0 ? 0 : (size_t)sai::fused_workspace_words(batch) * sizeof(int32_t);
}

int sai_paged_mqa_logits_topk(const uint8_t* q_fp8, const uint8_t* kv_cache, int64_t num_pages, int32_t page_size,
                              const float* weights, const int32_t* context_lens, const int32_t* block_table,
                              int64_t block_table_stride, int32_t batch, int32_t next_n, int32_t heads,
                              int32_t head_dim, float* logits, int64_t logits_stride, int64_t max_model_len,
                              int32_t k, int32_t* indices, int64_t indices_stride, void* workspace,
                              size_t workspace_bytes, uint32_t* status, sai_stream_t stream) {
  using namespace sai;
  LogitsArgs a;
  const int rc = check_logits(q_fp8, kv_cache, num_pages, page_size, weights, context_lens, block_table,
                              block_table_stride, batch, next_n, heads, head_dim, logits, logits_stride,
                              max_model_len, SAI_KV_PAGE_SPLIT, status, a);
  if (rc != SAI_OK) return rc;
  if (k < 1 || indices_stride < k || !indices) return SAI_ERR_INVALID_ARGUMENT;
  if (k > 65536 || max_model_len > INT32_MAX) return SAI_ERR_UNSUPPORTED;
  if (indices_stride > (INT64_MAX / 8) / ((int64_t)batch * next_n + 1)) return SAI_ERR_INVALID_ARGUMENT;
  if (!aligned(indices, 4) || !aligned(workspace, 4)) return SAI_ERR_MISALIGNED;
  if (batch == 0) return SAI_OK;
  if (workspace == nullptr || workspace_bytes < (size_t)fused_workspace_words(batch) * sizeof(int32_t))
    return SAI_ERR_WORKSPACE;
  a.indices = indices; a.idx_stride = indices_stride; a.k = k;
  a.req_counter = static_cast<int32_t*>(workspace);
  return from_cuda(launch_logits_tc(a, reinterpret_cast<cudaStream_t>(stream)));
}

int sai_paged_mqa_logits_topk_static(const uint8_t* q_fp8, const uint8_t* kv_cache, int64_t num_pages,
                                     int32_t page_size, const float* weights, const int32_t* context_lens,
                                     const int32_t* block_table, int64_t block_table_stride, int32_t batch,
                                     int32_t next_n, int32_t heads, int32_t head_dim, float* logits,
                                     int64_t logits_stride, int64_t max_model_len, int32_t k, int32_t* indices,
                                     int64_t indices_stride, uint32_t* status, sai_stream_t stream) {
  using namespace sai;
  LogitsArgs a;
  const int rc = check_logits(q_fp8, kv_cache, num_pages, page_size, weights, context_lens, block_table,
                              block_table_stride, batch, next_n, heads, head_dim, logits, logits_stride,
                              max_model_len, SAI_KV_PAGE_SPLIT, status, a);
  if (rc != SAI_OK) return rc;
  if (k < 1 || indices_stride < k || !indices) return SAI_ERR_INVALID_ARGUMENT;
  if (k > 65536 || max_model_len > INT32_MAX) return SAI_ERR_UNSUPPORTED;
  if (indices_stride > (INT64_MAX / 8) / ((int64_t)batch * next_n + 1)) return SAI_ERR_INVALID_ARGUMENT;
  if (!aligned(indices, 4)) return SAI_ERR_MISALIGNED;
  if (batch > kStaticMaxBatch) return SAI_ERR_WORKSPACE;
  if (batch == 0) return SAI_OK;
  int32_t* counters = nullptr;
  const int sc = static_counters(&counters);
  if (sc != SAI_OK) return sc;
  a.indices = indices; a.idx_stride = indices_stride; a.k = k;
  a.req_counter = counters;
  return from_cuda(launch_logits_tc(a, reinterpret_cast<cudaStream_t>(stream)));
}

int sai_paged_mqa_logits_topk_static_reset(sai_stream_t stream) {
  using namespace sai;
  int32_t* counters = nullptr;
  const int sc = static_counters(&counters);
  if (sc != SAI_OK) return sc;
  return from_cuda(cudaMemsetAsync(counters, 0, sizeof(int32_t) * fused_workspace_words(kStaticMaxBatch),
                                   reinterpret_cast<cudaStream_t>(stream)));
}

int sai_indexer_k_quant_insert(const uint16_t* k_bf16, int64_t num_tokens, int32_t head_dim,
                               const int64_t* slot_mapping, uint8_t* kv_cache, int64_t num_pages,
                               int32_t page_size, int32_t kv_layout, uint32_t* status, sai_stream_t stream) {
  using namespace sai;
  if (num_tokens < 0 || head_dim < 1 || num_pages < 1 || page_size < 1) return SAI_ERR_INVALID_ARGUMENT;
  if (num_tokens == 0) return SAI_OK;                     // an empty batch may pass null pointers
  if (!k_bf16 || !slot_mapping || !kv_cache) return SAI_ERR_INVALID_ARGUMENT;
  if (kv_layout != SAI_KV_PAGE_SPLIT && kv_layout != SAI_KV_INTERLEAVED) return SAI_ERR_INVALID_ARGUMENT;
  if (head_dim != kHeadDim || !supported_page_size(page_size)) return SAI_ERR_UNSUPPORTED;
  if (num_pages > (INT64_MAX / 4) / ((int64_t)page_size * kTokenBytes)) return SAI_ERR_INVALID_ARGUMENT;
  if (num_tokens > INT64_MAX / (8 * kHeadDim)) return SAI_ERR_INVALID_ARGUMENT;
  if (!aligned(k_bf16, 16) || !aligned(slot_mapping, 8) || !aligned(kv_cache, 16) || !aligned(status, 4))
    return SAI_ERR_MISALIGNED;
  return from_cuda(launch_k_quant_insert(k_bf16, num_tokens, slot_mapping, kv_cache, num_pages, page_size, kv_layout,
                                         status, reinterpret_cast<cudaStream_t>(stream)));
}

int sai_gather_selected_kv(const int32_t* indices, int64_t indices_stride, int32_t rows, int32_t k, int32_t next_n,
                           const int32_t* block_table, int64_t block_table_stride, int32_t page_size,
                           const uint8_t* kv_pool, int64_t num_pages, int32_t row_bytes, int64_t* row_ids,
                           uint8_t* out, uint32_t* status, sai_stream_t stream) {
  using namespace sai;
  if (rows < 0 || k < 1 || next_n < 1 || indices_stride < k || block_table_stride < 1 || page_size < 1 ||
      num_pages < 1 || row_bytes < 1)
    return SAI_ERR_INVALID_ARGUMENT;
  if (rows == 0) return SAI_OK;
  if (!indices || !block_table || (!row_ids && !out) || (out && !kv_pool)) return SAI_ERR_INVALID_ARGUMENT;
  if (row_bytes % 16 != 0 || row_bytes > 4096 || page_size > 65536) return SAI_ERR_UNSUPPORTED;
  if (num_pages > (INT64_MAX / 4) / ((int64_t)page_size * row_bytes)) return SAI_ERR_INVALID_ARGUMENT;
  if (indices_stride > (INT64_MAX / 8) / ((int64_t)rows + 1)) return SAI_ERR_INVALID_ARGUMENT;
  if (block_table_stride > (INT64_MAX / 8) / ((int64_t)rows + 1)) return SAI_ERR_INVALID_ARGUMENT;
  if ((int64_t)rows * k > INT64_MAX / 4096) return SAI_ERR_INVALID_ARGUMENT;
  if (!aligned(indices, 4) || !aligned(block_table, 4) || !aligned(kv_pool, 16) || !aligned(row_ids, 8) ||
      !aligned(out, 16) || !aligned(status, 4))
    return SAI_ERR_MISALIGNED;
  GatherArgs a;
  a.indices = indices; a.idx_stride = indices_stride; a.rows = rows; a.k = k; a.next_n = next_n;
  a.block_table = block_table; a.bt_stride = block_table_stride; a.page_size = page_size;
  a.pool = kv_pool; a.num_pages = num_pages; a.row_bytes = row_bytes; a.row_ids = row_ids; a.out = out;
  a.status = status;
  return from_cuda(launch_gather_rows(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t sai_top_k_workspace_bytes(int32_t rows, int64_t max_len, int32_t k) {
  if (rows < 0 || max_len < 0 || k < 1) return 0;
  return sai::topk_workspace_bytes(rows, max_len, k);
}

int sai_top_k_per_row_decode(const float* logits, int64_t logits_stride, const int32_t* context_lens,
                             int32_t batch, int32_t next_n, int64_t max_model_len, int32_t k,
                             int32_t* indices, int64_t indices_stride, void* workspace, size_t workspace_bytes,
                             sai_stream_t stream) {
  using namespace sai;
  if (batch < 0 || next_n < 1 || max_model_len < 1 || logits_stride < max_model_len || k < 1 ||
      indices_stride < k)
    return SAI_ERR_INVALID_ARGUMENT;
  if (!logits || !context_lens || !indices) return SAI_ERR_INVALID_ARGUMENT;
  if (k > 65536 || max_model_len > INT32_MAX) return SAI_ERR_UNSUPPORTED;
  const int64_t rows = (int64_t)batch * next_n;
  if (rows > INT32_MAX) return SAI_ERR_UNSUPPORTED;
  if (logits_stride > (INT64_MAX / 8) / (rows + 1) || indices_stride > (INT64_MAX / 8) / (rows + 1))
    return SAI_ERR_INVALID_ARGUMENT;
  if (!aligned(logits, 4) || !aligned(context_lens, 4) || !aligned(indices, 4)) return SAI_ERR_MISALIGNED;
  const size_t need = topk_workspace_bytes((int)rows, max_model_len, k);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need)) return SAI_ERR_WORKSPACE;
  if (rows == 0) return SAI_OK;

  TopKArgs a;
  a.logits = logits; a.stride = logits_stride; a.context_lens = context_lens; a.batch = batch;
  a.next_n = next_n; a.width = max_model_len; a.k = k; a.indices = indices; a.out_stride = indices_stride;
  return from_cuda(launch_topk(a, reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
