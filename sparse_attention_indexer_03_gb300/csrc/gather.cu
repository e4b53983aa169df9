// Consumer gather: the KV rows of the tokens the top-k selected, addressed
// through the block table with int64 row ids (ATOM PR 2533, "[MLA] Address
// Triton decode KV rows with int64 ids": row id * row stride must be formed
// in 64 bits; an int32 product wraps past row 2^31 / 576).
//
// A warp takes 8 (row, index) entries at a time: lanes 0-7 read the 8 indices
// and their table entries and form the row ids; then the warp copies the 8
// rows, 16 bytes per lane per unit, issuing up to 8 loads per lane before
// storing them, so a whole batch of rows is in flight at once.  HBM-bound:
// each selected row is read once and written once.
#include "common.cuh"
#include "ptx.cuh"

namespace sai {
namespace {

constexpr int kGatherWarps = 8;
constexpr int kEntries = 8;        // entries per warp batch
constexpr int kUnitsInFlight = 8;  // 16-byte loads per lane before the stores

__global__ void __launch_bounds__(kGatherWarps * 32)
gather_rows_kernel(GatherArgs a) {
  ptx::wait_prerequisites();
  const int lane = threadIdx.x & 31;
  const int64_t n_entries = (int64_t)a.rows * a.k;
  const int upe = a.row_bytes / 16;                          // 16-byte units per row
  const int64_t warps = (int64_t)gridDim.x * kGatherWarps;
  for (int64_t e0 = ((int64_t)blockIdx.x * kGatherWarps + (threadIdx.x >> 5)) * kEntries; e0 < n_entries;
       e0 += warps * kEntries) {
    int64_t rid = -1;
    bool bad = false;
    if (lane < kEntries && e0 + lane < n_entries) {
      const int64_t e = e0 + lane;
      const int64_t r = e / a.k, i = e - r * a.k;
      const int32_t t = a.indices[r * a.idx_stride + i];
      if (t >= 0) {
        const int64_t b = r / a.next_n;
        const int64_t entry = t / a.page_size;
        if (entry < a.bt_stride) {
          const int64_t page = a.block_table[b * a.bt_stride + entry];   // widened before use
          if (page >= 0 && page < a.num_pages) rid = page * a.page_size + t % a.page_size;
          else bad = true;
        } else {
          bad = true;
        }
      }
      if (a.row_ids) a.row_ids[e] = rid;
    }
    if (bad) raise_status(a.status, SAI_STATUS_BAD_PAGE);
    if (!a.out) continue;
    const int n_here = (int)min((int64_t)kEntries, n_entries - e0);
    const int units = n_here * upe;
    for (int q0 = 0; q0 < units; q0 += 32 * kUnitsInFlight) {
      uint4 v[kUnitsInFlight];
#pragma unroll
      for (int m = 0; m < kUnitsInFlight; ++m) {
        const int q = q0 + m * 32 + lane;
        const int j = min(q, units - 1) / upe;                 // entry of this unit (all lanes shuffle)
        const int64_t rj = __shfl_sync(0xffffffffu, rid, j);
        v[m] = make_uint4(0, 0, 0, 0);
        if (q < units && rj >= 0) {
          const int u = q - j * upe;
          v[m] = __ldg(reinterpret_cast<const uint4*>(a.pool + rj * a.row_bytes) + u);   // 64-bit offset
        }
      }
#pragma unroll
      for (int m = 0; m < kUnitsInFlight; ++m) {
        const int q = q0 + m * 32 + lane;
        if (q < units) {
          const int j = q / upe, u = q - j * upe;
          reinterpret_cast<uint4*>(a.out + (e0 + j) * a.row_bytes)[u] = v[m];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_gather_rows(const GatherArgs& a, cudaStream_t stream) {
  const int64_t n_entries = (int64_t)a.rows * a.k;
  if (n_entries == 0) return cudaSuccess;
  const int64_t blocks_needed = (n_entries + kGatherWarps * kEntries - 1) / (kGatherWarps * kEntries);
  const int sms = device_sm_count();
  const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 8;        // grid-stride beyond 8 CTAs per SM
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(blocks_needed < cap ? blocks_needed : cap));
  cfg.blockDim = dim3(kGatherWarps * 32);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // start while the top-k drains
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gather_rows_kernel, a);
}

}  // namespace sai
