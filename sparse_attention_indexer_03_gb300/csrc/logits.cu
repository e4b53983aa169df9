// FP8 paged MQA logits on the sm_103a tensor cores.
//
//   logits[r, t] = sum_h w[r, h] * ReLU(q[b, j, h] . k[t]) * scale[t]   (t < ctx_r)
//   logits[r, t] = -inf                                                 (ctx_r <= t < W)
//
// (the op `deepgemm_fp8_paged_mqa_logits` of aiter PR 4244, "small
// reproducer"; rows r = b * next_n + j; MTP row j sees ctx_b - next_n + j + 1
// tokens).
//
// One persistent CTA per SM, warp-specialised:
//   warps 0-2  producers, taking the tiles round-robin: block-table reads
//              (int64 widened, bounds-checked, copied ahead with cp.async) and
//              TMA gathers of the K pages into a ring of 128-token stages.  A
//              stage holds 128/P pages of P < 128 tokens, each its own pair of
//              TMA boxes, values and scales loaded separately (aiter PR 6626,
//              "paged MQA logits: 8-token pages ...", section 1), or half of a
//              256-token page.  A copy instruction costs the issuing warp
//              hundreds of cycles whatever its size, so a tile's page copies
//              go out as one warp-wide instruction (one lane per page) and
//              three warps issue in parallel (two where the ring is too
//              shallow for three: see ring_waits_unambiguous).  Warp 0 also
//              computes the work partition.  Q [next_n * H, 128] of each
//              request is loaded once into one of two Q slots.
//              Interleaved caches (IL; each token's 128 value bytes, then its
//              4 scale bytes, as the aiter PR 4244 reproducer builds them):
//              the 132-byte token pitch is no tensor-map stride, so a lane
//              bulk-copies its page as stored into the stage, and once the
//              tile has landed the warp rewrites it in place into the layout
//              above; the MMA and the epilogue are the same.
//   warp 3     TMEM allocation and the MMA issuer: tcgen05.mma kind::f8f6f4,
//              A = the K stage (128 tokens x 128 B, K-major, 128-byte
//              swizzle), B = Q (whole rows j, <= 256 columns per job), fp32
//              accumulators in a ring of TMEM stages.  On decode-like shapes
//              (one job of <= 128 columns per tile) with pages of >= 64
//              tokens, warp 2 is a second MMA issuer taking the odd tiles
//              (Cfg::DUAL; compiled in logits_dual.cu) and warps 0-1 produce.
//   warps 4-11 two epilogue warpgroups taking alternate jobs: tcgen05.ld of a
//              token's accumulator row, ReLU, per-head weight, scale, -inf
//              mask, coalesced stores at a 64-bit row base (aiter PR 4244,
//              "Fix"); then their share of the -inf fill of columns past the
//              last tile of each request.
//
// Work partition: the 128-token tiles of all requests, in request order,
// split into equal contiguous ranges, one per CTA; the fill split the same
// way in units of (row, 4096 columns).  Each CTA derives its range from
// context_lens itself, with no global scratch and no atomics.  (The fused
// launch adds per-request counters and a ready-row queue in its workspace,
// and shares a fill-heavy launch's fill units through one counter there.)
//
// Every wait is bounded: when one runs out, the CTA raises SAI_STATUS_TIMEOUT,
// stops, lets its in-flight copies and MMAs drain (again bounded), frees its
// TMEM and exits.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "ptx.cuh"
#include "select.cuh"

namespace sai {
namespace {

constexpr int kTile = 128;                       // tokens per MMA tile (M)
constexpr int kProducers = 3;                    // warps 0 .. kProducers - 1 may produce
constexpr int kMmaWarp = kProducers;             // then the MMA warp
constexpr int kFirstEpiWarp = kProducers + 1;    // then two epilogue warpgroups
constexpr int kEpiWarps = 8;
constexpr int kThreadsTc = (kProducers + 1 + kEpiWarps) * 32;
constexpr int kStageBytes = kTile * kHeadDim;    // 16 KB of K values per stage
constexpr int kScaleSlot = kTile * kScaleBytes;  // 512 B of scales per stage, in token order
constexpr int kFillCols = 4096;
constexpr long long kWaitBudget = 1LL << 31;     // SM clock cycles before a wait gives up
constexpr int kMaxSmem = 232448;                 // dynamic shared memory per CTA on sm_100-family

constexpr int kFlagNew = 1, kFlagLast = 2;
constexpr int kLookahead = 8;                    // tiles of page ids copied ahead of the producer

struct TcParams {
  const int32_t* context_lens;
  const int32_t* block_table;
  int64_t bt_stride;
  const uint8_t* kv;
  int64_t num_pages;
  int page_size;
  const float* weights;
  float* logits;
  int64_t stride;
  int64_t width;
  int64_t cap;          // min(W, bt_stride * P): longest context a row can have
  int batch;
  uint32_t* status;
  // fused top-k (null indices: logits only)
  int32_t* indices;
  int64_t idx_stride;
  int k;
  int32_t* req_counter;   // fused top-k workspace, zero between launches: [batch] tiles counted in
                          // so far, [4 * batch] ready-row queue, head, tail, done
};

// Batches up to this many requests have their context lengths copied into
// shared memory by the partition, so the walks over requests read them there.
constexpr int kCtxSmem = 512;

// An interleaved stage: a tile of tokens as stored (128 * 132 = 16,896 B),
// rewritten in place into the 16 KB MMA layout; rounded to 1 KB so every
// stage base keeps the 128-byte swizzle's 1024-byte alignment.
constexpr int kStageBytesIl = (kTile * kTokenBytes + 1023) / 1024 * 1024;

// The producers wait for a stage's release by phase parity, which cannot tell
// the release of the stage's use u - 1 from that of use u - 2: the wait is
// sound only if use u - 2 is known released when it starts.  A producer warp
// has seen the releases of its own earlier tiles' predecessors (tiles
// i - m * producers - stages, m >= 1).  Releases come from the epilogue
// warpgroups: when a tile is several jobs, every release needs both
// warpgroups, so releases complete in tile order and stages >= producers is
// enough; when a tile is one job, the two warpgroups take alternate tiles and
// only releases two tiles apart are ordered, so some m must leave
// stages - m * producers even and non-negative.
constexpr bool ring_waits_unambiguous(int stages, int producers, int jobs_per_tile) {
  if (stages < producers) return false;
  if (jobs_per_tile > 1) return true;
  for (int m = 1; m * producers <= stages; ++m)
    if ((stages - m * producers) % 2 == 0) return true;
  return false;
}

constexpr int deepest_sound_ring(int fit, int producers, int jobs_per_tile) {
  for (int st = fit; st >= 2; --st)
    if (ring_waits_unambiguous(st, producers, jobs_per_tile)) return st;
  return 0;
}

// IL: K pages in the interleaved layout (each token's 128 value bytes then its
// 4 scale bytes), copied into the stage as stored and rewritten there into the
// MMA layout by the producers.
template <int NEXT_N, int H, bool IL = false, bool DUAL_OK = false>
struct Cfg {
  static constexpr int N = NEXT_N * H;
  static constexpr int NC = N <= 256 ? N : (N % 256 == 0 ? 256 : H);   // accumulator columns per job
  static constexpr int C = N / NC;                                     // jobs per tile
  static constexpr int ROWS = NC / H;                                  // rows j per job
  static constexpr int ACC = NC <= 128 ? 4 : 2;                        // TMEM accumulator stages
  static constexpr int TMEM_COLS = ACC * NC <= 256 ? 256 : 512;
  static constexpr int QBOX = N <= 256 ? N : (N % 256 == 0 ? 256 : 192);
  static constexpr int Q_BYTES = N * kHeadDim;
  static constexpr uint32_t IDESC = ptx::idesc_e4m3_f32(kTile, NC);
  // K ring depth: as many 128-token stages as fit beside two Q slots (at
  // most 8), with as many producer warps (3, else 2) as keep the ring's
  // parity waits sound.
  static constexpr int FIXED = 1024 + 2 * Q_BYTES + kProducers * kLookahead * 32 * 4 + 8 * (4 + 2 * ACC + 2) + 64 +
                               kCtxSmem * 4;
  static constexpr int STAGE_BYTES = IL ? kStageBytesIl : kStageBytes;
  // The tile's head weights [next_n, H] fp32 come into the stage with its K
  // pages when the epilogue's sums are long (N >= 256; page-split caches:
  // interleaved ones lose a stage to it): read there, not from global memory.
  static constexpr bool STAGE_W = !IL && N >= 256;
  static constexpr int W_BYTES = STAGE_W ? NEXT_N * H * 4 : 0;
  static constexpr int PER_STAGE = STAGE_BYTES + kScaleSlot + 16 + 16 + (IL ? 8 : 0) + W_BYTES;
  static constexpr int FIT = (kMaxSmem - FIXED) / PER_STAGE < 8 ? (kMaxSmem - FIXED) / PER_STAGE : 8;
  // Tiles of one job of at most 128 columns (decode-like shapes: the MMA
  // warp's per-tile loop, not the tensor pipe, sets the tile rate): two MMA
  // warps take alternate tiles (warp kMmaWarp the even ones, warp 2 the odd
  // ones), each with its own two of the four accumulators, fed by two
  // producer warps.  An even ring gives every stage to one MMA warp.  Only
  // where the launch asks for it (DUAL_OK: pages of 64 tokens or more, at
  // most two per tile): a tile of small pages costs its producer a copy-
  // engine operation per page and scale run, and two producers fall behind.
  static constexpr bool DUAL = DUAL_OK && !IL && C == 1 && N <= 128;
  static constexpr int PRODUCERS = DUAL ? 2 : (ring_waits_unambiguous(FIT, kProducers, C) ? kProducers : 2);
  static constexpr int STAGES = deepest_sound_ring(FIT, PRODUCERS, C);
  static_assert(STAGES >= 2 && ring_waits_unambiguous(STAGES, PRODUCERS, C), "shared memory");
  static_assert(!DUAL || (STAGES % 2 == 0 && ACC % 2 == 0 && kMmaWarp == 3), "two MMA warps");
  static_assert(N % QBOX == 0 && NC % 16 == 0 && NC <= 256 && ACC * NC <= 512, "shape");
};

struct Part {        // this CTA's share of the work
  int b0, t0, n_tiles;
  int fb0, fu0, n_units;
  int n_sel;         // rows longer than k (the fused top-k's queue length)
  int u_total;       // fill units of the launch where they outweigh its tiles four times over (else -1)
};

struct SmemLayout {
  uint32_t k, q, sc, meta, wst, ids, bar, misc, ctx, total;
};

__host__ __device__ inline SmemLayout smem_layout(int stages, int q_bytes, int acc, bool il, int w_bytes) {
  SmemLayout L;
  L.k = 0;
  L.q = L.k + stages * (il ? kStageBytesIl : kStageBytes);
  L.sc = L.q + 2 * q_bytes;
  L.meta = L.sc + stages * kScaleSlot;
  L.wst = L.meta + stages * 16;                        // per-stage head weights (w_bytes each, may be 0)
  L.ids = L.wst + stages * w_bytes;
  L.bar = L.ids + kProducers * kLookahead * 32 * 4;
  L.misc = L.bar + 8 * (2 * stages + 4 + 2 * acc + 2 + (il ? stages : 0));
  L.ctx = L.misc + 64;
  L.total = L.ctx + kCtxSmem * 4;
  return L;
}

__device__ __forceinline__ int64_t ctx_eff(int64_t raw, int64_t cap) { return raw < 0 ? 0 : (raw > cap ? cap : raw); }

__device__ __forceinline__ int64_t warp_sum64(int64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ int64_t warp_incl_scan64(int64_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int64_t n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Tiles of request b (compute part) and its fill units.
__device__ __forceinline__ int64_t req_tiles(int64_t ce) { return (ce + kTile - 1) / kTile; }
template <int NEXT_N>
__device__ __forceinline__ int64_t req_units(int64_t ce, int64_t W) {
  const int64_t fs = min(W, req_tiles(ce) * kTile);
  return (int64_t)NEXT_N * ((W - fs + kFillCols - 1) / kFillCols);
}

// Balanced split of n units over g parts: part i gets [begin(i), begin(i + 1)).
__device__ __forceinline__ int64_t split_begin(int64_t n, int64_t g, int64_t i) {
  const int64_t q = n / g, r = n % g;
  return q * i + (i < r ? i : r);
}

// Warp 0: split the tiles and the fill units of all requests evenly across
// the grid and locate this CTA's first tile and first fill unit.  For up to
// 32 * kCtxRegs requests, lane l reads requests [l * R, (l + 1) * R) once
// (R = ceil(batch / 32)) and one warp scan over the lane totals places every
// request; larger batches are scanned 32 requests at a time.
constexpr int kCtxRegs = 16;

template <int NEXT_N>
__device__ void compute_partition(const TcParams& p, Part* part, int32_t* ctx_s, int lane) {
  const int64_t G = gridDim.x, cta = blockIdx.x;
  int b0 = 0, t0 = 0, fb0 = 0, fu0 = 0;
  int64_t tb = 0, te = 0, ub = 0, ue = 0;
  int64_t with_tiles = 0;                            // rows longer than k (per lane, then summed)
  int64_t u_all = -1;                                // fill units of a fill-heavy launch
  bool clamped = false;
  static_assert(32 * kCtxRegs == kCtxSmem, "every request of a staged batch is read by the register path");
  if (p.batch <= 32 * kCtxRegs) {
    const int R = (p.batch + 31) / 32;
    // Every load of the lane's lengths is in flight before the first use;
    // the per-request sums then cover the lane's R requests only.
    int32_t rl[kCtxRegs], tl[kCtxRegs], ul[kCtxRegs];
#pragma unroll
    for (int x = 0; x < kCtxRegs; ++x) {
      const int b = lane * R + x;
      rl[x] = x < R && b < p.batch ? p.context_lens[b] : 0;
      tl[x] = 0;
      ul[x] = 0;
    }
    int64_t lt = 0, lu = 0;
#pragma unroll
    for (int x = 0; x < kCtxRegs; ++x) {
      if (x >= R) break;
      const int b = lane * R + x;
      if (b >= p.batch) continue;
      const int64_t raw = rl[x];
      ctx_s[b] = rl[x];
      clamped |= raw < 0 || raw > p.cap;
      const int64_t ce = ctx_eff(raw, p.cap);
      tl[x] = (int32_t)req_tiles(ce);
      ul[x] = (int32_t)req_units<NEXT_N>(ce, p.width);
      lt += tl[x];
      lu += ul[x];
      if (p.k > 0)
        for (int j = 0; j < NEXT_N; ++j) with_tiles += row_context(raw, NEXT_N, j, p.cap) > p.k ? 1 : 0;
    }
    const int64_t it = warp_incl_scan64(lt, lane), iu = warp_incl_scan64(lu, lane);
    const int64_t T = __shfl_sync(0xffffffffu, it, 31), U = __shfl_sync(0xffffffffu, iu, 31);
    u_all = U > 4 * T ? U : -1;
    tb = split_begin(T, G, cta); te = split_begin(T, G, cta + 1);
    ub = split_begin(U, G, cta); ue = split_begin(U, G, cta + 1);
    int fb = -1, ft = 0, gb = -1, gu = 0;
    int64_t at = it - lt, au = iu - lu;              // units before this lane's first request
#pragma unroll
    for (int x = 0; x < kCtxRegs; ++x) {
      if (x >= R) break;
      if (tl[x] > 0 && at <= tb && tb < at + tl[x]) { fb = lane * R + x; ft = (int)(tb - at); }
      if (ul[x] > 0 && au <= ub && ub < au + ul[x]) { gb = lane * R + x; gu = (int)(ub - au); }
      at += tl[x];
      au += ul[x];
    }
    const uint32_t bt = __ballot_sync(0xffffffffu, fb >= 0), bu = __ballot_sync(0xffffffffu, gb >= 0);
    if (bt) { b0 = __shfl_sync(0xffffffffu, fb, __ffs(bt) - 1); t0 = __shfl_sync(0xffffffffu, ft, __ffs(bt) - 1); }
    if (bu) { fb0 = __shfl_sync(0xffffffffu, gb, __ffs(bu) - 1); fu0 = __shfl_sync(0xffffffffu, gu, __ffs(bu) - 1); }
  } else {
    int64_t T = 0, U = 0;
    for (int b = lane; b < p.batch; b += 32) {
      const int64_t raw = p.context_lens[b];
      clamped |= raw < 0 || raw > p.cap;
      const int64_t ce = ctx_eff(raw, p.cap);
      T += req_tiles(ce);
      U += req_units<NEXT_N>(ce, p.width);
      if (p.k > 0)
        for (int j = 0; j < NEXT_N; ++j) with_tiles += row_context(raw, NEXT_N, j, p.cap) > p.k ? 1 : 0;
    }
    T = warp_sum64(T);
    U = warp_sum64(U);
    u_all = U > 4 * T ? U : -1;
    tb = split_begin(T, G, cta); te = split_begin(T, G, cta + 1);
    ub = split_begin(U, G, cta); ue = split_begin(U, G, cta + 1);
    int64_t ct = 0, cu = 0;
    bool got_t = tb >= te, got_u = ub >= ue;
    for (int base = 0; base < p.batch && !(got_t && got_u); base += 32) {
      const int b = base + lane;
      const int64_t ce = b < p.batch ? ctx_eff(p.context_lens[b], p.cap) : 0;
      const int64_t x = b < p.batch ? req_tiles(ce) : 0;
      const int64_t y = b < p.batch ? req_units<NEXT_N>(ce, p.width) : 0;
      const int64_t xi = warp_incl_scan64(x, lane), yi = warp_incl_scan64(y, lane);
      const bool ht = !got_t && x > 0 && ct + xi - x <= tb && tb < ct + xi;
      const bool hu = !got_u && y > 0 && cu + yi - y <= ub && ub < cu + yi;
      const uint32_t bt = __ballot_sync(0xffffffffu, ht), bu = __ballot_sync(0xffffffffu, hu);
      if (bt) {
        const int src = __ffs(bt) - 1;
        b0 = __shfl_sync(0xffffffffu, b, src);
        t0 = (int)__shfl_sync(0xffffffffu, tb - (ct + xi - x), src);
        got_t = true;
      }
      if (bu) {
        const int src = __ffs(bu) - 1;
        fb0 = __shfl_sync(0xffffffffu, b, src);
        fu0 = (int)__shfl_sync(0xffffffffu, ub - (cu + yi - y), src);
        got_u = true;
      }
      ct += __shfl_sync(0xffffffffu, xi, 31);
      cu += __shfl_sync(0xffffffffu, yi, 31);
    }
  }
  if (blockIdx.x == 0 && __any_sync(0xffffffffu, clamped) && lane == 0) raise_status(p.status, SAI_STATUS_CTX_CLAMPED);
  with_tiles = warp_sum64(with_tiles);
  if (lane == 0) {
    part->b0 = b0; part->t0 = t0; part->n_tiles = (int)(te - tb);
    part->fb0 = fb0; part->fu0 = fu0; part->n_units = (int)(ue - ub);
    part->n_sel = (int)with_tiles;
    part->u_total = u_all < (int64_t(1) << 30) ? (int)u_all : -1;
  }
}

// L2 prefetch of the block-table entries the launch may read (each row's
// first min(stride, ceil(cap / P)) entries), split evenly over the CTAs: run
// while the partition reads the context lengths, it turns the producers'
// first page-id reads into L2 hits.  A prefetch only loads lines into L2, so
// it may run before the previous kernel in the stream has completed.
__device__ void prefetch_block_table(const TcParams& p, int lane) {
  const int64_t used = min(p.bt_stride, (p.cap + p.page_size - 1) / p.page_size);
  const int64_t lines_per_row = (used * 4 + 127) / 128 + 1;      // + 1: a row need not start on a line
  const int64_t total = (int64_t)p.batch * lines_per_row;
  const int64_t per = (total + gridDim.x - 1) / gridDim.x;
  const int64_t x0 = (int64_t)blockIdx.x * per, x1 = min(total, x0 + per);
  for (int64_t x = x0 + lane; x < x1; x += 32) {
    const int64_t r = x / lines_per_row, l = x - r * lines_per_row;
    const char* row = reinterpret_cast<const char*>(p.block_table + r * p.bt_stride);
    if (l * 128 < used * 4) ptx::prefetch_l2(row + l * 128);
  }
}

// Context lengths of requests [base, base + 32) held one per lane, so a warp
// walking requests in order reads them from registers.
struct CtxCache {
  const int32_t* staged = nullptr;                 // shared-memory copy, if the batch has one
  int base = -1000000;
  int64_t mine = 0;
  __device__ __forceinline__ int64_t get(const TcParams& p, int b, int lane) {
    if (b < base || b >= base + 32) {              // warp-uniform
      base = b;
      mine = (b + lane < p.batch) ? (int64_t)(staged ? staged[b + lane] : p.context_lens[b + lane]) : 0;
    }
    return __shfl_sync(0xffffffffu, mine, b - base);
  }
};

// Position (request b, tile t) in the walk over a CTA's tiles, with the
// request's raw and clamped context and its tile count.
struct Cursor {
  int b = 0, t = 0;
  int64_t raw = 0, ce = 0, nt = 0;
  __device__ __forceinline__ void load(const TcParams& p, CtxCache& cc, int lane) {
    raw = cc.get(p, b, lane);
    ce = ctx_eff(raw, p.cap);
    nt = req_tiles(ce);
  }
  __device__ __forceinline__ void start(const TcParams& p, int b0, int t0, CtxCache& cc, int lane) {
    b = b0;
    t = t0;
    load(p, cc, lane);
  }
  // Next tile; skips requests without tiles (the partition guarantees one
  // follows).  Returns 1 when the tile belongs to a new request.
  __device__ __forceinline__ int advance(const TcParams& p, CtxCache& cc, int lane) {
    if (++t < nt) return 0;
    t = 0;
    do {
      ++b;
      load(p, cc, lane);
    } while (nt == 0 && b + 1 < p.batch);
    return 1;
  }
};

// The same walk for one thread (no warp shuffles), counting the requests
// entered: q is the Q load index of the current tile's request.
struct ScalarCursor {
  int b = 0, t = 0, q = 0;
  int64_t nt = 0;
  const int32_t* staged = nullptr;
  __device__ __forceinline__ void load(const TcParams& p) {
    nt = req_tiles(ctx_eff(staged ? staged[b] : p.context_lens[b], p.cap));
  }
  __device__ __forceinline__ void start(const TcParams& p, int b0, int t0) {
    b = b0;
    t = t0;
    q = 0;
    load(p);
  }
  __device__ __forceinline__ void advance(const TcParams& p) {
    if (++t < nt) return;
    t = 0;
    do {
      ++b;
      load(p);
    } while (nt == 0 && b + 1 < p.batch);
    ++q;
  }
};

// ---- fused top-k: rows go to a ready queue, every CTA selects from it ---------
// Each CTA adds, per request it touched, the number of that request's tiles it
// processed to the request's counter once its logits are stored and fenced;
// the CTA whose addition completes the request's tile count resets the
// counter to 0 and publishes the request: its rows longer than k go onto a
// queue of ready rows, its shorter ones (indices 0 .. n - 1, then -1) it
// writes itself.  Every CTA, once its tiles are done, takes rows from the
// queue (one atomic on its head per row, the next taken before the current
// row is selected) and selects them, reading the logits through L2; so the
// selection is spread over the whole grid and starts as soon as a request is
// complete.  The queue's length (the launch's rows longer than k) comes from
// the partition.  A queue entry not yet written (its request still has tiles
// in flight on another CTA) is waited for, with a bounded wait; the grid is
// one CTA per SM, so every CTA is resident.  The last CTA to finish resets
// the queue's head, tail and done count and the fill counter; the workspace
// is all zero again.  Requests without tiles get their -1 rows from CTA
// (b mod grid).  Where the -inf fill outweighs the tiles (more than four
// fill units per tile) the two epilogue warpgroups select (NT = 256) while
// the other warps keep writing the fill; elsewhere all warps select
// (NT = 384).  Named barrier 1 joins the selecting threads; the drained
// K-stage ring and Q slots hold the selection's histograms and staged keys.
template <int NT>
struct TailBar {
  __device__ __forceinline__ void operator()() const { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }
};

__device__ __forceinline__ bool fill_heavy(const Part& pt) { return pt.n_units > 4 * pt.n_tiles; }

template <int NEXT_N, int NT>
__device__ void fused_topk(const TcParams& p, const Part& pt, uint8_t* ring, int ring_bytes, int etid,
                           const int32_t* staged, const volatile int* abort_flag) {
  auto ctx_of = [&](int b) -> int64_t { return staged ? staged[b] : p.context_lens[b]; };
  static_assert(NT == 256 || NT == 384, "the epilogue warpgroups, or every warp of the CTA");
  const TailBar<NT> ebar;
  uint32_t* hist = reinterpret_cast<uint32_t*>(ring);
  auto* sh = reinterpret_cast<SelectShared<NT>*>(ring + kSelectSmem);
  volatile int* word = reinterpret_cast<volatile int*>(ring + kSelectSmem + 512);   // [0] row, [1] done count
  int* done_list = reinterpret_cast<int*>(ring + kSelectSmem + 520);           // requests completed here
  constexpr int kDoneMax = (1024 - 520) / 4;
  uint32_t* key_base = reinterpret_cast<uint32_t*>(ring + kSelectSmem + 1024);
  const int key_cap = (ring_bytes - (int)kSelectSmem - 1024) / 4 - 3;
  int32_t* counter = p.req_counter;
  int32_t* queue = p.req_counter + p.batch;
  int32_t* qctl = p.req_counter + 5 * (int64_t)p.batch;     // head, tail, done
  const int k = p.k;
  const int lane = etid & 31;
  auto write_short = [&](int64_t row, int64_t n, int tid, int nthreads) {
    int32_t* out = p.indices + row * p.idx_stride;          // 64-bit row base
    for (int i = tid; i < k; i += nthreads) out[i] = i < n ? i : -1;
  };
  __threadfence();                                   // this thread's logits are visible device-wide
  ebar();
  // Publish: the first warp walks this CTA's tiles 32 requests at a time
  // (lane l takes request b + l).  Of each request it completes, the rows
  // longer than k go onto the queue; the others (indices 0 .. n - 1, then
  // -1) are written here, by the whole group from a list of the completed
  // requests (by the warp itself once the list is full).
  int h_next = -1;                                   // the next queue entry this CTA takes (thread 0)
  if (etid < 32) {
    int n_done = 0;
    if (*abort_flag == 0) {
      int b = pt.b0, left = pt.n_tiles;
      int64_t t = pt.t0;
      while (left > 0) {
        const int bb = b + lane;
        const int64_t raw = bb < p.batch ? ctx_of(bb) : 0;
        const int64_t nt = bb < p.batch ? req_tiles(ctx_eff(raw, p.cap)) : 0;
        const int64_t avail = lane == 0 ? nt - t : nt;
        const int64_t incl = warp_incl_scan64(avail, lane);
        const int64_t m = min(avail, max((int64_t)0, (int64_t)left - (incl - avail)));
        bool done = false;
        if (m > 0) {
          const int old = atomicAdd(&counter[bb], (int)m);
          done = (int64_t)old + m == nt;
          if (done) counter[bb] = 0;                 // the last contributor restores zero
        }
        int n_long = 0;
        if (done)
          for (int j = 0; j < NEXT_N; ++j) n_long += row_context(raw, NEXT_N, j, p.cap) > k ? 1 : 0;
        const uint32_t db = __ballot_sync(0xffffffffu, done);
        const int long_incl = __reduce_add_sync(0xffffffffu, n_long);
        int base = 0;
        if (lane == 0 && long_incl > 0) base = atomicAdd(&qctl[1], long_incl);
        base = __shfl_sync(0xffffffffu, base, 0);
        // Every contributor fenced its logits before its addition, which a
        // completing lane's addition observed: fence, then publish the rows.
        if (done) __threadfence();
        // Each completing lane's queue position: the long rows of the lanes below it.
        int excl = n_long;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, excl, o);
          if (lane >= o) excl += y;
        }
        excl -= n_long;
        if (done) {
          int pos = base + excl;
          for (int j = 0; j < NEXT_N; ++j)
            if (row_context(raw, NEXT_N, j, p.cap) > k) atomicExch(&queue[pos++], bb * NEXT_N + j + 1);
        }
        // The short rows: through the list, or by this warp once it is full.
        const int rank = __popc(db & ((1u << lane) - 1u));
        const bool listed = done && n_done + rank < kDoneMax;
        if (listed) done_list[n_done + rank] = bb;
        if (done && !listed)
          for (int j = 0; j < NEXT_N; ++j) {
            const int64_t n = row_context(raw, NEXT_N, j, p.cap);
            if (n <= k) {
              int32_t* out = p.indices + ((int64_t)bb * NEXT_N + j) * p.idx_stride;
              for (int i = 0; i < k; ++i) out[i] = i < n ? i : -1;
            }
          }
        n_done = min(kDoneMax, n_done + __popc(db));
        const int64_t total = __shfl_sync(0xffffffffu, incl, 31);
        if (total >= left) break;
        left -= (int)total;
        b += 32;
        t = 0;
      }
    }
    if (lane == 0) word[1] = n_done;
    if (etid == 0 && *abort_flag == 0 && pt.n_sel > 0) h_next = atomicAdd(&qctl[0], 1);
  }
  ebar();
  {
    const int n_done = word[1];
    for (int x = 0; x < n_done; ++x) {
      const int bb = done_list[x];
      const int64_t raw = ctx_of(bb);
      for (int j = 0; j < NEXT_N; ++j) {
        const int64_t n = row_context(raw, NEXT_N, j, p.cap);
        if (n <= k) write_short((int64_t)bb * NEXT_N + j, n, etid, NT);
      }
    }
  }
  // Select: one row at a time from the queue, until past its last long row.
  // Thread 0 takes the entry after the current one before the group selects
  // the current row, so the atomic's round trip overlaps the work.
  for (;;) {
    if (etid == 0) {
      int row = -1;
      const int h = *abort_flag ? pt.n_sel : h_next;
      if (h >= 0 && h < pt.n_sel) {
        const long long t0 = clock64();
        int v;
        while ((v = atomicAdd(&queue[h], 0)) == 0) {
          if (*abort_flag || clock64() - t0 > kWaitBudget) {
            raise_status(p.status, SAI_STATUS_TIMEOUT);
            break;
          }
          __nanosleep(256);
        }
        if (v != 0) {
          queue[h] = 0;
          row = v - 1;
          __threadfence();                           // the row's logits, from every CTA that wrote them
          h_next = atomicAdd(&qctl[0], 1);
        }
      }
      word[0] = row;
    }
    ebar();
    const int row = word[0];
    if (row < 0) break;
    const int bb = row / NEXT_N, j = row - bb * NEXT_N;
    const int64_t n = row_context(ctx_of(bb), NEXT_N, j, p.cap);
    int32_t* out = p.indices + (int64_t)row * p.idx_stride;  // 64-bit row base
    const float* lrow = p.logits + (int64_t)row * p.stride;
    if (n <= key_cap) {
      topk_row_staged<NT>(lrow, (int)n, k, out, *sh, hist, key_base, etid, ebar);
    } else {
      topk_row_stream<NT>(lrow, n, k, out, *sh, hist, etid, ebar);
    }
    ebar();                                          // word[0] read by all before it is rewritten
  }
  for (int bb = blockIdx.x; bb < p.batch; bb += gridDim.x) {
    if (req_tiles(ctx_eff(ctx_of(bb), p.cap)) != 0) continue;
    for (int j = 0; j < NEXT_N; ++j) {
      int32_t* out = p.indices + ((int64_t)bb * NEXT_N + j) * p.idx_stride;
      for (int i = etid; i < k; i += NT) out[i] = -1;
    }
  }
}

// -inf fill of the columns past each request's last tile, in units of
// (row, 4096 columns) taken from a counter, so warps with time to spare
// (producers waiting for ring space, any warp once its role is done) share
// it.  Each warp keeps its own position in the walk over the requests: the
// units it takes only move forward.  By default each CTA fills its own
// share of the units from a shared-memory counter.  The fused launch, whose
// CTAs spend unequal times selecting rows, shares every unit of the launch
// through one counter in global memory instead (`whole` set), so the CTAs
// that select less fill more; a warp that fills until its role is done
// takes kClaim units at a time there (`batch`), a warp that fills only
// while it waits takes one, so that it never drops units it has claimed.
constexpr int kClaim = 4;

template <int NEXT_N>
struct Filler {
  const TcParams* p;
  int* next;
  int n_units, lane, b, step, claim, claim_end;
  CtxCache cc;
  int64_t u_in, ucur, fs, chunks;

  __device__ __forceinline__ void init(const TcParams& pp, const Part& pt, int* counter, const int32_t* staged,
                                       int ln, bool whole = false, bool batch = false) {
    p = &pp;
    next = counter;
    n_units = whole ? pt.u_total : pt.n_units;
    step = whole && batch ? kClaim : 1;
    claim = claim_end = 0;
    lane = ln;
    cc.staged = staged;
    b = whole ? 0 : pt.fb0;
    u_in = whole ? 0 : pt.fu0;
    ucur = 0;
    const int64_t ce = n_units > 0 ? ctx_eff(cc.get(pp, b, lane), pp.cap) : 0;
    fs = min(pp.width, req_tiles(ce) * kTile);
    chunks = (pp.width - fs + kFillCols - 1) / kFillCols;
  }

  // Takes and writes one unit; false when none is left.  Warp-uniform.
  __device__ bool unit() {
    if (claim >= claim_end) {
      int u = 0;
      if (lane == 0) u = atomicAdd(next, step);
      u = __shfl_sync(0xffffffffu, u, 0);
      if (u >= n_units) return false;
      claim = u;
      claim_end = min(n_units, u + step);
    }
    const int u = claim++;
    u_in += u - ucur;
    ucur = u;
    while (u_in >= NEXT_N * chunks && b < p->batch) {   // move to the request holding unit u
      u_in -= NEXT_N * chunks;
      ++b;
      if (b >= p->batch) break;
      const int64_t ce = ctx_eff(cc.get(*p, b, lane), p->cap);
      fs = min(p->width, req_tiles(ce) * kTile);
      chunks = (p->width - fs + kFillCols - 1) / kFillCols;
    }
    if (b >= p->batch) return false;                     // never past the last row
    const int j = (int)(u_in / chunks);
    const int64_t c0 = fs + (u_in % chunks) * kFillCols;
    const int64_t c1 = min(p->width, c0 + kFillCols);
    float* row = p->logits + ((int64_t)b * NEXT_N + j) * p->stride;    // 64-bit row base
    int64_t head = (int64_t)(((16 - (reinterpret_cast<uintptr_t>(row + c0) & 15)) & 15) >> 2);
    head = min(head, c1 - c0);
    if (lane < head) row[c0 + lane] = -INFINITY;
    const int64_t v0 = c0 + head;
    const int64_t nv = (c1 - v0) >> 2;
    float4* vrow = reinterpret_cast<float4*>(row + v0);
    const float4 ninf = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    for (int64_t x = lane; x < nv; x += 32) vrow[x] = ninf;
    const int64_t tail0 = v0 + nv * 4;
    if (tail0 + lane < c1) row[tail0 + lane] = -INFINITY;
    return true;
  }
};

template <int NEXT_N, int H, bool FUSED, bool IL, bool DUAL_OK>
__global__ void __launch_bounds__(kThreadsTc, 1)
logits_tc_kernel(const __grid_constant__ CUtensorMap tmap_kv, const __grid_constant__ CUtensorMap tmap_q,
                 const TcParams p) {
  using K = Cfg<NEXT_N, H, IL, DUAL_OK>;
  constexpr int NP = K::PRODUCERS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int stages = K::STAGES;
  const SmemLayout L = smem_layout(stages, K::Q_BYTES, K::ACC, IL, K::W_BYTES);
  const uint32_t s_base = ptx::smem_addr(smem);
  const uint32_t s_k = s_base + L.k, s_q = s_base + L.q;
  float* scales = reinterpret_cast<float*>(smem + L.sc);
  int4* meta = reinterpret_cast<int4*>(smem + L.meta);
  const uint32_t bar = s_base + L.bar;
  // barrier addresses
  auto full = [&](int s) { return bar + 8u * s; };
  auto kempty = [&](int s) { return bar + 8u * (stages + s); };
  auto qfull = [&](int q) { return bar + 8u * (2 * stages + q); };
  auto qempty = [&](int q) { return bar + 8u * (2 * stages + 2 + q); };
  auto tfull = [&](int a) { return bar + 8u * (2 * stages + 4 + a); };
  auto tempty = [&](int a) { return bar + 8u * (2 * stages + 4 + K::ACC + a); };
  const uint32_t drain = bar + 8u * (2 * stages + 4 + 2 * K::ACC);       // [0] MMA warp, [1] the second one
  auto stgbar = [&](int s) { return bar + 8u * (2 * stages + 4 + 2 * K::ACC + 2 + s); };   // IL staging
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  int* fill_next = reinterpret_cast<int*>(smem + L.misc + 8);      // next -inf fill unit to take
  Part* part = reinterpret_cast<Part*>(smem + L.misc + 16);
  int32_t* ctx_s = reinterpret_cast<int32_t*>(smem + L.ctx);
  const int32_t* staged = p.batch <= kCtxSmem ? ctx_s : nullptr;   // written by the partition

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- set-up --------------------------------------------------------------
  if (warp == 0) {
    if (lane == 0) {
      if constexpr (!IL) ptx::prefetch_tensormap(&tmap_kv);
      ptx::prefetch_tensormap(&tmap_q);
    }
    // The context lengths' lines are pulled into L2 first (a prefetch returns
    // nothing, so it may run while the previous kernel still works); then,
    // since inputs may come from that kernel and the logits buffer may still
    // be read by it, wait for it before touching either.
    for (int64_t x = (int64_t)lane * 32; x < p.batch; x += 32 * 32) ptx::prefetch_l2(p.context_lens + x);
    ptx::wait_prerequisites();
    compute_partition<NEXT_N>(p, part, ctx_s, lane);
  } else if (warp == 1) {
    prefetch_block_table(p, lane);
  } else if (warp == kMmaWarp) {
    if (lane == 0) {
      for (int s = 0; s < stages; ++s) {
        ptx::mbar_init(full(s), 1);
        ptx::mbar_init(kempty(s), 4 * K::C);   // every epilogue warp of the tile's jobs
      }
      for (int q = 0; q < 2; ++q) {
        ptx::mbar_init(qfull(q), 1);
        ptx::mbar_init(qempty(q), K::DUAL ? 2 : 1);    // each MMA warp commits every Q load's release
      }
      for (int a = 0; a < K::ACC; ++a) {
        ptx::mbar_init(tfull(a), 1);
        ptx::mbar_init(tempty(a), 4);
      }
      ptx::mbar_init(drain, 1);
      ptx::mbar_init(drain + 8u, 1);
      if constexpr (IL)
        for (int s = 0; s < stages; ++s) ptx::mbar_init(stgbar(s), 1);
      *abort_flag = 0;
      *fill_next = 0;
      ptx::fence_barrier_init();
    }
    __syncwarp();
    ptx::tmem_alloc(ptx::smem_addr(tmem_holder), K::TMEM_COLS);
  }
  ptx::wait_prerequisites();
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  const Part pt = *part;
  // A fused launch whose fill outweighs its tiles four times over fills from
  // one counter for the whole grid (the word after the ready queue's head,
  // tail and done count); the choice is the same for every CTA.  Elsewhere
  // the producers' fill while they wait would pay a global atomic per unit.
  const bool whole_fill = FUSED && pt.u_total >= 0;
  int* fill_ctr = whole_fill ? p.req_counter + 5 * (int64_t)p.batch + 3 : fill_next;
  // The next kernel in the stream (top-k) may be scheduled now; it still
  // waits for this grid to complete before it reads the logits.
  ptx::launch_dependents();

  auto fail = [&]() {
    *abort_flag = 1;
    raise_status(p.status, SAI_STATUS_TIMEOUT);
  };

  if (warp < NP) {
    // ---- producers: warp pw issues tiles pw, pw + NP, ... ------------------------
    // A tile's copies go out as two warp instructions: lane l loads the values
    // of page l of the tile (a 128-byte swizzled tensor box), then its scales
    // (a contiguous bulk copy).
    const int pw = warp;
    const uint64_t pol_k = ptx::policy_evict_first();
    const uint64_t pol_q = ptx::policy_evict_last();
    const int P = p.page_size;
    const int ppt = P >= kTile ? 1 : kTile / P;          // pages per tile (<= 16)
    const int log2p = __ffs(P) - 1;                      // P is a power of two
    const int tok_per_box = P >= kTile ? kTile : P;
    const uint32_t box_bytes = (uint32_t)tok_per_box * kTokenBytes;
    const int pl = lane;                                 // page of the tile this lane serves
    const int own = pt.n_tiles > pw ? (pt.n_tiles - pw + NP - 1) / NP : 0;
    // Two cursors over this CTA's tiles: `cur` at this warp's tile being
    // issued, `la` kLookahead own tiles ahead, whose page ids are copied into a
    // shared-memory ring with cp.async so their latency overlaps the pipeline.
    // q_seq counts the requests entered before `cur`'s (its Q slot is q_seq & 1).
    // Warp 0 alone loads Q, for every request in order as its cursor crosses
    // request starts (its own tiles' and the other warps'): waiting on a Q
    // slot's release in sequence keeps each parity wait unambiguous.
    const bool q_here = pw == 0;
    CtxCache cc, cc_la;
    cc.staged = cc_la.staged = staged;
    Cursor cur, la;
    int q_seq = 0, ci = 0;                               // ci: tile index of `cur`
    bool qok = true;
    auto issue_q = [&](int b, int seq) {
      const int qs = seq & 1;
      if (!ptx::mbar_wait_warp(qempty(qs), ((uint32_t)(seq >> 1) & 1u) ^ 1u, abort_flag, kWaitBudget)) {
        qok = false;
        if (lane == 0) fail();
        return;
      }
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(qfull(qs), K::Q_BYTES);
        for (int x = 0; x < K::N / K::QBOX; ++x)
          ptx::tma_load_2d(s_q + qs * K::Q_BYTES + x * K::QBOX * kHeadDim, &tmap_q, 0, b * K::N + x * K::QBOX,
                           qfull(qs), pol_q);
      }
    };
    // Advance `cur` one tile; warp 0 loads Q for a request it enters.
    auto step = [&]() {
      const int entered = cur.advance(p, cc, lane);
      ++ci;
      q_seq += entered;
      if (entered && q_here && qok) issue_q(cur.b, q_seq);
    };
    if (own > 0) {
      cur.start(p, pt.b0, pt.t0, cc, lane);
      if (q_here) issue_q(cur.b, 0);
      for (int x = 0; x < pw; ++x) step();
      la = cur;
    }
    const uint32_t ring = s_base + L.ids + (uint32_t)(pw * kLookahead * 32 * 4);
    const int32_t* ring_ptr = reinterpret_cast<const int32_t*>(smem + L.ids) + pw * kLookahead * 32;
    int la_j = 0;
    auto issue_ids = [&]() {
      if (la_j < own) {
        const int64_t tok0 = (int64_t)la.t * kTile + (P >= kTile ? 0 : (int64_t)lane * P);
        const bool v = lane < ppt && tok0 < la.ce;
        const int32_t* src = p.block_table + (v ? (int64_t)la.b * p.bt_stride + (tok0 >> log2p) : 0);
        ptx::cp_async_4(ring + (uint32_t)(((la_j % kLookahead) * 32 + lane) * 4), src, v ? 4u : 0u);
        if (la_j + 1 < own)
          for (int x = 0; x < NP; ++x) la.advance(p, cc_la, lane);
        ++la_j;
      }
      ptx::cp_async_commit();
    };
    // Interleaved tiles: once a tile's pages have landed in its stage as
    // stored, the warp rewrites them in place (values into the swizzled
    // K-major layout, scales into token order), then marks the stage full.
    // Lane (c, r0) moves 16-byte value chunk c of tokens r0, r0 + 4, ...:
    // the 132-byte token pitch leaves the source words 4-byte aligned and
    // puts the 32 lanes' words in 32 distinct banks.
    auto finish_il = [&](int fs, uint32_t fph, bool fbad) -> bool {
      if (!ptx::mbar_wait_warp(stgbar(fs), fph, abort_flag, kWaitBudget)) {
        if (lane == 0) fail();
        const int zero_flag = 0;
        ptx::mbar_wait_warp(stgbar(fs), fph, &zero_flag, 1LL << 26);    // the copies land before exit
        return false;
      }
      // Token r's rewritten row [128 r, 128 r + 128) overlaps the stored
      // bytes of tokens <= r only, so the warp rewrites 16 tokens at a time
      // in increasing order, reading all 16 (values and scales) before
      // writing any.
      uint8_t* st = smem + L.k + fs * K::STAGE_BYTES;
      const int c = lane & 7;
#pragma unroll 1
      for (int m = 0; m < kTile / 16; ++m) {
        uint4 v[4];
        float sv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = (lane >> 3) + 4 * u + 16 * m;
          const uint32_t* w = reinterpret_cast<const uint32_t*>(st + r * kTokenBytes + c * 16);
          v[u] = make_uint4(w[0], w[1], w[2], w[3]);
          sv[u] = c == 0 ? *reinterpret_cast<const float*>(st + r * kTokenBytes + kHeadDim) : 0.f;
        }
        __syncwarp();
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = (lane >> 3) + 4 * u + 16 * m;
          *reinterpret_cast<uint4*>(st + r * kHeadDim + ((c ^ (r & 7)) << 4)) = v[u];
          if (c == 0) scales[fs * kTile + r] = sv[u];
        }
      }
      __syncwarp();
      if (fbad)
        for (int x = 0; x < tok_per_box; ++x) scales[fs * kTile + (P >= kTile ? 0 : pl * P) + x] = __int_as_float(0x7fc00000);
      ptx::fence_proxy_async_smem();                   // generic stores, then the MMA's async-proxy reads
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(full(fs));
      return true;
    };
    // Warps other than 0 issue their next tile's copies before rewriting the
    // current tile, so two of their tiles are in flight.  Holding tile i
    // while waiting for the release of tile i + NP - stages is deadlock-free
    // when stages > NP: that release needs only earlier tiles.  Warp 0 does
    // not hold: its Q loads wait for releases that may need its own tile.
    const bool hold = IL && stages > NP && pw != 0;
    int held_s = -1;                                   // stage of the held tile, -1 if none
    uint32_t held_ph = 0;
    bool held_bad = false;
    // While the ring is full the warp writes -inf fill units; once none is
    // left it waits (bounded).  Only where the fill outweighs the tiles: a
    // unit (16 KB of stores) would otherwise delay the next tile's copies on
    // a short, latency-bound launch.
    Filler<NEXT_N> filler;
    filler.init(p, pt, fill_ctr, staged, lane, whole_fill);
    bool fill_left = pt.n_units > pt.n_tiles;
    auto wait_filling = [&](uint32_t b, uint32_t parity) -> bool {
      while (fill_left && !__all_sync(0xffffffffu, ptx::mbar_test(b, parity))) {
        if (*abort_flag) return false;
        fill_left = filler.unit();
      }
      return ptx::mbar_wait_warp(b, parity, abort_flag, kWaitBudget);
    };
    // Only the first tile's page ids go out before its K copies; the rest of
    // the lookahead follows them, off the first tile's latency chain.
    issue_ids();
    bool ok = true;
    int j = 0;
    for (; j < own && ok; ++j) {
      const int i = pw + j * NP;
      const int s = i % stages;
      const uint32_t ph = (uint32_t)(i / stages) & 1u;
      const bool is_new = (i == 0) || (cur.t == 0);
      const bool is_last = (cur.t == cur.nt - 1) || (i == pt.n_tiles - 1);
      if (!qok) { ok = false; break; }
      if (!wait_filling(kempty(s), ph ^ 1u)) { ok = false; if (lane == 0) fail(); break; }
      if (j == 0) ptx::cp_async_wait<0>();                    // page ids of this tile have landed
      else ptx::cp_async_wait<kLookahead - 1>();
      const int64_t tok0 = (int64_t)cur.t * kTile + (P >= kTile ? 0 : (int64_t)pl * P);
      const bool need = pl < ppt && tok0 < cur.ce;
      const int64_t pg = (int64_t)ring_ptr[(j % kLookahead) * 32 + pl];   // widened before use
      const bool bad = need && (pg < 0 || pg >= p.num_pages);
      const bool load = need && !bad;
      const uint32_t nload = __popc(__ballot_sync(0xffffffffu, load));
      if constexpr (IL) {
        // The tile's pages as stored (P * 132 contiguous bytes, 16-byte
        // aligned since P is a multiple of 4) come into the stage with bulk
        // copies, one lane per page; finish_il rewrites them in place.
        if (bad) raise_status(p.status, SAI_STATUS_BAD_PAGE);
        if (lane == 0) {
          meta[s] = make_int4(cur.b, cur.t, (int)max((int64_t)INT32_MIN, min((int64_t)INT32_MAX, cur.raw)),
                              (is_new ? kFlagNew : 0) | (is_last ? kFlagLast : 0) | (q_seq << 8));
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_expect_tx(stgbar(s), nload * box_bytes + K::W_BYTES);
        __syncwarp();
        if (load) {
          const int y = P > kTile ? (cur.t & 1) * kTile : 0;                     // half of a 256-token page
          const uint8_t* src = p.kv + pg * (int64_t)P * kTokenBytes + (int64_t)y * kTokenBytes;
          const uint32_t dst = s_k + s * K::STAGE_BYTES + (P >= kTile ? 0 : pl * box_bytes);
          ptx::bulk_load(dst, src, box_bytes, stgbar(s), pol_k);
        }
        if (K::STAGE_W && lane == 31)
          ptx::bulk_load(s_base + L.wst + s * K::W_BYTES, p.weights + (int64_t)cur.b * NEXT_N * H, K::W_BYTES,
                         stgbar(s), pol_q);
        if (hold) {                                    // rewrite the previous tile while this one lands
          const int prev_s = held_s;
          const uint32_t prev_ph = held_ph;
          const bool prev_bad = held_bad;
          held_s = s;                                  // (so an exit below still drains its copies)
          held_ph = ph;
          held_bad = bad;
          if (prev_s >= 0 && !finish_il(prev_s, prev_ph, prev_bad)) { ok = false; break; }
        } else if (!finish_il(s, ph, bad)) {
          ok = false;
          break;
        }
      } else {
        if (bad) {
          for (int x = 0; x < tok_per_box; ++x) scales[s * kTile + (P >= kTile ? 0 : pl * P) + x] = __int_as_float(0x7fc00000);
          ptx::fence_proxy_async_smem();
          raise_status(p.status, SAI_STATUS_BAD_PAGE);
        }
        if (lane == 0) {
          meta[s] = make_int4(cur.b, cur.t, (int)max((int64_t)INT32_MIN, min((int64_t)INT32_MAX, cur.raw)),
                              (is_new ? kFlagNew : 0) | (is_last ? kFlagLast : 0) | (q_seq << 8));
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive_expect_tx(full(s), nload * box_bytes + K::W_BYTES);
        __syncwarp();
        if (K::STAGE_W && lane == 31)
          ptx::bulk_load(s_base + L.wst + s * K::W_BYTES, p.weights + (int64_t)cur.b * NEXT_N * H, K::W_BYTES,
                         full(s), pol_q);
        if (load) {
          const int y = P > kTile ? (cur.t & 1) * kTile : 0;                       // half of a 256-token page
          const uint32_t dst = s_k + s * kStageBytes + (P >= kTile ? 0 : pl * P * kHeadDim);
          ptx::tma_load_3d(dst, &tmap_kv, 0, y, (int)pg, full(s), pol_k);
          const uint8_t* src = p.kv + pg * (int64_t)P * kTokenBytes + (int64_t)P * kHeadDim + (int64_t)y * kScaleBytes;
          const uint32_t sdst = s_base + L.sc + s * kScaleSlot + (P >= kTile ? 0 : pl * P * kScaleBytes);
          ptx::bulk_load(sdst, src, (uint32_t)tok_per_box * kScaleBytes, full(s), pol_k);
        }
      }
      __syncwarp();
      if (j == 0)
        for (int k = 1; k < kLookahead; ++k) issue_ids();     // the lookahead, after the first copies
      issue_ids();                                             // refill the slot just read
      if (j + 1 < own)
        for (int x = 0; x < NP; ++x) step();
    }
    if (held_s >= 0) {
      if (ok) {
        ok = finish_il(held_s, held_ph, held_bad);
      } else {
        const int zero_flag = 0;
        ptx::mbar_wait_warp(stgbar(held_s), held_ph, &zero_flag, 1LL << 26);   // its copies land before exit
      }
    }
    // Warp 0 still loads Q for requests that start in the other warps' last tiles.
    if (q_here && ok && own > 0)
      while (ci + 1 < pt.n_tiles && qok) step();
    ok = ok && qok;
    ptx::cp_async_wait<0>();
    if (!IL && !ok) {
      // Let this warp's copies already issued land before the CTA exits (an
      // interleaved tile's copies have always landed before its stage is full).
      const int zero_flag = 0;
      const int i_end = pw + j * NP;
      for (int k2 = max(0, i_end - stages); k2 < i_end; ++k2)
        if (k2 % NP == pw)
          ptx::mbar_wait_warp(full(k2 % stages), (uint32_t)(k2 / stages) & 1u, &zero_flag, 1LL << 26);
    }
  } else if (warp == kMmaWarp || (K::DUAL && warp == 2)) {
    // ---- MMA issuer(s) ----------------------------------------------------------
    // One warp issues every tile; with DUAL, warp kMmaWarp the even tiles and
    // warp 2 the odd ones.  Tile i's job goes to accumulator i % ACC, which
    // the epilogue releases in tile order, so the two warps' accumulators
    // are disjoint.  Q loads (one per request, in order, slot q & 1, issued
    // by producer warp 0, which waits for each slot's release in order): the
    // single warp waits for a request's Q at its first tile and releases it
    // after its last.  Two warps each wait for every Q load in order (also
    // those of requests whose tiles all went to the other warp), and each
    // walks the tiles itself (a scalar cursor), so that right after its last
    // tile of a request, before its next tile has landed, it commits the
    // release of every load before its next tile's request; a Q slot's
    // release needs both commits.  (Releasing only on reading the next
    // tile's request can deadlock: producer warp 0 may be waiting for that
    // release before it issues that very tile.)  A warp waits for load q only
    // after load q - 2 has landed and commits load q's release only after
    // waiting for it, so each parity wait and each arrival is on the phase
    // it means (simulated in the protocol tests).
    const int mw = warp == kMmaWarp ? 0 : 1;
    const uint32_t my_drain = drain + 8u * (uint32_t)mw;
    if (lane == 0) {
      int q_count = 0, acc_count = 0;                  // single warp
      int q_waited = 0, q_done = 0;                    // DUAL: Q loads waited for / released by this warp
      ScalarCursor sc;                                 // DUAL: at this warp's current tile
      sc.staged = staged;
      if (K::DUAL && pt.n_tiles > mw) {
        sc.start(p, pt.b0, pt.t0);
        if (mw == 1) sc.advance(p);
      }
      // DUAL: wait for load j (in order), then commit its release.
      auto wait_q = [&](int j) {
        return ptx::mbar_wait(qfull(j & 1), (uint32_t)(j >> 1) & 1u, abort_flag, kWaitBudget);
      };
      bool aborted = false;
      for (int i = K::DUAL ? mw : 0; i < pt.n_tiles; i += K::DUAL ? 2 : 1) {
        const int s = i % stages;
        int qs;
        if constexpr (K::DUAL) {
          const int qi = sc.q;                         // this tile's request's Q load
          bool qok_mma = true;
          for (; qok_mma && q_waited <= qi; ++q_waited) qok_mma = wait_q(q_waited);
          if (!qok_mma) { fail(); aborted = true; break; }
          qs = qi & 1;
        }
        // The stage and Q barriers are completed by TMA, not by tcgen05
        // operations, so no tcgen05 fence is needed after these waits.
        if (!ptx::mbar_wait(full(s), (uint32_t)(i / stages) & 1u, abort_flag, kWaitBudget)) { fail(); aborted = true; break; }
        const int4 m = meta[s];
        if constexpr (!K::DUAL) {
          qs = (m.w >> 8) & 1;
          if (m.w & kFlagNew) {
            if (!ptx::mbar_wait(qfull(qs), (uint32_t)(q_count >> 1) & 1u, abort_flag, kWaitBudget)) { fail(); aborted = true; break; }
            ++q_count;
          }
        }
        bool ok = true;
#pragma unroll 1
        for (int c = 0; c < K::C; ++c, ++acc_count) {
          const int job = K::DUAL ? i : acc_count;     // DUAL: one job per tile
          const int a = job % K::ACC;
          if (!ptx::mbar_wait(tempty(a), ((uint32_t)(job / K::ACC) & 1u) ^ 1u, abort_flag, kWaitBudget)) { ok = false; break; }
          ptx::tc_fence_after();
          const uint32_t d = tmem_base + (uint32_t)(a * K::NC);
          const uint64_t adesc = ptx::desc_kmajor_sw128(s_k + s * K::STAGE_BYTES);
          const uint64_t bdesc = ptx::desc_kmajor_sw128(s_q + qs * K::Q_BYTES + c * K::NC * kHeadDim);
#pragma unroll
          for (int k = 0; k < kHeadDim / 32; ++k)       // 32 bytes of K per instruction: +2 in 16-byte units
            ptx::mma_f8f6f4(d, adesc + 2 * k, bdesc + 2 * k, K::IDESC, k > 0 ? 1u : 0u);
          ptx::mma_commit(tfull(a));
        }
        if (!ok) { fail(); aborted = true; break; }
        if constexpr (K::DUAL) {
          // Release the loads before the next own tile's request (all those
          // waited for, past the last tile).
          int q_next = sc.q + 1;
          if (i + 2 < pt.n_tiles) {
            sc.advance(p);
            sc.advance(p);
            q_next = sc.q;
          }
          bool qok_mma = true;
          while (q_done < q_next) {
            if (q_done == q_waited) {
              qok_mma = wait_q(q_waited);
              if (!qok_mma) break;
              ++q_waited;
            }
            ptx::mma_commit(qempty(q_done & 1));
            ++q_done;
          }
          if (!qok_mma) { fail(); aborted = true; break; }
        } else if (m.w & kFlagLast) {
          // The stage is released by the epilogue warps of its jobs, each after
          // its accumulator is complete, hence after every MMA reading the stage.
          ptx::mma_commit(qempty(qs));
        }
      }
      // After an abort, the MMAs already issued complete before TMEM is freed
      // (otherwise the epilogue has already seen every one of them complete).
      if (aborted) {
        const int zero_flag = 0;
        ptx::mma_commit(my_drain);
        ptx::mbar_wait(my_drain, 0, &zero_flag, 1LL << 28);
      }
    }
    __syncwarp();
  } else if (warp >= kFirstEpiWarp) {   // (a producer warp left idle by Cfg::PRODUCERS goes on to the fill)
    // ---- epilogue ---------------------------------------------------------------
    const int ew = warp - kFirstEpiWarp;
    const int wg = ew >> 2;
    const int quarter = warp & 3;                 // TMEM lanes this warp may read
    const int token = quarter * 32 + lane;
    const uint32_t t_lane = tmem_base + ((uint32_t)(quarter * 32) << 16);
    const int jobs = pt.n_tiles * K::C;
    for (int a = wg; a < jobs; a += 2) {
      const int i = a / K::C, c = a % K::C, s = i % stages;
      const int acc = a % K::ACC;
      // The stage's data (and its meta) first: the first weights can then be
      // read while the MMA of this job completes.
      if (!ptx::mbar_wait_warp(full(s), (uint32_t)(i / stages) & 1u, abort_flag, kWaitBudget)) { if (lane == 0) fail(); break; }
      const int4 m = meta[s];
      const float sc = scales[s * kTile + token];
      // Weights of the job's rows: float4 f of row c * ROWS + jr is ldw(jr * H / 4 + f).
      const float4* w0 = reinterpret_cast<const float4*>(p.weights + ((int64_t)m.x * NEXT_N + c * K::ROWS) * H);
      const uint32_t ws0 = s_base + L.wst + s * K::W_BYTES + c * K::ROWS * H * 4;
      auto ldw = [&](int f) { return K::STAGE_W ? ptx::lds128(ws0 + 16u * f) : __ldg(w0 + f); };
      float4 wn[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) wn[x] = ldw(x);
      if (!ptx::mbar_wait_warp(tfull(acc), (uint32_t)(a / K::ACC) & 1u, abort_flag, kWaitBudget)) { if (lane == 0) fail(); break; }
      __syncwarp();
      // The stage is released here unless its staged weights are still to be
      // read by the sums below.
      if (!K::STAGE_W && lane == 0) ptx::mbar_arrive(kempty(s));
      ptx::tc_fence_after();
      float out[K::ROWS];
#pragma unroll
      for (int jr = 0; jr < K::ROWS; ++jr) {
        // Eight independent partial sums, held as four pairs updated by
        // paired fp32 FMAs: one dependent chain of H fused multiply-adds would
        // bound the epilogue by FMA latency.
        float2 part[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                          make_float2(0.f, 0.f)};
#pragma unroll
        for (int h0 = 0; h0 < H; h0 += 64) {         // two 32-column TMEM loads, one wait
          uint32_t v[64];
          ptx::tmem_ld_32(t_lane + (uint32_t)(acc * K::NC + jr * H + h0), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
          ptx::tmem_ld_32(t_lane + (uint32_t)(acc * K::NC + jr * H + h0 + 32), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
          float4 w4[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) w4[x] = (jr == 0 && h0 == 0 && x < 8) ? wn[x] : ldw(jr * (H / 4) + (h0 >> 2) + x);
          ptx::tmem_ld_wait();
          ptx::tmem_regs_ready(v);
#pragma unroll
          for (int x = 0; x < 16; ++x) {
            float2* q = part + 2 * (x & 1);
            const float2 r01 = make_float2(fmaxf(__uint_as_float(v[4 * x + 0]), 0.f),
                                           fmaxf(__uint_as_float(v[4 * x + 1]), 0.f));
            const float2 r23 = make_float2(fmaxf(__uint_as_float(v[4 * x + 2]), 0.f),
                                           fmaxf(__uint_as_float(v[4 * x + 3]), 0.f));
            q[0] = __ffma2_rn(make_float2(w4[x].x, w4[x].y), r01, q[0]);
            q[1] = __ffma2_rn(make_float2(w4[x].z, w4[x].w), r23, q[1]);
          }
        }
        out[jr] = ((part[0].x + part[0].y) + (part[1].x + part[1].y)) +
                  ((part[2].x + part[2].y) + (part[3].x + part[3].y));
      }
      ptx::tc_fence_before();
      __syncwarp();                                  // every lane's weight reads are done
      if (K::STAGE_W && lane == 0) ptx::mbar_arrive(kempty(s));
      if (lane == 0) ptx::mbar_arrive(tempty(acc));
      const int64_t col = (int64_t)m.y * kTile + token;
      if (col < p.width) {
#pragma unroll
        for (int jr = 0; jr < K::ROWS; ++jr) {
          const int j = c * K::ROWS + jr;
          const int64_t n_r = row_context(m.z, NEXT_N, j, p.cap);
          const int64_t r = (int64_t)m.x * NEXT_N + j;
          p.logits[r * p.stride + col] = col < n_r ? out[jr] * sc : -INFINITY;   // 64-bit row base
        }
      }
    }
  }

  // ---- -inf fill past each request's last tile --------------------------------
  // Every warp takes units from a shared counter once its role is done (the
  // producers also while they wait for ring space).  With the fused top-k the
  // epilogue warps select rows first and then join the fill.
  auto run_fill = [&]() {
    Filler<NEXT_N> f;
    f.init(p, pt, fill_ctr, staged, lane, whole_fill, true);
    while (f.unit()) {
    }
  };
  if constexpr (FUSED) {
    if (fill_heavy(pt)) {      // the epilogue warpgroups select rows while the other warps fill
      if (warp >= kFirstEpiWarp)
        fused_topk<NEXT_N, 256>(p, pt, smem + L.k, (int)(L.sc - L.k), (int)threadIdx.x - kFirstEpiWarp * 32,
                                staged, abort_flag);
    } else {                   // every warp selects, then fills
      fused_topk<NEXT_N, kThreadsTc>(p, pt, smem + L.k, (int)(L.sc - L.k), (int)threadIdx.x, staged, abort_flag);
    }
    run_fill();
  } else {
    run_fill();
  }

  // ---- tear-down ----------------------------------------------------------------
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, K::TMEM_COLS);
  }
  if constexpr (FUSED) {
    // The last CTA out resets the ready queue's head, tail and done count
    // and the fill counter: every CTA has taken its last row and unit by then.
    if (threadIdx.x == 0) {
      int32_t* qctl = p.req_counter + 5 * (int64_t)p.batch;
      __threadfence();
      if (atomicAdd(&qctl[2], 1) == (int)gridDim.x - 1) {
        qctl[0] = 0;
        qctl[1] = 0;
        qctl[2] = 0;
        qctl[3] = 0;
      }
    }
  }
}

// ---------------------------------------------------------------- host side
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// Encoded tensor maps keyed by (base, rows, box, rank): a decode loop calls
// with the same buffers every step and skips re-encoding.  The map depends
// only on the key, so a hit is always valid; entries are replaced round-robin.
struct TmapKey {
  const void* base;
  uint64_t extent;
  uint32_t box;
  uint32_t rank;
  bool operator==(const TmapKey& o) const {
    return base == o.base && extent == o.extent && box == o.box && rank == o.rank;
  }
};

constexpr int kTmapCache = 32;
struct TmapCache {
  std::mutex mu;
  TmapKey keys[kTmapCache] = {};
  CUtensorMap maps[kTmapCache];
  int dev[kTmapCache] = {};
  int next = 0;
};

TmapCache& tmap_cache() {
  static TmapCache c;
  return c;
}

bool tmap_lookup(const TmapKey& k, CUtensorMap* out) {
  int d = 0;
  cudaGetDevice(&d);
  TmapCache& c = tmap_cache();
  std::lock_guard<std::mutex> g(c.mu);
  for (int i = 0; i < kTmapCache; ++i)
    if (c.keys[i].base != nullptr && c.keys[i] == k && c.dev[i] == d) {
      *out = c.maps[i];
      return true;
    }
  return false;
}

void tmap_store(const TmapKey& k, const CUtensorMap& m) {
  int d = 0;
  cudaGetDevice(&d);
  TmapCache& c = tmap_cache();
  std::lock_guard<std::mutex> g(c.mu);
  c.keys[c.next] = k;
  c.maps[c.next] = m;
  c.dev[c.next] = d;
  c.next = (c.next + 1) % kTmapCache;
}

EncodeTiled encode_fn() {
  static EncodeTiled fn = nullptr;
  if (fn == nullptr) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  }
  return fn;
}

template <int NEXT_N, int H, bool FUSED, bool IL, bool DUAL_OK = false>
cudaError_t launch_tc(const LogitsArgs& a, cudaStream_t stream) {
  using K = Cfg<NEXT_N, H, IL, DUAL_OK>;
  EncodeTiled enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const int P = a.page_size;
  CUtensorMap tkv, tq;
  if (!IL) {   // the interleaved layout's pages are bulk copies, without a tensor map
    const uint64_t np = (uint64_t)(a.num_pages < (int64_t)INT32_MAX ? a.num_pages : (int64_t)INT32_MAX);
    const TmapKey key{a.kv, np, (uint32_t)P, 3};
    if (!tmap_lookup(key, &tkv)) {
      const cuuint64_t dims[3] = {(cuuint64_t)kHeadDim, (cuuint64_t)P, (cuuint64_t)np};
      const cuuint64_t strides[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)P * kTokenBytes};
      const cuuint32_t box[3] = {(cuuint32_t)kHeadDim, (cuuint32_t)min(P, kTile), 1};
      const cuuint32_t es[3] = {1, 1, 1};
      if (enc(&tkv, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(a.kv), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
      tmap_store(key, tkv);
    }
  }
  {
    const TmapKey key{a.q, (uint64_t)a.batch * K::N, (uint32_t)K::QBOX, 2};
    if (!tmap_lookup(key, &tq)) {
      const cuuint64_t dims[2] = {(cuuint64_t)kHeadDim, (cuuint64_t)a.batch * K::N};
      const cuuint64_t strides[1] = {(cuuint64_t)kHeadDim};
      const cuuint32_t box[2] = {(cuuint32_t)kHeadDim, (cuuint32_t)K::QBOX};
      const cuuint32_t es[2] = {1, 1};
      if (enc(&tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(a.q), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
      tmap_store(key, tq);
    }
  }
  if (IL) tkv = tq;                                      // never read
  const SmemLayout L = smem_layout(K::STAGES, K::Q_BYTES, K::ACC, IL, K::W_BYTES);
  const size_t smem = (size_t)L.total + 1024;
  if (smem > (size_t)kMaxSmem) return cudaErrorInvalidConfiguration;
  static int smem_set[64] = {0};
  static_assert(!FUSED || K::STAGES * kStageBytes + 2 * K::Q_BYTES >= (int)kSelectSmem + 1024 + 4 * 8192,
                "fused top-k scratch (and the keys of 8192-column rows) fit the drained K stages and Q slots");
  cudaError_t e = ensure_dynamic_smem(logits_tc_kernel<NEXT_N, H, FUSED, IL, DUAL_OK>, smem, smem_set);
  if (e != cudaSuccess) return e;

  TcParams p;
  p.context_lens = a.context_lens; p.block_table = a.block_table; p.bt_stride = a.bt_stride;
  p.kv = a.kv; p.num_pages = a.num_pages; p.page_size = P; p.weights = a.weights;
  p.logits = a.logits; p.stride = a.stride; p.width = a.width;
  p.cap = min(a.width, a.bt_stride * (int64_t)P);
  p.batch = a.batch; p.status = a.status;
  p.indices = a.indices; p.idx_stride = a.idx_stride; p.k = a.k; p.req_counter = a.req_counter;
  const int grid = device_sm_count();
  if (grid <= 0) return cudaErrorNoDevice;
  // Programmatic dependent launch: the CTAs may be scheduled (barrier set-up,
  // TMEM allocation) while the previous kernel in the stream drains.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreadsTc);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t le = cudaLaunchKernelEx(&cfg, logits_tc_kernel<NEXT_N, H, FUSED, IL, DUAL_OK>, tkv, tq, p);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

}  // namespace

#if defined(SAI_LOGITS_DUAL)
// Page-split caches with pages of 64 tokens or more, on the shapes whose
// tiles are one job of at most 128 columns: two MMA warps (Cfg::DUAL).
cudaError_t launch_logits_tc_dual(const LogitsArgs& a, cudaStream_t stream) {
  const bool fused = a.indices != nullptr;
  switch (a.next_n * 1000 + a.heads) {
    case 1064: return fused ? launch_tc<1, 64, true, false, true>(a, stream) : launch_tc<1, 64, false, false, true>(a, stream);
    case 2064: return fused ? launch_tc<2, 64, true, false, true>(a, stream) : launch_tc<2, 64, false, false, true>(a, stream);
    case 1128: return fused ? launch_tc<1, 128, true, false, true>(a, stream) : launch_tc<1, 128, false, false, true>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}
#elif !defined(SAI_LOGITS_INTERLEAVED)
cudaError_t launch_logits_tc(const LogitsArgs& a, cudaStream_t stream) {
  const bool fused = a.indices != nullptr;
  const int shape = a.next_n * 1000 + a.heads;
  if (a.page_size >= 64 && (shape == 1064 || shape == 2064 || shape == 1128)) return launch_logits_tc_dual(a, stream);
  switch (shape) {
    case 1064: return fused ? launch_tc<1, 64, true, false>(a, stream) : launch_tc<1, 64, false, false>(a, stream);
    case 2064: return fused ? launch_tc<2, 64, true, false>(a, stream) : launch_tc<2, 64, false, false>(a, stream);
    case 3064: return fused ? launch_tc<3, 64, true, false>(a, stream) : launch_tc<3, 64, false, false>(a, stream);
    case 4064: return fused ? launch_tc<4, 64, true, false>(a, stream) : launch_tc<4, 64, false, false>(a, stream);
    case 1128: return fused ? launch_tc<1, 128, true, false>(a, stream) : launch_tc<1, 128, false, false>(a, stream);
    case 2128: return fused ? launch_tc<2, 128, true, false>(a, stream) : launch_tc<2, 128, false, false>(a, stream);
    case 3128: return fused ? launch_tc<3, 128, true, false>(a, stream) : launch_tc<3, 128, false, false>(a, stream);
    case 4128: return fused ? launch_tc<4, 128, true, false>(a, stream) : launch_tc<4, 128, false, false>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}
#else
cudaError_t launch_logits_tc_interleaved(const LogitsArgs& a, cudaStream_t stream) {
  if (a.indices != nullptr) return cudaErrorInvalidValue;   // the fused launch reads page-split caches only
  switch (a.next_n * 1000 + a.heads) {
    case 1064: return launch_tc<1, 64, false, true>(a, stream);
    case 2064: return launch_tc<2, 64, false, true>(a, stream);
    case 3064: return launch_tc<3, 64, false, true>(a, stream);
    case 4064: return launch_tc<4, 64, false, true>(a, stream);
    case 1128: return launch_tc<1, 128, false, true>(a, stream);
    case 2128: return launch_tc<2, 128, false, true>(a, stream);
    case 3128: return launch_tc<3, 128, false, true>(a, stream);
    case 4128: return launch_tc<4, 128, false, true>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}
#endif

}  // namespace sai
