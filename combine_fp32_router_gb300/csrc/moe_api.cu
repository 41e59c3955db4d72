// C ABI of libmoe.so (declared in include/moe.h): argument validation on the host, the
// workspace carve-up, and the launch sequence of each entry point on the caller's stream.
// The host path allocates no memory and does not synchronise (except moe_get_error); the
// checks are plain integer tests, in the spirit of the report translation's section 2.1
// (itsolotime.com): argument checking belongs in compiled host code, not in Python.
#include <atomic>
#include <cstdlib>
#include <cstring>
#include <new>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

std::atomic<uint64_t> g_wait_ns{2000000000ull};
std::atomic<int> g_debug_flags{0};

// CTA pairs (256-row tiles, tcgen05 cta_group::2) or single CTAs (128-row tiles) for the
// grouped GEMMs; both give bitwise identical results.  The environment variable
// MOE_GEMM_PAIR, read once per process, selects: "0" single CTAs only, "1" pairs wherever
// an expert can fill a pair tile, unset (or anything else) the size rule of row_pairs.
enum PairMode { kPairsOff = 0, kPairsOn = 1, kPairsAuto = 2 };
PairMode pair_mode() {
  static const PairMode v = [] {
    const char* e = std::getenv("MOE_GEMM_PAIR");
    if (e && e[0] == '0' && e[1] == 0) return kPairsOff;
    if (e && e[0] == '1' && e[1] == 0) return kPairsOn;
    return kPairsAuto;
  }();
  return v;
}
bool use_pairs() { return pair_mode() != kPairsOff; }


// CTA pairs for the row-grouped GEMMs (the experts' 256-row pair tiles, chosen per expert on
// the device; the rest in a second, single-CTA launch): only when some expert can fill a pair
// tile (T > 128) and the layer is large enough that the second launch's ramp and tail are
// paid back, T k d d_ff >= 2^37 (GEMM1 >= 0.55 TFLOP).  Measured on GB300: T=4096, d=2048,
// E=64, top-6, d_ff=1024 (T k d d_ff = 5.2e10) runs 7% faster on single CTAs alone;
// T=8192, d=4096, E=128, top-8, d_ff=1536 (4.1e11) 3% faster with pairs.
bool row_pairs(int64_t T, int k, int d, int dff) {
  if (pair_mode() == kPairsOff || T <= kTileRows) return false;
  const double work = static_cast<double>(T) * k * d * dff;
  return pair_mode() == kPairsOn || work >= 137438953472.0;
}

// The size rule of the swapped-operand kinds (weight columns or rows x row blocks, every expert
// on CTA pairs in one launch): small batches (T <= 128), wherever the row-tile kernels would use
// CTA pairs, and from T k d d_ff >= 2^36 (half the row-pair threshold).  Measured on GB300:
//  * T=4096, d=2048, E=64, top-6, d_ff=1024 (5.2e10): forward 0.335 ms on single-CTA row
//    tiles, 0.385 swapped;
//  * T=1024, d=4096, E=64, top-8, d_ff=1536 (5.2e10): 0.508 / 0.512 ms;
//  * T=2048, d=4096, E=32, top-8, d_ff=1536 (1.0e11): 0.551 / 0.528 ms, backward 1.200 / 1.139;
//  * T=1..128 with d=7168, E=256, top-8, d_ff=2048: 2-18% faster swapped; the T=16384 layer
//    of that shape and T=8192, d=4096, E=128, top-8, d_ff=1536: 1-2%.
bool swap_size(int64_t T, int k, int d, int dff) {
  if (T <= kTileRows || row_pairs(T, k, d, dff)) return true;
  const double work = static_cast<double>(T) * k * d * dff;
  return pair_mode() == kPairsAuto && work >= 68719476736.0;
}

// Forward GEMMs with swapped operands by the size rule above; the row-tile kernels (single
// CTAs) below it.  MOE_FWD_SWAP="0" turns the swapped kernels off, "1" uses them for every
// size; MOE_GEMM_PAIR="0" (single CTAs only) turns them off too.  Read once per process;
// every choice gives bitwise the same rows.
bool forward_swap(int64_t T, int k, int d, int dff) {
  static const int mode = [] {
    const char* e = std::getenv("MOE_FWD_SWAP");
    if (e && e[0] == '0' && e[1] == 0) return 0;
    if (e && e[0] == '1' && e[1] == 0) return 1;
    return 2;
  }();
  if (mode == 0 || !use_pairs()) return false;
  return mode == 1 || swap_size(T, k, d, dff);
}

// The backward's dX GEMM with swapped operands (every expert on CTA pairs in one launch) by the
// same size rule as the forward's (measured on GB300: the fwd_bwd workload, T=8192, d=4096,
// E=128, top-8, d_ff=1536, whose 5-tile experts otherwise run on single CTAs in a second
// launch; and T=2048, d=4096, E=32, top-8, d_ff=1536, dX 0.344 -> 0.294 ms).
// MOE_BWD_SWAP="0" keeps the row-tile kernels, "1" swaps at every size; read once per process.
// Bitwise the same dX rows either way.
bool backward_swap(int64_t T, int k, int d, int dff) {
  static const int mode = [] {
    const char* e = std::getenv("MOE_BWD_SWAP");
    if (e && e[0] == '0' && e[1] == 0) return 0;
    if (e && e[0] == '1' && e[1] == 0) return 1;
    return 2;
  }();
  if (mode == 0 || !use_pairs()) return false;
  return mode == 1 || swap_size(T, k, d, dff);
}

// The backward's dH GEMM with swapped operands, by the same rule unless MOE_BWD_DH_SWAP ("0"
// or "1") overrides it; read once per process.  Bitwise the same dA and dB rows either way.
bool backward_swap_dh(int64_t T, int k, int d, int dff) {
  static const int mode = [] {
    const char* e = std::getenv("MOE_BWD_DH_SWAP");
    if (e && e[0] == '0' && e[1] == 0) return 0;
    if (e && e[0] == '1' && e[1] == 0) return 1;
    return 2;
  }();
  if (mode == 0 || !use_pairs()) return false;
  return mode == 1 || backward_swap(T, k, d, dff);
}

// Whether the swapped GEMM1 copies the permuted rows itself (its copy warps write x_perm
// block by block in the order its tiles read them, so the copy runs under the MMAs) instead
// of the dispatch's scatter kernel.  MOE_FWD_ROW_COPY="0" keeps the scatter's copies, "1"
// (or unset) the GEMM's; read once per process.  Bitwise the same rows either way.
bool gemm_row_copy() {
  static const int mode = [] {
    const char* e = std::getenv("MOE_FWD_ROW_COPY");
    if (e && e[0] == '0' && e[1] == 0) return 0;
    return 1;
  }();
  return mode == 1;
}

// The swapped GEMMs as one persistent launch (GEMM2 of a row block after its GEMM1 tiles) for
// T <= 64, where one launch's ramp and tail matter (measured on GB300: tiny 0.037 -> 0.034 ms,
// T=1 at d=7168, E=256, top-8, d_ff=2048 0.158 -> 0.154 ms; T=8 and larger layers within
// noise or slower, e.g. the T=16384 layer 9.67 -> 9.88 ms).  MOE_FWD_FUSED "1" forces it,
// "0" turns it off; read once per process.  Bitwise the same rows as two launches.
bool forward_fused(int64_t T) {
  static const int mode = [] {
    const char* e = std::getenv("MOE_FWD_FUSED");
    if (e && e[0] == '0' && e[1] == 0) return 0;
    if (e && e[0] == '1' && e[1] == 0) return 1;
    return 2;
  }();
  return mode == 1 || (mode == 2 && T <= 64);
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// moe_forward_host's staging at the end of the workspace: x, logits, out (256-byte aligned)
size_t host_io_bytes(int64_t T, int d, int E) {
  const size_t t = static_cast<size_t>(T);
  return round_up(t * d * 2, 256) + round_up(t * E * 4, 256) + round_up(t * d * 2, 256);
}


bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks shared by every entry point.  `need_gemm` adds the tile-shape constraints of the
// expert GEMMs (d and d_ff multiples of 128).
moe_status_t check_dims(int64_t T, int d, int E, int k, int dff, bool need_gemm) {
  if (T < 0 || d <= 0 || E <= 0 || k <= 0 || k > E || (need_gemm && dff <= 0))
    return MOE_ERR_INVALID_ARG;
  if (E > kMaxE || k > kMaxK || d > 65536 || d % 8 != 0) return MOE_ERR_UNSUPPORTED;
  if (need_gemm && (d % 128 != 0 || dff % 128 != 0 || dff > 65536)) return MOE_ERR_UNSUPPORTED;
  if (T > (int64_t{1} << 31) / k) return MOE_ERR_UNSUPPORTED;
  if (T * k + static_cast<int64_t>(kTileRows) * E >= (int64_t{1} << 31))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int num_sms_of_current_device() {
  static std::atomic<int> cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (dev >= 0 && dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 152;
  if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

moe_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                                    \
  do {                                                   \
    const cudaError_t e_ = (expr);                       \
    if (e_ != cudaSuccess) return MOE_ERR_CUDA;          \
  } while (0)

void record(cudaEvent_t* ev, int i, cudaStream_t s) {
  if (ev && ev[i]) cudaEventRecord(ev[i], s);
}

}  // namespace

WsLayout make_layout(int64_t T, int d, int E, int k, int dff) {
  WsLayout L;
  L.T = T;
  L.d = d;
  L.E = E;
  L.k = k;
  L.dff = dff;
  L.P = T * k;
  L.nblk = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  // every non-empty expert segment is padded to a multiple of 128 rows
  const int64_t busy = L.P < E ? L.P : E;
  L.P_pad = round_up(static_cast<size_t>(L.P + (kTileRows - 1) * busy), kTileRows);
  L.max_mt = L.P_pad / kTileRows;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += round_up(bytes ? bytes : 1, 256);
    return o;
  };
  const size_t P = static_cast<size_t>(L.P), Pp = static_cast<size_t>(L.P_pad);
  L.err = take(sizeof(DevErr));
  L.hist = take(static_cast<size_t>(L.nblk) * E * 4);
  L.bbase = take(static_cast<size_t>(L.nblk) * E * 4);
  L.route_total = off;
  L.counts = take(static_cast<size_t>(E) * 4);
  L.offsets = take(static_cast<size_t>(E + 1) * 4);
  L.poff = take(static_cast<size_t>(E + 1) * 4);
  L.n_mt = take(16);
  L.mt_expert = take(static_cast<size_t>(L.max_mt) * 4);
  L.mt_row0 = take(static_cast<size_t>(L.max_mt) * 4);
  L.n_pt = take(16);
  L.pt_expert = take(static_cast<size_t>(L.max_mt) * 4);
  L.pt_row0 = take(static_cast<size_t>(L.max_mt) * 4);
  L.n_lo = take(16);
  L.lo_expert = take(static_cast<size_t>(L.max_mt) * 4);
  L.lo_row0 = take(static_cast<size_t>(L.max_mt) * 4);
  L.n_st = take(16);  // 256-row blocks: never more than the 128-row tiles
  L.st_expert = take(static_cast<size_t>(L.max_mt) * 4);
  L.st_row0 = take(static_cast<size_t>(L.max_mt) * 4);
  L.done1 = take(static_cast<size_t>(L.max_mt) * 4);
  L.topk = take(P * 4);
  L.gate = take(P * 4);
  L.pos = take(P * 4);
  L.perm = take(Pp * 4);
  L.xperm = take(Pp * d * 2);
  L.H = take(Pp * dff * 2);
  L.Y = take(Pp * d * 2);  // bf16 expert output rows
  L.seg = take(P / (k > 0 ? k : 1) * static_cast<size_t>(d / 128) * 4);  // [T, d/128] counters
  L.xscale = take(static_cast<size_t>(T) * 4);  // FP8 payload: one scale per token
  L.fwd_total = off;
  L.Asave = take(Pp * dff * 4);
  L.Bsave = take(Pp * dff * 4);
  L.dO = take(Pp * d * 2);
  L.dAB = take(Pp * 2 * dff * 2);
  L.dXp = take(Pp * d * 4);
  L.bwd_total = off;
  return L;
}

TileTables tile_tables(const WsLayout& L, char* w) {
  TileTables tt;
  tt.n_mt = reinterpret_cast<int32_t*>(w + L.n_mt);
  tt.mt_expert = reinterpret_cast<int32_t*>(w + L.mt_expert);
  tt.mt_row0 = reinterpret_cast<int32_t*>(w + L.mt_row0);
  tt.n_pt = reinterpret_cast<int32_t*>(w + L.n_pt);
  tt.pt_expert = reinterpret_cast<int32_t*>(w + L.pt_expert);
  tt.pt_row0 = reinterpret_cast<int32_t*>(w + L.pt_row0);
  tt.n_lo = reinterpret_cast<int32_t*>(w + L.n_lo);
  tt.lo_expert = reinterpret_cast<int32_t*>(w + L.lo_expert);
  tt.lo_row0 = reinterpret_cast<int32_t*>(w + L.lo_row0);
  tt.n_st = reinterpret_cast<int32_t*>(w + L.n_st);
  tt.st_expert = reinterpret_cast<int32_t*>(w + L.st_expert);
  tt.st_row0 = reinterpret_cast<int32_t*>(w + L.st_row0);
  tt.done1 = reinterpret_cast<int32_t*>(w + L.done1);
  tt.max_mt = L.max_mt;
  return tt;
}

}  // namespace moe

namespace moe {
moe_status_t check_route_args(const void* x, const void* logits, int64_t T, int d, int E, int k,
                              const void* topk_idx, const void* gate, const void* counts,
                              const void* offsets, const void* perm, const void* pos,
                              const void* x_perm) {
  moe_status_t st = check_dims(T, d, E, k, 0, false);
  if (st != MOE_OK) return st;
  if (!counts || !offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !logits || !topk_idx || !gate || !perm || !pos || !x_perm))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, logits, topk_idx, gate, counts, offsets, perm, pos, x_perm};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_route_workspace_bytes(int64_t T, int E, int k) {
  if (check_dims(T, 8, E, k, 0, false) != MOE_OK) return 0;
  return make_layout(T, 8, E, k, 128).route_total;
}

size_t moe_workspace_bytes(int64_t T, int d, int E, int k, int d_ff, int needs) {
  if (check_dims(T, d, E, k, d_ff, true) != MOE_OK) return 0;
  if (needs & ~(MOE_WS_BACKWARD | MOE_WS_HOST_IO)) return 0;
  const WsLayout L = make_layout(T, d, E, k, d_ff);
  return ((needs & MOE_WS_BACKWARD) ? L.bwd_total : L.fwd_total) +
         ((needs & MOE_WS_HOST_IO) ? host_io_bytes(T, d, E) : 0);
}

moe_status_t moe_route_dispatch(const moe_bf16_t* x, const float* logits, int64_t T, int d,
                                int E, int k, int32_t* topk_idx, float* gate, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* pos,
                                moe_bf16_t* x_perm, void* ws, size_t ws_bytes,
                                cudaStream_t stream) {
  moe_status_t st = check_route_args(x, logits, T, d, E, k, topk_idx, gate, counts, offsets,
                                     perm, pos, x_perm);
  if (st != MOE_OK) return st;
  if (!ws) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  const WsLayout L = make_layout(T, d, E, k, 128);
  if (ws_bytes < L.route_total) return MOE_ERR_WORKSPACE;

  char* w = static_cast<char*>(ws);
  DevErr* err = reinterpret_cast<DevErr*>(w + L.err);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(DevErr), stream));
  if (T == 0) {
    MOE_TRY(cudaMemsetAsync(counts, 0, static_cast<size_t>(E) * 4, stream));
    MOE_TRY(cudaMemsetAsync(offsets, 0, static_cast<size_t>(E + 1) * 4, stream));
    return MOE_OK;
  }
  int32_t* hist = reinterpret_cast<int32_t*>(w + L.hist);
  int32_t* bbase = reinterpret_cast<int32_t*>(w + L.bbase);
  MOE_TRY(launch_route_topk(logits, T, E, k, topk_idx, gate, pos, hist, err, stream));
  MOE_TRY(launch_scan_cols(hist, L.nblk, E, bbase, counts, stream));
  // unpadded rows: the padded offsets are the offsets themselves
  MOE_TRY(launch_offsets(counts, E, 1, nullptr, offsets, nullptr, err, stream));
  MOE_TRY(launch_scatter(x, T, d, E, k, topk_idx, bbase, offsets, pos, perm, x_perm, L.P, err,
                         stream));
  return MOE_OK;
}

namespace moe {
namespace {
// Host-side argument checks of moe_forward (nothing is launched).
moe_status_t check_forward(const moe_bf16_t* x, const float* logits, const moe_bf16_t* W1,
                           const moe_bf16_t* W3, const moe_bf16_t* W2, int64_t T, int d, int E,
                           int k, int d_ff, const moe_bf16_t* out, const void* ws,
                           size_t ws_bytes, int flags) {
  moe_status_t st = check_dims(T, d, E, k, d_ff, true);
  if (st != MOE_OK) return st;
  if (!W1 || !W2 || !ws) return MOE_ERR_INVALID_ARG;
  if (!W3 && d_ff % 256 != 0) return MOE_ERR_UNSUPPORTED;  // squared ReLU: 256-column tiles
  if (T > 0 && (!x || !logits || !out)) return MOE_ERR_INVALID_ARG;
  if (flags & ~(MOE_FWD_SAVE_FOR_BACKWARD | MOE_FWD_FUSED_COMBINE | MOE_FWD_GATHER_ROWS))
    return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, logits, W1, W3, W2, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  const bool save = (flags & MOE_FWD_SAVE_FOR_BACKWARD) != 0;
  const WsLayout L = make_layout(T, d, E, k, d_ff);
  if (ws_bytes < (save ? L.bwd_total : L.fwd_total)) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}
}  // namespace
}  // namespace moe

moe_status_t moe_forward(const moe_bf16_t* x, const float* logits, const moe_bf16_t* W1,
                         const moe_bf16_t* W3, const moe_bf16_t* W2, int64_t T, int d, int E,
                         int k, int d_ff, moe_bf16_t* out, void* ws, size_t ws_bytes, int flags,
                         cudaEvent_t* stage_events, cudaStream_t stream) {
  moe_status_t st = check_forward(x, logits, W1, W3, W2, T, d, E, k, d_ff, out, ws, ws_bytes,
                                  flags);
  if (st != MOE_OK) return st;
  const bool save = (flags & MOE_FWD_SAVE_FOR_BACKWARD) != 0;
  const WsLayout L = make_layout(T, d, E, k, d_ff);

  char* w = static_cast<char*>(ws);
  DevErr* err = reinterpret_cast<DevErr*>(w + L.err);
  record(stage_events, 0, stream);
  // a batch of T <= 128 is dispatched in one launch, which also clears the error record
  const bool small = T > 0 && T <= kRouteTokensPerBlock && (g_debug_flags.load() & 2) == 0;
  if (!small) MOE_TRY(cudaMemsetAsync(err, 0, sizeof(DevErr), stream));
  if (T == 0) {
    for (int i = 1; i < MOE_FWD_NUM_EVENTS; ++i) record(stage_events, i, stream);
    return MOE_OK;
  }
  int32_t* hist = reinterpret_cast<int32_t*>(w + L.hist);
  int32_t* bbase = reinterpret_cast<int32_t*>(w + L.bbase);
  int32_t* counts = reinterpret_cast<int32_t*>(w + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  int32_t* poff = reinterpret_cast<int32_t*>(w + L.poff);
  int32_t* topk = reinterpret_cast<int32_t*>(w + L.topk);
  float* gate = reinterpret_cast<float*>(w + L.gate);
  int32_t* pos = reinterpret_cast<int32_t*>(w + L.pos);
  int32_t* perm = reinterpret_cast<int32_t*>(w + L.perm);
  uint16_t* xperm = reinterpret_cast<uint16_t*>(w + L.xperm);

  // dispatch: route, count, prefix sums (rows padded to 128 per expert), stable permute.
  // With MOE_FWD_GATHER_ROWS (and no backward, which reads x_perm as a K operand) GEMM1
  // gathers its rows from x itself: the dispatch copy of the next tiles overlaps the MMAs of
  // the current ones.
  const bool gather = !save && (flags & MOE_FWD_GATHER_ROWS) != 0;
  // the plain forward runs both GEMMs with swapped operands on CTA pairs; the row-gather and
  // fused-combine variants keep the row-tile kernels
  const bool swap = forward_swap(T, k, d, d_ff) && !gather &&
                    (flags & MOE_FWD_FUSED_COMBINE) == 0;
  // above the single-launch dispatch's batch size, the swapped GEMM1 copies the rows
  // (gemm_row_copy); the one-launch pair of GEMMs (forward_fused) reads rows the dispatch
  // copied
  const bool copy_in_gemm =
      T > kRouteTokensPerBlock && swap && !forward_fused(T) && gemm_row_copy();
  const TileTables tt = tile_tables(L, w);
  const int num_sms = num_sms_of_current_device();
  if (small) {
    // one launch for the whole dispatch of a small batch
    MOE_TRY(launch_dispatch_small(logits, x, T, d, E, k, kTileRows, topk, gate, pos, perm,
                                  counts, offsets, poff, &tt, gather ? nullptr : xperm, L.P_pad,
                                  num_sms, err, stream));
    // zero x padding rows when the backward will read them as a K operand
    if (save) MOE_TRY(launch_pad_rows(counts, poff, E, nullptr, xperm, 2ll * d, stream));
  } else {
    MOE_TRY(launch_route_topk(logits, T, E, k, topk, gate, pos, hist, err, stream));
    MOE_TRY(launch_scan_cols(hist, L.nblk, E, bbase, counts, stream));
    MOE_TRY(launch_offsets(counts, E, kTileRows, offsets, poff, &tt, err, stream));
    MOE_TRY(launch_scatter(x, T, d, E, k, topk, bbase, poff, pos, perm,
                           (gather || copy_in_gemm) ? nullptr : xperm, L.P_pad, err, stream));
    // padding rows: perm = -1; zero x rows when the backward will read them as a K operand
    MOE_TRY(launch_pad_rows(counts, poff, E, perm, save ? xperm : nullptr, 2ll * d, stream));
  }
  record(stage_events, 1, stream);

  GemmCtx c{};
  c.L = &L;
  c.ws = w;
  c.x = x;
  c.W1 = W1;
  c.W3 = W3;
  c.W2 = W2;
  c.save_ab = save ? 1 : 0;
  c.err = err;
  c.wait_ns = g_wait_ns.load();
  c.debug_flags = g_debug_flags.load();
  c.num_sms = num_sms;
  c.pair = row_pairs(T, k, d, d_ff);
  c.fuse_combine = (flags & MOE_FWD_FUSED_COMBINE) != 0;
  c.gated = W3 != nullptr;
  c.gather_x = gather;
  c.copy_rows = copy_in_gemm;
  c.out = out;
  c.swap = swap;
  if (c.swap && forward_fused(T)) {
    // both GEMMs in one launch: the GEMM1 and GEMM2 stage events bracket it together
    MOE_TRY(launch_gemm_fwd_fused(c, stream));
    record(stage_events, 2, stream);
    record(stage_events, 3, stream);
    MOE_TRY(launch_combine(reinterpret_cast<const uint16_t*>(w + L.Y), L.P_pad, gate, pos, T, k,
                           d, out, err, stream));
    record(stage_events, 4, stream);
    return MOE_OK;
  }
  MOE_TRY(c.swap ? launch_gemm_fwd1_swap(c, stream) : launch_gemm_fwd1(c, stream));
  record(stage_events, 2, stream);
  if (c.fuse_combine) {
    // GEMM2 combines each token as soon as its k expert rows are written
    const int bn2 = (d % 256 == 0) ? 256 : 128;
    MOE_TRY(cudaMemsetAsync(w + L.seg, 0, static_cast<size_t>(T) * (d / bn2) * 4, stream));
    MOE_TRY(launch_gemm_fwd2(c, stream));
    record(stage_events, 3, stream);
    record(stage_events, 4, stream);
    return MOE_OK;
  }
  MOE_TRY(c.swap ? launch_gemm_fwd2_swap(c, stream) : launch_gemm_fwd2(c, stream));
  record(stage_events, 3, stream);
  MOE_TRY(launch_combine(reinterpret_cast<const uint16_t*>(w + L.Y), L.P_pad, gate, pos, T, k, d,
                         out, err, stream));
  record(stage_events, 4, stream);
  return MOE_OK;
}

moe_status_t moe_quantize_weights_fp8(const moe_bf16_t* W, int E, int K, int N, uint8_t* Wq,
                                      float* scales, cudaStream_t stream) {
  if (E < 1 || K < 1 || N < 1 || K % 128 != 0 || N % 128 != 0) return MOE_ERR_UNSUPPORTED;
  if (!W || !Wq || !scales || !aligned16(W) || !aligned16(Wq) || !aligned16(scales))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(launch_quantize_weights_fp8(W, E, K, N, Wq, scales, stream));
  return MOE_OK;
}

moe_status_t moe_forward_fp8(const moe_bf16_t* x, const float* logits, const uint8_t* W1q,
                             const uint8_t* W3q, const float* w1_scale, const float* w3_scale,
                             const moe_bf16_t* W2, int64_t T, int d, int E, int k, int d_ff,
                             moe_bf16_t* out, void* ws, size_t ws_bytes,
                             cudaEvent_t* stage_events, cudaStream_t stream) {
  moe_status_t st = check_dims(T, d, E, k, d_ff, true);
  if (st != MOE_OK) return st;
  if (!W1q || !W3q || !w1_scale || !w3_scale || !W2 || !ws) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x || !logits || !out)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {x, logits, W1q, W3q, w1_scale, w3_scale, W2, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  const WsLayout L = make_layout(T, d, E, k, d_ff);
  if (ws_bytes < L.fwd_total) return MOE_ERR_WORKSPACE;

  char* w = static_cast<char*>(ws);
  DevErr* err = reinterpret_cast<DevErr*>(w + L.err);
  record(stage_events, 0, stream);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(DevErr), stream));
  if (T == 0) {
    for (int i = 1; i < MOE_FWD_NUM_EVENTS; ++i) record(stage_events, i, stream);
    return MOE_OK;
  }
  int32_t* hist = reinterpret_cast<int32_t*>(w + L.hist);
  int32_t* bbase = reinterpret_cast<int32_t*>(w + L.bbase);
  int32_t* counts = reinterpret_cast<int32_t*>(w + L.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  int32_t* poff = reinterpret_cast<int32_t*>(w + L.poff);
  int32_t* topk = reinterpret_cast<int32_t*>(w + L.topk);
  float* gate = reinterpret_cast<float*>(w + L.gate);
  int32_t* pos = reinterpret_cast<int32_t*>(w + L.pos);
  int32_t* perm = reinterpret_cast<int32_t*>(w + L.perm);

  // dispatch with the FP8 payload: route, count, prefix sums, E4M3 rows + row scales
  MOE_TRY(launch_route_topk(logits, T, E, k, topk, gate, pos, hist, err, stream));
  MOE_TRY(launch_scan_cols(hist, L.nblk, E, bbase, counts, stream));
  const TileTables tt = tile_tables(L, w);
  MOE_TRY(launch_offsets(counts, E, kTileRows, offsets, poff, &tt, err, stream));
  MOE_TRY(launch_scatter_fp8(x, T, d, E, k, topk, bbase, poff, pos, perm,
                             reinterpret_cast<uint8_t*>(w + L.xperm),
                             reinterpret_cast<float*>(w + L.xscale), L.P_pad, err, stream));
  MOE_TRY(launch_pad_rows(counts, poff, E, perm, nullptr, 0, stream));
  record(stage_events, 1, stream);

  GemmCtx c{};
  c.L = &L;
  c.ws = w;
  c.x = x;
  c.W2 = W2;
  c.W1q = W1q;
  c.W3q = W3q;
  c.wscale1 = w1_scale;
  c.wscale3 = w3_scale;
  c.err = err;
  c.wait_ns = g_wait_ns.load();
  c.debug_flags = g_debug_flags.load();
  c.num_sms = num_sms_of_current_device();
  c.pair = row_pairs(T, k, d, d_ff);
  c.gated = true;
  c.out = out;
  MOE_TRY(launch_gemm_fwd1_fp8(c, stream));
  record(stage_events, 2, stream);
  // GEMM2 takes the bf16 H rows as in moe_forward, swapped by the same rule
  MOE_TRY(forward_swap(T, k, d, d_ff) ? launch_gemm_fwd2_swap(c, stream)
                                      : launch_gemm_fwd2(c, stream));
  record(stage_events, 3, stream);
  MOE_TRY(launch_combine(reinterpret_cast<const uint16_t*>(w + L.Y), L.P_pad, gate, pos, T, k, d,
                         out, err, stream));
  record(stage_events, 4, stream);
  return MOE_OK;
}

size_t moe_expert_workspace_bytes(int64_t n_rows, int d, int E, int d_ff) {
  if (check_dims(n_rows, d, E, 1, d_ff, true) != MOE_OK) return 0;
  return make_layout(n_rows, d, E, 1, d_ff).fwd_total;
}

// The expert stage on the caller's rows: the tile tables from the caller's counts, then the
// swapped GEMM1 and GEMM2 with the caller's rows as the row operand and y_rows as GEMM2's
// output (the workspace holds the tables and H).  The same kernels as moe_forward's, so each
// row's results are bitwise moe_forward's.
moe_status_t moe_expert_forward(const moe_bf16_t* rows, const int32_t* counts, int64_t n_rows,
                                int d, int E, int d_ff, const moe_bf16_t* W1,
                                const moe_bf16_t* W3, const moe_bf16_t* W2, moe_bf16_t* y_rows,
                                void* ws, size_t ws_bytes, cudaStream_t stream) {
  moe_status_t st = check_dims(n_rows, d, E, 1, d_ff, true);
  if (st != MOE_OK) return st;
  if (!counts || !W1 || !W2 || !ws) return MOE_ERR_INVALID_ARG;
  if (!W3 && d_ff % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (n_rows > 0 && (!rows || !y_rows)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {rows, W1, W3, W2, y_rows};
  for (const void* q : ptrs)
    if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(counts) & 3u) != 0) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  const WsLayout L = make_layout(n_rows, d, E, 1, d_ff);
  if (ws_bytes < L.fwd_total) return MOE_ERR_WORKSPACE;
  char* w = static_cast<char*>(ws);
  DevErr* err = reinterpret_cast<DevErr*>(w + L.err);
  MOE_TRY(cudaMemsetAsync(err, 0, sizeof(DevErr), stream));
  if (n_rows == 0) return MOE_OK;
  int32_t* cnt = reinterpret_cast<int32_t*>(w + L.counts);
  MOE_TRY(cudaMemcpyAsync(cnt, counts, static_cast<size_t>(E) * 4, cudaMemcpyDeviceToDevice,
                          stream));
  const TileTables tt = tile_tables(L, w);
  MOE_TRY(launch_offsets(cnt, E, kTileRows, reinterpret_cast<int32_t*>(w + L.offsets),
                         reinterpret_cast<int32_t*>(w + L.poff), &tt, err, stream));
  GemmCtx c{};
  c.L = &L;
  c.ws = w;
  c.W1 = W1;
  c.W3 = W3;
  c.W2 = W2;
  c.err = err;
  c.wait_ns = g_wait_ns.load();
  c.debug_flags = g_debug_flags.load();
  c.num_sms = num_sms_of_current_device();
  c.gated = W3 != nullptr;
  c.rows = rows;
  c.y = y_rows;
  c.rows_cap = n_rows;
  MOE_TRY(launch_gemm_fwd1_swap(c, stream));
  MOE_TRY(launch_gemm_fwd2_swap(c, stream));
  return MOE_OK;
}

moe_status_t moe_combine(const moe_bf16_t* y_rows, int64_t n_rows, const float* gate,
                         const int32_t* pos, int64_t T, int k, int d, moe_bf16_t* out,
                         void* err_word, cudaStream_t stream) {
  if (T < 0 || k < 1 || d <= 0 || n_rows < 0) return MOE_ERR_INVALID_ARG;
  if (k > kMaxK || d % 8 != 0 || d > 65536 || T > (int64_t{1} << 31) / k)
    return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!y_rows || n_rows < 1 || !gate || !pos || !out || !err_word) return MOE_ERR_INVALID_ARG;
  if (!aligned16(y_rows) || !aligned16(out) || !aligned16(err_word)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(gate) & 3u) != 0 || (reinterpret_cast<uintptr_t>(pos) & 3u) != 0)
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(launch_combine(y_rows, n_rows, gate, pos, T, k, d, out,
                         static_cast<DevErr*>(err_word), stream));
  return MOE_OK;
}

struct moe_forward_graph {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

moe_status_t moe_forward_graph_create(const moe_bf16_t* x, const float* logits,
                                      const moe_bf16_t* W1, const moe_bf16_t* W3,
                                      const moe_bf16_t* W2, int64_t T, int d, int E, int k,
                                      int d_ff, moe_bf16_t* out, void* ws, size_t ws_bytes,
                                      int flags, moe_forward_graph_t* graph) {
  if (!graph) return MOE_ERR_INVALID_ARG;
  *graph = nullptr;
  moe_status_t st = check_forward(x, logits, W1, W3, W2, T, d, E, k, d_ff, out, ws, ws_bytes,
                                  flags);
  if (st != MOE_OK) return st;
  // record the launches of one moe_forward on a private stream (nothing runs), then
  // instantiate them
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return MOE_ERR_CUDA;
  cudaGraph_t g = nullptr;
  if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(cs);
    return MOE_ERR_CUDA;
  }
  st = moe_forward(x, logits, W1, W3, W2, T, d, E, k, d_ff, out, ws, ws_bytes, flags, nullptr,
                   cs);
  const cudaError_t ce = cudaStreamEndCapture(cs, &g);
  cudaStreamDestroy(cs);
  if (st != MOE_OK || ce != cudaSuccess || !g) {
    if (g) cudaGraphDestroy(g);
    return st != MOE_OK ? st : MOE_ERR_CUDA;
  }
  cudaGraphExec_t ex = nullptr;
  if (cudaGraphInstantiate(&ex, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    return MOE_ERR_CUDA;
  }
  auto* h = new (std::nothrow) moe_forward_graph{g, ex};
  if (!h) {
    cudaGraphExecDestroy(ex);
    cudaGraphDestroy(g);
    return MOE_ERR_CUDA;
  }
  *graph = h;
  return MOE_OK;
}

moe_status_t moe_forward_graph_launch(moe_forward_graph_t graph, cudaStream_t stream) {
  if (!graph) return MOE_ERR_INVALID_ARG;
  return cudaGraphLaunch(graph->exec, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

void moe_forward_graph_destroy(moe_forward_graph_t graph) {
  if (!graph) return;
  cudaGraphExecDestroy(graph->exec);
  cudaGraphDestroy(graph->graph);
  delete graph;
}

namespace {
// moe_forward_host and moe_forward_host_pipelined: the input copies on `copy`, the layer on
// `stream`, the output copy on `copy`.  With two streams, inputs_ready / layer_done order
// them (recorded and waited on here); with one, stream order does.
moe_status_t forward_host_impl(const moe_bf16_t* x_host, const float* logits_host,
                               const moe_bf16_t* W1, const moe_bf16_t* W3, const moe_bf16_t* W2,
                               int64_t T, int d, int E, int k, int d_ff, moe_bf16_t* out_host,
                               void* ws, size_t ws_bytes, int flags, cudaEvent_t* stage_events,
                               cudaStream_t stream, cudaStream_t copy, cudaEvent_t inputs_ready,
                               cudaEvent_t layer_done) {
  moe_status_t st = check_dims(T, d, E, k, d_ff, true);
  if (st != MOE_OK) return st;
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!x_host || !logits_host || !out_host)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  const WsLayout L = make_layout(T, d, E, k, d_ff);
  const bool save = (flags & MOE_FWD_SAVE_FOR_BACKWARD) != 0;
  const size_t io = host_io_bytes(T, d, E);
  const size_t layer = save ? L.bwd_total : L.fwd_total;
  if (ws_bytes < layer + io) return MOE_ERR_WORKSPACE;
  // staging at the end of ws; the layer's own region stays [0, io0), as for moe_forward
  const size_t io0 = (ws_bytes - io) & ~static_cast<size_t>(255);
  char* w = static_cast<char*>(ws);
  moe_bf16_t* x = reinterpret_cast<moe_bf16_t*>(w + io0);
  float* logits = reinterpret_cast<float*>(w + io0 + round_up(static_cast<size_t>(T) * d * 2, 256));
  moe_bf16_t* out = reinterpret_cast<moe_bf16_t*>(
      w + io0 + round_up(static_cast<size_t>(T) * d * 2, 256) +
      round_up(static_cast<size_t>(T) * E * 4, 256));
  const size_t xb = static_cast<size_t>(T) * d * 2, lb = static_cast<size_t>(T) * E * 4;
  if (T > 0) {
    MOE_TRY(cudaMemcpyAsync(x, x_host, xb, cudaMemcpyHostToDevice, copy));
    MOE_TRY(cudaMemcpyAsync(logits, logits_host, lb, cudaMemcpyHostToDevice, copy));
  }
  if (copy != stream) {
    MOE_TRY(cudaEventRecord(inputs_ready, copy));
    MOE_TRY(cudaStreamWaitEvent(stream, inputs_ready, 0));
  }
  st = moe_forward(x, logits, W1, W3, W2, T, d, E, k, d_ff, out, ws, io0, flags, stage_events,
                   stream);
  if (st != MOE_OK) return st;
  if (copy != stream) {
    MOE_TRY(cudaEventRecord(layer_done, stream));
    MOE_TRY(cudaStreamWaitEvent(copy, layer_done, 0));
  }
  if (T > 0) MOE_TRY(cudaMemcpyAsync(out_host, out, xb, cudaMemcpyDeviceToHost, copy));
  return MOE_OK;
}
}  // namespace

moe_status_t moe_forward_host(const moe_bf16_t* x_host, const float* logits_host,
                              const moe_bf16_t* W1, const moe_bf16_t* W3, const moe_bf16_t* W2,
                              int64_t T, int d, int E, int k, int d_ff, moe_bf16_t* out_host,
                              void* ws, size_t ws_bytes, int flags, cudaEvent_t* stage_events,
                              cudaStream_t stream) {
  return forward_host_impl(x_host, logits_host, W1, W3, W2, T, d, E, k, d_ff, out_host, ws,
                           ws_bytes, flags, stage_events, stream, stream, nullptr, nullptr);
}

moe_status_t moe_forward_host_pipelined(const moe_bf16_t* x_host, const float* logits_host,
                                        const moe_bf16_t* W1, const moe_bf16_t* W3,
                                        const moe_bf16_t* W2, int64_t T, int d, int E, int k,
                                        int d_ff, moe_bf16_t* out_host, void* ws,
                                        size_t ws_bytes, int flags, cudaEvent_t* stage_events,
                                        cudaStream_t stream, cudaStream_t copy_stream,
                                        cudaEvent_t inputs_ready, cudaEvent_t layer_done) {
  if (!inputs_ready || !layer_done || inputs_ready == layer_done) return MOE_ERR_INVALID_ARG;
  return forward_host_impl(x_host, logits_host, W1, W3, W2, T, d, E, k, d_ff, out_host, ws,
                           ws_bytes, flags, stage_events, stream, copy_stream, inputs_ready,
                           layer_done);
}

moe_status_t moe_backward(const moe_bf16_t* dy, const moe_bf16_t* x, const float* logits,
                          const moe_bf16_t* W1, const moe_bf16_t* W3, const moe_bf16_t* W2,
                          int64_t T, int d, int E, int k, int d_ff, moe_bf16_t* dx, float* dW1,
                          float* dW3, float* dW2, float* dgate, float* dlogits, void* ws,
                          size_t ws_bytes, cudaEvent_t* stage_events, cudaStream_t stream) {
  moe_status_t st = check_dims(T, d, E, k, d_ff, true);
  if (st != MOE_OK) return st;
  if (!W1 || !W2 || !dW1 || !dW2 || !ws) return MOE_ERR_INVALID_ARG;
  if (!W3 != !dW3) return MOE_ERR_INVALID_ARG;  // no W3 (squared ReLU): no dW3 either
  if (!W3 && d_ff % 256 != 0) return MOE_ERR_UNSUPPORTED;
  if (T > 0 && (!dy || !x || !logits || !dx || !dgate)) return MOE_ERR_INVALID_ARG;
  const void* ptrs[] = {dy, x, logits, W1, W3, W2, dx, dW1, dW3, dW2, dgate, dlogits};
  for (const void* p : ptrs)
    if (!aligned16(p)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return MOE_ERR_INVALID_ARG;
  const WsLayout L = make_layout(T, d, E, k, d_ff);
  if (ws_bytes < L.bwd_total) return MOE_ERR_WORKSPACE;

  char* w = static_cast<char*>(ws);
  DevErr* err = reinterpret_cast<DevErr*>(w + L.err);
  record(stage_events, 0, stream);
  if (T == 0) {
    const size_t wb = static_cast<size_t>(E) * d * d_ff * 4;
    MOE_TRY(cudaMemsetAsync(dW1, 0, wb, stream));
    if (dW3) MOE_TRY(cudaMemsetAsync(dW3, 0, wb, stream));
    MOE_TRY(cudaMemsetAsync(dW2, 0, wb, stream));
    for (int i = 1; i < MOE_BWD_NUM_EVENTS; ++i) record(stage_events, i, stream);
    return MOE_OK;
  }
  const int32_t* counts = reinterpret_cast<const int32_t*>(w + L.counts);
  const int32_t* poff = reinterpret_cast<const int32_t*>(w + L.poff);
  const int32_t* topk = reinterpret_cast<const int32_t*>(w + L.topk);
  const float* gate = reinterpret_cast<const float*>(w + L.gate);
  const int32_t* pos = reinterpret_cast<const int32_t*>(w + L.pos);
  uint16_t* dO = reinterpret_cast<uint16_t*>(w + L.dO);

  // the dX rows' buffer is free until the dX GEMM: it holds the gate grads' partial sums
  MOE_TRY(launch_bwd_gate(dy, reinterpret_cast<const uint16_t*>(w + L.Y), gate, pos, topk, T, k,
                          d, E, dO, dgate, dlogits, reinterpret_cast<float*>(w + L.dXp), stream));
  MOE_TRY(launch_pad_rows(counts, poff, E, nullptr, dO, 2ll * d, stream));
  record(stage_events, 1, stream);

  GemmCtx c{};
  c.L = &L;
  c.ws = w;
  c.x = x;
  c.W1 = W1;
  c.W3 = W3;
  c.W2 = W2;
  c.dW1 = dW1;
  c.dW3 = dW3;
  c.dW2 = dW2;
  c.err = err;
  c.wait_ns = g_wait_ns.load();
  c.debug_flags = g_debug_flags.load();
  c.num_sms = num_sms_of_current_device();
  c.pair = row_pairs(T, k, d, d_ff);  // dH and dX: row-grouped like the forward
  c.gated = W3 != nullptr;
  MOE_TRY(backward_swap_dh(T, k, d, d_ff) ? launch_gemm_dh_swap(c, stream)
                                          : launch_gemm_dh(c, stream));
  record(stage_events, 2, stream);
  MOE_TRY(backward_swap(T, k, d, d_ff) ? launch_gemm_dx_swap(c, stream)
                                       : launch_gemm_dx(c, stream));
  record(stage_events, 3, stream);
  MOE_TRY(launch_combine_f32(reinterpret_cast<const float*>(w + L.dXp), pos, T, k, d, dx,
                             stream));
  record(stage_events, 4, stream);
  c.pair = use_pairs();  // the weight gradients pair on 256 output rows instead
  MOE_TRY(launch_gemm_dw2(c, stream));
  record(stage_events, 5, stream);
  MOE_TRY(launch_gemm_dw13(c, stream));
  record(stage_events, 6, stream);
  return MOE_OK;
}

moe_status_t moe_get_error(const void* ws, cudaStream_t stream) {
  if (!ws) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
  DevErr e{};
  if (cudaMemcpy(&e, ws, sizeof e, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status_t>(e.status);
}

void moe_set_wait_timeout_ns(uint64_t ns) { g_wait_ns.store(ns ? ns : 1); }

void moe_debug_set_flags(int flags) { g_debug_flags.store(flags); }

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_DEVICE_BOUNDS: return "device-side index out of range";
  }
  return "unknown status";
}

}  // extern "C"
