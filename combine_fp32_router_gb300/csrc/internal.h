// Host-side declarations shared between the translation units of libmoe.so.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "moe.h"

namespace moe {

constexpr int kRouteTokensPerBlock = 128;  // tokens per routing CTA (4 ranking chunks of 32)
constexpr int kTileRows = 128;             // rows of one expert GEMM tile; padded row unit
constexpr int kPairOddMinTiles = 7;        // CTA pairs for an odd tile count from this many
constexpr int kMaxK = 16;
constexpr int kMaxE = 1024;

struct DevErr;

// Workspace carve-up (byte offsets from ws, each 256-byte aligned).
struct WsLayout {
  int64_t T = 0, P = 0, P_pad = 0, max_mt = 0, nblk = 0;
  int d = 0, E = 0, k = 0, dff = 0;
  size_t err = 0, hist = 0, bbase = 0, counts = 0, offsets = 0, poff = 0, n_mt = 0,
         mt_expert = 0, mt_row0 = 0, n_pt = 0, pt_expert = 0, pt_row0 = 0, n_lo = 0,
         lo_expert = 0, lo_row0 = 0, n_st = 0, st_expert = 0, st_row0 = 0, done1 = 0, topk = 0,
         gate = 0,
         pos = 0, perm = 0, xperm = 0, H = 0, Y = 0, Asave = 0, Bsave = 0, dO = 0, dAB = 0,
         dXp = 0, seg = 0, xscale = 0;
  size_t route_total = 0, fwd_total = 0, bwd_total = 0;
};

WsLayout make_layout(int64_t T, int d, int E, int k, int dff);

// Argument checks of the dispatch entry points (sizes, null pointers, 16-byte alignment),
// shared by moe_route_dispatch and moe_route_dispatch_noalloc (moe_api.cu).
moe_status_t check_route_args(const void* x, const void* logits, int64_t T, int d, int E, int k,
                              const void* topk_idx, const void* gate, const void* counts,
                              const void* offsets, const void* perm, const void* pos,
                              const void* x_perm);

// ---- routing / dispatch / combine launches (route.cu) -----------------------------------
cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int32_t* topk,
                              float* gate, int32_t* pos_local, int32_t* hist, DevErr* err,
                              cudaStream_t s);
cudaError_t launch_scan_cols(const int32_t* hist, int64_t nblk, int E, int32_t* bbase,
                             int32_t* counts, cudaStream_t s);
struct TileTables;
// The whole dispatch of T <= 128 tokens in one launch (route, counts, offsets and tables as
// launch_offsets, pos, perm with -1 on padding rows, and the row copies unless x_perm is
// null); E <= 1024.  Bitwise the results of the multi-kernel sequence.  It first clears the
// error record `err`, so no memset precedes it.
cudaError_t launch_dispatch_small(const float* logits, const uint16_t* x, int64_t T, int d,
                                  int E, int k, int align, int32_t* topk, float* gate,
                                  int32_t* pos, int32_t* perm, int32_t* counts,
                                  int32_t* offsets, int32_t* poff, const TileTables* tables,
                                  uint16_t* x_perm, int64_t rows_cap, int num_sms, DevErr* err,
                                  cudaStream_t s);
// offsets (unpadded, may be null), poff (rows padded to `align`), and when align == 128
// the tile tables: every 128-row tile (n_mt, mt_expert, mt_row0); the 256-row pair tiles
// (n_pt, pt_expert, pt_row0: two consecutive 128-row tiles of one expert); each expert's odd
// last 128-row tile (n_lo, lo_expert, lo_row0), which pairs leave over; and the blocks of up
// to 256 rows of the swapped forward GEMMs (n_st, st_expert, st_row0: every expert's rows
// cut from its first row in 256-row steps, the last block partial).
struct TileTables {
  int32_t *n_mt, *mt_expert, *mt_row0, *n_pt, *pt_expert, *pt_row0, *n_lo, *lo_expert, *lo_row0;
  int32_t *n_st, *st_expert, *st_row0;
  int32_t* done1;  // per 256-row block: GEMM1 halves stored (both GEMMs in one launch); zeroed
  int64_t max_mt;
};
// The tile tables of a workspace laid out by L.
TileTables tile_tables(const WsLayout& L, char* ws);
cudaError_t launch_offsets(const int32_t* counts, int E, int align, int32_t* offsets,
                           int32_t* poff, const TileTables* tables, DevErr* err,
                           cudaStream_t s);
cudaError_t launch_scatter(const uint16_t* x, int64_t T, int d, int E, int k,
                           const int32_t* topk, const int32_t* bbase, const int32_t* poff,
                           int32_t* pos, int32_t* perm, uint16_t* x_perm, int64_t rows_cap,
                           DevErr* err, cudaStream_t s);
// The stable permute with the FP8 payload: E4M3 rows (d bytes) and a row scale per token.
cudaError_t launch_scatter_fp8(const uint16_t* x, int64_t T, int d, int E, int k,
                               const int32_t* topk, const int32_t* bbase, const int32_t* poff,
                               int32_t* pos, int32_t* perm, uint8_t* x_perm, float* xscale,
                               int64_t rows_cap, DevErr* err, cudaStream_t s);
// E4M3 weights, transposed to [E][N][K], with per-(expert, column) scales [E][N].
cudaError_t launch_quantize_weights_fp8(const uint16_t* W, int E, int K, int N, uint8_t* Wq,
                                        float* scales, cudaStream_t s);
// Padding rows of every expert segment: perm = -1 and (if rows != null) zero bytes.
cudaError_t launch_pad_rows(const int32_t* counts, const int32_t* poff, int E, int32_t* perm,
                            void* rows, int64_t row_bytes, cudaStream_t s);
// y_rows holds rows_cap rows; a pos outside them records MOE_ERR_DEVICE_BOUNDS in err
cudaError_t launch_combine(const uint16_t* y_rows, int64_t rows_cap, const float* gate,
                           const int32_t* pos, int64_t T, int k, int d, uint16_t* out,
                           DevErr* err, cudaStream_t s);
// `part`: scratch of T * ceil(d / 1024) * k floats (per-block partial dot products).
cudaError_t launch_bwd_gate(const uint16_t* dy, const uint16_t* y_rows, const float* gate,
                            const int32_t* pos, const int32_t* topk, int64_t T, int k, int d,
                            int E, uint16_t* dO_rows, float* dgate, float* dlogits, float* part,
                            cudaStream_t s);
cudaError_t launch_combine_f32(const float* rows, const int32_t* pos, int64_t T, int k, int d,
                               uint16_t* out, cudaStream_t s);

// ---- grouped GEMMs (gemm_fwd.cu, gemm_bwd.cu) ------------------------------------------
struct GemmCtx {
  const WsLayout* L;
  char* ws;
  const uint16_t *x, *W1, *W3, *W2;
  float *dW1, *dW3, *dW2;
  int save_ab;
  DevErr* err;
  uint64_t wait_ns;
  int debug_flags;
  int num_sms;
  bool pair;  // 256-row tiles on CTA pairs (tcgen05 cta_group::2)
  bool swap;  // forward GEMMs with weight columns as M and row blocks as N (one pair launch)
  bool fuse_combine;     // GEMM2 also combines finished tokens into `out`
  bool gather_x;         // GEMM1 gathers its A rows from x (no x_perm)
  bool copy_rows;        // the swapped GEMM1 writes x_perm itself, block by block
  // the rows the swapped forward GEMMs read and GEMM2's output rows: the workspace's x_perm
  // and Y unless set (moe_expert_forward: the caller's buffers of rows_cap rows)
  const uint16_t* rows;
  uint16_t* y;
  int64_t rows_cap;
  uint16_t* out;         // layer output [T, d] (fused combine)
  bool gated;            // SwiGLU (W1, W3); false: squared ReLU on W1 alone
  // FP8 GEMM1: transposed E4M3 weights [E][dff][d] and their scales [E][dff]
  const uint8_t *W1q, *W3q;
  const float *wscale1, *wscale3;
};
cudaError_t launch_gemm_fwd1(const GemmCtx& c, cudaStream_t s);   // H = SwiGLU(Xp W1, Xp W3)
cudaError_t launch_gemm_fwd1_fp8(const GemmCtx& c, cudaStream_t s);  // H from E4M3 Xp, W1, W3
cudaError_t launch_gemm_fwd2(const GemmCtx& c, cudaStream_t s);   // Y = H W2
// the same two GEMMs with swapped operands (weight columns x row blocks), CTA pairs
cudaError_t launch_gemm_fwd1_swap(const GemmCtx& c, cudaStream_t s);
cudaError_t launch_gemm_fwd2_swap(const GemmCtx& c, cudaStream_t s);
// both swapped GEMMs in one persistent CTA-pair launch (GEMM2 of a block after its GEMM1)
cudaError_t launch_gemm_fwd_fused(const GemmCtx& c, cudaStream_t s);
cudaError_t launch_gemm_dh(const GemmCtx& c, cudaStream_t s);     // dA,dB from dO W2^T
// the same with swapped operands (W2 rows x row blocks), CTA pairs, one launch
cudaError_t launch_gemm_dh_swap(const GemmCtx& c, cudaStream_t s);
cudaError_t launch_gemm_dx(const GemmCtx& c, cudaStream_t s);     // dXp = dA W1^T + dB W3^T
// the same with swapped operands ([W1|W3] rows x row blocks), CTA pairs, one launch
cudaError_t launch_gemm_dx_swap(const GemmCtx& c, cudaStream_t s);
cudaError_t launch_gemm_dw2(const GemmCtx& c, cudaStream_t s);    // dW2 = H^T dO
cudaError_t launch_gemm_dw13(const GemmCtx& c, cudaStream_t s);   // dW1|dW3 = Xp^T [dA|dB]

// tensor-map encoder from the driver, resolved once
void* tensor_map_encoder();

}  // namespace moe
