// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// The expert stage is Linear -> SwiGLU -> Linear per expert (DeepSeek-V4 report reading,
// 10100.com, section on fine-grained EP overlap; report translation, itsolotime.com,
// section 1.4: gate, up and down projections, 6hd FLOP per token-expert pair).  Every kind
// below is one persistent, warp-specialised kernel:
//   warp 0      TMA producer (one lane): operand tiles -> a ring of shared-memory stages
//   warp 1      MMA issuer (one lane): tcgen05.mma 128 x BN x K into a TMEM accumulator
//               (bf16: K = 16; E4M3: K = 32; with CTA pairs, rank 0 issues M = 256)
//   warp 2      TMEM allocator
//   warps 4..7  epilogue: tcgen05.ld of the accumulator, activation, global stores (the
//               row-tile dH pair launch and kFwd1TW: warps 4..11, two per TMEM lane
//               quadrant, each taking half of the accumulator)
// Two TMEM accumulators alternate so the epilogue of tile i overlaps the MMAs of tile i+1.
// GEMM1 with rows gathered from x (opt-in) adds warp 2 as a second row-copying warp next to
// warp 0 and warp 3 (one lane) as the proxy-fence thread.
//
// Batch invariance and determinism (report translation, section 3; 10100.com reading):
// the tile shape (128 x BN x 64 bf16 or 128 E4M3 elements), the K order and therefore each
// output element's accumulation order are fixed by the model sizes alone, never by T or by
// the expert loads; there is no split-K and no atomic accumulation; which CTA computes a
// tile does not change its value.
//
// Row layout: the permuted rows of every expert start at a multiple of 128 (padded
// offsets), so each 128-row tile belongs to one expert; padding rows are masked in the
// epilogues (or written as zeros where a later K-over-rows GEMM reads them).
#pragma once

#include <cuda.h>

#include <atomic>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace moe {

enum GemmKind : int {
  kFwd1 = 0,  // H = bf16(silu(Xp W1) * (Xp W3)), optional fp32 A/B save   (rows x dff)
  kFwd2 = 1,  // Y = H W2 (bf16 rows, the combine's payload)                (rows x d)
  kDh = 2,    // dH = dO W2^T -> dA, dB (bf16) through the SwiGLU backward (rows x dff)
  kDx = 3,    // dXp = [dA|dB] [W1|W3]^T (fp32)                            (rows x d)
  kDw2 = 4,   // dW2[e] = H^T dO (fp32)                                    (dff x d)
  kDw13 = 5,  // [dW1|dW3][e] = Xp^T [dA|dB] (fp32)                         (d x 2dff)
  kFwd1F8 = 6,  // GEMM1 + SwiGLU on the FP8 payload: Xp and W1 / W3 in E4M3 (K-major), the
                // row and column scales applied in the epilogue                (rows x dff)
  // The forward GEMMs with the operands swapped: the expert's weight columns are the M
  // operand (256 per CTA pair, MN-major straight from the weights' row-major layout) and the
  // expert's permuted rows the N operand (a block of up to 256 rows, K-major), so a tile's N
  // follows the rows the block really holds (32, 64, 128 or 256) and an expert with few rows
  // costs few MMAs; heavy and light experts then share one persistent CTA-pair launch.
  kFwd1T = 7,   // H^T = [W1|W3]^T Xp^T -> SwiGLU -> H                      (dff x rows)
  kFwd2T = 8,   // Y^T = W2^T H^T (bf16 rows)                                (d x rows)
  // Both swapped GEMMs in one persistent launch: every GEMM1 tile first, then every GEMM2
  // tile; a GEMM2 tile of a row block starts loading H only when all GEMM1 tiles of that
  // block have stored theirs (a per-block counter), so GEMM2 of the first blocks runs while
  // GEMM1 of the last ones still computes, and one launch's ramp and tail serve both.
  kFwdT = 9,
  // The backward's dX rows swapped the same way: the expert's W1 / W3 rows (d of them, 256
  // per CTA pair) are the M operand, K-major as stored ([d][dff]: K = dff contiguous), and a
  // block of up to 256 rows of [dA|dB] the N operand, so every expert runs on CTA pairs in
  // one launch whatever its tile count.
  kDxT = 10,    // dXp^T = [W1|W3] [dA|dB]^T (fp32 rows)                     (d x rows)
  // and dH: the expert's W2 rows (d_ff of them, K = d contiguous) as the M operand, a block of
  // dO rows as N; the epilogue applies the saved multipliers per (row, d_ff column)
  kDhT = 11,    // dH^T = W2 dO^T -> dA, dB (bf16)                            (dff x rows)
  // kFwd1T with 8 epilogue warps (two per TMEM lane quadrant, alternate 32-row chunks) and 5
  // stages: its SwiGLU epilogue keeps up with short main loops of full row blocks (K = d of
  // 2048: GEMM1 of the T=4096, d=2048, E=64, top-6, d_ff=1024 layer 0.238 -> 0.187 ms on
  // GB300; the T=16384, d=7168, E=256 layer 5.71 -> 5.63 ms), while layers of mostly light
  // experts, which stream weights, keep the sixth stage of kFwd1T (T=128 and T=1024 of the
  // d=7168 layer: 2.23 vs 2.28 ms and 1.029 vs 1.059 ms)
  kFwd1TW = 12,
};

template <int KIND>
struct KindTraits {
  static constexpr bool kRowsM = (KIND <= kDx || KIND == kFwd1F8);  // M = permuted rows
  static constexpr bool kSwap = (KIND == kFwd1T || KIND == kFwd2T || KIND == kFwdT ||
                                 KIND == kDxT || KIND == kDhT || KIND == kFwd1TW);  // N = rows
  static constexpr int kAmn =
      (KIND == kDw2 || KIND == kDw13 || (kSwap && KIND != kDxT && KIND != kDhT)) ? 1 : 0;
  static constexpr int kBmn = (KIND == kDh || KIND == kDx || KIND == kFwd1F8 || kSwap) ? 0 : 1;
  // K blocks (of 64) per pipeline stage: two for the swapped GEMM2 and dX (3 stages of 64 KB:
  // one producer / MMA-issuer handshake per 128 K), one elsewhere.  Measured on GB300 against
  // one for every swapped kind, 3 alternations: GEMM2 of the T=16384, d=7168, E=256, top-8,
  // d_ff=2048 layer 2.87 -> 2.77 ms, dX of T=8192, d=4096, E=128, top-8, d_ff=1536 1.171 ->
  // 1.159 ms; GEMM1 (5.61 -> 5.57 there, but +0.6% at T=2048, +1.6% at T=128) and dH (+2.7%)
  // keep one.  Bitwise the same results.
  static constexpr int kKPS = (KIND == kFwd2T || KIND == kDxT) ? 2 : 1;
};

// Epilogue warps of a launch: 4, one per TMEM lane quadrant, or 8 for the row-tile dH pair
// launch, whose epilogue (the saved multipliers of dA and dB read from HBM, 12 bytes of
// traffic per accumulator element) is slower than its MMAs with 4 warps, and for kFwd1TW;
// two warps then share a lane quadrant and split the accumulator.  (The swapped dH runs
// faster with 4 warps and the sixth stage they leave room for: measured on GB300, 0.697 ->
// 0.662 ms at the fwd_bwd workload, T=8192, d=4096, E=128, top-8, d_ff=1536.)
template <int KIND, bool PAIR>
struct EpiCfg {
  static constexpr int kWarps = ((KIND == kDh || KIND == kFwd1TW) && PAIR) ? 8 : 4;
  static constexpr int kThreads = 128 + 32 * kWarps;  // + producer, MMA, TMEM, spare warps
};

struct GemmParams {
  // expert activation: 1 = SwiGLU (W1 and W3), 0 = squared ReLU on W1 alone (no gate
  // projection): GEMM1 tiles then hold 256 columns of A = Xp W1, dH gives dA only, dX and
  // dW1 take K = N = d_ff
  int gated;
  // FP8 GEMM1: per-token row scales [T] and per-(expert, column) weight scales [E, dff]
  const float* xscale;
  const float* wscale1;
  const float* wscale3;
  // fp32 output tiles written by TMA stores (32 x 32 boxes, 128-byte swizzle) when tma_store:
  // c0 = out0, c1 = out1
  CUtensorMap mapC0, mapC1;
  int tma_store;
  int E, d, dff;
  int nb;   // BN blocks along N
  int nkb;  // 64-wide K blocks (row-grouped kinds)
  int mb;   // 128-row blocks along M (K-over-rows kinds)
  const int32_t* n_mt;
  const int32_t* mt_expert;
  const int32_t* mt_row0;
  const int32_t* counts;
  const int32_t* poff;
  void* out0;
  void* out1;
  float* save_a;
  float* save_b;
  int save_ab;
  DevErr* err;
  uint64_t wait_ns;
  int debug_flags;
  int64_t max_tiles;  // tiles the workspace tables can describe
  int64_t rows_cap;   // permuted rows allocated in the workspace
  const int32_t* n_pt;       // 256-row pair tiles (two 128-row tiles of one expert)
  const int32_t* pt_expert;
  const int32_t* pt_row0;
  int M;                     // M extent of the K-over-rows kinds (d or d_ff)
  // GEMM2 with the combine fused in (see combine_segment)
  int fuse_combine;
  // GEMM1 reading its A rows straight from x (rows gathered by token with cp.async)
  int gather_x;
  const uint16_t* gather_src;  // x [T, d] bf16
  const int32_t* perm;       // permuted row -> pair t*k + j
  const int32_t* pos;        // pair -> permuted row
  const float* gate;         // [T, k]
  int32_t* seg_count;        // [T, nb]: rows of (token, N block) written so far
  uint16_t* comb_out;        // [T, d] bf16 layer output
  int k;
  // swapped forward kinds: the table of 256-row blocks (expert, first row) and tensor maps of
  // the row operand with boxes of 16, 32, 64 and 128 rows (the rows a CTA takes of a block)
  const int32_t* n_st;
  const int32_t* st_expert;
  const int32_t* st_row0;
  CUtensorMap mapR[4];
  // both GEMMs in one launch (kFwdT): GEMM2's column blocks and K blocks, the row maps of H
  // (GEMM2's N operand), and the per-row-block count of GEMM1 tile halves (one per CTA of a
  // pair) whose H rows are stored
  int nb2, nkb2;
  CUtensorMap mapR2[4];
  int32_t* done1;
  // swapped GEMM1 copying its own rows: warps 2 and 3 of every CTA write
  // copy_dst[r] = gather_src[perm[r] / k] block by block, counting each block's finished
  // units in done1; a tile's loads wait for its block
  int copy_rows;
  uint16_t* copy_dst;
};

// Row copy units of a 256-row block (4 rows each).
constexpr int kCopyUnits = 64;

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB
// L2 eviction priority of the operand loads of the row-grouped forward GEMMs: 0 = default,
// 1 = evict_last, 2 = evict_first.  A = permuted rows, B = expert weights.
constexpr int kL2HintA = 0;
constexpr int kL2HintB = 1;

template <int BN, bool PAIR = false, int EPI_WARPS = 4, int KPS = 1>
struct GemmCfg {
  // a CTA pair holds half of the B tile in each CTA
  static constexpr int kBLocal = PAIR ? BN / 2 : BN;
  static constexpr uint32_t kBBytes = kBLocal * kBK * 2;
  // one K block's A and B tiles; a stage holds KPS of them back to back
  static constexpr uint32_t kSubBytes = kABytes + kBBytes;
  // 32 KB of K blocks: 6 (5 with 8 epilogue warps); 48 KB: 4; divided among KPS per stage
  static constexpr int kStages =
      ((kSubBytes <= 32768) ? (EPI_WARPS > 4 ? 5 : 6) : 4) / KPS;
  static_assert(kStages >= 2, "a ring of at least two stages");
  static constexpr uint32_t kStageBytes = KPS * kSubBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;
  // full, empty, tfull x2, tempty x2, drain, gathered-rows landed
  static constexpr int kBars = 3 * kStages + 5;
  // one 1024-aligned 5 KB region per epilogue warp: a 32 x 33 fp32 transpose buffer, or the
  // 32 x 32 fp32 staging box of a TMA store
  static constexpr size_t kEpiWarpBytes = 5120;
  static constexpr size_t kEpiBytes = EPI_WARPS * kEpiWarpBytes;
  // + 128 bytes: TMEM address, abort flag, fill counters and the two rings of per-fill
  // load bytes (this CTA's and, with pairs, the peer's)
  static constexpr size_t kSmemBytes = static_cast<size_t>(kStages) * kStageBytes + 1024 +
                                       kEpiBytes + 8 * kBars + 128;
  static_assert(kStageBytes % 1024 == 0, "stages keep the epilogue regions 1024-aligned");
  static_assert(kSmemBytes <= 232448, "fits the opt-in shared memory of a CTA (227 KB)");
};

struct TileInfo {
  int e;      // expert
  int row0;   // first permuted row (row-grouped) / first K row (K-over-rows)
  int nvalid; // valid rows of the tile (row-grouped)
  int m0;     // first M index (K-over-rows)
  int n0;     // first N index
  int nk;     // number of 64-wide K blocks
  int mvalid; // valid M rows of this CTA's 128 (K-over-rows kinds)
  int nseg;   // rows of this CTA inside the expert's padded row segment (rows-grouped kinds);
              // with PAIR the second half of an expert's last tile can lie past the segment,
              // on the next expert's rows, and must not be written
  int box;    // swapped kinds: rows of the block each CTA loads (16, 32, 64 or 128); N = 2 box
  int part;   // swapped kinds: 1 = GEMM1 (+ SwiGLU) tile, 2 = GEMM2 tile
  int st;     // swapped kinds: index of the row block in the block table
  bool bad;   // tile tables out of range: every role skips the tile
};

// Tile -> (expert, rows, N block, K blocks) for this CTA.  With PAIR a tile is 256 rows of
// one expert (rows-grouped kinds: two consecutive 128-row tiles; K-over-rows kinds: 256 rows
// of M) and CTA rank r of the pair owns rows [128 r, 128 r + 128) of it.
template <int KIND, int BN, bool PAIR>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int tile, int rank) {
  TileInfo ti;
  ti.box = kBM;
  if constexpr (KindTraits<KIND>::kRowsM) {
    const int mt = tile / p.nb;
    ti.n0 = (tile % p.nb) * BN;
    if constexpr (PAIR) {
      ti.e = p.pt_expert[mt];
      const int r0 = p.pt_row0[mt];
      ti.bad = ti.e < 0 || ti.e >= p.E || r0 < 0 || r0 + kBM > p.rows_cap;
      ti.row0 = r0 + kBM * rank;
    } else {
      ti.e = p.mt_expert[mt];
      ti.row0 = p.mt_row0[mt];
      ti.bad = ti.e < 0 || ti.e >= p.E || ti.row0 < 0 || ti.row0 + kBM > p.rows_cap;
    }
    ti.nvalid = ti.bad ? 0 : p.poff[ti.e] + p.counts[ti.e] - ti.row0;
    ti.nseg = ti.bad ? 0 : p.poff[ti.e + 1] - ti.row0;
    ti.m0 = 0;
    ti.nk = p.nkb;
    ti.mvalid = kBM;
  } else if constexpr (KindTraits<KIND>::kSwap) {
    // a block of up to 256 rows of one expert x one block of weight columns: 128 h columns
    // (64 per CTA, each with its W1 and W3 column) for GEMM1, 256 without the gate
    // projection or for GEMM2 (128 per CTA)
    // part: 1 GEMM1, 2 GEMM2, 3 the backward's dX, 4 its dH
    int part = KIND == kFwd2T ? 2 : (KIND == kDxT ? 3 : (KIND == kDhT ? 4 : 1)), t = tile,
        nbp = p.nb, nk = p.nkb;
    if constexpr (KIND == kFwdT) {
      const int n1 = p.n_st[0] * p.nb;  // GEMM1 tiles come first
      if (tile >= n1) {
        part = 2;
        t = tile - n1;
        nbp = p.nb2;
        nk = p.nkb2;
      }
    }
    const int st = t / nbp;
    ti.part = part;
    ti.st = st;
    ti.n0 = (t % nbp) * ((part == 1 && p.gated) ? 128 : 256);
    ti.e = p.st_expert[st];
    ti.row0 = p.st_row0[st];
    ti.bad = ti.e < 0 || ti.e >= p.E || ti.row0 < 0 || ti.row0 >= p.rows_cap;
    ti.nvalid = 0;
    ti.nseg = 0;
    if (!ti.bad) {
      const int nv = p.poff[ti.e] + p.counts[ti.e] - ti.row0;
      const int ns = p.poff[ti.e + 1] - ti.row0;
      ti.nvalid = nv < 2 * kBM ? nv : 2 * kBM;
      ti.nseg = ns < 2 * kBM ? ns : 2 * kBM;
      ti.bad = ti.nvalid < 1 || ti.nseg < ti.nvalid || ti.row0 + ti.nseg > p.rows_cap;
      if (ti.bad) ti.nvalid = ti.nseg = 0;
    }
    const int half = (ti.nvalid + 1) / 2;
    ti.box = half <= 16 ? 16 : (half <= 32 ? 32 : (half <= 64 ? 64 : 128));
    ti.m0 = 0;
    ti.nk = nk;
    ti.mvalid = kBM;
  } else {
    const int per_e = p.mb * p.nb;
    ti.e = tile / per_e;
    const int rem = tile % per_e;
    ti.m0 = (rem / p.nb) * (PAIR ? 2 * kBM : kBM) + (PAIR ? kBM * rank : 0);
    ti.n0 = (rem % p.nb) * BN;
    ti.row0 = p.poff[ti.e];
    ti.nk = (p.poff[ti.e + 1] - p.poff[ti.e]) / kBK;
    ti.nvalid = kBM;
    ti.nseg = kBM;
    ti.mvalid = p.M - ti.m0 < kBM ? (p.M - ti.m0 > 0 ? p.M - ti.m0 : 0) : kBM;
    ti.bad = ti.row0 < 0 || ti.nk < 0 || ti.row0 + ti.nk * kBK > p.rows_cap;
  }
  return ti;
}

__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + expf(-a)); }

// What the forward saves for the backward's dH epilogue, per h element: the multipliers of dh
// in dA = dh * b silu'(a) and dB = dh * silu(a), with silu'(a) = s (1 + a (1 - s)) and
// s = sigmoid(a); without the gate projection dA = dh * 2 relu(a).  The backward then needs one
// multiply per output instead of an exp and a division.
__device__ __forceinline__ void swiglu_bwd_mults(float a, float b, float* ma, float* mb) {
  const float sg = 1.0f / (1.0f + expf(-a));
  *ma = b * (sg * (1.0f + a * (1.0f - sg)));
  *mb = a * sg;
}
__device__ __forceinline__ float relu2_bwd_mult(float a) { return 2.0f * fmaxf(a, 0.0f); }

__device__ __forceinline__ void st_zero32(void* p) {  // 32 bytes of zeros
  const uint4 z = make_uint4(0u, 0u, 0u, 0u);
  st_v4(p, z);
  st_v4(static_cast<char*>(p) + 16, z);
}
__device__ __forceinline__ void st_f32x16(float* p, const float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    st_v4(p + 4 * i, make_uint4(__float_as_uint(v[4 * i]), __float_as_uint(v[4 * i + 1]),
                                __float_as_uint(v[4 * i + 2]), __float_as_uint(v[4 * i + 3])));
}
__device__ __forceinline__ void st_bf16x16(uint16_t* p, const float (&v)[16]) {
  st_v4(p, make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                      pack_bf16x2(v[6], v[7])));
  st_v4(p + 8, make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                          pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15])));
}
__device__ __forceinline__ void ld_f32x16(const float* p, float (&v)[16]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 u = ld_v4(p + 4 * i);
    v[4 * i] = __uint_as_float(u.x);
    v[4 * i + 1] = __uint_as_float(u.y);
    v[4 * i + 2] = __uint_as_float(u.z);
    v[4 * i + 3] = __uint_as_float(u.w);
  }
}

// ---------------------------------------------------------------------------- fused combine
// GEMM2 can run the combine itself.  When an epilogue warp has stored its 32 rows of a tile,
// each row's lane counts one more finished row of its (token, N block) segment (integer
// atomics: exact whatever their order).  A lane that brings a segment to k rows has the
// whole warp combine it right away: out[t, cols] = bf16(sum_j gate[t,j] * Y[pos[t,j], cols])
// over the bf16 output rows Y
// with fp32 fused multiply-adds in slot order, the same arithmetic as the stand-alone
// combine, so the result is bitwise identical.  The combine of earlier experts' tokens thus
// runs under the MMAs of later experts (the accumulator is double-buffered, so the epilogue
// has a whole tile's main loop to finish).
template <int BN>
__device__ __forceinline__ void combine_segment(const GemmParams& p, int seg, int lane) {
  constexpr int CPL = BN / 32;  // columns per lane (8 or 4)
  const int t = seg / p.nb, nblk = seg % p.nb;
  int row = 0;
  float g = 0.0f;
  if (lane < p.k) {
    row = p.pos[static_cast<int64_t>(t) * p.k + lane];
    g = p.gate[static_cast<int64_t>(t) * p.k + lane];
  }
  const int col = nblk * BN + lane * CPL;
  const uint16_t* Y = static_cast<const uint16_t*>(p.out0);  // bf16 output rows
  float4 y[kMaxK][CPL / 4];
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    const int rj = __shfl_sync(0xFFFFFFFFu, row, j);
    if (j < p.k) {
      const uint16_t* src = Y + static_cast<int64_t>(rj) * p.d + col;
#pragma unroll
      for (int c4 = 0; c4 < CPL / 4; ++c4) {
        const uint2 u = __ldcg(reinterpret_cast<const uint2*>(src) + c4);
        y[j][c4] = make_float4(bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y));
      }
    }
  }
  float acc[CPL];
#pragma unroll
  for (int c = 0; c < CPL; ++c) acc[c] = 0.0f;
#pragma unroll
  for (int j = 0; j < kMaxK; ++j) {
    const float gj = __shfl_sync(0xFFFFFFFFu, g, j);
    if (j < p.k) {
#pragma unroll
      for (int c4 = 0; c4 < CPL / 4; ++c4) {
        acc[4 * c4 + 0] = __fmaf_rn(gj, y[j][c4].x, acc[4 * c4 + 0]);
        acc[4 * c4 + 1] = __fmaf_rn(gj, y[j][c4].y, acc[4 * c4 + 1]);
        acc[4 * c4 + 2] = __fmaf_rn(gj, y[j][c4].z, acc[4 * c4 + 2]);
        acc[4 * c4 + 3] = __fmaf_rn(gj, y[j][c4].w, acc[4 * c4 + 3]);
      }
    }
  }
  uint16_t* o = p.comb_out + static_cast<int64_t>(t) * p.d + col;
  if constexpr (CPL == 8) {
    st_v4(o, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                        pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
  } else {
    *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
  }
}

// 32 consecutive accumulator columns of this lane's row
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  float a[16], b[16];
  tmem_ld16x2(taddr, taddr + 16, a, b);
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    v[i] = a[i];
    v[16 + i] = b[i];
  }
}

// Each epilogue warp owns 32 accumulator rows (one per lane) and writes them 32 columns at a
// time.  A lane holds 32 consecutive values of its own row; the warp transposes the 32 x 32
// chunk through a padded shared buffer (32 x 33 floats, conflict-free both ways) so that every
// global store instruction writes whole 128-byte lines of 4 (fp32) or 8 (bf16) rows.
// Rows [0, nstore) of the chunk are written; base points at (row 0, first column of chunk).
template <bool BF16>
__device__ __forceinline__ void store_chunk(float* buf, const float (&v)[32], char* base,
                                            int64_t row_bytes, int nstore, int lane) {
#pragma unroll
  for (int c = 0; c < 32; ++c) buf[lane * 33 + c] = v[c];
  __syncwarp();
  if constexpr (BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int row = 8 * i + (lane >> 2), c0 = (lane & 3) * 8;
      const float* src = buf + row * 33 + c0;
      if (row < nstore)
        st_v4(base + row * row_bytes + c0 * 2,
              make_uint4(pack_bf16x2(src[0], src[1]), pack_bf16x2(src[2], src[3]),
                         pack_bf16x2(src[4], src[5]), pack_bf16x2(src[6], src[7])));
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int row = 4 * i + (lane >> 3), c0 = (lane & 7) * 4;
      const float* src = buf + row * 33 + c0;
      if (row < nstore)
        st_v4(base + row * row_bytes + c0 * 4,
              make_uint4(__float_as_uint(src[0]), __float_as_uint(src[1]),
                         __float_as_uint(src[2]), __float_as_uint(src[3])));
    }
  }
  __syncwarp();
}

// 32 rows (one per lane) x 32 fp32 columns to global memory with one TMA store of box (x, y).
// The warp writes the box into its staging region in the 128-byte-swizzled layout the tensor
// map expects (16-byte chunk c of row r at chunk c ^ (r & 7)), then lane 0 issues the store.
// Before the warp rewrites the region, lane 0 waits until the previous store has read it.
__device__ __forceinline__ void store_chunk_tma(uint32_t stage, const float (&v)[32],
                                                const CUtensorMap* map, int x, int y, int lane) {
  if (lane == 0) bulk_wait_read_all();
  __syncwarp();
  const uint32_t row = stage + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t dst = row + static_cast<uint32_t>((c ^ (lane & 7)) * 16);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst),
                 "r"(__float_as_uint(v[4 * c])), "r"(__float_as_uint(v[4 * c + 1])),
                 "r"(__float_as_uint(v[4 * c + 2])), "r"(__float_as_uint(v[4 * c + 3]))
                 : "memory");
  }
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, stage, x, y);
    bulk_commit();
  }
}

// Epilogue of one tile for one epilogue warp (rows q*32 .. q*32+31 of the accumulator).
// `tacc` is the warp's TMEM address (lane base q*32, accumulator column 0); `r` = q*32 + lane.
// `part` of `nparts` (dH with 8 epilogue warps: 2) selects the warp's share of the chunks.
template <int KIND, int BN>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const TileInfo& ti,
                                              uint32_t tacc, int q, int lane, float* buf,
                                              uint32_t stage, int part, int nparts) {
  const int r = q * 32 + lane;
  const bool valid = r < ti.nvalid;
  const int w0 = q * 32;  // first row of this warp
  auto clamp_rows = [&](int n) { return n - w0 < 0 ? 0 : (n - w0 > 32 ? 32 : n - w0); };
  if constexpr (KIND == kFwd1 || KIND == kFwd1F8) {
    if (KIND == kFwd1 && !p.gated) {
      // h = relu(a)^2 over the tile's 256 accumulator columns (h columns n0 ..)
      const int64_t row0 = ti.row0 + w0;
      char* H = reinterpret_cast<char*>(static_cast<uint16_t*>(p.out0) + row0 * p.dff + ti.n0);
      const int nstore = clamp_rows(ti.nseg);      // pad rows are written as zeros
      const int nsave = clamp_rows(ti.nvalid);
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        float a[32], h[32];
        tmem_ld32(tacc + ch * 32, a);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float rl = fmaxf(a[i], 0.0f);
          h[i] = valid ? rl * rl : 0.0f;
        }
        store_chunk<true>(buf, h, H + ch * 64, 2ll * p.dff, nstore, lane);
        if (p.save_ab) {
          // dA's multiplier 2 relu(a)
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = relu2_bwd_mult(a[i]);
          char* SA = reinterpret_cast<char*>(p.save_a + row0 * p.dff + ti.n0 + ch * 32);
          store_chunk<false>(buf, a, SA, 4ll * p.dff, nsave, lane);
        }
      }
      return;
    }
    constexpr int HALF = BN / 2;
    const int c0 = ti.n0 / 2;  // h column of this tile's first accumulator column
    const int64_t row0 = ti.row0 + w0;
    char* H = reinterpret_cast<char*>(static_cast<uint16_t*>(p.out0) + row0 * p.dff + c0);
    const int nstore = clamp_rows(ti.nseg);      // pad rows are written as zeros
    const int nsave = clamp_rows(ti.nvalid);
    float rscale = 1.0f;  // FP8: the row's (token's) scale
    if (KIND == kFwd1F8 && valid) rscale = p.xscale[p.perm[ti.row0 + r] / p.k];
#pragma unroll 1
    for (int ch = 0; ch < HALF / 32; ++ch) {
      float a[32], b[32], h[32];
      tmem_ld32(tacc + ch * 32, a);
      tmem_ld32(tacc + HALF + ch * 32, b);
      if constexpr (KIND == kFwd1F8) {
        // dequantize: A = (sum of E4M3 products) * row scale * column scale
        const float* s1 = p.wscale1 + static_cast<int64_t>(ti.e) * p.dff + c0 + ch * 32;
        const float* s3 = p.wscale3 + static_cast<int64_t>(ti.e) * p.dff + c0 + ch * 32;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          a[i] *= rscale * __ldg(s1 + i);
          b[i] *= rscale * __ldg(s3 + i);
        }
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = valid ? silu_f(a[i]) * b[i] : 0.0f;
      store_chunk<true>(buf, h, H + ch * 64, 2ll * p.dff, nstore, lane);
      if (p.save_ab) {
        // dA's and dB's multipliers b silu'(a) and silu(a), in place of a and b
#pragma unroll
        for (int i = 0; i < 32; ++i) swiglu_bwd_mults(a[i], b[i], &a[i], &b[i]);
        char* SA = reinterpret_cast<char*>(p.save_a + row0 * p.dff + c0 + ch * 32);
        char* SB = reinterpret_cast<char*>(p.save_b + row0 * p.dff + c0 + ch * 32);
        store_chunk<false>(buf, a, SA, 4ll * p.dff, nsave, lane);
        store_chunk<false>(buf, b, SB, 4ll * p.dff, nsave, lane);
      }
    }
  } else if constexpr (KIND == kFwd2 || KIND == kDx) {
    const int64_t row0 = ti.row0 + w0;
    const int nstore = clamp_rows(ti.nvalid);
    if constexpr (KIND == kFwd2) {
      // bf16 output rows (the combine's payload), through the bf16 transpose
      char* out = reinterpret_cast<char*>(static_cast<uint16_t*>(p.out0) + row0 * p.d + ti.n0);
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        float v[32];
        tmem_ld32(tacc + ch * 32, v);
        store_chunk<true>(buf, v, out + ch * 64, 2ll * p.d, nstore, lane);
      }
    } else {
      // fp32 dX rows.  TMA stores write all 32 rows of the warp: rows past the expert's count
      // are padding rows of its own segment (zeros: their A rows are zero), which nothing reads
      char* out = reinterpret_cast<char*>(static_cast<float*>(p.out0) + row0 * p.d + ti.n0);
      const bool tma = p.tma_store && clamp_rows(ti.nseg) == 32;
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        float v[32];
        tmem_ld32(tacc + ch * 32, v);
        if (tma) {
          store_chunk_tma(stage, v, &p.mapC0, ti.n0 + ch * 32, static_cast<int>(row0), lane);
        } else {
          if (p.tma_store && lane == 0) bulk_wait_read_all();  // the region may still be read
          __syncwarp();
          store_chunk<false>(buf, v, out + ch * 128, 4ll * p.d, nstore, lane);
        }
      }
    }
    if constexpr (KIND == kFwd2) {
      if (p.fuse_combine) {
        __threadfence();  // this lane's row stores are visible device-wide ...
        __syncwarp();     // ... before any lane of the warp counts its row as finished
        int seg = -1;
        if (valid) {
          const int pair = p.perm[ti.row0 + r];
          seg = (pair / p.k) * p.nb + ti.n0 / BN;
          if (atomicAdd(&p.seg_count[seg], 1) != p.k - 1) seg = -1;
        }
        unsigned ready = __ballot_sync(0xFFFFFFFFu, seg >= 0);
        if (ready) __threadfence();  // the other rows of those segments are visible
        while (ready) {
          const int src = __ffs(ready) - 1;
          ready &= ready - 1;
          combine_segment<BN>(p, __shfl_sync(0xFFFFFFFFu, seg, src), lane);
        }
      }
    }
  } else if constexpr (KIND == kDh) {
    // The warp puts its 32 x 32 chunk of dH through the padded shared buffer, then works row
    // by row: 8 lanes per row read the row's saved multipliers of dA and dB (16 bytes each,
    // whole 128-byte lines), multiply and store dA and dB (8 bytes each).
    const int64_t row0 = ti.row0 + w0;
    uint16_t* dA0 = static_cast<uint16_t*>(p.out0) + row0 * (2 * p.dff) + ti.n0;
    const float* sa0 = p.save_a + row0 * p.dff + ti.n0;
    const float* sb0 = p.save_b + row0 * p.dff + ti.n0;
    const int nstore = clamp_rows(ti.nseg);      // pad rows are written as zeros
    const int nval = clamp_rows(ti.nvalid);
    const int rsub = lane >> 3, c4 = (lane & 7) * 4;
    const int ch_end = (part + 1) * (BN / 32) / nparts;
#pragma unroll 1
    for (int ch = part * (BN / 32) / nparts; ch < ch_end; ++ch) {
      // all 16 loads of the chunk in flight first; the accumulator read and the shared
      // transpose run under their latency
      uint4 ua[8], ub[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + rsub;
        if (rr < nval) {
          ua[i] = ld_v4(sa0 + rr * p.dff + ch * 32 + c4);
          ub[i] = p.gated ? ld_v4(sb0 + rr * p.dff + ch * 32 + c4) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float dh[32];
      tmem_ld32(tacc + ch * 32, dh);
#pragma unroll
      for (int c = 0; c < 32; ++c) buf[lane * 33 + c] = dh[c];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + rsub;
        if (rr < nstore) {
          float da[4] = {0.0f, 0.0f, 0.0f, 0.0f}, db[4] = {0.0f, 0.0f, 0.0f, 0.0f};
          if (rr < nval) {
            const float av[4] = {__uint_as_float(ua[i].x), __uint_as_float(ua[i].y),
                                 __uint_as_float(ua[i].z), __uint_as_float(ua[i].w)};
            const float bv[4] = {__uint_as_float(ub[i].x), __uint_as_float(ub[i].y),
                                 __uint_as_float(ub[i].z), __uint_as_float(ub[i].w)};
            // the forward saved dA's and dB's multipliers (b silu'(a) and silu(a), or
            // 2 relu(a) without the gate projection) in place of a and b
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float g = buf[rr * 33 + c4 + q];
              da[q] = g * av[q];
              db[q] = g * bv[q];
            }
          }
          uint16_t* o = dA0 + rr * (2 * p.dff) + ch * 32 + c4;
          *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(da[0], da[1]), pack_bf16x2(da[2], da[3]));
          if (p.gated)
            *reinterpret_cast<uint2*>(o + p.dff) =
                make_uint2(pack_bf16x2(db[0], db[1]), pack_bf16x2(db[2], db[3]));
        }
      }
      __syncwarp();
    }
  } else {
    // K-over-rows kinds: output rows m0 + w0 .. of expert e's weight gradient.
    char* out;
    int64_t row_bytes;
    if constexpr (KIND == kDw2) {
      row_bytes = 4ll * p.d;
      out = reinterpret_cast<char*>(static_cast<float*>(p.out0) +
                                    (static_cast<int64_t>(ti.e) * p.dff + ti.m0 + w0) * p.d + ti.n0);
    } else {
      row_bytes = 4ll * p.dff;
      const bool first = ti.n0 < p.dff;
      float* basep = static_cast<float*>(first ? p.out0 : p.out1);
      out = reinterpret_cast<char*>(basep + (static_cast<int64_t>(ti.e) * p.d + ti.m0 + w0) * p.dff +
                                    (first ? ti.n0 : ti.n0 - p.dff));
    }
    const int nstore = clamp_rows(ti.mvalid);
    const CUtensorMap* cmap = &p.mapC0;
    int cx = ti.n0, cy;
    if constexpr (KIND == kDw2) {
      cy = ti.e * p.dff + ti.m0 + w0;
    } else {
      cy = ti.e * p.d + ti.m0 + w0;
      if (ti.n0 >= p.dff) {
        cmap = &p.mapC1;
        cx = ti.n0 - p.dff;
      }
    }
#pragma unroll 1
    for (int ch = 0; ch < BN / 32; ++ch) {
      float v[32];
      if (ti.nk > 0) {
        tmem_ld32(tacc + ch * 32, v);
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      }
      if (p.tma_store && nstore == 32) {
        store_chunk_tma(stage, v, cmap, cx + ch * 32, cy, lane);
      } else {
        if (p.tma_store && lane == 0) bulk_wait_read_all();
        __syncwarp();
        store_chunk<false>(buf, v, out + ch * 128, row_bytes, nstore, lane);
      }
    }
  }
}

// Epilogue of the swapped forward kinds for one epilogue warp: TMEM lanes are this CTA's
// weight columns (one per lane of warp q's quadrant), TMEM columns the block's rows.  The
// warp walks the rows 32 at a time; for each row, the 32 lanes write 32 consecutive output
// columns.
//  * kFwd1T with W3: lanes 0-63 hold A = Xp W1 and lanes 64-127 B = Xp W3 for the same 64 h
//    columns, so warp q (A) and warp q + 2 (B) swap their 32 x 32 chunks through shared
//    memory and each finishes half of the chunk's rows: h = bf16(silu(A) B).  Padding rows of
//    the expert's segment get h = 0 (a later K-over-rows GEMM reads them).
//  * kFwd1T without W3: h = bf16(relu(A)^2) over 128 W1 columns.
//  * kDxT: fp32 dX rows over 128 d columns (as kFwd2T, columns past d are not stored).
//  * kDhT: dA and dB rows (bf16) over 128 d_ff columns; where a launch runs two warps per lane
//    quadrant, they take alternate 32-row chunks (`half` of `nhalves`).
//  * kFwd2T: Y rows (bf16) over 128 W2 columns (columns past d, when d is not a multiple of
//    256, are neither loaded as real data nor stored).
template <int KIND>
__device__ __forceinline__ void epilogue_swap(const GemmParams& p, const TileInfo& ti,
                                              uint32_t tacc, int q, int lane, float* mine,
                                              const float* partner, int rank, int half,
                                              int nhalves) {
  const int nch = (ti.nvalid + 31) / 32;
  const int64_t row0 = ti.row0;
  if constexpr (KIND == kDhT) {
    // Each 32 x 32 chunk (lane = d_ff column, register = row) goes through `mine` transposed;
    // then 8 lanes per row read the row's saved multipliers of dA and dB (16 bytes each, whole
    // 128-byte lines), multiply and store 8 bytes of dA and of dB.  Padding rows of the
    // expert's segment get zeros (dW1 / dW3 read them as K rows).
    const int c0 = ti.n0 + 128 * rank + 32 * q;  // first d_ff column of this warp
    if (c0 >= p.dff) return;  // warp-uniform: d_ff % 256 == 128, rank 1's last columns
    uint16_t* dA0 = static_cast<uint16_t*>(p.out0) + row0 * (2 * p.dff) + c0;
    const float* sa0 = p.save_a + row0 * p.dff + c0;
    const float* sb0 = p.save_b + row0 * p.dff + c0;
    const int rsub = lane >> 3, c4 = (lane & 7) * 4;
#pragma unroll 1
    for (int ch = half; ch < nch; ch += nhalves) {
      const int nval = ti.nvalid - ch * 32, nstore = ti.nseg - ch * 32;  // may exceed 32
      // all 16 loads of the chunk in flight first; the accumulator read and the shared
      // transpose run under their latency
      uint4 ua[8], ub[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int64_t r = ch * 32 + 4 * i + rsub;
        ua[i] = ub[i] = make_uint4(0u, 0u, 0u, 0u);
        if (4 * i + rsub < nval) {
          ua[i] = ld_v4(sa0 + r * p.dff + c4);
          if (p.gated) ub[i] = ld_v4(sb0 + r * p.dff + c4);
        }
      }
      float v[32];
      tmem_ld32(tacc + ch * 32, v);
#pragma unroll
      for (int j = 0; j < 32; ++j) mine[j * 33 + lane] = v[j];
      __syncwarp();
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + rsub;
        if (rr < nstore) {
          // rows past the valid ones multiply zeros (their saved multipliers are not read)
          const float av[4] = {__uint_as_float(ua[i].x), __uint_as_float(ua[i].y),
                               __uint_as_float(ua[i].z), __uint_as_float(ua[i].w)};
          const float bv[4] = {__uint_as_float(ub[i].x), __uint_as_float(ub[i].y),
                               __uint_as_float(ub[i].z), __uint_as_float(ub[i].w)};
          float da[4], db[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const float g = mine[rr * 33 + c4 + u];
            da[u] = rr < nval ? g * av[u] : 0.0f;
            db[u] = rr < nval ? g * bv[u] : 0.0f;
          }
          uint16_t* o = dA0 + (ch * 32 + rr) * static_cast<int64_t>(2 * p.dff) + c4;
          *reinterpret_cast<uint2*>(o) =
              make_uint2(pack_bf16x2(da[0], da[1]), pack_bf16x2(da[2], da[3]));
          if (p.gated)
            *reinterpret_cast<uint2*>(o + p.dff) =
                make_uint2(pack_bf16x2(db[0], db[1]), pack_bf16x2(db[2], db[3]));
        }
      }
      __syncwarp();  // the stores' reads of `mine` are done before the next chunk rewrites it
    }
    // padding rows of the segment past the last chunk: 4 rows per instruction
    const uint2 z = make_uint2(0u, 0u);
    for (int r = nch * 32 + 4 * half + rsub; r < ti.nseg; r += 4 * nhalves) {
      uint16_t* o = dA0 + r * static_cast<int64_t>(2 * p.dff) + c4;
      *reinterpret_cast<uint2*>(o) = z;
      if (p.gated) *reinterpret_cast<uint2*>(o + p.dff) = z;
    }
    return;
  }
  if constexpr (KIND == kDxT) {
    // fp32 dX rows over this CTA's 128 d columns: per chunk of 32 rows, each row's 32
    // columns of the warp in one 128-byte store (lane = column)
    const int col = ti.n0 + 128 * rank + 32 * q + lane;
    const bool live = ti.n0 + 128 * rank < p.d;  // warp-uniform: d is a multiple of 128
    float* X = static_cast<float*>(p.out0);
#pragma unroll 1
    for (int ch = 0; ch < nch; ++ch) {
      float v[32];
      tmem_ld32(tacc + ch * 32, v);
      if (!live) continue;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int r = ch * 32 + j;
        if (r < ti.nvalid) X[(row0 + r) * p.d + col] = v[j];
      }
    }
    return;
  }
  if (ti.part == 1) {
    uint16_t* H = static_cast<uint16_t*>(p.out0);
    if (p.gated) {
      const bool is_a = q < 2;
      const int col = ti.n0 + 64 * rank + 32 * (q & 1) + lane;  // h column of this lane
      // named barrier of the warp pair: 1 and 2, or 5 and 6 for the second warp of each lane
      // quadrant (3 and 4 are the tile-level barriers)
      const int bar = 1 + (q & 1) + 4 * half;
      const int j0 = is_a ? 0 : 16;
#pragma unroll 1
      for (int ch = half; ch < nch; ch += nhalves) {
        float v[32];
        tmem_ld32(tacc + ch * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) mine[lane * 33 + j] = v[j];
        named_bar_sync(bar, 64);
        float hv[16];
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int j = j0 + jj;
          const float x0 = mine[lane * 33 + j], x1 = partner[lane * 33 + j];
          const float av = is_a ? x0 : x1, bv = is_a ? x1 : x0;
          const int r = ch * 32 + j;
          hv[jj] = r < ti.nvalid ? silu_f(av) * bv : 0.0f;
          if (p.save_ab && r < ti.nvalid) {
            // dA's and dB's multipliers for the backward, of this warp's half of the rows
            float ma, mb;
            swiglu_bwd_mults(av, bv, &ma, &mb);
            p.save_a[(row0 + r) * p.dff + col] = ma;
            p.save_b[(row0 + r) * p.dff + col] = mb;
          }
        }
        named_bar_sync(bar, 64);  // the partner has read `mine`
        // the warp's 16 rows x 32 h columns as bf16 through `mine` (row pitch 64 bytes), then
        // 16-byte stores: each instruction writes 8 rows x 64 bytes
        uint16_t* hb = reinterpret_cast<uint16_t*>(mine);
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) hb[jj * 32 + lane] = bf16_bits(hv[jj]);
        __syncwarp();
#pragma unroll
        for (int it = 0; it < 2; ++it) {
          const int jj = (it * 32 + lane) >> 2, piece = lane & 3;
          const int r = ch * 32 + j0 + jj;
          if (r < ti.nseg)
            st_v4(H + (row0 + r) * p.dff + (col - lane) + piece * 8,
                  *reinterpret_cast<const uint4*>(hb + jj * 32 + piece * 8));
        }
        __syncwarp();  // stores have read `mine` before the next chunk rewrites it
      }
      if (is_a)
        for (int r = nch * 32 + half; r < ti.nseg; r += nhalves) H[(row0 + r) * p.dff + col] = 0;
    } else {
      const int col = ti.n0 + 128 * rank + 32 * q + lane;
#pragma unroll 1
      for (int ch = half; ch < nch; ch += nhalves) {
        float v[32];
        tmem_ld32(tacc + ch * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int r = ch * 32 + j;
          if (p.save_ab && r < ti.nvalid)
            p.save_a[(row0 + r) * p.dff + col] = relu2_bwd_mult(v[j]);  // dA's multiplier
          if (r < ti.nseg) {
            const float rl = fmaxf(v[j], 0.0f);
            H[(row0 + r) * p.dff + col] = bf16_bits(r < ti.nvalid ? rl * rl : 0.0f);
          }
        }
      }
      for (int r = nch * 32 + half; r < ti.nseg; r += nhalves) H[(row0 + r) * p.dff + col] = 0;
    }
  } else {
    const int c0 = ti.n0 + 128 * rank + 32 * q;  // first output column of this warp
    const bool live = ti.n0 + 128 * rank < p.d;  // warp-uniform: d is a multiple of 128
    uint16_t* Y = static_cast<uint16_t*>(KIND == kFwdT ? p.out1 : p.out0);
    uint16_t* yb = reinterpret_cast<uint16_t*>(mine);
#pragma unroll 1
    for (int ch = half; ch < nch; ch += nhalves) {
      float v[32];
      tmem_ld32(tacc + ch * 32, v);
      if (!live) continue;
      // bf16 rows (the combine's payload): the warp's 32 rows x 32 columns through `mine`
      // (row pitch 64 bytes), then 16-byte stores, each instruction 8 rows x 64 bytes
#pragma unroll
      for (int j = 0; j < 32; ++j) yb[j * 32 + lane] = bf16_bits(v[j]);
      __syncwarp();
#pragma unroll
      for (int it = 0; it < 4; ++it) {
        const int j = (it * 32 + lane) >> 2, piece = lane & 3;
        const int r = ch * 32 + j;
        if (r < ti.nvalid)
          st_v4(Y + (row0 + r) * p.d + c0 + piece * 8,
                *reinterpret_cast<const uint4*>(yb + j * 32 + piece * 8));
      }
      __syncwarp();  // stores have read `mine` before the next chunk rewrites it
    }
  }
}

// PAIR: a cluster of two CTAs on two SMs computes one 256 x BN tile with
// tcgen05.mma.cta_group::2.  Each CTA loads its own 128 rows of A and half of B into its own
// shared memory; rank 0 issues the MMAs (M = 256), whose result lands in both CTAs' TMEM
// (128 rows each).  Both CTAs' loads complete on rank 0's full barrier (TMA .cta_group::2),
// armed by rank 0 for both, so the MMA issuer waits on the barrier the data itself lands
// on; rank 0's commits arrive on both CTAs' empty / tmem-full barriers (multicast); both
// epilogues release the accumulator on rank 0's tmem-empty barrier.
template <int KIND, int BN, bool PAIR>
__global__ void __launch_bounds__(EpiCfg<KIND, PAIR>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB0,
                        const __grid_constant__ CUtensorMap mapB1,
                        const __grid_constant__ GemmParams p) {
  constexpr int EW = EpiCfg<KIND, PAIR>::kWarps;
  constexpr int KPS = KindTraits<KIND>::kKPS;
  using Cfg = GemmCfg<BN, PAIR, EW, KPS>;
  using Tr = KindTraits<KIND>;
  constexpr int S = Cfg::kStages;
  constexpr int BL = Cfg::kBLocal;  // B columns held by this CTA
  constexpr uint32_t IDESC = KIND == kFwd1F8
                                 ? idesc_e4m3_f32(PAIR ? 2 * kBM : kBM, BN)
                                 : idesc_bf16_f32(PAIR ? 2 * kBM : kBM, BN, Tr::kAmn, Tr::kBmn);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t epi0 = base + S * Cfg::kStageBytes;  // epilogue regions (1024-aligned)
  const uint32_t bar0 = epi0 + static_cast<uint32_t>(Cfg::kEpiBytes);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  auto gather_bar = [&](int s) { return bar0 + 8u * (2 * S + 5 + s); };
  uint8_t* misc = gbase + S * Cfg::kStageBytes + Cfg::kEpiBytes + 8 * Cfg::kBars;
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  volatile uint32_t* consumed = reinterpret_cast<volatile uint32_t*>(misc + 8);
  volatile uint32_t* peer_issued = reinterpret_cast<volatile uint32_t*>(misc + 12);
  // bytes this CTA's TMA loads of the fill in each stage bring (written by the producer as
  // it arms / loads the stage), and the peer CTA's ring, sent over at exit (pairs)
  volatile uint32_t* tx_ring = reinterpret_cast<volatile uint32_t*>(misc + 16);
  volatile uint32_t* peer_tx = reinterpret_cast<volatile uint32_t*>(misc + 16 + 4 * S);
  static_assert(16 + 8 * S <= 128, "misc region");
  float* epi_buf = reinterpret_cast<float*>(gbase + S * Cfg::kStageBytes);
  // K block j (< KPS) of stage s
  auto stage_a = [&](int s, int j = 0) { return base + s * Cfg::kStageBytes + j * Cfg::kSubBytes; };
  auto stage_b = [&](int s, int j = 0) { return stage_a(s, j) + kABytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  const bool gather = KIND == kFwd1 && p.gather_x != 0;
  const bool copy = (KIND == kFwd1T || KIND == kFwd1TW) && p.copy_rows != 0;
  const int unit = PAIR ? static_cast<int>(blockIdx.x) / 2 : static_cast<int>(blockIdx.x);
  const int nunits = PAIR ? static_cast<int>(gridDim.x) / 2 : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    // A full barrier completes on its arming arrival (with the TMA bytes).  With gathered A
    // rows, each CTA's 32 producer lanes' cp.async arrivals complete its gather barrier, and
    // the CTA's gather-fence thread then adds one arrival on the full barrier (rank 0's, with
    // PAIR).
    const int full_count = !gather ? 1 : (PAIR ? 3 : 2);
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), full_count);
      mbar_init(empty_bar(s), 1);
      mbar_init(gather_bar(s), 64);  // the lanes of the two gathering warps
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), PAIR ? 2 * EW : EW);  // one arrival per epilogue warp (both CTAs)
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *consumed = 0u;
    *peer_issued = 0u;
    for (int s = 0; s < S; ++s) tx_ring[s] = peer_tx[s] = Cfg::kStageBytes;  // overwritten
    fence_mbar_init();
  }
  if (warp == 2) {
    if constexpr (PAIR) tmem_alloc_pair(smem_u32(const_cast<uint32_t*>(tmem_holder)), Cfg::kTmemCols);
    else tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_holder)), Cfg::kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  if constexpr (PAIR) cluster_sync_all();  // peer barriers initialised before any remote use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Programmatic dependent launch: the set-up above (barriers, TMEM) may overlap the end of
  // the previous kernel in the stream; global memory is touched only after it has completed.
  asm volatile("griddepcontrol.wait;" ::: "memory");

  int64_t ntiles64;
  if constexpr (Tr::kRowsM) ntiles64 = static_cast<int64_t>(PAIR ? p.n_pt[0] : p.n_mt[0]) * p.nb;
  else if constexpr (Tr::kSwap)
    ntiles64 = static_cast<int64_t>(p.n_st[0]) * (KIND == kFwdT ? p.nb + p.nb2 : p.nb);
  else ntiles64 = static_cast<int64_t>(p.E) * p.mb * p.nb;
  if (ntiles64 > p.max_tiles || ntiles64 < 0) {
    if (threadIdx.x == 0) set_error(p.err, MOE_ERR_DEVICE_BOUNDS, 10);
    ntiles64 = 0;
  }
  const int ntiles = static_cast<int>(ntiles64);

  auto wait_bar = [&](uint32_t bar, uint32_t par, volatile int* ab, int site) {
    if constexpr (PAIR) return mbar_wait_cluster(bar, par, ab, p.err, site, p.wait_ns);
    else return mbar_wait(bar, par, ab, p.err, site, p.wait_ns);
  };

  uint32_t issued = 0;
  int skipped = -1;

  if (warp == 0 || (gather && warp == 2)) {
    // ------------------------------------------------------------------ TMA producer
    // Lane 0 waits for each stage and issues the tile loads.  With gather_x the warp first
    // stages the token index of each of the tile's A rows (padding rows read token 0; they are
    // never stored), then every lane gathers 4 of the 128 rows per stage.  `fill`, `ok` and
    // `skipped` are lane 0's (the tile loop broadcasts `ok`).
    if (lane == 0) {
      tma_prefetch_desc(&mapA);
      tma_prefetch_desc(&mapB0);
      tma_prefetch_desc(&mapB1);
    }
    uint32_t fill = 0;
    bool ok = true;
    // with PAIR every load completes on rank 0's full barrier
    auto load = [&](uint32_t dst, const CUtensorMap* m, uint32_t fb, int x, int y) {
      if constexpr (PAIR) tma_load_2d_pair(dst, m, mapa_shared(fb, 0), x, y);
      else tma_load_2d(dst, m, fb, x, y);
    };
    const uint64_t pol_first = l2_policy_evict_first(), pol_last = l2_policy_evict_last();
    // forward operand loads with the eviction priority of kL2HintA / kL2HintB
    auto load_h = [&](int hint, uint32_t dst, const CUtensorMap* m, uint32_t fb, int x, int y) {
      if (hint == 0) {
        load(dst, m, fb, x, y);
      } else {
        const uint64_t pol = hint == 1 ? pol_last : pol_first;
        if constexpr (PAIR) tma_load_2d_pair_hint(dst, m, mapa_shared(fb, 0), x, y, pol);
        else tma_load_2d_hint(dst, m, fb, x, y, pol);
      }
    };
    for (int tile = unit; tile < ntiles; tile += nunits) {
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      const TileInfo ti = decode_tile<KIND, BN, PAIR>(p, tile, rank);
      if (ti.bad) {
        if (lane == 0) set_error(p.err, MOE_ERR_DEVICE_BOUNDS, 11);
        continue;
      }
      // gathered A rows: warp 0 copies rows [0, 64) of the CTA's 128, warp 2 rows [64, 128);
      // lane l takes chunk l & 7 of rows r0 + 4 i + (l >> 3).  Source rows in x (padding
      // rows read token 0; they are never stored):
      const uint16_t* src_row[kBM / 8];
      if (gather) {
        const int r0 = warp == 0 ? 0 : kBM / 2;
#pragma unroll
        for (int i = 0; i < kBM / 8; ++i) {
          const int rr = r0 + 4 * i + (lane >> 3);
          const int pr = rr < ti.nvalid ? p.perm[ti.row0 + rr] : -1;
          src_row[i] = p.gather_src + static_cast<int64_t>(pr >= 0 ? pr / p.k : 0) * p.d;
        }
      }
      const int nb0 = ti.n0 + rank * BL;  // first B column held by this CTA
      // lane 0: the tile loads of K block kb into (sa, sb), completing on fb (A too unless
      // gathered)
      auto load_kblock = [&](int kb, uint32_t fb, uint32_t sa, uint32_t sb) {
        const int k0 = kb * kBK;
        if constexpr (Tr::kSwap) {
          // A: this CTA's 128 weight columns as two 64-column boxes (MN-major); B: this CTA's
          // `box` rows of the block (K-major), by the tensor map of that box height
          if constexpr (KIND == kDxT) {
            // A: this CTA's 128 W1 (K < d_ff) or W3 rows, K-major: one box of 64 K x 128 rows;
            // past d (d % 256 == 128) the rows belong to the next expert or are zero fill, and
            // their results are not stored
            const int wrow = ti.e * p.d + ti.n0 + 128 * rank;
            if (k0 < p.dff) load_h(kL2HintB, sa, &mapB0, fb, k0, wrow);
            else load_h(kL2HintB, sa, &mapB1, fb, k0 - p.dff, wrow);
          } else if constexpr (KIND == kDhT) {
            // A: this CTA's 128 W2 rows (d_ff index), K-major (K = d): one box of 64 K x 128
            // rows; past d_ff (d_ff % 256 == 128) as for kDxT
            load_h(kL2HintB, sa, &mapB0, fb, k0, ti.e * p.dff + ti.n0 + 128 * rank);
          } else if (ti.part == 1) {
            const int wrow = ti.e * p.d + k0;
            if (p.gated) {
              const int c0 = ti.n0 + 64 * rank;  // W1 columns -> lanes 0-63, W3 -> 64-127
              load_h(kL2HintB, sa, &mapB0, fb, c0, wrow);
              load_h(kL2HintB, sa + 8192u, &mapB1, fb, c0, wrow);
            } else {
              const int c0 = ti.n0 + 128 * rank;
              load_h(kL2HintB, sa, &mapB0, fb, c0, wrow);
              load_h(kL2HintB, sa + 8192u, &mapB0, fb, c0 + 64, wrow);
            }
          } else {
            const int wrow = ti.e * p.dff + k0;
            const int c0 = ti.n0 + 128 * rank;  // past d (d % 256 == 128): zero fill
            const CUtensorMap* w2 = KIND == kFwdT ? &mapA : &mapB0;
            load_h(kL2HintB, sa, w2, fb, c0, wrow);
            load_h(kL2HintB, sa + 8192u, w2, fb, c0 + 64, wrow);
          }
          const int bi = ti.box == 16 ? 0 : (ti.box == 32 ? 1 : (ti.box == 64 ? 2 : 3));
          const CUtensorMap* rows = (KIND == kFwdT && ti.part == 2) ? &p.mapR2[bi] : &p.mapR[bi];
          load_h(kL2HintA, sb, rows, fb, k0, ti.row0 + rank * ti.box);
        } else if constexpr (KIND == kFwd1) {
          if (!p.gather_x) load_h(kL2HintA, sa, &mapA, fb, k0, ti.row0);
          const int wrow = ti.e * p.d + k0;
          const int h0 = ti.n0 / 2;  // first h column of the tile
          if (!p.gated) {
            // squared ReLU: every B column comes from W1 (CTA rank r of a pair: its half)
#pragma unroll
            for (int i = 0; i < BL / 64; ++i)
              load_h(kL2HintB, sb + 8192u * i, &mapB0, fb, nb0 + 64 * i, wrow);
          } else if constexpr (PAIR) {
            // rank 0 holds the W1 half of B, rank 1 the W3 half
            const CUtensorMap* wm = rank == 0 ? &mapB0 : &mapB1;
#pragma unroll
            for (int i = 0; i < BL / 64; ++i)
              load_h(kL2HintB, sb + 8192u * i, wm, fb, h0 + 64 * i, wrow);
          } else {
#pragma unroll
            for (int i = 0; i < BN / 128; ++i) {
              load_h(kL2HintB, sb + 8192u * i, &mapB0, fb, h0 + 64 * i, wrow);
              load_h(kL2HintB, sb + 8192u * (BN / 128 + i), &mapB1, fb, h0 + 64 * i, wrow);
            }
          }
        } else if constexpr (KIND == kFwd1F8) {
          // 128 K elements (bytes) per stage: A rows and the W1 / W3 rows (output columns) of
          // the transposed E4M3 weights, all K-major
          const int kb8 = kb * 128;
          const int wrow = ti.e * p.dff + ti.n0 / 2;
          load_h(kL2HintA, sa, &mapA, fb, kb8, ti.row0);
          if constexpr (PAIR) {
            load_h(kL2HintB, sb, rank == 0 ? &mapB0 : &mapB1, fb, kb8, wrow);
          } else {
            load_h(kL2HintB, sb, &mapB0, fb, kb8, wrow);
            load_h(kL2HintB, sb + 16384u, &mapB1, fb, kb8, wrow);
          }
        } else if constexpr (KIND == kFwd2) {
          load_h(kL2HintA, sa, &mapA, fb, k0, ti.row0);
#pragma unroll
          for (int i = 0; i < BL / 64; ++i)
            load_h(kL2HintB, sb + 8192u * i, &mapB0, fb, nb0 + 64 * i, ti.e * p.dff + k0);
        } else if constexpr (KIND == kDh) {
          load(sa, &mapA, fb, k0, ti.row0);
          load(sb, &mapB0, fb, k0, ti.e * p.dff + nb0);
        } else if constexpr (KIND == kDx) {
          load(sa, &mapA, fb, k0, ti.row0);
          if (k0 < p.dff) load(sb, &mapB0, fb, k0, ti.e * p.d + nb0);
          else load(sb, &mapB1, fb, k0 - p.dff, ti.e * p.d + nb0);
        } else {
          const int r = ti.row0 + k0;
          load(sa, &mapA, fb, ti.m0, r);
          load(sa + 8192u, &mapA, fb, ti.m0 + 64, r);
#pragma unroll
          for (int i = 0; i < BL / 64; ++i) load(sb + 8192u * i, &mapB0, fb, nb0 + 64 * i, r);
        }
      };
      // lane 0: arm stage s for the K blocks of the tile's stage `st` (KPS of them, fewer in a
      // last stage) and issue their loads; rank 0 arms its barrier for both CTAs' bytes, rank 1
      // only loads
      auto issue_stage = [&](int st, int s) {
        const uint32_t fb = full_bar(s);
        const int kb0 = st * KPS;
        const int nsub = ti.nk - kb0 < KPS ? ti.nk - kb0 : KPS;
        uint32_t tx = gather ? Cfg::kBBytes : Cfg::kSubBytes;
        if constexpr (Tr::kSwap) tx = kABytes + static_cast<uint32_t>(ti.box) * 128u;
        tx *= static_cast<uint32_t>(nsub);
        tx_ring[s] = tx;
        if (rank == 0) mbar_arrive_expect_tx(fb, PAIR ? 2 * tx : tx);
        for (int j = 0; j < nsub; ++j) load_kblock(kb0 + j, fb, stage_a(s, j), stage_b(s, j));
      };
      const int nst = (ti.nk + KPS - 1) / KPS;  // pipeline stages of the tile
      const bool skip_hook = (p.debug_flags & 1) && blockIdx.x == 0;
      if (gather) {
        // Warps 0 and 2 walk the K blocks together, each copying 64 of the stage's 128 A rows
        // with cp.async: each instruction moves 4 whole 128-byte row pieces (8 lanes per row, one
        // 16-byte chunk each), placed in the 128-byte-swizzled layout the MMA reads (chunk c
        // of row r at chunk c ^ (r & 7)); every lane arrives on the CTA's gather barrier when
        // its copies have landed.
        for (int kb = 0; kb < ti.nk; ++kb) {
          const int s = fill % S;
          const uint32_t ph = (fill / S) & 1u;
          bool got = true;
          if (lane == 0) got = wait_bar(empty_bar(s), ph ^ 1u, abort_flag, 1);
          if (!__shfl_sync(0xFFFFFFFFu, got, 0)) {
            ok = false;
            break;
          }
          const uint32_t fb = full_bar(s), sa = stage_a(s), sb = stage_b(s);
          if (skip_hook && fill == 0) {
            skipped = 0;  // test hook: this stage is never armed nor filled by this CTA
          } else {
            const int c = lane & 7;
            const int r0 = warp == 0 ? 0 : kBM / 2;
#pragma unroll
            for (int i = 0; i < kBM / 8; ++i) {
              const int rr = r0 + 4 * i + (lane >> 3);
              cp_async_16(sa + static_cast<uint32_t>(rr) * 128u +
                              static_cast<uint32_t>((c ^ (rr & 7)) * 16),
                          src_row[i] + kb * kBK + 8 * c);
            }
            cp_async_arrive_noinc(gather_bar(s));
            if (warp == 0 && lane == 0) issue_stage(kb, s);  // one K block per stage
          }
          ++fill;
        }
      } else if (lane == 0) {
        if (copy) {
          // the block's rows are copied by the grid's copy warps: wait for all its units, then
          // order their generic-proxy stores before this thread's TMA loads of the rows
          if (!wait_count(p.done1 + ti.st, kCopyUnits, abort_flag, p.err, 12, p.wait_ns)) {
            ok = false;
          } else {
            fence_proxy_async_global();
          }
        }
        if constexpr (KIND == kFwdT) {
          // a GEMM2 tile reads H rows that GEMM1 tiles of its block store: wait for all of
          // them (each CTA of a pair counts once), then order those generic-proxy stores
          // before this thread's async-proxy (TMA) loads
          if (ti.part == 2) {
            if (!wait_count(p.done1 + ti.st, 2 * p.nb, abort_flag, p.err, 9, p.wait_ns)) {
              ok = false;
            } else {
              fence_proxy_async_global();
            }
          }
        }
        for (int st = 0; st < nst && ok; ++st) {
          const int s = fill % S;
          const uint32_t ph = (fill / S) & 1u;
          if (!wait_bar(empty_bar(s), ph ^ 1u, abort_flag, 1)) {
            ok = false;
            break;
          }
          if (skip_hook && fill == 0) skipped = 0;  // test hook (see above)
          else issue_stage(st, s);
          ++fill;
        }
      }
      __syncwarp();
    }
    if (gather) cp_async_wait_all();  // no copy in flight into shared memory at exit
    issued = fill;
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ------------------------------------------------------------------ MMA issuer
    uint32_t fill = 0;
    int it = 0;
    bool ok = true;
    for (int tile = unit; tile < ntiles && ok; tile += nunits) {
      const TileInfo ti = decode_tile<KIND, BN, PAIR>(p, tile, 0);
      if (ti.bad) continue;
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1u;
      if (!wait_bar(tempty_bar(acc), aph ^ 1u, abort_flag, 2)) break;
      tc_fence_after();
      const uint32_t dtm = tmem_base + acc * BN;
      // swapped kinds: M = 256 weight columns, N = the block's rows (2 box)
      const uint32_t idesc = Tr::kSwap ? idesc_bf16_f32(2 * kBM, 2 * ti.box, Tr::kAmn, 0) : IDESC;
      const int nst = (ti.nk + KPS - 1) / KPS;
      for (int st = 0; st < nst; ++st) {
        const int s = fill % S;
        const uint32_t ph = (fill / S) & 1u;
        if (!wait_bar(full_bar(s), ph, abort_flag, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int kb0 = st * KPS;
        const int nsub = ti.nk - kb0 < KPS ? ti.nk - kb0 : KPS;
        for (int j = 0; j < nsub; ++j) {
          const uint32_t sa = stage_a(s, j), sb = stage_b(s, j);
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = Tr::kAmn ? smem_desc_sw128(sa + kk * 2048u, 8192u, 1024u)
                                         : smem_desc_sw128(sa + kk * 32u, 16u, 1024u);
            const uint64_t bd = Tr::kBmn ? smem_desc_sw128(sb + kk * 2048u, 8192u, 1024u)
                                         : smem_desc_sw128(sb + kk * 32u, 16u, 1024u);
            // bf16: K = 16 per instruction (32 bytes); E4M3: K = 32 (32 bytes), so the same
            // 32-byte descriptor step covers both
            const uint32_t accum = ((kb0 + j) | kk) != 0 ? 1u : 0u;
            if constexpr (KIND == kFwd1F8) {
              if constexpr (PAIR) umma_f8_pair(dtm, ad, bd, IDESC, accum);
              else umma_f8(dtm, ad, bd, IDESC, accum);
            } else {
              if constexpr (PAIR) umma_f16_pair(dtm, ad, bd, idesc, accum);
              else umma_f16(dtm, ad, bd, idesc, accum);
            }
          }
        }
        if constexpr (PAIR) umma_commit_pair(empty_bar(s), 3);
        else umma_commit(empty_bar(s));
        ++fill;
        *consumed = fill;
      }
      if (!ok) break;
      if constexpr (PAIR) umma_commit_pair(tfull_bar(acc), 3);
      else umma_commit(tfull_bar(acc));
      ++it;
    }
    // all MMAs issued by this thread complete before TMEM is released
    if constexpr (PAIR) umma_commit_pair(drain_bar, 1);
    else umma_commit(drain_bar);
    mbar_wait(drain_bar, 0u, nullptr, p.err, 4, p.wait_ns);
  } else if (gather && warp == 3 && lane == 0) {
    // ------------------------------------------------------------------ gather fence
    // cp.async writes shared memory through the generic proxy and the MMAs read it through
    // the async proxy.  Once a stage's gathered rows have landed in this CTA (its gather
    // barrier), this thread fences the proxies and passes one arrival on to the full
    // barrier the MMA issuer waits on (rank 0's with PAIR), so the issuer itself never
    // fences.
    uint32_t fill = 0;
    bool ok = true;
    for (int tile = unit; tile < ntiles && ok; tile += nunits) {
      const TileInfo ti = decode_tile<KIND, BN, PAIR>(p, tile, rank);
      if (ti.bad) continue;
      for (int kb = 0; kb < ti.nk; ++kb) {
        const int s = fill % S;
        if (!mbar_wait(gather_bar(s), (fill / S) & 1u, abort_flag, p.err, 8, p.wait_ns)) {
          ok = false;
          break;
        }
        fence_proxy_async_smem();
        if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(full_bar(s), 0));
        else mbar_arrive(full_bar(s));
        ++fill;
      }
    }
  } else if (copy && (warp == 2 || warp == 3)) {
    // ------------------------------------------------------------------ row copy
    // The permuted rows of the block table, in table order (the order the tiles consume
    // them): unit u is rows 4 (u % 64) .. + 3 of block u / 64, dealt round-robin over the
    // grid's copy warps.  Each lane loads its 16-byte pieces of the unit's rows, all in
    // flight together, then stores them; after the stores every lane fences and lane 0 adds
    // one to the block's count (release).  Units past a block's rows only count.
    const int n16 = p.d >> 3;
    int64_t nblk = p.n_st[0];
    if (nblk < 0 || nblk * p.nb > p.max_tiles) nblk = 0;  // the tile loops record the error
    const int64_t ncw = 2ll * gridDim.x;
    for (int64_t u = 2ll * blockIdx.x + (warp - 2); u < nblk * kCopyUnits; u += ncw) {
      const int st = static_cast<int>(u / kCopyUnits), sub = static_cast<int>(u % kCopyUnits);
      const int e = p.st_expert[st];
      const int64_t row0 = p.st_row0[st];
      int nv = 0;
      if (e >= 0 && e < p.E && row0 >= 0) {
        nv = p.poff[e] + p.counts[e] - static_cast<int>(row0) - 4 * sub;
        nv = nv < 0 ? 0 : (nv > 4 ? 4 : nv);
        if (row0 + 4 * sub + nv > p.rows_cap) nv = 0;
      }
      const uint4* src[4];
      uint4* dst[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int64_t row = row0 + 4 * sub + i;
        int pr = i < nv ? p.perm[row] : 0;
        if (pr < 0) {  // a valid row without its pair: recorded, and copied from token 0
          set_error(p.err, MOE_ERR_DEVICE_BOUNDS, 13);
          pr = 0;
        }
        src[i] = reinterpret_cast<const uint4*>(p.gather_src) + static_cast<int64_t>(pr / p.k) * n16;
        dst[i] = reinterpret_cast<uint4*>(p.copy_dst) + (i < nv ? row : 0) * n16;
      }
      // 16 loads of 16 bytes in flight per lane: 4 rows x 4 column steps
      for (int c = lane; c < n16; c += 128) {
        uint4 v[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (i < nv && c + 32 * j < n16) v[i][j] = ld_nc_v4(src[i] + c + 32 * j);
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (i < nv && c + 32 * j < n16) st_v4(dst[i] + c + 32 * j, v[i][j]);
      }
      __threadfence();  // this lane's stores are visible device-wide ...
      __syncwarp();     // ... before lane 0 counts the unit
      if (lane == 0) red_release_add(p.done1 + st, 1);
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int ew = warp - 4;  // epilogue warp index
    const int q = ew & 3;     // its TMEM lane quadrant (warp % 4)
    int it = 0;
    const uint32_t release_to = PAIR ? mapa_shared(tempty_bar(0), 0) : tempty_bar(0);
    for (int tile = unit; tile < ntiles; tile += nunits) {
      const TileInfo ti = decode_tile<KIND, BN, PAIR>(p, tile, rank);
      if (ti.bad) continue;
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1u;
      // warp-uniform decision: the tcgen05.ld below is .sync.aligned.  In the swapped kinds
      // all epilogue warps decide together (an AND over a named barrier), because they meet
      // at named barriers inside a tile (the chunk exchange of GEMM1, GEMM1's completion
      // count) and a warp that left could leave the others waiting there
      bool ok = __all_sync(0xFFFFFFFFu, wait_bar(tfull_bar(acc), aph, abort_flag, 5));
      if constexpr (Tr::kSwap) ok = named_bar_and(4, 32 * EW, ok);
      if (!ok) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if constexpr (Tr::kSwap) {
        epilogue_swap<KIND>(p, ti, tacc, q, lane, epi_buf + ew * (Cfg::kEpiWarpBytes / 4),
                            epi_buf + (ew ^ 2) * (Cfg::kEpiWarpBytes / 4), rank, ew >> 2,
                            EW / 4);
        if constexpr (KIND == kFwdT) {
          if (ti.part == 1) {
            // this CTA's H rows of the tile are stored: count them for the block's GEMM2
            // tiles (every epilogue thread's stores are made visible device-wide first)
            __threadfence();
            named_bar_sync(3, 32 * EW);
            if (ew == 0 && lane == 0) red_release_add(p.done1 + ti.st, 1);
          }
        }
      } else {
        epilogue_tile<KIND, BN>(p, ti, tacc, q, lane,
                                epi_buf + ew * (Cfg::kEpiWarpBytes / 4),
                                epi0 + ew * static_cast<uint32_t>(Cfg::kEpiWarpBytes), ew >> 2,
                                EW / 4);
      }
      tc_fence_before();
      __syncwarp();
      // The accumulator is free once every lane's tcgen05.ld has completed (they have: the
      // values are in registers).  The arrival is relaxed so that it does not wait for the
      // warp's global stores of this tile, which nothing on the MMA side reads.
      if (lane == 0) {
        if constexpr (PAIR) mbar_arrive_cluster_relaxed(release_to + 8u * acc);
        else mbar_arrive_relaxed(release_to + 8u * acc);
      }
      ++it;
    }
    if (p.tma_store && lane == 0) bulk_wait_all();  // stores done before the CTA exits
  }

  __syncthreads();
  // After an abort, wait for every operand load still in flight before TMEM is released and
  // the CTAs exit.  With PAIR all loads complete on rank 0's barriers: rank 1 reports how many
  // fills it issued, rank 0 re-balances the expected bytes of fills only one CTA issued and
  // waits for them, then both CTAs leave together.
  if constexpr (PAIR) {
    if (rank == 1 && warp == 0 && lane == 0) {
      st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(peer_issued)), 0), issued);
      for (int s = 0; s < S; ++s)
        st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t*>(peer_tx + s)), 0),
                              tx_ring[s]);
    }
    cluster_sync_all();
  }
  if (rank == 0 && warp == 0 && lane == 0) {
    const uint32_t iss_p = PAIR ? *peer_issued : 0u;
    const uint32_t last = issued > iss_p ? issued : iss_p;
    for (uint32_t f = *consumed; f < last; ++f) {
      const int s = f % S;
      const bool armed = f < issued && static_cast<int>(f) != skipped;
      if constexpr (PAIR) {
        // a fill rank 0 armed for both CTAs but the peer never loaded: complete the peer's
        // share (the same bytes: the same tile); a fill only the peer loaded: expect its bytes
        const bool peer_loaded = f < iss_p;
        if (!armed) mbar_arrive_expect_tx(full_bar(s), peer_loaded ? peer_tx[s] : 0u);
        else if (!peer_loaded) mbar_complete_tx(full_bar(s), tx_ring[s]);
      } else {
        if (!armed) continue;
      }
      const uint64_t t0 = global_ns();
      while (!mbar_try_wait(full_bar(s), (f / S) & 1u)) {
        if (global_ns() - t0 > p.wait_ns) break;
      }
    }
  }
  if constexpr (PAIR) {
    __syncthreads();
    cluster_sync_all();  // no load, remote arrival or MMA into the peer after this point
  }
  if (warp == 2) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    else tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
CUtensorMap make_map_2d(const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_rows, cudaError_t* st);
CUtensorMap make_store_map_f32(void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                               cudaError_t* st);

template <int KIND, int BN, bool PAIR>
cudaError_t run_grouped_gemm(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                             const GemmParams& p, int64_t max_tiles, int num_sms,
                             cudaStream_t s) {
  using Cfg = GemmCfg<BN, PAIR, EpiCfg<KIND, PAIR>::kWarps, KindTraits<KIND>::kKPS>;
  auto kern = grouped_gemm_kernel<KIND, BN, PAIR>;
  // the opt-in shared-memory size is a per-device function attribute: set it once per device
  // (two threads racing here both set the same value)
  static std::atomic<unsigned long long> attr_set_mask{0ull};
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit == 0ull || !(attr_set_mask.load(std::memory_order_acquire) & bit)) {
    st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(Cfg::kSmemBytes));
    if (st != cudaSuccess) return st;
    attr_set_mask.fetch_or(bit, std::memory_order_release);
  }
  GemmParams pp = p;
  pp.max_tiles = max_tiles;
  const int64_t units_max = PAIR ? num_sms / 2 : num_sms;
  int64_t units = max_tiles < units_max ? max_tiles : units_max;
  if (units < 1) units = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(PAIR ? 2 * units : units), 1, 1);
  cfg.blockDim = dim3(EpiCfg<KIND, PAIR>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = PAIR ? 2 : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, a, b0, b1, pp);
}

// A rows-grouped GEMM: with pairs, the 256-row pair tiles of the experts chosen for pairs
// run on CTA pairs, and the rest (their odd last 128-row tiles, and every tile of the other
// experts) on single CTAs in a second launch; both give bitwise the same rows.  `lo` carries
// that launch's tile table in place of the 128-row tile table; b0/b1 are the B maps of the
// pair launch (a K-major B box holds BN/2 rows there), sb0/sb1 those of single-CTA launches
// (BN rows).
template <int KIND, int BN>
cudaError_t run_rows_kind(bool pair, const CUtensorMap& a, const CUtensorMap& b0,
                          const CUtensorMap& b1, const CUtensorMap& sb0, const CUtensorMap& sb1,
                          const GemmParams& p, const GemmParams& lo, int64_t max_mt,
                          int num_sms, cudaStream_t s) {
  if (!pair) return run_grouped_gemm<KIND, BN, false>(a, sb0, sb1, p, max_mt * p.nb, num_sms, s);
  cudaError_t st = run_grouped_gemm<KIND, BN, true>(a, b0, b1, p, max_mt * p.nb, num_sms, s);
  if (st != cudaSuccess) return st;
  return run_grouped_gemm<KIND, BN, false>(a, sb0, sb1, lo, max_mt * lo.nb, num_sms, s);
}

}  // namespace moe
