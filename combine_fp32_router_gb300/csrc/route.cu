// Memory-bound kernels of the MoE layer: routing (top-k + softmax gate), per-expert
// counting and exclusive prefix sums, the stable row permute (dispatch), padding rows, the
// gate-weighted combine, and the per-token part of the backward.
//
// Dispatch -> Expert Compute -> Combine is the layer of "DeepSeek-V4 parallel strategy"
// (blog.lpkt.cn, EP section).  The combine reads the expert outputs as bf16 rows, the BF16
// combine payload of the report translation (itsolotime.com, section 1.4), and accumulates
// in fp32.  Determinism follows the
// report's section 3 and the 10100.com reading: no floating-point atomics anywhere; counts
// come from per-CTA shared-memory bit masks and histograms, positions from a fixed-order
// prefix sum, and every floating-point reduction runs in a fixed order that depends only on
// d and k.
#include <atomic>
#include <cfloat>
#include <climits>

#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace moe {

namespace {

// ------------------------------------------------------------------------------ routing
// Order key of a logit: an unsigned integer that sorts like the float (larger logit, larger
// key), with -0 folded into +0 so that the two compare equal (the lower expert index then
// wins the tie).
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v == 0.0f) v = 0.0f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float order_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

constexpr int kRouteWarps = 16;                                     // warps per routing CTA
constexpr int kRouteTokPerWarp = kRouteTokensPerBlock / kRouteWarps;  // top-k tokens per warp
static_assert(kRouteTokensPerBlock == 128 && kRouteTokPerWarp * kRouteWarps == 128, "");

// Top-k and gate of one token, by one warp: k rounds of a warp arg-max (a max-reduction of
// the order keys, then a min-reduction of the expert indices holding that key, so ties go
// to the lower index; the winner is marked taken), then a softmax over the k selected logits
// in fp32, summed in slot order.  v[c] is the logit of expert lane + 32 c.  Lane j < k
// receives slot j's expert and gate.
template <int EPL>
__device__ __forceinline__ void topk_token(const float (&v)[EPL], int E, int k, int lane,
                                           int* sel_e_out, float* gate_out) {
  uint32_t key[EPL];
#pragma unroll
  for (int c = 0; c < EPL; ++c) key[c] = order_key(v[c]);
  uint32_t live = 0;  // bit c: expert lane + 32c exists and is not yet taken
#pragma unroll
  for (int c = 0; c < EPL; ++c)
    if (lane + 32 * c < E) live |= 1u << c;
  int sel_e = 0;
  float sel_v = 0.0f;
  for (int j = 0; j < k; ++j) {
    uint32_t best = 0u;  // a lane with no live expert offers 0, never above a live key
#pragma unroll
    for (int c = 0; c < EPL; ++c)
      if (((live >> c) & 1u) && key[c] > best) best = key[c];
    const uint32_t bk = __reduce_max_sync(0xFFFFFFFFu, best);
    uint32_t mine = 0xFFFFFFFFu;
#pragma unroll
    for (int c = EPL - 1; c >= 0; --c)
      if (((live >> c) & 1u) && key[c] == bk) mine = static_cast<uint32_t>(lane + 32 * c);
    const uint32_t ew = __reduce_min_sync(0xFFFFFFFFu, mine);
    if ((ew & 31u) == static_cast<uint32_t>(lane)) live &= ~(1u << (ew >> 5));
    if (lane == j) {
      sel_e = static_cast<int>(ew);
      sel_v = order_value(bk);
    }
  }
  const float v0 = __shfl_sync(0xFFFFFFFFu, sel_v, 0);
  const float ex = (lane < k) ? expf(sel_v - v0) : 0.0f;
  float s = 0.0f;
  for (int j = 0; j < k; ++j) s += __shfl_sync(0xFFFFFFFFu, ex, j);
  *sel_e_out = sel_e;
  *gate_out = ex / s;
}

// Ranks inside one block of nt <= 128 tokens whose experts are in tok_e ([128][kMaxK]):
// per 32-token chunk (warps 0..3), a bit mask per expert (bit i = token i of the chunk chose
// it; `mask` [4][E] zeroed beforehand) gives each pair its rank among the chunk's earlier
// tokens, and the masks' popcounts the chunk bases.  On return tok_r[i][j] is pair (i, j)'s
// rank among the block's tokens routed to the same expert, and count[e] (shared or global
// memory) the block's tokens routed to e.  Every thread of the block calls it, after a
// barrier that follows the writes of tok_e; it ends with a barrier.
__device__ __forceinline__ void rank_block(uint32_t* mask, int32_t* wbase, const int32_t* tok_e,
                                           int32_t* tok_r, int nt, int E, int k,
                                           int32_t* count) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int i = w * 32 + lane;
  const bool valid = w < kRouteTokensPerBlock / 32 && i < nt;
  const int32_t* my_e = tok_e + i * kMaxK;
  int32_t* my_r = tok_r + i * kMaxK;
  if (valid)
    for (int j = 0; j < k; ++j) atomicOr(&mask[w * E + my_e[j]], 1u << lane);
  __syncwarp();
  if (valid)
    for (int j = 0; j < k; ++j) my_r[j] = __popc(mask[w * E + my_e[j]] & ((1u << lane) - 1u));
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int run = 0;
#pragma unroll
    for (int ww = 0; ww < kRouteTokensPerBlock / 32; ++ww) {
      wbase[ww * E + e] = run;
      run += __popc(mask[ww * E + e]);
    }
    count[e] = run;
  }
  __syncthreads();
  if (valid)
    for (int j = 0; j < k; ++j) my_r[j] += wbase[w * E + my_e[j]];
  __syncthreads();
}

// One CTA = 128 consecutive tokens.  Top-k: 16 warps x 8 tokens; a warp first loads the
// logits of NB of its tokens (EPL per lane each) so that their loads are in flight together,
// then runs topk_token per token.  rank_block then gives each pair its rank among the CTA's
// tokens routed to the same expert (pos_local) and the CTA's histogram row.
template <int EPL>
__global__ void __launch_bounds__(kRouteWarps * 32) route_topk_kernel(
    const float* __restrict__ logits, int64_t T, int E, int k, int32_t* __restrict__ topk,
    float* __restrict__ gate, int32_t* __restrict__ pos_local, int32_t* __restrict__ hist) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  constexpr int NB = EPL <= 8 ? 8 : (EPL <= 16 ? 4 : 2);
  static_assert(kRouteTokPerWarp % NB == 0, "");
  extern __shared__ uint32_t sm[];
  uint32_t* mask = sm;                                        // [4][E]
  int32_t* wbase = reinterpret_cast<int32_t*>(sm + 4 * E);   // [4][E]
  int32_t* tok_e = wbase + 4 * E;                             // [128][kMaxK]
  int32_t* tok_r = tok_e + kRouteTokensPerBlock * kMaxK;     // [128][kMaxK]

  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 4 * E; i += blockDim.x) mask[i] = 0u;

  const int64_t blk0 = static_cast<int64_t>(blockIdx.x) * kRouteTokensPerBlock;
  const int wt0 = w * kRouteTokPerWarp;
  for (int b0 = 0; b0 < kRouteTokPerWarp; b0 += NB) {
    float v[NB][EPL];
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int64_t t = blk0 + wt0 + b0 + i;
#pragma unroll
      for (int c = 0; c < EPL; ++c) {
        const int e = lane + 32 * c;
        v[i][c] = (t < T && e < E) ? __ldg(logits + t * E + e) : 0.0f;
      }
    }
#pragma unroll
    for (int i = 0; i < NB; ++i) {
      const int64_t t = blk0 + wt0 + b0 + i;
      if (t >= T) break;
      int sel_e;
      float g;
      topk_token<EPL>(v[i], E, k, lane, &sel_e, &g);
      if (lane < k) {
        topk[t * k + lane] = sel_e;
        gate[t * k + lane] = g;
        tok_e[(wt0 + b0 + i) * kMaxK + lane] = sel_e;
      }
    }
  }
  __syncthreads();
  const int64_t left = T - blk0;
  const int nt = left < kRouteTokensPerBlock ? static_cast<int>(left) : kRouteTokensPerBlock;
  rank_block(mask, wbase, tok_e, tok_r, nt, E, k, hist + static_cast<int64_t>(blockIdx.x) * E);
  for (int i = threadIdx.x; i < nt * k; i += blockDim.x)
    pos_local[blk0 * k + i] = tok_r[(i / k) * kMaxK + i % k];
}

// Column prefix over the routing CTAs: bbase[b][e] = sum_{b' < b} hist[b'][e], counts[e].
// One CTA per 32 experts; warp w owns a contiguous range of routing CTAs.
__global__ void __launch_bounds__(256) scan_cols_kernel(const int32_t* __restrict__ hist,
                                                        int64_t nblk, int E,
                                                        int32_t* __restrict__ bbase,
                                                        int32_t* __restrict__ counts) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  __shared__ int part[8][32];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int64_t ch = (nblk + 7) / 8;
  const int64_t b0 = w * ch, b1 = b0 + ch < nblk ? b0 + ch : nblk;
  int sum = 0;
  if (e < E)
    for (int64_t b = b0; b < b1; ++b) sum += hist[b * E + e];
  part[w][lane] = sum;
  __syncthreads();
  if (w == 0) {
    int run = 0;
    for (int ww = 0; ww < 8; ++ww) {
      const int v = part[ww][lane];
      part[ww][lane] = run;
      run += v;
    }
    if (e < E) counts[e] = run;
  }
  __syncthreads();
  int run = part[w][lane];
  if (e < E)
    for (int64_t b = b0; b < b1; ++b) {
      const int v = hist[b * E + e];
      bbase[b * E + e] = run;
      run += v;
    }
}

// Block-wide exclusive scan of one int per thread (blockDim.x == 1024).
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += o;
  }
  __syncthreads();
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  if (w == 0) {
    int x = warp_tot[lane];
    int xi = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, xi, off);
      if (lane >= off) xi += o;
    }
    warp_tot[lane] = xi - x;
    if (lane == 31) *total = xi;
  }
  __syncthreads();
  return warp_tot[w] + incl - v;
}

// Merge of two lists in proportion: element i of list A (length na) sits at relative time
// (i + 1/2) / na, element j of B (length nb) at (j + 1/2) / nb; ties go to the first list.
// merge_before(i) = number of B elements placed before element i of A; its position is
// i + merge_before(i).  Positions form a permutation of [0, na + nb) and keep each list's
// order.
__device__ __forceinline__ int merge_before(int i, int na, int nb, bool a_first) {
  if (nb == 0) return 0;
  const int64_t num = (2ll * i + 1) * nb - na;
  int64_t before;
  if (a_first) {   // B elements strictly earlier: (2j+1) na < (2i+1) nb
    before = num <= 0 ? 0 : (num + 2ll * na - 1) / (2ll * na);
  } else {         // B elements earlier or tied: (2j+1) na <= (2i+1) nb
    before = num < 0 ? 0 : num / (2ll * na) + 1;
  }
  return before > nb ? nb : static_cast<int>(before);
}

// Number of entries of the non-decreasing array incl[0..n) that are <= i: the owner of
// element i of a list whose per-expert inclusive prefix is incl.
__device__ __forceinline__ int owner_of(const int* incl, int n, int i) {
  int lo = 0, hi = n;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (incl[mid] <= i) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// One tile table: list A = experts with >= 2 tiles (bound by the tensor cores), list B = the
// others (one tile each, bound by reading their weights).  Each list keeps expert order; the
// two are merged in proportion so that the weight streams of light experts overlap the math
// of heavy ones instead of all coming last.  One thread per table entry.  The order changes
// no result: every tile is computed the same way wherever it runs.
__device__ __forceinline__ void fill_tile_table(const int* a_incl, const int* b_incl,
                                                const int* poff, int E, int na, int nb,
                                                int rows_per_tile, int32_t* t_expert,
                                                int32_t* t_row0) {
  for (int idx = threadIdx.x; idx < na + nb; idx += blockDim.x) {
    const bool in_a = idx < na;
    const int i = in_a ? idx : idx - na;
    const int* incl = in_a ? a_incl : b_incl;
    const int e = owner_of(incl, E, i);
    const int m = i - (e > 0 ? incl[e - 1] : 0);
    const int at = i + (in_a ? merge_before(i, na, nb, true) : merge_before(i, nb, na, false));
    t_expert[at] = e;
    t_row0[at] = poff[e] + m * rows_per_tile;
  }
}

// Offsets and tile tables of the expert counts, one CTA of 1024 threads (thread e holds
// expert e's count c, 0 past E): offsets (unpadded exclusive prefix and total, unless null),
// poff (rows padded to multiples of `align`, with the total), and with_tables the GEMM tile
// tables.  Every thread of the CTA calls it.
__device__ __forceinline__ void offsets_block(int c, int E, int align, int32_t* __restrict__ offsets,
                                              int32_t* __restrict__ poff, const TileTables& tt,
                                              int with_tables, DevErr* err) {
  __shared__ int warp_tot[32];
  __shared__ int total;
  __shared__ int s_poff[1024], s_a[1024], s_b[1024], s_pa[1024], s_pb[1024], s_sa[1024],
      s_sb[1024];
  const int e = threadIdx.x;
  const int pc = (c + align - 1) / align * align;
  const int off = block_exclusive_scan(c, warp_tot, &total);
  const int tot_c = total;
  if (offsets) {
    if (e < E) offsets[e] = off;
    if (e == 0) offsets[E] = tot_c;
  }
  const int poffv = block_exclusive_scan(pc, warp_tot, &total);
  const int tot_p = total;
  if (e < E) poff[e] = poffv;
  if (e == 0) poff[E] = tot_p;
  if (!with_tables) return;
  // 128-row tiles (the single-CTA schedule) and, for CTA pairs, 256-row pair tiles (two
  // consecutive 128-row tiles of one expert) plus a table for the single-CTA launch that runs
  // beside them.  An expert runs on pairs when its tile count is even, or odd and at least
  // kPairOddMinTiles; its odd last tile then goes to the single-CTA launch, which reads the
  // expert's weights a second time, a cost that the pair tiles' higher MMA rate repays only
  // from that many tiles on.  Every other expert runs all its tiles in the single-CTA launch
  // and reads its weights once.  Pair and single-CTA tiles compute bitwise the same rows, so
  // the choice changes no result.
  const int nm = pc / kTileRows;
  const bool paired = nm >= 2 && ((nm & 1) == 0 || nm >= kPairOddMinTiles);
  const int np = paired ? nm / 2 : 0;
  const int nlo = paired ? (nm & 1) : nm;  // tiles of the single-CTA launch
  const int ha = block_exclusive_scan(nm >= 2 ? nm : 0, warp_tot, &total) + (nm >= 2 ? nm : 0);
  const int H = total;
  const int lb = block_exclusive_scan(nm >= 2 ? 0 : nm, warp_tot, &total) + (nm >= 2 ? 0 : nm);
  const int L = total;
  const int pa = block_exclusive_scan(np >= 2 ? np : 0, warp_tot, &total) + (np >= 2 ? np : 0);
  const int PH = total;
  const int pb = block_exclusive_scan(np >= 2 ? 0 : np, warp_tot, &total) + (np >= 2 ? 0 : np);
  const int PL = total;
  const int los = block_exclusive_scan(nlo, warp_tot, &total);
  const int NLO = total;
  // blocks of up to 256 rows for the swapped forward GEMMs: experts with several blocks
  // (bound by the tensor cores) merged in proportion with the one-block experts (bound by
  // reading their weights)
  const int ns = (c + 2 * kTileRows - 1) / (2 * kTileRows);
  const int sa = block_exclusive_scan(ns >= 2 ? ns : 0, warp_tot, &total) + (ns >= 2 ? ns : 0);
  const int SH = total;
  const int sb = block_exclusive_scan(ns == 1 ? 1 : 0, warp_tot, &total) + (ns == 1 ? 1 : 0);
  const int SL = total;
  // every table holds at most sum(nm) <= max_mt entries (the padded rows bound the tiles)
  const bool fits = H + L <= tt.max_mt;
  if (e < E) {
    s_poff[e] = poffv;
    s_a[e] = ha;
    s_b[e] = lb;
    s_pa[e] = pa;
    s_pb[e] = pb;
    s_sa[e] = sa;
    s_sb[e] = sb;
    if (fits) {
      for (int i = 0; i < nlo; ++i) {  // nlo <= kPairOddMinTiles - 2 for experts not paired
        tt.lo_expert[los + i] = e;
        tt.lo_row0[los + i] = poffv + (nm - nlo + i) * kTileRows;
      }
    }
  }
  if (e == 0) {
    tt.n_mt[0] = fits ? H + L : 0;
    tt.n_pt[0] = fits ? PH + PL : 0;
    tt.n_lo[0] = fits ? NLO : 0;
    tt.n_st[0] = fits ? SH + SL : 0;
  }
  __syncthreads();
  if (!fits) {
    if (e == 0) set_error(err, MOE_ERR_DEVICE_BOUNDS, 100);
    return;
  }
  fill_tile_table(s_a, s_b, s_poff, E, H, L, kTileRows, tt.mt_expert, tt.mt_row0);
  fill_tile_table(s_pa, s_pb, s_poff, E, PH, PL, 2 * kTileRows, tt.pt_expert, tt.pt_row0);
  fill_tile_table(s_sa, s_sb, s_poff, E, SH, SL, 2 * kTileRows, tt.st_expert, tt.st_row0);
  if (tt.done1)
    for (int i = threadIdx.x; i < SH + SL; i += blockDim.x) tt.done1[i] = 0;
}

__global__ void __launch_bounds__(1024) offsets_kernel(const int32_t* __restrict__ counts, int E,
                                                       int align, int32_t* __restrict__ offsets,
                                                       int32_t* __restrict__ poff, TileTables tt,
                                                       int with_tables, DevErr* err) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  const int e = threadIdx.x;
  offsets_block(e < E ? counts[e] : 0, E, align, offsets, poff, tt, with_tables, err);
}

// Stable permute.  One warp per token: lanes j < k turn the CTA-local rank into the final
// row (padded expert offset + rank of earlier routing CTAs + local rank), write pos/perm,
// then (unless x_perm is null) the warp copies the token's row once from x and stores it k
// times (16-byte moves).
__global__ void __launch_bounds__(256) scatter_kernel(const uint4* __restrict__ x, int64_t T,
                                                      int d, int E, int k,
                                                      const int32_t* __restrict__ topk,
                                                      const int32_t* __restrict__ bbase,
                                                      const int32_t* __restrict__ poff,
                                                      int32_t* __restrict__ pos,
                                                      int32_t* __restrict__ perm,
                                                      uint4* __restrict__ x_perm,
                                                      int64_t rows_cap, DevErr* err) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int n16 = d >> 3;
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < T;
       t += nwarps) {
    int row = 0;
    if (lane < k) {
      const int64_t p = t * k + lane;
      const int e = topk[p];
      const int64_t b = t / kRouteTokensPerBlock;
      // the expert index is checked before it indexes poff and bbase, the row after
      row = (e >= 0 && e < E) ? poff[e] + bbase[b * E + e] + pos[p] : -1;
      if (row < 0 || row >= rows_cap) {
        set_error(reinterpret_cast<DevErr*>(err), MOE_ERR_DEVICE_BOUNDS, 200);
        row = -1;
      } else {
        pos[p] = row;
        perm[row] = static_cast<int32_t>(p);
      }
    }
    if (!x_perm) continue;  // indices only (the expert GEMM gathers rows from x itself)
    int rows[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) rows[j] = __shfl_sync(0xFFFFFFFFu, row, j);
    const uint4* src = x + t * n16;
    int c = lane;
    for (; c + 32 < n16; c += 64) {
      const uint4 v0 = ld_nc_v4(src + c), v1 = ld_nc_v4(src + c + 32);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k && rows[j] >= 0) {
          uint4* dst = x_perm + static_cast<int64_t>(rows[j]) * n16;
          st_v4(dst + c, v0);
          st_v4(dst + c + 32, v1);
        }
    }
    for (; c < n16; c += 32) {
      const uint4 v0 = ld_nc_v4(src + c);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k && rows[j] >= 0) st_v4(x_perm + static_cast<int64_t>(rows[j]) * n16 + c, v0);
    }
  }
}

// Single-launch dispatch for T <= 128 (one routing block): every CTA routes all T tokens
// itself (topk_token, rank_block: the same arithmetic as route_topk_kernel) and scans the
// counts, so no CTA waits for another.  CTA 0 clears the error record and writes the
// routing outputs (topk, gate, pos,
// perm of the tokens' rows, counts, and offsets_block's offsets, poff and tile tables); the
// other CTAs (CTA 0 too in a grid of one) set perm = -1 on the padding rows, a warp per
// expert, and copy the token rows to their permuted rows, work split by 16-byte column chunks
// (each chunk loaded once, stored k times).  Results equal those of route_topk, scan_cols,
// offsets, scatter and pad_rows's perm part.  1024 threads; dynamic shared memory as
// small_dispatch_smem.
template <int EPL>
__global__ void __launch_bounds__(1024) dispatch_small_kernel(
    const float* __restrict__ logits, const uint4* __restrict__ x, int T, int d, int E, int k,
    int align, int32_t* __restrict__ topk, float* __restrict__ gate, int32_t* __restrict__ pos,
    int32_t* __restrict__ perm, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ poff, TileTables tt, int with_tables, uint4* __restrict__ x_perm,
    int64_t rows_cap, DevErr* err) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  constexpr int NB = EPL <= 8 ? 4 : 1;  // tokens whose loads fly together (no spills)
  extern __shared__ uint32_t sm[];
  uint32_t* mask = sm;                                        // [4][E]
  int32_t* wbase = reinterpret_cast<int32_t*>(sm + 4 * E);   // [4][E]
  int32_t* tok_e = wbase + 4 * E;                             // [128][kMaxK]
  int32_t* tok_r = tok_e + kRouteTokensPerBlock * kMaxK;     // [128][kMaxK]: rank, then row
  int32_t* s_cnt = tok_r + kRouteTokensPerBlock * kMaxK;     // [E]
  int32_t* s_poff = s_cnt + E;                                // [E + 1]
  __shared__ int warp_tot[32];
  __shared__ int total;
  const bool lead = blockIdx.x == 0;
  const bool mover = !lead || gridDim.x == 1;  // pads perm and copies rows
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // the launch begins the layer's device work: CTA 0, the only one that records errors
  // here, clears the error record (ordered before its first record by the barriers below)
  if (lead && threadIdx.x == 0) *err = DevErr{};
  for (int i = threadIdx.x; i < 4 * E; i += blockDim.x) mask[i] = 0u;
  for (int t0 = w; t0 < T; t0 += 32 * NB) {
    float v[NB][EPL];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int t = t0 + 32 * b;
#pragma unroll
      for (int c = 0; c < EPL; ++c) {
        const int e = lane + 32 * c;
        v[b][c] = (t < T && e < E) ? __ldg(logits + static_cast<int64_t>(t) * E + e) : 0.0f;
      }
    }
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const int t = t0 + 32 * b;
      if (t >= T) break;
      int sel_e;
      float g;
      topk_token<EPL>(v[b], E, k, lane, &sel_e, &g);
      if (lane < k) {
        tok_e[t * kMaxK + lane] = sel_e;
        if (lead) {
          topk[t * k + lane] = sel_e;
          gate[t * k + lane] = g;
        }
      }
    }
  }
  __syncthreads();
  rank_block(mask, wbase, tok_e, tok_r, T, E, k, s_cnt);
  const int c = threadIdx.x < E ? s_cnt[threadIdx.x] : 0;
  if (lead) {
    if (threadIdx.x < E) counts[threadIdx.x] = c;
    offsets_block(c, E, align, offsets, poff, tt, with_tables, err);
  }
  // this CTA's copy of the padded offsets (the same scan as offsets_block's)
  const int pv = block_exclusive_scan((c + align - 1) / align * align, warp_tot, &total);
  if (threadIdx.x < E) s_poff[threadIdx.x] = pv;
  if (threadIdx.x == 0) s_poff[E] = total;
  __syncthreads();
  for (int i = threadIdx.x; i < T * k; i += blockDim.x) {
    const int t = i / k, j = i - t * k;
    int row = s_poff[tok_e[t * kMaxK + j]] + tok_r[t * kMaxK + j];
    if (row >= rows_cap) {
      if (lead) set_error(err, MOE_ERR_DEVICE_BOUNDS, 210);
      row = -1;
    } else if (lead) {
      pos[i] = row;
      perm[row] = i;
    }
    tok_r[t * kMaxK + j] = row;
  }
  if (!mover) return;
  const int nmov = gridDim.x > 1 ? gridDim.x - 1 : 1;
  const int mrank = gridDim.x > 1 ? blockIdx.x - 1 : 0;
  for (int e = mrank * 32 + w; e < E; e += nmov * 32) {
    const int64_t r1 = s_poff[e + 1] < rows_cap ? s_poff[e + 1] : rows_cap;
    for (int64_t r = s_poff[e] + s_cnt[e] + lane; r < r1; r += 32) perm[r] = -1;
  }
  __syncthreads();  // every row of tok_r is final
  if (!x_perm) return;
  const int n16 = d >> 3;
  const int64_t nchunks = static_cast<int64_t>(T) * n16;
  for (int64_t q = static_cast<int64_t>(mrank) * blockDim.x + threadIdx.x; q < nchunks;
       q += static_cast<int64_t>(nmov) * blockDim.x) {
    const int t = static_cast<int>(q / n16);
    const int col = static_cast<int>(q - static_cast<int64_t>(t) * n16);
    const uint4 v = ld_nc_v4(x + q);
    for (int j = 0; j < k; ++j) {
      const int row = tok_r[t * kMaxK + j];
      if (row >= 0) st_v4(x_perm + static_cast<int64_t>(row) * n16 + col, v);
    }
  }
}

// ------------------------------------------------------------------ FP8 dispatch payload
// E4M3 byte of v (round to nearest even, saturating at 448)
__device__ __forceinline__ uint32_t e4m3_byte(float v) {
  return static_cast<uint32_t>(__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3));
}
// E4M3 bytes of the 8 bf16 values in u, each divided by s (an fp32 division)
__device__ __forceinline__ uint2 e4m3_pack8(uint4 u, float s) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
  uint32_t b[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    b[2 * i] = e4m3_byte(bf16lo(w[i]) / s);
    b[2 * i + 1] = e4m3_byte(bf16hi(w[i]) / s);
  }
  return make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                    b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
}

// Stable permute with the FP8 payload: as scatter_kernel, but the warp first takes the
// token row's largest magnitude, stores the row scale s = amax / 448 (1 for a zero row) and
// writes each permuted copy as E4M3 bytes of x / s (d bytes per row).
__global__ void __launch_bounds__(256) scatter_fp8_kernel(const uint4* __restrict__ x, int64_t T,
                                                          int d, int E, int k,
                                                          const int32_t* __restrict__ topk,
                                                          const int32_t* __restrict__ bbase,
                                                          const int32_t* __restrict__ poff,
                                                          int32_t* __restrict__ pos,
                                                          int32_t* __restrict__ perm,
                                                          uint8_t* __restrict__ x_perm,
                                                          float* __restrict__ xscale,
                                                          int64_t rows_cap, DevErr* err) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int n16 = d >> 3;  // 16-byte chunks of 8 bf16 per row
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < T;
       t += nwarps) {
    int row = 0;
    if (lane < k) {
      const int64_t p = t * k + lane;
      const int e = topk[p];
      const int64_t b = t / kRouteTokensPerBlock;
      // the expert index is checked before it indexes poff and bbase, the row after
      row = (e >= 0 && e < E) ? poff[e] + bbase[b * E + e] + pos[p] : -1;
      if (row < 0 || row >= rows_cap) {
        set_error(err, MOE_ERR_DEVICE_BOUNDS, 201);
        row = -1;
      } else {
        pos[p] = row;
        perm[row] = static_cast<int32_t>(p);
      }
    }
    int rows[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) rows[j] = __shfl_sync(0xFFFFFFFFu, row, j);
    const uint4* src = x + t * n16;
    float amax = 0.0f;
    for (int c = lane; c < n16; c += 32) {
      const uint4 u = ld_nc_v4(src + c);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
        amax = fmaxf(amax, fmaxf(fabsf(bf16lo(w[i])), fabsf(bf16hi(w[i]))));
    }
    // the magnitudes are non-negative floats: their bit patterns order like the values
    amax = __uint_as_float(__reduce_max_sync(0xFFFFFFFFu, __float_as_uint(amax)));
    const float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    if (lane == 0) xscale[t] = s;
    for (int c = lane; c < n16; c += 32) {
      const uint2 q = e4m3_pack8(ld_nc_v4(src + c), s);
#pragma unroll
      for (int j = 0; j < kMaxK; ++j)
        if (j < k && rows[j] >= 0)
          *reinterpret_cast<uint2*>(x_perm + static_cast<int64_t>(rows[j]) * d + 8 * c) = q;
    }
  }
}

// E4M3 weights for the FP8 GEMM1: W [E][K][N] bf16 -> Wq [E][N][K] (transposed, so each
// output column is a K-contiguous row) and scales [E][N], s = amax over K / 448 (1 for a
// zero column), q = e4m3(w / s).  One CTA per (expert, 32 columns).
__global__ void __launch_bounds__(256) quantize_weights_fp8_kernel(
    const uint16_t* __restrict__ W, int K, int N, uint8_t* __restrict__ Wq,
    float* __restrict__ scales) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  __shared__ float red[8][32];
  __shared__ float sc[32];
  __shared__ uint8_t tile[32][36];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int n0 = blockIdx.x * 32;
  const int64_t e = blockIdx.y;
  const uint16_t* We = W + e * K * static_cast<int64_t>(N);
  float m = 0.0f;
  for (int kk = w; kk < K; kk += 8)
    m = fmaxf(m, fabsf(__uint_as_float(static_cast<uint32_t>(We[static_cast<int64_t>(kk) * N + n0 + lane]) << 16)));
  red[w][lane] = m;
  __syncthreads();
  if (w == 0) {
    float a = red[0][lane];
#pragma unroll
    for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i][lane]);
    const float s = a > 0.0f ? a / 448.0f : 1.0f;
    sc[lane] = s;
    scales[e * N + n0 + lane] = s;
  }
  __syncthreads();
  const float s = sc[lane];
  uint8_t* out = Wq + (e * N + n0) * static_cast<int64_t>(K);
  for (int k0 = 0; k0 < K; k0 += 32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int kk = k0 + w + 8 * i;
      const float v = __uint_as_float(static_cast<uint32_t>(We[static_cast<int64_t>(kk) * N + n0 + lane]) << 16);
      tile[w + 8 * i][lane] = static_cast<uint8_t>(e4m3_byte(v / s));
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int nn = w + 8 * i;
      out[static_cast<int64_t>(nn) * K + k0 + lane] = tile[lane][nn];
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(256) pad_rows_kernel(const int32_t* __restrict__ counts,
                                                       const int32_t* __restrict__ poff,
                                                       int32_t* __restrict__ perm,
                                                       uint4* __restrict__ rows,
                                                       int64_t row16) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  const int e = blockIdx.x;
  const int64_t r0 = static_cast<int64_t>(poff[e]) + counts[e];
  const int64_t r1 = poff[e + 1];
  if (perm)
    for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) perm[r] = -1;
  if (rows) {
    const int64_t n = (r1 - r0) * row16;
    uint4* base = rows + r0 * row16;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) st_v4(base + i, z);
  }
}

// Work unit of the combines: (token, block of kCombCols columns).  A warp takes units
// u, u + nwarps, ... of a grid sized to the GPU's resident capacity, so that the last wave is
// at most one unit per warp instead of a partial wave of whole blocks.
constexpr int kCombChunks = 128;  // 8-column chunks per unit (1024 columns, 4 per lane)

// Combine: out[t] = bf16( sum_j gate[t,j] * y[pos[t,j]] ) over the bf16 expert-output rows
// (the BF16 combine payload of the report translation, section 1.4), fp32 fused multiply-adds
// in slot order j = 0..k-1, one rounding at the end.  Each lane owns 8 consecutive columns per
// step (one 16-byte load per slot).  KC >= k bounds the slots.
// `cpu` chunks per work unit: kCombChunks, or 64 (one iteration per lane) for small batches,
// whose few units would otherwise leave each warp several dependent load rounds.
template <int KC>
__global__ void __launch_bounds__(256) combine_kernel(const uint4* __restrict__ y,
                                                      const float* __restrict__ gate,
                                                      const int32_t* __restrict__ pos,
                                                      int64_t T, int k, int d, int cpu,
                                                      int64_t rows_cap,
                                                      uint4* __restrict__ out, DevErr* err) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int n8 = d >> 3;
  const int upt = (n8 + cpu - 1) / cpu;
  for (int64_t u = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       u < T * upt; u += nwarps) {
    const int64_t t = u / upt;
    const int c0 = static_cast<int>(u - t * upt) * cpu;
    int row = 0;
    float g = 0.0f;
    if (lane < k) {
      row = pos[t * k + lane];
      g = gate[t * k + lane];
      if (row < 0 || row >= rows_cap) {  // recorded; row 0 is read instead
        set_error(err, MOE_ERR_DEVICE_BOUNDS, 220);
        row = 0;
      }
    }
    int rows[KC];
    float gs[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      rows[j] = __shfl_sync(0xFFFFFFFFu, row, j);
      gs[j] = __shfl_sync(0xFFFFFFFFu, g, j);
    }
    // two column steps (c and c + 32) per iteration: every slot's two 16-byte loads are in
    // flight together
#pragma unroll 1
    for (int c = c0 + lane; c < c0 + cpu && c < n8; c += 64) {
      const bool two = c + 32 < c0 + cpu && c + 32 < n8;
      uint4 v[2][KC];
#pragma unroll
      for (int j = 0; j < KC; ++j)
        if (j < k) {
          const uint4* src = y + static_cast<int64_t>(rows[j]) * n8 + c;
          v[0][j] = __ldg(src);
          if (two) v[1][j] = __ldg(src + 32);
        }
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        if (s2 == 1 && !two) break;
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
        for (int j = 0; j < KC; ++j)
          if (j < k) {
            const uint4 u = v[s2][j];
            acc[0] = __fmaf_rn(gs[j], bf16lo(u.x), acc[0]);
            acc[1] = __fmaf_rn(gs[j], bf16hi(u.x), acc[1]);
            acc[2] = __fmaf_rn(gs[j], bf16lo(u.y), acc[2]);
            acc[3] = __fmaf_rn(gs[j], bf16hi(u.y), acc[3]);
            acc[4] = __fmaf_rn(gs[j], bf16lo(u.z), acc[4]);
            acc[5] = __fmaf_rn(gs[j], bf16hi(u.z), acc[5]);
            acc[6] = __fmaf_rn(gs[j], bf16lo(u.w), acc[6]);
            acc[7] = __fmaf_rn(gs[j], bf16hi(u.w), acc[7]);
          }
        st_v4(out + t * n8 + c + 32 * s2,
              make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                         pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
      }
    }
  }
}

// dx[t] = bf16( sum_j rows[pos[t,j]] ) with fp32 rows, adds in slot order; same units.
template <int KC>
__global__ void __launch_bounds__(256) combine_f32_kernel(const float4* __restrict__ rowsp,
                                                          const int32_t* __restrict__ pos,
                                                          int64_t T, int k, int d,
                                                          uint4* __restrict__ out) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int n8 = d >> 3;
  const int upt = (n8 + kCombChunks - 1) / kCombChunks;
  for (int64_t u = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       u < T * upt; u += nwarps) {
    const int64_t t = u / upt;
    const int c0 = static_cast<int>(u - t * upt) * kCombChunks;
    const int row = lane < k ? pos[t * k + lane] : 0;
    int rows[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) rows[j] = __shfl_sync(0xFFFFFFFFu, row, j);
#pragma unroll 1
    for (int c = c0 + lane; c < c0 + kCombChunks && c < n8; c += 32) {
      float acc[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
      for (int j = 0; j < KC; ++j)
        if (j < k) {
          const float4* src = rowsp + (static_cast<int64_t>(rows[j]) * n8 + c) * 2;
          const float4 a = __ldg(src), b = __ldg(src + 1);
          acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
          acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
        }
      st_v4(out + t * n8 + c, make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                         pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7])));
    }
  }
}

// Backward of the combine and the gate, in two passes.
// Pass 1, per (token, column block) unit: dO[pos[t,j]] = bf16(gate[t,j] * dy[t]) and the
// block's partial dot products <y[pos[t,j]], dy[t]> (fp32: per-lane partials over the lane's
// columns of the block, then a fixed butterfly), stored to part[t][block][j].
// Pass 2, per token: dgate[t,j] = sum of the blocks' partials in block order,
// dlogits[t, e_j] = g_j (dgate_j - sum_i g_i dgate_i), 0 for unselected experts.
template <int KC>
__global__ void __launch_bounds__(256) bwd_gate_rows_kernel(
    const uint4* __restrict__ dy, const uint4* __restrict__ y, const float* __restrict__ gate,
    const int32_t* __restrict__ pos, int64_t T, int k, int d, uint4* __restrict__ dO,
    float* __restrict__ part) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int n8 = d >> 3;
  const int upt = (n8 + kCombChunks - 1) / kCombChunks;
  for (int64_t u = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
       u < T * upt; u += nwarps) {
    const int64_t t = u / upt;
    const int c0 = static_cast<int>(u - t * upt) * kCombChunks;
    int row = 0;
    float g = 0.0f;
    if (lane < k) {
      row = pos[t * k + lane];
      g = gate[t * k + lane];
    }
    int rows[KC];
    float gs[KC], dot[KC];
#pragma unroll
    for (int j = 0; j < KC; ++j) {
      rows[j] = __shfl_sync(0xFFFFFFFFu, row, j);
      gs[j] = __shfl_sync(0xFFFFFFFFu, g, j);
      dot[j] = 0.0f;
    }
    // two column steps (c and c + 32) per iteration: their dy and bf16 row loads are in
    // flight together; each slot's dot product still adds step c, then step c + 32
#pragma unroll 1
    for (int c = c0 + lane; c < c0 + kCombChunks && c < n8; c += 64) {
      const bool two = c + 32 < c0 + kCombChunks && c + 32 < n8;
      uint4 dv[2], yv[2][KC];
      dv[0] = ld_nc_v4(dy + t * n8 + c);
      if (two) dv[1] = ld_nc_v4(dy + t * n8 + c + 32);
#pragma unroll
      for (int j = 0; j < KC; ++j)
        if (j < k) {
          const uint4* src = y + static_cast<int64_t>(rows[j]) * n8 + c;  // bf16 row
          yv[0][j] = __ldg(src);
          if (two) yv[1][j] = __ldg(src + 32);
        }
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        if (s2 == 1 && !two) break;
        const uint32_t du[4] = {dv[s2].x, dv[s2].y, dv[s2].z, dv[s2].w};
        float dyf[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          dyf[2 * q] = bf16lo(du[q]);
          dyf[2 * q + 1] = bf16hi(du[q]);
        }
#pragma unroll
        for (int j = 0; j < KC; ++j)
          if (j < k) {
            const uint4 u4 = yv[s2][j];
            const float yf[8] = {bf16lo(u4.x), bf16hi(u4.x), bf16lo(u4.y), bf16hi(u4.y),
                                 bf16lo(u4.z), bf16hi(u4.z), bf16lo(u4.w), bf16hi(u4.w)};
#pragma unroll
            for (int q = 0; q < 8; ++q) dot[j] = __fmaf_rn(yf[q], dyf[q], dot[j]);
            uint4 o;
            o.x = pack_bf16x2(gs[j] * dyf[0], gs[j] * dyf[1]);
            o.y = pack_bf16x2(gs[j] * dyf[2], gs[j] * dyf[3]);
            o.z = pack_bf16x2(gs[j] * dyf[4], gs[j] * dyf[5]);
            o.w = pack_bf16x2(gs[j] * dyf[6], gs[j] * dyf[7]);
            st_v4(dO + static_cast<int64_t>(rows[j]) * n8 + c + 32 * s2, o);
          }
      }
    }
    float mine = 0.0f;
#pragma unroll
    for (int j = 0; j < KC; ++j)
      if (j < k) {
        float v = dot[j];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == j) mine = v;
      }
    if (lane < k) part[u * k + lane] = mine;
  }
}

__global__ void __launch_bounds__(256) bwd_gate_finish_kernel(
    const float* __restrict__ part, const float* __restrict__ gate,
    const int32_t* __restrict__ topk, int64_t T, int k, int upt, int E,
    float* __restrict__ dgate, float* __restrict__ dlogits) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t t = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; t < T;
       t += nwarps) {
    float dg = 0.0f, g = 0.0f;
    int ex = 0;
    if (lane < k) {
      for (int b = 0; b < upt; ++b) dg += part[(t * upt + b) * k + lane];
      g = gate[t * k + lane];
      ex = topk[t * k + lane];
      dgate[t * k + lane] = dg;
    }
    if (dlogits) {
      float sgd = 0.0f;
      for (int j = 0; j < k; ++j) sgd += __shfl_sync(0xFFFFFFFFu, g * dg, j);
      float* dl = dlogits + t * E;
      for (int e = lane; e < E; e += 32) dl[e] = 0.0f;
      __syncwarp();
      if (lane < k) dl[ex] = g * (dg - sgd);
    }
  }
}

int grid_for_warps(int64_t warps, int warps_per_block) {
  int64_t b = (warps + warps_per_block - 1) / warps_per_block;
  const int64_t cap = 152 * 16;
  if (b > cap) b = cap;
  if (b < 1) b = 1;
  return static_cast<int>(b);
}

// Blocks of `kern` (256 threads) resident on the whole current device at once, cached per
// device and kernel; 0 if the query fails.
template <typename K>
int resident_blocks(K kern) {
  static std::atomic<int> cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  const int c = cache[dev].load(std::memory_order_relaxed);
  if (c) return c;
  int per_sm = 0, sms = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  cache[dev].store(per_sm * sms, std::memory_order_relaxed);
  return per_sm * sms;
}

// Grid for a warp-per-unit kernel: one warp per unit, at most the resident capacity.
template <typename K>
int unit_grid(K kern, int64_t units) {
  int64_t b = (units + 7) / 8;
  const int cap = resident_blocks(kern);
  if (cap > 0 && b > cap) b = cap;
  if (b > (1ll << 30)) b = 1ll << 30;
  return static_cast<int>(b < 1 ? 1 : b);
}

// k -> kernel instantiation with KC = the next power of two >= k
#define MOE_DISPATCH_KC(k, KERNEL, ...)                      \
  ((k) <= 1 ? KERNEL<1>(__VA_ARGS__)                         \
   : (k) <= 2 ? KERNEL<2>(__VA_ARGS__)                       \
   : (k) <= 4 ? KERNEL<4>(__VA_ARGS__)                       \
   : (k) <= 8 ? KERNEL<8>(__VA_ARGS__)                       \
              : KERNEL<16>(__VA_ARGS__))

template <int KC>
cudaError_t launch_combine_kc(const uint16_t* y_rows, int64_t rows_cap, const float* gate,
                              const int32_t* pos, int64_t T, int k, int d, uint16_t* out,
                              DevErr* err, cudaStream_t s) {
  // one iteration per lane (two column steps) while the units do not fill the GPU's warps a
  // few times over
  const int64_t small_units = T * ((d / 8 + 63) / 64);
  const int cpu = small_units <= 8192 ? 64 : kCombChunks;
  const int64_t units = T * ((d / 8 + cpu - 1) / cpu);
  return launch_pdl(combine_kernel<KC>, dim3(unit_grid(combine_kernel<KC>, units)), dim3(256), 0,
                    s, reinterpret_cast<const uint4*>(y_rows), gate, pos, T, k, d, cpu, rows_cap,
                    reinterpret_cast<uint4*>(out), err);
}
template <int KC>
cudaError_t launch_combine_f32_kc(const float* rows, const int32_t* pos, int64_t T, int k, int d,
                                  uint16_t* out, cudaStream_t s) {
  const int64_t units = T * ((d / 8 + kCombChunks - 1) / kCombChunks);
  return launch_pdl(combine_f32_kernel<KC>, dim3(unit_grid(combine_f32_kernel<KC>, units)),
                    dim3(256), 0, s, reinterpret_cast<const float4*>(rows), pos, T, k, d,
                    reinterpret_cast<uint4*>(out));
}
template <int KC>
cudaError_t launch_bwd_gate_kc(const uint16_t* dy, const uint16_t* y_rows, const float* gate,
                               const int32_t* pos, int64_t T, int k, int d, uint16_t* dO_rows,
                               float* part, cudaStream_t s) {
  const int64_t units = T * ((d / 8 + kCombChunks - 1) / kCombChunks);
  return launch_pdl(bwd_gate_rows_kernel<KC>, dim3(unit_grid(bwd_gate_rows_kernel<KC>, units)),
                    dim3(256), 0, s, reinterpret_cast<const uint4*>(dy),
                    reinterpret_cast<const uint4*>(y_rows), gate, pos, T, k, d,
                    reinterpret_cast<uint4*>(dO_rows), part);
}

}  // namespace

cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int32_t* topk,
                              float* gate, int32_t* pos_local, int32_t* hist, DevErr* err,
                              cudaStream_t s) {
  (void)err;
  const int64_t nblk = (T + kRouteTokensPerBlock - 1) / kRouteTokensPerBlock;
  if (nblk == 0) return cudaSuccess;
  const size_t smem = (8 * static_cast<size_t>(E) + 2 * kRouteTokensPerBlock * kMaxK) * 4;
  const int epl = (E + 31) / 32;
  void (*kern)(const float*, int64_t, int, int, int32_t*, float*, int32_t*, int32_t*);
  if (epl <= 1) kern = route_topk_kernel<1>;
  else if (epl <= 2) kern = route_topk_kernel<2>;
  else if (epl <= 4) kern = route_topk_kernel<4>;
  else if (epl <= 8) kern = route_topk_kernel<8>;
  else if (epl <= 16) kern = route_topk_kernel<16>;
  else kern = route_topk_kernel<32>;
  cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
  if (st != cudaSuccess) return st;
  return launch_pdl(kern, dim3(static_cast<unsigned>(nblk)), dim3(kRouteWarps * 32), smem, s,
                    logits, T, E, k, topk, gate, pos_local, hist);
}

size_t small_dispatch_smem(int E) {
  return (10 * static_cast<size_t>(E) + 1 + 2 * kRouteTokensPerBlock * kMaxK) * 4;
}

cudaError_t launch_dispatch_small(const float* logits, const uint16_t* x, int64_t T, int d,
                                  int E, int k, int align, int32_t* topk, float* gate,
                                  int32_t* pos, int32_t* perm, int32_t* counts,
                                  int32_t* offsets, int32_t* poff, const TileTables* tables,
                                  uint16_t* x_perm, int64_t rows_cap, int num_sms, DevErr* err,
                                  cudaStream_t s) {
  if (T <= 0 || T > kRouteTokensPerBlock || E > 1024) return cudaErrorInvalidValue;
  const size_t smem = small_dispatch_smem(E);
  const int epl = (E + 31) / 32;
  void (*kern)(const float*, const uint4*, int, int, int, int, int, int32_t*, float*, int32_t*,
               int32_t*, int32_t*, int32_t*, int32_t*, TileTables, int, uint4*, int64_t,
               DevErr*);
  if (epl <= 1) kern = dispatch_small_kernel<1>;
  else if (epl <= 2) kern = dispatch_small_kernel<2>;
  else if (epl <= 4) kern = dispatch_small_kernel<4>;
  else if (epl <= 8) kern = dispatch_small_kernel<8>;
  else if (epl <= 16) kern = dispatch_small_kernel<16>;
  else kern = dispatch_small_kernel<32>;
  cudaError_t st = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        static_cast<int>(smem));
  if (st != cudaSuccess) return st;
  TileTables tt{};
  if (tables) tt = *tables;
  // CTA 0 for the routing outputs and tables, then one CTA per 1024 16-byte chunks of the
  // token rows (at least one), at most one CTA per SM
  const int64_t chunks = x_perm ? T * (d / 8) : 0;
  int64_t g = 1 + (chunks > 0 ? (chunks + 1023) / 1024 : 1);
  if (g > num_sms) g = num_sms;
  return launch_pdl(kern, dim3(static_cast<unsigned>(g)), dim3(1024), smem, s, logits,
                    reinterpret_cast<const uint4*>(x), static_cast<int>(T), d, E, k, align, topk,
                    gate, pos, perm, counts, offsets, poff, tt, tables ? 1 : 0,
                    reinterpret_cast<uint4*>(x_perm), rows_cap, err);
}

cudaError_t launch_scan_cols(const int32_t* hist, int64_t nblk, int E, int32_t* bbase,
                             int32_t* counts, cudaStream_t s) {
  return launch_pdl(scan_cols_kernel, dim3((E + 31) / 32), dim3(256), 0, s, hist, nblk, E, bbase,
                    counts);
}

cudaError_t launch_offsets(const int32_t* counts, int E, int align, int32_t* offsets,
                           int32_t* poff, const TileTables* tables, DevErr* err,
                           cudaStream_t s) {
  TileTables tt{};
  if (tables) tt = *tables;
  return launch_pdl(offsets_kernel, dim3(1), dim3(1024), 0, s, counts, E, align, offsets, poff, tt,
                    tables ? 1 : 0, err);
}

cudaError_t launch_scatter(const uint16_t* x, int64_t T, int d, int E, int k,
                           const int32_t* topk, const int32_t* bbase, const int32_t* poff,
                           int32_t* pos, int32_t* perm, uint16_t* x_perm, int64_t rows_cap,
                           DevErr* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(scatter_kernel, dim3(grid_for_warps(T, 8)), dim3(256), 0, s,
                    reinterpret_cast<const uint4*>(x), T, d, E, k, topk, bbase, poff, pos, perm,
                    reinterpret_cast<uint4*>(x_perm), rows_cap, err);
}

cudaError_t launch_scatter_fp8(const uint16_t* x, int64_t T, int d, int E, int k,
                               const int32_t* topk, const int32_t* bbase, const int32_t* poff,
                               int32_t* pos, int32_t* perm, uint8_t* x_perm, float* xscale,
                               int64_t rows_cap, DevErr* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(scatter_fp8_kernel, dim3(grid_for_warps(T, 8)), dim3(256), 0, s,
                    reinterpret_cast<const uint4*>(x), T, d, E, k, topk, bbase, poff, pos, perm,
                    x_perm, xscale, rows_cap, err);
}

cudaError_t launch_quantize_weights_fp8(const uint16_t* W, int E, int K, int N, uint8_t* Wq,
                                        float* scales, cudaStream_t s) {
  return launch_pdl(quantize_weights_fp8_kernel, dim3(N / 32, E), dim3(256), 0, s, W, K, N, Wq,
                    scales);
}

cudaError_t launch_pad_rows(const int32_t* counts, const int32_t* poff, int E, int32_t* perm,
                            void* rows, int64_t row_bytes, cudaStream_t s) {
  return launch_pdl(pad_rows_kernel, dim3(E), dim3(256), 0, s, counts, poff, perm,
                    reinterpret_cast<uint4*>(rows), row_bytes / 16);
}

cudaError_t launch_combine(const uint16_t* y_rows, int64_t rows_cap, const float* gate,
                           const int32_t* pos, int64_t T, int k, int d, uint16_t* out,
                           DevErr* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return MOE_DISPATCH_KC(k, launch_combine_kc, y_rows, rows_cap, gate, pos, T, k, d, out, err,
                         s);
}

cudaError_t launch_bwd_gate(const uint16_t* dy, const uint16_t* y_rows, const float* gate,
                            const int32_t* pos, const int32_t* topk, int64_t T, int k, int d,
                            int E, uint16_t* dO_rows, float* dgate, float* dlogits, float* part,
                            cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const cudaError_t st =
      MOE_DISPATCH_KC(k, launch_bwd_gate_kc, dy, y_rows, gate, pos, T, k, d, dO_rows, part, s);
  if (st != cudaSuccess) return st;
  const int upt = (d / 8 + kCombChunks - 1) / kCombChunks;
  return launch_pdl(bwd_gate_finish_kernel, dim3(grid_for_warps(T, 8)), dim3(256), 0, s, part,
                    gate, topk, T, k, upt, E, dgate, dlogits);
}

cudaError_t launch_combine_f32(const float* rows, const int32_t* pos, int64_t T, int k, int d,
                               uint16_t* out, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return MOE_DISPATCH_KC(k, launch_combine_f32_kc, rows, pos, T, k, d, out, s);
}

}  // namespace moe
