// Grouped expert GEMMs on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// The expert stage is Linear -> SwiGLU -> Linear per expert (DeepSeek-V4 report reading,
// 10100.com, section on fine-grained EP overlap; report translation, itsolotime.com,
// section 1.4: gate, up and down projections, 6hd FLOP per token-expert pair).  Every kind
// below is one persistent, warp-specialised kernel:
//   warp 0      TMA producer (one lane): operand tiles -> a ring of shared-memory stages
//   warp 1      MMA issuer (one lane): tcgen05.mma 128 x BN x 16 into a TMEM accumulator
//   warp 2      TMEM allocator
//   warps 4..7  epilogue: tcgen05.ld of the accumulator, activation, global stores
// Two TMEM accumulators alternate so the epilogue of tile i overlaps the MMAs of tile i+1.
//
// Batch invariance and determinism (report translation, section 3; 10100.com reading):
// the tile shape (128 x BN x 64), the K order and therefore each output element's
// accumulation order are fixed by the model sizes alone, never by T or by the expert
// loads; there is no split-K and no atomic accumulation; which CTA computes a tile does
// not change its value.
//
// Row layout: the permuted rows of every expert start at a multiple of 128 (padded
// offsets), so each 128-row tile belongs to one expert; padding rows are masked in the
// epilogues (or written as zeros where a later K-over-rows GEMM reads them).
#pragma once

#include <cuda.h>

#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace moe {

enum GemmKind : int {
  kFwd1 = 0,  // H = bf16(silu(Xp W1) * (Xp W3)), optional fp32 A/B save   (rows x dff)
  kFwd2 = 1,  // Y = H W2 (fp32 rows for the fp32 combine)                  (rows x d)
  kDh = 2,    // dH = dO W2^T -> dA, dB (bf16) through the SwiGLU backward (rows x dff)
  kDx = 3,    // dXp = [dA|dB] [W1|W3]^T (fp32)                            (rows x d)
  kDw2 = 4,   // dW2[e] = H^T dO (fp32)                                    (dff x d)
  kDw13 = 5,  // [dW1|dW3][e] = Xp^T [dA|dB] (fp32)                         (d x 2dff)
};

template <int KIND>
struct KindTraits {
  static constexpr bool kRowsM = (KIND <= kDx);      // M = permuted rows, K fixed
  static constexpr int kAmn = (KIND >= kDw2) ? 1 : 0;  // A operand MN-major?
  static constexpr int kBmn = (KIND == kDh || KIND == kDx) ? 0 : 1;
};

struct GemmParams {
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
};

constexpr int kBM = 128;
constexpr int kBK = 64;
constexpr uint32_t kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kEpiThreads = 128;

template <int BN>
struct GemmCfg {
  static constexpr int kStages = (BN == 256) ? 4 : 6;
  static constexpr uint32_t kBBytes = BN * kBK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kTmemCols = 2 * BN;
  static constexpr size_t kSmemBytes = static_cast<size_t>(kStages) * kStageBytes + 1024 + 256;
};

struct TileInfo {
  int e;      // expert
  int row0;   // first permuted row (row-grouped) / first K row (K-over-rows)
  int nvalid; // valid rows of the tile (row-grouped)
  int m0;     // first M index (K-over-rows)
  int n0;     // first N index
  int nk;     // number of 64-wide K blocks
  bool bad;   // tile tables out of range: every role skips the tile
};

template <int KIND, int BN>
__device__ __forceinline__ TileInfo decode_tile(const GemmParams& p, int tile) {
  TileInfo ti;
  if constexpr (KindTraits<KIND>::kRowsM) {
    const int mt = tile / p.nb;
    ti.n0 = (tile % p.nb) * BN;
    ti.e = p.mt_expert[mt];
    ti.row0 = p.mt_row0[mt];
    ti.nvalid = p.poff[ti.e] + p.counts[ti.e] - ti.row0;
    ti.m0 = 0;
    ti.nk = p.nkb;
    ti.bad = ti.e < 0 || ti.e >= p.E || ti.row0 < 0 || ti.row0 + kBM > p.rows_cap;
  } else {
    const int per_e = p.mb * p.nb;
    ti.e = tile / per_e;
    const int rem = tile % per_e;
    ti.m0 = (rem / p.nb) * kBM;
    ti.n0 = (rem % p.nb) * BN;
    ti.row0 = p.poff[ti.e];
    ti.nk = (p.poff[ti.e + 1] - p.poff[ti.e]) / kBK;
    ti.nvalid = kBM;
    ti.bad = ti.row0 < 0 || ti.nk < 0 || ti.row0 + ti.nk * kBK > p.rows_cap;
  }
  return ti;
}

__device__ __forceinline__ float silu_f(float a) { return a / (1.0f + expf(-a)); }

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

// Epilogue of one tile for one thread (= one accumulator row).
template <int KIND, int BN>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, const TileInfo& ti,
                                              uint32_t tacc, int r) {
  const bool valid = r < ti.nvalid;
  if constexpr (KIND == kFwd1) {
    constexpr int HALF = BN / 2;
    const int64_t row = ti.row0 + r;
    const int c0 = ti.n0 / 2;  // h column of this tile's first accumulator column
    uint16_t* H = static_cast<uint16_t*>(p.out0) + row * p.dff + c0;
#pragma unroll 1
    for (int ch = 0; ch < HALF / 16; ++ch) {
      float a[16], b[16];
      tmem_ld16x2(tacc + ch * 16, tacc + HALF + ch * 16, a, b);
      if (valid) {
        float h[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) h[i] = silu_f(a[i]) * b[i];
        st_bf16x16(H + ch * 16, h);
        if (p.save_ab) {
          st_f32x16(p.save_a + row * p.dff + c0 + ch * 16, a);
          st_f32x16(p.save_b + row * p.dff + c0 + ch * 16, b);
        }
      } else {
        st_zero32(H + ch * 16);
      }
    }
  } else if constexpr (KIND == kFwd2) {
    const int64_t row = ti.row0 + r;
    float* Y = static_cast<float*>(p.out0) + row * p.d + ti.n0;
#pragma unroll 1
    for (int ch = 0; ch < BN / 16; ++ch) {
      float v[16];
      tmem_ld16(tacc + ch * 16, v);
      if (valid) st_f32x16(Y + ch * 16, v);
    }
  } else if constexpr (KIND == kDh) {
    const int64_t row = ti.row0 + r;
    uint16_t* dA = static_cast<uint16_t*>(p.out0) + row * (2 * p.dff) + ti.n0;
    uint16_t* dB = dA + p.dff;
    const float* sa = p.save_a + row * p.dff + ti.n0;
    const float* sb = p.save_b + row * p.dff + ti.n0;
#pragma unroll 1
    for (int ch = 0; ch < BN / 16; ++ch) {
      float dh[16];
      tmem_ld16(tacc + ch * 16, dh);
      if (valid) {
        float a[16], b[16], da[16], db[16];
        ld_f32x16(sa + ch * 16, a);
        ld_f32x16(sb + ch * 16, b);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float sg = 1.0f / (1.0f + expf(-a[i]));
          da[i] = dh[i] * b[i] * (sg * (1.0f + a[i] * (1.0f - sg)));
          db[i] = dh[i] * (a[i] * sg);
        }
        st_bf16x16(dA + ch * 16, da);
        st_bf16x16(dB + ch * 16, db);
      } else {
        st_zero32(dA + ch * 16);
        st_zero32(dB + ch * 16);
      }
    }
  } else if constexpr (KIND == kDx) {
    const int64_t row = ti.row0 + r;
    float* out = static_cast<float*>(p.out0) + row * p.d + ti.n0;
#pragma unroll 1
    for (int ch = 0; ch < BN / 16; ++ch) {
      float v[16];
      tmem_ld16(tacc + ch * 16, v);
      if (valid) st_f32x16(out + ch * 16, v);
    }
  } else {
    // K-over-rows kinds: output row m0 + r of expert e's weight gradient.
    float* out;
    int ld;
    if constexpr (KIND == kDw2) {
      ld = p.d;
      out = static_cast<float*>(p.out0) +
            (static_cast<int64_t>(ti.e) * p.dff + ti.m0 + r) * p.d + ti.n0;
    } else {
      ld = p.dff;
      const bool first = ti.n0 < p.dff;
      float* base = static_cast<float*>(first ? p.out0 : p.out1);
      out = base + (static_cast<int64_t>(ti.e) * p.d + ti.m0 + r) * p.dff +
            (first ? ti.n0 : ti.n0 - p.dff);
    }
    (void)ld;
#pragma unroll 1
    for (int ch = 0; ch < BN / 16; ++ch) {
      float v[16];
      if (ti.nk > 0) {
        tmem_ld16(tacc + ch * 16, v);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = 0.0f;
      }
      st_f32x16(out + ch * 16, v);
    }
  }
}

template <int KIND, int BN>
__global__ void __launch_bounds__(256, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA,
                        const __grid_constant__ CUtensorMap mapB0,
                        const __grid_constant__ CUtensorMap mapB1, const GemmParams p) {
  using Cfg = GemmCfg<BN>;
  using Tr = KindTraits<KIND>;
  constexpr int S = Cfg::kStages;
  constexpr uint32_t IDESC = idesc_bf16_f32(kBM, BN, Tr::kAmn, Tr::kBmn);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bar0 = base + S * Cfg::kStageBytes;
  // barrier block: full[S], empty[S], tfull[2], tempty[2], drain  (8 bytes each)
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (S + s); };
  auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * S + 2 + a); };
  const uint32_t drain_bar = bar0 + 8u * (2 * S + 4);
  uint8_t* misc = gbase + S * Cfg::kStageBytes + 8 * (2 * S + 5);
  volatile uint32_t* tmem_holder = reinterpret_cast<volatile uint32_t*>(misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);
  volatile uint32_t* consumed = reinterpret_cast<volatile uint32_t*>(misc + 8);
  auto stage_a = [&](int s) { return base + s * Cfg::kStageBytes; };
  auto stage_b = [&](int s) { return base + s * Cfg::kStageBytes + kABytes; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull_bar(a), 1);
      mbar_init(tempty_bar(a), kEpiThreads);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    *consumed = 0u;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32(const_cast<uint32_t*>(tmem_holder)), Cfg::kTmemCols);
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;

  int64_t ntiles64;
  if constexpr (Tr::kRowsM) ntiles64 = static_cast<int64_t>(p.n_mt[0]) * p.nb;
  else ntiles64 = static_cast<int64_t>(p.E) * p.mb * p.nb;
  if (ntiles64 > p.max_tiles || ntiles64 < 0) {
    if (threadIdx.x == 0) set_error(p.err, MOE_ERR_DEVICE_BOUNDS, 10);
    ntiles64 = 0;
  }
  const int ntiles = static_cast<int>(ntiles64);

  uint32_t issued = 0;
  int skipped = -1;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------------ TMA producer
    tma_prefetch_desc(&mapA);
    tma_prefetch_desc(&mapB0);
    tma_prefetch_desc(&mapB1);
    uint32_t fill = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const TileInfo ti = decode_tile<KIND, BN>(p, tile);
      if (ti.bad) {
        set_error(p.err, MOE_ERR_DEVICE_BOUNDS, 11);
        continue;
      }
      for (int kb = 0; kb < ti.nk; ++kb) {
        const int s = fill % S;
        const uint32_t ph = (fill / S) & 1u;
        if (!mbar_wait(empty_bar(s), ph ^ 1u, abort_flag, p.err, 1, p.wait_ns)) {
          ok = false;
          break;
        }
        const uint32_t fb = full_bar(s), sa = stage_a(s), sb = stage_b(s);
        if ((p.debug_flags & 1) && blockIdx.x == 0 && fill == 0) {
          skipped = 0;  // test hook: this stage is never filled
        } else {
          mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          const int k0 = kb * kBK;
          if constexpr (KIND == kFwd1) {
            tma_load_2d(sa, &mapA, fb, k0, ti.row0);
            const int wrow = ti.e * p.d + k0;
#pragma unroll
            for (int i = 0; i < BN / 128; ++i) {
              tma_load_2d(sb + 8192u * i, &mapB0, fb, ti.n0 / 2 + 64 * i, wrow);
              tma_load_2d(sb + 8192u * (BN / 128 + i), &mapB1, fb, ti.n0 / 2 + 64 * i, wrow);
            }
          } else if constexpr (KIND == kFwd2) {
            tma_load_2d(sa, &mapA, fb, k0, ti.row0);
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
              tma_load_2d(sb + 8192u * i, &mapB0, fb, ti.n0 + 64 * i, ti.e * p.dff + k0);
          } else if constexpr (KIND == kDh) {
            tma_load_2d(sa, &mapA, fb, k0, ti.row0);
            tma_load_2d(sb, &mapB0, fb, k0, ti.e * p.dff + ti.n0);
          } else if constexpr (KIND == kDx) {
            tma_load_2d(sa, &mapA, fb, k0, ti.row0);
            if (k0 < p.dff) tma_load_2d(sb, &mapB0, fb, k0, ti.e * p.d + ti.n0);
            else tma_load_2d(sb, &mapB1, fb, k0 - p.dff, ti.e * p.d + ti.n0);
          } else {
            const int r = ti.row0 + k0;
            tma_load_2d(sa, &mapA, fb, ti.m0, r);
            tma_load_2d(sa + 8192u, &mapA, fb, ti.m0 + 64, r);
#pragma unroll
            for (int i = 0; i < BN / 64; ++i) tma_load_2d(sb + 8192u * i, &mapB0, fb, ti.n0 + 64 * i, r);
          }
        }
        ++fill;
      }
    }
    issued = fill;
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------------ MMA issuer
    uint32_t fill = 0;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
      const TileInfo ti = decode_tile<KIND, BN>(p, tile);
      if (ti.bad) continue;
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1u;
      if (!mbar_wait(tempty_bar(acc), aph ^ 1u, abort_flag, p.err, 2, p.wait_ns)) break;
      tc_fence_after();
      const uint32_t dtm = tmem_base + acc * BN;
      for (int kb = 0; kb < ti.nk; ++kb) {
        const int s = fill % S;
        const uint32_t ph = (fill / S) & 1u;
        if (!mbar_wait(full_bar(s), ph, abort_flag, p.err, 3, p.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = stage_a(s), sb = stage_b(s);
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t ad = Tr::kAmn ? smem_desc_sw128(sa + kk * 2048u, 8192u, 1024u)
                                       : smem_desc_sw128(sa + kk * 32u, 16u, 1024u);
          const uint64_t bd = Tr::kBmn ? smem_desc_sw128(sb + kk * 2048u, 8192u, 1024u)
                                       : smem_desc_sw128(sb + kk * 32u, 16u, 1024u);
          umma_f16(dtm, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
        }
        umma_commit(empty_bar(s));
        ++fill;
        *consumed = fill;
      }
      if (!ok) break;
      umma_commit(tfull_bar(acc));
      ++it;
    }
    // all MMAs issued by this thread complete before TMEM is released
    umma_commit(drain_bar);
    mbar_wait(drain_bar, 0u, nullptr, p.err, 4, p.wait_ns);
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ epilogue
    const int q = warp - 4;
    const int r = q * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const TileInfo ti = decode_tile<KIND, BN>(p, tile);
      if (ti.bad) continue;
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1u;
      // warp-uniform decision: the tcgen05.ld below is .sync.aligned
      const bool ok = mbar_wait(tfull_bar(acc), aph, abort_flag, p.err, 5, p.wait_ns);
      if (!__all_sync(0xFFFFFFFFu, ok)) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      epilogue_tile<KIND, BN>(p, ti, tacc, r);
      tc_fence_before();
      mbar_arrive(tempty_bar(acc));
      ++it;
    }
  }

  __syncthreads();
  if (warp == 0 && lane == 0) {
    // wait for every operand load still in flight (only after an abort)
    for (uint32_t f = *consumed; f < issued; ++f) {
      if (static_cast<int>(f) == skipped) continue;
      const int s = f % S;
      uint64_t t0 = global_ns();
      while (!mbar_try_wait(full_bar(s), (f / S) & 1u)) {
        if (global_ns() - t0 > p.wait_ns) break;
      }
    }
  }
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::kTmemCols);
  }
}

// ------------------------------------------------------------------ host side
CUtensorMap make_map_2d(const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_rows, cudaError_t* st);

template <int KIND, int BN>
cudaError_t run_grouped_gemm(const CUtensorMap& a, const CUtensorMap& b0, const CUtensorMap& b1,
                             const GemmParams& p, int64_t max_tiles, int num_sms,
                             cudaStream_t s) {
  using Cfg = GemmCfg<BN>;
  // the opt-in shared-memory size is a per-device function attribute: set it once per device
  static unsigned long long attr_set_mask = 0ull;
  int dev = 0;
  cudaError_t st = cudaGetDevice(&dev);
  if (st != cudaSuccess) return st;
  if (dev < 64 && !(attr_set_mask & (1ull << dev))) {
    st = cudaFuncSetAttribute(grouped_gemm_kernel<KIND, BN>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(Cfg::kSmemBytes));
    if (st != cudaSuccess) return st;
    attr_set_mask |= 1ull << dev;
  }
  GemmParams pp = p;
  pp.max_tiles = max_tiles;
  int64_t grid = max_tiles < num_sms ? max_tiles : num_sms;
  if (grid < 1) grid = 1;
  grouped_gemm_kernel<KIND, BN><<<static_cast<unsigned>(grid), 256, Cfg::kSmemBytes, s>>>(a, b0, b1, pp);
  return cudaGetLastError();
}

}  // namespace moe
