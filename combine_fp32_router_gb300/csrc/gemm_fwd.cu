// Forward grouped GEMMs: GEMM1 + SwiGLU (H) and GEMM2 (Y), plus the tensor-map helpers.
#include <mutex>

#include "gemm.cuh"

namespace moe {

void* tensor_map_encoder() {
  static void* fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = f;
  });
  return fn;
}

// 2-D bf16 tensor map with 128-byte swizzle: `rows` rows of `inner` elements, row pitch
// `row_bytes`; box of box_inner x box_rows elements (box_inner * 2 == 128 bytes).
CUtensorMap make_map_2d(const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                        uint32_t box_inner, uint32_t box_rows, cudaError_t* st) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  CUtensorMap m;
  std::memset(&m, 0, sizeof m);
  auto enc = reinterpret_cast<Encode>(tensor_map_encoder());
  if (!enc) {
    *st = cudaErrorNotSupported;
    return m;
  }
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) *st = cudaErrorInvalidValue;
  return m;
}

// 2-D byte (E4M3) tensor map with 128-byte swizzle: boxes of 128 bytes x box_rows rows.
CUtensorMap make_map_2d_u8(const void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                           uint32_t box_rows, cudaError_t* st) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  CUtensorMap m;
  std::memset(&m, 0, sizeof m);
  auto enc = reinterpret_cast<Encode>(tensor_map_encoder());
  if (!enc) {
    *st = cudaErrorNotSupported;
    return m;
  }
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {128, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) *st = cudaErrorInvalidValue;
  return m;
}

// 2-D fp32 tensor map for TMA stores of 32 x 32 boxes with 128-byte swizzle.
CUtensorMap make_store_map_f32(void* base, uint64_t inner, uint64_t rows, uint64_t row_bytes,
                               cudaError_t* st) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  CUtensorMap m;
  std::memset(&m, 0, sizeof m);
  auto enc = reinterpret_cast<Encode>(tensor_map_encoder());
  if (!enc) {
    *st = cudaErrorNotSupported;
    return m;
  }
  const cuuint64_t dims[2] = {inner, rows};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(&m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, base, dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) *st = cudaErrorInvalidValue;
  return m;
}

GemmParams base_params(const GemmCtx& c) {
  const WsLayout& L = *c.L;
  GemmParams p{};
  p.E = L.E;
  p.d = L.d;
  p.dff = L.dff;
  p.n_mt = reinterpret_cast<const int32_t*>(c.ws + L.n_mt);
  p.mt_expert = reinterpret_cast<const int32_t*>(c.ws + L.mt_expert);
  p.mt_row0 = reinterpret_cast<const int32_t*>(c.ws + L.mt_row0);
  p.n_pt = reinterpret_cast<const int32_t*>(c.ws + L.n_pt);
  p.pt_expert = reinterpret_cast<const int32_t*>(c.ws + L.pt_expert);
  p.pt_row0 = reinterpret_cast<const int32_t*>(c.ws + L.pt_row0);
  p.counts = reinterpret_cast<const int32_t*>(c.ws + L.counts);
  p.poff = reinterpret_cast<const int32_t*>(c.ws + L.poff);
  p.err = c.err;
  p.wait_ns = c.wait_ns;
  p.debug_flags = c.debug_flags;
  p.rows_cap = c.rows ? c.rows_cap : L.P_pad;
  p.gated = c.gated ? 1 : 0;
  return p;
}

// The same parameters with the leftover-tile table in place of the 128-row tile table.
GemmParams leftover_params(const GemmParams& p, const GemmCtx& c) {
  GemmParams lo = p;
  lo.n_mt = reinterpret_cast<const int32_t*>(c.ws + c.L->n_lo);
  lo.mt_expert = reinterpret_cast<const int32_t*>(c.ws + c.L->lo_expert);
  lo.mt_row0 = reinterpret_cast<const int32_t*>(c.ws + c.L->lo_row0);
  return lo;
}

cudaError_t launch_gemm_fwd1(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  cudaError_t st = cudaSuccess;
  // A rows: the permuted copy (with gather_x the kernel copies the rows from x itself and
  // this map is not read)
  const CUtensorMap a = make_map_2d(c.ws + L.xperm, L.d, L.P_pad, 2ull * L.d, 64, 128, &st);
  const CUtensorMap b0 = make_map_2d(c.W1, L.dff, static_cast<uint64_t>(L.E) * L.d, 2ull * L.dff, 64, 64, &st);
  // without W3 (squared ReLU) the second B map is never read
  const CUtensorMap b1 = make_map_2d(c.gated ? c.W3 : c.W1, L.dff, static_cast<uint64_t>(L.E) * L.d,
                                     2ull * L.dff, 64, 64, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = base_params(c);
  // SwiGLU: 128 h columns per tile (W1 half + W3 half = 256 accumulator columns);
  // squared ReLU: 256 h columns of W1 per tile
  p.nb = c.gated ? L.dff / 128 : L.dff / 256;
  p.nkb = L.d / kBK;
  p.out0 = c.ws + L.H;
  p.save_ab = c.save_ab;
  p.save_a = c.save_ab ? reinterpret_cast<float*>(c.ws + L.Asave) : nullptr;
  p.save_b = c.save_ab ? reinterpret_cast<float*>(c.ws + L.Bsave) : nullptr;
  p.gather_x = c.gather_x ? 1 : 0;
  p.gather_src = c.x;
  p.perm = reinterpret_cast<const int32_t*>(c.ws + L.perm);
  p.k = L.k;
  return run_rows_kind<kFwd1, 256>(c.pair, a, b0, b1, b0, b1, p, leftover_params(p, c), L.max_mt,
                                   c.num_sms, s);
}

cudaError_t launch_gemm_fwd1_fp8(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  cudaError_t st = cudaSuccess;
  // A = E4M3 permuted rows [P_pad][d] bytes; B = E4M3 W1 / W3 transposed, [E * dff][d] bytes
  // (one row per output column, K-major); 128 x 128-byte boxes for pairs and single CTAs
  const CUtensorMap a = make_map_2d_u8(c.ws + L.xperm, L.d, L.P_pad, L.d, 128, &st);
  const uint64_t wrows = static_cast<uint64_t>(L.E) * L.dff;
  const CUtensorMap b0 = make_map_2d_u8(c.W1q, L.d, wrows, L.d, 128, &st);
  const CUtensorMap b1 = make_map_2d_u8(c.W3q, L.d, wrows, L.d, 128, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = base_params(c);
  p.nb = L.dff / 128;  // 128 h columns per tile (W1 half + W3 half)
  p.nkb = L.d / 128;   // 128 K elements per stage
  p.out0 = c.ws + L.H;
  p.perm = reinterpret_cast<const int32_t*>(c.ws + L.perm);
  p.k = L.k;
  p.xscale = reinterpret_cast<const float*>(c.ws + L.xscale);
  p.wscale1 = c.wscale1;
  p.wscale3 = c.wscale3;
  return run_rows_kind<kFwd1F8, 256>(c.pair, a, b0, b1, b0, b1, p, leftover_params(p, c),
                                     L.max_mt, c.num_sms, s);
}

cudaError_t launch_gemm_fwd2(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  cudaError_t st = cudaSuccess;
  const CUtensorMap a = make_map_2d(c.ws + L.H, L.dff, L.P_pad, 2ull * L.dff, 64, 128, &st);
  const CUtensorMap b0 = make_map_2d(c.W2, L.d, static_cast<uint64_t>(L.E) * L.dff, 2ull * L.d, 64, 64, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = base_params(c);
  p.nkb = L.dff / kBK;
  p.out0 = c.ws + L.Y;
  const int BN = (L.d % 256 == 0) ? 256 : 128;
  p.nb = L.d / BN;
  p.fuse_combine = c.fuse_combine ? 1 : 0;
  p.perm = reinterpret_cast<const int32_t*>(c.ws + L.perm);
  p.pos = reinterpret_cast<const int32_t*>(c.ws + L.pos);
  p.gate = reinterpret_cast<const float*>(c.ws + L.gate);
  p.seg_count = reinterpret_cast<int32_t*>(c.ws + L.seg);
  p.comb_out = c.out;
  p.k = L.k;
  const GemmParams lo = leftover_params(p, c);
  if (BN == 256)
    return run_rows_kind<kFwd2, 256>(c.pair, a, b0, b0, b0, b0, p, lo, L.max_mt, c.num_sms, s);
  return run_rows_kind<kFwd2, 128>(c.pair, a, b0, b0, b0, b0, p, lo, L.max_mt, c.num_sms, s);
}

// Swapped forward GEMMs: one CTA-pair launch over every (row block, weight-column block).
// The row operand has four tensor maps, with boxes of 16, 32, 64 and 128 rows: each CTA of a
// pair loads half of the block's rows, rounded up to one of these.
cudaError_t row_maps(GemmParams& p, const void* rows, uint64_t inner, uint64_t nrows,
                     uint64_t row_bytes) {
  cudaError_t st = cudaSuccess;
  for (int i = 0; i < 4; ++i)
    p.mapR[i] = make_map_2d(rows, inner, nrows, row_bytes, 64, 16u << i, &st);
  return st;
}
GemmParams swap_params(const GemmCtx& c) {
  GemmParams p = base_params(c);
  p.n_st = reinterpret_cast<const int32_t*>(c.ws + c.L->n_st);
  p.st_expert = reinterpret_cast<const int32_t*>(c.ws + c.L->st_expert);
  p.st_row0 = reinterpret_cast<const int32_t*>(c.ws + c.L->st_row0);
  return p;
}

cudaError_t launch_gemm_fwd1_swap(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  cudaError_t st = cudaSuccess;
  // M operand: W1 and W3 viewed as [E d rows][dff] (64-column boxes of 64 K rows)
  const CUtensorMap w1 = make_map_2d(c.W1, L.dff, static_cast<uint64_t>(L.E) * L.d, 2ull * L.dff, 64, 64, &st);
  const CUtensorMap w3 = make_map_2d(c.gated ? c.W3 : c.W1, L.dff, static_cast<uint64_t>(L.E) * L.d,
                                     2ull * L.dff, 64, 64, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = swap_params(c);
  // the rows: the workspace's x_perm, or the caller's (moe_expert_forward; the map ends at
  // their last row, so nothing past it is read)
  if (c.rows) st = row_maps(p, c.rows, L.d, static_cast<uint64_t>(c.rows_cap), 2ull * L.d);
  else st = row_maps(p, c.ws + L.xperm, L.d, L.P_pad, 2ull * L.d);
  if (st != cudaSuccess) return st;
  p.nb = c.gated ? L.dff / 128 : L.dff / 256;
  p.nkb = L.d / kBK;
  p.out0 = c.ws + L.H;
  p.save_ab = c.save_ab;
  p.save_a = c.save_ab ? reinterpret_cast<float*>(c.ws + L.Asave) : nullptr;
  p.save_b = c.save_ab ? reinterpret_cast<float*>(c.ws + L.Bsave) : nullptr;
  if (c.copy_rows) {
    // the kernel's copy warps write the permuted rows the tiles read (see GemmParams)
    p.copy_rows = 1;
    p.copy_dst = reinterpret_cast<uint16_t*>(c.ws + L.xperm);
    p.gather_src = c.x;
    p.perm = reinterpret_cast<const int32_t*>(c.ws + L.perm);
    p.k = L.k;
    p.done1 = reinterpret_cast<int32_t*>(c.ws + L.done1);
  }
  // 8 epilogue warps (kFwd1TW) where an average expert fills a 256-row block, P >= 256 E:
  // measured on GB300 at d=7168, E=256, top-8, d_ff=2048, GEMM1 of T=16384 (P = 512 E)
  // 5.71 -> 5.63 ms, of T=1024 (P = 32 E) 1.029 -> 1.059 ms with 8 warps
  if (L.T > kTileRows && L.P >= 256ll * L.E)
    return run_grouped_gemm<kFwd1TW, 256, true>(w1, w1, w3, p, L.max_mt * p.nb, c.num_sms, s);
  return run_grouped_gemm<kFwd1T, 256, true>(w1, w1, w3, p, L.max_mt * p.nb, c.num_sms, s);
}

cudaError_t launch_gemm_fwd2_swap(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  cudaError_t st = cudaSuccess;
  // M operand: W2 viewed as [E dff rows][d] (64-column boxes of 64 K rows)
  const CUtensorMap w2 = make_map_2d(c.W2, L.d, static_cast<uint64_t>(L.E) * L.dff, 2ull * L.d, 64, 64, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = swap_params(c);
  st = row_maps(p, c.ws + L.H, L.dff, L.P_pad, 2ull * L.dff);
  if (st != cudaSuccess) return st;
  p.nb = (L.d + 255) / 256;  // d % 256 == 128: the last block's second CTA has no columns
  p.nkb = L.dff / kBK;
  p.out0 = c.y ? static_cast<void*>(c.y) : static_cast<void*>(c.ws + L.Y);
  return run_grouped_gemm<kFwd2T, 256, true>(w2, w2, w2, p, L.max_mt * p.nb, c.num_sms, s);
}

cudaError_t launch_gemm_fwd_fused(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  cudaError_t st = cudaSuccess;
  // M operands: W1 / W3 viewed as [E d rows][dff], W2 as [E dff rows][d] (64-column boxes)
  const CUtensorMap w1 = make_map_2d(c.W1, L.dff, static_cast<uint64_t>(L.E) * L.d, 2ull * L.dff, 64, 64, &st);
  const CUtensorMap w3 = make_map_2d(c.gated ? c.W3 : c.W1, L.dff, static_cast<uint64_t>(L.E) * L.d,
                                     2ull * L.dff, 64, 64, &st);
  const CUtensorMap w2 = make_map_2d(c.W2, L.d, static_cast<uint64_t>(L.E) * L.dff, 2ull * L.d, 64, 64, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = swap_params(c);
  st = row_maps(p, c.ws + L.xperm, L.d, L.P_pad, 2ull * L.d);
  if (st != cudaSuccess) return st;
  for (int i = 0; i < 4; ++i)
    p.mapR2[i] = make_map_2d(c.ws + L.H, L.dff, L.P_pad, 2ull * L.dff, 64, 16u << i, &st);
  if (st != cudaSuccess) return st;
  p.nb = c.gated ? L.dff / 128 : L.dff / 256;
  p.nkb = L.d / kBK;
  p.nb2 = (L.d + 255) / 256;
  p.nkb2 = L.dff / kBK;
  p.out0 = c.ws + L.H;
  p.out1 = c.ws + L.Y;
  p.done1 = reinterpret_cast<int32_t*>(c.ws + L.done1);
  p.save_ab = c.save_ab;
  p.save_a = c.save_ab ? reinterpret_cast<float*>(c.ws + L.Asave) : nullptr;
  p.save_b = c.save_ab ? reinterpret_cast<float*>(c.ws + L.Bsave) : nullptr;
  return run_grouped_gemm<kFwdT, 256, true>(w2, w1, w3, p, L.max_mt * (p.nb + p.nb2), c.num_sms,
                                            s);
}

}  // namespace moe
