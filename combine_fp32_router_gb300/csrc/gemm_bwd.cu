// Backward grouped GEMMs: dH (+ SwiGLU backward), dX rows, dW2, dW1/dW3.
#include "gemm.cuh"

namespace moe {

GemmParams base_params(const GemmCtx& c);
GemmParams leftover_params(const GemmParams& p, const GemmCtx& c);
GemmParams swap_params(const GemmCtx& c);
cudaError_t row_maps(GemmParams& p, const void* rows, uint64_t inner, uint64_t nrows,
                     uint64_t row_bytes);

namespace {
template <int KIND>
cudaError_t run_bn(int BN, bool pair, const CUtensorMap& a, const CUtensorMap& b0,
                   const CUtensorMap& b1, const GemmParams& p, int64_t tiles, int sms,
                   cudaStream_t s) {
  if (BN == 256) {
    if (pair) return run_grouped_gemm<KIND, 256, true>(a, b0, b1, p, tiles, sms, s);
    return run_grouped_gemm<KIND, 256, false>(a, b0, b1, p, tiles, sms, s);
  }
  if (pair) return run_grouped_gemm<KIND, 128, true>(a, b0, b1, p, tiles, sms, s);
  return run_grouped_gemm<KIND, 128, false>(a, b0, b1, p, tiles, sms, s);
}
}  // namespace

cudaError_t launch_gemm_dh(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  const int BN = (L.dff % 256 == 0) ? 256 : 128;
  const uint32_t brows = c.pair ? BN / 2 : BN;
  cudaError_t st = cudaSuccess;
  // A = dO rows (K = d, K-major); B = W2[e] viewed as [dff rows][d] (K-major)
  const CUtensorMap a = make_map_2d(c.ws + L.dO, L.d, L.P_pad, 2ull * L.d, 64, 128, &st);
  const CUtensorMap b0 = make_map_2d(c.W2, L.d, static_cast<uint64_t>(L.E) * L.dff, 2ull * L.d, 64, brows, &st);
  const CUtensorMap sb0 = make_map_2d(c.W2, L.d, static_cast<uint64_t>(L.E) * L.dff, 2ull * L.d, 64, BN, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = base_params(c);
  p.nb = L.dff / BN;
  p.nkb = L.d / kBK;
  p.out0 = c.ws + L.dAB;
  p.save_a = reinterpret_cast<float*>(c.ws + L.Asave);
  p.save_b = reinterpret_cast<float*>(c.ws + L.Bsave);
  const GemmParams lo = leftover_params(p, c);
  if (BN == 256) return run_rows_kind<kDh, 256>(c.pair, a, b0, b0, sb0, sb0, p, lo, L.max_mt, c.num_sms, s);
  return run_rows_kind<kDh, 128>(c.pair, a, b0, b0, sb0, sb0, p, lo, L.max_mt, c.num_sms, s);
}

cudaError_t launch_gemm_dx(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  const int BN = (L.d % 256 == 0) ? 256 : 128;
  const uint32_t brows = c.pair ? BN / 2 : BN;
  cudaError_t st = cudaSuccess;
  // A = [dA|dB] rows (K = 2 dff; squared ReLU: dA alone, K = dff); B = W1[e] / W3[e] viewed
  // as [d rows][dff] (K-major)
  const uint64_t kdim = (c.gated ? 2ull : 1ull) * L.dff;
  const uint16_t* w3 = c.gated ? c.W3 : c.W1;  // never read without the gate projection
  const CUtensorMap a = make_map_2d(c.ws + L.dAB, kdim, L.P_pad, 4ull * L.dff, 64, 128, &st);
  const CUtensorMap b0 = make_map_2d(c.W1, L.dff, static_cast<uint64_t>(L.E) * L.d, 2ull * L.dff, 64, brows, &st);
  const CUtensorMap b1 = make_map_2d(w3, L.dff, static_cast<uint64_t>(L.E) * L.d, 2ull * L.dff, 64, brows, &st);
  const CUtensorMap sb0 = make_map_2d(c.W1, L.dff, static_cast<uint64_t>(L.E) * L.d, 2ull * L.dff, 64, BN, &st);
  const CUtensorMap sb1 = make_map_2d(w3, L.dff, static_cast<uint64_t>(L.E) * L.d, 2ull * L.dff, 64, BN, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = base_params(c);
  p.nb = L.d / BN;
  p.nkb = static_cast<int>(kdim / kBK);
  p.out0 = c.ws + L.dXp;
  p.mapC0 = make_store_map_f32(c.ws + L.dXp, L.d, L.P_pad, 4ull * L.d, &st);
  if (st != cudaSuccess) return st;
  p.tma_store = 1;
  const GemmParams lo = leftover_params(p, c);
  if (BN == 256) return run_rows_kind<kDx, 256>(c.pair, a, b0, b1, sb0, sb1, p, lo, L.max_mt, c.num_sms, s);
  return run_rows_kind<kDx, 128>(c.pair, a, b0, b1, sb0, sb1, p, lo, L.max_mt, c.num_sms, s);
}

// dX rows with swapped operands: one CTA-pair launch over every (block of up to 256 rows,
// 256 d columns), the M operand W1 / W3 rows (K-major, K = d_ff each), the N operand the
// block's [dA|dB] rows.
cudaError_t launch_gemm_dx_swap(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  cudaError_t st = cudaSuccess;
  const uint64_t kdim = (c.gated ? 2ull : 1ull) * L.dff;
  const uint16_t* w3 = c.gated ? c.W3 : c.W1;  // never read without the gate projection
  // W1 / W3 viewed as [E d rows][dff]: boxes of 64 K columns x 128 rows
  const CUtensorMap w1m = make_map_2d(c.W1, L.dff, static_cast<uint64_t>(L.E) * L.d, 2ull * L.dff, 64, 128, &st);
  const CUtensorMap w3m = make_map_2d(w3, L.dff, static_cast<uint64_t>(L.E) * L.d, 2ull * L.dff, 64, 128, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = swap_params(c);
  st = row_maps(p, c.ws + L.dAB, kdim, L.P_pad, 4ull * L.dff);
  if (st != cudaSuccess) return st;
  p.nb = (L.d + 255) / 256;  // d % 256 == 128: the last block's second CTA has no columns
  p.nkb = static_cast<int>(kdim / kBK);
  p.out0 = c.ws + L.dXp;
  return run_grouped_gemm<kDxT, 256, true>(w1m, w1m, w3m, p, L.max_mt * p.nb, c.num_sms, s);
}

// dH with swapped operands: one CTA-pair launch over every (block of up to 256 rows, 256 d_ff
// columns), the M operand W2 rows (K-major, K = d), the N operand the block's dO rows; the
// epilogue applies the saved multipliers and writes dA and dB.
cudaError_t launch_gemm_dh_swap(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  cudaError_t st = cudaSuccess;
  // W2 viewed as [E dff rows][d]: boxes of 64 K columns x 128 rows
  const CUtensorMap w2m = make_map_2d(c.W2, L.d, static_cast<uint64_t>(L.E) * L.dff, 2ull * L.d, 64, 128, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = swap_params(c);
  st = row_maps(p, c.ws + L.dO, L.d, L.P_pad, 2ull * L.d);
  if (st != cudaSuccess) return st;
  p.nb = (L.dff + 255) / 256;  // d_ff % 256 == 128: the last block's second CTA has no columns
  p.nkb = L.d / kBK;
  p.out0 = c.ws + L.dAB;
  p.save_a = reinterpret_cast<float*>(c.ws + L.Asave);
  p.save_b = reinterpret_cast<float*>(c.ws + L.Bsave);
  return run_grouped_gemm<kDhT, 256, true>(w2m, w2m, w2m, p, L.max_mt * p.nb, c.num_sms, s);
}

cudaError_t launch_gemm_dw2(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  const int BN = (L.d % 256 == 0) ? 256 : 128;
  cudaError_t st = cudaSuccess;
  // A = H rows read as [K = rows][M = dff] (MN-major); B = dO rows [K = rows][N = d] (MN-major)
  const CUtensorMap a = make_map_2d(c.ws + L.H, L.dff, L.P_pad, 2ull * L.dff, 64, 64, &st);
  const CUtensorMap b0 = make_map_2d(c.ws + L.dO, L.d, L.P_pad, 2ull * L.d, 64, 64, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = base_params(c);
  p.M = L.dff;
  const int mrows = c.pair ? 2 * kBM : kBM;
  p.mb = (L.dff + mrows - 1) / mrows;
  p.nb = L.d / BN;
  p.out0 = c.dW2;
  p.mapC0 = make_store_map_f32(c.dW2, L.d, static_cast<uint64_t>(L.E) * L.dff, 4ull * L.d, &st);
  if (st != cudaSuccess) return st;
  p.tma_store = 1;
  const int64_t tiles = static_cast<int64_t>(L.E) * p.mb * p.nb;
  return run_bn<kDw2>(BN, c.pair, a, b0, b0, p, tiles, c.num_sms, s);
}

cudaError_t launch_gemm_dw13(const GemmCtx& c, cudaStream_t s) {
  const WsLayout& L = *c.L;
  const int BN = (L.dff % 256 == 0) ? 256 : 128;
  cudaError_t st = cudaSuccess;
  // A = x_perm rows [K = rows][M = d] (MN-major); B = [dA|dB] rows [K = rows][N = 2 dff]
  const CUtensorMap a = make_map_2d(c.ws + L.xperm, L.d, L.P_pad, 2ull * L.d, 64, 64, &st);
  const CUtensorMap b0 = make_map_2d(c.ws + L.dAB, 2ull * L.dff, L.P_pad, 4ull * L.dff, 64, 64, &st);
  if (st != cudaSuccess) return st;
  GemmParams p = base_params(c);
  p.M = L.d;
  const int mrows = c.pair ? 2 * kBM : kBM;
  p.mb = (L.d + mrows - 1) / mrows;
  p.nb = (c.gated ? 2 : 1) * L.dff / BN;  // squared ReLU: dW1 alone
  p.out0 = c.dW1;
  p.out1 = c.dW3;
  p.mapC0 = make_store_map_f32(c.dW1, L.dff, static_cast<uint64_t>(L.E) * L.d, 4ull * L.dff, &st);
  if (c.gated)
    p.mapC1 = make_store_map_f32(c.dW3, L.dff, static_cast<uint64_t>(L.E) * L.d, 4ull * L.dff, &st);
  if (st != cudaSuccess) return st;
  p.tma_store = 1;
  const int64_t tiles = static_cast<int64_t>(L.E) * p.mb * p.nb;
  return run_bn<kDw13>(BN, c.pair, a, b0, b0, p, tiles, c.num_sms, s);
}

}  // namespace moe
