// Fine-grained expert parallelism across GPUs: the exchange plan (host) and the row copies of
// its pull-based transport (device).
//
// The pages' method splits the experts across GPUs and processes each GPU's experts in
// waves: while wave i computes, the rows of wave i+1 are read from the GPUs that routed them
// and the outputs of wave i-1 are combined (DeepSeek-V4 report, Thai translation,
// itsolotime.com, section 1.2 and Figure 5; 10100.com reading, section on fine-grained EP
// overlap).  The reads are pull-based: each GPU reads its inputs from the other GPUs' memory
// instead of waiting to be sent them (the same page, section 1.4, bullet on communication
// primitives).
//
// This file holds what the path needs beyond the single-GPU layer:
//  * moe_ep_plan: from every rank's per-expert row counts (all-gathered [R][E]), the layout
//    of this rank's receive buffer and where each of its row segments lives in the sending
//    rank's permuted buffer; the rows of one expert arrive ordered by (source rank, source
//    row), which is (global token) order when the global batch is the ranks' batches
//    concatenated, so the expert GEMMs see exactly the rows a single-GPU dispatch of the
//    whole batch would give them, in the same order.
//  * moe_ep_return_plan: the reverse legs, for each expert of the layer, where this rank's
//    expert-output rows sit in the owner's receive-side output buffer.
//  * moe_ep_copy_rows: row segments copied from other ranks' buffers (peer device pointers)
//    with plain 16-byte loads and stores; one launch moves a whole wave.
// The planning is integer arithmetic in host code; nothing here allocates or synchronises.
#include <cstdint>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

int first_expert(int E, int R, int rank) {
  return static_cast<int>(static_cast<int64_t>(rank) * E / R);
}

// One warp per segment (segments strided over the grid), lanes across the 16-byte chunks
// of its rows.  Bounds: every row index is checked against the source and destination row
// counts; a segment that would leave them records MOE_ERR_DEVICE_BOUNDS and is skipped.
__global__ void __launch_bounds__(256) ep_copy_rows_kernel(
    const uint4* const* __restrict__ peers, int R, const int64_t* __restrict__ peer_rows,
    const int32_t* __restrict__ seg_src_rank, const int32_t* __restrict__ seg_src_row,
    const int32_t* __restrict__ seg_dst_row, const int32_t* __restrict__ seg_rows, int n_seg,
    int64_t row16, uint4* __restrict__ dst, int64_t dst_rows, DevErr* err) {
  griddep_wait();  // the previous kernel in the stream has finished (PDL)
  const int lane = threadIdx.x & 31;
  const int nwarps = static_cast<int>(gridDim.x * (blockDim.x >> 5));
  for (int sgi = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5); sgi < n_seg;
       sgi += nwarps) {
    const int s = seg_src_rank[sgi];
    const int64_t r0 = seg_src_row[sgi], d0 = seg_dst_row[sgi], n = seg_rows[sgi];
    if (s < 0 || s >= R || r0 < 0 || d0 < 0 || n < 0 || r0 + n > peer_rows[s] ||
        d0 + n > dst_rows) {
      if (lane == 0) set_error(err, MOE_ERR_DEVICE_BOUNDS, 300);
      continue;
    }
    const uint4* src = peers[s] + r0 * row16;
    uint4* out = dst + d0 * row16;
    const int64_t total = n * row16;  // 16-byte chunks of the segment (contiguous rows)
    for (int64_t i = lane; i < total; i += 32) st_v4(out + i, ld_nc_v4(src + i));
  }
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_ep_first_expert(int E, int R, int rank) {
  if (E <= 0 || R <= 0 || rank < 0 || rank > R) return -1;
  return first_expert(E, R, rank);
}

moe_status_t moe_ep_plan(const int32_t* counts_all, int R, int E, int rank, int row_align,
                         int wave_experts, int32_t* recv_off, int32_t* src_off,
                         int32_t* recv_counts, int32_t* wave_first, int32_t* n_waves) {
  if (!counts_all || !recv_off || !src_off || !recv_counts || !wave_first || !n_waves)
    return MOE_ERR_INVALID_ARG;
  if (R < 1 || E < 1 || R > E || rank < 0 || rank >= R || row_align < 1 || wave_experts < 1)
    return MOE_ERR_INVALID_ARG;
  const int e0 = first_expert(E, R, rank), e1 = first_expert(E, R, rank + 1);
  const int nloc = e1 - e0;
  for (int64_t i = 0; i < static_cast<int64_t>(R) * E; ++i)
    if (counts_all[i] < 0) return MOE_ERR_INVALID_ARG;
  int64_t at = 0;  // rows of the receive buffer so far (each expert padded to row_align)
  for (int i = 0; i < nloc; ++i) {
    const int e = e0 + i;
    int64_t n = 0;
    for (int s = 0; s < R; ++s) {
      // rows of expert e in source rank s's permuted buffer: after every lower expert's
      // (the exclusive prefix of s's counts)
      int64_t before = 0;
      for (int ep = 0; ep < e; ++ep) before += counts_all[static_cast<int64_t>(s) * E + ep];
      const int64_t c = counts_all[static_cast<int64_t>(s) * E + e];
      if (at + n > INT32_MAX - c || before > INT32_MAX) return MOE_ERR_UNSUPPORTED;
      recv_off[i * R + s] = static_cast<int32_t>(at + n);
      src_off[i * R + s] = static_cast<int32_t>(before);
      n += c;
    }
    recv_counts[i] = static_cast<int32_t>(n);
    at += (n + row_align - 1) / row_align * row_align;
    if (at > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  }
  recv_off[nloc * R] = static_cast<int32_t>(at);
  int w = 0;
  for (int i = 0; i < nloc; i += wave_experts) wave_first[w++] = i;
  wave_first[w] = nloc;
  *n_waves = w;
  return MOE_OK;
}

moe_status_t moe_ep_return_plan(const int32_t* counts_all, int R, int E, int rank,
                                int row_align, int32_t* owner, int32_t* owner_row,
                                int32_t* own_row) {
  if (!counts_all || !owner || !owner_row || !own_row) return MOE_ERR_INVALID_ARG;
  if (R < 1 || E < 1 || R > E || rank < 0 || rank >= R || row_align < 1)
    return MOE_ERR_INVALID_ARG;
  for (int r = 0; r < R; ++r) {
    // the owner's receive layout, recomputed from the same counts
    const int e0 = first_expert(E, R, r), e1 = first_expert(E, R, r + 1);
    int64_t at = 0;
    for (int e = e0; e < e1; ++e) {
      int64_t n = 0;
      for (int s = 0; s < R; ++s) {
        const int64_t c = counts_all[static_cast<int64_t>(s) * E + e];
        if (c < 0) return MOE_ERR_INVALID_ARG;
        if (s == rank) {
          owner[e] = r;
          owner_row[e] = static_cast<int32_t>(at + n);
        }
        n += c;
      }
      at += (n + row_align - 1) / row_align * row_align;
      if (at > INT32_MAX) return MOE_ERR_UNSUPPORTED;
    }
  }
  int64_t before = 0;
  for (int e = 0; e < E; ++e) {
    own_row[e] = static_cast<int32_t>(before);
    before += counts_all[static_cast<int64_t>(rank) * E + e];
  }
  return MOE_OK;
}

moe_status_t moe_ep_copy_rows(const void* const* peers, const int64_t* peer_rows, int R,
                              const int32_t* seg_src_rank, const int32_t* seg_src_row,
                              const int32_t* seg_dst_row, const int32_t* seg_rows, int n_seg,
                              int64_t row_bytes, void* dst, int64_t dst_rows, void* err_word,
                              cudaStream_t stream) {
  if (n_seg < 0 || R < 1 || row_bytes <= 0 || row_bytes % 16 != 0 || dst_rows < 0)
    return MOE_ERR_INVALID_ARG;
  if (n_seg == 0) return MOE_OK;
  if (!peers || !peer_rows || !seg_src_rank || !seg_src_row || !seg_dst_row || !seg_rows ||
      !dst || !err_word)
    return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dst) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(err_word) & 15u) != 0)
    return MOE_ERR_INVALID_ARG;
  int grid = (n_seg + 7) / 8;
  if (grid > 152 * 8) grid = 152 * 8;
  const cudaError_t e = launch_pdl(ep_copy_rows_kernel, dim3(grid), dim3(256), 0, stream,
                                   reinterpret_cast<const uint4* const*>(peers), R, peer_rows,
                                   seg_src_rank, seg_src_row, seg_dst_row, seg_rows, n_seg,
                                   row_bytes / 16, static_cast<uint4*>(dst), dst_rows,
                                   static_cast<DevErr*>(err_word));
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // extern "C"
