/*
 * moe.h - C ABI of libmoe.so: one Mixture-of-Experts expert layer on one GB300 GPU.
 *
 * The layer (sources by page title and section):
 *   - "DeepSeek-V4 parallel strategy" (blog.lpkt.cn), section on EP and the IB network:
 *     an MoE layer runs Dispatch -> Expert Compute -> Combine.
 *   - DeepSeek-V4 report reading (10100.com), section on fine-grained compute/communication
 *     overlap of the EP all-to-all: the expert stage is Linear + activation + Linear, and
 *     experts are processed in waves.
 *   - DeepSeek-V4 report, Thai translation (itsolotime.com), section 1.4: the activation is
 *     SwiGLU (gate, up and down projections, 6hd FLOP per token-expert pair) and the
 *     combine payload is BF16.  Section 3 and the 10100.com reading: every kernel is
 *     batch-invariant and deterministic (no global unordered atomic adds; per-unit buffers
 *     reduced in a fixed order).
 * Readings where the pages are silent:
 *   - routing is top-k over fp32 logits with ties going to the lower expert index (+0 and
 *     -0 compare equal); the gate is the softmax over the k selected logits, computed in
 *     fp32; slot j = 0..k-1 follows descending logit;
 *   - the permutation orders rows by (expert, token);
 *   - h = bf16(silu(x W1) * (x W3)) with silu(a) = a / (1 + exp(-a)); A = x W1 and B = x W3
 *     stay fp32; the expert outputs y_j = bf16(h W2) are bf16 rows (the BF16 combine payload
 *     of the report translation, section 1.4), combined as
 *     out_t = bf16(sum_j gate[t,j] * y_j), an fp32 accumulation in slot order.
 *
 * Conventions for every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, row-major, 16-byte
 *     aligned.  bf16 tensors are passed as moe_bf16_t (the raw 16-bit pattern).
 *   - Shapes: x [T,d], logits [T,E] fp32, W1 and W3 [E,d,d_ff], W2 [E,d_ff,d], out [T,d].
 *   - The library never allocates or frees device memory and never synchronises (except
 *     moe_get_error); only the graph entry points create (host and driver) objects.  Every
 *     launch is asynchronous on `stream`.  The workspace `ws` (device memory, 256-byte
 *     aligned, size from moe_workspace_bytes) is caller-owned; calls that share one ws must
 *     be ordered on the GPU (same stream, or synchronised).
 *   - The kernels are launched with programmatic stream serialization and each waits for
 *     the previous kernel in the stream to complete before touching global memory, so
 *     stream order holds as usual: work the caller queues before a call is visible to it,
 *     and a caller's own kernel queued after a call sees its outputs (a caller kernel that
 *     itself opts into programmatic serialization must wait the same way).
 *   - Argument errors are detected on the host before anything is launched and returned as
 *     a status; nothing is written then.  Problems detected on the device (a bounded wait
 *     that ran out, an index out of range) are recorded in an error word inside `ws` and
 *     read with moe_get_error.
 *   - Supported sizes: T >= 0 (T = 0 writes only the outputs that do not depend on T),
 *     1 <= k <= min(E, 16), 1 <= E <= 1024, d and d_ff multiples of 128, d <= 65536,
 *     d_ff <= 65536, T*k + 128*E < 2^31.  Violations return MOE_ERR_UNSUPPORTED.
 *   - Results are bitwise reproducible run to run, and each token's outputs are bitwise
 *     independent of the other tokens in the batch and of T.
 *   - Schedule overrides (environment variables, each read once per process; every choice
 *     gives bitwise the same results, only the kernels that compute them change):
 *     MOE_GEMM_PAIR "0" runs every GEMM on single CTAs, "1" uses CTA pairs whenever T > 128;
 *     MOE_FWD_SWAP, MOE_BWD_SWAP and MOE_BWD_DH_SWAP "0" / "1" turn the swapped-operand
 *     forward GEMMs, the backward's dX (and dH) and the backward's dH alone off / on at every
 *     size; MOE_FWD_FUSED "0" / "1" runs the two swapped forward GEMMs as two launches / one;
 *     MOE_FWD_ROW_COPY "0" has the dispatch copy the permuted rows instead of the swapped GEMM1.
 *     Unset, a size rule on T, k, d and d_ff chooses.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16_t; /* raw bfloat16 bit pattern */

typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, negative size, misalignment, k > E, ... */
  MOE_ERR_UNSUPPORTED = 2,   /* a size outside the supported bounds above             */
  MOE_ERR_WORKSPACE = 3,     /* ws_bytes smaller than the required workspace           */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed            */
  MOE_ERR_TIMEOUT = 5,       /* a bounded device-side wait ran out (moe_get_error)     */
  MOE_ERR_DEVICE_BOUNDS = 6  /* a device-side index check failed (moe_get_error)       */
} moe_status_t;

/* Flags of moe_forward. */
#define MOE_FWD_SAVE_FOR_BACKWARD 1 /* keep, per h element, dA's and dB's multipliers b silu'(a)
                                       * and silu(a) (fp32; 2 relu(a) without W3) in ws for
                                       * moe_backward */
#define MOE_FWD_FUSED_COMBINE 2     /* GEMM2 combines each token as soon as its k expert rows are
                                       written (the single-GPU form of the overlapped combine of
                                       waves); bitwise the same output as the default separate
                                       combine kernel, which is faster on GB300 */
#define MOE_FWD_GATHER_ROWS 4       /* GEMM1 copies its rows from x by token (cp.async into the
                                       operand stages) instead of reading a permuted copy (the
                                       overlapped dispatch of waves); bitwise the same output;
                                       slower on GB300; ignored with MOE_FWD_SAVE_FOR_BACKWARD
                                       (the backward needs the copy) */

/* Stage events: moe_forward records MOE_FWD_NUM_EVENTS events and moe_backward
 * MOE_BWD_NUM_EVENTS events on `stream` at its stage boundaries when `stage_events` is not
 * NULL (each a cudaEvent_t created by the caller).
 *   forward : [0] start, [1] after routing + dispatch, [2] after GEMM1 + SwiGLU,
 *             [3] after GEMM2, [4] after combine ([3] == [4] with MOE_FWD_FUSED_COMBINE).
 *   backward: [0] start, [1] after gate grads + dO, [2] after dH + SwiGLU backward,
 *             [3] after the dX GEMM, [4] after the dX combine, [5] after dW2, [6] after dW1/dW3. */
#define MOE_FWD_NUM_EVENTS 5
#define MOE_BWD_NUM_EVENTS 7

/* Bytes of workspace needed by moe_route_dispatch for (T, E, k). */
size_t moe_route_workspace_bytes(int64_t T, int E, int k);

/* Workspace needs, the bits of moe_workspace_bytes's last argument. */
#define MOE_WS_BACKWARD 1  /* moe_forward(..., MOE_FWD_SAVE_FOR_BACKWARD) + moe_backward */
#define MOE_WS_HOST_IO 2   /* moe_forward_host: device copies of x, logits and out */

/* Bytes of workspace needed by moe_forward, plus what the MOE_WS_* bits in `needs` add
 * (needs = 1, the former with_backward flag, is MOE_WS_BACKWARD).  Returns 0 for arguments
 * outside the supported bounds or an unknown bit. */
size_t moe_workspace_bytes(int64_t T, int d, int E, int k, int d_ff, int needs);

/*
 * Dispatch (routing, counting, prefix sum, stable permute).
 *   topk_idx [T,k] int32 : experts of token t in descending-logit order (ties: lower index)
 *   gate     [T,k] fp32  : softmax over the k selected logits
 *   counts   [E]   int32 : number of (token, slot) pairs routed to each expert
 *   offsets  [E+1] int32 : exclusive prefix sum of counts, offsets[E] = T*k
 *   perm     [T*k] int32 : perm[r] = t*k + j for the pair placed in permuted row r
 *   pos      [T*k] int32 : pos[t*k + j] = r (the inverse of perm)
 *   x_perm   [T*k,d] bf16: x_perm[r] = x[perm[r] / k], rows grouped by expert, ascending
 *                          token order inside each expert
 * Integer outputs and x_perm are exact (bitwise); gate is fp32.  Needs
 * moe_route_workspace_bytes(T, E, k) bytes of ws.
 */
moe_status_t moe_route_dispatch(const moe_bf16_t* x, const float* logits, int64_t T, int d,
                                int E, int k, int32_t* topk_idx, float* gate, int32_t* counts,
                                int32_t* offsets, int32_t* perm, int32_t* pos,
                                moe_bf16_t* x_perm, void* ws, size_t ws_bytes,
                                cudaStream_t stream);

/*
 * Forward of the whole layer: out [T,d] bf16.
 * W3 = NULL selects the expert without the gate projection (report translation, section 1.4,
 * activation bullet: a cheap element-wise activation with no exponential or division in
 * place of SwiGLU; squared ReLU is this library's reading): h = bf16(relu(x W1[e])^2), then
 * h W2[e] as below, with d_ff % 256 == 0 (else MOE_ERR_UNSUPPORTED).
 *   out_t = bf16( sum_j gate[t,j] * (h_tj W2[e_j]) ),  h_tj = bf16(silu(x_t W1[e_j]) * (x_t W3[e_j]))
 * with every matrix product accumulated in fp32 and the slot sum in fp32, in slot order.
 * ws must hold moe_workspace_bytes(T, d, E, k, d_ff, MOE_WS_BACKWARD if
 * MOE_FWD_SAVE_FOR_BACKWARD else 0) bytes; with MOE_FWD_SAVE_FOR_BACKWARD it keeps what
 * moe_backward needs.  stage_events: NULL or MOE_FWD_NUM_EVENTS events (see above).
 */
moe_status_t moe_forward(const moe_bf16_t* x, const float* logits, const moe_bf16_t* W1,
                         const moe_bf16_t* W3, const moe_bf16_t* W2, int64_t T, int d, int E,
                         int k, int d_ff, moe_bf16_t* out, void* ws, size_t ws_bytes, int flags,
                         cudaEvent_t* stage_events, cudaStream_t stream);

/*
 * FP8 dispatch payload (report translation, section 1.4: FP8 dispatch, BF16 combine).  The
 * readings of this library: each token row travels as E4M3 values with one fp32 scale per row,
 * s_t = amax_c |x_tc| / 448 (1 for an all-zero row), q = e4m3(x / s_t) (fp32 division, round
 * to nearest even, saturating at 448); the first projections use E4M3 weights with one fp32
 * scale per (expert, output column) over the input dimension, in the same format.  GEMM1 runs
 * on the tensor cores' FP8 path (tcgen05.mma kind::f8f6f4, fp32 accumulation) and applies the
 * row and column scales in its epilogue; h, W2, GEMM2 and the combine are as in moe_forward.
 * Forward only (no MOE_FWD_* flags).
 *
 * moe_quantize_weights_fp8: W [E,K,N] bf16 (device) -> Wq [E,N,K] E4M3 bytes (each output
 * column a K-contiguous row) and scales [E,N] fp32.  K and N multiples of 128.
 * moe_forward_fp8: x, logits, out and W2 as moe_forward; W1q, W3q [E,d_ff,d] and
 * w1_scale, w3_scale [E,d_ff] from moe_quantize_weights_fp8 of W1 and W3; ws as for
 * moe_forward without backward.
 */
moe_status_t moe_quantize_weights_fp8(const moe_bf16_t* W, int E, int K, int N, uint8_t* Wq,
                                      float* scales, cudaStream_t stream);
moe_status_t moe_forward_fp8(const moe_bf16_t* x, const float* logits, const uint8_t* W1q,
                             const uint8_t* W3q, const float* w1_scale, const float* w3_scale,
                             const moe_bf16_t* W2, int64_t T, int d, int E, int k, int d_ff,
                             moe_bf16_t* out, void* ws, size_t ws_bytes,
                             cudaEvent_t* stage_events, cudaStream_t stream);

/*
 * The launch-overhead path for small batches: one moe_forward captured into a CUDA graph and
 * replayed.  moe_forward_graph_create checks the arguments as moe_forward does, records
 * moe_forward(x, logits, W1, W3, W2, ..., out, ws, ws_bytes, flags) with exactly these
 * pointers and sizes on a private stream (stream capture: nothing runs) and instantiates it.
 * moe_forward_graph_launch replays it on `stream`: the layer on whatever x and logits hold
 * when the replay runs, into the same out and ws (calls sharing ws must be ordered, as for
 * moe_forward).  The handle owns the graph (host and driver objects, no device memory of the
 * library's own); moe_forward_graph_destroy releases it.  On failure *graph is NULL.
 */
typedef struct moe_forward_graph* moe_forward_graph_t;
moe_status_t moe_forward_graph_create(const moe_bf16_t* x, const float* logits,
                                      const moe_bf16_t* W1, const moe_bf16_t* W3,
                                      const moe_bf16_t* W2, int64_t T, int d, int E, int k,
                                      int d_ff, moe_bf16_t* out, void* ws, size_t ws_bytes,
                                      int flags, moe_forward_graph_t* graph);
moe_status_t moe_forward_graph_launch(moe_forward_graph_t graph, cudaStream_t stream);
void moe_forward_graph_destroy(moe_forward_graph_t graph);

/*
 * moe_forward with the batch in HOST memory: x_host [T,d] bf16 and logits_host [T,E] fp32
 * are copied into the end of the workspace, the layer runs on those copies, and out is copied
 * back to out_host [T,d] bf16.  The copies are asynchronous on `stream` (cudaMemcpyAsync);
 * with page-locked host buffers they overlap work on other streams, so a caller can run
 * batches on two streams with two workspaces and hide the copies behind the other batch's
 * layer.  The host buffers are read / written when the stream reaches the copies: keep x_host
 * and logits_host unchanged, and do not read out_host, until the stream has passed the call.
 * W1, W3, W2 and ws are device memory as for moe_forward.  ws must hold
 * moe_workspace_bytes(T, d, E, k, d_ff, MOE_WS_HOST_IO) bytes (| MOE_WS_BACKWARD with
 * MOE_FWD_SAVE_FOR_BACKWARD; moe_backward then takes the same ws and ws_bytes and device
 * x, logits, dy).  flags and stage_events as moe_forward: the events bracket the layer, after
 * the input copies and before the output copy.
 */
moe_status_t moe_forward_host(const moe_bf16_t* x_host, const float* logits_host,
                              const moe_bf16_t* W1, const moe_bf16_t* W3, const moe_bf16_t* W2,
                              int64_t T, int d, int E, int k, int d_ff, moe_bf16_t* out_host,
                              void* ws, size_t ws_bytes, int flags, cudaEvent_t* stage_events,
                              cudaStream_t stream);

/*
 * moe_forward_host for a loop that runs batches back to back: the input copies run on
 * copy_stream, the layer on `stream` once they have landed, and the output copy on
 * copy_stream once the layer has finished.  Successive calls on the same `stream` thus run
 * their layers one after the other (each grouped GEMM fills the whole GPU), while a call's
 * copies overlap the layers of the calls before and after it.  Two calls in flight need two
 * workspaces; calls that share a ws must also share copy_stream, which orders a call's input
 * copies after the previous call's output copy and hence after its layer.  inputs_ready and
 * layer_done are two distinct events created by the caller (cudaEventDisableTiming is
 * enough); the call records each and makes the other stream wait on it before returning, so
 * the next call may reuse them.  Arguments, workspace size and stage_events as
 * moe_forward_host (the events bracket the layer on `stream`).  copy_stream == stream gives
 * moe_forward_host.
 */
moe_status_t moe_forward_host_pipelined(const moe_bf16_t* x_host, const float* logits_host,
                                        const moe_bf16_t* W1, const moe_bf16_t* W3,
                                        const moe_bf16_t* W2, int64_t T, int d, int E, int k,
                                        int d_ff, moe_bf16_t* out_host, void* ws,
                                        size_t ws_bytes, int flags, cudaEvent_t* stage_events,
                                        cudaStream_t stream, cudaStream_t copy_stream,
                                        cudaEvent_t inputs_ready, cudaEvent_t layer_done);

/*
 * Backward of the layer for upstream gradient dy [T,d] bf16.  For the expert without the
 * gate projection (forward with W3 = NULL) pass W3 = NULL and dW3 = NULL.  Precondition: ws
 * holds the state of a moe_forward call with MOE_FWD_SAVE_FOR_BACKWARD on the same x,
 * logits, W1, W3, W2 and sizes, with nothing else using ws in between.
 * Outputs (all overwritten, none accumulated into):
 *   dx      [T,d]        bf16 : sum over slots j (in slot order, fp32) of dA W1^T + dB W3^T
 *   dW1,dW3 [E,d,d_ff]   fp32 : sum over the rows of each expert of x^T dA (resp. x^T dB)
 *   dW2     [E,d_ff,d]   fp32 : sum over the rows of each expert of h^T dO
 *   dgate   [T,k]        fp32 : <y_j, dy_t> with y_j the bf16 expert output row
 *   dlogits [T,E]        fp32 : gradient through the top-k softmax (0 for unselected
 *                               experts); may be NULL
 * with dO = gate * dy, dH = dO W2^T, dA = dH * B * silu'(A), dB = dH * silu(A) (without the
 * gate projection: dA = dH * 2 relu(A), no dB); dO, dA and dB are rounded to bf16 as GEMM
 * operands; every GEMM accumulates in fp32 in a fixed order.
 * stage_events: NULL or MOE_BWD_NUM_EVENTS events.
 */
moe_status_t moe_backward(const moe_bf16_t* dy, const moe_bf16_t* x, const float* logits,
                          const moe_bf16_t* W1, const moe_bf16_t* W3, const moe_bf16_t* W2,
                          int64_t T, int d, int E, int k, int d_ff, moe_bf16_t* dx, float* dW1,
                          float* dW3, float* dW2, float* dgate, float* dlogits, void* ws,
                          size_t ws_bytes, cudaEvent_t* stage_events, cudaStream_t stream);

/*
 * moe_route_dispatch without a workspace, for callers that cannot allocate device memory
 * (code inside a host framework that owns every device allocation, serving loops where an
 * allocation is not allowed, runtimes with a device memory budget fixed at start-up).  The
 * pages have no counterpart: it is a packaging of moe_route_dispatch, same arguments minus
 * ws/ws_bytes, same outputs and the same bit-exact results.
 * Its scratch is a 2 MiB array inside the library image, held in the device memory of every
 * GPU that loads the library until the process exits.  Limit: ceil(T/128) * E <= 262080
 * (for example T = 131072 tokens with E = 256, or T = 32640 with E = 1024); larger sizes
 * return MOE_ERR_UNSUPPORTED before anything is launched.  The first call on a device looks
 * up the array's device address (the device must be current) and keeps it for the life of
 * the process: make that first call before any stream capture, and do not reset the device
 * (cudaDeviceReset or a new primary context) after it.  Every call shares the array: calls
 * that overlap on the GPU (unordered streams, or several host threads) race and give
 * undefined results.  Device-side checks of this variant are recorded at the start of the
 * library's array; moe_route_dispatch_noalloc_get_error reads them.
 */
moe_status_t moe_route_dispatch_noalloc(const moe_bf16_t* x, const float* logits, int64_t T,
                                        int d, int E, int k, int32_t* topk_idx, float* gate,
                                        int32_t* counts, int32_t* offsets, int32_t* perm,
                                        int32_t* pos, moe_bf16_t* x_perm, cudaStream_t stream);

/* The device-side error record of moe_route_dispatch_noalloc on the current device:
 * synchronises `stream` (the stream of the last call), reads the record at the start of the
 * library's fixed array and returns it: MOE_OK when the last call on this device recorded no
 * device-side problem (each call clears the record first), MOE_ERR_DEVICE_BOUNDS when its
 * scatter met an index out of range.  Returns MOE_ERR_CUDA if the stream reports an error.
 * The pages have no counterpart; it belongs to the no-allocation dispatch. */
moe_status_t moe_route_dispatch_noalloc_get_error(cudaStream_t stream);

/* ---------------------------------------------------------------------------------------
 * Fine-grained expert parallelism across R GPUs: the exchange plan and the pull-based row
 * copies (DeepSeek-V4 report, Thai translation, itsolotime.com, section 1.2 and Figure 5:
 * each GPU's experts run in waves, wave i+1's rows are fetched and wave i-1's outputs
 * combined while wave i computes; section 1.4, communication-primitive bullet: the transfers
 * are pull-based reads of the other GPUs' memory; 10100.com reading, section on
 * fine-grained EP overlap).  Rank r of R owns experts [moe_ep_first_expert(E, R, r),
 * moe_ep_first_expert(E, R, r + 1)).  Each rank dispatches its own tokens
 * (moe_route_dispatch), all ranks exchange their per-expert counts ([R][E] int32, e.g. by an
 * all-gather), each rank pulls the rows of its experts from the other ranks into its receive
 * buffer (moe_ep_plan, moe_ep_copy_rows), runs the expert GEMMs on them, and each rank then
 * pulls its own rows' expert outputs back (moe_ep_return_plan, moe_ep_copy_rows) and
 * combines them as on one GPU.  The rows of an expert arrive ordered by (source rank, source
 * row), i.e. by global token when the global batch is the ranks' batches concatenated, so
 * every result is bitwise the single-GPU layer's on that batch.
 * ------------------------------------------------------------------------------------- */

/* First expert owned by `rank` of R (experts split into R contiguous blocks of floor/ceil
 * E/R); rank = R gives E.  -1 for invalid arguments. */
int moe_ep_first_expert(int E, int R, int rank);

/* Exchange plan of `rank` (host function, host memory; nothing is launched).
 * counts_all [R][E]: rows that each rank's dispatch routed to each expert.  For local expert
 * i (global expert first + i) and source rank s:
 *   recv_off[i*R + s]  first row of those rows in this rank's receive buffer; each expert's
 *                      rows start at a multiple of row_align (128 for the grouped GEMMs);
 *                      recv_off[n_local*R] = the receive buffer's row count,
 *   src_off[i*R + s]   first row of those rows in rank s's permuted buffer (the exclusive
 *                      prefix of s's counts: moe_route_dispatch's offsets on rank s),
 *   recv_counts[i]     rows of local expert i from all ranks,
 *   wave_first[w]      first local expert of wave w (waves of wave_experts experts),
 *                      wave_first[*n_waves] = n_local.
 * Output sizes: recv_off n_local*R + 1, src_off n_local*R, recv_counts n_local, wave_first
 * ceil(n_local / wave_experts) + 1 (n_local <= ceil(E / R)).  Errors: MOE_ERR_INVALID_ARG
 * (null pointer, R < 1, R > E, rank out of range, a negative count), MOE_ERR_UNSUPPORTED
 * (more than 2^31 - 1 rows). */
moe_status_t moe_ep_plan(const int32_t* counts_all, int R, int E, int rank, int row_align,
                         int wave_experts, int32_t* recv_off, int32_t* src_off,
                         int32_t* recv_counts, int32_t* wave_first, int32_t* n_waves);

/* Return plan of `rank` (host function, host memory): for every expert e of the layer,
 * owner[e] = the rank that computes it, owner_row[e] = the first row, in the owner's
 * receive-side buffers, of the rows this rank sent it, own_row[e] = the first of those rows
 * in this rank's permuted buffer.  Sizes E each.  Errors as moe_ep_plan. */
moe_status_t moe_ep_return_plan(const int32_t* counts_all, int R, int E, int rank,
                                int row_align, int32_t* owner, int32_t* owner_row,
                                int32_t* own_row);

/* Row segments copied into `dst` from other ranks' buffers with plain 16-byte loads and
 * stores (no TMA, no multicast): segment i copies seg_rows[i] rows starting at row
 * seg_src_row[i] of the buffer peers[seg_src_rank[i]] to rows starting at seg_dst_row[i]
 * of dst.  peers [R] and peer_rows [R] (rows each peer buffer holds) and the four segment
 * arrays [n_seg] are DEVICE arrays; each peers[s] is a device pointer this GPU can read (its
 * own memory, or a peer GPU's mapped by the caller).  row_bytes: a multiple of 16; dst holds
 * dst_rows rows.  A segment outside its source or destination records
 * MOE_ERR_DEVICE_BOUNDS in the 16-byte error word `err_word` (device memory, e.g. the start
 * of a workspace, read with moe_get_error) and is skipped.  Asynchronous on `stream`; the
 * caller orders it after the source rows are written on their GPUs. */
moe_status_t moe_ep_copy_rows(const void* const* peers, const int64_t* peer_rows, int R,
                              const int32_t* seg_src_rank, const int32_t* seg_src_row,
                              const int32_t* seg_dst_row, const int32_t* seg_rows, int n_seg,
                              int64_t row_bytes, void* dst, int64_t dst_rows, void* err_word,
                              cudaStream_t stream);

/* The expert stage alone (GEMM1 + SwiGLU, GEMM2) on rows the caller holds: an expert-
 * parallel owner's receive buffer, laid out by moe_ep_plan with row_align = 128.
 *   rows [n_rows, d] bf16 (device): local expert i's counts[i] rows start at row
 *        sum_{j<i} round_up(counts[j], 128); rows between the segments are not read into
 *        any result (any content),
 *   counts [E] int32 (DEVICE array), W1 / W3 [E, d, d_ff], W2 [E, d_ff, d] bf16: the E local
 *        experts (W3 = NULL: squared ReLU, d_ff a multiple of 256),
 *   y_rows [n_rows, d] bf16 (device): y = bf16(bf16(h) W2) of each row, in the same layout;
 *        rows between the segments are left as they were.
 * Each row's h and y are bitwise the ones moe_forward computes for the same token-expert
 * pair: every tile's arithmetic depends only on the model sizes.  ws: device memory of
 * moe_expert_workspace_bytes(n_rows, d, E, d_ff) bytes, 256-byte aligned, caller-owned; its
 * error record is read with moe_get_error.  Errors as moe_forward; a segment layout that does
 * not fit n_rows records MOE_ERR_DEVICE_BOUNDS (nothing past n_rows is written).
 * Asynchronous on `stream`. */
size_t moe_expert_workspace_bytes(int64_t n_rows, int d, int E, int d_ff);
moe_status_t moe_expert_forward(const moe_bf16_t* rows, const int32_t* counts, int64_t n_rows,
                                int d, int E, int d_ff, const moe_bf16_t* W1,
                                const moe_bf16_t* W3, const moe_bf16_t* W2, moe_bf16_t* y_rows,
                                void* ws, size_t ws_bytes, cudaStream_t stream);

/* The combine alone: out[t] = bf16(sum_j gate[t, j] * y_rows[pos[t, j]]), an fp32
 * accumulation in slot order j = 0..k-1, exactly as moe_forward's last stage (an expert-
 * parallel source rank combines the output rows it pulled back).  y_rows [n_rows, d] bf16,
 * gate [T, k] fp32, pos [T, k] int32, out [T, d] bf16: device memory.  A pos outside
 * [0, n_rows) records MOE_ERR_DEVICE_BOUNDS in the 16-byte error word err_word (device memory,
 * read with moe_get_error) and row 0 is read in its place.  Errors: MOE_ERR_INVALID_ARG (null
 * or misaligned pointers), MOE_ERR_UNSUPPORTED (k or d outside the layer's limits).
 * Asynchronous on `stream`. */
moe_status_t moe_combine(const moe_bf16_t* y_rows, int64_t n_rows, const float* gate,
                         const int32_t* pos, int64_t T, int k, int d, moe_bf16_t* out,
                         void* err_word, cudaStream_t stream);

/* Measurement probe (not part of the layer; the pages have no counterpart): the DRAM read
 * rate one SM sustains by load path.  Launches `ctas` CTAs (one per SM when ctas <= the SM
 * count), each streaming its own slice of floor(bytes / 152) bytes (rounded down to 16 KB)
 * of `buf` (device memory, 16-byte aligned, much larger than L2): mode 0 with 16-byte loads
 * by 512 threads, mode 1 / 2 with 16 KB bulk copies into 6 / 12 shared-memory stages, mode
 * 3 / 4 with the expert GEMMs' 2-D tensor-map boxes (two 64 x 64 bf16 boxes per stage, 6
 * stages) over the buffer viewed with 4 KB rows (a weight matrix's pattern) / 256-byte rows
 * (contiguous; each CTA then streams 256 bytes of each of its rows).  The
 * caller times the launch (events on `stream`); `out` (device, ctas uint32) receives 1 for a
 * CTA whose bounded wait ran out.  MOE_ERR_INVALID_ARG when the slices do not fit in buf. */
moe_status_t moe_probe_dram_read(const void* buf, size_t bytes, int ctas, int mode,
                                 uint32_t* out, cudaStream_t stream);

/* Synchronises `stream`, reads the device error word of `ws` and returns it (MOE_OK when
 * no device-side problem was recorded since the last moe_route_dispatch / moe_forward on
 * this ws, which clear it).  Returns MOE_ERR_CUDA if the stream reports an error. */
moe_status_t moe_get_error(const void* ws, cudaStream_t stream);

/* Upper bound, in nanoseconds, of every device-side wait of kernels launched after this
 * call (process-wide; default 2e9).  A wait that runs out records MOE_ERR_TIMEOUT and its
 * kernel returns without finishing the work. */
void moe_set_wait_timeout_ns(uint64_t ns);

/* Test hook, process-wide, 0 by default.  Bit 0: the first CTA of the next grouped-GEMM
 * launches skips its first operand load so that the matching wait runs out (used to test
 * the timeout path on a tiny problem with a short timeout).  Bit 1: moe_forward dispatches
 * batches of T <= 128 with the multi-kernel sequence of larger batches instead of its
 * single launch (both give bitwise the same workspace contents and output). */
void moe_debug_set_flags(int flags);

/* Short English description of a status code. */
const char* moe_status_string(moe_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H_ */
