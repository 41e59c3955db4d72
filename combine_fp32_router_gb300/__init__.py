"""Python binding of libmoe.so: one MoE expert layer on one GB300 GPU.

The functions below carry the names of the C entry points in ``include/moe.h`` and only
marshal arguments: they read sizes and device pointers off torch tensors, pass the current
CUDA stream, and turn a non-zero status into ``MoeError``.  Every step of the layer runs in
the library's CUDA kernels; there is no fallback.  torch provides device memory, streams
and events only.

Import fails loudly when ``libmoe.so`` has not been built (``build.build()``).
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_BOUNDS = 6
MOE_FWD_SAVE_FOR_BACKWARD = 1
MOE_FWD_FUSED_COMBINE = 2
MOE_FWD_GATHER_ROWS = 4
MOE_WS_BACKWARD = 1
MOE_WS_HOST_IO = 2
MOE_FWD_NUM_EVENTS = 5
MOE_BWD_NUM_EVENTS = 7

# Exported symbols of include/moe.h, in declaration order.
EXPORTS = ("moe_route_workspace_bytes", "moe_workspace_bytes", "moe_route_dispatch",
           "moe_forward", "moe_forward_fp8", "moe_quantize_weights_fp8",
           "moe_forward_graph_create", "moe_forward_graph_launch",
           "moe_forward_graph_destroy", "moe_forward_host", "moe_forward_host_pipelined",
           "moe_backward",
           "moe_route_dispatch_noalloc", "moe_route_dispatch_noalloc_get_error",
           "moe_ep_first_expert", "moe_ep_plan", "moe_ep_return_plan", "moe_ep_copy_rows",
           "moe_expert_workspace_bytes", "moe_expert_forward", "moe_combine",
           "moe_probe_dram_read", "moe_get_error", "moe_set_wait_timeout_ns",
           "moe_debug_set_flags", "moe_status_string")


class MoeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, moe_status_string(status), status))


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError("libmoe.so is missing: build it with "
                          "combine_fp32_router_gb300.build.build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    p, i, i64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    lib.moe_route_workspace_bytes.argtypes = [i64, i, i]
    lib.moe_route_workspace_bytes.restype = sz
    lib.moe_workspace_bytes.argtypes = [i64, i, i, i, i, i]
    lib.moe_workspace_bytes.restype = sz
    lib.moe_route_dispatch.argtypes = [p, p, i64, i, i, i] + [p] * 7 + [p, sz, p]
    lib.moe_route_dispatch.restype = i
    lib.moe_forward.argtypes = [p] * 5 + [i64, i, i, i, i, p, p, sz, i, p, p]
    lib.moe_quantize_weights_fp8.restype = i
    lib.moe_quantize_weights_fp8.argtypes = [p, i, i, i, p, p, p]
    lib.moe_forward_fp8.restype = i
    lib.moe_forward_fp8.argtypes = [p] * 7 + [i64, i, i, i, i, p, p, sz, p, p]
    lib.moe_forward_graph_create.restype = i
    lib.moe_forward_graph_create.argtypes = [p] * 5 + [i64, i, i, i, i, p, p, sz, i,
                                                       ctypes.POINTER(ctypes.c_void_p)]
    lib.moe_forward_graph_launch.restype = i
    lib.moe_forward_graph_launch.argtypes = [p, p]
    lib.moe_forward_graph_destroy.restype = None
    lib.moe_forward_graph_destroy.argtypes = [p]
    lib.moe_forward_host.restype = i
    lib.moe_forward_host.argtypes = [p] * 5 + [i64, i, i, i, i, p, p, sz, i, p, p]
    lib.moe_forward_host_pipelined.restype = i
    lib.moe_forward_host_pipelined.argtypes = [p] * 5 + [i64, i, i, i, i, p, p, sz, i, p] + [p] * 4
    lib.moe_forward.restype = i
    lib.moe_backward.argtypes = [p] * 6 + [i64, i, i, i, i] + [p] * 6 + [p, sz, p, p]
    lib.moe_backward.restype = i
    lib.moe_route_dispatch_noalloc.argtypes = [p, p, i64, i, i, i] + [p] * 7 + [p]
    lib.moe_route_dispatch_noalloc.restype = i
    lib.moe_get_error.argtypes = [p, p]
    lib.moe_get_error.restype = i
    lib.moe_route_dispatch_noalloc_get_error.argtypes = [p]
    lib.moe_route_dispatch_noalloc_get_error.restype = i
    lib.moe_ep_first_expert.argtypes = [i, i, i]
    lib.moe_ep_first_expert.restype = i
    lib.moe_ep_plan.argtypes = [p, i, i, i, i, i, p, p, p, p, p]
    lib.moe_ep_plan.restype = i
    lib.moe_ep_return_plan.argtypes = [p, i, i, i, i, p, p, p]
    lib.moe_ep_return_plan.restype = i
    lib.moe_ep_copy_rows.argtypes = [p, p, i, p, p, p, p, i, i64, p, i64, p, p]
    lib.moe_ep_copy_rows.restype = i
    lib.moe_expert_workspace_bytes.argtypes = [i64, i, i, i]
    lib.moe_expert_workspace_bytes.restype = sz
    lib.moe_expert_forward.argtypes = [p, p, i64, i, i, i, p, p, p, p, p, sz, p]
    lib.moe_expert_forward.restype = i
    lib.moe_combine.argtypes = [p, i64, p, p, i64, i, i, p, p, p]
    lib.moe_combine.restype = i
    lib.moe_probe_dram_read.argtypes = [p, sz, i, i, p, p]
    lib.moe_probe_dram_read.restype = i
    lib.moe_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
    lib.moe_set_wait_timeout_ns.restype = None
    lib.moe_debug_set_flags.argtypes = [i]
    lib.moe_debug_set_flags.restype = None
    lib.moe_status_string.argtypes = [i]
    lib.moe_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()


def _ptr(t):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor arguments must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _nptr(a):
    """Host numpy array -> pointer (the host-side planning entry points)."""
    return ctypes.c_void_p(a.ctypes.data)


def _nbytes(t):
    return t.numel() * t.element_size()


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _events(events):
    if events is None:
        return None
    handles = []
    for ev in events:
        if not ev.cuda_event:       # torch creates the CUDA event lazily on first record
            ev.record()
        handles.append(ev.cuda_event)
    return (ctypes.c_void_p * len(handles))(*handles)


def _check(st, where):
    if st != MOE_OK:
        raise MoeError(st, where)


def moe_status_string(status):
    return _lib.moe_status_string(int(status)).decode()


def moe_route_workspace_bytes(T, E, k):
    return int(_lib.moe_route_workspace_bytes(T, E, k))


def moe_workspace_bytes(T, d, E, k, d_ff, with_backward=False, host_io=False):
    needs = (MOE_WS_BACKWARD if with_backward else 0) | (MOE_WS_HOST_IO if host_io else 0)
    return int(_lib.moe_workspace_bytes(T, d, E, k, d_ff, needs))


def moe_route_dispatch(x, logits, k, topk_idx, gate, counts, offsets, perm, pos, x_perm, ws,
                       stream=None):
    """Routing + counts + offsets + stable permute into caller-owned outputs."""
    T, d = x.shape
    E = logits.shape[1]
    _check(_lib.moe_route_dispatch(_ptr(x), _ptr(logits), T, d, E, k, _ptr(topk_idx),
                                   _ptr(gate), _ptr(counts), _ptr(offsets), _ptr(perm),
                                   _ptr(pos), _ptr(x_perm), _ptr(ws), _nbytes(ws),
                                   _stream(stream)), "moe_route_dispatch")


def moe_forward(x, logits, W1, W3, W2, k, out, ws, flags=0, stage_events=None, stream=None):
    """Whole-layer forward into ``out`` [T, d] bf16."""
    T, d = x.shape
    E, _, d_ff = W1.shape
    _check(_lib.moe_forward(_ptr(x), _ptr(logits), _ptr(W1), _ptr(W3), _ptr(W2), T, d, E, k,
                            d_ff, _ptr(out), _ptr(ws), _nbytes(ws), int(flags),
                            _events(stage_events), _stream(stream)), "moe_forward")


def moe_quantize_weights_fp8(W, stream=None):
    """E4M3 copy of expert weights W [E, K, N] bf16 for moe_forward_fp8: returns
    (Wq [E, N, K] uint8, scales [E, N] fp32) (one scale per output column)."""
    E, K, N = W.shape
    Wq = torch.empty(E, N, K, dtype=torch.uint8, device=W.device)
    sc = torch.empty(E, N, dtype=torch.float32, device=W.device)
    _check(_lib.moe_quantize_weights_fp8(_ptr(W), E, K, N, _ptr(Wq), _ptr(sc), _stream(stream)),
           "moe_quantize_weights_fp8")
    return Wq, sc


def moe_forward_fp8(x, logits, W1q, W3q, w1_scale, w3_scale, W2, k, out, ws, stage_events=None,
                    stream=None):
    """Whole-layer forward with the FP8 dispatch payload (E4M3 rows and W1 / W3)."""
    T, d = x.shape
    E, d_ff, _ = W1q.shape
    _check(_lib.moe_forward_fp8(_ptr(x), _ptr(logits), _ptr(W1q), _ptr(W3q), _ptr(w1_scale),
                                _ptr(w3_scale), _ptr(W2), T, d, E, k, d_ff, _ptr(out), _ptr(ws),
                                _nbytes(ws), _events(stage_events), _stream(stream)),
           "moe_forward_fp8")


class ForwardGraph:
    """A moe_forward captured once (moe_forward_graph_create) and replayed with launch().  The
    tensors given at creation are baked in: replays read x and logits as they are then and
    write the same out.  close() (or garbage collection) releases the graph."""

    def __init__(self, handle, keep):
        self._h = handle
        self._keep = keep  # the captured tensors must outlive the graph

    def launch(self, stream=None):
        if not self._h:
            raise ValueError("graph already closed")
        _check(_lib.moe_forward_graph_launch(self._h, _stream(stream)), "moe_forward_graph_launch")

    def close(self):
        if self._h:
            _lib.moe_forward_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_forward_graph_create(x, logits, W1, W3, W2, k, out, ws, flags=0):
    """Capture moe_forward with these tensors into a replayable graph (ForwardGraph)."""
    T, d = x.shape
    E, _, d_ff = W1.shape
    h = ctypes.c_void_p()
    _check(_lib.moe_forward_graph_create(_ptr(x), _ptr(logits), _ptr(W1), _ptr(W3), _ptr(W2),
                                         T, d, E, k, d_ff, _ptr(out), _ptr(ws), _nbytes(ws),
                                         int(flags), ctypes.byref(h)),
           "moe_forward_graph_create")
    return ForwardGraph(h, (x, logits, W1, W3, W2, out, ws))


def moe_forward_host(x_host, logits_host, W1, W3, W2, k, out_host, ws, flags=0,
                     stage_events=None, stream=None):
    """Whole-layer forward with x, logits and out in host memory (page-locked for
    asynchronous copies); the weights and ``ws`` are device tensors."""
    T, d = x_host.shape
    E, _, d_ff = W1.shape
    _check(_lib.moe_forward_host(_ptr(x_host), _ptr(logits_host), _ptr(W1), _ptr(W3), _ptr(W2),
                                 T, d, E, k, d_ff, _ptr(out_host), _ptr(ws), _nbytes(ws),
                                 int(flags), _events(stage_events), _stream(stream)),
           "moe_forward_host")


def moe_forward_host_pipelined(x_host, logits_host, W1, W3, W2, k, out_host, ws, copy_stream,
                               events, flags=0, stage_events=None, stream=None):
    """moe_forward_host with the copies on ``copy_stream`` and the layer on ``stream``;
    ``events`` holds the two torch.cuda.Event objects the call records and waits on
    (inputs ready, layer done)."""
    T, d = x_host.shape
    E, _, d_ff = W1.shape
    ev = _events(events)
    if ev is None or len(ev) != 2:
        raise ValueError("events must hold two torch.cuda.Event objects")
    _check(_lib.moe_forward_host_pipelined(
        _ptr(x_host), _ptr(logits_host), _ptr(W1), _ptr(W3), _ptr(W2), T, d, E, k, d_ff,
        _ptr(out_host), _ptr(ws), _nbytes(ws), int(flags), _events(stage_events),
        _stream(stream), _stream(copy_stream), ev[0], ev[1]), "moe_forward_host_pipelined")


def moe_backward(dy, x, logits, W1, W3, W2, k, dx, dW1, dW3, dW2, dgate, dlogits, ws,
                 stage_events=None, stream=None):
    """Whole-layer backward (after moe_forward with MOE_FWD_SAVE_FOR_BACKWARD on ``ws``)."""
    T, d = x.shape
    E, _, d_ff = W1.shape
    _check(_lib.moe_backward(_ptr(dy), _ptr(x), _ptr(logits), _ptr(W1), _ptr(W3), _ptr(W2), T,
                             d, E, k, d_ff, _ptr(dx), _ptr(dW1), _ptr(dW3), _ptr(dW2),
                             _ptr(dgate), _ptr(dlogits), _ptr(ws), _nbytes(ws),
                             _events(stage_events), _stream(stream)), "moe_backward")


def moe_route_dispatch_noalloc(x, logits, k, topk_idx, gate, counts, offsets, perm, pos,
                               x_perm, stream=None):
    """moe_route_dispatch for callers that cannot allocate device memory: no workspace
    argument; the scratch is a fixed array inside the library (see include/moe.h for the size
    limit and the rule that calls must not overlap on the GPU)."""
    T, d = x.shape
    E = logits.shape[1]
    _check(_lib.moe_route_dispatch_noalloc(_ptr(x), _ptr(logits), T, d, E, k, _ptr(topk_idx),
                                           _ptr(gate), _ptr(counts), _ptr(offsets), _ptr(perm),
                                           _ptr(pos), _ptr(x_perm), _stream(stream)),
           "moe_route_dispatch_noalloc")


def moe_route_dispatch_noalloc_get_error(stream=None):
    """Synchronise the stream and return the device error status the last
    moe_route_dispatch_noalloc call on the current device recorded in the library's array."""
    return int(_lib.moe_route_dispatch_noalloc_get_error(_stream(stream)))


def moe_ep_first_expert(E, R, rank):
    """First expert owned by `rank` of R (rank = R gives E)."""
    return int(_lib.moe_ep_first_expert(int(E), int(R), int(rank)))


def moe_ep_plan(counts_all, rank, row_align=128, wave_experts=4):
    """Exchange plan of `rank` from every rank's per-expert counts (host int32 [R, E]):
    returns dict(recv_off [n_local, R], rows (receive buffer rows), src_off [n_local, R],
    recv_counts [n_local], waves (first local expert of each wave, plus n_local))."""
    import numpy as np
    c = np.ascontiguousarray(counts_all, dtype=np.int32)
    R, E = c.shape
    cap = -(-E // max(R, 1))                       # the most experts a rank can own
    recv_off = np.zeros(cap * R + 1, np.int32)
    src_off = np.zeros(cap * R, np.int32)
    recv_counts = np.zeros(cap, np.int32)
    wave_first = np.zeros(cap + 2, np.int32)
    n_waves = np.zeros(1, np.int32)
    _check(_lib.moe_ep_plan(_nptr(c), R, E, int(rank), int(row_align), int(wave_experts),
                            _nptr(recv_off), _nptr(src_off), _nptr(recv_counts),
                            _nptr(wave_first), _nptr(n_waves)), "moe_ep_plan")
    nloc = moe_ep_first_expert(E, R, rank + 1) - moe_ep_first_expert(E, R, rank)
    return dict(recv_off=recv_off[:nloc * R].reshape(nloc, R), rows=int(recv_off[nloc * R]),
                src_off=src_off[:nloc * R].reshape(nloc, R), recv_counts=recv_counts[:nloc],
                waves=wave_first[:int(n_waves[0]) + 1])


def moe_ep_return_plan(counts_all, rank, row_align=128):
    """For every expert: (owner rank, first row of this rank's rows in the owner's
    receive-side buffers, first row in this rank's permuted buffer), int32 arrays [E]."""
    import numpy as np
    c = np.ascontiguousarray(counts_all, dtype=np.int32)
    R, E = c.shape
    owner, owner_row, own_row = (np.zeros(E, np.int32) for _ in range(3))
    _check(_lib.moe_ep_return_plan(_nptr(c), R, E, int(rank), int(row_align), _nptr(owner),
                                   _nptr(owner_row), _nptr(own_row)), "moe_ep_return_plan")
    return owner, owner_row, own_row


def moe_ep_copy_rows(peers, peer_rows, seg_src_rank, seg_src_row, seg_dst_row, seg_rows, dst,
                     err_word, stream=None):
    """Row segments from other ranks' buffers into ``dst`` (device tensors: ``peers`` an
    int64 tensor of device addresses, ``peer_rows`` int64, the segment arrays int32);
    row size = dst's row size."""
    R = peers.numel()
    n_seg = seg_rows.numel()
    row_bytes = dst.stride(0) * dst.element_size()
    _check(_lib.moe_ep_copy_rows(_ptr(peers), _ptr(peer_rows), R, _ptr(seg_src_rank),
                                 _ptr(seg_src_row), _ptr(seg_dst_row), _ptr(seg_rows), n_seg,
                                 row_bytes, _ptr(dst), dst.shape[0], _ptr(err_word),
                                 _stream(stream)), "moe_ep_copy_rows")


def moe_expert_workspace_bytes(n_rows, d, E, d_ff):
    return int(_lib.moe_expert_workspace_bytes(int(n_rows), int(d), int(E), int(d_ff)))


def moe_expert_forward(rows, counts, W1, W3, W2, y_rows, ws, stream=None):
    """The expert stage on ``rows`` [n_rows, d] bf16 laid out with each local expert's
    ``counts`` (int32 device tensor [E]) rows starting on a 128-row boundary; writes
    ``y_rows`` [n_rows, d] bf16 (see include/moe.h)."""
    n_rows, d = rows.shape
    E, _, d_ff = W1.shape
    _check(_lib.moe_expert_forward(_ptr(rows), _ptr(counts), n_rows, d, E, d_ff, _ptr(W1),
                                   _ptr(W3), _ptr(W2), _ptr(y_rows), _ptr(ws), _nbytes(ws),
                                   _stream(stream)), "moe_expert_forward")


def moe_combine(y_rows, gate, pos, out, err_word, stream=None):
    """out [T, d] = bf16(sum_j gate[t, j] y_rows[pos[t, j]]), fp32 in slot order."""
    T, k = gate.shape
    d = out.shape[1]
    _check(_lib.moe_combine(_ptr(y_rows), y_rows.shape[0], _ptr(gate), _ptr(pos), T, k, d,
                            _ptr(out), _ptr(err_word), _stream(stream)), "moe_combine")


def moe_probe_dram_read(buf, ctas, mode, out, stream=None):
    """Launch the per-SM DRAM read probe over ``buf`` (see include/moe.h)."""
    _check(_lib.moe_probe_dram_read(_ptr(buf), _nbytes(buf), int(ctas), int(mode), _ptr(out),
                                    _stream(stream)), "moe_probe_dram_read")


def moe_get_error(ws, stream=None):
    """Synchronise the stream and return the device error status recorded in ``ws``."""
    return int(_lib.moe_get_error(_ptr(ws), _stream(stream)))


def moe_set_wait_timeout_ns(ns):
    _lib.moe_set_wait_timeout_ns(int(ns))


def moe_debug_set_flags(flags):
    _lib.moe_debug_set_flags(int(flags))


def library():
    """The loaded ctypes library (for callers that want the raw C ABI)."""
    return _lib
