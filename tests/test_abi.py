"""The C ABI without a GPU: libmoe.so loads, exports every function include/moe.h declares,
sizes its workspace, and rejects bad arguments on the host before launching anything."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", src)


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._load_builder().build()
    import combine_fp32_router_gb300 as moe
    return moe


def test_library_exports_every_declared_symbol(lib):
    names = _declared()
    assert set(names) == set(lib.EXPORTS)
    raw = lib.library()
    for n in names:
        assert hasattr(raw, n), n


def test_workspace_sizes(lib):
    small = lib.moe_workspace_bytes(64, 128, 8, 2, 256, False)
    big = lib.moe_workspace_bytes(64, 128, 8, 2, 256, True)
    assert 0 < small < big
    assert small % 256 == 0
    # the large skewed workload: padded rows P + 127 E, three row buffers of d bf16
    fwd = lib.moe_workspace_bytes(16384, 7168, 256, 8, 2048, False)
    P_pad = 16384 * 8 + 127 * 256
    assert fwd >= P_pad * 7168 * 2 * 2 + P_pad * 2048 * 2
    assert lib.moe_workspace_bytes(64, 100, 8, 2, 256, False) == 0      # d % 128 != 0
    assert lib.moe_workspace_bytes(64, 128, 8, 9, 256, False) == 0      # k > E
    assert lib.moe_workspace_bytes(64, 128, 2048, 2, 256, False) == 0   # E > 1024
    assert lib.moe_route_workspace_bytes(1000, 64, 6) > 0
    # host staging: x, logits, out copies at the end of the workspace
    hio = lib.moe_workspace_bytes(64, 128, 8, 2, 256, False, host_io=True)
    assert hio == small + 64 * 128 * 2 + 64 * 8 * 4 + 64 * 128 * 2  # each a multiple of 256
    assert lib.moe_workspace_bytes(64, 128, 8, 2, 256, True, host_io=True) == big + hio - small
    assert lib.library().moe_workspace_bytes(64, 128, 8, 2, 256, 4) == 0  # unknown need bit


def test_host_validation_rejects_before_launch(lib):
    raw = lib.library()
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    p = [fake] * 5
    st = raw.moe_forward(*p, 64, 128, 8, 9, 256, fake, fake, 1 << 30, 0, None, None)
    assert st == lib.MOE_ERR_INVALID_ARG                      # k > E
    st = raw.moe_forward(*p, 64, 100, 8, 2, 256, fake, fake, 1 << 30, 0, None, None)
    assert st == lib.MOE_ERR_UNSUPPORTED                      # d % 128 != 0
    st = raw.moe_forward(*p, -1, 128, 8, 2, 256, fake, fake, 1 << 30, 0, None, None)
    assert st == lib.MOE_ERR_INVALID_ARG                      # T < 0
    st = raw.moe_forward(*p, 64, 128, 8, 2, 256, fake, fake, 1 << 30, 8, None, None)
    assert st == lib.MOE_ERR_INVALID_ARG                      # unknown flag
    st = raw.moe_forward(*p, 64, 128, 8, 2, 256, fake, fake, 16, 0, None, None)
    assert st == lib.MOE_ERR_WORKSPACE                        # workspace too small
    mis = ctypes.c_void_p((1 << 20) + 8)
    st = raw.moe_forward(mis, *p[1:], 64, 128, 8, 2, 256, fake, fake, 1 << 30, 0, None, None)
    assert st == lib.MOE_ERR_INVALID_ARG                      # x not 16-byte aligned
    st = raw.moe_forward(None, *p[1:], 64, 128, 8, 2, 256, fake, fake, 1 << 30, 0, None, None)
    assert st == lib.MOE_ERR_INVALID_ARG                      # null x
    st = raw.moe_route_dispatch(fake, fake, 10, 64, 32, 17, *([fake] * 7), fake, 1 << 30, None)
    assert st == lib.MOE_ERR_UNSUPPORTED                      # k > 16
    st = raw.moe_backward(*([fake] * 6), 64, 128, 8, 2, 256, *([fake] * 6), fake, 16, None, None)
    assert st == lib.MOE_ERR_WORKSPACE
    assert lib.moe_status_string(lib.MOE_ERR_TIMEOUT) == "device-side wait timed out"


def test_forward_host_validation(lib):
    raw = lib.library()
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    w = [fake] * 3
    need = lib.moe_workspace_bytes(64, 128, 8, 2, 256, False, host_io=True)
    # null host buffers with T > 0
    st = raw.moe_forward_host(None, fake, *w, 64, 128, 8, 2, 256, fake, fake, need, 0, None, None)
    assert st == lib.MOE_ERR_INVALID_ARG
    st = raw.moe_forward_host(fake, fake, *w, 64, 128, 8, 2, 256, None, fake, need, 0, None, None)
    assert st == lib.MOE_ERR_INVALID_ARG
    # a workspace sized without the host staging, or without the backward state when saving
    small = lib.moe_workspace_bytes(64, 128, 8, 2, 256, False)
    st = raw.moe_forward_host(fake, fake, *w, 64, 128, 8, 2, 256, fake, fake, small, 0, None, None)
    assert st == lib.MOE_ERR_WORKSPACE
    st = raw.moe_forward_host(fake, fake, *w, 64, 128, 8, 2, 256, fake, fake, need,
                              lib.MOE_FWD_SAVE_FOR_BACKWARD, None, None)
    assert st == lib.MOE_ERR_WORKSPACE
    # shape checks as moe_forward
    st = raw.moe_forward_host(fake, fake, *w, 64, 100, 8, 2, 256, fake, fake, need, 0, None, None)
    assert st == lib.MOE_ERR_UNSUPPORTED


def test_forward_host_pipelined_validation(lib):
    raw = lib.library()
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    ev0, ev1 = ctypes.c_void_p(1 << 21), ctypes.c_void_p(1 << 22)
    w = [fake] * 3
    need = lib.moe_workspace_bytes(64, 128, 8, 2, 256, False, host_io=True)
    args = lambda: [fake, fake, *w, 64, 128, 8, 2, 256, fake, fake, need, 0, None, None, None]
    # both events are required, and they must differ
    assert raw.moe_forward_host_pipelined(*args(), None, ev1) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_forward_host_pipelined(*args(), ev0, None) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_forward_host_pipelined(*args(), ev0, ev0) == lib.MOE_ERR_INVALID_ARG
    # the rest as moe_forward_host
    a = args()
    a[0] = None
    assert raw.moe_forward_host_pipelined(*a, ev0, ev1) == lib.MOE_ERR_INVALID_ARG
    a = args()
    a[12] = lib.moe_workspace_bytes(64, 128, 8, 2, 256, False)
    assert raw.moe_forward_host_pipelined(*a, ev0, ev1) == lib.MOE_ERR_WORKSPACE
    a = args()
    a[6] = 100
    assert raw.moe_forward_host_pipelined(*a, ev0, ev1) == lib.MOE_ERR_UNSUPPORTED


def test_forward_graph_validation(lib):
    raw = lib.library()
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    h = ctypes.c_void_p(123)
    need = lib.moe_workspace_bytes(64, 128, 8, 2, 256, False)
    st = raw.moe_forward_graph_create(fake, fake, fake, fake, fake, 64, 128, 8, 9, 256, fake,
                                      fake, need, 0, ctypes.byref(h))
    assert st == lib.MOE_ERR_INVALID_ARG and not h.value          # k > E
    st = raw.moe_forward_graph_create(fake, fake, fake, fake, fake, 64, 128, 8, 2, 256, fake,
                                      fake, need - 256, 0, ctypes.byref(h))
    assert st == lib.MOE_ERR_WORKSPACE and not h.value
    assert raw.moe_forward_graph_launch(None, None) == lib.MOE_ERR_INVALID_ARG
    raw.moe_forward_graph_destroy(None)                           # no-op


def test_fp8_entry_points_validation(lib):
    raw = lib.library()
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    need = lib.moe_workspace_bytes(64, 128, 8, 2, 256, False)
    # weight quantization: K and N multiples of 128, non-null buffers
    assert raw.moe_quantize_weights_fp8(fake, 4, 100, 256, fake, fake, None) == lib.MOE_ERR_UNSUPPORTED
    assert raw.moe_quantize_weights_fp8(None, 4, 128, 256, fake, fake, None) == lib.MOE_ERR_INVALID_ARG
    # forward: k > E, missing scales, small workspace
    w = [fake] * 7
    assert raw.moe_forward_fp8(*w, 64, 128, 8, 9, 256, fake, fake, need, None, None) == \
        lib.MOE_ERR_INVALID_ARG
    args = [fake, fake, fake, fake, None, fake, fake]
    assert raw.moe_forward_fp8(*args, 64, 128, 8, 2, 256, fake, fake, need, None, None) == \
        lib.MOE_ERR_INVALID_ARG
    assert raw.moe_forward_fp8(*w, 64, 128, 8, 2, 256, fake, fake, need - 256, None, None) == \
        lib.MOE_ERR_WORKSPACE


def test_relu2_validation(lib):
    raw = lib.library()
    fake = ctypes.c_void_p(1 << 20)
    need = lib.moe_workspace_bytes(64, 128, 8, 2, 384, True)
    # no W3 needs d_ff % 256 == 0
    st = raw.moe_forward(fake, fake, fake, None, fake, 64, 128, 8, 2, 384, fake, fake, need, 0,
                         None, None)
    assert st == lib.MOE_ERR_UNSUPPORTED
    # backward: W3 and dW3 both present or both absent
    p = [fake] * 3
    st = raw.moe_backward(*p, fake, None, fake, 64, 128, 8, 2, 256, fake, fake, fake, fake, fake,
                          fake, fake, need, None, None)
    assert st == lib.MOE_ERR_INVALID_ARG


def test_expert_forward_and_combine_validation(lib):
    raw = lib.library()
    fake = ctypes.c_void_p(1 << 20)     # never dereferenced: validation fails first
    need = lib.moe_expert_workspace_bytes(1000, 256, 4, 256)
    assert need > 0 and need % 256 == 0
    assert lib.moe_expert_workspace_bytes(1000, 100, 4, 256) == 0     # d % 128 != 0
    assert lib.moe_expert_workspace_bytes(1000, 256, 2048, 256) == 0  # E > 1024
    args = lambda: [fake, fake, 1000, 256, 4, 256, fake, fake, fake, fake, fake, need, None]
    a = args()
    a[1] = None                                                        # null counts
    assert raw.moe_expert_forward(*a) == lib.MOE_ERR_INVALID_ARG
    a = args()
    a[11] = need - 256                                                 # workspace too small
    assert raw.moe_expert_forward(*a) == lib.MOE_ERR_WORKSPACE
    a = args()
    a[7] = None                                                        # no W3: d_ff % 256
    a[5] = 384
    assert raw.moe_expert_forward(*a) == lib.MOE_ERR_UNSUPPORTED
    a = args()
    a[0] = ctypes.c_void_p((1 << 20) + 8)                              # rows misaligned
    assert raw.moe_expert_forward(*a) == lib.MOE_ERR_INVALID_ARG
    # combine: k beyond 16, misaligned rows, no rows for T > 0; T = 0 launches nothing
    assert raw.moe_combine(fake, 10, fake, fake, 5, 17, 128, fake, fake, None) == \
        lib.MOE_ERR_UNSUPPORTED
    assert raw.moe_combine(ctypes.c_void_p((1 << 20) + 8), 10, fake, fake, 5, 2, 128, fake,
                           fake, None) == lib.MOE_ERR_INVALID_ARG
    assert raw.moe_combine(fake, 0, fake, fake, 5, 2, 128, fake, fake, None) == \
        lib.MOE_ERR_INVALID_ARG
    assert raw.moe_combine(None, 0, None, None, 0, 2, 128, None, None, None) == lib.MOE_OK
