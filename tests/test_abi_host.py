"""Host-side tests of the C ABI (no GPU): the library loads, exports every declared
symbol, and rejects bad arguments before touching a device."""
import ctypes
import re
import os

import pytest
import torch

import mixture_experts_layer_92_b300 as moe
from mixture_experts_layer_92_b300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(moe_\w+)\s*\(", src, re.M)))


def test_every_declared_symbol_is_exported():
    names = declared_symbols()
    assert len(names) >= 14
    lib = ctypes.CDLL(_lib.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(_lib.EXPORTED) == names


def test_capacity():
    assert moe.moe_capacity(1.25, 256, 2, 8) == 80
    assert moe.moe_capacity(1.0, 16384, 1, 128) == 128
    assert moe.moe_capacity(1.25, 64, 2, 8) == 20
    assert moe.moe_capacity(100.0, 50, 2, 4) == 50          # clamped: C = T means no drop
    assert moe.moe_capacity(0.0, 50, 2, 4) == 0
    assert moe.moe_capacity(1.0, 10, 1, 0) == -1
    assert moe.moe_capacity(-1.0, 10, 1, 2) == -1


def shape(**kw):
    base = dict(T=64, d=128, E=8, k=2, d_ff=256, gate="softmax_topk", dtype=torch.bfloat16)
    base.update(kw)
    return moe.make_shape(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(k=0), -1), (dict(k=9), -1), (dict(E=0), -1), (dict(E=1025, k=2), -1),
    (dict(T=-1), -1), (dict(d=0), -1), (dict(d_ff=0), -1), (dict(capacity=-1), -1),
    (dict(gate=7), -1), (dict(dtype=5), -1), (dict(d_ff_shared=-8), -1),
    (dict(d=100), -2), (dict(d_ff=260), -2), (dict(d_ff_shared=12), -2),
    (dict(T=1 << 30, k=2), -1),
    (dict(dtype=torch.float32, d=6), -2),
])
def test_invalid_shapes(kw, status):
    s = shape(**kw)
    assert moe.moe_check_shape(s) == status
    assert moe.moe_workspace_size(s) == 0
    assert _lib.LIB.moe_last_error_detail().decode() != ""


def test_valid_shapes_and_workspace_monotone():
    s1 = shape(T=64)
    s2 = shape(T=128)
    assert moe.moe_check_shape(s1) == 0
    n1, n2 = moe.moe_workspace_size(s1), moe.moe_workspace_size(s2)
    assert 0 < n1 < n2 and n1 % 256 == 0
    # the largest workload fits comfortably in HBM
    ds = shape(T=8192, d=7168, E=256, k=8, d_ff=2048, d_ff_shared=2048, gate="sigmoid_topk")
    assert moe.moe_workspace_size(ds) < 4 << 30


def test_workspace_dispatch_offsets():
    """The forward's perm, inv and offsets sit inside the workspace, apart from one another,
    4-byte aligned; expert-choice shapes and invalid shapes are refused."""
    for kw in (dict(T=64), dict(T=1000, E=128, k=1), dict(T=8192, d=7168, E=256, k=8, d_ff=2048,
                                                        gate="sigmoid_topk")):
        s = shape(**kw)
        n = moe.moe_workspace_size(s)
        po, io, oo = _lib.moe_workspace_dispatch_offsets(s)
        A, E = s.T * s.k, s.E
        spans = sorted([(po, po + 4 * A), (io, io + 4 * A), (oo, oo + 4 * (E + 1))])
        assert all(b <= n for _, b in spans)
        assert all(spans[i][1] <= spans[i + 1][0] for i in range(2))
        assert po % 4 == io % 4 == oo % 4 == 0
    with pytest.raises(_lib.MoeError) as ei:
        _lib.moe_workspace_dispatch_offsets(shape(T=64, gate="expert_choice"))
    assert ei.value.status == -2
    with pytest.raises(_lib.MoeError) as ei:
        _lib.moe_workspace_dispatch_offsets(shape(T=64, k=9))
    assert ei.value.status == -1


def _ws_bytes(n):
    return ctypes.c_size_t(n)


def test_entry_points_reject_before_any_launch():
    """Invalid arguments return an error on the host: no CUDA call is made, so these run
    on a machine without a GPU."""
    L = _lib.LIB
    s = shape()
    need = moe.moe_workspace_size(s)
    fake = ctypes.c_void_p(0x7f0000000000)          # never dereferenced
    null = ctypes.c_void_p(None)
    # no workspace
    assert L.moe_forward(ctypes.byref(s), fake, fake, null, fake, fake, fake, null, null, null,
                         fake, null, null, null, null, need, null) == -4
    # workspace too small
    assert L.moe_forward(ctypes.byref(s), fake, fake, null, fake, fake, fake, null, null, null,
                         fake, null, null, null, fake, need - 1, null) == -4
    # misaligned workspace
    assert L.moe_forward(ctypes.byref(s), fake, fake, null, fake, fake, fake, null, null, null,
                         fake, null, null, null, ctypes.c_void_p(0x7f0000000010), need, null) == -4
    # missing x
    assert L.moe_forward(ctypes.byref(s), null, fake, null, fake, fake, fake, null, null, null,
                         fake, null, null, null, fake, need, null) == -1
    # misaligned weight
    assert L.moe_forward(ctypes.byref(s), fake, fake, null, ctypes.c_void_p(0x7f0000000002), fake,
                         fake, null, null, null, fake, null, null, null, fake, need, null) == -1
    # shared expert declared but its weights missing
    s2 = shape(d_ff_shared=128)
    n2 = moe.moe_workspace_size(s2)
    assert L.moe_forward(ctypes.byref(s2), fake, fake, null, fake, fake, fake, null, null, null,
                         fake, null, null, null, fake, n2, null) == -1
    # wrong event count
    ev = (ctypes.c_void_p * 3)()
    assert L.moe_forward_events(ctypes.byref(s), fake, fake, null, fake, fake, fake, null, null,
                                null, fake, null, null, null, fake, need, null, ev, 3) == -1
    # dispatch without indices or logits
    assert L.moe_dispatch(ctypes.byref(s), null, null, fake, fake, fake, fake, fake, fake, need,
                          null) == -1
    # route without logits and without x
    assert L.moe_route_topk(ctypes.byref(s), null, fake, null, null, null, fake, fake, null, fake,
                            need, null) == -1
    # combine with a misaligned output
    assert L.moe_combine(ctypes.byref(s), fake, fake, null, ctypes.c_void_p(0x7f0000000004),
                         null) == -1
    assert L.moe_aux_loss(ctypes.byref(s), null, fake, fake, null) == -1
    # the host-memory forward checks everything before its first copy
    def host_fwd(xh=fake, yh=fake, xd=fake, yd=fake, lh=null, wsp=fake, nbytes=need):
        return L.moe_forward_host(ctypes.byref(s), xh, fake, null, fake, fake, fake, null, null,
                                  null, yh, lh, xd, yd, wsp, nbytes, null)
    assert host_fwd(xh=null) == -1
    assert host_fwd(yh=null) == -1
    assert host_fwd(xd=null) == -1
    assert host_fwd(yd=ctypes.c_void_p(0x7f0000000008)) == -1     # misaligned device y
    assert host_fwd(lh=ctypes.c_void_p(0x7f0000000002)) == -1     # misaligned host losses
    assert host_fwd(wsp=null) == -4
    assert host_fwd(nbytes=need - 1) == -4


def test_status_strings():
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert moe.moe_status_string(code) != "unknown status"
    assert moe.moe_status_string(42) == "unknown status"


@pytest.mark.parametrize("kw", [
    dict(d=96), dict(d_ff=200), dict(d_ff_shared=96), dict(E=12, k=2),
])
def test_backward_unsupported_shapes(kw):
    """bf16 layers need d, d_ff, d_ff_shared multiples of 64 and E a multiple of 8 for the
    backward pass: anything else is refused on the host (workspace size 0). fp32 layers have
    no tile constraints; expert-choice layers are supported."""
    s = shape(**kw)
    assert moe.moe_backward_workspace_size(s) == 0
    assert moe.moe_backward_workspace_size(shape(dtype=torch.float32, d=96, d_ff=200, E=12)) > 0
    ec = shape(gate="expert_choice", capacity=40)
    assert moe.moe_backward_workspace_size(ec) > moe.moe_workspace_size(ec) > 0


def test_backward_rejects_before_any_launch():
    L = _lib.LIB
    s = shape()
    need = moe.moe_backward_workspace_size(s)
    assert need > moe.moe_workspace_size(s) > 0 and need % 256 == 0
    fake = ctypes.c_void_p(0x7f0000000000)
    null = ctypes.c_void_p(None)

    def call(ws=fake, nbytes=need, x=fake, dy=fake, dw1=fake, dw1s=null, shp=s, ev=None, nev=0):
        return L.moe_backward(ctypes.byref(shp), x, fake, null, fake, fake, fake, null, null, null,
                              dy, 1.0, 1.0, fake, fake, null, dw1, fake, fake, dw1s, null, null,
                              null, null, ws, nbytes, null, ev, nev)
    assert call(ws=null) == -4
    assert call(nbytes=need - 1) == -4
    assert call(x=null) == -1
    assert call(dy=null) == -1
    assert call(dw1=null) == -1
    assert call(dw1=ctypes.c_void_p(0x7f0000000008)) == -1
    s2 = shape(d_ff_shared=128)
    assert call(shp=s2, nbytes=moe.moe_backward_workspace_size(s2)) == -1   # shared grads missing
    assert call(ev=(ctypes.c_void_p * 3)(), nev=3) == -1
    assert call(shp=shape(d=96)) == -2


def test_host_pipeline_rejects_before_any_cuda_call():
    """The host pipeline's argument checks run on the host; on a machine without a GPU its
    creation fails with MOE_ERR_CUDA and hands back no handle."""
    import torch
    L = _lib.LIB
    s = shape()
    h = ctypes.c_void_p()
    null = ctypes.c_void_p(None)
    fake = ctypes.c_void_p(0x7f0000000000)
    # two slots of x and y [T, d] and the losses, each rounded up to 256 bytes
    row_bytes = -(-s.T * s.d * (2 if s.dtype == 1 else 4) // 256) * 256
    need = L.moe_host_pipeline_buffer_size(ctypes.byref(s))
    assert need == 2 * (2 * row_bytes + 256)
    assert L.moe_host_pipeline_create(ctypes.byref(s), fake, need, None) == -1
    bad = shape()
    bad.k = bad.E + 1
    assert L.moe_host_pipeline_buffer_size(ctypes.byref(bad)) == 0
    assert L.moe_host_pipeline_create(ctypes.byref(bad), fake, need, ctypes.byref(h)) == -1
    assert h.value is None
    assert L.moe_host_pipeline_create(ctypes.byref(s), null, need, ctypes.byref(h)) == -4
    assert L.moe_host_pipeline_create(ctypes.byref(s), fake, need - 1, ctypes.byref(h)) == -4
    assert L.moe_host_pipeline_create(ctypes.byref(s), ctypes.c_void_p(0x7f0000000010), need,
                                      ctypes.byref(h)) == -4            # misaligned
    assert h.value is None
    assert L.moe_host_pipeline_forward(null, ctypes.byref(s), fake, fake, null, fake, fake, fake,
                                       null, null, null, fake, null, fake,
                                       moe.moe_workspace_size(s), null) == -1
    assert L.moe_host_pipeline_join(null, null) == -1
    assert L.moe_host_pipeline_destroy(null) == 0
    if not torch.cuda.is_available():
        assert L.moe_host_pipeline_create(ctypes.byref(s), fake, need, ctypes.byref(h)) == -3
        assert h.value is None


def test_selftest_rejects_bad_workspace_before_any_launch():
    """The bounded-wait diagnostic validates its workspace on the host (no GPU needed)."""
    L = _lib.LIB
    assert L.moe_selftest_wait_timeout(None, 4096, None) == -4
    assert L.moe_selftest_wait_timeout(ctypes.c_void_p(0x7f0000000008), 4096, None) == -4  # misaligned
    assert L.moe_selftest_wait_timeout(ctypes.c_void_p(0x7f0000000000), 8, None) == -4      # too small


def test_noalloc_rejects_before_any_launch():
    """moe_route_topk_noalloc checks its pointers and the gate mode on the host, like the
    workspace entry points: a misaligned pointer or an expert-choice layer is refused before
    any CUDA call (so this runs without a GPU)."""
    L = _lib.LIB
    s = shape()
    fake = ctypes.c_void_p(0x7f0000000000)          # never dereferenced
    odd = ctypes.c_void_p(0x7f0000000002)
    null = ctypes.c_void_p(None)
    call = lambda l, i, g, st, sh=s: L.moe_route_topk_noalloc(ctypes.byref(sh), l, i, g, st, null)
    assert call(null, fake, fake, null) == -1       # no logits
    assert call(odd, fake, fake, null) == -1        # misaligned logits
    assert call(fake, odd, fake, null) == -1        # misaligned indices
    assert call(fake, fake, odd, null) == -1        # misaligned gates
    assert call(fake, fake, fake, odd) == -1        # misaligned statistics
    assert "aligned" in _lib.LIB.moe_last_error_detail().decode()
    ec = shape(gate=3, capacity=16)
    assert call(fake, fake, fake, null, ec) == -2   # expert choice has no top-k step
    empty = shape(T=0)
    assert call(null, null, null, odd, empty) == -1  # checked even for an empty batch


def test_block_scaled_entry_points_reject_before_any_launch():
    """moe_forward_mx and moe_mx_quantize check shapes, formats and pointers on the host: no
    CUDA call is made for these (so this runs without a GPU)."""
    L = _lib.LIB
    fake = ctypes.c_void_p(0x7f0000000000)
    odd32 = ctypes.c_void_p(0x7f0000000010)         # 16- but not 32-byte aligned
    null = ctypes.c_void_p(None)
    s = shape(d=256, d_ff=256)
    need = _lib.moe_mx_workspace_size(s)
    assert need > moe.moe_workspace_size(s)         # the block-scaled operands come on top
    def fwd(fmt=0, sh=s, w=(fake,) * 6, nbytes=need, ws=fake):
        return L.moe_forward_mx(ctypes.byref(sh), fmt, fake, fake, null, *w, fake, null, null,
                                null, ws, nbytes, null, None, 0)
    assert fwd(fmt=7) == -1                         # unknown format
    assert fwd(sh=shape(d=200, d_ff=256)) == -2     # d % 256
    assert fwd(sh=shape(d=256, d_ff=200)) == -2     # d_ff % 128
    assert fwd(sh=shape(d=256, d_ff=256, dtype=torch.float32)) == -2
    assert fwd(sh=shape(d=256, d_ff=256, d_ff_shared=128)) == -2
    assert fwd(sh=shape(d=256, d_ff=256, gate=3, capacity=16)) == -2   # expert choice
    assert fwd(nbytes=need - 1) == -4               # the plain workspace is not enough
    assert fwd(w=(null,) + (fake,) * 5) == -1       # missing codes
    assert fwd(w=(fake, null) + (fake,) * 4) == -1  # missing scales
    assert fwd(fmt=1, w=(odd32,) + (fake,) * 5) == -1   # 4-bit codes need 32-byte alignment
    q = L.moe_mx_quantize
    assert q(fake, 4, 100, fake, fake, null, null) == -1     # K not a multiple of 32
    assert q(fake, -1, 64, fake, fake, null, null) == -1
    assert q(null, 4, 64, fake, fake, null, null) == -1
    assert q(fake, 4, 64, fake, null, null, null) == -1
    assert q(fake, 4, 64, fake, fake, ctypes.c_void_p(0x7f0000000010), null) == -4
    assert q(null, 0, 64, null, null, null, null) == 0       # nothing to do


@pytest.mark.parametrize("T", [1, 64, 4096])
def test_block_scaled_workspace_grows_with_the_layer(T):
    a = _lib.moe_mx_workspace_size(shape(T=T, d=256, d_ff=256))
    b = _lib.moe_mx_workspace_size(shape(T=T, d=512, d_ff=256))
    c = _lib.moe_mx_workspace_size(shape(T=T, d=256, d_ff=512))
    assert 0 < a < b and a < c
    assert a % 256 == 0
