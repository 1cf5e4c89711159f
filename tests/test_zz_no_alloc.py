"""ring_attn_bwd_static_scratch: the backward for callers that cannot allocate
device memory (no workspace argument to pass on, or device memory already fully
reserved by another allocator).  Its per-row statistics live in the library's
static device array instead of a caller workspace.

Checked through the C ABI against ring_attn_bwd (caller workspace) on the same
inputs: both run the same deterministic, atomic-free kernels on the same
statistics, so the gradients must be bit-identical.  Two calls on the problem
are separated by a call on other inputs and another shape, so a call that read
any part of the array before writing it would pick up stale statistics.  A
small case is also checked against the fp64 oracle, and problems beyond the
array's size are refused before any launch, after the same argument checks as
ring_attn_bwd.  The file is collected
last, and passes both alone in a fresh process and after every other test."""
import ctypes

import pytest
import torch

import ring_attn_gb300 as ra
from tests.helpers import assert_close, check_no_device_error, f64
from workload import make_qkv


@pytest.fixture(scope="module")
def lib():
    from ring_attn_gb300.build import build

    build()
    return ra.load()


def _fake(shape, dtype=ra.RA_BF16, data=0x10000):
    """A packed ra_tensor with a placeholder pointer, for calls refused before any launch."""
    t = ra._Tensor()
    t.data = data
    t.dtype = dtype
    t.ndim = len(shape)
    stride = 1
    for i in reversed(range(len(shape))):
        t.shape[i] = shape[i]
        t.stride[i] = stride
        stride *= shape[i]
    return t


def test_refuses_problems_beyond_the_static_scratch(lib):
    """b1 h64 s65536 needs 32 MiB of statistics: refused with its own status, no launch."""
    shp = (1, 64, 65536, 128)
    ts = [_fake(shp) for _ in range(5)]
    lse = _fake(shp[:3], ra.RA_FP32)
    grads = [_fake(shp) for _ in range(3)]
    assert lib.ring_attn_workspace_size(1, 1, 64, 65536, 128, 8) > ra.RA_STATIC_SCRATCH_BYTES
    st = lib.ring_attn_bwd_static_scratch(*(ctypes.byref(t) for t in ts), ctypes.byref(lse), 1, 8, 1,
                                          ctypes.c_float(0.088), *(ctypes.byref(t) for t in grads), None)
    assert st == 8
    assert b"static" in lib.ra_status_string(8)
    # argument errors still come first (65536 tokens do not split into 7 shards)
    st = lib.ring_attn_bwd_static_scratch(*(ctypes.byref(t) for t in ts), ctypes.byref(lse), 1, 7, 1,
                                          ctypes.c_float(0.088), *(ctypes.byref(t) for t in grads), None)
    assert st == 1
    # head_dim 96 is unsupported whatever the size: the same status as ring_attn_bwd gives
    shp96 = (1, 64, 65536, 96)
    ts96 = [_fake(shp96) for _ in range(5)]
    g96 = [_fake(shp96) for _ in range(3)]
    st = lib.ring_attn_bwd_static_scratch(*(ctypes.byref(t) for t in ts96), ctypes.byref(lse), 1, 8, 1,
                                          ctypes.c_float(0.1), *(ctypes.byref(t) for t in g96), None)
    assert st == 2
    # mismatched gradient shape: INVALID_ARG, not SCRATCH_LIMIT
    bad = [_fake(shp) for _ in range(2)] + [_fake((1, 64, 65536, 64))]
    st = lib.ring_attn_bwd_static_scratch(*(ctypes.byref(t) for t in ts), ctypes.byref(lse), 1, 8, 1,
                                          ctypes.c_float(0.088), *(ctypes.byref(t) for t in bad), None)
    assert st == 1


def _problem(b, h, s, d, layout, n, causal, seed):
    x = make_qkv(b, h, s, d, seed=seed, device="cuda")
    g = {k: ra.ring_attn_permute(t, layout, n) for k, t in x.items()}
    del x
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, causal)
    return g, out, lse


def _static(g, out, lse, layout, n, causal):
    grads = [torch.full_like(g["q"], float("nan")) for _ in range(3)]
    got = ra.ring_attn_bwd_static_scratch(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, causal,
                                          dq=grads[0], dk=grads[1], dv=grads[2])
    torch.cuda.synchronize()
    check_no_device_error(ra)
    return got


@pytest.mark.gpu
@pytest.mark.parametrize("b,h,s,d,layout,n,causal", [
    (1, 4, 4096, 128, "zigzag", 4, True),
    (2, 3, 1000, 64, "stripe", 2, False),
    (1, 32, 65536, 128, "zigzag", 8, True),  # needs exactly the 16 MiB the array holds
])
def test_matches_workspace_backward_twice(lib, b, h, s, d, layout, n, causal):
    assert ra.ring_attn_workspace_size(1, b, h, s, d, n) <= ra.RA_STATIC_SCRATCH_BYTES
    g, out, lse = _problem(b, h, s, d, layout, n, causal, seed=4242 + s)
    ref = ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, causal)
    torch.cuda.synchronize()
    # another problem between the two calls: other inputs, a different shape, and
    # (for the first two cases) more statistics rows than the problem under test
    other = (1, 8, 8192, 128, "contiguous", 4, True) if s < 65536 else (2, 3, 1000, 64, "stripe", 2, False)
    og, oout, olse = _problem(*other, seed=99)
    for call in range(2):
        got = _static(g, out, lse, layout, n, causal)
        for name, a, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(a, r), f"call {call} {name}: differs from ring_attn_bwd with a workspace"
        if call == 0:
            _static(og, oout, olse, *other[4:])
    del og, oout, olse


@pytest.mark.gpu
def test_small_case_against_the_oracle(lib):
    """b1 h2 s384 d64, causal zigzag over 3 shards, against the fp64 oracle."""
    import oracle

    b, h, s, d, layout, n, causal = 1, 2, 384, 64, "zigzag", 3, True
    x = make_qkv(b, h, s, d, seed=7, device="cpu")
    g = {k: ra.ring_attn_permute(t.cuda(), layout, n) for k, t in x.items()}
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, causal)
    dq, dk, dv = _static(g, out, lse, layout, n, causal)
    ref = oracle.attention_bwd(*(f64(x[k]) for k in ("q", "k", "v", "do")), d ** -0.5, causal)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(name, ra.ring_attn_unpermute(got, layout, n).cpu(), r)
