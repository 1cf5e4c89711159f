"""ring_attn_bwd_static_scratch: the backward for callers that cannot allocate
device memory (no workspace argument to pass on, or device memory already fully
reserved by another allocator).  Its per-row statistics live in the library's
static device array instead of a caller workspace.

Checked through the C ABI against ring_attn_bwd (caller workspace) on the same
inputs, for two calls in a row, within the parity tolerances; and a problem
beyond the array's size is refused before any launch.  The file is collected
last, and passes both alone in a fresh process and after every other test."""
import ctypes

import pytest
import torch

import ring_attn_gb300 as ra
from tests.helpers import TOL_MAX_ABS, TOL_REL_L2, check_no_device_error
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


def _close_on_device(name, got, ref):
    g, r = got.double(), ref.double()
    assert torch.isfinite(g).all(), f"{name}: non-finite values"
    mx = float((g - r).abs().max())
    assert mx <= TOL_MAX_ABS, f"{name}: max-abs {mx:.3e}"
    rel = float(torch.linalg.vector_norm(g - r) / torch.linalg.vector_norm(r).clamp_min(1e-30))
    assert rel <= TOL_REL_L2, f"{name}: rel-L2 {rel:.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("b,h,s,d,layout,n,causal", [
    (1, 4, 4096, 128, "zigzag", 4, True),
    (2, 3, 1000, 64, "stripe", 2, False),
    (1, 32, 65536, 128, "zigzag", 8, True),  # needs exactly the 16 MiB the array holds
])
def test_matches_workspace_backward_twice(lib, b, h, s, d, layout, n, causal):
    assert ra.ring_attn_workspace_size(1, b, h, s, d, n) <= ra.RA_STATIC_SCRATCH_BYTES
    x = make_qkv(b, h, s, d, seed=4242 + s, device="cuda")
    g = {k: ra.ring_attn_permute(t, layout, n) for k, t in x.items()}
    del x
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, causal)
    ref = ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, causal)
    for call in range(2):
        grads = [torch.full_like(g["q"], float("nan")) for _ in range(3)]
        got = ra.ring_attn_bwd_static_scratch(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, causal,
                                              dq=grads[0], dk=grads[1], dv=grads[2])
        torch.cuda.synchronize()
        check_no_device_error(ra)
        for name, a, r in zip(("dq", "dk", "dv"), got, ref):
            _close_on_device(f"call {call} {name}", a, r)
