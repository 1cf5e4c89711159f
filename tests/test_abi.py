"""CPU checks of the C ABI: the library loads, exports every declared symbol,
and rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

import ring_attn_gb300 as ra

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ringattn.h")


@pytest.fixture(scope="module")
def lib():
    from ring_attn_gb300.build import build

    build()
    return ra.load()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


def test_header_declares_the_binding_symbols():
    assert sorted(ra.EXPORTED_SYMBOLS) == _declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert getattr(lib, name) is not None


def test_status_strings_and_version(lib):
    assert lib.ra_status_string(0) == b"ok"
    assert b"workspace" in lib.ra_status_string(4)
    assert lib.ra_status_string(99) == b"unknown status"
    assert lib.ring_attn_version() == 200
    assert lib.ring_attn_debug_bounds() == 0


def test_workspace_size(lib):
    assert lib.ring_attn_workspace_size(0, 1, 2, 256, 64, 2) == 0
    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # 2 shards of 128 rows: no padding; D and lse2, one float per row each
    assert lib.ring_attn_workspace_size(1, 1, 2, 256, 64, 2) == 2 * r256(1 * 2 * 2 * 128 * 4)
    # 4 shards of 64 rows: each padded to 128
    assert lib.ring_attn_workspace_size(1, 1, 2, 256, 64, 4) == 2 * r256(1 * 2 * 4 * 128 * 4)
    assert lib.ring_attn_workspace_size(1, 0, 2, 256, 64, 2) == 0
    assert lib.ring_attn_workspace_size(1, 1, 2, 256, 64, 3) == 0


def _fake(shape, dtype=ra.RA_BF16, data=0x10000, strides=None):
    t = ra._Tensor()
    t.data = data
    t.dtype = dtype
    t.ndim = len(shape)
    if strides is None:
        strides = []
        acc = 1
        for n in reversed(shape):
            strides.insert(0, acc)
            acc *= n
    for i, n in enumerate(shape):
        t.shape[i] = n
        t.stride[i] = strides[i]
    return t


def _fwd(lib, q, k, v, out, lse, layout=0, n=2, causal=1, scale=0.125):
    return lib.ring_attn_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), layout, n, causal, scale,
                             ctypes.byref(out), ctypes.byref(lse), None, 0, None)


def test_fwd_rejects_bad_arguments_before_launch(lib):
    shp = (1, 2, 256, 64)
    ok = lambda: _fake(shp)  # noqa: E731
    lse = _fake((1, 2, 256), ra.RA_FP32)
    # null data pointer
    assert _fwd(lib, _fake(shp, data=0), ok(), ok(), ok(), lse) == 1
    # wrong dtype
    assert _fwd(lib, _fake(shp, ra.RA_FP32), ok(), ok(), ok(), lse) == 1
    # shape mismatch
    assert _fwd(lib, ok(), _fake((1, 2, 128, 64)), ok(), ok(), lse) == 1
    # grouped key / value heads: hk must divide h, and k and v agree
    q3 = _fake((1, 3, 256, 64))
    assert _fwd(lib, q3, ok(), ok(), _fake((1, 3, 256, 64)), _fake((1, 3, 256), ra.RA_FP32)) == 1
    assert _fwd(lib, ok(), _fake((1, 4, 256, 64)), _fake((1, 4, 256, 64)), ok(), lse) == 1
    assert _fwd(lib, ok(), ok(), _fake((1, 1, 256, 64)), ok(), lse) == 1
    # unsupported head dim
    assert _fwd(lib, _fake((1, 2, 256, 96)), _fake((1, 2, 256, 96)), _fake((1, 2, 256, 96)),
                _fake((1, 2, 256, 96)), lse) == 2
    # s not divisible by n_shards; zigzag needs 2N
    assert _fwd(lib, ok(), ok(), ok(), ok(), lse, n=3) == 1
    assert _fwd(lib, _fake((1, 2, 24, 64)), _fake((1, 2, 24, 64)), _fake((1, 2, 24, 64)), _fake((1, 2, 24, 64)),
                _fake((1, 2, 24), ra.RA_FP32), layout=1, n=8) == 1
    # bad layout, bad causal flag, bad scale
    assert _fwd(lib, ok(), ok(), ok(), ok(), lse, layout=3) == 1
    assert _fwd(lib, ok(), ok(), ok(), ok(), lse, causal=2) == 1
    assert _fwd(lib, ok(), ok(), ok(), ok(), lse, scale=0.0) == 1
    assert _fwd(lib, ok(), ok(), ok(), ok(), lse, scale=float("nan")) == 1
    # non-contiguous head dim and misaligned strides / pointers
    assert _fwd(lib, _fake(shp, strides=(32768, 16384, 64, 2)), ok(), ok(), ok(), lse) == 3
    assert _fwd(lib, _fake(shp, strides=(32768, 16384, 68, 1)), ok(), ok(), ok(), lse) == 3
    assert _fwd(lib, _fake(shp, data=0x10008), ok(), ok(), ok(), lse) == 3
    # lse shape
    assert _fwd(lib, ok(), ok(), ok(), ok(), _fake((1, 2, 128), ra.RA_FP32)) == 1


def test_bwd_rejects_missing_workspace(lib):
    shp = (1, 2, 256, 64)
    ts = [_fake(shp) for _ in range(5)]
    lse = _fake((1, 2, 256), ra.RA_FP32)
    grads = [_fake(shp) for _ in range(3)]
    r = lib.ring_attn_bwd(*(ctypes.byref(t) for t in ts), ctypes.byref(lse), 0, 2, 1, 0.125,
                          *(ctypes.byref(t) for t in grads), None, 0, None)
    assert r == 4
    r = lib.ring_attn_bwd(*(ctypes.byref(t) for t in ts), ctypes.byref(lse), 0, 2, 1, 0.125,
                          *(ctypes.byref(t) for t in grads), ctypes.c_void_p(0x100000), 16, None)
    assert r == 4


def test_varlen_rejects_bad_cu_seqlens(lib):
    q = _fake((64, 2, 64))
    lse = _fake((2, 64), ra.RA_FP32)

    def call(cu, n, maxlen=64, layout=0):
        arr = (ctypes.c_int32 * len(cu))(*cu)
        return lib.ring_attn_varlen_fwd(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), ctypes.c_void_p(0x1000),
                                        ctypes.cast(arr, ctypes.c_void_p), n, maxlen, layout, 2, 1, 0.125,
                                        ctypes.byref(q), ctypes.byref(lse), None, 0, None)

    assert call([1, 64], 1) == 1           # cu[0] != 0
    assert call([0, 40, 30, 64], 3) == 1   # decreasing
    assert call([0, 40, 64], 2, maxlen=10) == 1  # max_seqlen too small
    assert call([0, 40, 60], 2) == 1       # total does not match the tensors
    assert call([0, 64], 0) == 1           # no sequence
    assert call([0, 42, 64], 2, layout=1) == 1   # zigzag: 42 is not a multiple of 2 * n_shards
    assert call([0, 40, 64], 2, layout=2) == 2   # stripe varlen: not supported


def test_llama3_rejects_bad_rank_and_shapes(lib):
    k = _fake((64, 2, 64))
    lse = _fake((2, 16), ra.RA_FP32)

    def call(q, rank, n=4):
        arr = (ctypes.c_int32 * 3)(0, 40, 64)
        return lib.ring_attn_llama3_varlen_fwd(ctypes.byref(q), ctypes.byref(k), ctypes.byref(k),
                                               ctypes.c_void_p(0x1000), ctypes.cast(arr, ctypes.c_void_p), 2, 64,
                                               rank, n, 1, 0.125, ctypes.byref(q), ctypes.byref(lse), None)

    assert call(_fake((16, 2, 64)), 4) == 1        # rank outside [0, n_shards)
    assert call(_fake((16, 2, 64)), -1) == 1
    assert call(_fake((32, 2, 64)), 1) == 1        # q is not the rank's slice of total / n_shards rows
    assert call(_fake((16, 2, 64)), 0, n=3) == 1   # 64 tokens do not split into 3 ranks


def test_varlen_permute_rejects_bad_arguments(lib):
    x = _fake((64, 2, 64))

    def call(cu, n, layout, n_shards=2, seq_dim=0):
        arr = (ctypes.c_int32 * len(cu))(*cu)
        return lib.ring_attn_varlen_permute(ctypes.byref(x), ctypes.byref(x), ctypes.c_void_p(0x1000),
                                            ctypes.cast(arr, ctypes.c_void_p), n, layout, n_shards, seq_dim, None)

    assert call([0, 40, 60], 2, 1) == 1    # total does not match the sequence axis
    assert call([0, 42, 64], 2, 1) == 1    # zigzag length not a multiple of 2 * n_shards
    assert call([0, 40, 64], 2, 2) == 2    # stripe varlen: not supported
    assert call([0, 40, 64], 2, 1, seq_dim=3) == 1


def test_lse_merge_rejects_bad_shapes(lib):
    oa = _fake((2, 8, 128), ra.RA_FP32)
    la = _fake((2, 8), ra.RA_FP32)
    ob = _fake((2, 8, 128), ra.RA_BF16)
    lb = _fake((2, 8), ra.RA_FP32)
    bad = _fake((2, 9, 128), ra.RA_BF16)
    assert lib.lse_merge(ctypes.byref(oa), ctypes.byref(la), ctypes.byref(bad), ctypes.byref(lb), None) == 1
    assert lib.lse_merge(ctypes.byref(oa), ctypes.byref(la), ctypes.byref(ob), ctypes.byref(_fake((2, 8))), None) == 1
    big = _fake((2, 8, 256), ra.RA_FP32)
    assert lib.lse_merge(ctypes.byref(big), ctypes.byref(la), ctypes.byref(_fake((2, 8, 256))), ctypes.byref(lb),
                         None) == 2


def test_permute_rejects_bad_arguments(lib):
    x = _fake((1, 2, 12, 8))
    far = 0x100000  # a destination that does not overlap x, so each refusal below has its own cause
    assert lib.ring_attn_permute(ctypes.byref(x), ctypes.byref(_fake((1, 2, 10, 8), data=far)), 0, 2, 2, None) == 1
    assert lib.ring_attn_permute(ctypes.byref(x), ctypes.byref(_fake((1, 2, 12, 8), data=far)), 1, 4, 2,
                                 None) == 1  # 12 % 8
    assert lib.ring_attn_permute(ctypes.byref(x), ctypes.byref(_fake((1, 2, 12, 8), data=far)), 0, 2, 4, None) == 1
    # dims after seq_dim must be packed
    y = _fake((1, 2, 12, 8), strides=(384, 192, 16, 2))
    assert lib.ring_attn_permute(ctypes.byref(y), ctypes.byref(_fake((1, 2, 12, 8), data=far)), 0, 2, 2, None) == 1


def test_permute_refuses_overlapping_buffers(lib):
    """In place, or partly overlapping: refused before any launch (rows would be
    read after other blocks overwrote them)."""
    x = _fake((1, 2, 12, 8))  # 384 bytes at 0x10000
    for lay in (0, 1, 2):
        assert lib.ring_attn_permute(ctypes.byref(x), ctypes.byref(x), lay, 2, 2, None) == 1
        assert lib.ring_attn_unpermute(ctypes.byref(x), ctypes.byref(x), lay, 2, 2, None) == 1
    for off in (2, 128, 382):
        y = _fake((1, 2, 12, 8), data=0x10000 + off)
        assert lib.ring_attn_permute(ctypes.byref(x), ctypes.byref(y), 1, 2, 2, None) == 1
        y = _fake((1, 2, 12, 8), data=0x10000 - off)
        assert lib.ring_attn_unpermute(ctypes.byref(x), ctypes.byref(y), 1, 2, 2, None) == 1
    # a strided source whose rows interleave with the destination's
    xs = _fake((1, 2, 12, 8), strides=(384, 192, 16, 1))
    y = _fake((1, 2, 12, 8), data=0x10000 + 16)
    assert lib.ring_attn_permute(ctypes.byref(xs), ctypes.byref(y), 0, 2, 2, None) == 1
    x32 = _fake((12, 4), ra.RA_FP32)
    assert lib.ring_attn_varlen_permute(ctypes.byref(x32), ctypes.byref(x32), ctypes.c_void_p(0x1000),
                                        ctypes.cast((ctypes.c_int32 * 3)(0, 8, 12), ctypes.c_void_p), 2, 0, 2, 0,
                                        None) == 1


def test_knobs(lib):
    assert lib.ring_attn_set_knob(0, 10) == 1
    assert lib.ring_attn_set_knob(1, 8) == 1
    assert lib.ring_attn_set_knob(1, -1) == 1
    assert lib.ring_attn_set_knob(1, 7) == 0
    assert lib.ring_attn_set_knob(1, 2) == 0
    assert lib.ring_attn_set_knob(7, 0) == 1
    assert lib.ring_attn_set_knob(2, 5) == 1
    assert lib.ring_attn_set_knob(2, 0) == 0
    assert lib.ring_attn_set_knob(2, 1) == 0
    assert lib.ring_attn_set_knob(0, 4_000_000_000) == 0
    assert lib.ring_attn_set_knob(1, 0) == 0


def test_binding_refuses_cpu_tensors():
    import torch

    x = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ra.ring_attn_fwd(x, x, x)


def test_debug_bounds_variant_builds_and_exports_everything():
    """The RA_DEBUG_BOUNDS build (libringattn_dbg.so) exports the same C ABI and reports itself."""
    from ring_attn_gb300.build import build

    path = build(debug_bounds=True)
    dbg = ctypes.CDLL(path)
    for name in _declared_functions():
        assert hasattr(dbg, name), name
    dbg.ring_attn_debug_bounds.restype = ctypes.c_int32
    assert dbg.ring_attn_debug_bounds() == 1


def test_library_variant_selection(monkeypatch):
    monkeypatch.setenv("RA_LIB_VARIANT", "debug_bounds")
    assert ra.lib_path().endswith("libringattn_dbg.so")
    monkeypatch.setenv("RA_LIB_VARIANT", "")
    assert ra.lib_path().endswith("libringattn.so")
    monkeypatch.setenv("RA_LIB_VARIANT", "other")
    with pytest.raises(ValueError):
        ra.lib_path()


def test_varlen_workspace_sizes(lib):
    T = lambda total, h, d: -(-total * h * d * 2 // 256) * 256  # noqa: E731
    Lb = lambda total, h: -(-total * h * 4 // 256) * 256  # noqa: E731
    total, h, d, n = 131072, 32, 128, 8
    stats = lib.ring_attn_workspace_size(1, 1, h, total, d, n)
    assert lib.ring_attn_varlen_workspace_size(0, total, h, d, 0, n) == 0
    assert lib.ring_attn_varlen_workspace_size(1, total, h, d, 0, n) == stats
    M = Lb(total, 1)  # the token map and its inverse: total int32 each
    assert lib.ring_attn_varlen_workspace_size(0, total, h, d, 1, n) == 3 * T(total, h, d) + 2 * M
    # the backward copies dO, q, k, v; out and lse are read in place
    assert lib.ring_attn_varlen_workspace_size(1, total, h, d, 1, n) == stats + 4 * T(total, h, d) + 2 * M
    assert lib.ring_attn_varlen_workspace_size(0, total, h, 96, 1, n) == 0    # head_dim
    assert lib.ring_attn_varlen_workspace_size(0, total + 1, h, d, 1, n) == 0  # total % n_shards
    assert lib.ring_attn_varlen_workspace_size(0, total, h, d, 2, n) == 0     # stripe varlen
    assert ra.ring_attn_varlen_workspace_size(1, total, h, d, "zigzag", n) == lib.ring_attn_varlen_workspace_size(
        1, total, h, d, 1, n)
