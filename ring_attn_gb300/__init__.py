"""Python binding of libringattn (GB300 / sm_103a blockwise ring attention).

Every call marshals torch tensors into the C ABI declared in
``include/ringattn.h`` and launches the library's CUDA kernels on the current
torch stream.  torch only provides device memory and streams; no step of the
computation runs in Python or in torch.  There is no fallback: if the shared
library is missing or a tensor is not on a CUDA device the call raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

__all__ = [
    "LAYOUTS", "RingAttnError", "lib_path", "load", "ring_attn_fwd", "ring_attn_fwd_step", "ring_attn_bwd",
    "ring_attn_varlen_fwd", "ring_attn_varlen_bwd", "lse_merge", "ring_attn_permute", "ring_attn_unpermute",
    "ring_attn_workspace_size", "ring_attn_check_device_error", "ring_attn_set_knob", "ring_attn_version",
    "ring_attn_timing_enable", "ring_attn_timing_read", "ring_attn_bwd_static_scratch", "EXPORTED_SYMBOLS",
    "KERNELS", "RA_STATIC_SCRATCH_BYTES", "ring_attn_qkvpacked_fwd", "ring_attn_qkvpacked_bwd", "ring_attn_kvpacked_fwd",
    "ring_attn_kvpacked_bwd", "ring_attn_varlen_qkvpacked_fwd", "ring_attn_varlen_qkvpacked_bwd",
    "ring_attn_varlen_kvpacked_fwd", "ring_attn_varlen_kvpacked_bwd", "ring_attn_varlen_permute",
    "ring_attn_varlen_unpermute", "ring_attn_llama3_varlen_fwd", "ring_attn_llama3_varlen_bwd", "CuSeqlens",
]

LAYOUTS = {"contiguous": 0, "zigzag": 1, "stripe": 2}
RA_BF16, RA_FP32 = 0, 1
RA_OP_FWD, RA_OP_BWD = 0, 1
RA_KNOB_WAIT_LIMIT_NS, RA_KNOB_DEBUG_FLAGS, RA_KNOB_DKDV_PAIR = 0, 1, 2

# Every extern "C" symbol include/ringattn.h declares.
EXPORTED_SYMBOLS = (
    "ring_attn_fwd", "ring_attn_fwd_step", "lse_merge", "ring_attn_bwd", "ring_attn_varlen_fwd",
    "ring_attn_varlen_bwd", "ring_attn_permute", "ring_attn_unpermute", "ring_attn_workspace_size",
    "ring_attn_check_device_error", "ring_attn_set_knob", "ring_attn_timing_enable", "ring_attn_timing_read",
    "ra_status_string", "ring_attn_version", "ring_attn_bwd_static_scratch", "ring_attn_varlen_permute",
    "ring_attn_varlen_unpermute", "ring_attn_llama3_varlen_fwd", "ring_attn_llama3_varlen_bwd",
    "ring_attn_debug_bounds", "ring_attn_varlen_workspace_size",
)
RA_STATIC_SCRATCH_BYTES = 16 << 20
KERNELS = {"fwd": 0, "bwd_dkdv": 1, "bwd_pre": 2, "bwd_dq": 3, "permute": 4, "lse_merge": 5}


class RingAttnError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} (status {status})")
        self.status = status


class _Tensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


_LIB = None


def lib_path() -> str:
    """libringattn.so, or the debug-bounds variant libringattn_dbg.so when
    RA_LIB_VARIANT=debug_bounds (build it with build(debug_bounds=True))."""
    variant = os.environ.get("RA_LIB_VARIANT", "")
    if variant not in ("", "debug_bounds"):
        raise ValueError(f"RA_LIB_VARIANT={variant!r}: expected 'debug_bounds' or unset")
    name = "libringattn_dbg.so" if variant == "debug_bounds" else "libringattn.so"
    return os.path.join(os.path.dirname(os.path.abspath(__file__)), name)


def load():
    """Loads libringattn.so (raises if it has not been built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with ring_attn_gb300.build.build() "
                           "(or __graft_entry__.build()); there is no fallback path")
    lib = ctypes.CDLL(path)
    P, I32, I64, F32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    T = ctypes.POINTER(_Tensor)
    sig = {
        "ring_attn_fwd": [T, T, T, I32, I32, I32, F32, T, T, P, SZ, P],
        "ring_attn_fwd_step": [T, T, T, I32, I32, I32, F32, I32, T, T, P],
        "lse_merge": [T, T, T, T, P],
        "ring_attn_bwd": [T, T, T, T, T, T, I32, I32, I32, F32, T, T, T, P, SZ, P],
        "ring_attn_bwd_static_scratch": [T, T, T, T, T, T, I32, I32, I32, F32, T, T, T, P],
        "ring_attn_varlen_fwd": [T, T, T, P, P, I32, I32, I32, I32, I32, F32, T, T, P, SZ, P],
        "ring_attn_varlen_bwd": [T, T, T, T, T, T, P, P, I32, I32, I32, I32, I32, F32, T, T, T, P, SZ, P],
        "ring_attn_varlen_permute": [T, T, P, P, I32, I32, I32, I32, P],
        "ring_attn_llama3_varlen_fwd": [T, T, T, P, P, I32, I32, I32, I32, I32, F32, T, T, P],
        "ring_attn_llama3_varlen_bwd": [T, T, T, T, T, T, P, P, I32, I32, I32, I32, I32, F32, T, T, T, P, SZ, P],
        "ring_attn_varlen_unpermute": [T, T, P, P, I32, I32, I32, I32, P],
        "ring_attn_permute": [T, T, I32, I32, I32, P],
        "ring_attn_unpermute": [T, T, I32, I32, I32, P],
        "ring_attn_check_device_error": [P, ctypes.POINTER(I32)],
        "ring_attn_set_knob": [I32, I64],
        "ring_attn_timing_enable": [I32],
        "ring_attn_timing_read": [I32, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(I64)],
    }
    for name, args in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = I32
    lib.ring_attn_workspace_size.argtypes = [I32, I64, I64, I64, I64, I32]
    lib.ring_attn_workspace_size.restype = SZ
    lib.ring_attn_varlen_workspace_size.argtypes = [I32, I64, I64, I64, I32, I32]
    lib.ring_attn_varlen_workspace_size.restype = SZ
    lib.ra_status_string.argtypes = [I32]
    lib.ra_status_string.restype = ctypes.c_char_p
    lib.ring_attn_version.argtypes = []
    lib.ring_attn_version.restype = I32
    lib.ring_attn_debug_bounds.argtypes = []
    lib.ring_attn_debug_bounds.restype = I32
    _LIB = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        msg = load().ra_status_string(status).decode()
        raise RingAttnError(status, f"{what}: {msg}")


def _layout(layout) -> int:
    if isinstance(layout, str):
        if layout not in LAYOUTS:
            raise ValueError(f"unknown layout {layout!r}")
        return LAYOUTS[layout]
    return int(layout)


def _t(x: torch.Tensor) -> _Tensor:
    if not isinstance(x, torch.Tensor) or not x.is_cuda:
        raise ValueError("ring_attn_gb300 takes CUDA tensors only")
    if x.dtype == torch.bfloat16:
        dt = RA_BF16
    elif x.dtype == torch.float32:
        dt = RA_FP32
    else:
        raise ValueError(f"unsupported dtype {x.dtype}")
    if x.dim() > 4 or x.dim() < 1:
        raise ValueError("tensors must have 1 to 4 dimensions")
    t = _Tensor()
    t.data = x.data_ptr()
    t.dtype = dt
    t.ndim = x.dim()
    for i in range(x.dim()):
        t.shape[i] = x.shape[i]
        t.stride[i] = x.stride(i)
    return t


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _scale(scale, d):
    return float(1.0 / math.sqrt(d) if scale is None else scale)


def ring_attn_fwd(q, k, v, layout="contiguous", n_shards=1, causal=False, softmax_scale=None, out=None, lse=None,
                  stream=None):
    """Ring forward with the fp32 LSE merge fused.  q, k, v: (b, h, s, d) bf16 in layout order
    (k and v may have hk heads, hk dividing h: query head i uses key / value head i // (h // hk)).

    Returns (out (b, h, s, d) bf16, lse (b, h, s) fp32), both in layout order."""
    lib = load()
    b, h, s, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((b, h, s), dtype=torch.float32, device=q.device)
    tq, tk, tv, to, tl = _t(q), _t(k), _t(v), _t(out), _t(lse)
    _check(lib.ring_attn_fwd(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), _layout(layout), int(n_shards),
                             int(bool(causal)), _scale(softmax_scale, d), ctypes.byref(to), ctypes.byref(tl),
                             None, 0, _stream(stream)), "ring_attn_fwd")
    return out, lse


def ring_attn_fwd_step(q, k, v, step, layout="contiguous", n_shards=1, causal=False, softmax_scale=None,
                       out_blk=None, lse_blk=None, out_dtype=torch.float32, stream=None):
    """One ring step: every Q shard r against KV shard (r - step) mod N; block out and lse."""
    lib = load()
    b, h, s, d = q.shape
    if out_blk is None:
        out_blk = torch.empty((b, h, s, d), dtype=out_dtype, device=q.device)
    if lse_blk is None:
        lse_blk = torch.empty((b, h, s), dtype=torch.float32, device=q.device)
    tq, tk, tv, to, tl = _t(q), _t(k), _t(v), _t(out_blk), _t(lse_blk)
    _check(lib.ring_attn_fwd_step(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv), _layout(layout),
                                  int(n_shards), int(bool(causal)), _scale(softmax_scale, d), int(step),
                                  ctypes.byref(to), ctypes.byref(tl), _stream(stream)), "ring_attn_fwd_step")
    return out_blk, lse_blk


def lse_merge(out_acc, lse_acc, out_blk, lse_blk, stream=None):
    """In-place merge of a block result into (out_acc fp32, lse_acc fp32)."""
    lib = load()
    a, b_, c, d = _t(out_acc), _t(lse_acc), _t(out_blk), _t(lse_blk)
    _check(lib.lse_merge(ctypes.byref(a), ctypes.byref(b_), ctypes.byref(c), ctypes.byref(d), _stream(stream)),
           "lse_merge")
    return out_acc, lse_acc


def ring_attn_workspace_size(op, b, h, s, d, n_shards=1) -> int:
    return int(load().ring_attn_workspace_size(int(op), int(b), int(h), int(s), int(d), int(n_shards)))


def ring_attn_varlen_workspace_size(op, total, h, d, layout="contiguous", n_shards=1) -> int:
    """Bytes of a varlen call's workspace (for zigzag: the original-order copies, see the C header)."""
    return int(load().ring_attn_varlen_workspace_size(int(op), int(total), int(h), int(d), _layout(layout),
                                                      int(n_shards)))


def _ws_arg(workspace):
    """(pointer, bytes) of an optional workspace tensor."""
    if workspace is None:
        return None, 0
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()


def ring_attn_bwd(dout, q, k, v, out, lse, layout="contiguous", n_shards=1, causal=False, softmax_scale=None,
                  dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients (dq like q, dk and dv like k and v), bf16, layout order."""
    lib = load()
    b, h, s, d = q.shape
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = ring_attn_workspace_size(RA_OP_BWD, b, h, s, d, n_shards)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ts = [_t(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    r = [ctypes.byref(x) for x in ts]
    _check(lib.ring_attn_bwd(r[0], r[1], r[2], r[3], r[4], r[5], _layout(layout), int(n_shards), int(bool(causal)),
                             _scale(softmax_scale, d), r[6], r[7], r[8], ctypes.c_void_p(workspace.data_ptr()),
                             workspace.numel() * workspace.element_size(), _stream(stream)), "ring_attn_bwd")
    return dq, dk, dv


def ring_attn_bwd_static_scratch(dout, q, k, v, out, lse, layout="contiguous", n_shards=1, causal=False,
                                 softmax_scale=None, dq=None, dk=None, dv=None, stream=None):
    """ring_attn_bwd with the library's static device scratch instead of a workspace.

    The library call allocates nothing; only the outputs this wrapper creates when
    dq, dk or dv is None are allocated here, so callers that cannot allocate pass
    all three.  Calls that may overlap on the GPU race on the shared scratch."""
    lib = load()
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ts = [_t(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    r = [ctypes.byref(x) for x in ts]
    _check(lib.ring_attn_bwd_static_scratch(r[0], r[1], r[2], r[3], r[4], r[5], _layout(layout), int(n_shards),
                                            int(bool(causal)), _scale(softmax_scale, q.shape[-1]), r[6], r[7], r[8],
                                            _stream(stream)), "ring_attn_bwd_static_scratch")
    return dq, dk, dv


class CuSeqlens:
    """One cu_seqlens prepared once for repeated varlen calls.

    Holds the int32 host copy that the library validates before each launch and
    the device copy that its kernels read, so that a call given a CuSeqlens
    copies and allocates nothing for it (a plain list or tensor passed to a
    varlen call is copied to the device on every call)."""

    def __init__(self, cu_seqlens, device):
        if isinstance(cu_seqlens, torch.Tensor):
            host = cu_seqlens.detach().to("cpu", torch.int32).contiguous()
        else:
            host = torch.tensor(list(cu_seqlens), dtype=torch.int32)
        if host.dim() != 1 or host.numel() < 2:
            raise ValueError("cu_seqlens must be a 1-D array of n_seqs + 1 prefix sums")
        self.host = host
        self.dev = host.to(device)
        self.n_seqs = host.numel() - 1
        self.total = int(host[-1])
        self.max_seqlen = int((host[1:] - host[:-1]).max())


def _max_len(cu_seqlens, host):
    if isinstance(cu_seqlens, CuSeqlens):
        return cu_seqlens.max_seqlen
    return int((host[1:] - host[:-1]).max())


def _cu_pair(cu_seqlens, device):
    """(host, device) copies of cu_seqlens; a CuSeqlens is used as it is."""
    if isinstance(cu_seqlens, CuSeqlens):
        if cu_seqlens.dev.device != torch.device(device):
            raise ValueError(f"CuSeqlens was prepared for {cu_seqlens.dev.device}, not {device}")
        return cu_seqlens.host, cu_seqlens.dev
    c = CuSeqlens(cu_seqlens, device)
    return c.host, c.dev


def ring_attn_varlen_fwd(q, k, v, cu_seqlens, max_seqlen=None, n_shards=1, causal=True, softmax_scale=None,
                         out=None, lse=None, stream=None, layout="contiguous", workspace=None):
    """Packed sequences, one cu_seqlens.  q, k, v: (total, h, d) or (h, total, d) bf16 in
    layout order ("contiguous" slices of the packed buffer, or "zigzag" per sequence);
    k and v may have fewer heads than q (grouped-query attention, as in ring_attn_fwd).

    workspace: None allocates what ring_attn_varlen_workspace_size asks for (for
    zigzag, the original-order copies the library computes in); pass a tensor to
    reuse one (an empty tensor runs the zigzag kernels directly).
    Returns (out like q, lse (h, total) fp32)."""
    lib = load()
    host, dev = _cu_pair(cu_seqlens, q.device)
    n = host.numel() - 1
    total = int(host[-1])
    if max_seqlen is None:
        max_seqlen = _max_len(cu_seqlens, host)
    h = q.shape[1] if q.shape[0] == total else q.shape[0]
    d = q.shape[2]
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((h, total), dtype=torch.float32, device=q.device) if lse is None else lse
    if workspace is None:
        need = ring_attn_varlen_workspace_size(RA_OP_FWD, total, h, d, layout, n_shards)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device) if need else None
    wp, wb = _ws_arg(workspace)
    tq, tk, tv, to, tl = _t(q), _t(k), _t(v), _t(out), _t(lse)
    _check(lib.ring_attn_varlen_fwd(ctypes.byref(tq), ctypes.byref(tk), ctypes.byref(tv),
                                    ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(host.data_ptr()), n,
                                    int(max_seqlen), _layout(layout), int(n_shards), int(bool(causal)),
                                    _scale(softmax_scale, d), ctypes.byref(to), ctypes.byref(tl), wp, wb,
                                    _stream(stream)),
           "ring_attn_varlen_fwd")
    return out, lse


def ring_attn_varlen_bwd(dout, q, k, v, out, lse, cu_seqlens, max_seqlen=None, n_shards=1, causal=True,
                         softmax_scale=None, dq=None, dk=None, dv=None, workspace=None, stream=None,
                         layout="contiguous"):
    lib = load()
    host, dev = _cu_pair(cu_seqlens, q.device)
    n = host.numel() - 1
    total = int(host[-1])
    if max_seqlen is None:
        max_seqlen = _max_len(cu_seqlens, host)
    h = q.shape[1] if q.shape[0] == total else q.shape[0]
    d = q.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if workspace is None:
        ws_bytes = ring_attn_varlen_workspace_size(RA_OP_BWD, total, h, d, layout, n_shards)
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ts = [_t(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    r = [ctypes.byref(x) for x in ts]
    _check(lib.ring_attn_varlen_bwd(r[0], r[1], r[2], r[3], r[4], r[5], ctypes.c_void_p(dev.data_ptr()),
                                    ctypes.c_void_p(host.data_ptr()), n, int(max_seqlen), _layout(layout),
                                    int(n_shards), int(bool(causal)), _scale(softmax_scale, d), r[6], r[7], r[8],
                                    ctypes.c_void_p(workspace.data_ptr()),
                                    workspace.numel() * workspace.element_size(), _stream(stream)),
           "ring_attn_varlen_bwd")
    return dq, dk, dv


# ---------------------------------------------------------------------------- llama3 form
def _heads_of(x, rows):
    return x.shape[1] if x.shape[0] == rows else x.shape[0]


def ring_attn_llama3_varlen_fwd(q, k, v, cu_seqlens, rank, n_shards, causal=True, softmax_scale=None, max_seqlen=None,
                                out=None, lse=None, stream=None):
    """One rank of the llama3 form: q (L, h, d) or (h, L, d), the rank's contiguous slice of the
    packed buffer (L = total / n_shards); k, v: all total rows.  Returns (out like q, lse (h, L))."""
    lib = load()
    host, dev = _cu_pair(cu_seqlens, q.device)
    n = host.numel() - 1
    total = int(host[-1])
    if max_seqlen is None:
        max_seqlen = _max_len(cu_seqlens, host)
    L = total // int(n_shards)
    h, d = _heads_of(q, L), q.shape[2]
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((h, L), dtype=torch.float32, device=q.device) if lse is None else lse
    t = [_t(x) for x in (q, k, v, out, lse)]
    _check(lib.ring_attn_llama3_varlen_fwd(ctypes.byref(t[0]), ctypes.byref(t[1]), ctypes.byref(t[2]),
                                           ctypes.c_void_p(dev.data_ptr()), ctypes.c_void_p(host.data_ptr()), n,
                                           int(max_seqlen), int(rank), int(n_shards), int(bool(causal)),
                                           _scale(softmax_scale, d), ctypes.byref(t[3]), ctypes.byref(t[4]),
                                           _stream(stream)), "ring_attn_llama3_varlen_fwd")
    return out, lse


def ring_attn_llama3_varlen_bwd(dout, q, k, v, out, lse, cu_seqlens, rank, n_shards, causal=True, softmax_scale=None,
                                max_seqlen=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradient of one rank of the llama3 form: (dq of the rank's rows, the rank's contributions to dk, dv)."""
    lib = load()
    host, dev = _cu_pair(cu_seqlens, q.device)
    n = host.numel() - 1
    total = int(host[-1])
    if max_seqlen is None:
        max_seqlen = _max_len(cu_seqlens, host)
    L = total // int(n_shards)
    h, d = _heads_of(q, L), q.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    ws_bytes = ring_attn_workspace_size(RA_OP_BWD, 1, h, L, d, 1)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=q.device)
    ts = [_t(x) for x in (dout, q, k, v, out, lse, dq, dk, dv)]
    r = [ctypes.byref(x) for x in ts]
    _check(lib.ring_attn_llama3_varlen_bwd(r[0], r[1], r[2], r[3], r[4], r[5], ctypes.c_void_p(dev.data_ptr()),
                                           ctypes.c_void_p(host.data_ptr()), n, int(max_seqlen), int(rank),
                                           int(n_shards), int(bool(causal)), _scale(softmax_scale, d), r[6], r[7],
                                           r[8], ctypes.c_void_p(workspace.data_ptr()),
                                           workspace.numel() * workspace.element_size(), _stream(stream)),
           "ring_attn_llama3_varlen_bwd")
    return dq, dk, dv


# ---------------------------------------------------------------------------- packed forms
# The "kvpacked" / "qkvpacked" entry points of the "Ring Flash Attention" README
# (API list) take k and v, or q, k and v, stacked in one tensor.  They are
# strided views over the calls above: the kernels read the packed tensors in
# place through their strides, and the gradients are written into one packed
# tensor the same way.  Batched forms use the flash-attention packing
# (b, s, 3 or 2, h, d) with out and dout as (b, s, h, d); varlen forms use
# (total, 3 or 2, h, d) with out and dout as (total, h, d).  The sequence axis
# is in layout order, as everywhere in this library.

def _bshd(x):
    """(b, s, h, d) -> the (b, h, s, d) view the calls take."""
    return x.transpose(1, 2)


def ring_attn_qkvpacked_fwd(qkv, layout="contiguous", n_shards=1, causal=False, softmax_scale=None, out=None,
                            lse=None, stream=None):
    """qkv: (b, s, 3, h, d) bf16.  Returns (out (b, s, h, d) bf16, lse (b, h, s) fp32)."""
    b, s, three, h, d = qkv.shape
    if three != 3:
        raise ValueError("qkv must be (b, s, 3, h, d)")
    out = torch.empty((b, s, h, d), dtype=qkv.dtype, device=qkv.device) if out is None else out
    _, lse = ring_attn_fwd(_bshd(qkv[:, :, 0]), _bshd(qkv[:, :, 1]), _bshd(qkv[:, :, 2]), layout, n_shards, causal,
                           softmax_scale, out=_bshd(out), lse=lse, stream=stream)
    return out, lse


def ring_attn_qkvpacked_bwd(dout, qkv, out, lse, layout="contiguous", n_shards=1, causal=False, softmax_scale=None,
                            dqkv=None, workspace=None, stream=None):
    """Gradient of ring_attn_qkvpacked_fwd: dqkv (b, s, 3, h, d) bf16."""
    dqkv = torch.empty_like(qkv) if dqkv is None else dqkv
    ring_attn_bwd(_bshd(dout), _bshd(qkv[:, :, 0]), _bshd(qkv[:, :, 1]), _bshd(qkv[:, :, 2]), _bshd(out), lse,
                  layout, n_shards, causal, softmax_scale, dq=_bshd(dqkv[:, :, 0]), dk=_bshd(dqkv[:, :, 1]),
                  dv=_bshd(dqkv[:, :, 2]), workspace=workspace, stream=stream)
    return dqkv


def ring_attn_kvpacked_fwd(q, kv, layout="contiguous", n_shards=1, causal=False, softmax_scale=None, out=None,
                           lse=None, stream=None):
    """q: (b, s, h, d), kv: (b, s, 2, h, d) bf16.  Returns (out (b, s, h, d), lse (b, h, s))."""
    if kv.dim() != 5 or kv.shape[2] != 2:
        raise ValueError("kv must be (b, s, 2, h, d)")
    out = torch.empty_like(q) if out is None else out
    _, lse = ring_attn_fwd(_bshd(q), _bshd(kv[:, :, 0]), _bshd(kv[:, :, 1]), layout, n_shards, causal,
                           softmax_scale, out=_bshd(out), lse=lse, stream=stream)
    return out, lse


def ring_attn_kvpacked_bwd(dout, q, kv, out, lse, layout="contiguous", n_shards=1, causal=False, softmax_scale=None,
                           dq=None, dkv=None, workspace=None, stream=None):
    """Gradient of ring_attn_kvpacked_fwd: (dq (b, s, h, d), dkv (b, s, 2, h, d))."""
    dq = torch.empty_like(q) if dq is None else dq
    dkv = torch.empty_like(kv) if dkv is None else dkv
    ring_attn_bwd(_bshd(dout), _bshd(q), _bshd(kv[:, :, 0]), _bshd(kv[:, :, 1]), _bshd(out), lse, layout, n_shards,
                  causal, softmax_scale, dq=_bshd(dq), dk=_bshd(dkv[:, :, 0]), dv=_bshd(dkv[:, :, 1]),
                  workspace=workspace, stream=stream)
    return dq, dkv


def ring_attn_varlen_qkvpacked_fwd(qkv, cu_seqlens, max_seqlen=None, n_shards=1, causal=True, softmax_scale=None,
                                   out=None, lse=None, stream=None, layout="contiguous"):
    """qkv: (total, 3, h, d) bf16.  Returns (out (total, h, d), lse (h, total))."""
    if qkv.dim() != 4 or qkv.shape[1] != 3:
        raise ValueError("qkv must be (total, 3, h, d)")
    out = torch.empty_like(qkv[:, 0]) if out is None else out
    return ring_attn_varlen_fwd(qkv[:, 0], qkv[:, 1], qkv[:, 2], cu_seqlens, max_seqlen, n_shards, causal,
                                softmax_scale, out=out, lse=lse, stream=stream, layout=layout)


def ring_attn_varlen_qkvpacked_bwd(dout, qkv, out, lse, cu_seqlens, max_seqlen=None, n_shards=1, causal=True,
                                   softmax_scale=None, dqkv=None, workspace=None, stream=None, layout="contiguous"):
    """Gradient of ring_attn_varlen_qkvpacked_fwd: dqkv (total, 3, h, d)."""
    dqkv = torch.empty_like(qkv) if dqkv is None else dqkv
    ring_attn_varlen_bwd(dout, qkv[:, 0], qkv[:, 1], qkv[:, 2], out, lse, cu_seqlens, max_seqlen, n_shards, causal,
                         softmax_scale, dq=dqkv[:, 0], dk=dqkv[:, 1], dv=dqkv[:, 2], workspace=workspace,
                         stream=stream, layout=layout)
    return dqkv


def ring_attn_varlen_kvpacked_fwd(q, kv, cu_seqlens, max_seqlen=None, n_shards=1, causal=True, softmax_scale=None,
                                  out=None, lse=None, stream=None, layout="contiguous"):
    """q: (total, h, d), kv: (total, 2, h, d).  Returns (out (total, h, d), lse (h, total))."""
    if kv.dim() != 4 or kv.shape[1] != 2:
        raise ValueError("kv must be (total, 2, h, d)")
    return ring_attn_varlen_fwd(q, kv[:, 0], kv[:, 1], cu_seqlens, max_seqlen, n_shards, causal, softmax_scale,
                                out=out, lse=lse, stream=stream, layout=layout)


def ring_attn_varlen_kvpacked_bwd(dout, q, kv, out, lse, cu_seqlens, max_seqlen=None, n_shards=1, causal=True,
                                  softmax_scale=None, dq=None, dkv=None, workspace=None, stream=None,
                                  layout="contiguous"):
    """Gradient of ring_attn_varlen_kvpacked_fwd: (dq (total, h, d), dkv (total, 2, h, d))."""
    dq = torch.empty_like(q) if dq is None else dq
    dkv = torch.empty_like(kv) if dkv is None else dkv
    ring_attn_varlen_bwd(dout, q, kv[:, 0], kv[:, 1], out, lse, cu_seqlens, max_seqlen, n_shards, causal,
                         softmax_scale, dq=dq, dk=dkv[:, 0], dv=dkv[:, 1], workspace=workspace, stream=stream,
                         layout=layout)
    return dq, dkv


def ring_attn_varlen_permute(x, cu_seqlens, layout, n_shards, seq_dim=0, out=None, stream=None):
    """Packed original order -> layout order along seq_dim for one cu_seqlens (bit copy)."""
    lib = load()
    host, dev = _cu_pair(cu_seqlens, x.device)
    out = torch.empty_like(x) if out is None else out
    a, b_ = _t(x), _t(out)
    _check(lib.ring_attn_varlen_permute(ctypes.byref(a), ctypes.byref(b_), ctypes.c_void_p(dev.data_ptr()),
                                        ctypes.c_void_p(host.data_ptr()), host.numel() - 1, _layout(layout),
                                        int(n_shards), int(seq_dim), _stream(stream)), "ring_attn_varlen_permute")
    return out


def ring_attn_varlen_unpermute(y, cu_seqlens, layout, n_shards, seq_dim=0, out=None, stream=None):
    """Layout order -> packed original order along seq_dim (bit copy)."""
    lib = load()
    host, dev = _cu_pair(cu_seqlens, y.device)
    out = torch.empty_like(y) if out is None else out
    a, b_ = _t(y), _t(out)
    _check(lib.ring_attn_varlen_unpermute(ctypes.byref(a), ctypes.byref(b_), ctypes.c_void_p(dev.data_ptr()),
                                          ctypes.c_void_p(host.data_ptr()), host.numel() - 1, _layout(layout),
                                          int(n_shards), int(seq_dim), _stream(stream)), "ring_attn_varlen_unpermute")
    return out


def ring_attn_permute(x, layout, n_shards, seq_dim=2, out=None, stream=None):
    """Original token order -> layout order along seq_dim (bit copy)."""
    lib = load()
    out = torch.empty_like(x) if out is None else out
    a, b_ = _t(x), _t(out)
    _check(lib.ring_attn_permute(ctypes.byref(a), ctypes.byref(b_), _layout(layout), int(n_shards), int(seq_dim),
                                 _stream(stream)), "ring_attn_permute")
    return out


def ring_attn_unpermute(y, layout, n_shards, seq_dim=2, out=None, stream=None):
    """Layout order -> original token order along seq_dim (bit copy)."""
    lib = load()
    out = torch.empty_like(y) if out is None else out
    a, b_ = _t(y), _t(out)
    _check(lib.ring_attn_unpermute(ctypes.byref(a), ctypes.byref(b_), _layout(layout), int(n_shards),
                                   int(seq_dim), _stream(stream)), "ring_attn_unpermute")
    return out


def ring_attn_check_device_error(stream=None):
    """Synchronises the stream and returns (status, info); status 0 = no device-side error."""
    info = ctypes.c_int32(0)
    st = load().ring_attn_check_device_error(_stream(stream), ctypes.byref(info))
    return int(st), int(info.value)


def ring_attn_set_knob(knob: int, value: int):
    _check(load().ring_attn_set_knob(int(knob), int(value)), "ring_attn_set_knob")


def ring_attn_timing_enable(on: bool = True):
    """Bracket every library kernel launch with CUDA events (see ring_attn_timing_read)."""
    _check(load().ring_attn_timing_enable(int(bool(on))), "ring_attn_timing_enable")


def ring_attn_timing_read(kernel) -> tuple:
    """(total device ms, launches) of one kernel kind since the last read; resets it."""
    k = KERNELS[kernel] if isinstance(kernel, str) else int(kernel)
    ms = ctypes.c_double(0.0)
    n = ctypes.c_int64(0)
    _check(load().ring_attn_timing_read(k, ctypes.byref(ms), ctypes.byref(n)), "ring_attn_timing_read")
    return float(ms.value), int(n.value)


def ring_attn_version() -> int:
    return int(load().ring_attn_version())
