"""The backward's dQ pass runs as a persistent kernel by default
(RA_KNOB_PERSISTENT = 1): a CTA takes over the query tiles of CTAs that have
not started yet (cluster launch control) and overlaps each tile's set-up with
the previous tile.  It performs the same MMAs in the same order per query tile
as the one-tile-per-CTA kernel (knob 0), so dq must match it bit for bit; both
are also checked against the fp64 oracle on small cases.  The cases cover
grids far larger and far smaller than the number of SMs, query tiles without
key tiles, varlen sequences of every length class and a llama3 rank."""
import pytest
import torch

import oracle
from tests.helpers import assert_close, check_no_device_error, to_layout, to_original
from workload import cu_seqlens, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attn_gb300
    from ring_attn_gb300.build import build

    build()
    ring_attn_gb300.load()
    yield ring_attn_gb300
    ring_attn_gb300.ring_attn_set_knob(ring_attn_gb300.RA_KNOB_PERSISTENT, 1)


def _both(ra, fn):
    """fn() with the persistent dQ kernel, then with one query tile per CTA."""
    ra.ring_attn_set_knob(ra.RA_KNOB_PERSISTENT, 1)
    a = fn()
    torch.cuda.synchronize()
    ra.ring_attn_set_knob(ra.RA_KNOB_PERSISTENT, 0)
    try:
        b = fn()
        torch.cuda.synchronize()
    finally:
        ra.ring_attn_set_knob(ra.RA_KNOB_PERSISTENT, 1)
    check_no_device_error(ra)
    return a, b


@pytest.mark.parametrize("b,h,s,d,n,layout,causal", [
    (1, 1, 128, 64, 1, "contiguous", True),     # one query tile, one CTA
    (1, 2, 1000, 128, 2, "zigzag", True),
    (2, 3, 1000, 64, 4, "contiguous", False),
    (1, 4, 2304, 128, 3, "stripe", True),
    (1, 8, 4096, 128, 8, "zigzag", True),       # 256 query tiles: more CTAs than SMs
])
def test_persistent_dq_matches(ra, b, h, s, d, n, layout, causal):
    x = make_qkv(b, h, s, d, 5000 + s + n, with_do=True)
    scale = d ** -0.5
    g = {k: to_layout(ra, v.cuda(), layout, n) for k, v in x.items()}
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, causal, scale)

    def run():
        return ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, causal, scale)

    pers, one = _both(ra, run)
    for name, a, c in zip(("dq", "dk", "dv"), pers, one):
        assert torch.equal(a, c), f"{name}: persistent and one-tile kernels differ"
    if b * h * s <= 8 * 4096:
        ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal)
        assert_close("dq", to_original(ra, pers[0], layout, n).cpu(), ref[0])


@pytest.mark.parametrize("layout,lens,n", [
    ("contiguous", [100, 300, 1, 350, 273, 0, 1024], 4),
    ("contiguous", [1] * 40 + [88], 4),              # query tiles full of one-token sequences
    ("zigzag", [256, 640, 96, 1056], 4),
])
@pytest.mark.parametrize("causal", [False, True])
def test_persistent_dq_varlen(ra, layout, lens, n, causal):
    h, d = 2, 128
    cu = cu_seqlens(lens)
    x = make_qkv(1, h, int(cu[-1]), d, 5100 + len(lens), with_do=True)
    scale = d ** -0.5
    g = {k: ra.ring_attn_varlen_permute(v[0].transpose(0, 1).contiguous().cuda(), cu, layout, n, seq_dim=0)
         for k, v in x.items()}
    out, lse = ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cu, None, n, causal, scale, layout=layout)

    def run():
        return ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, cu, None, n, causal, scale,
                                       layout=layout)

    pers, one = _both(ra, run)
    for name, a, c in zip(("dq", "dk", "dv"), pers, one):
        assert torch.equal(a, c), f"{name}: persistent and one-tile kernels differ"
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal, cu_seqlens=cu)
    got = ra.ring_attn_varlen_unpermute(pers[0].contiguous(), cu, layout, n, seq_dim=0).cpu()
    assert_close("dq", got.transpose(0, 1).unsqueeze(0), ref[0])


def test_persistent_dq_llama3_rank(ra):
    lens, n, r, h, d = [300, 500, 224], 4, 2, 2, 64
    cu = cu_seqlens(lens)
    total = int(cu[-1])
    L = total // n
    x = make_qkv(1, h, total, d, 5200, with_do=True)
    g = {k: v[0].transpose(0, 1).contiguous().cuda() for k, v in x.items()}
    rows = slice(r * L, (r + 1) * L)
    q_loc, do_loc = g["q"][rows].contiguous(), g["do"][rows].contiguous()
    out, lse = ra.ring_attn_llama3_varlen_fwd(q_loc, g["k"], g["v"], cu, r, n, True, d ** -0.5)

    def run():
        return ra.ring_attn_llama3_varlen_bwd(do_loc, q_loc, g["k"], g["v"], out, lse, cu, r, n, True, d ** -0.5)

    pers, one = _both(ra, run)
    for name, a, c in zip(("dq", "dk", "dv"), pers, one):
        assert torch.equal(a, c), f"{name}: persistent and one-tile kernels differ"


def test_persistent_dq_benchmark_shape(ra):
    """b1 h32 s65536 d128, zigzag over 8 shards (16,384 query tiles on 152 SMs)."""
    b, h, s, d, n, layout = 1, 32, 65536, 128, 8, "zigzag"
    x = make_qkv(b, h, s, d, 5300, with_do=True, device="cuda")
    g = {k: ra.ring_attn_permute(v, layout, n) for k, v in x.items()}
    del x
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, True, d ** -0.5)

    def run():
        return ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, True, d ** -0.5)[0]

    pers, one = _both(ra, run)
    assert torch.equal(pers, one), "dq: persistent and one-tile kernels differ"
