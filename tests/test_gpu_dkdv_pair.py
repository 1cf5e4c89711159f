"""The dK / dV pass at head_dim 128 can run on CTA pairs (two SMs share each
M = 256 MMA; RA_KNOB_DKDV_PAIR = 1; the default is the one-CTA kernel).  These
cases check the pair kernel against the fp64 oracle and against the one-CTA
kernel (knob 0) on the same inputs, at the shapes where the pair's bookkeeping differs from one key tile per CTA: an
odd number of key tiles per shard (the odd CTA of the last pair lies past the
shard end), a ragged last tile, one tile per shard, shards whose two tiles meet
different query ranges, varlen sequences that straddle the pair's tiles, and one
llama3 rank."""
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
    ring_attn_gb300.ring_attn_set_knob(ring_attn_gb300.RA_KNOB_DKDV_PAIR, 0)


def _both(ra, fn):
    """fn() with the pair kernel, then with the one-CTA kernel."""
    ra.ring_attn_set_knob(ra.RA_KNOB_DKDV_PAIR, 1)
    try:
        a = fn()
    finally:
        ra.ring_attn_set_knob(ra.RA_KNOB_DKDV_PAIR, 0)
    b = fn()
    torch.cuda.synchronize()
    check_no_device_error(ra)
    return a, b


def _same_as_one_cta(name, pair, one):
    # the same products summed in the same order per SM: any difference is at most
    # the last bf16 rounding of the output
    d = (pair.float() - one.float()).abs()
    tol = 2.0 ** -7 * one.float().abs() + 1e-6
    assert bool((d <= tol).all()), f"{name}: pair and one-CTA kernels differ by {float(d.max()):.3e}"


@pytest.mark.parametrize("s,n,layout,causal", [
    (128, 1, "contiguous", True),    # one key tile: the pair's odd CTA has no keys
    (384, 1, "contiguous", False),   # three tiles: the last pair is half empty
    (384, 3, "stripe", True),        # one tile per shard
    (1000, 2, "zigzag", True),       # ragged last tile (500 keys per shard)
    (1000, 4, "contiguous", True),
    (2048, 4, "zigzag", True),       # four tiles per shard: both pairs full
    (2304, 3, "stripe", False),      # six tiles per shard
    (2560, 4, "contiguous", True),   # five tiles per shard (odd)
])
def test_pair_matches_oracle_and_one_cta(ra, s, n, layout, causal):
    b, h, d = 1, 2, 128
    x = make_qkv(b, h, s, d, 3000 + s + n, with_do=True)
    scale = d ** -0.5
    g = {k: to_layout(ra, v.cuda(), layout, n) for k, v in x.items()}
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, causal, scale)

    def run():
        return ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, causal, scale)

    pair, one = _both(ra, run)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal)
    for name, gp, go, r in zip(("dq", "dk", "dv"), pair, one, ref):
        _same_as_one_cta(name, gp, go)
        assert_close(name, to_original(ra, gp, layout, n).cpu(), r)


@pytest.mark.parametrize("layout,lens,n", [
    ("contiguous", [100, 300, 1, 350, 273], 4),       # sequences straddle the pair's two tiles
    ("contiguous", [1024], 2),
    ("zigzag", [256, 640, 96, 1056], 4),
])
@pytest.mark.parametrize("causal", [False, True])
def test_pair_varlen(ra, layout, lens, n, causal):
    h, d = 2, 128
    cu = cu_seqlens(lens)
    x = make_qkv(1, h, int(cu[-1]), d, 3100 + len(lens), with_do=True)
    scale = d ** -0.5
    g = {k: ra.ring_attn_varlen_permute(v[0].transpose(0, 1).contiguous().cuda(), cu, layout, n, seq_dim=0)
         for k, v in x.items()}
    out, lse = ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cu, None, n, causal, scale, layout=layout)

    def run():
        return ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, cu, None, n, causal, scale,
                                       layout=layout)

    pair, one = _both(ra, run)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal, cu_seqlens=cu)

    def back(t):
        return ra.ring_attn_varlen_unpermute(t.contiguous(), cu, layout, n, seq_dim=0).cpu()

    for name, gp, go, r in zip(("dq", "dk", "dv"), pair, one, ref):
        _same_as_one_cta(name, gp, go)
        assert_close(name, back(gp).transpose(0, 1).unsqueeze(0), r)


def test_pair_llama3_rank(ra):
    """Rank 1 holds the first key of the second sequence (token 300), where a
    causal dV collects its queries' dO at weights 1, 1/2, 1/3, ... and reaches
    |4-5|: dO is halved, the tolerance reading that
    tests/test_tolerance_readings.py supports."""
    lens, n, r, h, d = [300, 500, 224], 4, 1, 2, 128
    cu = cu_seqlens(lens)
    total = int(cu[-1])
    L = total // n
    x = make_qkv(1, h, total, d, 3200, with_do=True)
    x["do"] = (x["do"].float() * 0.5).to(torch.bfloat16)
    scale = d ** -0.5
    g = {k: v[0].transpose(0, 1).contiguous().cuda() for k, v in x.items()}
    rows = slice(r * L, (r + 1) * L)
    q_loc, do_loc = g["q"][rows].contiguous(), g["do"][rows].contiguous()
    out, lse = ra.ring_attn_llama3_varlen_fwd(q_loc, g["k"], g["v"], cu, r, n, True, scale)

    def run():
        return ra.ring_attn_llama3_varlen_bwd(do_loc, q_loc, g["k"], g["v"], out, lse, cu, r, n, True, scale)

    pair, one = _both(ra, run)
    want = oracle.llama3_rank_attention(x["q"], x["k"], x["v"], r, n, scale, True, cu_seqlens=cu,
                                        do=x["do"][:, :, rows])
    for name, gp, go, w in zip(("dq", "dk", "dv"), pair, one, want[2:]):
        _same_as_one_cta(name, gp, go)
        assert_close(name, gp.transpose(0, 1).unsqueeze(0).cpu(), w)


def test_pair_full_size_key_tiles_match_one_cta(ra):
    """The benchmark workload's shape (b1 h32 s65536 d128, zigzag over 8 shards),
    two heads: every dK / dV row of the pair kernel against the one-CTA kernel."""
    b, h, s, d, n, layout = 1, 2, 65536, 128, 8, "zigzag"
    x = make_qkv(b, h, s, d, 3300, with_do=True, device="cuda")
    g = {k: ra.ring_attn_permute(v, layout, n) for k, v in x.items()}
    del x
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, True, d ** -0.5)

    def run():
        return ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, True, d ** -0.5)

    pair, one = _both(ra, run)
    for name, gp, go in zip(("dq", "dk", "dv"), pair, one):
        assert bool(torch.isfinite(gp.float()).all()), name
        _same_as_one_cta(name, gp, go)
    assert torch.equal(pair[0], one[0]), "dq comes from the same deterministic kernel in both runs"
