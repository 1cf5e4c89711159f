"""Grouped-query attention: k and v (and dk, dv) with hk heads, q with h = G * hk,
query head i attending with key / value head i // G.  The pages only use
hk = h; the grouping follows the common convention (the same one as torch's
scaled_dot_product_attention with enable_gqa), which the oracle's own pins
check.  These cases compare the kernels with the fp64 oracle on every path
that takes k and v (batched layouts, one ring step + lse_merge, varlen in both
layouts, one llama3 rank, the static-scratch backward), and at the benchmark
workload's size with properties that hold at any size: the forward and dQ
equal, bit for bit, the same kernels run on k and v with every head repeated
G times, and dK / dV equal the sum over the group of the repeated run's
per-head gradients up to bf16 rounding."""
import pytest
import torch

import oracle
from tests.helpers import assert_close, assert_lse_close, check_no_device_error, lse_to_original, to_layout, to_original
from workload import cu_seqlens, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attn_gb300
    from ring_attn_gb300.build import build

    build()
    ring_attn_gb300.load()
    return ring_attn_gb300


def _gqa_inputs(b, h, hk, s, d, seed):
    """q, dO with h heads, k, v with hk heads (seeded, original order).

    dV of a key / value head sums the contributions of its G = h / hk query
    heads, so with unit dO its spread grows as sqrt(G); dO is scaled by
    1 / sqrt(G) (then rounded to bf16, the value both sides take) so that dV
    has the spread of plain multi-head attention with unit dO, which the 2e-2
    bound is stated for."""
    x = make_qkv(b, h, s, d, seed, with_do=True)
    y = make_qkv(b, hk, s, d, seed + 1, with_do=False)
    do = (x["do"].float() * (hk / h) ** 0.5).to(torch.bfloat16)
    return {"q": x["q"], "do": do, "k": y["k"], "v": y["v"]}


@pytest.mark.parametrize("b,h,hk,s,d,layout,n,causal", [
    (1, 4, 2, 1024, 128, "zigzag", 4, True),
    (1, 4, 1, 1000, 64, "contiguous", 2, True),     # one key / value head for all (multi-query)
    (2, 6, 2, 768, 128, "stripe", 3, False),        # G = 3, two batches
    (1, 8, 2, 520, 64, "zigzag", 2, True),          # ragged last tile (260 rows per shard)
    (1, 2, 1, 300, 128, "contiguous", 1, False),
])
def test_gqa_batched_fwd_bwd(ra, b, h, hk, s, d, layout, n, causal):
    x = _gqa_inputs(b, h, hk, s, d, 4000 + s + h)
    scale = d ** -0.5
    g = {k: to_layout(ra, v.cuda(), layout, n) for k, v in x.items()}
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, causal, scale)
    dq, dk, dv = ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, causal, scale)
    torch.cuda.synchronize()
    check_no_device_error(ra)
    assert dk.shape == x["k"].shape and dv.shape == x["v"].shape
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal)
    assert_close("out", to_original(ra, out, layout, n).cpu(), ro)
    assert_lse_close("lse", lse_to_original(ra, lse, layout, n).cpu(), rl)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(name, to_original(ra, got, layout, n).cpu(), r)


def test_gqa_ring_steps_and_merge(ra):
    """Every ring step on its own with grouped heads, merged with lse_merge."""
    b, h, hk, s, d, layout, n = 1, 4, 2, 1024, 64, "zigzag", 4
    x = _gqa_inputs(b, h, hk, s, d, 4100)
    scale = d ** -0.5
    g = {k: to_layout(ra, v.cuda(), layout, n) for k, v in x.items() if k != "do"}
    acc = torch.zeros((b, h, s, d), dtype=torch.float32, device="cuda")
    lacc = torch.full((b, h, s), float("-inf"), dtype=torch.float32, device="cuda")
    for step in range(n):
        ob, lb = ra.ring_attn_fwd_step(g["q"], g["k"], g["v"], step, layout, n, True, scale)
        ra.lse_merge(acc, lacc, ob, lb)
    torch.cuda.synchronize()
    check_no_device_error(ra)
    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, True)
    assert_close("out", to_original(ra, acc, layout, n).cpu(), ro)
    assert_lse_close("lse", lse_to_original(ra, lacc, layout, n).cpu(), rl)


@pytest.mark.parametrize("layout,lens,n,ws", [
    ("contiguous", [100, 300, 1, 350, 273], 4, False),
    ("zigzag", [256, 640, 96, 1056], 4, True),     # original-order copies in the workspace
    ("zigzag", [256, 640, 96, 1056], 4, False),    # zigzag chunks in place
])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_varlen(ra, layout, lens, n, ws, causal):
    h, hk, d = 4, 2, 128
    cu = cu_seqlens(lens)
    total = int(cu[-1])
    x = _gqa_inputs(1, h, hk, total, d, 4200 + len(lens))
    scale = d ** -0.5
    g = {k: ra.ring_attn_varlen_permute(v[0].transpose(0, 1).contiguous().cuda(), cu, layout, n, seq_dim=0)
         for k, v in x.items()}
    kw = {}
    if not ws:
        kw["workspace"] = torch.empty(ra.ring_attn_varlen_workspace_size(ra.RA_OP_FWD, total, h, d, "contiguous", n),
                                      dtype=torch.uint8, device="cuda")
    out, lse = ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cu, None, n, causal, scale, layout=layout, **kw)
    bw = {}
    if not ws:
        bw["workspace"] = torch.empty(ra.ring_attn_varlen_workspace_size(ra.RA_OP_BWD, total, h, d, "contiguous", n),
                                      dtype=torch.uint8, device="cuda")
    dq, dk, dv = ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, cu, None, n, causal, scale,
                                         layout=layout, **bw)
    torch.cuda.synchronize()
    check_no_device_error(ra)

    def back(t):
        return ra.ring_attn_varlen_unpermute(t.contiguous(), cu, layout, n, seq_dim=0).cpu()

    ro, rl = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, cu_seqlens=cu)
    assert_close("out", back(out).transpose(0, 1).unsqueeze(0), ro)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal, cu_seqlens=cu)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(name, back(got).transpose(0, 1).unsqueeze(0), r)


def test_gqa_llama3_rank(ra):
    lens, n, r, h, hk, d = [300, 500, 224], 4, 1, 4, 2, 64
    cu = cu_seqlens(lens)
    total = int(cu[-1])
    L = total // n
    x = _gqa_inputs(1, h, hk, total, d, 4300)
    scale = d ** -0.5
    g = {k: v[0].transpose(0, 1).contiguous().cuda() for k, v in x.items()}
    rows = slice(r * L, (r + 1) * L)
    q_loc, do_loc = g["q"][rows].contiguous(), g["do"][rows].contiguous()
    out, lse = ra.ring_attn_llama3_varlen_fwd(q_loc, g["k"], g["v"], cu, r, n, True, scale)
    dq, dk, dv = ra.ring_attn_llama3_varlen_bwd(do_loc, q_loc, g["k"], g["v"], out, lse, cu, r, n, True, scale)
    torch.cuda.synchronize()
    check_no_device_error(ra)
    want = oracle.llama3_rank_attention(x["q"], x["k"], x["v"], r, n, scale, True, cu_seqlens=cu,
                                        do=x["do"][:, :, rows])
    assert_close("out", out.transpose(0, 1).unsqueeze(0).cpu(), want[0])
    for name, got, w in zip(("dq", "dk", "dv"), (dq, dk, dv), want[2:]):
        assert_close(name, got.transpose(0, 1).unsqueeze(0).cpu(), w)


def test_gqa_static_scratch_and_pair_knob_match(ra):
    """The static-scratch backward gives the workspace backward's bits; with the
    CTA-pair knob on, grouped heads still take the one-CTA dK / dV kernel."""
    b, h, hk, s, d, layout, n = 1, 4, 2, 2048, 128, "zigzag", 4
    x = _gqa_inputs(b, h, hk, s, d, 4400)
    scale = d ** -0.5
    g = {k: to_layout(ra, v.cuda(), layout, n) for k, v in x.items()}
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, True, scale)
    want = ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, True, scale)
    got = ra.ring_attn_bwd_static_scratch(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, True, scale)
    ra.ring_attn_set_knob(ra.RA_KNOB_DKDV_PAIR, 1)
    try:
        pair = ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, True, scale)
    finally:
        ra.ring_attn_set_knob(ra.RA_KNOB_DKDV_PAIR, 0)
    torch.cuda.synchronize()
    check_no_device_error(ra)
    for name, w, a, p in zip(("dq", "dk", "dv"), want, got, pair):
        assert torch.equal(w, a), f"{name}: static scratch differs"
        assert torch.equal(w, p), f"{name}: pair knob changed a grouped-head result"


def test_gqa_full_size_matches_repeated_heads(ra):
    """The benchmark workload's sequence (s65536 d128, zigzag over 8 shards,
    causal) with h = 32 query heads over hk = 8 key / value heads, against the
    same kernels on k, v with every head repeated 4 times."""
    b, h, hk, s, d, layout, n = 1, 32, 8, 65536, 128, "zigzag", 8
    G = h // hk
    x = make_qkv(b, h, s, d, 4500, with_do=True, device="cuda")
    y = make_qkv(b, hk, s, d, 4501, with_do=False, device="cuda")
    q, do = ra.ring_attn_permute(x["q"], layout, n), ra.ring_attn_permute(x["do"], layout, n)
    k, v = ra.ring_attn_permute(y["k"], layout, n), ra.ring_attn_permute(y["v"], layout, n)
    del x, y
    scale = d ** -0.5
    out, lse = ra.ring_attn_fwd(q, k, v, layout, n, True, scale)
    dq, dk, dv = ra.ring_attn_bwd(do, q, k, v, out, lse, layout, n, True, scale)
    kr, vr = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
    out_r, lse_r = ra.ring_attn_fwd(q, kr, vr, layout, n, True, scale)
    assert torch.equal(out, out_r) and torch.equal(lse, lse_r), "forward differs from the repeated-head run"
    dq_r, dk_r, dv_r = ra.ring_attn_bwd(do, q, kr, vr, out_r, lse_r, layout, n, True, scale)
    torch.cuda.synchronize()
    check_no_device_error(ra)
    assert torch.equal(dq, dq_r), "dq differs from the repeated-head run"
    for name, got, rep in (("dk", dk, dk_r), ("dv", dv, dv_r)):
        parts = rep.float().view(b, hk, G, s, d)
        want = parts.sum(dim=2)
        # the grouped kernel rounds the fp32 sum once; the repeated run rounds each
        # head's gradient to bf16 before the sum
        tol = 2.0 ** -8 * (parts.abs().sum(dim=2) + want.abs()) + 1e-6
        err = (got.float() - want).abs()
        assert bool((err <= tol).all()), f"{name}: max excess {float((err - tol).max()):.3e}"
