"""GPU parity of the ring forward, the per-step forward + LSE merge, the
backward and the varlen forms against the fp64 oracle, element by element, on
sizes that span several 128-token tiles and ragged tails."""
import os

import numpy as np
import pytest
import torch

import oracle
from tests.helpers import (TOL_MAX_ABS, assert_close, assert_lse_close, check_no_device_error, f64, lse_to_original, to_layout,
                           to_original)
from workload import cu_seqlens, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attn_gb300
    from ring_attn_gb300.build import build

    build()
    ring_attn_gb300.load()
    return ring_attn_gb300


def _fwd_cases():
    cases = []
    for s in (1, 63, 64, 65, 127, 128, 129, 256, 1000):
        for n in (1, 2, 3, 4, 8):
            for layout in oracle.LAYOUTS:
                if s % n or (layout == "zigzag" and s % (2 * n)):
                    continue
                if n == 1 and layout != "contiguous":
                    continue
                for causal in (False, True):
                    cases.append((s, n, layout, causal))
    return cases


def _run_fwd(ra, b, h, s, d, n, layout, causal, seed):
    x = make_qkv(b, h, s, d, seed, with_do=False)
    scale = d ** -0.5
    g = {k: to_layout(ra, v.cuda(), layout, n) for k, v in x.items()}
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, causal, scale)
    check_no_device_error(ra)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal)
    assert_close("out", to_original(ra, out, layout, n).cpu(), ref_o)
    assert_lse_close("lse", lse_to_original(ra, lse, layout, n).cpu(), ref_l)
    return x, g, out, lse


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("s,n,layout,causal", _fwd_cases())
def test_fwd_parity_sweep(ra, d, s, n, layout, causal):
    _run_fwd(ra, 1, 2, s, d, n, layout, causal, seed=100 + s + n)


def test_fwd_tiny_noncausal_workload(ra):
    # b1 h2 s256 d64, non-causal, contiguous split into 4 shards of 64 tokens
    _run_fwd(ra, 1, 2, 256, 64, 4, "contiguous", False, seed=1001)


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
def test_fwd_batch_heads_and_multi_tile(ra, layout):
    _run_fwd(ra, 2, 3, 2048, 128, 4, layout, True, seed=7)


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("blk_dtype", [torch.float32, torch.bfloat16])
def test_step_blocks_then_merge(ra, layout, causal, blk_dtype):
    """Each ring step emits (out_blk, lse_blk); merging them with lse_merge in ring
    order equals full attention, and each block equals the oracle's block."""
    b, h, s, d, n = 1, 2, 768, 128, 4
    x = make_qkv(b, h, s, d, 55, with_do=False)
    scale = d ** -0.5
    g = {k: to_layout(ra, v.cuda(), layout, n) for k, v in x.items()}
    L = s // n
    tok = oracle.token_of_position(layout, n, s)
    ql, kl, vl = (oracle.permute(f64(x[k]), layout, n, axis=2) for k in ("q", "k", "v"))
    out_acc = torch.zeros(b, h, s, d, dtype=torch.float32, device="cuda")
    lse_acc = torch.full((b, h, s), -float("inf"), dtype=torch.float32, device="cuda")
    for t in range(n):
        ob, lb = ra.ring_attn_fwd_step(g["q"], g["k"], g["v"], t, layout, n, causal, scale, out_dtype=blk_dtype)
        check_no_device_error(ra)
        # block reference: Q shard r against KV shard (r - t) mod N
        for r in range(n):
            sk = (r - t) % n
            rq, rk = slice(r * L, (r + 1) * L), slice(sk * L, (sk + 1) * L)
            for hi in range(h):
                ro, rl = oracle.block_attention(ql[0, hi, rq], kl[0, hi, rk], vl[0, hi, rk], tok[rq], tok[rk],
                                                scale, causal)
                assert_close(f"out_blk t{t} r{r}", ob[0, hi, rq].cpu(), ro)
                assert_lse_close(f"lse_blk t{t} r{r}", lb[0, hi, rq].cpu(), rl)
        ra.lse_merge(out_acc, lse_acc, ob, lb)
    check_no_device_error(ra)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal)
    assert_close("merged out", to_original(ra, out_acc, layout, n).cpu(), ref_o)
    assert_lse_close("merged lse", lse_to_original(ra, lse_acc, layout, n).cpu(), ref_l)


def _bwd_cases():
    cases = []
    for s in (64, 65, 128, 129, 256, 1000):
        for n in (1, 2, 4, 8):
            for layout in oracle.LAYOUTS:
                if s % n or (layout == "zigzag" and s % (2 * n)):
                    continue
                if n == 1 and layout != "contiguous":
                    continue
                for causal in (False, True):
                    cases.append((s, n, layout, causal))
    return cases


def _run_bwd(ra, b, h, s, d, n, layout, causal, seed):
    x = make_qkv(b, h, s, d, seed, with_do=True)
    scale = d ** -0.5
    g = {k: to_layout(ra, v.cuda(), layout, n) for k, v in x.items()}
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], layout, n, causal, scale)
    dq, dk, dv = ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, layout, n, causal, scale)
    check_no_device_error(ra)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(name, to_original(ra, got, layout, n).cpu(), r)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("s,n,layout,causal", _bwd_cases())
def test_bwd_parity_sweep(ra, d, s, n, layout, causal):
    _run_bwd(ra, 1, 2, s, d, n, layout, causal, seed=300 + s + n)


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
def test_bwd_batch_heads_and_multi_tile(ra, layout):
    _run_bwd(ra, 2, 2, 2048, 128, 4, layout, True, seed=8)


# ----------------------------------------------------------------------------- varlen
def _varlen_case(lens, h, d, n, causal, seed, layout_thd=True):
    total = sum(lens)
    cu = cu_seqlens(lens)
    x = make_qkv(1, h, total, d, seed, with_do=True)
    return cu, x


@pytest.mark.parametrize("lens,n", [
    ([100, 1, 300, 27, 84], 4),          # short sequences, a 1-token one, crossing shard boundaries
    ([1000], 8),                         # one sequence spanning every shard
    ([128, 128, 256, 0, 512], 4),        # tile-aligned, with an empty sequence
    ([5] * 40 + [312], 2),               # many tiny sequences inside one tile
    ([700, 1300, 33, 2000, 15], 8),
])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("packed", ["thd", "htd"])
def test_varlen_fwd_bwd(ra, lens, n, causal, packed):
    h, d = 2, 128
    total = sum(lens)
    if total % n:
        pytest.skip("total not divisible by n_shards")
    cu, x = _varlen_case(lens, h, d, n, causal, seed=len(lens) + total)
    scale = d ** -0.5
    # (1, h, total, d) -> (total, h, d) or (h, total, d)
    if packed == "thd":
        g = {k: v[0].transpose(0, 1).contiguous().cuda() for k, v in x.items()}
    else:
        g = {k: v[0].contiguous().cuda() for k, v in x.items()}
    cu_t = torch.tensor(cu, dtype=torch.int32)
    out, lse = ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cu_t, None, n, causal, scale)
    dq, dk, dv = ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, cu_t, None, n, causal, scale)
    check_no_device_error(ra)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, cu_seqlens=cu)
    ref_g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal, cu_seqlens=cu)

    def back(t):
        t = t.cpu()
        return (t.transpose(0, 1) if packed == "thd" else t).unsqueeze(0)

    assert_close("out", back(out), ref_o)
    assert_lse_close("lse", lse.cpu().unsqueeze(0), ref_l)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref_g):
        assert_close(name, back(got), r)


# ----------------------------------------------------------------------------- zigzag varlen
@pytest.mark.parametrize("lens,n", [
    ([4, 132, 260, 0, 508], 2),
    ([128, 24, 320, 8], 4),
    ([6 * 20, 6 * 7, 6 * 50], 3),
    ([0, 4, 0, 8] * 300, 2),
])
def test_varlen_zigzag_permute_bit_exact(ra, lens, n):
    cu = cu_seqlens(lens)
    total = cu[-1]
    g = oracle.varlen_token_of_position("zigzag", n, cu)
    x16 = make_qkv(1, 3, total, 64, 11, with_do=False)["q"][0].transpose(0, 1).contiguous()  # (total, h, d)
    y = ra.ring_attn_varlen_permute(x16.cuda(), cu, "zigzag", n, seq_dim=0).cpu()
    assert torch.equal(y.view(torch.int16), x16[torch.from_numpy(g)].view(torch.int16))
    back = ra.ring_attn_varlen_unpermute(y.cuda(), cu, "zigzag", n, seq_dim=0).cpu()
    assert torch.equal(back.view(torch.int16), x16.view(torch.int16))
    x32 = torch.randn(2, total, generator=torch.Generator().manual_seed(5))  # (h, total) fp32, seq_dim 1
    y32 = ra.ring_attn_varlen_permute(x32.cuda(), cu, "zigzag", n, seq_dim=1).cpu()
    assert torch.equal(y32, x32[:, torch.from_numpy(g)])
    ident = ra.ring_attn_varlen_permute(x16.cuda(), cu, "contiguous", n, seq_dim=0).cpu()
    assert torch.equal(ident.view(torch.int16), x16.view(torch.int16))


@pytest.mark.parametrize("lens,n", [
    ([4, 132, 260, 0, 508], 2),            # a 4-token sequence, tile-crossing ones, an empty one
    ([128, 24, 320, 8], 4),
    ([16 * 70], 8),                        # one sequence: the batched zigzag split
    ([6 * 20, 6 * 7, 6 * 50, 6 * 1], 3),
    ([8] * 30 + [8 * 64], 4),              # many tiny sequences inside one tile
])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("path", ["original_order", "direct"])
def test_varlen_zigzag_fwd_bwd(ra, lens, n, causal, d, path):
    """Both ways a zigzag varlen call runs: in original token order inside the
    workspace (the binding's default), and on the zigzag order directly (a
    workspace too small for the copies)."""
    h = 2
    cu = cu_seqlens(lens)
    total = int(cu[-1])
    x = make_qkv(1, h, total, d, 300 + len(lens) + n, with_do=True)
    scale = d ** -0.5
    g = {k: ra.ring_attn_varlen_permute(v[0].transpose(0, 1).contiguous().cuda(), cu, "zigzag", n, seq_dim=0)
         for k, v in x.items()}
    if path == "direct":
        ws_f = torch.empty(0, dtype=torch.uint8, device="cuda")
        ws_b = torch.empty(ra.ring_attn_varlen_workspace_size(1, total, h, d, "contiguous", n), dtype=torch.uint8,
                           device="cuda")
    else:
        ws_f = ws_b = None
    out, lse = ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cu, None, n, causal, scale, layout="zigzag",
                                       workspace=ws_f)
    dq, dk, dv = ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, cu, None, n, causal, scale,
                                         layout="zigzag", workspace=ws_b)
    check_no_device_error(ra)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, cu_seqlens=cu)
    ref_g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal, cu_seqlens=cu)

    def back(t, seq_dim=0):
        return ra.ring_attn_varlen_unpermute(t.contiguous(), cu, "zigzag", n, seq_dim=seq_dim).cpu()

    assert_close("out", back(out).transpose(0, 1).unsqueeze(0), ref_o)
    assert_lse_close("lse", back(lse, 1).unsqueeze(0), ref_l)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref_g):
        assert_close(name, back(got).transpose(0, 1).unsqueeze(0), r)


# ----------------------------------------------------------------------------- many sequences
# More than 1024 sequences (three rounds of the warp-wide cu_seqlens search),
# most of them empty or a few tokens long.  dO is halved, a reading of the
# tolerance: with hundreds of short sequences a key near a sequence start collects
# its queries' dO at weights near 1, so |dV| reaches ~5 with unit-variance dO,
# and there the bf16 output rounding plus the bf16 P operand alone use up the
# 2e-2 absolute bound.  tests/test_tolerance_readings.py emulates exactly those
# two roundings on the fp64 oracle: 0.0207 (causal) and 0.0192 with unit dO,
# 0.0104 and 0.0096 with dO halved.
@pytest.mark.parametrize("layout,lens,n", [
    ("contiguous", [0, 2, 0, 0, 1, 3] * 200, 4),
    ("zigzag", [0, 4, 0, 8] * 300, 2),
])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_many_sequences(ra, layout, lens, n, causal):
    h, d = 2, 128
    cu = cu_seqlens(lens)
    x = make_qkv(1, h, cu[-1], d, 4242 + len(lens), with_do=True)
    x["do"] = (x["do"].float() * 0.5).to(torch.bfloat16)
    scale = d ** -0.5
    g = {k: ra.ring_attn_varlen_permute(v[0].transpose(0, 1).contiguous().cuda(), cu, layout, n, seq_dim=0)
         for k, v in x.items()}
    out, lse = ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cu, None, n, causal, scale, layout=layout)
    dq, dk, dv = ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, cu, None, n, causal, scale,
                                         layout=layout)
    check_no_device_error(ra)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, causal, cu_seqlens=cu)
    ref_g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, causal, cu_seqlens=cu)

    def back(t, seq_dim=0):
        return ra.ring_attn_varlen_unpermute(t.contiguous(), cu, layout, n, seq_dim=seq_dim).cpu()

    assert_close("out", back(out).transpose(0, 1).unsqueeze(0), ref_o)
    assert_lse_close("lse", back(lse, 1).unsqueeze(0), ref_l)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref_g):
        assert_close(name, back(got).transpose(0, 1).unsqueeze(0), r)


@pytest.mark.parametrize("n_seqs", [1, 31, 32, 33, 1023, 1024, 1025])
def test_varlen_search_boundaries(ra, n_seqs):
    """cu_seqlens sizes at the warp-wide search's round boundaries (32, 1024
    entries), random lengths of 0-12 tokens (empty sequences first and last
    included), causal contiguous shards; dO halved as in the many-sequence case
    (the tolerance reading that tests/test_tolerance_readings.py supports)."""
    rng = np.random.default_rng(77 + n_seqs)
    lens = [int(x) for x in rng.integers(0, 13, n_seqs)]
    lens[0] = 0
    lens[-1] = 0 if n_seqs > 1 else 16
    lens[n_seqs // 2] += 4 - sum(lens) % 4  # total divisible by the 4 shards
    h, d, n = 1, 64, 4
    cu = cu_seqlens(lens)
    x = make_qkv(1, h, cu[-1], d, 900 + n_seqs, with_do=True)
    x["do"] = (x["do"].float() * 0.5).to(torch.bfloat16)
    scale = d ** -0.5
    g = {k: v[0].transpose(0, 1).contiguous().cuda() for k, v in x.items()}
    out, lse = ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cu, None, n, True, scale)
    dq, dk, dv = ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, cu, None, n, True, scale)
    check_no_device_error(ra)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], scale, True, cu_seqlens=cu)
    ref_g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], scale, True, cu_seqlens=cu)
    back = lambda t: t.cpu().transpose(0, 1).unsqueeze(0)  # noqa: E731
    assert_close("out", back(out), ref_o)
    assert_lse_close("lse", lse.cpu().unsqueeze(0), ref_l)
    for name, got, r in zip(("dq", "dk", "dv"), (dq, dk, dv), ref_g):
        assert_close(name, back(got), r)


# ----------------------------------------------------------------------------- llama3 form
@pytest.mark.parametrize("lens,n", [
    ([100, 1, 300, 27, 84], 4),
    ([700, 1300, 33, 2000, 15], 8),
    ([256, 0, 128], 2),
])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("d", [64, 128])
def test_llama3_varlen_ranks(ra, lens, n, causal, d):
    """Every rank against the fp64 oracle; the ranks' dk / dv contributions sum
    to the full varlen backward of the same inputs."""
    h = 2
    cu = cu_seqlens(lens)
    total = cu[-1]
    if total % n:
        pytest.skip("total not divisible by n_shards")
    L = total // n
    x = make_qkv(1, h, total, d, 500 + len(lens) + n, with_do=True)
    scale = d ** -0.5
    g = {k: v[0].transpose(0, 1).contiguous().cuda() for k, v in x.items()}  # (total, h, d)
    dk_sum = torch.zeros(total, h, d, dtype=torch.float64, device="cuda")
    dv_sum = torch.zeros_like(dk_sum)
    for r in range(n):
        rows = slice(r * L, (r + 1) * L)
        q_loc, do_loc = g["q"][rows].contiguous(), g["do"][rows].contiguous()
        out, lse = ra.ring_attn_llama3_varlen_fwd(q_loc, g["k"], g["v"], cu, r, n, causal, scale)
        dq, dk, dv = ra.ring_attn_llama3_varlen_bwd(do_loc, q_loc, g["k"], g["v"], out, lse, cu, r, n, causal, scale)
        check_no_device_error(ra)
        want = oracle.llama3_rank_attention(x["q"], x["k"], x["v"], r, n, scale, causal, cu_seqlens=cu,
                                            do=x["do"][:, :, rows])
        assert_close(f"out r{r}", out.transpose(0, 1).unsqueeze(0).cpu(), want[0])
        assert_lse_close(f"lse r{r}", lse.unsqueeze(0).cpu(), want[1])
        assert_close(f"dq r{r}", dq.transpose(0, 1).unsqueeze(0).cpu(), want[2])
        assert_close(f"dk r{r}", dk.transpose(0, 1).unsqueeze(0).cpu(), want[3])
        assert_close(f"dv r{r}", dv.transpose(0, 1).unsqueeze(0).cpu(), want[4])
        dk_sum += dk.double()
        dv_sum += dv.double()
    out_f, lse_f = ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cu, None, n, causal, scale)
    _, dk_full, dv_full = ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out_f, lse_f, cu, None, n, causal,
                                                  scale)
    # each of the n contributions was rounded to bf16 (up to half an ulp of its
    # magnitude), so the max-abs bound grows with the number of ranks summed
    bound = TOL_MAX_ABS * (1 + n / 4)
    assert_close("sum dk", dk_sum.cpu(), dk_full.double().cpu(), max_abs=bound)
    assert_close("sum dv", dv_sum.cpu(), dv_full.double().cpu(), max_abs=bound)


# ----------------------------------------------------------------------------- bounded waits
def test_bounded_wait_reports_timeout_and_context_survives(ra):
    """The producer is told to skip the Q load, so the MMA and softmax warps'
    bounded waits run out: the kernel records RA_ERR_TIMEOUT and returns.  The
    same context then computes a correct result."""
    x = make_qkv(1, 1, 256, 64, 3, with_do=False)
    g = {k: v.cuda() for k, v in x.items()}
    try:
        ra.ring_attn_set_knob(ra.RA_KNOB_WAIT_LIMIT_NS, 2_000_000)
        ra.ring_attn_set_knob(ra.RA_KNOB_DEBUG_FLAGS, 1)
        ra.ring_attn_fwd(g["q"], g["k"], g["v"], "contiguous", 2, True, 0.125)
        st, info = ra.ring_attn_check_device_error()
    finally:
        ra.ring_attn_set_knob(ra.RA_KNOB_DEBUG_FLAGS, 0)
        ra.ring_attn_set_knob(ra.RA_KNOB_WAIT_LIMIT_NS, int(os.environ.get("RA_TEST_WAIT_LIMIT_NS", 4_000_000_000)))
    assert st == 6, (st, info)
    assert ra.ring_attn_check_device_error() == (0, 0)
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], "contiguous", 2, True, 0.125)
    check_no_device_error(ra)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.125, True)
    assert_close("out", out.cpu(), ref_o)
    assert_lse_close("lse", lse.cpu(), ref_l)


@pytest.mark.parametrize("flag", [2, 4], ids=["dkdv", "dq"])
def test_bounded_wait_backward_reports_timeout_and_context_survives(ra, flag):
    """The dK/dV kernel is told to skip its K / V load (flag 2), or the dQ
    kernel its Q / dO load (flag 4), so that kernel's bounded waits run out:
    the backward records RA_ERR_TIMEOUT and returns.  The same context then
    computes a correct backward."""
    x = make_qkv(1, 1, 512, 64, 5, with_do=True)
    g = {k: v.cuda() for k, v in x.items()}
    out, lse = ra.ring_attn_fwd(g["q"], g["k"], g["v"], "contiguous", 2, True, 0.125)
    check_no_device_error(ra)
    try:
        ra.ring_attn_set_knob(ra.RA_KNOB_WAIT_LIMIT_NS, 2_000_000)
        ra.ring_attn_set_knob(ra.RA_KNOB_DEBUG_FLAGS, flag)
        ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, "contiguous", 2, True, 0.125)
        st, info = ra.ring_attn_check_device_error()
    finally:
        ra.ring_attn_set_knob(ra.RA_KNOB_DEBUG_FLAGS, 0)
        ra.ring_attn_set_knob(ra.RA_KNOB_WAIT_LIMIT_NS, int(os.environ.get("RA_TEST_WAIT_LIMIT_NS", 4_000_000_000)))
    assert st == 6, (st, info)
    assert ra.ring_attn_check_device_error() == (0, 0)
    dq, dk, dv = ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, "contiguous", 2, True, 0.125)
    check_no_device_error(ra)
    ref = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], 0.125, True)
    for name, got, want in zip(("dq", "dk", "dv"), (dq, dk, dv), ref):
        assert_close(name, got.cpu(), want)


def test_outputs_are_finite_and_deterministic_shape_errors(ra):
    x = make_qkv(1, 2, 512, 128, 4, with_do=False)
    g = {k: v.cuda() for k, v in x.items()}
    with pytest.raises(ra.RingAttnError):
        ra.ring_attn_fwd(g["q"], g["k"][:, :, :256], g["v"], "contiguous", 2, True)
    with pytest.raises(ra.RingAttnError):
        ra.ring_attn_fwd(g["q"], g["k"], g["v"], "zigzag", 3, True)
    a, la = ra.ring_attn_fwd(g["q"], g["k"], g["v"], "stripe", 4, True)
    b, lb = ra.ring_attn_fwd(g["q"], g["k"], g["v"], "stripe", 4, True)
    assert torch.equal(a, b) and torch.equal(la, lb)
    assert torch.isfinite(a.float()).all() and torch.isfinite(la).all()
