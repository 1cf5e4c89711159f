"""Pins for the fp64 oracle: it is checked against things other than itself.

Each check ties the oracle to a fact the pages or the mathematics fix:
closed forms, invariants, the pages' layout examples, a library routine for
the special case that is plain attention (torch's scaled_dot_product_attention
in float64 on the CPU, with autograd for the gradient), central finite
differences, and the exactness of the ring's block-then-merge form.  The
mutation tests at the end plant plausible mistakes in the oracle and check
that one of these pins fails.
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as A
from workload import WORKLOADS, cu_seqlens, make_qkv, varlen_lengths

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(b, h, s, d, seed, with_do=False):
    t = make_qkv(b, h, s, d, seed, with_do=with_do)
    return {k: v.to(torch.float64).numpy() for k, v in t.items()}


def _sdpa(q, k, v, scale, causal, cu=None, grad_do=None):
    tq, tk, tv = (torch.tensor(x, dtype=torch.float64, requires_grad=grad_do is not None) for x in (q, k, v))
    mask = None
    if cu is not None:
        seg = torch.tensor(A.segment_ids(cu, q.shape[2]))
        mask = seg[:, None] == seg[None, :]
        if causal:
            mask = mask & torch.ones_like(mask).tril()
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=scale)
    else:
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=scale)
    if grad_do is None:
        return out.detach().numpy()
    out.backward(torch.tensor(grad_do, dtype=torch.float64))
    return out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


# --------------------------------------------------------------------------- layouts
def _parse_golden():
    rows = []
    with open(os.path.join(GOLDEN, "layout_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            head, toks = line.split(":")
            layout, n, s, r = head.split()
            prefix = False
            vals = []
            for t in toks.split():
                if t == "...":
                    prefix = True
                elif ".." in t:
                    a, b = t.split("..")
                    vals.extend(range(int(a), int(b) + 1))
                else:
                    vals.append(int(t))
            rows.append((layout, int(n), int(s), int(r), vals, prefix))
    return rows


@pytest.mark.parametrize("case", _parse_golden(), ids=lambda c: f"{c[0]}-N{c[1]}-s{c[2]}-r{c[3]}")
def test_layout_matches_pages_examples(case):
    layout, n, s, r, vals, prefix = case
    g = oracle.token_of_position(layout, n, s)
    L = s // n
    shard = g[r * L:(r + 1) * L]
    if prefix:
        assert list(shard[:len(vals)]) == vals
    else:
        assert list(shard) == vals


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
def test_layout_is_bijection_and_unpermute_inverts(layout, n):
    s = 2 * n * 12
    g = oracle.token_of_position(layout, n, s)
    assert sorted(g.tolist()) == list(range(s))
    x = np.arange(s * 3, dtype=np.float64).reshape(1, 1, s, 3)
    y = oracle.permute(x, layout, n, axis=2)
    assert np.array_equal(oracle.unpermute(y, layout, n, axis=2), x)
    # g is increasing inside every shard (the property tile classification relies on)
    L = s // n
    for r in range(n):
        assert np.all(np.diff(g[r * L:(r + 1) * L]) > 0)


def test_layout_rejects_bad_sizes():
    with pytest.raises(ValueError):
        oracle.token_of_position("zigzag", 4, 12)
    with pytest.raises(ValueError):
        oracle.token_of_position("stripe", 3, 10)
    with pytest.raises(ValueError):
        oracle.token_of_position("diagonal", 2, 8)


# --------------------------------------------------------------------------- closed forms
@pytest.mark.parametrize("causal", [False, True])
def test_zero_query_gives_uniform_weights(causal):
    x = _inputs(1, 2, 37, 8, 11)
    q = np.zeros_like(x["q"])
    out, lse = oracle.attention_fwd(q, x["k"], x["v"], 0.3, causal)
    s = q.shape[2]
    for i in range(s):
        n = i + 1 if causal else s
        np.testing.assert_allclose(out[:, :, i], x["v"][:, :, :n].mean(axis=2), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[:, :, i], math.log(n), rtol=0, atol=1e-12)


def test_zero_query_varlen_uniform_within_segment():
    lens = [5, 1, 9, 3]
    cu = cu_seqlens(lens)
    s = sum(lens)
    x = _inputs(1, 1, s, 4, 12)
    q = np.zeros_like(x["q"])
    out, lse = oracle.attention_fwd(q, x["k"], x["v"], 1.0, True, cu_seqlens=cu)
    for k in range(len(lens)):
        for i in range(cu[k], cu[k + 1]):
            n = i - cu[k] + 1
            np.testing.assert_allclose(out[0, 0, i], x["v"][0, 0, cu[k]:i + 1].mean(axis=0), atol=1e-12)
            assert abs(lse[0, 0, i] - math.log(n)) < 1e-12


def test_equal_keys_give_uniform_weights():
    x = _inputs(1, 1, 20, 8, 13)
    k = np.repeat(x["k"][:, :, :1], 20, axis=2)
    out, lse = oracle.attention_fwd(x["q"], k, x["v"], 0.5, False)
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(x["v"][0, 0].mean(axis=0), (20, 8)), atol=1e-12)
    np.testing.assert_allclose(lse[0, 0], 0.5 * x["q"][0, 0] @ k[0, 0, 0] + math.log(20), atol=1e-12)


def test_causal_row_zero_and_single_token():
    x = _inputs(2, 3, 9, 16, 14)
    sc = 0.25
    out, lse = oracle.attention_fwd(x["q"], x["k"], x["v"], sc, True)
    np.testing.assert_allclose(out[:, :, 0], x["v"][:, :, 0], atol=0)
    np.testing.assert_allclose(lse[:, :, 0], sc * np.einsum("bhd,bhd->bh", x["q"][:, :, 0], x["k"][:, :, 0]),
                               atol=1e-13)
    one = {k: v[:, :, :1] for k, v in x.items()}
    o1, _ = oracle.attention_fwd(one["q"], one["k"], one["v"], sc, False)
    np.testing.assert_array_equal(o1, one["v"])


def test_rows_of_p_sum_to_one():
    x = _inputs(1, 2, 50, 8, 15)
    v = np.ones_like(x["v"])
    for causal in (False, True):
        out, lse = oracle.attention_fwd(x["q"], x["k"], v, 0.7, causal)
        np.testing.assert_allclose(out, 1.0, atol=1e-12)
        # exp(S - lse) sums to one on each row
        S = 0.7 * np.einsum("bhid,bhjd->bhij", x["q"], x["k"])
        if causal:
            S = np.where(np.tril(np.ones((50, 50), bool)), S, -np.inf)
        np.testing.assert_allclose(np.exp(S - lse[..., None]).sum(-1), 1.0, atol=1e-12)


# --------------------------------------------------------------------------- library routine
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("s,d", [(4, 4), (33, 16), (130, 64)])
def test_matches_torch_sdpa_float64(causal, s, d):
    x = _inputs(2, 2, s, d, 16 + s)
    sc = 1.0 / math.sqrt(d)
    out, _ = oracle.attention_fwd(x["q"], x["k"], x["v"], sc, causal, row_block=32)
    np.testing.assert_allclose(out, _sdpa(x["q"], x["k"], x["v"], sc, causal), rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_matches_torch_sdpa_block_mask(causal):
    lens = [7, 1, 20, 4, 12]
    cu = cu_seqlens(lens)
    x = _inputs(1, 2, sum(lens), 8, 17)
    out, _ = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.4, causal, cu_seqlens=cu)
    np.testing.assert_allclose(out, _sdpa(x["q"], x["k"], x["v"], 0.4, causal, cu=cu), atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("varlen", [False, True])
def test_gradient_matches_torch_autograd(causal, varlen):
    lens = [6, 10, 3, 13] if varlen else None
    s = 32
    cu = cu_seqlens(lens) if varlen else None
    x = _inputs(1, 2, s, 8, 18, with_do=True)
    dq, dk, dv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], 0.35, causal, cu_seqlens=cu, row_block=7)
    _, tq, tk, tv = _sdpa(x["q"], x["k"], x["v"], 0.35, causal, cu=cu, grad_do=x["do"])
    for a, b in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-11)


# --------------------------------------------------------------------------- finite differences
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("varlen", [False, True])
def test_gradient_central_finite_differences(causal, varlen):
    s, d = 12, 6
    cu = cu_seqlens([5, 7]) if varlen else None
    x = _inputs(1, 1, s, d, 19, with_do=True)
    sc = 0.45
    dq, dk, dv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], sc, causal, cu_seqlens=cu)

    def loss(q, k, v):
        out, _ = oracle.attention_fwd(q, k, v, sc, causal, cu_seqlens=cu)
        return float((x["do"] * out).sum())

    h = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args = {n: x[n].copy() for n in ("q", "k", "v")}
            args[name][idx] += h
            fp = loss(args["q"], args["k"], args["v"])
            args[name][idx] -= 2 * h
            fm = loss(args["q"], args["k"], args["v"])
            num[idx] = (fp - fm) / (2 * h)
        rel = np.linalg.norm(num - grad) / max(np.linalg.norm(grad), 1e-30)
        assert rel <= 1e-6, (name, rel)


# --------------------------------------------------------------------------- ring form
@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_sharded_then_merged_equals_full(layout, n, causal):
    s = 2 * n * 5
    x = _inputs(1, 2, s, 8, 20 + n)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.5, causal)
    o, l = oracle.ring_attention_sharded(x["q"], x["k"], x["v"], layout, n, 0.5, causal)
    np.testing.assert_allclose(o, ref_o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, rtol=0, atol=1e-12)


@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_sharded_then_merged_equals_full(n, causal):
    lens = [9, 1, 17, 5, 24, 8]
    s = sum(lens)  # 64
    cu = cu_seqlens(lens)
    x = _inputs(1, 1, s, 8, 30 + n)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.5, causal, cu_seqlens=cu)
    o, l = oracle.ring_attention_sharded(x["q"], x["k"], x["v"], "contiguous", n, 0.5, causal, cu_seqlens=cu)
    np.testing.assert_allclose(o, ref_o, atol=1e-12)
    np.testing.assert_allclose(l, ref_l, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_online_softmax_form_equals_definition(causal):
    x = _inputs(1, 2, 70, 16, 40)
    ref, _ = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.25, causal)
    for blk in (1, 16, 64, 128):
        out = oracle.online_softmax_attention(x["q"], x["k"], x["v"], 0.25, causal, kv_block=blk)
        np.testing.assert_allclose(out, ref, atol=1e-12)
    lens = [30, 10, 30]
    cu = cu_seqlens(lens)
    ref, _ = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.25, causal, cu_seqlens=cu)
    out = oracle.online_softmax_attention(x["q"], x["k"], x["v"], 0.25, causal, kv_block=16, cu_seqlens=cu)
    np.testing.assert_allclose(out, ref, atol=1e-12)


def test_lse_merge_infinity_rules_and_self_merge():
    rng = np.random.default_rng(0)
    oa, ob = rng.standard_normal((4, 3)), rng.standard_normal((4, 3))
    la = np.array([0.5, -np.inf, 2.0, -np.inf])
    lb = np.array([-np.inf, 1.5, 2.0, -np.inf])
    o, l = oracle.lse_merge(oa, la, ob, lb)
    np.testing.assert_array_equal(o[0], oa[0])       # block empty: unchanged
    assert l[0] == 0.5
    np.testing.assert_array_equal(o[1], ob[1])       # accumulator empty: take the block
    assert l[1] == 1.5
    np.testing.assert_allclose(o[2], 0.5 * (oa[2] + ob[2]), atol=1e-15)  # equal lse: average
    assert abs(l[2] - (2.0 + math.log(2.0))) < 1e-15
    np.testing.assert_array_equal(o[3], 0.0)         # both empty
    assert l[3] == -np.inf
    assert not np.isnan(o).any()
    # merging a result with itself keeps out and adds log 2
    o2, l2 = oracle.lse_merge(oa, np.array([1.0, 2, 3, 4]), oa, np.array([1.0, 2, 3, 4]))
    np.testing.assert_allclose(o2, oa, atol=1e-15)
    np.testing.assert_allclose(l2, np.array([1.0, 2, 3, 4]) + math.log(2), atol=1e-15)


def test_sampled_rows_and_keys_match_full():
    lens = [20, 44]
    for cu in (None, cu_seqlens(lens)):
        for causal in (False, True):
            x = _inputs(1, 1, 64, 8, 50, with_do=True)
            q, k, v, do = (x[n][0, 0] for n in ("q", "k", "v", "do"))
            out, lse = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.3, causal, cu_seqlens=cu)
            dq, dk, dv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], 0.3, causal, cu_seqlens=cu)
            rows = [0, 5, 19, 20, 63]
            o_r, l_r, D_r, dq_r = oracle.attention_rows(q, k, v, rows, 0.3, causal, cu, do=do)
            np.testing.assert_allclose(o_r, out[0, 0, rows], atol=1e-13)
            np.testing.assert_allclose(l_r, lse[0, 0, rows], atol=1e-13)
            np.testing.assert_allclose(dq_r, dq[0, 0, rows], atol=1e-13)
            D = (do * out[0, 0]).sum(-1)
            dk_r, dv_r = oracle.key_grads(q, k, v, do, rows, lse[0, 0], D, 0.3, causal, cu)
            np.testing.assert_allclose(dk_r, dk[0, 0, rows], atol=1e-13)
            np.testing.assert_allclose(dv_r, dv[0, 0, rows], atol=1e-13)


# --------------------------------------------------------------------------- inputs
def test_varlen_lengths_recipe():
    w = WORKLOADS[5]
    lens = w.seq_lengths()
    assert len(lens) == 64 and sum(lens) == 131072 and min(lens) >= 1
    assert lens == varlen_lengths(64, 131072, 2000)
    assert (min(lens), max(lens)) == (275, 7634)
    assert sum(float(n) ** 2 for n in lens) * 8192 == pytest.approx(4.0427e12, rel=1e-4)
    cu = cu_seqlens(lens)
    assert cu[0] == 0 and cu[-1] == 131072 and np.all(np.diff(cu) > 0)


def test_inputs_are_seeded_bf16():
    a = make_qkv(1, 2, 16, 8, 7)
    b = make_qkv(1, 2, 16, 8, 7)
    for n in ("q", "k", "v", "do"):
        assert a[n].dtype == torch.bfloat16 and torch.equal(a[n], b[n])
    assert not torch.equal(a["q"], a["k"])


# --------------------------------------------------------------------------- planted mistakes
def _pins_hold():
    """A compact run of the pins above; False when any of them fails."""
    try:
        x = _inputs(1, 1, 16, 4, 60, with_do=True)
        for causal in (False, True):
            out, lse = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.6, causal)
            if not np.allclose(out, _sdpa(x["q"], x["k"], x["v"], 0.6, causal), atol=1e-11):
                return False
            q0 = np.zeros_like(x["q"])
            _, l0 = oracle.attention_fwd(q0, x["k"], x["v"], 0.6, causal)
            n = np.arange(1, 17) if causal else np.full(16, 16)
            if not np.allclose(l0[0, 0], np.log(n), atol=1e-12):
                return False
            _, tq, tk, tv = _sdpa(x["q"], x["k"], x["v"], 0.6, causal, grad_do=x["do"])
            g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], 0.6, causal)
            if not all(np.allclose(a, b, atol=1e-10) for a, b in zip(g, (tq, tk, tv))):
                return False
            for layout in oracle.LAYOUTS:
                o2, l2 = oracle.ring_attention_sharded(x["q"], x["k"], x["v"], layout, 4, 0.6, causal)
                if not (np.allclose(o2, out, atol=1e-12) and np.allclose(l2, lse, atol=1e-12)):
                    return False
        for case in _parse_golden():
            layout, nn, s, r, vals, prefix = case
            g = oracle.token_of_position(layout, nn, s)[r * (s // nn):(r + 1) * (s // nn)]
            if list(g[:len(vals)] if prefix else g) != vals:
                return False
        if not _varlen_zigzag_pins_hold():
            return False
        return True
    except (AssertionError, ValueError, IndexError, FloatingPointError):
        return False


# Zigzag varlen: the zigzag split applied to every packed sequence.  Worked by
# hand from that definition for cu_seqlens = [0, 4, 12], N = 2: sequence 0 has
# chunks {0}, {1}, {2}, {3} and sequence 1 chunks {4,5}, {6,7}, {8,9}, {10,11};
# shard 0 takes chunks 0 and 3 of each, shard 1 chunks 1 and 2.
_VZ_EXAMPLE = ([0, 4, 12], 2, [0, 3, 4, 5, 10, 11, 1, 2, 6, 7, 8, 9])


def _varlen_zigzag_pins_hold():
    cu, n, want = _VZ_EXAMPLE
    if list(oracle.varlen_token_of_position("zigzag", n, cu)) != want:
        return False
    for n in (1, 2, 3, 4):  # one sequence: the batched zigzag map
        if not np.array_equal(oracle.varlen_token_of_position("zigzag", n, [0, 48]),
                              oracle.token_of_position("zigzag", n, 48)):
            return False
    return True


def test_varlen_zigzag_layout_pins():
    assert _varlen_zigzag_pins_hold()


@pytest.mark.parametrize("n", [1, 2, 3, 4])
def test_varlen_zigzag_layout_structure(n):
    lens = [2 * n * m for m in (3, 1, 0, 5, 2)]
    cu = cu_seqlens(lens)
    g = oracle.varlen_token_of_position("zigzag", n, cu)
    total = cu[-1]
    assert sorted(g.tolist()) == list(range(total))  # a bijection
    L = total // n
    seg = oracle.segment_ids(cu, total)
    for r in range(n):
        loc = g[r * L:(r + 1) * L]
        assert np.all(np.diff(loc) > 0)  # increasing inside every shard
        for k in range(len(lens)):       # sequence k at local [cu[k]/N, cu[k+1]/N) of every shard
            assert np.all(seg[loc[cu[k] // n:cu[k + 1] // n]] == k)
    x = np.random.default_rng(3).standard_normal((2, total, 3))
    y = oracle.permute(x, "zigzag", n, axis=1, cu_seqlens=cu)
    assert np.array_equal(oracle.unpermute(y, "zigzag", n, axis=1, cu_seqlens=cu), x)
    assert np.array_equal(oracle.varlen_token_of_position("contiguous", n, cu), np.arange(total))


def test_varlen_zigzag_rejects_bad_sizes():
    with pytest.raises(ValueError):
        oracle.varlen_token_of_position("zigzag", 2, [0, 6])      # 6 is not a multiple of 4
    with pytest.raises(ValueError):
        oracle.varlen_token_of_position("stripe", 2, [0, 8])


@pytest.mark.parametrize("n", [1, 2, 3, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_varlen_zigzag_sharded_then_merged_equals_full(n, causal):
    lens = [2 * n * m for m in (2, 1, 4)]
    cu = cu_seqlens(lens)
    x = _inputs(1, 2, cu[-1], 8, 91 + n, with_do=False)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.5, causal, cu_seqlens=cu)
    o, l = oracle.ring_attention_sharded(x["q"], x["k"], x["v"], "zigzag", n, 0.5, causal, cu_seqlens=cu)
    assert np.allclose(o, ref_o, atol=1e-12, rtol=0)
    assert np.allclose(l, ref_l, atol=1e-12, rtol=0)


@pytest.mark.parametrize("n", [1, 2, 3, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_llama3_ranks_compose_to_full_attention(n, causal):
    """Outputs of the ranks concatenate to full varlen attention, and the ranks'
    dk / dv contributions sum to the full gradient (the gradient is linear in dO)."""
    lens = [5, 17, 0, 9, 29]
    cu = cu_seqlens(lens)
    s = cu[-1] + (-cu[-1]) % n
    if s != cu[-1]:
        lens[-1] += s - cu[-1]
        cu = cu_seqlens(lens)
    x = _inputs(1, 2, s, 8, 140 + n, with_do=True)
    ref_o, ref_l = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.45, causal, cu_seqlens=cu)
    ref_g = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], 0.45, causal, cu_seqlens=cu)
    L = s // n
    dk_sum = np.zeros_like(ref_g[1])
    dv_sum = np.zeros_like(ref_g[2])
    for r in range(n):
        rows = slice(r * L, (r + 1) * L)
        o, l, dq, dk, dv = oracle.llama3_rank_attention(x["q"], x["k"], x["v"], r, n, 0.45, causal, cu_seqlens=cu,
                                                        do=x["do"][:, :, rows])
        assert np.allclose(o, ref_o[:, :, rows], atol=1e-12, rtol=0)
        assert np.allclose(l, ref_l[:, :, rows], atol=1e-12, rtol=0)
        assert np.allclose(dq, ref_g[0][:, :, rows], atol=1e-12, rtol=0)
        dk_sum += dk
        dv_sum += dv
    assert np.allclose(dk_sum, ref_g[1], atol=1e-11, rtol=0)
    assert np.allclose(dv_sum, ref_g[2], atol=1e-11, rtol=0)


def test_pins_hold_on_the_unmodified_oracle():
    assert _pins_hold()


def _mutant_block_no_scale(q, k, v, gq, gk, scale, causal, segq=None, segk=None):
    return _ORIG_BLOCK(q, k, v, gq, gk, 1.0, causal, segq, segk)


def _mutant_block_strict_causal(q, k, v, gq, gk, scale, causal, segq=None, segk=None):
    if not causal:
        return _ORIG_BLOCK(q, k, v, gq, gk, scale, causal, segq, segk)
    # j < i instead of j <= i: shift the key indices by one
    return _ORIG_BLOCK(q, k, v, np.asarray(gq), np.asarray(gk) + 1, scale, causal, segq, segk)


def _mutant_block_log2(q, k, v, gq, gk, scale, causal, segq=None, segk=None):
    o, l = _ORIG_BLOCK(q, k, v, gq, gk, scale, causal, segq, segk)
    return o, l / math.log(2.0)


def _mutant_block_transposed_v(q, k, v, gq, gk, scale, causal, segq=None, segk=None):
    o, l = _ORIG_BLOCK(q, k, v, gq, gk, scale, causal, segq, segk)
    return o[::-1].copy(), l


def _mutant_merge_swapped(out_acc, lse_acc, out_blk, lse_blk):
    o, l = _ORIG_MERGE(out_blk, lse_acc, out_acc, lse_blk)
    return o, l


def _mutant_layout_zigzag(layout, n_shards, s):
    g = _ORIG_TOKEN(layout, n_shards, s)
    if layout == "zigzag":
        L = s // n_shards
        c = L // 2
        g = g.copy()
        for r in range(n_shards):   # second chunk taken as 2N-2-r (off by one)
            g[r * L + c:(r + 1) * L] = ((2 * n_shards - 2 - r) % (2 * n_shards)) * c + np.arange(c)
    return g


def _mutant_layout_stripe(layout, n_shards, s):
    g = _ORIG_TOKEN(layout, n_shards, s)
    if layout == "stripe":
        L = s // n_shards
        g = np.array([i * n_shards + (n_shards - 1 - r) for r in range(n_shards) for i in range(L)])
    return g


def _mutant_varlen_zigzag_order(layout, n_shards, cu_seqlens):
    g = _ORIG_VTOKEN(layout, n_shards, cu_seqlens)
    if layout == "zigzag":  # chunk 2N-1-r placed before chunk r in every sequence
        cu = list(cu_seqlens)
        out = []
        for r in range(n_shards):
            for k in range(len(cu) - 1):
                c = (cu[k + 1] - cu[k]) // (2 * n_shards)
                out += [cu[k] + (2 * n_shards - 1 - r) * c + o for o in range(c)]
                out += [cu[k] + r * c + o for o in range(c)]
        g = np.asarray(out, dtype=np.int64)
    return g


_ORIG_BLOCK = A.block_attention
_ORIG_VTOKEN = A.varlen_token_of_position
_ORIG_MERGE = A.lse_merge
_ORIG_TOKEN = A.token_of_position


@pytest.mark.parametrize("target,mutant", [
    ("block_attention", _mutant_block_no_scale),
    ("block_attention", _mutant_block_strict_causal),
    ("block_attention", _mutant_block_log2),
    ("block_attention", _mutant_block_transposed_v),
    ("lse_merge", _mutant_merge_swapped),
    ("token_of_position", _mutant_layout_zigzag),
    ("token_of_position", _mutant_layout_stripe),
    ("varlen_token_of_position", _mutant_varlen_zigzag_order),
], ids=lambda x: getattr(x, "__name__", x))
def test_planted_mistake_fails_a_pin(monkeypatch, target, mutant):
    monkeypatch.setattr(A, target, mutant)
    monkeypatch.setattr(oracle, target, mutant)
    assert not _pins_hold()


def test_planted_gradient_sign_error_fails_a_pin(monkeypatch):
    orig = A.attention_bwd

    def mutant(q, k, v, do, scale, causal, cu_seqlens=None, row_block=1024):
        dq, dk, dv = orig(q, k, v, do, scale, causal, cu_seqlens, row_block)
        return dq, -dk, dv          # a flipped sign in dS^T Q

    monkeypatch.setattr(A, "attention_bwd", mutant)
    monkeypatch.setattr(oracle, "attention_bwd", mutant)
    assert not _pins_hold()


# --------------------------------------------------------------------------- grouped-query attention
def _gqa_inputs(h, hk, s, d, seed):
    x = _inputs(1, h, s, d, seed, with_do=True)
    return {"q": x["q"], "k": x["k"][:, :hk], "v": x["v"][:, :hk], "do": x["do"]}


@pytest.mark.parametrize("h,hk", [(4, 1), (4, 2), (6, 3), (3, 3)])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_matches_torch_sdpa_enable_gqa(h, hk, causal):
    """Grouped-query heads against torch's own grouped-query attention (float64,
    autograd): query head i uses key / value head i // (h / hk)."""
    x = _gqa_inputs(h, hk, 20, 8, 300 + h + hk)
    sc = 0.4
    tq, tk, tv = (torch.tensor(x[n], dtype=torch.float64, requires_grad=True) for n in ("q", "k", "v"))
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=sc, enable_gqa=True)
    out.backward(torch.tensor(x["do"], dtype=torch.float64))
    o, _ = oracle.attention_fwd(x["q"], x["k"], x["v"], sc, causal)
    dq, dk, dv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], sc, causal)
    np.testing.assert_allclose(o, out.detach().numpy(), rtol=0, atol=1e-12)
    for a, ref in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
        assert a.shape == ref.shape
        np.testing.assert_allclose(a, ref.numpy(), rtol=0, atol=1e-11)


@pytest.mark.parametrize("causal", [False, True])
def test_gqa_gradient_central_finite_differences(causal):
    """The gradient of a shared key / value head collects every query head of its group."""
    s, d, h, hk = 10, 4, 4, 2
    x = _gqa_inputs(h, hk, s, d, 33)
    cu = cu_seqlens([4, 6])
    sc = 0.5
    dq, dk, dv = oracle.attention_bwd(x["q"], x["k"], x["v"], x["do"], sc, causal, cu_seqlens=cu)

    def loss(q, k, v):
        out, _ = oracle.attention_fwd(q, k, v, sc, causal, cu_seqlens=cu)
        return float((x["do"] * out).sum())

    eps = 1e-6
    for name, grad in (("q", dq), ("k", dk), ("v", dv)):
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            args = {n: x[n].copy() for n in ("q", "k", "v")}
            args[name][idx] += eps
            fp = loss(args["q"], args["k"], args["v"])
            args[name][idx] -= 2 * eps
            fm = loss(args["q"], args["k"], args["v"])
            num[idx] = (fp - fm) / (2 * eps)
        rel = np.linalg.norm(num - grad) / max(np.linalg.norm(grad), 1e-30)
        assert rel <= 1e-6, (name, rel)


def test_gqa_planted_interleaved_grouping_is_caught(monkeypatch):
    """A plausible mistake, key / value head i % hk instead of i // (h / hk),
    fails the torch comparison."""
    x = _gqa_inputs(4, 2, 12, 8, 41)
    tq, tk, tv = (torch.tensor(x[n], dtype=torch.float64) for n in ("q", "k", "v"))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=0.5, enable_gqa=True)
    monkeypatch.setattr(A, "_kv_head", lambda hi, h, hk: hi % hk)
    o, _ = oracle.attention_fwd(x["q"], x["k"], x["v"], 0.5, True)
    assert np.abs(o - ref.numpy()).max() > 1e-3


def test_gqa_rejects_head_counts_that_do_not_group():
    x = _gqa_inputs(4, 3, 8, 4, 42)
    with pytest.raises(ValueError):
        oracle.attention_fwd(x["q"], x["k"], x["v"], 0.5, True)
