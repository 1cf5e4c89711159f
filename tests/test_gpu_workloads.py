"""The benchmark workloads at full size, in the launch configuration that
bench.py times (fused ring forward, then the ring backward with a caller
workspace), checked against the fp64 oracle on sampled outputs it can afford,
plus properties that hold at any size:
  sum_j dK_j = 0 (rows of dS sum to zero) and sum_j dV_j = sum_i dO_i (rows of P
  sum to one), per head, within the rounding of bf16 outputs."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_close, assert_lse_close, check_no_device_error, f64
from workload import WORKLOADS, cu_seqlens, make_workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attn_gb300
    from ring_attn_gb300.build import build

    build()
    ring_attn_gb300.load()
    return ring_attn_gb300


def _sample_rows(s, n, rng, L):
    rows = {0, 1, s - 1, s - 2}
    for r in range(1, min(8, s // max(L, 1))):
        rows.update({r * L - 1, r * L})  # shard boundaries in original order
    rows.update(rng.integers(0, s, size=n).tolist())
    return np.array(sorted(rows))


def _run(ra, w):
    dev = torch.device("cuda")
    x = make_workload_inputs(w, device="cuda")
    scale = w.scale
    res = {"x": x}
    if w.varlen_seqs:
        lens = w.seq_lengths()
        cu = cu_seqlens(lens)
        res["cu"] = cu
        cu_t = torch.tensor(cu, dtype=torch.int32)
        # (h, total, d) in layout order (the identity for contiguous shards)
        g = {k: ra.ring_attn_varlen_permute(v[0].contiguous(), cu_t, w.layout, w.n_shards, seq_dim=1)
             for k, v in x.items()}
        back = lambda t: ra.ring_attn_varlen_unpermute(t, cu_t, w.layout, w.n_shards, seq_dim=1)  # noqa: E731
        out, lse = ra.ring_attn_varlen_fwd(g["q"], g["k"], g["v"], cu_t, None, w.n_shards, w.causal, scale,
                                           layout=w.layout)
        res["out"], res["lse"] = back(out).unsqueeze(0), back(lse).unsqueeze(0)
        if w.backward:
            dq, dk, dv = ra.ring_attn_varlen_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, cu_t, None, w.n_shards,
                                                 w.causal, scale, layout=w.layout)
            res["dq"], res["dk"], res["dv"] = back(dq).unsqueeze(0), back(dk).unsqueeze(0), back(dv).unsqueeze(0)
        del g
    else:
        g = {k: ra.ring_attn_permute(v, w.layout, w.n_shards) for k, v in x.items()}
        out = torch.empty_like(g["q"])
        lse = torch.empty((w.b, w.h, w.s), dtype=torch.float32, device=dev)
        ra.ring_attn_fwd(g["q"], g["k"], g["v"], w.layout, w.n_shards, w.causal, scale, out=out, lse=lse)
        back = lambda t: ra.ring_attn_unpermute(t, w.layout, w.n_shards)  # noqa: E731
        res["out"] = back(out)
        res["lse"] = back(lse)
        if w.backward:
            ws = torch.empty(ra.ring_attn_workspace_size(1, w.b, w.h, w.s, w.d, w.n_shards), dtype=torch.uint8, device=dev)
            dq, dk, dv = ra.ring_attn_bwd(g["do"], g["q"], g["k"], g["v"], out, lse, w.layout, w.n_shards,
                                          w.causal, scale, workspace=ws)
            res["dq"], res["dk"], res["dv"] = back(dq), back(dk), back(dv)
            del ws
        del g
    check_no_device_error(ra)
    return res


def _check_rows(w, res, heads, n_rows, seed):
    rng = np.random.default_rng(seed)
    cu = res.get("cu")
    rows = _sample_rows(w.s, n_rows, rng, w.shard_len)
    for h in heads:
        q, k, v = (res["x"][n][0, h].cpu() for n in ("q", "k", "v"))
        do = res["x"]["do"][0, h].cpu() if w.backward else None
        got = oracle.attention_rows(q, k, v, rows, w.scale, w.causal, cu, do=do)
        assert_close(f"out h{h}", res["out"][0, h, rows].cpu(), got[0])
        assert_lse_close(f"lse h{h}", res["lse"][0, h, rows].cpu(), got[1])
        if w.backward:
            assert_close(f"dq h{h}", res["dq"][0, h, rows].cpu(), got[3])


def _check_keys(w, res, h, keys):
    """dk, dv of selected keys need lse and D of every row that sees them."""
    cu = res.get("cu")
    q, k, v, do = (res["x"][n][0, h].cpu() for n in ("q", "k", "v", "do"))
    keys = np.asarray(sorted(keys))
    if cu is None:
        lo = int(keys.min()) if w.causal else 0
        rows = np.arange(lo, w.s)
    else:
        seg = oracle.segment_ids(cu, w.s)
        rows = np.unique(np.concatenate([np.arange(cu[seg[j]], cu[seg[j] + 1]) for j in keys]))
    _, lse_r, D_r, _ = oracle.attention_rows(q, k, v, rows, w.scale, w.causal, cu, do=do)
    lse = np.full(w.s, np.inf)  # rows outside `rows` never see these keys: P = 0 there
    D = np.zeros(w.s)
    lse[rows] = lse_r
    D[rows] = D_r
    dk, dv = oracle.key_grads(q, k, v, do, keys, lse, D, w.scale, w.causal, cu)
    assert_close(f"dk h{h}", res["dk"][0, h, keys].cpu(), dk)
    assert_close(f"dv h{h}", res["dv"][0, h, keys].cpu(), dv)


def _head_stats(w, res, h):
    """out, lse and D = rowsum(dO * out) of EVERY row of head h, from the fp64
    oracle's forward (row blocks of 1024 queries, so host memory stays bounded)."""
    cu = res.get("cu")
    q, k, v, do = (res["x"][n][0:1, h:h + 1].cpu() for n in ("q", "k", "v", "do"))
    out, lse = oracle.attention_fwd(q, k, v, w.scale, w.causal, cu_seqlens=cu, row_block=1024)
    D = (f64(do)[0, 0] * out[0, 0]).sum(axis=-1)
    return out[0, 0], lse[0, 0], D


def _check_keys_all_rows(w, res, h, keys, stats):
    """dk, dv of selected keys against the oracle, with lse and D of all rows."""
    cu = res.get("cu")
    q, k, v, do = (res["x"][n][0, h].cpu() for n in ("q", "k", "v", "do"))
    keys = np.asarray(sorted(keys))
    _, lse, D = stats
    dk, dv = oracle.key_grads(q, k, v, do, keys, lse, D, w.scale, w.causal, cu)
    assert_close(f"dk h{h} ({len(keys)} keys from {keys.min()})", res["dk"][0, h, keys].cpu(), dk)
    assert_close(f"dv h{h} ({len(keys)} keys from {keys.min()})", res["dv"][0, h, keys].cpu(), dv)


def _check_sums(w, res):
    dk = res["dk"][0].float()
    dv = res["dv"][0].float()
    do = res["x"]["do"][0].float()
    if res.get("cu") is not None:
        return  # per-sequence sums hold too, checked through sampled keys
    for h in range(w.h):
        s_dk = dk[h].double().sum(0)
        a_dk = dk[h].double().abs().sum(0)
        assert torch.all(s_dk.abs() <= 4e-3 * a_dk + 1e-3), f"sum dK h{h}"
        s_dv = dv[h].double().sum(0)
        a_dv = dv[h].double().abs().sum(0)
        ref = do[h].double().sum(0)
        assert torch.all((s_dv - ref).abs() <= 4e-3 * a_dv + 1e-3), f"sum dV h{h}"


def test_tiny_noncausal_full_output(ra):
    w = WORKLOADS[1]
    res = _run(ra, w)
    ref_o, ref_l = oracle.attention_fwd(res["x"]["q"], res["x"]["k"], res["x"]["v"], w.scale, w.causal)
    assert_close("out", res["out"].cpu(), ref_o)
    assert_lse_close("lse", res["lse"].cpu(), ref_l)


def test_causal_contiguous_fwd_h32_s16k(ra):
    w = WORKLOADS[2]
    res = _run(ra, w)
    _check_rows(w, res, heads=[0, 17, 31], n_rows=48, seed=2)
    assert torch.isfinite(res["out"].float()).all() and torch.isfinite(res["lse"]).all()


@pytest.mark.parametrize("wid", [3, 4])
def test_causal_fwd_bwd_full_size(ra, wid):
    """Sampled rows of two heads; then, for head 0, out and lse of every row and
    dk, dv of the keys that every shard's queries see: the first 128-token tile
    (zigzag: the start of chunk 0 of shard 0; stripe: local tile 0 of every
    shard), keys around the middle of the sequence and at chunk boundaries,
    and late keys, all against the oracle with lse and D of all rows."""
    w = WORKLOADS[wid]
    res = _run(ra, w)
    _check_rows(w, res, heads=[0, w.h - 1], n_rows=32, seed=wid)
    stats = _head_stats(w, res, 0)
    assert_close("out h0 (all rows)", res["out"][0, 0].cpu(), stats[0])
    assert_lse_close("lse h0 (all rows)", res["lse"][0, 0].cpu(), stats[1])
    rng = np.random.default_rng(wid)
    c = w.s // (2 * w.n_shards)
    _check_keys_all_rows(w, res, 0, range(0, 128), stats)
    mid = set(range(w.s // 2 - 8, w.s // 2 + 8)) | {c - 1, c, 3 * c - 1, 3 * c, 7 * c + 5}
    mid |= set(rng.integers(0, w.s, size=16).tolist())
    _check_keys_all_rows(w, res, 0, mid, stats)
    late = set((w.s - 1 - rng.integers(0, 2048, size=12)).tolist()) | {w.s - 1, w.s - 2048}
    _check_keys_all_rows(w, res, 0, late, stats)
    _check_sums(w, res)
    for n in ("out", "dq", "dk", "dv"):
        assert torch.isfinite(res[n].float()).all(), n


@pytest.mark.parametrize("wid", [5, 6])
def test_varlen_fwd_bwd_full_size(ra, wid):
    w = WORKLOADS[wid]
    res = _run(ra, w)
    _check_rows(w, res, heads=[0, 31], n_rows=48, seed=wid)
    cu = res["cu"]
    rng = np.random.default_rng(55)
    segs = rng.choice(len(cu) - 1, size=3, replace=False)
    keys = set()
    for sg in segs:
        keys.update(rng.integers(cu[sg], cu[sg + 1], size=4).tolist())
        keys.update({int(cu[sg]), int(cu[sg + 1] - 1)})
    _check_keys(w, res, 0, keys)
    # every row of head 0, and the first 128 keys of the longest sequence (the
    # keys with the most queries) with lse and D of all rows
    stats = _head_stats(w, res, 0)
    assert_close("out h0 (all rows)", res["out"][0, 0].cpu(), stats[0])
    assert_lse_close("lse h0 (all rows)", res["lse"][0, 0].cpu(), stats[1])
    longest = int(np.argmax(np.diff(cu)))
    _check_keys_all_rows(w, res, 0, range(int(cu[longest]), int(cu[longest]) + 128), stats)
    for n in ("out", "dq", "dk", "dv"):
        assert torch.isfinite(res[n].float()).all(), n
