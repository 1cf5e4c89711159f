"""kvpacked / qkvpacked forms ("Ring Flash Attention" README, API list): strided
views over the batched and varlen calls.  Each is checked bit for bit against
the unpacked call on contiguous copies of the same data (same kernels, same
values), and the batched qkvpacked form also against the fp64 oracle."""
import pytest
import torch

import oracle
from tests.helpers import assert_close, assert_lse_close, check_no_device_error

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


@pytest.fixture(scope="module")
def ra():
    import ring_attn_gb300
    from ring_attn_gb300.build import build

    build()
    ring_attn_gb300.load()
    return ring_attn_gb300


def _randn(*shape, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    return torch.randn(*shape, generator=g).to(BF16).cuda()


def _c(x):
    return x.contiguous()


@pytest.mark.parametrize("layout,n,causal,d", [("zigzag", 2, True, 64), ("stripe", 4, True, 128),
                                               ("contiguous", 2, False, 128)])
def test_qkvpacked_matches_unpacked(ra, layout, n, causal, d):
    b, s, h = 2, 512, 3
    qkv = _randn(b, s, 3, h, d, seed=71)  # layout order along s
    dout = _randn(b, s, h, d, seed=72)
    out, lse = ra.ring_attn_qkvpacked_fwd(qkv, layout, n, causal)
    q, k, v = (_c(qkv[:, :, i].transpose(1, 2)) for i in range(3))
    ref_o, ref_l = ra.ring_attn_fwd(q, k, v, layout, n, causal)
    assert torch.equal(out.transpose(1, 2), ref_o) and torch.equal(lse, ref_l)
    dqkv = ra.ring_attn_qkvpacked_bwd(dout, qkv, out, lse, layout, n, causal)
    dq, dk, dv = ra.ring_attn_bwd(_c(dout.transpose(1, 2)), q, k, v, ref_o, ref_l, layout, n, causal)
    for i, ref in enumerate((dq, dk, dv)):
        assert torch.equal(dqkv[:, :, i].transpose(1, 2), ref), i
    check_no_device_error(ra)
    # against the oracle, in original token order
    orig = lambda t, dim: ra.ring_attn_unpermute(_c(t), layout, n, seq_dim=dim)  # noqa: E731
    o_orig, l_orig = orig(out, 1), orig(lse, 2)
    qo, ko, vo = (orig(qkv[:, :, i], 1).transpose(1, 2).cpu() for i in range(3))
    want_o, want_l = oracle.attention_fwd(qo, ko, vo, d ** -0.5, causal)
    assert_close("out", o_orig.transpose(1, 2).cpu(), want_o)
    assert_lse_close("lse", l_orig.cpu(), want_l)


def test_kvpacked_matches_unpacked(ra):
    b, s, h, d = 1, 384, 2, 128
    q = _randn(b, s, h, d, seed=73)
    kv = _randn(b, s, 2, h, d, seed=74)
    dout = _randn(b, s, h, d, seed=75)
    out, lse = ra.ring_attn_kvpacked_fwd(q, kv, "zigzag", 3, True)
    qc, kc, vc = _c(q.transpose(1, 2)), _c(kv[:, :, 0].transpose(1, 2)), _c(kv[:, :, 1].transpose(1, 2))
    ref_o, ref_l = ra.ring_attn_fwd(qc, kc, vc, "zigzag", 3, True)
    assert torch.equal(out.transpose(1, 2), ref_o) and torch.equal(lse, ref_l)
    dq, dkv = ra.ring_attn_kvpacked_bwd(dout, q, kv, out, lse, "zigzag", 3, True)
    rq, rk, rv = ra.ring_attn_bwd(_c(dout.transpose(1, 2)), qc, kc, vc, ref_o, ref_l, "zigzag", 3, True)
    assert torch.equal(dq.transpose(1, 2), rq)
    assert torch.equal(dkv[:, :, 0].transpose(1, 2), rk) and torch.equal(dkv[:, :, 1].transpose(1, 2), rv)
    check_no_device_error(ra)


def test_varlen_packed_match_unpacked(ra):
    lens = [1, 130, 257, 0, 64, 316]
    cu = [0]
    for n_ in lens:
        cu.append(cu[-1] + n_)
    total, h, d = cu[-1], 2, 64
    qkv = _randn(total, 3, h, d, seed=76)
    dout = _randn(total, h, d, seed=77)
    out, lse = ra.ring_attn_varlen_qkvpacked_fwd(qkv, cu, n_shards=4)
    q, k, v = (_c(qkv[:, i]) for i in range(3))
    ref_o, ref_l = ra.ring_attn_varlen_fwd(q, k, v, cu, None, 4, True)
    assert torch.equal(out, ref_o) and torch.equal(lse, ref_l)
    dqkv = ra.ring_attn_varlen_qkvpacked_bwd(dout, qkv, out, lse, cu, n_shards=4)
    rq, rk, rv = ra.ring_attn_varlen_bwd(dout, q, k, v, ref_o, ref_l, cu, None, 4, True)
    for i, ref in enumerate((rq, rk, rv)):
        assert torch.equal(dqkv[:, i], ref), i
    # kv packed
    out2, lse2 = ra.ring_attn_varlen_kvpacked_fwd(q, _c(qkv[:, 1:]), cu, n_shards=4)
    assert torch.equal(out2, ref_o) and torch.equal(lse2, ref_l)
    dq2, dkv2 = ra.ring_attn_varlen_kvpacked_bwd(dout, q, _c(qkv[:, 1:]), out2, lse2, cu, n_shards=4)
    assert torch.equal(dq2, rq) and torch.equal(dkv2[:, 0], rk) and torch.equal(dkv2[:, 1], rv)
    check_no_device_error(ra)
