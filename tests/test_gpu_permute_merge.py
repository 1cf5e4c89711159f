"""GPU: shard-layout permutation (bit-exact against the oracle's index map) and
the standalone LSE merge (against the oracle's merge, including the -inf rules)."""
import numpy as np
import pytest
import torch

import oracle
from tests.helpers import assert_close, assert_lse_close, check_no_device_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ra():
    import ring_attn_gb300

    from ring_attn_gb300.build import build

    build()
    ring_attn_gb300.load()
    return ring_attn_gb300


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_permute_bit_exact(ra, layout, n, dtype):
    s = 2 * n * 37
    g = torch.Generator("cpu").manual_seed(5 + n)
    x = torch.randn(2, 3, s, 64, generator=g).to(dtype)
    xd = x.cuda()
    y = ra.ring_attn_permute(xd, layout, n, seq_dim=2)
    idx = torch.from_numpy(oracle.token_of_position(layout, n, s))
    ref = x[:, :, idx]
    assert torch.equal(y.cpu().view(torch.int16 if dtype == torch.bfloat16 else torch.int32),
                       ref.view(torch.int16 if dtype == torch.bfloat16 else torch.int32))
    back = ra.ring_attn_unpermute(y, layout, n, seq_dim=2)
    assert torch.equal(back.cpu(), x)
    check_no_device_error(ra)


@pytest.mark.parametrize("layout", oracle.LAYOUTS)
def test_permute_other_axes_and_strides(ra, layout):
    n, s = 4, 64
    g = torch.Generator("cpu").manual_seed(9)
    # lse-like tensor: sequence is the last axis
    x = torch.randn(2, 5, s, generator=g).cuda()
    y = ra.ring_attn_permute(x, layout, n, seq_dim=2)
    idx = torch.from_numpy(oracle.token_of_position(layout, n, s))
    assert torch.equal(y.cpu(), x.cpu()[:, :, idx])
    # varlen-like (total, h, d): sequence on axis 0, and a strided (sliced) source
    base = torch.randn(s, 6, 64, generator=g).to(torch.bfloat16).cuda()
    src = base[:, 1:5]
    y2 = ra.ring_attn_permute(src.contiguous(), layout, n, seq_dim=0)
    assert torch.equal(y2.cpu(), src.cpu()[idx])
    # odd row length (3 bf16 = 6 bytes): element-wise path
    z = torch.randn(1, 2, s, 3, generator=g).to(torch.bfloat16).cuda()
    assert torch.equal(ra.ring_attn_permute(z, layout, n).cpu(), z.cpu()[:, :, idx])
    check_no_device_error(ra)


def _merge_case(rows_shape, d, blk_dtype, seed):
    g = torch.Generator("cpu").manual_seed(seed)
    oa = torch.randn(*rows_shape, d, generator=g)
    ob = torch.randn(*rows_shape, d, generator=g).to(blk_dtype)
    la = torch.randn(*rows_shape, generator=g) * 3
    lb = torch.randn(*rows_shape, generator=g) * 3
    flat_a, flat_b = la.view(-1), lb.view(-1)
    n = flat_a.numel()
    flat_a[0:n:7] = -float("inf")
    flat_b[3:n:5] = -float("inf")
    flat_a[1:n:11] = -float("inf")
    flat_b[1:n:11] = -float("inf")
    return oa, la, ob, lb


@pytest.mark.parametrize("blk_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("shape,d", [((2, 3, 200), 128), ((7, 129), 64), ((2, 4, 50), 128), ((33,), 16),
                                     ((9, 31), 4)])
def test_lse_merge_matches_oracle(ra, blk_dtype, shape, d):
    oa, la, ob, lb = _merge_case(shape, d, blk_dtype, 3)
    ref_o, ref_l = oracle.lse_merge(oa.numpy().reshape(-1, d), la.numpy().reshape(-1),
                                    ob.float().numpy().reshape(-1, d), lb.numpy().reshape(-1))
    goa, gla = oa.cuda(), la.cuda()
    ra.lse_merge(goa, gla, ob.cuda(), lb.cuda())
    check_no_device_error(ra)
    assert_close("out_acc", goa.cpu().reshape(-1, d), ref_o, max_abs=1e-5, rel_l2=1e-6)
    assert_lse_close("lse_acc", gla.cpu().reshape(-1), ref_l, tol=1e-5)


@pytest.mark.parametrize("width", [256, 132])  # 132: rows 16-byte but not 32-byte aligned (4 columns per thread)
def test_lse_merge_strided_views(ra, width):
    g = torch.Generator("cpu").manual_seed(4)
    big_o = torch.randn(3, 40, width, generator=g)
    big_l = torch.randn(3, 80, generator=g)
    oa, la = big_o[:, :, :128], big_l[:, ::2]
    ob = torch.randn(3, 40, 128, generator=g).to(torch.bfloat16)
    lb = torch.randn(3, 40, generator=g)
    ref_o, ref_l = oracle.lse_merge(oa.numpy().reshape(-1, 128), la.numpy().reshape(-1),
                                    ob.float().numpy().reshape(-1, 128), lb.numpy().reshape(-1))
    gbo, gbl = big_o.cuda(), big_l.cuda()
    ra.lse_merge(gbo[:, :, :128], gbl[:, ::2], ob.cuda(), lb.cuda())
    check_no_device_error(ra)
    assert_close("out_acc", gbo[:, :, :128].cpu().reshape(-1, 128), ref_o, max_abs=1e-5, rel_l2=1e-6)
    assert_lse_close("lse_acc", gbl[:, ::2].cpu().reshape(-1), ref_l, tol=1e-5)
    # untouched neighbours
    assert torch.equal(gbo[:, :, 128:].cpu(), big_o[:, :, 128:])
    assert torch.equal(gbl[:, 1::2].cpu(), big_l[:, 1::2])
