"""GPU parity at every head dim the pages allow, not only multiples of 16.

MTPLX pull request #267, packed_dim sentence: q6 needs D % 4 == 0 (four fields per three bytes),
q4 D % 2 == 0, q8 any D.  Head dims that are not a multiple of 16 take the one-warp-per-row
kernels; codes, scales, dequantized rows and (with side channels) outlier values, positions and
sink rows must equal the oracle's bit for bit, over ragged sequences, appends at nonzero
positions into partially filled pages, rows whose fp16 scale is subnormal or zero, and exact ties.
"""
import numpy as np
import pytest
import torch

import kvgen
from oracle import side as osd
from oracle import symmetric as osym
from _gpu_util import cu_of, dev_tensor, i32, random_rows, u16

pytestmark = pytest.mark.gpu

DIMS = {8: [1, 4, 7, 8, 12, 20, 33, 36, 100, 252, 255],
        6: [4, 8, 12, 20, 36, 100, 252],
        4: [2, 4, 6, 8, 12, 20, 36, 98, 100, 252]}
CASES = [(b, d) for b in (8, 6, 4) for d in DIMS[b]]


def _ties(x, D):
    """Rows of exact half-integer quotients (ties) on scale-1 grids, one per width."""
    rng = np.random.default_rng(D)
    for r, q in ((1, 127), (2, 31), (3, 7)):
        if r < x.shape[0]:
            k = rng.integers(-2 * q, 2 * q + 1, size=D) / 2.0
            k[0] = q
            x[r] = k
    return x


@pytest.mark.parametrize("bits,D", CASES)
def test_quant_dequant_any_head_dim(kvq, cuda_dev, bits, D):
    H, ps = 3, 16
    lens, start = [0, 1, 15, 17, 100, 33], [0, 5, 0, 16, 3, 31]
    pps = (max(s + n for s, n in zip(start, lens)) + ps - 1) // ps
    pt = kvgen.random_page_table(40 + D, len(lens), pps)
    tot = int(sum(lens))
    x = _ties(random_rows(tot * H, D, 50 + D), D).reshape(-1, H, D)
    pool = kvq.Pool.empty(bits, H, D, ps, pt.size, cuda_dev)
    pool.codes.fill_(0xAB)
    pool.scales.fill_(7.0)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    args = (i32(pt, cuda_dev), i32(cu_of(lens), cuda_dev), i32(start, cuda_dev), err)
    kvq.kvq_quant_pack_paged([pool], [dev_tensor(x, cuda_dev)], *args)
    out = torch.full((tot, H, D), float("nan"), dtype=torch.float16, device=cuda_dev)
    kvq.kvq_dequant_paged([pool], [out], *args)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    op = osym.PagedPool(bits, H, D, ps, pt.size)
    op.codes[:] = 0xAB
    op.scales[:] = 7.0
    osym.quant_pack_paged(op, x, pt, cu_of(lens), np.asarray(start))
    od = osym.dequant_paged(op, pt, cu_of(lens), np.asarray(start))
    assert np.array_equal(pool.codes.cpu().numpy(), op.codes)   # untouched slots stay 0xAB
    assert np.array_equal(u16(pool.scales), op.scales.view(np.uint16))
    assert np.array_equal(u16(out), od.view(np.uint16))


SIDE_CASES = [(b, D, k, ns) for b in (8, 6, 4)
              for D, k, ns in ((4, 3, 2), (12, 1, 0), (20, 2, 4), (36, 8, 16), (100, 1, 1),
                               (252, 3, 4))]


@pytest.mark.parametrize("bits,D,k,n_sink", SIDE_CASES)
def test_side_channels_any_head_dim(kvq, cuda_dev, bits, D, k, n_sink):
    H, ps = 2, 16
    lens, starts = np.array([3, 40, 17]), np.array([0, 0, 2])
    nseq = len(lens)
    pt = kvgen.random_page_table(60 + D, nseq, int(((starts + lens).max() + ps - 1) // ps))
    tot = int(lens.sum())
    xs = []
    for i in range(2):
        x = kvgen.KVSpec(seed=61, layer=0, is_key=i == 0, n_seq=1, n_tok=tot, num_heads=H,
                         head_dim=D, n_outlier=min(4, D)).full_np()
        x[1, 0] = np.where(np.arange(D) % 3 == 0, -1.0, 1.0).astype(np.float16)   # ties everywhere
        x[2, 1, :] = 0
        x[2, 1, D // 2] = np.float16(-7.5)                                        # equal maxima
        x[2, 1, 0] = np.float16(7.5)
        xs.append(x)
    pools, sides, osides = [], [], []
    for _ in range(2):
        p = kvq.Pool.empty(bits, H, D, ps, pt.size, cuda_dev)
        p.codes.zero_()
        p.scales.zero_()
        pools.append(p)
        sides.append(kvq.Side.empty(p, k, n_sink, nseq, cuda_dev))
        osides.append(osd.SidePool(osym.PagedPool(bits, H, D, ps, pt.size), k, n_sink, nseq))
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    args = (i32(pt, cuda_dev), i32(cu_of(lens), cuda_dev), i32(starts, cuda_dev), err)
    kvq.kvq_quant_pack_paged_side(pools, sides, [dev_tensor(x, cuda_dev) for x in xs], *args)
    outs = [torch.full((tot, H, D), float("nan"), dtype=torch.float16, device=cuda_dev)
            for _ in range(2)]
    kvq.kvq_dequant_paged_side(pools, sides, outs, *args)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for x, osp in zip(xs, osides):
        osd.quant_pack_paged_side(osp, x, pt, cu_of(lens), starts)
    for p, sd, osp, o in zip(pools, sides, osides, outs):
        assert np.array_equal(p.codes.cpu().numpy(), osp.pool.codes)
        assert np.array_equal(u16(p.scales), osp.pool.scales.view(np.uint16))
        if k:
            assert np.array_equal(sd.out_idx.cpu().numpy(), osp.out_idx)
            assert np.array_equal(u16(sd.out_val), osp.out_val.view(np.uint16))
        if n_sink:
            assert np.array_equal(u16(sd.sink), osp.sink.view(np.uint16))
        ref = osd.dequant_paged_side(osp, pt, cu_of(lens), starts)
        assert np.array_equal(u16(o), ref.view(np.uint16))
