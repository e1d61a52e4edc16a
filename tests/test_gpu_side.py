"""GPU parity for the fp16 side channels on the symmetric path (attention sinks, dense-and-sparse
outliers): kvq_quant_pack_paged_side / kvq_dequant_paged_side against oracle/side.py bit for bit
(codes, scales, outlier values and positions, sink rows, dequantized rows)."""
import numpy as np
import pytest
import torch

import kvgen
from oracle import side as osd
from oracle import symmetric as osym
from _attn_checks import assert_attn_close
from _gpu_util import cu_of, dev_tensor, i32, u16

pytestmark = pytest.mark.gpu


def _rows(seed, is_key, n, H, D):
    x = kvgen.KVSpec(seed=seed, layer=0, is_key=is_key, n_seq=1, n_tok=n, num_heads=H,
                     head_dim=D).full_np()
    if n > 3:   # magnitude ties: a row of +-1 (ties everywhere) and one with two equal maxima
        x[1, 0] = np.where(np.arange(D) % 3 == 0, -1.0, 1.0).astype(np.float16)
        x[2, 0, 5] = x[2, 0, 9] = np.float16(-7.5)
        x[2, 0, 200 % D] = np.float16(7.5)
    return x


def _setup(kvq, dev, bits, H, D, ps, k, n_sink, lens, starts, seed=1):
    lens, starts = np.asarray(lens), np.asarray(starts)
    nseq = len(lens)
    pps = int(((starts + lens).max() + ps - 1) // ps)
    pt_np = kvgen.random_page_table(seed, nseq, pps)
    n_pages = pt_np.size
    pools, sides, opools, osides = [], [], [], []
    for _ in range(2):
        p = kvq.Pool.empty(bits, H, D, ps, n_pages, dev)
        p.codes.zero_()
        p.scales.zero_()
        pools.append(p)
        sides.append(kvq.Side.empty(p, k, n_sink, nseq, dev))
        op = osym.PagedPool(bits, H, D, ps, n_pages)
        opools.append(op)
        osides.append(osd.SidePool(op, k, n_sink, nseq))
    return pt_np, pools, sides, opools, osides


def _compare_state(pools, sides, opools, osides, n_sink):
    for p, sd, op, osp in zip(pools, sides, opools, osides):
        assert np.array_equal(p.codes.cpu().numpy(), op.codes)
        assert np.array_equal(u16(p.scales), op.scales.view(np.uint16))
        if sd.n_outlier:
            assert np.array_equal(sd.out_idx.cpu().numpy(), osp.out_idx)
            assert np.array_equal(u16(sd.out_val), osp.out_val.view(np.uint16))
        if n_sink:
            assert np.array_equal(u16(sd.sink), osp.sink.view(np.uint16))


@pytest.mark.parametrize("bits", [8, 6, 4])
@pytest.mark.parametrize("D,k,n_sink", [(256, 3, 4), (256, 8, 16), (128, 2, 0), (64, 0, 4),
                                        (256, 1, 1), (16, 8, 2), (48, 5, 2), (96, 3, 0)])
def test_quant_dequant_side_bit_exact(kvq, cuda_dev, bits, D, k, n_sink):
    H, ps = 4, 16
    lens, starts = [1, 5, 40, 100], [0, 0, 0, 0]
    pt_np, pools, sides, opools, osides = _setup(kvq, cuda_dev, bits, H, D, ps, k, n_sink,
                                                 lens, starts)
    tot = int(sum(lens))
    xs = [_rows(3, True, tot, H, D), _rows(3, False, tot, H, D)]
    cu = cu_of(lens)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_quant_pack_paged_side(pools, sides, [dev_tensor(x, cuda_dev) for x in xs],
                                  i32(pt_np, cuda_dev), i32(cu, cuda_dev), i32(starts, cuda_dev),
                                  err)
    for x, osp in zip(xs, osides):
        osd.quant_pack_paged_side(osp, x, pt_np, cu, np.asarray(starts))
    outs = [torch.full((tot, H, D), float("nan"), dtype=torch.float16, device=cuda_dev)
            for _ in range(2)]
    kvq.kvq_dequant_paged_side(pools, sides, outs, i32(pt_np, cuda_dev), i32(cu, cuda_dev),
                               i32(starts, cuda_dev), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _compare_state(pools, sides, opools, osides, n_sink)
    for o, osp in zip(outs, osides):
        want = osd.dequant_paged_side(osp, pt_np, cu, np.asarray(starts))
        assert np.array_equal(u16(o), want.view(np.uint16))


def _distinct(cands, D, n):
    """The first n distinct positions of cands taken modulo D."""
    out = []
    for c in cands:
        if c % D not in out:
            out.append(c % D)
        if len(out) == n:
            return out
    return out + [p for p in range(D) if p not in out][:n - len(out)]


def _selection_rows(D, k, rng):
    """Rows that stress the choice of outliers: the k + 1 largest magnitudes in one lane's
    elements (lanes hold units i and i + 8 of a row), equal outliers above the threshold, ties at
    the threshold (the k-th and (k+1)-th magnitudes equal, the lower position wins) and just
    below it, runs of equal maxima across lanes, subnormal rows, rows with exactly k and k - 1
    nonzeros, signed zeros, outliers at the row's ends; each crafted row sits between plain rows
    so a warp step sees rows with and without ties."""
    def base():
        return np.clip(rng.standard_normal(D) * 0.5, -2, 2).astype(np.float16)

    def put(r, pos, mags, signs=None):
        for i, (p, m) in enumerate(zip(pos, mags)):
            sg = -1.0 if signs is not None and i < len(signs) and signs[i] else 1.0
            r[p] = np.float16(sg * m)
        return r

    lane0 = [3, 130, 7, 140, 12, 135, 1, 129, 9, 14] if D > 128 else [3, 7, 12, 1, 9, 14, 0, 5]
    spread = [37 * i + 11 for i in range(2 * k + 4)]
    crafted = [
        put(base(), _distinct(lane0, D, k + 1), [9.0 - i for i in range(k + 1)]),
        put(base(), _distinct(spread, D, k), [10.0] * k, [i % 2 for i in range(k)]),
        # tie at the threshold, the later position first in the list
        put(base(), _distinct([D - 1, D // 2] + spread, D, k + 1),
            [6.0, 6.0] + [10.0 + i for i in range(k - 1)]),
        # tie just below the threshold
        put(base(), _distinct(spread, D, k + 2), [10.0 + i for i in range(k)] + [5.0, 5.0]),
        # three equal at the threshold
        put(base(), _distinct([D - 2, 5, D // 3] + spread, D, k + 2),
            [7.0, 7.0, 7.0] + [12.0 + i for i in range(k - 1)], [1, 0, 1]),
        # 2k + 1 equal maxima across the lanes
        put(base(), _distinct(spread[::-1], D, 2 * k + 1), [8.0] * (2 * k + 1)),
        (rng.standard_normal(D) * 2.0 ** -20).astype(np.float16),
        put(np.zeros(D, np.float16), _distinct(spread, D, k), rng.uniform(1, 5, k).tolist()),
        put(np.zeros(D, np.float16), _distinct(spread, D, max(k - 1, 0)),
            rng.uniform(1, 5, max(k - 1, 0)).tolist()),
        np.where(np.arange(D) % 5 == 0, np.float16(-0.0), np.float16(0.0)).astype(np.float16),
        put(base(), _distinct([0, D - 1, D - 2, 1, D - 3, 2], D, k + 1), [4.0, 3.5, 9.0, 3.5]
            + [3.0] * max(0, k - 3), [1, 0, 1, 0]),
    ]
    rows = []
    for r in crafted:
        rows.extend([base(), r, base()])
    return np.stack(rows)


@pytest.mark.parametrize("D,k", [(256, 3), (256, 1), (256, 2), (256, 0), (256, 5), (256, 8),
                                 (128, 3), (96, 3), (64, 2), (16, 3), (16, 8)])
def test_outlier_selection_cases(kvq, cuda_dev, D, k):
    bits, H, ps = 6, 4, 16
    rng = np.random.default_rng(1000 + 10 * D + k)
    rows = _selection_rows(D, k, rng)
    tot = -(-rows.shape[0] // H)
    pad = tot * H - rows.shape[0]
    rows = np.concatenate([rows, np.zeros((pad, D), np.float16)]).reshape(tot, H, D)
    rows_v = rows[::-1].copy()
    lens, starts = [tot], [0]
    pt_np, pools, sides, opools, osides = _setup(kvq, cuda_dev, bits, H, D, ps, k, 0, lens,
                                                 starts)
    cu = cu_of(lens)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_quant_pack_paged_side(pools, sides, [dev_tensor(rows, cuda_dev),
                                                 dev_tensor(rows_v, cuda_dev)],
                                  i32(pt_np, cuda_dev), i32(cu, cuda_dev), i32(starts, cuda_dev),
                                  err)
    for x, osp in zip((rows, rows_v), osides):
        osd.quant_pack_paged_side(osp, x, pt_np, cu, np.asarray(starts))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _compare_state(pools, sides, opools, osides, 0)


def test_append_across_the_sink_boundary(kvq, cuda_dev):
    """Appending to sequences at positions below and above n_sink: the sink buffer takes exactly
    the positions < n_sink, in place, and the rest of the state is untouched."""
    bits, H, D, ps, k, n_sink = 6, 2, 256, 16, 3, 4
    first, second = [2, 0, 30], [5, 3, 2]
    pt_np, pools, sides, opools, osides = _setup(kvq, cuda_dev, bits, H, D, ps, k, n_sink,
                                                 second, np.asarray(first))
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    seed = 10
    for lens, starts in ((first, [0, 0, 0]), (second, first)):
        tot = int(sum(lens))
        xs = [_rows(seed, True, tot, H, D), _rows(seed, False, tot, H, D)]
        seed += 1
        cu = cu_of(lens)
        kvq.kvq_quant_pack_paged_side(pools, sides, [dev_tensor(x, cuda_dev) for x in xs],
                                      i32(pt_np, cuda_dev), i32(cu, cuda_dev),
                                      i32(starts, cuda_dev), err)
        for x, osp in zip(xs, osides):
            osd.quant_pack_paged_side(osp, x, pt_np, cu, np.asarray(starts))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _compare_state(pools, sides, opools, osides, n_sink)


def test_side_rejects_bad_arguments(kvq, cuda_dev):
    p = kvq.Pool.empty(6, 2, 256, 16, 4, cuda_dev)
    x = torch.zeros((4, 2, 256), dtype=torch.float16, device=cuda_dev)
    pt, cu, st = i32([[0, 1, 2, 3]], cuda_dev), i32([0, 4], cuda_dev), i32([0], cuda_dev)
    with pytest.raises(kvq.KVQError):   # 9 outliers
        kvq.kvq_quant_pack_paged_side([p], [kvq.Side.empty(p, 9, 0, 1, cuda_dev)], [x], pt, cu, st)
    with pytest.raises(kvq.KVQError):   # 17 sinks
        kvq.kvq_quant_pack_paged_side([p], [kvq.Side.empty(p, 3, 17, 1, cuda_dev)], [x], pt, cu, st)
    sd = kvq.Side.empty(p, 3, 4, 1, cuda_dev)
    sd.out_val = None
    with pytest.raises(kvq.KVQError):
        kvq.kvq_quant_pack_paged_side([p], [sd], [x], pt, cu, st)


def test_full_size_prefill_sampled(kvq, cuda_dev):
    """The paged-prefill workload (16 layers x K/V x 8 seqs x 32,768 tokens x 4 heads x 256, page
    16), q6, 3 outliers per row (the page's 1 %), 4 sinks: sampled rows of every tensor are
    checked bit for bit -- packed codes, scale, outliers, and the dequantized row."""
    w = kvgen.WORKLOADS["paged_prefill_16L_8x32768_4x256"]
    L, nseq, ntok, H, D, ps = w["n_layers"], w["n_seq"], w["n_tok"], w["H"], w["D"], w["page_size"]
    bits, k, n_sink = 6, osd.outlier_count(D, 0.01), 4
    pt_np = kvgen.random_page_table(1, nseq, ntok // ps)
    pt = i32(pt_np, cuda_dev)
    cu = i32(np.arange(nseq + 1) * ntok, cuda_dev)
    st = i32(np.zeros(nseq), cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    rng = np.random.default_rng(4)
    for layer in (0, 15):   # two layers x K/V through the full-size launch shape
        specs = [kvgen.KVSpec(seed=w["seed"], layer=layer, is_key=kk, n_seq=nseq, n_tok=ntok,
                              num_heads=H, head_dim=D) for kk in (True, False)]
        xs = [s.full_torch(cuda_dev) for s in specs]
        pools = [kvq.Pool.empty(bits, H, D, ps, pt_np.size, cuda_dev) for _ in range(2)]
        sides = [kvq.Side.empty(p, k, n_sink, nseq, cuda_dev) for p in pools]
        kvq.kvq_quant_pack_paged_side(pools, sides, xs, pt, cu, st, err)
        outs = [torch.empty_like(x) for x in xs]
        kvq.kvq_dequant_paged_side(pools, sides, outs, pt, cu, st, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        tok = np.concatenate([rng.integers(0, nseq * ntok, 300), [0, 1, 3, 4, ntok, ntok + 3]])
        for spec, p, sd, out in zip(specs, pools, sides, outs):
            head = rng.integers(0, H, tok.size)
            x = spec.rows_np(tok * H + head)
            s, pos = tok // ntok, tok % ntok
            page, slot = pt_np[s, pos // ps], pos % ps
            packed, scale, opos, oval = osd.quant_pack_rows_side(x, bits, k)
            idx = [torch.from_numpy(a.astype(np.int64)).to(cuda_dev) for a in (page, head, slot)]
            assert np.array_equal(p.codes[idx[0], idx[1], idx[2]].cpu().numpy(), packed)
            assert np.array_equal(u16(p.scales[idx[0], idx[1], idx[2]]), scale.view(np.uint16))
            assert np.array_equal(sd.out_idx[idx[0], idx[1], idx[2]].cpu().numpy(), opos)
            assert np.array_equal(u16(sd.out_val[idx[0], idx[1], idx[2]]), oval.view(np.uint16))
            deq = osd.dequant_rows_side(packed, scale, opos, oval, bits, D)
            deq[pos < n_sink] = x[pos < n_sink]
            rows = out.view(-1, D)[torch.from_numpy(tok * H + head).to(cuda_dev)]
            assert np.array_equal(u16(rows), deq.view(np.uint16))
        del xs, pools, sides, outs
        torch.cuda.empty_cache()


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_side_tensors_aligned_to_16_but_not_32_bytes(kvq, cuda_dev, bits):
    """The fp16 rows take 256-bit accesses only when every tensor is 32-byte aligned; a call
    with a tensor offset by 16 bytes takes the 128-bit path, with the same results."""
    H, D, ps, k, n_sink = 4, 256, 16, 3, 4
    lens, starts = [1, 5, 40, 21], [0, 0, 0, 3]
    tot = int(sum(lens))
    xs = [_rows(5, True, tot, H, D), _rows(5, False, tot, H, D)]
    cu = cu_of(lens)

    def offset_view(a, elems):
        flat = torch.empty(a.size + 64, dtype=torch.float16, device=cuda_dev)
        v = flat[elems:elems + a.size].view(a.shape)
        v.copy_(torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev))
        return v

    for offs in ((16, 16), (16, 8)):   # fp16 elements: 32-byte aligned, then V off by 16 bytes
        pt_np, pools, sides, opools, osides = _setup(kvq, cuda_dev, bits, H, D, ps, k, n_sink,
                                                     lens, starts, seed=7)
        err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
        args = (i32(pt_np, cuda_dev), i32(cu, cuda_dev), i32(starts, cuda_dev), err)
        kvq.kvq_quant_pack_paged_side(pools, sides, [offset_view(x, o) for x, o in zip(xs, offs)],
                                      *args)
        outs = [offset_view(np.full((tot, H, D), np.float16(12345)), o) for o in offs]
        kvq.kvq_dequant_paged_side(pools, sides, outs, *args)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        for x, osp in zip(xs, osides):
            osd.quant_pack_paged_side(osp, x, pt_np, cu, np.asarray(starts))
        _compare_state(pools, sides, opools, osides, n_sink)
        for o, osp in zip(outs, osides):
            ref = osd.dequant_paged_side(osp, pt_np, cu, np.asarray(starts))
            assert np.array_equal(u16(o), ref.view(np.uint16))


# ---------------------------------------------------------------- decode attention


def _close(got, ref):
    assert_attn_close(got, ref, "side-channel decode attention")


@pytest.mark.parametrize("bits", [8, 6, 4])
@pytest.mark.parametrize("k,n_sink,ps", [(3, 4, 16), (0, 4, 16), (3, 0, 16), (8, 16, 32),
                                         (1, 1, 16), (4, 2, 16), (5, 2, 16)])
def test_decode_attn_side(kvq, cuda_dev, bits, k, n_sink, ps):
    H, G, D, L = 4, 6, 256, 2
    lens = [1, 3, 16, 17, 100, 1000, 0]
    nseq = len(lens)
    starts = [0] * nseq
    pt_np = None
    kps, vps, kss, vss, oks, ovs = [], [], [], [], [], []
    for layer in range(L):
        pt_np, pools, sides, opools, osides = _setup(kvq, cuda_dev, bits, H, D, ps, k, n_sink,
                                                     lens, starts)
        tot = int(sum(lens))
        xs = [_rows(20 + layer, True, tot, H, D), _rows(20 + layer, False, tot, H, D)]
        cu = cu_of(lens)
        kvq.kvq_quant_pack_paged_side(pools, sides, [dev_tensor(x, cuda_dev) for x in xs],
                                      i32(pt_np, cuda_dev), i32(cu, cuda_dev),
                                      i32(starts, cuda_dev))
        for x, osp in zip(xs, osides):
            osd.quant_pack_paged_side(osp, x, pt_np, cu, np.asarray(starts))
        kps.append(pools[0]); vps.append(pools[1]); kss.append(sides[0]); vss.append(sides[1])
        oks.append(osides[0]); ovs.append(osides[1])
    q = kvgen.queries_np(30, L, nseq, H * G, D)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
    ws = kvq.decode_workspace(kps, nseq, H * G, max(lens), cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_decode_attn_side(kps, vps, kss, vss, dev_tensor(q, cuda_dev), i32(pt_np, cuda_dev),
                             i32(lens, cuda_dev), max(lens), 1.0 / 16, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    for layer in range(L):
        ref = osd.decode_attention_paged_side(q[layer], oks[layer], ovs[layer], pt_np,
                                              np.asarray(lens), 1.0 / 16)
        _close(got[layer], ref)


@pytest.mark.parametrize("bits", [6, 4])
def test_decode_attn_side_stage_reuse(kvq, cuda_dev, bits):
    """2 layers x 8 sequences x 4 KV heads of up to 2,048 tokens: the split sizing gives each
    warp three or more tiles, so every stage is refilled by the copy engine while the residual
    tile of its previous tile is still in use -- the side terms must not read the stage after
    it is handed back.  Ragged lengths; every output checked against the oracle."""
    H, G, D, L, ps, k, n_sink = 4, 6, 256, 2, 16, 3, 4
    lens = [2048, 1900, 2047, 64, 2048, 1500, 1024, 2000]
    nseq = len(lens)
    starts = [0] * nseq
    kps, vps, kss, vss, oks, ovs = [], [], [], [], [], []
    pt_np = None
    for layer in range(L):
        pt_np, pools, sides, opools, osides = _setup(kvq, cuda_dev, bits, H, D, ps, k, n_sink,
                                                     lens, starts, seed=3)
        tot = int(sum(lens))
        xs = [_rows(40 + layer, True, tot, H, D), _rows(40 + layer, False, tot, H, D)]
        cu = cu_of(lens)
        kvq.kvq_quant_pack_paged_side(pools, sides, [dev_tensor(x, cuda_dev) for x in xs],
                                      i32(pt_np, cuda_dev), i32(cu, cuda_dev),
                                      i32(starts, cuda_dev))
        for x, osp in zip(xs, osides):
            osd.quant_pack_paged_side(osp, x, pt_np, cu, np.asarray(starts))
        kps.append(pools[0]); vps.append(pools[1]); kss.append(sides[0]); vss.append(sides[1])
        oks.append(osides[0]); ovs.append(osides[1])
    q = kvgen.queries_np(41, L, nseq, H * G, D)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
    ws = kvq.decode_workspace(kps, nseq, H * G, max(lens), cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_decode_attn_side(kps, vps, kss, vss, dev_tensor(q, cuda_dev), i32(pt_np, cuda_dev),
                             i32(lens, cuda_dev), max(lens), 1.0 / 16, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    for layer in range(L):
        ref = osd.decode_attention_paged_side(q[layer], oks[layer], ovs[layer], pt_np,
                                              np.asarray(lens), 1.0 / 16)
        _close(got[layer], ref)


def test_decode_attn_side_full_size_sampled(kvq, cuda_dev):
    """The bench's decode shape with side channels: 16 layers, 8 sequences x 32,768 tokens, 4 KV
    heads x 256, 24 query heads, q6, page 16, 3 outliers per row, 4 sinks; sampled (layer,
    sequence) outputs against the oracle's own quantization of those sequences."""
    w = kvgen.WORKLOADS["paged_prefill_16L_8x32768_4x256"]
    L, nseq, ntok, H, D, ps = w["n_layers"], w["n_seq"], w["n_tok"], w["H"], w["D"], w["page_size"]
    bits, k, n_sink, Hq = 6, 3, 4, 24
    pt_np = kvgen.random_page_table(1, nseq, ntok // ps)
    pt = i32(pt_np, cuda_dev)
    cu = i32(np.arange(nseq + 1) * ntok, cuda_dev)
    st = i32(np.zeros(nseq), cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kps, vps, kss, vss, specs = [], [], [], [], []
    for layer in range(L):
        sp = [kvgen.KVSpec(seed=w["seed"], layer=layer, is_key=kk, n_seq=nseq, n_tok=ntok,
                           num_heads=H, head_dim=D) for kk in (True, False)]
        pools = [kvq.Pool.empty(bits, H, D, ps, pt_np.size, cuda_dev) for _ in range(2)]
        sides = [kvq.Side.empty(p, k, n_sink, nseq, cuda_dev) for p in pools]
        xs = [s.full_torch(cuda_dev) for s in sp]
        kvq.kvq_quant_pack_paged_side(pools, sides, xs, pt, cu, st, err)
        del xs
        kps.append(pools[0]); vps.append(pools[1]); kss.append(sides[0]); vss.append(sides[1])
        specs.append(sp)
    q = kvgen.queries_torch(w["seed"], L, nseq, Hq, D, cuda_dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=cuda_dev)
    ws = kvq.decode_workspace(kps, nseq, Hq, ntok, cuda_dev)
    lens = i32(np.full(nseq, ntok), cuda_dev)
    kvq.kvq_decode_attn_side(kps, vps, kss, vss, q, pt, lens, ntok, 1.0 / 16, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    qn, got = q.cpu().numpy(), out.cpu().numpy().astype(np.float64)
    for layer, s in ((0, 0), (15, 7)):
        rows = np.arange(s * ntok * H, (s + 1) * ntok * H, dtype=np.int64)
        kx = specs[layer][0].rows_np(rows).reshape(ntok, H, D)
        vx = specs[layer][1].rows_np(rows).reshape(ntok, H, D)
        ops = [osd.SidePool(osym.PagedPool(bits, H, D, ps, ntok // ps), k, n_sink, 1)
               for _ in range(2)]
        table = np.arange(ntok // ps)[None, :]
        for x, op in zip((kx, vx), ops):
            osd.quant_pack_paged_side(op, x, table, np.array([0, ntok]), np.array([0]))
        ref = osd.decode_attention_paged_side(qn[layer, s:s + 1], ops[0], ops[1], table,
                                              np.array([ntok]), 1.0 / 16)
        _close(got[layer, s:s + 1], ref)
    del kps, vps, kss, vss
    torch.cuda.empty_cache()
