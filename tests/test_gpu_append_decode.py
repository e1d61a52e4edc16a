"""GPU parity: kvq_append_decode_attn (one decode step: quantize every sequence's new token into
its tail page and attend over the grown window, in one launch) against the oracle's decode step
(quantize-on-write, then dequantize + softmax in float64).  The appended rows are compared bit for
bit; the outputs within |gpu - ref| <= 2e-3 + 1e-3 * |ref| elementwise."""
import numpy as np
import pytest
import torch

import kvgen
from oracle import attention as oa
from oracle import symmetric as osym
from _attn_checks import assert_attn_close, decode_tiles_per_cta, needle_row, paged_needle_positions
from _gpu_util import cu_of, dev_tensor, i32

pytestmark = pytest.mark.gpu



def _close(got, ref):
    assert_attn_close(got, ref)


def _rows(seed, layer, is_key, n, H, D):
    return kvgen.KVSpec(seed=seed, layer=layer, is_key=is_key, n_seq=1, n_tok=n, num_heads=H,
                        head_dim=D).full_np()


def _check_new_rows(kp, okp, pt_np, lens, ps):
    for s, n in enumerate(lens):
        page, slot = int(pt_np[s, n // ps]), n % ps
        assert np.array_equal(kp.codes[page, :, slot].cpu().numpy(), okp.codes[page, :, slot])
        assert np.array_equal(kp.scales[page, :, slot].cpu().numpy().view(np.uint16),
                              okp.scales[page, :, slot].view(np.uint16))


@pytest.mark.parametrize("bits", [8, 6, 4])
@pytest.mark.parametrize("ps", [16, 32])
def test_decode_steps_ragged(kvq, cuda_dev, bits, ps):
    """Three decode steps over 2 layers and 7 sequences of ragged lengths (empty, page
    boundaries, one past a boundary, long); GQA 6:1."""
    L, H, G, D, steps = 2, 4, 6, 256, 3
    lens = np.array([0, 15, 16, 31, 100, 257, 1000])
    nseq = len(lens)
    pps = (int(lens.max()) + steps + ps - 1) // ps
    pt_np = kvgen.random_page_table(7, nseq, pps)
    pt = i32(pt_np, cuda_dev)
    n_pages = pt_np.size
    tot = int(lens.sum())
    kps, vps, okps, ovps = [], [], [], []
    for l in range(L):
        k, v = _rows(5, l, True, tot, H, D), _rows(5, l, False, tot, H, D)
        kp = kvq.Pool.empty(bits, H, D, ps, n_pages, cuda_dev)
        vp = kvq.Pool.empty(bits, H, D, ps, n_pages, cuda_dev)
        kvq.kvq_quant_pack_paged([kp, vp], [dev_tensor(k, cuda_dev), dev_tensor(v, cuda_dev)], pt,
                                 i32(cu_of(lens), cuda_dev), i32(np.zeros(nseq), cuda_dev))
        okp, ovp = osym.PagedPool(bits, H, D, ps, n_pages), osym.PagedPool(bits, H, D, ps, n_pages)
        osym.quant_pack_paged(okp, k, pt_np, cu_of(lens), np.zeros(nseq))
        osym.quant_pack_paged(ovp, v, pt_np, cu_of(lens), np.zeros(nseq))
        kps.append(kp); vps.append(vp); okps.append(okp); ovps.append(ovp)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    for step in range(steps):
        max_len = int(lens.max()) + 1
        kn = [_rows(100 + step, l, True, nseq, H, D) for l in range(L)]
        vn = [_rows(100 + step, l, False, nseq, H, D) for l in range(L)]
        q = kvgen.queries_np(200 + step, L, nseq, H * G, D)
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
        ws = kvq.decode_workspace(kps, nseq, H * G, max_len, cuda_dev)
        kvq.kvq_append_decode_attn(kps, vps, [dev_tensor(x, cuda_dev) for x in kn],
                                   [dev_tensor(x, cuda_dev) for x in vn], dev_tensor(q, cuda_dev),
                                   pt, i32(lens, cuda_dev), max_len, 1.0 / 16, out, ws, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.cpu().numpy().astype(np.float64)
        for l in range(L):
            ref = oa.append_decode_paged(q[l], okps[l], ovps[l], kn[l], vn[l], pt_np, lens,
                                         1.0 / 16)
            _close(got[l], ref)
            _check_new_rows(kps[l], okps[l], pt_np, lens, ps)
            _check_new_rows(vps[l], ovps[l], pt_np, lens, ps)
        lens = lens + 1


def test_unmapped_tail_page_is_reported_and_not_written(kvq, cuda_dev):
    """A sequence whose tail page id is out of the pool's range: the kernel's page check skips
    the tile (no write, no read) and sets KVQ_DEVERR_PAGE_RANGE; the other sequences are exact."""
    bits, H, G, D, ps = 6, 2, 2, 256, 16
    lens = np.array([20, 40])
    pt_np = np.array([[0, 1, 2], [3, 4, 5]], dtype=np.int32)
    n_pages = 6
    tot = int(lens.sum())
    k, v = _rows(6, 0, True, tot, H, D), _rows(6, 0, False, tot, H, D)
    kp = kvq.Pool.empty(bits, H, D, ps, n_pages, cuda_dev)
    vp = kvq.Pool.empty(bits, H, D, ps, n_pages, cuda_dev)
    kvq.kvq_quant_pack_paged([kp, vp], [dev_tensor(k, cuda_dev), dev_tensor(v, cuda_dev)],
                             i32(pt_np, cuda_dev), i32(cu_of(lens), cuda_dev),
                             i32(np.zeros(2), cuda_dev))
    okp, ovp = osym.PagedPool(bits, H, D, ps, n_pages), osym.PagedPool(bits, H, D, ps, n_pages)
    osym.quant_pack_paged(okp, k, pt_np, cu_of(lens), np.zeros(2))
    osym.quant_pack_paged(ovp, v, pt_np, cu_of(lens), np.zeros(2))
    bad_pt = pt_np.copy()
    bad_pt[1, 2] = 1000                     # position 40 of sequence 1 maps nowhere
    before = kp.codes.clone()
    kn, vn = _rows(7, 0, True, 2, H, D), _rows(7, 0, False, 2, H, D)
    q = kvgen.queries_np(8, 1, 2, H * G, D)
    out = torch.zeros(q.shape, dtype=torch.float32, device=cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    ws = kvq.decode_workspace([kp], 2, H * G, 41, cuda_dev)
    kvq.kvq_append_decode_attn([kp], [vp], [dev_tensor(kn, cuda_dev)], [dev_tensor(vn, cuda_dev)],
                               dev_tensor(q, cuda_dev), i32(bad_pt, cuda_dev), i32(lens, cuda_dev),
                               41, 1.0 / 16, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) & 1
    ref = oa.append_decode_paged(q[0, :1], okp, ovp, kn[:1], vn[:1], pt_np[:1], lens[:1], 1.0 / 16)
    _close(out.cpu().numpy()[0, :1].astype(np.float64), ref)
    after = kp.codes.cpu().numpy()
    changed = np.any(after != before.cpu().numpy(), axis=(1, 2, 3))
    assert list(np.nonzero(changed)[0]) == [int(pt_np[0, 1])]   # only sequence 0's tail page


def test_decode_step_64_ragged_sequences_full_size_sampled(kvq, cuda_dev):
    """The decode step of 64 sequences with lengths uniform in [1024, 65536], 16 layers, 4 KV
    heads x 256, 24 query heads, q6, page 16: the cache pages hold seeded random codes and
    scales; every appended row of sampled layers is checked bit for bit and the outputs of
    sampled (layer, sequence) pairs against the oracle's decode step on the same cache bytes."""
    w = kvgen.WORKLOADS["decode_append_16L_64seq_4x256"]
    L, nseq, H, D, ps, bits, Hq = w["n_layers"], w["n_seq"], w["H"], w["D"], w["page_size"], 6, 24
    lens = kvgen.decode_append_lengths(w["seed"], nseq).astype(np.int64)
    pages_per_seq = (lens + 1 + ps - 1) // ps
    max_pages = int(pages_per_seq.max())
    perm = kvgen.permutation(w["seed"], 77, int(pages_per_seq.sum()))
    pt_np = np.full((nseq, max_pages), -1, dtype=np.int32)
    o = 0
    for s in range(nseq):
        pt_np[s, :pages_per_seq[s]] = perm[o:o + pages_per_seq[s]]
        o += pages_per_seq[s]
    n_pages = int(pages_per_seq.sum())
    pt = i32(pt_np, cuda_dev)
    kps, vps = [], []
    for l in range(L):
        kp = kvq.Pool.empty(bits, H, D, ps, n_pages, cuda_dev)
        vp = kvq.Pool.empty(bits, H, D, ps, n_pages, cuda_dev)
        kvgen.fill_random_pool_(kp.codes, kp.scales, 1000 + 2 * l)
        kvgen.fill_random_pool_(vp.codes, vp.scales, 1001 + 2 * l)
        kps.append(kp); vps.append(vp)
    samples = [(0, int(np.argmin(lens))), (9, 17), (15, int(np.argmax(lens)))]
    # needles: in the sampled sequences the cached keys of the group's first query head are
    # replaced, at the tiles a schedule gets wrong, by the oracle's packed form of a key row along
    # that query's direction, so a lost or misplaced tile moves the output outside the tolerance
    qn = kvgen.queries_np(w["seed"], L, nseq, Hq, D)
    tpc = decode_tiles_per_cta(L, nseq, H, int(lens.max()) + 1,
                               torch.cuda.get_device_properties(cuda_dev).multi_processor_count)
    G = Hq // H
    for l, s in samples:
        for h in range(H):
            codes, sc = osym.quant_pack_rows(needle_row(qn[l, s, h * G], 1.0 / 16)[None], bits)
            for t in paged_needle_positions(int(lens[s]), tpc, stages=2):
                page, slot = int(pt_np[s, t // ps]), t % ps
                kps[l].codes[page, h, slot] = torch.from_numpy(codes[0]).to(cuda_dev)
                kps[l].scales[page, h, slot] = float(sc[0])
    host = {}
    for l, s in samples:   # the sampled sequences' cache bytes, taken before the step
        pages = torch.from_numpy(pt_np[s, :pages_per_seq[s]].astype(np.int64)).to(cuda_dev)
        pools = []
        for p in (kps[l], vps[l]):
            op = osym.PagedPool(bits, H, D, ps, int(pages_per_seq[s]))
            op.codes[:] = p.codes[pages].cpu().numpy()
            op.scales[:] = p.scales[pages].cpu().numpy()
            pools.append(op)
        host[(l, s)] = pools
    kn = [kvgen.KVSpec(seed=w["seed"], layer=l, is_key=True, n_seq=1, n_tok=nseq, num_heads=H,
                       head_dim=D).full_torch(cuda_dev) for l in range(L)]
    vn = [kvgen.KVSpec(seed=w["seed"], layer=l, is_key=False, n_seq=1, n_tok=nseq, num_heads=H,
                       head_dim=D).full_torch(cuda_dev) for l in range(L)]
    q = dev_tensor(qn, cuda_dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=cuda_dev)
    max_len = int(lens.max()) + 1
    ws = kvq.decode_workspace(kps, nseq, Hq, max_len, cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_append_decode_attn(kps, vps, kn, vn, q, pt, i32(lens, cuda_dev), max_len, 1.0 / 16,
                               out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for l in (0, 7, 15):
        for pool, new in ((kps[l], kn[l]), (vps[l], vn[l])):
            packed, scale = osym.quant_pack_rows(new.cpu().numpy(), bits)
            page = torch.from_numpy(pt_np[np.arange(nseq), lens // ps].astype(np.int64))
            slot = torch.from_numpy(lens % ps)
            got_c = pool.codes[page.to(cuda_dev), :, slot.to(cuda_dev)].cpu().numpy()
            got_s = pool.scales[page.to(cuda_dev), :, slot.to(cuda_dev)].cpu().numpy()
            assert np.array_equal(got_c, packed)
            assert np.array_equal(got_s.view(np.uint16), scale.view(np.uint16))
    got = out.cpu().numpy().astype(np.float64)
    for (l, s), (okp, ovp) in host.items():
        table = np.arange(int(pages_per_seq[s]))[None, :]
        ref = oa.append_decode_paged(qn[l, s:s + 1], okp, ovp, kn[l][s:s + 1].cpu().numpy(),
                                     vn[l][s:s + 1].cpu().numpy(), table, lens[s:s + 1], 1.0 / 16)
        _close(got[l, s:s + 1], ref)
    del kps, vps
    torch.cuda.empty_cache()
