"""GPU parity: kvq_quant_pack_paged and kvq_dequant_paged against the oracle, bit for bit.

Codes, scales and dequantized fp16 must be identical (the arithmetic is fixed: IEEE float32
divide, round-half-even, fp16 rounding).  Small cases span several tiles, ragged tails and the
degenerate rows; the full-size prefill and decode-append workloads run in the launch
configuration the benchmark times, checked on sampled rows (and on every appended row).  The
full-size prefill test also runs kvq_decode_attn over the pools it wrote, in the benchmark's
decode launch, against the oracle's attention on sampled (layer, sequence, head) triples.
"""
import numpy as np
import pytest
import torch

import kvgen
from oracle import attention as oa
from oracle import symmetric as osym
from _attn_checks import (Planted, assert_attn_close, decode_tiles_per_cta, needle_row,
                          paged_needle_positions, plant_needles)
from _gpu_util import (check_rows_against_oracle, cu_of, dev_tensor, i32, random_rows, u16)

pytestmark = pytest.mark.gpu


def _run(kvq, dev, x_list, bits, H, D, ps, lens, start, pt_np, n_pages, err=None):
    pools = [kvq.Pool.empty(bits, H, D, ps, n_pages, dev) for _ in x_list]
    for p in pools:
        p.codes.fill_(0xAB)
        p.scales.fill_(7.0)
    xs = [dev_tensor(x, dev) for x in x_list]
    pt = i32(pt_np, dev)
    cu = i32(cu_of(lens), dev)
    st = i32(start, dev)
    kvq.kvq_quant_pack_paged(pools, xs, pt, cu, st, err)
    outs = [torch.full_like(x, 12345) for x in xs]
    kvq.kvq_dequant_paged(pools, outs, pt, cu, st, err)
    torch.cuda.synchronize()
    return pools, outs


def _oracle(x_list, bits, H, D, ps, lens, start, pt_np, n_pages):
    res = []
    for x in x_list:
        p = osym.PagedPool(bits, H, D, ps, n_pages)
        p.codes[:] = 0xAB
        p.scales[:] = 7.0
        osym.quant_pack_paged(p, x, pt_np, cu_of(lens), np.asarray(start))
        res.append((p, osym.dequant_paged(p, pt_np, cu_of(lens), np.asarray(start))))
    return res


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_contiguous_roundtrip_one_layer(kvq, cuda_dev, bits):
    """q6 round-trip workload (and q8/q4): K, V [1 seq, 1024 tokens, 4 heads, 256], contiguous
    layout = one page of 1024 tokens with an identity table."""
    w = kvgen.WORKLOADS["q6_roundtrip_1x1024x4x256"]
    T, H, D = w["n_tok"], w["H"], w["D"]
    k = kvgen.KVSpec(seed=w["seed"], layer=0, is_key=True, n_seq=1, n_tok=T, num_heads=H,
                     head_dim=D).full_np()
    v = kvgen.KVSpec(seed=w["seed"], layer=0, is_key=False, n_seq=1, n_tok=T, num_heads=H,
                     head_dim=D).full_np()
    pt = np.zeros((1, 1), np.int32)
    pools, outs = _run(kvq, cuda_dev, [k, v], bits, H, D, T, [T], [0], pt, 1)
    ref = _oracle([k, v], bits, H, D, T, [T], [0], pt, 1)
    for (op, od), p, o in zip(ref, pools, outs):
        assert np.array_equal(p.codes.cpu().numpy(), op.codes)
        assert np.array_equal(u16(p.scales), op.scales.view(np.uint16))
        assert np.array_equal(u16(o), od.view(np.uint16))
    # the two all-zero rows store scale 0 and codes equal to the bias
    assert float(pools[0].scales[0, 0, 0]) == 0.0
    assert float(pools[1].scales[0, H - 1, T - 1]) == 0.0


@pytest.mark.parametrize("bits", [8, 6, 4])
@pytest.mark.parametrize("D", [16, 48, 64, 80, 96, 128, 192, 256])
def test_edge_rows_all_head_dims(kvq, cuda_dev, bits, D):
    """Magnitudes from fp16-subnormal scales to 2^11, outliers, zero rows, exact ties; ragged
    sequence lengths (0, 1, page-1, page, page+1, many pages) over a random page table; head
    dims whose rows take 1 to 16 units of 16 elements."""
    H, ps = 3, 16
    lens = [0, 1, 15, 16, 17, 100, 0, 333]
    pps = max((n + ps - 1) // ps for n in lens)
    pt = kvgen.random_page_table(5, len(lens), pps)
    x = random_rows(int(sum(lens)) * H, D, 11 + D).reshape(-1, H, D)
    pools, outs = _run(kvq, cuda_dev, [x], bits, H, D, ps, lens, [0] * len(lens), pt, pt.size)
    (op, od), = _oracle([x], bits, H, D, ps, lens, [0] * len(lens), pt, pt.size)
    assert np.array_equal(pools[0].codes.cpu().numpy(), op.codes)
    assert np.array_equal(u16(pools[0].scales), op.scales.view(np.uint16))
    assert np.array_equal(u16(outs[0]), od.view(np.uint16))


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_append_at_offsets_keeps_other_slots(kvq, cuda_dev, bits):
    """Appends at nonzero positions write only their own slots of the partially filled pages."""
    H, D, ps = 4, 256, 16
    start = [5, 16, 31, 0, 100]
    lens = [3, 1, 34, 0, 16]
    pps = (max(s + n for s, n in zip(start, lens)) + ps - 1) // ps
    pt = kvgen.random_page_table(6, len(lens), pps)
    x = random_rows(int(sum(lens)) * H, D, 21).reshape(-1, H, D)
    pools, outs = _run(kvq, cuda_dev, [x], bits, H, D, ps, lens, start, pt, pt.size)
    (op, od), = _oracle([x], bits, H, D, ps, lens, start, pt, pt.size)
    assert np.array_equal(pools[0].codes.cpu().numpy(), op.codes)   # untouched slots stay 0xAB
    assert np.array_equal(u16(pools[0].scales), op.scales.view(np.uint16))
    assert np.array_equal(u16(outs[0]), od.view(np.uint16))


def test_out_of_range_page_ids_are_skipped_and_reported(kvq, cuda_dev):
    H, D, ps, bits = 2, 64, 4, 6
    lens = [8, 8]
    pt = np.array([[0, 1], [2, 99]], np.int32)        # 99 >= num_pages = 3
    x = random_rows(16 * H, D, 31).reshape(-1, H, D)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    pools, outs = _run(kvq, cuda_dev, [x], bits, H, D, ps, lens, [0, 0], pt, 3, err)
    assert int(err.item()) == kvq.KVQ_DEVERR_PAGE_RANGE
    good = pt.copy()
    good[1, 1] = -1                                       # oracle: never touch the bad page
    p = osym.PagedPool(bits, H, D, ps, 3)
    p.codes[:] = 0xAB
    p.scales[:] = 7.0
    osym.quant_pack_paged(p, x[:12], good[:, :], cu_of([8, 4]), np.array([0, 0]))
    assert np.array_equal(pools[0].codes.cpu().numpy(), p.codes)
    out = outs[0].cpu().numpy()
    assert np.all(out[12:].view(np.uint16) == np.float16(12345).view(np.uint16))


def test_multi_tensor_call_and_determinism(kvq, cuda_dev):
    H, D, ps, bits = 4, 256, 16, 6
    lens = [40, 7]
    pt = kvgen.random_page_table(7, 2, 3)
    xs = [random_rows(47 * H, D, 40 + i).reshape(-1, H, D) for i in range(5)]
    a, _ = _run(kvq, cuda_dev, xs, bits, H, D, ps, lens, [0, 0], pt, pt.size)
    b, _ = _run(kvq, cuda_dev, xs, bits, H, D, ps, lens, [0, 0], pt, pt.size)
    ref = _oracle(xs, bits, H, D, ps, lens, [0, 0], pt, pt.size)
    for p, q, (op, _) in zip(a, b, ref):
        assert torch.equal(p.codes, q.codes) and torch.equal(p.scales, q.scales)
        assert np.array_equal(p.codes.cpu().numpy(), op.codes)


def test_zero_tokens_is_a_no_op(kvq, cuda_dev):
    H, D, ps = 4, 256, 16
    pool = kvq.Pool.empty(6, H, D, ps, 2, cuda_dev)
    pool.codes.fill_(1)
    x = torch.empty((0, H, D), dtype=torch.float16, device=cuda_dev)
    pt = i32([[0]], cuda_dev)
    kvq.kvq_quant_pack_paged([pool], [x], pt, i32([0, 0], cuda_dev), i32([0], cuda_dev))
    torch.cuda.synchronize()
    assert int(pool.codes.min()) == 1 and int(pool.codes.max()) == 1


# ------------------------------------------------------------------------ full-size workloads
# (layer, sequence, KV head) triples whose keys carry needles for the group's first query head,
# and whose decode outputs are checked against the oracle
NEEDLE_TRIPLES = [(0, 0, 0), (15, 7, 3), (7, 3, 2)]


@pytest.fixture(scope="module")
def prefill_inputs(cuda_dev):
    """The paged-prefill inputs, with needles planted in the keys of NEEDLE_TRIPLES at the tiles a
    decode schedule gets wrong (first/last tile, both sides of a split boundary, deep in a warp's
    stream, the middle split, the last token)."""
    w = kvgen.WORKLOADS["paged_prefill_16L_8x32768_4x256"]
    L, nseq, ntok, H, D = w["n_layers"], w["n_seq"], w["n_tok"], w["H"], w["D"]
    qn = kvgen.queries_np(w["seed"], L, nseq, 24, D)
    tpc = decode_tiles_per_cta(L, nseq, H, ntok,
                               torch.cuda.get_device_properties(cuda_dev).multi_processor_count)
    pos = paged_needle_positions(ntok, tpc, stages=2)
    specs, xs = [], []
    for layer in range(L):
        for is_key in (True, False):
            s = Planted(kvgen.KVSpec(seed=w["seed"], layer=layer, is_key=is_key, n_seq=nseq,
                                     n_tok=ntok, num_heads=H, head_dim=D))
            if is_key:
                for tl, ts, th in NEEDLE_TRIPLES:
                    if tl == layer:
                        plant_needles(s, ts, th, pos, needle_row(qn[layer, ts, th * (24 // H)],
                                                                 1.0 / 16.0))
            specs.append(s)
            xs.append(s.full_torch(cuda_dev))
    pt_np = kvgen.random_page_table(1, w["n_seq"], w["n_tok"] // w["page_size"])
    yield w, specs, xs, pt_np
    del xs
    torch.cuda.empty_cache()


def _decode_on_prefill_pools(kvq, dev, w, specs, pools, pt, bits):
    """kvq_decode_attn over the 16 packed layers, 8 sequences x 32,768 tokens, 24 query heads
    (GQA 6:1), softmax scale 1/16 -- the decode launch the benchmark times on these pools --
    against the oracle for sampled (layer, sequence, KV head) triples, within the decode
    tolerance |got - ref| <= 2e-3 + 1e-3 |ref|; every output must be finite."""
    H, D, nseq, ntok, L = w["H"], w["D"], w["n_seq"], w["n_tok"], w["n_layers"]
    hq, G, scale = 24, 24 // w["H"], 1.0 / 16.0
    q = kvgen.queries_torch(w["seed"], L, nseq, hq, D, dev)
    out = torch.full((L, nseq, hq, D), float("nan"), dtype=torch.float32, device=dev)
    ws = kvq.decode_workspace(pools[0::2], nseq, hq, ntok, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kvq.kvq_decode_attn(pools[0::2], pools[1::2], q, pt, i32([ntok] * nseq, dev), ntok, scale,
                        out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(got))
    qn = q.cpu().numpy()
    rng = np.random.default_rng(100 + bits)
    triples = list(NEEDLE_TRIPLES) + [
        (int(rng.integers(L)), int(rng.integers(nseq)), int(rng.integers(H))) for _ in range(2)]
    for layer, s, h in triples:
        rows = (s * ntok + np.arange(ntok, dtype=np.int64)) * H + h
        ks, vs = specs[2 * layer], specs[2 * layer + 1]
        k_hat = osym.dequant_rows(*osym.quant_pack_rows(ks.rows_np(rows), bits), bits, D)
        v_hat = osym.dequant_rows(*osym.quant_pack_rows(vs.rows_np(rows), bits), bits, D)
        ref = oa.attend(qn[layer, s, h * G:(h + 1) * G], k_hat[:, None, :], v_hat[:, None, :],
                        scale)
        assert_attn_close(got[layer, s, h * G:(h + 1) * G], ref, f"layer {layer} seq {s} head {h}")
    del out, ws


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_paged_prefill_full_size_sampled(kvq, cuda_dev, prefill_inputs, bits):
    """16 layers x {K,V} x 8 seqs x 32,768 tokens x 4 heads x 256, page 16, random table: one
    quant-pack call over all 32 tensors (the benchmark's launch), then one dequant call; 512
    sampled rows per tensor checked bit for bit, plus the first and last row of every sequence."""
    w, specs, xs, pt_np = prefill_inputs
    H, D, ps, nseq, ntok = w["H"], w["D"], w["page_size"], w["n_seq"], w["n_tok"]
    n_pages = pt_np.size
    pools = [kvq.Pool.empty(bits, H, D, ps, n_pages, cuda_dev) for _ in xs]
    pt = i32(pt_np, cuda_dev)
    cu = i32(cu_of([ntok] * nseq), cuda_dev)
    st = i32([0] * nseq, cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_quant_pack_paged(pools, xs, pt, cu, st, err)
    torch.cuda.synchronize()
    rng = np.random.default_rng(bits)
    n_rows = nseq * ntok * H
    edge = np.concatenate([[(s * ntok) * H, (s * ntok + ntok - 1) * H + H - 1]
                           for s in range(nseq)])
    for i, (spec, pool) in enumerate(zip(specs, pools)):
        rows = np.unique(np.concatenate([rng.integers(0, n_rows, 512), edge]))
        tok, head = rows // H, rows % H
        seq, pos = tok // ntok, tok % ntok
        check_rows_against_oracle(pool, spec.rows_np(rows), pt_np, seq, pos, head, bits)
    _decode_on_prefill_pools(kvq, cuda_dev, w, specs, pools, pt, bits)
    # dequant back (chunked in pairs of tensors to bound memory) and compare the sampled rows
    for i0 in range(0, len(xs), 8):
        outs = [torch.empty_like(xs[i]) for i in range(i0, i0 + 8)]
        kvq.kvq_dequant_paged(pools[i0:i0 + 8], outs, pt, cu, st, err)
        torch.cuda.synchronize()
        for j, out in enumerate(outs):
            spec = specs[i0 + j]
            rows = np.unique(rng.integers(0, n_rows, 256))
            ref = osym.dequant_rows(*osym.quant_pack_rows(spec.rows_np(rows), bits), bits, D)
            got = out.view(-1, D)[torch.from_numpy(rows).to(cuda_dev)].cpu().numpy()
            assert np.array_equal(got.view(np.uint16), ref.view(np.uint16))
        del outs
    assert int(err.item()) == 0
    del pools
    torch.cuda.empty_cache()


@pytest.mark.parametrize("n_new", [1, 8, 32])
def test_decode_append_full_size(kvq, cuda_dev, n_new):
    """64 sequences with cached lengths U[1024, 65536], each appends n_new tokens per layer across
    16 layers x {K,V}, into partially filled tail pages mapped by the host allocator.  Every
    appended row is checked; the slots before each append keep their prior bytes."""
    w = kvgen.WORKLOADS["decode_append_16L_64seq_4x256"]
    H, D, ps, nseq, L = w["H"], w["D"], w["page_size"], w["n_seq"], w["n_layers"]
    cur = kvgen.decode_append_lengths(w["seed"], nseq)
    max_pages = (int(cur.max()) + n_new + ps - 1) // ps
    table = torch.full((nseq, max_pages), -1, dtype=torch.int32)
    alloc = kvq.Allocator(nseq * 3)
    alloc.reserve(table, ps, cur, [n_new] * nseq)
    n_pages = nseq * 3
    pt_np = table.numpy().copy()
    pools, xs, specs = [], [], []
    for layer in range(L):
        for is_key in (True, False):
            s = kvgen.KVSpec(seed=w["seed"], layer=layer, is_key=is_key, n_seq=nseq,
                             n_tok=n_new, num_heads=H, head_dim=D, zero_rows=False)
            specs.append(s)
            xs.append(s.full_torch(cuda_dev))
            p = kvq.Pool.empty(6, H, D, ps, n_pages, cuda_dev)
            p.codes.fill_(0x5A)
            p.scales.fill_(3.0)
            pools.append(p)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_quant_pack_paged(pools, xs, i32(pt_np, cuda_dev), i32(cu_of([n_new] * nseq), cuda_dev),
                             i32(cur, cuda_dev), err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for spec, pool in zip(specs, pools):
        x = spec.full_np()
        p = osym.PagedPool(6, H, D, ps, n_pages)
        p.codes[:] = 0x5A
        p.scales[:] = 3.0
        osym.quant_pack_paged(p, x, pt_np, cu_of([n_new] * nseq), cur)
        assert np.array_equal(pool.codes.cpu().numpy(), p.codes)
        assert np.array_equal(u16(pool.scales), p.scales.view(np.uint16))


@pytest.mark.parametrize("bits", [8, 6, 4])
@pytest.mark.parametrize("D", [64, 256])
def test_tensors_aligned_to_16_but_not_32_bytes(kvq, cuda_dev, bits, D):
    """fp16 rows move in 256-bit accesses only when every tensor of a call is 32-byte aligned;
    tensors that are 16-byte aligned (what the API requires) take the 128-bit path.  Both must
    give the oracle's bytes and values: here K is 32-byte aligned and V is offset by 16 bytes in
    one call (the narrow path for both), then each alone."""
    H, ps = 3, 16
    lens, start = [5, 33, 17], [0, 3, 16]
    pps = (max(s + n for s, n in zip(start, lens)) + ps - 1) // ps
    pt = kvgen.random_page_table(90 + D, len(lens), pps)
    tot = int(sum(lens))
    x = [random_rows(tot * H, D, 91 + i).reshape(tot, H, D) for i in range(2)]

    def offset_view(a, elems):
        flat = torch.empty(a.size + 64, dtype=torch.float16, device=cuda_dev)
        v = flat[elems:elems + a.size].view(a.shape)
        v.copy_(torch.from_numpy(np.ascontiguousarray(a)).to(cuda_dev))
        return v

    ref = _oracle(x, bits, H, D, ps, lens, start, pt, pt.size)
    args = (i32(pt, cuda_dev), i32(cu_of(lens), cuda_dev), i32(start, cuda_dev))
    for offs in ((16, 8), (8, 8), (16, 16)):   # fp16 elements: 32 and 16 bytes
        xs = [offset_view(a, o) for a, o in zip(x, offs)]
        assert [t.data_ptr() % 32 for t in xs] == [2 * o % 32 for o in offs]
        pools = [kvq.Pool.empty(bits, H, D, ps, pt.size, cuda_dev) for _ in x]
        for p in pools:
            p.codes.fill_(0xAB)
            p.scales.fill_(7.0)
        kvq.kvq_quant_pack_paged(pools, xs, *args)
        outs = [offset_view(np.full(a.shape, np.float16(12345)), o) for a, o in zip(x, offs)]
        kvq.kvq_dequant_paged(pools, outs, *args)
        torch.cuda.synchronize()
        for (op, od), p, o in zip(ref, pools, outs):
            assert np.array_equal(p.codes.cpu().numpy(), op.codes)
            assert np.array_equal(u16(p.scales), op.scales.view(np.uint16))
            assert np.array_equal(u16(o), od.view(np.uint16))
