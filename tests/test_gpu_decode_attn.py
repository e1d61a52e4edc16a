"""GPU parity: kvq_decode_attn (reads packed pages) against the oracle's dequantize-then-softmax
attention in float64.  Tolerance: |gpu - ref| <= 2e-3 + 1e-3 * |ref| elementwise (float32
accumulation; the kernel multiplies the exact integer codes and applies each token's fp16 scale to
the scores (K) and to P (V), where the oracle rounds k_hat, v_hat to fp16 -- at most half an fp16
ulp apart; P times the V scale is rounded to fp16 for the tensor-core product)."""
import numpy as np
import pytest
import torch

import kvgen
from oracle import attention as oa
from oracle import symmetric as osym
from _attn_checks import (Planted, assert_attn_close, decode_tiles_per_cta, needle_row,
                          paged_needle_positions)
from _gpu_util import cu_of, dev_tensor, i32

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-3


def _build_cache(kvq, dev, bits, H, D, ps, lens, pt_np, k_np, v_np):
    n_pages = pt_np.size
    kp = kvq.Pool.empty(bits, H, D, ps, n_pages, dev)
    vp = kvq.Pool.empty(bits, H, D, ps, n_pages, dev)
    cu = i32(cu_of(lens), dev)
    st = i32([0] * len(lens), dev)
    pt = i32(pt_np, dev)
    kvq.kvq_quant_pack_paged([kp, vp], [dev_tensor(k_np, dev), dev_tensor(v_np, dev)], pt, cu, st)
    okp, ovp = osym.PagedPool(bits, H, D, ps, n_pages), osym.PagedPool(bits, H, D, ps, n_pages)
    osym.quant_pack_paged(okp, k_np, pt_np, cu_of(lens), np.zeros(len(lens)))
    osym.quant_pack_paged(ovp, v_np, pt_np, cu_of(lens), np.zeros(len(lens)))
    return kp, vp, okp, ovp, pt


def _attend(kvq, dev, kps, vps, q, pt, lens, scale):
    L, nseq, hq, D = q.shape
    out = torch.full((L, nseq, hq, D), float("nan"), dtype=torch.float32, device=dev)
    ws = kvq.decode_workspace(kps, nseq, hq, int(max(lens)), dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kvq.kvq_decode_attn(kps, vps, q, pt, i32(lens, dev), int(max(lens)), scale, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.cpu().numpy().astype(np.float64)


def _close(got, ref):
    assert_attn_close(got, ref)


@pytest.mark.parametrize("bits", [8, 6, 4])
@pytest.mark.parametrize("H,G", [(1, 1), (4, 6), (2, 8)])
def test_small_caches(kvq, cuda_dev, bits, H, G):
    D, ps = 256, 16
    lens = [1, 15, 16, 17, 100, 1000, 0]
    pps = max((n + ps - 1) // ps for n in lens)
    pt_np = kvgen.random_page_table(9, len(lens), pps)
    tot = int(sum(lens))
    k = kvgen.KVSpec(seed=4, layer=0, is_key=True, n_seq=1, n_tok=tot, num_heads=H,
                     head_dim=D).full_np()
    v = kvgen.KVSpec(seed=4, layer=0, is_key=False, n_seq=1, n_tok=tot, num_heads=H,
                     head_dim=D).full_np()
    kp, vp, okp, ovp, pt = _build_cache(kvq, cuda_dev, bits, H, D, ps, lens, pt_np, k, v)
    q = kvgen.queries_np(5, 1, len(lens), H * G, D)
    got = _attend(kvq, cuda_dev, [kp], [vp], dev_tensor(q, cuda_dev), pt, lens, 1 / 16)
    ref = oa.decode_attention_paged(q[0], okp, ovp, pt_np, np.array(lens), 1 / 16)
    _close(got[0], ref)
    assert np.all(got[0, len(lens) - 1] == 0)     # empty sequence


@pytest.mark.parametrize("ps", [1, 7, 32, 64])
def test_other_page_sizes(kvq, cuda_dev, ps):
    """Page sizes that are multiples of 16 stream pages through the bulk-copy ring; others
    gather rows one by one."""
    bits, H, G, D = 6, 2, 3, 256
    lens = [5, 130]
    pps = max((n + ps - 1) // ps for n in lens)
    pt_np = kvgen.random_page_table(10, len(lens), pps)
    tot = int(sum(lens))
    k = kvgen.KVSpec(seed=6, layer=1, is_key=True, n_seq=1, n_tok=tot, num_heads=H,
                     head_dim=D).full_np()
    v = kvgen.KVSpec(seed=6, layer=1, is_key=False, n_seq=1, n_tok=tot, num_heads=H,
                     head_dim=D).full_np()
    kp, vp, okp, ovp, pt = _build_cache(kvq, cuda_dev, bits, H, D, ps, lens, pt_np, k, v)
    q = kvgen.queries_np(7, 1, len(lens), H * G, D)
    got = _attend(kvq, cuda_dev, [kp], [vp], dev_tensor(q, cuda_dev), pt, lens, 0.0625)
    _close(got[0], oa.decode_attention_paged(q[0], okp, ovp, pt_np, np.array(lens), 0.0625))


def test_special_cases(kvq, cuda_dev):
    """Equal keys give the mean of v_hat; a single token gives v_hat itself."""
    bits, H, G, D, ps = 6, 1, 6, 256, 16
    T = 300
    k = np.repeat(kvgen.KVSpec(seed=8, layer=0, is_key=True, n_seq=1, n_tok=1, num_heads=H,
                               head_dim=D, zero_rows=False).full_np(), T, axis=0)
    v = kvgen.KVSpec(seed=8, layer=0, is_key=False, n_seq=1, n_tok=T, num_heads=H,
                     head_dim=D, zero_rows=False).full_np()
    lens = [T, 1]
    k2 = np.concatenate([k, k[:1]])
    v2 = np.concatenate([v, v[:1]])
    pt_np = kvgen.random_page_table(11, 2, (T + ps - 1) // ps)
    kp, vp, okp, ovp, pt = _build_cache(kvq, cuda_dev, bits, H, D, ps, lens, pt_np, k2, v2)
    q = kvgen.queries_np(12, 1, 2, H * G, D)
    got = _attend(kvq, cuda_dev, [kp], [vp], dev_tensor(q, cuda_dev), pt, lens, 1 / 16)
    vs, vc = osym.quantize_rows(v, bits)
    vhat = osym.dequantize_rows(vc, vs).astype(np.float64)
    # one token: p = 1, and the kernel multiplies the integer codes by P times the token's V scale,
    # so the output is the exact product code x scale -- the oracle's v_hat is that product
    # rounded to fp16, at most half an fp16 ulp away
    exact = vc[0, 0].astype(np.float64) * vs[0, 0].astype(np.float64)
    half_ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(vhat[0, 0]), 2 ** -14))) - 11)
    for j in range(G):
        assert np.allclose(got[0, 0, j], vhat[:, 0].mean(0), rtol=RTOL, atol=ATOL)
        assert np.array_equal(got[0, 1, j], exact)
        assert np.all(np.abs(got[0, 1, j] - vhat[0, 0]) <= half_ulp)


def test_multi_layer_call(kvq, cuda_dev):
    bits, H, G, D, ps, L = 4, 2, 6, 256, 16, 3
    lens = [77, 200]
    pt_np = kvgen.random_page_table(13, 2, 13)
    tot = int(sum(lens))
    kps, vps, refs = [], [], []
    q = kvgen.queries_np(14, L, 2, H * G, D)
    for layer in range(L):
        k = kvgen.KVSpec(seed=15, layer=layer, is_key=True, n_seq=1, n_tok=tot, num_heads=H,
                         head_dim=D).full_np()
        v = kvgen.KVSpec(seed=15, layer=layer, is_key=False, n_seq=1, n_tok=tot, num_heads=H,
                         head_dim=D).full_np()
        kp, vp, okp, ovp, pt = _build_cache(kvq, cuda_dev, bits, H, D, ps, lens, pt_np, k, v)
        kps.append(kp)
        vps.append(vp)
        refs.append(oa.decode_attention_paged(q[layer], okp, ovp, pt_np, np.array(lens), 0.0625))
    got = _attend(kvq, cuda_dev, kps, vps, dev_tensor(q, cuda_dev), pt, lens, 0.0625)
    for layer in range(L):
        _close(got[layer], refs[layer])


@pytest.mark.parametrize("bits", [6, 8, 4])
def test_full_context_262144_sampled(kvq, cuda_dev, bits):
    """The full-context workload: a 262,144-token paged cache, 16 layers x 4 KV heads x 256,
    page 16, random table, batch 1, 24 query heads (GQA 6:1), softmax scale 1/16, in one call
    over all layers.  Checked against the oracle for sampled (layer, KV head) pairs; every
    output must be finite.  In each sampled pair the keys carry needles for the group's first
    query head at the first and last tile, both sides of a split boundary, deep in a warp's
    stream, the middle split and the last token, so one lost or misplaced tile there falls
    outside the tolerance (which a whole-window average over 262,144 tokens would not show)."""
    w = kvgen.WORKLOADS["decode_attn_262144_16L_4x256_gqa6"]
    L, T, H, D, ps, hq = w["n_layers"], w["n_tok"], w["H"], w["D"], w["page_size"], w["Hq"]
    G = hq // H
    pt_np = kvgen.random_page_table(w["seed"] + 1, 1, T // ps)
    pt = i32(pt_np, cuda_dev)
    cu = i32([0, T], cuda_dev)
    st = i32([0], cuda_dev)
    samples = [(0, 0), (L - 1, H - 1)] if bits == 6 else [(L // 2, 1)]
    qn = kvgen.queries_np(w["seed"], L, 1, hq, D)
    tpc = decode_tiles_per_cta(L, 1, H, T, torch.cuda.get_device_properties(cuda_dev)
                               .multi_processor_count)
    pos = paged_needle_positions(T, tpc, stages=3 if bits == 4 else 2)
    kps, vps, specs = [], [], []
    for layer in range(L):
        pair = []
        for is_key in (True, False):
            s = Planted(kvgen.KVSpec(seed=w["seed"], layer=layer, is_key=is_key, n_seq=1,
                                     n_tok=T, num_heads=H, head_dim=D))
            if is_key:
                for sl, h in samples:
                    if sl == layer:
                        row = needle_row(qn[layer, 0, h * G], w["softmax_scale"])
                        for t in pos:
                            s.rows[t * H + h] = row
            x = s.full_torch(cuda_dev)
            p = kvq.Pool.empty(bits, H, D, ps, pt_np.size, cuda_dev)
            kvq.kvq_quant_pack_paged([p], [x], pt, cu, st)
            del x
            pair.append((s, p))
        specs.append((pair[0][0], pair[1][0]))
        kps.append(pair[0][1])
        vps.append(pair[1][1])
    q = dev_tensor(qn, cuda_dev)
    got = _attend(kvq, cuda_dev, kps, vps, q, pt, [T], w["softmax_scale"])
    assert np.all(np.isfinite(got))
    rows_all = np.arange(T, dtype=np.int64) * H
    for layer, h in samples:
        ks, vs = specs[layer]
        k_hat = osym.dequant_rows(*osym.quant_pack_rows(ks.rows_np(rows_all + h), bits), bits, D)
        v_hat = osym.dequant_rows(*osym.quant_pack_rows(vs.rows_np(rows_all + h), bits), bits, D)
        ref = oa.attend(qn[layer, 0, h * G:(h + 1) * G], k_hat[:, None, :], v_hat[:, None, :],
                        w["softmax_scale"])
        _close(got[layer, 0, h * G:(h + 1) * G], ref)
    del kps, vps
    torch.cuda.empty_cache()
