"""GPU parity at mid size: caches long enough that every warp of the decode attention streams
several tiles through its shared-memory ring, so stages are reused and mbarrier phases flip, and
ragged enough that splits end mid-stream.  Plain decode (q8/q6/q4), the fused append + decode
step and the packed KIVI attention are compared with the oracle on every output, within
|got - ref| <= 2e-3 + 1e-3 |ref|.  Needles (identical key rows along one query head's direction)
sit at the first and last tile, both sides of a split boundary, deep in a warp's stream, the
middle split and the last token of every sequence, so a lost, misplaced or stale tile there moves
the output far outside the tolerance (the CPU test test_needle_sensitivity shows that on the
oracle)."""
import numpy as np
import pytest
import torch

import kvgen
from oracle import attention as oa
from oracle import kivi_packed as okp
from oracle import symmetric as osym
from _attn_checks import (PlantedKivi, Planted, assert_attn_close, decode_splits_from_workspace,
                          decode_tiles_per_cta, kivi_needle_tokens, needle_row,
                          paged_needle_positions)
from _gpu_util import cu_of, dev_tensor, i32

pytestmark = pytest.mark.gpu

LENS = [4096, 1500, 333, 1777, 2048, 3001, 17, 640]
L, H, G, D, PS = 2, 4, 6, 256, 16
SCALE = 1.0 / 16
STAGES = {8: 2, 6: 2, 4: 3}   # stage ring of the staged decode kernel per width


def _cdiv(a, b):
    return -(-a // b)


def _sms(dev):
    return torch.cuda.get_device_properties(dev).multi_processor_count


def _planted_inputs(lens, q, tpc, bits, seed):
    """Per layer (Planted K, plain V spec) over the concatenated sequences, with needles for query
    head h * G + (s % G) of every (sequence s, KV head h)."""
    cu = cu_of(lens)
    tot = int(cu[-1])
    out = []
    for layer in range(L):
        ks = Planted(kvgen.KVSpec(seed=seed, layer=layer, is_key=True, n_seq=1, n_tok=tot,
                                  num_heads=H, head_dim=D))
        for s, n in enumerate(lens):
            pos = paged_needle_positions(int(n), tpc, STAGES[bits])
            for h in range(H):
                row = needle_row(q[layer, s, h * G + (s % G)], SCALE)
                for p in pos:
                    ks.rows[(int(cu[s]) + p) * H + h] = row
        vs = kvgen.KVSpec(seed=seed, layer=layer, is_key=False, n_seq=1, n_tok=tot, num_heads=H,
                          head_dim=D)
        out.append((ks, vs))
    return out


def _build(kvq, dev, bits, lens, q, tpc, seed, extra_pages=0):
    nseq = len(lens)
    pps = (max(lens) + extra_pages * PS + PS - 1) // PS
    pt_np = kvgen.random_page_table(seed + 1, nseq, pps)
    pt = i32(pt_np, dev)
    cu = cu_of(lens)
    kps, vps, okps, ovps = [], [], [], []
    for ks, vs in _planted_inputs(lens, q, tpc, bits, seed):
        k, v = ks.full_np(), vs.full_np()
        kp = kvq.Pool.empty(bits, H, D, PS, pt_np.size, dev)
        vp = kvq.Pool.empty(bits, H, D, PS, pt_np.size, dev)
        kvq.kvq_quant_pack_paged([kp, vp], [dev_tensor(k, dev), dev_tensor(v, dev)], pt,
                                 i32(cu, dev), i32(np.zeros(nseq), dev))
        okp_, ovp_ = osym.PagedPool(bits, H, D, PS, pt_np.size), osym.PagedPool(bits, H, D, PS,
                                                                               pt_np.size)
        osym.quant_pack_paged(okp_, k, pt_np, cu, np.zeros(nseq))
        osym.quant_pack_paged(ovp_, v, pt_np, cu, np.zeros(nseq))
        kps.append(kp); vps.append(vp); okps.append(okp_); ovps.append(ovp_)
    return kps, vps, okps, ovps, pt, pt_np


def _assert_ring_wraps(ws, nseq, max_len, tpc, bits):
    n_splits = decode_splits_from_workspace(ws.numel(), L, nseq, H)
    assert n_splits == _cdiv(_cdiv(max_len, 16), tpc), "split rule differs from the library's"
    assert tpc // 4 >= STAGES[bits] + 2, "each warp must stream past one turn of its ring"


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_decode_ring_wrap_ragged(kvq, cuda_dev, bits):
    nseq, max_len = len(LENS), max(LENS)
    tpc = decode_tiles_per_cta(L, nseq, H, max_len, _sms(cuda_dev))
    q = kvgen.queries_np(31, L, nseq, H * G, D)
    kps, vps, okps, ovps, pt, pt_np = _build(kvq, cuda_dev, bits, LENS, q, tpc, seed=32)
    ws = kvq.decode_workspace(kps, nseq, H * G, max_len, cuda_dev)
    _assert_ring_wraps(ws, nseq, max_len, tpc, bits)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_decode_attn(kps, vps, dev_tensor(q, cuda_dev), pt, i32(LENS, cuda_dev), max_len,
                        SCALE, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    for layer in range(L):
        ref = oa.decode_attention_paged(q[layer], okps[layer], ovps[layer], pt_np,
                                        np.array(LENS), SCALE)
        assert_attn_close(got[layer], ref, f"q{bits} layer {layer}")


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_append_decode_ring_wrap_ragged(kvq, cuda_dev, bits):
    """Two fused decode steps over the same ragged caches; the new key row of sequence 0 is a
    needle, so the token the kernel quantizes in the launch must be attended by it."""
    nseq, steps = len(LENS), 2
    lens = np.array(LENS)
    tpc = decode_tiles_per_cta(L, nseq, H, int(lens.max()) + 1, _sms(cuda_dev))
    q0 = kvgen.queries_np(41, L, nseq, H * G, D)
    kps, vps, okps, ovps, pt, pt_np = _build(kvq, cuda_dev, bits, LENS, q0, tpc, seed=42,
                                             extra_pages=1)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    for step in range(steps):
        max_len = int(lens.max()) + 1
        q = q0
        kn = [kvgen.KVSpec(seed=50 + step, layer=l, is_key=True, n_seq=1, n_tok=nseq,
                           num_heads=H, head_dim=D).full_np() for l in range(L)]
        vn = [kvgen.KVSpec(seed=50 + step, layer=l, is_key=False, n_seq=1, n_tok=nseq,
                           num_heads=H, head_dim=D).full_np() for l in range(L)]
        for l in range(L):
            for h in range(H):
                kn[l][0, h] = needle_row(q[l, 0, h * G], SCALE)
        ws = kvq.decode_workspace(kps, nseq, H * G, max_len, cuda_dev)
        _assert_ring_wraps(ws, nseq, max_len, tpc, bits)
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
        kvq.kvq_append_decode_attn(kps, vps, [dev_tensor(x, cuda_dev) for x in kn],
                                   [dev_tensor(x, cuda_dev) for x in vn], dev_tensor(q, cuda_dev),
                                   pt, i32(lens, cuda_dev), max_len, SCALE, out, ws, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.cpu().numpy().astype(np.float64)
        for l in range(L):
            ref = oa.append_decode_paged(q[l], okps[l], ovps[l], kn[l], vn[l], pt_np, lens, SCALE)
            assert_attn_close(got[l], ref, f"q{bits} step {step} layer {l}")
            for pool, opool in ((kps[l], okps[l]), (vps[l], ovps[l])):
                for s, n in enumerate(lens):
                    page, slot = int(pt_np[s, n // PS]), int(n % PS)
                    assert np.array_equal(pool.codes[page, :, slot].cpu().numpy(),
                                          opool.codes[page, :, slot])
        lens = lens + 1


def test_kivi_attention_ring_wrap(kvq, cuda_dev):
    """2 layers x 2 batch rows x 2 KV heads over 32,544 packed + 156 fp16 tokens: with few
    (layer, row, head) units every CTA takes many 64-token chunks, so each warp's 3-stage ring
    turns several times; needle key groups (stored exactly: a zero-range group) and needle
    residual tokens sit at the first chunk, a chunk boundary, mid-stream, the last packed group
    and in the fp16 window."""
    Lk, B, Hk, Gk, S, Dk, gs = 2, 2, 2, 4, 32768, 64, 32
    n_packed, offset, scale = 32544, 32700, 0.125
    q = kvgen.queries_np(61, Lk, B, Hk * Gk, Dk)
    toks = kivi_needle_tokens(n_packed, offset, gs)
    caches, ks_d, vs_d, host = [], [], [], []
    for layer in range(Lk):
        ks = PlantedKivi(kvgen.KiviSpec(seed=62, layer=layer, is_key=True, batch=B, num_heads=Hk,
                                        seq=S, head_dim=Dk))
        for b in range(B):
            for h in range(Hk):
                row = needle_row(q[layer, b, h * Gk + (b % Gk)], scale)
                for t in toks:
                    ks.rows[(b, h, t)] = row
        k = ks.full_np()
        v = kvgen.KiviSpec(seed=62, layer=layer, is_key=False, batch=B, num_heads=Hk, seq=S,
                           head_dim=Dk).full_np()
        host.append((k, v))
        caches.append(kvq.KiviPacked.empty(2, gs, B, Hk, S, Dk, cuda_dev))
        ks_d.append(dev_tensor(k, cuda_dev))
        vs_d.append(dev_tensor(v, cuda_dev))
    kvq.kivi_pack(caches, ks_d, vs_d, 0, n_packed)
    nbytes = kvq.kivi_decode_attn_workspace(Lk, B, Hk, Hk * Gk, Dk, offset)
    n_splits = nbytes // (Lk * B * Hk * 8 * (Dk + 4) * 4)
    chunks = _cdiv(_cdiv(offset, 16), 4)
    assert _cdiv(chunks, n_splits) // 4 >= 3 + 2, "each warp must stream past one ring turn"
    ws = torch.empty(max(16, nbytes), dtype=torch.uint8, device=cuda_dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kivi_decode_attn(caches, ks_d, vs_d, dev_tensor(q, cuda_dev), n_packed, offset, scale,
                         out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    for layer, (k, v) in enumerate(host):
        kp = okp.pack_keys(k[:, :, :n_packed], 2, gs)
        vp = okp.pack_values(v[:, :, :n_packed], 2, gs)
        ref = okp.decode_attention(q[layer], kp, vp, k[:, :, n_packed:offset],
                                   v[:, :, n_packed:offset], 2, gs, scale)
        assert_attn_close(got[layer], ref, f"KIVI layer {layer}")
