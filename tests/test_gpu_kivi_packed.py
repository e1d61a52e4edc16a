"""GPU parity for packed KIVI storage: kivi_pack against the oracle's packed form bit for bit
(codes, scales, zeros), and kivi_decode_attn (packed tokens plus the fp16 residual window)
against the oracle's dequantize-then-softmax attention within 2e-3 + 1e-3*|ref|."""
import numpy as np
import pytest
import torch

import kvgen
from oracle import kivi_packed as P
from _attn_checks import PlantedKivi, assert_attn_close, kivi_needle_tokens, needle_row
from _gpu_util import dev_tensor, u16

pytestmark = pytest.mark.gpu


def _layer(seed, layer, B, H, S, D):
    k = kvgen.KiviSpec(seed=seed, layer=layer, is_key=True, batch=B, num_heads=H, seq=S,
                       head_dim=D).full_np()
    v = kvgen.KiviSpec(seed=seed, layer=layer, is_key=False, batch=B, num_heads=H, seq=S,
                       head_dim=D).full_np()
    return k, v


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("gs,D", [(32, 64), (16, 64), (8, 64), (64, 64), (8, 32), (64, 128),
                                  (32, 256)])
def test_pack_bit_exact(kvq, cuda_dev, bits, gs, D):
    B, H, S, L = 2, 3, 4 * gs, 2
    lo, hi = gs, 3 * gs
    caches, ks, vs, ref = [], [], [], []
    for layer in range(L):
        k, v = _layer(11, layer, B, H, S, D)
        k[0, 0, gs:2 * gs, 5] = 1.25            # a constant channel group (scale underflows to 0)
        # exact ties (x - min) / scale = n + 1/2 under 2 bits: min 0, max 2.25, scale 0.75, and
        # the fp16 neighbours on both sides of each tie
        t3 = np.array([0.375, 1.125, 1.875], np.float16)
        ties = np.concatenate([np.array([0.0, 2.25], np.float16), t3,
                               np.nextafter(t3, np.float16(4)), np.nextafter(t3, np.float16(0)),
                               np.array([0.75, 1.5], np.float16)])
        k[1, 1, gs:2 * gs, 7] = np.resize(ties, gs)
        v[1, 2, gs + 3, :gs] = np.resize(ties, gs)
        caches.append(kvq.KiviPacked.empty(bits, gs, B, H, S, D, cuda_dev))
        ks.append(dev_tensor(k, cuda_dev))
        vs.append(dev_tensor(v, cuda_dev))
        ref.append((P.pack_keys(k[:, :, lo:hi], bits, gs), P.pack_values(v[:, :, lo:hi], bits, gs)))
    kvq.kivi_pack(caches, ks, vs, lo, hi)
    torch.cuda.synchronize()
    for c, ((kc, ksc, kz), (vc, vsc, vz)) in zip(caches, ref):
        assert np.array_equal(c.k_codes[:, :, lo:hi].cpu().numpy(), kc)
        assert np.array_equal(u16(c.k_scale[:, :, lo // gs:hi // gs]), ksc.view(np.uint16))
        assert np.array_equal(u16(c.k_zero[:, :, lo // gs:hi // gs]), kz.view(np.uint16))
        assert np.array_equal(c.v_codes[:, :, lo:hi].cpu().numpy(), vc)
        assert np.array_equal(u16(c.v_scale[:, :, lo:hi]), vsc.view(np.uint16))
        assert np.array_equal(u16(c.v_zero[:, :, lo:hi]), vz.view(np.uint16))
        # outside [lo, hi) nothing is written
        assert int(c.k_codes[:, :, :lo].count_nonzero()) == 0
        assert int(c.v_codes[:, :, hi:].count_nonzero()) == 0


def _attn_case(kvq, dev, L, B, H, G, S, n_packed, offset, gs=32, seed=12):
    D = 64
    caches, ks, vs, ref_in = [], [], [], []
    for layer in range(L):
        k, v = _layer(seed, layer, B, H, S, D)
        c = kvq.KiviPacked.empty(2, gs, B, H, S, D, dev)
        caches.append(c)
        ks.append(dev_tensor(k, dev))
        vs.append(dev_tensor(v, dev))
        ref_in.append((k, v))
    if n_packed:
        kvq.kivi_pack(caches, ks, vs, 0, n_packed)
    q = kvgen.queries_np(seed, L, B, H * G, D)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=dev)
    ws = torch.empty(max(16, kvq.kivi_decode_attn_workspace(L, B, H, H * G, D, offset)),
                     dtype=torch.uint8, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kvq.kivi_decode_attn(caches, ks, vs, dev_tensor(q, dev), n_packed, offset, 0.125, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    for layer, (k, v) in enumerate(ref_in):
        kp = P.pack_keys(k[:, :, :n_packed], 2, gs)
        vp = P.pack_values(v[:, :, :n_packed], 2, gs)
        ref = P.decode_attention(q[layer], kp, vp, k[:, :, n_packed:offset],
                                 v[:, :, n_packed:offset], 2, gs, 0.125)
        assert_attn_close(got[layer], ref, f"layer {layer}")


@pytest.mark.parametrize("n_packed,offset", [(0, 1), (0, 37), (32, 33), (96, 200), (256, 300),
                                             (512, 512), (224, 500), (480, 511)])
def test_attention_small(kvq, cuda_dev, n_packed, offset):
    _attn_case(kvq, cuda_dev, L=2, B=2, H=2, G=4, S=512, n_packed=n_packed, offset=offset)


@pytest.mark.parametrize("gs", [16, 64])
def test_attention_group_sizes(kvq, cuda_dev, gs):
    _attn_case(kvq, cuda_dev, L=1, B=3, H=4, G=8, S=256, n_packed=4 * gs if gs == 16 else 128,
               offset=230, gs=gs)


def test_full_size_pack_and_attend_sampled(kvq, cuda_dev):
    """16 layers x [16, 8, 4096, 64], 2-bit, group 32: pack the aged tokens [0, 3968) of every
    layer in one call, attend with 32 query heads (GQA 4:1) over 3968 packed + 128 residual
    tokens; the packed bytes of sampled (layer, b, h) slabs are checked exactly and the outputs of
    sampled layers within tolerance."""
    w = kvgen.WORKLOADS["kivi_flush_16L_16x8x4096x64"]
    L, B, H, S, D, gs = w["n_layers"], w["B"], w["H"], w["S"], w["D"], w["group_size"]
    n_packed, offset, Hq = 3968, 4096, 32
    G = Hq // H
    samples = [(0, 0, 0), (7, 5, 3), (15, 15, 7)]
    qn = kvgen.queries_np(w["seed"], L, B, Hq, D)
    needles = kivi_needle_tokens(n_packed, offset, gs)
    caches, ks, vs, specs = [], [], [], []
    for layer in range(L):
        # the sampled slabs' keys carry needle groups (stored exactly) and needle window tokens
        # for the group's first query head, so a lost or misplaced chunk moves that head's output
        # far outside the tolerance
        sk = PlantedKivi(kvgen.KiviSpec(seed=w["seed"], layer=layer, is_key=True, batch=B,
                                        num_heads=H, seq=S, head_dim=D))
        for sl, b, h in samples:
            if sl == layer:
                row = needle_row(qn[layer, b, h * G], 0.125)
                for t in needles:
                    sk.rows[(b, h, t)] = row
        sv = kvgen.KiviSpec(seed=w["seed"], layer=layer, is_key=False, batch=B, num_heads=H,
                            seq=S, head_dim=D)
        specs.append((sk, sv))
        ks.append(sk.full_torch(cuda_dev))
        vs.append(sv.full_torch(cuda_dev))
        caches.append(kvq.KiviPacked.empty(2, gs, B, H, S, D, cuda_dev))
    kvq.kivi_pack(caches, ks, vs, 0, n_packed)
    q = dev_tensor(qn, cuda_dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=cuda_dev)
    ws = torch.empty(kvq.kivi_decode_attn_workspace(L, B, H, Hq, D, offset), dtype=torch.uint8,
                     device=cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kivi_decode_attn(caches, ks, vs, q, n_packed, offset, 0.125, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    for layer, b, h in samples:
        sk, sv = specs[layer]
        k = sk.slab_np(b, h, 0, offset)[None, None]
        v = sv.slab_np(b, h, 0, offset)[None, None]
        kp = P.pack_keys(k[:, :, :n_packed], 2, gs)
        vp = P.pack_values(v[:, :, :n_packed], 2, gs)
        c = caches[layer]
        assert np.array_equal(c.k_codes[b, h, :n_packed].cpu().numpy(), kp[0][0, 0])
        assert np.array_equal(u16(c.k_scale[b, h, :n_packed // gs]), kp[1][0, 0].view(np.uint16))
        assert np.array_equal(c.v_codes[b, h, :n_packed].cpu().numpy(), vp[0][0, 0])
        assert np.array_equal(u16(c.v_zero[b, h, :n_packed]), vp[2][0, 0].view(np.uint16))
        ref = P.decode_attention(qn[layer, b:b + 1, h * G:(h + 1) * G], kp, vp,
                                 k[:, :, n_packed:], v[:, :, n_packed:], 2, gs, 0.125)[0]
        assert_attn_close(got[layer, b, h * G:(h + 1) * G], ref, f"layer {layer} b {b} h {h}")
    # the stored bytes are the page's estimate of a packed cache
    kb, vb = caches[0].nbytes(n_packed)
    assert (kb, vb) == P.packed_bytes(n_packed, B, H, D, 2, gs)
