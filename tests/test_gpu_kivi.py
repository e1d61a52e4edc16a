"""GPU parity: kivi_quant_dequant against the oracle's KIVI round trip, bit for bit.

Keys per channel (groups along tokens), values per token (groups along channels), in place on
the token slice [lo, hi); everything outside the slice must stay untouched.
"""
import numpy as np
import pytest
import torch

import kvgen
from oracle import kivi as ok
from _gpu_util import dev_tensor, u16

pytestmark = pytest.mark.gpu


def _pair(B, H, S, D, seed, layer=0):
    k = kvgen.KiviSpec(seed=seed, layer=layer, is_key=True, batch=B, num_heads=H, seq=S,
                       head_dim=D).full_np()
    v = kvgen.KiviSpec(seed=seed, layer=layer, is_key=False, batch=B, num_heads=H, seq=S,
                       head_dim=D).full_np()
    return k, v


@pytest.mark.parametrize("D", [8, 64, 96, 256])
@pytest.mark.parametrize("gs", [1, 5, 8, 32, 100])
@pytest.mark.parametrize("lo,hi", [(0, 64), (32, 160), (7, 50), (64, 65)])
def test_small_shapes_bit_exact(kvq, cuda_dev, D, gs, lo, hi):
    B, H, S = 2, 3, 200
    k, v = _pair(B, H, S, D, 1)
    k[0, 0, lo:hi, 3] = 2.5          # a constant channel and a row with ties
    v[1, 2, lo, :] = np.float16(np.arange(D) % 4 / 2.0)
    # exact ties of (x - min) / scale at 0.5, 1.5, 2.5 under 2 bits (min 0, max 2.25, scale
    # 0.75) and the fp16 neighbours on both sides, along a key channel and a value row
    t3 = np.array([0.375, 1.125, 1.875], np.float16)
    ties = np.concatenate([np.array([0.0, 2.25], np.float16), t3, np.nextafter(t3, np.float16(4)),
                           np.nextafter(t3, np.float16(0))])
    k[1, 1, lo:hi, 5 % D] = np.resize(ties, hi - lo)
    v[0, 1, (lo + hi) // 2, :] = np.resize(ties, D)
    kt, vt = dev_tensor(k, cuda_dev), dev_tensor(v, cuda_dev)
    kvq.kivi_quant_dequant([kt, vt], [True, False], lo, hi, gs, 3, 1e-8)
    torch.cuda.synchronize()
    ok.flush(k, v, lo, hi, gs, 3)
    assert np.array_equal(u16(kt), k.view(np.uint16))
    assert np.array_equal(u16(vt), v.view(np.uint16))


@pytest.mark.parametrize("levels", [1, 3, 15, 255])
def test_other_bit_widths(kvq, cuda_dev, levels):
    k, v = _pair(1, 2, 128, 64, 2)
    kt, vt = dev_tensor(k, cuda_dev), dev_tensor(v, cuda_dev)
    kvq.kivi_quant_dequant([kt, vt], [True, False], 0, 128, 32, levels, 1e-8)
    torch.cuda.synchronize()
    ok.flush(k, v, 0, 128, 32, levels)
    assert np.array_equal(u16(kt), k.view(np.uint16))
    assert np.array_equal(u16(vt), v.view(np.uint16))


def test_incremental_flushes_equal_one_shot(kvq, cuda_dev):
    """Boundary-driven flushes as tokens arrive one at a time give the same cache as one flush
    of the whole aged prefix (the chunking independence the page states)."""
    B, H, S, D, R, gs = 2, 2, 400, 64, 128, 32
    k, v = _pair(B, H, S, D, 3)
    a_k, a_v = dev_tensor(k, cuda_dev), dev_tensor(v, cuda_dev)
    b_k, b_v = dev_tensor(k, cuda_dev), dev_tensor(v, cuda_dev)
    nq = 0
    for offset in range(1, S + 1):
        hi = kvq.kivi_boundary(offset, R, gs)
        if hi > nq:
            kvq.kivi_quant_dequant([a_k, a_v], [True, False], nq, hi, gs, 3, 1e-8)
            nq = hi
    kvq.kivi_quant_dequant([b_k, b_v], [True, False], 0, kvq.kivi_boundary(S, R, gs), gs, 3,
                           1e-8)
    torch.cuda.synchronize()
    assert torch.equal(a_k, b_k) and torch.equal(a_v, b_v)


@pytest.mark.parametrize("lo,hi", [(3936, 3968), (3840, 3968)])
def test_flush_full_size(kvq, cuda_dev, lo, hi):
    """16 layers x {K,V} [16, 8, 4096, 64], 2 outlier channels x8 on keys, group 32, levels 3,
    residual 128: one call over all 32 tensors; the flushed slice is checked in full against the
    oracle and the neighbouring tokens must be unchanged."""
    w = kvgen.WORKLOADS["kivi_flush_16L_16x8x4096x64"]
    B, H, S, D = w["B"], w["H"], w["S"], w["D"]
    specs, xs, flags = [], [], []
    for layer in range(w["n_layers"]):
        for is_key in (True, False):
            s = kvgen.KiviSpec(seed=w["seed"], layer=layer, is_key=is_key, batch=B, num_heads=H,
                               seq=S, head_dim=D)
            specs.append(s)
            xs.append(s.full_torch(cuda_dev))
            flags.append(is_key)
    kvq.kivi_quant_dequant(xs, flags, lo, hi, w["group_size"], w["levels"], w["eps"])
    torch.cuda.synchronize()
    a0, a1 = lo - 16, hi + 16
    for s, x in zip(specs, xs):
        region = np.stack([np.stack([s.slab_np(b, h, a0, a1) for h in range(H)])
                           for b in range(B)])
        expect = region.copy()
        sl = expect[:, :, lo - a0:hi - a0, :]
        sl[...] = ok.quant_dequant_along(sl, -2 if s.is_key else -1, w["group_size"],
                                         w["levels"], w["eps"])
        got = x[:, :, a0:a1, :].cpu().numpy()
        assert np.array_equal(got.view(np.uint16), expect.view(np.uint16)), (s.layer, s.is_key)
    del xs
    torch.cuda.empty_cache()
