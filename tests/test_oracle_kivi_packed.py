"""Pins for the oracle's packed KIVI storage and the attention over it (see oracle/kivi_packed.py
for the readings).  Ties: hand-worked keys/values groups (tests/golden/kivi_packed.json); the
layout stores exactly the bytes of the page's packed-size estimate (``_quantized_bytes``);
whenever the group scale is already an fp16 value the packed round trip equals the page's
in-place round trip bit for bit; codes are nearest against the stored scale; attention special
cases and PyTorch SDPA in float64."""
import json

import numpy as np
import pytest
import torch

import kvgen
from oracle import attention as A
from oracle import kivi as K
from oracle import kivi_packed as P
from conftest import golden_path


def _g():
    with open(golden_path("kivi_packed.json")) as f:
        return json.load(f)


def _bits(a):
    return [f"{int(v):04x}" for v in np.asarray(a, np.float16).view(np.uint16).ravel()]


def test_golden_keys():
    g = _g()["keys"]
    x = np.array(g["x_tokens_by_channels"], np.float16)[None, None]      # [1, 1, 4, 4]
    codes, s16, z16 = P.pack_keys(x, g["bits"], g["group_size"])
    assert _bits(s16) == g["scale_bits"] and _bits(z16) == g["zero_bits"]
    assert [r.tobytes().hex() for r in codes[0, 0]] == g["packed_rows"]
    assert P.unpack_bits(codes, 2, 4)[0, 0].tolist() == g["codes"]
    xhat = P.unpack_keys(codes, s16, z16, g["bits"], g["group_size"], 4)
    assert xhat[0, 0].astype(np.float64).tolist() == g["xhat"]


def test_golden_values():
    g = _g()["values"]
    x = np.array(g["x_row"], np.float16)[None, None, None]                # [1, 1, 1, 4]
    codes, s16, z16 = P.pack_values(x, g["bits"], g["group_size"])
    assert _bits(s16) == g["scale_bits"] and _bits(z16) == g["zero_bits"]
    assert codes[0, 0, 0].tobytes().hex() == g["packed_row"]
    assert P.unpack_bits(codes, 2, 4)[0, 0, 0].tolist() == g["codes"]
    xhat = P.unpack_values(codes, s16, z16, g["bits"], g["group_size"], 4)
    assert xhat[0, 0, 0].astype(np.float64).tolist() == g["xhat"]
    # the page's in-place float32 round trip reconstructs 1.0 for the last element
    rt = K.quant_dequant_along(x, -1, 2, 3)
    assert float(rt[0, 0, 0, 3]) == 1.0


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("n,B,H,D,gs", [(160, 1, 4, 64, 32), (32, 2, 3, 64, 32), (128, 1, 8, 128, 64),
                                       (64, 4, 2, 96, 32), (96, 1, 1, 64, 16)])
def test_layout_stores_exactly_the_pages_estimate(bits, n, B, H, D, gs):
    k_est, v_est = K.quantized_bytes(n, B, H, D, bits, gs)
    assert P.packed_bytes(n, B, H, D, bits, gs) == (k_est, v_est)
    x = kvgen.KiviSpec(seed=1, layer=0, is_key=True, batch=B, num_heads=H, seq=n,
                       head_dim=D).full_np()
    kc, ks, kz = P.pack_keys(x, bits, gs)
    vc, vs, vz = P.pack_values(x, bits, gs)
    assert kc.nbytes + ks.nbytes + kz.nbytes == k_est
    assert vc.nbytes + vs.nbytes + vz.nbytes == v_est


def test_accounting_consistency_with_the_pages_reported_figure():
    g = _g()["accounting"]
    k, _ = P.packed_bytes(g["n"], g["batch"], g["num_heads"], g["head_dim"], g["bits"],
                          g["group_size"])
    assert k == g["key_bytes"]


def test_equals_the_in_place_round_trip_when_the_scale_is_fp16_exact():
    # ranges 3 * 2^k: range / 3 = 2^k is an fp16 value, so both forms use the same scale
    rng = np.random.default_rng(3)
    B, H, n, D = 2, 2, 64, 32
    e = rng.integers(-6, 4, size=(B, H, n // 32, 1, D))
    lo = rng.integers(-8, 8, size=(B, H, n // 32, 1, D)) * 2.0 ** e
    frac = rng.integers(0, 13, size=(B, H, n // 32, 32, D)) / 4.0       # multiples of 1/4 in [0, 3]
    frac[:, :, :, 0, :] = 0
    frac[:, :, :, 1, :] = 3
    x = (lo + frac * 2.0 ** e).reshape(B, H, n, D).astype(np.float16)
    assert np.all(x.astype(np.float64) == (lo + frac * 2.0 ** e).reshape(B, H, n, D))
    codes, s, z = P.pack_keys(x, 2, 32)
    assert np.array_equal(P.unpack_keys(codes, s, z, 2, 32, D).view(np.uint16),
                          K.quant_dequant_along(x, -2, 32, 3).view(np.uint16))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_codes_nearest_against_stored_scale_and_error_bound(bits):
    x = kvgen.KiviSpec(seed=5, layer=2, is_key=True, batch=2, num_heads=4, seq=128,
                       head_dim=64).full_np()
    L = P.levels_of(bits)
    for pack, unpack, axis in ((P.pack_keys, P.unpack_keys, -2), (P.pack_values, P.unpack_values, -1)):
        codes, s, z = pack(x, bits, 32)
        c = P.unpack_bits(codes, bits, 64).astype(np.float64)
        if axis == -2:
            s64 = np.repeat(s, 32, axis=2).astype(np.float64)
            z64 = np.repeat(z, 32, axis=2).astype(np.float64)
        else:
            gi = np.arange(64) // 32
            s64, z64 = s[..., gi].astype(np.float64), z[..., gi].astype(np.float64)
        r = (x.astype(np.float64) - z64) / s64
        inner = (c > 0) & (c < L)
        assert np.all(np.abs(r - c)[inner] <= 0.5 + 1e-6)
        assert np.all(r[c == 0] <= 0.5 + 1e-6) and np.all(r[c == L] >= L - 0.5 - 1e-6)
        xhat = unpack(codes, s, z, bits, 32, 64).astype(np.float64)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(xhat), 2 ** -14))) - 10)
        assert np.all(np.abs(xhat - x) <= s64 * (0.5 + 1e-6) + ulp)


def _packed_case(seed, B, H, G, n_q, n_res, D=64, bits=2, gs=32):
    ks = kvgen.KiviSpec(seed=seed, layer=0, is_key=True, batch=B, num_heads=H, seq=n_q + n_res,
                        head_dim=D)
    vs = kvgen.KiviSpec(seed=seed, layer=0, is_key=False, batch=B, num_heads=H,
                        seq=n_q + n_res, head_dim=D)
    k, v = ks.full_np(), vs.full_np()
    q = kvgen.queries_np(seed, 1, B, H * G, D)[0]
    kp = P.pack_keys(k[:, :, :n_q], bits, gs)
    vp = P.pack_values(v[:, :, :n_q], bits, gs)
    return q, k, v, kp, vp


def test_attention_matches_torch_sdpa_on_the_dequantized_cache():
    B, H, G, n_q, n_res, D = 2, 2, 4, 96, 37, 64
    q, k, v, kp, vp = _packed_case(7, B, H, G, n_q, n_res)
    out = P.decode_attention(q, kp, vp, k[:, :, n_q:], v[:, :, n_q:], 2, 32, 0.125)
    kh = np.concatenate([P.unpack_keys(*kp, 2, 32, D), k[:, :, n_q:]], axis=2).astype(np.float64)
    vh = np.concatenate([P.unpack_values(*vp, 2, 32, D), v[:, :, n_q:]], axis=2).astype(np.float64)
    qt = torch.from_numpy(q.astype(np.float64))[:, :, None, :]
    kt = torch.from_numpy(kh).repeat_interleave(G, 1)
    vt = torch.from_numpy(vh).repeat_interleave(G, 1)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=0.125)[:, :, 0]
    assert np.allclose(out, ref.numpy(), rtol=1e-12, atol=1e-13)


def test_attention_special_cases():
    B, H, G, D = 1, 1, 4, 64
    q, k, v, kp, vp = _packed_case(8, B, H, G, 0, 5)
    out = P.decode_attention(q, kp, vp, k, v, 2, 32, 0.125)          # no packed tokens
    ref = A.attend(q[0], k[0].transpose(1, 0, 2), v[0].transpose(1, 0, 2), 0.125)
    assert np.array_equal(out[0], ref)
    # equal keys everywhere -> uniform weights -> mean of the reconstructed values
    kk = np.repeat(k[:, :, :1], 64, axis=2)
    vv = kvgen.KiviSpec(seed=9, layer=0, is_key=False, batch=1, num_heads=1, seq=64,
                        head_dim=D).full_np()
    kp2, vp2 = P.pack_keys(kk[:, :, :32], 2, 32), P.pack_values(vv[:, :, :32], 2, 32)
    kh = P.unpack_keys(*kp2, 2, 32, D)
    assert np.array_equal(kh, kk[:, :, :32])   # constant channels: scale 0, exact zero point
    out = P.decode_attention(q, kp2, vp2, kk[:, :, 32:], vv[:, :, 32:], 2, 32, 0.125)
    vh = np.concatenate([P.unpack_values(*vp2, 2, 32, D), vv[:, :, 32:]], axis=2)
    assert np.allclose(out[0], vh[0, 0].astype(np.float64).mean(0), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- the cache protocol, packed
def _exact_scale_tokens(rng, B, H, n, D, gs):
    """Tokens whose every key group (gs tokens of a channel) and value group (gs channels of a
    token) spans exactly 3 * 2^e: range / 3 is an fp16 value, so the packed and the in-place
    round trips use the same scale and give the same fp16 values."""
    e = rng.integers(-4, 2, size=(B, H, n // gs, 1, 1))
    base = rng.integers(-6, 6, size=(B, H, n // gs, 1, 1)) * 2.0 ** e
    frac = rng.integers(0, 13, size=(B, H, n // gs, gs, D)) / 4.0
    frac[:, :, :, 0, :] = 0          # every key group holds its min and max
    frac[:, :, :, 1, :] = 3
    frac[..., 0::gs] = 0             # every value group holds its min and max
    frac[..., 1::gs] = 3
    x = (base + frac * 2.0 ** e).reshape(B, H, n, D)
    assert np.all(x.astype(np.float16).astype(np.float64) == x)
    return x.astype(np.float16)


def test_packed_protocol_equals_the_in_place_protocol_on_exact_scale_data():
    """update_and_fetch in chunks of 1..70 tokens: the packed cache's view equals the page's
    in-place fp16 cache bit for bit (same flush windows, same round-tripped values)."""
    rng = np.random.default_rng(11)
    B, H, D, gs, R, S = 2, 2, 64, 32, 128, 640
    k = _exact_scale_tokens(rng, B, H, S, D, gs)
    v = _exact_scale_tokens(rng, B, H, S, D, gs)
    ref = K.KiviCache(B, H, D, S, bit_width=2, group_size=gs, residual_length=R)
    pc = P.KiviPackedCache(B, H, D, S, bit_width=2, group_size=gs, residual_length=R)
    t = 0
    for n in [1, 5, 70, 31, 64, 1, 1, 128, 40, 200]:
        kr, vr = ref.update_and_fetch(k[:, :, t:t + n], v[:, :, t:t + n])
        pc.update(k[:, :, t:t + n], v[:, :, t:t + n])
        t += n
        assert pc.offset == ref.offset and pc.n_quantized == ref.n_quantized
        kp, vp = pc.fetch()
        assert np.array_equal(kp.view(np.uint16), kr.view(np.uint16))
        assert np.array_equal(vp.view(np.uint16), vr.view(np.uint16))


def test_packed_trim_rolls_back_like_the_page_and_keeps_round_tripped_rows():
    """Frontier after a trim = min(old, floor(offset / gs) * gs) (``_rollback_frontier``); the
    rows between the new frontier and the new offset hold their round-tripped values in the fp16
    window, and the view is unchanged on the kept tokens."""
    B, H, D, gs, R, S = 1, 2, 64, 32, 128, 512
    x = kvgen.KiviSpec(seed=8, layer=0, is_key=True, batch=B, num_heads=H, seq=S, head_dim=D)
    y = kvgen.KiviSpec(seed=8, layer=0, is_key=False, batch=B, num_heads=H, seq=S, head_dim=D)
    k, v = x.full_np(), y.full_np()
    pc = P.KiviPackedCache(B, H, D, S, group_size=gs, residual_length=R)
    pc.update(k[:, :, :400], v[:, :, :400])
    assert pc.n_quantized == 256
    before_k, before_v = pc.fetch()
    assert pc.trim(150) == 150 and pc.offset == 250 and pc.n_quantized == 224
    kk, vv = pc.fetch()
    assert np.array_equal(kk.view(np.uint16), before_k[:, :, :250].view(np.uint16))
    assert np.array_equal(vv.view(np.uint16), before_v[:, :, :250].view(np.uint16))
    assert not np.array_equal(pc.keys[:, :, 224:250], k[:, :, 224:250])   # round-tripped now
    assert pc.trim(1000) == 250 and pc.offset == 0 and pc.n_quantized == 0


def test_packed_requantize_after_trim_moves_values_by_at_most_one_step():
    """The page's bound on the double rounding: a row quantized, rolled back by a trim and
    quantized again differs from its first round trip by at most one step of the new group
    (plus half an fp16 ulp of each stored value)."""
    B, H, D, gs, R, S = 1, 2, 64, 32, 128, 640
    x = kvgen.KiviSpec(seed=9, layer=1, is_key=True, batch=B, num_heads=H, seq=S, head_dim=D)
    y = kvgen.KiviSpec(seed=9, layer=1, is_key=False, batch=B, num_heads=H, seq=S, head_dim=D)
    k, v = x.full_np(), y.full_np()
    pc = P.KiviPackedCache(B, H, D, S, group_size=gs, residual_length=R)
    pc.update(k[:, :, :420], v[:, :, :420])            # frontier 288
    first_k, first_v = (a.astype(np.float64) for a in pc.fetch())
    pc.trim(140)                                       # offset 280, frontier 256
    pc.update(k[:, :, 280:600], v[:, :, 280:600])      # re-flushes [256, 448)
    again_k, again_v = (a.astype(np.float64) for a in pc.fetch())
    rows = slice(256, 280)
    ks = np.repeat(pc.k_scale.astype(np.float64), gs, axis=2)[:, :, rows]
    vs = pc.v_scale.astype(np.float64)[:, :, rows][..., np.arange(D) // gs]
    for a, b, s in ((again_k, first_k, ks), (again_v, first_v, vs)):
        d = np.abs(a[:, :, rows] - b[:, :, rows])
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(b[:, :, rows]), 2 ** -14))) - 10)
        assert np.all(d <= s + ulp)
