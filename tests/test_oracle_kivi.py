"""Pins for the oracle's KIVI round trip, residual boundary, flush and trim.

Ties to the VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache": hand-worked groups and
boundaries (tests/golden/kivi_groups.json), and the invariants the page states -- a one-element
group collapses to scale = eps and round-trips exactly (``_quantization_boundary`` docstring),
the result does not depend on how the sequence was chunked (same docstring), keys group along
tokens and values along channels (module docstring), and re-quantizing after a trim moves a
value by at most one quantization step (``_rollback_frontier`` docstring).
"""
import json

import numpy as np
import pytest

import kvgen
from oracle import kivi as K
from conftest import golden_path


def _golden():
    with open(golden_path("kivi_groups.json")) as f:
        return json.load(f)


def test_golden_roundtrips():
    for case in _golden()["roundtrips"]:
        x = np.array(case["x"], dtype=np.float16)
        assert np.array_equal(x.astype(np.float64), np.array(case["x"])), case["name"]
        if case["axis"] == -2:       # keys: one channel, tokens along axis -2
            t = x.reshape(1, 1, -1, 1)
        else:                         # values: one token, channels along axis -1
            t = x.reshape(1, 1, 1, -1)
        out = K.quant_dequant_along(t, case["axis"], case["group_size"], 3, 1e-8).ravel()
        assert out.dtype == np.float16
        assert out.astype(np.float64).tolist() == case["out"], case["name"]


def test_golden_boundary():
    g = _golden()["boundary"]
    for offset, expect in g["cases"]:
        assert K.quantization_boundary(offset, g["residual_length"], g["group_size"]) == expect


def _kivi_rows(B, H, S, D, seed, is_key):
    spec = kvgen.KiviSpec(seed=seed, layer=0, is_key=is_key, batch=B, num_heads=H, seq=S,
                          head_dim=D)
    return spec.full_np()


@pytest.mark.parametrize("axis", [-2, -1])
def test_single_element_groups_are_exact(axis):
    x = _kivi_rows(2, 2, 8, 8, 1, True)
    out = K.quant_dequant_along(x, axis, 1, 3, 1e-8)
    assert np.array_equal(out.view(np.uint16), x.view(np.uint16))


def test_axes_keys_per_channel_values_per_token():
    """A channel that is constant over tokens survives the key round trip exactly (its key groups
    collapse); a token that is constant over channels survives the value round trip exactly."""
    x = _kivi_rows(1, 1, 32, 64, 2, True).astype(np.float32)
    x[:, :, :, 5] = 1.25
    out = K.quant_dequant_along(x.astype(np.float16), -2, 32, 3, 1e-8)
    assert np.all(out[:, :, :, 5] == np.float16(1.25))
    y = _kivi_rows(1, 1, 4, 64, 3, False).astype(np.float32)
    y[:, :, 2, :] = -0.5
    out = K.quant_dequant_along(y.astype(np.float16), -1, 32, 3, 1e-8)
    assert np.all(out[:, :, 2, :] == np.float16(-0.5))


def _brute_groups(x, axis, gs, levels, eps):
    """Scalar loops over each group of real elements only (no padding), float32 steps."""
    x = np.asarray(x)
    xm = np.moveaxis(x.astype(np.float32), axis, -1)
    out = np.empty_like(xm)
    L = xm.shape[-1]
    for idx in np.ndindex(xm.shape[:-1]):
        row = xm[idx]
        for g0 in range(0, L, gs):
            grp = row[g0:g0 + gs]
            lo, hi = np.float32(grp.min()), np.float32(grp.max())
            sc = max(np.float32(np.float32(hi - lo) / np.float32(levels)), np.float32(eps))
            for j, v in enumerate(grp):
                c = min(max(np.rint(np.float32(np.float32(v - lo) / sc)), 0), levels)
                out[idx + (g0 + j,)] = np.float32(np.float32(np.float32(c) * sc) + lo)
    return np.moveaxis(out, -1, axis).astype(x.dtype)


@pytest.mark.parametrize("axis,L,gs", [(-2, 37, 8), (-1, 24, 5), (-1, 64, 32), (-2, 64, 32)])
def test_ragged_tail_padding_equals_min_max_of_real_elements(axis, L, gs):
    shape = (2, 3, L, 16) if axis == -2 else (2, 3, 6, L)
    x = kvgen.normal_fp16_np(4, 50, np.arange(np.prod(shape))).reshape(shape)
    assert np.array_equal(K.quant_dequant_along(x, axis, gs, 3, 1e-8).view(np.uint16),
                          _brute_groups(x, axis, gs, 3, 1e-8).view(np.uint16))


def test_roundtrip_error_within_half_step():
    x = _kivi_rows(2, 4, 128, 64, 5, True)
    for axis in (-2, -1):
        out = K.quant_dequant_along(x, axis, 32, 3, 1e-8).astype(np.float64)
        xm = np.moveaxis(x.astype(np.float64), axis, -1)
        om = np.moveaxis(out, axis, -1)
        g = xm.reshape(xm.shape[:-1] + (-1, 32))
        step = (g.max(-1) - g.min(-1)) / 3
        err = np.abs(g - om.reshape(g.shape))
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(om.reshape(g.shape)), 2 ** -14))) - 10)
        assert np.all(err <= step[..., None] * (0.5 + 1e-5) + ulp / 2 + 1e-12)


def test_flush_result_does_not_depend_on_chunking():
    B, H, S, D = 2, 2, 400, 16
    keys = _kivi_rows(B, H, S, D, 6, True)
    values = _kivi_rows(B, H, S, D, 7, False)
    one = K.KiviCache(B, H, D, S)
    one.update_and_fetch(keys, values)
    tok = K.KiviCache(B, H, D, S)
    for t in range(S):
        tok.update_and_fetch(keys[:, :, t:t + 1], values[:, :, t:t + 1])
    rnd = K.KiviCache(B, H, D, S)
    cuts = [0, 1, 17, 64, 65, 200, 333, S]
    for a, b in zip(cuts[:-1], cuts[1:]):
        rnd.update_and_fetch(keys[:, :, a:b], values[:, :, a:b])
    for c in (tok, rnd):
        assert c.n_quantized == one.n_quantized == K.quantization_boundary(S, 128, 32)
        assert np.array_equal(c.keys.view(np.uint16), one.keys.view(np.uint16))
        assert np.array_equal(c.values.view(np.uint16), one.values.view(np.uint16))
    # the residual window stays exact fp16
    nq = one.n_quantized
    assert np.array_equal(one.keys[:, :, nq:], keys[:, :, nq:])
    assert not np.array_equal(one.keys[:, :, :nq], keys[:, :, :nq])


def test_flush_window_matches_update_and_fetch():
    """kivi flush of [lo, hi) equals what update_and_fetch does at that boundary."""
    B, H, S, D = 1, 2, 4096, 64
    keys = _kivi_rows(B, H, S, D, 8, True)
    values = _kivi_rows(B, H, S, D, 9, False)
    c = K.KiviCache(B, H, D, S)
    c.update_and_fetch(keys[:, :, :4064], values[:, :, :4064])
    assert c.n_quantized == 3936
    c.update_and_fetch(keys[:, :, 4064:], values[:, :, 4064:])
    assert c.n_quantized == 3968
    k2, v2 = keys.copy(), values.copy()
    K.flush(k2, v2, 0, 3936, 32, 3)
    K.flush(k2, v2, 3936, 3968, 32, 3)
    assert np.array_equal(k2.view(np.uint16), c.keys.view(np.uint16))
    assert np.array_equal(v2.view(np.uint16), c.values.view(np.uint16))


def test_trim_rolls_frontier_back_to_a_group_multiple():
    B, H, S, D = 1, 1, 300, 8
    keys = _kivi_rows(B, H, S, D, 10, True)
    values = _kivi_rows(B, H, S, D, 11, False)
    c = K.KiviCache(B, H, D, S)
    c.update_and_fetch(keys, values)
    assert c.n_quantized == 160
    assert c.trim(150) == 150 and c.offset == 150
    assert c.n_quantized == 128          # min(160, (150 // 32) * 32)
    assert c.trim(1000) == 150 and c.offset == 0 and c.n_quantized == 0


def test_requantize_after_trim_moves_values_by_at_most_one_step():
    B, H, S, D = 1, 2, 320, 16
    keys = _kivi_rows(B, H, S, D, 12, True)
    values = _kivi_rows(B, H, S, D, 13, False)
    c = K.KiviCache(B, H, D, S)
    c.update_and_fetch(keys, values)                  # frontier 192
    first_k = c.keys[:, :, :192].astype(np.float64).copy()
    c.trim(110)                                        # offset 210, frontier 192
    c.trim(30)                                         # offset 180, frontier 160
    assert c.n_quantized == 160
    c.update_and_fetch(keys[:, :, 180:], values[:, :, 180:])
    assert c.n_quantized == 192
    redo = c.keys[:, :, 160:192].astype(np.float64)
    grp = keys[:, :, 160:192].astype(np.float64)
    step = (grp.max(axis=2, keepdims=True) - grp.min(axis=2, keepdims=True)) / 3
    assert np.all(np.abs(redo - first_k[:, :, 160:192]) <= step * 1.0001 + 1e-3)
