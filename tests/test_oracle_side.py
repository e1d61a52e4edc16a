"""Pins for the oracle's side channels on the symmetric quantizer (oracle/side.py): outlier
selection against its definition by brute force, the special case k = 0 (the plain quantizer),
the dense scale from the (k+1)-th largest magnitude, exact outliers and sinks, the round-trip
bound with the dense scale, and attention special cases.

Source: VeloxQuant-MLX API docs, "veloxquant_mlx.cache.kvquant_cache module" (byte accounting;
Attention Sink-Aware quantization; the config's outlier fraction 0.01)."""
import itertools

import numpy as np
import pytest

import kvgen
from oracle import attention as A
from oracle import side as SD
from oracle import symmetric as S


def _rows(n, D, seed):
    return kvgen.KVSpec(seed=seed, layer=0, is_key=True, n_seq=1, n_tok=n, num_heads=1,
                        head_dim=D).full_np()[:, 0]


def test_outlier_count_from_the_pages_fraction():
    assert SD.outlier_count(256, 0.01) == 3
    assert SD.outlier_count(128, 0.01) == 2
    assert SD.outlier_count(64, 0.01) == 1
    assert SD.outlier_count(256, 0.0) == 0


def test_selection_brute_force_with_ties():
    """Every selected element beats every unselected one: larger magnitude, or equal magnitude
    and a lower position -- checked pairwise on all rows of magnitudes from a tiny set."""
    vals = np.array([0.0, 1.0, -1.0, 2.0, -2.0], np.float16)
    D, k = 5, 2
    for row in itertools.product(range(len(vals)), repeat=D):
        x = vals[list(row)][None, :]
        _, pos, val = SD.split_outliers(x, k)
        sel = set(int(p) for p in pos[0])
        assert len(sel) == k and list(pos[0]) == sorted(pos[0])
        for i in sel:
            for j in set(range(D)) - sel:
                ai, aj = abs(float(x[0, i])), abs(float(x[0, j]))
                assert ai > aj or (ai == aj and i < j)
        assert np.array_equal(val[0], x[0, pos[0].astype(int)])


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_k0_is_the_plain_quantizer(bits):
    x = _rows(64, 256, 3)
    packed, scale, pos, val = SD.quant_pack_rows_side(x, bits, 0)
    p2, s2 = S.quant_pack_rows(x, bits)
    assert np.array_equal(packed, p2) and np.array_equal(scale.view(np.uint16), s2.view(np.uint16))
    assert pos.shape == (64, 0) and val.shape == (64, 0)


@pytest.mark.parametrize("bits", [8, 6, 4])
@pytest.mark.parametrize("k", [1, 3, 8])
def test_dense_scale_exact_outliers_and_round_trip_bound(bits, k):
    x = _rows(200, 256, 4)
    x[7] = 0                                            # all-zero row
    packed, scale, pos, val = SD.quant_pack_rows_side(x, bits, k)
    qmax = S.qmax_for(bits)
    mags = np.sort(np.abs(x.astype(np.float64)), axis=1)
    want = (mags[:, -(k + 1)].astype(np.float32) / np.float32(qmax)).astype(np.float16)
    assert np.array_equal(scale.view(np.uint16), want.view(np.uint16))
    plain = S.quant_pack_rows(x, bits)[1]
    assert np.all(scale.astype(np.float64) <= plain.astype(np.float64))
    xh = SD.dequant_rows_side(packed, scale, pos, val, bits, 256).astype(np.float64)
    xf = x.astype(np.float64)
    is_out = np.zeros(x.shape, bool)
    np.put_along_axis(is_out, pos.astype(np.int64), True, axis=1)
    assert np.array_equal(xh[is_out], xf[is_out])      # outliers are exact
    s = scale.astype(np.float64)[:, None]
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(xh), 2 ** -14))) - 10)
    normal = (s >= 2 ** -14)[:, 0]
    err = np.abs(xf - xh)
    bound = s * (0.5 + 2 ** -17) + ulp / 2
    assert np.all((err <= bound)[normal][~is_out[normal]])
    # the outlier positions hold code 0 in the packed row
    codes = S.unpack(packed, bits, 256)
    assert np.all(np.take_along_axis(codes, pos.astype(np.int64), axis=1) == 0)


def test_paged_sinks_exact_and_the_rest_dequantized():
    bits, H, D, ps, k, n_sink = 6, 2, 256, 16, 3, 4
    lens = np.array([3, 20, 40])
    pt = kvgen.random_page_table(3, 3, 3)
    pool = S.PagedPool(bits, H, D, ps, 9)
    sp = SD.SidePool(pool, k, n_sink, 3)
    x = kvgen.KVSpec(seed=6, layer=0, is_key=False, n_seq=1, n_tok=int(lens.sum()), num_heads=H,
                     head_dim=D).full_np()
    cu = np.concatenate([[0], np.cumsum(lens)])
    SD.quant_pack_paged_side(sp, x, pt, cu, np.zeros(3, np.int64))
    back = SD.dequant_paged_side(sp, pt, cu, np.zeros(3, np.int64))
    for s in range(3):
        rows = x[cu[s]:cu[s + 1]]
        got = back[cu[s]:cu[s + 1]]
        n = min(n_sink, lens[s])
        assert np.array_equal(got[:n].view(np.uint16), rows[:n].view(np.uint16))
        p, sc, po, va = SD.quant_pack_rows_side(rows[n:], bits, k)
        want = SD.dequant_rows_side(p, sc, po, va, bits, D)
        assert np.array_equal(got[n:].view(np.uint16), want.view(np.uint16))


def test_attention_over_an_all_sink_cache_is_plain_attention_on_fp16():
    """n_sink >= the length: every token is exact fp16, so the attention is the plain definition
    on the fp16 cache."""
    bits, H, G, D, ps, k = 4, 2, 3, 256, 16, 2
    n = 10
    pt = np.arange(1)[None, :]
    kp, vp = S.PagedPool(bits, H, D, ps, 1), S.PagedPool(bits, H, D, ps, 1)
    ks, vs = SD.SidePool(kp, k, 16, 1), SD.SidePool(vp, k, 16, 1)
    kx = kvgen.KVSpec(seed=7, layer=0, is_key=True, n_seq=1, n_tok=n, num_heads=H, head_dim=D).full_np()
    vx = kvgen.KVSpec(seed=7, layer=0, is_key=False, n_seq=1, n_tok=n, num_heads=H, head_dim=D).full_np()
    cu = np.array([0, n])
    SD.quant_pack_paged_side(ks, kx, pt, cu, np.array([0]))
    SD.quant_pack_paged_side(vs, vx, pt, cu, np.array([0]))
    q = kvgen.queries_np(8, 1, 1, H * G, D)[0]
    out = SD.decode_attention_paged_side(q, ks, vs, pt, np.array([n]), 1 / 16)
    assert np.array_equal(out[0], A.attend(q[0], kx, vx, 1 / 16))
