"""Pins for the oracle's symmetric quantizer, q8/q6/q4 packing and paged scatter/gather.

Each check ties the oracle to something other than itself: the q6 byte-layout formula and the
packed_dim / bit-width statements of MTPLX pull request #267 ("feat(kv-cache): add q6 paged KV
quantization", description), hand-worked rows (tests/golden), brute force over every q6 field
value, an independent bit-stream packer, exact rational arithmetic, and the round-trip bound.
"""
import json
from fractions import Fraction

import numpy as np
import pytest

import kvgen
from oracle import symmetric as S
from conftest import golden_path


def _load(name):
    with open(golden_path(name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ bit-width table, packed_dim
def test_qmax_table_is_explicit_and_rejects_unknown_widths():
    assert S.QMAX == {8: 127, 6: 31, 4: 7}
    for bad in (0, 2, 3, 5, 7, 16, "6"):
        with pytest.raises(ValueError):
            S.qmax_for(bad)


def test_packed_dim_matches_page():
    g = _load("storage.json")
    for bits, pd in g["packed_dim_256"].items():
        assert S.packed_dim(256, int(bits)) == pd
    assert S.packed_dim(64, 6) == 48 and S.packed_dim(4, 6) == 3
    with pytest.raises(ValueError):
        S.packed_dim(6, 6)          # q6 requires D % 4 == 0
    with pytest.raises(ValueError):
        S.packed_dim(5, 4)          # q4 requires D % 2 == 0


# ------------------------------------------------------------------ q6 byte layout
def test_q6_golden_quadruples():
    for case in _load("q6_byte_layout.json")["cases"]:
        u = np.array(case["u"])
        got = S.pack_fields(u, 6).tobytes().hex()
        assert got == case["bytes"], case
        raw = np.frombuffer(bytes.fromhex(case["bytes"]), np.uint8)
        assert np.array_equal(S.unpack_fields(raw, 6, 4), u)


def test_q6_bruteforce_every_quadruple_is_a_24bit_little_endian_word():
    """All 64^4 quadruples: the page's three byte formulas equal the little-endian bytes of
    w = u0 | u1<<6 | u2<<12 | u3<<18, and unpack(pack(u)) == u."""
    r = np.arange(64, dtype=np.int64)
    u1, u2, u3 = np.meshgrid(r, r, r, indexing="ij")
    u1, u2, u3 = u1.ravel(), u2.ravel(), u3.ravel()
    for a in range(64):
        u0 = np.full_like(u1, a)
        u = np.stack([u0, u1, u2, u3], axis=-1)
        packed = S.pack_fields(u, 6)
        w = u0 | (u1 << 6) | (u2 << 12) | (u3 << 18)
        expect = np.stack([w & 0xFF, (w >> 8) & 0xFF, (w >> 16) & 0xFF], axis=-1)
        assert np.array_equal(packed, expect.astype(np.uint8))
        assert np.array_equal(S.unpack_fields(packed, 6, 4), u)


def test_q6_single_lane_values():
    """4 lanes x 64 values, the others zero: the value lands in the bits the formula says."""
    for lane in range(4):
        for v in range(64):
            u = np.zeros(4, dtype=np.int64)
            u[lane] = v
            b = S.pack_fields(u, 6).astype(np.int64)
            word = int(b[0]) | int(b[1]) << 8 | int(b[2]) << 16
            assert word == v << (6 * lane)


def _bitstream_pack(fields, bits):
    """Independent packer: append each field's bits, least significant first, to a bit stream."""
    out = []
    acc, n = 0, 0
    for f in fields:
        for k in range(bits):
            acc |= ((int(f) >> k) & 1) << n
            n += 1
            if n == 8:
                out.append(acc)
                acc, n = 0, 0
    assert n == 0
    return bytes(out)


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_packing_is_an_lsb_first_bit_stream(bits):
    rng = np.random.default_rng(7)
    for D in (4, 8, 64, 256):
        u = rng.integers(0, 1 << bits, size=D)
        assert S.pack_fields(u, bits).tobytes() == _bitstream_pack(u, bits)


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_unpack_is_defined_on_every_byte_string(bits):
    rng = np.random.default_rng(11)
    D = 256
    raw = rng.integers(0, 256, size=(1000, S.packed_dim(D, bits)), dtype=np.int64).astype(np.uint8)
    u = S.unpack_fields(raw, bits, D)
    assert u.min() >= 0 and u.max() < (1 << bits)
    assert np.array_equal(S.pack_fields(u, bits), raw)
    c = S.unpack(raw, bits, D)
    assert c.min() >= -(1 << (bits - 1)) and c.max() <= (1 << (bits - 1)) - 1


# ------------------------------------------------------------------ hand-worked rows
def test_golden_rows():
    for row in _load("symmetric_rows.json")["rows"]:
        bits = row["bits"]
        x = np.array([row["x"]], dtype=np.float16)
        assert np.array_equal(x.astype(np.float64)[0], np.array(row["x"])), row["name"]
        scale, codes = S.quantize_rows(x, bits)
        assert f"{int(scale.view(np.uint16)[0]):04x}" == row["scale_bits"], row["name"]
        assert codes[0].tolist() == row["codes"], row["name"]
        assert S.pack(codes, bits)[0].tobytes().hex() == row["packed"], row["name"]
        xhat = S.dequantize_rows(codes, scale)[0]
        assert xhat.astype(np.float64).tolist() == row["xhat"], row["name"]
        back = S.unpack(np.frombuffer(bytes.fromhex(row["packed"]), np.uint8), bits, x.shape[1])
        assert back.tolist() == row["codes"], row["name"]


# ------------------------------------------------------------------ properties on random rows
def _random_rows(n, D, seed):
    """Rows spanning many magnitudes (incl. subnormal-scale rows), outliers and zeros."""
    rng = np.random.default_rng(seed)
    base = kvgen.normal_fp16_np(seed, 99, np.arange(n * D)).reshape(n, D).astype(np.float32)
    mag = np.float32(2.0) ** rng.integers(-26, 12, size=(n, 1)).astype(np.float32)
    x = base * mag
    x[rng.random((n, D)) < 0.01] *= 10
    x[::97] = 0
    return np.clip(x, -65504, 65504).astype(np.float16)


def _f16_ulp(v):
    v = np.abs(v.astype(np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -14)))
    return 2.0 ** (e - 10)


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_scale_is_fp16_nearest_to_amax_over_qmax(bits):
    """Exact rational amax/qmax: the stored scale is the nearest fp16 (either neighbour only when
    the quotient sits within 2^-23 relative of an fp16 midpoint, where the float32 step may
    round first)."""
    x = _random_rows(400, 64, 1)
    scale, _ = S.quantize_rows(x, bits)
    qmax = S.QMAX[bits]
    for i in range(x.shape[0]):
        amax = Fraction(float(np.max(np.abs(x[i].astype(np.float64)))))
        q = amax / qmax
        s = Fraction(float(scale[i]))
        if q == 0:
            assert s == 0
            continue
        lo = Fraction(float(np.float16(float(q))))
        # neighbours of the float64-rounded candidate
        cands = {Fraction(float(v)) for v in
                 (np.nextafter(np.float16(lo), np.float16(-1)), np.float16(lo),
                  np.nextafter(np.float16(lo), np.float16(np.inf)))}
        best = min(abs(c - q) for c in cands)
        err = abs(s - q)
        assert err == best or abs(err - best) <= q * Fraction(1, 1 << 23), (i, float(q), float(s))


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_codes_are_nearest_against_stored_scale(bits):
    """|x/scale - c| <= 1/2 (+ the float32 quotient's rounding) for the stored fp16 scale, except
    where the clip bound applies (then |x|/scale lies just above qmax).  A code computed against
    the unrounded amax/qmax breaks this."""
    x = _random_rows(3000, 256, 2)
    scale, codes = S.quantize_rows(x, bits)
    qmax = S.QMAX[bits]
    s = scale.astype(np.float64)
    normal = s >= 2.0 ** -14
    r = x.astype(np.float64)[normal] / s[normal, None]
    c = codes[normal].astype(np.float64)
    dev = np.abs(r - c)
    clipped = (np.abs(c) == qmax) & (np.abs(r) > qmax)
    assert np.all(dev[~clipped] <= 0.5 + 2.0 ** -17)
    assert np.all(np.abs(r[clipped]) <= qmax * (1 + 2.0 ** -10))
    assert np.all(np.sign(r[clipped]) == np.sign(c[clipped]))


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_roundtrip_error_bound(bits):
    """|x - x_hat| <= scale*(1/2 + 2^-17) + ulp16(x_hat)/2 for fp16-normal scales; all-zero and
    underflowed rows reconstruct to 0."""
    x = _random_rows(3000, 256, 3)
    scale, codes = S.quantize_rows(x, bits)
    xhat = S.dequantize_rows(codes, scale)
    s = scale.astype(np.float64)
    normal = s >= 2.0 ** -14
    err = np.abs(x.astype(np.float64) - xhat.astype(np.float64))
    bound = s[:, None] * (0.5 + 2.0 ** -17) + 0.5 * _f16_ulp(xhat)
    assert np.all(err[normal] <= bound[normal])
    zero = s == 0
    assert np.all(xhat[zero] == 0) and np.all(codes[zero] == 0)
    frac = float(np.mean(err[normal] > 0.5 * s[normal][:, None]))
    assert frac < 0.01   # plain scale/2 fails only by the final fp16 rounding, rarely


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_amax_element_gets_qmax(bits):
    x = _random_rows(2000, 128, 4)
    scale, codes = S.quantize_rows(x, bits)
    normal = scale.astype(np.float64) >= 2.0 ** -14
    i = np.argmax(np.abs(x.astype(np.float32)), axis=1)
    c = codes[np.arange(len(i)), i]
    assert np.all(np.abs(c[normal]) == S.QMAX[bits])


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_exact_grid_rows_roundtrip_exactly(bits):
    """x = k * 2^e with integer |k| <= qmax and some |k| = qmax: the scale is exactly 2^e and
    the codes are k."""
    qmax = S.QMAX[bits]
    rng = np.random.default_rng(5)
    for e in (-20, -8, 0, 3):
        k = rng.integers(-qmax, qmax + 1, size=(50, 32))
        k[:, 0] = qmax * np.where(rng.random(50) < 0.5, -1, 1)
        x = (k.astype(np.float64) * 2.0 ** e).astype(np.float16)
        scale, codes = S.quantize_rows(x, bits)
        assert np.all(scale.astype(np.float64) == 2.0 ** e)
        assert np.array_equal(codes, k)
        assert np.array_equal(S.dequantize_rows(codes, scale), x)


# ------------------------------------------------------------------ paged scatter / gather
def _expected_location(pt, s, pos, ps):
    return int(pt[s][pos // ps]), pos % ps


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_paged_scatter_places_every_row_through_the_page_table(bits):
    H, D, ps = 2, 16, 4
    lens = [0, 5, 8, 13]
    pages_per_seq = 4
    pt = kvgen.random_page_table(1, len(lens), pages_per_seq)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    x = _random_rows(int(cu[-1]) * H, D, 6).reshape(-1, H, D)
    pool = S.PagedPool(bits, H, D, ps, pt.size)
    S.quant_pack_paged(pool, x, pt, cu, np.zeros(len(lens), np.int32))
    for s, n in enumerate(lens):
        for t in range(n):
            page, slot = _expected_location(pt, s, t, ps)
            for h in range(H):
                packed, scale = S.quant_pack_rows(x[cu[s] + t, h][None], bits)
                assert np.array_equal(pool.codes[page, h, slot], packed[0])
                assert pool.scales[page, h, slot].view(np.uint16) == scale.view(np.uint16)[0]
    back = S.dequant_paged(pool, pt, cu, np.zeros(len(lens), np.int32))
    sc, cd = S.quantize_rows(x, bits)
    assert np.array_equal(back.view(np.uint16), S.dequantize_rows(cd, sc).view(np.uint16))


def test_append_into_partial_pages_equals_one_shot():
    bits, H, D, ps = 6, 2, 8, 4
    lens0, add = np.array([3, 4, 6]), np.array([1, 5, 2])
    pt = kvgen.random_page_table(2, 3, 4)
    full = _random_rows(int((lens0 + add).sum()) * H, D, 7).reshape(-1, H, D)
    cu_full = np.concatenate([[0], np.cumsum(lens0 + add)])
    one = S.PagedPool(bits, H, D, ps, pt.size)
    S.quant_pack_paged(one, full, pt, cu_full, np.zeros(3, np.int32))
    two = S.PagedPool(bits, H, D, ps, pt.size)
    first = np.concatenate([full[cu_full[s]:cu_full[s] + lens0[s]] for s in range(3)])
    second = np.concatenate([full[cu_full[s] + lens0[s]:cu_full[s + 1]] for s in range(3)])
    S.quant_pack_paged(two, first, pt, np.concatenate([[0], np.cumsum(lens0)]), np.zeros(3))
    S.quant_pack_paged(two, second, pt, np.concatenate([[0], np.cumsum(add)]), lens0)
    assert np.array_equal(one.codes, two.codes)
    assert np.array_equal(one.scales.view(np.uint16), two.scales.view(np.uint16))
