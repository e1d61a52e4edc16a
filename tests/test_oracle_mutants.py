"""The oracle's pins reject plausible mistakes.

Each test plants one mistake in a copy of an oracle function (monkeypatched, CPU only). Then it
runs the pins that should catch it and requires at least one of them to fail.  The mistakes are
the kind a restatement of the pages could make:
- a scale kept in float32 instead of rounded to fp16;
- ties rounded away from zero;
- a q6 bias of 31;
- two q6 fields swapped in the byte layout;
- a KIVI divisor of levels + 1;
- a floor instead of a round;
- an off-by-one residual boundary;
- a dropped softmax scale;
- a GQA head map taken modulo the KV heads;
- the outlier tie broken toward the higher position;
- a paged scatter that ignores the page table;
- packed KIVI codes by floor;
- a packed KIVI zero point at the group maximum;
- an attention window missing its last token;
- a side-channel dense row that keeps its outliers.
"""
import numpy as np
import pytest

import test_oracle_attention as TA
import test_oracle_kivi as TK
import test_oracle_kivi_packed as TP
import test_oracle_side as TS
import test_oracle_symmetric as TY
from oracle import attention as A
from oracle import kivi as K
from oracle import kivi_packed as P
from oracle import side as SD
from oracle import symmetric as S


def _rejected(*pins):
    """True if at least one pin (a callable taking no arguments) fails."""
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError):
            return True
    return False


def _symmetric_pins():
    return (TY.test_golden_rows,
            lambda: TY.test_codes_are_nearest_against_stored_scale(6),
            lambda: TY.test_roundtrip_error_bound(6))


def test_the_unmutated_oracle_passes_every_pin_used_here():
    assert not _rejected(*_symmetric_pins(), TY.test_q6_golden_quadruples,
                         TK.test_golden_roundtrips, TK.test_golden_boundary,
                         TA.test_two_tokens_closed_form,
                         lambda: TA.test_matches_torch_sdpa_float64(37, 2, 3, 64),
                         TS.test_selection_brute_force_with_ties)


# ------------------------------------------------------------------ symmetric quantizer
def _quantize_with(scale_fn, round_fn):
    def quantize_rows(x16, bits):
        qmax = S.qmax_for(bits)
        x32 = np.asarray(x16, np.float16).astype(np.float32)
        amax = np.max(np.abs(x32), axis=-1)
        s32 = scale_fn(amax, qmax)
        zero = s32 == 0
        with np.errstate(divide="ignore", invalid="ignore"):
            q = x32 / s32[..., None]
        codes = np.clip(round_fn(q), -qmax, qmax)
        codes[zero] = 0
        return s32.astype(np.float16), codes.astype(np.int32)
    return quantize_rows


def _fp16_scale(amax, qmax):
    return (amax / np.float32(qmax)).astype(np.float16).astype(np.float32)


def test_scale_not_rounded_to_fp16_is_rejected(monkeypatch):
    monkeypatch.setattr(S, "quantize_rows",
                        _quantize_with(lambda a, q: a / np.float32(q), np.rint))
    assert _rejected(*_symmetric_pins())


def test_ties_away_from_zero_are_rejected(monkeypatch):
    away = lambda q: np.sign(q) * np.floor(np.abs(q) + 0.5)   # noqa: E731
    monkeypatch.setattr(S, "quantize_rows", _quantize_with(_fp16_scale, away))
    assert _rejected(*_symmetric_pins())


def test_wrong_q6_bias_is_rejected(monkeypatch):
    monkeypatch.setattr(S, "BIAS", {8: 0, 6: 31, 4: 8})
    assert _rejected(TY.test_golden_rows)


def test_swapped_q6_fields_are_rejected(monkeypatch):
    orig = S.pack_fields

    def pack_fields(u, bits):
        u = np.asarray(u, dtype=np.int64)
        if bits != 6:
            return orig(u, bits)
        q = u.reshape(u.shape[:-1] + (u.shape[-1] // 4, 4)).copy()
        q[..., [1, 2]] = q[..., [2, 1]]                   # u1 and u2 trade places
        return orig(q.reshape(u.shape), 6)
    monkeypatch.setattr(S, "pack_fields", pack_fields)
    assert _rejected(TY.test_q6_golden_quadruples)


# ------------------------------------------------------------------ KIVI
def _kivi_with(levels_off=0, round_fn=np.rint):
    def quant_dequant_along(x, axis, group_size, levels, eps=1e-8):
        gs = int(group_size)
        x32 = np.asarray(x).astype(np.float32)
        L = x32.shape[axis]
        ng = (L + gs - 1) // gs
        xm = np.moveaxis(x32, axis, -1)
        if ng * gs - L:
            xm = np.concatenate([xm, np.repeat(xm[..., -1:], ng * gs - L, axis=-1)], axis=-1)
        xg = xm.reshape(xm.shape[:-1] + (ng, gs))
        gmin, gmax = xg.min(-1, keepdims=True), xg.max(-1, keepdims=True)
        scale = np.maximum((gmax - gmin) / np.float32(levels + levels_off), np.float32(eps))
        codes = np.clip(round_fn((xg - gmin) / scale), 0, levels)
        recon = (codes * scale + gmin).reshape(xm.shape)[..., :L]
        return np.moveaxis(recon, -1, axis).astype(np.asarray(x).dtype)
    return quant_dequant_along


def test_kivi_golden_pins_pass_the_restated_round_trip(monkeypatch):
    monkeypatch.setattr(K, "quant_dequant_along", _kivi_with())
    assert not _rejected(TK.test_golden_roundtrips)


def test_kivi_levels_off_by_one_is_rejected(monkeypatch):
    monkeypatch.setattr(K, "quant_dequant_along", _kivi_with(levels_off=1))
    assert _rejected(TK.test_golden_roundtrips)


def test_kivi_floor_instead_of_round_is_rejected(monkeypatch):
    monkeypatch.setattr(K, "quant_dequant_along", _kivi_with(round_fn=np.floor))
    assert _rejected(TK.test_golden_roundtrips)


def test_kivi_boundary_off_by_one_is_rejected(monkeypatch):
    def boundary(offset, residual_length, group_size):
        aged = max(0, offset - residual_length + 1)
        return (aged // group_size) * group_size
    monkeypatch.setattr(K, "quantization_boundary", boundary)
    assert _rejected(TK.test_golden_boundary)


# ------------------------------------------------------------------ attention
def _attend_with(scale_used=True, head_map=lambda j, G, H: j // G):
    def attend(q16, k_hat, v_hat, softmax_scale):
        Hq, D = q16.shape
        T, H, _ = k_hat.shape
        G = Hq // H
        out = np.zeros((Hq, D))
        if T == 0:
            return out
        for j in range(Hq):
            h = head_map(j, G, H)
            k = k_hat[:, h, :].astype(np.float64)
            v = v_hat[:, h, :].astype(np.float64)
            s = (k @ q16[j].astype(np.float64)) * (softmax_scale if scale_used else 1.0)
            p = np.exp(s - s.max())
            out[j] = (p @ v) / p.sum()
        return out
    return attend


def _attention_pins():
    return (TA.test_two_tokens_closed_form,
            lambda: TA.test_matches_torch_sdpa_float64(37, 2, 3, 64))


def test_attention_restatement_passes(monkeypatch):
    monkeypatch.setattr(A, "attend", _attend_with())
    assert not _rejected(*_attention_pins())


def test_dropped_softmax_scale_is_rejected(monkeypatch):
    monkeypatch.setattr(A, "attend", _attend_with(scale_used=False))
    assert _rejected(*_attention_pins())


def test_gqa_head_map_modulo_is_rejected(monkeypatch):
    monkeypatch.setattr(A, "attend", _attend_with(head_map=lambda j, G, H: j % H))
    assert _rejected(*_attention_pins())


# ------------------------------------------------------------------ side channels
def test_outlier_tie_toward_higher_position_is_rejected(monkeypatch):
    def split_outliers(x16, k):
        D = x16.shape[-1]
        rows = x16.reshape(-1, D)
        mag = np.abs(rows.astype(np.float64))[:, ::-1]            # reversed: later first on ties
        order = (D - 1) - np.argsort(-mag, axis=1, kind="stable")
        pos = np.sort(order[:, :k], axis=1)
        dense = rows.copy()
        np.put_along_axis(dense, pos, np.float16(0), axis=1)
        val = np.take_along_axis(rows, pos, axis=1)
        shape = x16.shape[:-1]
        return (dense.reshape(x16.shape), pos.astype(np.uint8).reshape(shape + (k,)),
                val.reshape(shape + (k,)))
    monkeypatch.setattr(SD, "split_outliers", split_outliers)
    assert _rejected(TS.test_selection_brute_force_with_ties)


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_symmetric_restatement_passes(monkeypatch, bits):
    monkeypatch.setattr(S, "quantize_rows", _quantize_with(_fp16_scale, np.rint))
    assert not _rejected(TY.test_golden_rows,
                         lambda: TY.test_codes_are_nearest_against_stored_scale(bits))


# ------------------------------------------------------------------ paged scatter, packed KIVI
def test_scatter_ignoring_the_page_table_is_rejected(monkeypatch):
    def locate(page_table, seq, pos, page_size):
        pos = np.asarray(pos, dtype=np.int64)
        return seq * page_table.shape[1] + pos // page_size, pos % page_size
    monkeypatch.setattr(S, "locate", locate)
    assert _rejected(lambda: TY.test_paged_scatter_places_every_row_through_the_page_table(6))


def test_scatter_restatement_passes(monkeypatch):
    def locate(page_table, seq, pos, page_size):
        pos = np.asarray(pos, dtype=np.int64)
        return page_table[seq, pos // page_size].astype(np.int64), pos % page_size
    monkeypatch.setattr(S, "locate", locate)
    assert not _rejected(lambda: TY.test_paged_scatter_places_every_row_through_the_page_table(6))


def _packed_codes_with(round_fn):
    def _codes(x32, zero32, scale16, levels):
        s32 = scale16.astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            q = (x32 - zero32) / s32
        c = np.where(s32 == 0, 0, np.clip(round_fn(q), 0, levels))
        return c.astype(np.int64)
    return _codes


def test_packed_kivi_restatement_passes(monkeypatch):
    monkeypatch.setattr(P, "_codes", _packed_codes_with(np.rint))
    assert not _rejected(TP.test_golden_keys, TP.test_golden_values,
                         lambda: TP.test_codes_nearest_against_stored_scale_and_error_bound(2))


def test_packed_kivi_floor_codes_are_rejected(monkeypatch):
    monkeypatch.setattr(P, "_codes", _packed_codes_with(np.floor))
    assert _rejected(TP.test_golden_keys, TP.test_golden_values,
                     lambda: TP.test_codes_nearest_against_stored_scale_and_error_bound(2))


def test_packed_kivi_zero_at_the_group_max_is_rejected(monkeypatch):
    def _params(gmin32, gmax32, levels, eps):
        scale32 = np.maximum((gmax32 - gmin32) / np.float32(levels), np.float32(eps))
        return scale32.astype(np.float16), gmax32.astype(np.float16)
    monkeypatch.setattr(P, "_params", _params)
    assert _rejected(TP.test_golden_keys, TP.test_golden_values,
                     lambda: TP.test_codes_nearest_against_stored_scale_and_error_bound(2))


# ------------------------------------------------------------------ windows and dense rows
def test_attention_window_missing_its_last_token_is_rejected(monkeypatch):
    orig = A.gather_dequant

    def gather_dequant(pool, page_table, seq, length, heads=None):
        out = orig(pool, page_table, seq, length, heads)
        return out[:-1] if length > 1 else out
    monkeypatch.setattr(A, "gather_dequant", gather_dequant)
    assert _rejected(lambda: TA.test_paged_equals_contiguous(6))


def test_side_dense_row_keeping_its_outliers_is_rejected(monkeypatch):
    orig = SD.split_outliers

    def split_outliers(x16, k):
        _, pos, val = orig(x16, k)
        return x16.copy(), pos, val      # mistake: the outliers stay in the dense row
    monkeypatch.setattr(SD, "split_outliers", split_outliers)
    assert _rejected(lambda: TS.test_dense_scale_exact_outliers_and_round_trip_bound(6, 3))
