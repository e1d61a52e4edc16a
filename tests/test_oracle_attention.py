"""Pins for the oracle's decode attention (dequantize, then softmax(q k^T * scale) v in float64).

Source: MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", description
(plain KV quant dequantizes and runs SDPA).  Pinned to textbook special cases (one token; equal
keys -> uniform weights; two tokens in closed form) and to PyTorch's
scaled_dot_product_attention in float64 as an independent library routine.
"""
import math

import numpy as np
import pytest
import torch

import kvgen
from oracle import attention as A
from oracle import symmetric as S


def _fp16(shape, seed, tag=60):
    return kvgen.normal_fp16_np(seed, tag, np.arange(int(np.prod(shape)))).reshape(shape)


def test_single_token_returns_its_value():
    q = _fp16((6, 32), 1)
    k = _fp16((1, 1, 32), 2)
    v = _fp16((1, 1, 32), 3)
    out = A.attend(q, k, v, 0.25)
    assert np.array_equal(out, np.repeat(v[0].astype(np.float64), 6, axis=0))


def test_equal_keys_give_the_mean_of_values():
    q = _fp16((4, 16), 4)
    k = np.repeat(_fp16((1, 2, 16), 5), 50, axis=0)
    v = _fp16((50, 2, 16), 6)
    out = A.attend(q, k, v, 1.0)
    for j in range(4):
        assert np.allclose(out[j], v[:, j // 2].astype(np.float64).mean(0), rtol=0, atol=1e-12)


def test_two_tokens_closed_form():
    # scores 0 and 1: weights 1/(1+e) and e/(1+e)
    q = np.zeros((1, 4), np.float16)
    q[0, 0] = 1
    k = np.zeros((2, 1, 4), np.float16)
    k[1, 0, 0] = 1
    v = np.array([[[1, 0, 0, 2]], [[0, 1, 0, -2]]], np.float16)
    out = A.attend(q, k, v, 1.0)[0]
    e = math.e
    expect = np.array([1 / (1 + e), e / (1 + e), 0, 2 / (1 + e) - 2 * e / (1 + e)])
    assert np.allclose(out, expect, rtol=0, atol=1e-15)


@pytest.mark.parametrize("T,H,G,D", [(1, 1, 1, 8), (37, 2, 3, 64), (300, 4, 6, 256)])
def test_matches_torch_sdpa_float64(T, H, G, D):
    q = _fp16((H * G, D), 7)
    k = _fp16((T, H, D), 8)
    v = _fp16((T, H, D), 9)
    out = A.attend(q, k, v, 1.0 / math.sqrt(D))
    qt = torch.from_numpy(q.astype(np.float64)).view(1, H * G, 1, D)
    kt = torch.from_numpy(k.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    vt = torch.from_numpy(v.astype(np.float64)).permute(1, 0, 2).repeat_interleave(G, 0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=1.0 / math.sqrt(D))
    assert np.allclose(out, ref.view(H * G, D).numpy(), rtol=1e-12, atol=1e-13)


def test_empty_sequence_is_zero():
    out = A.attend(_fp16((6, 8), 1), np.zeros((0, 1, 8), np.float16),
                   np.zeros((0, 1, 8), np.float16), 1.0)
    assert np.all(out == 0)


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_paged_equals_contiguous(bits):
    H, G, D, ps = 2, 3, 32, 4
    lens = np.array([0, 1, 9, 16], np.int32)
    pt = kvgen.random_page_table(3, len(lens), 4)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    k = _fp16((int(cu[-1]), H, D), 10)
    v = _fp16((int(cu[-1]), H, D), 11)
    kp, vp = S.PagedPool(bits, H, D, ps, pt.size), S.PagedPool(bits, H, D, ps, pt.size)
    S.quant_pack_paged(kp, k, pt, cu, np.zeros(4, np.int32))
    S.quant_pack_paged(vp, v, pt, cu, np.zeros(4, np.int32))
    q = _fp16((len(lens), H * G, D), 12)
    out = A.decode_attention_paged(q, kp, vp, pt, lens, 0.125)
    for s in range(len(lens)):
        ref = A.decode_attention_fp16(q[s], k[cu[s]:cu[s + 1]], v[cu[s]:cu[s + 1]], bits, 0.125)
        assert np.array_equal(out[s], ref)


# ---------------------------------------------------------------- fused append + decode step
def _pools(bits, H, D, ps, pages):
    return S.PagedPool(bits, H, D, ps, pages), S.PagedPool(bits, H, D, ps, pages)


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_append_decode_on_empty_caches_returns_the_new_value(bits):
    """One cached token after the append: softmax of one score is 1, so every query head of KV
    head h returns the dequantized new value row of h."""
    nseq, H, G, D, ps = 3, 2, 3, 32, 16
    kp, vp = _pools(bits, H, D, ps, 8)
    pt = np.arange(nseq * 2).reshape(nseq, 2)
    kn, vn, q = _fp16((nseq, H, D), 11), _fp16((nseq, H, D), 12), _fp16((nseq, H * G, D), 13)
    out = A.append_decode_paged(q, kp, vp, kn, vn, pt, np.zeros(nseq, np.int64), 0.1)
    v_hat = S.dequant_rows(*S.quant_pack_rows(vn, bits), bits, D)
    for s in range(nseq):
        for j in range(H * G):
            assert np.array_equal(out[s, j], v_hat[s, j // G].astype(np.float64))


@pytest.mark.parametrize("bits", [6, 4])
def test_append_decode_writes_exactly_the_new_rows(bits):
    """The pools change only at (page_table[s][len // ps], h, len % ps), where they hold the
    quantizer's packed row and scale of the new token; a page boundary (len % ps == 0) is
    crossed for one sequence."""
    nseq, H, D, ps = 3, 2, 32, 16
    lens = np.array([5, 16, 31])
    pt = kvgen.random_page_table(4, nseq, 3)
    kp, vp = _pools(bits, H, D, ps, nseq * 3)
    kp.codes[:] = 0xA5
    kp.scales[:] = np.float16(0.5)
    before_c, before_s = kp.codes.copy(), kp.scales.copy()
    kn, vn, q = _fp16((nseq, H, D), 21), _fp16((nseq, H, D), 22), _fp16((nseq, 2 * H, D), 23)
    A.append_decode_paged(q, kp, vp, kn, vn, pt, lens, 0.2)
    packed, scale = S.quant_pack_rows(kn, bits)
    changed = np.zeros(kp.scales.shape, bool)
    for s in range(nseq):
        page, slot = pt[s, lens[s] // ps], lens[s] % ps
        changed[page, :, slot] = True
        assert np.array_equal(kp.codes[page, :, slot], packed[s])
        assert np.array_equal(kp.scales[page, :, slot].view(np.uint16), scale[s].view(np.uint16))
    assert np.array_equal(kp.codes[~changed], before_c[~changed])
    assert np.array_equal(kp.scales[~changed].view(np.uint16), before_s[~changed].view(np.uint16))


def test_append_decode_two_tokens_closed_form():
    """A cache of one token plus the new one: the weight of the new token is the logistic
    function of the score difference, o = v0 + (v1 - v0) / (1 + exp(s0 - s1))."""
    bits, H, D, ps = 8, 1, 16, 16
    kp, vp = _pools(bits, H, D, ps, 1)
    pt = np.zeros((1, 1), np.int64)
    k0, v0 = _fp16((1, H, D), 31), _fp16((1, H, D), 32)
    S.quant_pack_paged(kp, k0, pt, np.array([0, 1]), np.array([0]))
    S.quant_pack_paged(vp, v0, pt, np.array([0, 1]), np.array([0]))
    k1, v1, q = _fp16((1, H, D), 33), _fp16((1, H, D), 34), _fp16((1, 2, D), 35)
    out = A.append_decode_paged(q, kp, vp, k1, v1, pt, np.array([1]), 0.3)
    deq = lambda x: S.dequant_rows(*S.quant_pack_rows(x, bits), bits, D)[0, 0].astype(np.float64)
    kh0, kh1, vh0, vh1 = deq(k0), deq(k1), deq(v0), deq(v1)
    for j in range(2):
        qq = q[0, j].astype(np.float64)
        s0, s1 = 0.3 * float(qq @ kh0), 0.3 * float(qq @ kh1)
        ref = vh0 + (vh1 - vh0) / (1.0 + math.exp(s0 - s1))
        assert np.allclose(out[0, j], ref, rtol=1e-12, atol=1e-12)


def test_append_decode_steps_equal_one_prefill_write():
    """Appending T tokens one decode step at a time leaves the same pools as writing them in one
    quant-pack call (the write is per row, independent of how the tokens are batched)."""
    bits, H, D, ps, T = 6, 2, 32, 16, 40
    pt = kvgen.random_page_table(5, 1, 3)
    kp, vp = _pools(bits, H, D, ps, 3)
    kq, vq = _pools(bits, H, D, ps, 3)
    k, v = _fp16((T, H, D), 41), _fp16((T, H, D), 42)
    q = _fp16((1, H, D), 43)
    for t in range(T):
        A.append_decode_paged(q, kp, vp, k[t:t + 1], v[t:t + 1], pt, np.array([t]), 0.2)
    S.quant_pack_paged(kq, k, pt, np.array([0, T]), np.array([0]))
    S.quant_pack_paged(vq, v, pt, np.array([0, T]), np.array([0]))
    assert np.array_equal(kp.codes, kq.codes) and np.array_equal(vp.codes, vq.codes)
    assert np.array_equal(kp.scales.view(np.uint16), kq.scales.view(np.uint16))
