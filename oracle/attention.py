"""Decode attention over a quantized paged KV cache (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", description:
no kernel consumes the packed bytes; plain KV quant dequantizes and then runs SDPA.  So the
oracle's attention is exactly that: dequantize the cache with the oracle's own quantizer, then
compute softmax(q . k_hat * scale) . v_hat per query head, here in float64.

Readings where the pages are silent:
* one decode query per sequence attends to every cached token of that sequence (no mask);
* grouped-query attention maps query head j to KV head j // (Hq / H);
* the softmax is the max-subtracted exponential normalised by its sum;
* a sequence with no tokens has output 0.
"""
from __future__ import annotations

import numpy as np

from . import symmetric


def attend(q16: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, softmax_scale: float
           ) -> np.ndarray:
    """q16 [Hq, D]; k_hat, v_hat [T, H, D] (fp16, dequantized) -> float64 [Hq, D]."""
    Hq, D = q16.shape
    T, H, _ = k_hat.shape
    if Hq % H:
        raise ValueError("query heads must be a multiple of KV heads")
    G = Hq // H
    out = np.zeros((Hq, D), dtype=np.float64)
    if T == 0:
        return out
    q = q16.astype(np.float64)
    for j in range(Hq):
        h = j // G
        k = k_hat[:, h, :].astype(np.float64)
        v = v_hat[:, h, :].astype(np.float64)
        s = (k @ q[j]) * softmax_scale
        p = np.exp(s - s.max())
        out[j] = (p @ v) / p.sum()
    return out


def gather_dequant(pool: symmetric.PagedPool, page_table: np.ndarray, seq: int, length: int,
                   heads=None) -> np.ndarray:
    """Dequantize tokens [0, length) of one sequence -> fp16 [length, H, D] (heads subset
    optional; absent heads are left 0)."""
    out = np.zeros((length, pool.H, pool.D), dtype=np.float16)
    if length == 0:
        return out
    page, slot = symmetric.locate(page_table, seq, np.arange(length), pool.page_size)
    for h in (range(pool.H) if heads is None else heads):
        out[:, h] = symmetric.dequant_rows(pool.codes[page, h, slot],
                                           pool.scales[page, h, slot], pool.bits, pool.D)
    return out


def decode_attention_paged(q16: np.ndarray, k_pool: symmetric.PagedPool,
                           v_pool: symmetric.PagedPool, page_table: np.ndarray,
                           seq_lens: np.ndarray, softmax_scale: float) -> np.ndarray:
    """q16 [nseq, Hq, D] -> float64 [nseq, Hq, D] over the packed pools."""
    nseq, Hq, D = q16.shape
    out = np.zeros((nseq, Hq, D), dtype=np.float64)
    for s in range(nseq):
        n = int(seq_lens[s])
        k_hat = gather_dequant(k_pool, page_table, s, n)
        v_hat = gather_dequant(v_pool, page_table, s, n)
        out[s] = attend(q16[s], k_hat, v_hat, softmax_scale)
    return out


def append_decode_paged(q16: np.ndarray, k_pool: symmetric.PagedPool,
                        v_pool: symmetric.PagedPool, k_new16: np.ndarray, v_new16: np.ndarray,
                        page_table: np.ndarray, seq_lens: np.ndarray, softmax_scale: float
                        ) -> np.ndarray:
    """One decode step as the pages run it, in their order: quantize-on-write of every sequence's
    new token (k_new16, v_new16 [nseq, H, D]) at position seq_lens[s] through the page table,
    then dequantize the active window of seq_lens[s] + 1 tokens and attend.  The pools are
    updated in place.  q16 [nseq, Hq, D] -> float64 [nseq, Hq, D]."""
    lens = np.asarray(seq_lens, dtype=np.int64)
    cu = np.arange(len(lens) + 1)
    symmetric.quant_pack_paged(k_pool, k_new16, page_table, cu, lens)
    symmetric.quant_pack_paged(v_pool, v_new16, page_table, cu, lens)
    return decode_attention_paged(q16, k_pool, v_pool, page_table, lens + 1, softmax_scale)


def decode_attention_fp16(q16: np.ndarray, k16: np.ndarray, v16: np.ndarray, bits: int,
                          softmax_scale: float) -> np.ndarray:
    """Quantize an fp16 cache k16, v16 [T, H, D] with the oracle, dequantize, attend -> [Hq, D]."""
    ks, kc = symmetric.quantize_rows(k16, bits)
    vs, vc = symmetric.quantize_rows(v16, bits)
    return attend(q16, symmetric.dequantize_rows(kc, ks), symmetric.dequantize_rows(vc, vs),
                  softmax_scale)
