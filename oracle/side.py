"""fp16 side channels on the symmetric quantizer: attention sinks and dense-and-sparse outliers.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: VeloxQuant-MLX API docs, "veloxquant_mlx.cache.kvquant_cache module": the KVQuant cache
keeps "per-vector dense-and-sparse outlier isolation" with an "fp16 outlier side-channel (value +
position index)" (byte accounting), a default outlier fraction of 0.01 (config fields), and
"Attention Sink-Aware quantization": the first n_sink tokens of the sequence are restored to exact
fp16 and kept out of the fit.  The page's non-uniform (Lloyd-Max) levels are not on the pages and
are not used: the dense part here is the symmetric per-token-per-head quantizer of MTPLX pull
request #267 (module ``symmetric``).

Readings where the pages leave a step open:
* a vector is one (token, KV head) row of D elements;
* a row keeps k = ceil(fraction * D) outliers: its k elements of largest magnitude, ties to the
  lower position (k = 3 at D = 256 and the page's 0.01);
* the dense part is the row with the outliers set to 0, quantized by the symmetric quantizer, so
  its scale comes from the (k+1)-th largest magnitude and the outlier positions store code 0;
* the side channel of a row is k (fp16 value, uint8 position) pairs in ascending position order
  (D <= 256); dequantization writes the exact fp16 values over the dense reconstruction;
* a sink is a token at position < n_sink of its sequence; its K and V rows are kept exactly in an
  fp16 buffer [seq][n_sink][H][D] that dequantization and attention read instead of the pages
  (the packed rows of sinks are still written, as for any row).
"""
from __future__ import annotations

import math

import numpy as np

from . import attention, symmetric


def outlier_count(head_dim: int, fraction: float) -> int:
    """Outliers per row for an outlier fraction (the page's default is 0.01)."""
    if not 0.0 <= fraction < 1.0:
        raise ValueError("outlier fraction must be in [0, 1)")
    return int(math.ceil(fraction * head_dim))


def split_outliers(x16: np.ndarray, k: int):
    """fp16 rows [..., D] -> (dense fp16 [..., D] with the outliers zeroed, positions uint8
    [..., k] ascending, values fp16 [..., k])."""
    D = x16.shape[-1]
    if not 0 <= k < D:
        raise ValueError("need 0 <= k < D")
    rows = x16.reshape(-1, D)
    mag = np.abs(rows.astype(np.float64))
    # largest magnitude first; a stable sort keeps the lower position first among equals
    order = np.argsort(-mag, axis=1, kind="stable")
    pos = np.sort(order[:, :k], axis=1)
    dense = rows.copy()
    np.put_along_axis(dense, pos, np.float16(0), axis=1)
    val = np.take_along_axis(rows, pos, axis=1)
    shape = x16.shape[:-1]
    return (dense.reshape(x16.shape), pos.astype(np.uint8).reshape(shape + (k,)),
            val.reshape(shape + (k,)))


def quant_pack_rows_side(x16: np.ndarray, bits: int, k: int):
    """fp16 rows -> (packed uint8 rows, fp16 scales, positions, values)."""
    dense, pos, val = split_outliers(x16, k)
    packed, scale = symmetric.quant_pack_rows(dense, bits)
    return packed, scale, pos, val


def dequant_rows_side(packed, scale16, pos, val, bits: int, head_dim: int) -> np.ndarray:
    out = symmetric.dequant_rows(packed, scale16, bits, head_dim)
    flat = out.reshape(-1, head_dim)
    if flat.shape[0] == 0:
        return out
    np.put_along_axis(flat, pos.reshape(flat.shape[0], -1).astype(np.int64),
                      val.reshape(flat.shape[0], -1), axis=1)
    return flat.reshape(out.shape)


class SidePool:
    """Side channels of one (layer, K-or-V) pool: outliers per physical row and the sink rows."""

    def __init__(self, pool: symmetric.PagedPool, n_outlier: int, n_sink: int, max_seqs: int):
        self.pool, self.k, self.n_sink = pool, n_outlier, n_sink
        P, H, ps, D = pool.codes.shape[0], pool.H, pool.page_size, pool.D
        self.out_val = np.zeros((P, H, ps, n_outlier), np.float16)
        self.out_idx = np.zeros((P, H, ps, n_outlier), np.uint8)
        self.sink = np.zeros((max_seqs, n_sink, H, D), np.float16)


def quant_pack_paged_side(sp: SidePool, x16: np.ndarray, page_table: np.ndarray,
                          cu_new_tokens: np.ndarray, start_pos: np.ndarray) -> None:
    """As symmetric.quant_pack_paged, with each row's outliers split off, and sink positions
    copied exactly into the sink buffer."""
    pool = sp.pool
    for s in range(len(start_pos)):
        a, b = int(cu_new_tokens[s]), int(cu_new_tokens[s + 1])
        if b == a:
            continue
        pos = int(start_pos[s]) + np.arange(b - a)
        page, slot = symmetric.locate(page_table, s, pos, pool.page_size)
        packed, scale, opos, oval = quant_pack_rows_side(x16[a:b], pool.bits, sp.k)
        for h in range(pool.H):
            pool.codes[page, h, slot] = packed[:, h]
            pool.scales[page, h, slot] = scale[:, h]
            sp.out_idx[page, h, slot] = opos[:, h]
            sp.out_val[page, h, slot] = oval[:, h]
        sink = pos < sp.n_sink
        sp.sink[s, pos[sink]] = x16[a:b][sink]


def gather_dequant_side(sp: SidePool, page_table: np.ndarray, seq: int, length: int) -> np.ndarray:
    """Tokens [0, length) of one sequence -> fp16 [length, H, D]: sinks from the sink buffer, the
    rest dense dequantization with the outliers written back."""
    pool = sp.pool
    out = np.zeros((length, pool.H, pool.D), dtype=np.float16)
    if length == 0:
        return out
    page, slot = symmetric.locate(page_table, seq, np.arange(length), pool.page_size)
    for h in range(pool.H):
        out[:, h] = dequant_rows_side(pool.codes[page, h, slot], pool.scales[page, h, slot],
                                      sp.out_idx[page, h, slot], sp.out_val[page, h, slot],
                                      pool.bits, pool.D)
    n = min(sp.n_sink, length)
    out[:n] = sp.sink[seq, :n]
    return out


def dequant_paged_side(sp: SidePool, page_table: np.ndarray, cu_tokens: np.ndarray,
                       start_pos: np.ndarray) -> np.ndarray:
    """Gather rows cu_tokens[s]..cu_tokens[s+1] of sequence s (positions start_pos[s]...)."""
    pool = sp.pool
    total = int(cu_tokens[-1])
    out = np.zeros((total, pool.H, pool.D), dtype=np.float16)
    for s in range(len(start_pos)):
        a, b = int(cu_tokens[s]), int(cu_tokens[s + 1])
        if b == a:
            continue
        end = int(start_pos[s]) + (b - a)
        out[a:b] = gather_dequant_side(sp, page_table, s, end)[int(start_pos[s]):end]
    return out


def decode_attention_paged_side(q16: np.ndarray, k_side: SidePool, v_side: SidePool,
                                page_table: np.ndarray, seq_lens: np.ndarray,
                                softmax_scale: float) -> np.ndarray:
    """q16 [nseq, Hq, D] -> float64 [nseq, Hq, D]: attention over the side-channel cache."""
    nseq, Hq, D = q16.shape
    out = np.zeros((nseq, Hq, D), dtype=np.float64)
    for s in range(nseq):
        n = int(seq_lens[s])
        out[s] = attention.attend(q16[s], gather_dequant_side(k_side, page_table, s, n),
                                  gather_dequant_side(v_side, page_table, s, n), softmax_scale)
    return out
