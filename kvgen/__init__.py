"""Seeded synthetic K/V workloads, shared by the CUDA path's tests and bench and by the oracle.

This module holds no quantizer, packing, KIVI or attention arithmetic: it only makes inputs.

Every element is a pure function of ``(seed, tag, flat_index)`` (a counter-based generator), so
any row of a multi-gigabyte device tensor can be regenerated on the host, bit for bit, without
materialising the rest.  The same integer recipe is written twice, once over numpy arrays (host)
and once over torch tensors (any device); ``tests/test_kvgen.py`` checks that they agree.

Recipe for one N(0,1) fp16 element at flat index ``i`` (inverse-CDF sampling):

* one 32-bit word ``u = w(2i)``, where ``w(j) = fmix32(fmix32((j + s0) mod 2^32) ^ s1)`` and
  ``fmix32`` is the 32-bit finaliser of Austin Appleby's MurmurHash3 (public domain); ``(s0, s1)``
  are derived from ``(seed, tag)``;
* ``z`` is the standard normal quantile of ``(u + 1/2) / 2^32``, read from a table: nodes
  ``T[k]``, k = 0 .. 2^20, are the float64 quantiles at ``u = 4096 k`` (the last one at
  ``u = 2^32 - 1``) rounded to float32, with float32 slopes ``S[k] = (T[k+1] - T[k]) / 4096``;
  ``z = float32(T[u >> 12] + float32(float32(u & 4095) * S[u >> 12]))`` -- two IEEE float32
  operations, so the numpy and torch implementations agree bit for bit on any device.  The
  tails reach about +-6.3 sigma (the quantile of 2^-33); between nodes the inverse CDF is linear;
* channels chosen as outliers are multiplied by a float32 factor; the result is rounded to fp16
  (round to nearest even).

The shapes, the outlier channels and the zero rows follow the workloads they stand in for.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

MASK32 = 0xFFFFFFFF
_M1 = 0x85EBCA6B
_M2 = 0xC2B2AE35
_GOLDEN = 0x9E3779B1
_QBITS = 20                    # table nodes: 2^20 intervals of 4096 consecutive words
_QSHIFT = 32 - _QBITS
_QTABLE = None                  # (T, S) float32 numpy arrays, built on first use
_QTABLE_T = {}                  # torch copies per device

# tags: distinct generator streams
TAG_K = 1
TAG_V = 2
TAG_Q = 3
TAG_OUTLIER_K = 4
TAG_PAGES = 5
TAG_SEQLEN = 6
TAG_KIVI_K = 7
TAG_KIVI_V = 8
TAG_SAMPLE = 9


def _fmix32_py(h: int) -> int:
    h &= MASK32
    h ^= h >> 16
    h = (h * _M1) & MASK32
    h ^= h >> 13
    h = (h * _M2) & MASK32
    h ^= h >> 16
    return h


def stream_salt(seed: int, tag: int, sub: int = 0) -> tuple[int, int]:
    """Two 32-bit salts for stream (seed, tag, sub)."""
    a = _fmix32_py((seed * _GOLDEN + tag * 0x27D4EB2F + sub * 0x165667B1 + 1) & MASK32)
    b = _fmix32_py((a ^ (seed >> 32) ^ (tag << 16) ^ sub) + 0x7F4A7C15)
    return a, b


# ---------------------------------------------------------------- numpy (host) implementation
def _fmix32_np(h: np.ndarray) -> np.ndarray:
    h = h.astype(np.uint32, copy=True)
    h ^= h >> np.uint32(16)
    h *= np.uint32(_M1)
    h ^= h >> np.uint32(13)
    h *= np.uint32(_M2)
    h ^= h >> np.uint32(16)
    return h


def words_np(seed: int, tag: int, idx: np.ndarray, sub: int = 0) -> np.ndarray:
    """32-bit words w(idx) of stream (seed, tag, sub); idx int64 in [0, 2^32)."""
    s0, s1 = stream_salt(seed, tag, sub)
    idx = np.asarray(idx, dtype=np.int64)
    assert idx.size == 0 or (idx.min() >= 0 and idx.max() <= MASK32)
    x = ((idx + s0) & MASK32).astype(np.uint32)
    return _fmix32_np(_fmix32_np(x) ^ np.uint32(s1))


def _normal_quantiles(p: np.ndarray) -> np.ndarray:
    """Standard normal quantiles in float64: Acklam's rational approximation (relative error
    below 1.2e-9), then one Halley step on erfc, which takes it to float64 accuracy."""
    a = (-3.969683028665376e+01, 2.209460984245205e+02, -2.759285104469687e+02,
         1.383577518672690e+02, -3.066479806614716e+01, 2.506628277459239e+00)
    b = (-5.447609879822406e+01, 1.615858368580409e+02, -1.556989798598866e+02,
         6.680131188771972e+01, -1.328068155288572e+01)
    c = (-7.784894002430293e-03, -3.223964580411365e-01, -2.400758277161838e+00,
         -2.549732539343734e+00, 4.374664141464968e+00, 2.938163982698783e+00)
    d = (7.784695709041462e-03, 3.224671290700398e-01, 2.445134137142996e+00,
         3.754408661907416e+00)
    p = np.asarray(p, dtype=np.float64)
    x = np.empty_like(p)
    lo, hi = p < 0.02425, p > 1 - 0.02425
    mid = ~(lo | hi)
    q = np.sqrt(-2 * np.log(p[lo]))
    x[lo] = ((((((c[0] * q + c[1]) * q + c[2]) * q + c[3]) * q + c[4]) * q + c[5]) /
             ((((d[0] * q + d[1]) * q + d[2]) * q + d[3]) * q + 1))
    q = np.sqrt(-2 * np.log1p(-p[hi]))
    x[hi] = -((((((c[0] * q + c[1]) * q + c[2]) * q + c[3]) * q + c[4]) * q + c[5]) /
              ((((d[0] * q + d[1]) * q + d[2]) * q + d[3]) * q + 1))
    q = p[mid] - 0.5
    r = q * q
    x[mid] = ((((((a[0] * r + a[1]) * r + a[2]) * r + a[3]) * r + a[4]) * r + a[5]) * q /
              (((((b[0] * r + b[1]) * r + b[2]) * r + b[3]) * r + b[4]) * r + 1))
    erfc = np.vectorize(math.erfc)
    e = 0.5 * erfc(-x / math.sqrt(2.0)) - p
    u = e * math.sqrt(2.0 * math.pi) * np.exp(x * x / 2.0)
    return x - u / (1.0 + x * u / 2.0)


def quantile_table() -> tuple[np.ndarray, np.ndarray]:
    """(T, S): float32 nodes and slopes of the inverse-CDF table (see the module docstring)."""
    global _QTABLE
    if _QTABLE is None:
        n = 1 << _QBITS
        u = np.arange(n + 1, dtype=np.float64) * (1 << _QSHIFT)
        u[-1] = float(MASK32)
        t64 = _normal_quantiles((u + 0.5) / 2.0 ** 32)
        t = t64.astype(np.float32)
        slope = ((t[1:].astype(np.float64) - t[:-1].astype(np.float64))
                 / (u[1:] - u[:-1])).astype(np.float32)
        _QTABLE = (t[:-1].copy(), slope)
    return _QTABLE


def normal_fp16_np(seed: int, tag: int, idx: np.ndarray, sub: int = 0,
                   mult: np.ndarray | None = None) -> np.ndarray:
    """fp16 N(0,1) at flat indices idx; optional float32 multiplier per element."""
    idx = np.asarray(idx, dtype=np.int64)
    u = words_np(seed, tag, 2 * idx, sub)
    t, slope = quantile_table()
    k = (u >> np.uint32(_QSHIFT)).astype(np.int64)
    f = (u & np.uint32((1 << _QSHIFT) - 1)).astype(np.float32)
    z = t[k] + f * slope[k]
    if mult is not None:
        z = z * np.asarray(mult, dtype=np.float32)
    return z.astype(np.float16)


# ---------------------------------------------------------------- torch implementation
def _mul32_t(x, m: int):
    # (x * m) mod 2^32 for x in [0, 2^32) without int64 overflow: split x into 16-bit halves.
    return ((x & 0xFFFF) * m + (((x >> 16) * (m & 0xFFFF)) << 16)) & MASK32


def _fmix32_t(h):
    h = h ^ (h >> 16)
    h = _mul32_t(h, _M1)
    h = h ^ (h >> 13)
    h = _mul32_t(h, _M2)
    h = h ^ (h >> 16)
    return h


def words_torch(seed: int, tag: int, idx, sub: int = 0):
    s0, s1 = stream_salt(seed, tag, sub)
    x = (idx + s0) & MASK32
    return _fmix32_t(_fmix32_t(x) ^ s1)


def _quantile_table_torch(device):
    import torch
    key = str(device)
    if key not in _QTABLE_T:
        t, slope = quantile_table()
        _QTABLE_T[key] = (torch.from_numpy(t).to(device), torch.from_numpy(slope).to(device))
    return _QTABLE_T[key]


def normal_fp16_torch(seed: int, tag: int, idx, sub: int = 0, mult=None):
    import torch
    u = words_torch(seed, tag, 2 * idx, sub)
    t, slope = _quantile_table_torch(u.device)
    k = u >> _QSHIFT
    f = (u & ((1 << _QSHIFT) - 1)).to(torch.float32)
    z = t[k] + f * slope[k]
    if mult is not None:
        z = z * mult
    return z.to(torch.float16)


# ---------------------------------------------------------------- structure helpers (numpy only)
def outlier_channels(seed: int, tag: int, num_heads: int, head_dim: int, k: int) -> np.ndarray:
    """[num_heads, k] distinct channel ids per head (fixed for the workload)."""
    if k == 0:
        return np.zeros((num_heads, 0), dtype=np.int64)
    idx = np.arange(num_heads * head_dim, dtype=np.int64)
    w = words_np(seed, TAG_OUTLIER_K, idx, sub=tag).reshape(num_heads, head_dim)
    return np.sort(np.argsort(w, axis=1, kind="stable")[:, :k], axis=1)


def channel_multiplier(seed: int, tag: int, num_heads: int, head_dim: int, k: int,
                       factor: float) -> np.ndarray:
    """float32 [num_heads, head_dim]: `factor` on the outlier channels, 1 elsewhere."""
    m = np.ones((num_heads, head_dim), dtype=np.float32)
    ch = outlier_channels(seed, tag, num_heads, head_dim, k)
    for h in range(num_heads):
        m[h, ch[h]] = np.float32(factor)
    return m


def permutation(seed: int, tag: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n) (argsort of hashed keys), int32."""
    w = words_np(seed, tag, np.arange(n, dtype=np.int64))
    return np.argsort(w, kind="stable").astype(np.int32)


def uniform_ints(seed: int, tag: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers in [lo, hi] (inclusive), int64."""
    w = words_np(seed, tag, np.arange(n, dtype=np.int64)).astype(np.int64)
    return lo + (w % (hi - lo + 1))


# ---------------------------------------------------------------- K/V tensors in [tokens, H, D]
@dataclass(frozen=True)
class KVSpec:
    """One (layer, K-or-V) tensor of a batch of equal-length sequences, layout [seq*tok, H, D].

    Element (s, t, h, d) has flat index ((s*n_tok + t)*H + h)*D + d.  Keys carry `n_outlier`
    channels per head scaled by `outlier_factor`; keys have an all-zero row at (token 0, head 0)
    and values at (last token, head H-1) of every sequence when `zero_rows` is set.
    """
    seed: int
    layer: int
    is_key: bool
    n_seq: int
    n_tok: int
    num_heads: int
    head_dim: int
    n_outlier: int = 4
    outlier_factor: float = 10.0
    zero_rows: bool = True

    @property
    def tag(self) -> int:
        return TAG_K if self.is_key else TAG_V

    @property
    def n_rows(self) -> int:
        return self.n_seq * self.n_tok * self.num_heads

    def multiplier(self) -> np.ndarray:
        k = self.n_outlier if self.is_key else 0
        return channel_multiplier(self.seed, self.layer, self.num_heads, self.head_dim, k,
                                  self.outlier_factor)

    def zero_row_ids(self) -> np.ndarray:
        """Row ids (in units of [seq*tok*H]) that are forced to zero."""
        if not self.zero_rows:
            return np.zeros(0, dtype=np.int64)
        s = np.arange(self.n_seq, dtype=np.int64)
        if self.is_key:
            t, h = 0, 0
        else:
            t, h = self.n_tok - 1, self.num_heads - 1
        return (s * self.n_tok + t) * self.num_heads + h

    def rows_np(self, row_ids: np.ndarray) -> np.ndarray:
        """fp16 [len(row_ids), D] for the given row ids (row = (s*n_tok + t)*H + h)."""
        row_ids = np.asarray(row_ids, dtype=np.int64)
        D = self.head_dim
        idx = row_ids[:, None] * D + np.arange(D, dtype=np.int64)[None, :]
        mult = self.multiplier()[(row_ids % self.num_heads)]
        out = normal_fp16_np(self.seed, self.tag, idx, sub=self.layer, mult=mult)
        out[np.isin(row_ids, self.zero_row_ids())] = 0
        return out

    def full_np(self) -> np.ndarray:
        return self.rows_np(np.arange(self.n_rows, dtype=np.int64)).reshape(
            self.n_seq * self.n_tok, self.num_heads, self.head_dim)

    def full_torch(self, device, out=None, chunk_rows: int = 1 << 16):
        """Materialise on `device` (chunked, bounded temporaries)."""
        import torch
        D, H = self.head_dim, self.num_heads
        if out is None:
            out = torch.empty((self.n_seq * self.n_tok, H, D), dtype=torch.float16, device=device)
        flat = out.view(-1, D)
        mult = torch.from_numpy(self.multiplier()).to(device)
        d = torch.arange(D, dtype=torch.int64, device=device)
        for r0 in range(0, self.n_rows, chunk_rows):
            r1 = min(self.n_rows, r0 + chunk_rows)
            rows = torch.arange(r0, r1, dtype=torch.int64, device=device)
            idx = rows[:, None] * D + d[None, :]
            m = mult[rows % H]
            flat[r0:r1] = normal_fp16_torch(self.seed, self.tag, idx, sub=self.layer, mult=m)
        z = self.zero_row_ids()
        if z.size:
            flat[torch.from_numpy(z).to(device)] = 0
        return out


# ---------------------------------------------------------------- KIVI tensors [B, H, S, D]
@dataclass(frozen=True)
class KiviSpec:
    """One layer's K or V tensor for the KIVI cache, layout [B, H, S, D], flat index in that order.

    Keys carry `n_outlier` channels per head scaled by `outlier_factor`.
    """
    seed: int
    layer: int
    is_key: bool
    batch: int
    num_heads: int
    seq: int
    head_dim: int
    n_outlier: int = 2
    outlier_factor: float = 8.0

    @property
    def tag(self) -> int:
        return TAG_KIVI_K if self.is_key else TAG_KIVI_V

    def multiplier(self) -> np.ndarray:
        k = self.n_outlier if self.is_key else 0
        return channel_multiplier(self.seed, 1000 + self.layer, self.num_heads, self.head_dim, k,
                                  self.outlier_factor)

    def slab_np(self, b: int, h: int, t0: int, t1: int) -> np.ndarray:
        """fp16 [t1-t0, D] rows of (b, h) for tokens [t0, t1)."""
        D = self.head_dim
        base = ((b * self.num_heads + h) * self.seq)
        idx = (base + np.arange(t0, t1, dtype=np.int64))[:, None] * D + np.arange(D)[None, :]
        mult = np.broadcast_to(self.multiplier()[h][None, :], idx.shape)
        return normal_fp16_np(self.seed, self.tag, idx, sub=self.layer, mult=mult)

    def full_np(self) -> np.ndarray:
        out = np.empty((self.batch, self.num_heads, self.seq, self.head_dim), dtype=np.float16)
        for b in range(self.batch):
            for h in range(self.num_heads):
                out[b, h] = self.slab_np(b, h, 0, self.seq)
        return out

    def full_torch(self, device, out=None, chunk_rows: int = 1 << 16):
        import torch
        B, H, S, D = self.batch, self.num_heads, self.seq, self.head_dim
        if out is None:
            out = torch.empty((B, H, S, D), dtype=torch.float16, device=device)
        flat = out.view(-1, D)
        mult = torch.from_numpy(self.multiplier()).to(device)
        d = torch.arange(D, dtype=torch.int64, device=device)
        n_rows = B * H * S
        for r0 in range(0, n_rows, chunk_rows):
            r1 = min(n_rows, r0 + chunk_rows)
            rows = torch.arange(r0, r1, dtype=torch.int64, device=device)
            idx = rows[:, None] * D + d[None, :]
            m = mult[(rows // S) % H]
            flat[r0:r1] = normal_fp16_torch(self.seed, self.tag, idx, sub=self.layer, mult=m)
        return out


# ---------------------------------------------------------------- queries [n_layers, nseq, Hq, D]
def queries_np(seed: int, n_layers: int, nseq: int, hq: int, d: int) -> np.ndarray:
    idx = np.arange(n_layers * nseq * hq * d, dtype=np.int64)
    return normal_fp16_np(seed, TAG_Q, idx).reshape(n_layers, nseq, hq, d)


def queries_torch(seed: int, n_layers: int, nseq: int, hq: int, d: int, device):
    import torch
    idx = torch.arange(n_layers * nseq * hq * d, dtype=torch.int64, device=device)
    return normal_fp16_torch(seed, TAG_Q, idx).reshape(n_layers, nseq, hq, d)


# ---------------------------------------------------------------- page tables
def random_page_table(seed: int, nseq: int, pages_per_seq: int) -> np.ndarray:
    """int32 [nseq, pages_per_seq]: a seeded permutation of range(nseq*pages_per_seq), dealt out in
    order to the sequences."""
    perm = permutation(seed, TAG_PAGES, nseq * pages_per_seq)
    return perm.reshape(nseq, pages_per_seq)


def decode_append_lengths(seed: int, nseq: int, lo: int = 1024, hi: int = 65536) -> np.ndarray:
    """Existing cache lengths for the decode-append workload, uniform in [lo, hi]."""
    return uniform_ints(seed, TAG_SEQLEN, nseq, lo, hi).astype(np.int32)


# ---------------------------------------------------------------- random packed cache contents
def fill_random_pool_(codes, scales, seed: int) -> None:
    """Fill a packed pool in place with seeded random bytes: codes uniform over all byte values
    (every byte string is a valid packed row at every width) and fp16 scales log-uniform in
    [2^-10, 2^-4] (the scales of N(0, 1) rows with a few outliers).  Used where a cache is too
    large to produce by quantizing generated fp16 rows; the attention does the same work on any
    contents."""
    import torch
    g = torch.Generator(device=codes.device)
    g.manual_seed(seed)
    codes.copy_(torch.randint(0, 256, codes.shape, dtype=torch.uint8, device=codes.device,
                              generator=g))
    e = torch.rand(scales.shape, device=scales.device, generator=g, dtype=torch.float32)
    scales.copy_(torch.exp2(-10.0 + 6.0 * e).to(torch.float16))


# ---------------------------------------------------------------- the workloads
WORKLOADS = {
    # one layer, contiguous: K and V each [1 seq, 4 heads, 1024 tokens, D=256]
    "q6_roundtrip_1x1024x4x256": dict(seed=0, n_layers=1, n_seq=1, n_tok=1024, H=4, D=256,
                                      bits=6),
    # paged prefill: 16 layers x {K,V} x 8 seqs x 32768 tokens x 4 heads x 256, page 16
    "paged_prefill_16L_8x32768_4x256": dict(seed=0, n_layers=16, n_seq=8, n_tok=32768, H=4,
                                            D=256, page_size=16),
    # decode-step append: 64 seqs, lengths U[1024, 65536], append 1/8/32 tokens, 16 layers
    "decode_append_16L_64seq_4x256": dict(seed=2, n_layers=16, n_seq=64, H=4, D=256,
                                          page_size=16, appends=(1, 8, 32)),
    # KIVI flush: 16 layers x [16, 8, 4096, 64], gs 32, levels 3, residual 128
    "kivi_flush_16L_16x8x4096x64": dict(seed=3, n_layers=16, B=16, H=8, S=4096, D=64,
                                        group_size=32, levels=3, eps=1e-8, residual=128,
                                        flushes=((3936, 3968), (3840, 3968))),
    # decode attention over a 262,144-token paged cache, 16 layers, GQA 6:1
    "decode_attn_262144_16L_4x256_gqa6": dict(seed=0, n_layers=16, n_seq=1, n_tok=262144, H=4,
                                              D=256, Hq=24, page_size=16,
                                              softmax_scale=1.0 / 16.0),
}
