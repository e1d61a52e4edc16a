"""Packed KIVI storage and decode attention over it (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache".  The page keeps its cache in
fp16 and only estimates what a packed form would cost (module docstring, "Memory-savings caveat";
``_quantized_bytes`` / ``_account_bytes``): b-bit codes plus an fp16 (scale, zero) pair per group
-- per (token group, channel) for keys, per (token, channel group) for values.  This module is
that packed form, with the groups, axes, levels and eps of ``_quant_dequant_along``.

Readings where the pages leave a step open:
* zero = gmin, which is an fp16 value already (the minimum of fp16 inputs), so it is stored
  exactly; scale16 = fp16_rne(max(float32(gmax - gmin) / levels, float32(eps)));
* codes are computed against the stored fp16 scale (as the symmetric quantizer computes its codes
  against its stored scale): c = clip(rint_half_even(float32(x - gmin) / float32(scale16)), 0,
  levels); a group whose fp16 scale is 0 (range below fp16 resolution) stores codes 0;
* reconstruction keeps the page's two roundings: x_hat = fp16(float32(c * scale16) + gmin);
* codes are an LSB-first bit stream along the head dimension of each token row (element d at
  bits [b*d, b*d + b)), the same convention as the q4/q6 pages; b in {2, 4, 8};
* key groups start at token 0 of the cache (flushes are group-aligned); the value groups of a
  row start at channel 0 and the last one may be ragged;
* attention over the packed cache attends to the packed tokens [0, n_q) and to the fp16
  residual tokens [n_q, offset) of the same sequence, softmax(q . k_hat * scale) . v_hat, float64.
"""
from __future__ import annotations

import math

import numpy as np

from . import attention


def levels_of(bits: int) -> int:
    if bits not in (2, 4, 8):
        raise ValueError("packed KIVI supports 2, 4 or 8 bits")
    return (1 << bits) - 1


def _params(gmin32: np.ndarray, gmax32: np.ndarray, levels: int, eps: float):
    scale32 = np.maximum((gmax32 - gmin32) / np.float32(levels), np.float32(eps))
    return scale32.astype(np.float16), gmin32.astype(np.float16)


def _codes(x32: np.ndarray, zero32: np.ndarray, scale16: np.ndarray, levels: int) -> np.ndarray:
    s32 = scale16.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        q = (x32 - zero32) / s32
    c = np.clip(np.rint(q), 0, levels)
    c = np.where(s32 == 0, 0, c)
    return c.astype(np.int64)


def pack_bits(codes: np.ndarray, bits: int) -> np.ndarray:
    """int codes [..., D] -> uint8 [..., D*bits/8], LSB-first along the last axis."""
    D = codes.shape[-1]
    if (D * bits) % 8:
        raise ValueError("row of codes must fill whole bytes")
    per = 8 // bits
    c = codes.reshape(codes.shape[:-1] + (D // per, per))
    out = np.zeros(c.shape[:-1], dtype=np.int64)
    for k in range(per):
        out |= c[..., k] << (bits * k)
    return out.astype(np.uint8)


def unpack_bits(packed: np.ndarray, bits: int, D: int) -> np.ndarray:
    per = 8 // bits
    b = packed.astype(np.int64)
    parts = [(b >> (bits * k)) & ((1 << bits) - 1) for k in range(per)]
    return np.stack(parts, axis=-1).reshape(packed.shape[:-1] + (D,))


def pack_keys(x16: np.ndarray, bits: int, group_size: int, eps: float = 1e-8):
    """Keys [B, H, n, D] (n a multiple of group_size) -> (codes [B, H, n, D*b/8],
    scale16 [B, H, n/gs, D], zero16 [B, H, n/gs, D]); groups of gs tokens per channel."""
    L = levels_of(bits)
    B, H, n, D = x16.shape
    if n % group_size:
        raise ValueError("keys are packed in whole token groups")
    x32 = x16.astype(np.float32)
    xg = x32.reshape(B, H, n // group_size, group_size, D)
    scale16, zero16 = _params(xg.min(axis=3), xg.max(axis=3), L, eps)
    c = _codes(xg, zero16.astype(np.float32)[:, :, :, None, :], scale16[:, :, :, None, :], L)
    return pack_bits(c.reshape(B, H, n, D), bits), scale16, zero16


def pack_values(x16: np.ndarray, bits: int, group_size: int, eps: float = 1e-8):
    """Values [B, H, n, D] -> (codes [B, H, n, D*b/8], scale16 [B, H, n, G], zero16 [B, H, n, G]),
    G = ceil(D / gs) channel groups per token (the last one may be ragged)."""
    L = levels_of(bits)
    B, H, n, D = x16.shape
    G = (D + group_size - 1) // group_size
    x32 = x16.astype(np.float32)
    scale16 = np.zeros((B, H, n, G), np.float16)
    zero16 = np.zeros((B, H, n, G), np.float16)
    c = np.zeros((B, H, n, D), np.int64)
    for g in range(G):
        sl = slice(g * group_size, min(D, (g + 1) * group_size))
        s16, z16 = _params(x32[..., sl].min(axis=-1), x32[..., sl].max(axis=-1), L, eps)
        scale16[..., g], zero16[..., g] = s16, z16
        c[..., sl] = _codes(x32[..., sl], z16.astype(np.float32)[..., None], s16[..., None], L)
    return pack_bits(c, bits), scale16, zero16


def _recon(c: np.ndarray, scale16: np.ndarray, zero16: np.ndarray) -> np.ndarray:
    prod = c.astype(np.float32) * scale16.astype(np.float32)      # one rounding
    return (prod + zero16.astype(np.float32)).astype(np.float16)  # a second, then fp16


def unpack_keys(codes, scale16, zero16, bits: int, group_size: int, D: int) -> np.ndarray:
    c = unpack_bits(codes, bits, D)
    s = np.repeat(scale16, group_size, axis=2)[:, :, :c.shape[2]]
    z = np.repeat(zero16, group_size, axis=2)[:, :, :c.shape[2]]
    return _recon(c, s, z)


def unpack_values(codes, scale16, zero16, bits: int, group_size: int, D: int) -> np.ndarray:
    c = unpack_bits(codes, bits, D)
    gidx = np.arange(D) // group_size
    return _recon(c, scale16[..., gidx], zero16[..., gidx])


def packed_bytes(n: int, batch: int, num_heads: int, head_dim: int, bits: int,
                 group_size: int) -> tuple[int, int]:
    """Bytes this layout stores for n quantized tokens: (keys, values)."""
    B, H, D, gs = batch, num_heads, head_dim, group_size
    code = n * D * bits // 8 * H * B
    k = code + (n // gs) * D * 2 * 2 * H * B
    v = code + n * math.ceil(D / gs) * 2 * 2 * H * B
    return k, v


def decode_attention(q16: np.ndarray, k_packed, v_packed, k_res16: np.ndarray,
                     v_res16: np.ndarray, bits: int, group_size: int, softmax_scale: float
                     ) -> np.ndarray:
    """q16 [B, Hq, D]; k_packed = (codes, scale16, zero16) for tokens [0, n_q) of every batch
    row (same n_q); k_res16, v_res16 [B, H, n_res, D] the fp16 residual tokens.  -> float64
    [B, Hq, D]."""
    B, Hq, D = q16.shape
    kh = unpack_keys(*k_packed, bits, group_size, D)
    vh = unpack_values(*v_packed, bits, group_size, D)
    k_all = np.concatenate([kh, k_res16], axis=2)
    v_all = np.concatenate([vh, v_res16], axis=2)
    out = np.zeros((B, Hq, D), np.float64)
    for b in range(B):
        out[b] = attention.attend(q16[b], np.transpose(k_all[b], (1, 0, 2)),
                                  np.transpose(v_all[b], (1, 0, 2)), softmax_scale)
    return out


class KiviPackedCache:
    """The KIVI cache protocol of the page (``update_and_fetch``, ``trim`` with
    ``_rollback_frontier``) with the quantized region held in the packed form above.

    Tokens [0, n_quantized) are packed; tokens [n_quantized, offset) are the fp16 residual
    window.  A flush packs [n_quantized, boundary) from the fp16 rows (``update_and_fetch``).
    A trim pulls the frontier down to a group multiple; the rows between the new frontier and the
    new offset leave the packed region carrying their round-tripped values into the fp16 window
    (on the page they were round-tripped in place), so the next flush quantizes them a second time
    -- the double rounding the page bounds by one quantization step.
    """

    def __init__(self, batch: int, num_heads: int, head_dim: int, capacity: int,
                 bit_width: int = 2, group_size: int = 32, residual_length: int = 128,
                 eps: float = 1e-8):
        from . import kivi
        self._kivi = kivi
        B, H, D, S, gs = batch, num_heads, head_dim, capacity, group_size
        if S % gs:
            raise ValueError("capacity must be a multiple of group_size")
        self.bits, self.gs, self.residual_length, self.eps = bit_width, gs, residual_length, eps
        self.keys = np.zeros((B, H, S, D), np.float16)
        self.values = np.zeros((B, H, S, D), np.float16)
        cb = D * bit_width // 8
        G = -(-D // gs)
        self.k_codes = np.zeros((B, H, S, cb), np.uint8)
        self.k_scale = np.zeros((B, H, S // gs, D), np.float16)
        self.k_zero = np.zeros((B, H, S // gs, D), np.float16)
        self.v_codes = np.zeros((B, H, S, cb), np.uint8)
        self.v_scale = np.zeros((B, H, S, G), np.float16)
        self.v_zero = np.zeros((B, H, S, G), np.float16)
        self.offset = 0
        self.n_quantized = 0

    def update(self, keys: np.ndarray, values: np.ndarray) -> None:
        n = keys.shape[2]
        self.keys[:, :, self.offset:self.offset + n] = keys
        self.values[:, :, self.offset:self.offset + n] = values
        self.offset += n
        hi = self._kivi.quantization_boundary(self.offset, self.residual_length, self.gs)
        lo = self.n_quantized
        if hi > lo:
            gs = self.gs
            c, s, z = pack_keys(self.keys[:, :, lo:hi], self.bits, gs, self.eps)
            self.k_codes[:, :, lo:hi], self.k_scale[:, :, lo // gs:hi // gs] = c, s
            self.k_zero[:, :, lo // gs:hi // gs] = z
            c, s, z = pack_values(self.values[:, :, lo:hi], self.bits, gs, self.eps)
            self.v_codes[:, :, lo:hi], self.v_scale[:, :, lo:hi], self.v_zero[:, :, lo:hi] = c, s, z
            self.n_quantized = hi

    def _unpacked(self, lo: int, hi: int):
        D, gs = self.keys.shape[3], self.gs
        g0 = lo // gs
        g1 = -(-hi // gs)
        k = unpack_keys(self.k_codes[:, :, g0 * gs:g1 * gs], self.k_scale[:, :, g0:g1],
                        self.k_zero[:, :, g0:g1], self.bits, gs, D)[:, :, lo - g0 * gs:hi - g0 * gs]
        v = unpack_values(self.v_codes[:, :, lo:hi], self.v_scale[:, :, lo:hi],
                          self.v_zero[:, :, lo:hi], self.bits, gs, D)
        return k, v

    def trim(self, n: int) -> int:
        trimmed = min(self.offset, n)
        self.offset -= trimmed
        if trimmed:
            gs = self.gs
            new_nq = min(self.n_quantized, (max(self.offset, 0) // gs) * gs)
            hi = min(self.n_quantized, self.offset)
            if hi > new_nq:   # rows leaving the packed region keep their round-tripped values
                k, v = self._unpacked(new_nq, hi)
                self.keys[:, :, new_nq:hi], self.values[:, :, new_nq:hi] = k, v
            self.n_quantized = new_nq
        return trimmed

    def fetch(self):
        """The cache as attention sees it: unpacked [0, n_quantized) then the fp16 window."""
        nq, off = self.n_quantized, self.offset
        k, v = self._unpacked(0, nq)
        return (np.concatenate([k, self.keys[:, :, nq:off]], axis=2),
                np.concatenate([v, self.values[:, :, nq:off]], axis=2))
