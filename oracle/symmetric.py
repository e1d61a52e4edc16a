"""Symmetric per-token-per-head KV quantizer, q8/q6/q4 storage and paged scatter/gather (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization", description.

What the page fixes:
* one fp16 scale per row, a row being one (token, KV head) vector of D elements;
* clip bound qmax = 127 / 31 / 7 for 8 / 6 / 4 bits, an explicit table that raises on unknown
  widths (bit-width table paragraph);
* q6 codes biased by +32 into a 6-bit field and packed four per three bytes, little-endian:
  byte0 = u0 | (u1 & 0x03) << 6, byte1 = (u1 >> 2) | (u2 & 0x0F) << 4,
  byte2 = (u2 >> 4) | (u3 & 0x3F) << 2 (byte-layout formula);
* packed_dim(D, 6) = 3D/4 and q6 needs D % 4 == 0 (packed_dim sentence); q6 shares q4's uint8
  sub-byte storage branch.

Readings where the page is silent:
* scale = fp16_rne(float32(amax) / float32(qmax)), an IEEE float32 quotient rounded to fp16;
  codes are computed against that stored fp16 scale:
  c = clamp(rint_half_even(float32(x) / float32(scale)), -qmax, qmax);
* a row whose fp16 scale is 0 (all-zero row, or amax so small that amax/qmax underflows fp16)
  stores scale +0 and every code equal to 0 (stored field = the bias); it dequantizes to 0;
* q4: bias +8, element 2i in the low nibble of byte i (the same LSB-first bit stream as q6);
* q8: the signed code as an int8 two's-complement byte (bias 0);
* dequantization: x_hat = fp16_rne(float32(c) * float32(scale)) (the product is exact in fp32);
* inputs are finite fp16 (NaN/Inf are out of contract).
"""
from __future__ import annotations

import numpy as np

QMAX = {8: 127, 6: 31, 4: 7}
BIAS = {8: 0, 6: 32, 4: 8}


def qmax_for(bits: int) -> int:
    """Clip bound for a bit width; unknown widths raise (explicit table, no fall-through)."""
    if bits not in QMAX:
        raise ValueError(f"unsupported KV quantization width: {bits!r}")
    return QMAX[bits]


def packed_dim(head_dim: int, bits: int) -> int:
    """Bytes per packed row."""
    qmax_for(bits)
    if bits == 8:
        return head_dim
    if bits == 6:
        if head_dim % 4:
            raise ValueError("q6 needs head_dim % 4 == 0")
        return head_dim * 3 // 4
    if head_dim % 2:
        raise ValueError("q4 needs head_dim % 2 == 0")
    return head_dim // 2


# ---------------------------------------------------------------- quantize / dequantize
def quantize_rows(x16: np.ndarray, bits: int) -> tuple[np.ndarray, np.ndarray]:
    """Rows of fp16 [..., D] -> (fp16 scale [...], int32 codes [..., D] in [-qmax, qmax])."""
    qmax = qmax_for(bits)
    x16 = np.asarray(x16, dtype=np.float16)
    x32 = x16.astype(np.float32)
    if not np.all(np.isfinite(x32)):
        raise ValueError("non-finite input is out of contract")
    amax = np.max(np.abs(x32), axis=-1)                       # float32 max: exact
    scale16 = (amax / np.float32(qmax)).astype(np.float16)    # IEEE f32 divide, then RNE to fp16
    s32 = scale16.astype(np.float32)
    zero = s32 == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        q = x32 / s32[..., None]                              # IEEE f32 divide
    codes = np.clip(np.rint(q), -qmax, qmax)                  # rint: round half to even
    codes[zero] = 0
    return scale16, codes.astype(np.int32)


def dequantize_rows(codes: np.ndarray, scale16: np.ndarray) -> np.ndarray:
    """int codes [..., D] and fp16 scale [...] -> fp16 [..., D]."""
    prod = codes.astype(np.float32) * np.asarray(scale16, np.float16).astype(np.float32)[..., None]
    return prod.astype(np.float16)


# ---------------------------------------------------------------- pack / unpack
def encode(codes: np.ndarray, bits: int) -> np.ndarray:
    """Signed codes -> stored unsigned fields: +bias for q6/q4, int8 two's-complement byte for q8."""
    qmax = qmax_for(bits)
    codes = np.asarray(codes, dtype=np.int64)
    if codes.size and (codes.min() < -qmax or codes.max() > qmax):
        raise ValueError("code out of range")
    if bits == 8:
        return codes & 0xFF
    return codes + BIAS[bits]


def decode(fields: np.ndarray, bits: int) -> np.ndarray:
    """Stored unsigned fields -> signed codes (inverse of `encode`, defined on every field value)."""
    f = np.asarray(fields, dtype=np.int64)
    if bits == 8:
        return np.where(f >= 128, f - 256, f).astype(np.int32)
    return (f - BIAS[bits]).astype(np.int32)


def pack_fields(u: np.ndarray, bits: int) -> np.ndarray:
    """Unsigned fields [..., D] (each < 2^bits) -> uint8 [..., packed_dim(D, bits)]."""
    u = np.asarray(u, dtype=np.int64)
    D = u.shape[-1]
    pd = packed_dim(D, bits)
    if u.size and (u.min() < 0 or u.max() >= (1 << bits)):
        raise ValueError("field out of range")
    if bits == 8:
        return u.astype(np.uint8)
    if bits == 4:
        lo, hi = u[..., 0::2], u[..., 1::2]
        return (lo | (hi << 4)).astype(np.uint8)
    # q6: groups of four 6-bit fields -> three bytes, per the page's formula
    q = u.reshape(u.shape[:-1] + (D // 4, 4))
    u0, u1, u2, u3 = q[..., 0], q[..., 1], q[..., 2], q[..., 3]
    b0 = u0 | ((u1 & 0x03) << 6)
    b1 = (u1 >> 2) | ((u2 & 0x0F) << 4)
    b2 = (u2 >> 4) | ((u3 & 0x3F) << 2)
    out = np.stack([b0, b1, b2], axis=-1).reshape(u.shape[:-1] + (pd,))
    return (out & 0xFF).astype(np.uint8)


def unpack_fields(packed: np.ndarray, bits: int, head_dim: int) -> np.ndarray:
    """uint8 [..., packed_dim] -> unsigned fields [..., D] (inverse of `pack_fields`)."""
    qmax_for(bits)
    b = np.asarray(packed, dtype=np.uint8).astype(np.int64)
    if b.shape[-1] != packed_dim(head_dim, bits):
        raise ValueError("packed row has the wrong width")
    if bits == 8:
        return b
    if bits == 4:
        lo, hi = b & 0x0F, b >> 4
        return np.stack([lo, hi], axis=-1).reshape(b.shape[:-1] + (head_dim,))
    t = b.reshape(b.shape[:-1] + (head_dim // 4, 3))
    b0, b1, b2 = t[..., 0], t[..., 1], t[..., 2]
    u0 = b0 & 0x3F
    u1 = (b0 >> 6) | ((b1 & 0x0F) << 2)
    u2 = (b1 >> 4) | ((b2 & 0x03) << 4)
    u3 = b2 >> 2
    return np.stack([u0, u1, u2, u3], axis=-1).reshape(b.shape[:-1] + (head_dim,))


def pack(codes: np.ndarray, bits: int) -> np.ndarray:
    """Signed codes [..., D] -> uint8 [..., packed_dim(D, bits)]."""
    return pack_fields(encode(codes, bits), bits)


def unpack(packed: np.ndarray, bits: int, head_dim: int) -> np.ndarray:
    """uint8 [..., packed_dim] -> signed int32 codes [..., D]; decodes every byte string."""
    return decode(unpack_fields(packed, bits, head_dim), bits)


def quant_pack_rows(x16: np.ndarray, bits: int) -> tuple[np.ndarray, np.ndarray]:
    """fp16 rows -> (packed uint8 rows, fp16 scales)."""
    scale16, codes = quantize_rows(x16, bits)
    return pack(codes, bits), scale16


def dequant_rows(packed: np.ndarray, scale16: np.ndarray, bits: int, head_dim: int) -> np.ndarray:
    return dequantize_rows(unpack(packed, bits, head_dim), scale16)


# ---------------------------------------------------------------- paged storage
class PagedPool:
    """One (layer, K-or-V) page pool.

    codes  uint8  [num_pages, H, page_size, packed_dim]
    scales fp16   [num_pages, H, page_size]
    Token `pos` of sequence `s` lives at page page_table[s, pos // page_size], slot
    pos % page_size (a reading: the page does not fix the page layout).
    """

    def __init__(self, bits: int, num_heads: int, head_dim: int, page_size: int, num_pages: int):
        self.bits, self.H, self.D, self.page_size = bits, num_heads, head_dim, page_size
        self.pd = packed_dim(head_dim, bits)
        self.codes = np.zeros((num_pages, num_heads, page_size, self.pd), dtype=np.uint8)
        self.scales = np.zeros((num_pages, num_heads, page_size), dtype=np.float16)


def locate(page_table: np.ndarray, seq: int, pos, page_size: int):
    """(physical page, slot) of token `pos` of sequence `seq`."""
    pos = np.asarray(pos, dtype=np.int64)
    return page_table[seq, pos // page_size].astype(np.int64), pos % page_size


def quant_pack_paged(pool: PagedPool, x16: np.ndarray, page_table: np.ndarray,
                     cu_new_tokens: np.ndarray, start_pos: np.ndarray) -> None:
    """Quantize new tokens x16 [total, H, D] and write them into `pool` through the page table.

    Sequence s owns rows cu_new_tokens[s]:cu_new_tokens[s+1] of x16, which are its tokens
    start_pos[s], start_pos[s]+1, ...
    """
    for s in range(len(start_pos)):
        a, b = int(cu_new_tokens[s]), int(cu_new_tokens[s + 1])
        if b == a:
            continue
        pos = int(start_pos[s]) + np.arange(b - a)
        page, slot = locate(page_table, s, pos, pool.page_size)
        packed, scale16 = quant_pack_rows(x16[a:b], pool.bits)          # [n, H, pd], [n, H]
        for h in range(pool.H):
            pool.codes[page, h, slot] = packed[:, h]
            pool.scales[page, h, slot] = scale16[:, h]


def dequant_paged(pool: PagedPool, page_table: np.ndarray, cu_tokens: np.ndarray,
                  start_pos: np.ndarray) -> np.ndarray:
    """Gather and dequantize tokens back to fp16 [total, H, D] (same addressing as above)."""
    total = int(cu_tokens[-1])
    out = np.zeros((total, pool.H, pool.D), dtype=np.float16)
    for s in range(len(start_pos)):
        a, b = int(cu_tokens[s]), int(cu_tokens[s + 1])
        if b == a:
            continue
        pos = int(start_pos[s]) + np.arange(b - a)
        page, slot = locate(page_table, s, pos, pool.page_size)
        for h in range(pool.H):
            out[a:b, h] = dequant_rows(pool.codes[page, h, slot], pool.scales[page, h, slot],
                                       pool.bits, pool.D)
    return out
