"""KIVI asymmetric group quantize->dequantize, residual boundary, flush and trim (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache", class ``KIVIKVCache``:
``_quant_dequant_along`` (the round trip), ``_quantization_boundary`` (Algorithm 1 boundary),
``update_and_fetch`` (the in-place flush), ``_rollback_frontier`` / ``trim``.  The module
docstring fixes the axes: keys per channel (groups run along tokens), values per token (groups
run along channels); the config defaults are group size 32, residual 128, b = 2, and the class
sets levels = 2^b - 1 and eps = 1e-8.

The round trip follows the page's steps in their order, in float32:
cast to float32; split the chosen axis into groups of ``group_size`` (a ragged tail is padded by
repeating its last element); per group gmin, gmax; scale = max((gmax - gmin) / levels, eps);
codes = clip(round((x - gmin) / scale), 0, levels); recon = codes * scale + gmin; drop the pad;
cast back to the input dtype.

Readings where the page is silent:
* ``round`` is round-half-to-even (numpy/MLX ``round`` semantics);
* ``codes * scale + gmin`` is two float32 operations with two roundings (no fused multiply-add);
* ``eps`` is float32(1e-8) and ``levels`` is used as a float32 divisor;
* the final cast to fp16 rounds to nearest even;
* inputs are finite.
"""
from __future__ import annotations

import math

import numpy as np


def quant_dequant_along(x: np.ndarray, axis: int, group_size: int, levels: int,
                        eps: float = 1e-8) -> np.ndarray:
    """Round-trip `x` through KIVI group quantization along `axis` (groups start at index 0)."""
    gs = int(group_size)
    x32 = np.asarray(x).astype(np.float32)
    L = x32.shape[axis]
    n_groups = (L + gs - 1) // gs
    pad = n_groups * gs - L
    xm = np.moveaxis(x32, axis, -1)
    if pad:
        tail = np.repeat(xm[..., -1:], pad, axis=-1)
        xm = np.concatenate([xm, tail], axis=-1)
    xg = xm.reshape(xm.shape[:-1] + (n_groups, gs))
    gmin = xg.min(axis=-1, keepdims=True)
    gmax = xg.max(axis=-1, keepdims=True)
    scale = np.maximum((gmax - gmin) / np.float32(levels), np.float32(eps))
    codes = np.clip(np.rint((xg - gmin) / scale), 0, levels)
    recon = codes * scale          # one rounding
    recon = recon + gmin           # a second rounding
    recon = recon.reshape(xm.shape)[..., :L]
    recon = np.moveaxis(recon, -1, axis)
    return recon.astype(np.asarray(x).dtype)


def quantization_boundary(offset: int, residual_length: int, group_size: int) -> int:
    """Absolute position below which tokens may be quantized now: the aged-out count, snapped down
    to a multiple of the group size."""
    aged = max(0, offset - residual_length)
    return (aged // group_size) * group_size


def flush(keys: np.ndarray, values: np.ndarray, lo: int, hi: int, group_size: int, levels: int,
          eps: float = 1e-8) -> None:
    """In-place round trip of tokens [lo, hi) of [B, H, S, D] keys (per channel) and values
    (per token), as ``update_and_fetch`` does for the newly aged slice."""
    if hi <= lo:
        return
    keys[:, :, lo:hi, :] = quant_dequant_along(keys[:, :, lo:hi, :], -2, group_size, levels, eps)
    values[:, :, lo:hi, :] = quant_dequant_along(values[:, :, lo:hi, :], -1, group_size, levels,
                                                 eps)


class KiviCache:
    """fp16 KV cache with KIVI's residual window (the ``update_and_fetch`` / ``trim`` protocol)."""

    def __init__(self, batch: int, num_heads: int, head_dim: int, capacity: int,
                 bit_width: int = 2, group_size: int = 32, residual_length: int = 128):
        if not isinstance(bit_width, int):
            raise TypeError("bit_width must be a single int")
        self.levels = (1 << bit_width) - 1
        self.eps = 1e-8
        self.group_size = group_size
        self.residual_length = residual_length
        self.keys = np.zeros((batch, num_heads, capacity, head_dim), dtype=np.float16)
        self.values = np.zeros_like(self.keys)
        self.offset = 0
        self.n_quantized = 0

    def update_and_fetch(self, keys: np.ndarray, values: np.ndarray):
        S = keys.shape[2]
        self.keys[:, :, self.offset:self.offset + S] = keys
        self.values[:, :, self.offset:self.offset + S] = values
        self.offset += S
        boundary = quantization_boundary(self.offset, self.residual_length, self.group_size)
        if boundary > self.n_quantized:
            flush(self.keys, self.values, self.n_quantized, boundary, self.group_size,
                  self.levels, self.eps)
            self.n_quantized = boundary
        return self.keys[:, :, :self.offset], self.values[:, :, :self.offset]

    def trim(self, n: int) -> int:
        trimmed = min(self.offset, n)
        self.offset -= trimmed
        if trimmed:
            gs = self.group_size
            self.n_quantized = min(self.n_quantized, (max(self.offset, 0) // gs) * gs)
        return trimmed


def quantized_bytes(n: int, batch: int, num_heads: int, head_dim: int, bit_width: int,
                    group_size: int) -> tuple[int, int]:
    """(key, value) packed-byte cost of n group-aligned quantized tokens: codes at b bits plus an
    fp16 (scale, zero) pair per group -- per channel per token-group for keys, per token per
    channel-group for values (``_quantized_bytes``)."""
    B, H, D, gs = batch, num_heads, head_dim, group_size
    code = math.ceil(n * D * bit_width / 8) * H * B
    k = code + math.ceil(n / gs) * D * 2 * 2 * H * B
    v = code + n * math.ceil(D / gs) * 2 * 2 * H * B
    return k, v
