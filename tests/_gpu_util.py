"""Helpers shared by the GPU parity tests (not a test module)."""
from __future__ import annotations

import numpy as np
import torch

import kvgen
from oracle import symmetric as osym


def dev_tensor(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def i32(a, device) -> torch.Tensor:
    return torch.as_tensor(np.asarray(a, dtype=np.int32)).to(device)


def cu_of(lens) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.int32)


def u16(t) -> np.ndarray:
    a = t.cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
    return a.view(np.uint16)


def check_rows_against_oracle(pool, x_rows: np.ndarray, page_table: np.ndarray, seq: np.ndarray,
                              pos: np.ndarray, head: np.ndarray, bits: int) -> None:
    """Bit-exact: the GPU pool's bytes and scale for each sampled row equal the oracle's."""
    packed, scale = osym.quant_pack_rows(x_rows, bits)
    page = page_table[seq, pos // pool.page_size].astype(np.int64)
    slot = pos % pool.page_size
    idx = torch.from_numpy(np.stack([page, head, slot]).astype(np.int64))
    codes = pool.codes[idx[0].to(pool.codes.device), idx[1].to(pool.codes.device),
                       idx[2].to(pool.codes.device)].cpu().numpy()
    scales = pool.scales[idx[0].to(pool.codes.device), idx[1].to(pool.codes.device),
                         idx[2].to(pool.codes.device)].cpu().numpy()
    bad = np.nonzero(np.any(codes != packed, axis=1))[0]
    assert bad.size == 0, f"{bad.size} rows differ in codes, first row {bad[:4]}"
    assert np.array_equal(scales.view(np.uint16), scale.view(np.uint16)), "scales differ"


def random_rows(n: int, D: int, seed: int) -> np.ndarray:
    """Rows spanning many magnitudes (subnormal-scale rows included), outliers, zeros, ties."""
    rng = np.random.default_rng(seed)
    base = kvgen.normal_fp16_np(seed, 98, np.arange(n * D)).reshape(n, D).astype(np.float32)
    mag = np.float32(2.0) ** rng.integers(-26, 12, size=(n, 1)).astype(np.float32)
    x = base * mag
    x[rng.random((n, D)) < 0.01] *= 10
    x[::53] = 0
    # rows of exact half-integers on scale-1 grids (ties), one per width
    for r, q in ((1, 127), (2, 31), (3, 7)):
        if r < n:
            k = rng.integers(-2 * q, 2 * q + 1, size=D) / 2.0
            k[0] = q
            x[r] = k
    return np.clip(x, -65504, 65504).astype(np.float16)
