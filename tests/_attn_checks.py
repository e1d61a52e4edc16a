"""Attention checks shared by the parity tests (not a test module; no GPU needed).

* ``assert_attn_close``: the decode tolerance |got - ref| <= 2e-3 + 1e-3 |ref| elementwise, with a
  report of the max abs error, the max error / rms(ref) and the count outside.
* Needles: key rows planted along one query head's direction so that the softmax of that head is
  dominated by them.  Away from needles the whole-window output of a long cache is an average of
  hundreds of thousands of tokens, small against the absolute tolerance, so one lost or misplaced
  16-token tile can pass unseen; with identical needles the output of the needle head is the mean
  of the needle tokens' values, and dropping or moving any one of them shifts it far outside the
  tolerance.  The positions chosen are the places a tile schedule goes wrong: the first and last
  tile, the tiles on both sides of a split boundary, a tile deep in a warp's stream (after its
  stage ring has wrapped), the middle split and the last token.
* ``decode_tiles_per_cta`` restates the library's split rule for the paged decode attention so a
  test can place needles at split boundaries and assert that each warp's ring wraps; the tests
  cross-check it against the workspace size the library reports.

These helpers build inputs and compare outputs; they hold none of the method's arithmetic.
"""
from __future__ import annotations

import json
import os
from dataclasses import dataclass, field

import numpy as np

ATOL, RTOL = 2e-3, 1e-3
TILE = 16          # tokens per tile of the paged decode attention
WARPS = 4          # warps per CTA
NEEDLE_SCORE = 32.0   # target softmax logit of a needle for its query head


def attn_report(got: np.ndarray, ref: np.ndarray) -> dict:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(got - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    rms = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
    mx = float(err.max()) if err.size else 0.0
    tol_frac = float((err / (ATOL + RTOL * np.abs(ref))).max()) if err.size else 0.0
    return {"n_bad": int(bad.sum()), "max_abs_err": mx,
            "max_err_over_rms_ref": (mx / rms) if rms > 0 else float("inf") if mx > 0 else 0.0,
            "max_err_over_tol": tol_frac,
            "rms_ref": rms, "finite": bool(np.all(np.isfinite(got)))}


def attn_close(got, ref) -> bool:
    r = attn_report(got, ref)
    return r["n_bad"] == 0 and r["finite"]


def _log_margin(r: dict, ctx: str) -> None:
    """With KVQ_ATTN_MARGINS set to a file path, append this check's report to it (one JSON line
    per check, with the running test's id) -- how close each parity check came to the tolerance."""
    path = os.environ.get("KVQ_ATTN_MARGINS")
    if path:
        rec = dict(r, ctx=ctx, test=os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0])
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")


def assert_attn_close(got, ref, ctx: str = "") -> dict:
    r = attn_report(got, ref)
    _log_margin(r, ctx)
    assert r["finite"] and r["n_bad"] == 0, (
        f"{ctx}: {r['n_bad']} outside 2e-3 + 1e-3|ref|; max abs err {r['max_abs_err']:.3e}, "
        f"max err / rms(ref) {r['max_err_over_rms_ref']:.3e} (rms {r['rms_ref']:.3e})")
    return r


def needle_row(q_head: np.ndarray, softmax_scale: float, score: float = NEEDLE_SCORE) -> np.ndarray:
    """fp16 key row c * q with c chosen so that the exact logit q . k * scale is `score`."""
    q = np.asarray(q_head, dtype=np.float64)
    c = score / (softmax_scale * float(q @ q))
    return (c * q).astype(np.float16)


def decode_tiles_per_cta(n_layers: int, nseq: int, num_kv_heads: int, max_seq_len: int,
                         sms: int) -> int:
    """Tiles per CTA of the paged decode attention: about two resident waves of 3 CTAs per SM,
    at most 256 tiles per CTA, a multiple of the 4 warps."""
    tiles = -(-max_seq_len // TILE)
    units = n_layers * nseq * num_kv_heads
    want = -(-6 * sms // units)
    t = min(-(-tiles // want), 256)
    t = -(-t // WARPS) * WARPS
    return max(t, WARPS)


def decode_splits_from_workspace(ws_bytes: int, n_layers: int, nseq: int,
                                 num_kv_heads: int) -> int:
    """Split count implied by the workspace the library asks for (one float32 record of
    8 heads x (256 + 4) per (layer, sequence, KV head, split))."""
    per = n_layers * nseq * num_kv_heads * 8 * (256 + 4) * 4
    assert ws_bytes % per == 0
    return ws_bytes // per


def paged_needle_positions(length: int, tpc: int, stages: int) -> list[int]:
    """Token positions in a sequence of `length` tokens split into CTAs of `tpc` tiles (tiles
    dealt round-robin to 4 warps, each streaming through a ring of `stages` stages)."""
    if length <= 0:
        return []
    per_warp = tpc // WARPS
    deep_j = min(per_warp - 1, stages + 1)           # past one wrap of the ring when possible
    tiles = -(-length // TILE)
    n_splits = -(-tiles // tpc)
    mid = n_splits // 2
    cand = [0,                                        # first tile, warp 0
            TILE * (tpc - 1) + 7,                     # last tile of split 0 (warp 3)
            TILE * tpc + 3,                           # first tile of split 1
            TILE * (2 + WARPS * deep_j) + 11,         # warp 2, deep in its stream
            TILE * (mid * tpc + 1 + WARPS * deep_j) + 5,   # warp 1 of the middle split
            length - 1]                               # last token
    return sorted({p for p in cand if 0 <= p < length})


@dataclass
class Planted:
    """A K/V generator spec (kvgen.KVSpec) with some rows replaced: row id -> fp16 [D]."""
    spec: object
    rows: dict = field(default_factory=dict)

    def rows_np(self, row_ids) -> np.ndarray:
        row_ids = np.asarray(row_ids, dtype=np.int64)
        out = self.spec.rows_np(row_ids)
        for i, r in enumerate(row_ids):
            v = self.rows.get(int(r))
            if v is not None:
                out[i] = v
        return out

    def full_np(self) -> np.ndarray:
        s = self.spec
        flat = self.rows_np(np.arange(s.n_rows, dtype=np.int64))
        return flat.reshape(s.n_seq * s.n_tok, s.num_heads, s.head_dim)

    def full_torch(self, device):
        import torch
        x = self.spec.full_torch(device)
        if self.rows:
            ids = torch.tensor(sorted(self.rows), dtype=torch.int64, device=device)
            vals = np.stack([self.rows[i] for i in sorted(self.rows)])
            x.view(-1, self.spec.head_dim)[ids] = torch.from_numpy(vals).to(device)
        return x


def plant_needles(planted: Planted, seq: int, head: int, positions, key_row: np.ndarray) -> None:
    """Put `key_row` at (sequence seq, token p, KV head `head`) for every p in positions."""
    s = planted.spec
    for p in positions:
        planted.rows[(seq * s.n_tok + int(p)) * s.num_heads + head] = key_row


@dataclass
class PlantedKivi:
    """A KIVI generator spec (kvgen.KiviSpec) with some token rows replaced: (b, h, t) -> fp16."""
    spec: object
    rows: dict = field(default_factory=dict)

    def slab_np(self, b: int, h: int, t0: int, t1: int) -> np.ndarray:
        out = self.spec.slab_np(b, h, t0, t1)
        for (bb, hh, t), v in self.rows.items():
            if bb == b and hh == h and t0 <= t < t1:
                out[t - t0] = v
        return out

    def full_np(self) -> np.ndarray:
        s = self.spec
        out = s.full_np()
        for (b, h, t), v in self.rows.items():
            out[b, h, t] = v
        return out

    def full_torch(self, device):
        import torch
        x = self.spec.full_torch(device)
        for (b, h, t), v in self.rows.items():
            x[b, h, t] = torch.from_numpy(np.asarray(v)).to(device)
        return x


def kivi_needle_tokens(n_packed: int, offset: int, group_size: int, chunk: int = 64) -> list[int]:
    """Needle tokens of a KIVI cache: whole key groups in the packed region (a group of identical
    rows has a zero range, so its keys are stored exactly and every needle scores alike) at the
    first chunk, a chunk boundary, deep in the region and its last group; single tokens in the
    fp16 window."""
    toks = []
    groups = n_packed // group_size
    if groups > 0:
        gsel = {0, min(groups - 1, chunk // group_size), groups // 2 + 1, groups - 1}
        for gi in sorted(gsel):
            toks.extend(range(gi * group_size, (gi + 1) * group_size))
    for t in (n_packed, (n_packed + offset) // 2, offset - 1):
        if n_packed <= t < offset:
            toks.append(t)
    return sorted(set(toks))
