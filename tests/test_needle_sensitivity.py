"""The attention parity checks can see one lost or misplaced tile (CPU, oracle only).

At the full-context size a whole-window decode output averages 262,144 tokens, so its magnitude is
small against the absolute tolerance and one 16-token tile dropped from the cache moves it by less
than the tolerance.  The GPU parity tests therefore plant needles (identical key rows along one
query head's direction) at the tiles a schedule gets wrong: first and last tile, both sides of a
split boundary, deep in a warp's stream, the middle split, the last token.  Here the oracle's own
result on the needled input is compared, with the GPU tests' tolerance, against the oracle's
result on the same input with one tile lost, read from the wrong page, or read from a stale stage;
each mistake must fall outside the tolerance.  Mistakes are made in the oracle's input on the CPU,
never in a kernel.
"""
import numpy as np
import pytest

import kvgen
from oracle import attention as oa
from oracle import kivi_packed as okp
from oracle import symmetric as osym
from _attn_checks import (TILE, Planted, PlantedKivi, attn_close, attn_report, decode_tiles_per_cta,
                          kivi_needle_tokens, needle_row, paged_needle_positions, plant_needles)

W = kvgen.WORKLOADS["decode_attn_262144_16L_4x256_gqa6"]


@pytest.fixture(scope="module")
def full_context_head():
    """Layer 0, KV head 0 of the full-context workload, needles planted for query head 0, and
    the oracle's dequantized K and V of that head (q6)."""
    T, H, D, hq = W["n_tok"], W["H"], W["D"], W["Hq"]
    G = hq // H
    scale = W["softmax_scale"]
    q = kvgen.queries_np(W["seed"], W["n_layers"], 1, hq, D)[0, 0, :G]
    tpc = decode_tiles_per_cta(W["n_layers"], 1, H, T, 152)
    pos = paged_needle_positions(T, tpc, stages=2)
    ks = Planted(kvgen.KVSpec(seed=W["seed"], layer=0, is_key=True, n_seq=1, n_tok=T,
                              num_heads=H, head_dim=D))
    plant_needles(ks, 0, 0, pos, needle_row(q[0], scale))
    vs = kvgen.KVSpec(seed=W["seed"], layer=0, is_key=False, n_seq=1, n_tok=T, num_heads=H,
                      head_dim=D)
    rows = np.arange(T, dtype=np.int64) * H
    k_hat = osym.dequant_rows(*osym.quant_pack_rows(ks.rows_np(rows), 6), 6, D)
    v_hat = osym.dequant_rows(*osym.quant_pack_rows(vs.rows_np(rows), 6), 6, D)
    return q[:2], k_hat[:, None, :], v_hat[:, None, :], scale, pos, tpc


def _attend(q, k, v, scale):
    return oa.attend(q, k, v, scale)


def test_needles_dominate_their_head(full_context_head):
    q, k, v, scale, pos, _ = full_context_head
    ref = _attend(q[:1], k, v, scale)[0]
    mean_needles = v[pos, 0].astype(np.float64).mean(0)
    # the needle head's output is the mean of the needle tokens' values to far inside the tolerance
    assert np.abs(ref - mean_needles).max() < 1e-4
    assert len(pos) >= 5


def test_a_dropped_needle_tile_falls_outside_the_tolerance(full_context_head):
    q, k, v, scale, pos, _ = full_context_head
    ref = _attend(q, k, v, scale)
    for p in pos:
        t0 = (p // TILE) * TILE
        keep = np.r_[0:t0, t0 + TILE:k.shape[0]]
        got = _attend(q, k[keep], v[keep], scale)
        assert not attn_close(got[:1], ref[:1]), (p, attn_report(got[:1], ref[:1]))


def test_a_wrong_page_or_stale_stage_falls_outside_the_tolerance(full_context_head):
    """A page-table off-by-one (the needle's 16-token page read from the next page) and a stage
    read one ring turn late (the values of the tile two tiles earlier in the warp's stream: 2 stages,
    4 warps) both move the needle head's output outside the tolerance."""
    q, k, v, scale, pos, _ = full_context_head
    ref = _attend(q[:1], k, v, scale)
    T = k.shape[0]
    for p in pos:
        t0 = (p // TILE) * TILE
        nxt = t0 + TILE if t0 + TILE < T else t0 - TILE
        k2, v2 = k.copy(), v.copy()
        k2[t0:t0 + TILE], v2[t0:t0 + TILE] = k[nxt:nxt + TILE], v[nxt:nxt + TILE]
        assert not attn_close(_attend(q[:1], k2, v2, scale), ref), ("page", p)
        stale = t0 - 2 * 4 * TILE
        if stale >= 0:
            v3 = v.copy()
            v3[t0:t0 + TILE] = v[stale:stale + TILE]
            assert not attn_close(_attend(q[:1], k, v3, scale), ref), ("stage", p)


def test_kivi_needle_groups_store_exactly_and_are_seen():
    """A KIVI key group of identical needle rows has a zero range, so the packed keys reconstruct
    it exactly; dropping one 64-token chunk that holds needles moves the needle head's output
    outside the tolerance."""
    B, H, S, D, gs = 1, 1, 4096, 64, 32
    n_packed, offset, scale = 3968, 4096, 0.125
    q = kvgen.queries_np(3, 1, 1, 4, D)[0, 0]
    ks = PlantedKivi(kvgen.KiviSpec(seed=3, layer=0, is_key=True, batch=B, num_heads=H, seq=S,
                                    head_dim=D))
    vs = kvgen.KiviSpec(seed=3, layer=0, is_key=False, batch=B, num_heads=H, seq=S, head_dim=D)
    toks = kivi_needle_tokens(n_packed, offset, gs)
    row = needle_row(q[0], scale)
    for t in toks:
        ks.rows[(0, 0, t)] = row
    k = ks.full_np()
    v = vs.full_np()
    kp = okp.pack_keys(k[:, :, :n_packed], 2, gs)
    vp = okp.pack_values(v[:, :, :n_packed], 2, gs)
    k_hat = okp.unpack_keys(*kp, 2, gs, D)
    packed_needles = [t for t in toks if t < n_packed]
    assert np.array_equal(k_hat[0, 0, packed_needles].view(np.uint16),
                          np.broadcast_to(row, (len(packed_needles), D)).view(np.uint16))
    ref = okp.decode_attention(q[None], kp, vp, k[:, :, n_packed:offset], v[:, :, n_packed:offset],
                               2, gs, scale)[0]
    for t in (packed_needles[0], packed_needles[-1]):
        c0 = (t // 64) * 64
        keep = np.r_[0:c0, c0 + 64:n_packed]
        kp2 = okp.pack_keys(k[:, :, keep], 2, gs)
        vp2 = okp.pack_values(v[:, :, keep], 2, gs)
        got = okp.decode_attention(q[None], kp2, vp2, k[:, :, n_packed:offset],
                                   v[:, :, n_packed:offset], 2, gs, scale)[0]
        assert not attn_close(got[:1], ref[:1]), t
