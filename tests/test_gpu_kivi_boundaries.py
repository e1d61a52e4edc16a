"""GPU parity of the 2-bit KIVI flush at every fp16 value of chosen groups.

The 2-bit flush decides an element's code by comparing it, as fp16, with its group's three code
boundaries: for each code, the smallest fp16 value whose float32 difference from gmin reaches the
code's threshold.  These cases sweep every fp16 value (every k-th where there are too many)
between a group's min and max: groups whose boundaries fall among subnormals, around zero where
hundreds of fp16 values share one float32 difference, at the ends of the fp16 range, all-negative
and very narrow groups, and groups where eps sets the scale.  Keys (groups along tokens) and
values (groups along channels) at every value-group width the 2-bit kernel takes (one, two, three
and four 16-byte vectors), compared with the oracle's round trip bit for bit; and the same sweeps
through the packed form (2-bit codes against the stored fp16 scale), codes and group parameters
compared with the oracle's packing bit for bit, at head dim 64 (a warp per key token group) and
at other head dims.
"""
import numpy as np
import pytest
import torch

from oracle import kivi as ok
from oracle import kivi_packed as P
from _gpu_util import dev_tensor, u16

pytestmark = pytest.mark.gpu

_ALL = np.arange(65536, dtype=np.uint32).astype(np.uint16).view(np.float16)
_FINITE = np.sort(_ALL[np.isfinite(_ALL)].astype(np.float32), kind="stable").astype(np.float16)

CASES = [  # (gmin, gmax, eps)
    (-1.0, 1.0, 1e-8),            # middle boundary at 0: subnormals, both zeros
    (-1000.0, 1000.0, 1e-8),      # ~1000 fp16 values per float32 step of the difference near 0
    (-65504.0, 65504.0, 1e-8),    # the whole finite range
    (-2.0 ** -14, 2.0 ** -14, 1e-8),
    (0.0, 2.25, 1e-8),            # exact ties at 0.375, 1.125, 1.875
    (-3.0, -1.0, 1e-8),
    (5.0, 5.0078125, 1e-8),       # three fp16 ulps wide
    (-0.0, 3 * 2.0 ** -24, 1e-8),  # eps sets the scale
    (-0.001, 3000.0, 1e-8),
    (60000.0, 65504.0, 1e-8),
    (-65504.0, -60000.0, 1e-8),
    (-0.5, 0.75, 1e-3),
    (-1e-4, 1e-4, 1e-3),          # eps far above the range: everything is code 0 or 1
]
SHAPES = [(8, 64), (16, 64), (24, 96), (32, 64)]   # (group size, head dim)
PACK_SHAPES = [(8, 64), (16, 64), (32, 64), (64, 64), (32, 96), (16, 128)]


def _sweep(mn, mx, cap):
    f = _FINITE[(_FINITE >= np.float16(mn)) & (_FINITE <= np.float16(mx))]
    if len(f) > cap:
        f = f[np.linspace(0, len(f) - 1, cap).astype(np.int64)]
    return f


def _groups(vals, mn, mx, gs, n_groups, rng):
    """n_groups groups of gs elements: gmin, gmax and gs - 2 swept values (padded with gmin),
    shuffled within each group."""
    free = gs - 2
    flat = np.full(n_groups * free, np.float16(mn), dtype=np.float16)
    flat[:len(vals)] = vals
    g = np.empty((n_groups, gs), np.float16)
    g[:, 0] = np.float16(mn)
    g[:, 1] = np.float16(mx)
    g[:, 2:] = flat.reshape(n_groups, free)
    return rng.permuted(g, axis=1)


def _swept_pair(mn, mx, gs, D, cap=61440):
    """Key and value tensors [1, 1, S, D] whose groups (keys: gs tokens of a channel; values: gs
    channels of a token) hold gmin, gmax and the swept values."""
    assert D % gs == 0, "head dim must hold whole value groups here"
    vals = _sweep(mn, mx, cap)
    S = gs * -(-len(vals) // ((gs - 2) * D))
    n_groups = S * D // gs
    rng = np.random.default_rng(len(vals) + gs)
    gk = _groups(vals, mn, mx, gs, n_groups, rng)
    gv = _groups(vals[::-1].copy(), mn, mx, gs, n_groups, rng)
    # keys: group q = (token group q // D, channel q % D); values: (token q // (D / gs), slice)
    k = gk.reshape(S // gs, D, gs).transpose(0, 2, 1).reshape(1, 1, S, D).copy()
    v = gv.reshape(1, 1, S, D).copy()
    return k, v, S


@pytest.mark.parametrize("gs,D", SHAPES)
@pytest.mark.parametrize("mn,mx,eps", CASES)
def test_every_fp16_value_of_a_group(kvq, cuda_dev, gs, D, mn, mx, eps):
    k, v, S = _swept_pair(mn, mx, gs, D)
    kt, vt = dev_tensor(k, cuda_dev), dev_tensor(v, cuda_dev)
    kvq.kivi_quant_dequant([kt, vt], [True, False], 0, S, gs, 3, eps)
    torch.cuda.synchronize()
    ok.flush(k, v, 0, S, gs, 3, eps)
    assert np.array_equal(u16(kt), k.view(np.uint16))
    assert np.array_equal(u16(vt), v.view(np.uint16))


def _same_zero_param(got, ref):
    """Stored zeros (group minima) bit for bit, except that a group holding both -0 and +0 may
    store either as its minimum: the pages order no zeros, and neither the codes (x - (-0) equals
    x - (+0)) nor the reconstruction (c * scale + zero) depends on that sign."""
    both = ((got & 0x7fff) == 0) & ((ref & 0x7fff) == 0)
    return np.array_equal(np.where(both, 0, got), np.where(both, 0, ref))


@pytest.mark.parametrize("gs,D", PACK_SHAPES)
@pytest.mark.parametrize("mn,mx,eps", CASES)
def test_every_fp16_value_of_a_packed_group(kvq, cuda_dev, gs, D, mn, mx, eps):
    k, v, S = _swept_pair(mn, mx, gs, D)
    c = kvq.KiviPacked.empty(2, gs, 1, 1, S, D, cuda_dev)
    kvq.kivi_pack([c], [dev_tensor(k, cuda_dev)], [dev_tensor(v, cuda_dev)], 0, S, eps)
    torch.cuda.synchronize()
    kc, ksc, kz = P.pack_keys(k, 2, gs, eps)
    vc, vsc, vz = P.pack_values(v, 2, gs, eps)
    assert np.array_equal(u16(c.k_scale), ksc.view(np.uint16))
    assert _same_zero_param(u16(c.k_zero), kz.view(np.uint16))
    assert np.array_equal(c.k_codes.cpu().numpy(), kc)
    assert np.array_equal(u16(c.v_scale), vsc.view(np.uint16))
    assert _same_zero_param(u16(c.v_zero), vz.view(np.uint16))
    assert np.array_equal(c.v_codes.cpu().numpy(), vc)
