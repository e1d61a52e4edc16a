"""kvq_decode_attn_noalloc, the decode attention for callers that cannot allocate device memory
(its split partials live in the library's own static device array instead of a workspace the
caller allocates).  Called through the C ABI twice in a row -- the second call on a different
problem, over whatever the first left in the shared array -- and checked against
kvq_decode_attn with a workspace, within the attention tolerance of the other tests.  This file
is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import kvgen
from _gpu_util import cu_of, dev_tensor, i32

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-3


def _problem(kvq, dev, n_layers, lens, H, G, bits, seed):
    D, ps = 256, 16
    pps = max((n + ps - 1) // ps for n in lens)
    pt_np = kvgen.random_page_table(seed, len(lens), pps)
    pt = i32(pt_np, dev)
    cu = i32(cu_of(lens), dev)
    st = i32([0] * len(lens), dev)
    tot = int(sum(lens))
    kps, vps = [], []
    for layer in range(n_layers):
        for is_key, dst in ((True, kps), (False, vps)):
            x = kvgen.KVSpec(seed=seed, layer=layer, is_key=is_key, n_seq=1, n_tok=tot,
                             num_heads=H, head_dim=D).full_torch(dev)
            p = kvq.Pool.empty(bits, H, D, ps, pt_np.size, dev)
            kvq.kvq_quant_pack_paged([p], [x], pt, cu, st)
            dst.append(p)
    q = kvgen.queries_torch(seed, n_layers, len(lens), H * G, D, dev)
    return kps, vps, q, pt, i32(lens, dev), int(max(lens))


def _reference(kvq, dev, kps, vps, q, pt, lens_t, max_len):
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    ws = kvq.decode_workspace(kps, q.shape[1], q.shape[2], max_len, dev)
    kvq.kvq_decode_attn(kps, vps, q, pt, lens_t, max_len, 0.0625, out, ws)
    return out


def _noalloc_cabi(kvq, kps, vps, q, pt, lens_t, max_len, out, err):
    """Direct C-ABI call (ctypes), no workspace argument."""
    return kvq._lib.kvq_decode_attn_noalloc(
        kvq._pool_array(kps), kvq._pool_array(vps), len(kps), ctypes.c_void_p(q.data_ptr()),
        q.shape[2], ctypes.c_void_p(pt.data_ptr()), pt.shape[1],
        ctypes.c_void_p(lens_t.data_ptr()), q.shape[1], max_len, ctypes.c_float(0.0625),
        ctypes.c_void_p(out.data_ptr()), ctypes.c_void_p(err.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_decode_attention_matches_workspace_version_twice(kvq, cuda_dev):
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    problems = [
        # a few long sequences: the usual split count fits in the static array
        dict(n_layers=2, lens=[1000, 5000, 17], H=4, G=6, bits=6, seed=21),
        # 16 layers x 8 sequences x 4 heads: the split count is capped to fit the array
        dict(n_layers=16, lens=[700, 64, 1, 300, 900, 16, 33, 512], H=4, G=6, bits=8, seed=22),
    ]
    for prob in problems:
        kps, vps, q, pt, lens_t, max_len = _problem(kvq, cuda_dev, **prob)
        ref = _reference(kvq, cuda_dev, kps, vps, q, pt, lens_t, max_len)
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
        status = _noalloc_cabi(kvq, kps, vps, q, pt, lens_t, max_len, out, err)
        assert status == 0, kvq._lib.kvq_last_error()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got, want = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        bad = np.abs(got - want) > ATOL + RTOL * np.abs(want)
        assert not bad.any(), float(np.abs(got - want).max())


def test_noalloc_rejects_problems_beyond_its_scratch(kvq, cuda_dev):
    # 64 layers x 16 sequences x 4 heads = 4,096 units: more than the array holds with one split
    H, D, ps = 4, 256, 16
    pools = [kvq.Pool.empty(6, H, D, ps, 1, cuda_dev) for _ in range(64)]
    q = torch.zeros((64, 16, 24, D), dtype=torch.float16, device=cuda_dev)
    out = torch.zeros((64, 16, 24, D), dtype=torch.float32, device=cuda_dev)
    pt = torch.zeros((16, 1), dtype=torch.int32, device=cuda_dev)
    lens_t = torch.ones(16, dtype=torch.int32, device=cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    status = _noalloc_cabi(kvq, pools, pools, q, pt, lens_t, 1, out, err)
    assert status == 5
    assert b"static scratch" in kvq._lib.kvq_last_error()
