"""kvq_decode_attn_noalloc, the decode attention for callers that cannot allocate device memory
(its split partials live in the library's own static device array instead of a workspace the
caller allocates).  Called through the C ABI several times in a row -- each call on a different
problem, over whatever the one before left in the shared array -- and checked against
kvq_decode_attn with a workspace and against the oracle, within the attention tolerance of the
other tests.  One problem is large enough that the split count the workspace version would use
does not fit in the static array, so the entry point takes fewer, longer splits.  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import kvgen
from oracle import attention as oa
from oracle import symmetric as osym
from _attn_checks import assert_attn_close, decode_tiles_per_cta
from _gpu_util import cu_of, dev_tensor, i32

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 32 << 20          # the library's static scratch
RECORD_BYTES = 8 * (256 + 4) * 4  # one split's partial record per (layer, sequence, KV head)


def _problem(kvq, dev, n_layers, lens, H, G, bits, seed):
    """Pools quantized from generated rows, with the oracle's copies."""
    D, ps = 256, 16
    pps = max((n + ps - 1) // ps for n in lens)
    pt_np = kvgen.random_page_table(seed, len(lens), pps)
    pt = i32(pt_np, dev)
    cu = i32(cu_of(lens), dev)
    st = i32([0] * len(lens), dev)
    tot = int(sum(lens))
    kps, vps, host = [], [], []
    for layer in range(n_layers):
        pair = []
        for is_key, dst in ((True, kps), (False, vps)):
            x = kvgen.KVSpec(seed=seed, layer=layer, is_key=is_key, n_seq=1, n_tok=tot,
                             num_heads=H, head_dim=D).full_np()
            p = kvq.Pool.empty(bits, H, D, ps, pt_np.size, dev)
            kvq.kvq_quant_pack_paged([p], [dev_tensor(x, dev)], pt, cu, st)
            dst.append(p)
            op = osym.PagedPool(bits, H, D, ps, pt_np.size)
            osym.quant_pack_paged(op, x, pt_np, cu_of(lens), np.zeros(len(lens)))
            pair.append(op)
        host.append(pair)
    q = kvgen.queries_np(seed, n_layers, len(lens), H * G, D)
    return kps, vps, dev_tensor(q, dev), pt, i32(lens, dev), int(max(lens)), (q, host, pt_np)


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


def test_noalloc_decode_attention_matches_workspace_version_and_oracle(kvq, cuda_dev):
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    problems = [
        # a few long sequences (many splits per sequence)
        dict(n_layers=2, lens=[1000, 5000, 17], H=4, G=6, bits=6, seed=21),
        # 16 layers x 8 sequences x 4 heads: many (layer, sequence, head) units, short splits
        dict(n_layers=16, lens=[700, 64, 1, 300, 900, 16, 33, 512], H=4, G=6, bits=8, seed=22),
    ]
    for prob in problems:
        kps, vps, q, pt, lens_t, max_len, (qn, host, pt_np) = _problem(kvq, cuda_dev, **prob)
        ref = _reference(kvq, cuda_dev, kps, vps, q, pt, lens_t, max_len)
        out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
        status = _noalloc_cabi(kvq, kps, vps, q, pt, lens_t, max_len, out, err)
        assert status == 0, kvq._lib.kvq_last_error()
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        got = out.cpu().numpy().astype(np.float64)
        assert_attn_close(got, ref.cpu().numpy().astype(np.float64), "vs workspace version")
        for layer, (okp, ovp) in enumerate(host):
            want = oa.decode_attention_paged(qn[layer], okp, ovp, pt_np, np.array(prob["lens"]),
                                             0.0625)
            assert_attn_close(got[layer], want, f"vs oracle, layer {layer}")


def test_noalloc_caps_its_split_count_to_the_scratch(kvq, cuda_dev):
    """16 layers x 1 sequence x 4 KV heads x 262,144 tokens: the workspace version takes 64 splits
    of 256 tiles, one more than the static array holds (63 records of 16 x 4 partials), so the
    entry point takes 63 splits of 264 tiles.  The 16,384 logical pages of the sequence map onto
    a pool of 64 physical pages (page ids are only range-checked), so the problem needs no large
    allocation.  Checked against the workspace version on every output and against the oracle on
    two (layer, KV head) pairs."""
    L, H, G, D, ps, bits, T = 16, 4, 6, 256, 16, 6, 262144
    n_phys = 64
    units = L * 1 * H
    max_splits = SCRATCH_BYTES // (units * RECORD_BYTES)
    sms = torch.cuda.get_device_properties(cuda_dev).multi_processor_count
    tiles = T // 16
    usual = -(-tiles // decode_tiles_per_cta(L, 1, H, T, sms))
    assert usual > max_splits, "the problem must exceed the static scratch"
    # physical pages: one 1,024-token sequence quantized through the identity table
    ident = np.arange(n_phys, dtype=np.int32)[None]
    rng = np.random.default_rng(23)
    pt_np = rng.integers(0, n_phys, size=(1, tiles), dtype=np.int32)
    kps, vps, host = [], [], []
    for layer in range(L):
        pair = []
        for is_key, dst in ((True, kps), (False, vps)):
            x = kvgen.KVSpec(seed=24, layer=layer, is_key=is_key, n_seq=1, n_tok=n_phys * ps,
                             num_heads=H, head_dim=D).full_np()
            p = kvq.Pool.empty(bits, H, D, ps, n_phys, cuda_dev)
            kvq.kvq_quant_pack_paged([p], [dev_tensor(x, cuda_dev)], i32(ident, cuda_dev),
                                     i32([0, n_phys * ps], cuda_dev), i32([0], cuda_dev))
            dst.append(p)
            op = osym.PagedPool(bits, H, D, ps, n_phys)
            osym.quant_pack_paged(op, x, ident, np.array([0, n_phys * ps]), np.array([0]))
            pair.append(op)
        host.append(pair)
    qn = kvgen.queries_np(25, L, 1, H * G, D)
    q, pt, lens_t = dev_tensor(qn, cuda_dev), i32(pt_np, cuda_dev), i32([T], cuda_dev)
    ref = _reference(kvq, cuda_dev, kps, vps, q, pt, lens_t, T)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
    status = _noalloc_cabi(kvq, kps, vps, q, pt, lens_t, T, out, err)
    assert status == 0, kvq._lib.kvq_last_error()
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    assert_attn_close(got, ref.cpu().numpy().astype(np.float64), "vs workspace version")
    for layer, h in ((0, 0), (L - 1, H - 1)):
        okp, ovp = host[layer]
        k_hat = oa.gather_dequant(okp, pt_np, 0, T, heads=[h])
        v_hat = oa.gather_dequant(ovp, pt_np, 0, T, heads=[h])
        want = oa.attend(qn[layer, 0, h * G:(h + 1) * G], k_hat[:, h:h + 1], v_hat[:, h:h + 1],
                         0.0625)
        assert_attn_close(got[layer, 0, h * G:(h + 1) * G], want, f"vs oracle, layer {layer}")


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
