"""GPU parity at the largest counts one call accepts: 64 tensors (KVQ_MAX_TENSORS) in one
quant-pack / dequant / KIVI call, 64 layers in one decode-attention call, and 32 layers in one
KIVI protocol update (its K and V make 64 tensors) -- every tensor checked against the oracle."""
import numpy as np
import pytest
import torch

import kvgen
from oracle import attention as oa
from oracle import kivi as K
from oracle import symmetric as osym
from _gpu_util import cu_of, dev_tensor, i32, u16

pytestmark = pytest.mark.gpu


def _rows(seed, layer, is_key, n, H, D):
    return kvgen.KVSpec(seed=seed, layer=layer, is_key=is_key, n_seq=1, n_tok=n, num_heads=H,
                        head_dim=D).full_np()


def test_quant_dequant_64_tensors(kvq, cuda_dev):
    bits, H, D, ps = 6, 2, 64, 16
    lens = [5, 19]
    pt_np = kvgen.random_page_table(3, 2, 2)
    pt, cu, st = i32(pt_np, cuda_dev), i32(cu_of(lens), cuda_dev), i32([0, 0], cuda_dev)
    xs = [_rows(50 + i // 2, i // 2, i % 2 == 0, sum(lens), H, D) for i in range(64)]
    pools = [kvq.Pool.empty(bits, H, D, ps, pt_np.size, cuda_dev) for _ in xs]
    for p in pools:
        p.codes.zero_()
        p.scales.zero_()
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_quant_pack_paged(pools, [dev_tensor(x, cuda_dev) for x in xs], pt, cu, st, err)
    outs = [torch.empty((sum(lens), H, D), dtype=torch.float16, device=cuda_dev) for _ in xs]
    kvq.kvq_dequant_paged(pools, outs, pt, cu, st, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    for x, p, o in zip(xs, pools, outs):
        op = osym.PagedPool(bits, H, D, ps, pt_np.size)
        osym.quant_pack_paged(op, x, pt_np, cu_of(lens), np.zeros(2))
        assert np.array_equal(p.codes.cpu().numpy(), op.codes)
        assert np.array_equal(u16(o), osym.dequant_paged(op, pt_np, cu_of(lens), np.zeros(2)).view(np.uint16))


def test_decode_attention_64_layers(kvq, cuda_dev):
    bits, H, G, D, ps, L = 4, 1, 2, 256, 16, 64
    lens = [3, 17]
    pt_np = kvgen.random_page_table(4, 2, 2)
    pt, cu, st = i32(pt_np, cuda_dev), i32(cu_of(lens), cuda_dev), i32([0, 0], cuda_dev)
    kps, vps, refs = [], [], []
    q = kvgen.queries_np(5, L, 2, H * G, D)
    for layer in range(L):
        k, v = _rows(60, layer, True, sum(lens), H, D), _rows(60, layer, False, sum(lens), H, D)
        kp = kvq.Pool.empty(bits, H, D, ps, pt_np.size, cuda_dev)
        vp = kvq.Pool.empty(bits, H, D, ps, pt_np.size, cuda_dev)
        kvq.kvq_quant_pack_paged([kp, vp], [dev_tensor(k, cuda_dev), dev_tensor(v, cuda_dev)], pt,
                                 cu, st)
        okp, ovp = osym.PagedPool(bits, H, D, ps, pt_np.size), osym.PagedPool(bits, H, D, ps, pt_np.size)
        osym.quant_pack_paged(okp, k, pt_np, cu_of(lens), np.zeros(2))
        osym.quant_pack_paged(ovp, v, pt_np, cu_of(lens), np.zeros(2))
        kps.append(kp); vps.append(vp)
        refs.append(oa.decode_attention_paged(q[layer], okp, ovp, pt_np, np.array(lens), 1 / 16))
    out = torch.empty(q.shape, dtype=torch.float32, device=cuda_dev)
    ws = kvq.decode_workspace(kps, 2, H * G, max(lens), cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    kvq.kvq_decode_attn(kps, vps, dev_tensor(q, cuda_dev), pt, i32(lens, cuda_dev), max(lens),
                        1 / 16, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    for layer in range(L):
        ref = refs[layer]
        assert np.all(np.abs(got[layer] - ref) <= 2e-3 + 1e-3 * np.abs(ref))


def test_kivi_64_tensors_and_32_layer_protocol(kvq, cuda_dev):
    B, H, S, D, gs = 1, 2, 256, 64, 32
    xs = [kvgen.KiviSpec(seed=70 + i // 2, layer=i // 2, is_key=i % 2 == 0, batch=B, num_heads=H,
                         seq=S, head_dim=D).full_np() for i in range(64)]
    flags = [i % 2 == 0 for i in range(64)]
    dev = [dev_tensor(x, cuda_dev) for x in xs]
    kvq.kivi_quant_dequant(dev, flags, 32, 160, gs, 3, 1e-8)
    torch.cuda.synchronize()
    for x, f, d in zip(xs, flags, dev):
        want = x.copy()
        axis = -2 if f else -1
        want[:, :, 32:160] = K.quant_dequant_along(x[:, :, 32:160], axis, gs, 3)
        assert np.array_equal(u16(d), want.view(np.uint16))
    # the protocol over 32 layers (64 tensors): one append of 200 tokens, then a trim
    st = kvq.kivi_state_new(B, H, D, S, bits=2, group_size=gs, residual_length=64)
    kc = [torch.zeros((B, H, S, D), dtype=torch.float16, device=cuda_dev) for _ in range(32)]
    vc = [torch.zeros_like(kc[0]) for _ in range(32)]
    kn = [dev_tensor(np.ascontiguousarray(xs[2 * l][:, :, :200]), cuda_dev) for l in range(32)]
    vn = [dev_tensor(np.ascontiguousarray(xs[2 * l + 1][:, :, :200]), cuda_dev) for l in range(32)]
    kvq.kivi_update(st, kc, vc, kn, vn)
    torch.cuda.synchronize()
    assert (st.offset, st.n_quantized) == (200, 128)
    for l in (0, 31):
        ref = K.KiviCache(B, H, D, S, bit_width=2, group_size=gs, residual_length=64)
        rk, rv = ref.update_and_fetch(xs[2 * l][:, :, :200], xs[2 * l + 1][:, :, :200])
        assert np.array_equal(u16(kc[l][:, :, :200]), rk.view(np.uint16))
        assert np.array_equal(u16(vc[l][:, :, :200]), rv.view(np.uint16))
    assert kvq.kivi_trim(st, 90) == 90 and (st.offset, st.n_quantized) == (110, 96)
