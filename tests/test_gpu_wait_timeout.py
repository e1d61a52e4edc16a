"""The bounded stage waits give up cleanly (GPU).

The staged decode attention and the packed KIVI attention wait on an mbarrier for each tile's
bulk copies, with a bounded number of polls; a wait that runs out sets KVQ_DEVERR_TIMEOUT in the
caller's error word, drains the copies already in flight (with the normal bound, so every issued
copy completes before the block exits) and returns empty partials.  Here the two kernels are
built a second time with a stage-wait limit of 0 polls, so every first wait gives up at once while
its copies are still in flight; the call must return, report the timeout, produce the empty
result (zeros), and leave the context usable: the library's own build then computes the same
problem correctly.  No fault is planted and nothing waits without a bound."""
import ctypes
import concurrent.futures as cf
import os
import subprocess

import numpy as np
import pytest
import torch

import kvgen
from conftest import ROOT
from oracle import attention as oa
from oracle import kivi_packed as okp
from oracle import symmetric as osym
from _attn_checks import assert_attn_close
from _gpu_util import cu_of, dev_tensor, i32

pytestmark = pytest.mark.gpu

CSRC = os.path.join(ROOT, "paged_kv_cache_fp16_gb300", "csrc")


@pytest.fixture(scope="module")
def short_wait_lib(kvq):
    out_dir = os.path.join(ROOT, "tests", "_build")
    os.makedirs(out_dir, exist_ok=True)
    nvcc = os.environ.get("NVCC", "nvcc")
    flags = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-Xcompiler",
             "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include"),
             "-I", CSRC, "--expt-relaxed-constexpr", "-diag-suppress", "177",
             "-DKVQ_STAGE_WAIT_LIMIT=0"]
    srcs = ["decode_attn.cu", "kivi_packed.cu", "host.cpp"]

    def compile_one(name):
        obj = os.path.join(out_dir, "stage_wait0_" + name + ".o")
        subprocess.run([nvcc] + flags + ["-c", os.path.join(CSRC, name), "-o", obj], check=True,
                       capture_output=True)
        return obj

    with cf.ThreadPoolExecutor(len(srcs)) as ex:
        objs = list(ex.map(compile_one, srcs))
    so = os.path.join(out_dir, "kvq_stage_wait0.so")
    subprocess.run([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", so]
                   + objs, check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    P, I, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    pool_p = ctypes.POINTER(kvq.kvq_pool)
    lib.kvq_decode_attn.restype = I
    lib.kvq_decode_attn.argtypes = [pool_p, pool_p, I, P, I, P, I, P, I, I, F, P, P, S, P, P]
    lib.kivi_decode_attn.restype = I
    lib.kivi_decode_attn.argtypes = [ctypes.POINTER(kvq.kivi_packed), P, P, I, P, I, I, I, F, P,
                                     P, S, P, P]
    return lib


def test_decode_attention_stage_wait_timeout_is_reported(kvq, cuda_dev, short_wait_lib):
    bits, H, G, D, ps = 6, 2, 3, 256, 16
    lens = [100, 700]
    pt_np = kvgen.random_page_table(71, 2, 44)
    tot = int(sum(lens))
    k = kvgen.KVSpec(seed=72, layer=0, is_key=True, n_seq=1, n_tok=tot, num_heads=H,
                     head_dim=D).full_np()
    v = kvgen.KVSpec(seed=72, layer=0, is_key=False, n_seq=1, n_tok=tot, num_heads=H,
                     head_dim=D).full_np()
    kp = kvq.Pool.empty(bits, H, D, ps, pt_np.size, cuda_dev)
    vp = kvq.Pool.empty(bits, H, D, ps, pt_np.size, cuda_dev)
    pt = i32(pt_np, cuda_dev)
    kvq.kvq_quant_pack_paged([kp, vp], [dev_tensor(k, cuda_dev), dev_tensor(v, cuda_dev)], pt,
                             i32(cu_of(lens), cuda_dev), i32([0, 0], cuda_dev))
    q = dev_tensor(kvgen.queries_np(73, 1, 2, H * G, D), cuda_dev)
    lens_t = i32(lens, cuda_dev)
    ws = kvq.decode_workspace([kp], 2, H * G, max(lens), cuda_dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    st = short_wait_lib.kvq_decode_attn(
        kvq._pool_array([kp]), kvq._pool_array([vp]), 1, q.data_ptr(), H * G, pt.data_ptr(),
        pt.shape[1], lens_t.data_ptr(), 2, max(lens), 1.0 / 16, out.data_ptr(), ws.data_ptr(),
        ws.numel(), err.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) & kvq.KVQ_DEVERR_TIMEOUT
    assert torch.count_nonzero(out).item() == 0
    # the context is still usable: the library's build computes the same call correctly
    err.zero_()
    out.fill_(float("nan"))
    kvq.kvq_decode_attn([kp], [vp], q, pt, lens_t, max(lens), 1.0 / 16, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    okp_, ovp_ = osym.PagedPool(bits, H, D, ps, pt_np.size), osym.PagedPool(bits, H, D, ps,
                                                                           pt_np.size)
    osym.quant_pack_paged(okp_, k, pt_np, cu_of(lens), np.zeros(2))
    osym.quant_pack_paged(ovp_, v, pt_np, cu_of(lens), np.zeros(2))
    ref = oa.decode_attention_paged(q.cpu().numpy()[0], okp_, ovp_, pt_np, np.array(lens),
                                    1.0 / 16)
    assert_attn_close(out.cpu().numpy()[0].astype(np.float64), ref)


def test_kivi_attention_stage_wait_timeout_is_reported(kvq, cuda_dev, short_wait_lib):
    L, B, H, G, S, D, gs = 1, 2, 2, 4, 512, 64, 32
    n_packed, offset = 384, 450
    k = kvgen.KiviSpec(seed=74, layer=0, is_key=True, batch=B, num_heads=H, seq=S,
                       head_dim=D).full_torch(cuda_dev)
    v = kvgen.KiviSpec(seed=74, layer=0, is_key=False, batch=B, num_heads=H, seq=S,
                       head_dim=D).full_torch(cuda_dev)
    c = kvq.KiviPacked.empty(2, gs, B, H, S, D, cuda_dev)
    kvq.kivi_pack([c], [k], [v], 0, n_packed)
    q = dev_tensor(kvgen.queries_np(75, L, B, H * G, D), cuda_dev)
    nbytes = kvq.kivi_decode_attn_workspace(L, B, H, H * G, D, offset)
    ws = torch.empty(max(16, nbytes), dtype=torch.uint8, device=cuda_dev)
    out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    ks = (ctypes.c_void_p * 1)(k.data_ptr())
    vs = (ctypes.c_void_p * 1)(v.data_ptr())
    st = short_wait_lib.kivi_decode_attn(
        kvq._packed_array([c]), ks, vs, L, q.data_ptr(), H * G, n_packed, offset, 0.125,
        out.data_ptr(), ws.data_ptr(), ws.numel(), err.data_ptr(),
        torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) & kvq.KVQ_DEVERR_TIMEOUT
    assert torch.count_nonzero(out).item() == 0
    err.zero_()
    out.fill_(float("nan"))
    kvq.kivi_decode_attn([c], [k], [v], q, n_packed, offset, 0.125, out, ws, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    kn, vn = k.cpu().numpy(), v.cpu().numpy()
    ref = okp.decode_attention(q.cpu().numpy()[0], okp.pack_keys(kn[:, :, :n_packed], 2, gs),
                               okp.pack_values(vn[:, :, :n_packed], 2, gs),
                               kn[:, :, n_packed:offset], vn[:, :, n_packed:offset], 2, gs, 0.125)
    assert_attn_close(out.cpu().numpy()[0].astype(np.float64), ref)
