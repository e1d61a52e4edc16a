"""kvq_host_device_view: kernels reading page-locked host memory in place.  Quant-pack from a
HostView of pinned fp16 rows equals quant-pack from the same rows on the device, byte for byte;
pageable host memory is refused before any launch."""
import ctypes

import numpy as np
import pytest
import torch

import kvgen
from _gpu_util import cu_of, i32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("bits", [8, 6, 4])
def test_quant_pack_from_pinned_host_equals_device(kvq, cuda_dev, bits):
    H, D, ps, lens = 4, 256, 16, [37, 100]
    pt_np = kvgen.random_page_table(2, 2, 7)
    x = kvgen.KVSpec(seed=9, layer=0, is_key=True, n_seq=1, n_tok=sum(lens), num_heads=H,
                     head_dim=D).full_np()
    host = torch.from_numpy(x).pin_memory()
    view = kvq.HostView(host)
    pools = [kvq.Pool.empty(bits, H, D, ps, pt_np.size, cuda_dev) for _ in range(2)]
    for p in pools:
        p.codes.zero_()
        p.scales.zero_()
    pt, cu, st = i32(pt_np, cuda_dev), i32(cu_of(lens), cuda_dev), i32([0, 0], cuda_dev)
    kvq.kvq_quant_pack_paged([pools[0]], [host.to(cuda_dev)], pt, cu, st)
    kvq.kvq_quant_pack_paged([pools[1]], [view], pt, cu, st)
    torch.cuda.synchronize()
    assert torch.equal(pools[0].codes, pools[1].codes)
    assert torch.equal(pools[0].scales, pools[1].scales)


def test_pageable_host_memory_is_refused(kvq, cuda_dev):
    buf = np.zeros(1024, np.uint8)
    out = ctypes.c_void_p()
    assert kvq._lib.kvq_host_device_view(buf.ctypes.data, ctypes.byref(out)) == 5
    d = torch.zeros(16, device=cuda_dev)
    assert kvq._lib.kvq_host_device_view(d.data_ptr(), ctypes.byref(out)) == 0
    assert out.value == d.data_ptr()
