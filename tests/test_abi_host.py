"""C-ABI library (no GPU needed): it loads, exports every symbol include/kvq.h declares, and its
host logic (packed_dim, KIVI boundary, page allocator, argument validation) behaves as
specified.  No call here launches a kernel: every invalid argument is rejected on the host."""
import ctypes
import json
import os
import re
import subprocess

import numpy as np
import pytest

from conftest import ROOT, golden_path
from oracle import kivi as okivi
from oracle import symmetric as osym

HEADER = os.path.join(ROOT, "include", "kvq.h")


def _declared():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"KVQ_API[^;(]*?\b((?:kvq|kivi)_\w+)\s*\(", src)))


def test_library_exports_every_declared_symbol(kvq):
    names = _declared()
    assert len(names) >= 16
    lib = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", kvq.LIB_PATH], capture_output=True,
                         text=True).stdout
    exported = set(re.findall(r" T ((?:kvq|kivi)_\w+)", out))
    assert set(names) == exported


def test_version_and_status_strings(kvq):
    assert "sm_103a" in kvq.kvq_version()
    assert kvq._lib.kvq_status_string(6) == b"KVQ_ERR_CUDA"


def test_packed_dim_matches_oracle(kvq):
    for bits in (8, 6, 4):
        for d in range(1, 300):
            try:
                expect = osym.packed_dim(d, bits)
            except ValueError:
                expect = -1
            assert kvq.kvq_packed_dim(d, bits) == expect, (d, bits)
    for bits in (0, 2, 5, 7, 16):
        assert kvq.kvq_packed_dim(256, bits) == -1
    assert kvq.kvq_packed_dim(256, 6) == 192


def test_kivi_boundary_matches_golden_and_oracle(kvq):
    g = json.load(open(golden_path("kivi_groups.json")))["boundary"]
    for off, b in g["cases"]:
        assert kvq.kivi_boundary(off, g["residual_length"], g["group_size"]) == b
    for off in range(0, 700, 7):
        for R in (0, 1, 128):
            for gs in (1, 5, 32):
                assert kvq.kivi_boundary(off, R, gs) == okivi.quantization_boundary(off, R, gs)
    assert kvq.kivi_boundary(10, 0, 0) == -1 and kvq.kivi_boundary(10, -1, 4) == -1


def test_parse_mode_aliases(kvq):
    for m in ("q6", "6", "6bit", "int6", "uint6", 6, "Q6"):
        assert kvq.parse_mode(m) == 6
    assert kvq.parse_mode("q8") == 8 and kvq.parse_mode("q4") == 4
    for bad in ("q6_k", "q6_0", "q5", "fp16", ""):
        with pytest.raises(ValueError):
            kvq.parse_mode(bad)


def test_allocator(kvq):
    a = kvq.Allocator(10)
    assert a.free_count == 10
    ids = a.alloc(4)
    assert sorted(ids.tolist()) == [0, 1, 2, 3] and a.free_count == 6
    with pytest.raises(kvq.KVQError) as e:
        a.alloc(7)
    assert e.value.status == 7 and a.free_count == 6          # all or nothing
    with pytest.raises(kvq.KVQError):
        a.free(ids.new_tensor([1, 1]))                        # repeated id
    with pytest.raises(kvq.KVQError):
        a.free(ids.new_tensor([9]))                           # not allocated
    with pytest.raises(kvq.KVQError):
        a.free(ids.new_tensor([10]))                          # out of range
    assert a.free_count == 6
    a.free(ids[:2])
    assert a.free_count == 8
    with pytest.raises(kvq.KVQError):
        a.free(ids[:1])                                       # double free
    more = a.alloc(8)
    assert len(set(more.tolist()) | set(ids[2:].tolist())) == 10 and a.free_count == 0


def test_table_reserve_appends_into_partial_pages(kvq):
    import torch
    a = kvq.Allocator(100)
    pt = torch.full((3, 8), -1, dtype=torch.int32)
    a.reserve(pt, 16, [0, 0, 0], [16, 17, 0])
    assert (pt[0, :1] >= 0).all() and (pt[0, 1:] == -1).all()
    assert (pt[1, :2] >= 0).all() and (pt[1, 2:] == -1).all()
    assert (pt[2] == -1).all()
    before = pt.clone()
    a.reserve(pt, 16, [16, 17, 0], [1, 14, 0])          # seq 1 fills its partial page 1
    assert (pt[0, 1] >= 0) and torch.equal(pt[1], before[1])
    used = pt[pt >= 0]
    assert used.unique().numel() == used.numel() == 100 - a.free_count
    with pytest.raises(kvq.KVQError) as e:                  # beyond max_pages: unchanged
        a.reserve(pt, 16, [0, 0, 0], [0, 0, 16 * 9])
    assert e.value.status == 5
    snap, free = pt.clone(), a.free_count
    small = kvq.Allocator(1)
    with pytest.raises(kvq.KVQError) as e:
        small.reserve(pt, 16, [0, 0, 0], [0, 0, 40])        # needs 3, has 1
    assert e.value.status == 7 and torch.equal(pt, snap) and small.free_count == 1


# --------------------------------------------------------------------- host validation
FAKE = 0x10000  # aligned, never dereferenced: validation fails first


def _pool(kvq, bits=6, H=4, D=256, ps=16, pages=8, codes=FAKE, scales=FAKE):
    return kvq.kvq_pool(bits, H, D, ps, pages, codes, scales)


def _qp(kvq, pool, n=1, x=FAKE, total=16, nseq=1, max_pages=4, pt=FAKE, cu=FAKE, st=FAKE):
    pools = (kvq.kvq_pool * max(n, 1))(*([pool] * max(n, 1)))
    xs = (ctypes.c_void_p * max(n, 1))(*([x] * max(n, 1)))
    return kvq._lib.kvq_quant_pack_paged(pools, xs, n, pt, max_pages, cu, st, nseq, total, None,
                                         None)


def test_quant_pack_rejects_bad_arguments_before_launch(kvq):
    assert _qp(kvq, _pool(kvq, bits=5)) == 1
    assert _qp(kvq, _pool(kvq, bits=16)) == 1
    # head dims: exactly those kvq_packed_dim accepts, up to 256
    for bits in (8, 6, 4):
        for D in (0, 1, 2, 3, 4, 6, 10, 12, 20, 100, 252, 255, 256, 257, 264):
            want_ok = D <= 256 and kvq.kvq_packed_dim(D, bits) > 0
            got = _qp(kvq, _pool(kvq, bits=bits, D=D), total=0)
            assert (got == 0) == want_ok and (want_ok or got == 2), (bits, D, got)
    assert _qp(kvq, _pool(kvq, H=0)) == 2
    assert _qp(kvq, _pool(kvq, ps=0)) == 2
    assert _qp(kvq, _pool(kvq, codes=0)) == 3
    assert _qp(kvq, _pool(kvq, scales=FAKE + 2)) == 4
    assert _qp(kvq, _pool(kvq), x=FAKE + 8) == 4
    assert _qp(kvq, _pool(kvq), x=0) == 3
    assert _qp(kvq, _pool(kvq), n=0) == 5
    assert _qp(kvq, _pool(kvq), n=65) == 5
    assert _qp(kvq, _pool(kvq), total=-1) == 5
    assert _qp(kvq, _pool(kvq), max_pages=0) == 5
    assert _qp(kvq, _pool(kvq), pt=0) == 3
    assert b"KVQ_ERR_NULL" in kvq._lib.kvq_last_error()
    # mismatched pools in one call
    pools = (kvq.kvq_pool * 2)(_pool(kvq), _pool(kvq, bits=8))
    xs = (ctypes.c_void_p * 2)(FAKE, FAKE)
    assert kvq._lib.kvq_quant_pack_paged(pools, xs, 2, FAKE, 4, FAKE, FAKE, 1, 16, None,
                                         None) == 2


def test_dequant_rejects_bad_arguments_before_launch(kvq):
    pools = (kvq.kvq_pool * 1)(_pool(kvq, bits=3))
    xs = (ctypes.c_void_p * 1)(FAKE)
    assert kvq._lib.kvq_dequant_paged(pools, xs, 1, FAKE, 4, FAKE, FAKE, 1, 16, None, None) == 1


def test_kivi_rejects_bad_arguments_before_launch(kvq):
    xs = (ctypes.c_void_p * 2)(FAKE, FAKE)
    flags = (ctypes.c_int32 * 2)(1, 0)
    f = kvq._lib.kivi_quant_dequant
    assert f(xs, flags, 2, 1, 1, 64, 12, 0, 32, 32, 3, 1e-8, None) == 2     # D % 8
    assert f(xs, flags, 2, 1, 1, 64, 64, 40, 32, 32, 3, 1e-8, None) == 2    # lo > hi
    assert f(xs, flags, 2, 1, 1, 64, 64, 0, 65, 32, 3, 1e-8, None) == 2     # hi > S
    assert f(xs, flags, 2, 1, 1, 64, 64, 0, 32, 0, 3, 1e-8, None) == 2      # group 0
    assert f(xs, flags, 2, 1, 1, 64, 64, 0, 32, 32, 0, 1e-8, None) == 2     # levels 0
    assert f(xs, flags, 0, 1, 1, 64, 64, 0, 32, 32, 3, 1e-8, None) == 5
    bad = (ctypes.c_void_p * 2)(FAKE, FAKE + 4)
    assert f(bad, flags, 2, 1, 1, 64, 64, 0, 32, 32, 3, 1e-8, None) == 4
    assert f(xs, flags, 2, 1, 1, 64, 64, 16, 16, 32, 3, 1e-8, None) == 0    # empty: no launch


def test_decode_attn_rejects_bad_arguments_before_launch(kvq):
    f = kvq._lib.kvq_decode_attn
    P = lambda **kw: (kvq.kvq_pool * 1)(_pool(kvq, **kw))
    args = lambda kp, vp, hq=24, ws=1 << 30, maxlen=64: f(kp, vp, 1, FAKE, hq, FAKE, 4, FAKE, 1,
                                                         maxlen, 0.0625, FAKE, FAKE, ws, None,
                                                         None)
    assert args(P(D=128), P(D=128)) == 2            # head_dim 256 only
    assert args(P(), P(bits=8)) == 2                # K/V mismatch
    assert args(P(), P(), hq=18) == 2               # 18 % 4
    assert args(P(), P(), hq=36) == 2               # 9 query heads per KV head
    assert args(P(), P(), ws=16) == 8               # workspace too small
    assert args(P(), P(), maxlen=65) == 5           # beyond max_pages * page_size
    assert args(P(bits=7), P(bits=7)) == 1
    need = kvq.kvq_decode_attn_workspace(16, 1, 4, 24, 256, 16, 262144)
    assert need > 0 and need % 16 == 0


def _kp(kvq, bits=2, gs=32, B=1, H=2, S=128, D=64, ptr=FAKE):
    return kvq.kivi_packed(bits, gs, B, H, S, D, ptr, ptr, ptr, ptr, ptr, ptr)


def test_kivi_packed_rejects_bad_arguments_before_launch(kvq):
    C = lambda **kw: (kvq.kivi_packed * 1)(_kp(kvq, **kw))
    xs = (ctypes.c_void_p * 1)(FAKE)
    pack = lambda c, lo=0, hi=64, eps=1e-8, k=xs: kvq._lib.kivi_pack(c, k, xs, 1, lo, hi, eps, None)
    assert pack(C(bits=3)) == 1
    assert pack(C(gs=24)) == 2                      # group size not in {8, 16, 32, 64}
    assert pack(C(D=72)) == 2                       # head_dim % group_size
    assert pack(C(S=100)) == 5                      # capacity % group_size
    assert pack(C(ptr=FAKE + 2)) == 4
    assert pack(C(ptr=0)) == 3
    assert pack(C(), lo=16) == 2                    # lo not on a group boundary
    assert pack(C(), hi=160) == 2                   # beyond capacity
    assert pack(C(), eps=-1.0) == 5
    assert pack(C(), k=(ctypes.c_void_p * 1)(FAKE + 8)) == 4
    assert pack(C(), lo=64, hi=64) == 0             # empty: no launch
    two = (kvq.kivi_packed * 2)(_kp(kvq), _kp(kvq, H=3))
    assert kvq._lib.kivi_pack(two, (ctypes.c_void_p * 2)(FAKE, FAKE),
                              (ctypes.c_void_p * 2)(FAKE, FAKE), 2, 0, 64, 1e-8, None) == 2

    attn = lambda c, hq=8, n_packed=64, offset=100, ws=1 << 30: kvq._lib.kivi_decode_attn(
        c, xs, xs, 1, FAKE, hq, n_packed, offset, 0.125, FAKE, FAKE, ws, None, None)
    assert attn(C(bits=4)) == 2                     # the attention kernel reads 2-bit codes
    assert attn(C(D=128)) == 2                      # head_dim 64
    assert attn(C(gs=8)) == 2                       # group size a multiple of the 16-token tile
    assert attn(C(), hq=7) == 2                     # not a multiple of the 2 KV heads
    assert attn(C(), hq=18) == 2                    # 9 query heads per KV head
    assert attn(C(), n_packed=48) == 5              # not a whole group
    assert attn(C(), offset=60) == 5                # offset < n_packed
    assert attn(C(), offset=129) == 5               # beyond capacity
    assert attn(C(), ws=16) == 8
    assert kvq.kivi_decode_attn_workspace(1, 1, 2, 8, 64, 100) > 0


def test_append_decode_rejects_bad_arguments_before_launch(kvq):
    f = kvq._lib.kvq_append_decode_attn
    P = lambda **kw: (kvq.kvq_pool * 1)(_pool(kvq, **kw))
    xs = (ctypes.c_void_p * 1)(FAKE)
    call = lambda kp, vp, kn=xs, vn=xs, ws=1 << 30: f(kp, vp, 1, kn, vn, FAKE, 24, FAKE, 4, FAKE,
                                                     1, 64, 0.0625, FAKE, FAKE, ws, None, None)
    assert call(P(ps=8), P(ps=8)) == 2              # page size not a multiple of 16
    assert call(P(), P(), kn=None) == 3
    assert call(P(), P(), vn=(ctypes.c_void_p * 1)(0)) == 3
    assert call(P(), P(), kn=(ctypes.c_void_p * 1)(FAKE + 2)) == 4
    assert call(P(), P(), ws=16) == 8
    assert call(P(D=128), P(D=128)) == 2


def test_kivi_state_and_trim_follow_the_page_rollback(kvq):
    """kivi_trim is host arithmetic: offsets and frontiers follow the oracle's cache (the page's
    trim with _rollback_frontier) over a seeded sequence of appends and trims."""
    from oracle import kivi as K
    with pytest.raises(kvq.KVQError):
        kvq.kivi_state_new(1, 1, 12, 64)              # head_dim % 8
    with pytest.raises(kvq.KVQError):
        kvq.kivi_state_new(1, 1, 64, 64, bits=3)
    rng = np.random.default_rng(5)
    st = kvq.kivi_state_new(1, 1, 64, 4096, bits=2, group_size=32, residual_length=128)
    ref = K.KiviCache(1, 1, 8, 4096, bit_width=2, group_size=32, residual_length=128)
    for _ in range(300):
        if rng.random() < 0.7:
            n = int(rng.integers(1, 90))
            if ref.offset + n > 4096:
                continue
            ref.offset += n                            # the state part of update_and_fetch
            b = K.quantization_boundary(ref.offset, 128, 32)
            ref.n_quantized = max(ref.n_quantized, b)
            st.offset, st.n_quantized = ref.offset, ref.n_quantized
        else:
            n = int(rng.integers(0, 200))
            assert kvq.kivi_trim(st, n) == ref.trim(n)
            assert (st.offset, st.n_quantized) == (ref.offset, ref.n_quantized)


def test_kivi_protocol_rejects_bad_arguments_before_launch(kvq):
    st = kvq.kivi_state_new(1, 2, 64, 128, bits=2, group_size=32, residual_length=16)
    xs = (ctypes.c_void_p * 1)(FAKE)
    sp = ctypes.byref(st)
    f = kvq._lib.kivi_update
    assert f(sp, xs, xs, xs, xs, 1, 129, None) == 5                 # does not fit
    assert f(sp, xs, xs, None, xs, 1, 4, None) == 3
    assert f(sp, xs, (ctypes.c_void_p * 1)(FAKE + 2), xs, xs, 1, 4, None) == 4
    assert f(sp, xs, xs, xs, xs, 33, 4, None) == 5                  # at most 32 layers
    assert f(sp, xs, xs, xs, xs, 1, 0, None) == 0                   # nothing to do
    assert (st.offset, st.n_quantized) == (0, 0)
    C = (kvq.kivi_packed * 1)(kvq.kivi_packed(2, 32, 1, 2, 128, 64, FAKE, FAKE, FAKE, FAKE,
                                              FAKE, FAKE))
    bad = (kvq.kivi_packed * 1)(kvq.kivi_packed(2, 32, 1, 2, 256, 64, FAKE, FAKE, FAKE, FAKE,
                                                FAKE, FAKE))
    g = kvq._lib.kivi_packed_update
    assert g(sp, bad, xs, xs, xs, xs, 1, 4, None) == 2              # capacity differs
    assert g(sp, C, xs, xs, xs, xs, 1, 200, None) == 5
    out = ctypes.c_int(-1)
    assert kvq._lib.kivi_packed_trim(sp, C, xs, xs, 1, 5, ctypes.byref(out), None) == 0
    assert out.value == 0                                           # empty cache: nothing cut
    u = kvq._lib.kivi_unpack
    assert u(C, xs, xs, 1, 0, 129, None) == 2
    assert u(C, xs, xs, 1, 10, 5, None) == 2
    assert u(C, xs, xs, 1, 7, 7, None) == 0                         # empty: no launch


def _side(kvq, k=3, ns=4, max_seqs=1, val=FAKE, idx=FAKE, sink=FAKE):
    return kvq.kvq_side(k, ns, max_seqs, val, idx, sink)


def test_side_rejects_bad_arguments_before_launch(kvq):
    pools = (kvq.kvq_pool * 1)(_pool(kvq))
    xs = (ctypes.c_void_p * 1)(FAKE)
    S = lambda **kw: (kvq.kvq_side * 1)(_side(kvq, **kw))
    qp = lambda sd, nseq=1: kvq._lib.kvq_quant_pack_paged_side(pools, sd, xs, 1, FAKE, 4, FAKE,
                                                               FAKE, nseq, 16, None, None)
    dq = lambda sd: kvq._lib.kvq_dequant_paged_side(pools, sd, xs, 1, FAKE, 4, FAKE, FAKE, 1, 16,
                                                    None, None)
    assert qp(None) == 3                            # no side array
    assert qp(S(k=9)) == 5                          # more than KVQ_MAX_OUTLIERS
    assert qp(S(k=-1)) == 5
    assert qp(S(ns=17)) == 5                        # more than KVQ_MAX_SINKS
    assert qp(S(val=0)) == 3                        # outliers without value / position arrays
    assert qp(S(idx=0)) == 3
    assert qp(S(sink=0)) == 3                       # sinks without a buffer
    assert qp(S(val=FAKE + 2)) == 4
    assert qp(S(), nseq=2) == 5                     # the sink buffer holds one sequence
    assert dq(S(k=9)) == 5
    assert dq(S(idx=FAKE + 8)) == 4
    two = (kvq.kvq_pool * 2)(_pool(kvq), _pool(kvq))
    mixed = (kvq.kvq_side * 2)(_side(kvq, k=3), _side(kvq, k=2))
    assert kvq._lib.kvq_quant_pack_paged_side(two, mixed, (ctypes.c_void_p * 2)(FAKE, FAKE), 2,
                                              FAKE, 4, FAKE, FAKE, 1, 16, None, None) == 2

    P = lambda **kw: (kvq.kvq_pool * 1)(_pool(kvq, **kw))
    attn = lambda kp, vp, ks, vs, ws=1 << 30: kvq._lib.kvq_decode_attn_side(
        kp, vp, ks, vs, 1, FAKE, 24, FAKE, 4, FAKE, 1, 64, 0.0625, FAKE, FAKE, ws, None, None)
    assert attn(P(ps=8), P(ps=8), S(), S()) == 2    # the staged kernel needs pages of 16k
    assert attn(P(), P(), S(k=9), S(k=9)) == 5
    assert attn(P(), P(), S(), S(sink=0)) == 3
    assert attn(P(), P(), S(), S(), ws=16) == 8
