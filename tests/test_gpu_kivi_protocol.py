"""GPU parity for the KIVI cache protocol (update_and_fetch, trim with frontier rollback) in
both storage forms, step by step against the oracle's caches: the page's in-place fp16 cache
(oracle.kivi.KiviCache) and the packed form (oracle.kivi_packed.KiviPackedCache).  States are
compared exactly, cache contents bit for bit, and attention over the packed state within
|gpu - ref| <= 2e-3 + 1e-3 * |ref|."""
import numpy as np
import pytest
import torch

import kvgen
from oracle import kivi as K
from oracle import kivi_packed as P
from _attn_checks import assert_attn_close
from _gpu_util import dev_tensor, u16

pytestmark = pytest.mark.gpu

# (op, n): appends of various sizes (single tokens, chunks straddling group boundaries, a long
# prefill) and trims that cut inside a group, at a group edge and below the frontier
SCRIPT = [("u", 1), ("u", 5), ("u", 70), ("u", 31), ("u", 64), ("u", 1), ("u", 1), ("u", 128),
          ("t", 150), ("u", 40), ("t", 30), ("u", 200), ("t", 1), ("u", 17), ("t", 64),
          ("u", 96)]


class _Tokens:
    """A stream of new tokens [B, H, n, D] per layer, K and V, from the generator."""

    def __init__(self, L, B, H, D, total=2048, seed=21):
        self.k = [kvgen.KiviSpec(seed=seed, layer=l, is_key=True, batch=B, num_heads=H,
                                 seq=total, head_dim=D).full_np() for l in range(L)]
        self.v = [kvgen.KiviSpec(seed=seed, layer=l, is_key=False, batch=B, num_heads=H,
                                 seq=total, head_dim=D).full_np() for l in range(L)]
        self.t = 0

    def take(self, n):
        out = ([np.ascontiguousarray(x[:, :, self.t:self.t + n]) for x in self.k],
               [np.ascontiguousarray(x[:, :, self.t:self.t + n]) for x in self.v])
        self.t += n
        return out


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_in_place_protocol(kvq, cuda_dev, bits):
    L, B, H, D, S, gs, R = 2, 2, 3, 64, 1024, 32, 128
    st = kvq.kivi_state_new(B, H, D, S, bits=bits, group_size=gs, residual_length=R)
    kc = [torch.zeros((B, H, S, D), dtype=torch.float16, device=cuda_dev) for _ in range(L)]
    vc = [torch.zeros_like(kc[0]) for _ in range(L)]
    ref = [K.KiviCache(B, H, D, S, bit_width=bits, group_size=gs, residual_length=R)
           for _ in range(L)]
    toks = _Tokens(L, B, H, D)
    for op, n in SCRIPT:
        if op == "u":
            kn, vn = toks.take(n)
            kvq.kivi_update(st, kc, vc, [dev_tensor(x, cuda_dev) for x in kn],
                            [dev_tensor(x, cuda_dev) for x in vn])
            for l in range(L):
                ref[l].update_and_fetch(kn[l], vn[l])
        else:
            got = kvq.kivi_trim(st, n)
            for l in range(L):
                assert ref[l].trim(n) == got
        torch.cuda.synchronize()
        assert (st.offset, st.n_quantized) == (ref[0].offset, ref[0].n_quantized)
        off = st.offset
        for l in range(L):
            assert np.array_equal(u16(kc[l][:, :, :off]), ref[l].keys[:, :, :off].view(np.uint16))
            assert np.array_equal(u16(vc[l][:, :, :off]), ref[l].values[:, :, :off].view(np.uint16))


@pytest.mark.parametrize("bits,gs", [(2, 32), (2, 16), (4, 32), (8, 64)])
def test_packed_protocol_and_attention(kvq, cuda_dev, bits, gs):
    L, B, H, G, D, S, R = 2, 2, 2, 4, 64, 1024, 128
    st = kvq.kivi_state_new(B, H, D, S, bits=bits, group_size=gs, residual_length=R)
    kc = [torch.zeros((B, H, S, D), dtype=torch.float16, device=cuda_dev) for _ in range(L)]
    vc = [torch.zeros_like(kc[0]) for _ in range(L)]
    caches = [kvq.KiviPacked.empty(bits, gs, B, H, S, D, cuda_dev) for _ in range(L)]
    ref = [P.KiviPackedCache(B, H, D, S, bit_width=bits, group_size=gs, residual_length=R)
           for _ in range(L)]
    toks = _Tokens(L, B, H, D, seed=22)
    err = torch.zeros(1, dtype=torch.int32, device=cuda_dev)
    for step, (op, n) in enumerate(SCRIPT):
        if op == "u":
            kn, vn = toks.take(n)
            kvq.kivi_packed_update(st, caches, kc, vc, [dev_tensor(x, cuda_dev) for x in kn],
                                   [dev_tensor(x, cuda_dev) for x in vn])
            for l in range(L):
                ref[l].update(kn[l], vn[l])
        else:
            got = kvq.kivi_packed_trim(st, caches, kc, vc, n)
            for l in range(L):
                assert ref[l].trim(n) == got
        torch.cuda.synchronize()
        nq, off = st.n_quantized, st.offset
        assert (off, nq) == (ref[0].offset, ref[0].n_quantized)
        for l in range(L):
            c, r = caches[l], ref[l]
            assert np.array_equal(c.k_codes[:, :, :nq].cpu().numpy(), r.k_codes[:, :, :nq])
            assert np.array_equal(u16(c.k_scale[:, :, :nq // gs]), r.k_scale[:, :, :nq // gs].view(np.uint16))
            assert np.array_equal(u16(c.k_zero[:, :, :nq // gs]), r.k_zero[:, :, :nq // gs].view(np.uint16))
            assert np.array_equal(c.v_codes[:, :, :nq].cpu().numpy(), r.v_codes[:, :, :nq])
            assert np.array_equal(u16(c.v_scale[:, :, :nq]), r.v_scale[:, :, :nq].view(np.uint16))
            assert np.array_equal(u16(c.v_zero[:, :, :nq]), r.v_zero[:, :, :nq].view(np.uint16))
            assert np.array_equal(u16(kc[l][:, :, nq:off]), r.keys[:, :, nq:off].view(np.uint16))
            assert np.array_equal(u16(vc[l][:, :, nq:off]), r.values[:, :, nq:off].view(np.uint16))
        if bits == 2 and off > 0:   # attention over the packed state
            q = kvgen.queries_np(300 + step, L, B, H * G, D)
            out = torch.full(q.shape, float("nan"), dtype=torch.float32, device=cuda_dev)
            ws = torch.empty(max(16, kvq.kivi_decode_attn_workspace(L, B, H, H * G, D, off)),
                             dtype=torch.uint8, device=cuda_dev)
            kvq.kivi_decode_attn(caches, kc, vc, dev_tensor(q, cuda_dev), nq, off, 0.125, out, ws,
                                 err)
            torch.cuda.synchronize()
            assert int(err.item()) == 0
            got = out.cpu().numpy().astype(np.float64)
            for l in range(L):
                r = ref[l]
                kp = (r.k_codes[:, :, :nq], r.k_scale[:, :, :nq // gs], r.k_zero[:, :, :nq // gs])
                vp = (r.v_codes[:, :, :nq], r.v_scale[:, :, :nq], r.v_zero[:, :, :nq])
                want = P.decode_attention(q[l], kp, vp, r.keys[:, :, nq:off], r.values[:, :, nq:off],
                                          2, gs, 0.125)
                assert_attn_close(got[l], want, f"layer {l}")


def test_unpack_reconstructs_the_oracle_rows(kvq, cuda_dev):
    """kivi_unpack of a whole packed cache equals the oracle's unpack bit for bit (2/4/8 bits,
    group 8 to 64)."""
    B, H, S, D = 2, 3, 128, 64
    for bits, gs in ((2, 8), (4, 16), (8, 64), (2, 32)):
        k = kvgen.KiviSpec(seed=31, layer=0, is_key=True, batch=B, num_heads=H, seq=S,
                           head_dim=D).full_np()
        v = kvgen.KiviSpec(seed=31, layer=0, is_key=False, batch=B, num_heads=H, seq=S,
                           head_dim=D).full_np()
        c = kvq.KiviPacked.empty(bits, gs, B, H, S, D, cuda_dev)
        kvq.kivi_pack([c], [dev_tensor(k, cuda_dev)], [dev_tensor(v, cuda_dev)], 0, S)
        ko = torch.zeros((B, H, S, D), dtype=torch.float16, device=cuda_dev)
        vo = torch.zeros_like(ko)
        kvq.kivi_unpack([c], [ko], [vo], 16, 100)
        torch.cuda.synchronize()
        want_k = P.unpack_keys(*P.pack_keys(k, bits, gs), bits, gs, D)
        want_v = P.unpack_values(*P.pack_values(v, bits, gs), bits, gs, D)
        assert np.array_equal(u16(ko[:, :, 16:100]), want_k[:, :, 16:100].view(np.uint16))
        assert np.array_equal(u16(vo[:, :, 16:100]), want_v[:, :, 16:100].view(np.uint16))
        assert int(ko[:, :, :16].abs().sum()) == 0 and int(vo[:, :, 100:].abs().sum()) == 0
