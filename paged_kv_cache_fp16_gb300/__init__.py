"""Python binding of libkvq (quantized paged KV cache kernels for GB300, sm_103a).

Argument marshalling only: every step of the hot path runs in the CUDA library's kernels.  The
functions carry the C ABI's names (``include/kvq.h``) and take torch tensors for device memory;
they enqueue work on the current torch stream (or the one given) and never synchronize.

There is no fallback: if ``libkvq.so`` cannot be loaded, importing this package raises.
Build it with ``python -c "import __graft_entry__ as g; g.build()"`` or
``python paged_kv_cache_fp16_gb300/build.py``.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkvq.so")

KVQ_MAX_TENSORS = 64
KVQ_DEVERR_PAGE_RANGE = 1
KVQ_DEVERR_TIMEOUT = 2
STATUS = {0: "KVQ_OK", 1: "KVQ_ERR_BITS", 2: "KVQ_ERR_SHAPE", 3: "KVQ_ERR_NULL",
          4: "KVQ_ERR_ALIGN", 5: "KVQ_ERR_RANGE", 6: "KVQ_ERR_CUDA", 7: "KVQ_ERR_NOMEM",
          8: "KVQ_ERR_WORKSPACE"}


class KVQError(RuntimeError):
    """A libkvq entry point returned a non-OK status."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


class kvq_pool(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int64), ("codes", ctypes.c_void_p),
                ("scales", ctypes.c_void_p)]


class kivi_packed(ctypes.Structure):
    _fields_ = [("bits", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("k_codes", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("k_zero", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("v_zero", ctypes.c_void_p)]


class kvq_side(ctypes.Structure):
    _fields_ = [("n_outlier", ctypes.c_int32), ("n_sink", ctypes.c_int32),
                ("max_seqs", ctypes.c_int32), ("out_val", ctypes.c_void_p),
                ("out_idx", ctypes.c_void_p), ("sink", ctypes.c_void_p)]


class kivi_state(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("bits", ctypes.c_int32), ("group_size", ctypes.c_int32),
                ("residual_length", ctypes.c_int32), ("eps", ctypes.c_float),
                ("offset", ctypes.c_int32), ("n_quantized", ctypes.c_int32)]


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libkvq.so is not built ({LIB_PATH} missing); run paged_kv_cache_fp16_gb300/build.py")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, F, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
    pool_p = ctypes.POINTER(kvq_pool)
    sig = {
        "kvq_version": (ctypes.c_char_p, []),
        "kvq_last_error": (ctypes.c_char_p, []),
        "kvq_status_string": (ctypes.c_char_p, [I]),
        "kvq_packed_dim": (I, [I, I]),
        "kivi_boundary": (I, [I, I, I]),
        "kvq_alloc_create": (P, [I64]),
        "kvq_alloc_destroy": (None, [P]),
        "kvq_alloc_free_count": (I64, [P]),
        "kvq_alloc_pages": (I, [P, I64, P]),
        "kvq_free_pages": (I, [P, I64, P]),
        "kvq_table_reserve": (I, [P, P, I, I, P, P, I]),
        "kvq_quant_pack_paged": (I, [pool_p, P, I, P, I, P, P, I, I, P, P]),
        "kvq_dequant_paged": (I, [pool_p, P, I, P, I, P, P, I, I, P, P]),
        "kivi_quant_dequant": (I, [P, P, I, I, I, I, I, I, I, I, I, F, P]),
        "kvq_decode_attn_workspace": (S, [I, I, I, I, I, I, I]),
        "kvq_decode_attn": (I, [pool_p, pool_p, I, P, I, P, I, P, I, I, F, P, P, S, P, P]),
        "kvq_decode_attn_noalloc": (I, [pool_p, pool_p, I, P, I, P, I, P, I, I, F, P, P, P]),
        "kvq_append_decode_attn": (I, [pool_p, pool_p, I, P, P, P, I, P, I, P, I, I, F, P, P, S,
                                       P, P]),
        "kivi_pack": (I, [ctypes.POINTER(kivi_packed), P, P, I, I, I, F, P]),
        "kvq_quant_pack_paged_side": (I, [pool_p, ctypes.POINTER(kvq_side), P, I, P, I, P, P,
                                          I, I, P, P]),
        "kvq_decode_attn_side": (I, [pool_p, pool_p, ctypes.POINTER(kvq_side),
                                     ctypes.POINTER(kvq_side), I, P, I, P, I, P, I, I, F, P, P, S,
                                     P, P]),
        "kvq_dequant_paged_side": (I, [pool_p, ctypes.POINTER(kvq_side), P, I, P, I, P, P, I, I,
                                       P, P]),
        "kvq_host_device_view": (I, [P, ctypes.POINTER(ctypes.c_void_p)]),
        "kivi_state_init": (I, [ctypes.POINTER(kivi_state), I, I, I, I, I, I, I]),
        "kivi_update": (I, [ctypes.POINTER(kivi_state), P, P, P, P, I, I, P]),
        "kivi_trim": (I, [ctypes.POINTER(kivi_state), I]),
        "kivi_packed_update": (I, [ctypes.POINTER(kivi_state), ctypes.POINTER(kivi_packed), P, P,
                                   P, P, I, I, P]),
        "kivi_packed_trim": (I, [ctypes.POINTER(kivi_state), ctypes.POINTER(kivi_packed), P, P,
                                 I, I, ctypes.POINTER(ctypes.c_int), P]),
        "kivi_unpack": (I, [ctypes.POINTER(kivi_packed), P, P, I, I, I, P]),
        "kivi_decode_attn_workspace": (S, [I, I, I, I, I, I]),
        "kivi_decode_attn": (I, [ctypes.POINTER(kivi_packed), P, P, I, P, I, I, I, F, P, P, S,
                                 P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = _load()


def _check(status: int) -> None:
    if status != 0:
        raise KVQError(status, _lib.kvq_last_error().decode())


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        if torch.cuda.is_available():
            return torch.cuda.current_stream().cuda_stream
        return None
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr_array(tensors: Sequence[torch.Tensor]):
    arr = (ctypes.c_void_p * len(tensors))()
    for i, t in enumerate(tensors):
        arr[i] = t.data_ptr()
    return arr


def _cuda_tensor(t, dtype, name: str):
    if isinstance(t, HostView):   # page-locked host memory read in place by the kernel
        if t.dtype != dtype:
            raise TypeError(f"{name} must be {dtype}")
        return t
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# ------------------------------------------------------------------------------- host helpers
def kvq_version() -> str:
    return _lib.kvq_version().decode()


def kvq_packed_dim(head_dim: int, bits: int) -> int:
    return _lib.kvq_packed_dim(head_dim, bits)


def kivi_boundary(offset: int, residual_length: int = 128, group_size: int = 32) -> int:
    return _lib.kivi_boundary(offset, residual_length, group_size)


_MODES = {"q8": 8, "8": 8, "int8": 8, "q6": 6, "6": 6, "6bit": 6, "int6": 6, "uint6": 6,
          "q4": 4, "4": 4, "int4": 4}


def parse_mode(mode) -> int:
    """Quantization width from a mode name.  q6 aliases stay narrow (q6, 6, 6bit, int6, uint6);
    llama.cpp-style names such as q6_k or q6_0 are a different format and are rejected
    (MTPLX pull request #267, description, aliases paragraph)."""
    key = str(mode).strip().lower()
    if key not in _MODES:
        raise ValueError(f"unknown KV quantization mode {mode!r}")
    return _MODES[key]


@dataclass
class Pool:
    """Packed storage of one (layer, K-or-V) tensor: codes [num_pages, H, page_size, pd] uint8 and
    scales [num_pages, H, page_size] fp16."""
    bits: int
    num_heads: int
    head_dim: int
    page_size: int
    codes: torch.Tensor
    scales: torch.Tensor

    @staticmethod
    def empty(bits, num_heads, head_dim, page_size, num_pages, device="cuda"):
        pd = kvq_packed_dim(head_dim, bits)
        if pd < 0:
            raise ValueError("unsupported bits / head_dim")
        codes = torch.empty((num_pages, num_heads, page_size, pd), dtype=torch.uint8,
                            device=device)
        scales = torch.empty((num_pages, num_heads, page_size), dtype=torch.float16,
                             device=device)
        return Pool(bits, num_heads, head_dim, page_size, codes, scales)

    @property
    def num_pages(self) -> int:
        return self.codes.shape[0]

    def as_c(self) -> kvq_pool:
        return kvq_pool(self.bits, self.num_heads, self.head_dim, self.page_size,
                        self.num_pages, self.codes.data_ptr(), self.scales.data_ptr())


def _pool_array(pools: Sequence[Pool]):
    arr = (kvq_pool * len(pools))()
    for i, p in enumerate(pools):
        arr[i] = p.as_c()
    return arr


class Allocator:
    """Host page allocator (kvq_alloc_*): hands out page ids of a pool."""

    def __init__(self, num_pages: int):
        self._h = _lib.kvq_alloc_create(num_pages)
        if not self._h:
            raise ValueError("kvq_alloc_create failed")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _lib.kvq_alloc_destroy(h)
            self._h = None

    @property
    def free_count(self) -> int:
        return _lib.kvq_alloc_free_count(self._h)

    def alloc(self, n: int) -> torch.Tensor:
        out = torch.empty(n, dtype=torch.int32)
        _check(_lib.kvq_alloc_pages(self._h, n, out.data_ptr()))
        return out

    def free(self, ids: torch.Tensor) -> None:
        ids = ids.to(torch.int32).contiguous().cpu()
        _check(_lib.kvq_free_pages(self._h, ids.numel(), ids.data_ptr()))

    def reserve(self, page_table: torch.Tensor, page_size: int, cur_len, new_tokens) -> None:
        """Map pages for appends into a host int32 table [nseq, max_pages] (-1 = unmapped)."""
        if page_table.is_cuda or page_table.dtype != torch.int32 or not page_table.is_contiguous():
            raise TypeError("page_table must be a contiguous host int32 tensor")
        cur = torch.as_tensor(cur_len, dtype=torch.int32).contiguous()
        new = torch.as_tensor(new_tokens, dtype=torch.int32).contiguous()
        nseq, max_pages = page_table.shape
        _check(_lib.kvq_table_reserve(self._h, page_table.data_ptr(), max_pages, page_size,
                                      cur.data_ptr(), new.data_ptr(), nseq))


# ------------------------------------------------------------------------------- kernels
def _check_table(page_table: torch.Tensor, nseq: int, n_cu: int) -> None:
    if page_table.dim() != 2 or page_table.shape[0] < nseq:
        raise ValueError("page_table must be [nseq, max_pages] with a row per sequence")
    if n_cu != nseq + 1:
        raise ValueError("cu tensor must have nseq + 1 entries")


def kvq_quant_pack_paged(pools: Sequence[Pool], xs: Sequence[torch.Tensor],
                         page_table: torch.Tensor, cu_new_tokens: torch.Tensor,
                         start_pos: torch.Tensor, dev_err: torch.Tensor | None = None,
                         stream=None) -> None:
    """Quantize + pack new rows xs[i] (fp16 [total, H, D]) into pools[i] through page_table."""
    if len(pools) != len(xs):
        raise ValueError("one input tensor per pool")
    for i, x in enumerate(xs):
        _cuda_tensor(x, torch.float16, f"xs[{i}]")
    _cuda_tensor(page_table, torch.int32, "page_table")
    _cuda_tensor(cu_new_tokens, torch.int32, "cu_new_tokens")
    _cuda_tensor(start_pos, torch.int32, "start_pos")
    total = xs[0].shape[0] if xs else 0
    _check_table(page_table, start_pos.numel(), cu_new_tokens.numel())
    _check(_lib.kvq_quant_pack_paged(_pool_array(pools), _ptr_array(xs), len(xs),
                                     page_table.data_ptr(), page_table.shape[1],
                                     cu_new_tokens.data_ptr(), start_pos.data_ptr(),
                                     start_pos.numel(), total, _ptr(dev_err), _stream(stream)))


def kvq_dequant_paged(pools: Sequence[Pool], outs: Sequence[torch.Tensor],
                      page_table: torch.Tensor, cu_tokens: torch.Tensor, start_pos: torch.Tensor,
                      dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Gather + dequantize rows of pools[i] into outs[i] (fp16 [total, H, D])."""
    if len(pools) != len(outs):
        raise ValueError("one output tensor per pool")
    for i, o in enumerate(outs):
        _cuda_tensor(o, torch.float16, f"outs[{i}]")
    _cuda_tensor(page_table, torch.int32, "page_table")
    _cuda_tensor(cu_tokens, torch.int32, "cu_tokens")
    _cuda_tensor(start_pos, torch.int32, "start_pos")
    total = outs[0].shape[0] if outs else 0
    _check_table(page_table, start_pos.numel(), cu_tokens.numel())
    _check(_lib.kvq_dequant_paged(_pool_array(pools), _ptr_array(outs), len(outs),
                                  page_table.data_ptr(), page_table.shape[1],
                                  cu_tokens.data_ptr(), start_pos.data_ptr(), start_pos.numel(),
                                  total, _ptr(dev_err), _stream(stream)))


def kivi_quant_dequant(xs: Sequence[torch.Tensor], is_key: Sequence[bool], lo: int, hi: int,
                       group_size: int = 32, levels: int = 3, eps: float = 1e-8,
                       stream=None) -> None:
    """In-place KIVI round trip of tokens [lo, hi) of every fp16 [B, H, S, D] tensor."""
    if len(xs) != len(is_key):
        raise ValueError("one is_key flag per tensor")
    for i, x in enumerate(xs):
        _cuda_tensor(x, torch.float16, f"xs[{i}]")
        if x.dim() != 4 or x.shape != xs[0].shape:
            raise ValueError("all tensors must be [B, H, S, D] of one shape")
    B, H, S, D = xs[0].shape
    flags = (ctypes.c_int32 * len(xs))(*[1 if k else 0 for k in is_key])
    _check(_lib.kivi_quant_dequant(_ptr_array(xs), flags, len(xs), B, H, S, D, lo, hi,
                                   group_size, levels, eps, _stream(stream)))


def kvq_decode_attn_workspace(n_layers: int, nseq: int, num_kv_heads: int, num_q_heads: int,
                              head_dim: int, page_size: int, max_seq_len: int) -> int:
    return _lib.kvq_decode_attn_workspace(n_layers, nseq, num_kv_heads, num_q_heads, head_dim,
                                          page_size, max_seq_len)


def kvq_decode_attn(k_pools: Sequence[Pool], v_pools: Sequence[Pool], q: torch.Tensor,
                    page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                    softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                    dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Decode attention over packed pages: q fp16 [n_layers, nseq, Hq, D] -> out float32."""
    if len(k_pools) != len(v_pools):
        raise ValueError("one V pool per K pool")
    _cuda_tensor(q, torch.float16, "q")
    _cuda_tensor(out, torch.float32, "out")
    _cuda_tensor(page_table, torch.int32, "page_table")
    _cuda_tensor(seq_lens, torch.int32, "seq_lens")
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    n_layers, nseq, hq, _ = q.shape
    if page_table.dim() != 2 or page_table.shape[0] < nseq or seq_lens.numel() < nseq:
        raise ValueError("page_table needs a row and seq_lens an entry per sequence")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    _check(_lib.kvq_decode_attn(_pool_array(k_pools), _pool_array(v_pools), n_layers,
                                q.data_ptr(), hq, page_table.data_ptr(), page_table.shape[1],
                                seq_lens.data_ptr(), nseq, max_seq_len, softmax_scale,
                                out.data_ptr(), workspace.data_ptr(),
                                workspace.numel() * workspace.element_size(), _ptr(dev_err),
                                _stream(stream)))


def kvq_append_decode_attn(k_pools: Sequence[Pool], v_pools: Sequence[Pool],
                           k_new: Sequence[torch.Tensor], v_new: Sequence[torch.Tensor],
                           q: torch.Tensor, page_table: torch.Tensor, seq_lens: torch.Tensor,
                           max_seq_len: int, softmax_scale: float, out: torch.Tensor,
                           workspace: torch.Tensor, dev_err: torch.Tensor | None = None,
                           stream=None) -> None:
    """One decode step: write each sequence's new token (k_new[l], v_new[l] fp16 [nseq, H, D])
    at position seq_lens[s] of the pools, then attend over seq_lens[s] + 1 tokens.  seq_lens is
    not advanced; max_seq_len bounds seq_lens + 1."""
    if not (len(k_pools) == len(v_pools) == len(k_new) == len(v_new)):
        raise ValueError("one V pool and one new K/V tensor per K pool")
    _cuda_tensor(q, torch.float16, "q")
    _cuda_tensor(out, torch.float32, "out")
    _cuda_tensor(page_table, torch.int32, "page_table")
    _cuda_tensor(seq_lens, torch.int32, "seq_lens")
    n_layers, nseq, hq, D = q.shape
    for i, (k, v) in enumerate(zip(k_new, v_new)):
        _cuda_tensor(k, torch.float16, f"k_new[{i}]")
        _cuda_tensor(v, torch.float16, f"v_new[{i}]")
        if k.numel() < nseq * k_pools[i].num_heads * D or v.numel() != k.numel():
            raise ValueError("k_new/v_new need [nseq, H, D] rows")
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise TypeError("workspace must be a contiguous CUDA tensor")
    if page_table.dim() != 2 or page_table.shape[0] < nseq or seq_lens.numel() < nseq:
        raise ValueError("page_table needs a row and seq_lens an entry per sequence")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    _check(_lib.kvq_append_decode_attn(_pool_array(k_pools), _pool_array(v_pools), n_layers,
                                       _ptr_array(k_new), _ptr_array(v_new), q.data_ptr(), hq,
                                       page_table.data_ptr(), page_table.shape[1],
                                       seq_lens.data_ptr(), nseq, max_seq_len, softmax_scale,
                                       out.data_ptr(), workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(),
                                       _ptr(dev_err), _stream(stream)))


def kvq_decode_attn_noalloc(k_pools: Sequence[Pool], v_pools: Sequence[Pool], q: torch.Tensor,
                            page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                            softmax_scale: float, out: torch.Tensor,
                            dev_err: torch.Tensor | None = None, stream=None) -> None:
    """kvq_decode_attn without a workspace, for callers that cannot allocate device memory where
    they run attention: the split partials use the library's own 32 MiB device array (shared by
    all calls; calls that overlap on the GPU race).  Make the first call on a device before any
    stream capture (it looks up that array's address)."""
    if len(k_pools) != len(v_pools):
        raise ValueError("one V pool per K pool")
    _cuda_tensor(q, torch.float16, "q")
    _cuda_tensor(out, torch.float32, "out")
    _cuda_tensor(page_table, torch.int32, "page_table")
    _cuda_tensor(seq_lens, torch.int32, "seq_lens")
    n_layers, nseq, hq, _ = q.shape
    if page_table.dim() != 2 or page_table.shape[0] < nseq or seq_lens.numel() < nseq:
        raise ValueError("page_table needs a row and seq_lens an entry per sequence")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    _check(_lib.kvq_decode_attn_noalloc(_pool_array(k_pools), _pool_array(v_pools), n_layers,
                                        q.data_ptr(), hq, page_table.data_ptr(),
                                        page_table.shape[1], seq_lens.data_ptr(), nseq,
                                        max_seq_len, softmax_scale, out.data_ptr(), _ptr(dev_err),
                                        _stream(stream)))


@dataclass
class KiviPacked:
    """Packed KIVI storage of one layer (see include/kvq.h): b-bit codes plus fp16 scale/zero per
    group, keys per (token group, channel), values per (token, channel group)."""
    bits: int
    group_size: int
    batch: int
    num_heads: int
    capacity: int
    head_dim: int
    k_codes: torch.Tensor
    k_scale: torch.Tensor
    k_zero: torch.Tensor
    v_codes: torch.Tensor
    v_scale: torch.Tensor
    v_zero: torch.Tensor

    @staticmethod
    def empty(bits, group_size, batch, num_heads, capacity, head_dim, device="cuda"):
        B, H, S, D, gs = batch, num_heads, capacity, head_dim, group_size
        cb = D * bits // 8
        u8 = dict(dtype=torch.uint8, device=device)
        f16 = dict(dtype=torch.float16, device=device)
        return KiviPacked(bits, gs, B, H, S, D,
                          torch.zeros((B, H, S, cb), **u8),
                          torch.zeros((B, H, S // gs, D), **f16),
                          torch.zeros((B, H, S // gs, D), **f16),
                          torch.zeros((B, H, S, cb), **u8),
                          torch.zeros((B, H, S, D // gs), **f16),
                          torch.zeros((B, H, S, D // gs), **f16))

    def nbytes(self, n_tokens: int) -> tuple[int, int]:
        """(key, value) bytes this layout stores for the first n_tokens tokens."""
        B, H, D, gs = self.batch, self.num_heads, self.head_dim, self.group_size
        code = n_tokens * D * self.bits // 8 * H * B
        return code + n_tokens // gs * D * 4 * H * B, code + n_tokens * (D // gs) * 4 * H * B

    def as_c(self) -> kivi_packed:
        return kivi_packed(self.bits, self.group_size, self.batch, self.num_heads, self.capacity,
                           self.head_dim, self.k_codes.data_ptr(), self.k_scale.data_ptr(),
                           self.k_zero.data_ptr(), self.v_codes.data_ptr(),
                           self.v_scale.data_ptr(), self.v_zero.data_ptr())


def _packed_array(caches: Sequence[KiviPacked]):
    arr = (kivi_packed * len(caches))()
    for i, c in enumerate(caches):
        arr[i] = c.as_c()
    return arr


def kivi_pack(caches: Sequence[KiviPacked], ks: Sequence[torch.Tensor],
              vs: Sequence[torch.Tensor], lo: int, hi: int, eps: float = 1e-8,
              stream=None) -> None:
    """Pack tokens [lo, hi) of every layer's fp16 K/V [B, H, capacity, D] into caches."""
    if not (len(caches) == len(ks) == len(vs)):
        raise ValueError("one K and one V tensor per cache")
    for i, (k, v) in enumerate(zip(ks, vs)):
        _cuda_tensor(k, torch.float16, f"ks[{i}]")
        _cuda_tensor(v, torch.float16, f"vs[{i}]")
    _check(_lib.kivi_pack(_packed_array(caches), _ptr_array(ks), _ptr_array(vs), len(caches), lo,
                          hi, eps, _stream(stream)))


def kivi_state_new(batch: int, num_heads: int, head_dim: int, capacity: int, bits: int = 2,
                   group_size: int = 32, residual_length: int = 128) -> kivi_state:
    """An empty KIVI cache state (offset 0, frontier 0)."""
    st = kivi_state()
    _check(_lib.kivi_state_init(ctypes.byref(st), batch, num_heads, head_dim, capacity, bits,
                                group_size, residual_length))
    return st


def _new_tokens(ks, vs, st):
    n = None
    for i, (k, v) in enumerate(zip(ks, vs)):
        _cuda_tensor(k, torch.float16, f"k_new[{i}]")
        _cuda_tensor(v, torch.float16, f"v_new[{i}]")
        if k.dim() != 4 or k.shape != v.shape or k.shape[0] != st.batch or \
                k.shape[1] != st.num_heads or k.shape[3] != st.head_dim:
            raise ValueError("new tokens are [B, H, n, D] per layer, K and V alike")
        if n is not None and k.shape[2] != n:
            raise ValueError("every layer appends the same number of tokens")
        n = k.shape[2]
    return n or 0


def _caches(kc, vc, st):
    for i, (k, v) in enumerate(zip(kc, vc)):
        _cuda_tensor(k, torch.float16, f"k_cache[{i}]")
        _cuda_tensor(v, torch.float16, f"v_cache[{i}]")
        if k.shape != (st.batch, st.num_heads, st.capacity, st.head_dim) or v.shape != k.shape:
            raise ValueError("caches are [B, H, capacity, D] per layer")


def _new_arrays(k_new, v_new, n_layers, st):
    """(k array, v array, n) for the C call; None, None means no new tokens (flush only)."""
    if k_new is None and v_new is None:
        return None, None, 0
    if not (len(k_new) == len(v_new) == n_layers):
        raise ValueError("one new-token tensor per layer, K and V")
    n = _new_tokens(k_new, v_new, st)
    return _ptr_array(k_new), _ptr_array(v_new), n


def kivi_update(st: kivi_state, k_cache, v_cache, k_new=None, v_new=None, stream=None) -> None:
    """update_and_fetch on the in-place fp16 cache (all layers); advances `st`.  k_new / v_new:
    [B, H, n, D] per layer, or None to flush without appending."""
    if len(k_cache) != len(v_cache):
        raise ValueError("one K and one V cache per layer")
    _caches(k_cache, v_cache, st)
    ka, va, n = _new_arrays(k_new, v_new, len(k_cache), st)
    _check(_lib.kivi_update(ctypes.byref(st), _ptr_array(k_cache), _ptr_array(v_cache), ka, va,
                            len(k_cache), n, _stream(stream)))


def kivi_trim(st: kivi_state, n: int) -> int:
    """trim on the in-place cache (host only); returns the number of tokens dropped."""
    return _lib.kivi_trim(ctypes.byref(st), n)


def kivi_packed_update(st: kivi_state, caches: Sequence["KiviPacked"], k_cache, v_cache,
                       k_new=None, v_new=None, stream=None) -> None:
    """update_and_fetch with the quantized region packed; advances `st`.  k_new / v_new as in
    kivi_update."""
    if not (len(caches) == len(k_cache) == len(v_cache)):
        raise ValueError("one packed cache and one K and V cache per layer")
    _caches(k_cache, v_cache, st)
    ka, va, n = _new_arrays(k_new, v_new, len(caches), st)
    _check(_lib.kivi_packed_update(ctypes.byref(st), _packed_array(caches), _ptr_array(k_cache),
                                   _ptr_array(v_cache), ka, va, len(caches), n, _stream(stream)))


def kivi_packed_trim(st: kivi_state, caches: Sequence["KiviPacked"], k_cache, v_cache, n: int,
                     stream=None) -> int:
    """trim with the quantized region packed; returns the number of tokens dropped."""
    if not (len(caches) == len(k_cache) == len(v_cache)):
        raise ValueError("one packed cache and one cache per layer")
    _caches(k_cache, v_cache, st)
    out = ctypes.c_int(0)
    _check(_lib.kivi_packed_trim(ctypes.byref(st), _packed_array(caches), _ptr_array(k_cache),
                                 _ptr_array(v_cache), len(caches), n, ctypes.byref(out),
                                 _stream(stream)))
    return out.value


def kivi_unpack(caches: Sequence["KiviPacked"], k, v, lo: int, hi: int, stream=None) -> None:
    """Write the reconstruction of packed tokens [lo, hi) into fp16 k[l], v[l]."""
    for i, (a, b) in enumerate(zip(k, v)):
        _cuda_tensor(a, torch.float16, f"k[{i}]")
        _cuda_tensor(b, torch.float16, f"v[{i}]")
    _check(_lib.kivi_unpack(_packed_array(caches), _ptr_array(k), _ptr_array(v), len(caches), lo,
                            hi, _stream(stream)))


def kivi_decode_attn_workspace(n_layers: int, batch: int, num_heads: int, num_q_heads: int,
                               head_dim: int, offset: int) -> int:
    return _lib.kivi_decode_attn_workspace(n_layers, batch, num_heads, num_q_heads, head_dim,
                                           offset)


def kivi_decode_attn(caches: Sequence[KiviPacked], ks: Sequence[torch.Tensor],
                     vs: Sequence[torch.Tensor], q: torch.Tensor, n_packed: int, offset: int,
                     softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                     dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Decode attention over packed tokens [0, n_packed) and fp16 residual tokens
    [n_packed, offset): q fp16 [n_layers, B, Hq, D] -> out float32."""
    _cuda_tensor(q, torch.float16, "q")
    _cuda_tensor(out, torch.float32, "out")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    for i, (k, v) in enumerate(zip(ks, vs)):
        _cuda_tensor(k, torch.float16, f"ks[{i}]")
        _cuda_tensor(v, torch.float16, f"vs[{i}]")
    _check(_lib.kivi_decode_attn(_packed_array(caches), _ptr_array(ks), _ptr_array(vs),
                                 len(caches), q.data_ptr(), q.shape[2], n_packed, offset,
                                 softmax_scale, out.data_ptr(), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(),
                                 _ptr(dev_err), _stream(stream)))


@dataclass
class Side:
    """fp16 side channels of one pool (see kvq_side in include/kvq.h)."""
    n_outlier: int
    n_sink: int
    out_val: torch.Tensor | None
    out_idx: torch.Tensor | None
    sink: torch.Tensor | None

    @staticmethod
    def empty(pool: "Pool", n_outlier: int, n_sink: int, max_seqs: int, device="cuda") -> "Side":
        P, H, ps = pool.num_pages, pool.num_heads, pool.page_size
        k = max(n_outlier, 1)
        val = torch.zeros((P, H, ps, k), dtype=torch.float16, device=device) if n_outlier else None
        idx = torch.zeros((P, H, ps, k), dtype=torch.uint8, device=device) if n_outlier else None
        sink = (torch.zeros((max_seqs, n_sink, H, pool.head_dim), dtype=torch.float16,
                            device=device) if n_sink else None)
        return Side(n_outlier, n_sink, val, idx, sink)

    @property
    def max_seqs(self) -> int:
        return self.sink.shape[0] if self.sink is not None else 0

    def as_c(self) -> kvq_side:
        return kvq_side(self.n_outlier, self.n_sink, self.max_seqs, _ptr(self.out_val),
                        _ptr(self.out_idx), _ptr(self.sink))


def _side_array(sides):
    arr = (kvq_side * len(sides))()
    for i, sd in enumerate(sides):
        arr[i] = sd.as_c()
    return arr


def kvq_quant_pack_paged_side(pools: Sequence[Pool], sides: Sequence[Side],
                              x: Sequence[torch.Tensor], page_table: torch.Tensor,
                              cu_new_tokens: torch.Tensor, start_pos: torch.Tensor,
                              dev_err: torch.Tensor | None = None, stream=None) -> None:
    """kvq_quant_pack_paged with outliers split off and sink rows kept exactly."""
    if not (len(pools) == len(sides) == len(x)):
        raise ValueError("one side and one input per pool")
    for i, t in enumerate(x):
        _cuda_tensor(t, torch.float16, f"x[{i}]")
    _cuda_tensor(page_table, torch.int32, "page_table")
    total = x[0].shape[0]
    _check(_lib.kvq_quant_pack_paged_side(_pool_array(pools), _side_array(sides), _ptr_array(x),
                                          len(pools), page_table.data_ptr(), page_table.shape[1],
                                          cu_new_tokens.data_ptr(), start_pos.data_ptr(),
                                          start_pos.numel(), total, _ptr(dev_err),
                                          _stream(stream)))


def kvq_dequant_paged_side(pools: Sequence[Pool], sides: Sequence[Side],
                           out: Sequence[torch.Tensor], page_table: torch.Tensor,
                           cu_tokens: torch.Tensor, start_pos: torch.Tensor,
                           dev_err: torch.Tensor | None = None, stream=None) -> None:
    """kvq_dequant_paged with the outliers written back and sink rows exact."""
    if not (len(pools) == len(sides) == len(out)):
        raise ValueError("one side and one output per pool")
    for i, t in enumerate(out):
        _cuda_tensor(t, torch.float16, f"out[{i}]")
    _cuda_tensor(page_table, torch.int32, "page_table")
    total = out[0].shape[0]
    _check(_lib.kvq_dequant_paged_side(_pool_array(pools), _side_array(sides), _ptr_array(out),
                                       len(pools), page_table.data_ptr(), page_table.shape[1],
                                       cu_tokens.data_ptr(), start_pos.data_ptr(),
                                       start_pos.numel(), total, _ptr(dev_err), _stream(stream)))


def kvq_decode_attn_side(k_pools: Sequence[Pool], v_pools: Sequence[Pool],
                         k_sides: Sequence[Side], v_sides: Sequence[Side], q: torch.Tensor,
                         page_table: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                         softmax_scale: float, out: torch.Tensor, workspace: torch.Tensor,
                         dev_err: torch.Tensor | None = None, stream=None) -> None:
    """Decode attention over pools with sinks and outlier side channels."""
    if not (len(k_pools) == len(v_pools) == len(k_sides) == len(v_sides)):
        raise ValueError("one V pool and one side per pool")
    _cuda_tensor(q, torch.float16, "q")
    _cuda_tensor(out, torch.float32, "out")
    _cuda_tensor(page_table, torch.int32, "page_table")
    _cuda_tensor(seq_lens, torch.int32, "seq_lens")
    n_layers, nseq, hq, _ = q.shape
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    _check(_lib.kvq_decode_attn_side(_pool_array(k_pools), _pool_array(v_pools),
                                     _side_array(k_sides), _side_array(v_sides), n_layers,
                                     q.data_ptr(), hq, page_table.data_ptr(), page_table.shape[1],
                                     seq_lens.data_ptr(), nseq, max_seq_len, softmax_scale,
                                     out.data_ptr(), workspace.data_ptr(),
                                     workspace.numel() * workspace.element_size(), _ptr(dev_err),
                                     _stream(stream)))


class HostView:
    """A page-locked host tensor seen through its device address (kvq_host_device_view): pass it
    where an entry point takes device input and the kernel reads the host memory directly."""

    def __init__(self, t: torch.Tensor):
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise TypeError("HostView needs a contiguous page-locked host tensor")
        out = ctypes.c_void_p()
        _check(_lib.kvq_host_device_view(t.data_ptr(), ctypes.byref(out)))
        self.tensor, self.ptr = t, out.value
        self.shape, self.dtype = t.shape, t.dtype

    def data_ptr(self) -> int:
        return self.ptr

    def numel(self) -> int:
        return self.tensor.numel()

    def element_size(self) -> int:
        return self.tensor.element_size()


def decode_workspace(k_pools: Sequence[Pool], nseq: int, num_q_heads: int, max_seq_len: int,
                     device="cuda") -> torch.Tensor:
    """A workspace tensor of the size kvq_decode_attn needs."""
    p = k_pools[0]
    n = kvq_decode_attn_workspace(len(k_pools), nseq, p.num_heads, num_q_heads, p.head_dim,
                                  p.page_size, max_seq_len)
    return torch.empty(max(n, 16), dtype=torch.uint8, device=device)


__all__ = ["KVQError", "Pool", "Allocator", "parse_mode", "kvq_version", "kvq_packed_dim",
           "kivi_boundary", "kvq_quant_pack_paged", "kvq_dequant_paged", "kivi_quant_dequant",
           "kvq_decode_attn_workspace", "kvq_decode_attn", "kvq_decode_attn_noalloc",
           "kvq_append_decode_attn", "Side", "kvq_quant_pack_paged_side",
           "kvq_dequant_paged_side", "kvq_decode_attn_side",
           "KiviPacked", "kivi_pack", "kivi_decode_attn_workspace", "kivi_decode_attn",
           "kivi_state", "kivi_state_new", "kivi_update", "kivi_trim", "kivi_packed_update",
           "kivi_packed_trim", "kivi_unpack",
           "decode_workspace", "LIB_PATH"]
