"""CPU oracle for the quantized paged KV-cache hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its CPU-baseline leg and its
``--impl reference`` arm) may import this package.  The product path (the
``paged_kv_cache_fp16_gb300`` package and its CUDA library) never calls it, and this package
imports nothing from the product path.

It is a plain, slow, obviously correct numpy restatement of what the pages compute:

* ``symmetric``  -- the symmetric per-token-per-head quantizer with one fp16 scale per row,
  q8/q6/q4 storage (the q6 4-codes-in-3-bytes layout), ``packed_dim``, dequantization, and the
  paged scatter/gather through a page table.
  Source: MTPLX pull request #267, "feat(kv-cache): add q6 paged KV quantization"
  (description: quantizer paragraph, byte-layout formula, ``packed_dim`` sentence, bit-width
  table paragraph; "Implementation").
* ``kivi``       -- KIVI's asymmetric min/max group quantize->dequantize round trip, the
  residual-window boundary, the in-place flush of ``update_and_fetch`` and the frontier
  rollback of ``trim``.
  Source: VeloxQuant-MLX source page "veloxquant_mlx.cache.kivi_cache"
  (``KIVIKVCache._quant_dequant_along``, ``_quantization_boundary``, ``update_and_fetch``,
  ``_rollback_frontier``, ``trim``).
* ``kivi_packed`` -- the packed KIVI storage the page only estimates (b-bit codes plus an fp16
  (scale, zero) per group) and decode attention over it with the fp16 residual window.
  Source: the same page (module docstring, ``_quantized_bytes``, ``_account_bytes``).
* ``attention``  -- decode attention as the reference path computes it: dequantize the packed
  cache to fp16, then plain softmax(q k^T * scale) v, here in float64; and one decode step
  (write the new token, then attend over the grown window) in that order.
  Source: MTPLX pull request #267, description ("plain KV quant dequantizes and runs MLX SDPA").
* ``side``       -- fp16 side channels on the symmetric quantizer: attention sinks kept exactly and
  each row's largest-magnitude elements kept as (fp16 value, position) pairs.
  Source: VeloxQuant-MLX API docs, "veloxquant_mlx.cache.kvquant_cache module" (byte
  accounting: the fp16 outlier side channel; Attention Sink-Aware quantization).
* ``storage``    -- the storage arithmetic (bytes per token per KV head, whole-cache GiB).
  Source: MTPLX pull request #267, description, storage paragraph.

Readings taken where the pages are silent are listed in each module's docstring.
Pins (checks against values and properties the pages and mathematics fix) live in
``tests/test_oracle_*.py`` and ``tests/golden/``.
"""
from . import symmetric, kivi, kivi_packed, attention, storage, side  # noqa: F401
