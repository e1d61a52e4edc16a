"""Benchmark: one step of the quantized paged KV-cache hot path on the paged-prefill workload.

Workload (per GPU): 16 layers x {K, V} x 8 sequences x 32,768 tokens x 4 KV heads x D = 256 fp16,
page size 16, a seeded random page table; the KIVI cache 16 layers x {K, V} [16, 8, 4096, 64].
One step runs, in order:
  1. kvq_quant_pack_paged over all 32 K/V tensors (q6 by default)   -- symmetric quantize + pack
  2. kvq_dequant_paged over all 32 tensors                           -- gather + unpack + dequant
  3. kvq_decode_attn: one decode query per sequence (24 query heads, GQA 6:1) over the packed
     cache just written, all 16 layers in one call                  -- packed decode attention
  4. kivi_quant_dequant of the 128 aged tokens [3840, 3968) of all 32 KIVI tensors
The metric is algorithmic bytes moved per second (GB/s, 1e9) over the whole step; per-kernel
figures, the packed-decode tokens/s, the q8/q4 variants and the 262,144-token decode are reported
alongside.  Inputs are far larger than L2 (129 MB), so no explicit flush between steps.

`--impl reference` times the CPU oracle (the plain restatement of the pages) on a bounded sample
of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

# the CPU baseline is reported for the threads it uses: keep BLAS single-threaded
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import kvgen  # noqa: E402

METRIC = "KV quant+pack / dequant GB/s and % of HBM roofline; packed decode attn tok/s"
WL = kvgen.WORKLOADS["paged_prefill_16L_8x32768_4x256"]
KV = kvgen.WORKLOADS["kivi_flush_16L_16x8x4096x64"]
HQ = 24
SOFTMAX_SCALE = 1.0 / 16.0
KIVI_LO, KIVI_HI = 3840, 3968
KIVI_HQ = 32                      # GQA 4:1 over the KIVI cache's 8 KV heads
KIVI_BITS = 2
KIVI_OFFSET = KV["S"]             # decode at a full 4096-token cache
KIVI_NPACKED = KV["S"] - KV["residual"]   # 3968 packed tokens + a 128-token fp16 window
FALLBACK_HBM_GBS = 6800.0


def packed_dim(D, bits):
    return {8: D, 6: D * 3 // 4, 4: D // 2}[bits]


def bytes_quant(rows, D, bits):        # read fp16 row, write packed row + fp16 scale
    return rows * (2 * D + packed_dim(D, bits) + 2)


def bytes_decode(layers, tokens_total, H, D, bits, nseq, hq):
    kv = layers * tokens_total * H * 2 * (packed_dim(D, bits) + 2)
    return kv + layers * nseq * hq * D * (2 + 4)


def bytes_kivi(n_tensors, B, H, span, D):
    return n_tensors * B * H * span * D * 4


def kernel_source_hash(sources):
    """sha256 over the files a kernel is built from (paths relative to the repository): recorded
    ncu traffic is only valid for the code it measured."""
    import hashlib
    h = hashlib.sha256()
    for rel in sorted(sources):
        with open(os.path.join(ROOT, rel), "rb") as fh:
            h.update(rel.encode() + b"\0" + fh.read())
    return h.hexdigest()


def recorded_traffic(stage, bits):
    """DRAM bytes per launch from the committed ncu record, or None if the kernel's sources
    changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    e = rec.get("kernels", {}).get(f"{stage}/q{bits}")
    if e is None:
        return None
    try:
        if e.get("source_sha256") != kernel_source_hash(e.get("sources", [])):
            return None
    except OSError:
        return None
    return e.get("bytes_per_launch")


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"kvq_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s in sm if s >= 0.5 * max(sm)]
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- GPU arm
L2_FLUSH_BYTES = 256 << 20   # twice the GB300's 129 MB L2


def time_fn_flushed(fn, reps, warmup, stream, dev):
    """Median device time of one call of fn, the L2 flushed (a 256 MB buffer written) before each
    repetition; only the call itself is between the events."""
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        flush.fill_(0)
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(reps)]
    for i, (a, b) in enumerate(ev):
        flush.fill_(i & 0xFF)
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    del flush
    return statistics.median(a.elapsed_time(b) / 1e3 for a, b in ev)


def time_fn_graph(fn, reps, warmup, stream):
    """Device time of one call of fn with the calls back to back: reps calls captured in a CUDA
    graph and replayed, so the host's launch cost (the Python binding's argument marshalling) is
    not between them -- for calls of a few microseconds."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(reps):
            fn()
    g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    del g
    return a.elapsed_time(b) / 1e3 / reps


def roundtrip_extra(kvq, dev, steps, warmup, stream):
    """The q6 round trip of one layer: K and V each [1 seq, 1,024 tokens, 4 KV heads, 256] fp16
    (keys with 4 outlier channels per head x10; two all-zero rows), contiguous (one 1,024-token
    page per sequence, identity table): kvq_quant_pack_paged of both tensors in one call, then
    kvq_dequant_paged of both.  The working set (5.78 MB each way) fits in L2, so the L2 is flushed
    before every repetition and the figures are latency-bound, not HBM roofline figures."""
    w = kvgen.WORKLOADS["q6_roundtrip_1x1024x4x256"]
    T, H, D, bits = w["n_tok"], w["H"], w["D"], w["bits"]
    xs = [kvgen.KVSpec(seed=w["seed"], layer=0, is_key=k, n_seq=1, n_tok=T, num_heads=H,
                       head_dim=D).full_torch(dev) for k in (True, False)]
    pools = [kvq.Pool.empty(bits, H, D, T, 1, dev) for _ in xs]
    outs = [torch.empty_like(x) for x in xs]
    pt = torch.zeros((1, 1), dtype=torch.int32, device=dev)
    cu = torch.tensor([0, T], dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def quant():
        kvq.kvq_quant_pack_paged(pools, xs, pt, cu, st, err)

    def deq():
        kvq.kvq_dequant_paged(pools, outs, pt, cu, st, err)

    def both():
        quant()
        deq()

    reps = max(steps, 20)
    tq = time_fn_flushed(quant, reps, warmup, stream, dev)
    td = time_fn_flushed(deq, reps, warmup, stream, dev)
    tb = time_fn_flushed(both, reps, warmup, stream, dev)
    tbw = time_fn_graph(both, reps, warmup, stream)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError("device error word set in the round trip")
    nb = bytes_quant(2 * T * H, D, bits)
    return {"rows": 2 * T * H, "bytes_each_way": nb,
            "quant_pack_us": tq * 1e6, "quant_pack_GB_s": nb / tq / 1e9,
            "dequant_us": td * 1e6, "dequant_GB_s": nb / td / 1e9,
            "round_trip_us": tb * 1e6, "round_trip_GB_s": 2 * nb / tb / 1e9,
            "round_trip_us_l2_resident": tbw * 1e6,
            "l2": "L2-resident working set; L2 flushed (256 MB write) before each repetition; "
                  "median of the repetitions; latency-bound, not an HBM roofline figure"}


def append_extra(kvq, dev, steps, warmup, stream, bits=6):
    """kvq_quant_pack_paged of a decode-step append: 64 sequences with cached lengths uniform in
    [1,024, 65,536] append 1, 8 or 32 tokens each into their partially filled tail pages (mapped by
    the host allocator), 16 layers x {K, V} in one call.  Timed back to back from a CUDA graph (the
    step's new rows were just produced, so they sit in L2) and with the L2 flushed before each
    call."""
    wl = kvgen.WORKLOADS["decode_append_16L_64seq_4x256"]
    L, nseq, H, D, ps = wl["n_layers"], wl["n_seq"], wl["H"], wl["D"], wl["page_size"]
    cur = kvgen.decode_append_lengths(wl["seed"], nseq)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    res = {}
    for n_new in wl["appends"]:
        max_pages = (int(cur.max()) + n_new + ps - 1) // ps
        table = torch.full((nseq, max_pages), -1, dtype=torch.int32)
        alloc = kvq.Allocator(nseq * 4)
        alloc.reserve(table, ps, cur, [n_new] * nseq)
        pt = table.to(dev)
        pools = [kvq.Pool.empty(bits, H, D, ps, nseq * 4, dev) for _ in range(2 * L)]
        xs = [kvgen.KVSpec(seed=wl["seed"], layer=l, is_key=k, n_seq=nseq, n_tok=n_new,
                           num_heads=H, head_dim=D, zero_rows=False).full_torch(dev)
              for l in range(L) for k in (True, False)]
        cu = torch.tensor(np.arange(nseq + 1) * n_new, dtype=torch.int32, device=dev)
        st = torch.from_numpy(cur.astype(np.int32)).to(dev)

        def fn():
            kvq.kvq_quant_pack_paged(pools, xs, pt, cu, st, err)

        tw = time_fn_graph(fn, max(steps, 20), warmup, stream)
        tc = time_fn_flushed(fn, max(steps, 20), warmup, stream, dev)
        rows = 2 * L * nseq * n_new * H
        nb = bytes_quant(rows, D, bits)
        res[f"{n_new}_tok"] = {"rows": rows, "bytes": nb, "us": tw * 1e6, "GB_s": nb / tw / 1e9,
                               "us_l2_flushed": tc * 1e6, "GB_s_l2_flushed": nb / tc / 1e9,
                               "ideal_us_at_measured_peak": nb / (measured_peaks()[0] * 1e9) * 1e6}
        del pools, xs, alloc
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError("device error word set in the append extra")
    torch.cuda.empty_cache()
    return res


def kivi_flush_extra(w, steps, warmup, stream, dev, lo, hi):
    """A KIVI flush of tokens [lo, hi) of every layer's K and V (16 layers x [16, 8, 4096, 64]):
    32 tokens is one group, as decode reaches each group boundary; 128 tokens is the step's flush.
    Timed back to back from a CUDA graph and with the L2 flushed before each call."""

    def fn():
        w.kvq.kivi_quant_dequant(w.kivi, w.kivi_flags, lo, hi, KV["group_size"], KV["levels"],
                                 KV["eps"])

    t = time_fn_graph(fn, max(steps, 20), warmup, stream)
    tc = time_fn_flushed(fn, max(steps, 20), warmup, stream, dev)
    nb = bytes_kivi(len(w.kivi), KV["B"], KV["H"], hi - lo, KV["D"])
    return {"tokens": hi - lo, "bytes": nb, "us": t * 1e6, "GB_s": nb / t / 1e9,
            "us_l2_flushed": tc * 1e6, "GB_s_l2_flushed": nb / tc / 1e9}


def decode_step_extra(kvq, dev, steps, warmup, stream, bits=6):
    """One decode step of 64 sequences with lengths uniform in [1024, 65536] over 16 layers
    (4 KV heads x 256, 24 query heads, page 16): the fused kvq_append_decode_attn against the two
    calls it replaces (kvq_quant_pack_paged of the 64 new tokens, then kvq_decode_attn).  The
    cache pages hold seeded random codes and scales (the work does not depend on them); the new
    tokens and queries come from the generator.  Each timed step rewrites the same tail slots."""
    wl = kvgen.WORKLOADS["decode_append_16L_64seq_4x256"]
    L, nseq, H, D, ps = wl["n_layers"], wl["n_seq"], wl["H"], wl["D"], wl["page_size"]
    lens = kvgen.decode_append_lengths(wl["seed"], nseq).astype(np.int64)
    ppseq = (lens + 1 + ps - 1) // ps
    perm = kvgen.permutation(wl["seed"], 77, int(ppseq.sum()))
    pt_np = np.full((nseq, int(ppseq.max())), -1, dtype=np.int32)
    o = 0
    for s_ in range(nseq):
        pt_np[s_, :ppseq[s_]] = perm[o:o + ppseq[s_]]
        o += ppseq[s_]
    n_pages = int(ppseq.sum())
    pools = []
    for i in range(2 * L):
        p = kvq.Pool.empty(bits, H, D, ps, n_pages, dev)
        kvgen.fill_random_pool_(p.codes, p.scales, 1000 + i)
        pools.append(p)
    kps, vps = pools[0::2], pools[1::2]
    kn = [kvgen.KVSpec(seed=wl["seed"], layer=l, is_key=True, n_seq=1, n_tok=nseq, num_heads=H,
                       head_dim=D).full_torch(dev) for l in range(L)]
    vn = [kvgen.KVSpec(seed=wl["seed"], layer=l, is_key=False, n_seq=1, n_tok=nseq, num_heads=H,
                       head_dim=D).full_torch(dev) for l in range(L)]
    q = kvgen.queries_torch(wl["seed"], L, nseq, HQ, D, dev)
    out = torch.empty(q.shape, dtype=torch.float32, device=dev)
    pt = torch.from_numpy(pt_np).to(dev)
    lens_d = torch.from_numpy(lens.astype(np.int32)).to(dev)
    lens1_d = lens_d + 1
    cu = torch.arange(nseq + 1, dtype=torch.int32, device=dev)
    max_len = int(lens.max()) + 1
    ws = kvq.decode_workspace(kps, nseq, HQ, max_len, dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    new = [t for pair in zip(kn, vn) for t in pair]

    def fused():
        kvq.kvq_append_decode_attn(kps, vps, kn, vn, q, pt, lens_d, max_len, SOFTMAX_SCALE, out,
                                   ws, err)

    def separate():
        kvq.kvq_quant_pack_paged(pools, new, pt, cu, lens_d, err)
        kvq.kvq_decode_attn(kps, vps, q, pt, lens1_d, max_len, SOFTMAX_SCALE, out, ws, err)

    tf = time_fn(fused, steps, warmup, stream)
    ts = time_fn(separate, steps, warmup, stream)
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise RuntimeError("device error word set in the decode step")
    pd = packed_dim(D, bits)
    tok_heads = int((lens + 1).sum()) * L * H
    nbytes = (tok_heads * 2 * (pd + 2) + L * nseq * H * 2 * (2 * D + pd + 2)
              + L * nseq * HQ * D * (2 + 4))
    res = {"ms": tf * 1e3, "tok_s": nseq / tf, "GB_s": nbytes / tf / 1e9,
           "separate_ms": ts * 1e3, "separate_tok_s": nseq / ts, "bytes": nbytes,
           "cached_tokens": int(lens.sum())}
    del pools, kps, vps, kn, vn, new
    torch.cuda.empty_cache()
    return res


def kivi_loop_extra(kvq, dev, warmup, stream, passes=3):
    """The KIVI serving loop on the [16, 8, 4096, 64] x 16-layer cache (2-bit, group 32, residual
    128): from a prefill of 3,936 tokens (3,808 packed), 32 decode steps, each appending one token
    to every layer (kivi_packed_update; one flush of 32 tokens falls in the 32 steps) and running
    kivi_decode_attn for 32 query heads over the packed tokens and the fp16 window.  The state
    is restored to the post-prefill point before every pass (a pass rewrites the same bytes)."""
    L, B, H, S, D, gs = KV["n_layers"], KV["B"], KV["H"], KV["S"], KV["D"], KV["group_size"]
    prefill, steps = 3936, 32
    kc = [kvgen.KiviSpec(seed=KV["seed"], layer=l, is_key=True, batch=B, num_heads=H, seq=S,
                         head_dim=D).full_torch(dev) for l in range(L)]
    vc = [kvgen.KiviSpec(seed=KV["seed"], layer=l, is_key=False, batch=B, num_heads=H, seq=S,
                         head_dim=D).full_torch(dev) for l in range(L)]
    caches = [kvq.KiviPacked.empty(KIVI_BITS, gs, B, H, S, D, dev) for _ in range(L)]
    st = kvq.kivi_state_new(B, H, D, S, bits=KIVI_BITS, group_size=gs,
                            residual_length=KV["residual"])
    st.offset = prefill                      # the caches hold the prefill tokens already
    kvq.kivi_packed_update(st, caches, kc, vc)   # pack the aged prefill tokens
    nq0 = st.n_quantized
    # new tokens of each step, [B, H, 1, D] per layer (the generator's tokens 3936..3967)
    kn = [[kc[l][:, :, prefill + i:prefill + i + 1].clone() for l in range(L)] for i in range(steps)]
    vn = [[vc[l][:, :, prefill + i:prefill + i + 1].clone() for l in range(L)] for i in range(steps)]
    q = kvgen.queries_torch(KV["seed"] + 1, L, B, KIVI_HQ, D, dev)
    out = torch.empty((L, B, KIVI_HQ, D), dtype=torch.float32, device=dev)
    ws = torch.empty(kvq.kivi_decode_attn_workspace(L, B, H, KIVI_HQ, D, S), dtype=torch.uint8,
                     device=dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1.0 / np.sqrt(D)

    def one_pass():
        st.offset, st.n_quantized = prefill, nq0
        for i in range(steps):
            kvq.kivi_packed_update(st, caches, kc, vc, kn[i], vn[i])
            kvq.kivi_decode_attn(caches, kc, vc, q, st.n_quantized, st.offset, scale, out, ws, err)

    for _ in range(warmup):
        one_pass()
    torch.cuda.synchronize()
    times = []
    for _ in range(passes):
        st.offset, st.n_quantized = prefill, nq0
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(steps):
            kvq.kivi_packed_update(st, caches, kc, vc, kn[i], vn[i])
            kvq.kivi_decode_attn(caches, kc, vc, q, st.n_quantized, st.offset, scale, out, ws, err)
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) / 1e3)
    if int(err.item()) != 0:
        raise RuntimeError("device error word set in the KIVI loop")
    t = sum(times) / len(times)
    res = {"ms_per_step": t / steps * 1e3, "tok_s": B * steps / t, "steps": steps,
           "flushes": 1, "first_offset": prefill + 1}
    del kc, vc, caches, kn, vn
    torch.cuda.empty_cache()
    return res


def side_extra(w, kvq, dev, steps, warmup, stream, bits=6, n_sink=4, fraction=0.01):
    """The symmetric path with fp16 side channels on the paged-prefill workload: quant-pack with
    k = ceil(0.01 * D) = 3 outliers per row and 4 sink tokens per sequence, dequant, and decode
    attention (8 sequences x 24 query heads) over the result."""
    k = int(np.ceil(fraction * w.D))
    pools = w.make_pools(bits)
    sides = [kvq.Side.empty(p, k, n_sink, w.nseq, dev) for p in pools]
    q, out, ws = w.dec_buffers()

    def quant():
        kvq.kvq_quant_pack_paged_side(pools, sides, w.x, w.pt, w.cu, w.start, w.err)

    def deq():
        kvq.kvq_dequant_paged_side(pools, sides, w.deq, w.pt, w.cu, w.start, w.err)

    def attn():
        kvq.kvq_decode_attn_side(pools[0::2], pools[1::2], sides[0::2], sides[1::2], q, w.pt,
                                 w.lens, w.ntok, SOFTMAX_SCALE, out, ws, w.err)

    tq = time_fn(quant, steps, warmup, stream)
    td = time_fn(deq, steps, warmup, stream)
    ta = time_fn(attn, steps, warmup, stream)
    torch.cuda.synchronize()
    if int(w.err.item()) != 0:
        raise RuntimeError("device error word set in the side-channel extra")
    rows = w.L * 2 * w.nseq * w.ntok * w.H
    side_b = 3 * k                                       # fp16 value + uint8 position per outlier
    bq = rows * (2 * w.D + packed_dim(w.D, bits) + 2 + side_b)
    ba = (w.L * w.nseq * w.ntok * w.H * 2 * (packed_dim(w.D, bits) + 2 + side_b)
          + w.L * w.nseq * HQ * w.D * (2 + 4))
    res = {"outliers_per_row": k, "sinks": n_sink,
           "quant_pack_ms": tq * 1e3, "quant_pack_GB_s": bq / tq / 1e9,
           "dequant_ms": td * 1e3, "dequant_GB_s": bq / td / 1e9,
           "decode_attn_ms": ta * 1e3, "decode_attn_GB_s": ba / ta / 1e9,
           "decode_attn_tok_s": w.nseq / ta}
    del pools, sides
    torch.cuda.empty_cache()
    return res


class Workload:
    """Device-resident inputs and outputs of one replica (outputs allocated on first use)."""

    def __init__(self, kvq, dev, bits, layers=None):
        self.kvq, self.dev = kvq, dev
        L = WL["n_layers"] if layers is None else layers
        nseq, ntok, H, D, ps = WL["n_seq"], WL["n_tok"], WL["H"], WL["D"], WL["page_size"]
        self.L, self.nseq, self.ntok, self.H, self.D, self.ps = L, nseq, ntok, H, D, ps
        self.specs = [kvgen.KVSpec(seed=WL["seed"], layer=l, is_key=k, n_seq=nseq, n_tok=ntok,
                                   num_heads=H, head_dim=D)
                      for l in range(L) for k in (True, False)]
        self._x = None
        self.pt_np = kvgen.random_page_table(1, nseq, ntok // ps)
        self.pt = torch.from_numpy(self.pt_np).to(dev)
        self.pt1 = self.pt.reshape(1, -1).contiguous()      # one 262,144-token sequence
        self.cu = torch.tensor(np.arange(nseq + 1) * ntok, dtype=torch.int32, device=dev)
        self.start = torch.zeros(nseq, dtype=torch.int32, device=dev)
        self.lens = torch.full((nseq,), ntok, dtype=torch.int32, device=dev)
        self.lens1 = torch.tensor([nseq * ntok], dtype=torch.int32, device=dev)
        self.bits = bits
        self._pools = None
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self._deq = self._dec = self._dec1 = self._kivi = self._kp = None
        self.kivi_layers = KV["n_layers"] if layers is None else layers

    @property
    def x(self):
        """The paged-prefill fp16 inputs (16 GiB at 16 layers), generated on first use."""
        if self._x is None:
            self._x = [s.full_torch(self.dev) for s in self.specs]
        return self._x

    @property
    def pools(self):
        if self._pools is None:
            self._pools = {self.bits: self.make_pools(self.bits)}
        return self._pools

    @property
    def deq(self):
        if self._deq is None:
            self._deq = [torch.empty_like(t) for t in self.x]
        return self._deq

    def dec_buffers(self, full_context=False):
        if full_context:
            if self._dec1 is None:
                q = kvgen.queries_torch(WL["seed"] + 1, self.L, 1, HQ, self.D, self.dev)
                out = torch.empty((self.L, 1, HQ, self.D), dtype=torch.float32, device=self.dev)
                ws = self.kvq.decode_workspace(self.pools[self.bits][0::2], 1, HQ,
                                               self.nseq * self.ntok, self.dev)
                self._dec1 = (q, out, ws)
            return self._dec1
        if self._dec is None:
            q = kvgen.queries_torch(WL["seed"], self.L, self.nseq, HQ, self.D, self.dev)
            out = torch.empty((self.L, self.nseq, HQ, self.D), dtype=torch.float32,
                              device=self.dev)
            ws = self.kvq.decode_workspace(self.pools[self.bits][0::2], self.nseq, HQ,
                                           self.ntok, self.dev)
            self._dec = (q, out, ws)
        return self._dec

    @property
    def q(self):
        return self.dec_buffers()[0]

    @property
    def out(self):
        return self.dec_buffers()[1]

    @property
    def kivi(self):
        if self._kivi is None:
            self._kivi = [kvgen.KiviSpec(seed=KV["seed"], layer=l, is_key=k, batch=KV["B"],
                                         num_heads=KV["H"], seq=KV["S"], head_dim=KV["D"]
                                         ).full_torch(self.dev)
                          for l in range(self.kivi_layers) for k in (True, False)]
        return self._kivi

    @property
    def kivi_flags(self):
        return [k for _ in range(self.kivi_layers) for k in (True, False)]

    def kivi_packed(self):
        """(caches, ks, vs, q, out, workspace) of the packed KIVI cache (2-bit, group 32)."""
        if self._kp is None:
            L, B, H, S, D = self.kivi_layers, KV["B"], KV["H"], KV["S"], KV["D"]
            caches = [self.kvq.KiviPacked.empty(KIVI_BITS, KV["group_size"], B, H, S, D, self.dev)
                      for _ in range(L)]
            q = kvgen.queries_torch(KV["seed"], L, B, KIVI_HQ, D, self.dev)
            out = torch.empty((L, B, KIVI_HQ, D), dtype=torch.float32, device=self.dev)
            ws = torch.empty(self.kvq.kivi_decode_attn_workspace(L, B, H, KIVI_HQ, D, KIVI_OFFSET),
                             dtype=torch.uint8, device=self.dev)
            self._kp = (caches, self.kivi[0::2], self.kivi[1::2], q, out, ws)
        return self._kp

    def kivi_pack(self):
        caches, ks, vs = self.kivi_packed()[:3]
        self.kvq.kivi_pack(caches, ks, vs, 0, KIVI_NPACKED, KV["eps"])

    def kivi_attn(self, n_packed=KIVI_NPACKED):
        caches, ks, vs, q, out, ws = self.kivi_packed()
        self.kvq.kivi_decode_attn(caches, ks, vs, q, n_packed, KIVI_OFFSET,
                                  1.0 / np.sqrt(KV["D"]), out, ws)

    def kivi_packed_bytes(self):
        """Algorithmic bytes of the pack and of the two attention launches (packed / all fp16)."""
        L, B, H, D = self.kivi_layers, KV["B"], KV["H"], KV["D"]
        kb, vb = self.kivi_packed()[0][0].nbytes(KIVI_NPACKED)
        fp16_tok = B * H * D * 2 * 2            # K and V bytes of one token, all rows
        qo = B * KIVI_HQ * D * (2 + 4)
        return {"pack": L * (KIVI_NPACKED * fp16_tok + kb + vb),
                "attn_packed": L * (kb + vb + (KIVI_OFFSET - KIVI_NPACKED) * fp16_tok + qo),
                "attn_fp16": L * (KIVI_OFFSET * fp16_tok + qo)}

    def make_pools(self, bits):
        return [self.kvq.Pool.empty(bits, self.H, self.D, self.ps, self.pt_np.size, self.dev)
                for _ in range(2 * self.L)]

    # the four stages of one step
    def quant(self, bits):
        self.kvq.kvq_quant_pack_paged(self.pools[bits], self.x, self.pt, self.cu, self.start,
                                      self.err)

    def dequant(self, bits):
        self.kvq.kvq_dequant_paged(self.pools[bits], self.deq, self.pt, self.cu, self.start,
                                   self.err)

    def decode(self, bits):
        p = self.pools[bits]
        q, out, ws = self.dec_buffers()
        self.kvq.kvq_decode_attn(p[0::2], p[1::2], q, self.pt, self.lens, self.ntok,
                                 SOFTMAX_SCALE, out, ws, self.err)

    def decode_full_context(self, bits):
        p = self.pools[bits]
        q, out, ws = self.dec_buffers(full_context=True)
        self.kvq.kvq_decode_attn(p[0::2], p[1::2], q, self.pt1, self.lens1,
                                 self.nseq * self.ntok, SOFTMAX_SCALE, out, ws, self.err)

    def kivi_flush(self):
        self.kvq.kivi_quant_dequant(self.kivi, self.kivi_flags, KIVI_LO, KIVI_HI,
                                    KV["group_size"], KV["levels"], KV["eps"])

    def bytes(self, bits):
        rows = self.L * 2 * self.nseq * self.ntok * self.H
        return {
            "quant_pack": bytes_quant(rows, self.D, bits),
            "dequant": bytes_quant(rows, self.D, bits),
            "decode_attn": bytes_decode(self.L, self.nseq * self.ntok, self.H, self.D, bits,
                                        self.nseq, HQ),
            "kivi": bytes_kivi(len(self.kivi), KV["B"], KV["H"], KIVI_HI - KIVI_LO, KV["D"]),
        }


def time_step(w, bits, steps, stream):
    """Run `steps` steps with events between the stages; returns (total_s, per-stage seconds)."""
    names = ["quant_pack", "dequant", "decode_attn", "kivi"]
    fns = [lambda: w.quant(bits), lambda: w.dequant(bits), lambda: w.decode(bits), w.kivi_flush]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for k in range(steps):
        for i, fn in enumerate(fns):
            ev[k][i].record(stream)
            fn()
        ev[k][4].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    per = {n: [] for n in names}
    for k in range(steps):
        for i, n in enumerate(names):
            per[n].append(ev[k][i].elapsed_time(ev[k][i + 1]) / 1e3)
    return start.elapsed_time(end) / 1e3, per


def time_fn(fn, steps, warmup, stream):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / 1e3 / steps


def run_gpu(args):
    world, rank, local = dist_setup(args.gpus)
    import paged_kv_cache_fp16_gb300 as kvq
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    bits = args.bits
    w = Workload(kvq, dev, bits, layers=args.layers)
    if args.only:
        run_only(w, bits, args, stream)
        return
    B = w.bytes(bits)
    step_bytes = sum(B.values())

    for _ in range(args.warmup):
        w.quant(bits); w.dequant(bits); w.decode(bits); w.kivi_flush()
    torch.cuda.synchronize()
    if int(w.err.item()) != 0:
        raise RuntimeError("device error word set during warm-up")

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        total, per = time_step(w, bits, args.steps, stream)
        barrier(world)
        torch.cuda.synchronize()
    clocks = clk.summary()
    total = max_over_ranks(total, world, dev)
    ms_per_step = total / args.steps * 1e3
    value = world * step_bytes * args.steps / total / 1e9
    launches_per_step = 5   # quant, dequant, decode + merge, kivi (keys and values in one launch)

    stage = {}
    for n, ts in per.items():
        avg = sum(ts) / len(ts)
        stage[n] = {"ms": avg * 1e3, "GB_s": B[n] / avg / 1e9}
    stage["decode_attn"]["tok_s"] = w.nseq / (sum(per["decode_attn"]) / len(per["decode_attn"]))
    peak, peak_kind = measured_peaks()
    dom = max(per, key=lambda n: sum(per[n]))
    dom_avg = sum(per[dom]) / len(per[dom])
    achieved = B[dom] / dom_avg / 1e9
    roofline = {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1),
                "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
                "traffic": (args.traffic if args.traffic is not None
                            else recorded_traffic(dom, bits))}

    # end to end through the public API with host buffers (before the extras, which allocate and
    # free tens of GB)
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(w, kvq, bits, args, stream, world, dev, step_bytes)

    # extras outside the timed step: 262,144-token decode, q8/q4 variants
    extras = {}
    t = time_fn(lambda: w.decode_full_context(bits), args.steps, args.warmup, stream)
    extras["decode_attn_262144_1seq"] = {"ms": t * 1e3, "tok_s": 1.0 / t,
                                         "GB_s": bytes_decode(w.L, w.nseq * w.ntok, w.H, w.D,
                                                              bits, 1, HQ) / t / 1e9}
    if not args.no_widths:
        for b2 in (8, 4):
            if b2 == bits:
                continue
            w.pools[b2] = w.make_pools(b2)
            tq = time_fn(lambda: w.quant(b2), args.steps, args.warmup, stream)
            td = time_fn(lambda: w.dequant(b2), args.steps, args.warmup, stream)
            ta = time_fn(lambda: w.decode_full_context(b2), args.steps, args.warmup, stream)
            Bq = bytes_quant(w.L * 2 * w.nseq * w.ntok * w.H, w.D, b2)
            extras[f"q{b2}"] = {"quant_pack_GB_s": Bq / tq / 1e9, "dequant_GB_s": Bq / td / 1e9,
                                "decode_attn_262144_tok_s": 1.0 / ta,
                                "decode_attn_GB_s": bytes_decode(w.L, w.nseq * w.ntok, w.H, w.D,
                                                                 b2, 1, HQ) / ta / 1e9}
            del w.pools[b2]
            torch.cuda.empty_cache()

    # packed KIVI: pack the aged tokens of all 16 layers, decode over packed + residual, and the
    # same decode over the fp16 cache (n_packed = 0) for comparison
    if not args.no_kivi_packed:
        Bk = w.kivi_packed_bytes()
        tp = time_fn(w.kivi_pack, args.steps, args.warmup, stream)
        ta = time_fn(w.kivi_attn, args.steps, args.warmup, stream)
        tf = time_fn(lambda: w.kivi_attn(0), args.steps, args.warmup, stream)
        w.kivi_pack()
        extras["kivi_packed_2bit_16L_16x8x4096x64"] = {
            "pack_ms": tp * 1e3, "pack_GB_s": Bk["pack"] / tp / 1e9,
            "attn_ms": ta * 1e3, "attn_tok_s": KV["B"] / ta,
            "attn_GB_s": Bk["attn_packed"] / ta / 1e9,
            "attn_fp16_cache_ms": tf * 1e3, "attn_fp16_cache_tok_s": KV["B"] / tf,
            "attn_fp16_cache_GB_s": Bk["attn_fp16"] / tf / 1e9}
        del w._kp
        w._kp = None
        torch.cuda.empty_cache()

    # the symmetric path with fp16 sinks and outlier side channels
    if not args.no_side:
        extras["side_q6_k3_sink4"] = side_extra(w, kvq, dev, args.steps, args.warmup, stream)

    # the KIVI serving loop: append one token, flush every 32, attend over packed + window
    if not args.no_kivi_packed:
        extras["kivi_decode_loop_16L_16x8_2bit"] = kivi_loop_extra(kvq, dev, args.warmup, stream)

    # the small configurations: the q6 round trip of one layer, the decode-step appends and the
    # 32-token KIVI flush
    if not args.no_small:
        extras["q6_roundtrip_1x1024x4x256"] = roundtrip_extra(kvq, dev, args.steps, args.warmup,
                                                              stream)
        extras["append_q6_16L_64seq"] = append_extra(kvq, dev, args.steps, args.warmup, stream)
        for lo, hi in KV["flushes"]:
            extras[f"kivi_flush_{hi - lo}tok_16L"] = kivi_flush_extra(w, args.steps, args.warmup,
                                                                      stream, dev, lo, hi)

    # one decode step (append + attend) of 64 ragged sequences
    if not args.no_decode_step:
        extras["decode_step_64seq_ragged_16L_q6"] = decode_step_extra(kvq, dev, args.steps,
                                                                      args.warmup, stream)


    if int(w.err.item()) != 0:
        raise RuntimeError("device error word set")
    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
            "data": "synthetic (seeded counter-based generator, shapes of the pages' workloads)",
            "config": {"workload": "paged_prefill_16L_8x32768_4x256 step: quant-pack -> "
                                   "dequant -> packed decode attn (8 seqs x 24 q heads) -> "
                                   "KIVI flush 128 tok of 16L x [16,8,4096,64]",
                       "bits": bits, "layers": w.L, "seqs": w.nseq, "tokens_per_seq": w.ntok,
                       "kv_heads": w.H, "head_dim": w.D, "page_size": w.ps, "q_heads": HQ,
                       "l2": "inputs larger than L2 (no flush)",
                       "bytes_per_step": step_bytes, "parallelism": f"replicas x{world}"},
            "stages": {k: {kk: round(vv, 3) for kk, vv in v.items()} for k, v in stage.items()},
            "extras": _rounded(extras),
            "roofline": roofline,
            "e2e": e2e,
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))


def _rounded(obj):
    """The extras with floats rounded to 3 decimals, nested dicts included."""
    if isinstance(obj, dict):
        return {k: _rounded(v) for k, v in obj.items()}
    if isinstance(obj, float):
        return round(obj, 3)
    return obj


def run_only(w, bits, args, stream):
    """Profiling aid: run one stage warmup + steps times on a (possibly reduced) workload."""
    fn = {"quant_pack": lambda: w.quant(bits), "dequant": lambda: w.dequant(bits),
          "decode_attn": lambda: w.decode(bits), "kivi": w.kivi_flush,
          "decode_attn_262144": lambda: w.decode_full_context(bits),
          "kivi_pack": w.kivi_pack, "kivi_attn": w.kivi_attn,
          "kivi_attn_fp16": lambda: w.kivi_attn(0)}.get(args.only)
    if args.only.startswith("kivi"):   # the KIVI stages need none of the paged workload
        if args.only.startswith("kivi_attn"):
            w.kivi_pack()
    elif args.only.startswith("side_"):   # side channels: 3 outliers per row, 4 sinks
        kvq = w.kvq
        pools = w.pools[bits]
        sides = [kvq.Side.empty(p, int(np.ceil(0.01 * w.D)), 4, w.nseq, w.dev) for p in pools]
        q, out, ws = w.dec_buffers()
        fn = {"side_quant": lambda: kvq.kvq_quant_pack_paged_side(pools, sides, w.x, w.pt, w.cu,
                                                                  w.start, w.err),
              "side_dequant": lambda: kvq.kvq_dequant_paged_side(pools, sides, w.deq, w.pt, w.cu,
                                                                 w.start, w.err),
              "side_attn": lambda: kvq.kvq_decode_attn_side(pools[0::2], pools[1::2], sides[0::2],
                                                            sides[1::2], q, w.pt, w.lens, w.ntok,
                                                            SOFTMAX_SCALE, out, ws, w.err)}[args.only]
        kvq.kvq_quant_pack_paged_side(pools, sides, w.x, w.pt, w.cu, w.start, w.err)
    else:
        w.quant(bits)
    torch.cuda.synchronize()
    t = time_fn(fn, args.steps, args.warmup, stream)
    print(json.dumps({"profile_only": args.only, "layers": w.L, "bits": bits,
                      "ms": round(t * 1e3, 4), "err": int(w.err.item())}))


def run_e2e(w, kvq, bits, args, stream, world, dev, step_bytes):
    """Per step, through the public API: copy the step's fp16 K/V inputs (17 GB) and queries from
    pinned host memory, run the four stages, read the attention output back.  The copies run on a
    copy stream one layer at a time and each layer is quantized as soon as its copy lands (one
    kvq_quant_pack_paged call per layer), so the host link -- the bound of this loop -- never waits
    for the GPU: the next step's copy of a layer starts once this step's quantization has consumed
    it, under this step's dequantization, attention and KIVI flush."""
    host_x = [t.cpu().pin_memory() for t in w.x]
    host_q = w.q.cpu().pin_memory()
    host_out = torch.empty(w.out.shape, dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host_x) + host_q.numel() * 2
    d2h = host_out.numel() * 4
    copy = torch.cuda.Stream(device=dev)
    L = w.L
    landed = [torch.cuda.Event() for _ in range(L)]
    consumed = [torch.cuda.Event() for _ in range(L)]
    q_landed, decoded = torch.cuda.Event(), torch.cuda.Event()
    state = {"first": True}

    def step():
        for l in range(L):
            if not state["first"]:
                copy.wait_event(consumed[l])     # the previous step's quant has read layer l
            with torch.cuda.stream(copy):
                for i in (2 * l, 2 * l + 1):
                    w.x[i].copy_(host_x[i], non_blocking=True)
                landed[l].record(copy)
        if not state["first"]:
            copy.wait_event(decoded)             # the previous step's attention has read q
        with torch.cuda.stream(copy):
            w.q.copy_(host_q, non_blocking=True)
            q_landed.record(copy)
        for l in range(L):
            stream.wait_event(landed[l])
            kvq.kvq_quant_pack_paged(w.pools[bits][2 * l:2 * l + 2], w.x[2 * l:2 * l + 2], w.pt,
                                     w.cu, w.start, w.err)
            consumed[l].record(stream)
        w.dequant(bits)
        stream.wait_event(q_landed)
        w.decode(bits)
        decoded.record(stream)
        w.kivi_flush()
        host_out.copy_(w.out, non_blocking=True)
        state["first"] = False

    n = max(1, min(args.steps, 5))
    for _ in range(min(args.warmup, 2)):
        step()
    torch.cuda.synchronize()
    # the host link alone, just before the timed loop: the copies of the first 8 input tensors
    # (4 GiB) with nothing else running, best of three; the loop cannot beat h2d bytes / this rate
    p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    probe = host_x[:min(8, len(host_x))]

    def host_link():
        best = 0.0
        for _ in range(3):
            p0.record(copy)
            with torch.cuda.stream(copy):
                for i, hx in enumerate(probe):
                    w.x[i].copy_(hx, non_blocking=True)
            p1.record(copy)
            torch.cuda.synchronize()
            best = max(best, sum(t_.numel() * t_.element_size() for t_ in probe) /
                       (p0.elapsed_time(p1) / 1e3))
        return best

    link = host_link()
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    copy.wait_event(a)            # the timed region starts before the first copy
    for _ in range(n):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    t = max_over_ranks(a.elapsed_time(b) / 1e3, world, dev)
    link_after = host_link()   # the same probe right after the loop
    del host_x
    return {"value": round(world * step_bytes * n / t / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "ms_per_step": round(t / n * 1e3, 3),
            "host_link_GB_s": round(link / 1e9, 1),
            "host_link_after_GB_s": round(link_after / 1e9, 1),
            "host_link_floor_ms_per_step": round(h2d / link * 1e3, 1),
            "pipeline": "per-layer H2D on a copy stream overlapped with quant-pack"}


# ----------------------------------------------------------------------------- CPU (oracle) arm
_CPU_INPUTS = {}


def _cpu_inputs():
    """Seeded inputs of the CPU sample (generated once, outside the timed oracle work)."""
    if not _CPU_INPUTS:
        D, H, ps, n_tok = WL["D"], WL["H"], WL["page_size"], 4096
        _CPU_INPUTS["pt"] = kvgen.random_page_table(1, 1, n_tok // ps)
        _CPU_INPUTS["xs"] = [kvgen.KVSpec(seed=WL["seed"], layer=0, is_key=k, n_seq=1,
                                          n_tok=n_tok, num_heads=H, head_dim=D).full_np()
                             for k in (True, False)]
        _CPU_INPUTS["q"] = kvgen.queries_np(WL["seed"], 1, 1, HQ, D)
        _CPU_INPUTS["kivi"] = [kvgen.KiviSpec(seed=KV["seed"], layer=0, is_key=k, batch=1,
                                              num_heads=KV["H"], seq=KV["S"], head_dim=KV["D"]
                                              ).full_np() for k in (True, False)]
    return _CPU_INPUTS


def cpu_sample_step():
    """One bounded sample of the step, run through the oracle: returns algorithmic bytes."""
    from oracle import attention as oa
    from oracle import kivi as ok
    from oracle import symmetric as osym
    D, H, ps, n_tok = WL["D"], WL["H"], WL["page_size"], 4096
    inp = _cpu_inputs()
    pt = inp["pt"]
    pools = []
    for x in inp["xs"]:
        p = osym.PagedPool(6, H, D, ps, pt.size)
        osym.quant_pack_paged(p, x, pt, np.array([0, n_tok]), np.array([0]))
        osym.dequant_paged(p, pt, np.array([0, n_tok]), np.array([0]))
        pools.append(p)
    oa.decode_attention_paged(inp["q"][0], pools[0], pools[1], pt, np.array([n_tok]),
                              SOFTMAX_SCALE)
    kk, vv = (t.copy() for t in inp["kivi"])
    ok.flush(kk, vv, KIVI_LO, KIVI_HI, KV["group_size"], KV["levels"], KV["eps"])
    rows = 2 * n_tok * H
    return (2 * bytes_quant(rows, D, 6) + bytes_decode(1, n_tok, H, D, 6, 1, HQ)
            + bytes_kivi(2, 1, KV["H"], KIVI_HI - KIVI_LO, KV["D"]))


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


_POOL_BARRIER = None


def _cpu_pool_init(barrier):
    """Pool worker start-up: the shared barrier and this worker's inputs (outside any timing)."""
    global _POOL_BARRIER
    _POOL_BARRIER = barrier
    _cpu_inputs()


def _cpu_pool_task(n_iter):
    """One worker's share: wait until every worker is ready, then n_iter oracle samples.
    Returns (bytes, start, end) on the host's monotonic clock (common to all processes)."""
    _POOL_BARRIER.wait()
    t0 = time.perf_counter()
    total = 0
    for _ in range(n_iter):
        total += cpu_sample_step()
    return total, t0, time.perf_counter()


class OraclePool:
    """The oracle run on every host core at once: one spawned process per core (a process pool
    started with `spawn`, so no CUDA state is inherited), each running whole samples of the
    workload; BLAS stays single-threaded in every process."""

    def __init__(self, n_workers):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.n = n_workers
        self.barrier = ctx.Barrier(n_workers)
        self.pool = ctx.Pool(n_workers, initializer=_cpu_pool_init, initargs=(self.barrier,))

    def run(self, n_iter):
        """Every worker runs n_iter samples, all starting together; (bytes, wall seconds)."""
        res = self.pool.map(_cpu_pool_task, [n_iter] * self.n, chunksize=1)
        return sum(r[0] for r in res), max(r[2] for r in res) - min(r[1] for r in res)

    def close(self):
        self.pool.close()
        self.pool.join()


CPU_SAMPLE = ("1 layer K+V of 4,096 tokens x 4 heads x 256 quant-pack + dequant (q6, page 16), "
              "decode attn over it (24 q heads), KIVI flush of 128 tokens of 1 layer "
              "[1, 8, 4096, 64] K+V")


def cpu_baseline(seconds):
    """The oracle on one core for about `seconds`, then on every host core (one process per core,
    each running the same number of samples) for about as long."""
    _cpu_inputs()
    t0 = time.perf_counter()
    total, n = 0, 0
    while True:
        total += cpu_sample_step()
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    single = total / dt / 1e9
    cores = host_cores()
    out = {"value": round(single, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"{n} x ({CPU_SAMPLE}); {dt:.1f} s", "single_core_GB_s": round(single, 4)}
    if cores > 1:
        pool = OraclePool(cores)
        try:
            pool.run(1)                                 # every worker warm
            per = max(1, int(round(n * 1.0)))           # each core repeats the single-core run
            tot, wall = pool.run(per)
        finally:
            pool.close()
        out.update({"value": round(tot / wall / 1e9, 4), "cores": cores,
                    "sample": f"{cores} processes x {per} x ({CPU_SAMPLE}), {wall:.1f} s wall; "
                              f"single core: {n} x the same, {dt:.1f} s",
                    "all_cores_GB_s": round(tot / wall / 1e9, 4)})
    return out


def run_reference(args):
    """The oracle as it stands on the host cores: each step, every core (one spawned process per
    core) runs one sample of the step's workload, all starting together."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    cores = host_cores()
    pool = OraclePool(cores)
    try:
        for _ in range(max(1, args.warmup)):
            pool.run(1)
        total, dt = 0, 0.0
        for _ in range(args.steps):
            b, t = pool.run(1)
            total += b
            dt += t
    finally:
        pool.close()
    value = total / dt / 1e9
    sample = f"per step: {cores} processes x 1 x ({CPU_SAMPLE})"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic (seeded counter-based generator)",
        "config": {"workload": "paged_prefill_16L_8x32768_4x256 step, bounded sample per step",
                   "bits": 6},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["kvq", "reference"], default="kvq")
    ap.add_argument("--bits", type=int, default=6, choices=[8, 6, 4])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-widths", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--layers", type=int, default=None,
                    help="profiling only: fewer layers than the workload's 16")
    ap.add_argument("--only", default=None,
                    choices=["quant_pack", "dequant", "decode_attn", "kivi", "decode_attn_262144",
                             "kivi_pack", "kivi_attn", "kivi_attn_fp16", "side_quant",
                             "side_dequant", "side_attn"],
                    help="profiling only: run one stage and print its time, no bench line")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the side-channel (sinks + outliers) extra")
    ap.add_argument("--no-decode-step", action="store_true",
                    help="skip the fused append + decode step extra")
    ap.add_argument("--no-kivi-packed", action="store_true",
                    help="skip the packed KIVI pack/attention extras")
    ap.add_argument("--no-small", action="store_true",
                    help="skip the round-trip, append and 32-token flush extras")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per launch of the dominant kernel, if captured")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "kvq":
        ap.error("--warmup must be >= 3")
    if args.layers is not None and not args.only:
        ap.error("--layers is a profiling option: use it with --only")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
