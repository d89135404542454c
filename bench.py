"""Benchmark of the paged KV-cache hot path on GB300.

Step (the timed unit): one decode step of one layer on the long-context
workload -- B=8 sequences with contexts of 32K..128K tokens, H_Q=32, H_KV=8,
d=128, bf16, block size 16, shuffled physical blocks: write each sequence's
newest K/V token into the paged cache, then decode attention over it --
one launch of pa_paged_decode_step (--step two-call: pa_reshape_and_cache
followed by pa_paged_decode_attention).
Inputs are resident in HBM before the timed region; the KV cache (~2.9 GB)
is far larger than L2 (129 MB), so no flush is needed between steps.

Printed as one JSON line:
  value     decode KV GB/s: algorithmic bytes of the step / step time
  roofline  the decode attention kernel (one launch) against measured HBM
  e2e       the same metric through the C ABI with pinned HOST buffers, the
            per-step inputs copied in and the output copied back each step
  extras    cache-write tokens/s (32K-token prefill write, fp8/bf16/SWA) and
            the MLA K assembly (16K tokens), each over its own loop with an
            L2 flush (a 258 MB read) between iterations
  cpu_baseline  the CPU oracle on a bounded sample of the same workload

--impl reference times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("hbm_gbs"):
            return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def rank_seed(rank: int) -> int:
    """Seed of rank r's copy of the workload (rank 0 uses the spec's seed 4)."""
    return 4 + 1000 * rank


def reduce_over_ranks(value: float, op: str, device=None) -> float:
    """max or sum of a per-rank number over all ranks (identity without a
    process group); the only cross-rank traffic of the benchmark."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def bf16_peak():
    """Dense bf16 tensor TFLOP/s (measured burst, else the fallback)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        if d.get("bf16_tflops"):
            return float(d["bf16_tflops"])
    return 1900.0


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ------------------------------------------------------------- clocks ----
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while running."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in getattr(self, "lines", []):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        # samples under load: the top 80% (the sampler brackets the timed region)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------- helpers ----
def up(a, dtype, dev):
    import torch
    a = np.ascontiguousarray(a)
    t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).to(dev)
    return t.view(dtype) if dtype is not None else t


def traffic_record(kernel_file, workload, step, kv_dtype):
    """Per-launch DRAM bytes from the committed ncu records, if one was taken
    on the current source of the kernel and the same workload, step and KV
    format (else None)."""
    rec = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(rec):
        return None
    with open(rec) as f:
        d = json.load(f)
    # the kernel's source and the shared device header it includes
    hs = hashlib.sha256()
    for path in (kernel_file, os.path.join(os.path.dirname(kernel_file), "pa_internal.cuh")):
        with open(path, "rb") as f:
            hs.update(f.read())
    h = hs.hexdigest()[:16]
    for r in d.get("records", [d]):
        if (r.get("source_sha256_16") == h and r.get("workload") == workload
                and r.get("step") == step and r.get("kv_dtype") == kv_dtype):
            return r.get("dram_bytes_per_decode_call")
    return None


# ------------------------------------------------------------ our arm ----
class DecodeStep:
    """One variant of the decode step (block size, KV format, one launch or
    two) on the long-context workload, resident on the device."""

    def __init__(self, seed, block_size, kv_dtype, step, num_seqs, dev):
        import torch

        from paged_kv_cache_309_gb300 import pa
        from paged_kv_cache_309_gb300 import workloads as wl
        w = wl.long_context_decode(seed=seed, block_size=block_size, num_seqs=num_seqs)
        self.fp8 = kv_dtype == "e4m3"
        self.kv_dtype, self.step_kind = kv_dtype, step
        self.ksd = self.vsd = None
        if self.fp8:  # same sequences, an e4m3 cache with k_scale = v_scale = 0.05
            w = wl.as_fp8_history(w, seed=seed + 100)
            self.ksd = torch.tensor([0.05], dtype=torch.float32, device=dev)
            self.vsd = torch.tensor([0.05], dtype=torch.float32, device=dev)
        self.w = w
        B, HQ, HKV, d = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_size
        cache_t = torch.float8_e4m3fn if self.fp8 else torch.bfloat16
        self.kc, self.vc = up(w.k_cache, cache_t, dev), up(w.v_cache, cache_t, dev)
        self.q = up(w.q, torch.bfloat16, dev)
        self.nk, self.nv = up(w.new_k, torch.bfloat16, dev), up(w.new_v, torch.bfloat16, dev)
        self.sl = torch.from_numpy(w.slot_mapping).to(dev)
        self.bt = torch.from_numpy(w.block_tables).to(dev)
        self.cl = torch.from_numpy(w.context_lens).to(dev)
        self.out = torch.empty_like(self.q)
        self.mcl = w.max_context_len
        self.wsp = pa.decode_workspace(B, HQ, HKV, d, self.mcl, dev)
        self.splits, self.tps = pa.pa_paged_decode_plan(B, HKV, self.mcl)
        elt = 1 if self.fp8 else 2
        self.attn_bytes = wl.kv_bytes_read(w, elt=elt)  # algorithmic, decode attention
        self.write_bytes = B * HKV * d * 2 * (2 + elt) + B * 8  # new K/V read + written, slots
        self.step_bytes = self.attn_bytes + self.write_bytes
        self.fused = step == "fused"
        self.dev = dev

    def attention(self, q=None, nk=None, nv=None, sl=None, bt=None, cl=None):
        """The timed launch: the fused step, or the attention of the two-call step."""
        from paged_kv_cache_309_gb300 import pa
        q, bt, cl = (self.q if q is None else q, self.bt if bt is None else bt,
                     self.cl if cl is None else cl)
        if self.fused:
            pa.pa_paged_decode_step(self.out, q, self.nk if nk is None else nk,
                                    self.nv if nv is None else nv, self.sl if sl is None else sl,
                                    self.kc, self.vc, bt, cl, self.w.scale, self.mcl, self.wsp,
                                    k_scale=self.ksd, v_scale=self.vsd)
        else:
            pa.pa_paged_decode_attention(self.out, q, self.kc, self.vc, bt, cl, self.w.scale,
                                         self.mcl, self.wsp, k_scale=self.ksd, v_scale=self.vsd)

    def write(self, nk=None, nv=None, sl=None):
        """The cache write of the two-call step (nothing for the fused step)."""
        from paged_kv_cache_309_gb300 import pa
        if not self.fused:
            pa.pa_reshape_and_cache(self.nk if nk is None else nk, self.nv if nv is None else nv,
                                    self.kc, self.vc, self.sl if sl is None else sl, None,
                                    self.ksd, self.vsd)

    def timed(self, K, warmup, clock_device, barrier=None):
        """W untimed steps, then exactly K steps between a barrier and a
        synchronize on both sides; CUDA events on the launching stream around
        the whole region and around each timed attention launch; nvidia-smi
        samples the clocks meanwhile.  Returns (ms over the K steps, mean ms
        per attention launch, clock summary)."""
        import torch
        stream = torch.cuda.current_stream()
        for _ in range(warmup):
            self.write()
            self.attention()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(K)]
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if barrier:
            barrier()
        torch.cuda.synchronize()
        with ClockSampler(clock_device) as clk:
            start.record(stream)
            for i in range(K):
                self.write()
                ev[i][0].record(stream)
                self.attention()
                ev[i][1].record(stream)
            stop.record(stream)
            torch.cuda.synchronize()
        if barrier:
            barrier()
        return (start.elapsed_time(stop), statistics.mean(a.elapsed_time(b) for a, b in ev),
                clk.summary())

    def kernel_bytes(self):
        """Algorithmic bytes of the timed launch."""
        return self.step_bytes if self.fused else self.attn_bytes

    def traffic(self):
        return traffic_record(os.path.join(ROOT, "paged_kv_cache_309_gb300", "csrc", "decode.cu"),
                              self.w.name, self.step_kind, self.kv_dtype)


def run_ours(args):
    import torch
    import torch.distributed as dist

    from paged_kv_cache_309_gb300 import pa

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pa.library()  # fails loudly if the CUDA library is missing

    # ---------------- workload (rank r uses seed 4 + 1000 r: weak scaling)
    st = DecodeStep(rank_seed(rank), args.block_size, args.kv_dtype, args.step, args.num_seqs,
                    dev)
    w, fused, fp8 = st.w, st.fused, st.fp8
    B, HQ, HKV, d = w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_size
    stream = torch.cuda.current_stream()

    # ---------------- timed region: exactly K steps
    K = args.steps
    barrier = dist.barrier if ws_n > 1 else None
    ms_total, attn_ms_avg, clocks = st.timed(K, args.warmup, local, barrier)
    ms_total = reduce_over_ranks(ms_total, "max", dev)
    job_bytes = reduce_over_ranks(st.step_bytes, "sum", dev)   # every rank's own workload
    job_seqs = reduce_over_ranks(B, "sum", dev)
    assert pa.read_device_error(st.wsp) == 0, "device error word set"
    ms_step = ms_total / K
    value = job_bytes / (ms_step * 1e-3) / 1e9
    peak, peak_kind = hbm_peak()
    kernel_bytes = st.kernel_bytes()
    achieved = kernel_bytes / (attn_ms_avg * 1e-3) / 1e9

    # ---------------- end to end through the C ABI with pinned host buffers:
    # every step copies its inputs in (one pinned staging buffer holding q,
    # the new K/V rows, slot mapping, block tables and context lengths at
    # 256-byte aligned offsets: one host-to-device copy per step) and its
    # output back, over the same K
    parts = [np.ascontiguousarray(a) for a in (w.q.view(np.int16), w.new_k.view(np.int16),
                                               w.new_v.view(np.int16), w.slot_mapping,
                                               w.block_tables, w.context_lens)]
    offs, size = [], 0
    for a in parts:
        offs.append(size)
        size += (a.nbytes + 255) // 256 * 256
    hbuf = torch.empty(size, dtype=torch.uint8).pin_memory()
    hnp = hbuf.numpy()
    for a, o in zip(parts, offs):
        hnp[o:o + a.nbytes] = a.view(np.uint8).reshape(-1)
    dbuf = torch.empty(size, dtype=torch.uint8, device=dev)

    def dview(i, dtype):
        a = parts[i]
        return dbuf[offs[i]:offs[i] + a.nbytes].view(dtype).view(a.shape)

    dq, dk, dv = (dview(i, torch.int16) for i in range(3))
    dsl, dbt, dcl = dview(3, torch.int64), dview(4, torch.int32), dview(5, torch.int32)
    hout = torch.empty(st.out.shape, dtype=torch.int16).pin_memory()
    h2d = size
    d2h = hout.numel() * hout.element_size()

    def e2e_step():
        dbuf.copy_(hbuf, non_blocking=True)
        bq, bk, bv = (t.view(torch.bfloat16) for t in (dq, dk, dv))
        st.write(bk, bv, dsl)
        st.attention(bq, bk, bv, dsl, dbt, dcl)
        hout.copy_(st.out.view(torch.int16), non_blocking=True)

    for _ in range(args.warmup):
        e2e_step()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if barrier:
        barrier()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    e0.record(stream)
    for _ in range(K):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_wall_ms = (time.perf_counter() - t0) * 1e3 / K
    e2e_ms = reduce_over_ranks(e0.elapsed_time(e1), "max", dev) / K
    assert np.array_equal(hout.numpy(), st.out.view(torch.int16).cpu().numpy())

    result = {
        "metric": "paged decode-attn KV GB/s (% of HBM peak); cache-write tokens/s",
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": ws_n,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3 KV, bf16 q/out" if fp8 else "bf16",
        "data": ("synthetic (seeded random finite e4m3 KV codes, scale 0.05; N(0,1) bf16 q)"
                 if fp8 else "synthetic (seeded N(0,1) bf16, shuffled block pool)"),
        "config": {"workload": w.name, "num_seqs": B, "num_q_heads": HQ, "num_kv_heads": HKV,
                   "head_size": d, "block_size": w.block_size, "kv_dtype": args.kv_dtype,
                   "context_tokens": int(w.context_lens.sum()),
                   "max_context_len": st.mcl, "splits": st.splits, "tokens_per_split": st.tps,
                   "step": ("paged_decode_step (new-token write + attention, one launch)" if fused
                            else "reshape_and_cache(new tokens) + paged_decode_attention"),
                   "l2": "inputs larger than L2 (KV cache %.2f GB)" % (
                       2 * w.k_cache.nbytes / 1e9),
                   "parallelism": f"replicas x{ws_n} (independent sequences per GPU)"},
        "pct_of_hbm_peak": round(100 * value / peak, 2),
        "sequences_per_s": round(job_seqs / (ms_step * 1e-3), 1),
        "roofline": {"kernel": "paged_decode_split_tc_kernel" + (" (fused write, in-kernel merge)"
                                                                 if fused else " (in-kernel merge)"),
                     "bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": st.traffic(),
                     "bytes_per_launch": kernel_bytes, "avg_launch_us": round(attn_ms_avg * 1e3, 2)},
        "e2e": {"value": round(job_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 5), "host_wall_ms_per_step": round(e2e_wall_ms, 5),
                "steps": K, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": (1 if fused else 2) * K,
        "clocks": clocks,
    }
    del st, dq, dk, dv, dsl, dbt, dcl

    if rank == 0 and not args.no_extras:
        torch.cuda.empty_cache()
        result["extras"] = run_step_extras(args, dev, peak, local)
        result["extras"].update(run_extras(args, dev, peak))
    if rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws_n > 1:
        dist.destroy_process_group()


def run_step_extras(args, dev, peak, clock_device):
    """The other variants of the long-context decode step the benchmark's
    workload names -- block size 64 (bf16 cache) and an fp8 e4m3 cache with
    k_scale = v_scale = 0.05 (block size 16) -- each timed exactly like the
    main line (K steps after W warm-up steps, CUDA events, clocks sampled)."""
    import torch

    from paged_kv_cache_309_gb300 import pa
    ex = {}
    for bs, kv in ((64, "bf16"), (16, "e4m3")):
        if (bs, kv) == (args.block_size, args.kv_dtype):
            continue
        st = DecodeStep(rank_seed(0), bs, kv, "fused", args.num_seqs, dev)
        ms_total, attn_ms, clocks = st.timed(args.steps, args.warmup, clock_device)
        assert pa.read_device_error(st.wsp) == 0, "device error word set"
        ms_step = ms_total / args.steps
        kb = st.kernel_bytes()
        ach = kb / (attn_ms * 1e-3) / 1e9
        name = st.w.name
        ex[name] = {"step": "paged_decode_step (new-token write + attention, one launch)",
                    "block_size": bs, "kv_dtype": kv,
                    "k_scale": 0.05 if st.fp8 else None, "v_scale": 0.05 if st.fp8 else None,
                    "steps": args.steps, "warmup": args.warmup,
                    "ms_per_step": round(ms_step, 5),
                    "GB_per_s": round(st.step_bytes / (ms_step * 1e-3) / 1e9, 2),
                    "sequences_per_s": round(st.w.num_seqs / (ms_step * 1e-3), 1),
                    "context_tokens_per_s": round(int(st.w.context_lens.sum()) /
                                                  (ms_step * 1e-3), 1),
                    "roofline": {"kernel": "paged_decode_split_tc_kernel (fused write)",
                                 "bound": "hbm", "achieved": round(ach, 2), "peak": peak,
                                 "unit": "GB/s", "frac": round(ach / peak, 4),
                                 "traffic": st.traffic(), "bytes_per_launch": kb,
                                 "avg_launch_us": round(attn_ms * 1e3, 2)},
                    "clocks": clocks}
        del st
        torch.cuda.empty_cache()
    return ex


def timed_loop(fn, iters, warm, dev, flush_bytes=2 * L2_BYTES):
    """Median and mean device time of fn over `iters` calls.  Before each
    call, outside the timed events, L2 is flushed by READING a 258 MB buffer
    written once up front (a read leaves no dirty lines whose write-back
    would land inside the timed kernel), and the GPU is kept busy by a short
    device sleep while the host enqueues the call, so that host-side launch
    work does not show up as idle time between the events."""
    import torch
    scratch = torch.ones(flush_bytes // 4, dtype=torch.float32, device=dev)
    sink = torch.empty((), dtype=torch.float32, device=dev)
    for _ in range(warm):
        fn()
    times = []
    s = torch.cuda.current_stream()
    for _ in range(iters):
        torch.amax(scratch, dim=0, out=sink)
        torch.cuda._sleep(200_000)  # ~100 us at 2 GHz: covers the host's enqueue of fn
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        times.append((a, b))
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in times]
    return statistics.median(ms), statistics.mean(ms)


def run_extras(args, dev, peak):
    import torch

    from paged_kv_cache_309_gb300 import pa
    from paged_kv_cache_309_gb300 import workloads as wl
    ex = {}
    iters = args.extra_iters
    for variant in ("e4m3", "bf16", "e4m3_swa"):
        w = wl.prefill_write(variant=variant)
        H, d = w.key.shape[1:]
        cdt = torch.float8_e4m3fn if w.cache_dtype == "e4m3" else torch.bfloat16
        kc = torch.zeros((w.num_blocks, w.block_size, H, d), dtype=cdt, device=dev)
        vc = torch.zeros_like(kc)
        key, val = up(w.key, torch.bfloat16, dev), up(w.value, torch.bfloat16, dev)
        sl = torch.from_numpy(w.slot_mapping).to(dev)
        swa = None if w.swa_slot_mapping is None else torch.from_numpy(w.swa_slot_mapping).to(dev)
        ks = None if w.k_scale is None else torch.tensor([w.k_scale], dtype=torch.float32,
                                                         device=dev)
        vs = None if ks is None else ks.clone()
        fn = lambda: pa.pa_reshape_and_cache(key, val, kc, vc, sl, swa, ks, vs)
        med, mean = timed_loop(fn, iters, 3, dev)
        nbytes = wl.write_bytes(w)
        toks = w.key.shape[0]
        ex[w.name] = {"tokens_per_s": round(toks / (med * 1e-3), 1),
                      "written_tokens": wl.write_tokens_effective(w),
                      "GB_per_s": round(nbytes / (med * 1e-3) / 1e9, 2),
                      "frac_of_hbm_peak": round(nbytes / (med * 1e-3) / 1e9 / peak, 4),
                      "median_us": round(med * 1e3, 2), "algorithmic_bytes": nbytes}
    m = wl.mla_assembly()
    N = m.k_nope.shape[0]
    kn, kr = up(m.k_nope, torch.bfloat16, dev), up(m.k_rope, torch.bfloat16, dev)
    k = torch.empty((N, 128, 192), dtype=torch.bfloat16, device=dev)
    med, _ = timed_loop(lambda: pa.pa_concat_mla_k(k, kn, kr), iters, 3, dev)
    nbytes = N * (128 * 128 * 2 + 64 * 2 + 128 * 192 * 2)
    ex[m.name] = {"tokens_per_s": round(N / (med * 1e-3), 1),
                  "GB_per_s": round(nbytes / (med * 1e-3) / 1e9, 2),
                  "frac_of_hbm_peak": round(nbytes / (med * 1e-3) / 1e9 / peak, 4),
                  "median_us": round(med * 1e3, 2), "algorithmic_bytes": nbytes}
    # causal prefill: 4 fresh prompts of 8192 tokens, H_Q=32, H_KV=8, bs=16
    pw = wl.make_prefill("prefill_attention_b4_8k", 5, [8192] * 4, [8192] * 4, 32, 8, 128, 16)
    pq = up(pw.q, torch.bfloat16, dev)
    pout = torch.empty_like(pq)
    pkc, pvc = up(pw.k_cache, torch.bfloat16, dev), up(pw.v_cache, torch.bfloat16, dev)
    pbt = torch.from_numpy(pw.block_tables).to(dev)
    pcu = torch.from_numpy(pw.cu_seqlens_q).to(dev)
    pcl = torch.from_numpy(pw.context_lens).to(dev)
    perr = torch.zeros(1, dtype=torch.int32, device=dev)
    med, _ = timed_loop(lambda: pa.pa_paged_prefill_attention(pout, pq, pkc, pvc, pbt, pcu, pcl,
                                                              pw.scale, pw.max_q_len, perr),
                        max(3, iters // 5), 2, dev)
    flops = wl.prefill_flops(pw)
    ex[pw.name] = {"tokens_per_s": round(int(pw.cu_seqlens_q[-1]) / (med * 1e-3), 1),
                   "TFLOP_per_s": round(flops / (med * 1e-3) / 1e12, 2),
                   "frac_of_bf16_dense_peak": round(flops / (med * 1e-3) / 1e12 / bf16_peak(), 4),
                   "median_us": round(med * 1e3, 2), "causal_flops": flops}
    # the latent-cache write: [c_kv | k_pe] per token into [256, 64, 1, 576]
    # in one pass (pa_concat_and_cache_mla)
    ckv, kpe = up(m.c_kv, torch.bfloat16, dev), up(m.k_pe, torch.bfloat16, dev)
    cache = torch.zeros((m.num_blocks, m.block_size, 1, 576), dtype=torch.bfloat16, device=dev)
    sl = torch.from_numpy(m.slot_mapping).to(dev)
    med, _ = timed_loop(lambda: pa.pa_concat_and_cache_mla(ckv, kpe, cache, sl), iters, 3, dev)
    nbytes = N * (576 * 2 * 2 + 8)  # each row read and written once, plus its slot
    # context for a launch this short: a plain device-to-device copy of the same
    # rows (N x 1152 B read and written), timed the same way
    csrc = torch.empty(N * 576, dtype=torch.bfloat16, device=dev)
    cdst = torch.empty_like(csrc)
    cmed, _ = timed_loop(lambda: cdst.copy_(csrc), iters, 3, dev)
    del csrc, cdst
    ex["mla_latent_cache_write_16k"] = {"call": "pa_concat_and_cache_mla (one launch)",
                                        "tokens_per_s": round(N / (med * 1e-3), 1),
                                        "GB_per_s": round(nbytes / (med * 1e-3) / 1e9, 2),
                                        "frac_of_hbm_peak": round(nbytes / (med * 1e-3) / 1e9 /
                                                                  peak, 4),
                                        "median_us": round(med * 1e3, 2),
                                        "algorithmic_bytes": nbytes,
                                        "same_bytes_device_copy_us": round(cmed * 1e3, 2),
                                        "frac_of_same_bytes_copy_rate": round(cmed / med, 4)}
    # MLA decode over the latent cache (DeepSeek-V3-shaped: B=64, context
    # 512..4096, bs=64): 128 heads (tcgen05 kernel, heads on M) and 16 heads
    # (one TP8 shard, tcgen05 kernel with tokens on M); for 128 heads also
    # the absorbed chain
    for H in (128, 16):
        mw = wl.mla_decode(num_heads=H, with_weights=(H == 128))
        mq, mc = up(mw.q_lat, torch.bfloat16, dev), up(mw.latent_cache, torch.bfloat16, dev)
        mbt = torch.from_numpy(mw.block_tables).to(dev)
        mcl = torch.from_numpy(mw.context_lens).to(dev)
        mout = torch.empty((mw.num_seqs, H, 512), dtype=torch.bfloat16, device=dev)
        mws = pa.mla_decode_workspace(mw.num_seqs, H, mw.max_context_len, device=dev)
        attn = lambda: pa.pa_mla_decode_attention(mout, mq, mc, mbt, mcl, mw.scale,
                                                  mw.max_context_len, mws)
        med, _ = timed_loop(attn, iters, 3, dev)
        nbytes, flops = wl.mla_bytes_read(mw), wl.mla_flops(mw)
        rec = {"kernel": "tcgen05 2-CTA cluster" if H % 128 == 0 else
               ("tcgen05 tokens on M" if H % 64 else "mma.sync"),
               "tokens_attended_per_s": round(int(mw.context_lens.sum()) / (med * 1e-3), 1),
               "GB_per_s": round(nbytes / (med * 1e-3) / 1e9, 2),
               "frac_of_hbm_peak": round(nbytes / (med * 1e-3) / 1e9 / peak, 4),
               "TFLOP_per_s": round(flops / (med * 1e-3) / 1e12, 2),
               "frac_of_bf16_dense_peak": round(flops / (med * 1e-3) / 1e12 / bf16_peak(), 4),
               "median_us": round(med * 1e3, 2), "algorithmic_bytes": nbytes, "flops": flops}
        if H == 128:
            qn, qp = up(mw.q_nope, torch.bfloat16, dev), up(mw.q_pe, torch.bfloat16, dev)
            wuk, wuv = up(mw.w_uk, torch.bfloat16, dev), up(mw.w_uv, torch.bfloat16, dev)
            qlat = torch.empty_like(mq)
            o = torch.empty((mw.num_seqs, H, 128), dtype=torch.bfloat16, device=dev)
            a_med, _ = timed_loop(lambda: pa.pa_mla_absorb_q(qlat, qn, qp, wuk), iters, 3, dev)
            p_med, _ = timed_loop(lambda: pa.pa_mla_project_out(o, mout, wuv), iters, 3, dev)

            def chain():
                pa.pa_mla_absorb_q(qlat, qn, qp, wuk)
                pa.pa_mla_decode_attention(mout, qlat, mc, mbt, mcl, mw.scale,
                                           mw.max_context_len, mws)
                pa.pa_mla_project_out(o, mout, wuv)
            c_med, _ = timed_loop(chain, iters, 3, dev)
            rec.update({"absorb_q_us": round(a_med * 1e3, 2),
                        "project_out_us": round(p_med * 1e3, 2),
                        "chain_us": round(c_med * 1e3, 2),
                        "chain_seqs_per_s": round(mw.num_seqs / (c_med * 1e-3), 1)})
        ex[mw.name] = rec
    return ex


# ------------------------------------------------------ oracle timings ----
def _oracle_decode_sample(w, rows, max_tokens=None):
    """Run the oracle on (b, h) rows (optionally on the first max_tokens of
    each context); return (seconds, algorithmic KV bytes of the sample)."""
    import oracle
    lens = w.context_lens.copy()
    if max_tokens is not None:
        lens = np.minimum(lens, max_tokens).astype(np.int32)
    fp8 = w.k_cache.dtype == np.uint8
    kw = (dict(cache_dtype=oracle.E4M3, k_scale=w.meta["k_scale"], v_scale=w.meta["v_scale"])
          if fp8 else {})
    t0 = time.perf_counter()
    for b, h in rows:
        oracle.paged_decode_row(w.q, w.k_cache, w.v_cache, w.block_tables, lens, b, h, w.scale,
                                **kw)
    dt = time.perf_counter() - t0
    G = w.num_q_heads // w.num_kv_heads
    kv_groups = {(b, h // G) for b, h in rows}
    nbytes = sum(int(lens[b]) * w.head_size * (1 if fp8 else 2) * 2 for b, _ in kv_groups)
    return dt, nbytes


def host_cpu():
    """The host's CPU model (from /proc/cpuinfo; Arm cores report an
    implementer and part number instead of a name) and its core count."""
    model = None
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
        for key in ("model name", "Model", "CPU part"):
            for line in info.splitlines():
                if line.split(":")[0].strip() == key:
                    model = line.split(":", 1)[1].strip()
                    break
            if model:
                if key == "CPU part":
                    model = f"{platform.machine()} CPU part {model}"
                break
    except OSError:
        pass
    return {"cpu_model": model or platform.machine(), "nproc": os.cpu_count()}


def cpu_baseline(w, budget_s=15.0):
    """The oracle (single-threaded C, double precision) on sequence 0's
    query heads, as many KV-head groups as fit in about budget_s."""
    G = w.num_q_heads // w.num_kv_heads
    rows, spent, nbytes = [], 0.0, 0
    for g in range(w.num_kv_heads):
        grp = [(0, g * G + i) for i in range(G)]
        dt, nb = _oracle_decode_sample(w, grp)
        spent += dt
        nbytes += nb
        rows += grp
        if spent > budget_s:
            break
    return {"value": round(nbytes / spent / 1e9, 4), "unit": "GB/s", "cores": 1,
            "kind": "oracle", **host_cpu(),
            "sample": f"sequence 0 (context {int(w.context_lens[0])}), {len(rows)} query heads "
                      f"({len(rows) // G} KV heads), {spent:.1f} s"}


def run_reference(args):
    """The reference arm: the CPU oracle timed on the same workload, each
    step a bounded sample (one query-head group of one sequence, its context
    truncated so the whole run takes about two minutes)."""
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    from paged_kv_cache_309_gb300 import workloads as wl
    import oracle
    oracle.build()
    w = wl.long_context_decode(block_size=args.block_size)
    G = w.num_q_heads // w.num_kv_heads
    # calibrate the oracle's speed on one group, then size the per-step sample
    dt, nb = _oracle_decode_sample(w, [(0, i) for i in range(G)], max_tokens=4096)
    per_token = dt / 4096
    budget = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(max(64, min(int(w.context_lens.min()), budget / per_token)))
    steps_t = []
    for i in range(args.warmup + args.steps):
        b = i % w.num_seqs
        g = (i // w.num_seqs) % w.num_kv_heads
        dt, nb = _oracle_decode_sample(w, [(b, g * G + j) for j in range(G)], max_tokens=tokens)
        if i >= args.warmup:
            steps_t.append((dt, nb))
    tot_t = sum(t for t, _ in steps_t)
    tot_b = sum(b for _, b in steps_t)
    val = tot_b / tot_t / 1e9
    line = {"impl": "reference",
            "metric": "paged decode-attn KV GB/s (% of HBM peak); cache-write tokens/s",
            "value": round(val, 4), "unit": "GB/s", "n_gpus": ws_n, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(1e3 * tot_t / len(steps_t), 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,1) bf16, shuffled block pool)",
            "config": {"workload": w.name, "num_seqs": w.num_seqs, "num_q_heads": w.num_q_heads,
                       "num_kv_heads": w.num_kv_heads, "head_size": w.head_size,
                       "block_size": w.block_size},
            "cpu_baseline": {"value": round(val, 4), "unit": "GB/s", "cores": 1,
                             "kind": "oracle", **host_cpu(),
                             "sample": f"per step: one KV-head group ({G} query heads) of one "
                                       f"sequence over its first {tokens} tokens"},
            "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_mla_only(args):
    """MLA decode attention launches only (for an ncu capture of that kernel)."""
    import torch

    from paged_kv_cache_309_gb300 import build, pa
    from paged_kv_cache_309_gb300 import workloads as wl
    build.build()
    dev = torch.device("cuda", 0)
    w = wl.mla_decode(num_heads=args.mla_heads, with_weights=False)
    q, c = up(w.q_lat, torch.bfloat16, dev), up(w.latent_cache, torch.bfloat16, dev)
    bt, cl = torch.from_numpy(w.block_tables).to(dev), torch.from_numpy(w.context_lens).to(dev)
    out = torch.empty((w.num_seqs, w.num_heads, 512), dtype=torch.bfloat16, device=dev)
    ws = pa.mla_decode_workspace(w.num_seqs, w.num_heads, w.max_context_len, device=dev)
    pa.pa_mla_decode_attention(out, q, c, bt, cl, w.scale, w.max_context_len, ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps - 1):
        pa.pa_mla_decode_attention(out, q, c, bt, cl, w.scale, w.max_context_len, ws)
    e1.record()
    torch.cuda.synchronize()
    per = e0.elapsed_time(e1) / max(1, args.steps - 1)
    print(f"{w.name}: {args.steps} launches, {per * 1e3:.1f} us per launch (back to back), "
          f"device error word {pa.read_device_error(ws)}")


def run_proj_only(args):
    """MLA projection launches only (for an ncu capture of those kernels):
    --steps absorb launches, then --steps project launches, at B=64, 128
    heads; prints back-to-back and L2-flushed times."""
    import torch

    from paged_kv_cache_309_gb300 import build, pa
    from paged_kv_cache_309_gb300 import workloads as wl
    build.build()
    dev = torch.device("cuda", 0)
    w = wl.mla_decode(num_heads=128, with_weights=True)
    qn, qp = up(w.q_nope, torch.bfloat16, dev), up(w.q_pe, torch.bfloat16, dev)
    wuk, wuv = up(w.w_uk, torch.bfloat16, dev), up(w.w_uv, torch.bfloat16, dev)
    qlat = torch.empty((w.num_seqs, 128, 576), dtype=torch.bfloat16, device=dev)
    olat = torch.randn((w.num_seqs, 128, 512), device=dev).to(torch.bfloat16)
    out = torch.empty((w.num_seqs, 128, 128), dtype=torch.bfloat16, device=dev)
    for name, fn in (("absorb", lambda: pa.pa_mla_absorb_q(qlat, qn, qp, wuk)),
                     ("project", lambda: pa.pa_mla_project_out(out, olat, wuv))):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps - 1):
            fn()
        e1.record()
        torch.cuda.synchronize()
        per = e0.elapsed_time(e1) / max(1, args.steps - 1)
        med, _ = timed_loop(fn, max(3, args.steps), 2, dev)
        print(f"{name}: {args.steps} launches, {per * 1e3:.2f} us per launch back to back, "
              f"{med * 1e3:.2f} us median with L2 flushed")


def run_prefill_only(args):
    """Causal prefill launches only (for an ncu capture of that kernel)."""
    import torch

    from paged_kv_cache_309_gb300 import build, pa
    from paged_kv_cache_309_gb300 import workloads as wl
    build.build()
    dev = torch.device("cuda", 0)
    pw = wl.make_prefill("prefill_attention_b4_8k", 5, [8192] * 4, [8192] * 4, 32, 8, 128, 16)
    pq = up(pw.q, torch.bfloat16, dev)
    pout = torch.empty_like(pq)
    pkc, pvc = up(pw.k_cache, torch.bfloat16, dev), up(pw.v_cache, torch.bfloat16, dev)
    pbt, pcu = torch.from_numpy(pw.block_tables).to(dev), torch.from_numpy(pw.cu_seqlens_q).to(dev)
    pcl = torch.from_numpy(pw.context_lens).to(dev)
    perr = torch.zeros(1, dtype=torch.int32, device=dev)
    pa.pa_paged_prefill_attention(pout, pq, pkc, pvc, pbt, pcu, pcl, pw.scale, pw.max_q_len, perr)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps - 1):
        pa.pa_paged_prefill_attention(pout, pq, pkc, pvc, pbt, pcu, pcl, pw.scale, pw.max_q_len,
                                      perr)
    e1.record()
    torch.cuda.synchronize()
    per = e0.elapsed_time(e1) / max(1, args.steps - 1)
    tf = wl.prefill_flops(pw) / (per * 1e-3) / 1e12
    print(f"{pw.name}: {args.steps} launches, {per * 1e3:.1f} us per launch (back to back, "
          f"{tf:.1f} TFLOP/s), device error word {int(perr.item())}")


def run_write_only(args):
    """Cache-write launches only (for an ncu capture of those kernels):
    --steps launches each of the 32K-token prefill write to an e4m3 cache
    (scale 0.05), to a bf16 cache, to an e4m3 cache through the SWA table
    (window 4096), then of the 16K-token MLA latent-cache write."""
    import torch

    from paged_kv_cache_309_gb300 import build, pa
    from paged_kv_cache_309_gb300 import workloads as wl
    build.build()
    dev = torch.device("cuda", 0)

    def run(name, fn, nbytes):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps - 1):
            fn()
        e1.record()
        torch.cuda.synchronize()
        per = e0.elapsed_time(e1) / max(1, args.steps - 1)
        print(f"{name}: {args.steps} launches, {per * 1e3:.1f} us per launch (back to back, "
              f"{nbytes / (per * 1e-3) / 1e9:.0f} GB/s)")

    for variant in ("e4m3", "bf16", "e4m3_swa"):
        w = wl.prefill_write(variant=variant)
        H, d = w.key.shape[1:]
        cdt = torch.float8_e4m3fn if w.cache_dtype == "e4m3" else torch.bfloat16
        kc = torch.zeros((w.num_blocks, w.block_size, H, d), dtype=cdt, device=dev)
        vc = torch.zeros_like(kc)
        key, val = up(w.key, torch.bfloat16, dev), up(w.value, torch.bfloat16, dev)
        sl = torch.from_numpy(w.slot_mapping).to(dev)
        swa = None if w.swa_slot_mapping is None else torch.from_numpy(w.swa_slot_mapping).to(dev)
        ks = None if w.k_scale is None else torch.tensor([w.k_scale], dtype=torch.float32,
                                                         device=dev)
        vs = None if ks is None else ks.clone()
        run(w.name, lambda: pa.pa_reshape_and_cache(key, val, kc, vc, sl, swa, ks, vs),
            wl.write_bytes(w))
    m = wl.mla_assembly()
    N = m.c_kv.shape[0]
    ckv, kpe = up(m.c_kv, torch.bfloat16, dev), up(m.k_pe, torch.bfloat16, dev)
    cache = torch.zeros((m.num_blocks, m.block_size, 1, 576), dtype=torch.bfloat16, device=dev)
    msl = torch.from_numpy(m.slot_mapping).to(dev)
    run("mla_latent_cache_write_16k", lambda: pa.pa_concat_and_cache_mla(ckv, kpe, cache, msl),
        N * (576 * 2 * 2 + 8))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--block-size", type=int, default=16)
    ap.add_argument("--step", choices=["fused", "two-call"], default="fused",
                    help="decode step as one launch (pa_paged_decode_step) or write + attention")
    ap.add_argument("--kv-dtype", choices=["bf16", "e4m3"], default="bf16",
                    help="KV cache format of the decode step (e4m3: fp8 with scales)")
    ap.add_argument("--num-seqs", type=int, default=8,
                    help="sequences of the long-context workload (8; fewer for profiling)")
    ap.add_argument("--extra-iters", type=int, default=50)
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-only", action="store_true",
                    help="profiling aid: only run --steps causal prefill launches on the "
                         "4 x 8192-token workload (no JSON)")
    ap.add_argument("--write-only", action="store_true",
                    help="profiling aid: only run --steps cache-write launches of the 32K-token "
                         "prefill write (e4m3, bf16, e4m3 through the SWA table), then of the "
                         "16K-token MLA latent-cache write (no JSON)")
    ap.add_argument("--mla-proj", action="store_true",
                    help="profiling aid: only run --steps MLA absorb then project launches "
                         "(B=64, 128 heads; no JSON)")
    ap.add_argument("--mla-heads", type=int, default=0,
                    help="profiling aid: only run --steps MLA decode attention launches on the "
                         "B=64 context 512..4096 latent workload with this many heads (no JSON)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.mla_heads:
        run_mla_only(args)
        return
    if args.mla_proj:
        run_proj_only(args)
        return
    if args.prefill_only:
        run_prefill_only(args)
        return
    if args.write_only:
        run_write_only(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
