#!/usr/bin/env python
"""Benchmark of the LoRA-KV attention hot path on B300.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config all|NAME]
                  [--impl lrkv|reference] [--no-bk]

One step = one pass of the hot path over one batch of a workload, inputs
already resident in HBM: for the decode workloads the decode call; for the
prefill workload the append of the new chunk tokens plus the causal prefill;
for the mixed batch the append, then the decode and the prefill in one
``lrkv_attn_mixed`` call (the two run concurrently); its decode and prefill are
also timed alone, in a second loop, for their rooflines. With ``--config all`` (the
default) every bf16 workload is timed in turn in one process and reported under
``workloads.<name>``; the line's headline fields (value, roofline, e2e,
cpu_baseline) are those of the shared-context decode (Llama-3.1-8B-shaped
layer, 4 agents on one 8192-token context, rank 16), and ``prefill`` carries the
prefill kernel's TFLOP/s against the burst and the sustained bf16 peak.

Timing: L2 is flushed (a 512 MiB write) before every step, outside the timed
events; each part of the step is captured once into a CUDA graph (the same
library calls, the same kernels) and replayed, each replay bracketed by CUDA
events on the launching stream; the K steps are bracketed by a barrier and a
device synchronize, and the step time is the max over ranks. The e2e figure
calls the public API directly: per step one host-to-device copy of the step's
packed inputs from pinned memory, the library calls, one device-to-host copy
of the packed outputs. Under torchrun each rank holds its own disjoint share
of the contexts (weak scaling; no collective on the data path). Rank 0 prints
one JSON line. ``--impl reference`` times the fp64 CPU oracle instead (on the
host cores, rank 0 only). ``--no-bk`` runs attention with B_K = NULL (no K
adapter term, no rebuild): a diagnostic of the rebuild's cost, marked as such.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_CONFIG = "all"
ALL_WORKLOADS = ["shared_decode_llama8b", "prefill_chunk_llama8b", "long_decode_ministral8b",
                 "long_decode_codec_ministral8b", "prefill_chunk_codec_llama8b",
                 "mixed_batch_qwen3_1p7b", "prelr_decode_llama8b", "rebase_prefill_llama8b"]
HEADLINE = "shared_decode_llama8b"
PREFILL_HEADLINE = "prefill_chunk_llama8b"
METRIC = "LoRA-KV attention decode tok/s & GB/s (% of HBM), prefill TFLOP/s (% peak)"
FLUSH_BYTES = 512 << 20
KERNEL_SOURCES = {"decode": ["decode.cu", "lrkv_device.cuh", "tcgen05.cuh"],
                  "prefill": ["prefill.cu", "lrkv_device.cuh", "tcgen05.cuh"],
                  "append": ["append.cu", "lrkv_device.cuh", "tcgen05.cuh"]}


# ----------------------------------------------------------------- helpers
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


def kernel_sha(kind: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kind]:
        h.update(open(os.path.join(ROOT, "rank_cache_attention_flash_b300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def committed_traffic(workload: str, kind: str):
    """Per-launch DRAM bytes (read + write) of this part's kernel from a committed
    ncu capture, if the kernel's sources are unchanged since; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path)).get(workload, {}).get(kind)
    if not d or d.get("source_sha") != kernel_sha(kind):
        return None
    return d.get("dram_bytes_per_launch")


def workload_model(case):
    """Algorithmic bytes and flops of each call of one step (units: bytes, flop)."""
    sh = case.shape
    es = 4 if sh.dtype == "fp32" else 2
    D, R, Hkv, Hq = sh.head_dim, sh.rank, sh.n_kv_heads, sh.n_q_heads
    out = {}
    if case.dec_q.shape[0]:
        qs = case.dec_q_start.tolist()
        nbytes = flops = 0
        for c, s in enumerate(case.dec_ctx):
            L = case.seqs[s].total_len
            ads = case.dec_adapter[qs[c]:qs[c + 1]].tolist()
            rows = len(ads) * (Hq // Hkv)
            distinct = len({a for a in ads if a >= 0})
            # low-rank groups read: one (shared A), or each reading agent's own (agent-specific A)
            groups = max(1, distinct) if sh.lr_groups > 1 else 1
            # base part per token and kv head: K and V planes, or one compressed
            # chunk row (q8_0 keys, 3-bit values: (23 d + 64) / 16 bytes)
            base_tok = Hkv * (23 * D + 64) // 16 if sh.kv_codec else Hkv * D * 2 * es
            nbytes += L * (base_tok + 2 * R * groups * es)
            nbytes += distinct * 2 * R * Hkv * D * es
            nbytes += len(ads) * Hq * D * es * 2
            flops += L * Hkv * (distinct * 2 * R * D + rows * (4 * D + 2 * R))
            flops += len([a for a in ads if a >= 0]) * Hq * 2 * R * D
        out["decode"] = {"bytes": nbytes, "flops": flops, "units": int(case.dec_q.shape[0]),
                         "unit_name": "query tokens"}
    if case.pre_seq:
        qs = case.pre_q_start.tolist()
        pairs = 0
        nbytes = flops = 0
        for p, s in enumerate(case.pre_seq):
            L = case.seqs[s].total_len
            n = qs[p + 1] - qs[p]
            vis = n * (L - n) + n * (n + 1) // 2  # visible (query, key) pairs
            pairs += vis
            flops += Hq * vis * (4 * D + 2 * R)          # QK^T + PV + P L_V
            flops += Hkv * L * 2 * R * D                  # K rebuild (once per key)
            flops += n * Hq * 2 * R * D                   # O_lr B_V
            base_tok = Hkv * (23 * D + 64) // 16 if sh.kv_codec else Hkv * D * 2 * es
            nbytes += L * (base_tok + 2 * R * es) + 2 * n * Hq * D * es
        out["prefill"] = {"bytes": nbytes, "flops": flops, "units": int(qs[-1]),
                          "unit_name": "prefill tokens", "pairs": pairs}
    T = sum(b - a for _, a, b in case.step_appends())
    if T:
        N = 2 * Hkv * D + 2 * sh.lr_groups * R
        n_src = 2 if case.rebase else 1  # a re-based append reads two sets of hidden states
        out["append"] = {"bytes": (n_src * T * sh.hidden + N * sh.hidden + T * N) * es,
                         "flops": 2 * T * sh.hidden * N, "units": T, "unit_name": "appended tokens"}
    return out


class ClockSampler:
    """Samples the SM clock and clock-event reasons while running (read only):
    through NVML when the Python binding is present, else by running
    ``nvidia-smi --query-gpu ... -lms`` for the duration of the region."""

    FIELDS = ["clocks.sm", "clocks.max.sm", "clocks_event_reasons.hw_slowdown",
              "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
              "clocks_event_reasons.sw_power_cap"]
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int, interval_ms: int = 20):
        self.samples, self.reasons, self.max_mhz, self.error = [], set(), None, None
        self.interval = interval_ms
        self._stop = threading.Event()
        self._h = None
        self._proc = None
        self._bus = None
        try:
            import torch

            p = torch.cuda.get_device_properties(device_index)
            self._bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
        except Exception as e:
            self.error = f"bus id: {type(e).__name__}: {e}"
        try:
            import pynvml

            pynvml.nvmlInit()
            self._nv = pynvml
            self._h = (pynvml.nvmlDeviceGetHandleByPciBusId(self._bus.encode()) if self._bus
                       else pynvml.nvmlDeviceGetHandleByIndex(device_index))
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
        except Exception:
            self._h = None

    def _run(self):
        nv = self._nv
        reasons = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(nv, "nvmlDeviceGetCurrentClocksThrottleReasons")
        while not self._stop.is_set():
            try:
                self.samples.append(nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM))
                r = reasons(self._h)
                for bit, name in self.REASONS.items():
                    if r & bit:
                        self.reasons.add(name)
            except Exception as e:
                self.error = f"{type(e).__name__}: {e}"
            time.sleep(self.interval / 1e3)

    def __enter__(self):
        if self._h is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        else:
            import subprocess

            cmd = ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS), "--format=csv,noheader,nounits",
                   "-lms", str(self.interval)]
            if self._bus:
                cmd += ["-i", self._bus]
            try:
                self._proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
                time.sleep(0.2)  # let the first samples arrive before the region starts
            except Exception as e:
                self.error = f"nvidia-smi: {type(e).__name__}: {e}"
        return self

    def __exit__(self, *a):
        self._stop.set()
        if self._h is not None:
            self._t.join()
        elif self._proc is not None:
            time.sleep(0.05)
            self._proc.terminate()
            try:
                out, err = self._proc.communicate(timeout=5)
            except Exception:
                self._proc.kill()
                out, err = self._proc.communicate()
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            for line in out.splitlines():
                f = [x.strip() for x in line.split(",")]
                if len(f) != len(self.FIELDS):
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for name, v in zip(names, f[2:]):
                    if v.lower().startswith("active"):
                        self.reasons.add(name)
            if not self.samples:
                self.error = (err or "no samples").strip()[:200]

    def summary(self):
        med = statistics.median(self.samples) if self.samples else None
        out = {"sm_mhz": med, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
               "samples": len(self.samples)}
        if self.error and not self.samples:
            out["error"] = self.error
        return out


def reduce_step_time(total_ms_local: float, steps: int, world: int, device=None) -> float:
    """Per-step time of the whole job: the max over ranks of each rank's summed
    step time, divided by the step count (torch.distributed, any backend)."""
    import torch

    t = torch.tensor([total_ms_local], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist

        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item()) / steps


def job_throughput(units_per_rank: float, world: int, ms_per_step: float) -> float:
    """Units processed by all ranks per second (weak scaling: each rank its own replica)."""
    return world * units_per_rank / (ms_per_step / 1e3)


def oracle_threads() -> int:
    try:
        from threadpoolctl import threadpool_info

        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("internal_api") in ("openblas", "mkl", "blis")]
        if n:
            return max(n)
    except Exception:
        pass
    return len(os.sched_getaffinity(0))


# ----------------------------------------------------------- oracle timing
def oracle_sample(case, budget_s: float, model):
    """Times the fp64 oracle on a bounded sample of the workload. Returns
    (value, unit, seconds, description). Decode workloads: whole queries over
    their full context while the budget lasts (at least one query, or one query
    over a leading fraction of its context when even one exceeds the budget);
    prefill workloads: one sequence's chunk rows over the full context."""
    import numpy as np

    import oracle
    from oracle import polykv
    from tests.parity import _hidden, weights64

    sh = case.shape
    w64 = weights64(case)
    scale = 1.0 / math.sqrt(sh.head_dim)
    if "decode" in model and "prefill" not in model:
        qs = case.dec_q_start.tolist()
        done = 0.0
        t0 = time.perf_counter()
        n_full = 0
        for r in range(case.dec_q.shape[0]):
            c = next(i for i in range(len(case.dec_ctx)) if qs[i] <= r < qs[i + 1])
            L_full = case.seqs[case.dec_ctx[c]].total_len
            X, X_lr = _hidden(case, case.dec_ctx[c])
            if sh.kv_codec:
                polykv.decode_codec(X, case.dec_q[r:r + 1].double().numpy(), case.dec_adapter[r:r + 1].numpy(),
                                    w64, sh.n_kv_heads, sh.head_dim, sh.rope_base, scale)
            else:
                oracle.decode(X, case.dec_q[r:r + 1].double().numpy(), case.dec_adapter[r:r + 1].numpy(),
                              w64, sh.n_kv_heads, sh.head_dim, sh.rope_base, scale, X_lr=X_lr)
            done += 1.0
            n_full += 1
            if time.perf_counter() - t0 > budget_s:
                break
        dt = time.perf_counter() - t0
        return done / dt, "tok/s", dt, f"{n_full} decode queries over their full {L_full}-token contexts"
    if "prefill" in model and "decode" not in model:
        p = 0
        s = case.pre_seq[p]
        a, b = int(case.pre_q_start[p]), int(case.pre_q_start[p + 1])
        n = b - a
        rows = list(range(0, n, max(1, n // 16)))
        X, X_lr = _hidden(case, s)
        L = X.shape[0]
        t0 = time.perf_counter()
        oracle.attend(X, int(case.pre_adapter[p]), case.pre_q[a:b][rows].double().numpy(),
                      np.array([L - n + k for k in rows]), w64, sh.n_kv_heads, sh.head_dim, sh.rope_base, scale,
                      X_lr=X_lr)
        dt = time.perf_counter() - t0
        vis = sum(L - n + k + 1 for k in rows)
        fl = sh.n_q_heads * vis * (4 * sh.head_dim + 2 * sh.rank)
        return fl / dt / 1e12, "TFLOP/s", dt, f"{len(rows)} prefill rows of sequence 0 over {L} keys"
    # mixed: one decode query and one prefill sequence's sampled rows, in tokens/s
    t0 = time.perf_counter()
    c = 0
    X, X_lr = _hidden(case, case.dec_ctx[c])
    oracle.decode(X, case.dec_q[0:1].double().numpy(), case.dec_adapter[0:1].numpy(), w64, sh.n_kv_heads,
                  sh.head_dim, sh.rope_base, scale, X_lr=X_lr)
    p = 0
    s = case.pre_seq[p]
    a, b = int(case.pre_q_start[p]), int(case.pre_q_start[p + 1])
    X, X_lr = _hidden(case, s)
    oracle.prefill(X, case.pre_q[a:b].double().numpy(), int(case.pre_adapter[p]), w64, sh.n_kv_heads,
                   sh.head_dim, sh.rope_base, scale, X_lr=X_lr)
    dt = time.perf_counter() - t0
    return (1 + (b - a)) / dt, "tok/s", dt, f"1 decode query + 1 prefill chunk of {b - a} tokens"


def run_reference(args):
    """The base contract's reference arm: the fp64 CPU oracle as it stands."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from rank_cache_attention_flash_b300 import inputs as I

    config = HEADLINE if args.config == "all" else args.config
    case = I.FULL[config]()
    model = workload_model(case)
    budget = max(0.05, 150.0 / max(1, args.steps + args.warmup))
    # per-step sample: one query (or chunk rows) over a leading fraction of its
    # context, sized to the per-step budget; throughput in full-query units
    import numpy as np

    import oracle
    from oracle import polykv
    from tests.parity import _hidden, weights64

    sh = case.shape
    w64 = weights64(case)
    scale = 1.0 / math.sqrt(sh.head_dim)
    decode_like = "decode" in model and "prefill" not in model
    if decode_like:
        s = case.dec_ctx[0]
        L_full = case.seqs[s].total_len
        X_full, X_lr = _hidden(case, s)
        q = case.dec_q[0:1].double().numpy()
        ad = case.dec_adapter[0:1].numpy()

        def one(nt):
            if sh.kv_codec:
                polykv.decode_codec(X_full[:nt], q, ad, w64, sh.n_kv_heads, sh.head_dim, sh.rope_base, scale)
            else:
                oracle.decode(X_full[:nt], q, ad, w64, sh.n_kv_heads, sh.head_dim, sh.rope_base, scale,
                              X_lr=None if X_lr is None else X_lr[:nt])
    else:
        p = 0
        s = case.pre_seq[p]
        a, b = int(case.pre_q_start[p]), int(case.pre_q_start[p + 1])
        X_full, X_lr = _hidden(case, s)
        L_full = X_full.shape[0]
        qrow = case.pre_q[b - 1:b].double().numpy()

        def one(nt):
            oracle.attend(X_full[:nt], int(case.pre_adapter[p]), qrow, [nt - 1], w64, sh.n_kv_heads,
                          sh.head_dim, sh.rope_base, scale, X_lr=None if X_lr is None else X_lr[:nt])
    # calibrate tokens per step
    nt = min(L_full, 256)
    t0 = time.perf_counter()
    one(nt)
    per_tok = (time.perf_counter() - t0) / nt
    nt = int(max(16, min(L_full, budget / max(per_tok, 1e-9))))
    for _ in range(args.warmup):
        one(nt)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one(nt)
    dt = time.perf_counter() - t0
    units = args.steps * nt / L_full  # fractions of one full query
    value = units / dt
    cores = oracle_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": config},
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": f"per step: one query over the leading {nt} of its {L_full} keys "
                                       f"(counted as {nt}/{L_full} of a query)"},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- main
# Kernels of this library that one call of each part launches (bf16 path).
LAUNCHES_PER_CALL = {"append": 1, "decode": 2, "prefill": 1}


def cache_bytes(case):
    """LRKV cache bytes vs per-agent full caches over the decode contexts."""
    sh = case.shape
    es = 4 if sh.dtype == "fp32" else 2
    lr = full = 0
    if case.dec_q.shape[0]:
        qs = case.dec_q_start.tolist()
        for c, s in enumerate(case.dec_ctx):
            L = case.seqs[s].total_len
            readers = qs[c + 1] - qs[c]
            full += readers * L * sh.n_kv_heads * sh.head_dim * 2 * es
            base = sh.n_kv_heads * (23 * sh.head_dim + 64) // 16 if sh.kv_codec else sh.n_kv_heads * sh.head_dim * 2 * es
            lr += L * (base + 2 * sh.lr_groups * sh.rank * es)
    return {"lrkv": lr, "per_agent_full": full, "saving": full / lr} if full else None


def time_workload(name, args, world, rank, dev, pk):
    """Times one workload on this rank. Returns its report entry."""
    import torch

    from rank_cache_attention_flash_b300 import inputs as I
    from rank_cache_attention_flash_b300.harness import GpuCase

    case = I.build_shard(name, world, rank)
    model = workload_model(case)
    g = GpuCase(case, device=dev, no_bk=args.no_bk)
    g.setup()
    if "prefill" in model and "append" in model and "decode" not in model:
        kinds = ["append", "prefill"]
    else:
        kinds = [k for k in ("append", "decode", "prefill") if k in model]
    dominant = "decode" if "decode" in model else "prefill"
    stream = torch.cuda.current_stream(dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    calls = {"append": g.step_append, "decode": g.decode, "prefill": g.prefill, "mixed": g.mixed}
    # a step with both decode and prefill makes them one mixed call
    mixed = "decode" in kinds and "prefill" in kinds
    step_kinds = [k for k in kinds if not (mixed and k in ("decode", "prefill"))] + (["mixed"] if mixed else [])
    alone = ["decode", "prefill"] if mixed else []

    for i in range(args.warmup):
        flush.fill_(i & 0xFF)
        for k in step_kinds + alone:
            calls[k]()
    torch.cuda.synchronize()
    # Each part of the step is captured once into a CUDA graph and replayed in
    # the timed loop: the replay keeps host launch latency out of the device
    # timings (the kernels and their arguments are exactly the API call's).
    graphs = {}
    for k in step_kinds + alone:
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            calls[k]()
        graphs[k] = gr
    for i in range(3):
        flush.fill_(i & 0xFF)
        for k in step_kinds + alone:
            graphs[k].replay()
    torch.cuda.synchronize()
    K = args.steps
    evs = [{k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for k in step_kinds + alone} for _ in range(K)]
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    if world > 1:
        import torch.distributed as dist

        dist.barrier()
    torch.cuda.synchronize()
    host_t0 = time.perf_counter()
    with ClockSampler(dev.index) as clk:
        for i in range(K):
            flush.fill_(i & 0xFF)
            step_ev[i][0].record(stream)
            for k in step_kinds:
                evs[i][k][0].record(stream)
                graphs[k].replay()
                evs[i][k][1].record(stream)
            step_ev[i][1].record(stream)
        torch.cuda.synchronize()
        host_dt = time.perf_counter() - host_t0
        # the mixed call's two parts alone (each after its own flush), for
        # their rooflines; not part of the step time
        for i in range(K if alone else 0):
            for k in alone:
                flush.fill_(i & 0xFF)
                evs[i][k][0].record(stream)
                graphs[k].replay()
                evs[i][k][1].record(stream)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    part_ms = {k: sum(e[k][0].elapsed_time(e[k][1]) for e in evs) / K for k in step_kinds + alone}
    ms_per_step = reduce_step_time(sum(step_ms), K, world, dev)
    status = g.device_status()
    del graphs

    # ---- end to end through the public API: one packed copy in, one out
    # (the host enqueues each step while the GPU runs it: Python's garbage
    # collector stays off in this loop so a collection pause is not timed)
    import gc

    e_ms = []
    n_e2e = min(args.e2e_steps, 50 if dominant == "prefill" or len(kinds) > 1 else args.e2e_steps)
    gc.collect()
    gc.disable()
    for i in range(n_e2e + 3):
        flush.fill_(i & 0xFF)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        g.upload_inputs()
        for k in step_kinds:
            calls[k]()
        g.download_outputs()
        b.record(stream)
        b.synchronize()
        if i >= 3:
            e_ms.append(a.elapsed_time(b))
    gc.enable()
    e2e_ms = reduce_step_time(sum(e_ms), len(e_ms), world, dev)

    if dominant == "decode" and "prefill" not in model:
        unit = "tok/s"
        work = model["decode"]["units"]
    elif "decode" not in model:
        unit = "TFLOP/s"
        work = (model["prefill"]["flops"] + model.get("append", {"flops": 0})["flops"]) / 1e12
    else:
        unit = "tok/s"
        work = model["decode"]["units"] + model["prefill"]["units"]
    value = job_throughput(work, world, ms_per_step)
    e2e = {"value": job_throughput(work, world, e2e_ms), "unit": unit, "h2d_bytes_per_step": g.h2d_bytes,
           "d2h_bytes_per_step": g.d2h_bytes, "ms_per_step": e2e_ms, "ms_median": statistics.median(e_ms),
           "copies_per_step": {"h2d": 1, "d2h": 1}}

    parts = {}
    for k in kinds:
        ms = part_ms[k]
        m = model[k]
        parts[k] = {"ms": ms, "GB/s": m["bytes"] / (ms / 1e3) / 1e9, "TFLOP/s": m["flops"] / (ms / 1e3) / 1e12,
                    m["unit_name"]: m["units"]}
        parts[k]["frac_hbm"] = parts[k]["GB/s"] / pk["hbm_gbs"]
        parts[k]["frac_tensor"] = parts[k]["TFLOP/s"] / pk["bf16_tflops"]
        if pk.get("bf16_tflops_sustained"):
            parts[k]["frac_tensor_sustained"] = parts[k]["TFLOP/s"] / pk["bf16_tflops_sustained"]
        parts[k]["roofline"] = part_roofline(k, name, m, ms, pk)
    if mixed:
        parts["mixed"] = {"ms": part_ms["mixed"], "decode_and_prefill_alone_ms": part_ms["decode"] + part_ms["prefill"],
                          "note": "the step's decode and prefill in one lrkv_attn_mixed call, run concurrently; "
                                  "the decode and prefill entries are the same calls timed alone"}
    roof = parts[dominant]["roofline"]
    sh = case.shape
    entry = {
        "workload": name, "value": value, "unit": unit, "ms_per_step": ms_per_step, "steps": K,
        "dtype": "bf16" if sh.dtype == "bf16" else "fp32",
        "config": {"workload": name, "hidden": sh.hidden, "n_q_heads": sh.n_q_heads,
                   "n_kv_heads": sh.n_kv_heads, "head_dim": sh.head_dim, "rank": sh.rank,
                   "n_adapters": sh.n_adapters, "contexts": len(case.seqs),
                   "max_len": max(q.total_len for q in case.seqs),
                   "l2": f"flushed before every step ({FLUSH_BYTES >> 20} MiB write)",
                   "parallelism": f"weak x{world}: rank {rank} holds its own share of the contexts"},
        "roofline": roof, "parts": parts, "e2e": e2e,
        "gpu_launches": K * sum(LAUNCHES_PER_CALL[k] for k in kinds),
        **({"gpu_launches_parts_alone": K * sum(LAUNCHES_PER_CALL[k] for k in alone)} if alone else {}),
        "clocks": clk.summary(), "device_status": status, "host_s": host_dt,
    }
    if args.no_bk:
        entry["variant"] = "no_bk: attention without B_K (diagnostic, not the method's result)"
    cb = cache_bytes(case)
    if cb:
        entry["cache_bytes"] = cb
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, u, dt, desc = oracle_sample(case, args.cpu_budget, model)
        entry["cpu_baseline"] = {"value": v, "unit": u, "cores": oracle_threads(), "kind": "oracle",
                                 "sample": desc, "seconds": dt}
    del g, flush
    torch.cuda.empty_cache()
    return entry


def part_roofline(kind, workload, m, ms, pk):
    """Roofline of one part's kernel: bytes against HBM for decode, flops against
    the bf16 tensor peak for prefill and append (burst peak: each part is timed
    on its own, a fraction of a millisecond to a few milliseconds long)."""
    if kind == "decode":
        achieved = m["bytes"] / (ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"], "peak_source": pk["source"],
                "kernel": "lrkv_attn_decode (decode_kernel + combine_kernel)",
                "algorithmic_bytes_per_launch": m["bytes"], "launch_ms": ms,
                "traffic": committed_traffic(workload, "decode")}
    achieved = m["flops"] / (ms / 1e3) / 1e12
    r = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
         "frac": achieved / pk["bf16_tflops"], "peak_source": pk["source"] + " (burst)",
         "kernel": "lrkv_attn_prefill (prefill_kernel)" if kind == "prefill" else "lrkv_append (append kernel)",
         "algorithmic_flops_per_launch": m["flops"], "launch_ms": ms,
         "traffic": committed_traffic(workload, kind)}
    if pk.get("bf16_tflops_sustained"):
        r["frac_sustained"] = achieved / pk["bf16_tflops_sustained"]
    return r


def merge_clocks(entries):
    sums = [e["clocks"] for e in entries]
    med = [c["sm_mhz"] for c in sums if c.get("sm_mhz")]
    out = {"sm_mhz": statistics.median(med) if med else None,
           "sm_max_mhz": next((c["sm_max_mhz"] for c in sums if c.get("sm_max_mhz")), None),
           "reasons": sorted(set(r for c in sums for r in c.get("reasons", []))),
           "samples": sum(c.get("samples", 0) for c in sums)}
    errs = [c["error"] for c in sums if c.get("error")]
    if errs:
        out["error"] = errs[0]
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--config", default=DEFAULT_CONFIG, choices=["all"] + ALL_WORKLOADS + ["tiny_fp32_decode"])
    ap.add_argument("--impl", default="lrkv", choices=["lrkv", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0, help="seconds of oracle work per workload")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--no-bk", action="store_true", help="attention without B_K (diagnostic)")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist

    from rank_cache_attention_flash_b300 import lrkv

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lrkv.load()
    pk = peaks()

    names = ALL_WORKLOADS if args.config == "all" else [args.config]
    entries = {n: time_workload(n, args, world, rank, dev, pk) for n in names}
    head = entries[HEADLINE] if HEADLINE in entries else entries[names[0]]
    line = {
        "metric": METRIC, "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"], "data": "synthetic",
        "config": head["config"], "roofline": head["roofline"], "parts": head["parts"], "e2e": head["e2e"],
        "gpu_launches": sum(e["gpu_launches"] for e in entries.values()),
        "clocks": merge_clocks(list(entries.values())),
        "device_status": max(e["device_status"] for e in entries.values()),
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if "cache_bytes" in head:
        line["cache_bytes"] = head["cache_bytes"]
    if PREFILL_HEADLINE in entries:
        pr = entries[PREFILL_HEADLINE]["parts"]["prefill"]
        line["prefill"] = {"workload": PREFILL_HEADLINE, "TFLOP/s": pr["TFLOP/s"], "launch_ms": pr["ms"],
                           "frac_burst": pr["frac_tensor"], "frac_sustained": pr.get("frac_tensor_sustained"),
                           "peak_burst": pk["bf16_tflops"], "peak_sustained": pk.get("bf16_tflops_sustained")}
    if args.no_bk:
        line["variant"] = head.get("variant")
    if len(entries) > 1:
        line["workloads"] = entries
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
