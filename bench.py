"""Benchmark of the paged KV write + PagedAttention decode step on GB300.

One step = one pass of the whole hot path over one batch: the KV write of each
sequence's newest token (reshape_and_cache, one token per sequence), then the
decode of every sequence, split into 512-token partitions and merged when the
device's work-unit count calls for it (the library's own choice).

Default workload: the Llama-3-8B GQA decode (256 sequences, 32 query heads /
8 KV heads, head size 128, block size 16, bf16 KV, context lengths
log-uniform in [512, 4096], random block placement, seed 0x5EED0003).

Metric: KV GB/s = (logical K/V bytes read + Q + out + KV-write bytes) / step
time, on the device with inputs resident in HBM (1.8 GB of KV, far larger than
the 129 MB L2, so no flush is needed between steps). Also reported: decode
sequences per second per layer, the dominant kernel's roofline (the kernel
timed alone, graph-replayed for over a second, on method bytes), an
end-to-end figure through host buffers, the oracle timed on the host cores,
the SM clocks sampled during the timed region, and records of the other
four workloads (each step, its kernel alone, its own KV write; the
shared-prefix pool also with shared-prefix units).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config 1-5] [--form fused|separate|shared] [--configs LIST|none]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "paged-decode KV GB/s (fraction of GB300 HBM peak); decode seqs/sec per layer"
UNIT = "GB/s"
DEFAULT_CONFIG = 3
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "decode_partitions_llama3_8b_traffic.txt")
KERNEL_SOURCES = ["decode_mma.cuh", "decode_tma.cuh", "device_common.cuh", "kv_store.cuh"]


# ----------------------------------------------------------------------------- helpers

def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_141_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(config: int, partition_size: int, form: str, split: bool):
    """DRAM bytes per launch of the partition kernel from the committed ncu
    summary, if it was taken on the current kernel source and on this
    workload (configuration, partition size, fused or separate write)."""
    try:
        fields = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
        if fields.get("kernel_source_sha256") != kernel_source_hash():
            return None
        if (fields.get("workload") != f"configuration {config}"
                or int(fields.get("partition_size", -1)) != partition_size
                or fields.get("form") != form or not split):
            return None
        return float(fields["dram_bytes_per_launch"])
    except Exception:
        return None


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples every 200 ms."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def decode_kernel_label(case) -> str:
    """Which decode kernel the library runs for this workload (its dispatch
    rule: 16-bit query, cache of that type or E4M3, even group or none -> tensor-core
    kernel; other rows of 128/256/512 bytes with block size 8, 16 or a multiple
    of 32 -> tensor-TMA CUDA-core kernel; anything else -> bulk-copy kernel)."""
    eb = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}[case.cache_dtype]
    row = case.head_size * eb
    B = case.block_size
    tma = row in (128, 256, 512) and (B in (8, 16) or (B >= 32 and B % 32 == 0))
    if tma and case.q_dtype in ("f16", "bf16") and case.cache_dtype in (case.q_dtype, "e4m3") \
            and (case.group % 2 == 0 or case.group == 1):
        return "paged_decode_mma_kernel"
    return "paged_decode_tma_kernel" if tma else "paged_decode_simt_kernel"


def max_over_ranks(value_ms: float, world: int, device=None) -> float:
    """The slowest rank's time: an all-reduce MAX over the default process
    group (identity for one rank)."""
    if world <= 1:
        return value_ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([value_ms], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_gbs(bytes_per_rank: int, world: int, ms_per_step: float) -> float:
    """Weak scaling: every rank processes its own copy of the workload, so the
    job moves world x the bytes in the slowest rank's time."""
    return world * bytes_per_rank / (ms_per_step * 1e-3) / 1e9


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- workload

class Step:
    """Device-resident inputs of one decode step and the calls that run it.

    form "fused":    pa_write_decode_partitions (the KV write folded into the
                     partition kernel) then pa_merge; or pa_write_decode.
    form "separate": pa_reshape_and_cache, pa_decode_partitions, pa_merge; or
                     pa_reshape_and_cache, pa_decode.
    form "shared":   pa_write_decode_shared_prefix with the units of
                     pa_shared_prefix_plan (partition kernel with shared-prefix
                     units and the KV write, then the merge: one call).
    """

    def __init__(self, case, device, partition_size=512, form="fused"):
        import torch
        from paged_kv_cache_141_gb300 import binding as pk
        self.pk, self.torch, self.case, self.dev, self.form = pk, torch, case, device, form
        c = case
        self.P = partition_size

        def t(a, dt):
            a = np.ascontiguousarray(a)
            if dt == "bf16":
                return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
            return torch.from_numpy(a).to(device)

        self.q = t(c.query, c.q_dtype)
        self.kc = t(c.k_cache, c.cache_dtype)
        self.vc = t(c.v_cache, c.cache_dtype)
        self.bt = t(c.block_tables, "i32")
        self.cl = t(c.context_lens, "i32")
        self.nk = t(c.new_key, c.kv_dtype)
        self.nv = t(c.new_value, c.kv_dtype)
        self.ns = t(c.new_slots, "i64")
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        odt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[c.q_dtype]
        self.out = torch.empty(c.num_seqs, c.num_q_heads, c.head_size, dtype=odt, device=device)
        if c.prefill_key is not None:
            pk.reshape_and_cache(t(c.prefill_key, c.kv_dtype), t(c.prefill_value, c.kv_dtype),
                                 self.kc, self.vc, t(c.prefill_slots, "i64"), c.k_scale,
                                 c.v_scale, self.status)
        self.split = pk.choose(c.num_seqs, c.num_q_heads, c.num_kv_heads, c.max_context_len,
                               partition_size) == 1
        if form == "fused" and c.kv_dtype != c.q_dtype:
            self.form = form = "separate"     # the fused write takes tokens of the query type
        self.plan = None
        if form == "shared":
            # units of sequences sharing their leading partitions, planned on
            # the host from the block tables (outside any timed region)
            self.plan = pk.shared_prefix_plan(c.block_tables, c.context_lens, c.block_size,
                                              partition_size)
            self.plan_dev = self.plan.to(device)
            self.split = True
        self.ws = pk.alloc_workspace(c.num_seqs, c.num_q_heads, c.head_size, c.max_context_len,
                                     partition_size, device)
        self.views = pk.workspace_views(self.ws, c.num_seqs, c.num_q_heads, c.head_size,
                                        c.max_context_len, partition_size)
        self.calls = self._calls()

    def _calls(self):
        pk, c = self.pk, self.case

        def common():          # read at call time: the end-to-end loop swaps buffers
            return (self.bt, self.cl, c.max_context_len, c.scale)

        def write(stream=None):
            pk.reshape_and_cache(self.nk, self.nv, self.kc, self.vc, self.ns, c.k_scale,
                                 c.v_scale, self.status, stream)

        def write_decode(stream=None):
            pk.write_decode(self.out, self.q, self.nk, self.nv, self.kc, self.vc, self.ns,
                            *common(), c.k_scale, c.v_scale, self.status, stream)

        def write_partitions(stream=None):
            pk.write_decode_partitions(self.q, self.nk, self.nv, self.kc, self.vc, self.ns,
                                       *common(), self.ws, self.P, c.k_scale, c.v_scale,
                                       self.status, stream)

        def decode(stream=None):
            pk.decode(self.out, self.q, self.kc, self.vc, *common(), c.k_scale, c.v_scale,
                      self.status, stream)

        def partitions(stream=None):
            pk.decode_partitions(self.q, self.kc, self.vc, *common(), self.ws, self.P, c.k_scale,
                                 c.v_scale, self.status, stream)

        def merge(stream=None):
            tmp, ml, es = self.views
            pk.merge(self.out, tmp, ml, es, self.cl, self.P, self.status, stream)

        def shared_step(stream=None):
            sp, us, up = self.plan_dev
            kw = (dict(key=self.nk, value=self.nv, slot_mapping=self.ns)
                  if c.kv_dtype == c.q_dtype else {})
            if not kw:
                write(stream)
            pk.write_decode_shared_prefix(self.out, self.q, self.kc, self.vc, *common(), self.ws,
                                          sp, us, up, self.plan.max_unit_parts, self.P,
                                          k_scale=c.k_scale, v_scale=c.v_scale,
                                          dev_status=self.status, stream=stream, **kw)

        if self.form == "shared":
            return [("write+decode+merge", shared_step)]
        if self.form == "fused":
            if self.split:
                return [("write+decode", write_partitions), ("merge", merge)]
            return [("write+decode", write_decode)]
        if self.split:
            return [("reshape_and_cache", write), ("decode", partitions), ("merge", merge)]
        return [("reshape_and_cache", write), ("decode", decode)]

    @property
    def launches_per_step(self) -> int:
        return len(self.calls)

    def step(self, stream=None):
        for _, f in self.calls:
            f(stream)

    @property
    def main_call(self) -> str:
        """The call that runs the decode kernel (partition kernel or single
        pass; in the fused form it also stores the step's new tokens; in the
        shared form the whole step, partition kernel and merge)."""
        return {"fused": "write+decode", "shared": "write+decode+merge"}.get(self.form, "decode")

    def bytes_per_step(self) -> dict:
        """Algorithmic bytes, by the method's definition (no workspace).
        total: the step -- K/V read, Q read, out written, and the new tokens'
        K/V read and stored with their slots. main_kernel: the decode
        kernel's share -- K/V, Q and out, plus the new tokens in the fused
        form. partials: what the partition kernel writes for the merge to
        read (per-partition outputs, maxima and sums; 0 for the single
        pass), reported beside the method bytes and not counted in them."""
        c = self.case
        write = c.write_bytes()
        decode = c.kv_bytes() + c.qo_bytes()
        if self.split:
            parts = sum(-(-int(L) // self.P) for L in c.context_lens)
            partials = parts * c.num_q_heads * (c.head_size + 2) * 4
        else:
            partials = 0
        main = decode + (write if self.form in ("fused", "shared") else 0)
        return {"write": write, "decode": decode, "total": write + decode, "main_kernel": main,
                "partials": partials}


# ----------------------------------------------------------------------------- arms

def run_ours(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    from paged_kv_cache_141_gb300 import workloads as W
    case = W.config_case(args.config)
    from paged_kv_cache_141_gb300 import binding as pk
    P = (pk.partition_size(case.num_seqs, case.num_kv_heads, case.max_context_len)
         if args.partition_size == "auto" else int(args.partition_size))
    st = Step(case, device, P, args.form)
    stream = torch.cuda.current_stream(device)

    # correctness gate: one step, no device-side errors
    st.step()
    torch.cuda.synchronize()
    if int(st.status.item()) != 0:
        raise SystemExit(f"device status {int(st.status.item())} after the first step")

    # the clock sampler starts (and settles) before the warm-up, so that the
    # GPU goes from the warm-up straight into the timed region at full
    # clocks; it runs on through the kernel leg below (a second or more)
    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    time.sleep(0.25 if sampler else 0)
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()

    K = args.steps
    ncall = st.launches_per_step
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(K):
        for _, f in st.calls:
            f()
    t_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(total_ms, world, device)
    call_ms = run_call_leg(st, stream, max(8, min(64, K)))

    by = st.bytes_per_step()
    ms_per_step = total_ms / K
    value = whole_job_gbs(by["total"], world, ms_per_step)
    seqs_per_s = world * case.num_seqs / (ms_per_step * 1e-3)
    peak, peak_kind = hbm_peak()
    kernel = run_kernel_leg(st, device, args.kernel_seconds)
    clocks = sampler.stop() if sampler else None
    achieved = by["main_kernel"] / (kernel["ms"] * 1e-3) / 1e9
    unique = unique_record(case, by, world, ms_per_step, peak)

    graph = run_graph(st, max(20, min(1000, K)), device)
    write_step = run_write_step(st, device)
    write_bulk = run_write_bulk(st, device)
    e2e = run_e2e(st, max(20, min(200, K // 10)), device)
    form_used = st.form
    del st
    torch.cuda.empty_cache()
    others = None
    if rank == 0 and args.configs != "none":
        others = run_other_configs(args, device, [int(x) for x in args.configs.split(",")])
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(case, P, budget_s=args.cpu_seconds)
    if rank != 0:
        return
    split = "partitioned" if by["partials"] else "single-pass"
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": case.cache_dtype, "data": "synthetic",
        "config": {"workload": f"{case.name} (configuration {args.config})",
                   "num_seqs": case.num_seqs, "num_q_heads": case.num_q_heads,
                   "num_kv_heads": case.num_kv_heads, "head_size": case.head_size,
                   "block_size": case.block_size, "kv_dtype": case.cache_dtype,
                   "context_lens": "log-uniform [512, 4096]" if args.config == 3 else "see workloads",
                   "total_context_tokens": case.total_tokens, "partition_size": P,
                   "decode_form": f"{split}, {form_used}",
                   "l2": "inputs larger than L2 (KV pool %.2f GB vs 129 MB L2); no flush"
                         % (case.kv_bytes() / 1e9),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "frac_of_hbm_peak": round(value / peak, 4),
        **({"unique_bytes": unique} if unique else {}),
        "seqs_per_s_per_layer": round(seqs_per_s, 1),
        "bytes_per_step": by,
        "call_ms": {k: round(v, 5) for k, v in call_ms.items()},
        "call_ms_timing": "CUDA events around each call, a separate leg after the timed steps",
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": recorded_traffic(args.config, P, form_used, bool(by["partials"])),
                     "kernel": kernel["name"], "kernel_ms": round(kernel["ms"], 6),
                     "method_bytes_per_launch": by["main_kernel"],
                     "partials_bytes_per_launch": by["partials"],
                     "step_frac": round(value / peak, 4),
                     "timing": kernel["timing"],
                     "peak_kind": f"{peak_kind} (HBM copy, MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s"},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "graph": graph,
        "write_step": write_step,
        "write_bulk": write_bulk,
        "configs": others,
        "gpu_launches": K * ncall,
        "clocks": clocks,
    }
    print(json.dumps(line))


def run_call_leg(st: Step, stream, steps: int) -> dict:
    """Each call of the step on its own: CUDA events around every call of
    `steps` steps after the timed region (events between launches add a few
    microseconds of stream time, so they stay out of the timed loop)."""
    import torch
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(st.calls) + 1)]
          for _ in range(steps)]
    for e in ev:
        e[0].record(stream)
        for j, (_, f) in enumerate(st.calls):
            f()
            e[j + 1].record(stream)
    torch.cuda.synchronize()
    return {name: sum(e[j].elapsed_time(e[j + 1]) for e in ev) / steps
            for j, (name, _) in enumerate(st.calls)}


def unique_record(case, by, world, ms_per_step, peak):
    """Where sequences share blocks: the step's rate on each distinct cached
    token's K/V once (shared prefix blocks are read from L2 after the first
    reader), next to the logical-byte rate."""
    unique_kv = case.unique_kv_bytes()
    if unique_kv >= case.kv_bytes():
        return None
    ub = by["total"] - case.kv_bytes() + unique_kv
    ug = whole_job_gbs(ub, world, ms_per_step)
    return {"kv_bytes": unique_kv, "bytes_per_step": ub, "gbs": round(ug, 2),
            "frac_of_hbm_peak": round(ug / peak, 4),
            "note": "each distinct cached token's K/V once (shared prefix blocks count once)"}


def run_kernel_leg(st: Step, device, min_seconds: float = 1.0, per_graph: int = 20) -> dict:
    """The decode kernel alone (the step's main call: the partition kernel,
    or the single pass, with the KV write in the fused form): `per_graph`
    back-to-back launches captured in a CUDA graph and replayed until at
    least `min_seconds` have passed; CUDA events on the replaying stream.
    Every launch rewrites the same new tokens, so the pool is unchanged, and
    the K/V read (far larger than L2) comes from HBM each time."""
    import torch
    fn = dict(st.calls)[st.main_call]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(per_graph):
                fn(s)
    cur = torch.cuda.current_stream(device)
    cur.wait_stream(s)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    for _ in range(2):
        g.replay()
    a.record(cur)
    g.replay()
    b.record(cur)
    torch.cuda.synchronize()
    reps = max(10, int(math.ceil(min_seconds * 1e3 / max(a.elapsed_time(b), 1e-3))))
    a.record(cur)
    for _ in range(reps):
        g.replay()
    b.record(cur)
    torch.cuda.synchronize()
    if int(st.status.item()) != 0:
        raise SystemExit(f"device status {int(st.status.item())} after the kernel leg")
    total = a.elapsed_time(b)
    n = reps * per_graph
    if st.form == "shared":
        name = (decode_kernel_label(st.case) + " (partition kernel with shared-prefix units, KV "
                "write fused) + paged_merge_kernel")
    else:
        name = decode_kernel_label(st.case) + (
            (" (partition kernel" if st.split else " (single pass")
            + (", KV write fused)" if st.form == "fused" else ")"))
    return {"name": name, "ms": total / n, "launches": n,
            "timing": f"CUDA graph of {per_graph} launches of the kernel alone, replayed {reps} "
                      f"times ({n} launches, {total / 1e3:.2f} s), events on the replaying stream"}


def run_shared_step(case, device, partition_size, seconds: float = 0.5) -> dict | None:
    """Where sequences share their leading partitions' blocks: the step in
    the shared form (Step form "shared": pa_write_decode_shared_prefix, the
    partition kernel whose first CTAs read each unit's shared partitions once
    for its members, then the merge), launched eagerly and replayed as a CUDA
    graph. None when the plan finds no units."""
    import torch
    from paged_kv_cache_141_gb300 import binding as pk
    if pk.shared_prefix_plan(case.block_tables, case.context_lens, case.block_size,
                             partition_size).num_units == 0:
        return None                               # no sharing: nothing to build
    st = Step(case, device, partition_size, "shared")
    st.step()
    torch.cuda.synchronize()
    if int(st.status.item()) != 0:
        raise SystemExit(f"device status {int(st.status.item())} after the shared-prefix step")
    cur = torch.cuda.current_stream(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    for _ in range(3):
        st.step()
    a.record(cur)
    st.step()
    b.record(cur)
    torch.cuda.synchronize()
    n = max(20, int(seconds * 1e3 / max(a.elapsed_time(b), 1e-3)))
    a.record(cur)
    for _ in range(n):
        st.step()
    b.record(cur)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    graph = run_graph(st, n, device)
    by = st.bytes_per_step()
    peak, _ = hbm_peak()
    gbs = by["total"] / (ms * 1e-3) / 1e9
    unique = unique_record(case, by, 1, ms, peak)
    plan = st.plan
    rec = {"ms_per_step": round(ms, 5), "steps": n, "graph_ms_per_step": graph["ms_per_step"],
           "gbs": round(gbs, 2), "frac_of_hbm_peak": round(gbs / peak, 4),
           "seqs_per_s_per_layer": round(case.num_seqs / (ms * 1e-3), 1),
           **({"unique_bytes": unique} if unique else {}),
           "units": plan.num_units, "unit_members": int((plan.unit_seqs >= 0).sum()),
           "shared_partitions": int(plan.max_unit_parts),
           "launches": "partition kernel with shared-prefix units (KV write fused), merge",
           "note": "logical bytes as in the plain step; the shared partitions' K/V is read "
                   "once per unit of up to 4 sequences"}
    del st
    torch.cuda.empty_cache()
    return rec


def measure_config(index: int, device, partition_size, form="fused", step_seconds=0.3,
                   kernel_seconds=0.5) -> dict:
    """One workload's decode step and its kernel: the step launched eagerly
    (about step_seconds of steps), the kernel alone (run_kernel_leg), and
    the step's own KV write (run_write_step)."""
    import torch
    from paged_kv_cache_141_gb300 import binding as pk
    from paged_kv_cache_141_gb300 import workloads as W
    case = W.config_case(index)
    P = (pk.partition_size(case.num_seqs, case.num_kv_heads, case.max_context_len)
         if partition_size == "auto" else int(partition_size))
    st = Step(case, device, P, form)
    st.step()
    torch.cuda.synchronize()
    if int(st.status.item()) != 0:
        raise SystemExit(f"configuration {index}: device status {int(st.status.item())}")
    for _ in range(5):
        st.step()
    cur = torch.cuda.current_stream(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(cur)
    st.step()
    b.record(cur)
    torch.cuda.synchronize()
    n = max(20, int(step_seconds * 1e3 / max(a.elapsed_time(b), 1e-3)))
    a.record(cur)
    for _ in range(n):
        st.step()
    b.record(cur)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / n
    by = st.bytes_per_step()
    peak, _ = hbm_peak()
    gbs = by["total"] / (ms * 1e-3) / 1e9
    kern = run_kernel_leg(st, device, kernel_seconds)
    kg = by["main_kernel"] / (kern["ms"] * 1e-3) / 1e9
    graph = run_graph(st, max(20, n), device)
    ws = run_write_step(st, device)
    unique = unique_record(case, by, 1, ms, peak)
    shared = run_shared_step(case, device, P) if st.split else None
    rec = {"workload": f"{case.name} (configuration {index})", "num_seqs": case.num_seqs,
           "num_q_heads": case.num_q_heads, "num_kv_heads": case.num_kv_heads,
           "head_size": case.head_size, "kv_dtype": case.cache_dtype,
           "total_context_tokens": case.total_tokens, "partition_size": P,
           "decode_form": ("partitioned" if st.split else "single-pass") + ", " + st.form,
           "ms_per_step": round(ms, 5), "steps": n, "gbs": round(gbs, 2),
           "frac_of_hbm_peak": round(gbs / peak, 4),
           "seqs_per_s_per_layer": round(case.num_seqs / (ms * 1e-3), 1),
           "graph_ms_per_step": graph["ms_per_step"],
           "kernel": {"name": kern["name"], "ms": round(kern["ms"], 6),
                      "method_bytes_per_launch": by["main_kernel"],
                      "partials_bytes_per_launch": by["partials"], "gbs": round(kg, 1),
                      "frac": round(kg / peak, 4), "timing": kern["timing"]},
           "write_step": {"tokens_per_s": ws["tokens_per_s"], "us_per_launch": ws["us_per_launch"]},
           "bytes_per_step": by}
    if unique:
        rec["unique_bytes"] = unique
    if shared:
        rec["shared_prefix_step"] = shared
    del st
    torch.cuda.empty_cache()
    return rec


def run_other_configs(args, device, indices) -> dict:
    """Records for the other workloads (run_ours times the main one), with
    the SM clocks sampled across them. The long-context workload is also
    measured at the configured 512-token partitions next to the library's
    own choice."""
    import torch
    sampler = ClockSampler(torch.cuda.current_device())
    time.sleep(0.25)
    out = {}
    for i in indices:
        if i == args.config:
            continue
        out[str(i)] = measure_config(i, device, "auto", args.form)
        if i == 4:
            out["4@512"] = measure_config(i, device, 512, args.form)
    clocks = sampler.stop()
    out["clocks"] = clocks
    return out


PREFILL_METRIC = {
    "chunk512": "multi-query paged attention TFLOP/s (causal, algorithmic), 512-token prefill chunks",
    "spec8": "multi-query paged attention KV GB/s, 8-token speculative verification",
    "spec4": "multi-query paged attention KV GB/s, 4-token speculative verification",
    "spec2": "multi-query paged attention KV GB/s, 2-token speculative verification",
}


def prefill_queries(case, kind):
    """The query law of a multi-query workload: a 512-token chunk at the end
    of every context (capped at L_s), or 8, 4 or 2 draft tokens per
    sequence."""
    if kind == "chunk512":
        return ("fixed", np.minimum(512, case.context_lens))
    return ("fixed", np.minimum(int(kind[len("spec"):]), case.context_lens))


def prefill_work(case, qs: np.ndarray, seqs=None):
    """Algorithmic work of one multi-query step (or of the sequences `seqs`):
    FLOPs (QK^T and PV over each query token's causal prefix, 4 d per (query
    head, key)) and bytes (the K/V of every context once, Q read, out
    written)."""
    counts = np.diff(qs).astype(np.int64)
    L = case.context_lens.astype(np.int64)
    if seqs is not None:
        counts, L = counts[seqs], L[seqs]
    # keys seen by the Q_s tokens: sum_{i<Q} (L - Q + i + 1)
    keys = (counts * (L - counts) + counts * (counts + 1) // 2).sum()
    flops = 4 * case.head_size * case.num_q_heads * int(keys)
    eb = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}
    qo = 2 * int(counts.sum()) * case.num_q_heads * case.head_size * eb[case.q_dtype]
    kv = 2 * int(L.sum()) * case.num_kv_heads * case.head_size * eb[case.cache_dtype]
    return flops, kv + qo


def prefill_cpu_baseline(case, q, tensor: bool, budget_s: float = 12.0):
    """The oracle's multi-query attention, as it stands, on this host: one
    sequence at a time in a seeded order until the budget is spent; the rate
    in the line's unit over the work done."""
    import oracle
    kc, vc, _, _ = oracle_inputs(case)
    qs = q.query_start
    # a FLOP rate hardly depends on the context length: the shortest contexts
    # first keep one sequence's oracle time inside the budget; a byte rate
    # takes a seeded random order
    order = (np.argsort(case.context_lens, kind="stable") if tensor
             else np.random.default_rng(3).permutation(case.num_seqs))
    done, elapsed = [], 0.0
    for s_ in order:
        s_ = int(s_)
        rows = slice(int(qs[s_]), int(qs[s_ + 1]))
        t = time.perf_counter()
        oracle.paged_prefill(np.ascontiguousarray(q.query[rows]), case.q_dtype,
                             np.array([0, int(qs[s_ + 1] - qs[s_])], dtype=np.int32), kc, vc,
                             case.cache_dtype, np.ascontiguousarray(case.block_tables[s_:s_ + 1]),
                             np.ascontiguousarray(case.context_lens[s_:s_ + 1]),
                             case.num_kv_heads, case.block_size, case.scale, case.k_scale,
                             case.v_scale)
        elapsed += time.perf_counter() - t
        done.append(s_)
        if elapsed >= budget_s:
            break
    flops, nbytes = prefill_work(case, qs, np.array(done))
    value = flops / elapsed / 1e12 if tensor else nbytes / elapsed / 1e9
    return {"value": round(value, 6), "unit": "TFLOP/s" if tensor else "GB/s", "cores": 1,
            "kind": "oracle", **host_cpu(),
            "sample": f"{len(done)} of {case.num_seqs} sequences "
                      f"({'shortest contexts first, ' if tensor else ''}"
                      f"{int(np.diff(qs)[done].sum())} query tokens), single-threaded C oracle "
                      f"in fp64, {elapsed:.1f} s"}


def prefill_kernel_name(case, max_queries: int) -> str:
    """The kernel pa_paged_prefill selects for this workload, as the library
    reports it (pa_paged_prefill_kernel)."""
    from paged_kv_cache_141_gb300 import binding as pk
    code = {"f32": pk.PA_F32, "f16": pk.PA_F16, "bf16": pk.PA_BF16, "e4m3": pk.PA_FP8_E4M3}
    kind = pk.prefill_kernel(max_queries, case.num_q_heads, case.num_kv_heads, case.head_size,
                             case.block_size, case.num_blocks, code[case.q_dtype],
                             code[case.cache_dtype])
    e4m3 = case.cache_dtype == "e4m3"
    widened = ", E4M3 widened in registers" if e4m3 else ""
    products = case.q_dtype == "bf16" and case.head_size == 128
    tc_e4m3 = ", E4M3 products on kind::f8f6f4" if products else ", E4M3 tiles widened to binary16"
    return {
        "mma": f"paged_prefill_mma_kernel (warp-level MMA, one K/V pass for all rows{widened})",
        "mma_two_tiles": f"paged_prefill_mma2_kernel (warp-level MMA, two n-tiles per warp{widened})",
        "tc_two_tiles": "paged_prefill_tc2_kernel (two query tiles per CTA"
                        + (tc_e4m3 if e4m3 else "") + ")",
        "tc": "paged_prefill_tc_kernel" + (f" ({tc_e4m3[2:]})" if e4m3 else ""),
        "cuda_cores": "paged_decode_simt_kernel (one query token per work unit)",
    }[kind]


def run_prefill(args):
    """Multi-query paged attention (pa_paged_prefill) on the Llama-3-8B GQA
    pool: the kernel alone, K timed launches, CUDA events, clocks sampled."""
    import torch
    from paged_kv_cache_141_gb300 import binding as pk
    from paged_kv_cache_141_gb300 import workloads as W
    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    case = (W.config_case(args.config, num_seqs=args.num_seqs) if args.num_seqs
            else W.config_case(args.config))
    q = W.make_queries(case, prefill_queries(case, args.prefill))
    st = Step(case, device, 512, "separate")
    st.calls[0][1]()                       # the step's KV write: every context token stored
    query = torch.from_numpy(np.ascontiguousarray(q.query).view(np.int16)).view(
        torch.bfloat16).to(device) if case.q_dtype == "bf16" else torch.from_numpy(q.query).to(device)
    qstart = torch.from_numpy(q.query_start).to(device)
    out = torch.empty_like(query)
    # the order in which sequences start: longest context first, sorted on
    # the host from the lengths a serving scheduler holds, passed as an input
    host_order_np = pk.longest_first(case.context_lens)
    order = torch.from_numpy(host_order_np).to(device)

    def launch():
        pk.paged_prefill(out, query, qstart, st.kc, st.vc, st.bt, st.cl, q.max_queries,
                         case.max_context_len, case.scale, case.k_scale, case.v_scale, st.status,
                         seq_order=order)

    launch()
    torch.cuda.synchronize()
    if int(st.status.item()) != 0:
        raise SystemExit(f"device status {int(st.status.item())} after the first launch")
    K = args.steps
    stream = torch.cuda.current_stream(device)
    # sampler first, then the warm-up: no idle gap before the timed region
    sampler = ClockSampler(torch.cuda.current_device())
    time.sleep(0.25)
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(K):
        launch()
    b.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = a.elapsed_time(b) / K
    # end to end through the binding with host buffers: each step copies its
    # query tokens, query starts and lengths in from pinned memory, runs, and
    # reads the output back -- pipelined as a serving loop would run it: two
    # sets of device buffers alternate, copies in on one stream, the launch
    # on the compute stream, copies out on a third, events ordering every
    # buffer reuse
    host_q = torch.empty(query.shape, dtype=query.dtype, pin_memory=True)
    host_q.copy_(query.cpu())
    host_qs = torch.from_numpy(q.query_start).pin_memory()
    host_cl = st.cl.cpu().pin_memory()
    host_order = torch.from_numpy(host_order_np).pin_memory()
    host_out = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    dq = [query, torch.empty_like(query)]
    dqs = [qstart, torch.empty_like(qstart)]
    dcl = [st.cl, torch.empty_like(st.cl)]
    dord = [order, torch.empty_like(order)]
    dout = [out, torch.empty_like(out)]
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    in_ready = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    out_read = [torch.cuda.Event() for _ in range(2)]

    def e2e_run(count):
        for i in range(count):
            k = i % 2
            if i >= 2:
                s_in.wait_event(done[k])                 # step i-2 has used buffer k
            with torch.cuda.stream(s_in):
                dq[k].copy_(host_q, non_blocking=True)
                dqs[k].copy_(host_qs, non_blocking=True)
                dcl[k].copy_(host_cl, non_blocking=True)
                dord[k].copy_(host_order, non_blocking=True)
            in_ready[k].record(s_in)
            stream.wait_event(in_ready[k])
            if i >= 2:
                stream.wait_event(out_read[k])           # step i-2's output has left
            pk.paged_prefill(dout[k], dq[k], dqs[k], st.kc, st.vc, st.bt, dcl[k], q.max_queries,
                             case.max_context_len, case.scale, case.k_scale, case.v_scale,
                             st.status, seq_order=dord[k])
            done[k].record(stream)
            s_out.wait_event(done[k])
            with torch.cuda.stream(s_out):
                host_out[k].copy_(dout[k], non_blocking=True)
            out_read[k].record(s_out)

    ke = max(4, min(K, 20))
    e2e_run(4)
    torch.cuda.synchronize()
    ea = torch.cuda.Event(enable_timing=True)
    eb_ = torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    e2e_run(ke)
    eb_.record(s_out)                                  # after the last output has left
    torch.cuda.synchronize()
    e2e_ms = ea.elapsed_time(eb_) / ke
    h2d = (host_q.numel() * host_q.element_size() + host_qs.numel() * 4 + host_cl.numel() * 4
           + host_order.numel() * 4)
    d2h = host_out[0].numel() * host_out[0].element_size()

    flops, nbytes = prefill_work(case, q.query_start)
    tflops = flops / (ms * 1e-3) / 1e12
    gbs = nbytes / (ms * 1e-3) / 1e9
    peak_hbm, hk = hbm_peak()
    try:
        with open(PEAKS_FILE) as f:
            peak_tc, tk = float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except Exception:
        peak_tc, tk = 1700.0, "fallback"
    tensor = args.prefill == "chunk512"
    value, unit = (tflops, "TFLOP/s") if tensor else (gbs, "GB/s")
    e2e_value = (flops / (e2e_ms * 1e-3) / 1e12) if tensor else (nbytes / (e2e_ms * 1e-3) / 1e9)
    cpu = None if args.no_cpu_baseline else prefill_cpu_baseline(case, q, tensor,
                                                                   args.cpu_seconds)
    line = {
        "metric": PREFILL_METRIC[args.prefill], "value": round(value, 2), "unit": unit,
        "n_gpus": 1, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": case.cache_dtype, "data": "synthetic",
        "config": {"workload": f"{case.name} pool, {args.prefill} queries",
                   "num_seqs": case.num_seqs, "num_q_heads": case.num_q_heads,
                   "num_kv_heads": case.num_kv_heads, "head_size": case.head_size,
                   "block_size": case.block_size, "query_tokens": int(q.query_start[-1]),
                   "max_queries_per_seq": q.max_queries, "total_context_tokens": case.total_tokens,
                   "seq_order": "longest context first (host sort of the lengths, an input "
                                "copied in with them end to end)",
                   "l2": "KV pool %.2f GB vs 129 MB L2; no flush" % (case.kv_bytes() / 1e9)},
        "tflops": round(tflops, 2), "kv_q_o_gbs": round(gbs, 2),
        "flops_per_step": flops, "bytes_per_step": nbytes,
        "roofline": ({"bound": "tensor", "achieved": round(tflops, 2), "peak": peak_tc,
                      "unit": "TFLOP/s", "frac": round(tflops / peak_tc, 4), "traffic": None,
                      "peak_kind": f"{tk} bf16 sustained"}
                     if tensor else
                     {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak_hbm, "unit": "GB/s",
                      "frac": round(gbs / peak_hbm, 4), "traffic": None,
                      "peak_kind": f"{hk} HBM copy"}),
        "kernel": prefill_kernel_name(case, q.max_queries),
        "e2e": {"value": round(e2e_value, 2), "unit": unit, "ms_per_step": round(e2e_ms, 5),
                "steps": ke, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "pipelined": "inputs of step i+1 copied in and output of step i-1 copied "
                             "out while step i runs (two buffer sets, three streams)"},
        "cpu_baseline": cpu,
        "gpu_launches": K,
        "clocks": clocks,
    }
    print(json.dumps(line))


def run_write_step(st: Step, device, per_graph: int = 20, replays: int = 20):
    """The decode step's own KV write alone (one new token per sequence to
    its slot, as pa_reshape_and_cache in the separate form): device time per
    launch, from a CUDA graph of back-to-back launches (a launch from Python
    costs more host time than this write takes on the GPU), and tokens/s.
    Rewrites the same tokens, so the pool is unchanged."""
    import torch
    c, pk = st.case, st.pk

    def write(stream=None):
        pk.reshape_and_cache(st.nk, st.nv, st.kc, st.vc, st.ns, c.k_scale, c.v_scale,
                             st.status, stream)

    write()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for _ in range(per_graph):
                write(s)
    torch.cuda.current_stream(device).wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(replays):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (replays * per_graph)
    return {"tokens": c.num_seqs, "us_per_launch": round(ms * 1e3, 2),
            "tokens_per_s": round(c.num_seqs / (ms * 1e-3), 1), "bytes": c.write_bytes(),
            "kernel": "reshape_and_cache_kernel",
            "timing": f"CUDA graph of {per_graph} launches, replayed {replays} times"}


def run_write_bulk(st: Step, device, tokens: int | None = None, steps: int = 50):
    """The KV write alone in its bandwidth-bound regime: as many new tokens
    as the configuration's contexts hold (default; capped by the pool's free
    slots), of its head shape, scattered to seeded random distinct slots of
    the pool -- write tokens/s and bytes/s (input read + cache written +
    slots). Runs last: it overwrites pool slots."""
    import torch
    c, pk = st.case, st.pk
    slots_total = c.num_blocks * c.block_size
    tokens = min(c.total_tokens if tokens is None else tokens, slots_total - c.block_size)
    g = torch.Generator(device="cpu").manual_seed(0x5EED)
    slots = (torch.randperm(slots_total - c.block_size, generator=g)[:tokens] + c.block_size)
    slots = slots.to(torch.int64).to(device)                 # block 0 stays reserved
    dt = st.nk.dtype
    gd = torch.Generator(device=device).manual_seed(0x5EED)
    key = torch.randn(tokens, c.num_kv_heads, c.head_size, generator=gd, device=device).to(dt)
    value = torch.randn(tokens, c.num_kv_heads, c.head_size, generator=gd, device=device).to(dt)
    for _ in range(3):
        pk.reshape_and_cache(key, value, st.kc, st.vc, slots, c.k_scale, c.v_scale, st.status)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        pk.reshape_and_cache(key, value, st.kc, st.vc, slots, c.k_scale, c.v_scale, st.status)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    nbytes = c.write_bytes(tokens)
    peak, _ = hbm_peak()
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"tokens": tokens, "ms": round(ms, 5), "tokens_per_s": round(tokens / (ms * 1e-3), 1),
            "gbs": round(gbs, 1), "frac_of_hbm_peak": round(gbs / peak, 4),
            "bytes": nbytes, "kernel": "reshape_and_cache_kernel"}


def run_graph(st: Step, steps: int, device):
    """The step captured once in a CUDA graph (the library's calls are
    asynchronous on the caller's stream with no host synchronisation) and
    replayed: the same kernels without per-launch host overhead."""
    import torch
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            st.step(s)
    torch.cuda.current_stream(device).wait_stream(s)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream(device)
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        g.replay()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    by = st.bytes_per_step()["total"]
    return {"value": round(by / (ms * 1e-3) / 1e9, 2), "unit": UNIT, "ms_per_step": round(ms, 5),
            "steps": steps}


def run_e2e(st: Step, steps: int, device):
    """The same step through the public API with host buffers: every step
    copies its inputs from pinned host memory, runs the write and the decode,
    and reads its output back, as a serving loop would -- pipelined: two sets
    of device inputs/outputs alternate, host-to-device copies run on one
    stream, the step on the compute stream and the device-to-host read on a
    third, so step i+1's inputs arrive and step i-1's output leaves while step
    i computes (events order every reuse of a buffer)."""
    import torch
    names = ("q", "bt", "cl", "nk", "nv", "ns")
    host = {}
    for name in names:
        tdev = getattr(st, name)
        host[name] = torch.empty(tdev.shape, dtype=tdev.dtype, pin_memory=True)
        host[name].copy_(tdev.cpu())
    dev_in = [{n: getattr(st, n) for n in names}, {n: torch.empty_like(getattr(st, n)) for n in names}]
    dev_out = [st.out, torch.empty_like(st.out)]
    host_out = [torch.empty(st.out.shape, dtype=st.out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = host_out[0].numel() * host_out[0].element_size()
    comp = torch.cuda.current_stream(device)
    s_in = torch.cuda.Stream(device)
    s_out = torch.cuda.Stream(device)
    ev = lambda: [torch.cuda.Event() for _ in range(2)]
    in_ready, done, out_read = ev(), ev(), ev()
    saved = {n: getattr(st, n) for n in names + ("out",)}

    def run(count):
        for i in range(count):
            k = i % 2
            if i >= 2:
                s_in.wait_event(done[k])                 # step i-2 has used buffer k
            with torch.cuda.stream(s_in):
                for n in names:
                    dev_in[k][n].copy_(host[n], non_blocking=True)
            in_ready[k].record(s_in)
            comp.wait_event(in_ready[k])
            if i >= 2:
                comp.wait_event(out_read[k])             # step i-2's output has left
            for n in names:
                setattr(st, n, dev_in[k][n])
            st.out = dev_out[k]
            st.step(comp)
            done[k].record(comp)
            s_out.wait_event(done[k])
            with torch.cuda.stream(s_out):
                host_out[k].copy_(dev_out[k], non_blocking=True)
            out_read[k].record(s_out)

    run(4)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    comp.wait_event(a)
    run(steps)
    s_out.wait_event(done[(steps - 1) % 2])
    b.record(s_out)
    torch.cuda.synchronize()
    for n, t in saved.items():
        setattr(st, n, t)
    ms = a.elapsed_time(b) / steps
    by = st.bytes_per_step()["total"]
    return {"value": round(by / (ms * 1e-3) / 1e9, 2), "unit": UNIT, "ms_per_step": round(ms, 5),
            "steps": steps, "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipelined": "inputs of step i+1 copied in and output of step i-1 copied out "
                         "while step i runs (two buffer sets, three streams)"}


def host_cpu() -> dict:
    """This host's CPU model (x86 'model name'; Arm implementer/part codes)
    and hardware thread count, for the CPU-baseline record."""
    import platform
    model, impl, part = None, None, None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k = k.strip().lower()
                if k == "model name" and model is None:
                    model = v.strip()
                elif k == "cpu implementer" and impl is None:
                    impl = v.strip()
                elif k == "cpu part" and part is None:
                    part = v.strip()
    except OSError:
        pass
    if model is None and impl is not None:
        model = f"Arm implementer {impl} part {part}"
    return {"cpu_model": model or platform.machine(), "host_threads": os.cpu_count()}


def oracle_inputs(case):
    """The pool as the oracle sees it (E4M3 pools: the context tokens written
    through the oracle's own encoder) and the logical bytes per context token
    and per sequence's query + output."""
    import oracle
    kc, vc = case.k_cache, case.v_cache
    if case.prefill_key is not None:
        kc, vc = kc.copy(), vc.copy()
        rc = oracle.reshape_and_cache(case.prefill_key, case.prefill_value, kc, vc,
                                      case.prefill_slots, case.num_kv_heads, case.head_size,
                                      case.block_size, case.kv_dtype, case.cache_dtype,
                                      case.k_scale, case.v_scale)
        if rc != 0:
            raise SystemExit(f"oracle write of the prefill tokens failed ({rc})")
    eb = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}
    per_tok = 2 * case.num_kv_heads * case.head_size * eb[case.cache_dtype]
    qo = 2 * case.num_q_heads * case.head_size * eb[case.q_dtype]
    return kc, vc, per_tok, qo


def cpu_baseline(case, partition_size, budget_s=12.0):
    """The oracle, as it stands, on a bounded sample of the workload's
    sequences (single-threaded C, fp64), timed on this host."""
    import oracle
    order = np.random.default_rng(1).permutation(case.num_seqs)
    done, bytes_done = [], 0
    kc, vc, per_tok, qo = oracle_inputs(case)
    elapsed = 0.0
    for s in order:
        sl = slice(int(s), int(s) + 1)
        t = time.perf_counter()
        oracle.decode(np.ascontiguousarray(case.query[sl]), case.q_dtype, kc, vc, case.cache_dtype,
                      np.ascontiguousarray(case.block_tables[sl]),
                      np.ascontiguousarray(case.context_lens[sl]), case.num_kv_heads,
                      case.block_size, case.scale, case.k_scale, case.v_scale)
        elapsed += time.perf_counter() - t
        done.append(int(s))
        bytes_done += int(case.context_lens[s]) * per_tok + qo
        if elapsed >= budget_s:
            break
    return {"value": round(bytes_done / elapsed / 1e9, 4), "unit": UNIT, "cores": 1,
            "kind": "oracle", **host_cpu(),
            "sample": f"{len(done)} of {case.num_seqs} sequences ({sum(int(case.context_lens[s]) for s in done)} "
                      f"context tokens), single-threaded C oracle in fp64, {elapsed:.1f} s",
            "seqs_per_s": round(len(done) / elapsed, 3)}


def run_reference(args):
    """The oracle as the reference arm, on this host's cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from paged_kv_cache_141_gb300 import workloads as W
    import oracle
    case = W.config_case(args.config)
    kc, vc, per_tok, qo = oracle_inputs(case)
    order = np.random.default_rng(2).permutation(case.num_seqs)
    K, Wm = args.steps, args.warmup
    # each step decodes a slice of sequences sized so K + W steps take about
    # args.reference_seconds in total
    t = time.perf_counter()
    oracle.decode(np.ascontiguousarray(case.query[:1]), case.q_dtype, kc, vc,
                  case.cache_dtype, np.ascontiguousarray(case.block_tables[:1]),
                  np.ascontiguousarray(case.context_lens[:1]), case.num_kv_heads,
                  case.block_size, case.scale, case.k_scale, case.v_scale)
    per_seq = max(1e-4, (time.perf_counter() - t) / max(1, int(case.context_lens[0])) *
                  float(case.context_lens.mean()))
    n = max(1, int(args.reference_seconds / (K + Wm) / per_seq))
    n = min(n, case.num_seqs)
    cursor = 0

    def one_step():
        nonlocal cursor
        idx = np.array([order[(cursor + i) % case.num_seqs] for i in range(n)])
        cursor += n
        oracle.decode(np.ascontiguousarray(case.query[idx]), case.q_dtype, kc, vc,
                      case.cache_dtype, np.ascontiguousarray(case.block_tables[idx]),
                      np.ascontiguousarray(case.context_lens[idx]), case.num_kv_heads,
                      case.block_size, case.scale, case.k_scale, case.v_scale)
        return int(case.context_lens[idx].sum()) * per_tok + n * qo

    for _ in range(Wm):
        one_step()
    total, t0 = 0, time.perf_counter()
    for _ in range(K):
        total += one_step()
    el = time.perf_counter() - t0
    value = total / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": K, "warmup": Wm, "ms_per_step": round(el / K * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": case.cache_dtype, "data": "synthetic",
            "config": {"workload": f"{case.name} (configuration {args.config})",
                       "num_seqs": case.num_seqs, "num_q_heads": case.num_q_heads,
                       "num_kv_heads": case.num_kv_heads, "head_size": case.head_size,
                       "block_size": case.block_size, "kv_dtype": case.cache_dtype},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"{n} sequences per step of {case.num_seqs}, "
                                       f"single-threaded C oracle in fp64", **host_cpu()},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=DEFAULT_CONFIG, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--partition-size", default="auto",
                    help="tokens per partition, or 'auto' (the library's choice)")
    ap.add_argument("--form", choices=["fused", "separate", "shared"], default="fused",
                    help="how the step is launched (see Step); shared: shared-prefix units "
                         "(pa_write_decode_shared_prefix)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--kernel-seconds", type=float, default=1.2,
                    help="length of the kernel-only leg behind the roofline")
    ap.add_argument("--configs", default="1,2,4,5",
                    help="other workloads to record in the line ('none' to skip)")
    ap.add_argument("--reference-seconds", type=float, default=90.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill", choices=["chunk512", "spec8", "spec4", "spec2"], default=None,
                    help="time multi-query paged attention on the configuration's pool instead")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="with --prefill: fewer sequences of the same shape (small ncu captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.prefill:
        run_prefill(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
