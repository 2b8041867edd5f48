"""QSA layer-step benchmark on GB300.

Default workload: the decode batch (64 requests, contexts uniform in
[8192, 32768], one query row each; indexer 32 x 128 e4m3, compress_ratio 4,
token_topk 2048; GQA 32q / 4kv x 128 bf16, KV block 64), the configuration
the decode tokens/s metric is quoted on.  One step = one call of
qsa_layer_step (all four stages) over that batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline]

N > 1 runs under torchrun as independent replicas (one per GPU, no
collective on the data path: requests are independent), value = total rows
of all ranks / max time over ranks.  Between timed steps the L2 is flushed by
writing a 512 MiB buffer, then reading a separate 256 MiB buffer so that the
written lines are evicted (and written back) before the step instead of
during it; only the step itself sits between the CUDA events.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from learned_sparse_attention_gb300 import qsa as Q  # noqa: E402
from learned_sparse_attention_gb300 import workloads as W  # noqa: E402

METRIC = "QSA layer decode tokens/s and prefill rows/s at 1 GB300; % of HBM / fp8 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
FLUSH_BYTES = 512 << 20
DRAIN_BYTES = 256 << 20


def flush_l2(flush, drain, i):
    """Write a buffer larger than L2, then read another one larger than L2."""
    flush.fill_(i & 0xFF)
    return drain.sum()

# DRAM bytes per launch of the sparse GQA kernel on the decode batch, from one
# ncu capture (the decode-batch kernel-sections summary), keyed by a hash of
# the kernel sources it was taken on; any other source reports null.
GQA_TRAFFIC = {"74bde55c61c42a04": 270416896 + 3225856}
GQA_SOURCES = ("learned_sparse_attention_gb300/csrc/sparse_gqa.cu",
               "learned_sparse_attention_gb300/csrc/qsa_device.cuh")


# The inputs a layer step takes from its caller each step (the rest is state
# or configuration that stays on the device).
STEP_INPUTS = ("projected_q", "raw_keys", "positions", "q", "gate", "token_to_req",
               "query_start_loc", "logical_positions", "compressed_slots")


def pack_step_inputs(t: dict, keys, device, pin: bool):
    """One host buffer (pinned if `pin`) and one device buffer holding the
    tensors t[k] for k in keys in 256-byte aligned slots.  Returns (host
    buffer, device buffer, a copy of t whose entries for keys are slices of
    the device buffer); copying the host buffer into the device buffer sets
    all of them."""
    offs, total = [], 0
    for k in keys:
        offs.append(total)
        total += (t[k].numel() * t[k].element_size() + 255) // 256 * 256
    host_buf = torch.empty(total, dtype=torch.uint8, pin_memory=pin)
    dev_buf = torch.empty(total, dtype=torch.uint8, device=device)
    views = dict(t)
    for k, off in zip(keys, offs):
        src = t[k].contiguous()
        nb = src.numel() * src.element_size()
        host_buf[off:off + nb].copy_(src.reshape(-1).view(torch.uint8).cpu())
        views[k] = dev_buf[off:off + nb].view(src.dtype).view(src.shape)
    return host_buf, dev_buf, views


def unit_of(spec) -> str:
    """Rows of a prefill chunk are counted as prefill rows, all others as decode tokens."""
    return "prefill rows/s" if "prefill" in spec.name else "decode tokens/s"


def gqa_source_hash() -> str:
    """Hash of the GQA kernel sources with comments and blank lines removed
    (a comment edit does not change the kernel the counters were taken on)."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in GQA_SOURCES:
        with open(os.path.join(ROOT, f), encoding="utf-8") as fh:
            for line in fh:
                code = re.sub(r"//.*", "", line).rstrip()
                if code:
                    h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------- setup
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, local, backend):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
        return dist
    return None


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64,
                     device=device if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return FALLBACK_PEAKS, "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.device = device
        self.proc = None
        self.lines = []

    def start(self):
        sel = []
        try:
            bus = torch.cuda.get_device_properties(self.device).pci_bus_id
            sel = ["-i", f"{bus}"] if isinstance(bus, str) else []
        except Exception:
            sel = []
        cmd = ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- workload
def build(spec, device):
    wl = W.make_workload(spec, device=device)
    cfg = Q.make_cfg(spec.n_heads, spec.compress_ratio, spec.token_topk, spec.index_dtype,
                     spec.cpage, wl["cos_sin"].shape[0], state_size=spec.S,
                     mrope_section=spec.mrope_section, eps=spec.eps)
    gcfg = Q.make_gqa_cfg(spec.hq, spec.hkv, spec.page, wl["kv"].shape[0])
    mv = max(spec.contexts) // spec.compress_ratio
    packed = torch.empty((spec.rows, spec.packed_width), dtype=torch.int32, device=device)
    out = torch.empty_like(wl["q"])
    ws = torch.empty(Q.workspace_bytes(cfg, gcfg, spec.rows, spec.reqs, mv), dtype=torch.uint8,
                     device=device)
    return wl, cfg, gcfg, mv, packed, out, ws


def algorithmic_bytes(spec, wl, packed):
    """Bytes the method must move in one layer step, and in the sparse GQA
    kernel alone (the dominant kernel)."""
    counts = packed[:, -1].to(torch.int64).cpu().numpy()
    logical = wl["logical_positions"].cpu().numpy().astype(np.int64)
    qsl = wl["query_start_loc"].cpu().numpy()
    e_idx = 1 if spec.index_dtype == W.DTYPE_E4M3 else 2
    D, r = 128, spec.compress_ratio
    pk = packed.cpu().numpy()
    keys = kv = 0
    for q in range(spec.reqs):
        a, b = int(qsl[q]), int(qsl[q + 1])
        if b <= a:
            continue
        keys += ((int(logical[b - 1]) + 1) // r) * D * e_idx
        union = set()
        for row in range(a, b):
            union.update(pk[row, :counts[row]].tolist())
        kv += len(union) * spec.hkv * 2 * D * 2
    rows = spec.rows
    groups = int((wl["compressed_slots"] >= 0).sum().item())
    stage1 = rows * (spec.n_heads * D * 2 + 2 * D * 2 + spec.n_heads * D * e_idx) + groups * (
        (r - 1) * D * 2 + D * e_idx)
    main_io = rows * 3 * spec.hq * D * 2
    packed_io = rows * 2 * 4 * spec.packed_width
    step = keys + kv + stage1 + main_io + packed_io
    gqa = int(counts.sum()) * spec.hkv * 2 * D * 2 + main_io + rows * 4 * spec.packed_width
    return step, gqa, {"compressed_keys": keys, "kv_gather": kv, "stage1": stage1,
                       "main_qkv_gate_out": main_io, "packed": packed_io}


# --------------------------------------------------------------------------- CPU oracle
def oracle_sample(spec, wl, budget_s=15.0, max_rows=None):
    """Time the CPU oracle (as it stands) on whole requests of the workload
    until about budget_s seconds of CPU work; returns (rows/s, rows, secs)."""
    from oracle import qsa_oracle as O
    from tests.oracle_io import OracleState, f64

    st = OracleState(wl, with_kv=False)
    qsl = st.query_start_loc
    done_rows, spent = 0, 0.0
    for req in range(spec.reqs):
        a, b = int(qsl[req]), int(qsl[req + 1])
        if b <= a:
            continue
        # this request's KV blocks on the host, re-indexed 0..n-1 (marshalling)
        L = int(st.logical_positions[b - 1]) + 1
        nblk = -(-L // spec.page)
        blocks = st.block_table[req, :nblk]
        kv = f64(wl["kv"][torch.as_tensor(blocks, device=wl["kv"].device)])
        rows = list(range(a, b))
        sub = dict(
            projected_q=st.projected_q[a:b], raw_keys=st.raw_keys[a:b],
            positions=st.positions[a:b], cos_sin=st.cos_sin, q_norm_w=st.q_norm_w,
            k_norm_w=st.k_norm_w, ring=st.ring.copy(), ring_pos=None if st.ring_pos is None
            else st.ring_pos.copy(), ring_block_table=st.ring_block_table[req:req + 1],
            token_to_req=np.zeros(b - a, dtype=np.int64), query_start_loc=np.array([0, b - a]),
            logical_positions=st.logical_positions[a:b], ccache=st.ccache.copy(),
            compressed_slots=st.compressed_slots[a:b],
            cblock_table=st.cblock_table[req:req + 1], q=st.q[a:b], kv=kv,
            block_table=np.arange(nblk)[None, :], page=spec.page, gate=st.gate[a:b])
        t0 = time.perf_counter()
        O.layer_step(st.cfg, **sub)
        spent += time.perf_counter() - t0
        done_rows += len(rows)
        if spent >= budget_s or (max_rows and done_rows >= max_rows):
            break
    return done_rows / spent, done_rows, spent


def cpu_threads():
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


# --------------------------------------------------------------------------- arms
def run_reference(args):
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    spec = W.named_spec(args.workload)
    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    wl = W.make_workload(spec, device=device)
    for _ in range(args.warmup):
        oracle_sample(spec, wl, budget_s=0.0, max_rows=1)
    times, rows_total = [], 0
    t_all = 0.0
    for _ in range(args.steps):
        rate, rows, secs = oracle_sample(spec, wl, budget_s=args.ref_budget)
        times.append(secs)
        rows_total += rows
        t_all += secs
    value = rows_total / t_all
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit_of(spec),
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * t_all / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.name, "rows": spec.rows, "reqs": spec.reqs},
        "cpu_baseline": {"value": value, "unit": unit_of(spec), "cores": cpu_threads(),
                         "kind": "oracle",
                         "sample": f"whole requests of {spec.name} until ~{args.ref_budget}s "
                                   f"of CPU work per step ({rows_total} rows in total)"},
        "e2e": {"value": value, "unit": unit_of(spec), "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def prefill_report(device, steps, flush, drain):
    """The chunked-prefill workload (one request, 16384 new rows after a
    32768-token prefix): layer-step rows/s, and the index-logits kernel alone
    against the fp8 tensor peak (FLOPs = visible keys x heads x 128 x 2)."""
    spec = W.named_spec("chunked_prefill")
    wl, cfg, gcfg, mv, packed, out, ws = build(spec, device)
    sargs = Q.step_args(wl.t, packed, out, mv)
    stream = torch.cuda.current_stream()
    for _ in range(2):
        Q.layer_step(cfg, gcfg, sargs, ws)
    torch.cuda.synchronize()

    def timed(fn):
        ts = []
        for i in range(steps):
            flush_l2(flush, drain, i)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return statistics.median(ts)

    step_ms = timed(lambda: Q.layer_step(cfg, gcfg, sargs, ws))
    t = wl.t
    q_idx = torch.empty((spec.rows, spec.n_heads, 128),
                        dtype=torch.uint8 if spec.index_dtype == W.DTYPE_E4M3 else torch.bfloat16,
                        device=device)
    Q.compress(cfg, t["projected_q"], q_idx, t["raw_keys"], t["positions"], t["cos_sin"],
               t["q_norm_w"], t["k_norm_w"], t["ring"], t.get("ring_pos"), t["ring_block_table"],
               t["token_to_req"], t["query_start_loc"], t["logical_positions"], t["ccache"],
               t["compressed_slots"])
    logits = torch.empty((spec.rows, (mv + 3) // 4 * 4), dtype=torch.float32, device=device)
    lws = torch.empty(256, dtype=torch.uint8, device=device)
    logits_ms = timed(lambda: Q.index_logits(cfg, q_idx, t["ccache"], t["cblock_table"],
                                             t["token_to_req"], t["query_start_loc"],
                                             t["logical_positions"], logits, mv, lws))
    if Q.check_errors() != 0:
        raise RuntimeError("device error word set during the prefill measurement")
    vis = ((t["logical_positions"].long() + 1) // spec.compress_ratio).clamp(min=0)
    flops = float(vis.sum()) * spec.n_heads * 128 * 2
    peaks, peak_kind = load_peaks()
    fp8 = 2.0 * float(peaks["bf16_tflops"])
    tf = flops / (logits_ms / 1000.0) / 1e12
    res = {"workload": spec.name, "rows": spec.rows, "steps": steps,
           "ms_per_step": step_ms, "value": spec.rows / (step_ms / 1000.0), "unit": "prefill rows/s",
           "index_logits": {"bound": "tensor", "achieved": tf, "peak": fp8, "unit": "TFLOP/s",
                            "frac": tf / fp8, "kernel_ms": logits_ms, "flops_per_launch": flops,
                            "peak_source": f"2 x {peak_kind} bf16_tflops (nominal fp8/bf16 ratio)"}}
    del wl, packed, out, ws, logits, q_idx
    torch.cuda.empty_cache()
    return res


def run_ours(args):
    world, rank, local = dist_env()
    dist = init_dist(world, local, "nccl")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    spec = W.named_spec(args.workload)
    Q.load()
    wl, cfg, gcfg, mv, packed, out, ws = build(spec, device)
    sargs = Q.step_args(wl.t, packed, out, mv)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
    drain = torch.ones(DRAIN_BYTES // 4, dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream()

    def step_direct():
        Q.layer_step(cfg, gcfg, sargs, ws)

    for _ in range(args.warmup):
        step_direct()
    torch.cuda.synchronize()
    if Q.check_errors() != 0:
        raise RuntimeError("device error word set during warm-up")
    # The timed step replays one CUDA-graph capture of the same C-ABI call
    # (the call makes no host synchronisation, so it captures as is).
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device=device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        step_direct()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(graph):
        step_direct()
    torch.cuda.synchronize()

    def step():
        graph.replay()

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region: K steps, L2 flushed between them, events around each step
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(device)
    clocks.start()
    barrier(dist, device)
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush_l2(flush, drain, i)
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(dist, device)
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    t_total = max_over_ranks(dist, sum(step_ms), device)
    ms_per_step = t_total / args.steps
    value = world * spec.rows * args.steps / (t_total / 1000.0)

    # ---- per-kernel timing of the dominant kernel (stage 4) on the same stream
    ld = (mv + 3) // 4 * 4
    gws = ws  # the layer-step workspace is large enough for every stage call
    gev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        flush_l2(flush, drain, i)
        gev[i][0].record(stream)
        Q.sparse_gqa(gcfg, wl["q"], wl["kv"], wl["block_table"], packed, wl["token_to_req"],
                     wl["gate"], out, gws)
        gev[i][1].record(stream)
    torch.cuda.synchronize()
    gqa_ms = statistics.mean(a.elapsed_time(b) for a, b in gev)
    step_bytes, gqa_bytes, parts = algorithmic_bytes(spec, wl, packed)
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    achieved = gqa_bytes / (gqa_ms / 1000.0) / 1e9
    step_gbs = step_bytes / (ms_per_step / 1000.0) / 1e9

    # ---- end to end: host buffers in, output back, through the same C-ABI call.
    # The step's inputs sit in one pinned host buffer (256-byte aligned
    # slots) and travel in one copy to one device buffer whose slices are the
    # step's input tensors.
    host_buf, dev_buf, t_e2e = pack_step_inputs(wl.t, STEP_INPUTS, device, pin=True)
    sargs_e2e = Q.step_args(t_e2e, packed, out, mv)
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(wl.t[k].numel() * wl.t[k].element_size() for k in STEP_INPUTS)
    d2h = out_host.numel() * out_host.element_size()
    eev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    for i in range(args.steps):
        flush_l2(flush, drain, i)
        eev[i][0].record(stream)
        dev_buf.copy_(host_buf, non_blocking=True)
        Q.layer_step(cfg, gcfg, sargs_e2e, ws)
        out_host.copy_(out, non_blocking=True)
        eev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(dist, sum(a.elapsed_time(b) for a, b in eev), device) / args.steps
    e2e_value = world * spec.rows / (e2e_ms / 1000.0)
    if Q.check_errors() != 0:
        raise RuntimeError("device error word set during the timed steps")

    launches_per_step = Q.step_launches(cfg, gcfg, spec.rows, spec.reqs)
    prefill = None
    if rank == 0 and world == 1 and spec.name == "decode_batch" and not args.no_prefill:
        prefill = prefill_report(device, 3, flush, drain)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows_done, secs = oracle_sample(spec, wl, budget_s=args.ref_budget)
        cpu = {"value": rate, "unit": unit_of(spec), "cores": cpu_threads(), "kind": "oracle",
               "sample": f"{rows_done} rows (whole requests) of {spec.name}, {secs:.1f} s"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": unit_of(spec), "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3+bf16" if spec.index_dtype == W.DTYPE_E4M3 else "bf16",
            "data": "synthetic",
            "config": {"workload": spec.name, "rows": spec.rows, "reqs": spec.reqs,
                       "contexts": f"{min(spec.contexts)}..{max(spec.contexts)}",
                       "indexer": f"{spec.n_heads}x128 {'e4m3' if spec.index_dtype else 'bf16'}"
                                  f" r={spec.compress_ratio} topk={spec.token_topk}",
                       "gqa": f"{spec.hq}q/{spec.hkv}kv x128 bf16 page {spec.page}",
                       "parallelism": f"replicas x{world}",
                       "l2": f"flushed between steps ({FLUSH_BYTES >> 20} MiB write, then a "
                             f"{DRAIN_BYTES >> 20} MiB read to evict the written lines)"},
            "roofline": {"bound": "hbm", "kernel": "qsa sparse GQA (stage 4)",
                         "achieved": achieved, "peak": hbm, "unit": "GB/s",
                         "frac": achieved / hbm,
                         "traffic": (GQA_TRAFFIC.get(gqa_source_hash())
                                     if spec.name == "decode_batch" else None),
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "algorithmic_bytes_per_launch": gqa_bytes,
                         "kernel_ms": gqa_ms},
            "step_roofline": {"bound": "hbm", "achieved": step_gbs, "peak": hbm, "unit": "GB/s",
                              "frac": step_gbs / hbm, "algorithmic_bytes_per_step": step_bytes,
                              "parts": parts},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": unit_of(spec), "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
            "gpu_launches": launches_per_step * args.steps,
            "launch": "CUDA graph of one qsa_layer_step call (value); direct calls (e2e)",
            "clocks": clk,
            "prefill": prefill,
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_batch", choices=list(W.NAMED))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefill", action="store_true",
                    help="skip the chunked-prefill rows/s and index-logits measurement")
    ap.add_argument("--ref-budget", type=float, default=15.0)
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
