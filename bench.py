"""QSA layer-step benchmark on GB300.

Default workload: the decode batch (64 requests, contexts uniform in
[8192, 32768], one query row each; indexer 32 x 128 e4m3, compress_ratio 4,
token_topk 2048; GQA 32q / 4kv x 128 bf16, KV block 64), the configuration
the decode tokens/s metric is quoted on.  One step = one call of
qsa_layer_step (all four stages) over that batch.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-cpu-baseline] [--no-extra]

The default run also reports, in the same JSON line, the other workloads of
the metric: the chunked prefill (rows/s, the index-logits kernel against a
dense-fp8 peak measured in the same run, sparse GQA against its bf16 FLOPs),
the long-context decode and the MTP verify draft (step 0 plus three skip_topk
steps captured as one CUDA graph of qsa_mtp_steps).

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
GQA_TRAFFIC = {"3d78878b20f11825": 270419968 + 3646464}
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


def config_of(spec, world: int) -> dict:
    """The workload description printed by both arms."""
    return {"workload": spec.name, "rows": spec.rows, "reqs": spec.reqs,
            "contexts": f"{min(spec.contexts)}..{max(spec.contexts)}",
            "indexer": f"{spec.n_heads}x128 {'e4m3' if spec.index_dtype else 'bf16'}"
                       f" r={spec.compress_ratio} topk={spec.token_topk}",
            "gqa": f"{spec.hq}q/{spec.hkv}kv x128 "
                   f"{'e4m3 (static scales)' if spec.kv_dtype else 'bf16'} page {spec.page}",
            "parallelism": f"replicas x{world}",
            "l2": f"flushed between steps ({FLUSH_BYTES >> 20} MiB write, then a "
                  f"{DRAIN_BYTES >> 20} MiB read to evict the written lines)"}


def measure_fp8_peak(device, n=8192, reps=10):
    """Dense e4m3 x e4m3 -> bf16 GEMM throughput of the library GEMM
    (torch._scaled_mm, n^3, best of `reps`, CUDA events): the fp8 tensor
    peak the prefill index-logits kernel is quoted against."""
    try:
        a = torch.randn((n, n), device=device).to(torch.float8_e4m3fn)
        b = torch.randn((n, n), device=device).to(torch.float8_e4m3fn).t()  # column-major
        one = torch.ones((), device=device, dtype=torch.float32)
        fn = lambda: torch._scaled_mm(a, b, scale_a=one, scale_b=one, out_dtype=torch.bfloat16)
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        best = float("inf")
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        del a, b
        torch.cuda.empty_cache()
        return {"fp8_tflops": 2.0 * n ** 3 / (best / 1000.0) / 1e12, "ms": best,
                "how": f"torch._scaled_mm e4m3 {n}^3 -> bf16, best of {reps}, CUDA events"}
    except Exception as e:  # no fp8 GEMM in this torch build
        return {"fp8_tflops": None, "error": str(e)[:200]}


class CpuClock:
    """Wall and process CPU time around a region: cores = CPU s / wall s is
    the number of cores the region actually kept busy (BLAS threads included)."""

    def __init__(self):
        self.wall = self.cpu = 0.0

    def __enter__(self):
        self.w0, self.c0 = time.perf_counter(), time.process_time()
        return self

    def __exit__(self, *exc):
        self.wall += time.perf_counter() - self.w0
        self.cpu += time.process_time() - self.c0

    @property
    def cores(self) -> float:
        return round(self.cpu / self.wall, 2) if self.wall > 0 else 0.0


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
    ks = spec.kv_scale if spec.kv_dtype == W.DTYPE_E4M3 else 1.0
    gcfg = Q.make_gqa_cfg(spec.hq, spec.hkv, spec.page, wl["kv"].shape[0], kv_dtype=spec.kv_dtype,
                          k_scale=ks, v_scale=ks)
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
    e_kv = 1 if spec.kv_dtype == W.DTYPE_E4M3 else 2
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
        kv += len(union) * spec.hkv * 2 * D * e_kv
    rows = spec.rows
    groups = int((wl["compressed_slots"] >= 0).sum().item())
    stage1 = rows * (spec.n_heads * D * 2 + 2 * D * 2 + spec.n_heads * D * e_idx) + groups * (
        (r - 1) * D * 2 + D * e_idx)
    if spec.main_prep:  # projection rows in; q, gate and the rows' K/V out
        stage1 += rows * ((2 * spec.hq + 2 * spec.hkv) * D * 2 + 2 * spec.hq * D * 2
                          + spec.hkv * 2 * D * e_kv)
    main_io = rows * 3 * spec.hq * D * 2
    packed_io = rows * 2 * 4 * spec.packed_width
    step = keys + kv + stage1 + main_io + packed_io
    gqa = int(counts.sum()) * spec.hkv * 2 * D * e_kv + main_io + rows * 4 * spec.packed_width
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
    done_rows = 0
    clock = CpuClock()
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
        with clock:
            O.layer_step(st.cfg, **sub)
        done_rows += len(rows)
        if clock.wall >= budget_s or (max_rows and done_rows >= max_rows):
            break
    return done_rows / clock.wall, done_rows, clock.wall, clock.cores


def oracle_prefill_sample(spec, wl, nsample=192, seed=0):
    """The oracle on the chunked prefill: stage 1's pooling of every group the
    chunk completes (timed in full), then query prep, selection and sparse
    GQA of `nsample` seeded rows, extrapolated linearly to all rows.
    Returns (rows/s, seconds of the extrapolated step, cores, sample text)."""
    from oracle import qsa_oracle as O
    from tests.oracle_io import OracleState, f64

    st = OracleState(wl, with_kv=False)
    L = int(st.logical_positions[-1]) + 1
    nblk = -(-L // spec.page)
    kv = f64(wl["kv"][torch.as_tensor(st.block_table[0, :nblk], device=wl["kv"].device)])
    rows = np.sort(np.random.default_rng(seed).choice(spec.rows, size=nsample, replace=False))
    c1, c2 = CpuClock(), CpuClock()
    with c1:
        O.compress_stage(st.cfg, projected_q=None, raw_keys=st.raw_keys, positions=st.positions,
                         cos_sin=st.cos_sin, q_norm_w=st.q_norm_w, k_norm_w=st.k_norm_w,
                         ring=st.ring, ring_pos=st.ring_pos,
                         ring_block_table=st.ring_block_table, token_to_req=st.token_to_req,
                         query_start_loc=st.query_start_loc,
                         logical_positions=st.logical_positions, ccache=st.ccache,
                         compressed_slots=st.compressed_slots)
    with c2:
        for row in rows:
            q_idx = O.prep_query(st.cfg, st.projected_q[row], st.positions[row], st.cos_sin,
                                 st.q_norm_w)
            _, _, packed = O.select_row(st.cfg, q_idx, st.ccache, st.cblock_table[0],
                                        int(st.logical_positions[row]))
            n = int(packed[-1])
            O.sparse_gqa_row(st.q[row], kv, np.arange(nblk), packed[:n], spec.page, st.gate[row])
    total = c1.wall + c2.wall * spec.rows / nsample
    cores = round((c1.cpu + c2.cpu) / (c1.wall + c2.wall), 2)
    text = (f"stage-1 pooling of all {int((st.compressed_slots >= 0).sum())} groups "
            f"({c1.wall:.1f} s) + query prep, selection and sparse GQA of {nsample} seeded rows "
            f"({c2.wall:.1f} s) extrapolated x{spec.rows / nsample:.1f} to {spec.rows} rows")
    return spec.rows / total, total, cores, text


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
    rows_total, t_all, cores = 0, 0.0, []
    for _ in range(args.steps):
        rate, rows, secs, c = oracle_sample(spec, wl, budget_s=args.ref_budget)
        rows_total += rows
        t_all += secs
        cores.append(c)
    value = rows_total / t_all
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit_of(spec),
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * t_all / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(spec, 1),
        "cpu_baseline": {"value": value, "unit": unit_of(spec), "cores": max(cores),
                         "kind": "oracle",
                         "sample": f"whole requests of {spec.name} until ~{args.ref_budget}s "
                                   f"of CPU work per step ({rows_total} rows in total)"},
        "e2e": {"value": value, "unit": unit_of(spec), "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def capture(fn, device):
    """One CUDA graph of fn (a sequence of C-ABI calls without host sync)."""
    stream = torch.cuda.current_stream()
    side = torch.cuda.Stream(device=device)
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        fn()
    torch.cuda.synchronize()
    return graph


def timed(fn, steps, flush, drain):
    """Per-call CUDA-event times (ms) on the current stream, the L2 flushed
    and drained before every call, outside the events."""
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    for i in range(steps):
        flush_l2(flush, drain, i)
        ev[i][0].record(stream)
        fn()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def gqa_kernel_ms(wl, gcfg, packed, out, ws, steps, flush, drain):
    """The sparse GQA stage alone (the dominant kernel of a decode step)."""
    ts = timed(lambda: Q.sparse_gqa(gcfg, wl["q"], wl["kv"], wl["block_table"], packed,
                                    wl["token_to_req"], wl["gate"], out, ws), steps, flush, drain)
    return statistics.mean(ts)


def hbm_line(achieved_bytes, ms, hbm):
    gbs = achieved_bytes / (ms / 1000.0) / 1e9
    return {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
            "algorithmic_bytes": achieved_bytes, "ms": ms}


def decode_report(name, device, steps, warmup, flush, drain, hbm):
    """A decode workload other than the headline one: graph-replayed layer
    step (tokens/s, step against HBM) and its sparse GQA kernel alone."""
    spec = W.named_spec(name)
    wl, cfg, gcfg, mv, packed, out, ws = build(spec, device)
    main = Q.main_prep(wl.t, spec.eps) if spec.main_prep else None
    sargs = Q.step_args(wl.t, packed, out, mv, main=main)
    for _ in range(warmup):
        Q.layer_step(cfg, gcfg, sargs, ws)
    graph = capture(lambda: Q.layer_step(cfg, gcfg, sargs, ws), device)
    for _ in range(warmup):
        graph.replay()
    ms = statistics.mean(timed(graph.replay, steps, flush, drain))
    g_ms = gqa_kernel_ms(wl, gcfg, packed, out, ws, steps, flush, drain)
    if Q.check_errors() != 0:
        raise RuntimeError(f"device error word set during {name}")
    step_bytes, gqa_bytes, parts = algorithmic_bytes(spec, wl, packed)
    res = {"workload": name, "rows": spec.rows, "ms_per_step": ms, "steps": steps,
           "value": spec.rows / (ms / 1000.0), "unit": "decode tokens/s",
           "step_roofline": hbm_line(step_bytes, ms, hbm), "parts": parts,
           "gqa_roofline": hbm_line(gqa_bytes, g_ms, hbm),
           "launches_per_step": Q.step_launches(cfg, gcfg, spec.rows, spec.reqs)}
    del wl, packed, out, ws, graph
    torch.cuda.empty_cache()
    return res


def mtp_report(device, steps, warmup, flush, drain, hbm):
    """The MTP verify draft with MRoPE: step 0 selects, steps 1-3 reuse its
    packed buffer (skip_topk) with fresh per-step inputs.  The four steps are
    one qsa_mtp_steps call captured as one CUDA graph and replayed after an
    L2 flush; tokens/s counts every row once per step.  Step 0 and a skip
    step are also timed alone for the breakdown."""
    spec = W.named_spec("mtp_mrope")
    k = spec.mtp_steps
    wl, cfg, gcfg, mv, packed, out, ws = build(spec, device)
    per_step, outs = [], []
    for s in range(k):
        fresh = W.make_workload(spec, device=device, step=s, with_caches=False)
        t = dict(wl.t)
        for n in ("projected_q", "raw_keys", "positions", "q", "gate"):
            t[n] = fresh[n]
        outs.append(torch.empty_like(wl["q"]))
        per_step.append(Q.step_args(t, packed, outs[-1], mv))
    draft = lambda: Q.mtp_steps(cfg, gcfg, per_step, ws)
    for _ in range(warmup):
        draft()
    g_all = capture(draft, device)
    g0 = capture(lambda: Q.layer_step(cfg, gcfg, per_step[0], ws), device)
    g1 = capture(lambda: Q.layer_step(cfg, gcfg, per_step[1], ws, skip_topk=True), device)
    for _ in range(warmup):
        g_all.replay()
    cycle_ms = statistics.mean(timed(g_all.replay, steps, flush, drain))
    s0_ms = statistics.mean(timed(g0.replay, steps, flush, drain))
    s1_ms = statistics.mean(timed(g1.replay, steps, flush, drain))
    if Q.check_errors() != 0:
        raise RuntimeError("device error word set during the MTP draft")
    step_bytes, gqa_bytes, parts = algorithmic_bytes(spec, wl, packed)
    res = {"workload": spec.name, "rows": spec.rows, "draft_steps": k, "steps": steps,
           "draft_ms": cycle_ms, "value": k * spec.rows / (cycle_ms / 1000.0),
           "unit": "decode tokens/s", "step0_ms": s0_ms, "skip_step_ms": s1_ms,
           "step0_roofline": hbm_line(step_bytes, s0_ms, hbm), "parts_step0": parts,
           "launch": "one CUDA graph of qsa_mtp_steps (4 layer steps)",
           "launches_per_draft": Q.step_launches(cfg, gcfg, spec.rows, spec.reqs)
           + (k - 1) * Q.step_launches(cfg, gcfg, spec.rows, spec.reqs, skip_topk=True)}
    del wl, packed, out, ws, outs, per_step, g_all, g0, g1
    torch.cuda.empty_cache()
    return res


def projection_report(device, steps, flush, drain, bf16, hbm, hidden=4096):
    """The fused qkv + indexer projection GEMM of a 32q/4kv x 128 layer with
    a 32-head indexer over hidden = 4096 (synthetic weights; the pages do not
    give hidden_size), at the decode batch's 64 rows (bound by reading the
    weights) and the prefill chunk's 16384 rows (bound by the tensor cores)."""
    qc, iq, ik = (2 * 32 + 2 * 4) * 128, 32 * 128, 128
    ncols = qc + iq + ik
    g = torch.Generator(device=device).manual_seed(11)
    w = (torch.randn((ncols, hidden), generator=g, device=device) / hidden ** 0.5).to(torch.bfloat16)
    res = {"hidden": hidden, "columns": {"qkv": qc, "index_q": iq, "index_k": ik},
           "weights": "synthetic N(0, 1/hidden)"}
    for name, rows in (("decode_batch", 64), ("chunked_prefill", 16384)):
        x = torch.randn((rows, hidden), generator=g, device=device).to(torch.bfloat16)
        outs = [torch.empty((rows, c), dtype=torch.bfloat16, device=device) for c in (qc, iq, ik)]
        fn = lambda: Q.qkv_index_proj(x, w, *outs)
        fn()
        torch.cuda.synchronize()
        ms = statistics.median(timed(fn, steps, flush, drain))
        flops = 2.0 * rows * hidden * ncols
        nbytes = (ncols * hidden + rows * hidden + rows * ncols) * 2
        tf = flops / (ms / 1000.0) / 1e12
        gbs = nbytes / (ms / 1000.0) / 1e9
        res[name] = {"rows": rows, "ms": ms, "tflops": tf, "frac_bf16": tf / bf16,
                     "gbs": gbs, "frac_hbm": gbs / hbm, "flops": flops, "bytes": nbytes}
        del x, outs
    if Q.check_errors() != 0:
        raise RuntimeError("device error word set during the projection measurement")
    del w
    torch.cuda.empty_cache()
    return res


def prefill_report(device, steps, flush, drain, fp8, bf16, cpu_baseline):
    """The chunked-prefill workload (one request, 16384 new rows after a
    32768-token prefix): layer-step rows/s; the index-logits kernel alone
    against the measured dense-fp8 peak (FLOPs = visible keys x heads x 128
    x 2); the sparse GQA kernel alone against the bf16 peak (FLOPs = 4 x 128
    x Hq x selected tokens)."""
    spec = W.named_spec("chunked_prefill")
    wl, cfg, gcfg, mv, packed, out, ws = build(spec, device)
    sargs = Q.step_args(wl.t, packed, out, mv)
    for _ in range(2):
        Q.layer_step(cfg, gcfg, sargs, ws)
    torch.cuda.synchronize()
    step_ms = statistics.median(timed(lambda: Q.layer_step(cfg, gcfg, sargs, ws), steps,
                                      flush, drain))
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
    logits_ms = statistics.median(timed(
        lambda: Q.index_logits(cfg, q_idx, t["ccache"], t["cblock_table"], t["token_to_req"],
                               t["query_start_loc"], t["logical_positions"], logits, mv, lws),
        steps, flush, drain))
    gqa_ms = statistics.median(timed(
        lambda: Q.sparse_gqa(gcfg, wl["q"], wl["kv"], wl["block_table"], packed,
                             wl["token_to_req"], wl["gate"], out, ws), steps, flush, drain))
    if Q.check_errors() != 0:
        raise RuntimeError("device error word set during the prefill measurement")
    vis = ((t["logical_positions"].long() + 1) // spec.compress_ratio).clamp(min=0)
    flops = float(vis.sum()) * spec.n_heads * 128 * 2
    tf = flops / (logits_ms / 1000.0) / 1e12
    n_sel = float(packed[:, -1].long().sum())
    gflops = 4.0 * 128 * spec.hq * n_sel
    gtf = gflops / (gqa_ms / 1000.0) / 1e12
    res = {"workload": spec.name, "rows": spec.rows, "steps": steps,
           "ms_per_step": step_ms, "value": spec.rows / (step_ms / 1000.0), "unit": "prefill rows/s",
           "index_logits": {"bound": "tensor", "achieved": tf, "peak": fp8["fp8_tflops"],
                            "unit": "TFLOP/s",
                            "frac": tf / fp8["fp8_tflops"] if fp8.get("fp8_tflops") else None,
                            "kernel_ms": logits_ms, "flops_per_launch": flops,
                            "peak_source": "dense fp8 measured in this run: " + fp8.get("how", "")},
           "sparse_gqa": {"bound": "tensor", "achieved": gtf, "peak": bf16, "unit": "TFLOP/s",
                          "frac": gtf / bf16, "kernel_ms": gqa_ms, "flops_per_launch": gflops,
                          "peak_source": "MEASURED_PEAKS bf16_tflops (burst)"}}
    if cpu_baseline:
        rate, secs, cores, text = oracle_prefill_sample(spec, wl)
        res["cpu_baseline"] = {"value": rate, "unit": "prefill rows/s", "cores": cores,
                               "kind": "oracle", "sample": text}
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
    graph = capture(step_direct, device)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()

    # ---- timed region: K steps, L2 flushed between them, events around each step
    clocks = ClockSampler(device)
    clocks.start()
    barrier(dist, device)
    torch.cuda.synchronize()
    step_ms = timed(graph.replay, args.steps, flush, drain)
    barrier(dist, device)
    clk = clocks.stop()
    t_total = max_over_ranks(dist, sum(step_ms), device)
    ms_per_step = t_total / args.steps
    value = world * spec.rows * args.steps / (t_total / 1000.0)

    # ---- the dominant kernel (stage 4) alone, on the same stream
    gqa_ms = gqa_kernel_ms(wl, gcfg, packed, out, ws, args.steps, flush, drain)
    step_bytes, gqa_bytes, parts = algorithmic_bytes(spec, wl, packed)
    peaks, peak_kind = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    achieved = gqa_bytes / (gqa_ms / 1000.0) / 1e9
    step_gbs = step_bytes / (ms_per_step / 1000.0) / 1e9

    # ---- end to end: host buffers in, output back, through the same C-ABI call.
    # The caller produces the step's inputs in one pinned host staging buffer
    # (256-byte aligned slots); they travel in one copy to one device buffer
    # whose slices are the step's input tensors.
    host_buf, dev_buf, t_e2e = pack_step_inputs(wl.t, STEP_INPUTS, device, pin=True)
    sargs_e2e = Q.step_args(t_e2e, packed, out, mv)
    out_host = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    h2d = sum(wl.t[k].numel() * wl.t[k].element_size() for k in STEP_INPUTS)
    d2h = out_host.numel() * out_host.element_size()

    def e2e_step():
        dev_buf.copy_(host_buf, non_blocking=True)
        Q.layer_step(cfg, gcfg, sargs_e2e, ws)
        out_host.copy_(out, non_blocking=True)

    e2e_ms = max_over_ranks(dist, sum(timed(e2e_step, args.steps, flush, drain)), device) / args.steps
    e2e_value = world * spec.rows / (e2e_ms / 1000.0)
    if Q.check_errors() != 0:
        raise RuntimeError("device error word set during the timed steps")

    launches_per_step = Q.step_launches(cfg, gcfg, spec.rows, spec.reqs)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rate, rows_done, secs, cores = oracle_sample(spec, wl, budget_s=args.ref_budget)
        cpu = {"value": rate, "unit": unit_of(spec), "cores": cores, "kind": "oracle",
               "sample": f"{rows_done} rows (whole requests) of {spec.name}, {secs:.1f} s; "
                         f"cores = process CPU seconds / wall seconds"}
    del wl, packed, out, ws, graph, host_buf, dev_buf, t_e2e, sargs, sargs_e2e
    torch.cuda.empty_cache()

    extra = None
    if rank == 0 and world == 1 and spec.name == "decode_batch" and not args.no_extra:
        fp8 = measure_fp8_peak(device)
        bf16 = float(peaks["bf16_tflops"])
        extra = {"fp8_peak": fp8,
                 "prefill": prefill_report(device, 3, flush, drain, fp8, bf16,
                                           not args.no_cpu_baseline),
                 "long_decode": decode_report("long_decode", device, 10, 3, flush, drain, hbm),
                 "decode_batch_fp8kv": decode_report("decode_batch_fp8kv", device, 10, 3, flush,
                                                     drain, hbm),
                 "decode_batch_prepare": decode_report("decode_batch_prepare", device, 10, 3,
                                                       flush, drain, hbm),
                 "mtp_mrope": mtp_report(device, 10, 3, flush, drain, hbm),
                 "qkv_index_projection": projection_report(device, 5, flush, drain, bf16, hbm)}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": unit_of(spec), "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "e4m3+bf16" if spec.index_dtype == W.DTYPE_E4M3 else "bf16",
            "data": "synthetic",
            "config": config_of(spec, world),
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
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "inputs": "produced by the caller in one pinned staging buffer (no host "
                              "repacking); one H2D copy, the C-ABI call, one D2H copy per step"},
            "gpu_launches": launches_per_step * args.steps,
            "launch": "CUDA graph of one qsa_layer_step call (value); direct calls (e2e)",
            "clocks": clk,
            "other_workloads": extra,
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
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the other workloads (prefill, long decode, MTP draft) and the "
                         "fp8 peak probe in the default run")
    ap.add_argument("--ref-budget", type=float, default=15.0)
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
