"""Benchmark: verification attention on one GB300 (or N replicas).

One step = one spec_verify_attn call over the whole batch of the headline
workload (Llama-3-8B-shaped layer: B=4, L=32768, 32 query / 8 KV heads,
d=128, N=64-node random draft tree): the split-KV cache kernel plus the
log-sum-exp merge fused with the tree-masked draft block.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload C] [--impl native|reference]

Prints one JSON line (rank 0). `value` is achieved HBM TB/s = algorithmic K/V
bytes of all ranks / (max over ranks of the time per step); ms_per_step is the
step latency. Inputs (512 MiB of K/V) exceed the 129 MB L2, so no flush is
needed between steps. `--impl reference` times the CPU oracle (fp64, all host
cores) on a bounded sample of rows of the same workload.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from speculative_decoding_verification_77_gb300 import workloads as W  # noqa: E402

METRIC = "verify-attention µs/step and achieved HBM TB/s (% of 8 TB/s) at B=4, L=32k"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0

# DRAM bytes (read + written) per launch of the cache kernel from one ncu
# capture, keyed by the sha256 of the kernel source it was taken on and the
# workload; a changed kernel reports null. The captures and their commands are
# summarised in profiles/cache_attn_tc_llama3-8b-layer_ncu.md and
# profiles/cache_attn_tc_sparse-hybrid_ncu.md.
NCU_TRAFFIC = {
    ("cdb83f410f5b09e1", "llama3-8b-layer-B4-L32k-N64-tree"): 540_644_864 + 8_498_432,
    ("cdb83f410f5b09e1", "sparse-hybrid-B16-L32k-k2048-N8-chain"): 136_158_464 + 6_797_824,
}


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for fn in ("attn_tc.cu", "tc_pipe.cuh", "sm100.cuh", "common.cuh"):
        with open(os.path.join(ROOT, "speculative_decoding_verification_77_gb300", "csrc", fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled in the background."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        self.file.flush()
        self.file.seek(0)
        rows = []
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                whole, _, frac = parts[0].partition(".")
                ts = time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + float("0." + (frac or "0"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for r in rows if t0 - 1.0 <= r[0] <= t1 + 1.0]
        window = "timed" if inside else "bench"
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "window": window}


# ---------------------------------------------------------------------------
# native arm


def oracle_select_seconds(x) -> float:
    """Seconds the CPU oracle takes for the whole selection of a sparse workload (0 if dense)."""
    import oracle

    w = x["workload"]
    if not w.sparse:
        return 0.0
    t = time.perf_counter()
    oracle.select(x["draft_score"], x["target_score"], sink=w.sink, window=w.window, top_m=w.top_m,
                  budget=w.budget)
    return time.perf_counter() - t


def oracle_rows(x, rows, idx):
    import oracle

    oracle.attend(x["q"], x["k_cache"], x["v_cache"], x["k_draft"], x["v_draft"], x["parent"],
                  scale=x["scale"], rows=rows, idx=idx)


def oracle_baseline(x, rows_target_s: float = 10.0, max_rows: int | None = None):
    """Time the CPU oracle (as it stands) on a sample of rows; extrapolate to one step.

    A sparse step is the oracle selection of every sequence (timed whole) plus
    sparse attention over the chosen indices (timed on sampled rows)."""
    import oracle

    w = x["workload"]
    total_rows = w.B * w.N * w.Hq
    sel_s = oracle_select_seconds(x)
    idx = None
    if w.sparse:
        idx = oracle.select(x["draft_score"], x["target_score"], sink=w.sink, window=w.window,
                            top_m=w.top_m, budget=w.budget)[0]
    rng = np.random.default_rng(0)
    n = 16
    elapsed = 0.0
    done = 0
    while True:
        rows = rng.choice(total_rows, size=min(n, total_rows - done), replace=False)
        t = time.perf_counter()
        oracle_rows(x, rows, idx)
        dt = time.perf_counter() - t
        elapsed += dt
        done += len(rows)
        if elapsed >= rows_target_s or done >= total_rows or (max_rows and done >= max_rows):
            break
        n = min(total_rows, max(n, int(len(rows) * (rows_target_s - elapsed) / max(dt, 1e-3))))
    step_s = sel_s + elapsed / done * total_rows
    cores = len(os.sched_getaffinity(0))
    sel = f"selection of all {w.B} sequences {sel_s:.2f} s + " if w.sparse else ""
    return {"value": w.kv_bytes() / step_s / 1e12, "unit": "TB/s", "cores": cores, "kind": "oracle",
            "sample": f"{sel}{done} of {total_rows} output rows (fp64, OpenMP over rows), {elapsed:.1f} s, "
                      f"extrapolated to one step: {step_s:.2f} s/step"}


def run_native(args, ws_, rank, local):
    from speculative_decoding_verification_77_gb300 import ops

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = W.workload(args.workload)
    x = W.make_inputs(w)
    names = ["q", "k_cache", "v_cache", "k_draft", "v_draft", "parent"]
    if w.sparse:
        names += ["draft_score", "target_score"]
    host = {k: x[k].pin_memory() for k in names}
    g = {k: host[k].to(dev, non_blocking=True) for k in names}
    torch.cuda.synchronize()
    scale = x["scale"]
    out = torch.empty((w.B, w.N, w.Hq, w.d), dtype=torch.float32, device=dev)
    lse = torch.empty((w.B, w.N, w.Hq), dtype=torch.float32, device=dev)
    idx = torch.empty((w.B, max(w.budget, 1)), dtype=torch.int32, device=dev)
    cnt = torch.empty((w.B,), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(t):
        if w.sparse:
            ops.select_topk(t["draft_score"], t["target_score"], sink=w.sink, window=w.window, top_m=w.top_m,
                            budget=w.budget, idx=idx, count=cnt)
            return ops.verify_attn_sparse(t["q"], t["k_cache"], t["v_cache"], t["k_draft"], t["v_draft"],
                                          t["parent"], idx, scale=scale, out=out, lse=lse)
        return ops.verify_attn(t["q"], t["k_cache"], t["v_cache"], t["k_draft"], t["v_draft"], t["parent"],
                               scale=scale, out=out, lse=lse)

    # Inputs read per step smaller than 4x L2 (the sparse gather, the tiny case) get an L2 flush
    # before every step, outside the step's events; larger ones stream from HBM anyway.
    flush = w.kv_bytes() < 4 * L2_BYTES
    scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if flush else None

    for _ in range(args.warmup):
        step(g)
    torch.cuda.synchronize()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    kd_ev = [(ev(), ev()) for _ in range(args.steps)]
    st_ev = [(ev(), ev()) for _ in range(args.steps)]
    for a, b in kd_ev + st_ev:  # materialise the events before handing them to the library
        a.record(stream)
        b.record(stream)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(ws_)
    torch.cuda.synchronize()
    launches0 = ops.kernel_launches()
    t0 = time.time()
    for i in range(args.steps):
        if flush:
            scratch.fill_(float(i))
        st_ev[i][0].record(stream)
        step(g)
        st_ev[i][1].record(stream)
    torch.cuda.synchronize()
    launches = ops.kernel_launches() - launches0
    # The cache kernel's own duration, from a second pass of K steps with CUDA events that
    # the library records around that launch. An event between the cache kernel and the
    # merge stops the merge from starting early (programmatic dependent launch), so these
    # events stay out of the pass that gives the step time.
    for i in range(args.steps):
        if flush:
            scratch.fill_(float(i))
        ops.profile_events(*kd_ev[i])
        step(g)
    ops.profile_events(None, None)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(ws_)
    clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in st_ev) / args.steps
    kd_ms = sum(a.elapsed_time(b) for a, b in kd_ev) / args.steps
    ms_max = allreduce_max(ws_, ms, dev)

    # end to end through the public API: pinned host inputs -> device, verify, result -> host
    if args.no_e2e:
        e2e_ms = float("nan")
        return finish(args, ws_, rank, w, ms, ms_max, kd_ms, launches, None, None, e2e_ms, clocks, t0, t1, x,
                      flush)
    dbuf = {k: torch.empty_like(g[k]) for k in names}
    hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
    hlse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
    h2d = sum(host[k].numel() * host[k].element_size() for k in names)
    d2h = hout.numel() * 4 + hlse.numel() * 4

    def e2e_step():
        for k in names:
            dbuf[k].copy_(host[k], non_blocking=True)
        o, l_ = step(dbuf)
        hout.copy_(o, non_blocking=True)
        hlse.copy_(l_, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(ws_)
    e0, e1 = ev(), ev()
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = allreduce_max(ws_, e0.elapsed_time(e1) / args.steps, dev)
    return finish(args, ws_, rank, w, ms, ms_max, kd_ms, launches, h2d, d2h, e2e_ms, clocks, t0, t1, x, flush)


def finish(args, ws_, rank, w, ms, ms_max, kd_ms, launches, h2d, d2h, e2e_ms, clocks, t0, t1, x, flush):
    if rank != 0:
        return None
    peaks, peak_src = measured_peaks()
    kv = w.kv_bytes()
    achieved_gbs = kv / (kd_ms * 1e-3) / 1e9
    traffic = NCU_TRAFFIC.get((kernel_source_hash(), w.name))
    rec = {
        "metric": METRIC,
        "value": round(kv * ws_ / (ms_max * 1e-3) / 1e12, 4),
        "unit": "TB/s",
        "n_gpus": ws_,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5),
        "us_per_step": round(ms_max * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, " + ("softmax(4z) scores, " if w.sparse else "") +
                f"{w.tree} draft tree)",
        "config": config_of(w, ws_, kv, flush),
        "roofline": {"bound": "hbm", "kernel": kernel_name(w), "achieved": round(achieved_gbs, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
                     "peak_source": f"{peak_src} copy bandwidth", "traffic": traffic,
                     "kernel_ms": round(kd_ms, 5), "share_of_step": round(kd_ms / ms, 4),
                     "timing": "CUDA events around each cache-kernel launch, launching stream, second pass of K steps"},
        "gpu_launches": int(launches),
        "e2e": None if h2d is None else {
            "value": round(kv / (e2e_ms * 1e-3) / 1e12, 4), "unit": "TB/s", "ms_per_step": round(e2e_ms, 4),
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)},
        "clocks": clocks.summary(t0, t1),
    }
    if ws_ == 1 and not args.no_cpu_baseline:  # the CPU baseline is taken on rank 0 at N=1 only
        rec["cpu_baseline"] = oracle_baseline(x, rows_target_s=args.cpu_seconds)
    return rec


def config_of(w, ws_, kv, flush):
    c = {"workload": w.name, "B": w.B, "L": w.L, "Hq": w.Hq, "Hkv": w.Hkv, "d": w.d, "N": w.N,
         "tree": w.tree + (f" depth<={w.depth_max}" if w.tree == "random" else ""), "kv_bytes_per_step": kv,
         "l2": (f"L2 flushed before every step ({2 * L2_BYTES >> 20} MiB write, outside the step events)" if flush
                else f"inputs larger than L2 (K/V {kv >> 20} MiB vs 129 MB), no flush"),
         "parallelism": f"replicas x{ws_}"}
    if w.sparse:
        c.update(sink=w.sink, window=w.window, top_m=w.top_m, budget=w.budget,
                 step="spec_select_topk + spec_verify_attn_sparse")
    else:
        c["step"] = "spec_verify_attn"
    return c


def kernel_name(w):
    if w.sparse:
        return "cache_attn_tc<sparse> (tcgen05, cp.async row gather)"
    return "cache_attn_tc (tcgen05 split-KV)"


def barrier(ws_):
    if ws_ > 1:
        torch.distributed.barrier()


def allreduce_max(ws_, v: float, dev) -> float:
    if ws_ == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device=dev if torch.distributed.get_backend() == "nccl" else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle, timed as it stands


def run_reference(args, ws_, rank):
    if rank != 0:
        return None
    w = W.workload(args.workload)
    x = W.make_inputs(w)
    total_rows = w.B * w.N * w.Hq
    per_step_rows = max(8, min(total_rows, args.ref_rows))
    rng = np.random.default_rng(1)
    import oracle

    idx = None
    if w.sparse:
        idx = oracle.select(x["draft_score"], x["target_score"], sink=w.sink, window=w.window,
                            top_m=w.top_m, budget=w.budget)[0]
    sel_s = oracle_select_seconds(x)

    def one(rows):
        oracle_rows(x, rows, idx)

    for _ in range(args.warmup):
        one(rng.choice(total_rows, size=per_step_rows, replace=False))
    t = time.perf_counter()
    for _ in range(args.steps):
        one(rng.choice(total_rows, size=per_step_rows, replace=False))
    el = time.perf_counter() - t
    step_s = sel_s + el / (args.steps * per_step_rows) * total_rows
    value = w.kv_bytes() / step_s / 1e12
    cores = len(os.sched_getaffinity(0))
    sample = f"{per_step_rows} of {total_rows} output rows per step, extrapolated to the full step"
    if w.sparse:
        sample += f", plus the selection of all {w.B} sequences ({sel_s:.2f} s)"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TB/s", "n_gpus": ws_,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": dict(config_of(w, ws_, w.kv_bytes(), False), l2="n/a (CPU)",
                           parallelism="host cores (OpenMP)"),
            "cpu_baseline": {"value": round(value, 6), "unit": "TB/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 6), "unit": "TB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", type=int, default=2)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-rows", type=int, default=48)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end loop (for profiling runs)")
    args = ap.parse_args()
    ws_, rank, local = dist_env()
    if ws_ > 1:
        backend = "gloo" if args.impl == "reference" else "nccl"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    if args.impl == "reference":
        rec = run_reference(args, ws_, rank)
    else:
        rec = run_native(args, ws_, rank, local)
    if rec is not None:
        print(json.dumps(rec), flush=True)
    if ws_ > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
