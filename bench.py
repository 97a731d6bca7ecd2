"""Benchmark: verification attention on one GB300 (or N replicas).

One step = one verification call over the whole batch of a workload. The
contract line times the headline workload (Llama-3-8B-shaped layer: B=4,
L=32768, 32 query / 8 KV heads, d=128, N=64-node random draft tree): one
spec_verify_attn call, i.e. the split-KV cache kernel plus the log-sum-exp
merge with the tree-masked draft block.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload C] [--extras LIST]
                  [--impl native|reference]

Prints one JSON line (rank 0). `value` is achieved HBM TB/s = algorithmic K/V
bytes of all ranks / (max over ranks of the time per step); ms_per_step is the
step latency. The headline's 512 MiB of K/V exceed the 129 MB L2, so no flush is
needed between its steps. At N=1 the same run also times the other workloads
(tiny dense, sparse hybrid, Qwen2.5-72B-shaped layer, the tree-size sweep) and
reports them under "workloads", each with its own roofline fraction, oracle
baseline and clock record; the tree-size sweep also calibrates BASTION's budget
controller ("bastion"). `--impl reference` times the CPU oracle (fp64, all host
cores) on a bounded sample of rows of the same workload.
"""

from __future__ import annotations

import argparse
import dataclasses
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
NOMINAL_HBM_GBS = 8000.0
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SWEEP_N = (1, 4, 16, 64, 256)

# DRAM bytes (read + written) per launch of the cache kernel from one ncu
# capture, keyed by the sha256 of the kernel sources it was taken on and the
# workload; a changed kernel reports null.
NCU_TRAFFIC = {
    ("1a6c515c26ca7c5f", "llama3-8b-layer-B4-L32k-N64-tree"): 540_654_336 + 7_333_632,
    ("1a6c515c26ca7c5f", "sparse-hybrid-B16-L32k-k2048-N8-chain"): 135_812_096 + 6_123_264,
    # captured at L = 32k (1.08 GB of reads, 11.3 MB of partials written): reads scaled by 4
    ("1a6c515c26ca7c5f", "qwen2.5-72b-layer-B8-L128k-N32-tree"): 4 * 1_081_574_000 + 11_319_552,
    ("1a6c515c26ca7c5f", "tree-sweep-B8-L16k-N256-best-first"): 563_341_056 + 33_412_352,
    ("1a6c515c26ca7c5f", "tree-sweep-B8-L16k-N1-best-first"): 537_137_664 + 3_848_448,
}
NCU_TRAFFIC_NOTE = {
    "qwen2.5-72b-layer-B8-L128k-N32-tree": "from an ncu capture at L=32k: K/V reads x4 (they grow with L), "
                                           "partial writes as captured (they do not)",
    "tree-sweep-B8-L16k-N256-best-first": "G*N = 1024 rows per KV head make four 256-row units; one block of CTAs per "
                                          "row group walks the same tiles in step, so three of every four reads of a "
                                          "K/V tile hit L2 (1.11x the algorithmic bytes)",
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
            p = json.load(f)
        return {k: float(p.get(k, FALLBACK_PEAKS[k])) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


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
        self.rows = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    @staticmethod
    def parse(text: str):
        """(time, sm MHz, max sm MHz, [hw_slowdown, hw_thermal, sw_thermal, sw_power_cap]) per sample."""
        rows = []
        for line in text.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                whole, _, frac = parts[0].partition(".")
                ts = time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + float("0." + (frac or "0"))
                rows.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        return rows

    def peek(self):
        """The samples taken so far (the sampler keeps running)."""
        self.file.flush()
        with open(self.file.name) as f:
            return self.parse(f.read())

    def stop(self):
        if self.proc is not None:
            time.sleep(0.1)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = self.parse(self.file.read())
        self.file.close()
        os.unlink(self.file.name)
        self.rows = rows

    def summary(self, t0: float, t1: float, rows=None):
        """Samples taken between t0 and t1 (wall clock; the whole run if none fall inside)."""
        rows = (self.rows if rows is None else rows) or []
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        use = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(use), "window": "timed" if inside else "bench",
                "window_s": round(t1 - t0, 3)}


def clock_rejection(summary) -> str | None:
    """Why a timed region's clock record rejects it, or None: a hardware or thermal slowdown, or SM
    clocks held well below their maximum with no reason given (a clock lock left behind). A power
    cap keeps the measurement (it is noted in the record); no samples, no rejection."""
    if not summary or not summary.get("samples"):
        return None
    bad = [r for r in summary["reasons"] if r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")]
    if bad:
        return ", ".join(bad)
    mhz, top = summary.get("sm_mhz"), summary.get("sm_max_mhz")
    if mhz and top and mhz < 0.75 * top and not summary["reasons"]:
        return f"SM clock {mhz:.0f} of {top:.0f} MHz with no reason given"
    return None


# ---------------------------------------------------------------------------
# oracle (CPU baseline)


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
        n = min(total_rows - done, max(n, int(len(rows) * (rows_target_s - elapsed) / max(dt, 1e-3))))
        if n <= 0:
            break
    step_s = sel_s + elapsed / done * total_rows
    cores = len(os.sched_getaffinity(0))
    sel = f"selection of all {w.B} sequences {sel_s:.2f} s + " if w.sparse else ""
    return {"value": w.kv_bytes() / step_s / 1e12, "unit": "TB/s", "cores": cores, "kind": "oracle",
            "s_per_step": round(step_s, 4),
            "sample": f"{sel}{done} of {total_rows} output rows (fp64, OpenMP over rows), {elapsed:.1f} s, "
                      f"extrapolated to one step: {step_s:.2f} s/step"}


# ---------------------------------------------------------------------------
# native arm


class Case:
    """One workload with its inputs resident on the device and its step functions."""

    def __init__(self, w, dev, host_pinned: bool = False):
        self.w = w
        self.dev = dev
        self.x = W.make_inputs(w)
        names = ["q", "k_cache", "v_cache", "k_draft", "v_draft", "parent"]
        if w.sparse:
            names += ["draft_score", "target_score"]
        self.names = names
        self.host = {k: (self.x[k].pin_memory() if host_pinned else self.x[k]) for k in names}
        self.g = {k: self.host[k].to(dev, non_blocking=True) for k in names}
        torch.cuda.synchronize()
        self.scale = self.x["scale"]
        self.out = torch.empty((w.B, w.N, w.Hq, w.d), dtype=torch.float32, device=dev)
        self.lse = torch.empty((w.B, w.N, w.Hq), dtype=torch.float32, device=dev)
        self.idx = torch.empty((w.B, max(w.budget, 1)), dtype=torch.int32, device=dev)
        self.cnt = torch.empty((w.B,), dtype=torch.int32, device=dev)
        # Inputs read per step smaller than 4x L2 (the sparse gather, the tiny case) get an L2
        # flush before every step, outside the step's events; larger ones stream from HBM anyway.
        self.flush = w.kv_bytes() < 4 * L2_BYTES
        self.scratch = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev) if self.flush else None
        if w.sparse:  # the index set, for the attention-only timing
            self.select(self.g)

    def select(self, t):
        from speculative_decoding_verification_77_gb300 import ops

        w = self.w
        ops.select_topk(t["draft_score"], t["target_score"], sink=w.sink, window=w.window, top_m=w.top_m,
                        budget=w.budget, idx=self.idx, count=self.cnt)

    def attend(self, t):
        from speculative_decoding_verification_77_gb300 import ops

        if self.w.sparse:
            return ops.verify_attn_sparse(t["q"], t["k_cache"], t["v_cache"], t["k_draft"], t["v_draft"],
                                          t["parent"], self.idx, scale=self.scale, out=self.out, lse=self.lse)
        return ops.verify_attn(t["q"], t["k_cache"], t["v_cache"], t["k_draft"], t["v_draft"], t["parent"],
                               scale=self.scale, out=self.out, lse=self.lse)

    def step(self, t):
        if self.w.sparse:
            self.select(t)
        return self.attend(t)

    def do_flush(self, i):
        if self.flush:
            self.scratch.fill_(float(i))

    def release(self):
        for k in list(self.g):
            del self.g[k]
        self.scratch = None
        torch.cuda.synchronize()
        torch.cuda.empty_cache()


def ev():
    return torch.cuda.Event(enable_timing=True)


def time_loop(case, fn, stream, steps: int, min_seconds: float = 0.0):
    """Per-call device times (ms) of fn(case.g), CUDA events on the launching stream, an L2
    flush before each call when the case needs one. Runs at least `steps` calls and, with
    min_seconds > 0, repeats batches of them until the loop has kept the GPU busy that long
    (wall clock, flushes included), so that the clock sampler sees the load."""
    times = []
    start = time.time()
    while True:
        pairs = [(ev(), ev()) for _ in range(steps)]
        for i, (a, b) in enumerate(pairs):
            case.do_flush(i)
            a.record(stream)
            fn(case.g)
            b.record(stream)
        torch.cuda.synchronize()
        times += [a.elapsed_time(b) for a, b in pairs]
        if time.time() - start >= min_seconds:
            return times


def kernel_pass(case, stream, steps: int):
    """Mean device time (ms) of the cache-attention kernel alone: CUDA events that the
    library records around that launch on the launching stream. An event between the
    cache kernel and the merge stops the merge from starting early (programmatic
    dependent launch), so this pass is separate from the step timing."""
    from speculative_decoding_verification_77_gb300 import ops

    pairs = [(ev(), ev()) for _ in range(steps)]
    for a, b in pairs:  # materialise the events before handing them to the library
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(pairs):
        case.do_flush(i)
        ops.profile_events(a, b)
        case.step(case.g)
    ops.profile_events(None, None)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in pairs) / steps


def kernel_name(w):
    if w.sparse:
        return "cache_attn_tc<sparse> (tcgen05, cp.async row gather)"
    return "cache_attn_tc (tcgen05 split-KV)"


def roofline_entry(w, kernel_ms, peaks, peak_src):
    """Roofline of the cache kernel: algorithmic K/V bytes and QK^T + PV flops per launch over
    its mean duration, against the measured copy bandwidth and the sustained bf16 rate."""
    kv, fl = w.kv_bytes(), w.flops()
    gbs = kv / (kernel_ms * 1e-3) / 1e9
    tfl = fl / (kernel_ms * 1e-3) / 1e12
    t_hbm = kv / (peaks["hbm_gbs"] * 1e9)
    t_tc = fl / (peaks["bf16_tflops_sustained"] * 1e12)
    bound = "tensor" if t_tc > t_hbm else "hbm"
    r = {"bound": bound, "kernel": kernel_name(w), "kernel_us": round(kernel_ms * 1e3, 2),
         "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
         "frac_hbm_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
         "achieved_tflops": round(tfl, 1), "frac_tensor_sustained": round(tfl / peaks["bf16_tflops_sustained"], 4),
         "frac_bound": round((t_tc if bound == "tensor" else t_hbm) / (kernel_ms * 1e-3), 4),
         "traffic": NCU_TRAFFIC.get((kernel_source_hash(), w.name)),
         "peaks": f"{peak_src}: hbm {peaks['hbm_gbs']} GB/s, bf16 sustained {peaks['bf16_tflops_sustained']} TFLOP/s"}
    if r["traffic"] is not None:
        r["traffic_over_algorithmic"] = round(r["traffic"] / kv, 3)
        if w.name in NCU_TRAFFIC_NOTE:
            r["traffic_note"] = NCU_TRAFFIC_NOTE[w.name]
    return r


def time_extra(case, stream, args, peaks, peak_src, clocks_windows):
    """Per-workload entry: step time (>= args.extra_seconds of device time), the cache kernel
    alone, for sparse also the selection alone and the attention alone."""
    w = case.w
    for _ in range(3):
        case.step(case.g)
    torch.cuda.synchronize()
    t0 = time.time()
    steps = time_loop(case, case.step, stream, args.steps, args.extra_seconds)
    t1 = time.time()
    kd_ms = kernel_pass(case, stream, args.steps)
    step_ms = sum(steps) / len(steps)
    kv = w.kv_bytes()
    e = {"workload": w.name, "B": w.B, "L": w.L, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N,
         "tree": w.tree + (f" depth<={w.depth_max}" if w.tree == "random" else ""),
         "kv_bytes_per_step": kv, "flops_per_step": w.flops(),
         "us_per_step": round(step_ms * 1e3, 2), "tb_per_s": round(kv / (step_ms * 1e-3) / 1e12, 4),
         "frac_hbm_step": round(kv / (step_ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
         "steps_timed": len(steps), "device_s_timed": round(sum(steps) * 1e-3, 3),
         "l2": "flushed before every step (outside the events)" if case.flush else "inputs larger than L2, no flush",
         "roofline": roofline_entry(w, kd_ms, peaks, peak_src)}
    clocks_windows.append((e, t0, t1))
    if w.sparse:
        e.update(sink=w.sink, window=w.window, top_m=w.top_m, budget=w.budget,
                 step="spec_select_topk + spec_verify_attn_sparse")
        sel = time_loop(case, case.select, stream, args.steps, args.extra_seconds / 4)
        att = time_loop(case, case.attend, stream, args.steps, args.extra_seconds / 4)
        e["select_us"] = round(sum(sel) / len(sel) * 1e3, 2)
        e["attention_us"] = round(sum(att) / len(att) * 1e3, 2)
        e["attention_tb_per_s"] = round(kv / (sum(att) / len(att) * 1e-3) / 1e12, 4)
    else:
        e["step"] = "spec_verify_attn"
    return e


def time_importance(dev, stream, args, peaks, peak_src, windows):
    """The importance-score producer at the headline layer (B=4, L=32k, N=64): two listed heads
    of different KV heads, lse from the verify call. Algorithmic bytes: the K rows of the two
    heads' KV heads, 2 x B x L x 256 B."""
    from speculative_decoding_verification_77_gb300 import ops

    w = W.workload(2)
    case = Case(w, dev)
    # A call reads 67 MB, less than L2. Inputs larger than L2 instead of a flush: the listed
    # pair of heads rotates over four pairs on different KV heads ([3, 19], [7, 23], [11, 27],
    # [15, 31]: KV heads {0, 4}, {1, 5}, {2, 6}, {3, 7}), so a call's 67 MB of K were last read
    # four calls (268 MB) earlier. A write flush would leave L2 full of dirty lines, whose
    # write-back the next call pays for (23.3 against 20.4 us per call, same kernel).
    case.flush = False
    _, lse = case.attend(case.g)
    pairs = [torch.tensor([h, h + 16], dtype=torch.int32, device=dev) for h in (3, 7, 11, 15)]
    score = torch.empty((w.B, w.L), dtype=torch.float32, device=dev)
    calls = [0]

    def run(t):
        heads = pairs[calls[0] % len(pairs)]
        calls[0] += 1
        ops.importance_scores(t["q"], t["k_cache"], lse, heads, scale=case.scale, out=score)

    for _ in range(3):
        run(case.g)
    torch.cuda.synchronize()
    t0 = time.time()
    v = time_loop(case, run, stream, args.steps, args.extra_seconds / 2)
    t1 = time.time()
    ms = sum(v) / len(v)
    kbytes = 2 * w.B * w.L * w.d * 2
    gbs = kbytes / (ms * 1e-3) / 1e9
    e = {"workload": w.name + " importance scores, two heads on different KV heads", "us_per_call": round(ms * 1e3, 2),
         "k_bytes": kbytes, "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
         "kernel": "importance_tc (tcgen05: S^T = K Q^T per 128-token tile, TMEM lane per token)",
         "l2": "inputs larger than L2: the head pair rotates over four pairs (268 MB of K), no flush",
         "peaks": f"{peak_src}: hbm {peaks['hbm_gbs']} GB/s", "calls_timed": len(v)}
    windows.append((e, t0, t1))
    case.release()
    return e


def time_lse_merge(dev, stream, args, peaks, peak_src, windows):
    """The exported two-part log-sum-exp merge (spec_lse_merge) on 131,072 rows of d = 128:
    reads two partials (o, lse) and writes one, 1,548 B a row, 203 MB a call."""
    from speculative_decoding_verification_77_gb300 import ops

    rows, d = 131072, 128
    gen = torch.Generator().manual_seed(7)

    def one_set():
        return {"o_a": torch.randn((rows, d), generator=gen).to(dev), "o_b": torch.randn((rows, d), generator=gen).to(dev),
                "l_a": (4 * torch.randn((rows,), generator=gen)).to(dev),
                "l_b": (4 * torch.randn((rows,), generator=gen)).to(dev),
                "out": torch.empty((rows, d), dtype=torch.float32, device=dev),
                "lse": torch.empty((rows,), dtype=torch.float32, device=dev)}

    # inputs larger than L2 instead of a flush: three independent sets (203 MB each) in turn,
    # so a call's inputs were last touched two calls (406 MB) earlier
    sets = [one_set() for _ in range(3)]
    calls = [0]

    class _Rotating:
        g = None

        def do_flush(self, i):
            pass

    def run(_):
        t = sets[calls[0] % len(sets)]
        calls[0] += 1
        ops.lse_merge(t["o_a"], t["l_a"], t["o_b"], t["l_b"], out=t["out"], lse_out=t["lse"])

    for _ in range(3):
        run(None)
    torch.cuda.synchronize()
    t0 = time.time()
    v = time_loop(_Rotating(), run, stream, args.steps, args.extra_seconds / 4)
    t1 = time.time()
    ms = sum(v) / len(v)
    nbytes = rows * (3 * d * 4 + 3 * 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    e = {"workload": f"lse_merge2 {rows} rows x d={d} (synthetic partials)", "us_per_call": round(ms * 1e3, 2),
         "bytes": nbytes, "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
         "kernel": "lse_merge2 (one warp per row)",
         "l2": "inputs larger than L2: three independent sets of partials in turn, no flush",
         "peaks": f"{peak_src}: hbm {peaks['hbm_gbs']} GB/s", "calls_timed": len(v)}
    windows.append((e, t0, t1))
    del sets
    torch.cuda.empty_cache()
    return e


def time_fp8(dev, stream, args, peaks, peak_src, windows):
    """The headline layer (B=4, L=32k, N=64 tree) over an fp8 cache: the bf16 cache quantised to
    E4M3 codes with a scale per (sequence, KV head), verified through spec_verify_attn_ex (the
    tcgen05 kernel loads the codes by TMA and six warps convert them into its bf16 tiles).
    Algorithmic bytes: the codes, 1 B an element (268 MB)."""
    from speculative_decoding_verification_77_gb300 import ops

    w = W.workload(2)
    case = Case(w, dev)

    def quantize(c):
        amax = c.float().abs().amax(dim=(2, 3)).clamp_min(1e-30)
        sc = (amax / 448.0).to(torch.float32)
        return (c.float() / sc[:, :, None, None]).to(torch.float8_e4m3fn), sc

    kc, ks = quantize(case.g["k_cache"])
    vc, vs = quantize(case.g["v_cache"])
    for k in ("k_cache", "v_cache"):  # the bf16 caches are no longer needed
        del case.g[k]
    torch.cuda.empty_cache()
    g = case.g

    def run(t):
        ops.verify_attn_ex(t["q"], kc, vc, t["k_draft"], t["v_draft"], t["parent"], scale=case.scale, k_scale=ks,
                           v_scale=vs, out=case.out, lse=case.lse)

    for _ in range(3):
        run(g)
    torch.cuda.synchronize()
    t0 = time.time()
    v = time_loop(case, run, stream, args.steps, args.extra_seconds / 2)
    t1 = time.time()
    ms = sum(v) / len(v)
    nbytes = kc.numel() + vc.numel()
    gbs = nbytes / (ms * 1e-3) / 1e9
    e = {"workload": w.name + " over an E4M3 cache (scale per sequence and KV head)", "us_per_step": round(ms * 1e3, 2),
         "kv_bytes_per_step": nbytes, "achieved_gbs": round(gbs, 1), "frac_hbm": round(gbs / peaks["hbm_gbs"], 4),
         "kernel": "cache_attn_tc<fp8> (codes by TMA, converted to bf16 tiles by six warps) + merge",
         "l2": "inputs larger than L2, no flush", "peaks": f"{peak_src}: hbm {peaks['hbm_gbs']} GB/s",
         "steps_timed": len(v)}
    windows.append((e, t0, t1))
    case.release()
    return e


def bastion_calibration(sweep, marginals, peaks, args):
    """BASTION's budget controller calibrated on the measured tree-size sweep: T_verify(N) =
    a T_roof(N) + c fitted to the sweep's step times, then the best-first growth and the
    speedup stop over the sweep workload's drafter marginals. Times in microseconds."""
    from speculative_decoding_verification_77_gb300 import ops

    w = W.workload(5, 1)
    ns = [e["N"] for e in sweep]
    ts = [e["us_per_step"] for e in sweep]
    bytes0 = float(w.kv_bytes())
    bytes_per_node = float(w.B * (w.Hq * w.d * 2 + 2 * w.Hkv * w.d * 2 + w.Hq * (w.d + 1) * 4))
    flops_per_node = float(4 * w.B * w.Hq * w.L * w.d)
    bw = peaks["hbm_gbs"] * 1e3  # bytes per microsecond
    peak = peaks["bf16_tflops_sustained"] * 1e6  # flops per microsecond
    l_ar = ts[ns.index(1)] if 1 in ns else min(ts)
    t_draft = args.bastion_draft_ratio * l_ar
    plan = ops.budget_plan(marginals, args.bastion_n_max, t_draft=t_draft, l_ar=l_ar, bytes0=bytes0,
                           bytes_per_node=bytes_per_node, flops_per_node=flops_per_node, bw=bw, peak=peak,
                           cal_n=ns, cal_t=ts)
    n = plan["n"]
    return {"cal_n": ns, "cal_t_us": ts, "a": round(plan["a"], 6), "c_us": round(plan["c"], 4),
            "n_chosen": n, "speedup_at_chosen": round(plan["speedup"][n - 1], 4) if n >= 1 else None,
            "surrogate_at_chosen": round(float(sum(plan["rho"][:n])), 4),
            "n_eval": plan["n_eval"], "l_ar_us": round(l_ar, 3), "t_draft_us": round(t_draft, 3),
            "bytes0": bytes0, "bytes_per_node": bytes_per_node, "flops_per_node": flops_per_node,
            "marginals": "first sequence of the sweep workload (16 positions x 10 candidates, Dirichlet(0.3))",
            "assumptions": f"L_AR = measured step at N=1; T_draft = {args.bastion_draft_ratio} x L_AR"}


def run_native(args, ws_, rank, local):
    from speculative_decoding_verification_77_gb300 import ops

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    peaks, peak_src = measured_peaks()
    w = W.workload(args.workload, args.n)
    if args.seq_len is not None:  # a shorter cache of the same layer (small profiling captures)
        w = dataclasses.replace(w, L=args.seq_len, name=f"{w.name}@L{args.seq_len}")
    case = Case(w, dev, host_pinned=not args.no_e2e)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        case.step(case.g)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    # untimed steps before the timed ones, so that the clock record brackets the timed region
    t_pre = time.time()
    while time.time() - t_pre < args.clock_window:
        for i in range(20):
            case.do_flush(i)
            case.step(case.g)
        torch.cuda.synchronize()
    def timed_region():
        barrier(ws_)
        torch.cuda.synchronize()
        launches0 = ops.kernel_launches()
        evs = [(ev(), ev()) for _ in range(args.steps)]
        for i, (a, b) in enumerate(evs):
            case.do_flush(i)
            a.record(stream)
            case.step(case.g)
            b.record(stream)
        torch.cuda.synchronize()
        return evs, time.time(), ops.kernel_launches() - launches0

    st_ev, t1, launches = timed_region()
    # a clock record showing a slowdown (or a clock held low) rejects the timed region: measure it
    # once more, every rank together, and say why in the line
    rejected = clock_rejection(clocks.summary(t_pre, t1, clocks.peek()))
    remeasured = None
    if allreduce_max(ws_, 1.0 if rejected else 0.0, dev) > 0:
        remeasured = rejected or "another rank's clock record"
        t_pre = time.time()
        for i in range(20):
            case.do_flush(i)
            case.step(case.g)
        torch.cuda.synchronize()
        st_ev, t1, launches = timed_region()
    kd_ms = kernel_pass(case, stream, args.steps)
    barrier(ws_)
    ms = sum(a.elapsed_time(b) for a, b in st_ev) / args.steps
    ms_max = allreduce_max(ws_, ms, dev)

    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(case, stream, args, ws_, dev)
    x = case.x
    case.release()

    extras = {}
    bastion = None
    windows = []
    if ws_ == 1 and args.extras != "none":
        tokens = args.extras.split(",") if args.extras != "all" else ["1", "2", "3", "4", "5", "merge", "fp8"]
        wanted = [int(c) for c in tokens if c.isdigit()]
        sweep = []
        marginals = None
        for c in wanted:
            for n in (SWEEP_N if c == 5 else (None,)):
                wx = W.workload(c, n)
                if wx.name == w.name:  # the headline itself: same run, reuse its numbers below
                    continue
                cx = Case(wx, dev)
                e = time_extra(cx, stream, args, peaks, peak_src, windows)
                if not args.no_cpu_baseline:
                    e["cpu_baseline"] = oracle_baseline(cx.x, rows_target_s=args.extra_cpu_seconds)
                if c == 5:
                    sweep.append(e)
                    if marginals is None:
                        marginals = cx.x["trees"][0].marginals
                extras[wx.name] = e
                cx.release()
                del cx
        if 2 in wanted or "importance" in tokens:
            extras["importance-scores-llama3-8b-layer"] = time_importance(dev, stream, args, peaks, peak_src, windows)
        if "merge" in tokens:
            extras["lse-merge2-131072-rows"] = time_lse_merge(dev, stream, args, peaks, peak_src, windows)
        if "fp8" in tokens:
            extras["fp8-cache-llama3-8b-layer"] = time_fp8(dev, stream, args, peaks, peak_src, windows)
        if sweep and marginals is not None:
            head_e = None
            if w.tree == "best_first" and w.name.startswith("tree-sweep"):
                head_e = {"N": w.N, "us_per_step": round(ms * 1e3, 2)}
            pts = sorted(sweep + ([head_e] if head_e else []), key=lambda e: e["N"])
            bastion = bastion_calibration(pts, marginals, peaks, args)
    clocks.stop()
    for e, a, b in windows:
        e["clocks"] = clocks.summary(a, b)
    return finish(args, ws_, rank, w, ms, ms_max, kd_ms, launches, e2e, clocks, t_pre, t1, x, case.flush, peaks,
                  peak_src, extras, bastion, remeasured)


def run_e2e(case, stream, args, ws_, dev):
    """End to end through the public API, pipelined as a serving loop runs it: every step copies
    its inputs from pinned host memory to the device (on a copy stream, into one of two input
    buffers, so that step k + 1's copy runs under step k's compute), verifies on the launching
    stream and reads its result back to pinned host memory. The timed region holds every copy of
    every timed step."""
    bufs = [{k: torch.empty_like(case.g[k]) for k in case.names} for _ in range(2)]
    hout = torch.empty(case.out.shape, dtype=case.out.dtype, pin_memory=True)
    hlse = torch.empty(case.lse.shape, dtype=case.lse.dtype, pin_memory=True)
    h2d = sum(case.host[k].numel() * case.host[k].element_size() for k in case.names)
    d2h = hout.numel() * 4 + hlse.numel() * 4
    cstream = torch.cuda.Stream(dev)

    def run(n):
        copied = [torch.cuda.Event() for _ in range(2)]  # buffer j holds the inputs of its step
        freed = [torch.cuda.Event() for _ in range(2)]   # the step that read buffer j is done

        def copy_in(k):
            j = k % 2
            if k >= 2:
                cstream.wait_event(freed[j])
            with torch.cuda.stream(cstream):
                for name in case.names:
                    bufs[j][name].copy_(case.host[name], non_blocking=True)
            copied[j].record(cstream)

        cstream.wait_stream(stream)
        copy_in(0)
        for k in range(n):
            if k + 1 < n:
                copy_in(k + 1)
            stream.wait_event(copied[k % 2])
            o, l_ = case.step(bufs[k % 2])
            freed[k % 2].record(stream)
            hout.copy_(o, non_blocking=True)
            hlse.copy_(l_, non_blocking=True)

    run(max(1, args.warmup))
    torch.cuda.synchronize()
    barrier(ws_)
    e0, e1 = ev(), ev()
    e0.record(stream)
    run(args.steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = allreduce_max(ws_, e0.elapsed_time(e1) / args.steps, dev)
    del bufs
    return {"value": round(case.w.kv_bytes() / (e2e_ms * 1e-3) / 1e12, 4), "unit": "TB/s",
            "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "pipelined": "step k + 1's host-to-device copy under step k's compute (two input buffers)"}


def finish(args, ws_, rank, w, ms, ms_max, kd_ms, launches, e2e, clocks, t0, t1, x, flush, peaks, peak_src,
           extras, bastion, remeasured=None):
    if rank != 0:
        return None
    kv = w.kv_bytes()
    achieved_gbs = kv / (kd_ms * 1e-3) / 1e9
    traffic = NCU_TRAFFIC.get((kernel_source_hash(), w.name))
    rf = roofline_entry(w, kd_ms, peaks, peak_src)
    rec = {
        "metric": METRIC,
        "value": round(kv * ws_ / (ms_max * 1e-3) / 1e12, 4),
        "unit": "TB/s",
        "n_gpus": ws_,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5),
        "us_per_step": round(ms_max * 1e3, 2),
        "frac_hbm_step": round(kv / (ms_max * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
        "frac_hbm_step_nominal_8tbs": round(kv / (ms_max * 1e-3) / 1e9 / NOMINAL_HBM_GBS, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V, " + ("softmax(4z) scores, " if w.sparse else "") +
                f"{w.tree} draft tree)",
        "config": config_of(w, ws_, kv, flush),
        "roofline": {"bound": rf["bound"], "kernel": kernel_name(w), "achieved": round(achieved_gbs, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(achieved_gbs / peaks["hbm_gbs"], 4),
                     "frac_nominal_8tbs": round(achieved_gbs / NOMINAL_HBM_GBS, 4),
                     "peak_source": f"{peak_src} copy bandwidth", "traffic": traffic,
                     "kernel_ms": round(kd_ms, 5), "share_of_step": round(kd_ms / ms, 4),
                     "achieved_tflops": rf["achieved_tflops"], "frac_tensor_sustained": rf["frac_tensor_sustained"],
                     "timing": "CUDA events around each cache-kernel launch, launching stream, second pass of K steps"},
        "gpu_launches": int(launches),
        "e2e": e2e,
        "clocks": clocks.summary(t0, t1),
    }
    if remeasured:
        rec["clocks"]["remeasured"] = f"the first timed region's clock record showed {remeasured}"
    if extras:
        head = {"workload": w.name, "us_per_step": rec["us_per_step"], "tb_per_s": round(kv / (ms * 1e-3) / 1e12, 4),
                "frac_hbm_step": rec["frac_hbm_step"], "roofline": rf, "note": "the contract line above"}
        rec["workloads"] = {w.name: head, **extras}
    if bastion is not None:
        rec["bastion"] = bastion
    if ws_ == 1 and not args.no_cpu_baseline:  # the CPU baseline is taken on rank 0 at N=1 only
        rec["cpu_baseline"] = oracle_baseline(x, rows_target_s=args.cpu_seconds)
        if extras:
            rec["workloads"][w.name]["cpu_baseline"] = rec["cpu_baseline"]
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
    w = W.workload(args.workload, args.n)
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
    ap.add_argument("--n", type=int, default=None, help="draft-tree size of the tree-size sweep workload (5)")
    ap.add_argument("--seq-len", type=int, default=None,
                    help="cache length instead of the workload's own (small cases for ncu captures)")
    ap.add_argument("--extras", default="all",
                    help="other workloads timed in the same run at N=1: all, none, or a list like 1,3,4,5")
    ap.add_argument("--extra-seconds", type=float, default=1.0, help="device time per extra workload")
    ap.add_argument("--extra-cpu-seconds", type=float, default=2.0, help="oracle time per extra workload")
    ap.add_argument("--clock-window", type=float, default=0.5,
                    help="seconds of untimed steps before the timed ones, under the clock sampler")
    ap.add_argument("--bastion-draft-ratio", type=float, default=1.0)
    ap.add_argument("--bastion-n-max", type=int, default=512)
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
