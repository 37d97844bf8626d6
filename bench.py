"""Benchmark of the fused sparse-attention kernel (one JSON line on stdout).

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]

A step is one call of the whole fused path over one batch of synthetic tokens.  The
headline workload is the 1024-token decode (h_q 64, top-k 128 + 512 with ragged
lengths, NaN-filled stale rows); the line also carries the other workload sizes.
Timing: W untimed warm-up steps, then K steps; L2 is flushed (a 512 MiB write) before
every timed step, each step is timed with CUDA events on the launching stream, and
the K-step region is bracketed by a barrier and a device synchronize.  With N > 1
(torchrun) the ranks split one batch: rank r takes a contiguous slice of the workload's
tokens (query tokens are independent problems, so there is no collective on the data
path) and the value is the batch's tokens over the slowest rank's time (strong
scaling).  --replicas instead gives every rank its own copy of the whole workload (weak
scaling).

--impl reference times the CPU oracle (float64 numpy, test infrastructure) on
bounded samples of the same workload; only rank 0 runs it.
"""

from __future__ import annotations

import argparse
import re
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

HEADLINE = "decode1024"
METRIC = "sparse-attn tokens/s and us/call, s_q=1..2123; HBM GB/s and % of roofline"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
# the roofline the workload specification defines: the larger of the gathered bytes at
# 8 TB/s and the flops at the dense peak of the MMA precision used (fp16 operands, fp32
# accumulate: 2.25 PFLOP/s nominal on GB300)
SPEC_HBM_BPS = 8e12
SPEC_DENSE_FLOPS = 2.25e15


def spec_roofline_s(w) -> float:
    return max(algorithmic_bytes(w) / SPEC_HBM_BPS, algorithmic_flops(w) / SPEC_DENSE_FLOPS)


def algorithmic_bytes(w) -> int:
    """Bytes the path must move at least once: the valid gathered rows, q, the outputs,
    the index row, the length and the position of every token.  On the nvfp4_ds_mla
    cache the rows are 528 bytes (window columns) and 288 bytes (compressed columns)
    and q has 512 dims."""
    from top_sparse_mla_gb300 import workloads as W
    if w.kv_format == 1:
        cols = np.arange(w.topk)[None, :]
        live = (cols < w.topk_length[:, None]) & (w.indices >= 0)
        n_swa = int(live[:, :w.n_swa_cols].sum())
        n_cmp = int(live[:, w.n_swa_cols:].sum())
        per_tok = w.h_q * 512 * 2 + w.h_q * 512 + w.h_q * 16 + w.topk * 4 + 8
        return n_swa * 528 + n_cmp * 288 + w.s_q * per_tok
    n_valid = int(W.n_valid_rows(w).sum())
    per_tok = w.h_q * 576 * 2 + w.h_q * 512 + w.h_q * 16 + w.topk * 4 + 8
    return n_valid * 656 + w.s_q * per_tok


def algorithmic_flops(w) -> int:
    from top_sparse_mla_gb300 import workloads as W
    d_qk = 512 if w.kv_format == 1 else 576
    return int(W.n_valid_rows(w).sum()) * (2 * w.h_q * d_qk + 2 * w.h_q * 512)


def kernels_per_call(params, num_sms: int = 0) -> int:
    """Kernels one forward call launches: the fused kernel, preceded on the queue path
    (no token split, at most DSA_ORDER_MAX_TOKENS tokens) by the kernel that orders the
    queue.  Otherwise a memset clears the workspace header instead.  num_sms <= 0: the
    current device's SM count."""
    from top_sparse_mla_gb300 import native
    queue = native.dsa_sparse_attn_num_splits(params, num_sms) == 1
    return 2 if queue and params.s_q <= native.DSA_ORDER_MAX_TOKENS else 1


def profiled_traffic(workload_name: str):
    """DRAM bytes per launch (read + write) from the committed ncu summary of this
    workload, or None when the summary is missing or was taken on other kernel source
    (its recorded sha256 prefix of the kernel source must match the current one)."""
    here = os.path.dirname(os.path.abspath(__file__))
    path = os.path.join(here, "profiles", "dsa_fwd_kernel_decode1024_full.md")
    if workload_name != "decode1024" or not os.path.exists(path):
        return None
    src = b""
    for f in ("dsa_sparse_attn.cu", "ptx_sm103.cuh"):
        with open(os.path.join(here, "top_sparse_mla_gb300", "csrc", f), "rb") as fh:
            src += fh.read()
    digest = hashlib.sha256(src).hexdigest()[:16]
    text = open(path).read()
    m_hash = re.search(r"kernel-source-sha256-prefix: ([0-9a-f]{16})", text)
    m_traffic = re.search(r"traffic \(read \+ write\) per launch \| ([0-9.]+) MB", text)
    if not m_hash or not m_traffic or m_hash.group(1) != digest:
        return None
    return float(m_traffic.group(1)) * 1e6


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling every 200 ms while it runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.t_start = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def rank_workload(w, rank: int, world: int, replicas: bool = False):
    """The part of the batch this rank runs: its contiguous token slice of `w` (the caches
    are shared), or all of `w` in replica mode."""
    if world > 1 and not replicas:
        from top_sparse_mla_gb300 import sharding
        return sharding.shard(w, rank, world)
    return w


def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    return world, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def time_kernel(inp, out, steps: int, warmup: int, flush, events=True):
    """Per-step CUDA-event times (ms) of the fused call, L2 flushed before each step."""
    import torch
    from top_sparse_mla_gb300 import api
    for _ in range(warmup):
        flush.zero_()
        api.forward(inp, out)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        starts[i].record(st)
        api.forward(inp, out)
        ends[i].record(st)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def time_e2e(w, inp, out, steps: int, warmup: int, flush):
    """Same call with the step's inputs copied from pinned host memory and the result
    copied back, inside the timed span.  The KV caches and the norm weight stay resident
    on the device (persistent state, like model weights)."""
    import torch
    from top_sparse_mla_gb300 import api
    h_q = torch.from_numpy(w.q.view(np.int16)).pin_memory()
    h_idx = torch.from_numpy(w.indices).pin_memory()
    h_len = torch.from_numpy(w.topk_length).pin_memory()
    h_pos = torch.from_numpy(w.positions).pin_memory()
    h_fp8 = torch.empty(out.out_fp8.shape, dtype=torch.uint8).pin_memory()
    h_sf = torch.empty(out.out_sf.shape, dtype=torch.uint8).pin_memory()
    st = torch.cuda.current_stream()

    def step():
        inp.q.copy_(h_q, non_blocking=True)
        inp.indices.copy_(h_idx, non_blocking=True)
        inp.topk_length.copy_(h_len, non_blocking=True)
        inp.positions.copy_(h_pos, non_blocking=True)
        api.forward(inp, out)
        h_fp8.copy_(out.out_fp8, non_blocking=True)
        h_sf.copy_(out.out_sf, non_blocking=True)

    for _ in range(warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        step()
        b.record(st)
        b.synchronize()
        times.append(a.elapsed_time(b))
    h2d = sum(t.numel() * t.element_size() for t in (h_q, h_idx, h_len, h_pos))
    d2h = sum(t.numel() * t.element_size() for t in (h_fp8, h_sf))
    return times, h2d, d2h


def time_topk(s_q: int, n: int, k: int, flush, peak_gbs: float):
    """The index producer's top-k selection (include/dsa_topk.h) on seeded N(0,1) bf16
    logits: median CUDA-event time of 30 calls, L2 flushed before each; bytes are the
    logits read plus the index rows and lengths written."""
    import torch
    from top_sparse_mla_gb300 import native
    g = torch.Generator(device="cuda").manual_seed(7)
    logits = torch.randn((s_q, n), generator=g, device="cuda").to(torch.bfloat16)
    idx = torch.empty((s_q, k), dtype=torch.int32, device="cuda")
    tl = torch.empty((s_q,), dtype=torch.int32, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(3):
        native.dsa_topk_select(logits, k, idx, tl)
    ts = []
    for _ in range(30):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        native.dsa_topk_select(logits, k, idx, tl)
        b.record(st)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    med = statistics.median(ts)
    nbytes = s_q * n * 2 + s_q * k * 4 + s_q * 4
    return {"us_per_call_median": med * 1e3, "alg_bytes": nbytes, "alg_gbs": nbytes / (med * 1e-3) / 1e9,
            "frac_of_hbm_peak": nbytes / (med * 1e-3) / 1e9 / peak_gbs}


def time_kv_insert(n: int, n_rows: int, flush, peak_gbs: float):
    """The KV-cache insert (include/dsa_kv_insert.h): n seeded N(0,1) bf16 KV rows
    normalised, roped and quantised into random distinct rows of an n_rows-row pool;
    median CUDA-event time of 30 calls, L2 flushed before each.  Bytes: the KV rows, the
    positions and slots read, the 656-byte rows written."""
    import torch
    from top_sparse_mla_gb300 import native
    g = torch.Generator(device="cuda").manual_seed(9)
    kv = torch.randn((n, 576), generator=g, device="cuda").to(torch.bfloat16)
    w = (1 + 0.1 * torch.randn((512,), generator=g, device="cuda")).to(torch.bfloat16)
    pos = torch.randint(0, 32768, (n,), generator=g, device="cuda", dtype=torch.int32)
    slots = torch.randperm(n_rows, generator=g, device="cuda")[:n].to(torch.int64)
    pool = torch.zeros((n_rows, 656), dtype=torch.uint8, device="cuda")
    st = torch.cuda.current_stream()
    for _ in range(3):
        native.dsa_kv_insert(kv, pos, slots, w, pool)
    ts = []
    for _ in range(30):
        flush.zero_()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        native.dsa_kv_insert(kv, pos, slots, w, pool)
        b.record(st)
        b.synchronize()
        ts.append(a.elapsed_time(b))
    med = statistics.median(ts)
    nbytes = n * (576 * 2 + 4 + 8 + 656) + 512 * 2
    return {"us_per_call_median": med * 1e3, "alg_bytes": nbytes, "alg_gbs": nbytes / (med * 1e-3) / 1e9,
            "frac_of_hbm_peak": nbytes / (med * 1e-3) / 1e9 / peak_gbs, "tokens": n, "pool_rows": n_rows}


def cpu_oracle_rate(w, max_seconds: float = 20.0, min_tokens: int = 32):
    """Oracle tokens/s on a bounded prefix of the workload's tokens."""
    import oracle
    p = oracle.OracleParams(n_swa_cols=w.n_swa_cols)
    t0 = time.time()
    done = 0
    chunk = 16
    while done < w.s_q and (time.time() - t0 < max_seconds or done < min_tokens):
        sel = np.arange(done, min(done + chunk, w.s_q))
        oracle.sparse_mla_forward(w.q[sel], w.kv_swa, w.kv_cmp, w.indices[sel], w.topk_length[sel],
                                  w.positions[sel], w.norm_w, p)
        done += len(sel)
    dt = time.time() - t0
    return done / dt, done, dt


def run_reference(args):
    world, rank, _, pg = dist_setup(args.gpus)
    if rank != 0:
        return
    from top_sparse_mla_gb300 import workloads as W
    w = W.make(HEADLINE)
    import oracle
    p = oracle.OracleParams(n_swa_cols=w.n_swa_cols)
    per_step = 32
    cores = len(os.sched_getaffinity(0))

    def step(i):
        start = (i * per_step) % w.s_q
        sel = np.arange(start, min(start + per_step, w.s_q))
        oracle.sparse_mla_forward(w.q[sel], w.kv_swa, w.kv_cmp, w.indices[sel], w.topk_length[sel],
                                  w.positions[sel], w.norm_w, p)
        return len(sel)

    for i in range(args.warmup):
        step(i)
    t0 = time.time()
    toks = sum(step(args.warmup + i) for i in range(args.steps))
    dt = time.time() - t0
    value = toks / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "s_q_per_step": per_step, "h_q": w.h_q, "topk": w.topk},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"{toks} tokens of {w.name} ({per_step} per step), numpy float64, BLAS default threads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_native(args):
    import torch
    world, rank, local, pg = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    from top_sparse_mla_gb300 import api, native, workloads as W
    from top_sparse_mla_gb300.build import build
    build()
    native.library()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    peak, peak_kind = measured_peaks()

    w_full = W.make(args.workload)
    w = rank_workload(w_full, rank, world, args.replicas)
    inp = api.upload(w, "cuda")
    out = api.allocate_outputs(inp)
    sampler = ClockSampler(local)
    barrier(pg)
    torch.cuda.synchronize()
    t_wall = time.time()
    times = time_kernel(inp, out, args.steps, args.warmup, flush)
    torch.cuda.synchronize()
    barrier(pg)
    wall = time.time() - t_wall
    # keep the GPU under the same load long enough for the clock sampler to see it
    soak_end = time.time() + (0.0 if args.no_soak else 1.5)
    while time.time() < soak_end:
        time_kernel(inp, out, 20, 0, flush)
    clocks = sampler.stop()
    ms = statistics.mean(times)
    ms_max = max_over_ranks(pg, ms)
    tokens_total = w_full.s_q * (world if args.replicas else 1)
    value = tokens_total / (ms_max * 1e-3)
    b_alg = algorithmic_bytes(w)
    achieved = b_alg / (ms * 1e-3) / 1e9

    e2e = None
    if not args.skip_e2e:
        e2e_times, h2d, d2h = time_e2e(w, inp, out, max(3, min(args.steps, 20)), 2, flush)
        e2e_ms = max_over_ranks(pg, statistics.mean(e2e_times))
        e2e = {"value": tokens_total / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}

    per_config = {}
    if not args.skip_sweep and world == 1:
        for name in ("decode1", "decode64", "decode1024", "prefill2123", "decode1024_nvfp4", "decode1024_fp8q"):
            wc = W.make(name) if name != args.workload else w
            ic = api.upload(wc, "cuda") if name != args.workload else inp
            oc = api.allocate_outputs(ic)
            tc = time_kernel(ic, oc, 30, 5, flush)
            med = statistics.median(tc)
            bc = algorithmic_bytes(wc)
            per_config[name] = {"us_per_call_median": med * 1e3, "us_per_call_mean": statistics.mean(tc) * 1e3,
                                "tokens_per_s": wc.s_q / (med * 1e-3), "alg_bytes": bc,
                                "alg_gbs": bc / (med * 1e-3) / 1e9, "frac_of_hbm_peak": bc / (med * 1e-3) / 1e9 / peak,
                                "alg_tflops": algorithmic_flops(wc) / (med * 1e-3) / 1e12,
                                "spec_roofline_us": spec_roofline_s(wc) * 1e6,
                                "frac_of_spec_roofline": spec_roofline_s(wc) / (med * 1e-3),
                                "n_valid_rows": int(W.n_valid_rows(wc).sum())}
            if name != args.workload:
                del ic, oc
                torch.cuda.empty_cache()

    if not args.skip_sweep and world == 1:
        per_config["topk_1024x8192_k512"] = time_topk(1024, 8192, 512, flush, peak)
        per_config["kv_insert_4096_into_1M_rows"] = time_kv_insert(4096, 1 << 20, flush, peak)
        per_config["kv_insert_65536_into_1M_rows"] = time_kv_insert(65536, 1 << 20, flush, peak)

    cpu = None
    if rank == 0 and not args.skip_cpu:
        rate, ntok, dt = cpu_oracle_rate(w_full)
        cpu = {"value": rate, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
               "sample": f"first {ntok} tokens of {w_full.name} in {dt:.1f} s, numpy float64, BLAS default threads"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak" if (world == 1 or args.replicas) else "strong",
            "vs_baseline": None, "dtype": "f16", "data": "synthetic",
            "config": {"workload": w_full.name, "s_q": w_full.s_q, "h_q": w.h_q, "topk": w.topk,
                       "n_valid_rows": int(W.n_valid_rows(w_full).sum()),
                       "parallelism": (f"replicas x{world}" if args.replicas else f"token slices x{world}") if world > 1
                       else "single GPU",
                       "l2": "flushed before every timed step (512 MiB write)",
                       "operands": "E4M3 codes exact in fp16, fp32 block scales applied in fp32, q~ and P as "
                                   "fp16 hi + lo pairs, fp32 accumulate, MXFP8 out",
                       "timed_wall_s": wall},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         # the committed profile is of one launch of the whole workload: a token
                         # slice (N > 1) moves other bytes
                         "traffic": args.traffic if args.traffic is not None else
                         (profiled_traffic(args.workload) if world == 1 or args.replicas else None),
                         "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum, one launch "
                                           "(profiles/dsa_fwd_kernel_decode1024_full.md)",
                         "peak_source": peak_kind,
                         "alg_bytes_per_launch": b_alg,
                         "spec_roofline_us": spec_roofline_s(w) * 1e6,
                         "frac_of_spec_roofline": spec_roofline_s(w) / (ms * 1e-3),
                         "spec_roofline_definition": "max(alg bytes / 8 TB/s, alg flops / 2.25 PFLOP/s fp16 dense)"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * kernels_per_call(inp.params),
            "clocks": clocks,
            "per_config": per_config,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=HEADLINE, help="workload timed for the headline line")
    ap.add_argument("--skip-sweep", action="store_true", help="headline workload only")
    ap.add_argument("--skip-e2e", action="store_true", help="no host-buffer end-to-end timing")
    ap.add_argument("--no-soak", action="store_true", help="no clock-sampling soak after the timed steps")
    ap.add_argument("--skip-cpu", action="store_true", help="no CPU oracle baseline")
    ap.add_argument("--replicas", action="store_true",
                    help="with N > 1: every rank runs the whole workload (weak scaling) instead of a token slice")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the kernel from an ncu capture, if known")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_native(args)


if __name__ == "__main__":
    main()
