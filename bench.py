"""Benchmark: causal attention forward at B=4, H=32, S=8192, d=128 (bf16) on GB300.

One step = one call of the attention forward over the whole batch (one launch
of the tiled prefill kernel). Prints ONE JSON line on rank 0.

  value     algorithmic TFLOP/s (4*d per visible (query, key) pair), inputs
            resident in HBM, CUDA events on the launching stream, max over ranks
  e2e       same metric through the C ABI call that takes host buffers
            (fa_forward_host) with pinned host memory: every step's H2D of
            Q, K, V and D2H of O, LSE are inside the timed region
  roofline  achieved / measured bf16 tensor peak for the prefill kernel (with
            --workload of Sq <= 16, achieved GB/s / measured HBM bandwidth for
            the verify kernel fa_forward runs those shapes on)
  verify    the decode-shaped split-KV path (B=16, H=32, Sq=5, Sk=4096) against
            the measured HBM bandwidth (also as a draft tree and from paged caches)
  backward  dQ, dK, dV on the same workload (2.5x the forward's FLOPs)
  fp8       the FP8 (E4M3) forward on the same workload, against the FP8 peak
  cpu_baseline  the fp64 oracle on a bounded sample of rows, host cores

--impl reference times the fp64 CPU oracle instead (the only reference arm
this method has) on the same workload, metric and unit.
Multi-GPU (torchrun): every rank runs its own independent batch (weak
scaling, no collective on the data path); value = all ranks' FLOPs / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from exact_tiled_attention_03_gb300.inputs import HEADLINE, VERIFY, WORKLOADS, make_qkv, sample_rows, with_seed  # noqa: E402

METRIC = "causal attn fwd TFLOP/s (bf16, B=4,H=32,S=8192,d=128) and % of GB300 BF16 peak"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}


# ---------------------------------------------------------------- distributed helpers
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend, timeout_s: float = 600.0):
    """One process group for the job. A rank that dies ends the others' next
    collective with an error within `timeout_s` (or at once, when its
    connections close) instead of the backend's default wait."""
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend=backend,
                                             timeout=datetime.timedelta(seconds=timeout_s))


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def reduce_max(x: float, world: int, device=None) -> float:
    """Max over ranks (the job is as slow as its slowest rank)."""
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.SUM)
    return float(t.item())


def rank_workload(name: str, rank: int):
    """Each rank's own independent problem: same shape, seed offset by rank."""
    w = WORKLOADS[name]
    return with_seed(w, w.seed + 1000 * rank) if rank else w


# ---------------------------------------------------------------- measurement helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]), "hbm_gbs": float(d["hbm_gbs"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return dict(FALLBACK_PEAKS, source="fallback")


def source_hash(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ["exact_tiled_attention_03_gb300/csrc/fa_prefill_sm103.cu",
                   "exact_tiled_attention_03_gb300/csrc/fa_ptx.cuh",
                   "exact_tiled_attention_03_gb300/csrc/fa_schedule.cuh"]
VERIFY_SOURCES = ["exact_tiled_attention_03_gb300/csrc/fa_verify.cu",
                  "exact_tiled_attention_03_gb300/csrc/fa_ptx.cuh"]
FP8_SOURCES = ["exact_tiled_attention_03_gb300/csrc/fa_prefill_fp8_sm103.cu",
               "exact_tiled_attention_03_gb300/csrc/fa_ptx.cuh",
               "exact_tiled_attention_03_gb300/csrc/fa_schedule.cuh"]
BWD_SOURCES = ["exact_tiled_attention_03_gb300/csrc/fa_backward_sm103.cu",
               "exact_tiled_attention_03_gb300/csrc/fa_ptx.cuh"]


def ncu_traffic(kernel: str, sources, workload: str):
    """DRAM bytes per launch from the committed ncu summary; None if the
    kernel changed since or the capture was of another workload."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(kernel)
    if not d or d.get("source_sha") != source_hash(sources):
        return None
    if d["workload"].split()[0] != workload:
        return None
    return d["dram_bytes"] / d["units"]


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self._t = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = []
        for ts, line in self.lines:
            if t0 <= ts <= t1 + 0.15:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


def time_steps(fn, steps, stream):
    """Device time of `steps` back-to-back calls (CUDA events on `stream`)."""
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(steps):
        fn()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / 1e3


# ---------------------------------------------------------------- CPU oracle legs
def oracle_rows_flops(w, rows):
    return sum(4 * w.d * w.visible_keys(i) for _, _, i in rows)


def time_oracle_sample(w, q, k, v, budget_s: float, seed: int = 7, threads: int = 0):
    """Time the oracle (as it stands) on a seeded sample of rows sized to ~budget_s
    (threads = 0: the OpenMP default). The sample is sized from a probe large
    enough to occupy every thread (a small probe is dominated by per-call costs
    and would size the sample short), and topped up once if it still ran under
    60 % of the budget."""
    import numpy as np
    import oracle

    outs = []

    def run(rows, keep=True):
        t0 = time.perf_counter()
        res = oracle.attention(q, k, v, w.causal, w.scale, rows=rows, threads=threads)
        dt = time.perf_counter() - t0
        if keep:
            outs.append(res)
        return dt

    total = w.B * w.H * w.Sq
    probe = sample_rows(w, n_total=min(64 if threads == 1 else 512, total), seed=seed)
    per_flop = max(run(probe, keep=False), 1e-6) / oracle_rows_flops(w, probe)
    avg_row = w.exact_flops() / total
    rows, dt, fl = [], 0.0, 0.0
    for attempt in range(2):
        n = int(max(16, min(total, (budget_s - dt) / (per_flop * avg_row))))
        r = sample_rows(w, n_total=n, seed=seed + 1 + attempt)
        dt += run(r)
        fl += oracle_rows_flops(w, r)
        rows += r
        if dt >= 0.6 * budget_s or n >= total:
            break
        per_flop = dt / fl
    o_ref = np.concatenate([np.asarray(a).reshape(-1, w.d) for a, _ in outs])
    l_ref = np.concatenate([np.asarray(b).reshape(-1) for _, b in outs])
    return rows, dt, fl, (o_ref, l_ref)


TOL = {"o_max_abs": 2e-2, "o_mean_abs": 2e-3, "lse_max_abs": 1e-3}


def parity_of_rows(o_dev, lse_dev, rows, ref):
    """Element-wise errors of the GPU's O and LSE on `rows` against the oracle's
    values for the same rows (the parity bars of the benchmark spec's tolerance)."""
    import numpy as np

    o_ref, l_ref = ref
    idx = torch.tensor(rows, dtype=torch.long, device=o_dev.device)
    og = o_dev[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    lg = lse_dev[idx[:, 0], idx[:, 1], idx[:, 2]].double().cpu().numpy()
    fin = np.isfinite(l_ref)
    err = np.abs(og - o_ref)
    lerr = np.abs(lg[fin] - l_ref[fin]) if fin.any() else np.zeros(1)
    out = {"rows": len(rows), "o_max_abs": float(err.max()), "o_mean_abs": float(err.mean()),
           "lse_max_abs": float(lerr.max()),
           "masked_rows_match": bool(np.array_equal(np.isfinite(lg), fin))}
    out["pass"] = bool(out["masked_rows_match"] and all(out[k] <= v for k, v in TOL.items()))
    out["tol"] = TOL
    return out


def measure_exp_pipe(w, device, sptr):
    """The softmax's second bound: exp2 (MUFU) throughput from a microbenchmark,
    against the exponentials one step of the prefill kernel computes (every
    element of every computed tile; diagonal tiles are computed in full)."""
    from exact_tiled_attention_03_gb300 import _capi

    sms = torch.cuda.get_device_properties(device).multi_processor_count
    blocks, iters = sms * 8, 4096
    out = torch.empty(blocks * 256, dtype=torch.float32, device=device)
    for _ in range(3):
        _capi.check(_capi.fa_selftest_mufu(out, blocks, iters, sptr), "mufu")
    stream = torch.cuda.current_stream(device)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(5):
        _capi.check(_capi.fa_selftest_mufu(out, blocks, iters, sptr), "mufu")
    b.record(stream)
    torch.cuda.synchronize(device)
    rate = 5 * blocks * 256 * iters * 8 / (a.elapsed_time(b) * 1e-3)
    tiles = 0
    n_q = -(-w.Sq // 128)
    for qt in range(n_q):
        last = min(qt * 128 + 127, w.Sq - 1)
        tiles += -(-w.visible_keys(last) // 128)
    exps = w.B * w.H * tiles * 128 * 128
    return {"ex2_per_s": rate, "ex2_per_clk_per_sm_at_max_clock": rate / (sms * 2.07e9),
            "exps_per_step": exps, "ms_lower_bound": exps / rate * 1e3,
            "tensor_ms_lower_bound": w.exact_flops() / 1917.5e12 * 1e3}


MMA_FORMS = {0: "ss_n128", 1: "ss_2x_n64", 2: "ts_n128", 3: "ts_2x_n64", 4: "ss_n256",
             5: "e4m3_ss_n128", 6: "e4m3_ts_n128"}


def measure_mma_rate(device, sptr):
    """SM cycles per 128 x 128 x 128 tcgen05 product in each operand form (bf16,
    and E4M3 with .kind::f8f6f4), one CTA per SM, median over CTAs. 512 is the
    nominal dense bf16 rate."""
    from exact_tiled_attention_03_gb300 import _capi

    sms = torch.cuda.get_device_properties(device).multi_processor_count
    cyc = torch.empty(sms, dtype=torch.int64, device=device)
    iters, out = 1000, {}
    for mode, name in MMA_FORMS.items():
        for _ in range(2):
            _capi.check(_capi.fa_selftest_mma_rate(cyc, mode, sms, iters, sptr), "mma_rate")
        torch.cuda.synchronize(device)
        per = cyc.double().median().item() / (iters * (2 if mode == 4 else 1))
        out[name] = round(per, 1)
    return {"clk_per_128x128x128": out, "nominal": 512,
            "e4m3_over_bf16_rate": out["ss_n128"] / out["e4m3_ss_n128"]}


def run_reference(args, world, rank):
    """--impl reference: the fp64 CPU oracle on the same workload, rank 0 only
    (under a launcher every rank joins the process group, then the others exit)."""
    init_dist(world, "gloo")
    barrier(world)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return 0
    import oracle

    w = WORKLOADS[args.workload]
    q, k, v = make_qkv(w)
    cores = oracle.max_threads()
    total_budget = args.ref_budget
    rows_probe, dt_probe, fl_probe, _ = time_oracle_sample(w, q, k, v,
                                                           budget_s=min(2.0, total_budget / 4))
    per_flop = dt_probe / fl_probe
    avg_row = w.exact_flops() / (w.B * w.H * w.Sq)
    n_rows = int(max(1, total_budget / (args.steps + args.warmup) / (per_flop * avg_row)))
    times, flops = [], []
    for s in range(args.warmup + args.steps):
        rows = sample_rows(w, n_total=n_rows, seed=100 + s)
        t0 = time.perf_counter()
        oracle.attention(q, k, v, w.causal, w.scale, rows=rows)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
            flops.append(oracle_rows_flops(w, rows))
    value = sum(flops) / sum(times) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * sum(times) / len(times), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n_rows} seeded query rows of the workload per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def measure_backward(w, device, sptr, args, peaks):
    from exact_tiled_attention_03_gb300 import _capi

    q, k, v = (t.to(device) for t in make_qkv(w))
    g = torch.Generator(device=device).manual_seed(w.seed + 1)
    do = torch.randn(q.shape, generator=g, device=device).to(torch.bfloat16)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=device)
    _capi.check(_capi.fa_forward(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, w.causal, w.scale,
                                 sptr), "fa_forward")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    nb = _capi.fa_backward_workspace_size(w.B, w.H, w.Sq, w.Sk, w.d)
    ws = torch.empty(nb, dtype=torch.uint8, device=device)

    def step():
        st = _capi.fa_backward(q, k, v, o, lse, do, dq, dk, dv, w.B, w.H, w.Sq, w.Sk, w.d,
                               w.causal, w.scale, ws, nb, sptr)
        if st != 0:
            raise _capi.FAError(st, "fa_backward")

    for _ in range(args.warmup):
        step()
    n = max(10, args.steps // 4)
    per = time_steps(step, n, torch.cuda.current_stream(device)) / n
    _capi.check(_capi.fa_device_status(sptr), "device status after backward")
    flops = 2.5 * w.exact_flops()
    tf = flops / per / 1e12
    return {"workload": w.name, "ms_per_step": per * 1e3, "TFLOP/s": tf,
            "frac_bf16_peak": tf / peaks["bf16_tflops"], "flops_per_step": flops,
            "launches_per_step": 3, "kernels": "prep + dK/dV (4 GEMMs) + dQ (3 GEMMs)",
            "traffic": {k: ncu_traffic(k, BWD_SOURCES, w.name)
                        for k in ("fa_bwd_dkdv_kernel<128>", "fa_bwd_dq_kernel<128>")}}


OTHER_FORWARD = ("prefill_b4h32s2048d128_causal", "prefill_b4h32s2048d128_causal_q4",
                 "prefill_b1h32s32768d64_causal")


def measure_other_forward(device, sptr, args, peaks):
    """The other prefill configurations (2K, 2K with Q x 4, 32K at d = 64) through the
    same entry point, each against the bf16 tensor roofline."""
    from exact_tiled_attention_03_gb300 import _capi

    out = {}
    for name in OTHER_FORWARD:
        w = WORKLOADS[name]
        q, k, v = (t.to(device) for t in make_qkv(w))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=device)

        def step():
            st = _capi.fa_forward(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, w.causal, w.scale,
                                  sptr)
            if st != 0:
                raise _capi.FAError(st, "fa_forward")

        for _ in range(args.warmup):
            step()
        n = max(10, min(200, int(0.2 / max(1e-6, w.exact_flops() / 1e15))))
        per = time_steps(step, n, torch.cuda.current_stream(device)) / n
        _capi.check(_capi.fa_device_status(sptr), "device status after " + name)
        tf = w.exact_flops() / per / 1e12
        out[name] = {"ms_per_step": per * 1e3, "TFLOP/s": tf,
                     "frac_bf16_peak": tf / peaks["bf16_tflops"], "steps": n}
        del q, k, v, o, lse
    return out


def measure_fp8(w, device, sptr, args, peaks, mma_rate):
    """The FP8 forward (E4M3 Q, K, V with per-tensor descales, bf16 O) on the same
    workload and algorithmic FLOPs, against the FP8 dense peak: the measured
    bf16 burst peak times the measured ratio of the tcgen05 rates (cycles per
    128 x 128 x 128 product, bf16 over E4M3, both operands from shared memory)."""
    from exact_tiled_attention_03_gb300 import _capi
    from exact_tiled_attention_03_gb300.inputs import make_qkv_fp8

    q8, k8, v8, ds = make_qkv_fp8(w)
    q8, k8, v8 = (t.view(torch.uint8).to(device) for t in (q8, k8, v8))
    o = torch.empty((w.B, w.H, w.Sq, w.d), dtype=torch.bfloat16, device=device)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=device)

    def step():
        st = _capi.fa_forward_fp8(q8, k8, v8, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, w.causal,
                                  w.scale, ds[0], ds[1], ds[2], sptr)
        if st != 0:
            raise _capi.FAError(st, "fa_forward_fp8")

    for _ in range(args.warmup):
        step()
    n = max(10, args.steps // 2)
    per = time_steps(step, n, torch.cuda.current_stream(device)) / n
    _capi.check(_capi.fa_device_status(sptr), "device status after fp8")
    tf = w.exact_flops() / per / 1e12
    ratio = mma_rate["e4m3_over_bf16_rate"]
    peak = ratio * peaks["bf16_tflops"]
    return {"workload": w.name, "ms_per_step": per * 1e3, "TFLOP/s": tf, "peak": peak,
            "peak_source": f"{peaks['source']} bf16 burst x {ratio:.3f}, the measured "
                           "e4m3/bf16 rate ratio (tcgen05 kind::f8f6f4 microbenchmark)",
            "frac_of_nominal_2x": tf / (2.0 * peaks["bf16_tflops"]),
            "frac": tf / peak, "dtype": "e4m3 in, fp32 accumulate, bf16 out",
            "launches_per_step": 1,
            "traffic": ncu_traffic("fa_prefill_fp8_kernel", FP8_SOURCES, w.name)}


def measure_verify_variants(wv, device, sptr, args, peaks):
    """GB/s of the verify workload as a draft tree (random trees over the 5
    candidates) and read from a paged cache (random block table; page sizes
    16 and 64), against the same algorithmic bytes as the contiguous form."""
    from exact_tiled_attention_03_gb300 import _capi
    from exact_tiled_attention_03_gb300.inputs import make_tree_masks

    q, k, v = (t.to(device) for t in make_qkv(wv))
    o = torch.empty_like(q)
    lse = torch.empty((wv.B, wv.H, wv.Sq), dtype=torch.float32, device=device)
    n_split = _capi.fa_verify_auto_splits(wv.B, wv.H, wv.Sq, wv.Sk, wv.d)
    need = _capi.fa_verify_workspace_size(wv.B, wv.H, wv.Sq, wv.Sk, wv.d, n_split)
    ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)
    masks = make_tree_masks(wv.B, wv.Sq, seed=wv.seed).to(device)
    out = {}

    def timed(fn):
        for _ in range(args.warmup):
            fn()
        n = max(10, args.steps)
        per = time_steps(fn, n, torch.cuda.current_stream(device)) / n
        gbs = wv.io_bytes() / per / 1e9
        return {"us_per_step": per * 1e6, "GB/s": gbs, "frac": gbs / peaks["hbm_gbs"]}

    def tree():
        st = _capi.fa_verify_tree_forward(q, k, v, o, lse, wv.B, wv.H, wv.Sq, wv.Sk, wv.d, masks,
                                          wv.scale, n_split, ws, need, sptr)
        if st != 0:
            raise _capi.FAError(st, "fa_verify_tree_forward")
    out["tree"] = timed(tree)
    for P in (16, 64):
        n_lp = wv.Sk // P
        g = torch.Generator(device=device).manual_seed(wv.seed + P)
        perm = torch.randperm(wv.B * n_lp, generator=g, device=device)
        pages_k = k.reshape(wv.B, wv.H, n_lp, P, wv.d).permute(0, 2, 1, 3, 4).reshape(-1, wv.H, P, wv.d)
        pages_v = v.reshape(wv.B, wv.H, n_lp, P, wv.d).permute(0, 2, 1, 3, 4).reshape(-1, wv.H, P, wv.d)
        kp = torch.empty_like(pages_k)
        vp = torch.empty_like(pages_v)
        kp[perm] = pages_k
        vp[perm] = pages_v
        table = perm.reshape(wv.B, n_lp).to(torch.int32).contiguous()
        lens = torch.full((wv.B,), wv.Sk, dtype=torch.int32, device=device)

        def paged():
            st = _capi.fa_verify_paged_forward(q, kp, vp, table, lens, o, lse, wv.B, wv.H, wv.Sq,
                                               wv.d, kp.shape[0], P, n_lp, wv.Sk, 1, None,
                                               wv.scale, n_split, ws, need, sptr)
            if st != 0:
                raise _capi.FAError(st, "fa_verify_paged_forward")
        out[f"paged_p{P}"] = timed(paged)
        del kp, vp, pages_k, pages_v
    torch.cuda.synchronize()
    return out



def main_roofline(w, per_launch_s: float, peaks, n_split: int):
    """The roofline object of the main line and the launches per step.
    fa_forward runs decode-shaped problems (Sq <= FA_VERIFY_MAX_SQ) on the
    split-KV verify kernel, which is bound by HBM (n_split > 1 adds the combine
    launch), and the rest on the prefill kernel, bound by the tensor pipe."""
    from exact_tiled_attention_03_gb300._capi import FA_VERIFY_MAX_SQ

    if 0 < w.Sq <= FA_VERIFY_MAX_SQ:
        gbs = w.io_bytes() / per_launch_s / 1e9
        return ({"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                 "frac": gbs / peaks["hbm_gbs"], "peak_source": f"{peaks['source']} HBM copy",
                 "kernel": "fa_verify_split_kernel", "n_split": n_split,
                 "traffic": ncu_traffic("fa_verify_split_kernel", VERIFY_SOURCES, w.name)},
                1 if n_split == 1 else 2)
    achieved = w.exact_flops() / per_launch_s / 1e12
    return ({"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
             "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
             "peak_source": f"{peaks['source']} bf16 burst",
             "frac_sustained": achieved / peaks["bf16_tflops_sustained"],
             "peak_sustained": peaks["bf16_tflops_sustained"],
             "kernel": f"fa_prefill_kernel<{w.d}>",
             "traffic": ncu_traffic(f"fa_prefill_kernel<{w.d}>", PREFILL_SOURCES, w.name)},
            1)


def config_block(w, world):
    return {"workload": w.name, "B": w.B, "H": w.H, "Sq": w.Sq, "Sk": w.Sk, "d": w.d,
            "causal": w.causal, "scale": w.scale, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (no flush needed)",
            "flops_per_step": w.exact_flops(),
            "score_matrix_bytes_avoided": w.score_matrix_bytes()}


# ---------------------------------------------------------------- our arm
def run_ours(args, world, rank, local):
    import exact_tiled_attention_03_gb300 as fa
    from exact_tiled_attention_03_gb300 import _capi

    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    init_dist(world, "nccl")
    peaks = load_peaks()
    fa.load()

    w = rank_workload(args.workload, rank)
    q_h, k_h, v_h = make_qkv(w)
    q, k, v = q_h.to(device), k_h.to(device), v_h.to(device)
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.Sq), dtype=torch.float32, device=device)
    stream = torch.cuda.current_stream(device)
    sptr = stream.cuda_stream

    def step():
        st = _capi.fa_forward(q, k, v, o, lse, w.B, w.H, w.Sq, w.Sk, w.d, w.causal, w.scale, sptr)
        if st != 0:
            raise _capi.FAError(st, "fa_forward")

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    fa.check(fa.fa_device_status(sptr), "device status after warm-up")

    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        t0 = clk.mark()
        dt = time_steps(step, args.steps, stream)
        t1 = clk.mark()
        barrier(world)
    fa.check(fa.fa_device_status(sptr), "device status after timed region")
    dt_max = reduce_max(dt, world, device)
    flops_all = reduce_sum(float(w.exact_flops() * args.steps), world, device)
    value = flops_all / dt_max / 1e12
    per_launch_s = dt / args.steps
    clocks = clk.summary(t0, t1)
    ns = (_capi.fa_verify_auto_splits(w.B, w.H, w.Sq, w.Sk, w.d)
          if 0 < w.Sq <= _capi.FA_VERIFY_MAX_SQ else 0)
    roofline, launches_per_step = main_roofline(w, per_launch_s, peaks, ns)

    # the same step back to back for >= --sustained-s of device time, with its
    # own clock record: the steady state (power cap) next to the burst above
    sustained = None
    if args.sustained_s > 0:
        n_sus = max(args.steps, int(args.sustained_s / per_launch_s) + 1)
        with ClockSampler(local) as clk2:
            barrier(world)
            torch.cuda.synchronize()
            t0s = clk2.mark()
            ds = time_steps(step, n_sus, stream)
            t1s = clk2.mark()
            barrier(world)
        fa.check(fa.fa_device_status(sptr), "device status after sustained region")
        ds_max = reduce_max(ds, world, device)
        v_sus = reduce_sum(float(w.exact_flops() * n_sus), world, device) / ds_max / 1e12
        r_sus = main_roofline(w, ds / n_sus, peaks, ns)[0]
        sustained = {"value": v_sus, "unit": "TFLOP/s", "steps": n_sus, "device_s": ds_max,
                     "ms_per_step": 1e3 * ds_max / n_sus, "roofline_frac": r_sus["frac"],
                     "roofline_frac_sustained_peak": r_sus.get("frac_sustained"),
                     "clocks": clk2.summary(t0s, t1s)}

    # end to end through the C ABI call that takes host buffers (fa_forward_host):
    # pinned host inputs and outputs, every step's host-to-device and
    # device-to-host copies inside the timed region (pipelined by the call)
    e2e = None
    if not args.no_e2e:
        qp, kp, vp = q_h.pin_memory(), k_h.pin_memory(), v_h.pin_memory()
        op = torch.empty(o.shape, dtype=o.dtype, pin_memory=True)
        lp = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        ws_bytes = _capi.fa_forward_host_workspace_size(w.B, w.H, w.Sq, w.Sk, w.d)
        ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)

        def e2e_step():
            st = _capi.fa_forward_host(qp, kp, vp, op, lp, w.B, w.H, w.Sq, w.Sk, w.d, w.causal,
                                       w.scale, ws, ws_bytes, sptr)
            if st != 0:
                raise _capi.FAError(st, "fa_forward_host")

        for _ in range(3):
            e2e_step()
        n_e2e = max(3, min(20, args.steps // 10))
        barrier(world)
        de = time_steps(e2e_step, n_e2e, stream)
        de = reduce_max(de, world, device)
        fa.check(fa.fa_device_status(sptr), "device status after e2e")
        e2e = {"value": reduce_sum(float(w.exact_flops() * n_e2e), world, device) / de / 1e12,
               "unit": "TFLOP/s", "steps": n_e2e, "call": "fa_forward_host",
               "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in (qp, kp, vp)),
               "d2h_bytes_per_step": op.numel() * op.element_size() + lp.numel() * lp.element_size()}
        del ws

    # the decode-shaped verify path, against the HBM roofline
    verify = None
    verify_keep = None
    if not args.no_verify:
        wv = rank_workload(VERIFY, rank)
        qv, kv_, vv = (t.to(device) for t in make_qkv(wv))
        ov = torch.empty_like(qv)
        lv = torch.empty((wv.B, wv.H, wv.Sq), dtype=torch.float32, device=device)
        n_split = _capi.fa_verify_auto_splits(wv.B, wv.H, wv.Sq, wv.Sk, wv.d)
        need = _capi.fa_verify_workspace_size(wv.B, wv.H, wv.Sq, wv.Sk, wv.d, n_split)
        ws = torch.empty(max(need, 1), dtype=torch.uint8, device=device)

        def vstep():
            st = _capi.fa_verify_forward(qv, kv_, vv, ov, lv, wv.B, wv.H, wv.Sq, wv.Sk, wv.d,
                                         wv.causal, wv.scale, n_split, ws, need, sptr)
            if st != 0:
                raise _capi.FAError(st, "fa_verify_forward")

        def fstep():  # the main entry point: its own stream-ordered workspace
            st = _capi.fa_forward(qv, kv_, vv, ov, lv, wv.B, wv.H, wv.Sq, wv.Sk, wv.d, wv.causal,
                                  wv.scale, sptr)
            if st != 0:
                raise _capi.FAError(st, "fa_forward")

        n_v = max(200, args.steps)
        res = {}
        for name, fn in (("fa_forward", fstep), ("fa_verify_forward", vstep)):
            for _ in range(args.warmup):
                fn()
            res[name] = time_steps(fn, n_v, stream) / n_v
        fa.check(fa.fa_device_status(sptr), "device status after verify")
        per = res["fa_verify_forward"]
        gbs = wv.io_bytes() / per / 1e9
        gbs_f = wv.io_bytes() / res["fa_forward"] / 1e9
        verify = {"workload": wv.name, "us_per_step": per * 1e6, "GB/s": gbs,
                  "hbm_peak_GB/s": peaks["hbm_gbs"], "frac": gbs / peaks["hbm_gbs"],
                  "bytes_per_step": wv.io_bytes(), "n_split": n_split, "steps": n_v,
                  "launches_per_step": 1 if n_split == 1 else 2,
                  "via_fa_forward": {"us_per_step": res["fa_forward"] * 1e6, "GB/s": gbs_f,
                                     "frac": gbs_f / peaks["hbm_gbs"],
                                     "workspace": "library pool, stream-ordered"},
                  "traffic": ncu_traffic("fa_verify_split_kernel", VERIFY_SOURCES, wv.name)}
        del ws
        if rank == 0 and world == 1 and not args.no_cpu:
            verify_keep = (wv, tuple(t.cpu() for t in (qv, kv_, vv)), ov, lv)
        del qv, kv_, vv

    # the backward pass on the same workload (dQ, dK, dV by recomputation from
    # LSE); algorithmic FLOPs: 5 GEMMs of 2*d per visible pair = 2.5x forward
    backward = None
    if not args.no_backward:
        backward = measure_backward(w, device, sptr, args, peaks)

    # the tensor-pipe rates (bf16 and E4M3 forms) and the exp-pipe bound of the
    # prefill step (microbenchmarks)
    mma_rate = measure_mma_rate(device, sptr)
    exp_pipe = measure_exp_pipe(w, device, sptr)

    # the FP8 forward on the same workload
    fp8 = None
    if not args.no_fp8:
        fp8 = measure_fp8(w, device, sptr, args, peaks, mma_rate)

    # the other prefill configurations
    forward_other = None if args.no_other else measure_other_forward(device, sptr, args, peaks)

    # the verify step's tree-mask and paged-cache forms, same bytes and roofline
    verify_ext = None
    if not args.no_verify:
        verify_ext = measure_verify_variants(rank_workload(VERIFY, rank), device, sptr, args,
                                             peaks)

    # the CPU oracle on a bounded sample (rank 0, N = 1 only); the same rows
    # give the parity of the GPU outputs against the oracle
    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle

        cores = oracle.max_threads()
        rows, dtc, flc, ref = time_oracle_sample(w, q_h, k_h, v_h, budget_s=args.cpu_budget)
        rows1, dt1, fl1, _ = time_oracle_sample(w, q_h, k_h, v_h, budget_s=2.0, seed=11,
                                                threads=1)
        cpu = {"value": flc / dtc / 1e12, "unit": "TFLOP/s", "cores": cores,
               "kind": "oracle",
               "sample": f"{len(rows)} seeded query rows of {w.name} "
                         f"({flc:.3e} algorithmic FLOPs, {dtc:.1f} s)",
               "one_core_value": fl1 / dt1 / 1e12,
               "one_core_sample": f"{len(rows1)} rows, {dt1:.1f} s",
               "affinity_cpus": len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else None,
               "omp_num_threads": os.environ.get("OMP_NUM_THREADS"),
               "full_size_s_extrapolated": w.exact_flops() / (flc / dtc)}
        # the GPU's O and LSE on the rows the oracle just computed
        parity = {w.name: parity_of_rows(o, lse, rows, ref)}
        if verify_keep is not None:
            wv, (qv_h, kv_h, vv_h), ov, lv = verify_keep
            rv, dtv, flv, refv = time_oracle_sample(wv, qv_h, kv_h, vv_h, budget_s=3.0, seed=13)
            parity[wv.name] = parity_of_rows(ov, lv, rv, refv)
            cpu["verify"] = {"value": wv.io_bytes() * (flv / wv.exact_flops()) / dtv / 1e9,
                             "unit": "GB/s", "sample": f"{len(rv)} seeded query rows of "
                             f"{wv.name} ({dtv:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_block(w, world),
            "roofline": roofline,
            "pct_of_bf16_peak": 100.0 * value / world / peaks["bf16_tflops"],
            "fa_convention_tflops": w.fa_convention_flops() * args.steps * world / dt_max / 1e12,
            "e2e": e2e, "verify": verify, "verify_variants": verify_ext, "backward": backward,
            "fp8": fp8, "forward_other": forward_other, "exp_pipe": exp_pipe, "mma_rate": mma_rate,
            "cpu_baseline": cpu, "parity": parity, "sustained": sustained,
            "clocks": clocks,
            "gpu_launches": args.steps * launches_per_step,
            "gpu": torch.cuda.get_device_name(device),
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def launch_command(argv, n: int, port: int):
    """The torchrun command that runs this script as `n` ranks on this node
    (one process per GPU, rendezvous on 127.0.0.1)."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
            f"--nproc-per-node={n}", "--master-addr", "127.0.0.1", "--master-port", str(port),
            os.path.abspath(__file__)] + list(argv)


def launch_ranks(argv, n: int) -> int:
    """`bench.py --gpus N` started without a launcher: start N ranks under
    torchrun and return their exit status (rank 0 prints the line)."""
    import socket

    with socket.socket() as sock:
        sock.bind(("127.0.0.1", 0))
        port = sock.getsockname()[1]
    return subprocess.run(launch_command(argv, n, port)).returncode


def main(argv=None):
    argv = list(sys.argv[1:] if argv is None else argv)
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE, choices=sorted(WORKLOADS))
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-verify", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-backward", action="store_true")
    ap.add_argument("--no-fp8", action="store_true")
    ap.add_argument("--no-other", action="store_true",
                    help="skip the other prefill configurations (2K, 2K Q x 4, 32K d = 64)")
    ap.add_argument("--ref-budget", type=float, default=120.0,
                    help="--impl reference: seconds of oracle time for the whole run")
    ap.add_argument("--sustained-s", type=float, default=1.5,
                    help="device seconds of back-to-back steps for the sustained record (0: off)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return launch_ranks(argv, args.gpus)
    world, rank, local = dist_env()
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but the launcher started {world} ranks")
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
