"""Benchmark of the sparse MoE FFN layer forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-decode] [--no-cpu-baseline] [--all]

One step = one moe_forward (router + top-K + softmax, dispatch, routed and
shared expert FFN, combine) over one batch of the workload's synthetic tokens,
inputs resident in HBM.  Default workload: the largest single-GPU layer, the
DeepSeek-V3-shaped prefill chunk with Zipf load imbalance (T=16384, d=7168,
E=256, K=8, I=2048, one shared expert, bf16).  Every weight set is larger than
the 129 MB L2, so no flush is needed between steps.  Also reported: the
dominant stage (the expert FFN) against its roofline, timed over at least 100
repeats with its own clock record; the end-to-end number through the C ABI
with host buffers; the Mixtral-shaped prefill layer; the DeepSeek-V3-shaped
decode layer (T=8) in microseconds per call against the HBM roofline; the
token-count sweep on the DeepSeek-V3 shape (T = 1, 8, 64, 512, 4096) with its
HBM and tensor fractions; and the fp64 CPU oracle on a bounded sample of the
same workload.  Under torchrun every rank runs an independent replica on its
own tokens (weak scaling, no collective on the data path).

``--impl reference`` times the CPU oracle (the only reference this layer has)
on the host cores for the same workload and metric.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import moe_inputs as mi  # noqa: E402

DEFAULT_WORKLOAD = "dsv3_prefill_zipf"
DECODE_WORKLOAD = "dsv3_decode"
MIXTRAL_WORKLOAD = "mixtral_prefill"
SWEEP_T = "1,8,64,512,4096"
STAGE_REPEATS = 100   # the dominant stage's timed loop (>= 1 s of clock samples at prefill sizes)


def source_sha256() -> str:
    """sha256 (first 16 hex digits) over the library's sources and public
    header, in name order: the build a result or a profile was taken on."""
    import glob
    import hashlib
    h = hashlib.sha256()
    files = sorted(glob.glob(os.path.join(ROOT, "sparse_expert_ffn_moe_gb300", "csrc", "*"))) + \
        [os.path.join(ROOT, "include", "moe.h")]
    for f in files:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


# --------------------------------------------------------------------------- work accounting

def layer_flops(cfg) -> int:
    """Router GEMM + routed SwiGLU experts (K per token) + shared expert."""
    return (2 * cfg.T * cfg.d * cfg.E + 6 * cfg.T * cfg.K * cfg.d * cfg.I
            + 6 * cfg.T * cfg.d * cfg.Is)


def ffn_flops(cfg) -> int:
    return 6 * cfg.T * cfg.K * cfg.d * cfg.I + 6 * cfg.T * cfg.d * cfg.Is


def elem_bytes(cfg) -> int:
    return 2 if cfg.dtype == "bf16" else 4


def expert_bytes(cfg, inter: int) -> int:
    """Bytes of one expert's three matrices (E4M3: one byte per weight plus an
    fp32 scale per weight row, or per 128 x 128 block)."""
    if cfg.weights == "e4m3":
        return 3 * cfg.d * inter + 4 * (2 * inter + cfg.d)
    if cfg.weights == "e4m3b":
        return 3 * cfg.d * inter + 4 * 3 * (-(-cfg.d // 128)) * (-(-inter // 128))
    return elem_bytes(cfg) * 3 * cfg.d * inter


def fp8_calls(moe, cfg):
    """The layer and expert-stage entry points of an 8-bit-weight workload (row
    or block scales; 8-bit activations or not), or (None, None)."""
    if cfg.acts == "e4m3":
        if cfg.weights == "e4m3b":
            return moe.moe_forward_w8a8_blocks, moe.moe_expert_ffn_w8a8_blocks
        return moe.moe_forward_w8a8, moe.moe_expert_ffn_w8a8
    if cfg.weights == "e4m3b":
        return moe.moe_forward_fp8_blocks, moe.moe_expert_ffn_fp8_blocks
    if cfg.weights == "e4m3":
        return moe.moe_forward_fp8, moe.moe_expert_ffn_fp8
    return None, None


WEIGHT_FORMAT = {"e4m3": "e4m3 + fp32 row scales", "e4m3b": "e4m3 + fp32 128x128 block scales"}


def layer_bytes(cfg, n_active: int) -> int:
    """Algorithmic HBM bytes of one call: router weights, the weights of every
    expert that got at least one token, the shared expert, x in and y out.
    Permuted copies and intermediates are implementation traffic, not counted."""
    s = elem_bytes(cfg)
    shared = expert_bytes(cfg, cfg.Is) if cfg.Is else 0
    return (s * (cfg.E * cfg.d + 2 * cfg.T * cfg.d) + n_active * expert_bytes(cfg, cfg.I)
            + shared)


def ffn_stage_bytes(cfg, n_active: int) -> int:
    """Algorithmic bytes of the routed expert-FFN stage: the active experts'
    weights, the permuted rows in and the expert outputs out."""
    return n_active * expert_bytes(cfg, cfg.I) + 2 * elem_bytes(cfg) * cfg.T * cfg.K * cfg.d


class Forward:
    """One moe_forward (moe_forward_fp8 for 8-bit expert weights,
    moe_forward_w8a8 for 8-bit weights and activations) on fixed buffers; the
    argument structs are built once."""

    def __init__(self, moe, cfg, s, p, bias, ws, stream):
        self.moe, self.cfg, self.s, self.p, self.bias, self.ws, self.stream = (
            moe, cfg, s, p, bias, ws, stream)
        self.fp8 = moe.make_fp8_experts(p) if mi.is_fp8(cfg) else None
        self.fwd8 = fp8_calls(moe, cfg)[0]

    def __call__(self, x, y):
        m, p = self.moe, self.p
        if self.fp8 is not None:
            self.fwd8(self.s, x, p["w_g"], self.bias, self.fp8, y, self.ws, stream=self.stream)
        else:
            m.moe_forward(self.s, x, p["w_g"], self.bias, p["w_gate"], p["w_up"], p["w_down"],
                          p.get("ws_gate"), p.get("ws_up"), p.get("ws_down"), y, self.ws,
                          stream=self.stream)


def oracle_tokens(cfg, tokens, x_host, p_host, bias_host):
    """The oracle's per-token layer in the workload's weight format."""
    import oracle
    if mi.is_fp8(cfg):
        return oracle.forward_tokens_fp8(tokens, x_host, p_host["w_g"], p_host, cfg.K,
                                         dtype=cfg.dtype, bias=bias_host, router=cfg.router,
                                         act8=cfg.acts == "e4m3",
                                         blocks=cfg.weights == "e4m3b")
    return oracle.forward_tokens(tokens, x_host, p_host, cfg.K, dtype=cfg.dtype, bias=bias_host,
                                 router=cfg.router)


def launches_per_forward(cfg, gemv_limit: int = 0) -> int:
    """Kernels libmoe launches for one moe_forward (mirrors the host logic in
    moe_api.cu): router (GEMV or tcgen05) + top-K (one fused launch for at most
    16 tokens with MOE_FUSED_ROUTER=1), 3 dispatch kernels and the FFN
    plan (one fused launch when T*K <= 1024 and E <= 1024), the row gather when
    the tensor-core path may run,
    (2 GEMV kernels only for fp32 layers or a non-zero GEMV row limit), the
    single-SM tcgen05 gate/up and down GEMMs when needed, and the CTA-pair
    ones too when a group can hold more rows than one 128-row tile (or, with
    MOE_PAIR_MIN_ROWS set, at least that many rows), combine."""
    # small batches: the 3 dispatch kernels and the plan are one launch
    fused = cfg.T * cfg.K <= 1024 and cfg.E <= 1024 and \
        os.environ.get("MOE_FUSED_DISPATCH", "1") != "0"
    disp_plan = 1 if fused else 3 + 1
    # router + top-K: one fused launch for at most 16 tokens when MOE_FUSED_ROUTER=1
    router = 1 if 0 < cfg.T <= 16 and os.environ.get("MOE_FUSED_ROUTER", "0") == "1" else 2
    # block-scaled 8-bit weights take CTA-pair tiles only with MOE_W8_PAIR=1
    pair_ok = cfg.weights != "e4m3b" or os.environ.get("MOE_W8_PAIR", "0") == "1"
    if cfg.acts == "e4m3":
        # router + top-K, dispatch + plan, x quantiser, code gather,
        # tcgen05 gate/up, h quantiser (+ h_s), tcgen05 down -- the gate/up and
        # down twice when a group can take pair tiles -- combine
        pair = cfg.T > 128 and pair_ok
        return router + disp_plan + 1 + 1 + (2 if pair else 1) + (2 if cfg.Is else 1) \
            + (2 if pair else 1) + 1
    if mi.is_fp8(cfg):
        # router + top-K, 3 dispatch kernels and the plan, the 8-bit GEMV
        # (gate/up and down for each of its two group lists), and when a group
        # can exceed the GEMV limit: with two-plane activations (the default;
        # always with block scales) the x split and the plane gather, the
        # tcgen05 gate/up, the h split (+ h_s), the tcgen05 down -- gate/up and
        # down twice when a group can take pair tiles; with the codes widened
        # in the GEMM, the row gather and one gate/up and one down; combine
        # (row scales: no GEMV once some group can exceed 64 rows, i.e. T > 64)
        limit = int(os.environ.get("MOE_GEMV8_MAX_ROWS",
                                   "0" if cfg.weights == "e4m3" and cfg.T > 64 else "8"))
        gemv = (2 if limit > 0 else 0) + (2 if limit > 8 else 0)
        if cfg.T > limit and (os.environ.get("MOE_W8_PLANES", "1") != "0"
                              or cfg.weights == "e4m3b"):
            pair = cfg.T > 128 and pair_ok
            tc = 2 * (2 if pair else 1) + (2 if cfg.Is else 1)
            return router + disp_plan + 2 + gemv + tc + 1
        tc = 2 if cfg.T > limit else 0
        return router + disp_plan + 1 + gemv + tc + 1
    need_tc = cfg.dtype == "bf16" and cfg.T > gemv_limit
    # the permuted copy of the routed rows: not made when every row of the batch is
    # gathered inside the GEMM (by default, batches of at most 16 tokens)
    gather_max = int(os.environ.get("MOE_GATHER_MAX_ROWS", "16" if cfg.T <= 16 else "0"))
    gather = need_tc and cfg.T > gather_max
    gemv = cfg.dtype == "f32" or gemv_limit > 0
    pair_min = int(os.environ.get("MOE_PAIR_MIN_ROWS", "0"))
    pair = need_tc and (cfg.T >= pair_min if pair_min > 0 else cfg.T > 128)
    # small batches with a shared expert: its gate/up and down in two launches of
    # their own (beside the routing, on a side stream)
    apart = (2 if need_tc and not gemv and cfg.Is and not pair
             and cfg.T <= int(os.environ.get("MOE_SHARED_APART", "0")) else 0)
    return (router + disp_plan + (1 if gather else 0) + (2 if gemv else 0) + (2 if need_tc else 0)
            + (2 if pair else 0) + apart + 1)


# --------------------------------------------------------------------------- helpers

def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, interval_ms: int = 25):
        self.index = index
        self.interval_ms = interval_ms
        self.proc = None
        self.lines: list[str] = []
        self.reader = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
            # the timed region starts once samples are flowing
            t0 = time.time()
            while not self.lines and time.time() - t0 < 10:
                time.sleep(0.02)
        except (OSError, ValueError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.reader:
                self.reader.join(timeout=2)

    def summary(self) -> dict:
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            try:
                pw.append(float(parts[2]))
            except ValueError:
                pass
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
               "reasons": sorted(reasons), "samples": len(sm), "interval_ms": self.interval_ms}
        if pw:
            out["power_w_median"] = statistics.median(pw)
            out["power_w_max"] = max(pw)
        return out


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(v: float, ws: int) -> float:
    if ws <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(ws: int):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


# --------------------------------------------------------------------------- CPU oracle timing

def oracle_tokens_per_s(cfg, x_host, p_host, bias_host, budget_s: float = 15.0,
                        seed_name: str = "cpu_sample"):
    """The fp64 oracle as it stands on the host cores: the layer for a growing
    seeded sample of tokens until about budget_s of CPU time has been spent."""
    import oracle
    threads = oracle.default_threads()
    n, spent, done = max(1, threads), 0.0, 0
    t_start = time.perf_counter()
    while True:
        tokens = mi.sample_tokens(cfg.T, n, seed=cfg.seed, name=f"{seed_name}/{n}").numpy()
        t0 = time.perf_counter()
        oracle_tokens(cfg, tokens, x_host, p_host, bias_host)
        dt = time.perf_counter() - t0
        spent += dt
        done = len(tokens)
        rate = done / dt
        if spent >= budget_s * 0.4 or n >= cfg.T:
            return {"value": rate, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                    "sample": f"{done} seeded tokens of {cfg.name} (T={cfg.T}), full layer per "
                              f"token (router over all E, K routed experts, shared expert) in fp64; "
                              f"{time.perf_counter() - t_start:.1f} s of wall time"}
        n = min(cfg.T, max(n + 1, int(n * max(2.0, (budget_s * 0.5) / max(dt, 1e-3)))))


# --------------------------------------------------------------------------- our arm

def run_ours(args):
    import torch

    ws_n, rank, local = dist_env()
    if ws_n > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    import sparse_expert_ffn_moe_gb300 as moe

    peaks = load_peaks()
    cfg = mi.CONFIGS[args.workload]
    # every rank draws its own tokens (a replica serving a different batch)
    cfg_r = mi.LayerConfig(**{**cfg.__dict__, "seed": cfg.seed + rank})
    p = mi.make_weights(cfg_r, "cuda")
    x = mi.make_x(cfg_r, "cuda")
    bias = mi.make_bias(cfg_r, "cuda")
    s = moe.make_shape(cfg.T, cfg.d, cfg.E, cfg.K, cfg.I, cfg.Is, cfg.dtype, cfg.router)
    ws = moe.alloc_workspace(s)
    y = torch.empty_like(x)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()  # every input is written before the side stream reads it

    call = Forward(moe, cfg, s, p, bias, ws, stream)

    def fwd(xx=x, yy=y):
        call(xx, yy)

    # active experts of this batch (for the byte count), from the library's own routing
    n_active = count_active(moe, cfg, x, p, bias, stream)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            fwd()
    torch.cuda.synchronize()
    code = moe.moe_get_device_error(ws)
    if code:
        raise RuntimeError(f"device error during warm-up: {moe.status_string(code)}")

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(torch.cuda.current_device()) as clk:
        barrier(ws_n)
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            fwd()
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(ws_n)
    spread = step_stats(fwd, stream, args.steps)
    # dominant stage, timed alone on the same stream over >= STAGE_REPEATS calls, with
    # its own clock record: the expert FFN (tcgen05 gate/up GEMM with fused SiLU*mul,
    # then the down GEMM) of this batch
    with ClockSampler(torch.cuda.current_device()) as stage_clk:
        stage = time_expert_ffn(moe, cfg, x, p, bias, stream, max(STAGE_REPEATS, args.steps),
                                n_active)
    stage["clocks"] = stage_clk.summary()
    t_ms = ev0.elapsed_time(ev1) / args.steps
    t_ms_max = max_over_ranks(t_ms, ws_n)
    code = moe.moe_get_device_error(ws)
    if code:
        raise RuntimeError(f"device error in the timed region: {moe.status_string(code)}")

    tokens_per_s = cfg.T * ws_n / (t_ms_max / 1e3)
    e2e = time_e2e(call, stream, args.steps, x)
    e2e_ms = max_over_ranks(e2e["ms"], ws_n)

    result = {
        "metric": "MoE layer tokens/s",
        "value": tokens_per_s,
        "unit": "tokens/s",
        "n_gpus": ws_n,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": t_ms_max,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if cfg.acts == "e4m3" else cfg.dtype,
        "data": ("synthetic (seeded N(0,1) tokens, N(0,1/d) weights; no trained weights)"
                 if not mi.is_fp8(cfg) else
                 f"synthetic (seeded N(0,1) tokens; random E4M3 expert codes with fp32 "
                 f"{'row' if cfg.weights == 'e4m3' else '128x128 block'} scales; no trained "
                 f"weights)"),
        "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "E": cfg.E, "K": cfg.K,
                   "inter": cfg.I, "inter_shared": cfg.Is, "active_experts": n_active,
                   "expert_weights": WEIGHT_FORMAT.get(cfg.weights, cfg.dtype),
                   "expert_activations": ("e4m3 + fp32 row scales (x and h quantised per row)"
                                          if cfg.acts == "e4m3" else cfg.dtype),
                   "l2": "inputs larger than L2 (expert weights "
                         f"{cfg.E * expert_bytes(cfg, cfg.I) / 1e9:.2f} GB), no flush",
                   "parallelism": f"replicas x{ws_n} (independent batches, no collective)"},
        "layer": {"tflops": layer_flops(cfg) / (t_ms_max / 1e3) / 1e12,
                  "gbs": layer_bytes(cfg, n_active) / (t_ms_max / 1e3) / 1e9,
                  "flops": layer_flops(cfg), "alg_bytes": layer_bytes(cfg, n_active)},
        "roofline": stage_roofline(cfg, stage, peaks),
        "e2e": {"value": cfg.T * ws_n / (e2e_ms / 1e3), "unit": "tokens/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": e2e["h2d"],
                "d2h_bytes_per_step": e2e["d2h"]},
        "gpu_launches": launches_per_forward(cfg) * args.steps,
        # per-call spread, from a separate pass with an event between calls; the
        # back-to-back timed region lets each call's first kernels start while the
        # previous call's last ones finish (programmatic dependent launch), so
        # ms_per_step can sit below step_ms.median
        "step_ms": spread,
        "clocks": clk.summary(),
        "peaks": peaks,
        "source_sha256": source_sha256(),
    }
    if rank == 0:
        # the other workloads go last, so that they cannot disturb the lines above
        del call, ws, y
        torch.cuda.empty_cache()
        if not args.no_decode:
            result["decode"] = bench_decode(moe, peaks, args)
        if not args.no_extra and args.workload != MIXTRAL_WORKLOAD:
            result[MIXTRAL_WORKLOAD] = bench_workload(
                moe, mi.CONFIGS[MIXTRAL_WORKLOAD], peaks, steps=max(20, args.steps),
                graph=False, stage_repeats=max(STAGE_REPEATS, args.steps))
        if args.sweep_T:
            # the token-count sweep on the DeepSeek-V3 shape (uniform routing): the GEMV-like
            # to GEMM crossover against the HBM and tensor roofs
            base = mi.CONFIGS["dsv3_sweep_T8"]
            result["sweep"] = [
                bench_workload(moe, mi.CONFIGS.get(f"dsv3_sweep_T{t}", base.with_T(int(t))), peaks,
                               steps=max(20, args.steps), graph=int(t) <= 64)
                for t in args.sweep_T.split(",")]
        if args.all:
            result["workloads"] = bench_all(moe, peaks, args)
    if not args.no_cpu_baseline and rank == 0:
        torch.cuda.synchronize()
        hp = {k: mi.to_host_array(v) for k, v in p.items()}
        result["cpu_baseline"] = oracle_tokens_per_s(
            cfg_r, mi.to_host_array(x), hp,
            None if bias is None else bias.double().cpu().numpy(), budget_s=args.cpu_budget)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if ws_n > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def count_active(moe, cfg, x, p, bias, stream) -> int:
    import torch
    torch.cuda.synchronize()  # inputs were drawn on torch's current stream
    s = moe.make_shape(cfg.T, cfg.d, cfg.E, cfg.K, cfg.I, cfg.Is, cfg.dtype, cfg.router)
    ws = moe.alloc_workspace(s)
    idx = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device="cuda")
    moe.moe_route(s, x, p["w_g"], bias, None, None, idx, w, ws, stream=stream)
    torch.cuda.synchronize()
    return int(torch.unique(idx).numel())


def time_expert_ffn(moe, cfg, x, p, bias, stream, steps: int, n_active: int) -> dict:
    """Events around moe_expert_ffn (or moe_expert_ffn_fp8) alone: the routed
    experts of this batch."""
    import torch
    s = moe.make_shape(cfg.T, cfg.d, cfg.E, cfg.K, cfg.I, 0, cfg.dtype, cfg.router)
    ws = moe.alloc_workspace(s)
    n = cfg.T * cfg.K
    idx = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(cfg.E + 1, dtype=torch.int32, device="cuda")
    x_perm = torch.empty((n, cfg.d), dtype=x.dtype, device="cuda")
    y_perm = torch.empty((n, cfg.d), dtype=x.dtype, device="cuda")
    torch.cuda.synchronize()
    moe.moe_route(s, x, p["w_g"], bias, None, None, idx, w, ws, stream=stream)
    moe.moe_permute(s, idx, x, counts, offsets, None, None, x_perm, ws, stream=stream)

    fp8 = moe.make_fp8_experts(p) if mi.is_fp8(cfg) else None
    ffn8 = fp8_calls(moe, cfg)[1]

    def run():
        if fp8 is not None:
            ffn8(s, x_perm, offsets, fp8, y_perm, ws, stream=stream)
        else:
            moe.moe_expert_ffn(s, x_perm, offsets, p["w_gate"], p["w_up"], p["w_down"], y_perm,
                               ws, stream=stream)
    for _ in range(3):
        run()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"ms": ms, "flops": 6 * n * cfg.d * cfg.I, "bytes": ffn_stage_bytes(cfg, n_active),
            "repeats": steps}


# DRAM bytes (read + write) of one expert-FFN stage (its tcgen05 launches), from one
# ncu capture per workload, valid only for the ffn_tc.cu source it was taken on
# (sha256 prefix).
STAGE_TRAFFIC = {
    # the four GEMM launches of one stage call (pair and single gate/up, pair and single down)
    "dsv3_prefill_zipf": {"bytes": 9383788800 + 491185920 + 11156410112 + 44600320
                          + 2675092480 + 1703323648 + 5510793216 + 154811392,
                          "ffn_tc_sha256": "e21b475ffc96e160"},
    "mixtral_prefill": {"bytes": 1968544512 + 229080576 + 45312 + 1397152512 + 63691264 + 42240,
                        "ffn_tc_sha256": "e21b475ffc96e160"},
}


def stage_traffic(workload: str):
    import hashlib
    rec = STAGE_TRAFFIC.get(workload)
    if rec is None:
        return None
    path = os.path.join(ROOT, "sparse_expert_ffn_moe_gb300", "csrc", "ffn_tc.cu")
    with open(path, "rb") as f:
        sha = hashlib.sha256(f.read()).hexdigest()[:16]
    return rec["bytes"] if sha == rec["ffn_tc_sha256"] else None


def tensor_peak(cfg, peaks) -> tuple:
    """Dense tensor peak for the dtype the expert GEMMs multiply in: bf16 as
    measured, or (8-bit activations: E4M3 x E4M3) the measured bf16 peak times
    the nominal fp8 / bf16 ratio 4.5 / 2.25 = 2.  Two-plane activations run two
    E4M3 MMAs per bf16 one, the same tensor time: the bf16 peak."""
    if cfg.acts == "e4m3":
        return 2.0 * peaks["bf16_tflops"], (f"fp8 dense = 2 x measured bf16 burst "
                                            f"(nominal ratio), {peaks['source']}")
    return peaks["bf16_tflops"], f"bf16 dense, burst, {peaks['source']}"


def stage_roofline(cfg, stage, peaks) -> dict:
    """The expert-FFN stage against the roofline that binds it: the tensor
    pipe (dense, in the GEMMs' operand type) or HBM, whichever the stage comes
    closer to."""
    sec = stage["ms"] / 1e3
    tflops = stage["flops"] / sec / 1e12
    gbs = stage["bytes"] / sec / 1e9
    t_peak, t_kind = tensor_peak(cfg, peaks)
    t_frac, h_frac = tflops / t_peak, gbs / peaks["hbm_gbs"]
    planes = os.environ.get("MOE_W8_PLANES", "1") != "0" or cfg.weights == "e4m3b"
    kernel = ("expert FFN stage: tcgen05 gate/up GEMM (SiLU*mul epilogue) + tcgen05 down GEMM "
              + ("on E4M3 weights and E4M3 activations (kind::f8f6f4, + x and h quantisers)"
                 if cfg.acts == "e4m3" else
                 ("on E4M3 weights with bf16 activations as two E4M3 planes (kind::f8f6f4, "
                  "+ x and h splits)" if planes else "on E4M3 weights widened in-kernel")
                 + (", 128x128 block scales applied per 128-deep K block in registers"
                    if cfg.weights == "e4m3b" else "")
                 if mi.is_fp8(cfg) else
                 "(+ plan, empty GEMV launches)"))
    common = {"traffic": stage_traffic(cfg.name),
              "traffic_unit": "bytes per launch pair (DRAM read + write, ncu)",
              "kernel": kernel, "per_launch_flops": stage["flops"],
              "per_launch_bytes": stage["bytes"], "ms_per_launch": stage["ms"],
              "repeats": stage.get("repeats"), "other_frac": None}
    clk = stage.get("clocks")
    if clk and clk.get("sm_mhz"):
        # the clock behind the number: work per SM clock cycle of the whole GPU, and the
        # fraction of the peak scaled to the median SM clock sampled during the loop
        # (the measured peaks are taken as holding at the maximum SM clock)
        mhz, mx = clk["sm_mhz"], clk["sm_max_mhz"] or clk["sm_mhz"]
        common["clocks"] = clk
        common["per_cycle"] = {
            "flop_per_cycle": stage["flops"] / (sec * mhz * 1e6),
            "bytes_per_cycle": stage["bytes"] / (sec * mhz * 1e6),
            "tensor_frac_at_sampled_clock": t_frac * mx / mhz,
            "hbm_frac_at_sampled_clock": h_frac * mx / mhz}
    if t_frac >= h_frac:
        out = {"bound": "tensor", "achieved": tflops, "peak": t_peak,
               "unit": "TFLOP/s", "frac": t_frac, "peak_kind": t_kind}
        common["other_frac"] = {"hbm": h_frac}
        # the same against the measured back-to-back (power-capped) GEMM rate,
        # the ceiling that applies when the timed loop runs under sw_power_cap
        sus = peaks["bf16_tflops_sustained"] * (2.0 if cfg.acts == "e4m3" else 1.0)
        common["frac_of_sustained_peak"] = {"peak": sus, "frac": tflops / sus}
    else:
        out = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
               "frac": h_frac, "peak_kind": f"HBM copy, {peaks['source']}"}
        common["other_frac"] = {"tensor": t_frac}
    out.update(common)
    return out


def step_stats(fn, stream, steps: int) -> dict:
    """Per-call durations from an event between consecutive calls (a separate
    pass after the timed region, so the events cannot disturb it): median,
    standard deviation, min and max in ms."""
    import statistics
    import torch
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for i in range(steps):
            fn()
            ev[i + 1].record(stream)
    torch.cuda.synchronize()
    d = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return {"median": statistics.median(d), "std": statistics.pstdev(d), "min": min(d),
            "max": max(d), "n": steps}


def time_e2e(call, stream, steps, x_dev) -> dict:
    """Through the C ABI with host buffers: every step copies its x from pinned
    host memory to the device, runs the forward call and copies y back to pinned
    host memory, all inside the timed region.  Uploads and downloads run on two
    more streams with two device buffers each way, so step i+1's upload and step
    i-1's download overlap step i's compute (the usual serving pipeline); the
    events keep every buffer's reuse ordered."""
    import torch
    xh = x_dev.cpu().pin_memory()
    yh = [torch.empty_like(xh).pin_memory() for _ in range(2)]
    xd = [torch.empty_like(x_dev) for _ in range(2)]
    yd = [torch.empty_like(x_dev) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    up = [ev(), ev()]        # x copied into xd[b]
    done = [ev(), ev()]      # compute finished with xd[b] and wrote yd[b]
    down = [ev(), ev()]      # y copied out of yd[b]
    for b in range(2):       # every buffer starts free
        done[b].record(stream)
        down[b].record(d2h)

    def step(i):
        b = i & 1
        with torch.cuda.stream(h2d):
            h2d.wait_event(done[b])           # compute of step i-2 released xd[b]
            xd[b].copy_(xh, non_blocking=True)
            up[b].record(h2d)
        stream.wait_event(up[b])
        stream.wait_event(down[b])            # y of step i-2 copied out of yd[b]
        with torch.cuda.stream(stream):
            call(xd[b], yd[b])
            done[b].record(stream)
        with torch.cuda.stream(d2h):
            d2h.wait_event(done[b])
            yh[b].copy_(yd[b], non_blocking=True)
            down[b].record(d2h)

    for i in range(4):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d.wait_event(e0)                        # no timed copy starts before the clock does
    d2h.wait_event(e0)
    for i in range(steps):
        step(i)
    stream.wait_stream(d2h)                   # the last download is inside the timed region
    e1.record(stream)
    torch.cuda.synchronize()
    nbytes = xh.numel() * xh.element_size()
    return {"ms": e0.elapsed_time(e1) / steps, "h2d": nbytes, "d2h": nbytes}


def bench_decode(moe, peaks, args) -> dict:
    """DeepSeek-V3-shaped decode (T=8): microseconds per call against HBM, eager
    and as a replayed CUDA graph."""
    import torch
    cfg = mi.CONFIGS[DECODE_WORKLOAD]
    r = bench_workload(moe, cfg, peaks, steps=max(50, args.steps * 5), graph=True)
    return r


def bench_workload(moe, cfg, peaks, steps: int, graph: bool = False,
                   stage_repeats: int = 0) -> dict:
    import torch
    p = mi.make_weights(cfg, "cuda")
    x = mi.make_x(cfg, "cuda")
    bias = mi.make_bias(cfg, "cuda")
    s = moe.make_shape(cfg.T, cfg.d, cfg.E, cfg.K, cfg.I, cfg.Is, cfg.dtype, cfg.router)
    ws = moe.alloc_workspace(s)
    y = torch.empty_like(x)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()  # every input is written before the side stream reads it
    n_active = count_active(moe, cfg, x, p, bias, st)
    call = Forward(moe, cfg, s, p, bias, ws, st)

    def fwd():
        call(x, y)
    for _ in range(5):
        fwd()
    torch.cuda.synchronize()

    def timed(fn):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        for _ in range(steps):
            fn()
        e1.record(st)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    ms = timed(fwd)
    spread = step_stats(fwd, st, steps)
    out = {"workload": cfg.name, "T": cfg.T, "us_per_call": ms * 1e3,
           "us_per_call_median": spread["median"] * 1e3, "us_per_call_std": spread["std"] * 1e3,
           "tokens_per_s": cfg.T / (ms / 1e3), "active_experts": n_active,
           "alg_bytes": layer_bytes(cfg, n_active), "flops": layer_flops(cfg)}
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            fwd()
        def replay():
            with torch.cuda.stream(st):
                g.replay()
        replay()
        torch.cuda.synchronize()
        gms = timed(replay)
        out["us_per_call_graph"] = gms * 1e3
        ms = min(ms, gms)
    gbs = out["alg_bytes"] / (ms / 1e3) / 1e9
    tfs = out["flops"] / (ms / 1e3) / 1e12
    out["hbm_gbs"] = gbs
    out["hbm_frac"] = gbs / peaks["hbm_gbs"]
    out["tensor_tflops"] = tfs
    out["tensor_frac"] = tfs / tensor_peak(cfg, peaks)[0]
    code = moe.moe_get_device_error(ws)
    if code:
        raise RuntimeError(f"device error in {cfg.name}: {moe.status_string(code)}")
    if stage_repeats:
        # the expert-FFN stage of this batch against its roofline, with its clock record
        with ClockSampler(torch.cuda.current_device()) as clk:
            stage = time_expert_ffn(moe, cfg, x, p, bias, st, stage_repeats, n_active)
        stage["clocks"] = clk.summary()
        out["roofline"] = stage_roofline(cfg, stage, peaks)
    del p, x, y, ws
    torch.cuda.empty_cache()
    return out


def bench_all(moe, peaks, args) -> list:
    res = []
    for name in ("tiny_f32", "mixtral_prefill", "dsv3_decode", "dsv3_prefill_zipf",
                 *[f"dsv3_sweep_T{t}" for t in mi.SWEEP_T], "dsv3_decode_sigmoid",
                 "dsv3_decode_fp8", "dsv3_sweep_fp8_T64", "dsv3_sweep_fp8_T512",
                 "mixtral_prefill_fp8", "dsv3_decode_fp8b", "dsv3_sweep_fp8b_T512",
                 "mixtral_prefill_fp8b", "dsv3_decode_w8a8", "dsv3_sweep_w8a8_T512",
                 "dsv3_sweep_w8a8_T4096", "mixtral_prefill_w8a8", "dsv3_prefill_zipf_w8a8",
                 "dsv3_decode_w8a8b", "mixtral_prefill_w8a8b", "dsv3_prefill_zipf_w8a8b"):
        cfg = mi.CONFIGS[name]
        res.append(bench_workload(moe, cfg, peaks, steps=max(10, args.steps),
                                  graph=cfg.T <= 64))
    return res


# --------------------------------------------------------------------------- reduced expert pools

def pool_counts(moe, cfg, n_pool: int) -> list:
    """Per-expert row counts of a reduced pool with the workload's routing
    profile: the workload's per-expert counts (its own routing on the GPU),
    sorted, taken at every (E / n_pool)-th rank -- the hottest expert, and so on
    down to the coldest kept one."""
    import torch
    p = mi.make_weights(cfg, "cuda", only={"w_g"})
    x = mi.make_x(cfg, "cuda")
    bias = mi.make_bias(cfg, "cuda")
    s = moe.make_shape(cfg.T, cfg.d, cfg.E, cfg.K, cfg.I, cfg.Is, cfg.dtype, cfg.router)
    ws = moe.alloc_workspace(s)
    idx = torch.empty((cfg.T, cfg.K), dtype=torch.int32, device="cuda")
    w = torch.empty((cfg.T, cfg.K), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    moe.moe_route(s, x, p["w_g"], bias, None, None, idx, w, ws)
    counts = torch.bincount(idx.flatten().long(), minlength=cfg.E).cpu()
    ranked = torch.sort(counts, descending=True).values.tolist()
    step = max(1, cfg.E // n_pool)
    del p, x, ws, idx, w
    torch.cuda.empty_cache()
    return [int(c) for c in ranked[::step][:n_pool]]


def run_stage_pool(args):
    """The expert-FFN stage alone (moe_expert_ffn) on a reduced pool of
    args.stage_pool experts with the workload's routing profile (pool_counts):
    a few GB on the device, for counter captures of the stage's GEMMs."""
    import torch
    import sparse_expert_ffn_moe_gb300 as moe
    torch.cuda.set_device(0)
    cfg = mi.CONFIGS[args.workload]
    counts = pool_counts(moe, cfg, args.stage_pool)
    E, rows = len(counts), sum(counts)
    pcfg = mi.LayerConfig(f"{cfg.name}_pool{E}", T=rows, d=cfg.d, E=E, K=1, I=cfg.I,
                          dtype=cfg.dtype, weights=cfg.weights, acts=cfg.acts, seed=cfg.seed)
    p = mi.make_weights(pcfg, "cuda", only={"w_gate", "w_up", "w_down", "s_gate", "s_up",
                                            "s_down"})
    fp8 = moe.make_fp8_experts(p) if mi.is_fp8(cfg) else None
    ffn8 = fp8_calls(moe, cfg)[1]
    x_perm = mi.normal((rows, cfg.d), 1.0, cfg.dtype, "cuda", cfg.seed, "x_perm")
    y_perm = torch.empty_like(x_perm)
    offsets = torch.tensor([0] + list(np.cumsum(counts)), dtype=torch.int32, device="cuda")
    s = moe.make_shape(rows, cfg.d, E, 1, cfg.I, 0, cfg.dtype)
    ws = moe.alloc_workspace(s)
    st = torch.cuda.Stream()
    torch.cuda.synchronize()

    def run():
        if fp8 is not None:
            ffn8(s, x_perm, offsets, fp8, y_perm, ws, stream=st)
        else:
            moe.moe_expert_ffn(s, x_perm, offsets, p["w_gate"], p["w_up"], p["w_down"], y_perm,
                               ws, stream=st)
    for _ in range(max(3, args.warmup)):
        run()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    for _ in range(args.steps):
        run()
    e1.record(st)
    torch.cuda.synchronize()
    if moe.moe_get_device_error(ws):
        raise RuntimeError("device error in the expert stage")
    ms = e0.elapsed_time(e1) / args.steps
    flops = 6 * rows * cfg.d * cfg.I
    wbytes = E * expert_bytes(cfg, cfg.I)
    print(json.dumps({"workload": pcfg.name, "counts": counts, "rows": rows, "ms_per_stage": ms,
                      "tflops": flops / ms / 1e9, "weight_bytes": wbytes,
                      "alg_bytes": wbytes + 2 * elem_bytes(cfg) * rows * cfg.d,
                      "source_sha256": source_sha256()}), flush=True)


# --------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle timed on the host cores, same workload and metric."""
    ws_n, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    cfg = mi.CONFIGS[args.workload]
    import oracle
    # the seeded inputs are drawn where it is quick (22.6 GB of weights at the DeepSeek-V3
    # shape), then copied to host memory; the timed oracle runs on the host cores only
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    p = mi.make_weights(cfg, dev)
    x = mi.make_x(cfg, dev)
    bias = mi.make_bias(cfg, dev)
    hp = {k: mi.to_host_array(v) for k, v in p.items()}
    xh = mi.to_host_array(x)
    bh = None if bias is None else bias.double().cpu().numpy()
    del p, x
    if dev == "cuda":
        torch.cuda.empty_cache()
    threads = oracle.default_threads()
    # per-step sample sized so that warm-up + steps end within a few minutes
    per_step = max(threads, 16)
    times = []
    for i in range(args.warmup + args.steps):
        tokens = mi.sample_tokens(cfg.T, per_step, seed=cfg.seed, name=f"ref_step/{i}").numpy()
        t0 = time.perf_counter()
        oracle_tokens(cfg, tokens, xh, hp, bh)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    ms = 1e3 * sum(times) / len(times)
    value = per_step / (ms / 1e3)
    sample = (f"{per_step} seeded tokens of {cfg.name} per step, full layer per token in fp64 "
              f"(router, K routed experts, shared expert)")
    print(json.dumps({
        "impl": "reference", "metric": "MoE layer tokens/s", "value": value, "unit": "tokens/s",
        "n_gpus": ws_n, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": cfg.name, "T": cfg.T, "d": cfg.d, "E": cfg.E,
                                        "K": cfg.K, "inter": cfg.I, "inter_shared": cfg.Is},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(mi.CONFIGS))
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--all", action="store_true", help="also time every workload")
    ap.add_argument("--sweep-T", default=SWEEP_T, help="comma-separated token counts: time the "
                    "DeepSeek-V3 shape at each T (one JSON object per T under 'sweep'); "
                    "empty to skip")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the Mixtral prefill block")
    ap.add_argument("--stage-pool", type=int, default=0,
                    help="time only the expert stage on a pool of this many experts with the "
                         "workload's routing profile (for counter captures)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.stage_pool:
        run_stage_pool(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
