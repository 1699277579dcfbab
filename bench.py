"""Benchmark: GPT pre-LN layer forward + backward on GB300.

Default workload: one layer of the 96-layer GPT (b1 s4096 h8192, 64 heads of
128, ffn 32768) run as 8 tensor-parallel partitions on one GPU.  One step =
mc_layer_forward + mc_layer_backward over one batch (every kernel of the hot
path).  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload c1|c2|c3|c4|c4shard|c5] [--stage NAME]

--impl reference times the fp64 CPU oracle on this host's cores, on a bounded
sample of the same workload (a prefix of the sequence), with the same metric.
--stage NAME times one kernel alone (for profiling); its line is a
per-kernel measurement, not the step metric.
Under torchrun each rank runs an independent replica (weak scaling).
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

METRIC = "layer fwd+bwd tokens/s; BF16 TFLOP/s as % of GB300 dense tensor peak"
NOMINAL_BF16_TFLOPS = 2250.0

WORKLOADS = {
    "c1": dict(micro_batch=1, seq_len=128, hidden=768, heads=12, ffn_hidden=3072, tp_parts=2, head_dim=0),
    "c2": dict(micro_batch=4, seq_len=512, hidden=768, heads=12, ffn_hidden=3072, tp_parts=2, head_dim=0),
    "c3": dict(micro_batch=8, seq_len=1024, hidden=2048, heads=16, ffn_hidden=8192, tp_parts=4, head_dim=0),
    "c4": dict(micro_batch=1, seq_len=4096, hidden=8192, heads=64, ffn_hidden=32768, tp_parts=8, head_dim=0),
    "c4shard": dict(micro_batch=1, seq_len=4096, hidden=8192, heads=8, ffn_hidden=4096, tp_parts=1, head_dim=128),
    "c5": dict(micro_batch=1, seq_len=32768, hidden=4096, heads=32, ffn_hidden=16384, tp_parts=1, head_dim=0),
}
WORKLOAD_NAMES = {
    "c1": "gpt-layer b1 s128 h768 H12 d64 f3072 tp2",
    "c2": "gpt-layer b4 s512 h768 H12 d64 f3072 tp2",
    "c3": "gpt-layer b8 s1024 h2048 H16 d128 f8192 tp4",
    "c4": "gpt-layer b1 s4096 h8192 H64 d128 f32768 tp8 (one layer of the 96-layer GPT)",
    "c4shard": "gpt-layer shard b1 s4096 h8192 H8 d128 a1024 f4096 tp1 (one TP=8 rank alone)",
    "c5": "gpt-layer b1 s32768 h4096 H32 d128 f16384 tp1 (long sequence)",
}

# Kernels launched per step by mc_layer_forward + mc_layer_backward:
# forward 7 (LN, QKV, attention, out-proj, LN, fc1, fc2); backward 21
# (colsum x2 launches x3 sums, LN-backward x2 launches x2, 6 GEMMs,
# attention backward 3).
LAUNCHES_PER_STEP = 7 + 21


def launches_per_step(t_shards: int, recompute: bool, fp8: bool = False) -> int:
    """Kernel launches of one layer step; in sequence-parallel mode the
    per-token kernels and the reduce-scattered GEMMs run once per shard
    (forward 4t + 3, backward 8t + 13; t = 1 gives the 7 + 21 above).  The
    FP8 mode adds 3 launches per quantised tensor (amax, scale, cast): 8 in
    the forward (the 4 weights, ln1, O, ln2, g), 4 in the backward (dy, dhp,
    dx1, dQ|dK|dV)."""
    fwd = 4 * t_shards + 3 + (24 if fp8 else 0)
    return fwd + 8 * t_shards + 13 + (12 if fp8 else 0) + (fwd if recompute else 0)


def dims(w):
    d = w["head_dim"] or w["hidden"] // w["heads"]
    return dict(b=w["micro_batch"], s=w["seq_len"], T=w["micro_batch"] * w["seq_len"],
                h=w["hidden"], H=w["heads"], d=d, a=w["heads"] * d, f=w["ffn_hidden"],
                t=w["tp_parts"])


def layer_flops(w) -> float:
    """Algorithmic fwd+bwd flops: 3 x [2T(3ha + ah + 2hf) + 2 a b s (s+1)]."""
    D = dims(w)
    fwd = 2 * D["T"] * (3 * D["h"] * D["a"] + D["a"] * D["h"] + 2 * D["h"] * D["f"]) \
        + 2 * D["a"] * D["b"] * D["s"] * (D["s"] + 1)
    return 3.0 * fwd


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return {}


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers
def make_inputs(w, seed=0):
    from layer_inputs import LayerShape, make_layer_inputs
    shape = LayerShape(**w)
    return make_layer_inputs(shape, seed=seed)


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(world: int, tokens_per_replica: int, steps: int, max_ms: float) -> float:
    """Whole-job tokens/s of `world` independent replicas, timed by the
    slowest rank."""
    return world * tokens_per_replica * steps / (max_ms / 1e3)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- oracle timing
def prepare_oracle(w, prefix_tokens: int):
    """Inputs of a bounded sample of the workload for the fp64 oracle: the
    first `prefix_tokens` tokens of the sequence (micro-batch 1), full
    weights."""
    from layer_inputs import LayerShape, make_layer_inputs

    sample = dict(w)
    sample["micro_batch"] = 1
    sample["seq_len"] = min(prefix_tokens, w["seq_len"])
    shape = LayerShape(**sample)
    inp = make_layer_inputs(shape, seed=0)
    return shape, inp.params_f64(), inp.f64("x"), inp.f64("dy")


def oracle_step(prepared) -> float:
    """One fp64 oracle forward + backward; returns its wall time in seconds."""
    import oracle.layer as O

    shape, P, x, dy = prepared
    t0 = time.perf_counter()
    O.layer_forward_backward(shape, P, x, dy)
    return time.perf_counter() - t0


def record_card(device=None) -> dict:
    """Identity of the run, for the record: GPU, SM count, driver, CUDA and
    torch versions, host CPU model and thread count."""
    card = {"host_cpu": None, "host_threads": os.cpu_count()}
    try:
        import torch
        card["torch"] = torch.__version__
        card["cuda_runtime"] = torch.version.cuda
        if device is not None and torch.cuda.is_available():
            prop = torch.cuda.get_device_properties(device)
            card["gpu"] = prop.name
            card["sm_count"] = prop.multi_processor_count
            card["gpu_memory_gib"] = round(prop.total_memory / 2 ** 30, 1)
    except Exception:
        pass
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader"],
                             capture_output=True, text=True, timeout=20).stdout.split()
        card["driver"] = out[0] if out else None
    except (OSError, subprocess.TimeoutExpired):
        card["driver"] = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=20).stdout
        for ln in out.splitlines():
            if ln.lower().startswith("model name"):
                card["host_cpu"] = ln.split(":", 1)[1].strip()
                break
            if ln.lower().startswith("vendor id") and card["host_cpu"] is None:
                card["host_cpu"] = ln.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    return card


def oracle_extrapolated(w, prefixes=(64, 256), head_len=2048) -> dict:
    """Oracle tokens/s at the workload's full sequence length, extrapolated
    (not measured).  One fp64 layer step is timed on two prefixes of the
    sequence and modelled as c + alpha n + H beta n^2: c the per-step cost of
    the weights and their gradients, alpha the per-token products, beta the
    causal attention of one head, timed on its own (the oracle's attention
    forward + backward at `head_len` tokens).  The model is evaluated at the
    workload's micro_batch and seq_len."""
    import numpy as np

    import oracle.layer as O
    D = dims(w)
    n0 = min(head_len, w["seq_len"])
    rng = np.random.default_rng(0)
    q, k, v, do = (rng.standard_normal((n0, D["d"])) for _ in range(4))
    t0 = time.perf_counter()
    o, lse = O.causal_attention_forward(q, k, v)
    O.causal_attention_backward(q, k, v, o, lse, do)
    beta = (time.perf_counter() - t0) / (n0 * n0)
    ns, ts = [], []
    for n in prefixes:
        prepared = prepare_oracle(w, n)
        ns.append(prepared[0].seq_len)
        ts.append(oracle_step(prepared))
        del prepared
    if len(set(ns)) < 2:
        return {"value": None, "note": "sequence too short to extrapolate"}
    lin = [t - D["H"] * beta * n * n for n, t in zip(ns, ts)]
    alpha = max((lin[1] - lin[0]) / (ns[1] - ns[0]), 0.0)
    c = max(lin[0] - alpha * ns[0], 0.0)
    s_len, b = w["seq_len"], w["micro_batch"]
    t_full = c + alpha * b * s_len + b * D["H"] * beta * s_len * s_len
    return {"value": b * s_len / t_full, "unit": "tokens/s",
            "kind": "extrapolated, not measured",
            "prefix_tokens": ns, "prefix_seconds": ts,
            "model_seconds": {"c": c, "per_token": alpha, "per_head_token_pair": beta,
                              "attention_head_len_timed": n0},
            "seconds_per_step_at_config": t_full}


def oracle_threads() -> int:
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(var):
            return int(os.environ[var])
    return os.cpu_count() or 1


# ---------------------------------------------------------------- arms
def run_reference(args, world, rank):
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    prepared = prepare_oracle(w, args.ref_prefix)
    toks = prepared[0].seq_len
    for _ in range(args.warmup):
        oracle_step(prepared)
    per = [oracle_step(prepared) for _ in range(args.steps)]
    sec = sum(per) / len(per)
    value = toks / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAMES[args.workload], **w},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle_threads(),
                         "kind": "oracle",
                         "sample": f"first {toks} tokens of the sequence (micro-batch 1), full "
                                   f"weights, fp64 forward+backward per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "record_card": record_card(None),
    }
    line["cpu_baseline"]["cpu"] = line["record_card"].get("host_cpu")
    print(json.dumps(line), flush=True)


def stage_launcher(name, w, device, params=None, cp_parts=4):
    """One kernel of the step with the workload's shapes, inputs resident in
    HBM.  Returns (launch function, algorithmic flops or bytes per launch,
    unit, description)."""
    import torch

    from megatron_transformer_layer_gb300 import _lib as L
    D = dims(w)
    T, h, f, a, H, d, b, s = D["T"], D["h"], D["f"], D["a"], D["H"], D["d"], D["b"], D["s"]
    gen = torch.Generator(device=device).manual_seed(0)
    st = torch.cuda.current_stream(device)

    def rnd(*shape, scale=1.0, dtype=torch.bfloat16):
        return (torch.randn(*shape, device=device, generator=gen) * scale).to(dtype)

    if name == "gemm_fc1":
        A, B = rnd(T, h), (params["w_fc1"] if params else rnd(f, h, scale=0.02))
        bias = params["b_fc1"] if params else torch.zeros(f, device=device, dtype=torch.bfloat16)
        out, hp = rnd(T, f), rnd(T, f)

        def launch():
            rc = L.mc_gemm(T, f, h, A, h, 0, B, h, 0, out, f, L.MC_EPI_BIAS_GELU, bias=bias,
                           aux=hp, ldaux=f, stream=st)
            assert rc == 0, L.mc_strerror(rc)
        return launch, 2.0 * T * h * f, "flop", "gemm_tcgen05 fc1 forward (bias+GeLU epilogue)"
    if name == "gemm_fc1_fp8":
        # fc1 with E4M3 operands (per-tensor scales), quantised once outside the timing
        A32, B32 = rnd(T, h, dtype=torch.float32), rnd(f, h, scale=0.02, dtype=torch.float32)
        qa = torch.empty(T * h, dtype=torch.uint8, device=device)
        qb = torch.empty(f * h, dtype=torch.uint8, device=device)
        sa, sb = (torch.empty(1, device=device) for _ in range(2))
        scratch = torch.empty(L.mc_fp8_scratch_floats(), device=device)
        assert L.mc_fp8_quantize(A32, qa, sa, scratch, L.FP8_E4M3, stream=st) == 0
        assert L.mc_fp8_quantize(B32, qb, sb, scratch, L.FP8_E4M3, stream=st) == 0
        bias = torch.zeros(f, device=device, dtype=torch.bfloat16)
        out, hp = rnd(T, f), rnd(T, f)

        def launch():
            rc = L.mc_gemm_fp8(T, f, h, qa, h, L.FP8_E4M3, qb, h, L.FP8_E4M3, sa, sb, out, f,
                               L.MC_EPI_BIAS_GELU, bias=bias, aux=hp, ldaux=f, stream=st)
            assert rc == 0, L.mc_strerror(rc)
        return launch, 2.0 * T * h * f, "flop", "gemm_tcgen05 fc1 forward, E4M3 operands (kind::f8f6f4)"
    if name == "gemm_wgrad":
        A, B = rnd(T, f), rnd(T, h)           # dhp [T, f], ln2 [T, h]
        out = torch.empty(f, h, device=device, dtype=torch.float32)

        def launch():
            rc = L.mc_gemm(f, h, T, A, f, 1, B, h, 1, out, h, L.MC_EPI_STORE_F32, stream=st)
            assert rc == 0, L.mc_strerror(rc)
        return launch, 2.0 * T * h * f, "flop", "gemm_tcgen05 wgrad dW1 = dhp^T ln2 (MN-major A and B)"
    if name in ("attn_fwd", "attn_bwd", "attn_bwd_recompute"):
        qkv, o = rnd(T, 3 * a), rnd(T, a)
        lse = torch.empty(b * H * s, device=device, dtype=torch.float32)
        dout, dqkv = rnd(T, a), rnd(T, 3 * a)
        delta = torch.empty(b * H * s, device=device, dtype=torch.float32)
        assert L.mc_attention_forward(qkv, o, lse, b, s, H, d, stream=st) == 0
        causal = 2.0 * a * b * s * (s + 1)
        if name == "attn_fwd":
            def launch():
                assert L.mc_attention_forward(qkv, o, lse, b, s, H, d, stream=st) == 0
            return launch, causal, "flop", "causal attention forward"

        if name == "attn_bwd_recompute":
            def launch():
                assert L.mc_attention_backward(qkv, o, lse, dout, dqkv, delta, b, s, H, d,
                                               stream=st) == 0
            return launch, 2.0 * causal, "flop", \
                "causal attention backward (pre + dkdv + dq forming S, dP again)"
        nbytes = L.mc_attention_backward_ws_bytes(b, s, H, d)
        ds = torch.empty(nbytes, device=device, dtype=torch.uint8)

        def launch():
            assert L.mc_attention_backward_ws(qkv, o, lse, dout, dqkv, delta, b, s, H, d, ds,
                                              nbytes, stream=st) == 0
        return launch, 2.0 * causal, "flop", \
            "causal attention backward (pre + dkdv writing dS + dQ = dS K)"
    if name in ("attn_fwd_cp", "attn_bwd_cp"):
        cp = cp_parts
        qkv, o = rnd(T, 3 * a), rnd(T, a)
        lse = torch.empty(b * H * s, device=device, dtype=torch.float32)
        dout, dqkv = rnd(T, a), rnd(T, 3 * a)
        delta = torch.empty(b * H * s, device=device, dtype=torch.float32)
        nbytes = L.mc_attention_cp_workspace_bytes(b, s, H, d, cp)
        if nbytes == 0:
            raise SystemExit(f"seq_len {s} does not split into {2 * cp} whole 128-token chunks")
        ws = torch.empty(nbytes, device=device, dtype=torch.uint8)
        assert L.mc_attention_forward_cp(qkv, o, lse, b, s, H, d, cp, ws, nbytes, stream=st) == 0
        causal = 2.0 * a * b * s * (s + 1)
        if name == "attn_fwd_cp":
            def launch():
                assert L.mc_attention_forward_cp(qkv, o, lse, b, s, H, d, cp, ws, nbytes,
                                                 stream=st) == 0
            return launch, causal, "flop", f"context-parallel causal attention forward, cp {cp}"

        def launch():
            assert L.mc_attention_backward_cp(qkv, o, lse, dout, dqkv, delta, b, s, H, d, cp, ws,
                                              nbytes, stream=st) == 0
        return launch, 2.0 * causal, "flop", f"context-parallel causal attention backward, cp {cp}"
    if name == "ln_bwd":
        dln, x, resid = (torch.randn(T, h, device=device, generator=gen) for _ in range(3))
        mean = torch.zeros(T, device=device)
        rstd = torch.ones(T, device=device)
        gamma = torch.ones(h, device=device, dtype=torch.bfloat16)
        dx = torch.empty(T, h, device=device)
        dx16 = torch.empty(T, h, device=device, dtype=torch.bfloat16)
        dg, db, dc = (torch.empty(h, device=device) for _ in range(3))
        part = torch.empty(L.mc_layernorm_backward_scratch_floats(T, h), device=device)

        def launch():
            assert L.mc_layernorm_backward(dln, x, mean, rstd, gamma, resid, dx, dx16, dg, db, dc,
                                           0, part, T, h, stream=st) == 0
        # algorithmic bytes: read dln, x, resid (fp32), write dx fp32 + bf16
        return launch, float(T * h * (4 * 3 + 4 + 2)), "byte", "LayerNorm backward (+bf16 copy, colsums)"
    raise ValueError(name)


def time_launches(launch, device, steps, warmup):
    """Average ms per launch: CUDA events on the launching stream."""
    import torch
    st = torch.cuda.current_stream(device)
    for _ in range(warmup):
        launch()
    torch.cuda.synchronize(device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * steps)]
    for i in range(steps):
        ev[2 * i].record(st)
        launch()
        ev[2 * i + 1].record(st)
    torch.cuda.synchronize(device)
    ms = [ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(steps)]
    return sum(ms) / len(ms)


def run_stage(args, w, device):
    """Times one kernel of the step alone (used for profiling)."""
    launch, work, unit, desc = stage_launcher(args.stage, w, device, cp_parts=args.cp)
    ms = time_launches(launch, device, args.steps, max(args.warmup, 1))
    rate = work / (ms / 1e3)
    line = {"stage": args.stage, "kernel": desc, "workload": WORKLOAD_NAMES[args.workload],
            "ms_per_launch": ms}
    if unit == "flop":
        line["tflops"] = rate / 1e12
    else:
        line["gbs"] = rate / 1e9
    print(json.dumps(line), flush=True)


def sub_record(name, device, world, steps, warmup, peak_sustained, fp8=False, attention=True):
    """One more workload timed in the same run, device-resident: its step
    (forward + backward through the C ABI, CUDA events on the launching
    stream) and, with `attention`, its attention kernels alone.  `fp8`: the
    layer's GEMMs on 8-bit operands (MC_FP8_HYBRID)."""
    import numpy as np
    import torch

    from layer_inputs import LayerShape, make_layer_inputs
    from megatron_transformer_layer_gb300.layer import TransformerLayer, bf16_tensor
    w = WORKLOADS[name]
    D = dims(w)
    inp = make_layer_inputs(LayerShape(**w), seed=0)
    params = {k: bf16_tensor(v, device) for k, v in inp.params.items()}
    layer = TransformerLayer(**w, params=params, device=device, fp8=fp8)
    x = torch.from_numpy(inp.f64("x").reshape(-1, D["h"]).astype(np.float32)).to(device)
    dy = torch.from_numpy(inp.f64("dy").reshape(-1, D["h"]).astype(np.float32)).to(device)
    del inp
    y, dx = torch.empty_like(x), torch.empty_like(x)

    def step():
        layer.forward(x, y)
        layer.backward(dy, dx, x=x)

    ms = time_launches(step, device, steps, max(warmup, 3))
    ms = max_over_ranks(ms, world, device)
    if layer.device_status() != 0:
        raise SystemExit(f"{name}: device status {layer.device_status()}")
    flops = layer_flops(w)
    out = {"workload": WORKLOAD_NAMES[name], "steps": steps, "ms_per_step": ms,
           "tokens_per_s": world * D["T"] / (ms / 1e3),
           "tflops": flops / (ms / 1e3) / 1e12,
           "gemm_operands": "fp8 (E4M3 forward, E5M2 gradients)" if fp8 else "bf16"}
    if not fp8:
        out["frac_of_sustained"] = flops / (ms / 1e3) / 1e12 / peak_sustained
    del layer, params, x, dy, y, dx
    torch.cuda.empty_cache()
    for stage in (("attn_fwd", "attn_bwd") if attention else ()):
        launch, work, _, _ = stage_launcher(stage, w, device)
        sms = time_launches(launch, device, max(3, steps), 2)
        out[f"{stage}_ms"] = sms
        out[f"{stage}_tflops"] = work / (sms / 1e3) / 1e12
    torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    from megatron_transformer_layer_gb300 import _lib as L
    from megatron_transformer_layer_gb300.layer import TransformerLayer, bf16_tensor

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU for --impl ours")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = WORKLOADS[args.workload]
    if args.stage:
        run_stage(args, w, device)
        return
    D = dims(w)
    from layer_inputs import LayerShape, make_layer_inputs
    n_layers = args.layers
    layers, params, shared_ws = [], None, None
    for li in range(n_layers):
        inp_l = make_layer_inputs(LayerShape(**w), seed=0, layer=li)
        p_l = {k: bf16_tensor(v, device) for k, v in inp_l.params.items()}
        layers.append(TransformerLayer(**w, params=p_l, device=device, recompute=args.recompute,
                                       workspace=shared_ws, sequence_parallel=args.sp,
                                       fp8=args.fp8))
        if args.recompute:
            shared_ws = layers[-1].ws  # recomputation: one workspace for the whole stack
        if li == 0:
            inp, params = inp_l, p_l
    layer = layers[0]
    x = torch.from_numpy(inp.f64("x").reshape(-1, D["h"]).astype(np.float32)).to(device)
    dy = torch.from_numpy(inp.f64("dy").reshape(-1, D["h"]).astype(np.float32)).to(device)
    acts = [x] + [torch.empty_like(x) for _ in range(n_layers)]
    grads = [torch.empty_like(x) for _ in range(n_layers)]
    y, dx = acts[-1], grads[0]
    st = torch.cuda.current_stream(device)

    def step():
        # forward through the stack, then backward in reverse (fp32 residual
        # stream between layers)
        for li in range(n_layers):
            layers[li].forward(acts[li], acts[li + 1])
        g = dy
        for li in reversed(range(n_layers)):
            layers[li].backward(g, grads[li], x=acts[li])
            g = grads[li]

    for _ in range(max(args.warmup, 1)):
        step()
    torch.cuda.synchronize(device)
    if args.graph:
        # Capture one whole step (every launch of the stack's forward and
        # backward) and replay it: for launch-bound small shapes.  The first
        # calls above did the one-time set-up, and the step allocates nothing.
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize(device)
        eager_step = step

        def step():  # noqa: F811
            graph.replay()

        step()
        torch.cuda.synchronize(device)
        del eager_step
    status = max(abs(l.device_status()) for l in layers)
    if status != 0:
        raise SystemExit(f"device status {status}: {L.mc_strerror(status)}")

    # ---- device-resident timing (inputs already in HBM)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    step_ev = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    barrier(world)
    torch.cuda.synchronize(device)
    with ClockSampler(device.index if device.index is not None else 0) as clk:
        e0.record(st)
        step_ev[0].record(st)
        for i in range(args.steps):
            step()
            step_ev[i + 1].record(st)
        e1.record(st)
        torch.cuda.synchronize(device)
    barrier(world)
    ms_total = e0.elapsed_time(e1)
    per_step = [step_ev[i].elapsed_time(step_ev[i + 1]) for i in range(args.steps)]
    ms_total = max_over_ranks(ms_total, world, device)
    ms_step = ms_total / args.steps
    tokens = D["T"]
    value = replica_throughput(world, tokens, args.steps, ms_total)
    flops = layer_flops(w) * n_layers  # algorithmic: the recomputed forward is not counted
    tflops = flops / (ms_step / 1e3) / 1e12
    peaks = measured_peaks()
    peak = peaks.get("bf16_tflops_sustained") or 1710.0
    peak_burst = peaks.get("bf16_tflops") or 1900.0

    # ---- end to end through the public API with host buffers.  Every step
    # copies its inputs (x, dy) from pinned host memory and its results (y,
    # dx) back, all inside the timed region.  Pipelined as a training input
    # pipeline would be: step i+1's inputs go up on one copy stream and step
    # i's results come down on another while step i computes (device buffers
    # double-buffered, ordered by events).  The serial form (copy in, step,
    # copy out, one stream) is measured too.
    x_h = x.cpu().pin_memory()
    dy_h = dy.cpu().pin_memory()
    y_h = [torch.empty_like(x_h).pin_memory() for _ in range(2)]
    dx_h = [torch.empty_like(x_h).pin_memory() for _ in range(2)]
    x_d = [torch.empty_like(x) for _ in range(2)]
    dy_d = [torch.empty_like(dy) for _ in range(2)]
    y_d = [torch.empty_like(x) for _ in range(2)]
    dx_d = [torch.empty_like(x) for _ in range(2)]
    h2d_st, d2h_st = torch.cuda.Stream(device), torch.cuda.Stream(device)

    def compute(k):
        acts[0], acts[-1] = x_d[k], y_d[k]
        for li in range(n_layers):
            layers[li].forward(acts[li], acts[li + 1])
        g = dy_d[k]
        for li in reversed(range(n_layers)):
            out = dx_d[k] if li == 0 else grads[li]
            layers[li].backward(g, out, x=acts[li])
            g = out

    def e2e_serial(n):
        for _ in range(n):
            x_d[0].copy_(x_h, non_blocking=True)
            dy_d[0].copy_(dy_h, non_blocking=True)
            compute(0)
            y_h[0].copy_(y_d[0], non_blocking=True)
            dx_h[0].copy_(dx_d[0], non_blocking=True)

    def e2e_pipelined(n, start):
        ev = lambda: torch.cuda.Event()  # noqa: E731
        in_ready, in_free = [ev(), ev()], [ev(), ev()]
        out_ready, out_free = [ev(), ev()], [ev(), ev()]
        h2d_st.wait_stream(st)
        d2h_st.wait_stream(st)
        start.record(h2d_st)

        def upload(k):
            with torch.cuda.stream(h2d_st):
                x_d[k].copy_(x_h, non_blocking=True)
                dy_d[k].copy_(dy_h, non_blocking=True)
                in_ready[k].record(h2d_st)

        upload(0)
        for i in range(n):
            k = i & 1
            st.wait_event(in_ready[k])
            if i >= 2:
                st.wait_event(out_free[k])  # step i-2's results have been read out
            compute(k)
            out_ready[k].record(st)
            in_free[k].record(st)
            if i + 1 < n:
                if i >= 1:
                    h2d_st.wait_event(in_free[k ^ 1])  # step i-1 is done with its inputs
                upload(k ^ 1)
            with torch.cuda.stream(d2h_st):
                d2h_st.wait_event(out_ready[k])
                y_h[k].copy_(y_d[k], non_blocking=True)
                dx_h[k].copy_(dx_d[k], non_blocking=True)
                out_free[k].record(d2h_st)
        st.wait_stream(d2h_st)
        st.wait_stream(h2d_st)

    e2e_serial(2)
    e2e_pipelined(2, torch.cuda.Event(enable_timing=True))
    torch.cuda.synchronize(device)
    barrier(world)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_pipelined(args.steps, a0)
    a1.record(st)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(a0.elapsed_time(a1), world, device)
    e2e_value = replica_throughput(world, tokens, args.steps, e2e_ms)
    barrier(world)
    a0.record(st)
    e2e_serial(args.steps)
    a1.record(st)
    torch.cuda.synchronize(device)
    serial_ms = max_over_ranks(a0.elapsed_time(a1), world, device)
    e2e_serial_value = replica_throughput(world, tokens, args.steps, serial_ms)
    if not (torch.equal(y_h[0], y_h[1]) and torch.equal(dx_h[0], dx_h[1])):
        raise SystemExit("end-to-end steps disagree")
    h2d = 2 * x.numel() * 4
    d2h = 2 * x.numel() * 4

    # ---- dominant kernel: the tcgen05 GEMM variant with the largest share of
    # the step (the wgrad product, dW1 = dhp^T ln2), timed alone on this stream
    launch, gemm_flops, _, desc = stage_launcher("gemm_wgrad", w, device)
    gemm = time_launches(launch, device, max(5, min(args.steps, 20)), 2)
    achieved = gemm_flops / (gemm / 1e3) / 1e12
    roofline = {"bound": "tensor", "kernel": desc, "achieved": achieved, "peak": peak_burst,
                "unit": "TFLOP/s", "frac": achieved / peak_burst,
                "peak_kind": "bf16 burst, of measured (kernel timed alone)",
                "flops_per_launch": gemm_flops, "ms_per_launch": gemm,
                "traffic": TRAFFIC.get(args.workload)}
    launch_fc1, fc1_flops, _, _ = stage_launcher("gemm_fc1", w, device, params)
    fc1_ms = time_launches(launch_fc1, device, max(5, min(args.steps, 20)), 2)
    roofline["also_fc1_forward_tflops"] = fc1_flops / (fc1_ms / 1e3) / 1e12

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "ms_per_step_p50": statistics.median(per_step),
        "ms_per_step_p95": sorted(per_step)[max(0, int(round(0.95 * len(per_step))) - 1)],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8-hybrid" if args.fp8 else "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAMES[args.workload]
                   + (f", stack of {n_layers} layers" if n_layers > 1 else ""), **w,
                   "layers": n_layers,
                   "activation_recompute": bool(args.recompute),
                   "sequence_parallel": bool(args.sp),
                   "gemm_operands": "fp8 (E4M3 forward, E5M2 gradients)" if args.fp8 else "bf16",
                   "cuda_graph": bool(args.graph),
                   "l2": "inputs larger than L2 (1.6 GB of bf16 weights plus activations read per step)"
                   if args.workload == "c4" else "working set vs L2 not checked",
                   "parallelism": f"tp{w['tp_parts']} virtual partitions on one GPU; "
                                  f"{'replicas' if world > 1 else 'single GPU'}"},
        "tflops": tflops,
        "pct_of_peak": {"measured_sustained": tflops / peak, "nominal": tflops / NOMINAL_BF16_TFLOPS},
        "clocks": clk.summary(),
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "pipeline": "step i+1's inputs uploaded and step i's results read back on two "
                            "copy streams while step i computes (double-buffered)",
                "serial_value": e2e_serial_value},
        "gpu_launches": launches_per_step(w["tp_parts"] if args.sp else 1, args.recompute,
                                          args.fp8) * n_layers * args.steps,
        "memory": {"saved_bytes_per_layer": layer.saved_bytes,
                   "workspace_bytes_per_layer": layer.ws_bytes,
                   "workspace_shared_by_stack": bool(args.recompute)},
        "roofline": roofline,
    }
    line["record_card"] = record_card(device)
    if args.workload == "c4" and n_layers == 1 and not args.no_c5 and not args.recompute \
            and not args.graph and not args.sp and not args.fp8:
        # the long-sequence configuration (attention 40% of its flops), timed in
        # the same run; all ranks run it so that max-over-ranks still holds
        del layers, layer, acts, grads, x_d, dy_d, y_d, dx_d
        torch.cuda.empty_cache()
        line["c5"] = sub_record("c5", device, world, min(args.steps, 10), args.warmup, peak)
        # the same layer with its GEMMs on 8-bit operands, for comparison
        # (not the headline: the headline is the bf16 path)
        line["c4_fp8"] = sub_record("c4", device, world, min(args.steps, 20), args.warmup, peak,
                                    fp8=True, attention=False)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and n_layers == 1:
        prepared = prepare_oracle(w, args.ref_prefix)
        toks = prepared[0].seq_len
        sec = oracle_step(prepared)
        del prepared
        line["cpu_baseline"] = {"value": toks / sec, "unit": "tokens/s", "cores": oracle_threads(),
                                "kind": "oracle",
                                "cpu": line["record_card"].get("host_cpu"),
                                "sample": f"first {toks} tokens of the sequence (micro-batch 1), "
                                          f"full weights, one fp64 forward+backward",
                                "extrapolated_to_config": oracle_extrapolated(w)}
    if rank == 0:
        print(json.dumps(line), flush=True)


# dram__bytes_read.sum + dram__bytes_write.sum per launch of the timed wgrad
# GEMM, from one ncu capture of the current kernel build (c4 shapes); None
# for workloads not captured.
TRAFFIC = {"c4": 3.354e9}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="c4")
    ap.add_argument("--stage", choices=["gemm_fc1", "gemm_fc1_fp8", "gemm_wgrad", "attn_fwd",
                                        "attn_bwd_recompute",
                                        "attn_bwd",
                                        "attn_fwd_cp", "attn_bwd_cp", "ln_bwd"],
                    default=None)
    ap.add_argument("--ref-prefix", type=int, default=64,
                    help="tokens of the sequence the CPU oracle processes per sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-c5", action="store_true",
                    help="skip the long-sequence sub-record timed after the c4 workload")
    ap.add_argument("--tp-parts", type=int, default=0,
                    help="override the workload's tensor-parallel partition count")
    ap.add_argument("--graph", action="store_true",
                    help="capture one step in a CUDA graph and time its replays")
    ap.add_argument("--recompute", action="store_true",
                    help="activation recomputation: keep nothing between forward and backward")
    ap.add_argument("--fp8", action="store_true",
                    help="GEMMs on 8-bit operands (E4M3 forward, E5M2 gradients)")
    ap.add_argument("--sp", action="store_true",
                    help="sequence-parallel mode: per-token work launched per sequence shard")
    ap.add_argument("--layers", type=int, default=1,
                    help="time a stack of this many layers (distinct weights) per step")
    ap.add_argument("--cp", type=int, default=4,
                    help="context-parallel partitions for the attn_*_cp stages")
    args = ap.parse_args()
    if args.warmup < 3 and not args.stage and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    if args.tp_parts:
        WORKLOADS[args.workload] = dict(WORKLOADS[args.workload], tp_parts=args.tp_parts)
        WORKLOAD_NAMES[args.workload] = WORKLOAD_NAMES[args.workload].rsplit(" tp", 1)[0] \
            + f" tp{args.tp_parts}" if " tp" in WORKLOAD_NAMES[args.workload] else \
            WORKLOAD_NAMES[args.workload]
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
