#!/usr/bin/env python
"""Benchmark of one GDN-layer batched prefill on GB300.

Metric: GDN-layer prefill tokens/s on the 9B-like layer (hidden 4096, 16 q/k
heads and 32 v heads of dim 128, Q4_K weights, bf16 activations) at N = 32768
tokens, zero initial state, drawn gates (log a ~ U(-0.5, 0)).  One step is one
gdn_prefill call over the whole prompt: Q4_K decode of both weight matrices,
activation quantisation, input projection, conv, chunked delta rule, gated
norm, output projection.  Inputs (x 268 MB, workspace ~4 GB) are larger than
L2, so no flush is needed between steps.

Arms:
  default            the CUDA library (``value``: inputs resident in HBM;
                     ``e2e``: the same call fed from pinned host buffers, with
                     the host->device copy of x and the gates and the
                     device->host read of y inside the timed region);
  --impl reference   the fp64 CPU oracle on this machine's cores, each step a
                     bounded sample of the same workload.

Multi-GPU (torchrun, N ranks): the layer does not shard across GPUs here
("replicas only"): every rank prefills its own prompt on its own GPU, with no
data-path collective; timings are reduced (max) over ranks on the CPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, str(_CORES))

import numpy as np  # noqa: E402

METRIC = "GDN-layer prefill tokens/s at N=32768 (1 GB300); % int8 tensor / HBM roofline"
UNIT = "tokens/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="h4096")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-pass", type=int, default=12288, help="tokens per pass of the host-fed call")
    ap.add_argument("--seqs", type=int, default=None, help="--config decode: one batch size only (a profiling case)")
    ap.add_argument("--stage", choices=["in_proj", "delta_rule", "q6k_deq", "q4k_deq"], default=None,
                    help="time one stage kernel alone through its stage entry point (profiling case)")
    ap.add_argument("--tokens", type=int, default=None,
                    help="tokens per step (default: the workload's N); a smaller N is a profiling case, not the metric")
    return ap.parse_args()


# ------------------------------------------------------------------ distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo")
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def whole_job_rate(units_per_rank: int, world: int, ms_max: float) -> float:
    """Units per second of the whole job: every rank (an independent replica)
    processes units_per_rank per step; the step takes the slowest rank's time."""
    return units_per_rank * world / (ms_max / 1e3)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, kept with timestamps."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return []
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = time.mktime(time.strptime(f[0].split(".")[0], "%Y/%m/%d %H:%M:%S")) + float("0." + f[0].split(".")[1])
                rows.append({"t": ts, "sm": float(f[1]), "sm_max": float(f[2]), "power": f[3], "active": f[4],
                             "hw_slowdown": f[5], "hw_thermal_slowdown": f[6], "sw_thermal_slowdown": f[7],
                             "sw_power_cap": f[8]})
            except (ValueError, IndexError):
                continue
        return rows

    @staticmethod
    def summarize(rows, t0, t1):
        inside = [r for r in rows if t0 - 0.06 <= r["t"] <= t1 + 0.06] or rows
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        reasons = sorted({k for r in inside for k in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                                                        "sw_power_cap") if r[k].lower() == "active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in inside), "sm_max_mhz": max(r["sm_max"] for r in inside),
                "reasons": reasons, "samples": len(inside)}


REJECT = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}


# ------------------------------------------------------------------ roofline figures

def peaks():
    """Roofline denominators.  The projections run inside a step of a few ms
    timed over well under a second, so they take the burst tensor peak; the
    sustained one (a seconds-long loop under the power cap) is reported beside
    it.  sm_103a has no int8 tcgen05 kind: the int8 codes go through the fp16
    tensor path exactly, so the int8 roofline's denominator is the measured
    bf16 peak (fp16 runs at the bf16 rate)."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm": p["hbm_gbs"], "tensor": p["bf16_tflops"],
                "tensor_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "src": "of measured (MEASURED_PEAKS.json: hbm_gbs; bf16_tflops burst, fp16 at the bf16 rate)"}
    return {"hbm": 6800.0, "tensor": 1900.0, "tensor_sustained": 1700.0,
            "src": "of fallback (6.8 TB/s, 1.9 PFLOP/s burst bf16)"}


def stage_work(spec, n):
    """Algorithmic bytes (HBM-bound stages) or FLOPs (projections) per call: what
    the method has to move or compute, with int8 codes at one byte and bf16
    activations (the fp16 carriers of the codes and the fp32 intermediates this
    implementation keeps are its own choice and are not credited)."""
    H, hv, d = spec.hidden, spec.n_v_heads, spec.dk
    c_qk, c_v, c_conv, r_in = spec.c_qk, spec.c_v, spec.c_conv, spec.r_in
    w_el = r_in * H + H * c_v
    C = 64
    nch = (n + C - 1) // C
    return {
        # Q4_K blocks read (144 B / 256 weights) + int8 codes and fp32 row scales written
        "dequant": ("hbm", w_el * 144 / 256 + w_el * 1 + (r_in + H) * 4),
        # bf16 x read, int8 codes + scales written
        "act_quant": ("hbm", n * H * 2 + n * H * 1 + n * 4),
        "in_proj": ("tensor", 2.0 * n * r_in * H),
        # raw q|k|v read and conv output written (bf16 each); conv state
        "conv": ("hbm", n * c_conv * 2 * 2 + c_conv * 4 * 4),
        # q, k, v read and o written (bf16), gates read (fp32), the fp32 state in and out,
        # and one pass over the per-chunk intermediates of the chunked form
        # (U [C][dv] and W [C][dk] per chunk and value head, fp32)
        "delta_rule": ("hbm", n * c_conv * 2 + n * c_v * 2 + 2 * n * hv * 4 + 2 * hv * d * d * 4
                       + nch * hv * C * 2 * d * 4),
        # o and z read (bf16), int8 codes + scales written
        "gated_norm": ("hbm", n * c_v * 2 + n * c_v * 2 + n * c_v * 1 + n * 4),
        "out_proj": ("tensor", 2.0 * n * H * c_v),
    }


def traffic_from_profile(kernel_src: str, profile_md: str):
    """DRAM bytes per launch recorded in a committed ncu summary, if the kernel source is unchanged."""
    if not os.path.exists(profile_md):
        return None
    text = open(profile_md).read()
    m = re.search(r"kernel_source_sha256:\s*([0-9a-f]{64})", text)
    t = re.search(r"dram_bytes_per_launch_full_size:\s*([0-9.eE+]+)", text)
    if not m or not t:
        return None
    h = hashlib.sha256(open(kernel_src, "rb").read()).hexdigest()
    return float(t.group(1)) if h == m.group(1) else None


# ------------------------------------------------------------------ CPU oracle

def oracle_params(spec, layer):
    from oracle import q4k
    p = dict(wtype=spec.wtype, hidden=spec.hidden, n_qk_heads=spec.n_qk_heads, n_v_heads=spec.n_v_heads,
             dk=spec.dk, dv=spec.dv, conv_w=layer["conv_w"], A_log=layer["A_log"], dt_bias=layer["dt_bias"],
             norm_w=layer["norm_w"], eps_l2=1e-6, eps_rms=1e-6, q_scale=spec.dk ** -0.5)
    p["w_in"] = q4k.pack_q4k(layer["w_in"]) if spec.wtype == "q4k" else layer["w_in"]
    p["w_out"] = q4k.pack_q4k(layer["w_out"]) if spec.wtype == "q4k" else layer["w_out"]
    return p


def time_oracle(spec, layer, tok, n_sample):
    """Oracle (as it stands) on the first n_sample tokens; returns seconds."""
    from oracle import layer as OL
    p = oracle_params(spec, layer)
    t0 = time.perf_counter()
    OL.layer_forward(p, tok["x"][:n_sample], gate_log_a=tok["log_a"][:n_sample], gate_b=tok["b"][:n_sample])
    return time.perf_counter() - t0


# ------------------------------------------------------------------ arms

def run_reference(args, dist, spec):
    if dist.rank != 0:
        return
    from hybrid_gated_deltanet_q4k_gb300 import synth
    layer = synth.make_layer(spec)
    n_sample = 256
    tok = synth.make_tokens(spec, n_sample, seed=spec.seed + 10)
    for _ in range(args.warmup):
        time_oracle(spec, layer, tok, n_sample)
    times = [time_oracle(spec, layer, tok, n_sample) for _ in range(args.steps)]
    t = sum(times) / len(times)
    v = n_sample / t
    sample = (f"first {n_sample} tokens of the {spec.workload} workload per step (weights decoded each call, "
              f"recurrence one token at a time in fp64)")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": spec.workload, "tokens_per_step": n_sample},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": _CORES, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_ours(args, dist, spec):
    import ctypes

    import torch

    from hybrid_gated_deltanet_q4k_gb300 import lib as gl
    from hybrid_gated_deltanet_q4k_gb300 import synth
    from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer

    torch.cuda.set_device(dist.local)
    dev = f"cuda:{dist.local}"
    L = gl.load(build=True)
    n = args.tokens or spec.n_tokens
    layer = synth.make_layer(spec)
    tok = synth.make_tokens(spec, n, seed=spec.seed + 10 + dist.rank)
    dl = DeviceLayer(spec, layer, device=dev)
    x = torch.from_numpy(tok["x_bits"].view(np.int16)).to(dev).view(torch.bfloat16)
    la = torch.from_numpy(tok["log_a"]).to(dev)
    bb = torch.from_numpy(tok["b"]).to(dev)
    state, conv = dl.new_state()
    y = torch.empty(n, spec.hidden, dtype=torch.bfloat16, device=dev)
    ws = dl.new_workspace(n)
    stream = torch.cuda.current_stream()

    def step():
        conv.zero_()
        dl.prefill(x, None, state, conv, y, ws, gate_log_a=la, gate_b=bb)

    for _ in range(max(args.warmup, 3)):
        step()
    assert L.gdn_sync_status(stream.cuda_stream, check=False) == 0, L.last_error()

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(gl.GDN_N_STAGE_EVENTS)] for _ in range(K)]
    for row in ev:              # torch creates the CUDA event at its first record
        for e in row:
            e.record(stream)

    def timed():
        dist.barrier()
        torch.cuda.synchronize()
        t_host0 = time.time()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(K):
            arr = (ctypes.c_void_p * gl.GDN_N_STAGE_EVENTS)(*[e.cuda_event for e in ev[i]])
            L.gdn_set_stage_events(arr, gl.GDN_N_STAGE_EVENTS)
            step()
        e1.record(stream)
        L.gdn_set_stage_events(None, 0)
        torch.cuda.synchronize()
        t_host1 = time.time()
        dist.barrier()
        return e0.elapsed_time(e1) / K, t_host0, t_host1

    gpu_id = str(getattr(torch.cuda.get_device_properties(dist.local), "uuid", dist.local))
    if not gpu_id.startswith("GPU-") and len(gpu_id) == 36:
        gpu_id = "GPU-" + gpu_id
    sampler = ClockSampler(gpu_id)
    time.sleep(0.3)
    ms, h0, h1 = timed()
    clocks = ClockSampler.summarize(sampler.stop(), h0, h1)
    if REJECT & set(clocks["reasons"]):     # throttled: measure once more
        sampler = ClockSampler(gpu_id)
        time.sleep(0.3)
        ms, h0, h1 = timed()
        clocks = ClockSampler.summarize(sampler.stop(), h0, h1)
        clocks["remeasured"] = True
    assert L.gdn_sync_status(stream.cuda_stream, check=False) == 0, L.last_error()
    ms_max = dist.max(ms)

    # per-stage average durations (ms) from the stage events
    names = gl.STAGE_NAMES
    stage_ms = {nm: sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(K)) / K for j, nm in enumerate(names)}
    pk = peaks()
    work = stage_work(spec, n)
    # A stage that runs inside the previous one (the gated norm of each token
    # segment beside the delta rule's later segments) has an empty interval:
    # report the two as one stage.
    merged = []
    for nm in names:
        if merged and stage_ms[nm] < 0.005 and work[nm][0] == work[merged[-1]][0] == "hbm":
            prev = merged[-1]
            both = prev + "+" + nm
            stage_ms[both] = stage_ms.pop(prev) + stage_ms.pop(nm)
            work[both] = ("hbm", work[prev][1] + work[nm][1])
            merged[-1] = both
        else:
            merged.append(nm)
    names = merged
    stages = {}
    for nm in names:
        kind, amount = work[nm]
        sec = stage_ms[nm] / 1e3
        if kind == "tensor":
            a = amount / sec / 1e12
            stages[nm] = {"ms": stage_ms[nm], "bound": "tensor", "achieved": a, "unit": "TFLOP/s", "frac": a / pk["tensor"],
                          "frac_sustained": a / pk["tensor_sustained"]}
        else:
            a = amount / sec / 1e9
            stages[nm] = {"ms": stage_ms[nm], "bound": "hbm", "achieved": a, "unit": "GB/s", "frac": a / pk["hbm"]}
        if nm.startswith("delta_rule"):
            # the recurrence against the tensor roofline too: the chunked form's
            # FLOPs, N Hv (10 C dk + 6 dk^2) with chunks of C = 64
            fl = n * spec.n_v_heads * (10 * 64 * spec.dk + 6 * spec.dk * spec.dk)
            stages[nm]["tensor_achieved_tflops"] = fl / sec / 1e12
            stages[nm]["tensor_frac"] = fl / sec / 1e12 / pk["tensor"]
    dom = stages["in_proj"]
    traffic = traffic_from_profile(os.path.join(ROOT, "hybrid_gated_deltanet_q4k_gb300", "csrc", "k_gemm.cu"),
                                   os.path.join(ROOT, "profiles", "gemm_codes_in_proj_h4096_n32768.md"))
    roofline = {"bound": "tensor", "achieved": dom["achieved"], "peak": pk["tensor"], "unit": "TFLOP/s",
                "frac": dom["frac"], "traffic": traffic, "kernel": "gemm_codes_kernel (input projection, 3.316 TFLOP/launch)",
                "peak_source": pk["src"],
                "peak_sustained": pk["tensor_sustained"], "frac_sustained": dom["frac_sustained"],
                "int8_peak": "int8 codes on the fp16 tensor path (no int8 tcgen05 kind on sm_103a): "
                             "denominator = measured bf16/fp16 burst peak",
                "traffic_source": ("ncu dram__bytes_read.sum + dram__bytes_write.sum of one full-size input-projection "
                                   "launch, from profiles/gemm_codes_in_proj_h4096_n32768.md, used only while "
                                   "k_gemm.cu's sha256 matches the one recorded there (else null)")}

    # end to end through the public host-fed call: x and the drawn gates come
    # from pinned host memory and y goes back to it, every step; the library
    # overlaps the copies of neighbouring passes with the compute
    e2e = None
    if not args.no_e2e:
        xh = torch.from_numpy(tok["x_bits"].view(np.int16)).pin_memory()
        lah = torch.from_numpy(tok["log_a"]).pin_memory()
        bh = torch.from_numpy(tok["b"]).pin_memory()
        yh = torch.empty(n, spec.hidden, dtype=torch.int16).pin_memory()
        P = min(args.e2e_pass, n)
        wsh = dl.new_host_workspace(P, gates=True)

        def e2e_step():
            conv.zero_()
            dl.prefill_host(xh, None, state, conv, yh, wsh, pass_tokens=P, gate_log_a=lah, gate_b=bh)

        for _ in range(max(args.warmup, 3)):
            e2e_step()
        dist.barrier()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(K):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
        assert L.gdn_sync_status(stream.cuda_stream, check=False) == 0, L.last_error()
        e2e_ms = dist.max(e0.elapsed_time(e1) / K)
        e2e = {"value": whole_job_rate(n, dist.world, e2e_ms), "unit": UNIT,
               "h2d_bytes_per_step": xh.numel() * 2 + lah.numel() * 4 + bh.numel() * 4,
               "d2h_bytes_per_step": yh.numel() * 2, "ms_per_step": e2e_ms,
               "call": f"gdn_prefill_host, passes of {P} tokens"}
        del wsh

    cpu = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        n_sample = 1024
        t = time_oracle(spec, layer, tok, n_sample)
        cpu = {"value": n_sample / t, "unit": UNIT, "cores": _CORES, "kind": "oracle",
               "sample": f"first {n_sample} of the {n} tokens of {spec.workload} (one call: weight decode, "
                         f"projections as fp64 matmuls on the exact int8 operands, recurrence one token at a time)"}

    passes = 1
    # per step: weight decode (one launch, both matrices); per token pass: x
    # quantisation, input projection, conv, conv state, output projection, and
    # per token segment of the delta rule its prep, its state pass and its
    # gated norm (segments of 64 chunks, of 128 from 512 chunks on; one segment
    # up to 64 chunks)
    nch = (n + 63) // 64
    seg = 128 if nch >= 512 else 64
    segments = 1 if nch <= 64 else (nch + seg - 1) // seg
    launches = (1 + (5 + 3 * segments) * passes) * K
    if dist.rank == 0:
        print(json.dumps({
            "metric": METRIC, "value": whole_job_rate(n, dist.world, ms_max), "unit": UNIT, "n_gpus": dist.world,
            "steps": K, "warmup": max(args.warmup, 3), "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "dtype_detail": "int8 codes (exact in fp16) on fp16 tcgen05 tensor cores with exact int32 sums; "
                            "bf16 activations; fp32 conv/norm/recurrence state",
            "data": "synthetic (seeded random weights and inputs of the stated distributions)",
            "config": {"workload": spec.workload, "n_tokens": n, "hidden": spec.hidden,
                       "heads": f"{spec.n_qk_heads}x{spec.dk} q/k, {spec.n_v_heads}x{spec.dv} v",
                       "weights": "Q4_K", "state": "zero", "gates": "drawn, log a ~ U(-0.5,0)",
                       "l2": "no flush: inputs larger than L2 (x 268 MB, workspace %.1f GB)" % (ws.numel() / 1e9),
                       "parallelism": "replicas only" if dist.world > 1 else "single GPU"},
            "roofline": roofline, "stages": stages, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
            "clocks": clocks,
        }), flush=True)


def run_stage(args, spec):
    """One stage kernel alone, on the workload's shapes with `--tokens` rows (a profiling case)."""
    import ctypes

    import torch

    from hybrid_gated_deltanet_q4k_gb300 import lib as gl
    from hybrid_gated_deltanet_q4k_gb300 import synth
    from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer

    L = gl.load(build=True)
    n = args.tokens or spec.n_tokens
    H, r_in, hv, d = spec.hidden, spec.r_in, spec.n_v_heads, spec.dk
    nbf = 2 * spec.c_qk + 2 * spec.c_v
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    st = torch.cuda.current_stream().cuda_stream
    g = torch.Generator(device="cuda").manual_seed(0)
    if args.stage == "in_proj":
        wc = torch.empty(r_in, H, dtype=torch.float16, device="cuda")
        ws = torch.empty(r_in, dtype=torch.float32, device="cuda")
        L.gdn_q4k_deq_codes(gl.ptr(dl.dev["w_in"]), r_in, H, gl.ptr(wc), gl.ptr(ws), st)
        xc = torch.randint(-127, 128, (n, H), device="cuda", generator=g).to(torch.float16)
        sx = torch.rand(n, device="cuda", generator=g)
        out = torch.empty(n, nbf, dtype=torch.bfloat16, device="cuda")
        ba = torch.empty(n, 2 * hv, dtype=torch.float32, device="cuda")
        fn = lambda: L.gdn_gemm_codes(gl.ptr(xc), gl.ptr(sx), gl.ptr(wc), gl.ptr(ws), n, r_in, H, gl.ptr(out), nbf,  # noqa: E731
                                      nbf, gl.ptr(ba), 2 * hv, st)
        work, unit = 2.0 * n * r_in * H / 1e12, "TFLOP"
    elif args.stage in ("q6k_deq", "q4k_deq"):
        # step 1a alone on the input-projection matrix [R_in][H], each format:
        # HBM bytes = blocks read + int8 codes and fp32 scales written
        from hybrid_gated_deltanet_q4k_gb300.api import pack_q4k, pack_q6k
        q6 = args.stage == "q6k_deq"
        blocks = torch.from_numpy((pack_q6k if q6 else pack_q4k)(layer["w_in"])).cuda()
        q8 = torch.empty(r_in, H, dtype=torch.int8, device="cuda")
        sc = torch.empty(r_in, dtype=torch.float32, device="cuda")
        dec = L.q6k_deq_i8 if q6 else L.q4k_deq_i8
        fn = lambda: dec(gl.ptr(blocks), r_in, H, gl.ptr(q8), gl.ptr(sc), st)  # noqa: E731
        work, unit = (blocks.numel() + q8.numel() + 4 * r_in) / 1e9, "GB"
    else:
        s = dl.struct()
        qkv = (torch.randn(n, spec.c_conv, device="cuda", generator=g) * 0.05).to(torch.float16)
        la = -0.5 * torch.rand(n, hv, device="cuda", generator=g)
        b = torch.rand(n, hv, device="cuda", generator=g)
        stt = torch.zeros(hv, d, d, device="cuda")
        o = torch.empty(n, spec.c_v, dtype=torch.float16, device="cuda")
        nbytes = L.gdn_delta_rule_scratch_size(ctypes.byref(s), n)
        scratch = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        fn = lambda: L.gdn_delta_rule(ctypes.byref(s), gl.ptr(qkv), gl.ptr(la), gl.ptr(b), n, 0, gl.ptr(stt),  # noqa: E731
                                      gl.ptr(o), gl.ptr(scratch), nbytes, st)
        work, unit = n / 1e6, "Mtoken"
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    assert L.gdn_sync_status(st, check=False) == 0, L.last_error()
    ms = e0.elapsed_time(e1) / args.steps
    rate = work / (ms / 1e3)
    out = {"stage": args.stage, "workload": spec.workload, "tokens": n, "ms_per_launch": ms, "rate": rate,
           "rate_unit": unit + "/s"}
    pk = peaks()
    if unit == "GB":
        out["roofline"] = {"bound": "hbm", "achieved": rate, "peak": pk["hbm"], "unit": "GB/s",
                           "frac": rate / pk["hbm"], "peak_source": pk["src"]}
        # the oracle beside it: the same decode and quantisation of the first 256 rows
        from oracle import q4k as O4, q6k as O6, quant as OQ
        rs = 256
        fmt = O6 if args.stage == "q6k_deq" else O4
        blk = (O6.pack_q6k if args.stage == "q6k_deq" else O4.pack_q4k)(layer["w_in"][:rs])
        t0 = time.perf_counter()
        w = (O6.unpack_q6k if args.stage == "q6k_deq" else O4.unpack_q4k)(blk, rs, H)
        OQ.quant_rows_i8(w)
        t_or = time.perf_counter() - t0
        out["cpu_baseline"] = {"value": (blk.nbytes + rs * H + 4 * rs) / 1e9 / t_or, "unit": "GB/s", "cores": _CORES,
                               "kind": "oracle", "sample": f"the first {rs} rows of W_in ({fmt.__name__}: decode, int8 rows)"}
    elif unit == "TFLOP":
        out["roofline"] = {"bound": "tensor", "achieved": rate, "peak": pk["tensor"], "unit": "TFLOP/s",
                           "frac": rate / pk["tensor"], "peak_source": pk["src"]}
    print(json.dumps(out), flush=True)


def run_extend(args, spec):
    """Session-extend workload (8 sequences of the h2560 layer, each extending a
    saved 2048-token state by U[1, 4096] tokens): the extensions in one
    gdn_prefill_batch call against one gdn_prefill call per sequence, both
    timed with CUDA events, inputs resident.  A secondary measurement, not the
    headline metric."""
    import torch

    from hybrid_gated_deltanet_q4k_gb300 import lib as gl
    from hybrid_gated_deltanet_q4k_gb300 import synth
    from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer

    L = gl.load(build=True)
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    cases = synth.make_extend_case(spec)
    n = len(cases)
    pre, ext = cases[0]["prefix"], [c["extension"] for c in cases]
    cu = np.concatenate([[0], np.cumsum(ext)]).astype(np.int64)
    T = int(cu[-1])
    x = torch.from_numpy(np.concatenate([c["x_bits"][pre:] for c in cases]).view(np.int16)).cuda().view(torch.bfloat16)
    la = torch.from_numpy(np.concatenate([c["log_a"][pre:] for c in cases])).cuda()
    bb = torch.from_numpy(np.concatenate([c["b"][pre:] for c in cases])).cuda()
    rng = np.random.default_rng(7)
    s_saved = torch.from_numpy((0.05 * rng.standard_normal((n, spec.n_v_heads, spec.dv, spec.dk))).astype(np.float32)).cuda()
    c_saved = torch.from_numpy(rng.standard_normal((n, spec.c_conv, 3)).astype(np.float32)).cuda()
    st, cv = s_saved.clone(), c_saved.clone()
    y = torch.empty(T, spec.hidden, dtype=torch.bfloat16, device="cuda")
    wsb = dl.new_batch_workspace(T, n)
    wss = dl.new_workspace(max(ext))
    stream = torch.cuda.current_stream()

    def batch():
        dl.prefill_batch(x, cu, s_saved, st, cv, y, wsb, gate_log_a=la, gate_b=bb)

    def sequential():
        for i in range(n):
            a, b = int(cu[i]), int(cu[i + 1])
            dl.prefill(x[a:b], s_saved[i], st[i], cv[i], y[a:b], wss, gate_log_a=la[a:b], gate_b=bb[a:b])

    res = {}
    for name, fn in (("batch", batch), ("per_sequence", sequential)):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        assert L.gdn_sync_status(stream.cuda_stream, check=False) == 0, L.last_error()
        ms = e0.elapsed_time(e1) / args.steps
        res[name] = {"ms_per_step": ms, "value": T / (ms / 1e3)}
    # whole-call tensor roofline: the two projections' FLOPs over the batch call
    pk = peaks()
    tflop = 2.0 * T * (spec.r_in * spec.hidden + spec.hidden * spec.c_v) / 1e12
    tf = tflop / (res["batch"]["ms_per_step"] / 1e3)
    roofline = {"bound": "tensor", "achieved": tf, "peak": pk["tensor"], "unit": "TFLOP/s", "frac": tf / pk["tensor"],
                "peak_source": pk["src"],
                "work": f"both projections, {tflop:.3f} TFLOP per call, over the whole call's time (conv and delta "
                        "rule included: a lower bound on the projections' own rate)"}
    # the oracle beside it: the first 128 tokens of the first extension, from its saved state
    from oracle import layer as OL
    ns = min(128, ext[0])
    c0 = cases[0]
    t0 = time.perf_counter()
    OL.layer_forward(oracle_params(spec, layer), c0["x"][pre:pre + ns], S0=s_saved[0].cpu().numpy().astype(np.float64),
                     conv_tail=c_saved[0].cpu().numpy().astype(np.float64), gate_log_a=c0["log_a"][pre:pre + ns],
                     gate_b=c0["b"][pre:pre + ns])
    t_or = time.perf_counter() - t0
    cpu = {"value": ns / t_or, "unit": UNIT, "cores": _CORES, "kind": "oracle",
           "sample": f"the first {ns} tokens of the first sequence's extension, from its saved state (one call: "
                     "weight decode, fp64 projections on the exact int8 operands, recurrence one token at a time)"}
    print(json.dumps({"metric": "GDN-layer extend tokens/s, 8 sequences (1 GB300)", "unit": UNIT,
                      "value": res["batch"]["value"], "ms_per_step": res["batch"]["ms_per_step"],
                      "per_sequence_calls": res["per_sequence"], "steps": args.steps, "warmup": max(args.warmup, 3),
                      "roofline": roofline, "cpu_baseline": cpu,
                      "dtype": "int8", "data": "synthetic",
                      "config": {"workload": "extend_h2560_8seq", "hidden": spec.hidden, "prefix": pre,
                                 "extensions": ext, "tokens": T, "call": "gdn_prefill_batch"}}), flush=True)


def run_decode(args, spec):
    """Decode step of the 32k layer (h4096): one token for each of B sequences
    with saved states, every step through gdn_decode; inputs resident, timed
    with CUDA events.  HBM roofline: the Q4_K bytes of both weight matrices plus
    the states read and written, per step.  A secondary measurement."""
    import torch

    from hybrid_gated_deltanet_q4k_gb300 import lib as gl
    from hybrid_gated_deltanet_q4k_gb300 import synth
    from hybrid_gated_deltanet_q4k_gb300.api import DeviceLayer

    L = gl.load(build=True)
    layer = synth.make_layer(spec)
    dl = DeviceLayer(spec, layer)
    stream = torch.cuda.current_stream()
    pk = peaks()
    rows = []
    for B in ((args.seqs,) if args.seqs else (1, 8, 32)):
        tok = synth.make_tokens(spec, B, seed=90 + B)
        x = torch.from_numpy(tok["x_bits"].view(np.int16)).cuda().view(torch.bfloat16)
        la, bb = torch.from_numpy(tok["log_a"]).cuda(), torch.from_numpy(tok["b"]).cuda()
        st, cv = dl.new_batch_state(B)
        st.normal_(0, 0.05)
        y = torch.empty(B, spec.hidden, dtype=torch.bfloat16, device="cuda")
        ws = dl.new_decode_workspace(B)
        fn = lambda: dl.decode(x, st, cv, y, ws, gate_log_a=la, gate_b=bb)  # noqa: E731
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        # steps back to back: the layer's weights (38 MB) stay in L2 between steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        us_warm = e0.elapsed_time(e1) / args.steps * 1e3
        # L2 flushed before each step (as between the layers of a model): the
        # weights and states come from HBM; each step timed alone
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a0, a1 in evs:
            flush.fill_(1)
            a0.record(stream)
            fn()
            a1.record(stream)
        torch.cuda.synchronize()
        assert L.gdn_sync_status(stream.cuda_stream, check=False) == 0, L.last_error()
        us = sum(a0.elapsed_time(a1) for a0, a1 in evs) / args.steps * 1e3
        del flush
        wbytes = dl.dev["w_in"].numel() + dl.dev["w_out"].numel()
        sbytes = 2 * st.numel() * 4
        gbs = (wbytes + sbytes) / (us * 1e-6) / 1e9
        rows.append({"n_seqs": B, "us_per_step": us, "l2": "flushed before each step",
                     "us_per_step_l2_warm": us_warm, "tokens_per_s": B / (us * 1e-6), "hbm_bytes": wbytes + sbytes,
                     "achieved_gbs": gbs, "frac": gbs / pk["hbm"]})
    # the oracle beside it: one decode step of one sequence (weights decoded each call)
    from oracle import layer as OL
    tok = synth.make_tokens(spec, 1, seed=91)
    rng = np.random.default_rng(1)
    s0 = rng.normal(0, 0.05, size=(spec.n_v_heads, spec.dv, spec.dk))
    t0 = time.perf_counter()
    OL.layer_forward(oracle_params(spec, layer), tok["x"][:1], S0=s0, conv_tail=np.zeros((spec.c_conv, 3)),
                     gate_log_a=tok["log_a"][:1], gate_b=tok["b"][:1], decode=True)
    t_or = time.perf_counter() - t0
    cpu = {"value": 1.0 / t_or, "unit": "tokens/s", "us_per_step": t_or * 1e6, "cores": _CORES, "kind": "oracle",
           "sample": "one decode step of one sequence (B = 1): Q4_K decode of both matrices, fp64 products on the "
                     "exact int8 operands, one token of the recurrence"}
    print(json.dumps({"metric": "GDN-layer decode step (1 GB300)", "workload": spec.workload, "steps": args.steps,
                      "peak_gbs": pk["hbm"], "peak_source": pk["src"], "rows": rows, "cpu_baseline": cpu,
                      "dtype": "int8", "data": "synthetic", "call": "gdn_decode"}), flush=True)


def run_attn(args):
    """Prefill of a full-attention layer of the 9B-like hybrid (16 query heads
    over 4 key/value heads of 256; the pages give no sizes for these layers, so
    the GQA ratio and head size are a reading), N = 32768 causal, through
    gdn_attn_prefill; inputs resident, CUDA events.  Tensor roofline: the causal
    FLOPs 4 d Hq N (N + 1) / 2 against the bf16 peak (burst: the kernel timed
    alone).  A secondary measurement."""
    import torch

    from hybrid_gated_deltanet_q4k_gb300 import lib as gl
    from hybrid_gated_deltanet_q4k_gb300 import synth

    L = gl.load(build=True)
    n = args.tokens or 32768
    hq, hkv, d = 16, 4, 256
    inp = synth.make_attention(n, n, hq, hkv, d, seed=11)
    dev = lambda b: torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)  # noqa: E731
    q, k, v = dev(inp["q_bits"]), dev(inp["k_bits"]), dev(inp["v_bits"])
    o = torch.empty(n, hq, d, dtype=torch.bfloat16, device="cuda")
    nbytes = L.gdn_attn_workspace_size(n, hkv, d)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    fn = lambda: L.gdn_attn_prefill(gl.ptr(q), gl.ptr(k), gl.ptr(v), n, n, hq, hkv, d, 0.0, gl.ptr(o), gl.ptr(ws),  # noqa: E731
                                    nbytes, stream.cuda_stream)
    for _ in range(max(args.warmup, 3)):
        fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    assert L.gdn_sync_status(stream.cuda_stream, check=False) == 0, L.last_error()
    ms = e0.elapsed_time(e1) / args.steps
    flops = 4.0 * d * hq * n * (n + 1) / 2
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    peak = json.load(open(path))["bf16_tflops"] if os.path.exists(path) else 1900.0
    tf = flops / (ms / 1e3) / 1e12
    # the oracle beside it: the last 16 queries (the longest rows) against all keys,
    # scaled to tokens/s of the causal prefill by FLOPs (an average query does
    # (n + 1) / 2 of the n key products these do)
    from oracle.attention import attention as oracle_attention
    ns = min(16, n)
    t0 = time.perf_counter()
    oracle_attention(inp["q"][n - ns:], inp["k"], inp["v"])
    t_or = time.perf_counter() - t0
    f_sample = 4.0 * d * hq * ns * n
    cpu = {"value": f_sample / t_or / (flops / n), "unit": "tokens/s", "tflops": f_sample / t_or / 1e12,
           "cores": _CORES, "kind": "oracle",
           "sample": f"the last {ns} queries against all {n} keys, fp64 (tokens/s of the causal prefill at the same "
                     "FLOP rate)"}
    print(json.dumps({"metric": "full-attention layer prefill tokens/s (1 GB300)", "unit": "tokens/s",
                      "value": n / (ms / 1e3), "ms_per_step": ms, "steps": args.steps, "cpu_baseline": cpu,
                      "roofline": {"bound": "tensor", "achieved": tf, "peak": peak, "unit": "TFLOP/s", "frac": tf / peak,
                                   "peak_source": "of measured (MEASURED_PEAKS.json bf16_tflops, burst)"},
                      "dtype": "bf16", "data": "synthetic",
                      "config": {"workload": f"attn_causal_n{n}_hq{hq}_hkv{hkv}_d{d}", "call": "gdn_attn_prefill"}}),
          flush=True)


def main():
    args = parse()
    if args.config == "attn" and args.impl == "ours":
        run_attn(args)
        return
    if args.config == "decode" and args.impl == "ours":
        from hybrid_gated_deltanet_q4k_gb300 import synth
        run_decode(args, synth.SPECS["h4096"])
        return
    if args.config == "extend" and args.impl == "ours" and not args.stage:
        from hybrid_gated_deltanet_q4k_gb300 import synth
        run_extend(args, synth.SPECS["extend"])
        return
    if args.stage:
        from hybrid_gated_deltanet_q4k_gb300 import synth
        run_stage(args, synth.SPECS[args.config])
        return
    dist = Dist()
    from hybrid_gated_deltanet_q4k_gb300 import synth
    spec = synth.SPECS[args.config]
    try:
        if args.impl == "reference":
            run_reference(args, dist, spec)
        else:
            run_ours(args, dist, spec)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
