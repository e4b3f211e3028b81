#!/usr/bin/env python
"""TTT-E2E inner-loop prefill throughput on B300 (libttt, sm_103a).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 760m] [--impl ours|reference]

One step = every sequence of the workload's context (one for the 125M, 760M
and 3B workloads, four for the window/chunk sweep) through the inner loop:
for every chunk of b tokens, forward through all blocks, next-token
cross-entropy, backward through the last quarter of the blocks and the SGD
step on their MLP weights, then the window-cache commit.  Each step restarts
the sequences from the loaded weights (ttt_reset, inside the timed region).
value = tokens of all ranks / max over ranks of the device time of K steps
(CUDA events on the library's stream).

Multi-GPU: the inner loop is a serial chain within a sequence, so ranks are
independent replicas (their own sequences, seeds 1000 + rank*n_seqs + q); the
only collectives are the timing barrier and the max-reduction of the elapsed
time.

--impl reference times the float64 oracle (the method as written, numpy) on
the host cores on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from ttt_inputs import SHAPES, sequence_tokens, weight_blob  # noqa: E402

METRIC = "TTT prefill tokens/sec at 1 B300; % of bf16 tensor-core roofline"
PROFILE_EVERY = 8  # launches of the dominant class per bracketed one, in the timed region
UNIT = "tokens/s"
DATA = "synthetic: Zipf(1.1) token ids with repeated 32-token spans (sequence q of rank r: seed 1000 + r*n_seqs + q), N(0,0.02) weights (seed 0)"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return dict(hbm=j["hbm_gbs"], tc=j["bf16_tflops"], tc_sus=j["bf16_tflops_sustained"], kind="measured")
    return dict(hbm=6400.0, tc=1800.0, tc_sus=1400.0, kind="fallback")


def algorithmic_flops(s, T):
    """FLOPs the method needs for one T-token sequence (no recompute, no masked tiles).

    forward : T L (8d^2 + 4df) + 4d P L + 2dVT, P = sum_p min(p+1, k) window pairs
    backward: 2dVT (LM-head dX) + T (S-1)(8d^2 + 8df) + 6 T d f (first trainable block:
              dU, dW_down, dW_up only) + (S-1)(4d P + 4d O), O = own-chunk causal pairs
    """
    d, f, V, L, S, k, b = s.d_model, s.d_ff, s.vocab, s.n_layers, s.n_trainable, s.window, s.chunk
    pairs = sum(min(p + 1, k) for p in range(T)) if T <= k else k * (k + 1) // 2 + (T - k) * k
    own = sum(n * (n + 1) // 2 for n in [min(b, T - c) for c in range(0, T, b)])
    fwd = T * L * (8 * d * d + 4 * d * f) + 4 * d * pairs * L + 2 * d * V * T
    bwd = (2 * d * V * T + T * (S - 1) * (8 * d * d + 8 * d * f) + T * 6 * d * f
           + (S - 1) * (4 * d * pairs + 4 * d * own))
    return fwd + bwd


class Clocks:
    """nvidia-smi sampler (200 ms) over the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.p = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                       "-lms", "200", "-i", str(gpu_id)], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.p.terminate()
        try:
            self.p.wait(5)
        except subprocess.TimeoutExpired:
            self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [[x.strip() for x in r.split(",")] for r in self.f.read().strip().splitlines() if r.count(",") >= 7]
        os.unlink(self.f.name)

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(r[0]) for r in rows) if v is not None]
        mx = [v for v in (num(r[1]) for r in rows) if v is not None]
        pw = [v for v in (num(r[2]) for r in rows) if v is not None]
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(sm), "power_w_max": max(pw) if pw else None}


_UNPACKED = {}


def cpu_sample(shape, blob, tokens, n_tok):
    """Time the oracle on the first n_tok tokens (one inner-loop step) on the host cores."""
    from oracle import ttt_oracle as O
    try:
        from threadpoolctl import threadpool_info
        cores = max((i.get("num_threads", 1) for i in threadpool_info()), default=os.cpu_count())
    except Exception:
        cores = os.cpu_count()
    cfg = O.Config.from_shape(shape.replace(chunk=n_tok))
    key = (id(blob), n_tok)
    if key not in _UNPACKED:  # float64 parameters, converted once per process (untimed)
        _UNPACKED.clear()
        _UNPACKED[key] = O.unpack(blob, cfg)
    P = _UNPACKED[key]
    ids = np.asarray(tokens[:n_tok])
    tgt = O.chunk_targets(tokens, 0, n_tok)
    t0 = time.perf_counter()
    O.ttt_step(cfg, P, O.init_state(cfg), ids, tgt, shape.eta)
    dt = time.perf_counter() - t0
    return n_tok / dt, cores, dt


def max_over_ranks(x, dist, device):
    """The largest value of x over all ranks (the slowest replica's time); x when single-process."""
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_tokens_per_s(world, steps, tokens_per_step, seconds):
    """Whole-job throughput of `world` independent replicas, each processing
    tokens_per_step tokens per step, timed by the slowest one."""
    return world * steps * tokens_per_step / seconds


# DRAM bytes (read + write) of one steady-state launch (window full) of the attention
# forward at the 760M shape, from `ncu --set full` captures of this kernel: the
# frozen-block pass over 8192 queries, and a trainable block over one 1024-token chunk.
ATTN_FWD_TRAFFIC_760M = {"pass": 126.13e6 + 14.74e6, "step": 59.84e6 + 0.55e6}


def attn_fwd_traffic(shape, nc):
    """Average DRAM bytes per attention-forward launch over one step's launch mix (760M
    shape only; earlier chunks see partial windows and move fewer bytes, so this is an
    upper estimate), else None."""
    if ATTN_FWD_TRAFFIC_760M is None:
        return None
    if (shape.n_layers, shape.d_model, shape.window, shape.chunk) != (24, 1536, 8192, 1024):
        return None
    G = max(1, min(8192 // shape.chunk, shape.window // shape.chunk))
    passes = -(-nc // G) * (shape.n_layers - shape.n_trainable)
    steps = nc * shape.n_trainable
    t = ATTN_FWD_TRAFFIC_760M
    return (passes * t["pass"] + steps * t["step"]) / (passes + steps)


def chunk_major(tokens, b):
    """Inputs of ttt_prefill_chunk for every chunk of tokens [B][T]: the ids of chunk c
    as one [B][n_c] block after those of chunk c-1, and next[c][q], the token after
    chunk c of sequence q (-1 after the last)."""
    B, Tn = tokens.shape
    ids = np.concatenate([tokens[:, s:s + b].reshape(-1) for s in range(0, Tn, b)]).astype(np.int32)
    nxt = np.array([[tokens[q, s + b] if s + b < Tn else -1 for q in range(B)] for s in range(0, Tn, b)], np.int32)
    return ids, nxt


def workload_name(s):
    return (f"{s.n_layers}L d{s.d_model} H{s.n_heads} f{s.d_ff} V{s.vocab} k{s.window} b{s.chunk} "
            f"theta{s.rope_theta:g} eta{s.eta:g} {s.compute}: {s.n_seqs} x {s.seq_len} tokens")


def reference_tokens(steps, warmup, budget_s=120.0, s_per_token=0.025):
    """Tokens per oracle sample so that steps + warmup samples take about budget_s on the
    host cores (the float64 oracle runs the 760M shape at about s_per_token per token):
    a power of two between 64 and 1024, the workload's chunk."""
    n = budget_s / s_per_token / max(1, steps + warmup)
    t = 64
    while t * 2 <= min(n, 1024):
        t *= 2
    return t


def run_reference(a):
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    shape = SHAPES[a.workload]
    tokens = sequence_tokens(shape, 0)
    blob = weight_blob(shape)
    n_tok = a.cpu_tokens or reference_tokens(a.steps, a.warmup)
    for _ in range(a.warmup):
        cpu_sample(shape, blob, tokens, n_tok)
    secs, cores = [], None
    for _ in range(a.steps):
        _, cores, dt = cpu_sample(shape, blob, tokens, n_tok)
        secs.append(dt)
    value = a.steps * n_tok / sum(secs)
    sample = f"first {n_tok} tokens of sequence 0 as one inner-loop step (forward, loss, suffix backward, SGD)"
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": a.gpus,
           "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * sum(secs) / a.steps,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": DATA,
           "config": {"workload": workload_name(shape), "sample": sample},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)
    return 0


def run_ours(a):
    import torch
    import test_long_context_02_b300 as T

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    shape = SHAPES[a.workload]
    if a.tokens:
        shape = shape.replace(seq_len=a.tokens)
    # one step = every sequence of the workload's context (the window/chunk sweep holds 4)
    Tn, b, B = shape.seq_len, shape.chunk, shape.n_seqs
    nc = math.ceil(Tn / b)
    tokens = np.stack([sequence_tokens(shape, rank * B + q) for q in range(B)]).astype(np.int32)
    blob = weight_blob(shape)
    stream = torch.cuda.Stream()
    m = T.TTT.from_shape(shape, stream=stream.cuda_stream)
    m.load_weights(blob)
    d_tok = torch.tensor(tokens, dtype=torch.int32, device="cuda")
    d_loss = torch.zeros((B, nc), dtype=torch.float32, device="cuda")

    def one_step():
        m.reset()
        m.prefill_sequence_dev(d_tok, Tn, d_loss)

    for _ in range(a.warmup):
        one_step()
    m.sync()

    # per-class breakdown: one more step with every launch bracketed by events and the
    # context's streams run in issue order, so each launch is timed alone (not part of `value`)
    m.set_concurrency(False)
    m.profile(True)
    one_step()
    prof = m.profile_read()
    m.profile(False)
    m.set_concurrency(True)
    dom_name = max(prof, key=lambda k: prof[k]["ms"])

    # ---------------------------------------------------------------- timed region
    # only the dominant kernel class is bracketed by events here, for its live launch times,
    # and only one launch in PROFILE_EVERY: an event between two launches ends their
    # programmatic-launch overlap, so bracketing every launch would slow the timed steps
    clocks = Clocks(f"GPU-{torch.cuda.get_device_properties(local).uuid}")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    m.profile(True, classes=[dom_name], every=PROFILE_EVERY)
    barrier()
    torch.cuda.synchronize()
    l0 = m.launches
    ev0.record(stream)
    for _ in range(a.steps):
        one_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier()
    launches = m.launches - l0
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    dom = m.profile_read()[dom_name]
    m.profile(False)
    m.sync()
    losses = d_loss.cpu().numpy()
    if not np.all(np.isfinite(losses)):
        raise RuntimeError(f"non-finite chunk losses: {losses}")

    ms_max = max_over_ranks(ms, dist, "cuda")

    # ------------------------------------------------------------ end-to-end (host buffers)
    # The user's call on host memory: ttt_prefill_sequence uploads the step's tokens from
    # pinned memory, runs the sequence and downloads its chunk losses, all inside the timed
    # region.  The per-chunk API (ttt_prefill_chunk, one upload and one loss download per
    # chunk) is timed the same way as a second figure.
    e2e_steps = max(1, min(a.steps, 2))
    pin_tok = torch.tensor(tokens, dtype=torch.int32).pin_memory()
    # the per-chunk call takes [B][n] tokens of one chunk: the same ids, laid out chunk-major
    ctok, nxt = chunk_major(tokens, b)
    pin_ctok = torch.tensor(ctok, dtype=torch.int32).pin_memory()
    pin_next = torch.tensor(nxt).pin_memory()
    pin_loss = torch.zeros((B, nc), dtype=torch.float32).pin_memory()
    pin_closs = torch.zeros((nc, B), dtype=torch.float32).pin_memory()
    base_t, base_ct, base_n = pin_tok.data_ptr(), pin_ctok.data_ptr(), pin_next.data_ptr()
    base_l, base_cl = pin_loss.data_ptr(), pin_closs.data_ptr()

    def timed_host(run):
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for _ in range(e2e_steps):
            m.reset()
            run()
        torch.cuda.synchronize()
        dt = max_over_ranks(time.perf_counter() - t0, dist, "cuda")
        barrier()
        return dt

    def per_chunk():
        for ci in range(nc):
            s0 = ci * b
            n = min(b, Tn - s0)
            m._check(T.ttt_prefill_chunk(m._h, base_ct + 4 * B * s0, n, base_n + 4 * B * ci, base_cl + 4 * B * ci),
                     "ttt_prefill_chunk")

    e2e_s = timed_host(lambda: m._check(T.ttt_prefill_sequence(m._h, base_t, Tn, base_l), "ttt_prefill_sequence"))
    e2e_losses = pin_loss.numpy().copy()
    if not np.allclose(e2e_losses, losses, rtol=1e-3):
        raise RuntimeError(f"host-buffer sequence losses differ from the device-resident run: {e2e_losses} {losses}")
    e2e_chunk_s = timed_host(per_chunk)
    if not np.allclose(pin_closs.numpy().T, losses, rtol=1e-3):
        raise RuntimeError("per-chunk losses differ from the device-resident run")

    # --------------------------------------------------------------- reporting (rank 0)
    pk = peaks()
    alg = B * algorithmic_flops(shape, Tn)
    value = replica_tokens_per_s(world, a.steps, B * Tn, ms_max / 1e3)
    tc_frac = alg * a.steps / (ms / 1e3) / (pk["tc_sus"] * 1e12)
    total_ms = sum(v["ms"] for v in prof.values())
    avg_launch_ms = dom["ms"] / dom["launches"]
    def roofline(st):
        # the bound is the one whose peak takes longer for the class's algorithmic work
        # (the fused dW + SGD products, for example, move 8 B per fast weight)
        t_tc = st["alg_flops"] / (pk["tc_sus"] * 1e12)
        t_hbm = st["bytes"] / (pk["hbm"] * 1e9)
        if st["alg_flops"] > 0 and t_tc >= t_hbm:
            ach = st["alg_flops"] / (st["ms"] / 1e3) / 1e12
            return {"kernel": dom_name, "bound": "tensor", "achieved": ach, "peak": pk["tc_sus"], "unit": "TFLOP/s",
                    "frac": ach / pk["tc_sus"],
                    "traffic": attn_fwd_traffic(shape, nc) if dom_name == "attn_fwd" else None,
                    "peak_source": f"bf16_tflops_sustained ({pk['kind']}); burst {pk['tc']}",
                    "frac_of_burst": ach / pk["tc"], "avg_launch_ms": st["ms"] / st["launches"],
                    "launches_timed": st["launches"], "alg_flops_per_launch": st["alg_flops"] / st["launches"]}
        ach = st["bytes"] / (st["ms"] / 1e3) / 1e9
        return {"kernel": dom_name, "bound": "hbm", "achieved": ach, "peak": pk["hbm"], "unit": "GB/s",
                "frac": ach / pk["hbm"], "traffic": None, "avg_launch_ms": st["ms"] / st["launches"],
                "launches_timed": st["launches"], "alg_bytes_per_launch": st["bytes"] / st["launches"]}

    # timed region: the kernel shares the GPU with the other streams' kernels, so its launch
    # durations include that sharing; the isolated figure comes from the per-class step
    roof = dict(roofline(dom), launch_sample=f"1 in {PROFILE_EVERY} launches of the class, live in the timed region")
    roof_iso = dict(roofline(prof[dom_name]), note="same kernel, the per-class step: every launch alone, "
                    "the context's streams in issue order")
    kernels = {k: {"ms_per_step": round(v["ms"], 3), "share": round(v["ms"] / total_ms, 4),
                   "launches_per_step": v["launches"],
                   "alg_tflops": round(v["alg_flops"] / (v["ms"] / 1e3) / 1e12, 1) if v["alg_flops"] else None,
                   "exec_tflops": round(v["exec_flops"] / (v["ms"] / 1e3) / 1e12, 1) if v["exec_flops"] else None,
                   "hbm_gbs": round(v["bytes"] / (v["ms"] / 1e3) / 1e9, 1) if v["bytes"] else None}
               for k, v in sorted(prof.items(), key=lambda kv: -kv[1]["ms"])}
    if rank != 0:
        m.close()
        return 0
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": a.steps, "warmup": a.warmup,
           "ms_per_step": ms_max / a.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16" if shape.compute == "bf16" else "f32", "data": DATA,
           "config": {"workload": workload_name(shape), "tokens_per_step_per_gpu": B * Tn, "sequences": B,
                      "chunks": nc,
                      "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                      "l2": "working set larger than L2 (bf16 weights + window cache > 2 GB), no flush",
                      "timing": "CUDA events on the library stream; inside the timed region (the "
                                "context's streams overlapping, three per sequence lane, as the library runs "
                                "by default) only the dominant kernel class is bracketed by events, one "
                                f"launch in {PROFILE_EVERY}, on the stream each launch "
                                "goes to; the per-class table and roofline_isolated come from one extra "
                                "step with every launch bracketed and the streams in issue order",
                      "alg_gflop_per_token": alg / (B * Tn) / 1e9},
           "tc_roofline_frac": tc_frac,
           "tc_roofline_frac_of_burst": tc_frac * pk["tc_sus"] / pk["tc"],
           "roofline": roof, "roofline_isolated": roof_iso, "kernels": kernels, "clocks": clk, "gpu_launches": launches,
           "e2e": {"value": replica_tokens_per_s(world, e2e_steps, B * Tn, e2e_s), "unit": UNIT,
                   "h2d_bytes_per_step": 4 * B * Tn, "d2h_bytes_per_step": 4 * B * nc,
                   "api": "ttt_prefill_sequence, pinned host buffers (one upload, one download)",
                   "per_chunk_api": {"value": replica_tokens_per_s(world, e2e_steps, B * Tn, e2e_chunk_s),
                                     "h2d_bytes_per_step": 4 * B * (Tn + nc), "d2h_bytes_per_step": 4 * B * nc,
                                     "api": "ttt_prefill_chunk per chunk, pinned host buffers"}},
           "final_chunk_loss": float(losses[0, -1])}
    if world == 1 and not a.no_cpu_baseline:
        n_tok = a.cpu_tokens or 512
        v, cores, dt = cpu_sample(shape, blob, tokens[0], n_tok)
        out["cpu_baseline"] = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": f"first {n_tok} tokens as one inner-loop step, {dt:.1f} s"}
    print(json.dumps(out), flush=True)
    m.close()
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="760m", choices=sorted(SHAPES))
    ap.add_argument("--tokens", type=int, default=0, help="override the sequence length (smoke runs)")
    ap.add_argument("--cpu-tokens", type=int, default=None,
                    help="oracle sample size in tokens (default: 512 for cpu_baseline; for --impl reference, "
                         "sized so that warm-up and timed samples together take about two minutes)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    a = ap.parse_args()
    if a.warmup < 3:
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    return run_reference(a) if a.impl == "reference" else run_ours(a)


if __name__ == "__main__":
    sys.exit(main())
