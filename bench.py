#!/usr/bin/env python
"""Decode-step benchmark on GB300.

Workload (one JSON line on rank 0): the 24-layer Qwen2.5-0.5B-shaped decoder (hidden 896,
14 Q / 2 KV heads, head_dim 64, SwiGLU 4864, vocab 151936, tied head, fp16, seeded N(0, 0.02)
weights), continuous-batching decode at batch 32 (``--batch``), per-request contexts uniform in
[128, 1024], block size 16, physical blocks shuffled, the step captured as one CUDA graph and
replayed.  A "step" is one full decode iteration for every row: packed metadata upload, all
24 layers, the LM head to fp32 logits.

Reported:
  value      output tokens/s over K device-timed steps (CUDA events on the stream; metadata
             for each step prepared before the timed region, positions advancing every step).
  e2e        the same through the public API as a greedy decode loop: every step uploads its
             host metadata, runs, takes the argmax on the GPU and reads the token ids back to
             the host, which feed the next step.
  roofline   the dominant kernel (largest share of step time, measured with CUDA-event pairs
             around each launch in eager steps) against the measured HBM copy bandwidth.
  step_roofline  the whole step against max(FLOPs / tensor peak, bytes / HBM bandwidth).
  attention  the paged decode-attention kernel alone on its own workload (batch 256, 32 Q / 8
             KV heads, head_dim 128, bf16, contexts log-uniform in [512, 8192], 160k-block pool):
             algorithmic K/V bytes per launch / launch time.
  cpu_baseline  the fp64 CPU oracle on a bounded sample of the same workload.

``--impl reference`` times the CPU oracle alone (the reference arm).  Under torchrun each rank
runs an independent replica (no data-path collective; the step does not shard).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import synth  # noqa: E402
from transformer_decode_step_ns_gb300 import roofline as rl  # noqa: E402

METRIC = "decode output tokens/s at 1 GB300 (+ % of step roofline); paged-attn HBM GB/s"
WORKLOAD = "qwen2.5-0.5b-shape 24L fp16 decode, batch 32, ctx U[128,1024], bs16, graph replay"
SEED = synth.config_seed(1)
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ---------------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "samples": len(sm), "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------------- workload

class DecodeWorkload:
    """The decode workload on one GPU: model, KV pools, per-step metadata."""

    def __init__(self, batch: int, total_steps: int, use_graphs: bool = True):
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        self.shape = synth.qwen05b_shape(24)
        self.B = batch
        self.bs = 16
        t0 = time.time()
        self.w = synth.model_weights_device(self.shape, SEED)
        torch.cuda.synchronize()
        self.ctx = synth.ctx_uniform(SEED, "cfg1.ctx", batch, 128, 1024).astype(np.int64)
        grow = total_steps + 2
        self.mb = int(math.ceil((self.ctx.max() + 1 + grow) / self.bs)) + 1
        need = int(sum(math.ceil((c + 1 + grow) / self.bs) for c in self.ctx))
        self.num_blocks = need + batch
        self.dev = _lib.DecodeStep(self.shape, self.w, batch, self.mb, use_graphs=use_graphs)
        self.dev.kv_alloc(self.num_blocks, self.bs)
        # shuffle the physical free list: take every block, give them back in a seeded order
        ids = self.dev.reserve(self.num_blocks)
        perm = synth.permutation(SEED, "cfg1.pool", self.num_blocks)
        self.dev.release(ids[perm])
        self.tables = np.zeros((batch, self.mb), dtype=np.int32)
        for b in range(batch):
            n = int(math.ceil(self.ctx[b] / self.bs))
            self.tables[b, :n] = self.dev.reserve(n)
        stream = torch.cuda.current_stream().cuda_stream
        for l in range(self.shape.n_layers):
            k, v = self.dev.kv_layer_ptrs(l)
            n = self.dev.kv_pool_bytes() // 2
            synth.fill_normal_device(k, n, SEED, f"cfg1.k{l}", "f16", stream=stream)
            synth.fill_normal_device(v, n, SEED, f"cfg1.v{l}", "f16", stream=stream)
        torch.cuda.synchronize()
        self.positions = self.ctx.astype(np.int32).copy()
        self.tokens = synth.uniform_int(SEED, "cfg1.tokens", batch, 0,
                                        self.shape.vocab - 1).astype(np.int32)
        self.logits = torch.empty((batch, self.shape.vocab), dtype=torch.float32, device="cuda")
        self.setup_s = time.time() - t0

    def next_meta(self, tokens=None):
        """Advance every request by one token: allocate blocks as needed, map slots."""
        pos = self.positions.copy()
        slots = self.dev.prepare_step(pos, self.tables)
        meta = (self.tokens.copy() if tokens is None else np.asarray(tokens, np.int32),
                pos, self.tables.copy(), (pos + 1).astype(np.int32), slots)
        self.positions += 1
        return meta

    def step(self, meta):
        self.dev.step(*meta, self.logits)

    def meta_bytes(self) -> int:
        B, mb = self.B, self.mb
        o = 12 * B
        o = (o + 15) // 16 * 16 + 8 * B + 4 * B * mb
        return (o + 15) // 16 * 16 + 16


def kernel_bytes(shape, B, seq_lens):
    """Algorithmic bytes per launch for each kernel kind of one step (B rows)."""
    H, d, F, V = shape.hidden, shape.head_dim, shape.ffn, shape.vocab
    qd, kvd = shape.n_q_heads * d, shape.n_kv_heads * d
    e = 2
    return {
        "embed_rope": B * H * e + B * H * (4 + e) + B * (d // 2) * 8,
        "qkv": (qd + 2 * kvd) * H * e + B * H * e + B * (qd + 2 * kvd) * e,
        "attention": float(sum(seq_lens)) * kvd * 2 * e + 2 * B * qd * e,
        "o_proj": H * qd * e + B * qd * e + B * H * (8 + e),
        "gate_up": 2 * F * H * e + B * H * e + B * F * e,
        "down": H * F * e + B * F * e + B * H * (8 + e),
        "lm_head": V * H * e + B * H * e + B * V * 4,
    }


# ---------------------------------------------------------------------------------- oracle leg

def oracle_sample(model, host_k, host_v, meta, rows, bs):
    """Run the oracle on `rows` of one step; returns seconds."""
    import oracle
    tok, pos, tab, sl, slots = meta
    kp = [a.copy() for a in host_k]
    vp = [a.copy() for a in host_v]
    t0 = time.perf_counter()
    oracle.decode_step(model, kp, vp, tok[rows], pos[rows], tab[rows], sl[rows], slots[rows], bs)
    return time.perf_counter() - t0


def host_copy_of(wl):
    """Host copies (storage dtype) of the workload's weights and pools, for the oracle."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib

    def h(t):
        return t.cpu().numpy() if t is not None else None

    w = {"embed": h(wl.w["embed"]), "final_norm": h(wl.w["final_norm"]), "lm_head": None,
         "layers": [{k: h(v) for k, v in lw.items()} for lw in wl.w["layers"]]}
    ks, vs = [], []
    s = wl.shape
    for l in range(s.n_layers):
        k, v = wl.dev.kv_layer_ptrs(l)
        kk = np.empty((wl.num_blocks, s.n_kv_heads, wl.bs, s.head_dim), dtype=np.float16)
        vv = np.empty_like(kk)
        _lib.memcpy(kk.ctypes.data, k, kk.nbytes)
        _lib.memcpy(vv.ctypes.data, v, vv.nbytes)
        ks.append(kk)
        vs.append(vv)
    torch.cuda.synchronize()
    return w, ks, vs


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ---------------------------------------------------------------------------------- attention

def attention_workload(steps: int, warmup: int, batch: int = 256):
    """Paged decode attention alone; returns GB/s and per-launch ms."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    seed = synth.config_seed(2)
    n_q, n_kv, d, bs, nb = 32, 8, 128, 16, 160_000
    ctx = synth.ctx_log_uniform(seed, "cfg2.ctx", batch, 512, 8192)
    need = [int(math.ceil(c / bs)) for c in ctx]
    mb = 512
    perm = synth.permutation(seed, "cfg2.pool", nb)
    tab = np.zeros((batch, mb), dtype=np.int32)
    c = 0
    for b in range(batch):
        tab[b, : need[b]] = perm[c: c + need[b]]
        c += need[b]
    kp = torch.empty((nb, n_kv, bs, d), dtype=torch.bfloat16, device="cuda")
    vp = torch.empty_like(kp)
    stream = torch.cuda.current_stream().cuda_stream
    synth.fill_normal_device(kp.data_ptr(), kp.numel(), seed, "cfg2.k", "bf16", stream=stream)
    synth.fill_normal_device(vp.data_ptr(), vp.numel(), seed, "cfg2.v", "bf16", stream=stream)
    q = synth.normal_device(seed, "cfg2.q", (batch, n_q, d), "bf16")
    out = torch.empty_like(q)
    dt = torch.from_numpy(tab).cuda()
    dl = torch.from_numpy(ctx.astype(np.int32)).cuda()
    scale = 1.0 / math.sqrt(d)

    def launch():
        _lib.attn_decode(q, kp, vp, dt, dl, out, n_q, n_kv, d, bs, mb, nb, scale, "bf16")

    for _ in range(max(warmup, 3)):
        launch()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = max(steps, 10)
    e0.record()
    for _ in range(n):
        launch()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n
    nbytes = rl.attention_bytes(ctx, n_kv, d, 2)
    err = _lib.device_error()
    del kp, vp
    torch.cuda.empty_cache()
    return {"workload": "paged GQA decode attention, batch 256, 32Q/8KV, d128, bf16, "
                        "ctx log-uniform[512,8192], 160k-block pool",
            "gbs": nbytes / (ms * 1e-3) / 1e9, "ms_per_launch": ms, "bytes_per_launch": nbytes,
            "launches": n, "device_error": err}


# ---------------------------------------------------------------------------------- main arms

def read_traffic(kind):
    """Per-launch DRAM bytes from the committed ncu summary, when it matches this kernel."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) >= 2 and parts[0] == kind:
            try:
                return float(parts[1])
            except ValueError:
                return None
    return None


def run_ours(args, rank, world):
    import torch
    import __graft_entry__ as ge
    from transformer_decode_step_ns_gb300 import _lib
    ge.build()
    dev_idx = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev_idx)
    peaks, peaks_src = load_peaks()
    K, W = args.steps, args.warmup
    e2e_steps = max(5, min(K, 50))
    wl = DecodeWorkload(args.batch, total_steps=W + K + e2e_steps + 8)
    log(f"setup {wl.setup_s:.1f}s: {wl.num_blocks} blocks, mb {wl.mb}")

    # warm-up (captures the graph on the first step)
    for _ in range(W):
        wl.step(wl.next_meta())
    torch.cuda.synchronize()
    metas = [wl.next_meta() for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for m in metas:
        wl.step(m)
    e1.record()
    torch.cuda.synchronize()
    ms_total = e0.elapsed_time(e1)
    clk = clocks.stop()
    if world > 1:
        t = torch.tensor([ms_total], device="cuda")
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms_total = float(t.item())
    dev_err = wl.dev.device_error()
    info = wl.dev.info()
    ms_step = ms_total / K
    value = wl.B * K * world / (ms_total * 1e-3)

    # e2e: greedy decode loop through the public API, ids read back every step
    ids_dev = torch.empty(wl.B, dtype=torch.int32, device="cuda")
    ids_host = torch.empty(wl.B, dtype=torch.int32).pin_memory()
    toks = wl.tokens.copy()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        wl.step(wl.next_meta(toks))
        _lib.greedy_argmax(wl.logits, ids_dev)
        ids_host.copy_(ids_dev, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        toks = ids_host.numpy().copy()
    e2e_s = time.perf_counter() - t0
    e2e_value = wl.B * e2e_steps * world / e2e_s

    # per-kernel timing in eager steps (same kernels, same data)
    wl.dev.set_kernel_timing(True)
    for _ in range(3):
        wl.step(wl.next_meta())
    wl.dev.kernel_timing()  # discard the first eager steps
    for _ in range(5):
        wl.step(wl.next_meta())
    kt = wl.dev.kernel_timing()
    wl.dev.set_kernel_timing(False)
    eager_total = sum(v[1] for v in kt.values())
    kb = kernel_bytes(wl.shape, wl.B, metas[-1][3])
    dom = max(kt, key=lambda k: kt[k][1])
    launches, tot_ms = kt[dom]
    avg_ms = tot_ms / launches
    achieved = kb[dom] / (avg_ms * 1e-3) / 1e9
    hbm = float(peaks["hbm_gbs"])
    roof = {"kernel": f"gemm_kernel ({dom})" if dom not in ("attention", "embed_rope") else dom,
            "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
            "frac": achieved / hbm, "traffic": read_traffic(dom),
            "peak_source": "measured hbm_gbs (MEASURED_PEAKS.json)" if peaks_src == "measured"
            else "fallback 6.8 TB/s",
            "bytes_per_launch": kb[dom], "avg_launch_us": avg_ms * 1e3,
            "share_of_eager_step": tot_ms / eager_total,
            "kernel_shares": {k: round(v[1] / eager_total, 4) for k, v in kt.items()},
            "kernel_avg_us": {k: round(v[1] / v[0] * 1e3, 2) for k, v in kt.items()}}

    # whole-step roofline
    work = rl.decode_step_work(wl.shape, metas[-1][3])
    tflops = float(peaks.get("bf16_tflops_sustained", 1700)) * 1e12
    t_roof = rl.step_roofline_time(work.flops, work.total_bytes, tflops, hbm * 1e9)
    step_roof = {"roofline_us": t_roof * 1e6, "measured_us": ms_step * 1e3,
                 "frac": t_roof / (ms_step * 1e-3), "bytes": work.total_bytes,
                 "flops": work.flops,
                 "bound": "hbm" if work.total_bytes / (hbm * 1e9) >= work.flops / tflops
                 else "tensor"}

    attn = None
    if not args.skip_attention and rank == 0:
        attn = attention_workload(max(10, min(K, 50)), W)
        attn["frac_of_hbm"] = attn["gbs"] / hbm

    cpu = None
    if rank == 0 and not args.skip_cpu:
        import oracle
        hw, hk, hv = host_copy_of(wl)
        model = oracle.OracleModel.from_weights(wl.shape, hw)
        rows = np.arange(min(args.cpu_rows, wl.B))
        secs = oracle_sample(model, hk, hv, metas[0], rows, wl.bs)
        cpu = {"value": len(rows) / secs, "unit": "tokens/s", "cores": blas_threads(),
               "kind": "oracle",
               "sample": f"{len(rows)} of the {wl.B} requests through one full step (24 layers + "
                         f"LM head, fp64 numpy), {secs:.1f} s"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "model": "qwen2.5-0.5b-shaped (random init)",
                   "global_batch": wl.B * world, "seq_len": "ctx U[128,1024] + decode",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (988 MB of weights streamed per step)"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": wl.meta_bytes(),
                "d2h_bytes_per_step": wl.B * 4, "steps": e2e_steps,
                "loop": "greedy decode: host metadata upload, step, argmax, ids read back"},
        "roofline": roof,
        "step_roofline": step_roof,
        "attention": attn,
        "cpu_baseline": cpu,
        "clocks": clk,
        "gpu_launches": info.kernels_per_step * K,
        "kernels_per_step": info.kernels_per_step,
        "graph_capture_ms": info.last_capture_ms,
        "device_error": dev_err,
    }
    print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The oracle arm: the fp64 CPU oracle on bounded samples of the same workload."""
    if rank != 0:
        return
    import torch
    import __graft_entry__ as ge
    import oracle
    K, W = args.steps, args.warmup
    rows_per_step = max(1, args.ref_rows)
    if not torch.cuda.is_available():
        print(json.dumps({"impl": "reference", "unavailable":
                          "the seeded inputs are drawn on the GPU; no CUDA device"}))
        return
    ge.build()
    wl = DecodeWorkload(args.batch, total_steps=2)
    meta = wl.next_meta()
    hw, hk, hv = host_copy_of(wl)
    shape, bs, B = wl.shape, wl.bs, wl.B
    del wl
    model = oracle.OracleModel.from_weights(shape, hw)
    times = []
    for i in range(W + K):
        rows = (np.arange(rows_per_step) + i * rows_per_step) % B
        s = oracle_sample(model, hk, hv, meta, rows, bs)
        if i >= W:
            times.append(s)
    total = sum(times)
    value = rows_per_step * K / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": total / K * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "model": "qwen2.5-0.5b-shaped (random init)",
                       "global_batch": B, "seq_len": "ctx U[128,1024] + decode",
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": blas_threads(),
                             "kind": "oracle",
                             "sample": f"{rows_per_step} of {B} requests per step, one full "
                                       f"decode step each (24 layers + LM head, fp64)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--batch", type=int, default=32)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-attention", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=32)
    ap.add_argument("--ref-rows", type=int, default=4)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl" if args.impl == "ours" else "gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    main()
