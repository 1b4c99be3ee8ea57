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
    """nvidia-smi samples every 20 ms; the report keeps the samples taken inside the window
    marked by mark_start() / mark_stop() (host wall clock), else the ones nearest to it."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None
        self.path = None
        self.t0 = self.t1 = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20", "-i", str(self._device_index())],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    @staticmethod
    def _device_index():
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        local = int(os.environ.get("LOCAL_RANK", "0"))
        ids = [v for v in vis.split(",") if v.strip()]
        return ids[local].strip() if local < len(ids) else str(local)

    def has_samples(self) -> bool:
        return self.path is not None and os.path.getsize(self.path) > 0

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        import datetime
        samples = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((ts, float(parts[2]), float(parts[3]), parts[6:10]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        inside = [x for x in samples if self.t0 is not None and self.t0 <= x[0] <= self.t1]
        where = "inside the timed region"
        if not inside:
            # the region was shorter than the sampling period: the nearest samples either side
            mid = 0.5 * (self.t0 + self.t1) if self.t0 is not None else samples[-1][0]
            inside = sorted(samples, key=lambda x: abs(x[0] - mid))[:2]
            where = "nearest the timed region (shorter than the sampling period)"
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = set()
        for x in inside:
            for n, v in zip(names, x[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median([x[1] for x in inside])),
                "sm_max_mhz": float(max(x[2] for x in inside)),
                "samples": len(inside), "where": where, "reasons": sorted(reasons)}


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

class AttentionWorkload:
    """Paged decode attention alone: 32 Q / 8 KV heads, head_dim 128, bf16, block size 16,
    contexts log-uniform in [512, 8192], block tables drawn from a shuffled pool.

    Contexts are drawn for `max_batch` rows by index, so batch B uses the first B of them and
    batch 256 is the same input at any `max_batch`."""

    n_q, n_kv, d, bs, mb = 32, 8, 128, 16, 512

    def __init__(self, max_batch: int = 512, pool_blocks: int = 160_000):
        import torch
        seed = synth.config_seed(2)
        self.ctx = synth.ctx_log_uniform(seed, "cfg2.ctx", max_batch, 512, 8192)
        need = [int(math.ceil(c / self.bs)) for c in self.ctx]
        nb = max(pool_blocks, sum(need) + 1)
        self.nb = nb
        perm = synth.permutation(seed, "cfg2.pool", nb)
        tab = np.zeros((max_batch, self.mb), dtype=np.int32)
        c = 0
        for b in range(max_batch):
            tab[b, : need[b]] = perm[c: c + need[b]]
            c += need[b]
        self.kp = torch.empty((nb, self.n_kv, self.bs, self.d), dtype=torch.bfloat16,
                              device="cuda")
        self.vp = torch.empty_like(self.kp)
        stream = torch.cuda.current_stream().cuda_stream
        synth.fill_normal_device(self.kp.data_ptr(), self.kp.numel(), seed, "cfg2.k", "bf16",
                                 stream=stream)
        synth.fill_normal_device(self.vp.data_ptr(), self.vp.numel(), seed, "cfg2.v", "bf16",
                                 stream=stream)
        self.q = synth.normal_device(seed, "cfg2.q", (max_batch, self.n_q, self.d), "bf16")
        self.out = torch.empty_like(self.q)
        self.tab = torch.from_numpy(tab).cuda()
        self.lens = torch.from_numpy(self.ctx.astype(np.int32)).cuda()
        # a buffer larger than L2 (129 MB): writing it between launches evicts the K/V
        self.flush_buf = torch.empty(64 << 20, dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()

    def launch(self, B):
        from transformer_decode_step_ns_gb300 import _lib
        _lib.attn_decode(self.q[:B], self.kp, self.vp, self.tab[:B], self.lens[:B],
                         self.out[:B], self.n_q, self.n_kv, self.d, self.bs, self.mb, self.nb,
                         1.0 / math.sqrt(self.d), "bf16")

    def nbytes(self, B):
        return rl.attention_bytes(self.ctx[:B], self.n_kv, self.d, 2)

    def back_to_back(self, B, n, warmup):
        """Mean launch time of n launches in a row (only valid when the K/V exceed L2)."""
        import torch
        for _ in range(max(warmup, 3)):
            self.launch(B)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            self.launch(B)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    def flushed(self, B, n, warmup):
        """Mean launch time with L2 flushed before every launch (event pair per launch)."""
        import torch
        for _ in range(max(warmup, 3)):
            self.launch(B)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            self.flush_buf.zero_()
            a.record()
            self.launch(B)
            b.record()
        torch.cuda.synchronize()
        return sum(a.elapsed_time(b) for a, b in ev) / n

    def report(self, B, steps, warmup, hbm):
        ms = self.back_to_back(B, max(steps, 10), warmup)
        nbytes = self.nbytes(B)
        return {"workload": f"paged GQA decode attention, batch {B}, 32Q/8KV, d128, bf16, "
                            f"ctx log-uniform[512,8192], {self.nb}-block pool",
                "gbs": nbytes / (ms * 1e-3) / 1e9, "ms_per_launch": ms,
                "bytes_per_launch": nbytes, "launches": max(steps, 10),
                "frac_of_hbm": nbytes / (ms * 1e-3) / 1e9 / hbm,
                "l2": "K/V read per launch larger than L2, launches back to back"}

    def sweep(self, batches, hbm, n=10):
        rows = []
        for B in batches:
            ms = self.flushed(B, n, 3)
            nbytes = self.nbytes(B)
            rows.append({"batch": B, "us": round(ms * 1e3, 2), "bytes": nbytes,
                         "gbs": round(nbytes / (ms * 1e-3) / 1e9, 1),
                         "frac_of_hbm": round(nbytes / (ms * 1e-3) / 1e9 / hbm, 4)})
        return rows


SWEEP_BATCHES = [1, 2, 4, 8, 16, 32, 64, 128, 256, 512]


# ---------------------------------------------------------------------------------- nano-batches

class NanoLayerWorkload:
    """One LLaMA-2-70B-shaped layer (hidden 8192, 64 Q / 8 KV heads, head_dim 128, SwiGLU 28672,
    bf16, seeded N(0, 0.02) weights) over a dense batch of 2048 rows: 1024 decode requests with
    contexts uniform in [256, 2048], then one 1024-token prefill chunk as pseudo-requests
    (positions 0..1023 over one shared block table, each row attending to its prefix).  The
    step stops after the layer (no LM head).  The nano-batch split and attention CTA budget are
    chosen by the tuner (a pairwise attention/GEMM interference profile, then every split in
    multiples of 128 timed, then CTA budgets on the fastest splits)."""

    LABELS = {"1": [2048], "2": [1024, 1024], "2 uneven": [768, 1280], "3": [640, 640, 768],
              "4": [512, 512, 512, 512]}

    def __init__(self):
        import dataclasses
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        seed = synth.config_seed(3)
        # the vocabulary only feeds the embedding gather: tie it so no head is allocated
        self.shape = dataclasses.replace(synth.llama2_70b_layer_shape(), tie_embeddings=True)
        sh = self.shape
        self.bs = bs = 16
        n_dec, n_pre = 1024, 1024
        self.B = B = n_dec + n_pre
        self.w = synth.model_weights_device(sh, seed)
        ctx_dec = synth.ctx_uniform(seed, "cfg3.ctx", n_dec, 256, 2048).astype(np.int64)
        pos = np.concatenate([ctx_dec, np.arange(n_pre, dtype=np.int64)])
        self.mb = mb = int(math.ceil((ctx_dec.max() + 1) / bs))
        need_dec = [int(math.ceil((c + 1) / bs)) for c in ctx_dec]
        chunk_blocks = int(math.ceil(n_pre / bs))
        self.num_blocks = sum(need_dec) + chunk_blocks + 16
        self.dev = _lib.DecodeStep(sh, self.w, B, mb, use_graphs=True)
        self.dev.kv_alloc(self.num_blocks, bs)
        ids = self.dev.reserve(self.num_blocks)
        self.dev.release(ids[synth.permutation(seed, "cfg3.pool", self.num_blocks)])
        tab = np.zeros((B, mb), dtype=np.int32)
        for b in range(n_dec):
            tab[b, :need_dec[b]] = self.dev.reserve(need_dec[b])
        tab[n_dec:, :chunk_blocks] = self.dev.reserve(chunk_blocks)[None, :]
        stream = torch.cuda.current_stream().cuda_stream
        k, v = self.dev.kv_layer_ptrs(0)
        n = self.dev.kv_pool_bytes() // 2
        synth.fill_normal_device(k, n, seed, "cfg3.k0", "bf16", stream=stream)
        synth.fill_normal_device(v, n, seed, "cfg3.v0", "bf16", stream=stream)
        torch.cuda.synchronize()
        blk = tab[np.arange(B), pos // bs].astype(np.int64)
        self.meta = (synth.uniform_int(seed, "cfg3.tokens", B, 0, sh.vocab - 1).astype(np.int32),
                     pos.astype(np.int32), tab, (pos + 1).astype(np.int32), blk * bs + pos % bs)
        self.ctx_dec, self.n_pre = ctx_dec, n_pre

    def work(self):
        """Algorithmic FLOPs and bytes of the layer step (chunk K/V counted once)."""
        sh = self.shape
        h, f, d = sh.hidden, sh.ffn, sh.head_dim
        qd, kvd = sh.n_q_heads * d, sh.n_kv_heads * d
        lin = h * qd + 2 * h * kvd + qd * h + 3 * h * f
        seq = self.meta[3].astype(np.float64)
        flops = 2.0 * self.B * lin + 4.0 * qd * seq.sum()
        weights = (lin + 2 * h) * 2
        kv = (float((self.ctx_dec + 1).sum()) + self.n_pre) * 2 * kvd * 2
        kv_write = self.B * 2 * kvd * 2
        return flops, weights + kv + kv_write

    def time_variant(self, sizes, budget, steps, warmup):
        import torch
        self.dev.set_nanobatch(sizes, attn_cta_budget=budget)
        for _ in range(max(warmup, 3)):
            self.dev.step(*self.meta, None)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            self.dev.step(*self.meta, None)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    def serial_kernels(self):
        """Per-kind kernel time per step (µs) of the unsplit step, launched eagerly with an event
        pair around each launch (attention: the decode rows' and the chunk's kernels)."""
        self.dev.set_nanobatch(None)
        self.dev.set_kernel_timing(True)
        self.dev.step(*self.meta, None)
        self.dev.kernel_timing()
        steps = 3
        for _ in range(steps):
            self.dev.step(*self.meta, None)
        kt = self.dev.kernel_timing()
        self.dev.set_kernel_timing(False)
        return {k: round(v[1] / steps * 1e3, 1) for k, v in kt.items() if v[0]}

    def interference(self, reps=10):
        """R -> P of the decode rows' attention (capped at 8..128 CTAs) co-running with the
        gate projection of a 1024-row nano-batch (tuner.pair_profile)."""
        import torch
        from transformer_decode_step_ns_gb300 import _lib, tuner
        sh, bs = self.shape, self.bs
        n_dec = len(self.ctx_dec)
        tab = torch.from_numpy(self.meta[2][:n_dec].copy()).cuda()
        lens = torch.from_numpy(self.meta[3][:n_dec].copy()).cuda()
        q = torch.randn((n_dec, sh.n_q_heads * sh.head_dim), device="cuda").to(torch.bfloat16)
        out = torch.empty_like(q)
        k, v = self.dev.kv_layer_ptrs(0)
        wg = self.w["layers"][0]["w_gate"]
        x = torch.randn((1024, sh.hidden), device="cuda").to(torch.bfloat16)
        y = torch.empty((1024, sh.ffn), dtype=torch.float32, device="cuda")

        def attn(budget, stream):
            _lib.attn_decode(q, k, v, tab, lens, out, sh.n_q_heads, sh.n_kv_heads, sh.head_dim, bs,
                             self.mb, self.num_blocks, 1.0 / math.sqrt(sh.head_dim), "bf16",
                             stream=stream, cta_budget=budget)

        def gemm(stream):
            _lib.linear(wg, x, y, 1024, sh.ffn, sh.hidden, "bf16", stream=stream)

        prof = tuner.pair_profile(attn, gemm, reps=reps)
        prof["pair"] = (f"decode attention of the 1024 decode rows against the gate projection "
                        f"of 1024 rows ({sh.ffn} x {sh.hidden})")
        return prof

    def report(self, steps, warmup, peaks, tune=True):
        from transformer_decode_step_ns_gb300 import _lib, tuner
        flops, nbytes = self.work()
        tflops = float(peaks.get("bf16_tflops_sustained", 1700)) * 1e12
        hbm = float(peaks["hbm_gbs"]) * 1e9
        t_roof = rl.step_roofline_time(flops, nbytes, tflops, hbm)
        if not tune:  # the named splits only (a short command for profilers)
            rows = []
            for label, sizes in self.LABELS.items():
                ms = self.time_variant(None if len(sizes) == 1 else sizes, 0, steps, warmup)
                rows.append({"split": label, "sizes": sizes, "attn_cta_budget": 0,
                             "us": round(ms * 1e3, 1),
                             "frac_of_roofline": round(t_roof / (ms * 1e-3), 4)})
            best = min(rows, key=lambda r: r["us"])
            return {"workload": "LLaMA-2-70B-shaped layer, bf16, 1024 decode rows + 1024-token "
                                "prefill chunk, graph replay, no LM head (named splits, untuned)",
                    "roofline_us": round(t_roof * 1e6, 1), "variants": rows,
                    "tuned": {"sizes": best["sizes"], "attn_cta_budget": 0, "us": best["us"],
                              "frac_of_roofline": best["frac_of_roofline"]},
                    "device_error": _lib.device_error()}
        prof = self.interference()

        def step(sizes, budget):
            self.dev.set_nanobatch(sizes, attn_cta_budget=budget)
            self.dev.step(*self.meta, None)

        found = tuner.search(step, self.B, profile=prof, reps=max(3, min(steps, 10)))
        for r in found["table"]:
            r["frac_of_roofline"] = round(t_roof / (r["ms"] * 1e-3), 4)
        rows = []
        for label, sizes in self.LABELS.items():
            r = next(t for t in found["table"] if t["sizes"] == sizes and t["budget"] == 0)
            rows.append({"split": label, "sizes": sizes, "attn_cta_budget": 0,
                         "us": round(r["ms"] * 1e3, 1),
                         "tflops": round(flops / (r["ms"] * 1e-3) / 1e12, 1),
                         "frac_of_roofline": r["frac_of_roofline"]})
        best = found["best"]
        # the tuned configuration, timed again over the full step count
        ms = self.time_variant(None if len(best["sizes"]) == 1 else best["sizes"], best["budget"],
                               steps, warmup)
        tuned = {"sizes": best["sizes"], "attn_cta_budget": best["budget"], "us": round(ms * 1e3, 1),
                 "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
                 "frac_of_roofline": round(t_roof / (ms * 1e-3), 4)}
        self.dev.set_nanobatch(None)
        serial = self.serial_kernels()
        return {"workload": "LLaMA-2-70B-shaped layer, bf16, 1024 decode rows (ctx U[256,2048]) "
                            "+ 1024-token prefill chunk, graph replay, no LM head",
                "flops": flops, "bytes": nbytes, "roofline_us": round(t_roof * 1e6, 1),
                "bound": "tensor" if flops / tflops >= nbytes / hbm else "hbm",
                "tuned": tuned, "variants": rows, "interference": prof,
                "search": {"candidates": len(found["table"]), "budgets_kept": found["budgets_kept"],
                           "table": found["table"]},
                "serial_kernel_us": serial, "device_error": _lib.device_error()}


# ---------------------------------------------------------------------------------- continuous run

class ContinuousWorkload:
    """Continuous-batching decode of a 32-layer LLaMA-3-8B-shaped model (hidden 4096, 32 Q / 8
    KV heads, head_dim 128, SwiGLU 14336, vocab 128256, untied head, bf16, seeded N(0, 0.02)
    weights) at a constant batch of 256 requests.

    Every request starts with a context uniform in [512, 4096] (its K/V preloaded N(0, 1)) and
    decodes a length uniform in [100, 1000]; when it finishes it leaves (its blocks return to
    the pool) and a new request joins in its row.  Each step: join/leave bookkeeping and the
    host slot mapper, one ns_decode_step (graph replay), greedy argmax on the GPU and the ids
    read back to the host as the next tokens."""

    B, bs, ctx_lo, ctx_hi, dec_lo, dec_hi = 256, 16, 512, 4096, 100, 1000

    def __init__(self, max_joins: int = 100_000):
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        self.seed = seed = synth.config_seed(4)
        self.shape = sh = synth.llama3_8b_shape(32)
        B, bs = self.B, self.bs
        self.mb = mb = int(math.ceil((self.ctx_hi + self.dec_hi + 1) / bs))
        self.num_blocks = B * mb
        t0 = time.time()
        self.w = synth.model_weights_device(sh, seed)
        self.dev = _lib.DecodeStep(sh, self.w, B, mb, use_graphs=True)
        self.w = None  # the library holds its own copy
        torch.cuda.empty_cache()
        self.dev.kv_alloc(self.num_blocks, bs)
        ids = self.dev.reserve(self.num_blocks)
        self.dev.release(ids[synth.permutation(seed, "cfg4.pool", self.num_blocks)])
        stream = torch.cuda.current_stream().cuda_stream
        n = self.dev.kv_pool_bytes() // 2
        for l in range(sh.n_layers):
            k, v = self.dev.kv_layer_ptrs(l)
            synth.fill_normal_device(k, n, seed, f"cfg4.k{l}", "bf16", stream=stream)
            synth.fill_normal_device(v, n, seed, f"cfg4.v{l}", "bf16", stream=stream)
        torch.cuda.synchronize()
        # per-join draws, indexed by join number
        self.j_ctx = synth.ctx_uniform(seed, "cfg4.join.ctx", max_joins, self.ctx_lo, self.ctx_hi)
        self.j_len = synth.uniform_int(seed, "cfg4.join.len", max_joins, self.dec_lo, self.dec_hi)
        self.joins = 0
        self.tables = np.zeros((B, mb), dtype=np.int32)
        self.pos = np.zeros(B, dtype=np.int32)
        self.left = np.zeros(B, dtype=np.int64)
        for b in range(B):
            self.join(b)
        self.tokens = synth.uniform_int(seed, "cfg4.tokens", B, 0, sh.vocab - 1).astype(np.int32)
        self.logits = torch.empty((B, sh.vocab), dtype=torch.float32, device="cuda")
        self.setup_s = time.time() - t0

    def join(self, b):
        c = int(self.j_ctx[self.joins])
        self.left[b] = int(self.j_len[self.joins])
        self.joins += 1
        n = int(math.ceil(c / self.bs))
        self.tables[b] = 0
        self.tables[b, :n] = self.dev.reserve(n)
        self.pos[b] = c

    def leave(self, b):
        n = int(math.ceil(self.pos[b] / self.bs))
        self.dev.release(self.tables[b, :n].copy())

    def run(self, steps, peaks, nano=None):
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        self.dev.set_nanobatch(nano)
        ids_dev = torch.empty(self.B, dtype=torch.int32, device="cuda")
        ids_host = torch.empty(self.B, dtype=torch.int32).pin_memory()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        t_roof = 0.0
        tflops = float(peaks.get("bf16_tflops_sustained", 1700)) * 1e12
        hbm = float(peaks["hbm_gbs"]) * 1e9
        leaves = 0
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(steps):
            slots = self.dev.prepare_step(self.pos, self.tables)
            seq = self.pos + 1
            work = rl.decode_step_work(self.shape, seq)
            t_roof += rl.step_roofline_time(work.flops, work.total_bytes, tflops, hbm)
            ev[i][0].record()
            self.dev.step(self.tokens, self.pos, self.tables, seq, slots, self.logits)
            ev[i][1].record()
            _lib.greedy_argmax(self.logits, ids_dev)
            ids_host.copy_(ids_dev, non_blocking=True)
            torch.cuda.current_stream().synchronize()
            self.tokens = ids_host.numpy().copy()
            self.pos += 1
            self.left -= 1
            for b in np.nonzero(self.left == 0)[0]:
                self.leave(int(b))
                self.join(int(b))
                leaves += 1
        wall = time.perf_counter() - t0
        dev_ms = np.array([a.elapsed_time(b) for a, b in ev])
        return {"steps": steps, "nano_split": nano or [self.B], "leaves_and_joins": leaves,
                "device_ms_per_step_mean": float(dev_ms.mean()),
                "device_ms_per_step_median": float(np.median(dev_ms)),
                "tokens_per_s_device": self.B * steps / (dev_ms.sum() * 1e-3),
                "tokens_per_s_e2e": self.B * steps / wall,
                "roofline_ms_per_step_mean": t_roof / steps * 1e3,
                "frac_of_roofline": t_roof / (dev_ms.sum() * 1e-3),
                "graphs_cached": self.dev.info().graphs_cached,
                "device_error": self.dev.device_error()}

    def offload(self, steps, peaks, nano):
        """KV offload: steps with every step's new K/V mirrored to pinned host memory (each
        layer's rows copied while its attention and FFN run) against the same steps without;
        then the longest request saved to the host and reloaded into its blocks (contiguous
        transfer + device scatter), against plain copies of the same bytes."""
        import torch
        sh = self.shape
        row = 2 * sh.n_kv_heads * sh.head_dim
        mirror = torch.empty((sh.n_layers, self.B, row), dtype=torch.int16).pin_memory()
        self.dev.set_kv_offload(mirror)
        on = self.run(steps, peaks, nano)
        self.dev.set_kv_offload(None)
        off = self.run(steps, peaks, nano)
        b = int(np.argmax(self.pos))
        n = int(self.pos[b])
        tab = self.tables[b, :int(math.ceil(n / self.bs))].copy()
        host = torch.empty((sh.n_layers, n, row), dtype=torch.int16).pin_memory()
        dev_buf = torch.empty_like(host, device="cuda")
        nbytes = host.numel() * 2

        def timed(fn, reps=5):
            fn()
            torch.cuda.synchronize()
            a, z = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            z.record()
            torch.cuda.synchronize()
            return a.elapsed_time(z) / reps

        save_ms = timed(lambda: self.dev.kv_save(host, n, 0, tab))
        reload_ms = timed(lambda: self.dev.kv_reload(host, n, 0, tab))  # same bits, same blocks
        d2h_ms = timed(lambda: host.copy_(dev_buf, non_blocking=True))
        h2d_ms = timed(lambda: dev_buf.copy_(host, non_blocking=True))
        return {"mirror_bytes_per_step": sh.n_layers * self.B * row * 2,
                "ms_per_step_mirror_on": round(on["device_ms_per_step_median"], 3),
                "ms_per_step_mirror_off": round(off["device_ms_per_step_median"], 3),
                "request_tokens": n, "request_bytes": nbytes,
                "save_ms": round(save_ms, 3), "reload_ms": round(reload_ms, 3),
                "plain_d2h_ms": round(d2h_ms, 3), "plain_h2d_ms": round(h2d_ms, 3),
                "reload_gbs": round(nbytes / reload_ms * 1e-6, 1),
                "plain_h2d_gbs": round(nbytes / h2d_ms * 1e-6, 1),
                "device_error": self.dev.device_error()}

    def report(self, steps, peaks):
        # a short comparison of the nano-batch splits, then the full run with the faster one
        trial = {}
        for nano in (None, [128, 128]):
            trial[str(nano or [self.B])] = self.run(20, peaks, nano)["device_ms_per_step_median"]
        best = None if trial[str([self.B])] <= trial[str([128, 128])] else [128, 128]
        r = self.run(steps, peaks, best)
        r["split_trial_ms_per_step"] = trial
        # per-kind kernel time of eager steps (an event pair around each launch)
        self.dev.set_kernel_timing(True)
        self.run(2, peaks, best)
        self.dev.kernel_timing()
        self.run(3, peaks, best)
        kt = self.dev.kernel_timing()
        self.dev.set_kernel_timing(False)
        r["eager_kernel_us"] = {k: round(v[1] / v[0] * 1e3, 1) for k, v in kt.items() if v[0]}
        r["eager_kernel_launches_per_step"] = {k: v[0] // 3 for k, v in kt.items() if v[0]}
        r["kv_offload"] = self.offload(30, peaks, best)
        r["workload"] = ("LLaMA-3-8B-shaped 32L bf16, batch 256, ctx U[512,4096], decode lengths "
                         "U[100,1000] with leave/join, greedy argmax fed back, graph replay")
        r["setup_s"] = round(self.setup_s, 1)
        return r


# ---------------------------------------------------------------------------------- serving run

class ServingWorkload:
    """Constant-dense-batch serving of the 32-layer LLaMA-3-8B-shaped model (bf16, seeded
    N(0, 0.02) weights): 256 requests arrive at once with seeded prompts of lengths uniform in
    [128, 1024] and decode lengths uniform in [64, 256].  The library's batch former (ns_sched)
    forms every step at 512 tokens -- decode rows first, then prompt chunks at token granularity
    -- admitting prompts against their peak memory from a pool of 25 % of the requests' summed
    peaks, so prompts and decodes interleave as requests finish.  Steps with prompt chunks
    launch eagerly (their layouts vary); decode-only steps replay graphs padded to buckets of 64.
    Greedy argmax on the GPU; ids read back each step.  Run twice: with every prompt's full peak
    reserved at admission, and with peaks predicted from a decode length of 16, where requests
    that outgrow the pool are saved to pinned host memory and reloaded later."""

    D, n_req, bs = 512, 256, 16

    def __init__(self):
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        self.seed = seed = synth.config_seed(4)
        self.shape = sh = synth.llama3_8b_shape(32)
        n, bs = self.n_req, self.bs
        self.plen = synth.uniform_int(seed, "serve.plen", n, 128, 1024).astype(np.int64)
        self.new = synth.uniform_int(seed, "serve.new", n, 64, 256).astype(np.int64)
        self.mb = int(math.ceil((1024 + 256) / bs))
        peaks = sum(int(math.ceil((p + m - 1) / bs)) for p, m in zip(self.plen, self.new))
        self.num_blocks = int(0.25 * peaks)
        t0 = time.time()
        w = synth.model_weights_device(sh, seed)
        self.dev = _lib.DecodeStep(sh, w, self.D, self.mb, use_graphs=True)
        del w
        torch.cuda.empty_cache()
        self.dev.kv_alloc(self.num_blocks, bs)
        self.dev.set_graph_chunks(False)
        self.dev.set_graph_buckets(list(range(64, self.D + 1, 64)))
        self.prompts = [synth.uniform_int(seed, f"serve.prompt{i}", int(self.plen[i]), 0,
                                          sh.vocab - 1).astype(np.int32) for i in range(n)]
        self.setup_s = time.time() - t0

    def report(self):
        out = {"reserved_peaks": self.run(0), "predicted_peaks": self.run(16),
               "reserved_peaks_async": self.run(0, async_mode=True)}
        out.update({"workload": out["reserved_peaks"].pop("workload"), "num_blocks": self.num_blocks,
                    "setup_s": round(self.setup_s, 1)})
        out["predicted_peaks"].pop("workload")
        out["reserved_peaks_async"].pop("workload")
        return out

    def run(self, predicted_new, async_mode=False):
        """One pass over the requests.  Asynchronous: step k + 1 is formed and launched before
        step k's ids reach the host (its decode rows read them from the device argmax), and step
        k is committed after that launch, so the host's work overlaps the GPU's."""
        import collections
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        sh, D = self.shape, self.D
        former = _lib.BatchFormer(self.dev.pool(), D, self.mb, eos_token=-1,
                                  predicted_new_tokens=predicted_new)
        former.set_async(async_mode)
        for i in range(self.n_req):
            former.add(i, self.prompts[i], int(self.new[i]))
        store, inflight, saves, moved = {}, [], 0, 0
        logits = torch.empty((D, sh.vocab), dtype=torch.float32, device="cuda")
        ids_dev = torch.zeros(D, dtype=torch.int32, device="cuda")
        self.dev.set_token_source(ids_dev if async_mode else None)
        ids_host = [torch.empty(D, dtype=torch.int32).pin_memory() for _ in range(2)]
        done_ev = [torch.cuda.Event() for _ in range(2)]
        pending = collections.deque()
        rows_per_step, kinds, dev_ms = [], [], []
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        k = 0
        while former.counts()[3] < self.n_req:
            r = former.next()
            for kind, rid, n, table in former.moves():
                if kind == 0:  # preempted: its cached K/V go to pinned host memory
                    buf = torch.empty((sh.n_layers, n, self.dev.kv_row_elems()),
                                      dtype=torch.int16).pin_memory()
                    self.dev.kv_save(buf, n, 0, table)
                    store[rid] = buf
                    saves += 1
                else:          # resumed: reloaded into its new blocks before the step
                    buf = store.pop(rid)
                    self.dev.kv_reload(buf, n, 0, table)
                    inflight.append(buf)
                moved += n * sh.n_layers * self.dev.kv_row_elems() * 2
            B = len(r["token_ids"])
            if B == 0 and not pending:
                raise RuntimeError("the former formed an empty step with requests unfinished")
            if B:
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                self.dev.step(r["token_ids"], r["positions"], r["block_tables"], r["seq_lens"],
                              r["slot_mapping"], logits[:B])
                b.record()
                _lib.greedy_argmax(logits[:B], ids_dev[:B])
                ids_host[k % 2][:B].copy_(ids_dev[:B], non_blocking=True)
                dev_ms.append((a, b))
            done_ev[k % 2].record()
            pending.append((k % 2, B))
            k += 1
            if len(pending) == (2 if async_mode else 1):
                j, nb = pending.popleft()
                done_ev[j].synchronize()
                inflight.clear()
                former.commit(ids_host[j][:nb].numpy())
            if B == 0:
                continue
            rows_per_step.append(B)
            kinds.append("decode" if int(r["row_samples"].sum()) == B else "mixed")
        while pending:
            j, nb = pending.popleft()
            done_ev[j].synchronize()
            former.commit(ids_host[j][:nb].numpy())
        wall = time.perf_counter() - t0
        self.dev.set_token_source(None)
        dev_ms = np.array([a.elapsed_time(b) for a, b in dev_ms])
        kinds = np.array(kinds)
        rows = np.array(rows_per_step)
        out_tok = int(self.new.sum())
        all_tok = int(self.plen.sum() + self.new.sum() - self.n_req)  # rows fed: prompts + all but the last token
        return {"workload": ("LLaMA-3-8B-shaped 32L bf16, 256 requests (prompts U[128,1024], decode "
                             "U[64,256]), dense batch 512 tokens formed by ns_sched, pool 25% of "
                             "summed peaks, mixed steps eager, decode-only steps graph-replayed"),
                "steps": int(len(rows)), "wall_s": round(wall, 3),
                "output_tokens": out_tok, "prompt_tokens": int(self.plen.sum()),
                "output_tokens_per_s": round(out_tok / wall, 1),
                "rows_per_s": round(all_tok / wall, 1),
                "rows_per_step_mean": round(float(rows.mean()), 1),
                "steps_at_dense_size": round(float((rows == D).mean()), 4),
                "mixed_steps": int((kinds == "mixed").sum()),
                "device_ms_per_step_mixed": round(float(dev_ms[kinds == "mixed"].mean()), 3)
                if (kinds == "mixed").any() else None,
                "device_ms_per_step_decode": round(float(dev_ms[kinds == "decode"].mean()), 3)
                if (kinds == "decode").any() else None,
                "device_busy_frac": round(float(dev_ms.sum() * 1e-3 / wall), 4),
                "predicted_new_tokens": predicted_new, "asynchronous_formation": async_mode,
                "preemptions": saves,
                "kv_moved_bytes": moved,
                "graphs_cached": self.dev.info().graphs_cached,
                "device_error": self.dev.device_error()}


# ---------------------------------------------------------------------------------- KV transfers

class OffloadWorkload:
    """KV save and reload of one 4096-token request with the LLaMA-3-8B KV geometry (32 layers,
    8 KV heads, head_dim 128, bf16: 512 MiB of K/V rows), through a handle whose dense weights
    are small (hidden 1024, 8 Q heads, FFN 1024, vocab 1024) since only the cache is touched.
    The request's 256 blocks are a seeded permutation of a 1024-block pool.  Times, with CUDA
    events: ns_kv_save (gather kernel + one D2H copy) and ns_kv_reload (one H2D copy + scatter
    kernel) from pinned memory, and plain copies of the same bytes."""

    n_tok, bs = 4096, 16

    def __init__(self):
        import dataclasses
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        seed = synth.config_seed(4)
        sh = dataclasses.replace(synth.llama3_8b_shape(32), hidden=1024, n_q_heads=8, ffn=1024,
                                 vocab=1024, tie_embeddings=True)
        self.shape = sh
        nblk = self.n_tok // self.bs
        self.num_blocks = 4 * nblk
        w = synth.model_weights_device(sh, seed)
        self.dev = _lib.DecodeStep(sh, w, 1, nblk + 1, use_graphs=False)
        del w
        self.dev.kv_alloc(self.num_blocks, self.bs)
        stream = torch.cuda.current_stream().cuda_stream
        n = self.dev.kv_pool_bytes() // 2
        for l in range(sh.n_layers):
            k, v = self.dev.kv_layer_ptrs(l)
            synth.fill_normal_device(k, n, seed, f"off.k{l}", "bf16", stream=stream)
            synth.fill_normal_device(v, n, seed, f"off.v{l}", "bf16", stream=stream)
        self.table = synth.permutation(seed, "off.table", self.num_blocks)[:nblk].astype(np.int32)
        self.host = torch.empty((sh.n_layers, self.n_tok, self.dev.kv_row_elems()),
                                dtype=torch.int16).pin_memory()
        torch.cuda.synchronize()

    def report(self, reps=5):
        import torch
        nbytes = self.host.numel() * 2
        dev_buf = torch.empty_like(self.host, device="cuda")

        def timed(fn):
            fn()
            torch.cuda.synchronize()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            for _ in range(reps):
                fn()
            b.record()
            torch.cuda.synchronize()
            return a.elapsed_time(b) / reps

        save = timed(lambda: self.dev.kv_save(self.host, self.n_tok, 0, self.table))
        reload = timed(lambda: self.dev.kv_reload(self.host, self.n_tok, 0, self.table))
        d2h = timed(lambda: self.host.copy_(dev_buf, non_blocking=True))
        h2d = timed(lambda: dev_buf.copy_(self.host, non_blocking=True))
        return {"workload": "KV save/reload of one 4096-token request, 32 layers x 8 KV heads x d128 "
                            "bf16 (512 MiB of rows), 256 permuted blocks of a 1024-block pool, "
                            "pinned host memory",
                "bytes": nbytes, "save_ms": round(save, 3), "reload_ms": round(reload, 3),
                "plain_d2h_ms": round(d2h, 3), "plain_h2d_ms": round(h2d, 3),
                "save_gbs": round(nbytes / save * 1e-6, 1), "reload_gbs": round(nbytes / reload * 1e-6, 1),
                "plain_h2d_gbs": round(nbytes / h2d * 1e-6, 1), "plain_d2h_gbs": round(nbytes / d2h * 1e-6, 1),
                "device_error": self.dev.device_error()}


# ---------------------------------------------------------------------------------- projections alone

class GemmWorkload:
    """The LLaMA-3-8B projections alone through ns_linear (the step's GEMM kernel with a plain
    fp32 epilogue) at `rows` rows: QKV 6144 x 4096, O 4096 x 4096, gate/up 28672 x 4096, down
    4096 x 14336, bf16 weights N(0, 0.02) and activations N(0, 1) from the seed.  Each launch is
    timed alone with CUDA events after a write of 256 MiB that flushes L2; the median of `reps`."""

    SHAPES = {"qkv": (6144, 4096), "o": (4096, 4096), "gate_up": (28672, 4096), "down": (4096, 14336)}

    def __init__(self, rows):
        import torch
        self.rows = rows
        seed = synth.config_seed(4)
        self.w = {k: synth.normal_device(seed, f"gemm.{k}", (n, kk), "bf16", std=0.02)
                  for k, (n, kk) in self.SHAPES.items()}
        self.x = {k: synth.normal_device(seed, f"gemm.x.{k}", (rows, kk), "bf16")
                  for k, (n, kk) in self.SHAPES.items()}
        self.y = {k: torch.empty((rows, n), dtype=torch.float32, device="cuda")
                  for k, (n, kk) in self.SHAPES.items()}
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def report(self, peaks, reps=20):
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        tflops = float(peaks.get("bf16_tflops", 1900)) * 1e12
        hbm = float(peaks["hbm_gbs"]) * 1e9
        out = {}
        for k, (n, kk) in self.SHAPES.items():
            m = self.rows
            for _ in range(3):
                _lib.linear(self.w[k], self.x[k], self.y[k], m, n, kk, "bf16")
            ts = []
            for _ in range(reps):
                self.flush.zero_()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record()
                _lib.linear(self.w[k], self.x[k], self.y[k], m, n, kk, "bf16")
                b.record()
                torch.cuda.synchronize()
                ts.append(a.elapsed_time(b) * 1e-3)
            t = float(np.median(ts))
            flops = 2.0 * m * n * kk
            nbytes = n * kk * 2 + m * kk * 2 + m * n * 4
            roof = max(flops / tflops, nbytes / hbm)
            out[k] = {"us": round(t * 1e6, 1), "tflops": round(flops / t / 1e12, 1),
                      "gbs": round(nbytes / t / 1e9, 1), "roofline_us": round(roof * 1e6, 1),
                      "bound": "tensor" if flops / tflops >= nbytes / hbm else "hbm",
                      "frac_of_roofline": round(roof / t, 4)}
        return {"workload": f"LLaMA-3-8B projections alone at {self.rows} rows, bf16, L2 flushed "
                            "before each launch (peaks: burst bf16, HBM copy)",
                "projections": out, "device_error": _lib.device_error()}


# ---------------------------------------------------------------------------------- main arms

KERNEL_SOURCE = {"embed_rope": "k_misc.cu", "attention": "k_attn.cu", "qkv": "k_gemm.cu",
                 "o_proj": "k_gemm.cu", "gate_up": "k_gemm.cu", "down": "k_gemm.cu",
                 "lm_head": "k_gemm.cu", "prefill": "k_prefill.cu", "kv_copy": "k_misc.cu"}


def kernel_source_hash(kind):
    """sha256 (first 16 hex digits) of the device code of the kernel's source file (the text
    before its "host side" marker: launchers and launch-shape choices after it do not change
    what the kernel does) and of the shared device headers, with comments and whitespace
    removed (an edit of comments does not change the kernel)."""
    import hashlib
    import re
    base = kind.split("_cfg")[0]
    csrc = os.path.join(ROOT, "transformer_decode_step_ns_gb300", "csrc")
    h = hashlib.sha256()
    for f in (KERNEL_SOURCE.get(base, "k_gemm.cu"), "ns_ptx.cuh", "ns_internal.h"):
        with open(os.path.join(csrc, f)) as fh:
            src = fh.read()
        cut = re.search(r"^// -+ host side$", src, flags=re.M)
        if cut is not None:
            src = src[:cut.start()]
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()[:16]


def read_traffic(kind):
    """Per-launch DRAM bytes from the committed ncu summary, when it was taken on this kernel
    source (else None: the counters are stale)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) >= 3 and parts[0] == kind:
            try:
                nbytes = float(parts[1])
            except ValueError:
                return None
            return nbytes if parts[2] == kernel_source_hash(kind) else None
    return None


def replica_aggregate(ms_local: float, units_local: int, world: int):
    """Whole-job figures of independent replicas (the step does not shard): the slowest rank's
    time and the units every rank processed.  One collective per measurement, outside the
    timed region; the data path has none."""
    if world <= 1:
        return ms_local, units_local
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms_local], dtype=torch.float64, device=device)
    u = torch.tensor([units_local], dtype=torch.int64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), int(u.item())


def repeat_check(ms_a: float, n_a: int, ms_b: float, n_b: int, limit: float = 0.15):
    """The timed steps read as two back-to-back runs (first and second half): each run's ms per
    step and whether they differ by more than ``limit`` of the faster one (clocks that had not
    settled, or another tenant's load; such a number is re-measured).  None when a half is
    empty."""
    if n_a < 1 or n_b < 1:
        return None
    a, b = ms_a / n_a, ms_b / n_b
    spread = abs(a - b) / max(min(a, b), 1e-12)
    return {"ms_per_step_halves": [round(a, 4), round(b, 4)], "spread": round(spread, 4),
            "limit": limit, "flagged": spread > limit}


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
        warm_meta = wl.next_meta()
        wl.step(warm_meta)
    torch.cuda.synchronize()
    metas = [wl.next_meta() for _ in range(K)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler()
    clocks.start()
    # keep the GPU busy (untimed replays of the last warm-up step) until sampling is live
    t_wait = time.time()
    while not clocks.has_samples() and time.time() - t_wait < 5.0:
        for _ in range(20):
            wl.step(warm_meta)
        torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e_mid = torch.cuda.Event(enable_timing=True)
    half = K // 2
    clocks.mark_start()
    e0.record()
    for i, m in enumerate(metas):
        if i == half:
            e_mid.record()
        wl.step(m)
    e1.record()
    torch.cuda.synchronize()
    clocks.mark_stop()
    ms_total = e0.elapsed_time(e1)
    repeat = (repeat_check(e0.elapsed_time(e_mid), half, e_mid.elapsed_time(e1), K - half)
              if half >= 1 else None)
    clk = clocks.stop()
    ms_total, units = replica_aggregate(ms_total, wl.B * K, world)
    dev_err = wl.dev.device_error()
    info = wl.dev.info()
    graphs = wl.dev.graph_report()
    ms_step = ms_total / K
    value = units / (ms_total * 1e-3)

    # e2e: greedy decode through the public API.  Every step uploads its host metadata, runs,
    # takes the argmax on the GPU into the token buffer the next step reads (device token
    # source) and copies the ids to pinned host memory, where they are read one step late (the
    # end-of-sequence check of asynchronous batch formation)
    ids_dev = torch.from_numpy(wl.tokens.copy()).cuda()  # the first step's tokens
    host_ids = [torch.empty(wl.B, dtype=torch.int32).pin_memory() for _ in range(2)]
    evs = [torch.cuda.Event() for _ in range(2)]
    wl.dev.set_token_source(ids_dev)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    t0 = time.perf_counter()
    for k in range(e2e_steps):
        m = wl.next_meta()
        wl.dev.step(None, *m[1:], wl.logits)
        _lib.greedy_argmax(wl.logits, ids_dev)
        host_ids[k % 2].copy_(ids_dev, non_blocking=True)
        evs[k % 2].record()
        if k > 0:
            evs[(k - 1) % 2].synchronize()
            wl.tokens = host_ids[(k - 1) % 2].numpy().copy()
    evs[(e2e_steps - 1) % 2].synchronize()
    e2e_ms, e2e_units = replica_aggregate((time.perf_counter() - t0) * 1e3, wl.B * e2e_steps, world)
    e2e_value = e2e_units / (e2e_ms * 1e-3)
    wl.tokens = host_ids[(e2e_steps - 1) % 2].numpy().copy()
    wl.dev.set_token_source(None)

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

    # the same model at batch 1 and 8 (and the headline's 32): graph-replayed step time
    sweep = []
    if rank == 0:
        for B in (1, 8):
            sw = DecodeWorkload(B, total_steps=70)
            for _ in range(5):
                sw.step(sw.next_meta())
            sm = [sw.next_meta() for _ in range(50)]
            torch.cuda.synchronize()
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s0.record()
            for m in sm:
                sw.step(m)
            s1.record()
            torch.cuda.synchronize()
            ms = s0.elapsed_time(s1) / len(sm)
            wk = rl.decode_step_work(sw.shape, sm[-1][3])
            tr = rl.step_roofline_time(wk.flops, wk.total_bytes, tflops, hbm * 1e9)
            sweep.append({"batch": B, "ms_per_step": round(ms, 4), "tokens_per_s": round(B / (ms * 1e-3), 1),
                          "roofline_us": round(tr * 1e6, 1), "frac_of_roofline": round(tr / (ms * 1e-3), 4)})
            sw.dev.close()
            del sw
        sweep.append({"batch": wl.B, "ms_per_step": round(ms_step, 4), "tokens_per_s": round(value / world, 1),
                      "roofline_us": round(t_roof * 1e6, 1), "frac_of_roofline": round(t_roof / (ms_step * 1e-3), 4)})
        torch.cuda.empty_cache()

    attn = None
    if not args.skip_attention and rank == 0:
        aw = AttentionWorkload(max_batch=max(SWEEP_BATCHES))
        attn = aw.report(256, max(10, min(K, 50)), W, hbm)
        attn["sweep_l2_flushed"] = aw.sweep(SWEEP_BATCHES, hbm)
        attn["device_error"] = _lib.device_error()
        del aw
        torch.cuda.empty_cache()

    nano = None
    if not args.skip_nanobatch and rank == 0:
        nw = NanoLayerWorkload()
        nano = nw.report(20, 3, peaks)
        del nw
        torch.cuda.empty_cache()

    cont = None
    if not args.skip_continuous and rank == 0 and args.continuous_steps > 0:
        cw = ContinuousWorkload()
        cont = cw.report(args.continuous_steps, peaks)
        del cw
        torch.cuda.empty_cache()

    serve = None
    if not args.skip_serving and rank == 0:
        sw = ServingWorkload()
        serve = sw.report()
        del sw
        torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.skip_cpu:
        import oracle
        hw, hk, hv = host_copy_of(wl)
        model = oracle.OracleModel.from_weights(wl.shape, hw)
        rows = np.arange(min(args.cpu_rows, wl.B))
        secs, reps = 0.0, 0
        while reps < 1 or (secs < args.cpu_seconds and reps < 200):
            secs += oracle_sample(model, hk, hv, metas[reps % len(metas)], rows, wl.bs)
            reps += 1
        cpu = {"value": len(rows) * reps / secs, "unit": "tokens/s", "cores": blas_threads(),
               "kind": "oracle",
               "sample": f"{reps} decode steps of {len(rows)} of the {wl.B} requests (24 layers "
                         f"+ LM head each, fp64 numpy), {secs:.1f} s of CPU work"}

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
                "loop": "greedy decode: host metadata upload, step, argmax into the device token "
                        "source of the next step, ids copied to pinned host memory and read one "
                        "step late"},
        "roofline": roof,
        "step_roofline": step_roof,
        "batch_sweep": sweep,
        "attention": attn,
        "nanobatch_layer": nano,
        "continuous": cont,
        "serving": serve,
        "cpu_baseline": cpu,
        "clocks": clk,
        "repeat": repeat,
        "gpu_launches": info.kernels_per_step * K,
        "kernels_per_step": info.kernels_per_step,
        "graph_capture_ms": info.last_capture_ms,
        "graphs": [{k: (round(v, 3) if isinstance(v, float) else v) for k, v in g.items()}
                   for g in graphs],
        "device_error": dev_err,
    }
    print(json.dumps(line), flush=True)


def run_attention_only(args, rank, world):
    """Paged decode attention alone at one batch size (the attention workload's own line)."""
    import torch
    import __graft_entry__ as ge
    from transformer_decode_step_ns_gb300 import _lib
    ge.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    peaks, src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    B = args.attn_batch
    aw = AttentionWorkload(max_batch=B, pool_blocks=args.attn_pool_blocks)
    r = aw.report(B, args.steps, args.warmup, hbm)
    if rank != 0:
        return
    line = {"metric": "paged-attn HBM GB/s", "value": r["gbs"], "unit": "GB/s",
            "n_gpus": world, "steps": max(args.steps, 10), "warmup": args.warmup,
            "ms_per_step": r["ms_per_launch"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": r["workload"], "l2": r["l2"]},
            "roofline": {"bound": "hbm", "achieved": r["gbs"], "peak": hbm, "unit": "GB/s",
                         "frac": r["frac_of_hbm"], "traffic": read_traffic(f"attention_cfg2_b{B}"),
                         "peak_source": src},
            "device_error": _lib.device_error()}
    print(json.dumps(line), flush=True)


def run_extra_only(args, rank, world):
    """One of the extra workloads alone, as its own JSON line (--nanobatch-only,
    --continuous-only, --serving-only, --offload-only, --gemm-only)."""
    import torch
    import __graft_entry__ as ge
    ge.build()
    torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
    peaks, src = load_peaks()
    if args.nanobatch_only:
        nw = NanoLayerWorkload()
        r = nw.report(max(args.steps, 1), args.warmup, peaks, tune=not args.no_tune)
        line = {"metric": "70B-layer step time, dense batch 2048 (1024 decode + 1024 prefill)",
                "value": r["tuned"]["us"], "unit": "us", "higher_is_better": False,
                "n_gpus": world, "steps": max(args.steps, 1), "warmup": args.warmup,
                "dtype": "bf16", "data": "synthetic", "config": {"workload": r["workload"]},
                "nanobatch_layer": r}
    elif args.gemm_only:
        r = GemmWorkload(args.gemm_rows).report(peaks)
        tot = sum(v["us"] for v in r["projections"].values())
        roof = sum(v["roofline_us"] for v in r["projections"].values())
        line = {"metric": "projection time per layer, LLaMA-3-8B shapes", "unit": "us",
                "value": round(tot, 1), "higher_is_better": False, "n_gpus": world, "steps": 20,
                "warmup": 3, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": r["workload"]}, "frac_of_roofline": round(roof / tot, 4),
                "gemm": r}
    elif args.offload_only:
        r = OffloadWorkload().report()
        line = {"metric": "KV reload GB/s (contiguous H2D + scatter into pages)", "unit": "GB/s",
                "value": r["reload_gbs"], "higher_is_better": True, "n_gpus": world, "steps": 5,
                "warmup": 1, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": r["workload"]}, "offload": r}
    elif args.serving_only:
        r = ServingWorkload().report()
        line = {"metric": "serving output tokens/s, constant dense batch", "unit": "tokens/s",
                "value": max(r[k]["output_tokens_per_s"] for k in ("reserved_peaks", "predicted_peaks",
                                                                   "reserved_peaks_async")),
                "higher_is_better": True, "n_gpus": world,
                "steps": sum(r[k]["steps"] for k in ("reserved_peaks", "predicted_peaks", "reserved_peaks_async")),
                "warmup": 0, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": r["workload"]}, "serving": r}
    else:
        cw = ContinuousWorkload()
        r = cw.report(args.continuous_steps, peaks)
        line = {"metric": "decode output tokens/s, continuous batching", "unit": "tokens/s",
                "value": r["tokens_per_s_device"], "higher_is_better": True,
                "n_gpus": world, "steps": r["steps"], "warmup": 20, "dtype": "bf16",
                "data": "synthetic", "config": {"workload": r["workload"]}, "continuous": r}
    if rank == 0:
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
    ap.add_argument("--skip-nanobatch", action="store_true")
    ap.add_argument("--skip-continuous", action="store_true")
    ap.add_argument("--continuous-steps", type=int, default=2000)
    ap.add_argument("--skip-serving", action="store_true")
    ap.add_argument("--no-tune", action="store_true",
                    help="with --nanobatch-only: time the named splits only, no tuner")
    ap.add_argument("--offload-only", action="store_true",
                    help="time KV save/reload of one request alone")
    ap.add_argument("--gemm-only", action="store_true",
                    help="time the LLaMA-3-8B projections alone (--gemm-rows rows)")
    ap.add_argument("--gemm-rows", type=int, default=256)
    ap.add_argument("--serving-only", action="store_true",
                    help="run the batch-former serving workload alone")
    ap.add_argument("--nanobatch-only", action="store_true",
                    help="time the 70B-layer nano-batch workload alone")
    ap.add_argument("--continuous-only", action="store_true",
                    help="run the continuous-batching LLaMA-3-8B workload alone")
    ap.add_argument("--cpu-rows", type=int, default=32)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="minimum CPU time of the oracle baseline sample")
    ap.add_argument("--ref-rows", type=int, default=4)
    ap.add_argument("--attention-only", action="store_true",
                    help="time the paged attention workload alone at --attn-batch")
    ap.add_argument("--attn-batch", type=int, default=256)
    ap.add_argument("--attn-pool-blocks", type=int, default=160_000)
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
        elif args.attention_only:
            run_attention_only(args, rank, world)
        elif (args.nanobatch_only or args.continuous_only or args.serving_only or args.offload_only
              or args.gemm_only):
            run_extra_only(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            if dist.is_initialized():
                dist.destroy_process_group()


if __name__ == "__main__":
    main()
