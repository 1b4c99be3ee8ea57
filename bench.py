#!/usr/bin/env python
"""Decode-step benchmark on GB300.

Headline workload (one JSON line on rank 0): continuous-batching decode of a 32-layer
LLaMA-3-8B-shaped decoder (hidden 4096, 32 Q / 8 KV heads, head_dim 128, SwiGLU 14336, vocab
128256, untied head, bf16, seeded N(0, 0.02) weights) at a constant batch of 256 requests:
contexts uniform in [512, 4096], decode lengths uniform in [100, 1000], finished requests leave
and new ones join their rows, block size 16 over a shuffled pool, the step captured as a CUDA
graph and replayed, greedy argmax fed back on the device.  A "step" is one full decode
iteration for every row: packed metadata upload, all 32 layers, the LM head to fp32 logits, the
greedy argmax.

Reported:
  value      output tokens/s over K device-timed steps at the batch's steady state, after the
             e2e run (CUDA events on the stream; the metadata of every step, joins and leaves
             included, prepared before the region).
  e2e        the continuous run (--continuous-steps, 2000 by default) through the public API,
             host wall clock: every step the host slot mapper and bookkeeping, one metadata
             upload, graph replay, argmax into the next step's token source, ids to the host.
  roofline   the dominant kernel (paged decode attention: ~2/3 of the step) against the
             measured HBM copy bandwidth, from CUDA-event pairs around each launch of eager
             steps.
  step_roofline  the whole step against max(FLOPs / tensor peak, bytes / HBM bandwidth).
  cpu_baseline   the fp64 CPU oracle on a bounded sample of the same workload, on all host
             cores and on one (inputs drawn on the host, in a child process).
Extra objects: the 24-layer Qwen2.5-0.5B shape (batch 32 and batches 1, 8), the 2-layer Qwen
shape at batch 1 with L2 flushed, paged attention alone (batch 256 and an L2-flushed batch
sweep), the 70B-shaped layer's nano-batch tuning, the batch-former serving run and the KV
offload.

``--impl reference`` times the CPU oracle alone (the reference arm) on the same workload.
Under torchrun each rank runs an independent replica (no data-path collective; the step does
not shard).
"""
from __future__ import annotations

import os as _os
import sys as _sys

if "--oracle-leg" in _sys.argv or ("--impl" in _sys.argv and "reference" in _sys.argv):
    # the oracle's BLAS thread count is fixed when numpy loads: all host cores unless the
    # caller chose (the oracle legs set it for their child processes)
    _n = str(len(_os.sched_getaffinity(0)))
    for _k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        _os.environ.setdefault(_k, _n)

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
WORKLOAD = ("llama-3-8b-shape 32L bf16 continuous-batching decode, batch 256, ctx U[512,4096], "
            "decode U[100,1000] with leave/join, bs16, graph replay, greedy argmax fed back")
WORKLOAD_QWEN = "qwen2.5-0.5b-shape 24L fp16 decode, batch 32, ctx U[128,1024], bs16, graph replay"
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


def cfg4_first_step_host():
    """The continuous run's first step, built on the host alone with the allocator model: the
    same tokens, positions, block tables (the run's shuffled free list, blocks handed out row by
    row) and slots as ContinuousWorkload builds through the library's pool."""
    import oracle
    cw = ContinuousWorkload
    seed = synth.config_seed(4)
    sh = synth.llama3_8b_shape(32)
    B, bs = cw.B, cw.bs
    mb = cfg4_table_width(bs)
    nb = B * mb
    ctx = synth.ctx_uniform(seed, "cfg4.join.ctx", B, cw.ctx_lo, cw.ctx_hi)
    alloc = oracle.BlockAllocator(nb, bs)
    ids = np.array(alloc.alloc(nb))
    alloc.release(ids[synth.permutation(seed, "cfg4.pool", nb)])
    tab = np.zeros((B, mb), dtype=np.int32)
    for b in range(B):
        n = int(math.ceil(int(ctx[b]) / bs))
        tab[b, :n] = alloc.alloc(n)
    pos = ctx.astype(np.int32)
    slots = alloc.prepare_step(tab, pos)
    tok = synth.uniform_int(seed, "cfg4.tokens", B, 0, sh.vocab - 1).astype(np.int32)
    return tok, pos, tab, pos + 1, slots


class Cfg4OracleSample:
    """Inputs of the oracle on the continuous LLaMA-3-8B workload, drawn on the host from the
    seeded streams the GPU run uses (no GPU, no library): the first step of the batch of 256
    (contexts, tokens, block tables handed out by the allocator model from the run's shuffled
    free list) and, for the rows a sample takes, their cached K/V blocks.  The host draws layer
    0's weights (218 M values) and the LM head (525 M); every layer of the oracle's model reuses
    layer 0's weights and cache contents (drawing all 7 B weights on the host takes minutes), so
    each sampled step does the arithmetic of the full 32-layer step plus the head."""

    def __init__(self, workers):
        import oracle
        self.oracle = oracle
        self.sh = sh = synth.llama3_8b_shape(32)
        self.seed = seed = synth.config_seed(4)
        self.tok, self.pos, self.tab, self.seq, self.slots = cfg4_first_step_host()
        self.bs = bs = ContinuousWorkload.bs
        h, f, qd, kvd = sh.hidden, sh.ffn, sh.q_dim, sh.kv_dim
        shapes = {"wq": (qd, h), "wk": (kvd, h), "wv": (kvd, h), "wo": (h, qd),
                  "w_gate": (f, h), "w_up": (f, h), "w_down": (h, f)}
        t0 = time.perf_counter()
        layer = {k: synth.normal_threads(seed, f"layer0.{k}", shp, "bf16", 0.02, threads=workers)
                 for k, shp in shapes.items()}
        head = synth.normal_threads(seed, "lm_head", (sh.vocab, h), "bf16", 0.02, threads=workers)
        self.draw_s = time.perf_counter() - t0
        wid = lambda a: oracle.from_storage(a, "bf16")  # noqa: E731
        ones = wid(synth.to_storage(np.ones(h), "bf16"))
        l0 = {k: wid(v) for k, v in layer.items()}
        l0["attn_norm"], l0["ffn_norm"] = ones, ones
        self.layers = [l0] * sh.n_layers
        self.head = wid(head)
        self.final_norm = ones
        self.blk_elems = sh.n_kv_heads * bs * sh.head_dim

    def inputs(self, rows):
        """(model, k pools, v pools, token ids, positions, tables, seq_lens, slots) of `rows`,
        their blocks renumbered into a compact pool; the embedding rows of their tokens."""
        sh, bs, seed = self.sh, self.bs, self.seed
        rows = np.asarray(rows)
        used, index = [], {}
        ctab = np.zeros((len(rows), self.tab.shape[1]), dtype=np.int32)
        for i, r in enumerate(rows):
            for j in range(int(math.ceil(int(self.seq[r]) / bs))):
                b = int(self.tab[r, j])
                if b not in index:
                    index[b] = len(used)
                    used.append(b)
                ctab[i, j] = index[b]
        shp = (len(used), sh.n_kv_heads, bs, sh.head_dim)
        kp = np.stack([synth.normal_threads(seed, "cfg4.k0", (self.blk_elems,), "bf16",
                                            offset=b * self.blk_elems) for b in used]).reshape(shp)
        vp = np.stack([synth.normal_threads(seed, "cfg4.v0", (self.blk_elems,), "bf16",
                                            offset=b * self.blk_elems) for b in used]).reshape(shp)
        emb = np.stack([synth.normal(seed, "embed", (sh.hidden,), "bf16", std=0.02,
                                     offset=int(self.tok[r]) * sh.hidden) for r in rows])
        model = self.oracle.OracleModel(shape=sh, embed=self.oracle.from_storage(emb, "bf16"),
                                        final_norm=self.final_norm, lm_head=self.head,
                                        layers=self.layers)
        cslots = np.array([index[int(s) // bs] * bs + int(s) % bs for s in self.slots[rows]],
                          dtype=np.int64)
        # the same compact pool serves every layer (layer 0's contents)
        return (model, [kp] * sh.n_layers, [vp] * sh.n_layers, np.arange(len(rows), dtype=np.int32),
                self.pos[rows], ctab, self.seq[rows], cslots)

    def time_step(self, rows):
        """Seconds of one oracle decode step over `rows` (inputs built outside the timing)."""
        args = self.inputs(rows)
        t0 = time.perf_counter()
        self.oracle.decode_step(*args, self.bs)
        return time.perf_counter() - t0

    def describe(self, rows_per_step, steps):
        return (f"{steps} decode steps of {rows_per_step} of the 256 requests (rows taken in turn), "
                f"each a full 32-layer step + LM head in fp64 numpy; the 32 layers reuse layer 0's "
                f"seeded weights and cache contents (drawn on the host in {self.draw_s:.0f} s)")


def oracle_leg(args):
    """The oracle on bounded samples of the headline workload, timed on the host cores this
    process's BLAS was given; prints one JSON object."""
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", len(os.sched_getaffinity(0))))
    smp = Cfg4OracleSample(workers=len(os.sched_getaffinity(0)))
    R = max(1, args.ref_rows)
    secs, n = 0.0, 0
    while n < 1 or (secs < args.oracle_seconds and n < 200):
        rows = (np.arange(R) + n * R) % ContinuousWorkload.B
        secs += smp.time_step(rows)
        n += 1
    print(json.dumps({"value": R * n / secs, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                      "seconds": secs, "steps": n, "sample": smp.describe(R, n)}), flush=True)


# ---------------------------------------------------------------------------------- attention

class AttentionWorkload:
    """Paged decode attention alone: 32 Q / 8 KV heads, head_dim 128, bf16, block size 16,
    contexts log-uniform in [512, 8192], block tables drawn from a shuffled pool.

    Contexts are drawn for `max_batch` rows by index, so batch B uses the first B of them and
    batch 256 is the same input at any `max_batch`."""

    n_q, n_kv, d, bs, mb = 32, 8, 128, 16, 512

    def __init__(self, max_batch: int = 512, pool_blocks: int = 160_000, ctx_mix: str = "cfg2"):
        import torch
        seed = synth.config_seed(2)
        if ctx_mix == "cfg4":  # the continuous LLaMA-3-8B run's first-step contexts (+ this token)
            self.ctx = synth.ctx_uniform(synth.config_seed(4), "cfg4.join.ctx", max_batch, 512, 4096) + 1
        else:
            self.ctx = synth.ctx_log_uniform(seed, "cfg2.ctx", max_batch, 512, 8192)
        self.ctx_mix = ctx_mix
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
        mix = ("ctx uniform[513,4097] (the continuous run's first step)" if self.ctx_mix == "cfg4"
               else "ctx log-uniform[512,8192]")
        return {"workload": f"paged GQA decode attention, batch {B}, 32Q/8KV, d128, bf16, "
                            f"{mix}, {self.nb}-block pool",
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

    def time_variant(self, sizes, budget, steps, warmup, gemm_budget=0):
        import torch
        self.dev.set_nanobatch(sizes, attn_cta_budget=budget, gemm_cta_budget=gemm_budget)
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

        def step(sizes, budget, gemm_budget=0):
            self.dev.set_nanobatch(sizes, attn_cta_budget=budget, gemm_cta_budget=gemm_budget)
            self.dev.step(*self.meta, None)

        # projections of each nano-batch on g SMs (one persistent CTA per SM), the attention of
        # the other on the SMs they leave (two attention CTAs per SM), or uncapped
        import torch
        sms = int(torch.cuda.get_device_properties(0).multi_processor_count)
        pairs = [(g, 2 * (sms - g)) for g in (sms // 2, 2 * sms // 3, 4 * sms // 5, 9 * sms // 10)]
        pairs += [(2 * sms // 3, 0), (4 * sms // 5, 0)]
        found = tuner.search(step, self.B, profile=prof, reps=max(3, min(steps, 10)), gemm_pairs=pairs)
        for r in found["table"]:
            r["frac_of_roofline"] = round(t_roof / (r["ms"] * 1e-3), 4)
        rows = []
        for label, sizes in self.LABELS.items():
            r = next(t for t in found["table"] if t["sizes"] == sizes and t["budget"] == 0
                     and t["gemm_budget"] == 0)
            rows.append({"split": label, "sizes": sizes, "attn_cta_budget": 0,
                         "us": round(r["ms"] * 1e3, 1),
                         "tflops": round(flops / (r["ms"] * 1e-3) / 1e12, 1),
                         "frac_of_roofline": r["frac_of_roofline"]})
        best = found["best"]
        # the tuned configuration, timed again over the full step count
        ms = self.time_variant(None if len(best["sizes"]) == 1 else best["sizes"], best["budget"],
                               steps, warmup, best["gemm_budget"])
        tuned = {"sizes": best["sizes"], "attn_cta_budget": best["budget"],
                 "gemm_cta_budget": best["gemm_budget"], "us": round(ms * 1e3, 1),
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
    host slot mapper, one ns_decode_step (graph replay), greedy argmax on the GPU whose ids are
    the next step's tokens."""

    B, bs, ctx_lo, ctx_hi, dec_lo, dec_hi = 256, 16, 512, 4096, 100, 1000

    def __init__(self, max_joins: int = 100_000, n_layers: int = 32):
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        self.seed = seed = synth.config_seed(4)
        self.shape = sh = synth.llama3_8b_shape(n_layers)
        B, bs = self.B, self.bs
        self.mb = mb = cfg4_table_width()
        # the worst case (every row at its longest) for the full model; a truncated model (a
        # small case for profilers) gets the first step's blocks plus room for a few hundred
        # steps of growth and joins
        first = int(sum(math.ceil((int(c) + 1) / bs) for c in
                        synth.ctx_uniform(seed, "cfg4.join.ctx", B, self.ctx_lo, self.ctx_hi)))
        self.num_blocks = B * mb if n_layers == 32 else min(B * mb, first + 16 * mb)
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
        # greedy ids of the last step: the next step's tokens (device token source)
        self.ids_dev = torch.from_numpy(self.tokens.copy()).cuda()
        self.nano = None
        self.attn_budget = 0
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

    def next_meta(self):
        """This step's metadata (the slot mapper takes a block where a row crosses into one)."""
        slots = self.dev.prepare_step(self.pos, self.tables)
        return (self.pos.copy(), self.tables.copy(), (self.pos + 1).astype(np.int32), slots)

    def advance(self) -> int:
        """After a step: every row moves one position on; finished requests leave and new ones
        join their rows.  Returns the number of leave/join pairs."""
        self.pos += 1
        self.left -= 1
        done = np.nonzero(self.left == 0)[0]
        for b in done:
            self.leave(int(b))
            self.join(int(b))
        return len(done)

    def plan(self, n):
        """Metadata of the next n steps, prepared ahead (the host bookkeeping does not depend on
        the sampled tokens: requests leave at their drawn lengths)."""
        metas, leaves = [], 0
        for _ in range(n):
            metas.append(self.next_meta())
            leaves += self.advance()
        return metas, leaves

    def launch(self, meta):
        """One step through the public API, tokens read on the device from the previous step's
        greedy ids, and this step's greedy ids written back for the next."""
        from transformer_decode_step_ns_gb300 import _lib
        self.dev.step(None, *meta, self.logits)
        _lib.greedy_argmax(self.logits, self.ids_dev)

    def set_nano(self, nano, budget=None):
        self.nano = nano
        if budget is not None:
            self.attn_budget = budget
        self.dev.set_nanobatch(nano, attn_cta_budget=self.attn_budget if nano else 0)
        self.dev.set_token_source(self.ids_dev)

    def roofline_time(self, metas, peaks):
        tflops = float(peaks.get("bf16_tflops_sustained", 1700)) * 1e12
        hbm = float(peaks["hbm_gbs"]) * 1e9
        t, nbytes, flops = 0.0, 0.0, 0.0
        for m in metas:
            work = rl.decode_step_work(self.shape, m[2])
            t += rl.step_roofline_time(work.flops, work.total_bytes, tflops, hbm)
            nbytes += work.total_bytes
            flops += work.flops
        return t, nbytes, flops

    def headline(self, K, W, peaks, world):
        """W warm-up steps, then exactly K steps timed with CUDA events on the stream (bracketed
        by a barrier and synchronisation), metadata of every step prepared before the region,
        nvidia-smi sampling the clocks during it.  An event at the midpoint reads the K steps
        as two back-to-back runs."""
        import torch
        metas, leaves = self.plan(W + K)
        for m in metas[:W]:
            self.launch(m)
        torch.cuda.synchronize()
        timed = metas[W:]
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        clocks = ClockSampler()
        clocks.start()
        # keep the GPU busy (untimed repeats of the last warm-up step) until sampling is live
        t_wait = time.time()
        while not clocks.has_samples() and time.time() - t_wait < 5.0:
            for _ in range(5):
                self.launch(metas[W - 1])
            torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_mid = torch.cuda.Event(enable_timing=True)
        half = K // 2
        clocks.mark_start()
        e0.record()
        for i, m in enumerate(timed):
            if i == half:
                e_mid.record()
            self.launch(m)
        e1.record()
        torch.cuda.synchronize()
        clocks.mark_stop()
        ms_total = e0.elapsed_time(e1)
        repeat = (repeat_check(e0.elapsed_time(e_mid), half, e_mid.elapsed_time(e1), K - half)
                  if half >= 1 else None)
        t_roof, nbytes, flops = self.roofline_time(timed, peaks)
        return {"ms_total": ms_total, "repeat": repeat, "clocks": clocks.stop(),
                "roofline_s": t_roof, "bytes": nbytes, "flops": flops,
                "leaves_and_joins": leaves, "meta_bytes": cfg4_meta_bytes(self.B, self.mb)}

    def run_async(self, steps, peaks):
        """The end-to-end loop through the public API, as a server runs it: every step packs and
        uploads its host metadata (one pinned copy), replays the graph, takes the greedy argmax
        into the device token source of the next step and copies the ids to pinned host memory;
        the host reads them one step late (the end-of-sequence check of asynchronous batch
        formation) while the next step runs.  Host wall clock over the whole run."""
        import torch
        host_ids = [torch.empty(self.B, dtype=torch.int32).pin_memory() for _ in range(2)]
        evs = [torch.cuda.Event() for _ in range(2)]
        dev_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(steps)]
        t_roof, leaves = 0.0, 0
        tflops = float(peaks.get("bf16_tflops_sustained", 1700)) * 1e12
        hbm = float(peaks["hbm_gbs"]) * 1e9
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for k in range(steps):
            m = self.next_meta()
            work = rl.decode_step_work(self.shape, m[2])
            t_roof += rl.step_roofline_time(work.flops, work.total_bytes, tflops, hbm)
            dev_ev[k][0].record()
            self.launch(m)
            dev_ev[k][1].record()
            host_ids[k % 2].copy_(self.ids_dev, non_blocking=True)
            evs[k % 2].record()
            if k > 0:
                evs[(k - 1) % 2].synchronize()
                self.tokens = host_ids[(k - 1) % 2].numpy().copy()
            leaves += self.advance()
        evs[(steps - 1) % 2].synchronize()
        wall = time.perf_counter() - t0
        self.tokens = host_ids[(steps - 1) % 2].numpy().copy()
        dev_ms = np.array([a.elapsed_time(b) for a, b in dev_ev])
        return {"steps": steps, "nano_split": self.nano or [self.B], "leaves_and_joins": leaves,
                "wall_s": wall, "tokens_per_s": self.B * steps / wall,
                "device_ms_per_step_mean": float(dev_ms.mean()),
                "device_ms_per_step_median": float(np.median(dev_ms)),
                "roofline_ms_per_step_mean": t_roof / steps * 1e3,
                "frac_of_roofline_device": t_roof / (dev_ms.sum() * 1e-3),
                "graphs_cached": self.dev.info().graphs_cached,
                "device_error": self.dev.device_error()}

    def run(self, steps, peaks, nano=None):
        """Steps one at a time, each waited for (the split trial and the eager kernel timing)."""
        import torch
        self.set_nano(nano)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        metas = []
        for i in range(steps):
            m = self.next_meta()
            metas.append(m)
            ev[i][0].record()
            self.launch(m)
            ev[i][1].record()
            torch.cuda.current_stream().synchronize()
            self.advance()
        dev_ms = np.array([a.elapsed_time(b) for a, b in ev])
        t_roof, _, _ = self.roofline_time(metas, peaks)
        return {"steps": steps, "device_ms_per_step_median": float(np.median(dev_ms)),
                "frac_of_roofline": t_roof / (dev_ms.sum() * 1e-3),
                "attention_bytes": sum(rl.attention_bytes(m[2], self.shape.n_kv_heads,
                                                          self.shape.head_dim)
                                       + 4.0 * self.B * self.shape.q_dim for m in metas)
                * self.shape.n_layers}

    def pick_split(self, peaks):
        """A short comparison of the unsplit step and two nano-batches of 128 rows, the latter
        with the attention of each nano-batch uncapped or capped at one or one half CTA per SM
        (so that the other nano-batch's projections can run beside it on every SM: the NanoFlow
        page's co-running of memory- and compute-heavy nano-ops); the fastest is used for the
        rest of the run.  Returns (split, attention CTA budget, trial table)."""
        sms = int(__import__("torch").cuda.get_device_properties(0).multi_processor_count)
        trial, best = {}, (None, 0, float("inf"))
        for nano, budget in ((None, 0), ([128, 128], 0), ([128, 128], sms), ([128, 128], sms // 2)):
            self.attn_budget = budget
            ms = self.run(20, peaks, nano)["device_ms_per_step_median"]
            trial[f"{nano or [self.B]} attn_cta_budget={budget}"] = ms
            if ms < best[2]:
                best = (nano, budget, ms)
        self.set_nano(best[0], best[1])
        return best[0], best[1], trial

    def kernel_times(self, peaks):
        """Per-kind kernel times of eager steps (an event pair around each launch, on the stream
        the kernel runs on) and the attention kernel's achieved bandwidth: the algorithmic K/V
        (+ q in, o out) bytes of the timed steps over the attention launches' summed time."""
        self.dev.set_kernel_timing(True)
        self.run(2, peaks, self.nano)
        self.dev.kernel_timing()
        r = self.run(3, peaks, self.nano)
        kt = self.dev.kernel_timing()
        self.dev.set_kernel_timing(False)
        self.set_nano(self.nano)
        total = sum(v[1] for v in kt.values())
        n_attn, ms_attn = kt["attention"]
        return {"kernel_us": {k: round(v[1] / v[0] * 1e3, 1) for k, v in kt.items() if v[0]},
                "launches_per_step": {k: v[0] // 3 for k, v in kt.items() if v[0]},
                "shares": {k: round(v[1] / total, 4) for k, v in kt.items()},
                "attention_launches": n_attn, "attention_ms": ms_attn,
                "attention_bytes_per_launch": r["attention_bytes"] / n_attn,
                "attention_share": ms_attn / total}

    def offload(self, steps, peaks):
        """KV offload: steps with every step's new K/V mirrored to pinned host memory (each
        layer's rows copied while its attention and FFN run) against the same steps without;
        then the longest request saved to the host and reloaded into its blocks (contiguous
        transfer + device scatter), against plain copies of the same bytes."""
        import torch
        sh = self.shape
        row = 2 * sh.n_kv_heads * sh.head_dim
        mirror = torch.empty((sh.n_layers, self.B, row), dtype=torch.int16).pin_memory()
        self.dev.set_kv_offload(mirror)
        on = self.run(steps, peaks, self.nano)
        self.dev.set_kv_offload(None)
        off = self.run(steps, peaks, self.nano)
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

    def close(self):
        self.dev.set_token_source(None)
        self.dev.close()


def cfg4_table_width(bs: int = 16) -> int:
    """Block-table width of the continuous run: the longest context plus the longest decode."""
    return int(math.ceil((ContinuousWorkload.ctx_hi + ContinuousWorkload.dec_hi + 1) / bs))


def cfg4_meta_bytes(B: int, mb: int) -> int:
    """Bytes of one step's packed metadata upload (token ids, positions, lengths, slots, block
    tables, the logits pointer and two flags), as the library lays it out."""
    o = 12 * B
    o = (o + 15) // 16 * 16 + 8 * B + 4 * B * mb
    return (o + 15) // 16 * 16 + 16


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


def scaled_traffic(kind, algo_bytes):
    """Per-launch DRAM bytes of a launch moving `algo_bytes` algorithmic bytes, from the ncu
    summary of a smaller launch of the same kernel (its line gives the captured launch's
    algorithmic bytes as a fourth field): the captured traffic scaled by the ratio, valid when
    traffic grows in proportion to the units processed (K/V tokens read).  None when the
    counters are stale or absent."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    for line in open(p):
        parts = line.split()
        if len(parts) >= 4 and parts[0] == kind:
            try:
                dram, algo = float(parts[1]), float(parts[3])
            except ValueError:
                return None
            if parts[2] != kernel_source_hash(kind) or algo <= 0:
                return None
            return dram * algo_bytes / algo
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


class SmallStepWorkload:
    """The 2-layer Qwen2.5-0.5B-shaped decoder at batch 1 (the small parity case): 128 cached
    tokens in a seeded permutation of physical blocks 0-7, this step's token at position 128 in
    block 8, fp16 weights N(0, 0.02).  Each graph replay is timed alone after a 256 MiB write
    that flushes L2 (the step's 60 MB of layer weights would otherwise stay in L2 between
    replays)."""

    def __init__(self):
        import torch
        from transformer_decode_step_ns_gb300 import _lib
        self.shape = sh = synth.qwen05b_shape(2)
        seed = synth.config_seed(0)
        self.w = synth.model_weights_device(sh, seed)
        self.dev = _lib.DecodeStep(sh, self.w, 1, 9, use_graphs=True)
        self.dev.kv_alloc(9, 16)
        stream = torch.cuda.current_stream().cuda_stream
        n = self.dev.kv_pool_bytes() // 2
        for l in range(sh.n_layers):
            k, v = self.dev.kv_layer_ptrs(l)
            synth.fill_normal_device(k, n, seed, f"k{l}", "f16", stream=stream)
            synth.fill_normal_device(v, n, seed, f"v{l}", "f16", stream=stream)
        tab = np.zeros((1, 9), dtype=np.int32)
        tab[0, :8] = synth.permutation(seed, "cfg0.blocks", 8)
        tab[0, 8] = 8
        tok = synth.uniform_int(seed, "cfg0.token", 1, 0, sh.vocab - 1).astype(np.int32)
        self.meta = (tok, np.array([128], np.int32), tab, np.array([129], np.int32),
                     np.array([8 * 16], np.int64))
        self.logits = torch.empty((1, sh.vocab), dtype=torch.float32, device="cuda")
        self.flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def report(self, peaks, n=50, warmup=5):
        import torch
        for _ in range(warmup):
            self.dev.step(*self.meta, self.logits)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(n)]
        for a, b in ev:
            self.flush.zero_()
            a.record()
            self.dev.step(*self.meta, self.logits)
            b.record()
        torch.cuda.synchronize()
        ms = float(np.median([a.elapsed_time(b) for a, b in ev]))
        tflops = float(peaks.get("bf16_tflops", 1900)) * 1e12
        hbm = float(peaks["hbm_gbs"]) * 1e9
        work = rl.decode_step_work(self.shape, self.meta[3])
        t_roof = rl.step_roofline_time(work.flops, work.total_bytes, tflops, hbm)
        return {"workload": "qwen2.5-0.5b-shape 2L fp16 decode, batch 1, 128 cached tokens in "
                            "8 permuted blocks, graph replay, L2 flushed before each replay",
                "ms_per_step_median": round(ms, 4), "tokens_per_s": round(1.0 / (ms * 1e-3), 1),
                "replays": n, "bytes": work.total_bytes, "roofline_us": round(t_roof * 1e6, 2),
                "frac_of_roofline": round(t_roof / (ms * 1e-3), 4),
                "device_error": self.dev.device_error()}


def qwen_report(args, peaks, world):
    """The 24-layer Qwen2.5-0.5B-shaped decoder: batch 32 with its own roofline accounting (the
    dominant kernel by eager per-launch timing), then batches 1 and 8 (graph-replayed steps)."""
    import torch
    hbm = float(peaks["hbm_gbs"])
    tflops = float(peaks.get("bf16_tflops_sustained", 1700)) * 1e12
    K, W = max(args.steps, 20), args.warmup
    wl = DecodeWorkload(args.batch, total_steps=W + K + 16)
    for _ in range(W):
        wl.step(wl.next_meta())
    metas = [wl.next_meta() for _ in range(K)]
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for m in metas:
        wl.step(m)
    e1.record()
    torch.cuda.synchronize()
    ms_step = e0.elapsed_time(e1) / K
    wl.dev.set_kernel_timing(True)
    for _ in range(3):
        wl.step(wl.next_meta())
    wl.dev.kernel_timing()
    for _ in range(5):
        wl.step(wl.next_meta())
    kt = wl.dev.kernel_timing()
    wl.dev.set_kernel_timing(False)
    eager_total = sum(v[1] for v in kt.values())
    kb = kernel_bytes(wl.shape, wl.B, metas[-1][3])
    dom = max(kt, key=lambda k: kt[k][1])
    launches, tot_ms = kt[dom]
    achieved = kb[dom] / (tot_ms / launches * 1e-3) / 1e9
    work = rl.decode_step_work(wl.shape, metas[-1][3])
    t_roof = rl.step_roofline_time(work.flops, work.total_bytes, tflops, hbm * 1e9)
    out = {"workload": WORKLOAD_QWEN, "batch": wl.B, "ms_per_step": round(ms_step, 4),
           "tokens_per_s": round(wl.B / (ms_step * 1e-3), 1), "steps": K,
           "roofline_us": round(t_roof * 1e6, 1), "frac_of_roofline": round(t_roof / (ms_step * 1e-3), 4),
           "kernels_per_step": wl.dev.info().kernels_per_step,
           "dominant_kernel": {"kind": dom, "achieved_gbs": round(achieved, 1),
                               "frac_of_hbm": round(achieved / hbm, 4),
                               "traffic": read_traffic(dom), "share_of_eager_step": round(tot_ms / eager_total, 4)},
           "kernel_avg_us": {k: round(v[1] / v[0] * 1e3, 2) for k, v in kt.items()},
           "device_error": wl.dev.device_error()}
    wl.dev.close()
    del wl
    def timed(B, step_kernel):
        """Graph-replayed steps of batch B with the given ns_set_step_kernel mode."""
        sw = DecodeWorkload(B, total_steps=70)
        if step_kernel:
            sw.dev.set_step_kernel(1)
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
        row = {"batch": B, "ms_per_step": round(ms, 4), "tokens_per_s": round(B / (ms * 1e-3), 1),
               "roofline_us": round(tr * 1e6, 1), "frac_of_roofline": round(tr / (ms * 1e-3), 4),
               "kernels_per_step": sw.dev.info().kernels_per_step, "device_error": sw.dev.device_error()}
        sw.dev.close()
        del sw
        torch.cuda.empty_cache()
        return row

    out["batch_sweep"] = [timed(B, False) for B in (1, 8)]
    # the persistent step kernel (ns_set_step_kernel mode 1) on the same workloads
    out["step_kernel"] = [timed(B, True) for B in (1, 8, 32)]
    return out


def oracle_leg_subprocess(threads, seconds, rows):
    """Run the oracle leg in a child process whose BLAS uses `threads` threads (the thread count
    is fixed when numpy loads, so it cannot change inside this process).  The child draws its
    inputs on the host and loads no GPU code."""
    env = dict(os.environ)
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(threads)
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-leg", "--oracle-threads",
           str(threads), "--oracle-seconds", str(seconds), "--ref-rows", str(rows)]
    try:
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=900)
    except subprocess.TimeoutExpired:
        return {"unavailable": "oracle leg timed out"}
    for line in reversed(r.stdout.splitlines()):
        if line.startswith("{"):
            return json.loads(line)
    return {"unavailable": f"oracle leg failed (rc {r.returncode}): {r.stderr[-300:]}"}


def run_ours(args, rank, world):
    import torch
    import __graft_entry__ as ge
    from transformer_decode_step_ns_gb300 import _lib
    ge.build()
    dev_idx = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev_idx)
    peaks, peaks_src = load_peaks()
    hbm = float(peaks["hbm_gbs"])
    K, W = args.steps, args.warmup

    # ---- headline: continuous batching of the LLaMA-3-8B shape at batch 256
    cw = ContinuousWorkload()
    log(f"setup {cw.setup_s:.1f}s: {cw.num_blocks} blocks, mb {cw.mb}")
    best, budget, trial = cw.pick_split(peaks)
    # e2e: the continuous run through the public API, host metadata and token ids every step;
    # it also brings the batch to its steady state (every row has seen several requests leave
    # and join), where the headline's K steps are then timed
    if world > 1:
        torch.distributed.barrier()
    e2e_run = cw.run_async(max(1, args.continuous_steps), peaks)
    e2e_ms, e2e_units = replica_aggregate(e2e_run["wall_s"] * 1e3, cw.B * e2e_run["steps"], world)
    e2e_value = e2e_units / (e2e_ms * 1e-3)
    head = cw.headline(K, W, peaks, world)
    ms_total, units = replica_aggregate(head["ms_total"], cw.B * K, world)
    ms_step = ms_total / K
    value = units / (ms_total * 1e-3)
    info = cw.dev.info()
    graphs = cw.dev.graph_report()
    # kernels of the graph the timed steps replayed (the split trial captured others too), plus
    # the greedy argmax launched after each step
    n_split = len(best) if best else 1
    replayed = [g for g in graphs if g["n_split"] == n_split and g["with_lm"] == 1 and g["chunk_rows"] == 0]
    step_kernels = (replayed[0]["kernels"] if replayed else info.kernels_per_step) + 1
    kt = cw.kernel_times(peaks)
    offload = cw.offload(30, peaks) if rank == 0 and not args.skip_offload else None
    dev_err = cw.dev.device_error()
    cw.close()
    del cw
    torch.cuda.empty_cache()

    attn_us = kt["attention_ms"] / kt["attention_launches"] * 1e3
    achieved = kt["attention_bytes_per_launch"] / (attn_us * 1e-6) / 1e9
    roof = {"kernel": "attention (attn_decode_kernel)", "bound": "hbm", "achieved": achieved,
            "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": scaled_traffic("attention_cfg4", kt["attention_bytes_per_launch"]),
            "peak_source": "measured hbm_gbs (MEASURED_PEAKS.json)" if peaks_src == "measured"
            else "fallback 6.8 TB/s",
            "bytes_per_launch": kt["attention_bytes_per_launch"], "avg_launch_us": attn_us,
            "share_of_eager_step": kt["attention_share"], "kernel_shares": kt["shares"],
            "kernel_avg_us": kt["kernel_us"], "launches_per_step": kt["launches_per_step"]}
    t_roof = head["roofline_s"] / K
    step_roof = {"roofline_us": t_roof * 1e6, "measured_us": ms_step * 1e3,
                 "frac": t_roof / (ms_step * 1e-3), "bytes_per_step": head["bytes"] / K,
                 "flops_per_step": head["flops"] / K,
                 "bound": "hbm" if head["bytes"] / (hbm * 1e9) >= head["flops"] / (
                     float(peaks.get("bf16_tflops_sustained", 1700)) * 1e12) else "tensor",
                 "peaks": "measured HBM copy and sustained bf16" if peaks_src == "measured"
                 else "fallback"}

    # ---- the other workloads (rank 0 only)
    extras = {}
    if rank == 0:
        extras["qwen_24l"] = qwen_report(args, peaks, world) if not args.skip_qwen else None
        if not args.skip_small:
            sw = SmallStepWorkload()
            extras["qwen_2l_b1"] = sw.report(peaks)
            sw.dev.close()
            del sw
        if not args.skip_attention:
            aw = AttentionWorkload(max_batch=max(SWEEP_BATCHES))
            attn = aw.report(256, max(10, min(K, 50)), W, hbm)
            attn["sweep_l2_flushed"] = aw.sweep(SWEEP_BATCHES, hbm)
            attn["device_error"] = _lib.device_error()
            extras["attention"] = attn
            del aw
        torch.cuda.empty_cache()
        if not args.skip_nanobatch:
            nw = NanoLayerWorkload()
            extras["nanobatch_layer"] = nw.report(20, 3, peaks)
            nw.dev.close()
            del nw
            torch.cuda.empty_cache()
        if not args.skip_serving:
            sv = ServingWorkload()
            extras["serving"] = sv.report()
            del sv
            torch.cuda.empty_cache()

    cpu = None
    if rank == 0 and not args.skip_cpu:
        cores = len(os.sched_getaffinity(0))
        allc = oracle_leg_subprocess(cores, args.cpu_seconds, args.ref_rows)
        one = oracle_leg_subprocess(1, args.cpu_seconds, args.ref_rows)
        if "value" in allc:
            cpu = {"value": allc["value"], "unit": "tokens/s", "cores": allc["cores"],
                   "kind": "oracle", "sample": allc["sample"],
                   "single_thread": {"value": one.get("value"), "cores": 1,
                                     "sample": one.get("sample", one.get("unavailable"))}}
        else:
            cpu = {"unavailable": allc.get("unavailable"), "kind": "oracle"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K,
        "warmup": W, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "model": "llama-3-8b-shaped (random init)",
                   "global_batch": ContinuousWorkload.B * world,
                   "seq_len": "ctx U[512,4096] + decode U[100,1000], leave/join",
                   "nano_split": best or [ContinuousWorkload.B], "attn_cta_budget": budget,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (15 GB of weights and ~77 GB of K/V per step)"},
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": head["meta_bytes"],
                "d2h_bytes_per_step": ContinuousWorkload.B * 4, "steps": e2e_run["steps"],
                "loop": "continuous batching through the public API: every step the host slot "
                        "mapper and join/leave bookkeeping, one packed metadata upload, graph "
                        "replay, greedy argmax into the next step's device token source, ids "
                        "copied to pinned host memory and read one step late",
                "run": {k: (round(v, 4) if isinstance(v, float) else v) for k, v in e2e_run.items()}},
        "roofline": roof,
        "step_roofline": step_roof,
        "cpu_baseline": cpu,
        "clocks": head["clocks"],
        "repeat": head["repeat"],
        "gpu_launches": step_kernels * K,
        "kernels_per_step": step_kernels,
        "split_trial_ms_per_step": trial,
        "leaves_and_joins_in_timed_steps": head["leaves_and_joins"],
        "graph_capture_ms": info.last_capture_ms,
        "graphs": [{k: (round(v, 3) if isinstance(v, float) else v) for k, v in g.items()}
                   for g in graphs],
        "kv_offload": offload,
        "device_error": dev_err,
    }
    line.update(extras)
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
    aw = AttentionWorkload(max_batch=B, pool_blocks=args.attn_pool_blocks, ctx_mix=args.attn_ctx)
    r = aw.report(B, args.steps, args.warmup, hbm)
    if rank != 0:
        return
    line = {"metric": "paged-attn HBM GB/s", "value": r["gbs"], "unit": "GB/s",
            "n_gpus": world, "steps": max(args.steps, 10), "warmup": args.warmup,
            "ms_per_step": r["ms_per_launch"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": r["workload"], "l2": r["l2"]},
            "roofline": {"bound": "hbm", "achieved": r["gbs"], "peak": hbm, "unit": "GB/s",
                         "frac": r["frac_of_hbm"],
                         "traffic": (scaled_traffic("attention_cfg4", r["bytes_per_launch"])
                                     if args.attn_ctx == "cfg4" else read_traffic(f"attention_cfg2_b{B}")),
                         "peak_source": src},
            "device_error": _lib.device_error()}
    print(json.dumps(line), flush=True)


def run_extra_only(args, rank, world):
    """One of the extra workloads alone, as its own JSON line (--nanobatch-only,
    --continuous-only, --serving-only, --offload-only, --gemm-only, --qwen-only)."""
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
    elif args.qwen_only:
        r = qwen_report(args, peaks, world)
        line = {"metric": "decode output tokens/s, 24-layer Qwen2.5-0.5B shape", "unit": "tokens/s",
                "value": r["tokens_per_s"], "higher_is_better": True, "n_gpus": world,
                "steps": r["steps"], "warmup": args.warmup, "dtype": "f16", "data": "synthetic",
                "config": {"workload": r["workload"]}, "qwen_24l": r}
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
        cw = ContinuousWorkload(n_layers=args.layers)
        best, budget, trial = cw.pick_split(peaks)
        head = cw.headline(max(args.steps, 1), args.warmup, peaks, 1)
        r = cw.run_async(args.continuous_steps, peaks)
        r["split_trial_ms_per_step"] = trial
        r["kernels"] = cw.kernel_times(peaks)
        K = max(args.steps, 1)
        line = {"metric": "decode output tokens/s, continuous batching", "unit": "tokens/s",
                "value": ContinuousWorkload.B * K / (head["ms_total"] * 1e-3),
                "ms_per_step": head["ms_total"] / K, "higher_is_better": True,
                "n_gpus": world, "steps": K, "warmup": args.warmup, "dtype": "bf16",
                "data": "synthetic", "config": {"workload": WORKLOAD, "nano_split": best,
                                                 "attn_cta_budget": budget},
                "frac_of_roofline": head["roofline_s"] / (head["ms_total"] * 1e-3),
                "clocks": head["clocks"], "continuous": r}
        cw.close()
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_reference(args, rank, world):
    """The oracle arm: the fp64 CPU oracle on bounded samples of the headline workload, inputs
    drawn on the host (no GPU code is loaded)."""
    if rank != 0:
        return
    K, W = args.steps, args.warmup
    R = max(1, args.ref_rows)
    cores = int(os.environ.get("OPENBLAS_NUM_THREADS", len(os.sched_getaffinity(0))))
    smp = Cfg4OracleSample(workers=len(os.sched_getaffinity(0)))
    times = []
    for i in range(W + K):
        s_ = smp.time_step((np.arange(R) + i * R) % ContinuousWorkload.B)
        if i >= W:
            times.append(s_)
    total = sum(times)
    value = R * K / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": K, "warmup": W, "ms_per_step": total / K * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "model": "llama-3-8b-shaped (random init)",
                       "global_batch": ContinuousWorkload.B,
                       "seq_len": "ctx U[512,4096] + decode U[100,1000], leave/join",
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": smp.describe(R, K)},
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
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="minimum CPU time of each oracle baseline sample")
    ap.add_argument("--ref-rows", type=int, default=2)
    ap.add_argument("--attention-only", action="store_true",
                    help="time the paged attention workload alone at --attn-batch")
    ap.add_argument("--attn-batch", type=int, default=256)
    ap.add_argument("--attn-pool-blocks", type=int, default=160_000)
    ap.add_argument("--attn-ctx", default="cfg2", choices=["cfg2", "cfg4"],
                    help="context mix of --attention-only: the attention workload's own, or the "
                         "continuous LLaMA-3-8B run's")
    ap.add_argument("--layers", type=int, default=32,
                    help="with --continuous-only: layers of the LLaMA-3-8B shape (fewer: a small "
                         "case of the same kernels, e.g. for profilers)")
    ap.add_argument("--skip-qwen", action="store_true")
    ap.add_argument("--qwen-only", action="store_true",
                    help="run the 24-layer Qwen2.5-0.5B-shaped workloads alone (batch --batch, 1 and 8, "
                         "and the persistent step kernel at 1, 8 and 32)")
    ap.add_argument("--skip-small", action="store_true")
    ap.add_argument("--skip-offload", action="store_true")
    ap.add_argument("--oracle-leg", action="store_true",
                    help="internal: time the oracle on the headline workload and print JSON")
    ap.add_argument("--oracle-threads", type=int, default=0)
    ap.add_argument("--oracle-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.oracle_leg:
        oracle_leg(args)
        return
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
              or args.gemm_only or args.qwen_only):
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
