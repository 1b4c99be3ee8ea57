"""Seeded synthetic inputs for the decode step (weights, KV-cache contents, request mixes).

This module is the one piece of code that both sides of the parity tests use: the CPU oracle
and the CUDA library consume the arrays it draws.  It holds none of the decode step's
arithmetic -- only random numbers, storage-format rounding of those numbers, and the
bookkeeping of which synthetic request owns which physical cache block.

Generator (counter based, so any element can be drawn on its own, on the host or the GPU):

* ``mix64`` is the splitmix64 output function (Steele, Lea & Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014; constants as published by Vigna).
* Stream key for a named tensor: ``key = mix64(seed ^ mix64(fnv1a64(name)))``.
* Raw word ``i`` of a stream: ``w_i = mix64(key + (i + 1) * 0x9E3779B97F4A7C15 mod 2**64)``.
* Normal variate ``i`` (Box-Muller, one variate per word, fp64):
  ``u1 = ((w_i >> 32) + 1) / 2**32`` in (0, 1], ``u2 = (w_i & 0xffffffff) / 2**32`` in [0, 1),
  ``z = sqrt(-2 ln u1) * cos(6.283185307179586 * u2)``; the value ``mean + std * z`` is rounded
  fp64 -> fp32 -> storage type, each step round-to-nearest-even.
* Uniform double ``i``: ``(w_i >> 11) / 2**53``.

``synth/csrc/fill.cu`` implements the same definition on the GPU for pools too large to draw
on the host; both sides call the platform's own ``log``/``cos``/``sqrt`` in fp64, so their
outputs agree except where the two libraries round a transcendental differently in the last
fp64 bit and that bit decides a 16-bit rounding (probability ~2**-40 per element).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
TWO_PI = 6.283185307179586
_CHUNK = 1 << 22

F16 = "f16"
BF16 = "bf16"


def mix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 output function on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def fnv1a64(name: str) -> int:
    h = 0xCBF29CE484222325
    for byte in name.encode("utf-8"):
        h ^= byte
        h = (h * 0x100000001B3) & 0xFFFFFFFFFFFFFFFF
    return h


def stream_key(seed: int, name: str) -> int:
    tag = int(mix64(np.array([fnv1a64(name)], dtype=np.uint64))[0])
    return int(mix64(np.array([(seed ^ tag) & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64))[0])


def raw_words(key: int, start: int, count: int) -> np.ndarray:
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        state = np.uint64(key) + idx * GOLDEN
    return mix64(state)


def normal_f64(key: int, start: int, count: int) -> np.ndarray:
    w = raw_words(key, start, count)
    u1 = ((w >> np.uint64(32)).astype(np.float64) + 1.0) * (1.0 / 4294967296.0)
    u2 = (w & np.uint64(0xFFFFFFFF)).astype(np.float64) * (1.0 / 4294967296.0)
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(TWO_PI * u2)


def uniform_f64(key: int, start: int, count: int) -> np.ndarray:
    w = raw_words(key, start, count)
    return (w >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bfloat16 (nearest-even), returned as the uint16 bit pattern."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def to_storage(x64: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 -> fp32 -> storage type.  fp16 is numpy float16; bf16 is a uint16 bit array."""
    x32 = np.asarray(x64, dtype=np.float64).astype(np.float32)
    if dtype == F16:
        return x32.astype(np.float16)
    if dtype == BF16:
        return f32_to_bf16_bits(x32)
    raise ValueError(f"unknown storage dtype {dtype!r}")


def normal(seed: int, name: str, shape: Sequence[int], dtype: str, std: float = 1.0,
           mean: float = 0.0, offset: int = 0) -> np.ndarray:
    """Draw ``mean + std * N(0,1)`` of ``shape`` from stream ``name``, rounded to ``dtype``."""
    n = int(np.prod(shape)) if len(shape) else 1
    key = stream_key(seed, name)
    out = np.empty(n, dtype=np.float16 if dtype == F16 else np.uint16)
    for s in range(0, n, _CHUNK):
        c = min(_CHUNK, n - s)
        out[s:s + c] = to_storage(mean + std * normal_f64(key, offset + s, c), dtype)
    return out.reshape(shape)


def uniform_int(seed: int, name: str, count: int, lo: int, hi: int) -> np.ndarray:
    """Integers uniform on [lo, hi] (inclusive)."""
    u = uniform_f64(stream_key(seed, name), 0, count)
    return (lo + np.floor(u * (hi - lo + 1))).astype(np.int64).clip(lo, hi)


def log_uniform_int(seed: int, name: str, count: int, lo: int, hi: int) -> np.ndarray:
    """Integers log-uniform on [lo, hi]."""
    u = uniform_f64(stream_key(seed, name), 0, count)
    v = np.floor(np.exp(math.log(lo) + u * (math.log(hi + 1) - math.log(lo))))
    return v.astype(np.int64).clip(lo, hi)


def permutation(seed: int, name: str, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of range(n) driven by the counter stream."""
    u = uniform_f64(stream_key(seed, name), 0, max(n, 1))
    perm = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(u[n - 1 - i] * (i + 1))
        perm[i], perm[j] = perm[j], perm[i]
    return perm


# --------------------------------------------------------------------------------------------
# Model shapes and seeded weights
# --------------------------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class ModelShape:
    hidden: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rms_eps: float
    rope_theta: float
    dtype: str
    tie_embeddings: bool

    @property
    def q_dim(self) -> int:
        return self.n_q_heads * self.head_dim

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def param_count(self) -> int:
        h, f = self.hidden, self.ffn
        per_layer = (h * self.q_dim + 2 * h * self.kv_dim + self.q_dim * h
                     + 3 * h * f + 2 * h)
        head = 0 if self.tie_embeddings else self.vocab * h
        return self.vocab * h + self.n_layers * per_layer + h + head


def qwen05b_shape(n_layers: int = 24) -> ModelShape:
    """Qwen2.5-0.5B-shaped decoder (dims as the nanoserve page's model), fp16, tied head."""
    return ModelShape(hidden=896, n_layers=n_layers, n_q_heads=14, n_kv_heads=2, head_dim=64,
                      ffn=4864, vocab=151936, rms_eps=1e-6, rope_theta=1e6, dtype=F16,
                      tie_embeddings=True)


def llama3_8b_shape(n_layers: int = 32) -> ModelShape:
    return ModelShape(hidden=4096, n_layers=n_layers, n_q_heads=32, n_kv_heads=8, head_dim=128,
                      ffn=14336, vocab=128256, rms_eps=1e-5, rope_theta=5e5, dtype=BF16,
                      tie_embeddings=False)


def llama2_70b_layer_shape() -> ModelShape:
    return ModelShape(hidden=8192, n_layers=1, n_q_heads=64, n_kv_heads=8, head_dim=128,
                      ffn=28672, vocab=32000, rms_eps=1e-5, rope_theta=1e4, dtype=BF16,
                      tie_embeddings=False)


def tiny_shape(dtype: str = F16, n_layers: int = 2, hidden: int = 128, n_q_heads: int = 4,
               n_kv_heads: int = 2, head_dim: int = 32, ffn: int = 192, vocab: int = 96,
               tie: bool = True, theta: float = 1e4) -> ModelShape:
    return ModelShape(hidden=hidden, n_layers=n_layers, n_q_heads=n_q_heads,
                      n_kv_heads=n_kv_heads, head_dim=head_dim, ffn=ffn, vocab=vocab,
                      rms_eps=1e-6, rope_theta=theta, dtype=dtype, tie_embeddings=tie)


LAYER_KEYS = ("attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up", "w_down")


def model_weights(shape: ModelShape, seed: int, std: float = 0.02,
                  gamma_std: float = 0.0) -> Dict[str, object]:
    """Seeded weights: linear and embedding ~N(0, std); RMSNorm gains 1 (or N(1, gamma_std)).

    Linear weights are row-major [out_features][in_features] (y = x W^T).
    """
    dt = shape.dtype
    h = shape.hidden

    def gain(name):
        if gamma_std == 0.0:
            return to_storage(np.ones(h), dt)
        return normal(seed, name, (h,), dt, std=gamma_std, mean=1.0)

    layers = []
    for l in range(shape.n_layers):
        p = f"layer{l}."
        layers.append({
            "attn_norm": gain(p + "attn_norm"),
            "wq": normal(seed, p + "wq", (shape.q_dim, h), dt, std),
            "wk": normal(seed, p + "wk", (shape.kv_dim, h), dt, std),
            "wv": normal(seed, p + "wv", (shape.kv_dim, h), dt, std),
            "wo": normal(seed, p + "wo", (h, shape.q_dim), dt, std),
            "ffn_norm": gain(p + "ffn_norm"),
            "w_gate": normal(seed, p + "w_gate", (shape.ffn, h), dt, std),
            "w_up": normal(seed, p + "w_up", (shape.ffn, h), dt, std),
            "w_down": normal(seed, p + "w_down", (h, shape.ffn), dt, std),
        })
    return {
        "embed": normal(seed, "embed", (shape.vocab, h), dt, std),
        "final_norm": gain("final_norm"),
        "lm_head": None if shape.tie_embeddings else normal(seed, "lm_head", (shape.vocab, h),
                                                            dt, std),
        "layers": layers,
    }


# --------------------------------------------------------------------------------------------
# Paged-cache request mixes
# --------------------------------------------------------------------------------------------

@dataclasses.dataclass
class DecodeBatch:
    """One decode step's metadata for ``batch`` requests over a paged cache.

    ``ctx[b]`` cached tokens precede this step's token, which sits at position ``ctx[b]``;
    ``seq_lens = ctx + 1`` counts the cached tokens including this step's token.
    """
    token_ids: np.ndarray      # int32 [B]
    positions: np.ndarray      # int32 [B]
    seq_lens: np.ndarray       # int32 [B]
    block_tables: np.ndarray   # int32 [B, max_blocks_per_seq]; unused entries are 0
    slot_mapping: np.ndarray   # int64 [B]
    num_blocks: int
    block_size: int

    @property
    def batch(self) -> int:
        return int(self.token_ids.shape[0])


def decode_batch(seed: int, name: str, ctx: Sequence[int], vocab: int, block_size: int,
                 num_blocks: Optional[int] = None, max_blocks_per_seq: Optional[int] = None,
                 shared_table_rows: Optional[Sequence[int]] = None) -> DecodeBatch:
    """Assign physical blocks to requests from a shuffled free list.

    Each request b gets ceil((ctx[b] + 1) / block_size) blocks, so the block holding this
    step's token is already in its table.  Blocks are handed out in the order of a seeded
    permutation of the pool, so logical neighbours are scattered physically.
    ``shared_table_rows[b] = a`` makes row b reuse row a's blocks (prefill pseudo-requests).
    """
    ctx = np.asarray(ctx, dtype=np.int64)
    B = ctx.shape[0]
    need = (ctx + 1 + block_size - 1) // block_size
    own = np.ones(B, dtype=bool)
    if shared_table_rows is not None:
        own = np.array([shared_table_rows[b] == b for b in range(B)], dtype=bool)
    total = int(need[own].sum())
    if num_blocks is None:
        num_blocks = total
    if total > num_blocks:
        raise ValueError("pool too small for the requested contexts")
    mb = int(need.max()) if max_blocks_per_seq is None else max_blocks_per_seq
    perm = permutation(seed, name + ".pool", num_blocks)
    tables = np.zeros((B, mb), dtype=np.int32)
    cursor = 0
    for b in range(B):
        if own[b]:
            n = int(need[b])
            tables[b, :n] = perm[cursor:cursor + n]
            cursor += n
    for b in range(B):
        if not own[b]:
            a = shared_table_rows[b]
            tables[b] = tables[a]
    positions = ctx.astype(np.int32)
    seq_lens = (ctx + 1).astype(np.int32)
    blk = tables[np.arange(B), positions // block_size].astype(np.int64)
    slots = blk * block_size + positions % block_size
    toks = uniform_int(seed, name + ".tokens", B, 0, vocab - 1).astype(np.int32)
    return DecodeBatch(token_ids=toks, positions=positions, seq_lens=seq_lens,
                       block_tables=tables, slot_mapping=slots.astype(np.int64),
                       num_blocks=num_blocks, block_size=block_size)


def kv_pool(seed: int, name: str, num_blocks: int, n_kv_heads: int, block_size: int,
            head_dim: int, dtype: str, std: float = 1.0) -> np.ndarray:
    """A [num_blocks, n_kv_heads, block_size, head_dim] pool drawn N(0, std)."""
    return normal(seed, name, (num_blocks, n_kv_heads, block_size, head_dim), dtype, std)


def storage_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Widen fp16 / bf16-bits to fp64 (exact).  Harness convenience; the oracle has its own."""
    if dtype == F16:
        return np.asarray(x, dtype=np.float16).astype(np.float64)
    u = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


CONFIG_SEED = {0: 1000, 1: 1001, 2: 1002, 3: 1003, 4: 1004}


def config_seed(index: int) -> int:
    return CONFIG_SEED[index]


def ctx_uniform(seed: int, name: str, batch: int, lo: int, hi: int) -> np.ndarray:
    return uniform_int(seed, name, batch, lo, hi)


def ctx_log_uniform(seed: int, name: str, batch: int, lo: int, hi: int) -> np.ndarray:
    return log_uniform_int(seed, name, batch, lo, hi)


__all__: List[str] = [n for n in dir() if not n.startswith("_")]


# --------------------------------------------------------------------------------------------
# Device-side draws (same generator, for pools and weights too large to draw on the host)
# --------------------------------------------------------------------------------------------

_FILL_LIB = None


def _fill_lib():
    global _FILL_LIB
    if _FILL_LIB is None:
        import ctypes
        import os
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libsynth.so")
        if not os.path.exists(path):
            build_fill()
        L = ctypes.CDLL(path)
        L.synth_fill_normal.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_ulonglong,
                                        ctypes.c_ulonglong, ctypes.c_double, ctypes.c_double,
                                        ctypes.c_int, ctypes.c_void_p]
        L.synth_fill_normal.restype = ctypes.c_int
        _FILL_LIB = L
    return _FILL_LIB


def build_fill(force: bool = False) -> str:
    """Compile synth/csrc/fill.cu into synth/libsynth.so (sm_103a)."""
    import os
    import shutil
    import subprocess
    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "csrc", "fill.cu")
    out = os.path.join(here, "libsynth.so")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-shared", "-Xcompiler",
           "-fPIC", "-cudart", "shared", "-o", out, src]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for fill.cu:\n{r.stderr}")
    return out


def fill_normal_device(ptr: int, count: int, seed: int, name: str, dtype: str, std: float = 1.0,
                       mean: float = 0.0, offset: int = 0, stream: int = 0) -> None:
    """Write ``count`` draws of stream ``name`` (elements offset .. offset+count-1) at device
    address ``ptr`` in storage dtype: the same values ``normal()`` returns on the host."""
    r = _fill_lib().synth_fill_normal(ptr, count, stream_key(seed, name), offset, float(mean),
                                      float(std), 1 if dtype == BF16 else 0, stream or None)
    if r != 0:
        raise RuntimeError(f"synth_fill_normal failed ({r})")


def normal_device(seed: int, name: str, shape: Sequence[int], dtype: str, std: float = 1.0,
                  mean: float = 0.0):
    """A torch CUDA tensor (float16 / bfloat16) holding ``normal(seed, name, shape, ...)``."""
    import torch
    t = torch.empty(tuple(shape), dtype=torch.float16 if dtype == F16 else torch.bfloat16,
                    device="cuda")
    fill_normal_device(t.data_ptr(), t.numel(), seed, name, dtype, std, mean,
                       stream=torch.cuda.current_stream().cuda_stream)
    return t


_HOST_LIB = None


def build_host(force: bool = False) -> str:
    """Compile synth/csrc/fill_host.c into synth/libsynth_host.so (gcc, no FP contraction)."""
    import os
    import shutil
    import subprocess
    here = os.path.dirname(os.path.abspath(__file__))
    src = os.path.join(here, "csrc", "fill_host.c")
    out = os.path.join(here, "libsynth_host.so")
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    cc = shutil.which("gcc") or shutil.which("cc") or "gcc"
    cmd = [cc, "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-pthread",
           "-o", out, src, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"gcc failed for fill_host.c:\n{r.stderr}")
    return out


def _host_lib():
    global _HOST_LIB
    if _HOST_LIB is None:
        import ctypes
        L = ctypes.CDLL(build_host())
        L.synth_fill_normal_host.argtypes = [ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_ulonglong,
                                             ctypes.c_ulonglong, ctypes.c_double, ctypes.c_double,
                                             ctypes.c_int, ctypes.c_int]
        L.synth_fill_normal_host.restype = ctypes.c_int
        _HOST_LIB = L
    return _HOST_LIB


def normal_threads(seed: int, name: str, shape: Sequence[int], dtype: str, std: float = 1.0,
                   mean: float = 0.0, offset: int = 0, threads: int = 0) -> np.ndarray:
    """``normal()`` computed by the C twin on ``threads`` host threads (0: every core this
    process may use).  Same definition; both sides call their platform's own log/cos/sqrt in
    fp64, so an element can differ only where the two round a transcendental differently in
    the last fp64 bit and that bit decides the 16-bit rounding."""
    import os
    n = int(np.prod(shape)) if len(shape) else 1
    out = np.empty(n, dtype=np.float16 if dtype == F16 else np.uint16)
    t = threads if threads > 0 else len(os.sched_getaffinity(0))
    r = _host_lib().synth_fill_normal_host(out.ctypes.data, n, stream_key(seed, name), offset,
                                           float(mean), float(std), 1 if dtype == BF16 else 0, t)
    if r != 0:
        raise RuntimeError(f"synth_fill_normal_host failed ({r})")
    return out.reshape(shape)


def model_weights_device(shape: ModelShape, seed: int, std: float = 0.02,
                         gamma_std: float = 0.0) -> Dict[str, object]:
    """``model_weights`` drawn on the GPU (same values), as torch CUDA tensors."""
    import torch
    tdt = torch.float16 if shape.dtype == F16 else torch.bfloat16
    h = shape.hidden

    def gain(name):
        if gamma_std == 0.0:
            return torch.ones(h, dtype=tdt, device="cuda")
        return normal_device(seed, name, (h,), shape.dtype, std=gamma_std, mean=1.0)

    layers = []
    for l in range(shape.n_layers):
        p = f"layer{l}."
        layers.append({
            "attn_norm": gain(p + "attn_norm"),
            "wq": normal_device(seed, p + "wq", (shape.q_dim, h), shape.dtype, std),
            "wk": normal_device(seed, p + "wk", (shape.kv_dim, h), shape.dtype, std),
            "wv": normal_device(seed, p + "wv", (shape.kv_dim, h), shape.dtype, std),
            "wo": normal_device(seed, p + "wo", (h, shape.q_dim), shape.dtype, std),
            "ffn_norm": gain(p + "ffn_norm"),
            "w_gate": normal_device(seed, p + "w_gate", (shape.ffn, h), shape.dtype, std),
            "w_up": normal_device(seed, p + "w_up", (shape.ffn, h), shape.dtype, std),
            "w_down": normal_device(seed, p + "w_down", (h, shape.ffn), shape.dtype, std),
        })
    return {
        "embed": normal_device(seed, "embed", (shape.vocab, h), shape.dtype, std),
        "final_norm": gain("final_norm"),
        "lm_head": None if shape.tie_embeddings else normal_device(seed, "lm_head",
                                                                   (shape.vocab, h),
                                                                   shape.dtype, std),
        "layers": layers,
    }
