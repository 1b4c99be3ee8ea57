"""Roofline and step-cost arithmetic used by the benchmark.

Sources: "The roofline flips: why optimising small models is a different performance game",
sections "The bare mechanism: what the roofline says" (arithmetic intensity, the two
ceilings and the ridge point; decode AI ~ 2B FLOP/byte) and "The point of the title" /
"The maths that matter: a 3B on a 4090" (T_step ~ weight bytes / BW + T_fixed);
"The chef who calls out every order ...", "The maths that matters: when the GPU is left
waiting" (launch time = kernels x per-launch cost); "NanoFlow: LLM Serving Is Compute
Bound ...", opening section (compute-bound optimum = peak FLOPS / (2 n_params)).

The step roofline of the decode step is max(FLOPs / tensor peak, bytes / HBM bandwidth) over
the algorithmic work only: weights read once, cached K/V read once, new K/V and logits
written once.
"""
from __future__ import annotations

import dataclasses
from typing import Sequence


def ai_ridge(peak_flops: float, bandwidth: float) -> float:
    """Arithmetic intensity (FLOP/byte) where the memory and compute ceilings meet."""
    return peak_flops / bandwidth


def roofline_perf(peak_flops: float, bandwidth: float, ai: float) -> float:
    """Attainable FLOP/s = min(peak, BW x AI)."""
    return min(peak_flops, bandwidth * ai)


def ai_decode(batch: int) -> float:
    """Decode weight-GEMM intensity as the roofline page states it: ~2 FLOP per weight byte at
    batch 1, growing linearly with the batch that shares each weight read."""
    return 2.0 * batch


def t_hbm(nbytes: float, bandwidth: float) -> float:
    return nbytes / bandwidth


def t_step(nbytes: float, bandwidth: float, t_fixed: float) -> float:
    return nbytes / bandwidth + t_fixed


def t_launch(n_kernels: int, per_launch_s: float) -> float:
    return n_kernels * per_launch_s


def optimal_tokens_per_s(peak_flops: float, n_params: float) -> float:
    return peak_flops / (2.0 * n_params)


def step_roofline_time(flops: float, nbytes: float, peak_flops: float, bandwidth: float) -> float:
    return max(flops / peak_flops, nbytes / bandwidth)


@dataclasses.dataclass
class StepWork:
    weight_bytes: float
    kv_read_bytes: float
    kv_write_bytes: float
    act_bytes: float
    logits_bytes: float
    flops: float

    @property
    def total_bytes(self) -> float:
        return (self.weight_bytes + self.kv_read_bytes + self.kv_write_bytes + self.act_bytes
                + self.logits_bytes)


def decode_step_work(shape, seq_lens: Sequence[int], elt_bytes: int = 2,
                     n_layers: int = None) -> StepWork:
    """Algorithmic bytes and FLOPs of one decode step over ``len(seq_lens)`` rows.

    Weights: every linear weight once, plus the LM head (the embedding when tied; the embedding
    gather itself reads B rows).  KV read: sum_b seq_len_b * L * 2 * Hkv * d * elt.  FLOPs:
    2 * B * (linear params + LM head) + 4 * L * Hq * d * sum_b seq_len_b.
    """
    L = shape.n_layers if n_layers is None else n_layers
    B = len(seq_lens)
    h, f, d = shape.hidden, shape.ffn, shape.head_dim
    qd, kvd = shape.n_q_heads * d, shape.n_kv_heads * d
    lin_per_layer = h * qd + 2 * h * kvd + qd * h + 3 * h * f
    head = shape.vocab * h
    weights = (L * (lin_per_layer + 2 * h) + head + h) * elt_bytes
    ctx_total = float(sum(int(s) for s in seq_lens))
    kv_read = ctx_total * L * 2 * kvd * elt_bytes
    kv_write = B * L * 2 * kvd * elt_bytes
    act = B * h * elt_bytes
    logits = B * shape.vocab * 4
    flops = 2.0 * B * (L * lin_per_layer + head) + 4.0 * L * qd * ctx_total
    return StepWork(weights, kv_read, kv_write, act, logits, flops)


def attention_bytes(seq_lens: Sequence[int], n_kv_heads: int, head_dim: int,
                    elt_bytes: int = 2) -> float:
    """Algorithmic K+V bytes one decode-attention launch reads."""
    return float(sum(int(s) for s in seq_lens)) * n_kv_heads * head_dim * 2 * elt_bytes
