"""Shared test plumbing: device copies through PyTorch, error metrics, and one-step harnesses
that drive the library and the oracle on the same seeded inputs."""
from __future__ import annotations

import math

import numpy as np

import oracle
import synth


def rel_l2(got, ref) -> float:
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    return float(np.linalg.norm(got - ref) / (den if den > 0 else 1.0))


def to_dev(a: np.ndarray):
    import torch
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16))
    else:
        t = torch.from_numpy(a)
    return t.cuda()


def from_dev(t, dtype=None) -> np.ndarray:
    a = t.cpu().numpy()
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    return a


def storage_f64(a, dtype):
    return synth.storage_to_f64(a, dtype)


def attention_case(seed, lens, n_q, n_kv, d, dtype, bs=16, extra_blocks=5, mb=None):
    """q, pools and block tables for a decode-attention call (host arrays, storage dtype)."""
    lens = [int(x) for x in lens]
    B = len(lens)
    need = [math.ceil(n / bs) for n in lens]
    nb = sum(need) + extra_blocks
    mb = max(need) if mb is None else mb
    perm = synth.permutation(seed, "attn.pool", nb)
    tables = np.zeros((B, mb), dtype=np.int32)
    c = 0
    for b in range(B):
        tables[b, : need[b]] = perm[c: c + need[b]]
        c += need[b]
    q = synth.normal(seed, "attn.q", (B, n_q, d), dtype)
    kp = synth.normal(seed, "attn.k", (nb, n_kv, bs, d), dtype)
    vp = synth.normal(seed, "attn.v", (nb, n_kv, bs, d), dtype)
    return q, kp, vp, tables, np.array(lens, dtype=np.int32), nb


def run_attention(q, kp, vp, tables, lens, n_q, n_kv, d, dtype, nb, bs=16):
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    dq, dk, dv = to_dev(q), to_dev(kp), to_dev(vp)
    dt, dl = to_dev(tables), to_dev(lens)
    out = torch.zeros_like(dq)
    _lib.attn_decode(dq, dk, dv, dt, dl, out, n_q, n_kv, d, bs, tables.shape[1], nb,
                     1.0 / math.sqrt(d), dtype)
    torch.cuda.synchronize()
    return from_dev(out)


def oracle_attention(q, kp, vp, tables, lens, d, dtype):
    return oracle.paged_attention(storage_f64(q, dtype), kp, vp, tables, lens,
                                  1.0 / math.sqrt(d), dtype=dtype)
