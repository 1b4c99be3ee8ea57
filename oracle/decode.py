"""Plain fp64 definition of one pre-norm decoder decode step over a paged KV cache.

Test infrastructure only (see the package docstring).  Sources, by page title and section:

* "GPU waiting, not working" (nanoserve notes), table under "What I changed because of it":
  RoPE cos/sin built once per step because positions are shared by all layers; a fused
  RMSNorm; grouped-query attention without materialising the expanded K/V copy; one pinned
  host-to-device copy for step metadata; a faster token-to-cache-slot mapping; a fused paged
  attention kernel.  "The number that didn't fit": Qwen2.5-0.5B in fp16 is 943 MiB of weights.
* "NanoFlow: LLM Serving Is Compute Bound, and Your GPU Is Half Idle", "Four resource classes,
  one serialized queue": the layer's dense operators are the KQV projection, O projection,
  Up, Gate and Down; attention is the memory-bound decode attention; "Other" is the norm and
  RoPE.  "Nano-batching: manufacturing independence": different rows of the activation
  matrix are independent.

Readings where the pages are silent (each listed in the design notes): RMSNorm is
x / sqrt(mean(x^2) + eps) * gamma; RoPE pairs element i with i + d/2 ("rotate half") with
inverse frequency theta^(-2i/d); kv head of q head h is floor(h / G); the softmax scale is
1/sqrt(d); this step's token attends to itself; the FFN is SwiGLU, down(silu(gate) * up);
the LM head is tied to the embedding when the model says so; logits are fp32 on the GPU.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Optional, Sequence

import numpy as np

F16 = "f16"
BF16 = "bf16"


# ------------------------------------------------------------------------------------------
# storage formats (the cache and the weights are fp16 / bf16; the oracle computes in fp64)
# ------------------------------------------------------------------------------------------

def from_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of fp16 values or bf16 bit patterns (uint16) to fp64."""
    if dtype == F16:
        return np.asarray(x, dtype=np.float16).astype(np.float64)
    if dtype == BF16:
        bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def round_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp64 -> fp32 -> storage type, nearest-even at each step (IEEE 754 rounding).

    bf16 keeps the top 16 bits of the fp32 pattern; rounding adds 0x7fff plus the lowest kept
    bit before truncating, which is round-half-to-even on the dropped 16 bits.
    """
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    if dtype == F16:
        return x32.astype(np.float16)
    if dtype == BF16:
        u = np.ascontiguousarray(x32).view(np.uint32).astype(np.uint64)
        keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
        return ((u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)).astype(np.uint16)
    raise ValueError(dtype)


# ------------------------------------------------------------------------------------------
# the per-token operators
# ------------------------------------------------------------------------------------------

def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last axis ("fused RMSNorm", nanoserve notes, the change table).

    y = x / sqrt(mean(x^2) + eps) * gamma: no mean subtraction, no bias.
    """
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * gamma


def rope_tables(positions: Sequence[int], head_dim: int, theta: float):
    """cos/sin tables [B, d/2], built once per step and shared by every layer (nanoserve
    notes, the change table: positions are the same in all layers).

    inv_freq_i = theta^(-2i/d) for i < d/2; angle = position * inv_freq_i; fp64 throughout.
    """
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    inv_freq = np.power(float(theta), -2.0 * i / head_dim)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.cos(ang), np.sin(ang)


def rope_apply(x: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate each head of x [B, n_heads, d] by its token's angles, pairing i with i + d/2.

    (x_i, x_{i+d/2}) -> (x_i cos - x_{i+d/2} sin, x_{i+d/2} cos + x_i sin).
    """
    half = x.shape[-1] // 2
    lo, hi = x[..., :half], x[..., half:]
    c, s = cos[:, None, :], sin[:, None, :]
    return np.concatenate([lo * c - hi * s, hi * c + lo * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    """silu(x) = x * sigmoid(x)."""
    return x / (1.0 + np.exp(-x))


def swiglu(gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """The gated FFN activation silu(x W_gate^T) * (x W_up^T) ("Up/Gate", NanoFlow page,
    dense operator class)."""
    return silu(gate) * up


def gqa_group(h: int, n_q_heads: int, n_kv_heads: int) -> int:
    """KV head serving q head h: contiguous groups of G = Hq / Hkv q heads share one kv head
    (nanoserve notes: grouped-query attention instead of a G-times expanded K/V copy)."""
    return h // (n_q_heads // n_kv_heads)


def slot_of(block_table_row: np.ndarray, pos: int, block_size: int) -> int:
    """Physical cache slot of logical position pos: table[pos // bs] * bs + pos % bs
    (nanoserve notes: mapping tokens to cache slots; NanoFlow page: PagedAttention pages)."""
    return int(block_table_row[pos // block_size]) * block_size + pos % block_size


def softmax(s: np.ndarray) -> np.ndarray:
    """Max-subtracted softmax over the last axis."""
    e = np.exp(s - np.max(s, axis=-1, keepdims=True))
    return e / np.sum(e, axis=-1, keepdims=True)


def attention_weights(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """p_t = softmax_t(q . k_t * scale) for one query vector q [d] over keys k [T, d]."""
    return softmax((k @ q) * scale)


def dense_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """o = sum_t p_t v_t for one query over contiguous keys/values [T, d]."""
    return attention_weights(q, k, scale) @ v


def gather_tokens(pool: np.ndarray, block_table_row: np.ndarray, seq_len: int, kv_head: int,
                  block_size: int) -> np.ndarray:
    """Tokens 0..seq_len-1 of one kv head from a [num_blocks, Hkv, bs, d] pool, in logical
    order, read through the block table."""
    t = np.arange(seq_len)
    return pool[block_table_row[t // block_size], kv_head, t % block_size, :]


def paged_attention(q: np.ndarray, k_pool: np.ndarray, v_pool: np.ndarray,
                    block_tables: np.ndarray, seq_lens: np.ndarray, scale: float,
                    dtype: Optional[str] = None) -> np.ndarray:
    """Decode attention over a paged cache (nanoserve notes: the fused paged-attention kernel;
    NanoFlow page: decode attention is the memory-bound class).

    q [B, Hq, d] (fp64); pools [num_blocks, Hkv, bs, d], either fp64 or in storage format
    ``dtype``; for each request b and q head h, keys/values are tokens t < seq_lens[b] of kv
    head floor(h / G).  Returns o [B, Hq, d] in fp64.
    """
    B, n_q, d = q.shape
    n_kv, bs = k_pool.shape[1], k_pool.shape[2]
    out = np.zeros((B, n_q, d))
    for b in range(B):
        n = int(seq_lens[b])
        for g in range(n_kv):
            kk = gather_tokens(k_pool, block_tables[b], n, g, bs)
            vv = gather_tokens(v_pool, block_tables[b], n, g, bs)
            if dtype is not None:
                kk, vv = from_storage(kk, dtype), from_storage(vv, dtype)
            for h in range(n_q):
                if gqa_group(h, n_q, n_kv) == g:
                    out[b, h] = dense_attention(q[b, h], kk, vv, scale)
    return out


def greedy_argmax(logits: np.ndarray) -> np.ndarray:
    """Index of the largest logit per row; ties go to the lowest index."""
    return np.argmax(logits, axis=-1).astype(np.int32)


def param_bytes(shape, bytes_per_param: int = 2) -> int:
    """Weight bytes of the model (the nanoserve notes quote 943 MiB for Qwen2.5-0.5B fp16)."""
    return shape.param_count() * bytes_per_param


# ------------------------------------------------------------------------------------------
# the whole step
# ------------------------------------------------------------------------------------------

@dataclasses.dataclass
class OracleModel:
    """fp64 copies of a model's weights; ``shape`` carries the dims, eps, theta and dtype."""
    shape: object
    embed: np.ndarray
    final_norm: np.ndarray
    lm_head: np.ndarray
    layers: List[Dict[str, np.ndarray]]

    @classmethod
    def from_weights(cls, shape, weights) -> "OracleModel":
        dt = shape.dtype
        wid = lambda a: from_storage(a, dt)  # noqa: E731
        layers = [{k: wid(v) for k, v in lw.items()} for lw in weights["layers"]]
        embed = wid(weights["embed"])
        head = embed if weights["lm_head"] is None else wid(weights["lm_head"])
        return cls(shape=shape, embed=embed, final_norm=wid(weights["final_norm"]),
                   lm_head=head, layers=layers)


def decode_step(model: OracleModel, k_pools: List[np.ndarray], v_pools: List[np.ndarray],
                token_ids: np.ndarray, positions: np.ndarray, block_tables: np.ndarray,
                seq_lens: np.ndarray, slot_mapping: np.ndarray, block_size: int,
                trace: Optional[dict] = None, n_layers: Optional[int] = None) -> np.ndarray:
    """One decode step for a batch of requests; returns fp64 logits [B, vocab].

    ``k_pools[l]`` / ``v_pools[l]`` are layer l's caches [num_blocks, Hkv, bs, d] in storage
    format; this step's k and v are written into them at ``slot_mapping`` rounded to the
    storage type (the GPU stores them in that type and attends over the stored values).

    Per layer, in the order of a pre-norm decoder (NanoFlow page, dense classes KQV, O,
    Up/Gate, Down; "Other" is the norm and RoPE):
      n = RMSNorm(x; attn_norm); q, k, v = n Wq^T, n Wk^T, n Wv^T; RoPE(q), RoPE(k);
      cache[slot] <- k, v; o = attention over the request's tokens t < seq_len;
      x += o Wo^T; n = RMSNorm(x; ffn_norm); x += (silu(n Wg^T) * (n Wu^T)) Wd^T.
    Then logits = RMSNorm(x; final_norm) W_lm^T.  All rows' k/v are written before any row
    attends, so rows sharing a block table (a prefill chunk) see each other causally.

    ``trace``, when given, receives per layer (lists indexed by layer, fp64, before any
    storage rounding): "q" and "k" after RoPE [B, heads, d], "v", "attn" (o) [B, Hq, d],
    "resid_attn" (x after the attention block) and "resid" (x after the layer) [B, H].
    ``n_layers`` runs only the first layers before the final norm and head.
    """
    sh = model.shape
    dt = sh.dtype
    d, hq, hkv = sh.head_dim, sh.n_q_heads, sh.n_kv_heads
    B = len(token_ids)
    bs = block_size
    scale = 1.0 / np.sqrt(d)
    x = model.embed[np.asarray(token_ids, dtype=np.int64)].copy()
    cos, sin = rope_tables(positions, d, sh.rope_theta)
    blk = np.asarray(slot_mapping, dtype=np.int64) // bs
    off = np.asarray(slot_mapping, dtype=np.int64) % bs
    L = sh.n_layers if n_layers is None else n_layers
    for l in range(L):
        w = model.layers[l]
        n = rms_norm(x, w["attn_norm"], sh.rms_eps)
        q = (n @ w["wq"].T).reshape(B, hq, d)
        k = (n @ w["wk"].T).reshape(B, hkv, d)
        v = (n @ w["wv"].T).reshape(B, hkv, d)
        q = rope_apply(q, cos, sin)
        k = rope_apply(k, cos, sin)
        k_pools[l][blk, :, off, :] = round_storage(k, dt)
        v_pools[l][blk, :, off, :] = round_storage(v, dt)
        o = paged_attention(q, k_pools[l], v_pools[l], block_tables, seq_lens, scale, dtype=dt)
        x = x + o.reshape(B, hq * d) @ w["wo"].T
        x_attn = x
        n2 = rms_norm(x, w["ffn_norm"], sh.rms_eps)
        a = swiglu(n2 @ w["w_gate"].T, n2 @ w["w_up"].T)
        x = x + a @ w["w_down"].T
        if trace is not None:
            trace.setdefault("q", []).append(q)
            trace.setdefault("k", []).append(k)
            trace.setdefault("v", []).append(v)
            trace.setdefault("attn", []).append(o)
            trace.setdefault("resid_attn", []).append(x_attn.copy())
            trace.setdefault("resid", []).append(x.copy())
    nf = rms_norm(x, model.final_norm, sh.rms_eps)
    return nf @ model.lm_head.T
