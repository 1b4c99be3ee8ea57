"""Why a 32-layer bf16 model is checked against the fp64 oracle with a 5e-2 logits bound.

The oracle keeps every intermediate in fp64.  A tensor-core implementation in bf16 rounds the
operands of each matrix product (the normalised activations, q, the attention output, the
SwiGLU output) to bf16, whose unit roundoff is 2^-9.  With about six rounded operands per
layer adding independent relative errors to the residual stream, the logits move by roughly
sqrt(6 L) * 2^-9, i.e. ~2.7 % at L = 32 (fp16: 2^-11, ~0.6 % at 24 layers).  This test
measures that effect on the oracle alone (no GPU code): the fp64 oracle step against the same
step with the product operands rounded to bf16, for a 32-layer random-init model.
"""
import numpy as np

import oracle
import synth
from oracle.decode import (from_storage, paged_attention, rms_norm, rope_apply, rope_tables,
                           round_storage, swiglu)


def _operand_rounded_step(model, kp, vp, batch, bs):
    sh = model.shape
    d, hq, hkv = sh.head_dim, sh.n_q_heads, sh.n_kv_heads
    rnd = lambda x: from_storage(round_storage(x, sh.dtype), sh.dtype)  # noqa: E731
    B = len(batch.token_ids)
    x = model.embed[batch.token_ids].copy()
    cos, sin = rope_tables(batch.positions, d, sh.rope_theta)
    blk, off = batch.slot_mapping // bs, batch.slot_mapping % bs
    for l in range(sh.n_layers):
        w = model.layers[l]
        n = rnd(rms_norm(x, w["attn_norm"], sh.rms_eps))
        q = rnd(rope_apply((n @ w["wq"].T).reshape(B, hq, d), cos, sin))
        k = rope_apply((n @ w["wk"].T).reshape(B, hkv, d), cos, sin)
        v = (n @ w["wv"].T).reshape(B, hkv, d)
        kp[l][blk, :, off, :] = round_storage(k, sh.dtype)
        vp[l][blk, :, off, :] = round_storage(v, sh.dtype)
        o = rnd(paged_attention(q, kp[l], vp[l], batch.block_tables, batch.seq_lens,
                                1.0 / np.sqrt(d), dtype=sh.dtype))
        x = x + o.reshape(B, hq * d) @ w["wo"].T
        n2 = rnd(rms_norm(x, w["ffn_norm"], sh.rms_eps))
        x = x + rnd(swiglu(n2 @ w["w_gate"].T, n2 @ w["w_up"].T)) @ w["w_down"].T
    return rnd(rms_norm(x, model.final_norm, sh.rms_eps)) @ model.lm_head.T


def test_bf16_operands_move_32_layer_logits_by_a_few_percent():
    sh = synth.ModelShape(hidden=512, n_layers=32, n_q_heads=8, n_kv_heads=2, head_dim=64,
                          ffn=1408, vocab=1024, rms_eps=1e-5, rope_theta=5e5, dtype="bf16",
                          tie_embeddings=False)
    w = synth.model_weights(sh, 7)
    model = oracle.OracleModel.from_weights(sh, w)
    batch = synth.decode_batch(7, "b", [300, 1000], sh.vocab, 16)
    kp = [synth.kv_pool(7, f"k{l}", batch.num_blocks, 2, 16, 64, "bf16") for l in range(32)]
    vp = [synth.kv_pool(7, f"v{l}", batch.num_blocks, 2, 16, 64, "bf16") for l in range(32)]
    ref = oracle.decode_step(model, [a.copy() for a in kp], [a.copy() for a in vp],
                             batch.token_ids, batch.positions, batch.block_tables,
                             batch.seq_lens, batch.slot_mapping, 16)
    got = _operand_rounded_step(model, [a.copy() for a in kp], [a.copy() for a in vp], batch, 16)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    # beyond the 1e-2 bound that holds for shallow or fp16 models, inside the 5e-2 one
    assert 1e-2 < rel < 5e-2, rel
    assert np.abs(got - ref).max() < 0.2
