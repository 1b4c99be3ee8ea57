"""Pins of the CPU oracle against things other than itself (CPU only).

Each test checks the oracle against a closed form, a special case that reduces to a library
routine (PyTorch CPU fp64), brute force on tiny inputs, an invariant the method must keep,
or a number printed on the source pages.  They are chosen so that a plausible slip in the
oracle (a dropped term, a wrong sign, a transposed operand, a wrong head grouping or RoPE
pairing, an untied head, a missing residual) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ------------------------------------------------------------------ attention


def _scatter_pool(dense_list, tables, n_kv, bs, d, num_blocks):
    """Place each request's dense [T, Hkv, d] history into a pool through its block table."""
    pool = np.full((num_blocks, n_kv, bs, d), np.nan)
    for b, dense in enumerate(dense_list):
        for t in range(dense.shape[0]):
            pool[tables[b, t // bs], :, t % bs, :] = dense[t]
    return pool


def _paged_case(seed, B, n_q, n_kv, d, bs, lens):
    rng = _rng(seed)
    nblk = [math.ceil(n / bs) for n in lens]
    num_blocks = sum(nblk) + 3
    perm = rng.permutation(num_blocks)
    mb = max(nblk)
    tables = np.zeros((B, mb), dtype=np.int32)
    c = 0
    for b in range(B):
        tables[b, :nblk[b]] = perm[c:c + nblk[b]]
        c += nblk[b]
    kd = [rng.standard_normal((n, n_kv, d)) for n in lens]
    vd = [rng.standard_normal((n, n_kv, d)) for n in lens]
    q = rng.standard_normal((B, n_q, d))
    kp = _scatter_pool(kd, tables, n_kv, bs, d, num_blocks)
    vp = _scatter_pool(vd, tables, n_kv, bs, d, num_blocks)
    return q, kd, vd, kp, vp, tables, np.array(lens, dtype=np.int32)


def test_single_cached_token_returns_its_v():
    q, kd, vd, kp, vp, tables, lens = _paged_case(1, 3, 8, 2, 16, 4, [1, 1, 1])
    o = oracle.paged_attention(q, kp, vp, tables, lens, 0.25)
    for b in range(3):
        for h in range(8):
            g = h // 4
            np.testing.assert_array_equal(o[b, h], vd[b][0, g])


def test_softmax_rows_sum_to_one_and_are_positive():
    rng = _rng(2)
    s = rng.standard_normal((7, 33)) * 30.0
    p = oracle.softmax(s)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert (p > 0).all()
    # shift invariance and the two-element closed form sigmoid(a - b)
    np.testing.assert_allclose(oracle.softmax(s + 5.0), p, rtol=1e-12, atol=1e-15)
    two = oracle.softmax(np.array([[1.3, -0.4]]))
    np.testing.assert_allclose(two[0, 0], 1.0 / (1.0 + math.exp(-1.7)), rtol=1e-14)


@pytest.mark.parametrize("n_q,n_kv", [(8, 2), (4, 4), (6, 1)])
def test_paged_attention_matches_torch_sdpa_on_expanded_kv(n_q, n_kv):
    """Brute force: dense contiguous history, K/V explicitly repeated G times, torch SDPA."""
    bs, d = 4, 16
    lens = [1, 7, 40]
    q, kd, vd, kp, vp, tables, sl = _paged_case(3, 3, n_q, n_kv, d, bs, lens)
    scale = 1.0 / math.sqrt(d)
    o = oracle.paged_attention(q, kp, vp, tables, sl, scale)
    G = n_q // n_kv
    for b in range(3):
        K = torch.from_numpy(kd[b]).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq,T,d]
        V = torch.from_numpy(vd[b]).permute(1, 0, 2).repeat_interleave(G, dim=0)
        Q = torch.from_numpy(q[b])[:, None, :]
        ref = F.scaled_dot_product_attention(Q, K, V, scale=scale)[:, 0, :].numpy()
        np.testing.assert_allclose(o[b], ref, rtol=1e-12, atol=1e-13)


def test_gqa_equals_attention_over_the_expanded_copy():
    """Grouped-query sharing equals attention over the G-times expanded K/V (nanoserve notes)."""
    bs, d, n_q, n_kv = 4, 8, 8, 2
    q, kd, vd, kp, vp, tables, sl = _paged_case(4, 2, n_q, n_kv, d, bs, [9, 13])
    G = n_q // n_kv
    o_gqa = oracle.paged_attention(q, kp, vp, tables, sl, 0.3)
    o_mha = oracle.paged_attention(q, np.repeat(kp, G, axis=1), np.repeat(vp, G, axis=1),
                                   tables, sl, 0.3)
    np.testing.assert_array_equal(o_gqa, o_mha)


def test_all_equal_keys_give_mean_of_v():
    bs, d = 4, 8
    q, kd, vd, kp, vp, tables, sl = _paged_case(5, 2, 4, 2, d, bs, [6, 11])
    kp[:] = 0.7
    o = oracle.paged_attention(q, kp, vp, tables, sl, 0.5)
    for b in range(2):
        for h in range(4):
            np.testing.assert_allclose(o[b, h], vd[b][:, h // 2].mean(0), rtol=1e-12, atol=1e-14)


def test_block_pool_permutation_invariance():
    bs, d = 4, 8
    q, kd, vd, kp, vp, tables, sl = _paged_case(6, 3, 4, 2, d, bs, [5, 16, 23])
    o = oracle.paged_attention(q, kp, vp, tables, sl, 0.4)
    perm = _rng(7).permutation(kp.shape[0])          # new physical id of old block i = perm[i]
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    o2 = oracle.paged_attention(q, kp2, vp2, perm[tables].astype(np.int32), sl, 0.4)
    np.testing.assert_array_equal(o, o2)


def test_attention_reads_only_tokens_before_seq_len():
    bs, d = 4, 8
    q, kd, vd, kp, vp, tables, sl = _paged_case(8, 1, 2, 1, d, bs, [10])
    # slots 10, 11 of the last block are beyond seq_len: poison them
    blk = tables[0, 2]
    kp[blk, :, 2:, :] = 1e9
    vp[blk, :, 2:, :] = np.nan
    o = oracle.paged_attention(q, kp, vp, tables, sl, 0.4)
    assert np.isfinite(o).all()


# ------------------------------------------------------------------ RoPE


def test_rope_identity_at_position_zero_and_norm_preserving():
    rng = _rng(9)
    x = rng.standard_normal((3, 5, 16))
    c, s = oracle.rope_tables(np.zeros(3, dtype=np.int64), 16, 1e4)
    np.testing.assert_array_equal(oracle.rope_apply(x, c, s), x)
    pos = np.array([1, 77, 8191])
    c, s = oracle.rope_tables(pos, 16, 1e6)
    y = oracle.rope_apply(x, c, s)
    pair_norm = lambda z: z[..., :8] ** 2 + z[..., 8:] ** 2  # noqa: E731
    np.testing.assert_allclose(pair_norm(y), pair_norm(x), rtol=1e-12)


def test_rope_is_complex_rotation_of_half_pairs():
    """Closed form: z_i = x_i + j x_{i+d/2} multiplied by exp(j pos theta^(-2i/d))."""
    rng = _rng(10)
    d, theta = 32, 1e6
    pos = np.array([0, 3, 129, 4095])
    x = rng.standard_normal((4, 2, d))
    c, s = oracle.rope_tables(pos, d, theta)
    y = oracle.rope_apply(x, c, s)
    freqs = theta ** (-np.arange(0, d, 2) / d)
    z = (x[..., : d // 2] + 1j * x[..., d // 2:]) * np.exp(1j * pos[:, None, None] * freqs)
    np.testing.assert_allclose(y[..., : d // 2], z.real, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(y[..., d // 2:], z.imag, rtol=1e-10, atol=1e-12)


def test_rope_scores_depend_only_on_relative_position():
    rng = _rng(11)
    d = 16
    q = rng.standard_normal((1, 1, d))
    k = rng.standard_normal((1, 1, d))

    def score(m, n):
        cq, sq = oracle.rope_tables(np.array([m]), d, 1e4)
        ck, sk = oracle.rope_tables(np.array([n]), d, 1e4)
        return float((oracle.rope_apply(q, cq, sq) * oracle.rope_apply(k, ck, sk)).sum())

    base = score(9, 4)
    for shift in (1, 100, 3000):
        assert abs(score(9 + shift, 4 + shift) - base) < 1e-9
    assert abs(score(9, 5) - base) > 1e-6


# ------------------------------------------------------------------ RMSNorm, SwiGLU


def test_rms_norm_matches_torch_and_closed_forms():
    rng = _rng(12)
    x = rng.standard_normal((4, 64)) * 3.0
    g = rng.standard_normal(64)
    ref = F.rms_norm(torch.from_numpy(x), (64,), weight=torch.from_numpy(g), eps=1e-6).numpy()
    np.testing.assert_allclose(oracle.rms_norm(x, g, 1e-6), ref, rtol=1e-12, atol=1e-13)
    c = 0.01
    const = np.full((1, 64), c)
    np.testing.assert_allclose(oracle.rms_norm(const, np.ones(64), 1e-6),
                               c / math.sqrt(c * c + 1e-6), rtol=1e-13)
    y = oracle.rms_norm(x, np.ones(64), 0.0)
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(-1)), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.rms_norm(7.5 * x, g, 0.0), oracle.rms_norm(x, g, 0.0),
                               rtol=1e-12)


def test_silu_and_swiglu():
    x = np.linspace(-20, 20, 101)
    np.testing.assert_allclose(oracle.silu(x), F.silu(torch.from_numpy(x)).numpy(),
                               rtol=1e-13, atol=1e-300)
    assert oracle.silu(np.array([0.0]))[0] == 0.0
    g, u = np.array([2.0, -1.0]), np.array([3.0, 5.0])
    np.testing.assert_allclose(oracle.swiglu(g, u), g / (1 + np.exp(-g)) * u, rtol=1e-15)


# ------------------------------------------------------------------ storage formats


def test_storage_round_trip_matches_torch_rounding():
    rng = _rng(13)
    x = rng.standard_normal(4096) * 7.0
    for dt, tdt in (("f16", torch.float16), ("bf16", torch.bfloat16)):
        mine = oracle.from_storage(oracle.round_storage(x, dt), dt)
        ref = torch.from_numpy(x).to(torch.float32).to(tdt).to(torch.float64).numpy()
        np.testing.assert_array_equal(mine, ref)


def test_storage_rounding_of_exact_midpoints_is_half_to_even():
    """Values exactly halfway between two neighbours of the storage type (IEEE 754 round to
    nearest, ties to even): the fp32 patterns whose dropped 16 bits are 0x8000 (bf16) and the
    fp64 values halfway between fp16 neighbours, with even and odd kept last bits, of both
    signs, and at the edge where the rounding carries into the exponent; checked against torch's
    own conversion and the by-hand results."""
    # bf16: kept part 0x3F80 (1.0, even) and 0x3F81 (odd), 0x3FFF (odd, carries to 0x4000)
    pats = np.array([0x3F808000, 0x3F818000, 0x3FFF8000, 0xBF808000, 0xBF818000,
                     0x3F808001, 0x3F807FFF], dtype=np.uint32)
    x = pats.view(np.float32).astype(np.float64)
    got = oracle.round_storage(x, "bf16")
    np.testing.assert_array_equal(got, [0x3F80, 0x3F82, 0x4000, 0xBF80, 0xBF82, 0x3F81, 0x3F80])
    ref = torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy()
    np.testing.assert_array_equal(got, ref.view(np.uint16))
    # fp16: 1 + 2^-11 lies halfway between 1 and 1 + 2^-10 (ties to 1, the even one);
    # 1 + 3 * 2^-11 halfway between 1 + 2^-10 (odd) and 1 + 2^-9 (even)
    x = np.array([1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, -(1 + 2.0 ** -11), 2047.5 + 0.5])
    got = oracle.from_storage(oracle.round_storage(x, "f16"), "f16")
    np.testing.assert_array_equal(got, [1.0, 1 + 2.0 ** -9, -1.0, 2048.0])
    ref = torch.from_numpy(x).to(torch.float32).to(torch.float16).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, ref)


def test_greedy_argmax_breaks_ties_to_the_lowest_index():
    """Brute force: the first index holding the row maximum, on rows with many exact ties."""
    rng = _rng(17)
    logits = rng.integers(-3, 3, size=(64, 37)).astype(np.float64)
    logits[0] = 5.0                        # every entry ties
    logits[1, [4, 30]] = 9.0               # two maxima
    got = oracle.greedy_argmax(logits)
    for r in range(logits.shape[0]):
        first = next(i for i, v in enumerate(logits[r]) if v == max(logits[r]))
        assert got[r] == first
    assert got[0] == 0 and got[1] == 4


# ------------------------------------------------------------------ whole step


def _torch_step(shape, w, hist_k, hist_v, tokens, positions):
    """An independent PyTorch fp64 statement of the step over dense per-request histories.

    Uses F.rms_norm, F.linear, complex-exponential RoPE, F.scaled_dot_product_attention with
    an explicitly expanded K/V, F.silu; the current token's k/v are rounded through torch's
    own dtype conversion and appended to the history.
    """
    t = lambda a: torch.from_numpy(synth.storage_to_f64(a, shape.dtype))  # noqa: E731
    tdt = torch.float16 if shape.dtype == "f16" else torch.bfloat16
    d, hq, hkv, H = shape.head_dim, shape.n_q_heads, shape.n_kv_heads, shape.hidden
    E = t(w["embed"])
    head = E if w["lm_head"] is None else t(w["lm_head"])
    B = len(tokens)
    x = E[torch.as_tensor(tokens, dtype=torch.long)]
    freqs = shape.rope_theta ** (-torch.arange(0, d, 2, dtype=torch.float64) / d)
    rot = torch.polar(torch.ones(B, d // 2, dtype=torch.float64),
                      torch.as_tensor(positions, dtype=torch.float64)[:, None] * freqs)

    def rope(z):
        c = torch.complex(z[..., : d // 2], z[..., d // 2:]) * rot[:, None, :]
        return torch.cat([c.real, c.imag], dim=-1)

    for l, lw in enumerate(w["layers"]):
        n = F.rms_norm(x, (H,), weight=t(lw["attn_norm"]), eps=shape.rms_eps)
        q = rope(F.linear(n, t(lw["wq"])).view(B, hq, d))
        k = rope(F.linear(n, t(lw["wk"])).view(B, hkv, d))
        v = F.linear(n, t(lw["wv"])).view(B, hkv, d)
        k = k.to(torch.float32).to(tdt).to(torch.float64)
        v = v.to(torch.float32).to(tdt).to(torch.float64)
        outs = []
        for b in range(B):
            K = torch.cat([hist_k[l][b], k[b:b + 1]], 0)
            V = torch.cat([hist_v[l][b], v[b:b + 1]], 0)
            hist_k[l][b], hist_v[l][b] = K, V
            G = hq // hkv
            Ke = K.permute(1, 0, 2).repeat_interleave(G, 0)
            Ve = V.permute(1, 0, 2).repeat_interleave(G, 0)
            o = F.scaled_dot_product_attention(q[b][:, None, :], Ke, Ve, scale=d ** -0.5)
            outs.append(o[:, 0, :].reshape(hq * d))
        x = x + F.linear(torch.stack(outs), t(lw["wo"]))
        n2 = F.rms_norm(x, (H,), weight=t(lw["ffn_norm"]), eps=shape.rms_eps)
        a = F.silu(F.linear(n2, t(lw["w_gate"]))) * F.linear(n2, t(lw["w_up"]))
        x = x + F.linear(a, t(lw["w_down"]))
    nf = F.rms_norm(x, (H,), weight=t(w["final_norm"]), eps=shape.rms_eps)
    return F.linear(nf, head).numpy()


def _step_case(dtype, tie, seed=21, ctx=(0, 5, 17), gamma_std=0.1, bs=4):
    shape = synth.tiny_shape(dtype=dtype, tie=tie, n_layers=2, hidden=64, n_q_heads=4,
                             n_kv_heads=2, head_dim=16, ffn=96, vocab=80)
    w = synth.model_weights(shape, seed, std=0.08, gamma_std=gamma_std)
    batch = synth.decode_batch(seed, "batch", list(ctx), shape.vocab, bs, num_blocks=20,
                               max_blocks_per_seq=8)
    L, B, hkv, d = shape.n_layers, batch.batch, shape.n_kv_heads, shape.head_dim
    kpools, vpools, hist_k, hist_v = [], [], [], []
    for l in range(L):
        kp = synth.kv_pool(seed, f"k{l}", batch.num_blocks, hkv, bs, d, dtype)
        vp = synth.kv_pool(seed, f"v{l}", batch.num_blocks, hkv, bs, d, dtype)
        kpools.append(kp)
        vpools.append(vp)
        hk, hv = [], []
        for b in range(B):
            tt = np.arange(int(batch.positions[b]))
            blk = batch.block_tables[b, tt // bs]
            hk.append(torch.from_numpy(synth.storage_to_f64(kp[blk, :, tt % bs, :], dtype)))
            hv.append(torch.from_numpy(synth.storage_to_f64(vp[blk, :, tt % bs, :], dtype)))
        hist_k.append(hk)
        hist_v.append(hv)
    return shape, w, batch, kpools, vpools, hist_k, hist_v


@pytest.mark.parametrize("dtype,tie", [("f16", True), ("bf16", False)])
def test_decode_step_matches_independent_torch_statement(dtype, tie):
    shape, w, batch, kp, vp, hk, hv = _step_case(dtype, tie)
    model = oracle.OracleModel.from_weights(shape, w)
    logits = oracle.decode_step(model, kp, vp, batch.token_ids, batch.positions,
                                batch.block_tables, batch.seq_lens, batch.slot_mapping,
                                batch.block_size)
    ref = _torch_step(shape, w, hk, hv, batch.token_ids, batch.positions)
    np.testing.assert_allclose(logits, ref, rtol=1e-9, atol=1e-11)
    # the cache now holds this step's k/v at the mapped slots, as the torch history does
    for l in range(shape.n_layers):
        for b in range(batch.batch):
            s = int(batch.slot_mapping[b])
            got = synth.storage_to_f64(kp[l][s // 4, :, s % 4, :], dtype)
            np.testing.assert_array_equal(got, hk[l][b][-1].numpy())


@pytest.mark.parametrize("dtype,tie", [("f16", True), ("bf16", False)])
def test_step_flops_equal_torch_flop_count_of_the_independent_statement(dtype, tie):
    """The roofline's FLOPs of a step (projections, attention QK and PV, LM head) equal what
    PyTorch's own FLOP counter counts while running the independent statement of that step."""
    from torch.utils.flop_counter import FlopCounterMode
    from transformer_decode_step_ns_gb300 import roofline
    shape, w, batch, _, _, hk, hv = _step_case(dtype, tie)
    with FlopCounterMode(display=False) as fc:
        _torch_step(shape, w, hk, hv, batch.token_ids, batch.positions)
    assert fc.get_total_flops() == roofline.decode_step_work(shape, batch.seq_lens).flops


def test_zero_layers_pass_the_embedding_through_to_a_tied_head():
    """With Wo = Wd = 0 the residual stream is the embedding row; a tied head then scores the
    input token itself highest, and the logits equal rs * E[tok] . E^T exactly."""
    shape, w, batch, kp, vp, _, _ = _step_case("f16", True, gamma_std=0.0)
    for lw in w["layers"]:
        lw["wo"] = np.zeros_like(lw["wo"])
        lw["w_down"] = np.zeros_like(lw["w_down"])
    model = oracle.OracleModel.from_weights(shape, w)
    logits = oracle.decode_step(model, kp, vp, batch.token_ids, batch.positions,
                                batch.block_tables, batch.seq_lens, batch.slot_mapping, 4)
    E = synth.storage_to_f64(w["embed"], "f16")
    e = E[batch.token_ids]
    rs = 1.0 / np.sqrt((e * e).mean(-1, keepdims=True) + shape.rms_eps)
    np.testing.assert_allclose(logits, (e * rs) @ E.T, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(oracle.greedy_argmax(logits), batch.token_ids)


def test_decode_rows_are_independent():
    shape, w, batch, kp, vp, _, _ = _step_case("bf16", False)
    model = oracle.OracleModel.from_weights(shape, w)
    kp_all = [a.copy() for a in kp]
    vp_all = [a.copy() for a in vp]
    full = oracle.decode_step(model, kp_all, vp_all, batch.token_ids, batch.positions,
                              batch.block_tables, batch.seq_lens, batch.slot_mapping, 4)
    for b in range(batch.batch):
        sl = slice(b, b + 1)
        kk = [a.copy() for a in kp]
        vv = [a.copy() for a in vp]
        one = oracle.decode_step(model, kk, vv, batch.token_ids[sl], batch.positions[sl],
                                 batch.block_tables[sl], batch.seq_lens[sl],
                                 batch.slot_mapping[sl], 4)
        np.testing.assert_allclose(one[0], full[b], rtol=1e-12, atol=1e-13)


def test_uniform_attention_closed_form_through_the_whole_step():
    """Wq = 0 makes every score 0, so each q head's attention output is the plain mean of its
    kv head's V over the request's tokens t < seq_len, this step's own v included; with
    Wd = 0 and unit gains the layer is x += Wo . concat_h mean(V[:, h // G]) and the tied head
    gives rms(x) . E^T.  Written with np.mean over the dense histories (no softmax, no pool),
    so a wrong head grouping, an off-by-one seq_len, a missing write of this step's v before
    attending, or a rotation of v fails here."""
    shape, w, batch, kp, vp, _, hv = _step_case("f16", True, gamma_std=0.0)
    for lw in w["layers"]:
        lw["wq"] = np.zeros_like(lw["wq"])
        lw["w_down"] = np.zeros_like(lw["w_down"])
    model = oracle.OracleModel.from_weights(shape, w)
    logits = oracle.decode_step(model, kp, vp, batch.token_ids, batch.positions,
                                batch.block_tables, batch.seq_lens, batch.slot_mapping, 4)
    f64 = lambda a: synth.storage_to_f64(a, "f16")  # noqa: E731
    E = f64(w["embed"])
    hq, hkv, d, H = shape.n_q_heads, shape.n_kv_heads, shape.head_dim, shape.hidden
    G = hq // hkv
    rms = lambda z: z / np.sqrt((z * z).mean(-1, keepdims=True) + shape.rms_eps)  # noqa: E731
    x = E[batch.token_ids]
    for l, lw in enumerate(w["layers"]):
        v_new = rms(x) @ f64(lw["wv"]).T
        v_new = torch.from_numpy(v_new).to(torch.float32).to(torch.float16).double().numpy()
        o = np.zeros((batch.batch, hq * d))
        for b in range(batch.batch):
            V = np.concatenate([hv[l][b].numpy(), v_new[b].reshape(1, hkv, d)], 0)
            for h in range(hq):
                o[b, h * d:(h + 1) * d] = V[:, h // G, :].mean(0)
        x = x + o @ f64(lw["wo"]).T
    np.testing.assert_allclose(logits, rms(x) @ E.T, rtol=1e-9, atol=1e-11)


def test_prompt_chunk_equals_feeding_its_tokens_one_step_at_a_time():
    """A prompt chunk (rows of one request at consecutive positions over one block table, all
    in one step) is the same computation as decoding those tokens one per step: each row sees
    the cached tokens and the chunk's earlier rows, never its later ones (NanoFlow page,
    "Runtime details that keep the pipeline fed": prompts enter the dense batch as chunks
    next to decode rows).  Checked on logits and on the K/V left in the cache, with a decode
    row of another request in the same step."""
    bs, ctx0, n_chunk = 4, 5, 6
    shape, w, batch, kp, vp, _, _ = _step_case("bf16", False, ctx=(ctx0, 9))
    model = oracle.OracleModel.from_weights(shape, w)
    rng = _rng(31)
    chunk = rng.integers(0, shape.vocab, n_chunk).astype(np.int32)
    table = batch.block_tables[0].copy()
    assert (ctx0 + n_chunk + bs - 1) // bs <= len(table)
    # give the chunk's later positions blocks of their own (free blocks of the pool)
    used = set(batch.block_tables[:, :].ravel().tolist())
    n_have = (ctx0 + 1 + bs - 1) // bs
    free = [blk for blk in range(batch.num_blocks) if blk not in used]
    for i in range(n_have, (ctx0 + n_chunk + bs - 1) // bs):
        table[i] = free.pop()
    pos = np.arange(ctx0, ctx0 + n_chunk, dtype=np.int32)
    slots = np.array([table[p // bs] * bs + p % bs for p in pos], dtype=np.int64)

    # one step: the decode row of request 1, then the chunk of request 0
    kc = [a.copy() for a in kp]
    vc = [a.copy() for a in vp]
    tok = np.concatenate([batch.token_ids[1:2], chunk])
    posn = np.concatenate([batch.positions[1:2], pos])
    tabs = np.stack([batch.block_tables[1]] + [table] * n_chunk)
    lens = posn + 1
    sl = np.concatenate([batch.slot_mapping[1:2], slots])
    together = oracle.decode_step(model, kc, vc, tok, posn, tabs, lens, sl, bs)

    # the same tokens, one step each
    ks = [a.copy() for a in kp]
    vs = [a.copy() for a in vp]
    one_by_one = []
    for i in range(n_chunk):
        one_by_one.append(oracle.decode_step(model, ks, vs, chunk[i:i + 1], pos[i:i + 1],
                                             table[None], pos[i:i + 1] + 1, slots[i:i + 1],
                                             bs)[0])
    alone = oracle.decode_step(model, ks, vs, batch.token_ids[1:2], batch.positions[1:2],
                               batch.block_tables[1:2], batch.seq_lens[1:2],
                               batch.slot_mapping[1:2], bs)[0]
    np.testing.assert_allclose(together[1:], np.stack(one_by_one), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(together[0], alone, rtol=1e-9, atol=1e-11)
    for l in range(shape.n_layers):
        for a, b in ((kc[l], ks[l]), (vc[l], vs[l])):
            np.testing.assert_allclose(synth.storage_to_f64(a, "bf16"),
                                       synth.storage_to_f64(b, "bf16"), rtol=2 ** -7, atol=0)
    # and the chunk is causal: changing its last token changes no earlier row
    chunk2 = chunk.copy()
    chunk2[-1] = (chunk2[-1] + 1) % shape.vocab
    tok2 = np.concatenate([batch.token_ids[1:2], chunk2])
    other = oracle.decode_step(model, [a.copy() for a in kp], [a.copy() for a in vp], tok2,
                               posn, tabs, lens, sl, bs)
    np.testing.assert_array_equal(other[:-1], together[:-1])
    assert np.abs(other[-1] - together[-1]).max() > 1e-3


def test_qwen_shape_weight_bytes_match_the_printed_943_mib():
    g = json.load(open(os.path.join(GOLDEN, "pages_numbers.json")))["qwen05b_fp16_weights_mib"]
    mib = oracle.param_bytes(synth.qwen05b_shape()) / 2 ** 20
    assert abs(mib - g["value"]) <= g["tolerance_mib"]
    # the untied variant would be far off, which pins the tied head
    untied = synth.dataclasses.replace(synth.qwen05b_shape(), tie_embeddings=False)
    assert oracle.param_bytes(untied) / 2 ** 20 > g["value"] + 200
