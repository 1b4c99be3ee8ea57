"""The persistent step kernel (ns_set_step_kernel mode 1): one cooperative launch per decode
step of at most 32 rows.  Its logits and the K/V it writes match the oracle at the step
tolerances for every supported head shape, batch 1 to 32 and rows whose attention spans several
16-block units; a row's result does not depend on the rest of the batch (bitwise); a replayed
graph equals the eager launch (bitwise); steps it does not take run the per-stage kernels."""
import numpy as np
import pytest

import synth
from helpers import from_dev, to_dev
from test_gpu_step import Harness, _check_step, _tiny

pytestmark = pytest.mark.gpu


def _persistent(h: Harness) -> Harness:
    h.dev.set_step_kernel(1)
    return h


def _ctx(seed, n, lo, hi):
    return [int(v) for v in synth.uniform_int(seed, f"ctx{n}", n, lo, hi)]


@pytest.mark.parametrize("dtype,tie", [("bf16", True), ("f16", False)])
@pytest.mark.parametrize("ctx", [[300], [0, 5, 16, 300, 31], None])
def test_persistent_step_matches_oracle_head_dim_64(cuda_lib, dtype, tie, ctx):
    """head_dim 64, two q heads per kv head; batch 1, 5 and 32 (contexts up to 1100: rows of up
    to five 16-block attention units merged across CTAs)."""
    ctx = ctx if ctx is not None else _ctx(11, 32, 0, 1100)
    h = _persistent(Harness(_tiny(dtype, tie), 201, ctx))
    _check_step(h)
    assert h.dev.info().kernels_per_step == 1 or h.dev.info().graphs_cached == 1


@pytest.mark.parametrize("n_q,n_kv,dtype", [(8, 2, "bf16"), (8, 1, "f16"), (14, 2, "bf16")])
def test_persistent_step_matches_oracle_other_heads(cuda_lib, n_q, n_kv, dtype):
    """head_dim 128 with 4 and 8 q heads per kv head (the LLaMA groups), and the Qwen group of
    7 at head_dim 64; 24 rows with contexts up to 700."""
    d = 64 if n_q == 14 else 128
    shape = synth.ModelShape(hidden=n_q * d, n_layers=2, n_q_heads=n_q, n_kv_heads=n_kv,
                             head_dim=d, ffn=1280, vocab=1024, rms_eps=1e-5, rope_theta=5e5,
                             dtype=dtype, tie_embeddings=False)
    h = _persistent(Harness(shape, 211 + n_kv, _ctx(13, 24, 0, 700)))
    _check_step(h)


def test_persistent_step_qwen_shape_two_layers_batch1(cuda_lib):
    """The two-layer Qwen2.5-0.5B shape (hidden 896, 14/2 heads, ffn 4864, vocab 151936) at
    batch 1 with 128 cached tokens, and at batch 32 with contexts uniform in [128, 1024]."""
    shape = synth.qwen05b_shape(n_layers=2)
    w = synth.model_weights(shape, synth.config_seed(0))
    _check_step(_persistent(Harness(shape, 221, [128], weights=w)))
    _check_step(_persistent(Harness(shape, 222, _ctx(17, 32, 128, 1024), weights=w)))


def test_persistent_rows_do_not_depend_on_the_batch(cuda_lib):
    """Rows computed in a batch of 32, of 9 and alone: the same logits bitwise."""
    shape = _tiny("bf16")
    ctx = _ctx(19, 32, 0, 900)
    h = _persistent(Harness(shape, 231, ctx, use_graphs=False))
    full = h.run_gpu()
    for rows in (slice(3, 12), slice(31, 32), slice(0, 1)):
        h.upload_pools()
        part = h.run_gpu(rows=rows)
        np.testing.assert_array_equal(part, full[rows])


def test_persistent_graph_replay_equals_eager_bitwise(cuda_lib):
    shape = _tiny("f16")
    ctx = _ctx(23, 20, 0, 600)
    a = _persistent(Harness(shape, 241, ctx, use_graphs=True))
    b = _persistent(Harness(shape, 241, ctx, use_graphs=False))
    ga = a.run_gpu()
    np.testing.assert_array_equal(ga, b.run_gpu())
    assert b.dev.info().kernels_per_step == 1
    a.upload_pools()
    np.testing.assert_array_equal(a.run_gpu(), ga)
    assert a.dev.info().graphs_cached == 1


def test_steps_the_persistent_kernel_does_not_take_run_the_stage_kernels(cuda_lib):
    """33 rows, and nano-batched steps, run the per-stage kernels in mode 1: their logits equal
    a mode-0 handle's bitwise; switching back to mode 0 gives mode 0's results again."""
    shape = _tiny("bf16")
    ctx = _ctx(29, 33, 0, 500)
    ref = Harness(shape, 251, ctx)
    g_ref = ref.run_gpu()
    h = _persistent(Harness(shape, 251, ctx))
    np.testing.assert_array_equal(h.run_gpu(), g_ref)
    h.upload_pools()
    ref.upload_pools()
    r16 = ref.run_gpu(rows=slice(0, 16))
    h.dev.set_nanobatch([8, 8])
    np.testing.assert_array_equal(h.run_gpu(rows=slice(0, 16)), r16)
    h.dev.set_nanobatch(None)
    h.dev.set_step_kernel(0)
    h.upload_pools()
    np.testing.assert_array_equal(h.run_gpu(rows=slice(0, 16)), r16)


def test_persistent_step_with_device_tokens_and_graph_buckets(cuda_lib):
    """Bucketed graphs (a batch of 5 replays the graph of 8 with padding rows) and token ids
    read from the device: the real rows equal an exact eager step bitwise, padding rows write
    no logits, and only the real rows' slots change."""
    import torch
    shape = _tiny("bf16")
    ctx = _ctx(31, 8, 0, 400)
    exact = _persistent(Harness(shape, 261, ctx, use_graphs=False))
    bucket = _persistent(Harness(shape, 261, ctx))
    bucket.dev.set_graph_buckets([8])
    bt = bucket.batch
    n = 5
    ref = exact.run_gpu(rows=slice(0, n))
    ids_dev = to_dev(bt.token_ids[:8].copy())
    bucket.dev.set_token_source(ids_dev)
    big = torch.full((8, shape.vocab), float("nan"), dtype=torch.float32, device="cuda")
    bucket.dev.step(None, bt.positions[:n], bt.block_tables[:n], bt.seq_lens[:n],
                    bt.slot_mapping[:n], big[:n])
    torch.cuda.synchronize()
    assert bucket.dev.device_error() == 0
    got = from_dev(big)
    np.testing.assert_array_equal(got[:n].astype(np.float64), ref)
    assert np.isnan(got[n:]).all()
    ks, _ = bucket.download_pools()
    for l in range(shape.n_layers):
        changed = np.nonzero((ks[l] != bucket.kp[l]).any(axis=(1, 2, 3)))[0]
        assert set(changed.tolist()) <= {int(s) // 16 for s in bt.slot_mapping[:n]}


def test_persistent_step_without_lm_head_writes_the_same_cache(cuda_lib):
    """logits_out NULL: the step stops after the last layer; the K/V it writes equal those of
    the step with the LM head, bitwise."""
    shape = _tiny("f16")
    ctx = _ctx(37, 12, 0, 300)
    a = _persistent(Harness(shape, 271, ctx))
    b = _persistent(Harness(shape, 271, ctx))
    a.run_gpu()
    b.run_gpu(with_logits=False)
    ka, va = a.download_pools()
    kb, vb = b.download_pools()
    for l in range(shape.n_layers):
        np.testing.assert_array_equal(ka[l], kb[l])
        np.testing.assert_array_equal(va[l], vb[l])
