"""GPU parity of the whole decode step (ns_decode_step) against the oracle, plus the step's
bitwise properties: graph replay equals eager launch, nano-batched equals unsplit, and only
this step's slots of the KV cache change."""
import math

import numpy as np
import pytest

import oracle
import synth
from helpers import from_dev, rel_l2, storage_f64, to_dev

pytestmark = pytest.mark.gpu


def _tiny(dtype="bf16", tie=True, n_layers=2):
    return synth.ModelShape(hidden=256, n_layers=n_layers, n_q_heads=4, n_kv_heads=2, head_dim=64,
                            ffn=384, vocab=512, rms_eps=1e-6, rope_theta=1e4, dtype=dtype,
                            tie_embeddings=tie)


class Harness:
    """One model on the device and the same model + cache in the oracle."""

    def __init__(self, shape, seed, ctx, bs=16, extra_blocks=4, max_batch=None, mb=None,
                 use_graphs=True, gamma_std=0.1, weights=None, kv_std=1.0,
                 shared_table_rows=None):
        from transformer_decode_step_ns_gb300 import _lib
        self.shape, self.bs = shape, bs
        self.w = weights if weights is not None else synth.model_weights(shape, seed, gamma_std=gamma_std)
        need = sum(math.ceil((c + 1) / bs) for c in ctx)
        self.num_blocks = need + extra_blocks
        mb = mb or max(math.ceil((c + 1) / bs) for c in ctx) + 1
        self.batch = synth.decode_batch(seed, "batch", list(ctx), shape.vocab, bs,
                                        num_blocks=self.num_blocks, max_blocks_per_seq=mb,
                                        shared_table_rows=shared_table_rows)
        self.mb = mb
        self.kp = [synth.kv_pool(seed, f"k{l}", self.num_blocks, shape.n_kv_heads, bs,
                                 shape.head_dim, shape.dtype, kv_std) for l in range(shape.n_layers)]
        self.vp = [synth.kv_pool(seed, f"v{l}", self.num_blocks, shape.n_kv_heads, bs,
                                 shape.head_dim, shape.dtype, kv_std) for l in range(shape.n_layers)]
        self.dev = _lib.DecodeStep(shape, self.w, max_batch or len(ctx), mb, use_graphs=use_graphs)
        self.dev.kv_alloc(self.num_blocks, bs)
        self.upload_pools()

    def upload_pools(self):
        from transformer_decode_step_ns_gb300 import _lib
        for l in range(self.shape.n_layers):
            k, v = self.dev.kv_layer_ptrs(l)
            _lib.memcpy(k, self.kp[l].ctypes.data, self.kp[l].nbytes)
            _lib.memcpy(v, self.vp[l].ctypes.data, self.vp[l].nbytes)

    def download_pools(self):
        from transformer_decode_step_ns_gb300 import _lib
        ks, vs = [], []
        for l in range(self.shape.n_layers):
            k, v = self.dev.kv_layer_ptrs(l)
            kk = np.empty_like(self.kp[l])
            vv = np.empty_like(self.vp[l])
            _lib.memcpy(kk.ctypes.data, k, kk.nbytes)
            _lib.memcpy(vv.ctypes.data, v, vv.nbytes)
            ks.append(kk)
            vs.append(vv)
        return ks, vs

    def run_gpu(self, rows=None, with_logits=True):
        import torch
        b = self.batch
        sl = slice(None) if rows is None else rows
        B = len(b.token_ids[sl])
        logits = None
        if with_logits:
            logits = torch.full((B, self.shape.vocab), float("nan"), dtype=torch.float32,
                                device="cuda")
        self.dev.step(b.token_ids[sl], b.positions[sl], b.block_tables[sl], b.seq_lens[sl],
                      b.slot_mapping[sl], logits)
        torch.cuda.synchronize()
        assert self.dev.device_error() == 0
        return logits.cpu().numpy().astype(np.float64) if with_logits else None

    def run_oracle(self):
        b = self.batch
        model = oracle.OracleModel.from_weights(self.shape, self.w)
        kp = [a.copy() for a in self.kp]
        vp = [a.copy() for a in self.vp]
        logits = oracle.decode_step(model, kp, vp, b.token_ids, b.positions, b.block_tables,
                                    b.seq_lens, b.slot_mapping, self.bs)
        return logits, kp, vp


def _check_step(h: Harness):
    got = h.run_gpu()
    ref, kp_ref, vp_ref = h.run_oracle()
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) < 1e-2
    assert np.abs(got - ref).max() < 5e-2
    ks, vs = h.download_pools()
    dt = h.shape.dtype
    for l in range(h.shape.n_layers):
        for s in h.batch.slot_mapping:
            blk, off = int(s) // h.bs, int(s) % h.bs
            assert rel_l2(storage_f64(ks[l][blk, :, off], dt), storage_f64(kp_ref[l][blk, :, off], dt)) < 1e-2
            assert rel_l2(storage_f64(vs[l][blk, :, off], dt), storage_f64(vp_ref[l][blk, :, off], dt)) < 1e-2
    return got, ref


@pytest.mark.parametrize("dtype,tie", [("bf16", True), ("f16", False)])
def test_tiny_step_matches_oracle(cuda_lib, dtype, tie):
    h = Harness(_tiny(dtype, tie), 31, [0, 5, 16, 300])
    _check_step(h)


def test_qwen_shape_two_layers_batch1(cuda_lib):
    """Two-layer Qwen2.5-0.5B-shaped decoder, batch 1: 128 cached tokens whose blocks are a
    random permutation of physical blocks 0-7; this step's token takes block 8."""
    shape = synth.qwen05b_shape(n_layers=2)
    seed = synth.config_seed(0)
    w = synth.model_weights(shape, seed)
    h = Harness.__new__(Harness)
    from transformer_decode_step_ns_gb300 import _lib
    h.shape, h.bs, h.w = shape, 16, w
    perm = synth.permutation(seed, "cfg0.blocks", 8)
    tab = np.zeros((1, 9), dtype=np.int32)
    tab[0, :8] = perm
    tab[0, 8] = 8
    tok = synth.uniform_int(seed, "cfg0.token", 1, 0, shape.vocab - 1).astype(np.int32)
    h.batch = synth.DecodeBatch(token_ids=tok, positions=np.array([128], dtype=np.int32),
                                seq_lens=np.array([129], dtype=np.int32), block_tables=tab,
                                slot_mapping=np.array([8 * 16], dtype=np.int64), num_blocks=9,
                                block_size=16)
    h.num_blocks, h.mb = 9, 9
    h.kp = [synth.kv_pool(seed, f"k{l}", 9, 2, 16, 64, "f16") for l in range(2)]
    h.vp = [synth.kv_pool(seed, f"v{l}", 9, 2, 16, 64, "f16") for l in range(2)]
    h.dev = _lib.DecodeStep(shape, w, 1, 9, use_graphs=True)
    h.dev.kv_alloc(9, 16)
    h.upload_pools()
    got, ref = _check_step(h)
    assert int(np.argmax(got[0])) == int(np.argmax(ref[0])) or \
        abs(ref[0].max() - ref[0][int(np.argmax(got[0]))]) < 5e-2


@pytest.mark.parametrize("n_q,n_kv", [(8, 2), (8, 1)])
def test_head_dim_128_over_several_token_tiles(cuda_lib, n_q, n_kv):
    """head_dim 128 with 4 and 8 q heads per kv head (the LLaMA shapes), and 300 rows so every
    projection runs two token tiles (a ragged 160-row tile pair)."""
    shape = synth.ModelShape(hidden=512, n_layers=2, n_q_heads=n_q, n_kv_heads=n_kv, head_dim=128,
                             ffn=768, vocab=640, rms_eps=1e-5, rope_theta=5e5, dtype="bf16",
                             tie_embeddings=False)
    ctx = list(synth.uniform_int(81, "ctx300", 300, 0, 70))
    _check_step(Harness(shape, 81 + n_kv, ctx))


def test_nano_batches_across_both_gemm_kernels_equal_the_whole_batch_bitwise(cuda_lib):
    """2048 rows of a model whose unsplit projections (gate/up and the head: 152 feature tiles
    each) run the persistent kernel above 64 rows and the cluster kernel below, while the split
    ones (QKV, O, down) always run on clusters.  Unsplit, 40 + 2008 and 1024 + 1024 nano-batches
    give every row the same logits and cache bits through every fused epilogue (QKV with RoPE and
    the cache write, residual + norm, SwiGLU with the norm scale, the fp32 head), also with the
    persistent projections of the nano-batches capped at 40 or 7 CTAs and the attention at 50;
    sampled rows match the oracle."""
    shape = synth.ModelShape(hidden=512, n_layers=2, n_q_heads=32, n_kv_heads=4, head_dim=128,
                             ffn=9728, vocab=19456, rms_eps=1e-5, rope_theta=5e5, dtype="bf16",
                             tie_embeddings=False)
    ctx = list(synth.uniform_int(85, "ctx2048", 2048, 0, 70))
    h = Harness(shape, 86, ctx)
    got = h.run_gpu()
    ks0, vs0 = h.download_pools()
    for sizes, attn_cap, gemm_cap in (([40, 2008], 0, 0), ([1024, 1024], 0, 0), ([1024, 1024], 50, 40),
                                      ([40, 2008], 0, 7)):
        h.upload_pools()
        h.dev.set_nanobatch(sizes, attn_cta_budget=attn_cap, gemm_cta_budget=gemm_cap)
        np.testing.assert_array_equal(h.run_gpu(), got)
        ks, vs = h.download_pools()
        for l in range(shape.n_layers):
            np.testing.assert_array_equal(ks[l], ks0[l])
            np.testing.assert_array_equal(vs[l], vs0[l])
    # rows are independent: the oracle on a sample of them, over the same initial cache
    b = h.batch
    rows = np.array([0, 1, 39, 40, 1023, 1024, 2047])
    model = oracle.OracleModel.from_weights(shape, h.w)
    kp = [a.copy() for a in h.kp]
    vp = [a.copy() for a in h.vp]
    ref = oracle.decode_step(model, kp, vp, b.token_ids[rows], b.positions[rows], b.block_tables[rows],
                             b.seq_lens[rows], b.slot_mapping[rows], h.bs)
    assert rel_l2(got[rows], ref) < 1e-2 and np.abs(got[rows] - ref).max() < 5e-2


def test_wide_hidden_residual_epilogues_in_both_gemm_kernels(cuda_lib):
    """A hidden size of 19456 (152 feature tiles) leaves the O and down projections unsplit, so
    at 608 rows their residual + norm epilogue runs in the persistent kernel (three token tiles
    of 152 feature tiles: two per SM): unsplit and as 40 + 568 nano-batches (the 40 on
    clusters) give the same bits, and match the oracle."""
    shape = synth.ModelShape(hidden=19456, n_layers=1, n_q_heads=2, n_kv_heads=1, head_dim=128,
                             ffn=64, vocab=256, rms_eps=1e-5, rope_theta=5e5, dtype="bf16",
                             tie_embeddings=False)
    ctx = list(synth.uniform_int(87, "ctx608", 608, 0, 40))
    h = Harness(shape, 88, ctx)
    got = h.run_gpu()
    ref, kp_ref, vp_ref = h.run_oracle()
    # per-tensor relative L2 only: the 5e-2 max-abs bound is stated for logits of std ~0.6, and
    # this hidden size gives a head whose logits have std ~2.8
    assert rel_l2(got, ref) < 1e-2
    ks0, vs0 = h.download_pools()
    blk, off = h.batch.slot_mapping // h.bs, h.batch.slot_mapping % h.bs
    assert rel_l2(storage_f64(ks0[0][blk, :, off], "bf16"), storage_f64(kp_ref[0][blk, :, off], "bf16")) < 1e-2
    assert rel_l2(storage_f64(vs0[0][blk, :, off], "bf16"), storage_f64(vp_ref[0][blk, :, off], "bf16")) < 1e-2
    h.upload_pools()
    h.dev.set_nanobatch([40, 568])
    np.testing.assert_array_equal(h.run_gpu(), got)
    ks, vs = h.download_pools()
    np.testing.assert_array_equal(ks[0], ks0[0])
    np.testing.assert_array_equal(vs[0], vs0[0])


def test_graph_replay_equals_eager_bitwise(cuda_lib):
    shape = _tiny("bf16")
    a = Harness(shape, 41, [3, 40, 200], use_graphs=True)
    b = Harness(shape, 41, [3, 40, 200], use_graphs=False)
    ga = a.run_gpu()
    gb = b.run_gpu()
    np.testing.assert_array_equal(ga, gb)
    # a second replay of the captured graph on fresh caches gives the same answer
    a.upload_pools()
    np.testing.assert_array_equal(a.run_gpu(), ga)
    assert a.dev.info().graphs_cached == 1


def test_nano_batches_equal_the_whole_batch_bitwise(cuda_lib):
    shape = _tiny("bf16")
    ctx = [3, 40, 200, 17, 1, 600]
    whole = Harness(shape, 51, ctx)
    g_whole = whole.run_gpu()
    split = Harness(shape, 51, ctx)
    split.dev.set_nanobatch([2, 4])
    g_split = split.run_gpu()
    np.testing.assert_array_equal(g_split, g_whole)
    split3 = Harness(shape, 51, ctx, use_graphs=False)
    split3.dev.set_nanobatch([1, 3, 2], attn_cta_budget=3)
    np.testing.assert_array_equal(split3.run_gpu(), g_whole)


def test_prefill_chunk_rows_spanning_nano_batches(cuda_lib):
    """A prefill chunk as pseudo-requests (positions 0..C-1 over one shared block table) next
    to decode rows: matches the oracle, and every nano-batch split -- the chunk cut across
    nano-batches on both streams -- gives the unsplit result bitwise."""
    shape = _tiny("bf16")
    dec = [5, 70, 33]
    C = 40
    ctx = dec + list(range(C))
    last = len(ctx) - 1
    shared = list(range(len(dec))) + [last] * C
    h = Harness(shape, 71, ctx, shared_table_rows=shared)
    got, _ = _check_step(h)
    ks0, vs0 = h.download_pools()
    for sizes in ([16, 27], [10, 16, 17], [11, 11, 11, 10]):
        h.upload_pools()
        h.dev.set_nanobatch(sizes)
        np.testing.assert_array_equal(h.run_gpu(), got)
    # without an LM head the step writes the same KV cache bitwise
    h.upload_pools()
    h.dev.set_nanobatch([16, 27])
    h.run_gpu(with_logits=False)
    ks, vs = h.download_pools()
    for l in range(shape.n_layers):
        np.testing.assert_array_equal(ks[l], ks0[l])
        np.testing.assert_array_equal(vs[l], vs0[l])


def test_device_token_source_equals_host_tokens_bitwise(cuda_lib):
    """Three greedy steps with the tokens read back to the host and passed in, against the
    same steps reading the previous argmax from device memory: the same logits bitwise."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    shape = _tiny("bf16")
    ctx = [3, 40, 200]  # positions ctx .. ctx + 2 stay inside the rows' allocated blocks
    ha = Harness(shape, 91, ctx)
    hb = Harness(shape, 91, ctx)
    bt = ha.batch
    B = len(ctx)
    ids_dev = to_dev(bt.token_ids.copy())
    hb.dev.set_token_source(ids_dev)
    la = torch.empty((B, shape.vocab), dtype=torch.float32, device="cuda")
    lb = torch.empty_like(la)
    out_a = torch.empty(B, dtype=torch.int32, device="cuda")
    tok_a = bt.token_ids.copy()
    for s in range(3):
        pos = (bt.positions + s).astype(np.int32)
        slots = bt.block_tables[np.arange(B), pos // 16].astype(np.int64) * 16 + pos % 16
        ha.dev.step(tok_a, pos, bt.block_tables, pos + 1, slots, la)
        _lib.greedy_argmax(la, out_a)
        tok_a = from_dev(out_a)
        hb.dev.step(None, pos, bt.block_tables, pos + 1, slots, lb)
        _lib.greedy_argmax(lb, ids_dev)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(from_dev(la), from_dev(lb))
        np.testing.assert_array_equal(tok_a, from_dev(ids_dev))
    assert ha.dev.device_error() == 0 and hb.dev.device_error() == 0


def test_device_token_outside_the_vocabulary_is_recorded_and_replaced(cuda_lib):
    """A device token id outside [0, V) records NS_DEV_BAD_TOKEN (5) and the row embeds token 0:
    the logits equal those of the same step with token 0 given on the host, bitwise."""
    import torch
    shape = _tiny("bf16")
    ctx = [3, 40, 200]
    ha = Harness(shape, 93, ctx)
    hb = Harness(shape, 93, ctx)
    bt = ha.batch
    ids = bt.token_ids.copy()
    ids[1] = shape.vocab + 7
    ids_dev = to_dev(ids)
    ha.dev.set_token_source(ids_dev)
    la = torch.empty((3, shape.vocab), dtype=torch.float32, device="cuda")
    lb = torch.empty_like(la)
    ha.dev.step(None, bt.positions, bt.block_tables, bt.seq_lens, bt.slot_mapping, la)
    torch.cuda.synchronize()
    assert ha.dev.device_error() == 5
    host_ids = bt.token_ids.copy()
    host_ids[1] = 0
    hb.dev.step(host_ids, bt.positions, bt.block_tables, bt.seq_lens, bt.slot_mapping, lb)
    torch.cuda.synchronize()
    assert hb.dev.device_error() == 0
    np.testing.assert_array_equal(from_dev(la), from_dev(lb))


def test_graph_buckets_pad_batches_and_match_exact_graphs(cuda_lib):
    """With buckets {4, 8} a batch of 3 or 6 replays the graph of 4 or 8 with padding rows: the
    real rows' logits equal those of exact-size graphs bitwise, the padding rows write no
    logits (the rows after the caller's buffer keep their sentinel) and only the real rows'
    slots of the caller's pool change."""
    import torch
    shape = _tiny("bf16")
    ctx = [3, 40, 200, 17, 1, 600, 33, 9]
    exact = Harness(shape, 101, ctx)
    bucket = Harness(shape, 101, ctx)
    bucket.dev.set_graph_buckets([4, 8])
    bt = bucket.batch
    for n in (3, 6, 8, 4):
        exact.upload_pools()
        bucket.upload_pools()
        ref = exact.run_gpu(rows=slice(0, n))
        big = torch.full((8 + 2, shape.vocab), float("nan"), dtype=torch.float32, device="cuda")
        bucket.dev.step(bt.token_ids[:n], bt.positions[:n], bt.block_tables[:n], bt.seq_lens[:n],
                        bt.slot_mapping[:n], big[:n])
        torch.cuda.synchronize()
        assert bucket.dev.device_error() == 0
        got = big.cpu().numpy()
        np.testing.assert_array_equal(got[:n].astype(np.float64), ref)
        assert np.isnan(got[n:]).all()
        ks, vs = bucket.download_pools()
        for l in range(shape.n_layers):
            changed = np.nonzero((ks[l] != bucket.kp[l]).any(axis=(1, 2, 3)))[0]
            assert set(changed.tolist()) <= {int(s) // 16 for s in bt.slot_mapping[:n]}
    assert bucket.dev.info().graphs_cached == 2


@pytest.mark.parametrize("chunk,p0", [(15, 0), (16, 0), (33, 20)])
def test_prefill_chunk_threshold_and_offset(cuda_lib, chunk, p0):
    """A trailing run of 15 rows stays on the decode kernel, 16 or more go to the prefill-chunk
    kernel (a chunk that continues a prompt at position p0 > 0 reads its cached prefix too);
    both match the oracle."""
    shape = _tiny("bf16")
    dec = [7, 90]
    ctx = dec + list(range(p0, p0 + chunk))
    last = len(ctx) - 1
    shared = list(range(len(dec))) + [last] * chunk
    _check_step(Harness(shape, 111 + chunk, ctx, shared_table_rows=shared))


def test_attention_unit_queue_in_the_step_gives_the_same_bits(cuda_lib):
    """With the attention capped at 8 CTAs, 24 decode rows of 1100 to 2000 tokens hold at least
    six attention units per CTA, so the step launches the unit-queue variant (its graph reports
    attn_queue = 1); the logits and the cache equal bitwise those of the same step on the full
    grid, which takes the fixed deal, and match the oracle.  Graphs captured at start-up for that
    budget include both variants, and later steps replay them."""
    shape = _tiny("bf16")
    ctx = [int(v) for v in synth.uniform_int(91, "ctxq", 24, 1100, 2000)]
    full = Harness(shape, 301, ctx)
    got, _ = _check_step(full)
    assert [r["attn_queue"] for r in full.dev.graph_report()] == [0]
    ks0, vs0 = full.download_pools()
    capped = Harness(shape, 301, ctx)
    capped.dev.set_nanobatch(None, attn_cta_budget=8)
    capped.dev.capture_graphs([24])
    rep = capped.dev.graph_report()
    assert sorted(r["attn_queue"] for r in rep) == [0, 1] and all(r["batch"] == 24 for r in rep)
    np.testing.assert_array_equal(capped.run_gpu(), got)
    ks, vs = capped.download_pools()
    for l in range(shape.n_layers):
        np.testing.assert_array_equal(ks[l], ks0[l])
        np.testing.assert_array_equal(vs[l], vs0[l])
    assert capped.dev.info().graphs_cached == 2
    eager = Harness(shape, 301, ctx, use_graphs=False)
    eager.dev.set_nanobatch(None, attn_cta_budget=8)
    np.testing.assert_array_equal(eager.run_gpu(), got)
    assert eager.dev.device_error() == 0


def test_startup_capture_and_capture_report(cuda_lib):
    """Graphs captured at start-up for the buckets are the ones later steps replay (no new
    capture); the report lists each with its kernel count and capture time."""
    from transformer_decode_step_ns_gb300 import _lib
    shape = _tiny("bf16")
    ctx = [3, 40, 200, 17, 1, 600, 33, 9]
    h = Harness(shape, 161, ctx)
    h.dev.set_graph_buckets([4, 8])
    h.dev.capture_graphs([4, 8])
    rep = h.dev.graph_report()
    assert sorted(r["batch"] for r in rep) == [4, 8]
    for r in rep:
        assert r["kernels"] == 2 + 5 * shape.n_layers and r["capture_ms"] > 0
        assert r["with_lm"] == 1 and r["chunk_rows"] == 0 and r["n_split"] == 1
    h.run_gpu(rows=slice(0, 3))
    h.upload_pools()
    h.run_gpu()
    assert len(h.dev.graph_report()) == 2 and h.dev.info().graphs_cached == 2
    for bad in ([0], [9]):
        with pytest.raises(_lib.NSError):
            h.dev.capture_graphs(bad)
    eager = Harness(shape, 161, ctx, use_graphs=False)
    with pytest.raises(_lib.NSError):
        eager.dev.capture_graphs([4])


@pytest.mark.parametrize("tail", [25, 10])
def test_two_prompt_chunks_in_one_step(cuda_lib, tail):
    """Decode rows, then the rest of one prompt (positions 10..39), then the start of another
    (positions 0..tail-1), as a batch former lays them out: with a 25-row tail both prompts run
    as causal chunk kernels, with a 10-row tail (below the chunk threshold) the search stops and
    every row uses the decode kernel.  Both match the oracle, and a nano-batch split cutting
    through the first prompt gives the unsplit logits bitwise."""
    shape = _tiny("bf16")
    dec = [7, 90]
    first = list(range(10, 40))
    second = list(range(tail))
    ctx = dec + first + second
    ia, ib = len(dec) + len(first) - 1, len(ctx) - 1
    shared = list(range(len(dec))) + [ia] * len(first) + [ib] * len(second)
    h = Harness(shape, 171 + tail, ctx, shared_table_rows=shared)
    got, _ = _check_step(h)
    h.upload_pools()
    h.dev.set_nanobatch([20, len(ctx) - 20])
    np.testing.assert_array_equal(h.run_gpu(), got)


def test_graph_bucket_arguments_are_validated(cuda_lib):
    from transformer_decode_step_ns_gb300 import _lib
    h = Harness(_tiny("bf16"), 121, [3, 5])
    for bad in ([4, 2], [0, 2], [2, 3]):
        with pytest.raises(_lib.NSError) as e:
            h.dev.set_graph_buckets(bad)
        assert e.value.status == 1
    h.dev.set_graph_buckets([1, 2])
    h.dev.set_graph_buckets(None)


def test_step_at_the_largest_batch(cuda_lib):
    """4096 rows (the largest batch a handle takes: 16 token tiles of 256 in every projection),
    contexts 0..63 cycling; sampled rows match the oracle, which computes them alone."""
    shape = _tiny("bf16")
    ctx = [i % 64 for i in range(4096)]
    h = Harness(shape, 181, ctx, max_batch=4096)
    got = h.run_gpu()
    assert np.isfinite(got).all()
    rows = [0, 63, 1000, 2047, 4095]
    b = h.batch
    model = oracle.OracleModel.from_weights(h.shape, h.w)
    kp = [k.copy() for k in h.kp]
    vp = [v.copy() for v in h.vp]
    ref = oracle.decode_step(model, kp, vp, b.token_ids[rows], b.positions[rows], b.block_tables[rows],
                             b.seq_lens[rows], b.slot_mapping[rows], h.bs)
    assert rel_l2(got[rows], ref) < 1e-2
    assert np.abs(got[rows] - ref).max() < 5e-2


def test_rows_alone_equal_rows_in_batch_bitwise(cuda_lib):
    shape = _tiny("f16")
    ctx = [9, 33, 129]
    h = Harness(shape, 61, ctx, max_batch=3)
    full = h.run_gpu()
    for b in range(3):
        h.upload_pools()
        one = h.run_gpu(rows=slice(b, b + 1))
        np.testing.assert_array_equal(one[0], full[b])


def test_only_this_steps_slots_change(cuda_lib):
    shape = _tiny("bf16")
    h = Harness(shape, 71, [5, 31, 32, 100])
    before_k = [a.copy() for a in h.kp]
    h.run_gpu()
    ks, vs = h.download_pools()
    written = {(int(s) // 16, int(s) % 16) for s in h.batch.slot_mapping}
    for l in range(shape.n_layers):
        diff = np.argwhere((ks[l] != before_k[l]).any(axis=(1, 3)))
        assert {(int(b), int(o)) for b, o in diff} <= written
        diffv = np.argwhere((vs[l] != h.vp[l]).any(axis=(1, 3)))
        assert {(int(b), int(o)) for b, o in diffv} <= written


def test_decode_step_rejects_bad_metadata_before_launch(cuda_lib):
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    h = Harness(_tiny("bf16"), 81, [4, 20])
    b = h.batch
    logits = torch.zeros((2, 512), device="cuda")
    bad = b.slot_mapping.copy()
    bad[1] += 1
    with pytest.raises(_lib.NSError) as e:
        h.dev.step(b.token_ids, b.positions, b.block_tables, b.seq_lens, bad, logits)
    assert e.value.status == 1
    h.dev.set_nanobatch([1, 2])
    with pytest.raises(_lib.NSError):
        h.dev.step(b.token_ids, b.positions, b.block_tables, b.seq_lens, b.slot_mapping, logits)


def _trace_layer(h: Harness, layer: int):
    """The GPU's q, attention output, residual after the attention block and after the layer
    for ``layer`` (ns_set_trace), as fp64 host arrays, plus the step's logits."""
    import torch
    sh, B = h.shape, h.batch.batch
    qd = sh.n_q_heads * sh.head_dim
    R = h.dev.max_batch
    q = torch.zeros((R, qd), dtype=torch.int16, device="cuda")
    o = torch.zeros((R, qd), dtype=torch.int16, device="cuda")
    rm = torch.zeros((R, sh.hidden), dtype=torch.float32, device="cuda")
    ro = torch.zeros((R, sh.hidden), dtype=torch.float32, device="cuda")
    h.dev.set_trace(layer, q=q, attn=o, resid_mid=rm, resid_out=ro)
    logits = h.run_gpu()
    h.dev.set_trace(-1)
    dt = sh.dtype

    def bits(t):  # 16-bit storage patterns in the oracle's format (float16 values or bf16 bits)
        a = from_dev(t)[:B]
        return a.view(np.float16) if dt == "f16" else a
    return {"q": storage_f64(bits(q), dt).reshape(B, sh.n_q_heads, sh.head_dim),
            "attn": storage_f64(bits(o), dt).reshape(B, sh.n_q_heads, sh.head_dim),
            "resid_attn": rm[:B].cpu().numpy().astype(np.float64),
            "resid": ro[:B].cpu().numpy().astype(np.float64)}, logits


def _check_layers(h: Harness, split=None):
    """Every layer's tensors against the oracle's trace, each within relative L2 1e-2 (the
    stated per-tensor tolerance): q after RoPE, the k and v written to the cache, the attention
    output, the residual after the attention block and after the layer; then the logits."""
    b = h.batch
    model = oracle.OracleModel.from_weights(h.shape, h.w)
    kp = [a.copy() for a in h.kp]
    vp = [a.copy() for a in h.vp]
    tr = {}
    ref = oracle.decode_step(model, kp, vp, b.token_ids, b.positions, b.block_tables, b.seq_lens,
                             b.slot_mapping, h.bs, trace=tr)
    h.dev.set_nanobatch(split)
    dt = h.shape.dtype
    blk = b.slot_mapping // h.bs
    off = b.slot_mapping % h.bs
    errs = {}
    for l in range(h.shape.n_layers):
        got, logits = _trace_layer(h, l)
        for name in ("q", "attn", "resid_attn", "resid"):
            e = rel_l2(got[name], tr[name][l])
            errs[(l, name)] = e
            assert e < 1e-2, (l, name, e)
        ks, vs = h.download_pools()
        for name, pool, want in (("k", ks[l], tr["k"][l]), ("v", vs[l], tr["v"][l])):
            e = rel_l2(storage_f64(pool[blk, :, off, :], dt), want)
            errs[(l, name)] = e
            assert e < 1e-2, (l, name, e)
        assert rel_l2(logits, ref) < 1e-2 and np.abs(logits - ref).max() < 5e-2
    return errs


@pytest.mark.parametrize("dtype,tie", [("bf16", True), ("f16", False)])
def test_every_layer_tensor_matches_the_oracle(cuda_lib, dtype, tie):
    """Per-tensor parity inside the step, layer by layer (an error in one layer that a later
    layer damps would pass a logits-only check): a 4-layer model over ragged contexts that span
    block and superchunk boundaries."""
    shape = _tiny(dtype, tie, n_layers=4)
    h = Harness(shape, 61, [0, 5, 16, 300, 1100, 64])
    _check_layers(h)


def test_traced_tensors_of_nano_batches_equal_the_whole_batch_bitwise(cuda_lib):
    """The trace copies each nano-batch's rows on its own stream: the traced tensors of a split
    step equal the unsplit ones bit for bit, and both match the oracle per tensor."""
    shape = _tiny("bf16", n_layers=2)
    h = Harness(shape, 62, [3, 40, 200, 17, 1, 600])
    _check_layers(h, split=[2, 4])
    for l in range(2):
        h.dev.set_nanobatch(None)
        whole, lw = _trace_layer(h, l)
        h.dev.set_nanobatch([2, 4])
        part, lp = _trace_layer(h, l)
        np.testing.assert_array_equal(lw, lp)
        for k in whole:
            np.testing.assert_array_equal(whole[k], part[k])
    with pytest.raises(Exception):
        h.dev.set_trace(2, q=None)  # past the last layer
