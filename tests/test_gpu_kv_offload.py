"""KV offload and reload (NanoFlow page, "Runtime details that keep the pipeline fed"): the
rows a step mirrors to the host are the cache's own bits at the step's slots; saving a request,
reloading it into other blocks and decoding from there gives the same logits bitwise; every
copy is pure indexing, so every comparison here is exact."""
import math

import numpy as np
import pytest

import oracle
from test_gpu_step import Harness, _tiny

pytestmark = pytest.mark.gpu


def _pinned_rows(shape, n_rows):
    import torch
    return torch.zeros((shape.n_layers, n_rows, 2 * shape.n_kv_heads * shape.head_dim),
                       dtype=torch.int16).pin_memory()


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint16)


@pytest.mark.parametrize("graphs,split", [(False, None), (True, None), (True, [3, 5])])
def test_offload_mirror_is_the_cache_rows(cuda_lib, graphs, split):
    """After a step the host mirror holds, for every layer and row, the K and V the step wrote
    at the row's slot; mirroring changes no logit."""
    import torch
    shape = _tiny("bf16")
    ctx = [5, 17, 31, 40, 64, 3, 90, 15]
    h = Harness(shape, 131, ctx, use_graphs=graphs)
    mirror = _pinned_rows(shape, len(ctx))
    h.dev.set_kv_offload(mirror)
    if split:
        h.dev.set_nanobatch(split)
    on = h.run_gpu()
    ks, vs = h.download_pools()
    want = oracle.kv_rows(ks, vs, h.batch.slot_mapping)
    np.testing.assert_array_equal(_bits(mirror.numpy()), _bits(want))
    # the same step again without the mirror: identical logits and cache
    h.upload_pools()
    h.dev.set_kv_offload(None)
    off = h.run_gpu()
    np.testing.assert_array_equal(on, off)
    ks2, vs2 = h.download_pools()
    for l in range(shape.n_layers):
        np.testing.assert_array_equal(ks2[l], ks[l])
        np.testing.assert_array_equal(vs2[l], vs[l])
    torch.cuda.synchronize()


def test_offload_mirrors_prefill_chunk_rows_and_padding_is_harmless(cuda_lib):
    """A prefill chunk's rows are mirrored like decode rows; with graph buckets the real rows of
    a padded batch are still exact."""
    shape = _tiny("f16")
    dec = [9, 70]
    C = 20
    ctx = dec + list(range(C))
    last = len(ctx) - 1
    h = Harness(shape, 137, ctx, shared_table_rows=list(range(len(dec))) + [last] * C,
                max_batch=32)
    h.dev.set_graph_buckets([32])
    mirror = _pinned_rows(shape, 32)
    h.dev.set_kv_offload(mirror)
    h.run_gpu()
    ks, vs = h.download_pools()
    want = oracle.kv_rows(ks, vs, h.batch.slot_mapping)
    np.testing.assert_array_equal(_bits(mirror.numpy()[:, :len(ctx)]), _bits(want))


def test_save_reload_moves_a_request_to_other_blocks(cuda_lib):
    """Save one request's K/V (gather from its pages), check them against the cache, reload
    them in two pieces into fresh blocks, and decode its next token from the old and from the
    new blocks: the same logits bitwise."""
    import torch
    shape = _tiny("bf16")
    ctx = [40, 77, 130]
    bs = 16
    h = Harness(shape, 139, ctx, extra_blocks=24)
    h.run_gpu()
    r = 2
    n = int(h.batch.seq_lens[r])  # cached tokens of the request after the step
    nblk = math.ceil(n / bs)
    old = h.batch.block_tables[r, :nblk].copy()
    saved = np.zeros((shape.n_layers, n, 2 * shape.n_kv_heads * shape.head_dim), dtype=np.uint16)
    h.dev.kv_save(saved, n, 0, old)
    torch.cuda.synchronize()
    ks, vs = h.download_pools()
    np.testing.assert_array_equal(saved, _bits(oracle.kv_rows(ks, vs, oracle.request_slots(old, 0, n, bs))))
    # reload into fresh blocks: positions [0, 20) then [20, n), from pinned memory
    bt = h.batch
    used = {int(bt.block_tables[b, j]) for b in range(len(ctx))
            for j in range(math.ceil(int(bt.seq_lens[b]) / bs))}
    free = np.array(sorted(set(range(h.num_blocks)) - used), dtype=np.int32)
    assert free.size >= nblk
    new = free[np.random.default_rng(3).permutation(free.size)[:nblk]]
    src = torch.from_numpy(saved.view(np.int16))
    head = src[:, :20].contiguous().pin_memory()  # kept alive until the copies have run
    tail = src[:, 20:].contiguous().pin_memory()
    h.dev.kv_reload(head, 20, 0, new)
    h.dev.kv_reload(tail, n - 20, 20, new)
    torch.cuda.synchronize()
    assert h.dev.device_error() == 0
    ks2, vs2 = h.download_pools()
    np.testing.assert_array_equal(_bits(oracle.kv_rows(ks2, vs2, oracle.request_slots(new, 0, n, bs))), saved)
    # blocks other than the new ones are untouched
    for l in range(shape.n_layers):
        keep = np.setdiff1d(np.arange(h.num_blocks), new)
        np.testing.assert_array_equal(ks2[l][keep], ks[l][keep])
        np.testing.assert_array_equal(vs2[l][keep], vs[l][keep])
    # next token of the request from the old table and from the new one
    assert n % bs != 0  # the next position stays in the last block
    logits = []
    for tab_row in (old, new):
        tab = np.zeros((1, h.mb), dtype=np.int32)
        tab[0, :nblk] = tab_row
        pos = np.array([n], dtype=np.int32)
        slot = np.array([int(tab_row[n // bs]) * bs + n % bs], dtype=np.int64)
        out = torch.empty((1, shape.vocab), dtype=torch.float32, device="cuda")
        h.dev.step(np.array([7], dtype=np.int32), pos, tab, pos + 1, slot, out)
        torch.cuda.synchronize()
        logits.append(out.cpu().numpy())
    assert h.dev.device_error() == 0
    np.testing.assert_array_equal(logits[0], logits[1])


def test_offload_and_reload_arguments_are_validated(cuda_lib):
    from transformer_decode_step_ns_gb300 import _lib
    shape = _tiny("bf16")
    h = Harness(shape, 149, [3, 5])
    with pytest.raises(_lib.NSError):  # pageable host memory
        h.dev.set_kv_offload(np.zeros((shape.n_layers, 2, h.dev.kv_row_elems()), dtype=np.uint16))
    with pytest.raises(_lib.NSError):  # too small
        h.dev.set_kv_offload(_pinned_rows(shape, 1))
    rows = np.zeros((shape.n_layers, 4, h.dev.kv_row_elems()), dtype=np.uint16)
    for n_tok, first, table in ((4, 0, [h.num_blocks]),   # block id outside the pool
                                (4, 14, [0]),             # table shorter than the range
                                (0, 0, [0]),              # no tokens
                                (4, -1, [0])):            # negative position
        with pytest.raises(_lib.NSError) as e:
            h.dev.kv_reload(rows, n_tok, first, table)
        assert e.value.status == 1
    h.dev.kv_save(rows, 4, 0, [1])
    assert h.dev.device_error() == 0


def test_dense_batch_former_with_preemption_matches_the_oracle(cuda_lib):
    """Six prompts through the dense-batch former on a pool too small for their peaks
    (predicted decode length 1): prompts are chunked to fill each step, running requests are
    preempted (K/V saved to the host) and resumed (reloaded into other blocks).  Every
    generated token's logits equal, within the logits tolerance, the oracle run over that
    request alone (its prompt and generated tokens at positions 0 .. n-1)."""
    import torch
    import synth
    from transformer_decode_step_ns_gb300 import _lib
    from helpers import rel_l2
    shape = _tiny("bf16")
    bs, D, mb = 16, 24, 8
    w = synth.model_weights(shape, 151, gamma_std=0.1)
    dev = _lib.DecodeStep(shape, w, D, mb, use_graphs=False)
    dev.kv_alloc(12, bs)
    former = _lib.BatchFormer(dev.pool(), D, mb, eos_token=-1, predicted_new_tokens=1)
    rng = np.random.default_rng(151)
    prompts = {rid: rng.integers(0, shape.vocab, size=n).astype(np.int32)
               for rid, n in enumerate([40, 7, 23, 16, 31, 5])}
    for rid, p in prompts.items():
        former.add(rid, p, 12)
    store, got, saves, steps = {}, {rid: [] for rid in prompts}, 0, 0
    ids = torch.empty(D, dtype=torch.int32, device="cuda")
    while former.counts()[3] < len(prompts):
        steps += 1
        assert steps < 200
        rows = former.next()
        for kind, rid, n, table in former.moves():
            if kind == 0:
                store[rid] = np.zeros((shape.n_layers, n, dev.kv_row_elems()), dtype=np.uint16)
                dev.kv_save(store[rid], n, 0, table)
                saves += 1
            else:
                dev.kv_reload(store.pop(rid), n, 0, table)
        B = len(rows["token_ids"])
        assert B > 0
        logits = torch.empty((B, shape.vocab), dtype=torch.float32, device="cuda")
        dev.step(rows["token_ids"], rows["positions"], rows["block_tables"], rows["seq_lens"],
                 rows["slot_mapping"], logits)
        _lib.greedy_argmax(logits, ids[:B])
        torch.cuda.synchronize()
        assert dev.device_error() == 0
        lg = logits.cpu().numpy().astype(np.float64)
        for b in np.nonzero(rows["row_samples"])[0]:
            got[int(rows["row_request"][b])].append(lg[b])
        former.commit(ids[:B].cpu().numpy())
    assert saves > 0  # the pool forced preemption
    model = oracle.OracleModel.from_weights(shape, w)
    for rid, prompt in prompts.items():
        gen = former.tokens(rid)
        assert len(gen) == 12
        seq = np.concatenate([prompt, np.array(gen[:-1], dtype=np.int32)])
        T = len(seq)
        nblk = math.ceil(T / bs)
        pool_shape = (nblk, shape.n_kv_heads, bs, shape.head_dim)
        kp = [np.zeros(pool_shape, dtype=np.uint16) for _ in range(shape.n_layers)]
        vp = [np.zeros(pool_shape, dtype=np.uint16) for _ in range(shape.n_layers)]
        tab = np.tile(np.arange(mb, dtype=np.int32), (T, 1))
        pos = np.arange(T, dtype=np.int32)
        ref = oracle.decode_step(model, kp, vp, seq, pos, tab, pos + 1, pos.astype(np.int64), bs)
        ref = ref[len(prompt) - 1:]
        mine = np.stack(got[rid])
        assert mine.shape == ref.shape
        for i in range(len(ref)):
            assert rel_l2(mine[i], ref[i]) < 1e-2, (rid, i, rel_l2(mine[i], ref[i]))
            assert np.abs(mine[i] - ref[i]).max() < 5e-2, (rid, i)
        # greedy: each generated token is the argmax of the logits that produced it
        np.testing.assert_array_equal(np.argmax(mine, axis=1), gen)


def test_async_formation_generates_the_sync_tokens(cuda_lib):
    """The batch former forming each step before the previous one is committed (decode rows
    read their tokens from the previous step's device argmax) generates, greedily, exactly the
    tokens of synchronous formation (the same steps, rows independent of one another)."""
    import collections
    import torch
    import synth
    from transformer_decode_step_ns_gb300 import _lib
    shape = _tiny("bf16")
    bs, D, mb = 16, 24, 8
    w = synth.model_weights(shape, 157, gamma_std=0.1)
    rng = np.random.default_rng(157)
    prompts = {rid: rng.integers(0, shape.vocab, size=n).astype(np.int32)
               for rid, n in enumerate([33, 5, 20, 17, 9, 26])}
    out = {}
    for async_mode in (False, True):
        dev = _lib.DecodeStep(shape, w, D, mb, use_graphs=False)
        dev.kv_alloc(64, bs)
        ids = torch.zeros(D, dtype=torch.int32, device="cuda")
        dev.set_token_source(ids)
        former = _lib.BatchFormer(dev.pool(), D, mb, eos_token=-1)
        former.set_async(async_mode)
        for rid, p in prompts.items():
            former.add(rid, p, 10)
        logits = torch.empty((D, shape.vocab), dtype=torch.float32, device="cuda")
        pending = collections.deque()
        negative = 0
        for _ in range(200):
            r = former.next()
            B = len(r["token_ids"])
            negative += int((r["token_ids"] < 0).sum())
            if B:
                dev.step(r["token_ids"], r["positions"], r["block_tables"], r["seq_lens"],
                         r["slot_mapping"], logits[:B])
                _lib.greedy_argmax(logits[:B], ids[:B])
            pending.append(ids[:B].cpu().numpy().copy())  # read before the next step's argmax
            if len(pending) == (2 if async_mode else 1):
                former.commit(pending.popleft())
            if former.counts()[3] == len(prompts):
                break
        while pending:
            former.commit(pending.popleft())
        assert dev.device_error() == 0
        assert (negative > 0) == async_mode
        out[async_mode] = {rid: former.tokens(rid) for rid in prompts}
        dev.close()
    assert all(len(t) == 10 for t in out[False].values())
    assert out[True] == out[False]
