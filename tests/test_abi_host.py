"""C-ABI checks that need no GPU: the library loads, exports every symbol include/ns.h declares,
its host block pool reproduces the allocator model bit for bit, and host validation rejects
bad step metadata before anything is launched."""
import os
import re

import numpy as np
import pytest

import synth
from oracle.kvcache import AllocatorError, BlockAllocator
from transformer_decode_step_ns_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(_lib.LIB_PATH):
        from transformer_decode_step_ns_gb300 import _build
        _build.build()
    return _lib.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ns.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ns_[a-z_0-9]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 20
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(_lib.SYMBOLS)


def test_status_strings(L):
    assert L.ns_status_str(0) == b"NS_OK"
    assert L.ns_status_str(7) == b"NS_ERR_OUT_OF_BLOCKS"


def test_block_pool_matches_the_allocator_model_bit_for_bit(L):
    rng = np.random.default_rng(11)
    nb, bs, mb, B = 40, 16, 12, 6
    pool = _lib.BlockPool(nb, bs, mb)
    model = BlockAllocator(nb, bs)
    t_lib = np.zeros((B, mb), dtype=np.int32)
    t_mod = np.zeros((B, mb), dtype=np.int32)
    ctx = np.zeros(B, dtype=np.int64)
    for step in range(300):
        # a request leaves now and then; its slot restarts at position 0
        if rng.random() < 0.1:
            b = int(rng.integers(B))
            n = (int(ctx[b]) + bs - 1) // bs
            ids = t_lib[b, :n].copy()
            np.testing.assert_array_equal(ids, t_mod[b, :n])
            pool.release(ids)
            model.release(ids.tolist())
            if len(ids):  # returning them again is refused by both, with nothing changed
                with pytest.raises(_lib.NSError):
                    pool.release(ids[:1])
                with pytest.raises(AllocatorError):
                    model.release(ids[:1].tolist())
            ctx[b] = 0
            t_lib[b] = 0
            t_mod[b] = 0
        pos = ctx.astype(np.int32)
        try:
            s_mod = model.prepare_step(t_mod, pos)
            err_mod = None
        except AllocatorError as e:
            err_mod = e
        if err_mod is None:
            s_lib = pool.prepare_step(pos, t_lib)
            np.testing.assert_array_equal(s_lib, s_mod)
            np.testing.assert_array_equal(t_lib, t_mod)
            ctx += 1
            ctx[ctx >= mb * bs] = 0  # wrap long requests (release-free restart in the test)
        else:
            with pytest.raises(_lib.NSError):
                pool.prepare_step(pos, t_lib)
            np.testing.assert_array_equal(t_lib, t_mod)
        assert pool.free_count() == model.free_count()


def test_block_pool_errors(L):
    pool = _lib.BlockPool(2, 16, 4)
    tab = np.zeros((3, 4), dtype=np.int32)
    with pytest.raises(_lib.NSError) as e:
        pool.prepare_step(np.array([0, 0, 0]), tab)
    assert e.value.status == 7 and pool.free_count() == 2 and not tab.any()
    with pytest.raises(_lib.NSError) as e:
        pool.prepare_step(np.array([64]), np.zeros((1, 4), dtype=np.int32))
    assert e.value.status == 1
    with pytest.raises(_lib.NSError):
        pool.release([5])
    assert pool.reserve(2).tolist() == [0, 1]
    with pytest.raises(_lib.NSError):
        pool.reserve(1)
    # a block has one owner: returning a free block, or one block twice in a call, is refused
    # and leaves the free list as it was (the allocator model's rule)
    pool.release([1])
    for bad in ([1], [0, 0], [0, 1]):
        with pytest.raises(_lib.NSError) as e:
            pool.release(bad)
        assert e.value.status == 1 and pool.free_count() == 1
    pool.release([0])
    assert pool.free_count() == 2 and pool.reserve(2).tolist() == [1, 0]


def _meta(B=3, bs=16, mb=4, nb=20, vocab=50):
    db = synth.decode_batch(7, "m", [3, 17, 40], vocab, bs, num_blocks=nb, max_blocks_per_seq=mb)
    return db, dict(num_blocks=nb, block_size=bs, max_blocks_per_seq=mb, vocab=vocab, max_batch=8)


def _chk(kw, db, **over):
    a = dict(token_ids=db.token_ids.copy(), positions=db.positions.copy(),
             block_tables=db.block_tables.copy(), seq_lens=db.seq_lens.copy(),
             slot_mapping=db.slot_mapping.copy())
    a.update(over)
    return _lib.check_step_metadata(kw["num_blocks"], kw["block_size"], kw["max_blocks_per_seq"],
                                    kw["vocab"], kw["max_batch"], **a)


def test_step_metadata_validation(L):
    db, kw = _meta()
    assert _chk(kw, db) == 0
    bad_tok = db.token_ids.copy(); bad_tok[1] = 50
    assert _chk(kw, db, token_ids=bad_tok) == 1
    bad_len = db.seq_lens.copy(); bad_len[0] += 1
    assert _chk(kw, db, seq_lens=bad_len) == 1
    bad_tab = db.block_tables.copy(); bad_tab[2, 1] = 20
    assert _chk(kw, db, block_tables=bad_tab) == 1
    bad_tab = db.block_tables.copy(); bad_tab[2, 3] = -5   # beyond seq_len: ignored
    assert _chk(kw, db, block_tables=bad_tab) == 0
    bad_slot = db.slot_mapping.copy(); bad_slot[0] += 1
    assert _chk(kw, db, slot_mapping=bad_slot) == 1
    kw2 = dict(kw); kw2["max_batch"] = 2
    assert _chk(kw2, db) == 1
    # an empty step is refused (nothing to launch), as is a negative position
    empty = dict(token_ids=db.token_ids[:0], positions=db.positions[:0],
                 block_tables=db.block_tables[:0], seq_lens=db.seq_lens[:0],
                 slot_mapping=db.slot_mapping[:0])
    assert _chk(kw, db, **empty) == 1
    kw3 = dict(kw); kw3["max_blocks_per_seq"] = 4
    long_pos = db.positions.copy(); long_pos[2] = 64
    long_len = db.seq_lens.copy(); long_len[2] = 65
    assert _chk(kw3, db, positions=long_pos, seq_lens=long_len) == 1
    # the largest int32 position (seq_len wrapped to the smallest int32) is rejected before
    # p + 1 is formed or a table entry past the row is read
    huge_pos = db.positions.copy(); huge_pos[1] = 2 ** 31 - 1
    huge_len = db.seq_lens.copy(); huge_len[1] = -2 ** 31
    assert _chk(kw, db, positions=huge_pos, seq_lens=huge_len) == 1
    neg_pos = db.positions.copy(); neg_pos[0] = -1
    zero_len = db.seq_lens.copy(); zero_len[0] = 0
    assert _chk(kw, db, positions=neg_pos, seq_lens=zero_len) == 1
    # the last slot of a full table is accepted
    full_tab = db.block_tables.copy(); full_tab[2] = [3, 5, 7, 9]
    last_pos = db.positions.copy(); last_pos[2] = 63
    last_len = db.seq_lens.copy(); last_len[2] = 64
    last_slot = db.slot_mapping.copy(); last_slot[2] = 9 * 16 + 15
    assert _chk(kw, db, positions=last_pos, seq_lens=last_len, block_tables=full_tab,
                slot_mapping=last_slot) == 0


def test_binding_refuses_host_memory_where_kernels_read_device_memory(L):
    """A host buffer (numpy array or CPU tensor) passed where a kernel reads device memory, or
    a device buffer of the wrong type, is refused by the binding with INVALID_ARG before
    anything reaches the library."""
    import torch
    logits = torch.zeros((2, 5))
    ids = torch.zeros(2, dtype=torch.int32)
    for call in (lambda: _lib.greedy_argmax(logits, ids),
                 lambda: _lib.linear(np.zeros((128, 64), np.uint16), np.zeros((1, 64), np.uint16),
                                     torch.zeros((1, 128)), 1, 128, 64, "bf16"),
                 lambda: _lib.attn_decode(torch.zeros(8), torch.zeros(8), torch.zeros(8),
                                          np.zeros((1, 1), np.int32), np.ones(1, np.int32),
                                          torch.zeros(8), 2, 1, 64, 16, 1, 1, 0.125, "bf16")):
        with pytest.raises(_lib.NSError) as e:
            call()
        assert e.value.status == 1 and "device memory" in str(e.value)
    # raw device addresses pass through untouched (the caller vouches for them); None stays None
    assert _lib._dev(0x7F0000000000, "x") == 0x7F0000000000 and _lib._dev(None, "x") is None


class _FakeCuda:
    """Stands in for a CUDA tensor on a machine without a GPU.  The binding reads only these
    attributes before it calls the library; every call below has one bad argument and must be
    refused before the library is reached, so the address is never dereferenced."""
    is_cuda = True

    def __init__(self, n, dtype):
        import torch
        self.n, self.dtype = n, dtype
        self._size = torch.empty(0, dtype=dtype).element_size()

    def numel(self):
        return self.n

    def element_size(self):
        return self._size

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return 0x7F0000001000


def test_binding_refuses_short_or_mistyped_attention_buffers(L):
    """Each device buffer of the attention calls (ns_attn_decode, ns_attn_decode_noalloc) is
    checked against what the kernel reads or writes: q and out [batch][Hq][d], the pools
    [num_blocks][Hkv][bs][d] of 16-bit elements, block_tables int32 [batch][mb], seq_lens int32
    [batch], dev_err int32 [1].  A short or mistyped one is refused with INVALID_ARG."""
    import torch
    B, hq, hkv, d, bs, mb, nb = 3, 8, 2, 64, 16, 5, 20
    good = dict(q=(B * hq * d, torch.bfloat16), k_pool=(nb * hkv * bs * d, torch.bfloat16),
                v_pool=(nb * hkv * bs * d, torch.int16), block_tables=(B * mb, torch.int32),
                seq_lens=(B, torch.int32), out=(B * hq * d, torch.float16))
    bad = {"q": [(B * hq * d - 1, torch.bfloat16), (B * hq * d, torch.float32)],
           "k_pool": [(nb * hkv * bs * d - 1, torch.bfloat16), (nb * hkv * bs * d, torch.int32)],
           "v_pool": [(nb * hkv * bs * d - 8, torch.bfloat16), (nb * hkv * bs * d, torch.uint8)],
           "block_tables": [(B * mb - 1, torch.int32), (B * mb, torch.int64)],
           "seq_lens": [(B, torch.int64)],
           "out": [(B * hq * d - 1, torch.bfloat16), (B * hq * d, torch.float32)]}

    def args(**over):
        a = {k: _FakeCuda(*v) for k, v in good.items()}
        a.update({k: _FakeCuda(*v) for k, v in over.items()})
        if isinstance(a["seq_lens"], _FakeCuda):
            a["seq_lens"].shape = (B,)
        return a

    refused = 0
    for name, variants in bad.items():
        for v in variants:
            for noalloc in (False, True):
                a = args(**{name: v})
                fn = _lib.attn_decode_noalloc if noalloc else _lib.attn_decode
                with pytest.raises(_lib.NSError) as e:
                    fn(a["q"], a["k_pool"], a["v_pool"], a["block_tables"], a["seq_lens"],
                       a["out"], hq, hkv, d, bs, mb, nb, 0.125, "bf16")
                assert e.value.status == 1 and name in str(e.value), (name, v, str(e.value))
                refused += 1
    for err in ((0, torch.int32), (1, torch.int64)):
        a = args()
        with pytest.raises(_lib.NSError) as e:
            _lib.attn_decode_noalloc(a["q"], a["k_pool"], a["v_pool"], a["block_tables"],
                                     a["seq_lens"], a["out"], hq, hkv, d, bs, mb, nb, 0.125,
                                     "bf16", dev_err=_FakeCuda(*err))
        assert e.value.status == 1 and "dev_err" in str(e.value)
        refused += 1
    assert refused == 2 * 11 + 2


def test_binding_refuses_short_or_mistyped_linear_buffers(L):
    """ns_linear reads w [n][k] and x [m][k] (16-bit) and writes y [m][n] fp32."""
    import torch
    m, n, k = 4, 128, 64
    good = dict(w=(n * k, torch.bfloat16), x=(m * k, torch.bfloat16), y=(m * n, torch.float32))
    for name, v in (("w", (n * k - 1, torch.bfloat16)), ("w", (n * k, torch.float32)),
                    ("x", (m * k - 1, torch.bfloat16)), ("y", (m * n - 1, torch.float32)),
                    ("y", (m * n, torch.bfloat16))):
        a = {kk: _FakeCuda(*vv) for kk, vv in good.items()}
        a[name] = _FakeCuda(*v)
        with pytest.raises(_lib.NSError) as e:
            _lib.linear(a["w"], a["x"], a["y"], m, n, k, "bf16")
        assert e.value.status == 1 and name in str(e.value)


def test_binding_refuses_metadata_of_unequal_row_counts(L):
    db, kw = _meta()
    assert _chk(kw, db, seq_lens=db.seq_lens[:2]) == 1
    assert _chk(kw, db, slot_mapping=db.slot_mapping[:1]) == 1
    assert _chk(kw, db, block_tables=db.block_tables[:, :3]) == 1
    with pytest.raises(_lib.NSError) as e:
        _lib._same_rows(3, token_ids=np.zeros(3), seq_lens=np.zeros(2))
    assert e.value.status == 1 and "seq_lens" in str(e.value)


def _chunk_rule(pos, tabs, sl, bs, min_rows=16):
    """The documented rule, stated plainly: working back from the last row, grow a run while the
    previous row sits one position earlier and reads the same leading blocks as the run's last
    row; a run of at least min_rows rows is a chunk, a shorter one ends the search."""
    starts, end = [], len(pos)
    while end > 0:
        f = end - 1
        while f > 0:
            need = -(-int(sl[f - 1]) // bs)
            if pos[f - 1] != pos[f] - 1 or list(tabs[f - 1][:need]) != list(tabs[end - 1][:need]):
                break
            f -= 1
        if end - f < min_rows:
            break
        starts.insert(0, f)
        end = f
    return starts


def test_prompt_chunk_detection_by_hand_and_against_the_rule(L):
    bs, mb = 16, 8
    A = np.arange(0, 8, dtype=np.int32)
    Bt = np.arange(8, 16, dtype=np.int32)
    D = np.arange(16, 24, dtype=np.int32)

    def find(rows):
        pos = [p for p, _ in rows]
        return _lib.find_prompt_chunks(bs, pos, np.stack([t for _, t in rows]), [p + 1 for p in pos])

    dec = [(5, D), (9, D), (40, D)]
    assert find(dec) == []                                             # decode rows only
    assert find(dec + [(p, A) for p in range(16)]) == [3]              # exactly 16 rows: a chunk
    assert find(dec + [(p, A) for p in range(15)]) == []               # 15 rows: not one
    assert find(dec + [(p, A) for p in range(20)] + [(p, Bt) for p in range(30, 46)]) == [3, 23]
    # the first shorter run ends the search: the 20-row run before the 5-row one is not found
    assert find([(p, A) for p in range(20)] + [(p, D) for p in range(5)]
                + [(p, Bt) for p in range(16)]) == [25]
    # a position gap splits a run; so does a different block under the earlier row's tokens
    assert find([(p, A) for p in range(16)] + [(p, A) for p in range(17, 33)]) == [0, 16]
    other = A.copy()
    other[0] = 99
    assert find([(p, other) for p in range(16)] + [(p, A) for p in range(16, 32)]) == [0, 16]
    # entries past a row's own blocks do not matter: only the blocks its tokens occupy compare
    tail = A.copy()
    tail[7] = 77
    assert find([(p, tail) for p in range(16)] + [(p, A) for p in range(16, 24)]) == [0]
    # random layouts against the stated rule
    rng = np.random.default_rng(5)
    for _ in range(200):
        rows = []
        for _ in range(int(rng.integers(1, 6))):
            t = rng.permutation(64)[:mb].astype(np.int32)
            n = int(rng.integers(1, 40))
            p0 = int(rng.integers(0, mb * bs - n))
            rows += [(p0 + k, t) for k in range(n)]
        pos = [p for p, _ in rows]
        tabs = np.stack([t for _, t in rows])
        sl = [p + 1 for p in pos]
        assert _lib.find_prompt_chunks(bs, pos, tabs, sl) == _chunk_rule(pos, tabs, sl, bs)
    # bad lengths are refused before any table is read
    with pytest.raises(_lib.NSError):
        _lib.find_prompt_chunks(bs, [0], A[None], [0])
    with pytest.raises(_lib.NSError):
        _lib.find_prompt_chunks(bs, [127], A[None], [129])
    assert _lib.find_prompt_chunks(bs, [], np.zeros((0, mb), np.int32), []) == []


def test_block_pool_equals_the_model_on_arbitrary_call_sequences(L):
    """Property test: any sequence of reserve / release (valid, repeated, foreign or out of
    range ids) / prepare_step calls gives the library pool and the allocator model the same
    outcome (result or refusal) and the same free list after every call."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    nb, bs, mb = 12, 4, 6
    op = st.one_of(
        st.tuples(st.just("reserve"), st.integers(0, 5)),
        st.tuples(st.just("release"), st.lists(st.integers(-1, nb), max_size=4)),
        st.tuples(st.just("release_held"), st.integers(0, 30)),
        st.tuples(st.just("prepare"), st.lists(st.integers(0, mb * bs), min_size=1, max_size=3)),
    )

    @hyp.settings(max_examples=150, deadline=None, derandomize=True, database=None)
    @hyp.given(st.lists(op, max_size=40))
    def run(ops):
        pool, model = _lib.BlockPool(nb, bs, mb), BlockAllocator(nb, bs)
        held = []
        for kind, arg in ops:
            if kind == "release_held":
                arg = [held[arg % len(held)]] if held else []
                kind = "release"
            if kind == "reserve":
                calls = (lambda: pool.reserve(arg).tolist(), lambda: model.alloc(arg))
            elif kind == "release":
                calls = (lambda: pool.release(np.array(arg, np.int32)), lambda: model.release(arg))
            else:
                t_lib = np.zeros((len(arg), mb), np.int32)
                t_mod = np.zeros((len(arg), mb), np.int32)
                pos = np.array(arg, np.int32)
                calls = (lambda: pool.prepare_step(pos, t_lib).tolist(),
                         lambda: model.prepare_step(t_mod, pos).tolist())
            outcome = []
            for fn, errs in zip(calls, (_lib.NSError, AllocatorError)):
                try:
                    outcome.append(("ok", fn()))
                except errs:
                    outcome.append(("refused", None))
            assert outcome[0] == outcome[1], (kind, arg)
            if outcome[0][0] == "ok":
                if kind == "reserve":
                    held += outcome[0][1]
                elif kind == "release":
                    for i in arg:
                        held.remove(i)
                else:  # rows starting a block took one
                    held += [int(t_mod[r, p // bs]) for r, p in enumerate(arg) if p % bs == 0]
            assert pool.free_count() == model.free_count() == nb - len(held)
        rest = pool.reserve(pool.free_count()).tolist()
        assert rest == list(model.free)

    run()


def test_step_metadata_validation_equals_the_stated_rules(L):
    """Property test: on arbitrary (mostly invalid) metadata the library's host validation
    accepts exactly what the documented rules accept: 1 <= batch <= max_batch, token ids in
    [0, V), positions >= 0, seq_len = position + 1 <= max_blocks_per_seq * block_size, the
    table entries under a row's tokens inside the pool, slot = table[p / bs] * bs + p % bs."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    nb, bs, mb, vocab, max_batch = 6, 4, 3, 20, 4

    def rules(tok, pos, tab, sl, slot):
        if not 1 <= len(pos) <= max_batch:
            return 1
        for b in range(len(pos)):
            p, n = int(pos[b]), int(sl[b])
            if not 0 <= tok[b] < vocab or p < 0 or n != p + 1 or n > mb * bs:
                return 1
            if any(not 0 <= tab[b][j] < nb for j in range(-(-n // bs))):
                return 1
            if slot[b] != int(tab[b][p // bs]) * bs + p % bs:
                return 1
        return 0

    off = st.sampled_from([0, 0, 0, -1, 1])
    row = st.tuples(st.integers(-2, vocab + 1), st.integers(-2, mb * bs + 1), off,
                    st.lists(st.integers(-1, nb), min_size=mb, max_size=mb), off)
    seen = {0: 0, 1: 0}

    @hyp.settings(max_examples=400, deadline=None, derandomize=True, database=None)
    @hyp.given(st.lists(row, min_size=0, max_size=max_batch + 1))
    def run(rows):
        tok = np.array([r[0] for r in rows], np.int32)
        pos = np.array([r[1] for r in rows], np.int32)
        sl = np.array([r[1] + 1 + r[2] for r in rows], np.int32)       # right or off by one
        tab = np.array([r[3] for r in rows], np.int32).reshape(len(rows), mb)
        slot = np.array([int(r[3][min(max(r[1], 0) // bs, mb - 1)]) * bs + max(r[1], 0) % bs + r[4]
                         for r in rows], np.int64)                    # right or off by one
        got = _lib.check_step_metadata(nb, bs, mb, vocab, max_batch, tok, pos, tab, sl, slot)
        assert got == rules(tok, pos, tab, sl, slot)
        seen[got] += 1

    run()
    assert seen[0] >= 20 and seen[1] >= 20, seen  # both outcomes well exercised


def test_handle_setters_refuse_a_null_handle_without_touching_the_device(L):
    """ns_set_step_kernel, ns_set_nanobatch and ns_set_gemm_cta_budget return INVALID_ARG for a
    NULL handle (checked before any CUDA call)."""
    assert L.ns_set_step_kernel(None, 1) == 1
    assert L.ns_set_step_kernel(None, 0) == 1
    assert L.ns_set_gemm_cta_budget(None, 4) == 1
    assert L.ns_set_nanobatch(None, 1, None, 0) == 1
