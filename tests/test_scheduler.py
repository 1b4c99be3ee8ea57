"""The constant-dense-batch former (NanoFlow page, "Runtime details that keep the pipeline fed"):
the plain Python model is pinned by a worked example and by invariants over random runs; the
library's C++ former must reproduce the model bit for bit."""
import os

import numpy as np
import pytest

from oracle.kvcache import BlockAllocator
from oracle.scheduler import DenseBatchFormer, SchedulerError

KEYS = ("token_ids", "positions", "block_tables", "seq_lens", "slot_mapping", "row_request",
        "row_samples")


def _rows(st):
    return {k: getattr(st, k) for k in KEYS}


def test_worked_example_by_hand():
    """Dense target 8, block size 4: prompt A (5 tokens, 3 new) and B (6 tokens, 2 new)."""
    m = DenseBatchFormer(BlockAllocator(16, 4), dense_tokens=8, max_blocks_per_seq=4, eos_token=999)
    A, B = 7, 3
    m.add(A, [10, 11, 12, 13, 14], 3)
    m.add(B, [20, 21, 22, 23, 24, 25], 2)
    # step 1: A's whole prompt (blocks 0, 1), then 3 tokens of B (block 2)
    s = m.next()
    np.testing.assert_array_equal(s.token_ids, [10, 11, 12, 13, 14, 20, 21, 22])
    np.testing.assert_array_equal(s.positions, [0, 1, 2, 3, 4, 0, 1, 2])
    np.testing.assert_array_equal(s.slot_mapping, [0, 1, 2, 3, 4, 8, 9, 10])
    np.testing.assert_array_equal(s.row_request, [A] * 5 + [B] * 3)
    np.testing.assert_array_equal(s.row_samples, [0, 0, 0, 0, 1, 0, 0, 0])
    np.testing.assert_array_equal(s.block_tables[0], [0, 1, 0, 0])
    np.testing.assert_array_equal(s.block_tables[5], [2, 0, 0, 0])
    assert m.commit([0, 0, 0, 0, 30, 0, 0, 0]) == []
    # step 2: A decodes token 30 at position 5; B's last 3 prompt tokens (block 3 joins)
    s = m.next()
    np.testing.assert_array_equal(s.token_ids, [30, 23, 24, 25])
    np.testing.assert_array_equal(s.positions, [5, 3, 4, 5])
    np.testing.assert_array_equal(s.seq_lens, [6, 4, 5, 6])
    np.testing.assert_array_equal(s.slot_mapping, [5, 11, 12, 13])
    np.testing.assert_array_equal(s.row_samples, [1, 0, 0, 1])
    assert m.commit([31, 0, 0, 40]) == []
    # step 3: both decode; A reaches 3 new tokens, B 2: both finish, blocks return in order
    s = m.next()
    np.testing.assert_array_equal(s.token_ids, [31, 40])
    np.testing.assert_array_equal(s.positions, [6, 6])
    np.testing.assert_array_equal(s.slot_mapping, [6, 14])
    assert m.commit([32, 41]) == [A, B]
    assert m.tokens(A) == [30, 31, 32] and m.tokens(B) == [40, 41]
    assert list(m.pool.free) == list(range(4, 16)) + [0, 1, 2, 3]
    assert len(m.next().token_ids) == 0
    assert m.counts() == (0, 0, 0, 2)


def test_preemption_worked_example_by_hand():
    """Pool of 4 blocks of 4, predicted decode length 1 (optimistic): A (4 prompt tokens) and
    B (3) both decode 6 tokens.  B outgrows the pool at step 6, is saved and freed, and is
    reloaded into other blocks once A finishes."""
    m = DenseBatchFormer(BlockAllocator(4, 4), dense_tokens=4, max_blocks_per_seq=4,
                         eos_token=999, predicted_new=1)
    A, B = 1, 2
    m.add(A, [10, 11, 12, 13], 6)
    m.add(B, [20, 21, 22], 6)
    s = m.next()                                   # A's prompt fills the batch (block 0)
    np.testing.assert_array_equal(s.row_request, [A] * 4)
    m.commit([0, 0, 0, 50])
    s = m.next()                                   # A decodes at 4 (block 1); B admitted (block 2)
    np.testing.assert_array_equal(s.positions, [4, 0, 1, 2])
    np.testing.assert_array_equal(s.slot_mapping, [4, 8, 9, 10])
    m.commit([51, 0, 0, 60])
    for want_pos, want_slot in (([5, 3], [5, 11]), ([6, 4], [6, 12]), ([7, 5], [7, 13])):
        s = m.next()                               # B's position 4 takes block 3, the last
        np.testing.assert_array_equal(s.positions, want_pos)
        np.testing.assert_array_equal(s.slot_mapping, want_slot)
        assert m.moves == []
        m.commit([52, 61])
    s = m.next()                                   # A needs a block at 8: B (last) is preempted
    assert [(v.kind, v.rid, v.n_tokens, v.table) for v in m.moves] == [(0, B, 6, [2, 3])]
    np.testing.assert_array_equal(s.positions, [8])
    np.testing.assert_array_equal(s.slot_mapping, [8])   # block 2, freed by B, reused
    assert m.counts() == (0, 1, 1, 0)
    assert m.commit([53]) == [A]                   # A's sixth token: finished, blocks 0, 1, 2 back
    s = m.next()                                   # B resumes in blocks 3, 0 and decodes at 6
    assert [(v.kind, v.rid, v.n_tokens, v.table) for v in m.moves] == [(1, B, 6, [3, 0])]
    np.testing.assert_array_equal(s.positions, [6])
    np.testing.assert_array_equal(s.slot_mapping, [2])
    np.testing.assert_array_equal(s.token_ids, [61])
    m.commit([62])
    assert m.tokens(B) == [60, 61, 61, 61, 62] and m.counts() == (0, 1, 0, 1)


def _moves(m):
    return [(v.kind, v.rid, v.n_tokens, list(v.table)) for v in m.moves]


def test_preempted_requests_resume_first_in_first_out_by_hand():
    """Pool of 5 blocks of 4, predicted decode length 1.  Peaks: r0 (5 prompt tokens) 2 blocks,
    r1 (3), r2 (4), r3 (3) one each.  Step 0 places r0's prompt (blocks 0, 1) and r1's (block 2);
    step 1 decodes both and places r2's prompt (block 3) and two tokens of r3's (block 4).
    Step 2: r1 and r2 both cross into a new block with none free, so r2 (last running) is saved;
    step 4: r0 and r3 do the same, so r3 is saved too.  When r1 finishes, two blocks come back;
    resuming needs the cached tokens' blocks plus the block of the next position (2 each), so
    only one request fits: r2, saved first, resumes at step 5, and r3 only at step 7."""
    m = DenseBatchFormer(BlockAllocator(5, 4), dense_tokens=8, max_blocks_per_seq=8,
                         eos_token=999, predicted_new=1)
    for i, (pl, mn) in enumerate([(5, 8), (3, 5), (4, 3), (3, 4)]):
        m.add(i, list(range(100 * i, 100 * i + pl)), mn)
    want = {  # step: (rows' requests, positions, slots, moves)
        0: ([0, 0, 0, 0, 0, 1, 1, 1], [0, 1, 2, 3, 4, 0, 1, 2], [0, 1, 2, 3, 4, 8, 9, 10], []),
        1: ([0, 1, 2, 2, 2, 2, 3, 3], [5, 3, 0, 1, 2, 3, 0, 1], [5, 11, 12, 13, 14, 15, 16, 17], []),
        2: ([0, 1, 3], [6, 4, 2], [6, 12, 18], [(0, 2, 4, [3])]),
        3: ([0, 1, 3], [7, 5, 3], [7, 13, 19], []),
        4: ([0, 1], [8, 6], [16, 14], [(0, 3, 4, [4])]),
        5: ([0, 2], [9, 4], [17, 12], [(1, 2, 4, [2])]),
        6: ([0, 2], [10, 5], [18, 13], []),
        7: ([0, 3], [11, 4], [19, 12], [(1, 3, 4, [2])]),
        8: ([3], [5], [13], []),
    }
    for k in range(9):
        s = m.next()
        req, pos, slots, moves = want[k]
        np.testing.assert_array_equal(s.row_request, req, err_msg=f"step {k}")
        np.testing.assert_array_equal(s.positions, pos, err_msg=f"step {k}")
        np.testing.assert_array_equal(s.slot_mapping, slots, err_msg=f"step {k}")
        assert _moves(m) == moves, k
        if k == 4:
            assert list(m.swapped) == [2, 3]
        m.commit(np.full(len(s.token_ids), 50 + k, np.int32))
    assert m.counts() == (0, 0, 0, 4)
    assert m.tokens(2) == [51, 55, 56] and m.tokens(3) == [52, 53, 57, 58]


def test_no_resumption_in_a_step_that_preempts_by_hand():
    """Pool of 4 blocks of 4, predicted decode length 1.  r0 (4 prompt tokens, 6 new) runs
    alone until step 4, when r1 (4 prompt tokens) and r2 (1 token) arrive and take the last two
    blocks.  At step 5 r0 and r1 both need a new block and none is free: r2 (last running) is
    saved, which frees one block, still short, so r1 is saved too.  r2 would fit again at once,
    but a step that preempts resumes nothing; both come back at step 6, r2 first (saved
    first), once r0 has finished."""
    m = DenseBatchFormer(BlockAllocator(4, 4), dense_tokens=8, max_blocks_per_seq=8,
                         eos_token=999, predicted_new=1)
    m.add(0, [0, 1, 2, 3], 6)
    for k in range(4):
        m.commit(np.full(len(m.next().token_ids), 50 + k, np.int32))
    m.add(1, [100, 101, 102, 103], 3)
    m.add(2, [200], 3)
    s = m.next()
    np.testing.assert_array_equal(s.row_request, [0, 1, 1, 1, 1, 2])
    np.testing.assert_array_equal(s.slot_mapping, [7, 8, 9, 10, 11, 12])
    m.commit(np.full(6, 54, np.int32))
    s = m.next()
    assert _moves(m) == [(0, 2, 1, [3]), (0, 1, 4, [2])]
    np.testing.assert_array_equal(s.row_request, [0])
    np.testing.assert_array_equal(s.slot_mapping, [12])   # r0 takes block 3, r2's old block
    assert list(m.pool.free) == [2] and list(m.swapped) == [2, 1]
    assert m.commit([55]) == [0]
    s = m.next()
    assert _moves(m) == [(1, 2, 1, [2]), (1, 1, 4, [0])]
    np.testing.assert_array_equal(s.row_request, [2, 1])
    np.testing.assert_array_equal(s.positions, [1, 4])
    np.testing.assert_array_equal(s.slot_mapping, [9, 4])  # r1's position 4 takes block 1


def test_prompts_wait_while_a_preempted_request_cannot_resume_by_hand():
    """Pool of 6 blocks of 4, predicted decode length 1: A and S (8 prompt tokens each, 12 new)
    fill the pool; at step 5 A needs a block and S is saved (10 tokens, blocks 3, 4, 5).  P
    (2 prompt tokens, 1 new: a one-block peak) arrives at step 9, when one block is free after
    A's decode block: P alone would fit, but S needs 3 blocks to resume, so P waits; when A
    finishes, S resumes (blocks 5, 0, 1) and P starts in the same step."""
    m = DenseBatchFormer(BlockAllocator(6, 4), dense_tokens=8, max_blocks_per_seq=8,
                         eos_token=999, predicted_new=1)
    A, S, P = 1, 2, 3
    m.add(A, list(range(10, 18)), 12)
    m.add(S, list(range(20, 28)), 12)
    for k in range(13):
        if k == 9:
            m.add(P, [30, 31], 1)
        s = m.next()
        if k == 5:
            assert _moves(m) == [(0, S, 10, [3, 4, 5])]
        if 9 <= k <= 11:
            np.testing.assert_array_equal(s.row_request, [A])   # P waits, one block free
            assert m.counts() == (1, 1, 1, 0)
        if k == 12:
            assert _moves(m) == [(1, S, 10, [5, 0, 1])]
            np.testing.assert_array_equal(s.row_request, [S, P, P])
            np.testing.assert_array_equal(s.slot_mapping, [6, 8, 9])
        m.commit(np.full(len(s.token_ids), 5, np.int32))
    assert m.counts() == (0, 1, 0, 2)


def _random_run(form, rng, n_steps, vocab, eos, add_prob, max_prompt, max_new_hi):
    """Drive a former (model or library) with seeded arrivals and sampled tokens; yield each
    step's rows (or the error class) and finished ids."""
    next_id = 0
    for _ in range(n_steps):
        while rng.random() < add_prob:
            p = rng.integers(0, vocab, size=int(rng.integers(1, max_prompt + 1)))
            try:
                form.add(next_id, p, int(rng.integers(1, max_new_hi + 1)))
                yield ("add", next_id)
            except Exception as e:  # noqa: BLE001
                yield ("add_err", type(e).__name__)
            next_id += 1
        try:
            st = form.next()
        except Exception as e:  # noqa: BLE001
            yield ("next_err", type(e).__name__)
            continue
        rows = _rows(st) if not isinstance(st, dict) else st
        yield ("formed", rows, form.moves())
        n = len(rows["token_ids"])
        sampled = rng.integers(0, vocab, size=n).astype(np.int32)
        fin = form.commit(sampled)
        yield ("step", rows, list(fin))


class _ModelAdapter:
    """The model behind the library class's interface."""

    def __init__(self, m):
        self.m = m

    def add(self, rid, prompt, max_new):
        try:
            self.m.add(rid, prompt, max_new)
        except SchedulerError as e:
            raise RuntimeError(str(e))

    def next(self):
        try:
            return _rows(self.m.next())
        except SchedulerError as e:
            raise RuntimeError(str(e))

    def commit(self, sampled):
        return self.m.commit(sampled)

    def counts(self):
        return self.m.counts()

    def moves(self):
        return [(v.kind, v.rid, v.n_tokens, np.array(v.table, np.int32)) for v in self.m.moves]


CASES = [  # (dense, block size, pool blocks, blocks per seq, vocab, eos, add prob, max prompt,
    #      max new, predicted new)
    (8, 4, 64, 16, 50, 3, 0.5, 30, 6, 0),
    (16, 16, 12, 8, 20, 0, 0.6, 100, 20, 0),     # tight pool, peaks reserved
    (16, 16, 12, 8, 20, -1, 0.6, 100, 20, 2),    # tight pool, optimistic: preemption
    (33, 16, 400, 32, 1000, 7, 0.9, 200, 40, 0),
    (32, 4, 24, 32, 20, -1, 0.3, 60, 12, 3),     # preemption with chunked prompts
    (64, 4, 40, 32, 30, 5, 0.08, 60, 8, 0),      # short batches: prompts run out
    (1, 4, 8, 8, 10, 9, 0.3, 12, 4, 0),
]


@pytest.mark.parametrize("case", CASES)
def test_model_invariants_over_random_runs(case):
    D, bs, nb, mb, vocab, eos, ap, mp, mn, pn = case
    m = DenseBatchFormer(BlockAllocator(nb, bs), D, mb, eos, pn)
    rng = np.random.default_rng(11)
    placed = {}   # request -> prompt positions placed so far
    saved = {}    # preempted request -> cached tokens it was saved with
    for ev in _random_run(_ModelAdapter(m), rng, 300, vocab, eos, ap, mp, mn):
        if ev[0] == "formed":
            rows, moves = ev[1], ev[2]
            # saves come before reloads; a reload restores exactly what was saved, into as many
            # blocks as those tokens need; a request is saved at most once before it returns
            kinds = [v[0] for v in moves]
            assert kinds == sorted(kinds)
            assert not (0 in kinds and 1 in kinds)  # no resumption in a preempting step
            for kind, rid, n, table in moves:
                assert len(table) == -(-n // bs)
                if kind == 0:
                    assert rid not in saved
                    saved[rid] = n
                else:
                    assert saved.pop(rid) == n
            if pn == 0:
                assert moves == []  # peaks reserved: nothing is ever preempted
            continue
        if ev[0] != "step":
            continue
        rows, fin = ev[1], ev[2]
        n = len(rows["token_ids"])
        assert n <= D
        pos, tab, req, smp = rows["positions"], rows["block_tables"], rows["row_request"], rows["row_samples"]
        # slots follow the block table; no two rows share one
        want = tab[np.arange(n), pos // bs].astype(np.int64) * bs + pos % bs
        np.testing.assert_array_equal(rows["slot_mapping"], want)
        assert len(set(rows["slot_mapping"].tolist())) == n
        np.testing.assert_array_equal(rows["seq_lens"], pos + 1)
        # decode rows (requests past their prompt) come first
        is_dec = np.array([pos[b] >= len(m.req[int(req[b])].prompt) for b in range(n)], dtype=bool)
        assert not np.any(is_dec[1:] & ~is_dec[:-1])
        for b in range(n):
            r = m.req[int(req[b])]
            if not is_dec[b]:
                # prompt rows: consecutive positions, each placed once, in order, right token
                assert pos[b] == placed.get(r.rid, 0)
                placed[r.rid] = pos[b] + 1
                assert rows["token_ids"][b] == r.prompt[pos[b]]
                assert smp[b] == (1 if pos[b] == len(r.prompt) - 1 else 0)
            else:
                assert smp[b] == 1
        # finished requests: max_new reached or eos sampled, blocks returned
        for rid in fin:
            r = m.req[rid]
            assert r.finished and r.table == []
            assert len(r.gen) == r.max_new or r.gen[-1] == eos
    # blocks of live requests are disjoint and, with the free list, cover the pool exactly
    live = [b for r in m.req.values() for b in r.table]
    assert sorted(live + list(m.pool.free)) == list(range(nb))


@pytest.fixture(scope="module")
def L():
    from transformer_decode_step_ns_gb300 import _lib
    if not os.path.exists(_lib.LIB_PATH):
        pytest.skip("libns.so not built")
    return _lib


@pytest.mark.parametrize("case", CASES)
def test_library_former_matches_the_model_bit_for_bit(L, case):
    D, bs, nb, mb, vocab, eos, ap, mp, mn, pn = case
    model = _ModelAdapter(DenseBatchFormer(BlockAllocator(nb, bs), D, mb, eos, pn))
    pool = L.BlockPool(nb, bs, mb)
    lib_form = L.BatchFormer(pool, D, mb, eos, pn)
    a = _random_run(model, np.random.default_rng(5), 300, vocab, eos, ap, mp, mn)
    b = _random_run(lib_form, np.random.default_rng(5), 300, vocab, eos, ap, mp, mn)
    steps = 0
    for ea, eb in zip(a, b):
        assert ea[0] == eb[0], (ea, eb)
        if ea[0] == "formed":
            for k in KEYS:
                np.testing.assert_array_equal(ea[1][k], eb[1][k], err_msg=k)
            assert len(ea[2]) == len(eb[2])
            for va, vb in zip(ea[2], eb[2]):
                assert va[:3] == vb[:3]
                np.testing.assert_array_equal(va[3], vb[3])
        elif ea[0] == "step":
            steps += 1
            for k in KEYS:
                np.testing.assert_array_equal(ea[1][k], eb[1][k], err_msg=k)
            assert ea[2] == eb[2]
        elif ea[0] == "add":
            assert ea[1] == eb[1]
    assert steps > 0
    assert pool.free_count() == model.m.pool.free_count()
    ids = pool.reserve(pool.free_count())
    np.testing.assert_array_equal(ids, list(model.m.pool.free))


def test_library_former_errors(L):
    pool = L.BlockPool(2, 4, 4)
    f = L.BatchFormer(pool, 8, 4, 0)
    for args in ((0, [], 1), (0, [1], 0), (0, [1] * 16, 1), (-1, [1], 1), (0, [4, -1], 1)):
        with pytest.raises(L.NSError) as e:
            f.add(*args)
        assert e.value.status == 1
    f.add(0, [1, 2, 3, 4, 5, 6, 7], 1)   # 2 blocks: the whole pool
    f.add(1, [1, 2], 3)
    with pytest.raises(L.NSError):
        f.commit([0])                     # nothing formed yet
    s = f.next()
    assert len(s["token_ids"]) == 7       # B gets no row: the pool is empty
    with pytest.raises(L.NSError):
        f.next()                          # commit first
    with pytest.raises(L.NSError):
        f.commit([0] * 6)                 # wrong row count
    assert f.commit([5] * 7) == [0]       # max_new 1: finished, blocks back
    s = f.next()
    np.testing.assert_array_equal(s["token_ids"], [1, 2])
    f.commit([9, 9])
    assert f.counts() == (0, 1, 0, 1) and f.tokens(1) == [9]
    with pytest.raises(L.NSError):
        f.remove(1)                       # still running
    f.remove(0)                           # finished: forgotten
    assert f.counts() == (0, 1, 0, 0)
    with pytest.raises(L.NSError):
        f.tokens(0)
    assert L.BatchFormer(pool, 1, 4, 0).counts() == (0, 0, 0, 0)
    # with nothing to run, a step has no rows and commits nothing
    idle = L.BatchFormer(L.BlockPool(4, 4, 4), 8, 4, 0)
    s = idle.next()
    assert all(len(s[k]) == 0 for k in ("token_ids", "positions", "seq_lens", "slot_mapping"))
    assert idle.commit([]) == [] and idle.counts() == (0, 0, 0, 0)
    with pytest.raises(L.NSError):
        L.BatchFormer(pool, 4, 4, 0, -1)


def test_tuner_candidate_splits():
    from transformer_decode_step_ns_gb300 import tuner
    c = tuner.candidate_splits(2048)
    assert c[0] is None
    assert all(sum(s) == 2048 and all(v % 128 == 0 for v in s) for s in c[1:])
    two = [s for s in c[1:] if len(s) == 2]
    assert len(two) == 15 and [768, 1280] in two and [1024, 1024] in two
    assert sorted(s for s in c if s and len(s) == 3) == [[640, 640, 768], [640, 768, 640], [768, 640, 640]]
    assert [s for s in c if s and len(s) == 4] == [[512] * 4]
    # a batch that is not a multiple of 128: the last nano-batch takes the remainder
    c = tuner.candidate_splits(1000)
    assert all(sum(s) == 1000 for s in c[1:]) and [128, 872] in c
    # 7 units of 128 and 104 rows over: near-even thirds 3 + 2 + 2 units in every order, the
    # last part taking the 104
    assert sorted(s for s in c if s and len(s) == 3) == [[256, 256, 488], [256, 384, 360],
                                                          [384, 256, 360]]


def test_tuner_interference_row_arithmetic():
    from transformer_decode_step_ns_gb300 import tuner
    # attention best 100 us, capped solo 200, co-run 400; GEMM solo 50, co-run 80
    r = tuner.interference_row(64, 100e-6, 200e-6, 50e-6, 400e-6, 80e-6, 8)
    assert r["P_attn"] == 0.25 and r["P_attn_solo"] == 0.5
    assert r["P_gemm"] == r["R_gemm"] == 0.625 and r["R_attn"] == 0.375
    assert r["attn_us"] == 400.0 and r["gemm_us"] == 80.0 and r["n_gemm"] == 8


def test_tuner_search_measures_every_split_then_budgets_and_picks_the_fastest():
    """A synthetic step cost: two-way splits near 1280 + 768 are cheapest, and a CTA budget of
    96 helps only the best splits; the profile keeps budgets with co-run P_attn >= 0.5."""
    from transformer_decode_step_ns_gb300 import tuner
    calls = []

    def cost(sizes, budget):
        base = 4.0 if sizes is None else 3.7 + 0.001 * abs(sizes[0] - 1280) + 0.05 * (len(sizes) - 2)
        return base - (0.05 if budget == 96 else 0.0) + (0.01 if budget not in (0, 96) else 0.0)

    def step(sizes, budget):
        calls.append((None if sizes is None else tuple(sizes), budget))

    def timer(fn, reps):
        calls.clear()
        fn()
        (sizes, budget), = calls
        return cost(None if sizes is None else list(sizes), budget)

    profile = {"rows": [{"budget": b, "P_attn": 0.6 if b >= 96 else 0.3} for b in range(8, 129, 8)]}
    out = tuner.search(step, 2048, profile=profile, timer=timer)
    stage1 = [r for r in out["table"] if r["budget"] == 0]
    assert len(stage1) == len(tuner.candidate_splits(2048))
    assert out["budgets_kept"] == [96, 104, 112, 120, 128]
    assert len(out["table"]) == len(stage1) + 3 * 5
    assert out["best"]["sizes"] == [1280, 768] and out["best"]["budget"] == 96
    # without a profile every budget is tried on the three fastest splits
    out = tuner.search(step, 2048, timer=timer)
    assert len(out["table"]) == len(stage1) + 3 * 16
    # a budget exactly at min_p is kept; below it is not
    edge = {"rows": [{"budget": 8, "P_attn": 0.5}, {"budget": 16, "P_attn": 0.49},
                     {"budget": 24, "P_attn": 0.7}]}
    assert tuner.search(step, 2048, profile=edge, timer=timer)["budgets_kept"] == [8, 24]
    # fewer than two budgets clear min_p: the four with the highest co-run P_attn are tried
    low = {"rows": [{"budget": b, "P_attn": p} for b, p in
                    ((8, 0.1), (16, 0.45), (24, 0.2), (32, 0.3), (40, 0.05), (48, 0.4))]}
    assert tuner.search(step, 2048, profile=low, timer=timer)["budgets_kept"] == [16, 48, 32, 24]


def test_tuner_search_tries_gemm_budget_pairs_on_the_fastest_splits():
    """(GEMM budget, attention budget) pairs are timed on the three fastest multi-batch splits,
    after the attention budgets; a pair that helps wins, and every row records both budgets."""
    from transformer_decode_step_ns_gb300 import tuner
    calls = []

    def cost(sizes, budget, gemm_budget):
        base = 4.0 if sizes is None else 3.7 + 0.001 * abs(sizes[0] - 1024)
        return base - (0.2 if (gemm_budget, budget) == (100, 104) else 0.0)

    def step(sizes, budget, gemm_budget=0):
        calls.append((None if sizes is None else tuple(sizes), budget, gemm_budget))

    def timer(fn, reps):
        calls.clear()
        fn()
        (sizes, budget, gb), = calls
        return cost(None if sizes is None else list(sizes), budget, gb)

    pairs = [(76, 152), (100, 104), (128, 48)]
    out = tuner.search(step, 2048, budgets=(64,), timer=timer, gemm_pairs=pairs)
    n1 = len(tuner.candidate_splits(2048))
    assert len(out["table"]) == n1 + 3 * 1 + 3 * len(pairs)
    tail = out["table"][-3 * len(pairs):]
    assert [(r["gemm_budget"], r["budget"]) for r in tail[:3]] == pairs
    assert all(r["gemm_budget"] == 0 for r in out["table"][:n1 + 3])
    assert out["best"]["sizes"] == [1024, 1024]
    assert (out["best"]["gemm_budget"], out["best"]["budget"]) == (100, 104)


def test_async_formation_worked_example_by_hand():
    """Asynchronous formation: step 1 is formed before step 0 is committed, so its decode rows
    read their tokens from step 0's rows (-(row + 1)); B samples eos at step 0, which is seen
    only when step 0 commits, after B's row in step 1 exists: that row's token is dropped and
    B's blocks return at step 1's commit."""
    m = DenseBatchFormer(BlockAllocator(16, 4), dense_tokens=8, max_blocks_per_seq=4, eos_token=9)
    m.set_async(True)
    A, B = 1, 2
    m.add(A, [10, 11, 12], 3)
    m.add(B, [20, 21, 22, 23, 24], 2)
    s0 = m.next()
    np.testing.assert_array_equal(s0.token_ids, [10, 11, 12, 20, 21, 22, 23, 24])
    np.testing.assert_array_equal(s0.row_samples, [0, 0, 1, 0, 0, 0, 0, 1])
    s1 = m.next()                                   # formed before step 0 commits
    np.testing.assert_array_equal(s1.token_ids, [-3, -8])
    np.testing.assert_array_equal(s1.positions, [3, 5])
    with pytest.raises(SchedulerError):
        m.next()                                    # at most one formed step outstanding
    assert m.commit([0, 0, 50, 0, 0, 0, 0, 9]) == [B]   # B's eos, seen one step late
    s2 = m.next()
    np.testing.assert_array_equal(s2.token_ids, [-1])   # A only; its position 4 takes block 3
    np.testing.assert_array_equal(s2.slot_mapping, [12])
    assert m.commit([51, 77]) == []                 # B's extra token is dropped, blocks 1, 2 back
    assert m.tokens(B) == [9]
    assert m.commit([52]) == [A]
    assert m.tokens(A) == [50, 51, 52]
    assert list(m.pool.free) == list(range(4, 16)) + [1, 2, 0, 3]
    with pytest.raises(SchedulerError):
        DenseBatchFormer(BlockAllocator(4, 4), 4, 4, 0, predicted_new=3).set_async(True)


def _pipelined(form, rng, n_req, vocab, eos, max_prompt, max_new_hi, sampler, async_mode):
    """All requests arrive first; steps are formed and committed (one step late when
    asynchronous) until every request finishes.  Yields formed rows and commit results."""
    from collections import deque
    for i in range(n_req):
        form.add(i, rng.integers(0, vocab, size=int(rng.integers(1, max_prompt + 1))),
                 int(rng.integers(1, max_new_hi + 1)))
    pending = deque()
    for _ in range(5000):
        rows = form.next()
        yield ("formed", rows)
        pending.append(rows)
        if len(pending) == (2 if async_mode else 1):
            r = pending.popleft()
            yield ("commit", form.commit(sampler(r)))
        if form.counts()[3] == n_req:
            break
    while pending:
        r = pending.popleft()
        yield ("commit", form.commit(sampler(r)))


def _sampler_for(vocab):
    """The token a row samples depends only on its request and position."""
    def sample(rows):
        return np.array([(int(q) * 7919 + int(p) * 104729) % vocab
                         for q, p in zip(rows["row_request"], rows["positions"])], dtype=np.int32)
    return sample


ASYNC_CASES = [(16, 4, 200, 32, 30, 3, 20, 8), (33, 16, 400, 32, 100, 7, 60, 20)]


def _formed_blocks(rows, bs):
    """(request, block) of every block the rows of one formed step read or write."""
    out = set()
    for b in range(len(rows["token_ids"])):
        n = -(-int(rows["seq_lens"][b]) // bs)
        for blk in rows["block_tables"][b, :n]:
            out.add((int(rows["row_request"][b]), int(blk)))
    return out


@pytest.mark.parametrize("case", ASYNC_CASES)
def test_async_formation_generates_what_sync_formation_does(case):
    """With a sampler that depends only on (request, position), asynchronous and synchronous
    formation generate the same tokens for every request, and every block returns."""
    D, bs, nb, mb, vocab, eos, mp, mn = case
    outs = {}
    for async_mode in (False, True):
        model = _ModelAdapter(DenseBatchFormer(BlockAllocator(nb, bs), D, mb, eos))
        model.m.set_async(async_mode)
        n_req = 40
        for _ in _pipelined(model, np.random.default_rng(17), n_req, vocab, eos, mp, mn,
                            _sampler_for(vocab), async_mode):
            pass
        outs[async_mode] = {i: model.m.tokens(i) for i in range(n_req)}
        assert model.m.counts()[3] == n_req and model.m.pool.free_count() == nb
    assert outs[True] == outs[False]


@pytest.mark.parametrize("case", ASYNC_CASES)
def test_async_formation_keeps_the_blocks_of_formed_rows(case):
    """While a formed step is not committed, every block its rows read or write stays out of
    the free list and belongs to one request only, even after that request finished at the
    previous step's commit (its blocks return only once no formed row of it is uncommitted)."""
    D, bs, nb, mb, vocab, eos, mp, mn = case
    m = DenseBatchFormer(BlockAllocator(nb, bs), D, mb, eos)
    m.set_async(True)
    model = _ModelAdapter(m)
    pending = []
    late_rows = 0
    for ev in _pipelined(model, np.random.default_rng(23), 40, vocab, eos, mp, mn,
                         _sampler_for(vocab), True):
        if ev[0] == "formed":
            pending.append(ev[1])
        else:
            pending.pop(0)
        owned = set().union(*(_formed_blocks(r, bs) for r in pending)) if pending else set()
        assert not {blk for _, blk in owned} & set(m.pool.free)
        owner = {}
        for rid, blk in owned:
            assert owner.setdefault(blk, rid) == rid
        late_rows += sum(1 for r in pending for q in r["row_request"] if m.req[int(q)].finished)
    assert late_rows > 0  # the case does form rows for requests that already finished


@pytest.mark.parametrize("case", ASYNC_CASES)
def test_library_former_matches_the_model_in_both_formation_modes(L, case):
    """The library equals the model row for row, synchronous and asynchronous."""
    D, bs, nb, mb, vocab, eos, mp, mn = case
    for async_mode in (False, True):
        model = _ModelAdapter(DenseBatchFormer(BlockAllocator(nb, bs), D, mb, eos))
        pool = L.BlockPool(nb, bs, mb)
        lib_form = L.BatchFormer(pool, D, mb, eos)
        model.m.set_async(async_mode)
        lib_form.set_async(async_mode)
        n_req = 40
        a = _pipelined(model, np.random.default_rng(17), n_req, vocab, eos, mp, mn, _sampler_for(vocab), async_mode)
        b = _pipelined(lib_form, np.random.default_rng(17), n_req, vocab, eos, mp, mn, _sampler_for(vocab), async_mode)
        for ea, eb in zip(a, b):
            assert ea[0] == eb[0]
            if ea[0] == "formed":
                for k in KEYS:
                    np.testing.assert_array_equal(ea[1][k], eb[1][k], err_msg=k)
            else:
                assert ea[1] == eb[1]
        assert all(lib_form.tokens(i) == model.m.tokens(i) for i in range(n_req))


def test_model_refuses_negative_prompt_ids():
    """A negative id in a formed row names a token sampled on the device in the previous step,
    so a prompt may not contain one; the request is refused and nothing changes."""
    m = DenseBatchFormer(BlockAllocator(4, 4), 4, 4, 0)
    with pytest.raises(SchedulerError):
        m.add(0, [3, -2], 1)
    assert m.counts() == (0, 0, 0, 0)
    m.add(0, [3, 0], 1)
    assert m.counts() == (1, 0, 0, 0)


def test_library_former_equals_the_model_on_arbitrary_call_sequences(L):
    """Property test: any interleaving of add (valid or not), next, commit (right or wrong row
    count), remove and set_async gives the library and the model the same outcome -- the same
    rows, moves, finished ids and tokens, or a refusal on both sides -- with every peak
    reserved and with optimistic peaks."""
    hyp = pytest.importorskip("hypothesis")
    st = pytest.importorskip("hypothesis.strategies")
    nb, bs, mb, D, eos = 10, 4, 6, 6, 7
    op = st.one_of(
        st.tuples(st.just("add"), st.integers(-1, 5), st.integers(0, 14), st.integers(0, 6)),
        st.tuples(st.just("next"), st.just(0), st.just(0), st.just(0)),
        st.tuples(st.just("commit"), st.integers(0, 2), st.integers(0, 9), st.just(0)),
        st.tuples(st.just("remove"), st.integers(-1, 5), st.just(0), st.just(0)),
        st.tuples(st.just("async"), st.integers(0, 1), st.just(0), st.just(0)),
    )

    @hyp.settings(max_examples=200, deadline=None, derandomize=True, database=None)
    @hyp.given(st.lists(op, max_size=60), st.sampled_from([0, 2]))
    def run(ops, pred):
        lib_f = L.BatchFormer(L.BlockPool(nb, bs, mb), D, mb, eos, pred)
        mod = _ModelAdapter(DenseBatchFormer(BlockAllocator(nb, bs), D, mb, eos, pred))
        formed = []  # row counts of the formed, uncommitted steps (oldest first)
        for kind, a, b, c in ops:
            if kind == "add":
                calls = [lambda f: f.add(a, list(range(3, 3 + b)), c)] * 2
            elif kind == "next":
                calls = [lambda f: {k: v.tolist() for k, v in f.next().items()},
                         lambda f: {k: v.tolist() for k, v in f.next().items()}]
            elif kind == "commit":
                n = (formed[0] if formed else 0) + (a - 1 if a != 1 else 0)  # 1: the right count
                sampled = np.array([(b + 3 * r) % 10 for r in range(max(n, 0))], np.int32)
                calls = [lambda f: f.commit(sampled)] * 2
            elif kind == "remove":
                calls = [lambda f: f.remove(a), lambda f: f.m.remove(a)]
            else:
                calls = [lambda f: f.set_async(bool(a)), lambda f: f.m.set_async(bool(a))]
            out = []
            for fn, f in zip(calls, (lib_f, mod)):
                try:
                    r = fn(f)
                    out.append(("ok", r))
                except (L.NSError, RuntimeError, SchedulerError):
                    out.append(("refused", None))
            if out[0][0] == "ok" and kind == "next":
                assert out[0][1].keys() == {k: 0 for k in out[1][1]}.keys()
                for k in out[0][1]:
                    assert out[0][1][k] == out[1][1][k], k
                assert [(m[0], m[1], m[2], list(m[3])) for m in lib_f.moves()] == \
                       [(m[0], m[1], m[2], list(m[3])) for m in mod.moves()]
                formed.append(len(out[0][1]["token_ids"]))
            else:
                assert out[0] == out[1], (kind, a, b, c, out)
            if out[0][0] == "ok" and kind == "commit":
                formed.pop(0)
            assert lib_f.counts() == mod.counts()
        for rid in range(6):
            try:
                t_lib = lib_f.tokens(rid)
            except L.NSError:
                t_lib = None
            t_mod = mod.m.tokens(rid) if rid in mod.m.req else None
            assert t_lib == t_mod

    run()
