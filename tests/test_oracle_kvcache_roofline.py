"""CPU pins of the allocator model, the roofline arithmetic and the input generator."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
from oracle.kvcache import AllocatorError, BlockAllocator
from transformer_decode_step_ns_gb300 import roofline as rl

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))


# ------------------------------------------------------------------ allocator model


def test_allocator_model_fifo_and_slot_formula():
    a = BlockAllocator(6, 4)
    tables = np.zeros((2, 3), dtype=np.int32)
    slots = a.prepare_step(tables, np.array([0, 0]))
    assert tables[:, 0].tolist() == [0, 1] and slots.tolist() == [0, 4]
    slots = a.prepare_step(tables, np.array([1, 3]))
    assert slots.tolist() == [1, 7] and a.free_count() == 4
    slots = a.prepare_step(tables, np.array([4, 4]))
    assert tables[:, 1].tolist() == [2, 3] and slots.tolist() == [8, 12]
    a.release([1, 3])
    assert list(a.free) == [4, 5, 1, 3]
    # every slot decodes back to (block, offset) through the table
    for b in range(2):
        for p in range(6):
            s = oracle.slot_of(tables[b], p, 4)
            assert s // 4 == tables[b, p // 4] and s % 4 == p % 4


def test_allocator_model_errors_leave_state_unchanged():
    a = BlockAllocator(2, 4)
    tables = np.zeros((3, 2), dtype=np.int32)
    with pytest.raises(AllocatorError):
        a.prepare_step(tables, np.array([0, 0, 0]))
    assert a.free_count() == 2 and not tables.any()
    with pytest.raises(AllocatorError):
        a.prepare_step(tables, np.array([0, 8, 1]))
    assert a.free_count() == 2


def test_allocator_model_rejects_returning_a_block_it_does_not_hold():
    """A slot holds one token of one request, so a block returned twice (or never handed out)
    would later go to two requests at once; the release is refused and nothing changes."""
    a = BlockAllocator(4, 4)
    got = a.alloc(2)
    assert got == [0, 1]
    for bad in ([2], [0, 0], [1, 3], [0, 1, 0]):
        with pytest.raises(AllocatorError):
            a.release(bad)
        assert list(a.free) == [2, 3] and a.held == {0, 1}
    a.release([1])
    with pytest.raises(AllocatorError):
        a.release([1])
    assert list(a.free) == [2, 3, 1]
    tables = np.zeros((1, 2), dtype=np.int32)
    a.prepare_step(tables, np.array([0]))     # hands out block 2 through a table
    a.release([int(tables[0, 0]), 0])
    assert list(a.free) == [3, 1, 2, 0] and not a.held


def test_allocator_model_never_hands_out_a_block_twice():
    rng = np.random.default_rng(0)
    a = BlockAllocator(64, 16)
    owned = {}
    for step in range(400):
        if owned and rng.random() < 0.3:
            k = rng.choice(list(owned))
            a.release(owned.pop(k))
        else:
            n = int(rng.integers(1, 5))
            if n <= a.free_count():
                owned[step] = a.alloc(n)
        flat = [x for v in owned.values() for x in v]
        assert len(flat) == len(set(flat))
        assert len(flat) + a.free_count() == 64


# ------------------------------------------------------------------ roofline arithmetic


def test_kv_rows_layout_closed_form():
    """Every pool element holds its own flat index, so the row element at (l, t, c) must be the
    index of (block, head, offset, dim) that the row layout names: K heads first, then V."""
    L, nb, hkv, bs, d = 2, 5, 3, 4, 8
    base = np.arange(nb * hkv * bs * d, dtype=np.float64).reshape(nb, hkv, bs, d)
    kp = [base + 1e6 * l for l in range(L)]
    vp = [base + 1e6 * l + 5e5 for l in range(L)]
    slots = [17, 0, 9, 19]
    rows = oracle.kv_rows(kp, vp, slots)
    assert rows.shape == (L, len(slots), 2 * hkv * d)
    for l in range(L):
        for t, s in enumerate(slots):
            blk, off = divmod(s, bs)
            for c in range(2 * hkv * d):
                kv, col = divmod(c, hkv * d)
                h, i = divmod(col, d)
                want = ((blk * hkv + h) * bs + off) * d + i + 1e6 * l + 5e5 * kv
                assert rows[l, t, c] == want


def test_kv_scatter_inverts_kv_rows_and_touches_only_its_slots():
    rng = np.random.default_rng(7)
    L, nb, hkv, bs, d = 3, 6, 2, 4, 16
    slots = rng.permutation(nb * bs)[:9]
    rows = rng.standard_normal((L, len(slots), 2 * hkv * d))
    kp = [np.zeros((nb, hkv, bs, d)) for _ in range(L)]
    vp = [np.zeros((nb, hkv, bs, d)) for _ in range(L)]
    oracle.kv_scatter(kp, vp, rows, slots)
    np.testing.assert_array_equal(oracle.kv_rows(kp, vp, slots), rows)
    for l in range(L):
        # each slot's 2 * hkv * d elements, and nothing else, became nonzero
        assert np.count_nonzero(kp[l]) + np.count_nonzero(vp[l]) == len(slots) * 2 * hkv * d


def test_request_slots_by_hand():
    # table [5, 2, 9], block size 4, positions 3..8: block 5 offset 3, block 2 offsets 0..3,
    # block 9 offset 0
    got = oracle.request_slots(np.array([5, 2, 9]), 3, 6, 4)
    np.testing.assert_array_equal(got, [23, 8, 9, 10, 11, 36])


def test_bandwidth_floor_matches_nanoserve():
    g = GOLDEN["nanoserve_bandwidth_floor_ms"]
    nbytes = g["bytes_mib"] * 2 ** 20
    lo = rl.t_hbm(nbytes, g["bw_gbs_high"] * 1e9) * 1e3
    hi = rl.t_hbm(nbytes, g["bw_gbs_low"] * 1e9) * 1e3
    assert lo - g["tolerance_ms"] <= g["value_ms"] <= hi + g["tolerance_ms"]


def test_batch_scaling_tok_s_matches_nanoserve():
    g = GOLDEN["nanoserve_batch_scaling"]
    assert abs(1 / (g["step_ms_b1"] * 1e-3) / g["tok_s_b1"] - 1) < g["rel_tolerance"]
    assert abs(32 / (g["step_ms_b32"] * 1e-3) / g["tok_s_b32"] - 1) < g["rel_tolerance"]


def test_ridge_points_match_roofline_page():
    for key in ("ridge_h100_bf16", "ridge_4090_fp16"):
        g = GOLDEN[key]
        r = rl.ai_ridge(g["peak_tflops"] * 1e12, g["bw_tbs"] * 1e12)
        assert abs(r / g["value"] - 1) < g["rel_tolerance"]
    g = GOLDEN["decode_ai_crossing_batch"]
    assert rl.ai_decode(g["value"]) == pytest.approx(g["ridge"])
    # below the ridge the attainable rate is BW x AI, above it the peak
    assert rl.roofline_perf(989e12, 3.35e12, 10) == pytest.approx(33.5e12)
    assert rl.roofline_perf(989e12, 3.35e12, 1000) == pytest.approx(989e12)


def test_3b_4090_table_rows():
    g = GOLDEN["table_3b_4090"]
    bw = g["bw_tbs"] * 1e12
    assert 1 / rl.t_hbm(g["weights_gb_bf16"] * 1e9, bw) == pytest.approx(g["ceiling_tok_s"],
                                                                          rel=0.01)
    for row in g["rows"]:
        w = g["weights_gb_bf16"] if "BF16" in row["config"] else g["weights_gb_int4"]
        assert rl.t_hbm(w * 1e9, bw) * 1e3 == pytest.approx(row["t_hbm_ms"])
        ts = rl.t_step(w * 1e9, bw, row["t_fixed_ms"] * 1e-3)
        assert ts * 1e3 == pytest.approx(row["t_step_ms"])
        assert 1 / ts == pytest.approx(row["tok_s"], rel=0.01)


def test_launch_bound_70b_numbers():
    g = GOLDEN["launch_bound_70b"]
    t = rl.t_launch(g["layers"] * g["kernels_per_layer"], g["launch_us"] * 1e-6)
    assert t * 1e3 == pytest.approx(g["t_launch_ms"])
    tm = rl.t_hbm(g["weights_gb"] * 1e9, g["bw_tbs"] * 1e12)
    assert tm * 1e3 == pytest.approx(g["t_mem_ms"], rel=0.01)
    assert 1 / tm == pytest.approx(g["tok_s"], rel=0.02)


def test_nanoflow_optimum_formula_and_the_printed_inconsistency():
    g = GOLDEN["nanoflow_optimal"]
    v = rl.optimal_tokens_per_s(g["peak_tflops"] * 1e12, g["n_params_b"] * 1e9)
    assert v == pytest.approx(g["formula_value"])
    assert abs(v - g["printed_value"]) > 100


def test_step_work_counts_weights_once():
    shape = synth.qwen05b_shape()
    w = rl.decode_step_work(shape, [129])
    # weights plus the final norm: the 943 MiB figure
    assert abs(w.weight_bytes / 2 ** 20 - 943) < 1.0
    assert w.kv_read_bytes == 129 * 24 * 2 * 128 * 2
    assert rl.step_roofline_time(2e12, 1e9, 1e15, 1e12) == pytest.approx(2e-3)


# ------------------------------------------------------------------ input generator


@pytest.mark.parametrize("dtype,tie", [("f16", True), ("bf16", False)])
def test_step_weight_bytes_equal_the_arrays_a_step_reads(dtype, tie):
    """Brute force: every layer array (projections and both norm gains), the final norm and
    the head (the embedding when tied) of a generated model, byte for byte; the embedding table
    of an untied model is only gathered, B rows, and counts under activations."""
    shape = synth.tiny_shape(dtype=dtype, tie=tie, n_layers=3, hidden=64, n_q_heads=4,
                             n_kv_heads=2, head_dim=16, ffn=96, vocab=80)
    w = synth.model_weights(shape, 5)
    arrays = [a for lw in w["layers"] for a in lw.values()]
    arrays += [w["final_norm"], w["embed"] if tie else w["lm_head"]]
    assert len(arrays) == 9 * 3 + 2
    assert rl.decode_step_work(shape, [7, 1]).weight_bytes == sum(a.nbytes for a in arrays)


def test_attention_bytes_equal_the_kv_rows_a_launch_gathers():
    """Brute force: the bytes of the K and V rows gathered (``kv_rows``) for every cached token
    of every request, against the per-launch figure the roofline divides by."""
    rng = np.random.default_rng(3)
    nb, hkv, bs, d = 40, 2, 4, 8
    kp = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    vp = rng.standard_normal((nb, hkv, bs, d)).astype(np.float16)
    lens = [1, 4, 5, 17]
    ids = iter(rng.permutation(nb).tolist())
    total = 0
    for n in lens:
        table = np.array([next(ids) for _ in range(-(-n // bs))], dtype=np.int32)
        total += oracle.kv_rows([kp], [vp], oracle.request_slots(table, 0, n, bs)).nbytes
    assert rl.attention_bytes(lens, hkv, d, elt_bytes=2) == total


def test_generator_is_counter_based_and_seeded():
    a = synth.normal(5, "x", (1000,), "bf16")
    b = synth.normal(5, "x", (400,), "bf16", offset=600)
    np.testing.assert_array_equal(a[600:], b)
    assert not np.array_equal(a, synth.normal(6, "x", (1000,), "bf16"))
    assert not np.array_equal(a, synth.normal(5, "y", (1000,), "bf16"))
    z = synth.storage_to_f64(synth.normal(1, "big", (200000,), "f16"), "f16")
    assert abs(z.mean()) < 0.01 and abs(z.std() - 1) < 0.01


def test_splitmix64_reference_values():
    # splitmix64 seeded with 0: first outputs of the published generator
    out = synth.raw_words(0, 0, 3)
    assert [int(v) for v in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_decode_batch_tables_and_slots():
    db = synth.decode_batch(3, "t", [0, 15, 16, 40], 100, 16, num_blocks=20)
    used = [int(x) for b in range(4) for x in db.block_tables[b, : (int(db.seq_lens[b]) + 15) // 16]]
    assert len(used) == len(set(used))
    for b in range(4):
        assert db.slot_mapping[b] == oracle.slot_of(db.block_tables[b], int(db.positions[b]), 16)
    assert (db.seq_lens == db.positions + 1).all()
