"""Host-side rules of the benchmark's timing (no GPU): the timed steps read as two back-to-back
runs whose per-step times must agree within 15 %, else the number is flagged."""
import bench


def test_repeat_check_flags_a_spread_above_the_limit():
    r = bench.repeat_check(10.0, 10, 10.5, 10)
    assert r["ms_per_step_halves"] == [1.0, 1.05] and not r["flagged"]
    assert abs(r["spread"] - 0.05) < 1e-9
    r = bench.repeat_check(10.0, 10, 12.0, 10)
    assert r["flagged"] and abs(r["spread"] - 0.2) < 1e-9
    # halves of unequal length (odd step counts) compare per step; the faster half is the base
    r = bench.repeat_check(3.0, 3, 4.6, 4)
    assert r["ms_per_step_halves"] == [1.0, 1.15] and abs(r["spread"] - 0.15) < 1e-9
    assert not r["flagged"]
    assert bench.repeat_check(12.0, 10, 10.0, 10)["flagged"]


def test_repeat_check_needs_two_nonempty_halves():
    assert bench.repeat_check(0.0, 0, 5.0, 1) is None
    assert bench.repeat_check(5.0, 1, 0.0, 0) is None


def test_oracle_arm_builds_the_same_first_step_as_the_gpu_run():
    """The oracle arm draws its inputs on the host with the allocator model; the GPU run hands
    out blocks through the library's pool (ContinuousWorkload: every block reserved, given back
    in a seeded order, then each row's context reserved row by row, then the slot mapper).  The
    two give the same tables and slots, so the oracle samples the workload the GPU runs."""
    import math

    import numpy as np

    import synth
    from transformer_decode_step_ns_gb300 import _lib
    tok, pos, tab, seq, slots = bench.cfg4_first_step_host()
    cw = bench.ContinuousWorkload
    mb = bench.cfg4_table_width()
    nb = cw.B * mb
    seed = synth.config_seed(4)
    pool = _lib.BlockPool(nb, cw.bs, mb)
    ids = pool.reserve(nb)
    pool.release(ids[synth.permutation(seed, "cfg4.pool", nb)])
    ctx = synth.ctx_uniform(seed, "cfg4.join.ctx", 100_000, cw.ctx_lo, cw.ctx_hi)[:cw.B]
    t2 = np.zeros((cw.B, mb), dtype=np.int32)
    for b in range(cw.B):
        n = int(math.ceil(int(ctx[b]) / cw.bs))
        t2[b, :n] = pool.reserve(n)
    p2 = ctx.astype(np.int32)
    s2 = pool.prepare_step(p2, t2)
    np.testing.assert_array_equal(pos, p2)
    np.testing.assert_array_equal(tab, t2)
    np.testing.assert_array_equal(slots, s2)
    np.testing.assert_array_equal(seq, p2 + 1)
    assert tok.dtype == np.int32 and tok.shape == (cw.B,)


def test_meta_bytes_and_traffic_scaling(tmp_path, monkeypatch):
    """The upload size counts every metadata field of the packed layout (12 bytes of int32
    fields and an 8-byte slot per row, the block table, two 16-byte-aligned gaps, the logits
    pointer and two flags); traffic from a smaller captured launch scales by algorithmic bytes
    and is dropped when the kernel source has changed."""
    B, mb = 256, 319
    assert bench.cfg4_meta_bytes(B, mb) == 12 * B + 8 * B + 4 * B * mb + 16
    prof = tmp_path / "profiles"
    prof.mkdir()
    h = bench.kernel_source_hash("attention_cfg4")
    (prof / "ncu_traffic.txt").write_text(f"# x\nattention_cfg4 1000.0 {h} 800.0\n"
                                          f"attention_old 5.0 0000000000000000 1.0\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    import shutil
    shutil.copytree(bench.os.path.join(bench.os.path.dirname(bench.__file__),
                                       "transformer_decode_step_ns_gb300"),
                    tmp_path / "transformer_decode_step_ns_gb300")
    assert abs(bench.scaled_traffic("attention_cfg4", 1600.0) - 2000.0) < 1e-9
    assert bench.scaled_traffic("attention_old", 1.0) is None
    assert bench.scaled_traffic("missing", 1.0) is None
