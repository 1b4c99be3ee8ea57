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
