"""The seeded generator's host C twin (synth/csrc/fill_host.c) against its numpy definition:
the same values bit for bit, over offsets, both storage types, and the fp16 edge cases
(subnormal results, overflow to infinity, exact rounding midpoints)."""
import numpy as np
import pytest

import synth


@pytest.mark.parametrize("dtype,std,mean,offset", [
    ("bf16", 0.02, 0.0, 0), ("bf16", 1.0, 0.0, 987_654_321), ("f16", 1.0, 0.0, 12_345),
    ("f16", 3e-5, 0.0, 0), ("f16", 3e4, 0.0, 7), ("bf16", 0.1, 1.0, 3), ("f16", 0.05, 1.0, 99)])
def test_host_twin_equals_the_numpy_definition(dtype, std, mean, offset):
    n = 1 << 18
    with np.errstate(over="ignore"):
        want = synth.normal(31, "twin", (n,), dtype, std=std, mean=mean, offset=offset)
    for threads in (1, 3):
        got = synth.normal_threads(31, "twin", (n,), dtype, std=std, mean=mean, offset=offset,
                                   threads=threads)
        np.testing.assert_array_equal(got.view(np.uint16), want.view(np.uint16))


def test_host_twin_rounds_fp16_midpoints_to_even():
    """fp32 values exactly halfway between two fp16 values, written through the same
    fp64 -> fp32 -> fp16 path with mean = the value and std = 0."""
    for v in (1.0 + 2.0 ** -11, 1.0 + 3 * 2.0 ** -11, 2.0 ** -24 * 1.5, 65520.0):
        want = np.float32(v).astype(np.float16).view(np.uint16)
        got = synth.normal_threads(1, "mid", (1,), "f16", std=0.0, mean=v, threads=1)
        assert got.view(np.uint16)[0] == want, v
