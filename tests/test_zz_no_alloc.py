"""The allocation-free attention call, ns_attn_decode_noalloc.

It serves callers that may not call cudaMalloc (allocator or memory-pool callbacks, plugins
whose host owns all device memory, processes with a fixed device footprint): its scratch is a
fixed buffer inside the library.  These checks run it through the C ABI on two calls in a row
(the second finds the first call's leftovers in the shared buffer): each result equals
ns_attn_decode's bit for bit (the same kernel, grid and superchunk merge order) and the oracle
within the attention tolerance; a block id outside the pool is recorded in the caller's error
word while the other rows stay bitwise equal; an oversized request is refused.

The file name sorts last so that a run stopping at the first failure has run everything else.
"""
import math

import numpy as np
import pytest

from helpers import attention_case, from_dev, oracle_attention, rel_l2, storage_f64, to_dev

pytestmark = pytest.mark.gpu


def _both(case, n_q, n_kv, d, dtype, tab_override=None):
    """(noalloc output, ns_attn_decode output, the noalloc call's error word), storage dtype."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    q, kp, vp, tab, sl, nb = case
    dq, dk, dv, dl = to_dev(q), to_dev(kp), to_dev(vp), to_dev(sl)
    dt = to_dev(tab if tab_override is None else tab_override)
    ref = torch.zeros_like(dq)
    got = torch.full_like(dq, 7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    _lib.attn_decode(dq, dk, dv, dt, dl, ref, n_q, n_kv, d, 16, tab.shape[1], nb, scale, dtype)
    _lib.attn_decode_noalloc(dq, dk, dv, dt, dl, got, n_q, n_kv, d, 16, tab.shape[1], nb, scale,
                             dtype, dev_err=err)
    torch.cuda.synchronize()
    return from_dev(got), from_dev(ref), int(err.item())


def test_noalloc_matches_the_allocating_call_and_the_oracle_twice_in_a_row(cuda_lib):
    from transformer_decode_step_ns_gb300 import _lib
    cases = [
        ((32, 8, 128, "bf16"), [1, 17, 300, 700, 1100]),
        ((14, 2, 64, "f16"), [600, 5, 1040]),
    ]
    for (n_q, n_kv, d, dtype), lens in cases:
        case = attention_case(11, lens, n_q, n_kv, d, dtype)
        got, ref, err = _both(case, n_q, n_kv, d, dtype)
        assert err == 0 and _lib.device_error() == 0
        np.testing.assert_array_equal(got, ref)
        q, kp, vp, tab, sl, nb = case
        want = oracle_attention(q, kp, vp, tab, sl, d, dtype)
        g = storage_f64(got, dtype)
        assert np.isfinite(g).all()
        for b in range(len(lens)):
            assert rel_l2(g[b], want[b]) < 1e-2, (b, rel_l2(g[b], want[b]))
            assert np.abs(g[b] - want[b]).max() < 3e-2


def test_noalloc_records_a_bad_block_in_the_callers_error_word(cuda_lib):
    """A block id outside the pool: the kernel records NS_DEV_BAD_BLOCK (1) in dev_err and reads
    block 0 instead (no out-of-pool access); the other rows equal the allocating call bitwise."""
    from transformer_decode_step_ns_gb300 import _lib
    case = attention_case(21, [40, 300, 77], 32, 8, 128, "bf16")
    tab, nb = case[3], case[5]
    good, _, err = _both(case, 32, 8, 128, "bf16")
    assert err == 0
    bad = tab.copy()
    bad[0, 1] = nb + 5
    got, ref, err = _both(case, 32, 8, 128, "bf16", tab_override=bad)
    assert err == 1
    assert _lib.device_error() == 1  # the allocating call on the same table recorded it too
    np.testing.assert_array_equal(got[1:], good[1:])
    np.testing.assert_array_equal(got, ref)


def test_noalloc_refuses_requests_beyond_its_fixed_scratch(cuda_lib):
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    B, n_q, n_kv, d, mb = 1024, 64, 8, 128, 4096
    q = torch.zeros(B * n_q * d, dtype=torch.int16, device="cuda")
    pool = torch.zeros(n_kv * 16 * d, dtype=torch.int16, device="cuda")
    tab = torch.zeros(B * mb, dtype=torch.int32, device="cuda")
    sl = torch.ones(B, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.NSError) as e:
        _lib.attn_decode_noalloc(q, pool, pool, tab, sl, q, n_q, n_kv, d, 16, mb, 1, 0.1, "bf16")
    assert e.value.status == 1
    assert "fixed scratch" in str(e.value)
