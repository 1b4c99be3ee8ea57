"""The allocation-free attention call, ns_attn_decode_noalloc.

It serves callers that may not call cudaMalloc (allocator or memory-pool callbacks, plugins
whose host owns all device memory, processes with a fixed device footprint): its scratch is a
fixed buffer inside the library.  These checks run it through the C ABI and compare it with
ns_attn_decode on the same inputs, twice in a row (the second call finds the first call's
leftovers in the shared buffer), and check that an oversized request is refused.

The file name sorts last so that a run stopping at the first failure has run everything else.
"""
import math

import numpy as np
import pytest

from helpers import attention_case, from_dev, rel_l2, storage_f64, to_dev

pytestmark = pytest.mark.gpu


def _both(case, n_q, n_kv, d, dtype):
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    q, kp, vp, tab, sl, nb = case
    dq, dk, dv, dt, dl = to_dev(q), to_dev(kp), to_dev(vp), to_dev(tab), to_dev(sl)
    ref = torch.zeros_like(dq)
    got = torch.full_like(dq, 7)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    scale = 1.0 / math.sqrt(d)
    _lib.attn_decode(dq, dk, dv, dt, dl, ref, n_q, n_kv, d, 16, tab.shape[1], nb, scale, dtype)
    _lib.attn_decode_noalloc(dq, dk, dv, dt, dl, got, n_q, n_kv, d, 16, tab.shape[1], nb, scale,
                             dtype, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return storage_f64(from_dev(got), dtype), storage_f64(from_dev(ref), dtype)


def test_noalloc_matches_the_allocating_call_twice_in_a_row(cuda_lib):
    cases = [
        ((32, 8, 128, "bf16"), [1, 17, 300, 700, 1100]),
        ((14, 2, 64, "f16"), [600, 5, 1040]),
    ]
    for (n_q, n_kv, d, dtype), lens in cases:
        got, ref = _both(attention_case(11, lens, n_q, n_kv, d, dtype), n_q, n_kv, d, dtype)
        assert np.isfinite(got).all()
        for b in range(len(lens)):
            assert rel_l2(got[b], ref[b]) < 1e-2


def test_noalloc_refuses_requests_beyond_its_fixed_scratch(cuda_lib):
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    B, n_q, n_kv, d, mb = 1024, 64, 8, 128, 4096
    x = torch.zeros(16, dtype=torch.int16, device="cuda")
    sl = torch.ones(B, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.NSError) as e:
        _lib.attn_decode_noalloc(x, x, x, x, sl, x, n_q, n_kv, d, 16, mb, 1, 0.1, "bf16")
    assert e.value.status == 1
    assert "fixed scratch" in str(e.value)
