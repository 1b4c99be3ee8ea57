"""GPU parity of the individual kernels against the oracle, through the C ABI.

Tolerances: the decode-step requirement is per-tensor relative L2 <= 1e-2 for fp16/bf16
math; the projections (fp32 accumulation of exact 16-bit products) are held to 1e-4; where the
result is a copy of an input (single cached token) or must not depend on the rest of the
batch / the physical block order, the comparison is bitwise.
"""
import math

import numpy as np
import pytest

import synth
from helpers import (attention_case, from_dev, oracle_attention, rel_l2, run_attention,
                     storage_f64, to_dev)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n_q,n_kv,d,dtype,lens", [
    (32, 8, 128, "bf16", [1, 15, 16, 17, 255, 256, 257, 700]),
    (14, 2, 64, "f16", [129, 1, 600, 1040]),
    (64, 8, 128, "bf16", [3, 513, 1024]),
    (8, 8, 128, "f16", [40, 300]),
    (16, 8, 64, "bf16", [77, 1]),
])
def test_attention_matches_oracle(cuda_lib, n_q, n_kv, d, dtype, lens):
    q, kp, vp, tab, sl, nb = attention_case(3, lens, n_q, n_kv, d, dtype)
    got = storage_f64(run_attention(q, kp, vp, tab, sl, n_q, n_kv, d, dtype, nb), dtype)
    ref = oracle_attention(q, kp, vp, tab, sl, d, dtype)
    for b in range(len(lens)):
        assert rel_l2(got[b], ref[b]) < 1e-2, b
    assert np.abs(got - ref).max() < 3e-2


def test_attention_at_the_longest_supported_row(cuda_lib):
    """Rows of 65,536 tokens (4096 blocks: the 64-superchunk cap), one past half of it, and 1,
    next to each other; each matches the oracle."""
    lens = [65536, 32769, 1]
    q, kp, vp, tab, sl, nb = attention_case(13, lens, 32, 8, 128, "bf16", mb=4096)
    got = storage_f64(run_attention(q, kp, vp, tab, sl, 32, 8, 128, "bf16", nb), "bf16")
    ref = oracle_attention(q, kp, vp, tab, sl, 128, "bf16")
    for b in range(len(lens)):
        assert rel_l2(got[b], ref[b]) < 1e-2, b
    assert np.abs(got - ref).max() < 3e-2


def test_attention_single_cached_token_returns_v_exactly(cuda_lib):
    q, kp, vp, tab, sl, nb = attention_case(4, [1, 1, 1], 32, 8, 128, "bf16")
    got = run_attention(q, kp, vp, tab, sl, 32, 8, 128, "bf16", nb)
    for b in range(3):
        for h in range(32):
            np.testing.assert_array_equal(got[b, h], vp[tab[b, 0], h // 4, 0])


def test_attention_block_permutation_and_batch_independence_bitwise(cuda_lib):
    lens = [300, 17, 1200, 64]
    q, kp, vp, tab, sl, nb = attention_case(5, lens, 32, 8, 128, "bf16")
    base = run_attention(q, kp, vp, tab, sl, 32, 8, 128, "bf16", nb)
    perm = np.random.default_rng(0).permutation(nb)
    kp2 = np.empty_like(kp)
    vp2 = np.empty_like(vp)
    kp2[perm] = kp
    vp2[perm] = vp
    tab2 = np.where(tab >= 0, perm[tab], tab).astype(np.int32)
    out2 = run_attention(q, kp2, vp2, tab2, sl, 32, 8, 128, "bf16", nb)
    np.testing.assert_array_equal(out2, base)
    for b in range(len(lens)):
        one = run_attention(q[b:b + 1], kp, vp, tab[b:b + 1], sl[b:b + 1], 32, 8, 128, "bf16", nb)
        np.testing.assert_array_equal(one[0], base[b])


def test_attention_cta_budget_is_bitwise_neutral(cuda_lib):
    """Capping the attention at 1, 8 or 76 CTAs (the tuner's budgets) changes no bit."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    lens = [300, 17, 1200, 64, 2100, 5]
    q, kp, vp, tab, sl, nb = attention_case(6, lens, 32, 8, 128, "bf16")
    base = run_attention(q, kp, vp, tab, sl, 32, 8, 128, "bf16", nb)
    dq, dk, dv, dt, dl = to_dev(q), to_dev(kp), to_dev(vp), to_dev(tab), to_dev(sl)
    for budget in (1, 8, 76):
        out = torch.zeros_like(dq)
        _lib.attn_decode(dq, dk, dv, dt, dl, out, 32, 8, 128, 16, tab.shape[1], nb,
                         1.0 / math.sqrt(128), "bf16", cta_budget=budget)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(from_dev(out), base)
    with pytest.raises(_lib.NSError):
        _lib.check(_lib.lib().ns_attn_decode_capped(
            dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), dt.data_ptr(), dl.data_ptr(), dq.data_ptr(),
            6, 32, 8, 128, 16, tab.shape[1], nb, 0.1, 1, -1, None))  # negative budget


@pytest.mark.parametrize("n_q,n_kv,d,dtype", [(32, 8, 128, "bf16"), (14, 2, 64, "f16")])
def test_attention_unit_queue_and_fixed_deal_give_the_same_bits(cuda_lib, n_q, n_kv, d, dtype):
    """From six units per CTA on, a launch hands out its later units from a global counter,
    rows with the longest superchunks first; below that each CTA takes a fixed share.  Budgets
    of 4 and 16 CTAs put this batch (40 rows of 1 to 2100 tokens: superchunks of fewer blocks
    than warps next to ones of 33 to 64 blocks) in the queue, the full grid does not.  Every
    budget gives the same bits, which match the oracle; queued launches repeated back to back
    (the launch that takes the last ticket resets the counter) and a fixed-deal launch after
    them change nothing."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    lens = [1, 2, 3, 5, 7, 16, 17, 33, 64, 100, 513, 1024, 1025, 2047, 2100, 300, 1200, 48, 80,
            4] * 2
    q, kp, vp, tab, sl, nb = attention_case(27, lens, n_q, n_kv, d, dtype)
    base = run_attention(q, kp, vp, tab, sl, n_q, n_kv, d, dtype, nb)
    ref = oracle_attention(q, kp, vp, tab, sl, d, dtype)
    got = storage_f64(base, dtype)
    for b in range(len(lens)):
        assert rel_l2(got[b], ref[b]) < 1e-2, b
    dq, dk, dv, dt, dl = to_dev(q), to_dev(kp), to_dev(vp), to_dev(tab), to_dev(sl)
    for budget in (4, 4, 16, 16, 4, 0):
        out = torch.zeros_like(dq)
        _lib.attn_decode(dq, dk, dv, dt, dl, out, n_q, n_kv, d, 16, tab.shape[1], nb,
                         1.0 / math.sqrt(d), dtype, cta_budget=budget)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(from_dev(out), base)
    assert _lib.device_error() == 0


def test_attention_bounds_checks_record_errors_and_skip_the_access(cuda_lib):
    """The kernel's own checks (each substitutes a safe value before any memory access, so no
    fault is induced): a block id outside the pool records NS_DEV_BAD_BLOCK (1) and reads block 0
    instead; a seq_len beyond the block table records NS_DEV_BAD_LENGTH (3) and skips the row.
    The other rows' outputs are unchanged bitwise."""
    from transformer_decode_step_ns_gb300 import _lib
    q, kp, vp, tab, sl, nb = attention_case(21, [40, 300], 32, 8, 128, "bf16")
    good = run_attention(q, kp, vp, tab, sl, 32, 8, 128, "bf16", nb)
    assert _lib.device_error() == 0
    bad_tab = tab.copy()
    bad_tab[0, 1] = nb + 5
    out = run_attention(q, kp, vp, bad_tab, sl, 32, 8, 128, "bf16", nb)
    assert _lib.device_error() == 1
    np.testing.assert_array_equal(out[1], good[1])
    bad_sl = sl.copy()
    bad_sl[1] = tab.shape[1] * 16 + 1
    out = run_attention(q, kp, vp, tab, bad_sl, 32, 8, 128, "bf16", nb)
    assert _lib.device_error() == 3
    np.testing.assert_array_equal(out[0], good[0])
    assert _lib.device_error() == 0  # reading the word cleared it


def test_attention_rejects_unsupported_shapes(cuda_lib):
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    x = torch.zeros(16384, dtype=torch.int16, device="cuda")  # as large as either call reads
    t = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(_lib.NSError) as e:
        _lib.attn_decode(x, x, x, t, t, x, 12, 4, 96, 16, 1, 1, 0.1, "bf16")  # d = 96
    assert e.value.status == 4
    with pytest.raises(_lib.NSError) as e:
        _lib.attn_decode(x, x, x, t, t, x, 12, 5, 128, 16, 1, 1, 0.1, "bf16")  # Hq % Hkv
    assert e.value.status == 1


@pytest.mark.parametrize("m,n,k,dtype", [
    (1, 128, 64, "bf16"), (16, 256, 128, "f16"), (33, 1152, 896, "f16"),
    (7, 896, 4864, "bf16"), (32, 9728, 896, "f16"), (256, 384, 512, "bf16"),
    (300, 256, 1024, "bf16"), (1000, 512, 256, "f16"), (2048, 1024, 2048, "bf16"),
    # >= 152 output tiles: one split, tiles of 160 and 256 tokens staged in two passes
    (300, 19456, 256, "bf16"), (256, 19456, 512, "f16"),
])
def test_linear_matches_fp64(cuda_lib, m, n, k, dtype):
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    w = synth.normal(9, f"w{m}{n}{k}", (n, k), dtype, std=0.05)
    x = synth.normal(9, f"x{m}{n}{k}", (m, k), dtype)
    y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    _lib.linear(to_dev(w), to_dev(x), y, m, n, k, dtype)
    torch.cuda.synchronize()
    got = y.cpu().numpy().astype(np.float64)
    ref = storage_f64(x, dtype) @ storage_f64(w, dtype).T
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) < 1e-4
    assert _lib.device_error() == 0


def test_linear_rows_do_not_depend_on_the_batch(cuda_lib):
    """Row independence (NanoFlow: rows of the activation matrix are independent), bitwise."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    n, k = 1152, 896
    w = to_dev(synth.normal(10, "w", (n, k), "f16", std=0.05))
    x = synth.normal(10, "x", (40, k), "f16")
    full = torch.empty((40, n), dtype=torch.float32, device="cuda")
    _lib.linear(w, to_dev(x), full, 40, n, k, "f16")
    for lo, hi in ((0, 1), (3, 19), (19, 40)):
        part = torch.empty((hi - lo, n), dtype=torch.float32, device="cuda")
        _lib.linear(w, to_dev(x[lo:hi]), part, hi - lo, n, k, "f16")
        torch.cuda.synchronize()
        assert torch.equal(part, full[lo:hi])


@pytest.mark.parametrize("n,k,m,parts", [
    # 152 feature tiles: no k split; persistent from two 256-token tiles (257 rows) on
    (19456, 256, 600, ((0, 40), (40, 600), (7, 71), (100, 400), (0, 257), (256, 600))),
    (19456, 1024, 1100, ((0, 64), (64, 1100), (300, 812))),
])
def test_linear_rows_are_bitwise_the_same_in_either_gemm_kernel(cuda_lib, n, k, m, parts):
    """An unsplit weight runs the cluster kernel for short launches and the persistent kernel
    once it has two 256-token output tiles per SM; both accumulate the same k-blocks in the same order and apply the same epilogue roundings,
    so a row's result does not depend on which launch (or batch) it is in."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    w = to_dev(synth.normal(12, f"w{n}", (n, k), "bf16", std=0.05))
    x = synth.normal(12, f"x{n}", (m, k), "bf16")
    full = torch.empty((m, n), dtype=torch.float32, device="cuda")
    _lib.linear(w, to_dev(x), full, m, n, k, "bf16")
    for lo, hi in parts:
        part = torch.empty((hi - lo, n), dtype=torch.float32, device="cuda")
        _lib.linear(w, to_dev(x[lo:hi]), part, hi - lo, n, k, "bf16")
        torch.cuda.synchronize()
        assert torch.equal(part, full[lo:hi]), (lo, hi)
    assert _lib.device_error() == 0
    rows = np.r_[0:8, m - 8:m]
    ref = storage_f64(x[rows], "bf16") @ storage_f64(from_dev(w), "bf16").T
    assert rel_l2(full[rows].cpu().numpy(), ref) < 1e-4


def test_vocabulary_wide_head_at_decode_batches(cuda_lib):
    """A weight with four output tiles per SM (a vocabulary-wide head) runs the persistent kernel
    even at decode batches (1..64 rows, token tiles of 16..64): rows match fp64 and do not depend
    on the launch they are in."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    n, k, m = 4 * sms * 128, 256, 40
    w = to_dev(synth.normal(13, "wv", (n, k), "f16", std=0.05))
    x = synth.normal(13, "xv", (m, k), "f16")
    full = torch.empty((m, n), dtype=torch.float32, device="cuda")
    _lib.linear(w, to_dev(x), full, m, n, k, "f16")
    for lo, hi in ((0, 1), (3, 20), (20, 40)):
        part = torch.empty((hi - lo, n), dtype=torch.float32, device="cuda")
        _lib.linear(w, to_dev(x[lo:hi]), part, hi - lo, n, k, "f16")
        torch.cuda.synchronize()
        assert torch.equal(part, full[lo:hi]), (lo, hi)
    assert _lib.device_error() == 0
    ref = storage_f64(x, "f16") @ storage_f64(from_dev(w).view(np.float16), "f16").T
    assert rel_l2(full.cpu().numpy(), ref) < 1e-4


def test_greedy_argmax_ties_to_lowest(cuda_lib):
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    logits = torch.randn(5, 151936, device="cuda")
    logits[2, 7] = 50.0
    logits[2, 90000] = 50.0
    logits[4, :] = 1.0
    out = torch.empty(5, dtype=torch.int32, device="cuda")
    _lib.greedy_argmax(logits, out)
    ref = torch.argmax(logits, dim=-1).to(torch.int32)
    ref[2] = 7
    ref[4] = 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("vocab", [1, 5, 1001, 128256])
def test_greedy_argmax_slices_and_nan(cuda_lib, vocab):
    """The row is split over several CTAs: ragged and empty slices, a maximum in the last
    slice, ties across slices, and NaN (never chosen; an all-NaN row gives 0)."""
    import torch
    from transformer_decode_step_ns_gb300 import _lib
    g = torch.Generator(device="cpu").manual_seed(vocab)
    logits = torch.randn(6, vocab, generator=g).cuda()
    logits[1, :] = float("nan")
    logits[1, vocab // 2] = -3.0
    logits[2, vocab - 1] = 100.0
    logits[3, :] = float("nan")
    logits[4, :] = 2.0
    out = torch.empty(6, dtype=torch.int32, device="cuda")
    _lib.greedy_argmax(logits, out)
    ref = torch.argmax(logits, dim=-1).to(torch.int32)
    ref[1] = vocab // 2
    ref[2] = vocab - 1
    ref[3] = 0
    ref[4] = 0
    assert torch.equal(out.cpu(), ref.cpu())
