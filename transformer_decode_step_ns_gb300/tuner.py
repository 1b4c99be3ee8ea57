"""Offline nano-batch tuner: a pairwise interference profile and a small search.

NanoFlow page, "The part that is harder than it looks: allocating a GPU you cannot partition":
concurrent kernels share the GPU as the hardware decides, so a nano-op's resource share R is
inferred by co-running it with a partner and measuring the fraction P of its solo throughput it
keeps (a GEMM keeping 40 % has R = 0.4, its partner 0.6).  The page profiles that R -> P table
pairwise (compute against memory), caps the memory-bound op's thread blocks at 8 .. 128 in
steps of 8 and sweeps batch sizes in multiples of 128, then plans the nano-batch schedule with a
two-stage MILP.  Here:

* ``pair_profile`` co-runs the paged decode attention (memory-bound), capped at each CTA
  budget, with a projection GEMM (compute-bound) on a second stream and reports, per budget,
  both kernels' solo and co-run times, their P and the inferred R.
* ``search`` replaces the MILP by measurement: every split of the dense batch into 1 .. 4
  nano-batches whose sizes are multiples of 128 (two nano-batches: every cut; three and four:
  the near-even ones in every order) is timed as a captured, replayed step; the fastest
  multi-batch splits are then timed at the attention CTA budgets the profile keeps (those
  where attention retains at least ``min_p`` of its solo throughput while co-running; the four
  best when fewer than two do), then at the (GEMM budget, attention budget) pairs given, where
  the projections of each nano-batch are capped at a number of SMs and the attention takes what
  they leave, and the fastest configuration overall is returned with the whole table.

Everything here only times library calls; the step itself runs in the library's kernels.
"""
from __future__ import annotations

import itertools
from typing import Callable, Dict, List, Optional, Sequence, Tuple


def _events():
    import torch
    return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)


def _timed(fn: Callable[[], None], reps: int, warmup: int = 2) -> float:
    """Mean ms of fn() over reps calls on the current stream (CUDA events)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    a, b = _events()
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def interference_row(budget: int, t_attn_best: float, t_attn_capped: float, t_gemm_solo: float,
                     t_attn_corun: float, t_gemm_corun: float, n_gemm: int) -> Dict:
    """One row of the R -> P table from per-launch times (seconds): P of each op relative to its
    best solo run, R_gemm = P_gemm and R_attn = 1 - R_gemm (the page's inference of a share from
    the throughput an op keeps)."""
    p_g = t_gemm_solo / t_gemm_corun
    return {"budget": budget, "attn_capped_solo_us": round(t_attn_capped * 1e6, 1),
            "attn_us": round(t_attn_corun * 1e6, 1), "gemm_us": round(t_gemm_corun * 1e6, 1),
            "n_gemm": n_gemm, "P_attn": round(t_attn_best / t_attn_corun, 3),
            "P_attn_solo": round(t_attn_best / t_attn_capped, 3), "P_gemm": round(p_g, 3),
            "R_gemm": round(p_g, 3), "R_attn": round(1.0 - p_g, 3)}


def pair_profile(attn: Callable[[int, object], None], gemm: Callable[[object], None],
                 budgets: Sequence[int] = tuple(range(8, 129, 8)), reps: int = 6) -> Dict:
    """R -> P of decode attention against a GEMM.

    ``attn(budget, stream)`` launches the attention capped at ``budget`` CTAs (0: uncapped) on
    ``stream``; ``gemm(stream)`` launches the GEMM.  Per budget: the capped attention alone, then
    a co-run in which both streams start behind one event and stay busy for about the same solo
    time (``reps`` attention launches on one stream, as many GEMM launches as take that long
    alone on the other), each stream timed by its own events.  P is the throughput an op keeps
    relative to its best solo run (uncapped attention; the GEMM), R_gemm = P_gemm and
    R_attn = 1 - R_gemm.  Returns {"attn_solo_us", "gemm_solo_us", "rows": [{budget,
    attn_capped_solo_us, attn_us, gemm_us, n_gemm, P_attn, P_attn_solo, P_gemm, R_attn,
    R_gemm}]}, times per launch.
    """
    import torch
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(sb):
        t_attn = _timed(lambda: attn(0, sb), reps)
    with torch.cuda.stream(sa):
        t_gemm = _timed(lambda: gemm(sa), reps)
    rows = []
    for b in list(budgets):
        with torch.cuda.stream(sb):
            t_b = _timed(lambda: attn(b, sb), reps, warmup=1)
        n_g = max(1, int(round(reps * t_b / t_gemm)))
        torch.cuda.synchronize()
        start = torch.cuda.Event()
        start.record()
        sa.wait_event(start)
        sb.wait_event(start)
        ga, gb = _events()
        aa, ab = _events()
        ga.record(sa)
        for _ in range(n_g):
            gemm(sa)
        gb.record(sa)
        aa.record(sb)
        for _ in range(reps):
            attn(b, sb)
        ab.record(sb)
        torch.cuda.synchronize()
        ta = aa.elapsed_time(ab) / reps
        tg = ga.elapsed_time(gb) / n_g
        rows.append(interference_row(b, t_attn * 1e-3, t_b * 1e-3, t_gemm * 1e-3, ta * 1e-3, tg * 1e-3, n_g))
    return {"attn_solo_us": round(t_attn * 1e3, 1), "gemm_solo_us": round(t_gemm * 1e3, 1),
            "rows": rows}


def candidate_splits(batch: int, granularity: int = 128, max_nano: int = 4) -> List[Optional[List[int]]]:
    """None (unsplit), every two-way cut at multiples of ``granularity``, and the near-even
    three- and four-way splits (sizes multiples of ``granularity``, the last part taking any
    remainder) in every distinct order."""
    out: List[Optional[List[int]]] = [None]
    units = batch // granularity
    rem = batch - units * granularity
    for k in range(1, units):
        out.append([k * granularity, (units - k) * granularity + rem])
    for n in range(3, max_nano + 1):
        if units < n:
            break
        base, extra = divmod(units, n)
        parts = [base + (1 if i < extra else 0) for i in range(n)]
        seen = set()
        for perm in itertools.permutations(parts):
            if perm in seen:
                continue
            seen.add(perm)
            sizes = [p * granularity for p in perm]
            sizes[-1] += rem
            out.append(sizes)
    return out


def search(step: Callable[..., None], batch: int,
           profile: Optional[Dict] = None, granularity: int = 128, max_nano: int = 4,
           budgets: Sequence[int] = tuple(range(8, 129, 8)), min_p: float = 0.5, top: int = 3,
           reps: int = 5, timer: Optional[Callable[[Callable[[], None], int], float]] = None,
           gemm_pairs: Sequence[Tuple[int, int]] = ()) -> Dict:
    """Measure the candidate splits and CTA budgets of one dense batch.

    ``step(sizes, budget)`` runs one step with that nano-batch split (None: unsplit) and
    attention CTA budget (0: none); for a pair of ``gemm_pairs`` = (GEMM budget, attention
    budget) it is called as ``step(sizes, budget, gemm_budget)``.  Attention budgets come from
    ``profile`` when given (those whose co-run P_attn >= min_p, or the four best), else
    ``budgets``.  ``timer(fn, reps)`` returns the ms per call of fn (default: CUDA events).
    Returns {"best": {sizes, budget, gemm_budget, ms}, "table": [...], "budgets_kept"} in
    measurement order.
    """
    table = []
    timer = timer or _timed

    def run(sizes, budget, gemm_budget=0):
        if gemm_budget:
            ms = timer(lambda: step(sizes, budget, gemm_budget), reps)
        else:
            ms = timer(lambda: step(sizes, budget), reps)
        table.append({"sizes": sizes or [batch], "budget": budget, "gemm_budget": gemm_budget,
                      "ms": round(ms, 4)})
        return ms

    stage1 = [(run(s, 0), i, s) for i, s in enumerate(candidate_splits(batch, granularity, max_nano))]
    keep = list(budgets)
    if profile is not None:
        keep = [r["budget"] for r in profile["rows"] if r["P_attn"] >= min_p]
        if len(keep) < 2:  # nothing clears the bar: still try the four best
            keep = [r["budget"] for r in sorted(profile["rows"], key=lambda r: -r["P_attn"])[:4]]
    multi = sorted((t, i, s) for t, i, s in stage1 if s is not None)[:top]
    for _, _, s in multi:
        for b in keep:
            run(s, b)
    for _, _, s in multi:
        for g, b in gemm_pairs:
            run(s, b, g)
    best = min(table, key=lambda r: r["ms"])
    return {"best": best, "table": table, "budgets_kept": list(keep)}


__all__ = ["candidate_splits", "pair_profile", "search"]
