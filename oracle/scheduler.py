"""Reference model of the constant-dense-batch former (host-side batch formation).

Test infrastructure only.  The library's C++ former (``ns_sched_*``) must reproduce this model
bit for bit (same rows, same order, same block ids, same errors) on any sequence of calls.

Source: "NanoFlow: ..." page, "Runtime details that keep the pipeline fed": to keep the batch
shape constant, the scheduler takes the unfinished decode requests first and then fills the
batch up to exactly the target number of tokens with prefill chunks cut at token granularity
(the chunked-prefill idea it attributes to SarathiServe).  The details are this library's own
reading (the page gives none):

* One step has at most ``dense_tokens`` rows.  Decode rows come first, one per running request
  (requests whose prompt is complete), in the order their prompts completed; if more requests
  run than fit, the first ``dense_tokens`` do and the rest wait for a later step.
* The remaining rows go to prompts in arrival order.  A prompt contributes its next
  ``min(room, remaining)`` tokens as consecutive rows (positions done .. done + c - 1 over the
  request's own block table); if the block pool cannot hold them all the chunk is cut to what
  fits, and the fill stops at the first prompt that gets nothing.
* A row samples a token (``row_samples`` = 1) when it is a decode row or the last token of a
  prompt.  A prompt whose last row is formed joins the end of the running order at once (its
  first decode row comes in the next step).  After the step the caller commits the sampled
  tokens: a request finishes when it samples ``eos_token`` or reaches ``max_new_tokens``
  generated tokens, and its blocks return to the pool in table order.
* Prompt token ids are non-negative: a negative id in a formed row names a token sampled on the
  device (asynchronous formation, below).
* Blocks are reserved from the pool as positions cross block boundaries, decode rows first
  (in row order), then the chunks (in row order).
* Predicted peak memory (same passage: requests that outgrow their predicted peak are moved
  to the host and later reloaded, never recomputed).  A request's predicted peak is the blocks
  of its first prompt_len + min(max_new, predicted_new) - 1 positions (predicted_new = 0:
  max_new).  A prompt starts (gets its first row) only when the free blocks cover its predicted
  peak plus what the admitted requests (started prompts and running requests) still need to
  reach theirs and what the preempted requests need to resume (the blocks of their cached tokens
  and next position); started prompts always continue.
* When the first ``dense_tokens`` running requests need more new blocks than are free, the
  running request that started last is preempted (repeatedly): the caller saves its cached
  tokens (positions 0 .. prompt_len + generated - 2) from its blocks, the blocks return to the
  pool and the request waits, first in, first out, to be resumed.  In a step that preempted
  nothing, waiting requests resume in that order while the free blocks, after this step's
  decode blocks, cover the blocks of their cached tokens plus their next position: new blocks
  are reserved, the caller reloads the tokens into them, and the request runs again (last in
  the running order).  Moves are listed saves first; the caller performs them in order on the
  step's stream before the step.
* A decode row's token is the request's last generated token at position
  prompt_len + generated - 1; seq_len = position + 1; slot = table[p // bs] * bs + p % bs.
* Asynchronous formation (same passage: the batch of iteration i + 1 is formed before
  iteration i finishes, so an end-of-sequence token is seen one iteration late).  With it on, one
  formed step may be outstanding when the next is formed: a request whose previous row's token is
  not committed yet decodes the token sampled at that row, written as token id -(row + 1); a
  prompt joins the running order when its last row is formed (in either mode); a request counts
  its formed rows toward max_new_tokens, and one that samples eos keeps the row already formed
  for the next step, whose token is ignored, and returns its blocks once no formed row of it is
  outstanding.  It requires every peak reserved (predicted_new = 0), so nothing is preempted.
"""
from __future__ import annotations

from collections import deque
from dataclasses import dataclass, field
from typing import Dict, List, Optional

import numpy as np

from .kvcache import AllocatorError, BlockAllocator


class SchedulerError(RuntimeError):
    pass


@dataclass
class _Request:
    rid: int
    prompt: List[int]
    max_new: int
    peak: int                         # predicted peak, in blocks
    done: int = 0                     # prompt tokens already placed in a step
    gen: List[int] = field(default_factory=list)
    table: List[int] = field(default_factory=list)
    finished: bool = False
    inflight: List[tuple] = field(default_factory=list)   # (step, row) of formed sampling rows


@dataclass
class StepRows:
    token_ids: np.ndarray
    positions: np.ndarray
    block_tables: np.ndarray
    seq_lens: np.ndarray
    slot_mapping: np.ndarray
    row_request: np.ndarray
    row_samples: np.ndarray


@dataclass
class Move:
    kind: int           # 0: save the cached tokens from `table`, 1: reload them into `table`
    rid: int
    n_tokens: int
    table: List[int]


class DenseBatchFormer:
    def __init__(self, pool: BlockAllocator, dense_tokens: int, max_blocks_per_seq: int,
                 eos_token: int, predicted_new: int = 0):
        if dense_tokens < 1 or max_blocks_per_seq < 1 or predicted_new < 0:
            raise SchedulerError("dense_tokens, max_blocks_per_seq positive; predicted_new >= 0")
        self.pool, self.D, self.mb, self.eos = pool, dense_tokens, max_blocks_per_seq, eos_token
        self.pred = predicted_new
        self.req: Dict[int, _Request] = {}
        self.prefill: deque = deque()   # request ids with prompt left, arrival order
        self.running: List[int] = []    # request ids decoding, prompt-completion order
        self.swapped: deque = deque()   # preempted request ids, preemption order
        self.moves: List[Move] = []
        self.pending: deque = deque()   # (step number, StepRows) formed and not committed
        self.async_mode = False
        self.seq = 0

    def set_async(self, on: bool) -> None:
        if on and self.pred != 0:
            raise SchedulerError("asynchronous formation needs every peak reserved")
        if self.pending:
            raise SchedulerError("commit the formed steps first")
        self.async_mode = bool(on)

    def _blocks(self, n_pos: int) -> int:
        return -(-n_pos // self.pool.block_size)

    def add(self, rid: int, prompt, max_new: int) -> None:
        prompt = [int(t) for t in prompt]
        if rid in self.req or rid < 0:
            raise SchedulerError("request id in use or negative")
        if not prompt or max_new < 1:
            raise SchedulerError("empty prompt or max_new_tokens < 1")
        if min(prompt) < 0:
            raise SchedulerError("negative prompt token id")
        if len(prompt) + max_new > self.mb * self.pool.block_size:
            raise SchedulerError("prompt + max_new_tokens beyond the block table")
        if self._blocks(len(prompt) + max_new - 1) > self.pool.num_blocks:
            raise SchedulerError("prompt + max_new_tokens beyond the pool")
        new = max_new if self.pred == 0 else min(max_new, self.pred)
        self.req[rid] = _Request(rid, prompt, max_new, self._blocks(len(prompt) + new - 1))
        self.prefill.append(rid)

    def _pos_next(self, rid: int) -> int:
        """Position of a running request's next row; its cached tokens are 0 .. this - 1."""
        r = self.req[rid]
        return len(r.prompt) + len(r.gen) + len(r.inflight) - 1

    def _decoding(self) -> List[int]:
        """The running requests that get a decode row: the first dense_tokens of those whose
        formed rows have not reached max_new_tokens."""
        out = [rid for rid in self.running
               if len(self.req[rid].gen) + len(self.req[rid].inflight) < self.req[rid].max_new]
        return out[:self.D]

    def _decode_need(self) -> int:
        bs = self.pool.block_size
        return sum(1 for rid in self._decoding() if self._pos_next(rid) % bs == 0)

    def next(self) -> StepRows:
        if len(self.pending) >= (2 if self.async_mode else 1):
            raise SchedulerError("commit the previous step first")
        bs = self.pool.block_size
        self.moves = []
        # preempt the latest-started running request while the decode rows lack blocks
        preempted = False
        while self._decode_need() > len(self.pool.free):
            r = self.req[self.running.pop()]
            self.moves.append(Move(0, r.rid, self._pos_next(r.rid), list(r.table)))
            self.pool.release(r.table)
            r.table = []
            self.swapped.append(r.rid)
            preempted = True
        # resume preempted requests, first in first out, while they fit
        while not preempted and self.swapped:
            r = self.req[self.swapped[0]]
            n = self._pos_next(r.rid)
            extra = 1 if (len(self.running) < self.D and n % bs == 0) else 0
            if len(self.pool.free) - self._decode_need() < self._blocks(n) + extra:
                break
            self.swapped.popleft()
            r.table = self.pool.alloc(self._blocks(n))
            self.moves.append(Move(1, r.rid, n, list(r.table)))
            self.running.append(r.rid)
        rows = []  # (rid, token, pos, samples)
        for rid in self._decoding():
            r = self.req[rid]
            p = self._pos_next(rid)
            if p % bs == 0:
                r.table.append(self.pool.alloc(1)[0])
            tok = -(r.inflight[-1][1] + 1) if r.inflight else r.gen[-1]
            rows.append((rid, tok, p, 1))
        room = self.D - len(rows)
        for rid in list(self.prefill):
            if room <= 0:
                break
            r = self.req[rid]
            if r.done == 0:
                # admission: the free blocks must cover this request's predicted peak, what the
                # admitted requests still need to reach theirs, and what the preempted ones need
                # to resume
                owed = sum(max(0, q.peak - len(q.table)) for q in self.req.values()
                           if q.table and not q.finished)
                owed += sum(self._blocks(self._pos_next(i) + 1) for i in self.swapped)
                if len(self.pool.free) < r.peak + owed:
                    break
            c = min(room, len(r.prompt) - r.done)
            c = min(c, (len(r.table) + len(self.pool.free)) * bs - r.done)
            if c <= 0:
                break
            new = self._blocks(r.done + c) - len(r.table)
            if new > 0:
                r.table.extend(self.pool.alloc(new))
            for k in range(c):
                p = r.done + k
                rows.append((rid, r.prompt[p], p, 1 if p == len(r.prompt) - 1 else 0))
            r.done += c
            room -= c
        B = len(rows)
        step = self.seq
        self.seq += 1
        for b, (rid, tok, p, smp) in enumerate(rows):
            if smp:
                r = self.req[rid]
                if p == len(r.prompt) - 1:  # the prompt completes: the request runs from now
                    self.prefill.remove(rid)
                    self.running.append(rid)
                r.inflight.append((step, b))
        tab = np.zeros((B, self.mb), dtype=np.int32)
        out = StepRows(np.zeros(B, np.int32), np.zeros(B, np.int32), tab, np.zeros(B, np.int32),
                       np.zeros(B, np.int64), np.zeros(B, np.int32), np.zeros(B, np.int32))
        for b, (rid, tok, p, smp) in enumerate(rows):
            t = self.req[rid].table
            out.token_ids[b], out.positions[b], out.seq_lens[b] = tok, p, p + 1
            tab[b, :len(t)] = t
            out.slot_mapping[b] = t[p // bs] * bs + p % bs
            out.row_request[b], out.row_samples[b] = rid, smp
        self.pending.append((step, out))
        return out

    def commit(self, sampled) -> List[int]:
        """Sampled token of every row of the oldest formed step (read where row_samples = 1);
        returns the ids that finished, in row order."""
        if not self.pending:
            raise SchedulerError("no step to commit")
        if len(sampled) != len(self.pending[0][1].token_ids):
            raise SchedulerError("batch differs from the formed step")
        step, st = self.pending.popleft()
        finished = []
        for b in range(len(st.token_ids)):
            if not st.row_samples[b]:
                continue
            r = self.req[int(st.row_request[b])]
            r.inflight.remove((step, b))
            if not r.finished:  # a row formed after the request's eos: its token is dropped
                tok = int(sampled[b])
                r.gen.append(tok)
                if tok == self.eos or len(r.gen) == r.max_new:
                    r.finished = True
                    self.running.remove(r.rid)
                    finished.append(r.rid)
            if r.finished and not r.inflight and r.table:
                self.pool.release(r.table)
                r.table = []
        return finished

    def tokens(self, rid: int) -> List[int]:
        return list(self.req[rid].gen)

    def remove(self, rid: int) -> None:
        """Forget a finished request."""
        if rid not in self.req or not self.req[rid].finished or self.req[rid].inflight:
            raise SchedulerError("unknown or unfinished request (or a formed row not committed)")
        del self.req[rid]

    def counts(self):
        """(requests with prompt left, running, preempted, finished and not removed)."""
        fin = sum(1 for r in self.req.values() if r.finished)
        return len(self.prefill), len(self.running), len(self.swapped), fin


__all__ = ["AllocatorError", "DenseBatchFormer", "Move", "SchedulerError", "StepRows"]
