"""CPU oracle for one continuous-batching decode step over a paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, links or runs this package:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg and
``--impl reference`` arm use it.  It shares no code with the CUDA library (no kernels,
headers, helpers, tables or constant generators); the only common module is ``synth``,
which draws the seeded inputs and contains none of the step's arithmetic.

Everything here is plain numpy in fp64 on inputs widened exactly from their fp16/bf16
storage.  Each function states the passage of the source pages it follows.  The step is the
plain definition of a pre-norm decoder layer stack; fusion, paging, grouped-query sharing,
split-K, nano-batching and graph replay on the GPU side are exact re-orderings of it.

Parity status: every function below is pinned by a ``-m "not gpu"`` test against something
other than itself (closed forms, special cases that reduce to library routines, brute force,
invariants, or numbers printed on the pages).  The pages print no logits for any input, so
``decode_step`` as a whole is pinned by closed forms instead (zero Wo/Wd: the tied head scores
the input token; zero Wq: every head averages its kv head's V), by invariants (rows are
independent; a prompt chunk equals its tokens decoded one step at a time, causally) and by
an independent PyTorch statement over dense histories (``tests/test_oracle_pins.py``).
"""
from .decode import (  # noqa: F401
    OracleModel, attention_weights, dense_attention, decode_step, from_storage, gqa_group,
    greedy_argmax, paged_attention, param_bytes, rms_norm, rope_apply, rope_tables,
    round_storage, silu, slot_of, softmax, swiglu,
)
from .kvcache import BlockAllocator, kv_rows, kv_scatter, request_slots  # noqa: F401
