"""fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / reference leg may import this package.  The
product path (the CUDA library and its Python binding) never imports it and
shares no code with it.

Every function here is the plain definition written out in float64 with full
materialisation of the score matrix, one (batch, head) slice at a time.  No
tiling, no online softmax, no fusion.  The sources followed are

* "Stanford CS336 Assignment 2 (Systems)" handout, section 4 "FlashAttention-2":
  Eq. 4-6 (forward), Eq. 7-11 (standard backward), Eq. 12 (logsumexp),
  Eq. 13-19 (recompute backward and D), causal masking in problem
  ``flash_forward`` part (c);
* "CS336 Assignment 2: Systems" (blog), FlashAttention-2 section: the causal
  mask keeps key index <= query index;
* "[Attention] FlashAttention/Ring-Attention/混合序列并行的统一原理", the
  two-half softmax and output merge formulas.

Pins (tests/test_oracle_pins.py) tie these functions to closed forms, a
hand-worked example, invariants, finite differences and brute force, so a
dropped term, a sign or an index error here fails a test.
"""
from .attention import (  # noqa: F401
    scores,
    causal_keep,
    attention_fwd,
    attention_fwd_rows,
    attention_bwd,
    attention_bwd_from_output,
    attention_bwd_query_rows,
    attention_bwd_key_rows,
    round_to_storage,
    rowsum_o_do,
    partial_attention,
    merge_two_halves,
)
