"""Plain fp64 CPU oracle for prompt deduplication and split attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library (``prompt_deduplicated_shared_gb300``) and never
imports it.

Every function follows the text of the two method pages it cites:

* "How Prompt Deduplication Works" (trybrowzer.com/help/snowflake-research/
  how-prompt-deduplication-works), sections "Finding Prompt Groups",
  "Creating Deduplicated Batch", "Reconstructing Original Batch",
  "Split Attention Optimization", "Working with Packed/Unpacked Sequences"
  and "Correctness & Gradients";
* "Performance Benchmarks" (trybrowzer.com/help/snowflake-research/
  performance-benchmarks), section "Redundancy Analysis".

The method is exact (split attention reproduces full causal attention on every
duplicated sequence), so the oracle reaches each result by the slow, plain
route: it duplicates every prompt and runs textbook causal attention on each
``[prompt ; response]`` sequence in float64, with the backward pass through the
explicit softmax Jacobian.

Pins (see ``tests/test_oracle_*.py``): the pages' worked redundancy example and
group example, brute force on tiny inputs, an independent packed-mask
formulation, closed forms (all-equal keys, a single key), reductions to a
library routine (torch's float64 causal attention, torch autograd), and central
finite differences.  No function here is "parity unpinned".
"""

from .dedup import (  # noqa: F401
    find_prompt_groups,
    create_deduplicated_batch,
    reconstruct_sequences,
    reconstruct_backward,
    pack_rows,
    pack_rows_backward,
    ReconstructionInfo,
)
from .attention import (  # noqa: F401
    split_attention_fwd,
    split_attention_bwd,
    split_attention_fwd_rows,
    split_attention_bwd_sparse,
    row_key_sets,
)
from .accounting import (  # noqa: F401
    token_counts,
    attended_pairs,
    batch_stats,
)
