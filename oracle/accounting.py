"""Oracle: token, attended-pair, FLOP and byte accounting.

TEST INFRASTRUCTURE ONLY -- see the package docstring.

"Performance Benchmarks", "Redundancy Analysis" and "How Prompt Deduplication
Works", "Impact on Computation": a 10K-token prompt with 10 responses of 1K
tokens is 110K tokens in the batch but only 20K unique tokens, so 82% of the
work is repeated prompt work.  The page mixes K = 1000 ("10K x 10 + 1K x 10 =
110K") with the 1024-token sizes of the worked configuration; with K = 1024 the
exact figures are 112,640 and 20,480 tokens and a redundancy of 1 - 2/11.
"""

from __future__ import annotations

import numpy as np


def token_counts(prompt_lens, resp_lens_per_group):
    """Tokens of the duplicated batch and of the deduplicated packing.

    ``prompt_lens[g]`` is group g's prompt length, ``resp_lens_per_group[g]``
    the list of its members' response lengths.  Returns
    ``(total, unique, redundancy)`` with redundancy = 1 - unique/total."""
    total = 0
    unique = 0
    for P, lens in zip(prompt_lens, resp_lens_per_group):
        total += sum(P + n for n in lens)
        unique += P + sum(lens)
    return total, unique, (1.0 - unique / total) if total else 0.0


def attended_pairs(prompt_lens, resp_lens_per_group, duplicated=False):
    """Number of (query, key) pairs one head attends.  Causal attention over a
    sequence of n tokens attends n(n+1)/2 pairs.  Split attention: the prompt
    once (P(P+1)/2) plus, per response of length m, m*P prompt pairs and
    m(m+1)/2 response pairs.  ``duplicated=True`` counts the baseline that runs
    full causal attention on every [prompt ; response] sequence."""
    pairs = 0
    for P, lens in zip(prompt_lens, resp_lens_per_group):
        if duplicated:
            pairs += sum((P + m) * (P + m + 1) // 2 for m in lens)
        else:
            pairs += P * (P + 1) // 2 + sum(m * P + m * (m + 1) // 2 for m in lens)
    return pairs


def batch_stats(attention_mask, response_length):
    """Statistics of a normal (not deduplicated) batch from its attention mask
    ("Debugging & Analysis", "Batch Statistics": prompt length, response count
    with min/mean/max length, non-pad tokens and their share).  Reading: the
    prompt of row b is its first L - response_length positions, its response
    the rest; a row counts as a response when it holds at least one response
    token, and the response min/mean/max run over those rows.  Returns a dict
    of plain Python numbers."""
    m = np.asarray(attention_mask) != 0
    B, L = m.shape
    P = L - response_length
    plen = [int(m[b, :P].sum()) for b in range(B)]
    rlen = [int(m[b, P:].sum()) for b in range(B)]
    resp = [x for x in rlen if x > 0]
    non_pad = sum(plen) + sum(rlen)
    return {
        "rows": B,
        "prompt_len_min": min(plen) if B else 0,
        "prompt_len_max": max(plen) if B else 0,
        "prompt_len_mean": (sum(plen) / B) if B else 0.0,
        "responses": len(resp),
        "resp_len_min": min(resp) if resp else 0,
        "resp_len_max": max(resp) if resp else 0,
        "resp_len_mean": (sum(resp) / len(resp)) if resp else 0.0,
        "non_pad_tokens": non_pad,
        "total_positions": B * L,
        "non_pad_fraction": (non_pad / (B * L)) if B * L else 0.0,
    }
