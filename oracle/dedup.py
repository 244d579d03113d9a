"""Oracle: grouping, packing and reconstruction (plain Python/NumPy).

TEST INFRASTRUCTURE ONLY -- see the package docstring.

Citations are to "How Prompt Deduplication Works"
(trybrowzer.com/help/snowflake-research/how-prompt-deduplication-works).

Readings where the page is silent (each also listed in the design notes):

* Group order: groups are ordered by their smallest member index and members
  are ascending.  The page's example ``[[0, 1], [2, 3]]`` ("Finding Prompt
  Groups") is consistent with first-occurrence order, the plainest choice.
* With an attention mask the prompt key of a row also includes the mask over
  the prompt positions, so two rows whose prompt tokens agree but whose padding
  differs are different prompts.
* Packed position ids are copied from the source rows (prompt positions from
  the group's representative, response positions from the sample itself).
* ``use_unpad=True`` drops every position whose mask is 0 ("Working with
  Packed/Unpacked Sequences"; the page writes "unpacked" where the unpadded
  format is meant).
* Reconstruction fills every position that no packed row maps to with zeros.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class ReconstructionInfo:
    """Metadata to undo the pack ("Creating Deduplicated Batch": the returned
    reconstruction_info; "Working with Packed/Unpacked Sequences": the padding
    boundaries).  The field layout is ours; the page only calls it a dict of
    metadata.

    prompt_off[g]  packed row where group g's prompt slot starts
    prompt_slot[g] rows in that slot (P when padded, valid prompt tokens when
                   unpadded)
    prompt_len[g]  valid prompt tokens of the group's representative
    resp_off[b]    packed row where sample b's response slot starts
    resp_slot[b]   rows in that slot (R when padded, valid tokens when unpadded)
    resp_len[b]    valid response tokens of sample b
    group_of[b]    group index of sample b
    row_src[t]     (source sample, source position) of packed row t
    row_valid[t]   True where packed row t is a real (mask = 1) token
    """

    B: int
    L: int
    P: int
    use_unpad: bool
    prompt_groups: list
    prompt_off: np.ndarray
    prompt_slot: np.ndarray
    prompt_len: np.ndarray
    resp_off: np.ndarray
    resp_slot: np.ndarray
    resp_len: np.ndarray
    group_of: np.ndarray
    row_src: list = field(default_factory=list)
    row_valid: np.ndarray = None

    @property
    def T(self) -> int:
        return len(self.row_src)

    @property
    def G(self) -> int:
        return len(self.prompt_groups)


def find_prompt_groups(input_ids, response_length, attention_mask=None):
    """Group samples whose prompts are identical ("Finding Prompt Groups",
    "Phase 1: Prompt Detection & Deduplication").

    The prompt of row b is ``input_ids[b, :L - response_length]``.  Returns
    ``(prompt_groups, unique_prompts)``: a list of index lists and the
    ``[num_unique, prompt_len]`` array of each group's prompt tokens.
    """
    ids = np.asarray(input_ids)
    B, L = ids.shape
    P = L - int(response_length)
    if P < 0:
        raise ValueError("response_length exceeds the row length")
    mask = None if attention_mask is None else np.asarray(attention_mask)
    first_index_of_key = {}
    groups = []
    for b in range(B):
        key = tuple(int(x) for x in ids[b, :P])
        if mask is not None:
            key = key + tuple(int(x != 0) for x in mask[b, :P])
        if key not in first_index_of_key:
            first_index_of_key[key] = len(groups)
            groups.append([b])
        else:
            groups[first_index_of_key[key]].append(b)
    unique_prompts = np.stack([ids[grp[0], :P] for grp in groups]) if groups else \
        np.zeros((0, P), dtype=ids.dtype)
    return groups, unique_prompts


def _valid(mask, b, lo, hi):
    if mask is None:
        return list(range(lo, hi))
    return [p for p in range(lo, hi) if mask[b, p] != 0]


def create_deduplicated_batch(input_ids, position_ids, response_length,
                              prompt_groups, unique_prompts=None,
                              attention_mask=None, use_unpad=False):
    """Pack the batch into one sequence ``[1, T]`` laid out as
    ``[Prompt_1][Response_1_1][Response_1_2]...[Prompt_2][Response_2_1]...``
    ("Creating Deduplicated Batch", concatenation pattern).

    Returns ``(dedup_input_ids [1,T], dedup_position_ids [1,T],
    ReconstructionInfo)``.  ``position_ids=None`` stands for ``arange(L)`` on
    every row.
    """
    ids = np.asarray(input_ids)
    B, L = ids.shape
    R = int(response_length)
    P = L - R
    pos = np.tile(np.arange(L, dtype=np.int64), (B, 1)) if position_ids is None \
        else np.asarray(position_ids)
    mask = None if attention_mask is None else np.asarray(attention_mask)
    if use_unpad and mask is None:
        use_unpad = False  # nothing to drop without a mask

    G = len(prompt_groups)
    prompt_off = np.zeros(G, np.int64)
    prompt_slot = np.zeros(G, np.int64)
    prompt_len = np.zeros(G, np.int64)
    resp_off = np.zeros(B, np.int64)
    resp_slot = np.zeros(B, np.int64)
    resp_len = np.zeros(B, np.int64)
    group_of = np.full(B, -1, np.int64)
    row_src = []
    row_valid = []

    for g, members in enumerate(prompt_groups):
        rep = members[0]
        valid_p = _valid(mask, rep, 0, P)
        positions = valid_p if use_unpad else list(range(P))
        prompt_off[g] = len(row_src)
        prompt_slot[g] = len(positions)
        prompt_len[g] = len(valid_p)
        for p in positions:
            row_src.append((rep, p))
            row_valid.append(mask is None or mask[rep, p] != 0)
        for b in members:
            group_of[b] = g
            valid_r = _valid(mask, b, P, L)
            positions = valid_r if use_unpad else list(range(P, L))
            resp_off[b] = len(row_src)
            resp_slot[b] = len(positions)
            resp_len[b] = len(valid_r)
            for p in positions:
                row_src.append((b, p))
                row_valid.append(mask is None or mask[b, p] != 0)

    T = len(row_src)
    dedup_ids = np.zeros((1, T), dtype=ids.dtype)
    dedup_pos = np.zeros((1, T), dtype=pos.dtype)
    for t, (b, p) in enumerate(row_src):
        dedup_ids[0, t] = ids[b, p]
        dedup_pos[0, t] = pos[b, p]
    info = ReconstructionInfo(
        B=B, L=L, P=P, use_unpad=bool(use_unpad),
        prompt_groups=[list(m) for m in prompt_groups],
        prompt_off=prompt_off, prompt_slot=prompt_slot, prompt_len=prompt_len,
        resp_off=resp_off, resp_slot=resp_slot, resp_len=resp_len,
        group_of=group_of, row_src=row_src,
        row_valid=np.array(row_valid, dtype=bool))
    return dedup_ids, dedup_pos, info


def pack_rows(src, info: ReconstructionInfo):
    """Apply the pack's gather to any ``[B, L, ...]`` row tensor (hidden states,
    masks): packed row t takes ``src[row_src[t]]``."""
    src = np.asarray(src)
    out = np.zeros((info.T,) + src.shape[2:], dtype=src.dtype)
    for t, (b, p) in enumerate(info.row_src):
        out[t] = src[b, p]
    return out


def reconstruct_sequences(dedup_hidden, info: ReconstructionInfo):
    """Scatter the packed tensor back to ``[B, L, ...]`` ("Reconstructing
    Original Batch": for each output sample copy its unique prompt, then its
    response tokens).  Positions that no packed row maps to are zero."""
    x = np.asarray(dedup_hidden)
    if x.ndim >= 2 and x.shape[0] == 1 and x.shape[1] == info.T:
        x = x[0]
    out = np.zeros((info.B, info.L) + x.shape[1:], dtype=x.dtype)
    for g, members in enumerate(info.prompt_groups):
        lo = int(info.prompt_off[g])
        hi = lo + int(info.prompt_slot[g])
        for t in range(lo, hi):
            _, p = info.row_src[t]
            for b in members:
                out[b, p] = x[t]
    for b in range(info.B):
        lo = int(info.resp_off[b])
        hi = lo + int(info.resp_slot[b])
        for t in range(lo, hi):
            _, p = info.row_src[t]
            out[b, p] = x[t]
    return out


def reconstruct_backward(grad_out, info: ReconstructionInfo):
    """Adjoint of ``reconstruct_sequences`` ("Correctness & Gradients": the
    loss gradient of a shared prompt collects the contributions of every
    response of its group).  Packed row t receives the sum, over every output
    position that reconstruction copies it to, of the upstream gradient there:
    a group's prompt rows sum the gradients of all members' prompt copies, a
    response row takes its own sample's gradient.  Float64 result
    ``[T, ...]``; positions that reconstruction zero-fills contribute
    nothing."""
    g = np.asarray(grad_out, dtype=np.float64)
    out = np.zeros((info.T,) + g.shape[2:], dtype=np.float64)
    for gi, members in enumerate(info.prompt_groups):
        lo = int(info.prompt_off[gi])
        hi = lo + int(info.prompt_slot[gi])
        for t in range(lo, hi):
            _, p = info.row_src[t]
            for b in members:
                out[t] += g[b, p]
    for b in range(info.B):
        lo = int(info.resp_off[b])
        hi = lo + int(info.resp_slot[b])
        for t in range(lo, hi):
            _, p = info.row_src[t]
            out[t] += g[b, p]
    return out


def pack_rows_backward(grad_packed, info: ReconstructionInfo):
    """Adjoint of ``pack_rows`` ("Correctness & Gradients": gradients flow back
    through the deduplication step as well as the reconstruction).  Packed row
    t was read from source position ``row_src[t]``, so that position receives
    ``grad_packed[t]``; every source position is read at most once, so there
    is nothing to sum.  Positions the pack never read (the prompt rows of every
    group member but the representative, and the pads that ``use_unpad``
    dropped) receive zero.  Returns ``[B, L, ...]`` in the input's dtype."""
    g = np.asarray(grad_packed)
    if g.ndim >= 2 and g.shape[0] == 1 and g.shape[1] == info.T:
        g = g[0]
    out = np.zeros((info.B, info.L) + g.shape[1:], dtype=g.dtype)
    for t, (b, p) in enumerate(info.row_src):
        out[b, p] = g[t]
    return out

