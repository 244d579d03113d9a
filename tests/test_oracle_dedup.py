"""Pins for the oracle's grouping, packing and reconstruction (CPU only)."""

import itertools
import json
import os

import numpy as np
import pytest

import oracle
from oracle import accounting
from oracle.dedup import pack_rows
from dummy_batch import make_batch, WORKLOADS

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _brute_force_groups(ids, P, mask=None):
    """Pairwise row comparison + first-occurrence classes (independent of the
    oracle's dictionary of keys)."""
    B = ids.shape[0]
    rep = list(range(B))
    for b in range(B):
        for a in range(b):
            same = np.array_equal(ids[a, :P], ids[b, :P])
            if mask is not None:
                same = same and np.array_equal(mask[a, :P] != 0, mask[b, :P] != 0)
            if same:
                rep[b] = rep[a]
                break
    order = sorted(set(rep))
    return [[b for b in range(B) if rep[b] == r] for r in order]


def test_group_example_from_page():
    gold = _load("group_example.json")
    rng = np.random.default_rng(0)
    P, R = 16, 4
    pa, pb = rng.integers(0, 100, P), rng.integers(100, 200, P)
    ids = np.stack([np.concatenate([p, rng.integers(0, 100, R)]) for p in (pa, pa, pb, pb)])
    groups, uniq = oracle.find_prompt_groups(ids, R)
    assert groups == gold["prompt_groups"]
    assert uniq.shape == (gold["num_unique"], P)
    assert np.array_equal(uniq[0], pa) and np.array_equal(uniq[1], pb)


@pytest.mark.parametrize("seed", range(6))
def test_groups_brute_force(seed):
    rng = np.random.default_rng(seed)
    G, n, P, R = 1 + seed % 4, 1 + (seed * 7) % 5, 8 + seed, 3
    ids, mask, _ = make_batch(G, n, P, R, 5 if seed % 2 else 1000, seed)
    groups, uniq = oracle.find_prompt_groups(ids, R)
    assert groups == _brute_force_groups(ids, P)
    for g, members in enumerate(groups):
        for b in members:
            assert np.array_equal(ids[b, :P], uniq[g])
    # permutation equivariance: relabelled rows give relabelled classes
    perm = rng.permutation(ids.shape[0])
    g2, _ = oracle.find_prompt_groups(ids[perm], R)
    as_sets = sorted(sorted(int(perm[i]) for i in grp) for grp in g2)
    assert as_sets == sorted(sorted(grp) for grp in groups)


def test_groups_mask_is_part_of_key():
    ids = np.array([[5, 6, 7, 1], [5, 6, 7, 2], [5, 6, 7, 3]])
    mask = np.array([[1, 1, 1, 1], [0, 1, 1, 1], [1, 1, 1, 1]])
    groups, _ = oracle.find_prompt_groups(ids, 1, mask)
    assert groups == [[0, 2], [1]]
    assert groups == _brute_force_groups(ids, 3, mask)


def test_packing_pattern_from_page():
    gold = _load("packing_pattern.json")
    P, R = 3, 2
    tok = {"A": [1, 1, 1], "B": [2, 2, 2], "R1": [11, 11], "R2": [12, 12],
           "R3": [13, 13], "R4": [14, 14]}
    ids = np.array([tok[p] + tok[r] for p, r in gold["rows"]])
    groups, uniq = oracle.find_prompt_groups(ids, R)
    dids, dpos, info = oracle.create_deduplicated_batch(ids, None, R, groups, uniq)
    expect = sum((tok[x] for x in gold["packed"]), [])
    assert dids.tolist() == [expect]
    assert dpos.tolist() == [[0, 1, 2, 3, 4, 3, 4, 0, 1, 2, 3, 4, 3, 4]]
    assert info.prompt_off.tolist() == [0, 7]
    assert info.resp_off.tolist() == [3, 5, 10, 12]


def test_worked_example_counts():
    gold = _load("worked_example.json")
    K = gold["K_tokens"]
    P, n, R = gold["prompt_len"], gold["num_responses"], gold["response_len"]
    ids, _, _ = make_batch(1, n, P, R, 151936, 7)
    groups, uniq = oracle.find_prompt_groups(ids, R)
    assert len(groups) == 1 and len(groups[0]) == n
    dids, _, info = oracle.create_deduplicated_batch(ids, None, R, groups, uniq)
    total = ids.size
    unique = dids.shape[1]
    assert total == gold["total_tokens_K"] * K
    assert unique == gold["unique_tokens_K"] * K
    assert round(100 * (1 - unique / total)) == gold["redundancy_percent_rounded"]
    t, u, red = accounting.token_counts([P], [[R] * n])
    assert (t, u) == (total, unique) and abs(red - (1 - unique / total)) < 1e-15


@pytest.mark.parametrize("use_unpad", [False, True])
@pytest.mark.parametrize("prompt_pad", [None, (0, 5)])
def test_reconstruct_inverts_pack(use_unpad, prompt_pad):
    ids, mask, pos = make_batch(3, 3, 12, 6, 50, 11, resp_len_range=(1, 6),
                                prompt_pad_range=prompt_pad)
    R = 6
    groups, uniq = oracle.find_prompt_groups(ids, R, mask)
    dids, dpos, info = oracle.create_deduplicated_batch(
        ids, pos, R, groups, uniq, attention_mask=mask, use_unpad=use_unpad)
    back = oracle.reconstruct_sequences(dids[0][:, None], info)[..., 0]
    valid = mask != 0
    assert np.array_equal(back[valid], ids[valid])
    if use_unpad:
        assert np.all(back[~valid] == 0)
        assert info.T == int(mask.sum()) - sum(
            int(mask[m[0], :12].sum()) * (len(m) - 1) for m in groups)
    else:
        assert np.array_equal(back, ids)  # padded: every position round-trips
        assert info.T == len(groups) * 12 + ids.shape[0] * R
    # positions are copied from the source rows
    back_pos = oracle.reconstruct_sequences(dpos[0][:, None], info)[..., 0]
    assert np.array_equal(back_pos[valid], pos[valid])
    # any row tensor packs with the same gather; prompt positions of every
    # member come back from the group's representative (first member)
    hidden = np.arange(ids.size * 2, dtype=np.float32).reshape(ids.shape + (2,))
    ph = pack_rows(hidden, info)
    hb = oracle.reconstruct_sequences(ph, info)
    expect = hidden.copy()
    for members in groups:
        expect[members, :12] = hidden[members[0], :12]
    assert np.array_equal(hb[valid], expect[valid])


def test_pack_lengths_all_configs():
    for name, wl in WORKLOADS.items():
        if wl.resp_len_range is not None:
            continue
        T = wl.G * wl.P + wl.B * wl.R
        t, u, _ = accounting.token_counts([wl.P] * wl.G, [[wl.R] * wl.n] * wl.G)
        assert u == T and t == wl.B * wl.L, name


def test_pairs_brute_force():
    """attended_pairs against counting the entries of explicit attention masks."""
    for P, lens in [(5, [3, 0, 2]), (0, [4, 1]), (7, []), (3, [1])]:
        split = P * (P + 1) // 2  # prompt causal block, counted entry by entry below
        count = sum(1 for i in range(P) for j in range(P) if j <= i)
        assert count == split
        for m in lens:
            count += sum(1 for i in range(m) for j in range(P + m) if j < P or j - P <= i)
        assert accounting.attended_pairs([P], [lens]) == count
        dup = sum(sum(1 for i in range(P + m) for j in range(P + m) if j <= i) for m in lens)
        assert accounting.attended_pairs([P], [lens], duplicated=True) == dup


_ADJ_CASES = [
    # G, n, P, R, resp_len_range, prompt_pad_range, use_unpad
    (3, 3, 12, 6, (1, 6), None, False),
    (3, 3, 12, 6, (1, 6), (0, 5), True),
    (2, 4, 9, 5, None, None, False),
    (1, 5, 0, 7, (0, 7), None, True),   # no prompt
    (4, 2, 11, 0, None, None, False),   # no response
]


@pytest.mark.parametrize("case", _ADJ_CASES)
def test_reconstruct_backward_is_the_adjoint(case):
    """<reconstruct(x), y> = <x, reconstruct_backward(y)> for random x, y: the
    defining property of the adjoint, checked against the oracle's own
    reconstruction (itself pinned by reconstruct∘pack = identity)."""
    G, n, P, R, rlr, ppr, unpad = case
    ids, mask, pos = make_batch(G, n, P, R, 30, 17, resp_len_range=rlr, prompt_pad_range=ppr)
    if unpad and mask is None:
        mask = np.ones_like(ids, dtype=np.uint8)
    groups, uniq = oracle.find_prompt_groups(ids, R, mask)
    _, _, info = oracle.create_deduplicated_batch(ids, pos, R, groups, uniq, attention_mask=mask,
                                                  use_unpad=unpad)
    rng = np.random.default_rng(5)
    x = rng.standard_normal((info.T, 3))
    y = rng.standard_normal((ids.shape[0], ids.shape[1], 3))
    lhs = float(np.sum(oracle.reconstruct_sequences(x, info) * y))
    rhs = float(np.sum(x * oracle.reconstruct_backward(y, info)))
    assert abs(lhs - rhs) <= 1e-12 * (np.abs(x).sum() * np.abs(y).max() + 1.0)


def test_reconstruct_backward_special_cases():
    # all prompts distinct, padded layout: nothing is shared, so the adjoint is
    # the plain gather of the packed rows (pack_rows)
    ids, mask, pos = make_batch(5, 1, 8, 4, 1000, 3)
    groups, uniq = oracle.find_prompt_groups(ids, 4, mask)
    assert all(len(m) == 1 for m in groups)
    _, _, info = oracle.create_deduplicated_batch(ids, pos, 4, groups, uniq)
    y = np.random.default_rng(6).standard_normal(ids.shape + (2,))
    assert np.array_equal(oracle.reconstruct_backward(y, info), pack_rows(y, info))
    # one group of n members with equal upstream gradients: each prompt row
    # collects n times the gradient, each response row exactly its own
    n = 4
    ids, mask, pos = make_batch(1, n, 6, 3, 50, 4)
    groups, uniq = oracle.find_prompt_groups(ids, 3, mask)
    _, _, info = oracle.create_deduplicated_batch(ids, pos, 3, groups, uniq)
    y = np.ones(ids.shape + (1,))
    gp = oracle.reconstruct_backward(y, info)[:, 0]
    assert np.array_equal(gp[:6], np.full(6, float(n)))
    assert np.array_equal(gp[6:], np.ones(n * 3))


@pytest.mark.parametrize("case", _ADJ_CASES)
def test_pack_rows_backward_is_the_adjoint(case):
    """<pack(x), y> = <x, pack_backward(y)> for random x, y (the defining
    property of the adjoint), against the oracle's pack_rows, itself pinned by
    reconstruct∘pack = identity and the page's packing diagram."""
    G, n, P, R, rlr, ppr, unpad = case
    ids, mask, pos = make_batch(G, n, P, R, 30, 19, resp_len_range=rlr, prompt_pad_range=ppr)
    if unpad and mask is None:
        mask = np.ones_like(ids, dtype=np.uint8)
    groups, uniq = oracle.find_prompt_groups(ids, R, mask)
    _, _, info = oracle.create_deduplicated_batch(ids, pos, R, groups, uniq, attention_mask=mask,
                                                  use_unpad=unpad)
    rng = np.random.default_rng(8)
    x = rng.standard_normal((ids.shape[0], ids.shape[1], 3))
    y = rng.standard_normal((info.T, 3))
    lhs = float(np.sum(pack_rows(x, info) * y))
    rhs = float(np.sum(x * oracle.pack_rows_backward(y, info)))
    assert abs(lhs - rhs) <= 1e-12 * (np.abs(x).max() * np.abs(y).sum() + 1.0)


def test_pack_rows_backward_special_cases():
    """The pack reads every source position at most once, so its adjoint is a
    scatter: packing a tensor and mapping it back keeps exactly the positions
    the pack read -- the representative's whole row, and of every other member
    only the response -- and zeroes the rest (other members' prompts, pads
    dropped by use_unpad).  With all prompts distinct and no padding dropped it
    is the identity."""
    ids, mask, pos = make_batch(2, 3, 7, 4, 50, 21, resp_len_range=(1, 4))
    groups, uniq = oracle.find_prompt_groups(ids, 4, mask)
    x = np.random.default_rng(9).standard_normal(ids.shape + (2,))
    for unpad in (False, True):
        _, _, info = oracle.create_deduplicated_batch(ids, pos, 4, groups, uniq, attention_mask=mask,
                                                      use_unpad=unpad)
        back = oracle.pack_rows_backward(pack_rows(x, info), info)
        for g in groups:
            rep, others = g[0], g[1:]
            keep = np.ones(ids.shape[1], bool) if not unpad else mask[rep] != 0
            assert np.array_equal(back[rep][keep], x[rep][keep])
            assert not back[rep][~keep].any()
            for b in others:
                assert not back[b, :7].any()
                keep_r = np.ones(4, bool) if not unpad else mask[b, 7:] != 0
                assert np.array_equal(back[b, 7:][keep_r], x[b, 7:][keep_r])
                assert not back[b, 7:][~keep_r].any()
    ids, mask, pos = make_batch(5, 1, 8, 4, 1000, 3)
    groups, uniq = oracle.find_prompt_groups(ids, 4, mask)
    _, _, info = oracle.create_deduplicated_batch(ids, pos, 4, groups, uniq)
    x = np.random.default_rng(10).standard_normal(ids.shape + (2,))
    assert np.array_equal(oracle.pack_rows_backward(pack_rows(x, info), info), x)


def test_batch_stats_closed_form():
    """A batch built with known lengths: 3 rows, L = 10, response_length 4.
    Prompts hold 6, 4 and 6 valid tokens (left padded); responses 4, 0 and 2
    (right padded).  Every statistic follows by hand."""
    mask = np.zeros((3, 10), dtype=np.uint8)
    mask[0, 0:6] = 1; mask[0, 6:10] = 1
    mask[1, 2:6] = 1
    mask[2, 0:6] = 1; mask[2, 6:8] = 1
    st = accounting.batch_stats(mask, 4)
    assert (st["prompt_len_min"], st["prompt_len_max"]) == (4, 6)
    assert abs(st["prompt_len_mean"] - 16 / 3) < 1e-15
    assert (st["responses"], st["resp_len_min"], st["resp_len_max"]) == (2, 2, 4)
    assert st["resp_len_mean"] == 3.0
    assert (st["non_pad_tokens"], st["total_positions"]) == (22, 30)
    assert abs(st["non_pad_fraction"] - 22 / 30) < 1e-15


def test_batch_stats_against_generator():
    """make_batch draws the response lengths itself: the statistics must
    recover exactly what the generator reports back through the mask."""
    ids, mask, pos = make_batch(4, 5, 30, 12, 100, 9, resp_len_range=(3, 12), prompt_pad_range=(0, 7))
    st = accounting.batch_stats(mask, 12)
    rl = [int(r.sum()) for r in (mask[:, 30:] != 0)]
    pl = [int(r.sum()) for r in (mask[:, :30] != 0)]
    assert st["responses"] == 20 and st["resp_len_min"] == min(rl) and st["resp_len_max"] == max(rl)
    assert st["non_pad_tokens"] == sum(rl) + sum(pl) == int((mask != 0).sum())
