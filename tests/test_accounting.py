"""The bench's FLOP counter against the oracle's pinned pair counting.

Every TFLOP/s figure that bench.py prints is (4 + 10) * D * Hq * pairs over a
time, with `pairs` taken by ``bench.useful_pairs`` from the reconstruction
info arrays.  Here that function runs on the oracle's own reconstruction info
of every workload (padded and unpadded) and must equal
``oracle.attended_pairs`` exactly; that function is pinned against explicit
attention-mask counting in test_oracle_dedup.py.  The per-config totals are
also checked against the closed form of each configuration, worked by hand:
a group with prompt P and responses of lengths m_b attends
P(P+1)/2 + sum_b (m_b P + m_b (m_b + 1) / 2) pairs per head ("Split Attention
Optimization": prompt causal once, each response over the prompt and its own
causal prefix; "Performance Benchmarks", "Redundancy Analysis" for the worked
example's sizes).
"""

import numpy as np
import pytest

import bench
import oracle
from dummy_batch import WORKLOADS, make_batch, make_workload_batch


def _as_arrays(info):
    """The oracle's reconstruction info in the layout bench.useful_pairs reads
    (the GPU library's CSR grouping and per-group / per-sample lengths)."""
    groups = info.prompt_groups
    ptr = np.zeros(len(groups) + 1, dtype=np.int64)
    ptr[1:] = np.cumsum([len(g) for g in groups])
    members = np.array([b for g in groups for b in g], dtype=np.int64)
    return {"num_groups": len(groups), "group_ptr": ptr, "members": members,
            "prompt_len": np.asarray(info.prompt_len), "resp_len": np.asarray(info.resp_len)}


def _oracle_info(ids, mask, pos, R, use_unpad):
    groups, uniq = oracle.find_prompt_groups(ids, R, mask)
    if use_unpad and mask is None:
        mask = np.ones_like(ids, dtype=np.uint8)
    _, _, info = oracle.create_deduplicated_batch(ids, pos, R, groups, uniq, attention_mask=mask,
                                                  use_unpad=use_unpad)
    return info


def _oracle_pairs(info):
    return oracle.attended_pairs([int(info.prompt_len[g]) for g in range(info.G)],
                                 [[int(info.resp_len[b]) for b in grp] for grp in info.prompt_groups])


# hand-worked closed forms of the fixed-length configurations (pairs per head)
CLOSED_FORM = {
    # 2 x (128*129/2 + 2 (32*128 + 32*33/2))
    "tiny": 35_008,
    # 2 x (8192*8193/2 + 8 (512*8192 + 512*513/2))
    "qwen3_0p6b": 136_327_168,
    # 10240*10241/2 + 10 (1024*10240 + 1024*1025/2)
    "worked_example": 162_539_520,
    # 4 x (32768*32769/2 + 8 (2048*32768 + 2048*2049/2))
    "long_context": 4_362_174_464,
}


@pytest.mark.parametrize("wname", list(WORKLOADS))
@pytest.mark.parametrize("use_unpad", [False, True])
def test_bench_pairs_equal_oracle_pairs(wname, use_unpad):
    wl = WORKLOADS[wname]
    ids, mask, pos = make_workload_batch(wl, list(WORKLOADS).index(wname))
    info = _oracle_info(ids, mask, pos, wl.R, use_unpad)
    got = bench.useful_pairs(_as_arrays(info))
    assert got == _oracle_pairs(info)
    if wname in CLOSED_FORM:
        assert got == CLOSED_FORM[wname]
    if wl.resp_len_range is not None:
        # ragged responses: the count uses the valid lengths, not the padded width
        lens = [int(x) for x in info.resp_len]
        assert min(lens) >= wl.resp_len_range[0] and max(lens) <= wl.resp_len_range[1]
        assert got < oracle.attended_pairs([wl.P] * wl.G, [[wl.R] * wl.n] * wl.G)


@pytest.mark.parametrize("seed", [3, 4])
def test_bench_pairs_equal_oracle_key_sets(seed):
    """On small ragged, left-padded batches: the pair count equals the number of
    (query, key) entries of the oracle attention's own per-row key sets."""
    ids, mask, pos = make_batch(3, 3, 70, 40, 500, seed, resp_len_range=(1, 40), prompt_pad_range=(0, 20))
    for use_unpad in (False, True):
        info = _oracle_info(ids, mask, pos, 40, use_unpad)
        keysets = oracle.row_key_sets(info)
        entries = sum(len(keysets[t]) for t in range(info.T) if info.row_valid[t])
        assert bench.useful_pairs(_as_arrays(info)) == entries
