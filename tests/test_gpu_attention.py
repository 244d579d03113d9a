"""GPU parity of split attention (forward and backward) against the fp64
oracle.  Tolerances (outputs, LSE and all three gradients): fp32 max-abs 1e-3;
bf16 max-abs 2e-2 plus 2^-8 of the reference's magnitude, the rounding of the
bf16 output format itself (see gpu_util).

* dense parity on small and reduced shapes (every output element);
* full-size workloads: sampled query rows for the forward, and a sparse
  upstream gradient (dO = 0 outside a sampled row set) for the backward, where
  the oracle's exact gradients cost one row of attention per sampled row.
"""

import numpy as np
import pytest
import torch

import oracle
from dummy_batch import make_batch, WORKLOADS, make_workload_batch
from gpu_util import lib, oracle_pack, gpu_pack, qkv_inputs, max_abs, tol, DEV

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zr():
    return lib()


def _tc_expected(dtype, D):
    """bf16 attention runs on the tensor-core kernels for every GQA ratio
    (head_dim 64 or 128); float32 runs on the SIMT kernels."""
    return dtype == torch.bfloat16 and D in (64, 128)


def _run(zr, info, tq, tk, tv, tdo, backward=True):
    """Forward (and backward) through the C ABI; any error status fails the
    test.  The per-kernel event records show which kernels ran: the
    tensor-core forward and backward for bf16, none of them for float32."""
    zr.kernel_time_reset()
    zr.set_option("kernel_timing", 1)
    try:
        o, lse = zr.split_attn_fwd(info, tq, tk, tv)
        grads = zr.split_attn_bwd(info, tq, tk, tv, o, lse, tdo) if backward else None
        torch.cuda.synchronize()
        zr.check_status(info)
        launched = {n: zr.kernel_time(n)[1] for n in ("attn_fwd", "attn_bwd")}
    finally:
        zr.set_option("kernel_timing", 0)
        zr.kernel_time_reset()
    tc = _tc_expected(tq.dtype, tq.shape[2])
    assert launched["attn_fwd"] == (1 if tc else 0), launched
    assert launched["attn_bwd"] == (1 if tc and backward else 0), launched
    return o, lse, grads


DENSE = [
    # name, G, n, P, R, Hq, Hkv, D, dtype, resp_len_range, prompt_pad, use_unpad
    ("tiny-fp32", 2, 2, 128, 32, 2, 1, 64, torch.float32, None, None, False),
    ("fp32-ragged", 2, 3, 150, 70, 4, 2, 32, torch.float32, (1, 70), None, False),
    ("bf16-d128", 2, 3, 300, 140, 4, 2, 128, torch.bfloat16, None, None, False),
    ("bf16-d64-mha", 3, 2, 129, 257, 2, 2, 64, torch.bfloat16, (1, 257), None, False),
    ("bf16-d128-mha", 2, 2, 200, 130, 4, 4, 128, torch.bfloat16, (5, 130), None, False),
    ("bf16-d128-ratio3", 2, 2, 250, 100, 6, 2, 128, torch.bfloat16, (1, 100), None, False),
    ("bf16-d64-odd-heads", 2, 2, 140, 90, 5, 5, 64, torch.bfloat16, (1, 90), None, False),
    ("bf16-d128-ratio3-odd", 1, 3, 170, 60, 3, 1, 128, torch.bfloat16, (1, 60), None, False),
    ("bf16-unpad", 2, 4, 200, 100, 4, 2, 128, torch.bfloat16, (3, 100), None, True),
    ("bf16-leftpad", 2, 2, 190, 60, 4, 1, 128, torch.bfloat16, (1, 60), (1, 70), False),
    ("bf16-leftpad-unpad", 2, 2, 190, 60, 8, 2, 64, torch.bfloat16, (1, 60), (1, 70), True),
    ("bf16-no-prompt", 1, 3, 0, 200, 2, 1, 128, torch.bfloat16, None, None, False),
    ("bf16-no-response", 2, 1, 333, 0, 2, 1, 128, torch.bfloat16, None, None, False),
    ("bf16-d128-ratio4", 2, 2, 260, 120, 8, 2, 128, torch.bfloat16, (1, 120), None, False),
    ("bf16-d64-ratio8", 2, 2, 300, 90, 8, 1, 64, torch.bfloat16, (1, 90), None, False),
    ("bf16-many-groups-unpad", 5, 3, 100, 40, 4, 2, 128, torch.bfloat16, (1, 40), None, True),
    ("bf16-long-prompt", 1, 2, 700, 150, 2, 1, 128, torch.bfloat16, (1, 150), None, False),
]


@pytest.mark.parametrize("case", DENSE, ids=[c[0] for c in DENSE])
def test_dense_parity(zr, case):
    name, G, n, P, R, Hq, Hkv, D, dtype, rlr, ppr, unpad = case
    ids, mask, pos = make_batch(G, n, P, R, 1000, 77, resp_len_range=rlr, prompt_pad_range=ppr)
    if unpad and mask is None:
        mask = np.ones_like(ids, dtype=np.uint8)
    _, _, _, _, info_ref = oracle_pack(ids, mask, pos, R, unpad)
    _, _, _, _, info, T = gpu_pack(zr, ids, mask, pos, R, unpad, T_cap=max(info_ref.T, 1))
    (q, k, v, do), (tq, tk, tv, tdo) = qkv_inputs(T, Hq, Hkv, D, 5, dtype)
    o_ref, lse_ref = oracle.split_attention_fwd(q, k, v, info_ref)
    dq_ref, dk_ref, dv_ref = oracle.split_attention_bwd(q, k, v, do, info_ref)
    o, lse, (dq, dk, dv) = _run(zr, info, tq, tk, tv, tdo)
    t = tol(dtype)
    assert max_abs(o, o_ref) < t, "o"
    assert max_abs(lse, lse_ref.T) < t, "lse"
    assert max_abs(dq, dq_ref) < t, "dq"
    assert max_abs(dk, dk_ref) < t, "dk"
    assert max_abs(dv, dv_ref) < t, "dv"


def test_reduced_qwen_structure(zr):
    """16/8 heads, head_dim 128, prompt 2048, responses 256, 4 per group, 2
    groups: every element against the dense oracle."""
    ids, mask, pos = make_batch(2, 4, 2048, 256, 151936, 21)
    _, _, _, _, info_ref = oracle_pack(ids, mask, pos, 256, False)
    _, _, _, _, info, T = gpu_pack(zr, ids, mask, pos, 256, False, T_cap=info_ref.T)
    (q, k, v, do), (tq, tk, tv, tdo) = qkv_inputs(T, 16, 8, 128, 22, torch.bfloat16)
    o_ref, lse_ref = oracle.split_attention_fwd(q, k, v, info_ref)
    dq_ref, dk_ref, dv_ref = oracle.split_attention_bwd(q, k, v, do, info_ref)
    o, lse, (dq, dk, dv) = _run(zr, info, tq, tk, tv, tdo)
    assert max_abs(o, o_ref) < 2e-2
    assert max_abs(lse, lse_ref.T) < 2e-2
    assert max_abs(dq, dq_ref) < 2e-2
    assert max_abs(dk, dk_ref) < 2e-2
    assert max_abs(dv, dv_ref) < 2e-2


def _sample_rows(info, per_segment, rng):
    rows = []
    segs = [(int(info.prompt_off[g]), int(info.prompt_slot[g])) for g in range(info.G)]
    segs += [(int(info.resp_off[b]), int(info.resp_slot[b])) for b in range(info.B)]
    for lo, n in segs:
        if n == 0:
            continue
        pick = {lo, lo + n - 1}
        pick.update(int(x) for x in rng.integers(lo, lo + n, size=per_segment))
        rows.extend(sorted(pick))
    return sorted(set(t for t in rows if info.row_valid[t]))


# (workload, use_unpad, heads): heads overrides (Hq, Hkv, D) of the workload to
# run the same batch through another kernel configuration (head_dim 64, GQA 4)
FULL = [("qwen3_0p6b", False, None), ("worked_example", False, None), ("pipeline", False, None),
        ("pipeline", True, None), ("pipeline_nodedup", False, None), ("long_context", False, None),
        ("worked_example", False, (16, 4, 64))]


def _full_id(c):
    w, u, hd = c
    return f"{w}-{'unpad' if u else 'pad'}" + ("" if hd is None else f"-h{hd[0]}-{hd[1]}-d{hd[2]}")


@pytest.mark.parametrize("wname,use_unpad,heads", FULL, ids=[_full_id(c) for c in FULL])
def test_full_size_sampled(zr, wname, use_unpad, heads):
    """Every configuration at full size, in the launch configuration the bench
    uses: the forward on sampled query rows of every prompt and response, the
    backward with the upstream gradient zero outside a sampled row set (the
    exact gradients then need one row of attention per sampled row)."""
    wl = WORKLOADS[wname]
    idx = list(WORKLOADS).index(wname)
    ids, mask, pos = make_workload_batch(wl, idx)
    _, _, _, _, info_ref = oracle_pack(ids, mask, pos, wl.R, use_unpad)
    _, _, _, _, info, T = gpu_pack(zr, ids, mask, pos, wl.R, use_unpad, T_cap=info_ref.T)
    assert T == info_ref.T
    Hq, Hkv, D = heads if heads is not None else (wl.Hq, wl.Hkv, wl.D)
    (q, k, v, do), (tq, tk, tv, tdo) = qkv_inputs(T, Hq, Hkv, D, 100 + idx, torch.bfloat16)
    rng = np.random.default_rng(idx + (50 if use_unpad else 0))
    per = 2 if wname in ("long_context", "pipeline_nodedup") else 6
    rows = _sample_rows(info_ref, per, rng)
    keysets = oracle.row_key_sets(info_ref)
    o_ref, lse_ref = oracle.split_attention_fwd_rows(q, k, v, info_ref, rows, key_sets=keysets)
    sparse_do = np.zeros_like(do)
    bwd_rows = rows[::3] if wname in ("long_context", "pipeline_nodedup") else rows
    sparse_do[bwd_rows] = do[bwd_rows]
    tdo_sparse = torch.from_numpy(sparse_do).to(DEV, torch.bfloat16)
    want_bwd = wl.backward
    if want_bwd:
        dq_ref, dk_ref, dv_ref = oracle.split_attention_bwd_sparse(q, k, v, sparse_do, info_ref,
                                                                   bwd_rows, key_sets=keysets)
    o, lse, grads = _run(zr, info, tq, tk, tv, tdo_sparse, backward=want_bwd)
    assert max_abs(o[rows], o_ref) < 2e-2, "o"
    assert max_abs(lse[rows], lse_ref.T) < 2e-2, "lse"
    if want_bwd:
        dq, dk, dv = grads
        assert max_abs(dq, dq_ref) < 2e-2, "dq"
        assert max_abs(dk, dk_ref) < 2e-2, "dk"
        assert max_abs(dv, dv_ref) < 2e-2, "dv"


def test_kernel_timing_counts_launches_and_changes_nothing(zr):
    """The "kernel_timing" option brackets each tensor-core launch with events:
    one pair per launch under the kernel's name, outputs bit-identical."""
    ids, mask, pos = make_batch(2, 3, 300, 140, 1000, 78)
    _, _, _, _, info_ref = oracle_pack(ids, mask, pos, 140, False)
    _, _, _, _, info, T = gpu_pack(zr, ids, mask, pos, 140, False, T_cap=info_ref.T)
    _, (tq, tk, tv, tdo) = qkv_inputs(T, 4, 2, 128, 6, torch.bfloat16)

    def plain_run():
        o, lse = zr.split_attn_fwd(info, tq, tk, tv)
        grads = zr.split_attn_bwd(info, tq, tk, tv, o, lse, tdo)
        torch.cuda.synchronize()
        zr.check_status(info)
        return o, lse, grads

    plain = plain_run()
    zr.kernel_time_reset()
    zr.set_option("kernel_timing", 1)
    try:
        timed = plain_run()
        times = {n: zr.kernel_time(n) for n in ("attn_fwd", "attn_bwd_prep", "attn_bwd", "attn_dq_convert")}
    finally:
        zr.set_option("kernel_timing", 0)
        zr.kernel_time_reset()
    for n, (ms, count) in times.items():
        assert count == 1 and ms > 0.0, (n, ms, count)
    assert torch.equal(plain[0], timed[0]) and torch.equal(plain[1], timed[1])
    # dK and dV accumulate in a fixed order; dQ sums partials from different
    # CTAs in fp32 in arrival order, so two runs may differ in the last bits
    dq0, dk0, dv0 = plain[2]
    dq1, dk1, dv1 = timed[2]
    assert torch.equal(dk0, dk1) and torch.equal(dv0, dv1)
    assert float((dq0.float() - dq1.float()).abs().max()) <= 2.0 ** -7 * float(dq0.float().abs().max())
    assert zr.kernel_time("attn_fwd") == (0.0, 0)


def test_standard_qkv_path_equals_split_attention(zr):
    """The pages' exactness claim, checked on the GPU between the two
    strategies of "Split Attention Optimization": split attention on the
    deduplicated batch, then reconstruction, equals ordinary causal attention
    (identity grouping) on the reconstructed full Q, K, V at every valid
    position; and the standard path's dQ, dK, dV folded back with the
    reconstruction adjoint equal the split path's gradients when its upstream
    gradient is the adjoint of the standard one ("Correctness & Gradients").
    Both sides are bf16 GPU results, so the bound is twice the bf16 parity
    tolerance."""
    G, n, P, R, Hq, Hkv, D = 2, 3, 300, 140, 4, 2, 128
    ids, mask, pos = make_batch(G, n, P, R, 1000, 81, resp_len_range=(1, R))
    B, L = ids.shape
    t_ids = torch.from_numpy(ids).to(DEV)
    t_mask = torch.from_numpy(mask).to(DEV)
    t_pos = torch.from_numpy(pos).to(DEV)
    g = zr.find_prompt_groups(t_ids, R, t_mask, sync=True)
    T_ref = oracle_pack(ids, mask, pos, R, False)[4].T
    _, _, _, info, T = zr.pack_dedup(t_ids, t_pos, R, g, t_mask, T_cap=T_ref, sync=True)
    assert T == T_ref
    _, (tq, tk, tv, _) = qkv_inputs(T, Hq, Hkv, D, 12, torch.bfloat16)
    gi = zr.identity_groups(B, DEV)
    _, _, _, info_id, T_id = zr.pack_dedup(t_ids, t_pos, R, gi, t_mask, sync=True)
    assert T_id == B * L
    # forward: split, then reconstruct; versus reconstruct, then standard attention
    o, lse = zr.split_attn_fwd(info, tq, tk, tv)
    o_split = zr.reconstruct(info, o.view(T, Hq * D)).view(B, L, Hq, D)
    qf, kf, vf = (zr.reconstruct(info, x.view(T, -1)).view(B * L, x.shape[1], D) for x in (tq, tk, tv))
    o_std, lse_std = zr.split_attn_fwd(info_id, qf, kf, vf)
    torch.cuda.synchronize()
    valid = torch.from_numpy(mask != 0).to(DEV).view(B, L, 1, 1)
    tol = 2 * 2e-2
    diff = (o_split.float() - o_std.view(B, L, Hq, D).float()).abs() - 2 * 2.0 ** -8 * o_std.view(B, L, Hq, D).float().abs()
    assert float((diff * valid).max()) < tol
    # backward: upstream gradient on the full sequences, its adjoint on the packed rows
    dof = torch.randn((B, L, Hq, D), generator=torch.Generator().manual_seed(13)).to(DEV, torch.bfloat16)
    dof = dof * valid
    do_packed = zr.reconstruct_backward(info, dof.view(B, L, Hq * D)).view(T, Hq, D)
    dq, dk, dv = zr.split_attn_bwd(info, tq, tk, tv, o, lse, do_packed)
    dqf, dkf, dvf = zr.split_attn_bwd(info_id, qf, kf, vf, o_std, lse_std, dof.view(B * L, Hq, D))
    torch.cuda.synchronize()
    zr.check_status(info)
    zr.check_status(info_id)
    for got, full, name in ((dq, dqf, "dq"), (dk, dkf, "dk"), (dv, dvf, "dv")):
        ref = zr.reconstruct_backward(info, full.float().view(B, L, -1))[:T]
        d = (got.float().view(T, -1) - ref).abs() - 2 * 2.0 ** -8 * ref.abs()
        assert float(d.max()) < tol, name


def test_standard_strategy_against_oracle(zr):
    """The standard strategy ("Split Attention Optimization", split attention
    off: Q, K, V reconstructed to the full batch, then ordinary causal
    attention) against the oracle, element by element.  Q, K, V and dO are
    drawn on the deduplicated packed rows and reconstructed to [B, L] rows on
    both sides (the GPU reconstruction is bit-exact against the oracle's, see
    test_gpu_dedup); the GPU then runs its kernels over the identity grouping,
    and the oracle runs its duplicated per-sequence causal attention with
    every row its own group."""
    G, n, P, R, Hq, Hkv, D = 2, 3, 300, 140, 4, 2, 128
    ids, mask, pos = make_batch(G, n, P, R, 1000, 83, resp_len_range=(1, R))
    B, L = ids.shape
    _, _, _, _, info_ref = oracle_pack(ids, mask, pos, R, False)
    _, _, _, _, info, T = gpu_pack(zr, ids, mask, pos, R, False, T_cap=info_ref.T)
    (q, k, v, do), (tq, tk, tv, tdo) = qkv_inputs(T, Hq, Hkv, D, 15, torch.bfloat16)
    # reconstructed full-batch tensors, [B*L, H, D]
    qf_ref, kf_ref, vf_ref, dof_ref = (oracle.reconstruct_sequences(x.reshape(T, -1), info_ref)
                                       .reshape(B * L, x.shape[1], D) for x in (q, k, v, do))
    qf, kf, vf, dof = (zr.reconstruct(info, x.view(T, -1)).view(B * L, x.shape[1], D) for x in (tq, tk, tv, tdo))
    identity = [[b] for b in range(B)]
    _, _, info_id_ref = oracle.create_deduplicated_batch(ids, pos, R, identity, None, attention_mask=mask)
    assert info_id_ref.T == B * L
    o_ref, lse_ref = oracle.split_attention_fwd(qf_ref, kf_ref, vf_ref, info_id_ref)
    dq_ref, dk_ref, dv_ref = oracle.split_attention_bwd(qf_ref, kf_ref, vf_ref, dof_ref, info_id_ref)
    t_ids = torch.from_numpy(ids).to(DEV)
    gi = zr.identity_groups(B, DEV)
    _, _, _, info_id, T_id = zr.pack_dedup(t_ids, torch.from_numpy(pos).to(DEV), R, gi,
                                           torch.from_numpy(mask).to(DEV), sync=True)
    assert T_id == B * L
    o, lse, (dq, dk, dv) = _run(zr, info_id, qf, kf, vf, dof)
    assert max_abs(o, o_ref) < 2e-2, "o"
    assert max_abs(lse, lse_ref.T) < 2e-2, "lse"
    assert max_abs(dq, dq_ref) < 2e-2, "dq"
    assert max_abs(dk, dk_ref) < 2e-2, "dk"
    assert max_abs(dv, dv_ref) < 2e-2, "dv"
