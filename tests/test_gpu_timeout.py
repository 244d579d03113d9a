"""Failure detection of the tensor-core attention kernels, without a GPU fault.

Every mbarrier wait in those kernels is bounded.  The test option
"test_withhold_arrival" makes the CTA that takes the first work unit skip
one of its loads (the forward: the unit's Q tile; the backward: its K/V
tile), so the wait for it runs out after "wait_limit" cycles.  The CTA then
raises its abort flag, every role
leaves its loop, the producer waits for its own copies in flight, the MMA
warp waits for its own MMAs, TMEM is freed and the kernel returns; the
timeout lands in the reconstruction info's status words and zr_check_status
reports ZR_ERR_TIMEOUT.  Nothing traps or hangs: a following normal call on
the same context must pass parity against the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from dummy_batch import make_batch
from gpu_util import lib, oracle_pack, gpu_pack, qkv_inputs, max_abs

pytestmark = pytest.mark.gpu

SHORT_LIMIT = 20_000_000  # SM clock cycles: about 10 ms


@pytest.fixture(scope="module")
def zr():
    return lib()


def _case(zr):
    ids, mask, pos = make_batch(2, 3, 300, 140, 1000, 91, resp_len_range=(1, 140))
    _, _, _, _, info_ref = oracle_pack(ids, mask, pos, 140, False)
    _, _, _, _, info, T = gpu_pack(zr, ids, mask, pos, 140, False, T_cap=info_ref.T)
    (q, k, v, do), dev = qkv_inputs(T, 4, 2, 128, 17, torch.bfloat16)
    return info_ref, info, (q, k, v, do), dev


def _timed_out(zr, fn):
    zr.set_option("wait_limit", SHORT_LIMIT)
    zr.set_option("test_withhold_arrival", fn[0])
    try:
        out = fn[1]()
        torch.cuda.synchronize()  # the kernel returned: no hang, no fault
    finally:
        zr.set_option("test_withhold_arrival", 0)
        zr.set_option("wait_limit", 0)
    return out


def _normal_run_matches_oracle(zr, info_ref, info, host, dev):
    q, k, v, do = host
    tq, tk, tv, tdo = dev
    o, lse = zr.split_attn_fwd(info, tq, tk, tv)
    dq, dk, dv = zr.split_attn_bwd(info, tq, tk, tv, o, lse, tdo)
    torch.cuda.synchronize()
    zr.check_status(info)
    o_ref, lse_ref = oracle.split_attention_fwd(q, k, v, info_ref)
    dq_ref, dk_ref, dv_ref = oracle.split_attention_bwd(q, k, v, do, info_ref)
    assert max_abs(o, o_ref) < 2e-2 and max_abs(lse, lse_ref.T) < 2e-2
    assert max_abs(dq, dq_ref) < 2e-2 and max_abs(dk, dk_ref) < 2e-2 and max_abs(dv, dv_ref) < 2e-2


def test_forward_withheld_load_times_out_then_recovers(zr):
    info_ref, info, host, dev = _case(zr)
    tq, tk, tv, _ = dev
    _timed_out(zr, (1, lambda: zr.split_attn_fwd(info, tq, tk, tv)))
    with pytest.raises(zr.ZrError) as e:
        zr.check_status(info)
    assert e.value.status == zr.ZR_ERR_TIMEOUT
    zr.check_status(info)  # the report cleared the status word
    _normal_run_matches_oracle(zr, info_ref, info, host, dev)


def test_backward_withheld_load_times_out_then_recovers(zr):
    info_ref, info, host, dev = _case(zr)
    tq, tk, tv, tdo = dev
    o, lse = zr.split_attn_fwd(info, tq, tk, tv)
    torch.cuda.synchronize()
    zr.check_status(info)
    _timed_out(zr, (2, lambda: zr.split_attn_bwd(info, tq, tk, tv, o, lse, tdo)))
    with pytest.raises(zr.ZrError) as e:
        zr.check_status(info)
    assert e.value.status == zr.ZR_ERR_TIMEOUT
    _normal_run_matches_oracle(zr, info_ref, info, host, dev)
