"""GPU parity of grouping, packing and reconstruction against the oracle:
bit-exact, at small sizes and at the workloads' full sizes."""

import numpy as np
import pytest
import torch

from dummy_batch import make_batch, WORKLOADS, make_workload_batch
from gpu_util import lib, oracle_pack, gpu_pack, DEV

import oracle
from oracle.dedup import pack_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def zr():
    return lib()


def _check_pack(zr, ids, mask, pos, R, use_unpad):
    groups, uniq, dids, dpos, info = oracle_pack(ids, mask, pos, R, use_unpad)
    g, gids, gpos, gmask, ginfo, T = gpu_pack(zr, ids, mask, pos, R, use_unpad)
    assert g.num_groups_host == len(groups)
    assert g.as_lists() == groups
    G = len(groups)
    assert np.array_equal(g.unique_prompts[:G].cpu().numpy(), uniq)
    assert T == info.T
    assert np.array_equal(gids[:T].cpu().numpy(), dids)
    assert np.array_equal(gpos[:T].cpu().numpy(), dpos)
    ref_mask = np.array([1 if v else 0 for v in info.row_valid], dtype=np.uint8)
    assert np.array_equal(gmask[:T].cpu().numpy(), ref_mask)
    arr = ginfo.arrays()
    for name in ("prompt_off", "prompt_slot", "prompt_len"):
        assert np.array_equal(arr[name], getattr(info, name)), name
    for name in ("resp_off", "resp_slot", "resp_len", "group_of"):
        assert np.array_equal(arr[name], getattr(info, name)), name
    return ginfo, info, T


CASES = [
    ("tiny-contiguous", dict(G=2, n=2, P=128, R=32, vocab=32000, seed=1000, shuffle=False)),
    ("tiny-shuffled", dict(G=2, n=2, P=128, R=32, vocab=32000, seed=1001)),
    ("ragged", dict(G=3, n=5, P=77, R=45, vocab=50, seed=5, resp_len_range=(0, 45))),
    ("left-padded", dict(G=4, n=3, P=64, R=20, vocab=1000, seed=6, resp_len_range=(1, 20),
                          prompt_pad_range=(0, 30))),
    ("one-row", dict(G=1, n=1, P=9, R=3, vocab=10, seed=7)),
    ("no-response", dict(G=3, n=2, P=33, R=0, vocab=100, seed=8)),
    ("no-prompt", dict(G=1, n=6, P=0, R=19, vocab=100, seed=9)),
    ("all-distinct", dict(G=40, n=1, P=5, R=7, vocab=3, seed=10)),
    ("many-rows", dict(G=37, n=29, P=65, R=31, vocab=200, seed=11, resp_len_range=(0, 31))),
]


@pytest.mark.parametrize("use_unpad", [False, True])
@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_group_pack_reconstruct_small(zr, name, kw, use_unpad):
    ids, mask, pos = make_batch(**kw)
    R = kw["R"]
    if use_unpad and mask is None:
        mask = np.ones_like(ids, dtype=np.uint8)
    ginfo, info, T = _check_pack(zr, ids, mask, pos, R, use_unpad)
    # hidden rows: pack and reconstruct, bit-exact
    rng = np.random.default_rng(3)
    hidden = rng.standard_normal(ids.shape + (24,)).astype(np.float32)
    th = torch.from_numpy(hidden).to(DEV)
    packed = zr.pack_rows(ginfo, th)
    ref_packed = pack_rows(hidden, info)
    assert np.array_equal(packed[:T].cpu().numpy(), ref_packed)
    back = zr.reconstruct(ginfo, packed)
    ref_back = oracle.reconstruct_sequences(ref_packed, info)
    assert np.array_equal(back.cpu().numpy(), ref_back)
    zr.check_status(ginfo)


def test_forced_hash_collisions(zr):
    """With every prompt hashing alike, the exact comparison alone decides."""
    ids, mask, pos = make_batch(G=9, n=4, P=40, R=8, vocab=4, seed=12, resp_len_range=(1, 8))
    zr.set_option("weak_hash", 1)
    try:
        _check_pack(zr, ids, mask, pos, 8, False)
        # prompts that differ only in their last token
        ids2 = np.tile(np.arange(48, dtype=np.int64), (6, 1))
        ids2[::2, 39] = 7
        _check_pack(zr, ids2, None, np.tile(np.arange(48), (6, 1)), 8, False)
    finally:
        zr.set_option("weak_hash", 0)


def test_mask_is_part_of_the_prompt_key(zr):
    ids = np.array([[5, 6, 7, 1], [5, 6, 7, 2], [5, 6, 7, 3]], dtype=np.int64)
    mask = np.array([[1, 1, 1, 1], [0, 1, 1, 1], [1, 1, 1, 1]], dtype=np.uint8)
    t = torch.from_numpy(ids).to(DEV)
    g = zr.find_prompt_groups(t, 1, torch.from_numpy(mask).to(DEV), sync=True)
    assert g.as_lists() == [[0, 2], [1]]


def test_capacity_and_mask_errors(zr):
    ids, mask, pos = make_batch(G=2, n=3, P=16, R=8, vocab=100, seed=13)
    t_ids = torch.from_numpy(ids).to(DEV)
    g = zr.find_prompt_groups(t_ids, 8, sync=True)
    with pytest.raises(zr.ZrError) as e:
        zr.pack_dedup(t_ids, None, 8, g, T_cap=2 * 16 + 6 * 8 - 1, sync=True)
    assert e.value.status == zr.ZR_ERR_CAPACITY
    # asynchronous form: reported by check_status
    _, _, _, info, _ = zr.pack_dedup(t_ids, None, 8, g, T_cap=10)
    with pytest.raises(zr.ZrError) as e:
        zr.check_status(info)
    assert e.value.status == zr.ZR_ERR_CAPACITY
    bad = np.ones_like(ids, dtype=np.uint8)
    bad[0, 20] = 0  # a hole inside a response
    bad[0, 21] = 1
    bad[0, 22:] = 0
    tm = torch.from_numpy(bad).to(DEV)
    g = zr.find_prompt_groups(t_ids, 8, tm, sync=True)
    with pytest.raises(zr.ZrError) as e:
        zr.pack_dedup(t_ids, None, 8, g, tm, sync=True)
    assert e.value.status == zr.ZR_ERR_INVALID_ARG


@pytest.mark.parametrize("width,dtype", [(3, np.uint8), (9216, np.float32)], ids=["3B-rows", "36KB-rows"])
@pytest.mark.parametrize("use_unpad", [False, True])
def test_pack_reconstruct_row_widths(zr, width, dtype, use_unpad):
    """Rows narrower than a 16-byte vector and rows wider than one 32 KB work
    item: the copy kernels' byte path and one-row items, bit-exact."""
    kw = dict(G=3, n=3, P=21, R=13, vocab=40, seed=12, resp_len_range=(0, 13), prompt_pad_range=(0, 9))
    ids, mask, pos = make_batch(**kw)
    ginfo, info, T = _check_pack(zr, ids, mask, pos, kw["R"], use_unpad)
    rng = np.random.default_rng(4)
    if dtype == np.uint8:
        rows = rng.integers(0, 256, size=ids.shape + (width,), dtype=np.uint8)
    else:
        rows = rng.standard_normal(ids.shape + (width,)).astype(np.float32)
    th = torch.from_numpy(rows).to(DEV)
    packed = zr.pack_rows(ginfo, th)
    ref_packed = pack_rows(rows, info)
    assert np.array_equal(packed[:T].cpu().numpy(), ref_packed)
    back = zr.reconstruct(ginfo, packed)
    assert np.array_equal(back.cpu().numpy(), oracle.reconstruct_sequences(ref_packed, info))
    zr.check_status(ginfo)


@pytest.mark.parametrize("wname", ["qwen3_0p6b", "worked_example", "long_context", "pipeline",
                                   "pipeline_nodedup"])
def test_full_size_workloads(zr, wname):
    wl = WORKLOADS[wname]
    idx = list(WORKLOADS).index(wname)
    ids, mask, pos = make_workload_batch(wl, idx)
    for use_unpad in ([False, True] if mask is not None else [False]):
        ginfo, info, T = _check_pack(zr, ids, mask, pos, wl.R, use_unpad)
        if wl.hidden:
            rng = np.random.default_rng(idx)
            hidden = rng.standard_normal(ids.shape + (wl.hidden,), dtype=np.float32)
            th = torch.from_numpy(hidden).to(DEV, torch.bfloat16)
            packed = zr.pack_rows(ginfo, th)
            back = zr.reconstruct(ginfo, packed)
            hb = th.view(torch.int16).cpu().numpy()
            ref_packed = pack_rows(hb, info)
            assert np.array_equal(packed[:T].view(torch.int16).cpu().numpy(), ref_packed)
            ref_back = oracle.reconstruct_sequences(ref_packed, info)
            assert np.array_equal(back.view(torch.int16).cpu().numpy(), ref_back)
        zr.check_status(ginfo)


def _check_recon_backward(zr, ginfo, info, y, dtype):
    """GPU reconstruction adjoint against the oracle.  fp32 accumulation of n
    terms is within n * 2^-24 * sum|terms| of the exact sum (bound taken with
    n <= 64, i.e. 2^-18 * sum|terms|); bf16 adds one rounding of the result
    (2^-8 of its magnitude, the bf16 tolerance used throughout)."""
    ty = torch.from_numpy(y).to(DEV, dtype)
    yv = ty.float().cpu().numpy().astype(np.float64)  # the exact values the GPU sees
    got = zr.reconstruct_backward(ginfo, ty)
    torch.cuda.synchronize()
    zr.check_status(ginfo)
    T = info.T
    ref = oracle.reconstruct_backward(yv, info)
    absum = oracle.reconstruct_backward(np.abs(yv), info)
    g = got[:T].float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -18 * absum + (2.0 ** -8 * np.abs(ref) if dtype == torch.bfloat16 else 0.0) + 1e-30
    assert g.shape == ref.shape
    assert np.all(np.abs(g - ref) <= tol), float(np.max(np.abs(g - ref) - tol))
    assert torch.count_nonzero(got[T:]) == 0  # rows past T untouched (zero-initialised)


@pytest.mark.parametrize("use_unpad", [False, True])
@pytest.mark.parametrize("width,dtype", [(24, torch.float32), (3, torch.float32), (40, torch.bfloat16),
                                         (5, torch.bfloat16)], ids=["f32-24", "f32-3", "bf16-40", "bf16-5"])
@pytest.mark.parametrize("name,kw", [CASES[2], CASES[3], CASES[5], CASES[6], CASES[8]],
                         ids=[CASES[i][0] for i in (2, 3, 5, 6, 8)])
def test_reconstruct_backward_small(zr, name, kw, use_unpad, width, dtype):
    ids, mask, pos = make_batch(**kw)
    R = kw["R"]
    if use_unpad and mask is None:
        mask = np.ones_like(ids, dtype=np.uint8)
    ginfo, info, T = _check_pack(zr, ids, mask, pos, R, use_unpad)
    y = np.random.default_rng(8).standard_normal(ids.shape + (width,)).astype(np.float32)
    _check_recon_backward(zr, ginfo, info, y, dtype)


@pytest.mark.parametrize("wname", ["worked_example", "pipeline", "long_context"])
def test_reconstruct_backward_full_size(zr, wname):
    """Full-size grouping and layout (the pages' worked example, the pipeline
    batch with ragged responses, the long-context batch), narrow rows so the
    oracle's per-row loop stays small."""
    wl = WORKLOADS[wname]
    idx = list(WORKLOADS).index(wname)
    ids, mask, pos = make_workload_batch(wl, idx)
    for use_unpad in ([False, True] if mask is not None else [False]):
        ginfo, info, T = _check_pack(zr, ids, mask, pos, wl.R, use_unpad)
        y = np.random.default_rng(idx).standard_normal(ids.shape + (8,)).astype(np.float32)
        _check_recon_backward(zr, ginfo, info, y, torch.bfloat16)


@pytest.mark.parametrize("kw", [
    dict(G=4, n=5, P=30, R=12, vocab=100, seed=9, resp_len_range=(0, 12), prompt_pad_range=(0, 7)),
    dict(G=2, n=3, P=17, R=0, vocab=10, seed=2),
    dict(G=1, n=4, P=0, R=9, vocab=10, seed=3, resp_len_range=(0, 9)),
], ids=["ragged", "no-response", "no-prompt"])
def test_batch_stats_matches_oracle(zr, kw):
    ids, mask, pos = make_batch(**kw)
    R = kw["R"]
    t_ids = torch.from_numpy(ids).to(DEV)
    got = zr.batch_stats(t_ids, None if mask is None else torch.from_numpy(mask).to(DEV), R)
    ref = oracle.batch_stats(np.ones_like(ids) if mask is None else mask, R)
    assert got == ref  # integer counts, and means as the same double division


def test_batch_stats_full_size(zr):
    wl = WORKLOADS["pipeline"]
    ids, mask, pos = make_workload_batch(wl, list(WORKLOADS).index("pipeline"))
    got = zr.batch_stats(torch.from_numpy(ids).to(DEV), torch.from_numpy(mask).to(DEV), wl.R)
    assert got == oracle.batch_stats(mask, wl.R)
    assert got["responses"] == wl.B and 256 <= got["resp_len_min"] <= got["resp_len_max"] <= 1024


def _check_pack_backward(zr, ginfo, info, ids_shape, width, dtype, seed):
    """The pack adjoint is a copy: bit-exact against the oracle, every
    position written (unread ones zero)."""
    T = info.T
    gp = torch.from_numpy(np.random.default_rng(seed).standard_normal((ginfo.T_cap, width)).astype(np.float32))
    gp = gp.to(DEV, dtype)
    got = zr.pack_rows_backward(ginfo, gp)
    torch.cuda.synchronize()
    zr.check_status(ginfo)
    ref = oracle.pack_rows_backward(gp[:T].float().cpu().numpy(), info)
    assert tuple(got.shape) == tuple(ids_shape) + (width,)
    assert np.array_equal(got.float().cpu().numpy(), ref)


@pytest.mark.parametrize("use_unpad", [False, True])
@pytest.mark.parametrize("width,dtype", [(3, torch.float32), (40, torch.bfloat16), (1, torch.bfloat16)],
                         ids=["f32-3", "bf16-40", "bf16-1"])
@pytest.mark.parametrize("name,kw", [CASES[1], CASES[2], CASES[3], CASES[5], CASES[6], CASES[8]],
                         ids=[CASES[i][0] for i in (1, 2, 3, 5, 6, 8)])
def test_pack_rows_backward_small(zr, name, kw, use_unpad, width, dtype):
    ids, mask, pos = make_batch(**kw)
    R = kw["R"]
    if use_unpad and mask is None:
        mask = np.ones_like(ids, dtype=np.uint8)
    ginfo, info, T = _check_pack(zr, ids, mask, pos, R, use_unpad)
    _check_pack_backward(zr, ginfo, info, ids.shape, width, dtype, 12)


@pytest.mark.parametrize("use_unpad", [False, True])
@pytest.mark.parametrize("width,dtype", [(24, torch.float32), (3, torch.float32), (40, torch.bfloat16),
                                         (5, torch.bfloat16)], ids=["f32-24", "f32-3", "bf16-40", "bf16-5"])
@pytest.mark.parametrize("name,kw", [CASES[2], CASES[3], CASES[5], CASES[6], CASES[8]],
                         ids=[CASES[i][0] for i in (2, 3, 5, 6, 8)])
def test_reconstruct_pack_backward_small(zr, name, kw, use_unpad, width, dtype):
    """The fused round-trip gradient: bitwise equal to the reconstruction
    adjoint followed by the pack adjoint on the GPU, and within the fp32
    summation bound of the oracle's composition of the two."""
    ids, mask, pos = make_batch(**kw)
    R = kw["R"]
    if use_unpad and mask is None:
        mask = np.ones_like(ids, dtype=np.uint8)
    ginfo, info, T = _check_pack(zr, ids, mask, pos, R, use_unpad)
    y = np.random.default_rng(13).standard_normal(ids.shape + (width,)).astype(np.float32)
    ty = torch.from_numpy(y).to(DEV, dtype)
    fused = zr.reconstruct_pack_backward(ginfo, ty)
    two_step = zr.pack_rows_backward(ginfo, zr.reconstruct_backward(ginfo, ty))
    torch.cuda.synchronize()
    zr.check_status(ginfo)
    assert torch.equal(fused, two_step)
    yv = ty.float().cpu().numpy().astype(np.float64)
    ref = oracle.pack_rows_backward(oracle.reconstruct_backward(yv, info), info)
    absum = oracle.pack_rows_backward(oracle.reconstruct_backward(np.abs(yv), info), info)
    g = fused.float().cpu().numpy().astype(np.float64)
    tol = 2.0 ** -18 * absum + (2.0 ** -8 * np.abs(ref) if dtype == torch.bfloat16 else 0.0) + 1e-30
    assert np.all(np.abs(g - ref) <= tol), float(np.max(np.abs(g - ref) - tol))


@pytest.mark.parametrize("wname", ["worked_example", "pipeline", "long_context"])
def test_pack_backward_full_size(zr, wname):
    """Full-size layouts (padded and, with a mask, unpadded): the pack adjoint
    bit-exact against the oracle, the fused round trip bitwise equal to the
    two adjoints in sequence."""
    wl = WORKLOADS[wname]
    idx = list(WORKLOADS).index(wname)
    ids, mask, pos = make_workload_batch(wl, idx)
    for use_unpad in ([False, True] if mask is not None else [False]):
        ginfo, info, T = _check_pack(zr, ids, mask, pos, wl.R, use_unpad)
        _check_pack_backward(zr, ginfo, info, ids.shape, 8, torch.bfloat16, idx)
        ty = torch.randn(ids.shape + (64,), generator=torch.Generator().manual_seed(idx)).to(DEV, torch.bfloat16)
        fused = zr.reconstruct_pack_backward(ginfo, ty)
        two_step = zr.pack_rows_backward(ginfo, zr.reconstruct_backward(ginfo, ty))
        torch.cuda.synchronize()
        zr.check_status(ginfo)
        assert torch.equal(fused, two_step)
