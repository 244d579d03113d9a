"""Thin Python binding of libzr (ctypes).

Argument marshalling only: every step of the hot path runs in libzr's CUDA
kernels.  PyTorch supplies device memory and the current CUDA stream.  The
functions carry the names of the C entry points without the ``zr_`` prefix.
There is no CPU fallback: calling with CPU tensors, or without a built
``libzr.so``, raises.
"""

from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# ZR_LIBRARY selects another in-tree build of the same ABI, e.g. the
# bounds-checking libzr_debug.so (build(debug_bounds=True))
LIB_PATH = os.environ.get("ZR_LIBRARY") or os.path.join(_HERE, "libzr.so")

ZR_OK = 0
ZR_ERR_INVALID_ARG = 1
ZR_ERR_UNSUPPORTED = 2
ZR_ERR_CAPACITY = 3
ZR_ERR_WORKSPACE = 4
ZR_ERR_CUDA = 5
ZR_ERR_TIMEOUT = 6
ZR_ERR_NOT_IMPLEMENTED = 7
ZR_BF16 = 0
ZR_F32 = 1

_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64


class ZrGroupsC(ctypes.Structure):
    _fields_ = [("group_ptr", _vp), ("members", _vp), ("group_of", _vp), ("num_groups", _vp)]


class ZrReconInfoC(ctypes.Structure):
    _fields_ = [(n, _vp) for n in (
        "prompt_off", "prompt_slot", "prompt_len", "resp_off", "resp_slot", "resp_len",
        "group_ptr", "members", "group_of", "num_groups", "total_tokens", "status",
        "pack_segs", "recon_segs", "pad_segs", "row_prompt_len", "pack_order")] + [
        ("B", ctypes.c_int), ("L", ctypes.c_int), ("P", ctypes.c_int), ("use_unpad", ctypes.c_int),
        ("T_cap", _i64)]


class ZrBatchStatsC(ctypes.Structure):
    _fields_ = [(n, _i64) for n in ("rows", "responses", "non_pad_tokens", "total_positions",
                                    "prompt_len_min", "prompt_len_max", "resp_len_min", "resp_len_max")] + [
        (n, ctypes.c_double) for n in ("prompt_len_mean", "resp_len_mean", "non_pad_fraction")]


class ZrError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"zr status {status}: {msg}")
        self.status = status


_lib = None


def lib():
    """Load libzr.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libzr.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    sigs = {
        "zr_last_error": (ctypes.c_char_p, []),
        "zr_version": (ctypes.c_int, []),
        "zr_debug_bounds": (ctypes.c_int, []),
        "zr_kernel_launches": (_i64, []),
        "zr_set_option": (ctypes.c_int, [ctypes.c_char_p, _i64]),
        "zr_kernel_time": (ctypes.c_int, [ctypes.c_char_p, ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(_i64)]),
        "zr_kernel_time_reset": (ctypes.c_int, []),
        "zr_find_prompt_groups_workspace": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int]),
        "zr_find_prompt_groups": (ctypes.c_int, [_vp, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                 ctypes.POINTER(ZrGroupsC), _vp, _vp, _vp,
                                                 ctypes.c_size_t, _vp]),
        "zr_find_prompt_groups_noalloc": (ctypes.c_int, [_vp, _vp, ctypes.c_int, ctypes.c_int,
                                                         ctypes.c_int, ctypes.POINTER(ZrGroupsC), _vp,
                                                         _vp, _vp]),
        "zr_identity_groups": (ctypes.c_int, [ctypes.c_int, ctypes.POINTER(ZrGroupsC), _vp]),
        "zr_recon_info_bytes": (ctypes.c_size_t, [ctypes.c_int]),
        "zr_recon_info_bind": (ctypes.c_int, [ctypes.POINTER(ZrReconInfoC), _vp, ctypes.c_int,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_int, _i64]),
        "zr_pack_dedup": (ctypes.c_int, [_vp, _vp, _vp, ctypes.POINTER(ZrGroupsC), _vp, _vp, _vp,
                                         ctypes.POINTER(ZrReconInfoC), _vp, _vp]),
        "zr_pack_rows": (ctypes.c_int, [ctypes.POINTER(ZrReconInfoC), _vp, _i64, _vp, _vp]),
        "zr_reconstruct": (ctypes.c_int, [ctypes.POINTER(ZrReconInfoC), _vp, _i64, _vp, _vp]),
        "zr_reconstruct_backward": (ctypes.c_int, [ctypes.POINTER(ZrReconInfoC), _vp, _i64, ctypes.c_int, _vp,
                                                   _vp]),
        "zr_pack_rows_backward": (ctypes.c_int, [ctypes.POINTER(ZrReconInfoC), _vp, _i64, _vp, _vp]),
        "zr_reconstruct_pack_backward": (ctypes.c_int, [ctypes.POINTER(ZrReconInfoC), _vp, _i64, ctypes.c_int,
                                                        _vp, _vp]),
        "zr_batch_stats_workspace": (ctypes.c_size_t, [ctypes.c_int]),
        "zr_batch_stats_compute": (ctypes.c_int, [_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                                  ctypes.POINTER(ZrBatchStatsC), _vp, ctypes.c_size_t, _vp]),
        "zr_split_attn_workspace": (ctypes.c_size_t, [ctypes.POINTER(ZrReconInfoC), ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_int]),
        "zr_split_attn_fwd": (ctypes.c_int, [ctypes.POINTER(ZrReconInfoC), _vp, _vp, _vp, _vp, _vp,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_float, _vp, ctypes.c_size_t, _vp]),
        "zr_split_attn_bwd": (ctypes.c_int, [ctypes.POINTER(ZrReconInfoC), _vp, _vp, _vp, _vp, _vp,
                                             _vp, _vp, _vp, _vp, ctypes.c_int, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int, ctypes.c_float, _vp,
                                             ctypes.c_size_t, _vp]),
        "zr_check_status": (ctypes.c_int, [ctypes.POINTER(ZrReconInfoC), _vp, _vp]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _check(status: int):
    if status != ZR_OK:
        raise ZrError(status, lib().zr_last_error().decode())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("libzr works on CUDA tensors only (no CPU fallback)")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _rows(info, *ts):
    """The attention kernels address T_cap rows of every packed tensor."""
    for t in ts:
        if t is not None and t.shape[0] < info.T_cap:
            raise ValueError(f"packed tensors need T_cap = {info.T_cap} rows (got {t.shape[0]})")


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _aligned_empty(nbytes: int, device) -> torch.Tensor:
    t = torch.empty(max(int(nbytes), 1) + 256, dtype=torch.uint8, device=device)
    off = (-t.data_ptr()) % 256
    return t[off:off + max(int(nbytes), 1)]


def set_option(name: str, value: int):
    _check(lib().zr_set_option(name.encode(), int(value)))


def version() -> int:
    return lib().zr_version()


def debug_bounds() -> bool:
    """True when the loaded library is the bounds-checking debug build."""
    return lib().zr_debug_bounds() != 0


def kernel_launches() -> int:
    """zr_kernel_launches: kernels launched by libzr in this process."""
    return int(lib().zr_kernel_launches())


def kernel_time(name: str):
    """zr_kernel_time: (summed milliseconds, launch count) of the event pairs
    recorded for kernel `name` while the "kernel_timing" option was on."""
    ms = ctypes.c_double(0.0)
    n = _i64(0)
    _check(lib().zr_kernel_time(name.encode(), ctypes.byref(ms), ctypes.byref(n)))
    return ms.value, int(n.value)


def kernel_time_reset():
    """zr_kernel_time_reset: wait for and forget every recorded event pair."""
    _check(lib().zr_kernel_time_reset())


class Groups:
    """Output of find_prompt_groups: CSR groups on the device."""

    def __init__(self, B: int, device):
        self.B = B
        self.group_ptr = torch.empty(B + 1, dtype=torch.int32, device=device)
        self.members = torch.empty(B, dtype=torch.int32, device=device)
        self.group_of = torch.empty(B, dtype=torch.int32, device=device)
        self.num_groups = torch.empty(1, dtype=torch.int32, device=device)
        self.unique_prompts = None
        self.num_groups_host = None
        self.c = ZrGroupsC(_p(self.group_ptr), _p(self.members), _p(self.group_of),
                           _p(self.num_groups))

    def as_lists(self):
        """prompt_groups as a list of index lists (synchronises)."""
        G = int(self.num_groups.item())
        ptr = self.group_ptr.cpu().tolist()
        mem = self.members.cpu().tolist()
        return [mem[ptr[g]:ptr[g + 1]] for g in range(G)]


def find_prompt_groups(input_ids, response_length: int, attention_mask=None, unique=True,
                       sync=False, workspace=None, out: Groups | None = None) -> Groups:
    """zr_find_prompt_groups on ``input_ids [B, L]`` (int64, CUDA)."""
    _dev(input_ids, attention_mask)
    B, L = input_ids.shape
    g = out if out is not None else Groups(B, input_ids.device)
    P = L - int(response_length)
    if unique and g.unique_prompts is None:
        g.unique_prompts = torch.empty((B, P), dtype=torch.int64, device=input_ids.device)
    need = lib().zr_find_prompt_groups_workspace(B, L)
    ws = workspace if workspace is not None else _aligned_empty(need, input_ids.device)
    host = ctypes.c_int32(0)
    _check(lib().zr_find_prompt_groups(_p(input_ids), _p(attention_mask), B, L, int(response_length),
                                       ctypes.byref(g.c), _p(g.unique_prompts) if unique else None,
                                       ctypes.byref(host) if sync else None, _p(ws), ws.numel(),
                                       _stream(input_ids.device)))
    if sync:
        g.num_groups_host = host.value
    return g


def identity_groups(B: int, device) -> "Groups":
    """zr_identity_groups: every row its own group (the standard, not
    deduplicated, layout)."""
    g = Groups(B, device)
    _check(lib().zr_identity_groups(int(B), ctypes.byref(g.c), _stream(device)))
    return g


def find_prompt_groups_noalloc(input_ids, response_length: int, attention_mask=None, unique=True,
                               sync=False, out: Groups | None = None) -> Groups:
    """zr_find_prompt_groups_noalloc: the same grouping without a workspace
    (the library's own fixed device scratch; at most 4096 rows).  For callers
    that cannot allocate device memory; calls that overlap on the GPU race."""
    _dev(input_ids, attention_mask)
    B, L = input_ids.shape
    g = out if out is not None else Groups(B, input_ids.device)
    P = L - int(response_length)
    if unique and g.unique_prompts is None:
        g.unique_prompts = torch.empty((B, P), dtype=torch.int64, device=input_ids.device)
    host = ctypes.c_int32(0)
    _check(lib().zr_find_prompt_groups_noalloc(_p(input_ids), _p(attention_mask), B, L,
                                               int(response_length), ctypes.byref(g.c),
                                               _p(g.unique_prompts) if unique else None,
                                               ctypes.byref(host) if sync else None,
                                               _stream(input_ids.device)))
    if sync:
        g.num_groups_host = host.value
    return g


class ReconInfo:
    """Reconstruction info: one device buffer carved by zr_recon_info_bind."""

    def __init__(self, B: int, L: int, response_length: int, use_unpad: bool, T_cap: int, device):
        self.B, self.L, self.R = B, L, int(response_length)
        self.P = L - self.R
        self.use_unpad = bool(use_unpad)
        self.T_cap = int(T_cap)
        self.buffer = _aligned_empty(lib().zr_recon_info_bytes(B), device)
        self.c = ZrReconInfoC()
        _check(lib().zr_recon_info_bind(ctypes.byref(self.c), _p(self.buffer), B, L, self.R,
                                        int(use_unpad), self.T_cap))

    def _i32(self, name, n):
        ptr = getattr(self.c, name)
        base = self.buffer.data_ptr()
        off = ptr - base
        return self.buffer[off:off + 4 * n].view(torch.int32)

    @property
    def total_tokens(self):
        return self._i32("total_tokens", 1)

    def T(self) -> int:
        return int(self.total_tokens.item())

    def arrays(self, G=None):
        """Host copies of the metadata arrays (synchronises)."""
        G = int(self._i32("num_groups", 1).item()) if G is None else G
        out = {n: self._i32(n, self.B).cpu().numpy() for n in (
            "prompt_off", "prompt_slot", "prompt_len", "resp_off", "resp_slot", "resp_len",
            "group_of", "members")}
        for n in ("prompt_off", "prompt_slot", "prompt_len"):
            out[n] = out[n][:G]
        out["group_ptr"] = self._i32("group_ptr", self.B + 1).cpu().numpy()[:G + 1]
        out["num_groups"] = G
        out["T"] = self.T()
        return out


def pack_dedup(input_ids, position_ids, response_length: int, groups: Groups, attention_mask=None,
               use_unpad=False, T_cap=None, want_mask=False, sync=False, info: ReconInfo | None = None,
               out=None):
    """zr_pack_dedup: returns ``(dedup_ids [T_cap], dedup_pos [T_cap] or None,
    dedup_mask [T_cap] or None, info, T or None)``; T only when ``sync``."""
    _dev(input_ids, position_ids, attention_mask)
    B, L = input_ids.shape
    dev = input_ids.device
    T_cap = B * L if T_cap is None else int(T_cap)
    if info is None:
        info = ReconInfo(B, L, response_length, use_unpad, T_cap, dev)
    if out is None:
        ids = torch.empty(info.T_cap, dtype=torch.int64, device=dev)
        pos = torch.empty(info.T_cap, dtype=torch.int64, device=dev) if position_ids is not None else None
        msk = torch.empty(info.T_cap, dtype=torch.uint8, device=dev) if want_mask else None
    else:
        ids, pos, msk = out
    T_host = ctypes.c_int64(0)
    _check(lib().zr_pack_dedup(_p(input_ids), _p(position_ids), _p(attention_mask),
                               ctypes.byref(groups.c), _p(ids), _p(pos), _p(msk),
                               ctypes.byref(info.c), ctypes.byref(T_host) if sync else None,
                               _stream(dev)))
    return ids, pos, msk, info, (T_host.value if sync else None)


def pack_rows(info: ReconInfo, src, out=None):
    """zr_pack_rows: gather a ``[B, L, ...]`` tensor into ``[T_cap, ...]``."""
    _dev(src, out)
    row_bytes = src[0, 0].numel() * src.element_size()
    dst = out if out is not None else torch.empty((info.T_cap,) + tuple(src.shape[2:]),
                                                  dtype=src.dtype, device=src.device)
    _check(lib().zr_pack_rows(ctypes.byref(info.c), _p(src), row_bytes, _p(dst), _stream(src.device)))
    return dst


def reconstruct(info: ReconInfo, packed, out=None):
    """zr_reconstruct: scatter ``[T_cap, ...]`` back to ``[B, L, ...]``."""
    _dev(packed, out)
    row_bytes = packed[0].numel() * packed.element_size()
    dst = out if out is not None else torch.empty((info.B, info.L) + tuple(packed.shape[1:]),
                                                  dtype=packed.dtype, device=packed.device)
    _check(lib().zr_reconstruct(ctypes.byref(info.c), _p(packed), row_bytes, _p(dst),
                                _stream(packed.device)))
    return dst


def batch_stats(input_ids, attention_mask, response_length: int) -> dict:
    """zr_batch_stats_compute: statistics of a normal batch from its attention
    mask (``None``: every position valid); one stream synchronisation."""
    _dev(input_ids, attention_mask)
    B, L = int(input_ids.shape[0]), int(input_ids.shape[1])
    ws = _aligned_empty(lib().zr_batch_stats_workspace(B), input_ids.device)
    out = ZrBatchStatsC()
    _check(lib().zr_batch_stats_compute(_p(attention_mask), B, L, int(response_length), ctypes.byref(out),
                                        _p(ws), ws.numel(), _stream(input_ids.device)))
    return {name: getattr(out, name) for name, _ in ZrBatchStatsC._fields_}


def reconstruct_backward(info: ReconInfo, grad_out, out=None):
    """zr_reconstruct_backward: the adjoint of reconstruct, ``[B, L, ...]`` ->
    ``[T_cap, ...]`` (bf16 or fp32); shared prompt rows sum their members'
    gradients.  Rows past T of a new ``out`` are zero."""
    _dev(grad_out, out)
    if grad_out.dtype == torch.bfloat16:
        dt = ZR_BF16
    elif grad_out.dtype == torch.float32:
        dt = ZR_F32
    else:
        raise ValueError("reconstruct_backward takes bfloat16 or float32 gradients")
    W = grad_out[0, 0].numel()
    dst = out if out is not None else torch.zeros((info.T_cap,) + tuple(grad_out.shape[2:]),
                                                  dtype=grad_out.dtype, device=grad_out.device)
    _check(lib().zr_reconstruct_backward(ctypes.byref(info.c), _p(grad_out), W, dt, _p(dst),
                                         _stream(grad_out.device)))
    return dst


def pack_rows_backward(info: ReconInfo, grad_packed, out=None):
    """zr_pack_rows_backward: the adjoint of pack_rows, ``[T_cap, ...]`` ->
    ``[B, L, ...]`` (any dtype); positions the pack never read are zero."""
    _dev(grad_packed, out)
    row_bytes = grad_packed[0].numel() * grad_packed.element_size()
    dst = out if out is not None else torch.empty((info.B, info.L) + tuple(grad_packed.shape[1:]),
                                                  dtype=grad_packed.dtype, device=grad_packed.device)
    _check(lib().zr_pack_rows_backward(ctypes.byref(info.c), _p(grad_packed), row_bytes, _p(dst),
                                       _stream(grad_packed.device)))
    return dst


def reconstruct_pack_backward(info: ReconInfo, grad_out, out=None):
    """zr_reconstruct_pack_backward: the gradient of reconstruct(pack_rows(x))
    with respect to x in one pass, ``[B, L, ...]`` -> ``[B, L, ...]`` (bf16 or
    fp32)."""
    _dev(grad_out, out)
    W = grad_out[0, 0].numel()
    dst = out if out is not None else torch.empty_like(grad_out)
    _check(lib().zr_reconstruct_pack_backward(ctypes.byref(info.c), _p(grad_out), W, _dtype_code(grad_out),
                                              _p(dst), _stream(grad_out.device)))
    return dst


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return ZR_BF16
    if t.dtype == torch.float32:
        return ZR_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def attn_workspace(info: ReconInfo, Hq: int, Hkv: int, D: int, device):
    n = lib().zr_split_attn_workspace(ctypes.byref(info.c), Hq, Hkv, D)
    return _aligned_empty(n, device)


def split_attn_fwd(info: ReconInfo, q, k, v, softmax_scale=None, workspace=None, out=None):
    """zr_split_attn_fwd on packed ``q [T_cap,Hq,D]``, ``k, v [T_cap,Hkv,D]``.
    Returns ``(o [T_cap,Hq,D], lse [T_cap,Hq] float32)``."""
    _dev(q, k, v)
    _rows(info, q, k, v)
    Tc, Hq, D = q.shape
    Hkv = k.shape[1]
    ws = workspace if workspace is not None else attn_workspace(info, Hq, Hkv, D, q.device)
    if out is None:
        o = torch.empty_like(q)
        lse = torch.empty((Tc, Hq), dtype=torch.float32, device=q.device)
    else:
        o, lse = out
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check(lib().zr_split_attn_fwd(ctypes.byref(info.c), _p(q), _p(k), _p(v), _p(o), _p(lse), Hq, Hkv,
                                   D, _dtype_code(q), scale, _p(ws), ws.numel(), _stream(q.device)))
    return o, lse


def split_attn_bwd(info: ReconInfo, q, k, v, o, lse, dout, softmax_scale=None, workspace=None,
                   out=None):
    """zr_split_attn_bwd: returns ``(dq, dk, dv)``."""
    _dev(q, k, v, o, lse, dout)
    _rows(info, q, k, v, o, lse, dout)
    Tc, Hq, D = q.shape
    Hkv = k.shape[1]
    ws = workspace if workspace is not None else attn_workspace(info, Hq, Hkv, D, q.device)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    scale = 0.0 if softmax_scale is None else float(softmax_scale)
    _check(lib().zr_split_attn_bwd(ctypes.byref(info.c), _p(q), _p(k), _p(v), _p(o), _p(lse), _p(dout),
                                   _p(dq), _p(dk), _p(dv), Hq, Hkv, D, _dtype_code(q), scale, _p(ws),
                                   ws.numel(), _stream(q.device)))
    return dq, dk, dv


def check_status(info: ReconInfo, workspace=None):
    """zr_check_status: synchronise and raise on a device-reported error."""
    _check(lib().zr_check_status(ctypes.byref(info.c), _p(workspace),
                                 _stream(info.buffer.device)))


def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)
