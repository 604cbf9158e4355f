"""Exact attention forward for GB300 (sm_103a): Python binding of the C ABI.

The binding only marshals arguments to ``libfa_gb300.so`` (``include/fa.h``);
every step of the computation runs in the library's CUDA kernels.  PyTorch is
used for device memory and streams only.  There is no CPU fallback: if the
library is missing or a call fails, an exception is raised.

    from exact_attention_forward_08_gb300 import attention_forward
    o, lse = attention_forward(q, k, v, causal=True)   # q [B,Sq,Hq,d] bf16 on cuda
    o, lse = attention_forward_varlen(q, k, v, cu_q, cu_k)  # q [total_q,Hq,d], cu_q int32 [B+1]

Raw entry points with the C names: ``fa_fwd``, ``fa_fwd_ex``, ``fa_fwd_varlen``,
``fa_fwd_varlen_ex``, ``fa_varlen_workspace_size``, ``fa_varlen_plan_host``,
``fa_device_status``, ``fa_status_string``, ``fa_make_plan``, ``fa_plan_task``, ``fa_plan_set_grid``,
``fa_plan_block_masked``, ``fa_plan_first_masked_block``, ``fa_version``.
"""
from __future__ import annotations

import ctypes
import math
import os

from . import _build

__all__ = ["fa_fwd", "fa_fwd_ex", "fa_fwd_varlen", "fa_fwd_varlen_ex", "fa_varlen_workspace_size",
           "fa_varlen_plan_host", "fa_fwd_splitkv", "fa_splitkv_workspace_size", "fa_splitkv_num_splits",
           "attention_forward_splitkv", "fa_bwd", "fa_bwd_workspace_size", "attention_backward",
           "fa_bwd_varlen", "fa_bwd_varlen_workspace_size", "attention_backward_varlen",
           "fa_fwd_varlen_noalloc", "fa_noalloc_scratch_bytes", "fa_device_status", "fa_device_status_code", "fa_status_string", "fa_selftest_exp2", "fa_make_plan",
           "fa_plan_task", "fa_plan_set_grid", "fa_plan_block_masked", "fa_plan_first_masked_block", "fa_version", "FaOptions", "FaPlan",
           "FaTask", "FaVarlenTask", "attention_forward", "attention_forward_varlen", "FaError", "load_library",
           "LIB_PATH", "STATUS", "VARLEN_HEADER_BYTES"]

LIB_PATH = _build.LIB
STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_CUDA",
          4: "FA_ERR_DEVICE_TIMEOUT", 5: "FA_ERR_DEVICE_CHECK"}
FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT, FA_ERR_DEVICE_CHECK = range(6)


class FaError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)}" if what else STATUS.get(code, str(code)))


class FaOptions(ctypes.Structure):
    _fields_ = [("tau", ctypes.c_float), ("pack", ctypes.c_int), ("grid", ctypes.c_int),
                ("timeout_s", ctypes.c_double), ("debug_flags", ctypes.c_int), ("exp_emu", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("store_mode", ctypes.c_int), ("no_balance", ctypes.c_int),
                ("trace", ctypes.c_void_p), ("trace_ctas", ctypes.c_int), ("trace_cap", ctypes.c_int),
                ("stagger", ctypes.c_int)]


# bytes of the optional fixed-length scheduling workspace (fa_options.workspace)
SCHED_WORKSPACE_BYTES = 16


class FaPlan(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("batch", "heads_q", "heads_kv", "seqlen_q", "seqlen_k", "causal",
                                            "pack", "groups", "pos_per_tile", "tiles", "mblocks", "kv_blocks",
                                            "ratio", "section_units", "heavy_levels")] + [("num_tasks", ctypes.c_int64),
                                                                                          ("tail_first", ctypes.c_int64),
                                                                                          ("grid", ctypes.c_int)]


class FaTask(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int), ("g", ctypes.c_int), ("mblock", ctypes.c_int), ("kv_head", ctypes.c_int),
                ("pos0", ctypes.c_int * 2), ("n_blocks", ctypes.c_int * 2), ("key_split", ctypes.c_int)]


class FaVarlenTask(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in ("b", "g", "mblock", "reserved", "q_row0", "seqlen_q", "k_row0",
                                            "seqlen_k")]


# a varlen workspace holds the task count at byte 0 and the task records from this offset
VARLEN_HEADER_BYTES = 256

_lib = None

_I = ctypes.c_int
_P = ctypes.c_void_p
_FWD_ARGS = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float]


def load_library(path: str | None = None):
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise FaError(FA_ERR_CUDA, f"CUDA library not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p)
    lib.fa_fwd.argtypes = _FWD_ARGS + [_P]
    lib.fa_fwd.restype = _I
    lib.fa_fwd_ex.argtypes = _FWD_ARGS + [ctypes.POINTER(FaOptions), _P]
    lib.fa_fwd_ex.restype = _I
    lib.fa_options_default.argtypes = [ctypes.POINTER(FaOptions)]
    lib.fa_options_default.restype = None
    lib.fa_device_status.argtypes = [_P, ctypes.POINTER(_I)]
    lib.fa_device_status.restype = _I
    lib.fa_device_status_detail.argtypes = [_P, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_uint)]
    lib.fa_device_status_detail.restype = _I
    lib.fa_debug_rescale_count.argtypes = [_P, ctypes.POINTER(ctypes.c_uint)]
    lib.fa_debug_rescale_count.restype = _I
    lib.fa_status_string.argtypes = [_I]
    lib.fa_status_string.restype = ctypes.c_char_p
    lib.fa_version.argtypes = []
    lib.fa_version.restype = _I
    lib.fa_make_plan.argtypes = [_I] * 8 + [ctypes.c_int64, _I, ctypes.POINTER(FaPlan)]
    lib.fa_make_plan.restype = _I
    lib.fa_plan_task.argtypes = [ctypes.POINTER(FaPlan), ctypes.c_int64, ctypes.POINTER(FaTask)]
    lib.fa_plan_task.restype = _I
    lib.fa_plan_set_grid.argtypes = [ctypes.POINTER(FaPlan), _I]
    lib.fa_plan_set_grid.restype = _I
    lib.fa_plan_block_masked.argtypes = [ctypes.POINTER(FaPlan), _I, _I]
    lib.fa_plan_block_masked.restype = _I
    lib.fa_selftest_exp2.argtypes = [_P, _P, _P, _I, _P]
    lib.fa_selftest_exp2.restype = _I
    lib.fa_plan_first_masked_block.argtypes = [ctypes.POINTER(FaPlan), _I]
    lib.fa_plan_first_masked_block.restype = _I
    lib.fa_varlen_workspace_size.argtypes = [_I, _I, ctypes.c_int64]
    lib.fa_varlen_workspace_size.restype = ctypes.c_size_t
    vl = [_P, _P, _P, _P, _P, _P, _P, _I, ctypes.c_int64, ctypes.c_int64, _I, _I, _I, _I, _I, ctypes.c_float, _P,
          ctypes.c_size_t]
    lib.fa_fwd_varlen.argtypes = vl + [_P]
    lib.fa_fwd_varlen.restype = _I
    lib.fa_fwd_varlen_ex.argtypes = vl + [ctypes.POINTER(FaOptions), _P]
    lib.fa_fwd_varlen_ex.restype = _I
    lib.fa_fwd_splitkv.argtypes = _FWD_ARGS + [_I, _P, ctypes.c_size_t, _P]
    lib.fa_fwd_splitkv.restype = _I
    lib.fa_fwd_splitkv_ex.argtypes = _FWD_ARGS + [_I, _P, ctypes.c_size_t, ctypes.POINTER(FaOptions), _P]
    lib.fa_fwd_splitkv_ex.restype = _I
    lib.fa_splitkv_workspace_size.argtypes = [_I] * 5
    lib.fa_splitkv_workspace_size.restype = ctypes.c_size_t
    lib.fa_splitkv_num_splits.argtypes = [_I] * 10
    lib.fa_splitkv_num_splits.restype = _I
    bw = [_P] * 9 + [_I] * 8 + [ctypes.c_float, _P, ctypes.c_size_t]
    lib.fa_bwd.argtypes = bw + [_P]
    lib.fa_bwd.restype = _I
    bvl = [_P] * 11 + [_I, ctypes.c_int64, ctypes.c_int64] + [_I] * 5 + [ctypes.c_float, _P, ctypes.c_size_t]
    lib.fa_bwd_varlen.argtypes = bvl + [_P]
    lib.fa_bwd_varlen.restype = _I
    lib.fa_bwd_varlen_ex.argtypes = bvl + [ctypes.POINTER(FaOptions), _P]
    lib.fa_bwd_varlen_ex.restype = _I
    lib.fa_bwd_varlen_workspace_size.argtypes = [_I, _I, _I, ctypes.c_int64, ctypes.c_int64]
    lib.fa_bwd_varlen_workspace_size.restype = ctypes.c_size_t
    lib.fa_bwd_ex.argtypes = bw + [ctypes.POINTER(FaOptions), _P]
    lib.fa_bwd_ex.restype = _I
    lib.fa_bwd_workspace_size.argtypes = [_I, _I, _I]
    lib.fa_bwd_workspace_size.restype = ctypes.c_size_t
    lib.fa_fwd_varlen_noalloc.argtypes = vl[:16] + [_P]
    lib.fa_fwd_varlen_noalloc.restype = _I
    lib.fa_noalloc_scratch_bytes.argtypes = []
    lib.fa_noalloc_scratch_bytes.restype = ctypes.c_size_t
    lib.fa_varlen_plan_host.argtypes = [_P, _P] + [_I] * 6 + [ctypes.c_int64, _I, ctypes.POINTER(FaVarlenTask),
                                                             ctypes.c_int64, ctypes.POINTER(ctypes.c_int64)]
    lib.fa_varlen_plan_host.restype = _I
    if path is None:
        _lib = lib
    return lib


# ---------------------------------------------------------------------------
# raw C entry points (pointers and sizes)
# ---------------------------------------------------------------------------

def fa_fwd(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, scale, stream) -> int:
    """``fa_fwd`` of include/fa.h; pointer arguments are integers (device addresses)."""
    return load_library().fa_fwd(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v,
                                 int(causal), float(scale), stream)


def default_options() -> FaOptions:
    o = FaOptions()
    load_library().fa_options_default(ctypes.byref(o))
    return o


def fa_fwd_ex(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, scale, opts,
              stream) -> int:
    """``fa_fwd_ex``: ``opts`` is an ``FaOptions`` or None."""
    return load_library().fa_fwd_ex(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v,
                                    int(causal), float(scale), ctypes.byref(opts) if opts is not None else None,
                                    stream)


def fa_device_status(stream=None):
    """Synchronise ``stream`` and read/clear the device status through
    ``fa_device_status_detail``: (code, (code, site, block))."""
    out = _I(0)
    detail = (ctypes.c_uint * 3)()
    rc = load_library().fa_device_status_detail(stream, ctypes.byref(out), detail)
    if rc != FA_OK:
        raise FaError(rc, "fa_device_status_detail")
    return out.value, tuple(detail)


def fa_device_status_code(stream=None) -> int:
    """``fa_device_status``: synchronise ``stream``, read and clear the status code."""
    out = _I(0)
    rc = load_library().fa_device_status(stream, ctypes.byref(out))
    if rc != FA_OK:
        raise FaError(rc, "fa_device_status")
    return out.value


# fa_options.debug_flags bits
DEBUG_SKIP_P_ARRIVE = 1
DEBUG_COUNT_RESCALE = 2
DEBUG_CHECKS = 4        # the checking build of the forward kernel
DEBUG_PLANT_BAD_TASK = 8  # with DEBUG_CHECKS: task 0 decodes out of range (the checks must catch it)


def fa_debug_rescale_count(stream=None) -> int:
    """Synchronise ``stream``, read and clear the count of O rescales (forward
    calls made with ``debug_flags`` bit 1): one per warp of 32 rows and K/V
    block whose correction warps rescaled O."""
    out = ctypes.c_uint(0)
    rc = load_library().fa_debug_rescale_count(stream, ctypes.byref(out))
    if rc != FA_OK:
        raise FaError(rc, "fa_debug_rescale_count")
    return int(out.value)


def fa_selftest_exp2(x, y_fma, y_mufu, n, stream) -> int:
    """``fa_selftest_exp2``: device pointers as integers."""
    return load_library().fa_selftest_exp2(x, y_fma, y_mufu, n, stream)


def fa_status_string(code: int) -> str:
    return load_library().fa_status_string(code).decode()


def fa_version() -> int:
    return load_library().fa_version()


def fa_make_plan(batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, l2_bytes=0, pack=0) -> FaPlan:
    plan = FaPlan()
    rc = load_library().fa_make_plan(batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, int(causal), l2_bytes,
                                     pack, ctypes.byref(plan))
    if rc != FA_OK:
        raise FaError(rc, "fa_make_plan")
    return plan


def fa_plan_task(plan: FaPlan, task: int) -> FaTask:
    t = FaTask()
    rc = load_library().fa_plan_task(ctypes.byref(plan), task, ctypes.byref(t))
    if rc != FA_OK:
        raise FaError(rc, "fa_plan_task")
    return t


def fa_plan_set_grid(plan: FaPlan, grid: int) -> FaPlan:
    """Apply the balanced static order the kernel runs on `grid` CTAs (in place)."""
    rc = load_library().fa_plan_set_grid(ctypes.byref(plan), grid)
    if rc != FA_OK:
        raise FaError(rc, "fa_plan_set_grid")
    return plan


def fa_plan_block_masked(plan: FaPlan, pos0: int, j: int) -> bool:
    return bool(load_library().fa_plan_block_masked(ctypes.byref(plan), pos0, j))


def fa_plan_first_masked_block(plan: FaPlan, pos0: int) -> int:
    return load_library().fa_plan_first_masked_block(ctypes.byref(plan), pos0)


def fa_varlen_workspace_size(batch: int, heads_q: int, total_q: int) -> int:
    return load_library().fa_varlen_workspace_size(batch, heads_q, total_q)


def fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, batch, total_q, total_k, heads_q, heads_kv, d_qk, d_v, causal, scale,
                  workspace, workspace_bytes, stream) -> int:
    """``fa_fwd_varlen`` of include/fa.h; pointer arguments are integers (device addresses)."""
    return load_library().fa_fwd_varlen(q, k, v, o, lse, cu_q, cu_k, batch, total_q, total_k, heads_q, heads_kv, d_qk,
                                        d_v, int(causal), float(scale), workspace, workspace_bytes, stream)


def fa_fwd_varlen_ex(q, k, v, o, lse, cu_q, cu_k, batch, total_q, total_k, heads_q, heads_kv, d_qk, d_v, causal,
                     scale, workspace, workspace_bytes, opts, stream) -> int:
    return load_library().fa_fwd_varlen_ex(q, k, v, o, lse, cu_q, cu_k, batch, total_q, total_k, heads_q, heads_kv,
                                           d_qk, d_v, int(causal), float(scale), workspace, workspace_bytes,
                                           ctypes.byref(opts) if opts is not None else None, stream)


def fa_fwd_splitkv(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, scale,
                   num_splits, workspace, workspace_bytes, stream, opts=None) -> int:
    """``fa_fwd_splitkv_ex`` (``opts`` None: defaults); pointers as integers."""
    return load_library().fa_fwd_splitkv_ex(q, k, v, o, lse, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v,
                                            int(causal), float(scale), num_splits, workspace, workspace_bytes,
                                            ctypes.byref(opts) if opts is not None else None, stream)


def fa_splitkv_workspace_size(batch, heads_q, seqlen_q, d_v, num_splits) -> int:
    return load_library().fa_splitkv_workspace_size(batch, heads_q, seqlen_q, d_v, num_splits)


def fa_splitkv_num_splits(batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, num_sms, pack=0) -> int:
    return load_library().fa_splitkv_num_splits(batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, int(causal),
                                                pack, num_sms)


def attention_forward_splitkv(q, k, v, causal: bool = False, scale: float | None = None, num_splits: int = 0,
                              out=None, lse=None, workspace=None, stream=None, options: FaOptions | None = None):
    """Split-KV forward (decode / short Q): same tensors as ``attention_forward``.

    ``num_splits`` 0 lets the library choose; the workspace (uint8) is
    allocated for the count the call will use when not given.  Returns (O, LSE).
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise FaError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous 4-D bf16 CUDA tensor")
    B, Sq, Hq, dqk = q.shape
    _, Sk, Hkv, _ = k.shape
    dv = v.shape[3]
    if out is None:
        out = torch.empty((B, Sq, Hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    splits = num_splits
    if splits == 0:
        sms = torch.cuda.get_device_properties(q.device).multi_processor_count
        splits = fa_splitkv_num_splits(B, Hq, Hkv, Sq, Sk, dqk, dv, causal, sms,
                                       options.pack if options is not None else 0)
    need = fa_splitkv_workspace_size(B, Hq, Sq, dv, splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    s = 0.0 if scale is None else float(scale)
    rc = fa_fwd_splitkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(), B, Hq, Hkv, Sq, Sk,
                        dqk, dv, causal, s, num_splits, workspace.data_ptr(),
                        workspace.numel() * workspace.element_size(), sptr, options)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv")
    return out, lse


def fa_bwd_workspace_size(batch: int, heads_q: int, seqlen_q: int) -> int:
    return load_library().fa_bwd_workspace_size(batch, heads_q, seqlen_q)


def fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, batch, heads_q, heads_kv, seqlen_q, seqlen_k, d_qk, d_v, causal, scale,
           workspace, workspace_bytes, stream, opts=None) -> int:
    """``fa_bwd_ex`` of include/fa.h (``opts`` None: defaults); pointers as integers."""
    return load_library().fa_bwd_ex(q, k, v, o, lse, dout, dq, dk, dv, batch, heads_q, heads_kv, seqlen_q, seqlen_k,
                                    d_qk, d_v, int(causal), float(scale), workspace, workspace_bytes,
                                    ctypes.byref(opts) if opts is not None else None, stream)


def attention_backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None, dq=None, dk=None,
                       dv=None, workspace=None, stream=None, options: FaOptions | None = None):
    """(dQ, dK, dV) for bf16 CUDA tensors laid out as ``attention_forward``'s
    (q, k, v, its outputs o and lse, and dout = dLoss/dO).  Allocates the
    gradients and the workspace when not given."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise FaError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous 4-D bf16 CUDA tensor")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise FaError(FA_ERR_INVALID_ARG, "lse must be a contiguous fp32 CUDA tensor")
    B, Sq, Hq, dqk = q.shape
    _, Sk, Hkv, _ = k.shape
    dvh = v.shape[3]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = fa_bwd_workspace_size(B, Hq, Sq)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    s = 0.0 if scale is None else float(scale)
    rc = fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Sq, Sk, dqk, dvh, causal, s,
                workspace.data_ptr(), workspace.numel() * workspace.element_size(), sptr, options)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


def fa_fwd_varlen_noalloc(q, k, v, o, lse, cu_q, cu_k, batch, total_q, total_k, heads_q, heads_kv, d_qk, d_v,
                          causal, scale, stream) -> int:
    """``fa_fwd_varlen_noalloc``: the varlen call with the library's static scratch (no workspace)."""
    return load_library().fa_fwd_varlen_noalloc(q, k, v, o, lse, cu_q, cu_k, batch, total_q, total_k, heads_q,
                                                heads_kv, d_qk, d_v, int(causal), float(scale), stream)


def fa_noalloc_scratch_bytes() -> int:
    return load_library().fa_noalloc_scratch_bytes()


def fa_varlen_plan_host(cu_q, cu_k, heads_q, heads_kv, d_qk, d_v, causal, l2_bytes=0, pack=0):
    """Host copy of the planning kernel's task list for int sequences ``cu_q``, ``cu_k`` (length B + 1)."""
    batch = len(cu_q) - 1
    cq = (ctypes.c_int * len(cu_q))(*[int(x) for x in cu_q])
    ck = (ctypes.c_int * len(cu_k))(*[int(x) for x in cu_k])
    n = ctypes.c_int64(0)
    lib = load_library()
    rc = lib.fa_varlen_plan_host(cq, ck, batch, heads_q, heads_kv, d_qk, d_v, int(causal), l2_bytes, pack, None, 0,
                                 ctypes.byref(n))
    if rc != FA_OK:
        raise FaError(rc, "fa_varlen_plan_host")
    out = (FaVarlenTask * max(n.value, 1))()
    rc = lib.fa_varlen_plan_host(cq, ck, batch, heads_q, heads_kv, d_qk, d_v, int(causal), l2_bytes, pack, out,
                                 n.value, ctypes.byref(n))
    if rc != FA_OK:
        raise FaError(rc, "fa_varlen_plan_host")
    return list(out)[: n.value]


# ---------------------------------------------------------------------------
# torch convenience wrapper (allocation and argument marshalling only)
# ---------------------------------------------------------------------------

def attention_forward(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                      return_lse: bool = True, stream=None, options: FaOptions | None = None, workspace=None):
    """O (and LSE) for bf16 CUDA tensors q [B,Sq,Hq,dqk], k [B,Sk,Hkv,dqk], v [B,Sk,Hkv,dv].

    Allocates ``out`` [B,Sq,Hq,dv] bf16 and ``lse`` [B,Hq,Sq] fp32 when not given.
    ``workspace`` (a CUDA tensor of at least SCHED_WORKSPACE_BYTES bytes) selects
    dynamic task assignment (``fa_options.workspace``).  Launches on ``stream``
    (default: torch's current stream).  Raises FaError on any non-OK status.
    """
    import torch

    if workspace is not None:
        if not workspace.is_cuda or workspace.numel() * workspace.element_size() < SCHED_WORKSPACE_BYTES:
            raise FaError(FA_ERR_INVALID_ARG, f"workspace must be a CUDA tensor of >= {SCHED_WORKSPACE_BYTES} bytes")
        base = options if options is not None else default_options()
        options = FaOptions.from_buffer_copy(base)
        options.workspace = workspace.data_ptr()

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise FaError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous 4-D bf16 CUDA tensor")
    B, Sq, Hq, dqk = q.shape
    _, Sk, Hkv, _ = k.shape
    dv = v.shape[3]
    if out is None:
        out = torch.empty((B, Sq, Hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    s = 0.0 if scale is None else float(scale)
    rc = fa_fwd_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                   lse.data_ptr() if lse is not None else None, B, Hq, Hkv, Sq, Sk, dqk, dv, causal, s, options, sptr)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return (out, lse) if return_lse else out


def attention_forward_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, causal: bool = False, scale: float | None = None,
                             out=None, lse=None, return_lse: bool = True, workspace=None, stream=None,
                             options: FaOptions | None = None):
    """O (and LSE) of a variable-length batch: q [total_q,Hq,dqk], k [total_k,Hkv,dqk], v [total_k,Hkv,dv]
    bf16 CUDA tensors, cu_seqlens_q / cu_seqlens_k int32 CUDA tensors [B+1].

    Allocates ``out`` [total_q,Hq,dv] bf16, ``lse`` [Hq,total_q] fp32 and the
    planning workspace (uint8) when not given.  Bad cu_seqlens are detected on
    the device and reported by ``fa_device_status``.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise FaError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous 3-D bf16 CUDA tensor")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() or t.dim() != 1:
            raise FaError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous 1-D int32 CUDA tensor")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
        raise FaError(FA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must both hold batch + 1 offsets")
    batch = cu_seqlens_q.numel() - 1
    total_q, Hq, dqk = q.shape
    total_k, Hkv, _ = k.shape
    dv = v.shape[2]
    if out is None:
        out = torch.empty((total_q, Hq, dv), dtype=torch.bfloat16, device=q.device)
    if lse is None and return_lse:
        lse = torch.empty((Hq, total_q), dtype=torch.float32, device=q.device)
    need = fa_varlen_workspace_size(batch, Hq, total_q)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    s = 0.0 if scale is None else float(scale)
    rc = fa_fwd_varlen_ex(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr() if lse is not None else None, cu_seqlens_q.data_ptr(),
                          cu_seqlens_k.data_ptr(), batch, total_q, total_k, Hq, Hkv, dqk, dv, causal, s,
                          workspace.data_ptr(), workspace.numel(), options, sptr)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_varlen")
    return (out, lse) if return_lse else out


def flops(batch, heads_q, seqlen_q, seqlen_k, d_qk, d_v, causal) -> float:
    """2*B*Hq*Sq*Sk*(d_qk + d_v), halved for causal (the nominal convention)."""
    f = 2.0 * batch * heads_q * seqlen_q * seqlen_k * (d_qk + d_v)
    return f / 2 if causal else f


def default_scale(d_qk: int) -> float:
    return 1.0 / math.sqrt(d_qk)


def fa_bwd_varlen_workspace_size(batch: int, heads_q: int, heads_kv: int, total_q: int, total_k: int) -> int:
    return load_library().fa_bwd_varlen_workspace_size(batch, heads_q, heads_kv, total_q, total_k)


def fa_bwd_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_q, cu_k, batch, total_q, total_k, heads_q, heads_kv, d_qk,
                  d_v, causal, scale, workspace, workspace_bytes, stream, opts=None) -> int:
    """``fa_bwd_varlen_ex`` of include/fa.h (``opts`` None: defaults); pointers as integers."""
    return load_library().fa_bwd_varlen_ex(q, k, v, o, lse, dout, dq, dk, dv, cu_q, cu_k, batch, total_q, total_k,
                                           heads_q, heads_kv, d_qk, d_v, int(causal), float(scale), workspace,
                                           workspace_bytes, ctypes.byref(opts) if opts is not None else None,
                                           stream)


def attention_backward_varlen(q, k, v, o, lse, dout, cu_seqlens_q, cu_seqlens_k, causal: bool = False,
                              scale: float | None = None, dq=None, dk=None, dv=None, workspace=None, stream=None,
                              options: FaOptions | None = None):
    """(dQ, dK, dV) of a variable-length batch laid out as
    ``attention_forward_varlen``'s: q [total_q,Hq,dqk], k [total_k,Hkv,dqk],
    v [total_k,Hkv,dv], its outputs o [total_q,Hq,dv] and lse [Hq,total_q],
    dout like o; cu_seqlens int32 CUDA tensors [B+1].  Allocates the gradients
    and the workspace when not given."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise FaError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous 3-D bf16 CUDA tensor")
    if lse.dtype != torch.float32 or not lse.is_cuda or not lse.is_contiguous():
        raise FaError(FA_ERR_INVALID_ARG, "lse must be a contiguous fp32 CUDA tensor")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_cuda or not t.is_contiguous() or t.dim() != 1:
            raise FaError(FA_ERR_INVALID_ARG, f"{name} must be a contiguous 1-D int32 CUDA tensor")
    if cu_seqlens_q.numel() != cu_seqlens_k.numel() or cu_seqlens_q.numel() < 1:
        raise FaError(FA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must both hold batch + 1 offsets")
    batch = cu_seqlens_q.numel() - 1
    total_q, Hq, dqk = q.shape
    total_k, Hkv, _ = k.shape
    dvh = v.shape[2]
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = fa_bwd_varlen_workspace_size(batch, Hq, Hkv, total_q, total_k)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    sptr = stream.cuda_stream if hasattr(stream, "cuda_stream") else stream
    s = 0.0 if scale is None else float(scale)
    rc = fa_bwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), dout.data_ptr(),
                       dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_seqlens_q.data_ptr(), cu_seqlens_k.data_ptr(),
                       batch, total_q, total_k, Hq, Hkv, dqk, dvh, causal, s, workspace.data_ptr(),
                       workspace.numel() * workspace.element_size(), sptr, options)
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_varlen")
    return dq, dk, dv
