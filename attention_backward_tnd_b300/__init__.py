"""Python binding of the TND attention library (``libtndattn.so``).

Argument marshalling only: every step of the forward and the gradient runs in
the library's CUDA kernels.  The ``tnd_*`` functions mirror the C entry points
of ``include/tnd_attn.h`` one to one (integers for device pointers and the
stream); ``fwd`` and ``grad`` take torch CUDA tensors, allocate outputs and the
workspace with torch, and call those entry points on the current stream.
There is no fallback: without the built library every call raises.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtndattn.so")

TND_OK, TND_ERR_NULLPTR, TND_ERR_INVALID, TND_ERR_UNSUPPORTED = 0, 1, 2, 3
TND_ERR_WORKSPACE, TND_ERR_CUDA, TND_ERR_DEVICE_TIMEOUT, TND_ERR_DEVICE_CHECK = 4, 5, 6, 7
TND_F16, TND_BF16, TND_F32 = 0, 1, 2
TND_OPT_GRAD_PATH, TND_OPT_WAIT_LIMIT_MS, TND_OPT_PROFILE, TND_OPT_TEST_SKIP_LOAD, TND_OPT_DETERMINISTIC = 0, 1, 2, 3, 4

# exported symbols, in header order
SYMBOLS = ["tnd_attn_fwd_workspace_size", "tnd_attn_fwd", "tnd_attn_grad_workspace_size", "tnd_attn_grad",
           "tnd_attn_device_status", "tnd_status_string", "tnd_attn_set_option", "tnd_attn_profile_read",
           "tnd_attn_grad_plan", "tnd_attn_grad_static_ws", "tnd_attn_grad_static_ws_status"]


class TndError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: status {status} ({status_text(status)})")
        self.status = status


_lib = None
_i64, _u64, _f64, _vp, _int = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
_i64p = ctypes.POINTER(ctypes.c_int64)


def lib():
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library {LIB_PATH} is missing; build it with "
                               "attention_backward_tnd_b300.build.build()")
        L = ctypes.CDLL(LIB_PATH)
        ws_args = [_int, _i64, _i64p, _i64p, _i64p, _i64, _i64, _i64, _i64, _f64, _f64, _i64, _i64, _i64, _int,
                   _int, _int, ctypes.POINTER(ctypes.c_uint64)]
        L.tnd_attn_fwd_workspace_size.argtypes = ws_args
        L.tnd_attn_grad_workspace_size.argtypes = ws_args
        L.tnd_attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _int, _i64, _i64p, _i64p, _i64p,
                                   _i64, _i64, _i64, _i64, _f64, _f64, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _u64,
                                   _vp]
        L.tnd_attn_grad.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _int, _i64,
                                    _i64p, _i64p, _i64p, _i64, _i64, _i64, _i64, _f64, _f64, _i64, _i64, _i64, _vp,
                                    _vp, _vp, _vp, _vp, _u64, _vp]
        L.tnd_attn_device_status.argtypes = [_vp, _u64, _vp]
        L.tnd_status_string.argtypes = [_int]
        L.tnd_status_string.restype = ctypes.c_char_p
        L.tnd_attn_set_option.argtypes = [_int, _i64]
        L.tnd_attn_profile_read.argtypes = [ctypes.POINTER(ctypes.c_char_p), ctypes.POINTER(ctypes.c_double),
                                            _i64p, _int, ctypes.POINTER(ctypes.c_int), _int]
        L.tnd_attn_grad_plan.argtypes = [_i64, _i64p, _i64p, _i64p, _i64, _i64, _i64, _i64, _i64, _int, _i64p,
                                         _i64, _i64p, _i64p]
        L.tnd_attn_grad_static_ws.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _i64, _i64p,
                                              _i64p, _i64, _i64, _i64, _f64, _f64, _i64, _i64, _i64, _vp, _vp, _vp,
                                              _vp, _vp]
        L.tnd_attn_grad_static_ws_status.argtypes = [_vp]
        for name in SYMBOLS:
            if name != "tnd_status_string":
                getattr(L, name).restype = _int
        _lib = L
    return _lib


def status_text(status: int) -> str:
    try:
        return lib().tnd_status_string(status).decode()
    except Exception:  # pragma: no cover - library missing
        return "?"


def _cu(arr) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(arr, dtype=np.int64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_i64p)


def _pre(prefix):
    """Host prefix array (int64) or None, kept alive by the caller."""
    return None if prefix is None else _cu(prefix)


def _pp(arr):
    return None if arr is None else _p(arr)


# --- one-to-one wrappers of the C entry points --------------------------------------------

def tnd_attn_fwd_workspace_size(dtype, batch, cu_q, cu_kv, prefix, head_num, kv_head_num, head_dim, value_head_dim,
                                scale_value, keep_prob, pre_tokens, next_tokens, sparse_mode, has_drop_mask,
                                has_atten_mask, has_sink):
    cq, ck, pf, out = _cu(cu_q), _cu(cu_kv), _pre(prefix), ctypes.c_uint64(0)
    st = lib().tnd_attn_fwd_workspace_size(dtype, batch, _p(cq), _p(ck), _pp(pf), head_num, kv_head_num, head_dim,
                                           value_head_dim, scale_value, keep_prob, pre_tokens, next_tokens,
                                           sparse_mode,
                                           int(has_drop_mask), int(has_atten_mask), int(has_sink),
                                           ctypes.byref(out))
    return st, out.value


def tnd_attn_grad_workspace_size(dtype, batch, cu_q, cu_kv, prefix, head_num, kv_head_num, head_dim,
                                 value_head_dim, scale_value, keep_prob, pre_tokens, next_tokens, sparse_mode,
                                 has_drop_mask, has_atten_mask, has_sink):
    cq, ck, pf, out = _cu(cu_q), _cu(cu_kv), _pre(prefix), ctypes.c_uint64(0)
    st = lib().tnd_attn_grad_workspace_size(dtype, batch, _p(cq), _p(ck), _pp(pf), head_num, kv_head_num,
                                            head_dim, value_head_dim, scale_value, keep_prob, pre_tokens,
                                            next_tokens, sparse_mode,
                                            int(has_drop_mask), int(has_atten_mask), int(has_sink),
                                            ctypes.byref(out))
    return st, out.value


def tnd_attn_fwd(query, key, value, pse, pse_batch, pse_type, drop_mask, atten_mask, sink, dtype, batch, cu_q,
                 cu_kv, prefix, head_num, kv_head_num, head_dim, value_head_dim, scale_value, keep_prob, pre_tokens,
                 next_tokens, sparse_mode, attention_out, softmax_max, softmax_sum, workspace, workspace_size, stream):
    cq, ck, pf = _cu(cu_q), _cu(cu_kv), _pre(prefix)
    return lib().tnd_attn_fwd(query, key, value, pse, pse_batch, pse_type, drop_mask, atten_mask, sink, dtype, batch,
                              _p(cq), _p(ck), _pp(pf), head_num, kv_head_num, head_dim, value_head_dim, scale_value,
                              keep_prob, pre_tokens, next_tokens, sparse_mode, attention_out, softmax_max,
                              softmax_sum, workspace, workspace_size, stream)


def tnd_attn_grad(query, key, value, dy, pse, pse_batch, pse_type, drop_mask, atten_mask, softmax_max, softmax_sum,
                  attention_in, sink, dtype, batch, cu_q, cu_kv, prefix, head_num, kv_head_num, head_dim,
                  value_head_dim, scale_value, keep_prob, pre_tokens, next_tokens, sparse_mode, dq, dk, dv, dsink,
                  workspace, workspace_size, stream):
    cq, ck, pf = _cu(cu_q), _cu(cu_kv), _pre(prefix)
    return lib().tnd_attn_grad(query, key, value, dy, pse, pse_batch, pse_type, drop_mask, atten_mask, softmax_max,
                               softmax_sum, attention_in, sink, dtype, batch, _p(cq), _p(ck), _pp(pf), head_num,
                               kv_head_num, head_dim, value_head_dim, scale_value, keep_prob, pre_tokens,
                               next_tokens, sparse_mode, dq, dk, dv, dsink, workspace, workspace_size, stream)


def tnd_attn_grad_static_ws(query, key, value, dy, drop_mask, softmax_max, softmax_sum, attention_in, sink, dtype,
                            batch, cu_q, cu_kv, head_num, kv_head_num, head_dim, scale_value, keep_prob, pre_tokens,
                            next_tokens, sparse_mode, dq, dk, dv, dsink, stream):
    """tnd_attn_grad with the library's own fixed device workspace (no allocation)."""
    cq, ck = _cu(cu_q), _cu(cu_kv)
    return lib().tnd_attn_grad_static_ws(query, key, value, dy, drop_mask, softmax_max, softmax_sum, attention_in,
                                         sink, dtype, batch, _p(cq), _p(ck), head_num, kv_head_num, head_dim,
                                         scale_value, keep_prob, pre_tokens, next_tokens, sparse_mode, dq, dk, dv,
                                         dsink, stream)


TND_STATIC_WS_BYTES = 32 << 20


def tnd_attn_grad_static_ws_status(stream):
    """Device status of the last tnd_attn_grad_static_ws call on the current device (waits for `stream`)."""
    return lib().tnd_attn_grad_static_ws_status(stream)


def tnd_attn_device_status(workspace, workspace_size, stream):
    return lib().tnd_attn_device_status(workspace, workspace_size, stream)


def tnd_status_string(status: int) -> str:
    return lib().tnd_status_string(status).decode()


def tnd_attn_set_option(option: int, value: int) -> int:
    return lib().tnd_attn_set_option(option, value)


def tnd_attn_profile_read(reset: bool = False):
    """{kernel name: (total ms, launches)} recorded since the last reset."""
    cap = 32
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_double * cap)()
    n = (ctypes.c_int64 * cap)()
    count = ctypes.c_int(0)
    st = lib().tnd_attn_profile_read(names, ms, n, cap, ctypes.byref(count), int(reset))
    if st != TND_OK:
        raise TndError(st, "tnd_attn_profile_read")
    return {names[i].decode(): (ms[i], n[i]) for i in range(count.value)}


def tnd_attn_grad_plan(batch, cu_q, cu_kv, head_num, kv_head_num, pre_tokens, next_tokens, sparse_mode,
                       prefix=None, has_atten_mask=False):
    """(status, units int64 [n,5] = (b, g, j, first q block, end q block), kept pairs)."""
    cq, ck, pf = _cu(cu_q), _cu(cu_kv), _pre(prefix)
    n, kept = ctypes.c_int64(0), ctypes.c_int64(0)
    st = lib().tnd_attn_grad_plan(batch, _p(cq), _p(ck), _pp(pf), head_num, kv_head_num, pre_tokens, next_tokens,
                                  sparse_mode, int(has_atten_mask), None, 0, ctypes.byref(n), ctypes.byref(kept))
    if st != TND_OK:
        return st, None, None
    units = np.zeros((n.value, 5), dtype=np.int64)
    st = lib().tnd_attn_grad_plan(batch, _p(cq), _p(ck), _pp(pf), head_num, kv_head_num, pre_tokens, next_tokens,
                                  sparse_mode, int(has_atten_mask), _p(units), n.value, ctypes.byref(n),
                                  ctypes.byref(kept))
    return st, units, kept.value


# --- torch-tensor helpers -----------------------------------------------------------------

def dtype_code(t) -> int:
    import torch
    return {torch.float16: TND_F16, torch.bfloat16: TND_BF16, torch.float32: TND_F32}[t.dtype]


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _check_amask(atten_mask, cu_q, cu_kv):
    """The matrix must be a contiguous one-byte [S1Max, S2Max] tensor (the C ABI takes its pointer only)."""
    if atten_mask is None:
        return
    s1 = int(np.max(np.diff(_cu(cu_q))))
    s2 = int(np.max(np.diff(_cu(cu_kv))))
    if tuple(atten_mask.shape) != (s1, s2) or atten_mask.element_size() != 1 or not atten_mask.is_contiguous():
        raise ValueError(f"atten_mask must be a contiguous uint8/bool tensor of shape ({s1}, {s2})")


def _check_pse(pse, q, cu_kv, batch, pse_type=1) -> int:
    """pse must be a contiguous [B or 1, Nq, 1024, S2Max] tensor of q's dtype (pseType 0 / 1) or
    float32 slopes [B, Nq] or [Nq] (pseType 2 / 3); returns its first dim (0 = none)."""
    import torch
    if pse is None:
        return 0
    if pse_type in (2, 3):
        if pse.dtype != torch.float32 or not pse.is_contiguous() or pse.shape[-1] != q.shape[1] or \
                pse.dim() not in (1, 2) or (pse.dim() == 2 and pse.shape[0] != batch):
            raise ValueError(f"pseType {pse_type} takes contiguous float32 slopes [{batch}, {q.shape[1]}] "
                             f"or [{q.shape[1]}]")
        return batch if pse.dim() == 2 else 1
    s2 = int(np.max(np.diff(_cu(cu_kv))))
    if pse.dim() != 4 or pse.shape[0] not in (1, batch) or tuple(pse.shape[1:]) != (q.shape[1], 1024, s2) or \
            pse.dtype != q.dtype or not pse.is_contiguous():
        raise ValueError(f"pse must be a contiguous [{batch} or 1, {q.shape[1]}, 1024, {s2}] tensor of {q.dtype}")
    return int(pse.shape[0])


def _stream():
    import torch
    return torch.cuda.current_stream().cuda_stream


def fwd(q, k, v, cu_q: Sequence[int], cu_kv: Sequence[int], scale: float, keep_prob: float = 1.0,
        pre_tokens: int = 2147483647, next_tokens: int = 2147483647, sparse_mode: int = 0, drop_mask=None,
        sink=None, workspace=None, atten_mask=None, prefix=None, pse=None, pse_type: int = 1):
    """Forward on torch CUDA tensors: returns (out, softmax_max, softmax_sum) ([T,N,8] fp32 stats).
    atten_mask: uint8/bool CUDA tensor [S1Max, S2Max] (nonzero masks); prefix: host ints (sparse_mode 6);
    pse: CUDA tensor [B or 1, Nq, 1024, S2Max] in q's dtype (the last 1024 rows of each sequence's bias;
    pse_type 0 / 1), or float32 slopes [B, Nq] or [Nq] (pse_type 2 / 3: the bias is generated)."""
    import torch
    tq, nq, d = q.shape
    nkv, dv = k.shape[1], v.shape[2]
    batch = len(cu_q) - 1
    dt = dtype_code(q)
    _check_amask(atten_mask, cu_q, cu_kv)
    st, ws_bytes = tnd_attn_fwd_workspace_size(dt, batch, cu_q, cu_kv, prefix, nq, nkv, d, dv, scale, keep_prob,
                                               pre_tokens, next_tokens, sparse_mode, drop_mask is not None,
                                               atten_mask is not None, sink is not None)
    if st != TND_OK:
        raise TndError(st, "tnd_attn_fwd_workspace_size")
    out = torch.empty((tq, nq, dv), dtype=q.dtype, device=q.device)
    smax = torch.empty((tq, nq, 8), dtype=torch.float32, device=q.device)
    ssum = torch.empty((tq, nq, 8), dtype=torch.float32, device=q.device)
    if workspace is None or workspace.numel() < ws_bytes:
        workspace = torch.empty(max(ws_bytes, 256), dtype=torch.uint8, device=q.device)
    pb = _check_pse(pse, q, cu_kv, batch, pse_type)
    st = tnd_attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), _ptr(pse), pb, pse_type, _ptr(drop_mask),
                      _ptr(atten_mask), _ptr(sink), dt, batch, cu_q, cu_kv, prefix, nq, nkv, d, dv, scale,
                      keep_prob, pre_tokens, next_tokens, sparse_mode, out.data_ptr(), smax.data_ptr(), ssum.data_ptr(),
                      workspace.data_ptr(), workspace.numel(), _stream())
    if st != TND_OK:
        raise TndError(st, "tnd_attn_fwd")
    return out, smax, ssum


def grad_workspace_bytes(q, k, cu_q, cu_kv, scale, keep_prob=1.0, pre_tokens=2147483647,
                         next_tokens=2147483647, sparse_mode=0, has_drop=False, has_sink=False,
                         has_atten_mask=False, prefix=None, v=None) -> int:
    """Workspace bytes of the gradient (v gives the value head dim; default q's)."""
    dv = q.shape[2] if v is None else v.shape[2]
    st, n = tnd_attn_grad_workspace_size(dtype_code(q), len(cu_q) - 1, cu_q, cu_kv, prefix, q.shape[1], k.shape[1],
                                         q.shape[2], dv, scale, keep_prob, pre_tokens, next_tokens, sparse_mode,
                                         has_drop, has_atten_mask, has_sink)
    if st != TND_OK:
        raise TndError(st, "tnd_attn_grad_workspace_size")
    return n


def grad(q, k, v, dy, out, softmax_max, softmax_sum, cu_q, cu_kv, scale, keep_prob=1.0,
         pre_tokens=2147483647, next_tokens=2147483647, sparse_mode=0, drop_mask=None, sink=None,
         workspace=None, outputs=None, atten_mask=None, prefix=None, pse=None, pse_type: int = 1):
    """Gradient on torch CUDA tensors: returns (dq, dk, dv, dsink or None)."""
    import torch
    tq, nq, d = q.shape
    nkv, dvd = k.shape[1], v.shape[2]
    batch = len(cu_q) - 1
    dt = dtype_code(q)
    _check_amask(atten_mask, cu_q, cu_kv)
    if workspace is None:
        n = grad_workspace_bytes(q, k, cu_q, cu_kv, scale, keep_prob, pre_tokens, next_tokens, sparse_mode,
                                 drop_mask is not None, sink is not None, atten_mask is not None, prefix, v)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    if outputs is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        dsink = torch.empty(nq, dtype=torch.float32, device=q.device) if sink is not None else None
    else:
        dq, dk, dv, dsink = outputs
    pb = _check_pse(pse, q, cu_kv, batch, pse_type)
    st = tnd_attn_grad(q.data_ptr(), k.data_ptr(), v.data_ptr(), dy.data_ptr(), _ptr(pse), pb, pse_type,
                       _ptr(drop_mask), _ptr(atten_mask), softmax_max.data_ptr(), softmax_sum.data_ptr(),
                       out.data_ptr(), _ptr(sink), dt, batch, cu_q, cu_kv, prefix, nq, nkv, d, dvd, scale,
                       keep_prob, pre_tokens, next_tokens, sparse_mode, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                       _ptr(dsink), workspace.data_ptr(), workspace.numel(), _stream())
    if st != TND_OK:
        raise TndError(st, "tnd_attn_grad")
    return dq, dk, dv, dsink


def device_status(workspace) -> int:
    return tnd_attn_device_status(workspace.data_ptr(), workspace.numel(), _stream())
