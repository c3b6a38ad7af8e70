"""Python binding of libkvevict: head-adaptive KV-cache eviction and flat decode attention
on GB300 (sm_103a).

Every function here only marshals arguments (torch CUDA tensors to device
pointers, the current stream) and calls the C ABI declared in
``include/kvevict.h``; all computation runs in the library's CUDA kernels.
There is no CPU fallback: if ``libkvevict.so`` has not been built, or a tensor
is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "KV_OK", "KV_ERR_INVALID_ARG", "KV_ERR_UNSUPPORTED", "KV_ERR_WORKSPACE", "KV_ERR_CAPACITY",
    "KV_ERR_CUDA", "KV_ERR_DEVICE_CHECK", "KV_BF16", "KV_F32", "KV_SCORE_ADA", "KV_SCORE_LAVA",
    "KV_SCORE_CRITICAL", "KV_GROUP_MEAN", "KV_GROUP_MAX", "KV_OP_SCORE", "KV_OP_ALLOCATE",
    "KV_OP_COMPACT", "KV_OP_DECODE", "KvShape", "KvError", "lib", "library_path",
    "kv_workspace_size", "kv_score", "kv_crit_norm", "kv_allocate", "kv_allocate_capped",
    "kv_compact", "kv_recompact", "kv_recompact_workspace_size", "kv_window_terms",
    "kv_proj_score", "kv_compact_kappa", "kv_compact_streaming", "KV_TERMS_MEAN_POOLED",
    "KV_TERMS_L2",
    "KV_PROJ_CRIT_GQA", "KV_PROJ_LAPROX",
    "flat_decode_attn", "kv_check_device_status", "kv_status_string", "kv_kernel_launches",
    "flat_decode_attn_noalloc",
]

KV_OK, KV_ERR_INVALID_ARG, KV_ERR_UNSUPPORTED, KV_ERR_WORKSPACE = 0, 1, 2, 3
KV_ERR_CAPACITY, KV_ERR_CUDA, KV_ERR_DEVICE_CHECK = 4, 5, 6
KV_BF16, KV_F32 = 0, 1
KV_SCORE_ADA, KV_SCORE_LAVA, KV_SCORE_CRITICAL = 0, 1, 2
KV_GROUP_MEAN, KV_GROUP_MAX = 0, 1
KV_OP_SCORE, KV_OP_ALLOCATE, KV_OP_COMPACT, KV_OP_DECODE = 0, 1, 2, 3
KV_TERMS_MEAN_POOLED, KV_TERMS_L2 = 0, 1
KV_PROJ_CRIT_GQA, KV_PROJ_LAPROX = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.path.join(_HERE, "libkvevict.so")


class KvShape(ctypes.Structure):
    _fields_ = [(f, ctypes.c_int32) for f in
                ("batch", "layers", "hq", "hkv", "d", "n", "w", "pool", "dtype")]

    @classmethod
    def of(cls, batch, layers, hq, hkv, d, n, w, pool, dtype) -> "KvShape":
        if isinstance(dtype, str):
            dtype = KV_BF16 if dtype == "bf16" else KV_F32
        return cls(batch, layers, hq, hkv, d, n, w, pool, dtype)

    @classmethod
    def from_workload(cls, wl, batch: Optional[int] = None, layers: Optional[int] = None):
        return cls.of(wl.batch if batch is None else batch, wl.layers if layers is None else layers,
                      wl.hq, wl.hkv, wl.d, wl.n, wl.w, wl.pool, wl.dtype)


class KvError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__("%s: %s (status %d)" % (fn, kv_status_string(status), status))


_LIB = None
_vp, _sz, _i32, _u32, _f32, _i64 = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32,
                                     ctypes.c_uint32, ctypes.c_float, ctypes.c_int64)
_SIGS = {
    "kv_workspace_size": (_sz, [ctypes.c_int, ctypes.POINTER(KvShape)]),
    "kv_score": (ctypes.c_int, [ctypes.POINTER(KvShape), ctypes.c_int, ctypes.c_int, _vp, _vp, _vp,
                                _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "kv_crit_norm": (ctypes.c_int, [ctypes.POINTER(KvShape), _vp, _vp, _i32, _vp, _vp, _sz, _vp]),
    "kv_window_terms": (ctypes.c_int, [ctypes.POINTER(KvShape), ctypes.c_int, _vp, _vp, _vp, _vp,
                                       _sz, _vp]),
    "kv_proj_score": (ctypes.c_int, [ctypes.POINTER(KvShape), ctypes.c_int, _vp, _vp, _i32, _vp,
                                     _f32, _vp, _vp, _sz, _vp]),
    "kv_compact_streaming": (ctypes.c_int, [ctypes.POINTER(KvShape), _vp, _vp, _i32, _vp, _i32,
                                            _vp, _vp, _vp, _vp, _vp, _i64, _vp, _sz, _vp]),
    "kv_compact_kappa": (ctypes.c_int, [ctypes.POINTER(KvShape), _vp, _vp, _vp, _vp, _u32, _u32,
                                        _vp, _i32, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _sz,
                                        _vp]),
    "kv_allocate_capped": (ctypes.c_int, [ctypes.POINTER(KvShape), _vp, _vp, _vp, _u32, _u32,
                                          _vp, _vp, _vp, _sz, _vp]),
    "kv_recompact_workspace_size": (_sz, [_i64]),
    "kv_recompact": (ctypes.c_int, [ctypes.POINTER(KvShape), _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _sz,
                                    _vp]),
    "kv_allocate": (ctypes.c_int, [ctypes.POINTER(KvShape), _vp, _vp, ctypes.c_int, _u32, _u32,
                                   _vp, _vp, _vp, _sz, _vp]),
    "kv_compact": (ctypes.c_int, [ctypes.POINTER(KvShape), _vp, _vp, _vp, _vp, _u32, _u32, _f32,
                                  _vp, _i32, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _sz, _vp]),
    "flat_decode_attn": (ctypes.c_int, [ctypes.POINTER(KvShape), _vp, _vp, _vp, _vp, _vp, _vp,
                                        _vp, _i64, _f32, _vp, _vp, _sz, _vp]),
    "kv_check_device_status": (ctypes.c_int, [_vp, _vp, ctypes.POINTER(_u32)]),
    "kv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kv_kernel_launches": (ctypes.c_uint64, []),
    "flat_decode_attn_noalloc": (ctypes.c_int, [ctypes.POINTER(KvShape), _vp, _vp, _vp, _vp, _vp,
                                                _vp, _vp, _i64, _f32, _vp, _vp]),
}


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError("libkvevict.so is not built: run __graft_entry__.build() "
                               "or python -m kv_cache_eviction_gb300._build")
        L = ctypes.CDLL(path)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = L
    return _LIB


def _ptr(t) -> Optional[int]:
    """Device pointer of a CUDA tensor (None stays NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _nbytes(t) -> int:
    return 0 if t is None else t.numel() * t.element_size()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int) -> None:
    if st != KV_OK:
        raise KvError(fn, st)


def kv_status_string(status: int) -> str:
    return lib().kv_status_string(status).decode()


def kv_workspace_size(op: int, shape: KvShape) -> int:
    return int(lib().kv_workspace_size(op, ctypes.byref(shape)))


def kv_score(shape: KvShape, mode: int, group: int, q_win, k, v, w_o, model_dim: int, scores,
             crit_norm, ws, stream=None) -> None:
    st = lib().kv_score(ctypes.byref(shape), mode, group, _ptr(q_win), _ptr(k), _ptr(v), _ptr(w_o),
                        model_dim, _ptr(scores), _ptr(crit_norm), _ptr(ws), _nbytes(ws),
                        _stream(stream))
    _check("kv_score", st)


def kv_crit_norm(shape: KvShape, v, w_o, model_dim: int, crit_norm, ws, stream=None) -> None:
    st = lib().kv_crit_norm(ctypes.byref(shape), _ptr(v), _ptr(w_o), model_dim, _ptr(crit_norm),
                            _ptr(ws), _nbytes(ws), _stream(stream))
    _check("kv_crit_norm", st)


def kv_allocate(shape: KvShape, scores, budget, layer_entropy_mode: int, alpha_num: int,
                alpha_den: int, layer_budget, head_budget, ws, stream=None) -> None:
    st = lib().kv_allocate(ctypes.byref(shape), _ptr(scores), _ptr(budget), layer_entropy_mode,
                           alpha_num, alpha_den, _ptr(layer_budget), _ptr(head_budget), _ptr(ws),
                           _nbytes(ws), _stream(stream))
    _check("kv_allocate", st)


def kv_window_terms(shape: KvShape, kind: int, q_win, k, terms, ws, stream=None) -> None:
    st = lib().kv_window_terms(ctypes.byref(shape), kind, _ptr(q_win), _ptr(k), _ptr(terms),
                               _ptr(ws), _nbytes(ws), _stream(stream))
    _check("kv_window_terms", st)


def kv_proj_score(shape: KvShape, kind: int, v, w_o, model_dim: int, terms, eps: float, out, ws,
                  stream=None) -> None:
    st = lib().kv_proj_score(ctypes.byref(shape), kind, _ptr(v), _ptr(w_o), model_dim,
                             _ptr(terms), eps, _ptr(out), _ptr(ws), _nbytes(ws), _stream(stream))
    _check("kv_proj_score", st)


def kv_compact_streaming(shape: KvShape, k, v, sinks: int, head_budget, reserve: int, kept_idx,
                         cu_off, lens, k_flat, v_flat, flat_capacity_rows: int, ws,
                         stream=None) -> None:
    st = lib().kv_compact_streaming(ctypes.byref(shape), _ptr(k), _ptr(v), sinks,
                                    _ptr(head_budget), reserve, _ptr(kept_idx), _ptr(cu_off),
                                    _ptr(lens), _ptr(k_flat), _ptr(v_flat), flat_capacity_rows,
                                    _ptr(ws), _nbytes(ws), _stream(stream))
    _check("kv_compact_streaming", st)


def kv_compact_kappa(shape: KvShape, k, v, scores, kappa, crit_alpha_num: int,
                     crit_alpha_den: int, head_budget, reserve: int, kept_idx, cu_off, lens,
                     k_flat, v_flat, flat_capacity_rows: int, ws, stream=None) -> None:
    st = lib().kv_compact_kappa(ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(scores), _ptr(kappa),
                                crit_alpha_num, crit_alpha_den, _ptr(head_budget), reserve,
                                _ptr(kept_idx), _ptr(cu_off), _ptr(lens), _ptr(k_flat),
                                _ptr(v_flat), flat_capacity_rows, _ptr(ws), _nbytes(ws),
                                _stream(stream))
    _check("kv_compact_kappa", st)


def kv_allocate_capped(shape: KvShape, scores, budget, layer_cap, alpha_num: int, alpha_den: int,
                       layer_budget, head_budget, ws, stream=None) -> None:
    st = lib().kv_allocate_capped(ctypes.byref(shape), _ptr(scores), _ptr(budget),
                                  _ptr(layer_cap), alpha_num, alpha_den, _ptr(layer_budget),
                                  _ptr(head_budget), _ptr(ws), _nbytes(ws), _stream(stream))
    _check("kv_allocate_capped", st)


def kv_recompact_workspace_size(src_capacity_rows: int) -> int:
    return int(lib().kv_recompact_workspace_size(src_capacity_rows))


def kv_recompact(shape: KvShape, scores, head_budget, src_kept, src_cu, src_lens, src_k, src_v,
                 reserve: int, row_base, kept_idx, cu_off, lens, k_flat, v_flat, ws,
                 stream=None, src_capacity_rows=None, flat_capacity_rows=None) -> None:
    """src_kept / src_cu / src_lens None: the source is the uncompacted K/V."""
    src_cap = src_k.shape[0] if src_capacity_rows is None else src_capacity_rows
    if src_kept is None:
        src_cap = 0
    cap = k_flat.shape[0] if flat_capacity_rows is None else flat_capacity_rows
    st = lib().kv_recompact(ctypes.byref(shape), _ptr(scores), _ptr(head_budget), _ptr(src_kept),
                            _ptr(src_cu), _ptr(src_lens), _ptr(src_k), _ptr(src_v), src_cap,
                            reserve, _ptr(row_base), _ptr(kept_idx), _ptr(cu_off), _ptr(lens),
                            _ptr(k_flat), _ptr(v_flat), cap, _ptr(ws), _nbytes(ws),
                            _stream(stream))
    _check("kv_recompact", st)


def kv_compact(shape: KvShape, k, v, scores, crit_norm, crit_alpha_num: int, crit_alpha_den: int,
               crit_eps: float, head_budget, reserve: int, kept_idx, cu_off, lens, k_flat, v_flat,
               flat_capacity_rows: int, ws, stream=None) -> None:
    st = lib().kv_compact(ctypes.byref(shape), _ptr(k), _ptr(v), _ptr(scores), _ptr(crit_norm),
                          crit_alpha_num, crit_alpha_den, crit_eps, _ptr(head_budget), reserve,
                          _ptr(kept_idx), _ptr(cu_off), _ptr(lens), _ptr(k_flat), _ptr(v_flat),
                          flat_capacity_rows, _ptr(ws), _nbytes(ws), _stream(stream))
    _check("kv_compact", st)


def flat_decode_attn(shape: KvShape, q, k_new, v_new, k_flat, v_flat, cu_off, lens,
                     softmax_scale: float, out, ws, stream=None, flat_capacity_rows=None) -> None:
    cap = k_flat.shape[0] if flat_capacity_rows is None else flat_capacity_rows
    st = lib().flat_decode_attn(ctypes.byref(shape), _ptr(q), _ptr(k_new), _ptr(v_new),
                                _ptr(k_flat), _ptr(v_flat), _ptr(cu_off), _ptr(lens), cap,
                                softmax_scale, _ptr(out), _ptr(ws), _nbytes(ws), _stream(stream))
    _check("flat_decode_attn", st)


def flat_decode_attn_noalloc(shape: KvShape, q, k_new, v_new, k_flat, v_flat, cu_off, lens,
                             softmax_scale: float, out, stream=None,
                             flat_capacity_rows=None) -> None:
    """flat_decode_attn without a workspace: the library's fixed device scratch is used."""
    cap = k_flat.shape[0] if flat_capacity_rows is None else flat_capacity_rows
    st = lib().flat_decode_attn_noalloc(ctypes.byref(shape), _ptr(q), _ptr(k_new), _ptr(v_new),
                                        _ptr(k_flat), _ptr(v_flat), _ptr(cu_off), _ptr(lens), cap,
                                        softmax_scale, _ptr(out), _stream(stream))
    _check("flat_decode_attn_noalloc", st)


def kv_check_device_status(ws, stream=None) -> int:
    """Returns 0, or the first device check code recorded in `ws` (and clears it)."""
    info = _u32(0)
    st = lib().kv_check_device_status(_ptr(ws), _stream(stream), ctypes.byref(info))
    if st == KV_ERR_DEVICE_CHECK:
        return int(info.value)
    _check("kv_check_device_status", st)
    return 0


def kv_kernel_launches() -> int:
    """Kernels launched by the library in this process so far."""
    return int(lib().kv_kernel_launches())
