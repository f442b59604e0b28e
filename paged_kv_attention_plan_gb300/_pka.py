"""ctypes binding of libpka.so — argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but check types, pass raw pointers and raise on a non-zero status;
all work happens in the library's host planner and CUDA kernels.  The
binding refuses to run when libpka.so is missing (there is no fallback).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpka.so")

PKA_NHD, PKA_HND = 0, 1
PKA_MASK_NONE, PKA_MASK_CAUSAL, PKA_MASK_CUSTOM = 0, 1, 2
PKA_SPLIT_OFF, PKA_SPLIT_AUTO, PKA_SPLIT_FIXED = 0, 1, 2
PKA_KV_BF16, PKA_KV_FP8_E4M3 = 0, 1

STATUS = {0: "PKA_OK", 1: "PKA_ERR_INVALID_ARG", 2: "PKA_ERR_METADATA", 3: "PKA_ERR_UNSUPPORTED",
          4: "PKA_ERR_WORKSPACE", 5: "PKA_ERR_STALE_PLAN", 6: "PKA_ERR_CUDA",
          7: "PKA_ERR_DEVICE_TIMEOUT"}

EXPORTED = ["pka_status_str", "pka_version", "pka_validate", "pka_plan_create",
            "pka_plan_destroy", "pka_plan", "pka_plan_get_info", "pka_plan_wait", "pka_run",
            "pka_append_paged_kv_cache", "pka_merge_states", "pka_packbits",
            "pka_get_device_error", "pka_last_error", "pka_run_static_scratch",
            "pka_plan_cascade", "pka_selftest_bounded_wait", "pka_check_indices"]


class pka_params(ctypes.Structure):
    _fields_ = [("num_qo_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("layout", ctypes.c_int32), ("mask_mode", ctypes.c_int32),
                ("sm_scale", ctypes.c_float), ("kv_ragged", ctypes.c_int32),
                ("split_mode", ctypes.c_int32), ("fixed_split_pages", ctypes.c_int32),
                ("num_sms", ctypes.c_int32), ("graph_max_batch", ctypes.c_int32),
                ("graph_max_qo_rows", ctypes.c_int32), ("graph_max_kv_tokens", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float), ("decode_on_tensor_cores", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 1)]


class pka_plan_info(ctypes.Structure):
    _fields_ = [("int_ws_bytes", ctypes.c_uint64), ("float_ws_bytes", ctypes.c_uint64),
                ("num_requests", ctypes.c_int32), ("nnz_qo", ctypes.c_int32),
                ("total_kv", ctypes.c_int64), ("num_decode_ctas", ctypes.c_int32),
                ("num_decode_items", ctypes.c_int32), ("num_prefill_ctas", ctypes.c_int32),
                ("num_prefill_items", ctypes.c_int32), ("num_merge_tasks", ctypes.c_int32),
                ("num_partial_records", ctypes.c_int32),
                ("decode_chunk_tokens", ctypes.c_int32), ("num_decode_joins", ctypes.c_int32),
                ("kv_scratch_rows", ctypes.c_int32), ("reserved", ctypes.c_int32 * 3)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_ if f != "reserved"}


class PkaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status == 6:
            try:
                detail = " — " + lib().pka_last_error().decode()
            except Exception:
                pass
        super().__init__(f"{where}: {STATUS.get(status, status)} ({_str(status)}){detail}")


_lib = None


def lib():
    """Load libpka.so once; raise if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpka.so is missing ({LIB_PATH}); build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        P = ctypes.POINTER
        L.pka_status_str.restype = ctypes.c_char_p
        L.pka_status_str.argtypes = [ctypes.c_int]
        L.pka_version.argtypes = [P(i32), P(i32)]
        L.pka_validate.argtypes = [P(pka_params), i32, vp, vp, vp]
        L.pka_plan_create.argtypes = [P(vp)]
        L.pka_plan_destroy.argtypes = [vp]
        L.pka_plan_destroy.restype = None
        L.pka_plan.argtypes = [vp, P(pka_params), i32, vp, vp, vp, vp, sz, vp, sz, vp]
        L.pka_plan_cascade.argtypes = [vp, P(pka_params), i32, vp, vp, vp, vp, vp, sz, vp, sz,
                                       vp]
        L.pka_plan_get_info.argtypes = [vp, P(pka_plan_info)]
        L.pka_plan_wait.argtypes = [vp]
        L.pka_run.argtypes = [vp, P(pka_params), vp, vp, vp, i64, vp, vp, vp, vp, vp, sz, vp]
        L.pka_run_static_scratch.argtypes = [vp, P(pka_params), vp, vp, vp, i64, vp, vp, vp, vp,
                                             vp]
        L.pka_append_paged_kv_cache.argtypes = [P(pka_params), i32, vp, vp, vp, i64, vp, vp, vp,
                                                vp, vp, i64, vp]
        L.pka_merge_states.argtypes = [vp, vp, vp, i32, i32, i32, vp, vp, vp]
        L.pka_packbits.argtypes = [vp, i64, vp, vp]
        L.pka_get_device_error.argtypes = [P(i32), vp]
        L.pka_selftest_bounded_wait.argtypes = [i32, i32, vp]
        L.pka_check_indices.argtypes = [P(pka_params), i32, vp, vp, vp, i64, vp, i64, P(i64)]
        L.pka_last_error.argtypes = []
        L.pka_last_error.restype = ctypes.c_char_p
        for name in EXPORTED:
            if name not in ("pka_status_str", "pka_plan_destroy", "pka_last_error"):
                getattr(L, name).restype = ctypes.c_int
        _lib = L
    return _lib


def _str(status: int) -> str:
    try:
        return lib().pka_status_str(status).decode()
    except Exception:  # library missing while formatting an error
        return "?"


def _check(status: int, where: str):
    if status != 0:
        raise PkaError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return t.data_ptr()
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    raise TypeError(f"unsupported buffer type {type(t)}")


def _int32_host(a, name):
    """Host int32 metadata (numpy or CPU torch); int64 is rejected, not cast."""
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        if a.dtype != torch.int32:
            raise TypeError(f"{name} must be int32, got {a.dtype}")
        if a.is_cuda:
            raise TypeError(f"{name} must be a host tensor for planning")
        return np.ascontiguousarray(a.numpy())
    a = np.asarray(a)
    if a.dtype != np.int32:
        raise TypeError(f"{name} must be int32, got {a.dtype}")
    return np.ascontiguousarray(a)


def _dev(t, name, dtype):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _dev_pool(t, name, params=None):
    """K/V pool: the last three dims contiguous; pages may be strided (5-D view).
    bf16, or uint8 e4m3 codes when the params say so."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    want = (torch.uint8 if params is not None and params.kv_dtype == PKA_KV_FP8_E4M3
            else torch.bfloat16)
    if t.dtype != want:
        raise TypeError(f"{name} must be {want}, got {t.dtype}")
    if t.dim() >= 3 and (t.stride(-1) != 1 or t.stride(-2) != t.shape[-1]
                         or t.stride(-3) != t.shape[-1] * t.shape[-2]):
        raise ValueError(f"{name}: the last three dims must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def make_params(num_qo_heads, num_kv_heads, head_dim, page_size=1, layout="NHD",
                mask_mode="causal", sm_scale=0.0, kv_ragged=False, split_mode="auto",
                fixed_split_pages=1, num_sms=0, graph_max_batch=0, graph_max_qo_rows=0,
                graph_max_kv_tokens=0, kv_dtype="bf16", k_scale=1.0,
                v_scale=1.0, decode_on_tensor_cores=False) -> pka_params:
    p = pka_params()
    p.num_qo_heads, p.num_kv_heads, p.head_dim = num_qo_heads, num_kv_heads, head_dim
    p.page_size = page_size
    p.layout = {"NHD": PKA_NHD, "HND": PKA_HND}[layout] if isinstance(layout, str) else layout
    p.mask_mode = ({"none": PKA_MASK_NONE, "causal": PKA_MASK_CAUSAL, "custom": PKA_MASK_CUSTOM}
                   [mask_mode] if isinstance(mask_mode, str) else mask_mode)
    p.sm_scale = sm_scale
    p.kv_ragged = int(bool(kv_ragged))
    p.split_mode = ({"off": PKA_SPLIT_OFF, "auto": PKA_SPLIT_AUTO, "fixed": PKA_SPLIT_FIXED}
                    [split_mode] if isinstance(split_mode, str) else split_mode)
    p.fixed_split_pages = fixed_split_pages
    p.num_sms = num_sms
    p.graph_max_batch = graph_max_batch
    p.graph_max_qo_rows = graph_max_qo_rows
    p.graph_max_kv_tokens = graph_max_kv_tokens
    p.kv_dtype = ({"bf16": PKA_KV_BF16, "e4m3": PKA_KV_FP8_E4M3}[kv_dtype]
                  if isinstance(kv_dtype, str) else kv_dtype)
    p.k_scale, p.v_scale = k_scale, v_scale
    p.decode_on_tensor_cores = int(bool(decode_on_tensor_cores))
    return p


# ---------------------------------------------------------------------------
# The C entry points, one Python function each.
# ---------------------------------------------------------------------------

def pka_status_str(status: int) -> str:
    return _str(status)


def pka_version():
    a, b = ctypes.c_int32(), ctypes.c_int32()
    _check(lib().pka_version(ctypes.byref(a), ctypes.byref(b)), "pka_version")
    return a.value, b.value


def pka_validate(params, qo_indptr, kv_indptr, last_page_len) -> int:
    kv = _int32_host(kv_indptr, "kv_indptr")
    qo = _int32_host(qo_indptr, "qo_indptr")
    last = _int32_host(last_page_len, "last_page_len")
    return lib().pka_validate(ctypes.byref(params), len(kv) - 1, _ptr(qo), _ptr(kv), _ptr(last))


def pka_plan_create():
    h = ctypes.c_void_p()
    _check(lib().pka_plan_create(ctypes.byref(h)), "pka_plan_create")
    return h


def pka_plan_destroy(handle):
    if handle:
        lib().pka_plan_destroy(handle)


def pka_plan(handle, params, qo_indptr, kv_indptr, last_page_len, int_ws, pinned,
             stream=None, check=True) -> int:
    kv = _int32_host(kv_indptr, "kv_indptr")
    qo = _int32_host(qo_indptr, "qo_indptr")
    last = _int32_host(last_page_len, "last_page_len")
    ws_ptr = _ptr(int_ws) if int_ws is not None else None
    ws_bytes = int_ws.numel() * int_ws.element_size() if int_ws is not None else 0
    pin_bytes = (pinned.numel() * pinned.element_size() if isinstance(pinned, torch.Tensor)
                 else pinned.nbytes)
    st = _stream(stream) if int_ws is not None else None
    s = lib().pka_plan(handle, ctypes.byref(params), len(kv) - 1, _ptr(qo), _ptr(kv), _ptr(last),
                       ws_ptr, ws_bytes, _ptr(pinned), pin_bytes, st)
    if check:
        _check(s, "pka_plan")
    return s


def pka_plan_cascade(handle, params, levels, int_ws, pinned, stream=None, check=True) -> int:
    """``levels``: list, root first, of (qo_indptr, kv_indptr, last_page_len) host int32."""
    arrs = [tuple(_int32_host(a, n) for a, n in zip(lv, ("qo_indptr", "kv_indptr",
                                                          "last_page_len")))
            for lv in levels]
    n = len(arrs)
    nodes = np.asarray([len(a[1]) - 1 for a in arrs], dtype=np.int32)
    ptrs = [(ctypes.c_void_p * max(n, 1))(*[_ptr(a[i]) for a in arrs]) for i in range(3)]
    ws_ptr = _ptr(int_ws) if int_ws is not None else None
    ws_bytes = int_ws.numel() * int_ws.element_size() if int_ws is not None else 0
    pin_bytes = (pinned.numel() * pinned.element_size() if isinstance(pinned, torch.Tensor)
                 else pinned.nbytes)
    st = _stream(stream) if int_ws is not None else None
    s = lib().pka_plan_cascade(handle, ctypes.byref(params), n, _ptr(nodes),
                               ctypes.cast(ptrs[0], ctypes.c_void_p),
                               ctypes.cast(ptrs[1], ctypes.c_void_p),
                               ctypes.cast(ptrs[2], ctypes.c_void_p), ws_ptr, ws_bytes,
                               _ptr(pinned), pin_bytes, st)
    if check:
        _check(s, "pka_plan_cascade")
    return s


def pka_plan_get_info(handle) -> pka_plan_info:
    info = pka_plan_info()
    _check(lib().pka_plan_get_info(handle, ctypes.byref(info)), "pka_plan_get_info")
    return info


def pka_plan_wait(handle):
    _check(lib().pka_plan_wait(handle), "pka_plan_wait")


def pka_run(handle, params, q, k, v, page_stride, kv_indices, packed_mask, o, lse, float_ws,
            stream=None, check=True) -> int:
    bf16 = torch.bfloat16
    fws = float_ws.numel() * float_ws.element_size() if float_ws is not None else 0
    s = lib().pka_run(handle, ctypes.byref(params), _dev(q, "q", bf16),
                      _dev_pool(k, "k", params), _dev_pool(v, "v", params), int(page_stride),
                      _dev(kv_indices, "kv_indices", torch.int32),
                      _dev(packed_mask, "packed_mask", torch.uint8), _dev(o, "o", bf16),
                      _dev(lse, "lse", torch.float32), _ptr(float_ws), fws, _stream(stream))
    if check:
        _check(s, "pka_run")
    return s


def pka_run_static_scratch(handle, params, q, k, v, page_stride, kv_indices, packed_mask, o,
                           lse, stream=None, check=True) -> int:
    """pka_run with the split-KV scratch in the library's static device array
    (no workspace from the caller; see include/pka.h)."""
    bf16 = torch.bfloat16
    s = lib().pka_run_static_scratch(
        handle, ctypes.byref(params), _dev(q, "q", bf16), _dev_pool(k, "k", params),
        _dev_pool(v, "v", params),
        int(page_stride), _dev(kv_indices, "kv_indices", torch.int32),
        _dev(packed_mask, "packed_mask", torch.uint8), _dev(o, "o", bf16),
        _dev(lse, "lse", torch.float32), _stream(stream))
    if check:
        _check(s, "pka_run_static_scratch")
    return s


def pka_append_paged_kv_cache(params, k_new, v_new, append_indptr, kv_indptr, kv_indices,
                              last_page_len, k, v, page_stride, stream=None, check=True) -> int:
    bf16, i32 = torch.bfloat16, torch.int32
    s = lib().pka_append_paged_kv_cache(
        ctypes.byref(params), append_indptr.numel() - 1, _dev(k_new, "k_new", bf16),
        _dev(v_new, "v_new", bf16), _dev(append_indptr, "append_indptr", i32), k_new.shape[0],
        _dev(kv_indptr, "kv_indptr", i32), _dev(kv_indices, "kv_indices", i32),
        _dev(last_page_len, "last_page_len", i32), _dev_pool(k, "k", params),
        _dev_pool(v, "v", params),
        int(page_stride),
        _stream(stream))
    if check:
        _check(s, "pka_append_paged_kv_cache")
    return s


def pka_merge_states(v, s, indptr, v_out, s_out=None, stream=None):
    rows = indptr.numel() - 1
    _check(lib().pka_merge_states(_dev(v, "v", torch.float32), _dev(s, "s", torch.float32),
                                  _dev(indptr, "indptr", torch.int32), rows, v.shape[1],
                                  v.shape[2], _dev(v_out, "v_out", torch.bfloat16),
                                  _dev(s_out, "s_out", torch.float32), _stream(stream)),
           "pka_merge_states")


def pka_packbits(bools, out, stream=None):
    _check(lib().pka_packbits(_dev(bools, "bools", torch.uint8), bools.numel(),
                              _dev(out, "out", torch.uint8), _stream(stream)), "pka_packbits")


def pka_last_error() -> str:
    return lib().pka_last_error().decode()


def pka_get_device_error(stream=None) -> int:
    code = ctypes.c_int32()
    _check(lib().pka_get_device_error(ctypes.byref(code), _stream(stream)), "pka_get_device_error")
    return code.value


def pka_selftest_bounded_wait(arrive: bool, polls: int, stream=None):
    _check(lib().pka_selftest_bounded_wait(1 if arrive else 0, int(polls), _stream(stream)),
           "pka_selftest_bounded_wait")


def pka_check_indices(params, kv_indptr, kv_indices, last_page_len, num_pool_pages,
                      append_indptr=None):
    """Host check of a page table; returns (status, bad_index) without raising."""
    kv = _int32_host(kv_indptr, "kv_indptr")
    idx = _int32_host(kv_indices, "kv_indices")
    last = _int32_host(last_page_len, "last_page_len")
    app = _int32_host(append_indptr, "append_indptr")
    bad = ctypes.c_int64(-2)
    s = lib().pka_check_indices(ctypes.byref(params), len(kv) - 1, _ptr(app), _ptr(kv),
                                _ptr(idx), len(idx), _ptr(last), int(num_pool_pages),
                                ctypes.byref(bad))
    return s, bad.value
