"""Batched attention between a ragged query tensor and a paged KV cache
(CSR page table) on NVIDIA GB300, behind a plan/run C ABI (``libpka.so``).

``_pka`` mirrors the C entry points one to one; ``BatchAttention`` below only
owns the workspaces those calls need (device int workspace, pinned staging
buffer, device float workspace) and forwards to them.
"""
from __future__ import annotations

import torch

from . import _pka
from ._pka import (PKA_HND, PKA_KV_BF16, PKA_KV_FP8_E4M3, PKA_MASK_CAUSAL,  # noqa
                   PKA_MASK_CUSTOM, PKA_MASK_NONE, PKA_NHD,
                   PKA_SPLIT_AUTO, PKA_SPLIT_FIXED, PKA_SPLIT_OFF, PkaError, make_params,
                   pka_append_paged_kv_cache, pka_get_device_error, pka_last_error, pka_merge_states,
                   pka_packbits, pka_plan, pka_plan_cascade, pka_plan_create, pka_plan_destroy,
                   pka_plan_get_info,
                   pka_plan_wait, pka_run, pka_run_static_scratch, pka_status_str, pka_validate, pka_version,
                   pka_check_indices, pka_selftest_bounded_wait)

__all__ = ["BatchAttention", "make_params", "PkaError"] + [n for n in _pka.EXPORTED]

_WORKSPACE = 4


class BatchAttention:
    """Plan once per batch, run once per layer (the pages' plan/run contract)."""

    def __init__(self, device="cuda", int_ws_bytes=1 << 20, float_ws_bytes=16 << 20):
        _pka.lib()
        self.device = torch.device(device)
        self.handle = pka_plan_create()
        self.int_ws = torch.empty(int_ws_bytes, dtype=torch.uint8, device=self.device)
        self.pinned = torch.empty(int_ws_bytes, dtype=torch.uint8, pin_memory=True)
        self.float_ws = torch.empty(float_ws_bytes, dtype=torch.uint8, device=self.device)
        self.params = None
        self.info = None
        self._params_key = None
        self._params_cached = None

    def __del__(self):
        try:
            pka_plan_destroy(self.handle)
        except Exception:
            pass

    def plan(self, qo_indptr, kv_indptr, last_page_len, *, num_qo_heads, num_kv_heads, head_dim,
             page_size=1, layout="NHD", mask_mode="causal", sm_scale=0.0, kv_ragged=False,
             split_mode="auto", fixed_split_pages=1, num_sms=0, graph_max_batch=0,
             graph_max_qo_rows=0, graph_max_kv_tokens=0, kv_dtype="bf16", k_scale=1.0,
             v_scale=1.0, decode_on_tensor_cores=False, stream=None):
        key = (num_qo_heads, num_kv_heads, head_dim, page_size, layout, mask_mode, sm_scale,
               kv_ragged, split_mode, fixed_split_pages, num_sms, graph_max_batch,
               graph_max_qo_rows, graph_max_kv_tokens, kv_dtype, k_scale, v_scale,
               decode_on_tensor_cores)
        if key != self._params_key:  # the same parameters plan after plan: build them once
            self._params_cached = make_params(*key)
            self._params_key = key
        params = self._params_cached
        return self._plan(params, "pka_plan", lambda: pka_plan(
            self.handle, params, qo_indptr, kv_indptr, last_page_len, self.int_ws, self.pinned,
            stream, check=False))

    def plan_cascade(self, levels, *, num_qo_heads, num_kv_heads, head_dim, page_size=1,
                     layout="NHD", mask_mode="causal", sm_scale=0.0, split_mode="auto",
                     fixed_split_pages=1, num_sms=0, kv_dtype="bf16", k_scale=1.0, v_scale=1.0,
                     stream=None):
        """Multi-level cascade: ``levels`` lists, root first, each level's
        (qo_indptr, kv_indptr, last_page_len); run() then takes the levels'
        page ids concatenated in level order as kv_indices."""
        params = make_params(num_qo_heads, num_kv_heads, head_dim, page_size, layout, mask_mode,
                             sm_scale, False, split_mode, fixed_split_pages, num_sms,
                             kv_dtype=kv_dtype, k_scale=k_scale, v_scale=v_scale)
        return self._plan(params, "pka_plan_cascade", lambda: pka_plan_cascade(
            self.handle, params, levels, self.int_ws, self.pinned, stream, check=False))

    def _plan(self, params, where, call):
        s = call()
        if s == _WORKSPACE:
            info = pka_plan_get_info(self.handle)
            pka_plan_wait(self.handle)
            if info.int_ws_bytes <= min(self.int_ws.numel(), self.pinned.numel()):
                # not a buffer size: the batch exceeds the graph-mode capacities
                raise PkaError(s, where + ": " + pka_last_error())
            n = max(int(info.int_ws_bytes), self.int_ws.numel())
            self.int_ws = torch.empty(n, dtype=torch.uint8, device=self.device)
            self.pinned = torch.empty(n, dtype=torch.uint8, pin_memory=True)
            s = call()
        if s != 0:
            raise PkaError(s, where)
        self.params = params
        self.info = pka_plan_get_info(self.handle)
        if self.info.float_ws_bytes > self.float_ws.numel():
            self.float_ws = torch.empty(int(self.info.float_ws_bytes), dtype=torch.uint8,
                                        device=self.device)
        return self.info

    def run(self, q, k, v, kv_indices=None, packed_mask=None, *, page_stride=None, out=None,
            lse=None, return_lse=True, stream=None):
        if self.params is None:
            raise RuntimeError("plan() before run()")
        if out is None:
            out = torch.empty_like(q)
        if lse is None and return_lse:
            lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
        if page_stride is None:
            page_stride = k.stride(0) if not self.params.kv_ragged else 0
        pka_run(self.handle, self.params, q, k, v, page_stride, kv_indices, packed_mask, out, lse,
                self.float_ws, stream)
        return out, lse
