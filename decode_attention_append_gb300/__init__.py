"""GB300 (sm_103a) paged KV append + mixed-batch paged attention.

A thin ctypes binding over the C ABI of ``libdaa.so`` (declared in
``include/daa.h``).  It only marshals torch tensors into pointers and sizes:
every step of the computation runs in the library's CUDA kernels.  There is no
CPU or PyTorch fallback; if the library is missing the calls raise.

Entry points (same names as the C ABI, without the ``daa_`` prefix):

* ``kv_append(k_new, v_new, kv_pages, append_indptr, page_indices, kv_indptr,
  last_page_len)`` -- write each new token's K/V into its page slot.
* ``batch_attention(q, kv_pages, qo_indptr, kv_indptr, page_indices,
  last_page_len, causal, sm_scale, ...)`` -- attention for a batch mixing
  chunked-prefill requests (qo_len > 1, causal with the cache offset) and decode
  requests (qo_len = 1).
* ``batch_attention_tree(..., tree_mask, ...)`` -- the same attention with
  draft-tree masks over each request's new tokens (speculative-decoding
  verification of a tree of draft tokens).
* ``BatchAttention`` -- plans once from host copies of the page table and owns
  the workspace, for repeated calls over the same batch shape.

Tensors: bf16 ``q [nnz_qo, Hq, d]``, ``k_new/v_new [nnz_new, Hkv, d]``, page
pool ``kv_pages [num_pages, 2, Hkv, page_size, d]`` (K then V, HND inside a
page), int32 CSR arrays on the same CUDA device.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libdaa.so")
_lib = None
_lock = threading.Lock()

DAA_OK = 0
STATUS = {0: "ok", -1: "invalid argument", -2: "shape", -3: "page range", -4: "unsupported",
          -5: "CUDA error", -6: "workspace", -7: "alignment"}
KERNEL_NAMES = {1: "kv_append", 2: "decode_splitkv", 3: "softmax_merge", 4: "prefill_tc", 5: "decode_tc",
                6: "short_tc"}


class DaaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)} ({status})")
        self.status = status


class _Dims(ctypes.Structure):
    _fields_ = [("num_qo_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int64)]


class StepLayout(ctypes.Structure):
    """daa_step_layout: byte offsets of a host step's sections in its packed buffer."""
    _fields_ = [(n, ctypes.c_size_t) for n in ("qo_indptr", "kv_indptr", "page_indices", "last_page_len",
                                               "q", "k_new", "v_new", "total")]


class StepStreams(ctypes.Structure):
    """daa_step_streams: the streams and events of one host step."""
    _fields_ = [(n, ctypes.c_void_p) for n in ("upload_stream", "compute_stream", "download_stream",
                                               "uploaded", "computed", "downloaded", "inputs_free",
                                               "out_free")]


class PlanInfo(ctypes.Structure):
    """daa_plan_info: the record of a plan uploaded by ``batch_attention_plan``."""
    _fields_ = [("words", ctypes.c_int64 * 24)]


def library_path() -> str:
    return _LIB_PATH


def load_library():
    """Load libdaa.so (built by ``build.build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise ImportError(f"libdaa.so not built at {_LIB_PATH}; run decode_attention_append_gb300.build.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        vp, i32, i64, f32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
        lib.daa_status_string.restype = ctypes.c_char_p
        lib.daa_status_string.argtypes = [i32]
        lib.daa_version.restype = i32
        lib.daa_kv_append.restype = i32
        lib.daa_kv_append.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, _Dims, vp]
        lib.daa_batch_attention_workspace_size.restype = sz
        lib.daa_batch_attention_workspace_size.argtypes = [vp, vp, vp, i32, _Dims, ctypes.POINTER(i32)]
        lib.daa_batch_attention.restype = i32
        lib.daa_batch_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32, vp, vp,
                                            vp, sz, _Dims, vp]
        lib.daa_append_attention.restype = i32
        lib.daa_append_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32,
                                             vp, vp, vp, sz, _Dims, vp]
        lib.daa_batch_attention_tree.restype = i32
        lib.daa_batch_attention_tree.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, i32, f32,
                                                 vp, vp, vp, sz, _Dims, vp]
        lib.daa_batch_attention_noalloc.restype = i32
        lib.daa_batch_attention_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, f32,
                                                    vp, vp, _Dims, vp]
        lib.daa_batch_attention_shared_prefix_workspace_size.restype = sz
        lib.daa_batch_attention_shared_prefix_workspace_size.argtypes = [
            vp, vp, vp, i32, vp, vp, i32, _Dims, ctypes.POINTER(i32)]
        lib.daa_batch_attention_shared_prefix.restype = i32
        lib.daa_batch_attention_shared_prefix.argtypes = [
            vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, f32, vp, vp, vp, sz, _Dims, vp]
        lib.daa_append_attention_shared_prefix.restype = i32
        lib.daa_append_attention_shared_prefix.argtypes = [
            vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32, i32, f32, vp, vp, vp, sz,
            _Dims, vp]
        pinfo = ctypes.POINTER(PlanInfo)
        lib.daa_batch_attention_plan.restype = i32
        lib.daa_batch_attention_plan.argtypes = [vp, vp, vp, i32, vp, vp, i32, _Dims, vp, sz, pinfo, vp]
        lib.daa_batch_attention_run.restype = i32
        lib.daa_batch_attention_run.argtypes = [vp, vp, vp, vp, vp, vp, pinfo, i32, f32, vp, vp, vp, sz,
                                                _Dims, vp]
        lib.daa_append_attention_run.restype = i32
        lib.daa_append_attention_run.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, pinfo, i32, f32, vp, vp,
                                                 vp, sz, _Dims, vp]
        lib.daa_append_attention_host.restype = i32
        lib.daa_append_attention_host.argtypes = [vp, vp, ctypes.POINTER(StepLayout), i32, i32, f32, vp, vp,
                                                  vp, vp, sz, _Dims, ctypes.POINTER(StepStreams)]
        lib.daa_set_prefill_append_fusion.restype = i32
        lib.daa_set_prefill_append_fusion.argtypes = [i32]
        lib.daa_prefill_append_fusion.restype = i32
        lib.daa_prefill_append_fusion.argtypes = []
        lib.daa_selftest_bounded_wait.restype = i32
        lib.daa_selftest_bounded_wait.argtypes = [ctypes.POINTER(i32)]
        lib.daa_device_error.restype = i32
        lib.daa_device_error.argtypes = [ctypes.POINTER(i32), i32]
        lib.daa_trace_enable.restype = i32
        lib.daa_trace_enable.argtypes = [i32]
        lib.daa_trace_disable.restype = i32
        lib.daa_trace_read.restype = i32
        lib.daa_trace_read.argtypes = [ctypes.POINTER(i32), ctypes.POINTER(f32), i32]
        _lib = lib
        return lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        return ctypes.c_void_p(t.data_ptr())
    if isinstance(t, np.ndarray):
        return t.ctypes.data_as(ctypes.c_void_p)
    raise TypeError(type(t))


def _host_i32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _dev_i32(t: torch.Tensor, name: str) -> torch.Tensor:
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.int32 and t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous int32 CUDA tensor")
    return t


def _dev_bf16(t: torch.Tensor, name: str) -> torch.Tensor:
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
        raise TypeError(f"{name} must be a contiguous bf16 CUDA tensor")
    return t


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dims(kv_pages: torch.Tensor, num_qo_heads: int) -> _Dims:
    if kv_pages.dim() != 5 or kv_pages.shape[1] != 2:
        raise ValueError("kv_pages must be [num_pages, 2, Hkv, page_size, head_dim]")
    n, _, hkv, p, d = kv_pages.shape
    return _Dims(num_qo_heads, hkv, d, p, n)


def _check(st: int, what: str):
    if st != DAA_OK:
        raise DaaError(st, what)


def kv_append(k_new, v_new, kv_pages, append_indptr, page_indices, kv_indptr, last_page_len,
              stream=None) -> None:
    """Append new tokens' K/V into their pages (asynchronous on ``stream``)."""
    lib = load_library()
    _dev_bf16(k_new, "k_new"), _dev_bf16(v_new, "v_new"), _dev_bf16(kv_pages, "kv_pages")
    for n, t in (("append_indptr", append_indptr), ("page_indices", page_indices),
                 ("kv_indptr", kv_indptr), ("last_page_len", last_page_len)):
        _dev_i32(t, n)
    dims = _dims(kv_pages, kv_pages.shape[2])
    batch = append_indptr.numel() - 1
    _check(lib.daa_kv_append(_ptr(k_new), _ptr(v_new), _ptr(kv_pages), _ptr(append_indptr),
                             _ptr(page_indices), _ptr(kv_indptr), _ptr(last_page_len), batch,
                             k_new.shape[0], dims, _stream(stream)), "kv_append")


def batch_attention_workspace_size(h_qo_indptr, h_kv_indptr, h_last_page_len, num_qo_heads,
                                   num_kv_heads, head_dim, page_size, num_pages) -> int:
    lib = load_library()
    qo, kv, ll = _host_i32(h_qo_indptr), _host_i32(h_kv_indptr), _host_i32(h_last_page_len)
    st = ctypes.c_int32(0)
    n = lib.daa_batch_attention_workspace_size(_ptr(qo), _ptr(kv), _ptr(ll), len(qo) - 1,
                                               _Dims(num_qo_heads, num_kv_heads, head_dim,
                                                     page_size, num_pages), ctypes.byref(st))
    _check(st.value, "batch_attention_workspace_size")
    return int(n)


def _host_groups(prefix_groups):
    """(indptr, prefix_len) -> host int32 arrays and the group count."""
    ind, pl = (_host_i32(x) for x in prefix_groups)
    if len(ind) != len(pl) + 1:
        raise ValueError("prefix_groups: indptr must have one more entry than prefix_len")
    return ind, pl, len(pl)


def shared_prefix_workspace_size(h_qo_indptr, h_kv_indptr, h_last_page_len, prefix_groups,
                                 num_qo_heads, num_kv_heads, head_dim, page_size,
                                 num_pages) -> int:
    """Workspace bytes of ``batch_attention(..., prefix_groups=...)`` (and of
    ``append_attention`` with the same groups)."""
    lib = load_library()
    qo, kv, ll = _host_i32(h_qo_indptr), _host_i32(h_kv_indptr), _host_i32(h_last_page_len)
    gi, gl, ng = _host_groups(prefix_groups)
    st = ctypes.c_int32(0)
    n = lib.daa_batch_attention_shared_prefix_workspace_size(
        _ptr(qo), _ptr(kv), _ptr(ll), len(qo) - 1, _ptr(gi), _ptr(gl), ng,
        _Dims(num_qo_heads, num_kv_heads, head_dim, page_size, num_pages), ctypes.byref(st))
    _check(st.value, "shared_prefix_workspace_size")
    return int(n)


def _workspace_need(lib, hq, hk, hl, dims, groups, what):
    st = ctypes.c_int32(0)
    if groups is None:
        need = lib.daa_batch_attention_workspace_size(_ptr(hq), _ptr(hk), _ptr(hl), len(hq) - 1,
                                                      dims, ctypes.byref(st))
    else:
        gi, gl, ng = groups
        need = lib.daa_batch_attention_shared_prefix_workspace_size(
            _ptr(hq), _ptr(hk), _ptr(hl), len(hq) - 1, _ptr(gi), _ptr(gl), ng, dims,
            ctypes.byref(st))
    _check(st.value, what)
    return int(need)


def batch_attention(q, kv_pages, qo_indptr, kv_indptr, page_indices, last_page_len, causal=True,
                    sm_scale=None, out=None, lse=None, workspace=None, host_indptr=None,
                    stream=None, prefix_groups=None):
    """Mixed-batch paged attention.  Returns ``out`` (and fills ``lse`` if given).

    ``host_indptr`` = (h_qo_indptr, h_kv_indptr, h_last_page_len) host copies of
    the page table used for planning; when omitted they are copied from the
    device (a synchronisation).  ``workspace`` (uint8 CUDA tensor) is allocated
    by torch here when omitted; the library itself never allocates.

    ``prefix_groups`` = (indptr, prefix_len), host int arrays: group i is
    requests [indptr[i], indptr[i+1]) whose first prefix_len[i] keys sit in the
    same pages (a shared cached prefix).  The shared keys are then attended
    once for all the group's rows (``daa_batch_attention_shared_prefix``); the
    result is the same.
    """
    lib = load_library()
    _dev_bf16(q, "q"), _dev_bf16(kv_pages, "kv_pages")
    for n, t in (("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr), ("page_indices", page_indices),
                 ("last_page_len", last_page_len)):
        _dev_i32(t, n)
    Hq, d = q.shape[1], q.shape[2]
    dims = _dims(kv_pages, Hq)
    if sm_scale is None:
        sm_scale = 1.0 / float(d) ** 0.5
    if host_indptr is None:
        host_indptr = (qo_indptr, kv_indptr, last_page_len)
    hq, hk, hl = (_host_i32(x) for x in host_indptr)
    batch = len(hq) - 1
    if out is None:
        out = torch.empty_like(q)
    _dev_bf16(out, "out")
    if lse is not None and not (lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()):
        raise TypeError("lse must be a contiguous fp32 CUDA tensor")
    groups = None if prefix_groups is None else _host_groups(prefix_groups)
    need = _workspace_need(lib, hq, hk, hl, dims, groups, "batch_attention")
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if groups is None:
        st = lib.daa_batch_attention(_ptr(q), _ptr(kv_pages), _ptr(qo_indptr), _ptr(kv_indptr),
                                     _ptr(page_indices), _ptr(last_page_len), _ptr(hq), _ptr(hk),
                                     _ptr(hl), batch, int(bool(causal)), float(sm_scale), _ptr(out),
                                     _ptr(lse), _ptr(workspace), ws_bytes, dims, _stream(stream))
    else:
        gi, gl, ng = groups
        st = lib.daa_batch_attention_shared_prefix(
            _ptr(q), _ptr(kv_pages), _ptr(qo_indptr), _ptr(kv_indptr), _ptr(page_indices),
            _ptr(last_page_len), _ptr(hq), _ptr(hk), _ptr(hl), batch, _ptr(gi), _ptr(gl), ng,
            int(bool(causal)), float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
            dims, _stream(stream))
    _check(st, "batch_attention")
    return out


def batch_attention_tree(q, kv_pages, qo_indptr, kv_indptr, page_indices, last_page_len, tree_mask,
                         sm_scale=None, out=None, lse=None, workspace=None, host_indptr=None,
                         stream=None):
    """Causal mixed-batch attention in which new token i of a request sees,
    among its request's new tokens, itself and the earlier ones selected by
    its mask row (for a draft tree numbered parents-first: its ancestors).

    ``tree_mask``: contiguous int32 or uint32 CUDA tensor [nnz_qo, words], one
    row per query row; bit t (word t // 32, bit t % 32) selects new token t.
    Every request needs qo_len <= 32 * words.  Other arguments as
    ``batch_attention``."""
    lib = load_library()
    _dev_bf16(q, "q"), _dev_bf16(kv_pages, "kv_pages")
    for n, t in (("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr), ("page_indices", page_indices),
                 ("last_page_len", last_page_len)):
        _dev_i32(t, n)
    if not (isinstance(tree_mask, torch.Tensor) and tree_mask.is_cuda and tree_mask.dim() == 2
            and tree_mask.element_size() == 4 and tree_mask.is_contiguous()
            and not tree_mask.is_floating_point() and tree_mask.shape[0] == q.shape[0]):
        raise TypeError("tree_mask must be a contiguous [nnz_qo, words] int32/uint32 CUDA tensor")
    Hq, d = q.shape[1], q.shape[2]
    dims = _dims(kv_pages, Hq)
    if sm_scale is None:
        sm_scale = 1.0 / float(d) ** 0.5
    if host_indptr is None:
        host_indptr = (qo_indptr, kv_indptr, last_page_len)
    hq, hk, hl = (_host_i32(x) for x in host_indptr)
    batch = len(hq) - 1
    if out is None:
        out = torch.empty_like(q)
    _dev_bf16(out, "out")
    if lse is not None and not (lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()):
        raise TypeError("lse must be a contiguous fp32 CUDA tensor")
    if workspace is None:
        st = ctypes.c_int32(0)
        need = lib.daa_batch_attention_workspace_size(_ptr(hq), _ptr(hk), _ptr(hl), batch, dims,
                                                      ctypes.byref(st))
        _check(st.value, "batch_attention_tree")
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.daa_batch_attention_tree(_ptr(q), _ptr(kv_pages), _ptr(qo_indptr), _ptr(kv_indptr),
                                        _ptr(page_indices), _ptr(last_page_len), _ptr(hq), _ptr(hk),
                                        _ptr(hl), batch, _ptr(tree_mask), int(tree_mask.shape[1]),
                                        float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                        ws_bytes, dims, _stream(stream)),
           "batch_attention_tree")
    return out


def append_attention(k_new, v_new, q, kv_pages, qo_indptr, kv_indptr, page_indices, last_page_len,
                     causal=True, sm_scale=None, out=None, lse=None, workspace=None,
                     host_indptr=None, stream=None, prefix_groups=None):
    """``kv_append`` of this step's new K/V (rows laid out like ``q``) followed
    by ``batch_attention``, in one call: same results, with the attention
    kernels launched behind the append so that the work that does not read the
    appended rows overlaps it.  Arguments as ``batch_attention`` (including
    ``prefix_groups``)."""
    lib = load_library()
    _dev_bf16(k_new, "k_new"), _dev_bf16(v_new, "v_new")
    _dev_bf16(q, "q"), _dev_bf16(kv_pages, "kv_pages")
    for n, t in (("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr), ("page_indices", page_indices),
                 ("last_page_len", last_page_len)):
        _dev_i32(t, n)
    Hq, d = q.shape[1], q.shape[2]
    dims = _dims(kv_pages, Hq)
    if k_new.shape != (q.shape[0], dims.num_kv_heads, d) or v_new.shape != k_new.shape:
        raise ValueError("k_new and v_new must be [nnz_qo, Hkv, head_dim]")
    if sm_scale is None:
        sm_scale = 1.0 / float(d) ** 0.5
    if host_indptr is None:
        host_indptr = (qo_indptr, kv_indptr, last_page_len)
    hq, hk, hl = (_host_i32(x) for x in host_indptr)
    batch = len(hq) - 1
    if out is None:
        out = torch.empty_like(q)
    _dev_bf16(out, "out")
    if lse is not None and not (lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()):
        raise TypeError("lse must be a contiguous fp32 CUDA tensor")
    groups = None if prefix_groups is None else _host_groups(prefix_groups)
    if workspace is None:
        need = _workspace_need(lib, hq, hk, hl, dims, groups, "append_attention")
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if groups is None:
        st = lib.daa_append_attention(_ptr(k_new), _ptr(v_new), _ptr(q), _ptr(kv_pages),
                                      _ptr(qo_indptr), _ptr(kv_indptr), _ptr(page_indices),
                                      _ptr(last_page_len), _ptr(hq), _ptr(hk), _ptr(hl), batch,
                                      int(bool(causal)), float(sm_scale), _ptr(out), _ptr(lse),
                                      _ptr(workspace), ws_bytes, dims, _stream(stream))
    else:
        gi, gl, ng = groups
        st = lib.daa_append_attention_shared_prefix(
            _ptr(k_new), _ptr(v_new), _ptr(q), _ptr(kv_pages), _ptr(qo_indptr), _ptr(kv_indptr),
            _ptr(page_indices), _ptr(last_page_len), _ptr(hq), _ptr(hk), _ptr(hl), batch,
            _ptr(gi), _ptr(gl), ng, int(bool(causal)), float(sm_scale), _ptr(out), _ptr(lse),
            _ptr(workspace), ws_bytes, dims, _stream(stream))
    _check(st, "append_attention")
    return out


def batch_attention_noalloc(q, kv_pages, qo_indptr, kv_indptr, page_indices, last_page_len,
                            host_indptr, causal=True, sm_scale=None, out=None, lse=None,
                            stream=None):
    """``batch_attention`` without a workspace: the library's fixed device
    scratch array is used instead (see daa_batch_attention_noalloc in daa.h for
    its size limit and for why calls must not overlap on the GPU)."""
    lib = load_library()
    _dev_bf16(q, "q"), _dev_bf16(kv_pages, "kv_pages")
    for n, t in (("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr), ("page_indices", page_indices),
                 ("last_page_len", last_page_len)):
        _dev_i32(t, n)
    if q.dim() != 3:
        raise ValueError("q must be [nnz_qo, Hq, head_dim]")
    Hq, d = q.shape[1], q.shape[2]
    dims = _dims(kv_pages, Hq)
    if sm_scale is None:
        sm_scale = 1.0 / float(d) ** 0.5
    hq, hk, hl = (_host_i32(x) for x in host_indptr)
    if out is None:
        out = torch.empty_like(q)
    _dev_bf16(out, "out")
    if out.shape != q.shape:
        raise ValueError("out must have the shape of q")
    if lse is not None:
        if not (isinstance(lse, torch.Tensor) and lse.is_cuda and lse.dtype == torch.float32
                and lse.is_contiguous()):
            raise TypeError("lse must be a contiguous fp32 CUDA tensor")
        if tuple(lse.shape) != (q.shape[0], Hq):
            raise ValueError("lse must be [nnz_qo, Hq]")
    _check(lib.daa_batch_attention_noalloc(_ptr(q), _ptr(kv_pages), _ptr(qo_indptr), _ptr(kv_indptr),
                                           _ptr(page_indices), _ptr(last_page_len), _ptr(hq), _ptr(hk),
                                           _ptr(hl), len(hq) - 1, int(bool(causal)), float(sm_scale),
                                           _ptr(out), _ptr(lse), dims, _stream(stream)),
           "batch_attention_noalloc")
    return out


def batch_attention_plan(h_qo_indptr, h_kv_indptr, h_last_page_len, num_qo_heads, kv_pages,
                         workspace, prefix_groups=None, stream=None) -> PlanInfo:
    """Plan a batch once (host) and copy the plan into ``workspace``; the
    returned record is what ``batch_attention_run`` / ``append_attention_run``
    take.  ``workspace`` must hold at least the size query's bytes (with the
    same ``prefix_groups``)."""
    lib = load_library()
    _dev_bf16(kv_pages, "kv_pages")
    hq, hk, hl = (_host_i32(x) for x in (h_qo_indptr, h_kv_indptr, h_last_page_len))
    gi, gl, ng = _host_groups(prefix_groups) if prefix_groups is not None else (None, None, 0)
    dims = _dims(kv_pages, num_qo_heads)
    info = PlanInfo()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.daa_batch_attention_plan(_ptr(hq), _ptr(hk), _ptr(hl), len(hq) - 1, _ptr(gi), _ptr(gl),
                                        ng, dims, _ptr(workspace), ws_bytes, ctypes.byref(info),
                                        _stream(stream)), "batch_attention_plan")
    return info


def _run_args(q, kv_pages, qo_indptr, kv_indptr, page_indices, last_page_len, out, lse):
    _dev_bf16(q, "q"), _dev_bf16(kv_pages, "kv_pages")
    for n, t in (("qo_indptr", qo_indptr), ("kv_indptr", kv_indptr), ("page_indices", page_indices),
                 ("last_page_len", last_page_len)):
        _dev_i32(t, n)
    if out is None:
        out = torch.empty_like(q)
    _dev_bf16(out, "out")
    if lse is not None and not (lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()):
        raise TypeError("lse must be a contiguous fp32 CUDA tensor")
    return out


def batch_attention_run(q, kv_pages, qo_indptr, kv_indptr, page_indices, last_page_len, info,
                        workspace, causal=True, sm_scale=None, out=None, lse=None, stream=None):
    """Attention on a plan made by ``batch_attention_plan`` (kernels only)."""
    lib = load_library()
    out = _run_args(q, kv_pages, qo_indptr, kv_indptr, page_indices, last_page_len, out, lse)
    if sm_scale is None:
        sm_scale = 1.0 / float(q.shape[2]) ** 0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.daa_batch_attention_run(_ptr(q), _ptr(kv_pages), _ptr(qo_indptr), _ptr(kv_indptr),
                                       _ptr(page_indices), _ptr(last_page_len), ctypes.byref(info),
                                       int(bool(causal)), float(sm_scale), _ptr(out), _ptr(lse),
                                       _ptr(workspace), ws_bytes, _dims(kv_pages, q.shape[1]),
                                       _stream(stream)), "batch_attention_run")
    return out


def append_attention_run(k_new, v_new, q, kv_pages, qo_indptr, kv_indptr, page_indices,
                         last_page_len, info, workspace, causal=True, sm_scale=None, out=None,
                         lse=None, stream=None):
    """``append_attention`` on a plan made by ``batch_attention_plan``."""
    lib = load_library()
    _dev_bf16(k_new, "k_new"), _dev_bf16(v_new, "v_new")
    out = _run_args(q, kv_pages, qo_indptr, kv_indptr, page_indices, last_page_len, out, lse)
    if sm_scale is None:
        sm_scale = 1.0 / float(q.shape[2]) ** 0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib.daa_append_attention_run(_ptr(k_new), _ptr(v_new), _ptr(q), _ptr(kv_pages),
                                        _ptr(qo_indptr), _ptr(kv_indptr), _ptr(page_indices),
                                        _ptr(last_page_len), ctypes.byref(info), int(bool(causal)),
                                        float(sm_scale), _ptr(out), _ptr(lse), _ptr(workspace),
                                        ws_bytes, _dims(kv_pages, q.shape[1]), _stream(stream)),
           "append_attention_run")
    return out


@dataclass
class PageTable:
    """Device int32 CSR page table plus its host mirror (numpy)."""
    qo_indptr: torch.Tensor
    kv_indptr: torch.Tensor
    page_indices: torch.Tensor
    last_page_len: torch.Tensor
    h_qo_indptr: np.ndarray
    h_kv_indptr: np.ndarray
    h_last_page_len: np.ndarray

    @classmethod
    def from_host(cls, qo_indptr, kv_indptr, page_indices, last_page_len, device="cuda"):
        hq, hk, hp, hl = (_host_i32(x) for x in (qo_indptr, kv_indptr, page_indices, last_page_len))
        dev = lambda a: torch.from_numpy(a).to(device)  # noqa: E731
        return cls(dev(hq), dev(hk), dev(hp), dev(hl), hq, hk, hl)


class BatchAttention:
    """Plan-once / run-many wrapper for one batch shape (FlashInfer-style)."""

    def __init__(self, table: PageTable, num_qo_heads: int, kv_pages: torch.Tensor, causal=True,
                 sm_scale=None, prefix_groups=None):
        self.t = table
        self.kv_pages = kv_pages
        self.causal = causal
        self.Hq = num_qo_heads
        self.sm_scale = sm_scale if sm_scale is not None else 1.0 / float(kv_pages.shape[4]) ** 0.5
        self.prefix_groups = prefix_groups
        n, _, hkv, p, d = kv_pages.shape
        if prefix_groups is None:
            need = batch_attention_workspace_size(table.h_qo_indptr, table.h_kv_indptr,
                                                  table.h_last_page_len, num_qo_heads, hkv, d, p, n)
        else:
            need = shared_prefix_workspace_size(table.h_qo_indptr, table.h_kv_indptr,
                                                table.h_last_page_len, prefix_groups,
                                                num_qo_heads, hkv, d, p, n)
        self.workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=kv_pages.device)
        self.info = None  # set by plan(): run() and step() then launch the kernels only

    def plan(self, stream=None):
        """Upload the batch's plan once; later run() / step() calls (e.g. one per
        layer) reuse it until the next plan() or a tree-mask run."""
        t = self.t
        self.info = batch_attention_plan(t.h_qo_indptr, t.h_kv_indptr, t.h_last_page_len, self.Hq,
                                         self.kv_pages, self.workspace,
                                         prefix_groups=self.prefix_groups, stream=stream)
        return self.info

    def append(self, k_new, v_new, stream=None):
        t = self.t
        kv_append(k_new, v_new, self.kv_pages, t.qo_indptr, t.page_indices, t.kv_indptr,
                  t.last_page_len, stream=stream)

    def step(self, k_new, v_new, q, out=None, lse=None, stream=None):
        """append + run in one call (``append_attention``, or ``append_attention_run``
        on the stored plan)."""
        t = self.t
        if self.info is not None:
            return append_attention_run(k_new, v_new, q, self.kv_pages, t.qo_indptr, t.kv_indptr,
                                        t.page_indices, t.last_page_len, self.info, self.workspace,
                                        self.causal, self.sm_scale, out=out, lse=lse, stream=stream)
        return append_attention(k_new, v_new, q, self.kv_pages, t.qo_indptr, t.kv_indptr,
                                t.page_indices, t.last_page_len, self.causal, self.sm_scale,
                                out=out, lse=lse, workspace=self.workspace,
                                host_indptr=(t.h_qo_indptr, t.h_kv_indptr, t.h_last_page_len),
                                stream=stream, prefix_groups=self.prefix_groups)

    def run(self, q, out=None, lse=None, stream=None, tree_mask=None):
        """Attention over the batch; with ``tree_mask``, under draft-tree masks
        (``batch_attention_tree``; the batch must be causal)."""
        t = self.t
        if tree_mask is None and self.info is not None:
            return batch_attention_run(q, self.kv_pages, t.qo_indptr, t.kv_indptr, t.page_indices,
                                       t.last_page_len, self.info, self.workspace, self.causal,
                                       self.sm_scale, out=out, lse=lse, stream=stream)
        if tree_mask is not None:
            self.info = None  # the tree call plans into the workspace itself
            if self.prefix_groups is not None:
                raise ValueError("tree masks and prefix groups are not combined")
            if not self.causal:
                raise ValueError("a tree mask refines the causal rule")
            return batch_attention_tree(q, self.kv_pages, t.qo_indptr, t.kv_indptr, t.page_indices,
                                        t.last_page_len, tree_mask, self.sm_scale, out=out, lse=lse,
                                        workspace=self.workspace,
                                        host_indptr=(t.h_qo_indptr, t.h_kv_indptr,
                                                     t.h_last_page_len),
                                        stream=stream)
        return batch_attention(q, self.kv_pages, t.qo_indptr, t.kv_indptr, t.page_indices,
                               t.last_page_len, self.causal, self.sm_scale, out=out, lse=lse,
                               workspace=self.workspace,
                               host_indptr=(t.h_qo_indptr, t.h_kv_indptr, t.h_last_page_len),
                               stream=stream, prefix_groups=self.prefix_groups)


class HostStep:
    """Serving steps fed from pinned host memory, one library call each
    (``daa_append_attention_host``): upload the packed inputs, append +
    attention, read the output back.  Two sets of device buffers alternate, so
    step i + 1's upload and step i - 1's read-back overlap step i's kernels.

    ``sections``: the step's host tensors by name -- qo_indptr, kv_indptr,
    page_indices, last_page_len (int32) and q, k_new, v_new (bf16) -- packed
    once into one pinned buffer (``pack``; refill it with ``update``).  The
    page table must not change shape between steps (the workspace is sized for
    it).  ``step(i)`` enqueues step i on the current stream (compute) and two
    side streams; ``out(i)`` is step i's pinned output once ``done(i)`` has
    completed."""

    NAMES = ("qo_indptr", "kv_indptr", "page_indices", "last_page_len", "q", "k_new", "v_new")

    def __init__(self, sections, kv_pages, num_qo_heads, causal=True, sm_scale=None, workspace=None):
        lib = load_library()
        self.lib = lib
        dev = kv_pages.device
        self.kv_pages = kv_pages
        offs, at = {}, 0
        for n in self.NAMES:
            t = sections[n]
            offs[n] = at
            at += (t.numel() * t.element_size() + 255) // 256 * 256
        self.layout = StepLayout(*(offs[n] for n in self.NAMES), at)
        self.offsets = offs
        self.pack = torch.empty(at, dtype=torch.uint8, pin_memory=True)
        self.update(sections)
        hq, hk, hl = (sections[n].numpy() for n in ("qo_indptr", "kv_indptr", "last_page_len"))
        self.batch = len(hq) - 1
        q = sections["q"]
        self.dims = _dims(kv_pages, num_qo_heads)
        self.causal = int(bool(causal))
        self.sm_scale = float(sm_scale if sm_scale is not None else 1.0 / float(q.shape[2]) ** 0.5)
        if workspace is None:
            need = _workspace_need(lib, _host_i32(hq), _host_i32(hk), _host_i32(hl), self.dims, None,
                                   "HostStep")
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
        self.workspace = workspace
        self.d_inputs = [torch.empty(at, dtype=torch.uint8, device=dev) for _ in range(2)]
        self.d_out = [torch.empty(q.shape, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.h_out = [torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True) for _ in range(2)]
        self.up = torch.cuda.Stream(device=dev)
        self.down = torch.cuda.Stream(device=dev)
        self.events = [[torch.cuda.Event() for _ in range(3)] for _ in range(2)]
        cur = torch.cuda.current_stream(dev)
        for evs in self.events:  # events are created on first record
            for e in evs:
                e.record(cur)
        torch.cuda.synchronize(dev)
        self._args = []
        for k in range(2):
            up_ev, comp_ev, down_ev = (e.cuda_event for e in self.events[k])
            ss = StepStreams(self.up.cuda_stream, cur.cuda_stream, self.down.cuda_stream, up_ev, comp_ev,
                             down_ev, comp_ev, down_ev)
            self._args.append((ctypes.c_void_p(self.pack.data_ptr()),
                               ctypes.c_void_p(self.d_inputs[k].data_ptr()), ctypes.byref(self.layout),
                               self.batch, self.causal, ctypes.c_float(self.sm_scale),
                               ctypes.c_void_p(kv_pages.data_ptr()), ctypes.c_void_p(self.d_out[k].data_ptr()),
                               ctypes.c_void_p(self.h_out[k].data_ptr()),
                               ctypes.c_void_p(self.workspace.data_ptr()),
                               self.workspace.numel(), self.dims, ctypes.byref(ss), ss))
        self._stream = cur

    def update(self, sections):
        """Copy the step's host tensors into the pinned pack (wait for the
        previous step's ``uploaded`` event before calling this)."""
        for n in self.NAMES:
            t = sections[n].contiguous()
            nb = t.numel() * t.element_size()
            self.pack[self.offsets[n]:self.offsets[n] + nb].copy_(t.reshape(-1).view(torch.uint8))

    def step(self, i):
        """Enqueue step i (slot i % 2)."""
        a = self._args[i & 1]
        _check(self.lib.daa_append_attention_host(*a[:-1]), "append_attention_host")

    def done(self, i):
        """The event after which step i's output is in ``out(i)``."""
        return self.events[i & 1][2]

    def out(self, i):
        return self.h_out[i & 1]


def set_prefill_append_fusion(enable: bool) -> None:
    """Fused calls (``append_attention``, ``BatchAttention.step``): whether the
    prefill kernels read long chunks' own key tiles from k_new / v_new and write
    them into their pages themselves (True, the default) or the append kernel
    writes every row (False).  Results are identical."""
    _check(load_library().daa_set_prefill_append_fusion(int(bool(enable))),
           "set_prefill_append_fusion")


def prefill_append_fusion() -> bool:
    return bool(load_library().daa_prefill_append_fusion())


def device_error(reset: bool = True) -> int:
    """The library's device error word (0 = none); synchronises the device."""
    lib = load_library()
    code = ctypes.c_int32(0)
    _check(lib.daa_device_error(ctypes.byref(code), int(reset)), "device_error")
    return int(code.value)


def selftest_bounded_wait() -> bool:
    """Run the library's bounded wait on a barrier nothing completes; True when
    it gave up by its time limit (the device error word then holds 2)."""
    lib = load_library()
    flag = ctypes.c_int32(-1)
    _check(lib.daa_selftest_bounded_wait(ctypes.byref(flag)), "selftest_bounded_wait")
    return flag.value == 1


def trace_enable(capacity: int = 4096) -> None:
    _check(load_library().daa_trace_enable(capacity), "trace_enable")


def trace_disable() -> None:
    _check(load_library().daa_trace_disable(), "trace_disable")


def trace_read(max_records: int = 65536):
    """[(kernel name, milliseconds)] of the launches recorded since the last read."""
    lib = load_library()
    ids = (ctypes.c_int32 * max_records)()
    ms = (ctypes.c_float * max_records)()
    n = lib.daa_trace_read(ids, ms, max_records)
    return [(KERNEL_NAMES.get(ids[i], str(ids[i])), float(ms[i])) for i in range(n)]
