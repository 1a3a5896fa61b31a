"""daa_batch_attention_noalloc, the entry point for callers that cannot allocate
device memory (a serving engine whose HBM all belongs to its page pool, a
latency-critical path where cudaMalloc could synchronise the device, a
foreign-language host without a CUDA allocator).  Its scratch is the library's
fixed device array instead of a caller workspace.

Checked through the C ABI against daa_batch_attention (the workspace entry
point) within the parity tolerances of the other GPU tests, on two calls in a
row with different batches, so the second call runs over the first call's
leftover scratch contents.  This file is collected last and is self-contained:
it passes alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from synth import make_random_workload

pytestmark = pytest.mark.gpu

MAX_ERR, MEAN_ERR = 1.5e-2, 2e-3


def _setup(wl, dev):
    from gpu_support import gpu_fill, new_pool
    import decode_attention_append_gb300 as daa
    pool = new_pool(wl, dev)
    gpu_fill(wl, pool, dev)
    st = wl.step_table(0)
    q, kn, vn = wl.step_inputs(0)
    tab = daa.PageTable.from_host(st["qo_indptr"], st["kv_indptr"], st["page_indices"],
                                  st["last_page_len"], dev)
    daa.kv_append(kn.to(dev), vn.to(dev), pool, tab.qo_indptr, tab.page_indices, tab.kv_indptr,
                  tab.last_page_len)
    return pool, tab, q.to(dev)


def _call_noalloc(lib, wl, pool, tab, q, out, lse):
    import decode_attention_append_gb300 as daa
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    h = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    dims = daa._Dims(wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages)
    st = lib.daa_batch_attention_noalloc(
        p(q), p(pool), p(tab.qo_indptr), p(tab.kv_indptr), p(tab.page_indices), p(tab.last_page_len),
        h(tab.h_qo_indptr), h(tab.h_kv_indptr), h(tab.h_last_page_len), len(tab.h_qo_indptr) - 1,
        1, ctypes.c_float(wl.sm_scale), p(out), p(lse), dims,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.daa_status_string(st)


def _call_workspace(lib, wl, pool, tab, q, out, lse):
    import decode_attention_append_gb300 as daa
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    h = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    dims = daa._Dims(wl.num_qo_heads, wl.num_kv_heads, wl.head_dim, wl.page_size, wl.num_pages)
    status = ctypes.c_int32(0)
    nbytes = lib.daa_batch_attention_workspace_size(h(tab.h_qo_indptr), h(tab.h_kv_indptr),
                                                    h(tab.h_last_page_len), len(tab.h_qo_indptr) - 1,
                                                    dims, ctypes.byref(status))
    assert status.value == 0
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.daa_batch_attention(
        p(q), p(pool), p(tab.qo_indptr), p(tab.kv_indptr), p(tab.page_indices), p(tab.last_page_len),
        h(tab.h_qo_indptr), h(tab.h_kv_indptr), h(tab.h_last_page_len), len(tab.h_qo_indptr) - 1,
        1, ctypes.c_float(wl.sm_scale), p(out), p(lse), p(ws), ctypes.c_size_t(ws.numel()), dims,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.daa_status_string(st)
    return nbytes


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import decode_attention_append_gb300 as daa
    lib = daa.load_library()
    dev = torch.device("cuda:0")
    batches = [
        # mixed: a prefill chunk, long decodes that are split (partials + merge), short decodes
        make_random_workload(301, 8, 2, 128, 16, [(200, 1200), (1, 40000), (1, 300), (1, 9000)]),
        # a different shape on the second call: GQA 4:1, d 64, more splits
        make_random_workload(302, 8, 2, 64, 16, [(1, 30000), (37, 37), (1, 17), (1, 25000)]),
    ]
    for wl in batches:
        pool, tab, q = _setup(wl, dev)
        out_ref = torch.full_like(q, float("nan"))
        lse_ref = torch.full((q.shape[0], wl.num_qo_heads), float("nan"), device=dev)
        nbytes = _call_workspace(lib, wl, pool, tab, q, out_ref, lse_ref)
        assert nbytes > 0
        out = torch.full_like(q, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        _call_noalloc(lib, wl, pool, tab, q, out, lse)
        torch.cuda.synchronize()
        a, b = out.double(), out_ref.double()
        assert torch.isfinite(a).all()
        diff = (a - b).abs()
        assert diff.max().item() <= MAX_ERR and diff.mean().item() <= MEAN_ERR, (
            diff.max().item(), diff.mean().item())
        assert (lse - lse_ref).abs().max().item() <= 1e-3
    assert daa.device_error(reset=True) == 0
