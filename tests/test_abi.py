"""CPU-side checks of the C ABI: the library builds and loads, exports every
symbol the header declares, and rejects invalid arguments on the host before
touching the device.  No compute call runs here (there is no GPU)."""
import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from decode_attention_append_gb300 import build
    build.build()
    import decode_attention_append_gb300 as daa
    return daa.load_library()


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "daa.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(daa_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    syms = _declared_symbols()
    for s in ("daa_kv_append", "daa_batch_attention", "daa_batch_attention_workspace_size",
              "daa_append_attention", "daa_status_string", "daa_device_error", "daa_trace_enable",
              "daa_trace_read"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    missing = [s for s in _declared_symbols() if not hasattr(lib, s)]
    assert not missing, missing


def test_library_exports_nothing_undeclared(lib):
    import subprocess
    from decode_attention_append_gb300 import library_path
    out = subprocess.run(["nm", "-D", "--defined-only", library_path()], capture_output=True, text=True)
    if out.returncode != 0:
        pytest.skip("nm unavailable")
    exported = {ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln}
    daa_syms = {s for s in exported if s.startswith("daa_")}
    assert daa_syms == set(_declared_symbols())


def test_status_strings(lib):
    for code in range(0, -8, -1):
        s = lib.daa_status_string(code)
        assert s and s != b"unknown status"
    assert lib.daa_version() > 0


def _dims(Hq=4, Hkv=2, d=64, P=16, n=64):
    import decode_attention_append_gb300 as daa
    return daa._Dims(Hq, Hkv, d, P, n)


def _ws(lib, qo, kv, last, dims):
    st = ctypes.c_int32(0)
    qo, kv, last = (np.asarray(x, np.int32) for x in (qo, kv, last))
    n = lib.daa_batch_attention_workspace_size(qo.ctypes.data_as(ctypes.c_void_p),
                                               kv.ctypes.data_as(ctypes.c_void_p),
                                               last.ctypes.data_as(ctypes.c_void_p), len(qo) - 1,
                                               dims, ctypes.byref(st))
    return n, st.value


@pytest.mark.parametrize("qo,kv,last,dims,expect", [
    ([0, 2], [0, 1], [1], _dims(), -2),                 # qo_len 2 > kv_len 1
    ([0, 1], [0, 1], [0], _dims(), -2),                 # last_page_len 0 with a page
    ([0, 1], [0, 1], [17], _dims(), -2),                # last_page_len > page_size
    ([1, 1], [0, 1], [1], _dims(), -2),                 # indptr not starting at 0
    ([0, 3, 2], [0, 1, 2], [16, 16], _dims(), -2),      # decreasing qo_indptr
    ([0, 1], [0, 1], [1], _dims(d=96), -4),             # head_dim unsupported
    ([0, 1], [0, 1], [1], _dims(P=32), -4),             # page_size unsupported
    ([0, 1], [0, 1], [1], _dims(Hq=34, Hkv=2), -4),     # group size 17
    ([0, 1], [0, 1], [1], _dims(Hq=5, Hkv=2), -1),      # Hq not divisible by Hkv
    ([0, 1], [0, 1], [1], _dims(n=0), -1),              # empty pool
])
def test_host_validation_rejects(lib, qo, kv, last, dims, expect):
    n, st = _ws(lib, qo, kv, last, dims)
    assert st == expect and n == 0


def test_workspace_size_decode_and_prefill(lib):
    # two decodes of 40 and 73 tokens plus a 16-token chunk at offset 48: only
    # the plan is needed (the requests are short enough not to be split)
    n, st = _ws(lib, [0, 16, 17, 18], [0, 4, 7, 12], [16, 8, 9], _dims())
    assert st == 0 and n > 0 and n % 256 == 0
    n0, st0 = _ws(lib, [0], [0], [], _dims())
    assert st0 == 0 and n0 == 0


def test_workspace_grows_with_split_decodes(lib):
    # one long decode (40k tokens) gets split: partial outputs need space
    pages = 2500
    n_short, _ = _ws(lib, [0, 1], [0, 4], [16], _dims(Hq=8, Hkv=1, d=128))
    n_long, _ = _ws(lib, [0, 1], [0, pages], [16], _dims(Hq=8, Hkv=1, d=128, n=4096))
    assert n_long > n_short + 8 * 128 * 4


def test_null_pointers_rejected_before_any_launch(lib):
    import decode_attention_append_gb300 as daa
    d = _dims()
    st = lib.daa_kv_append(None, None, None, None, None, None, None, 1, 4, d, None)
    assert st == -1
    qo = np.asarray([0, 1], np.int32)
    kv = np.asarray([0, 1], np.int32)
    last = np.asarray([1], np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    st = lib.daa_batch_attention(None, None, None, None, None, None, p(qo), p(kv), p(last), 1, 1,
                                 0.125, None, None, None, 0, d, None)
    assert st == -1
    st = lib.daa_batch_attention(None, None, None, None, None, None, p(qo), p(kv), p(last), 1, 1,
                                 float("nan"), None, None, None, 0, d, None)
    assert st == -1
    assert daa.STATUS[-1] == "invalid argument"


def test_append_attention_rejects_before_any_launch(lib):
    """The fused call validates both halves on the host: missing or misaligned
    k_new / v_new, and everything batch_attention rejects."""
    d = _dims()
    qo = np.asarray([0, 1], np.int32)
    kv = np.asarray([0, 1], np.int32)
    last = np.asarray([1], np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    dev = lambda x: ctypes.c_void_p(x)  # noqa: E731  (never dereferenced: rejected first)
    args = [dev(0x10000), dev(0x20000), dev(0x30000), dev(0x40000), dev(0x50000)]
    ws = dev(0x100000)
    call = lambda kn, vn, scale=0.125, lastp=last: lib.daa_append_attention(  # noqa: E731
        kn, vn, dev(0x1000), *args, p(qo), p(kv), p(lastp), 1, 1, scale, dev(0x70000), None, ws,
        1 << 20, d, None)
    assert call(None, dev(0x2000)) == -1
    assert call(dev(0x2008), dev(0x3000)) == -7
    assert call(dev(0x2000), dev(0x3000), scale=0.0) == -1
    assert call(dev(0x2000), dev(0x3000), lastp=np.asarray([0], np.int32)) == -2


def test_misaligned_pointers_rejected(lib):
    d = _dims()
    st = lib.daa_kv_append(ctypes.c_void_p(0x1008), ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000),
                           ctypes.c_void_p(0x4000), ctypes.c_void_p(0x5000), ctypes.c_void_p(0x6000),
                           ctypes.c_void_p(0x7000), 1, 4, d, None)
    assert st == -7


def test_oracle_and_library_share_no_code():
    """The checker and the product are independent: no source of one includes,
    imports or links the other."""
    pkg = os.path.join(ROOT, "decode_attention_append_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in re.sub(r"(#|//).*", "", text), f
    for f in os.listdir(os.path.join(ROOT, "oracle")):
        if f.endswith((".py", ".c")):
            text = open(os.path.join(ROOT, "oracle", f)).read()
            assert "decode_attention_append_gb300" not in text and "daa.h" not in text, f


def test_tree_attention_rejects_before_any_launch(lib):
    """daa_batch_attention_tree: a mask is required, must be 4-byte aligned,
    needs at least one word per row and enough words for every request's new
    tokens (checked against the host mirror of qo_indptr)."""
    d = _dims()
    qo = np.asarray([0, 40], np.int32)     # one request of 40 new tokens
    kv = np.asarray([0, 3], np.int32)
    last = np.asarray([16], np.int32)
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    dev = lambda x: ctypes.c_void_p(x)  # noqa: E731  (never dereferenced: rejected first)
    call = lambda mask, words: lib.daa_batch_attention_tree(  # noqa: E731
        dev(0x10000), dev(0x20000), dev(0x30000), dev(0x40000), dev(0x50000), dev(0x60000),
        p(qo), p(kv), p(last), 1, mask, words, 0.125, dev(0x70000), None, dev(0x100000), 1 << 20,
        d, None)
    assert call(None, 2) == -1
    assert call(dev(0x8000), 0) == -1
    assert call(dev(0x8002), 2) == -7
    assert call(dev(0x8000), 1) == -2      # 40 tokens need 2 words


def _ws_groups(lib, qo, kv, last, dims, ind, plen, n=None):
    st = ctypes.c_int32(0)
    qo, kv, last = (np.asarray(x, np.int32) for x in (qo, kv, last))
    ind = None if ind is None else np.asarray(ind, np.int32)
    plen = None if plen is None else np.asarray(plen, np.int32)
    p = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    ng = (len(plen) if plen is not None else 0) if n is None else n
    size = lib.daa_batch_attention_shared_prefix_workspace_size(
        p(qo), p(kv), p(last), len(qo) - 1, p(ind), p(plen), ng, dims, ctypes.byref(st))
    return size, st.value


# three decodes (kv 300, 400, 500) that share a 256-token prefix; head_dim 128, GQA 8:1
_G_QO, _G_KV, _G_LAST = [0, 1, 2, 3], [0, 19, 44, 76], [12, 16, 4]


@pytest.mark.parametrize("ind,plen,n,expect", [
    ([0, 3], [256], -1, -1),          # negative group count
    (None, None, 1, -1),              # group arrays missing
    ([0, 4], [256], None, -2),        # group past the batch
    ([-1, 3], [256], None, -2),       # group before the batch
    ([2, 1], [256], None, -2),        # decreasing indptr
    ([0, 3], [250], None, -2),        # prefix not whole pages
    ([0, 3], [-16], None, -2),        # negative prefix
    ([0, 3], [304], None, -2),        # prefix longer than the first request's cached keys (299)
])
def test_shared_prefix_validation_rejects(lib, ind, plen, n, expect):
    size, st = _ws_groups(lib, _G_QO, _G_KV, _G_LAST, _dims(Hq=8, Hkv=1, d=128, n=256), ind, plen, n)
    assert st == expect and size == 0


def test_shared_prefix_workspace(lib):
    """No groups: the plain plan.  A 256-token prefix shared by three decodes:
    one partial row per decode for the shared part plus one for its own part."""
    dims = _dims(Hq=8, Hkv=1, d=128, n=256)
    plain, st = _ws(lib, _G_QO, _G_KV, _G_LAST, dims)
    assert st == 0
    none, st = _ws_groups(lib, _G_QO, _G_KV, _G_LAST, dims, None, None, 0)
    assert st == 0 and none == plain
    small, st = _ws_groups(lib, _G_QO, _G_KV, _G_LAST, dims, [0, 3], [112])  # under one tile
    assert st == 0 and small == plain
    shared, st = _ws_groups(lib, _G_QO, _G_KV, _G_LAST, dims, [0, 3], [256])
    assert st == 0 and shared >= plain + 2 * 3 * 8 * 128 * 4


def test_plan_and_run_reject_before_any_launch(lib):
    """daa_batch_attention_plan / _run: a plan record is required and checked
    (magic, dims) on the host; a workspace smaller than the plan is refused."""
    import decode_attention_append_gb300 as daa
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    dev = lambda x: ctypes.c_void_p(x)  # noqa: E731  (never dereferenced: rejected first)
    d = _dims(Hq=8, Hkv=1, d=128, n=256)
    qo, kv, last = (np.asarray(x, np.int32) for x in (_G_QO, _G_KV, _G_LAST))
    info = daa.PlanInfo()
    plan = lambda ws, nbytes, inf: lib.daa_batch_attention_plan(  # noqa: E731
        p(qo), p(kv), p(last), 3, None, None, 0, d, ws, nbytes, inf, None)
    assert plan(dev(0x100000), 1 << 20, None) == -1            # no record
    assert plan(dev(0x100000), 64, ctypes.byref(info)) == -6   # workspace too small
    assert plan(dev(0x100080), 1 << 20, ctypes.byref(info)) == -7  # misaligned workspace
    run = lambda inf, dims: lib.daa_batch_attention_run(  # noqa: E731
        dev(0x10000), dev(0x20000), dev(0x30000), dev(0x40000), dev(0x50000), dev(0x60000), inf, 1,
        0.125, dev(0x70000), None, dev(0x100000), 1 << 20, dims, None)
    assert run(None, d) == -1
    assert run(ctypes.byref(daa.PlanInfo()), d) == -1           # never written by a plan
    # an empty batch plans without touching the device; its record runs as a no-op
    e0 = np.zeros(1, np.int32)
    assert lib.daa_batch_attention_plan(p(e0), p(e0), None, 0, None, None, 0, d, None, 0,
                                        ctypes.byref(info), None) == 0
    assert run(ctypes.byref(info), d) == 0
    assert run(ctypes.byref(info), _dims(Hq=8, Hkv=1, d=64, n=256)) == -1  # other dims


def test_binding_prefix_groups_and_plan_records(lib):
    """Python binding, host side only: prefix groups are checked for shape
    before the library sees them; the shared-prefix workspace query follows
    the groups; an empty batch plans to a record without touching a device."""
    import decode_attention_append_gb300 as daa
    qo, kv, last = _G_QO, _G_KV, _G_LAST
    with pytest.raises(ValueError):
        daa.shared_prefix_workspace_size(qo, kv, last, ([0, 3], [256, 16]), 8, 1, 128, 16, 256)
    with pytest.raises(daa.DaaError):
        daa.shared_prefix_workspace_size(qo, kv, last, ([0, 3], [250]), 8, 1, 128, 16, 256)
    plain = daa.batch_attention_workspace_size(qo, kv, last, 8, 1, 128, 16, 256)
    assert daa.shared_prefix_workspace_size(qo, kv, last, ([0, 3], [0]), 8, 1, 128, 16, 256) == plain
    assert daa.shared_prefix_workspace_size(qo, kv, last, ([0, 3], [256]), 8, 1, 128, 16, 256) > plain
    rec = daa.PlanInfo()
    assert ctypes.sizeof(rec) == 24 * 8


def test_host_step_rejects_before_any_launch(lib):
    """daa_append_attention_host checks its layout and handles on the host:
    a NULL event, misaligned sections or device copy, sections past the
    buffer, and the fused call's own errors -- all before enqueuing anything
    (the device pointers here are never dereferenced)."""
    import decode_attention_append_gb300 as daa
    d = _dims()
    # one request: 1 new token over 1 cached; qo, kv, pages, last, q, k, v
    host = np.zeros(4096, np.uint8)
    ints = host[:256].view(np.int32)
    ints[0:2] = [0, 1]      # qo_indptr at 0
    ints[16:18] = [0, 1]    # kv_indptr at 64
    ints[32] = 7            # page_indices at 128
    ints[48] = 2            # last_page_len at 192
    lay = daa.StepLayout(0, 64, 128, 192, 256, 1280, 1536, 2048)
    ev = [ctypes.c_void_p(0x100 + 8 * i) for i in range(3)]
    ss = daa.StepStreams(None, None, None, ev[0], ev[1], ev[2], None, None)
    hp = host.ctypes.data_as(ctypes.c_void_p)
    dev = lambda x: ctypes.c_void_p(x)  # noqa: E731

    def call(layout=lay, streams=ss, d_inputs=dev(0x100000), scale=0.125):
        return lib.daa_append_attention_host(hp, d_inputs, ctypes.byref(layout), 1, 1, scale,
                                             dev(0x200000), dev(0x300000), dev(0x400000),
                                             dev(0x500000), 1 << 20, d, ctypes.byref(streams))
    bad = daa.StepStreams(None, None, None, ev[0], None, ev[2], None, None)
    assert call(streams=bad) == -1                                    # a NULL event
    assert call(d_inputs=dev(0x100010)) == -7                         # device copy not 256-aligned
    assert call(layout=daa.StepLayout(0, 64, 128, 194, 256, 1280, 1536, 2048)) == -7  # int32 offset
    assert call(layout=daa.StepLayout(0, 64, 128, 192, 264, 1280, 1536, 2048)) == -7  # bf16 offset
    assert call(layout=daa.StepLayout(0, 64, 128, 192, 256, 1280, 1536, 1600)) == -2  # v_new past the end
    assert call(scale=0.0) == -1                                      # the fused call's own check
    ints[48] = 0                                                      # last_page_len out of range
    assert call() == -2
