"""Host logic of the work plan, on the CPU: for random mixed batches, with and
without prefix groups, every query row must see each of its visible keys in
exactly one work item, and its partial results must be merged exactly once.

The plan is built by the library's own planner header, compiled with g++ into a
small harness (``plan_check.cpp``) that prints it.  What each item computes is
read the way the kernels read it:
  * a CUDA-core decode unit: the request's one row, keys [tok_begin, tok_end);
  * a tensor-core item of a request: its tokens tok0 .. tok0 + ntok + ntok1,
    keys [key_lo, min(key_hi, the row's causal end));
  * a prefix-group item: the rows q_row0 + tok0 .. of consecutive requests,
    keys [0, key_hi), which every one of those rows must see;
and a row writes either its output directly (one item covers all its keys) or
a partial to slot part + t * part_stride that one softmax_merge item names.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
P = 16


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ unavailable")
    inc = [os.path.join(ROOT, "include"), os.path.join(ROOT, "decode_attention_append_gb300", "csrc")]
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_check")
    cmd = [gxx, "-std=c++17", "-O1", *sum((["-I", i] for i in inc + [cuda_inc]), []),
           os.path.join(ROOT, "tests", "plan_check.cpp"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def _fmt(case):
    (Hq, Hkv, d, sms), qo, kv, last, groups = case
    parts = [f"{Hq} {Hkv} {d} {P} 1000000 {sms}", str(len(qo) - 1), " ".join(map(str, qo)),
             " ".join(map(str, kv)), " ".join(map(str, last))]
    if groups is None:
        parts.append("-1")
    else:
        ind, plen = groups
        parts += [str(len(plen)), " ".join(map(str, ind)), " ".join(map(str, plen))]
    return "\n".join(parts) + "\n"


def _plan(exe, cases):
    out = subprocess.run([exe], input="".join(_fmt(c) for c in cases), capture_output=True,
                         text=True, check=True).stdout
    plans, cur = [], None
    for ln in out.splitlines():
        f = ln.split()
        if f[0] == "S":
            cur = dict(status=int(f[1]), U=[], M=[], T=[])
        elif f[0] == "E":
            plans.append(cur)
        elif f[0] == "L":
            cur["L"] = list(map(int, f[1:]))
        else:
            cur[f[0]].append(list(map(int, f[1:])))
    assert len(plans) == len(cases)
    return plans


def _check(case, plan, causal=True):
    """Exact cover of every row's visible keys; every partial merged once."""
    (Hq, Hkv, d, sms), qo, kv, last, _ = case
    assert plan["status"] == 0
    batch = len(qo) - 1
    kv_len = [(kv[r + 1] - kv[r] - 1) * P + last[r] if kv[r + 1] > kv[r] else 0 for r in range(batch)]
    row_req = np.repeat(np.arange(batch), np.diff(qo))
    nrows = qo[-1]
    contrib = [[] for _ in range(nrows)]  # (key_lo, key_hi, slot or None)

    def vis_end(r, t):
        pos = kv_len[r] - (qo[r + 1] - qo[r]) + t
        return min(pos + 1, kv_len[r]) if causal else kv_len[r]

    for q_row, page_base, lo, hi, kl, part in plan["U"]:
        r = row_req[q_row]
        assert qo[r + 1] - qo[r] == 1 and kl == kv_len[r] and page_base == kv[r]
        contrib[q_row].append((lo, hi, part if part >= 0 else None))
    n_dec, n_short = plan["L"][3], plan["L"][4]
    for q_row0, qo_len, kl, page_base, tok0, ntok, ntok1, key_lo, key_hi, part, stride, kind in plan["T"]:
        assert key_lo % 128 == 0 and key_lo < key_hi
        for tt in range(tok0, tok0 + ntok + ntok1):
            row = q_row0 + tt
            r = row_req[row]
            slot = part + tt * stride if part >= 0 else None
            if kind == 1:  # prefix-group item: shared keys precede every row
                assert kl == key_hi and key_hi <= kv_len[r] - (qo[r + 1] - qo[r]) and slot is not None
                assert page_base == kv[row_req[q_row0]]
                contrib[row].append((0, key_hi, slot))
            else:
                assert q_row0 == qo[r] and qo_len == qo[r + 1] - qo[r] and kl == kv_len[r]
                assert page_base == kv[r]
                contrib[row].append((key_lo, min(key_hi, vis_end(r, tt)), slot))
    merged = {}
    for q_row, pb, n, extra in plan["M"]:
        assert q_row not in merged, "row merged twice"
        merged[q_row] = set(range(pb, pb + n)) | ({extra} if extra >= 0 else set())
    written = []
    for row in range(nrows):
        r = row_req[row]
        c = sorted(contrib[row])
        # the row's keys [0, vis_end) are covered exactly once
        at = 0
        for lo, hi, _ in c:
            assert lo == at, (row, c)
            at = max(at, hi)
        assert at == vis_end(r, row - qo[r]), (row, c)
        slots = [s for _, _, s in c if s is not None]
        if len(c) == 1 and slots == []:
            assert row not in merged
        else:
            assert len(slots) == len(c), "a split row written directly"
            assert merged.get(row) == set(slots), (row, slots, merged.get(row))
            written += slots
    assert len(written) == len(set(written)), "a partial slot written twice"
    assert all(0 <= s < plan["L"][5] for s in written)
    assert len(written) == sum(len(v) for v in merged.values())
    assert plan["L"][:3] == [len(plan["U"]), len(plan["M"]), len(plan["T"])]
    assert n_dec + n_short <= len(plan["T"])


SHAPES = [(32, 32, 128), (32, 8, 128), (12, 1, 128), (16, 2, 64), (8, 4, 64), (64, 8, 128),
          (16, 16, 64)]


def _random_case(rng, with_groups):
    Hq, Hkv, d = SHAPES[rng.integers(len(SHAPES))]
    sms = int(rng.choice([4, 16, 152]))
    batch = int(rng.integers(1, 11))
    qos, cached = [], []
    for _ in range(batch):
        kind = rng.integers(6)
        qo = [1, 1, int(rng.integers(2, 17)), int(rng.integers(17, 300)), int(rng.integers(300, 1200)),
              0][kind]
        c = int(rng.choice([rng.integers(0, 6000), 128 * rng.integers(0, 40) + rng.integers(-1, 2)]))
        c = max(c, 0 if qo else 1)
        qos.append(qo)
        cached.append(c)
    kvl = [q + c for q, c in zip(qos, cached)]
    qo = np.concatenate([[0], np.cumsum(qos)]).astype(int).tolist()
    npg = [-(-k // P) for k in kvl]
    kv = np.concatenate([[0], np.cumsum(npg)]).astype(int).tolist()
    last = [k - (n - 1) * P if n else 0 for k, n in zip(kvl, npg)]
    groups = None
    if with_groups:
        cuts = sorted(set([0, batch] + rng.integers(0, batch + 1, size=rng.integers(0, 4)).tolist()))
        ind, plen = [cuts[0]], []
        for a, b in zip(cuts[:-1], cuts[1:]):
            cap = min(cached[a:b]) if b > a else 0
            pl = int(rng.integers(0, cap // P + 1)) * P
            if rng.random() < 0.5:
                pl = cap // P * P  # the longest prefix the group allows
            ind.append(b)
            plen.append(pl)
        groups = (ind, plen)
    return (Hq, Hkv, d, sms), qo, kv, last, groups


@pytest.mark.parametrize("with_groups", [False, True])
@pytest.mark.parametrize("causal", [True, False])
def test_plan_covers_every_key_once(harness, with_groups, causal):
    rng = np.random.default_rng(20261202 + with_groups)
    cases = [_random_case(rng, with_groups) for _ in range(250)]
    for case, plan in zip(cases, _plan(harness, cases)):
        _check(case, plan, causal=causal)


def test_plan_prefix_groups_share_keys(harness):
    """Decodes over one 1024-token prefix: one group item per kv-head pass
    holds all their rows, each decode's own work starts at key 1024, and every
    decode row merges exactly two parts (shared + own) when unsplit."""
    n = 20
    kvl = [1024 + 1 + 37 * i for i in range(n)]
    npg = [-(-k // P) for k in kvl]
    kv = np.concatenate([[0], np.cumsum(npg)]).astype(int).tolist()
    case = ((32, 8, 128, 152), list(range(n + 1)), kv, [k - (m - 1) * P for k, m in zip(kvl, npg)],
            ([0, n], [1024]))
    plan = _plan(harness, [case])[0]
    _check(case, plan)
    groups = [t for t in plan["T"] if t[-1] == 1]
    assert len(groups) == 1 and groups[0][5] == n and groups[0][8] == 1024
    own = [t for t in plan["T"] if t[-1] == 0]
    assert own and all(t[7] >= 1024 for t in own)
    assert all(m[2] + (m[3] >= 0) >= 2 for m in plan["M"])


def test_plan_prefill_request_ends_a_run(harness):
    """A prefill request inside a group keeps the prefix in its own items and
    splits the group's decodes into two runs (two group items)."""
    reqs = [(1, 2000), (1, 2100), (600, 2600), (1, 1500), (1, 1600)]
    qo = np.concatenate([[0], np.cumsum([q for q, _ in reqs])]).astype(int).tolist()
    npg = [-(-k // P) for _, k in reqs]
    kv = np.concatenate([[0], np.cumsum(npg)]).astype(int).tolist()
    last = [k - (m - 1) * P for (_, k), m in zip(reqs, npg)]
    case = ((32, 8, 128, 152), qo, kv, last, ([0, 5], [1024]))
    plan = _plan(harness, [case])[0]
    _check(case, plan)
    groups = [t for t in plan["T"] if t[-1] == 1]
    assert sorted((t[0], t[5]) for t in groups) == [(0, 2), (602, 2)]
    prefill = [t for t in plan["T"] if t[-1] == 0 and t[1] == 600]
    assert prefill and all(t[7] == 0 and t[9] == -1 for t in prefill)


def _model_split(qos, kvs, Hkv, sms=152):
    """The planner's choice of tensor-core decode split for a batch with no
    prefill items, restated: pages per split for 2..8 items per SM, each
    scored by greedy most-keys-first assignment of its (split, kv head) units
    to 2 x SM persistent CTAs (64 keys of overhead per unit); first minimum."""
    import heapq
    pages = sum(-(-k // P) for q, k in zip(qos, kvs) if 1 <= q <= 16)
    ph = pages * Hkv
    best, best_split = None, None
    for per_sm in (2, 3, 4, 5, 6, 8):
        sp = (ph + sms * per_sm - 1) // (sms * per_sm)
        sp = max(32, min(2048, (sp + 7) // 8 * 8))
        units = []
        for q, k in zip(qos, kvs):
            if not 1 <= q <= 16:
                continue
            keys = k - q + 1
            n = -(-keys // (sp * P))
            units += [sp * P] * (n - 1) + [k - (n - 1) * sp * P]
        units = sorted(units * Hkv, reverse=True)
        h = [0] * (2 * sms)
        for u in units:
            heapq.heapreplace(h, h[0] + u + 64)
        m = max(h)
        if best is None or m < best:
            best, best_split = m, sp
    return best_split


def test_plan_decode_split_follows_the_assignment_model(harness):
    """GQA decode alone: the number of decode items equals the split the
    greedy-assignment model picks (GQA decode shard: 2 per SM, 362 items)."""
    from synth import make_workload
    rng = np.random.default_rng(77)
    batches = []
    wl = make_workload("gqa_decode_shard")
    batches.append(([r.qo_len for r in wl.steps[0].requests], [r.kv_len for r in wl.steps[0].requests],
                    wl.num_qo_heads, wl.num_kv_heads))
    for _ in range(12):
        n = int(rng.integers(8, 200))
        kvs = rng.integers(200, 40000, size=n).tolist()
        qos = [1 if rng.random() < 0.85 else int(rng.integers(2, 9)) for _ in range(n)]
        Hkv = int(rng.choice([1, 2, 8]))
        batches.append((qos, [max(k, q) for k, q in zip(kvs, qos)], 8 * Hkv, Hkv))
    for qos, kvs, Hq, Hkv in batches:
        qo = np.concatenate([[0], np.cumsum(qos)]).astype(int).tolist()
        npg = [-(-k // P) for k in kvs]
        kv = np.concatenate([[0], np.cumsum(npg)]).astype(int).tolist()
        last = [k - (m - 1) * P for k, m in zip(kvs, npg)]
        case = ((Hq, Hkv, 128, 152), qo, kv, last, None)
        plan = _plan(harness, [case])[0]
        _check(case, plan)
        sp = _model_split(qos, kvs, Hkv)
        # the Q rows of a verify request need qo_len * g <= 128 to stay in the decode launch
        g = Hq // Hkv
        expect = sum(-(-(k - q + 1) // (sp * P)) for q, k in zip(qos, kvs) if 1 <= q <= min(16, 128 // g))
        assert plan["L"][3] == expect, (plan["L"][3], expect, sp)
    gq = batches[0]
    assert _plan(harness, [((gq[2], gq[3], 128, 152),
                            np.concatenate([[0], np.cumsum(gq[0])]).astype(int).tolist(),
                            np.concatenate([[0], np.cumsum([-(-k // P) for k in gq[1]])]).astype(int).tolist(),
                            [k - (-(-k // P) - 1) * P for k in gq[1]], None)])[0]["L"][3] == 362
