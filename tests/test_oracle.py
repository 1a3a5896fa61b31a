"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here runs on the CPU.  Each targets a plausible mistake in the
oracle: a wrong causal offset or GQA mapping (library attention, chunk
equivalence), a wrong page/slot index in the append or the gather (HND layout
properties, dense brute force, page-permutation invariance), a dropped term in
the softmax or its log-sum-exp (merge identity, special cases, library
log-sum-exp), a wrong append byte count (the IO-overhead worked example).
"""
import copy
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import dense
from synth import (SENTINEL_BF16, Request, Step, chunk_schedule, make_prompt_workload,
                   make_random_workload, make_shared_prefix_workload, make_tree_workload,
                   make_workload, tree_mask_rows)
from support import oracle_pool, oracle_step

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _f64(t):
    return t.double().numpy()


TINY_CASES = [
    # (seed, Hq, Hkv, d, P, [(qo, kv), ...])
    (1, 4, 2, 8, 4, [(5, 5), (1, 7), (12, 30), (3, 3)]),
    (2, 3, 1, 8, 4, [(1, 1), (5, 17), (1, 16)]),
    (3, 4, 4, 64, 16, [(16, 64), (1, 40), (1, 73), (12, 12)]),
    (4, 6, 2, 8, 16, [(7, 21), (0, 9), (2, 2), (1, 33)]),
    (5, 2, 2, 8, 4, [(0, 0), (4, 4), (1, 5)]),
]


@pytest.mark.parametrize("case", TINY_CASES, ids=lambda c: f"seed{c[0]}")
@pytest.mark.parametrize("causal", [True, False])
def test_oracle_matches_dense_bruteforce(case, causal):
    seed, Hq, Hkv, d, P, reqs = case
    wl = make_random_workload(seed, Hq, Hkv, d, P, reqs, extra_pages=3)
    wl.causal = causal
    pool = oracle_pool(wl)
    out, lse, _ = oracle_step(wl, pool, 0)
    t = wl.step_table(0)
    q, _, _ = wl.step_inputs(0)
    dout, dlse, _ = dense.attention(_bits(q), pool, t["qo_indptr"], t["kv_indptr"], t["page_indices"],
                                    t["last_page_len"], causal, wl.sm_scale, Hq)
    assert out.shape == dout.shape
    np.testing.assert_allclose(out, dout, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, dlse, rtol=0, atol=1e-12)


def _contiguous_request(seed, Hq, Hkv, d, P, qo, kv):
    """One request whose pages are [0, 1, 2, ...] after a pool permutation, and
    the same request's dense K/V straight from the generator."""
    wl = make_random_workload(seed, Hq, Hkv, d, P, [(qo, kv)], extra_pages=5)
    pool = oracle_pool(wl)
    out, lse, _ = oracle_step(wl, pool, 0)
    q = wl.q_rows(0, kv - qo, kv)
    K = wl.k_rows(0, 0, kv)
    V = wl.v_rows(0, 0, kv)
    return wl, out, lse, q, K, V


@pytest.mark.parametrize("shape", [(4, 4, 16, 16, 9, 40), (8, 2, 64, 16, 1, 73), (6, 3, 32, 4, 13, 13),
                                   (12, 1, 128, 16, 17, 50)])
def test_oracle_matches_torch_sdpa(shape):
    """Library attention (torch SDPA in fp64) on K/V taken from the generator,
    not from the pool: pins the paged gather, the append, the scale, the GQA
    grouping and the bottom-right causal offset at once."""
    Hq, Hkv, d, P, qo, kv = shape
    wl, out, lse, q, K, V = _contiguous_request(11 + Hq, Hq, Hkv, d, P, qo, kv)
    g = Hq // Hkv
    Qt = _f64(q).transpose(1, 0, 2)                                  # [Hq, qo, d]
    Kt = np.repeat(_f64(K), g, axis=1).transpose(1, 0, 2)            # [Hq, kv, d]
    Vt = np.repeat(_f64(V), g, axis=1).transpose(1, 0, 2)
    mask = torch.ones(qo, kv, dtype=torch.bool).tril(diagonal=kv - qo)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(Qt), torch.from_numpy(Kt), torch.from_numpy(Vt), attn_mask=mask,
        scale=wl.sm_scale).numpy().transpose(1, 0, 2)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    scores = torch.from_numpy(np.einsum("hic,hjc->hij", Qt, Kt) * wl.sm_scale)
    scores = scores.masked_fill(~mask, -math.inf)
    ref_lse = torch.logsumexp(scores, dim=-1).numpy().T
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_oracle_matches_torch_sdpa_is_causal_full_prompt():
    """qo_len == kv_len: the library's own causal rule applies unchanged."""
    Hq, Hkv, d, P, L = 4, 2, 32, 16, 37
    wl, out, _, q, K, V = _contiguous_request(21, Hq, Hkv, d, P, L, L)
    Qt = torch.from_numpy(_f64(q).transpose(1, 0, 2).copy())
    Kt = torch.from_numpy(np.repeat(_f64(K), 2, axis=1).transpose(1, 0, 2).copy())
    Vt = torch.from_numpy(np.repeat(_f64(V), 2, axis=1).transpose(1, 0, 2).copy())
    ref = torch.nn.functional.scaled_dot_product_attention(Qt, Kt, Vt, is_causal=True,
                                                           scale=wl.sm_scale).numpy().transpose(1, 0, 2)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_weights_sum_to_one_and_masked_weights_zero():
    wl = make_random_workload(31, 4, 2, 16, 4, [(6, 19), (1, 9)], extra_pages=2)
    pool = oracle_pool(wl)
    oracle_step(wl, pool, 0)
    t = wl.step_table(0)
    q, _, _ = wl.step_inputs(0)
    for row in range(7):
        r = 0 if row < 6 else 1
        kv = 19 if r == 0 else 9
        pos = kv - (6 if r == 0 else 1) + (row if r == 0 else 0)
        for h in range(4):
            _, _, w = oracle.attention_keyrange(q, pool, t["qo_indptr"], t["kv_indptr"],
                                                t["page_indices"], t["last_page_len"], wl.sm_scale,
                                                4, row, h, 0, pos + 1, want_weights=True)
            assert np.all(w >= 0)
            assert abs(w.sum() - 1.0) <= 1e-12
    _, _, W = dense.attention(_bits(q), pool, t["qo_indptr"], t["kv_indptr"], t["page_indices"],
                              t["last_page_len"], True, wl.sm_scale, 4)
    W0 = W[0]                                       # [Hq, 6, 19]
    i = np.arange(6)[:, None]
    j = np.arange(19)[None, :]
    masked = np.broadcast_to(j > 19 - 6 + i, W0.shape)
    assert np.all(W0[masked] == 0.0)
    np.testing.assert_allclose(W0.sum(-1), 1.0, rtol=0, atol=1e-12)


def test_kv_len_one_returns_v_exactly():
    wl, out, lse, q, K, V = _contiguous_request(41, 4, 2, 64, 16, 1, 1)
    ref = np.repeat(_f64(V), 2, axis=1)[0]          # [Hq, d]
    assert np.array_equal(out[0], ref)
    s = np.einsum("hc,hc->h", _f64(q)[0], np.repeat(_f64(K), 2, axis=1)[0]) * wl.sm_scale
    np.testing.assert_allclose(lse[0], s, rtol=0, atol=1e-13)


def _pool_with_rows(wl, K, V):
    """Pool holding exactly the given K/V rows for the single request of wl."""
    pool = oracle.new_pool(wl.pool_shape(), SENTINEL_BF16)
    t = wl.step_table(0)
    kv = K.shape[0]
    oracle.kv_append(pool, K, V, [0, kv], t["page_indices"], t["kv_indptr"], t["last_page_len"])
    return pool, t


def test_identical_keys_give_mean_of_values():
    Hq, Hkv, d, P, kv = 2, 1, 16, 4, 11
    wl = make_random_workload(51, Hq, Hkv, d, P, [(1, kv)])
    K = wl.k_rows(0, 0, 1).repeat(kv, 1, 1)
    V = wl.v_rows(0, 0, kv)
    pool, t = _pool_with_rows(wl, K, V)
    q = wl.q_rows(0, 0, 1)
    out, _, _ = oracle.attention(q, pool, [0, 1], t["kv_indptr"], t["page_indices"],
                                 t["last_page_len"], True, wl.sm_scale, Hq)
    np.testing.assert_allclose(out[0], np.broadcast_to(_f64(V).mean(0)[0], (Hq, d)), rtol=0, atol=1e-12)


def test_single_dominant_key_selects_its_value():
    Hq, Hkv, d, P, kv, star = 1, 1, 16, 4, 9, 5
    wl = make_random_workload(61, Hq, Hkv, d, P, [(1, kv)])
    K = wl.k_rows(0, 0, kv)
    V = wl.v_rows(0, 0, kv)
    pool, t = _pool_with_rows(wl, K, V)
    q = (K[star:star + 1].float() * 100.0).to(torch.bfloat16)
    out, _, _ = oracle.attention(q, pool, [0, 1], t["kv_indptr"], t["page_indices"],
                                 t["last_page_len"], False, 1.0, Hq)
    np.testing.assert_allclose(out[0, 0], _f64(V)[star, 0], rtol=0, atol=1e-9)


def test_noncausal_equals_causal_for_decode():
    wl = make_random_workload(71, 4, 2, 32, 16, [(1, 40), (1, 1), (1, 17)])
    pool = oracle_pool(wl)
    out_c, lse_c, _ = oracle_step(wl, pool, 0)
    t = wl.step_table(0)
    q, _, _ = wl.step_inputs(0)
    out_n, lse_n, _ = oracle.attention(q, pool, t["qo_indptr"], t["kv_indptr"], t["page_indices"],
                                       t["last_page_len"], False, wl.sm_scale, 4)
    assert np.array_equal(out_c, out_n) and np.array_equal(lse_c, lse_n)


def _run_all_steps(wl):
    pool = oracle_pool(wl)
    outs = []
    for k in range(len(wl.steps)):
        outs.append(oracle_step(wl, pool, k))
    return pool, outs


@pytest.mark.parametrize("L,C,Hq,Hkv,d", [(64, 16, 4, 2, 64), (2048, 512, 2, 1, 16), (100, 37, 3, 1, 8)])
def test_chunked_prefill_equals_one_shot(L, C, Hq, Hkv, d):
    """#correctness: after ceil(L/C) chunks the cache is byte-identical to a
    one-shot prefill and every prompt token's attention output is the same."""
    seed = 81
    wc = make_prompt_workload(L, C, Hq, Hkv, d, 16, seed)
    wo = make_prompt_workload(L, L, Hq, Hkv, d, 16, seed)
    assert wc.num_pages == wo.num_pages and np.array_equal(wc.seqs[0].pages, wo.seqs[0].pages)
    pc, oc = _run_all_steps(wc)
    po, oo = _run_all_steps(wo)
    assert len(oc) == -(-L // C) and len(oo) == 1
    assert np.array_equal(pc, po)
    # sentinel everywhere outside the prompt's L token slots
    touched = np.zeros(pc.shape[0], bool)
    touched[wc.seqs[0].pages] = True
    assert np.all(pc[~touched] == SENTINEL_BF16)
    n_written = int(np.count_nonzero(pc != SENTINEL_BF16))
    assert n_written == L * 2 * Hkv * d
    chunk_out = np.concatenate([o[0] for o in oc], 0)
    np.testing.assert_allclose(chunk_out, oo[0][0], rtol=0, atol=1e-12)
    # FLOP invariant (#flops): same number of causal pairs either way
    assert sum(o[2] for o in oc) == oo[0][2] == L * (L + 1) // 2


def test_tiny_mixed_chunk_steps_match_one_shot_rows():
    """The tiny mixed workload: 4 steps of a 16-token chunk + 2 advancing decodes.
    The prompt rows of every step equal the one-shot prefill rows; the decodes
    equal a direct decode at the same kv_len."""
    wl = make_workload("tiny_mixed")
    pool, outs = _run_all_steps(wl)
    wo = make_prompt_workload(64, 64, 4, 2, 64, 16, wl.seed)
    # same values, different page ids: compare outputs only
    wo.seqs[0].pages = wl.seqs[0].pages.copy()
    wo.num_pages = wl.num_pages
    _, oo = _run_all_steps(wo)
    prompt = np.concatenate([o[0][:16] for o in outs], 0)
    np.testing.assert_allclose(prompt, oo[0][0], rtol=0, atol=1e-12)


def test_softmax_merge_of_cache_and_chunk_equals_full():
    """#correctness: attn_i = softmax_merge(scores over the cache, scores over the
    chunk) . [V_cache; V_chunk]."""
    wl = make_workload("tiny_mixed")
    pool = oracle_pool(wl)
    for k in range(len(wl.steps)):
        oracle_step(wl, pool, k)
        t = wl.step_table(k)
        q, _, _ = wl.step_inputs(k)
        args = (q, pool, t["qo_indptr"], t["kv_indptr"], t["page_indices"], t["last_page_len"],
                wl.sm_scale, 4)
        cached = 16 * k
        for i in range(16):
            pos = cached + i
            for h in range(4):
                of, lf, _ = oracle.attention_keyrange(*args, i, h, 0, pos + 1)
                oa, la, _ = oracle.attention_keyrange(*args, i, h, 0, cached)
                ob, lb, _ = oracle.attention_keyrange(*args, i, h, cached, pos + 1)
                om, lm = oracle.softmax_merge(np.stack([oa, ob]), np.array([la, lb]))
                np.testing.assert_allclose(om, of, rtol=0, atol=1e-12)
                assert abs(lm - lf) <= 1e-12
                if k == 0:
                    assert la == -math.inf      # empty cache part
    rng = np.random.default_rng(5)
    t = wl.step_table(len(wl.steps) - 1)
    q, _, _ = wl.step_inputs(len(wl.steps) - 1)
    args = (q, pool, t["qo_indptr"], t["kv_indptr"], t["page_indices"], t["last_page_len"],
            wl.sm_scale, 4)
    for _ in range(20):                         # random three-way splits of a decode row
        row, h, kv = 16, int(rng.integers(4)), 43
        a, b = sorted(rng.integers(0, kv + 1, 2))
        parts = [oracle.attention_keyrange(*args, row, h, lo, hi) for lo, hi in ((0, a), (a, b), (b, kv))]
        om, lm = oracle.softmax_merge(np.stack([p[0] for p in parts]), np.array([p[1] for p in parts]))
        of, lf, _ = oracle.attention_keyrange(*args, row, h, 0, kv)
        np.testing.assert_allclose(om, of, rtol=0, atol=1e-12)
        assert abs(lm - lf) <= 1e-12


def test_page_permutation_invariance():
    """Attention does not depend on which pool pages hold a request."""
    reqs = [(3, 20), (1, 33)]
    wa = make_random_workload(91, 4, 2, 16, 4, reqs, num_pages=40)
    wb = make_random_workload(91, 4, 2, 16, 4, reqs, num_pages=40)
    wb.seqs[0].pages = np.arange(len(wb.seqs[0].pages), dtype=np.int32) + 7
    wb.seqs[1].pages = np.arange(len(wb.seqs[1].pages), dtype=np.int32)[::-1].copy() + 20
    oa, la, _ = oracle_step(wa, oracle_pool(wa), 0)
    ob, lb, _ = oracle_step(wb, oracle_pool(wb), 0)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb)


def test_hnd_layout_properties():
    """"Disaggregated prefill and decode", "Sharded KV cache transfers": HND puts
    the head dimension before the tokens, so a page is one contiguous block and
    each head's slice of a page is contiguous.  Checked on the flat bytes."""
    num_pages, Hkv, P, d, page = 6, 3, 4, 2, 4
    pool = oracle.new_pool((num_pages, 2, Hkv, P, d), SENTINEL_BF16)
    # distinct exact small integers as bf16 tags: value = 1 + ((kv*Hkv + h)*P + t)*d + c
    tag = np.zeros((2, P, Hkv, d), np.float32)
    for kv in range(2):
        for t in range(P):
            for h in range(Hkv):
                for c in range(d):
                    tag[kv, t, h, c] = 1 + ((kv * Hkv + h) * P + t) * d + c
    kb = torch.from_numpy(tag[0]).to(torch.bfloat16)
    vb = torch.from_numpy(tag[1]).to(torch.bfloat16)
    oracle.kv_append(pool, kb, vb, [0, P], [page], [0, 1], [P])
    flat = pool.reshape(-1)
    vals = torch.from_numpy(flat.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    written = np.nonzero(flat != SENTINEL_BF16)[0]
    page_elems = 2 * Hkv * P * d
    assert written.min() == page * page_elems and written.max() == (page + 1) * page_elems - 1
    assert len(written) == page_elems                 # the page is one dense block
    block = vals[page * page_elems:(page + 1) * page_elems]
    at = 0
    for kv in range(2):                               # K block before V block
        for h in range(Hkv):                          # heads in order ...
            run = block[at:at + P * d]                # ... each a contiguous run of P*d
            expect = [tag[kv, t, h, c] for t in range(P) for c in range(d)]   # tokens in order
            assert list(run) == expect
            at += P * d


def test_io_overhead_worked_example():
    """#io-overhead: bytes the append writes for one chunk, times the layers,
    equals the page's printed 67,108,864 B."""
    g = _golden("io_overhead.json")
    C, layers, n_h, d_h = g["C"], g["L_layers"], g["n_h"], g["d_h"]
    P = 16
    wl = make_prompt_workload(C, C, n_h, n_h, d_h, P, 7, num_pages=2 * C // P)
    pool = oracle.new_pool(wl.pool_shape(), SENTINEL_BF16)
    before = pool.copy()
    t = wl.step_table(0)
    _, kn, vn = wl.step_inputs(0)
    oracle.kv_append(pool, kn, vn, t["qo_indptr"], t["page_indices"], t["kv_indptr"], t["last_page_len"])
    bytes_per_layer = int(np.count_nonzero(pool != before)) * 2
    assert bytes_per_layer * layers == g["bytes"]


def test_flop_invariant_worked_example():
    """#flops: sum over chunks of attended pairs = L(L+1)/2, and
    4 d Hq pairs gives the printed-formula FLOPs for L=2048."""
    g = _golden("flops.json")
    L, C = g["L"], g["C"]
    wc = make_prompt_workload(L, C, 1, 1, 8, 16, 3)
    wo = make_prompt_workload(L, L, 1, 1, 8, 16, 3)
    pc = sum(o[2] for o in _run_all_steps(wc)[1])
    po = _run_all_steps(wo)[1][0][2]
    assert pc == po == g["pairs"]
    assert 4 * g["d"] * g["Hq"] * pc == g["attention_flops"]


def test_chunk_schedule_worked_example():
    g = _golden("chunk_schedule.json")
    sched = chunk_schedule(g["L"], g["C"])
    assert [[a, b - 1] for a, b in sched] == g["chunks_inclusive"]


def test_oracle_rejects_bad_tables():
    pool = oracle.new_pool((4, 2, 1, 4, 8), SENTINEL_BF16)
    k = torch.zeros(2, 1, 8, dtype=torch.bfloat16)
    with pytest.raises(oracle.OracleError):          # page id out of range
        oracle.kv_append(pool, k, k, [0, 2], [9], [0, 1], [2])
    with pytest.raises(oracle.OracleError):          # qo_len > kv_len
        oracle.kv_append(pool, k, k, [0, 2], [1], [0, 1], [1])
    with pytest.raises(oracle.OracleError):          # last_page_len outside [1, P]
        oracle.kv_append(pool, k, k, [0, 2], [1], [0, 1], [5])


def test_sampled_rows_match_full_run():
    wl = make_workload("tiny_mixed")
    pool = oracle_pool(wl)
    full, lse, _ = oracle_step(wl, pool, 0)
    t = wl.step_table(0)
    q, _, _ = wl.step_inputs(0)
    sel = [17, 0, 5, 16]
    part, plse, _ = oracle.attention(q, pool, t["qo_indptr"], t["kv_indptr"], t["page_indices"],
                                     t["last_page_len"], True, wl.sm_scale, 4, sel_rows=sel)
    assert np.array_equal(part, full[sel]) and np.array_equal(plse, lse[sel])


# ------------------------------------------------------------- prefix caching
def test_prefix_cache_schedule_worked_example():
    """#prefix-cache-interaction: with the 1024-token system prompt cached, the
    2048-token prompt runs 2 chunks of 512 (user query 0-511, 512-1023)
    instead of 4."""
    g = _golden("prefix_cache_schedule.json")
    L, sp, C = g["system_prompt"] + g["user_query"], g["system_prompt"], g["C"]
    assert len(chunk_schedule(L, C)) == g["chunks_without_cache"]
    hit = chunk_schedule(L, C, cached=sp)
    assert [[a - sp, b - 1 - sp] for a, b in hit] == g["user_chunks_inclusive"]


def _shared_tiny(seed=61, Hq=4, Hkv=2, d=16, P=4):
    # prefix of 12 tokens (3 pages) shared by a prompt chunk, a longer prompt
    # chunk with cached tokens of its own, and three decodes
    return make_shared_prefix_workload("shared_tiny", Hq, Hkv, d, P, seed, 12,
                                       [(5, 17), (6, 27)], [13, 20, 31])


def test_shared_prefix_pages_equal_private_copies():
    """#prefix-cache-interaction: a prefix-cache hit only changes where the
    cached keys come from.  Requests that read one physical copy of the prefix
    pages give exactly the outputs of requests that each hold a private copy
    of the same values, and the step's append leaves the shared pages as they
    were."""
    ws = _shared_tiny()
    pool = oracle_pool(ws)
    shared_pages = ws.seqs[0].pages
    before = pool[shared_pages].copy()
    out_s, lse_s, _ = oracle_step(ws, pool, 0)
    assert np.array_equal(pool[shared_pages], before)
    # private copies: same values, each request's prefix in pages of its own
    wp = copy.copy(ws)
    wp.seqs = [type(s)(s.length, s.pages.copy(), s.prefix, s.prefix_len) for s in ws.seqs]
    nxt = ws.num_pages
    for s in wp.seqs[1:]:
        n = len(shared_pages)
        s.pages[:n] = np.arange(nxt, nxt + n)
        nxt += n
    wp.num_pages = nxt
    ppool = oracle.new_pool(wp.pool_shape(), SENTINEL_BF16)
    for i in range(1, len(wp.seqs)):   # each private copy gets the prefix rows
        n = wp.seqs[i].prefix_len
        t = wp._table([(i, n, n)])
        oracle.kv_append(ppool, ws.k_rows(0, 0, n), ws.v_rows(0, 0, n), t["qo_indptr"],
                         t["page_indices"], t["kv_indptr"], t["last_page_len"])
    it = ws.initial_table()
    k0, v0 = ws.initial_kv()
    nprefix = ws.seqs[1].prefix_len
    # the sequences' own cached tokens (after the prefix owner's span)
    own = wp._table([(s, hi - lo, hi) for s, lo, hi in ws.initial_spans() if s != 0])
    oracle.kv_append(ppool, k0[nprefix:], v0[nprefix:], own["qo_indptr"], own["page_indices"],
                     own["kv_indptr"], own["last_page_len"])
    assert it["qo_indptr"][1] == nprefix
    out_p, lse_p, _ = oracle_step(wp, ppool, 0)
    assert np.array_equal(out_s, out_p) and np.array_equal(lse_s, lse_p)


def test_shared_prefix_matches_torch_sdpa():
    """Library attention on K/V taken from the generator (shared prefix rows,
    then each request's own rows), not from the pool: pins the gather of
    shared pages and the causal offset of a chunk after a prefix hit."""
    ws = _shared_tiny(seed=62, Hq=6, Hkv=2, d=32, P=4)
    pool = oracle_pool(ws)
    out, lse, _ = oracle_step(ws, pool, 0)
    q, _, _ = ws.step_inputs(0)
    g = ws.group_size
    row = 0
    for r in ws.steps[0].requests:
        K, V = ws.k_rows(r.seq, 0, r.kv_len), ws.v_rows(r.seq, 0, r.kv_len)
        Qt = torch.from_numpy(_f64(q[row:row + r.qo_len]).transpose(1, 0, 2).copy())
        Kt = torch.from_numpy(np.repeat(_f64(K), g, axis=1).transpose(1, 0, 2).copy())
        Vt = torch.from_numpy(np.repeat(_f64(V), g, axis=1).transpose(1, 0, 2).copy())
        mask = torch.ones(r.qo_len, r.kv_len, dtype=torch.bool).tril(diagonal=r.kv_len - r.qo_len)
        ref = torch.nn.functional.scaled_dot_product_attention(Qt, Kt, Vt, attn_mask=mask,
                                                               scale=ws.sm_scale)
        np.testing.assert_allclose(out[row:row + r.qo_len], ref.numpy().transpose(1, 0, 2),
                                   rtol=0, atol=1e-12)
        row += r.qo_len
    assert row == out.shape[0]


def test_prefix_hit_equals_recompute():
    """#prefix-cache-interaction with #correctness: the 2 suffix chunks run
    after a prefix hit give the same outputs as the last 2 of the 4 chunks of
    the same prompt computed from scratch, and the pages end up holding the
    same bytes."""
    L, C, sp, Hq, Hkv, d, P = 64, 16, 32, 4, 2, 16, 4
    # A: prefix hit -- the system prompt (seq 0) is cached and shared; the
    # prompt (seq 1) runs its two suffix chunks as two steps
    wa = make_shared_prefix_workload("hit", Hq, Hkv, d, P, 71, sp, [(C, sp + C)], [])
    wa.seqs[1].length = L
    extra = np.arange(wa.num_pages, wa.num_pages + (L - sp - C) // P, dtype=np.int32)
    wa.seqs[1].pages = np.concatenate([wa.seqs[1].pages, extra])
    wa.num_pages += len(extra)
    wa.steps = [Step([Request(1, b - a, b)]) for a, b in chunk_schedule(L, C, cached=sp)]
    pa = oracle_pool(wa)
    outs_a = [oracle_step(wa, pa, k) for k in range(len(wa.steps))]
    # B: the same prompt values from scratch, 4 chunks, private pages
    wb = make_prompt_workload(L, C, Hq, Hkv, d, P, 71, num_pages=wa.num_pages)
    wb.seqs[0].pages = wa.seqs[1].pages.copy()
    wb.rows_into = lambda out, seq, kind, lo, hi: wa.rows_into(out, 1, kind, lo, hi)
    pb = oracle_pool(wb)
    outs_b = [oracle_step(wb, pb, k) for k in range(len(wb.steps))]
    assert len(outs_a) == 2 and len(outs_b) == 4
    for (oa, la, na), (ob, lb, nb) in zip(outs_a, outs_b[2:]):
        np.testing.assert_allclose(oa, ob, rtol=0, atol=1e-12)
        np.testing.assert_allclose(la, lb, rtol=0, atol=1e-12)
        assert na == nb
    assert np.array_equal(pa[wa.seqs[1].pages], pb[wb.seqs[0].pages])


# --------------------------------------------------------------- tree masks
TREE_CASES = [
    # (seed, Hq, Hkv, d, P, trees (nodes, cached, roots), decodes, prompts)
    (201, 4, 2, 16, 4, [(9, 14, 1), (1, 5, 1), (33, 40, 3)], [11], [(6, 20)]),
    (202, 6, 2, 8, 16, [(40, 3, 1), (17, 0, 17), (64, 70, 2)], [], []),
    (203, 2, 2, 8, 4, [(5, 0, 1), (70, 9, 1)], [3, 30], [(3, 3)]),
]


def _tree_run(case):
    seed, Hq, Hkv, d, P, trees, decodes, prompts = case
    wl = make_tree_workload(f"tree_{seed}", Hq, Hkv, d, P, seed, trees, decodes, prompts)
    pool = oracle_pool(wl)
    out, lse, pairs = oracle_step(wl, pool, 0)
    return wl, pool, out, lse, pairs


@pytest.mark.parametrize("case", TREE_CASES, ids=lambda c: f"seed{c[0]}")
def test_tree_mask_matches_dense_bruteforce(case):
    """The C oracle's tree visibility against the NumPy brute force's masked
    score matrix (unpacked mask bits, strict lower triangle, diagonal)."""
    wl, pool, out, lse, _ = _tree_run(case)
    t = wl.step_table(0)
    q, _, _ = wl.step_inputs(0)
    dout, dlse, _ = dense.attention(_bits(q), pool, t["qo_indptr"], t["kv_indptr"], t["page_indices"],
                                    t["last_page_len"], True, wl.sm_scale, wl.num_qo_heads,
                                    tree_mask=wl.tree_mask(0))
    np.testing.assert_allclose(out, dout, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, dlse, rtol=0, atol=1e-12)


@pytest.mark.parametrize("case", TREE_CASES, ids=lambda c: f"seed{c[0]}")
def test_tree_node_equals_its_branch_as_a_sequence(case):
    """EAGLE: a draft token is verified against the accepted prefix and its own
    branch.  Each tree node's output equals library attention (torch SDPA,
    fp64) of its query over the cached keys followed by the keys of its
    root-to-node path, walked from the parent array (not from the mask)."""
    wl, pool, out, lse, pairs = _tree_run(case)
    q, _, _ = wl.step_inputs(0)
    g = wl.group_size
    row, n_pairs = 0, 0
    for r in wl.steps[0].requests:
        cached = r.kv_len - r.qo_len
        K, V = wl.k_rows(r.seq, 0, r.kv_len), wl.v_rows(r.seq, 0, r.kv_len)
        par = r.parents if r.parents is not None else np.arange(r.qo_len) - 1
        for i in range(r.qo_len):
            path, j = [], i
            while j >= 0:
                path.append(j)
                j = int(par[j])
            keys = list(range(cached)) + [cached + j for j in reversed(path)]
            n_pairs += len(keys)
            Kp = torch.from_numpy(np.repeat(_f64(K[keys]), g, axis=1).transpose(1, 0, 2).copy())
            Vp = torch.from_numpy(np.repeat(_f64(V[keys]), g, axis=1).transpose(1, 0, 2).copy())
            Qi = torch.from_numpy(_f64(q[row + i:row + i + 1]).transpose(1, 0, 2).copy())
            ref = torch.nn.functional.scaled_dot_product_attention(Qi, Kp, Vp, scale=wl.sm_scale)
            np.testing.assert_allclose(out[row + i], ref.numpy()[:, 0], rtol=0, atol=1e-12)
            ref_lse = torch.logsumexp(torch.einsum("hqc,hkc->hqk", Qi, Kp) * wl.sm_scale, -1)
            np.testing.assert_allclose(lse[row + i], ref_lse.numpy()[:, 0], rtol=0, atol=1e-12)
        row += r.qo_len
    assert pairs == n_pairs


def test_chain_mask_equals_causal():
    """A mask row holding every earlier new token is the plain causal rule:
    outputs bit-identical to attention without a mask."""
    wl = make_random_workload(211, 4, 2, 16, 4, [(40, 47), (1, 9), (33, 33)], extra_pages=2)
    mask = np.concatenate([tree_mask_rows(np.arange(n) - 1, 2) for n in (40, 1, 33)], 0)
    pa, pb = oracle_pool(wl), oracle_pool(wl)
    oa, la, na = oracle_step(wl, pa, 0)
    ob, lb, nb = oracle_step(wl, pb, 0, tree_mask=mask)
    assert np.array_equal(oa, ob) and np.array_equal(la, lb) and na == nb


def test_tree_mask_arguments_checked():
    wl = make_random_workload(212, 2, 1, 8, 4, [(40, 41)], extra_pages=1)
    pool = oracle_pool(wl)
    t = wl.step_table(0)
    q, _, _ = wl.step_inputs(0)
    args = (q, pool, t["qo_indptr"], t["kv_indptr"], t["page_indices"], t["last_page_len"])
    with pytest.raises(oracle.OracleError):          # 40 new tokens need 2 words
        oracle.attention(*args, True, 0.3, 2, tree_mask=np.zeros((40, 1), np.uint32))
    with pytest.raises(oracle.OracleError):          # a tree mask needs the causal rule
        oracle.attention(*args, False, 0.3, 2, tree_mask=np.zeros((40, 2), np.uint32))


@pytest.mark.parametrize("case", TREE_CASES[:2], ids=lambda c: f"seed{c[0]}")
def test_tree_mask_bits_on_and_above_diagonal_are_ignored(case):
    """Only bits of earlier new tokens count: a token always sees itself and
    never a later token, whatever its row holds there.  Scrambling every bit
    on or above the diagonal (the self bit cleared or set, later bits random)
    leaves the outputs bit-identical."""
    wl, _, out, lse, pairs = _tree_run(case)
    mask = wl.tree_mask(0).copy()
    rng = np.random.default_rng(7)
    row = 0
    for r in wl.steps[0].requests:
        for i in range(r.qo_len):
            for j in range(i, 32 * mask.shape[1]):
                w, b = divmod(j, 32)
                if j == i or rng.random() < 0.5:
                    mask[row + i, w] ^= np.uint32(1 << b)
        row += r.qo_len
    pool = oracle_pool(wl)
    o2, l2, p2 = oracle_step(wl, pool, 0, tree_mask=mask)
    assert np.array_equal(out, o2) and np.array_equal(lse, l2) and pairs == p2
