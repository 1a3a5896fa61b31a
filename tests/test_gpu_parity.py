"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Both sides read the same seeded inputs from ``synth`` and each builds its own
page pool with its own append.  Acceptance (task statement of the method):
* kv_append and the page layout: bit-exact, sentinel bytes untouched;
* attention (bf16 in, fp32 accumulate, bf16 out) against the fp64 oracle:
  max |err| <= 1.5e-2 and mean |err| <= 2e-3; relative L2 <= 1e-2 as a
  stricter diagnostic; natural-log LSE within 1e-3 (the GPU sums fp32
  exponentials, so only fp32 rounding separates it from the fp64 value);
* GPU chunked vs one-shot prefill within 1e-2.
"""
import numpy as np
import pytest
import torch

import oracle
from synth import (SENTINEL_BF16, make_prefix_groups_workload, make_prompt_workload,
                   make_random_workload, make_shared_prefix_workload, make_tree_workload,
                   make_workload, tree_mask_rows)
from support import err_stats, oracle_pool, oracle_step

pytestmark = pytest.mark.gpu

MAX_ERR, MEAN_ERR, REL_L2, LSE_ERR = 1.5e-2, 2e-3, 1e-2, 1e-3


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _check(out, lse, ref, ref_lse, what):
    got = out.double().numpy()
    mx, mean, rel = err_stats(got, ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert mx <= MAX_ERR and mean <= MEAN_ERR and rel <= REL_L2, (what, mx, mean, rel)
    if lse is not None:
        le = np.abs(lse.double().numpy() - ref_lse).max()
        assert le <= LSE_ERR, (what, "lse", le)
    return mx, mean, rel


def _run_both(wl, dev, sel_rows=None, compare_pool=True, fused=False, groups=False):
    from gpu_support import compact, gpu_fill, gpu_step, new_pool, pool_bits
    cw, mapping = compact(wl)
    opool = oracle_pool(cw)
    gpool = new_pool(wl, dev)
    gpu_fill(wl, gpool, dev)
    stats = []
    for k in range(len(wl.steps)):
        out, lse = gpu_step(wl, gpool, k, dev, fused=fused, groups=groups)
        ref, ref_lse, _ = oracle_step(cw, opool, k, sel_rows=sel_rows)
        if sel_rows is not None:
            out, lse = out[sel_rows], lse[sel_rows]
        stats.append(_check(out, lse, ref, ref_lse, f"{wl.name} step {k}"))
    if compare_pool:
        orig = np.asarray(sorted(mapping), np.int64)
        new = np.asarray([mapping[int(p)] for p in orig], np.int64)
        g = pool_bits(gpool[torch.from_numpy(orig).to(dev)])
        assert np.array_equal(g, opool[new]), f"{wl.name}: page bytes differ"
        # pages no request owns stay sentinel
        untouched = torch.ones(wl.num_pages, dtype=torch.bool, device=dev)
        untouched[torch.from_numpy(orig).to(dev)] = False
        assert bool((gpool.view(torch.int16)[untouched] == SENTINEL_BF16).all())
    return stats


def test_tiny_mixed_all_steps_bit_exact_pool(dev):
    from gpu_support import gpu_fill, gpu_step, new_pool, pool_bits
    wl = make_workload("tiny_mixed")
    opool = oracle_pool(wl)
    gpool = new_pool(wl, dev)
    gpu_fill(wl, gpool, dev)
    for k in range(len(wl.steps)):
        out, lse = gpu_step(wl, gpool, k, dev)
        ref, ref_lse, _ = oracle_step(wl, opool, k)
        _check(out, lse, ref, ref_lse, f"tiny step {k}")
        assert np.array_equal(pool_bits(gpool), opool), f"pool differs after step {k}"


EDGE = [
    # (seed, Hq, Hkv, d, [(qo, kv), ...], causal)
    (101, 4, 4, 128, [(1, 1), (1, 17), (2, 2), (3, 40)], True),
    (102, 8, 1, 128, [(129, 300), (1, 5000), (0, 33), (128, 128)], True),
    (103, 12, 1, 128, [(37, 1000), (1, 4097), (1, 16)], True),
    (104, 6, 2, 64, [(5, 5), (17, 100), (1, 7)], True),
    (105, 16, 1, 128, [(300, 300), (1, 20000)], True),
    (106, 2, 2, 64, [(255, 1000), (1, 1)], True),
    (107, 8, 1, 128, [(129, 300), (1, 5000), (0, 33), (128, 128)], False),
    (108, 4, 2, 128, [(16, 16)] * 3 + [(1, 2049)] * 5, True),
    (109, 32, 8, 128, [(512, 2048)] + [(1, 1024 + 97 * i) for i in range(8)], True),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"seed{c[0]}")
def test_edge_cases(dev, case):
    seed, Hq, Hkv, d, reqs, causal = case
    wl = make_random_workload(seed, Hq, Hkv, d, 16, reqs, extra_pages=7)
    wl.causal = causal
    _run_both(wl, dev)


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 1, 128), (12, 1, 128), (16, 2, 64)])
def test_tensor_core_decode_tile_counts(dev, Hq, Hkv, d):
    """GQA decode runs as single-tile tensor-core items with S double-buffered:
    kv lengths around 128-key tile boundaries give 1..17 tiles per item, odd and
    even, full and ragged last tiles, split and unsplit requests."""
    kvs = [1, 2, 127, 128, 129, 200, 255, 256, 257, 384, 385, 1000, 2047, 2048, 2049]
    wl = make_random_workload(113 + Hq, Hq, Hkv, d, 16, [(1, kv) for kv in kvs], extra_pages=5)
    _run_both(wl, dev)


VERIFY = [
    # (Hq, Hkv, d, causal): verify batches (qo 2..16) mixed with decodes; long kv
    # forces many key splits, kv = 128k + small puts a split boundary inside
    # the last qo keys
    (32, 32, 128, True),
    (8, 2, 64, True),
    (32, 4, 128, True),
    (12, 1, 128, True),
    (16, 1, 128, False),
]


@pytest.mark.parametrize("case", VERIFY, ids=lambda c: f"Hq{c[0]}_Hkv{c[1]}_d{c[2]}_{'c' if c[3] else 'nc'}")
def test_verify_batches(dev, case):
    """Small multi-token requests (speculative-decoding verify) run as key-split
    items of the tensor-core decode kernel with one softmax_merge per token."""
    Hq, Hkv, d, causal = case
    vmax = min(16, 128 // (Hq // Hkv))
    qos = [q for q in (2, 3, 4, 7, 8, 16) if q <= vmax]
    reqs = [(q, kv) for q, kv in zip(qos * 2, [20000, 4097, 129, 3000, 8195, 640, 17, 20483, 2051, 520, 16, 12000])]
    reqs += [(1, 9000), (1, 130)]
    wl = make_random_workload(131 + Hq + d, Hq, Hkv, d, 16, reqs, extra_pages=9)
    wl.causal = causal
    _run_both(wl, dev)


SHORT = [
    # (seed, Hq, Hkv, d, [(qo, kv), ...], causal): requests whose rows fit two
    # 128-row Q tiles (verify cap < qo <= 256 / g) run on the single-CTA kernel,
    # key-split when long; qo = 256 / g + 1 is the first pair-prefill request
    (121, 8, 8, 128, [(17, 40000), (200, 3000), (256, 256), (257, 900), (1, 5000), (150, 50000)], True),
    (122, 32, 8, 128, [(17, 12000), (33, 33), (64, 7000), (65, 7000), (40, 300)], True),
    (123, 12, 1, 128, [(11, 30000), (20, 20), (21, 5000), (1, 3000)], True),
    (124, 8, 1, 128, [(100, 5000), (17, 17), (32, 9000)], False),
    (125, 16, 4, 64, [(40, 9000), (84, 84), (64, 64)], True),
]


@pytest.mark.parametrize("case", SHORT, ids=lambda c: f"seed{c[0]}")
def test_short_requests(dev, case):
    """Short multi-token requests: one or two Q tiles on the single-CTA kernel,
    key splits merged per token, against the oracle."""
    seed, Hq, Hkv, d, reqs, causal = case
    wl = make_random_workload(seed, Hq, Hkv, d, 16, reqs, extra_pages=7)
    wl.causal = causal
    _run_both(wl, dev)


def test_decode_kv_len_one_returns_v(dev):
    from gpu_support import gpu_fill, gpu_step, new_pool
    wl = make_random_workload(111, 8, 2, 128, 16, [(1, 1), (1, 1)])
    gpool = new_pool(wl, dev)
    gpu_fill(wl, gpool, dev)
    out, _ = gpu_step(wl, gpool, 0, dev)
    for r in range(2):
        v = wl.v_rows(r, 0, 1)[0]                          # [Hkv, d]
        expect = v.repeat_interleave(4, dim=0)             # head h reads kv head h // 4
        assert torch.equal(out[r], expect)


@pytest.mark.parametrize("name", ["mha_decode", "chunked_prefill_mixed", "gqa_decode_shard",
                                  "prefix_shared"])
def test_config_full_rows(dev, name):
    _run_both(make_workload(name), dev)


def test_long_prefill_sampled_rows(dev):
    """The long-prompt prefill batch (4 x 8192 new over 8192 cached, GQA 64/8,
    + 64 decodes) on ~1,100 rows checked one by one against the oracle:
    * prompt 0: one row in every 128-row Q tile (16 tokens x 8 heads each), at
      a rotating offset inside the tile, so every tile slot of every four-tile
      pair item, on both CTAs of the pair, is checked;
    * every prompt: the last row before and the first row after every 128-key
      tile boundary along the diagonal (the masked diagonal tiles and the key
      tile that is read as a whole for the first time), and the chunk's edges;
    * all 64 decode rows.
    The pool is compared byte for byte."""
    wl = make_workload("long_prefill")
    qo = 8192
    tpt = 128 // wl.group_size  # tokens per 128-row Q tile
    prompt_rows = [t * tpt + (7 * t) % tpt for t in range(qo // tpt)]
    for p in range(4):
        base = p * qo
        prompt_rows += [base, base + 1, base + qo - 1]
        for b in range(128, qo, 128):
            prompt_rows += [base + b - 1, base + b]
    decode_rows = list(range(4 * qo, 4 * qo + 64))
    sel = sorted(set(prompt_rows)) + decode_rows
    assert len(set(r // tpt for r in prompt_rows if r < qo)) == qo // tpt
    # the fused call, as the benchmark runs it: the prompts' new key tiles come
    # from k_new / v_new and are written into the pages by the prefill kernel
    _run_both(wl, dev, sel_rows=sel, fused=True)


@pytest.mark.parametrize("fused", [False, True])
def test_chunked_vs_one_shot_gpu(dev, fused):
    """#correctness on the GPU: 4 chunks of 512 vs one 2048-token prefill give
    a byte-identical cache and outputs within 1e-2 (two calls, or the fused
    call whose prefill kernel appends the chunk itself)."""
    from gpu_support import gpu_fill, gpu_step, new_pool, pool_bits
    wc = make_prompt_workload(2048, 512, 32, 8, 128, 16, 1003, decodes=[1500, 3000])
    wo = make_prompt_workload(2048, 2048, 32, 8, 128, 16, 1003)
    wo.num_pages = wc.num_pages
    wo.seqs[0].pages = wc.seqs[0].pages.copy()
    pc, po = new_pool(wc, dev), new_pool(wo, dev)
    gpu_fill(wc, pc, dev)
    gpu_fill(wo, po, dev)
    chunks = [gpu_step(wc, pc, k, dev, fused=fused)[0][:512] for k in range(4)]
    one, _ = gpu_step(wo, po, 0, dev, fused=fused)
    pages = torch.from_numpy(wc.seqs[0].pages.astype(np.int64)).to(dev)
    assert np.array_equal(pool_bits(pc[pages]), pool_bits(po[pages]))
    diff = (torch.cat(chunks, 0).double() - one.double()).abs().max().item()
    assert diff <= 1e-2, diff


@pytest.mark.parametrize("name", ["tiny_mixed", "mha_decode", "chunked_prefill_mixed",
                                  "gqa_decode_shard", "prefix_shared"])
def test_append_attention_against_oracle(dev, name):
    """The fused call (append, then attention launched behind it as
    programmatic dependent launches) against the oracle: pool bytes bit-exact,
    outputs within the attention tolerance, every step."""
    _run_both(make_workload(name), dev, fused=True)


@pytest.mark.parametrize("case", [EDGE[1], EDGE[4], EDGE[7], EDGE[8]], ids=lambda c: f"seed{c[0]}")
def test_append_attention_equals_two_calls(dev, case):
    """Same kernels, same plan: the fused call and kv_append + batch_attention
    give bit-identical pools, outputs and LSE (only the schedule differs)."""
    from gpu_support import gpu_fill, gpu_step, new_pool, pool_bits
    seed, Hq, Hkv, d, reqs, causal = case
    wl = make_random_workload(seed, Hq, Hkv, d, 16, reqs, extra_pages=7)
    wl.causal = causal
    pa, pb = new_pool(wl, dev), new_pool(wl, dev)
    gpu_fill(wl, pa, dev)
    gpu_fill(wl, pb, dev)
    for k in range(len(wl.steps)):
        oa, la = gpu_step(wl, pa, k, dev, fused=True)
        ob, lb = gpu_step(wl, pb, k, dev, fused=False)
        assert torch.equal(oa.view(torch.int16), ob.view(torch.int16)), f"step {k}: out differs"
        assert torch.equal(la, lb), f"step {k}: lse differs"
    assert np.array_equal(pool_bits(pa), pool_bits(pb))


FUSED_PREFILL = [
    # (seed, Hq, Hkv, head_dim, [(qo, kv), ...], causal): prefill requests with
    # their append fused in -- head_dim 128 on the CTA-pair kernel, head_dim 64
    # on the single-CTA kernel.  Cached prefixes that are whole 128-key tiles
    # (every new tile read from k_new) and that are not (the tile holding both
    # cached and new keys is read from the pages after the append); ragged last
    # tiles; requests of several items; requests whose new keys never fill a
    # whole 128-aligned tile (nothing fused); decode and short requests beside
    # them.
    (141, 32, 8, 128, [(512, 2048), (300, 1000), (129, 129), (1, 3000), (40, 700)], True),  # g 4
    (142, 64, 8, 128, [(1000, 3000), (77, 207), (1, 500), (33, 33)], True),                # g 8
    (143, 12, 1, 128, [(333, 4000), (150, 150), (21, 600), (1, 900)], True),               # g 12
    (144, 16, 1, 128, [(600, 2500), (200, 1111), (1, 40)], True),                          # g 16
    (145, 8, 8, 128, [(700, 1700), (257, 300), (1, 64)], True),                            # g 1
    (146, 32, 8, 128, [(300, 900), (513, 513), (1, 100)], False),                          # not causal
    (147, 8, 4, 64, [(512, 2048), (300, 1000), (129, 129), (1, 3000), (40, 700)], True),   # g 2
    (148, 32, 4, 64, [(1000, 3000), (77, 207), (1, 500), (33, 33), (17, 400)], True),     # g 8
    (149, 8, 8, 64, [(700, 1700), (257, 300), (1, 64)], False),                            # g 1, not causal
]


@pytest.mark.parametrize("case", FUSED_PREFILL, ids=lambda c: f"seed{c[0]}")
def test_fused_prefill_append(dev, case):
    """The fused call with the prefill kernel appending its chunk's own key
    tiles ("Chunked prefill", #io-overhead): pool bytes bit-exact against the
    oracle's append (and sentinel pages untouched), outputs within tolerance."""
    import decode_attention_append_gb300 as daa
    seed, Hq, Hkv, d, reqs, causal = case
    assert daa.prefill_append_fusion()
    wl = make_random_workload(seed, Hq, Hkv, d, 16, reqs, extra_pages=9)
    wl.causal = causal
    _run_both(wl, dev, fused=True)


@pytest.mark.parametrize("case", [FUSED_PREFILL[i] for i in (0, 2, 5, 6, 7)],
                         ids=lambda c: f"seed{c[0]}")
def test_fused_prefill_append_matches_unfused_bitwise(dev, case):
    """Fusion on and off run the same arithmetic on the same bits (a tile read
    from k_new holds exactly the bytes the append writes): identical outputs,
    LSE and pools."""
    import decode_attention_append_gb300 as daa
    from gpu_support import gpu_fill, gpu_step, new_pool, pool_bits
    seed, Hq, Hkv, d, reqs, causal = case
    wl = make_random_workload(seed, Hq, Hkv, d, 16, reqs, extra_pages=9)
    wl.causal = causal
    res = []
    try:
        for on in (False, True):
            daa.set_prefill_append_fusion(on)
            pool = new_pool(wl, dev)
            gpu_fill(wl, pool, dev)
            out, lse = gpu_step(wl, pool, 0, dev, fused=True)
            res.append((out, lse, pool_bits(pool)))
    finally:
        daa.set_prefill_append_fusion(True)
    (oa, la, pa), (ob, lb, pb) = res
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la, lb)
    assert np.array_equal(pa, pb)


SHARED = [
    # (seed, Hq, Hkv, d, prefix_len, prompt chunks (qo, kv), decode kv_lens)
    # g = 2: CUDA-core decode splits, a 7-token verify request, pair prefill
    (91, 8, 4, 128, 48, [(40, 100), (7, 60)], [49, 120, 300]),
    # g = 4, head_dim 64: tensor-core decode and the single-CTA prefill kernel
    (92, 16, 4, 64, 64, [(100, 250)], [65, 1000, 77]),
    # g = 12: twenty decodes over one 256-token prefix, a chunk right after it
    (93, 12, 1, 128, 256, [(12, 268), (300, 556)], [257 + 37 * i for i in range(20)]),
]


@pytest.mark.parametrize("case", SHARED, ids=lambda c: f"seed{c[0]}")
@pytest.mark.parametrize("fused", [False, True])
def test_shared_prefix_pages(dev, case, fused):
    """Prefix-cache hits ("Chunked prefill", #prefix-cache-interaction): every
    request reads the same physical prefix pages; outputs match the oracle and
    the append leaves the shared pages untouched (pool bit-exact)."""
    seed, Hq, Hkv, d, sp, prompts, decodes = case
    wl = make_shared_prefix_workload(f"shared_{seed}", Hq, Hkv, d, 16, seed, sp, prompts, decodes)
    _run_both(wl, dev, fused=fused)


@pytest.mark.parametrize("case", SHARED, ids=lambda c: f"seed{c[0]}")
def test_shared_prefix_groups_small_cases(dev, case):
    """The same batches through the shared-prefix call: prefixes under one
    128-key tile are planned as without groups, the 256-token one is attended
    once for the group's decodes and verify request."""
    seed, Hq, Hkv, d, sp, prompts, decodes = case
    wl = make_shared_prefix_workload(f"shared_{seed}", Hq, Hkv, d, 16, seed, sp, prompts, decodes)
    _run_both(wl, dev, groups=True)


def _dec(kv0, n, step):
    return [(1, kv0 + step * i) for i in range(n)]


CASCADE = [
    # (seed, Hq, Hkv, d, layout, causal).  Runs of decode / verify / short
    # requests inside a group attend its shared 128-key tiles once; a prefill
    # request in a group ends a run and keeps the prefix in its own items.
    # g = 4, head_dim 128: decodes, a verify and a short request share a
    # 1024-token prefix (pair kernel group items, tensor-core decode splits
    # after the prefix); a prompt chunk splits the group into two runs; a second
    # group whose prefix (400 tokens) is not whole tiles; solo requests between
    (401, 32, 8, 128, [("group", 1024, _dec(1025, 12, 131) + [(7, 1500), (40, 2000), (200, 1400)]
                        + _dec(3000, 5, 17)),
                       ("solo", 1, 777), ("solo", 100, 900),
                       ("group", 400, _dec(401, 4, 300) + [(9, 1000)])], True),
    # g = 1 (MHA): CUDA-core decode splits after the prefix; 40 rows of one Q
    # tile in the group item
    (402, 16, 16, 128, [("group", 512, _dec(513, 40, 61))], True),
    # g = 8, head_dim 64: group items on the single-CTA prefill kernel; a
    # member whose only own key is its new token (kv = prefix + 1)
    (403, 16, 2, 64, [("group", 384, _dec(385, 9, 203) + [(20, 700), (3, 387)])], True),
    # g = 12: 30 decodes and a 10-token verify request over 1024 shared keys
    (404, 12, 1, 128, [("solo", 1, 5000), ("group", 1024, _dec(1100, 30, 97) + [(10, 2500)])], True),
    # not causal: every row sees all its keys, the shared ones included
    (405, 32, 8, 128, [("group", 640, _dec(700, 8, 211) + [(12, 900), (64, 1200)])], False),
    # a group of one member and a group with a prefix under one tile: no group
    # items (the plan of the plain call)
    (406, 32, 8, 128, [("group", 1024, [(1, 2000)]), ("group", 96, _dec(100, 6, 50))], True),
]


@pytest.mark.parametrize("case", CASCADE, ids=lambda c: f"seed{c[0]}")
@pytest.mark.parametrize("fused", [False, True])
def test_shared_prefix_groups(dev, case, fused):
    """daa_batch_attention_shared_prefix / daa_append_attention_shared_prefix
    ("Chunked prefill", #prefix-cache-interaction with the softmax_merge of
    #correctness): outputs and LSE against the oracle, pool bit-exact."""
    seed, Hq, Hkv, d, layout, causal = case
    wl = make_prefix_groups_workload(f"groups_{seed}", Hq, Hkv, d, 16, seed, layout, causal=causal)
    _run_both(wl, dev, fused=fused, groups=True)


def test_shared_prefix_groups_match_plain_call(dev):
    """The shared-prefix call and the plain call agree row by row (only the
    fp32 summation order differs); groups that yield no group item give the
    plain call's bits exactly."""
    from gpu_support import gpu_fill, gpu_step, new_pool
    for seed, exact in ((401, False), (406, True)):
        case = next(c for c in CASCADE if c[0] == seed)
        wl = make_prefix_groups_workload(f"groups_{seed}", *case[1:4], 16, seed, case[4])
        outs = []
        for groups in (False, True):
            pool = new_pool(wl, dev)
            gpu_fill(wl, pool, dev)
            outs.append(gpu_step(wl, pool, 0, dev, groups=groups))
        (oa, la), (ob, lb) = outs
        if exact:
            assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
            assert torch.equal(la, lb)
        else:
            assert (oa.float() - ob.float()).abs().max().item() <= 1e-2
            assert (la - lb).abs().max().item() <= 1e-4


def test_prefix_shared_workload_groups(dev):
    _run_both(make_workload("prefix_shared"), dev, groups=True)


TREES = [
    # (seed, Hq, Hkv, d, trees (nodes, cached, roots), decode kv_lens, prompts (qo, kv))
    # g = 1: every tree is a key-split verify item; CUDA-core decodes beside them
    (301, 8, 8, 128, [(16, 300, 1), (9, 1000, 2), (5, 40, 1)], [100, 700], []),
    # g = 4: a 16-node tree as a verify item, larger trees on the pair prefill
    # kernel, a plain chunk in the same masked batch (10 mask words per row)
    (302, 32, 8, 128, [(64, 1500, 1), (40, 200, 3), (16, 5000, 1), (100, 30, 1)], [900], [(300, 1200)]),
    # g = 8, head_dim 64: verify item and the single-CTA prefill kernel
    (303, 16, 2, 64, [(48, 700, 1), (12, 90, 1)], [64], []),
    # g = 12: 10 tokens per Q tile; a 10-node verify item, a 33-node tree
    (304, 12, 1, 128, [(10, 3000, 1), (33, 4000, 2)], [2000], []),
]


@pytest.mark.parametrize("case", TREES, ids=lambda c: f"seed{c[0]}")
def test_tree_verify(dev, case):
    """Draft-tree verification ("Accelerating Sonar through speculation",
    EAGLE): every new token attends to the cached prefix and its own branch of
    the tree, through daa_batch_attention_tree, against the oracle."""
    seed, Hq, Hkv, d, trees, decodes, prompts = case
    wl = make_tree_workload(f"tree_{seed}", Hq, Hkv, d, 16, seed, trees, decodes, prompts)
    _run_both(wl, dev)


def test_tree_verify_workload(dev):
    _run_both(make_workload("tree_verify"), dev)


def test_chain_mask_matches_unmasked_bitwise(dev):
    """A mask row selecting every earlier new token is the causal rule: the
    tree variant of the kernels returns the plain call's bits exactly."""
    import decode_attention_append_gb300 as daa
    from gpu_support import gpu_fill, new_pool
    wl = make_random_workload(305, 32, 8, 128, 16, [(200, 900), (12, 400), (1, 77), (64, 64), (7, 20)],
                              extra_pages=5)
    pool = new_pool(wl, dev)
    gpu_fill(wl, pool, dev)
    st = wl.step_table(0)
    q, kn, vn = wl.step_inputs(0)
    tab = daa.PageTable.from_host(st["qo_indptr"], st["kv_indptr"], st["page_indices"],
                                  st["last_page_len"], dev)
    runner = daa.BatchAttention(tab, wl.num_qo_heads, pool, sm_scale=wl.sm_scale)
    runner.append(kn.to(dev), vn.to(dev))
    qd = q.to(dev)
    mask = np.concatenate([tree_mask_rows(np.arange(r.qo_len) - 1, 7) for r in wl.steps[0].requests])
    la = torch.empty(q.shape[0], wl.num_qo_heads, device=dev)
    lb = torch.empty_like(la)
    oa = runner.run(qd, lse=la)
    ob = runner.run(qd, lse=lb, tree_mask=torch.from_numpy(mask.view(np.int32)).to(dev))
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(la, lb)


def test_no_device_error_recorded(dev):
    import decode_attention_append_gb300 as daa
    assert daa.device_error(reset=True) == 0


@pytest.mark.parametrize("Hq,Hkv,d", [(32, 4, 128), (16, 2, 64)])
def test_persistent_decode_many_units(dev, Hq, Hkv, d):
    """The persistent decode kernel over thousands of short units: every CTA
    runs many of them back to back (barrier phases carried across units),
    most end in a partial key tile (stale V rows zeroed by the MMA warp),
    one-token and verify items interleave, and the same plan then runs again
    (the work counter resets itself)."""
    import decode_attention_append_gb300 as daa
    from gpu_support import gpu_fill, new_pool
    rng = np.random.default_rng(Hq * 7 + d)
    reqs = [(1, int(k)) for k in rng.integers(1, 400, size=1600)]
    reqs += [(int(q), int(q + c)) for q, c in zip(rng.integers(2, 9, size=200), rng.integers(0, 500, size=200))]
    order = rng.permutation(len(reqs))
    reqs = [reqs[i] for i in order]
    wl = make_random_workload(900 + Hq, Hq, Hkv, d, 16, reqs, extra_pages=11)
    stats = _run_both(wl, dev)
    assert stats
    # the same plan, run twice more on a stored plan: identical bits
    pool = new_pool(wl, dev)
    gpu_fill(wl, pool, dev)
    st = wl.step_table(0)
    tab = daa.PageTable.from_host(st["qo_indptr"], st["kv_indptr"], st["page_indices"],
                                  st["last_page_len"], dev)
    runner = daa.BatchAttention(tab, wl.num_qo_heads, pool, sm_scale=wl.sm_scale)
    q, kn, vn = wl.step_inputs(0)
    runner.append(kn.to(dev), vn.to(dev))
    qd = q.to(dev)
    ref = runner.run(qd).clone()
    runner.plan()
    for _ in range(2):
        out = runner.run(qd)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert daa.device_error(reset=True) == 0
