"""Seeded request batches shaped like the pages' workloads.

Sources of the shapes (all synthetic; no dataset is involved):

* "Chunked prefill" (k4i.top), section "The core idea" (#core-idea): a 2048-token
  prompt cut into chunks of C=512 and interleaved with decode requests under a
  token budget T = C_prefill + N_decode.
* "Disaggregated prefill and decode" (Perplexity), section "Prefill vs decode
  performance": decode requests carry qo_len=1, prefill requests carry large
  qo_len, and attention cost grows with kv_len.

Five named workloads mirror the five configurations of the benchmark spec
(tiny mixed batch, 7B-class MHA decode, chunked-prefill mixed batch, large-model
GQA decode shard, long-prompt prefill).  Values are bf16 rounded (RNE) from fp32
N(0,1) draws; every draw comes from a ``torch.Generator`` seeded from a
``numpy.random.SeedSequence`` of (workload seed, sequence id, tensor kind,
token block), so one sequence's tensors can be regenerated without drawing the
others.

Data model
----------
A *sequence* is one user request with a final length (tokens) and the list of
page ids reserved for it.  A *step* is one call of the hot path: a list of
(sequence, qo_len, kv_len) entries, where ``kv_len`` counts the tokens that
attention reads *after* this step's append (the cached prefix plus the qo_len
new tokens).  Before the first step of a workload, each sequence already holds
``kv_len - qo_len`` cached tokens of its first step.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

# bf16 quiet-NaN bit pattern used to fill pages (and page slots) that hold no
# token; any read of one poisons an output, and any stray write is visible in a
# byte comparison.
SENTINEL_BF16 = 0x7FC1

# tensor kinds for seeding
_KIND_Q, _KIND_K, _KIND_V = 0, 1, 2
_BLOCK = 256  # tokens per independently seeded block


@dataclass
class Seq:
    length: int                 # final number of tokens of the sequence
    pages: np.ndarray           # int32 page ids reserved, ceil(length / page_size) of them
    prefix: int = -1            # sequence whose first prefix_len tokens (and pages) this one shares
    prefix_len: int = 0         # shared tokens, a multiple of page_size


@dataclass
class Request:
    seq: int                    # index into Workload.seqs
    qo_len: int                 # new tokens appended and attended this step
    kv_len: int                 # tokens attended after the append (cached + new)
    parents: Optional[np.ndarray] = None  # draft tree over the new tokens: parent index or -1


@dataclass
class Step:
    requests: List[Request]


@dataclass
class Workload:
    name: str
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    page_size: int
    num_pages: int
    seed: int
    seqs: List[Seq]
    steps: List[Step]
    causal: bool = True
    description: str = ""

    # ------------------------------------------------------------------ shapes
    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def group_size(self) -> int:
        return self.num_qo_heads // self.num_kv_heads

    def pool_shape(self) -> Tuple[int, int, int, int, int]:
        """[num_pages, 2 (K then V), num_kv_heads, page_size, head_dim]."""
        return (self.num_pages, 2, self.num_kv_heads, self.page_size, self.head_dim)

    def npages(self, kv_len: int) -> int:
        return -(-kv_len // self.page_size)

    # --------------------------------------------------------- page-table arrays
    def _table(self, entries: Sequence[Tuple[int, int, int]]):
        """CSR page table for (seq, n_new, kv_len) entries (int32 numpy arrays)."""
        P = self.page_size
        qo_indptr = [0]
        kv_indptr = [0]
        pages: List[np.ndarray] = []
        last = []
        for s, n_new, kv_len in entries:
            qo_indptr.append(qo_indptr[-1] + n_new)
            n = self.npages(kv_len)
            pages.append(self.seqs[s].pages[:n])
            kv_indptr.append(kv_indptr[-1] + n)
            last.append(0 if kv_len == 0 else kv_len - (n - 1) * P)
        page_indices = (np.concatenate(pages) if pages else np.zeros(0)).astype(np.int32)
        return dict(
            qo_indptr=np.asarray(qo_indptr, np.int32),
            kv_indptr=np.asarray(kv_indptr, np.int32),
            page_indices=page_indices,
            last_page_len=np.asarray(last, np.int32),
        )

    def step_table(self, k: int):
        """Page table of step k; ``qo_indptr`` doubles as the append indptr."""
        return self._table([(r.seq, r.qo_len, r.kv_len) for r in self.steps[k].requests])

    def initial_entries(self) -> List[Tuple[int, int]]:
        """(seq, cached tokens) held before the first step each sequence appears in."""
        seen = {}
        for st in self.steps:
            for r in st.requests:
                if r.seq not in seen:
                    seen[r.seq] = r.kv_len - r.qo_len
        return sorted(seen.items())

    def initial_spans(self) -> List[Tuple[int, int, int]]:
        """(seq, lo, hi): token ranges written before the first step.  A shared
        prefix is written once, under the sequence that owns it; a sequence that
        shares it writes only its own tokens [prefix_len, cached)."""
        spans, owners = [], {}
        for s, c in self.initial_entries():
            q = self.seqs[s]
            lo = 0
            if q.prefix >= 0:
                owners[q.prefix] = max(owners.get(q.prefix, 0), q.prefix_len)
                lo = q.prefix_len
            if c > lo:
                spans.append((s, lo, c))
        for p, n in sorted(owners.items()):
            if all(x[0] != p for x in spans):
                spans.insert(0, (p, 0, n))
        return spans

    def initial_table(self):
        """Page table that appends every sequence's initially cached prefix."""
        return self._table([(s, hi - lo, hi) for s, lo, hi in self.initial_spans()])

    # ------------------------------------------------------------------- values
    def _block(self, seq: int, kind: int, block: int) -> torch.Tensor:
        heads = self.num_qo_heads if kind == _KIND_Q else self.num_kv_heads
        ss = np.random.SeedSequence([self.seed, seq, kind, block])
        g = torch.Generator().manual_seed(int(ss.generate_state(1, np.uint64)[0]))
        t = torch.randn(_BLOCK, heads, self.head_dim, generator=g, dtype=torch.float32)
        t = t.to(torch.bfloat16)
        return t

    def rows_into(self, out: torch.Tensor, seq: int, kind: int, lo: int, hi: int) -> None:
        """Write bf16 rows [lo, hi) of tensor ``kind`` of sequence ``seq`` into out[:hi-lo]."""
        q = self.seqs[seq] if seq < len(self.seqs) else None
        if q is not None and q.prefix >= 0 and lo < q.prefix_len and kind != _KIND_Q:
            # the shared tokens are the prefix owner's
            n = min(hi, q.prefix_len) - lo
            self.rows_into(out[:n], q.prefix, kind, lo, lo + n)
            if hi > q.prefix_len:
                self.rows_into(out[n:], seq, kind, q.prefix_len, hi)
            return
        at = 0
        b = lo // _BLOCK
        while lo + at < hi:
            blk = self._block(seq, kind, b)
            s0 = lo + at - b * _BLOCK
            n = min(_BLOCK - s0, hi - lo - at)
            out[at:at + n].copy_(blk[s0:s0 + n])
            at += n
            b += 1

    def rows(self, seq: int, kind: int, lo: int, hi: int) -> torch.Tensor:
        """bf16 rows [lo, hi) of tensor ``kind`` of sequence ``seq``: [hi-lo, H, d]."""
        heads = self.num_qo_heads if kind == _KIND_Q else self.num_kv_heads
        out = torch.empty(max(0, hi - lo), heads, self.head_dim, dtype=torch.bfloat16)
        if hi > lo:
            self.rows_into(out, seq, kind, lo, hi)
        return out

    def q_rows(self, seq, lo, hi):
        return self.rows(seq, _KIND_Q, lo, hi)

    def k_rows(self, seq, lo, hi):
        return self.rows(seq, _KIND_K, lo, hi)

    def v_rows(self, seq, lo, hi):
        return self.rows(seq, _KIND_V, lo, hi)

    def _gather(self, kind: int, spans: Sequence[Tuple[int, int, int]]) -> torch.Tensor:
        heads = self.num_qo_heads if kind == _KIND_Q else self.num_kv_heads
        n = sum(hi - lo for _, lo, hi in spans)
        out = torch.empty(n, heads, self.head_dim, dtype=torch.bfloat16)
        at = 0
        for seq, lo, hi in spans:
            if hi > lo:
                self.rows_into(out[at:at + hi - lo], seq, kind, lo, hi)
                at += hi - lo
        return out

    def initial_kv(self) -> Tuple[torch.Tensor, torch.Tensor]:
        """K and V of every sequence's initially cached prefix, concatenated."""
        spans = self.initial_spans()
        return self._gather(_KIND_K, spans), self._gather(_KIND_V, spans)

    def step_inputs(self, k: int) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
        """(q [nnz_qo, Hq, d], k_new [nnz_qo, Hkv, d], v_new) of step k, bf16."""
        spans = [(r.seq, r.kv_len - r.qo_len, r.kv_len) for r in self.steps[k].requests]
        return self._gather(_KIND_Q, spans), self._gather(_KIND_K, spans), self._gather(_KIND_V, spans)

    # ------------------------------------------------------------ tree masks
    def prefix_groups(self, k: int = 0):
        """Prefix groups of step k, as the shared-prefix calls take them:
        (indptr, prefix_len) int32 arrays, group i being requests
        [indptr[i], indptr[i+1]).  A maximal run of consecutive requests whose
        sequences share one prefix (same owner and length) is a group; the
        requests between such runs form groups of prefix length 0."""
        reqs = self.steps[k].requests
        key = lambda r: (self.seqs[r.seq].prefix, self.seqs[r.seq].prefix_len)  # noqa: E731
        indptr, plen = [0], []
        i = 0
        while i < len(reqs):
            j = i + 1
            shared = key(reqs[i])[0] >= 0
            while j < len(reqs) and (key(reqs[j]) == key(reqs[i]) if shared
                                     else key(reqs[j])[0] < 0):
                j += 1
            indptr.append(j)
            plen.append(key(reqs[i])[1] if shared else 0)
            i = j
        return np.asarray(indptr, np.int32), np.asarray(plen, np.int32)

    def has_tree(self, k: int = 0) -> bool:
        return any(r.parents is not None for r in self.steps[k].requests)

    def tree_mask(self, k: int = 0, words: Optional[int] = None) -> np.ndarray:
        """uint32 [nnz_qo, words] mask rows of step k (see ``tree_mask_rows``);
        requests without a tree get the chain (every earlier new token)."""
        reqs = self.steps[k].requests
        W = words or max(1, -(-max(r.qo_len for r in reqs) // 32))
        rows = []
        for r in reqs:
            par = r.parents if r.parents is not None else np.arange(r.qo_len) - 1
            rows.append(tree_mask_rows(par, W))
        return np.concatenate(rows, 0) if rows else np.zeros((0, W), np.uint32)

    # ------------------------------------------------------------- accounting
    def summary(self, k: int = 0) -> Dict:
        reqs = self.steps[k].requests
        pre = [r for r in reqs if r.qo_len > 1]
        dec = [r for r in reqs if r.qo_len == 1]
        return dict(
            name=self.name, requests=len(reqs), prefill_requests=len(pre),
            decode_requests=len(dec), nnz_qo=sum(r.qo_len for r in reqs),
            kv_tokens=sum(r.kv_len for r in reqs),
            pages_used=sum(self.npages(r.kv_len) for r in reqs),
            num_pages=self.num_pages, Hq=self.num_qo_heads, Hkv=self.num_kv_heads,
            head_dim=self.head_dim, page_size=self.page_size,
        )


def chunk_schedule(L: int, C: int, cached: int = 0) -> List[Tuple[int, int]]:
    """0-based token ranges [start, end) of the chunks of an L-token prompt.

    "Chunked prefill" (k4i.top), #core-idea and #correctness: chunk s (1-based)
    covers tokens (s-1)C+1 .. sC; in 0-based half-open form [(s-1)C, min(sC, L)).
    Section "Relation to prefix caching" (#prefix-cache-interaction): when the
    first `cached` tokens hit the prefix cache they are skipped, and only the
    uncached suffix is cut into chunks of C.
    """
    n = L - cached
    return [(cached + s * C, cached + min((s + 1) * C, n)) for s in range(-(-n // C))]


def random_tree(gen: torch.Generator, n: int, roots: int = 1) -> np.ndarray:
    """Parent index of each of n draft-tree nodes in topological order (a
    random recursive tree: node i hangs under a uniformly drawn earlier node;
    the first `roots` nodes hang under the cached prefix, parent -1)."""
    par = np.full(n, -1, np.int64)
    for i in range(roots, n):
        par[i] = int(torch.randint(0, i, (1,), generator=gen))
    return par


def tree_mask_rows(parents: np.ndarray, words: int) -> np.ndarray:
    """Encode a draft tree as attention-mask rows: uint32 [n, words], bit j of
    row i (word j // 32, bit j % 32) set when new token j is an ancestor of new
    token i.  Bit i (the token itself) is set too.  Input layout only: the
    encoding of which earlier draft tokens each token may see."""
    n = len(parents)
    assert n <= 32 * words
    rows = np.zeros((n, words), np.uint32)
    for i in range(n):
        j = i
        while j >= 0:
            rows[i, j // 32] |= np.uint32(1 << (j % 32))
            j = int(parents[j])
            assert j < i
    return rows


def _alloc_pages(gen: torch.Generator, num_pages: int, lengths: Sequence[int], P: int) -> List[np.ndarray]:
    """Random page assignment: a permutation of the pool, consecutive entries per sequence."""
    perm = torch.randperm(num_pages, generator=gen).numpy().astype(np.int32)
    out, at = [], 0
    for L in lengths:
        n = -(-L // P)
        if at + n > num_pages:
            raise ValueError("page pool too small for the workload")
        out.append(perm[at:at + n].copy())
        at += n
    return out


def _pool_pages(pages_used: int) -> int:
    """Next power of two >= twice the pages used (pool size where none is stated)."""
    return 1 << max(0, (2 * pages_used - 1).bit_length())


def _single_step(name, Hq, Hkv, d, P, seed, prompts, decodes, num_pages=None, description=""):
    """prompts: list of (qo_len, kv_len); decodes: list of kv_len (qo_len = 1)."""
    lengths = [kv for _, kv in prompts] + list(decodes)
    used = sum(-(-L // P) for L in lengths)
    if num_pages is None:
        num_pages = _pool_pages(used)
    gen = torch.Generator().manual_seed(seed + 7919)
    pages = _alloc_pages(gen, num_pages, lengths, P)
    seqs = [Seq(L, pg) for L, pg in zip(lengths, pages)]
    reqs = [Request(i, qo, kv) for i, (qo, kv) in enumerate(prompts)]
    reqs += [Request(len(prompts) + j, 1, kv) for j, kv in enumerate(decodes)]
    return Workload(name, Hq, Hkv, d, P, num_pages, seed, seqs, [Step(reqs)], description=description)


def make_shared_prefix_workload(name, Hq, Hkv, d, P, seed, prefix_len, prompts, decodes, description=""):
    """One step over a prefix shared by every request (a prefix-cache hit).

    Sequence 0 owns the shared prefix (prefix_len tokens, whole pages) and is
    not itself a request.  prompts: (qo_len, kv_len) chunks of prompts whose
    first prefix_len tokens are the shared prefix; decodes: kv_len of decode
    requests that share it too.  Each request's page list is the prefix's
    pages followed by pages of its own."""
    assert prefix_len % P == 0
    lengths = [kv for _, kv in prompts] + list(decodes)
    own = [L - prefix_len for L in lengths]
    used = prefix_len // P + sum(-(-x // P) for x in own)
    num_pages = _pool_pages(used)
    gen = torch.Generator().manual_seed(seed + 7919)
    pages = _alloc_pages(gen, num_pages, [prefix_len] + own, P)
    seqs = [Seq(prefix_len, pages[0])]
    for L, pg in zip(lengths, pages[1:]):
        seqs.append(Seq(L, np.concatenate([pages[0], pg]).astype(np.int32), 0, prefix_len))
    reqs = [Request(1 + i, qo, kv) for i, (qo, kv) in enumerate(prompts)]
    reqs += [Request(1 + len(prompts) + j, 1, kv) for j, kv in enumerate(decodes)]
    return Workload(name, Hq, Hkv, d, P, num_pages, seed, seqs, [Step(reqs)], description=description)


def make_prefix_groups_workload(name, Hq, Hkv, d, P, seed, layout, causal=True, description=""):
    """One step over a batch whose requests hit several cached prefixes.

    layout, in batch order: ("group", prefix_len, [(qo_len, kv_len), ...]) --
    requests whose first prefix_len tokens (whole pages) are one shared prefix,
    owned by a sequence that is not itself a request -- and ("solo", qo_len,
    kv_len) requests with pages of their own."""
    lengths, plan = [], []  # plan: (owner index or -1, prefix_len, qo, kv) per request
    for ent in layout:
        if ent[0] == "group":
            _, pl, reqs = ent
            assert pl % P == 0
            owner = len(lengths)
            lengths.append(pl)
            for qo, kv in reqs:
                plan.append((owner, pl, qo, kv))
                lengths.append(kv - pl)
        else:
            _, qo, kv = ent
            plan.append((-1, 0, qo, kv))
            lengths.append(kv)
    used = sum(-(-L // P) for L in lengths)
    num_pages = _pool_pages(used)
    pages = _alloc_pages(torch.Generator().manual_seed(seed + 7919), num_pages, lengths, P)
    seqs, reqs, at = [], [], 0
    for ent in layout:
        if ent[0] == "group":
            owner = len(seqs)
            seqs.append(Seq(ent[1], pages[at]))
            at += 1
            for qo, kv in ent[2]:
                own = np.concatenate([pages[owner], pages[at]]).astype(np.int32)
                reqs.append(Request(len(seqs), qo, kv))
                seqs.append(Seq(kv, own, owner, ent[1]))
                at += 1
        else:
            reqs.append(Request(len(seqs), ent[1], ent[2]))
            seqs.append(Seq(ent[2], pages[at]))
            at += 1
    wl = Workload(name, Hq, Hkv, d, P, num_pages, seed, seqs, [Step(reqs)], description=description)
    wl.causal = causal
    return wl


def make_tree_workload(name, Hq, Hkv, d, P, seed, trees, decodes=(), prompts=(), num_pages=None,
                       description=""):
    """One step of draft-tree verification ("Accelerating Sonar through
    speculation", section EAGLE).  trees: (n_nodes, cached tokens, roots) per
    verify request -- its n_nodes draft tokens are appended after the cached
    ones and attended through the tree mask; decodes: kv_len of decode
    requests; prompts: (qo_len, kv_len) of plain causal chunks."""
    gen = torch.Generator().manual_seed(seed + 104729)
    lengths = [c + n for n, c, _ in trees] + [kv for _, kv in prompts] + list(decodes)
    used = sum(-(-x // P) for x in lengths)
    if num_pages is None:
        num_pages = _pool_pages(used)
    pages = _alloc_pages(torch.Generator().manual_seed(seed + 7919), num_pages, lengths, P)
    seqs = [Seq(L, pg) for L, pg in zip(lengths, pages)]
    reqs = [Request(i, n, c + n, random_tree(gen, n, roots)) for i, (n, c, roots) in enumerate(trees)]
    at = len(trees)
    reqs += [Request(at + i, qo, kv) for i, (qo, kv) in enumerate(prompts)]
    at += len(prompts)
    reqs += [Request(at + i, 1, kv) for i, kv in enumerate(decodes)]
    return Workload(name, Hq, Hkv, d, P, num_pages, seed, seqs, [Step(reqs)], description=description)


CONFIG_NAMES = ["tiny_mixed", "mha_decode", "chunked_prefill_mixed", "gqa_decode_shard", "long_prefill"]
# further workloads beyond the five configurations
EXTRA_NAMES = ["prefix_shared", "tree_verify", "long_prefill_d64", "first_chunk_prefill"]


def make_workload(name: str) -> Workload:
    """The five named workloads (seed = 1000 + 1-based config number)."""
    if name == "tiny_mixed":
        # 1 prompt of 64 tokens prefilled in 4 chunks of 16 + decodes at kv 40 and 73
        # that each advance one token per step (continuous batching).
        Hq, Hkv, d, P, num_pages, seed = 4, 2, 64, 16, 64, 1001
        lengths = [64, 40 + 3, 73 + 3]
        gen = torch.Generator().manual_seed(seed + 7919)
        pages = _alloc_pages(gen, num_pages, lengths, P)
        seqs = [Seq(L, pg) for L, pg in zip(lengths, pages)]
        steps = []
        for k, (c0, c1) in enumerate(chunk_schedule(64, 16)):
            steps.append(Step([Request(0, c1 - c0, c1), Request(1, 1, 40 + k), Request(2, 1, 73 + k)]))
        return Workload(name, Hq, Hkv, d, P, num_pages, seed, seqs, steps,
                        description="1 prompt L=64 in 4 chunks of C=16 + 2 decodes (kv 40, 73); "
                                    "Hq 4 / Hkv 2, d 64, P 16, 64-page pool")
    if name == "mha_decode":
        seed = 1002
        g = torch.Generator().manual_seed(seed)
        kv = torch.randint(512, 4096 + 1, (32,), generator=g).tolist()
        return _single_step(name, 32, 32, 128, 16, seed, [], kv,
                            description="32 decodes, kv ~ U[512,4096], Hq=Hkv=32, d 128, P 16, "
                                        "+ append of 1 token each")
    if name == "chunked_prefill_mixed":
        seed = 1003
        g = torch.Generator().manual_seed(seed)
        kv = torch.randint(1024, 4096 + 1, (32,), generator=g).tolist()
        return _single_step(name, 32, 8, 128, 16, seed, [(512, 2048)], kv,
                            description="2048-token prompt at chunk [1536,2048) + 32 decodes "
                                        "kv ~ U[1024,4096]; Hq 32 / Hkv 8, d 128, P 16")
    if name == "gqa_decode_shard":
        seed = 1004
        g = torch.Generator().manual_seed(seed)
        z = torch.randn(128, generator=g, dtype=torch.float64)
        kv = torch.exp(math.log(8192.0) + math.log(2.0) * z).round().clamp(1024, 32768).long().tolist()
        return _single_step(name, 12, 1, 128, 16, seed, [], kv, num_pages=300_000,
                            description="128 decodes, kv log-normal (median 8192, sigma ln 2, "
                                        "clip [1024,32768]); Hq 12 / Hkv 1, d 128, P 16, 300k-page pool")
    if name == "long_prefill":
        seed = 1005
        g = torch.Generator().manual_seed(seed)
        kv = torch.randint(2048, 16384 + 1, (64,), generator=g).tolist()
        return _single_step(name, 64, 8, 128, 16, seed, [(8192, 16384)] * 4, kv,
                            description="4 prompts of 16384 at chunk 2 of 2 (8192 new over 8192 "
                                        "cached) + 64 decodes kv ~ U[2048,16384]; Hq 64 / Hkv 8, d 128")
    if name == "prefix_shared":
        # "Chunked prefill", #prefix-cache-interaction: a 1024-token system
        # prompt hits the prefix cache, so a 2048-token prompt needs only its
        # two 512-token suffix chunks.  One prompt at each of those chunks, and
        # 64 decode requests that share the same system prompt, all reading its
        # 64 pages in place.
        seed = 1006
        g = torch.Generator().manual_seed(seed)
        kv = (1024 + torch.randint(512, 3072 + 1, (64,), generator=g)).tolist()
        return make_shared_prefix_workload(name, 32, 8, 128, 16, seed, 1024, [(512, 1536), (512, 2048)], kv,
                                   description="1024-token system prompt shared by every request "
                                               "(64 pages read in place): prompts at suffix chunks "
                                               "[1024,1536) and [1536,2048) + 64 decodes kv = 1024 + "
                                               "U[512,3072]; Hq 32 / Hkv 8, d 128, P 16")
    if name == "tree_verify":
        # "Accelerating Sonar through speculation", section EAGLE: the target
        # model verifies a tree of draft tokens under a custom attention mask.
        # 32 requests, each a 64-node draft tree (random recursive tree, one
        # root) over kv ~ U[1024, 4096] cached tokens; 7B-class GQA 32 / 8.
        seed = 1007
        g = torch.Generator().manual_seed(seed)
        cached = torch.randint(1024, 4096 + 1, (32,), generator=g).tolist()
        return make_tree_workload(name, 32, 8, 128, 16, seed, [(64, c, 1) for c in cached],
                                  description="32 verify requests, each a 64-node draft tree "
                                              "(random recursive tree) over kv ~ U[1024,4096] cached "
                                              "tokens under its tree mask; Hq 32 / Hkv 8, d 128, P 16")
    if name == "long_prefill_d64":
        # the long-prompt prefill batch at head_dim 64 (small-model heads, as
        # in the tiny mixed batch): prefill items run the single-CTA
        # tensor-core kernel instead of CTA pairs
        seed = 1008
        g = torch.Generator().manual_seed(seed)
        kv = torch.randint(1024, 8192 + 1, (32,), generator=g).tolist()
        return _single_step(name, 32, 4, 64, 16, seed, [(4096, 8192)] * 4, kv,
                            description="4 prompts of 8192 at chunk 2 of 2 (4096 new over 4096 "
                                        "cached) + 32 decodes kv ~ U[1024,8192]; Hq 32 / Hkv 4, d 64")
    if name == "first_chunk_prefill":
        # "Chunked prefill", #core-idea: the first chunk of a prompt has no
        # cached prefix, so every key the chunk attends to is appended in the
        # same step; 4 prompts' first 8192-token chunks + 64 decodes, GQA 64/8
        seed = 1009
        g = torch.Generator().manual_seed(seed)
        kv = torch.randint(2048, 16384 + 1, (64,), generator=g).tolist()
        return _single_step(name, 64, 8, 128, 16, seed, [(8192, 8192)] * 4, kv,
                            description="first 8192-token chunks of 4 prompts (nothing cached) "
                                        "+ 64 decodes kv ~ U[2048,16384]; Hq 64 / Hkv 8, d 128")
    raise KeyError(name)


def make_prompt_workload(L: int, C: int, Hq: int, Hkv: int, d: int, P: int, seed: int,
                         num_pages: int | None = None, decodes: Sequence[int] = ()) -> Workload:
    """One L-token prompt prefilled in chunks of C (one step per chunk), plus
    optional decode sequences that advance one token per step.  C >= L gives the
    one-shot prefill of the same prompt with the same pages and values."""
    sched = chunk_schedule(L, C)
    nsteps = len(sched)
    lengths = [L] + [kv + nsteps - 1 for kv in decodes]
    used = sum(-(-x // P) for x in lengths)
    if num_pages is None:
        num_pages = _pool_pages(used)
    gen = torch.Generator().manual_seed(seed + 7919)
    pages = _alloc_pages(gen, num_pages, lengths, P)
    seqs = [Seq(x, pg) for x, pg in zip(lengths, pages)]
    steps = []
    for k, (c0, c1) in enumerate(sched):
        reqs = [Request(0, c1 - c0, c1)]
        reqs += [Request(1 + j, 1, kv + k) for j, kv in enumerate(decodes)]
        steps.append(Step(reqs))
    return Workload(f"prompt_L{L}_C{C}", Hq, Hkv, d, P, num_pages, seed, seqs, steps,
                    description=f"prompt L={L} in chunks of C={C}")


def make_random_workload(seed: int, Hq: int, Hkv: int, d: int, P: int, reqs: Sequence[Tuple[int, int]],
                         num_pages: int | None = None, extra_pages: int = 0) -> Workload:
    """Single step with explicit (qo_len, kv_len) per request (edge-case tests)."""
    lengths = [kv for _, kv in reqs]
    used = sum(-(-x // P) for x in lengths)
    if num_pages is None:
        num_pages = max(1, used + extra_pages)
    gen = torch.Generator().manual_seed(seed + 7919)
    pages = _alloc_pages(gen, num_pages, lengths, P)
    seqs = [Seq(x, pg) for x, pg in zip(lengths, pages)]
    step = Step([Request(i, qo, kv) for i, (qo, kv) in enumerate(reqs)])
    return Workload(f"random_{seed}", Hq, Hkv, d, P, num_pages, seed, seqs, [step])
