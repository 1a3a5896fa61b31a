// Host-side plan of one batch_attention call, shared by the workspace entry
// point and the no-allocation entry point (which instantiates it over
// fixed-capacity static containers).
//
// "Disaggregated prefill and decode" (Perplexity), "Prefill vs decode
// performance": attention parallelises over requests and over kv_len.  Work is
// split three ways:
//  * decode requests (qo_len == 1) whose kv head serves g >= kTcDecodeMinGroup
//    query heads, and small multi-token requests (verify batches, qo_len up to
//    plan_verify_max), go to the tensor-core kernel as key-split work items
//    (their qo_len x g rows fill one M = 128 tile); the K/V bytes then stream
//    at memory rate while the CUDA cores only run the softmax;
//  * other decode requests go to the CUDA-core split-KV kernel as page-aligned
//    key splits;
//  * short multi-token requests whose rows fit two 128-row Q tiles (larger
//    verify steps, e.g. draft trees) become items of the single-CTA
//    tensor-core kernel, both tiles sharing every K/V tile; their keys are cut
//    only when one request holds more keys than an SM's share of the batch;
//  * longer prefill requests become items of 128-row tiles of packed
//    (token, query head) rows for the tensor-core kernels -- four tiles on a
//    pair of SMs for head_dim 128, two tiles on one SM otherwise -- longest
//    key range first.
// Split decode requests get consecutive partial slots and one softmax_merge
// item ("Chunked prefill" (k4i.top), #correctness).
#pragma once
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <functional>
#include <vector>

#include "../../include/daa.h"
#include "launch.h"

namespace daa {

constexpr int kPlanPageSize = 16;
constexpr int kTcDecodeMinGroup = 4;
// Requests with 2 <= qo_len <= this many tokens (and qo_len * g <= 128) -- e.g.
// the draft tokens of a speculative-decoding verify step -- are memory bound
// like decode: they run as key-split items of the tensor-core decode kernel
// (all their rows in one 128-row tile, K/V read once per split).
constexpr int kVerifyMaxTokens = 16;

inline int plan_verify_max(int g) { return std::min(kVerifyMaxTokens, kPrefillTileRows / g); }
constexpr size_t kPlanAlign = 256;

inline size_t plan_align_up(size_t x) { return (x + kPlanAlign - 1) & ~(kPlanAlign - 1); }

// Prefill items span four Q tiles and run on CTA pairs (head_dim 128), else two
// Q tiles on one CTA.
inline bool plan_prefill_quads(const daa_dims& d) { return d.head_dim == 128; }

inline daa_status plan_check_dims(const daa_dims& d) {
  if (d.num_qo_heads <= 0 || d.num_kv_heads <= 0 || d.head_dim <= 0 || d.page_size <= 0 ||
      d.num_pages <= 0 || d.num_qo_heads % d.num_kv_heads != 0)
    return DAA_ERR_INVALID_ARG;
  if (d.head_dim != 64 && d.head_dim != 128) return DAA_ERR_UNSUPPORTED;
  if (d.page_size != kPlanPageSize) return DAA_ERR_UNSUPPORTED;
  const int g = d.num_qo_heads / d.num_kv_heads;
  if (g < 1 || g > 16) return DAA_ERR_UNSUPPORTED;
  // slices of the pool must be addressable by 32-bit TMA coordinates
  if (d.num_pages * 2 * (int64_t)d.num_kv_heads > (int64_t)INT32_MAX) return DAA_ERR_UNSUPPORTED;
  return DAA_OK;
}

// Requests that share a cached prefix (a prefix-cache hit, "Chunked prefill",
// #prefix-cache-interaction): group i is requests [indptr[i], indptr[i+1]),
// consecutive, whose first prefix_len[i] tokens sit in the same pages.  Host
// arrays.
struct PrefixGroups {
  const int32_t* indptr;      // [n + 1], non-decreasing, within [0, batch]
  const int32_t* prefix_len;  // [n], multiples of the page size
  int32_t n;
};

// Offsets of the workspace sections (bytes).  Tensor-core items are stored
// as three consecutive groups, each launched as its own kernel: prefill items,
// short items (single-CTA kernel, head_dim 128 only; for head_dim 64 they join
// the prefill group, which runs the same kernel), decode / verify items.
// The plan ends with one zeroed 256-byte block (off_sched): the work counter
// the persistent decode kernel takes its items from, reset by every call's
// plan copy.
struct PlanLayout {
  int n_units = 0, n_merges = 0, n_tiles = 0, n_dec_tiles = 0, n_short_tiles = 0, n_parts = 0;
  size_t off_units = 0, off_merges = 0, off_tiles = 0, off_sched = 0, plan_bytes = 0;
  size_t off_part_o = 0, off_part_lse = 0, total = 0;
};

// Makespan, in keys, of greedy longest-first assignment of the tensor-core
// decode units to `workers` persistent CTAs (each takes the next unit when it
// is free), for key splits of `split_keys`; every unit also costs `overhead`
// keys.  unit_keys(r, f) calls f(keys) for each split of request r, and every
// split is repeated for each of `heads` kv heads.  Returns -1 when the batch
// is too large to model (then a fixed target is used).  Allocation-free: a
// fixed heap on the stack and a per-thread buffer for the last splits.
template <class UnitKeys>
int64_t plan_lpt_makespan(int batch, int heads, int workers, int64_t split_keys, int64_t overhead,
                          UnitKeys&& unit_keys) {
  constexpr int kMaxWorkers = 1024, kMaxTail = 8192;
  thread_local int32_t tail[kMaxTail];
  if (workers <= 0 || workers > kMaxWorkers) return -1;
  int64_t n_full = 0;  // splits of exactly split_keys keys (all but each request's last)
  int n_tail = 0;
  for (int r = 0; r < batch; ++r) {
    bool ok = true;
    unit_keys(r, [&](int64_t keys) {
      if (keys == split_keys) ++n_full;
      else if (n_tail < kMaxTail) tail[n_tail++] = (int32_t)keys;
      else ok = false;
    });
    if (!ok) return -1;
  }
  n_full *= heads;
  // full splits first (the longest): workers end up one full unit apart
  int64_t heap[kMaxWorkers];
  const int64_t per = n_full / workers, extra = n_full % workers;
  for (int w = 0; w < workers; ++w) heap[w] = (per + (w < extra ? 1 : 0)) * (split_keys + overhead);
  std::make_heap(heap, heap + workers, std::greater<int64_t>());
  std::sort(tail, tail + n_tail, std::greater<int32_t>());
  for (int i = 0; i < n_tail; ++i)
    for (int h = 0; h < heads; ++h) {
      std::pop_heap(heap, heap + workers, std::greater<int64_t>());
      heap[workers - 1] += tail[i] + overhead;
      std::push_heap(heap, heap + workers, std::greater<int64_t>());
    }
  return *std::max_element(heap, heap + workers);
}

// Vec: push_back(const T&) -> bool (false when full), size(), data(), clear().
// With `groups`: within each group, every maximal run of consecutive requests
// with 1 <= qo_len <= two Q tiles (decode, verify and short requests) that has
// two or more such members attends the group's shared keys -- whole 128-key
// tiles of its prefix -- once for all its rows (prefix-group items), and each
// member's own items start after them; softmax_merge then combines each row's
// prefix partial with its own.  Prefill requests of a group keep the prefix in
// their own items: their Q tiles are full already, so sharing would only add
// partials to merge.  Without groups the plan allocates nothing beyond the
// Vecs.
template <class UnitVec, class MergeVec, class TileVec>
daa_status plan_batch(const int32_t* qo, const int32_t* kv, const int32_t* last, int32_t batch,
                      const daa_dims& d, int sms, UnitVec& units, MergeVec& merges,
                      TileVec& tiles, PlanLayout& lay, const PrefixGroups* groups = nullptr) {
  units.clear();
  merges.clear();
  tiles.clear();
  lay = PlanLayout{};
  daa_status st = plan_check_dims(d);
  if (st != DAA_OK) return st;
  if (batch < 0) return DAA_ERR_INVALID_ARG;
  if (batch == 0) return DAA_OK;
  if (!qo || !kv || !last) return DAA_ERR_INVALID_ARG;
  if (qo[0] != 0 || kv[0] != 0) return DAA_ERR_SHAPE;
  const int P = d.page_size;
  const int g = d.num_qo_heads / d.num_kv_heads;
  const bool tc_decode = g >= kTcDecodeMinGroup;
  const int verify_max = plan_verify_max(g);

  const int tpt = kPrefillTileRows / g;  // tokens per 128-row Q tile
  const int short_max = 2 * tpt;
  const bool quads = plan_prefill_quads(d);
  int64_t dec_pages = 0, short_pages = 0;
  for (int r = 0; r < batch; ++r) {
    const int64_t nq = (int64_t)qo[r + 1] - qo[r];
    const int64_t np = (int64_t)kv[r + 1] - kv[r];
    if (nq < 0 || np < 0) return DAA_ERR_SHAPE;
    if (np > 0 && (last[r] < 1 || last[r] > P)) return DAA_ERR_SHAPE;
    const int64_t kv_len = np > 0 ? (np - 1) * P + last[r] : 0;
    if (nq > kv_len || kv_len > INT32_MAX / 2) return DAA_ERR_SHAPE;
    if (nq >= 1 && nq <= verify_max) dec_pages += np;
    else if (nq > verify_max && nq <= short_max) short_pages += np;
  }
  // prefix-group runs (see above): shared keys and the partial slot of row 0
  // of each member, per request; slots [0, group_rows) hold the runs' rows
  struct Run {
    int r0, r1, sk, slot0;
  };
  std::vector<Run> runs;
  std::vector<int32_t> shared_keys, shared_slot;
  int group_rows = 0;
  if (groups && groups->n > 0) {
    if (!groups->indptr || !groups->prefix_len) return DAA_ERR_INVALID_ARG;
    if (groups->indptr[0] < 0 || groups->indptr[groups->n] > batch) return DAA_ERR_SHAPE;
    shared_keys.assign(batch, 0);
    shared_slot.assign(batch, -1);
    for (int i = 0; i < groups->n; ++i) {
      const int b0 = groups->indptr[i], b1 = groups->indptr[i + 1];
      const int pl = groups->prefix_len[i];
      if (b1 < b0 || pl < 0 || pl % P != 0) return DAA_ERR_SHAPE;
      for (int r = b0; r < b1; ++r) {
        const int np = kv[r + 1] - kv[r];
        const int64_t kv_len = np > 0 ? (int64_t)(np - 1) * P + last[r] : 0;
        if (pl > kv_len - (qo[r + 1] - qo[r])) return DAA_ERR_SHAPE;  // the prefix is cached
      }
      const int sk = pl / kPrefillTileRows * kPrefillTileRows;
      if (sk == 0) continue;
      for (int r = b0; r < b1;) {
        const int nq = qo[r + 1] - qo[r];
        if (nq > short_max || nq == 0) {  // a prefill request ends a run; runs start with rows
          ++r;
          continue;
        }
        int r1 = r, members = 0;
        for (; r1 < b1 && qo[r1 + 1] - qo[r1] <= short_max; ++r1)
          if (qo[r1 + 1] > qo[r1]) ++members;
        if (members >= 2) {
          runs.push_back(Run{r, r1, sk, group_rows});
          for (int m = r; m < r1; ++m) {
            shared_keys[m] = sk;
            shared_slot[m] = group_rows + (qo[m] - qo[r]);
          }
          group_rows += qo[r1] - qo[r];
        }
        r = r1;
      }
    }
    // the shared keys are not read again by the members' own splits
    for (int r = 0; r < batch; ++r) {
      const int64_t nq = (int64_t)qo[r + 1] - qo[r];
      if (nq >= 1 && nq <= verify_max) dec_pages -= shared_keys[r] / P;
      else if (nq > verify_max && nq <= short_max) short_pages -= shared_keys[r] / P;
    }
  }
  auto shared_of = [&](int r) -> int { return shared_keys.empty() ? 0 : shared_keys[r]; };
  const int64_t page_heads = dec_pages * d.num_kv_heads;

  // split sizes (pages).  CUDA-core splits: about twenty per SM (ten per CTA
  // slot), so the longest split is a small fraction of the pass while the
  // split-KV partials stay few.  Tensor-core splits: whole 128-key tiles.  With
  // prefill items beside them, about six items per SM: the prefill holds its
  // SMs for tens of microseconds, the decode CTAs that start after it take
  // items late, and shorter items keep that tail short.  Alone, the count of
  // items per SM (2 .. 8) whose greedy assignment to the persistent CTAs ends
  // first.  Measured on GB300: MHA decode 20 CUDA-core splits per SM 7% faster
  // than 40 or 80; chunked-prefill mixed batch 6 tensor-core items per SM 9%
  // faster than 4; GQA decode shard 2 per SM 4% faster than 4, 3 and 5 per SM
  // 20% slower (the model's ranking).
  bool prefill_beside = groups && groups->n > 0;  // prefix-group items join the prefill launch
  for (int r = 0; r < batch && !prefill_beside; ++r) prefill_beside = qo[r + 1] - qo[r] > short_max;
  int64_t cur_split = 0;  // split (pages) being modelled below
  auto tc_split_for = [&](int64_t per_sm) {
    int64_t sp = (page_heads + (int64_t)sms * per_sm - 1) / ((int64_t)sms * per_sm);
    sp = (sp + 7) / 8 * 8;
    return std::max<int64_t>(32, std::min<int64_t>(2048, sp));
  };
  int64_t split_tc = tc_split_for(prefill_beside ? 6 : 4);
  if (!prefill_beside && tc_decode) {
    // alone on the GPU, the persistent decode CTAs take their units greedily,
    // most keys first, so the split whose units pack the CTAs most evenly is
    // found by simulating that (GB300: this model ranks 2 < 4 < 6 < 8 < 5 < 3
    // items per SM for the GQA decode shard exactly as measured)
    auto unit_keys = [&](int r, auto&& emit) {
      const int nq = qo[r + 1] - qo[r];
      if (nq < 1 || nq > verify_max) return;
      const int np = kv[r + 1] - kv[r];
      const int64_t kv_len = (int64_t)(np - 1) * P + last[r];
      const int64_t keys = kv_len - nq + 1 - shared_of(r);
      const int64_t sk_ = (int64_t)cur_split * P;
      const int64_t n = (keys + sk_ - 1) / sk_;
      for (int64_t s2 = 0; s2 + 1 < n; ++s2) emit(sk_);
      emit(kv_len - shared_of(r) - (n - 1) * sk_);
    };
    int64_t best = -1;
    for (int64_t per_sm : {2, 3, 4, 5, 6, 8}) {
      cur_split = tc_split_for(per_sm);
      const int64_t m = plan_lpt_makespan(batch, d.num_kv_heads, 2 * sms, cur_split * P,
                                          /*overhead=*/64, unit_keys);
      if (m < 0) break;
      if (best < 0 || m < best) {
        best = m;
        split_tc = cur_split;
      }
    }
  }
  int64_t split_cc = (page_heads + (int64_t)sms * 20 - 1) / ((int64_t)sms * 20);
  split_cc = std::max<int64_t>(16, std::min<int64_t>(1024, split_cc));

  // short items: one item's keys at most an SM's share of the short requests'
  // K/V (so the longest item bounds the pass), whole 128-key tiles
  int64_t split_short = (short_pages * d.num_kv_heads + sms - 1) / sms;
  split_short = std::max<int64_t>(32, (split_short + 7) / 8 * 8);

  // prefix-group items first: each run's rows hold consecutive partial slots
  // (one per token, in row order) from slot 0, named by their merge items
  lay.n_parts = group_rows;
  for (const Run& run : runs) {
    const int rows = qo[run.r1] - qo[run.r0];
    for (int t0 = 0; t0 < rows; t0 += (quads ? 4 : 2) * tpt) {
      PrefillTile t{};
      t.q_row0 = qo[run.r0];
      t.qo_len = rows;
      t.kv_len = run.sk;
      t.page_base = kv[run.r0];
      t.tok0 = t0;
      if (quads) {
        t.ntok = std::min(4 * tpt, rows - t0);
        t.ntok1 = 0;
      } else {
        t.ntok = std::min(tpt, rows - t0);
        t.ntok1 = t.ntok == tpt ? std::max(0, std::min(tpt, rows - t0 - tpt)) : 0;
      }
      t.key_lo = 0;
      t.key_hi = run.sk;
      t.part = run.slot0;
      t.part_stride = 1;
      t.kind = kTilePrefixGroup;
      if (!tiles.push_back(t)) return DAA_ERR_WORKSPACE;
    }
  }

  // decode (qo_len 1), verify (qo_len 2 .. verify_max) and short
  // (verify_max < qo_len <= short_max) requests: key-split items
  for (int r = 0; r < batch; ++r) {
    const int nq = qo[r + 1] - qo[r];
    if (nq < 1 || nq > short_max) continue;
    const bool is_short = nq > verify_max;
    const bool on_tc = tc_decode || nq > 1;
    const int64_t split = is_short ? split_short : on_tc ? split_tc : split_cc;
    const int np = kv[r + 1] - kv[r];
    const int kv_len = (np - 1) * P + last[r];
    const int sk = shared_of(r);  // keys a prefix-group item covers
    // splits cut the keys token 0 can see past the shared ones, [sk, kv_len -
    // nq], so every split starts at a key each token sees; the last split also
    // takes the tail
    const int64_t vis = (int64_t)kv_len - nq + 1;
    const int nsplit = (int)((vis - sk + split * P - 1) / (split * P));
    // partial slots: token t of split s at part0 + t * nsplit + s, so each
    // token's splits are consecutive for its softmax_merge item (which also
    // takes the row's prefix partial when sk > 0)
    int part0 = -1;
    if (nsplit > 1 || sk > 0) {
      const int32_t pbase = sk > 0 ? shared_slot[r] : -1;
      for (int t = 0; t < nq; ++t)
        if (!merges.push_back(MergeItem{qo[r] + t, lay.n_parts + t * nsplit, nsplit,
                                        sk > 0 ? pbase + t : -1}))
          return DAA_ERR_WORKSPACE;
      part0 = lay.n_parts;
      lay.n_parts += nsplit * nq;
    }
    for (int s = 0; s < nsplit; ++s) {
      const int lo = (int)(sk + s * split * P);
      const int hi = s == nsplit - 1 ? kv_len : (int)(sk + (s + 1) * split * P);
      if (on_tc) {
        PrefillTile t{};
        t.q_row0 = qo[r];
        t.qo_len = nq;
        t.kv_len = kv_len;
        t.page_base = kv[r];
        t.tok0 = 0;
        t.ntok = std::min(nq, tpt);   // short items: two Q tiles
        t.ntok1 = nq - t.ntok;
        t.key_lo = lo;
        t.key_hi = hi;
        t.part = part0 >= 0 ? part0 + s : -1;
        t.part_stride = nsplit;
        if (!tiles.push_back(t)) return DAA_ERR_WORKSPACE;
      } else {
        DecodeUnit u{};
        u.q_row = qo[r];
        u.page_base = kv[r];
        u.tok_begin = lo;
        u.tok_end = hi;
        u.kv_len = kv_len;
        u.part = part0 >= 0 ? part0 + s : -1;
        if (!units.push_back(u)) return DAA_ERR_WORKSPACE;
      }
    }
  }
  // longest splits first (only the last split of a request is shorter)
  std::sort(units.data(), units.data() + units.size(), [](const DecodeUnit& x, const DecodeUnit& y) {
    const int a = x.tok_end - x.tok_begin, b = y.tok_end - y.tok_begin;
    return a != b ? a > b : (x.q_row != y.q_row ? x.q_row < y.q_row : x.tok_begin < y.tok_begin);
  });

  // prefill: 128-row Q tiles of packed (token, query head) rows (tpt tokens
  // each).  head_dim 128: items of four tiles for a CTA pair (ntok = the item's
  // tokens); otherwise pairs of tiles for one CTA (ntok, ntok1 per tile).
  for (int r = 0; r < batch; ++r) {
    const int nq = qo[r + 1] - qo[r];
    if (nq <= short_max) continue;
    const int np = kv[r + 1] - kv[r];
    const int kv_len = (np - 1) * P + last[r];
    for (int t0 = 0; t0 < nq; t0 += (quads ? 4 : 2) * tpt) {
      PrefillTile t{};
      t.q_row0 = qo[r];
      t.qo_len = nq;
      t.kv_len = kv_len;
      t.page_base = kv[r];
      t.tok0 = t0;
      if (quads) {
        t.ntok = std::min(4 * tpt, nq - t0);
        t.ntok1 = 0;
      } else {
        t.ntok = std::min(tpt, nq - t0);
        t.ntok1 = t.ntok == tpt ? std::max(0, std::min(tpt, nq - t0 - tpt)) : 0;
      }
      t.key_lo = 0;
      t.key_hi = kv_len;
      t.part = -1;
      if (!tiles.push_back(t)) return DAA_ERR_WORKSPACE;
    }
  }
  // tensor-core items in launch groups -- prefill items, short items (their
  // own group only where prefill runs on CTA pairs), decode / verify items --
  // most work first within each group
  auto group = [=](const PrefillTile& t) {
    if (t.kind == kTilePrefixGroup) return 0;  // with the prefill items
    if (t.qo_len <= verify_max) return 2;
    return quads && t.qo_len <= short_max ? 1 : 0;
  };
  // work of an item: keys read by its last row, counted once per Q tile
  auto work = [=](const PrefillTile& t) -> int64_t {
    const bool pair = quads && group(t) == 0;  // up to four tiles on a CTA pair
    const int toks = t.ntok + t.ntok1;
    const int ntiles = pair ? (toks + tpt - 1) / tpt : (t.ntok1 > 0 ? 2 : 1);
    const int end = t.kind == kTilePrefixGroup
                        ? t.key_hi
                        : std::min(t.key_hi, t.kv_len - t.qo_len + t.tok0 + toks);
    return (int64_t)(end - t.key_lo) * ntiles;
  };
  // Sort keys computed once per item (a comparator that recomputes them made
  // the sort most of the host time of a call: ~70 us for 362 items), then the
  // items permuted in place.  Batches past the key buffer sort directly.
  struct SortKey {
    int64_t work;
    int32_t group, q_row0, tok0, key_lo, idx, pad;
  };
  auto key_less = [](const SortKey& x, const SortKey& y) {
    if (x.group != y.group) return x.group < y.group;
    if (x.work != y.work) return x.work > y.work;
    if (x.q_row0 != y.q_row0) return x.q_row0 < y.q_row0;
    return x.tok0 != y.tok0 ? x.tok0 < y.tok0 : x.key_lo < y.key_lo;
  };
  constexpr int kMaxSortKeys = 16384;
  thread_local SortKey sort_keys[kMaxSortKeys];
  const int n_tiles = (int)tiles.size();
  PrefillTile* td = tiles.data();
  if (n_tiles <= kMaxSortKeys) {
    for (int i = 0; i < n_tiles; ++i)
      sort_keys[i] = SortKey{work(td[i]), group(td[i]), td[i].q_row0, td[i].tok0, td[i].key_lo, i, 0};
    std::sort(sort_keys, sort_keys + n_tiles, key_less);
    // position i takes item sort_keys[i].idx: follow each cycle of the
    // permutation once, marking placed positions with idx = -1
    for (int i = 0; i < n_tiles; ++i) {
      if (sort_keys[i].idx < 0 || sort_keys[i].idx == i) continue;
      const PrefillTile first = td[i];
      int at = i;
      while (true) {
        const int from = sort_keys[at].idx;
        sort_keys[at].idx = -1;
        if (from == i) {
          td[at] = first;
          break;
        }
        td[at] = td[from];
        at = from;
      }
    }
  } else {
    std::sort(td, td + n_tiles, [&](const PrefillTile& x, const PrefillTile& y) {
      return key_less(SortKey{work(x), group(x), x.q_row0, x.tok0, x.key_lo, 0, 0},
                      SortKey{work(y), group(y), y.q_row0, y.tok0, y.key_lo, 0, 0});
    });
  }
  for (size_t i = 0; i < tiles.size(); ++i) {
    const int gi = group(tiles.data()[i]);
    lay.n_dec_tiles += gi == 2 ? 1 : 0;
    lay.n_short_tiles += gi == 1 ? 1 : 0;
  }

  lay.n_units = (int)units.size();
  lay.n_merges = (int)merges.size();
  lay.n_tiles = (int)tiles.size();
  size_t off = 0;
  lay.off_units = off;
  off = plan_align_up(off + units.size() * sizeof(DecodeUnit));
  lay.off_merges = off;
  off = plan_align_up(off + merges.size() * sizeof(MergeItem));
  lay.off_tiles = off;
  off = plan_align_up(off + tiles.size() * sizeof(PrefillTile));
  lay.off_sched = off;
  off += kPlanAlign;
  lay.plan_bytes = off;
  lay.off_part_o = off;
  off = plan_align_up(off + (size_t)lay.n_parts * d.num_qo_heads * d.head_dim * sizeof(float));
  lay.off_part_lse = off;
  off = plan_align_up(off + (size_t)lay.n_parts * d.num_qo_heads * sizeof(float));
  lay.total = (units.size() == 0 && tiles.size() == 0) ? 0 : off;
  return DAA_OK;
}

// Copy the plan into a host staging buffer laid out as the workspace head.
template <class UnitVec, class MergeVec, class TileVec>
void plan_stage(const PlanLayout& lay, const UnitVec& units, const MergeVec& merges,
                const TileVec& tiles, uint8_t* host) {
  std::memset(host, 0, lay.plan_bytes);
  if (units.size()) std::memcpy(host + lay.off_units, units.data(), units.size() * sizeof(DecodeUnit));
  if (merges.size()) std::memcpy(host + lay.off_merges, merges.data(), merges.size() * sizeof(MergeItem));
  if (tiles.size()) std::memcpy(host + lay.off_tiles, tiles.data(), tiles.size() * sizeof(PrefillTile));
}

}  // namespace daa
