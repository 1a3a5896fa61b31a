// Host-only harness for tests/test_plan.py: builds the library's work plan for
// batches read from stdin and prints it, so the test can check on the CPU that
// every (query row, visible key) pair is attended exactly once and that every
// row's partial results are merged.  Compiled with g++ against the library's
// planner header; runs no CUDA call.
//
// Input, per case (whitespace separated):
//   Hq Hkv head_dim page_size num_pages sms
//   batch  qo_indptr[batch+1]  kv_indptr[batch+1]  last_page_len[batch]
//   n_groups  (if n_groups >= 0: prefix_indptr[n_groups+1] prefix_len[n_groups])
// (n_groups = -1: the plain plan).  Output, per case: "S status", then
//   "U q_row page_base tok_begin tok_end kv_len part" per decode unit,
//   "M q_row part_begin n_parts extra" per merge item,
//   "T q_row0 qo_len kv_len page_base tok0 ntok ntok1 key_lo key_hi part part_stride kind"
//   per tensor-core item (launch order),
//   "L n_units n_merges n_tiles n_dec_tiles n_short_tiles n_parts", and "E".
#include <cstdio>
#include <vector>

#include "planner.h"

namespace {

template <class T>
struct Vec {
  std::vector<T> v;
  bool push_back(const T& x) {
    v.push_back(x);
    return true;
  }
  size_t size() const { return v.size(); }
  T* data() { return v.data(); }
  const T* data() const { return v.data(); }
  void clear() { v.clear(); }
};

bool read_ints(std::vector<int32_t>& a, int n) {
  a.resize(n);
  for (int i = 0; i < n; ++i)
    if (std::scanf("%d", &a[i]) != 1) return false;
  return true;
}

}  // namespace

int main() {
  int Hq, Hkv, d, P, sms;
  long long num_pages;
  while (std::scanf("%d %d %d %d %lld %d", &Hq, &Hkv, &d, &P, &num_pages, &sms) == 6) {
    int batch, ng;
    std::vector<int32_t> qo, kv, last, ind, plen;
    if (std::scanf("%d", &batch) != 1 || !read_ints(qo, batch + 1) || !read_ints(kv, batch + 1) ||
        !read_ints(last, batch) || std::scanf("%d", &ng) != 1)
      return 2;
    daa::PrefixGroups groups{};
    if (ng >= 0) {
      if (!read_ints(ind, ng + 1) || !read_ints(plen, ng)) return 2;
      groups.indptr = ind.data();
      groups.prefix_len = plen.data();
      groups.n = ng;
    }
    daa_dims dims{Hq, Hkv, d, P, num_pages};
    Vec<daa::DecodeUnit> units;
    Vec<daa::MergeItem> merges;
    Vec<daa::PrefillTile> tiles;
    daa::PlanLayout lay;
    const daa_status st = daa::plan_batch(qo.data(), kv.data(), last.data(), batch, dims, sms,
                                          units, merges, tiles, lay, ng >= 0 ? &groups : nullptr);
    std::printf("S %d\n", (int)st);
    for (const auto& u : units.v)
      std::printf("U %d %d %d %d %d %d\n", u.q_row, u.page_base, u.tok_begin, u.tok_end, u.kv_len,
                  u.part);
    for (const auto& m : merges.v)
      std::printf("M %d %d %d %d\n", m.q_row, m.part_begin, m.n_parts, m.extra);
    for (const auto& t : tiles.v)
      std::printf("T %d %d %d %d %d %d %d %d %d %d %d %d\n", t.q_row0, t.qo_len, t.kv_len,
                  t.page_base, t.tok0, t.ntok, t.ntok1, t.key_lo, t.key_hi, t.part, t.part_stride,
                  t.kind);
    std::printf("L %d %d %d %d %d %d\nE\n", lay.n_units, lay.n_merges, lay.n_tiles, lay.n_dec_tiles,
                lay.n_short_tiles, lay.n_parts);
  }
  return 0;
}
