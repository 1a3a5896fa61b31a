// C ABI of libdaa: argument validation, the host-side plan of the batch, and
// the launches.  Host code only (plus the device error word).
//
// The plan follows "Disaggregated prefill and decode" (Perplexity), "Prefill vs
// decode performance": attention parallelises over requests and over kv_len.
// Decode requests (qo_len == 1) are cut into page-aligned key splits so that the
// number of CTAs covers the SMs several times over and no single split is long
// enough to leave a tail; their partial results are combined by softmax_merge
// ("Chunked prefill" (k4i.top), #correctness).  Prefill requests (qo_len > 1)
// are cut into 128-row tiles of packed (token, query head) rows, longest causal
// key range first.  The plan is built from the host mirrors of the indptr
// arrays, so no call waits on the device.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/daa.h"
#include "launch.h"

namespace daa {

__device__ int g_daa_device_error = 0;

int* device_error_word() {
  static int* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_daa_device_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<int*>(p);
  }
  return addr[dev];
}

namespace {

constexpr int kPageSize = 16;
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;
  }
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

daa_status check_dims(const daa_dims& d) {
  if (d.num_qo_heads <= 0 || d.num_kv_heads <= 0 || d.head_dim <= 0 || d.page_size <= 0 ||
      d.num_pages <= 0)
    return DAA_ERR_INVALID_ARG;
  if (d.num_qo_heads % d.num_kv_heads != 0) return DAA_ERR_INVALID_ARG;
  if (d.head_dim != 64 && d.head_dim != 128) return DAA_ERR_UNSUPPORTED;
  if (d.page_size != kPageSize) return DAA_ERR_UNSUPPORTED;
  const int g = d.num_qo_heads / d.num_kv_heads;
  if (g < 1 || g > 16) return DAA_ERR_UNSUPPORTED;
  // slices of the pool must be addressable by 32-bit TMA coordinates
  if (d.num_pages * 2 * (int64_t)d.num_kv_heads > (int64_t)INT32_MAX) return DAA_ERR_UNSUPPORTED;
  return DAA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

struct HostPlan {
  std::vector<DecodeUnit> units;
  std::vector<MergeItem> merges;
  std::vector<PrefillTile> tiles;
  int n_parts = 0;
  size_t off_units = 0, off_merges = 0, off_tiles = 0, plan_bytes = 0;
  size_t off_part_o = 0, off_part_lse = 0, total = 0;
};

daa_status make_plan(const int32_t* qo, const int32_t* kv, const int32_t* last, int32_t batch,
                     const daa_dims& d, int sms, HostPlan& pl) {
  daa_status st = check_dims(d);
  if (st != DAA_OK) return st;
  if (batch < 0) return DAA_ERR_INVALID_ARG;
  if (batch > 0 && (!qo || !kv || !last)) return DAA_ERR_INVALID_ARG;
  if (batch == 0) return DAA_OK;
  if (qo[0] != 0 || kv[0] != 0) return DAA_ERR_SHAPE;
  const int P = d.page_size;
  const int g = d.num_qo_heads / d.num_kv_heads;
  const int64_t Hkv = d.num_kv_heads;

  int64_t dec_pages = 0;
  for (int r = 0; r < batch; ++r) {
    const int64_t nq = (int64_t)qo[r + 1] - qo[r];
    const int64_t np = (int64_t)kv[r + 1] - kv[r];
    if (nq < 0 || np < 0) return DAA_ERR_SHAPE;
    if (np > 0 && (last[r] < 1 || last[r] > P)) return DAA_ERR_SHAPE;
    const int64_t kv_len = np > 0 ? (np - 1) * P + last[r] : 0;
    if (nq > kv_len) return DAA_ERR_SHAPE;
    if (kv_len > INT32_MAX / 2) return DAA_ERR_SHAPE;
    if (nq == 1) dec_pages += np;
  }

  // decode split size (pages): enough CTAs that the longest split is a small
  // fraction of the whole pass, never fewer pages than fill the copy pipeline
  const int64_t page_heads = dec_pages * Hkv;
  int64_t split = (page_heads + (int64_t)sms * 40 - 1) / ((int64_t)sms * 40);
  split = std::max<int64_t>(16, std::min<int64_t>(1024, split));

  std::vector<DecodeUnit> full_units, tail_units;
  for (int r = 0; r < batch; ++r) {
    const int nq = qo[r + 1] - qo[r];
    if (nq != 1) continue;
    const int np = kv[r + 1] - kv[r];
    const int kv_len = (np - 1) * P + last[r];
    const int nsplit = (int)((np + split - 1) / split);
    const int part0 = nsplit > 1 ? pl.n_parts : -1;
    if (nsplit > 1) {
      pl.merges.push_back(MergeItem{qo[r], pl.n_parts, nsplit, 0});
      pl.n_parts += nsplit;
    }
    for (int s = 0; s < nsplit; ++s) {
      DecodeUnit u{};
      u.q_row = qo[r];
      u.page_base = kv[r];
      u.tok_begin = (int)(s * split * P);
      u.tok_end = std::min<int>(kv_len, (int)((s + 1) * split * P));
      u.kv_len = kv_len;
      u.part = part0 >= 0 ? part0 + s : -1;
      (u.tok_end - u.tok_begin == split * P ? full_units : tail_units).push_back(u);
    }
  }
  std::stable_sort(tail_units.begin(), tail_units.end(), [](const DecodeUnit& x, const DecodeUnit& y) {
    return (x.tok_end - x.tok_begin) > (y.tok_end - y.tok_begin);
  });
  pl.units = std::move(full_units);
  pl.units.insert(pl.units.end(), tail_units.begin(), tail_units.end());

  // prefill tiles: pairs of 128-row tiles (ntok * g <= 128 packed rows each;
  // the second tile's tokens in pad0), longest key range first
  const int tpt = kPrefillTileRows / g;
  std::vector<std::pair<int, PrefillTile>> tw;
  for (int r = 0; r < batch; ++r) {
    const int nq = qo[r + 1] - qo[r];
    if (nq < 2) continue;
    const int np = kv[r + 1] - kv[r];
    const int kv_len = (np - 1) * P + last[r];
    for (int t0 = 0; t0 < nq; t0 += 2 * tpt) {
      PrefillTile t{};
      t.q_row0 = qo[r];
      t.qo_len = nq;
      t.kv_len = kv_len;
      t.page_base = kv[r];
      t.tok0 = t0;
      t.ntok = std::min(tpt, nq - t0);
      t.pad0 = t.ntok == tpt ? std::max(0, std::min(tpt, nq - t0 - tpt)) : 0;  // second tile
      const int keys = std::min(kv_len, kv_len - nq + t0 + t.ntok + t.pad0);
      tw.emplace_back(keys, t);
    }
  }
  std::stable_sort(tw.begin(), tw.end(),
                   [](const auto& x, const auto& y) { return x.first > y.first; });
  for (auto& x : tw) pl.tiles.push_back(x.second);

  size_t off = 0;
  pl.off_units = off;
  off = align_up(off + pl.units.size() * sizeof(DecodeUnit));
  pl.off_merges = off;
  off = align_up(off + pl.merges.size() * sizeof(MergeItem));
  pl.off_tiles = off;
  off = align_up(off + pl.tiles.size() * sizeof(PrefillTile));
  pl.plan_bytes = off;
  pl.off_part_o = off;
  off = align_up(off + (size_t)pl.n_parts * d.num_qo_heads * d.head_dim * sizeof(float));
  pl.off_part_lse = off;
  off = align_up(off + (size_t)pl.n_parts * d.num_qo_heads * sizeof(float));
  pl.total = (pl.units.empty() && pl.tiles.empty()) ? 0 : off;
  return DAA_OK;
}

// ------------------------------------------------------------------ tracing
struct Tracer {
  std::mutex mu;
  bool on = false;
  int cap = 0, n = 0;
  std::vector<cudaEvent_t> b, e;
  std::vector<int32_t> id;
  void clear_events() {
    for (auto ev : b) cudaEventDestroy(ev);
    for (auto ev : e) cudaEventDestroy(ev);
    b.clear();
    e.clear();
    id.clear();
    cap = n = 0;
  }
};
Tracer& tracer() {
  static Tracer t;
  return t;
}

template <typename F>
cudaError_t traced(int32_t kid, cudaStream_t s, F&& launch) {
  Tracer& t = tracer();
  int slot = -1;
  {
    std::lock_guard<std::mutex> g(t.mu);
    if (t.on && t.n < t.cap) slot = t.n++;
  }
  if (slot >= 0) {
    t.id[slot] = kid;
    cudaEventRecord(t.b[slot], s);
  }
  cudaError_t err = launch();
  if (slot >= 0) cudaEventRecord(t.e[slot], s);
  return err;
}

std::vector<uint8_t>& staging() {
  thread_local std::vector<uint8_t> buf;
  return buf;
}

}  // namespace
}  // namespace daa

using namespace daa;

extern "C" {

const char* daa_status_string(daa_status s) {
  switch (s) {
    case DAA_OK: return "ok";
    case DAA_ERR_INVALID_ARG: return "invalid argument";
    case DAA_ERR_SHAPE: return "inconsistent shapes (indptr, qo_len > kv_len or last_page_len)";
    case DAA_ERR_PAGE_RANGE: return "page range";
    case DAA_ERR_UNSUPPORTED: return "unsupported shape (head_dim, page_size or group size)";
    case DAA_ERR_CUDA: return "CUDA error";
    case DAA_ERR_WORKSPACE: return "workspace missing or too small";
    case DAA_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
  }
  return "unknown status";
}

int32_t daa_version(void) { return 100; }

daa_status daa_kv_append(const void* k_new, const void* v_new, void* kv_pages,
                         const int32_t* append_indptr, const int32_t* page_indices,
                         const int32_t* kv_indptr, const int32_t* last_page_len, int32_t batch,
                         int32_t nnz_new, daa_dims dims, void* stream) {
  daa_status st = check_dims(dims);
  if (st != DAA_OK) return st;
  if (batch < 0 || nnz_new < 0) return DAA_ERR_INVALID_ARG;
  if (nnz_new == 0 || batch == 0) return nnz_new == 0 ? DAA_OK : DAA_ERR_SHAPE;
  if (!k_new || !v_new || !kv_pages || !append_indptr || !page_indices || !kv_indptr ||
      !last_page_len)
    return DAA_ERR_INVALID_ARG;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(kv_pages)) return DAA_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* err = device_error_word();
  cudaError_t e = traced(kKernelAppend, s, [&] {
    return launch_kv_append(k_new, v_new, kv_pages, append_indptr, page_indices, kv_indptr,
                            last_page_len, batch, nnz_new, dims.num_kv_heads, dims.head_dim,
                            dims.num_pages, num_sms(), err, s);
  });
  return e == cudaSuccess ? DAA_OK : DAA_ERR_CUDA;
}

size_t daa_batch_attention_workspace_size(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                          const int32_t* h_last_page_len, int32_t batch,
                                          daa_dims dims, daa_status* status) {
  HostPlan pl;
  daa_status st = make_plan(h_qo_indptr, h_kv_indptr, h_last_page_len, batch, dims, num_sms(), pl);
  if (status) *status = st;
  return st == DAA_OK ? pl.total : 0;
}

daa_status daa_batch_attention(const void* q, const void* kv_pages, const int32_t* qo_indptr,
                               const int32_t* kv_indptr, const int32_t* page_indices,
                               const int32_t* last_page_len, const int32_t* h_qo_indptr,
                               const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
                               int32_t batch, int32_t causal, float sm_scale, void* out,
                               float* lse_out, void* workspace, size_t workspace_bytes,
                               daa_dims dims, void* stream) {
  if (!(std::isfinite(sm_scale))) return DAA_ERR_INVALID_ARG;
  HostPlan pl;
  daa_status st = make_plan(h_qo_indptr, h_kv_indptr, h_last_page_len, batch, dims, num_sms(), pl);
  if (st != DAA_OK) return st;
  if (pl.units.empty() && pl.tiles.empty()) return DAA_OK;
  if (!q || !kv_pages || !qo_indptr || !kv_indptr || !page_indices || !last_page_len || !out)
    return DAA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_pages) || !aligned16(out)) return DAA_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(lse_out) & 3) != 0) return DAA_ERR_ALIGNMENT;
  if (!workspace || workspace_bytes < pl.total) return DAA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DAA_ERR_ALIGNMENT;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  std::vector<uint8_t>& host = staging();
  host.assign(pl.plan_bytes, 0);
  if (!pl.units.empty())
    std::memcpy(host.data() + pl.off_units, pl.units.data(), pl.units.size() * sizeof(DecodeUnit));
  if (!pl.merges.empty())
    std::memcpy(host.data() + pl.off_merges, pl.merges.data(), pl.merges.size() * sizeof(MergeItem));
  if (!pl.tiles.empty())
    std::memcpy(host.data() + pl.off_tiles, pl.tiles.data(), pl.tiles.size() * sizeof(PrefillTile));
  if (cudaMemcpyAsync(ws, host.data(), pl.plan_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DAA_ERR_CUDA;

  int* err = device_error_word();
  const int g = dims.num_qo_heads / dims.num_kv_heads;
  const float sc = sm_scale * 1.4426950408889634f;
  const int nnz_qo = h_qo_indptr[batch];
  cudaError_t e = cudaSuccess;

  if (!pl.tiles.empty()) {
    PrefillArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.pool = static_cast<const uint16_t*>(kv_pages);
    a.page_indices = page_indices;
    a.tiles = reinterpret_cast<const PrefillTile*>(ws + pl.off_tiles);
    a.n_tiles = (int)pl.tiles.size();
    a.Hq = dims.num_qo_heads;
    a.Hkv = dims.num_kv_heads;
    a.group = g;
    a.head_dim = dims.head_dim;
    a.num_pages = dims.num_pages;
    a.nnz_qo = nnz_qo;
    a.causal = causal ? 1 : 0;
    a.sm_scale_log2 = sc;
    a.out = static_cast<uint16_t*>(out);
    a.lse_out = lse_out;
    a.err = err;
    e = traced(kKernelPrefill, s, [&] { return launch_prefill(a, s); });
    if (e != cudaSuccess) return DAA_ERR_CUDA;
  }
  if (!pl.units.empty()) {
    DecodeArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.pool = static_cast<const uint16_t*>(kv_pages);
    a.page_indices = page_indices;
    a.units = reinterpret_cast<const DecodeUnit*>(ws + pl.off_units);
    a.n_units = (int)pl.units.size();
    a.Hq = dims.num_qo_heads;
    a.Hkv = dims.num_kv_heads;
    a.group = g;
    a.head_dim = dims.head_dim;
    a.num_pages = dims.num_pages;
    a.sm_scale_log2 = sc;
    a.out = static_cast<uint16_t*>(out);
    a.lse_out = lse_out;
    a.part_o = reinterpret_cast<float*>(ws + pl.off_part_o);
    a.part_lse = reinterpret_cast<float*>(ws + pl.off_part_lse);
    a.err = err;
    e = traced(kKernelDecode, s, [&] { return launch_decode(a, s); });
    if (e != cudaSuccess) return DAA_ERR_CUDA;
    if (!pl.merges.empty()) {
      MergeArgs m{};
      m.items = reinterpret_cast<const MergeItem*>(ws + pl.off_merges);
      m.n_items = (int)pl.merges.size();
      m.Hq = dims.num_qo_heads;
      m.head_dim = dims.head_dim;
      m.part_o = a.part_o;
      m.part_lse = a.part_lse;
      m.out = a.out;
      m.lse_out = lse_out;
      e = traced(kKernelMerge, s, [&] { return launch_merge(m, s); });
      if (e != cudaSuccess) return DAA_ERR_CUDA;
    }
  }
  return DAA_OK;
}

daa_status daa_device_error(int32_t* code, int32_t reset) {
  if (!code) return DAA_ERR_INVALID_ARG;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_daa_device_error, sizeof(int)) != cudaSuccess) return DAA_ERR_CUDA;
  *code = v;
  if (reset) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_daa_device_error, &zero, sizeof(int)) != cudaSuccess) return DAA_ERR_CUDA;
  }
  return DAA_OK;
}

daa_status daa_trace_enable(int32_t capacity) {
  if (capacity <= 0) return DAA_ERR_INVALID_ARG;
  Tracer& t = tracer();
  std::lock_guard<std::mutex> g(t.mu);
  t.clear_events();
  t.b.resize(capacity);
  t.e.resize(capacity);
  t.id.assign(capacity, 0);
  for (int i = 0; i < capacity; ++i) {
    if (cudaEventCreate(&t.b[i]) != cudaSuccess || cudaEventCreate(&t.e[i]) != cudaSuccess) {
      t.b.resize(i);
      t.e.resize(i);
      t.clear_events();
      return DAA_ERR_CUDA;
    }
  }
  t.cap = capacity;
  t.n = 0;
  t.on = true;
  return DAA_OK;
}

daa_status daa_trace_disable(void) {
  Tracer& t = tracer();
  std::lock_guard<std::mutex> g(t.mu);
  t.on = false;
  t.clear_events();
  return DAA_OK;
}

int32_t daa_trace_read(int32_t* kernel_ids, float* milliseconds, int32_t max_records) {
  Tracer& t = tracer();
  std::lock_guard<std::mutex> g(t.mu);
  int32_t n = std::min(t.n, max_records);
  for (int i = 0; i < n; ++i) {
    float ms = -1.f;
    if (cudaEventSynchronize(t.e[i]) == cudaSuccess) cudaEventElapsedTime(&ms, t.b[i], t.e[i]);
    if (kernel_ids) kernel_ids[i] = t.id[i];
    if (milliseconds) milliseconds[i] = ms;
  }
  t.n = 0;
  return n;
}

}  // extern "C"
