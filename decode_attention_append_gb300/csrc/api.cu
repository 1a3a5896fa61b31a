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
#include <atomic>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/daa.h"
#include "launch.h"
#include "planner.h"
#include "ptx.cuh"

namespace daa {

__device__ int g_daa_device_error = 0;
__device__ int g_daa_selftest_flag = 0;

// Self-test of the bounded wait every kernel uses: one thread waits on the
// first phase of an mbarrier that nothing arrives on.  The wait must give up
// after its time limit, record kDevErrBarrierTimeout and let the kernel exit.
__global__ void selftest_wait_kernel(int* err, int* gave_up) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbar_init();
  *gave_up = mbar_wait(&bar, 0, err) ? 0 : 1;
}

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

constexpr size_t kAlign = kPlanAlign;

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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// growable plan containers (reused per host thread, so steady-state calls do
// not allocate)
template <class T>
struct HostVec {
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

struct HostPlan {
  HostVec<DecodeUnit> units;
  HostVec<MergeItem> merges;
  HostVec<PrefillTile> tiles;
  PlanLayout lay;
};

HostPlan& host_plan() {
  thread_local HostPlan p;
  return p;
}

daa_status make_plan(const int32_t* qo, const int32_t* kv, const int32_t* last, int32_t batch,
                     const daa_dims& d, int sms, HostPlan& pl,
                     const PrefixGroups* groups = nullptr) {
  return plan_batch(qo, kv, last, batch, d, sms, pl.units, pl.merges, pl.tiles, pl.lay, groups);
}

// Host prefix groups of a shared-prefix call, checked for null arrays and a
// negative count (the planner checks them against the page table).
// What daa_batch_attention_plan leaves in the caller's daa_plan_info: the
// plan's layout in the workspace and the shapes it was made for.
struct PlanRecord {
  int64_t magic;
  int64_t num_qo_heads, num_kv_heads, head_dim, page_size, num_pages;
  int64_t batch, nnz_qo;
  PlanLayout lay;
  // rows the append kernel of a fused run covers with the prefill append
  // fused (append_span at the fusion threshold of these dims)
  int32_t fused_span_begin, fused_span_end;
};
constexpr int64_t kPlanMagic = 0x4441415f504c414eLL;  // "DAA_PLAN"
static_assert(sizeof(PlanRecord) <= sizeof(daa_plan_info), "daa_plan_info too small");

daa_status make_groups(const int32_t* h_prefix_indptr, const int32_t* h_prefix_len,
                       int32_t n_groups, PrefixGroups& g) {
  if (n_groups < 0) return DAA_ERR_INVALID_ARG;
  if (n_groups > 0 && (!h_prefix_indptr || !h_prefix_len)) return DAA_ERR_INVALID_ARG;
  g.indptr = h_prefix_indptr;
  g.prefix_len = h_prefix_len;
  g.n = n_groups;
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

bool tracing() {
  Tracer& t = tracer();
  std::lock_guard<std::mutex> g(t.mu);
  return t.on;
}

std::vector<uint8_t>& staging() {
  thread_local std::vector<uint8_t> buf;
  return buf;
}

// Fused calls: whether the prefill kernels read their chunk's own key tiles
// from k_new / v_new and write them into the pages themselves (1, the
// default), or the append kernel writes every row and the prefill reads them
// back from the pages (0).  Results are identical either way.
std::atomic<int> g_fuse_prefill_append{1};

// The smallest qo_len whose rows the prefill kernel appends in a fused call:
// requests planned as prefill items (more rows than two 128-row Q tiles hold:
// CTA-pair items for head_dim 128, single-CTA items for head_dim 64); 0 when
// nothing is fused.
int fuse_threshold(const daa_dims& d) {
  const int g = d.num_qo_heads / d.num_kv_heads;
  return 2 * (kPrefillTileRows / g) + 1;
}
int fuse_min_qo_for(const daa_dims& d) {
  return g_fuse_prefill_append.load(std::memory_order_relaxed) ? fuse_threshold(d) : 0;
}

}  // namespace

daa_status launch_all(const LaunchSet& ls, const PlanLayout& lay, cudaStream_t s, bool trace,
                      bool after_append) {
  const daa_dims& dims = ls.dims;
  const int g = dims.num_qo_heads / dims.num_kv_heads;
  const float sc = ls.sm_scale * 1.4426950408889634f;
  uint8_t* ws = static_cast<uint8_t*>(ls.scratch);
  float* part_o = reinterpret_cast<float*>(ws + lay.off_part_o);
  float* part_lse = reinterpret_cast<float*>(ws + lay.off_part_lse);
  auto run = [&](int32_t kid, auto&& f) -> cudaError_t {
    return trace ? traced(kid, s, f) : f();
  };
  // programmatic launches, except while the tracer brackets every launch with
  // events (each kernel is then timed alone)
  bool programmatic = after_append && !(trace && tracing());
  if (lay.n_tiles > 0) {
    PrefillArgs a{};
    a.q = static_cast<const uint16_t*>(ls.q);
    a.pool = static_cast<const uint16_t*>(ls.kv_pages);
    a.page_indices = ls.page_indices;
    a.tiles = reinterpret_cast<const PrefillTile*>(ws + lay.off_tiles);
    a.n_tiles = lay.n_tiles - lay.n_dec_tiles - lay.n_short_tiles;
    a.short_tiles = a.tiles + a.n_tiles;
    a.n_short_tiles = lay.n_short_tiles;
    a.dec_tiles = a.short_tiles + a.n_short_tiles;
    a.n_dec_tiles = lay.n_dec_tiles;
    a.Hq = dims.num_qo_heads;
    a.Hkv = dims.num_kv_heads;
    a.group = g;
    a.head_dim = dims.head_dim;
    a.num_pages = dims.num_pages;
    a.nnz_qo = ls.nnz_qo;
    a.causal = ls.causal ? 1 : 0;
    a.sm_scale_log2 = sc;
    a.out = static_cast<uint16_t*>(ls.out);
    a.lse_out = ls.lse_out;
    a.part_o = part_o;
    a.part_lse = part_lse;
    a.tree_mask = ls.tree_mask;
    a.mask_words = ls.mask_words;
    a.err = ls.err;
    a.dec_counter = reinterpret_cast<int*>(ws + lay.off_sched);
    a.sms = ls.sms;
    a.k_new = static_cast<const uint16_t*>(ls.k_new);
    a.v_new = static_cast<const uint16_t*>(ls.v_new);
    a.pool_w = const_cast<uint16_t*>(static_cast<const uint16_t*>(ls.kv_pages));
    a.fuse_min_qo = ls.k_new && ls.v_new ? ls.fuse_min_qo : 0;
    if (a.n_tiles > 0) {
      const bool quads = plan_prefill_quads(dims);
      if (run(kKernelPrefill, [&] {
            return quads ? launch_prefill_pair(a, s, programmatic)
                         : launch_prefill(a, a.tiles, a.n_tiles, s, programmatic);
          }) != cudaSuccess)
        return DAA_ERR_CUDA;
      programmatic = !(trace && tracing());
    }
    if (a.n_short_tiles > 0) {
      if (run(kKernelShort, [&] {
            return launch_prefill(a, a.short_tiles, a.n_short_tiles, s, programmatic);
          }) != cudaSuccess)
        return DAA_ERR_CUDA;
      programmatic = !(trace && tracing());
    }
    if (a.n_dec_tiles > 0) {
      if (run(kKernelTcDecode, [&] { return launch_tc_decode(a, s, programmatic); }) != cudaSuccess)
        return DAA_ERR_CUDA;
      programmatic = !(trace && tracing());
    }
  }
  if (lay.n_units > 0) {
    DecodeArgs a{};
    a.q = static_cast<const uint16_t*>(ls.q);
    a.pool = static_cast<const uint16_t*>(ls.kv_pages);
    a.page_indices = ls.page_indices;
    a.units = reinterpret_cast<const DecodeUnit*>(ws + lay.off_units);
    a.n_units = lay.n_units;
    a.Hq = dims.num_qo_heads;
    a.Hkv = dims.num_kv_heads;
    a.group = g;
    a.head_dim = dims.head_dim;
    a.num_pages = dims.num_pages;
    a.sm_scale_log2 = sc;
    a.out = static_cast<uint16_t*>(ls.out);
    a.lse_out = ls.lse_out;
    a.part_o = part_o;
    a.part_lse = part_lse;
    a.err = ls.err;
    if (run(kKernelDecode, [&] { return launch_decode(a, s, programmatic); }) != cudaSuccess)
      return DAA_ERR_CUDA;
    programmatic = !(trace && tracing());
  }
  if (lay.n_merges > 0) {
    MergeArgs m{};
    m.items = reinterpret_cast<const MergeItem*>(ws + lay.off_merges);
    m.n_items = lay.n_merges;
    m.Hq = dims.num_qo_heads;
    m.head_dim = dims.head_dim;
    m.part_o = part_o;
    m.part_lse = part_lse;
    m.out = static_cast<uint16_t*>(ls.out);
    m.lse_out = ls.lse_out;
    if (run(kKernelMerge, [&] { return launch_merge(m, s, programmatic); }) != cudaSuccess)
      return DAA_ERR_CUDA;
  }
  return DAA_OK;
}

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
  daa_status st = plan_check_dims(dims);
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
                            last_page_len, batch, 0, nnz_new, dims.num_kv_heads, dims.head_dim,
                            dims.num_pages, num_sms(), /*fuse_min_qo=*/0, err, s);
  });
  return e == cudaSuccess ? DAA_OK : DAA_ERR_CUDA;
}

size_t daa_batch_attention_workspace_size(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                          const int32_t* h_last_page_len, int32_t batch,
                                          daa_dims dims, daa_status* status) {
  HostPlan& pl = host_plan();
  daa_status st = make_plan(h_qo_indptr, h_kv_indptr, h_last_page_len, batch, dims, num_sms(), pl);
  if (status) *status = st;
  return st == DAA_OK ? pl.lay.total : 0;
}

size_t daa_batch_attention_shared_prefix_workspace_size(
    const int32_t* h_qo_indptr, const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
    int32_t batch, const int32_t* h_prefix_indptr, const int32_t* h_prefix_len, int32_t n_groups,
    daa_dims dims, daa_status* status) {
  PrefixGroups g{};
  daa_status st = make_groups(h_prefix_indptr, h_prefix_len, n_groups, g);
  HostPlan& pl = host_plan();
  if (st == DAA_OK)
    st = make_plan(h_qo_indptr, h_kv_indptr, h_last_page_len, batch, dims, num_sms(), pl, &g);
  if (status) *status = st;
  return st == DAA_OK ? pl.lay.total : 0;
}

}  // extern "C"

namespace {

// Work a caller enqueues once the arguments have been checked and before the
// call's own work (the host step's input upload); a failure is returned as is.
struct BeforeEnqueue {
  daa_status (*fn)(void* ctx);
  void* ctx;
};

// Shared body of daa_batch_attention and daa_append_attention: validate, plan,
// stage the plan, then (fused call) launch the append, then the attention.
daa_status attention_call(const void* k_new, const void* v_new, const void* q,
                          const void* kv_pages, const int32_t* qo_indptr,
                          const int32_t* kv_indptr, const int32_t* page_indices,
                          const int32_t* last_page_len, const int32_t* h_qo_indptr,
                          const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
                          int32_t batch, int32_t causal, float sm_scale, void* out,
                          float* lse_out, void* workspace, size_t workspace_bytes,
                          const daa_dims& dims, void* stream, bool fused,
                          const uint32_t* tree_mask = nullptr, int32_t mask_words = 0,
                          const PrefixGroups* groups = nullptr,
                          const BeforeEnqueue* before = nullptr) {
  if (!(std::isfinite(sm_scale)) || !(sm_scale > 0.f)) return DAA_ERR_INVALID_ARG;
  HostPlan& pl = host_plan();
  daa_status st =
      make_plan(h_qo_indptr, h_kv_indptr, h_last_page_len, batch, dims, num_sms(), pl, groups);
  if (st != DAA_OK) return st;
  if (tree_mask) {
    // the mask refines the causal rule; each request's new tokens fit its rows
    if (!causal || mask_words < 1) return DAA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(tree_mask) & 3) != 0) return DAA_ERR_ALIGNMENT;
    for (int r = 0; r < batch; ++r)
      if ((int64_t)h_qo_indptr[r + 1] - h_qo_indptr[r] > 32 * (int64_t)mask_words)
        return DAA_ERR_SHAPE;
  }
  const PlanLayout& lay = pl.lay;
  if (lay.n_units == 0 && lay.n_tiles == 0) return DAA_OK;
  if (!q || !kv_pages || !qo_indptr || !kv_indptr || !page_indices || !last_page_len || !out)
    return DAA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_pages) || !aligned16(out)) return DAA_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(lse_out) & 3) != 0) return DAA_ERR_ALIGNMENT;
  if (fused) {
    if (!k_new || !v_new) return DAA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return DAA_ERR_ALIGNMENT;
  }
  if (!workspace || workspace_bytes < lay.total) return DAA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DAA_ERR_ALIGNMENT;
  if (before) {
    st = before->fn(before->ctx);
    if (st != DAA_OK) return st;
  }

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  std::vector<uint8_t>& host = staging();
  if (host.size() < lay.plan_bytes) host.resize(lay.plan_bytes);
  plan_stage(lay, pl.units, pl.merges, pl.tiles, host.data());
  if (cudaMemcpyAsync(ws, host.data(), lay.plan_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DAA_ERR_CUDA;
  const int nnz_qo = h_qo_indptr[batch];
  // the tree call never fuses (its mask path appends separately)
  const int fuse_min_qo = fused && !tree_mask ? fuse_min_qo_for(dims) : 0;
  // the append kernel covers only the rows the prefill kernels do not write
  const AppendSpan span = fused ? append_span(h_qo_indptr, h_kv_indptr, h_last_page_len, batch,
                                              dims.page_size, fuse_min_qo)
                                : AppendSpan{0, 0};
  const bool appended = span.end > span.begin;
  if (appended) {
    int* err = device_error_word();
    cudaError_t e = traced(kKernelAppend, s, [&] {
      return launch_kv_append(k_new, v_new, const_cast<void*>(kv_pages), qo_indptr, page_indices,
                              kv_indptr, last_page_len, batch, span.begin, span.end - span.begin,
                              dims.num_kv_heads, dims.head_dim, dims.num_pages, num_sms(),
                              fuse_min_qo, err, s);
    });
    if (e != cudaSuccess) return DAA_ERR_CUDA;
  }
  LaunchSet ls{};
  ls.q = q;
  ls.kv_pages = kv_pages;
  ls.page_indices = page_indices;
  ls.dims = dims;
  ls.causal = causal;
  ls.sm_scale = sm_scale;
  ls.nnz_qo = nnz_qo;
  ls.out = out;
  ls.lse_out = lse_out;
  ls.tree_mask = tree_mask;
  ls.mask_words = tree_mask ? mask_words : 0;
  ls.scratch = ws;
  ls.err = device_error_word();
  ls.sms = num_sms();
  if (fused) {
    ls.k_new = k_new;
    ls.v_new = v_new;
    ls.fuse_min_qo = fuse_min_qo;
  }
  return launch_all(ls, lay, s, /*trace=*/true, /*after_append=*/appended);
}

}  // namespace

extern "C" {

daa_status daa_batch_attention(const void* q, const void* kv_pages, const int32_t* qo_indptr,
                               const int32_t* kv_indptr, const int32_t* page_indices,
                               const int32_t* last_page_len, const int32_t* h_qo_indptr,
                               const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
                               int32_t batch, int32_t causal, float sm_scale, void* out,
                               float* lse_out, void* workspace, size_t workspace_bytes,
                               daa_dims dims, void* stream) {
  return attention_call(nullptr, nullptr, q, kv_pages, qo_indptr, kv_indptr, page_indices,
                        last_page_len, h_qo_indptr, h_kv_indptr, h_last_page_len, batch, causal,
                        sm_scale, out, lse_out, workspace, workspace_bytes, dims, stream, false);
}

daa_status daa_append_attention(const void* k_new, const void* v_new, const void* q,
                                void* kv_pages, const int32_t* qo_indptr,
                                const int32_t* kv_indptr, const int32_t* page_indices,
                                const int32_t* last_page_len, const int32_t* h_qo_indptr,
                                const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
                                int32_t batch, int32_t causal, float sm_scale, void* out,
                                float* lse_out, void* workspace, size_t workspace_bytes,
                                daa_dims dims, void* stream) {
  return attention_call(k_new, v_new, q, kv_pages, qo_indptr, kv_indptr, page_indices,
                        last_page_len, h_qo_indptr, h_kv_indptr, h_last_page_len, batch, causal,
                        sm_scale, out, lse_out, workspace, workspace_bytes, dims, stream, true);
}

daa_status daa_batch_attention_tree(const void* q, const void* kv_pages,
                                    const int32_t* qo_indptr, const int32_t* kv_indptr,
                                    const int32_t* page_indices, const int32_t* last_page_len,
                                    const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                    const int32_t* h_last_page_len, int32_t batch,
                                    const uint32_t* tree_mask, int32_t mask_words, float sm_scale,
                                    void* out, float* lse_out, void* workspace,
                                    size_t workspace_bytes, daa_dims dims, void* stream) {
  if (!tree_mask) return DAA_ERR_INVALID_ARG;
  return attention_call(nullptr, nullptr, q, kv_pages, qo_indptr, kv_indptr, page_indices,
                        last_page_len, h_qo_indptr, h_kv_indptr, h_last_page_len, batch, 1,
                        sm_scale, out, lse_out, workspace, workspace_bytes, dims, stream, false,
                        tree_mask, mask_words);
}

daa_status daa_batch_attention_shared_prefix(
    const void* q, const void* kv_pages, const int32_t* qo_indptr, const int32_t* kv_indptr,
    const int32_t* page_indices, const int32_t* last_page_len, const int32_t* h_qo_indptr,
    const int32_t* h_kv_indptr, const int32_t* h_last_page_len, int32_t batch,
    const int32_t* h_prefix_indptr, const int32_t* h_prefix_len, int32_t n_groups, int32_t causal,
    float sm_scale, void* out, float* lse_out, void* workspace, size_t workspace_bytes,
    daa_dims dims, void* stream) {
  PrefixGroups g{};
  daa_status st = make_groups(h_prefix_indptr, h_prefix_len, n_groups, g);
  if (st != DAA_OK) return st;
  return attention_call(nullptr, nullptr, q, kv_pages, qo_indptr, kv_indptr, page_indices,
                        last_page_len, h_qo_indptr, h_kv_indptr, h_last_page_len, batch, causal,
                        sm_scale, out, lse_out, workspace, workspace_bytes, dims, stream, false,
                        nullptr, 0, &g);
}

daa_status daa_append_attention_shared_prefix(
    const void* k_new, const void* v_new, const void* q, void* kv_pages, const int32_t* qo_indptr,
    const int32_t* kv_indptr, const int32_t* page_indices, const int32_t* last_page_len,
    const int32_t* h_qo_indptr, const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
    int32_t batch, const int32_t* h_prefix_indptr, const int32_t* h_prefix_len, int32_t n_groups,
    int32_t causal, float sm_scale, void* out, float* lse_out, void* workspace,
    size_t workspace_bytes, daa_dims dims, void* stream) {
  PrefixGroups g{};
  daa_status st = make_groups(h_prefix_indptr, h_prefix_len, n_groups, g);
  if (st != DAA_OK) return st;
  return attention_call(k_new, v_new, q, kv_pages, qo_indptr, kv_indptr, page_indices,
                        last_page_len, h_qo_indptr, h_kv_indptr, h_last_page_len, batch, causal,
                        sm_scale, out, lse_out, workspace, workspace_bytes, dims, stream, true,
                        nullptr, 0, &g);
}

daa_status daa_batch_attention_plan(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                    const int32_t* h_last_page_len, int32_t batch,
                                    const int32_t* h_prefix_indptr, const int32_t* h_prefix_len,
                                    int32_t n_groups, daa_dims dims, void* workspace,
                                    size_t workspace_bytes, daa_plan_info* info, void* stream) {
  if (!info) return DAA_ERR_INVALID_ARG;
  std::memset(info, 0, sizeof(*info));
  PrefixGroups g{};
  daa_status st = make_groups(h_prefix_indptr, h_prefix_len, n_groups, g);
  if (st != DAA_OK) return st;
  HostPlan& pl = host_plan();
  st = make_plan(h_qo_indptr, h_kv_indptr, h_last_page_len, batch, dims, num_sms(), pl,
                 n_groups > 0 ? &g : nullptr);
  if (st != DAA_OK) return st;
  const PlanLayout& lay = pl.lay;
  if (lay.total > 0) {
    if (!workspace || workspace_bytes < lay.total) return DAA_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DAA_ERR_ALIGNMENT;
    std::vector<uint8_t>& host = staging();
    if (host.size() < lay.plan_bytes) host.resize(lay.plan_bytes);
    plan_stage(lay, pl.units, pl.merges, pl.tiles, host.data());
    if (cudaMemcpyAsync(workspace, host.data(), lay.plan_bytes, cudaMemcpyHostToDevice,
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return DAA_ERR_CUDA;
  }
  PlanRecord rec{};
  rec.magic = kPlanMagic;
  rec.num_qo_heads = dims.num_qo_heads;
  rec.num_kv_heads = dims.num_kv_heads;
  rec.head_dim = dims.head_dim;
  rec.page_size = dims.page_size;
  rec.num_pages = dims.num_pages;
  rec.batch = batch;
  rec.nnz_qo = batch > 0 ? h_qo_indptr[batch] : 0;
  rec.lay = lay;
  const AppendSpan span = append_span(h_qo_indptr, h_kv_indptr, h_last_page_len, batch,
                                      dims.page_size, fuse_threshold(dims));
  rec.fused_span_begin = span.begin;
  rec.fused_span_end = span.end;
  std::memcpy(info, &rec, sizeof(rec));
  return DAA_OK;
}

}  // extern "C"

namespace {

// Shared body of the two run calls: check the plan record against the call,
// then (fused) the append and the attention kernels.
daa_status run_call(const void* k_new, const void* v_new, const void* q, const void* kv_pages,
                    const int32_t* qo_indptr, const int32_t* kv_indptr,
                    const int32_t* page_indices, const int32_t* last_page_len,
                    const daa_plan_info* info, int32_t causal, float sm_scale, void* out,
                    float* lse_out, void* workspace, size_t workspace_bytes, daa_dims dims,
                    void* stream, bool fused) {
  if (!info) return DAA_ERR_INVALID_ARG;
  PlanRecord rec;
  std::memcpy(&rec, info, sizeof(rec));
  if (rec.magic != kPlanMagic || rec.num_qo_heads != dims.num_qo_heads ||
      rec.num_kv_heads != dims.num_kv_heads || rec.head_dim != dims.head_dim ||
      rec.page_size != dims.page_size || rec.num_pages != dims.num_pages)
    return DAA_ERR_INVALID_ARG;
  if (!(std::isfinite(sm_scale)) || !(sm_scale > 0.f)) return DAA_ERR_INVALID_ARG;
  const PlanLayout& lay = rec.lay;
  if (lay.n_units == 0 && lay.n_tiles == 0) return DAA_OK;
  if (!q || !kv_pages || !qo_indptr || !kv_indptr || !page_indices || !last_page_len || !out)
    return DAA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv_pages) || !aligned16(out)) return DAA_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(lse_out) & 3) != 0) return DAA_ERR_ALIGNMENT;
  if (fused) {
    if (!k_new || !v_new) return DAA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new)) return DAA_ERR_ALIGNMENT;
  }
  if (!workspace || workspace_bytes < lay.total) return DAA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1)) != 0) return DAA_ERR_ALIGNMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int nnz_qo = (int)rec.nnz_qo;
  const int fuse_min_qo = fused ? fuse_min_qo_for(dims) : 0;
  // rows the append kernel covers: those of the stored span with the fusion
  // on, every row with it off
  const AppendSpan span = !fused ? AppendSpan{0, 0}
                          : fuse_min_qo > 0 ? AppendSpan{rec.fused_span_begin, rec.fused_span_end}
                                            : AppendSpan{0, nnz_qo};
  const bool appended = span.end > span.begin;
  if (appended) {
    int* err = device_error_word();
    cudaError_t e = traced(kKernelAppend, s, [&] {
      return launch_kv_append(k_new, v_new, const_cast<void*>(kv_pages), qo_indptr, page_indices,
                              kv_indptr, last_page_len, (int)rec.batch, span.begin,
                              span.end - span.begin, dims.num_kv_heads, dims.head_dim,
                              dims.num_pages, num_sms(), fuse_min_qo, err, s);
    });
    if (e != cudaSuccess) return DAA_ERR_CUDA;
  }
  LaunchSet ls{};
  ls.q = q;
  ls.kv_pages = kv_pages;
  ls.page_indices = page_indices;
  ls.dims = dims;
  ls.causal = causal;
  ls.sm_scale = sm_scale;
  ls.nnz_qo = nnz_qo;
  ls.out = out;
  ls.lse_out = lse_out;
  ls.scratch = workspace;
  ls.err = device_error_word();
  ls.sms = num_sms();
  if (fused) {
    ls.k_new = k_new;
    ls.v_new = v_new;
    ls.fuse_min_qo = fuse_min_qo;
  }
  return launch_all(ls, lay, s, /*trace=*/true, /*after_append=*/appended);
}

}  // namespace

extern "C" {

daa_status daa_batch_attention_run(const void* q, const void* kv_pages, const int32_t* qo_indptr,
                                   const int32_t* kv_indptr, const int32_t* page_indices,
                                   const int32_t* last_page_len, const daa_plan_info* info,
                                   int32_t causal, float sm_scale, void* out, float* lse_out,
                                   void* workspace, size_t workspace_bytes, daa_dims dims,
                                   void* stream) {
  return run_call(nullptr, nullptr, q, kv_pages, qo_indptr, kv_indptr, page_indices,
                  last_page_len, info, causal, sm_scale, out, lse_out, workspace, workspace_bytes,
                  dims, stream, false);
}

daa_status daa_append_attention_run(const void* k_new, const void* v_new, const void* q,
                                    void* kv_pages, const int32_t* qo_indptr,
                                    const int32_t* kv_indptr, const int32_t* page_indices,
                                    const int32_t* last_page_len, const daa_plan_info* info,
                                    int32_t causal, float sm_scale, void* out, float* lse_out,
                                    void* workspace, size_t workspace_bytes, daa_dims dims,
                                    void* stream) {
  return run_call(k_new, v_new, q, kv_pages, qo_indptr, kv_indptr, page_indices, last_page_len,
                  info, causal, sm_scale, out, lse_out, workspace, workspace_bytes, dims, stream,
                  true);
}

}  // extern "C"

namespace {

// The host step's upload, enqueued by attention_call once every argument has
// passed its checks: the packed inputs on the upload stream (after the
// previous reader of the device copy), then the compute stream waits for them
// and for the previous read-back of the output buffer.
struct HostStepUpload {
  const void* h_inputs;
  void* d_inputs;
  size_t bytes;
  const daa_step_streams* ss;
};

daa_status host_step_upload(void* ctx) {
  const HostStepUpload& u = *static_cast<const HostStepUpload*>(ctx);
  cudaStream_t us = static_cast<cudaStream_t>(u.ss->upload_stream);
  cudaStream_t cs = static_cast<cudaStream_t>(u.ss->compute_stream);
  cudaEvent_t uploaded = static_cast<cudaEvent_t>(u.ss->uploaded);
  if (u.ss->inputs_free &&
      cudaStreamWaitEvent(us, static_cast<cudaEvent_t>(u.ss->inputs_free), 0) != cudaSuccess)
    return DAA_ERR_CUDA;
  if (cudaMemcpyAsync(u.d_inputs, u.h_inputs, u.bytes, cudaMemcpyHostToDevice, us) != cudaSuccess ||
      cudaEventRecord(uploaded, us) != cudaSuccess || cudaStreamWaitEvent(cs, uploaded, 0) != cudaSuccess)
    return DAA_ERR_CUDA;
  if (u.ss->out_free &&
      cudaStreamWaitEvent(cs, static_cast<cudaEvent_t>(u.ss->out_free), 0) != cudaSuccess)
    return DAA_ERR_CUDA;
  return DAA_OK;
}

}  // namespace

extern "C" {

daa_status daa_append_attention_host(const void* h_inputs, void* d_inputs,
                                     const daa_step_layout* layout, int32_t batch, int32_t causal,
                                     float sm_scale, void* kv_pages, void* d_out, void* h_out,
                                     void* workspace, size_t workspace_bytes, daa_dims dims,
                                     const daa_step_streams* streams) {
  if (!h_inputs || !d_inputs || !layout || !streams || !d_out || !h_out) return DAA_ERR_INVALID_ARG;
  if (!streams->uploaded || !streams->computed || !streams->downloaded) return DAA_ERR_INVALID_ARG;
  if (batch < 0) return DAA_ERR_INVALID_ARG;
  daa_status st = plan_check_dims(dims);
  if (st != DAA_OK) return st;
  const daa_step_layout& L = *layout;
  // every section inside the buffer; int32 sections 4-byte aligned, bf16 ones
  // 16-byte aligned (the device copy starts on a 256-byte boundary)
  if ((reinterpret_cast<uintptr_t>(d_inputs) & (kAlign - 1)) != 0) return DAA_ERR_ALIGNMENT;
  const size_t ints[4] = {L.qo_indptr, L.kv_indptr, L.page_indices, L.last_page_len};
  const size_t vecs[3] = {L.q, L.k_new, L.v_new};
  for (size_t o : ints)
    if (o % 4 != 0) return DAA_ERR_ALIGNMENT;
  for (size_t o : vecs)
    if (o % 16 != 0) return DAA_ERR_ALIGNMENT;
  const uint8_t* h = static_cast<const uint8_t*>(h_inputs);
  uint8_t* d = static_cast<uint8_t*>(d_inputs);
  auto fits = [&](size_t off, size_t n) { return off <= L.total && n <= L.total - off; };
  if (!fits(L.qo_indptr, 4 * ((size_t)batch + 1)) || !fits(L.kv_indptr, 4 * ((size_t)batch + 1)) ||
      !fits(L.last_page_len, 4 * (size_t)batch))
    return DAA_ERR_SHAPE;
  const int32_t* h_qo = reinterpret_cast<const int32_t*>(h + L.qo_indptr);
  const int32_t* h_kv = reinterpret_cast<const int32_t*>(h + L.kv_indptr);
  const int32_t* h_last = reinterpret_cast<const int32_t*>(h + L.last_page_len);
  if (batch > 0 && (h_qo[batch] < 0 || h_kv[batch] < 0)) return DAA_ERR_SHAPE;
  const size_t nnz_qo = batch > 0 ? (size_t)h_qo[batch] : 0;
  const size_t row_q = (size_t)dims.num_qo_heads * dims.head_dim * 2;
  const size_t row_kv = (size_t)dims.num_kv_heads * dims.head_dim * 2;
  if (!fits(L.page_indices, 4 * (size_t)(batch > 0 ? h_kv[batch] : 0)) || !fits(L.q, nnz_qo * row_q) ||
      !fits(L.k_new, nnz_qo * row_kv) || !fits(L.v_new, nnz_qo * row_kv))
    return DAA_ERR_SHAPE;
  cudaStream_t us = static_cast<cudaStream_t>(streams->upload_stream);
  cudaStream_t cs = static_cast<cudaStream_t>(streams->compute_stream);
  cudaStream_t ds = static_cast<cudaStream_t>(streams->download_stream);
  HostStepUpload up{h_inputs, d_inputs, L.total, streams};
  BeforeEnqueue before{host_step_upload, &up};
  if (nnz_qo == 0) {
    // no query rows: nothing to compute or read back; the events still mark
    // this step on their streams
    if (cudaEventRecord(static_cast<cudaEvent_t>(streams->uploaded), us) != cudaSuccess ||
        cudaEventRecord(static_cast<cudaEvent_t>(streams->computed), cs) != cudaSuccess ||
        cudaEventRecord(static_cast<cudaEvent_t>(streams->downloaded), ds) != cudaSuccess)
      return DAA_ERR_CUDA;
    return DAA_OK;
  }
  st = attention_call(d + L.k_new, d + L.v_new, d + L.q, kv_pages,
                      reinterpret_cast<const int32_t*>(d + L.qo_indptr),
                      reinterpret_cast<const int32_t*>(d + L.kv_indptr),
                      reinterpret_cast<const int32_t*>(d + L.page_indices),
                      reinterpret_cast<const int32_t*>(d + L.last_page_len), h_qo, h_kv, h_last,
                      batch, causal, sm_scale, d_out, nullptr, workspace, workspace_bytes, dims, cs,
                      /*fused=*/true, nullptr, 0, nullptr, &before);
  if (st != DAA_OK) return st;
  cudaEvent_t computed = static_cast<cudaEvent_t>(streams->computed);
  if (cudaEventRecord(computed, cs) != cudaSuccess || cudaStreamWaitEvent(ds, computed, 0) != cudaSuccess ||
      cudaMemcpyAsync(h_out, d_out, nnz_qo * row_q, cudaMemcpyDeviceToHost, ds) != cudaSuccess ||
      cudaEventRecord(static_cast<cudaEvent_t>(streams->downloaded), ds) != cudaSuccess)
    return DAA_ERR_CUDA;
  return DAA_OK;
}

daa_status daa_set_prefill_append_fusion(int32_t enable) {
  if (enable != 0 && enable != 1) return DAA_ERR_INVALID_ARG;
  g_fuse_prefill_append.store(enable, std::memory_order_relaxed);
  return DAA_OK;
}

int32_t daa_prefill_append_fusion(void) { return g_fuse_prefill_append.load(std::memory_order_relaxed); }

daa_status daa_selftest_bounded_wait(int32_t* gave_up) {
  if (!gave_up) return DAA_ERR_INVALID_ARG;
  int* err = device_error_word();
  void* flag = nullptr;
  if (!err || cudaGetSymbolAddress(&flag, g_daa_selftest_flag) != cudaSuccess) return DAA_ERR_CUDA;
  selftest_wait_kernel<<<1, 32>>>(err, static_cast<int*>(flag));
  if (cudaGetLastError() != cudaSuccess) return DAA_ERR_CUDA;
  int v = -1;
  if (cudaMemcpyFromSymbol(&v, g_daa_selftest_flag, sizeof(int)) != cudaSuccess) return DAA_ERR_CUDA;
  *gave_up = v;
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
