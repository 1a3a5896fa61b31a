// daa_batch_attention_noalloc: the mixed-batch attention call for callers that
// cannot allocate device memory (see include/daa.h for who they are).
//
// Its scratch -- the work plan and the split-KV partial outputs of the decode
// kernel -- lives in a file-scope __device__ array of fixed size instead of a
// caller-provided workspace.  Host code never uses the array's name as an
// address: on the first call on each device, with that device current, the
// device address is looked up with cudaGetSymbolAddress and cached.  The plan
// is built into fixed-size static host buffers, so the call allocates no device
// memory and no host heap memory either.  The plan and the launches are the
// library's ordinary ones (planner.h, launch_all); only where the scratch lives
// differs.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/daa.h"
#include "launch.h"
#include "planner.h"

namespace daa {
namespace {

constexpr size_t kScratchBytes = (size_t)DAA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxUnits = 16384;
constexpr int kMaxMerges = 16384;
constexpr int kMaxTiles = 16384;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_scratch[DAA_NOALLOC_SCRATCH_BYTES];

// Fixed-capacity container with the interface plan_batch expects; lives in
// static storage, never allocates.
template <class T, int N>
struct FixedVec {
  T items[N];
  int n = 0;
  bool push_back(const T& x) {
    if (n >= N) return false;
    items[n++] = x;
    return true;
  }
  size_t size() const { return (size_t)n; }
  T* data() { return items; }
  const T* data() const { return items; }
  void clear() { n = 0; }
};

std::mutex g_mu;                       // guards the static host buffers below
uint8_t* g_scratch_ptr[kMaxDevices];   // device address of g_noalloc_scratch, per device
FixedVec<DecodeUnit, kMaxUnits> g_units;
FixedVec<MergeItem, kMaxMerges> g_merges;
FixedVec<PrefillTile, kMaxTiles> g_tiles;
alignas(256) uint8_t g_staging[kMaxUnits * sizeof(DecodeUnit) + kMaxMerges * sizeof(MergeItem) +
                               kMaxTiles * sizeof(PrefillTile) + 4 * kPlanAlign];

// Per-device set-up: resolve the scratch array's device address.
daa_status scratch_for_current_device(uint8_t** out, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DAA_ERR_CUDA;
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return DAA_ERR_CUDA;
    g_scratch_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return DAA_ERR_CUDA;
  *sms = n;
  return DAA_OK;
}

}  // namespace
}  // namespace daa

using namespace daa;

extern "C" daa_status daa_batch_attention_noalloc(
    const void* q, const void* kv_pages, const int32_t* qo_indptr, const int32_t* kv_indptr,
    const int32_t* page_indices, const int32_t* last_page_len, const int32_t* h_qo_indptr,
    const int32_t* h_kv_indptr, const int32_t* h_last_page_len, int32_t batch, int32_t causal,
    float sm_scale, void* out, float* lse_out, daa_dims dims, void* stream) {
  if (!std::isfinite(sm_scale) || !(sm_scale > 0.f)) return DAA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  uint8_t* scratch = nullptr;
  int sms = 0;
  daa_status st = scratch_for_current_device(&scratch, &sms);
  if (st != DAA_OK) return st;
  PlanLayout lay;
  // the same plan as daa_batch_attention, built in the static containers
  st = plan_batch(h_qo_indptr, h_kv_indptr, h_last_page_len, batch, dims, sms, g_units, g_merges,
                  g_tiles, lay);
  if (st != DAA_OK) return st;
  if (lay.n_units == 0 && lay.n_tiles == 0) return DAA_OK;
  if (lay.total > kScratchBytes) return DAA_ERR_WORKSPACE;
  if (!q || !kv_pages || !qo_indptr || !kv_indptr || !page_indices || !last_page_len || !out)
    return DAA_ERR_INVALID_ARG;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!a16(q) || !a16(kv_pages) || !a16(out) || (reinterpret_cast<uintptr_t>(lse_out) & 3))
    return DAA_ERR_ALIGNMENT;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  plan_stage(lay, g_units, g_merges, g_tiles, g_staging);
  // the staging buffer is pageable: the copy has read it by the time this returns
  if (cudaMemcpyAsync(scratch, g_staging, lay.plan_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DAA_ERR_CUDA;
  LaunchSet ls{};
  ls.q = q;
  ls.kv_pages = kv_pages;
  ls.page_indices = page_indices;
  ls.dims = dims;
  ls.causal = causal;
  ls.sm_scale = sm_scale;
  ls.nnz_qo = h_qo_indptr[batch];
  ls.out = out;
  ls.lse_out = lse_out;
  ls.scratch = scratch;
  ls.err = device_error_word();
  ls.sms = sms;
  return launch_all(ls, lay, s, /*trace=*/false, /*after_append=*/false);
}
