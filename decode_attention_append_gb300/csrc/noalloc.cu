// daa_batch_attention_noalloc: the mixed-batch attention call for callers that
// cannot allocate device memory (see include/daa.h for who they are).
//
// Its scratch -- the work plan and the split-KV partial outputs of the decode
// kernel -- lives in a file-scope __device__ array of fixed size instead of a
// caller-provided workspace.  Host code never uses the array's name as an
// address: on the first call on each device, with that device current, the
// device address is looked up with cudaGetSymbolAddress and cached.  The plan
// is built into fixed-size static host buffers, so the call allocates no device
// memory and no host heap memory either.  The kernels are the library's
// ordinary ones; only where their scratch lives differs.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/daa.h"
#include "launch.h"

namespace daa {
namespace {

constexpr size_t kScratchBytes = (size_t)DAA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxUnits = 16384;
constexpr int kMaxMerges = 16384;
constexpr int kMaxTiles = 16384;
constexpr int kMaxDevices = 64;
constexpr int kPage = 16;
constexpr size_t kAlign = 256;

static __device__ __align__(256) uint8_t g_noalloc_scratch[DAA_NOALLOC_SCRATCH_BYTES];

std::mutex g_mu;                       // guards the static host buffers below
uint8_t* g_scratch_ptr[kMaxDevices];   // device address of g_noalloc_scratch, per device
DecodeUnit g_units[kMaxUnits];
MergeItem g_merges[kMaxMerges];
PrefillTile g_tiles[kMaxTiles];
int32_t g_tile_keys[kMaxTiles];
int32_t g_order[kMaxTiles];
alignas(256) uint8_t g_staging[kMaxUnits * sizeof(DecodeUnit) + kMaxMerges * sizeof(MergeItem) +
                               kMaxTiles * sizeof(PrefillTile) + 4 * kAlign];

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

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

daa_status check_dims(const daa_dims& d) {
  if (d.num_qo_heads <= 0 || d.num_kv_heads <= 0 || d.head_dim <= 0 || d.page_size <= 0 ||
      d.num_pages <= 0 || d.num_qo_heads % d.num_kv_heads != 0)
    return DAA_ERR_INVALID_ARG;
  if (d.head_dim != 64 && d.head_dim != 128) return DAA_ERR_UNSUPPORTED;
  if (d.page_size != kPage) return DAA_ERR_UNSUPPORTED;
  const int g = d.num_qo_heads / d.num_kv_heads;
  if (g < 1 || g > 16) return DAA_ERR_UNSUPPORTED;
  if (d.num_pages * 2 * (int64_t)d.num_kv_heads > (int64_t)INT32_MAX) return DAA_ERR_UNSUPPORTED;
  return DAA_OK;
}

struct Counts {
  int units = 0, merges = 0, tiles = 0, parts = 0;
  size_t off_units = 0, off_merges = 0, off_tiles = 0, plan_bytes = 0;
  size_t off_part_o = 0, off_part_lse = 0, total = 0;
};

// The same split of the work as daa_batch_attention (decode splits of
// max(16, min(1024, ceil(page_heads / (40 * SMs)))) pages; 128-row prefill
// tiles, paired two per CTA), written into the static buffers.  Unit and tile order do not affect
// any result.
daa_status plan_fixed(const int32_t* qo, const int32_t* kv, const int32_t* last, int32_t batch,
                      const daa_dims& d, int sms, Counts& c) {
  daa_status st = check_dims(d);
  if (st != DAA_OK) return st;
  if (batch < 0) return DAA_ERR_INVALID_ARG;
  if (batch == 0) return DAA_OK;
  if (!qo || !kv || !last) return DAA_ERR_INVALID_ARG;
  if (qo[0] != 0 || kv[0] != 0) return DAA_ERR_SHAPE;
  const int P = d.page_size;
  const int g = d.num_qo_heads / d.num_kv_heads;
  int64_t dec_pages = 0;
  for (int r = 0; r < batch; ++r) {
    const int64_t nq = (int64_t)qo[r + 1] - qo[r];
    const int64_t np = (int64_t)kv[r + 1] - kv[r];
    if (nq < 0 || np < 0) return DAA_ERR_SHAPE;
    if (np > 0 && (last[r] < 1 || last[r] > P)) return DAA_ERR_SHAPE;
    const int64_t kv_len = np > 0 ? (np - 1) * P + last[r] : 0;
    if (nq > kv_len || kv_len > INT32_MAX / 2) return DAA_ERR_SHAPE;
    if (nq == 1) dec_pages += np;
  }
  const int64_t page_heads = dec_pages * d.num_kv_heads;
  int64_t split = (page_heads + (int64_t)sms * 40 - 1) / ((int64_t)sms * 40);
  split = std::max<int64_t>(16, std::min<int64_t>(1024, split));

  for (int r = 0; r < batch; ++r) {
    if (qo[r + 1] - qo[r] != 1) continue;
    const int np = kv[r + 1] - kv[r];
    const int kv_len = (np - 1) * P + last[r];
    const int nsplit = (int)((np + split - 1) / split);
    if (c.units + nsplit > kMaxUnits) return DAA_ERR_WORKSPACE;
    int part0 = -1;
    if (nsplit > 1) {
      if (c.merges >= kMaxMerges) return DAA_ERR_WORKSPACE;
      g_merges[c.merges++] = MergeItem{qo[r], c.parts, nsplit, 0};
      part0 = c.parts;
      c.parts += nsplit;
    }
    for (int s = 0; s < nsplit; ++s) {
      DecodeUnit u{};
      u.q_row = qo[r];
      u.page_base = kv[r];
      u.tok_begin = (int)(s * split * P);
      u.tok_end = std::min<int>(kv_len, (int)((s + 1) * split * P));
      u.kv_len = kv_len;
      u.part = part0 >= 0 ? part0 + s : -1;
      g_units[c.units++] = u;
    }
  }
  std::sort(g_units, g_units + c.units, [](const DecodeUnit& x, const DecodeUnit& y) {
    return (x.tok_end - x.tok_begin) > (y.tok_end - y.tok_begin);
  });

  const int tpt = kPrefillTileRows / g;
  int nt = 0;
  for (int r = 0; r < batch; ++r) {
    const int nq = qo[r + 1] - qo[r];
    if (nq < 2) continue;
    const int np = kv[r + 1] - kv[r];
    const int kv_len = (np - 1) * P + last[r];
    for (int t0 = 0; t0 < nq; t0 += 2 * tpt) {
      if (nt >= kMaxTiles) return DAA_ERR_WORKSPACE;
      PrefillTile t{};
      t.q_row0 = qo[r];
      t.qo_len = nq;
      t.kv_len = kv_len;
      t.page_base = kv[r];
      t.tok0 = t0;
      t.ntok = std::min(tpt, nq - t0);
      t.pad0 = t.ntok == tpt ? std::max(0, std::min(tpt, nq - t0 - tpt)) : 0;  // second tile
      g_tile_keys[nt] = std::min(kv_len, kv_len - nq + t0 + t.ntok + t.pad0);
      g_order[nt] = nt;
      g_tiles[nt++] = t;
    }
  }
  std::sort(g_order, g_order + nt, [](int a, int b) {
    return g_tile_keys[a] != g_tile_keys[b] ? g_tile_keys[a] > g_tile_keys[b] : a < b;
  });
  c.tiles = nt;

  size_t off = 0;
  c.off_units = off;
  off = align_up(off + c.units * sizeof(DecodeUnit));
  c.off_merges = off;
  off = align_up(off + c.merges * sizeof(MergeItem));
  c.off_tiles = off;
  off = align_up(off + c.tiles * sizeof(PrefillTile));
  c.plan_bytes = off;
  c.off_part_o = off;
  off = align_up(off + (size_t)c.parts * d.num_qo_heads * d.head_dim * sizeof(float));
  c.off_part_lse = off;
  off = align_up(off + (size_t)c.parts * d.num_qo_heads * sizeof(float));
  c.total = off;
  if (c.total > kScratchBytes) return DAA_ERR_WORKSPACE;

  std::memcpy(g_staging + c.off_units, g_units, c.units * sizeof(DecodeUnit));
  std::memcpy(g_staging + c.off_merges, g_merges, c.merges * sizeof(MergeItem));
  PrefillTile* dst = reinterpret_cast<PrefillTile*>(g_staging + c.off_tiles);
  for (int i = 0; i < nt; ++i) dst[i] = g_tiles[g_order[i]];
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
  if (!std::isfinite(sm_scale)) return DAA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(g_mu);
  uint8_t* scratch = nullptr;
  int sms = 0;
  daa_status st = scratch_for_current_device(&scratch, &sms);
  if (st != DAA_OK) return st;
  Counts c;
  st = plan_fixed(h_qo_indptr, h_kv_indptr, h_last_page_len, batch, dims, sms, c);
  if (st != DAA_OK) return st;
  if (c.units == 0 && c.tiles == 0) return DAA_OK;
  if (!q || !kv_pages || !qo_indptr || !kv_indptr || !page_indices || !last_page_len || !out)
    return DAA_ERR_INVALID_ARG;
  auto a16 = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  if (!a16(q) || !a16(kv_pages) || !a16(out) || (reinterpret_cast<uintptr_t>(lse_out) & 3))
    return DAA_ERR_ALIGNMENT;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // the staging buffer is pageable: the copy has read it by the time this returns
  if (cudaMemcpyAsync(scratch, g_staging, c.plan_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return DAA_ERR_CUDA;
  int* err = device_error_word();
  const int g = dims.num_qo_heads / dims.num_kv_heads;
  const float sc = sm_scale * 1.4426950408889634f;
  if (c.tiles > 0) {
    PrefillArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.pool = static_cast<const uint16_t*>(kv_pages);
    a.page_indices = page_indices;
    a.tiles = reinterpret_cast<const PrefillTile*>(scratch + c.off_tiles);
    a.n_tiles = c.tiles;
    a.Hq = dims.num_qo_heads;
    a.Hkv = dims.num_kv_heads;
    a.group = g;
    a.head_dim = dims.head_dim;
    a.num_pages = dims.num_pages;
    a.nnz_qo = h_qo_indptr[batch];
    a.causal = causal ? 1 : 0;
    a.sm_scale_log2 = sc;
    a.out = static_cast<uint16_t*>(out);
    a.lse_out = lse_out;
    a.err = err;
    if (launch_prefill(a, s) != cudaSuccess) return DAA_ERR_CUDA;
  }
  if (c.units > 0) {
    DecodeArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.pool = static_cast<const uint16_t*>(kv_pages);
    a.page_indices = page_indices;
    a.units = reinterpret_cast<const DecodeUnit*>(scratch + c.off_units);
    a.n_units = c.units;
    a.Hq = dims.num_qo_heads;
    a.Hkv = dims.num_kv_heads;
    a.group = g;
    a.head_dim = dims.head_dim;
    a.num_pages = dims.num_pages;
    a.sm_scale_log2 = sc;
    a.out = static_cast<uint16_t*>(out);
    a.lse_out = lse_out;
    a.part_o = reinterpret_cast<float*>(scratch + c.off_part_o);
    a.part_lse = reinterpret_cast<float*>(scratch + c.off_part_lse);
    a.err = err;
    if (launch_decode(a, s) != cudaSuccess) return DAA_ERR_CUDA;
    if (c.merges > 0) {
      MergeArgs m{};
      m.items = reinterpret_cast<const MergeItem*>(scratch + c.off_merges);
      m.n_items = c.merges;
      m.Hq = dims.num_qo_heads;
      m.head_dim = dims.head_dim;
      m.part_o = a.part_o;
      m.part_lse = a.part_lse;
      m.out = a.out;
      m.lse_out = lse_out;
      if (launch_merge(m, s) != cudaSuccess) return DAA_ERR_CUDA;
    }
  }
  return DAA_OK;
}
