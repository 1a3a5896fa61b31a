// Host-side launchers of the CUDA kernels (one translation unit each).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/daa.h"
#include "plan.h"

namespace daa {

// Address of this library's device error word on the current device.
int* device_error_word();

// Launch `kern` on `s`; with `programmatic`, as a programmatic dependent launch
// (its CTAs may start while the previous kernel on the stream is still running
// and must call grid_dep_wait before reading what that kernel writes).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, bool programmatic, Args... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = programmatic ? attr : nullptr;
  cfg.numAttrs = programmatic ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Key tiles are 128 keys; with the prefill append fused (fuse_min_qo > 0), a
// request with qo_len >= fuse_min_qo has its new tokens at positions
// >= fused_from(kv_len, qo_len) written by the prefill kernel, not the append.
constexpr int kFuseTileKeys = 128;
__host__ __device__ inline int fused_from(int kv_len, int qo_len) {
  const int c = kv_len - qo_len;
  return (c + kFuseTileKeys - 1) / kFuseTileKeys * kFuseTileKeys;
}

// Appends rows [row_begin, row_begin + n_rows) of k_new / v_new (all rows:
// 0, nnz_new).  fuse_min_qo: 0 appends every row of that span; otherwise rows
// that the prefill kernel writes itself (see fused_from) are skipped.
cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* pool,
                             const int32_t* append_indptr, const int32_t* page_indices,
                             const int32_t* kv_indptr, const int32_t* last_page_len, int batch,
                             int row_begin, int n_rows, int Hkv, int head_dim, int64_t num_pages,
                             int num_sms, int fuse_min_qo, int* err, cudaStream_t stream);

// The span of rows the append kernel of a fused call must cover: every row
// except those the prefill kernels write (a request's new tokens from
// fused_from on when qo_len >= fuse_min_qo).  Host side, from the host copies
// of the lengths; begin == end when there is none.
struct AppendSpan {
  int begin, end;
};
AppendSpan append_span(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                       const int32_t* h_last_page_len, int batch, int page_size, int fuse_min_qo);

struct DecodeArgs {
  const uint16_t* q;            // [nnz_qo][Hq][d]
  const uint16_t* pool;         // [num_pages][2][Hkv][P][d]
  const int32_t* page_indices;
  const DecodeUnit* units;      // device
  int n_units;
  int Hq, Hkv, group;           // group = Hq / Hkv
  int head_dim;
  int64_t num_pages;
  float sm_scale_log2;          // sm_scale * log2(e)
  uint16_t* out;                // [nnz_qo][Hq][d]
  float* lse_out;               // [nnz_qo][Hq] natural log, or null
  float* part_o;                // [n_parts][Hq][d]
  float* part_lse;              // [n_parts][Hq] (log2 domain)
  int* err;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream, bool programmatic);

struct MergeArgs {
  const MergeItem* items;       // device
  int n_items;
  int Hq, head_dim;
  const float* part_o;
  const float* part_lse;
  uint16_t* out;
  float* lse_out;
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream, bool programmatic);

struct PrefillArgs {
  const uint16_t* q;
  const uint16_t* pool;
  const int32_t* page_indices;
  const PrefillTile* tiles;     // device: prefill items
  int n_tiles;
  const PrefillTile* short_tiles;  // device: short multi-token items (single-CTA kernel)
  int n_short_tiles;
  const PrefillTile* dec_tiles; // device: decode and verify items
  int n_dec_tiles;
  int Hq, Hkv, group, head_dim;
  int64_t num_pages;
  int nnz_qo;
  int causal;
  float sm_scale_log2;
  uint16_t* out;
  float* lse_out;
  float* part_o;                // split items: [n_parts][Hq][d]
  float* part_lse;              // split items: [n_parts][Hq] (log2 domain)
  const uint32_t* tree_mask;    // draft-tree mask rows [nnz_qo][mask_words], or null
  int mask_words;
  int* err;
  int* dec_counter;             // persistent decode kernel: [0] work counter, [1] CTAs
                                // finished; zero before a launch, reset to zero by it
  int sms;                      // SMs of the device (persistent grid size)
  // Prefill append fused into the prefill kernels (the fused call
  // only; fuse_min_qo == 0 otherwise).  For a prefill item of a request with
  // qo_len >= fuse_min_qo, key tiles from fused_from(kv_len, qo_len) on are
  // read from k_new / v_new (rows laid out like q) instead of the pool, and the
  // item that holds a tile's first new token writes the tile's rows into their
  // pages (pool_w).
  const uint16_t* k_new;        // [nnz_qo][Hkv][d]
  const uint16_t* v_new;
  uint16_t* pool_w;
  int fuse_min_qo;
};
// Rows of packed (token, head) a prefill tile holds.
constexpr int kPrefillTileRows = 128;
// Single-CTA tensor-core kernel over `tiles` (pairs of 128-row Q tiles: the
// prefill items for head_dim 64, the short items for head_dim 128), and the
// decode instantiation over the decode / verify items (one Q tile, two CTAs
// per SM).
cudaError_t launch_prefill(const PrefillArgs& a, const PrefillTile* tiles, int n_tiles,
                           cudaStream_t stream, bool programmatic);
// head_dim 128: prefill items of four Q tiles on clusters of two CTAs
// (tcgen05 cta_group::2); grid (2 * n_tiles, Hkv).
cudaError_t launch_prefill_pair(const PrefillArgs& a, cudaStream_t stream, bool programmatic);
cudaError_t launch_tc_decode(const PrefillArgs& a, cudaStream_t stream, bool programmatic);

// Everything one batch_attention call launches, given its plan in `scratch`
// (the workspace, or the no-allocation entry point's static array).
struct LaunchSet {
  const void* q;
  const void* kv_pages;
  const int32_t* page_indices;
  daa_dims dims;
  int causal;
  float sm_scale;
  int nnz_qo;
  void* out;
  float* lse_out;
  const uint32_t* tree_mask;    // draft-tree mask rows, or null
  int mask_words;
  void* scratch;
  int* err;
  int sms;
  // the fused call's new rows and the fusion threshold (see PrefillArgs)
  const void* k_new;
  const void* v_new;
  int fuse_min_qo;
};
struct PlanLayout;
// The kernels run in the order prefill, decode, softmax_merge; each after the
// first is a programmatic dependent launch, and so is the first when
// `after_append` (this call's own kv_append kernel precedes it on the stream).
// Ordering contract, kept by the kernels:
//  * every CTA that reads rows the append wrote (all prefill CTAs, the last
//    key split of each decode request) calls grid_dep_wait first; so does
//    every softmax_merge CTA.  The completion of a kernel therefore implies the
//    completion of the kernel before it, and the last kernel's completion (what
//    later stream work waits for) implies that of the whole chain;
//  * the other decode splits read only cached rows and overlap the kernel
//    before them.
daa_status launch_all(const LaunchSet& ls, const PlanLayout& lay, cudaStream_t s, bool trace,
                      bool after_append);

}  // namespace daa
