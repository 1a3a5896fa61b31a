// Host-side launchers of the CUDA kernels (one translation unit each).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/daa.h"
#include "plan.h"

namespace daa {

// Address of this library's device error word on the current device.
int* device_error_word();

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* pool,
                             const int32_t* append_indptr, const int32_t* page_indices,
                             const int32_t* kv_indptr, const int32_t* last_page_len, int batch,
                             int nnz_new, int Hkv, int head_dim, int64_t num_pages, int num_sms,
                             int* err, cudaStream_t stream);

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
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream);

struct MergeArgs {
  const MergeItem* items;       // device
  int n_items;
  int Hq, head_dim;
  const float* part_o;
  const float* part_lse;
  uint16_t* out;
  float* lse_out;
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);

struct PrefillArgs {
  const uint16_t* q;
  const uint16_t* pool;
  const int32_t* page_indices;
  const PrefillTile* tiles;     // device: prefill items
  int n_tiles;
  const PrefillTile* dec_tiles; // device: one-token (decode) items
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
  int* err;
};
// Rows of packed (token, head) a prefill tile holds.
constexpr int kPrefillTileRows = 128;
// Tensor-core kernel over the prefill items (pairs of 128-row Q tiles) and
// over the one-token decode items (a smaller instantiation, two CTAs per SM).
cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream);
cudaError_t launch_tc_decode(const PrefillArgs& a, cudaStream_t stream);

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
  void* scratch;
  int* err;
  int sms;
};
struct PlanLayout;
daa_status launch_all(const LaunchSet& ls, const PlanLayout& lay, cudaStream_t s, bool trace);

}  // namespace daa
