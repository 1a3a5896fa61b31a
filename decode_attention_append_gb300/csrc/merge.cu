// softmax_merge of split-KV partial attentions.
//
// "Chunked prefill" (k4i.top), #correctness: attention over a key set equals
// the online-softmax merge of attentions over a partition of it.  With parts
// (o_p normalised over its own keys, lse_p in the log2 domain):
//   M = max_p lse_p,  w_p = 2^(lse_p - M),  o = sum_p w_p o_p / sum_p w_p,
//   lse = M + log2 sum_p w_p   (reported as natural log).
// One warp per (query row, query head); lanes stride the d dimension so every
// partial row is read with coalesced 16-byte loads.  A row's parts are its
// n_parts consecutive key-split slots plus, when it follows a shared prefix
// attended once for a group of requests, the slot holding that prefix part.
#include "launch.h"
#include "ptx.cuh"

namespace daa {
namespace {

constexpr int kMergeWarps = 4;

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) softmax_merge_kernel(const MergeArgs a) {
  constexpr int EPL = D / 32;  // elements per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.y * kMergeWarps + warp;
  grid_dep_wait();  // the partials come from the decode kernel launched before
  if (hq >= a.Hq) return;
  const MergeItem it = a.items[blockIdx.x];
  const int n = it.n_parts + (it.extra >= 0 ? 1 : 0);
  auto slot = [&](int p) -> int64_t { return p < it.n_parts ? it.part_begin + p : it.extra; };

  float M = -INFINITY;
  for (int p = lane; p < n; p += 32) M = fmaxf(M, a.part_lse[slot(p) * a.Hq + hq]);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));

  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int p = 0; p < n; ++p) {
    const int64_t sl = slot(p);
    const float w = ex2_approx(a.part_lse[sl * a.Hq + hq] - M);
    wsum += w;
    const float* po = a.part_o + (sl * a.Hq + hq) * D + lane * EPL;
    if constexpr (EPL == 4) {
      const float4 v = *reinterpret_cast<const float4*>(po);
      acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
      acc[2] = fmaf(w, v.z, acc[2]); acc[3] = fmaf(w, v.w, acc[3]);
    } else {
      const float2 v = *reinterpret_cast<const float2*>(po);
      acc[0] = fmaf(w, v.x, acc[0]); acc[1] = fmaf(w, v.y, acc[1]);
    }
  }
  const float inv = 1.f / wsum;
  uint16_t* dst = a.out + ((int64_t)it.q_row * a.Hq + hq) * D + lane * EPL;
  if constexpr (EPL == 4) {
    uint2 pk;
    pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0 && a.lse_out)
    a.lse_out[(int64_t)it.q_row * a.Hq + hq] = (M + __log2f(wsum)) * 0.69314718055994531f;
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream, bool programmatic) {
  if (a.n_items <= 0) return cudaSuccess;
  const dim3 grid(a.n_items, (a.Hq + kMergeWarps - 1) / kMergeWarps), block(32 * kMergeWarps);
  return a.head_dim == 128
             ? launch_kernel(softmax_merge_kernel<128>, grid, block, 0, stream, programmatic, a)
             : launch_kernel(softmax_merge_kernel<64>, grid, block, 0, stream, programmatic, a);
}

}  // namespace daa
