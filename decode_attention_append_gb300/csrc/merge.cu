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
#include <type_traits>

#include "launch.h"
#include "ptx.cuh"

namespace daa {
namespace {

constexpr int kMergeWarps = 4;
constexpr int kMergeBatch = 4;  // partial rows loaded per batch (8 measured slower)

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) softmax_merge_kernel(const MergeArgs a) {
  constexpr int EPL = D / 32;  // elements per lane
  using Vec = typename std::conditional<EPL == 4, float4, float2>::type;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.y * kMergeWarps + warp;
  // the item comes from the plan, copied before any kernel of the call ran
  const MergeItem it = a.items[blockIdx.x];
  grid_dep_wait();  // the partials come from the kernels launched before
  if (hq >= a.Hq) return;
  const int n = it.n_parts + (it.extra >= 0 ? 1 : 0);
  auto slot = [&](int p) -> int64_t { return p < it.n_parts ? it.part_begin + p : it.extra; };

  // lane l holds part p0 + l's LSE: the running max over all parts first
  float lse_l = lane < n ? a.part_lse[slot(lane) * a.Hq + hq] : -INFINITY;
  float M = lse_l;
  for (int p = lane + 32; p < n; p += 32) M = fmaxf(M, a.part_lse[slot(p) * a.Hq + hq]);
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));

  // then, 32 parts at a time, each lane's weight, and the partial rows four
  // at a time (independent loads in flight instead of one round trip per part)
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int p0 = 0; p0 < n; p0 += 32) {
    if (p0 > 0) lse_l = p0 + lane < n ? a.part_lse[slot(p0 + lane) * a.Hq + hq] : -INFINITY;
    const float w_l = p0 + lane < n ? ex2_approx(lse_l - M) : 0.f;
    wsum += w_l;
    const int m = min(32, n - p0);
    for (int q = 0; q < m; q += kMergeBatch) {
      Vec v[kMergeBatch];
      float w[kMergeBatch];
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        w[u] = __shfl_sync(0xffffffffu, w_l, (q + u) & 31);
        if (q + u < m) {
          v[u] = *reinterpret_cast<const Vec*>(a.part_o + (slot(p0 + q + u) * a.Hq + hq) * D + lane * EPL);
        } else {
          w[u] = 0.f;
          v[u] = Vec{};
        }
      }
#pragma unroll
      for (int u = 0; u < kMergeBatch; ++u) {
        if constexpr (EPL == 4) {
          acc[0] = fmaf(w[u], v[u].x, acc[0]); acc[1] = fmaf(w[u], v[u].y, acc[1]);
          acc[2] = fmaf(w[u], v[u].z, acc[2]); acc[3] = fmaf(w[u], v[u].w, acc[3]);
        } else {
          acc[0] = fmaf(w[u], v[u].x, acc[0]); acc[1] = fmaf(w[u], v[u].y, acc[1]);
        }
      }
    }
  }
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, m);
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
