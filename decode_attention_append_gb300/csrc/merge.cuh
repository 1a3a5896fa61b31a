// softmax_merge of one (query row, query head) by one warp, shared by the
// merge kernel and by the persistent decode kernel (whose last unit of a row
// merges it in place).
//
// "Chunked prefill" (k4i.top), #correctness: attention over a key set equals
// the online-softmax merge of attentions over a partition of it.  With parts
// (o_p normalised over its own keys, lse_p in the log2 domain):
//   M = max_p lse_p,  w_p = 2^(lse_p - M),  o = sum_p w_p o_p / sum_p w_p,
//   lse = M + log2 sum_p w_p   (reported as natural log).
// A row's parts are its n_parts consecutive key-split slots plus, when it
// follows a shared prefix attended once for a group of requests, the slot
// holding that prefix part.  Lanes stride the d dimension (16-byte loads);
// partials are read through L2 (.cg): other CTAs wrote them.
#pragma once
#include <type_traits>

#include "launch.h"
#include "ptx.cuh"

namespace daa {

constexpr int kMergeBatch = 4;  // partial rows loaded per batch (8 measured slower)

template <int D>
__device__ __forceinline__ void merge_row_head(const MergeItem& it, int Hq, int hq,
                                               const float* __restrict__ part_o,
                                               const float* __restrict__ part_lse,
                                               uint16_t* __restrict__ out, float* lse_out,
                                               int lane) {
  constexpr int EPL = D / 32;  // elements per lane
  using Vec = typename std::conditional<EPL == 4, float4, float2>::type;
  const int n = it.n_parts + (it.extra >= 0 ? 1 : 0);
  auto slot = [&](int p) -> int64_t { return p < it.n_parts ? it.part_begin + p : it.extra; };

  // lane l holds part p0 + l's LSE: the running max over all parts first
  float lse_l = lane < n ? __ldcg(part_lse + slot(lane) * Hq + hq) : -INFINITY;
  float M = lse_l;
  for (int p = lane + 32; p < n; p += 32) M = fmaxf(M, __ldcg(part_lse + slot(p) * Hq + hq));
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, m));

  // then, 32 parts at a time, each lane's weight, and the partial rows four
  // at a time (independent loads in flight instead of one round trip per part)
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float wsum = 0.f;
  for (int p0 = 0; p0 < n; p0 += 32) {
    if (p0 > 0) lse_l = p0 + lane < n ? __ldcg(part_lse + slot(p0 + lane) * Hq + hq) : -INFINITY;
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
          v[u] = __ldcg(reinterpret_cast<const Vec*>(part_o + (slot(p0 + q + u) * Hq + hq) * D + lane * EPL));
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
  uint16_t* dst = out + ((int64_t)it.q_row * Hq + hq) * D + lane * EPL;
  if constexpr (EPL == 4) {
    uint2 pk;
    pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<uint32_t*>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
  if (lane == 0 && lse_out)
    lse_out[(int64_t)it.q_row * Hq + hq] = (M + __log2f(wsum)) * 0.69314718055994531f;
}

}  // namespace daa
