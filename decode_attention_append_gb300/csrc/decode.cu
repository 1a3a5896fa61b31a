// Split-KV decode attention (qo_len == 1) over HND pages, on CUDA cores.
//
// "Disaggregated prefill and decode" (Perplexity), "Prefill vs decode
// performance": decode attention is memory bound and can be split over
// requests and over kv_len.  "Chunked prefill" (k4i.top), #correctness: the
// partial attentions over disjoint key ranges are combined by softmax_merge
// (the merge kernel), so each CTA handles one page-aligned key range (a split)
// of one request for one kv head.
//
// CTA organisation (G = query heads per kv head):
//   - a "page group" of NWH warps shares one ring of NSTAGE shared-memory
//     stages; each stage holds one page's K slice and V slice for this kv head
//     (2 x page_size x d bf16, contiguous in HND), filled by two 1-D TMA bulk
//     copies issued by one lane and tracked by an mbarrier;
//   - the NWH warps of a group split the G query heads (HPW per warp), so one
//     page read from HBM serves every query head of its group (GQA packing);
//   - NPG page groups per CTA take pages round-robin and keep separate
//     online-softmax states, merged in shared memory at the end.
// Inside a warp, 16 lanes cover one token's d-vector (8 dims each for d=128)
// and the two half-warps take alternate tokens.  q.k partial sums are reduced
// across the 16 lanes with a reduce-scatter of warp shuffles (each level halves
// the values a lane holds); it leaves every lane owning whole scores of one
// token for HPW/2 heads, so the online-softmax update (max, exp2, sum) runs in
// all lanes at once with 4-level shuffle reductions over the page's tokens.
// Scores live in the log2 domain (q is pre-scaled by sm_scale * log2 e).  The
// FMAs are packed two-wide (sm_100 FFMA2).
#include <cfloat>

#include "launch.h"
#include "ptx.cuh"

namespace daa {
namespace {

constexpr int kP = 16;

template <int D, int G>
struct DecodeShape {
  static constexpr int HPW = G >= 16 ? 8 : (G >= 12 ? 6 : (G >= 4 ? 4 : G));  // heads per warp
  static constexpr int NWH = (G + HPW - 1) / HPW;     // warps sharing a page
  static constexpr int NPG = NWH >= 4 ? 1 : 4 / NWH;  // page groups per CTA
  static constexpr int NWARPS = NWH * NPG;
  static constexpr int THREADS = 32 * NWARPS;
  static constexpr int DPL = D / 16;                  // dims per lane
  static constexpr int DP2 = DPL / 2;                 // float2 pairs per lane
  static constexpr int ITERS = kP / 2;                // two tokens per warp step
  static constexpr int SLICE = kP * D * 2;            // bytes of one head's K (or V) page slice
  static constexpr int STAGE = 2 * SLICE;
  static constexpr int NSTAGE = NPG >= 4 ? 3 : (NPG == 2 ? 4 : (NWH >= 2 ? 5 : 6));
  static constexpr int RING = NPG * NSTAGE * STAGE;
  static constexpr int NRED = ITERS * HPW;            // partial dots per lane per page
  static constexpr int NF = HPW >= 2 ? HPW / 2 : 1;   // scores a lane owns after the reduce
  static_assert(HPW == 1 || HPW % 2 == 0, "heads per warp");
  static constexpr int MERGE_BYTES = NPG * G * (D + 2) * 4;
  static constexpr int BODY = RING > MERGE_BYTES ? RING : MERGE_BYTES;
  static constexpr int BARS = 2 * NPG * NSTAGE * 8;
  static constexpr int SCORES = NWARPS * kP * HPW * 4;
  static constexpr int ALPHA = NWARPS * HPW * 4;
  static constexpr int SMEM = BODY + BARS + SCORES + ALPHA;
};

// Reduce-scatter over the 16 lanes of a half-warp: on entry every lane holds N
// partial sums; on exit lane li holds the full sums of entries
// [li * N/16, li * N/16 + N/16) (N >= 16), or of entry li >> 1 (N == 8).
template <int N, int M>
__device__ __forceinline__ void reduce_scatter16(float* v, int li) {
  if constexpr (M > 0) {
    if constexpr (N >= 2) {
      constexpr int H = N / 2;
      const bool upper = (li & M) != 0;
#pragma unroll
      for (int i = 0; i < H; ++i) {
        const float a = v[i], b = v[H + i];
        const float send = upper ? a : b;
        const float keep = upper ? b : a;
        v[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
      }
      reduce_scatter16<H, M / 2>(v, li);
    } else {
      v[0] += __shfl_xor_sync(0xffffffffu, v[0], M);
      reduce_scatter16<1, M / 2>(v, li);
    }
  }
}

// One row slice of DPL bf16 values -> DPL/2 float2 pairs (exact widening).
template <int DPL>
__device__ __forceinline__ void load_row_f2(const uint8_t* p, float2 (&f)[DPL / 2]) {
  if constexpr (DPL == 8) {
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    f[0] = make_float2(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x));
    f[1] = make_float2(bf16lo_to_f32(w.y), bf16hi_to_f32(w.y));
    f[2] = make_float2(bf16lo_to_f32(w.z), bf16hi_to_f32(w.z));
    f[3] = make_float2(bf16lo_to_f32(w.w), bf16hi_to_f32(w.w));
  } else {
    const uint2 w = *reinterpret_cast<const uint2*>(p);
    f[0] = make_float2(bf16lo_to_f32(w.x), bf16hi_to_f32(w.x));
    f[1] = make_float2(bf16lo_to_f32(w.y), bf16hi_to_f32(w.y));
  }
}

__device__ __forceinline__ uint16_t f32_to_bf16_rn(float x) {
  return static_cast<uint16_t>(pack_bf16x2(x, 0.f) & 0xFFFFu);
}

template <int D, int G>
__global__ void __launch_bounds__(DecodeShape<D, G>::THREADS)
decode_splitkv_kernel(const DecodeArgs a) {
  using S = DecodeShape<D, G>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::BODY);
  uint64_t* empty = full + S::NPG * S::NSTAGE;
  float* s_scores = reinterpret_cast<float*>(empty + S::NPG * S::NSTAGE);
  float* s_alpha = s_scores + S::NWARPS * kP * S::HPW;

  const DecodeUnit u = a.units[blockIdx.x];
  const int kvh = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / S::NWH;
  const int wh = warp - grp * S::NWH;
  const int hb = wh * S::HPW;  // first head (within the group of G) of this warp
  const int half = lane >> 4, li = lane & 15;

  const int pg_lo = u.tok_begin / kP;
  const int pg_hi = (u.tok_end + kP - 1) / kP;
  const int npg_unit = pg_hi - pg_lo;
  const int my_n = npg_unit > grp ? (npg_unit - grp + S::NPG - 1) / S::NPG : 0;

  if (threadIdx.x == 0) {
    grid_dep_launch();  // the merge pass may launch; it waits for this grid
    for (int i = 0; i < S::NPG * S::NSTAGE; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], S::NWH);
    }
    fence_mbar_init();
  }
  __syncthreads();

  uint64_t* gfull = full + grp * S::NSTAGE;
  uint64_t* gempty = empty + grp * S::NSTAGE;
  uint8_t* gring = ring + grp * S::NSTAGE * S::STAGE;
  const bool producer = (wh == 0 && lane == 0);

  // page id of the group's k-th page (the producer loads the next one a page
  // ahead, so the global-load latency is off the refill path)
  auto page_id = [&](int k) -> int64_t {
    return k < my_n ? (int64_t)__ldg(a.page_indices + u.page_base + pg_lo + grp + k * S::NPG) : -1;
  };
  auto issue = [&](int k, int64_t page) {
    const int stage = k % S::NSTAGE;
    if (page < 0 || page >= a.num_pages) {
      set_device_error(a.err, kDevErrPageRange);
      mbar_arrive(&gfull[stage]);  // completes the phase with no bytes; data is stale
      return;
    }
    uint8_t* dst = gring + stage * S::STAGE;
    mbar_arrive_expect_tx(&gfull[stage], 2 * S::SLICE);
    const uint16_t* kp = a.pool + ((page * 2 + 0) * a.Hkv + kvh) * (int64_t)(kP * D);
    const uint16_t* vp = a.pool + ((page * 2 + 1) * a.Hkv + kvh) * (int64_t)(kP * D);
    bulk_g2s(dst, kp, S::SLICE, &gfull[stage]);
    bulk_g2s(dst + S::SLICE, vp, S::SLICE, &gfull[stage]);
  };

  int64_t next_page = -1;  // producer: id of page k + NSTAGE
  if (producer) {
    const int n0 = my_n < S::NSTAGE ? my_n : S::NSTAGE;
    int64_t ids[S::NSTAGE];
#pragma unroll
    for (int k = 0; k < S::NSTAGE; ++k) ids[k] = page_id(k);
    // only the split holding the request's last page reads a row appended in
    // this step: it alone waits for the kernel launched before this one
    if (u.tok_end >= u.kv_len) grid_dep_wait();
    for (int k = 0; k < n0; ++k) issue(k, ids[k]);
    next_page = page_id(S::NSTAGE);
  }

  // q rows of this warp's heads, scaled into the log2 domain
  float2 q2[S::HPW][S::DP2];
#pragma unroll
  for (int j = 0; j < S::HPW; ++j) {
    const int hg = hb + j;
    if (hg < a.group) {
      const int hq = kvh * a.group + hg;
      const uint8_t* qp = reinterpret_cast<const uint8_t*>(
          a.q + ((int64_t)u.q_row * a.Hq + hq) * D + li * S::DPL);
      float2 f[S::DP2];
      load_row_f2<S::DPL>(qp, f);
#pragma unroll
      for (int c = 0; c < S::DP2; ++c)
        q2[j][c] = make_float2(f[c].x * a.sm_scale_log2, f[c].y * a.sm_scale_log2);
    } else {
#pragma unroll
      for (int c = 0; c < S::DP2; ++c) q2[j][c] = make_float2(0.f, 0.f);
    }
  }

  float2 o2[S::HPW][S::DP2];
#pragma unroll
  for (int j = 0; j < S::HPW; ++j)
#pragma unroll
    for (int c = 0; c < S::DP2; ++c) o2[j][c] = make_float2(0.f, 0.f);

  // online-softmax state of the NF heads this lane owns after the reduce:
  // token t_own of each page, heads hj(f) = (li & 1) * NF + f (head 0 if HPW == 1)
  float m_run[S::NF], l_run[S::NF];
#pragma unroll
  for (int f = 0; f < S::NF; ++f) {
    m_run[f] = -INFINITY;
    l_run[f] = 0.f;
  }
  const int t_own = 2 * (li >> 1) + half;
  const int hj0 = S::HPW == 1 ? 0 : (li & 1) * S::NF;
  const bool writer = S::HPW > 1 || (li & 1) == 0;

  float* sw = s_scores + warp * kP * S::HPW;
  float* aw = s_alpha + warp * S::HPW;

  for (int k = 0; k < my_n; ++k) {
    const int stage = k % S::NSTAGE;
    const uint32_t parity = (k / S::NSTAGE) & 1;
    mbar_wait(&gfull[stage], parity, a.err);
    const uint8_t* kbuf = gring + stage * S::STAGE;
    const uint8_t* vbuf = kbuf + S::SLICE;
    const int tok0 = (pg_lo + grp + k * S::NPG) * kP;
    const int valid = min(kP, u.tok_end - tok0);

    // ---- scores s[t][j] = q_j . k_t (log2 domain)
    float part[S::NRED];
#pragma unroll
    for (int it = 0; it < S::ITERS; ++it) {
      const int t = 2 * it + half;
      float2 kf[S::DP2];
      load_row_f2<S::DPL>(kbuf + (t * D + li * S::DPL) * 2, kf);
#pragma unroll
      for (int j = 0; j < S::HPW; ++j) {
        float2 acc = __fmul2_rn(q2[j][0], kf[0]);
#pragma unroll
        for (int c = 1; c < S::DP2; ++c) acc = __ffma2_rn(q2[j][c], kf[c], acc);
        part[it * S::HPW + j] = acc.x + acc.y;
      }
    }
    reduce_scatter16<S::NRED, 8>(part, li);

    // ---- online softmax over this page's tokens, all lanes at once
    const bool tok_ok = t_own < valid;
    float p[S::NF], alpha[S::NF];
#pragma unroll
    for (int f = 0; f < S::NF; ++f) {
      const float s = tok_ok ? part[f] : -INFINITY;
      float mx = s;
#pragma unroll
      for (int msk = 2; msk <= 16; msk <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, msk));
      const float m_new = fmaxf(m_run[f], mx);
      alpha[f] = ex2_approx(m_run[f] - m_new);
      p[f] = ex2_approx(s - m_new);
      float sum = p[f];
#pragma unroll
      for (int msk = 2; msk <= 16; msk <<= 1) sum += __shfl_xor_sync(0xffffffffu, sum, msk);
      l_run[f] = l_run[f] * alpha[f] + sum;
      m_run[f] = m_new;
    }
    if (writer) {
#pragma unroll
      for (int f = 0; f < S::NF; ++f) sw[t_own * S::HPW + hj0 + f] = p[f];
      if (half == 0 && li < 2) {
#pragma unroll
        for (int f = 0; f < S::NF; ++f) aw[hj0 + f] = alpha[f];
      }
    }
    __syncwarp();

    // ---- o = alpha * o + sum_t p_t v_t
#pragma unroll
    for (int j = 0; j < S::HPW; ++j) {
      const float al = aw[j];
      const float2 al2 = make_float2(al, al);
#pragma unroll
      for (int c = 0; c < S::DP2; ++c) o2[j][c] = __fmul2_rn(o2[j][c], al2);
    }
#pragma unroll
    for (int it = 0; it < S::ITERS; ++it) {
      const int t = 2 * it + half;
      if (t < valid) {
        float2 vf[S::DP2];
        load_row_f2<S::DPL>(vbuf + (t * D + li * S::DPL) * 2, vf);
#pragma unroll
        for (int j = 0; j < S::HPW; ++j) {
          const float pj = sw[t * S::HPW + j];
          const float2 p2 = make_float2(pj, pj);
#pragma unroll
          for (int c = 0; c < S::DP2; ++c) o2[j][c] = __ffma2_rn(p2, vf[c], o2[j][c]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&gempty[stage]);
    if (producer && k + S::NSTAGE < my_n) {
      mbar_wait(&gempty[stage], parity, a.err);
      issue(k + S::NSTAGE, next_page);
      next_page = page_id(k + S::NSTAGE + 1);
    }
  }

  // ---- combine the two half-warps (same running max), then the page groups
#pragma unroll
  for (int j = 0; j < S::HPW; ++j)
#pragma unroll
    for (int c = 0; c < S::DP2; ++c) {
      o2[j][c].x += __shfl_xor_sync(0xffffffffu, o2[j][c].x, 16);
      o2[j][c].y += __shfl_xor_sync(0xffffffffu, o2[j][c].y, 16);
    }

  __syncthreads();  // ring is free: reuse it for the merge
  float* mo = reinterpret_cast<float*>(ring);   // [NPG][G][D]
  float* mm = mo + S::NPG * G * D;              // [NPG][G]
  float* ml = mm + S::NPG * G;                  // [NPG][G]
  if (half == 0) {
#pragma unroll
    for (int j = 0; j < S::HPW; ++j) {
      const int hg = hb + j;
      if (hg < G) {
#pragma unroll
        for (int c = 0; c < S::DP2; ++c) {
          mo[(grp * G + hg) * D + li * S::DPL + 2 * c] = o2[j][c].x;
          mo[(grp * G + hg) * D + li * S::DPL + 2 * c + 1] = o2[j][c].y;
        }
      }
    }
    if (li < 2 && writer) {
#pragma unroll
      for (int f = 0; f < S::NF; ++f) {
        const int hg = hb + hj0 + f;
        if (hg < G) {
          mm[grp * G + hg] = m_run[f];
          ml[grp * G + hg] = l_run[f];
        }
      }
    }
  }
  __syncthreads();

  const int group = a.group;
  for (int i = threadIdx.x; i < group * D; i += S::THREADS) {
    const int hg = i / D, c = i - hg * D;
    float M = -INFINITY;
#pragma unroll
    for (int g = 0; g < S::NPG; ++g) M = fmaxf(M, mm[g * G + hg]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int g = 0; g < S::NPG; ++g) {
      const float w = ex2_approx(mm[g * G + hg] - M);
      L += w * ml[g * G + hg];
      O += w * mo[(g * G + hg) * D + c];
    }
    const float inv = 1.f / L;
    const int hq = kvh * group + hg;
    const float lse2 = M + __log2f(L);
    if (u.part < 0) {
      a.out[((int64_t)u.q_row * a.Hq + hq) * D + c] = f32_to_bf16_rn(O * inv);
      if (c == 0 && a.lse_out) a.lse_out[(int64_t)u.q_row * a.Hq + hq] = lse2 * 0.69314718055994531f;
    } else {
      a.part_o[((int64_t)u.part * a.Hq + hq) * D + c] = O * inv;
      if (c == 0) a.part_lse[(int64_t)u.part * a.Hq + hq] = lse2;
    }
  }
}

template <int D, int G>
cudaError_t launch_decode_t(const DecodeArgs& a, cudaStream_t stream, bool programmatic) {
  using S = DecodeShape<D, G>;
  auto kern = decode_splitkv_kernel<D, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(a.n_units, a.Hkv), dim3(S::THREADS), S::SMEM, stream,
                       programmatic, a);
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t stream, bool pr) {
  const int g = a.group;
  if (g <= 1) return launch_decode_t<D, 1>(a, stream, pr);
  if (g <= 2) return launch_decode_t<D, 2>(a, stream, pr);
  if (g <= 4) return launch_decode_t<D, 4>(a, stream, pr);
  if (g <= 8) return launch_decode_t<D, 8>(a, stream, pr);
  if (g <= 12) return launch_decode_t<D, 12>(a, stream, pr);
  return launch_decode_t<D, 16>(a, stream, pr);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t stream, bool programmatic) {
  if (a.n_units <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_decode_d<128>(a, stream, programmatic)
                           : launch_decode_d<64>(a, stream, programmatic);
}

}  // namespace daa
