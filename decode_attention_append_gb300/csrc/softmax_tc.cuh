// Softmax warps of the tensor-core attention kernels: one thread per packed
// query row (its TMEM lane), a warpgroup per 128-row Q tile.
//
// "Chunked prefill" (k4i.top), #correctness: token i of a chunk attends to the
// keys j <= its absolute position, cached prefix and chunk alike, through one
// online softmax.  Per key tile the thread loads its row of S from TMEM, masks
// keys at or past row_end, raises a lazily kept running max (only when it
// grows by more than 2^8, so O is rescaled in TMEM rarely), writes
// P = 2^(s * scale - m) as bf16 over the first KT/2 columns of S (the A
// operand of PV), and hands P to the MMA issuer through release_p.  The
// epilogue divides O by the running sum and writes bf16 rows (or, for a key
// split, fp32 partial rows in the log2 domain for softmax_merge).
#pragma once
#include "launch.h"
#include "ptx.cuh"

namespace daa {

constexpr float kRescaleThreshold = 8.0f;  // log2 domain

// Per-row output target of the epilogue.
struct SoftmaxRowOut {
  int q_row;     // token row of q / out / lse_out
  int hq;        // query head
  bool write;    // the row holds a real (token, head)
  int part;      // partial slot (key split) or -1
};

// Draft-tree mask of one row ("Accelerating Sonar through speculation", EAGLE:
// a tree of draft tokens is verified under a custom attention mask).  The
// request's new tokens sit at keys draft0 + t; this row's token `tok` sees all
// cached keys, itself, and each earlier new token t < tok whose bit t is set in
// `bits` (word t / 32, bit t % 32).  bits == nullptr: no mask.
struct TreeRow {
  const uint32_t* bits;
  int words;
  int draft0;
  int tok;
};

// Keys key0 .. key0 + 31 that the row's mask hides (bit b = key key0 + b):
// earlier new tokens whose mask bit is clear.  Cached keys, the row's own key
// and later keys are never hidden here (later keys fall past row_end).
__device__ __forceinline__ uint32_t tree_hidden_word(const TreeRow& tr, int key0) {
  const int rel0 = key0 - tr.draft0;  // new-token index of bit 0
  const int lo_b = max(0, -rel0);                 // first bit inside [0, tok)
  const int hi_b = min(32, tr.tok - rel0);        // one past the last
  if (tr.bits == nullptr || hi_b <= lo_b) return 0u;
  uint32_t m;
  if (rel0 >= 0) {
    const int q = rel0 >> 5;
    const uint32_t w0 = q < tr.words ? __ldg(tr.bits + q) : 0u;
    const uint32_t w1 = q + 1 < tr.words ? __ldg(tr.bits + q + 1) : 0u;
    m = __funnelshift_r(w0, w1, rel0 & 31);
  } else {
    m = __ldg(tr.bits) << lo_b;  // lo_b = -rel0 in 1 .. 31
  }
  const uint32_t hi_mask = hi_b >= 32 ? 0xffffffffu : ((1u << hi_b) - 1u);
  const uint32_t inwin = hi_mask & ~((1u << lo_b) - 1u);
  return inwin & ~m;
}

// TREE: the kernel variant for draft-tree masks (tr describes the row's mask);
// the plain variant carries no mask code at all.
// tmem_s0: TMEM address (lane field = this warp's 32 lanes) of S buffer 0; S
// buffer b sits at tmem_s0 + b * KT.  tmem_o: this warp's lanes of O.
// dbuf: S alternates between buffers 0 and 1 per key tile (single Q tile);
// otherwise buffer `sbuf` is used for every tile.
// j0: key tiles this CTA's MMA issuer processed before this item (a persistent
// CTA runs item after item; the S buffers and the phases of s_full and o_done
// continue across items).  0 for a CTA that runs one item.
template <int D, int KT, bool TREE, class ReleaseP>
__device__ __forceinline__ void tc_softmax_rows(const PrefillArgs& a, uint32_t tmem_s0,
                                                uint32_t tmem_o, uint64_t* s_full,
                                                uint64_t* o_done_q, int sbuf, bool dbuf,
                                                int n_kt, int kt0, int row_end,
                                                const SoftmaxRowOut& ro, const TreeRow& tr,
                                                ReleaseP&& release_p, int j0 = 0) {
  const float sc = a.sm_scale_log2;
  float m_run = -INFINITY, l_run = 0.f;

  for (int j = 0; j < n_kt; ++j) {
    const int b = dbuf ? ((j0 + j) & 1) : sbuf;
    const uint32_t ph = dbuf ? (((j0 + j) >> 1) & 1) : (j & 1);
    const uint32_t tmem_s = tmem_s0 + b * KT;
    mbar_wait(&s_full[b], ph, a.err);
    tc_fence_after();
    float s[KT];
#pragma unroll
    for (int c = 0; c < KT; c += 32) tmem_ld32f(tmem_s + c, s + c);
    tmem_wait_ld();
    const int kb = (kt0 + j) * KT;
    const int lim = row_end - kb;  // keys [kb, kb + lim) are valid
    // tree mask: only tiles that hold an earlier new token of some row
    if (TREE && __any_sync(0xffffffffu, kb + KT > tr.draft0 && kb < tr.draft0 + tr.tok)) {
#pragma unroll
      for (int k = 0; k < KT / 32; ++k) {
        const uint32_t hid = tree_hidden_word(tr, kb + 32 * k);
#pragma unroll
        for (int b = 0; b < 32; ++b) s[32 * k + b] = ((hid >> b) & 1u) ? -INFINITY : s[32 * k + b];
      }
    }
    if (!__all_sync(0xffffffffu, lim >= KT)) {
#pragma unroll
      for (int c = 0; c < KT; ++c) s[c] = (c < lim) ? s[c] : -INFINITY;
    }
    // row max of the raw scores (sm_scale > 0, so it commutes with scaling),
    // as independent chains over 32 columns each
    float mx[KT / 32];
#pragma unroll
    for (int k = 0; k < KT / 32; ++k) {
      mx[k] = s[32 * k];
#pragma unroll
      for (int i2 = 1; i2 < 31; i2 += 2) mx[k] = fmax3(mx[k], s[32 * k + i2], s[32 * k + i2 + 1]);
      mx[k] = fmaxf(mx[k], s[32 * k + 31]);
    }
    float mt = mx[0];
#pragma unroll
    for (int k = 1; k < KT / 32; ++k) mt = fmaxf(mt, mx[k]);
    mt *= sc;
    float m_use = m_run;
    float alpha = 1.f;
    if (mt > m_run + kRescaleThreshold) {
      m_use = mt;
      alpha = ex2_approx(m_run - mt);  // 0 on the first tile
    }
    // P = 2^(s * scale - m) as bf16 pairs over the first KT/2 columns of S
    // (the A operand of PV), 32 columns at a time so each chunk of s dies early
    // a row with no visible key yet (possible in a key split) keeps m = -inf:
    // subtract 0 instead so its masked scores give p = 0, not NaN
    const float m_sub = m_use == -INFINITY ? 0.f : m_use;
    const float2 sc2 = make_float2(sc, sc);
    const float2 nm2 = make_float2(-m_sub, -m_sub);
    float2 sum2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < KT / 2; c += 32) {
      uint32_t r[32];
#pragma unroll
      for (int i2 = 0; i2 < 32; ++i2) {
        const float2 t = __ffma2_rn(make_float2(s[2 * (c + i2)], s[2 * (c + i2) + 1]), sc2, nm2);
        const float2 pp = make_float2(ex2_approx(t.x), ex2_approx(t.y));
        sum2 = __fadd2_rn(sum2, pp);
        r[i2] = pack_bf16x2(pp.x, pp.y);
      }
      tmem_st32(tmem_s + c, r);
    }
    const float sum = sum2.x + sum2.y;
    l_run = l_run * alpha + sum;
    m_run = m_use;
    const bool warp_rescale = __any_sync(0xffffffffu, alpha != 1.f) && j > 0;

    // O (TMEM) is rescaled once PV of the previous tile is done with it
    if (warp_rescale) {
      mbar_wait(o_done_q, (j0 + j - 1) & 1, a.err);
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D; c += 64) {  // two 32-column loads in flight per wait
        float o[64];
        tmem_ld32f(tmem_o + c, o);
        tmem_ld32f(tmem_o + c + 32, o + 32);
        tmem_wait_ld();
        uint32_t r[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int i2 = 0; i2 < 32; ++i2) r[i2] = __float_as_uint(o[32 * h + i2] * alpha);
          tmem_st32(tmem_o + c + 32 * h, r);
        }
      }
    }
    // o_done must never run two phases ahead of this thread's parity waits:
    // with S double-buffered, S(j) done only implies PV(j-2) done, so consume
    // the phase of PV(j-1) before PV(j) can be issued (normally no wait).
    if (j > 0 && !warp_rescale) mbar_wait(o_done_q, (j0 + j - 1) & 1, a.err);
    tmem_wait_st();
    tc_fence_before();
    __syncwarp();
    release_p(b);
  }

  // ---- epilogue: O / l -> bf16 rows of out; lse
  mbar_wait(o_done_q, (j0 + n_kt - 1) & 1, a.err);
  tc_fence_after();
  const float inv = l_run > 0.f ? 1.f / l_run : 0.f;  // no visible key: o = 0, lse = -inf
  const bool partial = ro.part >= 0;  // key split: fp32 partial for softmax_merge
  uint16_t* dst = a.out + ((int64_t)ro.q_row * a.Hq + ro.hq) * D;
  float* pdst = a.part_o + ((int64_t)ro.part * a.Hq + ro.hq) * D;
#pragma unroll
  for (int c = 0; c < D; c += 64) {  // two 32-column loads in flight per wait
    float o[64];
    tmem_ld32f(tmem_o + c, o);
    tmem_ld32f(tmem_o + c + 32, o + 32);
    tmem_wait_ld();
    if (ro.write && partial) {
#pragma unroll
      for (int i2 = 0; i2 < 64; i2 += 4)
        *reinterpret_cast<float4*>(pdst + c + i2) =
            make_float4(o[i2] * inv, o[i2 + 1] * inv, o[i2 + 2] * inv, o[i2 + 3] * inv);
    } else if (ro.write) {
#pragma unroll
      for (int i2 = 0; i2 < 64; i2 += 8) {
        uint4 v;
        v.x = pack_bf16x2(o[i2 + 0] * inv, o[i2 + 1] * inv);
        v.y = pack_bf16x2(o[i2 + 2] * inv, o[i2 + 3] * inv);
        v.z = pack_bf16x2(o[i2 + 4] * inv, o[i2 + 5] * inv);
        v.w = pack_bf16x2(o[i2 + 6] * inv, o[i2 + 7] * inv);
        *reinterpret_cast<uint4*>(dst + c + i2) = v;
      }
    }
  }
  if (ro.write) {
    const float lse2 = m_run + __log2f(l_run);
    if (partial)
      a.part_lse[(int64_t)ro.part * a.Hq + ro.hq] = lse2;
    else if (a.lse_out)
      a.lse_out[(int64_t)ro.q_row * a.Hq + ro.hq] = lse2 * 0.69314718055994531f;
  }
}

}  // namespace daa
