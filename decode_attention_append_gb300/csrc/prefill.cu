// Prefill-chunk attention (qo_len > 1, causal with a cache offset) on the
// sm_103a tensor cores (tcgen05 + tensor memory).
//
// "Chunked prefill" (k4i.top), #correctness: new token i of a chunk sits at
// absolute position kv_len - qo_len + i and attends to every key j <= that
// position: the cached prefix (all of it) plus the causal part of its own
// chunk; both parts flow through one online softmax here.  #flops: the work
// is 4 d per (query, key) pair, a dense contraction, hence the tensor cores.
// "Disaggregated prefill and decode", "Sharded KV cache transfers": pages are
// HND, so one (page, head) K or V slice is a contiguous [page_size][d] block,
// which a 3-D tensor map over the pool fetches as one TMA box per 64 columns.
//
// CTA = one PrefillTile x one kv head, 128 threads.  The tile packs the g query
// heads of the kv head token-major into M = 128 rows (row = token * g + head),
// so every K/V tile loaded from HBM serves all g query heads (GQA packing).
// Per 128-key tile kt:
//   S = Q K^T          tcgen05.mma M=128 N=128 K=16 x (d/16), S in TMEM
//   P = exp2(S*scale - m) per row (thread = row = TMEM lane), P bf16 -> smem
//   O += P V           tcgen05.mma M=128 N=d K=16 x 8, O in TMEM
// The running max is raised lazily (only when it grows by more than 2^8), and
// O is rescaled in TMEM only then.  Thread 0 issues TMA and MMAs; K/V tiles
// are double buffered so the next tile's pages stream in during this tile.
#include <cuda.h>

#include "launch.h"
#include "ptx.cuh"

namespace daa {
namespace {

constexpr int kP = 16;
constexpr int kRows = kPrefillTileRows;  // 128
constexpr int kKeys = 128;               // keys per K/V tile (8 pages)
constexpr int kPagesPerTile = kKeys / kP;
constexpr int kThreads = 128;
constexpr float kRescaleThreshold = 8.0f;  // log2 domain

struct __align__(64) PrefillParams {
  CUtensorMap tmap_q;     // q viewed as [nnz_qo][Hq][d], box {64, g, 128/g}
  CUtensorMap tmap_kv;    // pool viewed as [num_pages*2*Hkv][P][d], box {64, P, 1}
  PrefillArgs a;
};

template <int D>
struct PrefillSmem {
  static constexpr int KB = D / 64;                 // 64-column (128-byte) blocks per row
  static constexpr int Q_BYTES = kRows * D * 2;     // 128 rows
  static constexpr int T_BYTES = kKeys * D * 2;     // one K or V tile
  static constexpr int P_BYTES = kRows * kKeys * 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K0 = OFF_Q + Q_BYTES;
  static constexpr int OFF_V0 = OFF_K0 + T_BYTES;
  static constexpr int OFF_K1 = OFF_V0 + T_BYTES;
  static constexpr int OFF_V1 = OFF_K1 + T_BYTES;
  static constexpr int OFF_P = OFF_V1 + T_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int NBAR = 8;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_TMEM + 16;
  static constexpr int ALLOC = BYTES + 1024;        // slack to align the base to 1024
  static constexpr int TMEM_COLS = 256;             // S: [0,128)  O: [128, 128+D)
};

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr) {
  // K-major, 128-byte swizzle: 8-row atoms of 1024 bytes stacked along M/N.
  return smem_desc_sw128(addr, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t addr, uint32_t lbo) {
  // MN-major, 128-byte swizzle: 64 MN-elements x 8 K-rows per atom; LBO =
  // stride between 64-element MN blocks, SBO = stride between 8-row K groups.
  return smem_desc_sw128(addr, lbo, 1024);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ PrefillParams prm) {
  using L = PrefillSmem<D>;
  const PrefillArgs& a = prm.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_bar = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_bar = bars + 5;
  uint64_t* o_bar = bars + 6;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);

  const PrefillTile tile = a.tiles[blockIdx.x];
  const int kvh = blockIdx.y;
  const int g = a.group;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int rows_valid = tile.ntok * g;

  // key range this tile needs
  const int pos_first = tile.kv_len - tile.qo_len + tile.tok0;
  const int pos_last = pos_first + tile.ntok - 1;
  const int kv_end = a.causal ? min(tile.kv_len, pos_last + 1) : tile.kv_len;
  const int n_kt = (kv_end + kKeys - 1) / kKeys;
  const int npages_req = (tile.kv_len + kP - 1) / kP;

  if (tid == 0) {
    prefetch_tmap(&prm.tmap_q);
    prefetch_tmap(&prm.tmap_kv);
    mbar_init(q_bar, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    mbar_init(s_bar, 1);
    mbar_init(o_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, L::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;
  const uint32_t tmem_o = tmem + 128;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  const uint32_t sQ = smem_u32(smem + L::OFF_Q);
  const uint32_t sK[2] = {smem_u32(smem + L::OFF_K0), smem_u32(smem + L::OFF_K1)};
  const uint32_t sV[2] = {smem_u32(smem + L::OFF_V0), smem_u32(smem + L::OFF_V1)};
  const uint32_t sP = smem_u32(smem + L::OFF_P);
  uint8_t* kbuf[2] = {smem + L::OFF_K0, smem + L::OFF_K1};
  uint8_t* vbuf[2] = {smem + L::OFF_V0, smem + L::OFF_V1};

  // ---- producer helpers (thread 0 only)
  auto load_kv = [&](int kt, int st) {
    const int pg0 = kt * kPagesPerTile;
    int np = npages_req - pg0;
    np = np > kPagesPerTile ? kPagesPerTile : np;
    mbar_arrive_expect_tx(&kv_full[st], (uint32_t)(np * 2 * kP * D * 2));
    for (int i = 0; i < np; ++i) {
      int64_t page = a.page_indices[tile.page_base + pg0 + i];
      if (page < 0 || page >= a.num_pages) {
        set_device_error(a.err, kDevErrPageRange);
        page = 0;  // fetch a valid page instead; the output is undefined anyway
      }
      const int32_t kslice = (int32_t)((page * 2 + 0) * a.Hkv + kvh);
      const int32_t vslice = (int32_t)((page * 2 + 1) * a.Hkv + kvh);
#pragma unroll
      for (int b = 0; b < L::KB; ++b) {
        tma_load_3d(kbuf[st] + b * (kKeys * 128) + i * (kP * 128), &prm.tmap_kv, b * 64, 0, kslice,
                    &kv_full[st]);
        tma_load_3d(vbuf[st] + b * (kKeys * 128) + i * (kP * 128), &prm.tmap_kv, b * 64, 0, vslice,
                    &kv_full[st]);
      }
    }
  };
  auto issue_s = [&](int st) {
    constexpr uint32_t idesc = idesc_bf16_f32(kRows, kKeys, 0, 0);
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k >> 2) * (kRows * 128) + (k & 3) * 32;
      const uint32_t koff = (k >> 2) * (kKeys * 128) + (k & 3) * 32;
      tc_mma_ss(tmem_s, desc_kmajor(sQ + off), desc_kmajor(sK[st] + koff), idesc, k > 0 ? 1u : 0u);
    }
    tc_commit(s_bar);
  };
  auto issue_pv = [&](int st, int kt) {
    constexpr uint32_t idesc = idesc_bf16_f32(kRows, D, 0, 1);
#pragma unroll
    for (int k = 0; k < kKeys / 16; ++k) {
      const uint32_t poff = (k >> 2) * (kRows * 128) + (k & 3) * 32;
      const uint32_t voff = k * (16 * 128);
      tc_mma_ss(tmem_o, desc_kmajor(sP + poff), desc_mnmajor(sV[st] + voff, kKeys * 128), idesc,
                (kt > 0 || k > 0) ? 1u : 0u);
    }
    tc_commit(o_bar);
    tc_commit(&kv_empty[st]);
  };

  if (tid == 0) {
    const int d_blocks = L::KB;
    mbar_arrive_expect_tx(q_bar, (uint32_t)(rows_valid > 0 ? (kRows / g) * g * D * 2 : 0));
    for (int b = 0; b < d_blocks; ++b)
      tma_load_3d(smem + L::OFF_Q + b * (kRows * 128), &prm.tmap_q, b * 64, kvh * g,
                  tile.q_row0 + tile.tok0, q_bar);
    load_kv(0, 0);
    if (n_kt > 1) load_kv(1, 1);
    mbar_wait(q_bar, 0, a.err);
    mbar_wait(&kv_full[0], 0, a.err);
    tc_fence_after();
    issue_s(0);
  }

  // ---- per-row softmax state (thread = row)
  const int row = tid;
  const int tl = row / g;
  const bool row_ok = row < rows_valid;
  const int qpos = pos_first + tl;  // absolute position of this row's token
  const int row_end = a.causal ? min(qpos + 1, tile.kv_len) : tile.kv_len;  // keys j < row_end
  float m_run = -INFINITY, l_run = 0.f;
  const float sc = a.sm_scale_log2;

  for (int kt = 0; kt < n_kt; ++kt) {
    const int st = kt & 1;
    mbar_wait(s_bar, kt & 1, a.err);
    tc_fence_after();

    // scores of this row for keys kt*128 .. +128
    float s[kKeys];
#pragma unroll
    for (int c = 0; c < kKeys; c += 32) {
      uint32_t r[32];
      tmem_ld32(tmem_s + lane_off + c, r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) s[c + i] = __uint_as_float(r[i]);
    }
    const int key0 = kt * kKeys;
    const int lim = row_end - key0;  // keys [key0, key0 + lim) are valid
    float mt = -INFINITY;
#pragma unroll
    for (int c = 0; c < kKeys; ++c) {
      s[c] = (c < lim) ? s[c] * sc : -INFINITY;
      mt = fmaxf(mt, s[c]);
    }
    float m_use = m_run;
    float alpha = 1.f;
    if (mt > m_run + kRescaleThreshold) {
      m_use = mt;
      alpha = ex2_approx(m_run - mt);  // 0 on the first tile
    }
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < kKeys; ++c) {
      s[c] = ex2_approx(s[c] - m_use);
      sum += s[c];
    }
    l_run = l_run * alpha + sum;
    m_run = m_use;
    const bool warp_rescale = __any_sync(0xffffffffu, alpha != 1.f) && kt > 0;

    // PV of the previous tile must be done before P (smem) and O (TMEM) change
    if (kt > 0) {
      mbar_wait(o_bar, (kt - 1) & 1, a.err);
      tc_fence_after();
    }
    if (warp_rescale) {
#pragma unroll
      for (int c = 0; c < D; c += 32) {
        uint32_t r[32];
        tmem_ld32(tmem_o + lane_off + c, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
        tmem_st32(tmem_o + lane_off + c, r);
      }
      tmem_wait_st();
    }
    // P row -> smem, K-major 128-byte swizzle: 16-byte chunk ch of row `row`
    // in 64-key block b lives at b*16K + row*128 + ((ch ^ (row & 7)) * 16)
#pragma unroll
    for (int cc = 0; cc < kKeys / 8; ++cc) {
      uint4 v;
      v.x = pack_bf16x2(s[cc * 8 + 0], s[cc * 8 + 1]);
      v.y = pack_bf16x2(s[cc * 8 + 2], s[cc * 8 + 3]);
      v.z = pack_bf16x2(s[cc * 8 + 4], s[cc * 8 + 5]);
      v.w = pack_bf16x2(s[cc * 8 + 6], s[cc * 8 + 7]);
      const int b = cc >> 3, ch = cc & 7;
      uint8_t* dst = smem + L::OFF_P + b * (kRows * 128) + row * 128 + ((ch ^ (row & 7)) << 4);
      *reinterpret_cast<uint4*>(dst) = v;
    }
    // keys past the request's last token (stale slots, or pages not loaded)
    // must hold finite values in V: zero those rows of the last tile
    const int tile_keys = tile.kv_len - key0;
    if (tile_keys < kKeys) {
      mbar_wait(&kv_full[st], (kt >> 1) & 1, a.err);
      if (row >= tile_keys) {
#pragma unroll
        for (int b = 0; b < L::KB; ++b) {
          uint4* dst = reinterpret_cast<uint4*>(vbuf[st] + b * (kKeys * 128) + row * 128);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) dst[ch] = make_uint4(0, 0, 0, 0);
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    if (tid == 0) {
      tc_fence_after();
      issue_pv(st, kt);
      if (kt + 1 < n_kt) {
        mbar_wait(&kv_full[st ^ 1], ((kt + 1) >> 1) & 1, a.err);
        issue_s(st ^ 1);
      }
      if (kt + 2 < n_kt) {
        mbar_wait(&kv_empty[st], (kt >> 1) & 1, a.err);
        load_kv(kt + 2, st);
      }
    }
  }

  // ---- epilogue: O / l -> bf16 rows of out; lse
  mbar_wait(o_bar, (n_kt - 1) & 1, a.err);
  tc_fence_after();
  const float inv = 1.f / l_run;
  const int hg = row - tl * g;
  const int q_row = tile.q_row0 + tile.tok0 + tl;
  const int hq = kvh * g + hg;
  const bool write = row_ok && (tile.tok0 + tl) < tile.qo_len;
  uint16_t* dst = a.out + ((int64_t)q_row * a.Hq + hq) * D;
#pragma unroll
  for (int c = 0; c < D; c += 32) {
    uint32_t r[32];
    tmem_ld32(tmem_o + lane_off + c, r);
    tmem_wait_ld();
    if (write) {
#pragma unroll
      for (int i = 0; i < 32; i += 8) {
        uint4 v;
        v.x = pack_bf16x2(__uint_as_float(r[i + 0]) * inv, __uint_as_float(r[i + 1]) * inv);
        v.y = pack_bf16x2(__uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv);
        v.z = pack_bf16x2(__uint_as_float(r[i + 4]) * inv, __uint_as_float(r[i + 5]) * inv);
        v.w = pack_bf16x2(__uint_as_float(r[i + 6]) * inv, __uint_as_float(r[i + 7]) * inv);
        *reinterpret_cast<uint4*>(dst + c + i) = v;
      }
    }
  }
  if (write && a.lse_out)
    a.lse_out[(int64_t)q_row * a.Hq + hq] = (m_run + __log2f(l_run)) * 0.69314718055994531f;

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_relinquish();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// --------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &p, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

template <int D>
cudaError_t launch_prefill_d(const PrefillArgs& a, cudaStream_t stream) {
  using L = PrefillSmem<D>;
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return cudaErrorNotSupported;
  PrefillParams prm;
  prm.a = a;
  const int g = a.group;
  const int tpt = kRows / g;
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.Hq, (cuuint64_t)a.nnz_qo};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hq * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)tpt};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&prm.tmap_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)a.q, dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)kP, (cuuint64_t)a.num_pages * 2 * a.Hkv};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)kP * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kP, 1};
    cuuint32_t es[3] = {1, 1, 1};
    if (enc(&prm.tmap_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)a.pool, dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kern = prefill_tc_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_tiles, a.Hkv);
  kern<<<grid, kThreads, L::ALLOC, stream>>>(prm);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (a.n_tiles <= 0) return cudaSuccess;
  return a.head_dim == 128 ? launch_prefill_d<128>(a, stream) : launch_prefill_d<64>(a, stream);
}

}  // namespace daa
