// Prefill-chunk attention (qo_len > 1, causal with a cache offset) on the
// sm_103a tensor cores (tcgen05 + tensor memory), warp specialised.
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
// CTA = a pair of 128-row Q tiles of one request and one kv head (the second
// tile may be absent).  Each tile packs the g query heads of the kv head
// token-major into M = 128 rows (row = token * g + head), so every K/V tile
// loaded from HBM serves 2 x 128 query rows.  Warp roles:
//   warps 0-3 / 4-7  softmax of Q tile 0 / 1 (thread = row = TMEM lane)
//   warp 8           TMA producer: Q tiles, then K_0, V_0, K_1, V_1, ... into a
//                    ring of RS shared-memory stages (one 128-key tile each)
//   warp 9           MMA issuer (one lane)
//   warp 10          page writer of the fused append (below); otherwise a second
//                    TMA producer (the odd ring items)
// Tensor memory: S_q / P_q at q*KT, O_q at 2*KT + q*D (512 columns for pairs).
//   S_q = Q_q K_j^T      A = Q (smem), B = K (smem), fp32 S in TMEM
//   P_q (bf16) overwrites the first 64 columns of S_q (softmax, tcgen05.st)
//   O_q += P_q V_j       A = P (TMEM), B = V (smem, MN-major), fp32 O in TMEM
// Per key tile the MMA warp issues PV_0(j), S_0(j+1), PV_1(j), S_1(j+1): S_q(j+1)
// follows PV_q(j) in the tensor pipe, which reads P_q(j) from the columns
// S_q(j+1) overwrites; the other tile's softmax runs meanwhile (ping-pong).
// A CTA with a single Q tile (decode splits, a request's last odd tile) instead
// double-buffers S over both S regions, so S(j+1) is ready while softmax works
// on tile j, and PV(j) is followed by S(j+2) into the buffer it just read.
// V tiles of head_dim 128 are page-major in shared memory: one TMA box per
// (page, head) slice lands as its two 64-column panels of 16 rows, and each
// PV step of 16 keys reads one page (a K tile stays column-block-major, as
// the S MMA's K-major operand needs, at two boxes per page).
// Softmax keeps a lazily raised running max (raised only when it grows by
// more than 2^8) and rescales O in TMEM only then.  V rows past the request's
// last key (stale slots, or pages not loaded) are zeroed by the producer
// before the last PV so they cannot poison it.
//
// Fused append ("Chunked prefill", #io-overhead: the chunk's new K/V go to the
// cache once; "Disaggregated prefill and decode", "KV Messenger": they are
// valid in the pages once the step's attention has run).  In a fused append +
// attention call, a prefill item's key tiles that lie wholly in its request's
// chunk -- from the first 128-aligned key at or after the cached prefix --
// are loaded straight from k_new / v_new (rows laid out like q) instead of
// from the pages, so they need not wait for the append kernel; the item that
// holds a tile's first new token also writes the tile's rows into their pages
// from shared memory (warp 10), and the append kernel skips those rows.
#include <cuda.h>

#include <algorithm>
#include <climits>

#include "launch.h"
#include "ptx.cuh"
#include "softmax_tc.cuh"

namespace daa {
namespace {

constexpr int kP = 16;
constexpr int kRows = kPrefillTileRows;  // 128 packed query rows per Q tile
// 4-D tiled TMA load through a tensor map (coordinates innermost first).
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const void* tmap, int32_t c0, int32_t c1,
                                            int32_t c2, int32_t c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(smem_dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

struct __align__(64) PrefillParams {
  CUtensorMap tmap_q;     // q viewed as [nnz_qo][Hq][d], box {64, g, 128/g}
  CUtensorMap tmap_q1;    // the same view, box {64, g, 1} (one-token decode items)
  CUtensorMap tmap_kv;    // pool viewed as [num_pages*2*Hkv][P][d], box {64, P, 1}
  CUtensorMap tmap_kn;    // k_new viewed as [nnz_qo][Hkv][d], box {64, 1, KT} (fused append)
  CUtensorMap tmap_vn;    // v_new, the same view and box
  CUtensorMap tmap_vp;    // pool as [slices][half][P][64], box {64, P, 2, 1}: one page (d = 128)
  PrefillArgs a;
  const PrefillTile* tiles;
};

// One instantiation of the kernel: head dim D, KT keys per K/V tile, at most
// NQX Q tiles per CTA, MIN_BLOCKS CTAs meant to share an SM.
//   <D, 128, 2, 1>  prefill pairs (and, for head_dim 128, short items): 224 KB
//                   of shared memory, 512 TMEM columns
//   <D,  64, 1, 2>  decode splits: ~100 KB, 256 TMEM columns, two CTAs per SM
//                   with two producer warps each (more independent TMA issue
//                   loops per SM stream K/V faster)
template <int D_, int KT_, int NQX_, int MINB_>
struct TcCfg {
  static constexpr int D = D_, KT = KT_, NQX = NQX_, MIN_BLOCKS = MINB_;
  static constexpr int PPT = KT / kP;               // pages per K/V tile
  static constexpr int KB = D / 64;                 // 64-column (128-byte) blocks per row
  // prefill instantiations (Q-tile pairs) carry the fused append's page writer
  static constexpr bool WRITES = NQX == 2;
  static constexpr int THREADS = 32 * (4 * NQX + 2 + (WRITES ? 1 : 0) + (NQX == 1 ? 1 : 0));
  // the decode instantiation's second TMA producer warp (one warp's issue loop
  // paced the page stream; two overlap their issue)
  static constexpr int PRODUCER2 = 4 * NQX + 2;
  static constexpr int PRODUCER = 4 * NQX;          // warp ids
  static constexpr int MMA = 4 * NQX + 1;
  static constexpr int WRITER = 4 * NQX + 2;        // when WRITES
  static constexpr int Q_BYTES = kRows * D * 2;
  static constexpr int T_BYTES = KT * D * 2;        // one K or V tile
  static constexpr int BUDGET = MINB_ == 1 ? 231424 : 114688;
  static constexpr int FIXED = NQX * Q_BYTES + 512 + 1024;
  static constexpr int RS_FIT = (BUDGET - FIXED) / T_BYTES;
  static constexpr int RS = RS_FIT < 12 ? RS_FIT : 12;  // ring stages
  static constexpr int OFF_Q = 0;                   // [NQX]
  static constexpr int OFF_RING = NQX * Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + RS * T_BYTES;
  // barriers: q_full, ring_full[RS], ring_empty[RS], s_full[2], p_full[2],
  // o_done[2], v_clean
  static constexpr int NBAR = 1 + 2 * RS + 6 + 1;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_TMEM + 16;
  static constexpr int ALLOC = BYTES + 1024;        // slack to align the base to 1024
  // TMEM: S / P buffers at columns 0 and KT, O_q at O_COL + q * D
  static constexpr int O_COL = 2 * KT;
  static constexpr int TMEM_COLS = 2 * KT + NQX * D <= 256 ? 256 : 512;
  static_assert(RS >= 3, "ring too shallow");
  static_assert(ALLOC <= (MINB_ == 1 ? 232448 : 115712), "shared memory budget");
};
using CfgPrefill128 = TcCfg<128, 128, 2, 1>;
using CfgPrefill64 = TcCfg<64, 128, 2, 1>;
using CfgDecode128 = TcCfg<128, 64, 1, 2>;
using CfgDecode64 = TcCfg<64, 64, 1, 2>;

__device__ __forceinline__ uint64_t desc_kmajor(uint32_t addr) {
  // K-major, 128-byte swizzle: 8-row atoms of 1024 bytes stacked along M/N.
  return smem_desc_sw128(addr, 16, 1024);
}
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t addr, uint32_t lbo) {
  // MN-major, 128-byte swizzle: 64 MN-elements x 8 K-rows per atom; LBO =
  // stride between 64-element MN blocks, SBO = stride between 8-row K groups.
  return smem_desc_sw128(addr, lbo, 1024);
}

// Ring item order.  Pairs of Q tiles (nq == 2) consume K_0, V_0, K_1, V_1, ...
// A single Q tile double-buffers S, so S runs one tile ahead of PV and the
// consumption order is K_0, K_1, V_0, K_2, V_1, ..., K_{n-1}, V_{n-2}, V_{n-1}.
__device__ __forceinline__ int ring_tile(int i, int nq, int n) {
  if (nq == 2) return i >> 1;
  if (i == 0) return 0;
  if (i & 1) {  // i = 2t + 1: K_{t+1}, or V_{n-1} for the last item
    const int t = i >> 1;
    return t + 1 < n ? t + 1 : t;
  }
  return (i >> 1) - 1;  // i = 2t + 2: V_t
}
__device__ __forceinline__ bool ring_is_v(int i, int nq, int n) {
  if (nq == 2) return i & 1;
  if (i == 0) return false;
  if (i & 1) return (i >> 1) + 1 >= n;
  return true;
}
// Ring index of K_j / V_j in the single-tile order above.
__device__ __forceinline__ int ring_k_index(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int ring_v_index(int j, int n) { return j <= n - 2 ? 2 * j + 2 : 2 * n - 1; }

template <class C, bool TREE>
__device__ __forceinline__ void tc_attention(const PrefillParams& prm) {
  using L = C;
  constexpr int D = C::D, KT = C::KT, PPT = C::PPT, RS = C::RS;
  const PrefillArgs& a = prm.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* ring_full = bars + 1;
  uint64_t* ring_empty = ring_full + RS;
  uint64_t* s_full = ring_empty + RS;  // [2]
  uint64_t* p_full = s_full + 2;       // [2]
  uint64_t* o_done = p_full + 2;       // [2]
  uint64_t* v_clean = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_TMEM);

  const PrefillTile tile = prm.tiles[blockIdx.x];
  const int kvh = blockIdx.y;
  const int g = a.group;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int nq = C::NQX == 2 && tile.ntok1 > 0 ? 2 : 1;  // Q tiles in this CTA
  const bool one_token = tile.ntok == 1 && nq == 1;

  // key tiles kt0 .. kt0 + n_kt - 1 cover keys [key_lo, kend); causal rows mask
  // beyond their own position.  A prefix-group item's keys (a cached prefix
  // shared by several requests) precede every one of its rows: no mask.
  const bool prefix_group = tile.kind == kTilePrefixGroup;
  const bool causal = a.causal && !prefix_group;
  const int pos_first = tile.kv_len - tile.qo_len + tile.tok0;
  const int ntok_all = tile.ntok + tile.ntok1;
  const int kv_end = causal ? min(tile.kv_len, pos_first + ntok_all) : tile.kv_len;
  const int kend = min(kv_end, tile.key_hi);
  const int kt0 = tile.key_lo / KT;
  const int n_kt = (kend + KT - 1) / KT - kt0;
  const int npages_req = (tile.kv_len + kP - 1) / kP;
  const bool last_partial = tile.kv_len - (kt0 + n_kt - 1) * KT < KT;
  // warps of each Q tile that hold real rows (the others skip the softmax)
  const int act0 = (tile.ntok * g + 31) / 32;
  const int act1 = (tile.ntok1 * g + 31) / 32;

  // fused append: key tiles from fuse_key on are the chunk's own keys, read
  // from k_new / v_new; this item writes into the pages each such tile whose
  // first new token (kb - first_new_key) is one of its own tokens, so every
  // new row is written once per kv head
  const int first_new_key = tile.kv_len - tile.qo_len;
  // (head_dim 64 only: head_dim-128 prefill runs on CTA pairs, and the short
  // items here stay below the fusion threshold)
  const bool fuse = C::WRITES && C::KB == 1 && a.fuse_min_qo > 0 && !prefix_group &&
                    tile.qo_len >= a.fuse_min_qo;
  const int fuse_key = fuse ? fused_from(tile.kv_len, tile.qo_len) : INT_MAX;
  auto owns = [&](int kt) {  // kt: key tile index
    const int kb = kt * KT, t = kb - first_new_key;
    return kb >= fuse_key && t >= tile.tok0 && t < tile.tok0 + ntok_all;
  };
  const int own_lo = max(fuse_key, first_new_key + tile.tok0);  // first key whose tile it may own
  const bool writer_on = fuse && (own_lo + KT - 1) / KT * KT < first_new_key + tile.tok0 + ntok_all;

  if (tid == 0) {
    prefetch_tmap(one_token ? (const void*)&prm.tmap_q1 : (const void*)&prm.tmap_q);
    prefetch_tmap(&prm.tmap_kv);
    if (fuse) {
      prefetch_tmap(&prm.tmap_kn);
      prefetch_tmap(&prm.tmap_vn);
    }
    mbar_init(q_full, 1);
    for (int i = 0; i < RS; ++i) {
      mbar_init(&ring_full[i], 1);
      // MMA completion, plus the page writer once it has copied the stage out
      mbar_init(&ring_empty[i], writer_on ? 2 : 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&s_full[q], 1);
      mbar_init(&p_full[q], q == 0 || nq == 1 ? act0 : act1);
      mbar_init(&o_done[q], 1);
    }
    mbar_init(v_clean, 1);
    fence_mbar_init();
  }
  if (warp == C::MMA) {
    tmem_alloc(tmem_slot, L::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) grid_dep_launch();  // the next kernel may start its CTAs

  // Two producers when the item has no page to write: the page writer's warp
  // issues the odd ring items, the producer warp the even ones.  One warp's
  // issue loop (a wait, an arrive and the page boxes per stage) paced the
  // stream at about 32 GB/s per SM; two overlap their issue.
  const int n_prod = C::WRITES && !writer_on ? 2 : 1;
  if (warp == C::PRODUCER || (n_prod == 2 && warp == C::WRITER)) {
    // ------------------------------------------------------------ producer
    const int pw = warp == C::PRODUCER ? 0 : 1;  // this warp issues ring items i = pw (mod n_prod)
    // Page ids of ring item i: lane l (< 8) holds the id of the item's l-th
    // page.  Fetched with one coalesced load per item, one item ahead, so its
    // latency overlaps the wait for a free stage; each lane then issues the
    // TMA boxes of its own page (issue spread over lanes runs faster than
    // from one lane; either way, 2 KB page boxes cap the per-SM load rate).
    auto load_ids = [&](int i) -> int64_t {
      if (i >= 2 * n_kt) return -1;
      const int pg0 = (kt0 + ring_tile(i, nq, n_kt)) * PPT;
      const int np = min(PPT, npages_req - pg0);
      return lane < np ? (int64_t)__ldg(a.page_indices + tile.page_base + pg0 + lane) : -1;
    };
    if (lane == 0 && pw == 0) {
      const int tpt = one_token ? 1 : kRows / g;
      const void* tmap_q = one_token ? (const void*)&prm.tmap_q1 : (const void*)&prm.tmap_q;
      mbar_arrive_expect_tx(q_full, (uint32_t)(nq * tpt * g * D * 2));
      for (int q = 0; q < nq; ++q)
        for (int b = 0; b < L::KB; ++b)
          tma_load_3d(smem + L::OFF_Q + q * L::Q_BYTES + b * (kRows * 128), tmap_q, b * 64,
                      kvh * g, tile.q_row0 + tile.tok0 + q * tile.ntok, q_full);
    }
    int64_t pid = load_ids(pw);
    // the request's last qo_len keys are the rows appended in this step: the
    // first ring item that reaches them waits for the kernel launched before
    // this one (tiles of cached keys stream while that kernel still runs).  A
    // prefix-group item reads only cached keys.
    const int first_new = prefix_group ? tile.kv_len : tile.kv_len - tile.qo_len;
    bool dep_waited = false;
    for (int i = pw; i < 2 * n_kt; i += n_prod) {
      const int64_t pid_next = load_ids(i + n_prod);
      const int st = i % RS;
      const bool is_v = ring_is_v(i, nq, n_kt);
      const int pg0 = (kt0 + ring_tile(i, nq, n_kt)) * PPT;
      uint8_t* buf = smem + L::OFF_RING + st * L::T_BYTES;
      if (pg0 * kP >= fuse_key) {
        // the chunk's own keys, from k_new / v_new (row = q_row0 + key - first
        // new key); rows past the request's end are other requests' rows or
        // zero fill, masked like stale slots
        if (lane == 0) {
          if (i >= RS) mbar_wait(&ring_empty[st], ((i / RS) - 1) & 1, a.err);
          mbar_arrive_expect_tx(&ring_full[st], (uint32_t)L::T_BYTES);
          const int row = tile.q_row0 + (pg0 * kP - first_new_key);
#pragma unroll
          for (int b = 0; b < L::KB; ++b)
            tma_load_3d(buf + b * (KT * 128), is_v ? (const void*)&prm.tmap_vn : (const void*)&prm.tmap_kn,
                        b * 64, kvh, row, &ring_full[st]);
        }
        __syncwarp();
        pid = pid_next;
        continue;
      }
      if (!dep_waited && (pg0 / PPT + 1) * KT > first_new) {
        grid_dep_wait();
        dep_waited = true;
      }
      const int np = min(PPT, npages_req - pg0);
      if (lane == 0) {
        if (i >= RS) mbar_wait(&ring_empty[st], ((i / RS) - 1) & 1, a.err);
        mbar_arrive_expect_tx(&ring_full[st], (uint32_t)(np * kP * D * 2));
      }
      __syncwarp();
      if (lane < np) {
        int64_t page = pid;
        if (page < 0 || page >= a.num_pages) {
          set_device_error(a.err, kDevErrPageRange);
          page = 0;  // fetch a valid page instead; the output is undefined anyway
        }
        const int32_t slice = (int32_t)((page * 2 + (is_v ? 1 : 0)) * a.Hkv + kvh);
        if (is_v && L::KB == 2) {  // the whole page in one box, page-major
          tma_load_4d(buf + lane * (2 * kP * 128), &prm.tmap_vp, 0, 0, 0, slice, &ring_full[st]);
        } else {
#pragma unroll
          for (int b = 0; b < L::KB; ++b)
            tma_load_3d(buf + b * (KT * 128) + lane * (kP * 128), &prm.tmap_kv, b * 64, 0, slice,
                        &ring_full[st]);
        }
      }
      pid = pid_next;
    }
    // a prefix-group item reads no appended row, and a fused item may read
    // none, but they still wait before they exit: a launch may hold nothing
    // else, and the kernels after it rely on its completion implying that of
    // the kernel before it.  (Key splits of cached rows need not: their
    // request's last split waits.)
    if ((prefix_group || fuse) && !dep_waited) grid_dep_wait();
    __syncwarp();
    if (last_partial && (2 * n_kt - 1) % n_prod == pw) {  // the last ring item's producer
      // last V tile: rows past the request's last key must hold finite values
      const int i = 2 * n_kt - 1, st = i % RS;  // V of the last tile is the last ring item
      const int tile_keys = tile.kv_len - (kt0 + n_kt - 1) * KT;
      uint8_t* buf = smem + L::OFF_RING + st * L::T_BYTES;
      mbar_wait(&ring_full[st], (i / RS) & 1, a.err);
      const int nz = (KT - tile_keys) * 8;  // 16-byte chunks per 64-column block
      for (int idx = lane; idx < nz * L::KB; idx += 32) {
        const int b = idx / nz, rem = idx - b * nz;
        const int r = tile_keys + (rem >> 3), ch = rem & 7;
        uint8_t* at = L::KB == 2 ? buf + (r >> 4) * (2 * kP * 128) + b * (kP * 128) + (r & 15) * 128
                                 : buf + b * (KT * 128) + r * 128;
        *reinterpret_cast<uint4*>(at + ch * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(v_clean);
    }
  } else if (warp == C::MMA) {
    // ----------------------------------------------------------------- MMA
    // The whole warp runs this converged; one elected lane issues each MMA and
    // commit (waits are taken by every lane, then the warp reconverges).
    constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, KT, 0, 0);
    constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, D, 0, 1);
    const uint32_t sQ = smem_u32(smem + L::OFF_Q);
    const uint32_t sR = smem_u32(smem + L::OFF_RING);
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      mbar_wait(bar, parity, a.err);
      __syncwarp();
    };
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) tc_commit(bar);
      __syncwarp();
    };
    // S = Q K^T into TMEM columns [col, col + KT): Q tile at sq, K tile in ring stage st
    auto issue_s = [&](uint32_t col, uint32_t sq, int st) {
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * (kRows * 128) + (k & 3) * 32;
        const uint32_t koff = (k >> 2) * (KT * 128) + (k & 3) * 32;
        const uint64_t da = desc_kmajor(sq + off);
        const uint64_t db = desc_kmajor(sR + st * L::T_BYTES + koff);
        if (elect_one()) tc_mma_ss(tmem + col, da, db, idesc_s, k > 0 ? 1u : 0u);
      }
      __syncwarp();
    };
    // O (columns [ocol, ocol + D)) += P (bf16 in columns [pcol, pcol + KT/2)) V (ring stage st;
    // head_dim 128: page-major, page k's two 64-column panels 2 KB apart)
    auto issue_pv = [&](uint32_t ocol, uint32_t pcol, int st, bool accumulate) {
#pragma unroll
      for (int k = 0; k < KT / 16; ++k) {
        const uint64_t db = L::KB == 2 ? desc_mnmajor(sR + st * L::T_BYTES + k * (2 * 16 * 128), 16 * 128)
                                       : desc_mnmajor(sR + st * L::T_BYTES + k * (16 * 128), KT * 128);
        if (elect_one())
          tc_mma_ts(tmem + ocol, tmem + pcol + k * 8, db, idesc_o, (accumulate || k > 0) ? 1u : 0u);
      }
      __syncwarp();
    };
    wait(q_full, 0);
    wait(&ring_full[0], 0);
    tc_fence_after();
    if (nq == 1) {
      // single Q tile: S double-buffered in TMEM columns [0, KT) and [KT, 2 KT)
      issue_s(0, sQ, 0);
      commit(&s_full[0]);
      commit(&ring_empty[0]);
      if (n_kt > 1) {
        const int ik = ring_k_index(1), sk = ik % RS;
        wait(&ring_full[sk], (ik / RS) & 1);
        tc_fence_after();
        issue_s(KT, sQ, sk);
        commit(&s_full[1]);
        commit(&ring_empty[sk]);
      }
      for (int j = 0; j < n_kt; ++j) {
        const int b = j & 1;
        const int iv = ring_v_index(j, n_kt), sv = iv % RS;
        wait(&ring_full[sv], (iv / RS) & 1);
        if (j == n_kt - 1 && last_partial) wait(v_clean, 0);
        wait(&p_full[b], (j >> 1) & 1);
        tc_fence_after();
        issue_pv(C::O_COL, b * KT, sv, j > 0);
        commit(&o_done[0]);
        commit(&ring_empty[sv]);
        if (j + 2 < n_kt) {  // S(j+2) into the buffer PV(j) just read
          const int ik = ring_k_index(j + 2), sk = ik % RS;
          wait(&ring_full[sk], (ik / RS) & 1);
          tc_fence_after();
          issue_s(b * KT, sQ, sk);
          commit(&s_full[b]);
          commit(&ring_empty[sk]);
        }
      }
    } else if constexpr (C::NQX == 2) {
      for (int q = 0; q < nq; ++q) {
        issue_s(q * KT, sQ + q * L::Q_BYTES, 0);
        commit(&s_full[q]);
      }
      commit(&ring_empty[0]);
      for (int j = 0; j < n_kt; ++j) {
        const int iv = 2 * j + 1, sv = iv % RS;
        const int ik = 2 * j + 2, sk = ik % RS;
        wait(&ring_full[sv], (iv / RS) & 1);
        if (j == n_kt - 1 && last_partial) wait(v_clean, 0);
        bool k_ready = false;
        for (int q = 0; q < nq; ++q) {
          wait(&p_full[q], j & 1);
          tc_fence_after();
          issue_pv(C::O_COL + q * D, q * KT, sv, j > 0);
          commit(&o_done[q]);
          if (j + 1 < n_kt) {
            if (!k_ready) {
              wait(&ring_full[sk], (ik / RS) & 1);
              tc_fence_after();
              k_ready = true;
            }
            issue_s(q * KT, sQ + q * L::Q_BYTES, sk);
            commit(&s_full[q]);
          }
        }
        commit(&ring_empty[sv]);
        if (j + 1 < n_kt) commit(&ring_empty[sk]);
      }
    }
  } else if (C::WRITES && warp == C::WRITER) {
    // ----------------------------------------------------- page writer
    // Fused append: write every owned K or V tile from shared memory into the
    // pages.  A page whose 16 slots are all keys of the request goes out as
    // TMA stores of the same {64, 16, 1} boxes the loads use (the TMA unit
    // undoes the 128-byte swizzle); the request's partial last page goes out
    // row by row with plain stores (16-byte chunk c of stage row R sits at
    // chunk c ^ (R % 8)), so no slot at or past kv_len is written.  The writer
    // releases every ring stage (ring_empty counts it) once its stores have
    // read the stage.
    if (writer_on) {
      for (int i = 0; i < 2 * n_kt; ++i) {
        const int st = i % RS;
        mbar_wait(&ring_full[st], (i / RS) & 1, a.err);
        const int kt = kt0 + ring_tile(i, nq, n_kt);
        if (owns(kt)) {
          const uint8_t* buf = smem + L::OFF_RING + st * L::T_BYTES;
          const bool is_v = ring_is_v(i, nq, n_kt);
          const int key0 = kt * KT;
          // lane l < PPT: page l of the tile
          int64_t page = -1;
          int keys = 0;  // keys of the request on page l
          if (lane < PPT) {
            keys = min(kP, tile.kv_len - (key0 + lane * kP));
            if (keys > 0) {
              page = __ldg(a.page_indices + tile.page_base + key0 / kP + lane);
              if (page < 0 || page >= a.num_pages) {
                set_device_error(a.err, kDevErrPageRange);
                page = -1;
              }
            }
          }
          if (page >= 0 && keys == kP) {
            const int32_t slice = (int32_t)((page * 2 + (is_v ? 1 : 0)) * a.Hkv + kvh);
#pragma unroll
            for (int b = 0; b < L::KB; ++b)
              tma_store_3d(&prm.tmap_kv, b * 64, 0, slice, buf + b * (KT * 128) + lane * (kP * 128));
            bulk_commit();
          }
          // the partial last page (at most one per tile): plain stores
          const uint32_t part_mask = __ballot_sync(0xffffffffu, page >= 0 && keys < kP);
          if (part_mask) {
            const int pl = __ffs(part_mask) - 1;
            const int pkeys = __shfl_sync(0xffffffffu, keys, pl);
            const int64_t ppage = __shfl_sync(0xffffffffu, page, pl);
            constexpr int nch = D / 8;  // 16-byte chunks per row
            uint16_t* row0 = a.pool_w + (((ppage * 2 + (is_v ? 1 : 0)) * a.Hkv + kvh) * kP) * D;
            for (int idx = lane; idx < pkeys * nch; idx += 32) {
              const int sl = idx / nch, ch = idx - sl * nch;
              const int b = ch >> 3, cc = ch & 7;
              const int R = pl * kP + sl;  // row within the stage's panels
              const uint4 v = *reinterpret_cast<const uint4*>(buf + b * (KT * 128) + R * 128 +
                                                              ((cc ^ (R & 7)) << 4));
              reinterpret_cast<uint4*>(row0 + sl * D)[ch] = v;
            }
          }
          if (page >= 0 && keys == kP) bulk_wait_read();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring_empty[st]);
      }
      bulk_wait_all();
    }
  } else if (warp / 4 < nq && (warp & 3) < ((warp >> 2) == 0 ? act0 : act1)) {
    // ------------------------------------------------------------- softmax
    const int q = warp >> 2;
    const int row = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int q_ntok = q == 0 ? tile.ntok : tile.ntok1;
    const int q_tok0 = tile.tok0 + q * tile.ntok;  // first token of this Q tile
    const int tl = row / g;
    const int qpos = tile.kv_len - tile.qo_len + q_tok0 + tl;
    const int row_end = min(causal ? min(qpos + 1, tile.kv_len) : tile.kv_len, kend);  // keys < row_end
    SoftmaxRowOut ro;
    ro.q_row = tile.q_row0 + q_tok0 + tl;
    ro.hq = kvh * g + (row - tl * g);
    ro.write = row < q_ntok * g;
    // partial slot of token t (counted from the first token of the request,
    // or of the group): part + t * part_stride
    ro.part = tile.part >= 0 ? tile.part + (q_tok0 + tl) * tile.part_stride : -1;
    TreeRow tr;
    tr.bits = TREE && ro.write && !prefix_group ? a.tree_mask + (int64_t)ro.q_row * a.mask_words
                                                : nullptr;
    tr.words = a.mask_words;
    tr.draft0 = prefix_group ? tile.kv_len : tile.kv_len - tile.qo_len;  // no draft keys
    tr.tok = prefix_group ? 0 : q_tok0 + tl;
    tc_softmax_rows<D, KT, TREE>(a, tmem + lane_off, tmem + C::O_COL + q * D + lane_off, s_full, &o_done[q],
                           q, nq == 1, n_kt, kt0, row_end, ro, tr, [&](int b) {
                             if (lane == 0) mbar_arrive(&p_full[b]);
                           });
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, L::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Persistent decode / verify kernel: the items of the decode launch (key
// splits of decode and small verify requests, one Q tile each) run on a grid
// of two CTAs per SM, each CTA taking item after item from a work counter in
// the plan's order (most keys first), so the last wave is never partly empty
// and each CTA pays its set-up (barriers, TMEM, tensor-map prefetch) once.
// Across items the pipeline does not drain: the producers stream the next
// item's K/V tiles while the MMA issuer and the softmax warps finish the
// current one.  Per CTA, ring stages, S buffers and the phases of s_full,
// p_full and o_done follow running counts of ring items and key tiles over
// all its items, exactly as within one item.  Hand-offs across items:
//   item_full / item_empty [2]  item index from the first producer to the MMA
//                               warp, the four softmax warps and the second
//                               producer (two slots)
//   q_empty      the last S of an item is done: Q may be overwritten
//   o_free       the epilogue of an item has read O: the next PV may overwrite
// The MMA warp itself zeroes the stale rows of a request's last V tile once
// it has landed, just before the PV that reads it.  (Taking the next item
// from the counter a ring's depth before the current one ends was measured
// slower: it unbalances the last items.)  Softmax
// warps that hold no real row of an item skip it; warp 0 arrives on p_full
// and o_free on their behalf.
template <class C>
struct PersistLayout {
  static constexpr int RS = C::RS;
  // barriers after C::OFF_BAR, then two item slots and the TMEM address
  static constexpr int NBAR = 2 + 2 * RS + 2 + 2 + 1 + 1 + 2 + 2 + 1;
  static constexpr int OFF_SLOT = C::OFF_BAR + NBAR * 8;  // item slots [2], S-done count
  static constexpr int OFF_ITEM = OFF_SLOT + 16;          // the two slots' descriptors
  static constexpr int OFF_TMEM = OFF_ITEM + 2 * (int)sizeof(PrefillTile);
  static constexpr int ALLOC = OFF_TMEM + 16 + 1024;
  static_assert(C::NQX == 1, "one Q tile per item");
  static_assert(ALLOC <= (C::MIN_BLOCKS == 1 ? 232448 : 115712), "shared memory budget");
};

template <class C, bool TREE>
__device__ __forceinline__ void tc_decode_persistent(const PrefillParams& prm) {
  using PL = PersistLayout<C>;
  constexpr int D = C::D, KT = C::KT, PPT = C::PPT, RS = C::RS;
  const PrefillArgs& a = prm.a;
  // work units: (item, kv head), item-major, so the heads of one item are
  // consecutive and the plan's order (most keys first) is kept
  const int n_units = a.n_dec_tiles * a.Hkv;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_empty = bars + 1;
  uint64_t* ring_full = bars + 2;         // [RS]
  uint64_t* ring_empty = ring_full + RS;  // [RS]
  uint64_t* s_full = ring_empty + RS;     // [2]
  uint64_t* p_full = s_full + 2;          // [2]
  uint64_t* o_done = p_full + 2;
  uint64_t* o_free = o_done + 1;
  uint64_t* item_full = o_free + 1;       // [2]
  uint64_t* item_empty = item_full + 2;   // [2]
  uint64_t* drained = item_empty + 2;     // the MMA warp's last MMAs have completed
  volatile int* item_slot = reinterpret_cast<volatile int*>(smem + PL::OFF_SLOT);  // [2]
  // index of the last S tile known complete (-1: none), written by the MMA warp
  volatile int* s_done_upto = item_slot + 2;
  // the descriptor of the unit in each mailbox slot, copied there by the
  // producer, so the MMA and softmax warps start a unit without a global load
  PrefillTile* item_tile = reinterpret_cast<PrefillTile*>(smem + PL::OFF_ITEM);  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + PL::OFF_TMEM);

  const int g = a.group;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    prefetch_tmap(&prm.tmap_q1);
    prefetch_tmap(&prm.tmap_q);
    prefetch_tmap(&prm.tmap_kv);
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int i = 0; i < RS; ++i) {
      mbar_init(&ring_full[i], 1);
      mbar_init(&ring_empty[i], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], 4);
      mbar_init(&item_full[b], 1);
      mbar_init(&item_empty[b], 6);  // the MMA warp, the four softmax warps, the second producer
    }
    mbar_init(o_done, 1);
    mbar_init(o_free, 4);
    mbar_init(drained, 1);
    *s_done_upto = -1;
    fence_mbar_init();
  }
  if (warp == C::MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) grid_dep_launch();

  // Item geometry shared by the roles (same formulas as the one-item kernel).
  struct Geo {
    int n_kt, kt0, kend, npages_req, act;
    bool last_partial, one_token;
  };
  auto geometry = [&](const PrefillTile& t) {
    Geo q;
    const int pos_first = t.kv_len - t.qo_len + t.tok0;
    const int kv_end = a.causal ? min(t.kv_len, pos_first + t.ntok) : t.kv_len;
    q.kend = min(kv_end, t.key_hi);
    q.kt0 = t.key_lo / KT;
    q.n_kt = (q.kend + KT - 1) / KT - q.kt0;
    q.npages_req = (t.kv_len + kP - 1) / kP;
    q.last_partial = t.kv_len - (q.kt0 + q.n_kt - 1) * KT < KT;
    q.one_token = t.ntok == 1;
    q.act = (t.ntok * g + 31) / 32;
    return q;
  };

  if (warp == C::PRODUCER || warp == C::PRODUCER2) {
    // ------------------------------------------------------------ producer
    // Two producer warps: the first takes each unit from the work counter,
    // publishes it in the mailbox and loads Q; the second reads the unit from
    // the mailbox like the consumers do.  Of each unit's ring items, the first
    // issues the even ones and the second the odd ones (K and V of a key tile
    // go to different warps), each with its own page-id pipeline.
    const int pw = warp == C::PRODUCER ? 0 : 1;
    int64_t r0 = 0;       // ring items issued before the current item
    bool dep_waited = false;
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      int unit = n_units;
      if (pw == 0) {
        if (lane == 0) {
          const bool ok = k < 2 || mbar_wait(&item_empty[slot], ((k >> 1) - 1) & 1, a.err);
          unit = ok ? atomicAdd(a.dec_counter, 1) : n_units;
          item_slot[slot] = unit;
          if (unit < n_units) item_tile[slot] = prm.tiles[unit / a.Hkv];
          mbar_arrive(&item_full[slot]);  // release: the slot's writes precede it
        }
        unit = __shfl_sync(0xffffffffu, unit, 0);
        if (unit >= n_units) break;
        __syncwarp();
      } else {
        const bool ok = mbar_wait(&item_full[slot], (k >> 1) & 1, a.err);
        unit = ok ? item_slot[slot] : n_units;
        __syncwarp();
        if (unit >= n_units) {
          if (lane == 0) mbar_arrive(&item_empty[slot]);
          break;
        }
      }
      const PrefillTile tile = item_tile[slot];
      __syncwarp();
      if (pw == 1 && lane == 0) mbar_arrive(&item_empty[slot]);  // descriptor read
      const int kvh = unit % a.Hkv;
      const Geo ge = geometry(tile);
      const int n_kt = ge.n_kt;
      auto load_ids = [&](int i) -> int64_t {
        if (i >= 2 * n_kt) return -1;
        const int pg0 = (ge.kt0 + ring_tile(i, 1, n_kt)) * PPT;
        const int np = min(PPT, ge.npages_req - pg0);
        return lane < np ? (int64_t)__ldg(a.page_indices + tile.page_base + pg0 + lane) : -1;
      };
      int64_t pid = load_ids(pw);
      if (lane == 0 && pw == 0) {
        // Q, once the previous item's last S has read it
        if (k > 0) mbar_wait(q_empty, (k - 1) & 1, a.err);
        const int tpt = ge.one_token ? 1 : kRows / g;
        const void* tmap_q = ge.one_token ? (const void*)&prm.tmap_q1 : (const void*)&prm.tmap_q;
        mbar_arrive_expect_tx(q_full, (uint32_t)(tpt * g * D * 2));
        for (int b = 0; b < C::KB; ++b)
          tma_load_3d(smem + C::OFF_Q + b * (kRows * 128), tmap_q, b * 64, kvh * g,
                      tile.q_row0 + tile.tok0, q_full);
      }
      const int first_new = tile.kv_len - tile.qo_len;
      for (int i = pw; i < 2 * n_kt; i += 2) {
        const int64_t pid_next = load_ids(i + 2);
        const int64_t rg = r0 + i;
        const int st = (int)(rg % RS);
        const uint32_t ph = (uint32_t)((rg / RS) & 1);
        const bool is_v = ring_is_v(i, 1, n_kt);
        const int pg0 = (ge.kt0 + ring_tile(i, 1, n_kt)) * PPT;
        if (!dep_waited && (pg0 / PPT + 1) * KT > first_new) {
          grid_dep_wait();
          dep_waited = true;
        }
        const int np = min(PPT, ge.npages_req - pg0);
        uint8_t* buf = smem + C::OFF_RING + st * C::T_BYTES;
        if (lane == 0) {
          if (rg >= RS) mbar_wait(&ring_empty[st], ph ^ 1u, a.err);
          mbar_arrive_expect_tx(&ring_full[st], (uint32_t)(np * kP * D * 2));
        }
        __syncwarp();
        if (lane < np) {
          int64_t page = pid;
          if (page < 0 || page >= a.num_pages) {
            set_device_error(a.err, kDevErrPageRange);
            page = 0;  // fetch a valid page instead; the output is undefined anyway
          }
          const int32_t slice = (int32_t)((page * 2 + (is_v ? 1 : 0)) * a.Hkv + kvh);
          if (is_v && C::KB == 2) {  // the whole page in one box, page-major
            tma_load_4d(buf + lane * (2 * kP * 128), &prm.tmap_vp, 0, 0, 0, slice, &ring_full[st]);
          } else {
#pragma unroll
            for (int b = 0; b < C::KB; ++b)
              tma_load_3d(buf + b * (KT * 128) + lane * (kP * 128), &prm.tmap_kv, b * 64, 0, slice,
                          &ring_full[st]);
          }
        }
        pid = pid_next;
      }
      r0 += 2 * n_kt;
    }
    // the last CTA to finish resets the work counter (dec_counter[0]) and the
    // finish count (dec_counter[1]) for the next launch on this plan: every
    // CTA has taken its last ticket before it counts itself finished
    if (pw == 0 && lane == 0 && atomicAdd(a.dec_counter + 1, 1) == (int)(gridDim.x * gridDim.y) - 1) {
      atomicExch(a.dec_counter, 0);
      atomicExch(a.dec_counter + 1, 0);
    }
  } else if (warp == C::MMA) {
    // ----------------------------------------------------------------- MMA
    constexpr uint32_t idesc_s = idesc_bf16_f32(kRows, KT, 0, 0);
    constexpr uint32_t idesc_o = idesc_bf16_f32(kRows, D, 0, 1);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sR = smem_u32(smem + C::OFF_RING);
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      const bool ok = mbar_wait(bar, parity, a.err);
      __syncwarp();
      return ok;
    };
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) tc_commit(bar);
      __syncwarp();
    };
    auto issue_s = [&](uint32_t col, int st) {
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * (kRows * 128) + (k & 3) * 32;
        const uint32_t koff = (k >> 2) * (KT * 128) + (k & 3) * 32;
        const uint64_t da = desc_kmajor(sQ + off);
        const uint64_t db = desc_kmajor(sR + st * C::T_BYTES + koff);
        if (elect_one()) tc_mma_ss(tmem + col, da, db, idesc_s, k > 0 ? 1u : 0u);
      }
      __syncwarp();
    };
    auto issue_pv = [&](uint32_t pcol, int st, bool accumulate) {
#pragma unroll
      for (int k = 0; k < KT / 16; ++k) {
        const uint64_t db = C::KB == 2 ? desc_mnmajor(sR + st * C::T_BYTES + k * (2 * 16 * 128), 16 * 128)
                                       : desc_mnmajor(sR + st * C::T_BYTES + k * (16 * 128), KT * 128);
        if (elect_one())
          tc_mma_ts(tmem + C::O_COL, tmem + pcol + k * 8, db, idesc_o, (accumulate || k > 0) ? 1u : 0u);
      }
      __syncwarp();
    };
    int64_t r0 = 0;  // ring items consumed before the current item
    int j0 = 0;      // key tiles before the current item
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      const bool ok = wait(&item_full[slot], (k >> 1) & 1);
      const int unit = ok ? item_slot[slot] : n_units;
      PrefillTile tile{};
      if (unit < n_units) tile = item_tile[slot];  // read before the slot is released
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      if (unit >= n_units) break;
      const Geo ge = geometry(tile);
      const int n_kt = ge.n_kt;
      auto stage = [&](int i) { return (int)((r0 + i) % RS); };
      auto phase = [&](int i) { return (uint32_t)(((r0 + i) / RS) & 1); };
      auto sbuf = [&](int j) { return (uint32_t)((j0 + j) & 1); };
      // S(j) into buffer (j0 + j) & 1: S of the first two tiles, then per tile
      // PV(j) and S(j + 2) into the buffer PV(j) just read
      auto s_tile = [&](int j) {
        const int ik = ring_k_index(j);
        wait(&ring_full[stage(ik)], phase(ik));
        tc_fence_after();
        issue_s(sbuf(j) * KT, stage(ik));
        commit(&s_full[sbuf(j)]);
        commit(&ring_empty[stage(ik)]);
        if (j == n_kt - 1) commit(q_empty);  // Q may be replaced
      };
      // every S tile before this item has completed (the last one issued is
      // S(j0 - 1); waiting for it is within one phase of s_full): publish that
      // for the softmax warps that join this item after skipping others
      if (j0 > 0) {
        wait(&s_full[(j0 - 1) & 1], ((j0 - 1) >> 1) & 1);
        if (lane == 0) *s_done_upto = j0 - 1;
        __syncwarp();
      }
      wait(q_full, k & 1);
      s_tile(0);
      if (n_kt > 1) s_tile(1);
      if (k > 0) wait(o_free, (k - 1) & 1);  // the previous epilogue has read O
      for (int j = 0; j < n_kt; ++j) {
        const int iv = ring_v_index(j, n_kt);
        wait(&ring_full[stage(iv)], phase(iv));
        if (j == n_kt - 1 && ge.last_partial) {
          // V rows past the request's last key (stale slots, pages not loaded)
          // must be finite for PV: zero them in shared memory
          const int keys = tile.kv_len - (ge.kt0 + n_kt - 1) * KT;
          uint8_t* buf = smem + C::OFF_RING + stage(iv) * C::T_BYTES;
          const int nz = (KT - keys) * 8;  // 16-byte chunks per 64-column block
          for (int x = lane; x < nz * C::KB; x += 32) {
            const int b = x / nz, rem = x - b * nz;
            const int r = keys + (rem >> 3), ch = rem & 7;
            uint8_t* at = C::KB == 2 ? buf + (r >> 4) * (2 * kP * 128) + b * (kP * 128) + (r & 15) * 128
                                     : buf + b * (KT * 128) + r * 128;
            *reinterpret_cast<uint4*>(at + ch * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }
        wait(&p_full[sbuf(j)], ((j0 + j) >> 1) & 1);
        tc_fence_after();
        issue_pv(sbuf(j) * KT, stage(iv), j > 0);
        commit(o_done);
        commit(&ring_empty[stage(iv)]);
        if (j + 2 < n_kt) s_tile(j + 2);
      }
      r0 += 2 * n_kt;
      j0 += n_kt;
    }
    // every MMA this warp issued has completed before the CTA frees its tensor
    // memory, whatever the softmax warps have observed
    commit(drained);
    wait(drained, 0);
  } else {
    // ------------------------------------------------------------- softmax
    const int row = tid & 127;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    int j0 = 0;
    for (int k = 0;; ++k) {
      const int slot = k & 1;
      const bool ok = mbar_wait(&item_full[slot], (k >> 1) & 1, a.err);
      const int unit = ok ? item_slot[slot] : n_units;
      PrefillTile tile{};
      if (unit < n_units) tile = item_tile[slot];  // read before the slot is released
      __syncwarp();
      if (lane == 0) mbar_arrive(&item_empty[slot]);
      if (unit >= n_units) break;
      const int kvh = unit % a.Hkv;
      const Geo ge = geometry(tile);
      // warp 0 always holds a real row; it arrives for the warps that do not
      const uint32_t cnt = warp == 0 ? (uint32_t)(5 - ge.act) : 1u;
      if (warp < ge.act) {
        // A warp other than warp 0 skips the items that hold no row of its
        // lanes, without waiting on their S tiles.  A parity wait must not run
        // two phases ahead of its barrier, so before its first S wait here it
        // waits until every S before this item is known complete (published by
        // the MMA warp; a count, which cannot alias).
        if (warp > 0) {
          const uint64_t t0 = global_timer_ns();
          while (*s_done_upto < j0 - 1) {
            if (global_timer_ns() - t0 > kWaitLimitNs ||
                *reinterpret_cast<volatile int*>(a.err) == kDevErrBarrierTimeout) {
              set_device_error(a.err, kDevErrBarrierTimeout);
              break;
            }
          }
        }
        const int tl = row / g;
        const int qpos = tile.kv_len - tile.qo_len + tile.tok0 + tl;
        const int row_end = min(a.causal ? min(qpos + 1, tile.kv_len) : tile.kv_len, ge.kend);
        SoftmaxRowOut ro;
        ro.q_row = tile.q_row0 + tile.tok0 + tl;
        ro.hq = kvh * g + (row - tl * g);
        ro.write = row < tile.ntok * g;
        ro.part = tile.part >= 0 ? tile.part + (tile.tok0 + tl) * tile.part_stride : -1;
        TreeRow tr;
        tr.bits = TREE && ro.write ? a.tree_mask + (int64_t)ro.q_row * a.mask_words : nullptr;
        tr.words = a.mask_words;
        tr.draft0 = tile.kv_len - tile.qo_len;
        tr.tok = tile.tok0 + tl;
        tc_softmax_rows<D, KT, TREE>(a, tmem + lane_off, tmem + C::O_COL + lane_off, s_full, o_done,
                                     0, true, ge.n_kt, ge.kt0, row_end, ro, tr,
                                     [&](int b) {
                                       if (lane == 0) mbar_arrive_cnt(&p_full[b], cnt);
                                     },
                                     j0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cnt(o_free, cnt);  // O of this item has been read
      }
      j0 += ge.n_kt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// One entry per role, so profilers and traces tell the two apart.
template <class C, bool TREE>
__global__ void __launch_bounds__(C::THREADS, C::MIN_BLOCKS)
prefill_tc_kernel(const __grid_constant__ PrefillParams prm) {
  tc_attention<C, TREE>(prm);
}
template <class C, bool TREE>
__global__ void __launch_bounds__(C::THREADS, C::MIN_BLOCKS)
decode_tc_kernel(const __grid_constant__ PrefillParams prm) {
  tc_decode_persistent<C, TREE>(prm);
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

template <class C, bool kDecode>
cudaError_t launch_tc(const PrefillArgs& a, const PrefillTile* tiles, int n_tiles,
                      cudaStream_t stream, bool programmatic) {
  if (n_tiles <= 0) return cudaSuccess;
  constexpr int D = C::D;
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return cudaErrorNotSupported;
  PrefillParams prm;
  prm.a = a;
  prm.tiles = tiles;
  const int g = a.group;
  const int tpt = kRows / g;
  auto encode_q = [&](CUtensorMap* m, int tokens) {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.Hq, (cuuint64_t)a.nnz_qo};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hq * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)tokens};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, (void*)a.q, dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  if (!encode_q(&prm.tmap_q, tpt) || !encode_q(&prm.tmap_q1, 1)) return cudaErrorInvalidValue;
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
  if (D == 128) {
    // one V page per box: [slices][half][P rows][64 columns] (the halves' stride
    // is 128 bytes, the rows' 256), so a page lands as two 16-row panels
    cuuint64_t dims[4] = {64, (cuuint64_t)kP, 2, (cuuint64_t)a.num_pages * 2 * a.Hkv};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, 128, (cuuint64_t)kP * D * 2};
    cuuint32_t box[4] = {64, (cuuint32_t)kP, 2, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    if (enc(&prm.tmap_vp, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, (void*)a.pool, dims, strides, box,
            es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  if (!kDecode && a.fuse_min_qo > 0) {
    // the fused call's new rows: [nnz_qo][Hkv][d], boxes of one key tile
    for (int v = 0; v < 2; ++v) {
      cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.Hkv, (cuuint64_t)a.nnz_qo};
      cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hkv * D * 2};
      cuuint32_t box[3] = {64, 1, (cuuint32_t)C::KT};
      cuuint32_t es[3] = {1, 1, 1};
      if (enc(v ? &prm.tmap_vn : &prm.tmap_kn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              (void*)(v ? a.v_new : a.k_new), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  // decode: a persistent grid of MIN_BLOCKS CTAs per SM (over all kv heads),
  // each taking items from the work counter; otherwise one CTA per item
  int alloc = C::ALLOC;
  dim3 grid(n_tiles, a.Hkv);
  if constexpr (kDecode) {
    alloc = PersistLayout<C>::ALLOC;
    const int64_t units = (int64_t)n_tiles * a.Hkv;
    const int slots = C::MIN_BLOCKS * (a.sms > 0 ? a.sms : 1);
    grid = dim3((unsigned)std::min<int64_t>(units, slots), 1);
  }
  auto go = [&](void (*kern)(PrefillParams)) -> cudaError_t {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, alloc);
    if (e != cudaSuccess) return e;
    return launch_kernel(kern, grid, dim3(C::THREADS), alloc, stream, programmatic, prm);
  };
  // the draft-tree variant only when the call carries a mask
  if constexpr (kDecode)
    return a.tree_mask ? go(decode_tc_kernel<C, true>) : go(decode_tc_kernel<C, false>);
  else
    return a.tree_mask ? go(prefill_tc_kernel<C, true>) : go(prefill_tc_kernel<C, false>);
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const PrefillTile* tiles, int n_tiles,
                           cudaStream_t stream, bool pr) {
  return a.head_dim == 128 ? launch_tc<CfgPrefill128, false>(a, tiles, n_tiles, stream, pr)
                           : launch_tc<CfgPrefill64, false>(a, tiles, n_tiles, stream, pr);
}

cudaError_t launch_tc_decode(const PrefillArgs& a, cudaStream_t stream, bool pr) {
  return a.head_dim == 128 ? launch_tc<CfgDecode128, true>(a, a.dec_tiles, a.n_dec_tiles, stream, pr)
                           : launch_tc<CfgDecode64, true>(a, a.dec_tiles, a.n_dec_tiles, stream, pr);
}

}  // namespace daa
