// Prefill-chunk attention (qo_len > 1) on pairs of SMs: tcgen05 with
// cta_group::2, head_dim 128.
//
// "Chunked prefill" (k4i.top), #correctness / #flops: the same computation as
// the single-CTA tensor-core kernel (one online softmax over the cached prefix
// and the causal part of the chunk).  What changes is how K/V reach the tensor
// cores.  With 16-token pages a K or V tile is assembled from 2 KB TMA boxes
// (one per page and 64-column half), and one SM takes in such boxes at about
// 20 bytes per clock -- below the ~30 bytes per clock two 128-row Q tiles need
// at the tensor-core rate.  A cluster of two CTAs issues each MMA once for
// M = 256 rows (128 in each CTA) and splits the B operand between them, so each
// SM loads only half of every K tile (64 keys) and half of every V tile (64 of
// the 128 columns): half the boxes and bytes per SM for the same work.
//
// Cluster = (CTA 0, CTA 1), one work item = up to four 128-row Q tiles of one
// request and kv head; CTA r holds tiles r and 2 + r (local tiles 0 and 1), so
// the M = 256 MMA of local tile q covers the adjacent tiles 2q and 2q + 1.
// Per CTA the warp roles are those of the single-CTA kernel:
//   warps 0-3 / 4-7  softmax of local Q tile 0 / 1 (thread = row = TMEM lane)
//   warp 8           TMA producer of this CTA's halves: Q tiles, then K_0, V_0,
//                    K_1, V_1, ... into a ring of RS half-tile stages (16 KB)
//   warp 9           CTA 0: MMA issuer for the pair; CTA 1: relays "my half of
//                    stage s has landed" to CTA 0 (remote mbarrier arrive)
//   warp 10          page writer of the fused append (below); idle otherwise
//
// Fused append ("Chunked prefill", #io-overhead: the chunk's new K/V are
// written to the cache once; "Disaggregated prefill and decode", "KV
// Messenger": they are valid in the pages once the step's attention has run).
// In a fused append + attention call, key tiles of a request that lie wholly
// in its chunk -- from the first 128-aligned key at or after the cached prefix
// -- are loaded straight from k_new / v_new (rows laid out like q) instead of
// from the pages, so they need not wait for the append kernel, and the item
// holding a tile's first new token also writes the tile's rows into their
// pages from shared memory (warp 10); the append kernel skips those rows.  The
// tile that holds both cached and new keys (when the prefix is not a multiple
// of 128 keys) is still read from the pages after the append.
// Tensor memory per CTA: S_q / P_q at q*128, O_q at 256 + q*128 (512 columns).
// Completion of the pair's MMAs is committed to the barriers of both CTAs
// (multicast); both CTAs' softmax warps hand P to CTA 0's issuer by arriving on
// its p_full barrier.  Every tcgen05 instruction of this kernel uses
// cta_group::2, as the instruction set requires within one kernel.
#include <cuda.h>

#include <climits>

#include "launch.h"
#include "ptx.cuh"
#include "softmax_tc.cuh"

namespace daa {
namespace {

constexpr int kP = 16;
constexpr int kRows = kPrefillTileRows;

struct __align__(64) PairParams {
  CUtensorMap tmap_q;   // q viewed as [nnz_qo][Hq][d], box {64, g, 128/g}
  CUtensorMap tmap_kv;  // pool viewed as [num_pages*2*Hkv][P][d], box {64, P, 1}
  CUtensorMap tmap_kn;  // k_new viewed as [nnz_qo][Hkv][d], box {64, 1, 64} (fused append)
  CUtensorMap tmap_vn;  // v_new, the same view, box {64, 1, 128}
  PrefillArgs a;
  const PrefillTile* tiles;
};

// ------------------------------------------------- cluster / cta_group::2 ops
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
// Arrive once on the mbarrier at the same shared-memory offset in CTA `rank`
// of the cluster (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint64_t* bar, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}
// The same without release semantics.  Used to hand P (in this CTA's tensor
// memory) to CTA 0's issuer -- the stores are already complete
// (tcgen05.wait::st, then tcgen05.fence::before_thread_sync), and the release
// form measured ~800 clocks per arrive on this critical path -- and to tell
// CTA 0 that this CTA's half of a ring stage (its own TMA loads, observed
// complete) has landed.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint64_t* bar, uint32_t rank) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(bar)), "r"(rank));
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* smem_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(smem_slot)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// D (TMEM of both CTAs) (+)= A (M = 256: 128 rows in each CTA's smem) * B
// (N split in half between the two CTAs' smem).
__device__ __forceinline__ void mma_pair_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// The same with A read from each CTA's own TMEM (its 128 rows).
__device__ __forceinline__ void mma_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the barrier at this offset in both CTAs once the pair's previously
// issued MMAs complete.
__device__ __forceinline__ void commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 "
      "[%0], %1;" ::"r"(smem_u32(bar)),
      "h"((uint16_t)3)
      : "memory");
}

struct PairCfg {
  static constexpr int D = 128, KT = 128, PPT = KT / kP;
  static constexpr int THREADS = 352;
  static constexpr int PRODUCER = 8, MMA = 9, WRITER = 10;
  static constexpr int Q_BYTES = kRows * D * 2;           // one 128-row Q tile (32 KB)
  static constexpr int H_BYTES = KT * D;                  // half of a K or V tile (16 KB)
  static constexpr int BUDGET = 231424;
  static constexpr int FIXED = 2 * Q_BYTES + 512 + 1024;
  static constexpr int RS_FIT = (BUDGET - FIXED) / H_BYTES;
  static constexpr int RS = RS_FIT < 12 ? RS_FIT : 12;    // ring stages (half tiles)
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = 2 * Q_BYTES;
  static constexpr int OFF_BAR = OFF_RING + RS * H_BYTES;
  // q_full, q_peer, ring_full[RS], ring_empty[RS], peer_full[RS], s_full[2],
  // p_full[2], o_done[2], v_clean
  static constexpr int NBAR = 2 + 3 * RS + 7;
  static constexpr int OFF_TMEM = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_TMEM + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static constexpr int O_COL = 2 * KT;
  static constexpr int TMEM_COLS = 512;
  static_assert(RS >= 6, "ring too shallow");
  static_assert(ALLOC <= 232448, "shared memory budget");
};

__device__ __forceinline__ uint64_t desc_kmajor_p(uint32_t addr) { return smem_desc_sw128(addr, 16, 1024); }
__device__ __forceinline__ uint64_t desc_mnmajor_p(uint32_t addr) {
  // one 64-column N block per CTA: LBO is not used
  return smem_desc_sw128(addr, PairCfg::KT * 128, 1024);
}

template <bool TREE>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairCfg::THREADS, 1)
prefill_pair_kernel(const __grid_constant__ PairParams prm) {
  using C = PairCfg;
  constexpr int D = C::D, KT = C::KT, PPT = C::PPT, RS = C::RS;
  const PrefillArgs& a = prm.a;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* q_peer = bars + 1;
  uint64_t* ring_full = bars + 2;
  uint64_t* ring_empty = ring_full + RS;
  uint64_t* peer_full = ring_empty + RS;
  uint64_t* s_full = peer_full + RS;  // [2]
  uint64_t* p_full = s_full + 2;      // [2]
  uint64_t* o_done = p_full + 2;      // [2]
  uint64_t* v_clean = o_done + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM);

  const uint32_t rank = cluster_ctarank();
  const PrefillTile tile = prm.tiles[blockIdx.x >> 1];
  const int kvh = blockIdx.y;
  const int g = a.group;
  const int tpt = kRows / g;  // tokens per Q tile
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_tiles = (tile.ntok + tpt - 1) / tpt;  // Q tiles of the item (1..4)
  const int nq = (n_tiles + 1) >> 1;                 // M = 256 tile pairs (1 or 2)

  // key tiles kt0 .. kt0 + n_kt - 1 cover keys [key_lo, kend); causal rows mask
  // beyond their own position.  A prefix-group item's keys (a cached prefix
  // shared by several requests) precede every one of its rows: no mask.
  const bool prefix_group = tile.kind == kTilePrefixGroup;
  const bool causal = a.causal && !prefix_group;
  const int pos_first = tile.kv_len - tile.qo_len + tile.tok0;
  const int kv_end = causal ? min(tile.kv_len, pos_first + tile.ntok) : tile.kv_len;
  const int kend = min(kv_end, tile.key_hi);
  const int kt0 = tile.key_lo / KT;
  const int n_kt = (kend + KT - 1) / KT - kt0;
  const int npages_req = (tile.kv_len + kP - 1) / kP;
  const bool last_partial = tile.kv_len - (kt0 + n_kt - 1) * KT < KT;

  // fused append: key tiles from fuse_key on are the chunk's own keys, read
  // from k_new / v_new; this item writes into the pages each such tile whose
  // first new token (kb - first_new_key) is one of its own tokens, so every
  // new row is written once per kv head
  const int first_new_key = tile.kv_len - tile.qo_len;
  const bool fuse = a.fuse_min_qo > 0 && !prefix_group && tile.qo_len >= a.fuse_min_qo;
  const int fuse_key = fuse ? fused_from(tile.kv_len, tile.qo_len) : INT_MAX;
  auto owns = [&](int j) {
    const int kb = (kt0 + j) * KT, t = kb - first_new_key;
    return kb >= fuse_key && t >= tile.tok0 && t < tile.tok0 + tile.ntok;
  };
  const int own_lo = max(fuse_key, first_new_key + tile.tok0);  // first key whose tile it may own
  const bool writer_on =
      fuse && (own_lo + KT - 1) / KT * KT < first_new_key + tile.tok0 + tile.ntok;

  if (tid == 0) {
    prefetch_tmap(&prm.tmap_q);
    prefetch_tmap(&prm.tmap_kv);
    if (fuse) {
      prefetch_tmap(&prm.tmap_kn);
      prefetch_tmap(&prm.tmap_vn);
    }
    mbar_init(q_full, 1);
    mbar_init(q_peer, 1);
    for (int i = 0; i < RS; ++i) {
      mbar_init(&ring_full[i], 1);
      // MMA completion, plus the page writer once it has copied the stage out
      mbar_init(&ring_empty[i], writer_on ? 2 : 1);
      mbar_init(&peer_full[i], 1);
    }
    for (int q = 0; q < 2; ++q) {
      mbar_init(&s_full[q], 1);
      mbar_init(&p_full[q], 8);  // the tile pair's 4 + 4 softmax warps
      mbar_init(&o_done[q], 1);
    }
    mbar_init(v_clean, 2);
    fence_mbar_init();
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == C::MMA) {
    tmem_alloc_pair(tmem_slot, C::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrive or commit
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (tid == 0) grid_dep_launch();

  if (warp == C::PRODUCER) {
    // ------------------------------------------------------------ producer
    // This CTA's half of K tile j: keys [64 r, 64 r + 64) = pages 4r .. 4r+3,
    // both 64-column blocks, as two [64 rows][128 B] panels.  Its half of V tile
    // j: all 8 pages, column block r, as one [128 rows][128 B] panel.
    // Page ids of key tile j: lane l (< 8) holds the id of the tile's l-th
    // page (K_j and V_j share them).  Loaded coalesced, four tiles ahead, in a
    // register pipeline, so the id latency never stalls the issue loop.
    auto load_ids = [&](int j) -> int64_t {
      if (j >= n_kt) return -1;
      const int pg0 = (kt0 + j) * PPT;
      const int np = min(PPT, npages_req - pg0);
      return lane < np ? (int64_t)__ldg(a.page_indices + tile.page_base + pg0 + lane) : -1;
    };
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, (uint32_t)(nq * tpt * g * D * 2));
      for (int q = 0; q < nq; ++q) {
        const int t = 2 * q + (int)rank;  // tile of the item held in local slot q
        for (int b = 0; b < 2; ++b)
          tma_load_3d(smem + C::OFF_Q + q * C::Q_BYTES + b * (kRows * 128), &prm.tmap_q, b * 64,
                      kvh * g, tile.q_row0 + tile.tok0 + t * tpt, q_full);
      }
    }
    int64_t id0 = load_ids(0), id1 = load_ids(1), id2 = load_ids(2), id3 = load_ids(3);
    // the request's last qo_len keys are the rows appended in this step: the
    // first key tile that reaches them waits for the kernel launched before
    // this one (tiles of cached keys stream while that kernel still runs).  A
    // prefix-group item reads only cached keys.
    const int first_new = prefix_group ? tile.kv_len : tile.kv_len - tile.qo_len;
    bool dep_waited = false;
    for (int i = 0; i < 2 * n_kt; ++i) {
      const int st = i % RS;
      const bool is_v = i & 1;
      const int kb = (kt0 + (i >> 1)) * KT;
      const int pg0 = kb / kP;
      uint8_t* buf = smem + C::OFF_RING + st * C::H_BYTES;
      if (kb >= fuse_key) {
        // the chunk's own keys, from k_new / v_new (row = q_row0 + key - first
        // new key); rows past the request's end are other requests' rows or
        // zero fill, masked like stale slots
        if (lane == 0) {
          if (i >= RS) mbar_wait(&ring_empty[st], ((i / RS) - 1) & 1, a.err);
          mbar_arrive_expect_tx(&ring_full[st], (uint32_t)C::H_BYTES);
          const int row = tile.q_row0 + (kb - first_new_key);
          if (is_v) {
            tma_load_3d(buf, &prm.tmap_vn, (int)rank * 64, kvh, row, &ring_full[st]);
          } else {
#pragma unroll
            for (int b = 0; b < 2; ++b)
              tma_load_3d(buf + b * (64 * 128), &prm.tmap_kn, b * 64, kvh, row + 64 * (int)rank,
                          &ring_full[st]);
          }
        }
        __syncwarp();
        if (is_v) {  // tile done: shift the id pipeline
          id0 = id1;
          id1 = id2;
          id2 = id3;
          id3 = load_ids((i >> 1) + 4);
        }
        continue;
      }
      if (!dep_waited && kb + KT > first_new) {
        grid_dep_wait();
        dep_waited = true;
      }
      const int np = min(PPT, npages_req - pg0);
      const int kp = max(0, min(4, np - 4 * (int)rank));  // pages of this CTA's K half
      if (lane == 0) {
        if (i >= RS) mbar_wait(&ring_empty[st], ((i / RS) - 1) & 1, a.err);
        mbar_arrive_expect_tx(&ring_full[st], (uint32_t)((is_v ? np : 2 * kp) * kP * 128));
      }
      __syncwarp();
      const bool mine = is_v ? lane < np : (lane >= 4 * (int)rank && lane < 4 * (int)rank + kp);
      if (mine) {
        int64_t page = id0;
        if (page < 0 || page >= a.num_pages) {
          set_device_error(a.err, kDevErrPageRange);
          page = 0;  // fetch a valid page instead; the output is undefined anyway
        }
        const int32_t slice = (int32_t)((page * 2 + (is_v ? 1 : 0)) * a.Hkv + kvh);
        if (is_v) {
          tma_load_3d(buf + lane * (kP * 128), &prm.tmap_kv, (int)rank * 64, 0, slice, &ring_full[st]);
        } else {
          const int p = lane - 4 * (int)rank;
#pragma unroll
          for (int b = 0; b < 2; ++b)
            tma_load_3d(buf + b * (64 * 128) + p * (kP * 128), &prm.tmap_kv, b * 64, 0, slice,
                        &ring_full[st]);
        }
      }
      if (is_v) {  // tile done: shift the id pipeline
        id0 = id1;
        id1 = id2;
        id2 = id3;
        id3 = load_ids((i >> 1) + 4);
      }
    }
    // an item that read no appended row from the pages (a prefix-group item,
    // or one whose new keys all came from k_new) still waits before it exits:
    // a launch may hold nothing else, and the kernels after it rely on its
    // completion implying that of the kernel before it
    if (!dep_waited) grid_dep_wait();
    __syncwarp();
    if (last_partial) {
      // this CTA's half of the last V tile: rows past the request's last key
      // must hold finite values
      const int i = 2 * n_kt - 1, st = i % RS;
      const int tile_keys = tile.kv_len - (kt0 + n_kt - 1) * KT;
      uint8_t* buf = smem + C::OFF_RING + st * C::H_BYTES;
      mbar_wait(&ring_full[st], (i / RS) & 1, a.err);
      for (int idx = lane; idx < (KT - tile_keys) * 8; idx += 32) {
        const int r = tile_keys + (idx >> 3), ch = idx & 7;
        *reinterpret_cast<uint4*>(buf + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(v_clean);
        else
          mbar_arrive_cluster(v_clean, 0);
      }
    }
  } else if (warp == C::MMA && rank == 1) {
    // ------------------------------------------------------ relay (CTA 1)
    // CTA 0 issues MMAs that read this CTA's shared memory: tell it when each
    // of this CTA's Q tiles and ring stages has landed.  The stage arrives are
    // relaxed: the bytes are this CTA's own TMA loads, complete once its
    // ring_full phase is observed, and this thread publishes no writes of its
    // own.  The release form cost ~1100 clocks per ring item here, about two
    // thirds of this warp's time, and CTA 0 waited on it.
    mbar_wait(q_full, 0, a.err);
    __syncwarp();
    if (lane == 0) mbar_arrive_cluster(q_peer, 0);
    for (int i = 0; i < 2 * n_kt; ++i) {
      const int st = i % RS;
      mbar_wait(&ring_full[st], (i / RS) & 1, a.err);
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster_relaxed(&peer_full[st], 0);
    }
  } else if (warp == C::MMA) {
    // ------------------------------------------------- MMA issuer (CTA 0)
    // Converged warp, one elected lane issues (see elect_one).
    constexpr uint32_t idesc_s = idesc_bf16_f32(2 * kRows, KT, 0, 0);
    constexpr uint32_t idesc_o = idesc_bf16_f32(2 * kRows, D, 0, 1);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sR = smem_u32(smem + C::OFF_RING);
    auto wait = [&](uint64_t* bar, uint32_t parity) {
      mbar_wait(bar, parity, a.err);
      __syncwarp();
    };
    auto commit = [&](uint64_t* bar) {
      if (elect_one()) commit_pair(bar);
      __syncwarp();
    };
    auto wait_stage = [&](int i) {  // both CTAs' halves of ring item i
      const int st = i % RS;
      wait(&ring_full[st], (i / RS) & 1);
      wait(&peer_full[st], (i / RS) & 1);
      tc_fence_after();
    };
    auto issue_s = [&](int q, int st) {  // S_q = Q_q K^T (N = 128 keys, 64 per CTA)
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint64_t da = desc_kmajor_p(sQ + q * C::Q_BYTES + (k >> 2) * (kRows * 128) + (k & 3) * 32);
        const uint64_t db = desc_kmajor_p(sR + st * C::H_BYTES + (k >> 2) * (64 * 128) + (k & 3) * 32);
        if (elect_one()) mma_pair_ss(tmem + q * KT, da, db, idesc_s, k > 0 ? 1u : 0u);
      }
      __syncwarp();
    };
    auto issue_pv = [&](int q, int st, bool accumulate) {  // O_q += P_q V (N = 128, 64 per CTA)
#pragma unroll
      for (int k = 0; k < KT / 16; ++k) {
        const uint64_t db = desc_mnmajor_p(sR + st * C::H_BYTES + k * (16 * 128));
        if (elect_one())
          mma_pair_ts(tmem + C::O_COL + q * D, tmem + q * KT + k * 8, db, idesc_o,
                      (accumulate || k > 0) ? 1u : 0u);
      }
      __syncwarp();
    };
    wait(q_full, 0);
    wait(q_peer, 0);
    wait_stage(0);
    for (int q = 0; q < nq; ++q) {
      issue_s(q, 0);
      commit(&s_full[q]);
    }
    commit(&ring_empty[0]);
    for (int j = 0; j < n_kt; ++j) {
      const int iv = 2 * j + 1, sv = iv % RS;
      const int ik = 2 * j + 2, sk = ik % RS;
      wait_stage(iv);
      if (j == n_kt - 1 && last_partial) wait(v_clean, 0);
      bool k_ready = false;
      for (int q = 0; q < nq; ++q) {
        wait(&p_full[q], j & 1);
        tc_fence_after();
        issue_pv(q, sv, j > 0);
        commit(&o_done[q]);
        if (j + 1 < n_kt) {
          if (!k_ready) {
            wait_stage(ik);
            k_ready = true;
          }
          issue_s(q, sk);
          commit(&s_full[q]);
        }
      }
      commit(&ring_empty[sv]);
      if (j + 1 < n_kt) commit(&ring_empty[sk]);
    }
  } else if (warp == C::WRITER) {
    // ----------------------------------------------------- page writer
    // Fused append: write this CTA's part of every owned tile from shared
    // memory into the pages (K: keys [64 r, 64 r + 64) of the tile, both
    // 64-column halves; V: all 128 keys, columns [64 r, 64 r + 64)).  A page
    // whose 16 slots are all keys of the request goes out as TMA stores of the
    // same {64, 16, 1} boxes the loads use (the TMA unit undoes the 128-byte
    // swizzle); the request's partial last page goes out row by row with plain
    // stores (16-byte chunk c of stage row R sits at chunk c ^ (R % 8)), so no
    // slot at or past kv_len is written.  The writer releases every ring stage
    // (ring_empty counts it) once its stores have read the stage.
    if (writer_on) {
      for (int i = 0; i < 2 * n_kt; ++i) {
        const int st = i % RS;
        mbar_wait(&ring_full[st], (i / RS) & 1, a.err);
        if (owns(i >> 1)) {
          const uint8_t* buf = smem + C::OFF_RING + st * C::H_BYTES;
          const bool is_v = i & 1;
          const int kb = (kt0 + (i >> 1)) * KT;
          const int key0 = is_v ? kb : kb + 64 * (int)rank;  // first key of this CTA's part
          const int npg = is_v ? 8 : 4;                       // pages of this CTA's part
          // lane l < npg: page l of the part
          int64_t page = -1;
          int keys = 0;  // keys of the request on page l
          if (lane < npg) {
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
            if (is_v) {
              tma_store_3d(&prm.tmap_kv, (int)rank * 64, 0, slice, buf + lane * (kP * 128));
            } else {
#pragma unroll
              for (int b = 0; b < 2; ++b)
                tma_store_3d(&prm.tmap_kv, b * 64, 0, slice, buf + b * (64 * 128) + lane * (kP * 128));
            }
            bulk_commit();
          }
          // the partial last page (at most one per part): plain stores
          const uint32_t part_mask = __ballot_sync(0xffffffffu, page >= 0 && keys < kP);
          if (part_mask) {
            const int pl = __ffs(part_mask) - 1;
            const int pkeys = __shfl_sync(0xffffffffu, keys, pl);
            const int64_t ppage = __shfl_sync(0xffffffffu, page, pl);
            const int nch = is_v ? 8 : 16;  // 16-byte chunks per row of this part
            uint16_t* row0 = a.pool_w + (((ppage * 2 + (is_v ? 1 : 0)) * a.Hkv + kvh) * kP) * D;
            for (int idx = lane; idx < pkeys * nch; idx += 32) {
              const int sl = idx / nch, ch = idx - sl * nch;
              const int b = is_v ? 0 : ch >> 3, cc = ch & 7;
              const int R = pl * kP + sl;  // row within this CTA's panel
              const uint4 v = *reinterpret_cast<const uint4*>(buf + b * (64 * 128) + R * 128 +
                                                              ((cc ^ (R & 7)) << 4));
              reinterpret_cast<uint4*>(row0 + sl * D)[(is_v ? (int)rank : b) * 8 + cc] = v;
            }
          }
          if (page >= 0 && keys == kP) bulk_wait_read();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring_empty[st]);
      }
      bulk_wait_all();
    }
  } else if (warp / 4 < nq) {
    // ------------------------------------------------------------- softmax
    // Every warp of a live tile pair runs (rows past the item's tokens compute
    // values that are not written): CTA 0's issuer counts 8 arrivals per P.
    const int q = warp >> 2;
    const int row = tid & 127;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const int t = 2 * q + (int)rank;
    const int q_tok0 = tile.tok0 + t * tpt;  // first token of this Q tile
    const int q_ntok = max(0, min(tpt, tile.ntok - t * tpt));
    const int tl = row / g;
    const int qpos = tile.kv_len - tile.qo_len + q_tok0 + tl;
    const int row_end = min(causal ? min(qpos + 1, tile.kv_len) : tile.kv_len, kend);
    SoftmaxRowOut ro;
    ro.q_row = tile.q_row0 + q_tok0 + tl;
    ro.hq = kvh * g + (row - tl * g);
    ro.write = row < q_ntok * g;
    // partial slot of token t (counted from the first token of the request, or
    // of the group) when the item covers only part of the row's keys
    ro.part = tile.part >= 0 ? tile.part + (q_tok0 + tl) * tile.part_stride : -1;
    TreeRow tr;
    tr.bits = TREE && ro.write && !prefix_group ? a.tree_mask + (int64_t)ro.q_row * a.mask_words
                                                : nullptr;
    tr.words = a.mask_words;
    tr.draft0 = prefix_group ? tile.kv_len : tile.kv_len - tile.qo_len;  // no draft keys
    tr.tok = prefix_group ? 0 : q_tok0 + tl;
    tc_softmax_rows<D, KT, TREE>(a, tmem + lane_off, tmem + C::O_COL + q * D + lane_off, s_full, &o_done[q],
                           q, false, n_kt, kt0, row_end, ro, tr, [&](int b) {
                             if (lane == 0) {
                               if (rank == 0)
                                 mbar_arrive(&p_full[b]);
                               else
                                 mbar_arrive_cluster_relaxed(&p_full[b], 0);
                             }
                           });
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // neither CTA leaves while the pair's MMAs or arrives may reach it
  if (warp == C::MMA) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, C::TMEM_COLS);
  }
}

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

}  // namespace

cudaError_t launch_prefill_pair(const PrefillArgs& a, cudaStream_t stream, bool programmatic) {
  if (a.n_tiles <= 0) return cudaSuccess;
  if (a.head_dim != 128) return cudaErrorInvalidValue;
  constexpr int D = 128;
  EncodeTiledFn enc = get_encode_fn();
  if (!enc) return cudaErrorNotSupported;
  PairParams prm;
  prm.a = a;
  prm.tiles = a.tiles;
  const int g = a.group;
  {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.Hq, (cuuint64_t)a.nnz_qo};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hq * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)g, (cuuint32_t)(kRows / g)};
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
  if (a.fuse_min_qo > 0) {
    // the fused call's new rows: [nnz_qo][Hkv][d], K boxes of 64 rows (this
    // CTA's half of a key tile), V boxes of 128 rows
    for (int v = 0; v < 2; ++v) {
      cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)a.Hkv, (cuuint64_t)a.nnz_qo};
      cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)a.Hkv * D * 2};
      cuuint32_t box[3] = {64, 1, v ? 128u : 64u};
      cuuint32_t es[3] = {1, 1, 1};
      if (enc(v ? &prm.tmap_vn : &prm.tmap_kn, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
              (void*)(v ? a.v_new : a.k_new), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    }
  }
  // the draft-tree variant only when the call carries a mask
  auto kern = a.tree_mask ? prefill_pair_kernel<true> : prefill_pair_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PairCfg::ALLOC);
  if (e != cudaSuccess) return e;
  return launch_kernel(kern, dim3(2 * a.n_tiles, a.Hkv), dim3(PairCfg::THREADS),
                       PairCfg::ALLOC, stream, programmatic, prm);
}

}  // namespace daa
