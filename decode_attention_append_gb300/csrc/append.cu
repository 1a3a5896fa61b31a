// KV append: scatter each new token's K and V rows into its page slot.
//
// "Chunked prefill" (k4i.top), #correctness: after a chunk the new k, v
// vectors are appended to the KV cache (K_cache += [k_{(s-1)C+1} .. k_{sC}]);
// #io-overhead: the append moves C x 2 x Hkv x d x 2 bytes per layer.
// "Disaggregated prefill and decode" (Perplexity), "Sharded KV cache
// transfers": HND pages, so head h of token slot s is one contiguous d-row.
//
// Bandwidth design: the (token row, K/V, head, 16-byte chunk) space is cut into
// equal contiguous ranges, one per CTA, sized from the SM count so that small
// appends (one token per request) still spread over every SM and large ones
// give each thread ~16 chunks in flight.  The owner request of each row a CTA
// touches is found once (binary search over append_indptr) into shared memory;
// then all threads stream 16-byte chunks with read-only, no-allocate loads.
// Source rows are contiguous ([Hkv][d] per token); each destination (head,
// slot) row is 2*d contiguous bytes, so warps write whole 128-byte lines.
// In a fused append + attention call the prefill kernels write the rows of
// long prefill requests from their first 128-aligned key tile on themselves
// (they read those tiles from k_new / v_new anyway); this kernel then skips
// them (fuse_min_qo > 0), and its grid covers only the span of rows
// [row_begin, row_begin + n_rows) that holds the others.
#include "launch.h"
#include "ptx.cuh"

namespace daa {

namespace {

constexpr int kAppendThreads = 128;
constexpr int kAppendMaxRows = 64;

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int D>
__global__ void __launch_bounds__(kAppendThreads)
kv_append_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                 uint4* __restrict__ pool, const int32_t* __restrict__ append_indptr,
                 const int32_t* __restrict__ page_indices, const int32_t* __restrict__ kv_indptr,
                 const int32_t* __restrict__ last_page_len, int batch, int row_begin, int n_rows,
                 int Hkv, int chunks_per_cta, int64_t num_pages, int fuse_min_qo, int* err) {
  constexpr int P = 16;
  constexpr int CH = D / 8;  // 16-byte chunks per (head, slot) row
  __shared__ int64_t s_dst[kAppendMaxRows];  // chunk index of (page, K, head 0, slot, 0); -1 = skip

  // the attention kernels of a fused call may start their CTAs now: the ones
  // that read appended rows wait for this grid to complete
  if (threadIdx.x == 0) grid_dep_launch();

  const int per_row = 2 * Hkv * CH;
  // chunk indices count from row row_begin
  const int64_t total = (int64_t)n_rows * per_row;
  const int64_t first = (int64_t)blockIdx.x * chunks_per_cta;
  const int64_t last = min(first + chunks_per_cta, total);
  const int row0 = (int)(first / per_row);
  const int nrows = (int)((last - 1) / per_row) - row0 + 1;
  if (threadIdx.x < nrows) {
    const int row = row_begin + row0 + threadIdx.x;
    int lo = 0, hi = batch - 1;  // largest r with append_indptr[r] <= row
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(append_indptr + mid) <= row) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int a0 = __ldg(append_indptr + r), a1 = __ldg(append_indptr + r + 1);
    const int p0 = __ldg(kv_indptr + r), np = __ldg(kv_indptr + r + 1) - p0;
    const int last_len = np > 0 ? __ldg(last_page_len + r) : 0;
    const int64_t kv_len = np > 0 ? (int64_t)(np - 1) * P + last_len : 0;
    const int n_new = a1 - a0;
    int64_t dst = -1;
    if (row < a0 || row >= a1 || n_new > kv_len || (np > 0 && (last_len < 1 || last_len > P))) {
      set_device_error(err, kDevErrShape);
    } else {
      const int64_t pos = kv_len - n_new + (row - a0);
      const int64_t page = __ldg(page_indices + p0 + pos / P);
      if (fuse_min_qo > 0 && n_new >= fuse_min_qo && pos >= fused_from((int)kv_len, n_new)) {
        // written by the prefill kernel of this fused call, from the same rows
      } else if (page < 0 || page >= num_pages) {
        set_device_error(err, kDevErrPageRange);
      } else {
        dst = ((page * 2) * Hkv * P + (pos % P)) * CH;
      }
    }
    s_dst[threadIdx.x] = dst;
  }
  __syncthreads();

  // flat chunk index i over (row, kv, head, c), c fastest
  constexpr int U = 4;
  for (int64_t base = first + threadIdx.x; base < last; base += kAppendThreads * U) {
    uint4 val[U];
    int64_t dst[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t i = base + (int64_t)u * kAppendThreads;
      dst[u] = -1;
      if (i < last) {
        const int row = (int)(i / per_row);
        const int rem = (int)(i - (int64_t)row * per_row);
        const int kv = rem / (Hkv * CH);
        const int hc = rem - kv * (Hkv * CH);  // h * CH + c
        const int h = hc / CH, c = hc - h * CH;
        const int64_t d0 = s_dst[row - row0];
        if (d0 >= 0) {
          const uint4* src = (kv == 0 ? k_new : v_new) + (int64_t)(row_begin + row) * Hkv * CH + hc;
          val[u] = ld_stream(src);
          dst[u] = d0 + ((int64_t)kv * Hkv + h) * P * CH + c;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (dst[u] >= 0) pool[dst[u]] = val[u];
  }
}

}  // namespace

AppendSpan append_span(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                       const int32_t* h_last_page_len, int batch, int page_size, int fuse_min_qo) {
  AppendSpan sp{batch > 0 ? h_qo_indptr[batch] : 0, 0};
  for (int r = 0; r < batch; ++r) {
    const int n_new = h_qo_indptr[r + 1] - h_qo_indptr[r];
    if (n_new <= 0) continue;
    int keep = n_new;  // the request's rows the append kernel writes: its first `keep`
    if (fuse_min_qo > 0 && n_new >= fuse_min_qo) {
      const int np = h_kv_indptr[r + 1] - h_kv_indptr[r];
      const int kv_len = np > 0 ? (np - 1) * page_size + h_last_page_len[r] : 0;
      keep = fused_from(kv_len, n_new) - (kv_len - n_new);
      keep = keep < 0 ? 0 : (keep > n_new ? n_new : keep);
    }
    if (keep > 0) {
      sp.begin = h_qo_indptr[r] < sp.begin ? h_qo_indptr[r] : sp.begin;
      sp.end = h_qo_indptr[r] + keep > sp.end ? h_qo_indptr[r] + keep : sp.end;
    }
  }
  if (sp.end <= sp.begin) sp = AppendSpan{0, 0};
  return sp;
}

cudaError_t launch_kv_append(const void* k_new, const void* v_new, void* pool,
                             const int32_t* append_indptr, const int32_t* page_indices,
                             const int32_t* kv_indptr, const int32_t* last_page_len, int batch,
                             int row_begin, int n_rows, int Hkv, int head_dim, int64_t num_pages,
                             int num_sms, int fuse_min_qo, int* err, cudaStream_t stream) {
  if (n_rows <= 0 || batch <= 0) return cudaSuccess;
  const int per_row = 2 * Hkv * (head_dim / 8);
  const int64_t total = (int64_t)n_rows * per_row;
  // ~4 CTAs per SM for small appends, up to 16 chunks per thread for large ones,
  // and never more rows per CTA than the shared row table holds
  int64_t cpc = (total + (int64_t)num_sms * 4 - 1) / ((int64_t)num_sms * 4);
  cpc = ((cpc + kAppendThreads - 1) / kAppendThreads) * kAppendThreads;
  cpc = cpc < kAppendThreads ? kAppendThreads : (cpc > 16 * kAppendThreads ? 16 * kAppendThreads : cpc);
  const int64_t max_cpc = (int64_t)(kAppendMaxRows - 1) * per_row;
  if (cpc > max_cpc) cpc = max_cpc;
  const int64_t grid = (total + cpc - 1) / cpc;
  if (grid > INT32_MAX) return cudaErrorInvalidValue;
  if (head_dim == 128) {
    kv_append_kernel<128><<<(unsigned)grid, kAppendThreads, 0, stream>>>(
        (const uint4*)k_new, (const uint4*)v_new, (uint4*)pool, append_indptr, page_indices,
        kv_indptr, last_page_len, batch, row_begin, n_rows, Hkv, (int)cpc, num_pages, fuse_min_qo,
        err);
  } else {
    kv_append_kernel<64><<<(unsigned)grid, kAppendThreads, 0, stream>>>(
        (const uint4*)k_new, (const uint4*)v_new, (uint4*)pool, append_indptr, page_indices,
        kv_indptr, last_page_len, batch, row_begin, n_rows, Hkv, (int)cpc, num_pages, fuse_min_qo,
        err);
  }
  return cudaGetLastError();
}

}  // namespace daa
