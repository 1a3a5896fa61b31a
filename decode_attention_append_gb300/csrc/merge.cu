// softmax_merge of split-KV partial attentions: one warp per (query row,
// query head); the arithmetic is merge_row_head (merge.cuh).
#include "merge.cuh"

namespace daa {
namespace {

constexpr int kMergeWarps = 4;

template <int D>
__global__ void __launch_bounds__(32 * kMergeWarps) softmax_merge_kernel(const MergeArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hq = blockIdx.y * kMergeWarps + warp;
  // the item comes from the plan, copied before any kernel of the call ran
  const MergeItem it = a.items[blockIdx.x];
  grid_dep_wait();  // the partials come from the kernels launched before
  if (hq >= a.Hq) return;
  merge_row_head<D>(it, a.Hq, hq, a.part_o, a.part_lse, a.out, a.lse_out, lane);
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
