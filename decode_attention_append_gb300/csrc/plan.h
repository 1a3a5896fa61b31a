// Work descriptors that the host planner writes into the workspace and the
// kernels read.  Plain 32-byte PODs so one cudaMemcpyAsync moves the whole plan.
#pragma once
#include <cstddef>
#include <cstdint>

namespace daa {

// One split of the keys of one decode request (qo_len == 1).  The decode kernel
// runs one CTA per (unit, kv head).  Splits are page aligned.
struct DecodeUnit {
  int32_t q_row;      // row of q / out / lse_out
  int32_t page_base;  // index into page_indices of the request's first page
  int32_t tok_begin;  // first key of this split (multiple of page_size)
  int32_t tok_end;    // one past the last key of this split
  int32_t kv_len;     // keys of the whole request
  int32_t part;       // partial slot, or -1 when the split covers the request
  int32_t pad0, pad1;
};

// softmax_merge of the partials of one query row: n_parts consecutive slots
// from part_begin (the key splits of its request), plus slot `extra` when the
// row's shared prefix was attended by a prefix-group item (else -1).
struct MergeItem {
  int32_t q_row;
  int32_t part_begin;  // first partial slot
  int32_t n_parts;     // consecutive slots to merge
  int32_t extra;       // one more slot (the row's shared-prefix partial), or -1
};

// A work item of the tensor-core kernel: one or two 128-row tiles of packed
// query rows of one request, over keys [key_lo, min(key_hi, causal end)).
// Tile 0 holds new tokens [tok0, tok0 + ntok) of the request, tile 1 (if
// ntok1 > 0) the next ntok1 tokens; each token brings all g query heads of a
// kv head, packed token-major into ntok * g <= 128 rows per tile.  One CTA per
// (item, kv head); both tiles share every K/V tile the CTA loads.  Prefill
// pairs cover all keys and write the output; a decode or verify request (all
// its qo_len tokens in tile 0) may be split over 128-key-aligned key ranges,
// each writing partial (o, lse) rows to slots part + t * part_stride for
// softmax_merge.
struct PrefillTile {
  int32_t q_row0;     // row of the request's first new token
  int32_t qo_len;
  int32_t kv_len;
  int32_t page_base;
  int32_t tok0;       // first new-token index (0-based within the request)
  int32_t ntok;       // tokens in tile 0
  int32_t ntok1;      // tokens in tile 1 (0: no second tile)
  int32_t key_lo;     // first key (multiple of 128)
  int32_t key_hi;     // one past the last key
  int32_t part;       // partial slot, or -1: write out / lse_out directly
  int32_t part_stride;  // key-split multi-token item: token t of the request writes its
                        // partial to slot part + t * part_stride
  int32_t kind;       // kTileRequest, or kTilePrefixGroup (see below)
};

// Tile kinds.  A prefix-group item attends the query rows of several
// consecutive requests that share a cached prefix to the keys of that prefix
// (read once for all of them): q_row0 / qo_len span the group's rows,
// kv_len = key_hi = the shared keys (a multiple of 128), page_base = the first
// request's page list; every row sees every key (the prefix precedes all new
// tokens), and row t of the group writes its partial to slot part + t.
// The plan is copied to the device every call, so the item stays small: a
// plan under 64 KB is copied inline with the launches.

static_assert(sizeof(DecodeUnit) == 32, "DecodeUnit layout");
static_assert(sizeof(MergeItem) == 16, "MergeItem layout");
constexpr int32_t kTileRequest = 0;
constexpr int32_t kTilePrefixGroup = 1;

static_assert(sizeof(PrefillTile) == 48, "PrefillTile layout");

// Kernel ids reported by the tracer.
enum KernelId : int32_t {
  kKernelAppend = 1,
  kKernelDecode = 2,
  kKernelMerge = 3,
  kKernelPrefill = 4,
  kKernelTcDecode = 5,
  kKernelShort = 6,   // short multi-token items on the single-CTA kernel (head_dim 128)
};

}  // namespace daa
