/*
 * daa.h -- C ABI of libdaa: paged KV append and mixed-batch paged attention
 * (chunked-prefill requests and decode requests in one batch) for sm_103a.
 *
 * The operation, from the pages it follows:
 *  - "Chunked prefill" (k4i.top), section "Why chunking does not change the
 *    result" (#correctness): a prompt is processed in chunks; token i of a
 *    chunk attends to every position j <= i, i.e. to the cached prefix written
 *    by earlier chunks plus the causal part of its own chunk, and the two parts
 *    combine by softmax_merge; after each chunk its new k, v vectors are
 *    appended to the KV cache.  Section "IO overhead" (#io-overhead) sizes that
 *    append: C x 2 x n_h x d_h x 2 bytes per layer.
 *  - "Disaggregated prefill and decode" (Perplexity), section "Prefill vs decode
 *    performance": decode requests carry qo_len = 1 and are memory bound,
 *    prefill requests carry large qo_len and are compute bound; attention can
 *    be split over requests and over kv_len.  Section "Sharded KV cache
 *    transfers" with the figure "NHD and HND KV cache layouts": the cache is
 *    paged in the HND layout (heads before tokens), so each head's slice of a
 *    page is contiguous.  Section "KV Messenger": KV entries are valid after
 *    the append and before attention reads them.
 *
 * Conventions shared by every call
 *  - All tensors are bf16 (bit patterns, 2 bytes per element), row-major and
 *    contiguous, on the device unless a parameter says "host".
 *  - Page pool `kv_pages`: [num_pages][2][Hkv][page_size][head_dim]; index 0 of
 *    the second dimension holds K, index 1 holds V (HND inside each page).
 *  - Page table (CSR): request r owns pages page_indices[kv_indptr[r] ..
 *    kv_indptr[r+1]); its length after this step's append is
 *    kv_len_r = (npages_r - 1) * page_size + last_page_len[r]
 *    (kv_len_r = 0 when it owns no page).  1 <= last_page_len[r] <= page_size
 *    whenever npages_r > 0.  The caller allocates pages; the table already
 *    covers the post-append length.  A page that receives appended tokens
 *    belongs to one request alone; pages that hold only cached tokens may be
 *    listed by several requests (a prefix-cache hit: "Chunked prefill",
 *    #prefix-cache-interaction), which read them in place.
 *  - Query / new-token rows (CSR): request r owns rows qo_indptr[r] ..
 *    qo_indptr[r+1]) of q, k_new, v_new and out; qo_len_r <= kv_len_r.  The new
 *    token i of request r sits at absolute position kv_len_r - qo_len_r + i.
 *  - GQA: query head h reads kv head h / (Hq / Hkv) (contiguous groups).
 *  - Ownership: the caller owns every buffer; the library allocates no device
 *    memory.  Pointers must be 16-byte aligned.
 *  - Ordering: work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and runs asynchronously; call daa_kv_append before
 *    daa_batch_attention on the same stream.  No call synchronises the device.
 *  - Errors: argument checks run on the host before anything is enqueued and
 *    return a negative daa_status; nothing is thrown across the ABI.  Device
 *    kernels never read or write outside the pool or the given arrays: a page
 *    id outside [0, num_pages) or an inconsistent length seen on the device is
 *    skipped and recorded in a device error word (daa_device_error).
 *  - Supported: head_dim in {64, 128}; page_size 16; 1 <= Hq/Hkv <= 16 with Hq
 *    divisible by Hkv.  Other shapes return DAA_ERR_UNSUPPORTED.
 */
#ifndef DAA_H_
#define DAA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DAA_OK = 0,
  DAA_ERR_INVALID_ARG = -1, /* null pointer, negative count, bad scalar */
  DAA_ERR_SHAPE = -2,       /* indptr not monotonic, qo_len > kv_len, bad last_page_len */
  DAA_ERR_PAGE_RANGE = -3,  /* page count inconsistent with the pool */
  DAA_ERR_UNSUPPORTED = -4, /* head_dim / page_size / group size outside the support matrix */
  DAA_ERR_CUDA = -5,        /* a CUDA runtime call or launch failed */
  DAA_ERR_WORKSPACE = -6,   /* workspace missing or smaller than the size query */
  DAA_ERR_ALIGNMENT = -7    /* a pointer is not 16-byte aligned */
} daa_status;

typedef struct {
  int32_t num_qo_heads; /* Hq */
  int32_t num_kv_heads; /* Hkv */
  int32_t head_dim;     /* d */
  int32_t page_size;    /* P (tokens per page) */
  int64_t num_pages;    /* pages in the pool */
} daa_dims;

/* Human-readable name of a status code (static storage). */
const char* daa_status_string(daa_status s);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int32_t daa_version(void);

/*
 * KV append ("Chunked prefill", #correctness: K_cache += [k_{(s-1)C+1} .. k_{sC}];
 * #io-overhead for its size).
 *
 * For every request r and each of its n_r = append_indptr[r+1] - append_indptr[r]
 * new tokens t (0 <= t < n_r), writes
 *   kv_pages[p][0][h][s][:] = k_new[append_indptr[r] + t][h][:]
 *   kv_pages[p][1][h][s][:] = v_new[append_indptr[r] + t][h][:]
 * for every kv head h, where pos = kv_len_r - n_r + t,
 * p = page_indices[kv_indptr[r] + pos / page_size] and s = pos % page_size.
 * A bit-exact copy; nothing else in the pool is touched.
 *
 *  k_new, v_new   device, bf16 [nnz_new][Hkv][head_dim]
 *  kv_pages       device, bf16 pool (see conventions), written
 *  append_indptr  device, int32 [batch + 1], append_indptr[batch] == nnz_new
 *                 (the same array as qo_indptr of the attention call)
 *  page_indices   device, int32 [kv_indptr[batch]]
 *  kv_indptr      device, int32 [batch + 1]
 *  last_page_len  device, int32 [batch], post-append
 *  batch, nnz_new host scalars (batch >= 0, nnz_new >= 0)
 *  dims           shapes; num_qo_heads is not used here but must be valid
 *  stream         cudaStream_t
 * Errors: DAA_ERR_INVALID_ARG / _UNSUPPORTED / _ALIGNMENT on the host,
 * DAA_ERR_CUDA if the launch fails.  Lengths and page ids are checked on the
 * device (see daa_device_error).
 */
daa_status daa_kv_append(const void* k_new, const void* v_new, void* kv_pages,
                         const int32_t* append_indptr, const int32_t* page_indices,
                         const int32_t* kv_indptr, const int32_t* last_page_len, int32_t batch,
                         int32_t nnz_new, daa_dims dims, void* stream);

/*
 * Bytes of device workspace daa_batch_attention needs for this batch (0 if
 * none).  Reads the host mirrors only; a pure function of its arguments and of
 * the current device's SM count.  Returns 0 and sets *status (if non-NULL) to
 * an error for invalid input.
 */
size_t daa_batch_attention_workspace_size(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                          const int32_t* h_last_page_len, int32_t batch,
                                          daa_dims dims, daa_status* status);

/*
 * Mixed-batch paged attention ("Chunked prefill", #correctness; "Disaggregated
 * prefill and decode", "Prefill vs decode performance").
 *
 * For every request r, new token i and query head h (kv head hk = h / (Hq/Hkv)),
 * with pos = kv_len_r - qo_len_r + i and key range J = {j : j <= pos} when
 * causal (J = {j < kv_len_r} otherwise):
 *   s_j = sm_scale * q[row][h][:] . K_r[j][hk][:]
 *   out[row][h][:] = sum_{j in J} softmax_J(s)_j * V_r[j][hk][:]      (bf16, RNE)
 *   lse_out[row][h] = ln sum_{j in J} exp(s_j)                          (fp32)
 * where row = qo_indptr[r] + i and K_r / V_r are read from the request's pages.
 * Routing (results do not depend on it): requests with qo_len = 1 run a
 * split-KV decode kernel (CUDA cores when a kv head serves fewer than 4 query
 * heads, tensor cores otherwise); requests with 2 <= qo_len <= min(16, 128 / g)
 * (g = Hq / Hkv; e.g. speculative-decoding verify steps) run as key-split
 * items of the tensor-core decode kernel; requests up to 256 / g tokens (two
 * 128-row tiles of packed query rows) run as items of the single-CTA
 * tensor-core kernel, key-split when long; longer requests run the
 * tensor-core prefill kernel.  Split requests are combined by the softmax_merge pass, one
 * merge per token.  Rows of requests with qo_len = 0 do not exist; nothing is
 * written.
 *
 *  q              device, bf16 [nnz_qo][Hq][head_dim]
 *  kv_pages       device, bf16 pool (read only)
 *  qo_indptr, kv_indptr, page_indices, last_page_len    device int32 (as above)
 *  h_qo_indptr, h_kv_indptr, h_last_page_len            host int32 copies of
 *                 the same arrays; used to validate and to plan the split of the
 *                 work on the host, so the call never waits on the device
 *  batch          number of requests
 *  causal         1: keys j <= pos; 0: all kv_len keys
 *  sm_scale       score scale, e.g. 1/sqrt(head_dim); must be finite and > 0
 *  out            device, bf16 [nnz_qo][Hq][head_dim], written
 *  lse_out        device, fp32 [nnz_qo][Hq] natural-log LSE, or NULL
 *  workspace      device scratch of at least
 *                 daa_batch_attention_workspace_size(...) bytes (NULL if 0);
 *                 the call owns it until the enqueued work completes
 *  stream         cudaStream_t
 * Errors: DAA_ERR_* on the host before any launch; DAA_ERR_CUDA on a failed
 * launch or copy.
 */
daa_status daa_batch_attention(const void* q, const void* kv_pages, const int32_t* qo_indptr,
                               const int32_t* kv_indptr, const int32_t* page_indices,
                               const int32_t* last_page_len, const int32_t* h_qo_indptr,
                               const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
                               int32_t batch, int32_t causal, float sm_scale, void* out,
                               float* lse_out, void* workspace, size_t workspace_bytes,
                               daa_dims dims, void* stream);

/*
 * daa_kv_append followed by daa_batch_attention in one call, on one plan
 * ("Disaggregated prefill and decode", section "KV Messenger": entries are
 * valid after the append and before attention; "Chunked prefill", #correctness:
 * each chunk's new k, v are appended and attended to in the same step).
 *
 * The new tokens of request r are its query rows: k_new, v_new are
 * [nnz_qo][Hkv][head_dim] with the row layout of q (append_indptr = qo_indptr,
 * nnz_new = h_qo_indptr[batch]).  The result -- pool bytes, out, lse_out -- is
 * exactly that of the two calls in sequence on the same stream.  What differs
 * is the schedule: the plan copy is issued before the append, and the
 * attention kernels are launched behind the append as programmatic dependent
 * launches, so their set-up and the key splits that read only cached rows
 * overlap the append (the CTAs that read an appended row wait for it).
 *
 * The append of long prefill chunks is fused into their attention ("Chunked
 * prefill", #io-overhead: the chunk's K/V are written to the cache once).  A
 * request with more new tokens than two 128-row tiles of packed (token, query
 * head) rows hold (qo_len > 2 * (128 / (Hq / Hkv))) runs on a prefill kernel
 * (CTA pairs for head_dim 128, one CTA per two tiles for head_dim 64).  Its
 * key tiles that lie wholly in the chunk -- keys from the first multiple of 128
 * at or after kv_len - qo_len -- are read by that kernel straight from k_new /
 * v_new, and written into their pages by it from the same tiles; the append
 * kernel writes only the other rows.  The pages end up with exactly the bytes
 * the plain append writes.
 * daa_set_prefill_append_fusion(0) turns this off (every row then goes
 * through the append kernel and is read back from the pages).
 *
 *  k_new, v_new   device, bf16 [nnz_qo][Hkv][head_dim]
 *  kv_pages       device, bf16 pool, written (the appended rows) and read
 *  other arguments as daa_batch_attention, with the same workspace size
 *  (daa_batch_attention_workspace_size).
 * Errors: those of both calls, all checked on the host before anything is
 * enqueued.
 */
daa_status daa_append_attention(const void* k_new, const void* v_new, const void* q,
                                void* kv_pages, const int32_t* qo_indptr,
                                const int32_t* kv_indptr, const int32_t* page_indices,
                                const int32_t* last_page_len, const int32_t* h_qo_indptr,
                                const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
                                int32_t batch, int32_t causal, float sm_scale, void* out,
                                float* lse_out, void* workspace, size_t workspace_bytes,
                                daa_dims dims, void* stream);

/*
 * One serving step fed from host memory: upload the step's inputs, run
 * daa_append_attention on them, read the output back -- one call per step,
 * every copy and kernel asynchronous, so consecutive steps overlap when the
 * caller alternates two sets of device buffers.  It feeds the attention and
 * the append as a serving loop does ("Accelerating Sonar through
 * speculation", section "Inference with speculative decoding": a step's input
 * tokens and KV page information are packed into one buffer on the host and
 * the metadata is then copied to GPU memory).
 *
 * Inputs: one pinned host buffer `h_inputs` of layout->total bytes holding,
 * at the byte offsets of `layout`, the step's qo_indptr, kv_indptr,
 * page_indices, last_page_len (int32, 4-byte aligned offsets) and q, k_new,
 * v_new (bf16, 16-byte aligned offsets), with the shapes of
 * daa_append_attention.  The call reads the page table from this host buffer
 * to plan (no device sync), copies the whole buffer to `d_inputs` (device,
 * 256-byte aligned, layout->total bytes) on the upload stream, runs the append
 * and the attention on the compute stream from the device copy, and copies
 * out ([nnz_qo][Hq][head_dim] bf16 in `d_out`) back to `h_out` (pinned host)
 * on the download stream.  `workspace` is that of daa_append_attention.
 *
 * Ordering (all cudaEvent_t / cudaStream_t, created by the caller):
 *   upload:   waits for streams->inputs_free (if not NULL: the previous step
 *             that read this d_inputs has finished computing), copies, records
 *             streams->uploaded;
 *   compute:  waits for uploaded and for streams->out_free (if not NULL: the
 *             previous read-back of this d_out has finished), runs the kernels,
 *             records streams->computed;
 *   download: waits for computed, copies, records streams->downloaded.
 * h_inputs must not change until `uploaded` has completed; h_out holds the
 * output once `downloaded` has completed.  A batch with no query rows copies
 * nothing and only records the three events.
 *
 * Errors: those of daa_append_attention, plus DAA_ERR_INVALID_ARG for a NULL
 * buffer, layout, stream set or event, DAA_ERR_ALIGNMENT for misaligned
 * offsets or d_inputs, DAA_ERR_SHAPE when a section runs past layout->total.
 * All are found before anything is enqueued.
 */
typedef struct {
  size_t qo_indptr, kv_indptr, page_indices, last_page_len; /* int32 sections */
  size_t q, k_new, v_new;                                   /* bf16 sections */
  size_t total;                                             /* bytes uploaded */
} daa_step_layout;

typedef struct {
  void* upload_stream;   /* cudaStream_t */
  void* compute_stream;  /* cudaStream_t */
  void* download_stream; /* cudaStream_t */
  void* uploaded;        /* cudaEvent_t, recorded by the call */
  void* computed;        /* cudaEvent_t, recorded by the call */
  void* downloaded;      /* cudaEvent_t, recorded by the call */
  void* inputs_free;     /* cudaEvent_t waited for, or NULL */
  void* out_free;        /* cudaEvent_t waited for, or NULL */
} daa_step_streams;

daa_status daa_append_attention_host(const void* h_inputs, void* d_inputs,
                                     const daa_step_layout* layout, int32_t batch, int32_t causal,
                                     float sm_scale, void* kv_pages, void* d_out, void* h_out,
                                     void* workspace, size_t workspace_bytes, daa_dims dims,
                                     const daa_step_streams* streams);

/*
 * Switch of the fused prefill append of daa_append_attention,
 * daa_append_attention_shared_prefix and daa_append_attention_run ("Chunked
 * prefill", #io-overhead; see daa_append_attention): 1 (the default) lets the
 * prefill kernels read their chunk's own key tiles from k_new / v_new and
 * write them into the pages; 0 appends every row with the append kernel.
 * Results (pool bytes, out, lse_out) are identical; only the work differs.
 * Process-wide; takes effect for calls made after it returns.
 * Errors: DAA_ERR_INVALID_ARG for a value other than 0 or 1.
 */
daa_status daa_set_prefill_append_fusion(int32_t enable);

/* The current setting of daa_set_prefill_append_fusion (0 or 1). */
int32_t daa_prefill_append_fusion(void);

/*
 * Mixed-batch paged attention under draft-tree masks, for verifying the draft
 * tokens of speculative decoding ("Accelerating Sonar through speculation"
 * (Perplexity), section EAGLE: a tree of draft tokens is checked by the target
 * model in one pass under a custom attention mask; each draft token is scored
 * against the accepted prefix and its own branch of the tree).
 *
 * Computes daa_batch_attention with causal = 1, except that new token i of a
 * request sees, among the request's new tokens, only itself and the earlier
 * ones its mask row selects.  With pos0 = kv_len - qo_len (the key of new token
 * 0), token i's key set is
 *   J = {j < pos0}  U  {pos0 + i}  U  {pos0 + t : t < i, bit t of its row set}.
 * Mask rows: tree_mask is uint32 [nnz_qo][mask_words] on the device, one row
 * per query row (the row layout of q); bit t of a row is word t / 32, bit
 * t % 32 (t counts the request's new tokens from 0).  Bits t >= i are ignored:
 * a token always sees itself and never a later new token, so a row of all
 * earlier bits set is plain causal attention and every request of a mixed
 * batch can be given that way.  For a draft tree whose nodes are numbered so
 * that parents precede children, row i holds the bits of i's ancestors.
 * Requests with qo_len = 1 are unaffected (their key set is the same).
 *
 *  tree_mask      device, uint32 [nnz_qo][mask_words], 4-byte aligned
 *  mask_words     words per row; every request needs qo_len <= 32 * mask_words
 *  other arguments as daa_batch_attention (no `causal`: the rule is causal),
 *  with the same workspace size (daa_batch_attention_workspace_size).
 * Errors: those of daa_batch_attention; DAA_ERR_INVALID_ARG for a NULL mask or
 * mask_words < 1, DAA_ERR_SHAPE when a request has more than 32 * mask_words
 * new tokens, DAA_ERR_ALIGNMENT for a misaligned mask.  Only tiles of keys
 * that hold earlier new tokens of a row evaluate the mask; the cached prefix
 * streams exactly as in daa_batch_attention.
 */
daa_status daa_batch_attention_tree(const void* q, const void* kv_pages,
                                    const int32_t* qo_indptr, const int32_t* kv_indptr,
                                    const int32_t* page_indices, const int32_t* last_page_len,
                                    const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                    const int32_t* h_last_page_len, int32_t batch,
                                    const uint32_t* tree_mask, int32_t mask_words, float sm_scale,
                                    void* out, float* lse_out, void* workspace,
                                    size_t workspace_bytes, daa_dims dims, void* stream);

/*
 * Mixed-batch paged attention for requests that share a cached prefix, with
 * that prefix's keys read once for the whole group ("Chunked prefill"
 * (k4i.top), #prefix-cache-interaction: the cached blocks of a prefix hit are
 * skipped, only the suffix is computed; #correctness: attention over a key set
 * is the softmax_merge of attentions over a partition of it).
 *
 * The result -- out, lse_out -- is that of daa_batch_attention on the same
 * arguments (equal up to fp32 rounding order).  What differs is the schedule.
 * Within a group, every run of consecutive decode, verify and short requests
 * (1 <= qo_len <= two 128-row Q tiles of packed (token, head) rows) with two
 * or more such members has the query rows of all its members (one per new
 * token and query head) attended to the group's shared keys in one pass, the
 * rows of several requests packed into the same 128-row tensor-core tiles.
 * Only whole 128-key tiles of the prefix are shared; the rest of it is read
 * per request.  Each member's own items then cover only the keys after the
 * shared part, and softmax_merge combines the two parts per row.  K/V bytes of
 * the shared prefix are read once per run instead of once per request.
 * Prefill requests of a group (and runs of one member) attend the prefix in
 * their own items: their Q tiles are full already.
 *
 * Groups (host arrays): group i is requests [h_prefix_indptr[i],
 * h_prefix_indptr[i+1]) -- consecutive requests, groups in request order --
 * whose first h_prefix_len[i] keys are the same tokens in the same pages: for
 * every request r of the group, page_indices[kv_indptr[r] + p] is the same
 * page for every p < h_prefix_len[i] / page_size.  The library cannot check
 * this (page ids live only on the device); a group that breaks it gives wrong
 * outputs, never an access outside the pool.  h_prefix_len[i] must be a
 * multiple of page_size and cached: at most kv_len_r - qo_len_r for every
 * request of the group.  Requests in no group are planned as in
 * daa_batch_attention; a request between two groups may sit in a group of
 * prefix length 0.
 *
 *  h_prefix_indptr  host int32 [n_groups + 1], non-decreasing, in [0, batch]
 *  h_prefix_len     host int32 [n_groups]
 *  n_groups         >= 0 (0: exactly daa_batch_attention's plan)
 *  workspace        at least daa_batch_attention_shared_prefix_workspace_size(...)
 *                   bytes with the same groups
 *  other arguments as daa_batch_attention / daa_append_attention.
 * Errors: those of daa_batch_attention; DAA_ERR_INVALID_ARG for n_groups < 0
 * or NULL group arrays with n_groups > 0; DAA_ERR_SHAPE for a group outside
 * [0, batch], a decreasing indptr, a prefix length that is negative, not a
 * multiple of page_size, or longer than some member's cached keys.
 */
size_t daa_batch_attention_shared_prefix_workspace_size(
    const int32_t* h_qo_indptr, const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
    int32_t batch, const int32_t* h_prefix_indptr, const int32_t* h_prefix_len, int32_t n_groups,
    daa_dims dims, daa_status* status);

daa_status daa_batch_attention_shared_prefix(
    const void* q, const void* kv_pages, const int32_t* qo_indptr, const int32_t* kv_indptr,
    const int32_t* page_indices, const int32_t* last_page_len, const int32_t* h_qo_indptr,
    const int32_t* h_kv_indptr, const int32_t* h_last_page_len, int32_t batch,
    const int32_t* h_prefix_indptr, const int32_t* h_prefix_len, int32_t n_groups, int32_t causal,
    float sm_scale, void* out, float* lse_out, void* workspace, size_t workspace_bytes,
    daa_dims dims, void* stream);

/* daa_append_attention (append, then attention, in one call) with the prefix
 * groups of daa_batch_attention_shared_prefix. */
daa_status daa_append_attention_shared_prefix(
    const void* k_new, const void* v_new, const void* q, void* kv_pages, const int32_t* qo_indptr,
    const int32_t* kv_indptr, const int32_t* page_indices, const int32_t* last_page_len,
    const int32_t* h_qo_indptr, const int32_t* h_kv_indptr, const int32_t* h_last_page_len,
    int32_t batch, const int32_t* h_prefix_indptr, const int32_t* h_prefix_len, int32_t n_groups,
    int32_t causal, float sm_scale, void* out, float* lse_out, void* workspace,
    size_t workspace_bytes, daa_dims dims, void* stream);

/*
 * Plan once, run many times.  The plan of a batch -- how its requests are cut
 * into work items ("Disaggregated prefill and decode", "Prefill vs decode
 * performance": attention splits over requests and over kv_len) -- depends
 * only on the page table's lengths.  In a model, every attention layer of a
 * step reads the same table, so one plan serves all of them.
 * daa_batch_attention_plan builds it on the host and copies it into the head
 * of the workspace (one cudaMemcpyAsync on `stream`).  daa_batch_attention_run
 * and daa_append_attention_run then launch only the kernels.  The outputs are
 * bit-identical to daa_batch_attention / daa_append_attention on the same
 * arguments, with and without prefix groups.
 *
 * daa_plan_info is plain data: the workspace layout and the shapes the plan
 * was made for.  The plan stays valid while the workspace is not written by
 * anything else (another plan, or a call that plans for itself) and the page
 * table's lengths (qo_indptr, kv_indptr, last_page_len) are unchanged.  The
 * pages themselves and q, k_new, v_new may change between runs.  Runs of one
 * plan must not overlap on the GPU: they share the workspace's partials.
 *
 *  plan: the host arrays of daa_batch_attention (plus the prefix groups of
 *        daa_batch_attention_shared_prefix; n_groups = 0 for none), the
 *        workspace (at least the matching workspace-size query's bytes; may be
 *        NULL when that size is 0), `info` (written), `stream`.
 *  run:  the device arrays of daa_batch_attention, `info`, then causal,
 *        sm_scale, out, lse_out, the workspace, the dims the plan was made
 *        for, `stream`.  The page table passed must be the one planned.
 * Errors: plan -- those of the size query; DAA_ERR_INVALID_ARG for a NULL info;
 * DAA_ERR_WORKSPACE / DAA_ERR_ALIGNMENT for the workspace; DAA_ERR_CUDA if the
 * copy fails.  run -- DAA_ERR_INVALID_ARG for an info that no plan call wrote or
 * whose dims differ from `dims`; otherwise those of daa_batch_attention.
 */
typedef struct {
  int64_t words[24];
} daa_plan_info;

daa_status daa_batch_attention_plan(const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                    const int32_t* h_last_page_len, int32_t batch,
                                    const int32_t* h_prefix_indptr, const int32_t* h_prefix_len,
                                    int32_t n_groups, daa_dims dims, void* workspace,
                                    size_t workspace_bytes, daa_plan_info* info, void* stream);

daa_status daa_batch_attention_run(const void* q, const void* kv_pages, const int32_t* qo_indptr,
                                   const int32_t* kv_indptr, const int32_t* page_indices,
                                   const int32_t* last_page_len, const daa_plan_info* info,
                                   int32_t causal, float sm_scale, void* out, float* lse_out,
                                   void* workspace, size_t workspace_bytes, daa_dims dims,
                                   void* stream);

/* daa_append_attention on a plan: the append of k_new, v_new, then the
 * attention kernels launched behind it (as daa_append_attention). */
daa_status daa_append_attention_run(const void* k_new, const void* v_new, const void* q,
                                    void* kv_pages, const int32_t* qo_indptr,
                                    const int32_t* kv_indptr, const int32_t* page_indices,
                                    const int32_t* last_page_len, const daa_plan_info* info,
                                    int32_t causal, float sm_scale, void* out, float* lse_out,
                                    void* workspace, size_t workspace_bytes, daa_dims dims,
                                    void* stream);

/* Size of the device scratch array behind daa_batch_attention_noalloc (48 MiB). */
#define DAA_NOALLOC_SCRATCH_BYTES (48u * 1024u * 1024u)

/*
 * daa_batch_attention for callers that cannot allocate device memory.  The
 * pages describe no such call; it has no counterpart there.
 *
 * Who needs it: a caller with no device allocator at the call site -- e.g. a
 * serving engine that has handed all free HBM to its KV page pool and keeps no
 * allocator to carve a workspace from, code on a latency-critical path where a
 * cudaMalloc/cudaFree could synchronise the device, or a foreign-language host
 * with no binding to a CUDA allocator.  It computes exactly what
 * daa_batch_attention computes, with the same arguments minus the workspace.
 *
 * Scratch: the work plan and the split-KV partial outputs live in one
 * file-scope __device__ array of DAA_NOALLOC_SCRATCH_BYTES bytes, which every
 * GPU that loads the library holds until the process exits.  The call makes no
 * cudaMalloc/cudaFree and no other allocation (device or host heap); its plan
 * is built in fixed-size static host buffers.  A batch whose scratch would
 * exceed the array, or that needs more than 16384 decode splits, 16384 split
 * requests or 16384 prefill tiles, is rejected with DAA_ERR_WORKSPACE before
 * anything is enqueued.
 *
 * Set-up: the first call on each device (with that device current) looks up
 * the array's device address with cudaGetSymbolAddress and caches it.  The
 * cached address belongs to the device context it was looked up in: after
 * cudaDeviceReset (or anything else that destroys the primary context) it is
 * stale, so do not call this entry point again in a process that has reset the
 * device.
 *
 * Sharing: every call, on every stream and host thread, uses the same array,
 * which keeps the last call's contents.  Nothing in it has to start at zero --
 * every byte a call reads was written earlier in that same call -- but calls
 * whose GPU work overlaps (concurrent streams, or calls from several host
 * threads without ordering between their streams) race on the scratch and
 * produce wrong results.  Serialise them, e.g. by issuing all such calls on one
 * stream.  Host-side calls are serialised by an internal mutex.
 *
 * Arguments, layouts and the other errors are those of daa_batch_attention.
 */
daa_status daa_batch_attention_noalloc(const void* q, const void* kv_pages,
                                       const int32_t* qo_indptr, const int32_t* kv_indptr,
                                       const int32_t* page_indices, const int32_t* last_page_len,
                                       const int32_t* h_qo_indptr, const int32_t* h_kv_indptr,
                                       const int32_t* h_last_page_len, int32_t batch,
                                       int32_t causal, float sm_scale, void* out, float* lse_out,
                                       daa_dims dims, void* stream);

/*
 * Reads the device error word of the current device into *code (0 = none, 1 =
 * page id out of range, 2 = a bounded wait timed out, 3 = inconsistent request
 * lengths) and clears it when `reset` is non-zero.  Synchronises the device.
 * Kernels never trap on these: a page id outside the pool is replaced by page
 * 0 (or, in the append, the row is skipped), so the outputs of that call are
 * undefined but the context stays usable.  Every wait inside a kernel is
 * bounded (1 s); one that runs out records code 2 and the kernel runs on to its
 * exit.  While the word holds code 2, waits of later launches give up at once,
 * so clear it (reset = 1) after a timeout has been reported.
 */
daa_status daa_device_error(int32_t* code, int32_t reset);

/*
 * Health check of the bounded waits (no counterpart on the pages): launches a
 * one-thread kernel on the legacy default stream that waits on an mbarrier
 * phase nothing completes, with the same bounded wait the attention kernels
 * use, and returns after that wait has given up (about 1 s).  *gave_up = 1 when
 * the wait ended by its limit; the device error word then holds code 2 (read
 * and clear it with daa_device_error).  Synchronises the device.
 */
daa_status daa_selftest_bounded_wait(int32_t* gave_up);

/*
 * Per-kernel timing with CUDA events.  While enabled, every kernel the library
 * launches is bracketed by two events on its stream (up to `capacity` launches
 * are kept, older ones dropped).  daa_trace_read synchronises on the recorded
 * events and copies out up to `max_records` (kernel id, milliseconds) pairs in
 * launch order, returning how many were written, then clears the record.
 * Kernel ids: 1 kv_append, 2 decode split-KV (CUDA cores), 3 softmax_merge,
 * 4 tensor-core prefill, 5 tensor-core decode split-KV (decode and verify
 * items), 6 tensor-core short multi-token items (head_dim 128: requests whose
 * rows fit two 128-row Q tiles).
 */
daa_status daa_trace_enable(int32_t capacity);
daa_status daa_trace_disable(void);
int32_t daa_trace_read(int32_t* kernel_ids, float* milliseconds, int32_t max_records);

#ifdef __cplusplus
}
#endif

#endif /* DAA_H_ */
