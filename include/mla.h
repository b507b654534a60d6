/*
 * mla.h -- C ABI of the multi-head latent attention (MLA) decode library.
 *
 * The library implements the inference path that the MLA pages describe:
 * cache only the latent c_s = W^DKV h_s and the rotated decoupled key
 * R_s k^R_s of every token, fold W^UK into the query, attend in latent
 * space, and apply W^UV and W^O once to the attended latent.
 *   - "Multi-head latent attention (MLA)" (ai-knowledge-tree, pillar E3),
 *     sections 2 (down-projection, up-projections, folding) and 3
 *     (decoupled RoPE key; score = content term + rotary term).
 *   - "Attention, Part 2: MQA, GQA and MLA" (ishwarj.com), "The MLA
 *     equations", "The trick that makes it fast: never rebuild at all"
 *     (absorbed inference path), "Why position needs its own key".
 *   - "How DeepSeek Rewrote the Transformer" (zhichai.net), "Absorbed
 *     projections" (the value is the first d_c numbers of the key row).
 * For prompts and long chunks it also rebuilds the per-head keys and values
 * from the cached latent ("The MLA equations") and attends over them
 * (mla_prefill_kv, mla_prefill_attention): the same result, fewer flops
 * once a chunk has more than a few dozen tokens.
 *
 * Conventions shared by every call:
 *   - Every array pointer is a DEVICE pointer (cudaMalloc'd or torch
 *     memory) owned by the caller, row-major and contiguous, 16-byte
 *     aligned.  The library allocates no device memory at run time (the
 *     scratch of mla_decode_paged_noalloc is a static array of the library
 *     image).
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on it and returns; results are
 *     ready when the stream reaches that point.
 *   - Calls return an mla_status.  Host-side argument checks run before any
 *     launch; when one fails nothing is launched.  Conditions that only the
 *     device can see (a block id outside the pool, a sequence length outside
 *     [T_q, max_blocks_per_seq * 64], a wait that ran out) are recorded in a
 *     per-device error word; mla_check_status() reports and clears it.
 *     Affected output rows are written as zeros, never read out of bounds.
 *   - dtype codes: MLA_F32 (IEEE float) and MLA_BF16 (bfloat16).  Casts to
 *     bfloat16 round to nearest even.  Accumulation is always in float.
 *   - Cache layout ("paged pool"): kv_cache is [num_blocks, 64, D] with
 *     D = d_c + d_r; row r of block k holds one token's [c ; R k^R].
 *     block_table is int32 [B, max_blocks_per_seq]; token s of sequence b
 *     lives in block block_table[b, s / 64], row s % 64.  Entries past a
 *     sequence's last block are never read.
 *   - Thread safety: calls keep no per-call state on the host or device
 *     besides the error word, and may be made from several host threads.
 */
#ifndef MLA_H
#define MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define MLA_OK              0
#define MLA_ERR_INVALID_ARG 1  /* host check failed; nothing launched        */
#define MLA_ERR_UNSUPPORTED 2  /* valid but unsupported dims/dtype combination */
#define MLA_ERR_CUDA        3  /* a CUDA call failed; see mla_last_cuda_error */
#define MLA_ERR_WORKSPACE   4  /* workspace NULL or smaller than required     */
#define MLA_ERR_TIMEOUT     5  /* a device wait gave up (bounded spin)        */
#define MLA_ERR_BAD_INDEX   6  /* device saw a bad block id or sequence length */
#define MLA_ERR_BAD_RECORD  7  /* the merge found split records that no partial
                                  pass wrote (a partial pass that gave up, or
                                  mla_decode_combine without its partial pass) */

/* dtype codes */
#define MLA_F32  0
#define MLA_BF16 1

/* tokens per cache block; the only supported page size */
#define MLA_PAGE_SIZE 64

/*
 * mla_cache_append -- write new tokens' rows into the paged cache.
 *
 * For i < n_new, with b = seq_ids[i], s = positions[i]:
 *   row (b, s) <- [ c[i, 0:d_c] ; RoPE_s(k_rope[i, 0:d_r]) ]
 * i.e. the cached row of "The MLA equations" (c = W_dkv x, kr = rope(W_kr x))
 * and section 3 of the ai-knowledge-tree page: the latent is stored as is,
 * only the decoupled key is rotated.  RoPE rotates adjacent pairs
 * (x[2j], x[2j+1]) by s * base^(-2j/d_r) (RoFormer form); the angle and the
 * rotation are evaluated in double precision, then cast to cache_dtype.
 *
 *   c          [n_new, d_c]  dtype_in        latent of each new token
 *   k_rope     [n_new, d_r]  dtype_in        UNrotated decoupled key
 *   seq_ids    [n_new]       int32           sequence of each token (< B)
 *   positions  [n_new]       int32           token position s within it
 *   block_table[B, max_blocks_per_seq] int32
 *   kv_cache   [num_blocks, 64, d_c + d_r]  cache_dtype, written in place
 * d_r must be even.  Host errors: NULL pointers, n_new < 0, B < 1, d_c < 1,
 * d_r < 0 or odd, page_size != 64.  Device errors (MLA_ERR_BAD_INDEX):
 * seq_ids[i] outside [0, B), position < 0 or >= max_blocks_per_seq * 64,
 * block id outside [0, num_blocks); such rows are skipped.  n_new == 0
 * launches nothing.
 */
int mla_cache_append(const void* c, const void* k_rope, int dtype_in,
                     const int32_t* seq_ids, const int32_t* positions, int n_new,
                     const int32_t* block_table, int B, int max_blocks_per_seq,
                     void* kv_cache, int cache_dtype, int num_blocks, int page_size,
                     int d_c, int d_r, float rope_base, void* stream);

/*
 * mla_absorb_query -- fold W^UK into the query and rotate the rotary query.
 *
 *   q_lat[n, h, 0:d_c]      = W^UK_h^T q_nope[n, h, :]      (float accumulate)
 *   q_lat[n, h, d_c:d_c+d_r] = RoPE_{positions[n]}(q_rope[n, h, :])
 * where W^UK_h is rows h*d_h .. (h+1)*d_h-1 of w_uk [H*d_h, d_c]
 * ("The trick that makes it fast": the new query is multiplied by the
 * transposed per-head key up-projection once, and the result is compared
 * with the cached latents directly.)
 *
 *   q_nope [N, H, d_h]   dtype        content query W^Q h
 *   q_rope [N, H, d_r]   dtype        UNrotated rotary query W^QR h
 *   positions [N]        int32        position of each query token
 *   w_uk   [H*d_h, d_c]  dtype
 *   q_lat  [N, H, d_c + d_r]  q_dtype (output)
 * Host errors: NULL pointers, non-positive dims, odd d_r, N < 0.
 */
int mla_absorb_query(const void* q_nope, const void* q_rope, const int32_t* positions,
                     const void* w_uk, int dtype, int N, int H, int d_h, int d_c,
                     int d_r, float rope_base, void* q_lat, int q_dtype, void* stream);

/*
 * mla_decode_workspace_size -- bytes of scratch mla_decode_paged needs for
 * the split-KV partial results on the CURRENT device (it depends on the
 * device's SM count and on which kernel the shape selects).  Returns 0 for
 * invalid dims.
 */
size_t mla_decode_workspace_size(int B, int T_q, int H, int d_c, int d_r, int dtype);

/*
 * mla_decode_paged -- latent-space attention of T_q new query tokens per
 * sequence against that sequence's paged cache (the decode hot path).
 *
 * For sequence b with L_b = seqlens[b] cached rows (INCLUDING the T_q new
 * tokens, which the caller appended first), query token t at position
 * L_b - T_q + t, head h, and row C_s = cache row of token s:
 *   z_s   = softmax_scale * q_lat[b,t,h,:] . C_s          (content + rotary)
 *   p     = softmax over visible s (s <= L_b - T_q + t if causal, else all)
 *   o_lat[b,t,h,:] = sum_s p_s C_s[0:d_c]                 (V = first d_c)
 *   lse[b,t,h]     = natural log of sum_s exp(z_s)
 * ("The trick that makes it fast": scores and the softmax-weighted sum are
 * taken over the cached latents themselves; section 3 of the
 * ai-knowledge-tree page: score = content term + positional term.)
 *
 *   q_lat    [B, T_q, H, D]              dtype (MLA_BF16 or MLA_F32)
 *   kv_cache [num_blocks, 64, D]         same dtype
 *   block_table [B, max_blocks_per_seq]  int32
 *   seqlens  [B]                         int32, device
 *   o_lat    [B, T_q, H, d_c]            float (output)
 *   lse      [B, T_q, H]                 float (output) or NULL
 *   workspace, workspace_bytes           >= mla_decode_workspace_size(...)
 * Long or ragged batches are split into page ranges processed in parallel
 * (partial softmax results in the workspace) and merged by a log-sum-exp
 * combine kernel.  The bf16 shape d_c = 512, d_r = 64 runs the tensor-core
 * (tcgen05/TMEM) kernel, any H*T_q (rows in groups of up to 128, see
 * mla_decode_row_groups); every other shape a CUDA-core kernel.
 * Host errors: NULL pointers, B/T_q/H < 1, d_c < 1 or > 512, d_r < 0,
 * D > 1024, page_size != 64, max_blocks_per_seq < 1, num_blocks < 1.
 * Device errors (MLA_ERR_BAD_INDEX): L_b < T_q or L_b > 64*max_blocks_per_seq
 * (that sequence's outputs are zero), a block id outside [0, num_blocks)
 * (that page is treated as absent).  MLA_ERR_TIMEOUT: a bounded wait in the
 * tensor-core kernel gave up; its outputs are then undefined but the context
 * stays usable.
 */
int mla_decode_paged(const void* q_lat, const void* kv_cache, int dtype,
                     const int32_t* block_table, const int32_t* seqlens,
                     int B, int T_q, int H, int d_c, int d_r, int page_size,
                     int max_blocks_per_seq, int num_blocks,
                     float softmax_scale, int causal,
                     void* workspace, size_t workspace_bytes,
                     float* o_lat, float* lse, void* stream);

/*
 * mla_decode_paged_noalloc -- mla_decode_paged without a caller workspace.
 * (An engineering variant: the pages have no counterpart of it.)
 *
 * For callers that have no way to get device memory at the point of the
 * call: a plain C or C++ host that holds only the pointers it was handed and
 * has no allocator of its own, or a serving process that gave all free device
 * memory to its cache pool at start-up, so that a workspace would have to
 * come from cudaMalloc, which can fail there and stalls the whole device.
 *
 * Same arguments and results as mla_decode_paged, minus workspace and
 * workspace_bytes.  The split workspace lives in a file-scope device array
 * of this library, 64 MiB per device: shapes whose
 * mla_decode_workspace_size(...) exceeds 64 MiB are rejected with
 * MLA_ERR_WORKSPACE (nothing launched).  The call allocates nothing (no
 * cudaMalloc, no library that allocates); nothing in the scratch has to
 * start at zero, because the partial pass writes every record the merge
 * reads within the same call.
 * The scratch is shared by all calls on a device: two calls that may overlap
 * in time (different streams, or different host threads) race on it; issue
 * them on one stream.  The first call on a device looks the scratch address
 * up (cudaGetSymbolAddress; it may load the module), so make that first call
 * before any stream capture begins.
 */
int mla_decode_paged_noalloc(const void* q_lat, const void* kv_cache, int dtype,
                             const int32_t* block_table, const int32_t* seqlens,
                             int B, int T_q, int H, int d_c, int d_r, int page_size,
                             int max_blocks_per_seq, int num_blocks,
                             float softmax_scale, int causal,
                             float* o_lat, float* lse, void* stream);

/*
 * mla_decode_paged_partial / mla_decode_combine -- the two launches that
 * make up mla_decode_paged, exposed separately (same arguments) so that a
 * caller can time, overlap or reorder them.  mla_decode_paged_partial runs
 * the split-KV attention pass: sequences handled by a single worker get
 * their final o_lat/lse, the others leave partial results in the workspace.
 * mla_decode_combine then merges the partial results (log-sum-exp
 * weighting) and writes zeros for sequences of invalid length.  Calling the
 * partial pass, then the combine, on one stream, with unchanged arguments
 * and workspace, is exactly mla_decode_paged.
 */
int mla_decode_paged_partial(const void* q_lat, const void* kv_cache, int dtype,
                             const int32_t* block_table, const int32_t* seqlens,
                             int B, int T_q, int H, int d_c, int d_r, int page_size,
                             int max_blocks_per_seq, int num_blocks,
                             float softmax_scale, int causal,
                             void* workspace, size_t workspace_bytes,
                             float* o_lat, float* lse, void* stream);
int mla_decode_combine(const void* q_lat, const void* kv_cache, int dtype,
                       const int32_t* block_table, const int32_t* seqlens,
                       int B, int T_q, int H, int d_c, int d_r, int page_size,
                       int max_blocks_per_seq, int num_blocks,
                       float softmax_scale, int causal,
                       void* workspace, size_t workspace_bytes,
                       float* o_lat, float* lse, void* stream);

/*
 * mla_decode_step -- one decode step of the absorbed MLA layer in one call:
 * the chain "The MLA equations" / "The trick that makes it fast" describe for
 * new tokens (cache the latent and the rotated decoupled key, absorb W^UK
 * into the query, attend in latent space).
 *
 * For sequence b with L_b = seqlens[b] cached rows INCLUDING its T_q new
 * tokens, new token t sits at position s = L_b - T_q + t and has flat index
 * i = b * T_q + t.  In stream order:
 *   1. q_lat[b, t, h] = [ W^UK_h^T q_nope[i, h] ; RoPE_s(q_rope[i, h]) ]
 *      (as mla_absorb_query, stored in the cache dtype in the workspace);
 *   2. cache row (b, s) <- [ c_new[i] ; RoPE_s(k_rope_new[i]) ]
 *      (as mla_cache_append);
 *   3. o_lat, lse = mla_decode_paged over the cache with q_lat.
 * The cache append is launched as a programmatic dependent of the query
 * absorption (its launch overlaps the absorption's tail).
 *
 *   q_nope [B*T_q, H, d_h], q_rope [B*T_q, H, d_r], w_uk [H*d_h, d_c],
 *   c_new [B*T_q, d_c], k_rope_new [B*T_q, d_r]: all in `dtype`, the cache's
 *   dtype; the other arguments as for mla_decode_paged.
 *   workspace: >= mla_decode_step_workspace_size(...) bytes, 256-byte aligned
 *   (q_lat first, then the decode's split workspace).
 * Host errors: those of the three calls; MLA_ERR_WORKSPACE for a small or
 * misaligned workspace.  Device errors: as the three calls (a position
 * outside the block table, a bad block id, an invalid length).
 */
size_t mla_decode_step_workspace_size(int B, int T_q, int H, int d_c, int d_r, int dtype);
int mla_decode_step(const void* q_nope, const void* q_rope, const void* w_uk, int d_h,
                    const void* c_new, const void* k_rope_new, void* kv_cache, int dtype,
                    const int32_t* block_table, const int32_t* seqlens,
                    int B, int T_q, int H, int d_c, int d_r, int page_size,
                    int max_blocks_per_seq, int num_blocks, float softmax_scale, int causal,
                    float rope_base, void* workspace, size_t workspace_bytes,
                    float* o_lat, float* lse, void* stream);

/*
 * mla_absorb_output -- apply W^UV per head, then W^O, to the attended latent.
 *
 *   o[n, h, v] = sum_c w_uv[h*d_h + v, c] * o_lat[n, h, c]
 *   out[n, j]  = sum_{h,v} w_o[j, h*d_h + v] * o[n, h, v]
 * ("The trick that makes it fast": the value up-projection is applied once,
 * to the attended latent, followed by the output projection.)
 *
 *   o_lat [N, H, d_c] float;  w_uv [H*d_h, d_c] dtype;  w_o [d, H*d_h] dtype
 *   out   [N, d] float (output)
 * bf16 weights with d_c % 64 == 0, d_h % 8 == 0, d % 4 == 0 and 16-byte
 * aligned pointers run on the tensor cores: o_lat and o enter as bf16 value
 * plus bf16 remainder (about fp32 accuracy), K of the second product is split
 * across the grid and the partial sums are added in a fixed order; the call
 * allocates and frees a scratch buffer in stream order on `stream`.  Other
 * shapes and fp32 weights run on CUDA cores.
 * Host errors: NULL pointers, non-positive dims, H*d_h > 32768.  Device
 * errors: MLA_ERR_TIMEOUT (tensor-core path).
 */
int mla_absorb_output(const float* o_lat, const void* w_uv, const void* w_o, int dtype,
                      int N, int H, int d_h, int d_c, int d, float* out, void* stream);

/*
 * mla_merge_output_weights -- fold W^UV into W^O: one d x d_c matrix per head
 * ("How DeepSeek Rewrote the Transformer", the absorbed inference path: the
 * value up-projection can be merged into the output projection).
 *
 *   w_merged[j, h*d_c + c] = sum_v w_o[j, h*d_h + v] * w_uv[h*d_h + v, c]
 *
 *   w_uv [H*d_h, d_c] bf16;  w_o [d, H*d_h] bf16
 *   w_merged [d, H*d_c] bf16 (output; fp32 sums rounded once)
 * A one-time weight transform: it allocates and frees a scratch copy of w_uv
 * (H*d_h*d_c*2 bytes) in stream order on `stream`.
 * Host errors: MLA_ERR_INVALID_ARG (non-positive dims, d_c % 8 or d % 4 not
 * zero, NULL or not 16-byte aligned pointers); MLA_ERR_UNSUPPORTED for
 * dtype != MLA_BF16 or d_h % 64 != 0.  Device errors: MLA_ERR_TIMEOUT (a
 * bounded wait gave up; w_merged then holds no result).  Asynchronous.
 */
int mla_merge_output_weights(const void* w_uv, const void* w_o, int dtype, int H, int d_h, int d_c,
                             int d, void* w_merged, void* stream);

/*
 * mla_absorb_output_merged -- the output projection with merged weights:
 *
 *   out[n, j] = sum_{h, c} w_merged[j, h*d_c + c] * o_lat[n, h, c]
 *
 * equal (up to rounding) to mla_absorb_output with the weights merged by
 * mla_merge_output_weights.  o_lat is rounded to bf16 (like the weights)
 * and the products are summed in fp32 on the tensor cores, split along
 * H*d_c; the splits are added in a fixed order, so the result is
 * deterministic.  It reads d*H*d_c weights against H*d_h*(d_c + d) unmerged:
 * more whenever d_h < d_c.
 *
 *   o_lat [N, H, d_c] float;  w_merged [d, H*d_c] bf16;  out [N, d] float
 *   workspace: >= mla_absorb_output_merged_workspace_size(N, H, d_c, d)
 *              bytes, 256-byte aligned (a bf16 copy of o_lat and the fp32
 *              partial sums)
 * Host errors: MLA_ERR_INVALID_ARG (bad sizes, NULL or unaligned pointers),
 * MLA_ERR_UNSUPPORTED (dtype != MLA_BF16), MLA_ERR_WORKSPACE.  Device
 * errors: MLA_ERR_TIMEOUT.  Asynchronous on `stream`.
 */
size_t mla_absorb_output_merged_workspace_size(int N, int H, int d_c, int d);   /* 0: invalid */
int mla_absorb_output_merged(const float* o_lat, const void* w_merged, int dtype, int N, int H,
                             int d_c, int d, void* workspace, size_t workspace_bytes, float* out,
                             void* stream);

/*
 * mla_decode_split_plan -- HOST helper: which split workers mla_decode_paged
 * assigns to each sequence, for a given worker count and item cost (no
 * device needed).
 *
 * Work is laid on a cost axis: each valid sequence b covers item_cost units
 * (the fixed cost of one work item: loading its query rows and writing its
 * output) followed by ceil(L_b / 64) units, one per page (T pages, U units in
 * all).  The axis is cut into W' = min(num_workers, floor(U / (item_cost + 1)))
 * ranges whose sizes differ by at most one unit, so every active worker
 * carries about the same cost; each range holds at least one page.  For each
 * b, first_worker[b] / last_worker[b] get the first and last worker holding
 * one of its pages (-1 for a sequence whose length is outside
 * [T_q, 64 * max_blocks_per_seq]).  A sequence with first == last is finished
 * by one worker; otherwise its partial results are merged by the
 * log-sum-exp combine.  item_cost = 0 is the plain even split of the pages;
 * mla_decode_paged uses mla_decode_item_cost() of the shape.  Returns the
 * total page count through *total_pages (may be NULL).  All pointers are host
 * pointers.
 * Host errors: NULL arrays, B < 1, T_q < 1, max_blocks_per_seq < 1,
 * num_workers < 1, item_cost outside [0, 1024].
 */
int mla_decode_split_plan(const int32_t* seqlens_host, int B, int T_q, int max_blocks_per_seq,
                          int num_workers, int item_cost, int32_t* first_worker,
                          int32_t* last_worker, int64_t* total_pages);

/*
 * mla_decode_item_cost -- the item cost (in pages) mla_decode_paged gives the
 * split partition for a shape: measured for the tensor-core kernel (about 5
 * at 128 query rows, 3 at 32), 0 for the CUDA-core kernel.  Returns -1 for
 * invalid dims.  Host only; needs no device.
 */
int mla_decode_item_cost(int T_q, int H, int d_c, int d_r, int dtype);

/*
 * mla_decode_row_groups -- how many row groups the decode forms of a
 * sequence's T_q * H query rows: the tensor-core kernel handles at most 128
 * rows per work item, so a sequence with more rows becomes G = ceil(rows/128)
 * work items over the same pages (rows [128 g, 128 g + 128)); 1 for the
 * CUDA-core kernel.  The split partition then runs over the B * G virtual
 * sequences in order (sequence-major): mla_decode_split_plan gives their
 * workers when each length is repeated G times.  Returns -1 for invalid dims.
 * Host only; needs no device.
 */
int mla_decode_row_groups(int T_q, int H, int d_c, int d_r, int dtype);

/*
 * mla_decode_num_workers -- the worker count mla_decode_paged uses for this
 * shape on the CURRENT device (depends on its SM count and on the kernel the
 * shape selects).  Returns 0 for invalid dims or when no device is usable.
 */
int mla_decode_num_workers(int B, int T_q, int H, int d_c, int d_r, int dtype);

/*
 * mla_decode_path -- which attention kernel mla_decode_paged selects for a
 * shape: 1 = tensor-core kernel (tcgen05/TMEM), 0 = CUDA-core kernel,
 * -1 = invalid dims.  Host only; needs no device.
 */
int mla_decode_path(int T_q, int H, int d_c, int d_r, int dtype);

/*
 * ---- Prefill with rebuilt per-head keys and values ----
 *
 * For a chunk of T_q new tokens per sequence, attention can run on the
 * per-head keys k_{s,h} = [W^UK_h c_s ; R_s k^R_s] and values
 * v_{s,h} = W^UV_h c_s rebuilt from the latent cache ("Attention, Part 2:
 * MQA, GQA and MLA", the MLA equations; "Multi-head latent attention (MLA)",
 * section 2: absorbing W^UK and W^UV or applying them to the cached latent
 * gives the same result).  Per (query, key, head) that costs
 * 2 (d_h + d_r) + 2 d_h flops instead of the absorbed path's
 * 2 (d_c + d_r) + 2 d_c, plus 4 d_c d_h per (cached row, head) for the
 * rebuild: the cheaper way once a chunk has more than a few dozen tokens.
 * The output is per head (o_h, d_h wide), ready for W^O; the absorbed path's
 * o_lat is the same o_h before W^UV.
 *
 * Supported: bf16, d_c = 512, d_h = 128, d_r = 64, page_size = 64
 * (MLA_ERR_UNSUPPORTED otherwise; there is no other kernel for these calls).
 *
 * Rebuilt buffers: R = mla_prefill_kv_rows(max_blocks_per_seq) rows per
 * sequence (64 * max_blocks_per_seq rounded up to a multiple of 128);
 * k_nope and v are bf16 [B, H, R, d_h] (head-major: the keys of one head are
 * contiguous), k_rope is bf16 [B, R, d_r]; row s of sequence b is cached
 * token s.  All device pointers, owned by the caller,
 * 16-byte aligned.
 */
int mla_prefill_kv_rows(int max_blocks_per_seq);   /* 0 for invalid input; host only */

/*
 * mla_prefill_use_rebuild -- HOST helper: which way to run a chunk of T_q new
 * tokens per sequence over sequences of L cached rows (the chunk included).
 * Returns 1 when attention over rebuilt keys (mla_prefill_kv +
 * mla_prefill_attention) is expected to be faster than the absorbed decode
 * (mla_decode_paged with T_q query tokens), 0 when the absorbed decode is,
 * or when the rebuild path does not support the shape, and -1 for invalid
 * input.  The estimate uses whole-GPU costs measured on B300: about 2.9 us
 * per group of 128 query rows and 4096 cached rows for the absorbed decode
 * (each group streams the pages once); about 168 us per 4096 rows at 128
 * heads for the rebuild, scaled by rows x heads; and 980 TFLOP/s for the
 * attention over rebuilt keys.  At H = 128 it switches near T_q = 66.  Needs
 * no device.
 */
int mla_prefill_use_rebuild(int T_q, int L, int H, int d_c, int d_r, int d_h, int dtype);

/*
 * mla_prefill_kv -- rebuild k_nope[b, h, s] = W^UK_h c_s, v[b, h, s] =
 * W^UV_h c_s and copy k_rope[b, s] = R_s k^R_s (the cached rotary key) for
 * every cached row s < seqlens[b] of every sequence, reading the paged cache
 * through block_table as mla_decode_paged does.  w_uk and w_uv are bf16
 * [H * d_h, d_c] (row h * d_h + i is output feature i of head h).  Rows from
 * seqlens[b] up to the next multiple of 128 are written as zeros (the
 * attention call reads them, masked); later rows are not touched.
 * Host errors: MLA_ERR_INVALID_ARG (bad sizes, NULL or unaligned pointers),
 * MLA_ERR_UNSUPPORTED.  Device errors (MLA_ERR_BAD_INDEX, via
 * mla_check_status): seqlens[b] < 0 or > 64 * max_blocks_per_seq (nothing
 * written for b), a block id outside [0, num_blocks) (its page reads as
 * zeros).  MLA_ERR_TIMEOUT: a bounded wait in the kernel gave up.
 * Asynchronous on `stream`.
 */
int mla_prefill_kv(const void* kv_cache, int dtype, const int32_t* block_table,
                   const int32_t* seqlens, int B, int d_c, int d_r, int page_size,
                   int max_blocks_per_seq, int num_blocks, const void* w_uk, const void* w_uv,
                   int H, int d_h, void* k_nope, void* v, void* k_rope, void* stream);

/*
 * mla_prefill_kv_chunk -- the same rebuild for one chunk of a chunked
 * prefill ("Attention, Part 2: MQA, GQA and MLA" and "The MLA equations",
 * T > 1 new tokens after earlier ones): only the chunk's rows
 * s in [seqlens[b] - T_new, seqlens[b]) are rebuilt into the caller's
 * buffers, plus the zero rows past seqlens[b] up to the next multiple of 128;
 * earlier rows keep what the earlier chunks' calls wrote.  T_new = 0 rebuilds
 * every row (mla_prefill_kv).  The buffers must have been written for the
 * earlier rows (by mla_prefill_kv or earlier chunks) and hold zeros or later
 * rows' data past them.  Errors as mla_prefill_kv, and MLA_ERR_INVALID_ARG for
 * T_new < 0.
 */
int mla_prefill_kv_chunk(const void* kv_cache, int dtype, const int32_t* block_table,
                         const int32_t* seqlens, int B, int d_c, int d_r, int page_size,
                         int max_blocks_per_seq, int num_blocks, const void* w_uk, const void* w_uv,
                         int H, int d_h, int T_new, void* k_nope, void* v, void* k_rope, void* stream);

/*
 * mla_prefill_attention -- causal softmax attention of T_q new tokens per
 * sequence over the rebuilt keys and values.  Query t of sequence b sits at
 * position seqlens[b] - T_q + t (seqlens counts every cached row, the new
 * tokens' included) and sees keys 0 .. that position.  q_nope is bf16
 * [B, T_q, H, d_h] (the content query q^C_h); q_rope is bf16
 * [B, T_q, H, d_r], NOT rotated: the call rotates it by the query's position
 * (adjacent pairs, theta_i = rope_base^(-2i/d_r), as mla_absorb_query).
 * k_nope, v, k_rope as written by mla_prefill_kv for the same
 * max_blocks_per_seq (rows from seqlens[b] to the next multiple of 128 must
 * be finite).  Outputs: o [B, T_q, H, d_h] fp32 = sum_s p_s v_{s,h};
 * lse [B, T_q, H] fp32 natural-log log-sum-exp of the scaled scores, or NULL.
 * Host errors: MLA_ERR_INVALID_ARG (bad sizes, softmax_scale <= 0, NULL or
 * unaligned pointers), MLA_ERR_UNSUPPORTED.  Device errors (MLA_ERR_BAD_INDEX):
 * seqlens[b] < T_q or > 64 * max_blocks_per_seq (zeros written for b).
 * MLA_ERR_TIMEOUT: a bounded wait gave up.  Asynchronous on `stream`.
 * Scheduling: one persistent CTA per SM takes (pair of query tiles, head)
 * items from a work counter in device memory that belongs to `stream` (the
 * first 64 streams that call it on a device get one each; the kernel leaves
 * it at zero).  Launches on one stream run in order, so they never share a
 * counter while running; later streams, and the per-thread default stream,
 * take items in a fixed order instead.  The result is the same bits either
 * way.  A CUDA graph that captured this call keeps the capturing stream's
 * counter: do not run two instances of such a graph at the same time.
 */
int mla_prefill_attention(const void* q_nope, const void* q_rope, int dtype, const void* k_nope,
                          const void* v, const void* k_rope, const int32_t* seqlens, int B,
                          int T_q, int H, int d_h, int d_r, int max_blocks_per_seq,
                          float rope_base, float softmax_scale, float* o, float* lse,
                          void* stream);

/* Text for a status code (static storage). */
const char* mla_status_string(int status);

/* Text of the last CUDA error seen by this host thread ("" if none). */
const char* mla_last_cuda_error(void);

/*
 * mla_check_status -- wait for `stream`, then read and clear the current
 * device's error word.  Returns MLA_OK, MLA_ERR_TIMEOUT, MLA_ERR_BAD_INDEX,
 * MLA_ERR_BAD_RECORD (the first of these three that was recorded, in this
 * order) or MLA_ERR_CUDA.
 */
int mla_check_status(void* stream);

/*
 * mla_test_set_wait_fault -- test hook for the bounded device waits (no
 * counterpart in the pages; failure detection of this library).
 *   skip_load > 0: every later tensor-core decode launch (mla_decode_paged,
 *     its partial stage, mla_decode_step, mla_decode_paged_noalloc) leaves
 *     out the shared-memory load of the skip_load-th page of split worker 0,
 *     and every bounded wait of the kernel gives up after wait_us
 *     microseconds (1000 if 0) instead of 2 s.  The wait for the missing page
 *     then runs out: the kernel records MLA_ERR_TIMEOUT, drains its copies
 *     and MMAs, frees its tensor memory and returns, and mla_check_status
 *     reports MLA_ERR_TIMEOUT.  Outputs of such a call are unspecified.
 *   skip_load == 0: back to normal operation.
 * Process-wide (all devices, all host threads).  Returns MLA_OK, or
 * MLA_ERR_INVALID_ARG for skip_load < 0.
 */
int mla_test_set_wait_fault(int skip_load, unsigned wait_us);

/*
 * mla_test_force_splits -- TEST KNOB (process-wide): cap the split workers
 * of mla_decode_paged (and of mla_decode_workspace_size and
 * mla_decode_num_workers, which must see the same value) at num_workers, so
 * that tests can run the same batch with 1, 2, ... splits and compare.  The
 * cost-weighted partition then cuts the pages into at most that many ranges
 * (fewer when the batch is small).  0 restores the default; values above the
 * device's worker count have no effect.  Returns MLA_OK, or
 * MLA_ERR_INVALID_ARG for a negative value.  Not for concurrent use.
 */
int mla_test_force_splits(int num_workers);

/* Library ABI version (major * 100 + minor). */
int mla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H */
