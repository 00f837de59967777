/*
 * pkv.h -- C ABI of the paged-KV attention library (libpkv.so, sm_103a).
 *
 * Attention over a paged KV cache: K/V of every request live in fixed-size
 * physical blocks of 16 or 32 tokens, and a per-request block table maps the
 * request's logical block i to a physical block, so that scattered blocks are
 * read as one contiguous sequence ("PagedAttention과 RadixAttention으로 LLM KV
 * 캐시 최적화", section 02).  Requests may share physical prefix blocks
 * (same page, section 03: RadixAttention reuses the longest cached prefix and
 * computes only the suffix).
 *
 * Memory layouts (all row-major, all device memory unless stated):
 *   k_cache, v_cache  [num_blocks][num_kv_heads][block_size][head_dim]
 *                     elements of cache_dtype (fp8: one byte per code)
 *   q, out            [tokens][num_q_heads][head_dim]   act dtype (f16 / bf16)
 *   k_new, v_new      [tokens][num_kv_heads][head_dim]  act dtype
 *   block_tables      int32 [batch][max_blocks_per_seq]
 *   seq_lens          int32 [batch]
 *   slot_mapping      int64 [tokens]; slot = physical_block * block_size + offset,
 *                     a negative slot means "do not write this token"
 *   GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *
 * Ownership: the caller owns and allocates every device buffer, including
 * the workspace; the library allocates no device memory.  Its own state: a
 * per-device cache of the SM count, the device error word and the scratch
 * array of pkv_paged_decode_attn_noalloc (module globals), and the host
 * objects of the prefix index (pkv_radix_create .. pkv_radix_destroy).
 *
 * Execution: every call only validates its arguments on the host and enqueues
 * kernels on `stream`; it returns before the GPU work finishes.  Buffers must
 * stay alive until the stream reaches that point.
 *
 * Errors: argument errors are detected on the host and returned before any
 * launch (PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE).  A
 * failed launch returns PKV_ERR_CUDA.  Data errors found on the device (a
 * block id or slot outside the pool, a sequence longer than its block table)
 * never fault: the offending element is skipped or read as zero, and the
 * first such event is recorded in a device error word read by
 * pkv_get_device_error().
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,   /* null pointer, negative size, Hq % Hkv != 0, ... */
  PKV_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, block_size, dtype combo */
  PKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than *_workspace_bytes() */
  PKV_ERR_CUDA = 4,          /* a CUDA runtime/driver call or a launch failed */
  PKV_ERR_NO_SPACE = 5       /* prefix index: no free block even after evicting every
                                unlocked leaf */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

/* Device error word values (pkv_get_device_error). */
#define PKV_DEVERR_NONE 0
#define PKV_DEVERR_BAD_BLOCK 1     /* block table entry outside [0, num_blocks) */
#define PKV_DEVERR_BAD_SLOT 2      /* slot_mapping entry outside the pool */
#define PKV_DEVERR_BAD_LENGTH 3    /* seq_len / prefix+suffix beyond the table or hint */
#define PKV_DEVERR_TIMEOUT 4       /* a bounded wait on an asynchronous copy ran out */
#define PKV_DEVERR_TOO_MANY_BLOCKS 5 /* chain hash: a request has more full blocks than max_blocks */

/* Description of one layer's KV pool.
 *   head_dim in {64, 128}; block_size in {16, 32};
 *   cache_dtype: PKV_F16, PKV_BF16 or PKV_FP8_E4M3;
 *   k_scale / v_scale: per-tensor dequantisation scales of an fp8 cache
 *   (value = code * scale; append stores e4m3(x / scale)).  Ignored (must be
 *   finite and > 0) for 16-bit caches.  The pages name the fp8_e4m3 format
 *   only ("KV Cache 완전 정리 — PagedAttention vs RadixAttention, SGLang이
 *   빠른 이유", section "FP8 KV 캐시"); one fp32 scale per tensor is this
 *   library's convention. */
typedef struct {
  int32_t num_blocks;
  int32_t block_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  pkv_dtype cache_dtype;
  float k_scale;
  float v_scale;
} pkv_cache_desc;

/* ---------------------------------------------------------------------------
 * pkv_kv_append -- write the K/V rows of new tokens into their cache slots.
 *
 * "KV Cache에 대해 알아보자 (Feat. Attention)", §3: at every decode step the
 * new token's K and V are added to the cache.  Token t, kv head g is stored at
 * block slot_mapping[t] / block_size, offset slot_mapping[t] % block_size.
 *   16-bit cache: act dtype must equal the cache dtype; the bits are copied.
 *   fp8 cache:    code = e4m3(fp32(x) / k_scale) (resp. v_scale), rounded to
 *                 nearest-even, saturated to +-448.
 * k_new / v_new: [num_tokens][num_kv_heads][head_dim] act dtype, device.
 * slot_mapping:  int64 [num_tokens], device.  Negative = skip.  A slot whose
 *                block lies outside the pool is skipped and reported in the
 *                device error word.
 * num_tokens == 0 is a no-op.  Several tokens writing the same slot: one of
 * them wins (unspecified which).
 * ------------------------------------------------------------------------- */
pkv_status pkv_kv_append(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                         const void* k_new, const void* v_new, pkv_dtype act_dtype,
                         const int64_t* slot_mapping, int32_t num_tokens,
                         cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_decode_attn -- one query token per request attends over all of the
 * request's cached tokens, read through its block table.
 *
 * Definition: out[b,h] = softmax_t(sm_scale * q[b,h] . K[b,t,g]) V[b,t,g] for
 * t < seq_lens[b], g = h / (Hq/Hkv) ("KV Cache에 대해 알아보자 (Feat.
 * Attention)", §1 formula, §3 decode step; the block-table read of
 * "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 02).
 * seq_lens count the current token: its K/V must already be in the cache
 * (pkv_kv_append first).
 *
 * The work is split over the sequence (split-KV): each split runs an online
 * softmax over its pages and a second pass merges the splits with their
 * log-sum-exp, which reproduces the one-pass softmax exactly up to rounding.
 *
 * q, out:        [batch][num_q_heads][head_dim] act dtype (f16 or bf16).
 *                16-bit cache: act dtype == cache dtype.  fp8 cache: either.
 * block_tables:  int32 [batch][max_blocks_per_seq].  Entries past a request's
 *                last block are never read.
 * seq_lens:      int32 [batch], each in [0, min(max_seq_len,
 *                max_blocks_per_seq*block_size)].  seq_len 0 gives out = 0,
 *                lse = -inf.
 * sm_scale:      softmax scale (1/sqrt(head_dim) for the textbook formula).
 * max_seq_len:   host-side upper bound of seq_lens; sizes the split plan.
 * num_splits:    0 = choose automatically; > 0 forces at most that many splits
 *                (1 = single pass, no merge).
 * lse_out:       nullable float [batch][num_q_heads], natural-log LSE.
 * workspace:     device scratch of pkv_decode_workspace_bytes() bytes (may be
 *                NULL when that is 0).  Concurrent calls need separate
 *                workspaces.
 * Host memory:   q, out, block_tables, seq_lens, lse_out (and k_new / v_new
 *                of pkv_paged_decode_attn_append) are read and written with
 *                plain loads and stores, so they may also be pinned host
 *                memory that the GPU addresses directly (zero-copy over a
 *                coherent host link, as on Grace-Blackwell): the bytes then
 *                cross the link inside the kernels.  The caches and the
 *                workspace must be device memory (the caches are read by
 *                TMA).
 * Supported: head_dim 64/128, block_size 16/32, any GQA group
 * num_q_heads/num_kv_heads.  One CTA takes up to 8 query heads of a kv head:
 * a group of more than 8 is split into chunks of 8 heads whose CTAs each read
 * the kv head's pages (K/V bytes are read once per chunk, mostly from L2
 * after the first).
 * ------------------------------------------------------------------------- */
size_t pkv_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t batch,
                                  int32_t num_q_heads, int32_t max_seq_len,
                                  int32_t num_splits);

pkv_status pkv_paged_decode_attn(const pkv_cache_desc* desc, const void* k_cache,
                                 const void* v_cache, const void* q, void* out,
                                 pkv_dtype act_dtype, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t batch, int32_t num_q_heads, float sm_scale,
                                 int32_t max_seq_len, int32_t num_splits, float* lse_out,
                                 void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_decode_attn_append -- decode with the current token appended by
 * the decode kernel itself.
 *
 * "KV Cache에 대해 알아보자 (Feat. Attention)", §3: each decode step adds the
 * new token's K and V to the cache and then attends over the whole cache,
 * the new token included.  This call does both in one launch: the same result
 * and the same cache bytes as pkv_kv_append of k_new/v_new into the slot of
 * position seq_lens[b]-1 (physical block block_tables[b][(n-1)/bs], offset
 * (n-1) % bs) followed by pkv_paged_decode_attn, without the separate launch
 * and the second read of the new rows.
 *
 * k_new, v_new:  [batch][num_kv_heads][head_dim] act dtype, device,
 *                16-byte aligned; request b's row goes to position
 *                seq_lens[b]-1 (requests with seq_lens[b] == 0 append nothing).
 * k_cache, v_cache: written at those slots (fp8: e4m3(fp32(x) / scale),
 *                correctly rounded division, saturating round-to-nearest-even,
 *                exactly as pkv_kv_append); the slots must not be shared by
 *                two requests of the call.
 * Everything else as pkv_paged_decode_attn.  A slot whose block id lies
 * outside the pool is not written and is reported in the device error word.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_decode_attn_append(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                                        const void* k_new, const void* v_new, const void* q,
                                        void* out, pkv_dtype act_dtype,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* seq_lens, int32_t batch,
                                        int32_t num_q_heads, float sm_scale, int32_t max_seq_len,
                                        int32_t num_splits, float* lse_out, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_decode_attn_noalloc -- the same decode as pkv_paged_decode_attn,
 * for callers that cannot allocate device memory.
 *
 * The pages describe no such call; it exists for integration only.  Some
 * callers have no way to obtain a workspace: a plugin inside an engine that
 * owns all device memory and passes in only the tensors of the call, or a
 * latency-critical path where cudaMalloc (which may synchronise the device or
 * fail under memory pressure) is not allowed.  This entry point takes no
 * workspace: the split-KV partials go to a scratch array compiled into the
 * library, PKV_NOALLOC_SCRATCH_BYTES (16 MiB) per device, held by every GPU
 * that loads the library until the process exits.  The call allocates
 * nothing.
 *
 * Arguments, layouts and results are those of pkv_paged_decode_attn.
 * Errors: PKV_ERR_WORKSPACE if the split plan for these arguments needs more
 * than PKV_NOALLOC_SCRATCH_BYTES (pkv_decode_workspace_bytes() tells the
 * size; a smaller num_splits, e.g. 1, needs none), before anything is
 * enqueued; PKV_ERR_CUDA if the scratch address cannot be obtained.
 * The first call on each device looks up the scratch array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.
 * All calls on one device share the scratch array and leave their partials
 * in it: calls whose work overlaps on the GPU (other streams, concurrent graph
 * branches) race and may produce wrong results.  Serialise them.
 * ------------------------------------------------------------------------- */
#define PKV_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

pkv_status pkv_paged_decode_attn_noalloc(const pkv_cache_desc* desc, const void* k_cache,
                                         const void* v_cache, const void* q, void* out,
                                         pkv_dtype act_dtype, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                         int32_t batch, int32_t num_q_heads, float sm_scale,
                                         int32_t max_seq_len, int32_t num_splits,
                                         float* lse_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_decode_attn_shared_prefix -- decode for groups of requests that
 * share a cached prefix, the prefix attended once per group.
 *
 * "KV Cache 완전 정리 — PagedAttention vs RadixAttention, SGLang이 빠른 이유",
 * section "RadixAttention — SGLang의 혁신", and "PagedAttention과
 * RadixAttention으로 LLM KV 캐시 최적화", section 03: many requests share one
 * long prefix (a system prompt) whose KV blocks are stored once.  Plain
 * decode reads those blocks once per request; this call computes the
 * prefix's attention for all (request, head) rows of a group in one dense
 * pass on the tensor cores, attends each request's own tokens with the
 * split-KV decode kernel, and merges the parts with their log-sum-exps,
 * which equals attention over the whole sequence up to rounding.
 *
 * Groups: request b belongs to group g when group_indptr[g] <= b <
 * group_indptr[g+1]; group_indptr (int32 [num_groups+1], device) rises from 0
 * to batch.  group_prefix_lens (int32 [num_groups], device): P_g, the tokens
 * every member of the group holds with the same K/V (0 = none).  Only whole
 * blocks are shared: with W_g = floor(P_g / block_size) * block_size, tokens
 * 0 .. W_g-1 of every member are read once for the group, through the block
 * table of its first member (block_tables[group_indptr[g]]; the other
 * members' entries for them are not read), and tokens W_g .. seq_lens[b]-1
 * through the member's own table.  P_g <= seq_lens[b] for every member (else
 * the device error word reports PKV_DEVERR_BAD_LENGTH).  A request that no
 * group covers is attended over its whole sequence through its own table and
 * reported the same way.
 *
 * k_new, v_new:  nullable together; as pkv_paged_decode_attn_append (the
 *                current token, position seq_lens[b]-1, must lie at or after
 *                W_g).
 * desc:          an fp8 cache's k_scale / v_scale are applied in both parts
 *                (scores and outputs), as in pkv_paged_decode_attn.
 * max_group_size: host bound of the members per group (sizes the prefix pass).
 * max_prefix_len: host bound of P_g.  When the groups give few work items,
 *                the prefix pass cuts each group's W_g shared keys into chunks
 *                of whole 128-key tiles (at most 8, at least 256 keys each
 *                except the last), so that the pass fills about a quarter of
 *                the SMs beside the own-token decode; every chunk's partial is
 *                one more term of the LSE merge.  Keys beyond the chunks the
 *                hint allows are not attended and set PKV_DEVERR_BAD_LENGTH.
 * max_suffix_len: host bound of seq_lens[b] - P_g (sizes the split plan).
 * num_splits:    as pkv_paged_decode_attn, for the members' own tokens.
 * workspace:     pkv_shared_prefix_decode_workspace_bytes() bytes, 256-byte
 *                aligned (always needed).
 * q:             16-byte aligned.  Everything else as pkv_paged_decode_attn.
 * Streams: the prefix pass runs on a side stream the library keeps per device
 * (highest priority), forked from `stream` by an event at the call and joined
 * back before the merge, so it overlaps the decode of the members' own
 * tokens; the call as a whole is ordered on `stream` like any other and can
 * be captured into a CUDA graph.  Calls on one device from several host
 * threads are serialised around the fork and join.
 * Supported: head_dim 64/128, block_size 16/32, f16 or bf16 cache with the
 * same act dtype or an fp8 e4m3 cache with either, GQA groups
 * num_q_heads/num_kv_heads of 1 .. 128 (one 128-row tile holds 128 / group
 * members x group heads), sm_scale > 0.
 * ------------------------------------------------------------------------- */
size_t pkv_shared_prefix_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t batch,
                                                int32_t num_q_heads, int32_t max_prefix_len,
                                                int32_t max_suffix_len, int32_t num_splits);

pkv_status pkv_paged_decode_attn_shared_prefix(
    const pkv_cache_desc* desc, void* k_cache, void* v_cache, const void* k_new,
    const void* v_new, const void* q, void* out, pkv_dtype act_dtype,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
    int32_t batch, int32_t num_q_heads, float sm_scale, const int32_t* group_indptr,
    const int32_t* group_prefix_lens, int32_t num_groups, int32_t max_group_size,
    int32_t max_prefix_len, int32_t max_suffix_len, int32_t num_splits, float* lse_out,
    void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_extend_attn -- suffix prefill over a cached prefix.
 *
 * "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03: when
 * the longest cached prefix of a request has P tokens, only the remaining
 * suffix is computed (2,000-token request with 1,900 cached -> 100 prefilled).
 * Request b owns query rows q_indptr[b] .. q_indptr[b+1]-1; its row i sits at
 * position P_b + i (P_b = prefix_lens[b]) and attends to keys 0 .. P_b + i:
 * every cached prefix token plus the suffix causally.  The suffix's own K/V
 * must already be in the cache at positions P_b .. P_b+S_b-1 (pkv_kv_append
 * first), so every key is read through the block table.
 *
 * q, out:        [q_indptr[batch]][num_q_heads][head_dim] act dtype.
 * q_indptr:      int32 [batch+1], device, non-decreasing, q_indptr[0] = 0.
 * prefix_lens:   int32 [batch], device.
 * sm_scale:      softmax scale, finite and > 0.
 * max_suffix_len / max_total_len: host-side upper bounds of S_b and P_b+S_b.
 * total_q_rows:  q_indptr[batch] (host value; sizes the grid).
 * lse_out:       nullable float [q_indptr[batch]][num_q_heads], natural log.
 * workspace:     optional: pkv_extend_workspace_bytes() is 0 for every cache
 *                dtype, and NULL, 0 is always accepted.  An fp8 cache is then
 *                read as codes and each K/V tile is widened inside the kernel
 *                (exactly: e4m3 fits f16 and bf16), with k_scale applied to
 *                the scores and v_scale to the output; the tensor cores take
 *                P as f16, so a bf16 cache's V tiles are converted to f16 the
 *                same way.  Given pkv_extend_widen_workspace_bytes() bytes or
 *                more, 256-byte aligned (any contents), the call first widens
 *                each cache block its requests read once (a block shared by
 *                several requests included) into 16-bit copies of the pools
 *                there -- V as f16 for bf16, and for fp8 also K in the
 *                queries' type -- and the kernel reads those.  The same
 *                conversions either way, so the results are bit-identical,
 *                except for an fp8 cache under bf16 queries: the per-tile
 *                path rounds the queries to f16 for S = Q K^T, this one keeps
 *                them bf16 (K widened to bf16 exactly), no less accurate.  A
 *                smaller or misaligned workspace, an f16 cache, and batches
 *                of more than 65,535 requests take the per-tile path.  Calls
 *                that run at the same time need workspaces of their own.
 * Device-side checks: a request whose rows q_indptr[b] .. q_indptr[b+1]-1
 * do not lie inside [0, total_q_rows) is not computed (nothing is written for
 * it), and suffix rows beyond max_suffix_len are not computed; both set
 * PKV_DEVERR_BAD_LENGTH.  Block ids outside the pool read zeros
 * (PKV_DEVERR_BAD_BLOCK).
 * Supported: head_dim 64/128, block_size 16/32, GQA groups
 * num_q_heads/num_kv_heads of 1 .. 128 (a 128-row tile holds 128 / group
 * suffix tokens x group heads); cache dtype equal to the act dtype (f16,
 * bf16) or fp8 e4m3 with either act dtype.
 * ------------------------------------------------------------------------- */
size_t pkv_extend_workspace_bytes(const pkv_cache_desc* desc, int32_t batch,
                                  int32_t num_q_heads, int32_t total_q_rows,
                                  int32_t max_total_len);
/* Bytes of the optional widening workspace of pkv_paged_extend_attn: the V
 * pool in 16-bit elements for a bf16 cache (the K and V pools for an fp8
 * cache), then int32 claims (a counter, and a flag and a list entry per block),
 * each part 256-byte aligned; 0 for an f16 cache (and for an invalid desc). */
size_t pkv_extend_widen_workspace_bytes(const pkv_cache_desc* desc);

pkv_status pkv_paged_extend_attn(const pkv_cache_desc* desc, const void* k_cache,
                                 const void* v_cache, const void* q, void* out,
                                 pkv_dtype act_dtype, const int32_t* q_indptr,
                                 const int32_t* prefix_lens, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, int32_t batch,
                                 int32_t num_q_heads, float sm_scale, int32_t total_q_rows,
                                 int32_t max_suffix_len, int32_t max_total_len,
                                 float* lse_out, void* workspace, size_t workspace_bytes,
                                 cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * pkv_paged_extend_attn_shared_prefix -- suffix prefill for groups of
 * requests that share a cached prefix.
 *
 * "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", sections 02-03:
 * requests that share a prompt prefix point their block tables at the same
 * physical blocks, and only each request's suffix is computed.  The result is
 * that of pkv_paged_extend_attn on the same arguments (every row i of request
 * b attends to keys 0 .. P_b + i through b's block table); the call differs in
 * how the work is laid out.  The suffix rows of a group's requests are packed
 * back to back into 128-row tiles (no tile is padded at a request's end), and
 * each tile pair reads the group's shared blocks once for all of its rows,
 * then each of its requests' remaining keys (its unshared prefix tail and its
 * suffix) with the other requests' rows masked.
 *
 * group_indptr:      int32 [num_groups+1], device: group g is requests
 *                    group_indptr[g] .. group_indptr[g+1]-1 (consecutive in
 *                    q_indptr order); the groups partition 0 .. batch-1.
 * group_shared_lens: int32 [num_groups], device: W_g, the tokens whose blocks
 *                    every member of group g shares (the same physical block
 *                    ids in the first W_g / block_size entries of their
 *                    tables), rounded down to whole blocks by the kernel.
 *                    Every member with rows must have prefix_lens[b] >= W_g.
 *                    W_g = 0 is allowed (rows are still packed).
 * max_group_rows:    host-side upper bound of the suffix rows of a group
 *                    (q_indptr[group_indptr[g+1]] - q_indptr[group_indptr[g]]);
 *                    it sizes the grid.
 * workspace:         NULL, or pkv_extend_shared_prefix_workspace_bytes()
 *                    bytes of device memory, 256-byte aligned (any contents;
 *                    the size is 0 for an f16 cache).  The tensor cores take
 *                    P as f16, so a bf16 cache's V tiles, and an fp8 cache's K
 *                    and V tiles, are otherwise converted to f16 tile by tile
 *                    in shared memory.  With a workspace, the call first
 *                    widens the pages it reads (each group's shared blocks
 *                    once, every request's own blocks) into f16 copies of
 *                    those pools there -- V for bf16 (as f16), K and V for fp8
 *                    (K in the queries' type, V as f16: twice an fp8 cache's
 *                    size, memory traded for speed) -- and the kernel reads
 *                    them from it.  The same conversions either way, so the
 *                    results are bit-identical, except for an fp8 cache under
 *                    bf16 queries: the per-tile path rounds the queries to f16
 *                    for S = Q K^T, this one keeps them bf16 (K widened to
 *                    bf16 exactly), no less accurate.  A workspace smaller
 *                    than the size, or misaligned, gives PKV_ERR_WORKSPACE.
 *                    Batches of more than 65,535 requests do not use it.
 *                    Calls that run at the same time need workspaces of their
 *                    own.
 * Everything else as pkv_paged_extend_attn.
 * Device-side checks: a group whose request range or rows are not valid, rows
 * beyond max_group_rows, and a request whose prefix is shorter than W_g or
 * whose keys do not fit its block table are not computed (nothing is written
 * for the rows of the tile pairs concerned) and set PKV_DEVERR_BAD_LENGTH.
 * Supported: as pkv_paged_extend_attn.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_extend_attn_shared_prefix(
    const pkv_cache_desc* desc, const void* k_cache, const void* v_cache, const void* q, void* out,
    pkv_dtype act_dtype, const int32_t* q_indptr, const int32_t* prefix_lens,
    const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t batch, int32_t num_q_heads,
    float sm_scale, int32_t total_q_rows, const int32_t* group_indptr,
    const int32_t* group_shared_lens, int32_t num_groups, int32_t max_group_rows,
    int32_t max_total_len, float* lse_out, void* workspace, size_t workspace_bytes,
    cudaStream_t stream);
/* Bytes of the optional workspace of pkv_paged_extend_attn_shared_prefix: the
 * V pool in 16-bit elements for a bf16 cache, the K and V pools in 16-bit
 * elements for an fp8 cache, 0 for an f16 cache (and for an invalid desc). */
size_t pkv_extend_shared_prefix_workspace_bytes(const pkv_cache_desc* desc);

/* ---------------------------------------------------------------------------
 * pkv_paged_extend_attn_append -- suffix prefill with the suffix's K/V written
 * into the cache by the same call.
 *
 * "KV Cache에 대해 알아보자 (Feat. Attention)", §3: the K/V of every processed
 * token go into the cache; "PagedAttention과 RadixAttention으로 LLM KV 캐시
 * 최적화", section 03: only the suffix after the cached prefix is computed.
 * Same result and same cache bytes as pkv_kv_append of k_new/v_new into
 * positions prefix_lens[b] + i of request b (physical block
 * block_tables[b][(prefix_lens[b]+i)/bs], offset (prefix_lens[b]+i) % bs)
 * followed by pkv_paged_extend_attn, in one call without a slot mapping: the
 * append kernel derives each row's slot from q_indptr, prefix_lens and the
 * block table, then the extend kernel runs (two launches in stream order).
 * Writing the rows from inside the extend kernel was built and measured
 * slower (the extra warp code displaced the softmax loop's instructions).
 *
 * k_new, v_new:  [total_q_rows][num_kv_heads][head_dim], the act dtype,
 *                device, 16-byte aligned; row q_indptr[b] + i is suffix token
 *                i of request b.  An fp8 cache stores e4m3(fp32(x) / scale)
 *                exactly as pkv_kv_append.
 * Everything else as pkv_paged_extend_attn.  A suffix slot whose block id
 * lies outside the pool is not written and is reported in the device error
 * word.
 * ------------------------------------------------------------------------- */
pkv_status pkv_paged_extend_attn_append(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                                        const void* k_new, const void* v_new, const void* q,
                                        void* out, pkv_dtype act_dtype, const int32_t* q_indptr,
                                        const int32_t* prefix_lens, const int32_t* block_tables,
                                        int32_t max_blocks_per_seq, int32_t batch,
                                        int32_t num_q_heads, float sm_scale, int32_t total_q_rows,
                                        int32_t max_suffix_len, int32_t max_total_len,
                                        float* lse_out, cudaStream_t stream);

/* ---------------------------------------------------------------------------
 * Prefix index (host): radix tree over token ids with leaf-first LRU eviction.
 *
 * "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03: the KV
 * of finished requests stays on token paths of a radix tree, a new request
 * reuses the longest matching path and prefills only the rest, and when
 * memory runs short unused leaf branches are evicted first (least recently
 * used first) so that interior prefixes shared by many requests survive.
 * With paged KV only whole blocks are shared: edge labels, matches and
 * insertions are whole numbers of block_size tokens (a prefix that ends inside
 * a block is matched up to the block before it).
 *
 * The index owns the physical block ids [0, num_blocks) of one cache pool.
 * A block is free, held by the caller (pkv_radix_alloc, until pkv_radix_insert
 * adopts it or pkv_radix_free returns it), or held by the tree (evictable once
 * no match holds it).  All arrays here are host memory owned by the caller;
 * the index keeps no pointer to them.  Not thread-safe.  The typical request:
 *   match(tokens) -> P matched tokens, their blocks (locked);
 *   alloc(blocks for the remaining tokens) -> block table = matched + new;
 *   kv_append the suffix K/V, paged_extend_attn with prefix_len = P;
 *   insert(tokens, block table) -> the tree adopts the new full blocks and
 *   hands back any block it already held under the same tokens;
 *   release(tokens, P) unlocks the matched path; free() the partial tail block
 *   when the request is done with it.
 * ------------------------------------------------------------------------- */
typedef struct pkv_radix_index pkv_radix_index;

typedef struct {
  int32_t num_blocks;       /* pool size */
  int32_t free_blocks;      /* not held by anyone */
  int32_t tree_blocks;      /* held by the tree */
  int32_t caller_blocks;    /* allocated and not yet inserted or freed */
  int32_t nodes;            /* tree nodes (edges), the root not counted */
  int32_t evictable_leaves; /* leaves that no match holds */
} pkv_radix_stats_t;

/* New index over block ids [0, num_blocks) of a pool with block_size tokens
 * per block; every block starts free.  *out = NULL on error. */
pkv_status pkv_radix_create(int32_t block_size, int32_t num_blocks, pkv_radix_index** out);
void pkv_radix_destroy(pkv_radix_index* index);

/* Longest cached prefix of tokens[0, num_tokens) in whole blocks: its length
 * in *matched_tokens and its physical blocks, in order, in blocks_out (room for
 * blocks_cap).  The path is locked (never evicted) until pkv_radix_release and
 * marked as used now.  blocks_cap too small -> PKV_ERR_INVALID_ARG, nothing
 * locked, *matched_tokens still set. */
pkv_status pkv_radix_match(pkv_radix_index* index, const int32_t* tokens, int32_t num_tokens,
                           int32_t* blocks_out, int32_t blocks_cap, int32_t* matched_tokens);

/* Unlock a path locked by pkv_radix_match (same tokens, the matched length). */
pkv_status pkv_radix_release(pkv_radix_index* index, const int32_t* tokens,
                             int32_t matched_tokens);

/* count free blocks for the caller, evicting unlocked leaves (least recently
 * used first) as needed; PKV_ERR_NO_SPACE when even that is not enough (the
 * evictions made so far stay made, nothing is allocated). */
pkv_status pkv_radix_alloc(pkv_radix_index* index, int32_t count, int32_t* blocks_out);

/* Return caller-held blocks to the pool. */
pkv_status pkv_radix_free(pkv_radix_index* index, const int32_t* blocks, int32_t count);

/* The tree takes the full blocks of tokens[0, num_tokens) with their physical
 * blocks blocks[0, num_tokens / block_size): blocks it already holds under the
 * same tokens stay the tree's; a caller block standing for such a block is
 * freed and reported in released_out (room for num_tokens / block_size, may be
 * NULL) / *num_released; the remaining blocks are adopted.  A partial last
 * block is not taken.  Blocks that are free, or twice in the list ->
 * PKV_ERR_INVALID_ARG with no change. */
pkv_status pkv_radix_insert(pkv_radix_index* index, const int32_t* tokens, int32_t num_tokens,
                            const int32_t* blocks, int32_t* released_out, int32_t* num_released);

/* Evict unlocked leaves, least recently used first, until num_blocks blocks
 * are freed or nothing is evictable; *freed = blocks freed. */
pkv_status pkv_radix_evict(pkv_radix_index* index, int32_t num_blocks, int32_t* freed);

pkv_status pkv_radix_stats(const pkv_radix_index* index, pkv_radix_stats_t* out);

/* ---------------------------------------------------------------------------
 * pkv_chain_hash -- chain hashes of full KV blocks (block identifiers).
 *
 * "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 05: a
 * block's hash combines its parent block's hash with the block's token ids
 * (and optional extra data), so equal token prefixes give equal chains and a
 * request's first miss marks where new blocks begin; section 06: a per-tenant
 * salt in the identifier keeps tenants apart.  The pages fix no hash; this one
 * (G = 0x9E3779B97F4A7C15, mix = the SplitMix64 finalizer):
 *   content(block) = c after c = mix(c + G + (uint32)token) over the block's
 *                    tokens, from c = 0;
 *   h[0] = mix((salt ^ content(block 0)) + G),
 *   h[i] = mix((h[i-1] ^ content(block i)) + G).
 * Extra data (a LoRA or multimodal id) belongs in the salt.
 *
 * tokens:        int32 [token_indptr[batch]], device; request b owns
 *                tokens[token_indptr[b] .. token_indptr[b+1]).
 * token_indptr:  int32 [batch+1], device, non-decreasing.
 * salts:         uint64 [batch], device, or NULL (salt 0).
 * hashes:        uint64 [batch][max_blocks], device: request b's full blocks
 *                (len / block_size of them) get hashes[b][0 ..); a partial
 *                last block gets none; other entries are left untouched.  A
 *                request with more full blocks than max_blocks gets the first
 *                max_blocks and PKV_DEVERR_TOO_MANY_BLOCKS in the error word.
 * block_size:    1 .. 4096 tokens.
 * ------------------------------------------------------------------------- */
pkv_status pkv_chain_hash(const int32_t* tokens, const int32_t* token_indptr, int32_t batch,
                          int32_t block_size, const uint64_t* salts, uint64_t* hashes,
                          int32_t max_blocks, cudaStream_t stream);

/* Human-readable name of a status code (static string, never NULL). */
const char* pkv_status_string(pkv_status status);

/* Read (and optionally clear) the device error word of the current device.
 * Synchronises `stream`.  Returns PKV_OK and writes the word to *word. */
pkv_status pkv_get_device_error(int32_t* word, int32_t clear, cudaStream_t stream);

/* Library version, major*10000 + minor*100 + patch.  2.0.0: the shared-prefix
 * extend takes a workspace (two arguments before the stream).  2.1.0:
 * pkv_extend_widen_workspace_bytes; the plain extend uses a workspace of that
 * size (its signature unchanged). */
int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
