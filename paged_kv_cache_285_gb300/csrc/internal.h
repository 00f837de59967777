// Internal launch interfaces shared by the C-ABI layer (api.cu) and the
// kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

enum : int {
  DT_F16 = 0,
  DT_BF16 = 1,
  DT_E4M3 = 2,
  // extend with K read as bf16 and V pages widened to f16 beforehand (a
  // widening pass): a bf16 cache's K with its V shadow pool, or an fp8 cache's
  // K and V shadow pools (bf16 queries)
  DT_BF16_V16 = 3
};

constexpr int kSubTokens = 16;  // tokens per staged K/V tile (one MMA row block)

struct DecodeParams {
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const void* q;
  void* out;
  float* lse_out;     // nullable, natural log
  float* ws_o;        // [B][Hq][S][D] fp32 partials (S > 1)
  float* ws_lse;      // [B][Hq][S] base-2 LSE partials
  int32_t* err;       // device error word
  int max_blocks;     // block table row length
  int num_blocks;
  int batch;
  int num_q_heads;
  int num_kv_heads;
  int group;          // Hq / Hkv (a CTA takes up to 8 of them)
  int bs_shift;       // log2(block_size)
  int chunk;          // tokens per split, multiple of 16
  int num_splits;     // S of the plan
  float scale_log2;   // sm_scale * log2(e) (* k_scale for fp8)
  float out_scale;    // v_scale for fp8, else 1
};

// Per-call extras of a decode launch, a kernel argument of their own:
// widening DecodeParams changes how the decode loop is register-allocated.
//  - fused append (k_new null: none): the current token's K/V rows
//    [B][Hkv][D] in the act dtype, written to position seq_len-1 before it is
//    read;
//  - shared-prefix groups (cascade launches only): requests
//    [group_indptr[g], group_indptr[g+1]) share their first
//    group_prefix_lens[g] tokens, which a prefix pass attends once for the
//    group; the decode then covers each request's tokens from there on and
//    its partials start at workspace slot 1 (slot 0 is the prefix's).
struct DecodeExtraParams {
  const void* k_new;
  const void* v_new;
  void* k_cache;
  void* v_cache;
  float k_scale;      // fp8 store scales and their fp32 reciprocals
  float v_scale;
  float k_rcp;
  float v_rcp;
  const int32_t* group_indptr;       // [num_groups + 1]
  const int32_t* group_prefix_lens;  // [num_groups]
  int num_groups;
  int2* ws_span;                     // [batch] (first own token, length), for the merge
  // workspace slots 0 .. prefix_slots-1 hold the shared prefix's partials, one
  // per chunk of prefix_chunk keys (a prefix of W tokens fills the first
  // ceil(W / prefix_chunk)); the own tokens' splits follow them
  int prefix_slots;
  int prefix_chunk;
  int prefix_chunks;  // chunks the prefix pass computes (<= prefix_slots)
};

// Division of unsigned n < 2^31 by a divisor fixed for a launch, as a
// multiply-high and a shift (Granlund & Montgomery, "Division by invariant
// integers using multiplication", 1994): with l = ceil(log2 d) and
// m = floor(2^32 (2^l - d) / d) + 1, n / d = (umulhi(n, m) + n) >> l.
struct FastDiv {
  uint32_t d, m, l;
#ifdef __CUDACC__
  __host__ __device__
#endif
  uint32_t div(uint32_t n) const {
#ifdef __CUDA_ARCH__
    return (__umulhi(n, m) + n) >> l;
#else
    return (uint32_t)((((uint64_t)n * m) >> 32) + n) >> l;
#endif
  }
#ifdef __CUDACC__
  __host__ __device__
#endif
  uint32_t mod(uint32_t n) const { return n - div(n) * d; }
};
inline FastDiv make_fastdiv(uint32_t d) {
  FastDiv f{d, 0u, 0u};
  while ((1ull << f.l) < d) ++f.l;
  f.m = (uint32_t)((((uint64_t)1 << 32) * ((1ull << f.l) - d)) / d + 1);
  return f;
}

struct AppendParams {
  void* k_cache;
  void* v_cache;
  const void* k_new;
  const void* v_new;
  const int64_t* slots;          // null: slots from the extend layout below
  int32_t* err;
  int64_t num_tokens;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int num_blocks;
  float k_scale;
  float v_scale;
  float k_rcp;         // RN(1 / k_scale), RN(1 / v_scale)
  float v_rcp;
  // slots == null: token t is suffix row t of an extend call (request b with
  // q_indptr[b] <= t < q_indptr[b+1]) at position prefix_lens[b] + t - q_indptr[b]
  const int32_t* q_indptr;
  const int32_t* prefix_lens;
  const int32_t* block_tables;
  int batch;
  int max_blocks;
  // set by the launcher
  int bs_shift;       // log2(block_size)
  int rows_fit32;     // num_tokens * num_kv_heads < 2^31
  FastDiv div_hkv;    // by num_kv_heads
};

struct ExtendParams {
  const int32_t* q_indptr;
  const int32_t* prefix_lens;
  const int32_t* block_tables;
  // shared-prefix extend: requests group_indptr[g] .. group_indptr[g+1]-1
  // form group g and share their first group_shared[g] tokens' blocks
  // (null otherwise)
  const int32_t* group_indptr;
  const int32_t* group_shared;
  const void* q;
  void* out;
  float* lse_out;
  int32_t* err;
  int max_blocks;
  int num_blocks;
  int batch;
  int num_q_heads;
  int num_kv_heads;
  int group;            // Hq / Hkv, 1 .. 128
  int tok;              // suffix tokens per 128-row tile: 128 / group (rounded down)
  int bs_shift;
  int total_rows;
  int tiles_per_head;   // ceil(max_suffix_len / tok)
  int num_items;        // ceil(tiles_per_head / 2) * num_kv_heads * batch (pairs of tiles)
  int num_ctas;         // persistent grid: min(num_items, SM count)
  int out_32b;          // out is 32-byte aligned: rows are written with 32-byte stores
  int out_tma;          // whole row tiles of out are stored by TMA (through the output map)
  int kchunks;          // prefix pass: key chunks per pair of row tiles (1 otherwise)
  int kchunk_keys;      // prefix pass: keys per chunk, a multiple of 128
  FastDiv div_pairs;    // by ceil(tiles_per_head / 2) * kchunks
  FastDiv div_hkv;      // by num_kv_heads
  FastDiv div_req;      // by ceil(tiles_per_head / 2) * num_kv_heads (items per request)
  float scale_log2;
  float out_scale;
};

// Partial output of the extend kernel's prefix pass: row q (request b, head h:
// q = b * num_q_heads + h) over key chunk c writes O / l to
// o[q * o_stride + c * head_dim .. + head_dim) and the base-2 LSE to
// lse[q * lse_stride + c] (o 32-byte aligned, o_stride a multiple of 8).
struct ExtendPartialParams {
  float* o;
  float* lse;
  int64_t o_stride;
  int64_t lse_stride;
};

// Each returns a cudaError_t from the launch.
cudaError_t launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const DecodeParams& p, const DecodeExtraParams& ap, int head_dim,
                          int cache_dt, int act_dt, cudaStream_t stream);
// Decode over each request's tokens after its group's shared prefix, partials
// in the workspace slots after the prefix's, then (after `merge_after`, the
// prefix pass's completion, when not null) the merge with the prefix's
// partials (slots 0 .. prefix_slots-1).
cudaError_t launch_decode_cascade(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                  const DecodeParams& p, const DecodeExtraParams& ap, int head_dim,
                                  int cache_dt, int act_dt, cudaStream_t stream,
                                  cudaEvent_t merge_after);
size_t decode_smem_bytes(int head_dim, int cache_dt);
cudaError_t launch_append(const AppendParams& p, int cache_dt, int act_dt, cudaStream_t stream);
// Chain hashes of the full blocks of each request's token ids.
struct ChainHashParams {
  const int32_t* tokens;        // [token_indptr[batch]]
  const int32_t* token_indptr;  // [batch + 1]
  const uint64_t* salts;        // [batch] or null (salt 0)
  uint64_t* hashes;             // [batch][max_blocks]
  int32_t* err;                 // device error word
  int block_size;
  int max_blocks;
};
cudaError_t launch_chain_hash(const ChainHashParams& p, int batch, cudaStream_t stream);

// kmap/vmap: page maps of the K and V caches (16-bit or fp8 codes); qmap: the
// query rows, dims {head_dim, num_q_heads, total_rows}, box {64, group, tok}.
// omap: the output rows, the same dims and box as qmap (whole 16-bit row
// tiles are stored through it when p.out_tma is set).
cudaError_t launch_extend(const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const CUtensorMap& qmap, const CUtensorMap& omap, const ExtendParams& p,
                          int head_dim, int cache_dt, int act_dt, cudaStream_t stream);
// The prefix pass: ExtendParams over groups (q_indptr = group offsets into
// the batch, prefix_lens = the groups' shared prefix lengths); see extend.cu.
cudaError_t launch_extend_prefix_pass(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                      const CUtensorMap& qmap, const ExtendParams& p,
                                      const ExtendPartialParams& pp, int head_dim, int cache_dt,
                                      int act_dt, cudaStream_t stream);
// Shared-prefix extend: the rows of each group's requests packed into
// 128-row tiles; every row attends to the group's shared prefix and to its
// own request's remaining keys in one online softmax.
cudaError_t launch_extend_shared(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const CUtensorMap& qmap, const CUtensorMap& omap,
                                 const ExtendParams& p, int head_dim, int cache_dt, int act_dt,
                                 cudaStream_t stream);
bool extend_supported(int head_dim, int cache_dt, int act_dt, int group);
// The pages a shared-prefix extend reads (each group's shared blocks through
// its first member's table, every request's own blocks through its own),
// widened into 16-bit pools of the cache's shape and block ids: a bf16 cache's
// V pages into v16 as f16 (k16 unused); an fp8 cache's K pages into k16 in the
// queries' type act_dt and its V pages into v16 as f16 (the codes' values,
// exactly).  p: the call's ExtendParams (tables, lengths, groups).  Pages out
// of the pool are skipped (the extend kernel reports them).
cudaError_t launch_widen(int cache_dt, int act_dt, const void* k_cache, const void* v_cache,
                         void* k16, void* v16, const ExtendParams& p, int num_groups, int head_dim,
                         int block_size, int max_total_len, cudaStream_t stream);
// The same for a plain extend (no groups): every request's pages, each block
// widened once although requests may share it.  claims: int32 scratch of
// 1 + 2 * p.num_blocks entries (any contents; a counter and a flag per block
// are zeroed first on `stream`, then a list of the blocks claimed is built and
// widened by a grid of 8 * sm_count CTAs at most).
cudaError_t launch_widen_claim(int cache_dt, int act_dt, const void* k_cache,
                               const void* v_cache, void* k16, void* v16, int* claims,
                               const ExtendParams& p, int head_dim, int block_size,
                               int max_total_len, int sm_count, cudaStream_t stream);

}  // namespace pkv
