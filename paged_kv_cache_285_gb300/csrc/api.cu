// C ABI of libpkv.so: argument validation, split planning, TMA descriptors and
// launches.  Every check runs on the host before anything is enqueued.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <mutex>

#include "../../include/pkv.h"
#include "internal.h"

using namespace pkv;

// Device error word: first data error seen by any kernel (see pkv.h).
__device__ int32_t g_pkv_error_word = 0;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  std::once_flag once;
  int sm_count = 0;
  int32_t* err = nullptr;
  cudaError_t init_error = cudaSuccess;
  // side stream of the shared-prefix decode, created on first use: its
  // prefix pass runs there, beside the decode of the members' own tokens on
  // the caller's stream (fork / join events order both against the caller's
  // stream; the mutex keeps concurrent callers' fork and join apart)
  std::once_flag side_once;
  std::mutex side_mu;
  cudaStream_t side = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  cudaError_t side_error = cudaSuccess;
};
DeviceState g_dev[kMaxDevices];

DeviceState* device_state(cudaError_t* e) {
  int dev = 0;
  *e = cudaGetDevice(&dev);
  if (*e != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= kMaxDevices) {
    *e = cudaErrorInvalidDevice;
    return nullptr;
  }
  DeviceState* s = &g_dev[dev];
  std::call_once(s->once, [s, dev]() {
    cudaError_t r = cudaDeviceGetAttribute(&s->sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (r == cudaSuccess) r = cudaGetSymbolAddress(reinterpret_cast<void**>(&s->err), g_pkv_error_word);
    s->init_error = r;
  });
  *e = s->init_error;
  return s->init_error == cudaSuccess ? s : nullptr;
}

cudaError_t side_stream(DeviceState* s) {
  std::call_once(s->side_once, [s]() {
    int least = 0, greatest = 0;
    cudaError_t r = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (r == cudaSuccess) r = cudaStreamCreateWithPriority(&s->side, cudaStreamNonBlocking, greatest);
    if (r == cudaSuccess) r = cudaEventCreateWithFlags(&s->fork, cudaEventDisableTiming);
    if (r == cudaSuccess) r = cudaEventCreateWithFlags(&s->join, cudaEventDisableTiming);
    s->side_error = r;
  });
  return s->side_error;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int elem_bytes(pkv_dtype d) { return d == PKV_FP8_E4M3 ? 1 : 2; }

bool valid_dtype(pkv_dtype d) { return d == PKV_F16 || d == PKV_BF16 || d == PKV_FP8_E4M3; }

pkv_status check_desc(const pkv_cache_desc* d) {
  if (!d) return PKV_ERR_INVALID_ARG;
  if (d->num_blocks <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0 || d->block_size <= 0)
    return PKV_ERR_INVALID_ARG;
  if (!valid_dtype(d->cache_dtype)) return PKV_ERR_INVALID_ARG;
  if (!(d->head_dim == 64 || d->head_dim == 128)) return PKV_ERR_UNSUPPORTED;
  if (!(d->block_size == 16 || d->block_size == 32)) return PKV_ERR_UNSUPPORTED;
  if (d->cache_dtype == PKV_FP8_E4M3) {
    if (!(std::isfinite(d->k_scale) && d->k_scale > 0.f && std::isfinite(d->v_scale) &&
          d->v_scale > 0.f))
      return PKV_ERR_INVALID_ARG;
  }
  if ((int64_t)d->num_blocks * d->num_kv_heads > (int64_t)INT32_MAX) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

pkv_status check_act(const pkv_cache_desc* d, pkv_dtype act) {
  if (act != PKV_F16 && act != PKV_BF16) return PKV_ERR_INVALID_ARG;
  if (d->cache_dtype != PKV_FP8_E4M3 && d->cache_dtype != act) return PKV_ERR_UNSUPPORTED;
  return PKV_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// One 16-token tile of one kv head per TMA box row group:
// dims {head_dim, block_size, num_blocks*Hkv}, box {min(128B row) , 16, 1}.
pkv_status make_page_map(CUtensorMap* m, const void* base, const pkv_cache_desc* d) {
  auto enc = encode_fn();
  if (!enc) return PKV_ERR_CUDA;
  const int elem = elem_bytes(d->cache_dtype);
  const int rowb = d->head_dim * elem;
  const int chunkb = rowb < 128 ? rowb : 128;
  cuuint64_t dims[3] = {(cuuint64_t)d->head_dim, (cuuint64_t)d->block_size,
                        (cuuint64_t)d->num_blocks * (cuuint64_t)d->num_kv_heads};
  cuuint64_t strides[2] = {(cuuint64_t)rowb, (cuuint64_t)rowb * (cuuint64_t)d->block_size};
  cuuint32_t box[3] = {(cuuint32_t)(chunkb / elem), (cuuint32_t)kSubTokens, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUtensorMapDataType dt =
      elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const CUtensorMapSwizzle sw =
      chunkb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  CUresult r = enc(m, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

// Query rows of the extend call as a 3-D map {head_dim, num_q_heads, rows}:
// one box {64, group, 128 / group} is the 64-dim column block of a row tile of
// (suffix token, head of the group) rows, 128-byte swizzled.
pkv_status make_q_map(CUtensorMap* m, const void* q, int head_dim, int num_q_heads,
                      int total_rows, int group) {
  auto enc = encode_fn();
  if (!enc) return PKV_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)total_rows};
  cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2u, (cuuint64_t)head_dim * 2u * (cuuint64_t)num_q_heads};
  cuuint32_t box[3] = {64u, (cuuint32_t)group, (cuuint32_t)(128 / group)};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims, strides, box,
                   estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PKV_OK : PKV_ERR_CUDA;
}

int ceil_div(int64_t a, int64_t b) { return (int)((a + b - 1) / b); }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Work decomposition of an extend launch: rows of one (request, kv head) in
// tiles of `tok` suffix tokens x `group` heads, a work item = a pair of tiles,
// one persistent CTA per SM.  False if the item count overflows.
bool plan_extend(ExtendParams& p, int batch, int num_kv_heads, int group, int max_rows_per_request,
                 int sm_count) {
  p.group = group;
  p.tok = 128 / group;
  p.kchunks = 1;
  p.kchunk_keys = 0;
  p.tiles_per_head = ceil_div((int64_t)max_rows_per_request, p.tok);
  const int64_t pairs = (p.tiles_per_head + 1) / 2;
  const int64_t items = pairs * num_kv_heads * batch;
  if (items > INT32_MAX || pairs * num_kv_heads > UINT32_MAX / 2) return false;
  p.num_items = (int)items;
  p.div_pairs = make_fastdiv((uint32_t)pairs);
  p.div_hkv = make_fastdiv((uint32_t)num_kv_heads);
  p.div_req = make_fastdiv((uint32_t)(pairs * num_kv_heads));
  p.num_ctas = (int)std::min<int64_t>(items, sm_count > 0 ? sm_count : 1);
  return true;
}

// Softmax scale in base 2 with an fp8 cache's k_scale folded in (scores are
// computed on the codes), and the output scale (v_scale for fp8, else 1).
float score_scale_log2(const pkv_cache_desc* d, float sm_scale) {
  const double kscale = d->cache_dtype == PKV_FP8_E4M3 ? (double)d->k_scale : 1.0;
  return (float)((double)sm_scale * kscale * 1.4426950408889634);
}
float output_scale(const pkv_cache_desc* d) {
  return d->cache_dtype == PKV_FP8_E4M3 ? d->v_scale : 1.0f;
}

struct DecodePlan {
  int chunk = 0;
  int splits = 0;
  size_t ws_bytes = 0;
  size_t ws_lse_offset = 0;
  size_t ws_span_offset = 0;  // cascade: int2 (first own token, length) per request
};

// Split plan: the sequence is cut into runs of `chunk` tokens (a multiple of
// 16).  Automatic: aim for about six waves of two CTAs per SM over the worst
// case batch*Hkv*max_seq_len, runs between 128 and 4096 tokens.
DecodePlan plan_decode(const pkv_cache_desc* d, int batch, int hq, int max_seq_len,
                       int forced, int sm_count) {
  DecodePlan pl;
  const int max_sub = max_seq_len > 0 ? ceil_div(max_seq_len, kSubTokens) : 1;
  int chunk_sub;
  if (forced > 0) {
    chunk_sub = ceil_div(max_sub, forced);
  } else {
    const int64_t work = (int64_t)max_sub * batch * d->num_kv_heads;
    const int64_t target = 6LL * 2LL * (sm_count > 0 ? sm_count : 148);
    chunk_sub = ceil_div(work, target);
    if (chunk_sub < 8) chunk_sub = 8;
    if (chunk_sub > 256) chunk_sub = 256;
  }
  if (chunk_sub < 1) chunk_sub = 1;
  pl.chunk = chunk_sub * kSubTokens;
  pl.splits = ceil_div(max_sub, chunk_sub);
  if (pl.splits < 1) pl.splits = 1;
  if (pl.splits > 1) {
    const size_t o_bytes = (size_t)batch * hq * pl.splits * d->head_dim * sizeof(float);
    pl.ws_lse_offset = (o_bytes + 255) & ~(size_t)255;
    pl.ws_bytes = pl.ws_lse_offset + (size_t)batch * hq * pl.splits * sizeof(float);
  }
  return pl;
}

}  // namespace

extern "C" {

pkv_status pkv_chain_hash(const int32_t* tokens, const int32_t* token_indptr, int32_t batch,
                          int32_t block_size, const uint64_t* salts, uint64_t* hashes,
                          int32_t max_blocks, cudaStream_t stream) {
  if (batch < 0 || block_size <= 0 || block_size > 4096 || max_blocks < 0) return PKV_ERR_INVALID_ARG;
  if (batch == 0 || max_blocks == 0) return PKV_OK;
  if (!tokens || !token_indptr || !hashes) return PKV_ERR_INVALID_ARG;
  if (!aligned(hashes, 8) || (salts && !aligned(salts, 8)) || !aligned(tokens, 4))
    return PKV_ERR_INVALID_ARG;
  cudaError_t e;
  DeviceState* ds = device_state(&e);
  if (!ds) return PKV_ERR_CUDA;
  ChainHashParams p;
  p.tokens = tokens;
  p.token_indptr = token_indptr;
  p.salts = salts;
  p.hashes = hashes;
  p.err = ds->err;
  p.block_size = block_size;
  p.max_blocks = max_blocks;
  e = launch_chain_hash(p, batch, stream);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

const char* pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_NO_SPACE: return "PKV_ERR_NO_SPACE";
    default: return "PKV_ERR_UNKNOWN";
  }
}

int32_t pkv_version(void) { return 20100; }

pkv_status pkv_get_device_error(int32_t* word, int32_t clear, cudaStream_t stream) {
  if (!word) return PKV_ERR_INVALID_ARG;
  cudaError_t e;
  DeviceState* ds = device_state(&e);
  if (!ds) return PKV_ERR_CUDA;
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, ds->err, sizeof(int32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (clear && cudaMemsetAsync(ds->err, 0, sizeof(int32_t), stream) != cudaSuccess)
    return PKV_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PKV_ERR_CUDA;
  *word = host;
  return PKV_OK;
}

pkv_status pkv_kv_append(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                         const void* k_new, const void* v_new, pkv_dtype act_dtype,
                         const int64_t* slot_mapping, int32_t num_tokens, cudaStream_t stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if ((st = check_act(desc, act_dtype)) != PKV_OK) return st;
  if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k_cache || !v_cache || !k_new || !v_new || !slot_mapping) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
    return PKV_ERR_INVALID_ARG;
  cudaError_t e;
  DeviceState* ds = device_state(&e);
  if (!ds) return PKV_ERR_CUDA;
  AppendParams p{};
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.k_new = k_new;
  p.v_new = v_new;
  p.slots = slot_mapping;
  p.err = ds->err;
  p.num_tokens = num_tokens;
  p.num_kv_heads = desc->num_kv_heads;
  p.head_dim = desc->head_dim;
  p.block_size = desc->block_size;
  p.num_blocks = desc->num_blocks;
  p.k_scale = desc->k_scale;
  p.v_scale = desc->v_scale;
  e = launch_append(p, (int)desc->cache_dtype, (int)act_dtype, stream);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

size_t pkv_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t batch, int32_t num_q_heads,
                                  int32_t max_seq_len, int32_t num_splits) {
  if (check_desc(desc) != PKV_OK || batch <= 0 || num_q_heads <= 0 || max_seq_len < 0 ||
      num_splits < 0)
    return 0;
  cudaError_t e;
  DeviceState* ds = device_state(&e);
  const int sms = ds ? ds->sm_count : 0;
  return plan_decode(desc, batch, num_q_heads, max_seq_len, num_splits, sms).ws_bytes;
}

}  // extern "C"

// Plan of a shared-prefix decode: the decode split plan over the requests'
// own tokens, plus workspace slots for the shared prefix's partials (one per
// key chunk, at most kMaxPrefixChunks, chunks of at least kMinPrefixChunk keys)
// per (request, head), always merged.
constexpr int kMaxPrefixChunks = 8;
constexpr int kMinPrefixChunk = 256;
int prefix_slots_for(int max_prefix_len) {
  const int by_len = ceil_div(std::max(max_prefix_len, 1), kMinPrefixChunk);
  return std::min(kMaxPrefixChunks, std::max(1, by_len));
}
static DecodePlan plan_cascade(const pkv_cache_desc* d, int batch, int hq, int max_prefix_len,
                               int max_suffix_len, int forced, int sm_count) {
  // a member's own tokens start at its group's prefix rounded down to whole
  // blocks: up to block_size - 1 more than seq_len - prefix
  DecodePlan pl = plan_decode(d, batch, hq, max_suffix_len + d->block_size - 1, forced, sm_count);
  const size_t slots = (size_t)pl.splits + prefix_slots_for(max_prefix_len);
  pl.ws_lse_offset = align256((size_t)batch * hq * slots * d->head_dim * sizeof(float));
  pl.ws_span_offset = align256(pl.ws_lse_offset + (size_t)batch * hq * slots * sizeof(float));
  pl.ws_bytes = pl.ws_span_offset + (size_t)batch * 2 * sizeof(int32_t);
  return pl;
}

extern "C" {

size_t pkv_shared_prefix_decode_workspace_bytes(const pkv_cache_desc* desc, int32_t batch,
                                                int32_t num_q_heads, int32_t max_prefix_len,
                                                int32_t max_suffix_len, int32_t num_splits) {
  if (check_desc(desc) != PKV_OK || batch <= 0 || num_q_heads <= 0 || max_prefix_len < 0 ||
      max_suffix_len < 0 || num_splits < 0)
    return 0;
  cudaError_t e;
  DeviceState* ds = device_state(&e);
  const int sms = ds ? ds->sm_count : 0;
  return plan_cascade(desc, batch, num_q_heads, max_prefix_len, max_suffix_len, num_splits, sms)
      .ws_bytes;
}

pkv_status pkv_paged_decode_attn_shared_prefix(
    const pkv_cache_desc* desc, void* k_cache, void* v_cache, const void* k_new, const void* v_new,
    const void* q, void* out, pkv_dtype act_dtype, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
    float sm_scale, const int32_t* group_indptr, const int32_t* group_prefix_lens,
    int32_t num_groups, int32_t max_group_size, int32_t max_prefix_len, int32_t max_suffix_len,
    int32_t num_splits, float* lse_out, void* workspace, size_t workspace_bytes,
    cudaStream_t stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if ((st = check_act(desc, act_dtype)) != PKV_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || num_groups < 0 ||
      max_group_size < 0 || max_prefix_len < 0 || max_suffix_len < 0 || num_splits < 0 ||
      !std::isfinite(sm_scale) || !(sm_scale > 0.f))
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % desc->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int group = num_q_heads / desc->num_kv_heads;
  if (!extend_supported(desc->head_dim, (int)desc->cache_dtype, (int)act_dtype, group))
    return PKV_ERR_UNSUPPORTED;
  if (batch == 0) return PKV_OK;
  if (num_groups == 0 || max_group_size == 0) return PKV_ERR_INVALID_ARG;
  if (batch > 65535 || desc->num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (!k_cache || !v_cache || !q || !out || !block_tables || !seq_lens || !group_indptr ||
      !group_prefix_lens)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 2))
    return PKV_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID_ARG;
  if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))) return PKV_ERR_INVALID_ARG;
  cudaError_t e;
  DeviceState* ds = device_state(&e);
  if (!ds) return PKV_ERR_CUDA;
  const DecodePlan pl = plan_cascade(desc, batch, num_q_heads, max_prefix_len, max_suffix_len,
                                     num_splits, ds->sm_count);
  if (!workspace || workspace_bytes < pl.ws_bytes || !aligned(workspace, 256))
    return PKV_ERR_WORKSPACE;
  if (pl.splits > 65535) return PKV_ERR_UNSUPPORTED;
  CUtensorMap kmap, vmap, qmap;
  if ((st = make_page_map(&kmap, k_cache, desc)) != PKV_OK) return st;
  if ((st = make_page_map(&vmap, v_cache, desc)) != PKV_OK) return st;
  if ((st = make_q_map(&qmap, q, desc->head_dim, num_q_heads, batch, group)) != PKV_OK) return st;
  float* ws_o = reinterpret_cast<float*>(workspace);
  float* ws_lse = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.ws_lse_offset);
  const int prefix_slots = prefix_slots_for(max_prefix_len);
  const int slots = pl.splits + prefix_slots;
  const float scale_log2 = score_scale_log2(desc, sm_scale);

  // 1. the shared prefixes, once per group, on the tensor cores -> one
  //    partial per key chunk in the first prefix_slots slots (on the side
  //    stream, beside step 2)
  ExtendParams pe{};
  pe.q_indptr = group_indptr;
  pe.prefix_lens = group_prefix_lens;
  pe.block_tables = block_tables;
  pe.q = q;
  pe.out = nullptr;
  pe.lse_out = nullptr;
  pe.err = ds->err;
  pe.max_blocks = max_blocks_per_seq;
  pe.num_blocks = desc->num_blocks;
  pe.batch = num_groups;
  pe.num_q_heads = num_q_heads;
  pe.num_kv_heads = desc->num_kv_heads;
  pe.out_32b = 0;
  pe.bs_shift = desc->block_size == 16 ? 4 : 5;
  pe.total_rows = batch;
  pe.scale_log2 = scale_log2;
  pe.out_scale = output_scale(desc);
  if (!plan_extend(pe, num_groups, desc->num_kv_heads, group, max_group_size, ds->sm_count))
    return PKV_ERR_UNSUPPORTED;
  // The prefix's keys in chunks of whole key tiles when the groups give few
  // work items: the pass runs beside the own-token decode and should take
  // about a quarter of the SMs (measured on the shared-prompt layer: 32 items
  // of 8 key tiles beside the decode, 55 us per call; 128 items of 2 tiles run
  // before it, 75 us).  Each chunk's partial is one more term of the LSE
  // merge; at most prefix_slots chunks.
  const int key_tiles = std::max(1, ceil_div(max_prefix_len, 128));
  const int quarter = std::max(1, (ds->sm_count > 0 ? ds->sm_count : 4) / 4);
  const int want = std::max(1, quarter / pe.num_items);
  const int chunk_tiles = ceil_div(key_tiles, std::min(std::min(want, prefix_slots), key_tiles));
  pe.kchunks = ceil_div(key_tiles, chunk_tiles);
  pe.kchunk_keys = chunk_tiles * 128;
  {
    const int64_t items = (int64_t)pe.num_items * pe.kchunks;
    const uint32_t pairs = (uint32_t)((pe.tiles_per_head + 1) / 2);
    if (items > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    pe.num_items = (int)items;
    pe.div_pairs = make_fastdiv(pairs * (uint32_t)pe.kchunks);
    pe.div_req = make_fastdiv(pairs * (uint32_t)pe.kchunks * (uint32_t)desc->num_kv_heads);
    pe.num_ctas = (int)std::min<int64_t>(items, ds->sm_count > 0 ? ds->sm_count : 1);
  }
  ExtendPartialParams pp{};
  pp.o = ws_o;
  pp.lse = ws_lse;
  pp.o_stride = (int64_t)slots * desc->head_dim;
  pp.lse_stride = slots;
  if (side_stream(ds) != cudaSuccess) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(ds->side_mu);
  e = cudaEventRecord(ds->fork, stream);
  if (e != cudaSuccess) return PKV_ERR_CUDA;
  e = cudaStreamWaitEvent(ds->side, ds->fork, 0);
  if (e == cudaSuccess)
    e = launch_extend_prefix_pass(kmap, vmap, qmap, pe, pp, desc->head_dim,
                                  (int)desc->cache_dtype, (int)act_dtype, ds->side);
  // join even after a failure, so that the caller's stream (or a capture in
  // progress) never keeps the side stream forked
  const cudaError_t ej = cudaEventRecord(ds->join, ds->side);
  if (e != cudaSuccess || ej != cudaSuccess) {
    cudaStreamWaitEvent(stream, ds->join, 0);
    return PKV_ERR_CUDA;
  }

  // 2. each request's own tokens (current token appended first) -> the slots
  //    after the prefix's, then, once the prefix pass has joined, the merge
  //    of all of them
  DecodeParams p;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.q = q;
  p.out = out;
  p.lse_out = lse_out;
  p.ws_o = ws_o;
  p.ws_lse = ws_lse;
  p.err = ds->err;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = desc->num_blocks;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = desc->num_kv_heads;
  p.group = group;
  p.bs_shift = desc->block_size == 16 ? 4 : 5;
  p.chunk = pl.chunk;
  p.num_splits = pl.splits;
  p.scale_log2 = scale_log2;
  p.out_scale = output_scale(desc);
  DecodeExtraParams ap{};
  ap.k_new = k_new;
  ap.v_new = v_new;
  ap.k_cache = k_cache;
  ap.v_cache = v_cache;
  ap.k_scale = desc->k_scale;
  ap.v_scale = desc->v_scale;
  ap.k_rcp = (float)(1.0 / (double)desc->k_scale);
  ap.v_rcp = (float)(1.0 / (double)desc->v_scale);
  ap.group_indptr = group_indptr;
  ap.group_prefix_lens = group_prefix_lens;
  ap.num_groups = num_groups;
  ap.ws_span = reinterpret_cast<int2*>(static_cast<uint8_t*>(workspace) + pl.ws_span_offset);
  ap.prefix_slots = prefix_slots;
  ap.prefix_chunk = pe.kchunk_keys;
  ap.prefix_chunks = pe.kchunks;
  e = launch_decode_cascade(kmap, vmap, p, ap, desc->head_dim, (int)desc->cache_dtype,
                            (int)act_dtype, stream, ds->join);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// Decode, optionally with the current token's K/V (k_new/v_new, [B][Hkv][D]
// act dtype) appended to position seq_len-1 inside the decode kernel.
static pkv_status decode_common(const pkv_cache_desc* desc, const void* k_cache,
                                const void* v_cache, const void* k_new, const void* v_new,
                                const void* q, void* out, pkv_dtype act_dtype,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* seq_lens, int32_t batch, int32_t num_q_heads,
                                float sm_scale, int32_t max_seq_len, int32_t num_splits,
                                float* lse_out, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if ((st = check_act(desc, act_dtype)) != PKV_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_seq_len < 0 ||
      num_splits < 0 || !std::isfinite(sm_scale))
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % desc->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int group = num_q_heads / desc->num_kv_heads;
  if (batch == 0) return PKV_OK;
  if (batch > 65535 || desc->num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
  if (!k_cache || !v_cache || !q || !out || !block_tables || !seq_lens)
    return PKV_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 4) || !aligned(out, 2))
    return PKV_ERR_INVALID_ARG;
  if ((k_new == nullptr) != (v_new == nullptr)) return PKV_ERR_INVALID_ARG;
  if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16))) return PKV_ERR_INVALID_ARG;
  cudaError_t e;
  DeviceState* ds = device_state(&e);
  if (!ds) return PKV_ERR_CUDA;
  const DecodePlan pl = plan_decode(desc, batch, num_q_heads, max_seq_len, num_splits, ds->sm_count);
  if (pl.ws_bytes > 0 && (!workspace || workspace_bytes < pl.ws_bytes || !aligned(workspace, 256)))
    return PKV_ERR_WORKSPACE;
  if (pl.splits > 65535) return PKV_ERR_UNSUPPORTED;
  CUtensorMap kmap, vmap;
  if ((st = make_page_map(&kmap, k_cache, desc)) != PKV_OK) return st;
  if ((st = make_page_map(&vmap, v_cache, desc)) != PKV_OK) return st;
  DecodeParams p;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.q = q;
  p.out = out;
  p.lse_out = lse_out;
  p.ws_o = pl.ws_bytes ? reinterpret_cast<float*>(workspace) : nullptr;
  p.ws_lse = pl.ws_bytes ? reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) + pl.ws_lse_offset)
                         : nullptr;
  p.err = ds->err;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = desc->num_blocks;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = desc->num_kv_heads;
  p.group = group;
  p.bs_shift = desc->block_size == 16 ? 4 : 5;
  p.chunk = pl.chunk;
  p.num_splits = pl.splits;
  p.scale_log2 = score_scale_log2(desc, sm_scale);
  p.out_scale = output_scale(desc);
  DecodeExtraParams ap{};
  ap.k_new = k_new;
  ap.v_new = v_new;
  ap.k_cache = const_cast<void*>(k_cache);
  ap.v_cache = const_cast<void*>(v_cache);
  ap.k_scale = desc->k_scale;
  ap.v_scale = desc->v_scale;
  ap.k_rcp = (float)(1.0 / (double)desc->k_scale);
  ap.v_rcp = (float)(1.0 / (double)desc->v_scale);
  e = launch_decode(kmap, vmap, p, ap, desc->head_dim, (int)desc->cache_dtype, (int)act_dtype,
                    stream);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

pkv_status pkv_paged_decode_attn(const pkv_cache_desc* desc, const void* k_cache,
                                 const void* v_cache, const void* q, void* out,
                                 pkv_dtype act_dtype, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t batch, int32_t num_q_heads, float sm_scale,
                                 int32_t max_seq_len, int32_t num_splits, float* lse_out,
                                 void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return decode_common(desc, k_cache, v_cache, nullptr, nullptr, q, out, act_dtype, block_tables,
                       max_blocks_per_seq, seq_lens, batch, num_q_heads, sm_scale, max_seq_len,
                       num_splits, lse_out, workspace, workspace_bytes, stream);
}

pkv_status pkv_paged_decode_attn_append(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                                        const void* k_new, const void* v_new, const void* q,
                                        void* out, pkv_dtype act_dtype,
                                        const int32_t* block_tables, int32_t max_blocks_per_seq,
                                        const int32_t* seq_lens, int32_t batch,
                                        int32_t num_q_heads, float sm_scale, int32_t max_seq_len,
                                        int32_t num_splits, float* lse_out, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream) {
  if (!k_new || !v_new) return PKV_ERR_INVALID_ARG;
  return decode_common(desc, k_cache, v_cache, k_new, v_new, q, out, act_dtype, block_tables,
                       max_blocks_per_seq, seq_lens, batch, num_q_heads, sm_scale, max_seq_len,
                       num_splits, lse_out, workspace, workspace_bytes, stream);
}

size_t pkv_extend_workspace_bytes(const pkv_cache_desc* desc, int32_t batch, int32_t num_q_heads,
                                  int32_t total_q_rows, int32_t max_total_len) {
  // every dtype, fp8 included, is read straight from the cache: no scratch
  (void)desc; (void)batch; (void)num_q_heads; (void)total_q_rows; (void)max_total_len;
  return 0;
}

}  // extern "C"

// Shared-prefix extend: the groups (null group_indptr: plain extend).
struct ExtendGroups {
  const int32_t* group_indptr;
  const int32_t* group_shared;
  int32_t num_groups;
  int32_t max_group_rows;
};

// Extend, optionally with the suffix's K/V (k_new/v_new, [rows][Hkv][D] in
// the act dtype) written into the cache before the extend kernel runs, or
// (groups) with the rows of each group's requests packed into shared tiles.
// Workspace the shared-prefix extend can use: f16 copies of the pools (the same
// block ids) into which the call widens the pages it reads, so that the kernel
// takes them as f16 instead of converting every tile -- the V pool of a bf16
// cache, the K and V pools of an fp8 cache (K first); none for an f16 cache.
static size_t shared_prefix_pool16_bytes(const pkv_cache_desc* d) {
  return align256((size_t)d->num_blocks * d->num_kv_heads * d->block_size * d->head_dim * 2);
}
static size_t shared_prefix_widen_bytes(const pkv_cache_desc* d) {
  if (d->cache_dtype == PKV_BF16) return shared_prefix_pool16_bytes(d);
  if (d->cache_dtype == PKV_FP8_E4M3) return 2 * shared_prefix_pool16_bytes(d);
  return 0;
}
// The plain extend's optional workspace: the same pools, then a counter, a
// claim flag per block and a list of the blocks claimed (requests may share
// blocks without the call knowing it).
static size_t plain_widen_bytes(const pkv_cache_desc* d) {
  const size_t pools = shared_prefix_widen_bytes(d);
  return pools ? pools + align256((1 + 2 * (size_t)d->num_blocks) * sizeof(int32_t)) : 0;
}

static pkv_status extend_common(const pkv_cache_desc* desc, const void* k_cache,
                                const void* v_cache, const void* k_new, const void* v_new,
                                const void* q, void* out, pkv_dtype act_dtype,
                                const int32_t* q_indptr, const int32_t* prefix_lens,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                int32_t batch, int32_t num_q_heads, float sm_scale,
                                int32_t total_q_rows, int32_t max_suffix_len,
                                int32_t max_total_len, float* lse_out, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream,
                                const ExtendGroups* groups = nullptr) {
  pkv_status st = check_desc(desc);
  if (st != PKV_OK) return st;
  if ((st = check_act(desc, act_dtype)) != PKV_OK) return st;
  if (batch < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || total_q_rows < 0 ||
      max_suffix_len < 0 || max_total_len < 0 || !std::isfinite(sm_scale) || !(sm_scale > 0.f))
    return PKV_ERR_INVALID_ARG;
  if (num_q_heads % desc->num_kv_heads != 0) return PKV_ERR_INVALID_ARG;
  const int group = num_q_heads / desc->num_kv_heads;
  if (!extend_supported(desc->head_dim, (int)desc->cache_dtype, (int)act_dtype, group))
    return PKV_ERR_UNSUPPORTED;
  // no call needs scratch; either may take one to widen the pages it reads
  // once instead of per tile (a plain call whose workspace is smaller than
  // that, such as the 0 bytes of pkv_extend_workspace_bytes, does without)
  const size_t plain_bytes = groups ? 0 : plain_widen_bytes(desc);
  const bool widen_plain = !groups && workspace != nullptr && plain_bytes > 0 &&
                           workspace_bytes >= plain_bytes && aligned(workspace, 256) &&
                           batch <= 65535;
  const size_t widen_bytes = groups ? shared_prefix_widen_bytes(desc) : 0;
  // (the widening pass takes one CTA row per request: larger batches keep the
  // per-tile conversion)
  const bool widen = groups && workspace != nullptr && widen_bytes > 0 && batch <= 65535;
  if (widen && (workspace_bytes < widen_bytes || !aligned(workspace, 256))) return PKV_ERR_WORKSPACE;
  if (groups) {
    if (groups->num_groups < 0 || groups->max_group_rows < 0 || groups->num_groups > batch)
      return PKV_ERR_INVALID_ARG;
    if (batch > 0 && groups->num_groups == 0) return PKV_ERR_INVALID_ARG;
  }
  const int32_t rows_hint = groups ? groups->max_group_rows : max_suffix_len;
  if (batch == 0 || total_q_rows == 0 || rows_hint == 0) return PKV_OK;
  if (!k_cache || !v_cache || !q || !out || !block_tables || !q_indptr || !prefix_lens)
    return PKV_ERR_INVALID_ARG;
  if (groups && (!groups->group_indptr || !groups->group_shared)) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16))
    return PKV_ERR_INVALID_ARG;
  cudaError_t e;
  DeviceState* ds = device_state(&e);
  if (!ds) return PKV_ERR_CUDA;
  CUtensorMap kmap, vmap, qmap, omap;
  if ((st = make_page_map(&kmap, k_cache, desc)) != PKV_OK) return st;
  if ((st = make_page_map(&vmap, v_cache, desc)) != PKV_OK) return st;
  if ((st = make_q_map(&qmap, q, desc->head_dim, num_q_heads, total_q_rows, group)) != PKV_OK)
    return st;
  // the output has q's shape and layout: the same map over out
  if ((st = make_q_map(&omap, out, desc->head_dim, num_q_heads, total_q_rows, group)) != PKV_OK)
    return st;
  ExtendParams p{};
  p.q_indptr = q_indptr;
  p.prefix_lens = prefix_lens;
  p.block_tables = block_tables;
  p.group_indptr = groups ? groups->group_indptr : nullptr;
  p.group_shared = groups ? groups->group_shared : nullptr;
  p.q = q;
  p.out = out;
  p.lse_out = lse_out;
  p.err = ds->err;
  p.max_blocks = max_blocks_per_seq;
  p.num_blocks = desc->num_blocks;
  p.batch = batch;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = desc->num_kv_heads;
  p.out_32b = aligned(out, 32) ? 1 : 0;
  p.out_tma = 1;
  p.bs_shift = desc->block_size == 16 ? 4 : 5;
  p.total_rows = total_q_rows;
  p.scale_log2 = score_scale_log2(desc, sm_scale);
  p.out_scale = output_scale(desc);
  // work items per (request or group, kv head): pairs of row tiles
  if (!plan_extend(p, groups ? groups->num_groups : batch, desc->num_kv_heads, group, rows_hint,
                   ds->sm_count))
    return PKV_ERR_UNSUPPORTED;
  if (groups) {
    int cache_dt = (int)desc->cache_dtype;
    if (widen) {
      // the pages the call reads, widened in the workspace (same block ids),
      // then read by the kernel through maps over those pools: V as f16, an
      // fp8 cache's K in the queries' type; the scales of an fp8 cache stay
      // folded into p's softmax and output scales
      pkv_cache_desc d16 = *desc;
      d16.cache_dtype = PKV_F16;
      const bool fp8 = desc->cache_dtype == PKV_FP8_E4M3;
      void* k16 = fp8 ? workspace : nullptr;
      void* v16 = static_cast<uint8_t*>(workspace) + (fp8 ? shared_prefix_pool16_bytes(desc) : 0);
      if (fp8 && (st = make_page_map(&kmap, k16, &d16)) != PKV_OK) return st;
      if ((st = make_page_map(&vmap, v16, &d16)) != PKV_OK) return st;
      e = launch_widen(fp8 ? DT_E4M3 : DT_BF16, (int)act_dtype, k_cache, v_cache, k16, v16, p,
                       groups->num_groups, desc->head_dim, desc->block_size, max_total_len, stream);
      if (e != cudaSuccess) return PKV_ERR_CUDA;
      // K bf16 (cache or widened) with f16 V; an fp8 cache under f16 queries
      // is then an f16 cache
      cache_dt = act_dtype == PKV_BF16 ? DT_BF16_V16 : DT_F16;
    }
    e = launch_extend_shared(kmap, vmap, qmap, omap, p, desc->head_dim, cache_dt, (int)act_dtype,
                             stream);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
  }
  if (k_new) {
    // the suffix's K/V first (its slots computed from the extend layout), then
    // the extend kernel reads them back; two launches in stream order
    AppendParams ap{};
    ap.k_cache = const_cast<void*>(k_cache);
    ap.v_cache = const_cast<void*>(v_cache);
    ap.k_new = k_new;
    ap.v_new = v_new;
    ap.slots = nullptr;
    ap.err = ds->err;
    ap.num_tokens = total_q_rows;
    ap.num_kv_heads = desc->num_kv_heads;
    ap.head_dim = desc->head_dim;
    ap.block_size = desc->block_size;
    ap.num_blocks = desc->num_blocks;
    ap.k_scale = desc->k_scale;
    ap.v_scale = desc->v_scale;
    ap.q_indptr = q_indptr;
    ap.prefix_lens = prefix_lens;
    ap.block_tables = block_tables;
    ap.batch = batch;
    ap.max_blocks = max_blocks_per_seq;
    e = launch_append(ap, (int)desc->cache_dtype, (int)act_dtype, stream);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
  }
  int cache_dt = (int)desc->cache_dtype;
  if (widen_plain) {
    // the pages the call reads, each block widened once (claimed in the
    // workspace) into 16-bit pools read through maps over them
    pkv_cache_desc d16 = *desc;
    d16.cache_dtype = PKV_F16;
    const bool fp8 = desc->cache_dtype == PKV_FP8_E4M3;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    void* k16 = fp8 ? base : nullptr;
    void* v16 = base + (fp8 ? shared_prefix_pool16_bytes(desc) : 0);
    int32_t* claims = reinterpret_cast<int32_t*>(base + shared_prefix_widen_bytes(desc));
    if (fp8 && (st = make_page_map(&kmap, k16, &d16)) != PKV_OK) return st;
    if ((st = make_page_map(&vmap, v16, &d16)) != PKV_OK) return st;
    e = launch_widen_claim(fp8 ? DT_E4M3 : DT_BF16, (int)act_dtype, k_cache, v_cache, k16, v16,
                           claims, p, desc->head_dim, desc->block_size, max_total_len,
                           ds->sm_count, stream);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    cache_dt = act_dtype == PKV_BF16 ? DT_BF16_V16 : DT_F16;
  }
  e = launch_extend(kmap, vmap, qmap, omap, p, desc->head_dim, cache_dt, (int)act_dtype, stream);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" {

pkv_status pkv_paged_extend_attn(const pkv_cache_desc* desc, const void* k_cache,
                                 const void* v_cache, const void* q, void* out,
                                 pkv_dtype act_dtype, const int32_t* q_indptr,
                                 const int32_t* prefix_lens, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, int32_t batch, int32_t num_q_heads,
                                 float sm_scale, int32_t total_q_rows, int32_t max_suffix_len,
                                 int32_t max_total_len, float* lse_out, void* workspace,
                                 size_t workspace_bytes, cudaStream_t stream) {
  return extend_common(desc, k_cache, v_cache, nullptr, nullptr, q, out, act_dtype, q_indptr,
                       prefix_lens, block_tables, max_blocks_per_seq, batch, num_q_heads,
                       sm_scale, total_q_rows, max_suffix_len, max_total_len, lse_out, workspace,
                       workspace_bytes, stream);
}

size_t pkv_extend_widen_workspace_bytes(const pkv_cache_desc* desc) {
  if (check_desc(desc) != PKV_OK) return 0;
  return plain_widen_bytes(desc);
}

size_t pkv_extend_shared_prefix_workspace_bytes(const pkv_cache_desc* desc) {
  if (check_desc(desc) != PKV_OK) return 0;
  return shared_prefix_widen_bytes(desc);
}

pkv_status pkv_paged_extend_attn_shared_prefix(
    const pkv_cache_desc* desc, const void* k_cache, const void* v_cache, const void* q, void* out,
    pkv_dtype act_dtype, const int32_t* q_indptr, const int32_t* prefix_lens,
    const int32_t* block_tables, int32_t max_blocks_per_seq, int32_t batch, int32_t num_q_heads,
    float sm_scale, int32_t total_q_rows, const int32_t* group_indptr,
    const int32_t* group_shared_lens, int32_t num_groups, int32_t max_group_rows,
    int32_t max_total_len, float* lse_out, void* workspace, size_t workspace_bytes,
    cudaStream_t stream) {
  const ExtendGroups groups{group_indptr, group_shared_lens, num_groups, max_group_rows};
  return extend_common(desc, k_cache, v_cache, nullptr, nullptr, q, out, act_dtype, q_indptr,
                       prefix_lens, block_tables, max_blocks_per_seq, batch, num_q_heads,
                       sm_scale, total_q_rows, max_group_rows, max_total_len, lse_out, workspace,
                       workspace_bytes, stream, &groups);
}

pkv_status pkv_paged_extend_attn_append(const pkv_cache_desc* desc, void* k_cache, void* v_cache,
                                        const void* k_new, const void* v_new, const void* q,
                                        void* out, pkv_dtype act_dtype, const int32_t* q_indptr,
                                        const int32_t* prefix_lens, const int32_t* block_tables,
                                        int32_t max_blocks_per_seq, int32_t batch,
                                        int32_t num_q_heads, float sm_scale, int32_t total_q_rows,
                                        int32_t max_suffix_len, int32_t max_total_len,
                                        float* lse_out, cudaStream_t stream) {
  if (!k_new || !v_new) return PKV_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16)) return PKV_ERR_INVALID_ARG;
  return extend_common(desc, k_cache, v_cache, k_new, v_new, q, out, act_dtype, q_indptr,
                       prefix_lens, block_tables, max_blocks_per_seq, batch, num_q_heads,
                       sm_scale, total_q_rows, max_suffix_len, max_total_len, lse_out, nullptr, 0,
                       stream);
}

}  // extern "C"
