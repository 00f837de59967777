// Paged decode for callers that cannot allocate device memory.
//
// pkv_paged_decode_attn needs a caller-provided workspace for its split-KV
// partial results.  Some callers cannot provide one: code that runs where a
// device allocation is not allowed or not available to it -- for example a
// plugin inside an engine that owns all device memory and hands out only the
// tensors of a call, or a real-time path where cudaMalloc (which can
// synchronise the device and may fail under memory pressure) is forbidden.
// For them, pkv_paged_decode_attn_noalloc runs the same decode with the
// partials placed in a fixed scratch array that is part of this library's
// device image, so the call itself allocates nothing.
//
// The array is PKV_NOALLOC_SCRATCH_BYTES long and exists on every device that
// loads the library, for as long as the process lives.  All calls on a device
// share it: two calls whose kernels overlap on the GPU (different streams, or
// graph branches running concurrently) race on it and may return wrong
// results.  Nothing in it needs to start at zero -- every partial is written
// before it is read within the same call -- so it is never cleared.
#include <mutex>

#include "../../include/pkv.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Per-device cache of the scratch array's device address.  Only a successful
// lookup is kept: a failed one (for example a sticky error left by earlier
// unrelated work, or a first call made while a stream is being captured) is
// retried by the next call instead of failing every later call on that device.
struct ScratchState {
  std::mutex mu;
  void* ptr = nullptr;
};
ScratchState g_scratch[kMaxDevices];

// Device address of the scratch array on the current device.  In host code the
// array's name is only a host-side stand-in, so the address must be asked of
// the runtime, once per device, while that device is current.
void* scratch_for_current_device(pkv_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *st = PKV_ERR_CUDA;
    return nullptr;
  }
  ScratchState* s = &g_scratch[dev];
  std::lock_guard<std::mutex> lock(s->mu);
  if (!s->ptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) {
      *st = PKV_ERR_CUDA;
      return nullptr;
    }
    s->ptr = p;
  }
  *st = PKV_OK;
  return s->ptr;
}

}  // namespace

extern "C" pkv_status pkv_paged_decode_attn_noalloc(
    const pkv_cache_desc* desc, const void* k_cache, const void* v_cache, const void* q,
    void* out, pkv_dtype act_dtype, const int32_t* block_tables, int32_t max_blocks_per_seq,
    const int32_t* seq_lens, int32_t batch, int32_t num_q_heads, float sm_scale,
    int32_t max_seq_len, int32_t num_splits, float* lse_out, cudaStream_t stream) {
  const size_t need =
      pkv_decode_workspace_bytes(desc, batch, num_q_heads, max_seq_len, num_splits);
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;
  pkv_status st;
  void* scratch = scratch_for_current_device(&st);
  if (!scratch) return st;
  return pkv_paged_decode_attn(desc, k_cache, v_cache, q, out, act_dtype, block_tables,
                               max_blocks_per_seq, seq_lens, batch, num_q_heads, sm_scale,
                               max_seq_len, num_splits, lse_out, scratch,
                               (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}
