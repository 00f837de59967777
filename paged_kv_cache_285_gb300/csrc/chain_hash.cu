// Chain hashes of full KV blocks, as block identifiers for prefix caching.
//
// "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 05: each
// KV block's hash is built from its parent block's hash, the block's token ids
// and optional extra data (a LoRA or multimodal id), so equal token prefixes
// give equal hash chains and a new request allocates from its first miss;
// section 06: a per-tenant salt goes into the identifier so that equal
// prompts of different tenants never share blocks.  The pages fix no hash
// function.  This one is built on the SplitMix64 finalizer (Vigna):
//   mix(z): z ^= z >> 30; z *= 0xBF58476D1CE4E5B9; z ^= z >> 27;
//           z *= 0x94D049BB133111EB; z ^= z >> 31
//   content(block) = c after c = mix(c + G + t) for each token id t (as an
//                    unsigned 32-bit value), c starting at 0, G = 0x9E3779B97F4A7C15
//   h_i = mix((h_{i-1} ^ content(block i)) + G), h_{-1} = the request's salt
// (extra data goes into the salt).  Two levels so that the block contents
// hash in parallel and only the cheap chain step is sequential.
#include "internal.h"

namespace pkv {

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;
constexpr int kThreads = 64;         // warp 0: chain; warp 1: block contents
constexpr int kRoundBlocks = 32;     // blocks per round, one per content lane
constexpr int kRoundTokens = 1024;   // tokens staged per round (fewer blocks if larger)
constexpr int kStages = 3;           // token buffers: copy r+2, hash r+1, (free)

// Blocks per round: one per content lane, at most kRoundTokens tokens, at least 1.
__host__ __device__ __forceinline__ int round_blocks(int block_size) {
  const int c = kRoundTokens / block_size;
  return c < 1 ? 1 : (c > kRoundBlocks ? kRoundBlocks : c);
}

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

__device__ __forceinline__ void cp_async4(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem))),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_1() {
  asm volatile("cp.async.wait_group 1;" ::: "memory");
}

// One CTA of two warps per request, in rounds of round_blocks() blocks.  In
// round r the whole CTA starts the asynchronous copy of round r+2's tokens
// into shared memory, warp 1 hashes the contents of round r+1 (one block per
// lane), and lane 0 of warp 0 runs the chain over round r's contents; warp 0
// then stores round r's hashes with coalesced writes.  Only the chain is
// sequential, so a request takes about (its blocks) x (one chain step).
__global__ void __launch_bounds__(kThreads) chain_hash_kernel(const ChainHashParams p) {
  extern __shared__ int32_t tok_s[];  // kStages x round_blocks x block_size tokens
  __shared__ uint64_t content_s[2][kRoundBlocks];
  __shared__ uint64_t chain_s[kRoundBlocks];
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bs = p.block_size;
  const int cb = round_blocks(bs);
  const int stage_tok = cb * bs;
  const int64_t base = p.token_indptr[b];
  const int64_t len = (int64_t)p.token_indptr[b + 1] - base;
  int64_t nblk = len > 0 ? len / bs : 0;
  if (nblk > p.max_blocks) {
    if (threadIdx.x == 0 && p.err) atomicCAS(p.err, 0, 5);
    nblk = p.max_blocks;
  }
  const int64_t nrounds = (nblk + cb - 1) / cb;
  auto nb_of = [&](int64_t r) -> int {
    const int64_t left = nblk - r * cb;
    return (int)(left < cb ? left : cb);
  };
  // Start the copy of round r's tokens (an empty group past the end keeps the
  // group count per thread uniform).
  auto copy_round = [&](int64_t r) {
    if (r < nrounds) {
      const int ntok = nb_of(r) * bs;
      const int32_t* src = p.tokens + base + r * (int64_t)stage_tok;
      int32_t* dst = tok_s + (int)(r % kStages) * stage_tok;
      for (int i = threadIdx.x; i < ntok; i += kThreads) cp_async4(dst + i, src + i);
    }
    cp_async_commit();
  };
  auto hash_round = [&](int64_t r) {  // warp 1
    if (r < nrounds && lane < nb_of(r)) {
      const int32_t* t = tok_s + (int)(r % kStages) * stage_tok + lane * bs;
      uint64_t c = 0;
      for (int j = 0; j < bs; ++j) c = mix64(c + kGolden + (uint64_t)(uint32_t)t[j]);
      content_s[r & 1][lane] = c;
    }
  };

  copy_round(0);
  copy_round(1);
  cp_async_wait_1();
  __syncthreads();
  if (warp == 1) hash_round(0);
  uint64_t h = p.salts ? p.salts[b] : 0ull;  // lane 0 of warp 0 carries the chain
  for (int64_t r = 0; r < nrounds; ++r) {
    copy_round(r + 2);
    cp_async_wait_1();  // this thread's copies of round r+1 have landed
    __syncthreads();    // ... and everyone's; round r's contents are complete
    if (warp == 1) {
      hash_round(r + 1);
    } else {
      const int nb = nb_of(r);
      if (lane == 0) {
        const uint64_t* cs = content_s[r & 1];
        for (int i = 0; i < nb; ++i) {
          h = mix64((h ^ cs[i]) + kGolden);
          chain_s[i] = h;
        }
      }
      __syncwarp();
      if (lane < nb) p.hashes[(int64_t)b * p.max_blocks + r * cb + lane] = chain_s[lane];
      __syncwarp();
    }
  }
}

}  // namespace

cudaError_t launch_chain_hash(const ChainHashParams& p, int batch, cudaStream_t stream) {
  if (batch <= 0) return cudaSuccess;
  const size_t smem = (size_t)kStages * round_blocks(p.block_size) * p.block_size * sizeof(int32_t);
  if (smem > 40 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(chain_hash_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  chain_hash_kernel<<<batch, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
