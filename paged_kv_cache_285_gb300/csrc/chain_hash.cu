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
// hash in parallel and only the cheap chain step is sequential: one pass
// hashes every block's contents at once, a second runs each request's chain.
#include "internal.h"

namespace pkv {

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;
constexpr int kContentThreads = 128;  // blocks per CTA of the content pass
constexpr int kMaxChunkCtas = 16;     // content-pass CTAs per request, at most

__device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z ^= z >> 30;
  z *= 0xBF58476D1CE4E5B9ull;
  z ^= z >> 27;
  z *= 0x94D049BB133111EBull;
  z ^= z >> 31;
  return z;
}

// Full blocks of request b (at most max_blocks; more sets the error word when
// `report`).
__device__ __forceinline__ int64_t full_blocks(const ChainHashParams& p, int b, int64_t* base,
                                               bool report) {
  *base = p.token_indptr[b];
  const int64_t len = (int64_t)p.token_indptr[b + 1] - *base;
  int64_t n = len > 0 ? len / p.block_size : 0;
  if (n > p.max_blocks) {
    if (report && p.err) atomicCAS(p.err, 0, 5);
    n = p.max_blocks;
  }
  return n;
}

// Pass 1, all blocks in parallel: CTA (b, y) folds the tokens of blocks
// y * kContentThreads + threadIdx.x, then every gridDim.y * kContentThreads
// further, of request b into their content hashes, stored where the blocks'
// chain hashes go.
__global__ void __launch_bounds__(kContentThreads) block_content_kernel(const ChainHashParams p) {
  const int b = blockIdx.x;
  int64_t base;
  const int64_t nblk = full_blocks(p, b, &base, blockIdx.y == 0 && threadIdx.x == 0);
  const int bs = p.block_size;
  for (int64_t j = (int64_t)blockIdx.y * kContentThreads + threadIdx.x; j < nblk;
       j += (int64_t)gridDim.y * kContentThreads) {
    const int32_t* t = p.tokens + base + j * bs;
    uint64_t c = 0;
    if ((bs & 3) == 0 && (reinterpret_cast<uintptr_t>(t) & 15) == 0) {
      const int4* t4 = reinterpret_cast<const int4*>(t);
      for (int k = 0; k < bs / 4; ++k) {
        const int4 v = __ldg(t4 + k);
        c = mix64(c + kGolden + (uint64_t)(uint32_t)v.x);
        c = mix64(c + kGolden + (uint64_t)(uint32_t)v.y);
        c = mix64(c + kGolden + (uint64_t)(uint32_t)v.z);
        c = mix64(c + kGolden + (uint64_t)(uint32_t)v.w);
      }
    } else {
      for (int k = 0; k < bs; ++k) c = mix64(c + kGolden + (uint64_t)(uint32_t)__ldg(t + k));
    }
    p.hashes[(int64_t)b * p.max_blocks + j] = c;
  }
}

__device__ __forceinline__ void cp_async8(void* dst_smem, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(
                   static_cast<uint32_t>(__cvta_generic_to_shared(dst_smem))),
               "l"(src)
               : "memory");
}

// Pass 2, one lane per request: the chain over the contents of pass 1, in
// place.  Only this step is sequential; one warp instruction advances 32
// requests' chains.  The contents go through shared memory in tiles of 32
// requests x 32 blocks, four buffers deep: while warp 0 chains tile t (lane
// l along row l), warp 1 writes tile t-1 back and starts copying tile t+2
// in, both row-wise (coalesced), so a copy has a whole tile's time to land.  Rows are padded to 33 entries, so lane l's column
// reads hit distinct banks.
constexpr int kTile = 32;
constexpr int kBufs = 4;
__global__ void __launch_bounds__(64) chain_kernel(const ChainHashParams p, int batch) {
  __shared__ uint64_t tile[kBufs][kTile][kTile + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b0 = blockIdx.x * kTile;
  const int nrows = batch - b0 < kTile ? batch - b0 : kTile;
  const int b = b0 + lane;
  int64_t base;
  const int nblk = lane < nrows ? (int)full_blocks(p, b, &base, false) : 0;  // <= max_blocks
  const int ntile = (__reduce_max_sync(0xffffffffu, nblk) + kTile - 1) / kTile;
  int nr[kTile];  // every row's length, in registers (rows past the batch: 0)
#pragma unroll
  for (int r = 0; r < kTile; ++r) nr[r] = __shfl_sync(0xffffffffu, nblk, r);
  uint64_t* const rows = p.hashes + (int64_t)b0 * p.max_blocks;
  // warp 1: start copying tile t in (row r, columns lane); one group per
  // call, empty past the end, so that "all but the newest group" is tile t-1
  auto fetch = [&](int t) {
    if (t < ntile) {
      const int j = t * kTile + lane;
#pragma unroll
      for (int r = 0; r < kTile; ++r)
        if (j < nr[r]) cp_async8(&tile[t % kBufs][r][lane], rows + (int64_t)r * p.max_blocks + j);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  auto landed_but_newest = [&]() {
    asm volatile("cp.async.wait_group 1;" ::: "memory");
    __syncwarp();
  };
  // warp 1: write tile t back
  auto store = [&](int t) {
    const int j = t * kTile + lane;
#pragma unroll
    for (int r = 0; r < kTile; ++r)
      if (j < nr[r]) rows[(int64_t)r * p.max_blocks + j] = tile[t % kBufs][r][lane];
  };

  if (warp == 1) {
    fetch(0);
    fetch(1);
    landed_but_newest();  // tile 0
  }
  __syncthreads();
  uint64_t h = (lane < nrows && p.salts) ? p.salts[b] : 0ull;  // warp 0's chains
  for (int t = 0; t < ntile; ++t) {
    if (warp == 0) {
      uint64_t* row = tile[t % kBufs][lane];
      int kend = nblk - t * kTile;  // this lane's blocks in tile t
      kend = kend < 0 ? 0 : (kend > kTile ? kTile : kend);
      int k0 = 0;
      for (; k0 + 8 <= kend; k0 += 8) {  // 8 contents to registers, then 8 steps
        uint64_t c[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) c[k] = row[k0 + k];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          h = mix64((h ^ c[k]) + kGolden);
          row[k0 + k] = h;
        }
      }
      for (; k0 < kend; ++k0) {
        h = mix64((h ^ row[k0]) + kGolden);
        row[k0] = h;
      }
    } else {
      if (t >= 1) store(t - 1);
      fetch(t + 2);
      landed_but_newest();  // tile t+1
    }
    __syncthreads();  // tile t chained, tile t+1 in, tile t-1 out
  }
  if (warp == 1 && ntile > 0) store(ntile - 1);
}

}  // namespace

cudaError_t launch_chain_hash(const ChainHashParams& p, int batch, cudaStream_t stream) {
  if (batch <= 0 || p.max_blocks <= 0) return cudaSuccess;
  // at most kMaxChunkCtas CTAs per request; the device knows the lengths
  const int64_t chunks = ((int64_t)p.max_blocks + kContentThreads - 1) / kContentThreads;
  const dim3 grid1((unsigned)batch, (unsigned)(chunks < kMaxChunkCtas ? chunks : kMaxChunkCtas));
  block_content_kernel<<<grid1, kContentThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  chain_kernel<<<(unsigned)((batch + kTile - 1) / kTile), 64, 0, stream>>>(p, batch);
  return cudaGetLastError();
}

}  // namespace pkv
