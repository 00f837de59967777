// KV append: scatter the K/V rows of new tokens into their cache slots.
//
// "KV Cache에 대해 알아보자 (Feat. Attention)", §3: at each decode step the
// new token's K and V are added to the cache; with paging the destination is
// the token's slot (physical block, offset) -- "PagedAttention과
// RadixAttention으로 LLM KV 캐시 최적화", section 02.
//
// One thread moves 8 elements of one (token, kv head) row for K and for V (16
// for the fp8 store), with coalesced 16-byte loads and stores.
// 16-bit caches copy the bits; fp8 caches store e4m3(fp32(x) / scale) -- the
// correctly rounded fp32 quotient (a multiply by the reciprocal, with the
// division only where the two could round differently) and a saturating
// round-to-nearest-even convert (cvt.rn.satfinite).  Slots whose block lies outside the pool are
// skipped and reported in the error word; negative slots are skipped silently.
#include "internal.h"
#include "ptx.cuh"

namespace pkv {

namespace {

template <int AT>
__device__ __forceinline__ float act_to_f32(uint16_t bits) {
  if constexpr (AT == DT_BF16) return __uint_as_float((uint32_t)bits << 16);
  else return __half2float(__ushort_as_half(bits));
}

// Elements of a row one thread moves: 8 (one 16-byte input vector) for a
// 16-bit copy; 16 for the fp8 store (two input vectors per tensor in flight
// and one 16-byte store of codes).
template <int CT>
__host__ __device__ constexpr int append_ept() { return CT == DT_E4M3 ? 16 : 8; }

template <int CT, int AT, int HD>
__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
  constexpr int EPT = append_ept<CT>();
  constexpr int VPR = HD / EPT;  // threads per row (a power of two)
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = p.num_tokens * p.num_kv_heads * VPR;
  if (idx >= total) return;
  const int v = (int)(idx & (VPR - 1));
  const int64_t row = (int64_t)((uint64_t)idx / VPR);  // (token, kv head) row
  int64_t t;
  int g;
  if (p.rows_fit32) {  // row < 2^31: the kv-head split as a multiply-high
    const uint32_t q = p.div_hkv.div((uint32_t)row);
    t = q;
    g = (int)((uint32_t)row - q * (uint32_t)p.num_kv_heads);
  } else {
    t = row / p.num_kv_heads;
    g = (int)(row - t * p.num_kv_heads);
  }
  const int64_t bmask = p.block_size - 1;  // block sizes are powers of two
  int64_t slot;
  if (p.slots) {
    slot = p.slots[t];
  } else {
    int lo = 0, hi = p.batch;  // the request of suffix row t
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (__ldg(p.q_indptr + mid) <= t) lo = mid;
      else hi = mid;
    }
    const int64_t pos = (int64_t)__ldg(p.prefix_lens + lo) + (t - __ldg(p.q_indptr + lo));
    if (pos < 0 || (pos >> p.bs_shift) >= p.max_blocks) {
      if (v == 0 && p.err) atomicCAS(p.err, 0, 3);
      return;
    }
    const int32_t b = __ldg(p.block_tables + (int64_t)lo * p.max_blocks + (pos >> p.bs_shift));
    // a negative block id is outside the pool too (reported below)
    slot = ((b < 0 ? (int64_t)p.num_blocks : (int64_t)b) << p.bs_shift) + (pos & bmask);
  }
  if (slot < 0) return;
  const int64_t blk = slot >> p.bs_shift, off = slot & bmask;
  if (blk >= p.num_blocks) {
    if (v == 0 && p.err) atomicCAS(p.err, 0, 2);
    return;
  }
  const int64_t src = idx * EPT;  // row * HD + v * EPT
  const int64_t dst = (((blk * p.num_kv_heads + g) << p.bs_shift) + off) * HD + v * EPT;
  const uint4* ksrc = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.k_new) + src);
  const uint4* vsrc = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.v_new) + src);
  if constexpr (CT != DT_E4M3) {
    const uint4 kx = __ldg(ksrc), vx = __ldg(vsrc);
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.k_cache) + dst) = kx;
    *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.v_cache) + dst) = vx;
  } else {
    const uint4 kx0 = __ldg(ksrc), kx1 = __ldg(ksrc + 1);
    const uint4 vx0 = __ldg(vsrc), vx1 = __ldg(vsrc + 1);
    const uint32_t kw[8] = {kx0.x, kx0.y, kx0.z, kx0.w, kx1.x, kx1.y, kx1.z, kx1.w};
    const uint32_t vw[8] = {vx0.x, vx0.y, vx0.z, vx0.w, vx1.x, vx1.y, vx1.z, vx1.w};
    uint32_t ko[4], vo[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      uint32_t kb = 0, vb = 0;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint32_t wk = kw[2 * h + q], wv = vw[2 * h + q];
        const float k0 = quot_for_e4m3(act_to_f32<AT>((uint16_t)(wk & 0xFFFFu)), p.k_scale, p.k_rcp);
        const float k1 = quot_for_e4m3(act_to_f32<AT>((uint16_t)(wk >> 16)), p.k_scale, p.k_rcp);
        const float v0 = quot_for_e4m3(act_to_f32<AT>((uint16_t)(wv & 0xFFFFu)), p.v_scale, p.v_rcp);
        const float v1 = quot_for_e4m3(act_to_f32<AT>((uint16_t)(wv >> 16)), p.v_scale, p.v_rcp);
        kb |= f32x2_to_e4m3x2(k0, k1) << (16 * q);
        vb |= f32x2_to_e4m3x2(v0, v1) << (16 * q);
      }
      ko[h] = kb;
      vo[h] = vb;
    }
    *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.k_cache) + dst) = make_uint4(ko[0], ko[1], ko[2], ko[3]);
    *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.v_cache) + dst) = make_uint4(vo[0], vo[1], vo[2], vo[3]);
  }
}

template <int CT, int AT>
cudaError_t launch_append_t(const AppendParams& in, cudaStream_t stream) {
  const int64_t total = in.num_tokens * in.num_kv_heads * (in.head_dim / append_ept<CT>());
  if (total == 0) return cudaSuccess;
  AppendParams p = in;
  p.bs_shift = p.block_size == 16 ? 4 : 5;
  p.k_rcp = (float)(1.0 / (double)p.k_scale);
  p.v_rcp = (float)(1.0 / (double)p.v_scale);
  p.rows_fit32 = p.num_tokens * p.num_kv_heads < ((int64_t)1 << 31) ? 1 : 0;
  p.div_hkv = make_fastdiv((uint32_t)p.num_kv_heads);
  const unsigned blocks = (unsigned)((total + 255) / 256);
  if (p.head_dim == 64) append_kernel<CT, AT, 64><<<blocks, 256, 0, stream>>>(p);
  else append_kernel<CT, AT, 128><<<blocks, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int cache_dt, int act_dt, cudaStream_t stream) {
  if (cache_dt == DT_F16 && act_dt == DT_F16) return launch_append_t<DT_F16, DT_F16>(p, stream);
  if (cache_dt == DT_BF16 && act_dt == DT_BF16) return launch_append_t<DT_BF16, DT_BF16>(p, stream);
  if (cache_dt == DT_E4M3 && act_dt == DT_F16) return launch_append_t<DT_E4M3, DT_F16>(p, stream);
  if (cache_dt == DT_E4M3 && act_dt == DT_BF16) return launch_append_t<DT_E4M3, DT_BF16>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pkv
