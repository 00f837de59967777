// fp8 (e4m3) pages -> 16-bit shadow pages for the extend path.
//
// The extend kernel's tensor-core products take 16-bit operands of one type
// (Q with K, P with V).  For an fp8 cache ("PagedAttention과 RadixAttention으로
// LLM KV 캐시 최적화", fp8 KV with a per-tensor scale) every physical page
// that some request of the call reads is first widened into a shadow pool of
// the activation dtype, with the same [num_blocks][Hkv][bs][D] layout, so the
// block tables apply unchanged.  Pages shared by many requests (a common
// prefix) are claimed once through a per-block flag and widened once.  The
// per-tensor scales are not applied here: k_scale is folded into the softmax
// scale and v_scale into the output scale by the caller, so the widening is
// exact (an e4m3 value has 4 significant bits and a 2^-9 .. 448 range, which
// both f16 and bf16 hold).
#include "internal.h"
#include "ptx.cuh"

namespace pkv {

namespace {

template <int AT>
__global__ void __launch_bounds__(256)
dequant_pages_kernel(const DequantParams p) {
  const int b = blockIdx.y, lb = blockIdx.x;
  const int S = p.q_indptr[b + 1] - p.q_indptr[b];
  const int kv_total = p.prefix_lens[b] + S;
  if (kv_total <= 0 || (lb << p.bs_shift) >= kv_total || lb >= p.max_blocks) return;
  const int blk = p.block_tables[(int64_t)b * p.max_blocks + lb];
  if (blk < 0 || blk >= p.num_blocks) return;  // reported by the extend kernel
  __shared__ int claim;
  if (threadIdx.x == 0) claim = atomicCAS(p.flags + blk, 0, 1);
  __syncthreads();
  if (claim != 0) return;  // another request's CTA widens this page
  const int64_t base = (int64_t)blk * p.page_elems;
  const uint2* k8 = reinterpret_cast<const uint2*>(p.k8 + base);
  const uint2* v8 = reinterpret_cast<const uint2*>(p.v8 + base);
  uint4* k16 = reinterpret_cast<uint4*>(p.k16 + base);
  uint4* v16 = reinterpret_cast<uint4*>(p.v16 + base);
  for (int i = threadIdx.x; i < p.page_elems / 8; i += blockDim.x) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const uint2 c = t ? v8[i] : k8[i];  // 8 codes
      uint32_t h[4];
      h[0] = e4m3x2_to_f16x2(c.x & 0xFFFFu);
      h[1] = e4m3x2_to_f16x2(c.x >> 16);
      h[2] = e4m3x2_to_f16x2(c.y & 0xFFFFu);
      h[3] = e4m3x2_to_f16x2(c.y >> 16);
      if (AT == DT_BF16) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h[q]));
          h[q] = pack2<true>(f.x, f.y);  // exact: at most 4 significant bits
        }
      }
      (t ? v16 : k16)[i] = make_uint4(h[0], h[1], h[2], h[3]);
    }
  }
}

}  // namespace

cudaError_t launch_dequant_pages(const DequantParams& p, int batch, int blocks_per_seq, int act_dt,
                                 cudaStream_t stream) {
  if (batch <= 0 || blocks_per_seq <= 0) return cudaSuccess;
  if (p.page_elems % 8 != 0 || batch > 65535) return cudaErrorInvalidValue;
  const dim3 grid(blocks_per_seq, batch);
  if (act_dt == DT_BF16) dequant_pages_kernel<DT_BF16><<<grid, 256, 0, stream>>>(p);
  else dequant_pages_kernel<DT_F16><<<grid, 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace pkv
