// Paged extend (suffix prefill) on the 5th-generation tensor cores.
//
// "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03: the
// longest cached prefix is reused and only the suffix is computed; prefill is
// compute-bound ("KV Cache에 대해 알아보자 (Feat. Attention)", §3), so this
// is the one dense contraction of the path and runs on tcgen05 with TMEM
// accumulators.
//
// One CTA owns a 128-row tile of packed (suffix token, query head) rows of
// one (request, kv head): with a GQA group of G heads the tile holds 128/G
// consecutive suffix tokens x G heads, all sharing the same K/V.  Row r
// (token i, head j) attends to keys 0 .. prefix + i.  Keys are consumed in
// tiles of 128 read through the block table.
//
// Warp roles (256 threads):
//   warp 0      TMA producer: the Q tile once (3-D map over q), then per key
//               tile the K tile (double-buffered) and the V tile, each as
//               sixteen 16-token x 64-dim boxes addressed through the block
//               table, 128-byte swizzled.
//   warp 1      TMEM owner (512 columns: two S buffers + O) and, on one lane,
//               the MMA issuer: S = Q K^T (M=128, N=128, K=128) into the free
//               S buffer, then O += P V for the previous tile.
//   warps 2-3   V^T builders: each V tile is transposed to [dim][key] and
//               converted to f16 (ldmatrix.trans -> cvt -> stmatrix), zeroing
//               keys past the sequence end, so that the PV product is a
//               K-major f16 x f16 MMA.
//   warps 4-7   softmax (one thread per row): S row from TMEM, causal mask on
//               the diagonal tiles, running max with lazy rescaling (O in TMEM
//               is rescaled only when the max grows by more than 2^8), P in
//               f16 to shared memory, final O / l and LSE.
// P is kept in f16 (11-bit significand) because bf16 P alone would put the
// relative L2 error of the output near 1.5e-3.
#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int BM = 128;       // rows per tile
constexpr int BN = 128;       // keys per tile
constexpr int HD = 128;       // head dim
constexpr int NTHREADS = 256;
constexpr int TILE = BM * HD * 2;   // 32 KB: 128 x 128 16-bit elements
constexpr int CHUNK = 16384;        // one 64-element column block [128 rows][128 B]

constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE;   // two stages
constexpr int OFF_V = OFF_K + 2 * TILE;
constexpr int OFF_VT = OFF_V + TILE;
constexpr int OFF_P = OFF_VT + TILE;
constexpr int OFF_BAR = OFF_P + TILE;
enum {
  B_Q = 0, B_KFULL = 1, B_KFREE = 3, B_VFULL = 5, B_VFREE = 6, B_VTFULL = 7,
  B_SFULL = 8, B_SFREE = 10, B_PFULL = 12, B_PVDONE = 13, NBAR = 14
};
constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_TMEMSLOT + 16 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;     // S buffers at columns 0 and 128
constexpr uint32_t TM_O = 256;   // O accumulator at column 256
constexpr float kLn2f = 0.6931471805599453f;

// byte offset of (row, 16-byte unit) in a [128 rows][128 B] 128B-swizzled block
__device__ __forceinline__ uint32_t sw_off(int row, int unit) {
  return (uint32_t)(row * 128 + ((unit ^ (row & 7)) << 4));
}

__device__ __forceinline__ void set_err(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

template <int CT>
__global__ void __launch_bounds__(NTHREADS, 1)
extend_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
              const __grid_constant__ CUtensorMap vmap, const ExtendParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_TMEMSLOT);
  const uint32_t s_base = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

  const int tile = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int TOK = BM / G;
  const int row0 = p.q_indptr[b];
  const int S = p.q_indptr[b + 1] - row0;
  const int i0 = tile * TOK;
  if (i0 >= S) return;  // CTA-uniform: no tokens in this tile
  const int ntok = min(TOK, S - i0);
  const int P = p.prefix_lens[b];
  const int bs = 1 << p.bs_shift;
  const int cap = p.max_blocks * bs;
  int kv_total = P + S;
  int k_hi = P + i0 + ntok;  // keys this tile needs
  if (P < 0 || kv_total > cap) {
    if (threadIdx.x == 0) set_err(p.err, 3);
    kv_total = min(max(kv_total, 0), cap);
    k_hi = min(max(k_hi, 1), max(cap, 1));
  }
  const int T = (k_hi + BN - 1) / BN;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&qmap);
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    mbar_init(bar(B_Q), 1);
    mbar_init(bar(B_KFULL), 1);
    mbar_init(bar(B_KFULL + 1), 1);
    mbar_init(bar(B_KFREE), 1);
    mbar_init(bar(B_KFREE + 1), 1);
    mbar_init(bar(B_VFULL), 1);
    mbar_init(bar(B_VFREE), 2);
    mbar_init(bar(B_VTFULL), 2);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_SFULL + 1), 1);
    mbar_init(bar(B_SFREE), 4);
    mbar_init(bar(B_SFREE + 1), 4);
    mbar_init(bar(B_PFULL), 4);
    mbar_init(bar(B_PVDONE), 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(B_Q), TILE);
      for (int c = 0; c < 2; ++c)
        tma_load_3d(s_base + OFF_Q + c * CHUNK, &qmap, bar(B_Q), c * 64, g * G, row0 + i0);
    }
    const int32_t* bt = p.block_tables + (int64_t)b * p.max_blocks;
    for (int kt = 0; kt < T && ok; ++kt) {
      const int s = kt & 1;
      const int key0 = kt * BN + 16 * (lane & 7);
      int blk = -1;
      if (lane < 8 && key0 < k_hi) {
        blk = bt[key0 >> p.bs_shift];
        if (blk < 0 || blk >= p.num_blocks) {
          set_err(p.err, 1);
          blk = -1;  // the TMA fills an out-of-range box with zeros
        }
      }
      const int page = blk < 0 ? -1 : blk * p.num_kv_heads + g;
      const int rip = key0 & (bs - 1);
      if (kt >= 2 && !mbar_wait(bar(B_KFREE + s), ((kt - 2) >> 1) & 1)) { ok = false; break; }
      int pg[8], rr[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        pg[j] = __shfl_sync(0xFFFFFFFFu, page, j);
        rr[j] = __shfl_sync(0xFFFFFFFFu, rip, j);
      }
      if (lane == 0) {
        const uint32_t dst = s_base + OFF_K + s * TILE;
        mbar_arrive_expect_tx(bar(B_KFULL + s), TILE);
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_3d(dst + c * CHUNK + j * 2048, &kmap, bar(B_KFULL + s), c * 64, rr[j], pg[j]);
      }
      if (kt >= 1 && !mbar_wait(bar(B_VFREE), (kt - 1) & 1)) { ok = false; break; }
      if (lane == 0) {
        const uint32_t dst = s_base + OFF_V;
        mbar_arrive_expect_tx(bar(B_VFULL), TILE);
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_3d(dst + c * CHUNK + j * 2048, &vmap, bar(B_VFULL), c * 64, rr[j], pg[j]);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t qk_fmt = (CT == DT_BF16) ? 1u : 0u;
      constexpr uint32_t idesc_qk = umma_idesc_f16(qk_fmt, qk_fmt, BM, BN);
      constexpr uint32_t idesc_pv = umma_idesc_f16(0u, 0u, BM, HD);
      auto issue_pv = [&](int u) -> bool {
        if (!mbar_wait(bar(B_PFULL), u & 1)) return false;
        if (!mbar_wait(bar(B_VTFULL), u & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK + (kk & 3) * 32;
          umma_f16(tmem + TM_O, umma_desc_sw128(s_base + OFF_P + off),
                   umma_desc_sw128(s_base + OFF_VT + off), idesc_pv, (u > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(bar(B_PVDONE));
        return true;
      };
      ok = mbar_wait(bar(B_Q), 0);
      for (int kt = 0; kt < T && ok; ++kt) {
        const int s = kt & 1;
        if (!mbar_wait(bar(B_KFULL + s), (kt >> 1) & 1)) { ok = false; break; }
        if (kt >= 2 && !mbar_wait(bar(B_SFREE + s), ((kt - 2) >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK + (kk & 3) * 32;
          umma_f16(tmem + TM_S + s * BN, umma_desc_sw128(s_base + OFF_Q + off),
                   umma_desc_sw128(s_base + OFF_K + s * TILE + off), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_SFULL + s));
        umma_commit(bar(B_KFREE + s));
        if (kt >= 1 && !issue_pv(kt - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(T - 1);
    }
    __syncwarp();
  } else if (warp < 4) {
    // ------------------------------------------------------------ V^T builders
    const int ct = threadIdx.x - 64;  // 0..63
    for (int kt = 0; kt < T && ok; ++kt) {
      if (!mbar_wait(bar(B_VFULL), kt & 1)) { ok = false; break; }
      if (kt >= 1 && !mbar_wait(bar(B_PVDONE), (kt - 1) & 1)) { ok = false; break; }
      const int kbase = kt * BN;
      // 64 groups of four 8x8 blocks; this warp takes 32 of them
      for (int q = ct >> 5; q < 64; q += 2) {
        const int kb2 = q >> 3, dq = q & 7;
        const int jm = lane >> 3, rw = lane & 7;
        // source: row = key, 16 B = 8 dims
        const int key_s = kb2 * 16 + (jm >> 1) * 8 + rw;
        const int dim_s = dq * 16 + (jm & 1) * 8;
        uint32_t r[4];
        ldsm_x4_t(s_base + OFF_V + (dim_s >> 6) * CHUNK + sw_off(key_s, (dim_s & 63) >> 3), r);
        // r[j]: rows = dims db_j + gid, cols = keys kb_j + 2tig, +1
        const int gid = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int kb_j = kb2 * 16 + (j >> 1) * 8;
          uint32_t v = to_f16x2<CT == DT_BF16>(r[j]);
          const int k0 = kbase + kb_j + 2 * tig;
          if (k0 >= kv_total) v &= 0xFFFF0000u;
          if (k0 + 1 >= kv_total) v &= 0x0000FFFFu;
          r[j] = v;
          (void)gid;
        }
        // destination: row = dim, 16 B = 8 keys
        const int dim_d = dq * 16 + (jm & 1) * 8 + rw;
        const int key_d = kb2 * 16 + (jm >> 1) * 8;
        stsm_x4(s_base + OFF_VT + (key_d >> 6) * CHUNK + sw_off(dim_d, (key_d & 63) >> 3), r[0], r[1],
                r[2], r[3]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(B_VFREE));
        mbar_arrive(bar(B_VTFULL));
      }
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qw = warp & 3;
    const int r = qw * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(qw * 32) << 16;
    const int lim = P + i0 + r / G;  // last key this row may see
    float m_run = -INFINITY, l_run = 0.f;
    for (int kt = 0; kt < T && ok; ++kt) {
      const int s = kt & 1;
      if (!mbar_wait(bar(B_SFULL + s), (kt >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      float x[BN];
      {
        uint32_t raw[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_addr + TM_S + s * BN + c * 32, raw[c]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j) x[c * 32 + j] = __uint_as_float(raw[c][j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SFREE + s));

      const int key0 = kt * BN;
      const bool need_mask = key0 + BN - 1 > P + i0;
      float mt = -INFINITY;
#pragma unroll
      for (int j = 0; j < BN; ++j) {
        float v = x[j] * p.scale_log2;
        if (need_mask && key0 + j > lim) v = -INFINITY;
        x[j] = v;
        mt = fmaxf(mt, v);
      }
      float m_new = m_run;
      if (mt > m_run + 8.f) m_new = mt;
      const float alpha = fast_exp2(m_run - m_new);
      uint32_t pk[BN / 2];
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < BN / 2; ++j) {
        const float p0 = fast_exp2(x[2 * j] - m_new), p1 = fast_exp2(x[2 * j + 1] - m_new);
        sum += p0 + p1;
        pk[j] = pack2<false>(p0, p1);
      }
      l_run = l_run * alpha + sum;
      if (kt >= 1) {
        if (!mbar_wait(bar(B_PVDONE), (kt - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const bool mine = (m_new != m_run);
        if (__any_sync(0xFFFFFFFFu, mine)) {
          const float f = mine ? alpha : 1.f;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_addr + TM_O + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
            tmem_st32(tmem + lane_addr + TM_O + c * 32, o);
          }
          tmem_wait_st();
        }
      }
      m_run = m_new;
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const uint32_t addr = s_base + OFF_P + (u >> 3) * CHUNK + sw_off(r, u & 7);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * u]),
                     "r"(pk[4 * u + 1]), "r"(pk[4 * u + 2]), "r"(pk[4 * u + 3])
                     : "memory");
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
    }
    // ---- epilogue: O / l -> out, LSE
    if (ok && mbar_wait(bar(B_PVDONE), (T - 1) & 1)) {
      tc_fence_after();
      const bool valid = (r / G) < ntok;
      const int64_t orow = (int64_t)(row0 + i0 + r / G) * p.num_q_heads + g * G + (r % G);
      const float inv = 1.f / l_run;
      const float osc = inv * p.out_scale;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_addr + TM_O + c * 32, o);
        tmem_wait_ld();
        if (valid) {
          uint32_t w[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            w[j] = pack2<CT == DT_BF16>(__uint_as_float(o[2 * j]) * osc,
                                        __uint_as_float(o[2 * j + 1]) * osc);
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + orow * HD + c * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      }
      if (valid && p.lse_out) p.lse_out[orow] = (m_run + log2f(l_run)) * kLn2f;
    } else {
      ok = false;
    }
  }

  if (!ok) set_err(p.err, 4);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace

bool extend_supported(int head_dim, int cache_dt, int act_dt, int group) {
  if (head_dim != HD) return false;
  if (!(cache_dt == DT_F16 || cache_dt == DT_BF16) || act_dt != cache_dt) return false;
  return group == 1 || group == 2 || group == 4 || group == 8;
}

cudaError_t launch_extend(const CUtensorMap& qmap, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const ExtendParams& p, int head_dim, int cache_dt, int act_dt,
                          cudaStream_t stream) {
  if (!extend_supported(head_dim, cache_dt, act_dt, p.group)) return cudaErrorInvalidValue;
  dim3 grid(p.tiles_per_head, p.num_kv_heads, p.batch);
  if (cache_dt == DT_BF16) {
    auto k = extend_kernel<DT_BF16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    k<<<grid, NTHREADS, SMEM_BYTES, stream>>>(qmap, kmap, vmap, p);
  } else {
    auto k = extend_kernel<DT_F16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    k<<<grid, NTHREADS, SMEM_BYTES, stream>>>(qmap, kmap, vmap, p);
  }
  return cudaGetLastError();
}

}  // namespace pkv
