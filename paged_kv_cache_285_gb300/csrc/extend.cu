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
// Measured on this part, an MMA that reads its A operand from shared memory
// runs at ~60% of the tensor peak for this shape, one that reads A from TMEM
// at the full peak, so both A operands (Q for S = Q K^T, P for O += P V) live
// in TMEM.  TMEM (512 columns): two fp32 S buffers, the O accumulator, the Q
// tile and one f16 P tile.  An S buffer is released as soon as the softmax
// has its row in registers, so S = Q K^T of tile k+2 never waits for a PV
// product to drain; the P tile is rewritten once PV of the previous tile is
// done.  Shared memory holds only 3-stage K and V rings.
//
// Warp roles (384 threads):
//   warps 0,11  TMA producers for the K and the V ring: per key tile sixteen
//               16-token x 64-dim boxes addressed through the block table
//               (block ids prefetched into registers), 128-byte swizzled.
//   warp 1      TMEM owner and, on one lane, the MMA issuer: S = Q K^T
//               (A = Q in TMEM, B = K tile K-major, M=N=K=128), then
//               O += P V for the previous tile (A = P in TMEM, B = the V tile
//               as loaded, [key][dim], read as an MN-major operand).
//   warps 2-3,  V converters: bf16 V tiles are turned into f16 in place and
//   8-10        keys past the sequence end are zeroed (they may hold NaN).
//   warps 4-7   softmax (one thread per row): stores its Q row into TMEM,
//               then per tile reads its 128-column S row from TMEM with one
//               wait, takes the row max (causal mask on diagonal tiles), keeps
//               a running max with lazy rescaling (O in TMEM is rescaled only
//               when the max grows by more than 2^8) and writes f16 P; finally
//               O / l and the LSE.
// P is f16 (11 significant bits) because bf16 P alone would put the relative
// L2 error of the output near 1.5e-3; V is therefore converted to f16 (bf16
// values beyond +-65504 are outside this path's range).
#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int BM = 128;       // rows per tile
constexpr int BN = 128;       // keys per tile
constexpr int HD = 128;       // head dim
constexpr int NTHREADS = 384;
constexpr int NCONV = 160;    // V converter threads (warps 2, 3, 8-10)
constexpr int NST = 3;        // K and V ring depth
constexpr int TILE = BN * HD * 2;   // 32 KB: 128 x 128 16-bit elements
constexpr int CHUNK = 16384;        // one 64-element column block [128 rows][128 B]

constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + NST * TILE;
constexpr int OFF_BAR = OFF_V + NST * TILE;
enum {
  B_Q = 0,
  B_KFULL = 1, B_KFREE = B_KFULL + NST,
  B_VFULL = B_KFREE + NST, B_VFREE = B_VFULL + NST, B_VCONV = B_VFREE + NST,
  B_SFULL = B_VCONV + NST, B_SFREE = B_SFULL + 2, B_PFULL = B_SFREE + 2, B_PVDONE = B_PFULL + 1,
  NBAR = B_PVDONE + 1
};
constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_TMEMSLOT + 16 + 1024;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;     // two fp32 S buffers, columns 0 and 128
constexpr uint32_t TM_O = 256;   // O accumulator, 128 columns
constexpr uint32_t TM_Q = 384;   // Q tile: 64 columns of 16-bit pairs
constexpr uint32_t TM_P = 448;   // P tile: 64 columns of f16 pairs
constexpr float kLn2f = 0.6931471805599453f;

__device__ __forceinline__ void set_err(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

template <int CT>
__global__ void __launch_bounds__(NTHREADS, 1)
extend_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
              const ExtendParams p) {
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
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    mbar_init(bar(B_Q), 4);
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_KFREE + i), 1);
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_VFREE + i), 1);
      mbar_init(bar(B_VCONV + i), NCONV / 32);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_SFULL + i), 1);
      mbar_init(bar(B_SFREE + i), 4);
    }
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

  if (warp == 0 || warp == 11) {
    // ------------------------------------------------------------ producers
    // warp 0 streams K tiles, warp 11 V tiles, each through its own ring, so
    // that a K load never queues behind a V buffer that is still in use.
    // Block ids: lane l holds sub-tile (32 w + l) of window w, the next
    // window is fetched one window ahead.
    const bool is_k = (warp == 0);
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    const int full0 = is_k ? B_KFULL : B_VFULL, free0 = is_k ? B_KFREE : B_VFREE;
    const uint32_t ring = s_base + (is_k ? OFF_K : OFF_V);
    const int32_t* bt = p.block_tables + (int64_t)b * p.max_blocks;
    auto fetch = [&](int w) -> int {
      const int key0 = (w * 32 + lane) * 16;  // sub-tile = 16 keys
      int page = -1;
      if (key0 < k_hi) {
        const int blk = bt[key0 >> p.bs_shift];
        if (blk < 0 || blk >= p.num_blocks) set_err(p.err, 1);  // TMA zero-fills page -1
        else page = blk * p.num_kv_heads + g;
      }
      return page;
    };
    int win = 0, cur = fetch(0), nxt = fetch(1);
    for (int kt = 0; kt < T && ok; ++kt) {
      const int s = kt % NST;
      if ((kt >> 2) > win) {  // 4 tiles x 8 sub-tiles per window
        cur = nxt;
        ++win;
        nxt = fetch(win + 1);
      }
      int pg[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) pg[j] = __shfl_sync(0xFFFFFFFFu, cur, (kt & 3) * 8 + j);
      if (kt >= NST && !mbar_wait(bar(free0 + s), (uint32_t)((kt / NST - 1) & 1))) { ok = false; break; }
      if (lane == 0) {
        const uint32_t dst = ring + s * TILE;
        mbar_arrive_expect_tx(bar(full0 + s), TILE);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int rip = (kt * BN + 16 * j) & (bs - 1);
#pragma unroll
          for (int c = 0; c < 2; ++c)
            tma_load_3d(dst + c * CHUNK + j * 2048, map, bar(full0 + s), c * 64, rip, pg[j]);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t qk_fmt = (CT == DT_BF16) ? 1u : 0u;
      constexpr uint32_t idesc_qk = umma_idesc_f16(qk_fmt, qk_fmt, BM, BN);
      // P (A, f16 in TMEM) x V (B, f16, MN-major: the V tile as loaded, [key][dim])
      constexpr uint32_t idesc_pv = umma_idesc_f16(0u, 0u, BM, HD) | (1u << 16);
      auto issue_pv = [&](int u) -> bool {
        const int us = u % NST;
        if (!mbar_wait(bar(B_PFULL), u & 1)) return false;
        if (!mbar_wait(bar(B_VCONV + us), (u / NST) & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          umma_f16_ts(tmem + TM_O, tmem + TM_P + kk * 8,
                      umma_desc_sw128_mn(s_base + OFF_V + us * TILE + kk * 2048, CHUNK), idesc_pv,
                      (u > 0 || kk > 0) ? 1u : 0u);
        umma_commit(bar(B_PVDONE));  // P buffer and O are free again
        umma_commit(bar(B_VFREE + us));
        return true;
      };
      ok = mbar_wait(bar(B_Q), 0);
      for (int kt = 0; kt < T && ok; ++kt) {
        const int sb = kt & 1, ks = kt % NST;
        if (!mbar_wait(bar(B_KFULL + ks), (kt / NST) & 1)) { ok = false; break; }
        // S buffer sb is free once the softmax has read S(kt-2) into registers
        if (kt >= 2 && !mbar_wait(bar(B_SFREE + sb), ((kt - 2) >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * CHUNK + (kk & 3) * 32;
          umma_f16_ts(tmem + TM_S + sb * BN, tmem + TM_Q + kk * 8,
                      umma_desc_sw128(s_base + OFF_K + ks * TILE + off), idesc_qk, kk > 0 ? 1u : 0u);
        }
        umma_commit(bar(B_SFULL + sb));
        umma_commit(bar(B_KFREE + ks));
        if (kt >= 1 && !issue_pv(kt - 1)) { ok = false; break; }
      }
      if (ok) ok = issue_pv(T - 1);
    }
    __syncwarp();
  } else if (warp < 4 || warp >= 8) {
    // ------------------------------------------------------------ V converters (2, 3, 8-10)
    // In place, per 16-byte unit: bf16 -> f16 (the PV product is f16 x f16),
    // and keys at or past the sequence end -> 0 (they may hold anything, and
    // 0 * NaN is NaN).  The swizzle only permutes units inside a 128-byte key
    // row, so the key of a unit is its byte offset / 128 within its block.
    const int ct = warp < 4 ? threadIdx.x - 64 : threadIdx.x - 192;  // 0..159
    for (int kt = 0; kt < T && ok; ++kt) {
      const int vs = kt % NST;
      if (!mbar_wait(bar(B_VFULL + vs), (kt / NST) & 1)) { ok = false; break; }
      const int kbase = kt * BN;
      const bool tail = kbase + BN > kv_total;
      if (CT == DT_BF16 || tail) {
        uint8_t* vt = smem + OFF_V + vs * TILE;
        constexpr int PER = (TILE / 16 + NCONV - 1) / NCONV;  // 13 units of 16 bytes
        uint4 w[PER];
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int u = ct + i * NCONV;
          if (u < TILE / 16) w[i] = *reinterpret_cast<const uint4*>(vt + u * 16);
        }
#pragma unroll
        for (int i = 0; i < PER; ++i) {
          const int u = ct + i * NCONV;
          if (u >= TILE / 16) break;
          const int key = kbase + ((u * 16) % CHUNK) / 128;
          if (key >= kv_total) {
            w[i] = make_uint4(0u, 0u, 0u, 0u);
          } else if (CT == DT_BF16) {
            w[i].x = to_f16x2<true>(w[i].x);
            w[i].y = to_f16x2<true>(w[i].y);
            w[i].z = to_f16x2<true>(w[i].z);
            w[i].w = to_f16x2<true>(w[i].w);
          }
          *reinterpret_cast<uint4*>(vt + u * 16) = w[i];
        }
        fence_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_VCONV + vs));
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int qw = warp & 3;
    const int r = qw * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(qw * 32) << 16;
    const int lim = P + i0 + r / G;  // last key this row may see
    const bool valid = (r / G) < ntok;
    const int64_t qrow = (int64_t)(row0 + i0 + r / G) * p.num_q_heads + g * G + (r % G);
    // Q row -> TMEM (64 columns of 16-bit pairs, the QK A operand); rows
    // past the suffix get zeros
    {
      const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) + qrow * HD);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 w = valid ? __ldg(src + c * 4 + j) : make_uint4(0u, 0u, 0u, 0u);
          v[4 * j] = w.x; v[4 * j + 1] = w.y; v[4 * j + 2] = w.z; v[4 * j + 3] = w.w;
        }
        tmem_st16(tmem + lane_addr + TM_Q + c * 16, v);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_Q));
    }
    float m_run = -INFINITY, l_run = 0.f;
    for (int kt = 0; kt < T && ok; ++kt) {
      const int sb = kt & 1;
      if (!mbar_wait(bar(B_SFULL + sb), (kt >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const uint32_t srow = tmem + lane_addr + TM_S + sb * BN;
      const int key0 = kt * BN;
      const bool diag = key0 + BN - 1 > P + i0;  // tile reaches past some row's limit
      // the whole S row: four 32-column loads, one wait
      uint32_t raw[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(srow + c * 32, raw[c]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_SFREE + sb));  // S is in registers: buffer free
      if (diag) {  // causal mask on the tile that reaches past some row's limit
        const int nvis = lim - key0;  // keys key0 .. key0+nvis are visible
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c * 32 + j > nvis) raw[c][j] = __float_as_uint(-INFINITY);
      }
      // row max over 8 independent accumulators (one running max would be a
      // 128-long dependent chain)
      float mx[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) mx[a] = -INFINITY;
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int j = 0; j < 32; ++j) mx[j & 7] = fmaxf(mx[j & 7], __uint_as_float(raw[c][j]));
      const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                             fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * p.scale_log2;
      float m_new = m_run;
      if (mt > m_run + 8.f) m_new = mt;
      const float alpha = fast_exp2(m_run - m_new);
      const bool mine = (m_new != m_run);
      if (kt >= 1 && __any_sync(0xFFFFFFFFu, mine)) {
        // rescale O in TMEM: wait until PV(kt-1) has finished accumulating
        if (!mbar_wait(bar(B_PVDONE), (kt - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const float f = mine ? alpha : 1.f;
#pragma unroll 1
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
      m_run = m_new;
      // p = 2^(s*scale - m) as f16 pairs, streamed 32 keys at a time into the P
      // tile once PV(kt-1) has consumed P(kt-1)
      if (kt >= 1 && !mbar_wait(bar(B_PVDONE), (kt - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      float sm[8];
#pragma unroll
      for (int a = 0; a < 8; ++a) sm[a] = 0.f;
      const float sc = p.scale_log2, neg_m = -m_new;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t pk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(raw[c][2 * j]), sc, neg_m));
          const float p1 = fast_exp2(fmaf(__uint_as_float(raw[c][2 * j + 1]), sc, neg_m));
          sm[j & 7] += p0 + p1;
          pk[j] = pack2<false>(p0, p1);
        }
        tmem_st16(tmem + lane_addr + TM_P + c * 16, pk);
      }
      const float sum = ((sm[0] + sm[1]) + (sm[2] + sm[3])) + ((sm[4] + sm[5]) + (sm[6] + sm[7]));
      l_run = l_run * alpha + sum;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_PFULL));
    }
    // ---- epilogue: O / l -> out, LSE
    if (ok && mbar_wait(bar(B_PVDONE), (T - 1) & 1)) {
      tc_fence_after();
      const float osc = p.out_scale / l_run;
#pragma unroll 1
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
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + qrow * HD + c * 32);
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
      }
      if (valid && p.lse_out) p.lse_out[qrow] = (m_run + log2f(l_run)) * kLn2f;
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

cudaError_t launch_extend(const CUtensorMap& kmap, const CUtensorMap& vmap, const ExtendParams& p,
                          int head_dim, int cache_dt, int act_dt, cudaStream_t stream) {
  if (!extend_supported(head_dim, cache_dt, act_dt, p.group)) return cudaErrorInvalidValue;
  dim3 grid(p.tiles_per_head, p.num_kv_heads, p.batch);
  if (cache_dt == DT_BF16) {
    auto k = extend_kernel<DT_BF16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    k<<<grid, NTHREADS, SMEM_BYTES, stream>>>(kmap, vmap, p);
  } else {
    auto k = extend_kernel<DT_F16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    k<<<grid, NTHREADS, SMEM_BYTES, stream>>>(kmap, vmap, p);
  }
  return cudaGetLastError();
}

}  // namespace pkv
