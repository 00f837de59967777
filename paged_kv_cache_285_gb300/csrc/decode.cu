// Paged decode attention for sm_103a.
//
// One query token per request attends over all of the request's cached
// tokens, read through its block table ("PagedAttention과 RadixAttention으로
// LLM KV 캐시 최적화", section 02; the step itself: "KV Cache에 대해
// 알아보자 (Feat. Attention)", §3 Decode 단계 -- memory-bound, the whole cache
// is read every step).
//
// Design (memory-bound stream, so every byte is read once and the arithmetic
// stays far below the HBM roofline):
//   * grid (split, kv head x head chunk, request).  A split is a fixed-length
//     run of the sequence; up to 8 query heads of one kv head share one CTA
//     (the N = 8 side of the MMA), so with GQA groups of up to 8 every K/V
//     byte is fetched once per step; larger groups are cut into chunks of 8
//     heads, one CTA each, which read the same pages (the second read mostly
//     from L2).
//   * each warp owns every NW-th 16-token tile of the split and runs its own
//     NS-deep TMA pipeline: lane 0 issues cp.async.bulk.tensor copies of the
//     K and V tiles (128-byte swizzled, conflict-free ldmatrix) completing on a
//     per-stage mbarrier; the warp's block ids are prefetched 32 at a time into
//     registers and handed to lane 0 with a shuffle.
//   * scores S^T[token][head] = K q^T and O^T[dim][head] += V^T P^T on the
//     warp-level tensor cores (mma.m16n8k16, fp32 accumulate), tokens on the M
//     side so a GQA group of up to 8 heads fills the N=8 side.  P^T comes from
//     S^T's accumulator registers by an in-register 8x8 transpose (movmatrix).
//     bf16 caches split P into bf16 hi+lo parts (two PV products) so that P
//     keeps ~16 bits; f16 and fp8 caches use f16 P.  fp8 codes are widened to
//     f16 exactly in registers (cvt e4m3x2 -> f16x2); k_scale is folded into
//     the softmax scale and v_scale into the output scale.
//   * online softmax in base 2 (running max and sum per head column, max
//     reduced over the 8 lanes that hold a column with xor-shuffles).
//   * warps are combined through shared memory with their (max, sum); a split
//     either writes the final output (single-split requests) or a normalised
//     partial plus its log-sum-exp, merged by merge_kernel.
#include "internal.h"
#include "ptx.cuh"

namespace pkv {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr float kLn2 = 0.6931471805599453f;

template <int HD, int CT, int NW, int NS>
struct DecodeCfg {
  static constexpr int ELEM = (CT == DT_E4M3) ? 1 : 2;
  static constexpr int ROWB = HD * ELEM;                // bytes of one token row
  static constexpr int CHUNKB = ROWB < 128 ? ROWB : 128;  // swizzle span (64 or 128)
  static constexpr int NCH = ROWB / CHUNKB;             // TMA boxes per tile
  static constexpr int TILEB = kSubTokens * ROWB;       // one 16-token K (or V) tile
  static constexpr int STAGEB = 2 * TILEB;              // K tile + V tile
  static constexpr int STAGE_AREA = NW * NS * STAGEB;
  static constexpr int MT = HD / 16;                    // output m-tiles (dims)
  static constexpr bool MMA_BF16 = (CT == DT_BF16);
  static constexpr int COMB_BYTES = NW * 8 * HD * 4 + NW * 8 * 2 * 4;
  static constexpr int AREA = STAGE_AREA > COMB_BYTES ? STAGE_AREA : COMB_BYTES;
  static constexpr int SMEM = 1024 /*align slack*/ + AREA + NW * NS * 8;
};

// Byte offset of (token t, row byte x) inside a staged tile, matching the TMA
// swizzle: the tile is NCH boxes of [16 tokens][CHUNKB bytes]; 16-byte unit
// bits [4, 4+log2(CHUNKB/16)) are XORed with address bits [7, ...).
template <int CHUNKB>
__device__ __forceinline__ uint32_t tile_off(int t, int x) {
  const uint32_t o = (uint32_t)((x / CHUNKB) * (kSubTokens * CHUNKB) + t * CHUNKB + (x % CHUNKB));
  if constexpr (CHUNKB == 128) return o ^ ((o >> 3) & 0x70u);
  else if constexpr (CHUNKB == 64) return o ^ ((o >> 3) & 0x30u);
  else return o;
}

// Which head dim an accumulator row holds: 16-bit caches keep dims in order,
// fp8 tiles interleave them (see the PV product below).
template <int CT>
__device__ __forceinline__ int out_dim(int u, int row) {
  if constexpr (CT == DT_E4M3) {
    const int pp = u >> 1, e = u & 1;
    return 32 * pp + (row >= 8 ? 16 : 0) + 2 * (row & 7) + e;
  } else {
    return 16 * u + row;
  }
}

__device__ __forceinline__ void set_err(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

template <int AT>
__device__ __forceinline__ void store_act(void* base, int64_t idx, float v) {
  if constexpr (AT == DT_BF16) {
    reinterpret_cast<__nv_bfloat16*>(base)[idx] = __float2bfloat16_rn(v);
  } else {
    reinterpret_cast<__half*>(base)[idx] = __float2half_rn(v);
  }
}

template <int AT>
__device__ __forceinline__ float load_act(const void* base, int64_t idx) {
  if constexpr (AT == DT_BF16) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  } else {
    return __half2float(reinterpret_cast<const __half*>(base)[idx]);
  }
}

// A 16-bit activation value (its bits) widened to fp32.
template <int AT>
__device__ __forceinline__ float to_f32_bits(uint32_t bits16) {
  if constexpr (AT == DT_BF16) return __uint_as_float(bits16 << 16);
  else return __half2float(__ushort_as_half((unsigned short)bits16));
}

// Shared-prefix length of request b's group (group_indptr is non-decreasing
// from 0 to batch; the search stays inside the arrays whatever they hold).
// A request that no group covers gets -1: no shared prefix, reported.
__device__ __forceinline__ int group_prefix_len(const DecodeExtraParams& ap, int b) {
  if (b < __ldg(ap.group_indptr) || b >= __ldg(ap.group_indptr + ap.num_groups)) return -1;
  int lo = 0, hi = ap.num_groups;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(ap.group_indptr + mid) <= b) lo = mid;
    else hi = mid;
  }
  return __ldg(ap.group_prefix_lens + lo);
}

// CASC: a cascade launch (tokens from the group's shared prefix on; partials
// in the workspace slots after the prefix's chunks, always merged).
template <int HD, int CT, int AT, int NW, int NS, bool CASC>
__global__ void __launch_bounds__(NW * 32)
decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
              const DecodeParams p, const DecodeExtraParams ap) {
  using C = DecodeCfg<HD, CT, NW, NS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::AREA);

  // split is the slowest grid dimension: every request's first chunk runs
  // before any second chunk, so the partial and empty last splits form the tail
  const int b = blockIdx.y, split = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;
  const int G = p.group;
  // kv head g, chunk hc of its query heads: heads hb .. hb + GC - 1
  const int nhc = (G + 7) >> 3;
  const int g = (int)blockIdx.x / nhc, hc = (int)blockIdx.x - g * nhc;
  const int hb = g * G + hc * 8, GC = min(8, G - hc * 8);
  const int bs = 1 << p.bs_shift;

  int n = p.seq_lens[b];
  int tb = 0;  // first token of this launch (cascade: the end of the shared prefix)
  if constexpr (CASC) tb = group_prefix_len(ap, b);
  const int cap = min(p.max_blocks * bs, (tb > 0 ? tb : 0) + p.num_splits * p.chunk);
  if (n < 0 || n > cap) {
    if (threadIdx.x == 0 && split == 0) set_err(p.err, 3);
    n = n < 0 ? 0 : cap;
  }
  if constexpr (CASC) {
    if (tb < 0 || tb > n) {
      if (threadIdx.x == 0 && split == 0) set_err(p.err, 3);
      tb = tb < 0 ? 0 : n;
    }
    tb = (tb >> p.bs_shift) << p.bs_shift;  // only whole blocks are shared
    // the merge reads the request's span from here instead of searching again
    if (split == 0 && blockIdx.x == 0 && threadIdx.x == 0) ap.ws_span[b] = make_int2(tb, n);
  }
  const int t0 = tb + split * p.chunk;
  if (t0 >= n) {
    if constexpr (CASC) {
      // nothing after the prefix; the current token cannot be appended there
      if (ap.k_new != nullptr && split == 0 && n > 0 && threadIdx.x == 0) set_err(p.err, 3);
    } else if (split == 0) {  // empty sequence: out = 0, lse = -inf
      for (int idx = threadIdx.x; idx < GC * HD; idx += NW * 32) {
        const int h = hb + idx / HD;
        store_act<AT>(p.out, ((int64_t)b * p.num_q_heads + h) * HD + idx % HD, 0.f);
        if (p.lse_out && idx % HD == 0) p.lse_out[(int64_t)b * p.num_q_heads + h] = -INFINITY;
      }
    }
    return;
  }
  const int t1 = min(n, t0 + p.chunk);
  const int nsub = (t1 - t0 + kSubTokens - 1) / kSubTokens;
  const int nsplit_b = (n - tb + p.chunk - 1) / p.chunk;
  const int cnt = warp < nsub ? (nsub - warp + NW - 1) / NW : 0;

  if (ap.k_new != nullptr && split == nsplit_b - 1) {
    // Fused append: this CTA covers position n-1, the current token; its K/V
    // rows of kv head g go to their slot before any tile of this CTA is
    // loaded (TMA reads the slot after the proxy fence and the barrier
    // below).  Same bytes as the separate append: a 16-bit copy, or
    // e4m3(fp32(x) / scale) from the correctly rounded quotient and a
    // saturating round-to-nearest-even convert.  With a group of more than 8
    // heads every head chunk's CTA writes the row (the same bytes), before its
    // own read of it.
    const int pos = n - 1;
    const int blk = p.block_tables[(int64_t)b * p.max_blocks + (pos >> p.bs_shift)];
    constexpr int VPR = HD / 8;  // 16-byte input vectors per row
    if (blk < 0 || blk >= p.num_blocks) {
      if (threadIdx.x == 0) set_err(p.err, 2);
    } else if (threadIdx.x < 2 * VPR) {
      const bool isv = threadIdx.x >= VPR;
      const int e = (threadIdx.x % VPR) * 8;
      const int64_t src = ((int64_t)b * p.num_kv_heads + g) * HD + e;
      const int64_t dst = (((int64_t)blk * p.num_kv_heads + g) * bs + (pos & (bs - 1))) * HD + e;
      const uint4 x = __ldg(reinterpret_cast<const uint4*>(
          reinterpret_cast<const uint16_t*>(isv ? ap.v_new : ap.k_new) + src));
      void* cache = isv ? ap.v_cache : ap.k_cache;
      if constexpr (CT != DT_E4M3) {
        *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(cache) + dst) = x;
      } else {
        const float sc = isv ? ap.v_scale : ap.k_scale;
        const float rc = isv ? ap.v_rcp : ap.k_rcp;
        const uint32_t w[4] = {x.x, x.y, x.z, x.w};
        uint32_t o[2];
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          uint32_t ob = 0;
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const uint32_t ww = w[2 * h2 + q2];
            const float a0 = quot_for_e4m3(to_f32_bits<AT>(ww & 0xFFFFu), sc, rc);
            const float a1 = quot_for_e4m3(to_f32_bits<AT>(ww >> 16), sc, rc);
            ob |= f32x2_to_e4m3x2(a0, a1) << (16 * q2);
          }
          o[h2] = ob;
        }
        *reinterpret_cast<uint2*>(reinterpret_cast<uint8_t*>(cache) + dst) = make_uint2(o[0], o[1]);
      }
      fence_proxy_async_global();
    }
  }

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    for (int i = 0; i < NW * NS; ++i) mbar_init(smem_u32(&bars[i]), 1);
    fence_mbar_init();
  }
  __syncthreads();

  // ---- query fragments (B operand: k = head dim, n = head in group) --------
  constexpr bool MMA_BF16 = C::MMA_BF16;
  uint32_t qf[HD / 16][2];
  {
    const int h = hb + gid;
    const int64_t qbase = ((int64_t)b * p.num_q_heads + h) * HD;
#pragma unroll
    for (int s = 0; s < HD / 16; ++s) {
      int d0, d1, d2, d3;
      if constexpr (CT == DT_E4M3) {  // permuted k order, see the fp8 score product
        d0 = 16 * s + 4 * tig; d1 = d0 + 1; d2 = d0 + 2; d3 = d0 + 3;
      } else {
        d0 = 16 * s + 2 * tig; d1 = d0 + 1; d2 = d0 + 8; d3 = d0 + 9;
      }
      if (gid < GC) {
        if constexpr (CT != DT_E4M3) {
          qf[s][0] = *reinterpret_cast<const uint32_t*>(
              reinterpret_cast<const uint16_t*>(p.q) + qbase + d0);
          qf[s][1] = *reinterpret_cast<const uint32_t*>(
              reinterpret_cast<const uint16_t*>(p.q) + qbase + d2);
        } else {
          qf[s][0] = pack2<false>(load_act<AT>(p.q, qbase + d0), load_act<AT>(p.q, qbase + d1));
          qf[s][1] = pack2<false>(load_act<AT>(p.q, qbase + d2), load_act<AT>(p.q, qbase + d3));
        }
      } else {
        qf[s][0] = 0u;
        qf[s][1] = 0u;
      }
    }
  }

  // ---- block ids of this warp's tiles, 32 at a time in registers ------------
  const int32_t* bt_row = p.block_tables + (int64_t)b * p.max_blocks;
  auto fetch = [&](int win) -> int {
    const int i = win * 32 + lane;
    int blk = -1;
    if (i < cnt) {
      const int tok = t0 + kSubTokens * (warp + i * NW);
      blk = bt_row[tok >> p.bs_shift];
      if (blk < 0 || blk >= p.num_blocks) {
        set_err(p.err, 1);
        blk = -1;  // TMA fills out-of-range tiles with zeros
      }
    }
    return blk;
  };
  int win_cur = 0;
  int bw_cur = fetch(0), bw_next = fetch(1);
  auto blk_of = [&](int i) -> int {  // called by all lanes with a warp-uniform, rising i
    while ((i >> 5) > win_cur) {
      bw_cur = bw_next;
      ++win_cur;
      bw_next = fetch(win_cur + 1);
    }
    return __shfl_sync(kFull, bw_cur, i & 31);
  };

  uint8_t* wstage = smem + warp * NS * C::STAGEB;
  const uint32_t wstage_s = smem_u32(wstage);
  const uint32_t wbar_s = smem_u32(&bars[warp * NS]);
  auto issue = [&](int i, int blk) {  // lane 0 only
    const int s = i % NS;
    const uint32_t bar = wbar_s + 8 * s;
    const uint32_t kdst = wstage_s + s * C::STAGEB;
    const uint32_t vdst = kdst + C::TILEB;
    const int tok = t0 + kSubTokens * (warp + i * NW);
    const int row = tok & (bs - 1);
    const int page = blk < 0 ? -1 : blk * p.num_kv_heads + g;
    mbar_arrive_expect_tx(bar, C::STAGEB);
#pragma unroll
    for (int ch = 0; ch < C::NCH; ++ch)
      tma_load_3d(kdst + ch * kSubTokens * C::CHUNKB, &kmap, bar, ch * (C::CHUNKB / C::ELEM), row, page);
#pragma unroll
    for (int ch = 0; ch < C::NCH; ++ch)
      tma_load_3d(vdst + ch * kSubTokens * C::CHUNKB, &vmap, bar, ch * (C::CHUNKB / C::ELEM), row, page);
  };

  {
    const int pre = cnt < NS ? cnt : NS;
    for (int i = 0; i < pre; ++i) {
      const int blk = blk_of(i);
      if (lane == 0) issue(i, blk);
    }
  }

  float acc[C::MT][4];
#pragma unroll
  for (int u = 0; u < C::MT; ++u) acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
  float m_e = -INFINITY, m_o = -INFINITY, l_e = 0.f, l_o = 0.f;
  int done = 0;  // tiles consumed (all issued tiles are waited on before exit)
  bool timed_out = false;

  for (int i = 0; i < cnt; ++i) {
    const int s = i % NS;
    if (!mbar_wait(wbar_s + 8 * s, (uint32_t)((i / NS) & 1))) {
      timed_out = true;
      break;
    }
    done = i + 1;
    const uint32_t kb = wstage_s + s * C::STAGEB;
    const uint32_t vb = kb + C::TILEB;
    const int tok0 = t0 + kSubTokens * (warp + i * NW);
    const int nvalid = min(kSubTokens, t1 - tok0);

    // ---- S^T (16 tokens x 8 heads) = K_tile . q^T --------------------------
    float sc[4] = {0.f, 0.f, 0.f, 0.f};
    {
      const int t = (lane & 7) + ((lane >> 3) & 1) * 8;
      if constexpr (CT != DT_E4M3) {
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          uint32_t a[4];
          ldsm_x4(kb + tile_off<C::CHUNKB>(t, (kk * 16 + (lane >> 4) * 8) * 2), a);
          mma16816<MMA_BF16>(sc, a, qf[kk][0], qf[kk][1]);
        }
      } else {
        // fp8: one ldmatrix row is 16 codes of one token; thread (gid,tig)
        // receives codes 4tig..4tig+3 and maps them to logical k slots
        // {2tig,2tig+1} and {2tig+8,2tig+9}; q uses the same permutation.
#pragma unroll
        for (int kp = 0; kp < HD / 32; ++kp) {
          uint32_t r[4];
          ldsm_x4(kb + tile_off<C::CHUNKB>(t, (2 * kp + (lane >> 4)) * 16), r);
          uint32_t a[4];
          a[0] = e4m3x2_to_f16x2(r[0] & 0xFFFFu);
          a[2] = e4m3x2_to_f16x2(r[0] >> 16);
          a[1] = e4m3x2_to_f16x2(r[1] & 0xFFFFu);
          a[3] = e4m3x2_to_f16x2(r[1] >> 16);
          mma16816<false>(sc, a, qf[2 * kp][0], qf[2 * kp][1]);
          a[0] = e4m3x2_to_f16x2(r[2] & 0xFFFFu);
          a[2] = e4m3x2_to_f16x2(r[2] >> 16);
          a[1] = e4m3x2_to_f16x2(r[3] & 0xFFFFu);
          a[3] = e4m3x2_to_f16x2(r[3] >> 16);
          mma16816<false>(sc, a, qf[2 * kp + 1][0], qf[2 * kp + 1][1]);
        }
      }
    }

    // ---- online softmax (base 2) over this tile, per head column --------------
    float s0 = sc[0] * p.scale_log2, s1 = sc[1] * p.scale_log2;
    float s2 = sc[2] * p.scale_log2, s3 = sc[3] * p.scale_log2;
    if (gid >= nvalid) { s0 = -INFINITY; s1 = -INFINITY; }
    if (gid + 8 >= nvalid) { s2 = -INFINITY; s3 = -INFINITY; }
    float mx_e = fmaxf(s0, s2), mx_o = fmaxf(s1, s3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      mx_e = fmaxf(mx_e, __shfl_xor_sync(kFull, mx_e, off));
      mx_o = fmaxf(mx_o, __shfl_xor_sync(kFull, mx_o, off));
    }
    const float mn_e = fmaxf(m_e, mx_e), mn_o = fmaxf(m_o, mx_o);
    const float al_e = fast_exp2(m_e - mn_e), al_o = fast_exp2(m_o - mn_o);
    m_e = mn_e;
    m_o = mn_o;
    const float p0 = fast_exp2(s0 - mn_e), p1 = fast_exp2(s1 - mn_o);
    const float p2 = fast_exp2(s2 - mn_e), p3 = fast_exp2(s3 - mn_o);
    l_e = l_e * al_e + (p0 + p2);
    l_o = l_o * al_o + (p1 + p3);
#pragma unroll
    for (int u = 0; u < C::MT; ++u) {
      acc[u][0] *= al_e;
      acc[u][1] *= al_o;
      acc[u][2] *= al_e;
      acc[u][3] *= al_o;
    }

    // ---- P^T as the B operand: transpose the S^T accumulator layout ----------
    uint32_t bh0, bh1, bl0 = 0u, bl1 = 0u;
    if constexpr (MMA_BF16) {
      const uint32_t h0 = pack2<true>(p0, p1), h1 = pack2<true>(p2, p3);
      const uint32_t r0 = pack2<true>(p0 - lo_f32<true>(h0), p1 - hi_f32<true>(h0));
      const uint32_t r1 = pack2<true>(p2 - lo_f32<true>(h1), p3 - hi_f32<true>(h1));
      bh0 = movmatrix_t(h0);
      bh1 = movmatrix_t(h1);
      bl0 = movmatrix_t(r0);
      bl1 = movmatrix_t(r1);
    } else {
      bh0 = movmatrix_t(pack2<false>(p0, p1));
      bh1 = movmatrix_t(pack2<false>(p2, p3));
    }

    // Zero the V values of tokens past the sequence end (they may hold
    // anything, and 0 * inf would poison the sum).
    const uint32_t mlo = (2 * tig < nvalid ? 0x0000FFFFu : 0u) | (2 * tig + 1 < nvalid ? 0xFFFF0000u : 0u);
    const uint32_t mhi = (2 * tig + 8 < nvalid ? 0x0000FFFFu : 0u) | (2 * tig + 9 < nvalid ? 0xFFFF0000u : 0u);

    // ---- O^T[dim][head] += V^T . P^T -----------------------------------------
    {
      const int j = lane >> 3;
      const int t = (lane & 7) + (j >> 1) * 8;
      if constexpr (CT != DT_E4M3) {
#pragma unroll
        for (int u = 0; u < C::MT; ++u) {
          uint32_t a[4];
          ldsm_x4_t(vb + tile_off<C::CHUNKB>(t, (u * 16 + (j & 1) * 8) * 2), a);
          a[0] &= mlo; a[1] &= mlo; a[2] &= mhi; a[3] &= mhi;
          mma16816<MMA_BF16>(acc[u], a, bh0, bh1);
          if constexpr (MMA_BF16) mma16816<true>(acc[u], a, bl0, bl1);
        }
      } else {
        // fp8: an 8x8 b16 transpose of codes gives thread (gid,tig) the bytes
        // V[2tig][d], V[2tig][d+1], V[2tig+1][d], V[2tig+1][d+1] with
        // d = 16*seg + 2*gid; a byte permute pairs equal dims of the two
        // tokens, which widen to the (k = token) pairs the A operand wants.
#pragma unroll
        for (int pp = 0; pp < HD / 32; ++pp) {
          uint32_t r[4];
          ldsm_x4_t(vb + tile_off<C::CHUNKB>(t, (2 * pp + (j & 1)) * 16), r);
          r[0] = __byte_perm(r[0] & mlo, 0, 0x3120);
          r[1] = __byte_perm(r[1] & mlo, 0, 0x3120);
          r[2] = __byte_perm(r[2] & mhi, 0, 0x3120);
          r[3] = __byte_perm(r[3] & mhi, 0, 0x3120);
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            uint32_t a[4];
            a[0] = e4m3x2_to_f16x2(e ? (r[0] >> 16) : (r[0] & 0xFFFFu));
            a[1] = e4m3x2_to_f16x2(e ? (r[1] >> 16) : (r[1] & 0xFFFFu));
            a[2] = e4m3x2_to_f16x2(e ? (r[2] >> 16) : (r[2] & 0xFFFFu));
            a[3] = e4m3x2_to_f16x2(e ? (r[3] >> 16) : (r[3] & 0xFFFFu));
            mma16816<false>(acc[2 * pp + e], a, bh0, bh1);
          }
        }
      }
    }

    __syncwarp();
    if (i + NS < cnt) {
      const int blk = blk_of(i + NS);
      if (lane == 0) issue(i + NS, blk);
    }
  }

  if (timed_out) {
    // Drain this warp's copies still in flight (bounded) before shared memory
    // is reused or the CTA exits.
    const int issued = min(cnt, done + NS);
    for (int i = done; i < issued; ++i) (void)mbar_wait(wbar_s + 8 * (i % NS), (uint32_t)((i / NS) & 1));
    if (lane == 0) set_err(p.err, 4);
  }

  // ---- combine the warps of this CTA -------------------------------------------
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l_e += __shfl_xor_sync(kFull, l_e, off);
    l_o += __shfl_xor_sync(kFull, l_o, off);
  }
  __syncthreads();  // every warp is done with its stages: reuse them
  float* sm_o = reinterpret_cast<float*>(smem);        // [NW][8][HD]
  float* sm_m = sm_o + NW * 8 * HD;                    // [NW][8]
  float* sm_l = sm_m + NW * 8;                         // [NW][8]
#pragma unroll
  for (int u = 0; u < C::MT; ++u) {
    const int d_lo = out_dim<CT>(u, gid), d_hi = out_dim<CT>(u, gid + 8);
    sm_o[(warp * 8 + 2 * tig) * HD + d_lo] = acc[u][0];
    sm_o[(warp * 8 + 2 * tig + 1) * HD + d_lo] = acc[u][1];
    sm_o[(warp * 8 + 2 * tig) * HD + d_hi] = acc[u][2];
    sm_o[(warp * 8 + 2 * tig + 1) * HD + d_hi] = acc[u][3];
  }
  if (gid == 0) {
    sm_m[warp * 8 + 2 * tig] = m_e;
    sm_m[warp * 8 + 2 * tig + 1] = m_o;
    sm_l[warp * 8 + 2 * tig] = l_e;
    sm_l[warp * 8 + 2 * tig + 1] = l_o;
  }
  __syncthreads();

  const bool direct = !CASC && (nsplit_b == 1);
  // cascade: the shared prefix's chunks hold the first slots
  const int kSlot0 = CASC ? ap.prefix_slots : 0;
  const int nslots = p.num_splits + kSlot0;
  for (int idx = threadIdx.x; idx < GC * HD; idx += NW * 32) {
    const int jh = idx / HD, d = idx % HD;
    float mstar = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) mstar = fmaxf(mstar, sm_m[w * 8 + jh]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = fast_exp2(sm_m[w * 8 + jh] - mstar);
      L += f * sm_l[w * 8 + jh];
      O += f * sm_o[(w * 8 + jh) * HD + d];
    }
    const float res = (O / L) * p.out_scale;
    const float lse2 = mstar + log2f(L);
    const int h = hb + jh;
    const int64_t bh = (int64_t)b * p.num_q_heads + h;
    if (direct) {
      store_act<AT>(p.out, bh * HD + d, res);
      if (p.lse_out && d == 0) p.lse_out[bh] = lse2 * kLn2;
    } else {
      p.ws_o[(bh * nslots + kSlot0 + split) * HD + d] = res;
      if (d == 0) p.ws_lse[bh * nslots + kSlot0 + split] = lse2;
    }
  }
}

// Merge the splits of one (request, head) per warp:
//   lse* = log2 sum_s 2^lse_s,  out = sum_s 2^(lse_s - lse*) o_s.
// Cascade: the shared prefix's chunks (slots 0 .. npc-1, when the group has a
// prefix) and the request's own splits (slots prefix_slots ..).
template <int HD, int AT, bool CASC>
__global__ void __launch_bounds__(128) merge_kernel(const DecodeParams p, const DecodeExtraParams ap) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bh = (int64_t)blockIdx.x * 4 + warp;
  if (bh >= (int64_t)p.batch * p.num_q_heads) return;
  const int b = (int)(bh / p.num_q_heads);
  constexpr int PER = HD / 32;
  int n, tb = 0;
  if constexpr (CASC) {
    // The usual row has one prefix chunk (slot 0) and one own split (slot
    // prefix_slots): both are loaded beside the request's span, so that such
    // a row waits on one round trip instead of two.
    const int ns0 = p.num_splits + ap.prefix_slots;
    const float* o0 = p.ws_o + bh * ns0 * HD + lane * PER;
    const float* o1 = o0 + (int64_t)ap.prefix_slots * HD;
    float a0[PER], a1[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) {
      a0[e] = o0[e];
      a1[e] = o1[e];
    }
    const float l0 = p.ws_lse[bh * ns0], l1 = p.ws_lse[bh * ns0 + ap.prefix_slots];
    // (first own token, clamped length) as the split kernel settled them
    const int2 span = ap.ws_span[b];
    tb = span.x;
    n = span.y;
    const bool one_chunk = tb > 0 && (tb <= ap.prefix_chunk || ap.prefix_chunks == 1);
    if (one_chunk && n > tb && n - tb <= p.chunk) {
      const float m = fmaxf(l0, l1);
      const float w0 = fast_exp2(l0 - m), w1 = fast_exp2(l1 - m);
      const float inv = 1.f / (w0 + w1);
#pragma unroll
      for (int e = 0; e < PER; ++e)
        store_act<AT>(p.out, bh * HD + lane * PER + e, (w0 * a0[e] + w1 * a1[e]) * inv);
      if (p.lse_out && lane == 0) p.lse_out[bh] = (m + log2f(w0 + w1)) * kLn2;
      return;
    }
  } else {
    const int bs = 1 << p.bs_shift;
    n = p.seq_lens[b];
    const int cap = min(p.max_blocks * bs, p.num_splits * p.chunk);
    n = n < 0 ? 0 : (n > cap ? cap : n);
  }
  const int ns = (n - tb + p.chunk - 1) / p.chunk;
  if (!CASC && ns <= 1) return;  // written directly by the split kernel
  const int kSlot0 = CASC ? ap.prefix_slots : 0;
  const int nslots = p.num_splits + kSlot0;
  // partial i of this row: the prefix's chunks first, then the own splits
  const int npc =
      (CASC && tb > 0) ? min((tb + ap.prefix_chunk - 1) / ap.prefix_chunk, ap.prefix_chunks) : 0;
  const int cnt = npc + ns;
  auto slot = [&](int i) { return i < npc ? i : kSlot0 + (i - npc); };
  if (cnt <= 0) {  // no token at all: out = 0, lse = -inf
#pragma unroll
    for (int k = 0; k < PER; ++k) store_act<AT>(p.out, bh * HD + lane * PER + k, 0.f);
    if (p.lse_out && lane == 0) p.lse_out[bh] = -INFINITY;
    return;
  }
  const float* lse = p.ws_lse + bh * nslots;
  const float* po = p.ws_o + bh * nslots * HD + lane * PER;
  // the first kPre partials are loaded together with the LSEs (they do not
  // depend on the max), so the merge waits on one round trip, not two
  constexpr int kPre = 8;
  float pre[kPre][PER];
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    if (k < cnt) {
#pragma unroll
      for (int e = 0; e < PER; ++e) pre[k][e] = 0.f;
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(po + (int64_t)slot(k) * HD);
        pre[k][0] = v.x; pre[k][1] = v.y; pre[k][2] = v.z; pre[k][3] = v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(po + (int64_t)slot(k) * HD);
        pre[k][0] = v.x; pre[k][1] = v.y;
      }
    }
  }
  float m = -INFINITY;
  for (int i = lane; i < cnt; i += 32) m = fmaxf(m, lse[slot(i)]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, off));
  float o[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) o[k] = 0.f;
  float L = 0.f;
#pragma unroll
  for (int k = 0; k < kPre; ++k) {
    if (k < cnt) {
      const float w = fast_exp2(lse[slot(k)] - m);
      L += w;
#pragma unroll
      for (int e = 0; e < PER; ++e) o[e] += w * pre[k][e];
    }
  }
  for (int i = kPre; i < cnt; ++i) {  // rows with more than kPre partials
    const int s = slot(i);
    const float w = fast_exp2(lse[s] - m);
    L += w;
    if constexpr (PER == 4) {
      const float4 v = *reinterpret_cast<const float4*>(po + (int64_t)s * HD);
      o[0] += w * v.x; o[1] += w * v.y; o[2] += w * v.z; o[3] += w * v.w;
    } else {
      const float2 v = *reinterpret_cast<const float2*>(po + (int64_t)s * HD);
      o[0] += w * v.x; o[1] += w * v.y;
    }
  }
  const float inv = 1.f / L;
#pragma unroll
  for (int k = 0; k < PER; ++k) store_act<AT>(p.out, bh * HD + lane * PER + k, o[k] * inv);
  if (p.lse_out && lane == 0) p.lse_out[bh] = (m + log2f(L)) * kLn2;
}

constexpr int kNW = 4;

template <int HD, int CT>
constexpr int stages_for() {
  // ~12 KB of copies in flight per warp (at least two stages): CTAs of 48-64 KB,
  // so three or four share an SM (four is also the register limit at ~123
  // registers).  More CTAs in flight beat deeper pipelines: on GB300, fp8 d128
  // at 3 stages took 180 us where 6 took 206 us (70B-shaped layer), bf16 d128
  // at 2 stages 98.6 us where 3 took 99.2 us (8B-shaped layer).
  constexpr int st = DecodeCfg<HD, CT, kNW, 1>::STAGEB;
  constexpr int ns = (12 * 1024) / st;
  return ns < 2 ? 2 : (ns > 8 ? 8 : ns);
}

// NSO > 0 overrides the pipeline depth (stages per warp), NW the warps per CTA.
template <int HD, int CT, int AT, bool CASC, int NSO = 0, int NW = kNW>
cudaError_t launch_decode_t(const CUtensorMap& kmap, const CUtensorMap& vmap,
                            const DecodeParams& p, const DecodeExtraParams& ap,
                            cudaStream_t stream, cudaEvent_t merge_after = nullptr) {
  constexpr int NS = NSO > 0 ? NSO : stages_for<HD, CT>();
  using C = DecodeCfg<HD, CT, NW, NS>;
  auto kern = decode_kernel<HD, CT, AT, NW, NS, CASC>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_kv_heads * ((p.group + 7) / 8), p.batch, p.num_splits);
  kern<<<grid, NW * 32, C::SMEM, stream>>>(kmap, vmap, p, ap);
  e = cudaGetLastError();
  if (e != cudaSuccess || (!CASC && p.num_splits <= 1)) return e;
  if (merge_after != nullptr && (e = cudaStreamWaitEvent(stream, merge_after, 0)) != cudaSuccess)
    return e;
  const int64_t pairs = (int64_t)p.batch * p.num_q_heads;
  merge_kernel<HD, AT, CASC><<<(unsigned)((pairs + 3) / 4), 128, 0, stream>>>(p, ap);
  return cudaGetLastError();
}

}  // namespace

size_t decode_smem_bytes(int head_dim, int cache_dt) {
  switch (head_dim * 4 + cache_dt) {
    case 64 * 4 + DT_F16: return DecodeCfg<64, DT_F16, kNW, stages_for<64, DT_F16>()>::SMEM;
    case 64 * 4 + DT_BF16: return DecodeCfg<64, DT_BF16, kNW, stages_for<64, DT_BF16>()>::SMEM;
    case 64 * 4 + DT_E4M3: return DecodeCfg<64, DT_E4M3, kNW, stages_for<64, DT_E4M3>()>::SMEM;
    case 128 * 4 + DT_F16: return DecodeCfg<128, DT_F16, kNW, stages_for<128, DT_F16>()>::SMEM;
    case 128 * 4 + DT_BF16: return DecodeCfg<128, DT_BF16, kNW, stages_for<128, DT_BF16>()>::SMEM;
    case 128 * 4 + DT_E4M3: return DecodeCfg<128, DT_E4M3, kNW, stages_for<128, DT_E4M3>()>::SMEM;
    default: return 0;
  }
}

cudaError_t launch_decode(const CUtensorMap& kmap, const CUtensorMap& vmap, const DecodeParams& p,
                          const DecodeExtraParams& ap, int head_dim, int cache_dt, int act_dt,
                          cudaStream_t stream) {
#define PKV_DEC(HD, CT, AT)                                              \
  if (head_dim == HD && cache_dt == CT && act_dt == AT)                  \
    return launch_decode_t<HD, CT, AT, false>(kmap, vmap, p, ap, stream);
  PKV_DEC(64, DT_F16, DT_F16)
  PKV_DEC(64, DT_BF16, DT_BF16)
  PKV_DEC(64, DT_E4M3, DT_F16)
  PKV_DEC(64, DT_E4M3, DT_BF16)
  PKV_DEC(128, DT_F16, DT_F16)
  PKV_DEC(128, DT_BF16, DT_BF16)
  PKV_DEC(128, DT_E4M3, DT_F16)
  PKV_DEC(128, DT_E4M3, DT_BF16)
#undef PKV_DEC
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_cascade(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                  const DecodeParams& p, const DecodeExtraParams& ap, int head_dim,
                                  int cache_dt, int act_dt, cudaStream_t stream,
                                  cudaEvent_t merge_after) {
  if (!ap.group_indptr || !ap.group_prefix_lens || ap.num_groups <= 0 || !p.ws_o)
    return cudaErrorInvalidValue;
  // Short runs per CTA (the members' own tokens are typically a few hundred):
  // small CTAs of two warps with two stages each (~33 KB at bf16 d128), so
  // that many fit on an SM and their fixed costs (setup, first copy,
  // epilogue) overlap.  Shared-prompt layer, 320 tokens per CTA: 50.5 us,
  // against 51.5 (2 warps, 1 stage), 53.1 (4 warps, 1 stage), 59.6 (4 warps,
  // 3 stages) and 65.5 (8 warps, 1 stage).  Long runs keep the plain decode's
  // configuration.
  const bool short_runs = p.chunk <= 512;
#define PKV_CASC(HD, CT, AT)                                                                   \
  if (head_dim == HD && cache_dt == CT && act_dt == AT)                                        \
    return short_runs                                                                          \
               ? launch_decode_t<HD, CT, AT, true, 2, 2>(kmap, vmap, p, ap, stream, merge_after) \
               : launch_decode_t<HD, CT, AT, true>(kmap, vmap, p, ap, stream, merge_after);
  PKV_CASC(64, DT_F16, DT_F16)
  PKV_CASC(64, DT_BF16, DT_BF16)
  PKV_CASC(64, DT_E4M3, DT_F16)
  PKV_CASC(64, DT_E4M3, DT_BF16)
  PKV_CASC(128, DT_F16, DT_F16)
  PKV_CASC(128, DT_BF16, DT_BF16)
  PKV_CASC(128, DT_E4M3, DT_F16)
  PKV_CASC(128, DT_E4M3, DT_BF16)
#undef PKV_CASC
  return cudaErrorInvalidValue;
}

}  // namespace pkv
