// Paged extend (suffix prefill) on the 5th-generation tensor cores.
//
// "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03: the
// longest cached prefix is reused and only the suffix is computed; prefill is
// compute-bound ("KV Cache에 대해 알아보자 (Feat. Attention)", §3), so this
// is the one dense contraction of the path and runs on tcgen05 with TMEM
// accumulators.
//
// Work item: a 128-row tile of packed (suffix token, query head) rows of one
// (request, kv head): with a GQA group of G heads the tile holds 128/G
// consecutive suffix tokens x G heads, all sharing the same K/V.  Row r
// (token i, head j) attends to keys 0 .. prefix + i.  Keys are consumed in
// tiles of 128 read through the block table.
//
// The kernel is persistent: one CTA per SM walks the items with a fixed
// stride, and every pipeline (K and V rings, S, P, O) runs straight through
// item boundaries, so loading the next item's Q, block ids and first K/V
// tiles, and writing the previous item's output, overlap the tensor work.
//
// Measured on this part, an MMA that reads its A operand from shared memory
// runs well below the tensor peak for this shape, one that reads A from TMEM
// at the peak, so both A operands (Q for S = Q K^T, P for O += P V) live in
// TMEM.  TMEM: one fp32 S tile, the O accumulator, two Q tiles and two f16 P
// tiles.  Q arrives by TMA in a shared-memory stage and is copied into the
// TMEM Q tile of its item (tcgen05.cp).  The S tile is released as soon as the
// softmax has its row in registers, so S = Q K^T of the next key tile runs
// while the softmax works; P of key tile n goes to P buffer n mod 2 while
// O += P V of tile n-1 reads the other.  Every reuse of a TMEM or
// shared-memory buffer is ordered by an mbarrier.
//
// Warp roles (384 threads):
//   warp 0      TMA producer of the Q stage (per item) and of the K ring: per
//               key tile sixteen 16-token x 64-dim boxes addressed through the
//               block table (block ids prefetched into registers), 128-byte
//               swizzled.
//   warp 11     TMA producer of the V ring, the same way.
//   warp 1      TMEM owner and, on one lane, the MMA issuer: Q stage -> TMEM,
//               S = Q K^T (A = Q in TMEM, B = K tile K-major, M=N=K=128), then
//               O += P V for the previous key tile (A = P in TMEM, B = the V
//               tile as loaded, [key][dim], read as an MN-major operand).
//   warps 2-3,  V converters: bf16 V tiles are turned into f16 in place and
//   8-10        keys past the sequence end are zeroed (they may hold NaN).
//   warps 4-7   softmax (one thread per row): per key tile reads its
//               128-column S row from TMEM with one wait, takes the row max
//               (causal mask on diagonal tiles), keeps a running max with lazy
//               rescaling (O in TMEM is rescaled only when the max grows by
//               more than 2^8) and writes f16 P; at the end of an item O / l
//               and the LSE.
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
constexpr int NTHREADS = 512;
constexpr int NCONV = 128;    // V converter threads (warps 2, 3, 8, 9: one per SM sub-partition)
constexpr int NSMX = 8;       // softmax warps: two per SM sub-partition
constexpr int NST = 3;        // K and V ring depth
constexpr int TILE = BN * HD * 2;   // 32 KB: 128 x 128 16-bit elements
constexpr int CHUNK = 16384;        // one 64-element column block [128 rows][128 B]

constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + NST * TILE;
constexpr int OFF_XM = OFF_V + NST * TILE;   // row-max exchange [2 tiles][2 halves][128 rows] f32
constexpr int OFF_XL = OFF_XM + 2 * 2 * BM * 4;   // row-sum exchange [2 halves][128 rows] f32
constexpr int OFF_BAR = OFF_XL + 2 * BM * 4;
enum {
  B_KFULL = 0, B_VFULL = B_KFULL + NST, B_VCONV = B_VFULL + NST,
  // S(n) = Q K^T of key tile n done: S is readable, K stage n mod NST free
  B_SDONE = B_VCONV + NST,
  // O += P V of key tile n done: P buffer n mod 2, O and V stage n mod NST free
  B_PVDONE = B_SDONE + NST,
  B_SFREE = B_PVDONE + NST,   // every softmax warp has its half of S in registers
  B_PFULL = B_SFREE + 1,      // [2] P buffer written
  B_QFULL = B_PFULL + 2,      // [2] TMEM Q tile i written
  B_QDONE = B_QFULL + 2,      // [2] every S = Q K^T of the item using TMEM Q tile i done
  B_OFREE = B_QDONE + 2,      // the item's O has been read out of TMEM
  B_MX = B_OFREE + 1,         // [2] partial row maxima of key tile n written (slot n mod 2)
  B_LX = B_MX + 2,            // partial row sums of the item written
  NBAR = B_LX + 1
};
constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_TMEMSLOT + 16 + 1024;
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TM_S = 0;     // fp32 S tile, 128 columns
constexpr uint32_t TM_O = 128;   // O accumulator, 128 columns
constexpr uint32_t TM_Q = 256;   // two Q tiles of 64 columns of 16-bit pairs
constexpr uint32_t TM_P = 384;   // two P tiles of 64 columns of f16 pairs
constexpr float kLn2f = 0.6931471805599453f;

__device__ __forceinline__ void set_err(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// Per-request values an item needs, loaded one item ahead.
struct ItemRaw {
  int r0, r1, prefix;
};

struct Item {
  int b, g, i0, ntok, P, S, row0, kv_total, k_hi, T;
};

__device__ __forceinline__ ItemRaw load_raw(const ExtendParams& p, int item) {
  ItemRaw r{0, 0, 0};
  if (item < p.num_items) {
    const int b = item / (p.tiles_per_head * p.num_kv_heads);
    r.r0 = __ldg(p.q_indptr + b);
    r.r1 = __ldg(p.q_indptr + b + 1);
    r.prefix = __ldg(p.prefix_lens + b);
  }
  return r;
}

// false: the tile holds no suffix rows (the same answer in every role)
__device__ __forceinline__ bool derive(const ExtendParams& p, int item, const ItemRaw& r, Item& it) {
  const int tile = item % p.tiles_per_head;
  const int rest = item / p.tiles_per_head;
  it.g = rest % p.num_kv_heads;
  it.b = rest / p.num_kv_heads;
  const int TOK = BM / p.group;
  it.row0 = r.r0;
  it.S = r.r1 - r.r0;
  it.i0 = tile * TOK;
  if (it.i0 >= it.S) return false;
  it.ntok = min(TOK, it.S - it.i0);
  it.P = r.prefix;
  const int cap = p.max_blocks << p.bs_shift;
  it.kv_total = it.P + it.S;
  it.k_hi = it.P + it.i0 + it.ntok;  // keys this tile needs
  if (it.P < 0 || it.kv_total > cap) {
    set_err(p.err, 3);
    it.kv_total = min(max(it.kv_total, 0), cap);
    it.k_hi = min(max(it.k_hi, 1), max(cap, 1));
  }
  it.T = (it.k_hi + BN - 1) / BN;
  return true;
}

// The next item at or after `from` (stride apart) that holds suffix rows;
// p.num_items when there is none.
__device__ __forceinline__ int next_item(const ExtendParams& p, int from, int stride, Item& it) {
  for (int item = from; item < p.num_items; item += stride)
    if (derive(p, item, load_raw(p, item), it)) return item;
  return p.num_items;
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
  float* xmax = reinterpret_cast<float*>(smem + OFF_XM);
  float* xsum = reinterpret_cast<float*>(smem + OFF_XL);
  const uint32_t s_base = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int item0 = blockIdx.x, stride = gridDim.x;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(B_KFULL + i), 1);
      mbar_init(bar(B_VFULL + i), 1);
      mbar_init(bar(B_VCONV + i), NCONV / 32);
      mbar_init(bar(B_SDONE + i), 1);
      mbar_init(bar(B_PVDONE + i), 1);
    }
    mbar_init(bar(B_SFREE), NSMX);
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(B_PFULL + i), NSMX);
      mbar_init(bar(B_QFULL + i), NCONV / 32);
      mbar_init(bar(B_QDONE + i), 1);
      mbar_init(bar(B_MX + i), NSMX);
    }
    mbar_init(bar(B_OFREE), NSMX);
    mbar_init(bar(B_LX), NSMX);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  // registers: launched with 128 per thread (512 x 128); the two softmax
  // warpgroups (warps 4-7 and 12-15) raise their budget to 152, the other two
  // lower theirs to 104: 2 x 152 + 2 x 104 = 4 x 128.
  static_assert(2 * 152 + 2 * 104 == 4 * 128, "register split must equal the launch budget");
  if ((warp >= 4 && warp < 8) || warp >= 12) {
    regs_inc<152>();
    // ------------------------------------------------------------ softmax
    // Two warps per row quarter: half h takes keys 64h .. 64h+63 of every
    // key tile and dims 64h .. 64h+63 of O.  The row max is combined through
    // shared memory every key tile, the row sum once per item.
    const int h = warp >= 12 ? 1 : 0;
    const int qw = warp & 3;
    const int r = qw * 32 + lane;
    const uint32_t lane_addr = (uint32_t)(qw * 32) << 16;
    const uint32_t srow = tmem + lane_addr + TM_S + h * 64;
    const uint32_t orow = tmem + lane_addr + TM_O + h * 64;
    int n = 0, js = 0;
    // Output rows are written back late: the packed half row of the previous
    // item stays in registers and goes out in two groups of four 16-byte
    // stores, one group per key tile of the next item, so the row-strided
    // stores drain behind the softmax instead of stalling it.
    uint32_t w[32];
    uint4* pdst = nullptr;
    int pstage = 2;  // next group to store; 2: nothing pending
    auto store_group = [&]() {
      if (pstage < 2) {
#pragma unroll
        for (int g4 = 0; g4 < 2; ++g4)
          if (g4 == pstage) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              pdst[4 * g4 + q] = make_uint4(w[16 * g4 + 4 * q], w[16 * g4 + 4 * q + 1],
                                            w[16 * g4 + 4 * q + 2], w[16 * g4 + 4 * q + 3]);
          }
        ++pstage;
      }
    };
    ItemRaw nxt_raw = load_raw(p, item0);
    for (int item = item0; ok && item < p.num_items; item += stride) {
      const ItemRaw raw = nxt_raw;
      nxt_raw = load_raw(p, item + stride);
      Item it;
      if (!derive(p, item, raw, it)) continue;
      const int kdiag = it.P + it.i0;  // a row's last visible key is kdiag + its token
      float m_run = -INFINITY, l_run = 0.f;
      for (int kt = 0; kt < it.T; ++kt, ++n) {
        const int pb = n & 1;
        if (!mbar_wait(bar(B_SDONE + n % NST), (n / NST) & 1)) { ok = false; break; }
        tc_fence_after();
        const int key0 = kt * BN;
        if (key0 + BN - 1 > kdiag) {
          // causal mask on a tile that reaches past some row's limit (keys
          // key0 .. key0+nvis are visible): applied in TMEM one 32-column
          // chunk at a time, a short rolled loop that runs on one or two key
          // tiles per item
          const int nvis = kdiag + r / G - key0 - h * 64;
          const uint32_t ninf = __float_as_uint(-INFINITY);
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t t[32];
            tmem_ld32(srow + c * 32, t);
            tmem_wait_ld();
            const int lc = nvis - c * 32;
#pragma unroll
            for (int q = 0; q < 32; ++q) t[q] = (q > lc) ? ninf : t[q];
            tmem_st32(srow + c * 32, t);
          }
          tmem_wait_st();
        }
        // this half of the S row: two 32-column loads, one wait
        uint32_t sr[2][32];
#pragma unroll
        for (int c = 0; c < 2; ++c) tmem_ld32(srow + c * 32, sr[c]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_SFREE));  // S is in registers
        // partial row max: three-input max over 8 independent accumulators
        float mx[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx[a] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int q = 0; q < 16; ++q)
            mx[q & 7] = fmax3(mx[q & 7], __uint_as_float(sr[c][2 * q]), __uint_as_float(sr[c][2 * q + 1]));
        const float mpart = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                                  fmaxf(mx[6], mx[7]));
        // combine with the other half through shared memory (slot n mod 2)
        float* xm = xmax + (n & 1) * (2 * BM);
        xm[h * BM + r] = mpart;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_MX + (n & 1)));
        if (!mbar_wait(bar(B_MX + (n & 1)), (n >> 1) & 1)) { ok = false; break; }
        const float mt = fmaxf(mpart, xm[(1 - h) * BM + r]) * p.scale_log2;
        float m_new = m_run;
        if (mt > m_run + 8.f) m_new = mt;
        const float alpha = fast_exp2(m_run - m_new);
        const bool mine = (m_new != m_run);
        if (kt >= 1 && __any_sync(0xFFFFFFFFu, mine)) {
          // rescale this half of O in TMEM once PV(n-1) has finished
          if (!mbar_wait(bar(B_PVDONE + (n - 1) % NST), ((n - 1) / NST) & 1)) { ok = false; break; }
          tc_fence_after();
          const float f = mine ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld32(orow + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * f);
            tmem_st32(orow + c * 32, o);
          }
          tmem_wait_st();
        }
        m_run = m_new;
        // p = 2^(s*scale - m) as f16 pairs into this half of P buffer pb, once
        // PV(n-2) has consumed P(n-2); pairs of keys through the packed fp32 pipe
        if (n >= 2 && !mbar_wait(bar(B_PVDONE + (n - 2) % NST), ((n - 2) / NST) & 1)) { ok = false; break; }
        tc_fence_after();
        float2 sm[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) sm[a] = make_float2(0.f, 0.f);
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nm2 = make_float2(-m_new, -m_new);
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float2 x = __ffma2_rn(
                make_float2(__uint_as_float(sr[c][2 * q]), __uint_as_float(sr[c][2 * q + 1])), sc2, nm2);
            const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
            sm[q & 3] = __fadd2_rn(sm[q & 3], pe);
            pk[q] = pack2<false>(pe.x, pe.y);
          }
          tmem_st16(tmem + lane_addr + TM_P + pb * 64 + h * 32 + c * 16, pk);
        }
        const float sum = ((sm[0].x + sm[1].x) + (sm[2].x + sm[3].x)) +
                          ((sm[0].y + sm[1].y) + (sm[2].y + sm[3].y));
        l_run = l_run * alpha + sum;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_PFULL + pb));
        store_group();
      }
      if (!ok) break;
      // ---- item epilogue: the row sum of both halves, O out of TMEM (then O
      // is free for the next item), O / l -> out, LSE
      xsum[h * BM + r] = l_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_LX));
      const int u = n - 1;  // last key tile of this item
      if (!mbar_wait(bar(B_PVDONE + u % NST), (u / NST) & 1)) { ok = false; break; }
      if (!mbar_wait(bar(B_LX), js & 1)) { ok = false; break; }
      const float l_tot = l_run + xsum[(1 - h) * BM + r];
      tc_fence_after();
      while (pstage < 2) store_group();  // the previous item's row, if still pending
      const float osc = p.out_scale / l_tot;
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t o[32];
        tmem_ld32(orow + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int q = 0; q < 16; ++q)
          w[c * 16 + q] = pack2<CT == DT_BF16>(__uint_as_float(o[2 * q]) * osc,
                                               __uint_as_float(o[2 * q + 1]) * osc);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_OFREE));
      if ((r / G) < it.ntok) {
        const int64_t qrow = (int64_t)(it.row0 + it.i0 + r / G) * p.num_q_heads + it.g * G + (r % G);
        pdst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + qrow * HD + h * 64);
        pstage = 0;
        if (h == 0 && p.lse_out) p.lse_out[qrow] = (m_run + log2f(l_tot)) * kLn2f;
      }
      ++js;
    }
    while (pstage < 2) store_group();
  } else {
    regs_dec<104>();
    if (warp == 0 || warp == 11) {
      // ------------------------------------------------------------ producers
      // warp 0 streams K tiles, warp 11 V tiles, each through its own ring,
      // so that a K load never queues behind a V buffer that is still in use.
      // Block ids: lane l holds sub-tile (32 w + l) of window w, the next
      // window is fetched one window ahead.
      const bool is_k = (warp == 0);
      const CUtensorMap* map = is_k ? &kmap : &vmap;
      // a stage is free once the MMA that read it has completed
      const int full0 = is_k ? B_KFULL : B_VFULL, free0 = is_k ? B_SDONE : B_PVDONE;
      const uint32_t ring = s_base + (is_k ? OFF_K : OFF_V);
      int n = 0;  // key tiles so far
      ItemRaw nxt_raw = load_raw(p, item0);
      for (int item = item0; ok && item < p.num_items; item += stride) {
        const ItemRaw raw = nxt_raw;
        nxt_raw = load_raw(p, item + stride);
        Item it;
        if (!derive(p, item, raw, it)) continue;
        const int32_t* bt = p.block_tables + (int64_t)it.b * p.max_blocks;
        auto fetch = [&](int wi) -> int {
          const int key0 = (wi * 32 + lane) * 16;  // sub-tile = 16 keys
          int page = -1;
          if (key0 < it.k_hi) {
            const int blk = bt[key0 >> p.bs_shift];
            if (blk < 0 || blk >= p.num_blocks) set_err(p.err, 1);  // TMA zero-fills page -1
            else page = blk * p.num_kv_heads + it.g;
          }
          return page;
        };
        int win = 0, cur = fetch(0), nxt = fetch(1);
        for (int kt = 0; kt < it.T; ++kt, ++n) {
          const int s = n % NST;
          if ((kt >> 2) > win) {  // 4 tiles x 8 sub-tiles per window
            cur = nxt;
            ++win;
            nxt = fetch(win + 1);
          }
          int pg[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) pg[q] = __shfl_sync(0xFFFFFFFFu, cur, (kt & 3) * 8 + q);
          if (n >= NST && !mbar_wait(bar(free0 + s), (uint32_t)((n / NST - 1) & 1))) { ok = false; break; }
          if (lane == 0) {
            const uint32_t dst = ring + s * TILE;
            mbar_arrive_expect_tx(bar(full0 + s), TILE);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const int rip = (kt * BN + 16 * q) & ((1 << p.bs_shift) - 1);
#pragma unroll
              for (int c = 0; c < 2; ++c)
                tma_load_3d(dst + c * CHUNK + q * 2048, map, bar(full0 + s), c * 64, rip, pg[q]);
            }
          }
        }
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the loop (every operand is warp-uniform); one
      // elected lane issues the MMAs and commits.
      {
        constexpr uint32_t qk_fmt = (CT == DT_BF16) ? 1u : 0u;
        constexpr uint32_t idesc_qk = umma_idesc_f16(qk_fmt, qk_fmt, BM, BN);
        // P (A, f16 in TMEM) x V (B, f16, MN-major: the V tile as loaded, [key][dim])
        constexpr uint32_t idesc_pv = umma_idesc_f16(0u, 0u, BM, HD) | (1u << 16);
        // O += P V of key tile u; `first`: the first key tile of item ju, which
        // overwrites O once the previous item's O has been read out
        auto issue_pv = [&](int u, bool first, int ju) -> bool {
          const int us = u % NST, pb = u & 1;  // V stage, P buffer
          if (!mbar_wait(bar(B_PFULL + pb), (u >> 1) & 1)) return false;
          if (!mbar_wait(bar(B_VCONV + us), (u / NST) & 1)) return false;
          if (first && ju >= 1 && !mbar_wait(bar(B_OFREE), (ju - 1) & 1)) return false;
          tc_fence_after();
          const uint64_t vdesc = umma_desc_sw128_mn(s_base + OFF_V + us * TILE, CHUNK);
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk)
              umma_f16_ts(tmem + TM_O, tmem + TM_P + pb * 64 + kk * 8, vdesc + (uint64_t)(kk * 2048 >> 4),
                          idesc_pv, (!first || kk > 0) ? 1u : 0u);
            umma_commit(bar(B_PVDONE + us));
          }
          __syncwarp();
          return true;
        };
        int n = 0, j = 0;
        bool have_prev = false, prev_first = false;
        int prev_n = 0, prev_j = 0;
        ItemRaw nxt_raw = load_raw(p, item0);
        for (int item = item0; ok && item < p.num_items; item += stride) {
          const ItemRaw raw = nxt_raw;
          nxt_raw = load_raw(p, item + stride);
          Item it;
          if (!derive(p, item, raw, it)) continue;
          const int qb = j & 1;
          if (!mbar_wait(bar(B_QFULL + qb), (j >> 1) & 1)) { ok = false; break; }
          for (int kt = 0; kt < it.T; ++kt, ++n) {
            const int ks = n % NST;
            if (!mbar_wait(bar(B_KFULL + ks), (n / NST) & 1)) { ok = false; break; }
            // the S tile is free once the softmax has read S(n-1) into registers
            if (n >= 1 && !mbar_wait(bar(B_SFREE), (n - 1) & 1)) { ok = false; break; }
            tc_fence_after();
            const uint64_t kdesc = umma_desc_sw128(s_base + OFF_K + ks * TILE);
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < HD / 16; ++kk) {
                const uint32_t off = (kk >> 2) * CHUNK + (kk & 3) * 32;
                umma_f16_ts(tmem + TM_S, tmem + TM_Q + qb * 64 + kk * 8, kdesc + (uint64_t)(off >> 4),
                            idesc_qk, kk > 0 ? 1u : 0u);
              }
              umma_commit(bar(B_SDONE + ks));
              if (kt == it.T - 1) umma_commit(bar(B_QDONE + qb));
            }
            __syncwarp();
            if (have_prev && !issue_pv(prev_n, prev_first, prev_j)) { ok = false; break; }
            have_prev = true;
            prev_n = n;
            prev_first = (kt == 0);
            prev_j = j;
          }
          ++j;
        }
        if (ok && have_prev) ok = issue_pv(prev_n, prev_first, prev_j);
      }
      __syncwarp();
    } else if (warp != 10) {
      // ------------------------------------------------------------ V converters and Q loaders (2, 3, 8, 9)
      // V: in place, per 16-byte unit: bf16 -> f16 (the PV product is
      // f16 x f16), and keys at or past the sequence end -> 0 (they may hold
      // anything, and 0 * NaN is NaN).  The swizzle only permutes units inside
      // a 128-byte key row, so the key of a unit is its byte offset / 128
      // within its block.
      // Q: warp w writes rows 32 (w mod 4) .. +31 of TMEM Q tile j mod 2 for
      // item j, one item ahead (after the first V tile of the item before).
      const int cw = warp == 2 ? 0 : warp == 3 ? 1 : warp == 8 ? 2 : 3;
      const int ct = cw * 32 + lane;  // 0..127
      const int rq = (warp & 3) * 32 + lane;  // Q row (TMEM lane) this thread writes
      constexpr int PER = TILE / 16 / NCONV;  // 16 units of 16 bytes per thread
      static_assert(PER * NCONV * 16 == TILE, "converter units");
      auto load_q = [&](const Item& iq, int jq) -> bool {
        const int qb = jq & 1;
        if (jq >= 2 && !mbar_wait(bar(B_QDONE + qb), ((jq - 2) >> 1) & 1)) return false;
        tc_fence_after();
        const bool valid = (rq / G) < iq.ntok;
        const int64_t qrow = (int64_t)(iq.row0 + iq.i0 + rq / G) * p.num_q_heads + iq.g * G + (rq % G);
        const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const uint16_t*>(p.q) + qrow * HD);
        uint4 qv[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) qv[i] = valid ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t qaddr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + TM_Q + qb * 64;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[16];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            v[4 * i] = qv[4 * c + i].x; v[4 * i + 1] = qv[4 * c + i].y;
            v[4 * i + 2] = qv[4 * c + i].z; v[4 * i + 3] = qv[4 * c + i].w;
          }
          tmem_st16(qaddr + c * 16, v);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_QFULL + qb));
        return true;
      };
      int n = 0, j = 0;
      Item cur;
      int item = next_item(p, item0, stride, cur);
      if (item < p.num_items) ok = load_q(cur, 0);
      while (ok && item < p.num_items) {
        Item nxt;
        const int nitem = next_item(p, item + stride, stride, nxt);
        for (int kt = 0; kt < cur.T; ++kt, ++n) {
          const int vs = n % NST;
          if (!mbar_wait(bar(B_VFULL + vs), (n / NST) & 1)) { ok = false; break; }
          const int kbase = kt * BN;
          uint4* vt = reinterpret_cast<uint4*>(smem + OFF_V + vs * TILE);
          if (kbase + BN > cur.kv_total) {  // tail tile: zero the keys past the end
#pragma unroll 4
            for (int i = 0; i < PER; ++i) {
              const int uu = ct + i * NCONV;
              uint4 x = vt[uu];
              if (kbase + ((uu * 16) % CHUNK) / 128 >= cur.kv_total) {
                x = make_uint4(0u, 0u, 0u, 0u);
              } else if (CT == DT_BF16) {
                x.x = to_f16x2<true>(x.x);
                x.y = to_f16x2<true>(x.y);
                x.z = to_f16x2<true>(x.z);
                x.w = to_f16x2<true>(x.w);
              }
              vt[uu] = x;
            }
            fence_async_smem();
          } else if (CT == DT_BF16) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {  // two batches of 8 loads in flight
              uint4 x[PER / 2];
#pragma unroll
              for (int i = 0; i < PER / 2; ++i) x[i] = vt[ct + (hh * (PER / 2) + i) * NCONV];
#pragma unroll
              for (int i = 0; i < PER / 2; ++i) {
                x[i].x = to_f16x2<true>(x[i].x);
                x[i].y = to_f16x2<true>(x[i].y);
                x[i].z = to_f16x2<true>(x[i].z);
                x[i].w = to_f16x2<true>(x[i].w);
                vt[ct + (hh * (PER / 2) + i) * NCONV] = x[i];
              }
            }
            fence_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(B_VCONV + vs));
          if (kt == 0 && nitem < p.num_items && !load_q(nxt, j + 1)) { ok = false; break; }
        }
        cur = nxt;
        item = nitem;
        ++j;
      }
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
  if (p.num_items <= 0 || p.num_ctas <= 0) return cudaErrorInvalidValue;
  const dim3 grid(p.num_ctas);
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
