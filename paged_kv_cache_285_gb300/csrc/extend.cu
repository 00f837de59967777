// Paged extend (suffix prefill) on the 5th-generation tensor cores.
//
// "PagedAttention과 RadixAttention으로 LLM KV 캐시 최적화", section 03: the
// longest cached prefix is reused and only the suffix is computed; prefill is
// compute-bound ("KV Cache에 대해 알아보자 (Feat. Attention)", §3), so this
// is the one dense contraction of the path and runs on tcgen05 with TMEM
// accumulators.
//
// Rows: a 128-row tile packs (suffix token, query head) rows of one
// (request, kv head): with a GQA group of G heads it holds tok = 128/G
// consecutive suffix tokens x G heads (row = token * G + head), all sharing
// the same K/V.  Row r (token i, head j) attends to keys 0 .. prefix + i.
// Keys are consumed in tiles of 128 read through the block table.
//
// Work item: two consecutive row tiles A and B of one (request, kv head).
// Both use every K/V tile, and their softmaxes run on separate warps in
// ping-pong: while the softmax of A works on S_A, the tensor core computes
// O_B += P_B V and S_B = Q_B K^T, and the other way round, so the tensor core
// and the softmax warps overlap instead of waiting for each other.  The kernel
// is persistent: one CTA per SM walks the items with a fixed stride and every
// pipeline runs through item boundaries.
//
// TMEM (512 columns): S_A, S_B (fp32, 128 columns each) and O_A, O_B (fp32,
// head_dim columns each).  P of a tile is written as f16 over the first 64
// columns of its own S once the softmax has S in registers, and O += P V
// reads it from there; the next S = Q K^T of that tile is issued after that PV
// by the same thread (MMAs of one thread execute in issue order).  Shared
// memory: Q of three row tiles (the A and B tiles of an item and one tile of
// the next), K and V rings.  S = Q K^T reads both operands from shared memory,
// O += P V reads P from TMEM and V, as loaded ([key][dim]), as an MN-major
// operand.
//
// Warp roles (512 threads):
//   warp 0        TMA producer of Q tiles and of the K ring (block ids
//                 prefetched into registers, 16-token boxes, swizzled).
//   warp 1        TMEM owner and MMA issuer: the whole warp runs the loop with
//                 warp-uniform operands, one elected lane issues.
//   warp 2        TMA producer of the V ring.
//   warps 4-7     softmax of tile A (one thread per row), warps 8-11 of tile
//                 B: row max with lazy rescaling (O is rescaled in TMEM only
//                 when the max grows by more than 2^8), f16 P, and at the end
//                 of an item O / l and the LSE.
//   warps 12-15   converters: bf16 V tiles become f16 in place; fp8 (e4m3) K
//                 and V tiles are widened to f16 (exactly), one key row per
//                 thread, and with bf16 queries each Q tile is converted to
//                 f16 once per item, so S = Q K^T runs in f16; V keys past the
//                 sequence end are zeroed (they may hold NaN, and 0 * NaN is
//                 NaN).
// P is f16 (11 significant bits) because bf16 P alone would put the relative
// L2 error of the output near 1.5e-3; V is therefore f16 (bf16 values beyond
// +-65504 are outside this path's range).
//
// fp8 caches ("KV Cache 완전 정리 — PagedAttention vs RadixAttention, SGLang이
// 빠른 이유", "FP8 KV 캐시": half the bytes of a 16-bit cache) are read as
// codes: the TMA copies one byte per element, the converter warps widen each
// tile in shared memory, and the per-tensor scales are folded into the softmax
// scale (k_scale) and the output scale (v_scale), so no 16-bit copy of the
// cache exists anywhere.  bf16 queries over an fp8 cache are taken as f16
// (exact within the f16 range; query values beyond +-65504 are outside this
// path's range, like bf16 V values).
//
// Prefix pass (PP = true), for decode over a prefix shared by a group of
// requests: each group is one pseudo-request whose rows are the group
// members' query vectors (one token each), keys are the group's P shared
// tokens read through its first member's block table, every row sees all P
// of them and no other.  The keys are cut into chunks of kchunk_keys, one work
// item each (so that a few groups still fill the GPU), and each row's result
// over a chunk leaves as an fp32 partial (O / l and the base-2 LSE) in the
// chunk's slot, for an LSE merge with the member's own tokens.
#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int BM = 128;       // rows per tile
constexpr int BN = 128;       // keys per tile
constexpr int NTHREADS = 512;
constexpr int NCONV = 128;    // converter threads (warps 12-15), one per key row
constexpr int NQB = 3;        // Q tile buffers
constexpr int CHUNK = 16384;  // one 64-element column block of a 16-bit tile: [128 rows][128 B]

template <int HD, int CT, int AT>
struct ExtCfg {
  static constexpr bool FP8 = (CT == DT_E4M3);
  // S = Q K^T runs in f16 for fp8 caches: K codes widen to f16 with one
  // convert per pair, and bf16 queries (QCVT) are converted to f16 once per
  // item instead of K to bf16 at every key tile
  static constexpr bool QCVT = FP8 && (AT == DT_BF16);
  static constexpr bool QK_BF16 = !FP8 && (AT == DT_BF16);
  static constexpr int NCH = HD / 64;           // 64-element column blocks per 16-bit row
  static constexpr int NST = HD == 64 ? 3 : 2;  // K and V ring depth
  static constexpr int T16 = BM * HD * 2;       // a 16-bit tile (Q, K or V): 16 or 32 KB
  static constexpr int T8 = BN * HD;            // an fp8 K or V tile as loaded
  // fp8 tiles are loaded into the first half of their 16-bit slot and widened
  // in place at d128 (each converter thread owns one key row, and the 16-bit
  // bytes of that row's dims 0-63 are exactly its fp8 row); at d64 a 16-bit
  // row covers two fp8 rows, so the fp8 tiles get a staging ring of their own
  static constexpr bool STAGE8 = FP8 && HD == 64;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + NQB * T16;
  static constexpr int OFF_V = OFF_K + NST * T16;
  static constexpr int OFF_K8 = OFF_V + NST * T16;
  static constexpr int OFF_V8 = OFF_K8 + (STAGE8 ? NST * T8 : 0);
  static constexpr int OFF_BAR = OFF_V8 + (STAGE8 ? NST * T8 : 0);
  enum {
    B_KFULL = 0,              // [stage] K tile loaded
    B_VFULL = B_KFULL + NST,  // [stage] V tile loaded
    B_KCONV = B_VFULL + NST,  // [stage] fp8 K tile widened
    B_VCONV = B_KCONV + NST,  // [stage] V tile converted / tail zeroed
    B_KFREE = B_VCONV + NST,  // [stage] S_B(n) = Q_B K(n)^T done (S_A(n) before it): K stage free
    B_VFREE = B_KFREE + NST,  // [stage] O_B += P_B V(n) done (O_A's before it): V stage free
    B_SDONE = B_VFREE + NST,  // [2] S_x(n) = Q_x K(n)^T done
    B_PFULL = B_SDONE + 2,    // [2] P_x(n) written
    B_QFULL = B_PFULL + 2,    // [tile x][item parity] Q tile x of the item loaded
    B_QCONV = B_QFULL + 4,    // [tile x][item parity] Q tile x converted to f16 (fp8 cache, bf16 q)
    B_QFREE = B_QCONV + 4,    // [item parity] the item's last S_B = Q_B K^T done
    B_ODONE = B_QFREE + 2,    // the item's last O_B += P_B V done (O_A's before it)
    B_OFREE = B_ODONE + 1,    // [2] O_x of the item read out of TMEM
    B_EST = B_OFREE + 2,      // [2] tile x's output rows staged in shared memory (4 warps)
    B_EFREE = B_EST + 2,      // [2] tile x done with the staging buffer (its store has read it)
    NBAR = B_EFREE + 2
  };
  static constexpr int OFF_TMEMSLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TMEMSLOT + 16 + 1024;
  static_assert(SMEM <= 232448, "shared memory per CTA");
  // where the fp8 codes of stage s of the K (isv false) or V ring are loaded
  __host__ __device__ static constexpr int src8(bool isv, int s) {
    return STAGE8 ? (isv ? OFF_V8 : OFF_K8) + s * T8 : (isv ? OFF_V : OFF_K) + s * T16;
  }
};

// Whole output tiles leave through shared memory and TMA stores issued by warp
// 3, except in the shared-prefix kernel over fp8 codes at d128, whose segment
// walk, in-place widening and Q conversion already fill the instruction cache
// (with the stores: 904-910 against 879-881 us; the plain fp8 d128 kernel
// gains, 855 against 877).
template <int HD, int CT, bool SX>
__host__ __device__ constexpr bool out_tma_for() { return !(CT == DT_E4M3 && HD == 128 && SX); }

constexpr uint32_t TMEM_COLS = 512;
__host__ __device__ constexpr uint32_t tm_s(int x) { return (uint32_t)x * 128u; }  // S_x, then P_x
template <int HD>
__host__ __device__ constexpr uint32_t tm_o(int x) { return 256u + (uint32_t)x * HD; }  // O_x
constexpr float kLn2f = 0.6931471805599453f;

__device__ __forceinline__ void set_err(int32_t* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

// ---- converters ---------------------------------------------------------------
// A 16-bit tile is NCH column blocks of [128 key rows][128 B] in the 128-byte
// swizzle: logical 16-byte unit u of row t sits at unit u ^ (t & 7).  The
// swizzle only permutes units inside a row, so a unit's key row is its byte
// offset within its column block / 128.

// A 16-bit V tile in place, 16-byte units spread over the converter threads
// (thread ct takes units ct, ct + 128, ...: consecutive threads, consecutive
// units): bf16 -> f16 (CVT), and units of keys at or past kv_end -> zeros
// (TAIL; key0 is the tile's first key).  Measured faster than one key row per
// thread on the benchmark's bf16 tiles (896 against 945 us per call).
// A bf16 Q tile to f16 in place, once per item: a rolled loop (four units in
// flight per pass), so that this cold code takes little instruction cache
// beside the key-tile loops.
template <int HD>
__device__ __forceinline__ void conv_q_tile(uint8_t* tile, int ct) {
  constexpr int PER = BM * HD * 2 / 16 / NCONV;  // 16-byte units per thread
  uint4* v4 = reinterpret_cast<uint4*>(tile);
#pragma unroll 1
  for (int hh = 0; hh < PER; hh += 4) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = v4[ct + (hh + i) * NCONV];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[i].x = to_f16x2<true>(v[i].x);
      v[i].y = to_f16x2<true>(v[i].y);
      v[i].z = to_f16x2<true>(v[i].z);
      v[i].w = to_f16x2<true>(v[i].w);
      v4[ct + (hh + i) * NCONV] = v[i];
    }
  }
}

template <int HD, bool CVT, bool TAIL>
__device__ __forceinline__ void conv_tile16(uint8_t* tile, int ct, int key0, int kv_end) {
  constexpr int PER = BN * HD * 2 / 16 / NCONV;  // 16-byte units per thread
  uint4* v4 = reinterpret_cast<uint4*>(tile);
  if constexpr (TAIL) {
#pragma unroll 4
    for (int i = 0; i < PER; ++i) {
      const int uu = ct + i * NCONV;
      uint4 v = v4[uu];
      if (key0 + ((uu * 16) % CHUNK) / 128 >= kv_end) {
        v = make_uint4(0u, 0u, 0u, 0u);
      } else if (CVT) {
        v.x = to_f16x2<true>(v.x);
        v.y = to_f16x2<true>(v.y);
        v.z = to_f16x2<true>(v.z);
        v.w = to_f16x2<true>(v.w);
      }
      v4[uu] = v;
    }
  } else {
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {  // four batches of PER / 4 loads in flight
      uint4 v[PER / 4];
#pragma unroll
      for (int i = 0; i < PER / 4; ++i) v[i] = v4[ct + (hh * (PER / 4) + i) * NCONV];
#pragma unroll
      for (int i = 0; i < PER / 4; ++i) {
        v[i].x = to_f16x2<true>(v[i].x);
        v[i].y = to_f16x2<true>(v[i].y);
        v[i].z = to_f16x2<true>(v[i].z);
        v[i].w = to_f16x2<true>(v[i].w);
        v4[ct + (hh * (PER / 4) + i) * NCONV] = v[i];
      }
    }
  }
}

// Two e4m3 codes (low byte first) -> a 16-bit pair of OUT (exact).
template <int OUT>
__device__ __forceinline__ uint32_t widen2(uint32_t two) {
  const uint32_t h = e4m3x2_to_f16x2(two);
  if constexpr (OUT == DT_BF16) return pack2<true>(lo_f32<false>(h), hi_f32<false>(h));
  else return h;
}

// 16 codes -> 16 OUT values in two 16-byte units.
template <int OUT>
__device__ __forceinline__ void widen16(const uint4& a, uint4& lo, uint4& hi) {
  lo = make_uint4(widen2<OUT>(a.x & 0xFFFFu), widen2<OUT>(a.x >> 16), widen2<OUT>(a.y & 0xFFFFu),
                  widen2<OUT>(a.y >> 16));
  hi = make_uint4(widen2<OUT>(a.z & 0xFFFFu), widen2<OUT>(a.z >> 16), widen2<OUT>(a.w & 0xFFFFu),
                  widen2<OUT>(a.w >> 16));
}

// Fp8 key row t (codes at src) -> 16-bit row t of the tile at dst, or zeros.
//  d128: src == dst (in place).  The fp8 row is 128 B at t * 128 in the
//        128-byte swizzle (logical unit u = dims 16u .. 16u+15 at u ^ (t & 7)),
//        and 16-bit unit w of row t in column block 0 sits at the same place as
//        fp8 unit w: dims 64-127 go to column block 1 (past the fp8 tile)
//        first, then fp8 units 3, 2 -> 16-bit units 7 .. 4 and fp8 units 1, 0
//        -> units 3 .. 0, so every store lands on fp8 units already read.  No
//        other thread touches the row.
//  d64:  src is a separate staging tile: 64 B rows at t * 64 in the 64-byte
//        swizzle (unit u at u ^ ((t >> 1) & 3)).
// A swizzled offset row + 16 (u ^ c) is (row | 16 c) ^ 16 u: one xor with a
// constant per unit.
template <int HD, int OUT>
__device__ __forceinline__ void widen_row(const uint8_t* src, uint8_t* dst, int t, bool zero) {
  const uint32_t sbase = (HD == 128) ? ((uint32_t)t * 128u) | (((uint32_t)t & 7u) << 4)
                                     : ((uint32_t)t * 64u) | ((((uint32_t)t >> 1) & 3u) << 4);
  const uint32_t dbase = ((uint32_t)t * 128u) | (((uint32_t)t & 7u) << 4);
#pragma unroll
  for (int pr = HD / 32 - 1; pr >= 0; --pr) {  // fp8 unit pairs (2pr, 2pr+1), highest first
    uint4 a[2];
    if (!zero) {
#pragma unroll
      for (int j = 0; j < 2; ++j)
        a[j] = *reinterpret_cast<const uint4*>(src + (sbase ^ (uint32_t)((2 * pr + j) << 4)));
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int u = 2 * pr + j;  // dims 16u .. 16u+15: block u / 4, 16-bit units 2(u%4), 2(u%4)+1
      uint8_t* blk = dst + (u >> 2) * CHUNK;
      uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
      if (!zero) widen16<OUT>(a[j], lo, hi);
      *reinterpret_cast<uint4*>(blk + (dbase ^ (uint32_t)((2 * (u & 3)) << 4))) = lo;
      *reinterpret_cast<uint4*>(blk + (dbase ^ (uint32_t)((2 * (u & 3) + 1) << 4))) = hi;
    }
  }
}

// Per-request values an item needs, loaded one item ahead.  Shared-prefix
// extend (SX): per-group values (rows r0 .. r1-1 of requests ga .. gb-1,
// `prefix` = the group's shared prefix length).
struct ItemRaw {
  int r0, r1, prefix, ga, gb;
};

// Tsh, r_lo, r_hi (SX): the shared prefix's key tiles, and the requests that
// hold the item's first and last rows.
struct Item {
  int b, g, i0, ntok[2], P, S, row0, kv_total, k_lo, k_hi, T, slot, Tsh, r_lo, r_hi;
};

template <bool SX>
__device__ __forceinline__ ItemRaw load_raw(const ExtendParams& p, int item) {
  ItemRaw r{0, 0, 0, 0, 0};
  if (item < p.num_items) {
    const int b = (int)p.div_req.div((uint32_t)item);
    if constexpr (SX) {
      r.ga = __ldg(p.group_indptr + b);
      r.gb = __ldg(p.group_indptr + b + 1);
      if (r.ga >= 0 && r.ga <= r.gb && r.gb <= p.batch) {
        r.r0 = __ldg(p.q_indptr + r.ga);
        r.r1 = __ldg(p.q_indptr + r.gb);
      } else {
        r.r0 = 0;
        r.r1 = -1;  // rejected by derive()
      }
      r.prefix = __ldg(p.group_shared + b);
    } else {
      r.r0 = __ldg(p.q_indptr + b);
      r.r1 = __ldg(p.q_indptr + b + 1);
      r.prefix = __ldg(p.prefix_lens + b);
    }
  }
  return r;
}

// A run of key tiles that the same rows may see through the same block
// table: the whole key range of a plain or prefix-pass item, or (SX) the
// group's shared prefix (req = -1, every row) or request req's own keys.
struct Seg {
  int req, k_lo, k_hi, kv_total, tiles;
};

// SX: request r's keys past the group's shared prefix (it.P) up to its last
// row in the item; none if it has no rows.
__device__ __forceinline__ Seg own_seg(const ExtendParams& p, const Item& it, int r) {
  Seg sg;
  sg.req = r;
  const int qs = __ldg(p.q_indptr + r), qe = __ldg(p.q_indptr + r + 1);
  const int pr = __ldg(p.prefix_lens + r);
  const int last = min(qe, it.row0 + it.i0 + it.ntok[0] + it.ntok[1]) - qs;  // r's rows in the item
  sg.k_lo = it.P;
  sg.k_hi = pr + last;
  sg.kv_total = pr + (qe - qs);
  sg.tiles = (qe > qs && sg.k_hi > sg.k_lo) ? (sg.k_hi - sg.k_lo + BN - 1) / BN : 0;
  return sg;
}

// The request of rows lo .. hi-1 (q_indptr order) that holds row t: the last
// one starting at or before t, so empty requests are passed over.
__device__ __forceinline__ int find_req(const int32_t* q_indptr, int lo, int hi, int t) {
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(q_indptr + mid) <= t) lo = mid;
    else hi = mid;
  }
  return lo;
}

// find_req by the whole warp (t the same in every lane): each round reads 32
// entries spread over the span at once and keeps the stretch between the last
// one at or before t and the next, so 256 requests take two rounds of one
// load each instead of eight dependent loads.
__device__ __forceinline__ int find_req_warp(const int32_t* q_indptr, int lo, int hi, int t) {
  const int lane = threadIdx.x & 31;
  while (hi - lo > 1) {
    const int step = (hi - lo + 31) >> 5;
    const int idx = lo + lane * step;
    const int v = idx < hi ? __ldg(q_indptr + idx) : INT_MAX;
    const unsigned m = __ballot_sync(0xFFFFFFFFu, v <= t);
    const int k = m ? 31 - __clz(m) : 0;
    lo += k * step;
    hi = min(hi, lo + step);
  }
  return lo;
}

// The key tiles of an item walked in order, segment by segment; every role
// walks them the same way.
struct SegIter {
  Seg sg;
  int st;  // tile within the segment
  int rr;  // SX: the next request whose own keys follow
};

template <bool SX>
__device__ __forceinline__ void seg_next_nonempty(const ExtendParams& p, const Item& it, SegIter& si) {
  if constexpr (SX) {
    while (si.st >= si.sg.tiles && si.rr <= it.r_hi) {
      si.sg = own_seg(p, it, si.rr++);
      si.st = 0;
    }
  }
}

template <bool SX>
__device__ __forceinline__ void seg_begin(const ExtendParams& p, const Item& it, SegIter& si) {
  if constexpr (!SX) return;  // a plain or prefix-pass item is one run: tile kt at k_lo + kt * BN
  si.sg.req = -1;
  si.sg.k_lo = it.k_lo;
  si.sg.k_hi = it.k_hi;
  si.sg.kv_total = it.kv_total;
  si.sg.tiles = SX ? it.Tsh : it.T;
  si.st = 0;
  si.rr = it.r_lo;
  seg_next_nonempty<SX>(p, it, si);
}

template <bool SX>
__device__ __forceinline__ void seg_advance(const ExtendParams& p, const Item& it, SegIter& si) {
  if constexpr (SX) {
    ++si.st;
    seg_next_nonempty<SX>(p, it, si);
  }
}

// false: the item has no work (the same answer in every role): tile A holds no
// suffix rows, the request's rows are not a valid range of the call's rows,
// or, in the prefix pass, the group shares no prefix or none in this item's
// key chunk.  Rows beyond the max_suffix_len hint (or max_group_size in the
// prefix pass), and prefix keys beyond the last chunk, are not computed and
// are reported as a length error.  SX: the item is a pair of tiles of the
// group's rows (requests packed back to back); a group whose request range or
// rows are not valid, or a request in the item whose prefix is shorter than
// the group's shared prefix or whose keys do not fit its block table, is not
// computed and is reported as a length error.
template <bool PP, bool SX>
__device__ __forceinline__ bool derive(const ExtendParams& p, int item, const ItemRaw& r, Item& it) {
  const uint32_t rest = p.div_pairs.div((uint32_t)item);
  int pair = item - (int)(rest * p.div_pairs.d);
  int kc = 0;  // prefix pass: the item's key chunk
  if constexpr (PP) {
    kc = pair % p.kchunks;
    pair /= p.kchunks;
  }
  it.b = (int)p.div_hkv.div(rest);
  it.g = (int)(rest - (uint32_t)it.b * p.div_hkv.d);
  const int TOK = p.tok;
  it.row0 = r.r0;
  it.S = r.r1 - r.r0;
  if constexpr (!PP) {
    // the output rows written below must lie inside the call's rows
    if (r.r0 < 0 || it.S < 0 || r.r1 > p.total_rows) {
      set_err(p.err, 3);
      return false;
    }
  }
  it.Tsh = 0;
  it.r_lo = 0;
  it.r_hi = -1;
  it.i0 = 2 * pair * TOK;  // first token of tile A; tile B follows it
  if (it.i0 >= it.S) return false;
  if ((pair + 1) * p.kchunks == (int)p.div_pairs.d && it.i0 + 2 * TOK < it.S) set_err(p.err, 3);
  it.ntok[0] = min(TOK, it.S - it.i0);
  it.ntok[1] = max(0, min(TOK, it.S - it.i0 - TOK));
  it.P = r.prefix;
  const int cap = p.max_blocks << p.bs_shift;
  if constexpr (SX) {
    it.P = (max(it.P, 0) >> p.bs_shift) << p.bs_shift;  // only whole blocks are shared
    if (it.P > cap) {
      set_err(p.err, 3);
      return false;
    }
    it.slot = 0;
    it.k_lo = 0;
    it.k_hi = it.P;
    it.kv_total = it.P;
    it.Tsh = (it.P + BN - 1) / BN;
    const int t_first = it.row0 + it.i0, t_last = t_first + it.ntok[0] + it.ntok[1] - 1;
    it.r_lo = find_req_warp(p.q_indptr, r.ga, r.gb, t_first);
    it.r_hi = find_req_warp(p.q_indptr, it.r_lo, r.gb, t_last);
    int T = it.Tsh;
    for (int rq = it.r_lo; rq <= it.r_hi; ++rq) {
      const Seg sg = own_seg(p, it, rq);
      const int pr = __ldg(p.prefix_lens + rq);
      if (sg.kv_total > pr && (pr < it.P || sg.kv_total > cap)) {  // a request with rows
        set_err(p.err, 3);
        return false;
      }
      T += sg.tiles;
    }
    it.T = T;
    return T > 0;
  }
  if constexpr (PP) {
    // the group's first member supplies the block table and must exist
    if (it.row0 < 0 || it.row0 >= p.total_rows) {
      set_err(p.err, 3);
      return false;
    }
    it.P = (it.P >> p.bs_shift) << p.bs_shift;  // only whole blocks are shared
    it.k_lo = kc * p.kchunk_keys;
    if (it.P <= 0 || it.k_lo >= it.P) return false;
    if (kc == p.kchunks - 1 && it.k_lo + p.kchunk_keys < it.P) set_err(p.err, 3);
    it.kv_total = min(it.P, it.k_lo + p.kchunk_keys);  // this chunk's keys end here
    it.k_hi = it.kv_total;
    it.slot = kc;
  } else {
    it.k_lo = 0;
    it.slot = 0;
    it.kv_total = it.P + it.S;
    it.k_hi = it.P + it.i0 + it.ntok[0] + it.ntok[1];  // keys the pair needs
  }
  if (it.P < 0 || it.kv_total > cap) {
    set_err(p.err, 3);
    it.kv_total = min(max(it.kv_total, 0), cap);
    it.k_hi = min(max(it.k_hi, 1), max(cap, 1));
    if (it.k_hi <= it.k_lo) return false;  // every item that runs has a key tile
  }
  it.T = (it.k_hi - it.k_lo + BN - 1) / BN;
  return true;
}

// HD: head dim (64 or 128); CT: cache dtype (f16, bf16 or e4m3); AT: the
// activation dtype of q and out (equal to CT for 16-bit caches); PP: the
// prefix pass; SX: shared-prefix extend.
template <int HD, int CT, int AT, bool PP, bool SX>
__global__ void __launch_bounds__(NTHREADS, 1)
extend_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
              const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap omap,
              const ExtendParams p, const ExtendPartialParams pp) {
  using C = ExtCfg<HD, CT, AT>;
  constexpr int NST = C::NST;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEMSLOT);
  const uint32_t s_base = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return smem_u32(&bars[i]); };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int TOK = p.tok;
  const int item0 = blockIdx.x, stride = gridDim.x;

  if (threadIdx.x == 0) {
    prefetch_tensormap(&kmap);
    prefetch_tensormap(&vmap);
    prefetch_tensormap(&qmap);
    for (int i = 0; i < NST; ++i) {
      mbar_init(bar(C::B_KFULL + i), 1);
      mbar_init(bar(C::B_VFULL + i), 1);
      mbar_init(bar(C::B_KCONV + i), NCONV / 32);
      mbar_init(bar(C::B_VCONV + i), NCONV / 32);
      mbar_init(bar(C::B_KFREE + i), 1);
      mbar_init(bar(C::B_VFREE + i), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(bar(C::B_SDONE + x), 1);
      mbar_init(bar(C::B_PFULL + x), 4);
      mbar_init(bar(C::B_QFULL + 2 * x), 1);
      mbar_init(bar(C::B_QFULL + 2 * x + 1), 1);
      mbar_init(bar(C::B_QCONV + 2 * x), NCONV / 32);
      mbar_init(bar(C::B_QCONV + 2 * x + 1), NCONV / 32);
      mbar_init(bar(C::B_QFREE + x), 1);
      mbar_init(bar(C::B_OFREE + x), 4);
      mbar_init(bar(C::B_EST + x), 4);
      mbar_init(bar(C::B_EFREE + x), 1);
    }
    mbar_init(bar(C::B_ODONE), 1);
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  // registers: launched with 128 per thread (512 x 128); the two softmax
  // warpgroups (warps 4-7 and 8-11) raise their budget to 184, the producer /
  // MMA warpgroup (0-3) lowers its to 96 and the converters (12-15) to 48
  // (fp8 caches, whose converters widen K and V: 88 and 56); the shares add up
  // to the launch budget, 4 x 128.
  constexpr int kRegsProd = C::FP8 ? 88 : 96, kRegsConv = C::FP8 ? 56 : 48;
  static_assert(2 * 184 + kRegsProd + kRegsConv == 4 * 128,
                "register split must equal the launch budget");
  if (warp >= 4 && warp < 12) {
    regs_inc<184>();
    // ------------------------------------------------------------ softmax of tile x
    const int x = warp >= 8 ? 1 : 0;
    const int qw = warp & 3;
    const int r = qw * 32 + lane;
    const int rtok = r / G, rhead = r - rtok * G;  // this row's token in the tile and head in the group
    const uint32_t lane_addr = (uint32_t)(qw * 32) << 16;
    const uint32_t srow = tmem + lane_addr + tm_s(x);
    const uint32_t orow = tmem + lane_addr + tm_o<HD>(x);
    int n = 0, js = 0;
    ItemRaw nxt_raw = load_raw<SX>(p, item0);
    for (int item = item0; ok && item < p.num_items; item += stride) {
      const ItemRaw raw = nxt_raw;
      nxt_raw = load_raw<SX>(p, item + stride);
      Item it;
      if (!derive<PP, SX>(p, item, raw, it)) continue;
      const int i0x = it.i0 + x * TOK;  // first token of this tile
      // a row's last visible key is kdiag + its token (prefix pass: the chunk's
      // last key for all)
      const int kdiag = PP ? it.kv_total - 1 : it.P + i0x;
      // SX: this row's request and its last visible key (rows past the
      // group's end see nothing)
      int row_req = -2, row_lim = -1;
      if constexpr (SX) {
        if (rtok < it.ntok[x]) {
          const int tg = it.row0 + i0x + rtok;
          row_req = find_req(p.q_indptr, it.r_lo, it.r_hi + 1, tg);
          row_lim = __ldg(p.prefix_lens + row_req) + (tg - __ldg(p.q_indptr + row_req));
        }
      }
      SegIter si;
      seg_begin<SX>(p, it, si);
      float m_run = -INFINITY, l_run = 0.f;
      for (int kt = 0; kt < it.T; ++kt, ++n, seg_advance<SX>(p, it, si)) {
        if (!mbar_wait(bar(C::B_SDONE + x), n & 1)) { ok = false; break; }
        tc_fence_after();
        const int key0 = SX ? si.sg.k_lo + si.st * BN : it.k_lo + kt * BN;
        // keys key0 .. key0 + nvis of the tile are visible to this row
        int nvis;
        bool masked;
        if constexpr (SX) {
          // the shared prefix: keys before its end, up to the row's limit;
          // a request's own keys: only that request's rows, causally
          const int lim = si.sg.req < 0 ? min(it.P - 1, row_lim) : (row_req == si.sg.req ? row_lim : -1);
          nvis = lim - key0;
          masked = __any_sync(0xFFFFFFFFu, nvis < BN - 1);
        } else {
          nvis = kdiag + (PP ? 0 : rtok) - key0;
          masked = key0 + BN - 1 > kdiag;
        }
        // Scores past a row's limit become -inf.  Plain 16-bit kernels mask the
        // loaded row in registers (~130 cycles); the fp8, prefix-pass and
        // shared-prefix kernels, whose hot loops already fill the instruction
        // cache, rewrite the tile in TMEM with a short rolled loop instead
        // (~600 cycles, but 4 KB less code: the unrolled register form cost
        // them 3-7 %).  Either runs on one or two key tiles per item.
        constexpr bool kRegMask = !SX && !PP && !C::FP8;
        const uint32_t ninf = __float_as_uint(-INFINITY);
        if (!kRegMask && masked) {
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
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
        // the whole S row: four 32-column loads, one wait
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(srow + c * 32, sr[c]);
        tmem_wait_ld();
        if (kRegMask && masked) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int q = 0; q < 32; ++q) sr[c][q] = (c * 32 + q > nvis) ? ninf : sr[c][q];
        }
        // row max: three-input max over 8 independent accumulators
        float mx[8];
#pragma unroll
        for (int a = 0; a < 8; ++a) mx[a] = -INFINITY;
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int q = 0; q < 16; ++q)
            mx[q & 7] = fmax3(mx[q & 7], __uint_as_float(sr[c][2 * q]), __uint_as_float(sr[c][2 * q + 1]));
        const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], mx[5]),
                               fmaxf(mx[6], mx[7])) * p.scale_log2;
        float m_new = m_run;
        if (mt > m_run + 8.f) m_new = mt;
        // SX: a row that has seen no key yet keeps m = -inf and takes 0 as
        // the exponent's base, so its masked scores give exact zeros
        const float m_base = (SX && m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = fast_exp2(m_run - m_base);
        const bool mine = (m_new != m_run);
        if (kt >= 1 && __any_sync(0xFFFFFFFFu, mine)) {
          // rescale O_x in TMEM (its last PV completed before S_x(n) did)
          const float f = mine ? alpha : 1.f;
#pragma unroll 1
          for (int c = 0; c < HD / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(orow + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * f);
            tmem_st32(orow + c * 32, o);
          }
        }
        m_run = m_new;
        // p = 2^(s*scale - m) as f16 pairs over the first 64 columns of S_x;
        // pairs of keys through the packed fp32 pipe
        float2 sm[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) sm[a] = make_float2(0.f, 0.f);
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
        const float2 nm2 = make_float2(-m_base, -m_base);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float2 xv = __ffma2_rn(
                make_float2(__uint_as_float(sr[c][2 * q]), __uint_as_float(sr[c][2 * q + 1])), sc2, nm2);
            const float2 pe = make_float2(fast_exp2(xv.x), fast_exp2(xv.y));
            sm[q & 3] = __fadd2_rn(sm[q & 3], pe);
            pk[q] = pack2<false>(pe.x, pe.y);
          }
          tmem_st16(srow + c * 16, pk);
        }
        const float sum = ((sm[0].x + sm[1].x) + (sm[2].x + sm[3].x)) +
                          ((sm[0].y + sm[1].y) + (sm[2].y + sm[3].y));
        l_run = l_run * alpha + sum;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_PFULL + x));
      }
      if (!ok) break;
      // ---- item epilogue: O_x out of TMEM (then it is free for the next
      // item), O / l -> out, LSE
      if (!mbar_wait(bar(C::B_ODONE), js & 1)) { ok = false; break; }
      tc_fence_after();
      // a whole tile of 16-bit output rows leaves through shared memory and
      // TMA stores (a tile with fewer rows, whose box would reach the next
      // request's rows, and the prefix pass's fp32 partials are stored by
      // each thread)
      const bool staged = out_tma_for<HD, CT, SX>() && !PP && p.out_tma && it.ntok[x] == TOK;
      const float osc = p.out_scale / l_run;
      if constexpr (PP) {
        // fp32 O / l straight from TMEM (the whole row before one wait), then
        // the LSE
        const int req = it.row0 + i0x + rtok;  // the group member of this row
        const bool valid = rtok < it.ntok[x] && req >= 0 && req < p.total_rows;
        const int64_t qrow = (int64_t)req * p.num_q_heads + it.g * G + rhead;
        float* dst = pp.o + qrow * pp.o_stride + it.slot * HD;
        {
          uint32_t o[HD / 32][32];
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) tmem_ld32(orow + c * 32, o[c]);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int c = 0; c < HD / 32; ++c) {
#pragma unroll
              for (int q = 0; q < 32; ++q) o[c][q] = __float_as_uint(__uint_as_float(o[c][q]) * osc);
#pragma unroll
              for (int q = 0; q < 4; ++q) st_global_v8(dst + c * 32 + 8 * q, &o[c][8 * q]);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_OFREE + x));
        if (valid) pp.lse[qrow * pp.lse_stride + it.slot] = m_run + log2f(l_run);
      } else {
        // O / l packed to 16-bit in registers; then O_x is free in TMEM.  The
        // whole row is loaded before one wait (the score registers are free
        // by now): one TMEM round trip instead of one per 32 columns
        uint32_t w[HD / 2];
        {
          uint32_t o[HD / 32][32];
#pragma unroll
          for (int c = 0; c < HD / 32; ++c) tmem_ld32(orow + c * 32, o[c]);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < HD / 32; ++c)
#pragma unroll
            for (int q = 0; q < 16; ++q)
              w[c * 16 + q] = pack2<AT == DT_BF16>(__uint_as_float(o[c][2 * q]) * osc,
                                                   __uint_as_float(o[c][2 * q + 1]) * osc);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_OFREE + x));
        if (staged) {
          // the rows go to shared memory in the layout of a Q tile (128-byte
          // rows, 128-byte swizzle, one block per 64 dims) and leave in TMA
          // stores: 128 coalesced boxes instead of 32 row-strided cache lines
          // per warp store, issued by warp 3.  Tile B writes after tile A's
          // store has read the buffer.
          if (x == 1 && !mbar_wait(bar(C::B_EFREE), js & 1)) { ok = false; break; }
          uint8_t* stg = smem + C::OFF_Q + ((2 * js + 1) % NQB) * C::T16;
#pragma unroll
          for (int c = 0; c < HD / 64; ++c)
#pragma unroll
            for (int u = 0; u < 8; ++u)
              *reinterpret_cast<uint4*>(stg + c * CHUNK + r * 128 + ((u ^ (r & 7)) << 4)) =
                  make_uint4(w[c * 32 + 4 * u], w[c * 32 + 4 * u + 1], w[c * 32 + 4 * u + 2],
                             w[c * 32 + 4 * u + 3]);
          fence_async_smem();
          if (p.lse_out && rtok < it.ntok[x]) {
            const int64_t qrow = (int64_t)(it.row0 + i0x + rtok) * p.num_q_heads + it.g * G + rhead;
            p.lse_out[qrow] = (m_run + log2f(l_run)) * kLn2f;
          }
        } else if (rtok < it.ntok[x]) {
          const int64_t qrow = (int64_t)(it.row0 + i0x + rtok) * p.num_q_heads + it.g * G + rhead;
          uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) + qrow * HD;
          if (p.out_32b) {
            // 32-byte stores: half the L1 requests of 16-byte ones for the
            // row-strided output
#pragma unroll
            for (int q = 0; q < HD / 16; ++q) st_global_v8(dst + 16 * q, &w[8 * q]);
          } else {
            uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
            for (int q = 0; q < HD / 8; ++q) d4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
          }
          if (p.lse_out) p.lse_out[qrow] = (m_run + log2f(l_run)) * kLn2f;
        }
      }
      // the tile's rows are staged (or it has none to stage): warp 3 takes
      // over.  Every warp arrives once per item, so that the phase counts items.
      if constexpr (out_tma_for<HD, CT, SX>()) {
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_EST + x));
      }
      ++js;
    }
  } else if (warp < 4) {
    regs_dec<kRegsProd>();
    if (warp == 0 || warp == 2) {
      // ------------------------------------------------------------ producers
      // warp 0: Q tiles and the K ring; warp 2: the V ring.  Block ids: lane l
      // holds sub-tile (32 w + l) of window w, the next window is fetched one
      // window ahead.
      const bool is_k = (warp == 0);
      const CUtensorMap* map = is_k ? &kmap : &vmap;
      // a K stage is free once S_B of its tile is done (S_A was issued before
      // it), a V stage once O_B += P_B V is
      const int full0 = is_k ? C::B_KFULL : C::B_VFULL, free0 = is_k ? C::B_KFREE : C::B_VFREE;
      // Q tile x of item j goes to buffer (2j + x) mod 3; the buffer was last
      // used by tile B of item j-2 (x = 0) or tile A of item j-1 (x = 1)
      const uint32_t qbytes = (uint32_t)(C::NCH * 128 * G * TOK);  // the boxes' bytes
      auto load_q = [&](const Item& it, int jq, int xq) -> bool {
        int good = 1;
        if (lane == 0) {
          const int prev = jq - 2 + xq;  // item whose last S_B frees the buffer
          if (prev >= 0 && !mbar_wait(bar(C::B_QFREE + (prev & 1)), (prev >> 1) & 1)) good = 0;
          // tile A's buffer is where item j-2 staged its output
          if (out_tma_for<HD, CT, SX>() && good && xq == 0 && jq >= 2 &&
              !mbar_wait(bar(C::B_EFREE + 1), (jq - 2) & 1))
            good = 0;
          if (good) {
            const uint32_t dst = s_base + C::OFF_Q + ((2 * jq + xq) % NQB) * C::T16;
            const uint32_t fb = bar(C::B_QFULL + 2 * xq + (jq & 1));
            mbar_arrive_expect_tx(fb, qbytes);
#pragma unroll
            for (int c = 0; c < C::NCH; ++c)
              tma_load_3d(dst + c * CHUNK, &qmap, fb, c * 64, it.g * G, it.row0 + it.i0 + xq * TOK);
          }
        }
        return __shfl_sync(0xFFFFFFFFu, good, 0) != 0;
      };
      int n = 0, j = 0;
      ItemRaw nxt_raw = load_raw<SX>(p, item0);
      for (int item = item0; ok && item < p.num_items; item += stride) {
        const ItemRaw raw = nxt_raw;
        nxt_raw = load_raw<SX>(p, item + stride);
        Item it;
        if (!derive<PP, SX>(p, item, raw, it)) continue;
        if (is_k && !load_q(it, j, 0)) { ok = false; break; }
        SegIter si;
        seg_begin<SX>(p, it, si);
        const int32_t* bt = p.block_tables;
        int sk_lo = 0, sk_hi = 0;  // the segment's keys
        auto fetch = [&](int wi) -> int {
          const int key0 = sk_lo + (wi * 32 + lane) * 16;  // sub-tile = 16 keys
          int page = -1;
          if (key0 < sk_hi) {
            const int blk = bt[key0 >> p.bs_shift];
            if (blk < 0 || blk >= p.num_blocks) set_err(p.err, 1);  // TMA zero-fills page -1
            else page = blk * p.num_kv_heads + it.g;
          }
          return page;
        };
        int win = 0, cur = -1, nxt = -1;
        for (int kt = 0; kt < it.T; ++kt, ++n, seg_advance<SX>(p, it, si)) {
          const int s = n % NST;
          const int st = SX ? si.st : kt;  // tile within the segment
          if (st == 0) {
            // a segment's table: the prefix pass reads the group's first
            // member's (row0 = its index); a shared prefix (SX) is read
            // through the table of the item's first request, whose blocks
            // for it are the group's
            const int breq = SX ? (si.sg.req < 0 ? it.r_lo : si.sg.req) : (PP ? it.row0 : it.b);
            bt = p.block_tables + (int64_t)breq * p.max_blocks;
            sk_lo = SX ? si.sg.k_lo : it.k_lo;
            sk_hi = SX ? si.sg.k_hi : it.k_hi;
            win = 0;
            cur = fetch(0);
            nxt = fetch(1);
          } else if ((st >> 2) > win) {  // 4 tiles x 8 sub-tiles per window
            cur = nxt;
            ++win;
            nxt = fetch(win + 1);
          }
          int pg[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) pg[q] = __shfl_sync(0xFFFFFFFFu, cur, (st & 3) * 8 + q);
          if (n >= NST && !mbar_wait(bar(free0 + s), (uint32_t)((n / NST - 1) & 1))) { ok = false; break; }
          if (lane == 0) {
            const uint32_t fb = bar(full0 + s);
            if constexpr (C::FP8) {
              // one box of 16 keys x head_dim codes per sub-tile
              const uint32_t dst = s_base + C::src8(!is_k, s);
              mbar_arrive_expect_tx(fb, C::T8);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int rip = (sk_lo + st * BN + 16 * q) & ((1 << p.bs_shift) - 1);
                tma_load_3d(dst + q * 16 * HD, map, fb, 0, rip, pg[q]);
              }
            } else {
              const uint32_t dst = s_base + (is_k ? C::OFF_K : C::OFF_V) + s * C::T16;
              mbar_arrive_expect_tx(fb, C::T16);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                const int rip = (sk_lo + st * BN + 16 * q) & ((1 << p.bs_shift) - 1);
#pragma unroll
                for (int c = 0; c < C::NCH; ++c)
                  tma_load_3d(dst + c * CHUNK + q * 2048, map, fb, c * 64, rip, pg[q]);
              }
            }
          }
          // Q of tile B once tile A of the previous item is done with its buffer
          if (is_k && kt == min(1, it.T - 1) && !load_q(it, j, 1)) { ok = false; break; }
        }
        ++j;
      }
    } else if (warp == 3) {
      if constexpr (out_tma_for<HD, CT, SX>()) {
      // ------------------------------------------------------------ output stores
      // Per item and tile: once the softmax warps have staged a whole tile of
      // 16-bit output rows in tile B's Q buffer, TMA-store it, wait until the
      // stores have read the buffer and release it (tile A first; tile B
      // stages only after tile A's store has read, and the Q load of tile A
      // two items on waits for tile B's release).  Waiting here keeps the
      // softmax warps off the TMA engine's queue.
      int js = 0;
      ItemRaw nxt_raw = load_raw<SX>(p, item0);
      for (int item = item0; ok && item < p.num_items; item += stride) {
        const ItemRaw raw = nxt_raw;
        nxt_raw = load_raw<SX>(p, item + stride);
        Item it;
        if (!derive<PP, SX>(p, item, raw, it)) continue;
        const uint32_t stg = s_base + C::OFF_Q + ((2 * js + 1) % NQB) * C::T16;
#pragma unroll 1
        for (int x = 0; x < 2 && ok; ++x) {
          const bool staged = !PP && p.out_tma && it.ntok[x] == TOK;
          // every item, staged or not: this warp stays in step with the barrier
          if (!mbar_wait(bar(C::B_EST + x), js & 1)) { ok = false; break; }
          if (staged) {
            if (lane == 0) {
#pragma unroll
              for (int c = 0; c < C::NCH; ++c)
                tma_store_3d(&omap, stg + c * CHUNK, c * 64, it.g * G, it.row0 + it.i0 + x * TOK);
              bulk_commit();
              bulk_wait_read_all();
            }
            __syncwarp();
          }
          if (lane == 0) mbar_arrive(bar(C::B_EFREE + x));
        }
        ++js;
      }
      // the stores complete before the CTA exits
      if (lane == 0) bulk_wait_all();
      }
    } else if (warp == 1) {
      // ------------------------------------------------------------ MMA issuer
      // The whole warp runs the loop (every operand is warp-uniform); one
      // elected lane issues the MMAs and commits.  Order per key tile n:
      // O_A += P_A(n-1) V(n-1), S_A(n), O_B += P_B(n-1) V(n-1), S_B(n): each
      // S_x(n) overwrites P_x(n-1) after the PV that reads it.
      constexpr uint32_t qk_fmt = C::QK_BF16 ? 1u : 0u;
      constexpr uint32_t idesc_qk = umma_idesc_f16(qk_fmt, qk_fmt, BM, BN);
      constexpr uint32_t idesc_pv = umma_idesc_f16(0u, 0u, BM, HD) | (1u << 16);
      // K is ready for the MMA once loaded, or, for fp8 codes, once widened;
      // Q once loaded, or once converted to f16
      const int kready0 = C::FP8 ? C::B_KCONV : C::B_KFULL;
      const int qready0 = C::QCVT ? C::B_QCONV : C::B_QFULL;
      // O_x += P_x(u) V(u); `first`: the first key tile of item ju, which
      // overwrites O_x once the previous item's O_x has been read out
      auto issue_pv = [&](int xx, int u, bool first, int ju) -> bool {
        if (!mbar_wait(bar(C::B_PFULL + xx), u & 1)) return false;
        if (xx == 0 && !mbar_wait(bar(C::B_VCONV + u % NST), (u / NST) & 1)) return false;
        if (first && ju >= 1 && !mbar_wait(bar(C::B_OFREE + xx), (ju - 1) & 1)) return false;
        tc_fence_after();
        const uint64_t vdesc = umma_desc_sw128_mn(s_base + C::OFF_V + (u % NST) * C::T16, CHUNK);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_f16_ts(tmem + tm_o<HD>(xx), tmem + tm_s(xx) + kk * 8, vdesc + (uint64_t)(kk * 2048 >> 4),
                        idesc_pv, (!first || kk > 0) ? 1u : 0u);
        }
        __syncwarp();
        return true;
      };
      auto issue_qk = [&](int xx, int nn, int qbuf) {
        const uint64_t kdesc = umma_desc_sw128(s_base + C::OFF_K + (nn % NST) * C::T16);
        const uint64_t qdesc = umma_desc_sw128(s_base + C::OFF_Q + qbuf * C::T16);
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint64_t off = (uint64_t)(((kk >> 2) * CHUNK + (kk & 3) * 32) >> 4);
            umma_f16(tmem + tm_s(xx), qdesc + off, kdesc + off, idesc_qk, kk > 0 ? 1u : 0u);
          }
          umma_commit(bar(C::B_SDONE + xx));
        }
        __syncwarp();
      };
      auto commit = [&](int b) {
        if (elect_one()) umma_commit(bar(b));
        __syncwarp();
      };
      int n = 0, j = 0;
      bool have_prev = false, prev_first = false, prev_last = false;
      int prev_n = 0, prev_j = 0;
      ItemRaw nxt_raw = load_raw<SX>(p, item0);
      for (int item = item0; ok && item < p.num_items; item += stride) {
        const ItemRaw raw = nxt_raw;
        nxt_raw = load_raw<SX>(p, item + stride);
        Item it;
        if (!derive<PP, SX>(p, item, raw, it)) continue;
        const int qa = (2 * j) % NQB, qb = (2 * j + 1) % NQB;
        for (int kt = 0; kt < it.T; ++kt, ++n) {
          if constexpr (C::FP8 && HD == 128) {
            // the same order as a rolled loop over the two tiles: half the
            // issue code, which the fp8 d128 kernel (in-place widening, Q
            // conversion) needs more than the unrolled form's shorter path
            // (878 against 942 us; bf16 would take 827 against 785, fp8 d64
            // 693 against 679)
#pragma unroll 1
            for (int xx = 0; xx < 2; ++xx) {
              if (have_prev) {
                if (!issue_pv(xx, prev_n, prev_first, prev_j)) { ok = false; break; }
                if (xx == 1) {
                  commit(C::B_VFREE + prev_n % NST);
                  if (prev_last) commit(C::B_ODONE);
                }
              }
              if (xx == 0 && !mbar_wait(bar(kready0 + n % NST), (n / NST) & 1)) { ok = false; break; }
              if (kt == 0 && !mbar_wait(bar(qready0 + 2 * xx + (j & 1)), (j >> 1) & 1)) { ok = false; break; }
              tc_fence_after();
              issue_qk(xx, n, xx ? qb : qa);
            }
            if (!ok) break;
          } else {
            if (have_prev && !issue_pv(0, prev_n, prev_first, prev_j)) { ok = false; break; }
            if (!mbar_wait(bar(kready0 + n % NST), (n / NST) & 1)) { ok = false; break; }
            if (kt == 0 && !mbar_wait(bar(qready0 + (j & 1)), (j >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            issue_qk(0, n, qa);
            if (have_prev) {
              if (!issue_pv(1, prev_n, prev_first, prev_j)) { ok = false; break; }
              commit(C::B_VFREE + prev_n % NST);
              if (prev_last) commit(C::B_ODONE);
            }
            if (kt == 0 && !mbar_wait(bar(qready0 + 2 + (j & 1)), (j >> 1) & 1)) { ok = false; break; }
            tc_fence_after();
            issue_qk(1, n, qb);
          }
          commit(C::B_KFREE + n % NST);
          if (kt == it.T - 1) commit(C::B_QFREE + (j & 1));
          have_prev = true;
          prev_n = n;
          prev_first = (kt == 0);
          prev_last = (kt == it.T - 1);
          prev_j = j;
        }
        ++j;
      }
      if (ok && have_prev) {
        ok = issue_pv(0, prev_n, prev_first, prev_j) && issue_pv(1, prev_n, prev_first, prev_j);
        if (ok) {
          commit(C::B_VFREE + prev_n % NST);
          commit(C::B_ODONE);
        }
      }
    }
  } else {
    regs_dec<kRegsConv>();
    {
      // ------------------------------------------------------------ converters (12-15)
      // Per key tile: fp8 K rows are widened to the activation dtype (then the
      // S MMA may read the tile); V becomes f16 (bf16 or fp8 sources) and keys
      // at or past the sequence end become zeros (then the PV MMA may read the
      // tile).  fp8 tiles: thread t owns key row t.
      const int t = threadIdx.x - 384;  // 0..127
      int n = 0, j = 0;
      // bf16 Q tile x of item j -> f16 in place (fp8 caches: S runs in f16)
      auto conv_q = [&](int xq) -> bool {
        if (!mbar_wait(bar(C::B_QFULL + 2 * xq + (j & 1)), (j >> 1) & 1)) return false;
        conv_q_tile<HD>(smem + C::OFF_Q + ((2 * j + xq) % NQB) * C::T16, t);
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_QCONV + 2 * xq + (j & 1)));
        return true;
      };
      ItemRaw nxt_raw = load_raw<SX>(p, item0);
      for (int item = item0; ok && item < p.num_items; item += stride) {
        const ItemRaw raw = nxt_raw;
        nxt_raw = load_raw<SX>(p, item + stride);
        Item it;
        if (!derive<PP, SX>(p, item, raw, it)) continue;
        SegIter si;
        seg_begin<SX>(p, it, si);
        for (int kt = 0; kt < it.T; ++kt, ++n, seg_advance<SX>(p, it, si)) {
          const int s = n % NST;
          const uint32_t ph = (uint32_t)((n / NST) & 1);
          // order of the first key tile: Q_A, K, Q_B, V (the MMA's order of use;
          // the producer loads Q_B after the first K tile)
          if constexpr (C::QCVT) {
            if (kt == 0 && !conv_q(0)) { ok = false; break; }
          }
          if constexpr (C::FP8) {
            if (!mbar_wait(bar(C::B_KFULL + s), ph)) { ok = false; break; }
            widen_row<HD, DT_F16>(smem + C::src8(false, s), smem + C::OFF_K + s * C::T16, t, false);
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_KCONV + s));
          }
          if constexpr (C::QCVT) {
            if (kt == 0 && !conv_q(1)) { ok = false; break; }
          }
          if (!mbar_wait(bar(C::B_VFULL + s), ph)) { ok = false; break; }
          // keys at or past the segment's end are zeroed (a shared prefix's
          // last tile reaches into one member's own keys, which no row of the
          // segment sees)
          const int kbase = SX ? si.sg.k_lo + si.st * BN : it.k_lo + kt * BN;
          const int kv_end = SX ? si.sg.kv_total : it.kv_total;
          const bool zero = kbase + t >= kv_end;
          uint8_t* vt = smem + C::OFF_V + s * C::T16;
          if constexpr (C::FP8) {
            widen_row<HD, DT_F16>(smem + C::src8(true, s), vt, t, zero);
            fence_async_smem();
          } else if (kbase + BN > kv_end) {  // tail tile: zero the keys past the end
            conv_tile16<HD, CT == DT_BF16, true>(vt, t, kbase, kv_end);
            fence_async_smem();
          } else if constexpr (CT == DT_BF16) {
            conv_tile16<HD, true, false>(vt, t, kbase, kv_end);
            fence_async_smem();
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(C::B_VCONV + s));
        }
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
  if (head_dim != 64 && head_dim != 128) return false;
  if (!(act_dt == DT_F16 || act_dt == DT_BF16)) return false;
  if (!(cache_dt == act_dt || cache_dt == DT_E4M3)) return false;
  return group >= 1 && group <= BM;
}

namespace {

template <int HD, int CT, int AT, bool PP, bool SX>
cudaError_t launch_extend_t(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                            const CUtensorMap& omap, const ExtendParams& p,
                            const ExtendPartialParams& pp, cudaStream_t stream) {
  auto k = extend_kernel<HD, CT, AT, PP, SX>;
  constexpr int smem = ExtCfg<HD, CT, AT>::SMEM;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  k<<<dim3(p.num_ctas), NTHREADS, smem, stream>>>(kmap, vmap, qmap, omap, p, pp);
  return cudaGetLastError();
}

template <bool PP, bool SX>
cudaError_t launch_extend_any(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                              const CUtensorMap& omap, const ExtendParams& p,
                              const ExtendPartialParams& pp, int head_dim, int cache_dt, int act_dt,
                              cudaStream_t stream) {
  // K bf16 with V widened to f16 beforehand is checked as a bf16 cache
  const int checked_dt = cache_dt == DT_BF16_V16 ? DT_BF16 : cache_dt;
  if (!extend_supported(head_dim, checked_dt, act_dt, p.group)) return cudaErrorInvalidValue;
  if (p.num_items <= 0 || p.num_ctas <= 0 || p.tok != BM / p.group) return cudaErrorInvalidValue;
#define PKV_EXT(HD, CT, AT)                                    \
  if (head_dim == HD && cache_dt == CT && act_dt == AT)        \
    return launch_extend_t<HD, CT, AT, PP, SX>(kmap, vmap, qmap, omap, p, pp, stream);
  if constexpr (!PP) {
    PKV_EXT(128, DT_BF16_V16, DT_BF16)
    PKV_EXT(64, DT_BF16_V16, DT_BF16)
  }
  PKV_EXT(128, DT_F16, DT_F16)
  PKV_EXT(128, DT_BF16, DT_BF16)
  PKV_EXT(128, DT_E4M3, DT_F16)
  PKV_EXT(128, DT_E4M3, DT_BF16)
  PKV_EXT(64, DT_F16, DT_F16)
  PKV_EXT(64, DT_BF16, DT_BF16)
  PKV_EXT(64, DT_E4M3, DT_F16)
  PKV_EXT(64, DT_E4M3, DT_BF16)
#undef PKV_EXT
  return cudaErrorInvalidValue;
}

// Pages of a shared-prefix extend widened into 16-bit shadow pools with the
// cache's block ids, so that the extend kernel reads them without converting
// and its converter warps only zero the keys past a segment's end: a bf16
// cache's V pages to f16 (SRC = DT_BF16), or an fp8 cache's K pages to KOUT
// (the queries' type, so that S = Q K^T needs no query conversion) and V
// pages to f16 (SRC = DT_E4M3; every e4m3 value is exact in both).
// Request r (the k-th member of its group of n) widens its own blocks, from
// the group's shared prefix to its last key, and every n-th of the group's
// shared blocks from the k-th on (read through the group's first member's
// table), so a long shared prefix is spread over the members.  CTA (x, r)
// takes every gridDim.x-th block of r's list from the x-th.  bf16 -> f16
// rounds to nearest (+-inf beyond the f16 range) as the converter warps do.
template <int SRC, int OUT>
__device__ __forceinline__ void widen_block(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                            int in_vec) {
  // in_vec 16-byte input vectors: bf16 -> one f16 vector each, e4m3 -> two
  for (int u0 = threadIdx.x; u0 < in_vec; u0 += 8 * 256) {
    uint4 x[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (u0 + e * 256 < in_vec) x[e] = __ldg(src + u0 + e * 256);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int u = u0 + e * 256;
      if (u < in_vec) {
        if constexpr (SRC == DT_BF16) {
          x[e].x = to_f16x2<true>(x[e].x);
          x[e].y = to_f16x2<true>(x[e].y);
          x[e].z = to_f16x2<true>(x[e].z);
          x[e].w = to_f16x2<true>(x[e].w);
          dst[u] = x[e];
        } else {
          uint4 lo, hi;
          widen16<OUT>(x[e], lo, hi);
          dst[2 * u] = lo;
          dst[2 * u + 1] = hi;
        }
      }
    }
  }
}

template <int SRC, int KOUT>
__global__ void __launch_bounds__(256) widen_kernel(const uint4* __restrict__ k,
                                                    const uint4* __restrict__ v,
                                                    uint4* __restrict__ k16, uint4* __restrict__ v16,
                                                    const ExtendParams p, int num_groups,
                                                    int in_vec) {
  const int r = blockIdx.y;
  if (r < __ldg(p.group_indptr) || r >= __ldg(p.group_indptr + num_groups)) return;
  int lo = 0, hi = num_groups;  // r's group: the last g with group_indptr[g] <= r
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(p.group_indptr + mid) <= r) lo = mid;
    else hi = mid;
  }
  const int first = __ldg(p.group_indptr + lo);
  const int members = __ldg(p.group_indptr + lo + 1) - first, kk = r - first;
  const int total = __ldg(p.prefix_lens + r) + (__ldg(p.q_indptr + r + 1) - __ldg(p.q_indptr + r));
  const int nb = min(p.max_blocks, (max(total, 0) + (1 << p.bs_shift) - 1) >> p.bs_shift);
  const int ws = min(max(__ldg(p.group_shared + lo), 0) >> p.bs_shift, p.max_blocks);
  const int n_own = max(nb - ws, 0);
  const int n_shared = ws > kk ? (ws - kk + members - 1) / members : 0;
  const int out_vec = SRC == DT_BF16 ? in_vec : 2 * in_vec;
  for (int t = blockIdx.x; t < n_own + n_shared; t += gridDim.x) {
    const int row = t < n_own ? r : first;
    const int i = t < n_own ? ws + t : kk + (t - n_own) * members;
    const int blk = __ldg(p.block_tables + (int64_t)row * p.max_blocks + i);
    if (blk < 0 || blk >= p.num_blocks) continue;
    if constexpr (SRC == DT_E4M3)
      widen_block<SRC, KOUT>(k + (int64_t)blk * in_vec, k16 + (int64_t)blk * out_vec, in_vec);
    widen_block<SRC, DT_F16>(v + (int64_t)blk * in_vec, v16 + (int64_t)blk * out_vec, in_vec);
  }
}

// Plain extend: the pages each request reads (blocks 0 .. ceil((P + S) /
// block_size) - 1 of its table), widened once per block although requests
// may share blocks.  claims = [count][flag per block][list]: the claim pass
// gives thread (x, r, t) blocks 256 x + t, 256 (x + gridDim.x) + t, ... of
// request r; the first request to set a block's flag (zeroed before the pass)
// appends it to the list.  The widening pass then spreads the list over a
// grid of persistent CTAs, so that the blocks of a shared prefix, which the
// requests that start first win, do not queue up in those requests' CTAs.
__global__ void __launch_bounds__(256) claim_kernel(int* claims, const ExtendParams p) {
  const int r = blockIdx.y;
  const int total = __ldg(p.prefix_lens + r) + (__ldg(p.q_indptr + r + 1) - __ldg(p.q_indptr + r));
  const int nb = min(p.max_blocks, (max(total, 0) + (1 << p.bs_shift) - 1) >> p.bs_shift);
  // the grid is sized from the call's length hint; a request past it loops
  for (int base = blockIdx.x * 256; base < nb; base += gridDim.x * 256) {
    const int i = base + threadIdx.x;
    int blk = -1;
    if (i < nb) blk = __ldg(p.block_tables + (int64_t)r * p.max_blocks + i);
    const bool won = blk >= 0 && blk < p.num_blocks && atomicCAS(claims + 1 + blk, 0, 1) == 0;
    // one list slot reservation per warp
    const unsigned m = __ballot_sync(0xffffffffu, won);
    if (m != 0) {
      const int lane = threadIdx.x & 31, leader = __ffs(m) - 1;
      int slot = 0;
      if (lane == leader) slot = atomicAdd(claims, __popc(m));
      slot = __shfl_sync(0xffffffffu, slot, leader);
      if (won) claims[1 + p.num_blocks + slot + __popc(m & ((1u << lane) - 1))] = blk;
    }
  }
}

template <int SRC, int KOUT>
__global__ void __launch_bounds__(256) widen_list_kernel(const uint4* __restrict__ k,
                                                         const uint4* __restrict__ v,
                                                         uint4* __restrict__ k16,
                                                         uint4* __restrict__ v16,
                                                         const int* __restrict__ claims,
                                                         int num_blocks, int in_vec) {
  const int n = min(claims[0], num_blocks);
  const int* list = claims + 1 + num_blocks;
  const int out_vec = SRC == DT_BF16 ? in_vec : 2 * in_vec;
  for (int j = blockIdx.x; j < n; j += gridDim.x) {
    const int blk = list[j];
    if constexpr (SRC == DT_E4M3)
      widen_block<SRC, KOUT>(k + (int64_t)blk * in_vec, k16 + (int64_t)blk * out_vec, in_vec);
    widen_block<SRC, DT_F16>(v + (int64_t)blk * in_vec, v16 + (int64_t)blk * out_vec, in_vec);
  }
}

}  // namespace

cudaError_t launch_widen_claim(int cache_dt, int act_dt, const void* k_cache,
                               const void* v_cache, void* k16, void* v16, int* claims,
                               const ExtendParams& p, int head_dim, int block_size,
                               int max_total_len, int sm_count, cudaStream_t stream) {
  if (!v_cache || !v16 || !claims || p.batch <= 0 || p.num_blocks <= 0 || sm_count <= 0)
    return cudaErrorInvalidValue;
  if (cache_dt != DT_BF16 && (cache_dt != DT_E4M3 || !k_cache || !k16)) return cudaErrorInvalidValue;
  const int elem = cache_dt == DT_BF16 ? 2 : 1;
  const int in_vec = p.num_kv_heads * block_size * head_dim * elem / 16;
  const int max_nb = std::min(p.max_blocks, (std::max(max_total_len, 1) + block_size - 1) / block_size);
  dim3 grid((unsigned)((max_nb + 255) / 256), (unsigned)p.batch);
  if (grid.y > 65535) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(claims, 0, (size_t)(1 + p.num_blocks) * sizeof(int), stream);
  if (e != cudaSuccess) return e;
  claim_kernel<<<grid, 256, 0, stream>>>(claims, p);
  // 8 CTAs of 256 threads fill an SM
  const int ctas = std::min(8 * sm_count, p.num_blocks);
  const uint4* k = static_cast<const uint4*>(k_cache);
  const uint4* v = static_cast<const uint4*>(v_cache);
  uint4* k16v = static_cast<uint4*>(k16);
  uint4* v16v = static_cast<uint4*>(v16);
  if (cache_dt == DT_BF16)
    widen_list_kernel<DT_BF16, DT_F16><<<ctas, 256, 0, stream>>>(k, v, k16v, v16v, claims,
                                                                   p.num_blocks, in_vec);
  else if (act_dt == DT_BF16)
    widen_list_kernel<DT_E4M3, DT_BF16><<<ctas, 256, 0, stream>>>(k, v, k16v, v16v, claims,
                                                                    p.num_blocks, in_vec);
  else
    widen_list_kernel<DT_E4M3, DT_F16><<<ctas, 256, 0, stream>>>(k, v, k16v, v16v, claims,
                                                                   p.num_blocks, in_vec);
  return cudaGetLastError();
}

cudaError_t launch_widen(int cache_dt, int act_dt, const void* k_cache, const void* v_cache,
                         void* k16, void* v16, const ExtendParams& p, int num_groups, int head_dim,
                         int block_size, int max_total_len, cudaStream_t stream) {
  if (!v_cache || !v16 || !p.group_indptr || !p.group_shared || num_groups <= 0 || p.batch <= 0)
    return cudaErrorInvalidValue;
  if (cache_dt != DT_BF16 && (cache_dt != DT_E4M3 || !k_cache || !k16)) return cudaErrorInvalidValue;
  const int elem = cache_dt == DT_BF16 ? 2 : 1;
  const int in_vec = p.num_kv_heads * block_size * head_dim * elem / 16;
  // a request's list is at most its own blocks plus its share of the shared
  // ones, both bounded by its table; about 16 blocks per CTA at the hint's length
  const int max_nb = std::min(p.max_blocks, (std::max(max_total_len, 1) + block_size - 1) / block_size);
  dim3 grid((unsigned)std::max(1, std::min(8, (max_nb + 15) / 16)), (unsigned)p.batch);
  if (grid.y > 65535) return cudaErrorInvalidValue;
  const uint4* k = static_cast<const uint4*>(k_cache);
  const uint4* v = static_cast<const uint4*>(v_cache);
  uint4* k16v = static_cast<uint4*>(k16);
  uint4* v16v = static_cast<uint4*>(v16);
  if (cache_dt == DT_BF16)
    widen_kernel<DT_BF16, DT_F16><<<grid, 256, 0, stream>>>(k, v, k16v, v16v, p, num_groups, in_vec);
  else if (act_dt == DT_BF16)
    widen_kernel<DT_E4M3, DT_BF16><<<grid, 256, 0, stream>>>(k, v, k16v, v16v, p, num_groups, in_vec);
  else
    widen_kernel<DT_E4M3, DT_F16><<<grid, 256, 0, stream>>>(k, v, k16v, v16v, p, num_groups, in_vec);
  return cudaGetLastError();
}

cudaError_t launch_extend(const CUtensorMap& kmap, const CUtensorMap& vmap, const CUtensorMap& qmap,
                          const CUtensorMap& omap, const ExtendParams& p, int head_dim,
                          int cache_dt, int act_dt, cudaStream_t stream) {
  return launch_extend_any<false, false>(kmap, vmap, qmap, omap, p, ExtendPartialParams{},
                                         head_dim, cache_dt, act_dt, stream);
}

cudaError_t launch_extend_shared(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const CUtensorMap& qmap, const CUtensorMap& omap,
                                 const ExtendParams& p, int head_dim, int cache_dt, int act_dt,
                                 cudaStream_t stream) {
  if (!p.group_indptr || !p.group_shared) return cudaErrorInvalidValue;
  return launch_extend_any<false, true>(kmap, vmap, qmap, omap, p, ExtendPartialParams{},
                                        head_dim, cache_dt, act_dt, stream);
}

cudaError_t launch_extend_prefix_pass(const CUtensorMap& kmap, const CUtensorMap& vmap,
                                      const CUtensorMap& qmap, const ExtendParams& p,
                                      const ExtendPartialParams& pp, int head_dim, int cache_dt,
                                      int act_dt, cudaStream_t stream) {
  if (!pp.o || !pp.lse || p.out_tma) return cudaErrorInvalidValue;
  // the partials are stored by each thread: the output map is not read
  return launch_extend_any<true, false>(kmap, vmap, qmap, qmap, p, pp, head_dim, cache_dt, act_dt,
                                        stream);
}

}  // namespace pkv
