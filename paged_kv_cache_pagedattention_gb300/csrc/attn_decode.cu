// PagedAttention decode on tensor cores.
//
// decode_mma_kernel: one CTA handles (request, KV head, head group of <= 8 query
// heads, partition of the context).  [NOTES] "Decode": the single new query token
// of a request reads every cached K/V of that request; [LINEAGE] "PagedAttention":
// K/V are read through the block table; the partitions' partial softmax states are
// merged afterwards by the rescale-and-add rule of [AGENTIC] "Online softmax".
//
// shared_prefix_kernel: one CTA handles (group of sequences whose block tables
// share leading entries, KV head, head group, partition of the shared prefix).
// [AGENTIC] "統一分頁 + 共用池": forked requests point at the same physical blocks;
// here each shared (block, head) tile is loaded once and one warp per member
// applies that member's query heads to it.  The members' private remainders run in
// decode_mma_kernel from their first private token, and the merge combines both.
// A member whose entry for a declared-shared block names another physical block
// (a stale or wrong declaration) gets that block as a stage of its own, read by its
// warp alone, so every member attends exactly its own blocks.
//
// Data movement.  Each (physical block, KV head) tile of K or V is contiguous in
// HBM (block_size x head_size elements).  TMA bulk-tensor copies land a tile in
// shared memory through a 4-D tensor map as head_size*elem/128 pieces of
// [block_size tokens][128 bytes] with the 128-byte swizzle, so eight consecutive
// tokens of one 16-byte column sit in eight different bank groups: the ldmatrix /
// 16-byte shared loads below are free of bank conflicts.  Copies complete on
// mbarrier transaction counts.  In decode_mma_kernel each warp owns a private ring
// and its lane 0 refills a stage as soon as the warp has consumed it; in
// shared_prefix_kernel a producer warp fills a CTA ring that all member warps read
// (full / empty mbarriers).  Whether a stage holds a valid block is recorded in
// shared memory by the issuing lane before its mbarrier arrive.
//
// Math.  The query heads that share a KV head are the N = 8 columns of a warp MMA
// m16n8k16 (grouped-query reuse: every K/V element loaded serves all of them):
//   S^T[token][head]   = K[token][:] . Q[head][:]       (M = 16 tokens, K = head dim)
//   O^T[dim][head]    += V^T[dim][token] . P^T[token][head]  (M = 16 dims, K = 16 tokens)
// P^T comes from the S^T accumulators through movmatrix (an in-register 8x8
// transpose).  The softmax runs on the accumulators in fp32 with a running max per
// head (log2 units), sums l from the same rounded P that feeds the MMA, and
// rescales O when the max grows.  FP8 tiles are converted to f16 exactly (cvt
// e4m3x2 / e5m2x2 -> f16x2) in registers; NVFP4 tiles (E2M1 codes + E4M3 block
// scales, copied whole with one 1-D bulk copy each) are converted code pair by code
// pair (cvt e2m1x2 -> f16x2) and multiplied by their block scale in f16, which is
// exact (at most 6 significant bits, magnitudes within f16's normal range).  The
// fp32 scales are folded into the score multiplier (k_scale) and the output
// (v_scale); q is scaled by a power of two per head so that it fits f16 exactly.
#include "pa_common.cuh"

namespace pa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int KVDT, int HEAD, int BS>
struct DecodeGeom {
  static constexpr bool kFp8 = is_fp8<KVDT>();
  static constexpr bool kFp4 = is_nvfp4<KVDT>();
  static constexpr bool kScaled = kFp8 || kFp4;  // f16 MMAs on converted codes
  static constexpr int kElemBytes = kFp8 ? 1 : 2;
  // code bytes of one token of one head; NVFP4 block scales follow the code rows
  static constexpr int kRowBytes = kFp4 ? HEAD / 2 : HEAD * kElemBytes;
  static constexpr int kCodeBytes = BS * kRowBytes;
  static constexpr int kTileBytes = kFp4 ? nvfp4_tile_bytes(BS, HEAD) : kCodeBytes;
  static constexpr int kMTiles = BS / 16;
  static constexpr int kKSteps = HEAD / 16;
  static constexpr int kDTiles = HEAD / 16;
  // per-warp ring (decode).  NVFP4 decode is bound by instruction latency rather than
  // HBM: three stages keep four CTAs (16 warps) per SM within shared memory and the
  // 128-register cap; measured 1.065 -> 0.994 ms on the NVFP4 decode workload.
  // 16-bit tiles: two stages (3 CTAs per SM instead of 2): Llama decode 95.9 -> 92.8
  // us, agentic span 0.384 -> 0.373 ms; FP8 keeps three, four for 2 KB tiles (block 16:
  // the CTA stays at 48 -> 64 KB, three per SM; FP8 mixed step 1.468 -> 1.454 ms).
  static constexpr int kStages = kFp4 ? 3 : kTileBytes <= 4096 ? (kFp8 ? (kTileBytes <= 2048 ? 4 : 3) : 2) : 2;
  static constexpr int kSharedStages = kTileBytes <= 4096 ? 6 : 4;       // CTA ring (shared prefix)
  static_assert(kFp4 ? HEAD == 128 : kRowBytes % 128 == 0, "token rows must be whole 128-byte rows");
  static_assert(kTileBytes % 16 == 0, "tiles are whole 16-byte pieces");
  // byte offset of 16-byte chunk `chunk` of token `tok` inside a tile
  static __device__ __forceinline__ uint32_t off(int tok, int chunk) {
    return static_cast<uint32_t>((chunk >> 3) * BS * 128) + swz128(tok, chunk & 7);
  }
};

// Per-warp attention state for one query row and its <= 8 heads (columns 2qq, 2qq+1
// of the accumulators belong to this thread: heads A and B).
template <int HEAD>
struct WarpState {
  float acc[HEAD / 16][4];
  float mA, mB, lA, lB;
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int i = 0; i < HEAD / 16; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    mA = mB = -INFINITY;
    lA = lB = 0.f;
  }
};

// B-operand fragments of the query (k = head dim, n = query head of the group) and
// the score multipliers (log2 units) of this thread's accumulator columns.
template <int QDT, int KVDT, int HEAD>
__device__ __forceinline__ void load_query(const AttnParams& p, long long row, int h0, int nh,
                                           uint32_t (&qb)[HEAD / 16][2], float& cA, float& cB) {
  using QE = Elem<QDT>;
  constexpr int KS = HEAD / 16;
  const int lane = threadIdx.x & 31;
  const int qn = lane >> 2, qq = lane & 3;
  const float base_c = p.scale * kLog2e;
  const typename QE::T* qrow =
      reinterpret_cast<const typename QE::T*>(p.q) + (row * p.num_q_heads + h0 + qn) * HEAD;
  if constexpr (!is_scaled<KVDT>()) {
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(qrow);
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[ks][0] = qn < nh ? qw[8 * ks + qq] : 0u;
      qb[ks][1] = qn < nh ? qw[8 * ks + 4 + qq] : 0u;
    }
    cA = cB = base_c;
  } else {
    // k-step ks, B rows (2qq, 2qq+1) <-> dims 32qq + 4ks + {0,1}; rows (2qq+8, 2qq+9) <-> +{2,3}
    float amax = 0.f;
    float qv[KS][4];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qv[ks][e] = qn < nh ? QE::load(qrow + 32 * qq + 4 * ks + e) : 0.f;
        amax = fmaxf(amax, fabsf(qv[ks][e]));
      }
    amax = warp_max_xor(amax, 1, 2);
    int ex = 0;
    frexpf(amax, &ex);  // amax < 2^ex
    int sh = 15 - ex;   // |q| * 2^sh < 2^15, exact in f16
    sh = max(-100, min(100, sh));
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qb[ks][0] = pack2<PA_F16>(ldexpf(qv[ks][0], sh), ldexpf(qv[ks][1], sh));
      qb[ks][1] = pack2<PA_F16>(ldexpf(qv[ks][2], sh), ldexpf(qv[ks][3], sh));
    }
    const float my_c = ldexpf(base_c * p.k_scale[(h0 / p.group) * p.scale_stride], -sh);
    cA = __shfl_sync(0xffffffffu, my_c, 8 * qq);      // head 2qq lives in lanes 8qq..8qq+3
    cB = __shfl_sync(0xffffffffu, my_c, 8 * qq + 4);  // head 2qq+1
  }
}

// One block of block_size tokens (K tile at `tile`, V tile at `tile + tile_bytes`)
// folded into a warp's state; tokens lo .. rem-1 of the block are attended (lo > 0
// only in the block where a sliding window starts; the tokens before it are older
// cached tokens, finite, so only their scores are masked).
template <int QDT, int KVDT, int HEAD, int BS>
__device__ __forceinline__ void attend_block(const uint8_t* tile, int rem, int lo, const uint32_t (&qb)[HEAD / 16][2],
                                             float cA, float cB, WarpState<HEAD>& w) {
  using G = DecodeGeom<KVDT, HEAD, BS>;
  constexpr bool kFp8 = G::kFp8;
  constexpr bool kFp4 = G::kFp4;
  constexpr int MDT = G::kScaled ? PA_F16 : QDT;
  constexpr int TB = G::kTileBytes;
  const int lane = threadIdx.x & 31, qq = lane & 3;
  const uint32_t kbase = smem_u32(tile);
  const uint32_t vbase = kbase + TB;

  // ---- S^T = K Q^T
  float sc[G::kMTiles][4];
#pragma unroll
  for (int mt = 0; mt < G::kMTiles; ++mt) {
    float sc2[4] = {0.f, 0.f, 0.f, 0.f};  // second, independent accumulation chain
    sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
    if constexpr (kFp4) {
      // rows tA, tB; this thread's 32 dims 32qq .. 32qq+31 are 16 code bytes (k-step ks:
      // bytes 2ks, 2ks+1 = dims 32qq + 4ks + 0..3) and block scales 2qq (ks < 4), 2qq+1
      const int tA = 16 * mt + (lane >> 2), tB = tA + 8;
      const uint4 ka = *reinterpret_cast<const uint4*>(tile + tA * G::kRowBytes + 16 * qq);
      const uint4 kb = *reinterpret_cast<const uint4*>(tile + tB * G::kRowBytes + 16 * qq);
      const uint32_t sa = fp8x2_to_f16x2<PA_FP8_E4M3>(
          *reinterpret_cast<const uint16_t*>(tile + G::kCodeBytes + tA * (HEAD / 16) + 2 * qq));
      const uint32_t sb = fp8x2_to_f16x2<PA_FP8_E4M3>(
          *reinterpret_cast<const uint16_t*>(tile + G::kCodeBytes + tB * (HEAD / 16) + 2 * qq));
      const uint32_t sa0 = __byte_perm(sa, 0, 0x1010), sa1 = __byte_perm(sa, 0, 0x3232);
      const uint32_t sb0 = __byte_perm(sb, 0, 0x1010), sb1 = __byte_perm(sb, 0, 0x3232);
      const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w};
      const uint32_t wb[4] = {kb.x, kb.y, kb.z, kb.w};
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {  // word wi: bytes 4wi .. 4wi+3 = k-steps 2wi, 2wi+1
        uint32_t fa[4], fb[4];
        fp4x8_to_f16x2x4(wa[wi], fa);
        fp4x8_to_f16x2x4(wb[wi], fb);
        const uint32_t scA = wi < 2 ? sa0 : sa1, scB = wi < 2 ? sb0 : sb1;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ks = 2 * wi + h;
          const uint32_t a0 = hmul2_u32(fa[2 * h], scA), a2 = hmul2_u32(fa[2 * h + 1], scA);
          const uint32_t a1 = hmul2_u32(fb[2 * h], scB), a3 = hmul2_u32(fb[2 * h + 1], scB);
          if (h) mma_16816<PA_F16>(sc2, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
          else mma_16816<PA_F16>(sc[mt], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
        }
      }
    } else if constexpr (!kFp8) {
#pragma unroll
      for (int ks = 0; ks < G::kKSteps; ++ks) {
        const int tok = 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int chunk = 2 * ks + (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(kbase + G::off(tok, chunk), a0, a1, a2, a3);
        if (ks & 1) mma_16816<MDT>(sc2, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
        else mma_16816<MDT>(sc[mt], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
      }
    } else {
      const int tA = 16 * mt + (lane >> 2), tB = tA + 8;
      const uint4 ka0 = *reinterpret_cast<const uint4*>(tile + swz128(tA, 2 * qq));
      const uint4 ka1 = *reinterpret_cast<const uint4*>(tile + swz128(tA, 2 * qq + 1));
      const uint4 kb0 = *reinterpret_cast<const uint4*>(tile + swz128(tB, 2 * qq));
      const uint4 kb1 = *reinterpret_cast<const uint4*>(tile + swz128(tB, 2 * qq + 1));
      const uint32_t wa[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
      const uint32_t wb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
#pragma unroll
      for (int ks = 0; ks < G::kKSteps; ++ks) {
        uint32_t a0, a1, a2, a3;
        fp8x4_to_f16x2x2<KVDT>(wa[ks], a0, a2);
        fp8x4_to_f16x2x2<KVDT>(wb[ks], a1, a3);
        if (ks & 1) mma_16816<PA_F16>(sc2, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
        else mma_16816<PA_F16>(sc[mt], a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) sc[mt][e] += sc2[e];
  }

  // ---- online softmax on the accumulators (columns 2qq, 2qq+1 = heads A, B).
  // Scores stay raw here; the positive multipliers cA / cB (scale * log2 e, and
  // k_scale for FP8) are applied inside the exponent.  The running max m is kept in
  // scaled (log2) units and is only raised when a block's max exceeds it by more
  // than kRescaleSlack: until then P = 2^(s*c - m) <= 2^kRescaleSlack and O, l need
  // no rescale.  The final normalisation divides by l computed with the same m, so
  // the result is the same softmax.
  if (rem < BS || lo > 0) {  // tokens past the sequence end or before the window: -inf
#pragma unroll
    for (int mt = 0; mt < G::kMTiles; ++mt) {
      const int t0 = 16 * mt + (lane >> 2);
      if (t0 >= rem || t0 < lo) sc[mt][0] = sc[mt][1] = -INFINITY;
      if (t0 + 8 >= rem || t0 + 8 < lo) sc[mt][2] = sc[mt][3] = -INFINITY;
    }
  }
  float mxA = -INFINITY, mxB = -INFINITY;
#pragma unroll
  for (int mt = 0; mt < G::kMTiles; ++mt) {
    mxA = fmaxf(mxA, fmaxf(sc[mt][0], sc[mt][2]));
    mxB = fmaxf(mxB, fmaxf(sc[mt][1], sc[mt][3]));
  }
  mxA = warp_max_xor(mxA, 4, 16) * cA;
  mxB = warp_max_xor(mxB, 4, 16) * cB;
  if (__any_sync(0xffffffffu, mxA > w.mA + kRescaleSlack || mxB > w.mB + kRescaleSlack)) {
    const float nA = fmaxf(w.mA, mxA), nB = fmaxf(w.mB, mxB);
    const float alA = nA == -INFINITY ? 1.f : ex2_approx(w.mA - nA);
    const float alB = nB == -INFINITY ? 1.f : ex2_approx(w.mB - nB);
    w.mA = nA;
    w.mB = nB;
    w.lA *= alA;
    w.lB *= alB;
#pragma unroll
    for (int dt = 0; dt < G::kDTiles; ++dt) {
      w.acc[dt][0] *= alA;
      w.acc[dt][1] *= alB;
      w.acc[dt][2] *= alA;
      w.acc[dt][3] *= alB;
    }
  }
  const float uA = w.mA == -INFINITY ? 0.f : w.mA, uB = w.mB == -INFINITY ? 0.f : w.mB;
  uint32_t pb[G::kMTiles][2];
  float addA = 0.f, addB = 0.f;
#pragma unroll
  for (int mt = 0; mt < G::kMTiles; ++mt) {
    const uint32_t X = pack2<MDT>(ex2_approx(fmaf(sc[mt][0], cA, -uA)), ex2_approx(fmaf(sc[mt][1], cB, -uB)));
    const uint32_t Y = pack2<MDT>(ex2_approx(fmaf(sc[mt][2], cA, -uA)), ex2_approx(fmaf(sc[mt][3], cB, -uB)));
    const float2 fx = unpack2<MDT>(X), fy = unpack2<MDT>(Y);
    addA += fx.x + fy.x;
    addB += fx.y + fy.y;
    pb[mt][0] = movmatrix_trans(X);
    pb[mt][1] = movmatrix_trans(Y);
  }
  w.lA += addA;
  w.lB += addB;

  // ---- O^T += V^T P^T; V tokens past the valid ones are zeroed (their P is 0,
  // their bits arbitrary)
  const bool tail = rem < BS;
#pragma unroll
  for (int kt = 0; kt < G::kMTiles; ++kt) {
    if constexpr (kFp4) {
      // this thread owns dims 16*(lane>>2) .. +15 (one block-scale group) of tokens
      // 16kt + {2qq, 2qq+1, 2qq+8, 2qq+9}: 8 code bytes per token.  Odd quads read the
      // second token of each pair first, so that one load instruction touches rows
      // 0, 3, 4, 7 (or 1, 2, 5, 6) of eight: two 64-byte rows per 128-byte bank line.
      const int rr = lane >> 2;
      const uint8_t* vt = tile + TB;
      const int tk = 16 * kt + 2 * qq;
      const int odd = qq & 1;
      uint2 v0 = *reinterpret_cast<const uint2*>(vt + (tk + odd) * G::kRowBytes + 8 * rr);
      uint2 v1 = *reinterpret_cast<const uint2*>(vt + (tk + 1 - odd) * G::kRowBytes + 8 * rr);
      uint2 v2 = *reinterpret_cast<const uint2*>(vt + (tk + 8 + odd) * G::kRowBytes + 8 * rr);
      uint2 v3 = *reinterpret_cast<const uint2*>(vt + (tk + 9 - odd) * G::kRowBytes + 8 * rr);
      const uint8_t* vs = vt + G::kCodeBytes + rr;
      uint32_t s01 = vs[tk * (HEAD / 16)] | (static_cast<uint32_t>(vs[(tk + 1) * (HEAD / 16)]) << 8);
      uint32_t s89 = vs[(tk + 8) * (HEAD / 16)] | (static_cast<uint32_t>(vs[(tk + 9) * (HEAD / 16)]) << 8);
      if (tail) {  // tokens past the end: zero codes and zero scales
        if (tk + odd >= rem) v0 = make_uint2(0, 0);
        if (tk + 1 - odd >= rem) v1 = make_uint2(0, 0);
        if (tk + 8 + odd >= rem) v2 = make_uint2(0, 0);
        if (tk + 9 - odd >= rem) v3 = make_uint2(0, 0);
        if (tk >= rem) s01 &= 0xff00u;
        if (tk + 1 >= rem) s01 &= 0x00ffu;
        if (tk + 8 >= rem) s89 &= 0xff00u;
        if (tk + 9 >= rem) s89 &= 0x00ffu;
      }
      const uint32_t f01 = fp8x2_to_f16x2<PA_FP8_E4M3>(static_cast<uint16_t>(s01));  // (token tk, tk+1)
      const uint32_t f89 = fp8x2_to_f16x2<PA_FP8_E4M3>(static_cast<uint16_t>(s89));
      // (first-read, second-read) -> (token tk, token tk+1) halves
      const uint32_t sel_lo = odd ? 0x1054u : 0x5410u, sel_hi = odd ? 0x3276u : 0x7632u;
#pragma unroll
      for (int wi = 0; wi < 2; ++wi) {  // word wi of each token: bytes 4wi .. 4wi+3 = d-tiles 4wi ..
        uint32_t x0[4], y0[4], x1[4], y1[4];
        fp4x8_to_f16x2x4(wi ? v0.y : v0.x, x0);
        fp4x8_to_f16x2x4(wi ? v1.y : v1.x, y0);
        fp4x8_to_f16x2x4(wi ? v2.y : v2.x, x1);
        fp4x8_to_f16x2x4(wi ? v3.y : v3.x, y1);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t a0 = hmul2_u32(__byte_perm(x0[j], y0[j], sel_lo), f01);
          const uint32_t a1 = hmul2_u32(__byte_perm(x0[j], y0[j], sel_hi), f01);
          const uint32_t a2 = hmul2_u32(__byte_perm(x1[j], y1[j], sel_lo), f89);
          const uint32_t a3 = hmul2_u32(__byte_perm(x1[j], y1[j], sel_hi), f89);
          mma_16816<PA_F16>(w.acc[4 * wi + j], a0, a1, a2, a3, pb[kt][0], pb[kt][1]);
        }
      }
    } else if constexpr (!kFp8) {
      const int tk = 16 * kt + 2 * qq;  // tokens of this thread's A halves: tk, tk+1, tk+8, tk+9
      const uint32_t m01 = (tk < rem ? 0xffffu : 0u) | (tk + 1 < rem ? 0xffff0000u : 0u);
      const uint32_t m23 = (tk + 8 < rem ? 0xffffu : 0u) | (tk + 9 < rem ? 0xffff0000u : 0u);
#pragma unroll
      for (int dt = 0; dt < G::kDTiles; ++dt) {
        const int tok = 16 * kt + (lane & 7) + 8 * (lane >> 4);
        const int chunk = 2 * dt + ((lane >> 3) & 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_trans(vbase + G::off(tok, chunk), a0, a1, a2, a3);
        if (tail) {
          a0 &= m01;
          a1 &= m01;
          a2 &= m23;
          a3 &= m23;
        }
        mma_16816<MDT>(w.acc[dt], a0, a1, a2, a3, pb[kt][0], pb[kt][1]);
      }
    } else {
      // this thread owns dims 16*(lane>>2) .. +15 of tokens 16kt + {2qq, 2qq+1, 2qq+8, 2qq+9}
      const int rr = lane >> 2;
      const uint8_t* vt = tile + TB;
      const int tk = 16 * kt + 2 * qq;
      uint4 v[4];
      v[0] = *reinterpret_cast<const uint4*>(vt + swz128(tk, rr));
      v[1] = *reinterpret_cast<const uint4*>(vt + swz128(tk + 1, rr));
      v[2] = *reinterpret_cast<const uint4*>(vt + swz128(tk + 8, rr));
      v[3] = *reinterpret_cast<const uint4*>(vt + swz128(tk + 9, rr));
      if (tail) {
        if (tk >= rem) v[0] = make_uint4(0, 0, 0, 0);
        if (tk + 1 >= rem) v[1] = make_uint4(0, 0, 0, 0);
        if (tk + 8 >= rem) v[2] = make_uint4(0, 0, 0, 0);
        if (tk + 9 >= rem) v[3] = make_uint4(0, 0, 0, 0);
      }
      const uint32_t w0[4] = {v[0].x, v[0].y, v[0].z, v[0].w};
      const uint32_t w1[4] = {v[1].x, v[1].y, v[1].z, v[1].w};
      const uint32_t w2[4] = {v[2].x, v[2].y, v[2].z, v[2].w};
      const uint32_t w3[4] = {v[3].x, v[3].y, v[3].z, v[3].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // word k: dims 16rr + 4k .. +3 = d-tiles 2k, 2k+1
        // byte-interleave the token pairs: 16-bit halves = (token t, token t+1) of one dim
        uint32_t c01[4], c89[4];
        fp8x4_to_f16x2x2<KVDT>(__byte_perm(w0[k], w1[k], 0x5140), c01[0], c01[1]);
        fp8x4_to_f16x2x2<KVDT>(__byte_perm(w0[k], w1[k], 0x7362), c01[2], c01[3]);
        fp8x4_to_f16x2x2<KVDT>(__byte_perm(w2[k], w3[k], 0x5140), c89[0], c89[1]);
        fp8x4_to_f16x2x2<KVDT>(__byte_perm(w2[k], w3[k], 0x7362), c89[2], c89[3]);
        mma_16816<PA_F16>(w.acc[2 * k], c01[0], c01[1], c89[0], c89[1], pb[kt][0], pb[kt][1]);
        mma_16816<PA_F16>(w.acc[2 * k + 1], c01[2], c01[3], c89[2], c89[3], pb[kt][0], pb[kt][1]);
      }
    }
  }
}

// Output dimensions of accumulator elements 0/1 (dA) and 2/3 (dB) of d-tile dt.
template <bool kScaled>
__device__ __forceinline__ void acc_dims(int dt, int lane, int& dA, int& dB) {
  const int rr = lane >> 2;
  dA = kScaled ? 16 * rr + 2 * dt : 16 * dt + rr;
  dB = kScaled ? dA + 1 : dA + 8;
}

// Copies of the K and V tiles of (physical block phys, KV head kvh) into st and
// st + tile bytes, completing on `bar`: tensor-map copies landing as swizzled
// 128-byte pieces, or for NVFP4 one 1-D bulk copy per tile (read as laid out).
template <int KVDT, int HEAD, int BS>
__device__ __forceinline__ void load_kv_tiles(uint8_t* st, const AttnParams& p, const CUtensorMap* tmk,
                                              const CUtensorMap* tmv, int kvh, int phys, uint64_t* bar) {
  using G = DecodeGeom<KVDT, HEAD, BS>;
  constexpr int TB = G::kTileBytes;
  mbar_arrive_expect_tx(bar, 2 * TB);
  if constexpr (G::kFp4) {
    const long long off = ((long long)phys * p.num_kv_heads + kvh) * TB;
    bulk_load(st, static_cast<const uint8_t*>(p.k_cache) + off, TB, bar);
    bulk_load(st + TB, static_cast<const uint8_t*>(p.v_cache) + off, TB, bar);
  } else {
    tma_load_4d(st, tmk, 0, kvh * BS, 0, phys, bar);
    tma_load_4d(st + TB, tmv, 0, kvh * BS, 0, phys, bar);
  }
}

template <int KVDT, int HEAD, int BS, int NW>
constexpr int decode_smem_bytes() {
  using G = DecodeGeom<KVDT, HEAD, BS>;
  return NW * G::kStages * 2 * G::kTileBytes + NW * G::kStages * (8 + 4) + 1024;
}

template <int QDT, int KVDT, int HEAD, int BS, int NW>
__global__ void __launch_bounds__(NW * 32, is_nvfp4<KVDT>() ? 4 : 1)
    decode_mma_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
  using G = DecodeGeom<KVDT, HEAD, BS>;
  using QE = Elem<QDT>;
  constexpr int ST = G::kStages;
  constexpr int TB = G::kTileBytes;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + NW * ST * 2 * TB);
  int* stage_ok = reinterpret_cast<int*>(bars + NW * ST);
  __shared__ int s_failed;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = blockIdx.x;
  const int kvh = blockIdx.y / p.num_head_groups;
  const int hg = blockIdx.y % p.num_head_groups;
  const int z = blockIdx.z;

  int row = r;
  if (p.query_start_loc != nullptr) {
    if (plan_rejected(p)) return;
    const int q0 = p.query_start_loc[r];
    if (p.query_start_loc[r + 1] - q0 != 1) return;  // multi-token rows go elsewhere
    row = q0;
  }
  const int seq_len = p.seq_lens[r];
  const int h0 = kvh * p.group + hg * 8;
  const int nh = min(8, p.group - hg * 8);
  const bool ok = seq_len >= 1 && seq_len <= p.max_seq_len &&
                  (long long)seq_len <= (long long)p.max_blocks_per_seq * BS;
  typename QE::T* out = reinterpret_cast<typename QE::T*>(p.out);
  if (!ok) {
    if (z == 0) {
      for (int i = threadIdx.x; i < nh * HEAD; i += NW * 32)
        out[((long long)row * p.num_q_heads + h0 + i / HEAD) * HEAD + (i % HEAD)] = QE::from_float(0.f);
      if (threadIdx.x == 0 && blockIdx.y == 0) flag_error(p.err, PA_ERRFLAG_SEQ_LEN);
    }
    return;
  }
  // tokens [start, seq_len) are this kernel's; [0, start) belong to the shared-prefix
  // kernel, or lie before the sliding window's origin block (never read)
  const int shared_start = p.query_start_loc == nullptr ? shared_prefix_tokens(p, r) : 0;
  const int start = max(shared_start, window_origin(p, seq_len, 1));
  const int nblk = (seq_len + BS - 1) / BS;
  const int pb = p.part / BS;
  const int sb0 = start / BS;
  const int b0 = sb0 + z * pb;
  if (b0 >= nblk) return;
  const int b1 = min(b0 + pb, nblk);
  const int nparts = (nblk - sb0 + pb - 1) / pb;
  // this row's partials follow those of its shared prefix (none under a window)
  const int shared_parts = shared_start > 0 ? (shared_start + p.part_shared - 1) / p.part_shared : 0;

  if (threadIdx.x == 0) {
    s_failed = 0;
    if constexpr (!G::kFp4) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
    }
    for (int i = 0; i < NW * ST; ++i) mbar_init(bars + i, 1);
    fence_mbar_init();
  }
  __syncthreads();

  const int32_t* table = p.block_tables + (long long)r * p.max_blocks_per_seq;
  const int nmine = (b1 - b0 > warp) ? (b1 - b0 - warp + NW - 1) / NW : 0;
  uint8_t* ring = smem + warp * ST * 2 * TB;
  uint64_t* wbars = bars + warp * ST;
  int* wok = stage_ok + warp * ST;

  // Block-table entries of this warp's blocks, 32 at a time in registers (lane l
  // holds the entry of the warp's block index base + l); the next window is loaded
  // one window ahead so the issuing lane never waits on a table read.
  auto load_window = [&](int base) {
    const int i = base + lane;
    return i < nmine ? table[b0 + warp + i * NW] : -1;
  };
  int tbl = load_window(0), tbl_next = load_window(32);
  // Lane 0 issues the copies of the warp's block index i into stage i % ST and
  // records in shared memory whether the block is valid (read after the wait).
  auto issue = [&](int i, int phys) {
    if (lane == 0) {
      const int s = i % ST;
      const bool valid = phys >= 0 && phys < p.num_blocks;
      wok[s] = valid;
      if (!valid) {
        flag_error(p.err, PA_ERRFLAG_BLOCK_TABLE);
        mbar_arrive(wbars + s);  // completes the phase with no data; the block is skipped
      } else {
        load_kv_tiles<KVDT, HEAD, BS>(ring + s * 2 * TB, p, &tmk, &tmv, kvh, phys, wbars + s);
      }
    }
  };
  for (int i = 0; i < min(ST, nmine); ++i) issue(i, __shfl_sync(0xffffffffu, tbl, i));

  uint32_t qb[G::kKSteps][2];
  float cA, cB;
  load_query<QDT, KVDT, HEAD>(p, row, h0, nh, qb, cA, cB);
  WarpState<HEAD> w;
  w.init();
  bool failed = false;
  int consumed = 0;

  for (int i = 0; i < nmine; ++i) {
    const int s = i % ST;
    const bool got = mbar_wait_bounded(wbars + s, (i / ST) & 1);
    if (!__all_sync(0xffffffffu, got)) {
      failed = true;
      break;
    }
    consumed = i + 1;
    if (wok[s]) {
      const int jb = b0 + warp + i * NW;
      // first key attended (sliding window), relative to the block
      const int lo = p.window > 0 ? seq_len - p.window - jb * BS : 0;
      attend_block<QDT, KVDT, HEAD, BS>(ring + s * 2 * TB, seq_len - jb * BS, lo, qb, cA, cB, w);
    }
    __syncwarp();
    const int j = i + ST;
    if (j < nmine) {
      if ((j & 31) == 0) {
        tbl = tbl_next;
        tbl_next = load_window(j + 32);
      }
      const int phys = __shfl_sync(0xffffffffu, tbl, j & 31);
      if (lane == 0) fence_proxy_async();
      issue(j, phys);
    }
  }
  if (failed) {
    // a copy never completed: record it, give the copies still in flight a bounded
    // chance to land, and write nothing for this CTA
    if (lane == 0) {
      flag_error(p.err, PA_ERRFLAG_TIMEOUT);
      for (int i = consumed; i < min(consumed + ST, nmine); ++i)
        (void)mbar_wait_bounded(wbars + (i % ST), (i / ST) & 1, 100000000ull);
    }
    s_failed = 1;
  }

  // ---- merge the warps' states through shared memory
  w.lA = warp_sum_xor(w.lA, 4, 16);
  w.lB = warp_sum_xor(w.lB, 4, 16);
  __syncthreads();
  if (s_failed) return;
  float* red = reinterpret_cast<float*>(smem);  // [NW][8][HEAD]
  float* rm = red + NW * 8 * HEAD;              // [NW][8]
  float* rl = rm + NW * 8;                      // [NW][8]
  {
    const int qq = lane & 3;
#pragma unroll
    for (int dt = 0; dt < G::kDTiles; ++dt) {
      int dA, dB;
      acc_dims<G::kScaled>(dt, lane, dA, dB);
      red[(warp * 8 + 2 * qq) * HEAD + dA] = w.acc[dt][0];
      red[(warp * 8 + 2 * qq + 1) * HEAD + dA] = w.acc[dt][1];
      red[(warp * 8 + 2 * qq) * HEAD + dB] = w.acc[dt][2];
      red[(warp * 8 + 2 * qq + 1) * HEAD + dB] = w.acc[dt][3];
    }
    if (lane < 4) {
      rm[warp * 8 + 2 * lane] = w.mA;
      rm[warp * 8 + 2 * lane + 1] = w.mB;
      rl[warp * 8 + 2 * lane] = w.lA;
      rl[warp * 8 + 2 * lane + 1] = w.lB;
    }
  }
  __syncthreads();
  const float vscale = G::kScaled ? p.v_scale[kvh * p.scale_stride] : 1.f;
  const long long pbase = p.part_off ? (long long)p.part_off[r] : (long long)row * p.max_partitions;
  const bool direct = nparts == 1 && !p.force_partials;
  for (int idx = threadIdx.x; idx < nh * HEAD; idx += NW * 32) {
    const int n = idx / HEAD, dd = idx % HEAD;
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < NW; ++ww)
      if (rl[ww * 8 + n] > 0.f) M = fmaxf(M, rm[ww * 8 + n]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int ww = 0; ww < NW; ++ww) {
      const float lw = rl[ww * 8 + n];
      if (lw > 0.f) {
        const float f = exp2f(rm[ww * 8 + n] - M);
        L = fmaf(lw, f, L);
        O = fmaf(red[(ww * 8 + n) * HEAD + dd], f, O);
      }
    }
    O *= vscale;
    const int h = h0 + n;
    if (direct) {
      out[((long long)row * p.num_q_heads + h) * HEAD + dd] = QE::from_float(L > 0.f ? O / L : 0.f);
    } else {
      const long long pi = pbase + shared_parts + z;
      p.ws_acc[(pi * p.num_q_heads + h) * HEAD + dd] = O;
      if (dd == 0) p.ws_ml[pi * p.num_q_heads + h] = make_float2(M, L);
    }
  }
}

// ------------------------------------------------------------------ shared prefix

constexpr int kMaxGroup = 8;

template <int KVDT, int HEAD, int BS>
constexpr int shared_smem_bytes() {
  using G = DecodeGeom<KVDT, HEAD, BS>;
  return G::kSharedStages * 2 * G::kTileBytes + G::kSharedStages * (8 + 8 + 4) + 1024;
}

// grid: (group, KV head x head group, partition of the shared prefix); block: one
// warp per group member (up to the group size bound) + one producer warp.
template <int QDT, int KVDT, int HEAD, int BS>
__global__ void __launch_bounds__((kMaxGroup + 1) * 32)
    shared_prefix_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv) {
  using G = DecodeGeom<KVDT, HEAD, BS>;
  constexpr int ST = G::kSharedStages;
  constexpr int TB = G::kTileBytes;

  const int g = blockIdx.x;
  const int kvh = blockIdx.y / p.num_head_groups, hg = blockIdx.y % p.num_head_groups;
  const int z = blockIdx.z;
  const int s0 = p.group_start[g], s1 = p.group_start[g + 1];
  const int nm = s1 - s0;
  const int nwarps = blockDim.x >> 5;
  if (s0 < 0 || s1 > p.num_seqs || nm < 2 || nm > nwarps - 1) return;
  const int S = group_shared_tokens(p, g, s0, s1);
  if (S == 0) return;
  const int nsb = S / BS, pb = p.part_shared / BS;
  const int b0 = z * pb;
  if (b0 >= nsb) return;
  const int nblocks = min(b0 + pb, nsb) - b0;
  const int h0 = kvh * p.group + hg * 8;
  const int nh = min(8, p.group - hg * 8);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * 2 * TB);
  uint64_t* empty = full + ST;
  int* stage_ok = reinterpret_cast<int*>(empty + ST);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    if constexpr (!G::kFp4) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
    }
    for (int i = 0; i < ST; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, nm);
    }
    fence_mbar_init();
  }
  __syncthreads();
  if (warp == nm) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint32_t all = (1u << nm) - 1u;
      int gi = 0;  // stages issued so far
      for (int i = 0; i < nblocks; ++i) {
        const int jb = b0 + i;
        // the common case, checked first: every member names the first member's block
        const int lead = p.block_tables[(long long)s0 * p.max_blocks_per_seq + jb];
        bool same = lead >= 0 && lead < p.num_blocks;
        for (int m = 1; m < nm; ++m) same &= p.block_tables[(long long)(s0 + m) * p.max_blocks_per_seq + jb] == lead;
        if (same) {
          const int s = gi % ST;
          if (gi >= ST && !mbar_wait_bounded(empty + s, ((gi / ST) - 1) & 1)) {
            flag_error(p.err, PA_ERRFLAG_TIMEOUT);
            return;  // the members time out on the full barrier and write nothing
          }
          stage_ok[s] = (int)all | kStageLast;
          load_kv_tiles<KVDT, HEAD, BS>(smem + s * 2 * TB, p, &tmk, &tmv, kvh, lead, full + s);
          ++gi;
          continue;
        }
        // otherwise one stage per distinct physical block the members name, and an
        // empty last stage when none is in range
        int e[kMaxShareMembers];
        load_share_entries(p, s0, nm, jb, e);
        uint32_t done = 0, mask = 0;
        int phys = 0;
        int m = next_share_stage(p, e, nm, done, mask, phys);
        if (m >= 0 && mask != all) flag_error(p.err, PA_ERRFLAG_SHARED_MISMATCH);
        do {
          uint32_t mask_n = 0;
          int phys_n = 0, mn = -1;
          if (m >= 0) {
            done |= mask;
            mn = next_share_stage(p, e, nm, done, mask_n, phys_n);
          }
          const int s = gi % ST;
          if (gi >= ST && !mbar_wait_bounded(empty + s, ((gi / ST) - 1) & 1)) {
            flag_error(p.err, PA_ERRFLAG_TIMEOUT);
            return;  // the members time out on the full barrier and write nothing
          }
          stage_ok[s] = (m >= 0 ? (int)mask : 0) | (mn < 0 ? kStageLast : 0);
          if (m < 0)
            mbar_arrive(full + s);  // empty phase: no member reads this block
          else
            load_kv_tiles<KVDT, HEAD, BS>(smem + s * 2 * TB, p, &tmk, &tmv, kvh, phys, full + s);
          ++gi;
          m = mn;
          mask = mask_n;
          phys = phys_n;
        } while (m >= 0);
      }
    }
    return;
  }
  if (warp > nm) return;

  // ------------------------------------------------------------------ members
  const int seq = s0 + warp;
  uint32_t qb[G::kKSteps][2];
  float cA, cB;
  load_query<QDT, KVDT, HEAD>(p, seq, h0, nh, qb, cA, cB);
  WarpState<HEAD> w;
  w.init();
  int gi = 0;  // stages consumed so far
  for (int i = 0; i < nblocks; ++i) {
    bool last = false;
    while (!last) {  // the block's stages; this member reads the one naming its block
      const int s = gi % ST;
      const bool got = mbar_wait_bounded(full + s, (gi / ST) & 1);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
        return;
      }
      const int rec = stage_ok[s];
      last = (rec & kStageLast) != 0;
      if ((rec >> warp) & 1) attend_block<QDT, KVDT, HEAD, BS>(smem + s * 2 * TB, BS, 0, qb, cA, cB, w);
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
      ++gi;
    }
  }

  // ---- this member's partial state for partition z of its shared prefix
  w.lA = warp_sum_xor(w.lA, 4, 16);
  w.lB = warp_sum_xor(w.lB, 4, 16);
  const float vscale = G::kScaled ? p.v_scale[kvh * p.scale_stride] : 1.f;
  const long long pi = (long long)seq * p.max_partitions + z;
  const int qq = lane & 3;
  const int hA = 2 * qq, hB = 2 * qq + 1;
#pragma unroll
  for (int dt = 0; dt < G::kDTiles; ++dt) {
    int dA, dB;
    acc_dims<G::kScaled>(dt, lane, dA, dB);
    if (hA < nh) {
      float* wa = p.ws_acc + (pi * p.num_q_heads + h0 + hA) * HEAD;
      wa[dA] = w.acc[dt][0] * vscale;
      wa[dB] = w.acc[dt][2] * vscale;
    }
    if (hB < nh) {
      float* wb = p.ws_acc + (pi * p.num_q_heads + h0 + hB) * HEAD;
      wb[dA] = w.acc[dt][1] * vscale;
      wb[dB] = w.acc[dt][3] * vscale;
    }
  }
  if (lane < 4) {
    if (hA < nh) p.ws_ml[pi * p.num_q_heads + h0 + hA] = make_float2(w.mA, w.lA);
    if (hB < nh) p.ws_ml[pi * p.num_q_heads + h0 + hB] = make_float2(w.mB, w.lB);
  }
}

template <int QDT, int KVDT, int HEAD, int BS>
cudaError_t launch_t(const AttnParams& p, int grid_z, const CUtensorMap* tk, const CUtensorMap* tv,
                     cudaStream_t stream) {
  constexpr int NW = 4;
  constexpr int smem = decode_smem_bytes<KVDT, HEAD, BS, NW>();
  constexpr auto kern = decode_mma_kernel<QDT, KVDT, HEAD, BS, NW>;
  cudaError_t e = set_smem<kern>(smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_seqs, p.num_kv_heads * p.num_head_groups, grid_z);
  kern<<<grid, NW * 32, smem, stream>>>(p, *tk, *tv);
  return cudaGetLastError();
}

template <int QDT, int KVDT, int HEAD, int BS>
cudaError_t launch_shared_t(const AttnParams& p, int grid_z, const CUtensorMap* tk, const CUtensorMap* tv,
                            cudaStream_t stream) {
  constexpr int smem = shared_smem_bytes<KVDT, HEAD, BS>();
  constexpr auto kern = shared_prefix_kernel<QDT, KVDT, HEAD, BS>;
  cudaError_t e = set_smem<kern>(smem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.num_groups, p.num_kv_heads * p.num_head_groups, grid_z);
  kern<<<grid, (p.max_group_size + 1) * 32, smem, stream>>>(p, *tk, *tv);
  return cudaGetLastError();
}

template <int QDT, int KVDT, bool kShared>
cudaError_t launch_shape(const AttnParams& p, int grid_z, const CUtensorMap* tk,
                         const CUtensorMap* tv, cudaStream_t s) {
  const int d = p.head_size, bs = p.block_size;
#define PA_SHAPE(D, B)                                                      \
  if (d == D && bs == B)                                                   \
    return kShared ? launch_shared_t<QDT, KVDT, D, B>(p, grid_z, tk, tv, s) \
                   : launch_t<QDT, KVDT, D, B>(p, grid_z, tk, tv, s);
  if constexpr (!is_scaled<KVDT>()) {
    PA_SHAPE(128, 16)
    PA_SHAPE(128, 32)
    PA_SHAPE(64, 16)
    PA_SHAPE(64, 32)
  } else {
    PA_SHAPE(128, 16)
    PA_SHAPE(128, 32)
  }
#undef PA_SHAPE
  return cudaErrorInvalidValue;
}

template <bool kShared>
cudaError_t dispatch(const AttnParams& p, int q_dtype, int kv_dtype, int grid_z, const CUtensorMap* tk,
                     const CUtensorMap* tv, cudaStream_t s) {
  if (q_dtype == PA_BF16 && kv_dtype == PA_BF16) return launch_shape<PA_BF16, PA_BF16, kShared>(p, grid_z, tk, tv, s);
  if (q_dtype == PA_F16 && kv_dtype == PA_F16) return launch_shape<PA_F16, PA_F16, kShared>(p, grid_z, tk, tv, s);
  if (q_dtype == PA_BF16 && kv_dtype == PA_FP8_E4M3)
    return launch_shape<PA_BF16, PA_FP8_E4M3, kShared>(p, grid_z, tk, tv, s);
  if (q_dtype == PA_F16 && kv_dtype == PA_FP8_E4M3)
    return launch_shape<PA_F16, PA_FP8_E4M3, kShared>(p, grid_z, tk, tv, s);
  if (q_dtype == PA_BF16 && kv_dtype == PA_FP8_E5M2)
    return launch_shape<PA_BF16, PA_FP8_E5M2, kShared>(p, grid_z, tk, tv, s);
  if (q_dtype == PA_F16 && kv_dtype == PA_FP8_E5M2)
    return launch_shape<PA_F16, PA_FP8_E5M2, kShared>(p, grid_z, tk, tv, s);
  if (q_dtype == PA_BF16 && kv_dtype == PA_NVFP4) return launch_shape<PA_BF16, PA_NVFP4, kShared>(p, grid_z, tk, tv, s);
  if (q_dtype == PA_F16 && kv_dtype == PA_NVFP4) return launch_shape<PA_F16, PA_NVFP4, kShared>(p, grid_z, tk, tv, s);
  return cudaErrorInvalidValue;
}

}  // namespace

bool decode_mma_supported(int q_dtype, int kv_dtype, int head_size, int block_size, int group) {
  (void)group;
  const bool q16 = q_dtype == PA_BF16 || q_dtype == PA_F16;
  if (!q16) return false;
  if (kv_dtype == q_dtype) return (head_size == 64 || head_size == 128) && (block_size == 16 || block_size == 32);
  if (kv_dtype == PA_FP8_E4M3 || kv_dtype == PA_FP8_E5M2 || kv_dtype == PA_NVFP4)
    return head_size == 128 && (block_size == 16 || block_size == 32);
  return false;
}

cudaError_t launch_decode_mma(const AttnParams& p, int q_dtype, int kv_dtype, int grid_z,
                              const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                              cudaStream_t stream) {
  return dispatch<false>(p, q_dtype, kv_dtype, grid_z, tmap_k, tmap_v, stream);
}

cudaError_t launch_shared_prefix(const AttnParams& p, int q_dtype, int kv_dtype, int grid_z,
                                 const CUtensorMap* tmap_k, const CUtensorMap* tmap_v,
                                 cudaStream_t stream) {
  if (p.max_group_size < 2 || p.max_group_size > kMaxGroup || p.num_groups <= 0) return cudaErrorInvalidValue;
  return dispatch<true>(p, q_dtype, kv_dtype, grid_z, tmap_k, tmap_v, stream);
}

}  // namespace pa
