// Prefill (multi-token) rows of a varlen batch on the 5th-generation tensor cores:
// tcgen05.mma with operands in shared memory and accumulators in tensor memory.
//
// [LINEAGE] "Chunked prefill" / [ARCH] Part 2: a prefill chunk's query tokens attend
// the request's cached prefix and, causally, the chunk itself; [NOTES] "Prefill 与
// Decode": this work is dense and compute-bound.
//
// A persistent grid (one CTA per SM) whose CTAs claim tiles in turn from a counter: a
// tile is a work item of the varlen plan (request, first query row, partition of the
// keys) for one (KV head, group of <= 8 query heads); the K/V ring's stages and every
// barrier's phase run on from one tile to the next.  A tile's 256 query rows are
// (token, head) pairs, token-major (row = token * GP + head, GP = the head group
// padded to a power of two), split into two tiles of 128 rows; row r of a tile lives
// in TMEM lane r.  Keys stream in chunks of 64 tokens (whole paged blocks) staged by
// TMA, and every chunk serves both tiles.  Per tile and chunk i:
//   S(i)  = Q K(i)^T    M = 128 rows, N = 64 keys, K = head dim   -> TMEM (2 buffers)
//   P(i)  = softmax numerators of S(i), 16-bit, written over S(i) -> TMEM
//   O    += P(i) V(i)   M = 128 rows, N = head dim, K = 64 keys   -> TMEM (A from TMEM)
// Warps:
//   0-3, 4-7  softmax of tile 0, tile 1: one row per thread; read S(i) from TMEM,
//             keep the running max (log2 units, raised only when a chunk exceeds it
//             by more than kRescaleSlack; then O is rescaled in TMEM) and sum, write
//             P(i) over the first 32 columns of S(i)'s buffer (two values a column);
//   8, 9      TMA producers of K (one piece of one block per copy) and V (one block
//             per copy), from a block-table window read by their lanes;
//   10, 11    MMA issuers of tile 0, tile 1 (warp 10 also owns TMEM): PV(i) once
//             P(i) is written, then S(i+2) into the buffer PV(i) frees.  A thread's
//             MMAs run in issue order, so S(i+2) never overwrites P(i) before PV(i)
//             has read it; the softmax of chunk i+1 overlaps PV(i) and S(i+2).
// FP8 and NVFP4 caches: the producers copy whole (block, head) tiles of codes into a
// staging ring (NVFP4 with 1-D bulk copies, tiles as laid out in HBM) and four
// converter warps widen them to f16 in the layouts below.
// Shared memory: Q and each K chunk are K-major, [64-element piece][row][128 bytes];
// V is MN-major (head dim contiguous) and kept as the cache lays it out per block,
// [block][piece][token][128 bytes], one TMA box per block; every operand uses the
// 128-byte swizzle.
#include <algorithm>

#include "pa_common.cuh"

namespace pa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kRows = 128;        // query rows per tile = TMEM lanes
constexpr int kTiles = 2;         // tiles per CTA, sharing every K/V chunk
constexpr int kChunk = 64;        // keys per chunk
constexpr int kProducerWarp = 4 * kTiles;  // K copies; the next warp issues the V copies
constexpr int kMmaWarp = 4 * kTiles + 2;   // one MMA warp per tile; the first owns TMEM
constexpr int kConvWarp = kMmaWarp + kTiles;  // FP8 caches: four warps widen K/V to f16
constexpr int kConvThreads = 128;
template <bool F8>
constexpr int threads_tc() { return (kConvWarp + (F8 ? kConvThreads / 32 : 0)) * 32; }
constexpr int kSBufs = 2;         // S / P buffers per tile, 64 TMEM columns each
constexpr int kOCol = 128;        // a tile's O: columns [128, 128 + head dim) of its 256
constexpr int kTileCols = 256;
constexpr int kTmemCols = kTiles * kTileCols;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Shared-memory matrix descriptor: start address, leading and stride byte offsets,
// descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Instruction descriptor, kind::f16 with fp32 accumulation: operand format 0 = f16,
// 1 = bf16 (A and B alike); A K-major; B K-major (0) or MN-major (1).
__device__ __forceinline__ uint32_t umma_idesc(int M, int N, uint32_t fmt, uint32_t b_mn_major) {
  uint32_t d = 1u << 4;
  d |= fmt << 7;
  d |= fmt << 10;
  d |= b_mn_major << 16;
  d |= (uint32_t)(N >> 3) << 17;
  d |= (uint32_t)(M >> 4) << 24;
  return d;
}

__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// D (+)= A B with A read from TMEM (rows in lanes, two 16-bit values per column).
__device__ __forceinline__ void umma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// Arrive once on `bar` when every MMA this thread has issued so far has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// One lane of the (converged) warp: issues the single-thread tcgen05 operations while
// their operands stay warp-uniform.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred != 0;
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic) and the three-input maximum.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 f2_unpack(uint64_t v) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
  return r;
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive TMEM columns of the warp's 32 lanes (thread i reads lane base + i).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

template <int HEAD, int BS, bool F8 = false, bool F4 = false>
struct TcGeom {
  static constexpr int kPieces = HEAD / 64;                 // 128-byte pieces of an f16 row
  static constexpr int kBlocks = kChunk / BS;               // paged blocks per chunk
  static constexpr int kStages = F8 ? 3 : (HEAD == 128 ? 4 : 8);  // f16 K/V ring depth, chunks
  static constexpr int kPiece = kChunk * 128;               // one K piece of a chunk (64 keys)
  static constexpr int kKvBytes = kPieces * kPiece;         // K (or V) of one chunk
  static constexpr int kStageBytes = 2 * kKvBytes;          // K then V
  static constexpr int kBlockTx = kPieces * BS * 128;       // bytes of one (block, head) tile
  static constexpr int kQPiece = kRows * 128;
  static constexpr int kQTile = kPieces * kQPiece;
  // FP8 / NVFP4 caches: the copies land in a staging ring, [K | V][block][tile bytes]
  // (FP8: [token][head-dim bytes]; NVFP4: code rows, then block-scale rows)
  static constexpr int kStgStages = F8 ? 3 : 0;
  static constexpr int kStgBlock = F4 ? nvfp4_tile_bytes(BS, HEAD) : BS * HEAD;  // one (block, head) tile
  static constexpr int kStgKv = kBlocks * kStgBlock;
  static constexpr int kStgOff = kTiles * kQTile + kStages * kStageBytes;
  static constexpr int kBarOff = kStgOff + kStgStages * 2 * kStgKv;
  // full[S], empty[S]; per tile s_full[2], p_full[2], o_done[2]; mma_fin;
  // stg_full[SG], stg_empty[SG]; the TMEM address
  static constexpr int kNumBars = 2 * kStages + 3 * kSBufs * kTiles + 1 + 2 * kStgStages;
  static constexpr int kSmem = 1024 + kBarOff + 8 * kNumBars + 16;
  static_assert(kBlocks * BS == kChunk, "block size must divide the chunk");
  static_assert(kSBufs * 64 <= kOCol && kOCol + HEAD <= kTileCols, "TMEM columns");
  static_assert(kSmem <= 227 * 1024, "shared memory");
  static_assert(!F8 || HEAD == 128, "FP8 rows are one 128-byte piece");
  static_assert(kStgBlock % 16 == 0, "staged tiles are whole 16-byte pieces");
};

// Byte offset, inside a chunk's V, of key `key`'s row in piece `pc`.
template <int HEAD, int BS>
__device__ __forceinline__ uint32_t v_row_off(int key, int pc) {
  return (uint32_t)((key / BS) * (HEAD / 64) * BS * 128 + pc * BS * 128 + (key % BS) * 128);
}

template <int QDT, int KVDT, int HEAD, int BS>
__global__ void __launch_bounds__(threads_tc<is_scaled<KVDT>()>(), 1)
    prefill_tc_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
  constexpr bool kCvt = is_scaled<KVDT>();  // codes staged, then widened to f16
  constexpr bool kFp4 = is_nvfp4<KVDT>();
  constexpr int ODT = kCvt ? PA_F16 : QDT;  // MMA operand type (FP8 K/V are widened to f16)
  using G = TcGeom<HEAD, BS, kCvt, kFp4>;
  using QE = Elem<QDT>;
  constexpr int ST = G::kStages;
  constexpr int NB = G::kBlocks;

  if (plan_rejected(p)) return;
  // Persistent: each CTA claims (work item, KV head group) tiles from a counter the
  // plan kernel zeroes, so launches of any size share one list.  Claims run over the
  // whole-partition items first, then over the rest (each row tile's last, shorter
  // partition); within each class the item runs fastest, so the row tiles that read
  // one partition of one KV head are in flight together and share it through L2.
  const int nwork = *p.work_count;
  const int nfull = *p.work_full;
  const int ny = p.num_kv_heads * p.num_head_groups;
  const int total = nwork * ny;
  const int total_full = nfull * ny;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint8_t* sQ = smem;                                   // [tile][piece][row][128 bytes]
  uint8_t* sKV = sQ + kTiles * G::kQTile;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + G::kBarOff);
  uint64_t* empty = full + ST;
  // Per tile t and buffer b (chunk i uses b = i % 2, phase i / 2): s_full when S(i)
  // is in TMEM, p_full when P(i) is, o_done when PV(i) has completed.  The next use
  // of a buffer's barrier always follows its waiter's observation of the previous
  // phase (S(i+2) is issued after PV(i), PV(i) after p_full(i)), so no waiter can
  // fall two phases behind.
  uint64_t* s_full = empty + ST;                        // [tile][2]
  uint64_t* p_full = s_full + kTiles * kSBufs;
  uint64_t* o_done = p_full + kTiles * kSBufs;
  uint64_t* mma_fin = o_done + kTiles * kSBufs;
  // FP8: stg_full when a chunk's codes have landed in staging, stg_empty when the
  // converters have widened them (the f16 `full` is then arrived by the converters)
  uint64_t* stg_full = mma_fin + 1;
  uint64_t* stg_empty = stg_full + G::kStgStages;
  uint8_t* sStg = smem + G::kStgOff;                    // [stage][K | V][block][token][bytes]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(stg_empty + G::kStgStages);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

  __shared__ int s_next, s_abort;  // the next claimed tile; set when a wait gave up
  constexpr int RS = kCvt ? G::kStgStages : ST;  // the copy ring: staged codes, or the f16 stages
  uint64_t* rfull = kCvt ? stg_full : full;
  uint64_t* rempty = kCvt ? stg_empty : empty;

  // ---- set-up: barriers, the first claim, TMEM
  if (tid == 0) {
    if constexpr (!kFp4) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
    }
    for (int i = 0; i < ST; ++i) {
      mbar_init(full + i, kCvt ? kConvThreads : 2);  // the converters, or the K and V producers
      mbar_init(empty + i, kTiles);                 // every tile's MMA warp
    }
    for (int i = 0; i < G::kStgStages; ++i) {
      mbar_init(stg_full + i, 2);
      mbar_init(stg_empty + i, kConvThreads);
    }
    for (int i = 0; i < kTiles * kSBufs; ++i) {
      mbar_init(s_full + i, 1);
      mbar_init(p_full + i, kRows);
      mbar_init(o_done + i, 1);
    }
    mbar_init(mma_fin, kTiles);
    fence_mbar_init();
    s_next = atomicAdd(p.work_claim, 1);
    s_abort = 0;
  }
  __syncthreads();
  int L = s_next;
  if (L >= total) return;
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  int gch = 0;             // ring chunks of earlier tiles: stages and phases run on
  int tch0 = 0, tch1 = 0;  // each tile's chunks of earlier tiles: its S / P / O phases run on
  int g_issued = 0;        // producers: ring chunks issued so far
  for (;;) {
    const int lc = L < total_full ? L : L - total_full;  // index within the claim's class
    const int nc = L < total_full ? nfull : nwork - nfull;
    const int x = (L < total_full ? 0 : nfull) + lc % nc, y = lc / nc;
    const int4 item = p.work[x];
    const int r = item.x, row0 = item.y, z = item.z;
    const int kvh = y / p.num_head_groups, hg = y % p.num_head_groups;
    const int h0 = kvh * p.group + hg * 8;
    const int nh = min(8, p.group - hg * 8);
    int gp = 1;
    while (gp < min(p.group, 8)) gp <<= 1;
    const int tile_tokens = kRows / gp;                   // query tokens of one 128-row tile
    const int qs = p.query_start_loc[r];
    const int q_len = p.query_start_loc[r + 1] - qs;
    const int seq_len = p.seq_lens[r];
    const int t0 = row0 - qs;                             // first token of the CTA in its request
    const int ntok = min(kTiles * tile_tokens, q_len - t0);
    const int pos0 = seq_len - q_len + t0;                // position of the CTA's first token
    const int part = p.part_pf;
    // partitions count from the request's origin (0, or the block where the first
    // query's sliding window starts)
    const int origin = window_origin(p, seq_len, q_len);
    const int parts_req = (seq_len - origin + part - 1) / part;
    const int k0 = origin + z * part;
    // chunks start at the block holding the first key the CTA's first row attends
    const int klo = p.window > 0 ? max(k0, max(0, pos0 - p.window + 1) / BS * BS) : k0;
    // keys [klo, k1) of this partition that some row of tile t attends -> its chunks
    auto tile_chunks = [&](int t) {
      const int nt = min(ntok, (t + 1) * tile_tokens) - t * tile_tokens;
      if (nt <= 0) return 0;
      const int k1t = min(k0 + part, p.causal ? pos0 + t * tile_tokens + nt : seq_len);
      return k1t > klo ? (k1t - klo + kChunk - 1) / kChunk : 0;
    };
    static_assert(kTiles == 2, "two tiles per CTA");
    const int nch_t[kTiles] = {tile_chunks(0), tile_chunks(1)};
    const int k1 = min(k0 + part, p.causal ? pos0 + ntok : seq_len);
    const int nch = k1 > klo ? (k1 - klo + kChunk - 1) / kChunk : 0;  // = the largest nch_t
    const int kb_first = klo / BS;
    // keys held by the blocks a chunk loads end at the last block that reaches k1; V
    // rows past them (or past seq_len) are zeroed before they meet P.  Only the last
    // chunk can hold such rows; the last tile that reads it zeroes them.
    const int kv_loaded_end = min(seq_len, (k1 + BS - 1) / BS * BS);
    const bool tail_chunk = nch > 0 && klo + nch * kChunk > kv_loaded_end;
    const int zero_tile = nch_t[kTiles - 1] == nch ? kTiles - 1 : 0;

    // CTA row R = token * gp + head; tile R / 128, TMEM lane R % 128
    const int row_tok = tid / gp, row_head = tid % gp;
    const bool row_valid = tid < kTiles * kRows && row_tok < ntok && row_head < nh;
    const int row_pos = pos0 + row_tok;
    // FP8 caches: the row is scaled by 2^q_shift so that f16 holds it exactly (max |q|
    // below 2^15); the softmax multiplier takes 2^-q_shift back
    int q_shift = 0;
    if (tid < kTiles * kRows) {
      const uint4* src = row_valid ? reinterpret_cast<const uint4*>(
                                         reinterpret_cast<const typename QE::T*>(p.q) +
                                         ((long long)(row0 + row_tok) * p.num_q_heads + h0 + row_head) * HEAD)
                                   : nullptr;
      uint8_t* dst = sQ + (tid / kRows) * G::kQTile;
      if constexpr (!kCvt) {
#pragma unroll
        for (int c = 0; c < HEAD / 8; ++c) {
          const uint4 v = src ? src[c] : make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4*>(dst + (c >> 3) * G::kQPiece + swz128(tid % kRows, c & 7)) = v;
        }
      } else {
        float amax = 0.f;
        for (int c = 0; c < HEAD / 8 && src; ++c) {
          const uint4 v = src[c];
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack2<QDT>(w[e]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
        int ex = 0;
        frexpf(amax, &ex);  // amax < 2^ex
        q_shift = max(-100, min(100, 15 - ex));
#pragma unroll 4
        for (int c = 0; c < HEAD / 8; ++c) {
          const uint4 v = src ? src[c] : make_uint4(0, 0, 0, 0);
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
          uint32_t h[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = unpack2<QDT>(w[e]);
            h[e] = pack2<PA_F16>(ldexpf(f.x, q_shift), ldexpf(f.y, q_shift));
          }
          *reinterpret_cast<uint4*>(dst + (c >> 3) * G::kQPiece + swz128(tid % kRows, c & 7)) =
              make_uint4(h[0], h[1], h[2], h[3]);
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();  // the Q tiles are in place; every role of the previous tile is done
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int32_t* table = p.block_tables + (long long)r * p.max_blocks_per_seq;

    if (warp == kProducerWarp || warp == kProducerWarp + 1) {
      // ------------------------------------------------------------ TMA producers
      // Lane j holds block table entry kb_first + 32 w + j of window w; the next window
      // is prefetched.  An elected lane of the first warp copies a chunk's K one piece
      // of one block at a time; the second warp's copies V one whole block at a time.
      // Each arrives once per chunk on full with its own byte count.  With an FP8 cache
      // both copy whole (block, head) tiles of codes into the staging ring instead.
      const bool is_v = warp != kProducerWarp;
      const int kb_end = (k1 + BS - 1) / BS;  // blocks [kb_first, kb_end) are loaded
      auto load_window = [&](int w) {
        const int kb = kb_first + 32 * w + lane;
        return kb < kb_end ? table[kb] : -1;
      };
      int cur_w = 0;
      int win = load_window(0);
      int win_next = load_window(1);
      for (int i = 0; i < nch; ++i) {
        const int g = gch + i;  // the chunk's place in the ring, counted across work items
        const int s = g % RS;
        if (g >= RS && !__all_sync(0xffffffffu, mbar_wait_bounded(rempty + s, ((g / RS) - 1) & 1))) {
          if (lane == 0) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
          s_abort = 1;
          break;
        }
        const int w = (i * NB) >> 5;  // NB divides 32: a chunk's blocks share one window
        if (w != cur_w) {
          win = win_next;
          win_next = load_window(w + 1);
          cur_w = w;
        }
        int phys[NB];
        int nvalid = 0;
#pragma unroll
        for (int b = 0; b < NB; ++b) {
          const int e = __shfl_sync(0xffffffffu, win, (i * NB + b) & 31);
          const bool in_range = kb_first + i * NB + b < kb_end;
          const bool ok_b = in_range && e >= 0 && e < p.num_blocks;
          if (in_range && !ok_b && lane == 0 && !is_v) flag_error(p.err, PA_ERRFLAG_BLOCK_TABLE);
          phys[b] = ok_b ? e : -1;
          nvalid += ok_b;
        }
        if (kCvt && elect_one()) {
          uint8_t* sg = sStg + s * 2 * G::kStgKv + (is_v ? G::kStgKv : 0);
          if (nvalid == 0) {
            mbar_arrive(rfull + s);
          } else {
            mbar_arrive_expect_tx(rfull + s, (uint32_t)(nvalid * G::kStgBlock));
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              if (phys[b] < 0) continue;
              if constexpr (kFp4) {  // a whole tile, as laid out in HBM
                const void* src = static_cast<const uint8_t*>(is_v ? p.v_cache : p.k_cache) +
                                  ((long long)phys[b] * p.num_kv_heads + kvh) * G::kStgBlock;
                bulk_load(sg + b * G::kStgBlock, src, G::kStgBlock, rfull + s);
              } else {
                tma_load_4d(sg + b * G::kStgBlock, is_v ? &tmv : &tmk, 0, kvh * BS, 0, phys[b], rfull + s);
              }
            }
          }
        } else if (!kCvt && elect_one()) {
          uint8_t* sk = sKV + s * G::kStageBytes;
          if (nvalid == 0) {
            mbar_arrive(full + s);
          } else {
            mbar_arrive_expect_tx(full + s, (uint32_t)(nvalid * G::kBlockTx));
#pragma unroll
            for (int b = 0; b < NB; ++b) {
              if (phys[b] < 0) continue;
              if (is_v) {
                tma_load_4d(sk + G::kKvBytes + b * G::kBlockTx, &tmv, 0, kvh * BS, 0, phys[b], full + s);
              } else {
#pragma unroll
                for (int pc = 0; pc < G::kPieces; ++pc)
                  tma_load_4d(sk + pc * G::kPiece + b * BS * 128, &tmk, 0, kvh * BS, pc, phys[b], full + s);
              }
            }
          }
        }
        __syncwarp();
        g_issued = g + 1;
      }
    } else if (kCvt && warp >= kConvWarp) {
      // ------------------------------------------------------------ FP8 / NVFP4 converters
      // Chunk i: wait for its codes in staging and for its f16 stage to be free, widen
      // every code to f16 exactly (every e4m3 value and every finite e5m2 value is an
      // f16 value; NVFP4: E2M1 value x E4M3 block scale, at most 6 significant bits
      // and within f16's normal range; the fp32 scales are applied later) into the
      // K-major K layout and the per-block V layout, release the staging slot and mark
      // the f16 stage full.
      // Thread t owns one row: K row t (t < 64) or V row t - 64.  Reading group g of
      // a row and writing its two f16 chunks touch eight different 16-byte bank groups
      // across any eight consecutive rows, so neither side has bank conflicts.
      if constexpr (kCvt) {
      const int ct = tid - kConvWarp * 32;
      const int tensor = ct / kChunk, key = ct % kChunk;
      const int blk = key / BS, tok = key % BS, sw = key & 7;  // tok & 7 == key & 7
      for (int i = 0; i < nch; ++i) {
        const int g = gch + i;
        const int s = g % ST, ss = g % G::kStgStages;
        bool ok = mbar_wait_bounded(stg_full + ss, (g / G::kStgStages) & 1);
        if (g >= ST) ok = ok && mbar_wait_bounded(empty + s, ((g / ST) - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
          s_abort = 1;
          break;
        }
        const uint8_t* stile = sStg + ss * 2 * G::kStgKv + tensor * G::kStgKv + blk * G::kStgBlock;
        uint8_t* sk = sKV + s * G::kStageBytes;
        uint8_t* drow = tensor == 0 ? sk + key * 128 : sk + G::kKvBytes + blk * G::kBlockTx + tok * 128;
        const int piece_stride = tensor == 0 ? G::kPiece : BS * 128;
        if constexpr (kFp4) {
          // a 64-byte code row and its 8 block scales; the row's four 16-byte chunks are
          // read in an order rotated by row pair, so a warp's reads spread over the bank
          // line (64-byte rows) and its writes stay on distinct banks (rows differ in
          // their swizzle)
          const uint8_t* crow = stile + tok * (HEAD / 2);
          const uint2 sc8 = *reinterpret_cast<const uint2*>(stile + BS * (HEAD / 2) + tok * (HEAD / 16));
          const uint64_t sc64 = (static_cast<uint64_t>(sc8.y) << 32) | sc8.x;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int cc = (c + (key >> 1)) & 3;  // chunk: groups 2cc, 2cc+1 = dims 32cc .. 32cc+31
            const uint4 codes = *reinterpret_cast<const uint4*>(crow + 16 * cc);
            const uint32_t sp = fp8x2_to_f16x2<PA_FP8_E4M3>(static_cast<uint16_t>(sc64 >> (16 * cc)));
            const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {  // group g = 2cc + hh: codes 16 g .. 16 g + 15
              const int g = 2 * cc + hh;
              const uint32_t sg = __byte_perm(sp, 0, hh ? 0x3232 : 0x1010);
              uint32_t lo[4], hi[4];
              fp4x8_to_f16x2x4(cw[2 * hh], lo);
              fp4x8_to_f16x2x4(cw[2 * hh + 1], hi);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                lo[e] = hmul2_u32(lo[e], sg);
                hi[e] = hmul2_u32(hi[e], sg);
              }
              uint8_t* row = drow + (g >> 2) * piece_stride;
              const int ch = (2 * g) & 7;
              *reinterpret_cast<uint4*>(row + ((ch ^ sw) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
              *reinterpret_cast<uint4*>(row + (((ch + 1) ^ sw) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            }
          }
        } else {
          const uint8_t* srow = stile + tok * 128;
#pragma unroll
          for (int g = 0; g < 8; ++g) {  // codes 16 g .. 16 g + 15 -> f16 chunks 2g, 2g+1 (mod 8) of piece g / 4
            const uint4 codes = *reinterpret_cast<const uint4*>(srow + ((g ^ sw) << 4));
            const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
            uint32_t h[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) fp8x4_to_f16x2x2<KVDT>(cw[e], h[2 * e], h[2 * e + 1]);
            uint8_t* row = drow + (g >> 2) * piece_stride;
            const int cc = (2 * g) & 7;
            *reinterpret_cast<uint4*>(row + ((cc ^ sw) << 4)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(row + (((cc + 1) ^ sw) << 4)) = make_uint4(h[4], h[5], h[6], h[7]);
          }
        }
        fence_proxy_async();  // generic-proxy writes, read next by the tensor core
        mbar_arrive(stg_empty + ss);
        mbar_arrive(full + s);
      }
      }
    } else if (warp >= kMmaWarp && warp < kConvWarp) {
      // ------------------------------------------------------------ MMA issuers
      // One warp per tile follows that tile's schedule (descriptors stay
      // warp-uniform); an elected lane issues each group of MMAs and its commit.  Per
      // chunk i: PV(i) as soon as P(i) is in TMEM, then S(i+2) into the buffer PV(i)
      // frees.  The two tiles' streams run independently on the tensor core.
      const int t = warp - kMmaWarp;
      const int my_nch = t == 0 ? nch_t[0] : nch_t[1];
      const int tc = t == 0 ? tch0 : tch1;  // this tile's S / P / O sequence runs on across items
      const uint32_t fmt = ODT == PA_BF16 ? 1u : 0u;
      const uint32_t id_s = umma_idesc(kRows, kChunk, fmt, 0);
      const uint32_t id_o = umma_idesc(kRows, HEAD, fmt, 1);
      // descriptor start addresses count 16-byte units: offsets are added pre-shifted
      const uint64_t qd = umma_desc(smem_u32(sQ) + t * G::kQTile, 16, 1024);
      const uint64_t kd0 = umma_desc(smem_u32(sKV), 16, 1024);
      const uint64_t vd0 = umma_desc(smem_u32(sKV) + G::kKvBytes, BS * 128, 1024);
      const uint32_t tT = tmem + t * kTileCols;
      uint64_t* my_p_full = p_full + t * kSBufs;
      auto issue_s = [&](int j) {
        const uint64_t kd = kd0 + (uint64_t)((((gch + j) % ST) * G::kStageBytes) >> 4);
        const uint32_t d = tT + ((tc + j) % kSBufs) * 64;
        if (elect_one()) {
#pragma unroll
          for (int ks = 0; ks < HEAD / 16; ++ks) {
            const uint32_t qo = ((ks >> 2) * G::kQPiece + (ks & 3) * 32) >> 4;
            const uint32_t ko = ((ks >> 2) * G::kPiece + (ks & 3) * 32) >> 4;
            umma(d, qd + qo, kd + ko, id_s, ks > 0 ? 1u : 0u);
          }
          umma_commit(s_full + t * kSBufs + (tc + j) % kSBufs);
        }
        __syncwarp();
      };
      auto wait_all = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity));
      };
      bool ok = true;
      for (int j = 0; ok && j < kSBufs && j < my_nch; ++j) {
        ok = wait_all(full + (gch + j) % ST, ((gch + j) / ST) & 1);
        if (!ok) break;
        tc_fence_after();
        issue_s(j);
      }
      for (int i = 0; ok && i < nch; ++i) {
        const int g = gch + i, ci = tc + i;
        if (i >= my_nch) {
          // This tile does not read chunk i.  It still releases the stage once, after
          // the chunk has landed (so it never arrives twice within one phase).
          if (!(ok = wait_all(full + g % ST, (g / ST) & 1))) break;
          if (elect_one()) mbar_arrive(empty + g % ST);
          __syncwarp();
          continue;
        }
        // a tail chunk's V is read only after its zeroing tile has written P(i)
        const int cz = (zero_tile == 0 ? tch0 : tch1) + i;
        if (tail_chunk && i == nch - 1 && t != zero_tile &&
            !(ok = wait_all(p_full + zero_tile * kSBufs + cz % kSBufs, (cz / kSBufs) & 1)))
          break;
        if (!(ok = wait_all(my_p_full + ci % kSBufs, (ci / kSBufs) & 1))) break;
        tc_fence_after();
        const uint64_t vd = vd0 + (uint64_t)(((g % ST) * G::kStageBytes) >> 4);
        const uint32_t pt = tT + (ci % kSBufs) * 64;
        if (elect_one()) {
#pragma unroll
          for (int ks = 0; ks < kChunk / 16; ++ks)
            umma_tmem_a(tT + kOCol, pt + ks * 8, vd + (uint64_t)(v_row_off<HEAD, BS>(16 * ks, 0) >> 4), id_o,
                        (i > 0 || ks > 0) ? 1u : 0u);
          umma_commit(o_done + t * kSBufs + ci % kSBufs);
          umma_commit(empty + g % ST);
        }
        __syncwarp();
        const int j = i + kSBufs;
        if (j < my_nch) {
          if (!(ok = wait_all(full + (gch + j) % ST, ((gch + j) / ST) & 1))) break;
          tc_fence_after();
          issue_s(j);
        }
      }
      if (!ok) {
        if (lane == 0) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
        s_abort = 1;
      }
    } else {
      // ------------------------------------------------------------ softmax warps
      // Warps 4t .. 4t+3 serve tile t; thread = TMEM lane = row of the tile.
      const int t = warp >> 2;
      const int my_nch = t == 0 ? nch_t[0] : nch_t[1];
      const int tc = t == 0 ? tch0 : tch1;
      const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
      const uint32_t tT = tmem + t * kTileCols;
      const uint32_t tO = tT + kOCol;
      uint64_t* my_s_full = s_full + t * kSBufs;
      uint64_t* my_p_full = p_full + t * kSBufs;
      uint64_t* my_o_done = o_done + t * kSBufs;
      // score multiplier in log2 units; FP8: the K scale and the row's f16 shift too
      const float c = kCvt ? ldexpf(p.scale * kLog2e * p.k_scale[kvh * p.scale_stride], -q_shift) : p.scale * kLog2e;
      const float out_scale = kCvt ? p.v_scale[kvh * p.scale_stride] : 1.f;
      const int row_limit = p.causal ? min(k1, row_pos + 1) : k1;  // this row attends keys < row_limit
      const int row_lo = p.window > 0 ? max(0, row_pos - p.window + 1) : 0;  // ... and keys >= row_lo
      float m = -INFINITY, l = 0.f;
      bool fail = false;
      for (int i = 0; i < my_nch; ++i) {
        const int base = klo + i * kChunk;
        const int ci = tc + i, g = gch + i;
        const uint32_t tS = tT + (ci % kSBufs) * 64;
        const bool got = mbar_wait_bounded(my_s_full + ci % kSBufs, (ci / kSBufs) & 1);
        if (!__all_sync(0xffffffffu, got)) {
          fail = true;
          break;
        }
        tc_fence_after();
        uint32_t sr[kChunk];
        tmem_ld32(tS + lane_base, sr);
        tmem_ld32(tS + 32 + lane_base, sr + 32);
        tmem_wait_ld();
        float sc[kChunk];
#pragma unroll
        for (int j = 0; j < kChunk; ++j) sc[j] = __uint_as_float(sr[j]);
        const int rem = row_limit - base;  // keys of this chunk the row attends: [lo_rem, rem)
        const int lo_rem = row_lo - base;
        if (rem < kChunk || lo_rem > 0) {
#pragma unroll
          for (int j = 0; j < kChunk; ++j)
            if (j >= rem || j < lo_rem) sc[j] = -INFINITY;
        }
        // row maximum: eight independent chains of three-input maxima
        float mq[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float x = max3(sc[8 * q], sc[8 * q + 1], sc[8 * q + 2]);
          x = max3(x, sc[8 * q + 3], sc[8 * q + 4]);
          x = max3(x, sc[8 * q + 5], sc[8 * q + 6]);
          mq[q] = fmaxf(x, sc[8 * q + 7]);
        }
        const float mx = max3(max3(mq[0], mq[1], mq[2]), max3(mq[3], mq[4], mq[5]), fmaxf(mq[6], mq[7])) * c;
        const bool need = mx > m + kRescaleSlack;
        float al = 1.f;
        if (need) {
          const float nm = fmaxf(m, mx);
          al = ex2_approx(m - nm);  // 0 while the row had no key yet
          m = nm;
          l *= al;
        }
        const float u = m == -INFINITY ? 0.f : m;
        // p = 2^(s c - u) on pairs of keys; the row sum in four packed accumulators
        const uint64_t c2 = f2_pack(c, c), nu2 = f2_pack(-u, -u);
        uint32_t pk[kChunk / 2];
        uint64_t acc2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int j = 0; j < kChunk / 2; ++j) {
          const float2 x = f2_unpack(f2_fma(f2_pack(sc[2 * j], sc[2 * j + 1]), c2, nu2));
          const float e0 = ex2_approx(x.x), e1 = ex2_approx(x.y);
          acc2[j & 3] = f2_add(acc2[j & 3], f2_pack(e0, e1));
          pk[j] = pack2<ODT>(e0, e1);
        }
        const float2 lsum = f2_unpack(f2_add(f2_add(acc2[0], acc2[1]), f2_add(acc2[2], acc2[3])));
        l += lsum.x + lsum.y;
        // O is rescaled only once PV(i-1) has completed
        if (__any_sync(0xffffffffu, need) && i > 0) {
          const bool done = mbar_wait_bounded(my_o_done + (ci - 1) % kSBufs, ((ci - 1) / kSBufs) & 1);
          if (!__all_sync(0xffffffffu, done)) {
            fail = true;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int cb = 0; cb < HEAD; cb += 32) {
            uint32_t o[32];
            tmem_ld32(tO + cb + lane_base, o);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * al);
            tmem_st32(tO + cb + lane_base, o);
          }
        }
        // P(i) over the first half of S(i)'s columns
        tmem_st32(tS + lane_base, pk);
        // V rows past the loaded keys may hold any bits; their P is 0, so they are
        // zeroed to keep 0 * V finite.  Each thread's stores precede its own arrival
        // on p_full, which every PV of this chunk waits for.
        if (tail_chunk && t == zero_tile && i == nch - 1) {
          const bool landed = mbar_wait_bounded(full + g % ST, (g / ST) & 1);
          const int vrem = kv_loaded_end - base;
          const int rr = tid % kRows;
          if (landed && rr < G::kPieces * kChunk) {
            const int key = rr % kChunk, pc = rr / kChunk;
            if (key >= vrem) {
              uint4* d = reinterpret_cast<uint4*>(sKV + (g % ST) * G::kStageBytes + G::kKvBytes +
                                                  v_row_off<HEAD, BS>(key, pc));
#pragma unroll
              for (int q = 0; q < 8; ++q) d[q] = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async();
        }
        tmem_wait_st();
        // Observe PV(i-2): every phase of both o_done barriers is waited for in order
        // and never more than one phase late, so the parity waits stay unambiguous.
        if (i >= kSBufs) {
          const bool done = mbar_wait_bounded(my_o_done + ci % kSBufs, ((ci - kSBufs) / kSBufs) & 1);
          if (!__all_sync(0xffffffffu, done)) {
            fail = true;
            break;
          }
        }
        tc_fence_before();
        mbar_arrive(my_p_full + ci % kSBufs);
      }
      if (!fail && my_nch > 0) {
        const int cl = tc + my_nch - 1;
        const bool done = mbar_wait_bounded(my_o_done + cl % kSBufs, (cl / kSBufs) & 1);
        fail = !__all_sync(0xffffffffu, done);
        tc_fence_after();
      }
      if (fail) {
        if (lane == 0) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
        s_abort = 1;
      } else {
        // ---- epilogue: thread = row; direct output when the row needs one partition,
        // else its partial state (unnormalised O, max in log2 units, sum)
        const int kv_len = p.causal ? row_pos + 1 : seq_len;
        const int parts_row = (kv_len - origin + part - 1) / part;
        const bool write = row_valid && z < parts_row;
        const bool direct = parts_row == 1;
        const int tq = t0 + row_tok;
        const int head = h0 + row_head;
        const float inv = l > 0.f ? out_scale / l : 0.f;
        const long long pi = (long long)p.part_off[r] + (long long)tq * parts_req + z;
        typename QE::T* o_row =
            reinterpret_cast<typename QE::T*>(p.out) + ((long long)(qs + tq) * p.num_q_heads + head) * HEAD;
        float* w_row = p.ws_acc + (pi * p.num_q_heads + head) * HEAD;
#pragma unroll 1
        for (int cb = 0; cb < HEAD; cb += 32) {
          uint32_t o[32];
          if (my_nch > 0) {
            tmem_ld32(tO + cb + lane_base, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0u;
          }
          if (!write) continue;
          if (direct) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint4 v;
              v.x = pack2<QDT>(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
              v.y = pack2<QDT>(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
              v.z = pack2<QDT>(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
              v.w = pack2<QDT>(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
              *reinterpret_cast<uint4*>(o_row + cb + 8 * q) = v;
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q)
              *reinterpret_cast<float4*>(w_row + cb + 4 * q) =
                  make_float4(__uint_as_float(o[4 * q]) * out_scale, __uint_as_float(o[4 * q + 1]) * out_scale,
                              __uint_as_float(o[4 * q + 2]) * out_scale, __uint_as_float(o[4 * q + 3]) * out_scale);
          }
        }
        if (write && !direct) p.ws_ml[pi * p.num_q_heads + head] = make_float2(m, l);
      }
    }

    gch += nch;
    tch0 += nch_t[0];
    tch1 += nch_t[1];
    if (tid == 0) s_next = atomicAdd(p.work_claim, 1);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    L = s_next;
    if (L >= total || s_abort) break;
  }

  // ---- teardown: every MMA completes and every copy lands before TMEM is released
  // and the CTA leaves
  if (warp >= kMmaWarp && warp < kConvWarp) {
    if (elect_one()) umma_commit(mma_fin);
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait_bounded(mma_fin, 0)) && lane == 0) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
  } else if ((warp == kProducerWarp || warp == kProducerWarp + 1) && lane == 0) {
    for (int j = max(0, g_issued - RS); j < g_issued; ++j)
      if (!mbar_wait_bounded(rfull + j % RS, (j / RS) & 1)) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

template <int QDT, int KVDT, int HEAD, int BS>
cudaError_t launch_tc_t(const AttnParams& p, int num_items, int max_ctas, const CUtensorMap* tk,
                        const CUtensorMap* tv, cudaStream_t stream) {
  constexpr bool kCvt = is_scaled<KVDT>();
  constexpr int smem = TcGeom<HEAD, BS, kCvt, is_nvfp4<KVDT>()>::kSmem;
  constexpr auto kern = prefill_tc_kernel<QDT, KVDT, HEAD, BS>;
  const cudaError_t e = set_smem<kern>(smem);
  if (e != cudaSuccess) return e;
  const long long tiles = (long long)num_items * p.num_kv_heads * p.num_head_groups;
  const int grid = static_cast<int>(std::min<long long>(tiles, std::max(1, max_ctas)));
  kern<<<grid, threads_tc<kCvt>(), smem, stream>>>(p, *tk, *tv);
  return cudaGetLastError();
}

template <int QDT, int KVDT>
cudaError_t launch_tc_shape(const AttnParams& p, int num_items, int max_ctas, const CUtensorMap* tk,
                            const CUtensorMap* tv, cudaStream_t s) {
  const int d = p.head_size, bs = p.block_size;
  if (d == 128 && bs == 16) return launch_tc_t<QDT, KVDT, 128, 16>(p, num_items, max_ctas, tk, tv, s);
  if (d == 128 && bs == 32) return launch_tc_t<QDT, KVDT, 128, 32>(p, num_items, max_ctas, tk, tv, s);
  if (d == 128 && bs == 64) return launch_tc_t<QDT, KVDT, 128, 64>(p, num_items, max_ctas, tk, tv, s);
  if constexpr (!is_scaled<KVDT>()) {
    if (d == 64 && bs == 16) return launch_tc_t<QDT, KVDT, 64, 16>(p, num_items, max_ctas, tk, tv, s);
    if (d == 64 && bs == 32) return launch_tc_t<QDT, KVDT, 64, 32>(p, num_items, max_ctas, tk, tv, s);
    if (d == 64 && bs == 64) return launch_tc_t<QDT, KVDT, 64, 64>(p, num_items, max_ctas, tk, tv, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

// Query tokens of one prefill CTA: two 128-row tiles whose rows are (token, head)
// pairs, the head group padded to a power of two, at most 8 heads per tile.
int prefill_tile_tokens(int group) {
  int g8 = 1;
  while (g8 < group && g8 < 8) g8 <<= 1;
  return kTiles * kRows / g8;
}

bool prefill_tc_supported(int q_dtype, int kv_dtype, int head_size, int block_size) {
  if (!(q_dtype == PA_BF16 || q_dtype == PA_F16)) return false;
  if (!(block_size == 16 || block_size == 32 || block_size == 64)) return false;
  if (kv_dtype == PA_FP8_E4M3 || kv_dtype == PA_FP8_E5M2 || kv_dtype == PA_NVFP4)
    return head_size == 128;  // converted rows are one 128-byte piece of codes (FP8) / 64 bytes (NVFP4)
  return kv_dtype == q_dtype && (head_size == 64 || head_size == 128);
}

cudaError_t launch_prefill_tc(const AttnParams& p, int q_dtype, int kv_dtype, int num_items, int max_ctas,
                              const CUtensorMap* tmap_k, const CUtensorMap* tmap_v, cudaStream_t stream) {
  if (num_items <= 0) return cudaSuccess;
  if (kv_dtype == PA_FP8_E4M3) {
    if (q_dtype == PA_BF16) return launch_tc_shape<PA_BF16, PA_FP8_E4M3>(p, num_items, max_ctas, tmap_k, tmap_v, stream);
    if (q_dtype == PA_F16) return launch_tc_shape<PA_F16, PA_FP8_E4M3>(p, num_items, max_ctas, tmap_k, tmap_v, stream);
    return cudaErrorInvalidValue;
  }
  if (kv_dtype == PA_FP8_E5M2) {
    if (q_dtype == PA_BF16) return launch_tc_shape<PA_BF16, PA_FP8_E5M2>(p, num_items, max_ctas, tmap_k, tmap_v, stream);
    if (q_dtype == PA_F16) return launch_tc_shape<PA_F16, PA_FP8_E5M2>(p, num_items, max_ctas, tmap_k, tmap_v, stream);
    return cudaErrorInvalidValue;
  }
  if (kv_dtype == PA_NVFP4) {
    if (q_dtype == PA_BF16) return launch_tc_shape<PA_BF16, PA_NVFP4>(p, num_items, max_ctas, tmap_k, tmap_v, stream);
    if (q_dtype == PA_F16) return launch_tc_shape<PA_F16, PA_NVFP4>(p, num_items, max_ctas, tmap_k, tmap_v, stream);
    return cudaErrorInvalidValue;
  }
  if (kv_dtype != q_dtype) return cudaErrorInvalidValue;
  if (q_dtype == PA_BF16) return launch_tc_shape<PA_BF16, PA_BF16>(p, num_items, max_ctas, tmap_k, tmap_v, stream);
  if (q_dtype == PA_F16) return launch_tc_shape<PA_F16, PA_F16>(p, num_items, max_ctas, tmap_k, tmap_v, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
