// FlashAttention-2 style tiles on the warp-level tensor-core MMA (m16n8k16) for the
// shared prefixes of sequence groups.
//
// [AGENTIC] "統一分頁 + 共用池": forked sequences point at the same physical blocks,
// so the rows that read one shared block are gathered into one tile and the block
// is loaded once.  A tile holds up to 128 query rows; the group's K/V blocks stream
// through a ring of TMA stages (full / empty mbarriers) filled by one producer warp.
// Per 16-token block and consumer warp (16 rows each, Q fragments and the O
// accumulator in registers):
//   S = Q K^T   (m16n8k16, M = 16 rows, N = 8 tokens, K = head dim)
//   online softmax per row (running max / sum in log2 units, exp2, fp32)
//   O += P V    (P straight from the S accumulators as the A operand)
// Rows write partial states (unnormalised O, max, sum) that the merge combines with
// the members' private remainders.
#include <algorithm>

#include "pa_common.cuh"

namespace pa {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

template <int HEAD, int BS>
struct PrefillGeom {
  static constexpr int kRowBytes = HEAD * 2;
  static constexpr int kTileBytes = BS * kRowBytes;
  static constexpr int kStages = kTileBytes <= 4096 ? 8 : 5;
  static constexpr int kKSteps = HEAD / 16;  // QK k-steps over the head dim
  static constexpr int kNTok = BS / 8;       // QK n-tiles over tokens
  static constexpr int kNDim = HEAD / 8;     // PV n-tiles over the head dim
  static __device__ __forceinline__ uint32_t off(int tok, int chunk) {
    return static_cast<uint32_t>((chunk >> 3) * BS * 128) + swz128(tok, chunk & 7);
  }
};

// Online-softmax state of the two query rows a thread holds in an FA2 tile
// (warp rows lane/4 and lane/4 + 8): O accumulators over the head dim, running max
// in log2 units, running sum.
template <int HEAD>
struct RowState {
  float acc[HEAD / 8][4];
  float m[2], l[2];
  __device__ __forceinline__ void init() {
#pragma unroll
    for (int i = 0; i < HEAD / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
  }
};

// Raw scores S = Q K^T of one block: 16 rows x block_size keys, m16n8k16 with the
// Q rows as A (registers) and the K tile as B (ldmatrix, conflict-free layout).
template <int QDT, int HEAD, int BS>
__device__ __forceinline__ void fa2_scores(uint32_t kbase, const uint32_t (&qa)[HEAD / 16][4],
                                           float (&sc)[BS / 8][4]) {
  using G = PrefillGeom<HEAD, BS>;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int nt = 0; nt < G::kNTok; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < G::kKSteps; ++ks) {
#pragma unroll
    for (int np2 = 0; np2 < G::kNTok / 2; ++np2) {
      const int mi = lane >> 3;
      const int tok = 16 * np2 + (lane & 7) + 8 * (mi >> 1);
      const int chunk = 2 * ks + (mi & 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kbase + G::off(tok, chunk), b0, b1, b2, b3);
      mma_16816<QDT>(sc[2 * np2], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
      mma_16816<QDT>(sc[2 * np2 + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
    }
  }
}

// Softmax and O += P V for one block.  `sc` holds raw scores, -inf where masked;
// the positive multiplier c (scale * log2 e) is applied inside the exponent.  The
// running max is raised only when a block exceeds it by more than kRescaleSlack
// (then O and l are rescaled); P feeds the PV MMA straight from the S registers.
// V tokens at or past `rem` are zeroed (their P is 0, their bits arbitrary).
template <int QDT, int HEAD, int BS>
__device__ __forceinline__ void fa2_softmax_pv(uint32_t vbase, float (&sc)[BS / 8][4], float c, int rem,
                                               RowState<HEAD>& st) {
  using G = PrefillGeom<HEAD, BS>;
  const int lane = threadIdx.x & 31;
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < G::kNTok; ++nt) {
    mx[0] = fmaxf(mx[0], fmaxf(sc[nt][0], sc[nt][1]));
    mx[1] = fmaxf(mx[1], fmaxf(sc[nt][2], sc[nt][3]));
  }
  mx[0] = warp_max_xor(mx[0], 1, 2) * c;
  mx[1] = warp_max_xor(mx[1], 1, 2) * c;
  if (__any_sync(0xffffffffu, mx[0] > st.m[0] + kRescaleSlack || mx[1] > st.m[1] + kRescaleSlack)) {
    float al[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float nm = fmaxf(st.m[h], mx[h]);
      al[h] = nm == -INFINITY ? 1.f : ex2_approx(st.m[h] - nm);
      st.m[h] = nm;
      st.l[h] *= al[h];
    }
#pragma unroll
    for (int dn = 0; dn < G::kNDim; ++dn) {
      st.acc[dn][0] *= al[0];
      st.acc[dn][1] *= al[0];
      st.acc[dn][2] *= al[1];
      st.acc[dn][3] *= al[1];
    }
  }
  const float u0 = st.m[0] == -INFINITY ? 0.f : st.m[0], u1 = st.m[1] == -INFINITY ? 0.f : st.m[1];
  uint32_t pa[G::kNTok][2];
  float add0 = 0.f, add1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < G::kNTok; ++nt) {
    pa[nt][0] = pack2<QDT>(ex2_approx(fmaf(sc[nt][0], c, -u0)), ex2_approx(fmaf(sc[nt][1], c, -u0)));
    pa[nt][1] = pack2<QDT>(ex2_approx(fmaf(sc[nt][2], c, -u1)), ex2_approx(fmaf(sc[nt][3], c, -u1)));
    const float2 f0 = unpack2<QDT>(pa[nt][0]), f1 = unpack2<QDT>(pa[nt][1]);
    add0 += f0.x + f0.y;
    add1 += f1.x + f1.y;
  }
  st.l[0] += add0;
  st.l[1] += add1;
#pragma unroll
  for (int kt = 0; kt < BS / 16; ++kt) {
    const int tk = 16 * kt + 2 * (lane & 3);
    const bool tail = rem < 16 * kt + 16;
    const uint32_t m01 = (tk < rem ? 0xffffu : 0u) | (tk + 1 < rem ? 0xffff0000u : 0u);
    const uint32_t m23 = (tk + 8 < rem ? 0xffffu : 0u) | (tk + 9 < rem ? 0xffff0000u : 0u);
#pragma unroll
    for (int dp = 0; dp < G::kNDim / 2; ++dp) {
      const int mi = lane >> 3;
      const int tok = 16 * kt + (lane & 7) + 8 * (mi & 1);
      const int chunk = 2 * dp + (mi >> 1);
      uint32_t b0, b1, b2, b3;
      ldsm_x4_trans(vbase + G::off(tok, chunk), b0, b1, b2, b3);
      if (tail) {
        b0 &= m01;
        b1 &= m23;
        b2 &= m01;
        b3 &= m23;
      }
      mma_16816<QDT>(st.acc[2 * dp], pa[2 * kt][0], pa[2 * kt][1], pa[2 * kt + 1][0], pa[2 * kt + 1][1], b0, b1);
      mma_16816<QDT>(st.acc[2 * dp + 1], pa[2 * kt][0], pa[2 * kt][1], pa[2 * kt + 1][0], pa[2 * kt + 1][1], b2,
                     b3);
    }
  }
}

// Softmax and O += P V for two whole blocks at once (every token valid): one running-
// max update for the 2 x block_size scores, then both blocks' PV products.  Twice the
// independent MMA and exp2 work per step for the scheduler to interleave.
template <int QDT, int HEAD, int BS>
__device__ __forceinline__ void fa2_softmax_pv2(uint32_t vbase0, uint32_t vbase1, float (&sc)[2][BS / 8][4],
                                                float c, RowState<HEAD>& st) {
  using G = PrefillGeom<HEAD, BS>;
  const int lane = threadIdx.x & 31;
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int nt = 0; nt < G::kNTok; ++nt) {
      mx[0] = fmaxf(mx[0], fmaxf(sc[b][nt][0], sc[b][nt][1]));
      mx[1] = fmaxf(mx[1], fmaxf(sc[b][nt][2], sc[b][nt][3]));
    }
  mx[0] = warp_max_xor(mx[0], 1, 2) * c;
  mx[1] = warp_max_xor(mx[1], 1, 2) * c;
  if (__any_sync(0xffffffffu, mx[0] > st.m[0] + kRescaleSlack || mx[1] > st.m[1] + kRescaleSlack)) {
    float al[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float nm = fmaxf(st.m[h], mx[h]);
      al[h] = nm == -INFINITY ? 1.f : ex2_approx(st.m[h] - nm);
      st.m[h] = nm;
      st.l[h] *= al[h];
    }
#pragma unroll
    for (int dn = 0; dn < G::kNDim; ++dn) {
      st.acc[dn][0] *= al[0];
      st.acc[dn][1] *= al[0];
      st.acc[dn][2] *= al[1];
      st.acc[dn][3] *= al[1];
    }
  }
  const float u0 = st.m[0] == -INFINITY ? 0.f : st.m[0], u1 = st.m[1] == -INFINITY ? 0.f : st.m[1];
  uint32_t pa[2][G::kNTok][2];
  float add0 = 0.f, add1 = 0.f;
#pragma unroll
  for (int b = 0; b < 2; ++b)
#pragma unroll
    for (int nt = 0; nt < G::kNTok; ++nt) {
      pa[b][nt][0] = pack2<QDT>(ex2_approx(fmaf(sc[b][nt][0], c, -u0)), ex2_approx(fmaf(sc[b][nt][1], c, -u0)));
      pa[b][nt][1] = pack2<QDT>(ex2_approx(fmaf(sc[b][nt][2], c, -u1)), ex2_approx(fmaf(sc[b][nt][3], c, -u1)));
      const float2 f0 = unpack2<QDT>(pa[b][nt][0]), f1 = unpack2<QDT>(pa[b][nt][1]);
      add0 += f0.x + f0.y;
      add1 += f1.x + f1.y;
    }
  st.l[0] += add0;
  st.l[1] += add1;
#pragma unroll
  for (int b = 0; b < 2; ++b) {
    const uint32_t vbase = b ? vbase1 : vbase0;
#pragma unroll
    for (int kt = 0; kt < BS / 16; ++kt) {
#pragma unroll
      for (int dp = 0; dp < G::kNDim / 2; ++dp) {
        const int mi = lane >> 3;
        const int tok = 16 * kt + (lane & 7) + 8 * (mi & 1);
        const int chunk = 2 * dp + (mi >> 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_trans(vbase + G::off(tok, chunk), b0, b1, b2, b3);
        mma_16816<QDT>(st.acc[2 * dp], pa[b][2 * kt][0], pa[b][2 * kt][1], pa[b][2 * kt + 1][0],
                       pa[b][2 * kt + 1][1], b0, b1);
        mma_16816<QDT>(st.acc[2 * dp + 1], pa[b][2 * kt][0], pa[b][2 * kt][1], pa[b][2 * kt + 1][0],
                       pa[b][2 * kt + 1][1], b2, b3);
      }
    }
  }
}

// A-operand fragments of two query rows (zero when the row pointer is null).
template <int HEAD>
__device__ __forceinline__ void load_query_rows(const uint32_t* q0, const uint32_t* q1, uint32_t (&qa)[HEAD / 16][4]) {
  const int qq = threadIdx.x & 3;
#pragma unroll
  for (int ks = 0; ks < HEAD / 16; ++ks) {
    qa[ks][0] = q0 ? q0[8 * ks + qq] : 0u;
    qa[ks][1] = q1 ? q1[8 * ks + qq] : 0u;
    qa[ks][2] = q0 ? q0[8 * ks + 4 + qq] : 0u;
    qa[ks][3] = q1 ? q1[8 * ks + 4 + qq] : 0u;
  }
}

template <int HEAD, int BS>
constexpr int prefill_smem_bytes() {
  using G = PrefillGeom<HEAD, BS>;
  return G::kStages * 2 * G::kTileBytes + G::kStages * (8 + 8 + 4) + 1024;
}

// Shared-prefix tiles.  [AGENTIC] "統一分頁 + 共用池": forked sequences point at
// the same physical blocks.  A work item is (group of sequences sharing leading
// blocks, KV head, head group, partition of the shared prefix); its query rows are
// the (member, head) pairs of the group, member-major (row = member * GP + head),
// so every shared K/V tile is loaded once and serves every member's heads.  All
// shared keys precede every member's query position: no mask.  Each row writes a
// partial state at its sequence's shared partition z; the members' private tokens
// are attended by the decode kernel and the merge combines both.
//
// The declaration is checked block by block: when a member's entry names another
// physical block than the first member's (a stale share after copy-on-write, or a
// wrong one), that block is loaded as a stage of its own and only that member's rows
// read it (next_share_stage), so every member attends exactly its own blocks.
//
// The grid is persistent: as many CTAs as fit on the GPU at once, each taking work
// items blockIdx.x, blockIdx.x + gridDim.x, ... (items of groups that share nothing,
// or past a group's shared length, are skipped by every warp alike).  The ring's
// stage and phase run on across items, so the producer streams the next item's
// blocks while the consumers finish the current one.
template <int QDT, int HEAD, int BS>
__global__ void __launch_bounds__(kThreads, 1)
    shared_prefix_tile_kernel(const AttnParams p, const __grid_constant__ CUtensorMap tmk,
                              const __grid_constant__ CUtensorMap tmv, int parts) {
  using G = PrefillGeom<HEAD, BS>;
  constexpr int ST = G::kStages;
  constexpr int TB = G::kTileBytes;

  const int nwc = (int)(blockDim.x >> 5) - 1;  // consumer warps
  int gp = 1;
  while (gp < min(p.group, 8)) gp <<= 1;
  const int ny = p.num_kv_heads * p.num_head_groups;
  const long long total = (long long)p.num_groups * ny * parts;
  // Item `it` -> its group's first sequence s0, members nm, KV head, first query head,
  // heads, partition and blocks; false when the item has no work.
  struct Item {
    int s0, nm, kvh, h0, nh, z, b0, nblocks;
  };
  auto decode_item = [&](long long it, Item& w) -> bool {
    w.z = (int)(it % parts);
    const long long gy = it / parts;
    const int y = (int)(gy % ny), g = (int)(gy / ny);
    w.kvh = y / p.num_head_groups;
    const int hg = y % p.num_head_groups;
    w.s0 = p.group_start[g];
    const int s1 = p.group_start[g + 1];
    w.nm = s1 - w.s0;
    if (w.nm < 2 || w.nm * gp > 16 * nwc) return false;
    const int S = group_shared_tokens(p, g, w.s0, s1);
    if (S == 0) return false;
    const int pb = p.part_shared / BS, nsb = S / BS;
    w.b0 = w.z * pb;
    if (w.b0 >= nsb) return false;
    w.nblocks = min(w.b0 + pb, nsb) - w.b0;
    w.h0 = w.kvh * p.group + hg * 8;
    w.nh = min(8, p.group - hg * 8);
    return true;
  };

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + ST * 2 * TB);
  uint64_t* empty = full + ST;
  int* stage_ok = reinterpret_cast<int*>(empty + ST);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    tma_prefetch_desc(&tmk);
    tma_prefetch_desc(&tmv);
    for (int i = 0; i < ST; ++i) {
      mbar_init(full + i, 1);
      mbar_init(empty + i, nwc);
    }
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == nwc) {
    // ---------------------------------------------------------------- producer
    // The whole warp reads the block-table entries, a window of 32 blocks at a time
    // (lane j: block base + j, every member's entry, loads issued together), one window
    // ahead; lane 0 issues the copies.  The members' entries must name the first
    // member's block (checked per window); a block where they do not takes the
    // per-member path (next_share_stage) on lane 0.
    long long gi = 0;  // stages issued so far, over all items
    // entries of one window: the first member's block, and whether every member names it
    auto window = [&](const Item& w, int base, int& lead, bool& same) {
      const int jb = w.b0 + base + lane;
      lead = -1;
      same = false;
      if (base + lane < w.nblocks) {
        int e[kMaxShareMembers];
        load_share_entries(p, w.s0, w.nm, jb, e);
        lead = e[0];
        same = lead >= 0 && lead < p.num_blocks;
#pragma unroll
        for (int m = 1; m < kMaxShareMembers; ++m) same &= m >= w.nm || e[m] == lead;
      }
    };
    for (long long it = blockIdx.x; it < total; it += gridDim.x) {
      Item w;
      if (!decode_item(it, w)) continue;
      const uint32_t all = (1u << w.nm) - 1u;
      int lead_cur, lead_next;
      bool same_cur, same_next;
      window(w, 0, lead_cur, same_cur);
      window(w, 32, lead_next, same_next);
      for (int i = 0; i < w.nblocks; ++i) {
        if (i > 0 && (i & 31) == 0) {
          lead_cur = lead_next;
          same_cur = same_next;
          window(w, i + 32, lead_next, same_next);
        }
        const int lead = __shfl_sync(0xffffffffu, lead_cur, i & 31);
        const bool same = __shfl_sync(0xffffffffu, same_cur ? 1 : 0, i & 31) != 0;
        int stop = 0;
        if (lane == 0) {
          if (same) {  // the common case: one stage, every member
            const int s = (int)(gi % ST);
            if (gi >= ST && !mbar_wait_bounded(empty + s, (uint32_t)((gi / ST) - 1) & 1)) {
              flag_error(p.err, PA_ERRFLAG_TIMEOUT);
              stop = 1;  // the consumers time out on the full barrier and write nothing
            } else {
              stage_ok[s] = (int)all | kStageLast;
              uint8_t* st = smem + s * 2 * TB;
              mbar_arrive_expect_tx(full + s, 2 * TB);
              tma_load_4d(st, &tmk, 0, w.kvh * BS, 0, lead, full + s);
              tma_load_4d(st + TB, &tmv, 0, w.kvh * BS, 0, lead, full + s);
              ++gi;
            }
          } else {
            // one stage per distinct physical block the members name, and an empty
            // last stage when none is in range
            const int jb = w.b0 + i;
            int e[kMaxShareMembers];
            load_share_entries(p, w.s0, w.nm, jb, e);
            uint32_t done = 0, mask = 0;
            int phys = 0;
            int m = next_share_stage(p, e, w.nm, done, mask, phys);
            if (m >= 0 && mask != all) flag_error(p.err, PA_ERRFLAG_SHARED_MISMATCH);
            do {
              uint32_t mask_n = 0;
              int phys_n = 0, mn = -1;
              if (m >= 0) {
                done |= mask;
                mn = next_share_stage(p, e, w.nm, done, mask_n, phys_n);
              }
              const int s = (int)(gi % ST);
              if (gi >= ST && !mbar_wait_bounded(empty + s, (uint32_t)((gi / ST) - 1) & 1)) {
                flag_error(p.err, PA_ERRFLAG_TIMEOUT);
                stop = 1;
                break;
              }
              stage_ok[s] = (m >= 0 ? (int)mask : 0) | (mn < 0 ? kStageLast : 0);
              if (m < 0) {
                mbar_arrive(full + s);  // empty phase: no member reads this block
              } else {
                uint8_t* st = smem + s * 2 * TB;
                mbar_arrive_expect_tx(full + s, 2 * TB);
                tma_load_4d(st, &tmk, 0, w.kvh * BS, 0, phys, full + s);
                tma_load_4d(st + TB, &tmv, 0, w.kvh * BS, 0, phys, full + s);
              }
              ++gi;
              m = mn;
              mask = mask_n;
              phys = phys_n;
            } while (m >= 0);
          }
        }
        if (__shfl_sync(0xffffffffu, stop, 0)) return;
      }
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  const float c = p.scale * kLog2e;
  long long gi = 0;  // stages consumed so far, over all items
  for (long long it = blockIdx.x; it < total; it += gridDim.x) {
    Item w;
    if (!decode_item(it, w)) continue;
    const uint32_t all = (1u << w.nm) - 1u;
    int rm[2], rn[2];
    bool rvalid[2];
    const uint32_t* qw[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int rho = 16 * warp + (lane >> 2) + 8 * h;
      rm[h] = rho / gp;
      rn[h] = rho % gp;
      rvalid[h] = rm[h] < w.nm && rn[h] < w.nh;
      qw[h] = rvalid[h] ? reinterpret_cast<const uint32_t*>(
                              reinterpret_cast<const typename Elem<QDT>::T*>(p.q) +
                              ((long long)(w.s0 + rm[h]) * p.num_q_heads + w.h0 + rn[h]) * HEAD)
                        : nullptr;
    }
    const bool warp_active = (16 * warp) / gp < w.nm;
    const bool all_valid = __all_sync(0xffffffffu, rvalid[0] && rvalid[1]);
    // members whose rows this warp holds
    const int m_lo = (16 * warp) / gp, m_hi = min((16 * warp + 15) / gp, w.nm - 1);
    const uint32_t warp_members = warp_active ? (((2u << m_hi) - 1u) & ~((1u << m_lo) - 1u)) : 0u;
    uint32_t qa[G::kKSteps][4];
    load_query_rows<HEAD>(qw[0], qw[1], qa);
    RowState<HEAD> st;
    st.init();
    // the common case: every stage is a whole block read by every member, taken two
    // blocks at a time (one block when the item has one left, or when the next
    // stage is not such a block)
    const int fast = (int)all | kStageLast;
    int i = 0;
    int s = 0, rec = 0;
    bool have = false;  // stage s of block i waited for and rec read already
    while (i < w.nblocks) {
      if (!have) {
        s = (int)(gi % ST);
        const bool got = mbar_wait_bounded(full + s, (uint32_t)(gi / ST) & 1);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
          return;
        }
        rec = stage_ok[s];
      }
      have = true;
      if (rec != fast) break;  // the rest of the item takes the general path
      int s1 = -1, rec1 = 0;
      if (i + 1 < w.nblocks) {
        s1 = (int)((gi + 1) % ST);
        const bool got = mbar_wait_bounded(full + s1, (uint32_t)((gi + 1) / ST) & 1);
        if (!__all_sync(0xffffffffu, got)) {
          if (lane == 0) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
          return;
        }
        rec1 = stage_ok[s1];
      }
      const bool two = s1 >= 0 && rec1 == fast;
      if (warp_active) {
        const uint32_t kbase = smem_u32(smem + s * 2 * TB);
        if (two) {
          const uint32_t kbase1 = smem_u32(smem + s1 * 2 * TB);
          float sc[2][G::kNTok][4];
          fa2_scores<QDT, HEAD, BS>(kbase, qa, sc[0]);
          fa2_scores<QDT, HEAD, BS>(kbase1, qa, sc[1]);
          if (!all_valid) {  // padding rows (no member / head) take no part
#pragma unroll
            for (int b = 0; b < 2; ++b)
#pragma unroll
              for (int nt = 0; nt < G::kNTok; ++nt) {
                if (!rvalid[0]) sc[b][nt][0] = sc[b][nt][1] = -INFINITY;
                if (!rvalid[1]) sc[b][nt][2] = sc[b][nt][3] = -INFINITY;
              }
          }
          fa2_softmax_pv2<QDT, HEAD, BS>(kbase + TB, kbase1 + TB, sc, c, st);
        } else {
          float sc[G::kNTok][4];
          fa2_scores<QDT, HEAD, BS>(kbase, qa, sc);
          if (!all_valid) {
#pragma unroll
            for (int nt = 0; nt < G::kNTok; ++nt) {
              if (!rvalid[0]) sc[nt][0] = sc[nt][1] = -INFINITY;
              if (!rvalid[1]) sc[nt][2] = sc[nt][3] = -INFINITY;
            }
          }
          fa2_softmax_pv<QDT, HEAD, BS>(kbase + TB, sc, c, BS, st);
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(empty + s);
        if (two) mbar_arrive(empty + s1);
      }
      if (two) {
        i += 2;
        gi += 2;
        have = false;
      } else {
        i += 1;
        gi += 1;
        have = s1 >= 0;  // the next block's stage was waited for above
        s = s1;
        rec = rec1;
      }
    }
    // the general path, from the stage waited for above: each stage read by the
    // members that name its block, a block ending on its last stage
    while (i < w.nblocks) {
      const uint32_t readers = (uint32_t)(rec & kStageMembers);
      if (readers & warp_members) {
        const bool r0 = rvalid[0] && ((readers >> rm[0]) & 1u);
        const bool r1 = rvalid[1] && ((readers >> rm[1]) & 1u);
        const uint32_t kbase = smem_u32(smem + s * 2 * TB);
        float sc[G::kNTok][4];
        fa2_scores<QDT, HEAD, BS>(kbase, qa, sc);
#pragma unroll
        for (int nt = 0; nt < G::kNTok; ++nt) {
          if (!r0) sc[nt][0] = sc[nt][1] = -INFINITY;
          if (!r1) sc[nt][2] = sc[nt][3] = -INFINITY;
        }
        fa2_softmax_pv<QDT, HEAD, BS>(kbase + TB, sc, c, BS, st);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + s);
      ++gi;
      if (rec & kStageLast) ++i;
      if (i == w.nblocks) break;
      s = (int)(gi % ST);
      const bool got = mbar_wait_bounded(full + s, (uint32_t)(gi / ST) & 1);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) flag_error(p.err, PA_ERRFLAG_TIMEOUT);
        return;
      }
      rec = stage_ok[s];
    }

    // ---- each valid row's partial state for shared partition z
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      st.l[h] = warp_sum_xor(st.l[h], 1, 2);
      if (!rvalid[h]) continue;
      const long long pi = (long long)(w.s0 + rm[h]) * p.max_partitions + w.z;
      const int head = w.h0 + rn[h];
      float* wa = p.ws_acc + (pi * p.num_q_heads + head) * HEAD;
      const int dcol = 2 * (lane & 3);
#pragma unroll
      for (int dn = 0; dn < G::kNDim; ++dn)
        *reinterpret_cast<float2*>(wa + 8 * dn + dcol) = make_float2(st.acc[dn][2 * h], st.acc[dn][2 * h + 1]);
      if ((lane & 3) == 0) p.ws_ml[pi * p.num_q_heads + head] = make_float2(st.m[h], st.l[h]);
    }
  }
}

template <int QDT, int HEAD, int BS>
cudaError_t launch_shared_t(const AttnParams& p, int grid_z, const CUtensorMap* tk, const CUtensorMap* tv,
                            cudaStream_t stream) {
  constexpr int smem = prefill_smem_bytes<HEAD, BS>();
  constexpr auto kern = shared_prefix_tile_kernel<QDT, HEAD, BS>;
  cudaError_t e = set_smem<kern>(smem);
  if (e != cudaSuccess) return e;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return cudaErrorInvalidDevice;
  }
  int gp = 1;
  while (gp < (p.group < 8 ? p.group : 8)) gp <<= 1;
  const int nwc = (p.max_group_size * gp + 15) / 16;
  const int threads = (nwc + 1) * 32;
  // Resident CTAs per SM at this block size, cached per device as one word
  // (threads << 32 | CTAs) so that a host thread never pairs one call's thread count
  // with another's CTA count.
  static std::atomic<unsigned long long> occupancy[kMaxDevices] = {};
  int resident = 0;
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  if (tracked) {
    const unsigned long long w = occupancy[dev].load(std::memory_order_relaxed);
    if ((int)(w >> 32) == threads) resident = (int)(w & 0xffffffffu);
  }
  if (resident < 1) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kern, threads, smem) != cudaSuccess ||
        resident < 1) {
      (void)cudaGetLastError();
      resident = 1;
    }
    if (tracked)
      occupancy[dev].store(((unsigned long long)threads << 32) | (unsigned)resident, std::memory_order_relaxed);
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) {
    (void)cudaGetLastError();
    sms = 1;
  }
  const long long items = (long long)p.num_groups * p.num_kv_heads * p.num_head_groups * grid_z;
  if (items <= 0) return cudaSuccess;  // no shared partition to attend
  const long long grid = std::min<long long>(items, (long long)resident * sms);
  kern<<<static_cast<unsigned>(grid), threads, smem, stream>>>(p, *tk, *tv, grid_z);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_shared_prefix_tiles(const AttnParams& p, int q_dtype, int grid_z, const CUtensorMap* tk,
                                       const CUtensorMap* tv, cudaStream_t s) {
  const int d = p.head_size, bs = p.block_size;
  if (p.max_group_size < 2 || p.max_group_size > 8 || p.num_groups <= 0) return cudaErrorInvalidValue;
#define PA_SHAPE(Q, D, B) \
  if (q_dtype == Q && d == D && bs == B) return launch_shared_t<Q, D, B>(p, grid_z, tk, tv, s);
  PA_SHAPE(PA_BF16, 128, 16)
  PA_SHAPE(PA_BF16, 128, 32)
  PA_SHAPE(PA_BF16, 64, 16)
  PA_SHAPE(PA_BF16, 64, 32)
  PA_SHAPE(PA_F16, 128, 16)
  PA_SHAPE(PA_F16, 128, 32)
  PA_SHAPE(PA_F16, 64, 16)
  PA_SHAPE(PA_F16, 64, 32)
#undef PA_SHAPE
  return cudaErrorInvalidValue;
}

}  // namespace pa
