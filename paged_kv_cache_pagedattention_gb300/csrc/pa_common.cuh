// Device-side building blocks shared by the library's kernels: element types,
// parameter blocks, the error word, and thin inline-PTX wrappers for mbarriers,
// TMA bulk-tensor copies, ldmatrix / movmatrix and the warp-level tensor-core MMA.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "pa_internal.h"

namespace pa {

// ---------------------------------------------------------------- host side

constexpr int kMaxDevices = 64;

// Opt kernel kKernel into `smem` bytes of dynamic shared memory on the current
// device, once per device.  The per-device flags are atomics: host threads may
// launch at once, and a repeated opt-in only repeats the same call.
template <auto kKernel>
cudaError_t set_smem(int smem) {
  static std::atomic<bool> done[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return cudaErrorInvalidDevice;
  }
  const bool tracked = dev >= 0 && dev < kMaxDevices;
  if (tracked && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kKernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // consume it: the caller reports the failure
    return e;
  }
  if (tracked) done[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

// ---------------------------------------------------------------- elements

template <int DT>
struct Elem;
template <>
struct Elem<PA_F32> {
  using T = float;
  static constexpr int bytes = 4;
  static __device__ __forceinline__ float load(const T* p) { return *p; }
  static __device__ __forceinline__ T from_float(float x) { return x; }
};
template <>
struct Elem<PA_F16> {
  using T = __half;
  static constexpr int bytes = 2;
  static __device__ __forceinline__ float load(const T* p) { return __half2float(*p); }
  static __device__ __forceinline__ T from_float(float x) { return __float2half_rn(x); }
};
template <>
struct Elem<PA_BF16> {
  using T = __nv_bfloat16;
  static constexpr int bytes = 2;
  static __device__ __forceinline__ float load(const T* p) { return __bfloat162float(*p); }
  static __device__ __forceinline__ T from_float(float x) { return __float2bfloat16_rn(x); }
};
template <>
struct Elem<PA_FP8_E4M3> {
  using T = uint8_t;
  static constexpr int bytes = 1;
  static __device__ __forceinline__ float load(const T* p) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(*p), __NV_E4M3);
    return __half2float(__half(h));
  }
};
template <>
struct Elem<PA_FP8_E5M2> {
  using T = uint8_t;
  static constexpr int bytes = 1;
  static __device__ __forceinline__ float load(const T* p) {
    __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(*p), __NV_E5M2);
    return __half2float(__half(h));
  }
};

// FP8 cache formats (codes with a per-tensor scale).
template <int DT>
constexpr bool is_fp8() { return DT == PA_FP8_E4M3 || DT == PA_FP8_E5M2; }
// NVFP4 cache format: per (block, KV head) tile, block_size rows of head/2 bytes of
// E2M1 codes (element 2i in the low nibble of byte i), then block_size rows of
// head/16 E4M3 block scales; values carry the fp32 scale as FP8 does.
template <int DT>
constexpr bool is_nvfp4() { return DT == PA_NVFP4; }
// Cache formats whose values carry an fp32 scale (k_scale / v_scale).
template <int DT>
constexpr bool is_scaled() { return is_fp8<DT>() || is_nvfp4<DT>(); }

__device__ __forceinline__ void flag_error(unsigned* err, unsigned bits) {
  if (err) atomicOr(err, bits);
}

__device__ __forceinline__ int ceil_div_dev(int a, int b) { return (a + b - 1) / b; }

// Index of the first partial row of query row `row`, and the partition count of
// the row's request (see pa_internal.h, AttnParams).
__device__ __forceinline__ long long partial_base(const AttnParams& p, int request, int row,
                                                  int row_in_request, int parts_of_request) {
  if (p.part_off) return (long long)p.part_off[request] + (long long)row_in_request * parts_of_request;
  return (long long)row * p.max_partitions;
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ uint32_t smem_u32(const void* ptr) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(ptr));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns` nanoseconds.
// Returns false on timeout.  Every thread that calls it polls on its own.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled bulk-tensor copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// 4-D tiled bulk-tensor copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

// Byte offset of 16-byte chunk `chunk` (0..7) of 128-byte row `row` inside a tile
// written by TMA with CU_TENSOR_MAP_SWIZZLE_128B (tile base 1024-byte aligned).
__device__ __forceinline__ uint32_t swz128(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// ---------------------------------------------------------------- warp MMA

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a) {
  uint32_t d;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}

template <int DT>
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1);

template <>
__device__ __forceinline__ void mma_16816<PA_BF16>(float (&c)[4], uint32_t a0, uint32_t a1,
                                                   uint32_t a2, uint32_t a3, uint32_t b0,
                                                   uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <>
__device__ __forceinline__ void mma_16816<PA_F16>(float (&c)[4], uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint32_t b0,
                                                  uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Pack two fp32 into one register of two 16-bit elements (lo = a), round to nearest.
template <int DT>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<PA_BF16>(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
template <>
__device__ __forceinline__ uint32_t pack2<PA_F16>(float a, float b) {
  __half2 v = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The two fp32 values of a packed pair (exact widening).
template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t v);
template <>
__device__ __forceinline__ float2 unpack2<PA_BF16>(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}
template <>
__device__ __forceinline__ float2 unpack2<PA_F16>(uint32_t v) {
  __half2 h = *reinterpret_cast<__half2*>(&v);
  return __half22float2(h);
}

// Two FP8 codes (low byte first) -> two f16 in one register, exact (every e4m3 and
// every finite e5m2 value is an f16 value).
template <int DT>
__device__ __forceinline__ uint32_t fp8x2_to_f16x2(uint16_t codes) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(codes),
                                             DT == PA_FP8_E5M2 ? __NV_E5M2 : __NV_E4M3);
  return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// Four FP8 codes (one 32-bit word) -> two f16 pairs: bytes 0, 1 -> lo, bytes 2, 3 ->
// hi; exact.  The word is split into its 16-bit halves by the conversion's operand
// unpack, not by shifts and masks.
template <int DT>
__device__ __forceinline__ void fp8x4_to_f16x2x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  if constexpr (DT == PA_FP8_E5M2)
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "cvt.rn.f16x2.e5m2x2 %0, h0;\n\tcvt.rn.f16x2.e5m2x2 %1, h1;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  else
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, h0;\n\tcvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}

// Eight E2M1 codes (one 32-bit word; byte j holds codes 2j in its low nibble and
// 2j+1 in its high nibble) -> four f16 pairs r[j], exact (every E2M1 value is an
// f16 value).
__device__ __forceinline__ void fp4x8_to_f16x2x4(uint32_t w, uint32_t (&r)[4]) {
  asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
      "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
      : "r"(w));
}

// Elementwise product of two f16 pairs, rounded to nearest.
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 1-D bulk copy global -> shared of `bytes` bytes (a multiple of 16, both addresses
// 16-byte aligned), completion counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// 2^x with the hardware approximation (MUFU); 2^-inf = +0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Online-softmax running max: a block whose max exceeds it by at most this much
// (log2 units) is accumulated against the stale max without rescaling.
constexpr float kRescaleSlack = 8.0f;

__device__ __forceinline__ float warp_max_xor(float v, int lane_mask_lo, int lane_mask_hi) {
  for (int m = lane_mask_lo; m <= lane_mask_hi; m <<= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

__device__ __forceinline__ float warp_sum_xor(float v, int lane_mask_lo, int lane_mask_hi) {
  for (int m = lane_mask_lo; m <= lane_mask_hi; m <<= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

}  // namespace pa

namespace pa {

// Sliding window ([AGENTIC] "為什麼需要「分頁」記憶體管理": only the most recent
// fixed range is attended; blocks that leave it are reclaimed).  A request's
// split-K partitions start at its origin: the block holding the first key its
// first query attends.  Blocks before the origin are never read.
__device__ __forceinline__ int window_origin(const AttnParams& p, int seq_len, int q_len) {
  if (p.window <= 0) return 0;
  const int first = max(0, seq_len - q_len - p.window + 1);
  return first / p.block_size * p.block_size;
}

// Where a query row sits: its request, position, the keys it attends and the
// split-K partitioning of those keys.
struct RowInfo {
  int request;
  int q_len;
  int j;          // row index inside its request
  int seq_len;
  int pos;        // position of the query token: seq_len - q_len + j
  int kv_len;     // keys attended end here: pos + 1 (causal) or seq_len
  int lo;         // first key attended (sliding window), else 0
  int origin;     // first key of the request's partition 0 (block aligned)
  int part;       // partition tokens for this request
  int parts_req;  // partitions covering origin .. seq_len (sizes the request's partial rows)
  int parts_row;  // partitions covering origin .. kv_len (the ones this row uses)
  bool ok;
};

__device__ __forceinline__ RowInfo row_info(const AttnParams& p, int row) {
  RowInfo ri;
  if (p.query_start_loc == nullptr) {
    ri.request = row;
    ri.q_len = 1;
    ri.j = 0;
  } else {
    int lo = 0, hi = p.num_seqs;  // first r with qsl[r+1] > row
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (p.query_start_loc[mid + 1] <= row) lo = mid + 1; else hi = mid;
    }
    ri.request = lo < p.num_seqs ? lo : p.num_seqs - 1;
    const int s = p.query_start_loc[ri.request];
    ri.q_len = p.query_start_loc[ri.request + 1] - s;
    ri.j = row - s;
  }
  ri.seq_len = p.seq_lens[ri.request];
  ri.ok = ri.seq_len >= 1 && ri.seq_len <= p.max_seq_len &&
          (long long)ri.seq_len <= (long long)p.max_blocks_per_seq * p.block_size &&
          ri.q_len >= 1 && ri.q_len <= ri.seq_len && ri.j >= 0 && ri.j < ri.q_len;
  ri.pos = ri.seq_len - ri.q_len + ri.j;
  ri.kv_len = p.causal ? ri.pos + 1 : ri.seq_len;
  ri.lo = p.window > 0 ? max(0, ri.pos - p.window + 1) : 0;
  ri.origin = window_origin(p, ri.seq_len, ri.q_len);
  ri.part = ri.q_len == 1 ? p.part : p.part_pf;
  ri.parts_req = ri.ok ? ceil_div_dev(ri.seq_len - ri.origin, ri.part) : 0;
  ri.parts_row = ri.ok ? ceil_div_dev(ri.kv_len - ri.origin, ri.part) : 0;
  return ri;
}

// Shared-prefix decode.  Group g is the run of sequences group_start[g] ..
// group_start[g+1]-1; its members' block tables agree on their first
// group_shared_blocks[g] entries.  The shared length used is that count clamped so
// every member holds that many full blocks; groups of one sequence, or larger than
// max_group_size, share nothing.
__device__ __forceinline__ int group_shared_tokens(const AttnParams& p, int g, int s0, int s1) {
  if (s0 < 0 || s1 > p.num_seqs || s1 - s0 < 2 || s1 - s0 > p.max_group_size) return 0;
  int sb = p.group_shared_blocks[g];
  for (int m = s0; m < s1; ++m) {
    const int len = p.seq_lens[m];
    // an out-of-range length (flagged by the decode kernel) shares nothing, so no table
    // entry past the row is ever read
    if (len < 1 || len > p.max_seq_len || (long long)len > (long long)p.max_blocks_per_seq * p.block_size)
      return 0;
    sb = min(sb, len / p.block_size);
  }
  return sb > 0 ? sb * p.block_size : 0;
}

// Stages of one declared-shared block.  [AGENTIC] "統一分頁 + 共用池": blocks are
// shared by reference count and copied on write, so a group's declaration can be
// stale (a member already holds a private copy of a block) or simply wrong.  Each
// distinct physical block that the members' entries name for logical block jb gets a
// stage of its own, read only by the members that name it; in the common case every
// member names the first member's block and there is one stage.  A stage record holds
// the reading members in bits 0..7 and kStageLast on the block's last stage.
constexpr int kStageLast = 0x100;
constexpr int kStageMembers = 0xff;

constexpr int kMaxShareMembers = 8;

// The members' block-table entries for logical block jb of the group whose nm
// (<= kMaxShareMembers) members start at sequence s0, loaded together (independent
// loads, issued back to back); -1 past the last member.
__device__ __forceinline__ void load_share_entries(const AttnParams& p, int s0, int nm, int jb,
                                                   int (&e)[kMaxShareMembers]) {
#pragma unroll
  for (int m = 0; m < kMaxShareMembers; ++m)
    e[m] = m < nm ? p.block_tables[(long long)(s0 + m) * p.max_blocks_per_seq + jb] : -1;
}

// The next stage of a block whose members' entries are `e`: the first member not in
// `done` whose entry is a physical block in range, with `mask` the members not in
// `done` that name the same block, and `phys` that block.  Returns that member, or -1
// when every member is done.  Members met with an entry outside [0, num_blocks) join
// `done` without a stage and flag PA_ERRFLAG_BLOCK_TABLE (those tokens are skipped, as
// pa_decode skips them).
__device__ __forceinline__ int next_share_stage(const AttnParams& p, const int (&e)[kMaxShareMembers], int nm,
                                                uint32_t& done, uint32_t& mask, int& phys) {
#pragma unroll
  for (int m = 0; m < kMaxShareMembers; ++m) {
    if (m >= nm || ((done >> m) & 1u)) continue;
    if (e[m] < 0 || e[m] >= p.num_blocks) {
      flag_error(p.err, PA_ERRFLAG_BLOCK_TABLE);
      done |= 1u << m;
      continue;
    }
    uint32_t mk = 0;
#pragma unroll
    for (int m2 = 0; m2 < kMaxShareMembers; ++m2)
      if (m2 >= m && m2 < nm && !((done >> m2) & 1u) && e[m2] == e[m]) mk |= 1u << m2;
    mask = mk;
    phys = e[m];
    return m;
  }
  return -1;
}

// Tokens at the start of sequence `seq` processed by the shared-prefix kernel.
__device__ __forceinline__ int shared_prefix_tokens(const AttnParams& p, int seq) {
  if (p.group_start == nullptr || p.num_groups <= 0) return 0;
  int lo = 0, hi = p.num_groups;  // first g with group_start[g+1] > seq
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (p.group_start[mid + 1] <= seq) lo = mid + 1; else hi = mid;
  }
  if (lo >= p.num_groups) return 0;
  const int s0 = p.group_start[lo], s1 = p.group_start[lo + 1];
  if (seq < s0 || seq >= s1) return 0;
  return group_shared_tokens(p, lo, s0, s1);
}

// Varlen launches do nothing when query_start_loc was found inconsistent (the plan
// kernel has flagged it); this keeps every row and partial index in range.
__device__ __forceinline__ bool plan_rejected(const AttnParams& p) {
  return p.query_start_loc != nullptr && p.plan_ok != nullptr && *p.plan_ok == 0;
}

__device__ __forceinline__ long long row_partial_base(const AttnParams& p, const RowInfo& ri,
                                                      int row) {
  return partial_base(p, ri.request, row, ri.j, ri.parts_req);
}

}  // namespace pa
