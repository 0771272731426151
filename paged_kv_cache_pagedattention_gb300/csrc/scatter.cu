// reshape_and_cache: write each new token's K and V rows into its slot of the
// paged cache.  [NOTES] "Prefill 与 Decode" (prefill stores every prompt token's
// K/V, decode appends the new token's); [ARCH] Part 1, forward pass (slot_mapping
// built during input preparation).  Slot s -> block s / block_size, offset
// s % block_size; negative slots are padding.
//
// One thread moves one 16-byte piece of a destination row (same dtype: a straight
// copy of 16 bytes; FP8: 16 codes quantised from 16 source elements; NVFP4: 16
// elements into 8 code bytes and one block-scale byte).  Threads of a warp cover
// consecutive pieces of consecutive rows, so the source reads and the destination
// writes are coalesced.
#include "pa_common.cuh"

namespace pa {

namespace {

__global__ void __launch_bounds__(256) scatter_copy_kernel(const ScatterParams p, int elem_bytes) {
  const int pieces = p.head_size * elem_bytes / 16;  // per (token, head) row
  const long long per_token = (long long)p.num_kv_heads * pieces;
  const long long total = (long long)p.num_tokens * per_token;
  const long long limit = (long long)p.num_blocks * p.block_size;
  for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < total;
       u += (long long)gridDim.x * blockDim.x) {
    const long long t = u / per_token;
    const int rem = static_cast<int>(u - t * per_token);
    const int h = rem / pieces, c = rem % pieces;
    // the source pieces do not depend on the slot: their loads go out with the slot's
    const long long src = (t * p.num_kv_heads + h) * pieces + c;
    const uint4 kv = reinterpret_cast<const uint4*>(p.key)[src];
    const uint4 vv = reinterpret_cast<const uint4*>(p.value)[src];
    const long long slot = p.slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= limit) {
      flag_error(p.err, PA_ERRFLAG_SLOT);
      continue;
    }
    const long long blk = slot / p.block_size, off = slot % p.block_size;
    const long long dst = ((blk * p.num_kv_heads + h) * p.block_size + off) * pieces + c;
    reinterpret_cast<uint4*>(p.k_cache)[dst] = kv;
    reinterpret_cast<uint4*>(p.v_cache)[dst] = vv;
  }
}

// x / scale in IEEE fp32 (correctly rounded division), then FP8 (e4m3 or e5m2)
// round-to-nearest-even with saturation to the largest finite value, via the CUDA
// conversion intrinsic.
template <int CDT>
__device__ __forceinline__ uint8_t quant_fp8(float x, float scale) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x, scale), __NV_SATFINITE,
                                                    CDT == PA_FP8_E5M2 ? __NV_E5M2 : __NV_E4M3));
}

template <int SRC, int CDT>
__global__ void __launch_bounds__(256) scatter_fp8_kernel(const ScatterParams p) {
  using SE = Elem<SRC>;
  const int pieces = p.head_size / 16;  // 16 codes per piece
  const long long per_token = (long long)p.num_kv_heads * pieces;
  const long long total = (long long)p.num_tokens * per_token;
  const long long limit = (long long)p.num_blocks * p.block_size;
  for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < total;
       u += (long long)gridDim.x * blockDim.x) {
    const long long t = u / per_token;
    const int rem = static_cast<int>(u - t * per_token);
    const int h = rem / pieces, c = rem % pieces;
    // the codes do not depend on the slot: their loads go out with the slot's
    const long long slot = p.slot_mapping[t];
    const float ks = p.k_scale[h * p.scale_stride], vs = p.v_scale[h * p.scale_stride];
    const long long src = ((t * p.num_kv_heads + h) * p.head_size) + c * 16;
    const typename SE::T* ksrc = reinterpret_cast<const typename SE::T*>(p.key) + src;
    const typename SE::T* vsrc = reinterpret_cast<const typename SE::T*>(p.value) + src;
    uint32_t kw[4], vw[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      uint32_t kb = 0, vb = 0;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        kb |= static_cast<uint32_t>(quant_fp8<CDT>(SE::load(ksrc + 4 * w + b), ks)) << (8 * b);
        vb |= static_cast<uint32_t>(quant_fp8<CDT>(SE::load(vsrc + 4 * w + b), vs)) << (8 * b);
      }
      kw[w] = kb;
      vw[w] = vb;
    }
    if (slot < 0) continue;
    if (slot >= limit) {
      flag_error(p.err, PA_ERRFLAG_SLOT);
      continue;
    }
    const long long blk = slot / p.block_size, off = slot % p.block_size;
    const long long dst = ((blk * p.num_kv_heads + h) * p.block_size + off) * p.head_size + c * 16;
    reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.k_cache) + dst)[0] = make_uint4(kw[0], kw[1], kw[2], kw[3]);
    reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.v_cache) + dst)[0] = make_uint4(vw[0], vw[1], vw[2], vw[3]);
  }
}

// E2M1 code of y: round to nearest with ties to the even code, saturating at 6,
// sign kept.  The magnitude code counts the midpoints between neighbouring E2M1
// magnitudes (0, 0.5, 1, 1.5, 2, 3, 4, 6) that |y| lies above; at a midpoint the
// comparison is strict or not so that the tie lands on the even code.
__device__ __forceinline__ uint32_t e2m1_code(float y) {
  const float a = fabsf(y);
  const uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) + (a >= 3.5f) +
                     (a > 5.0f);
  return c | (signbit(y) ? 8u : 0u);
}

// NVFP4 quantisation of one group of 16 source elements with fp32 scale s: block
// scale code e4m3(amax / (6 s)), codes e2m1(x / (s b)) packed low nibble first;
// zero codes when the block scale is zero.
template <int SRC>
__device__ __forceinline__ void quant_nvfp4_group(const typename Elem<SRC>::T* src, float s, uint2& codes,
                                                  uint8_t& scale) {
  float x[16];
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    x[i] = Elem<SRC>::load(src + i);
    amax = fmaxf(amax, fabsf(x[i]));
  }
  const float q = __fdiv_rn(amax, __fmul_rn(6.0f, s));
  scale = static_cast<uint8_t>(__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3));
  const float b = __half2float(__half(__nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(scale), __NV_E4M3)));
  uint32_t w[2] = {0u, 0u};
  if (b != 0.f) {
    const float den = __fmul_rn(s, b);
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i >> 3] |= e2m1_code(__fdiv_rn(x[i], den)) << (4 * (i & 7));
  }
  codes = make_uint2(w[0], w[1]);
}

// One thread per group of 16 elements of a (token, head) row, K and V; consecutive
// threads cover consecutive groups of a row, so the 8-byte code stores and the
// scale bytes of a row are written side by side.
template <int SRC>
__global__ void __launch_bounds__(256) scatter_nvfp4_kernel(const ScatterParams p) {
  using SE = Elem<SRC>;
  const int d = p.head_size, bs = p.block_size;
  const int groups = d / 16;
  const long long per_token = (long long)p.num_kv_heads * groups;
  const long long total = (long long)p.num_tokens * per_token;
  const long long limit = (long long)p.num_blocks * bs;
  const long long tile = nvfp4_tile_bytes(bs, d);
  for (long long u = (long long)blockIdx.x * blockDim.x + threadIdx.x; u < total;
       u += (long long)gridDim.x * blockDim.x) {
    const long long t = u / per_token;
    const int rem = static_cast<int>(u - t * per_token);
    const int h = rem / groups, g = rem % groups;
    // the codes do not depend on the slot: their loads go out with the slot's
    const long long slot = p.slot_mapping[t];
    const long long src = (t * p.num_kv_heads + h) * d + g * 16;
    uint2 kcodes, vcodes;
    uint8_t ksc, vsc;
    quant_nvfp4_group<SRC>(reinterpret_cast<const typename SE::T*>(p.key) + src, p.k_scale[h * p.scale_stride],
                           kcodes, ksc);
    quant_nvfp4_group<SRC>(reinterpret_cast<const typename SE::T*>(p.value) + src, p.v_scale[h * p.scale_stride],
                           vcodes, vsc);
    if (slot < 0) continue;
    if (slot >= limit) {
      flag_error(p.err, PA_ERRFLAG_SLOT);
      continue;
    }
    const long long blk = slot / bs;
    const int off = static_cast<int>(slot % bs);
    const long long tbase = (blk * p.num_kv_heads + h) * tile;
    const long long code_at = tbase + off * (d / 2) + g * 8;
    const long long scale_at = tbase + (long long)bs * (d / 2) + off * (d / 16) + g;
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.k_cache) + code_at) = kcodes;
    static_cast<uint8_t*>(p.k_cache)[scale_at] = ksc;
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.v_cache) + code_at) = vcodes;
    static_cast<uint8_t*>(p.v_cache)[scale_at] = vsc;
  }
}

int scatter_grid(long long units) {
  long long blocks = (units + 255) / 256;
  if (blocks > 152LL * 64) blocks = 152LL * 64;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t launch_reshape_and_cache(const ScatterParams& p, int src_dtype, int cache_dtype,
                                     cudaStream_t stream) {
  if (p.num_tokens == 0) return cudaSuccess;
  if (src_dtype == cache_dtype) {
    const int eb = src_dtype == PA_F32 ? 4 : (src_dtype == PA_F16 || src_dtype == PA_BF16 ? 2 : 1);
    const long long units = (long long)p.num_tokens * p.num_kv_heads * (p.head_size * eb / 16);
    scatter_copy_kernel<<<scatter_grid(units), 256, 0, stream>>>(p, eb);
    return cudaGetLastError();
  }
  if (cache_dtype == PA_NVFP4) {
    const long long units = (long long)p.num_tokens * p.num_kv_heads * (p.head_size / 16);
    const int g = scatter_grid(units);
    if (src_dtype == PA_F32) scatter_nvfp4_kernel<PA_F32><<<g, 256, 0, stream>>>(p);
    else if (src_dtype == PA_F16) scatter_nvfp4_kernel<PA_F16><<<g, 256, 0, stream>>>(p);
    else if (src_dtype == PA_BF16) scatter_nvfp4_kernel<PA_BF16><<<g, 256, 0, stream>>>(p);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
  }
  if (cache_dtype != PA_FP8_E4M3 && cache_dtype != PA_FP8_E5M2) return cudaErrorInvalidValue;
  const long long units = (long long)p.num_tokens * p.num_kv_heads * (p.head_size / 16);
  const int g = scatter_grid(units);
  const bool e5 = cache_dtype == PA_FP8_E5M2;
#define PA_Q(S) \
  e5 ? (scatter_fp8_kernel<S, PA_FP8_E5M2><<<g, 256, 0, stream>>>(p), 0) \
     : (scatter_fp8_kernel<S, PA_FP8_E4M3><<<g, 256, 0, stream>>>(p), 0)
  if (src_dtype == PA_F32) PA_Q(PA_F32);
  else if (src_dtype == PA_F16) PA_Q(PA_F16);
  else if (src_dtype == PA_BF16) PA_Q(PA_BF16);
  else return cudaErrorInvalidValue;
#undef PA_Q
  return cudaGetLastError();
}

}  // namespace pa
