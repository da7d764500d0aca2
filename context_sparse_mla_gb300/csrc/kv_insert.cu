// kv_insert.cu -- latent KV-cache insertion: each token's all-gathered latent
// KV row (bf16, 512 latent + 64 rope) written to its cache slot, as bf16 or as
// the fp8 layout the sparse attention reads (E4M3 latent with one fp32 scale
// per 128-channel group, bf16 rope).
//
// "[Core] Add MRV2 virtual-batch PCP for MLA", Summary (sparse MLA cache
// insertion) and "DualChunkSwap partitioning" (the all-gathered latent KV is
// what the insertion writes); the fp8_ds_mla cache dtype of "[Feature][PCP]
// Add DeepSeek-V4.1-Flash support".  The quantisation rule is the library's
// own: per group, scale = amax / 448 in binary32 (1 for an all-zero group),
// code = E4M3(x / scale) with the quotient in binary32, rounded to nearest
// even, saturating at +-448.
//
// HBM-bound: per token 1152 B read, 576 x 2 B (bf16) or 512 + 16 + 128 B
// (fp8) written.  A warp takes two tokens at a time, all their loads in
// flight before the first store; per token, lane l moves latent 16-byte
// chunks l and l + 32 (each warp access one contiguous 512 B span), lanes 0-7
// the rope; the 16 chunks of a 128-channel group sit in one half-warp, whose
// shuffle reduction gives the group's amax.
#include <cmath>

#include "cpmla_internal.cuh"

namespace cpmla {
namespace {

constexpr int kInsThreads = 128;

// two binary32 -> two E4M3 codes (lo in the low byte), round to nearest
// even, saturating to +-448 (NaN stays NaN)
__device__ __forceinline__ uint16_t e4m3x2_rn_sat(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// x / b rounded to nearest even in binary32, from y = RN(1/b): q0 = RN(x y)
// lies within one ulp of x / b, so the remainder x - b q0 is exact in one FMA
// and RN(q0 + r y) = RN(x / b) -- Markstein's correction step of division by
// a correctly rounded reciprocal (Markstein 1990; Muller et al., "Handbook of
// Floating-Point Arithmetic", the FMA-based division chapter).  It holds while
// b and 1/b are normal and finite; the quotients that fall below the normal
// range are below 2^-126, where every E4M3 code is a zero, so the codes match
// those of the exact quotient there too.
__device__ __forceinline__ float div_by_recip(float x, float b, float y) {
  const float q0 = __fmul_rn(x, y);
  const float r = __fmaf_rn(-q0, b, x);
  return __fmaf_rn(r, y, q0);
}

__device__ __forceinline__ void bf16x8_to_float(const uint4 &v, float *x) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// tokens whose loads a warp has in flight at once: two, with one pass of
// 128-thread blocks over the tokens (measured on the 131072-token insertion:
// 0.0452 ms at two, 0.0503 at four, 0.0514 at one; 256-thread blocks and
// grids capped at 8-16 blocks per SM were slower)
constexpr int kTokPerWarp = 2;

__global__ void __launch_bounds__(kInsThreads)
    kv_insert_kernel(const __nv_bfloat16 *__restrict__ kv, int64_t kv_stride, int n,
                     const int64_t *__restrict__ slot, int fmt, __nv_bfloat16 *__restrict__ cache,
                     uint8_t *__restrict__ cache_fp8, float *__restrict__ cache_scale,
                     __nv_bfloat16 *__restrict__ cache_rope, int64_t s_cache, int *status) {
  const int lane = threadIdx.x & 31;
  const int64_t n_warps = (int64_t)gridDim.x * (kInsThreads / 32);
  for (int64_t t0 = ((int64_t)blockIdx.x * (kInsThreads / 32) + (threadIdx.x >> 5)) * kTokPerWarp;
       t0 < n; t0 += n_warps * kTokPerWarp) {
    // every load of the warp's tokens first (the insertion is bound by how
    // many bytes each SM has in flight), then each token's stores
    uint4 c0[kTokPerWarp], c1[kTokPerWarp], rope[kTokPerWarp];
    int64_t s[kTokPerWarp];
#pragma unroll
    for (int u = 0; u < kTokPerWarp; ++u) {
      const int64_t t = t0 + u;
      s[u] = -1;
      c0[u] = c1[u] = rope[u] = make_uint4(0, 0, 0, 0);
      if (t < n) {
        const uint4 *src = reinterpret_cast<const uint4 *>(kv + t * kv_stride);
        c0[u] = __ldg(src + lane);       // latent chunk lane (group lane / 16)
        c1[u] = __ldg(src + lane + 32);  // latent chunk lane + 32 (group 2 + lane / 16)
        if (lane < 8) rope[u] = __ldg(src + 64 + lane);
        s[u] = slot[t];
      }
    }
#pragma unroll
    for (int u = 0; u < kTokPerWarp; ++u) {
      const int64_t su = s[u];
      if (su < 0) continue;
      if (su >= s_cache) {
        if (lane == 0) record_status(status, CPMLA_ERR_INDEX);
        continue;
      }
      if (fmt == CPMLA_KV_BF16) {
        uint4 *dst = reinterpret_cast<uint4 *>(cache + su * CPMLA_DQK);
        dst[lane] = c0[u];
        dst[lane + 32] = c1[u];
        if (lane < 8) dst[64 + lane] = rope[u];
        continue;
      }
      uint2 codes[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        float x[8];
        bf16x8_to_float(k == 0 ? c0[u] : c1[u], x);
        float amax = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1)
          amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));  // within the half-warp
        const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
        uint32_t p[4];
        if (scale >= 1.17549435e-38f && scale <= 3.40282347e38f) {
          // one correctly rounded reciprocal per group, three operations a code
          const float y = __frcp_rn(scale);
#pragma unroll
          for (int i = 0; i < 4; ++i)
            p[i] = e4m3x2_rn_sat(div_by_recip(x[2 * i], scale, y),
                                 div_by_recip(x[2 * i + 1], scale, y));
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i)
            p[i] = e4m3x2_rn_sat(__fdiv_rn(x[2 * i], scale), __fdiv_rn(x[2 * i + 1], scale));
        }
        codes[k] = make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
        if ((lane & 15) == 0) cache_scale[su * 4 + 2 * k + (lane >> 4)] = scale;
      }
      uint2 *dst8 = reinterpret_cast<uint2 *>(cache_fp8 + su * CPMLA_DV);
      dst8[lane] = codes[0];
      dst8[lane + 32] = codes[1];
      if (lane < 8) reinterpret_cast<uint4 *>(cache_rope + su * CPMLA_DROPE)[lane] = rope[u];
    }
  }
}

}  // namespace
}  // namespace cpmla

extern "C" int mla_kv_cache_insert(const void *kv, int64_t kv_token_stride, int n,
                                   const int64_t *slot_mapping, int kv_format, void *cache,
                                   void *cache_fp8, float *cache_scale, void *cache_rope,
                                   int64_t s_cache, void *stream) {
  using namespace cpmla;
  const char *fn = "mla_kv_cache_insert";
  CPMLA_CHECK_ARG(n >= 0, "%s: n=%d < 0", fn, n);
  CPMLA_CHECK_ARG(kv_format == CPMLA_KV_BF16 || kv_format == CPMLA_KV_FP8_E4M3_G128,
                  "%s: unknown kv_format %d", fn, kv_format);
  CPMLA_CHECK_ARG(kv_token_stride >= CPMLA_DQK && kv_token_stride % 8 == 0,
                  "%s: kv_token_stride=%lld must be >= 576 and a multiple of 8", fn,
                  (long long)kv_token_stride);
  CPMLA_CHECK_ARG(s_cache >= 1, "%s: s_cache=%lld < 1", fn, (long long)s_cache);
  if (n == 0) return CPMLA_OK;
  CPMLA_CHECK_ARG(kv && slot_mapping, "%s: kv and slot_mapping are required", fn);
  CPMLA_CHECK_ARG(((uintptr_t)kv & 15) == 0, "%s: kv must be 16-byte aligned", fn);
  if (kv_format == CPMLA_KV_BF16) {
    CPMLA_CHECK_ARG(cache && ((uintptr_t)cache & 15) == 0,
                    "%s: cache must be non-NULL and 16-byte aligned", fn);
  } else {
    CPMLA_CHECK_ARG(cache_fp8 && cache_scale && cache_rope,
                    "%s: the fp8 cache needs cache_fp8, cache_scale and cache_rope", fn);
    CPMLA_CHECK_ARG(((uintptr_t)cache_fp8 & 15) == 0 && ((uintptr_t)cache_rope & 15) == 0 &&
                        ((uintptr_t)cache_scale & 3) == 0,
                    "%s: cache_fp8 and cache_rope must be 16-byte aligned", fn);
  }
  int *status = status_word();
  if (!status) return fail(CPMLA_ERR_CUDA, "%s: status word unavailable", fn);
  const int64_t per_block = (kInsThreads / 32) * kTokPerWarp;  // tokens per block
  const int64_t grid = ((int64_t)n + per_block - 1) / per_block;
  kv_insert_kernel<<<(unsigned)grid, kInsThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const __nv_bfloat16 *>(kv), kv_token_stride, n, slot_mapping, kv_format,
      static_cast<__nv_bfloat16 *>(cache), static_cast<uint8_t *>(cache_fp8), cache_scale,
      static_cast<__nv_bfloat16 *>(cache_rope), s_cache, status);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "mla_kv_cache_insert: launch");
  return CPMLA_OK;
}
