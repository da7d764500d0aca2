// merge.cu -- global LSE merge of partial MLA attention results, attention sink
// applied once, output restored to global token order.
//
// "[DeepSeekV4][PCP] Enable context-parallel prefill for hybrid KV and
// MegaMoE", "Implementation summary": the PCP ranks' partial (output, LSE) are
// merged globally by LSE and attn_sink is applied only once; "Main
// challenges": it must not be applied per rank.  "[Core] Add MRV2
// virtual-batch PCP for MLA", "DualChunkSwap partitioning": results return to
// global scheduled-token order.  The sink is one extra logit per head with a
// zero value vector, so after the merge O is scaled by 1 / (1 + e^(sink - L)).
//
// The kernel is bandwidth-bound: per (token, head) it reads 2 KB of fp32
// partial output per contributing partial plus one LSE, and writes 1 KB of
// bf16 plus one LSE.  One warp owns one (token, head) row; each lane moves four
// 16-byte vectors so that every warp access is one contiguous 512 B (load) or
// 256 B (store) span.
#include <cmath>

#include "cpmla_internal.cuh"

namespace cpmla {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kVecPerLane = CPMLA_DV / (32 * 4);  // 4 float4 per lane

__device__ __forceinline__ float4 ld_stream(const float4 *p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_stream_bf16x4(void *p, float a, float b, float c, float d) {
  __nv_bfloat162 lo = __floats2bfloat162_rn(a, b);
  __nv_bfloat162 hi = __floats2bfloat162_rn(c, d);
  uint32_t ulo = *reinterpret_cast<uint32_t *>(&lo);
  uint32_t uhi = *reinterpret_cast<uint32_t *>(&hi);
  asm volatile("st.global.cs.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(ulo), "r"(uhi) : "memory");
}

__global__ void __launch_bounds__(kMergeThreads)
    lse_merge_kernel(const float *__restrict__ o_part, const float *__restrict__ lse_part,
                     int64_t n_part, int H, const int32_t *__restrict__ contrib_off,
                     const int32_t *__restrict__ contrib_rows, int T,
                     const float *__restrict__ sink, __nv_bfloat16 *__restrict__ o_out,
                     float *__restrict__ lse_out, const int32_t *__restrict__ out_tok,
                     int T_out, int *status) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * (kMergeThreads / 32) + (threadIdx.x >> 5);
  const int64_t n_warps = (int64_t)gridDim.x * (kMergeThreads / 32);
  const int64_t total = (int64_t)T * H;
  for (int64_t gh = warp; gh < total; gh += n_warps) {
    const int64_t g = gh / H;
    const int h = (int)(gh - g * H);
    // where merged row g goes: itself, or token out_tok[g] (a list of tokens)
    int64_t go = g;
    if (out_tok) {
      go = out_tok[g];
      if (go < 0 || go >= T_out) {
        if (lane == 0) record_status(status, CPMLA_ERR_INDEX);
        continue;
      }
    }
    int c0, c1;
    if (contrib_off) {
      c0 = contrib_off[g];
      c1 = contrib_off[g + 1];
    } else {
      c0 = (int)g;
      c1 = (int)g + 1;
    }
    float acc[kVecPerLane * 4];
#pragma unroll
    for (int i = 0; i < kVecPerLane * 4; ++i) acc[i] = 0.f;
    // L = max + ln sum exp(lse_c - max) over the valid partials; a contrib
    // row outside [0, n_part) is skipped and recorded here, before anything
    // else depends on it (also when it is the token's only partial)
    float mx = -INFINITY;
    for (int c = c0; c < c1; ++c) {
      const int r = contrib_rows[c];
      if (r < 0 || (int64_t)r >= n_part) {
        if (lane == 0) record_status(status, CPMLA_ERR_INDEX);
        continue;
      }
      mx = fmaxf(mx, lse_part[(int64_t)r * H + h]);
    }
    float L = -INFINITY;
    if (mx != -INFINITY) {
      float z = 0.f;
      for (int c = c0; c < c1; ++c) {
        const int r = contrib_rows[c];
        if (r < 0 || (int64_t)r >= n_part) continue;
        z += expf(lse_part[(int64_t)r * H + h] - mx);
      }
      L = mx + logf(z);
      for (int c = c0; c < c1; ++c) {
        const int r = contrib_rows[c];
        if (r < 0 || (int64_t)r >= n_part) continue;
        const float l = lse_part[(int64_t)r * H + h];
        if (l == -INFINITY) continue;
        const float w = expf(l - L);
        const float4 *src =
            reinterpret_cast<const float4 *>(o_part + ((int64_t)r * H + h) * CPMLA_DV);
#pragma unroll
        for (int i = 0; i < kVecPerLane; ++i) {
          const float4 v = ld_stream(src + lane + 32 * i);
          acc[4 * i + 0] += w * v.x;
          acc[4 * i + 1] += w * v.y;
          acc[4 * i + 2] += w * v.z;
          acc[4 * i + 3] += w * v.w;
        }
      }
      // the sink, once, after the merge
      if (sink) {
        const float f = 1.f / (1.f + expf(sink[h] - L));
#pragma unroll
        for (int i = 0; i < kVecPerLane * 4; ++i) acc[i] *= f;
      }
    }
    __nv_bfloat16 *dst = o_out + (go * H + h) * CPMLA_DV;
#pragma unroll
    for (int i = 0; i < kVecPerLane; ++i)
      st_stream_bf16x4(dst + 4 * (lane + 32 * i), acc[4 * i], acc[4 * i + 1], acc[4 * i + 2],
                       acc[4 * i + 3]);
    if (lane == 0) lse_out[go * H + h] = L;
  }
}

}  // namespace
}  // namespace cpmla

extern "C" int lse_merge_with_sink(const float *o_part, const float *lse_part, int64_t n_part,
                                   int H, const int32_t *contrib_off,
                                   const int32_t *contrib_rows, int T, const float *sink,
                                   void *o_out, float *lse_out, void *stream) {
  using namespace cpmla;
  CPMLA_CHECK_ARG(T >= 0 && n_part >= 0, "lse_merge_with_sink: negative size");
  CPMLA_CHECK_ARG(H >= 1 && H <= 1024, "lse_merge_with_sink: H=%d outside 1..1024", H);
  if (T == 0) return CPMLA_OK;
  CPMLA_CHECK_ARG(contrib_rows && o_out && lse_out,
                  "lse_merge_with_sink: contrib_rows/o_out/lse_out is NULL");
  CPMLA_CHECK_ARG(n_part == 0 || (o_part && lse_part),
                  "lse_merge_with_sink: o_part/lse_part is NULL");
  CPMLA_CHECK_ARG(((uintptr_t)o_part & 15) == 0 && ((uintptr_t)o_out & 15) == 0,
                  "lse_merge_with_sink: o_part and o_out must be 16-byte aligned");
  int *status = status_word();
  if (!status) return fail(CPMLA_ERR_CUDA, "lse_merge_with_sink: status word unavailable");
  int dev = 0, n_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const int64_t rows = (int64_t)T * H;
  const int64_t want = (rows + (kMergeThreads / 32) - 1) / (kMergeThreads / 32);
  // 8 resident CTAs of 256 threads per SM keep enough 16-byte loads in flight
  const int64_t cap = (int64_t)(n_sm > 0 ? n_sm : 152) * 8;
  const int grid = (int)(want < cap ? want : cap);
  lse_merge_kernel<<<grid, kMergeThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      o_part, lse_part, n_part, H, contrib_off, contrib_rows, T, sink,
      static_cast<__nv_bfloat16 *>(o_out), lse_out, nullptr, T, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "lse_merge_with_sink: launch");
  return CPMLA_OK;
}

namespace cpmla {
// The merge for a list of tokens: merged row i (partials contrib_off[i] ..
// contrib_off[i+1]-1) goes to token out_tok[i] of o_out / lse_out [T_out].
int launch_merge_to_tokens(const float *o_part, const float *lse_part, int64_t n_part, int H,
                           const int32_t *contrib_off, const int32_t *contrib_rows, int n,
                           const float *sink, void *o_out, float *lse_out,
                           const int32_t *out_tok, int T_out, int *status, cudaStream_t st) {
  int dev = 0, n_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const int64_t rows = (int64_t)n * H;
  const int64_t want = (rows + (kMergeThreads / 32) - 1) / (kMergeThreads / 32);
  const int64_t cap = (int64_t)(n_sm > 0 ? n_sm : 152) * 8;
  const int grid = (int)(want < cap ? want : cap);
  if (grid <= 0) return CPMLA_OK;
  lse_merge_kernel<<<grid, kMergeThreads, 0, st>>>(o_part, lse_part, n_part, H, contrib_off,
                                                   contrib_rows, n, sink,
                                                   static_cast<__nv_bfloat16 *>(o_out), lse_out,
                                                   out_tok, T_out, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "split-KV merge: launch");
  return CPMLA_OK;
}
}  // namespace cpmla
