// attn_common.cuh -- pieces shared by the dense and the sparse partial-attention
// kernels: work-item arguments, the P^T shared-memory layout, warp
// transpose-reductions, conversions and the elected bounded wait.
//
// Both kernels compute, for each shard row (token g at position t) and head h,
// the partial attention of "[DeepSeekV4][PCP] Enable context-parallel prefill
// for hybrid KV and MegaMoE", "Implementation summary": O and LSE over the
// row's keys, no sink.  Scores use the 576-wide absorbed latent+rope key;
// values are the 512-wide latent ("[Core] Add MRV2 virtual-batch PCP for MLA",
// "DualChunkSwap partitioning": every shard reads the full latent KV).
#pragma once

#include "cpmla_internal.cuh"

namespace cpmla {


constexpr int kTileKeys = 128;                     // keys per KV tile (MMA M)
constexpr int kKbDims = 64;                        // dims per k-block (128 B rows)
constexpr int kLatKb = CPMLA_DV / kKbDims;         // 8 latent k-blocks
constexpr int kKb = CPMLA_DQK / kKbDims;           // 9 k-blocks incl. rope
constexpr int kKbBytes = kTileKeys * kKbDims * 2;  // 16 KB
constexpr int kThreads = 384;
constexpr int kSoftmaxWarp0 = 4;

struct AttnArgs {
  const __nv_bfloat16 *q;
  int64_t q_stride;  // elements between tokens
  int H;
  const __nv_bfloat16 *kv;
  const uint8_t *kv8;
  const float *kv_scale;
  const __nv_bfloat16 *kv_rope;
  int64_t s_kv;
  const int64_t *kv_start;
  const int32_t *rows;
  const int32_t *pos;
  const int32_t *req;
  int n_rows;
  const int32_t *kv_lo;
  const int32_t *kv_hi;
  const int32_t *topk;
  int k;
  // Optional top-k window per shard row (split-KV rows): row i reads entries
  // ent_lo[i] .. ent_lo[i] + ent_len - 1 of its token's list (clipped to k);
  // NULL = the whole list.
  const int32_t *ent_lo;
  int ent_len;
  float scale_log2;  // softmax scale * log2(e)
  float *o_part;
  float *lse_part;
  // Merged output (o_out non-NULL): instead of o_part / lse_part, the owner
  // row of each global token writes its (single) partial merged with the sink
  // straight to the token's place in o_out (bf16) and lse_out.
  __nv_bfloat16 *o_out;
  float *lse_out;
  const float *sink;         // [H] or NULL
  const int32_t *owner_row;  // [T]: the shard row that owns global token g
  int T;
  int hc;         // heads per CTA
  int g;          // tokens per CTA
  int n_hgroups;  // H / hc
  int *status;
};

// The part of its token's top-k list a sparse shard row reads: entries
// [e0, e0 + *len) of the row of global token g.
__device__ __forceinline__ const int32_t *topk_window(const AttnArgs &a, int row, int64_t g,
                                                      int *len) {
  int e0 = 0, n = a.k;
  if (a.ent_lo) {
    e0 = a.ent_lo[row];
    e0 = e0 < 0 ? 0 : (e0 > a.k ? a.k : e0);
    n = a.k - e0 < a.ent_len ? a.k - e0 : a.ent_len;
  }
  *len = n;
  return a.topk + g * a.k + e0;
}

// Sink factor of a merged row with natural-log LSE L: 1 / (1 + e^(sink - L)),
// written as the merge kernel computes it, so that a fused epilogue and the
// partial + merge path give the same bits; 0 for an empty row.
__device__ __forceinline__ float sink_factor(const float *sink, int h, float L) {
  if (L == -INFINITY) return 0.f;
  return sink ? 1.f / (1.f + expf(sink[h] - L)) : 1.f;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// P^T layout for the PV GEMM's B operand: MN-major, N = R rows per key row,
// swizzle width = R*2 bytes (16 rows: 32 B, 32: 64 B, 64: 128 B).
template <int R>
struct PLayout {
  static constexpr uint32_t swz = R == 64 ? kSwz128 : (R == 32 ? kSwz64 : kSwz32);
  static constexpr int row_bytes = R * 2;
  __device__ static __forceinline__ int chunk_xor(int key) {
    return R == 64 ? (key & 7) : (R == 32 ? ((key >> 1) & 3) : ((key >> 2) & 1));
  }
};

// Transpose-reduction of N per-lane values across the 32 lanes of a warp
// (N = 32: afterwards lane l holds row l in v[0]; N = 16: lane l holds row
// l/2).  Each step trades half of the values with the partner lane, so it
// takes N-1 shuffles instead of 5N.
template <int N, bool kMax>
__device__ __forceinline__ void warp_transpose_reduce(float *v, int lane) {
  int n = N;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    if (n > 1) {
      const bool upper = (lane & off) != 0;
      const int h = n >> 1;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < h) {
          const float mine = upper ? v[h + i] : v[i];
          const float give = upper ? v[i] : v[h + i];
          const float got = __shfl_xor_sync(0xffffffffu, give, off);
          v[i] = kMax ? fmaxf(mine, got) : mine + got;
        }
      }
      n = h;
    } else {
      const float got = __shfl_xor_sync(0xffffffffu, v[0], off);
      v[0] = kMax ? fmaxf(v[0], got) : v[0] + got;
    }
  }
}

// e4m3 pair -> two floats (exact), low byte first.
// Two E4M3 codes (low byte -> low half) -> two fp16, exactly: every E4M3
// value, subnormals and NaN included, is an fp16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  return h2;
}

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
  __half2 t = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&t);
}

// Two bf16 (one 32-bit word) -> two fp16, rounded to nearest.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  return pack_f16x2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&t);
}

// Elected bounded wait whose result every thread of a named-barrier group
// sees (so no thread skips a barrier the others enter).
__device__ __forceinline__ bool group_wait(uint64_t *bar, uint32_t parity, int t, int bar_id,
                                           int *flag_pair, int &seq, volatile int *abort,
                                           int *status) {
  int *f = flag_pair + (seq & 1);
  ++seq;
  if (t == 0) *f = mbar_wait(bar, parity, abort, status) ? 1 : 0;
  named_bar_sync(bar_id, 128);
  return *reinterpret_cast<volatile int *>(f) != 0;
}

// Options of attn_entry beyond the public entry points' arguments.
struct AttnExtra {
  const int32_t *ent_lo = nullptr;  // per-row top-k window (sparse)
  int ent_len = 0;
  bool one_row_per_item = false;     // dense: one shard row per work item
  const char *fn = nullptr;          // entry-point name for error messages
};

// Argument checks, work decomposition and launch of the partial-attention
// kernels (attn.cu); the public entry points and the split-KV path call it.
int attn_entry(bool sparse, const void *q, int64_t q_token_stride, int H, int kv_format,
               const void *kv, const void *kv_fp8, const float *kv_scale, const void *kv_rope,
               int64_t s_kv, const int64_t *kv_start, const int32_t *rows, const int32_t *pos,
               const int32_t *req, int n_rows, const int32_t *kv_lo, const int32_t *kv_hi,
               const int32_t *topk, int k, float softmax_scale, float *o_part, float *lse_part,
               const int32_t *owner_row, int T, const float *sink, void *o_out, float *lse_out,
               void *stream, const AttnExtra &extra);

// The merge of merge.cu for a list of tokens: merged row i (partials
// contrib_off[i] .. contrib_off[i+1]-1) is written to token out_tok[i] of
// o_out / lse_out (T_out tokens).
int launch_merge_to_tokens(const float *o_part, const float *lse_part, int64_t n_part, int H,
                           const int32_t *contrib_off, const int32_t *contrib_rows, int n,
                           const float *sink, void *o_out, float *lse_out,
                           const int32_t *out_tok, int T_out, int *status, cudaStream_t st);

// Launchers (one per translation unit); n_items CTAs, one work item each.
// Dense: tm_q = Q as [T, H, 576] in boxes of 64 dims x hc heads x 1 token
// (used when hc is a multiple of 8).
int launch_dense(const AttnArgs &args, const CUtensorMap &tm_kv, const CUtensorMap &tm_q,
                 int n_items, cudaStream_t st);
// Sparse (attn_sparse_wide.cu): bf16 KV with R = 16, 32 or 64 heads per CTA,
// or fp8 KV with R = 16.  One-row gather maps: bf16: tm_kv = tm_rope = the
// KV (box 64 x 1, 128-byte swizzle); fp8: tm_kv = the E4M3 codes (box 128 x
// 1, no swizzle), tm_rope = the bf16 rope (box 64 x 1, 128-byte swizzle).
// bf16: tm_q = Q as [T, H, 576] in boxes of 64 dims x R heads x 1 token,
// 128-byte swizzle (fp8 reads Q with plain loads; tm_q unused).
int launch_sparse_wide(bool fp8, int R, const AttnArgs &args, const CUtensorMap &tm_kv,
                       const CUtensorMap &tm_q, const CUtensorMap &tm_rope, int n_items,
                       cudaStream_t st);

}  // namespace cpmla
