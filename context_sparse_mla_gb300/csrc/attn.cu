// attn.cu -- C-ABI entry points of the partial-attention kernels: argument
// checks, work decomposition and launch.
//
// mla_partial_attn_dense / mla_partial_attn_sparse compute, for every shard
// row of all P virtual shards in one launch, the partial attention of
// "[DeepSeekV4][PCP] Enable context-parallel prefill for hybrid KV and
// MegaMoE", "Implementation summary" (O and LSE over the row's keys, no sink),
// over the full latent KV ("[Core] Add MRV2 virtual-batch PCP for MLA",
// "DualChunkSwap partitioning").  mla_attn_dense_merged /
// mla_attn_sparse_merged run the same kernels with the merge folded into
// their epilogue for the query-partitioned case, where every token has one
// partial: its owner row applies the sink once and writes bf16 O and the LSE
// in global token order, the merge kernel's arithmetic for one partial.  The
// kernels live in attn_dense.cu and attn_sparse_wide.cu.
#include <cmath>
#include <cstring>
#include <mutex>

#include "attn_common.cuh"

namespace cpmla {
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

int attn_entry(bool sparse, const void *q, int64_t q_token_stride, int H, int kv_format,
               const void *kv, const void *kv_fp8, const float *kv_scale, const void *kv_rope,
               int64_t s_kv, const int64_t *kv_start, const int32_t *rows, const int32_t *pos,
               const int32_t *req, int n_rows, const int32_t *kv_lo, const int32_t *kv_hi,
               const int32_t *topk, int k, float softmax_scale, float *o_part, float *lse_part,
               const int32_t *owner_row, int T, const float *sink, void *o_out, float *lse_out,
               void *stream, const AttnExtra &extra) {
  const bool merged = o_out != nullptr;
  const char *fn = extra.fn ? extra.fn
                   : merged ? (sparse ? "mla_attn_sparse_merged" : "mla_attn_dense_merged")
                            : (sparse ? "mla_partial_attn_sparse" : "mla_partial_attn_dense");
  CPMLA_CHECK_ARG(n_rows >= 0, "%s: n_rows=%d < 0", fn, n_rows);
  CPMLA_CHECK_ARG(H >= 1 && H <= 128 && (H <= 64 || H % 64 == 0),
                  "%s: H=%d unsupported (1..64, or a multiple of 64 up to 128)", fn, H);
  CPMLA_CHECK_ARG(kv_format == CPMLA_KV_BF16 || kv_format == CPMLA_KV_FP8_E4M3_G128,
                  "%s: unknown kv_format %d", fn, kv_format);
  if (!sparse && kv_format != CPMLA_KV_BF16)
    return fail(CPMLA_ERR_UNSUPPORTED, "%s: dense attention takes CPMLA_KV_BF16 only", fn);
  if (sparse && kv_format == CPMLA_KV_FP8_E4M3_G128 && H > 16 && H % 16 != 0)
    return fail(CPMLA_ERR_UNSUPPORTED,
                "%s: H=%d over the fp8 cache must be at most 16 or a multiple of 16", fn, H);
  CPMLA_CHECK_ARG(std::isfinite(softmax_scale) && softmax_scale > 0.f, "%s: bad softmax_scale",
                  fn);
  CPMLA_CHECK_ARG(q_token_stride >= (int64_t)H * CPMLA_DQK && q_token_stride % 8 == 0,
                  "%s: q_token_stride=%lld must be >= H*576 and a multiple of 8", fn,
                  (long long)q_token_stride);
  CPMLA_CHECK_ARG(s_kv >= 1 && s_kv <= INT32_MAX, "%s: s_kv=%lld outside 1..2^31-1", fn,
                  (long long)s_kv);
  if (sparse) CPMLA_CHECK_ARG(k >= 1 && k <= 65536, "%s: k=%d outside 1..65536", fn, k);
  if (merged) CPMLA_CHECK_ARG(T >= 0, "%s: T=%d < 0", fn, T);
  if (n_rows == 0) return CPMLA_OK;
  CPMLA_CHECK_ARG(q && kv_start && rows && pos && req, "%s: a required pointer is NULL", fn);
  if (merged) {
    CPMLA_CHECK_ARG(owner_row && lse_out, "%s: owner_row, o_out and lse_out are required", fn);
    CPMLA_CHECK_ARG(((uintptr_t)o_out & 15) == 0, "%s: o_out must be 16-byte aligned", fn);
  }
  else
    CPMLA_CHECK_ARG(o_part && lse_part, "%s: o_part and lse_part are required", fn);
  CPMLA_CHECK_ARG(((uintptr_t)q & 15) == 0, "%s: q must be 16-byte aligned", fn);
  if (kv_format == CPMLA_KV_BF16) {
    CPMLA_CHECK_ARG(kv != nullptr && ((uintptr_t)kv & 15) == 0,
                    "%s: kv must be non-NULL and 16-byte aligned", fn);
  } else {
    CPMLA_CHECK_ARG(kv_fp8 && kv_scale && kv_rope, "%s: fp8 KV needs kv_fp8, kv_scale, kv_rope",
                    fn);
    CPMLA_CHECK_ARG(((uintptr_t)kv_fp8 & 15) == 0 && ((uintptr_t)kv_rope & 15) == 0 &&
                        ((uintptr_t)kv_scale & 15) == 0,
                    "%s: kv_fp8, kv_scale and kv_rope must be 16-byte aligned", fn);
  }
  if (sparse) CPMLA_CHECK_ARG(topk != nullptr, "%s: topk_idx is NULL", fn);
  int *status = status_word();
  if (!status) return fail(CPMLA_ERR_CUDA, "%s: status word unavailable", fn);

  AttnArgs args{};
  args.q = static_cast<const __nv_bfloat16 *>(q);
  args.q_stride = q_token_stride;
  args.H = H;
  args.kv = static_cast<const __nv_bfloat16 *>(kv);
  args.kv8 = static_cast<const uint8_t *>(kv_fp8);
  args.kv_scale = kv_scale;
  args.kv_rope = static_cast<const __nv_bfloat16 *>(kv_rope);
  args.s_kv = s_kv;
  args.kv_start = kv_start;
  args.rows = rows;
  args.pos = pos;
  args.req = req;
  args.n_rows = n_rows;
  args.kv_lo = kv_lo;
  args.kv_hi = kv_hi;
  args.topk = topk;
  args.k = k;
  args.ent_lo = extra.ent_lo;
  args.ent_len = extra.ent_len;
  args.scale_log2 = softmax_scale * 1.4426950408889634f;
  args.o_part = o_part;
  args.lse_part = lse_part;
  args.o_out = static_cast<__nv_bfloat16 *>(o_out);
  args.lse_out = lse_out;
  args.sink = sink;
  args.owner_row = owner_row;
  args.T = T;
  args.status = status;

  // rows per CTA: dense packs G tokens x Hc heads into R = 64; sparse keeps one
  // token (its keys are its own) with up to 32 heads
  int R;
  if (!sparse) {
    args.hc = H <= 64 ? H : 64;
    // a work item takes g = 64 / hc consecutive shard rows over the union
    // of their key ranges; rows that split one token's keys go one per item
    args.g = extra.one_row_per_item ? 1 : 64 / args.hc;
    R = 64;
  } else {
    // one token per CTA.  fp8 works on 16 heads at a time (its four P^T
    // matrices and five score accumulators are sized for R = 16); bf16 takes
    // up to 64 (all heads of a 64-head token in one CTA, so its keys are
    // gathered once)
    const int hmax = kv_format == CPMLA_KV_FP8_E4M3_G128 ? 16 : 64;
    args.hc = H <= hmax ? H : hmax;
    if (H > hmax && H % hmax != 0)
      return fail(CPMLA_ERR_UNSUPPORTED, "%s: H=%d > %d must be a multiple of %d", fn, H, hmax,
                  hmax);
    args.g = 1;
    R = args.hc <= 16 ? 16 : (args.hc <= 32 ? 32 : 64);
  }
  args.n_hgroups = H / args.hc;
  const int64_t n_groups = (n_rows + args.g - 1) / args.g;
  const int64_t n_items = n_groups * args.n_hgroups;
  CPMLA_CHECK_ARG(n_items <= INT32_MAX, "%s: too many work items", fn);

  EncodeTiledFn enc = encode_fn();
  if (!enc) return fail(CPMLA_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", fn);
  // 2D map over a row-major [s_kv, width] array, box [box_w x box_h]
  auto encode = [&](CUtensorMap *tm, CUtensorMapDataType dt, const void *base, int width,
                    int elem_bytes, int box_w, int box_h, CUtensorMapSwizzle swz) {
    memset(tm, 0, sizeof *tm);
    cuuint64_t dims[2] = {(cuuint64_t)width, (cuuint64_t)s_kv};
    cuuint64_t strides[1] = {(cuuint64_t)width * elem_bytes};
    cuuint32_t box[2] = {(cuuint32_t)box_w, (cuuint32_t)box_h};
    cuuint32_t estr[2] = {1, 1};
    return enc(tm, dt, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (sparse) {
    // one-row boxes for four-row TMA gathers: bf16 rows of 64 dims with the
    // MMA's 128-byte swizzle (the KV, or the fp8 layout's rope), and raw fp8
    // codes of 128 dims, unswizzled
    CUtensorMap tm_kv, tm_rope;
    CUresult cr2;
    if (kv_format == CPMLA_KV_BF16) {
      cr2 = encode(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kv, CPMLA_DQK, 2, kKbDims, 1,
                   CU_TENSOR_MAP_SWIZZLE_128B);
      tm_rope = tm_kv;
    } else {
      cr2 = encode(&tm_kv, CU_TENSOR_MAP_DATA_TYPE_UINT8, kv_fp8, CPMLA_DV, 1, 128, 1,
                   CU_TENSOR_MAP_SWIZZLE_NONE);
      if (cr2 == CUDA_SUCCESS)
        cr2 = encode(&tm_rope, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kv_rope, CPMLA_DROPE, 2,
                     CPMLA_DROPE, 1, CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (cr2 != CUDA_SUCCESS)
      return fail(CPMLA_ERR_CUDA, "%s: tensor map encode failed (%d)", fn, (int)cr2);
    if (kv_format == CPMLA_KV_BF16) {
      // Q as [T tokens, H heads, 576] with the token stride; one box is the
      // 64 dims of one k-block for R consecutive heads of one token, in the
      // MMA's 128-byte-swizzled K-major layout (heads past H read as zero)
      CUtensorMap tm_q;
      memset(&tm_q, 0, sizeof tm_q);
      const int64_t T_q = (int64_t)(merged ? T : 0);
      cuuint64_t qdims[3] = {(cuuint64_t)CPMLA_DQK, (cuuint64_t)H,
                             (cuuint64_t)(T_q > 0 ? T_q : INT32_MAX)};
      cuuint64_t qstr[2] = {(cuuint64_t)CPMLA_DQK * 2, (cuuint64_t)q_token_stride * 2};
      cuuint32_t qbox[3] = {(cuuint32_t)kKbDims, (cuuint32_t)R, 1};
      cuuint32_t qes[3] = {1, 1, 1};
      const CUresult cq = enc(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q),
                              qdims, qstr, qbox, qes, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (cq != CUDA_SUCCESS)
        return fail(CPMLA_ERR_CUDA, "%s: Q tensor map encode failed (%d)", fn, (int)cq);
      return launch_sparse_wide(false, R, args, tm_kv, tm_q, tm_rope, (int)n_items, st);
    }
    return launch_sparse_wide(true, 16, args, tm_kv, tm_kv, tm_rope, (int)n_items, st);
  }
  // 128-key x 64-dim tiles of the bf16 KV
  CUtensorMap tm;
  const CUresult cr = encode(&tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kv, CPMLA_DQK, 2, kKbDims,
                             kTileKeys, CU_TENSOR_MAP_SWIZZLE_128B);
  if (cr != CUDA_SUCCESS) return fail(CPMLA_ERR_CUDA, "%s: tensor map encode failed (%d)", fn, (int)cr);
  // Q as for the sparse kernel, in boxes of 64 dims x hc heads x 1 token (the
  // kernel uses it when hc is a multiple of 8)
  CUtensorMap tm_q;
  memset(&tm_q, 0, sizeof tm_q);
  {
    const int64_t T_q = (int64_t)(merged ? T : 0);
    cuuint64_t qdims[3] = {(cuuint64_t)CPMLA_DQK, (cuuint64_t)H,
                           (cuuint64_t)(T_q > 0 ? T_q : INT32_MAX)};
    cuuint64_t qstr[2] = {(cuuint64_t)CPMLA_DQK * 2, (cuuint64_t)q_token_stride * 2};
    cuuint32_t qbox[3] = {(cuuint32_t)kKbDims, (cuuint32_t)args.hc, 1};
    cuuint32_t qes[3] = {1, 1, 1};
    const CUresult cq = enc(&tm_q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), qdims,
                            qstr, qbox, qes, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cq != CUDA_SUCCESS)
      return fail(CPMLA_ERR_CUDA, "%s: Q tensor map encode failed (%d)", fn, (int)cq);
  }
  return launch_dense(args, tm, tm_q, (int)n_items, st);
}

}  // namespace cpmla

extern "C" int mla_partial_attn_dense(const void *q, int64_t q_token_stride, int H, int kv_format,
                                      const void *kv, const void *kv_fp8, const float *kv_scale,
                                      const void *kv_rope, int64_t s_kv, const int64_t *kv_start,
                                      const int32_t *rows, const int32_t *pos, const int32_t *req,
                                      int n_rows, const int32_t *kv_lo, const int32_t *kv_hi,
                                      float softmax_scale, float *o_part, float *lse_part,
                                      void *stream) {
  return cpmla::attn_entry(false, q, q_token_stride, H, kv_format, kv, kv_fp8, kv_scale, kv_rope,
                           s_kv, kv_start, rows, pos, req, n_rows, kv_lo, kv_hi, nullptr, 0,
                           softmax_scale, o_part, lse_part, nullptr, 0, nullptr, nullptr,
                           nullptr, stream, cpmla::AttnExtra{});
}

extern "C" int mla_partial_attn_sparse(const void *q, int64_t q_token_stride, int H,
                                       int kv_format, const void *kv, const void *kv_fp8,
                                       const float *kv_scale, const void *kv_rope, int64_t s_kv,
                                       const int64_t *kv_start, const int32_t *rows,
                                       const int32_t *pos, const int32_t *req, int n_rows,
                                       const int32_t *kv_lo, const int32_t *kv_hi,
                                       const int32_t *topk_idx, int k, float softmax_scale,
                                       float *o_part, float *lse_part, void *stream) {
  return cpmla::attn_entry(true, q, q_token_stride, H, kv_format, kv, kv_fp8, kv_scale, kv_rope,
                           s_kv, kv_start, rows, pos, req, n_rows, kv_lo, kv_hi, topk_idx, k,
                           softmax_scale, o_part, lse_part, nullptr, 0, nullptr, nullptr,
                           nullptr, stream, cpmla::AttnExtra{});
}

extern "C" int mla_attn_dense_merged(const void *q, int64_t q_token_stride, int H, int kv_format,
                                     const void *kv, const void *kv_fp8, const float *kv_scale,
                                     const void *kv_rope, int64_t s_kv, const int64_t *kv_start,
                                     const int32_t *rows, const int32_t *pos, const int32_t *req,
                                     int n_rows, const int32_t *kv_lo, const int32_t *kv_hi,
                                     float softmax_scale, const int32_t *owner_row, int T,
                                     const float *sink, void *o_out, float *lse_out,
                                     void *stream) {
  using namespace cpmla;
  CPMLA_CHECK_ARG(n_rows == 0 || o_out, "mla_attn_dense_merged: o_out is NULL");
  return attn_entry(false, q, q_token_stride, H, kv_format, kv, kv_fp8, kv_scale, kv_rope, s_kv,
                    kv_start, rows, pos, req, n_rows, kv_lo, kv_hi, nullptr, 0, softmax_scale,
                    nullptr, nullptr, owner_row, T, sink, o_out, lse_out, stream, AttnExtra{});
}

extern "C" int mla_attn_sparse_merged(const void *q, int64_t q_token_stride, int H, int kv_format,
                                      const void *kv, const void *kv_fp8, const float *kv_scale,
                                      const void *kv_rope, int64_t s_kv, const int64_t *kv_start,
                                      const int32_t *rows, const int32_t *pos, const int32_t *req,
                                      int n_rows, const int32_t *kv_lo, const int32_t *kv_hi,
                                      const int32_t *topk_idx, int k, float softmax_scale,
                                      const int32_t *owner_row, int T, const float *sink,
                                      void *o_out, float *lse_out, void *stream) {
  using namespace cpmla;
  CPMLA_CHECK_ARG(n_rows == 0 || o_out, "mla_attn_sparse_merged: o_out is NULL");
  return attn_entry(true, q, q_token_stride, H, kv_format, kv, kv_fp8, kv_scale, kv_rope, s_kv,
                    kv_start, rows, pos, req, n_rows, kv_lo, kv_hi, topk_idx, k, softmax_scale,
                    nullptr, nullptr, owner_row, T, sink, o_out, lse_out, stream, AttnExtra{});
}
