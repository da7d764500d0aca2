// split_kv.cu -- attention of a list of tokens whose keys are split into parts
// computed side by side (split-KV, flash-decoding style), then merged by LSE
// with the attention sink applied once.
//
// "[Core] Add MRV2 virtual-batch PCP for MLA", "PCP algorithm": decode rows
// are replicated on every PCP rank; "[DeepSeekV4][PCP] Enable context-parallel
// prefill for hybrid KV and MegaMoE", "Implementation summary": partial
// (output, LSE) pairs are merged globally by LSE and the sink is applied once.
// A decode row has one query and a long context (or a long top-k list), so
// one work item per row leaves most of the GPU idle; here row i's keys are cut
// into n_split parts -- the replicated rows of the pages each take one part
// instead of all of it -- and each part is its own work item:
//   dense:  part s of a row at position t takes positions
//           [floor((t+1) s / n), floor((t+1)(s+1) / n) - 1]
//   sparse: part s takes entries [s ke, (s+1) ke) of the row's top-k list,
//           ke = ceil(k / n)
// Three launches on the caller's stream: the parts' row arrays (built in the
// workspace), the partial attention of all parts (the kernels of
// attn_dense.cu / attn_sparse*.cu), and the merge of each token's parts.
#include <cmath>

#include "attn_common.cuh"

namespace cpmla {
namespace {

constexpr int kSplitMax = 64;

// Workspace sections, each 256-byte aligned.
struct SplitLayout {
  size_t rows, pos, req, lo, hi, off, crow, o, lse, total;
};

SplitLayout split_layout(int H, int64_t n, int ns) {
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t m = (size_t)n * ns;
  SplitLayout L{};
  size_t at = 0;
  L.rows = at;
  at += up(m * 4);
  L.pos = at;
  at += up(m * 4);
  L.req = at;
  at += up(m * 4);
  L.lo = at;
  at += up(m * 4);
  L.hi = at;
  at += up(m * 4);
  L.off = at;
  at += up((size_t)(n + 1) * 4);
  L.crow = at;
  at += up(m * 4);
  L.o = at;
  at += up(m * H * CPMLA_DV * 4);
  L.lse = at;
  at += up(m * H * 4);
  L.total = at;
  return L;
}

// One thread per (token, part): the part's shard-row arrays, its key range
// (dense) or top-k window start (sparse), and the merge's CSR of parts.
__global__ void split_rows_kernel(const int32_t *__restrict__ tokens,
                                  const int32_t *__restrict__ pos,
                                  const int32_t *__restrict__ req, int n, int ns, int k,
                                  int sparse, int32_t *rows, int32_t *rpos, int32_t *rreq,
                                  int32_t *lo, int32_t *hi, int32_t *off, int32_t *crow) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t m = (int64_t)n * ns;
  if (i >= m) return;
  const int tk = (int)(i / ns), s = (int)(i - (int64_t)tk * ns);
  const int t = pos[tk];
  rows[i] = tokens[tk];
  rpos[i] = t;
  rreq[i] = req[tk];
  if (sparse) {
    lo[i] = s * ((k + ns - 1) / ns);
    hi[i] = 0;
  } else {
    const int64_t span = (int64_t)t + 1;
    lo[i] = (int)(span * s / ns);
    hi[i] = (int)(span * (s + 1) / ns) - 1;  // below lo: an empty part
  }
  crow[i] = (int)i;
  if (s == 0) off[tk] = (int)(tk * (int64_t)ns);
  if (i == m - 1) off[n] = (int)m;
}

}  // namespace

// The split-KV path with the workspace at a given device address (the public
// entry points pass the caller's buffer or the library's own).
int split_kv_run(const char *fn, const void *q, int64_t q_token_stride, int H, int kv_format,
                 const void *kv, const void *kv_fp8, const float *kv_scale, const void *kv_rope,
                 int64_t s_kv, const int64_t *kv_start, const int32_t *tokens,
                 const int32_t *pos, const int32_t *req, int n_tokens, const int32_t *topk_idx,
                 int k, int n_split, float softmax_scale, const float *sink, int T, void *o_out,
                 float *lse_out, void *workspace, size_t workspace_bytes, void *stream) {
  CPMLA_CHECK_ARG(n_tokens >= 0, "%s: n_tokens=%d < 0", fn, n_tokens);
  CPMLA_CHECK_ARG(n_split >= 1 && n_split <= kSplitMax, "%s: n_split=%d outside 1..%d", fn,
                  n_split, kSplitMax);
  CPMLA_CHECK_ARG(H >= 1 && H <= 128, "%s: H=%d outside 1..128", fn, H);
  CPMLA_CHECK_ARG((int64_t)n_tokens * n_split <= INT32_MAX, "%s: too many parts", fn);
  CPMLA_CHECK_ARG(T >= 1 || n_tokens == 0, "%s: T=%d", fn, T);
  if (topk_idx) CPMLA_CHECK_ARG(k >= 1 && k <= 65536, "%s: k=%d outside 1..65536", fn, k);
  if (n_tokens == 0) return CPMLA_OK;
  CPMLA_CHECK_ARG(tokens && pos && req && o_out && lse_out, "%s: a required pointer is NULL", fn);
  const SplitLayout L = split_layout(H, n_tokens, n_split);
  CPMLA_CHECK_ARG(workspace != nullptr && ((uintptr_t)workspace & 255) == 0,
                  "%s: workspace must be non-NULL and 256-byte aligned", fn);
  CPMLA_CHECK_ARG(workspace_bytes >= L.total, "%s: workspace of %zu bytes, %zu needed", fn,
                  workspace_bytes, L.total);
  int *status = status_word();
  if (!status) return fail(CPMLA_ERR_CUDA, "%s: status word unavailable", fn);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *rows = reinterpret_cast<int32_t *>(ws + L.rows);
  int32_t *rpos = reinterpret_cast<int32_t *>(ws + L.pos);
  int32_t *rreq = reinterpret_cast<int32_t *>(ws + L.req);
  int32_t *lo = reinterpret_cast<int32_t *>(ws + L.lo);
  int32_t *hi = reinterpret_cast<int32_t *>(ws + L.hi);
  int32_t *off = reinterpret_cast<int32_t *>(ws + L.off);
  int32_t *crow = reinterpret_cast<int32_t *>(ws + L.crow);
  float *o_part = reinterpret_cast<float *>(ws + L.o);
  float *lse_part = reinterpret_cast<float *>(ws + L.lse);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool sparse = topk_idx != nullptr;
  const int m = n_tokens * n_split;
  split_rows_kernel<<<(m + 255) / 256, 256, 0, st>>>(tokens, pos, req, n_tokens, n_split, k,
                                                     sparse ? 1 : 0, rows, rpos, rreq, lo, hi,
                                                     off, crow);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "split-KV rows: launch");
  AttnExtra ex;
  ex.fn = fn;
  if (sparse) {
    ex.ent_lo = lo;
    ex.ent_len = (k + n_split - 1) / n_split;
  } else {
    ex.one_row_per_item = true;
  }
  int rc = attn_entry(sparse, q, q_token_stride, H, kv_format, kv, kv_fp8, kv_scale, kv_rope,
                      s_kv, kv_start, rows, rpos, rreq, m, sparse ? nullptr : lo,
                      sparse ? nullptr : hi, topk_idx, k, softmax_scale, o_part, lse_part,
                      nullptr, 0, nullptr, nullptr, nullptr, stream, ex);
  if (rc != CPMLA_OK) return rc;
  return launch_merge_to_tokens(o_part, lse_part, m, H, off, crow, n_tokens, sink, o_out, lse_out,
                                tokens, T, status, st);
}

}  // namespace cpmla

extern "C" size_t mla_attn_split_kv_workspace_size(int H, int n_tokens, int n_split) {
  if (H < 1 || n_tokens < 0 || n_split < 1) return 0;
  return cpmla::split_layout(H, n_tokens, n_split).total;
}

extern "C" int mla_attn_split_kv(const void *q, int64_t q_token_stride, int H, int kv_format,
                                 const void *kv, const void *kv_fp8, const float *kv_scale,
                                 const void *kv_rope, int64_t s_kv, const int64_t *kv_start,
                                 const int32_t *tokens, const int32_t *pos, const int32_t *req,
                                 int n_tokens, const int32_t *topk_idx, int k, int n_split,
                                 float softmax_scale, const float *sink, int T, void *o_out,
                                 float *lse_out, void *workspace, size_t workspace_bytes,
                                 void *stream) {
  return cpmla::split_kv_run("mla_attn_split_kv", q, q_token_stride, H, kv_format, kv, kv_fp8,
                             kv_scale, kv_rope, s_kv, kv_start, tokens, pos, req, n_tokens,
                             topk_idx, k, n_split, softmax_scale, sink, T, o_out, lse_out,
                             workspace, workspace_bytes, stream);
}
