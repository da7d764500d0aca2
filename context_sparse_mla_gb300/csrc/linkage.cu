// linkage.cu -- ratio-2 compressor linkage across DualChunkSwap chunks (host)
// and the gather of the linked rows (device).
//
// "[Feature][PCP] Add DeepSeek-V4.1-Flash support", "Overview" and
// "Implementation": ratio-2 groups are compressed on each rank's local token
// rows; a pair split across two PCP chunks is closed with the preceding
// chunk's last row, and only the last (fp32) row of each local chunk is
// gathered; "Rank-local Compressor Revision" lists the cases the linkage must
// get right (PCP2/4, replicated short prefills, empty ranks, request
// isolation, newest open ring rows).  The chunks are those of
// "[Core] Add MRV2 virtual-batch PCP for MLA", "DualChunkSwap partitioning".
// Readings where the pages are silent: a ratio-2 group is the pair of request
// positions (2m, 2m+1); decode requests have no chunks.  The compressor's own
// arithmetic (its learned scores) is not on the pages and not built here.
#include <climits>
#include <vector>

#include "cpmla_internal.cuh"

namespace {

constexpr int kMaxShards = 1024;

int check_linkage_batch(const char *fn, int P, int B, const int32_t *cu, const uint8_t *dec,
                        int64_t *n_links) {
  CPMLA_CHECK_ARG(P >= 1 && P <= kMaxShards, "%s: P=%d outside 1..%d", fn, P, kMaxShards);
  CPMLA_CHECK_ARG(B >= 0, "%s: B=%d < 0", fn, B);
  CPMLA_CHECK_ARG(cu != nullptr, "%s: cu_seqlens is NULL", fn);
  CPMLA_CHECK_ARG(B == 0 || dec != nullptr, "%s: is_decode is NULL", fn);
  CPMLA_CHECK_ARG(cu[0] == 0, "%s: cu_seqlens[0]=%d, expected 0", fn, cu[0]);
  int64_t prefills = 0;
  for (int b = 0; b < B; ++b) {
    CPMLA_CHECK_ARG(cu[b + 1] >= cu[b], "%s: cu_seqlens decreases at request %d", fn, b);
    if (!dec[b]) ++prefills;
  }
  const int64_t n = prefills * 2 * P;
  CPMLA_CHECK_ARG(n <= INT32_MAX, "%s: %lld entries exceed int32", fn, (long long)n);
  *n_links = n;
  return CPMLA_OK;
}

}  // namespace

extern "C" int pcp_ratio2_linkage_size(int P, int B, const int32_t *cu_seqlens,
                                       const uint8_t *is_decode, int64_t *n_links) {
  CPMLA_CHECK_ARG(n_links != nullptr, "pcp_ratio2_linkage_size: n_links is NULL");
  return check_linkage_batch("pcp_ratio2_linkage_size", P, B, cu_seqlens, is_decode, n_links);
}

extern "C" int pcp_ratio2_linkage(int P, int B, const int32_t *cu_seqlens,
                                  const int32_t *q_start_pos, const uint8_t *is_decode,
                                  int32_t *first, int32_t *last, int32_t *pred,
                                  int32_t *pred_shard, int32_t *flags) {
  const char *fn = "pcp_ratio2_linkage";
  int64_t n = 0;
  int rc = check_linkage_batch(fn, P, B, cu_seqlens, is_decode, &n);
  if (rc != CPMLA_OK) return rc;
  CPMLA_CHECK_ARG(B == 0 || q_start_pos != nullptr, "%s: q_start_pos is NULL", fn);
  CPMLA_CHECK_ARG(n == 0 || (first && last && pred && pred_shard && flags),
                  "%s: an output array is NULL", fn);
  for (int b = 0; b < B; ++b)
    CPMLA_CHECK_ARG(q_start_pos[b] >= 0 &&
                        (int64_t)q_start_pos[b] + cu_seqlens[b + 1] - cu_seqlens[b] <= INT32_MAX,
                    "%s: bad start position %d for request %d", fn, q_start_pos[b], b);
  const int nc = 2 * P;
  // per chunk of the request being filled: its start, length and the nearest
  // earlier non-empty chunk (whose last row is the predecessor)
  std::vector<int32_t> lo(nc), len(nc), prev(nc);
  // entries of shard r for prefill request number k sit at (r * prefills + k) * 2
  const int64_t prefills = n / (2 * P);
  int64_t k = 0;
  for (int b = 0; b < B; ++b) {
    if (is_decode[b]) continue;
    const int32_t g0 = cu_seqlens[b], S = cu_seqlens[b + 1] - g0, q0 = q_start_pos[b];
    const int32_t base = S / nc, extra = S % nc;
    int last_nonempty = -1;
    for (int c = 0; c < nc; ++c) {
      lo[c] = c * base + (c < extra ? c : extra);
      len[c] = base + (c < extra ? 1 : 0);
      prev[c] = last_nonempty;
      if (len[c] > 0) last_nonempty = c;
    }
    for (int r = 0; r < P; ++r) {
      const int mine[2] = {r, nc - 1 - r};
      for (int h = 0; h < 2; ++h) {
        const int c = mine[h];
        const int64_t e = (r * prefills + k) * 2 + h;
        first[e] = last[e] = pred[e] = pred_shard[e] = -1;
        flags[e] = 0;
        if (len[c] == 0) continue;
        first[e] = g0 + lo[c];
        last[e] = g0 + lo[c] + len[c] - 1;
        const int32_t p_first = q0 + lo[c], p_last = q0 + lo[c] + len[c] - 1;
        int32_t f = 0;
        if (p_first & 1) {
          // the chunk opens on the second row of a pair
          f |= 1;
          if (prev[c] >= 0) {
            pred[e] = g0 + lo[prev[c]] + len[prev[c]] - 1;
            pred_shard[e] = prev[c] < P ? prev[c] : nc - 1 - prev[c];
          } else {
            f |= 2;  // the first row of the pair came in an earlier step
          }
        }
        if (!(p_last & 1)) {
          f |= 4;  // the chunk closes on the first row of a pair
          if (lo[c] + len[c] == S) f |= 8;
        }
        flags[e] = f;
      }
    }
    ++k;
  }
  return CPMLA_OK;
}

// ------------------------------------------------------------ row gather
namespace cpmla {
namespace {

constexpr int kGatherThreads = 256;

// One warp per output row: out[i, :] = src[idx[i], :] (16-byte vectors), or
// zeros for idx[i] == -1; an index outside [-1, n_src) is recorded and its
// row zeroed.
__global__ void __launch_bounds__(kGatherThreads)
    gather_rows_kernel(const float *__restrict__ src, int64_t src_stride, int64_t n_src, int D,
                       int n, const int32_t *__restrict__ idx, float *__restrict__ out,
                       int64_t out_stride, int *status) {
  const int lane = threadIdx.x & 31;
  const int64_t w0 = ((int64_t)blockIdx.x * kGatherThreads + threadIdx.x) >> 5;
  const int64_t nw = ((int64_t)gridDim.x * kGatherThreads) >> 5;
  const int nv = D >> 2;
  for (int64_t i = w0; i < n; i += nw) {
    const int j = idx[i];
    const bool bad = j < -1 || (int64_t)j >= n_src;
    if (bad && lane == 0) record_status(status, CPMLA_ERR_INDEX);
    float4 *dst = reinterpret_cast<float4 *>(out + i * out_stride);
    if (j < 0 || bad) {
      for (int v = lane; v < nv; v += 32) dst[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      continue;
    }
    const float4 *s = reinterpret_cast<const float4 *>(src + (int64_t)j * src_stride);
    for (int v = lane; v < nv; v += 32) dst[v] = __ldg(s + v);
  }
}

}  // namespace
}  // namespace cpmla

extern "C" int pcp_gather_rows_f32(const float *src, int64_t src_row_stride, int64_t n_src, int D,
                                   int n, const int32_t *idx, float *out, int64_t out_row_stride,
                                   void *stream) {
  using namespace cpmla;
  const char *fn = "pcp_gather_rows_f32";
  CPMLA_CHECK_ARG(n >= 0 && n_src >= 0, "%s: negative size", fn);
  CPMLA_CHECK_ARG(D >= 4 && D % 4 == 0, "%s: D=%d must be a positive multiple of 4", fn, D);
  CPMLA_CHECK_ARG(src_row_stride >= D && src_row_stride % 4 == 0 && out_row_stride >= D &&
                      out_row_stride % 4 == 0,
                  "%s: row strides must be >= D and multiples of 4", fn);
  if (n == 0) return CPMLA_OK;
  CPMLA_CHECK_ARG(idx && out && (n_src == 0 || src), "%s: a required pointer is NULL", fn);
  CPMLA_CHECK_ARG(((uintptr_t)src & 15) == 0 && ((uintptr_t)out & 15) == 0,
                  "%s: src and out must be 16-byte aligned", fn);
  int *status = status_word();
  if (!status) return fail(CPMLA_ERR_CUDA, "%s: status word unavailable", fn);
  int dev = 0, n_sm = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
  const int64_t blocks = (n + (kGatherThreads / 32) - 1) / (kGatherThreads / 32);
  const int64_t cap = (int64_t)(n_sm > 0 ? n_sm : 152) * 8;
  const int grid = (int)(blocks < cap ? blocks : cap);
  gather_rows_kernel<<<grid, kGatherThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      src, src_row_stride, n_src, D, n, idx, out, out_row_stride, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "pcp_gather_rows_f32: launch");
  return CPMLA_OK;
}
