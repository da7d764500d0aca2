// split_kv_noalloc.cu -- the split-KV attention of split_kv.cu for callers that
// cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: code hosted inside
// another framework that owns every device allocation and hands its plugins
// only their inputs and outputs, or a serving loop that has fixed its memory
// at start-up and may not call cudaMalloc afterwards (cudaMalloc can
// synchronise the device and fragments a pool sized in advance).  For them
// this entry point takes the parts' partial results in a fixed array of this
// library's own device memory instead of a caller workspace.  The caller still
// passes the inputs and the outputs; nothing is allocated or freed here.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds CPMLA_SPLIT_KV_STATIC_BYTES of it until the process exits.
// Host code cannot use the array's name as a device address (in host code
// the name is a host-side stand-in); its device address is looked up once per
// device, with that device current, by cudaGetSymbolAddress on the first call
// made on that device -- so make that first call before any stream capture.
// Every call on a device shares the one array and its contents are whatever
// the last call left: nothing in it has to start at zero (each call writes
// every byte it reads before reading it), but calls whose work can overlap on
// the GPU (other streams, or another host thread) race on it.
#include <mutex>

#include "attn_common.cuh"

namespace cpmla {

int split_kv_run(const char *fn, const void *q, int64_t q_token_stride, int H, int kv_format,
                 const void *kv, const void *kv_fp8, const float *kv_scale, const void *kv_rope,
                 int64_t s_kv, const int64_t *kv_start, const int32_t *tokens,
                 const int32_t *pos, const int32_t *req, int n_tokens, const int32_t *topk_idx,
                 int k, int n_split, float softmax_scale, const float *sink, int T, void *o_out,
                 float *lse_out, void *workspace, size_t workspace_bytes, void *stream);

namespace {

static __device__ __align__(256) uint8_t g_split_kv_scratch[CPMLA_SPLIT_KV_STATIC_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_split_kv_scratch on the current device, looked up once
// per device; CPMLA_OK, or an error code with its message recorded.
int scratch_address(const char *fn, void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "mla_attn_split_kv_noalloc: current device");
  if (dev < 0 || dev >= kMaxDevices)
    return fail(CPMLA_ERR_UNSUPPORTED, "%s: device %d beyond the %d this entry point serves", fn,
                dev, kMaxDevices);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_split_kv_scratch);
    if (e != cudaSuccess)
      return cuda_fail(e, "mla_attn_split_kv_noalloc: address of the static scratch array");
    if (p == nullptr)
      return fail(CPMLA_ERR_CUDA, "%s: the static scratch array has no device address", fn);
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return CPMLA_OK;
}

}  // namespace
}  // namespace cpmla

extern "C" int mla_attn_split_kv_noalloc(const void *q, int64_t q_token_stride, int H,
                                         int kv_format, const void *kv, const void *kv_fp8,
                                         const float *kv_scale, const void *kv_rope,
                                         int64_t s_kv, const int64_t *kv_start,
                                         const int32_t *tokens, const int32_t *pos,
                                         const int32_t *req, int n_tokens,
                                         const int32_t *topk_idx, int k, int n_split,
                                         float softmax_scale, const float *sink, int T,
                                         void *o_out, float *lse_out, void *stream) {
  using namespace cpmla;
  const char *fn = "mla_attn_split_kv_noalloc";
  if (n_tokens > 0 && H >= 1 && n_split >= 1) {
    const size_t need = mla_attn_split_kv_workspace_size(H, n_tokens, n_split);
    if (need > (size_t)CPMLA_SPLIT_KV_STATIC_BYTES)
      return fail(CPMLA_ERR_ARG,
                  "%s: %d tokens x %d parts x %d heads need %zu bytes of scratch, beyond the "
                  "%zu-byte static array; use fewer tokens or parts per call, or "
                  "mla_attn_split_kv with a workspace",
                  fn, n_tokens, n_split, H, need, (size_t)CPMLA_SPLIT_KV_STATIC_BYTES);
  }
  void *scratch = nullptr;
  if (n_tokens > 0) {
    const int rc = scratch_address(fn, &scratch);
    if (rc != CPMLA_OK) return rc;
  }
  return split_kv_run(fn, q, q_token_stride, H, kv_format, kv, kv_fp8, kv_scale, kv_rope, s_kv,
                      kv_start, tokens, pos, req, n_tokens, topk_idx, k, n_split, softmax_scale,
                      sink, T, o_out, lse_out, scratch, (size_t)CPMLA_SPLIT_KV_STATIC_BYTES,
                      stream);
}
