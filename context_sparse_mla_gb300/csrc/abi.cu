// abi.cu -- error reporting, version and the per-device status word.
#include <cstring>
#include <mutex>

#include "cpmla_internal.cuh"

namespace cpmla {

// First fault a kernel recorded on this device (0 = none).  Kernels get its
// device address as an argument (see status_word()).
__device__ int g_status_word;

namespace {
thread_local char t_msg[512] = "";
constexpr int kMaxDevices = 64;
int *g_status_addr[kMaxDevices] = {};
std::mutex g_status_mu;
}  // namespace

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof t_msg, fmt, ap);
  va_end(ap);
}

int fail(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(t_msg, sizeof t_msg, fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char *what) {
  return fail(CPMLA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int *status_word() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    g_status_addr[dev] = static_cast<int *>(p);
  }
  return g_status_addr[dev];
}

}  // namespace cpmla

namespace cpmla {
namespace {
// One thread waits, with the kernels' bounded wait, on a barrier that nothing
// will ever arrive at; the wait gives up after limit_ns and records
// CPMLA_ERR_TIMEOUT, exactly as a stalled pipeline stage would.
__global__ void wait_timeout_selftest_kernel(int *status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
}
}  // namespace
}  // namespace cpmla

extern "C" int cpmla_selftest_wait_timeout(unsigned int limit_ms, void *stream) {
  CPMLA_CHECK_ARG(limit_ms >= 1 && limit_ms <= 2000,
                  "cpmla_selftest_wait_timeout: limit_ms=%u outside 1..2000", limit_ms);
  int *status = cpmla::status_word();
  if (!status) return cpmla::fail(CPMLA_ERR_CUDA, "cpmla_selftest_wait_timeout: status word unavailable");
  cpmla::wait_timeout_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      status, (unsigned long long)limit_ms * 1000000ull);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cpmla::cuda_fail(e, "cpmla_selftest_wait_timeout: launch");
  return CPMLA_OK;
}

extern "C" const char *cpmla_last_error(void) { return cpmla::t_msg; }

extern "C" int cpmla_version(void) { return 100; }

extern "C" int cpmla_device_status(int *status, int clear) {
  CPMLA_CHECK_ARG(status != nullptr, "cpmla_device_status: status is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cpmla::cuda_fail(e, "cpmla_device_status: synchronize");
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, cpmla::g_status_word, sizeof v);
  if (e != cudaSuccess) return cpmla::cuda_fail(e, "cpmla_device_status: read");
  *status = v;
  if (clear) {
    int z = 0;
    e = cudaMemcpyToSymbol(cpmla::g_status_word, &z, sizeof z);
    if (e != cudaSuccess) return cpmla::cuda_fail(e, "cpmla_device_status: clear");
  }
  return CPMLA_OK;
}
