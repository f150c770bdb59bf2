// api.cu — status and error reporting, device properties, and the
// copy-ceiling kernel of libgf.
#include <stdarg.h>
#include <stdio.h>


#include "gf_internal.cuh"

namespace gf {

static thread_local char g_msg[512] = "";

void set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
}

int cuda_fail(cudaError_t e, const char* what) {
  set_error("%s: %s", what, cudaGetErrorString(e));
  return GF_ECUDA;
}

int device_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cached[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// 16-byte vector copy, four independent loads in flight per thread.
__global__ void __launch_bounds__(256) k_copy(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                              size_t n) {
  size_t stride = (size_t)gridDim.x * blockDim.x;
  size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    uint4 a = __ldcs(src + i), b = __ldcs(src + i + stride);
    uint4 c = __ldcs(src + i + 2 * stride), d = __ldcs(src + i + 3 * stride);
    __stcs(dst + i, a);
    __stcs(dst + i + stride, b);
    __stcs(dst + i + 2 * stride, c);
    __stcs(dst + i + 3 * stride, d);
  }
  for (; i < n; i += stride) __stcs(dst + i, __ldcs(src + i));
}

}  // namespace gf

using namespace gf;

extern "C" {

const char* gf_last_error(void) { return g_msg; }

int gf_version(void) { return 2; }

long long gf_packed_bytes(int wdtype, int N, int K) {
  if (wdtype < 0 || wdtype > 2 || N <= 0 || K <= 0 || K % per_chunk(wdtype)) return -1;
  return packed_bytes(wdtype, N, K, 32);
}

int gf_copy_ceiling(const void* src, void* dst, size_t bytes, gf_stream stream) {
  if (!src || !dst || bytes % 16) {
    set_error("gf_copy_ceiling: null pointer or size not a multiple of 16");
    return GF_EINVAL;
  }
  if (!aligned16(src) || !aligned16(dst)) {
    set_error("gf_copy_ceiling: pointers must be 16-byte aligned");
    return GF_EALIGN;
  }
  if (bytes == 0) return GF_OK;
  int sms = device_sms();
  k_copy<<<sms * 8, 256, 0, (cudaStream_t)stream>>>((const uint4*)src, (uint4*)dst, bytes / 16);
  GF_CUDA(cudaGetLastError());
  return GF_OK;
}

static_assert(GF_DEVERR_WAIT_FULL == ERR_WAIT_FULL && GF_DEVERR_WAIT_EMPTY == ERR_WAIT_EMPTY &&
                  GF_DEVERR_WAIT_GRID == ERR_WAIT_GRID && GF_DEVERR_WAIT_CTA == ERR_WAIT_CTA &&
                  GF_DEVERR_DRAIN == ERR_DRAIN && GF_DEVERR_BAD_PROGRAM == ERR_BAD_PROGRAM &&
                  GF_DEVERR_BAD_POS == ERR_BAD_POS && GF_DEVERR_BAD_TOKEN == ERR_BAD_TOKEN &&
                  GF_DEVERR_WAIT_ROUTER == ERR_WAIT_ROUTER && GF_DEVERR_WAIT_COMBINE == ERR_WAIT_COMBINE &&
                  GF_DEVERR_WAIT_HEAD == ERR_WAIT_HEAD,
              "public and internal device error codes agree");

int gf_device_error(void) {
  GF_CUDA(cudaDeviceSynchronize());
  int* p = device_err_ptr();
  if (!p) return GF_ECUDA;
  int v = 0;
  GF_CUDA(cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost));
  int zero = 0;
  GF_CUDA(cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice));
  return v;
}

}  // extern "C"
