// abi.cu - library-wide entry points: version and per-thread error text.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"

namespace {
thread_local char g_last_error[512] = "";
}

namespace sdm {

int set_error(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

int sticky_gdn_chunk(int32_t *bits);
int sticky_sse_chunk(int32_t *bits);

int check_launch(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SDM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return SDM_OK;
}

}  // namespace sdm

extern "C" int sdm_version(void) { return 10000; }

extern "C" const char *sdm_last_error(void) { return g_last_error; }

// sdm_check: wait for `stream`, then report the caller's device error word
// and every timeout the library recorded since the last check.
extern "C" int sdm_check(const int32_t *dev_err, void *stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return sdm::set_error(SDM_ERR_CUDA, "sdm_check: %s", cudaGetErrorString(e));
  int32_t bits = 0;
  if (dev_err) {
    e = cudaMemcpy(&bits, dev_err, sizeof bits, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return sdm::set_error(SDM_ERR_CUDA, "sdm_check: %s", cudaGetErrorString(e));
  }
  int rc = sdm::sticky_gdn_chunk(&bits);
  if (rc == SDM_OK) rc = sdm::sticky_sse_chunk(&bits);
  if (rc != SDM_OK) return rc;
  if (bits == 0) return SDM_OK;
  return sdm::set_error(SDM_ERR_DEVICE, "device error bits 0x%x:%s%s%s%s", static_cast<unsigned>(bits),
                        (bits & SDM_DEVERR_INDEX_RANGE) ? " index out of range;" : "",
                        (bits & SDM_DEVERR_INDEX_REPEAT) ? " repeated write slot;" : "",
                        (bits & SDM_DEVERR_NONFINITE) ? " non-finite score or logit;" : "",
                        (bits & SDM_DEVERR_TIMEOUT) ? " a bounded on-device wait gave up (outputs and state invalid);"
                                                    : "");
}
