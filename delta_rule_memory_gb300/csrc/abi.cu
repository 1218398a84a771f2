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

int check_launch(const char *what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(SDM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return SDM_OK;
}

}  // namespace sdm

extern "C" int sdm_version(void) { return 10000; }

extern "C" const char *sdm_last_error(void) { return g_last_error; }
