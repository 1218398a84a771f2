// common.cuh - small helpers shared by the libsdm kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sdm.h"

namespace sdm {

constexpr unsigned kFull = 0xffffffffu;

// Set the thread-local error text (abi.cu) and return `code`.
int set_error(int code, const char *fmt, ...);
// Check the last launch; on failure record the CUDA error text.
int check_launch(const char *what);

inline bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Monotone map float -> uint32: a > b (as floats, not NaN) <=> key(a) > key(b).
__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(b);
}

// Timeouts of bounded on-device waits are never dropped: besides the caller's
// optional error word, every one is OR-ed into this translation unit's own
// device word, which sdm_check() reads (and clears) through the accessor that
// SDM_STICKY_ACCESSOR defines in the same file.
static __device__ int32_t g_sticky_err;

__device__ __forceinline__ void report_timeout(int32_t *err) {
  if (err) atomicOr(err, SDM_DEVERR_TIMEOUT);
  atomicOr(&g_sticky_err, SDM_DEVERR_TIMEOUT);
}

// host side: read this file's sticky word into *bits and clear it
#define SDM_STICKY_ACCESSOR(name)                                                        \
  int name(int32_t *bits) {                                                              \
    int32_t v = 0;                                                                       \
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_sticky_err, sizeof v);                    \
    if (e != cudaSuccess) return set_error(SDM_ERR_CUDA, "sdm_check: %s", cudaGetErrorString(e)); \
    if (v) {                                                                             \
      const int32_t zero = 0;                                                            \
      e = cudaMemcpyToSymbol(g_sticky_err, &zero, sizeof zero);                          \
      if (e != cudaSuccess) return set_error(SDM_ERR_CUDA, "sdm_check: %s", cudaGetErrorString(e)); \
    }                                                                                    \
    *bits |= v;                                                                          \
    return SDM_OK;                                                                       \
  }

__device__ __forceinline__ float bf16_to_f32(uint16_t h) { return __uint_as_float(uint32_t(h) << 16); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// cp.async (non-bulk, generic proxy) of 4, 8 or 16 bytes global -> shared.
template <int BYTES>
__device__ __forceinline__ void cp_async(void *smem_dst, const void *gmem_src) {
  static_assert(BYTES == 4 || BYTES == 8 || BYTES == 16, "cp.async size");
  if constexpr (BYTES == 16) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src)
                 : "memory");
  } else {
    asm volatile("cp.async.ca.shared.global [%0], [%1], %2;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src),
                 "n"(BYTES)
                 : "memory");
  }
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

}  // namespace sdm
