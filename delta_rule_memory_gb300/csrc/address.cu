// address.cu - product-key addressing (Sparse Delta Memory deck, "Product keys
// select addresses without scoring every slot", Secs. 2 and 3.1).
//
// One warp per token-head row.  Each stage is an exact warp-level top-k over
// (key descending, id ascending), where key is the order-preserving uint32
// image of an fp32 score:
//   * every lane holds E candidates in registers, sorted locally;
//   * per output rank, one redux.sync max finds the best head key, one
//     redux.sync min picks the lowest id among lanes holding that key, and the
//     winning lane pops its head.
// Stage 1 and 2 select the top-k of each score half (ids = positions); stage 3
// forms the k*k fp32 sums s1[a] + s2[b] (ids = a*sqrtN + b) and selects the
// top-W; the weights are the softmax of the selected sums.
#include <climits>

#include "common.cuh"

namespace sdm {
namespace {

constexpr int kAddrWarps = 8;

template <int E>
__device__ __forceinline__ void local_sort(uint32_t (&key)[E], int (&id)[E]) {
  // odd-even transposition sort, descending by (key, -id)
#pragma unroll
  for (int pass = 0; pass < E; ++pass) {
#pragma unroll
    for (int i = pass & 1; i + 1 < E; i += 2) {
      const bool sw = key[i + 1] > key[i] || (key[i + 1] == key[i] && id[i + 1] < id[i]);
      const uint32_t k0 = key[i], k1 = key[i + 1];
      const int i0 = id[i], i1 = id[i + 1];
      key[i] = sw ? k1 : k0;
      key[i + 1] = sw ? k0 : k1;
      id[i] = sw ? i1 : i0;
      id[i + 1] = sw ? i0 : i1;
    }
  }
}

// Exact top-`count` of the warp's 32*E (key, id) pairs.  Padding entries carry
// key 0 and id INT_MAX; ids of real entries are distinct.  On return, rank r
// (r < count) sits in lane r % 32, output slot r / 32.
template <int E, int OUTS>
__device__ __forceinline__ void warp_topk(uint32_t (&key)[E], int (&id)[E], int count, uint32_t (&okey)[OUTS],
                                          int (&oid)[OUTS]) {
  const int lane = threadIdx.x & 31;
  local_sort(key, id);
#pragma unroll
  for (int o = 0; o < OUTS; ++o) {
    okey[o] = 0;
    oid[o] = INT_MAX;
  }
  for (int r = 0; r < count; ++r) {
    const uint32_t m = __reduce_max_sync(kFull, key[0]);
    const int cand = (key[0] == m) ? id[0] : INT_MAX;
    const int wid = __reduce_min_sync(kFull, cand);
    const bool pop = (key[0] == m) && (id[0] == wid);
#pragma unroll
    for (int e = 0; e + 1 < E; ++e) {
      key[e] = pop ? key[e + 1] : key[e];
      id[e] = pop ? id[e + 1] : id[e];
    }
    if (pop) {
      key[E - 1] = 0;
      id[E - 1] = INT_MAX;
    }
#pragma unroll
    for (int o = 0; o < OUTS; ++o) {
      if (r == lane + 32 * o) {
        okey[o] = m;
        oid[o] = wid;
      }
    }
  }
}

template <int E>
__global__ void __launch_bounds__(kAddrWarps * 32) address_kernel(const float *__restrict__ s1,
                                                                  const float *__restrict__ s2, long rows,
                                                                  int sqrtN, int k, int W,
                                                                  int32_t *__restrict__ idx_out,
                                                                  float *__restrict__ w_out,
                                                                  int32_t *__restrict__ dev_err) {
  const int lane = threadIdx.x & 31;
  const long row = static_cast<long>(blockIdx.x) * kAddrWarps + (threadIdx.x >> 5);
  if (row >= rows) return;  // warp-uniform

  // --- stage 1 and 2: top-k of each half (one lane holds rank `lane`) ---
  float hv[2];
  int hid[2];
  bool bad = false;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const float *src = (half == 0 ? s1 : s2) + row * sqrtN;
    uint32_t key[E];
    int id[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const int j = lane + 32 * e;
      const bool in = j < sqrtN;
      const float x = in ? src[j] : 0.f;
      bad |= in && !isfinite(x);
      key[e] = in ? order_key(x) : 0u;
      id[e] = in ? j : INT_MAX;
    }
    uint32_t ok[1];
    int oi[1];
    warp_topk<E, 1>(key, id, k, ok, oi);
    hv[half] = key_value(ok[0]);
    hid[half] = oi[0];
  }
  if (__any_sync(kFull, bad) && lane == 0 && dev_err) atomicOr(dev_err, SDM_DEVERR_NONFINITE);

  // --- stage 3: the k*k candidate sums, top-W ---
  uint32_t key[E];
  int id[E];
  const int kk = k * k;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int c = lane + 32 * e;
    const int x = c / k, y = c - (c / k) * k;
    const float av = __shfl_sync(kFull, hv[0], x & 31);
    const float bv = __shfl_sync(kFull, hv[1], y & 31);
    const int ai = __shfl_sync(kFull, hid[0], x & 31);
    const int bi = __shfl_sync(kFull, hid[1], y & 31);
    const bool in = c < kk;
    key[e] = in ? order_key(__fadd_rn(av, bv)) : 0u;
    id[e] = in ? ai * sqrtN + bi : INT_MAX;
  }
  uint32_t ok[2];
  int oi[2];
  warp_topk<E, 2>(key, id, W, ok, oi);

  // --- weights: softmax over the W selected sums (max = rank 0) ---
  const float smax = key_value(__shfl_sync(kFull, ok[0], 0));
  float ex[2];
  float part = 0.f;
#pragma unroll
  for (int o = 0; o < 2; ++o) {
    const int r = lane + 32 * o;
    ex[o] = (r < W) ? expf(key_value(ok[o]) - smax) : 0.f;
    part += ex[o];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
#pragma unroll
  for (int o = 0; o < 2; ++o) {
    const int r = lane + 32 * o;
    if (r < W) {
      idx_out[row * W + r] = oi[o];
      w_out[row * W + r] = ex[o] / part;
    }
  }
}

int pow2_at_least(int n) {
  int e = 1;
  while (e < n) e <<= 1;
  return e;
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" int sdm_address(const float *s1, const float *s2, int B, int T, int H, int sqrtN, int k, int W,
                           int32_t *idx_out, float *w_out, int32_t *dev_err, void *stream) {
  if (!s1 || !s2 || !idx_out || !w_out) return set_error(SDM_ERR_INVALID_ARG, "sdm_address: null pointer");
  if (B < 0 || T < 0 || H < 0) return set_error(SDM_ERR_INVALID_ARG, "sdm_address: negative size");
  if (sqrtN < 1 || sqrtN > 512 || k < 1 || k > 32 || k > sqrtN || W < 1 || W > 64 || W > k * k)
    return set_error(SDM_ERR_SHAPE, "sdm_address: need 1<=sqrtN<=512, 1<=k<=min(32,sqrtN), 1<=W<=min(64,k*k)");
  if (!aligned(s1, 4) || !aligned(s2, 4) || !aligned(idx_out, 4) || !aligned(w_out, 4) ||
      (dev_err && !aligned(dev_err, 4)))
    return set_error(SDM_ERR_ALIGN, "sdm_address: pointers must be 4-byte aligned");
  const long rows = static_cast<long>(B) * T * H;
  if (rows >= (1L << 31)) return set_error(SDM_ERR_SHAPE, "sdm_address: B*T*H must be < 2^31");
  if (rows == 0) return SDM_OK;
  const int E = pow2_at_least(max((sqrtN + 31) / 32, (k * k + 31) / 32));
  const dim3 grid(static_cast<unsigned>((rows + kAddrWarps - 1) / kAddrWarps));
  const dim3 block(kAddrWarps * 32);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (E) {
    case 1: address_kernel<1><<<grid, block, 0, st>>>(s1, s2, rows, sqrtN, k, W, idx_out, w_out, dev_err); break;
    case 2: address_kernel<2><<<grid, block, 0, st>>>(s1, s2, rows, sqrtN, k, W, idx_out, w_out, dev_err); break;
    case 4: address_kernel<4><<<grid, block, 0, st>>>(s1, s2, rows, sqrtN, k, W, idx_out, w_out, dev_err); break;
    case 8: address_kernel<8><<<grid, block, 0, st>>>(s1, s2, rows, sqrtN, k, W, idx_out, w_out, dev_err); break;
    case 16: address_kernel<16><<<grid, block, 0, st>>>(s1, s2, rows, sqrtN, k, W, idx_out, w_out, dev_err); break;
    case 32: address_kernel<32><<<grid, block, 0, st>>>(s1, s2, rows, sqrtN, k, W, idx_out, w_out, dev_err); break;
    default: return set_error(SDM_ERR_SHAPE, "sdm_address: unsupported size");
  }
  return check_launch("sdm_address");
}
