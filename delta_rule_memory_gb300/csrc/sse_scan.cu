// sse_scan.cu - Sparse State Expansion scan (SSE deck, "One gate controls both
// writes and reads", Eqs. 9-14; "SSE routes tokens into shared-parameter state
// partitions"; "A memory decays only when its partition is visited").
//
// Two kernels:
//   route  - one warp per token-head: top-k partitions by router logit (ties to
//            the lower index), their softmax gates over all N partitions (not
//            renormalised), and the max / inverse normaliser of the key-logit
//            softmax over the c rows.  One small record per token.
//   scan   - one CTA per (batch, head, 16-column tile).  All N+1 partitions of
//            that column tile live in shared memory for the whole sequence; per
//            token only the k routed partitions and the shared one are touched
//            (decay, write, read), two columns per thread with packed fp32x2
//            arithmetic.  Per-token inputs are prefetched P tokens ahead with
//            cp.async; one CTA barrier per token (two with the delta write).
//
// Write modes: additive (the deck's SSE: S^p[j,:] += g kk_j v after the
// decay) and delta, where the rows of a visited partition share one residual
// v - vhat_p, vhat_p = sum_j kk_j alpha_j S^p[j,:] (the Sparse Delta Memory
// deck's shared residual, Fig. 2, with row weights kk and strength g).
#include <climits>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "sse_group.cuh"

namespace sdm {
namespace {

constexpr int kSseDT = 16;        // columns per CTA
constexpr int kSseThreads = 256;  // 16 columns x 16 row groups
constexpr int kSseP = 4;          // tokens prefetched ahead
constexpr int kSseMaxTopk = 8;

using ssegrp::rec_words;

// ---------------------------------------------------------------------------
// Routing prepass.
// ---------------------------------------------------------------------------
// Routing with one thread per token-head, for N <= kRouteThreadN without the
// key-logit statistics (the chunked path): the same selection (order keys,
// ties to the lower partition) and gates e = softmax over all N logits, the
// normaliser summed in partition order.
constexpr int kRouteThreadN = 16;

__global__ void __launch_bounds__(256) sse_route_thread_kernel(const float *__restrict__ route, long tokens, int N,
                                                               int topk, uint32_t *__restrict__ rec,
                                                               int32_t *__restrict__ sel_out,
                                                               int32_t *__restrict__ dev_err) {
  const long tok = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  bool bad = false;
  if (tok < tokens) {
    const float *lg = route + tok * N;
    uint32_t key[kRouteThreadN];
    float lv[kRouteThreadN];
    uint32_t kmax = 0u;
#pragma unroll
    for (int j = 0; j < kRouteThreadN; ++j) {
      lv[j] = j < N ? lg[j] : 0.f;
      bad |= j < N && !isfinite(lv[j]);
      key[j] = j < N ? order_key(lv[j]) : 0u;
      kmax = max(kmax, key[j]);
    }
    const float lmax = key_value(kmax);
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < kRouteThreadN; ++j)
      if (j < N) z += expf(lv[j] - lmax);
    uint32_t *r = rec + tok * rec_words(topk);
    uint32_t taken = 0u;
    for (int s = 0; s < topk; ++s) {
      uint32_t best = 0u;
      int bid = -1;
#pragma unroll
      for (int j = 0; j < kRouteThreadN; ++j) {  // first (lowest) id wins ties
        const bool cand = j < N && !((taken >> j) & 1u) && (bid < 0 || key[j] > best);
        if (cand) {
          best = key[j];
          bid = j;
        }
      }
      taken |= 1u << bid;
      r[s] = static_cast<uint32_t>(bid);
      r[topk + s] = __float_as_uint(expf(key_value(best) - lmax) / z);
      if (sel_out) sel_out[tok * topk + s] = bid;
    }
  }
  if (__any_sync(kFull, bad) && (threadIdx.x & 31) == 0 && dev_err) atomicOr(dev_err, SDM_DEVERR_NONFINITE);
}

__global__ void __launch_bounds__(256) sse_route_kernel(const float *__restrict__ route, const float *__restrict__ klog,
                                                        long tokens, int N, int topk, int c, bool kstats,
                                                        uint32_t *__restrict__ rec, int32_t *__restrict__ sel_out,
                                                        int32_t *__restrict__ dev_err) {
  const int lane = threadIdx.x & 31;
  const long tok = static_cast<long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (tok >= tokens) return;  // warp-uniform
  const float *lg = route + tok * N;
  // two logits per lane: ids lane and lane + 32
  uint32_t key[2];
  int id[2];
  float lv[2];
  bool bad = false;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int j = lane + 32 * e;
    const bool in = j < N;
    lv[e] = in ? lg[j] : -INFINITY;
    bad |= in && !isfinite(lv[e]);
    key[e] = in ? order_key(lv[e]) : 0u;
    id[e] = in ? j : INT_MAX;
  }
  // softmax over all N logits
  const float lmax = key_value(__reduce_max_sync(kFull, max(key[0], key[1])));
  float z = 0.f;
#pragma unroll
  for (int e = 0; e < 2; ++e) z += (lane + 32 * e < N) ? expf(lv[e] - lmax) : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(kFull, z, off);
  // top-k: sort each lane's pair, then redux rounds
  if (key[1] > key[0] || (key[1] == key[0] && id[1] < id[0])) {
    const uint32_t tk = key[0]; key[0] = key[1]; key[1] = tk;
    const int ti = id[0]; id[0] = id[1]; id[1] = ti;
  }
  uint32_t *r = rec + tok * rec_words(topk);
  for (int s = 0; s < topk; ++s) {
    const uint32_t m = __reduce_max_sync(kFull, key[0]);
    const int wid = __reduce_min_sync(kFull, key[0] == m ? id[0] : INT_MAX);
    if (key[0] == m && id[0] == wid) {
      key[0] = key[1]; id[0] = id[1];
      key[1] = 0u; id[1] = INT_MAX;
    }
    if (lane == 0) {
      r[s] = static_cast<uint32_t>(wid);
      r[topk + s] = __float_as_uint(expf(key_value(m) - lmax) / z);
      if (sel_out) sel_out[tok * topk + s] = wid;
    }
  }
  // key-logit softmax statistics over the c rows (c <= 128: four per lane);
  // the chunked path computes them where it reads the logits
  if (!kstats) {
    if (__any_sync(kFull, bad) && lane == 0 && dev_err) atomicOr(dev_err, SDM_DEVERR_NONFINITE);
    return;
  }
  const float *kl = klog + tok * c;
  float kv[4];
  uint32_t km = 0u;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int j = lane + 32 * e;
    kv[e] = j < c ? kl[j] : -INFINITY;
    bad |= j < c && !isfinite(kv[e]);
    km = max(km, j < c ? order_key(kv[e]) : 0u);
  }
  const float kmax = key_value(__reduce_max_sync(kFull, km));
  float kz = 0.f;
#pragma unroll
  for (int e = 0; e < 4; ++e) kz += (lane + 32 * e < c) ? expf(kv[e] - kmax) : 0.f;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) kz += __shfl_xor_sync(kFull, kz, off);
  if (lane == 0) {
    r[2 * topk] = __float_as_uint(kmax);
    r[2 * topk + 1] = __float_as_uint(1.0f / kz);
  }
  if (__any_sync(kFull, bad) && lane == 0 && dev_err) atomicOr(dev_err, SDM_DEVERR_NONFINITE);
}

// ---------------------------------------------------------------------------
// The scan.
// ---------------------------------------------------------------------------
struct SseArgs {
  float *state;
  const float *klog, *alpha;
  const uint16_t *q, *v;
  const uint32_t *rec;
  float *y;
  int T, H, N, c, d, topk, tiles, rw, mode;
};

// per-token input slot, in 16-byte chunks: klog[c], alpha[c], q[c] bf16,
// v[16] bf16, routing record
struct SseSlot {
  static __host__ __device__ int klog_off() { return 0; }
  static __host__ __device__ int alpha_off(int c) { return c; }        // in words
  static __host__ __device__ int q_off(int c) { return 2 * c; }        // words
  static __host__ __device__ int v_off(int c) { return 2 * c + c / 2; }
  static __host__ __device__ int rec_off(int c) { return 2 * c + c / 2 + kSseDT / 2; }
  static __host__ __device__ int words(int c, int rw) { return rec_off(c) + rw; }
};

// packed fp32x2 helpers (one instruction for two lanes of math)
__device__ __forceinline__ unsigned long long pk(float x, float y) {
  return (static_cast<unsigned long long>(__float_as_uint(y)) << 32) | __float_as_uint(x);
}
__device__ __forceinline__ float2 upk(unsigned long long v) {
  return make_float2(__uint_as_float(static_cast<uint32_t>(v)), __uint_as_float(static_cast<uint32_t>(v >> 32)));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Thread (pair cp = tid % 8, row group rg = tid / 8) owns columns 2cp, 2cp+1
// of the tile and rows rg, rg+32, rg+64, rg+96 of every partition; the read
// is summed over the four row groups of a warp with shuffles, then over the
// eight warps through shared memory (summed after the next token's barrier).
constexpr int kSseRows = 32;  // row groups
constexpr int kSseRPT = 4;    // rows per thread (c <= 128)

template <int MODE>  // SSE_WRITE_ADDITIVE or SSE_WRITE_DELTA
__global__ void __launch_bounds__(kSseThreads) sse_scan_kernel(const SseArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;
  const int cp = tid & 7;
  const int rg = tid >> 3;
  const int tile = blockIdx.x % a.tiles;
  const long bh = blockIdx.x / a.tiles;
  const int h = static_cast<int>(bh % a.H);
  const long b = bh / a.H;
  const int c = a.c, d = a.d, N = a.N, T = a.T, H = a.H, topk = a.topk;
  const int parts = N + 1;

  float *S = reinterpret_cast<float *>(smem_raw);            // [parts][c][16]
  float *red = S + static_cast<size_t>(parts) * c * kSseDT;   // [2][8 warps][16]
  float *redv = red + 2 * 8 * kSseDT;  // delta write: [topk+1][8 warps][16] predictions
  uint32_t *ring = reinterpret_cast<uint32_t *>(redv + (MODE == SSE_WRITE_DELTA ? (kSseMaxTopk + 1) * 8 * kSseDT : 0));
  const int slot_words = SseSlot::words(c, a.rw);
  const int col0 = tile * kSseDT;

  float *gS = a.state + bh * static_cast<long>(parts) * c * d;
  for (int e = tid; e < parts * c * (kSseDT / 4); e += kSseThreads) {
    const int row = e / (kSseDT / 4), q4 = e % (kSseDT / 4);
    *reinterpret_cast<float4 *>(S + row * kSseDT + 4 * q4) =
        *reinterpret_cast<const float4 *>(gS + static_cast<long>(row) * d + col0 + 4 * q4);
  }

  const long tok0 = b * T * H + h;
  const int n_klog = c / 4, n_alpha = c / 4, n_q = c / 8, n_v = kSseDT / 8, n_rec = a.rw / 4;
  const int n_chunks = n_klog + n_alpha + n_q + n_v + n_rec;
  auto issue = [&](int t) {
    if (tid >= n_chunks) return;
    const long tok = tok0 + static_cast<long>(t) * H;
    uint32_t *sl = ring + (t % (kSseP + 1)) * slot_words;
    int q = tid;
    if (q < n_klog) { cp_async<16>(sl + SseSlot::klog_off() + 4 * q, a.klog + tok * c + 4 * q); return; }
    q -= n_klog;
    if (q < n_alpha) { cp_async<16>(sl + SseSlot::alpha_off(c) + 4 * q, a.alpha + tok * c + 4 * q); return; }
    q -= n_alpha;
    if (q < n_q) { cp_async<16>(sl + SseSlot::q_off(c) + 4 * q, a.q + tok * c + 8 * q); return; }
    q -= n_q;
    if (q < n_v) { cp_async<16>(sl + SseSlot::v_off(c) + 4 * q, a.v + tok * d + col0 + 8 * q); return; }
    q -= n_v;
    cp_async<16>(sl + SseSlot::rec_off(c) + 4 * q, a.rec + tok * a.rw + 4 * q);
  };
  for (int t = 0; t < kSseP; ++t) {
    if (t < T) issue(t);
    cp_async_commit();
  }

  auto emit_y = [&](int t) {  // threads 0..15: column tid, sum of the 8 warp partials of token t
    const float *rd = red + (t & 1) * 8 * kSseDT;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) acc += rd[w * kSseDT + tid];
    a.y[(tok0 + static_cast<long>(t) * H) * d + col0 + tid] = acc;
  };

  for (int t = 0; t < T; ++t) {
    cp_async_wait<kSseP - 1>();
    __syncthreads();
    if (t + kSseP < T) issue(t + kSseP);
    cp_async_commit();
    if (t > 0 && tid < kSseDT) emit_y(t - 1);
    const uint32_t *sl = ring + (t % (kSseP + 1)) * slot_words;
    const float *kl = reinterpret_cast<const float *>(sl + SseSlot::klog_off());
    const float *al = reinterpret_cast<const float *>(sl + SseSlot::alpha_off(c));
    const uint16_t *qq = reinterpret_cast<const uint16_t *>(sl + SseSlot::q_off(c));
    const uint32_t vw = sl[SseSlot::v_off(c) + cp];  // bf16 pair: columns 2cp, 2cp+1
    const uint32_t *rc = sl + SseSlot::rec_off(c);
    const float kmax = __uint_as_float(rc[2 * topk]);
    const float kinv = __uint_as_float(rc[2 * topk + 1]);
    const unsigned long long v2 = pk(bf16_to_f32(vw & 0xffff), bf16_to_f32(vw >> 16));
    // per own row: decay pair, key weight kk_j, query q_j
    unsigned long long a2[kSseRPT], q2[kSseRPT];
    float kk[kSseRPT];
    bool in[kSseRPT];
#pragma unroll
    for (int i = 0; i < kSseRPT; ++i) {
      const int j = rg + kSseRows * i;
      in[i] = j < c;
      const int jj = in[i] ? j : 0;
      kk[i] = __expf(kl[jj] - kmax) * kinv;
      a2[i] = pk(al[jj], al[jj]);
      const float qv = bf16_to_f32(qq[jj]);
      q2[i] = pk(qv, qv);
    }
    if (MODE == SSE_WRITE_DELTA) {
      // the decayed prediction of every visited partition, summed over rows
      for (int s = 0; s <= topk; ++s) {
        const int p = s < topk ? static_cast<int>(rc[s]) : N;
        const float *Sp = S + static_cast<size_t>(p) * c * kSseDT + 2 * cp;
        unsigned long long acc = 0ull;
#pragma unroll
        for (int i = 0; i < kSseRPT; ++i) {
          if (in[i]) {
            const int j = rg + kSseRows * i;
            const float ka = kk[i] * al[j];
            acc = fma2(pk(ka, ka), *reinterpret_cast<const unsigned long long *>(Sp + j * kSseDT), acc);
          }
        }
        float2 pv = upk(acc);
#pragma unroll
        for (int m = 8; m <= 16; m <<= 1) {
          pv.x += __shfl_xor_sync(kFull, pv.x, m);
          pv.y += __shfl_xor_sync(kFull, pv.y, m);
        }
        if (lane < 8) *reinterpret_cast<float2 *>(redv + (s * 8 + warp) * kSseDT + 2 * cp) = pv;
      }
      __syncthreads();
    }
    unsigned long long part = 0ull;
    for (int s = 0; s <= topk; ++s) {
      const int p = s < topk ? static_cast<int>(rc[s]) : N;
      const float g = s < topk ? __uint_as_float(rc[topk + s]) : 1.0f;
      float *Sp = S + static_cast<size_t>(p) * c * kSseDT + 2 * cp;
      unsigned long long src = v2;  // what is written: v (additive) or v - vhat_p (delta)
      if (MODE == SSE_WRITE_DELTA) {
        float2 vh = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < 8; ++w) {
          const float2 t2 = *reinterpret_cast<const float2 *>(redv + (s * 8 + w) * kSseDT + 2 * cp);
          vh.x += t2.x;
          vh.y += t2.y;
        }
        const float2 vf = upk(v2);
        src = pk(vf.x - vh.x, vf.y - vh.y);
      }
      unsigned long long inner = 0ull;
#pragma unroll
      for (int i = 0; i < kSseRPT; ++i) {
        if (in[i]) {
          const int j = rg + kSseRows * i;
          unsigned long long *cell = reinterpret_cast<unsigned long long *>(Sp + j * kSseDT);
          const float gk = g * kk[i];
          const unsigned long long x = fma2(a2[i], *cell, mul2(pk(gk, gk), src));  // alpha_j S + g kk_j src
          *cell = x;
          inner = fma2(q2[i], x, inner);
        }
      }
      part = fma2(pk(g, g), inner, part);
    }
    float2 pv = upk(part);
#pragma unroll
    for (int m = 8; m <= 16; m <<= 1) {  // the warp's four row groups
      pv.x += __shfl_xor_sync(kFull, pv.x, m);
      pv.y += __shfl_xor_sync(kFull, pv.y, m);
    }
    if (lane < 8) *reinterpret_cast<float2 *>(red + (t & 1) * 8 * kSseDT + warp * kSseDT + 2 * cp) = pv;
  }
  cp_async_wait<0>();
  __syncthreads();
  if (T > 0 && tid < kSseDT) emit_y(T - 1);
  for (int e = tid; e < parts * c * (kSseDT / 4); e += kSseThreads) {
    const int row = e / (kSseDT / 4), q4 = e % (kSseDT / 4);
    *reinterpret_cast<float4 *>(gS + static_cast<long>(row) * d + col0 + 4 * q4) =
        *reinterpret_cast<const float4 *>(S + row * kSseDT + 4 * q4);
  }
}

size_t sse_smem_bytes(int N, int c, int topk, int mode) {
  const size_t pred = mode == SSE_WRITE_DELTA ? (kSseMaxTopk + 1) * 8 * kSseDT : 0;
  return sizeof(float) * (static_cast<size_t>(N + 1) * c * kSseDT + 2 * 8 * kSseDT + pred) +
         sizeof(uint32_t) * (kSseP + 1) * SseSlot::words(c, rec_words(topk));
}

}  // namespace
}  // namespace sdm

using namespace sdm;

namespace sdm {
size_t sse_chunk_workspace_size(int B, int T, int H, int N, int topk, int write_mode);
bool sse_chunk_supported(int write_mode, int N, int topk, int c, int d);
int launch_sse_chunk(float *state, const uint32_t *rec, int rw, const float *klog, const uint16_t *q,
                     const uint16_t *v, const float *alpha, int write_mode, int B, int T, int H, int N, int topk,
                     float *y, unsigned char *chunk_ws, int32_t *err, cudaStream_t st);
}  // namespace sdm

// Both writes with c = d = 128 run as a chunked prefill by partition once T
// reaches one chunk (the additive write in sse_chunk.cu's GLA chunk form, the
// delta write in the KDA chunk form of gdn_chunk.cu); other shapes and short
// sequences run token by token.  SDM_SSE_PATH=recurrent forces the
// token-by-token kernel, SDM_SSE_PATH=chunk the chunked path for any T.
static bool use_sse_chunk(int write_mode, int T, int N, int topk, int c, int d) {
  if (!sse_chunk_supported(write_mode, N, topk, c, d)) return false;
  const char *path = getenv("SDM_SSE_PATH");
  if (path && strcmp(path, "recurrent") == 0) return false;
  if (path && strcmp(path, "chunk") == 0) return true;
  return T >= 64;
}

static size_t rec_bytes(int B, int T, int H, int topk) {
  const size_t n = static_cast<size_t>(B) * T * H * rec_words(topk) * sizeof(uint32_t);
  return (n + 255) & ~static_cast<size_t>(255);
}

extern "C" size_t sse_scan_workspace_size(int B, int T, int H, int N, int topk, int c, int d, int write_mode) {
  if (B <= 0 || T <= 0 || H <= 0 || N <= 0 || topk <= 0) return 0;
  size_t n = rec_bytes(B, T, H, topk);
  if (use_sse_chunk(write_mode, T, N, topk, c, d)) n += sse_chunk_workspace_size(B, T, H, N, topk, write_mode);
  return n;
}

extern "C" int sse_scan(float *state, const float *route_logits, int topk, const float *k_logits, const uint16_t *q,
                        const uint16_t *v, const float *alpha, int write_mode, int B, int T, int H, int N, int c, int d,
                        float *y,
                        int32_t *sel_out, void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream) {
  if (!state || !route_logits || !k_logits || !q || !v || !alpha || !y)
    return set_error(SDM_ERR_INVALID_ARG, "sse_scan: null pointer");
  if (B < 0 || T < 0 || H < 0) return set_error(SDM_ERR_INVALID_ARG, "sse_scan: negative size");
  if (write_mode != SSE_WRITE_ADDITIVE && write_mode != SSE_WRITE_DELTA)
    return set_error(SDM_ERR_UNSUPPORTED, "sse_scan: write_mode must be SSE_WRITE_ADDITIVE or SSE_WRITE_DELTA");
  if (N < 1 || N > 64 || topk < 1 || topk > N || topk > kSseMaxTopk)
    return set_error(SDM_ERR_SHAPE, "sse_scan: need 1 <= topk <= min(N, 8), N <= 64");
  if (c < 16 || c > 128 || c % 16 != 0 || d < kSseDT || d % kSseDT != 0)
    return set_error(SDM_ERR_SHAPE, "sse_scan: need c %% 16 == 0, 16 <= c <= 128, d %% 16 == 0");
  int dev = 0, smem_blk = 0;
  if (!aligned(state, 16) || !aligned(y, 4) || !aligned(k_logits, 16) || !aligned(alpha, 16) ||
      !aligned(q, 16) || !aligned(v, 16) || !aligned(route_logits, 4) || (sel_out && !aligned(sel_out, 4)) ||
      (dev_err && !aligned(dev_err, 4)))
    return set_error(SDM_ERR_ALIGN, "sse_scan: state, k_logits, alpha, q, v need 16-byte alignment");
  if (B == 0 || T == 0 || H == 0) return SDM_OK;
  if (static_cast<long>(B) * T * H * (topk + 1) >= INT_MAX || T >= (1 << 27))
    return set_error(SDM_ERR_SHAPE, "sse_scan: B*T*H*(topk+1) must stay below 2^31 and T below 2^27");
  const size_t need = sse_scan_workspace_size(B, T, H, N, topk, c, d, write_mode);
  if (!workspace || workspace_bytes < need)
    return set_error(SDM_ERR_INVALID_ARG, "sse_scan: workspace of %zu bytes needed", need);
  if (!aligned(workspace, 16)) return set_error(SDM_ERR_ALIGN, "sse_scan: workspace must be 16-byte aligned");
  const bool chunk = use_sse_chunk(write_mode, T, N, topk, c, d);
  const size_t smem = sse_smem_bytes(N, c, topk, write_mode);
  if (chunk) {
    if (!aligned(y, 16)) return set_error(SDM_ERR_ALIGN, "sse_scan: y must be 16-byte aligned");
  } else {
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (smem > static_cast<size_t>(smem_blk))
      return set_error(SDM_ERR_SHAPE, "sse_scan: (N+1)*c too large for the shared-memory resident state");
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long tokens = static_cast<long>(B) * T * H;
  uint32_t *rec = static_cast<uint32_t *>(workspace);
  if (chunk && N <= kRouteThreadN)
    sse_route_thread_kernel<<<static_cast<unsigned>((tokens + 255) / 256), 256, 0, st>>>(route_logits, tokens, N, topk,
                                                                                       rec, sel_out, dev_err);
  else
    sse_route_kernel<<<static_cast<unsigned>((tokens + 7) / 8), 256, 0, st>>>(route_logits, k_logits, tokens, N,
                                                                             topk, c, !chunk, rec, sel_out, dev_err);
  int rc = check_launch("sse_scan: route kernel");
  if (rc != SDM_OK) return rc;

  if (chunk)
    return launch_sse_chunk(state, rec, rec_words(topk), k_logits, q, v, alpha, write_mode, B, T, H, N, topk, y,
                            static_cast<unsigned char *>(workspace) + rec_bytes(B, T, H, topk), dev_err, st);

  SseArgs args;
  args.state = state;
  args.klog = k_logits;
  args.alpha = alpha;
  args.q = q;
  args.v = v;
  args.rec = rec;
  args.y = y;
  args.T = T;
  args.H = H;
  args.N = N;
  args.c = c;
  args.d = d;
  args.topk = topk;
  args.tiles = d / kSseDT;
  args.rw = rec_words(topk);
  args.mode = write_mode;
  auto kern = write_mode == SSE_WRITE_DELTA ? sse_scan_kernel<SSE_WRITE_DELTA> : sse_scan_kernel<SSE_WRITE_ADDITIVE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return check_launch("sse_scan: set shared memory");
  const long blocks = static_cast<long>(B) * H * args.tiles;
  kern<<<static_cast<unsigned>(blocks), kSseThreads, smem, st>>>(args);
  return check_launch("sse_scan: scan kernel");
}
