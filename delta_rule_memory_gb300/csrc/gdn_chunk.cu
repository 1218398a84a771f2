// gdn_chunk.cu - dense Gated DeltaNet scan in chunkwise (WY / triangular-solve)
// form on the tcgen05 tensor cores (Sparse Delta Memory deck, App. A.1-A.2,
// Eq. 7, dense case; Linear Attention Architectures deck, "GDN and KDA change
// the granularity of forgetting", Eqs. 15-17).
//
// Within a chunk of C = 64 tokens, with lambda_i = sum_{j<=i} log alpha_j,
// gamma_i = exp(lambda_i), the token recurrence is equivalent to
//   (I + A) U = diag(beta) (V - diag(gamma) K S0),  A_ij = beta_i e^{l_i-l_j} k_i.k_j (j < i)
//   Y   = diag(gamma) Q S0 + Mq U,                  Mq_ij = e^{l_i-l_j} q_i.k_j   (j <= i)
//   S_C = gamma_C S0 + Khat^T U,                    Khat_j = e^{l_C-l_j} k_j
// Every state contraction is written transposed so that its M dimension is
// d_v = 128 and the state S^T (d_v x d_k, fp32) stays in tensor memory as an
// accumulator for the whole sequence.  Operands that are not exact in bf16
// (the state, R, U, T, Mq, Khat) are split into bf16 hi + lo and multiplied
// as hi*hi + hi*lo + lo*hi, which keeps fp32-level accuracy.  Decay ratios
// are always formed as exp(l_i - l_j) with j <= i.
//
// One CTA (256 threads, one tensor-memory allocation of 512 columns) runs one
// (batch, head) sequence chunk by chunk.  Thread (row d = tid % 128,
// half = tid / 128) owns tensor-memory lane d and half of each tile's columns.
#include <climits>

#include "common.cuh"
#include "umma.cuh"

namespace sdm {
namespace {

using namespace umma;

constexpr int kC = 64;      // tokens per chunk
constexpr int kDK = 128;    // key width
constexpr int kDV = 128;    // value width (the MMA M)
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 20;  // polls (about 0.1 s) before an mbarrier wait gives up

// tensor-memory columns (fp32)
constexpr uint32_t kColS = 0;     // S^T          [128 x 128]
constexpr uint32_t kColGP = 128;  // [K;Q] K^T    [128 x 64]: rows 0..63 = K K^T, 64..127 = Q K^T
constexpr uint32_t kColX = 192;   // S0^T K^T     [128 x 64]
constexpr uint32_t kColY1 = 256;  // S0^T Q^T     [128 x 64]
constexpr uint32_t kColU = 320;   // U^T          [128 x 64]
constexpr uint32_t kColY2 = 384;  // U^T Mq^T     [128 x 64]
constexpr uint32_t kTmemCols = 512;

// shared memory (bytes); operand tiles are K-major, no swizzle (umma.cuh)
constexpr uint32_t kOffKQ = 0;                            // [K;Q]: 128 rows x 128, bf16          32 KB
constexpr uint32_t kOffSh = kOffKQ + 128 * kDK * 2;       // S^T hi: 128 x 128 bf16               32 KB
constexpr uint32_t kOffSl = kOffSh + 128 * kDK * 2;       // S^T lo                               32 KB
constexpr uint32_t kOffRU = kOffSl + 128 * kDK * 2;       // R^T / U^T hi+lo: 2 x 128 x 64 bf16   32 KB
constexpr uint32_t kOffT = kOffRU + 2 * 128 * kC * 2;     // T hi+lo: 2 x 64 x 64 bf16            16 KB
constexpr uint32_t kOffM = kOffT + 2 * kC * kC * 2;       // Mq hi+lo                             16 KB
constexpr uint32_t kOffKh = kOffM + 2 * kC * kC * 2;      // Khat^T hi+lo: 2 x 128 x 64 bf16      32 KB
constexpr uint32_t kOffGate = kOffKh + 2 * 128 * kC * 2;  // per buffer: log alpha, beta, lambda, gamma, e^(l_C-l_j)
constexpr uint32_t kOffBar = kOffGate + 10 * kC * 4;
constexpr uint32_t kSmemBytes = kOffBar + 64;
// scratch views during the triangular solve (regions free at that time)
constexpr int kLd = kC + 1;                        // padded fp32 row stride
constexpr uint32_t kOffA = kOffKh;                 // L = I + A, fp32 [64][65]
constexpr uint32_t kOffTf = kOffRU;                // L^-1, fp32 [64][65]
constexpr uint32_t kOffZ = kOffRU + kC * kLd * 4;  // block products, fp32 [3][16][16]
static_assert(kC * kLd * 4 <= 2 * 128 * kC * 2, "A fits in the Khat region");
static_assert(kC * kLd * 4 + 3 * 256 * 4 <= 2 * 128 * kC * 2, "L^-1 and Z fit in the R/U region");

struct ChunkArgs {
  float *state;
  const uint16_t *q, *k, *v;
  const float *alpha, *beta;
  float *y;
  int T, H;
  int32_t *err;
};

__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, int lane_base, uint32_t col) {
  return base + (static_cast<uint32_t>(lane_base) << 16) + col;
}

// 8 consecutive fp32 -> one 16-byte chunk of bf16 hi and one of bf16 lo
// (hi = bf16(x), lo = bf16(x - hi), converted two at a time)
__device__ __forceinline__ void store_split8(unsigned char *hi, unsigned char *lo, uint32_t off, const float *x) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 hb = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    const float2 hf = __bfloat1622float2(hb);
    const __nv_bfloat162 lb = __floats2bfloat162_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y);
    h[e] = *reinterpret_cast<const uint32_t *>(&hb);
    l[e] = *reinterpret_cast<const uint32_t *>(&lb);
  }
  *reinterpret_cast<uint4 *>(hi + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4 *>(lo + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// issue `ksteps` MMAs of K = 16 into d (M = 128, N); A and B K-major tiles
// whose rows hold ka and kb elements
__device__ __forceinline__ void mma_tile(uint32_t d, uint32_t a, int ka, uint32_t b, int kb, int ksteps, int N,
                                         bool accumulate) {
  const uint32_t idesc = idesc_bf16_f32(128, N);
  for (int s = 0; s < ksteps; ++s) {
    const uint64_t ad = smem_desc(a + s * 256, 128, ka * 16);
    const uint64_t bd = smem_desc(b + s * 256, 128, kb * 16);
    mma_bf16(d, ad, bd, idesc, accumulate || s > 0);
  }
}

__global__ void __launch_bounds__(kThreads, 1) gdn_chunk_kernel(const ChunkArgs a) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int row = tid & 127;  // tensor-memory lane / value row d
  const int half = tid >> 7;  // which half of each tile's columns
  const int lane_base = 32 * (warp & 3);
  const long bh = blockIdx.x;
  const int h = static_cast<int>(bh % a.H);
  const long b = bh / a.H;
  const int T = a.T, H = a.H;
  const long tok0 = b * T * H + h;  // token t -> tok0 + t*H

  unsigned char *sKQ = sm + kOffKQ, *sSh = sm + kOffSh, *sSl = sm + kOffSl;
  unsigned char *sRh = sm + kOffRU, *sRl = sm + kOffRU + 128 * kC * 2;
  unsigned char *sTh = sm + kOffT, *sTl = sm + kOffT + kC * kC * 2;
  unsigned char *sMh = sm + kOffM, *sMl = sm + kOffM + kC * kC * 2;
  unsigned char *sKhh = sm + kOffKh, *sKhl = sm + kOffKh + 128 * kC * 2;
  float *gate = reinterpret_cast<float *>(sm + kOffGate);  // [2 buffers][log alpha, beta, lambda, gamma, tail][64]
  float *sA = reinterpret_cast<float *>(sm + kOffA);
  float *sTf = reinterpret_cast<float *>(sm + kOffTf);
  float *sZ = reinterpret_cast<float *>(sm + kOffZ);
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kOffBar);
  uint32_t *holder = reinterpret_cast<uint32_t *>(sm + kOffBar + 40);
  const uint32_t mbGP = smem_addr(bars + 0), mbXY = smem_addr(bars + 1), mbU = smem_addr(bars + 2),
                 mbYS = smem_addr(bars + 3), mbEnd = smem_addr(bars + 4);

  if (tid == 0) {
    mbar_init(mbGP, 1);
    mbar_init(mbXY, 1);
    mbar_init(mbU, 1);
    mbar_init(mbYS, 1);
    mbar_init(mbEnd, 1);
  }
  if (warp == 0) tmem_alloc(smem_addr(holder), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  bool failed = false;
  // every thread waits, then the CTA agrees: either all continue or all stop
  auto wait_ok = [&](uint32_t mb, uint32_t parity) -> bool {
    const bool ok = mbar_wait(mb, parity, kWaitLimit);
    tc_fence_after();
    return __syncthreads_and(ok) != 0;
  };

  // ---- the initial state: S^T into tensor memory and its bf16 split into smem
  float *gS = a.state + bh * kDK * kDV;
  for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
    float x[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) x[e] = gS[static_cast<long>(c0 + e) * kDV + row];  // S[c][d]
    tmem_st16(tmem_addr(tmem, lane_base, kColS + c0), x);
    store_split8(sSh, sSl, kmajor_off(row, c0, kDK), x);
    store_split8(sSh, sSl, kmajor_off(row, c0 + 8, kDK), x + 8);
  }
  tmem_st_wait();

  // ---- per-chunk inputs: K and Q rows into the [K;Q] tile, gates into smem
  auto load_chunk = [&](int c, int buf) {
    const int t0 = c * kC;
    for (int id = tid; id < 128 * (kDK / 8); id += kThreads) {
      const int r = id >> 4, k8 = id & 15;
      const int t = t0 + (r & 63);
      unsigned char *dst = sKQ + kmajor_off(r, k8 * 8, kDK);
      if (t < T) {
        const uint16_t *src = (r < 64 ? a.k : a.q) + (tok0 + static_cast<long>(t) * H) * kDK + k8 * 8;
        cp_async<16>(dst, src);
      } else {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    if (tid < kC) {
      const int t = t0 + tid;
      float *g = gate + buf * 5 * kC;
      g[tid] = t < T ? __logf(a.alpha[tok0 + static_cast<long>(t) * H]) : 0.f;  // padding: alpha = 1
      g[kC + tid] = t < T ? a.beta[tok0 + static_cast<long>(t) * H] : 0.f;       // padding: beta = 0
    }
  };
  // this thread's 32 values of V for a chunk (column d, tokens half*32 ..)
  uint16_t vreg[32];
  auto load_v = [&](int c) {
    const int t0 = c * kC + half * 32;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int t = t0 + i;
      vreg[i] = t < T ? a.v[(tok0 + static_cast<long>(t) * H) * kDV + row] : static_cast<uint16_t>(0);
    }
  };

  const int nchunks = (T + kC - 1) / kC;
  if (nchunks > 0) {
    load_chunk(0, 0);
    load_v(0);
  }
  cp_async_commit();
  for (int c = 0; c < nchunks; ++c) {
    const int buf = c & 1;
    const uint32_t par = static_cast<uint32_t>(c & 1);
    float *g = gate + buf * 5 * kC;  // [0]: log alpha, [1]: beta, [2]: lambda, [3]: gamma, [4]: e^(l_C - l_j)
    cp_async_wait<0>();
    // lambda = inclusive prefix sum of log alpha (two warps of 32 tokens)
    if (warp < 2) {
      float x = g[tid];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(kFull, x, o);
        if ((tid & 31) >= o) x += y;
      }
      g[2 * kC + tid] = x;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) g[2 * kC + tid] += g[2 * kC + 31];
    __syncthreads();
    if (tid < kC) {
      g[3 * kC + tid] = __expf(g[2 * kC + tid]);
      g[4 * kC + tid] = __expf(g[2 * kC + kC - 1] - g[2 * kC + tid]);
    }
    tc_fence_after();

    // ---- MMAs that need only the chunk's K, Q and the incoming state
    if (tid == 0) {
      const uint32_t kq = smem_addr(sKQ);
      const uint32_t kblk = kq, qblk = kq + 8 * (kDK * 16);  // rows 0..63 = K, 64..127 = Q
      mma_tile(tmem + kColGP, kq, kDK, kblk, kDK, kDK / 16, kC, false);  // [K;Q] K^T
      mma_commit(mbGP);
      mma_tile(tmem + kColX, smem_addr(sSh), kDK, kblk, kDK, kDK / 16, kC, false);  // S^T K^T
      mma_tile(tmem + kColX, smem_addr(sSl), kDK, kblk, kDK, kDK / 16, kC, true);
      mma_tile(tmem + kColY1, smem_addr(sSh), kDK, qblk, kDK, kDK / 16, kC, false);  // S^T Q^T
      mma_tile(tmem + kColY1, smem_addr(sSl), kDK, qblk, kDK, kDK / 16, kC, true);
      mma_commit(mbXY);
    }

    // ---- A (decayed, gated K K^T) and Mq (decayed Q K^T) from the GP tile
    if (!wait_ok(mbGP, par)) { failed = true; break; }
    const float *lam = g + 2 * kC;
    {
      const int i = row & 63;
      const float li = lam[i];
      const float bi = g[kC + i];
      for (int j0 = half * 32; j0 < half * 32 + 32; j0 += 16) {
        float x[16];
        tmem_ld16(tmem_addr(tmem, lane_base, kColGP + j0), x);
        tmem_ld_wait();
        if (row < 64) {  // strictly lower part of L = I + A (the unit diagonal is implicit)
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = j0 + e;
            sA[i * kLd + j] = j < i ? bi * __expf(li - lam[j]) * x[e] : 0.f;
          }
        } else {  // Mq, lower part including the diagonal
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = j0 + e;
            x[e] = j <= i ? __expf(li - lam[j]) * x[e] : 0.f;
          }
          store_split8(sMh, sMl, kmajor_off(i, j0, kC), x);
          store_split8(sMh, sMl, kmajor_off(i, j0 + 8, kC), x + 8);
        }
      }
    }
    __syncthreads();

    // ---- T = (I + A)^-1 diag(beta): 16x16 diagonal blocks by substitution ...
    if (tid < 64) {
      const int I = tid >> 4, cc = tid & 15, o = I * 16;
      float xv[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) {
        float acc = (r == cc) ? 1.f : 0.f;
#pragma unroll
        for (int j = 0; j < r; ++j) acc -= sA[(o + r) * kLd + o + j] * xv[j];
        xv[r] = acc;
      }
#pragma unroll
      for (int r = 0; r < 16; ++r) sTf[(o + r) * kLd + o + cc] = xv[r];
    }
    __syncthreads();
    // ... then the blocks below the diagonal, one block distance at a time:
    // X_IJ = -L_II^-1 sum_{K=J}^{I-1} L_IK X_KJ
    for (int dist = 1; dist < 4; ++dist) {
      const int npairs = 4 - dist;
      for (int oi = tid; oi < npairs * 256; oi += kThreads) {
        const int p = oi >> 8, r = (oi >> 4) & 15, cc = oi & 15;
        const int J = p, I = p + dist;
        float acc = 0.f;
        for (int K = J; K < I; ++K)
#pragma unroll
          for (int kk = 0; kk < 16; ++kk)
            acc += sA[(I * 16 + r) * kLd + K * 16 + kk] * sTf[(K * 16 + kk) * kLd + J * 16 + cc];
        sZ[p * 256 + r * 16 + cc] = acc;
      }
      __syncthreads();
      for (int oi = tid; oi < npairs * 256; oi += kThreads) {
        const int p = oi >> 8, r = (oi >> 4) & 15, cc = oi & 15;
        const int J = p, I = p + dist;
        float acc = 0.f;
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) acc += sTf[(I * 16 + r) * kLd + I * 16 + kk] * sZ[p * 256 + kk * 16 + cc];
        sTf[(I * 16 + r) * kLd + J * 16 + cc] = -acc;
      }
      __syncthreads();
    }
    // T = L^-1 diag(beta) (lower triangle), split into the B-operand tile
    {
      const int i = tid >> 2, j0 = (tid & 3) * 16;
      float x[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = j0 + e;
        x[e] = j <= i ? sTf[i * kLd + j] * g[kC + j] : 0.f;
      }
      store_split8(sTh, sTl, kmajor_off(i, j0, kC), x);
      store_split8(sTh, sTl, kmajor_off(i, j0 + 8, kC), x + 8);
    }
    __syncthreads();  // sA (in the Khat region) is no longer read
    // Khat^T[c][j] = exp(lambda_C - lambda_j) k_j[c] (B operand of the state update)
    {
      const float *tail = g + 4 * kC;  // e^(lambda_C - lambda_j)
      for (int j0 = half * 32; j0 < half * 32 + 32; j0 += 8) {
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int j = j0 + e;
          const uint16_t kb = *reinterpret_cast<const uint16_t *>(sKQ + kmajor_off(j, row, kDK));
          x[e] = tail[j] * bf16_to_f32(kb);
        }
        store_split8(sKhh, sKhl, kmajor_off(row, j0, kC), x);
      }
    }

    // ---- R^T = V^T - (S0^T K^T) diag(gamma), split into the A-operand tile
    if (!wait_ok(mbXY, par)) { failed = true; break; }
    {
      const float *gam = g + 3 * kC;
      for (int i0 = half * 32; i0 < half * 32 + 32; i0 += 16) {
        float x[16];
        tmem_ld16(tmem_addr(tmem, lane_base, kColX + i0), x);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = bf16_to_f32(vreg[i0 - half * 32 + e]) - gam[i0 + e] * x[e];
        store_split8(sRh, sRl, kmajor_off(row, i0, kC), x);
        store_split8(sRh, sRl, kmajor_off(row, i0 + 8, kC), x + 8);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the chunk's K, Q and V are consumed: prefetch the next chunk
    if (c + 1 < nchunks) {
      load_chunk(c + 1, buf ^ 1);
      load_v(c + 1);
    }
    cp_async_commit();

    // ---- U^T = R^T T^T
    if (tid == 0) {
      const uint32_t rh = smem_addr(sRh), rl = smem_addr(sRl), th = smem_addr(sTh), tl = smem_addr(sTl);
      mma_tile(tmem + kColU, rh, kC, th, kC, kC / 16, kC, false);
      mma_tile(tmem + kColU, rh, kC, tl, kC, kC / 16, kC, true);
      mma_tile(tmem + kColU, rl, kC, th, kC, kC / 16, kC, true);
      mma_commit(mbU);
    }
    if (!wait_ok(mbU, par)) { failed = true; break; }
    // U^T split into the A-operand tile (over R, whose reads are complete);
    // S^T scaled by gamma_C in tensor memory before the state update
    {
      for (int i0 = half * 32; i0 < half * 32 + 32; i0 += 16) {
        float x[16];
        tmem_ld16(tmem_addr(tmem, lane_base, kColU + i0), x);
        tmem_ld_wait();
        store_split8(sRh, sRl, kmajor_off(row, i0, kC), x);
        store_split8(sRh, sRl, kmajor_off(row, i0 + 8, kC), x + 8);
      }
      const float gC = g[3 * kC + kC - 1];
      for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
        float x[16];
        tmem_ld16(tmem_addr(tmem, lane_base, kColS + c0), x);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] *= gC;
        tmem_st16(tmem_addr(tmem, lane_base, kColS + c0), x);
      }
      tmem_st_wait();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- Y2^T = U^T Mq^T and S^T += U^T Khat
    if (tid == 0) {
      const uint32_t uh = smem_addr(sRh), ul = smem_addr(sRl);
      const uint32_t mh = smem_addr(sMh), ml = smem_addr(sMl), kh = smem_addr(sKhh), kl = smem_addr(sKhl);
      mma_tile(tmem + kColY2, uh, kC, mh, kC, kC / 16, kC, false);
      mma_tile(tmem + kColY2, uh, kC, ml, kC, kC / 16, kC, true);
      mma_tile(tmem + kColY2, ul, kC, mh, kC, kC / 16, kC, true);
      mma_tile(tmem + kColS, uh, kC, kh, kC, kC / 16, kDK, true);
      mma_tile(tmem + kColS, uh, kC, kl, kC, kC / 16, kDK, true);
      mma_tile(tmem + kColS, ul, kC, kh, kC, kC / 16, kDK, true);
      mma_commit(mbYS);
    }
    if (!wait_ok(mbYS, par)) { failed = true; break; }

    // ---- y = gamma_i (S0^T Q^T)[:, i] + (U^T Mq^T)[:, i], and the new state's split
    {
      const float *gam = g + 3 * kC;
      const int t0 = c * kC;
      for (int i0 = half * 32; i0 < half * 32 + 32; i0 += 16) {
        float y1[16], y2[16];
        tmem_ld16(tmem_addr(tmem, lane_base, kColY1 + i0), y1);
        tmem_ld16(tmem_addr(tmem, lane_base, kColY2 + i0), y2);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int t = t0 + i0 + e;
          if (t < T) a.y[(tok0 + static_cast<long>(t) * H) * kDV + row] = fmaf(gam[i0 + e], y1[e], y2[e]);
        }
      }
      for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
        float x[16];
        tmem_ld16(tmem_addr(tmem, lane_base, kColS + c0), x);
        tmem_ld_wait();
        store_split8(sSh, sSl, kmajor_off(row, c0, kDK), x);
        store_split8(sSh, sSl, kmajor_off(row, c0 + 8, kDK), x + 8);
      }
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  cp_async_wait<0>();
  if (failed) {
    // stop cleanly: wait (bounded) for this CTA's tensor-core work, report
    if (tid == 0) mma_commit(mbEnd);
    mbar_wait(mbEnd, 0, kWaitLimit);
    if (tid == 0 && a.err) atomicOr(a.err, SDM_DEVERR_TIMEOUT);
  } else {
    // ---- the final state back to HBM (S[c][d] = S^T[d][c])
    for (int c0 = half * 64; c0 < half * 64 + 64; c0 += 16) {
      float x[16];
      tmem_ld16(tmem_addr(tmem, lane_base, kColS + c0), x);
      tmem_ld_wait();
#pragma unroll
      for (int e = 0; e < 16; ++e) gS[static_cast<long>(c0 + e) * kDV + row] = x[e];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

// launched by gdn_scan for dense GDN with d_k = d_v = 128
int launch_gdn_chunk(float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                     const float *beta, int B, int T, int H, float *y, int32_t *err, cudaStream_t st) {
  ChunkArgs args;
  args.state = state;
  args.q = q;
  args.k = k;
  args.v = v;
  args.alpha = alpha;
  args.beta = beta;
  args.y = y;
  args.T = T;
  args.H = H;
  args.err = err;
  if (cudaFuncSetAttribute(gdn_chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kSmemBytes)) != cudaSuccess)
    return check_launch("gdn_scan: set shared memory");
  gdn_chunk_kernel<<<static_cast<unsigned>(static_cast<long>(B) * H), kThreads, kSmemBytes, st>>>(args);
  return check_launch("gdn_scan: chunk kernel");
}

}  // namespace sdm
