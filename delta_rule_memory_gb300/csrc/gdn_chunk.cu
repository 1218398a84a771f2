// gdn_chunk.cu - dense Gated DeltaNet scan in chunkwise (WY / triangular-solve)
// form on the tcgen05 tensor cores (Sparse Delta Memory deck, App. A.1-A.2,
// Eq. 7, dense case; Linear Attention Architectures deck, "GDN and KDA change
// the granularity of forgetting", Eqs. 15-17).
//
// Within a chunk of C = 64 tokens, with lambda_i = sum_{j<=i} log alpha_j,
// gamma_i = exp(lambda_i), L = I + A, A_ij = beta_i e^{l_i-l_j} k_i.k_j (j < i)
// and T = L^-1 diag(beta), the token recurrence is equivalent to
//   U   = T V - T diag(gamma) K S0 = Ut - W S0
//   Y   = diag(gamma) Q S0 + Mq U,     Mq_ij = e^{l_i-l_j} q_i.k_j   (j <= i)
//   S_C = gamma_C S0 + Khat^T U,       Khat_j = e^{l_C-l_j} k_j
// Only the products with S0 and with U depend on the state, so the work is
// split in two kernels:
//   gdn_prep_kernel  - every chunk in parallel (persistent CTAs): A, the
//                      triangular inverse, T, then W and Ut by MMA, Mq and
//                      Khat, written to the workspace as ready-made operand
//                      tiles of the second kernel.
//   gdn_chain_pair_kernel - two CTAs per (batch, head), each owning 64 of
//                      the value columns, chunk after chunk: two rounds of
//                      MMAs on the state (fp32, held in the registers of the
//                      worker warps), fed by a producer warp; the next
//                      chunk's tiles stream in with bulk asynchronous copies
//                      meanwhile.  Every contraction has M = 128 (tokens of
//                      [W; Q], or key channels) and N = 64 (the columns).
//   gdn_chain_kernel - the same chain on one CTA per (batch, head), taken
//                      when the pairs would not all be resident at once;
//                      there every state contraction is written transposed
//                      so that its M is d_v = 128.
// Operands that are not exact in bf16 (state, U, T, W, Mq, Khat) are split
// into bf16 hi + lo and multiplied as hi*hi + hi*lo + lo*hi, which keeps
// fp32-level accuracy.  Decay ratios are always formed as exp(l_i - l_j) with
// j <= i.
#include <climits>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "sse_group.cuh"
#include "umma.cuh"

namespace sdm {
namespace {

using namespace umma;

constexpr int kC = 64;      // tokens per chunk
constexpr int kDK = 128;    // key width
constexpr int kDV = 128;    // value width (the MMA M)
constexpr int kThreads = 256;
constexpr uint32_t kWaitLimit = 1u << 20;  // polls (about 0.1 s) before an mbarrier wait gives up

// ---- one chunk's tiles in the workspace (bytes; K-major no-swizzle bf16 tiles, umma.cuh)
// W hi, then Q, then W lo: [W hi; Q] is one MN-major B operand of N = 128
// tokens (X and Y1 of the chain in one MMA group)
constexpr uint32_t kUW = 0;       // W hi            [64 i][128 c]   16 KB, MN-major (8 tokens per 16 B)
constexpr uint32_t kUQ = 16384;   // Q               [64 i][128 c]   16 KB, MN-major
constexpr uint32_t kUWl = 32768;  // W lo            [64 i][128 c]   16 KB, MN-major
constexpr uint32_t kUMq = 49152;  // Mq hi, lo       [64 i][64 j]     8 KB each
constexpr uint32_t kUKh = 65536;  // Khat hi, lo     [64 j][128 c]   16 KB each, MN-major B of S^T += U^T Khat
constexpr uint32_t kUG = 98304;   // gamma_i         fp32 [64]
constexpr uint32_t kUU = 98560;   // Ut = T V        fp32 [64 i][128 d]
constexpr uint32_t kUnit = kUU + kC * kDV * 4;
constexpr uint32_t kWBytes = kUMq - kUW;  // W and Q: one bulk copy (phase 1 operands)
constexpr uint32_t kMBytes = kUG - kUMq;  // Mq and Khat: one bulk copy (phase 2 operands)
constexpr uint32_t kGBytes = kUU - kUG;   // gamma
static_assert(kUnit % 16 == 0 && kWBytes % 16 == 0 && kMBytes % 16 == 0, "bulk copies need 16-byte multiples");

__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, int lane_base, uint32_t col) {
  return base + (static_cast<uint32_t>(lane_base) << 16) + col;
}

// ===========================================================================
// Kernel 1: the state-independent part of every chunk.
//
// Operand tiles (umma.cuh) are read either K-major or MN-major: the K and V
// tiles as loaded, [64 j][128 c] with 8 consecutive c per 16-byte row, are
// the K-major B operand of K K^T and also the MN-major A operands of
// W^T = K^T (T diag(gamma))^T and Ut^T = V^T T^T (descriptor: LBO = 2048, the
// stride between 8-token groups; SBO = 128, the stride between 8-column
// groups).  Two CTAs share an SM.
// ===========================================================================
struct PrepArgs {
  const uint16_t *q, *k, *v;
  const float *alpha, *beta;
  unsigned char *ws;
  int T, H, nchunks;
  long units;  // B * H * nchunks
  int32_t *err;
};

constexpr int kPrepCtasPerSm = 2;
constexpr int kLd = kC + 4;  // fp32 row stride of the solve (rows 16-byte aligned, 4 banks apart)
constexpr uint32_t kSolve = kC * kLd * 4;
// shared memory (bytes)
constexpr uint32_t kPK = 0;                     // K rows [64 j][128 c]                    16 KB
constexpr uint32_t kPQ = kPK + 16384;           // Q rows [64 i][128 c] (rows 64..127 of [K;Q]); then L = I + A
constexpr uint32_t kPV = kPQ + kSolve;          // V rows [64 j][128 d]                    16 KB
constexpr uint32_t kPT = kPV + 16384;           // T hi, lo [64 i][64 j]; block products during the solve
constexpr uint32_t kPTG = kPT + 16384;          // T diag(gamma) hi, lo                    16 KB
constexpr uint32_t kPTf = kPTG + 16384;         // L^-1, fp32 [64][kLd]
constexpr uint32_t kPGate = kPTf + kSolve;      // alpha, beta, lambda, gamma, tail [64] each
constexpr uint32_t kPBar = kPGate + 5 * kC * 4;
constexpr uint32_t kPrepSmem = kPBar + 64;
constexpr uint32_t kPColGP = 0, kPColW = 64, kPColU = 128, kPrepTmemCols = 256;
static_assert(2 * (kPrepSmem + 1024) <= 228 * 1024, "two preparation CTAs per SM");

// L^-1 for L = I + A, A strictly lower triangular (fp32, row stride kLd): the
// 16x16 diagonal blocks by substitution, then the blocks below the diagonal
// one block distance at a time, X_IJ = -L_II^-1 sum_{K=J}^{I-1} L_IK X_KJ,
// each thread computing a 1 x 4 strip with 16-byte loads.  Reads only the
// strictly lower part of sA; writes the lower triangle (diagonal included) of
// sTf; sZ holds 768 floats of block products.  kNamed = 0: called by every
// thread of the CTA (at least 192), synchronising the CTA; else by threads
// 0 .. kNamed-1 only (kNamed >= 192), synchronising them on named barrier 1.
template <int kNamed = 0>
__device__ __forceinline__ void solve_sync() {
  if (kNamed == 0)
    __syncthreads();
  else
    asm volatile("bar.sync 1, %0;\n" ::"n"(kNamed) : "memory");
}
template <int kNamed = 0>
__device__ __forceinline__ void solve_unit_lower(const float *sA, float *sTf, float *sZ, int tid) {
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
  solve_sync<kNamed>();
  // ... then the blocks below the diagonal, one block distance at a time:
  // X_IJ = -L_II^-1 sum_{K=J}^{I-1} L_IK X_KJ.  A thread computes a 1 x 4
  // strip (pair p, row r, columns c4..c4+3) with 16-byte loads.
#pragma unroll
  for (int dist = 1; dist < 4; ++dist) {
    const bool mine = tid < (4 - dist) * 64;
    const int p = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
    const int J = p, I = p + dist;
    if (mine) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int K = 0; K < dist; ++K) {
        const float *arow = sA + (I * 16 + r) * kLd + (J + K) * 16;
        const float *xcol = sTf + (J + K) * 16 * kLd + J * 16 + c4;
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4) {
          const float4 av = *reinterpret_cast<const float4 *>(arow + k4);
          const float aa[4] = {av.x, av.y, av.z, av.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 xv = *reinterpret_cast<const float4 *>(xcol + (k4 + e) * kLd);
            acc[0] = fmaf(aa[e], xv.x, acc[0]);
            acc[1] = fmaf(aa[e], xv.y, acc[1]);
            acc[2] = fmaf(aa[e], xv.z, acc[2]);
            acc[3] = fmaf(aa[e], xv.w, acc[3]);
          }
        }
      }
      *reinterpret_cast<float4 *>(sZ + p * 256 + r * 16 + c4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
    solve_sync<kNamed>();
    if (mine) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      const float *xrow = sTf + (I * 16 + r) * kLd + I * 16;
      const float *zcol = sZ + p * 256 + c4;
#pragma unroll
      for (int k4 = 0; k4 < 16; k4 += 4) {
        const float4 xv = *reinterpret_cast<const float4 *>(xrow + k4);
        const float xx[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float4 zv = *reinterpret_cast<const float4 *>(zcol + (k4 + e) * 16);
          acc[0] = fmaf(xx[e], zv.x, acc[0]);
          acc[1] = fmaf(xx[e], zv.y, acc[1]);
          acc[2] = fmaf(xx[e], zv.z, acc[2]);
          acc[3] = fmaf(xx[e], zv.w, acc[3]);
        }
      }
      *reinterpret_cast<float4 *>(sTf + (I * 16 + r) * kLd + J * 16 + c4) =
          make_float4(-acc[0], -acc[1], -acc[2], -acc[3]);
    }
    solve_sync<kNamed>();
  }
}

__global__ void __launch_bounds__(kThreads, kPrepCtasPerSm) gdn_prep_kernel(const PrepArgs a) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int row = tid & 127;
  const int half = tid >> 7;
  const int lane_base = 32 * (warp & 3);
  const int T = a.T, H = a.H;

  unsigned char *sK = sm + kPK, *sQ = sm + kPQ, *sV = sm + kPV;
  unsigned char *sTh = sm + kPT, *sTl = sm + kPT + 8192, *sTGh = sm + kPTG, *sTGl = sm + kPTG + 8192;
  float *sA = reinterpret_cast<float *>(sm + kPQ);
  float *sTf = reinterpret_cast<float *>(sm + kPTf);
  float *sZ = reinterpret_cast<float *>(sm + kPT);
  float *al = reinterpret_cast<float *>(sm + kPGate);
  float *be = al + kC, *lam = al + 2 * kC, *gam = al + 3 * kC, *tail = al + 4 * kC;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kPBar);
  uint32_t *holder = reinterpret_cast<uint32_t *>(sm + kPBar + 32);
  const uint32_t mbGP = smem_addr(bars + 0), mbW = smem_addr(bars + 1), mbEnd = smem_addr(bars + 2);

  if (tid == 0) {
    mbar_init(mbGP, 1);
    mbar_init(mbW, 1);
    mbar_init(mbEnd, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(holder), kPrepTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  // descriptors at k-step 0 (MN-major A: k-step advances 4096 bytes = 256 units)
  const uint64_t dKmn = smem_desc(smem_addr(sK), 2048, 128), dVmn = smem_desc(smem_addr(sV), 2048, 128);
  const uint64_t dTh = smem_desc(smem_addr(sTh), 128, kC * 16), dTl = smem_desc(smem_addr(sTl), 128, kC * 16);
  const uint64_t dTGh = smem_desc(smem_addr(sTGh), 128, kC * 16), dTGl = smem_desc(smem_addr(sTGl), 128, kC * 16);
  const uint32_t idMN = idesc_bf16_f32(128, kC) | (1u << 15);  // A MN-major

  bool failed = false;
  // every thread waits, then the CTA agrees: either all continue or all stop
  auto wait_ok = [&](uint32_t mb, uint32_t parity) -> bool {
    const bool ok = mbar_wait(mb, parity, kWaitLimit);
    tc_fence_before();
    const bool all = __syncthreads_and(ok) != 0;
    tc_fence_after();
    return all;
  };

  int it = 0;
  for (long u = blockIdx.x; u < a.units; u += gridDim.x, ++it) {
    const uint32_t par = static_cast<uint32_t>(it & 1);
    unsigned char *ws = a.ws + u * kUnit;
    const long bh = u / a.nchunks;
    const int t0 = static_cast<int>(u - bh * a.nchunks) * kC;
    const long tok0 = (bh / H) * T * H + bh % H;

    // ---- inputs: K, Q, V rows (8 columns per 16-byte piece), alpha, beta
    // (padding tokens: k = q = v = 0, alpha = 1, beta = 0)
    for (int id = tid; id < 3 * kC * 16; id += kThreads) {
      const int m = id >> 10, r = (id >> 4) & 63, k8 = id & 15;
      const int t = t0 + r;
      unsigned char *dst = sm + (m == 0 ? kPK : m == 1 ? kPQ : kPV) + kmajor_off(r, k8 * 8, kDK);
      if (t < T)
        cp_async<16>(dst, (m == 0 ? a.k : m == 1 ? a.q : a.v) + (tok0 + static_cast<long>(t) * H) * kDK + k8 * 8);
      else
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    if (tid < 2 * kC) {  // the thread that loads alpha_i / beta_i is the one that first reads it
      const int t = t0 + (tid & 63);
      if (t < T)
        cp_async<4>(al + tid, (tid < kC ? a.alpha : a.beta) + tok0 + static_cast<long>(t) * H);
      else
        al[tid] = tid < kC ? 1.f : 0.f;
    }
    cp_async_commit();
    cp_async_wait<0>();
    // lambda = inclusive prefix sum of log2 alpha (two warps of 32 tokens; log2
    // units, so every decay factor below is one ex2)
    if (warp < 2) {
      float x = lg2_approx(al[tid]);
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(kFull, x, o);
        if ((tid & 31) >= o) x += y;
      }
      lam[tid] = x;
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {  // G = [K;Q] K^T: rows 0..63 K K^T, 64..127 Q K^T
      const uint64_t dKQ = smem_desc(smem_addr(sK), 128, kDK * 16);
      const uint32_t idG = idesc_bf16_f32(128, kC);
#pragma unroll
      for (int ks = 0; ks < kDK / 16; ++ks) mma_bf16(tmem + kPColGP, dKQ + 16u * ks, dKQ + 16u * ks, idG, ks > 0);
      mma_commit(mbGP);
    }
    if (warp == 1) lam[tid] += lam[31];
    __syncthreads();
    if (tid < kC) {
      gam[tid] = ex2_approx(lam[tid]);
      tail[tid] = ex2_approx(lam[kC - 1] - lam[tid]);
    }
    __syncthreads();
    // Q tile to the workspace MN-major (8 tokens of one key per 16 bytes,
    // the layout of W); Khat hi/lo: the K tile with row j scaled by
    // e^(lambda_C - lambda_j), the MN-major B operand of the chain's state update
    // (each warp transposes four 8x8 core matrices per ldmatrix: token group
    // ig, key groups 4m..4m+3; lane t then holds tokens 2(t%4), 2(t%4)+1 of
    // key 8(4m+j) + t/4 and stores them as 4 bytes of that key's 16-byte piece)
    for (int o = warp; o < 32; o += kThreads / 32) {
      const int ig = o >> 2, m = o & 3, lane = tid & 31;
      uint32_t r[4];
      ldsm_x4_trans(smem_addr(sQ) + ig * 2048 + (4 * m + (lane >> 3)) * 128 + (lane & 7) * 16, r);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = 8 * (4 * m + j) + (lane >> 2);
        *reinterpret_cast<uint32_t *>(ws + kUQ + ig * 2048 + (c >> 3) * 128 + (c & 7) * 16 + (lane & 3) * 4) = r[j];
      }
    }
    for (int o = tid; o < 1024; o += kThreads) {
      const uint4 kv = reinterpret_cast<const uint4 *>(sK)[o];
      const int j = ((o >> 7) << 3) | (o & 7);  // row of the 16-byte piece o (kmajor_off with K = 128)
      const float tj = tail[j];
      const uint32_t kw[4] = {kv.x, kv.y, kv.z, kv.w};
      float x[8];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[2 * e] = tj * bf16_to_f32(static_cast<uint16_t>(kw[e] & 0xffff));
        x[2 * e + 1] = tj * bf16_to_f32(static_cast<uint16_t>(kw[e] >> 16));
      }
      store_split8(ws + kUKh, ws + kUKh + 16384, o * 16, x);
    }

    // ---- A (decayed, gated K K^T) and Mq (decayed Q K^T) from G
    if (!wait_ok(mbGP, par)) { failed = true; break; }
    {
      const int i = row & 63;
      const float li = lam[i];
      const float bi = be[i];
      for (int j0 = half * 32; j0 < half * 32 + 32; j0 += 16) {
        // a block of 16 columns above every row of the warp is skipped (warp-uniform)
        const bool any = __any_sync(kFull, j0 <= i);
        float x[16];
        if (any) {
          tmem_ld16(tmem_addr(tmem, lane_base, kPColGP + j0), x);
          tmem_ld_wait();
        }
        if (row < 64) {  // strictly lower part of L = I + A (the solve reads no other entry)
          if (any) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const int j = j0 + e;
              if (j < i) sA[i * kLd + j] = bi * ex2_approx(li - lam[j]) * x[e];
            }
          }
        } else {  // Mq, lower part including the diagonal, to the workspace
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int j = j0 + e;
            x[e] = (any && j <= i) ? ex2_approx(li - lam[j]) * x[e] : 0.f;
          }
          store_split8(ws + kUMq, ws + kUMq + 8192, kmajor_off(i, j0, kC), x);
          store_split8(ws + kUMq, ws + kUMq + 8192, kmajor_off(i, j0 + 8, kC), x + 8);
        }
      }
    }
    __syncthreads();

    // ---- L^-1 (unit lower triangular inverse of I + A)
    solve_unit_lower(sA, sTf, sZ, tid);
    // T = L^-1 diag(beta) and T diag(gamma), lower triangles, as B-operand tiles
    // (8 consecutive threads take 8 consecutive rows: conflict-free stores)
    {
      const int i = ((tid >> 5) << 3) | (tid & 7), j0 = ((tid >> 3) & 3) * 16;
      float x[16], xg[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const int j = j0 + e;
        x[e] = j <= i ? sTf[i * kLd + j] * be[j] : 0.f;
        xg[e] = x[e] * gam[j];
      }
      store_split8(sTh, sTl, kmajor_off(i, j0, kC), x);
      store_split8(sTh, sTl, kmajor_off(i, j0 + 8, kC), x + 8);
      store_split8(sTGh, sTGl, kmajor_off(i, j0, kC), xg);
      store_split8(sTGh, sTGl, kmajor_off(i, j0 + 8, kC), xg + 8);
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- W^T = K^T (T diag(gamma))^T and Ut^T = V^T T^T (A MN-major)
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks) {
        mma_bf16(tmem + kPColW, dKmn + 256u * ks, dTGh + 16u * ks, idMN, ks > 0);
        mma_bf16(tmem + kPColW, dKmn + 256u * ks, dTGl + 16u * ks, idMN, true);
        mma_bf16(tmem + kPColU, dVmn + 256u * ks, dTh + 16u * ks, idMN, ks > 0);
        mma_bf16(tmem + kPColU, dVmn + 256u * ks, dTl + 16u * ks, idMN, true);
      }
      mma_commit(mbW);
    }
    if (tid < kC) reinterpret_cast<float *>(ws + kUG)[tid] = gam[tid];
    if (!wait_ok(mbW, par)) { failed = true; break; }
    // Ut[i][d] to the workspace (thread d: coalesced over d); W (lane c,
    // tokens i) as the MN-major B operand of the chain: 8 consecutive i of
    // column c per 16 bytes, at (i/8)*2048 + (c/8)*128 + (c%8)*16
    {
      float *gU = reinterpret_cast<float *>(ws + kUU);
      for (int i0 = half * 32; i0 < half * 32 + 32; i0 += 16) {
        float x[16];
        tmem_ld16(tmem_addr(tmem, lane_base, kPColU + i0), x);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) gU[(i0 + e) * kDV + row] = x[e];
        tmem_ld16(tmem_addr(tmem, lane_base, kPColW + i0), x);
        tmem_ld_wait();
        const uint32_t off = (i0 >> 3) * 2048 + (row >> 3) * 128 + (row & 7) * 16;
        store_split8(ws + kUW, ws + kUWl, off, x);
        store_split8(ws + kUW, ws + kUWl, off + 2048, x + 8);
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  if (failed) {
    // a tensor-core wait ran out: drain this CTA's MMAs (bounded) and report;
    // the chain kernel then reads invalid tiles but ends normally
    if (tid == 0) mma_commit(mbEnd);
    mbar_wait(mbEnd, 0, kWaitLimit);
    if (tid == 0) report_timeout(a.err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kPrepTmemCols);
}

// ===========================================================================
// Kernel 1 for KDA (a decay per key channel; Linear Attention Architectures
// deck, "GDN and KDA change the granularity of forgetting", Eqs. 18-20).
//
// With lambda_ir = sum_{t<=i} log alpha_tr (per channel r, within the chunk),
// the chunk form keeps the shape of the GDN one, but every decay sits inside
// the channel sums:
//   A_ij  = beta_i sum_r k_ir k_jr e^{lambda_ir - lambda_jr}         (j < i)
//   Mq_ij = sum_r q_ir k_jr e^{lambda_ir - lambda_jr}                (j <= i)
//   Qt_i = q_i (.) e^{lambda_i},  Kt_i = k_i (.) e^{lambda_i},
//   Khat_j = k_j (.) e^{lambda_C - lambda_j},  gamma_C = e^{lambda_C}
//   T = (I + A)^-1 diag(beta),  W = T Kt,  Ut = T V
// and the chain runs  U = Ut - W S0,  Y = Qt S0 + Mq U,
// S_C = diag(gamma_C) S0 + Khat^T U.
// A and Mq cannot be one K K^T product: each pair needs its own per-channel
// decay.  Every pair j < i of the chunk is split at the highest bit in which
// i and j differ (level l = 0..5, half size h = 32 >> l): i lies in the right
// half and j in the left half of a segment of 2h tokens whose left half ends
// at token b, so the decay is e^{lambda_i - lambda_b} e^{lambda_b - lambda_j},
// two factors that are each a decay ratio of at most 1 (no factor is ever an
// inverse decay).  Levels 0-3 become two tcgen05 products of block-referenced
// operands (levels 0+1, then 2+3):
//   rows  [k_i; q_i] (.) e^{lambda_i - lambda_b}  (right-half tokens)
//   cols  k_j (.) e^{lambda_b - lambda_j}         (left-half tokens)
// of which only the pairs in the same segment are kept.  Pairs inside a block
// of 4 tokens (levels 4, 5) and the diagonal of Mq are summed on the CUDA
// cores with running products of alpha.  One CTA of 16 warps per SM,
// persistent over units; independent phases run on separate warp groups at
// once, and the next unit's inputs load as this unit's buffers free up.
// ===========================================================================
// ---- one KDA chunk's tiles in the workspace (bytes)
constexpr uint32_t kVW = 0;        // W hi            [64 i][128 c]   MN-major, as kUW
constexpr uint32_t kVQ = 16384;    // Qt hi           [64 i][128 c]   MN-major
constexpr uint32_t kVWl = 32768;   // W lo
constexpr uint32_t kVQl = 49152;   // Qt lo
constexpr uint32_t kVMq = 65536;   // Mq hi, lo       [64 i][64 j]
constexpr uint32_t kVKh = 81920;   // Khat hi, lo     [64 j][128 c]
constexpr uint32_t kVG = 114688;   // gamma_C         fp32 [128] (per key channel)
constexpr uint32_t kVU = 115200;   // Ut = T V        fp32 [64 i][128 d]
constexpr uint32_t kVUnit = kVU + kC * kDV * 4;
static_assert(kVUnit % 16 == 0 && kVMq % 16 == 0 && (kVG - kVMq) % 16 == 0 && (kVU - kVG) % 16 == 0,
              "bulk copies need 16-byte multiples");

// the three instances of the per-channel-decay preparation
constexpr int kModeKda = 0;   // KDA: k, q, v, alpha, beta per token
constexpr int kModeGdn2 = 1;  // GDN2: erase rows e = b (.) k, T = (I + A)^-1, Ut = T (w (.) v)
constexpr int kModeSse = 2;   // SSE delta write: the visits of one partition (keys kk = softmax of the
                              // key logits, beta = the gate, reads scaled by the gate)
// the SSE delta unit: the KDA unit with each visit's staging row after gamma_C
constexpr uint32_t kSRows = kVG + 512;  // int32 [64], -1 for padding visits
constexpr uint32_t kSU = kVU + 256;     // Ut
constexpr uint32_t kSUnit = kVUnit + 256;

struct KdaPrepArgs {
  const uint16_t *q, *k, *v;
  const float *alpha, *beta;
  const float *b_erase, *w_write;  // GDN2 only: erase gate [B,T,H,dk], write gate [B,T,H,dv]
  // SSE delta only: key logits [B,T,H,c], routing records, group tables
  const float *klog;
  const uint32_t *rec, *grp;
  int N, topk, rw, umax;
  long gwords;
  unsigned char *ws;
  int T, H, nchunks;
  long units;  // B * H * nchunks
  int32_t *err;
};

constexpr int kLdL = kDK + 4;  // fp32 row stride of lambda (8 consecutive rows hit distinct banks)
constexpr int kLdS = kC + 1;   // fp32 row stride of the A / Mq staging (a column is conflict-free)
// shared memory (bytes)
constexpr uint32_t kKK = 0;                       // K tile bf16 [64][128] K-major          16 KB
constexpr uint32_t kKQ = 16384;                   // Q tile                                 16 KB
constexpr uint32_t kKV = 32768;                   // V tile                                 16 KB
constexpr uint32_t kKLam = 49152;                 // lambda fp32 [64][kLdL]
constexpr uint32_t kKAl = kKLam + kC * kLdL * 4;  // alpha fp32 [64][128]; then L = I + A fp32 [64][kLd]
                                                  // (the solve's input) and the Mq staging [64][kLdS]
constexpr uint32_t kKAlBytes = kC * kLd * 4 + kC * kLdS * 4;
constexpr uint32_t kKOp = kKAl + kKAlBytes;       // level operands: rows hi, lo [128][128], cols hi, lo [64][128]
constexpr uint32_t kKOpBytes = 98304;
constexpr uint32_t kKGate = kKOp + kKOpBytes;     // beta [2][64], block-of-4 sums [16][16]; SSE: visit
                                                  // token-heads [2][64], staging rows [2][64], unit
                                                  // info [2][4] (two buffers: this unit, the next)
constexpr uint32_t kKBar = kKGate + (2 * kC + 256 + 4 * kC + 8) * 4;
constexpr uint32_t kKdaSmem = kKBar + 64;
// inside the operand region once the level products are done
constexpr uint32_t kOL = 0;                       // GDN2's Z hi/lo (32 KB) once T is written
constexpr uint32_t kOTf = kOL + kSolve;           // L^-1
constexpr uint32_t kOZ = kOTf + kSolve;           // block products of the solve (768 floats)
constexpr uint32_t kOT = kOZ + 4096;              // T hi, lo [64 i][64 j]
constexpr uint32_t kOKt = kOT + 16384;            // Kt hi, lo [64][128]
static_assert(kKAlBytes >= kC * kDK * 4, "alpha fits the staging region");
static_assert(kOKt + 32768 <= kKOpBytes, "solve and Kt fit the operand region");
static_assert(kOL + 32768 <= kOZ, "GDN2's Z hi/lo fits below the solve's block products");
static_assert(kKdaSmem <= 227 * 1024, "one KDA preparation CTA per SM");
constexpr int kKThreads = 512;  // 16 warps (at most 128 registers a thread)
constexpr uint32_t kKColG1 = 0, kKColG2 = 64, kKColW = 128, kKColU = 192, kKdaTmemCols = 256;

// 8 key channels c0..c0+7 of token t as fp32: the bf16 K tile, plus (SSE
// delta: the keys are fp32 row weights kept as bf16 hi + lo) the lo tile
template <int MODE>
__device__ __forceinline__ void load_k8(const unsigned char *sK, const unsigned char *sKlo, int t, int c0,
                                        float (&x)[8]) {
  const uint4 hr = *reinterpret_cast<const uint4 *>(sK + kmajor_off(t, c0, kDK));
  const uint32_t hw[4] = {hr.x, hr.y, hr.z, hr.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    x[2 * e] = bf16_to_f32(static_cast<uint16_t>(hw[e] & 0xffff));
    x[2 * e + 1] = bf16_to_f32(static_cast<uint16_t>(hw[e] >> 16));
  }
  if (MODE == kModeSse) {
    const uint4 lr = *reinterpret_cast<const uint4 *>(sKlo + kmajor_off(t, c0, kDK));
    const uint32_t lw[4] = {lr.x, lr.y, lr.z, lr.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[2 * e] += bf16_to_f32(static_cast<uint16_t>(lw[e] & 0xffff));
      x[2 * e + 1] += bf16_to_f32(static_cast<uint16_t>(lw[e] >> 16));
    }
  }
}

// Operands of the level pair (la, lb) into the operand region: rows
// [k@la; q@la; k@lb; q@lb] of the right-half tokens (32 each) and cols
// [k@la; k@lb] of the left-half tokens, hi/lo K-major.  A thread takes 8
// channels of one token of one level (a right-half token gives its k row and
// its q row from one set of decay factors); 8 consecutive threads take 8
// consecutive operand rows (one 128-byte core-matrix row group), so the
// stores are conflict-free.
// GDN2: the k rows of A are e_t = b_t (.) k_t (the erase gate times the key),
// read as gb[t * gstride + c] for the chunk's valid tokens t < nvalid.
// lam holds lambda in log2 units, so each factor is one 2^x.
// Item k of a thread (k = 0..3): rows for k < 2, level LA for even k; the
// operand row w and channel group g are the thread's own for every k.
template <int MODE, int LA, int LB>
__device__ __forceinline__ void kda_level_operands(const unsigned char *sK, const unsigned char *sKlo,
                                                   const unsigned char *sQ, const float *lam, unsigned char *op,
                                                   int tid, const float *gb, long gstride, int nvalid) {
  constexpr bool G2 = MODE == kModeGdn2;
  static_assert(kKThreads == 512, "four items per thread");
  const int w = (((tid >> 7) & 3) << 3) | (tid & 7), g = (tid >> 3) & 15;
  // GDN2: the erase gates of this thread's two row items, loaded from global
  // memory before any of the work that needs them
  float4 gbr[2][2];
  if (G2) {
#pragma unroll
    for (int ls = 0; ls < 2; ++ls) {
      const int sh = 5 - (ls ? LB : LA), h = 1 << sh;
      const int t = 2 * h * (w >> sh) + h + (w & (h - 1));
      gbr[ls][0] = gbr[ls][1] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (t < nvalid) {
        gbr[ls][0] = __ldg(reinterpret_cast<const float4 *>(gb + t * gstride + 8 * g));
        gbr[ls][1] = __ldg(reinterpret_cast<const float4 *>(gb + t * gstride + 8 * g + 4));
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const bool is_row = k < 2;
    const int lsel = k & 1;                                            // 0: level LA, 1: level LB
    const int lvl = lsel ? LB : LA;
    const int sh = 5 - lvl, h = 1 << sh, seg = w >> sh;
    const int b = 2 * h * seg + h - 1;                                 // last token of the left half
    const int t = is_row ? b + 1 + (w & (h - 1)) : b - h + 1 + (w & (h - 1));
    const float4 lt0 = *reinterpret_cast<const float4 *>(lam + t * kLdL + 8 * g);
    const float4 lt1 = *reinterpret_cast<const float4 *>(lam + t * kLdL + 8 * g + 4);
    const float4 lb0 = *reinterpret_cast<const float4 *>(lam + b * kLdL + 8 * g);
    const float4 lb1 = *reinterpret_cast<const float4 *>(lam + b * kLdL + 8 * g + 4);
    const float dt[8] = {lt0.x - lb0.x, lt0.y - lb0.y, lt0.z - lb0.z, lt0.w - lb0.w,
                         lt1.x - lb1.x, lt1.y - lb1.y, lt1.z - lb1.z, lt1.w - lb1.w};
    // right-half row: e^{lambda_t - lambda_b} (t > b); left-half col: e^{lambda_b - lambda_t} (t <= b)
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = ex2_approx(is_row ? dt[e] : -dt[e]);
    float x[8];
    load_k8<MODE>(sK, sKlo, t, 8 * g, x);
#pragma unroll
    for (int e = 0; e < 8; ++e) x[e] *= f[e];
    if (G2 && is_row) {
      const float4 b0 = lsel ? gbr[1][0] : gbr[0][0], b1 = lsel ? gbr[1][1] : gbr[0][1];
      const float bv[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= bv[e];
    }
    if (is_row) {
      store_split8(op, op + 32768, kmajor_off(64 * lsel + w, 8 * g, kDK), x);
      const uint4 qr = *reinterpret_cast<const uint4 *>(sQ + kmajor_off(t, 8 * g, kDK));
      const uint32_t qw[4] = {qr.x, qr.y, qr.z, qr.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[2 * e] = bf16_to_f32(static_cast<uint16_t>(qw[e] & 0xffff)) * f[2 * e];
        x[2 * e + 1] = bf16_to_f32(static_cast<uint16_t>(qw[e] >> 16)) * f[2 * e + 1];
      }
      store_split8(op, op + 32768, kmajor_off(64 * lsel + 32 + w, 8 * g, kDK), x);
    } else {
      store_split8(op + 65536, op + 81920, kmajor_off(32 * lsel + w, 8 * g, kDK), x);
    }
  }
}

// The pairs of the level pair (la, lb) kept from the product in tensor memory
// (lanes = operand rows, columns = operand cols) into the A / Mq staging.
// Warp w reads lanes 32*(w%4) (one row kind) and 8 of its level's 32 columns.
// A entries (beta applied; none for GDN2) go straight into L = I + A (row
// stride kLd), of which the solve reads only the strictly lower part.
template <int MODE>
__device__ __forceinline__ void kda_level_extract(int la, int lb, uint32_t tmem_col, float *sL, float *sMst,
                                                  const float *be, int warp, int lane) {
  constexpr bool G2 = MODE == kModeGdn2;
  const int sub = warp & 3, qtr = warp >> 2;
  const int lvl = sub < 2 ? la : lb;
  const int sh = 5 - lvl, h = 1 << sh;
  float x[8];
  tmem_ld8(tmem_col + (static_cast<uint32_t>(32 * sub) << 16) + 32 * (sub >> 1) + 8 * qtr, x);
  tmem_ld_wait();
  const int u = lane, seg = u >> sh;
  const int ti = 2 * h * seg + h + (u & (h - 1));
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int v = 8 * qtr + e;
    if ((v >> sh) == seg) {
      const int tj = 2 * h * seg + (v & (h - 1));
      if (sub & 1)
        sMst[ti * kLdS + tj] = x[e];
      else
        sL[ti * kLd + tj] = G2 ? x[e] : be[ti] * x[e];
    }
  }
}

__device__ __forceinline__ void kda_issue_level_mma(uint32_t tmem_d, uint32_t op_addr, uint32_t mbar) {
  const uint64_t dLh = smem_desc(op_addr, 128, kDK * 16), dLl = smem_desc(op_addr + 32768, 128, kDK * 16);
  const uint64_t dRh = smem_desc(op_addr + 65536, 128, kDK * 16), dRl = smem_desc(op_addr + 81920, 128, kDK * 16);
  const uint32_t id = idesc_bf16_f32(128, 64);
#pragma unroll
  for (int ks = 0; ks < kDK / 16; ++ks) {
    mma_bf16(tmem_d, dLh + 16u * ks, dRh + 16u * ks, id, ks > 0);
    mma_bf16(tmem_d, dLh + 16u * ks, dRl + 16u * ks, id, true);
    mma_bf16(tmem_d, dLl + 16u * ks, dRh + 16u * ks, id, true);
  }
  mma_commit(mbar);
}

template <int MODE>
__global__ void __launch_bounds__(kKThreads, 1) kda_prep_kernel(const KdaPrepArgs a) {
  constexpr bool G2 = MODE == kModeGdn2, SSE = MODE == kModeSse;
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int row = tid & 127;
  const int lane_base = 32 * (warp & 3);
  const int T = a.T, H = a.H;

  // SSE: the V tile's slot holds the keys' lo tile, and V arrives late in the
  // operand region (free once the level products are done)
  unsigned char *sK = sm + kKK, *sQ = sm + kKQ, *sKlo = sm + kKV;
  unsigned char *sV = SSE ? sm + kKOp : sm + kKV;
  float *lam = reinterpret_cast<float *>(sm + kKLam);
  float *al = reinterpret_cast<float *>(sm + kKAl);
  float *sL = reinterpret_cast<float *>(sm + kKAl), *sMst = sL + kC * kLd;
  unsigned char *op = sm + kKOp;
  float *sTf = reinterpret_cast<float *>(op + kOTf);
  float *sZ = reinterpret_cast<float *>(op + kOZ);
  unsigned char *sTh = op + kOT, *sTl = op + kOT + 8192, *sKth = op + kOKt, *sKtl = op + kOKt + 16384;
  // per unit, two buffers (this unit's and the next one's, whose inputs load
  // while this one finishes): beta (SSE: the visits' gates) and, SSE only, the
  // token-head (-1: padding) and staging row of each visit and the unit's
  // partition, first position, visit count and list offset
  float *be_all = reinterpret_cast<float *>(sm + kKGate);
  float *w4 = be_all + 2 * kC;
  int *rtok_all = reinterpret_cast<int *>(w4 + 256);
  int *rrow_all = rtok_all + 2 * kC;
  int *info_all = rrow_all + 2 * kC;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kKBar);
  uint32_t *holder = reinterpret_cast<uint32_t *>(sm + kKBar + 32);
  const uint32_t mbG = smem_addr(bars + 0), mbW = smem_addr(bars + 1), mbEnd = smem_addr(bars + 2);
  const uint32_t mbU = smem_addr(bars + 3);  // Ut^T = V^T T^T done (V free), KDA and SSE

  if (tid == 0) {
    mbar_init(mbG, 1);
    mbar_init(mbW, 1);
    mbar_init(mbEnd, 1);
    mbar_init(mbU, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(holder), kKdaTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;
  const uint32_t op_addr = smem_addr(op);
  // W^T = Kt^T T^T and Ut^T = V^T T^T: A operands MN-major (k-step = 16 tokens = 4096 bytes)
  const uint64_t dKtmn_h = smem_desc(smem_addr(sKth), 2048, 128), dKtmn_l = smem_desc(smem_addr(sKtl), 2048, 128);
  const uint64_t dVmn = smem_desc(smem_addr(sV), 2048, 128);
  const uint64_t dZmn_h = smem_desc(smem_addr(op + kOL), 2048, 128), dZmn_l = smem_desc(smem_addr(op + kOL + 16384), 2048, 128);
  const uint64_t dTh = smem_desc(smem_addr(sTh), 128, kC * 16), dTl = smem_desc(smem_addr(sTl), 128, kC * 16);
  const uint32_t idMN = idesc_bf16_f32(128, kC) | (1u << 15);

  bool failed = false;
  auto wait_ok = [&](uint32_t mb, uint32_t parity) -> bool {
    const bool ok = mbar_wait(mb, parity, kWaitLimit);
    tc_fence_before();
    const bool all = __syncthreads_and(ok) != 0;
    tc_fence_after();
    return all;
  };

  // SSE: units past the (batch, head)'s own count are skipped (uniform over the CTA)
  auto unit_valid = [&](long u) -> bool {
    if (!SSE) return true;
    const long bh = u / a.umax;
    return static_cast<int>(u - bh * a.umax) < static_cast<int>(a.grp[bh * a.gwords + ssegrp::kGFirst + a.N]);
  };
  auto next_unit = [&](long u) -> long {
    for (u += gridDim.x; u < a.units && !unit_valid(u); u += gridDim.x) {
    }
    return u;
  };
  // SSE: the visits of unit u (a chunk of 64 visits of one partition of its
  // (batch, head), sse_group.cuh) into buffer b: token-heads, staging rows,
  // gates (the write strength of the delta rule).  Synchronises the CTA.
  auto sse_setup = [&](long u, int b) {
    const long bh = u / a.umax;
    const int uu = static_cast<int>(u - bh * a.umax);
    const uint32_t *g = a.grp + bh * a.gwords;
    const int N = a.N;
    int *info = info_all + 4 * b;
    if (warp == 0) {
      const int nS = (T + kC - 1) / kC;
      int p = N, pos0 = uu * kC, cnt = T, off = 0;
      if (uu >= nS) {  // routed: the last partition whose first unit is <= uu
        const bool c0 = lane < N && static_cast<int>(g[ssegrp::kGFirst + lane]) <= uu;
        const bool c1 = lane + 32 < N && static_cast<int>(g[ssegrp::kGFirst + lane + 32]) <= uu;
        p = __popc(__ballot_sync(kFull, c0)) + __popc(__ballot_sync(kFull, c1)) - 1;
        pos0 = (uu - static_cast<int>(g[ssegrp::kGFirst + p])) * kC;
        cnt = static_cast<int>(g[ssegrp::kGCnt + p]);
        off = static_cast<int>(g[ssegrp::kGOff + p]);
      }
      if (lane == 0) {
        info[0] = p;
        info[1] = pos0;
        info[2] = cnt;
        info[3] = off;
      }
    }
    __syncthreads();
    if (tid < kC) {
      const int p = info[0], pos = info[1] + tid, topk = a.topk;
      int tl = -1, srow = -1;
      float gate = 0.f;
      if (pos < info[2]) {
        int t = pos, r = topk;  // the shared partition: every token, slot topk, gate 1
        if (p < N) {
          const uint32_t e = g[ssegrp::kGHdr + info[3] + pos];
          t = static_cast<int>(e >> 4);
          r = static_cast<int>(e & 15u);
        }
        tl = static_cast<int>((bh / H * T + t) * H + bh % H);
        gate = r < topk ? __uint_as_float(a.rec[static_cast<long>(tl) * a.rw + topk + r]) : 1.f;
        srow = tl * (topk + 1) + r;
      }
      rtok_all[b * kC + tid] = tl;
      rrow_all[b * kC + tid] = srow;
      be_all[b * kC + tid] = gate;
    }
    __syncthreads();
  };
  // ---- inputs of unit u into buffer b, in three groups issued as their
  // destinations free up (padding: k = q = v = 0, alpha = 1, beta = 0):
  // Q (SSE: the visits' q rows) ...
  auto load_q = [&](long u, int b) {
    const int *rt = rtok_all + b * kC;
    const long bh = SSE ? 0 : u / a.nchunks;
    const int t0 = SSE ? 0 : static_cast<int>(u - bh * a.nchunks) * kC;
    const long tok0 = (bh / H) * T * H + bh % H;
    for (int id = tid; id < kC * 16; id += kKThreads) {
      const int r = id >> 4, k8 = id & 15;
      unsigned char *dst = sQ + kmajor_off(r, k8 * 8, kDK);
      const bool valid = SSE ? rt[r] >= 0 : t0 + r < T;
      const long src = SSE ? static_cast<long>(rt[r]) : tok0 + static_cast<long>(t0 + r) * H;
      if (valid)
        cp_async<16>(dst, a.q + src * kDK + k8 * 8);
      else
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  };
  // ... alpha, beta and K (SSE: the key logits, into the lambda buffer) ...
  auto load_kal = [&](long u, int b) {
    const int *rt = rtok_all + b * kC;
    const long bh = SSE ? 0 : u / a.nchunks;
    const int t0 = SSE ? 0 : static_cast<int>(u - bh * a.nchunks) * kC;
    const long tok0 = (bh / H) * T * H + bh % H;
    if (SSE) {
      for (int id = tid; id < kC * (kDK / 4); id += kKThreads) {
        const int r = id >> 5, c4 = id & 31;
        if (rt[r] >= 0)
          cp_async<16>(lam + r * kLdL + 4 * c4, a.klog + static_cast<long>(rt[r]) * kDK + 4 * c4);
        else
          *reinterpret_cast<float4 *>(lam + r * kLdL + 4 * c4) = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    } else {
      for (int id = tid; id < kC * 16; id += kKThreads) {
        const int r = id >> 4, k8 = id & 15;
        unsigned char *dst = sK + kmajor_off(r, k8 * 8, kDK);
        if (t0 + r < T)
          cp_async<16>(dst, a.k + (tok0 + static_cast<long>(t0 + r) * H) * kDK + k8 * 8);
        else
          *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    for (int id = tid; id < kC * (kDK / 4); id += kKThreads) {
      const int r = id >> 5, c4 = id & 31;
      const bool valid = SSE ? rt[r] >= 0 : t0 + r < T;
      const long src = SSE ? static_cast<long>(rt[r]) : tok0 + static_cast<long>(t0 + r) * H;
      if (valid)
        cp_async<16>(al + r * kDK + 4 * c4, a.alpha + src * kDK + 4 * c4);
      else
        *reinterpret_cast<float4 *>(al + r * kDK + 4 * c4) = make_float4(1.f, 1.f, 1.f, 1.f);
    }
    if (tid < kC && !G2 && !SSE) {
      float *bb = be_all + b * kC;
      if (t0 + tid < T)
        cp_async<4>(bb + tid, a.beta + tok0 + static_cast<long>(t0 + tid) * H);
      else
        bb[tid] = 0.f;
    }
    cp_async_commit();
  };
  // ... and V (SSE: loaded inside the unit, below)
  auto load_v = [&](long u) {
    const long bh = u / a.nchunks;
    const int t0 = static_cast<int>(u - bh * a.nchunks) * kC;
    const long tok0 = (bh / H) * T * H + bh % H;
    for (int id = tid; id < kC * 16; id += kKThreads) {
      const int r = id >> 4, k8 = id & 15;
      unsigned char *dst = sV + kmajor_off(r, k8 * 8, kDV);
      if (t0 + r < T)
        cp_async<16>(dst, a.v + (tok0 + static_cast<long>(t0 + r) * H) * kDV + k8 * 8);
      else
        *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
    cp_async_commit();
  };

  int it = 0;  // units done by this CTA (the parity of the W/U barrier)
  int buf = 0;
  long u = next_unit(static_cast<long>(blockIdx.x) - static_cast<long>(gridDim.x));
  if (u < a.units) {
    if (SSE) sse_setup(u, 0);
    load_q(u, 0);
    load_kal(u, 0);
    if (!SSE) load_v(u);
  }
  for (; u < a.units; buf ^= 1) {
    const long un = next_unit(u);
    const bool has_next = un < a.units;
    if (SSE && has_next) sse_setup(un, buf ^ 1);
    float *be = be_all + buf * kC;
    const int *rtok = rtok_all + buf * kC;
    const int *rrow = rrow_all + buf * kC;
    unsigned char *ws = a.ws + u * (SSE ? kSUnit : kVUnit);
    const long bh = SSE ? u / a.umax : u / a.nchunks;
    const int t0 = SSE ? 0 : static_cast<int>(u - bh * a.nchunks) * kC;
    const long tok0 = (bh / H) * T * H + bh % H;
    // GDN2 gates of the chunk's tokens: row t at gb[t * gstride], valid for t < nvalid
    const long gstride = static_cast<long>(H) * kDK;
    const int nvalid = T - t0 < kC ? T - t0 : kC;
    const float *gb = G2 ? a.b_erase + (tok0 + static_cast<long>(t0) * H) * kDK : nullptr;
    const float *gw = G2 ? a.w_write + (tok0 + static_cast<long>(t0) * H) * kDV : nullptr;
    cp_async_wait<0>();
    __syncthreads();
    if (SSE) {
      // kk = softmax of each visit's key logits, in place (a warp takes 4 rows,
      // a lane 4 channels); padding visits get kk = 0
      constexpr int kRowsPerWarp = kC / (kKThreads / 32);
#pragma unroll
      for (int e = 0; e < kRowsPerWarp; ++e) {
        const int i = kRowsPerWarp * warp + e;
        float4 *x = reinterpret_cast<float4 *>(lam + i * kLdL) + lane;
        float4 v = *x;
        if (rtok[i] >= 0) {  // warp-uniform
          const bool bad = !(isfinite(v.x) && isfinite(v.y) && isfinite(v.z) && isfinite(v.w));
          if (__any_sync(kFull, bad) && lane == 0 && a.err) atomicOr(a.err, SDM_DEVERR_NONFINITE);
          float m = fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, o));
          v.x = __expf(v.x - m);
          v.y = __expf(v.y - m);
          v.z = __expf(v.z - m);
          v.w = __expf(v.w - m);
          float z = (v.x + v.y) + (v.z + v.w);
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(kFull, z, o);
          const float zi = 1.0f / z;
          v = make_float4(v.x * zi, v.y * zi, v.z * zi, v.w * zi);
        } else {
          v = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        *x = v;
      }
      __syncthreads();
      // kk as bf16 hi + lo K-major tiles (8 consecutive threads: 8 consecutive rows)
      for (int id = tid; id < kC * 16; id += kKThreads) {
        const int t = ((id >> 7) << 3) | (id & 7), g = (id >> 3) & 15;
        const float4 k0 = *reinterpret_cast<const float4 *>(lam + t * kLdL + 8 * g);
        const float4 k1 = *reinterpret_cast<const float4 *>(lam + t * kLdL + 8 * g + 4);
        const float x[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
        store_split8(sK, sKlo, kmajor_off(t, 8 * g, kDK), x);
      }
      __syncthreads();
    }

    // ---- two groups of 8 warps at once:
    // warps 0-7: pairs inside each block of 4 tokens (and the diagonal of Mq)
    // with running products of alpha.  A thread sums 8 channels of one block
    // (two halves of 4), then the 16 threads of the block reduce-scatter their
    // 16 partial sums (outputs 0-5: A at (1,0),(2,0),(2,1),(3,0),(3,1),(3,2);
    // 6-15: Mq at (0,0),(1,0),(1,1),(2,0),(2,1),(2,2),(3,0),(3,1),(3,2),(3,3)).
    // The lanes of a warp alternate between its two blocks, so a quarter-warp's
    // 16-byte row loads fall on two bank groups, not one.
    // warps 8-15: lambda, the running sum of log alpha over the chunk (kept in
    // log2 units: every decay factor below is a 2^x), two threads per channel
    // (tokens 0-31 and 32-63); the second half then adds the first's total.
    if (tid < 256) {
      const int blk = 2 * warp + (lane & 1), cg = lane >> 1;
      uint4 kraw[4], klraw[4], qraw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = 4 * blk + i;
        kraw[i] = *reinterpret_cast<const uint4 *>(sK + kmajor_off(t, 8 * cg, kDK));
        if (SSE) klraw[i] = *reinterpret_cast<const uint4 *>(sKlo + kmajor_off(t, 8 * cg, kDK));
        qraw[i] = *reinterpret_cast<const uint4 *>(sQ + kmajor_off(t, 8 * cg, kDK));
      }
      float v[16];
#pragma unroll
      for (int o = 0; o < 16; ++o) v[o] = 0.f;
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {
        // channels 8 cg + 4 hc .. + 3: words 2 hc, 2 hc + 1 of each raw row
        float kf[4][4], qf[4][4], af[4][4], ef[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int t = 4 * blk + i;
          const uint32_t kw[2] = {hc ? kraw[i].z : kraw[i].x, hc ? kraw[i].w : kraw[i].y};
          const uint32_t qw[2] = {hc ? qraw[i].z : qraw[i].x, hc ? qraw[i].w : qraw[i].y};
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            kf[i][2 * e] = bf16_to_f32(static_cast<uint16_t>(kw[e] & 0xffff));
            kf[i][2 * e + 1] = bf16_to_f32(static_cast<uint16_t>(kw[e] >> 16));
            qf[i][2 * e] = bf16_to_f32(static_cast<uint16_t>(qw[e] & 0xffff));
            qf[i][2 * e + 1] = bf16_to_f32(static_cast<uint16_t>(qw[e] >> 16));
          }
          if (SSE) {
            const uint32_t lw[2] = {hc ? klraw[i].z : klraw[i].x, hc ? klraw[i].w : klraw[i].y};
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              kf[i][2 * e] += bf16_to_f32(static_cast<uint16_t>(lw[e] & 0xffff));
              kf[i][2 * e + 1] += bf16_to_f32(static_cast<uint16_t>(lw[e] >> 16));
            }
          }
          const float4 a4 = *reinterpret_cast<const float4 *>(al + t * kDK + 8 * cg + 4 * hc);
          af[i][0] = a4.x; af[i][1] = a4.y; af[i][2] = a4.z; af[i][3] = a4.w;
          // left factors of A: k (beta applied later) or e = b (.) k (GDN2)
          float bv[4] = {1.f, 1.f, 1.f, 1.f};
          if (G2) {
            bv[0] = bv[1] = bv[2] = bv[3] = 0.f;
            if (t < nvalid) {
              const float4 b4 = __ldg(reinterpret_cast<const float4 *>(gb + t * gstride + 8 * cg + 4 * hc));
              bv[0] = b4.x; bv[1] = b4.y; bv[2] = b4.z; bv[3] = b4.w;
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) ef[i][e] = bv[e] * kf[i][e];
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float p10 = af[1][c], p21 = af[2][c], p32 = af[3][c];
          const float p20 = p21 * p10, p31 = p32 * p21, p30 = p32 * p20;
          v[0] = fmaf(ef[1][c] * kf[0][c], p10, v[0]);
          v[1] = fmaf(ef[2][c] * kf[0][c], p20, v[1]);
          v[2] = fmaf(ef[2][c] * kf[1][c], p21, v[2]);
          v[3] = fmaf(ef[3][c] * kf[0][c], p30, v[3]);
          v[4] = fmaf(ef[3][c] * kf[1][c], p31, v[4]);
          v[5] = fmaf(ef[3][c] * kf[2][c], p32, v[5]);
          v[6] = fmaf(qf[0][c], kf[0][c], v[6]);
          v[7] = fmaf(qf[1][c] * kf[0][c], p10, v[7]);
          v[8] = fmaf(qf[1][c], kf[1][c], v[8]);
          v[9] = fmaf(qf[2][c] * kf[0][c], p20, v[9]);
          v[10] = fmaf(qf[2][c] * kf[1][c], p21, v[10]);
          v[11] = fmaf(qf[2][c], kf[2][c], v[11]);
          v[12] = fmaf(qf[3][c] * kf[0][c], p30, v[12]);
          v[13] = fmaf(qf[3][c] * kf[1][c], p31, v[13]);
          v[14] = fmaf(qf[3][c] * kf[2][c], p32, v[14]);
          v[15] = fmaf(qf[3][c], kf[3][c], v[15]);
        }
      }
      // reduce-scatter over the block's 16 threads (lanes of one parity): the
      // thread with channel group l ends with output l
      const int l = cg;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const bool up = l & 8;
        const float send = up ? v[e] : v[e + 8];
        const float keep = up ? v[e + 8] : v[e];
        v[e] = keep + __shfl_xor_sync(kFull, send, 16);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const bool up = l & 4;
        const float send = up ? v[e] : v[e + 4];
        const float keep = up ? v[e + 4] : v[e];
        v[e] = keep + __shfl_xor_sync(kFull, send, 8);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const bool up = l & 2;
        const float send = up ? v[e] : v[e + 2];
        const float keep = up ? v[e + 2] : v[e];
        v[e] = keep + __shfl_xor_sync(kFull, send, 4);
      }
      {
        const bool up = l & 1;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(kFull, send, 2);
      }
      w4[16 * blk + l] = v[0];
    } else {
      const int r = tid & (kDK - 1), hf = (tid >> 7) & 1;
      float la[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) la[e] = al[(32 * hf + e) * kDK + r];
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) {
        acc += lg2_approx(la[e]);
        lam[(32 * hf + e) * kLdL + r] = acc;
      }
    }
    __syncthreads();
    if (tid >= 384) {
      const int r = tid & (kDK - 1);
      const float base = lam[31 * kLdL + r];
#pragma unroll
      for (int e = 0; e < 32; ++e) lam[(32 + e) * kLdL + r] += base;
    }
    __syncthreads();

    // ---- levels 0 and 1 on the tensor cores
    kda_level_operands<MODE, 0, 1>(sK, sKlo, sQ, lam, op, tid, gb, gstride, nvalid);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) kda_issue_level_mma(tmem + kKColG1, op_addr, mbG);
    // meanwhile (warps 1-15; warp 0's issuing thread waits on the tensor core):
    // Qt (MN-major: 8 tokens of one key per 16 bytes), Khat and gamma_C to the
    // workspace (q transposed by ldmatrix, four 8x8 core matrices per warp and
    // step: lane t holds tokens 2(t%4), 2(t%4)+1 of key 8(4m+j) + t/4)
    for (int o = warp - 1; warp > 0 && o < 32; o += kKThreads / 32 - 1) {
      const int ig = o >> 2, m = o & 3;
      uint32_t r[4];
      ldsm_x4_trans(smem_addr(sQ) + ig * 2048 + (4 * m + (lane >> 3)) * 128 + (lane & 7) * 16, r);
      const int t0 = 8 * ig + 2 * (lane & 3);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = 8 * (4 * m + j) + (lane >> 2);
        // (SSE: the read of the visit is scaled by its gate)
        const float g0 = SSE ? be[t0] : 1.f, g1 = SSE ? be[t0 + 1] : 1.f;
        const float x0 = g0 * bf16_to_f32(static_cast<uint16_t>(r[j] & 0xffff)) * ex2_approx(lam[t0 * kLdL + c]);
        const float x1 = g1 * bf16_to_f32(static_cast<uint16_t>(r[j] >> 16)) * ex2_approx(lam[(t0 + 1) * kLdL + c]);
        const __nv_bfloat162 hb = __floats2bfloat162_rn(x0, x1);
        const float2 hf = __bfloat1622float2(hb);
        const __nv_bfloat162 lb = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
        const uint32_t off = ig * 2048 + (c >> 3) * 128 + (c & 7) * 16 + (lane & 3) * 4;
        *reinterpret_cast<__nv_bfloat162 *>(ws + kVQ + off) = hb;
        *reinterpret_cast<__nv_bfloat162 *>(ws + kVQl + off) = lb;
      }
    }
    for (int id = tid - 32; tid >= 32 && id < kC * 16; id += kKThreads - 32) {
      // Khat = k (.) e^{lambda_C - lambda_t}, K-major
      const int t = ((id >> 7) << 3) | (id & 7), g = (id >> 3) & 15;
      const float4 t0v = *reinterpret_cast<const float4 *>(lam + t * kLdL + 8 * g);
      const float4 t1v = *reinterpret_cast<const float4 *>(lam + t * kLdL + 8 * g + 4);
      const float4 e0v = *reinterpret_cast<const float4 *>(lam + (kC - 1) * kLdL + 8 * g);
      const float4 e1v = *reinterpret_cast<const float4 *>(lam + (kC - 1) * kLdL + 8 * g + 4);
      const float d[8] = {e0v.x - t0v.x, e0v.y - t0v.y, e0v.z - t0v.z, e0v.w - t0v.w,
                          e1v.x - t1v.x, e1v.y - t1v.y, e1v.z - t1v.z, e1v.w - t1v.w};
      float x[8];
      load_k8<MODE>(sK, sKlo, t, 8 * g, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) x[e] *= ex2_approx(d[e]);
      store_split8(ws + kVKh, ws + kVKh + 16384, kmajor_off(t, 8 * g, kDK), x);
    }
    if (tid >= 32 && tid < 32 + kDK)
      reinterpret_cast<float *>(ws + kVG)[tid - 32] = ex2_approx(lam[(kC - 1) * kLdL + tid - 32]);
    if (!wait_ok(mbG, 0)) { failed = true; break; }
    kda_level_extract<MODE>(0, 1, tmem + kKColG1, sL, sMst, be, warp, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    // ---- levels 2 and 3
    kda_level_operands<MODE, 2, 3>(sK, sKlo, sQ, lam, op, tid, gb, gstride, nvalid);
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) kda_issue_level_mma(tmem + kKColG2, op_addr, mbG);
    // the Q tile is free: the next unit's q rows
    if (has_next) load_q(un, buf ^ 1);
    if (tid >= 32 && tid < 288) {  // meanwhile: the block-of-4 sums into the staging
      const int blk = (tid - 32) >> 4, o = (tid - 32) & 15;
      // (i, j) of output o inside the block (4 bits each, output 0 lowest):
      // i = 1,2,2,3,3,3,0,1,1,2,2,2,3,3,3,3  j = 0,0,1,0,1,2,0,0,1,0,1,2,0,1,2,3
      const uint64_t oi = 0x3333222110333221ull, oj = 0x3210210100210100ull;
      const int i = 4 * blk + static_cast<int>((oi >> (4 * o)) & 15);
      const int j = 4 * blk + static_cast<int>((oj >> (4 * o)) & 15);
      if (o < 6)
        sL[i * kLd + j] = G2 ? w4[tid - 32] : be[i] * w4[tid - 32];
      else
        sMst[i * kLdS + j] = w4[tid - 32];
    }
    if (!wait_ok(mbG, 1)) { failed = true; break; }
    kda_level_extract<MODE>(2, 3, tmem + kKColG2, sL, sMst, be, warp, lane);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (SSE) {
      // V rows of the visits into the operand region, free now: they land
      // while the solve runs
      for (int id = tid; id < kC * 16; id += kKThreads) {
        const int r = id >> 4, k8 = id & 15;
        unsigned char *dst = sV + kmajor_off(r, k8 * 8, kDV);
        if (rtok[r] >= 0)
          cp_async<16>(dst, a.v + static_cast<long>(rtok[r]) * kDV + k8 * 8);
        else
          *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
      }
      cp_async_commit();
    }

    if (tid < 256) {
      solve_unit_lower<256>(sL, sTf, sZ, tid);
    } else {
      // meanwhile (warps 8-15): Mq (lower, diagonal included) to the workspace
      // (8 consecutive threads take 8 consecutive rows: one contiguous
      // 128-byte piece) ...  (GDN2: the erase gates of the thread's Et items
      // are loaded first, so their latency passes under the Mq store)
      float4 eb[4][2];
      if (G2) {
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          const int id = tid - 256 + s4 * (kKThreads - 256);
          const int t = ((id >> 7) << 3) | (id & 7), g = (id >> 3) & 15;
          eb[s4][0] = eb[s4][1] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (t < nvalid) {
            eb[s4][0] = __ldg(reinterpret_cast<const float4 *>(gb + t * gstride + 8 * g));
            eb[s4][1] = __ldg(reinterpret_cast<const float4 *>(gb + t * gstride + 8 * g + 4));
          }
        }
      }
      for (int id = tid - 256; id < kC * 8; id += kKThreads - 256) {
        const int i = ((id >> 6) << 3) | (id & 7), j0 = ((id >> 3) & 7) * 8;
        float x[8];
        const float gi = SSE ? be[i] : 1.f;  // SSE: the read of visit i is scaled by its gate
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = j0 + e <= i ? gi * sMst[i * kLdS + j0 + e] : 0.f;
        store_split8(ws + kVMq, ws + kVMq + 8192, kmajor_off(i, j0, kC), x);
      }
      // ... and Kt = k (.) e^{lambda} (KDA) or Et = b (.) k (.) e^{lambda}
      // (GDN2), hi/lo operand tiles
#pragma unroll
      for (int s4 = 0; s4 < 4; ++s4) {
        const int id = tid - 256 + s4 * (kKThreads - 256);
        const int t = ((id >> 7) << 3) | (id & 7), g = (id >> 3) & 15;
        const float4 t0v = *reinterpret_cast<const float4 *>(lam + t * kLdL + 8 * g);
        const float4 t1v = *reinterpret_cast<const float4 *>(lam + t * kLdL + 8 * g + 4);
        const float lt[8] = {t0v.x, t0v.y, t0v.z, t0v.w, t1v.x, t1v.y, t1v.z, t1v.w};
        float kx[8];
        load_k8<MODE>(sK, sKlo, t, 8 * g, kx);
        float bv[8] = {1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f, 1.f};
        if (G2) {
          bv[0] = eb[s4][0].x; bv[1] = eb[s4][0].y; bv[2] = eb[s4][0].z; bv[3] = eb[s4][0].w;
          bv[4] = eb[s4][1].x; bv[5] = eb[s4][1].y; bv[6] = eb[s4][1].z; bv[7] = eb[s4][1].w;
        }
        float x[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) x[e] = kx[e] * bv[e] * ex2_approx(lt[e]);
        store_split8(sKth, sKtl, kmajor_off(t, 8 * g, kDK), x);
      }
    }
    __syncthreads();
    // GDN2: the write gates of the thread's two Z items, loaded before T is built
    float4 zw[2][2];
    if (G2) {
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int id = tid + s2 * kKThreads;
        const int t = ((id >> 7) << 3) | (id & 7), g = (id >> 3) & 15;
        zw[s2][0] = zw[s2][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (t < nvalid) {
          zw[s2][0] = __ldg(reinterpret_cast<const float4 *>(gw + t * static_cast<long>(H) * kDV + 8 * g));
          zw[s2][1] = __ldg(reinterpret_cast<const float4 *>(gw + t * static_cast<long>(H) * kDV + 8 * g + 4));
        }
      }
    }
    // T = L^-1 diag(beta) (KDA) or L^-1 (GDN2), lower triangle, hi/lo (8
    // consecutive threads take 8 consecutive rows: conflict-free stores)
    {
      const int i = ((tid >> 6) << 3) | (tid & 7), j0 = ((tid >> 3) & 7) * 8;
      float x[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int j = j0 + e;
        x[e] = j <= i ? (G2 ? sTf[i * kLd + j] : sTf[i * kLd + j] * be[j]) : 0.f;
      }
      store_split8(sTh, sTl, kmajor_off(i, j0, kC), x);
    }
    if (G2) {
      // Z = w (.) v, hi/lo K-major [64 t][128 d] into the solve buffers (free
      // once T is written): the MN-major A operand of Ut^T = Z^T T^T
      __syncthreads();
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int id = tid + s2 * kKThreads;
        const int t = ((id >> 7) << 3) | (id & 7), g = (id >> 3) & 15;
        const uint4 raw = *reinterpret_cast<const uint4 *>(sV + kmajor_off(t, 8 * g, kDV));
        const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
        const float wv[8] = {zw[s2][0].x, zw[s2][0].y, zw[s2][0].z, zw[s2][0].w,
                             zw[s2][1].x, zw[s2][1].y, zw[s2][1].z, zw[s2][1].w};
        float x[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          x[2 * e] = bf16_to_f32(static_cast<uint16_t>(rw[e] & 0xffff)) * wv[2 * e];
          x[2 * e + 1] = bf16_to_f32(static_cast<uint16_t>(rw[e] >> 16)) * wv[2 * e + 1];
        }
        store_split8(op + kOL, op + kOL + 16384, kmajor_off(t, 8 * g, kDV), x);
      }
    }
    if (SSE) cp_async_wait<0>();
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // ---- Ut^T = V^T T^T (V is exact: two passes; KDA and SSE: first, on its
    // own commit, so the V tile frees early) and W^T = Kt^T T^T (three)
    if (tid == 0) {
      if (!G2) {
#pragma unroll
        for (int ks = 0; ks < kC / 16; ++ks) {
          mma_bf16(tmem + kKColU, dVmn + 256u * ks, dTh + 16u * ks, idMN, ks > 0);
          mma_bf16(tmem + kKColU, dVmn + 256u * ks, dTl + 16u * ks, idMN, true);
        }
        mma_commit(mbU);
      }
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks) {
        mma_bf16(tmem + kKColW, dKtmn_h + 256u * ks, dTh + 16u * ks, idMN, ks > 0);
        mma_bf16(tmem + kKColW, dKtmn_h + 256u * ks, dTl + 16u * ks, idMN, true);
        mma_bf16(tmem + kKColW, dKtmn_l + 256u * ks, dTh + 16u * ks, idMN, true);
        if (G2) {
          mma_bf16(tmem + kKColU, dZmn_h + 256u * ks, dTh + 16u * ks, idMN, ks > 0);
          mma_bf16(tmem + kKColU, dZmn_h + 256u * ks, dTl + 16u * ks, idMN, true);
          mma_bf16(tmem + kKColU, dZmn_l + 256u * ks, dTh + 16u * ks, idMN, true);
        }
      }
      mma_commit(mbW);
    }
    // K, alpha, beta and lambda are free: the next unit's, while the products
    // run; V too as soon as no product reads it (GDN2's Ut takes z = w (.) v,
    // built before the products; KDA's reads V and completes first)
    if (has_next) load_kal(un, buf ^ 1);
    if (has_next && G2) load_v(un);
    if (has_next && !SSE && !G2) {
      if (!wait_ok(mbU, static_cast<uint32_t>(it & 1))) { failed = true; break; }
      load_v(un);
    }
    if (!wait_ok(mbW, static_cast<uint32_t>(it & 1))) { failed = true; break; }
    if (SSE && tid < kC) reinterpret_cast<int *>(ws + kSRows)[tid] = rrow[tid];
    {
      float *gU = reinterpret_cast<float *>(ws + (SSE ? kSU : kVU));
      {
        const int i0 = 16 * (tid >> 7);  // a quarter of the tokens per group of 4 warps
        float x[16];
        tmem_ld16(tmem_addr(tmem, lane_base, kKColU + i0), x);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) gU[(i0 + e) * kDV + row] = x[e];
        tmem_ld16(tmem_addr(tmem, lane_base, kKColW + i0), x);
        tmem_ld_wait();
        const uint32_t off = (i0 >> 3) * 2048 + (row >> 3) * 128 + (row & 7) * 16;
        store_split8(ws + kVW, ws + kVWl, off, x);
        store_split8(ws + kVW, ws + kVWl, off + 2048, x + 8);
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    ++it;
    u = un;
  }
  cp_async_wait<0>();  // (a wait that ran out may leave the next unit's loads in flight)
  if (failed) {
    if (tid == 0) mma_commit(mbEnd);
    mbar_wait(mbEnd, 0, kWaitLimit);
    if (tid == 0) report_timeout(a.err);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kKdaTmemCols);
}

// ===========================================================================
// Kernel 2: the chain of chunks of one (batch, head).
//
// Warps 0-15 (workers): warp w owns tensor-memory lanes 32*(w%4) .. +31
// (value rows d) and quarter w/4 of each tile's columns; it keeps its 32
// columns of S^T in registers.  Warp 16 (producer, one lane) issues the bulk
// copies and the MMAs.  Per chunk, the state's own chain first and the output
// behind it (the tensor pipe runs one thread's MMAs in order):
//   phase 1  [X | Y1] = S0^T [W^T | Q^T] as one MMA group of N = 128,
//            issued in two column groups as the workers publish the bf16
//            split of S0 (S_ready[g]); the next chunk's W and Q load as soon
//            as it is done;
//   workers  U^T = Ut^T - X, split, published (U_ready);
//   phase 2  D = U^T Khat; then Y2 = U^T Mq^T;
//   workers  S^T <- gamma_C S^T + D, split for the next phase 1; then
//            y = gamma_i Y1 + Y2 (GDN) or Y1 + Y2 (KDA).
// ===========================================================================
struct ChainArgs {
  float *state;
  const unsigned char *ws;
  float *y;
  int T, H, nchunks;
  // SSE delta only: the group tables, units per (batch, head), routed
  // partitions, (batch, head) count, the visits' staging rows
  const uint32_t *grp;
  long gwords, bhn;
  int umax, N;
  float *stage;
  int drop_signal;  // test hook: the first X-done signal is never sent, so the workers' bounded wait runs out
  int32_t *err;
};

constexpr int kWorkers = 512;
constexpr int kChainThreads = kWorkers + 32;

// tensor-memory columns (fp32)
constexpr uint32_t kColD = 0;     // U^T Khat     [128 d x 128 c]
constexpr uint32_t kColXY = 128;  // [S0^T W^T | S0^T Q^T]  [128 x (64 + 64)], one MMA group of N = 128;
                                  // two buffers by chunk parity (chunk c+1's group may be issued
                                  // while the workers still read chunk c's Y1)
constexpr uint32_t kColY2 = 384;  // U^T Mq^T     [128 x 64]
constexpr uint32_t kChainTmemCols = 512;

// shared memory (bytes) and the unit layout the chain reads, GDN or KDA
constexpr uint32_t kCS = 0;               // S^T hi, lo [128 d][128 c]        2 x 32 KB
constexpr uint32_t kCU = kCS + 65536;     // U^T hi, lo [128 d][64 j]         2 x 16 KB
constexpr uint32_t kCW = kCU + 32768;     // W hi, lo, then Q (GDN) or Qt hi, lo (KDA): one bulk copy
constexpr int kNBar = 12;
// CM: 0 GDN, 1 KDA / GDN2, 2 SSE delta (the KDA layout plus each visit's
// staging row after gamma_C)
template <int CM>
struct ChainLayout {
  static constexpr bool KDA = CM >= 1;
  static constexpr uint32_t unit = CM == 2 ? kSUnit : KDA ? kVUnit : kUnit;
  static constexpr uint32_t w_off = KDA ? kVW : kUW;                 // W, Q / Qt
  static constexpr uint32_t w_bytes = KDA ? kVMq - kVW : kWBytes;
  static constexpr uint32_t m_off = KDA ? kVMq : kUMq;               // Mq, Khat
  static constexpr uint32_t m_bytes = KDA ? kVG - kVMq : kMBytes;
  static constexpr uint32_t g_off = KDA ? kVG : kUG;                 // gamma_C per channel (KDA) / gamma_i (GDN)
  static constexpr uint32_t g_bytes = CM == 2 ? kSU - kVG : KDA ? kVU - kVG : kGBytes;
  static constexpr uint32_t u_off = CM == 2 ? kSU : KDA ? kVU : kUU;  // Ut
  static constexpr uint32_t cm = kCW + w_bytes;                      // Mq hi, lo, Khat hi, lo
  static constexpr uint32_t cg = cm + m_bytes;                       // gammas, two buffers
  static constexpr uint32_t cbar = cg + 2 * g_bytes;
  static constexpr uint32_t smem = cbar + kNBar * 8 + 16;
  static_assert(smem <= 227 * 1024, "chain shared memory");
};

// bounded wait (about 0.13 s) that also gives up as soon as another thread has
constexpr uint32_t kHintedWaitLimit = 1u << 17;
__device__ __forceinline__ bool chain_wait(uint32_t mbar, uint32_t parity, volatile int *abort_flag) {
  return mbar_wait_hinted(mbar, parity, kHintedWaitLimit, abort_flag);
}
// the producer's waits: a busy wait (one thread), so it issues the moment an operand is ready
constexpr uint32_t kSpinWaitLimit = 1u << 24;
__device__ __forceinline__ bool producer_wait(uint32_t mbar, uint32_t parity, volatile int *abort_flag) {
  return mbar_wait_spin(mbar, parity, kSpinWaitLimit, abort_flag);
}

// the chain of one (batch, head) (SSE: one (batch, head, partition)) on the
// CTA `cta` of the launch
template <int CM>
__device__ __forceinline__ void chain_single(const ChainArgs &a, long cta) {
  using L = ChainLayout<CM>;
  constexpr bool KDA = CM >= 1, SSE = CM == 2;
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int T = a.T, H = a.H;
  long bh = cta, u0;
  int n;
  float *gS;
  if (SSE) {
    // one (batch, head, partition), the shared partitions first (the longest
    // chains); its units are consecutive in the (batch, head)'s unit space
    int p;
    if (cta < a.bhn) {
      p = a.N;
    } else {
      bh = (cta - a.bhn) / a.N;
      p = static_cast<int>((cta - a.bhn) % a.N);
    }
    const uint32_t *g = a.grp + bh * a.gwords;
    int first = 0, count = (T + kC - 1) / kC;
    if (p < a.N) {
      first = static_cast<int>(g[ssegrp::kGFirst + p]);
      count = static_cast<int>(g[ssegrp::kGFirst + p + 1]) - first;
    }
    if (count == 0) return;  // a partition nobody visited keeps its state (the whole CTA leaves)
    u0 = bh * a.umax + first;
    n = count;
    gS = a.state + (bh * (a.N + 1) + p) * static_cast<long>(kDK * kDV);
  } else {
    n = a.nchunks;
    u0 = bh * n;
    gS = a.state + bh * kDK * kDV;
  }
  const long tok0 = (bh / H) * T * H + bh % H;  // token t -> tok0 + t*H (GDN / KDA)

  unsigned char *sSh = sm + kCS, *sSl = sm + kCS + 32768;
  unsigned char *sUh = sm + kCU, *sUl = sm + kCU + 16384;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::cbar);
  // barriers: 0 W, 1 M, 2-3 gamma buffers, 4 phase 1 ([X | Y1]) done, 5 unused,
  // 6 Y2 done (the chunk's last MMA), 7 D done, 8-9 S_ready[g], 10 U_ready, 11 drain
  auto bar = [&](int i) { return smem_addr(bars + i); };
  uint32_t *holder = reinterpret_cast<uint32_t *>(sm + L::cbar + kNBar * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::cbar + kNBar * 8 + 4);

  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(bar(i), 1);
    for (int i = 8; i < 11; ++i) mbar_init(bar(i), kWorkers / 32);  // one arrival per worker warp
    mbar_init(bar(11), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(holder), kChainTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;

  if (warp < kWorkers / 32) {
    // ------------------------------------------------------------ workers
    const int row = 32 * (warp & 3) + (tid & 31), qtr = warp >> 2;
    const uint32_t lanes = tmem + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
    // waits agree across the warp (its tensor-memory loads are warp-wide)
    auto wwait = [&](uint32_t mb, uint32_t parity) -> bool {
      return __all_sync(kFull, chain_wait(mb, parity, abort_flag)) != 0;
    };
    float S[32];  // S^T[row][32*qtr + j]
#pragma unroll
    for (int j = 0; j < 32; ++j) S[j] = gS[static_cast<long>(32 * qtr + j) * kDV + row];
    // publish the bf16 split of columns [32*qtr + 16g, +16) of S^T
    // a warp's stores are fenced towards the tensor core by every lane, then
    // ordered within the warp, then released by one arrival
    auto publish_s = [&](int g) {
      store_split8(sSh, sSl, kmajor_off(row, 32 * qtr + 16 * g, kDK), S + 16 * g);
      store_split8(sSh, sSl, kmajor_off(row, 32 * qtr + 16 * g + 8, kDK), S + 16 * g + 8);
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if ((tid & 31) == 0) mbar_arrive(bar(8 + g));
    };
    publish_s(0);
    publish_s(1);
    float ut[16];  // Ut[16*qtr + e][row] of the next chunk
    auto load_ut = [&](int c) {
      const float *src = reinterpret_cast<const float *>(a.ws + (u0 + c) * L::unit + L::u_off) + row;
#pragma unroll
      for (int e = 0; e < 16; ++e) ut[e] = __ldg(src + (16 * qtr + e) * kDV);
    };
    load_ut(0);
    for (int c = 0; c < n; ++c) {
      const uint32_t par = static_cast<uint32_t>(c & 1);
      const bool last = c + 1 == n;
      // U^T = Ut^T - X for this warp's 16 tokens
      if (!wwait(bar(4), par)) break;
      {
        float x[16];
        tmem_ld16(lanes + kColXY + 128 * (c & 1) + 16 * qtr, x);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = ut[e] - x[e];
        store_split8(sUh, sUl, kmajor_off(row, 16 * qtr, kC), x);
        store_split8(sUh, sUl, kmajor_off(row, 16 * qtr + 8, kC), x + 8);
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if ((tid & 31) == 0) mbar_arrive(bar(10));
      }
      if (!last) load_ut(c + 1);
      // this chunk's gammas (loaded long before; checked while D runs)
      if (!wwait(bar(2 + (c & 1)), static_cast<uint32_t>((c >> 1) & 1))) break;
      // S^T <- gamma_C S^T + D (KDA: gamma_C per key channel, i.e. per column
      // of S^T), published group by group for the next phase 1.  D completing
      // also means Y1 (issued before it) no longer reads the published S.
      if (!wwait(bar(7), par)) break;
      const float *gbuf = reinterpret_cast<const float *>(sm + L::cg + (c & 1) * L::g_bytes);
      if (CM != 1) {
#pragma unroll
        for (int g = 0; g < 2; ++g) {
          float x[16];
          tmem_ld16(lanes + kColD + 32 * qtr + 16 * g, x);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e)
            S[16 * g + e] = fmaf(gbuf[KDA ? 32 * qtr + 16 * g + e : kC - 1], S[16 * g + e], x[e]);
          if (!last) publish_s(g);
        }
      } else {
        // KDA / GDN2 (measured faster this way; GDN and the SSE write slower):
        // both column groups of D in flight at once, then fold and publish group by group
        float x0[16], x1[16];
        tmem_ld16(lanes + kColD + 32 * qtr, x0);
        tmem_ld16(lanes + kColD + 32 * qtr + 16, x1);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) S[e] = fmaf(gbuf[32 * qtr + e], S[e], x0[e]);
        if (!last) publish_s(0);
#pragma unroll
        for (int e = 0; e < 16; ++e) S[16 + e] = fmaf(gbuf[32 * qtr + 16 + e], S[16 + e], x1[e]);
        if (!last) publish_s(1);
      }
      if (last) {
#pragma unroll
        for (int j = 0; j < 32; ++j) gS[static_cast<long>(32 * qtr + j) * kDV + row] = S[j];
      }
      // y = gamma_i Y1 + Y2 (GDN) or Y1 + Y2 (KDA: the decay is inside Qt),
      // off the state's critical path
      if (!wwait(bar(6), par)) break;
      {
        const float *gam = gbuf + 16 * qtr;
        const int *srow = reinterpret_cast<const int *>(gbuf + kDK) + 16 * qtr;  // SSE: the visits' staging rows
        const int t0 = c * kC + 16 * qtr;
        float *yp = SSE ? nullptr : a.y + (tok0 + static_cast<long>(t0) * H) * kDV + row;
#pragma unroll
        for (int h8 = 0; h8 < 16; h8 += 8) {
          float y1[8], y2[8];
          tmem_ld8(lanes + kColXY + 128 * (c & 1) + 64 + 16 * qtr + h8, y1);
          tmem_ld8(lanes + kColY2 + 16 * qtr + h8, y2);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            if (SSE) {
              const int r = srow[h8 + e];
              if (r >= 0) a.stage[static_cast<long>(r) * kDV + row] = y1[e] + y2[e];
            } else if (t0 + h8 + e < T) {
              yp[static_cast<long>(h8 + e) * H * kDV] = KDA ? y1[e] + y2[e] : fmaf(gam[h8 + e], y1[e], y2[e]);
            }
          }
        }
      }
    }
  } else if (tid == kWorkers) {
    // ------------------------------------------------------------ producer
    const uint32_t sh = smem_addr(sSh), sl = smem_addr(sSl), uh = smem_addr(sUh), ul = smem_addr(sUl);
    // W region: W hi, Q / Qt hi, W lo, (KDA) Qt lo, all MN-major with 8-token
    // groups 2048 bytes apart, so [W hi; Q hi] and [W lo; Qt lo] are B
    // operands of N = 128 tokens
    const uint32_t wh = smem_addr(sm + kCW), wl = wh + 32768;
    const uint32_t mh = smem_addr(sm + L::cm), ml = mh + 8192, kh = mh + 16384, kl = mh + 32768;
    const uint32_t id64 = idesc_bf16_f32(128, kC), id128 = idesc_bf16_f32(128, kDK);
    // operand descriptors at k-step 0; k-step ks starts 256 bytes further on,
    // i.e. 16 in the descriptor's address field
    const uint64_t dSh = smem_desc(smem_addr(sSh), 128, kDK * 16), dSl = smem_desc(smem_addr(sSl), 128, kDK * 16);
    const uint64_t dWQh = smem_desc(wh, 128, 2048), dWQl = smem_desc(wl, 128, 2048);
    const uint64_t dUh = smem_desc(smem_addr(sUh), 128, kC * 16), dUl = smem_desc(smem_addr(sUl), 128, kC * 16);
    const uint64_t dMh = smem_desc(mh, 128, kC * 16), dMl = smem_desc(ml, 128, kC * 16);
    const uint64_t dKh = smem_desc(kh, 2048, 128), dKl = smem_desc(kl, 2048, 128);
    const uint32_t id64w = id64 | (1u << 16), id128w = id128 | (1u << 16), id128k = id128 | (1u << 16);  // B MN-major
    // k-step ks: A advances 256 bytes (16 in the descriptor); B by bstep
    auto mma = [&](uint32_t d, uint64_t A, uint64_t Bm, int ks, uint32_t idesc, bool acc, uint32_t bstep = 16u) {
      mma_bf16(d, A + 16u * ks, Bm + bstep * ks, idesc, acc);
    };
    int w_issued = 0, w_done = 0, m_issued = 0, m_done = 0, g_issued = 0;
    auto load = [&](int which, int c) {
      const unsigned char *src = a.ws + (u0 + c) * L::unit;
      fence_async_smem();
      if (which == 0) {
        mbar_expect_tx(bar(0), L::w_bytes);
        bulk_g2s(wh, src + L::w_off, L::w_bytes, bar(0));
        ++w_issued;
      } else {
        mbar_expect_tx(bar(1), L::m_bytes);
        bulk_g2s(mh, src + L::m_off, L::m_bytes, bar(1));
        mbar_expect_tx(bar(2 + (c & 1)), L::g_bytes);
        bulk_g2s(smem_addr(sm + L::cg + (c & 1) * L::g_bytes), src + L::g_off, L::g_bytes, bar(2 + (c & 1)));
        ++m_issued;
        ++g_issued;
      }
    };
    // the operands of chunk c into L2 ahead of their copies (pieces of at most 48 KB)
    auto prefetch = [&](int c) {
      const unsigned char *pf = a.ws + (u0 + c) * L::unit;
      prefetch_l2(pf + L::w_off, L::w_bytes / 2);
      prefetch_l2(pf + L::w_off + L::w_bytes / 2, L::w_bytes / 2);
      prefetch_l2(pf + L::m_off, L::m_bytes + L::g_bytes);
      prefetch_l2(pf + L::u_off, L::unit - L::u_off);
    };
    if (n > 1) prefetch(1);
    load(0, 0);
    load(1, 0);
    bool ok = true;
    for (int c = 0; c < n && ok; ++c) {
      const uint32_t par = static_cast<uint32_t>(c & 1);
      if (c + 2 < n) prefetch(c + 2);  // chunk c + 2 into L2 while this one runs
      // phase 1: [X | Y1] = S0^T [W^T | Q^T] as each column group g (k-steps
      // g, g + 2, g + 4, g + 6) of S^T is published: S hi x [W hi; Q], S hi x
      // W lo (GDN, N = 64: Q is exact) or S hi x [W lo; Qt lo] (KDA), S lo x
      // [W hi; Q]
      const uint32_t xy = tmem + kColXY + 128 * (c & 1);
      ok = producer_wait(bar(0), par, abort_flag);
      if (ok) ++w_done;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (ok) ok = producer_wait(bar(8 + g), par, abort_flag);
        if (!ok) break;
#pragma unroll
        for (int ks = g; ks < 8; ks += 2) {
          mma(xy, dSh, dWQh, ks, id128w, ks != 0);
          mma(xy, dSh, dWQl, ks, KDA ? id128w : id64w, true);
          mma(xy, dSl, dWQh, ks, id128w, true);
        }
      }
      if (!ok) break;
      if (!(a.drop_signal && c == 0)) mma_commit(bar(4));
      // the W region is free once the group is done: the next chunk's W and Q
      if (c + 1 < n) {
        ok = producer_wait(bar(4), par, abort_flag);
        if (!ok) break;
        load(0, c + 1);
      }
      // phase 2: D = U^T Khat first (the state update waits for it), then
      // Y2 = U^T Mq^T
      ok = producer_wait(bar(1), par, abort_flag);
      if (ok) ++m_done;
      if (ok) ok = producer_wait(bar(10), par, abort_flag);
      if (!ok) break;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma(tmem + kColD, dUh, dKh, ks, id128k, ks != 0, 256u);
        mma(tmem + kColD, dUh, dKl, ks, id128k, true, 256u);
        mma(tmem + kColD, dUl, dKh, ks, id128k, true, 256u);
      }
      mma_commit(bar(7));
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma(tmem + kColY2, dUh, dMh, ks, id64, ks != 0);
        mma(tmem + kColY2, dUh, dMl, ks, id64, true);
        mma(tmem + kColY2, dUl, dMh, ks, id64, true);
      }
      mma_commit(bar(6));
      if (c + 1 < n) {
        // the next chunk's Mq, Khat and gammas once Y2 (the chunk's last MMA,
        // which reads Mq) is done
        ok = producer_wait(bar(6), par, abort_flag);
        if (ok) load(1, c + 1);
      }
    }
    // every MMA issued has completed before tensor memory is freed (also when
    // a worker's wait ran out after this loop ended) ...
    mma_commit(bar(11));
    mbar_wait(bar(11), 0, kWaitLimit);
    // ... and every bulk copy has landed before the CTA exits: at most the last
    // copy into each buffer can be unobserved (bounded waits; in the normal
    // path all have been seen complete already)
    if (w_done < w_issued) mbar_wait(bar(0), static_cast<uint32_t>((w_issued - 1) & 1), kWaitLimit);
    if (m_done < m_issued) mbar_wait(bar(1), static_cast<uint32_t>((m_issued - 1) & 1), kWaitLimit);
    for (int gb = 0; gb < 2; ++gb) {
      const int loads = (g_issued + 1 - gb) / 2;  // gamma copies issued into buffer gb
      if (loads > 0) mbar_wait(bar(2 + gb), static_cast<uint32_t>((loads - 1) & 1), kWaitLimit);
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) report_timeout(a.err);
  if (warp == 0) tmem_dealloc(tmem, kChainTmemCols);
}

template <int CM>
__global__ void __maxnreg__(96) gdn_chain_kernel(const ChainArgs a) {
  chain_single<CM>(a, blockIdx.x);
}


// ===========================================================================
// Kernel 2, split by value columns: the chain of one (batch, head) on a pair
// of CTAs, CTA h of the pair owning value columns [64h, 64h + 64).  Each
// value column evolves independently, so the two CTAs never communicate.
// The products are turned so that every MMA has M = 128 and N = 64 (the
// CTA's columns):
//   phase 1  [X; Y1] = [W; Q] S0      A = [W; Q] (128 tokens, MN-major from the
//                                      unit), B = S0 (d_k x 64, MN-major);
//   workers  U = Ut - X (token rows, warps of lanes 0-63), split, published;
//   phase 2  D = Khat^T U              A = Khat^T (MN-major from the unit);
//            Y2 = [0; Mq] U            A = Mq below 64 zero rows, so Y2 lands
//                                      in the lanes of Y1;
//   workers  S <- gamma_C S + D (all 16 warps, lane = key channel), split for
//            the next phase 1; y = gamma_i Y1 + Y2 (GDN) or Y1 + Y2 (KDA) on
//            the warps of lanes 64-127.
// Against one CTA per (b, h) this halves the state update per thread and
// gives the output to the warps that have no U to form.
// ===========================================================================
constexpr uint32_t kQS = 0;              // S hi, lo [128 c][64 d] MN-major      2 x 16 KB
constexpr uint32_t kQU = kQS + 32768;    // U hi, lo [64 i][64 d] MN-major       2 x 8 KB
constexpr uint32_t kQW = kQU + 16384;    // W hi | Q (Qt) hi | W lo | Qt lo (KDA) or zeros (GDN)   64 KB
constexpr uint32_t kQM = kQW + 65536;    // zeros | Mq hi | zeros | Mq lo | Khat hi | Khat lo        64 KB
constexpr uint32_t kQG = kQM + 65536;    // gammas, two buffers
constexpr uint32_t kQColXY = 0;          // [X; Y1] [128 x 64], two buffers by chunk parity
constexpr uint32_t kQColD = 128;         // D       [128 c x 64 d]
constexpr uint32_t kQColY2 = 192;        // Y2      [128 x 64] (rows 64-127), two buffers
constexpr uint32_t kQTmemCols = 512;
// CM as the single form's: 0 GDN, 1 KDA / GDN2, 2 SSE delta (the KDA layout
// plus each visit's staging row after gamma_C)
template <int CM>
struct PairLayout {
  static constexpr bool KDA = CM >= 1;
  static constexpr uint32_t unit = CM == 2 ? kSUnit : KDA ? kVUnit : kUnit;
  static constexpr uint32_t w_off = KDA ? kVW : kUW;
  static constexpr uint32_t w_bytes = KDA ? kVMq - kVW : kWBytes;    // 64 KB (KDA) or 48 KB (GDN)
  static constexpr uint32_t m_off = KDA ? kVMq : kUMq;               // Mq hi, Mq lo, Khat hi, Khat lo
  static constexpr uint32_t m_bytes = KDA ? kVG - kVMq : kMBytes;    // 48 KB
  static constexpr uint32_t g_off = KDA ? kVG : kUG;
  static constexpr uint32_t g_bytes = CM == 2 ? kSU - kVG : KDA ? kVU - kVG : kGBytes;
  static constexpr uint32_t u_off = CM == 2 ? kSU : KDA ? kVU : kUU;
  static constexpr uint32_t cbar = kQG + 2 * g_bytes;
  static constexpr uint32_t smem = cbar + kNBar * 8 + 16;
  static_assert(m_bytes == 49152 && w_bytes <= 65536, "unit regions");
  static_assert(smem <= 227 * 1024 && smem > 114 * 1024, "one pair CTA per SM (its 512 tensor-memory columns)");
};
// MN-major tile of 64 columns (S: rows = key channels, U: rows = tokens):
// 8 consecutive columns per 16 bytes, 8-row groups 1024 bytes apart
__device__ __forceinline__ uint32_t mn64_off(int r, int d) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (d >> 3) * 128 + (r & 7) * 16 + (d & 7) * 2);
}

// the chain of one (batch, head) on CTA `cta` of a pair (cta / 2 is the pair);
// SSE delta: the chain of the (batch, head)'s shared partition, which every
// token visits (its units are the first ceil(T / 64) of the (batch, head))
template <int CM>
__device__ __forceinline__ void chain_pair(const ChainArgs &a, long cta) {
  using L = PairLayout<CM>;
  constexpr bool KDA = CM >= 1, SSE = CM == 2;
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int T = a.T, H = a.H;
  const long bh = cta >> 1;
  const int d0 = 64 * static_cast<int>(cta & 1);  // this CTA's value columns
  const int n = SSE ? (T + kC - 1) / kC : a.nchunks;
  const long u0 = SSE ? bh * a.umax : bh * n;
  float *gS = a.state + (SSE ? bh * (a.N + 1) + a.N : bh) * static_cast<long>(kDK * kDV);
  const long tok0 = (bh / H) * T * H + bh % H;

  unsigned char *sSh = sm + kQS, *sSl = sm + kQS + 16384;
  unsigned char *sUh = sm + kQU, *sUl = sm + kQU + 8192;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + L::cbar);
  // barriers: 0 W, 1 M, 2-3 gamma buffers, 4 phase 1 done, 6 Y2 done (the
  // chunk's last MMA), 7 D done, 8-9 S_ready[g] (key channels 64g..64g+63),
  // 10 U_ready, 11 drain
  auto bar = [&](int i) { return smem_addr(bars + i); };
  uint32_t *holder = reinterpret_cast<uint32_t *>(sm + L::cbar + kNBar * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + L::cbar + kNBar * 8 + 4);

  if (tid == 0) {
    for (int i = 0; i < 8; ++i) mbar_init(bar(i), 1);
    for (int i = 8; i < 11; ++i) mbar_init(bar(i), kWorkers / 64);  // one arrival per worker warp of the half
    mbar_init(bar(11), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(smem_addr(holder), kQTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *holder;

  if (warp < kWorkers / 32) {
    // ------------------------------------------------------------ workers
    // warp w: tensor-memory lanes 32 q .. 32 q + 31 (q = w % 4), value columns
    // 16 qtr .. 16 qtr + 15 of the CTA's 64 (qtr = w / 4)
    const int q = warp & 3, qtr = warp >> 2;
    const int row = 32 * q + lane;  // key channel (state), token (q < 2: X) or token + 64 (q >= 2: Y)
    const int dc = 16 * qtr;        // first of this thread's 16 columns
    const uint32_t lanes = tmem + (static_cast<uint32_t>(32 * q) << 16);
    auto wwait = [&](uint32_t mb, uint32_t parity) -> bool {
      return __all_sync(kFull, chain_wait(mb, parity, abort_flag)) != 0;
    };
    // zero rows of the operand regions that no copy writes: above Mq hi and
    // Mq lo (Y2's A), and (GDN) the Q lo slot of phase 1's lo pass
    {
      uint4 *z0 = reinterpret_cast<uint4 *>(sm + kQM), *z1 = reinterpret_cast<uint4 *>(sm + kQM + 16384);
      for (int i = tid; i < 512; i += kWorkers) z0[i] = z1[i] = make_uint4(0u, 0u, 0u, 0u);
      if (!KDA) {
        uint4 *z2 = reinterpret_cast<uint4 *>(sm + kQW + 49152);
        for (int i = tid; i < 1024; i += kWorkers) z2[i] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    float S[16];  // S[row][d0 + dc + e]
    {
      const float4 *src = reinterpret_cast<const float4 *>(gS + static_cast<long>(row) * kDV + d0 + dc);
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4) {
        const float4 x = src[e4];
        S[4 * e4] = x.x;
        S[4 * e4 + 1] = x.y;
        S[4 * e4 + 2] = x.z;
        S[4 * e4 + 3] = x.w;
      }
    }
    // the bf16 split of this thread's 16 state columns, released by one
    // arrival per warp on S_ready[q / 2]
    auto publish_s = [&]() {
      store_split8(sSh, sSl, mn64_off(row, dc), S);
      store_split8(sSh, sSl, mn64_off(row, dc + 8), S + 8);
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(8 + (q >> 1)));
    };
    publish_s();
    float ut[16];  // Ut[row][d0 + dc + e] of the next chunk (q < 2)
    auto load_ut = [&](int c) {
      const float4 *src = reinterpret_cast<const float4 *>(
          reinterpret_cast<const float *>(a.ws + (u0 + c) * L::unit + L::u_off) + static_cast<long>(row) * kDV + d0 + dc);
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4) {
        const float4 x = __ldg(src + e4);
        ut[4 * e4] = x.x;
        ut[4 * e4 + 1] = x.y;
        ut[4 * e4 + 2] = x.z;
        ut[4 * e4 + 3] = x.w;
      }
    };
    if (q < 2) load_ut(0);
    for (int c = 0; c < n; ++c) {
      const uint32_t par = static_cast<uint32_t>(c & 1);
      const bool last = c + 1 == n;
      if (q < 2) {
        // U = Ut - X for token `row`
        if (!wwait(bar(4), par)) break;
        float x[16];
        tmem_ld16(lanes + kQColXY + 64 * (c & 1) + dc, x);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) x[e] = ut[e] - x[e];
        store_split8(sUh, sUl, mn64_off(row, dc), x);
        store_split8(sUh, sUl, mn64_off(row, dc + 8), x + 8);
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(10));
        if (!last) load_ut(c + 1);
      }
      // this chunk's gammas (loaded long before)
      if (!wwait(bar(2 + (c & 1)), static_cast<uint32_t>((c >> 1) & 1))) break;
      const float *gbuf = reinterpret_cast<const float *>(sm + kQG + (c & 1) * L::g_bytes);
      // GDN's gamma_i of this thread's output token, read before the state is
      // published (the buffer is refilled two chunks on)
      const float gi = (!KDA && q >= 2) ? gbuf[row - 64] : 1.f;
      // SSE: the staging row of this thread's visit (-1 for padding)
      const int sr = (SSE && q >= 2) ? reinterpret_cast<const int *>(gbuf + kDK)[row - 64] : -1;
      // S <- gamma_C S + D; D completing also means phase 1 no longer reads S
      if (!wwait(bar(7), par)) break;
      {
        float x[16];
        tmem_ld16(lanes + kQColD + dc, x);
        tmem_ld_wait();
        const float g = gbuf[KDA ? row : kC - 1];  // KDA: gamma_C per key channel; GDN: gamma of the chunk's last token
#pragma unroll
        for (int e = 0; e < 16; ++e) S[e] = fmaf(g, S[e], x[e]);
      }
      if (!last) {
        publish_s();
      } else {
        float4 *dst = reinterpret_cast<float4 *>(gS + static_cast<long>(row) * kDV + d0 + dc);
#pragma unroll
        for (int e4 = 0; e4 < 4; ++e4) dst[e4] = make_float4(S[4 * e4], S[4 * e4 + 1], S[4 * e4 + 2], S[4 * e4 + 3]);
      }
      if (q >= 2) {
        // y = gamma_i Y1 + Y2 (GDN) or Y1 + Y2 (KDA: the decay is inside Qt)
        if (!wwait(bar(6), par)) break;
        float y1[16], y2[16];
        tmem_ld16(lanes + kQColXY + 64 * (c & 1) + dc, y1);
        tmem_ld16(lanes + kQColY2 + 64 * (c & 1) + dc, y2);
        tmem_ld_wait();
        const int t = c * kC + row - 64;
        if (SSE ? sr >= 0 : t < T) {
          float4 *yp = reinterpret_cast<float4 *>(
              SSE ? a.stage + static_cast<long>(sr) * kDV + d0 + dc : a.y + (tok0 + static_cast<long>(t) * H) * kDV + d0 + dc);
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            float o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) o[e] = KDA ? y1[4 * e4 + e] + y2[4 * e4 + e] : fmaf(gi, y1[4 * e4 + e], y2[4 * e4 + e]);
            yp[e4] = make_float4(o[0], o[1], o[2], o[3]);
          }
        }
      }
    }
  } else if (tid == kWorkers) {
    // ------------------------------------------------------------ producer
    const uint32_t wh = smem_addr(sm + kQW), wl = wh + 32768;  // [W hi; Q hi], [W lo; Qt lo or zeros]
    const uint32_t mz = smem_addr(sm + kQM);                    // zeros | Mq hi | zeros | Mq lo | Khat hi | Khat lo
    const uint32_t kh = mz + 32768, kl = mz + 49152;
    // phase 1: A [W; Q] MN-major (LBO 128 along key channels, SBO 2048 along
    // tokens), B = S MN-major (LBO 1024 along key channels, SBO 128 along
    // value columns); a k-step of 16 key channels advances A 256 bytes, B 2048
    const uint64_t dAh = smem_desc(wh, 128, 2048), dAl = smem_desc(wl, 128, 2048);
    const uint64_t dSh = smem_desc(smem_addr(sSh), 1024, 128), dSl = smem_desc(smem_addr(sSl), 1024, 128);
    // phase 2: A = Khat^T MN-major (LBO 2048 along tokens, SBO 128 along key
    // channels; a k-step of 16 tokens advances 4096 bytes); A = [0; Mq]
    // K-major (LBO 128, SBO 1024; 256 bytes a k-step), starting 64 zero rows
    // (8 KB) above Mq; B = U MN-major (LBO 1024, SBO 128; 2048 bytes a k-step)
    const uint64_t dKh = smem_desc(kh, 2048, 128), dKl = smem_desc(kl, 2048, 128);
    const uint64_t dMh = smem_desc(mz, 128, 1024), dMl = smem_desc(mz + 16384, 128, 1024);
    const uint64_t dUh = smem_desc(smem_addr(sUh), 1024, 128), dUl = smem_desc(smem_addr(sUl), 1024, 128);
    const uint32_t idMM = idesc_bf16_f32(128, 64) | (1u << 15) | (1u << 16);  // A and B MN-major
    const uint32_t idKM = idesc_bf16_f32(128, 64) | (1u << 16);                // A K-major, B MN-major
    int w_issued = 0, w_done = 0, m_issued = 0, m_done = 0, g_issued = 0;
    auto load = [&](int which, int c) {
      const unsigned char *src = a.ws + (u0 + c) * L::unit;
      fence_async_smem();
      if (which == 0) {
        mbar_expect_tx(bar(0), L::w_bytes);
        bulk_g2s(wh, src + L::w_off, L::w_bytes, bar(0));
        ++w_issued;
      } else {
        // Mq hi below its zero rows; Mq lo, Khat hi and Khat lo (contiguous in
        // the unit) below the second zero rows
        mbar_expect_tx(bar(1), L::m_bytes);
        bulk_g2s(mz + 8192, src + L::m_off, 8192, bar(1));
        bulk_g2s(mz + 24576, src + L::m_off + 8192, L::m_bytes - 8192, bar(1));
        mbar_expect_tx(bar(2 + (c & 1)), L::g_bytes);
        bulk_g2s(smem_addr(sm + kQG + (c & 1) * L::g_bytes), src + L::g_off, L::g_bytes, bar(2 + (c & 1)));
        ++m_issued;
        ++g_issued;
      }
    };
    auto prefetch = [&](int c) {
      const unsigned char *pf = a.ws + (u0 + c) * L::unit;
      prefetch_l2(pf + L::w_off, L::w_bytes / 2);
      prefetch_l2(pf + L::w_off + L::w_bytes / 2, L::w_bytes / 2);
      prefetch_l2(pf + L::m_off, L::m_bytes + L::g_bytes);
      prefetch_l2(pf + L::u_off, L::unit - L::u_off);
    };
    if (n > 1) prefetch(1);
    load(0, 0);
    load(1, 0);
    bool ok = true;
    for (int c = 0; c < n && ok; ++c) {
      const uint32_t par = static_cast<uint32_t>(c & 1);
      if (c + 2 < n) prefetch(c + 2);
      // phase 1, key channels 64 g .. 64 g + 63 (k-steps 4 g .. 4 g + 3) as
      // their half of S is published: A hi x S hi, A lo x S hi, A hi x S lo
      const uint32_t xy = tmem + kQColXY + 64 * (c & 1);
      ok = producer_wait(bar(0), par, abort_flag);
      if (ok) ++w_done;
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        if (ok) ok = producer_wait(bar(8 + g), par, abort_flag);
        if (!ok) break;
#pragma unroll
        for (int ks = 4 * g; ks < 4 * g + 4; ++ks) {
          mma_bf16(xy, dAh + 16u * ks, dSh + 128u * ks, idMM, ks != 0);
          mma_bf16(xy, dAl + 16u * ks, dSh + 128u * ks, idMM, true);
          mma_bf16(xy, dAh + 16u * ks, dSl + 128u * ks, idMM, true);
        }
      }
      if (!ok) break;
      if (!(a.drop_signal && c == 0)) mma_commit(bar(4));
      if (c + 1 < n) {
        ok = producer_wait(bar(4), par, abort_flag);
        if (!ok) break;
        load(0, c + 1);
      }
      // phase 2: D = Khat^T U (the state update waits for it), then Y2
      ok = producer_wait(bar(1), par, abort_flag);
      if (ok) ++m_done;
      if (ok) ok = producer_wait(bar(10), par, abort_flag);
      if (!ok) break;
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(tmem + kQColD, dKh + 256u * ks, dUh + 128u * ks, idMM, ks != 0);
        mma_bf16(tmem + kQColD, dKl + 256u * ks, dUh + 128u * ks, idMM, true);
        mma_bf16(tmem + kQColD, dKh + 256u * ks, dUl + 128u * ks, idMM, true);
      }
      mma_commit(bar(7));
      const uint32_t y2 = tmem + kQColY2 + 64 * (c & 1);
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        mma_bf16(y2, dMh + 16u * ks, dUh + 128u * ks, idKM, ks != 0);
        mma_bf16(y2, dMl + 16u * ks, dUh + 128u * ks, idKM, true);
        mma_bf16(y2, dMh + 16u * ks, dUl + 128u * ks, idKM, true);
      }
      mma_commit(bar(6));
      if (c + 1 < n) {
        ok = producer_wait(bar(6), par, abort_flag);
        if (ok) load(1, c + 1);
      }
    }
    mma_commit(bar(11));
    mbar_wait(bar(11), 0, kWaitLimit);
    if (w_done < w_issued) mbar_wait(bar(0), static_cast<uint32_t>((w_issued - 1) & 1), kWaitLimit);
    if (m_done < m_issued) mbar_wait(bar(1), static_cast<uint32_t>((m_issued - 1) & 1), kWaitLimit);
    for (int gb = 0; gb < 2; ++gb) {
      const int loads = (g_issued + 1 - gb) / 2;
      if (loads > 0) mbar_wait(bar(2 + gb), static_cast<uint32_t>((loads - 1) & 1), kWaitLimit);
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) report_timeout(a.err);
  if (warp == 0) tmem_dealloc(tmem, kQTmemCols);
}

template <int CM>
__global__ void __maxnreg__(96) gdn_chain_pair_kernel(const ChainArgs a) {
  chain_pair<CM>(a, blockIdx.x);
}

// SSE delta write: the shared partitions' chains (the longest: every token
// visits them) on CTA pairs, first, then the routed partitions' chains on one
// CTA each, in one launch
__global__ void __maxnreg__(96) gdn_chain_sse_kernel(const ChainArgs a) {
  if (static_cast<long>(blockIdx.x) < 2 * a.bhn)
    chain_pair<2>(a, blockIdx.x);
  else
    chain_single<2>(a, static_cast<long>(blockIdx.x) - a.bhn);
}

}  // namespace

// workspace of the chunked GDN path: one unit of tiles per chunk
size_t gdn_chunk_workspace_size(int B, int T, int H) {
  const long units = static_cast<long>(B) * H * ((T + kC - 1) / kC);
  const size_t n = static_cast<size_t>(units) * kUnit;
  return (n + 255) & ~static_cast<size_t>(255);
}

// Test hook for the failure path: SDM_TEST_DROP_SIGNAL=1 makes the chain
// kernels skip one mbarrier signal, so a bounded on-device wait runs out and
// the call reports SDM_DEVERR_TIMEOUT (outputs invalid) with the context
// still usable.  Read per call; off unless set.
int test_drop_signal() {
  const char *s = getenv("SDM_TEST_DROP_SIGNAL");
  return (s && s[0] == '1') ? 1 : 0;
}

// The chain's form: a CTA pair per (b, h) (value columns split) when every
// pair is resident at once, else one CTA per (b, h).  SDM_GDN_CHAIN=single or
// =pair forces one form (read per call).
bool chain_in_pairs(long bh, int sms) {
  const char *s = getenv("SDM_GDN_CHAIN");
  if (s && strcmp(s, "single") == 0) return false;
  if (s && strcmp(s, "pair") == 0) return true;
  return 2 * bh <= sms;
}

// launched by gdn_scan for dense GDN with d_k = d_v = 128
int launch_gdn_chunk(float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                     const float *beta, int B, int T, int H, float *y, void *workspace, int32_t *err,
                     cudaStream_t st) {
  const int nchunks = (T + kC - 1) / kC;
  const long units = static_cast<long>(B) * H * nchunks;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

  PrepArgs pa{};
  pa.q = q;
  pa.k = k;
  pa.v = v;
  pa.alpha = alpha;
  pa.beta = beta;
  pa.ws = ws;
  pa.T = T;
  pa.H = H;
  pa.nchunks = nchunks;
  pa.units = units;
  pa.err = err;
  if (cudaFuncSetAttribute(gdn_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kPrepSmem)) != cudaSuccess)
    return check_launch("gdn_scan: set shared memory");
  const long pmax = static_cast<long>(sms) * kPrepCtasPerSm;
  const long pgrid = units < pmax ? units : pmax;
  gdn_prep_kernel<<<static_cast<unsigned>(pgrid), kThreads, kPrepSmem, st>>>(pa);
  const int rc = check_launch("gdn_scan: chunk preparation kernel");
  if (rc != SDM_OK) return rc;

  ChainArgs ca{};
  ca.state = state;
  ca.ws = ws;
  ca.y = y;
  ca.T = T;
  ca.H = H;
  ca.nchunks = nchunks;
  ca.err = err;
  ca.drop_signal = test_drop_signal();
  const long bh = static_cast<long>(B) * H;
  if (chain_in_pairs(bh, sms)) {
    constexpr uint32_t pair_smem = PairLayout<0>::smem;
    if (cudaFuncSetAttribute(gdn_chain_pair_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(pair_smem)) != cudaSuccess)
      return check_launch("gdn_scan: set shared memory");
    gdn_chain_pair_kernel<0><<<static_cast<unsigned>(2 * bh), kChainThreads, pair_smem, st>>>(ca);
    return check_launch("gdn_scan: chunk chain kernel");
  }
  constexpr uint32_t chain_smem = ChainLayout<0>::smem;
  if (cudaFuncSetAttribute(gdn_chain_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(chain_smem)) != cudaSuccess)
    return check_launch("gdn_scan: set shared memory");
  gdn_chain_kernel<0><<<static_cast<unsigned>(bh), kChainThreads, chain_smem, st>>>(ca);
  return check_launch("gdn_scan: chunk chain kernel");
}

// workspace of the chunked KDA path: one unit of tiles per chunk
size_t kda_chunk_workspace_size(int B, int T, int H) {
  const long units = static_cast<long>(B) * H * ((T + kC - 1) / kC);
  const size_t n = static_cast<size_t>(units) * kVUnit;
  return (n + 255) & ~static_cast<size_t>(255);
}

// launched by gdn_scan for KDA (a decay per key channel) and by gdn2_scan for
// GDN2 (b_erase, w_write non-null), both with d_k = d_v = 128
int launch_kda_chunk(float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                     const float *beta, const float *b_erase, const float *w_write, int B, int T, int H, float *y,
                     void *workspace, int32_t *err, cudaStream_t st) {
  const int nchunks = (T + kC - 1) / kC;
  const long units = static_cast<long>(B) * H * nchunks;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const bool g2 = b_erase != nullptr;

  KdaPrepArgs pa{};
  pa.q = q;
  pa.k = k;
  pa.v = v;
  pa.alpha = alpha;
  pa.beta = beta;
  pa.b_erase = b_erase;
  pa.w_write = w_write;
  pa.ws = ws;
  pa.T = T;
  pa.H = H;
  pa.nchunks = nchunks;
  pa.units = units;
  pa.err = err;
  const long pgrid = units < sms ? units : sms;
  if (g2) {
    if (cudaFuncSetAttribute(kda_prep_kernel<kModeGdn2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kKdaSmem)) != cudaSuccess)
      return check_launch("gdn2_scan: set shared memory");
    kda_prep_kernel<kModeGdn2><<<static_cast<unsigned>(pgrid), kKThreads, kKdaSmem, st>>>(pa);
  } else {
    if (cudaFuncSetAttribute(kda_prep_kernel<kModeKda>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kKdaSmem)) != cudaSuccess)
      return check_launch("gdn_scan: set shared memory");
    kda_prep_kernel<kModeKda><<<static_cast<unsigned>(pgrid), kKThreads, kKdaSmem, st>>>(pa);
  }
  const int rc = check_launch(g2 ? "gdn2_scan: chunk preparation kernel" : "gdn_scan: KDA chunk preparation kernel");
  if (rc != SDM_OK) return rc;

  ChainArgs ca{};
  ca.state = state;
  ca.ws = ws;
  ca.y = y;
  ca.T = T;
  ca.H = H;
  ca.nchunks = nchunks;
  ca.err = err;
  ca.drop_signal = test_drop_signal();
  const long bh = static_cast<long>(B) * H;
  if (chain_in_pairs(bh, sms)) {
    constexpr uint32_t pair_smem = PairLayout<1>::smem;
    if (cudaFuncSetAttribute(gdn_chain_pair_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(pair_smem)) != cudaSuccess)
      return check_launch("gdn_scan: set shared memory");
    gdn_chain_pair_kernel<1><<<static_cast<unsigned>(2 * bh), kChainThreads, pair_smem, st>>>(ca);
    return check_launch(g2 ? "gdn2_scan: chunk chain kernel" : "gdn_scan: KDA chunk chain kernel");
  }
  constexpr uint32_t chain_smem = ChainLayout<1>::smem;
  if (cudaFuncSetAttribute(gdn_chain_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(chain_smem)) != cudaSuccess)
    return check_launch("gdn_scan: set shared memory");
  gdn_chain_kernel<1><<<static_cast<unsigned>(bh), kChainThreads, chain_smem, st>>>(ca);
  return check_launch(g2 ? "gdn2_scan: chunk chain kernel" : "gdn_scan: KDA chunk chain kernel");
}

// bytes of one unit of the SSE delta prefill (sse_chunk.cu sizes the workspace)
size_t sse_delta_unit_bytes() { return kSUnit; }

// launched by sse_scan's chunked path for the delta write, after the routing
// and group kernels: the chunk preparation of every unit (its visits gathered
// from the group table), then one chain CTA per (batch, head, partition)
// writing each visit's gated read to its staging row
int launch_sse_delta_chunk(float *state, const uint32_t *rec, int rw, const uint32_t *grp, long gwords, int umax,
                           const float *klog, const uint16_t *q, const uint16_t *v, const float *alpha, int B, int T,
                           int H, int N, int topk, unsigned char *units, float *stage, int32_t *err, cudaStream_t st) {
  const long bhn = static_cast<long>(B) * H;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

  KdaPrepArgs pa{};
  pa.q = q;
  pa.v = v;
  pa.alpha = alpha;
  pa.klog = klog;
  pa.rec = rec;
  pa.grp = grp;
  pa.N = N;
  pa.topk = topk;
  pa.rw = rw;
  pa.umax = umax;
  pa.gwords = gwords;
  pa.ws = units;
  pa.T = T;
  pa.H = H;
  pa.nchunks = umax;
  pa.units = bhn * umax;
  pa.err = err;
  if (cudaFuncSetAttribute(kda_prep_kernel<kModeSse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kKdaSmem)) != cudaSuccess)
    return check_launch("sse_scan: set shared memory");
  const long pgrid = pa.units < sms ? pa.units : sms;
  kda_prep_kernel<kModeSse><<<static_cast<unsigned>(pgrid), kKThreads, kKdaSmem, st>>>(pa);
  int rc = check_launch("sse_scan: delta chunk preparation kernel");
  if (rc != SDM_OK) return rc;

  ChainArgs ca{};
  ca.state = state;
  ca.ws = units;
  ca.T = T;
  ca.H = H;
  ca.nchunks = umax;
  ca.grp = grp;
  ca.gwords = gwords;
  ca.bhn = bhn;
  ca.umax = umax;
  ca.N = N;
  ca.stage = stage;
  ca.err = err;
  ca.drop_signal = test_drop_signal();
  if (chain_in_pairs(bhn, sms)) {
    constexpr uint32_t sse_smem =
        PairLayout<2>::smem > ChainLayout<2>::smem ? PairLayout<2>::smem : ChainLayout<2>::smem;
    if (cudaFuncSetAttribute(gdn_chain_sse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(sse_smem)) != cudaSuccess)
      return check_launch("sse_scan: set shared memory");
    gdn_chain_sse_kernel<<<static_cast<unsigned>(bhn * (N + 2)), kChainThreads, sse_smem, st>>>(ca);
    return check_launch("sse_scan: delta chunk chain kernel");
  }
  constexpr uint32_t chain_smem = ChainLayout<2>::smem;
  if (cudaFuncSetAttribute(gdn_chain_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(chain_smem)) != cudaSuccess)
    return check_launch("sse_scan: set shared memory");
  gdn_chain_kernel<2><<<static_cast<unsigned>(bhn * (N + 1)), kChainThreads, chain_smem, st>>>(ca);
  return check_launch("sse_scan: delta chunk chain kernel");
}

SDM_STICKY_ACCESSOR(sticky_gdn_chunk)

}  // namespace sdm
