// chunked_scan.cu - the sparse delta-rule memory scan in chunked form (Sparse
// Delta Memory deck, "Training parallelizes within chunks and recurs across
// chunks" and "Backup: sparse interactions drive the triangular solve",
// App. A.1-A.2, Eq. 7): the same result as sdm_scan (shared residual or
// additive write), with the work inside a chunk of C = 64 tokens done in
// parallel instead of token by token.
//
// Within a chunk, lambda_i(s) is the sum of log alpha over the tokens j <= i
// that write slot s (the slot's decay clock), u_i = v_i - vhat_i token i's
// shared residual, and
//   (I + A diag(beta)) u = v - p,       p_i = sum_n k_in e^{lambda_i(s_in)} M0[s_in]
//   A[i,j] = sum_{n,m: s_in = s_jm} k_in k_jm e^{lambda_i(s) - lambda_j(s)}   (j < i)
//   y_i = sum_m r_im e^{lambda_i(rho_im)} M0[rho_im] + sum_{j<=i} beta_j Qr[i,j] u_j
//   Qr[i,j] = sum_{m,n: rho_im = s_jn} r_im k_jn e^{lambda_i(rho) - lambda_j(rho)}
//   M_C[s] = e^{lambda_C(s)} M0[s] + sum_{j writes s} beta_j k_j(s) e^{lambda_C(s) - lambda_j(s)} u_j
// (additive write: u = v).  Two kernels:
//   chunk_prep_kernel  - every chunk in parallel: sorts the chunk's write
//                        pairs by (slot, token), accumulates the decay clocks
//                        along each slot's run, builds A and Qr row by row
//                        (one thread per token, deterministic), inverts
//                        I + A diag(beta), and writes T, beta Qr and the
//                        per-pair coefficients to the workspace.
//   chunk_chain_kernel - one CTA per (batch, head, 32-column tile), chunks in
//                        order: every gather of a chunk at once, u = T (v - p),
//                        y, and one scatter per distinct written slot.
#include <climits>

#include "common.cuh"

namespace sdm {
namespace {

constexpr int kCC = 64;         // tokens per chunk
constexpr int kCS = 16;         // slots per token (W, R <= 16)
constexpr int kCP = kCC * kCS;  // pair slots per chunk: pair p = 16 * token + position
constexpr int kCLd = kCC + 4;   // padded fp32 row stride of the solve
constexpr int kPrepThreads = 256;

// one chunk's record in the workspace (bytes)
constexpr uint32_t kXT = 0;                    // T = (I + A diag beta)^-1, fp32 [64][64]
constexpr uint32_t kXQ = kXT + kCC * kCC * 4;  // beta_j Qr[i][j], fp32 [64][64]
constexpr uint32_t kXWs = kXQ + kCC * kCC * 4; // write pairs: slot, int32 (-1: none)
constexpr uint32_t kXWcp = kXWs + kCP * 4;     // k_in e^{lambda_i(s)}
constexpr uint32_t kXWsc = kXWcp + kCP * 4;    // beta_i k_in e^{lambda_C(s) - lambda_i(s)}
constexpr uint32_t kXWln = kXWsc + kCP * 4;    // int32: 1 + previous pair of the slot's run (0: none) | kLast
constexpr uint32_t kXWdc = kXWln + kCP * 4;    // e^{lambda_C(s)} (last pair of a run)
constexpr uint32_t kXRs = kXWdc + kCP * 4;     // read pairs: slot, int32 (-1: none)
constexpr uint32_t kXRc = kXRs + kCP * 4;      // r_im e^{lambda_i(rho)}
constexpr uint32_t kXUnit = kXRc + kCP * 4;
constexpr int32_t kLast = 1 << 30;
static_assert(kXUnit % 16 == 0, "16-byte records");

struct ChunkArgs {
  float *state;
  const void *v;
  const float *alpha, *beta;
  const int32_t *idx_w, *idx_r;
  const float *w_w, *w_r;
  float *y;
  unsigned char *ws;
  int32_t *err;
  int T, H, N, d_v, W, R, additive, v_bf16, nchunks, tiles;
};

// X = L^-1 for a unit lower-triangular 64 x 64 L given by its strict lower
// part sL (row stride kCLd): 16 x 16 diagonal blocks by substitution, then the
// blocks below, one block distance at a time: X_IJ = -X_II sum_{K=J}^{I-1} L_IK X_KJ
__device__ void unit_lower_inverse(const float *sL, float *sX, float *sZ, int tid) {
  if (tid < 64) {
    const int I = tid >> 4, cc = tid & 15, o = I * 16;
    float xv[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float acc = (r == cc) ? 1.f : 0.f;
#pragma unroll
      for (int j = 0; j < r; ++j) acc -= sL[(o + r) * kCLd + o + j] * xv[j];
      xv[r] = acc;
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) sX[(o + r) * kCLd + o + cc] = xv[r];
  }
  __syncthreads();
#pragma unroll
  for (int dist = 1; dist < 4; ++dist) {
    const bool mine = tid < (4 - dist) * 64;
    const int p = tid >> 6, r = (tid >> 2) & 15, c4 = (tid & 3) * 4;
    const int J = p, I = p + dist;
    if (mine) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int K = 0; K < dist; ++K)
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
          const float l = sL[(I * 16 + r) * kCLd + (J + K) * 16 + kk];
          const float4 x = *reinterpret_cast<const float4 *>(sX + ((J + K) * 16 + kk) * kCLd + J * 16 + c4);
          acc[0] = fmaf(l, x.x, acc[0]);
          acc[1] = fmaf(l, x.y, acc[1]);
          acc[2] = fmaf(l, x.z, acc[2]);
          acc[3] = fmaf(l, x.w, acc[3]);
        }
      *reinterpret_cast<float4 *>(sZ + p * 256 + r * 16 + c4) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    }
    __syncthreads();
    if (mine) {
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int kk = 0; kk < 16; ++kk) {
        const float x = sX[(I * 16 + r) * kCLd + I * 16 + kk];
        const float4 z = *reinterpret_cast<const float4 *>(sZ + p * 256 + kk * 16 + c4);
        acc[0] = fmaf(x, z.x, acc[0]);
        acc[1] = fmaf(x, z.y, acc[1]);
        acc[2] = fmaf(x, z.z, acc[2]);
        acc[3] = fmaf(x, z.w, acc[3]);
      }
      *reinterpret_cast<float4 *>(sX + (I * 16 + r) * kCLd + J * 16 + c4) =
          make_float4(-acc[0], -acc[1], -acc[2], -acc[3]);
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Kernel 1: the state-independent part of every chunk.
// ---------------------------------------------------------------------------
// shared memory of the preparation kernel (bytes)
constexpr uint32_t kPKeys = 0;                      // (slot * 64 + token) << 32 | pair, ascending   [1024] u64
constexpr uint32_t kPLam = kPKeys + kCP * 8;        // decay clock of the slot at each sorted position [1024] f32
constexpr uint32_t kPWk = kPLam + kCP * 4;          // write weight of each pair                        [1024] f32
constexpr uint32_t kPA = kPWk + kCP * 4;            // A, then L = A diag(beta)                        [64][68] f32
constexpr uint32_t kPX = kPA + kCC * kCLd * 4;      // L^-1                                            [64][68] f32
constexpr uint32_t kPZ = kPX + kCC * kCLd * 4;      // block products                                  [3][256] f32
constexpr uint32_t kPLa = kPZ + 3 * 256 * 4;        // log alpha, beta of each token                    [2][64] f32
constexpr uint32_t kPPos = kPLa + 2 * kCC * 4;      // sorted position of each pair (-1: none)          [1024] i16
constexpr uint32_t kPrepSmemC = kPPos + kCP * 2;

__global__ void __launch_bounds__(kPrepThreads) chunk_prep_kernel(const ChunkArgs a) {
  extern __shared__ __align__(16) unsigned char smp[];
  unsigned long long *keys = reinterpret_cast<unsigned long long *>(smp + kPKeys);
  float *lamq = reinterpret_cast<float *>(smp + kPLam);
  float *wk = reinterpret_cast<float *>(smp + kPWk);
  float *sA = reinterpret_cast<float *>(smp + kPA);
  float *sX = reinterpret_cast<float *>(smp + kPX);
  float *sZ = reinterpret_cast<float *>(smp + kPZ);
  float *la = reinterpret_cast<float *>(smp + kPLa), *be = la + kCC;
  int16_t *pos = reinterpret_cast<int16_t *>(smp + kPPos);
  const int tid = threadIdx.x;
  const long unit = blockIdx.x;
  const long bh = unit / a.nchunks;
  const int c = static_cast<int>(unit - bh * a.nchunks);
  const int T = a.T, H = a.H, W = a.W, R = a.R;
  const long tok0 = (bh / H) * T * H + bh % H;
  const int t0 = c * kCC;
  const int L = min(kCC, T - t0);
  unsigned char *ws = a.ws + unit * kXUnit;
  bool bad_range = false, bad_repeat = false;

  if (tid < kCC) {
    const long tok = tok0 + static_cast<long>(t0 + tid) * H;
    la[tid] = tid < L ? __logf(a.alpha[tok]) : 0.f;
    be[tid] = tid < L ? a.beta[tok] : 0.f;
  }
  for (int p = tid; p < kCP; p += kPrepThreads) {
    const int i = p >> 4, n = p & 15;
    int slot = -1;
    float w = 0.f;
    if (i < L && n < W) {
      const long tok = tok0 + static_cast<long>(t0 + i) * H;
      slot = a.idx_w[tok * W + n];
      w = a.w_w[tok * W + n];
      if (static_cast<unsigned>(slot) >= static_cast<unsigned>(a.N)) { bad_range = true; slot = -1; w = 0.f; }
    }
    wk[p] = w;
    pos[p] = -1;
    keys[p] = slot < 0 ? ~0ull
                       : (static_cast<unsigned long long>(static_cast<unsigned>(slot) * 64u + i) << 32) | p;
  }
  for (int e = tid; e < kCC * kCLd; e += kPrepThreads) sA[e] = 0.f;
  __syncthreads();
  // bitonic sort of the 1024 keys
  for (int k = 2; k <= kCP; k <<= 1)
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int t = tid; t < kCP; t += kPrepThreads) {
        const int o = t ^ j;
        if (o > t) {
          const unsigned long long x = keys[t], y = keys[o];
          if ((x > y) == ((t & k) == 0)) {
            keys[t] = y;
            keys[o] = x;
          }
        }
      }
      __syncthreads();
    }
  auto slot_of = [&](int q) { return static_cast<unsigned>(keys[q] >> 38); };        // key >> 32 >> 6
  auto tok_of = [&](int q) { return static_cast<int>((keys[q] >> 32) & 63); };
  auto pair_of = [&](int q) { return static_cast<int>(keys[q] & 0xffffffffu); };
  auto valid = [&](int q) { return keys[q] != ~0ull; };
  // decay clocks along each slot's run (runs sorted by token)
  for (int q = tid; q < kCP; q += kPrepThreads) {
    if (!valid(q)) continue;
    pos[pair_of(q)] = static_cast<int16_t>(q);
    float lam = la[tok_of(q)];
    for (int r = q - 1; r >= 0 && slot_of(r) == slot_of(q); --r) lam += la[tok_of(r)];
    lamq[q] = lam;
    if (q > 0 && (keys[q - 1] >> 32) == (keys[q] >> 32)) bad_repeat = true;  // a slot twice in one token
  }
  __syncthreads();
  // A (row i: the write pairs of token i and the earlier writes of their slots),
  // Qr and the read coefficients (row i: the reads of token i)
  float *gQ = reinterpret_cast<float *>(ws + kXQ);
  if (tid < kCC) {
    const int i = tid;
    float qrow[kCC];
#pragma unroll
    for (int j = 0; j < kCC; ++j) qrow[j] = 0.f;
    if (i < L) {
      for (int n = 0; n < W; ++n) {
        const int q = pos[i * kCS + n];
        if (q < 0) continue;
        const int p = i * kCS + n;
        const unsigned s = slot_of(q);
        for (int r = q - 1; r >= 0 && slot_of(r) == s; --r)
          sA[i * kCLd + tok_of(r)] += wk[p] * wk[pair_of(r)] * __expf(lamq[q] - lamq[r]);
      }
      const long tok = tok0 + static_cast<long>(t0 + i) * H;
      for (int m = 0; m < R; ++m) {
        const int rho = a.idx_r[tok * R + m];
        const float rw = a.w_r[tok * R + m];
        float coef = 0.f;
        int slot_out = -1;
        if (static_cast<unsigned>(rho) < static_cast<unsigned>(a.N)) {
          slot_out = rho;
          // the last write of rho at a token <= i: largest key <= (rho*64 + i) << 32 | max
          const unsigned long long bound = (static_cast<unsigned long long>(static_cast<unsigned>(rho) * 64u + i) << 32) |
                                           0xffffffffull;
          int lo = 0, hi = kCP;  // first position with key > bound
          while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (keys[mid] <= bound) lo = mid + 1;
            else hi = mid;
          }
          const int ql = lo - 1;
          float lam_i = 0.f;
          if (ql >= 0 && valid(ql) && slot_of(ql) == static_cast<unsigned>(rho)) {
            lam_i = lamq[ql];
            for (int r = ql; r >= 0 && slot_of(r) == static_cast<unsigned>(rho); --r)
              qrow[tok_of(r)] += rw * wk[pair_of(r)] * __expf(lam_i - lamq[r]) * be[tok_of(r)];
          }
          coef = rw * __expf(lam_i);
        } else {
          bad_range = true;
        }
        reinterpret_cast<int32_t *>(ws + kXRs)[i * kCS + m] = slot_out;
        reinterpret_cast<float *>(ws + kXRc)[i * kCS + m] = coef;
      }
    }
#pragma unroll
    for (int j = 0; j < kCC; ++j) gQ[i * kCC + j] = qrow[j];
    for (int m = (i < L ? R : 0); m < kCS; ++m) {
      reinterpret_cast<int32_t *>(ws + kXRs)[i * kCS + m] = -1;
      reinterpret_cast<float *>(ws + kXRc)[i * kCS + m] = 0.f;
    }
  }
  // the write pairs' coefficients, run links and end-of-chunk decays
  for (int p = tid; p < kCP; p += kPrepThreads) {
    const int q = pos[p];
    const bool ok = q >= 0;
    int32_t slot = -1, ln = 0;
    float cp = 0.f, sc = 0.f, dc = 0.f;
    if (ok) {
      const unsigned s = slot_of(q);
      int qe = q;
      while (qe + 1 < kCP && valid(qe + 1) && slot_of(qe + 1) == s) ++qe;
      const int i = p >> 4;
      slot = static_cast<int32_t>(s);
      cp = wk[p] * __expf(lamq[q]);
      sc = be[i] * wk[p] * __expf(lamq[qe] - lamq[q]);
      ln = (q > 0 && valid(q - 1) && slot_of(q - 1) == s) ? 1 + pair_of(q - 1) : 0;
      if (qe == q) {
        ln |= kLast;
        dc = __expf(lamq[q]);
      }
    }
    reinterpret_cast<int32_t *>(ws + kXWs)[p] = slot;
    reinterpret_cast<float *>(ws + kXWcp)[p] = cp;
    reinterpret_cast<float *>(ws + kXWsc)[p] = sc;
    reinterpret_cast<int32_t *>(ws + kXWln)[p] = ln;
    reinterpret_cast<float *>(ws + kXWdc)[p] = dc;
  }
  __syncthreads();
  // T = (I + A diag(beta))^-1 (identity for the additive write)
  if (!a.additive) {
    for (int e = tid; e < kCC * kCC; e += kPrepThreads) {
      const int i = e >> 6, j = e & 63;
      sA[i * kCLd + j] = j < i ? sA[i * kCLd + j] * be[j] : 0.f;
    }
    __syncthreads();
    unit_lower_inverse(sA, sX, sZ, tid);
  }
  float *gT = reinterpret_cast<float *>(ws + kXT);
  for (int e = tid; e < kCC * kCC; e += kPrepThreads) {
    const int i = e >> 6, j = e & 63;
    gT[e] = a.additive ? (i == j ? 1.f : 0.f) : (j <= i ? sX[i * kCLd + j] : 0.f);
  }
  const int any_range = __syncthreads_or(bad_range), any_repeat = __syncthreads_or(bad_repeat);
  if (tid == 0 && a.err && any_range) atomicOr(a.err, SDM_DEVERR_INDEX_RANGE);
  if (tid == 0 && a.err && any_repeat) atomicOr(a.err, SDM_DEVERR_INDEX_REPEAT);
}

// ---------------------------------------------------------------------------
// Kernel 2: chunks in order, one CTA per (batch, head, 32-column tile).
// Warp w computes tokens 8w .. 8w+7 of a chunk; lane = column.
// ---------------------------------------------------------------------------
constexpr int kChainThreadsC = 256;
constexpr int kRS = 33;  // padded row stride of the [64][32] per-column tiles

__global__ void __launch_bounds__(kChainThreadsC) chunk_chain_kernel(const ChunkArgs a) {
  extern __shared__ __align__(16) unsigned char smc[];
  unsigned char *rec = smc;                                        // the chunk's record (kXUnit bytes)
  float *sr = reinterpret_cast<float *>(smc + kXUnit);             // v - p   [64][33]
  float *su = sr + kCC * kRS;                                      // u       [64][33]
  const float *sT = reinterpret_cast<const float *>(rec + kXT);
  const float *sQ = reinterpret_cast<const float *>(rec + kXQ);
  const int32_t *sWs = reinterpret_cast<const int32_t *>(rec + kXWs);
  const float *sWcp = reinterpret_cast<const float *>(rec + kXWcp);
  const float *sWsc = reinterpret_cast<const float *>(rec + kXWsc);
  const int32_t *sWln = reinterpret_cast<const int32_t *>(rec + kXWln);
  const float *sWdc = reinterpret_cast<const float *>(rec + kXWdc);
  const int32_t *sRs = reinterpret_cast<const int32_t *>(rec + kXRs);
  const float *sRc = reinterpret_cast<const float *>(rec + kXRc);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tile = static_cast<int>(blockIdx.x % a.tiles);
  const long bh = blockIdx.x / a.tiles;
  const int T = a.T, H = a.H, d_v = a.d_v, W = a.W, R = a.R;
  const long tok0 = (bh / H) * T * H + bh % H;
  const int col = tile * 32 + lane;
  const bool active = col < d_v;
  const int ccol = active ? col : 0;
  float *M = a.state + bh * static_cast<long>(a.N) * d_v + ccol;

  for (int c = 0; c < a.nchunks; ++c) {
    const int t0 = c * kCC;
    const int L = min(kCC, T - t0);
    const uint4 *src = reinterpret_cast<const uint4 *>(a.ws + (bh * a.nchunks + c) * kXUnit);
    for (int e = tid; e < static_cast<int>(kXUnit / 16); e += kChainThreadsC) reinterpret_cast<uint4 *>(rec)[e] = src[e];
    __syncthreads();
    // every gather of the chunk: p (write rows) and the chunk-start part of y (read rows)
    float y0[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = warp * 8 + k;
      float r = 0.f, yy = 0.f;
      if (i < L) {
        const long tok = tok0 + static_cast<long>(t0 + i) * H;
        const float vv = a.v_bf16 ? bf16_to_f32(static_cast<const uint16_t *>(a.v)[tok * d_v + ccol])
                                  : static_cast<const float *>(a.v)[tok * d_v + ccol];
        // the token's 16 write rows and 16 read rows, all loads in flight at once
        float gw[kCS], gr[kCS];
#pragma unroll
        for (int n = 0; n < kCS; ++n) {
          const int sw = (!a.additive && n < W) ? sWs[i * kCS + n] : -1;
          const int sr_ = n < R ? sRs[i * kCS + n] : -1;
          gw[n] = sw >= 0 ? M[static_cast<long>(sw) * d_v] : 0.f;
          gr[n] = sr_ >= 0 ? M[static_cast<long>(sr_) * d_v] : 0.f;
        }
        float p = 0.f;
#pragma unroll
        for (int n = 0; n < kCS; ++n) {
          p = fmaf(sWcp[i * kCS + n], gw[n], p);   // unused pairs have coefficient 0
          yy = fmaf(sRc[i * kCS + n], gr[n], yy);
        }
        r = vv - p;
      }
      sr[i * kRS + lane] = r;
      y0[k] = yy;
    }
    __syncthreads();
    // u = T (v - p)
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = warp * 8 + k;
      float u = 0.f;
      for (int j = 0; j <= i; ++j) u = fmaf(sT[i * kCC + j], sr[j * kRS + lane], u);
      su[i * kRS + lane] = u;
    }
    __syncthreads();
    // y = chunk-start reads + beta Qr u
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = warp * 8 + k;
      if (i < L) {
        float yy = y0[k];
        for (int j = 0; j <= i; ++j) yy = fmaf(sQ[i * kCC + j], su[j * kRS + lane], yy);
        if (active) a.y[(tok0 + static_cast<long>(t0 + i) * H) * d_v + col] = yy;
      }
    }
    // one scatter per distinct written slot, by the warp holding its run's last
    // pair; 32 pairs at a time: their old rows are loaded together, then updated
    for (int base = warp * (kCP / 8); base < (warp + 1) * (kCP / 8); base += 32) {
      float old[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int p = base + k;
        old[k] = (sWln[p] & kLast) ? M[static_cast<long>(sWs[p]) * d_v] : 0.f;
      }
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const int p = base + k;
        if (!(sWln[p] & kLast)) continue;
        float val = sWdc[p] * old[k];
        for (int q = p; q >= 0;) {
          val = fmaf(sWsc[q], su[(q >> 4) * kRS + lane], val);
          q = (sWln[q] & 0xffff) - 1;
        }
        if (active) M[static_cast<long>(sWs[p]) * d_v] = val;
      }
    }
    __syncthreads();
  }
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" size_t sdm_scan_chunked_workspace_size(int B, int T, int H, int W, int R) {
  if (B <= 0 || T <= 0 || H <= 0 || W <= 0 || R <= 0) return 0;
  const size_t chunks = static_cast<size_t>(B) * H * ((T + kCC - 1) / kCC);
  return chunks * kXUnit;
}

extern "C" int sdm_scan_chunked(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
                                const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r,
                                const float *w_r, int R, int B, int T, int H, int N, int d_v, int resid_mode, float *y,
                                void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream) {
  if (!state || !v || !alpha || !beta || !idx_w || !w_w || !idx_r || !w_r || !y)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan_chunked: null pointer");
  if (B < 0 || T < 0 || H < 0 || N < 1 || d_v < 1)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan_chunked: bad sizes");
  if (W < 1 || W > kCS || R < 1 || R > kCS) return set_error(SDM_ERR_SHAPE, "sdm_scan_chunked: need 1 <= W, R <= 16");
  if (N > (1 << 25)) return set_error(SDM_ERR_SHAPE, "sdm_scan_chunked: N must be at most 2^25");
  if (v_dtype != SDM_DTYPE_F32 && v_dtype != SDM_DTYPE_BF16)
    return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan_chunked: v_dtype must be SDM_DTYPE_F32 or SDM_DTYPE_BF16");
  if (resid_mode != SDM_RESID_SHARED && resid_mode != SDM_RESID_ADDITIVE)
    return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan_chunked: resid_mode must be SDM_RESID_SHARED or SDM_RESID_ADDITIVE");
  if (!aligned(state, 4) || !aligned(y, 4) || (dev_err && !aligned(dev_err, 4)))
    return set_error(SDM_ERR_ALIGN, "sdm_scan_chunked: 4-byte alignment needed");
  if (B == 0 || T == 0 || H == 0) return SDM_OK;
  const size_t need = sdm_scan_chunked_workspace_size(B, T, H, W, R);
  if (!workspace || workspace_bytes < need)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan_chunked: workspace of %zu bytes needed", need);
  if (!aligned(workspace, 16)) return set_error(SDM_ERR_ALIGN, "sdm_scan_chunked: workspace must be 16-byte aligned");

  ChunkArgs args;
  args.state = state;
  args.v = v;
  args.alpha = alpha;
  args.beta = beta;
  args.idx_w = idx_w;
  args.idx_r = idx_r;
  args.w_w = w_w;
  args.w_r = w_r;
  args.y = y;
  args.ws = static_cast<unsigned char *>(workspace);
  args.err = dev_err;
  args.T = T;
  args.H = H;
  args.N = N;
  args.d_v = d_v;
  args.W = W;
  args.R = R;
  args.additive = resid_mode == SDM_RESID_ADDITIVE;
  args.v_bf16 = v_dtype == SDM_DTYPE_BF16;
  args.nchunks = (T + kCC - 1) / kCC;
  args.tiles = (d_v + 31) / 32;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long units = static_cast<long>(B) * H * args.nchunks;
  if (cudaFuncSetAttribute(chunk_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kPrepSmemC)) != cudaSuccess)
    return check_launch("sdm_scan_chunked: set shared memory");
  chunk_prep_kernel<<<static_cast<unsigned>(units), kPrepThreads, kPrepSmemC, st>>>(args);
  const int rc = check_launch("sdm_scan_chunked: preparation kernel");
  if (rc != SDM_OK) return rc;
  const size_t smem = kXUnit + 2 * kCC * kRS * sizeof(float);
  if (cudaFuncSetAttribute(chunk_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return check_launch("sdm_scan_chunked: set shared memory");
  const long blocks = static_cast<long>(B) * H * args.tiles;
  chunk_chain_kernel<<<static_cast<unsigned>(blocks), kChainThreadsC, smem, st>>>(args);
  return check_launch("sdm_scan_chunked: chain kernel");
}
