// sse_chunk.cu - the SSE scan as a prefill: the visits of every partition
// grouped into one time-ordered subsequence (varlen), each subsequence run in
// chunkwise GLA form on the tcgen05 tensor cores, the visits' partial reads
// summed per token (SSE deck, "Varlen groups tokens while preserving causal
// order"; "One gate controls both writes and reads", Eqs. 9-14; "A memory
// decays only when its partition is visited").
//
// Along the subsequence of a partition (every token for the shared one), with
// gate g_i (e^p of the router softmax; 1 for the shared partition) and row
// weights kk_i = softmax of the key logits, the recurrence is
//   S_i = diag(alpha_i) S_{i-1} + g_i kk_i^T v_i,      o_i = g_i q_i S_i.
// Within a chunk of C = 64 visits, every decay factor a product of alphas
// over a range of the chunk's visits:
//   O    = Qt S0 + A V,          Qt_i = g_i q_i * prod_{t<=i} alpha_t
//   A_ij = g_i g_j sum_r q_ir kk_jr prod_{t=j+1..i} alpha_tr       (j <= i)
//   S_C  = diag(gamma) S0 + Kh^T V,   Kh_j = g_j kk_j * prod_{t>j} alpha_t,
//   gamma = prod_t alpha_t.
// A is formed from blocks of 16 visits: within a block by running products,
// across blocks with the block boundaries as reference points (product in the
// later block up to i, whole blocks between, product in the earlier block
// after j), so no factor is ever a quotient and nothing over- or underflows
// into a wrong value.
//
// Launches after the routing prepass of sse_scan.cu:
//   group    one CTA per (batch, head): stable counting sort of the visits by
//            partition; per partition its visit list and its range of units
//            (one unit = one chunk of one partition)
//   prep     every unit in parallel on the CUDA cores: A, Qt, Kh, gamma and
//            the gathered V, stored as ready-made tcgen05 operand tiles
//   chain    one CTA per (batch, head, partition), the shared partitions
//            first (the longest chains): S^T (d x c, fp32) in the registers
//            of 16 worker warps; a producer lane issues the bulk copies and
//            the MMAs  D = V^T Kh  and  O^T = V^T A^T + S0^T Qt^T;  the
//            workers fold S^T <- gamma S^T + D and stage O^T per visit
//   combine  y[token] = its staged visits summed in a fixed order (routed
//            ranks, then the shared partition)
// Operands that are not exact in bf16 (state, Qt, A, Kh) are split into bf16
// hi + lo; q and v are bf16 inputs and enter as they are.
#include <climits>

#include "common.cuh"
#include "sse_group.cuh"
#include "umma.cuh"

namespace sdm {
namespace {

using namespace umma;

constexpr int kC = 64;      // visits per chunk
constexpr int kCh = 128;    // c: rows of a partition (key width)
constexpr int kD = 128;     // d: value width (the MMA M)
constexpr int kMaxTopk = ssegrp::kMaxTopk;
constexpr int kMaxN = ssegrp::kMaxN;
constexpr uint32_t kWaitLimit = 1u << 20;  // polls (about 0.1 s) before an mbarrier wait gives up
constexpr uint32_t kHintedWaitLimit = 1u << 17;  // polls of up to 1 us each (the workers' suspending waits)
constexpr uint32_t kSpinWaitLimit = 1u << 24;    // non-blocking polls (the producer's busy waits)

// ---- one unit in the workspace (bytes)
constexpr uint32_t kXQ = 0;       // Qt hi, lo   [64 i][128 r] K-major, 16 KB each
constexpr uint32_t kXA = 32768;   // A hi, lo    [64 i][64 j]  K-major, 8 KB each
constexpr uint32_t kXV = 49152;   // V           [64 j][128 d] bf16 (read MN-major as V^T)
constexpr uint32_t kXK = 65536;   // Kh hi, lo   [64 j][128 r] (read MN-major as the B of V^T Kh)
constexpr uint32_t kXG = 98304;   // gamma       fp32 [128]
constexpr uint32_t kXR = 98816;   // staging row of each visit, int32 [64] (-1: padding)
constexpr uint32_t kXUnit = 99072;
constexpr uint32_t kXQBytes = kXA - kXQ;    // the S-dependent operand (one bulk copy)
constexpr uint32_t kXYBytes = kXG - kXA;    // A, V, Kh (one bulk copy)
constexpr uint32_t kXZBytes = kXUnit - kXG; // gamma and rows (one bulk copy, double-buffered)
static_assert(kXUnit % 16 == 0 && kXYBytes % 16 == 0 && kXZBytes % 16 == 0, "bulk copies need 16-byte multiples");

// ---- group table of one (batch, head): sse_group.cuh
using ssegrp::group_words;
using ssegrp::kGCnt;
using ssegrp::kGFirst;
using ssegrp::kGHdr;
using ssegrp::kGOff;
using ssegrp::units_max;

// ===========================================================================
// group: per (batch, head), the visits sorted by partition, time order kept.
// ===========================================================================
constexpr int kGroupThreads = 1024;

__global__ void __launch_bounds__(kGroupThreads) sse_group_kernel(const uint32_t *__restrict__ rec, int T, int H, int N,
                                                                  int topk, int rw, uint32_t *__restrict__ grp,
                                                                  long gwords) {
  __shared__ int cnt[kMaxN];
  __shared__ int base[kMaxN];
  __shared__ int wcnt[kGroupThreads / 32][kMaxN];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const long bh = blockIdx.x;
  const long b = bh / H;
  const int h = static_cast<int>(bh % H);
  uint32_t *g = grp + bh * gwords;
  if (tid < kMaxN) cnt[tid] = 0;
  __syncthreads();
  for (int t = tid; t < T; t += kGroupThreads) {
    const uint32_t *r = rec + ((b * T + t) * H + h) * rw;
#pragma unroll
    for (int s = 0; s < kMaxTopk; ++s)
      if (s < topk) atomicAdd(&cnt[r[s]], 1);
  }
  __syncthreads();
  if (tid == 0) {
    int off = 0, u = (T + kC - 1) / kC;
    for (int p = 0; p < N; ++p) {
      g[kGFirst + p] = static_cast<uint32_t>(u);
      g[kGCnt + p] = static_cast<uint32_t>(cnt[p]);
      g[kGOff + p] = static_cast<uint32_t>(off);
      base[p] = off;
      off += cnt[p];
      u += (cnt[p] + kC - 1) / kC;
    }
    g[kGFirst + N] = static_cast<uint32_t>(u);
  }
  __syncthreads();
  uint32_t *ent = g + kGHdr;
  for (int t0 = 0; t0 < T; t0 += kGroupThreads) {
    const int t = t0 + tid;
    int ids[kMaxTopk];
    unsigned masks[kMaxTopk];
    const uint32_t *r = rec + ((b * T + (t < T ? t : 0)) * H + h) * rw;
#pragma unroll
    for (int s = 0; s < kMaxTopk; ++s) {
      ids[s] = (t < T && s < topk) ? static_cast<int>(r[s]) : -1;
      masks[s] = 0u;
    }
    // per partition: which lanes of the warp visit it
    for (int p = 0; p < N; ++p) {
      bool mine = false;
#pragma unroll
      for (int s = 0; s < kMaxTopk; ++s) mine |= ids[s] == p;
      const unsigned m = __ballot_sync(kFull, mine);
#pragma unroll
      for (int s = 0; s < kMaxTopk; ++s)
        if (ids[s] == p) masks[s] = m;
      if (lane == 0) wcnt[warp][p] = __popc(m);
    }
    __syncthreads();
    if (tid < N) {  // exclusive scan over the warps, on top of the partition's running base
      int run = base[tid];
      for (int w = 0; w < kGroupThreads / 32; ++w) {
        const int x = wcnt[w][tid];
        wcnt[w][tid] = run;
        run += x;
      }
      base[tid] = run;
    }
    __syncthreads();
#pragma unroll
    for (int s = 0; s < kMaxTopk; ++s) {
      if (ids[s] >= 0) {
        const int pos = wcnt[warp][ids[s]] + __popc(masks[s] & ((1u << lane) - 1u));
        ent[pos] = (static_cast<uint32_t>(t) << 4) | static_cast<uint32_t>(s);
      }
    }
    __syncthreads();
  }
}

// ===========================================================================
// prep: the state-independent operands of every unit (CUDA cores).
// ===========================================================================
struct PrepArgs {
  const uint16_t *q, *v;
  const float *klog, *alpha;
  const uint32_t *rec, *grp;
  unsigned char *units;
  int T, H, N, topk, rw, umax;
  long gwords, total;  // total = B * H * umax
  int32_t *err;
};

constexpr int kPThreads = 256;
constexpr int kLdA = 132;  // fp32 row stride of the alpha / kk arrays (rows 4 banks apart)
constexpr int kLdF = 68;   // fp32 row stride of A
// shared memory (bytes)
constexpr uint32_t kPq = 0;                          // q bf16 [64][128]
constexpr uint32_t kPal = kPq + kC * kCh * 2;        // alpha, then q * (product in the block up to i)
constexpr uint32_t kPkk = kPal + kC * kLdA * 4;      // key logits, then kk, then kk * (product in the block after j)
constexpr uint32_t kPAf = kPkk + kC * kLdA * 4;      // A fp32 [64][kLdF]
constexpr uint32_t kPPb = kPAf + kC * kLdF * 4;      // block products, prefix, suffix [3][4][128]
constexpr uint32_t kPRow = kPPb + 3 * 4 * kCh * 4;   // per visit: token-head, slot, gate
constexpr uint32_t kPInfo = kPRow + 3 * kC * 4;      // the unit: partition, first position, visits, list offset
constexpr uint32_t kPrepSmem = kPInfo + 16;
static_assert(2 * (kPrepSmem + 1024) <= 228 * 1024, "two preparation CTAs per SM");

__global__ void __launch_bounds__(kPThreads, 2) sse_prep_kernel(const PrepArgs a) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint16_t *sq = reinterpret_cast<uint16_t *>(sm + kPq);
  float *sal = reinterpret_cast<float *>(sm + kPal);
  float *skk = reinterpret_cast<float *>(sm + kPkk);
  float *sA = reinterpret_cast<float *>(sm + kPAf);
  float *sP = reinterpret_cast<float *>(sm + kPPb), *sPre = sP + 4 * kCh, *sSuf = sP + 8 * kCh;
  int *rtok = reinterpret_cast<int *>(sm + kPRow), *rslot = rtok + kC;
  float *rg = reinterpret_cast<float *>(rslot + kC);
  int *info = reinterpret_cast<int *>(sm + kPInfo);
  const int T = a.T, H = a.H, N = a.N, topk = a.topk;
  const int nS = (T + kC - 1) / kC;

  for (long ug = blockIdx.x; ug < a.total; ug += gridDim.x) {
    const long bh = ug / a.umax;
    const int uu = static_cast<int>(ug - bh * a.umax);
    const uint32_t *g = a.grp + bh * a.gwords;
    if (uu >= static_cast<int>(g[kGFirst + N])) continue;  // beyond this (batch, head)'s units: uniform
    if (warp == 0) {
      int p = N, pos0 = uu * kC, cnt = T, off = 0;
      if (uu >= nS) {  // routed: the last partition whose first unit is <= uu
        const bool c0 = lane < N && static_cast<int>(g[kGFirst + lane]) <= uu;
        const bool c1 = lane + 32 < N && static_cast<int>(g[kGFirst + lane + 32]) <= uu;
        p = __popc(__ballot_sync(kFull, c0)) + __popc(__ballot_sync(kFull, c1)) - 1;
        pos0 = (uu - static_cast<int>(g[kGFirst + p])) * kC;
        cnt = static_cast<int>(g[kGCnt + p]);
        off = static_cast<int>(g[kGOff + p]);
      }
      if (lane == 0) {
        info[0] = p;
        info[1] = pos0;
        info[2] = cnt;
        info[3] = off;
      }
    }
    __syncthreads();
    const long b = bh / H;
    const int h = static_cast<int>(bh % H);
    if (tid < kC) {
      const int p = info[0], pos = info[1] + tid;
      int tk = -1, slot = topk;
      float gate = 0.f;
      if (pos < info[2]) {
        int t = pos, r = topk;
        if (p < N) {
          const uint32_t e = g[kGHdr + info[3] + pos];
          t = static_cast<int>(e >> 4);
          r = static_cast<int>(e & 15u);
        }
        const long tl = (b * T + t) * H + h;
        const uint32_t *rc = a.rec + tl * a.rw;
        gate = r < topk ? __uint_as_float(rc[topk + r]) : 1.f;
        tk = static_cast<int>(tl);
        slot = r;
      }
      rtok[tid] = tk;
      rslot[tid] = slot;
      rg[tid] = gate;
    }
    __syncthreads();
    unsigned char *unit = a.units + ug * kXUnit;

    // ---- q, key logits, alpha rows (padding: q = 0, logits 0, alpha = 1)
    for (int id = tid; id < kC * 16; id += kPThreads) {  // q: 16 pieces per row
      const int i = id >> 4, k = id & 15;
      const long tk = rtok[i];
      uint16_t *dst = sq + i * kCh + 8 * k;
      if (tk >= 0) cp_async<16>(dst, a.q + tk * kCh + 8 * k);
      else *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    for (int id = tid; id < kC * 32; id += kPThreads) {  // key logits and alpha: 32 pieces per row each
      const int i = id >> 5, k = id & 31;
      const long tk = rtok[i];
      float *dk = skk + i * kLdA + 4 * k, *da = sal + i * kLdA + 4 * k;
      if (tk >= 0) {
        cp_async<16>(dk, a.klog + tk * kCh + 4 * k);
        cp_async<16>(da, a.alpha + tk * kCh + 4 * k);
      } else {
        *reinterpret_cast<uint4 *>(dk) = make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<float4 *>(da) = make_float4(1.f, 1.f, 1.f, 1.f);
      }
    }
    cp_async_commit();
    // V tile (8 values of d per 16 bytes, the K-tile layout) and the staging
    // rows, straight to the workspace
    for (int id = tid; id < kC * 16; id += kPThreads) {
      const int j = id >> 4, d8 = id & 15;
      const long tk = rtok[j];
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (tk >= 0) x = __ldg(reinterpret_cast<const uint4 *>(a.v + tk * kD + 8 * d8));
      *reinterpret_cast<uint4 *>(unit + kXV + kmajor_off(j, 8 * d8, kD)) = x;
    }
    if (tid < kC) reinterpret_cast<int *>(unit + kXR)[tid] = rtok[tid] >= 0 ? rtok[tid] * (topk + 1) + rslot[tid] : -1;
    cp_async_wait<0>();
    __syncthreads();
    // kk = softmax of each visit's key logits (warp: 8 rows, lane: 4 channels)
#pragma unroll 2
    for (int e = 0; e < kC / 8; ++e) {
      const int i = (kC / 8) * warp + e;
      float4 *x = reinterpret_cast<float4 *>(skk + i * kLdA) + lane;
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
        v.x *= zi;
        v.y *= zi;
        v.z *= zi;
        v.w *= zi;
      } else {
        v = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      *x = v;
    }
    __syncthreads();

    // ---- A, diagonal blocks: thread (block J, rows i and i + 8, channel
    // slice cs) walks j from row i + 8 down to the block start with qf_r =
    // q_ir prod_{t=j+1..i} alpha_tr for both rows, so every key and decay row
    // it loads serves two rows; its channels are the float4 groups cs, cs+8,
    // cs+16, cs+24 (the 8 slices of a row read distinct banks)
    {
      const int J = tid >> 6, il = (tid >> 3) & 7, cs = tid & 7;
      const int ia = 16 * J + il, ib = ia + 8;
      float qa[16], qb[16];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const uint2 wa = *reinterpret_cast<const uint2 *>(sq + ia * kCh + 4 * (cs + 8 * m));
        const uint2 wb = *reinterpret_cast<const uint2 *>(sq + ib * kCh + 4 * (cs + 8 * m));
        qa[4 * m] = bf16_to_f32(static_cast<uint16_t>(wa.x & 0xffffu));
        qa[4 * m + 1] = bf16_to_f32(static_cast<uint16_t>(wa.x >> 16));
        qa[4 * m + 2] = bf16_to_f32(static_cast<uint16_t>(wa.y & 0xffffu));
        qa[4 * m + 3] = bf16_to_f32(static_cast<uint16_t>(wa.y >> 16));
        qb[4 * m] = bf16_to_f32(static_cast<uint16_t>(wb.x & 0xffffu));
        qb[4 * m + 1] = bf16_to_f32(static_cast<uint16_t>(wb.x >> 16));
        qb[4 * m + 2] = bf16_to_f32(static_cast<uint16_t>(wb.y & 0xffffu));
        qb[4 * m + 3] = bf16_to_f32(static_cast<uint16_t>(wb.y >> 16));
      }
      for (int jl = (il | 3) + 8; jl >= 0; --jl) {  // warp-uniform trip count (a warp holds 4 consecutive il)
        const bool acta = jl <= il, actb = jl <= il + 8;
        const int j = 16 * J + jl;
        const float *kr = skk + j * kLdA;
        float acc_a = 0.f, acc_b = 0.f;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 kv = *reinterpret_cast<const float4 *>(kr + 4 * (cs + 8 * m));
          acc_a = fmaf(qa[4 * m], kv.x, acc_a);
          acc_a = fmaf(qa[4 * m + 1], kv.y, acc_a);
          acc_a = fmaf(qa[4 * m + 2], kv.z, acc_a);
          acc_a = fmaf(qa[4 * m + 3], kv.w, acc_a);
          acc_b = fmaf(qb[4 * m], kv.x, acc_b);
          acc_b = fmaf(qb[4 * m + 1], kv.y, acc_b);
          acc_b = fmaf(qb[4 * m + 2], kv.z, acc_b);
          acc_b = fmaf(qb[4 * m + 3], kv.w, acc_b);
        }
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) {
          acc_a += __shfl_xor_sync(kFull, acc_a, o);
          acc_b += __shfl_xor_sync(kFull, acc_b, o);
        }
        if (cs == 0) {
          if (acta) sA[ia * kLdF + j] = acc_a;
          if (actb) sA[ib * kLdF + j] = acc_b;
        }
        const float *ar = sal + j * kLdA;  // toward j - 1: include alpha_j
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float4 av = *reinterpret_cast<const float4 *>(ar + 4 * (cs + 8 * m));
          if (acta) {
            qa[4 * m] *= av.x;
            qa[4 * m + 1] *= av.y;
            qa[4 * m + 2] *= av.z;
            qa[4 * m + 3] *= av.w;
          }
          if (actb) {
            qb[4 * m] *= av.x;
            qb[4 * m + 1] *= av.y;
            qb[4 * m + 2] *= av.z;
            qb[4 * m + 3] *= av.w;
          }
        }
      }
    }
    __syncthreads();

    // ---- block products; then per channel and block the running products:
    // alpha -> q * F (F = product in the block up to i), kk -> kk * R (R =
    // product in the block after j)
    {  // thread (column r, blocks 2hb and 2hb+1) is the only one touching that column of those blocks
      const int r = tid & 127, hb = tid >> 7;
#pragma unroll
      for (int Jh = 0; Jh < 2; ++Jh) {
        const int J = 2 * hb + Jh;
        float al[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) al[k] = sal[(16 * J + k) * kLdA + r];
        float P = 1.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) P *= al[k];
        sP[J * kCh + r] = P;
        float F = 1.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const int i = 16 * J + k;
          F *= al[k];
          sal[i * kLdA + r] = bf16_to_f32(sq[i * kCh + r]) * F;
        }
        float R = 1.f;
#pragma unroll
        for (int k = 15; k >= 0; --k) {
          const int j = 16 * J + k;
          skk[j * kLdA + r] *= R;
          R *= al[k];
        }
      }
    }
    __syncthreads();
    {
      const int r = tid & 127, hb = tid >> 7;
      float pb[4];
#pragma unroll
      for (int K = 0; K < 4; ++K) pb[K] = sP[K * kCh + r];
      if (hb == 0) reinterpret_cast<float *>(unit + kXG)[r] = ((pb[0] * pb[1]) * pb[2]) * pb[3];
#pragma unroll
      for (int Jh = 0; Jh < 2; ++Jh) {
        const int J = 2 * hb + Jh;
        float pre = 1.f, suf = 1.f;
#pragma unroll
        for (int K = 0; K < 4; ++K) {
          if (K < J) pre *= pb[K];
          if (K > J) suf *= pb[K];
        }
        sPre[J * kCh + r] = pre;
        sSuf[J * kCh + r] = suf;
      }
    }
    __syncthreads();

    // ---- A, blocks below the diagonal: A_ij = sum_r qF_ir mid_r kkR_jr with
    // mid = the whole blocks between J and I.  Thread pair (tid, tid^1): a
    // 4 x 4 tile, rows 16I + rq + 4e, columns j0..j0+3, the two threads taking
    // the float4 channel groups 8m + 4ch + u (ch = 0, 1), which puts the 8
    // lanes of a quarter-warp (4 row offsets x 2 channel halves) on distinct
    // banks
    if (tid < 192) {
      const int ch = tid & 1, tt = tid >> 1;
      const int rq = tt & 3, gq = tt >> 2;  // gq: (I, J, jq) as below, 24 of them
      int I, J, jq;
      if (gq < 4) {
        I = 1; J = 0; jq = gq;
      } else if (gq < 12) {
        I = 2; J = (gq - 4) >> 2; jq = (gq - 4) & 3;
      } else {
        I = 3; J = (gq - 12) >> 2; jq = (gq - 12) & 3;
      }
      const int i0 = 16 * I + rq, j0 = 16 * J + 4 * jq;
      const int gap = I - J;  // warp-uniform
      const float *m0 = sP + (J + 1) * kCh, *m1 = sP + (J + 2) * kCh;
      float acc[4][4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int f = 0; f < 4; ++f) acc[e][f] = 0.f;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int k4 = 8 * m + 4 * ch + u;
          float4 mid = make_float4(1.f, 1.f, 1.f, 1.f);
          if (gap >= 2) mid = *reinterpret_cast<const float4 *>(m0 + 4 * k4);
          if (gap == 3) {
            const float4 m2 = *reinterpret_cast<const float4 *>(m1 + 4 * k4);
            mid.x *= m2.x;
            mid.y *= m2.y;
            mid.z *= m2.z;
            mid.w *= m2.w;
          }
          float4 kv[4];
#pragma unroll
          for (int f = 0; f < 4; ++f) {
            kv[f] = *reinterpret_cast<const float4 *>(skk + (j0 + f) * kLdA + 4 * k4);
            if (gap >= 2) {
              kv[f].x *= mid.x;
              kv[f].y *= mid.y;
              kv[f].z *= mid.z;
              kv[f].w *= mid.w;
            }
          }
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float4 qv = *reinterpret_cast<const float4 *>(sal + (i0 + 4 * e) * kLdA + 4 * k4);
#pragma unroll
            for (int f = 0; f < 4; ++f) {
              acc[e][f] = fmaf(qv.x, kv[f].x, acc[e][f]);
              acc[e][f] = fmaf(qv.y, kv[f].y, acc[e][f]);
              acc[e][f] = fmaf(qv.z, kv[f].z, acc[e][f]);
              acc[e][f] = fmaf(qv.w, kv[f].w, acc[e][f]);
            }
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e)
#pragma unroll
        for (int f = 0; f < 4; ++f) acc[e][f] += __shfl_xor_sync(0xffffffffu, acc[e][f], 1);
      if (ch == 0) {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          *reinterpret_cast<float4 *>(sA + (i0 + 4 * e) * kLdF + j0) =
              make_float4(acc[e][0], acc[e][1], acc[e][2], acc[e][3]);
      }
    }
    __syncthreads();

    // ---- operand tiles: A (lower triangle, gated), Qt, Kh as bf16 hi/lo
    for (int id = tid; id < kC * 8; id += kPThreads) {
      const int i = id >> 3, j0 = (id & 7) * 8;
      const float gi = rg[i];
      float x[8];
#pragma unroll
      for (int h4 = 0; h4 < 8; h4 += 4) {  // kLdF and j0 are multiples of 4; rg is 16-byte aligned
        const float4 a4 = *reinterpret_cast<const float4 *>(sA + i * kLdF + j0 + h4);
        const float4 g4 = *reinterpret_cast<const float4 *>(rg + j0 + h4);
        const float av[4] = {a4.x, a4.y, a4.z, a4.w}, gv[4] = {g4.x, g4.y, g4.z, g4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) x[h4 + e] = j0 + h4 + e <= i ? av[e] * gi * gv[e] : 0.f;
      }
      store_split8(unit + kXA, unit + kXA + 8192, kmajor_off(i, j0, kC), x);
    }
    {  // thread: block J, channels r0..r0+7, rows 16J + il + 4m (m < 4), so the
       // block's prefix and suffix products are loaded once
      const int r0 = (tid & 15) * 8, il = (tid >> 4) & 3, J = tid >> 6;
      float pr[8], sf[8];
#pragma unroll
      for (int h4 = 0; h4 < 8; h4 += 4) {  // 16-byte rows: kLdA and r0 are multiples of 4
        const float4 p4 = *reinterpret_cast<const float4 *>(sPre + J * kCh + r0 + h4);
        const float4 s4 = *reinterpret_cast<const float4 *>(sSuf + J * kCh + r0 + h4);
        pr[h4] = p4.x; pr[h4 + 1] = p4.y; pr[h4 + 2] = p4.z; pr[h4 + 3] = p4.w;
        sf[h4] = s4.x; sf[h4 + 1] = s4.y; sf[h4 + 2] = s4.z; sf[h4 + 3] = s4.w;
      }
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const int i = 16 * J + il + 4 * m;
        const float gi = rg[i];
        float x[8], y[8];
#pragma unroll
        for (int h4 = 0; h4 < 8; h4 += 4) {
          const float4 qf = *reinterpret_cast<const float4 *>(sal + i * kLdA + r0 + h4);
          const float4 kr = *reinterpret_cast<const float4 *>(skk + i * kLdA + r0 + h4);
          x[h4] = gi * qf.x * pr[h4];
          x[h4 + 1] = gi * qf.y * pr[h4 + 1];
          x[h4 + 2] = gi * qf.z * pr[h4 + 2];
          x[h4 + 3] = gi * qf.w * pr[h4 + 3];
          y[h4] = gi * kr.x * sf[h4];
          y[h4 + 1] = gi * kr.y * sf[h4 + 1];
          y[h4 + 2] = gi * kr.z * sf[h4 + 2];
          y[h4 + 3] = gi * kr.w * sf[h4 + 3];
        }
        store_split8(unit + kXQ, unit + kXQ + 16384, kmajor_off(i, r0, kCh), x);
        store_split8(unit + kXK, unit + kXK + 16384, kmajor_off(i, r0, kCh), y);
      }
    }
    __syncthreads();  // shared memory is reused by the next unit
  }
}

// ===========================================================================
// chain: the units of one partition in order.
//
// Warps 0-15 (workers): warp w owns tensor-memory lanes 32*(w%4) .. +31
// (value columns d) and quarter w/4 of the rows r (S) and of the unit's
// visits (O).  Warp 16 (producer, one lane) issues the bulk copies and the
// MMAs.  Per unit c (buffers b = c % 2 for Qt, gamma/rows, D and O; one
// buffer for A/V/Kh):
//   producer  D[b] = V^T Kh and O[b]^T = V^T A^T (state-independent), then,
//             once the workers have published S0: O[b]^T += S0^T Qt^T; then
//             the copies: A/V/Kh of unit c+1 as soon as D[b] and V^T A^T are
//             done, Qt of unit c+2 once this unit's MMAs are
//   workers   S^T <- gamma S^T + D[b] as soon as D[b] is done, published as
//             bf16 hi/lo for unit c+1 once this unit's MMAs no longer read
//             S0; O[b]^T staged per visit
// Qt is double-buffered so that the next unit's copy is long done when its
// state-dependent MMAs can start: the per-unit cycle is the tensor pipe's
// work plus the state's publish, not a copy's latency.
// ===========================================================================
struct ChainArgs {
  float *state;
  const unsigned char *units;
  const uint32_t *grp;
  float *stage;
  int T, N, umax;
  long bh_count, gwords;
  int drop_signal;  // test hook: the first unit's MMA-done signal is never sent (bounded waits run out)
  int32_t *err;
};

constexpr int kWorkers = 512;
constexpr int kChainThreads = kWorkers + 32;
// tensor-memory columns (fp32): D[2] 128 each, O[2] 64 each
constexpr uint32_t kColD = 0, kColO = 256, kChainTmemCols = 512;
// shared memory (bytes)
constexpr uint32_t kSS = 0;                      // S^T hi, lo [128 d][128 r]   2 x 32 KB
constexpr uint32_t kSX = 65536;                  // Qt hi, lo                   2 x 32 KB (two units)
constexpr uint32_t kSY = kSX + 2 * kXQBytes;     // A hi, lo, V, Kh hi, lo      64 KB
constexpr uint32_t kSZ = kSY + kXYBytes;         // gamma + rows                2 x 768 B
constexpr uint32_t kSBar = kSZ + 2 * kXZBytes;
constexpr int kNBar = 13;
constexpr uint32_t kChainSmem = kSBar + kNBar * 8 + 16;
static_assert(kChainSmem <= 227 * 1024, "chain shared memory");

__global__ void __maxnreg__(96) sse_chain_kernel(const ChainArgs a) {
  extern __shared__ __align__(1024) unsigned char sm[];
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  long bh;
  int p;
  if (blockIdx.x < a.bh_count) {  // the shared partitions first: the longest chains
    bh = blockIdx.x;
    p = a.N;
  } else {
    const long k = blockIdx.x - a.bh_count;
    bh = k / a.N;
    p = static_cast<int>(k - bh * a.N);
  }
  const uint32_t *g = a.grp + bh * a.gwords;
  const int u0 = p == a.N ? 0 : static_cast<int>(g[kGFirst + p]);
  const int n = p == a.N ? (a.T + kC - 1) / kC : static_cast<int>(g[kGFirst + p + 1]) - u0;
  if (n <= 0) return;  // a partition no token visits keeps its state (CTA-uniform)
  const unsigned char *ub = a.units + (bh * a.umax + u0) * static_cast<long>(kXUnit);
  float *gS = a.state + (bh * (a.N + 1) + p) * static_cast<long>(kCh * kD);

  unsigned char *sSh = sm + kSS, *sSl = sm + kSS + 32768;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + kSBar);
  // barriers: 0-1 Qt loaded [b], 2 A/V/Kh loaded, 3-4 gamma/rows loaded [b], 5 MMAs of the unit done,
  // 6 S published (workers), 7-8 D[b] and O[b] read (workers), 9 drain, 10-11 D[b] done,
  // 12 A/V/Kh read (D and V^T A^T done)
  enum { kBarX = 0, kBarY = 2, kBarZ = 3, kBarMma = 5, kBarS = 6, kBarFree = 7, kBarDrain = 9, kBarD = 10,
         kBarYFree = 12 };
  auto bar = [&](int i) { return smem_addr(bars + i); };
  uint32_t *holder = reinterpret_cast<uint32_t *>(sm + kSBar + kNBar * 8);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + kSBar + kNBar * 8 + 4);

  if (tid == 0) {
    for (int i = 0; i < kNBar; ++i)
      mbar_init(bar(i), (i == kBarS || i == kBarFree || i == kBarFree + 1) ? kWorkers : 1);
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
    auto wwait = [&](uint32_t mb, uint32_t parity) -> bool {
      return __all_sync(kFull, mbar_wait_hinted(mb, parity, kHintedWaitLimit, abort_flag)) != 0;
    };
    float S[32];  // S^T[row][32*qtr + j] = S[32*qtr + j][row]
#pragma unroll
    for (int j = 0; j < 32; ++j) S[j] = gS[static_cast<long>(32 * qtr + j) * kD + row];
    auto publish = [&]() {
#pragma unroll
      for (int g8 = 0; g8 < 4; ++g8) store_split8(sSh, sSl, kmajor_off(row, 32 * qtr + 8 * g8, kCh), S + 8 * g8);
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarS));
    };
    publish();
    for (int c = 0; c < n; ++c) {
      const int b = c & 1;
      const bool last = c + 1 == n;
      if (!wwait(bar(kBarZ + b), static_cast<uint32_t>((c >> 1) & 1))) break;
      if (!wwait(bar(kBarD + b), static_cast<uint32_t>((c >> 1) & 1))) break;
      const unsigned char *z = sm + kSZ + b * kXZBytes;
      const float *gam = reinterpret_cast<const float *>(z) + 32 * qtr;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        float x[16];
        tmem_ld16(lanes + kColD + 128 * b + 32 * qtr + 16 * hh, x);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) S[16 * hh + e] = fmaf(gam[16 * hh + e], S[16 * hh + e], x[e]);
      }
      // the unit's MMAs done: the published S0 is no longer read and O[b] is complete
      if (!wwait(bar(kBarMma), static_cast<uint32_t>(c & 1))) break;
      if (!last) publish();
      {
        const int *rows = reinterpret_cast<const int *>(z + (kXR - kXG)) + 16 * qtr;
        float o[16];
        tmem_ld16(lanes + kColO + 64 * b + 16 * qtr, o);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int rr = rows[e];
          if (rr >= 0) a.stage[static_cast<long>(rr) * kD + row] = o[e];
        }
      }
      tc_fence_before();
      mbar_arrive(bar(kBarFree + b));
      if (last) {
#pragma unroll
        for (int j = 0; j < 32; ++j) gS[static_cast<long>(32 * qtr + j) * kD + row] = S[j];
      }
    }
  } else if (tid == kWorkers) {
    // ------------------------------------------------------------ producer
    const uint32_t sh = smem_addr(sSh), sl = smem_addr(sSl);
    const uint32_t xq = smem_addr(sm + kSX);
    const uint64_t dSh = smem_desc(sh, 128, kCh * 16), dSl = smem_desc(sl, 128, kCh * 16);
    const uint32_t idO = idesc_bf16_f32(128, kC), idOv = idO | (1u << 15);
    const uint32_t idD = idesc_bf16_f32(128, kCh) | (1u << 15) | (1u << 16);
    int x_issued[2] = {0, 0}, x_done[2] = {0, 0}, y_issued = 0, y_done = 0, z_issued[2] = {0, 0};
    auto load_x = [&](int c) {  // Qt of unit c into buffer c % 2
      const int b = c & 1;
      fence_async_smem();
      mbar_expect_tx(bar(kBarX + b), kXQBytes);
      bulk_g2s(xq + b * kXQBytes, ub + static_cast<long>(c) * kXUnit + kXQ, kXQBytes, bar(kBarX + b));
      ++x_issued[b];
    };
    auto load_y = [&](int c) {  // A, V, Kh of unit c
      fence_async_smem();
      mbar_expect_tx(bar(kBarY), kXYBytes);
      bulk_g2s(smem_addr(sm + kSY), ub + static_cast<long>(c) * kXUnit + kXA, kXYBytes, bar(kBarY));
      ++y_issued;
    };
    auto load_z = [&](int c) {  // gamma and rows of unit c into buffer c % 2
      const int b = c & 1;
      fence_async_smem();
      mbar_expect_tx(bar(kBarZ + b), kXZBytes);
      bulk_g2s(smem_addr(sm + kSZ + b * kXZBytes), ub + static_cast<long>(c) * kXUnit + kXG, kXZBytes, bar(kBarZ + b));
      ++z_issued[b];
    };
    auto prefetch = [&](int c) {
      const unsigned char *pf = ub + static_cast<long>(c) * kXUnit;
      prefetch_l2(pf, kXV);
      prefetch_l2(pf + kXV, kXUnit - kXV);
    };
    // a busy wait (one thread), so the producer issues the moment an operand is ready
    auto wait = [&](int i, uint32_t parity) { return mbar_wait_spin(bar(i), parity, kSpinWaitLimit, abort_flag); };
    if (n > 1) prefetch(1);
    load_x(0);
    if (n > 1) load_x(1);
    load_y(0);
    load_z(0);
    const uint32_t ya = smem_addr(sm + kSY);
    const uint32_t yv = ya + (kXV - kXA), yk = ya + (kXK - kXA);
    const uint64_t dAh = smem_desc(ya, 128, kC * 16), dAl = smem_desc(ya + 8192, 128, kC * 16);
    // V^T (A operand) and Kh (B operand) are MN-major: 8 consecutive d (or
    // r) per 16 bytes, 8-visit groups 2048 bytes apart; a k-step of 16
    // visits is 4096 bytes (256 in the descriptor)
    const uint64_t dV = smem_desc(yv, 2048, 128);
    const uint64_t dKh = smem_desc(yk, 2048, 128), dKl = smem_desc(yk + 16384, 2048, 128);
    bool ok = true;
    for (int c = 0; c < n && ok; ++c) {
      const int b = c & 1;
      if (c + 2 < n) prefetch(c + 2);
      // state-independent MMAs of unit c
      ok = wait(kBarY, static_cast<uint32_t>(c & 1));
      if (ok) ++y_done;
      if (ok && c >= 2) ok = wait(kBarFree + b, static_cast<uint32_t>(((c - 2) >> 1) & 1));  // D[b], O[b] read
      if (!ok) break;
      const uint32_t tD = tmem + kColD + 128 * b, tO = tmem + kColO + 64 * b;
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks) {
        mma_bf16(tD, dV + 256u * ks, dKh + 256u * ks, idD, ks > 0);
        mma_bf16(tD, dV + 256u * ks, dKl + 256u * ks, idD, true);
      }
      mma_commit(bar(kBarD + b));
#pragma unroll
      for (int ks = 0; ks < kC / 16; ++ks) {
        mma_bf16(tO, dV + 256u * ks, dAh + 16u * ks, idOv, ks > 0);
        mma_bf16(tO, dV + 256u * ks, dAl + 16u * ks, idOv, true);
      }
      mma_commit(bar(kBarYFree));
      // the state-dependent part
      ok = wait(kBarX + b, static_cast<uint32_t>((c >> 1) & 1));
      if (ok) ++x_done[b];
      if (ok) ok = wait(kBarS, static_cast<uint32_t>(c & 1));  // S0 of unit c published
      if (!ok) break;
      const uint32_t xb = xq + b * kXQBytes;
      const uint64_t dQh = smem_desc(xb, 128, kCh * 16), dQl = smem_desc(xb + 16384, 128, kCh * 16);
#pragma unroll
      for (int ks = 0; ks < kCh / 16; ++ks) {
        mma_bf16(tO, dSh + 16u * ks, dQh + 16u * ks, idO, true);
        mma_bf16(tO, dSh + 16u * ks, dQl + 16u * ks, idO, true);
        mma_bf16(tO, dSl + 16u * ks, dQh + 16u * ks, idO, true);
      }
      if (!(a.drop_signal && c == 0)) mma_commit(bar(kBarMma));
      if (c + 1 < n) {
        // unit c+1's A/V/Kh once unit c's state-independent MMAs have read
        // theirs; its gamma/rows once the workers are done with unit c-1's
        ok = wait(kBarYFree, static_cast<uint32_t>(c & 1));
        if (ok) load_y(c + 1);
        if (ok && c >= 1) ok = wait(kBarFree + (b ^ 1), static_cast<uint32_t>(((c - 1) >> 1) & 1));
        if (ok) load_z(c + 1);
        // unit c+2's Qt into this buffer once this unit's MMAs have read it
        if (ok && c + 2 < n) {
          ok = wait(kBarMma, static_cast<uint32_t>(c & 1));
          if (ok) load_x(c + 2);
        }
      }
    }
    // every MMA issued has completed before tensor memory is freed (also when
    // a worker's wait ran out after this loop ended)
    mma_commit(bar(kBarDrain));
    mbar_wait(bar(kBarDrain), 0, kWaitLimit);
    // and every bulk copy has landed before the CTA exits (bounded waits; in
    // the normal path they have all been seen complete already)
    if (y_done < y_issued) mbar_wait(bar(kBarY), static_cast<uint32_t>((y_issued - 1) & 1), kWaitLimit);
    for (int bb = 0; bb < 2; ++bb) {
      if (x_done[bb] < x_issued[bb])
        mbar_wait(bar(kBarX + bb), static_cast<uint32_t>((x_issued[bb] - 1) & 1), kWaitLimit);
      if (z_issued[bb] > 0) mbar_wait(bar(kBarZ + bb), static_cast<uint32_t>((z_issued[bb] - 1) & 1), kWaitLimit);
    }
    if (!ok) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (tid == 0 && *abort_flag) report_timeout(a.err);
  if (warp == 0) tmem_dealloc(tmem, kChainTmemCols);
}

// ===========================================================================
// combine: y[token] = the sum of its visits' staged rows
// ===========================================================================
__global__ void __launch_bounds__(256) sse_combine_kernel(const float4 *__restrict__ stage, float4 *__restrict__ y,
                                                          long n4, int slots) {
  constexpr int kD4 = kD / 4;
  for (long e = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n4;
       e += static_cast<long>(gridDim.x) * blockDim.x) {
    const long tok = e / kD4;
    const int c4 = static_cast<int>(e - tok * kD4);
    const float4 *s = stage + tok * slots * kD4 + c4;
    float4 acc = __ldg(s);
    for (int k = 1; k < slots; ++k) {
      const float4 x = __ldg(s + k * kD4);
      acc.x += x.x;
      acc.y += x.y;
      acc.z += x.z;
      acc.w += x.w;
    }
    y[e] = acc;
  }
}

inline size_t round256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

}  // namespace

size_t sse_delta_unit_bytes();  // gdn_chunk.cu
int launch_sse_delta_chunk(float *state, const uint32_t *rec, int rw, const uint32_t *grp, long gwords, int umax,
                           const float *klog, const uint16_t *q, const uint16_t *v, const float *alpha, int B, int T,
                           int H, int N, int topk, unsigned char *units, float *stage, int32_t *err, cudaStream_t st);

// Workspace bytes of the chunked path beyond the routing records: group
// tables, the units (the additive write's or, for the delta write, the KDA
// chunk form's), the staging rows.
size_t sse_chunk_workspace_size(int B, int T, int H, int N, int topk, int write_mode) {
  const size_t bh = static_cast<size_t>(B) * H;
  const size_t unit = write_mode == SSE_WRITE_DELTA ? sse_delta_unit_bytes() : static_cast<size_t>(kXUnit);
  return round256(bh * group_words(T, topk) * 4) + round256(bh * units_max(T, N, topk) * unit) +
         round256(bh * T * static_cast<size_t>(topk + 1) * kD * 4);
}

// Shapes the chunked path takes: c = d = 128, either write.
bool sse_chunk_supported(int write_mode, int N, int topk, int c, int d) {
  return (write_mode == SSE_WRITE_ADDITIVE || write_mode == SSE_WRITE_DELTA) && c == kCh && d == kD && N <= kMaxN &&
         topk <= kMaxTopk;
}

int test_drop_signal();  // gdn_chunk.cu: the SDM_TEST_DROP_SIGNAL test hook

namespace {

// the additive write's preparation and chain (the units and staging rows of
// the chunked path)
int launch_sse_additive_chunk(float *state, const uint32_t *rec, int rw, const uint32_t *grp, long gwords, int umax,
                              const float *klog, const uint16_t *q, const uint16_t *v, const float *alpha, long bhn,
                              int T, int H, int N, int topk, unsigned char *units, float *stage, int32_t *err,
                              int sms, cudaStream_t st) {
  PrepArgs pa;
  pa.q = q;
  pa.v = v;
  pa.klog = klog;
  pa.alpha = alpha;
  pa.rec = rec;
  pa.grp = grp;
  pa.units = units;
  pa.T = T;
  pa.H = H;
  pa.N = N;
  pa.topk = topk;
  pa.rw = rw;
  pa.umax = umax;
  pa.gwords = gwords;
  pa.total = bhn * umax;
  pa.err = err;
  if (cudaFuncSetAttribute(sse_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kPrepSmem)) != cudaSuccess)
    return check_launch("sse_scan: set shared memory");
  const long pmax = static_cast<long>(sms) * 2;
  sse_prep_kernel<<<static_cast<unsigned>(pa.total < pmax ? pa.total : pmax), kPThreads, kPrepSmem, st>>>(pa);
  const int rc = check_launch("sse_scan: chunk preparation kernel");
  if (rc != SDM_OK) return rc;

  ChainArgs ca;
  ca.state = state;
  ca.units = units;
  ca.grp = grp;
  ca.stage = stage;
  ca.T = T;
  ca.N = N;
  ca.umax = umax;
  ca.bh_count = bhn;
  ca.gwords = gwords;
  ca.err = err;
  ca.drop_signal = test_drop_signal();
  if (cudaFuncSetAttribute(sse_chain_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kChainSmem)) != cudaSuccess)
    return check_launch("sse_scan: set shared memory");
  sse_chain_kernel<<<static_cast<unsigned>(bhn * (N + 1)), kChainThreads, kChainSmem, st>>>(ca);
  return check_launch("sse_scan: chunk chain kernel");
}

}  // namespace

// launched by sse_scan after the routing prepass (rec: the routing records;
// chunk_ws: sse_chunk_workspace_size bytes, 256-byte aligned)
int launch_sse_chunk(float *state, const uint32_t *rec, int rw, const float *klog, const uint16_t *q,
                     const uint16_t *v, const float *alpha, int write_mode, int B, int T, int H, int N, int topk,
                     float *y, unsigned char *chunk_ws, int32_t *err, cudaStream_t st) {
  const long bhn = static_cast<long>(B) * H;
  const long gwords = group_words(T, topk);
  const int umax = units_max(T, N, topk);
  const size_t unit = write_mode == SSE_WRITE_DELTA ? sse_delta_unit_bytes() : static_cast<size_t>(kXUnit);
  uint32_t *grp = reinterpret_cast<uint32_t *>(chunk_ws);
  unsigned char *units = chunk_ws + round256(static_cast<size_t>(bhn) * gwords * 4);
  float *stage = reinterpret_cast<float *>(units + round256(static_cast<size_t>(bhn) * umax * unit));
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);

  sse_group_kernel<<<static_cast<unsigned>(bhn), kGroupThreads, 0, st>>>(rec, T, H, N, topk, rw, grp, gwords);
  int rc = check_launch("sse_scan: group kernel");
  if (rc != SDM_OK) return rc;
  if (write_mode == SSE_WRITE_DELTA)
    rc = launch_sse_delta_chunk(state, rec, rw, grp, gwords, umax, klog, q, v, alpha, B, T, H, N, topk, units, stage,
                                err, st);
  else
    rc = launch_sse_additive_chunk(state, rec, rw, grp, gwords, umax, klog, q, v, alpha, bhn, T, H, N, topk, units,
                                   stage, err, sms, st);
  if (rc != SDM_OK) return rc;

  const long n4 = bhn * T * (kD / 4);
  const long cgrid = (n4 + 255) / 256 < static_cast<long>(sms) * 8 ? (n4 + 255) / 256 : static_cast<long>(sms) * 8;
  sse_combine_kernel<<<static_cast<unsigned>(cgrid), 256, 0, st>>>(reinterpret_cast<const float4 *>(stage),
                                                                    reinterpret_cast<float4 *>(y), n4, topk + 1);
  return check_launch("sse_scan: combine kernel");
}

SDM_STICKY_ACCESSOR(sticky_sse_chunk)

}  // namespace sdm
