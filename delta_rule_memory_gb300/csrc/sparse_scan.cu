// sparse_scan.cu - the sparse delta-rule memory scan (Sparse Delta Memory
// deck, "Selected slots decay and update; other slots persist", Eqs. 3-5, and
// "A v1 inconsistency matters for reproducing the update", Fig. 2).
//
// Design (HBM-bound gather/scatter of fp32 table rows):
//   * Every value column evolves independently (the addresses do not depend on
//     the table), so one warp owns one (batch, head, column tile) slice of the
//     table for the whole sequence: no inter-warp synchronisation exists.
//   * Lane l owns CPL consecutive columns of the tile.  It copies exactly those
//     columns of every row it needs (cp.async, 4*CPL bytes), computes them and
//     stores them, so row data never crosses lanes.
//   * The rows of token t+P are prefetched while token t is computed (P-deep
//     ring in shared memory).  A row written by one of the last P tokens is
//     stale in that prefetch; a prepass kernel finds, for every (token, slot),
//     the most recent writer within the window, and the scan takes the row
//     from that writer's slot in the shared-memory history instead.
#include <climits>
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace sdm {
namespace {

constexpr uint16_t kHzNone = 0xffff;     // take the prefetched row
constexpr uint16_t kHzInvalid = 0xfffe;  // index out of range: read zeros, no store

__host__ __device__ inline int hz_stride(int W, int R) { return (W + R + 1) & ~1; }

// ---------------------------------------------------------------------------
// Hazard prepass: one thread per (token, slot).  hz[tok][s] for write slot
// s < W (look back d = 1..P) and read slot W + j (look back d = 0..P):
// (d << 8) | slot of the most recent token t - d whose write list holds the
// same row, kHzNone if none, kHzInvalid if the index is out of range.
// ---------------------------------------------------------------------------
__global__ void hazard_kernel(const int32_t *__restrict__ idx_w, const int32_t *__restrict__ idx_r, int W, int R,
                              int T, int H, int N, int window, long total, uint16_t *__restrict__ hz,
                              int32_t *__restrict__ dev_err) {
  const long tid = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tid >= total) return;
  const int WR = W + R;
  const long tok = tid / WR;
  const int s = static_cast<int>(tid - tok * WR);
  const long bt = tok / H;
  const int t = static_cast<int>(bt % T);
  const bool is_w = s < W;
  const int my = is_w ? idx_w[tok * W + s] : idx_r[tok * R + (s - W)];
  uint16_t code = kHzNone;
  int err = 0;
  if (my < 0 || my >= N) {
    code = kHzInvalid;
    err |= SDM_DEVERR_INDEX_RANGE;
  } else {
    if (is_w) {
      for (int j = 0; j < s; ++j)
        if (idx_w[tok * W + j] == my) err |= SDM_DEVERR_INDEX_REPEAT;
    }
    const int dmax = min(window, t);
    for (int d = is_w ? 1 : 0; d <= dmax && code == kHzNone; ++d) {
      const int32_t *lst = idx_w + (tok - static_cast<long>(d) * H) * W;
      for (int j = W - 1; j >= 0; --j) {
        if (lst[j] == my) {
          code = static_cast<uint16_t>((d << 8) | j);
          break;
        }
      }
    }
  }
  hz[tok * hz_stride(W, R) + s] = code;
  if (err && dev_err) atomicOr(dev_err, err);
}

// ---------------------------------------------------------------------------
// The scan.  One CTA of NG warps per (batch, head, column tile of tw <= 128
// columns).  Lane l owns columns [4l, 4l+4) of the tile (a float4 quad); warp
// g owns the write slots and read slots j == g (mod NG) of every token, so a
// token's rows are processed by all warps at once.  Per token:
//   B1  barrier: this token's rows (prefetched P tokens ago) have landed;
//       issue the prefetch of token t+P (rows) and t+2P (metadata);
//   2.  decay own write rows, partial shared prediction -> red1
//   B2  barrier (shared residual only): v_hat = sum over warps
//   3.  delta write of own write rows (history ring + table in HBM); read own
//       read rows -> partial y -> red2 (summed by warp 0 after the next B1).
// Rings in shared memory: incoming write rows (P+1 slots), post-write history
// (P+1 slots, the forwarding source), incoming read rows (P+1), metadata
// (2P+1).  A read slot that names a row written by the same token (distance
// 0) recomputes that row's new value from the same inputs, so no warp reads a
// history slot while another warp is writing it.
// ---------------------------------------------------------------------------
struct ScanArgs {
  float *state;
  const void *v;
  const float *alpha, *beta;
  const int32_t *idx_w, *idx_r;
  const float *w_w, *w_r;
  const uint16_t *hz;
  float *y;
  int W, R, T, H, N, d_v, mode, v_bf16, tiles, tw, hzs;
};

constexpr int kNG = 8;  // warps (row groups) per CTA

template <int SLOTS>
struct alignas(16) ScanMeta {
  int32_t iw[SLOTS];
  float ww[SLOTS];
  int32_t ir[SLOTS];
  float wr[SLOTS];
  uint16_t hz[2 * SLOTS];
  uint32_t vraw[128];  // tw fp32 values or tw/2 words of bf16 pairs
  float ab[4];         // alpha, beta
};

template <int SLOTS>
__host__ __device__ inline size_t scan_smem_bytes(int P, int tw) {
  const size_t rows = static_cast<size_t>(3) * (P + 1) * SLOTS * tw * sizeof(float);
  return rows + static_cast<size_t>(2 * P + 1) * sizeof(ScanMeta<SLOTS>) + 3 * kNG * 32 * sizeof(float4);
}

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 x) { *reinterpret_cast<float4 *>(p) = x; }
__device__ __forceinline__ float4 f4_fma(float s, float4 x, float4 acc) {
  return make_float4(fmaf(s, x.x, acc.x), fmaf(s, x.y, acc.y), fmaf(s, x.z, acc.z), fmaf(s, x.w, acc.w));
}
__device__ __forceinline__ float4 f4_scale(float s, float4 x) { return make_float4(s * x.x, s * x.y, s * x.z, s * x.w); }
__device__ __forceinline__ float4 f4_add(float4 a, float4 b) {
  return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float4 f4_sub(float4 a, float4 b) {
  return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w);
}

template <int P, int SLOTS>
__global__ void __launch_bounds__(kNG * 32, 1) sparse_scan_kernel(const ScanArgs a) {
  using Meta = ScanMeta<SLOTS>;
  constexpr int NI = P + 1, NH = P + 1, NR = P + 1, NM = 2 * P + 1;
  constexpr int NT = kNG * 32;
  constexpr int WPG = (SLOTS + kNG - 1) / kNG;           // write (or read) slots per warp
  constexpr int KMAX = (2 * SLOTS * 32 + NT - 1) / NT;  // row chunks per thread per token
  extern __shared__ __align__(16) unsigned char smem_raw[];

  const int tid = threadIdx.x, lane = tid & 31, g = tid >> 5;
  const int tile = blockIdx.x % a.tiles;
  const long bh = blockIdx.x / a.tiles;
  const int h = static_cast<int>(bh % a.H);
  const long b = bh / a.H;
  const int W = a.W, R = a.R, T = a.T, H = a.H, d_v = a.d_v, N = a.N;
  const int col0 = tile * a.tw;
  const int tw = min(a.tw, d_v - col0);  // this tile's width, a multiple of 4
  const int nq = tw >> 2;                // active quads (lanes)
  const int RS = a.tw;                   // smem row stride (floats)
  const bool qa = lane < nq;

  float *inW = reinterpret_cast<float *>(smem_raw);
  float *hist = inW + NI * SLOTS * RS;
  float *inR = hist + NH * SLOTS * RS;
  Meta *meta = reinterpret_cast<Meta *>(inR + NR * SLOTS * RS);
  float4 *red1 = reinterpret_cast<float4 *>(meta + NM);  // [NG][32]
  float4 *red2 = red1 + kNG * 32;                         // [2][NG][32]

  float *table = a.state + bh * static_cast<long>(N) * d_v + col0;
  const long tok0 = b * T * H + h;

  // this thread's row chunks: chunk c = tid + k*NT of the (W+R) x nq grid
  int ck_row[KMAX], ck_q[KMAX];
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    const int c = tid + k * NT;
    const int row = nq > 0 ? c / nq : 0;
    ck_row[k] = (c < (W + R) * nq) ? row : -1;
    ck_q[k] = c - row * nq;
  }

  const int v_words = a.v_bf16 ? tw / 2 : tw;
  const int hz_words = a.hzs / 2;
  const int m_total = 2 * W + 2 * R + hz_words + v_words + 2;

  auto issue_meta = [&](int t) {
    Meta &m = meta[t % NM];
    const long tok = tok0 + static_cast<long>(t) * H;
    for (int q = tid; q < m_total; q += NT) {
      int r = q;
      void *dst;
      const void *src;
      if (r < W) { dst = &m.iw[r]; src = a.idx_w + tok * W + r; }
      else if ((r -= W) < W) { dst = &m.ww[r]; src = a.w_w + tok * W + r; }
      else if ((r -= W) < R) { dst = &m.ir[r]; src = a.idx_r + tok * R + r; }
      else if ((r -= R) < R) { dst = &m.wr[r]; src = a.w_r + tok * R + r; }
      else if ((r -= R) < hz_words) {
        dst = reinterpret_cast<uint32_t *>(m.hz) + r;
        src = reinterpret_cast<const uint32_t *>(a.hz + tok * a.hzs) + r;
      } else if ((r -= hz_words) < v_words) {
        dst = &m.vraw[r];
        src = a.v_bf16 ? static_cast<const void *>(static_cast<const uint16_t *>(a.v) + tok * d_v + col0 + 2 * r)
                       : static_cast<const void *>(static_cast<const float *>(a.v) + tok * d_v + col0 + r);
      } else {
        r -= v_words;
        dst = &m.ab[r];
        src = (r == 0 ? a.alpha : a.beta) + tok;
      }
      cp_async<4>(dst, src);
    }
  };
  auto issue_rows = [&](int t) {
    const Meta &m = meta[t % NM];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int row = ck_row[k];
      if (row < 0) continue;
      const bool isw = row < W;
      const int j = isw ? row : row - W;
      const int i = isw ? m.iw[j] : m.ir[j];
      float *dst = (isw ? inW + (t % NI) * SLOTS * RS : inR + (t % NR) * SLOTS * RS) + j * RS + 4 * ck_q[k];
      if (static_cast<unsigned>(i) < static_cast<unsigned>(N))
        cp_async<16>(dst, table + static_cast<long>(i) * d_v + 4 * ck_q[k]);
    }
  };

  // prologue: metadata of tokens [0, P), then P groups (rows of j, meta of j+P)
  for (int t = 0; t < P && t < T; ++t) issue_meta(t);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  for (int j = 0; j < P; ++j) {
    if (j + P < T) issue_meta(j + P);
    if (j < T) issue_rows(j);
    cp_async_commit();
  }

  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int t = 0; t < T; ++t) {
    cp_async_wait<P - 1>();
    __syncthreads();  // B1
    if (t > 0 && g == 0 && qa) {
      const float4 *rd = red2 + ((t - 1) & 1) * kNG * 32;
      float4 acc = rd[lane];
#pragma unroll
      for (int w = 1; w < kNG; ++w) acc = f4_add(acc, rd[w * 32 + lane]);
      st4(a.y + (tok0 + static_cast<long>(t - 1) * H) * d_v + col0 + 4 * lane, acc);
    }
    if (t + 2 * P < T) issue_meta(t + 2 * P);
    if (t + P < T) issue_rows(t + P);
    cp_async_commit();

    const Meta &m = meta[t % NM];
    const float al = m.ab[0], be = m.ab[1];
    float4 vv = zero4;
    if (qa) {
      if (a.v_bf16) {
        const uint32_t w0 = m.vraw[2 * lane], w1 = m.vraw[2 * lane + 1];
        vv = make_float4(bf16_to_f32(w0 & 0xffff), bf16_to_f32(w0 >> 16), bf16_to_f32(w1 & 0xffff),
                         bf16_to_f32(w1 >> 16));
      } else {
        vv = make_float4(__uint_as_float(m.vraw[4 * lane]), __uint_as_float(m.vraw[4 * lane + 1]),
                         __uint_as_float(m.vraw[4 * lane + 2]), __uint_as_float(m.vraw[4 * lane + 3]));
      }
    }
    const float *cur_in = inW + (t % NI) * SLOTS * RS + 4 * lane;
    auto hist_row = [&](int d, int s) { return hist + ((t - d) % NH) * SLOTS * RS + s * RS + 4 * lane; };
    // the row a write slot starts from (before decay)
    auto write_src = [&](int j) -> float4 {
      const uint16_t code = m.hz[j];
      if (code == kHzNone) return ld4(cur_in + j * RS);
      if (code == kHzInvalid) return zero4;
      return ld4(hist_row(code >> 8, code & 0xff));
    };

    // phase 2: selective decay of the written rows, partial shared prediction
    float4 md[WPG];
    float4 vh = zero4;
#pragma unroll
    for (int i = 0; i < WPG; ++i) {
      const int j = g + kNG * i;
      md[i] = zero4;
      if (j < W && qa) {
        md[i] = f4_scale(al, write_src(j));
        vh = f4_fma(m.ww[j], md[i], vh);
      }
    }
    if (a.mode == SDM_RESID_SHARED) {
      red1[g * 32 + lane] = vh;
      __syncthreads();  // B2
      vh = red1[lane];
#pragma unroll
      for (int w = 1; w < kNG; ++w) vh = f4_add(vh, red1[w * 32 + lane]);
    }
    const float4 base = a.mode == SDM_RESID_SHARED ? f4_sub(vv, vh) : vv;
    auto new_row = [&](float4 mdj, float gj) -> float4 {
      const float4 resid = a.mode == SDM_RESID_PERSLOT ? f4_sub(vv, mdj) : base;
      return f4_fma(gj, resid, mdj);
    };

    // phase 3: delta write into the history ring and the table
    float *cur_hist = hist + (t % NH) * SLOTS * RS + 4 * lane;
#pragma unroll
    for (int i = 0; i < WPG; ++i) {
      const int j = g + kNG * i;
      if (j < W && qa) {
        const float4 nw = new_row(md[i], be * m.ww[j]);
        st4(cur_hist + j * RS, nw);
        const int row = m.iw[j];
        if (m.hz[j] != kHzInvalid && static_cast<unsigned>(row) < static_cast<unsigned>(N))
          st4(table + static_cast<long>(row) * d_v + 4 * lane, nw);
      }
    }
    // read after the write
    float4 yp = zero4;
    const float *cur_r = inR + (t % NR) * SLOTS * RS + 4 * lane;
#pragma unroll
    for (int i = 0; i < WPG; ++i) {
      const int j = g + kNG * i;
      if (j < R && qa) {
        const uint16_t code = m.hz[W + j];
        float4 x;
        if (code == kHzNone) {
          x = ld4(cur_r + j * RS);
        } else if (code == kHzInvalid) {
          x = zero4;
        } else if ((code >> 8) == 0) {
          const int s = code & 0xff;  // written by this token: recompute its new value
          x = new_row(f4_scale(al, write_src(s)), be * m.ww[s]);
        } else {
          x = ld4(hist_row(code >> 8, code & 0xff));
        }
        yp = f4_fma(m.wr[j], x, yp);
      }
    }
    red2[(t & 1) * kNG * 32 + g * 32 + lane] = yp;
  }
  cp_async_wait<0>();
  __syncthreads();
  if (T > 0 && g == 0 && qa) {
    const float4 *rd = red2 + ((T - 1) & 1) * kNG * 32;
    float4 acc = rd[lane];
#pragma unroll
    for (int w = 1; w < kNG; ++w) acc = f4_add(acc, rd[w * 32 + lane]);
    st4(a.y + (tok0 + static_cast<long>(T - 1) * H) * d_v + col0 + 4 * lane, acc);
  }
}

int env_int(const char *name, int dflt) {
  const char *s = getenv(name);
  return (s && *s) ? atoi(s) : dflt;
}

size_t smem_dispatch(int slots, int P, int tw) {
  return slots == 16 ? scan_smem_bytes<16>(P, tw) : scan_smem_bytes<64>(P, tw);
}

template <int P, int SLOTS>
int launch_scan(const ScanArgs &args, long blocks, cudaStream_t st) {
  const size_t smem = scan_smem_bytes<SLOTS>(P, args.tw);
  auto kern = sparse_scan_kernel<P, SLOTS>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return check_launch("sdm_scan: set shared memory");
  kern<<<static_cast<unsigned>(blocks), kNG * 32, smem, st>>>(args);
  return check_launch("sdm_scan: scan kernel");
}

int launch_dispatch(int slots, int P, const ScanArgs &args, long blocks, cudaStream_t st) {
#define SDM_LS(S, PP) \
  if (slots == S && P == PP) return launch_scan<PP, S>(args, blocks, st);
  SDM_LS(16, 4) SDM_LS(16, 6) SDM_LS(16, 8) SDM_LS(64, 4) SDM_LS(64, 6) SDM_LS(64, 8)
#undef SDM_LS
  return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan: no kernel for slots=%d window=%d", slots, P);
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" size_t sdm_scan_workspace_size(int B, int T, int H, int W, int R) {
  if (B <= 0 || T <= 0 || H <= 0 || W <= 0 || R <= 0) return 0;
  const size_t n = static_cast<size_t>(B) * T * H * hz_stride(W, R) * sizeof(uint16_t);
  return (n + 255) & ~static_cast<size_t>(255);
}

extern "C" int sdm_scan(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
                        const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r, const float *w_r, int R,
                        int B, int T, int H, int N, int d_v, int resid_mode, float *y, void *workspace,
                        size_t workspace_bytes, int32_t *dev_err, void *stream) {
  if (!state || !v || !alpha || !beta || !idx_w || !w_w || !idx_r || !w_r || !y)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan: null pointer");
  if (B < 0 || T < 0 || H < 0 || N < 1 || d_v < 1)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan: bad sizes");
  if (W < 1 || W > 64 || R < 1 || R > 64) return set_error(SDM_ERR_SHAPE, "sdm_scan: need 1 <= W, R <= 64");
  if (d_v % 4 != 0) return set_error(SDM_ERR_SHAPE, "sdm_scan: d_v must be a multiple of 4");
  if (v_dtype != SDM_DTYPE_F32 && v_dtype != SDM_DTYPE_BF16)
    return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan: v_dtype must be SDM_DTYPE_F32 or SDM_DTYPE_BF16");
  if (resid_mode != SDM_RESID_SHARED && resid_mode != SDM_RESID_PERSLOT && resid_mode != SDM_RESID_ADDITIVE)
    return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan: unknown resid_mode %d", resid_mode);
  if (!aligned(state, 16) || !aligned(y, 16) || !aligned(v, 4) || !aligned(alpha, 4) || !aligned(beta, 4) ||
      !aligned(idx_w, 4) || !aligned(w_w, 4) || !aligned(idx_r, 4) || !aligned(w_r, 4) ||
      (dev_err && !aligned(dev_err, 4)))
    return set_error(SDM_ERR_ALIGN, "sdm_scan: state and y need 16-byte, other arrays 4-byte alignment");
  if (static_cast<double>(B) * T * H * (W + R) >= 9.0e18) return set_error(SDM_ERR_SHAPE, "sdm_scan: too large");
  if (B == 0 || T == 0 || H == 0) return SDM_OK;
  const size_t need = sdm_scan_workspace_size(B, T, H, W, R);
  if (!workspace || workspace_bytes < need)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan: workspace of %zu bytes needed", need);
  if (!aligned(workspace, 16)) return set_error(SDM_ERR_ALIGN, "sdm_scan: workspace must be 16-byte aligned");

  // Launch shape: one CTA of 8 warps per (b, h, column tile).  Every CTA
  // runs the whole sequence, so the grid should be one wave: split d_v into
  // as many tiles (<= 128 columns each) as the SMs allow, then take the
  // deepest prefetch window whose shared-memory rings fit.
  const int slots = (W <= 16 && R <= 16) ? 16 : 64;
  int dev = 0, smem_blk = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long bh_count = static_cast<long>(B) * H;
  const int quads = d_v / 4;
  const int tiles_min = (quads + 31) / 32;
  long tiles_want = sms / bh_count;
  if (tiles_want > quads) tiles_want = quads;
  int tiles = static_cast<int>(tiles_want > tiles_min ? tiles_want : tiles_min);
  tiles = env_int("SDM_SCAN_TILES", tiles);
  if (tiles < tiles_min) tiles = tiles_min;
  if (tiles > quads) tiles = quads;
  int tw = 4 * ((quads + tiles - 1) / tiles);
  int window = 0;
  const int want_window = env_int("SDM_SCAN_WINDOW", 0);
  for (int p : {8, 6, 4}) {
    if (want_window && p != want_window) continue;
    if (smem_dispatch(slots, p, tw) <= static_cast<size_t>(smem_blk)) { window = p; break; }
  }
  if (window == 0) {  // narrower tiles until the smallest window fits
    window = want_window ? want_window : 4;
    while (tw > 4 && smem_dispatch(slots, window, tw) > static_cast<size_t>(smem_blk)) tw -= 4;
    if (smem_dispatch(slots, window, tw) > static_cast<size_t>(smem_blk))
      return set_error(SDM_ERR_SHAPE, "sdm_scan: W/R too large for shared memory");
  }
  tiles = (d_v + tw - 1) / tw;

  ScanArgs args;
  args.state = state;
  args.v = v;
  args.alpha = alpha;
  args.beta = beta;
  args.idx_w = idx_w;
  args.idx_r = idx_r;
  args.w_w = w_w;
  args.w_r = w_r;
  args.hz = static_cast<const uint16_t *>(workspace);
  args.y = y;
  args.W = W;
  args.R = R;
  args.T = T;
  args.H = H;
  args.N = N;
  args.d_v = d_v;
  args.mode = resid_mode;
  args.v_bf16 = v_dtype == SDM_DTYPE_BF16;
  args.tiles = tiles;
  args.tw = tw;
  args.hzs = hz_stride(W, R);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long total = static_cast<long>(B) * T * H * (W + R);
  hazard_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(
      idx_w, idx_r, W, R, T, H, N, window, total, static_cast<uint16_t *>(workspace), dev_err);
  int rc = check_launch("sdm_scan: hazard kernel");
  if (rc != SDM_OK) return rc;
  return launch_dispatch(slots, window, args, bh_count * tiles, st);
}

// ---------------------------------------------------------------------------
// sdm_scan_noalloc: sdm_scan for callers that cannot hand over device scratch
// memory.  The hazard table lives in a fixed, file-scope device array instead
// of a caller workspace.  Host code cannot use the array's name as a device
// address, so the address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached; the first call
// on a device does this lookup, so make that first call before capturing any
// stream.  Every call shares the one array: calls that can overlap on the GPU
// (different streams, or several host threads) race on it and must be
// serialised by the caller.  The hazard table is fully rewritten by every
// call, so nothing has to be cleared between calls.
// ---------------------------------------------------------------------------
namespace sdm {
namespace {
constexpr size_t kStaticScratchBytes = static_cast<size_t>(8) << 20;  // 8 MiB per device
__device__ __align__(256) unsigned char g_scan_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

int static_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(SDM_ERR_CUDA, "sdm_scan_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scan_scratch);
    if (e != cudaSuccess || !p)
      return set_error(SDM_ERR_CUDA, "sdm_scan_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return SDM_OK;
}
}  // namespace
}  // namespace sdm

extern "C" int sdm_scan_noalloc(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
                                const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r,
                                const float *w_r, int R, int B, int T, int H, int N, int d_v, int resid_mode,
                                float *y, int32_t *dev_err, void *stream) {
  if (B < 0 || T < 0 || H < 0 || W < 1 || W > 64 || R < 1 || R > 64)
    return set_error(SDM_ERR_SHAPE, "sdm_scan_noalloc: bad sizes");
  const size_t need = sdm_scan_workspace_size(B, T, H, W, R);
  if (need > sdm::kStaticScratchBytes)
    return set_error(SDM_ERR_SHAPE,
                     "sdm_scan_noalloc: B*T*H*(W+R) too large: needs %zu bytes of scratch, the static array holds "
                     "%zu; use sdm_scan with a workspace",
                     need, sdm::kStaticScratchBytes);
  if (B == 0 || T == 0 || H == 0) return SDM_OK;
  void *scratch = nullptr;
  const int rc = sdm::static_scratch(&scratch);
  if (rc != SDM_OK) return rc;
  return sdm_scan(state, v, v_dtype, alpha, beta, idx_w, w_w, W, idx_r, w_r, R, B, T, H, N, d_v, resid_mode, y,
                  scratch, sdm::kStaticScratchBytes, dev_err, stream);
}
