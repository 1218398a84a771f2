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
// The scan.
// ---------------------------------------------------------------------------
struct ScanArgs {
  float *state;
  const void *v;
  const float *alpha, *beta;
  const int32_t *idx_w, *idx_r;
  const float *w_w, *w_r;
  const uint16_t *hz;
  float *y;
  int W, R, T, H, N, d_v, mode, v_bf16, tiles, hzs;
  long total_warps;
};

template <int CPL, int SLOTS, int P>
struct ScanLayout {
  static constexpr int TC = 32 * CPL;  // tile columns
  static constexpr int NW = 2 * P + 1; // write-row ring: P in flight, current, P history
  static constexpr int NR = P + 1;     // read-row ring: P in flight, current
  static constexpr int NM = 2 * P + 1; // per-token metadata ring
  struct alignas(16) Meta {
    int32_t iw[SLOTS];
    float ww[SLOTS];
    int32_t ir[SLOTS];
    float wr[SLOTS];
    uint16_t hz[2 * SLOTS];
    uint32_t vraw[TC];  // TC fp32 or TC/2 words of bf16 pairs
    float ab[2];        // alpha, beta
  };
  static constexpr size_t kRowsBytes = static_cast<size_t>(NW + NR) * SLOTS * TC * sizeof(float);
  static constexpr size_t kZeroOffset = kRowsBytes + NM * sizeof(Meta);  // one all-zero row
  static constexpr size_t kWarpBytes = (kZeroOffset + TC * sizeof(float) + 127) & ~static_cast<size_t>(127);
  static_assert(sizeof(Meta) % 16 == 0 && kRowsBytes % 16 == 0, "16-byte alignment of the warp's regions");
};

template <int CPL>
__device__ __forceinline__ void load_cols(const float *p, float (&x)[CPL]) {
  if constexpr (CPL == 4) {
    const float4 q = *reinterpret_cast<const float4 *>(p);
    x[0] = q.x; x[1] = q.y; x[2] = q.z; x[3] = q.w;
  } else if constexpr (CPL == 2) {
    const float2 q = *reinterpret_cast<const float2 *>(p);
    x[0] = q.x; x[1] = q.y;
  } else {
    x[0] = *p;
  }
}
template <int CPL>
__device__ __forceinline__ void store_cols(float *p, const float (&x)[CPL]) {
  if constexpr (CPL == 4) {
    *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
  } else if constexpr (CPL == 2) {
    *reinterpret_cast<float2 *>(p) = make_float2(x[0], x[1]);
  } else {
    *p = x[0];
  }
}

template <int CPL, int SLOTS, int P>
__global__ void __launch_bounds__(256) sparse_scan_kernel(const ScanArgs a) {
  using L = ScanLayout<CPL, SLOTS, P>;
  using Meta = typename L::Meta;
  constexpr int TC = L::TC;
  extern __shared__ __align__(16) unsigned char smem_raw[];

  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const long gw = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + wib;
  if (gw >= a.total_warps) return;  // warp-uniform; the kernel has no CTA barrier
  const int tile = static_cast<int>(gw % a.tiles);
  const long bh = gw / a.tiles;
  const int h = static_cast<int>(bh % a.H);
  const long b = bh / a.H;

  unsigned char *base = smem_raw + static_cast<size_t>(wib) * L::kWarpBytes;
  float(*wring)[SLOTS][TC] = reinterpret_cast<float(*)[SLOTS][TC]>(base);
  float(*rring)[SLOTS][TC] = reinterpret_cast<float(*)[SLOTS][TC]>(base + sizeof(float) * L::NW * SLOTS * TC);
  Meta *meta = reinterpret_cast<Meta *>(base + L::kRowsBytes);
  float *zero_row = reinterpret_cast<float *>(base + L::kZeroOffset);

  const int lc = lane * CPL;               // first column of this lane inside the tile
  const int col = tile * TC + lc;          // absolute column
  const bool active = col < a.d_v;
  const int W = a.W, R = a.R, T = a.T, H = a.H, d_v = a.d_v;
  float *table = a.state + bh * static_cast<long>(a.N) * d_v;  // [N, d_v] of this (b, h)
  const long tok0 = b * T * H + h;                               // token t -> tok0 + t*H

  // words of metadata per token, in copy order
  const int v_words = a.v_bf16 ? TC / 2 : TC;
  const int hz_words = a.hzs / 2;
  const int m_total = 2 * W + 2 * R + hz_words + v_words + 2;

  auto issue_meta = [&](int t) {
    Meta &m = meta[t % L::NM];
    const long tok = tok0 + static_cast<long>(t) * H;
    for (int q = lane; q < m_total; q += 32) {
      int r = q;
      void *dst;
      const void *src;
      bool ok = true;
      if (r < W) { dst = &m.iw[r]; src = a.idx_w + tok * W + r; }
      else if ((r -= W) < W) { dst = &m.ww[r]; src = a.w_w + tok * W + r; }
      else if ((r -= W) < R) { dst = &m.ir[r]; src = a.idx_r + tok * R + r; }
      else if ((r -= R) < R) { dst = &m.wr[r]; src = a.w_r + tok * R + r; }
      else if ((r -= R) < hz_words) {
        dst = reinterpret_cast<uint32_t *>(m.hz) + r;
        src = reinterpret_cast<const uint32_t *>(a.hz + tok * a.hzs) + r;
      } else if ((r -= hz_words) < v_words) {
        const int c0 = tile * TC + (a.v_bf16 ? 2 * r : r);
        ok = c0 < d_v;
        dst = &m.vraw[r];
        src = a.v_bf16 ? static_cast<const void *>(static_cast<const uint16_t *>(a.v) + tok * d_v + c0)
                       : static_cast<const void *>(static_cast<const float *>(a.v) + tok * d_v + c0);
      } else {
        r -= v_words;
        dst = &m.ab[r];
        src = (r == 0 ? a.alpha : a.beta) + tok;
      }
      if (ok) cp_async<4>(dst, src);
    }
  };
  auto issue_rows = [&](int t) {
    const Meta &m = meta[t % L::NM];
    if (!active) return;
    float(*wr)[TC] = wring[t % L::NW];
    float(*rr)[TC] = rring[t % L::NR];
    for (int j = 0; j < W; ++j) {
      const int i = m.iw[j];
      if (static_cast<unsigned>(i) < static_cast<unsigned>(a.N))
        cp_async<4 * CPL>(&wr[j][lc], table + static_cast<long>(i) * d_v + col);
    }
    for (int j = 0; j < R; ++j) {
      const int i = m.ir[j];
      if (static_cast<unsigned>(i) < static_cast<unsigned>(a.N))
        cp_async<4 * CPL>(&rr[j][lc], table + static_cast<long>(i) * d_v + col);
    }
  };

  // prologue: metadata of tokens [0, P) first, then P groups that each carry
  // the metadata of token j+P and the rows of token j.
  for (int t = 0; t < P && t < T; ++t) issue_meta(t);
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  for (int j = 0; j < P; ++j) {
    if (j + P < T) issue_meta(j + P);
    if (j < T) issue_rows(j);
    cp_async_commit();
  }

#pragma unroll
  for (int c = 0; c < CPL; ++c) zero_row[lc + c] = 0.f;
  for (int t = 0; t < T; ++t) {
    // group t-P (rows of t, metadata of t+P) has landed
    cp_async_wait<P - 1>();
    __syncwarp();
    if (t + 2 * P < T) issue_meta(t + 2 * P);
    if (t + P < T) issue_rows(t + P);
    cp_async_commit();

    const Meta &m = meta[t % L::NM];
    float(*cur)[TC] = wring[t % L::NW];
    const float al = m.ab[0], be = m.ab[1];
    float vv[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      if (a.v_bf16) {
        const uint32_t wd = m.vraw[(lc + c) >> 1];
        vv[c] = bf16_to_f32(static_cast<uint16_t>(((lc + c) & 1) ? (wd >> 16) : (wd & 0xffff)));
      } else {
        vv[c] = __uint_as_float(m.vraw[lc + c]);
      }
    }
    auto src_row = [&](uint16_t code, const float *prefetched) -> const float * {
      if (code == kHzNone) return prefetched;
      if (code == kHzInvalid) return zero_row + lc;
      const int d = code >> 8, s = code & 0xff;
      return &wring[(t - d) % L::NW][s][lc];
    };

    if (active) {
      // shared prediction from the decayed rows (Fig. 2)
      float vh[CPL] = {};
      if (a.mode == SDM_RESID_SHARED) {
        for (int j = 0; j < W; ++j) {
          float x[CPL];
          load_cols<CPL>(src_row(m.hz[j], &cur[j][lc]), x);
          const float wj = m.ww[j];
#pragma unroll
          for (int c = 0; c < CPL; ++c) vh[c] = fmaf(wj, al * x[c], vh[c]);
        }
      }
      // selective decay and delta write
      for (int j = 0; j < W; ++j) {
        const uint16_t code = m.hz[j];
        float x[CPL];
        load_cols<CPL>(src_row(code, &cur[j][lc]), x);
        const float g = be * m.ww[j];
        float nw[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
          const float md = al * x[c];
          const float resid = a.mode == SDM_RESID_SHARED ? vv[c] - vh[c]
                              : a.mode == SDM_RESID_PERSLOT ? vv[c] - md
                                                            : vv[c];
          nw[c] = fmaf(g, resid, md);
        }
        store_cols<CPL>(&cur[j][lc], nw);
        if (code != kHzInvalid && static_cast<unsigned>(m.iw[j]) < static_cast<unsigned>(a.N))
          store_cols<CPL>(table + static_cast<long>(m.iw[j]) * d_v + col, nw);
      }
      // read after the write
      float acc[CPL] = {};
      const float(*rr)[TC] = rring[t % L::NR];
      for (int j = 0; j < R; ++j) {
        float x[CPL];
        load_cols<CPL>(src_row(m.hz[W + j], &rr[j][lc]), x);
        const float rj = m.wr[j];
#pragma unroll
        for (int c = 0; c < CPL; ++c) acc[c] = fmaf(rj, x[c], acc[c]);
      }
      store_cols<CPL>(a.y + (tok0 + static_cast<long>(t) * H) * d_v + col, acc);
    }
  }
  cp_async_wait<0>();
}

struct Tuning {
  int cpl, window, warps_per_cta;
};

int env_int(const char *name, int dflt) {
  const char *s = getenv(name);
  return (s && *s) ? atoi(s) : dflt;
}

template <int CPL, int SLOTS, int P>
size_t warp_bytes() {
  return ScanLayout<CPL, SLOTS, P>::kWarpBytes;
}

size_t warp_bytes_dispatch(int cpl, int slots, int p) {
#define SDM_WB(C, S, PP) \
  if (cpl == C && slots == S && p == PP) return warp_bytes<C, S, PP>();
  SDM_WB(1, 16, 4) SDM_WB(2, 16, 4) SDM_WB(4, 16, 4) SDM_WB(1, 16, 8) SDM_WB(2, 16, 8) SDM_WB(4, 16, 8)
  SDM_WB(1, 64, 4) SDM_WB(2, 64, 4) SDM_WB(4, 64, 4) SDM_WB(1, 64, 8) SDM_WB(2, 64, 8) SDM_WB(4, 64, 8)
#undef SDM_WB
  return 0;
}

template <int CPL, int SLOTS, int P>
int launch_scan(const ScanArgs &args, int wpc, cudaStream_t st) {
  using L = ScanLayout<CPL, SLOTS, P>;
  const size_t smem = L::kWarpBytes * wpc;
  auto kern = sparse_scan_kernel<CPL, SLOTS, P>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return check_launch("sdm_scan: set shared memory");
  const long blocks = (args.total_warps + wpc - 1) / wpc;
  kern<<<static_cast<unsigned>(blocks), wpc * 32, smem, st>>>(args);
  return check_launch("sdm_scan: scan kernel");
}

int launch_dispatch(int cpl, int slots, int p, const ScanArgs &args, int wpc, cudaStream_t st) {
#define SDM_LS(C, S, PP) \
  if (cpl == C && slots == S && p == PP) return launch_scan<C, S, PP>(args, wpc, st);
  SDM_LS(1, 16, 4) SDM_LS(2, 16, 4) SDM_LS(4, 16, 4) SDM_LS(1, 16, 8) SDM_LS(2, 16, 8) SDM_LS(4, 16, 8)
  SDM_LS(1, 64, 4) SDM_LS(2, 64, 4) SDM_LS(4, 64, 4) SDM_LS(1, 64, 8) SDM_LS(2, 64, 8) SDM_LS(4, 64, 8)
#undef SDM_LS
  return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan: no kernel for cpl=%d slots=%d window=%d", cpl, slots, p);
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

  // Tuning: columns per lane (cpl), prefetch window (tokens in flight) and
  // warps per CTA.  Every warp runs the whole sequence, so the launch must be
  // a single wave: pick the first (window, cpl) whose warps all fit at once.
  const int slots = (W <= 16 && R <= 16) ? 16 : 64;
  int dev = 0, smem_blk = 0, smem_sm = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  static const int kOrder[][2] = {{1, 8}, {2, 8}, {1, 4}, {2, 4}, {4, 4}, {4, 8}};
  int cpl = 0, window = 0;
  for (const auto &o : kOrder) {
    const size_t wb = warp_bytes_dispatch(o[0], slots, o[1]);
    if (wb == 0 || wb > static_cast<size_t>(smem_blk)) continue;
    const long tiles_o = (d_v + 32 * o[0] - 1) / (32 * o[0]);
    const long warps_o = static_cast<long>(B) * H * tiles_o;
    const long per_sm = static_cast<long>(smem_sm - 1024) / static_cast<long>(wb);
    if (cpl == 0) { cpl = o[0]; window = o[1]; }  // fallback: first that fits a CTA
    if (per_sm >= 1 && warps_o <= per_sm * sms) { cpl = o[0]; window = o[1]; break; }
  }
  cpl = env_int("SDM_SCAN_CPL", cpl);
  window = env_int("SDM_SCAN_WINDOW", window);
  if ((cpl != 1 && cpl != 2 && cpl != 4) || (window != 4 && window != 8))
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan: SDM_SCAN_CPL must be 1/2/4 and SDM_SCAN_WINDOW 4/8");
  const size_t wb = warp_bytes_dispatch(cpl, slots, window);
  if (wb == 0 || wb > static_cast<size_t>(smem_blk))
    return set_error(SDM_ERR_SHAPE, "sdm_scan: W/R too large for shared memory");
  const int tc = 32 * cpl;
  const int tiles = (d_v + tc - 1) / tc;
  const long total_warps = static_cast<long>(B) * H * tiles;
  const int fit = static_cast<int>(static_cast<size_t>(smem_blk) / wb);
  int wpc = env_int("SDM_SCAN_WARPS", 0);
  if (wpc <= 0) {
    const long per_sm = (total_warps + sms - 1) / sms;
    wpc = static_cast<int>(per_sm < 1 ? 1 : per_sm);
  }
  wpc = min(min(wpc, fit), 8);

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
  args.hzs = hz_stride(W, R);
  args.total_warps = total_warps;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long total = static_cast<long>(B) * T * H * (W + R);
  hazard_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, st>>>(
      idx_w, idx_r, W, R, T, H, N, window, total, static_cast<uint16_t *>(workspace), dev_err);
  int rc = check_launch("sdm_scan: hazard kernel");
  if (rc != SDM_OK) return rc;
  return launch_dispatch(cpl, slots, window, args, wpc, st);
}
