// sparse_backward.cu - gradients of the sparse delta-rule memory scan by
// undoing its writes (Sparse Delta Memory deck, "Training parallelizes within
// chunks and recurs across chunks" and "Backup: undoing writes avoids
// repeated full-table snapshots", App. A.3).
//
// The forward (sdm_scan_train) leaves M_T in the table and logs, per token,
// the written rows as they were before the token's decay.  Walking the tokens
// backwards with M = M_t and G = dL/dM_t:
//   read   y = sum_i r_i M[i]:       dr_i = <dy, M[i]>,  G[i] += r_i dy
//   write  M[i_j] = m_j + beta w_j rho_j,  m_j = alpha undo_j,
//          rho_j = v - sum_k w_k m_k (shared) | v - m_j (per-slot) | v (additive):
//            g      = beta sum_j w_j G_j          -> dv
//            dbeta  = sum_j w_j <G_j, rho_j>
//            dw_j   = beta <G_j, rho_j>  (- <g, m_j> for the shared residual)
//            dm_j   = G_j - w_j g | G_j (1 - beta w_j) | G_j
//            dalpha = sum_j <dm_j, undo_j>
//          then G[i_j] = alpha dm_j and M[i_j] = undo_j (M_{t-1}).
// Every value column is independent: one warp per (batch, head, 32-column
// tile), one column per lane, so a lane is the only reader and writer of its
// column of M and G and needs no synchronisation.  The column sums (dr, dw,
// dalpha, dbeta) are reduced over the warp and written per tile; a second
// kernel adds the tiles in a fixed order.
#include <climits>

#include "common.cuh"

namespace sdm {
namespace {

struct BackArgs {
  float *state, *dstate;
  const void *v;
  const float *alpha, *beta;
  const int32_t *idx_w, *idx_r;
  const float *w_w, *w_r;
  const float *undo, *dy;
  float *dv;
  float *part;  // [tiles][B*T*H][R + W + 2]: per-tile column sums
  int32_t *err;
  int T, H, N, d_v, W, R, mode, v_bf16, tiles;
  long total_warps;
};

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

template <int MODE>
__global__ void __launch_bounds__(128) sparse_backward_kernel(const BackArgs a) {
  const int lane = threadIdx.x & 31;
  const long gw = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= a.total_warps) return;  // warp-uniform
  const int tile = static_cast<int>(gw % a.tiles);
  const long bh = gw / a.tiles;
  const int h = static_cast<int>(bh % a.H);
  const long b = bh / a.H;
  const int T = a.T, H = a.H, N = a.N, d_v = a.d_v, W = a.W, R = a.R;
  const int col = tile * 32 + lane;
  const bool active = col < d_v;
  const int ccol = active ? col : 0;  // inactive lanes read column 0 and store nothing
  float *M = a.state + bh * static_cast<long>(N) * d_v + ccol;
  float *G = a.dstate + bh * static_cast<long>(N) * d_v + ccol;
  const int np = R + W + 2;
  int bad = 0;

  for (int t = T - 1; t >= 0; --t) {
    const long tok = (b * T + t) * H + h;
    const float al = a.alpha[tok], be = a.beta[tok];
    const float vc = a.v_bf16 ? bf16_to_f32(static_cast<const uint16_t *>(a.v)[tok * d_v + ccol])
                              : static_cast<const float *>(a.v)[tok * d_v + ccol];
    const float dyc = a.dy[tok * d_v + ccol];
    // this tile's column sums of token tok: [tile][B*T*H][np], B*H*T = (total_warps / tiles) * T rows
    float *pt = a.part + (static_cast<long>(tile) * (a.total_warps / a.tiles) * T + tok) * np;
    // ---- the read after the write
    for (int i = 0; i < R; ++i) {
      const int row = a.idx_r[tok * R + i];
      float dr = 0.f;
      if (static_cast<unsigned>(row) < static_cast<unsigned>(N)) {
        const long o = static_cast<long>(row) * d_v;
        dr = active ? dyc * M[o] : 0.f;
        if (active) G[o] = fmaf(a.w_r[tok * R + i], dyc, G[o]);
      } else {
        bad = 1;
      }
      dr = warp_sum(dr);
      if (lane == 0) pt[i] = dr;
    }
    // ---- the write
    const int32_t *iw = a.idx_w + tok * W;
    const float *ww = a.w_w + tok * W;
    const float *un = a.undo + tok * static_cast<long>(W) * d_v + ccol;
    float vh = 0.f, gs = 0.f;
    for (int j = 0; j < W; ++j) {
      const int row = iw[j];
      const bool ok = static_cast<unsigned>(row) < static_cast<unsigned>(N);
      const float m = al * un[static_cast<long>(j) * d_v];
      const float Gj = ok ? G[static_cast<long>(row) * d_v] : 0.f;
      if (MODE == SDM_RESID_SHARED) vh = fmaf(ww[j], m, vh);
      gs = fmaf(ww[j], Gj, gs);
    }
    gs *= be;
    const float res_sh = vc - vh;
    if (active) a.dv[tok * d_v + col] = gs;
    float dbeta = 0.f, dalpha = 0.f;
    for (int j = 0; j < W; ++j) {
      const int row = iw[j];
      const bool ok = static_cast<unsigned>(row) < static_cast<unsigned>(N);
      if (!ok) bad = 1;
      const long o = static_cast<long>(ok ? row : 0) * d_v;
      const float u = un[static_cast<long>(j) * d_v];
      const float m = al * u;
      const float Gj = ok ? G[o] : 0.f;
      const float rho = MODE == SDM_RESID_SHARED ? res_sh : MODE == SDM_RESID_PERSLOT ? vc - m : vc;
      dbeta = fmaf(ww[j] * Gj, rho, dbeta);
      float dw = be * Gj * rho;
      if (MODE == SDM_RESID_SHARED) dw = fmaf(-gs, m, dw);
      const float dm = MODE == SDM_RESID_SHARED ? fmaf(-ww[j], gs, Gj)
                       : MODE == SDM_RESID_PERSLOT ? Gj * (1.f - be * ww[j]) : Gj;
      dalpha = fmaf(dm, u, dalpha);
      if (active && ok) {
        G[o] = al * dm;
        M[o] = u;  // undo: the row as it was before this token
      }
      dw = warp_sum(active ? dw : 0.f);
      if (lane == 0) pt[R + j] = dw;
    }
    dalpha = warp_sum(active ? dalpha : 0.f);
    dbeta = warp_sum(active ? dbeta : 0.f);
    if (lane == 0) {
      pt[R + W] = dalpha;
      pt[R + W + 1] = dbeta;
    }
  }
  if (bad && lane == 0 && a.err) atomicOr(a.err, SDM_DEVERR_INDEX_RANGE);
}

// The same step for W, R <= 16 with every row of a token loaded at once into
// registers (one memory round trip per token instead of one per slot).  A
// write slot whose row is also read by the token takes the read's gradient
// from registers; the gradient rows are stored read slots first, then write
// slots, so a row in both ends with the write slot's value, which includes it.
template <int MODE>
__global__ void __launch_bounds__(128) sparse_backward_kernel16(const BackArgs a) {
  constexpr int S = 16;
  const int lane = threadIdx.x & 31;
  const long gw = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= a.total_warps) return;  // warp-uniform
  const int tile = static_cast<int>(gw % a.tiles);
  const long bh = gw / a.tiles;
  const int h = static_cast<int>(bh % a.H);
  const long b = bh / a.H;
  const int T = a.T, H = a.H, N = a.N, d_v = a.d_v, W = a.W, R = a.R;
  const int col = tile * 32 + lane;
  const bool active = col < d_v;
  const int ccol = active ? col : 0;
  float *M = a.state + bh * static_cast<long>(N) * d_v + ccol;
  float *G = a.dstate + bh * static_cast<long>(N) * d_v + ccol;
  const int np = R + W + 2;
  bool bad = false;
  // slot data: lane k < 16 holds read slot k, lane 16 + k write slot k
  const int ks = lane & 15;
  const bool is_w = lane >= 16;
  const bool has = ks < (is_w ? W : R);
  auto tok_of = [&](int t) { return (b * T + t) * H + h; };

  // Software pipeline over the reversed tokens: the slot ids of token t-2 and
  // the rows, gates, v and dy of token t-1 are loaded while token t is
  // computed.  A lane is the only reader and writer of its column, so a row
  // of token t-1 that token t then stores was prefetched stale (the load came
  // first in program order); those few slots are loaded again after the
  // stores.
  struct Scal { float al, be, vc, dyc; };
  auto load_ids = [&](int t, int &id, float &wt) {
    const long tok = tok_of(t);
    id = has ? (is_w ? a.idx_w[tok * W + ks] : a.idx_r[tok * R + ks]) : -1;
    wt = has ? (is_w ? a.w_w[tok * W + ks] : a.w_r[tok * R + ks]) : 0.f;
  };
  auto load_tok = [&](int t, int id, float (&Mr)[S], float (&Gr)[S], float (&Gw)[S], float (&U)[S], Scal &sc) {
    const long tok = tok_of(t);
    sc.al = a.alpha[tok];
    sc.be = a.beta[tok];
    sc.vc = a.v_bf16 ? bf16_to_f32(static_cast<const uint16_t *>(a.v)[tok * d_v + ccol])
                     : static_cast<const float *>(a.v)[tok * d_v + ccol];
    sc.dyc = a.dy[tok * d_v + ccol];
#pragma unroll
    for (int k = 0; k < S; ++k) {  // every row of the token at once
      const int ri = __shfl_sync(kFull, id, k), wi = __shfl_sync(kFull, id, 16 + k);
      const bool okr = static_cast<unsigned>(ri) < static_cast<unsigned>(N);
      const bool okw = static_cast<unsigned>(wi) < static_cast<unsigned>(N);
      Mr[k] = okr ? M[static_cast<long>(ri) * d_v] : 0.f;
      Gr[k] = okr ? G[static_cast<long>(ri) * d_v] : 0.f;
      Gw[k] = okw ? G[static_cast<long>(wi) * d_v] : 0.f;
      U[k] = k < W ? a.undo[(tok * W + k) * static_cast<long>(d_v) + ccol] : 0.f;
    }
  };
  float Mr[S], Gr[S], Gw[S], U[S], nMr[S], nGr[S], nGw[S], nU[S];
  Scal sc, nsc;
  int my_id = -1, n_id = -1;
  float my_wt = 0.f, n_wt = 0.f;
  if (T > 0) {
    load_ids(T - 1, my_id, my_wt);
    load_tok(T - 1, my_id, Mr, Gr, Gw, U, sc);
  }
  if (T > 1) load_ids(T - 2, n_id, n_wt);

  for (int t = T - 1; t >= 0; --t) {
    const long tok = tok_of(t);
    if (t >= 1) load_tok(t - 1, n_id, nMr, nGr, nGw, nU, nsc);  // next token's rows (prefetch)
    int nn_id = -1;
    float nn_wt = 0.f;
    if (t >= 2) load_ids(t - 2, nn_id, nn_wt);                   // and the ids after it
    const float al = sc.al, be = sc.be, vc = sc.vc, dyc = sc.dyc;
    float *pt = a.part + (static_cast<long>(tile) * (a.total_warps / a.tiles) * T + tok) * np;
    bad |= has && static_cast<unsigned>(my_id) >= static_cast<unsigned>(N);
    // a write lane finds the read slot (if any) with its row
    int my_match = -1;
#pragma unroll
    for (int i = 0; i < S; ++i) {
      const int ri = __shfl_sync(kFull, my_id, i);
      if (is_w && has && ri == my_id) my_match = i;
    }
    // per-lane column partials of the token's sums: [0, 16) dr_i, [16, 32) dw_j
    float part[2 * S];
    // the read after the write
#pragma unroll
    for (int i = 0; i < S; ++i) {
      part[i] = (i < R && active) ? dyc * Mr[i] : 0.f;
      if (i < R) Gr[i] = fmaf(__shfl_sync(kFull, my_wt, i), dyc, Gr[i]);
    }
    // a written row that is also read takes the read gradient (same fma as its read slot)
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const int mi = __shfl_sync(kFull, my_match, 16 + j);
      const float wr = __shfl_sync(kFull, my_wt, mi & 15);
      if (mi >= 0) Gw[j] = fmaf(wr, dyc, Gw[j]);
    }
    // the write
    float vh = 0.f, gs = 0.f;
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const float wj = __shfl_sync(kFull, my_wt, 16 + j);
      if (MODE == SDM_RESID_SHARED) vh = fmaf(wj, al * U[j], vh);
      gs = fmaf(wj, Gw[j], gs);
    }
    gs *= be;
    const float res_sh = vc - vh;
    if (active) a.dv[tok * d_v + col] = gs;
    float dbeta = 0.f, dalpha = 0.f;
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const float wj = __shfl_sync(kFull, my_wt, 16 + j);
      part[S + j] = 0.f;
      if (j < W) {
        const float m = al * U[j];
        const float rho = MODE == SDM_RESID_SHARED ? res_sh : MODE == SDM_RESID_PERSLOT ? vc - m : vc;
        dbeta = fmaf(wj * Gw[j], rho, dbeta);
        float dw = be * Gw[j] * rho;
        if (MODE == SDM_RESID_SHARED) dw = fmaf(-gs, m, dw);
        const float dm = MODE == SDM_RESID_SHARED ? fmaf(-wj, gs, Gw[j])
                         : MODE == SDM_RESID_PERSLOT ? Gw[j] * (1.f - be * wj) : Gw[j];
        dalpha = fmaf(dm, U[j], dalpha);
        Gw[j] = al * dm;
        part[S + j] = active ? dw : 0.f;
      }
    }
    dalpha = warp_sum(active ? dalpha : 0.f);
    dbeta = warp_sum(active ? dbeta : 0.f);
    // reduce-scatter of the 32 partials over the warp (31 shuffles): lane l
    // ends with the column sum of partial l
#pragma unroll
    for (int o = 16, n = 2 * S; o >= 1; o >>= 1, n >>= 1) {
      const bool upper = (lane & o) != 0;
#pragma unroll
      for (int i = 0; i < n / 2; ++i) {
        const float send = upper ? part[i] : part[i + n / 2];
        const float recv = __shfl_xor_sync(kFull, send, o);
        part[i] = (upper ? part[i + n / 2] : part[i]) + recv;
      }
    }
    if (lane < S ? lane < R : lane - S < W) pt[lane < S ? lane : R + lane - S] = part[0];
    if (lane == 0) {
      pt[R + W] = dalpha;
      pt[R + W + 1] = dbeta;
    }
    // stores: read rows, then written rows (gradient and the undone table row),
    // with the streaming hint (evict first) so that L2 stays with the gathers
    // of the tokens still to come (measured: training step 19.77 -> 19.54 ms)
#pragma unroll
    for (int i = 0; i < S; ++i) {
      const int ri = __shfl_sync(kFull, my_id, i);
      if (active && static_cast<unsigned>(ri) < static_cast<unsigned>(N)) __stcs(&G[static_cast<long>(ri) * d_v], Gr[i]);
    }
#pragma unroll
    for (int j = 0; j < S; ++j) {
      const int wi = __shfl_sync(kFull, my_id, 16 + j);
      if (active && static_cast<unsigned>(wi) < static_cast<unsigned>(N)) {
        __stcs(&G[static_cast<long>(wi) * d_v], Gw[j]);
        __stcs(&M[static_cast<long>(wi) * d_v], U[j]);
      }
    }
    if (t >= 1) {
      // slots of token t-1 whose row token t just stored: load them again
      bool hit = false;
#pragma unroll
      for (int k = 0; k < 2 * S; ++k) hit |= __shfl_sync(kFull, my_id, k) == n_id;
      const unsigned stale = __ballot_sync(kFull, hit && static_cast<unsigned>(n_id) < static_cast<unsigned>(N));
      if (stale) {  // warp-uniform
#pragma unroll
        for (int k = 0; k < S; ++k) {
          const int ri = __shfl_sync(kFull, n_id, k), wi = __shfl_sync(kFull, n_id, 16 + k);
          if ((stale >> k) & 1u) {
            nMr[k] = M[static_cast<long>(ri) * d_v];
            nGr[k] = G[static_cast<long>(ri) * d_v];
          }
          if ((stale >> (16 + k)) & 1u) nGw[k] = G[static_cast<long>(wi) * d_v];
        }
      }
#pragma unroll
      for (int k = 0; k < S; ++k) {
        Mr[k] = nMr[k];
        Gr[k] = nGr[k];
        Gw[k] = nGw[k];
        U[k] = nU[k];
      }
      sc = nsc;
      my_id = n_id;
      my_wt = n_wt;
      n_id = nn_id;
      n_wt = nn_wt;
    }
  }
  if (__any_sync(kFull, bad) && lane == 0 && a.err) atomicOr(a.err, SDM_DEVERR_INDEX_RANGE);
}

// Addressing backward (SDM deck, Secs. 2 / 3.1): w = softmax of the W selected
// sums s_i = s1[a_i] + s2[b_i]; ds_i = w_i (dw_i - sum_j w_j dw_j) lands on
// s1[a_i] and s2[b_i], every other score gets 0.  One warp per row; the warp
// zeroes the row, then adds the slots in order (deterministic).
__global__ void __launch_bounds__(256) address_backward_kernel(const int32_t *idx, const float *w, const float *dw,
                                                               long rows, int sqrtN, int W, float *ds1, float *ds2,
                                                               int32_t *err) {
  const int lane = threadIdx.x & 31;
  const long r = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (r >= rows) return;  // warp-uniform
  float *d1 = ds1 + r * sqrtN, *d2 = ds2 + r * sqrtN;
  for (int a = lane; a < sqrtN; a += 32) d1[a] = d2[a] = 0.f;
  float wv[2], dv2[2], ds[2];
  int id[2];
  float dot = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int j = lane + 32 * k;
    const bool in = j < W;
    id[k] = in ? idx[r * W + j] : -1;
    wv[k] = in ? w[r * W + j] : 0.f;
    dv2[k] = in ? dw[r * W + j] : 0.f;
    dot = fmaf(wv[k], dv2[k], dot);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(kFull, dot, o);
#pragma unroll
  for (int k = 0; k < 2; ++k) ds[k] = wv[k] * (dv2[k] - dot);
  __syncwarp();
  bool bad = false;
  for (int j = 0; j < W; ++j) {
    const int k = j >> 5;
    const float g = __shfl_sync(kFull, k ? ds[1] : ds[0], j & 31);
    const int i = __shfl_sync(kFull, k ? id[1] : id[0], j & 31);
    if (lane == 0) {
      if (static_cast<unsigned>(i) < static_cast<unsigned>(sqrtN * sqrtN)) {
        d1[i / sqrtN] += g;
        d2[i % sqrtN] += g;
      } else {
        bad = true;
      }
    }
  }
  if (bad && err) atomicOr(err, SDM_DEVERR_INDEX_RANGE);
}

// sum of the per-tile column sums, tile by tile in order
__global__ void sparse_backward_reduce(const float *part, long rows, int np, int tiles, int W, int R, float *dw_r,
                                       float *dw_w, float *dalpha, float *dbeta) {
  const long i = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= rows * np) return;
  const long tok = i / np;
  const int k = static_cast<int>(i - tok * np);
  float s = 0.f;
  for (int t = 0; t < tiles; ++t) s += part[(static_cast<long>(t) * rows + tok) * np + k];
  if (k < R) dw_r[tok * R + k] = s;
  else if (k < R + W) dw_w[tok * W + (k - R)] = s;
  else if (k == R + W) dalpha[tok] = s;
  else dbeta[tok] = s;
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" size_t sdm_scan_backward_workspace_size(int B, int T, int H, int W, int R, int d_v) {
  if (B <= 0 || T <= 0 || H <= 0 || W <= 0 || R <= 0 || d_v <= 0) return 0;
  const size_t n = static_cast<size_t>((d_v + 31) / 32) * B * T * H * (W + R + 2) * sizeof(float);
  return (n + 255) & ~static_cast<size_t>(255);
}

extern "C" int sdm_scan_backward(float *state, float *dstate, const void *v, int v_dtype, const float *alpha,
                                 const float *beta, const int32_t *idx_w, const float *w_w, int W,
                                 const int32_t *idx_r, const float *w_r, int R, int B, int T, int H, int N, int d_v,
                                 int resid_mode, const float *undo, const float *dy, float *dv, float *dalpha,
                                 float *dbeta, float *dw_w, float *dw_r, void *workspace, size_t workspace_bytes,
                                 int32_t *dev_err, void *stream) {
  if (!state || !dstate || !v || !alpha || !beta || !idx_w || !w_w || !idx_r || !w_r || !undo || !dy || !dv ||
      !dalpha || !dbeta || !dw_w || !dw_r)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan_backward: null pointer");
  if (B < 0 || T < 0 || H < 0 || N < 1 || d_v < 1)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan_backward: bad sizes");
  if (W < 1 || W > 64 || R < 1 || R > 64) return set_error(SDM_ERR_SHAPE, "sdm_scan_backward: need 1 <= W, R <= 64");
  if (v_dtype != SDM_DTYPE_F32 && v_dtype != SDM_DTYPE_BF16)
    return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan_backward: v_dtype must be SDM_DTYPE_F32 or SDM_DTYPE_BF16");
  if (resid_mode != SDM_RESID_SHARED && resid_mode != SDM_RESID_PERSLOT && resid_mode != SDM_RESID_ADDITIVE)
    return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan_backward: unknown resid_mode %d", resid_mode);
  if (!aligned(state, 4) || !aligned(dstate, 4) || !aligned(undo, 4) || !aligned(dy, 4) || !aligned(dv, 4) ||
      (dev_err && !aligned(dev_err, 4)))
    return set_error(SDM_ERR_ALIGN, "sdm_scan_backward: fp32 tensors need 4-byte alignment");
  if (static_cast<double>(B) * T * H >= 2.0e9) return set_error(SDM_ERR_SHAPE, "sdm_scan_backward: B*T*H too large");
  if (B == 0 || T == 0 || H == 0) return SDM_OK;
  const size_t need = sdm_scan_backward_workspace_size(B, T, H, W, R, d_v);
  if (!workspace || workspace_bytes < need)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan_backward: workspace of %zu bytes needed", need);

  BackArgs args;
  args.state = state;
  args.dstate = dstate;
  args.v = v;
  args.alpha = alpha;
  args.beta = beta;
  args.idx_w = idx_w;
  args.idx_r = idx_r;
  args.w_w = w_w;
  args.w_r = w_r;
  args.undo = undo;
  args.dy = dy;
  args.dv = dv;
  args.part = static_cast<float *>(workspace);
  args.err = dev_err;
  args.T = T;
  args.H = H;
  args.N = N;
  args.d_v = d_v;
  args.W = W;
  args.R = R;
  args.mode = resid_mode;
  args.v_bf16 = v_dtype == SDM_DTYPE_BF16;
  args.tiles = (d_v + 31) / 32;
  args.total_warps = static_cast<long>(B) * H * args.tiles;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned blocks = static_cast<unsigned>((args.total_warps + 3) / 4);
  if (W <= 16 && R <= 16) {
    if (resid_mode == SDM_RESID_SHARED) sparse_backward_kernel16<SDM_RESID_SHARED><<<blocks, 128, 0, st>>>(args);
    else if (resid_mode == SDM_RESID_PERSLOT) sparse_backward_kernel16<SDM_RESID_PERSLOT><<<blocks, 128, 0, st>>>(args);
    else sparse_backward_kernel16<SDM_RESID_ADDITIVE><<<blocks, 128, 0, st>>>(args);
  } else {
    if (resid_mode == SDM_RESID_SHARED) sparse_backward_kernel<SDM_RESID_SHARED><<<blocks, 128, 0, st>>>(args);
    else if (resid_mode == SDM_RESID_PERSLOT) sparse_backward_kernel<SDM_RESID_PERSLOT><<<blocks, 128, 0, st>>>(args);
    else sparse_backward_kernel<SDM_RESID_ADDITIVE><<<blocks, 128, 0, st>>>(args);
  }
  int rc = check_launch("sdm_scan_backward: kernel");
  if (rc != SDM_OK) return rc;
  const long rows = static_cast<long>(B) * T * H;
  const int np = W + R + 2;
  const unsigned rb = static_cast<unsigned>((rows * np + 255) / 256);
  sparse_backward_reduce<<<rb, 256, 0, st>>>(args.part, rows, np, args.tiles, W, R, dw_r, dw_w, dalpha, dbeta);
  return check_launch("sdm_scan_backward: reduce kernel");
}

extern "C" int sdm_address_backward(const int32_t *idx, const float *w, const float *dw, int B, int T, int H,
                                    int sqrtN, int W, float *ds1, float *ds2, int32_t *dev_err, void *stream) {
  if (!idx || !w || !dw || !ds1 || !ds2) return set_error(SDM_ERR_INVALID_ARG, "sdm_address_backward: null pointer");
  if (B < 0 || T < 0 || H < 0 || sqrtN < 1) return set_error(SDM_ERR_INVALID_ARG, "sdm_address_backward: bad sizes");
  if (W < 1 || W > 64) return set_error(SDM_ERR_SHAPE, "sdm_address_backward: need 1 <= W <= 64");
  if (static_cast<long>(sqrtN) * sqrtN > INT_MAX) return set_error(SDM_ERR_SHAPE, "sdm_address_backward: sqrtN too large");
  if (!aligned(idx, 4) || !aligned(w, 4) || !aligned(dw, 4) || !aligned(ds1, 4) || !aligned(ds2, 4) ||
      (dev_err && !aligned(dev_err, 4)))
    return set_error(SDM_ERR_ALIGN, "sdm_address_backward: 4-byte alignment needed");
  const long rows = static_cast<long>(B) * T * H;
  if (rows == 0) return SDM_OK;
  address_backward_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      idx, w, dw, rows, sqrtN, W, ds1, ds2, dev_err);
  return check_launch("sdm_address_backward");
}
