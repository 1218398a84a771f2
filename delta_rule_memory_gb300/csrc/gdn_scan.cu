// gdn_scan.cu - dense Gated DeltaNet / KDA scan (Linear Attention Architectures
// deck, "GDN and KDA change the granularity of forgetting", Eqs. 15-20) and
// GDN2 (same deck, "GDN2 separates key-side erase and value-side write",
// Eqs. 21-24): the C ABI entry points, and the token-by-token fp32 kernel used
// for KDA, GDN2 and widths other than d_k = d_v = 128 (dense GDN at 128 x 128
// runs chunkwise on the tensor cores, gdn_chunk.cu).
//
// One CTA per (batch, head, 32-column tile of the value dimension); the
// dk x 32 state tile stays in registers for the whole sequence (thread
// (warp w, lane l) holds rows w, w+8, ... of column l).  Per token: decay the
// rows, reduce the decayed prediction over rows (one barrier), write, and
// reduce the read over rows (reduced by the next token's barrier).  Per-token
// inputs are prefetched P tokens ahead with cp.async.
#include <cstdlib>

#include "common.cuh"

namespace sdm {
namespace {

constexpr int kGdnCols = 32;
constexpr int kGdnWarps = 8;
constexpr int kGdnP = 4;

struct GdnArgs {
  float *state;
  const uint16_t *q, *k, *v;
  const float *alpha, *beta;
  const float *berase, *wwrite;  // GDN2 gates (gdn2 = 1), else unused
  float *y;
  int T, H, dk, dv, per_channel, gdn2, tiles;
};

// per-token slot (32-bit words): k[dk] bf16, q[dk] bf16, v[32] bf16,
// alpha[dk or 1], then beta (GDN, KDA) or b_erase[dk], w_write[32] (GDN2),
// padded to a multiple of 4 words
__host__ __device__ inline int gdn_slot_words(int dk, int gdn2) {
  return (dk + 16 + dk + (gdn2 ? dk + 32 : 1) + 3) & ~3;
}

template <int RPT>  // rows per thread = dk / 8
__global__ void __launch_bounds__(kGdnWarps * 32) gdn_recurrent_kernel(const GdnArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int tile = blockIdx.x % a.tiles;
  const long bh = blockIdx.x / a.tiles;
  const int h = static_cast<int>(bh % a.H);
  const long b = bh / a.H;
  const int dk = a.dk, dv = a.dv, T = a.T, H = a.H;
  const int col = tile * kGdnCols + lane;

  float *redP = reinterpret_cast<float *>(smem_raw);          // [8][32]
  float *redY = redP + kGdnWarps * kGdnCols;                  // [2][8][32]
  uint32_t *ring = reinterpret_cast<uint32_t *>(redY + 2 * kGdnWarps * kGdnCols);
  const int sw = gdn_slot_words(dk, a.gdn2);
  const int k_off = 0, q_off = dk / 2, v_off = dk, a_off = dk + 16, b_off = dk + 16 + dk;
  const int e_off = b_off, w_off = b_off + dk;  // GDN2: erase gate b[dk], write gate w[32 columns]

  float *gS = a.state + bh * static_cast<long>(dk) * dv;
  float s[RPT];
#pragma unroll
  for (int i = 0; i < RPT; ++i) s[i] = gS[static_cast<long>(warp + kGdnWarps * i) * dv + col];

  const long tok0 = b * T * H + h;
  const int n_k = dk / 8, n_q = dk / 8, n_v = kGdnCols / 8, n_a = a.per_channel ? dk / 4 : 0;
  const int n_e = a.gdn2 ? dk / 4 : 0, n_w = a.gdn2 ? kGdnCols / 4 : 0;
  auto issue = [&](int t) {
    const long tok = tok0 + static_cast<long>(t) * H;
    uint32_t *sl = ring + (t % (kGdnP + 1)) * sw;
    const int tid = threadIdx.x;
    int q = tid;
    if (q < n_k) { cp_async<16>(sl + k_off + 4 * q, a.k + tok * dk + 8 * q); return; }
    q -= n_k;
    if (q < n_q) { cp_async<16>(sl + q_off + 4 * q, a.q + tok * dk + 8 * q); return; }
    q -= n_q;
    if (q < n_v) { cp_async<16>(sl + v_off + 4 * q, a.v + tok * dv + tile * kGdnCols + 8 * q); return; }
    q -= n_v;
    if (q < n_a) { cp_async<16>(sl + a_off + 4 * q, a.alpha + tok * dk + 4 * q); return; }
    q -= n_a;
    if (q < n_e) { cp_async<16>(sl + e_off + 4 * q, a.berase + tok * dk + 4 * q); return; }
    q -= n_e;
    if (q < n_w) { cp_async<16>(sl + w_off + 4 * q, a.wwrite + tok * dv + tile * kGdnCols + 4 * q); return; }
    q -= n_w;
    if (a.gdn2) return;
    if (!a.per_channel) {
      if (q == 0) cp_async<4>(sl + a_off, a.alpha + tok);
      else if (q == 1) cp_async<4>(sl + b_off, a.beta + tok);
    } else if (q == 0) {
      cp_async<4>(sl + b_off, a.beta + tok);
    }
  };
  for (int t = 0; t < kGdnP; ++t) {
    if (t < T) issue(t);
    cp_async_commit();
  }

  for (int t = 0; t < T; ++t) {
    cp_async_wait<kGdnP - 1>();
    __syncthreads();
    if (t + kGdnP < T) issue(t + kGdnP);
    cp_async_commit();
    if (t > 0 && warp == 0) {
      const float *rd = redY + ((t - 1) & 1) * kGdnWarps * kGdnCols;
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < kGdnWarps; ++w) acc += rd[w * kGdnCols + lane];
      a.y[(tok0 + static_cast<long>(t - 1) * H) * dv + col] = acc;
    }
    const uint32_t *sl = ring + (t % (kGdnP + 1)) * sw;
    const uint16_t *kk = reinterpret_cast<const uint16_t *>(sl + k_off);
    const uint16_t *qq = reinterpret_cast<const uint16_t *>(sl + q_off);
    const uint16_t *vv = reinterpret_cast<const uint16_t *>(sl + v_off);
    const float *al = reinterpret_cast<const float *>(sl + a_off);
    const float *eb = reinterpret_cast<const float *>(sl + e_off);  // GDN2 erase gate b
    const float *wg = reinterpret_cast<const float *>(sl + w_off);  // GDN2 write gate w
    const float be = a.gdn2 ? 0.f : __uint_as_float(sl[b_off]);
    // decay every row (D_alpha S), then the decayed prediction S~^T k
    // (GDN2: at the erase key e = b (.) k)
    float pp = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int j = warp + kGdnWarps * i;
      const float aj = a.per_channel ? al[j] : al[0];
      const float kj = bf16_to_f32(kk[j]);
      s[i] *= aj;
      pp = fmaf(s[i], a.gdn2 ? eb[j] * kj : kj, pp);
    }
    redP[warp * kGdnCols + lane] = pp;
    __syncthreads();
    float pred = 0.f;
#pragma unroll
    for (int w = 0; w < kGdnWarps; ++w) pred += redP[w * kGdnCols + lane];
    const float vl = bf16_to_f32(vv[lane]);
    const float r = a.gdn2 ? fmaf(wg[lane], vl, -pred) : be * (vl - pred);  // GDN2: w (.) v - pred
    float yp = 0.f;
#pragma unroll
    for (int i = 0; i < RPT; ++i) {
      const int j = warp + kGdnWarps * i;
      s[i] = fmaf(bf16_to_f32(kk[j]), r, s[i]);
      yp = fmaf(s[i], bf16_to_f32(qq[j]), yp);
    }
    redY[(t & 1) * kGdnWarps * kGdnCols + warp * kGdnCols + lane] = yp;
  }
  cp_async_wait<0>();
  __syncthreads();
  if (T > 0 && warp == 0) {
    const float *rd = redY + ((T - 1) & 1) * kGdnWarps * kGdnCols;
    float acc = 0.f;
#pragma unroll
    for (int w = 0; w < kGdnWarps; ++w) acc += rd[w * kGdnCols + lane];
    a.y[(tok0 + static_cast<long>(T - 1) * H) * dv + col] = acc;
  }
#pragma unroll
  for (int i = 0; i < RPT; ++i) gS[static_cast<long>(warp + kGdnWarps * i) * dv + col] = s[i];
}

// one CTA per (batch, head, 32-column tile)
int launch_recurrent(GdnArgs &args, int B, cudaStream_t st, const char *what) {
  args.tiles = args.dv / kGdnCols;
  const size_t smem = sizeof(float) * 3 * kGdnWarps * kGdnCols +
                      sizeof(uint32_t) * (kGdnP + 1) * gdn_slot_words(args.dk, args.gdn2);
  const long blocks = static_cast<long>(B) * args.H * args.tiles;
  switch (args.dk) {
    case 16: gdn_recurrent_kernel<2><<<static_cast<unsigned>(blocks), kGdnWarps * 32, smem, st>>>(args); break;
    case 32: gdn_recurrent_kernel<4><<<static_cast<unsigned>(blocks), kGdnWarps * 32, smem, st>>>(args); break;
    case 64: gdn_recurrent_kernel<8><<<static_cast<unsigned>(blocks), kGdnWarps * 32, smem, st>>>(args); break;
    default: gdn_recurrent_kernel<16><<<static_cast<unsigned>(blocks), kGdnWarps * 32, smem, st>>>(args); break;
  }
  return check_launch(what);
}

}  // namespace

size_t gdn_chunk_workspace_size(int B, int T, int H);
size_t kda_chunk_workspace_size(int B, int T, int H);
int launch_kda_chunk(float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                     const float *beta, const float *b_erase, const float *w_write, int B, int T, int H, float *y,
                     void *workspace, int32_t *err, cudaStream_t st);
int launch_gdn_chunk(float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                     const float *beta, int B, int T, int H, float *y, void *workspace, int32_t *err,
                     cudaStream_t st);

// dense GDN and KDA at d_k = d_v = 128 run chunkwise on the tensor cores;
// every other shape runs token by token.  SDM_GDN_PATH=recurrent forces the
// token-by-token kernel (for cross-checks).
static bool use_chunked(int dk, int dv, int per_channel) {
  (void)per_channel;
  const char *path = getenv("SDM_GDN_PATH");
  const bool want_recurrent = path && path[0] == 'r';
  return dk == 128 && dv == 128 && !want_recurrent;
}

static size_t chunk_workspace_size(int B, int T, int H, int per_channel) {
  return per_channel ? kda_chunk_workspace_size(B, T, H) : gdn_chunk_workspace_size(B, T, H);
}

}  // namespace sdm

using namespace sdm;

extern "C" size_t gdn_scan_workspace_size(int B, int T, int H, int dk, int dv, int per_channel) {
  if (B <= 0 || T <= 0 || H <= 0 || !use_chunked(dk, dv, per_channel)) return 0;
  return chunk_workspace_size(B, T, H, per_channel);
}

extern "C" int gdn_scan(float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                        int per_channel, const float *beta, int B, int T, int H, int dk, int dv, float *y,
                        void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream) {
  if (!state || !q || !k || !v || !alpha || !beta || !y) return set_error(SDM_ERR_INVALID_ARG, "gdn_scan: null pointer");
  if (B < 0 || T < 0 || H < 0) return set_error(SDM_ERR_INVALID_ARG, "gdn_scan: negative size");
  if ((dk != 16 && dk != 32 && dk != 64 && dk != 128) || dv < 32 || dv % 32 != 0 || dv > 256)
    return set_error(SDM_ERR_SHAPE, "gdn_scan: need dk in {16,32,64,128}, dv %% 32 == 0, dv <= 256");
  if (per_channel != 0 && per_channel != 1) return set_error(SDM_ERR_UNSUPPORTED, "gdn_scan: per_channel must be 0/1");
  if (!aligned(state, 16) || !aligned(y, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(alpha, per_channel ? 16 : 4) || !aligned(beta, 4))
    return set_error(SDM_ERR_ALIGN, "gdn_scan: state, y, q, k, v (and KDA alpha) need 16-byte alignment");
  if (B == 0 || T == 0 || H == 0) return SDM_OK;
  if (dev_err && !aligned(dev_err, 4)) return set_error(SDM_ERR_ALIGN, "gdn_scan: dev_err must be 4-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (use_chunked(dk, dv, per_channel)) {
    const size_t need = chunk_workspace_size(B, T, H, per_channel);
    if (!workspace || workspace_bytes < need)
      return set_error(SDM_ERR_INVALID_ARG, "gdn_scan: workspace of %zu bytes needed", need);
    if (!aligned(workspace, 16)) return set_error(SDM_ERR_ALIGN, "gdn_scan: workspace must be 16-byte aligned");
    if (per_channel)
      return launch_kda_chunk(state, q, k, v, alpha, beta, nullptr, nullptr, B, T, H, y, workspace, dev_err, st);
    return launch_gdn_chunk(state, q, k, v, alpha, beta, B, T, H, y, workspace, dev_err, st);
  }
  GdnArgs args{};
  args.state = state;
  args.q = q;
  args.k = k;
  args.v = v;
  args.alpha = alpha;
  args.beta = beta;
  args.y = y;
  args.T = T;
  args.H = H;
  args.dk = dk;
  args.dv = dv;
  args.per_channel = per_channel;
  return launch_recurrent(args, B, st, "gdn_scan");
}

extern "C" size_t gdn2_scan_workspace_size(int B, int T, int H, int dk, int dv) {
  if (B <= 0 || T <= 0 || H <= 0 || !use_chunked(dk, dv, 1)) return 0;
  return kda_chunk_workspace_size(B, T, H);
}

extern "C" int gdn2_scan(float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                         const float *b_erase, const float *w_write, int B, int T, int H, int dk, int dv, float *y,
                         void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream) {
  if (!state || !q || !k || !v || !alpha || !b_erase || !w_write || !y)
    return set_error(SDM_ERR_INVALID_ARG, "gdn2_scan: null pointer");
  if (B < 0 || T < 0 || H < 0) return set_error(SDM_ERR_INVALID_ARG, "gdn2_scan: negative size");
  if ((dk != 16 && dk != 32 && dk != 64 && dk != 128) || dv < 32 || dv % 32 != 0 || dv > 256)
    return set_error(SDM_ERR_SHAPE, "gdn2_scan: need dk in {16,32,64,128}, dv %% 32 == 0, dv <= 256");
  if (!aligned(state, 16) || !aligned(y, 16) || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(alpha, 16) || !aligned(b_erase, 16) || !aligned(w_write, 16))
    return set_error(SDM_ERR_ALIGN, "gdn2_scan: every tensor needs 16-byte alignment");
  if (B == 0 || T == 0 || H == 0) return SDM_OK;
  if (dev_err && !aligned(dev_err, 4)) return set_error(SDM_ERR_ALIGN, "gdn2_scan: dev_err must be 4-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (use_chunked(dk, dv, 1)) {
    const size_t need = kda_chunk_workspace_size(B, T, H);
    if (!workspace || workspace_bytes < need)
      return set_error(SDM_ERR_INVALID_ARG, "gdn2_scan: workspace of %zu bytes needed", need);
    if (!aligned(workspace, 16)) return set_error(SDM_ERR_ALIGN, "gdn2_scan: workspace must be 16-byte aligned");
    return launch_kda_chunk(state, q, k, v, alpha, nullptr, b_erase, w_write, B, T, H, y, workspace, dev_err, st);
  }
  GdnArgs args{};
  args.state = state;
  args.q = q;
  args.k = k;
  args.v = v;
  args.alpha = alpha;
  args.berase = b_erase;
  args.wwrite = w_write;
  args.y = y;
  args.T = T;
  args.H = H;
  args.dk = dk;
  args.dv = dv;
  args.per_channel = 1;
  args.gdn2 = 1;
  return launch_recurrent(args, B, st, "gdn2_scan");
}
