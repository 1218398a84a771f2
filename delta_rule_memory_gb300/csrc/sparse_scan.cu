// sparse_scan.cu - the sparse delta-rule memory scan (Sparse Delta Memory
// deck, "Selected slots decay and update; other slots persist", Eqs. 3-5, and
// "A v1 inconsistency matters for reproducing the update", Fig. 2).
//
// The table is HBM-resident fp32 [B,H,N,d_v]; every token gathers its write
// and read rows, decays and updates the written ones, scatters them back and
// reads.  Every value column evolves independently (the addresses do not
// depend on the table), so the work splits into (batch, head, 32-column tile)
// slices, one warp each, with no synchronisation between warps.
//
// Inside a warp, lane = q + 8 r: q picks a float4 column quad of the tile, r a
// row subgroup; lane (q, r) owns write slots and read slots r, r+4, r+8, ...
// of every token.  It copies exactly those row quads (cp.async, 16 bytes),
// decays and updates them; the shared prediction v_hat and the read y are
// summed over the four subgroups with two xor-shuffles.
//
// The rows of token t+P are prefetched while token t is computed.  A row that
// one of the last P tokens wrote is stale in that prefetch, so a prepass
// kernel writes, for every token, one packed record (slot ids, weights, gates,
// and for every slot the shared-memory row to take it from: the prefetched
// copy, a row of the post-write history ring, or - for a read of a row this
// token writes - "recompute").  Records are laid out so a lane reads its own
// slots with 16-byte loads.
#include <climits>
#include <cstdlib>
#include <mutex>

#include "common.cuh"

namespace sdm {
namespace {

// source codes of a slot (see above)
constexpr uint16_t kSrcIncoming = 0x8000;   // the prefetched copy of this slot's row
constexpr uint16_t kSrcZero = 0xffff;       // padding or out-of-range index: zero row, no store
constexpr uint16_t kSrcRecompute = 0x4000;  // | s: read of write slot s of the same token
// otherwise: row ((t - d) % (P + 1)) * SLOTS + s of the history ring

// Packed per-token record, 16-byte aligned.  Slot positions are permuted so
// lane subgroup r finds its 2*RPL slots (RPL write then RPL read) contiguous:
// position r*2*RPL + k is write slot r + 4k (k < RPL) or read slot
// r + 4(k - RPL) (k >= RPL).
template <int SLOTS>
struct alignas(16) TokenRec {
  int32_t idx[2 * SLOTS];
  float w[2 * SLOTS];
  uint16_t src[2 * SLOTS];
  float alpha, beta;
  float pad[2];
};

template <int SLOTS>
__host__ __device__ constexpr size_t rec_bytes() { return sizeof(TokenRec<SLOTS>); }

__host__ __device__ inline int pick_slots(int W, int R) { return (W <= 16 && R <= 16) ? 16 : 64; }

// ---------------------------------------------------------------------------
// Prepass: one thread per (token, record position).
// ---------------------------------------------------------------------------
template <int SLOTS>
__global__ void record_kernel(const int32_t *__restrict__ idx_w, const float *__restrict__ w_w,
                              const int32_t *__restrict__ idx_r, const float *__restrict__ w_r,
                              const float *__restrict__ alpha, const float *__restrict__ beta, int W, int R, int T,
                              int H, int N, int window, long total, TokenRec<SLOTS> *__restrict__ rec,
                              int32_t *__restrict__ dev_err) {
  constexpr int RPL = SLOTS / 4;
  const long tid = static_cast<long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (tid >= total) return;
  const long tok = tid / (2 * SLOTS);
  const int pos = static_cast<int>(tid - tok * 2 * SLOTS);
  const int r = pos / (2 * RPL), k = pos % (2 * RPL);
  const bool is_w = k < RPL;
  const int j = r + 4 * (is_w ? k : k - RPL);
  const int t = static_cast<int>((tok / H) % T);
  TokenRec<SLOTS> &o = rec[tok];
  if (pos == 0) {
    o.alpha = alpha[tok];
    o.beta = beta[tok];
    o.pad[0] = o.pad[1] = 0.f;
  }
  const int n = is_w ? W : R;
  if (j >= n) {  // padding slot
    o.idx[pos] = -1;
    o.w[pos] = 0.f;
    o.src[pos] = kSrcZero;
    return;
  }
  const int my = is_w ? idx_w[tok * W + j] : idx_r[tok * R + j];
  o.idx[pos] = my;
  o.w[pos] = is_w ? w_w[tok * W + j] : w_r[tok * R + j];
  int err = 0;
  uint16_t code = kSrcIncoming;
  if (my < 0 || my >= N) {
    code = kSrcZero;
    err |= SDM_DEVERR_INDEX_RANGE;
  } else {
    if (is_w) {
      for (int jj = 0; jj < j; ++jj)
        if (idx_w[tok * W + jj] == my) err |= SDM_DEVERR_INDEX_REPEAT;
    }
    const int dmax = min(window, t);
    for (int d = is_w ? 1 : 0; d <= dmax && code == kSrcIncoming; ++d) {
      const int32_t *lst = idx_w + (tok - static_cast<long>(d) * H) * W;
      for (int s = W - 1; s >= 0; --s) {
        if (lst[s] == my) {
          code = d == 0 ? static_cast<uint16_t>(kSrcRecompute | s)
                        : static_cast<uint16_t>(((t - d) % (window + 1)) * SLOTS + s);
          break;
        }
      }
    }
  }
  o.src[pos] = code;
  if (err && dev_err) atomicOr(dev_err, err);
}

// ---------------------------------------------------------------------------
// The scan.
// ---------------------------------------------------------------------------
struct ScanArgs {
  float *state;
  const void *v;
  const void *rec;
  float *y;
  int T, H, N, d_v, v_bf16, tiles;
  long total_warps;
};

template <int P, int SLOTS>
struct ScanLayout {
  static constexpr int NI = P + 1;      // incoming rows: P in flight + current
  static constexpr int NH = P + 1;      // post-write history: current + P back
  static constexpr int NM = 2 * P + 1;  // records: needed from t-P (row issue) to t
  static constexpr size_t kSlotBytes = static_cast<size_t>(SLOTS) * 32 * sizeof(float);
  static constexpr size_t kRecOff = 3 * NI * kSlotBytes;  // inW, hist, inR rings
  static constexpr size_t kVOff = kRecOff + NM * rec_bytes<SLOTS>();
  static constexpr size_t kZeroOff = kVOff + NM * 128;      // 32 columns of v per record, fp32 or bf16
  static constexpr size_t kWarpBytes = kZeroOff + 128;      // one all-zero 32-float row
};

__device__ __forceinline__ float4 ld4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ void st4(float *p, float4 x) { *reinterpret_cast<float4 *>(p) = x; }
__device__ __forceinline__ float4 fma4(float s, float4 x, float4 c) {
  return make_float4(fmaf(s, x.x, c.x), fmaf(s, x.y, c.y), fmaf(s, x.z, c.z), fmaf(s, x.w, c.w));
}
__device__ __forceinline__ float4 mul4(float s, float4 x) { return make_float4(s * x.x, s * x.y, s * x.z, s * x.w); }
__device__ __forceinline__ float4 sub4(float4 a, float4 b) {
  return make_float4(a.x - b.x, a.y - b.y, a.z - b.z, a.w - b.w);
}
__device__ __forceinline__ float4 xsum4(float4 a) {  // sum over the four row subgroups (lane bits 3, 4)
#pragma unroll
  for (int m = 8; m <= 16; m <<= 1) {
    a.x += __shfl_xor_sync(kFull, a.x, m);
    a.y += __shfl_xor_sync(kFull, a.y, m);
    a.z += __shfl_xor_sync(kFull, a.z, m);
    a.w += __shfl_xor_sync(kFull, a.w, m);
  }
  return a;
}

template <int P, int SLOTS, int MODE>
__global__ void __launch_bounds__(128) sparse_scan_kernel(const ScanArgs a) {
  using L = ScanLayout<P, SLOTS>;
  using Rec = TokenRec<SLOTS>;
  constexpr int RPL = SLOTS / 4;
  constexpr int SLOT_F = SLOTS * 32;  // floats per ring slot
  constexpr int REC_CHUNKS = static_cast<int>(sizeof(Rec) / 16);
  static_assert(REC_CHUNKS + 8 <= 32 || SLOTS == 64, "one copy per lane for the 16-slot record");
  extern __shared__ __align__(16) unsigned char smem_raw[];

  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const long gw = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + wib;
  if (gw >= a.total_warps) return;  // warp-uniform; no CTA-wide barrier below
  const int tile = static_cast<int>(gw % a.tiles);
  const long bh = gw / a.tiles;
  const int h = static_cast<int>(bh % a.H);
  const long b = bh / a.H;
  const int T = a.T, H = a.H, d_v = a.d_v;
  const int q = lane & 7, r = lane >> 3;
  const int col = tile * 32 + 4 * q;
  const bool active = col < d_v;

  unsigned char *base = smem_raw + static_cast<size_t>(wib) * L::kWarpBytes;
  float *inW = reinterpret_cast<float *>(base);
  float *hist = inW + L::NI * SLOT_F;
  float *inR = hist + L::NH * SLOT_F;
  Rec *recs = reinterpret_cast<Rec *>(base + L::kRecOff);
  uint32_t *vbuf = reinterpret_cast<uint32_t *>(base + L::kVOff);  // [NM][32 words]
  float *zrow = reinterpret_cast<float *>(base + L::kZeroOff);
  zrow[lane] = 0.f;

  float *table = a.state + bh * static_cast<long>(a.N) * d_v + col;  // this lane's quad of row 0
  const long tok0 = b * T * H + h;
  const Rec *grec = static_cast<const Rec *>(a.rec);
  const int lq = 4 * q;  // this lane's column offset inside a 32-float ring row

  // per token: the record (REC_CHUNKS x 16 B) and 32 columns of v
  // (8 x 8 B of bf16 or 8 x 16 B of fp32); one copy per lane
  auto issue_meta = [&](int t) {
    const long tok = tok0 + static_cast<long>(t) * H;
    const int slot = t % L::NM;
    for (int c = lane; c < REC_CHUNKS + 8; c += 32) {
      if (c < REC_CHUNKS) {
        cp_async<16>(reinterpret_cast<unsigned char *>(recs + slot) + 16 * c,
                     reinterpret_cast<const unsigned char *>(grec + tok) + 16 * c);
      } else {
        const int vc = c - REC_CHUNKS;  // columns 4vc .. 4vc+3
        if (tile * 32 + 4 * vc < d_v) {
          if (a.v_bf16)
            cp_async<8>(vbuf + slot * 32 + 2 * vc, static_cast<const uint16_t *>(a.v) + tok * d_v + tile * 32 + 4 * vc);
          else
            cp_async<16>(vbuf + slot * 32 + 4 * vc, static_cast<const float *>(a.v) + tok * d_v + tile * 32 + 4 * vc);
        }
      }
    }
  };
  // the row quads this lane consumes: write slots r+4k into inW, read slots into inR
  auto issue_rows = [&](int t) {
    if (!active) return;
    const Rec &m = recs[t % L::NM];
    int id[2 * RPL];
#pragma unroll
    for (int k = 0; k < 2 * RPL; k += 4) {
      const int4 x = *reinterpret_cast<const int4 *>(m.idx + r * 2 * RPL + k);
      id[k] = x.x; id[k + 1] = x.y; id[k + 2] = x.z; id[k + 3] = x.w;
    }
    float *dw = inW + (t % L::NI) * SLOT_F + lq;
    float *dr = inR + (t % L::NI) * SLOT_F + lq;
#pragma unroll
    for (int k = 0; k < 2 * RPL; ++k) {
      const int i = id[k];
      const int j = r + 4 * (k < RPL ? k : k - RPL);
      if (static_cast<unsigned>(i) < static_cast<unsigned>(a.N))
        cp_async<16>((k < RPL ? dw : dr) + j * 32, table + static_cast<long>(i) * d_v);
    }
  };

  // prologue: records of tokens [0, P), then P groups (rows of j, record of j+P)
  for (int t = 0; t < P && t < T; ++t) issue_meta(t);
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  for (int j = 0; j < P; ++j) {
    if (j + P < T) issue_meta(j + P);
    if (j < T) issue_rows(j);
    cp_async_commit();
  }

  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int t = 0; t < T; ++t) {
    cp_async_wait<P - 1>();
    __syncwarp();
    if (t + 2 * P < T) issue_meta(t + 2 * P);
    if (t + P < T) issue_rows(t + P);
    cp_async_commit();

    const Rec &m = recs[t % L::NM];
    const float al = m.alpha, be = m.beta;
    const uint32_t *vw = vbuf + (t % L::NM) * 32;
    float4 vv;
    if (a.v_bf16) {
      const uint32_t w0 = vw[2 * q], w1 = vw[2 * q + 1];
      vv = make_float4(bf16_to_f32(w0 & 0xffff), bf16_to_f32(w0 >> 16), bf16_to_f32(w1 & 0xffff),
                       bf16_to_f32(w1 >> 16));
    } else {
      vv = make_float4(__uint_as_float(vw[4 * q]), __uint_as_float(vw[4 * q + 1]), __uint_as_float(vw[4 * q + 2]),
                       __uint_as_float(vw[4 * q + 3]));
    }
    const float *cur_w = inW + (t % L::NI) * SLOT_F + lq;
    const float *cur_r = inR + (t % L::NI) * SLOT_F + lq;
    float *cur_h = hist + (t % L::NH) * SLOT_F + lq;
    // this lane's 2*RPL slots: ids, weights and source codes, vector loads
    int my_idx[RPL];
    float my_w[2 * RPL];
    uint16_t my_src[2 * RPL];
#pragma unroll
    for (int k = 0; k < RPL; k += 4) {
      const int4 x = *reinterpret_cast<const int4 *>(m.idx + r * 2 * RPL + k);
      my_idx[k] = x.x; my_idx[k + 1] = x.y; my_idx[k + 2] = x.z; my_idx[k + 3] = x.w;
    }
#pragma unroll
    for (int k = 0; k < 2 * RPL; k += 4) {
      const float4 x = *reinterpret_cast<const float4 *>(m.w + r * 2 * RPL + k);
      my_w[k] = x.x; my_w[k + 1] = x.y; my_w[k + 2] = x.z; my_w[k + 3] = x.w;
    }
#pragma unroll
    for (int k = 0; k < 2 * RPL; k += 8) {
      const uint4 x = *reinterpret_cast<const uint4 *>(m.src + r * 2 * RPL + k);
      const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        my_src[k + 2 * e] = static_cast<uint16_t>(u[e] & 0xffff);
        my_src[k + 2 * e + 1] = static_cast<uint16_t>(u[e] >> 16);
      }
    }
    // shared-memory address of the row a slot starts from (branch-free):
    // the prefetched copy, a history row, or the zero row
    auto row_addr = [&](uint16_t code, const float *incoming) -> const float * {
      const float *hrow = hist + (code < L::NH * SLOTS ? code : 0) * 32 + lq;
      return code == kSrcIncoming ? incoming : (code == kSrcZero ? zrow + lq : hrow);
    };

    // selective decay of the written rows and the shared prediction (Fig. 2)
    float4 md[RPL];
    float4 vh = zero4;
#pragma unroll
    for (int k = 0; k < RPL; ++k) md[k] = ld4(row_addr(my_src[k], cur_w + (r + 4 * k) * 32));
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      md[k] = mul4(al, md[k]);
      if (MODE == SDM_RESID_SHARED) vh = fma4(my_w[k], md[k], vh);
    }
    // read rows (prefetched, history, or zero); reads of a row this token
    // writes are patched below
    float4 xr[RPL];
    bool recomp = false;
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const uint16_t code = my_src[RPL + k];
      const bool rc = code != kSrcIncoming && code != kSrcZero && (code & kSrcRecompute);
      recomp |= rc;
      xr[k] = ld4(rc ? zrow + lq : row_addr(code, cur_r + (r + 4 * k) * 32));
    }
    float4 base4 = vv;
    if (MODE == SDM_RESID_SHARED) base4 = sub4(vv, xsum4(vh));
    auto new_row = [&](float4 mdk, float gk) -> float4 {
      return fma4(gk, MODE == SDM_RESID_PERSLOT ? sub4(vv, mdk) : base4, mdk);
    };

    // delta write: history ring (forwarding source) and the table in HBM
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const float4 nw = new_row(md[k], be * my_w[k]);
      st4(cur_h + (r + 4 * k) * 32, nw);
      const int i = my_idx[k];
      if (active && static_cast<unsigned>(i) < static_cast<unsigned>(a.N))
        st4(table + static_cast<long>(i) * d_v, nw);
    }
    // rare: a read of a row written by this same token -> recompute its new value
    if (__any_sync(kFull, recomp)) {
#pragma unroll
      for (int k = 0; k < RPL; ++k) {
        const uint16_t code = my_src[RPL + k];
        if (code != kSrcIncoming && code != kSrcZero && (code & kSrcRecompute)) {
          const int s = code & 0xff;                     // write slot s of this token
          const int ps = (s & 3) * 2 * RPL + (s >> 2);   // its record position
          const float4 x0 = ld4(row_addr(m.src[ps], cur_w + s * 32));
          xr[k] = new_row(mul4(al, x0), be * m.w[ps]);
        }
      }
    }
    // read after the write
    float4 yp = zero4;
#pragma unroll
    for (int k = 0; k < RPL; ++k) yp = fma4(my_w[RPL + k], xr[k], yp);
    yp = xsum4(yp);
    if (r == 0 && active) st4(a.y + (tok0 + static_cast<long>(t) * H) * d_v + col, yp);
  }
  cp_async_wait<0>();
}

int env_int(const char *name, int dflt) {
  const char *s = getenv(name);
  return (s && *s) ? atoi(s) : dflt;
}

template <int P, int SLOTS>
size_t warp_bytes() { return ScanLayout<P, SLOTS>::kWarpBytes; }

size_t warp_bytes_dispatch(int slots, int P) {
  if (slots == 16) return P == 4 ? warp_bytes<4, 16>() : P == 6 ? warp_bytes<6, 16>() : warp_bytes<8, 16>();
  return P == 4 ? warp_bytes<4, 64>() : 0;
}

template <int P, int SLOTS, int MODE>
int launch_scan(const ScanArgs &args, int wpc, cudaStream_t st) {
  const size_t smem = ScanLayout<P, SLOTS>::kWarpBytes * wpc;
  auto kern = sparse_scan_kernel<P, SLOTS, MODE>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return check_launch("sdm_scan: set shared memory");
  const long blocks = (args.total_warps + wpc - 1) / wpc;
  kern<<<static_cast<unsigned>(blocks), wpc * 32, smem, st>>>(args);
  return check_launch("sdm_scan: scan kernel");
}

template <int P, int SLOTS>
int launch_mode(int mode, const ScanArgs &args, int wpc, cudaStream_t st) {
  if (mode == SDM_RESID_SHARED) return launch_scan<P, SLOTS, SDM_RESID_SHARED>(args, wpc, st);
  if (mode == SDM_RESID_PERSLOT) return launch_scan<P, SLOTS, SDM_RESID_PERSLOT>(args, wpc, st);
  return launch_scan<P, SLOTS, SDM_RESID_ADDITIVE>(args, wpc, st);
}

int launch_dispatch(int slots, int P, int mode, const ScanArgs &args, int wpc, cudaStream_t st) {
  if (slots == 16 && P == 4) return launch_mode<4, 16>(mode, args, wpc, st);
  if (slots == 16 && P == 6) return launch_mode<6, 16>(mode, args, wpc, st);
  if (slots == 16 && P == 8) return launch_mode<8, 16>(mode, args, wpc, st);
  if (slots == 64 && P == 4) return launch_mode<4, 64>(mode, args, wpc, st);
  return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan: no kernel for slots=%d window=%d", slots, P);
}

size_t record_bytes(int W, int R) { return pick_slots(W, R) == 16 ? rec_bytes<16>() : rec_bytes<64>(); }

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" size_t sdm_scan_workspace_size(int B, int T, int H, int W, int R) {
  if (B <= 0 || T <= 0 || H <= 0 || W <= 0 || R <= 0 || W > 64 || R > 64) return 0;
  const size_t n = static_cast<size_t>(B) * T * H * record_bytes(W, R);
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
  if (!aligned(state, 16) || !aligned(y, 16) || !aligned(v, v_dtype == SDM_DTYPE_F32 ? 16 : 8) ||
      !aligned(alpha, 4) || !aligned(beta, 4) || !aligned(idx_w, 4) || !aligned(w_w, 4) || !aligned(idx_r, 4) ||
      !aligned(w_r, 4) || (dev_err && !aligned(dev_err, 4)))
    return set_error(SDM_ERR_ALIGN, "sdm_scan: state, y (and fp32 v) need 16-byte alignment, bf16 v 8-byte, "
                                    "the rest 4-byte");
  if (static_cast<double>(B) * T * H >= 2.0e9) return set_error(SDM_ERR_SHAPE, "sdm_scan: B*T*H too large");
  if (B == 0 || T == 0 || H == 0) return SDM_OK;
  const size_t need = sdm_scan_workspace_size(B, T, H, W, R);
  if (!workspace || workspace_bytes < need)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan: workspace of %zu bytes needed", need);
  if (!aligned(workspace, 16)) return set_error(SDM_ERR_ALIGN, "sdm_scan: workspace must be 16-byte aligned");

  // Launch shape: B*H*ceil(d_v/32) independent warps.  Each runs the whole
  // sequence, so all must be resident at once; take the deepest prefetch
  // window whose shared-memory rings still let every warp fit in one wave.
  const int slots = pick_slots(W, R);
  int dev = 0, smem_blk = 0, smem_sm = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = (d_v + 31) / 32;
  const long total_warps = static_cast<long>(B) * H * tiles;
  const int want_window = env_int("SDM_SCAN_WINDOW", 0);
  int window = 0, wpc = 1;
  for (int p : {8, 6, 4}) {
    if (want_window && p != want_window) continue;
    const size_t wb = warp_bytes_dispatch(slots, p);
    if (wb == 0 || wb > static_cast<size_t>(smem_blk)) continue;
    for (int c : {4, 2, 1}) {  // warps per CTA
      if (c * wb > static_cast<size_t>(smem_blk)) continue;
      const long ctas_sm = static_cast<long>(smem_sm) / static_cast<long>(c * wb + 1024);
      if (window == 0) { window = p; wpc = c; }  // fallback: the first that fits at all
      if (ctas_sm >= 1 && total_warps <= ctas_sm * c * sms) { window = p; wpc = c; goto chosen; }
    }
  }
chosen:
  if (window == 0) return set_error(SDM_ERR_SHAPE, "sdm_scan: W/R too large for shared memory");
  wpc = env_int("SDM_SCAN_WARPS", wpc);
  if (wpc < 1 || static_cast<size_t>(wpc) * warp_bytes_dispatch(slots, window) > static_cast<size_t>(smem_blk))
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan: SDM_SCAN_WARPS does not fit");

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long total = static_cast<long>(B) * T * H * 2 * slots;
  const unsigned rblocks = static_cast<unsigned>((total + 255) / 256);
  if (slots == 16)
    record_kernel<16><<<rblocks, 256, 0, st>>>(idx_w, w_w, idx_r, w_r, alpha, beta, W, R, T, H, N, window, total,
                                               static_cast<TokenRec<16> *>(workspace), dev_err);
  else
    record_kernel<64><<<rblocks, 256, 0, st>>>(idx_w, w_w, idx_r, w_r, alpha, beta, W, R, T, H, N, window, total,
                                               static_cast<TokenRec<64> *>(workspace), dev_err);
  int rc = check_launch("sdm_scan: record kernel");
  if (rc != SDM_OK) return rc;

  ScanArgs args;
  args.state = state;
  args.v = v;
  args.rec = workspace;
  args.y = y;
  args.T = T;
  args.H = H;
  args.N = N;
  args.d_v = d_v;
  args.v_bf16 = v_dtype == SDM_DTYPE_BF16;
  args.tiles = tiles;
  args.total_warps = total_warps;
  return launch_dispatch(slots, window, resid_mode, args, wpc, st);
}

// ---------------------------------------------------------------------------
// sdm_scan_noalloc: sdm_scan for callers that cannot hand over device scratch
// memory.  The per-token records live in a fixed, file-scope device array instead
// of a caller workspace.  Host code cannot use the array's name as a device
// address, so the address is looked up once per device with
// cudaGetSymbolAddress (with that device current) and cached; the first call
// on a device does this lookup, so make that first call before capturing any
// stream.  Every call shares the one array: calls that can overlap on the GPU
// (different streams, or several host threads) race on it and must be
// serialised by the caller.  Every call rewrites all the records it reads, so
// nothing has to be cleared between calls.
// ---------------------------------------------------------------------------
namespace sdm {
namespace {
constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB per device
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
