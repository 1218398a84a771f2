// sparse_scan.cu - the sparse delta-rule memory scan (Sparse Delta Memory
// deck, "Selected slots decay and update; other slots persist", Eqs. 3-5, and
// "A v1 inconsistency matters for reproducing the update", Fig. 2).
//
// The table is HBM-resident fp32 [B,H,N,d_v]; every token gathers its write
// and read rows, decays and updates the written ones, scatters them back and
// reads.  Every value column evolves independently (the addresses do not
// depend on the table), so the work splits into (batch, head, column tile)
// slices of TW = 32 or 16 columns, one warp each, with no synchronisation
// between warps (16-column tiles double the warps for small batches).
//
// Inside a warp, lane = q + Q r with Q = TW/4: q picks a float4 column quad of
// the tile, r one of RG = 32/Q row subgroups; lane (q, r) owns write slots and
// read slots r, r+RG, r+2RG, ... of every token.  It copies exactly those row
// quads (cp.async, 16 bytes), decays and updates them; the shared prediction
// v_hat and the read y are summed over the subgroups with xor-shuffles.
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
#include <cuda.h>
#include <mutex>

#include "common.cuh"

namespace sdm {
namespace {

// A slot's source is stored as the number of a tile row (TW floats) of the
// warp's shared memory, numbered across the rings of ScanLayout: the
// prefetched copy, a post-write history row or the zero row.  A read of a
// row the same token writes is kRecompute | write slot.
constexpr uint16_t kRecompute = 0x8000;

// Packed per-token record, 16-byte aligned.  Slot positions are permuted so
// lane subgroup r finds its 2*RPL slots (RPL write then RPL read) contiguous:
// position r*2*RPL + k is write slot r + RG k (k < RPL) or read slot
// r + RG (k - RPL) (k >= RPL), RG the number of row subgroups of the tile.
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

// Column tile of a warp: TW columns as Q float4 quads, RG row subgroups.
template <int TW>
struct Tile {
  static_assert(TW == 16 || TW == 32, "16- or 32-column tiles");
  static constexpr int Q = TW / 4;
  static constexpr int RG = 32 / Q;
  static constexpr int RB = TW * 4;  // bytes of one tile row
};

template <int P, int SLOTS, int TW>
struct ScanLayout {
  static constexpr int RB = Tile<TW>::RB;
  static constexpr int NI = P + 1;      // incoming rows: P in flight + current
  static constexpr int NH = P + 1;      // post-write history: current + P back
  static constexpr int NM = 2 * P + 1;  // records: needed from t-P (row issue) to t
  // tile-row numbers of the rings
  static constexpr int kRowW = 0;                    // incoming write rows [NI][SLOTS]
  static constexpr int kRowH = NI * SLOTS;           // history [NH][SLOTS]
  static constexpr int kRowR = (NI + NH) * SLOTS;    // incoming read rows [NI][SLOTS]
  static constexpr int kRowZero = (2 * NI + NH) * SLOTS;
  static constexpr size_t kRecOff = static_cast<size_t>(kRowZero + 1) * RB;
  static constexpr size_t kVOff = kRecOff + NM * rec_bytes<SLOTS>();
  static constexpr size_t kWarpBytes = kVOff + NM * RB;  // TW columns of v per record, fp32 or bf16
  static_assert(kRowZero < kRecompute, "row numbers must stay below the recompute flag");
  static_assert(kRecOff % 16 == 0 && kVOff % 16 == 0 && kWarpBytes % 16 == 0, "16-byte aligned regions");
};


// ---------------------------------------------------------------------------
// Prepass: resolves, for every slot, which shared-memory row the scan warp
// reads it from at token t: write slot j -> its prefetched copy, or the
// history row of the most recent earlier token (within the prefetch window P)
// that wrote the same table row; read slot j -> likewise, or kRecompute | s
// when write slot s of the same token holds the row; out-of-range ids and
// padding -> the zero row.  A CTA takes TB consecutive tokens of one (batch,
// head), one thread per (token, record position), and first stages the write
// lists of tokens t0 - P .. t0 + TB - 1 in shared memory, so every hazard
// search reads shared memory only.
// ---------------------------------------------------------------------------
constexpr int kRecThreads = 256;

template <int P, int SLOTS, int TW>
__global__ void __launch_bounds__(kRecThreads) record_kernel(
    const int32_t *__restrict__ idx_w, const float *__restrict__ w_w, const int32_t *__restrict__ idx_r,
    const float *__restrict__ w_r, const float *__restrict__ alpha, const float *__restrict__ beta, int W, int R,
    int T, int H, int N, int t_blocks, TokenRec<SLOTS> *__restrict__ rec, int32_t *__restrict__ dev_err) {
  using L = ScanLayout<P, SLOTS, TW>;
  constexpr int RG = Tile<TW>::RG;
  constexpr int RPL = SLOTS / RG;
  constexpr int PPOS = 2 * SLOTS;            // record positions per token
  constexpr int TB = kRecThreads / PPOS;     // tokens per CTA
  constexpr int NROW = TB + P;               // staged write lists
  __shared__ __align__(16) int32_t sw[NROW * SLOTS];
  const long bh = blockIdx.x / t_blocks;
  const int t0 = static_cast<int>(blockIdx.x - bh * t_blocks) * TB;
  const long b = bh / H;
  const int h = static_cast<int>(bh - b * H);
  for (int id = threadIdx.x; id < NROW * SLOTS; id += kRecThreads) {
    const int tt = t0 - P + id / SLOTS, s = id % SLOTS;
    int32_t x = -1;  // matches no valid id
    if (tt >= 0 && tt < T && s < W) x = idx_w[((b * T + tt) * H + h) * W + s];
    sw[id] = x;
  }
  __syncthreads();
  const int tl = threadIdx.x / PPOS, pos = threadIdx.x % PPOS;
  const int t = t0 + tl;
  if (t >= T) return;
  const long tok = (b * T + t) * H + h;
  const int r = pos / (2 * RPL), k = pos % (2 * RPL);
  const bool is_w = k < RPL;
  const int j = r + RG * (is_w ? k : k - RPL);
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
    o.src[pos] = static_cast<uint16_t>(L::kRowZero);
    return;
  }
  const int32_t *own = sw + (tl + P) * SLOTS;
  const int my = is_w ? own[j] : idx_r[tok * R + j];
  o.idx[pos] = my;
  o.w[pos] = is_w ? w_w[tok * W + j] : w_r[tok * R + j];
  int err = 0;
  int code = is_w ? L::kRowW + (t % L::NI) * SLOTS + j : L::kRowR + (t % L::NI) * SLOTS + j;
  if (my < 0 || my >= N) {
    code = L::kRowZero;
    err |= SDM_DEVERR_INDEX_RANGE;
  } else {
    // the nearest earlier writer: smallest distance d, then the largest slot
    // s; walking d downwards and s upwards, the last match is that one
    int hit = -1;
#pragma unroll
    for (int d = P; d >= 0; --d) {
      const int4 *row = reinterpret_cast<const int4 *>(sw + (tl + P - d) * SLOTS);
#pragma unroll
      for (int s4 = 0; s4 < SLOTS / 4; ++s4) {
        const int4 x = row[s4];
        const int xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int s = 4 * s4 + e;
          if (d == 0) {
            if (xs[e] == my) {
              if (is_w && s < j) err |= SDM_DEVERR_INDEX_REPEAT;
              if (!is_w) hit = s;
            }
          } else if (xs[e] == my) {
            hit = (d << 8) | s;
          }
        }
      }
    }
    if (hit >= 0) {
      const int d = hit >> 8, s = hit & 0xff;
      code = d == 0 ? (kRecompute | s) : L::kRowH + ((t - d) % L::NH) * SLOTS + s;
    }
  }
  o.src[pos] = static_cast<uint16_t>(code);
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
  float *undo;  // optional [B,T,H,W,d_v]: the written rows before each token's decay
  int T, H, N, d_v, v_bf16, tiles, W;
  long total_warps;
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
template <int Q>
__device__ __forceinline__ float4 xsum4(float4 a) {  // sum over the row subgroups (lane bits from log2 Q up)
#pragma unroll
  for (int m = Q; m <= 16; m <<= 1) {
    a.x += __shfl_xor_sync(kFull, a.x, m);
    a.y += __shfl_xor_sync(kFull, a.y, m);
    a.z += __shfl_xor_sync(kFull, a.z, m);
    a.w += __shfl_xor_sync(kFull, a.w, m);
  }
  return a;
}

template <int P, int SLOTS, int TW, int MODE, bool LOG>  // LOG: also write the undo log
__global__ void __launch_bounds__(128) sparse_scan_kernel(const ScanArgs a) {
  using L = ScanLayout<P, SLOTS, TW>;
  using Rec = TokenRec<SLOTS>;
  constexpr int Q = Tile<TW>::Q, RG = Tile<TW>::RG, RB = Tile<TW>::RB;
  constexpr int RPL = SLOTS / RG;
  constexpr int SLOT_B = SLOTS * RB;  // bytes per ring slot
  constexpr int REC_CHUNKS = static_cast<int>(sizeof(Rec) / 16);
  extern __shared__ __align__(16) unsigned char smem_raw[];

  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const long gw = static_cast<long>(blockIdx.x) * (blockDim.x >> 5) + wib;
  if (gw >= a.total_warps) return;  // warp-uniform; no CTA-wide barrier below
  const int tile = static_cast<int>(gw % a.tiles);
  const long bh = gw / a.tiles;
  const int h = static_cast<int>(bh % a.H);
  const long b = bh / a.H;
  const int T = a.T, d_v = a.d_v;
  const int q = lane % Q, r = lane / Q;
  const int col = tile * TW + 4 * q;
  const bool active = col < d_v;

  unsigned char *base = smem_raw + static_cast<size_t>(wib) * L::kWarpBytes;
  unsigned char *lbase = base + 16 * q;  // this lane's quad inside any 128-byte row
  Rec *recs = reinterpret_cast<Rec *>(base + L::kRecOff);
  uint32_t *vbuf = reinterpret_cast<uint32_t *>(base + L::kVOff);  // [NM][TW words]
  if (lane < TW) reinterpret_cast<float *>(base + L::kRowZero * RB)[lane] = 0.f;
  auto row_ptr = [&](int row) -> const float * {
    return reinterpret_cast<const float *>(lbase + min(row, L::kRowZero) * RB);
  };

  const size_t rowbytes = static_cast<size_t>(d_v) * sizeof(float);
  const unsigned char *table = reinterpret_cast<const unsigned char *>(a.state + bh * static_cast<long>(a.N) * d_v + col);
  unsigned char *table_w = reinterpret_cast<unsigned char *>(a.state + bh * static_cast<long>(a.N) * d_v + col);
  const long tok0 = b * T * a.H + h;
  const long tok_stride = a.H;

  // per-token global sources (this token's record and v), advanced one token
  // at a time; chunk c < REC_CHUNKS is 16 bytes of the record, the next Q are
  // the v columns 4vc .. 4vc+3 of this tile
  const int esz = a.v_bf16 ? 2 : 4;
  const unsigned char *rec_tok = reinterpret_cast<const unsigned char *>(static_cast<const Rec *>(a.rec) + tok0);
  const unsigned char *v_tok = static_cast<const unsigned char *>(a.v) + (tok0 * d_v + tile * TW) * esz;
  const long rec_step = tok_stride * static_cast<long>(sizeof(Rec));
  const long v_step = tok_stride * d_v * esz;
  int meta_slot = 0;  // ring slot of the next record to fetch
  auto issue_meta = [&]() {
    for (int c = lane; c < REC_CHUNKS + Q; c += 32) {
      if (c < REC_CHUNKS) {
        cp_async<16>(reinterpret_cast<unsigned char *>(recs + meta_slot) + 16 * c, rec_tok + 16 * c);
      } else {
        const int vc = c - REC_CHUNKS;
        if (tile * TW + 4 * vc < d_v) {
          unsigned char *dst = reinterpret_cast<unsigned char *>(vbuf + meta_slot * TW) + vc * 4 * esz;
          if (a.v_bf16) cp_async<8>(dst, v_tok + vc * 8);
          else cp_async<16>(dst, v_tok + vc * 16);
        }
      }
    }
    rec_tok += rec_step;
    v_tok += v_step;
    meta_slot = meta_slot + 1 == L::NM ? 0 : meta_slot + 1;
  };
  // the row quads this lane consumes: write slots r+RG k and read slots r+RG k
  int fetch_rec = 0, fetch_ring = 0;  // record slot and row-ring slot of the next token to fetch
  auto issue_rows = [&]() {
    if (active) {
      const Rec &m = recs[fetch_rec];
      const int4 *ip = reinterpret_cast<const int4 *>(m.idx + r * 2 * RPL);
      unsigned char *dw = lbase + (L::kRowW * RB + fetch_ring * SLOT_B);
      unsigned char *dr = lbase + (L::kRowR * RB + fetch_ring * SLOT_B);
#pragma unroll
      for (int k4 = 0; k4 < 2 * RPL / 4; ++k4) {
        const int4 x = ip[k4];
        const int ids[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = 4 * k4 + e;
          const int j = r + RG * (k < RPL ? k : k - RPL);
          if (static_cast<unsigned>(ids[e]) < static_cast<unsigned>(a.N))
            cp_async<16>((k < RPL ? dw : dr) + j * RB, table + static_cast<size_t>(ids[e]) * rowbytes);
        }
      }
    }
    fetch_rec = fetch_rec + 1 == L::NM ? 0 : fetch_rec + 1;
    fetch_ring = fetch_ring + 1 == L::NI ? 0 : fetch_ring + 1;
  };

  // prologue: records of tokens [0, P), then P groups (rows of j, record of j+P)
  for (int t = 0; t < P && t < T; ++t) issue_meta();
  cp_async_commit();
  cp_async_wait<0>();
  __syncwarp();
  for (int j = 0; j < P; ++j) {
    if (j + P < T) issue_meta();
    if (j < T) issue_rows();
    cp_async_commit();
  }

  float *yp_out = a.y + tok0 * d_v + col;
  const long y_step = tok_stride * d_v;
  float *undo_out = LOG ? a.undo + tok0 * a.W * d_v + col : nullptr;
  const long undo_step = tok_stride * a.W * d_v;
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  int cur_rec = 0, cur_ring = 0;
  for (int t = 0; t < T; ++t) {
    cp_async_wait<P - 1>();
    __syncwarp();
    if (t + 2 * P < T) issue_meta();
    if (t + P < T) issue_rows();
    cp_async_commit();

    const Rec &m = recs[cur_rec];
    const float al = m.alpha, be = m.beta;
    const uint32_t *vw = vbuf + cur_rec * TW;
    float4 vv;
    if (a.v_bf16) {
      const uint2 w2 = *reinterpret_cast<const uint2 *>(vw + 2 * q);
      vv = make_float4(bf16_to_f32(w2.x & 0xffff), bf16_to_f32(w2.x >> 16), bf16_to_f32(w2.y & 0xffff),
                       bf16_to_f32(w2.y >> 16));
    } else {
      vv = *reinterpret_cast<const float4 *>(vw + 4 * q);
    }
    // this lane's slots: ids (write), weights and source rows, vector loads
    int my_idx[RPL];
    float my_w[2 * RPL];
    int my_src[2 * RPL];
#pragma unroll
    for (int k = 0; k < RPL; k += 4) {  // the first RPL of the lane's positions are its write slots
      const int4 x = *reinterpret_cast<const int4 *>(m.idx + r * 2 * RPL + k);
      const int xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (k + e < RPL) my_idx[k + e] = xs[e];
    }
#pragma unroll
    for (int k = 0; k < 2 * RPL; k += 4) {
      const float4 x = *reinterpret_cast<const float4 *>(m.w + r * 2 * RPL + k);
      my_w[k] = x.x; my_w[k + 1] = x.y; my_w[k + 2] = x.z; my_w[k + 3] = x.w;
    }
    if constexpr (2 * RPL % 8 == 0) {
#pragma unroll
      for (int k = 0; k < 2 * RPL; k += 8) {
        const uint4 x = *reinterpret_cast<const uint4 *>(m.src + r * 2 * RPL + k);
        const uint32_t u[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          my_src[k + 2 * e] = static_cast<int>(u[e] & 0xffff);
          my_src[k + 2 * e + 1] = static_cast<int>(u[e] >> 16);
        }
      }
    } else {
      const uint2 x = *reinterpret_cast<const uint2 *>(m.src + r * 2 * RPL);
      my_src[0] = static_cast<int>(x.x & 0xffff);
      my_src[1] = static_cast<int>(x.x >> 16);
      my_src[2] = static_cast<int>(x.y & 0xffff);
      my_src[3] = static_cast<int>(x.y >> 16);
    }

    // selective decay of the written rows and the shared prediction (Fig. 2)
    float4 md[RPL];
    float4 vh = zero4;
#pragma unroll
    for (int k = 0; k < RPL; ++k) md[k] = ld4(row_ptr(my_src[k]));
    if (LOG) {  // the undo log: write slot j = r + RG k before the decay
#pragma unroll
      for (int k = 0; k < RPL; ++k)
        if (active && r + RG * k < a.W) st4(undo_out + static_cast<long>(r + RG * k) * d_v, md[k]);
      undo_out += undo_step;
    }
    // read rows; a read of a row this token writes is patched below
    float4 xr[RPL];
    bool recomp = false;
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int code = my_src[RPL + k];
      const bool rc = (code & kRecompute) != 0;
      recomp |= rc;
      xr[k] = ld4(row_ptr(rc ? L::kRowZero : code));
    }
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      md[k] = mul4(al, md[k]);
      if (MODE == SDM_RESID_SHARED) vh = fma4(my_w[k], md[k], vh);
    }
    float4 base4 = vv;
    if (MODE == SDM_RESID_SHARED) base4 = sub4(vv, xsum4<Q>(vh));
    auto new_row = [&](float4 mdk, float gk) -> float4 {
      return fma4(gk, MODE == SDM_RESID_PERSLOT ? sub4(vv, mdk) : base4, mdk);
    };

    // delta write: history ring (forwarding source) and the table in HBM.  The
    // table rows and y are stored with the streaming hint (evict first): a
    // written row is rarely gathered again before it would leave L2 anyway,
    // and keeping written lines out of the way leaves L2 to the gathers
    // (measured: the 1.4B-layer scan 2.77 -> 2.66 ms).  The undo log keeps
    // normal stores: the backward reads it, newest first, right after.
    unsigned char *hslot = lbase + (L::kRowH * RB + cur_ring * SLOT_B);
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const float4 nw = new_row(md[k], be * my_w[k]);
      st4(reinterpret_cast<float *>(hslot + (r + RG * k) * RB), nw);
      const int i = my_idx[k];
      if (active && static_cast<unsigned>(i) < static_cast<unsigned>(a.N))
        __stcs(reinterpret_cast<float4 *>(table_w + static_cast<size_t>(i) * rowbytes), nw);
    }
    // rare: a read of a row written by this same token -> recompute its new value
    if (__any_sync(kFull, recomp)) {
#pragma unroll
      for (int k = 0; k < RPL; ++k) {
        const int code = my_src[RPL + k];
        if (code & kRecompute) {
          const int sw = code & 0xff;                       // write slot of this token
          const int ps = (sw % RG) * 2 * RPL + (sw / RG);  // its record position
          xr[k] = new_row(mul4(al, ld4(row_ptr(m.src[ps]))), be * m.w[ps]);
        }
      }
    }
    // read after the write
    float4 yp = zero4;
#pragma unroll
    for (int k = 0; k < RPL; ++k) yp = fma4(my_w[RPL + k], xr[k], yp);
    yp = xsum4<Q>(yp);
    if (r == 0 && active) __stcs(reinterpret_cast<float4 *>(yp_out), yp);
    yp_out += y_step;
    cur_rec = cur_rec + 1 == L::NM ? 0 : cur_rec + 1;
    cur_ring = cur_ring + 1 == L::NI ? 0 : cur_ring + 1;
  }
  cp_async_wait<0>();
}

int env_int(const char *name, int dflt) {
  const char *s = getenv(name);
  return (s && *s) ? atoi(s) : dflt;
}

template <int P, int SLOTS, int TW>
size_t warp_bytes() { return ScanLayout<P, SLOTS, TW>::kWarpBytes; }

size_t warp_bytes_dispatch(int slots, int P, int tw) {
  if (slots == 16 && tw == 32)
    return P == 4 ? warp_bytes<4, 16, 32>() : P == 6 ? warp_bytes<6, 16, 32>() : warp_bytes<8, 16, 32>();
  if (slots == 16 && tw == 16)
    return P == 4 ? warp_bytes<4, 16, 16>() : P == 6 ? warp_bytes<6, 16, 16>() : warp_bytes<8, 16, 16>();
  return (P == 4 && tw == 32) ? warp_bytes<4, 64, 32>() : 0;
}

template <int P, int SLOTS, int TW, int MODE>
int launch_scan(const ScanArgs &args, int wpc, cudaStream_t st) {
  const size_t smem = ScanLayout<P, SLOTS, TW>::kWarpBytes * wpc;
  auto kern =
      args.undo ? sparse_scan_kernel<P, SLOTS, TW, MODE, true> : sparse_scan_kernel<P, SLOTS, TW, MODE, false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return check_launch("sdm_scan: set shared memory");
  const long blocks = (args.total_warps + wpc - 1) / wpc;
  kern<<<static_cast<unsigned>(blocks), wpc * 32, smem, st>>>(args);
  return check_launch("sdm_scan: scan kernel");
}

template <int P, int SLOTS, int TW>
int launch_mode(int mode, const ScanArgs &args, int wpc, cudaStream_t st) {
  if (mode == SDM_RESID_SHARED) return launch_scan<P, SLOTS, TW, SDM_RESID_SHARED>(args, wpc, st);
  if (mode == SDM_RESID_PERSLOT) return launch_scan<P, SLOTS, TW, SDM_RESID_PERSLOT>(args, wpc, st);
  return launch_scan<P, SLOTS, TW, SDM_RESID_ADDITIVE>(args, wpc, st);
}

int launch_dispatch(int slots, int P, int tw, int mode, const ScanArgs &args, int wpc, cudaStream_t st) {
  if (slots == 16 && tw == 32 && P == 4) return launch_mode<4, 16, 32>(mode, args, wpc, st);
  if (slots == 16 && tw == 32 && P == 6) return launch_mode<6, 16, 32>(mode, args, wpc, st);
  if (slots == 16 && tw == 32 && P == 8) return launch_mode<8, 16, 32>(mode, args, wpc, st);
  if (slots == 16 && tw == 16 && P == 4) return launch_mode<4, 16, 16>(mode, args, wpc, st);
  if (slots == 16 && tw == 16 && P == 6) return launch_mode<6, 16, 16>(mode, args, wpc, st);
  if (slots == 16 && tw == 16 && P == 8) return launch_mode<8, 16, 16>(mode, args, wpc, st);
  if (slots == 64 && tw == 32 && P == 4) return launch_mode<4, 64, 32>(mode, args, wpc, st);
  return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan: no kernel for slots=%d window=%d tile=%d", slots, P, tw);
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

static int scan_core(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
                     const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r, const float *w_r, int R,
                     int B, int T, int H, int N, int d_v, int resid_mode, float *y, float *undo, void *workspace,
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

  // Launch shape: B*H*ceil(d_v/TW) independent warps.  Each runs the whole
  // sequence, so all must be resident at once.  Per-warp speed is bound by
  // its own per-token chain, so more warps (16-column tiles) go first; for
  // each tile width take the deepest prefetch window whose shared-memory rings
  // still let every warp fit in one wave.  SDM_SCAN_TILE / SDM_SCAN_WINDOW /
  // SDM_SCAN_WARPS force a choice.
  const int slots = pick_slots(W, R);
  int dev = 0, smem_blk = 0, smem_sm = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&smem_blk, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int want_window = env_int("SDM_SCAN_WINDOW", 0), want_tile = env_int("SDM_SCAN_TILE", 0);
  int window = 0, wpc = 1, tw = 0;
  for (int w_t : {16, 32}) {
    if (want_tile && w_t != want_tile) continue;
    const long warps_t = static_cast<long>(B) * H * ((d_v + w_t - 1) / w_t);
    for (int p : {8, 6, 4}) {
      if (want_window && p != want_window) continue;
      const size_t wb = warp_bytes_dispatch(slots, p, w_t);
      if (wb == 0 || wb > static_cast<size_t>(smem_blk)) continue;
      for (int c : {4, 2, 1}) {  // warps per CTA
        if (c * wb > static_cast<size_t>(smem_blk)) continue;
        const long ctas_sm = static_cast<long>(smem_sm) / static_cast<long>(c * wb + 1024);
        if (window == 0) { window = p; wpc = c; tw = w_t; }  // fallback: the first that fits at all
        if (ctas_sm >= 1 && warps_t <= ctas_sm * c * sms) { window = p; wpc = c; tw = w_t; goto chosen; }
      }
    }
  }
chosen:
  if (window == 0) return set_error(SDM_ERR_SHAPE, "sdm_scan: W/R too large for shared memory");
  wpc = env_int("SDM_SCAN_WARPS", wpc);
  if (wpc < 1 || static_cast<size_t>(wpc) * warp_bytes_dispatch(slots, window, tw) > static_cast<size_t>(smem_blk))
    return set_error(SDM_ERR_INVALID_ARG, "sdm_scan: SDM_SCAN_WARPS does not fit");
  const int tiles = (d_v + tw - 1) / tw;
  const long total_warps = static_cast<long>(B) * H * tiles;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int rec_tb = kRecThreads / (2 * slots);  // tokens per prepass CTA
  const int t_blocks = (T + rec_tb - 1) / rec_tb;
  const unsigned rblocks = static_cast<unsigned>(static_cast<long>(B) * H * t_blocks);
#define SDM_REC(PP, S, TT)                                                                                  \
  record_kernel<PP, S, TT><<<rblocks, kRecThreads, 0, st>>>(idx_w, w_w, idx_r, w_r, alpha, beta, W, R, T, H, N, \
                                                            t_blocks, static_cast<TokenRec<S> *>(workspace), dev_err)
  if (slots == 16 && tw == 32 && window == 4) SDM_REC(4, 16, 32);
  else if (slots == 16 && tw == 32 && window == 6) SDM_REC(6, 16, 32);
  else if (slots == 16 && tw == 32 && window == 8) SDM_REC(8, 16, 32);
  else if (slots == 16 && tw == 16 && window == 4) SDM_REC(4, 16, 16);
  else if (slots == 16 && tw == 16 && window == 6) SDM_REC(6, 16, 16);
  else if (slots == 16 && tw == 16 && window == 8) SDM_REC(8, 16, 16);
  else SDM_REC(4, 64, 32);
#undef SDM_REC
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
  args.undo = undo;
  args.W = W;
  return launch_dispatch(slots, window, tw, resid_mode, args, wpc, st);
}

extern "C" int sdm_scan(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
                        const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r, const float *w_r, int R,
                        int B, int T, int H, int N, int d_v, int resid_mode, float *y, void *workspace,
                        size_t workspace_bytes, int32_t *dev_err, void *stream) {
  return scan_core(state, v, v_dtype, alpha, beta, idx_w, w_w, W, idx_r, w_r, R, B, T, H, N, d_v, resid_mode, y,
                   nullptr, workspace, workspace_bytes, dev_err, stream);
}

extern "C" int sdm_scan_train(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
                              const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r, const float *w_r,
                              int R, int B, int T, int H, int N, int d_v, int resid_mode, float *y, float *undo,
                              void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream) {
  if (!undo) return set_error(SDM_ERR_INVALID_ARG, "sdm_scan_train: null undo log");
  if (!aligned(undo, 16)) return set_error(SDM_ERR_ALIGN, "sdm_scan_train: the undo log needs 16-byte alignment");
  return scan_core(state, v, v_dtype, alpha, beta, idx_w, w_w, W, idx_r, w_r, R, B, T, H, N, d_v, resid_mode, y,
                   undo, workspace, workspace_bytes, dev_err, stream);
}

// ---------------------------------------------------------------------------
// sdm_scan_noalloc: sdm_scan for callers that cannot hand over device scratch
// memory.  The per-token records live in a fixed, file-scope device array instead
// of a caller workspace.  Host code cannot use the array's name as a device
// address, so the address is looked up with cudaGetSymbolAddress (with the
// device current) and cached per device together with the id of the CUDA
// context it was taken in; a call made in another context (the device's
// primary context destroyed and created again, e.g. after cudaDeviceReset)
// looks it up again, because the module, and with it the array, may then sit
// elsewhere.  The first call in a context does this lookup, so make that first
// call before capturing any stream.  Every call shares the one array: calls
// that can overlap on the GPU (different streams, or several host threads)
// race on it and must be serialised by the caller.  Every call rewrites all the
// records it reads, so nothing has to be cleared between calls.
// ---------------------------------------------------------------------------
namespace sdm {
namespace {
constexpr size_t kStaticScratchBytes = static_cast<size_t>(32) << 20;  // 32 MiB per device
__device__ __align__(256) unsigned char g_scan_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};

// id of the current CUDA context (unique for the life of the process), read
// through the driver entry points the runtime hands out, so that the library
// does not link the driver library itself
int current_context_id(unsigned long long *id) {
  using GetCurrentFn = CUresult (*)(CUcontext *);
  using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  if (!get_current || !get_id) {
    void *f1 = nullptr, *f2 = nullptr;
    cudaDriverEntryPointQueryResult q1, q2;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return set_error(SDM_ERR_CUDA, "sdm_scan_noalloc: driver entry points cuCtxGetCurrent/cuCtxGetId unavailable");
    get_current = reinterpret_cast<GetCurrentFn>(f1);
    get_id = reinterpret_cast<GetIdFn>(f2);
  }
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, id) != CUDA_SUCCESS)
    return set_error(SDM_ERR_CUDA, "sdm_scan_noalloc: no current CUDA context");
  return SDM_OK;
}

int static_scratch(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(SDM_ERR_CUDA, "sdm_scan_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_error(SDM_ERR_UNSUPPORTED, "sdm_scan_noalloc: device %d", dev);
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  unsigned long long ctx_id = 0;
  if (!g_scratch_addr[dev]) {
    // the first lookup on this device: the runtime makes the primary context
    // current here if no context is yet
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scan_scratch);
    if (e != cudaSuccess || !p)
      return set_error(SDM_ERR_CUDA, "sdm_scan_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    const int rc = current_context_id(&ctx_id);
    if (rc != SDM_OK) return rc;
    g_scratch_addr[dev] = p;
    g_scratch_ctx[dev] = ctx_id;
  } else {
    const int rc = current_context_id(&ctx_id);
    if (rc != SDM_OK) return rc;
    if (ctx_id != g_scratch_ctx[dev]) {
      void *p = nullptr;
      e = cudaGetSymbolAddress(&p, g_scan_scratch);
      if (e != cudaSuccess || !p)
        return set_error(SDM_ERR_CUDA, "sdm_scan_noalloc: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      g_scratch_addr[dev] = p;
      g_scratch_ctx[dev] = ctx_id;
    }
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
