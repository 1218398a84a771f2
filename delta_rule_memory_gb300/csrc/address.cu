// address.cu - product-key addressing (Sparse Delta Memory deck, "Product keys
// select addresses without scoring every slot", Secs. 2 and 3.1).
//
// One warp per token-head row (persistent warps).  Each stage is an exact
// warp-level top-k over (key descending, id ascending), where key is the
// order-preserving uint32 image of an fp32 score: candidates sit in lane
// registers, and per output rank one redux.sync max finds the best key, one
// redux.sync min the lowest id holding it, and the lane holding that id (ids
// are unique) pops it.  Stage 1 and 2 select the top-k of each score half
// (ids = positions), first filtering by a provable lower bound of the k-th
// score (the k-th largest lane maximum, from a bitonic sort of the warp); the
// two halves' selections run interleaved, so each redux chain hides the
// other's latency.  Stage 3 forms the
// fp32 sums s1[a] + s2[b] (ids = a*sqrtN + b) of only the candidates that can
// reach the top-W (a staircase of the two sorted halves), checks that no sum
// outside it ties the W-th, and selects the top-W; the weights are the
// softmax of the selected sums.
#include <climits>
#include <cstring>

#include "common.cuh"

namespace sdm {
namespace {

constexpr int kAddrWarps = 8;

template <int E>
__device__ __forceinline__ void local_sort(uint32_t (&key)[E], int (&id)[E]) {
  // odd-even transposition sort, descending by (key, -id)
#pragma unroll
  for (int pass = 0; pass < E; ++pass) {
#pragma unroll
    for (int i = pass & 1; i + 1 < E; i += 2) {
      const bool sw = key[i + 1] > key[i] || (key[i + 1] == key[i] && id[i + 1] < id[i]);
      const uint32_t k0 = key[i], k1 = key[i + 1];
      const int i0 = id[i], i1 = id[i + 1];
      key[i] = sw ? k1 : k0;
      key[i + 1] = sw ? k0 : k1;
      id[i] = sw ? i1 : i0;
      id[i + 1] = sw ? i0 : i1;
    }
  }
}

// Exact top-`count` of the warp's 32*E (key, id) pairs.  Padding entries carry
// key 0 and id INT_MAX; ids of real entries are distinct.  On return, rank r
// (r < count) sits in lane r % 32, output slot r / 32.
template <int E, int OUTS>
__device__ __forceinline__ void warp_topk(uint32_t (&key)[E], int (&id)[E], int count, uint32_t (&okey)[OUTS],
                                          int (&oid)[OUTS]) {
  const int lane = threadIdx.x & 31;
  local_sort(key, id);
#pragma unroll
  for (int o = 0; o < OUTS; ++o) {
    okey[o] = 0;
    oid[o] = INT_MAX;
  }
  for (int r = 0; r < count; ++r) {
    const uint32_t m = __reduce_max_sync(kFull, key[0]);
    const int cand = (key[0] == m) ? id[0] : INT_MAX;
    const int wid = __reduce_min_sync(kFull, cand);
    const bool pop = (key[0] == m) && (id[0] == wid);
#pragma unroll
    for (int e = 0; e + 1 < E; ++e) {
      key[e] = pop ? key[e + 1] : key[e];
      id[e] = pop ? id[e + 1] : id[e];
    }
    if (pop) {
      key[E - 1] = 0;
      id[E - 1] = INT_MAX;
    }
#pragma unroll
    for (int o = 0; o < OUTS; ++o) {
      if (r == lane + 32 * o) {
        okey[o] = m;
        oid[o] = wid;
      }
    }
  }
}

// Exact top-`count` of up to 64 (key, id) pairs held two per lane: sorted
// pair, then one redux round per output rank (as warp_topk, cheaper pops).
__device__ __forceinline__ void warp_topk2(uint32_t k0, int i0, uint32_t k1, int i1, int count, uint32_t (&okey)[2],
                                           int (&oid)[2]) {
  const int lane = threadIdx.x & 31;
  if (k1 > k0 || (k1 == k0 && i1 < i0)) {
    const uint32_t tk = k0; k0 = k1; k1 = tk;
    const int ti = i0; i0 = i1; i1 = ti;
  }
  okey[0] = okey[1] = 0;
  oid[0] = oid[1] = INT_MAX;
  for (int r = 0; r < count; ++r) {
    const uint32_t m = __reduce_max_sync(kFull, k0);
    const int wid = __reduce_min_sync(kFull, k0 == m ? i0 : INT_MAX);
    const bool pop = k0 == m && i0 == wid;
    k0 = pop ? k1 : k0;
    i0 = pop ? i1 : i0;
    k1 = pop ? 0u : k1;
    i1 = pop ? INT_MAX : i1;
    if (r == lane) { okey[0] = m; oid[0] = wid; }
    if (r == lane + 32) { okey[1] = m; oid[1] = wid; }
  }
}

// Exact top-`count` (count <= 32) of up to 64 (key, id) pairs held two per
// lane, where the ids of real entries are unique and at least `count` entries
// are real.  Per output rank one redux.sync max finds the best key, one
// redux.sync min the lowest id holding it, and the lane holding that id (ids
// are unique) pops it; lane 0 records the rank in `rbuf` (32 entries of the
// warp's own scratch).  On return lane r holds rank r (r < count).
__device__ __forceinline__ void warp_topk2_fast(uint32_t k0, int i0, uint32_t k1, int i1, int count, uint2 *rbuf,
                                                uint32_t &okey, int &oid) {
  const int lane = threadIdx.x & 31;
  if (k1 > k0 || (k1 == k0 && i1 < i0)) {
    const uint32_t tk = k0; k0 = k1; k1 = tk;
    const int ti = i0; i0 = i1; i1 = ti;
  }
#pragma unroll 4
  for (int r = 0; r < count; ++r) {
    const uint32_t m = __reduce_max_sync(kFull, k0);
    const int wid = __reduce_min_sync(kFull, k0 == m ? i0 : INT_MAX);
    const bool pop = i0 == wid;
    k0 = pop ? k1 : k0;
    i0 = pop ? i1 : i0;
    k1 = pop ? 0u : k1;
    i1 = pop ? INT_MAX : i1;
    if (lane == 0) rbuf[r] = make_uint2(m, static_cast<unsigned>(wid));
  }
  __syncwarp();
  const uint2 e = lane < count ? rbuf[lane] : make_uint2(0u, static_cast<unsigned>(INT_MAX));
  __syncwarp();
  okey = e.x;
  oid = static_cast<int>(e.y);
}

// warp_topk2_fast on two independent candidate sets at once (the two score
// halves of a row): their redux chains interleave, so each hides the other's
// latency.  Results go through rbufA / rbufB (32 entries each).
__device__ __forceinline__ void warp_topk2_fast_x2(uint2 ca0, uint2 ca1, uint2 cb0, uint2 cb1, int count,
                                                   uint2 *rbufA, uint2 *rbufB, uint2 &outA, uint2 &outB) {
  const int lane = threadIdx.x & 31;
  uint32_t ka0 = ca0.x, ka1 = ca1.x, kb0 = cb0.x, kb1 = cb1.x;
  int ia0 = static_cast<int>(ca0.y), ia1 = static_cast<int>(ca1.y);
  int ib0 = static_cast<int>(cb0.y), ib1 = static_cast<int>(cb1.y);
  if (ka1 > ka0 || (ka1 == ka0 && ia1 < ia0)) {
    const uint32_t tk = ka0; ka0 = ka1; ka1 = tk;
    const int ti = ia0; ia0 = ia1; ia1 = ti;
  }
  if (kb1 > kb0 || (kb1 == kb0 && ib1 < ib0)) {
    const uint32_t tk = kb0; kb0 = kb1; kb1 = tk;
    const int ti = ib0; ib0 = ib1; ib1 = ti;
  }
#pragma unroll 2
  for (int r = 0; r < count; ++r) {
    const uint32_t ma = __reduce_max_sync(kFull, ka0);
    const uint32_t mb = __reduce_max_sync(kFull, kb0);
    const int wa = __reduce_min_sync(kFull, ka0 == ma ? ia0 : INT_MAX);
    const int wb = __reduce_min_sync(kFull, kb0 == mb ? ib0 : INT_MAX);
    const bool pa = ia0 == wa, pb = ib0 == wb;
    ka0 = pa ? ka1 : ka0;
    ia0 = pa ? ia1 : ia0;
    ka1 = pa ? 0u : ka1;
    ia1 = pa ? INT_MAX : ia1;
    kb0 = pb ? kb1 : kb0;
    ib0 = pb ? ib1 : ib0;
    kb1 = pb ? 0u : kb1;
    ib1 = pb ? INT_MAX : ib1;
    if (lane == 0) {
      rbufA[r] = make_uint2(ma, static_cast<unsigned>(wa));
      rbufB[r] = make_uint2(mb, static_cast<unsigned>(wb));
    }
  }
  __syncwarp();
  const uint2 pad = make_uint2(0u, static_cast<unsigned>(INT_MAX));
  outA = lane < count ? rbufA[lane] : pad;
  outB = lane < count ? rbufB[lane] : pad;
  __syncwarp();
}

// Both halves' lower bounds at once: v packs two 16-bit keys (the top half of
// each score half's lane maximum); a bitonic sort of the warp, descending in
// each 16-bit half independently (max.u16x2 / min.u16x2), then lane k-1's
// pair.  Truncation is monotone, so the result is the truncated k-th largest
// lane maximum of each half: still a lower bound of that half's k-th score.
__device__ __forceinline__ uint32_t warp_kth_largest_x2(uint32_t v, int k) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int blk = 2; blk <= 32; blk <<= 1) {
#pragma unroll
    for (int j = blk >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(kFull, v, j);
      const bool desc = (lane & blk) == 0, lower = (lane & j) == 0;
      uint32_t r;
      if (lower == desc)
        asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(o));
      else
        asm("min.u16x2 %0, %1, %2;" : "=r"(r) : "r"(v), "r"(o));
      v = r;
    }
  }
  return __shfl_sync(kFull, v, k - 1);
}

// Candidates of one score half: the entries with key >= tau compacted into
// cbuf in ballot order (at most 64 stored); returns how many qualified.
template <int E>
__device__ __forceinline__ int count_compact(const uint32_t (&key)[E], int n, uint32_t tau, uint2 *cbuf) {
  const int lane = threadIdx.x & 31;
  int basepos = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const bool in = key[e] >= tau && lane + 32 * e < n;
    const unsigned bal = __ballot_sync(kFull, in);
    const int pos = basepos + __popc(bal & ((1u << lane) - 1));
    if (in && pos < 64) cbuf[pos] = make_uint2(key[e], lane + 32 * e);
    basepos += __popc(bal);
  }
  return basepos;
}

// The k-th largest (k <= 32) of the 32 lanes' values: a bitonic sort of the
// warp, descending, then lane k-1's value.
__device__ __forceinline__ uint32_t warp_kth_largest(uint32_t v, int k) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int blk = 2; blk <= 32; blk <<= 1) {
#pragma unroll
    for (int j = blk >> 1; j > 0; j >>= 1) {
      const uint32_t o = __shfl_xor_sync(kFull, v, j);
      const bool desc = (lane & blk) == 0, lower = (lane & j) == 0;
      v = (lower == desc) ? max(v, o) : min(v, o);
    }
  }
  return __shfl_sync(kFull, v, k - 1);
}

// Top-k of one score half (positions 0..n-1, E values per lane at lane+32e).
// Fast path: tau = the k-th largest of the 32 lane maxima is a lower bound of
// the k-th largest score, so every top-k element has key >= tau; when at most
// 64 elements qualify they are compacted (ballot order) and selected exactly.
// Otherwise the full per-lane sorted selection runs.  Returns rank `lane`.
template <int E>
__device__ __forceinline__ void half_topk(const uint32_t (&key)[E], int n, int k, uint2 *cbuf, uint32_t &okey,
                                          int &oid) {
  const int lane = threadIdx.x & 31;
  uint32_t lm = 0;
#pragma unroll
  for (int e = 0; e < E; ++e) lm = max(lm, key[e]);
  int cnt = 0;
  uint32_t tau = 0;
  if (E > 2) {
    // k-th largest lane maximum
    tau = warp_kth_largest(lm, k);
#pragma unroll
    for (int e = 0; e < E; ++e) cnt += __popc(__ballot_sync(kFull, key[e] >= tau && lane + 32 * e < n));
  }
  if (E > 2 && cnt <= 64) {
    int basepos = 0;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const bool in = key[e] >= tau && lane + 32 * e < n;
      const unsigned bal = __ballot_sync(kFull, in);
      if (in) cbuf[basepos + __popc(bal & ((1u << lane) - 1))] = make_uint2(key[e], lane + 32 * e);
      basepos += __popc(bal);
    }
    __syncwarp();
    const uint2 c0 = lane < cnt ? cbuf[lane] : make_uint2(0u, static_cast<unsigned>(INT_MAX));
    const uint2 c1 = lane + 32 < cnt ? cbuf[lane + 32] : make_uint2(0u, static_cast<unsigned>(INT_MAX));
    __syncwarp();
    // cnt >= k real candidates with unique positions
    warp_topk2_fast(c0.x, static_cast<int>(c0.y), c1.x, static_cast<int>(c1.y), k, cbuf, okey, oid);
  } else if (E <= 2) {
    uint32_t k0 = key[0], k1 = E > 1 ? key[E - 1] : 0u;
    int i0 = lane < n ? lane : INT_MAX, i1 = (E > 1 && lane + 32 < n) ? lane + 32 : INT_MAX;
    if (!(lane < n)) k0 = 0u;
    if (!(E > 1 && lane + 32 < n)) k1 = 0u;
    uint32_t ok[2];
    int oi[2];
    warp_topk2(k0, i0, k1, i1, k, ok, oi);
    okey = ok[0];
    oid = oi[0];
  } else {
    uint32_t kk[E];
    int id[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kk[e] = lane + 32 * e < n ? key[e] : 0u;
      id[e] = lane + 32 * e < n ? lane + 32 * e : INT_MAX;
    }
    uint32_t ok[1];
    int oi[1];
    warp_topk<E, 1>(kk, id, k, ok, oi);
    okey = ok[0];
    oid = oi[0];
  }
}

// The pruned candidate set P = {(x, y) : (x+1)(y+1) <= W} of the k x k grid
// of sorted half ranks, in column-major order: every slot outside P is
// dominated by at least W slots of P (the sorted halves make the sum monotone
// in x and y), so the top-W lies in P unless the W-th sum ties with a sum
// outside P.  Entry e (e < n, n <= 64) is (x[e], y[e]); corner[x] is the
// first y outside P in column x (k if none).  Built on the host from (k, W).
struct Staircase {
  int8_t x[64], y[64];
  int8_t corner[32];
  int n;
};

Staircase make_staircase(int k, int W) {
  Staircase st;
  memset(&st, 0, sizeof(st));
  int n = 0;
  for (int x = 0; x < k; ++x) {
    const int cnt = min(k, W / (x + 1));
    for (int y = 0; y < cnt; ++y, ++n)
      if (n < 64) {
        st.x[n] = static_cast<int8_t>(x);
        st.y[n] = static_cast<int8_t>(y);
      }
    st.corner[x] = static_cast<int8_t>(min(k, W / (x + 1)));
  }
  st.n = n;
  return st;
}

// One warp per row, persistent over rows.  E1 = score values per lane of a
// half; E3 = per-lane candidates of the full k*k fallback (8 or 32).
template <int E1, int E3>
__global__ void __launch_bounds__(kAddrWarps * 32, (E1 <= 8 && E3 <= 8) ? 4 : 1) address_kernel(const float *__restrict__ s1,
                                                                  const float *__restrict__ s2, long rows,
                                                                  int sqrtN, int k, int W, const Staircase sc,
                                                                  int32_t *__restrict__ idx_out,
                                                                  float *__restrict__ w_out,
                                                                  int32_t *__restrict__ dev_err) {
  __shared__ uint2 cbuf_all[kAddrWarps][128];
  const int lane = threadIdx.x & 31;
  uint2 *cbuf = cbuf_all[threadIdx.x >> 5];
  // lane owns entries lane and lane + 32 of the staircase P
  int px[2], py[2];
#pragma unroll
  for (int o = 0; o < 2; ++o) {
    const int e = lane + 32 * o;
    px[o] = e < sc.n ? sc.x[e] : -1;
    py[o] = e < sc.n ? sc.y[e] : -1;
  }
  const bool pruned_ok = sc.n <= 64;
  // corner of the complement of P in column x = lane: (x, floor(W/(x+1))) if inside the k x k grid
  const int corner_y = lane < k ? sc.corner[lane] : k;

  const long stride = static_cast<long>(gridDim.x) * kAddrWarps;
  for (long row = static_cast<long>(blockIdx.x) * kAddrWarps + (threadIdx.x >> 5); row < rows; row += stride) {
    // --- stage 1 and 2: top-k of each half (lane holds rank `lane`) ---
    float hv[2];
    int hid[2];
    bool bad = false;
    uint32_t key1[E1], key2[E1];
#pragma unroll
    for (int e = 0; e < E1; ++e) {
      const int j = lane + 32 * e;
      const float x1 = j < sqrtN ? s1[row * sqrtN + j] : 0.f;
      const float x2 = j < sqrtN ? s2[row * sqrtN + j] : 0.f;
      bad |= j < sqrtN && (!isfinite(x1) || !isfinite(x2));
      key1[e] = j < sqrtN ? order_key(x1) : 0u;
      key2[e] = j < sqrtN ? order_key(x2) : 0u;
    }
    bool both_fast = false;
    if (E1 > 2) {
      // both halves at once: tau of each (the k-th largest lane maximum, a
      // lower bound of the k-th largest score), the candidates >= tau, and
      // when both sets hold at most 64 the two exact selections interleaved
      uint32_t lm1 = 0, lm2 = 0;
#pragma unroll
      for (int e = 0; e < E1; ++e) {
        lm1 = max(lm1, key1[e]);
        lm2 = max(lm2, key2[e]);
      }
      const uint32_t tp = warp_kth_largest_x2((lm1 & 0xffff0000u) | (lm2 >> 16), k);
      const uint32_t tau1 = tp & 0xffff0000u, tau2 = tp << 16;
      const int cnt1 = count_compact<E1>(key1, sqrtN, tau1, cbuf);
      const int cnt2 = count_compact<E1>(key2, sqrtN, tau2, cbuf + 64);
      if (cnt1 <= 64 && cnt2 <= 64) {
        __syncwarp();
        const uint2 pad = make_uint2(0u, static_cast<unsigned>(INT_MAX));
        const uint2 a0 = lane < cnt1 ? cbuf[lane] : pad, a1 = lane + 32 < cnt1 ? cbuf[lane + 32] : pad;
        const uint2 b0 = lane < cnt2 ? cbuf[64 + lane] : pad, b1 = lane + 32 < cnt2 ? cbuf[64 + lane + 32] : pad;
        __syncwarp();
        uint2 oa, ob;
        warp_topk2_fast_x2(a0, a1, b0, b1, k, cbuf, cbuf + 64, oa, ob);
        hv[0] = key_value(oa.x);
        hid[0] = static_cast<int>(oa.y);
        hv[1] = key_value(ob.x);
        hid[1] = static_cast<int>(ob.y);
        both_fast = true;
      }
    }
    if (!both_fast) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t ok;
        int oi;
        half_topk<E1>(half == 0 ? key1 : key2, sqrtN, k, cbuf, ok, oi);
        hv[half] = key_value(ok);
        hid[half] = oi;
      }
    }
    if (__any_sync(kFull, bad) && lane == 0 && dev_err) atomicOr(dev_err, SDM_DEVERR_NONFINITE);

    // --- stage 3: top-W of the k*k sums s1[a_x] + s2[b_y] ---
    uint32_t ok[2];
    int oi[2];
    bool done = false;
    if (pruned_ok) {
      uint32_t ck[2];
      int ci[2];
#pragma unroll
      for (int o = 0; o < 2; ++o) {
        const int x = px[o] < 0 ? 0 : px[o], y = py[o] < 0 ? 0 : py[o];
        const float av = __shfl_sync(kFull, hv[0], x);
        const float bv = __shfl_sync(kFull, hv[1], y);
        const int ai = __shfl_sync(kFull, hid[0], x);
        const int bi = __shfl_sync(kFull, hid[1], y);
        ck[o] = px[o] >= 0 ? order_key(__fadd_rn(av, bv)) : 0u;
        ci[o] = px[o] >= 0 ? ai * sqrtN + bi : INT_MAX;
      }
      if (W <= 32) {  // the staircase holds at least W candidates with unique slot ids
        warp_topk2_fast(ck[0], ci[0], ck[1], ci[1], W, cbuf, ok[0], oi[0]);
        ok[1] = 0u;
        oi[1] = INT_MAX;
      } else {
        warp_topk2(ck[0], ci[0], ck[1], ci[1], W, ok, oi);
      }
      // exactness: the best sum outside P sits on one of its corners
      const uint32_t kw = __shfl_sync(kFull, (W - 1) < 32 ? ok[0] : ok[1], (W - 1) & 31);
      const float bcorner = __shfl_sync(kFull, hv[1], corner_y < k ? corner_y : 0);
      const bool tie = lane < k && corner_y < k && order_key(__fadd_rn(hv[0], bcorner)) >= kw;
      done = !__any_sync(kFull, tie);
    }
    if (!done) {  // full k*k candidate set
      uint32_t key[E3];
      int id[E3];
      const int kk = k * k;
#pragma unroll
      for (int e = 0; e < E3; ++e) {
        const int c = lane + 32 * e;
        const int x = c / k, y = c - (c / k) * k;
        const float av = __shfl_sync(kFull, hv[0], x & 31);
        const float bv = __shfl_sync(kFull, hv[1], y & 31);
        const int ai = __shfl_sync(kFull, hid[0], x & 31);
        const int bi = __shfl_sync(kFull, hid[1], y & 31);
        const bool in = c < kk;
        key[e] = in ? order_key(__fadd_rn(av, bv)) : 0u;
        id[e] = in ? ai * sqrtN + bi : INT_MAX;
      }
      warp_topk<E3, 2>(key, id, W, ok, oi);
    }

    // --- weights: softmax over the W selected sums (max = rank 0) ---
    const float smax = key_value(__shfl_sync(kFull, ok[0], 0));
    float ex[2];
    float part = 0.f;
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      const int r = lane + 32 * o;
      ex[o] = (r < W) ? __expf(key_value(ok[o]) - smax) : 0.f;
      part += ex[o];
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(kFull, part, off);
    const float inv = 1.0f / part;
#pragma unroll
    for (int o = 0; o < 2; ++o) {
      const int r = lane + 32 * o;
      if (r < W) {
        idx_out[row * W + r] = oi[o];
        w_out[row * W + r] = ex[o] * inv;
      }
    }
  }
}

int pow2_at_least(int n) {
  int e = 1;
  while (e < n) e <<= 1;
  return e;
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" int sdm_address(const float *s1, const float *s2, int B, int T, int H, int sqrtN, int k, int W,
                           int32_t *idx_out, float *w_out, int32_t *dev_err, void *stream) {
  if (!s1 || !s2 || !idx_out || !w_out) return set_error(SDM_ERR_INVALID_ARG, "sdm_address: null pointer");
  if (B < 0 || T < 0 || H < 0) return set_error(SDM_ERR_INVALID_ARG, "sdm_address: negative size");
  if (sqrtN < 1 || sqrtN > 512 || k < 1 || k > 32 || k > sqrtN || W < 1 || W > 64 || W > k * k)
    return set_error(SDM_ERR_SHAPE, "sdm_address: need 1<=sqrtN<=512, 1<=k<=min(32,sqrtN), 1<=W<=min(64,k*k)");
  if (!aligned(s1, 4) || !aligned(s2, 4) || !aligned(idx_out, 4) || !aligned(w_out, 4) ||
      (dev_err && !aligned(dev_err, 4)))
    return set_error(SDM_ERR_ALIGN, "sdm_address: pointers must be 4-byte aligned");
  const long rows = static_cast<long>(B) * T * H;
  if (rows >= (1L << 31)) return set_error(SDM_ERR_SHAPE, "sdm_address: B*T*H must be < 2^31");
  if (rows == 0) return SDM_OK;
  const int E1 = pow2_at_least((sqrtN + 31) / 32);
  const int E3 = pow2_at_least((k * k + 31) / 32);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  long blocks = (rows + kAddrWarps - 1) / kAddrWarps;
  if (blocks > static_cast<long>(sms) * 8) blocks = static_cast<long>(sms) * 8;
  const dim3 grid(static_cast<unsigned>(blocks));
  const dim3 block(kAddrWarps * 32);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const Staircase sc = make_staircase(k, W);
#define SDM_AK(A, C) \
  address_kernel<A, C><<<grid, block, 0, st>>>(s1, s2, rows, sqrtN, k, W, sc, idx_out, w_out, dev_err)
#define SDM_AK_E3(A)            \
  if (E3 <= 8) SDM_AK(A, 8);    \
  else SDM_AK(A, 32);
  switch (E1) {
    case 1: SDM_AK_E3(1); break;
    case 2: SDM_AK_E3(2); break;
    case 4: SDM_AK_E3(4); break;
    case 8: SDM_AK_E3(8); break;
    default: SDM_AK_E3(16); break;
  }
#undef SDM_AK_E3
#undef SDM_AK
  return check_launch("sdm_address");
}
