// host_path.cu - the whole sparse step from host buffers, with transfers
// overlapped with compute.
//
// The sequence is cut into chunks of at most chunk_T tokens: the first and
// the last are a quarter of chunk_T, so the pipeline fills (the first chunk's
// inputs cross before any compute) and drains (the last chunk's y crosses
// after it) quickly, and the tokens between are split evenly into chunks of
// at most chunk_T.  For chunk c (staging slot c % 2) four streams run a
// software pipeline:
//   copy-in  : the chunk's score halves, v, alpha and beta, host -> device
//   address  : write and read addressing (independent of the table, so chunk
//              c+1's runs while chunk c is scanned)
//   compute  : the scan (the caller's stream; the table continues from chunk
//              to chunk)
//   copy-out : the chunk's y, device -> host
// Events order each stage after the one it depends on and keep a staging
// slot from being refilled before its previous chunk has left it.  Rows of a
// chunk are strided in the host layout [B,T,H,...], so every transfer is one
// 2-D copy (B rows).
#include <cstring>

#include "common.cuh"

namespace sdm {
namespace {

constexpr size_t kAlign = 256;
size_t align_up(size_t n) { return (n + kAlign - 1) & ~(kAlign - 1); }

// byte sizes of one staging slot's buffers for a chunk of Tc tokens
struct Slot {
  size_t s, v, g, iw, ir, y, ws;  // score half, v, one gate, write ids/weights, read ids/weights, y, scan workspace
  size_t total;
  Slot(int B, int Tc, int H, int sqrtN, int d_v, int W, int R, int esz) {
    const size_t th = static_cast<size_t>(B) * Tc * H;
    s = align_up(th * sqrtN * 4);
    v = align_up(th * d_v * esz);
    g = align_up(th * 4);
    iw = align_up(th * W * 4);
    ir = align_up(th * R * 4);
    y = align_up(th * d_v * 4);
    ws = align_up(sdm_scan_workspace_size(B, Tc, H, W, R));
    total = 4 * s + v + 2 * g + 2 * iw + 2 * ir + y + ws;
  }
};

// Chunk start of chunk c under the schedule above (c = nchunks gives T).
struct Schedule {
  int T, edge, mid_n, mid_base, mid_extra, n;
  Schedule(int T_, int chunk_T) : T(T_) {
    edge = chunk_T / 4 > 0 ? chunk_T / 4 : 1;
    if (T <= chunk_T) {  // one chunk
      edge = T;
      mid_n = mid_base = mid_extra = 0;
      n = 1;
      return;
    }
    const int mid = T - 2 * edge;  // >= 0: edge <= chunk_T / 2 < T / 2, or edge = 1 < T
    mid_n = (mid + chunk_T - 1) / chunk_T;
    mid_base = mid_n ? mid / mid_n : 0;
    mid_extra = mid_n ? mid % mid_n : 0;  // the first mid_extra middle chunks take one token more
    n = mid_n + 2;
  }
  int start(int c) const {
    if (c <= 0) return 0;
    if (n == 1 || c >= n) return T;
    const int m = c - 1;  // middle chunks before chunk c
    if (m >= mid_n) return T - edge;
    return edge + m * mid_base + (m < mid_extra ? m : mid_extra);
  }
};

int copy_chunk_2d(void *dst, const void *src, size_t feat_bytes, int B, int T, int H, int t0, int Tc, bool to_host,
                  cudaStream_t st) {
  const size_t row = static_cast<size_t>(Tc) * H * feat_bytes;   // one batch's chunk
  const size_t full = static_cast<size_t>(T) * H * feat_bytes;   // one batch's whole sequence
  const size_t off = static_cast<size_t>(t0) * H * feat_bytes;
  cudaError_t e;
  if (to_host)
    e = cudaMemcpy2DAsync(static_cast<char *>(dst) + off, full, src, row, row, B, cudaMemcpyDeviceToHost, st);
  else
    e = cudaMemcpy2DAsync(dst, row, static_cast<const char *>(src) + off, full, row, B, cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return set_error(SDM_ERR_CUDA, "sdm_forward_host: copy: %s", cudaGetErrorString(e));
  return SDM_OK;
}

}  // namespace
}  // namespace sdm

using namespace sdm;

extern "C" size_t sdm_forward_host_workspace_size(int B, int T, int H, int sqrtN, int d_v, int W, int R, int v_dtype,
                                                  int chunk_T) {
  if (B <= 0 || T <= 0 || H <= 0 || sqrtN <= 0 || d_v <= 0 || W <= 0 || R <= 0 || chunk_T <= 0) return 0;
  const int Tc = chunk_T < T ? chunk_T : T;
  const Slot sl(B, Tc, H, sqrtN, d_v, W, R, v_dtype == SDM_DTYPE_BF16 ? 2 : 4);
  return 2 * sl.total;
}

extern "C" int sdm_forward_host(const float *s1w, const float *s2w, const float *s1r, const float *s2r, const void *v,
                                int v_dtype, const float *alpha, const float *beta, int B, int T, int H, int sqrtN,
                                int k, int W, int R, int d_v, int resid_mode, float *state, float *y, int chunk_T,
                                void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream) {
  if (!s1w || !s2w || !s1r || !s2r || !v || !alpha || !beta || !state || !y || !workspace)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_forward_host: null pointer");
  if (B < 0 || T < 0 || H < 0 || chunk_T <= 0) return set_error(SDM_ERR_INVALID_ARG, "sdm_forward_host: bad sizes");
  if (v_dtype != SDM_DTYPE_F32 && v_dtype != SDM_DTYPE_BF16)
    return set_error(SDM_ERR_UNSUPPORTED, "sdm_forward_host: v_dtype must be SDM_DTYPE_F32 or SDM_DTYPE_BF16");
  if (B == 0 || T == 0 || H == 0) return SDM_OK;
  const size_t need = sdm_forward_host_workspace_size(B, T, H, sqrtN, d_v, W, R, v_dtype, chunk_T);
  if (need == 0) return set_error(SDM_ERR_SHAPE, "sdm_forward_host: bad sizes");
  if (workspace_bytes < need)
    return set_error(SDM_ERR_INVALID_ARG, "sdm_forward_host: workspace of %zu bytes needed", need);
  if (!aligned(workspace, kAlign)) return set_error(SDM_ERR_ALIGN, "sdm_forward_host: workspace must be 256-byte aligned");

  const int esz = v_dtype == SDM_DTYPE_BF16 ? 2 : 4;
  const int Tc = chunk_T < T ? chunk_T : T;
  const Slot sl(B, Tc, H, sqrtN, d_v, W, R, esz);
  cudaStream_t compute = static_cast<cudaStream_t>(stream);
  cudaStream_t cin = nullptr, cout = nullptr, caddr = nullptr;
  cudaEvent_t start = nullptr, in_done[2] = {}, addr_done[2] = {}, comp_done[2] = {}, out_done[2] = {};
  int rc = SDM_OK;
  auto ok = [&](cudaError_t e, const char *what) {
    if (e != cudaSuccess && rc == SDM_OK) rc = set_error(SDM_ERR_CUDA, "sdm_forward_host: %s: %s", what, cudaGetErrorString(e));
    return rc == SDM_OK;
  };
  ok(cudaStreamCreateWithFlags(&cin, cudaStreamNonBlocking), "stream");
  ok(cudaStreamCreateWithFlags(&cout, cudaStreamNonBlocking), "stream");
  ok(cudaStreamCreateWithFlags(&caddr, cudaStreamNonBlocking), "stream");
  ok(cudaEventCreateWithFlags(&start, cudaEventDisableTiming), "event");
  for (int i = 0; i < 2; ++i) {
    ok(cudaEventCreateWithFlags(&in_done[i], cudaEventDisableTiming), "event");
    ok(cudaEventCreateWithFlags(&addr_done[i], cudaEventDisableTiming), "event");
    ok(cudaEventCreateWithFlags(&comp_done[i], cudaEventDisableTiming), "event");
    ok(cudaEventCreateWithFlags(&out_done[i], cudaEventDisableTiming), "event");
  }
  // everything already queued on the caller's stream comes first
  if (rc == SDM_OK && ok(cudaEventRecord(start, compute), "record")) {
    ok(cudaStreamWaitEvent(cin, start, 0), "wait");
    ok(cudaStreamWaitEvent(cout, start, 0), "wait");
    ok(cudaStreamWaitEvent(caddr, start, 0), "wait");
  }

  const Schedule sched(T, Tc);
  const int nchunks = sched.n;
  for (int c = 0; c < nchunks && rc == SDM_OK; ++c) {
    const int s = c & 1;
    const int t0 = sched.start(c);
    const int tc = sched.start(c + 1) - t0;
    char *base = static_cast<char *>(workspace) + s * sl.total;
    float *d_s[4];
    for (int i = 0; i < 4; ++i) d_s[i] = reinterpret_cast<float *>(base + i * sl.s);
    char *p = base + 4 * sl.s;
    void *d_vb = p; p += sl.v;
    float *d_a = reinterpret_cast<float *>(p); p += sl.g;
    float *d_b = reinterpret_cast<float *>(p); p += sl.g;
    int32_t *d_iw = reinterpret_cast<int32_t *>(p); p += sl.iw;
    float *d_ww = reinterpret_cast<float *>(p); p += sl.iw;
    int32_t *d_ir = reinterpret_cast<int32_t *>(p); p += sl.ir;
    float *d_wr = reinterpret_cast<float *>(p); p += sl.ir;
    float *d_y = reinterpret_cast<float *>(p); p += sl.y;
    void *d_ws = p;

    // copy-in (after chunk c-2 left this slot's inputs)
    if (c >= 2 && !ok(cudaStreamWaitEvent(cin, comp_done[s], 0), "wait")) break;
    const float *hs[4] = {s1w, s2w, s1r, s2r};
    for (int i = 0; i < 4 && rc == SDM_OK; ++i)
      rc = copy_chunk_2d(d_s[i], hs[i], static_cast<size_t>(sqrtN) * 4, B, T, H, t0, tc, false, cin);
    if (rc == SDM_OK) rc = copy_chunk_2d(d_vb, v, static_cast<size_t>(d_v) * esz, B, T, H, t0, tc, false, cin);
    if (rc == SDM_OK) rc = copy_chunk_2d(d_a, alpha, 4, B, T, H, t0, tc, false, cin);
    if (rc == SDM_OK) rc = copy_chunk_2d(d_b, beta, 4, B, T, H, t0, tc, false, cin);
    if (rc != SDM_OK || !ok(cudaEventRecord(in_done[s], cin), "record")) break;

    // addressing (after its inputs landed; this slot's previous ids were read
    // by chunk c-2's scan, which the copy-in already waited for)
    if (!ok(cudaStreamWaitEvent(caddr, in_done[s], 0), "wait")) break;
    rc = sdm_address(d_s[0], d_s[1], B, tc, H, sqrtN, k, W, d_iw, d_ww, dev_err, caddr);
    if (rc == SDM_OK) rc = sdm_address(d_s[2], d_s[3], B, tc, H, sqrtN, k, R, d_ir, d_wr, dev_err, caddr);
    if (rc != SDM_OK || !ok(cudaEventRecord(addr_done[s], caddr), "record")) break;

    // scan (after the addressing and after chunk c-2's y left this slot)
    if (!ok(cudaStreamWaitEvent(compute, addr_done[s], 0), "wait")) break;
    if (c >= 2 && !ok(cudaStreamWaitEvent(compute, out_done[s], 0), "wait")) break;
    rc = sdm_scan(state, d_vb, v_dtype, d_a, d_b, d_iw, d_ww, W, d_ir, d_wr, R, B, tc, H, sqrtN * sqrtN, d_v,
                  resid_mode, d_y, d_ws, sl.ws, dev_err, compute);
    if (rc != SDM_OK || !ok(cudaEventRecord(comp_done[s], compute), "record")) break;

    // copy-out
    if (!ok(cudaStreamWaitEvent(cout, comp_done[s], 0), "wait")) break;
    rc = copy_chunk_2d(y, d_y, static_cast<size_t>(d_v) * 4, B, T, H, t0, tc, true, cout);
    if (rc != SDM_OK || !ok(cudaEventRecord(out_done[s], cout), "record")) break;
  }
  // the caller's stream completes only after the last y copy
  if (cout) {
    cudaEvent_t fin = nullptr;
    if (cudaEventCreateWithFlags(&fin, cudaEventDisableTiming) == cudaSuccess) {
      cudaEventRecord(fin, cout);
      cudaStreamWaitEvent(compute, fin, 0);
      cudaEventRecord(fin, cin);
      cudaStreamWaitEvent(compute, fin, 0);
      cudaEventRecord(fin, caddr);
      cudaStreamWaitEvent(compute, fin, 0);
      cudaEventDestroy(fin);
    }
  }
  // streams and events are released once their queued work completes
  for (int i = 0; i < 2; ++i) {
    if (in_done[i]) cudaEventDestroy(in_done[i]);
    if (addr_done[i]) cudaEventDestroy(addr_done[i]);
    if (comp_done[i]) cudaEventDestroy(comp_done[i]);
    if (out_done[i]) cudaEventDestroy(out_done[i]);
  }
  if (start) cudaEventDestroy(start);
  if (cin) cudaStreamDestroy(cin);
  if (cout) cudaStreamDestroy(cout);
  if (caddr) cudaStreamDestroy(caddr);
  return rc;
}
