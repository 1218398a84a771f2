/*
 * sdm.h - C ABI of libsdm.so: the sparse-routed gated delta-rule memory scan
 * on one GB300 (sm_103a).
 *
 * The method: a recurrent memory table per (batch, head) that each token
 * addresses sparsely, decays only where it writes, updates with a delta rule
 * and reads after the write.  Sources (reading decks of the three papers):
 *   [SDM]  "Sparse Delta Memory" deck: "Product keys select addresses without
 *          scoring every slot" (Secs. 2, 3.1); "Selected slots decay and
 *          update; other slots persist" (Eqs. 3-5); "A v1 inconsistency
 *          matters for reproducing the update" (Fig. 2 shared residual).
 *   [LAA]  "Linear Attention Architectures" deck: "GDN and KDA change the
 *          granularity of forgetting" (Eqs. 15-20).
 *   [SSE]  "Sparse State Expansion" deck: "One gate controls both writes and
 *          reads" (Eqs. 9-14); "SSE routes tokens into shared-parameter state
 *          partitions" (shared partition); "A memory decays only when its
 *          partition is visited".
 *
 * Conventions for every call below.
 *   - Tensor pointers are DEVICE pointers (cudaMalloc'd or PyTorch-owned),
 *     row-major and contiguous in the layout given.  The caller owns every
 *     buffer; the library keeps no pointer after a call returns and allocates
 *     no device memory.  Scratch space, where needed, is passed in by the
 *     caller and sized by the matching *_workspace_size() call.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  All calls
 *     are asynchronous and stream-ordered; none synchronises the host.
 *   - Return value: SDM_OK (0) or one of the SDM_ERR_* codes.  On an error
 *     return nothing has been launched and no output was touched, except for
 *     SDM_ERR_CUDA (a launch failed; see sdm_last_error()).  Errors found on
 *     the device (bad indices, non-finite scores) are OR-ed as SDM_DEVERR_*
 *     bits into the optional `dev_err` word, which the caller reads after
 *     synchronising; the kernels never trap.
 *   - bf16 arguments are uint16_t bit patterns.
 *   - Calls are thread-safe: they hold no global state apart from the
 *     thread-local error text.
 */
#ifndef SDM_H_
#define SDM_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define SDM_API __attribute__((visibility("default")))
#else
#define SDM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define SDM_OK 0
#define SDM_ERR_INVALID_ARG 1  /* null pointer, negative size, small workspace */
#define SDM_ERR_SHAPE 2        /* sizes inconsistent or beyond the limits below */
#define SDM_ERR_ALIGN 3        /* pointer not aligned as required */
#define SDM_ERR_UNSUPPORTED 4  /* unknown dtype or mode */
#define SDM_ERR_CUDA 5         /* a CUDA launch or copy failed */
#define SDM_ERR_DEVICE 6       /* sdm_check: a device-side error was recorded */

/* Device-side error bits (OR-ed into *dev_err when dev_err != NULL). */
#define SDM_DEVERR_INDEX_RANGE 1  /* a slot index outside [0, N) (skipped) */
#define SDM_DEVERR_INDEX_REPEAT 2 /* a slot repeated within one token's write list */
#define SDM_DEVERR_NONFINITE 4    /* a NaN or infinite score or logit */
#define SDM_DEVERR_TIMEOUT 8      /* a bounded on-device wait gave up; outputs invalid */

/*
 * A timeout (SDM_DEVERR_TIMEOUT) leaves that call's y AND the state it updated
 * in place undefined; every later call that continues the state builds on the
 * corrupt values.  So timeouts are never dropped: each one is also recorded in
 * a library-owned device word, whether or not the call had a dev_err.
 */

/*
 * Environment variables read at each call (all optional; unset = the library's
 * own choice):
 *   SDM_SCAN_TILE=16|32, SDM_SCAN_WINDOW=4|6|8, SDM_SCAN_WARPS=1..4
 *       sdm_scan / sdm_scan_train: column-tile width, prefetch window and warps
 *       per CTA of the scan kernel (default: the 16-column tile if every warp
 *       fits in one wave, then the deepest window that does, 4 warps per CTA).
 *   SDM_GDN_PATH=recurrent|chunk    gdn_scan: force the token-recurrent or the
 *       chunked tensor-core path (shape rules permitting).
 *   SDM_SSE_PATH=recurrent|chunk    sse_scan: force the token-by-token or the
 *       chunked prefill path (shape rules permitting).
 *   SDM_TEST_DROP_SIGNAL=1          test hook: the chunked GDN, KDA, GDN2 and
 *       SSE chain kernels skip one internal signal, so a bounded on-device wait runs out
 *       and the call reports SDM_DEVERR_TIMEOUT (its outputs are invalid; the
 *       CUDA context stays usable).  Never set in normal use.
 */

/* Element types of the value input of sdm_scan. */
#define SDM_DTYPE_F32 0
#define SDM_DTYPE_BF16 1

/* Residual of the sparse write (sdm_scan). */
#define SDM_RESID_SHARED 0   /* [SDM] Fig. 2: v_hat = sum_j w_j M~[j]; M[i] = M~[i] + beta w_i (v - v_hat) */
#define SDM_RESID_PERSLOT 1  /* [SDM] printed Eq. 4: M[i] = M~[i] + beta w_i (v - M~[i]) */
#define SDM_RESID_ADDITIVE 2 /* additive write, no residual: M[i] = M~[i] + beta w_i v */

/* sse_scan write modes */
#define SSE_WRITE_ADDITIVE 0 /* [SSE] Eqs. 9-14: S^p[j,:] = alpha_j S^p[j,:] + g kk_j v */
#define SSE_WRITE_DELTA 1    /* shared residual per partition: v replaced by v - sum_j kk_j alpha_j S^p[j,:] */

/* Library version (major*10000 + minor*100 + patch). */
SDM_API int sdm_version(void);

/* Text of the last error raised by a call on this host thread ("" if none). */
SDM_API const char *sdm_last_error(void);

/*
 * sdm_check - the device-side status check.  Synchronises `stream`, then reads
 * the caller's error word `dev_err` (optional; not cleared) and the library's
 * own timeout record (cleared by this call).  Returns SDM_OK if no bit is set,
 * SDM_ERR_DEVICE if any is (sdm_last_error() names the bits), SDM_ERR_CUDA if
 * the synchronisation or a read failed.  Not capturable (it synchronises);
 * call it after a step, not inside one.
 */
SDM_API int sdm_check(const int32_t *dev_err, void *stream);

/*
 * sdm_address - product-key addressing, [SDM] "Product keys select addresses
 * without scoring every slot" (Secs. 2 and 3.1).  Called once for the write
 * halves (W = |I^w|) and once for the read halves (W = |I^r|).
 *
 * For every token-head row r in [0, B*T*H):
 *   1. keep the top-k entries of s1[r] and of s2[r] (value descending, ties
 *      to the lower index);
 *   2. form only the k*k candidate scores s1[a] + s2[b] (one fp32 addition,
 *      round to nearest) with slot id a*sqrtN + b;
 *   3. select the top-W candidates by (score descending, slot id ascending);
 *   4. w = softmax over the W selected scores (no temperature).
 *
 * s1, s2  : fp32 [B,T,H,sqrtN] score halves.
 * idx_out : int32 [B,T,H,W] selected slot ids in rank order (bit-exact).
 * w_out   : fp32 [B,T,H,W] softmax weights, same order.
 * dev_err : optional; SDM_DEVERR_NONFINITE if a score is NaN/inf.
 * Limits: 1 <= sqrtN <= 512, 1 <= k <= min(32, sqrtN), 1 <= W <= min(64, k*k),
 *         B*T*H < 2^31.  Pointers 4-byte aligned.
 */
SDM_API int sdm_address(const float *s1, const float *s2, int B, int T, int H, int sqrtN, int k, int W,
                int32_t *idx_out, float *w_out, int32_t *dev_err, void *stream);

/*
 * Scratch bytes sdm_scan needs for these sizes: one packed record per
 * token-head (its slot ids, weights, gates and where each slot's row is read
 * from), 336 bytes when W, R <= 16 and 1296 bytes otherwise, rounded up to
 * 256.  0 for invalid sizes.
 */
SDM_API size_t sdm_scan_workspace_size(int B, int T, int H, int W, int R);

/*
 * sdm_scan - the sparse delta-rule memory scan, [SDM] Eqs. 3-5 with the
 * Fig. 2 shared residual by default.  For each (b, h), tokens in order:
 *   M~[i] = alpha_t M[i]                 for i in I^w only (selective decay)
 *   M[i]  = M~[i] + beta_t w_i * resid   resid per resid_mode (SDM_RESID_*)
 *   rows not in I^w keep their bits
 *   y_t   = sum_{i in I^r} r_i M[i]      read after the write
 *
 * state     : fp32 [B,H,N,d_v], updated in place (M_0 in, M_T out).  Calling
 *             again with the same buffer continues the sequence.
 * v         : [B,T,H,d_v], fp32 or bf16 per v_dtype.
 * alpha,beta: fp32 [B,T,H] per-head forget and input gates.
 * idx_w,w_w : int32 / fp32 [B,T,H,W] write slots and weights (from sdm_address).
 * idx_r,w_r : int32 / fp32 [B,T,H,R] read slots and weights.
 * y         : fp32 [B,T,H,d_v].
 * workspace : device scratch of at least sdm_scan_workspace_size(B,T,H,W,R)
 *             bytes, 16-byte aligned; contents need no initialisation.
 *             Calls sharing one workspace must not overlap on the GPU.
 * dev_err   : optional; SDM_DEVERR_INDEX_RANGE (that slot is read as zero and
 *             not written) and SDM_DEVERR_INDEX_REPEAT (result for that token
 *             unspecified, memory-safe).
 * Limits: 1 <= W, R <= 64; d_v % 4 == 0; N >= 1; B*T*H < 2e9.  state, y
 *         and fp32 v 16-byte aligned; bf16 v 8-byte; alpha, beta, idx, w
 *         4-byte.
 */
SDM_API int sdm_scan(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
             const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r, const float *w_r, int R,
             int B, int T, int H, int N, int d_v, int resid_mode, float *y, void *workspace,
             size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * Device bytes sdm_forward_host needs as staging for these sizes (two chunk
 * buffers of every input and output plus the scan's records); 0 for invalid
 * sizes.
 */
SDM_API size_t sdm_forward_host_workspace_size(int B, int T, int H, int sqrtN, int d_v, int W, int R, int v_dtype,
                                               int chunk_T);

/*
 * sdm_forward_host - one whole sparse step from HOST buffers: write and read
 * addressing ([SDM] "Product keys select addresses ...") and the scan ([SDM]
 * Eqs. 3-5), i.e. sdm_address twice and sdm_scan, with the per-step inputs
 * and y in host memory and the table resident on the device.
 *
 * The sequence is processed in chunks of at most chunk_T tokens: the first
 * and the last hold chunk_T/4 tokens (at least 1), so that the pipeline fills
 * and drains quickly, and the tokens between are split evenly (a sequence of
 * at most chunk_T tokens is one chunk).  Chunk c+1's inputs are copied in,
 * and its addressing runs, while chunk c is scanned and chunk c-1's y is
 * copied out (three internal streams for the copies and the addressing,
 * ordered by events after the work already queued on `stream`, and before
 * anything queued on `stream` afterwards; the scans run on `stream`).  Results are
 * bit-identical to one sdm_address/sdm_address/sdm_scan sequence on the whole
 * input (the scan continues its table across chunks).
 *
 * s1w, s2w, s1r, s2r : host fp32 [B,T,H,sqrtN] write and read score halves.
 * v          : host [B,T,H,d_v], fp32 or bf16 per v_dtype.
 * alpha, beta: host fp32 [B,T,H].
 * state      : DEVICE fp32 [B,H,N,d_v], N = sqrtN^2, updated in place.
 * y          : host fp32 [B,T,H,d_v], written when `stream` reaches the end
 *              of this call's work (synchronise `stream` before reading it).
 * workspace  : DEVICE scratch, 256-byte aligned, at least
 *              sdm_forward_host_workspace_size(...) bytes.
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to overlap compute; pageable memory works but serialises.
 * Limits and errors: those of sdm_address and sdm_scan.
 */
SDM_API int sdm_forward_host(const float *s1w, const float *s2w, const float *s1r, const float *s2r, const void *v,
                             int v_dtype, const float *alpha, const float *beta, int B, int T, int H, int sqrtN, int k,
                             int W, int R, int d_v, int resid_mode, float *state, float *y, int chunk_T,
                             void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * sdm_scan_noalloc - sdm_scan for callers that cannot give the library device
 * scratch memory.  The papers have no counterpart: this is an interface
 * convenience of this library, not a step of the method.
 *
 * Some callers cannot call cudaMalloc at the point where they run the scan:
 * hosts that hand out all device memory from their own pool and forbid raw
 * allocations once running (an allocation can synchronise the device and
 * fragments the pool), or plug-in code that receives only its input and
 * output buffers.  This entry point takes the same arguments as sdm_scan
 * minus the workspace, and keeps its scratch (the per-token records) in one
 * fixed 32 MiB array in device memory that every GPU loading this library
 * holds until the process exits.  It allocates nothing and frees nothing.
 *
 * Limit: sdm_scan_workspace_size(B,T,H,W,R) <= 32 MiB, i.e. B*T*H <= 99864
 * when W, R <= 16 (336 bytes per token-head) and B*T*H <= 25890 when either
 * is larger (1296 bytes); larger calls return SDM_ERR_SHAPE and launch nothing.
 * Set-up: the first call on a device looks up the array's device address
 * (with that device current) and remembers it for the current CUDA context; a
 * call from a new context on that device (after cudaDeviceReset, say) looks it
 * up again.  Make the first call in each context before any stream capture.
 * Sharing: all calls in the process share the one array, which keeps the last
 * call's contents (nothing in it needs clearing: every call rewrites what it
 * reads).  Calls that can overlap on the GPU - on different streams, or from
 * several host threads - race on it; serialise them.
 */
SDM_API int sdm_scan_noalloc(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
                     const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r, const float *w_r, int R,
                     int B, int T, int H, int N, int d_v, int resid_mode, float *y, int32_t *dev_err,
                     void *stream);

/*
 * Scratch bytes sdm_scan_chunked needs: one 60 KB record per chunk of 64
 * tokens and (batch, head).
 */
SDM_API size_t sdm_scan_chunked_workspace_size(int B, int T, int H, int W, int R);

/*
 * sdm_scan_chunked - the same scan as sdm_scan (shared residual or additive
 * write) in chunked form ([SDM] "Training parallelizes within chunks and
 * recurs across chunks", "Backup: sparse interactions drive the triangular
 * solve", App. A.1-A.2, Eq. 7).  Within a chunk of C = 64 tokens, with
 * lambda_i(s) the sum of log alpha over the tokens j <= i that write slot s:
 *   (I + A diag(beta)) u = v - p,   p_i = sum_n k_in e^{lambda_i(s_in)} M0[s_in],
 *   A[i,j] = sum_{s_in = s_jm} k_in k_jm e^{lambda_i(s) - lambda_j(s)} (j < i);
 *   y_i and the end-of-chunk rows follow from u (see chunked_scan.cu).
 * All the gathers of a chunk are independent, so the work inside a chunk is
 * parallel; chunks run in order.  Results equal sdm_scan's up to fp32
 * rounding.
 *
 * Arguments as sdm_scan; resid_mode SDM_RESID_SHARED or SDM_RESID_ADDITIVE
 * (SDM_RESID_PERSLOT: SDM_ERR_UNSUPPORTED); W, R <= 16; N <= 2^25.
 * workspace : sdm_scan_chunked_workspace_size() bytes, 16-byte aligned.
 * dev_err   : optional; SDM_DEVERR_INDEX_RANGE / SDM_DEVERR_INDEX_REPEAT.
 */
SDM_API int sdm_scan_chunked(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
                             const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r, const float *w_r,
                             int R, int B, int T, int H, int N, int d_v, int resid_mode, float *y, void *workspace,
                             size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * sdm_address_backward - gradient of the addressing weights with respect to
 * the two score halves ([SDM] Secs. 2 / 3.1).  The selection is piecewise
 * constant; the weights are w = softmax of the W selected sums
 * s_i = s1[a_i] + s2[b_i] (i = a_i sqrtN + b_i), so
 *   ds_i = w_i (dw_i - sum_j w_j dw_j),  ds1[a_i] += ds_i,  ds2[b_i] += ds_i
 * and every other score gets 0.
 *
 * idx, w : int32 / fp32 [B,T,H,W], as sdm_address returned them.
 * dw     : fp32 [B,T,H,W], dL/dw (e.g. from sdm_scan_backward).
 * ds1, ds2 : fp32 [B,T,H,sqrtN] out (overwritten).
 * dev_err : optional; SDM_DEVERR_INDEX_RANGE for an id outside [0, sqrtN^2).
 * Deterministic: one warp per row, slots added in order.
 */
SDM_API int sdm_address_backward(const int32_t *idx, const float *w, const float *dw, int B, int T, int H, int sqrtN,
                                 int W, float *ds1, float *ds2, int32_t *dev_err, void *stream);

/*
 * sdm_scan_train - sdm_scan that also keeps the undo log the backward needs
 * ([SDM] "Backup: undoing writes avoids repeated full-table snapshots",
 * App. A.3: the forward keeps only the sparse update information, T W d_v
 * values, instead of table snapshots).
 *
 * Arguments as sdm_scan, plus
 * undo : fp32 [B,T,H,W,d_v], 16-byte aligned, written: undo[b,t,h,j,:] is
 *        row idx_w[b,t,h,j] of the table as it was just before token t
 *        (before the decay).  For the 1.4B-layer shape: 61 KB per token-head.
 * y, the final table and the error codes are identical to sdm_scan's.
 */
SDM_API int sdm_scan_train(float *state, const void *v, int v_dtype, const float *alpha, const float *beta,
                           const int32_t *idx_w, const float *w_w, int W, const int32_t *idx_r, const float *w_r,
                           int R, int B, int T, int H, int N, int d_v, int resid_mode, float *y, float *undo,
                           void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * Scratch bytes sdm_scan_backward needs: per 32-column tile of d_v and per
 * token-head, R + W + 2 fp32 partial column sums, rounded up to 256.
 */
SDM_API size_t sdm_scan_backward_workspace_size(int B, int T, int H, int W, int R, int d_v);

/*
 * sdm_scan_backward - gradients of sdm_scan through its undo log, walking the
 * tokens backwards (same deck, App. A.3).  For token t (last to first), with
 * M = M_t and G = dL/dM_t:
 *   read   dL/dw_r[i] = <dy_t, M[idx_r[i]]>,   G[idx_r[i]] += w_r[i] dy_t
 *   write  M[i_j] = m_j + beta w_j rho_j with m_j = alpha undo_j and rho_j the
 *          residual of resid_mode; G_j = G[i_j]; g = beta sum_j w_j G_j:
 *          dL/dv_t = g;  dL/dbeta = sum_j w_j <G_j, rho_j>;
 *          dL/dw_w[j] = beta <G_j, rho_j> (- <g, m_j> for SDM_RESID_SHARED);
 *          dm_j = G_j - w_j g (shared) | G_j (1 - beta w_j) (per-slot) | G_j;
 *          dL/dalpha = sum_j <dm_j, undo_j>;  then G[i_j] = alpha dm_j and
 *          M[i_j] = undo_j.
 *
 * state  : fp32 [B,H,N,d_v]: M_T (as sdm_scan_train left it) in, M_0 out
 *          (bit-identical to the table before the forward).
 * dstate : fp32 [B,H,N,d_v]: dL/dM_T in (zeros if the loss ignores the final
 *          table), dL/dM_0 out.
 * v, v_dtype, alpha, beta, idx_w, w_w, W, idx_r, w_r, R, sizes, resid_mode :
 *          exactly as given to sdm_scan_train.
 * undo   : its log.   dy : fp32 [B,T,H,d_v], dL/dy.
 * dv     : fp32 [B,T,H,d_v] out.   dalpha, dbeta : fp32 [B,T,H] out.
 * dw_w   : fp32 [B,T,H,W] out.     dw_r : fp32 [B,T,H,R] out.
 * workspace : sdm_scan_backward_workspace_size() bytes.
 * dev_err : optional; SDM_DEVERR_INDEX_RANGE for an id outside [0, N) (skipped).
 * Work: one warp per (batch, head, 32 columns), one column per lane, then a
 *       deterministic reduction of the column sums over the tiles.
 */
SDM_API int sdm_scan_backward(float *state, float *dstate, const void *v, int v_dtype, const float *alpha,
                              const float *beta, const int32_t *idx_w, const float *w_w, int W,
                              const int32_t *idx_r, const float *w_r, int R, int B, int T, int H, int N, int d_v,
                              int resid_mode, const float *undo, const float *dy, float *dv, float *dalpha,
                              float *dbeta, float *dw_w, float *dw_r, void *workspace, size_t workspace_bytes,
                              int32_t *dev_err, void *stream);

/*
 * Scratch bytes gdn_scan needs.  At dk = dv = 128 (the chunked tensor-core
 * path) one tile set per chunk of 64 tokens (the operands of the
 * state-dependent products): GDN 131,328 bytes, KDA 147,968 bytes,
 * rounded up to 256 (about 2.1 / 2.3 KB per token-head).  Every other shape
 * and SDM_GDN_PATH=recurrent need none (0).
 */
SDM_API size_t gdn_scan_workspace_size(int B, int T, int H, int dk, int dv, int per_channel);

/*
 * gdn_scan - dense Gated DeltaNet (per_channel = 0) or Kimi Delta Attention
 * (per_channel = 1), [LAA] Eqs. 15-20, with the state stored key-major
 * (S = W^T, rows are key channels):
 *   S~   = D_alpha S              (GDN: every row scaled by alpha_t)
 *   pred = S~^T k_t               (decay-adjusted prediction)
 *   S    = S~ + beta_t k_t (v_t - pred)^T
 *   y_t  = S^T q_t                (unnormalised read after the write)
 * This is sdm_scan with every row selected, write weights k_t and read
 * weights q_t ([SDM] "A v1 inconsistency ...": the dense limit).
 *
 * state : fp32 [B,H,dk,dv] in place.
 * q, k  : bf16 [B,T,H,dk];  v : bf16 [B,T,H,dv].
 * alpha : fp32 [B,T,H] (GDN) or [B,T,H,dk] (KDA).   beta : fp32 [B,T,H].
 * y     : fp32 [B,T,H,dv].
 * workspace : device scratch of gdn_scan_workspace_size() bytes, 16-byte
 *           aligned, owned by the caller (NULL allowed when that size is 0);
 *           its contents on return are undefined.  Too small: SDM_ERR_INVALID_ARG.
 * dev_err : optional; SDM_DEVERR_TIMEOUT if a bounded wait of the tensor-core
 *           kernels gave up (outputs then invalid).
 * Kernels: GDN and KDA with dk = dv = 128 run chunkwise (64 tokens) on the
 *          tensor cores ([SDM] App. A.1-A.2, Eq. 7, dense case): a kernel
 *          parallel over all chunks prepares each chunk's state-independent
 *          operands in the workspace, then two CTAs per (batch, head), each
 *          owning half of the value columns, run the chunks in order with the
 *          state in registers (one CTA per (batch, head) when 2*B*H exceeds
 *          the SM count; SDM_GDN_CHAIN=pair|single forces one form).  KDA's per-channel
 *          decays sit inside the chunk's pair sums; each pair's decay is
 *          formed as a product of two decay ratios of at most 1 about a
 *          segment boundary, never with an inverse decay.  alpha must lie in
 *          (0, 1].  Other widths run token by token in fp32.
 * Limits: dk in {16, 32, 64, 128}; dv % 32 == 0, dv <= 256.  state and y
 *         16-byte aligned; q, k, v 16-byte aligned (dk, dv multiples of 8).
 */
SDM_API int gdn_scan(float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                     int per_channel, const float *beta, int B, int T, int H, int dk, int dv, float *y,
                     void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * gdn2_scan - GDN2, [LAA] "GDN2 separates key-side erase and value-side
 * write", Eqs. 21-24, state stored key-major (S = W^T):
 *   S~   = D_alpha S                  (per-key-channel decay, as KDA)
 *   e    = b (.) k,   z = w (.) v     (erase gate on keys, write gate on values)
 *   S    = S~ + k (z - S~^T e)^T      (the outer product takes k, not e)
 *   y_t  = S^T q_t
 * b = w = beta 1 is KDA.
 *
 * Chunk form (dk = dv = 128): the KDA chunk form of gdn_scan with the erase
 * rows e_i in place of beta_i k_i (A_ij = sum_r e_ir k_jr e^{lambda_ir -
 * lambda_jr}, W = (I + A)^-1 (e (.) e^{lambda})) and Ut = (I + A)^-1 z, on
 * the same two tensor-core kernels; other widths run token by token.
 *
 * state   : fp32 [B,H,dk,dv] in place.
 * q, k    : bf16 [B,T,H,dk];  v : bf16 [B,T,H,dv].
 * alpha   : fp32 [B,T,H,dk] in (0, 1].  b_erase : fp32 [B,T,H,dk].  w_write : fp32 [B,T,H,dv].
 * y       : fp32 [B,T,H,dv].
 * workspace : device scratch of gdn2_scan_workspace_size() bytes, 16-byte
 *           aligned (NULL allowed when that size is 0); contents undefined on
 *           return.  Too small: SDM_ERR_INVALID_ARG.
 * dev_err : optional; SDM_DEVERR_TIMEOUT if a bounded wait of the tensor-core
 *           kernels gave up (outputs then invalid).
 * Limits: dk in {16, 32, 64, 128}; dv % 32 == 0, dv <= 256; every tensor
 *         16-byte aligned.
 */
SDM_API size_t gdn2_scan_workspace_size(int B, int T, int H, int dk, int dv);
SDM_API int gdn2_scan(float *state, const uint16_t *q, const uint16_t *k, const uint16_t *v, const float *alpha,
                      const float *b_erase, const float *w_write, int B, int T, int H, int dk, int dv, float *y,
                      void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream);

/*
 * Scratch bytes sse_scan needs for these sizes and write mode: one routing
 * record per token (selected partitions, their gates, and the max and
 * inverse normaliser of the row softmax), rounded up to 256 bytes; when the
 * call takes the chunked prefill path (below) also, per (batch, head), the
 * visit lists grouped by partition, one operand unit per chunk of 64 visits
 * (at most ceil(T/64) + floor((topk*T + 63*N)/64) units; 99,072 bytes each
 * for the additive write, 148,224 for the delta write), and one staging row
 * of d fp32 per visit.  Read SDM_SSE_PATH at the call, so query it under the
 * same environment as sse_scan.
 */
SDM_API size_t sse_scan_workspace_size(int B, int T, int H, int N, int topk, int c, int d, int write_mode);

/*
 * sse_scan - Sparse State Expansion, [SSE] Eqs. 9-14, with N routed
 * partitions plus one always-active shared partition (index N):
 *   e_t  = softmax(route_t) over all N partitions (not renormalised)
 *   T_t  = top-k of route_t (value descending, ties to the lower index)
 *   kk_t = softmax(k_logits_t) over the c rows of a partition
 *   for p in T_t (gate g = e_t[p]) and p = N (g = 1):
 *       S^p[j,:] = alpha_t[j] S^p[j,:] + g kk_t[j] r_p      (j < c)
 *       r_p = v_t                                  (write_mode SSE_WRITE_ADDITIVE)
 *       r_p = v_t - sum_j kk_t[j] alpha_t[j] S^p[j,:]   (SSE_WRITE_DELTA: the
 *             partition's rows share one residual, the [SDM] Fig. 2 shared
 *             residual with row weights kk and strength g; the SSE deck names
 *             delta-rule transitions as follow-up work without a formula)
 *   unvisited partitions keep their bits (their decay clock stops)
 *   y_t  = sum_p g_p sum_j q_t[j] S^p[j,:]                 (after the write)
 *
 * Paths.  Either write with c = d = 128 and T >= 64 runs as a prefill by
 * varlen grouping ([SSE] "Varlen groups tokens while preserving causal
 * order"): the visits of each partition gathered in time order, each group
 * run in chunks of 64 visits on the tensor cores, and every token's visit
 * outputs summed in a fixed order (routed ranks, then the shared partition),
 * so results are deterministic.  The additive write takes the chunkwise GLA
 * form; the delta write is the gated delta rule with a decay per key row, so
 * it takes the chunk form of the per-channel-decay (KDA) scan with keys kk,
 * write strength g and every read scaled by g (the shared partitions'
 * chains, the longest, on CTA pairs as gdn_scan's; SDM_GDN_CHAIN=single puts
 * every chain on one CTA).  Everything else runs token
 * by token with the partitions resident in shared memory.  The
 * environment variable SDM_SSE_PATH=recurrent forces the token-by-token
 * kernel; SDM_SSE_PATH=chunk the chunked path for any T (same shape rules).
 *
 * state       : fp32 [B,H,N+1,c,d] in place.
 * route_logits: fp32 [B,T,H,N].  k_logits : fp32 [B,T,H,c].
 * q           : bf16 [B,T,H,c].  v : bf16 [B,T,H,d].  alpha : fp32 [B,T,H,c].
 * write_mode  : SSE_WRITE_ADDITIVE or SSE_WRITE_DELTA (else SDM_ERR_UNSUPPORTED).
 * y           : fp32 [B,T,H,d].
 * sel_out     : optional int32 [B,T,H,topk], the selected partitions in rank order.
 * workspace   : device scratch of at least sse_scan_workspace_size() bytes,
 *               16-byte aligned.
 * dev_err     : optional; SDM_DEVERR_NONFINITE if a logit is NaN/inf;
 *               SDM_DEVERR_TIMEOUT if a tensor-core wait of the chunked path
 *               gave up (its outputs are then invalid).
 * Limits: 1 <= topk <= N <= 64, topk <= 8; c % 16 == 0, 16 <= c <= 128;
 *         d % 16 == 0; B*T*H*(topk+1) < 2^31, T < 2^27.  state, k_logits,
 *         alpha, q, v 16-byte aligned; y 4-byte aligned (16 on the chunked
 *         path).  Token by token, (N+1)*c*16 fp32 must fit in shared memory.
 */
SDM_API int sse_scan(float *state, const float *route_logits, int topk, const float *k_logits, const uint16_t *q,
             const uint16_t *v, const float *alpha, int write_mode, int B, int T, int H, int N, int c, int d,
             float *y, int32_t *sel_out, void *workspace, size_t workspace_bytes, int32_t *dev_err, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SDM_H_ */
