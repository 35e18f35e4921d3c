/*
 * xhc.h -- C ABI of the xHC per-sublayer residual-stream update on one GPU
 * (NVIDIA B300, sm_103a).
 *
 * Method: "xHC: Expanded Hyper-Connections" (qingkeai.online research
 * retrospective).  Per token the residual state is N streams of width C
 * (section "Scaling N"); the sublayer input is a dense read over all N
 * streams weighted by H^pre (section "Dense read, sparse write"); the
 * sublayer output `out` is expanded along the sequence by three causal
 * depthwise convolutions of kernel size 4, 8 and 12 stacked with the raw
 * output (section "Temporal Feature Augmentation"); only k active streams are
 * rewritten, by a Sinkhorn-normalised k x k mix H^res of the active streams
 * plus an H^post combination of the four components; the other streams pass
 * through unchanged (sections "Scaling N", "Dense read, sparse write").
 *
 * Formulation used (the pages' formulas were lost; these choices are fixed by
 * the project specification), per token with v = vec X (length N*C, index
 * n*C + c), P = N + 4k + k*k:
 *   rstd = 1 / sqrt(mean(v^2) + eps)         z = rstd * (W v),  W: [P, N*C]
 *   hpre = sigmoid(z[0:N])                    hpost[i][c] = sigmoid(z[N + 4i + c])
 *   Hres = Sinkhorn(exp(Z - max Z)), Z[i][j] = z[N + 4k + k*i + j];
 *          each Sinkhorn iteration normalises rows, then columns
 *   x_in = sum_n hpre[n] X[n]
 *   u0 = out[t];  u_j[t][c] = sum_{tau < K_j} w_j[c][tau] out[t - tau][c]
 *          (K = 4, 8, 12; zero before the start of each sequence)
 *   X'[a_i] = sum_j Hres[i][j] X[a_j] + sum_c hpost[i][c] u_c   (i < k)
 *   X'[n]   = X[n] for streams n not in the active list a.
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller, except the
 *     active-index list `idx`, which is a HOST array of k int32.
 *   - Layouts are dense row-major: X, X', dX' and dX are [B, S, N, C];
 *     out, x_in, dx_in, dout are [B, S, C]; conv weights w4, w8, w12 are
 *     [C, 4], [C, 8], [C, 12] (tap tau multiplies out[t - tau]); W and dW are
 *     [P, N*C]; hpre [B, S, N]; hpost [B, S, k, 4]; hres [B, S, k, k];
 *     saved [B, S, P + 1] holds the logits z followed by rstd.
 *   - Activations (X, out, x_in, dX', dx_in, dX, dout, u, saved_active) use
 *     the shape's dtype (fp32 or bf16); W, conv weights, coefficients and
 *     weight gradients are always fp32.  Arithmetic accumulates in fp32;
 *     bf16 results are rounded to nearest even.
 *   - Every pointer must be 16-byte aligned; C * sizeof(dtype) must be a
 *     multiple of 16.
 *   - Work is enqueued asynchronously on `stream`; nothing synchronises the
 *     host.  Gradients are written, not accumulated.
 *   - On any error status nothing has been launched, except XHC_ERR_CUDA,
 *     which reports a launch failure (see xhc_last_cuda_error).
 *   - The library allocates no device memory.  Entry points that need
 *     scratch take a caller workspace and report its size.
 *   - Limits: 1 <= N <= 16, 1 <= k <= min(N, 4), 0 <= sinkhorn_iters <= 64.
 *     B * S == 0 is a valid empty call that launches nothing.
 */
#ifndef XHC_H_
#define XHC_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* xhc_stream_t; /* same type as cudaStream_t */

enum {
  XHC_F32 = 0,
  XHC_BF16 = 1
};

enum {
  XHC_OK = 0,
  XHC_ERR_SHAPE = 1,     /* bad B, S, N, C, k, iteration count or eps */
  XHC_ERR_INDEX = 2,     /* idx missing, repeated or outside [0, N) */
  XHC_ERR_ALIGN = 3,     /* a pointer is not 16-byte aligned */
  XHC_ERR_DTYPE = 4,     /* unsupported dtype */
  XHC_ERR_WORKSPACE = 5, /* workspace missing or too small */
  XHC_ERR_CUDA = 6,      /* a kernel launch failed */
  XHC_ERR_TIMEOUT = 7,   /* a bounded device-side wait gave up */
  XHC_ERR_ARG = 8        /* a required pointer is NULL */
};

typedef struct xhc_shape {
  int B, S, N, C, k;
  int dtype;          /* XHC_F32 or XHC_BF16 */
  int sinkhorn_iters; /* 20 in the method's setting */
  float eps;          /* rmsnorm epsilon, 1e-6 in the method's setting */
  int gram_schmidt;   /* 0: write back u_0..u_3 as they are (default);
                         1: orthogonalise them first by modified Gram-Schmidt
                         (section "Conv / Gram-Schmidt"), see
                         xhc_sublayer_fwd.  Other values: XHC_ERR_SHAPE. */
} xhc_shape_t;

/* Human-readable name of a status code.  Never NULL. */
const char* xhc_status_string(int status);

/* cudaError_t of the most recent XHC_ERR_CUDA in this process (0 if none). */
int xhc_last_cuda_error(void);

/*
 * Status of the library's bounded device-side waits.  Synchronises `stream`,
 * returns XHC_ERR_TIMEOUT if a kernel gave up waiting since the last call (the
 * affected outputs are then undefined) and clears the record; XHC_OK
 * otherwise.
 */
int xhc_device_status(xhc_stream_t stream);

/*
 * Limit of the library's bounded device-side waits (mbarrier waits of the
 * tensor-core kernels), in nanoseconds, for kernels launched after the call;
 * 0 restores the default of 2 s.  A wait that runs out records
 * XHC_ERR_TIMEOUT for xhc_device_status, and every wait of the kernels in
 * flight then gives up at once; before a kernel ends, each of its roles waits
 * (again within the limit) for the asynchronous copies and tensor-core
 * operations it issued, so nothing is left writing its shared memory or
 * tensor memory.  Synchronises the device (call it between steps).  The
 * pages have no counterpart: failure detection of this library.
 * Returns XHC_OK, or XHC_ERR_CUDA.
 */
int xhc_set_wait_limit_ns(unsigned long long ns);

/*
 * Failure-detection test hook (the pages have no counterpart): the next
 * coefficient projection this process launches (the first kernel of
 * xhc_coeffs, xhc_sublayer_fwd and the other forward entry points) issues
 * none of its loads, so the waits of its tensor-core and math roles run out
 * after the wait limit with nothing in flight.  That call's outputs are
 * undefined; xhc_device_status then returns XHC_ERR_TIMEOUT and clears the
 * record, and later calls run normally.  Returns XHC_OK.
 */
int xhc_debug_starve_next_projection(void);

/*
 * Debug build record (the pages have no counterpart; a stand-in for a
 * memory checker).  libxhc_debug.so, built with -DXHC_DEBUG, checks every
 * global load and store of the forward update and the backward column pass
 * against the extents of the buffers of that launch (as the shape gives
 * them); an access outside all of them is skipped and the first one is
 * recorded.  This call synchronises the device and returns 1 with the
 * source line of the access in *line and its address in *address (then
 * clears the record), 0 when nothing was recorded, -1 in a release build
 * (which checks nothing), -2 on a CUDA error.  line and address may be NULL.
 */
int xhc_debug_record(unsigned long long* line, unsigned long long* address);

/*
 * Self-test of the debug build's checker: one checked 4-byte load from
 * byte 128 of `buf` with only the first 64 bytes of `buf` registered, result
 * to out[0].  `buf` must hold at least 256 bytes (so that even an unchecked
 * load stays inside it) and be 16-byte aligned; `out` at least 4 bytes.  A
 * debug build skips the load (out[0] = 0) and records it; a release build
 * performs it.  Asynchronous on `stream`.  XHC_OK, XHC_ERR_ALIGN or
 * XHC_ERR_CUDA.
 */
int xhc_debug_selftest(const float* buf, float* out, xhc_stream_t stream);

/* Number of projection rows P = N + 4k + k^2 for a shape. */
int xhc_num_logits(const xhc_shape_t* sh);

/*
 * xhc_coeffs -- coefficient generation and dense read.
 * Section "Scaling N" (H^pre, H^post, H^res from the state; Sinkhorn) and
 * section "Dense read, sparse write" (the input is read from all N streams).
 *   X      [B,S,N,C] dtype, read.
 *   W      [P, N*C] fp32, read.
 *   hpre   [B,S,N], hpost [B,S,k,4], hres [B,S,k,k] fp32, written.
 *   saved  [B,S,P+1] fp32 (z then rstd), written; may be NULL.
 *   x_in   [B,S,C] dtype, written; may be NULL (no dense read).
 */
int xhc_coeffs(const xhc_shape_t* sh, const void* X, const float* W,
               float* hpre, float* hpost, float* hres, float* saved,
               void* x_in, xhc_stream_t stream);

/*
 * xhc_tfa -- Temporal Feature Augmentation components u_1, u_2, u_3.
 * Section "Temporal Feature Augmentation": three causal depthwise
 * convolutions, kernel sizes 4, 8, 12, each channel independent along the
 * sequence; u_0 is `out` itself and is not written.
 *   out          [B,S,C] dtype, read.
 *   w4, w8, w12  [C,4], [C,8], [C,12] fp32, read; all three required.
 *   u            [3,B,S,C] dtype, written (u_1, u_2, u_3).
 */
int xhc_tfa(const xhc_shape_t* sh, const void* out, const float* w4,
            const float* w8, const float* w12, void* u, xhc_stream_t stream);

/*
 * xhc_sparse_update -- the sparse write given coefficients.
 * Section "Dense read, sparse write": only the k streams in idx are
 * rewritten; section "Temporal Feature Augmentation" for the components.
 *   X_in   [B,S,N,C] dtype, read.
 *   X_out  [B,S,N,C] dtype, written.  X_out == X_in updates in place and
 *          writes only the k active rows; otherwise the N-k inactive rows are
 *          copied as well.  Partial overlap is not allowed.
 *   out    [B,S,C] dtype, read.
 *   w4, w8, w12  fp32 conv weights, or all three NULL for no convolution
 *          branches (u_1 = u_2 = u_3 = 0).
 *   hpost  [B,S,k,4] fp32, hres [B,S,k,k] fp32, read.
 *   idx    host int32[k]: slot i rewrites stream idx[i].
 */
int xhc_sparse_update(const xhc_shape_t* sh, const void* X_in, void* X_out,
                      const void* out, const float* w4, const float* w8,
                      const float* w12, const float* hpost, const float* hres,
                      const int32_t* idx, xhc_stream_t stream);

/*
 * Workspace of the fused forward (bytes).  xhc_fwd_workspace_bytes() is enough
 * for every call of the shape; xhc_fwd_workspace_need() is what a call needs
 * when the caller keeps the logits (keeps_saved != 0: `saved` is non-NULL) or
 * not.  The bf16 path uses it for a per-token coefficient block (48 fp32 per
 * token) and a bf16 hi/lo split copy of W (2 x 48 x N*C bf16), and, when
 * `saved` is NULL, for the logits (P + 1 fp32 per token).
 */
size_t xhc_fwd_workspace_bytes(const xhc_shape_t* sh);
size_t xhc_fwd_workspace_need(const xhc_shape_t* sh, int keeps_saved);

/*
 * xhc_sublayer_fwd -- the whole per-sublayer update: coefficients, dense
 * read, TFA and sparse write (all sections cited above).
 *   With sh->gram_schmidt = 1 the four components are orthogonalised per
 *   token before the write-back (section "Conv / Gram-Schmidt"): u_0 is kept
 *   and each of u_1, u_2, u_3 in turn loses its projection onto every
 *   orthogonalised component before it; a projection onto a component whose
 *   residual is at most 1e-6 of its own squared norm (a zero or dependent
 *   component) is skipped.  The library forms the per-token Gram matrix of
 *   the components and applies the steps to the coefficients (exact up to
 *   rounding).  Supported with conv weights on the bf16 path: the forward
 *   for C a multiple of 64, the backward for C a multiple of 128
 *   (XHC_ERR_DTYPE otherwise); without conv weights it changes nothing.  The
 *   forward workspace grows by 48 bytes per token per 256 channels.
 *   xhc_tfa and xhc_sparse_update (with conv weights) return XHC_ERR_ARG for
 *   such a shape: they handle raw components only.
 *   X_in, X_out  as in xhc_sparse_update (X_out == X_in: in place).
 *   out, w4, w8, w12, idx  as in xhc_sparse_update.
 *   W      [P, N*C] fp32.
 *   x_in   [B,S,C] dtype, written; may be NULL.
 *   saved  [B,S,P+1] fp32 (z, rstd), written; may be NULL.
 *   saved_active  [B,S,k,C] dtype: the k active rows of X_in before the
 *          update (slot order), written; may be NULL.  Needed by the backward
 *          when the state is updated in place.
 *   workspace, ws_bytes  at least xhc_fwd_workspace_need(sh, saved != NULL)
 *          bytes (NULL/0 when that is 0); xhc_fwd_workspace_bytes() always
 *          suffices.
 */
int xhc_sublayer_fwd(const xhc_shape_t* sh, const void* X_in, void* X_out,
                     const void* out, const float* w4, const float* w8,
                     const float* w12, const float* W, const int32_t* idx,
                     void* x_in, float* saved, void* saved_active,
                     void* workspace, size_t ws_bytes, xhc_stream_t stream);

/*
 * xhc_sublayer_fwd_noalloc -- xhc_sublayer_fwd for callers that cannot
 * allocate device memory.  The paper has no counterpart; this is a library
 * convenience.  Some callers only receive their input and output buffers and
 * may not call the CUDA allocator (a plugin or custom-op hook running inside
 * another framework's memory pool, a C caller without a workspace of its
 * own).  This entry point takes the same arguments as xhc_sublayer_fwd minus
 * the workspace, and uses a fixed 32 MiB scratch area built into the library
 * (a device array that every GPU which loads the library keeps until the
 * process exits) in place of the workspace.
 *   Limit: xhc_fwd_workspace_need(sh, saved != NULL) must be at most 32 MiB.
 *          At N = 16, k = 4 in bf16 a call needs 3072 * C bytes (a bf16 split
 *          copy of W) plus 192 bytes per token with `saved` given, 388
 *          without: at C = 2048 about 141,000 and 70,000 tokens.  Larger
 *          calls return XHC_ERR_WORKSPACE before touching the GPU.
 *   The first call on each device looks up the scratch address on that
 *   device; make that first call before any stream capture.  The lookup
 *   makes the driver load the library's device code on that device, which
 *   reserves the 32 MiB there (the driver's doing, not an allocation call by
 *   this library): when the device's memory is already taken, for example
 *   by a caching pool, that first call can fail with XHC_ERR_CUDA
 *   (out of memory).  The address is cached per device and context; after a
 *   cudaDeviceReset the next call looks it up again in the new context.
 *   Every call shares the one scratch area: calls whose work overlaps on the
 *   GPU (different streams, or different threads) race and must be ordered
 *   by the caller.  The area keeps the last call's contents; nothing in it
 *   needs to start at zero.
 *   No cudaMalloc, cudaFree or other allocating routine is called.
 */
int xhc_sublayer_fwd_noalloc(const xhc_shape_t* sh, const void* X_in,
                             void* X_out, const void* out, const float* w4,
                             const float* w8, const float* w12, const float* W,
                             const int32_t* idx, void* x_in, float* saved,
                             void* saved_active, xhc_stream_t stream);

/*
 * xhc_sublayer_fwd_routed -- the sublayer update with per-token active sets
 * chosen by a router (section "Dense read, sparse write").  Per token:
 *   scores  s = sigmoid(W_r . LN(vec X)), LN over all N*C entries, no gain
 *           or bias, eps = sh->eps;
 *   slots   the n_fixed streams `fixed` (host, ordered) first, then the top
 *           k - n_fixed other streams by score (descending, ties to the lower
 *           index);
 *   update  as xhc_sublayer_fwd with those slots, a routed slot's write-back
 *           sum_c H^post[i][c] u_c multiplied by its stream's score.
 *   W_r      [N, N*C] fp32, read.
 *   tok_idx  [B,S,k] int32 device, written: the slots.
 *   rrec     [B,S,2N+2] fp32 device, written: per token the scores s (N),
 *            the logits W_r . LN(vec X) (N), the LayerNorm mean and its
 *            standard deviation sqrt(var + eps) (the backward reads them).
 *   saved_active  [B,S,k,C], the active rows before the update in slot order
 *            (may be NULL).
 *   workspace, ws_bytes  at least xhc_fwd_routed_workspace_bytes() bytes
 *            (required).
 * Other arguments as in xhc_sublayer_fwd.  bf16 with C a multiple of 64
 * (XHC_ERR_DTYPE otherwise); not combined with gram_schmidt (XHC_ERR_ARG);
 * bad `fixed` lists give XHC_ERR_INDEX.  The router's logits come from the
 * same projection pass as the coefficients (W_r adds N rows to it).
 */
size_t xhc_fwd_routed_workspace_bytes(const xhc_shape_t* sh);
int xhc_sublayer_fwd_routed(const xhc_shape_t* sh, const void* X_in,
                            void* X_out, const void* out, const float* w4,
                            const float* w8, const float* w12, const float* W,
                            const float* W_r, const int32_t* fixed,
                            int n_fixed, void* x_in, float* saved,
                            void* saved_active, int32_t* tok_idx,
                            float* rrec, void* workspace, size_t ws_bytes,
                            xhc_stream_t stream);

/*
 * xhc_stack_fwd -- forward of a stack of L sublayers on one state, in place,
 * with each sublayer's update fused with the next sublayer's coefficient
 * projection (section "Beyond N=16": xHC-Flash reorders the reads and writes
 * of consecutive sublayers to lower the traffic per sublayer).  Sublayer l
 * reads the state that sublayer l - 1 wrote and applies the update of
 * xhc_sublayer_fwd with its own out[l], conv weights, W[l] and index list.
 * One pass over the state per sublayer: it forms sublayer l's dense read and
 * sparse write and, from the updated tile still on chip, sublayer l+1's
 * coefficients.  A first pass computes sublayer 0's coefficients.
 *   X        [B,S,N,C] bf16 device, read and written (the final state).
 *   out      host array of L device pointers, out[l] [B,S,C] bf16.
 *   w4, w8, w12  NULL, or host arrays of L device pointers ([C,4], [C,8],
 *            [C,12] fp32); per sublayer all three or none (no TFA).
 *   W        host array of L device pointers, W[l] [P, N*C] fp32.
 *   idx      host int32 [L*k]: sublayer l's slots at idx + l*k.
 *   x_in     NULL, or host array of L device pointers (entries may be NULL):
 *            sublayer l's dense read [B,S,C] bf16, written.
 *   saved    NULL, or host array of L device pointers (entries may be NULL):
 *            sublayer l's logits and rstd [B,S,P+1] fp32, written.
 *   workspace, ws_bytes  at least xhc_stack_fwd_workspace_bytes() bytes.
 * bf16 only (XHC_ERR_DTYPE), C a multiple of 64 and P <= 48
 * (XHC_ERR_SHAPE); L >= 1 (XHC_ERR_ARG).  With sh->gram_schmidt each
 * sublayer's components are orthogonalised as in xhc_sublayer_fwd.  The
 * state between sublayers is the bf16 state in memory.  Inference form: the
 * old active rows are not saved (training uses xhc_sublayer_fwd per
 * sublayer).  On error nothing is launched.
 */
size_t xhc_stack_fwd_workspace_bytes(const xhc_shape_t* sh);
int xhc_stack_fwd(const xhc_shape_t* sh, int L, void* X,
                  const void* const* out, const float* const* w4,
                  const float* const* w8, const float* const* w12,
                  const float* const* W, const int32_t* idx,
                  void* const* x_in, float* const* saved, void* workspace,
                  size_t ws_bytes, xhc_stream_t stream);

/*
 * xhc_sublayer_bwd_routed -- exact reverse mode of xhc_sublayer_fwd_routed
 * (the active sets are the forward's, a constant; unchosen scores get no
 * gradient).
 *   X_state  [B,S,N,C] dtype.  If saved_active is NULL it is the state BEFORE
 *            the update and is only read.  Otherwise it is the state AFTER an
 *            in-place forward (X_out == X_in): the call first writes the
 *            saved old active rows back at each token's slots, so that on
 *            return X_state holds the state before the update (what the
 *            backward of the sublayer below reads).  Slot entries of tok_idx
 *            outside [0, N) are skipped by that write.
 *   saved_active  [B,S,k,C] dtype from the in-place forward, or NULL.
 *   saved, tok_idx, rrec  the forward's outputs (required).
 *   dW_r     [N, N*C] fp32, written.
 * Other arguments as in xhc_sublayer_bwd.  bf16 with C a multiple of 128 and
 * P + N <= 64 (XHC_ERR_DTYPE otherwise); workspace at least
 * xhc_bwd_routed_workspace_bytes() bytes.
 */
size_t xhc_bwd_routed_workspace_bytes(const xhc_shape_t* sh);
int xhc_sublayer_bwd_routed(const xhc_shape_t* sh, void* X_state,
                            const void* saved_active, const void* out, const float* w4, const float* w8,
                            const float* w12, const float* W,
                            const float* W_r, const int32_t* fixed,
                            int n_fixed, const float* saved,
                            const int32_t* tok_idx, const float* rrec,
                            const void* dXp, const void* dx_in, void* dX,
                            void* dout, float* dw4, float* dw8, float* dw12,
                            float* dW, float* dW_r, void* workspace,
                            size_t ws_bytes, xhc_stream_t stream);

/* Workspace the backward needs (bytes). */
size_t xhc_bwd_workspace_bytes(const xhc_shape_t* sh);

/*
 * xhc_sublayer_bwd -- exact reverse mode of xhc_sublayer_fwd, including the
 * pass back through every Sinkhorn iteration.
 *   X_state  [B,S,N,C] dtype.  If saved_active is NULL it is the state BEFORE
 *            the update; otherwise it is the state AFTER the in-place update
 *            and the k old active rows are read from saved_active.
 *   saved_active  [B,S,k,C] dtype or NULL (see X_state).
 *   out, w4, w8, w12, W, idx  the forward's inputs (conv weights all NULL for
 *            no convolution branches).
 *   saved    [B,S,P+1] fp32 from the forward, or NULL to recompute it.
 *   dXp      [B,S,N,C] dtype: dL/dX', read.
 *   dx_in    [B,S,C] dtype: dL/dx_in, or NULL when x_in carries no gradient.
 *   dX       [B,S,N,C] dtype: dL/dX, written.  dX must not be dXp
 *            (XHC_ERR_ARG).
 *   With sh->gram_schmidt = 1 the gradient is taken back through the
 *   Gram-Schmidt step of the forward (same support as xhc_sublayer_fwd).
 *   dout     [B,S,C] dtype: dL/dout, written.
 *   dw4, dw8, dw12  [C,4], [C,8], [C,12] fp32, written (NULL when the conv
 *            weights are NULL).
 *   dW       [P, N*C] fp32, written.
 *   workspace, ws_bytes  at least xhc_bwd_workspace_bytes() bytes.
 */
int xhc_sublayer_bwd(const xhc_shape_t* sh, const void* X_state,
                     const void* saved_active, const void* out,
                     const float* w4, const float* w8, const float* w12,
                     const float* W, const int32_t* idx, const float* saved,
                     const void* dXp, const void* dx_in, void* dX, void* dout,
                     float* dw4, float* dw8, float* dw12, float* dW,
                     void* workspace, size_t ws_bytes, xhc_stream_t stream);

/*
 * xhc_hres_active_weights -- H^res logits from the k active streams only.
 * Section "Dense read, sparse write": only the k active streams take part in
 * the residual mixing, so its logits can be generated from their k*C state
 * entries alone (cost O(k^3 C) instead of growing with N).  This builds the
 * full projection that every other entry point takes, so the variant runs
 * through them unchanged:
 *   W_pp   [N + 4k, N*C] fp32, read: the H^pre and H^post rows (whole state).
 *   W_ra   [k*k, k*C] fp32, read: the H^res rows over vec(X[a_0], ..,
 *          X[a_{k-1}]) (slot order of idx).
 *   idx    host, k entries (as in xhc_sparse_update).
 *   W      [P, N*C] fp32, written: W_pp, then the H^res rows with W_ra in the
 *          columns of the active streams and zeros elsewhere.
 * rstd stays the rmsnorm scale of the whole state.
 */
int xhc_hres_active_weights(const xhc_shape_t* sh, const float* W_pp,
                            const float* W_ra, const int32_t* idx, float* W,
                            xhc_stream_t stream);

/*
 * xhc_hres_active_grad -- dL/dW_ra [k*k, k*C] fp32 (written) from the
 * gradient dW [P, N*C] (read) of the projection built by
 * xhc_hres_active_weights: the active streams' columns of its H^res rows.
 */
int xhc_hres_active_grad(const xhc_shape_t* sh, const float* dW,
                         const int32_t* idx, float* dW_ra, xhc_stream_t stream);

/*
 * xhc_copy -- device-to-device copy of `bytes` bytes with 16-byte vector
 * loads and stores.  Used to measure the HBM copy bandwidth in the same
 * process as the update kernels.  Both pointers 16-byte aligned, bytes a
 * multiple of 16; the ranges must not overlap.
 */
int xhc_copy(const void* src, void* dst, size_t bytes, xhc_stream_t stream);

/*
 * Optional per-kernel timing.  While enabled (on != 0), every kernel the
 * library launches is bracketed by two CUDA events recorded on the stream it
 * runs on.  xhc_timing_collect waits for the recorded events, writes for each
 * distinct kernel name its launch count and total milliseconds (names: up to
 * max_kernels entries of 48 bytes each, NUL-terminated), clears the record
 * and returns the number of entries written (a negative status on a CUDA
 * error).  Any of names / counts / total_ms may be NULL.  Not thread-safe:
 * enable it only around single-threaded use of the library.
 */
int xhc_timing_enable(int on);
int xhc_timing_collect(char* names, int* counts, float* total_ms, int max_kernels);

#ifdef __cplusplus
}
#endif

#endif /* XHC_H_ */
