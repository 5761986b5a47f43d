/*
 * osattn.h - C ABI of libosattn, a fused scaled-dot-product attention forward
 * pass for one NVIDIA GB300 (sm_103a), built on the one-pass online-softmax
 * normaliser, with its backward pass and the standalone row softmax.
 *
 * Sources (cited by page title and section):
 *   [Ch6]  "CUDA 算子工程：手写 FlashAttention v2 之路", chapter 6
 *          "Softmax 与 Online Softmax" (yangyitao.com): the online (m, l)
 *          recurrence (§6.3.1), the guarded combine (§6.4, §6.4.1), LSE
 *          (§6.5), the blocked attention loop (§6.6), the fused additive
 *          mask (§6.7.3).
 *   [XXQK] m.xxqk.cn/news/563265 (article on parallel softmax and
 *          FlashAttention): the attention problem statement (§1.1), the
 *          inner loop with scale and mask and the single final O / l (§4.1),
 *          the causal diagonal-block pitfall (§6.3).
 *
 * Entry points:
 *   forward        osattn_fwd, osattn_fwd_strided (any (b, h, row) strides),
 *                  osattn_fwd_splitkv / _noalloc (key axis split and merged),
 *                  osattn_fwd_offload (host-memory tensors, pipelined copies)
 *   backward       osattn_bwd, osattn_bwd_strided, osattn_bwd_offload
 *   row softmax    osattn_softmax_rows, osattn_softmax_rows_offload
 *   helpers        workspace sizes, status strings, the device status word,
 *                  the version, and test hooks for the bounded waits
 *
 * Every entry point is callable from C; no C++ or framework types cross it.
 */
#ifndef OSATTN_H
#define OSATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define OSATTN_VERSION 1

/* Element types of Q, K, V and O (LSE is always fp32). */
#define OSATTN_BF16 0 /* bfloat16; runs on the tcgen05 tensor-core kernel */
#define OSATTN_FP32 1 /* float32; runs on the SIMT kernel (full fp32 FMA) */
#define OSATTN_FP16 2 /* IEEE float16; runs on the tcgen05 tensor-core kernel */

/* Status codes. */
#define OSATTN_OK 0
#define OSATTN_ERR_INVALID_ARG 1 /* null pointer, size < 1, misalignment, non-finite scale */
#define OSATTN_ERR_UNSUPPORTED 2 /* d or dtype outside the supported set */
#define OSATTN_ERR_CUDA 3        /* a CUDA call failed (launch, attribute, tensor map) */
#define OSATTN_ERR_TIMEOUT 4     /* a device-side wait ran past its limit (reported by
                                    osattn_get_device_status only) */
#define OSATTN_ERR_SCRATCH_LIMIT 5 /* osattn_fwd_splitkv_noalloc: the problem's partials need
                                      more than OSATTN_NOALLOC_SCRATCH_BYTES */

/*
 * osattn_fwd - attention forward with online softmax.
 *
 * Computes, for every batch b < B, head h < H and query row i < Nq,
 *     s_j    = scale * <Q[b,h,i,:], K[b,h,j,:]>                  ([XXQK] §1.1)
 *     J      = { j < min(max(key_len[b], 0), Nkv) and (causal == 0 or j <= i) }
 *     O[b,h,i,:] = sum_{j in J} e^{s_j} V[b,h,j,:] / sum_{j in J} e^{s_j}
 *     LSE[b,h,i] = log sum_{j in J} e^{s_j}        (natural log, [Ch6] §6.5)
 * by streaming K/V tiles with the running row max m and adjusted sum l
 * ([Ch6] §6.3.1, §6.6), rescaling the accumulated O only when m changes and
 * dividing by l once at the end ([XXQK] §4.1).  A row with J empty (keys all
 * masked) gets O = 0 and LSE = -inf, never NaN.
 *
 * Arguments
 *   Q        device, [B, H, Nq, d] contiguous, element type `dtype` (read)
 *   K, V     device, [B, H, Nkv, d] contiguous, element type `dtype` (read)
 *   O        device, [B, H, Nq, d] contiguous, element type `dtype` (written)
 *   LSE      device, [B, H, Nq] contiguous fp32 (written)
 *   B, H, Nq, Nkv   >= 1
 *   d        head dimension: 64 or 128
 *   scale    finite multiplier of the logits (1/sqrt(d) for the usual SDPA)
 *   causal   0: no causal mask; non-zero: key j visible to query i iff j <= i
 *            (top-left aligned, the same index for queries and keys)
 *   key_len  device int32 [B] or NULL; keys j >= key_len[b] are masked
 *            (values are clamped to [0, Nkv]; NULL means Nkv for every b).
 *            Combined with `causal` by logical AND.
 *   dtype    OSATTN_BF16, OSATTN_FP16 (tensor cores, fp32 accumulation,
 *            P rounded to the input type before P.V) or OSATTN_FP32 (SIMT)
 *   stream   cudaStream_t to enqueue on (NULL: the legacy default stream)
 *
 * Layout and alignment: Q, K, V and O must be 16-byte aligned; LSE and
 * key_len 4-byte aligned.  The d axis is fastest, then the sequence axis,
 * then H, then B.  O and LSE must not overlap the inputs.
 *
 * Ownership: all buffers are owned by the caller and stay owned by it.  The
 * call allocates no device memory and keeps no per-call state; it may read
 * device properties and set kernel attributes once per device.
 *
 * Asynchrony and errors: the call validates its arguments on the host, then
 * enqueues the kernel on `stream` and returns.  Results are valid once the
 * stream has reached that point.  The return value covers host validation
 * (OSATTN_ERR_INVALID_ARG / OSATTN_ERR_UNSUPPORTED, nothing enqueued) and
 * launch failures (OSATTN_ERR_CUDA, read with cudaGetLastError, no
 * synchronisation).  Device-side timeouts are reported by
 * osattn_get_device_status.  Nothing is printed and nothing aborts.
 */
int osattn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
               int B, int H, int Nq, int Nkv, int d, float scale, int causal,
               const int32_t* key_len, int dtype, void* stream);

/*
 * osattn_fwd_strided - osattn_fwd on tensors with arbitrary strides, e.g.
 * the [B, N, H, d] layout a fused QKV projection leaves behind, without a
 * transposing copy.  Same computation, masking, results and errors as
 * osattn_fwd.
 *
 *   q_strides, k_strides, v_strides, o_strides
 *            host int64[3] each, or NULL: element strides of the B, H and
 *            sequence axes of Q, K, V and O (the d axis always has stride 1).
 *            NULL means the contiguous [B, H, N, d] layout, so osattn_fwd is
 *            this call with four NULLs.  Each stride must be >= 1, a multiple
 *            of 16 bytes (8 elements for bf16/fp16, 4 for fp32) and below
 *            2^40 bytes; otherwise OSATTN_ERR_INVALID_ARG.  Strides are read
 *            during the call only.  Views may interleave (Q, K and V slices
 *            of one packed tensor); O must not alias any input, and distinct
 *            (b, h, i) of O must not share memory.
 *   LSE      always [B, H, Nq] contiguous fp32.
 */
int osattn_fwd_strided(const void* Q, const void* K, const void* V, void* O, float* LSE,
                       int B, int H, int Nq, int Nkv, int d, const int64_t* q_strides,
                       const int64_t* k_strides, const int64_t* v_strides,
                       const int64_t* o_strides, float scale, int causal,
                       const int32_t* key_len, int dtype, void* stream);

/*
 * osattn_fwd_offload - osattn_fwd for inputs and outputs that live in host
 * memory: copies Q, K, V in, runs the forward pass and copies O and LSE out,
 * pipelined over chunks of heads so that the copy of one chunk in, the
 * attention of the previous one and the copy out of the one before that
 * overlap (one host-to-device and one device-to-host stream of the
 * library's; the chunks' attention launches alternate between `stream` and
 * a compute stream of the library's, so that one chunk's launch starts on
 * the SMs the end of the previous one leaves idle).  Same result as
 * osattn_fwd on the copied data.
 *
 *   Q_host, K_host, V_host   host, contiguous [B, H, N, d] (read); pinned
 *                            (page-locked) memory for the copies to overlap
 *   O_host, LSE_host         host, contiguous [B, H, Nq, d] / [B, H, Nq] (written)
 *   Q, K, V, O, LSE          device buffers of the same shapes (overwritten;
 *                            used as staging, and hold the inputs and outputs
 *                            afterwards); alignment as for osattn_fwd
 *   B .. dtype               as for osattn_fwd (key_len is a device array)
 *   heads_per_chunk          heads per pipeline chunk, within one batch entry
 *                            (larger than H: one chunk per batch entry); 0
 *                            picks enough heads for one wave of CTAs per
 *                            chunk; negative -> OSATTN_ERR_INVALID_ARG
 *   stream                   the copies wait for work enqueued on `stream`
 *                            before the call, and `stream` completes only
 *                            after the last copy out: synchronize `stream`
 *                            (or wait on an event recorded on it) before
 *                            reading O_host and LSE_host
 *
 * Errors as for osattn_fwd (a null host pointer is OSATTN_ERR_INVALID_ARG).
 * Calls from several host threads are serialised while they enqueue.
 */
int osattn_fwd_offload(const void* Q_host, const void* K_host, const void* V_host, void* O_host,
                       float* LSE_host, void* Q, void* K, void* V, void* O, float* LSE, int B,
                       int H, int Nq, int Nkv, int d, float scale, int causal,
                       const int32_t* key_len, int dtype, int heads_per_chunk, void* stream);

/* Largest num_splits osattn_fwd_splitkv accepts. */
#define OSATTN_MAX_SPLITS 128

/*
 * osattn_splitkv_workspace_bytes - device workspace osattn_fwd_splitkv needs:
 * num_splits * B*H*Nq * (d + 1) fp32 values (a normalised partial O row and
 * its partial LSE per key range).  Returns 0 for sizes < 1.
 */
size_t osattn_splitkv_workspace_bytes(int B, int H, int Nq, int d, int num_splits);

/*
 * osattn_fwd_splitkv - the same result as osattn_fwd (same arguments,
 * layouts, masking and fully-masked-row rule), computed with the key axis
 * cut into num_splits ranges so that few (b, h) rows with long key sequences
 * still fill the GPU.
 *
 * Each CTA runs the online-softmax loop over one key range and writes a
 * partial O_s = O / l_s (fp32) and lse_s = m_s + ln l_s; a second kernel
 * folds the partials of every row with the guarded (m, l) combine of [Ch6]
 * §6.4.1 - the two-stage reduction [Ch6] §6.7.1 describes for a row split
 * across blocks - and writes O and LSE.  A key range with no visible
 * key contributes the (-inf, 0) identity.
 *
 *   dtype            OSATTN_BF16 or OSATTN_FP16 (OSATTN_FP32 -> OSATTN_ERR_UNSUPPORTED);
 *                    O is written in that type
 *   num_splits       1 .. OSATTN_MAX_SPLITS (else OSATTN_ERR_INVALID_ARG); ranges are
 *                    equal cuts of each 256-row query block's 128-key tiles, so
 *                    splits beyond the tile count receive empty ranges
 *   workspace        caller-owned device memory, 16-byte aligned, at least
 *                    osattn_splitkv_workspace_bytes(B, H, Nq, d, num_splits) bytes
 *                    (else OSATTN_ERR_INVALID_ARG); overwritten by the call and
 *                    free for other use once the stream passes it
 *
 * Both kernels are enqueued on `stream`; the call allocates nothing.
 * Errors as for osattn_fwd.
 */
int osattn_fwd_splitkv(const void* Q, const void* K, const void* V, void* O, float* LSE,
                       int B, int H, int Nq, int Nkv, int d, float scale, int causal,
                       const int32_t* key_len, int dtype, int num_splits, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Size of the scratch array built into the library for
 * osattn_fwd_splitkv_noalloc (32 MiB on every GPU that loads the library). */
#define OSATTN_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * osattn_fwd_splitkv_noalloc - osattn_fwd_splitkv without a caller-provided
 * workspace, for callers that cannot allocate device memory: an application
 * whose own memory manager owns the device budget and forbids other
 * allocations, or a latency-critical path that cannot pay for cudaMalloc's
 * implicit synchronisation.  (The pages have no counterpart; this is an
 * interface convenience, not part of the method.)
 *
 * Same arguments, results and errors as osattn_fwd_splitkv, minus the
 * workspace: the partial results go to a fixed array of
 * OSATTN_NOALLOC_SCRATCH_BYTES compiled into the library.  A problem with
 * osattn_splitkv_workspace_bytes(B, H, Nq, d, num_splits) greater than that
 * is rejected with OSATTN_ERR_SCRATCH_LIMIT before anything is enqueued;
 * use fewer splits, or osattn_fwd_splitkv with your own workspace.
 *
 * Arguments are checked first, with the statuses osattn_fwd_splitkv
 * returns; OSATTN_ERR_SCRATCH_LIMIT only follows for valid arguments.
 *
 * The call allocates nothing.  Its first call on a device looks up that
 * device's copy of the array (cudaGetSymbolAddress, with the device
 * current) and keeps the address; make that first call before any stream
 * capture.  The address belongs to the runtime's primary context: the entry
 * point assumes the caller uses that context and does not reset the device
 * (cudaDeviceReset) between calls.  Every call on a device shares the one
 * array and leaves its contents behind; a successful call writes every
 * partial it reads, so nothing in it has to start at zero.  After
 * osattn_get_device_status reports OSATTN_ERR_TIMEOUT, O and LSE of the
 * calls since the last status read may hold data left in the array by
 * earlier calls: discard them.  Calls whose kernels can overlap on the GPU
 * (for example on two streams without ordering between them) race on the
 * array and give undefined results: order them on one stream or with events.
 */
int osattn_fwd_splitkv_noalloc(const void* Q, const void* K, const void* V, void* O,
                               float* LSE, int B, int H, int Nq, int Nkv, int d, float scale,
                               int causal, const int32_t* key_len, int dtype, int num_splits,
                               void* stream);

/*
 * osattn_bwd_workspace_bytes - device workspace osattn_bwd needs: one fp32
 * per query row (B*H*Nq floats).  Returns 0 for sizes < 1.
 */
size_t osattn_bwd_workspace_bytes(int B, int H, int Nq);

/*
 * osattn_bwd - gradients of osattn_fwd for an upstream gradient dO.
 *
 * With P_ij = e^{s_ij - LSE_i} on the visible keys J_i (s, J and LSE exactly
 * as in osattn_fwd; the forward pass keeps LSE per row so that the backward
 * pass can rebuild P, [Ch6] §6.5, recomputing the scores, [XXQK] §5.2):
 *     D_i   = <dO_i, O_i>
 *     dS_ij = P_ij (<dO_i, V_j> - D_i)
 *     dQ_i  = scale * sum_j dS_ij K_j
 *     dK_j  = scale * sum_i dS_ij Q_i
 *     dV_j  = sum_i P_ij dO_i
 * (the chain rule on the forward definition).  Rows with J empty contribute
 * nothing; keys no row sees get dK = dV = 0.
 *
 *   Q, K, V   device, as for osattn_fwd (contiguous [B, H, N, d]) (read)
 *   O, LSE    device, the outputs of osattn_fwd for these Q, K, V, scale,
 *             causal and key_len (read)
 *   dO        device, [B, H, Nq, d] contiguous, element type `dtype` (read)
 *   dQ        device, [B, H, Nq, d] contiguous, element type `dtype` (written)
 *   dK, dV    device, [B, H, Nkv, d] contiguous, element type `dtype` (written)
 *   B .. key_len   as for osattn_fwd
 *   dtype     OSATTN_BF16, OSATTN_FP16 (tensor cores: P and dS rounded to the
 *             input type for the products, fp32 accumulation) or OSATTN_FP32
 *             (SIMT FMAs and expf throughout, for the fp32 forward)
 *   workspace caller-owned device memory, 16-byte aligned, at least
 *             osattn_bwd_workspace_bytes(B, H, Nq) bytes (else
 *             OSATTN_ERR_INVALID_ARG); overwritten, free once the stream
 *             passes the call
 *
 * dO, dQ, dK, dV must be 16-byte aligned and must not overlap each other or
 * the inputs.  Three kernels are enqueued on `stream` (D, then dK/dV, then
 * dQ); each output element is written by one CTA (one thread for fp32), so
 * the results do not depend on scheduling.  The call allocates nothing.  Errors as for
 * osattn_fwd.
 */
int osattn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
               const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int Nq, int Nkv,
               int d, float scale, int causal, const int32_t* key_len, int dtype,
               void* workspace, size_t workspace_bytes, void* stream);

/*
 * osattn_bwd_offload - osattn_bwd for tensors that live in host memory:
 * copies Q, K, V, O, dO and LSE in, computes the gradients and copies dQ,
 * dK and dV out, pipelined over chunks of heads as osattn_fwd_offload
 * (when Nq is not a multiple of 4 every chunk's kernels run on `stream`:
 * the chunks then share the start of the workspace).  Same results as
 * osattn_bwd on the copied data.
 *
 *   *_host     host, contiguous (Q, O, dO, dQ [B, H, Nq, d]; K, V, dK, dV
 *              [B, H, Nkv, d]; LSE [B, H, Nq] fp32); inputs read, dQ_host,
 *              dK_host, dV_host written; pinned memory for the copies to
 *              overlap the compute
 *   Q .. dV    device buffers of the same shapes (overwritten staging)
 *   B .. dtype, workspace, workspace_bytes   as for osattn_bwd
 *   heads_per_chunk   as for osattn_fwd_offload (0: two waves of dK/dV
 *              CTAs per chunk)
 *   stream     as for osattn_fwd_offload
 *
 * Errors as for osattn_bwd (a null host pointer is OSATTN_ERR_INVALID_ARG).
 */
int osattn_bwd_offload(const void* Q_host, const void* K_host, const void* V_host,
                       const void* O_host, const void* dO_host, const float* LSE_host,
                       void* dQ_host, void* dK_host, void* dV_host, void* Q, void* K, void* V,
                       void* O, void* dO, float* LSE, void* dQ, void* dK, void* dV, int B, int H,
                       int Nq, int Nkv, int d, float scale, int causal, const int32_t* key_len,
                       int dtype, void* workspace, size_t workspace_bytes, int heads_per_chunk,
                       void* stream);

/*
 * osattn_bwd_strided - osattn_bwd on tensors with arbitrary strides (e.g.
 * the [B, N, H, d] layout), without transposing copies.  Same computation,
 * results and errors as osattn_bwd.
 *
 *   q_strides .. dv_strides
 *            host int64[3] each, or NULL: element strides of the B, H and
 *            sequence axes of Q, K, V, O, dO, dQ, dK and dV (the d axis
 *            always has stride 1; NULL means the contiguous [B, H, N, d]
 *            layout, so osattn_bwd is this call with eight NULLs).  Each
 *            stride must be >= 1, a multiple of 16 bytes (8 elements) and
 *            below 2^40 bytes; otherwise OSATTN_ERR_INVALID_ARG.  Read during
 *            the call only.  Distinct rows of dQ, dK and dV must not share
 *            memory, and the outputs must not overlap the inputs.
 *   LSE      always [B, H, Nq] contiguous fp32.
 */
int osattn_bwd_strided(const void* Q, const void* K, const void* V, const void* O,
                       const void* dO, const float* LSE, void* dQ, void* dK, void* dV, int B,
                       int H, int Nq, int Nkv, int d, const int64_t* q_strides,
                       const int64_t* k_strides, const int64_t* v_strides,
                       const int64_t* o_strides, const int64_t* do_strides,
                       const int64_t* dq_strides, const int64_t* dk_strides,
                       const int64_t* dv_strides, float scale, int causal,
                       const int32_t* key_len, int dtype, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * osattn_softmax_rows - row softmax of a [rows, N] matrix with the online
 * (m, l) normaliser of [Ch6] §6.4: per row,
 *     y_i = e^{x_i - m} / l,  m = max_i x_i,  l = sum_i e^{x_i - m},
 *     LSE = m + ln l                                          ([Ch6] §6.5)
 * with per-thread states merged by the guarded combine of [Ch6] §6.4.1.
 * Rows of up to 32768 elements are held in registers: read once and written
 * once; longer rows are read twice.  -inf entries act as the additive mask
 * of [Ch6] §6.7.3; a row of only -inf gives y = 0 and LSE = -inf (no NaN).
 *
 *   in, out  device, [rows, N] contiguous, element type `dtype` (bf16, fp16
 *            or fp32);
 *            element-aligned; in == out (in place) is allowed
 *   lse      device fp32 [rows], or NULL to skip it
 *   rows, N  >= 1
 *   stream   cudaStream_t (NULL: legacy default stream)
 * Errors: OSATTN_ERR_INVALID_ARG (null/size/alignment), OSATTN_ERR_UNSUPPORTED
 * (dtype), OSATTN_ERR_CUDA (launch).  Asynchronous like osattn_fwd.
 */
int osattn_softmax_rows(const void* in, void* out, float* lse, int64_t rows, int N, int dtype,
                        void* stream);

/*
 * osattn_softmax_rows_offload - osattn_softmax_rows for a matrix in host
 * memory: copies it in, normalises and copies y (and LSE) out, pipelined
 * over chunks of rows as osattn_fwd_offload does over heads.  Same result as
 * osattn_softmax_rows on the copied data.
 *
 *   in_host    host, [rows, N] row-major, element type `dtype` (read); pinned
 *              memory for the copies to overlap
 *   out_host   host, [rows, N] (written)
 *   lse_host   host fp32 [rows] (written) or NULL; NULL exactly when `lse` is
 *   in, out, lse   device buffers of the same shapes (overwritten staging)
 *   rows_per_chunk   rows per pipeline chunk; 0 picks 16 chunks; negative ->
 *              OSATTN_ERR_INVALID_ARG
 *   stream     as for osattn_fwd_offload
 *
 * Errors as for osattn_softmax_rows (null host pointers, or lse_host and lse
 * not both given or both NULL: OSATTN_ERR_INVALID_ARG; rows above 2^31 - 1:
 * OSATTN_ERR_INVALID_ARG).
 */
int osattn_softmax_rows_offload(const void* in_host, void* out_host, float* lse_host, void* in,
                                void* out, float* lse, int64_t rows, int N, int dtype,
                                int64_t rows_per_chunk, void* stream);

/* Static, human-readable text for a status code (never NULL). */
const char* osattn_status_string(int status);

/*
 * osattn_get_device_status - synchronises `stream`, then returns and clears
 * the device status word of the current device: OSATTN_OK, or
 * OSATTN_ERR_TIMEOUT if a kernel's bounded wait on an mbarrier ran past its
 * limit since the last call (that kernel returned early; its outputs are
 * undefined).  Returns OSATTN_ERR_CUDA if the synchronisation itself fails.
 * Every device-side wait in libosattn is bounded; none traps.
 */
int osattn_get_device_status(void* stream);

/* OSATTN_VERSION of the built library. */
int osattn_version(void);

/*
 * Test hooks (no counterpart on the pages; they exist so the failure path can
 * be exercised without faulting a GPU).
 *
 * osattn_set_wait_limit_ns - sets the time limit (nanoseconds, >= 1000) that
 *   every device-side wait of later launches on any device uses; returns the
 *   previous limit.  Default 4e9 (4 s).  Values below 1000 are clamped.
 * osattn_test_wait_timeout - enqueues a one-warp kernel that waits on an
 *   mbarrier nobody arrives on, with the current limit; the wait gives up,
 *   records OSATTN_ERR_TIMEOUT in the status word and the kernel returns.
 *   Returns OSATTN_OK or OSATTN_ERR_CUDA (launch failure).
 */
uint64_t osattn_set_wait_limit_ns(uint64_t ns);
int osattn_test_wait_timeout(void* stream);

/* Site code of the first wait that gave up, as read by the most recent
 * osattn_get_device_status call that returned OSATTN_ERR_TIMEOUT (0 if none).
 * Codes identify the waiting role (producer, MMA issuer, softmax, epilogue). */
int osattn_last_timeout_site(void);

/*
 * osattn_step_trace_read - profiling hook (no counterpart in the method).
 * A library built with OSATTN_STEP_TRACE=1 (a separate profiling build,
 * never the product) records SM clock stamps at the phases of every K/V
 * step of the first 8 CTAs of each bf16/fp16 forward launch: long long
 * [8 CTAs][7 roles][128 steps][4 stamps]; role 0/1 = softmax of query tile
 * 0/1, its first warp (S seen, S in registers, alpha published, P
 * published); role 2 = MMA warp (K/V seen, P of tile 0 seen, P of tile 1
 * seen, step issued); role 3/4 = P published by each of the four softmax
 * warps of tile 0/1; role 5/6 = correction of tile 0/1, its first warp
 * (alpha seen, O rescaled, arrived, and 1 if the warp rescaled O - a flag,
 * not a clock).  Then long long [4096 CTAs][6] for the first 4096 CTAs of
 * the last launch: global-timer nanoseconds at start, end of setup, first S
 * seen, epilogue start (tile 0) and end, and the SM it ran on.
 * Copies them to `host` (bytes >= *needed) after the stream has
 * synchronised.  *needed (if not NULL) gets the size.  Returns OSATTN_OK,
 * OSATTN_ERR_INVALID_ARG (buffer too small) or, in a product build,
 * OSATTN_ERR_UNSUPPORTED.
 */
int osattn_step_trace_read(void* host, size_t bytes, size_t* needed);

#ifdef __cplusplus
}
#endif

#endif /* OSATTN_H */
