/*
 * fa.h -- C ABI of fused exact attention for GB300 (sm_103a): the forward (with masks and a
 * split-K/V form), its backward, and host-buffer forms of both.
 *
 * The operation ("FlashAttention 优化原理与实现要点解析" §1, §2, §4.3, §5, §7):
 *
 *     S = scale * Q K^T            (per batch b and head h; never written to memory)
 *     S[i, j] = -inf  for j > i    (only when causal: a query sees keys at positions <= its own)
 *     P = softmax(S) row-wise
 *     O = P V
 *     LSE[i] = m_i + ln(l_i),  m_i = max_j S[i, j],  l_i = sum_j exp(S[i, j] - m_i)
 *
 * computed tile by tile with online softmax: the running row maximum m and sum l are
 * rescaled by exp(m_old - m_new) as each K/V tile arrives, the unnormalised O is rescaled by
 * the same factor, and O is divided by l once at the end (same page §4.2, §4.3, §6). The
 * statistics m and l are the ones the forward keeps for the backward pass
 * ("FlashAttention V2 核心原理与架构设计" §2.3); they are returned combined as one fp32
 * log-sum-exp per row, in natural-log units of the scaled scores.
 *
 * Layout. q, k, v, o: [B, N, H, d], dense and contiguous: element (b, n, h, c) sits at
 * ((b*N + n)*H + h)*d + c. This is the [B, N, H, D] layout of the page's PyTorch wrapper
 * ("FlashAttention V2 核心原理与架构设计" §5.2). lse: [B, H, N] fp32, element (b, h, n) at
 * (b*H + h)*N + n.
 *
 * Ownership. Every pointer is owned by the caller and is a device pointer, except the host
 * buffers of fa_fwd_host and fa_bwd_host. The library allocates no device memory per call and
 * frees nothing. Calls are asynchronous: they only enqueue work on `stream` and return.
 *
 * Threading. The entry points are thread-safe; per-device state (the device-side error word,
 * the kernel attributes) is set up on first use of each device.
 */
#ifndef FA_GB300_FA_H
#define FA_GB300_FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. NULL means the legacy default stream. */
typedef struct CUstream_st* fa_stream_t;

/* Storage type of q, k, v and o (lse is always fp32). */
enum fa_dtype {
    FA_BF16 = 0,
    FA_FP16 = 1
};

/* Return codes. 0 is success; every error is negative. */
enum fa_status {
    FA_OK = 0,
    FA_ERR_NULL = -1,     /* a required pointer is NULL */
    FA_ERR_SHAPE = -2,    /* B, H or N < 1; d not 64 or 128; or B*N*H*d does not fit int64 */
    FA_ERR_DTYPE = -3,    /* dtype is not an fa_dtype */
    FA_ERR_ALIGN = -4,    /* q, k, v or o not 16-byte aligned; lse or seqlens_k not 4-byte */
    FA_ERR_ALIAS = -5,    /* o or lse overlaps q, k, v or seqlens_k, or o overlaps lse */
    FA_ERR_ARCH = -6,     /* the current device is not compute capability 10.3 (sm_103) */
    FA_ERR_LAUNCH = -7,   /* the kernel launch failed (the CUDA error is not cleared) */
    FA_ERR_TIMEOUT = -8,  /* a kernel wait ran past its limit; outputs are undefined */
    FA_ERR_SCALE = -9,    /* scale is not finite */
    FA_ERR_CUDA = -10,    /* a CUDA runtime or driver query failed */
    FA_ERR_WORKSPACE = -11, /* workspace smaller than fa_fwd_splitkv_workspace_size() */
    FA_ERR_POINTER = -12    /* a device-side argument is not device memory of the current device */
};

/*
 * fa_fwd -- O = softmax(scale * Q K^T [+ causal mask]) V and LSE, for all B*H heads.
 *
 *   q, k, v  [B, N, H, d] dtype, device, 16-byte aligned, read only
 *   o        [B, N, H, d] dtype, device, 16-byte aligned, written (every element)
 *   lse      [B, H, N] fp32, device, 4-byte aligned, written (every element)
 *   B, H, N  batch, heads, sequence length (>= 1 each); queries and keys share N
 *   d        head dimension: 64 or 128
 *   causal   0: every query sees all N keys; nonzero: query i sees keys 0..i
 *   scale    multiplier of Q K^T, used as given (typically 1/sqrt(d)); must be finite
 *   dtype    FA_BF16 or FA_FP16; the matrix products take this type, accumulate in fp32,
 *            and the probabilities P are rounded to this type before P V
 *   stream   CUDA stream the work is enqueued on
 *
 * Returns FA_OK once the work is enqueued. On a host-detected error (every code except
 * FA_ERR_TIMEOUT) nothing is enqueued and the outputs are untouched. Every device-side pointer
 * is looked up (cudaPointerGetAttributes) before anything is enqueued: host memory, memory of
 * another device or an unknown address gives FA_ERR_POINTER instead of a faulting kernel.
 * Kernel waits are bounded: if one runs out, the kernel records FA_ERR_TIMEOUT in a per-device
 * error word (read it with fa_get_device_error) and exits without hanging the device.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
           int N, int d, int causal, float scale, int dtype, fa_stream_t stream);

/*
 * fa_fwd_masked -- fa_fwd with the padding and sliding-window masks named next to the causal
 * mask in "FlashAttention 优化原理与实现要点解析" §8. Key j is visible to query i of batch b
 * only when all of these hold:
 *   j < len_b                  padding: len_b = seqlens_k[b] clamped to [0, N], or N when
 *                              seqlens_k is NULL (keys at or past len_b do not exist)
 *   j <= i                     when causal is nonzero
 *   j >= i - window_left       when window_left >= 0 (negative: no bound)
 *   j <= i + window_right      when window_right >= 0 (negative: no bound)
 * A query with no visible key gets O = 0 and LSE = -inf. K/V tiles with no visible key for any
 * query of a Q tile are never loaded or multiplied.
 *
 *   seqlens_k  device int32 [B], 4-byte aligned, read only, or NULL; it must not overlap o or
 *              lse (FA_ERR_ALIAS). Its values are read by the kernel, not checked on the host.
 *   everything else as in fa_fwd; fa_fwd(...) equals fa_fwd_masked(..., -1, -1, NULL, ...).
 */
int fa_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                  int H, int N, int d, int causal, int window_left, int window_right,
                  const int* seqlens_k, float scale, int dtype, fa_stream_t stream);

/*
 * fa_fwd_splitkv -- the forward with fewer queries than keys and with each (b, h, Q block)'s
 * K/V range cut into num_splits parts computed by separate CTAs, then merged. This is the
 * combination with FlashDecoding that "FlashAttention V2 核心原理与架构设计" §5.1 suggests for
 * very long sequences: when B * H * ceil(Nq / 256) is small against the number of SMs (few
 * heads, few queries, e.g. decoding), the parts fill the GPU. The merge applies the online-
 * softmax rule of "FlashAttention 优化原理与实现要点解析" §4.2 to whole parts: with part s
 * giving O_s (normalised by its own sum) and LSE_s, LSE = ln sum_s e^{LSE_s} and
 * O = sum_s e^{LSE_s - LSE} O_s.
 *
 *   q, o       [B, Nq, H, d];  k, v  [B, Nk, H, d] with Nk >= Nq;  lse  [B, H, Nq] fp32
 *              The queries are the last Nq positions of the sequence: query i sits at
 *              position i + Nk - Nq, and causal / window bounds are relative to it (so Nq = 1
 *              with causal sees every key: one decoding step).
 *   num_splits 1..128 parts; 1 needs no workspace (workspace may then be NULL).
 *   workspace  device memory of at least fa_fwd_splitkv_workspace_size(B, H, Nq, d,
 *              num_splits) bytes, 16-byte aligned, owned by the caller; it must not overlap any
 *              input or output. It holds the parts (fp32) until the merge kernel, enqueued on
 *              the same stream, has read them; calls that share a workspace must not overlap.
 *   everything else as in fa_fwd_masked.
 */
int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int Nq, int Nk, int d, int causal, int window_left, int window_right,
                   const int* seqlens_k, float scale, int dtype, int num_splits,
                   void* workspace, size_t workspace_bytes, fa_stream_t stream);

/* Bytes of workspace fa_fwd_splitkv needs: B*H*Nq*num_splits*(d + 1)*4; 0 for one part. */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int Nq, int d, int num_splits);

/* A part count for fa_fwd_splitkv on a GPU with num_sms SMs: the count (1..128, each part
 * keeping at least 2 K/V tiles of 128 keys) that minimises waves of CTAs x (K/V tiles per part
 * + 4), a model of one CTA per SM streaming its tiles after a fixed start-up cost. */
int fa_fwd_splitkv_num_splits(int B, int H, int Nq, int Nk, int num_sms);

/*
 * fa_fwd_splitkv_noalloc -- fa_fwd_splitkv for callers that cannot allocate device memory at
 * call time: a plugin running inside a host that owns the whole device-memory budget, or a
 * latency-critical loop where an allocation (and the synchronisation it may imply) is not
 * acceptable. The pages have no counterpart of this entry point; it is a deployment aid.
 *
 * Instead of a caller-provided workspace it uses one 8 MiB (8 * 2^20 bytes) device buffer
 * built into the library, which every GPU that loads the library keeps until the process
 * exits. It allocates nothing: no cudaMalloc, no cudaFree, no allocating library call. The
 * caller still passes q, k, v, o, lse (and seqlens_k) exactly as for fa_fwd_splitkv.
 *
 *   - Calls whose parts need more than 8 MiB (fa_fwd_splitkv_workspace_size(B, H, Nq, d,
 *     num_splits) > 8 MiB) return FA_ERR_WORKSPACE and enqueue nothing; use fewer parts, or
 *     fa_fwd_splitkv with a workspace of your own.
 *   - The first call on each device looks up the buffer's device address (with that device
 *     current) and keeps it for the device's context; after a device reset the next call looks
 *     it up again. Make the first call on a device, and the first after a reset, before any
 *     stream capture.
 *   - All calls on a device share the buffer, which keeps the last call's contents. Nothing in
 *     it needs clearing: each call writes every part it reads. Calls that overlap on the GPU
 *     (on different streams without ordering between them) race on the buffer.
 *   - Every argument means what it means for fa_fwd_splitkv, and is checked in the same way
 *     first, with the same return codes; only then are parts that do not fit the buffer
 *     refused (FA_ERR_WORKSPACE). A failed address lookup returns FA_ERR_CUDA and leaves no
 *     CUDA error pending.
 */
int fa_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                           int B, int H, int Nq, int Nk, int d, int causal, int window_left,
                           int window_right, const int* seqlens_k, float scale, int dtype,
                           int num_splits, fa_stream_t stream);

/*
 * fa_fwd_host -- fa_fwd on host buffers: the inputs are copied to device buffers, the forward
 * runs there, and O and LSE are copied back, in groups of heads so that the copies of one
 * group overlap the computation of another (each group is packed into a compact problem in the
 * device buffers and unpacked on the way back). (The pages have no counterpart; this is the
 * end-to-end form of fa_fwd for data that lives in host memory.)
 *
 *   q_h, k_h, v_h  [B, N, H, d] dtype, host memory: inputs
 *   o_h            [B, N, H, d] dtype, host memory: output
 *   lse_h          [B, H, N] fp32, host memory: output
 *   q_d, k_d, v_d, o_d, lse_d  device buffers of the same sizes, owned by the caller, the
 *                  arguments of the fa_fwd calls made here (same alignment and aliasing rules);
 *                  their previous contents are overwritten
 *   B, H, N, d, causal, scale, dtype: as in fa_fwd
 * Page-locked (pinned) host memory lets the copies run asynchronously; with pageable memory
 * the call is still correct but the copies do not overlap. Work is enqueued on `stream` and on
 * two copy streams and three kernel streams the library keeps per device (the groups' kernels
 * take the kernel streams in turn, so that they overlap one another); `stream` reaches
 * completion (O and LSE in host memory) after everything enqueued here, so synchronise
 * `stream` before reading o_h, lse_h, and keep every buffer alive until then. Returns as fa_fwd; on a host-detected error nothing is
 * enqueued. Calls from several threads are serialised while they enqueue.
 */
int fa_fwd_host(const void* q_h, const void* k_h, const void* v_h, void* o_h, float* lse_h,
                void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d, int B, int H, int N,
                int d, int causal, float scale, int dtype, fa_stream_t stream);

/*
 * fa_fwd_host_masked -- fa_fwd_host for the attention of fa_fwd_masked: the same window
 * (window_left, window_right) and key lengths (seqlens_k: DEVICE int32 [B], 4-byte aligned, or
 * NULL; the head groups span every batch, so it applies to each of them unchanged). Every other
 * argument, the streams and the return codes as in fa_fwd_host; fa_fwd_host(...) equals
 * fa_fwd_host_masked(..., -1, -1, NULL, ...).
 */
int fa_fwd_host_masked(const void* q_h, const void* k_h, const void* v_h, void* o_h,
                       float* lse_h, void* q_d, void* k_d, void* v_d, void* o_d, float* lse_d,
                       int B, int H, int N, int d, int causal, int window_left,
                       int window_right, const int* seqlens_k, float scale, int dtype,
                       fa_stream_t stream);

/*
 * fa_bwd -- gradients of the forward: dQ, dK, dV of L = sum(dO * O) for O = fa_fwd(q, k, v).
 * The forward keeps, per row, the softmax statistics the backward needs ("FlashAttention V2
 * 核心原理与架构设计" §2.3 keeps m and l; here their combination LSE = m + ln l), so the
 * backward rebuilds P_ij = exp(scale <q_i, k_j> - LSE_i) tile by tile without storing it:
 *   dV = P^T dO,  dP = dO V^T,  dS = P (dP - D) with D_i = <dO_i, O_i>,
 *   dQ = scale dS K,  dK = scale dS^T Q.
 *
 *   q, k, v, o   [B, N, H, d] dtype: the forward's inputs and output
 *   dout         [B, N, H, d] dtype: the gradient of the loss with respect to o
 *   lse          [B, H, N] fp32: the forward's LSE for the same q, k, v, causal and scale
 *   dq, dk, dv   [B, N, H, d] dtype, written (every element)
 *   causal, scale, dtype, d: as in fa_fwd (window and key-length masks: fa_bwd_masked)
 *   workspace    device memory of at least fa_bwd_workspace_size(B, H, N, d) bytes, 16-byte
 *                aligned, owned by the caller, not overlapping any other argument: fp32 dQ
 *                partial sums and D. Calls sharing a workspace must not overlap.
 * Returns as fa_fwd; on a host-detected error nothing is enqueued. Enqueues three kernels on
 * `stream`: D and a cleared dQ accumulator, the main kernel (one CTA per (b, h, 128-key
 * block)), and the rounding of dQ.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
           int causal, float scale, int dtype, void* workspace, size_t workspace_bytes,
           fa_stream_t stream);

/*
 * fa_bwd_masked -- fa_bwd for the attention fa_fwd_masked computes with Nq = Nk = N: the same
 * window (window_left, window_right; negative = no bound) and per-batch key lengths (seqlens_k:
 * device int32 [B], 4-byte aligned, or NULL), on top of `causal`. The gradients are those of
 * that masked attention: a key no query sees gets dK = dV = 0, a query that sees no key gets
 * dQ = 0 (its forward LSE is -inf). `lse` must come from fa_fwd_masked with the same masks.
 * Every other argument, the workspace and the return codes as in fa_bwd (seqlens_k must not
 * overlap an output).
 */
int fa_bwd_masked(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, int B, int H, int N, int d,
                  int causal, int window_left, int window_right, const int* seqlens_k,
                  float scale, int dtype, void* workspace, size_t workspace_bytes,
                  fa_stream_t stream);

/* Bytes of workspace fa_bwd needs: B*H*N*(d + 1)*4. */
size_t fa_bwd_workspace_size(int B, int H, int N, int d);

/*
 * fa_bwd_host -- fa_bwd on host buffers, in the manner of fa_fwd_host: q, k, v, o, dout and
 * lse are copied to device buffers group of heads by group of heads, fa_bwd runs on each group
 * packed into a compact problem, and dQ, dK, dV are copied back, so that the copies of one
 * group overlap the computation of another. (No counterpart in the pages; the end-to-end form
 * of fa_bwd for data that lives in host memory.)
 *
 *   q_h, k_h, v_h, o_h, do_h  [B, N, H, d] dtype, host memory: inputs (do_h is dO)
 *   lse_h          [B, H, N] fp32, host memory: the forward's LSE
 *   dq_h, dk_h, dv_h  [B, N, H, d] dtype, host memory: outputs
 *   q_d ... dv_d   device buffers of the same sizes, owned by the caller, pairwise disjoint,
 *                  16-byte aligned (lse_d 4-byte); their previous contents are overwritten
 *   workspace      as in fa_bwd for the whole problem. With at least
 *                  fa_bwd_workspace_size(B, H, N, d) + 128 bytes every group gets a part of its
 *                  own (at a 16-byte aligned offset) and the groups' kernels overlap on the
 *                  kernel streams; with less, the groups run one after another and reuse the
 *                  start of it in turn
 *   B, H, N, d, causal, scale, dtype: as in fa_bwd
 * Streams, pinned memory, synchronisation and errors as in fa_fwd_host: synchronise `stream`
 * before reading dq_h, dk_h, dv_h.
 */
int fa_bwd_host(const void* q_h, const void* k_h, const void* v_h, const void* o_h,
                const void* do_h, const float* lse_h, void* dq_h, void* dk_h, void* dv_h,
                void* q_d, void* k_d, void* v_d, void* o_d, void* do_d, float* lse_d,
                void* dq_d, void* dk_d, void* dv_d, void* workspace, size_t workspace_bytes,
                int B, int H, int N, int d, int causal, float scale, int dtype,
                fa_stream_t stream);

/*
 * fa_bwd_host_masked -- fa_bwd_host for the attention of fa_bwd_masked (window and key lengths,
 * seqlens_k a DEVICE int32 [B] array or NULL, as in fa_fwd_host_masked). Every other argument
 * as in fa_bwd_host; fa_bwd_host(...) equals fa_bwd_host_masked(..., -1, -1, NULL, ...).
 */
int fa_bwd_host_masked(const void* q_h, const void* k_h, const void* v_h, const void* o_h,
                       const void* do_h, const float* lse_h, void* dq_h, void* dk_h, void* dv_h,
                       void* q_d, void* k_d, void* v_d, void* o_d, void* do_d, float* lse_d,
                       void* dq_d, void* dk_d, void* dv_d, void* workspace,
                       size_t workspace_bytes, int B, int H, int N, int d, int causal,
                       int window_left, int window_right, const int* seqlens_k, float scale,
                       int dtype, fa_stream_t stream);

/* Static English text for a status code (never NULL). */
const char* fa_error_string(int code);

/*
 * fa_get_device_error -- synchronise `stream`, then return and clear the current device's
 * error word: FA_OK when no kernel wait has run out since the last call, FA_ERR_TIMEOUT
 * otherwise, FA_ERR_CUDA when the synchronisation or the read failed.
 */
int fa_get_device_error(fa_stream_t stream);

/*
 * fa_selftest_wait_timeout -- diagnostic for the failure path every kernel wait shares: enqueues
 * on `stream` one warp that waits, with the kernels' own bounded wait, on a barrier nothing ever
 * completes, for `limit_us` microseconds (1 .. 1e6); the wait runs out, the kernel records
 * FA_ERR_TIMEOUT in the device error word and exits. fa_get_device_error(stream) then returns
 * FA_ERR_TIMEOUT (and clears it), and the device stays usable. (Not on the pages: a check of
 * this library's error reporting.) Returns FA_OK once enqueued, FA_ERR_SHAPE for a limit out of
 * range, FA_ERR_ARCH / FA_ERR_CUDA / FA_ERR_LAUNCH as fa_fwd.
 */
int fa_selftest_wait_timeout(int limit_us, fa_stream_t stream);

/* ABI version of this header: 1. */
int fa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FA_H */
