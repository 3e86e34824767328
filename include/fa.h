/*
 * fa.h — C ABI of the fused exact-attention library (libfa.so), sm_103a.
 *
 * Computes exact scaled-dot-product attention O = softmax(mask(Q K^T * scale)) V
 * as a fused FlashAttention-2-style forward that never writes the N x N score
 * matrix, plus the recompute backward.
 *
 * Layouts (all tensors dense, row-major, no padding between rows):
 *   q, k, v, o, dO, dq, dk, dv : [B, N, H, d]  (the pages' [B, T, C], C = H*d)
 *   lse                        : [B, H, N] float32, natural log
 * Square self-attention only: queries and keys share N.  The causal mask is
 * top-left aligned: query i sees keys j <= i.
 *
 * Ownership: every pointer is a DEVICE pointer owned and allocated by the
 * caller; the library never allocates device memory in these calls and keeps
 * no pointer after a call returns.  Every call is asynchronous on `stream`
 * (a cudaStream_t passed as void*, NULL = legacy default stream) and never
 * synchronises.  Outputs must not alias inputs.
 *
 * Errors: arguments are validated on the host before anything is launched;
 * an invalid call returns an error code and launches nothing.  A launch
 * failure returns FA_ERR_CUDA.  Kernels never trap: every device-side wait is
 * bounded, and a wait that runs out records FA_ERR_TIMEOUT in a device status
 * word that fa_sync_status() reads.
 */
#ifndef FA_H
#define FA_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned, non-finite scale */
  FA_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. d > 128, dtype) */
  FA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  FA_ERR_TIMEOUT = 4       /* a bounded device wait ran out (see fa_sync_status) */
} fa_status;

typedef enum {
  FA_DTYPE_F32 = 0,   /* float32 storage, float32 arithmetic (SIMT path) */
  FA_DTYPE_BF16 = 1,  /* bf16 storage, fp32 accumulation (tcgen05 path) */
  FA_DTYPE_F16 = 2    /* fp16 storage, fp32 accumulation (tcgen05 path); |values| < 65504 */
} fa_dtype;

/*
 * fa_fwd — fused attention forward.
 *
 * Source: "Flash Attention 2 — forward pass notes", sections "The algorithm"
 * (S = Q K^T scale, causal mask S[i,j] = -inf for j > i, P = softmax(S),
 * O = P V) and "Loop (per (b, h, Q-tile))" (online m, l, O with rescale
 * alpha = exp(m_old - m_new), causal block skip, out-of-range keys scored
 * -inf), and "What's still needed for full FA2" item 1 (save
 * L = m_final + log(l_final) per row).
 *
 *   q, k, v  in : [B, N, H, d], element type `dtype`
 *   o       out : [B, N, H, d], element type `dtype`
 *   lse     out : [B, H, N] float32, natural log of sum_j exp(scale q.k_j)
 *   B, H, N     : >= 1;  B*H <= 2^31-1 rows of work
 *   d           : head dimension, a multiple of 8 in [8, 128]
 *   scale       : finite multiplier of the scores (1/sqrt(d) usually)
 *   causal      : 0 = no mask, nonzero = query i sees keys j <= i
 *   stream      : cudaStream_t (void*)
 * Alignment: q, k, v, o 16-byte aligned; lse 4-byte aligned.
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int H, int N, int d, float scale, int causal,
                 fa_dtype dtype, void* stream);

/*
 * fa_bwd_workspace_size — bytes of device workspace fa_bwd needs:
 * the D = rowsum(dO * O) buffer, [B, H, N] float32, rounded up to 256 bytes.
 * Returns 0 for non-positive sizes.
 */
size_t fa_bwd_workspace_size(int B, int H, int N);

/*
 * fa_bwd — attention backward with recompute, no float atomics.
 *
 * Source: "Flash Attention 2 — backward pass notes", section "The math (FA2
 * backward with recompute)": D = <dO, O> per query row, P = exp(S - L)
 * recomputed from q, k and the saved L, dP = dO V^T, dS = P (dP - D),
 * dQ = scale dS K, dK = scale dS^T Q, dV = P^T dO; and section "Why the WGSL
 * kernel isn't shipped this turn", options 1 and 3: a D pre-pass into a
 * [B, H, N] buffer, then one kernel that owns a K tile (dK, dV) and one that
 * owns a Q tile (dQ).
 *
 *   q, k, v, o, dO  in : [B, N, H, d], element type `dtype`
 *   lse             in : [B, H, N] float32 from fa_fwd on the same inputs
 *   dq, dk, dv     out : [B, N, H, d], element type `grad_dtype`
 *   grad_dtype         : `dtype`, or FA_DTYPE_F32 for float32 gradients
 *   workspace          : device scratch of >= fa_bwd_workspace_size(B,H,N)
 *                        bytes, 256-byte aligned; contents on entry ignored;
 *                        on return it holds D as float32 [B, H, N]
 *   other arguments as in fa_fwd.
 * Rows whose lse is -inf (no visible key) contribute nothing.
 *
 * 16-bit paths (bf16, fp16): D is first taken from the 16-bit O as above,
 * then refined in the dQ kernel to the fp32 sum_j P_ij dP_ij (the same
 * quantity without O's storage rounding), and dQ is corrected accordingly;
 * dS is staged for the tensor cores in fp16, so |Q|, |K| and |dS| must stay
 * below 65504 (fp16 storage: every input and output too).
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dO,
                 void* dq, void* dk, void* dv,
                 int B, int H, int N, int d, float scale, int causal,
                 fa_dtype dtype, fa_dtype grad_dtype,
                 void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_bwd_phase — one step of fa_bwd, for callers that schedule or time the
 * backward's kernels separately.  fa_bwd is exactly phases 0, 1, 2 in order
 * on one stream, and the phases must be run in that order:
 *   0: the D pre-pass, D = rowsum(dO * O) into the workspace
 *      ("Flash Attention 2 — backward pass notes", option 1 of "Why the WGSL
 *      kernel isn't shipped this turn");
 *   1: the kernel that owns Q tiles and writes dQ (16-bit paths: also
 *      refines D in the workspace);
 *   2: the kernel that owns K tiles and writes dK and dV (option 3).
 * Arguments, validation and errors as fa_bwd; phase outside [0, 2] returns
 * FA_ERR_INVALID_ARG.
 */
fa_status fa_bwd_phase(int phase, const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dO,
                       void* dq, void* dk, void* dv,
                       int B, int H, int N, int d, float scale, int causal,
                       fa_dtype dtype, fa_dtype grad_dtype,
                       void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_sync_status — synchronises `stream`, then returns and clears the device
 * status word of the current device: FA_OK, or FA_ERR_TIMEOUT if a kernel's
 * bounded wait ran out since the last call (its outputs are then undefined),
 * or FA_ERR_CUDA if the synchronisation itself failed.
 */
fa_status fa_sync_status(void* stream);

/*
 * fa_bwd_noalloc — fa_bwd without a workspace argument, for callers that
 * must not allocate device memory at call time (for example code whose
 * device memory belongs to a host framework's pool, or a latency-critical
 * path that cannot afford cudaMalloc).  The pages have no counterpart: this
 * is a convenience of this library.
 *
 * The D scratch is a fixed array of FA_BWD_NOALLOC_MAX_ROWS floats (16 MiB)
 * inside the library's device image, present on every GPU that loads the
 * library until the process exits.  Calls with B*H*N above that return
 * FA_ERR_UNSUPPORTED and launch nothing.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress, with that device
 * current), so make that first call before any stream capture.  All calls on
 * a device share the array: calls whose GPU work overlaps (other streams,
 * unordered host threads) race on it and produce wrong gradients.  No call
 * allocates device memory.  Otherwise arguments, results and errors are
 * those of fa_bwd.
 */
#define FA_BWD_NOALLOC_MAX_ROWS (1u << 22)
fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                         const float* lse, const void* dO,
                         void* dq, void* dk, void* dv,
                         int B, int H, int N, int d, float scale, int causal,
                         fa_dtype dtype, fa_dtype grad_dtype, void* stream);

/* fa_status_string — static, human-readable name of a status code. */
const char* fa_status_string(fa_status s);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
