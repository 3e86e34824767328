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
 *      kernel isn't shipped this turn"); with 16-bit inputs and d <= 64 it
 *      launches nothing, because phase 1 forms D from the O and dO rows it
 *      loads;
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
 * fa_bwd_prepass — 1 if fa_bwd's phase 0 (the D pre-pass) launches a kernel
 * for this head dim and input type, 0 if it is empty (16-bit inputs with
 * d <= 64: phase 1 forms D itself); for callers that time the phases.  No
 * argument checks: it only reports the rule.
 */
int fa_bwd_prepass(int d, fa_dtype dtype);

/*
 * fa_sync_status — synchronises `stream`, then returns and clears the device
 * status word of the current device: FA_OK, or FA_ERR_TIMEOUT if a kernel's
 * bounded wait ran out since the last call (its outputs are then undefined),
 * or FA_ERR_CUDA if the synchronisation itself failed.
 *
 * The status word is one int per device, shared by every stream and every
 * caller on that device (it is not in the caller's workspace).  A timeout
 * recorded by a kernel on stream A is therefore returned, and cleared, by
 * whichever fa_sync_status call on that device reads it first, whatever
 * stream that call names; and since only `stream` is synchronised, a kernel
 * still running on another stream may record a timeout after the read.
 * Callers that run library kernels on several streams and need to know
 * which call timed out should synchronise all of those streams (e.g.
 * cudaDeviceSynchronize) before calling fa_sync_status, or serialise the
 * calls they want to tell apart.
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

/*
 * Split-KV forward: the keys of each head are cut into slices, every
 * (Q tile, key slice) pair is an independent piece of work, and the per-slice
 * results are merged afterwards.  This spreads a few long heads over every SM
 * (few heads x long N, where whole Q tiles are too few to fill the GPU), and
 * the merge is the exchange step a context-parallel forward would need.
 *
 * Source: "Flash Attention 2 — forward pass notes", section "Loop (per
 * (b, h, Q-tile))": the softmax of a concatenation of key blocks is the
 * merge of the blocks' (m, l) states; and the "Lesson K23, fused attention"
 * facts page, `sources.onlineSoftmax.claims[2]`: the (m, l) pairs combine
 * with an associative, commutative operator, so the reduction may run in
 * parallel and in any order.
 *
 * Slices: keys [s*keys_per_split, (s+1)*keys_per_split) for
 * s < num_splits = ceil(N / keys_per_split).  Row i READS slice s when it
 * sees at least one key there: with causal, iff s*keys_per_split <= i;
 * without, always.
 */

/*
 * fa_fwd_partial — attention of every query row over each key slice alone.
 * For every (row i, slice s) that row i reads:
 *   lse_part[s, b, h, i] = log sum_{j in s, visible} exp(scale q_i.k_j)
 *   o_part[s, b, i, h, :] = sum_{j in s, visible} exp(scale q_i.k_j - lse_part) v_j
 * (O normalised over the slice; float32, no rounding to 16 bits).  Entries of
 * slices a row does not read are not written.
 *
 *   q, k, v        in : [B, N, H, d], element type `dtype` (BF16 or F16;
 *                       F32 returns FA_ERR_UNSUPPORTED)
 *   o_part        out : [num_splits, B, N, H, d] float32, 16-byte aligned
 *   lse_part      out : [num_splits, B, H, N] float32
 *   keys_per_split    : a positive multiple of 256
 *   other arguments as in fa_fwd.  Outputs must not overlap inputs or each other.
 */
fa_status fa_fwd_partial(const void* q, const void* k, const void* v,
                         float* o_part, float* lse_part,
                         int B, int H, int N, int d, float scale, int causal,
                         fa_dtype dtype, int keys_per_split, void* stream);

/*
 * fa_merge — combine per-slice results into the attention output.  For each
 * row i, over the slices s it reads (see above) whose lse_part is not -inf:
 *   L_i = log sum_s exp(lse_part[s, i]),
 *   O_i = sum_s exp(lse_part[s, i] - L_i) o_part[s, i]
 * (the (m, l) merge, with every slice's state written as m = lse, l = 1).
 * A slice whose lse_part is -inf contributes nothing and its o_part is not
 * read; a row with no contribution gets O = 0 and L = -inf.  O is rounded
 * once to `dtype`.
 *
 *   o_part, lse_part  in : as written by fa_fwd_partial (any producer that
 *                          follows the same layout and slice rule)
 *   num_splits           : >= 1 slices present in o_part / lse_part; row i
 *                          reads at most ceil(N / keys_per_split) of them
 *   keys_per_split       : >= 1 (the slice width the partials were made with)
 *   o                out : [B, N, H, d], element type `dtype` (F32, BF16, F16),
 *                          16-byte aligned
 *   lse              out : [B, H, N] float32
 */
fa_status fa_merge(const float* o_part, const float* lse_part, int num_splits,
                   int keys_per_split, int causal, void* o, float* lse,
                   int B, int H, int N, int d, fa_dtype dtype, void* stream);

/*
 * fa_fwd_splitkv_keys_per_split — the slice width fa_fwd_splitkv uses for
 * `num_splits` requested slices: 256 * ceil(N / (256 num_splits)).  The
 * slices actually used, ceil(N / that), may be fewer than requested.
 * Returns 0 for non-positive arguments.
 */
int fa_fwd_splitkv_keys_per_split(int N, int num_splits);

/*
 * fa_fwd_splitkv_workspace_size — bytes of device workspace fa_fwd_splitkv
 * needs for `num_splits` requested slices: o_part and lse_part for the
 * slices used, each rounded up to 256 bytes.  Returns 0 for invalid sizes.
 */
size_t fa_fwd_splitkv_workspace_size(int B, int H, int N, int d, int num_splits);

/*
 * fa_fwd_splitkv — fa_fwd computed as fa_fwd_partial then fa_merge on one
 * stream, with o_part and lse_part in `workspace` (o_part first, then
 * lse_part at the next 256-byte boundary).  Same results as fa_fwd up to
 * rounding order.  num_splits >= 1 (see fa_fwd_splitkv_keys_per_split);
 * workspace 256-byte aligned, >= fa_fwd_splitkv_workspace_size(...) bytes,
 * not overlapping any argument.  Other arguments as in fa_fwd; dtype BF16 or
 * F16.
 */
fa_status fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal,
                         fa_dtype dtype, int num_splits,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_bwd_host — fa_fwd then fa_bwd on HOST buffers: the inputs are copied
 * in, the outputs copied out, all inside the call's stream order.  The pages
 * have no counterpart; this is the library's end-to-end entry point.
 *
 * The batch is processed in chunks of `batch_chunk` sequences through two
 * device slots in `workspace`, so that the copy-in of chunk c+1 and the
 * copy-out of chunk c-1 overlap the kernels of chunk c (two internal copy
 * streams, created once per device, plus the caller's stream for the
 * kernels).  Host buffers should be page-locked (cudaHostAlloc /
 * cudaHostRegister); pageable buffers give correct results without overlap.
 *
 *   q, k, v, dO      in : HOST, [B, N, H, d], element type `dtype`
 *   o               out : HOST, [B, N, H, d], `dtype`
 *   lse             out : HOST, [B, H, N] float32
 *   dq, dk, dv      out : HOST, [B, N, H, d], `grad_dtype`
 *   batch_chunk         : >= 1 sequences per chunk (min(batch_chunk, B) used)
 *   workspace           : DEVICE, 256-byte aligned, >=
 *                         fa_fwd_bwd_host_workspace_size(min(batch_chunk, B),
 *                         H, N, d, dtype, grad_dtype) bytes
 *   other arguments as in fa_fwd and fa_bwd.
 * The call returns once everything is queued; the host outputs are complete
 * after `stream` is synchronised (then also check fa_sync_status).  Host
 * outputs must not overlap host inputs.  Concurrent calls on one device are
 * queued one after another.
 */
size_t fa_fwd_bwd_host_workspace_size(int batch_chunk, int H, int N, int d, fa_dtype dtype,
                                      fa_dtype grad_dtype);
fa_status fa_fwd_bwd_host(const void* q, const void* k, const void* v, const void* dO,
                          void* o, float* lse, void* dq, void* dk, void* dv,
                          int B, int H, int N, int d, float scale, int causal,
                          fa_dtype dtype, fa_dtype grad_dtype, int batch_chunk,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * fa_fwd_unfused — the unfused forward, kept as a measured comparison for
 * fa_fwd (not the fused method).
 *
 * Source: "Lesson K23, fused attention" facts page, `sources.flashAttention`
 * (Algorithm 0) and block `traffic`: S = scale Q K^T is written to global
 * memory, a row softmax reads S and writes P, then O = P V reads P, so each
 * head moves its N x N matrices through DRAM (4 N^2 bytes of extra memory).
 * Here S is float32 [B, H, N, N] in `workspace`; the row softmax writes
 * exp(S - m) (16-bit) over the first half of each S row and the row sums l;
 * O = (exp(S - m) V) / l, the product in float32, divided and rounded once
 * by the library's kernel.  The two matrix products are plain cuBLAS GEMMs
 * (16-bit inputs, float32 accumulation) loaded on first use.  Same outputs
 * as fa_fwd (o, lse), up to rounding.
 *
 *   q, k, v, o, lse, B, H, N, d, scale, causal : as in fa_fwd
 *   dtype      : BF16 or F16 (F32 returns FA_ERR_UNSUPPORTED)
 *   workspace  : DEVICE, 256-byte aligned, >= fa_fwd_unfused_workspace_size
 *                (B, H, N, d) bytes: S (4 B H N^2), the float32 product
 *                (4 B N H d), l (4 B H N), each rounded up to 256 bytes, then
 *                the GEMMs' workspace (32 MiB)
 * Returns FA_ERR_UNSUPPORTED if cuBLAS cannot be loaded.  The first call on
 * a device creates a cuBLAS handle; calls are serialised on the host.
 */
size_t fa_fwd_unfused_workspace_size(int B, int H, int N, int d);
fa_status fa_fwd_unfused(const void* q, const void* k, const void* v, void* o, float* lse,
                         int B, int H, int N, int d, float scale, int causal,
                         fa_dtype dtype, void* workspace, size_t workspace_bytes,
                         void* stream);

/*
 * fa_fwd_tf32x3 — float32 forward on the tensor cores.
 *
 * Same operation and outputs as fa_fwd with FA_DTYPE_F32 ("Flash Attention 2
 * — forward pass notes", sections "Loop (per (b, h, Q-tile))" and "What's
 * still needed for full FA2" item 1), computed with tcgen05 kind::tf32
 * products instead of the float32 FMA pipes.  Every float32 input x is
 * split into hi (x rounded to tf32) and lo (x - hi rounded to tf32), and each
 * product is taken as hi*hi + hi*lo + lo*hi (3xTF32), in Q K^T and in P V
 * alike; accumulation, the softmax and the outputs are float32.  The
 * relative error per product is at most about 3 * 2^-22.  Inputs must be
 * finite with |x| < 2^127.
 *
 *   q, k, v   in : [B, N, H, d] float32
 *   o        out : [B, N, H, d] float32;  lse out : [B, H, N] float32
 *   d            : a multiple of 8 in [8, 128]; d <= 64 runs 64-key blocks,
 *                  d in (64, 128] 32-key blocks (the hi/lo Q tile of 128
 *                  rows then takes 128 KB of shared memory)
 *   workspace    : DEVICE, 256-byte aligned, >= fa_fwd_tf32x3_workspace_size
 *                  (B, H, N, d) bytes: the hi/lo split of q, k and v (v
 *                  transposed per head), 6 float32 copies of an input
 *   other arguments as in fa_fwd.
 */
size_t fa_fwd_tf32x3_workspace_size(int B, int H, int N, int d);
fa_status fa_fwd_tf32x3(const float* q, const float* k, const float* v, float* o, float* lse,
                        int B, int H, int N, int d, float scale, int causal,
                        void* workspace, size_t workspace_bytes, void* stream);

/* fa_status_string — static, human-readable name of a status code. */
const char* fa_status_string(fa_status s);

/*
 * fa_bwd_tf32x3 — float32 backward on the tensor cores: the gradients of
 * fa_fwd / fa_fwd_tf32x3 ("Flash Attention 2 — backward pass notes", "The
 * math (FA2 backward with recompute)", split as option 3 of "Why the WGSL
 * kernel isn't shipped this turn": one kernel per query tile writes dQ, one
 * per key tile writes dK and dV, D = rowsum(dO * O) first) with every product
 * taken as three tcgen05 kind::tf32 products of hi / lo tf32 parts
 * (hi*hi + hi*lo + lo*hi).
 *   q, k, v, o, dO : DEVICE, float32 [B, N, H, d], 16-byte aligned
 *   lse            : DEVICE, float32 [B, H, N] (the forward's)
 *   dq, dk, dv     : DEVICE, float32 [B, N, H, d], 16-byte aligned, written
 *   d              : a multiple of 8, at most 64 (FA_ERR_UNSUPPORTED above)
 *   workspace      : DEVICE, 256-byte aligned, >= fa_bwd_tf32x3_workspace_size
 *                    bytes (D, the hi / lo copies of Q, K, V, dO and the
 *                    transposed hi / lo copies of Q, K, dO); caller-owned
 * Validation, aliasing rules, errors and the status word as fa_bwd.
 */
size_t fa_bwd_tf32x3_workspace_size(int B, int H, int N, int d);
fa_status fa_bwd_tf32x3(const float* q, const float* k, const float* v, const float* o,
                        const float* lse, const float* dO, float* dq, float* dk, float* dv,
                        int B, int H, int N, int d, float scale, int causal, void* workspace,
                        size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_H */
