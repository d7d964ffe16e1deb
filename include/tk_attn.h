/*
 * tk_attn.h -- C ABI of the GB300 (sm_103a) fused attention forward.
 *
 * One call computes, for every batch b and head h,
 *
 *     O   = softmax(scale * Q K^T [+ causal mask]) V
 *     LSE = per query row, ln(sum_j exp(scale * <Q_i, K_j>)) over the keys j
 *           the row may see
 *
 * in one fused kernel: the N x N score matrix never reaches global memory
 * (online softmax over key tiles, one division by the row sum at the end).
 *
 * The computation is the attention forward pass of the "ThunderKittens"
 * attention kernel (10100.com/article/71410160, section "writing a kernel
 * with TK": attn_fwd_template, whose consumer::compute forms Q K^T, keeps a
 * running row max and row sum in the exp2 domain with scale*log2(e) folded
 * in, rescales the partial output and adds P V; consumer::finish divides by
 * the row sum), together with the ragged-tail masking of the inner-loop
 * excerpt on alanwu.xyz/posts/thunderkittens (keys past the end take -inf).
 * Readings taken where the pages are silent:
 *   - LSE is in natural log and includes scale: LSE_i = scale*max_j s_ij +
 *     ln(sum_j exp(scale*(s_ij - max_j s_ij))) with s_ij = <Q_i, K_j>.  The
 *     pages store no LSE.
 *   - causal = 1 means key j is visible to query i iff j <= i (top-left
 *     aligned, equal query and key lengths).  The pages have no mask.
 *   - scale is a runtime argument (the pages hard-code 1/sqrt(D)); it must
 *     be finite and > 0, because the kernel takes the row maximum of the
 *     unscaled scores, as the pages do.
 *
 * All entry points are thread-safe.  None of them allocates device memory.
 */
#ifndef TK_ATTN_H
#define TK_ATTN_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
enum {
    TK_OK = 0,
    TK_ERR_NULL_PTR = 1,           /* a required pointer is NULL                       */
    TK_ERR_BAD_SHAPE = 2,          /* B, H or N < 1, or B*H*N*D overflows               */
    TK_ERR_UNSUPPORTED_D = 3,      /* head dim other than 64 or 128                      */
    TK_ERR_MISALIGNED = 4,         /* Q, K, V or O not 16-byte aligned, LSE not 4-byte   */
    TK_ERR_BAD_SCALE = 5,          /* scale not finite or not > 0                         */
    TK_ERR_ALIAS = 6,              /* O or LSE overlaps an input, or O overlaps LSE       */
    TK_ERR_BAD_FLAG = 7,           /* causal not 0 or 1                                   */
    TK_ERR_UNSUPPORTED_DEVICE = 8, /* current device is not compute capability 10.3       */
    TK_ERR_CUDA = 9,               /* a CUDA runtime/driver call or the launch failed     */
    TK_ERR_DEVICE_TIMEOUT = 10,    /* a bounded wait inside a kernel gave up (see below) */
    TK_ERR_NOT_DEVICE_MEMORY = 11  /* a pointer is not device (or managed) memory        */
};

/*
 * tk_attn_fwd -- fused attention forward.
 *
 * Arguments
 *   Q, K, V  device pointers, bf16, contiguous [B, H, N, D] (row stride D,
 *            head stride N*D, batch stride H*N*D elements), 16-byte aligned.
 *   O        device pointer, bf16, contiguous [B, H, N, D], 16-byte aligned.
 *            Written: O[b,h,i,:] = sum_j P_ij V[b,h,j,:], rounded to bf16
 *            (round to nearest even).
 *   LSE      device pointer, fp32, contiguous [B, H, N], 4-byte aligned.
 *            Written: the natural-log log-sum-exp of row i's scaled scores.
 *   B, H, N  batch, heads, sequence length (queries = keys = N); each >= 1.
 *            Any N >= 1: the last key tile is masked, the last query tile's
 *            extra rows are neither computed into nor stored.
 *   D        head dimension: 64 or 128.
 *   causal   0: every query sees every key; 1: query i sees keys j <= i.
 *   scale    multiplier of Q K^T, finite and > 0 (usually 1/sqrt(D)).
 *   stream   CUDA stream the kernel is enqueued on (0 = legacy default).
 *
 * Ownership: the caller owns every buffer; the library keeps no pointer
 * after the call returns and allocates nothing.  It caches, per device, the
 * SM count and the kernel attributes.  O and LSE must not overlap Q, K, V or
 * each other.
 *
 * Semantics: asynchronous.  The call validates its arguments, enqueues one
 * kernel on `stream` and returns without synchronising; O and LSE are valid
 * once the stream reaches that point.  Results are deterministic: the same
 * inputs give bitwise-identical outputs on every call.
 *
 * Errors: invalid arguments are reported before anything is enqueued and
 * leave O and LSE untouched (codes 1-8 and 11).  TK_ERR_CUDA reports a failed launch
 * or runtime call (see tk_attn_last_cuda_error).  Waits inside the kernel are
 * bounded in time; if one gives up, the kernel stops early, its outputs are
 * undefined, and tk_attn_device_status reports TK_ERR_DEVICE_TIMEOUT.
 */
int tk_attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE,
                int64_t B, int64_t H, int64_t N, int64_t D, int causal, float scale,
                cudaStream_t stream);

/*
 * tk_attn_device_status -- synchronises `stream`, then reads and clears the
 * current device's kernel status word.  Returns TK_OK if no bounded wait of
 * any kernel of this library on this device has given up since the last
 * call, TK_ERR_DEVICE_TIMEOUT if one has, TK_ERR_CUDA if the synchronisation
 * itself failed.  *detail (may be NULL) receives the role and step at which
 * the first wait gave up (0 if none).
 */
int tk_attn_device_status(cudaStream_t stream, uint32_t *detail);

/*
 * tk_attn_selftest_timeout -- enqueues a one-CTA kernel that waits, with the
 * same bounded wait the attention kernel uses, on a shared-memory barrier
 * that nothing signals, for at most `limit_ns` nanoseconds (clamped to
 * [1e3, 5e9]).  The wait gives up, records TK_ERR_DEVICE_TIMEOUT in the
 * status word and the kernel returns normally: no trap, no hang.  Used to
 * test the failure path; read the result with tk_attn_device_status.
 */
int tk_attn_selftest_timeout(uint64_t limit_ns, cudaStream_t stream);

/* Static English description of a status code (never NULL). */
const char *tk_attn_strerror(int code);

/* The cudaError_t of the most recent TK_ERR_CUDA on this thread (0 if none). */
int tk_attn_last_cuda_error(void);

/* Library ABI version: (major << 16) | minor. */
int tk_attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* TK_ATTN_H */
