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

#include <stddef.h>
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
    TK_ERR_UNSUPPORTED_D = 3,      /* head dim the entry point does not take              */
    TK_ERR_MISALIGNED = 4,         /* Q, K, V or O not 16-byte aligned, LSE not 4-byte   */
    TK_ERR_BAD_SCALE = 5,          /* scale not finite or not > 0                         */
    TK_ERR_ALIAS = 6,              /* O or LSE overlaps an input, or O overlaps LSE       */
    TK_ERR_BAD_FLAG = 7,           /* causal not 0 or 1                                   */
    TK_ERR_UNSUPPORTED_DEVICE = 8, /* current device is not compute capability 10.3       */
    TK_ERR_CUDA = 9,               /* a CUDA runtime/driver call or the launch failed     */
    TK_ERR_DEVICE_TIMEOUT = 10,    /* a bounded wait inside a kernel gave up (see below) */
    TK_ERR_NOT_DEVICE_MEMORY = 11, /* a pointer is not device (or managed) memory        */
    TK_ERR_WORKSPACE = 12,         /* workspace too small or not 256-byte aligned         */
    TK_ERR_NOALLOC_TOO_LARGE = 13  /* tk_attn_bwd_noalloc: workspace need above 32 MiB    */
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
 *   D        head dimension: 32, 64, 96, 128 or 256 (the backward: 32, 64, 96
 *            or 128).
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
 * tk_attn_fwd_kv -- the same forward for Nq queries against Nkv keys
 * (attention inference over a cache: a block of new queries attends to every
 * earlier key and to itself; the groovesquid.com summary of the
 * ThunderKittens paper lists "attention inference" among its kernels).
 *
 * Arguments as tk_attn_fwd, except
 *   Q, O     bf16 [B, H, Nq, D];  LSE fp32 [B, H, Nq].
 *   K, V     bf16 [B, H, Nkv, D].
 *   Nq, Nkv  query and key rows, each >= 1 (any values, ragged tails masked).
 *   causal   0: every query sees every key.  1: the queries stand at the end
 *            of the key sequence, query i at position i + Nkv - Nq, and see
 *            keys j <= i + Nkv - Nq; needs Nkv >= Nq (else TK_ERR_BAD_SHAPE).
 * With Nq = Nkv = N it is tk_attn_fwd.  Semantics, ownership and errors as
 * tk_attn_fwd.
 */
int tk_attn_fwd_kv(const void *Q, const void *K, const void *V, void *O, float *LSE,
                   int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D, int causal,
                   float scale, cudaStream_t stream);

/*
 * tk_attn_fwd_workspace_bytes -- device workspace tk_attn_fwd_ws needs on
 * the current device for this shape: nonzero only without the causal mask,
 * at a head dim below 256, with at least 4 key tiles (Nkv > 384), when the
 * work units (pairs of 128-row query tiles, B*H*ceil(ceil(Nq/128)/2) of
 * them) fill some rounds of one unit per SM and leave a last round at most
 * half full.  Then each unit of that round is split in two by key tiles:
 * 2*T pieces for T tail units need 2*T*2*128*(D+1)*4 bytes of partial
 * results (rounded up to 256) plus T*64 bytes of counters (rounded up to
 * 256).  0 for any other shape, including one tk_attn_fwd_ws rejects.
 * There is no counterpart on the pages: it balances the last round on this
 * GPU's SM count.
 */
size_t tk_attn_fwd_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D, int causal);

/*
 * tk_attn_fwd_ws -- tk_attn_fwd_kv with the last, partial round of work
 * units split by key tiles when tk_attn_fwd_workspace_bytes says so.  A
 * split unit's two pieces each leave O/l (fp32) and their LSE in the
 * workspace; the piece that publishes second merges them,
 *     LSE = m + ln(w_a + w_b),  w = exp(LSE_piece - m),  m = max(LSE_a, LSE_b)
 *     O   = (w_a O_a + w_b O_b) / (w_a + w_b),
 * the same combination of partial softmax sums the online softmax uses
 * across key tiles, with unfused fp32 products and sums so that the result
 * does not depend on which piece merges.  Deterministic.
 *
 * Arguments as tk_attn_fwd_kv, plus
 *   workspace        device memory of at least tk_attn_fwd_workspace_bytes
 *                    bytes for this shape, 256-byte aligned, not overlapping
 *                    any other argument; may be NULL when that size is 0
 *                    (then this is tk_attn_fwd_kv).  Owned by the caller,
 *                    overwritten; no clearing is needed between calls.  Two
 *                    calls in flight at once need two workspaces.
 *   workspace_bytes  its size.
 * Errors as tk_attn_fwd_kv, plus TK_ERR_WORKSPACE (too small or
 * misaligned), TK_ERR_NULL_PTR (NULL where one is needed) and TK_ERR_ALIAS
 * (the workspace overlapping an argument).
 */
int tk_attn_fwd_ws(const void *Q, const void *K, const void *V, void *O, float *LSE, void *workspace,
                   size_t workspace_bytes, int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D,
                   int causal, float scale, cudaStream_t stream);

/*
 * tk_attn_bwd_workspace_bytes -- device workspace tk_attn_bwd needs for a
 * problem of this shape: an fp32 dQ accumulator over whole 128-row query
 * tiles (B*H*ceil(N/128)*128*Dk floats, Dk = 64 for D = 32 or 64 and 128 for
 * D = 96 or 128: head dims 32 and 96 run on the 64- and 128-column kernels,
 * their missing columns read as zeros) and two fp32 row values over the same
 * padded rows, Delta_i = <dO_i, O_i> and -LSE_i*log2(e); each section
 * 256-byte aligned.
 * Returns 0 for shapes tk_attn_bwd rejects: TK_ERR_BAD_SHAPE, or a head dim
 * other than 32, 64, 96 and 128 (TK_ERR_UNSUPPORTED_D).
 */
size_t tk_attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D);

/*
 * tk_attn_bwd -- attention backward: the gradients of L = sum(O * dO) with
 * respect to Q, K and V for O = softmax(scale * Q K^T [+ causal mask]) V.
 * The pages list attention backwards among the kernels built with the same
 * tiles (groovesquid.com summary of the ThunderKittens paper, "attention
 * backwards"); it is the chain rule through the forward above:
 *     P_ij  = exp(scale <Q_i,K_j> - LSE_i)   (LSE from tk_attn_fwd)
 *     dV_j  = sum_i P_ij dO_i
 *     dS_ij = scale * P_ij (<dO_i,V_j> - <dO_i,O_i>)
 *     dQ_i  = sum_j dS_ij K_j,   dK_j = sum_i dS_ij Q_i
 * P and dS are rounded to bf16 for the tensor-core products (as the forward
 * rounds P); dQ accumulates in fp32 across key tiles.
 *
 * Arguments
 *   Q, K, V   the forward's inputs (device, bf16 [B,H,N,D], 16-byte aligned).
 *   O, LSE    the forward's outputs for them (bf16 [B,H,N,D]; fp32 [B,H,N]).
 *   dO        gradient of the loss with respect to O (bf16 [B,H,N,D]).
 *   dQ, dK, dV  outputs, bf16 [B,H,N,D], 16-byte aligned, written in full.
 *   workspace device memory of at least tk_attn_bwd_workspace_bytes(B,H,N,D)
 *             bytes, 256-byte aligned; owned by the caller, overwritten.
 *   B, H, N, D, causal, scale, stream: as for tk_attn_fwd.
 *
 * Semantics: asynchronous on `stream` (three kernels: row values, main,
 * dQ rounding).  dK and dV are deterministic; dQ sums fp32 contributions of
 * the key tiles with bulk atomic adds, so its last bits may vary between
 * runs.
 * Errors: as tk_attn_fwd, plus TK_ERR_NULL_PTR for a NULL workspace and
 * TK_ERR_WORKSPACE (too small or misaligned).  Outputs must not overlap the
 * inputs, each other or the workspace (TK_ERR_ALIAS).
 */
int tk_attn_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                const float *LSE, void *dQ, void *dK, void *dV, void *workspace,
                size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t D, int causal,
                float scale, cudaStream_t stream);

/*
 * tk_attn_bwd_noalloc -- tk_attn_bwd without a caller workspace.  The paper
 * has no counterpart: this entry point exists for callers that cannot
 * allocate device memory, for instance code running under a framework or
 * pool allocator that owns all of the device's memory (a raw cudaMalloc
 * would fail or fragment it), or a latency-critical path that cannot take
 * cudaMalloc's implicit device-wide synchronisation.  It allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library routine.
 *
 * The workspace is a fixed 32 MiB array inside the library (every device
 * that loads the library holds it until the process exits).  Problems whose
 * workspace (tk_attn_bwd_workspace_bytes) exceeds 32 MiB are rejected with
 * TK_ERR_NOALLOC_TOO_LARGE before anything is enqueued; with D = 128 that is
 * B*H*N above about 64 thousand rows.
 *
 * Arguments, results and errors are those of tk_attn_bwd without
 * `workspace` and `workspace_bytes`.  The first call on a device looks up
 * the array's device address (once per device, with that device current);
 * make that first call before any stream capture.  All calls share the one
 * array and it keeps the last call's contents (each call re-zeroes what it
 * accumulates into), so calls whose work overlaps on the GPU -- on
 * different streams without ordering between them -- race: serialise them.
 */
int tk_attn_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                        const float *LSE, void *dQ, void *dK, void *dV, int64_t B, int64_t H,
                        int64_t N, int64_t D, int causal, float scale, cudaStream_t stream);

/*
 * tk_gemm_workspace_bytes -- device workspace tk_gemm needs on the current
 * device for this shape: 0 when the schedule has no stream-K part (also for a
 * shape tk_gemm rejects), else one 128 x 256 fp32 partial-sum slot per CTA of
 * the grid (a pair of CTAs shares a 256 x 256 slot) plus one counter per
 * stream-K tile, each section 256-byte aligned.
 */
size_t tk_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int stream_k);

/*
 * tk_gemm_uses_pairs -- 1 if tk_gemm runs this shape on CTA pairs on the
 * current device (see tk_gemm), 0 if on single CTAs; 0 also for a shape or
 * flag tk_gemm rejects, or when no device is usable.  Enqueues nothing.
 */
int tk_gemm_uses_pairs(int64_t M, int64_t N, int64_t K, int stream_k);

/*
 * tk_gemm -- C = A op(B) on the same TMA + tcgen05 pipeline as the attention
 * kernels, with a persistent grid, an L2-grouped tile order and stream-K for
 * the last wave.  The pages name GEMM as the workload the tile abstractions
 * are built around and threadblock swizzle plus persistent grid + stream-K
 * as the cures for its L2 hit rate and wave quantisation
 * (10100.com/article/71410160, section on grid-level abstraction).
 * Large problems (at least one wave of 256 x 256 tiles over pairs of SMs,
 * K >= 768) run on CTA pairs (two-SM tcgen05 products, each SM loading half
 * of each operand tile); there stream-K splits the last waves only below four
 * waves of pair tiles.  Either path gives the same C bit for bit when no tile
 * is split in K (each output element is one fp32 dot product in k order).
 *
 *   C[m,n] = sum_k A[m,k] * B'[k,n],  fp32 accumulation, C rounded to bf16
 *            (round to nearest even), where B' = B^T if b_kmajor else B.
 *
 * Arguments
 *   A          device bf16 [M, K] row-major, 16-byte aligned.
 *   B          device bf16 [N, K] row-major if b_kmajor = 1 (C = A B^T), or
 *              [K, N] row-major if b_kmajor = 0 (C = A B); 16-byte aligned.
 *   C          device bf16 [M, N] row-major, 16-byte aligned, written in full.
 *   workspace  device memory of at least tk_gemm_workspace_bytes(M,N,K,
 *              stream_k) bytes, 256-byte aligned (may be NULL when that is 0).
 *   M, N, K    >= 1; K and N multiples of 8 (16-byte row strides).
 *   b_kmajor   0 or 1, as above.
 *   stream_k   1: split the last wave's tiles in K over all SMs when the
 *              tiles do not fill whole waves; 0: whole tiles only.
 *   stream     CUDA stream (0 = legacy default).
 * Semantics: asynchronous on `stream` (a memset of the stream-K counters and
 * one kernel).  Deterministic: the stream-K partial sums are added in a fixed
 * order.  Errors: TK_ERR_NULL_PTR, TK_ERR_BAD_SHAPE, TK_ERR_BAD_FLAG,
 * TK_ERR_MISALIGNED, TK_ERR_ALIAS (C or the workspace overlapping an input or
 * each other), TK_ERR_WORKSPACE, TK_ERR_NOT_DEVICE_MEMORY,
 * TK_ERR_UNSUPPORTED_DEVICE, TK_ERR_CUDA; all reported before anything is
 * enqueued.  Bounded waits as for the attention kernels.
 */
int tk_gemm(const void *A, const void *B, void *C, void *workspace, size_t workspace_bytes, int64_t M,
            int64_t N, int64_t K, int b_kmajor, int stream_k, cudaStream_t stream);

/*
 * tk_based_fwd -- causal Based linear attention (the linear-attention kernel
 * the pages list as "Based Linear Attention", thebeat.tech "ThunderKittens
 * 2.0", New Kernels; the formula is the Based feature map, the second-order
 * Taylor expansion of exp):
 *     s_ij  = scale <Q_i, K_j>,   w_ij = 1 + s_ij + s_ij^2 / 2   (j <= i)
 *     DEN_i = sum_j w_ij,         O_i  = sum_j w_ij V_j / DEN_i
 * computed in linear time: chunks of 128 rows, a running state of the
 * feature map's 153 features in TMEM, tensor-core products for the
 * in-chunk and carried parts.
 *
 * Arguments
 *   Q, K   device bf16 [B, H, N, Dqk], Dqk = 16, 16-byte aligned.
 *   V, O   device bf16 [B, H, N, Dv], Dv = 64, 16-byte aligned (O written).
 *   DEN    device fp32 [B, H, N], 4-byte aligned (written): the normaliser,
 *          so O_i * DEN_i is the unnormalised sum.
 *   scale  finite, > 0 (usually 1/sqrt(Dqk) = 0.25).
 * Semantics, ownership and errors as tk_attn_fwd (TK_ERR_UNSUPPORTED_D for
 * any other Dqk, Dv).  Deterministic.
 */
int tk_based_fwd(const void *Q, const void *K, const void *V, void *O, float *DEN, int64_t B, int64_t H,
                 int64_t N, int64_t Dqk, int64_t Dv, float scale, cudaStream_t stream);

/*
 * tk_based_workspace_bytes -- the workspace tk_based_fwd_ws needs on the
 * current device for [B, H, N]:
 *   - B*H below the SM count: B*H * n_seg * 51,200 bytes (rounded up to 256)
 *     for the partial states of n_seg segments per head (0 when the heads
 *     are too short to split);
 *   - B*H above the SM count, where one CTA per head would leave more than
 *     eight 128-row chunks per SM idle in the last wave ((waves * SMs - B*H)
 *     * ceil(N/128) > 8 * SMs): B*H * 51,200 bytes (rounded up to 256) for
 *     the states of heads split between two CTAs, plus B*H * 64 bytes
 *     (rounded up to 256) of flags (balanced schedule);
 *   - otherwise 0 (one CTA walks each head, as in tk_based_fwd).
 * 0 also for an invalid shape (tk_based_fwd_ws then reports it).
 */
size_t tk_based_workspace_bytes(int64_t B, int64_t H, int64_t N);

/*
 * tk_based_fwd_ws -- tk_based_fwd with the work balanced over the SMs.
 * With fewer heads than SMs the sequence is split into segments: a first
 * pass forms each segment's partial state sum_j [V_j | 1] phi(K_j)^T (fp32,
 * into `workspace`), then one CTA per segment starts from the sum of the
 * partial states before it; same result as tk_based_fwd up to the order of
 * fp32 additions.  With more heads than SMs and a last wave of heads that
 * would leave SMs idle for long, the heads' chunks, laid end to end, are cut
 * into one equal run per SM: a head
 * split between two CTAs passes its exact fp32 state from the first to the
 * second through `workspace`, and the result is bitwise that of
 * tk_based_fwd (one kernel, launched cooperatively so that every CTA is
 * resident).  There is no counterpart on the pages for either split.
 *
 * Arguments as tk_based_fwd, plus
 *   workspace        device memory of at least tk_based_workspace_bytes(B,H,N)
 *                    bytes, 256-byte aligned, not overlapping any other
 *                    argument; may be NULL when that size is 0 (then this is
 *                    tk_based_fwd).  Owned by the caller, overwritten.
 *   workspace_bytes  its size.
 * Semantics: asynchronous on `stream` (two kernels when segmented).
 * Deterministic.  Errors as tk_based_fwd, plus TK_ERR_WORKSPACE (too small
 * or misaligned), TK_ERR_NULL_PTR (NULL where one is needed) and
 * TK_ERR_ALIAS (the workspace overlapping an argument).
 */
int tk_based_fwd_ws(const void *Q, const void *K, const void *V, void *O, float *DEN, void *workspace,
                    size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t Dqk, int64_t Dv, float scale,
                    cudaStream_t stream);

/*
 * tk_hedgehog_fwd -- causal Hedgehog linear attention (the pages list
 * "LoLCATS Hedgehog Linear Attention", thebeat.tech "ThunderKittens 2.0", New
 * Kernels; the formula is the Hedgehog feature map):
 *     phi_q(x) = [softmax(x Wq), softmax(-x Wq)],  phi_k likewise with Wk
 *     w_ij = phi_q(Q_i) . phi_k(K_j)  (j <= i),   DEN_i = sum_j w_ij,
 *     O_i  = sum_j w_ij V_j / DEN_i
 * in linear time (128-row chunks, running state of the 128 features).
 *
 * Arguments
 *   Q, K, V, O   device bf16 [B, H, N, 64], 16-byte aligned (O written).
 *   Wq, Wk       device bf16 [H, Dqk = 64, F = 64] (the projection of head h
 *                is Wq[h], row-major [64][64]), 16-byte aligned.
 *   DEN          device fp32 [B, H, N] (written).
 *   Dqk, F, Dv   must be 64, 64, 64 (else TK_ERR_UNSUPPORTED_D).
 * Semantics, ownership and errors as tk_attn_fwd.  Deterministic.
 */
int tk_hedgehog_fwd(const void *Q, const void *K, const void *V, const void *Wq, const void *Wk, void *O,
                    float *DEN, int64_t B, int64_t H, int64_t N, int64_t Dqk, int64_t F, int64_t Dv,
                    cudaStream_t stream);

/*
 * tk_hedgehog_workspace_bytes / tk_hedgehog_fwd_ws -- tk_hedgehog_fwd with
 * the sequence split into segments when the B*H heads are fewer than the
 * SMs, as tk_based_workspace_bytes / tk_based_fwd_ws describe for Based: a
 * first pass forms each segment's fp32 partial state sum_j [V_j | 1]
 * phi_k(K_j)^T (B*H * n_seg * 40,960 bytes of workspace, rounded up to 256;
 * 0 when no split is needed or the shape is invalid), then one CTA per
 * segment starts from the sum of those before it.  Arguments as
 * tk_hedgehog_fwd plus `workspace` (device, 256-byte aligned, not
 * overlapping any argument; NULL allowed when the size is 0) and its size.
 * Errors as tk_hedgehog_fwd plus TK_ERR_WORKSPACE, TK_ERR_NULL_PTR and
 * TK_ERR_ALIAS for the workspace.  Deterministic.
 */
size_t tk_hedgehog_workspace_bytes(int64_t B, int64_t H, int64_t N);
int tk_hedgehog_fwd_ws(const void *Q, const void *K, const void *V, const void *Wq, const void *Wk, void *O,
                       float *DEN, void *workspace, size_t workspace_bytes, int64_t B, int64_t H, int64_t N,
                       int64_t Dqk, int64_t F, int64_t Dv, cudaStream_t stream);

/*
 * tk_attn_device_status -- synchronises `stream`, then reads and clears the
 * current device's kernel status word.  Returns TK_OK if no bounded wait of
 * any kernel of this library on this device has given up since the last
 * call, TK_ERR_DEVICE_TIMEOUT if one has, TK_ERR_CUDA if the synchronisation
 * itself failed.  *detail (may be NULL) receives the role and step at which
 * the first wait gave up (0 if none).
 *
 * Scope: the status word belongs to the library on one device, not to a
 * stream or a call.  Kernels of every stream on that device record into it,
 * and the first timeout since the last read wins (later ones are dropped).
 * The call synchronises only `stream`: a timeout raised by a kernel still
 * running on another stream is seen by whichever call reads the word after
 * that kernel has finished, and reading clears it for every caller.  A
 * program that needs per-stream attribution calls this once per stream with
 * the other streams idle (for instance after cudaDeviceSynchronize()).
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
