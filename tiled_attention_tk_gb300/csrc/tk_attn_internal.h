// tk_attn_internal.h -- types shared by the C-ABI layer and the kernel
// translation unit.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime_api.h>
#include <cstddef>
#include <cstdint>

namespace tk {

// Everything one launch of the fused forward kernel needs.  Passed by value
// as a __grid_constant__ kernel parameter (the tensor maps must stay in
// parameter space for TMA).
struct AttnParams {
    CUtensorMap tmQ;  // 3-D {D, Nq, B*H} bf16, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmK;  // 3-D {D, Nkv, B*H}, same box and swizzle
    CUtensorMap tmV;
    CUtensorMap tmO;  // the view of Q for O, for TMA stores
    CUtensorMap tmO32;  // the same view moved as 32-row boxes {64, 32, 1} (per-warp stores)
    void *O;          // bf16 [B*H, Nq, D]
    float *LSE;       // fp32 [B*H, Nq]
    int Nq;           // query rows
    int Nkv;          // key / value rows
    int offset;       // Nkv - Nq: causal query i sees keys j <= i + offset
    int BH;           // B * H
    int causal;       // 0 / 1
    int n_qtiles;     // ceil(Nq / 128)
    int n_kvtiles;    // ceil(Nkv / 128)
    int n_pairs;      // ceil(n_qtiles / 2): work units per head
    float scale;      // multiplier of Q K^T
    float scale_log2e;  // scale * log2(e): the exp2-domain factor
    // Tail split (non-causal only; split_pieces = 0: none).  The units of the
    // last, partial round run as two pieces each, over the first split_kv
    // key tiles and over the rest, on CTAs 0 .. split_pieces - 1 (tail unit
    // t on CTAs 2t and 2t + 1).  Each piece writes its O / l (fp32) and LSE
    // to `part`; the piece that publishes second merges the two.
    int split_round;                // the round whose units are split (= the full rounds)
    int split_pieces;               // 2 x the tail units
    int split_kv;                   // key tiles of the first piece
    float *part;                    // per piece and Q tile: 128 x D floats of O / l, then 128 LSE
    unsigned long long *ctr;        // per tail unit, Q tile and 32-row quarter: the last publisher's epoch
    unsigned long long epoch;       // this launch's tag (distinct for every split launch)
};

// Everything the backward kernels need.
struct BwdParams {
    CUtensorMap tmQ;   // 3-D {D, N, B*H} bf16 views, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmK;
    CUtensorMap tmV;
    CUtensorMap tmDO;
    const void *O;     // bf16 [B*H, N, D] (forward output)
    const void *dO;    // bf16 [B*H, N, D]
    const float *LSE;  // fp32 [B*H, N] (forward log-sum-exp)
    float *neg_delta;  // workspace: fp32 [B*H, n_tiles*128], -<dO_i, O_i> (0 past N)
    float *neg_lse2;   // workspace: fp32 [B*H, n_tiles*128], -LSE_i * log2(e) (-inf past N)
    float *dq_acc;     // workspace: fp32 dQ accumulator, per head [n_tiles][D/4][128][4]
    void *dQ;          // bf16 [B*H, N, D]
    void *dK;
    void *dV;
    int N;
    int D;             // head dim of the tensors (32, 64, 96, 128); the kernel's is 64 or 128
    int BH;
    int causal;
    int n_tiles;       // ceil(N / 128)
    float scale;
    float scale_log2e;
};

// Launches the backward pass (prep, main, dQ conversion) for head dim D.
cudaError_t launch_attn_bwd(int D, const BwdParams &p, int num_sms, cudaStream_t stream);

// Everything the GEMM kernel needs (C = A op(B), bf16 in and out, fp32 accumulation).
struct GemmParams {
    CUtensorMap tmA;   // 3-D {K, M, 1} bf16, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmB;   // b_kmajor: {K, N, 1}, box {64, 256, 1}; else {N, K, 1}, box {64, 64, 1}
    CUtensorMap tmC;   // {N, M, 1}, box {64, 32, 1}, for TMA stores
    float *partials;   // workspace: one 128 x 256 fp32 stream-K partial slot per CTA
    unsigned *counters;  // workspace: per stream-K tile, partials published (x4 warps)
    int M, N, K;
    int b_kmajor;      // 1: B is [N, K] (C = A B^T); 0: B is [K, N] (C = A B)
    int tiles_m, tiles_n, k_iters;
    int group_m;       // tile rows per L2 group of the tile order
    int dp_tiles;      // tiles [0, dp_tiles): whole tiles, round-robin over the CTAs
    int sk_tiles;      // tiles [dp_tiles, dp_tiles + sk_tiles): split in K (stream-K)
    int sk_iters_per_cta;  // K iterations of the stream-K range of each worker (CTA, or pair)
    int pair;          // 1: CTA pairs (cta_group::2) on 256 x 256 tiles; tiles_m counts 256-row tiles,
                       // tmB's box is {64, 128, 1} when b_kmajor, the schedule's CTAs are pairs
                       // (grid = 2 x pairs) and a partial slot is 256 x 256
};

cudaError_t launch_gemm(const GemmParams &p, int grid, cudaStream_t stream);
// CTA pairs of the GEMM's pair kernel that can be resident at once on the current device.
cudaError_t gemm_pair_capacity(int *pairs);
cudaError_t read_and_clear_gemm_status(uint32_t *status, uint32_t *detail);

// Everything the Based linear-attention kernel needs (Dqk = 16, Dv = 64).
struct BasedParams {
    CUtensorMap tmQ;   // 3-D {16, N, B*H} bf16, box {64, 128, 1} (columns 16..63 read as 0), 128-byte swizzle
    CUtensorMap tmK;
    CUtensorMap tmV;   // 3-D {64, N, B*H} bf16, box {64, 128, 1}
    CUtensorMap tmO;   // 3-D {64, N, B*H} bf16, box {32, 32, 1}, 64-byte swizzle (stores)
    void *O;           // bf16 [B*H, N, 64]
    float *DEN;        // fp32 [B*H, N]
    float *ws;         // segment states [B*H][n_seg][80][160] fp32 (n_seg > 1), else unused
    int N;
    int BH;
    int n_seg;         // segments per head (1: one CTA walks the whole head)
    int seg_chunks;    // 128-row chunks per segment
    float scale;
    // Balanced schedule (balanced = 1): the chunks of all heads cut into one
    // run per CTA; a head split between two CTAs passes its state through
    // `carry` ([B*H][80][160] fp32), each of the 8 compute warps raising its
    // own flag ([B*H][8], set to `epoch`, distinct for every launch).
    int balanced;
    float *carry;
    unsigned long long *flags;
    unsigned long long epoch;
};

cudaError_t launch_based(const BasedParams &p, cudaStream_t stream);
cudaError_t launch_based_states(const BasedParams &p, cudaStream_t stream);
cudaError_t read_and_clear_based_status(uint32_t *status, uint32_t *detail);

// Everything the Hedgehog linear-attention kernel needs (d = f = Dv = 64).
struct HedgehogParams {
    CUtensorMap tmQ;   // 3-D {64, N, B*H} bf16, box {64, 128, 1}, 128-byte swizzle
    CUtensorMap tmK;
    CUtensorMap tmV;
    CUtensorMap tmWq;  // 3-D {f, d, H} bf16 (W of head h: [d][f]), box {64, 64, 1}
    CUtensorMap tmWk;
    CUtensorMap tmO;   // 3-D {64, N, B*H} bf16, box {32, 32, 1}, 64-byte swizzle (stores)
    void *O;           // bf16 [B*H, N, 64]
    float *DEN;        // fp32 [B*H, N]
    float *ws;         // segment states [B*H][n_seg][80][128] fp32 (n_seg > 1), else unused
    int N;
    int H;
    int BH;
    int n_seg;         // segments per head (1: one CTA walks the whole head)
    int seg_chunks;    // 128-row chunks per segment
};

cudaError_t launch_hedgehog(const HedgehogParams &p, cudaStream_t stream);
cudaError_t launch_hedgehog_states(const HedgehogParams &p, cudaStream_t stream);
cudaError_t read_and_clear_hedgehog_status(uint32_t *status, uint32_t *detail);

// Size of the library-owned workspace behind tk_attn_bwd_noalloc.
constexpr size_t kNoAllocWorkspaceBytes = size_t(32) << 20;

// Device address of that workspace on the current device (looked up once
// per device, then cached).  Allocates nothing.
cudaError_t noalloc_workspace(void **ptr);

// Reads and clears the backward translation unit's status word (no sync).
cudaError_t read_and_clear_bwd_status(uint32_t *status, uint32_t *detail);

// Launches the fused forward kernel for head dim D (32, 64, 96 or 128).
cudaError_t launch_attn_fwd(int D, const AttnParams &p, int num_sms, cudaStream_t stream);

// The forward at head dim 256 (attn_fwd256.cu: one Q tile per unit, two S
// slots), and its device status word.
cudaError_t launch_attn_fwd256(const AttnParams &p, int num_sms, cudaStream_t stream);
cudaError_t read_and_clear_fwd256_status(uint32_t *status, uint32_t *detail);

// Launches the one-CTA bounded-wait self test.
cudaError_t launch_selftest_timeout(uint64_t limit_ns, cudaStream_t stream);

// Synchronises `stream`, reads and clears the device status word.
cudaError_t read_and_clear_status(cudaStream_t stream, uint32_t *status, uint32_t *detail);

}  // namespace tk
