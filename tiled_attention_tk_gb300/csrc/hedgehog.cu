// hedgehog.cu -- causal Hedgehog linear attention on tcgen05 (sm_103a, GB300).
//
// The pages list "LoLCATS Hedgehog Linear Attention" among the kernels built
// with the same tiles (thebeat.tech "ThunderKittens 2.0", New Kernels) without
// a formula.  The reading taken is the Hedgehog feature map, a softmax over a
// learned projection of the query (key) and over its negation:
//
//   phi_q(x) = [softmax(x Wq), softmax(-x Wq)],  phi_k(x) likewise with Wk
//   w_ij = phi_q(q_i) . phi_k(k_j),  O_i = sum_{j<=i} w_ij v_j / DEN_i,
//   DEN_i = sum_{j<=i} w_ij
//
// for d = 64 query/key dims, f = 64 features per half (128 in all) and
// value dim 64.  Same chunked linear form as the Based kernel: per 128-row
// chunk, Z = Q Wq and K Wk on the tensor core, the feature maps in the
// compute warps (into shared memory), S = phi(Q) phi(K)^T on the tensor core,
// the causal mask (P over S in TMEM), then [num | den] = P [V | 1] +
// phi(Q) S_{<c} and the state update S^T += [V | 1]^T phi(K).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tk_attn.h"
#include "tk_attn_internal.h"
#include "tk_ptx.cuh"
#include "tk_sync.cuh"

namespace tk {
namespace hedgehog {

constexpr int C = 128;             // rows per chunk
constexpr int DQK = 64;            // query / key dims
constexpr int FH = 64;             // features per half
constexpr int F = 2 * FH;          // feature dims of phi
constexpr int DV = 64;              // value dims: O rows leave as two 32-column boxes
constexpr int NV = 80;             // [num | den] columns (64 + 1, padded to a multiple of 16)
constexpr int NUM_THREADS = 320;   // two compute warpgroups, a TMA warp, an MMA warp
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ROLE_HH_PRODUCER = 15;
constexpr uint32_t ROLE_HH_MMA = 16;
constexpr uint32_t ROLE_HH_COMPUTE = 17;
constexpr uint32_t ROLE_HH_LAYOUT = 18;

constexpr uint32_t BOX = 128 * 128;                   // 128 rows x 128 bytes
constexpr uint32_t WBOX = 64 * 128;                   // 64 rows x 128 bytes
constexpr uint32_t SBOX = NV * 128;                   // 80 rows x 128 bytes
constexpr uint32_t OBOX = 32 * DV;                    // 32 rows x 64 bytes: one warp's O columns
constexpr uint32_t QK_OFF = 0;                        // Q, K boxes of the chunk Z is formed from next
constexpr uint32_t V_OFF = QK_OFF + 2 * BOX;          // V box of chunk c at + (c & 1) * BOX
constexpr uint32_t WQ_OFF = V_OFF + 2 * BOX;          // Wq [d][f]
constexpr uint32_t WK_OFF = WQ_OFF + WBOX;            // Wk [d][f]
constexpr uint32_t ONES_OFF = WK_OFF + WBOX;          // [row][col]: 1 in column 0
constexpr uint32_t PHIK_OFF = ONES_OFF + BOX;         // phi(K): 128 rows x 128 features (2 boxes)
constexpr uint32_t SPREV_OFF = PHIK_OFF + 2 * BOX;    // S (bf16, K-major): 80 rows x 128 features (2 boxes)
constexpr uint32_t OST_OFF = SPREV_OFF + 2 * SBOX;    // O staging: one 32 x 32 box per compute warp
constexpr uint32_t BAR_OFF = OST_OFF + 8 * OBOX;
constexpr int B_QKFULL = 0;        // Q, K of the next Z loaded
constexpr int B_QKEMPTY = 1;       // Z has read them
constexpr int B_VFULL = 2;         // + buffer (2)
constexpr int B_VEMPTY = 4;        // + buffer (2)
constexpr int B_WFULL = 6;         // Wq, Wk loaded
constexpr int B_ZFULL = 7;         // Q Wq, K Wk in TMEM
constexpr int B_PHIREADY = 8;      // phi(Q) in TMEM, phi(K) and the bf16 state of the chunks before in smem (8 warps)
constexpr int B_SFULL = 9;         // phi(Q) phi(K)^T in TMEM
constexpr int B_SREAD = 10;        // both groups hold their half of S in registers (8 warps)
constexpr int B_PREADY = 11;       // P in TMEM, the last O read out (8 warps)
constexpr int B_ODONE = 12;        // [num | den] of the chunk complete
constexpr int B_STDONE = 13;       // all products of the chunk done
constexpr int B_MMADONE = 14;
constexpr int NUM_BARS = 15;
constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
// The dynamic shared memory base is 1024-byte aligned (no static shared
// memory in this kernel); the kernel checks it and reports ROLE_HH_LAYOUT.
constexpr uint32_t SMEM_ALLOC = SMEM_USED;
static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");
static_assert(WQ_OFF % 1024 == 0 && ONES_OFF % 1024 == 0 && PHIK_OFF % 1024 == 0 && SPREV_OFF % 1024 == 0 &&
                  SBOX % 1024 == 0 &&
                  OST_OFF % 1024 == 0 && OBOX % 512 == 0,
              "swizzled boxes need 1024-byte (64-byte swizzle: 512-byte) alignment");

constexpr uint32_t T_Z = 0;        // Q Wq (cols 0..63), K Wk (64..127); then S
constexpr uint32_t T_O = 128;      // [num | den] fp32: 80 cols
constexpr uint32_t T_ST = 256;     // S^T fp32: 128 cols (lane = value column, 64 = the "1" row)
constexpr uint32_t T_P = 384;      // P (bf16, 64 cols): apart from S, so the next Z can be formed
                                   // as soon as S is read out
constexpr uint32_t T_PHIQ = 448;   // phi(Q) (bf16, 64 cols): the A operand of S and of the carried product

__device__ __forceinline__ uint32_t sw128(uint32_t box, int r, int c) { return box + r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ float fmin3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// phi(z) = [softmax(z), softmax(-z)] of one row's 64 projections (TMEM
// columns from `zcol`), as 64 packed bf16 pairs (zeros when `live` is false).
// The projections are read again for the second half, so that only one
// half's 64 exponentials are live at a time; pairs of columns go through the
// packed fp32 pipe.
__device__ __forceinline__ void phi_regs(uint32_t zcol, bool live, uint32_t (&pk)[64]) {
    constexpr float kLog2e = 1.4426950408889634f;
    uint32_t zr[64];
    tmem_ld64(zcol, zr);
    float zmax = __uint_as_float(zr[0]), zmin = zmax;
#pragma unroll
    for (int c = 1; c < FH; c += 2) {
        zmax = fmax3(zmax, __uint_as_float(zr[c]), __uint_as_float(zr[c + 1 < FH ? c + 1 : c]));
        zmin = fmin3(zmin, __uint_as_float(zr[c]), __uint_as_float(zr[c + 1 < FH ? c + 1 : c]));
    }
    // exp(z - zmax) = 2^(z log2e - zmax log2e); exp(zmin - z) = 2^(-z log2e + zmin log2e)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const float2 mul = half == 0 ? make_float2(kLog2e, kLog2e) : make_float2(-kLog2e, -kLog2e);
        const float off = half == 0 ? -zmax * kLog2e : zmin * kLog2e;
        const float2 add = make_float2(off, off);
        float2 e[FH / 2];
        float2 sum2 = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int part = 0; part < 2; ++part) {
            uint32_t zp[32];
            if (half == 1) tmem_ld32(zcol + part * 32, zp);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const int c = part * 32 + 2 * q;
                const float2 z2 = half == 0 ? make_float2(__uint_as_float(zr[c]), __uint_as_float(zr[c + 1]))
                                            : make_float2(__uint_as_float(zp[2 * q]), __uint_as_float(zp[2 * q + 1]));
                const float2 a = __ffma2_rn(z2, mul, add);
                e[c / 2] = make_float2(ex2(a.x), ex2(a.y));
                sum2 = __fadd2_rn(sum2, e[c / 2]);
            }
        }
        const float sc = live ? 1.0f / (sum2.x + sum2.y) : 0.0f;
        const float2 sc2 = make_float2(sc, sc);
#pragma unroll
        for (int q = 0; q < FH / 2; ++q) {
            const float2 v = __fmul2_rn(e[q], sc2);
            pk[half * 32 + q] = pack_bf16x2(v.x, v.y);
        }
    }
}

// Row r of a two-box 128-feature K-major tile from 64 packed bf16 pairs (phi(K));
// phi(Q) goes to TMEM instead.
__device__ __forceinline__ void phi_store(const uint32_t (&pk)[64], uint32_t tile, int r) {
#pragma unroll
    for (int half = 0; half < 2; ++half)
#pragma unroll
        for (int q = 0; q < 8; ++q)
            st_shared_v4(sw128(tile + half * BOX, r, q), pk[half * 32 + 4 * q], pk[half * 32 + 4 * q + 1],
                         pk[half * 32 + 4 * q + 2], pk[half * 32 + 4 * q + 3]);
}

__global__ void __launch_bounds__(NUM_THREADS, 1) hedgehog_kernel(const __grid_constant__ HedgehogParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    // A CTA walks one segment of a head: its chunks c0 .. c0 + n_chunks - 1
    // (the whole head unless the sequence is split into segments; then the
    // state of the chunks before c0 comes from the segment-state pass in
    // p.ws).  Chunk indices below are local to the segment.
    const int seg = blockIdx.x % p.n_seg;
    const int bh = blockIdx.x / p.n_seg;
    const int head = bh % p.H;
    const int c0 = seg * p.seg_chunks;
    const int n_chunks = min(p.seg_chunks, (p.N + C - 1) / C - c0);
    const bool has_prev = seg > 0;

    if (sbase & 1023u) {  // the swizzled layouts need it; uniform over the CTA, so every thread returns
        if (threadIdx.x == 0) record_timeout((ROLE_HH_LAYOUT << 24) | (sbase & 0xFFFFu));
        return;
    }
    if (warp == WARP_MMA) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(B_QKFULL), 1);
        mbar_init(bar(B_QKEMPTY), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_VFULL + b), 1);
            mbar_init(bar(B_VEMPTY + b), 1);
        }
        mbar_init(bar(B_WFULL), 1);
        mbar_init(bar(B_ZFULL), 1);
        mbar_init(bar(B_PHIREADY), 8);
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_SREAD), 8);
        mbar_init(bar(B_PREADY), 8);
        mbar_init(bar(B_ODONE), 1);
        mbar_init(bar(B_STDONE), 1);
        mbar_init(bar(B_MMADONE), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp < 4) {
        const int r = threadIdx.x;
        const uint32_t one = 0x3F80u;  // bf16 1.0 in the low half (column 0)
#pragma unroll
        for (int c = 0; c < 8; ++c) st_shared_v4(sw128(sbase + ONES_OFF, r, c), c == 0 ? one : 0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == WARP_TMA) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tmQ);
            tma_prefetch_desc(&p.tmK);
            tma_prefetch_desc(&p.tmV);
            tma_prefetch_desc(&p.tmWq);
            tma_prefetch_desc(&p.tmWk);
            mbar_arrive_expect_tx(bar(B_WFULL), 2 * WBOX);
            tma_load_3d(sbase + WQ_OFF, &p.tmWq, bar(B_WFULL), 0, 0, head);
            tma_load_3d(sbase + WK_OFF, &p.tmWk, bar(B_WFULL), 0, 0, head);
            // Q, K of chunk c into the single Q/K buffer once Z of chunk c-1 has
            // read it; V of chunk c into buffer c & 1 once chunk c-2's products have.
            int qk_issued = 0, v_issued = 0;
            bool ok = true;
            for (int c = 0; c < n_chunks; ++c) {
                const int b = c & 1;
                if (c >= 1 && !(ok = wait_bounded(bar(B_QKEMPTY), (c - 1) & 1, abort_flag,
                                                  (ROLE_HH_PRODUCER << 24) | (B_QKEMPTY << 16) | c)))
                    break;
                mbar_arrive_expect_tx(bar(B_QKFULL), 2 * BOX);
                tma_load_3d(sbase + QK_OFF, &p.tmQ, bar(B_QKFULL), 0, (c0 + c) * C, bh);
                tma_load_3d(sbase + QK_OFF + BOX, &p.tmK, bar(B_QKFULL), 0, (c0 + c) * C, bh);
                ++qk_issued;
                if (c >= 2 && !(ok = wait_bounded(bar(B_VEMPTY + b), ((c >> 1) - 1) & 1, abort_flag,
                                                  (ROLE_HH_PRODUCER << 24) | ((B_VEMPTY + b) << 16) | c)))
                    break;
                mbar_arrive_expect_tx(bar(B_VFULL + b), BOX);
                tma_load_3d(sbase + V_OFF + b * BOX, &p.tmV, bar(B_VFULL + b), 0, (c0 + c) * C, bh);
                ++v_issued;
            }
            if (!ok) {
                // let the loads in flight land before the CTA's shared memory goes away
                const uint64_t t0 = global_timer_ns();
                if (qk_issued > 0)
                    while (!mbar_try_wait(bar(B_QKFULL), (qk_issued - 1) & 1) && global_timer_ns() - t0 < kDrainLimitNs) {
                    }
                for (int j = v_issued - 2 < 0 ? 0 : v_issued - 2; j < v_issued; ++j)
                    while (!mbar_try_wait(bar(B_VFULL + (j & 1)), (j >> 1) & 1) &&
                           global_timer_ns() - t0 < kDrainLimitNs) {
                    }
                while (!mbar_try_wait(bar(B_WFULL), 0) && global_timer_ns() - t0 < kDrainLimitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the loop (operands stay warp-uniform); one
        // elected lane sends each block of products and each commit.
        {
            constexpr uint32_t ID_Z = idesc_bf16_f32(C, FH, 0, 1);       // X W: X K-major, W MN-major
            constexpr uint32_t ID_S = idesc_bf16_f32(C, C, 0, 0);        // phi(Q) phi(K)^T: A in TMEM
            constexpr uint32_t ID_INTRA = idesc_bf16_f32(C, NV, 0, 1);   // P [V | 1]: A in TMEM
            constexpr uint32_t ID_INTER = idesc_bf16_f32(C, NV, 0, 0);   // phi(Q) S: A in TMEM, B K-major
            constexpr uint32_t ID_STATE = idesc_bf16_f32(C, F, 1, 1);    // [V | 1]^T phi(K): both MN-major
            // Per chunk c, once both groups hold its S in registers: Q Wq and
            // K Wk of chunk c+1 (its feature maps are then formed while this
            // chunk's products run); once P is in TMEM: P [V|1], phi(Q) S_{<c},
            // the state update; once c+1's features are in place, phi(Q)
            // phi(K)^T of c+1.
            // Descriptors are formed once per operand; a k step adds its
            // compile-time offset to the start-address field (no carry:
            // shared memory is below 256 KB).
            const uint64_t qd = smem_desc_sw128(sbase + QK_OFF, 16, 1024), kd = smem_desc_sw128(sbase + QK_OFF + BOX, 16, 1024);
            const uint64_t wqd = smem_desc_sw128(sbase + WQ_OFF, WBOX, 1024), wkd = smem_desc_sw128(sbase + WK_OFF, WBOX, 1024);
            const uint64_t phikd = smem_desc_sw128(sbase + PHIK_OFF, 16, 1024), sprevd = smem_desc_sw128(sbase + SPREV_OFF, 16, 1024);
            const uint64_t phikmn = smem_desc_sw128(sbase + PHIK_OFF, BOX, 1024);
            const uint32_t hi = static_cast<uint32_t>(qd >> 32);  // every descriptor here has SBO 1024
            const uint32_t q_lo = static_cast<uint32_t>(qd), k_lo = static_cast<uint32_t>(kd);
            const uint32_t wq_lo = static_cast<uint32_t>(wqd), wk_lo = static_cast<uint32_t>(wkd);
            const uint32_t phik_lo = static_cast<uint32_t>(phikd), sprev_lo = static_cast<uint32_t>(sprevd);
            const uint32_t phikmn_lo = static_cast<uint32_t>(phikmn);
            auto issue_z = [&]() {  // Z = Q Wq, K Wk from the Q/K buffer, 16 of the 64 dims per step
                uint32_t qv[DQK / 16], kv[DQK / 16], wqv[DQK / 16], wkv[DQK / 16];
#pragma unroll
                for (int k = 0; k < DQK / 16; ++k) {
                    qv[k] = q_lo + ((k * 32) >> 4);
                    kv[k] = k_lo + ((k * 32) >> 4);
                    wqv[k] = wq_lo + ((k * 2048) >> 4);
                    wkv[k] = wk_lo + ((k * 2048) >> 4);
                }
                if (elect_one()) {
                    umma_ss_steps<DQK / 16>(tmem + T_Z, qv, hi, wqv, hi, ID_Z, 0u);
                    umma_ss_steps<DQK / 16>(tmem + T_Z + FH, kv, hi, wkv, hi, ID_Z, 0u);
                    umma_commit(bar(B_ZFULL));
                    umma_commit(bar(B_QKEMPTY));
                }
                __syncwarp();
            };
            auto issue_s = [&]() {  // S = phi(Q) phi(K)^T over the 128 features
                uint32_t phikv[F / 16];
#pragma unroll
                for (int k = 0; k < F / 16; ++k) phikv[k] = phik_lo + (((k / 4) * BOX + (k % 4) * 32) >> 4);
                if (elect_one()) {
                    umma_ts_steps<F / 16, 8>(tmem + T_Z, tmem + T_PHIQ, phikv, hi, ID_S, 0u);
                    umma_commit(bar(B_SFULL));
                }
                __syncwarp();
            };
            bool ok = wait_bounded(bar(B_WFULL), 0, abort_flag, (ROLE_HH_MMA << 24) | (B_WFULL << 16)) &&
                      wait_bounded(bar(B_QKFULL), 0, abort_flag, (ROLE_HH_MMA << 24) | (B_QKFULL << 16));
            if (ok) {
                tc_fence_after_sync();
                issue_z();
                if ((ok = wait_bounded(bar(B_PHIREADY), 0, abort_flag, (ROLE_HH_MMA << 24) | (B_PHIREADY << 16)))) {
                    tc_fence_after_sync();
                    issue_s();
                }
            }
            for (int c = 0; ok && c < n_chunks; ++c) {
                const int b = c & 1;
                const uint32_t ph = c & 1;
                const uint32_t vb = sbase + V_OFF + b * BOX;
                if (!(ok = wait_bounded(bar(B_SREAD), ph, abort_flag, (ROLE_HH_MMA << 24) | (B_SREAD << 16) | c)))
                    break;
                // Z of the next chunk over this chunk's S, which both groups have read out
                if (c + 1 < n_chunks) {
                    if (!(ok = wait_bounded(bar(B_QKFULL), (c + 1) & 1, abort_flag,
                                            (ROLE_HH_MMA << 24) | (B_QKFULL << 16) | (c + 1))))
                        break;
                    tc_fence_after_sync();
                    issue_z();
                }
                if (!(ok = wait_bounded(bar(B_PREADY), ph, abort_flag, (ROLE_HH_MMA << 24) | (B_PREADY << 16) | c)))
                    break;
                if (!(ok = wait_bounded(bar(B_VFULL + b), (c >> 1) & 1, abort_flag,
                                        (ROLE_HH_MMA << 24) | ((B_VFULL + b) << 16) | c)))
                    break;
                tc_fence_after_sync();
                // intra: [num | den] = P [V | 1]
                const uint32_t v1_lo = static_cast<uint32_t>(smem_desc_sw128(vb, ONES_OFF - (vb - sbase), 1024));
                uint32_t v1v[C / 16], pkv[C / 16], sprevv[F / 16];
#pragma unroll
                for (int k = 0; k < C / 16; ++k) {
                    v1v[k] = v1_lo + ((k * 2048) >> 4);
                    pkv[k] = phikmn_lo + ((k * 2048) >> 4);
                }
#pragma unroll
                for (int k = 0; k < F / 16; ++k) sprevv[k] = sprev_lo + (((k / 4) * SBOX + (k % 4) * 32) >> 4);
                if (elect_one()) {
                    umma_ts_steps<C / 16, 8>(tmem + T_O, tmem + T_P, v1v, hi, ID_INTRA, 0u);
                    // inter: [num | den] += phi(Q) S_{<c}
                    if (c > 0 || has_prev) umma_ts_steps<F / 16, 8>(tmem + T_O, tmem + T_PHIQ, sprevv, hi, ID_INTER, 1u);
                    umma_commit(bar(B_ODONE));
                    // state: S^T += [V | 1]^T phi(K)
                    umma_ss_steps<C / 16>(tmem + T_ST, v1v, hi, pkv, hi, ID_STATE, (c > 0 || has_prev) ? 1u : 0u);
                    umma_commit(bar(B_STDONE));
                    umma_commit(bar(B_VEMPTY + b));
                }
                __syncwarp();
                // S of the next chunk, once its features and this chunk's state are in smem
                if (c + 1 < n_chunks) {
                    if (!(ok = wait_bounded(bar(B_PHIREADY), ph ^ 1, abort_flag,
                                            (ROLE_HH_MMA << 24) | (B_PHIREADY << 16) | (c + 1))))
                        break;
                    tc_fence_after_sync();
                    issue_s();
                }
            }
            if (elect_one()) umma_commit(bar(B_MMADONE));
            __syncwarp();
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar(B_MMADONE), 0) && global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ compute warps
        // Two warpgroups over the same 128 rows (warp w reads TMEM lanes
        // 32 (w % 4) ..): group 0 forms phi(Q), the first half of P and of
        // the state copy, O columns 0..31 and DEN; group 1 forms phi(K) and
        // the second halves.  Per chunk c: S into registers (the tensor core
        // may then form Z of c+1) and P; chunk c+1's feature maps into
        // registers while chunk c's products run; once they are done, the
        // state copy and the feature maps into TMEM / smem (they feed c+1's
        // products); then O of chunk c through this warp's staging box and a
        // TMA store.
        const int i = threadIdx.x % 128;  // row of the chunk = TMEM lane; also row i of S^T
        const int grp = warp / 4;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
        const size_t head_row0 = static_cast<size_t>(bh) * p.N;
        const uint32_t zcol = lane_base + T_Z + grp * FH;
        // phi(Q) (group 0) into TMEM, phi(K) (group 1) into its smem tile
        auto put_phi = [&](const uint32_t (&pk)[64]) {
            if (grp == 0) {
                tmem_st32(lane_base + T_PHIQ, *reinterpret_cast<const uint32_t(*)[32]>(pk));
                tmem_st32(lane_base + T_PHIQ + 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32));
                tmem_st_wait();
            } else {
                phi_store(pk, sbase + PHIK_OFF, i);
            }
        };
        const uint32_t obox = sbase + OST_OFF + warp * OBOX;
        // bf16 copy of the state (rows 0..79 of S^T, this group's 64 features)
        // for the next chunk's carried product
        auto copy_state = [&]() {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t sv[32];
                tmem_ld32(lane_base + T_ST + grp * 64 + h2 * 32, sv);  // every lane loads; rows >= 80 are not stored
                if (i < NV) {
                    const uint32_t box = sbase + SPREV_OFF + grp * SBOX;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        st_shared_v4(sw128(box, i, h2 * 4 + q),
                                     pack_bf16x2(__uint_as_float(sv[8 * q]), __uint_as_float(sv[8 * q + 1])),
                                     pack_bf16x2(__uint_as_float(sv[8 * q + 2]), __uint_as_float(sv[8 * q + 3])),
                                     pack_bf16x2(__uint_as_float(sv[8 * q + 4]), __uint_as_float(sv[8 * q + 5])),
                                     pack_bf16x2(__uint_as_float(sv[8 * q + 6]), __uint_as_float(sv[8 * q + 7])));
                }
            }
        };
        if (has_prev) {
            // --- the state of the segments before this one: the sum of their fp32
            // partial states into the group's 64 columns of S^T (rows >= 65 are 0),
            // and its bf16 copy for the first chunk's carried product
            for (int blk = 0; blk < 64; blk += 16) {
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
                if (i < NV) {
                    for (int sp = 0; sp < seg; ++sp) {
                        const float4 *src = reinterpret_cast<const float4 *>(
                            p.ws + ((static_cast<size_t>(bh) * p.n_seg + sp) * NV + i) * F + grp * 64 + blk);
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 v = src[q];
                            acc[4 * q] += v.x;
                            acc[4 * q + 1] += v.y;
                            acc[4 * q + 2] += v.z;
                            acc[4 * q + 3] += v.w;
                        }
                    }
                }
                uint32_t u[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(acc[e]);
                tmem_st16(lane_base + T_ST + grp * 64 + blk, u);
            }
            tmem_st_wait();
            copy_state();
        }
        bool ok = wait_bounded(bar(B_ZFULL), 0, abort_flag, (ROLE_HH_COMPUTE << 24) | (B_ZFULL << 16));
        if (ok) {
            tc_fence_after_sync();
            uint32_t pk[64];
            phi_regs(zcol, grp == 0 || c0 * C + i < p.N, pk);  // phi(Q) always live; phi(K) zero past N
            put_phi(pk);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            warp_arrive(bar(B_PHIREADY), lane);
        }
        for (int c = 0; ok && c < n_chunks; ++c) {
            const uint32_t ph = c & 1;
            const int row = (c0 + c) * C + i;
            // --- this group's half of P = S under the causal mask (keys j <= i of the chunk and j < N)
            if (!(ok = wait_bounded(bar(B_SFULL), ph, abort_flag, (ROLE_HH_COMPUTE << 24) | (B_SFULL << 16) | c)))
                break;
            tc_fence_after_sync();
            {
                const int lim = p.N - 1 - (c0 + c) * C;  // last key of the chunk (j < N)
                const int jmax = min(i, lim);              // last key of the chunk this row sees
                // Per warp (rows r0 .. r0+31) and group (keys k0 .. k0+63): every key
                // hidden, every key seen, or a mix (the diagonal block, a ragged tail)
                const int r0 = (warp % 4) * 32, k0 = grp * 64;
                const int jlo = min(r0, lim), jhi = min(r0 + 31, lim);
                uint32_t pk[32];
                if (jhi < k0) {
                    tc_fence_before_sync();
                    warp_arrive(bar(B_SREAD), lane);
#pragma unroll
                    for (int e = 0; e < 32; ++e) pk[e] = 0u;
                } else {
                    uint32_t sr[64];
                    tmem_ld64(lane_base + T_Z + grp * 64, sr);
                    tc_fence_before_sync();
                    warp_arrive(bar(B_SREAD), lane);
                    if (jlo >= k0 + 63) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            pk[e] = pack_bf16x2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]));
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int j0 = k0 + 2 * e;
                            pk[e] = pack_bf16x2(j0 <= jmax ? __uint_as_float(sr[2 * e]) : 0.0f,
                                                j0 + 1 <= jmax ? __uint_as_float(sr[2 * e + 1]) : 0.0f);
                        }
                    }
                }
                tmem_st32(lane_base + T_P + grp * 32, pk);
            }
            tmem_st_wait();
            tc_fence_before_sync();
            warp_arrive(bar(B_PREADY), lane);
            if (c + 1 < n_chunks) {
                // --- chunk c+1's feature maps into registers (its Z follows this chunk's SREAD)
                if (!(ok = wait_bounded(bar(B_ZFULL), ph ^ 1, abort_flag,
                                        (ROLE_HH_COMPUTE << 24) | (B_ZFULL << 16) | (c + 1))))
                    break;
                tc_fence_after_sync();
                uint32_t pk[64];
                phi_regs(zcol, grp == 0 || row + C < p.N, pk);
                // --- chunk c's products done: the feature maps into TMEM / smem, then the state copy
                if (!(ok = wait_bounded(bar(B_STDONE), ph, abort_flag,
                                        (ROLE_HH_COMPUTE << 24) | (B_STDONE << 16) | c)))
                    break;
                tc_fence_after_sync();
                put_phi(pk);
                copy_state();
                fence_proxy_async_smem();
                tc_fence_before_sync();
                warp_arrive(bar(B_PHIREADY), lane);
            }
            // --- O_i = num_i / den_i, this group's 32 columns (read before the
            // group arrives on the next chunk's PREADY, after which the
            // tensor core overwrites them)
            if (!(ok = wait_bounded(bar(B_ODONE), ph, abort_flag, (ROLE_HH_COMPUTE << 24) | (B_ODONE << 16) | c)))
                break;
            tc_fence_after_sync();
            {
                uint32_t o[32], d[16];
                tmem_ld32(lane_base + T_O + grp * 32, o);
                tmem_ld16(lane_base + T_O + 64, d);
                const float den = __uint_as_float(d[0]);
                const float inv = 1.0f / den;
                const float2 inv2 = make_float2(inv, inv);
                // this warp's previous store has read its staging box
                if (lane == 0) tma_store_wait_read_all();
                __syncwarp();
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t w[4];
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        const float2 v = __fmul2_rn(
                            make_float2(__uint_as_float(o[8 * q + 2 * t]), __uint_as_float(o[8 * q + 2 * t + 1])), inv2);
                        w[t] = pack_bf16x2(v.x, v.y);
                    }
                    // 64-byte swizzle: 16-byte chunk q of row `lane` at chunk q ^ ((lane >> 1) & 3)
                    st_shared_v4(obox + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4), w[0], w[1], w[2], w[3]);
                }
                if (grp == 0 && row < p.N) p.DEN[head_row0 + row] = den;
                fence_proxy_async_smem();
                __syncwarp();
                const int row0 = (c0 + c) * C + (warp % 4) * 32;
                if (lane == 0 && row0 < p.N) {
                    tma_store_3d(&p.tmO, obox, grp * 32, row0, bh);  // rows past N are clipped
                    tma_store_commit();
                }
            }
        }
        if (lane == 0) tma_store_wait_all();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}


// ------------------------------------------------------------------ segment states
//
// For a head split into segments, each segment starts from the sum of the
// partial states of the segments before it.  This pass forms, per (head,
// segment) except the last, the partial state
//   dS^T = sum over the segment's rows of [v_j | 1] phi_k(k_j)^T   (fp32, 65 live rows x 128)
// with the main kernel's arithmetic (Z = K Wk on the tensor core, the same
// feature map, the same product), into ws[bh][seg].

// One half of phi(z) for one row: softmax(z) (half 0) or softmax(-z) (half 1)
// of the 64 projections at `zcol`, as 32 packed bf16 pairs, computed exactly
// as phi_regs computes that half.
__device__ __forceinline__ void phi_half(uint32_t zcol, bool live, int half, uint32_t (&pk)[32]) {
    constexpr float kLog2e = 1.4426950408889634f;
    uint32_t zr[64];
    tmem_ld64(zcol, zr);
    float zmax = __uint_as_float(zr[0]), zmin = zmax;
#pragma unroll
    for (int c = 1; c < FH; c += 2) {
        zmax = fmax3(zmax, __uint_as_float(zr[c]), __uint_as_float(zr[c + 1 < FH ? c + 1 : c]));
        zmin = fmin3(zmin, __uint_as_float(zr[c]), __uint_as_float(zr[c + 1 < FH ? c + 1 : c]));
    }
    const float2 mul = half == 0 ? make_float2(kLog2e, kLog2e) : make_float2(-kLog2e, -kLog2e);
    const float off = half == 0 ? -zmax * kLog2e : zmin * kLog2e;
    const float2 add = make_float2(off, off);
    float2 e[FH / 2];
    float2 sum2 = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int q = 0; q < FH / 2; ++q) {
        const float2 a = __ffma2_rn(make_float2(__uint_as_float(zr[2 * q]), __uint_as_float(zr[2 * q + 1])), mul, add);
        e[q] = make_float2(ex2(a.x), ex2(a.y));
        sum2 = __fadd2_rn(sum2, e[q]);
    }
    const float sc = live ? 1.0f / (sum2.x + sum2.y) : 0.0f;
    const float2 sc2 = make_float2(sc, sc);
#pragma unroll
    for (int q = 0; q < FH / 2; ++q) {
        const float2 v = __fmul2_rn(e[q], sc2);
        pk[q] = pack_bf16x2(v.x, v.y);
    }
}

namespace st {
constexpr uint32_t K_OFF = 0;                         // K box of chunk c at + (c & 1) * BOX
constexpr uint32_t V_OFF = K_OFF + 2 * BOX;           // V box likewise
constexpr uint32_t WK_OFF = V_OFF + 2 * BOX;          // Wk [d][f]
constexpr uint32_t ONES_OFF = WK_OFF + WBOX;
constexpr uint32_t PHIK_OFF = ONES_OFF + BOX;         // phi(K) of chunk c at + (c & 1) * 2 * BOX
constexpr uint32_t BAR_OFF = PHIK_OFF + 4 * BOX;
constexpr int B_FULL = 0;          // + buffer (2): K, V loaded
constexpr int B_FREE = 2;          // + buffer (2): the state product of the chunk in it is done
constexpr int B_ZFULL = 4;         // + buffer (2): K Wk in TMEM
constexpr int B_PHIKREADY = 6;     // + buffer (2): phi(K) in smem (8 warps)
constexpr int B_WFULL = 8;
constexpr int B_STDONE = 9;
constexpr int B_MMADONE = 10;
constexpr int NUM_BARS = 11;
constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t T_ZK = 0;       // K Wk of chunk c at + (c & 1) * 64
constexpr uint32_t T_STATE = 128;  // S^T fp32: 128 cols
static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");
static_assert(WK_OFF % 1024 == 0 && ONES_OFF % 1024 == 0 && PHIK_OFF % 1024 == 0, "swizzled boxes");
}  // namespace st

__global__ void __launch_bounds__(NUM_THREADS, 1) hedgehog_state_kernel(const __grid_constant__ HedgehogParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + st::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + st::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int seg = blockIdx.x % (p.n_seg - 1);   // every segment but the last
    const int bh = blockIdx.x / (p.n_seg - 1);
    const int head = bh % p.H;
    const int c0 = seg * p.seg_chunks;
    const int n_chunks = p.seg_chunks;

    if (warp == WARP_MMA) {
        tmem_alloc(smem_addr(tmem_slot), st::TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(st::B_FULL + b), 1);
            mbar_init(bar(st::B_FREE + b), 1);
            mbar_init(bar(st::B_ZFULL + b), 1);
            mbar_init(bar(st::B_PHIKREADY + b), 8);
        }
        mbar_init(bar(st::B_WFULL), 1);
        mbar_init(bar(st::B_STDONE), 1);
        mbar_init(bar(st::B_MMADONE), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp < 4) {
        const int r = threadIdx.x;
        const uint32_t one = 0x3F80u;  // bf16 1.0 in the low half (column 0)
#pragma unroll
        for (int c = 0; c < 8; ++c) st_shared_v4(sw128(sbase + st::ONES_OFF, r, c), c == 0 ? one : 0u, 0u, 0u, 0u);
        fence_proxy_async_smem();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == WARP_TMA) {
        if (lane == 0) {
            tma_prefetch_desc(&p.tmK);
            tma_prefetch_desc(&p.tmV);
            tma_prefetch_desc(&p.tmWk);
            mbar_arrive_expect_tx(bar(st::B_WFULL), WBOX);
            tma_load_3d(sbase + st::WK_OFF, &p.tmWk, bar(st::B_WFULL), 0, 0, head);
            int issued = 0;
            bool ok = true;
            for (int c = 0; c < n_chunks; ++c) {
                const int b = c & 1;
                if (c >= 2 && !(ok = wait_bounded(bar(st::B_FREE + b), ((c >> 1) - 1) & 1, abort_flag,
                                                  (ROLE_HH_PRODUCER << 24) | ((st::B_FREE + b) << 16) | c)))
                    break;
                mbar_arrive_expect_tx(bar(st::B_FULL + b), 2 * BOX);
                tma_load_3d(sbase + st::K_OFF + b * BOX, &p.tmK, bar(st::B_FULL + b), 0, (c0 + c) * C, bh);
                tma_load_3d(sbase + st::V_OFF + b * BOX, &p.tmV, bar(st::B_FULL + b), 0, (c0 + c) * C, bh);
                ++issued;
            }
            if (!ok) {
                const uint64_t t0 = global_timer_ns();
                for (int j = issued - 2 < 0 ? 0 : issued - 2; j < issued; ++j)
                    while (!mbar_try_wait(bar(st::B_FULL + (j & 1)), (j >> 1) & 1) && global_timer_ns() - t0 < kDrainLimitNs) {
                    }
                while (!mbar_try_wait(bar(st::B_WFULL), 0) && global_timer_ns() - t0 < kDrainLimitNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t ID_Z = idesc_bf16_f32(C, FH, 0, 1);      // K Wk: K K-major, W MN-major
            constexpr uint32_t ID_STATE = idesc_bf16_f32(C, F, 1, 1);   // [V | 1]^T phi(K): both MN-major
            auto issue_z = [&](int c) {
                const int b = c & 1;
                const uint32_t kb = sbase + st::K_OFF + b * BOX;
#pragma unroll
                for (int k = 0; k < DQK / 16; ++k)
                    umma_ss(tmem + st::T_ZK + b * FH, smem_desc_sw128(kb + k * 32, 16, 1024),
                            smem_desc_sw128(sbase + st::WK_OFF + k * 2048, WBOX, 1024), ID_Z, k > 0);
                umma_commit(bar(st::B_ZFULL + b));
            };
            bool ok = wait_bounded(bar(st::B_WFULL), 0, abort_flag, (ROLE_HH_MMA << 24) | (st::B_WFULL << 16));
            for (int c = 0; ok && c < 2 && c < n_chunks; ++c) {
                if (!(ok = wait_bounded(bar(st::B_FULL + c), 0, abort_flag, (ROLE_HH_MMA << 24) | ((st::B_FULL + c) << 16))))
                    break;
                tc_fence_after_sync();
                issue_z(c);
            }
            for (int c = 0; ok && c < n_chunks; ++c) {
                const int b = c & 1;
                const uint32_t vb = sbase + st::V_OFF + b * BOX;
                if (!(ok = wait_bounded(bar(st::B_PHIKREADY + b), (c >> 1) & 1, abort_flag,
                                        (ROLE_HH_MMA << 24) | ((st::B_PHIKREADY + b) << 16) | c)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    umma_ss(tmem + st::T_STATE, smem_desc_sw128(vb + k * 2048, st::ONES_OFF - (vb - sbase), 1024),
                            smem_desc_sw128(sbase + st::PHIK_OFF + b * 2 * BOX + k * 2048, BOX, 1024), ID_STATE,
                            (c > 0 || k > 0) ? 1u : 0u);
                umma_commit(bar(st::B_FREE + b));
                // Z of chunk c+2 into this buffer: its K is loaded once this chunk's products are done,
                // and the compute warps read this chunk's Z before they handed over phi(K)
                if (c + 2 < n_chunks) {
                    if (!(ok = wait_bounded(bar(st::B_FULL + b), ((c + 2) >> 1) & 1, abort_flag,
                                            (ROLE_HH_MMA << 24) | ((st::B_FULL + b) << 16) | (c + 2))))
                        break;
                    tc_fence_after_sync();
                    issue_z(c + 2);
                }
            }
            if (ok) umma_commit(bar(st::B_STDONE));
            umma_commit(bar(st::B_MMADONE));
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar(st::B_MMADONE), 0) && global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
            }
        }
        __syncwarp();
    } else {
        // group 0 forms softmax(z), group 1 softmax(-z) of K Wk, each into its box of phi(K)
        const int i = threadIdx.x % 128;
        const int grp = warp / 4;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
        bool ok = true;
        for (int c = 0; c < n_chunks; ++c) {
            const int b = c & 1;
            if (!(ok = wait_bounded(bar(st::B_ZFULL + b), (c >> 1) & 1, abort_flag,
                                    (ROLE_HH_COMPUTE << 24) | ((st::B_ZFULL + b) << 16) | c)))
                break;
            tc_fence_after_sync();
            uint32_t pk[32];
            phi_half(lane_base + st::T_ZK + b * FH, (c0 + c) * C + i < p.N, grp, pk);
            if (c >= 2 && !(ok = wait_bounded(bar(st::B_FREE + b), ((c >> 1) - 1) & 1, abort_flag,
                                              (ROLE_HH_COMPUTE << 24) | ((st::B_FREE + b) << 16) | c)))
                break;
            const uint32_t box = sbase + st::PHIK_OFF + b * 2 * BOX + grp * BOX;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                st_shared_v4(sw128(box, i, q), pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            warp_arrive(bar(st::B_PHIKREADY + b), lane);
        }
        if (ok && wait_bounded(bar(st::B_STDONE), 0, abort_flag, (ROLE_HH_COMPUTE << 24) | (st::B_STDONE << 16))) {
            tc_fence_after_sync();
            float *dst = p.ws + ((static_cast<size_t>(bh) * p.n_seg + seg) * NV + i) * F + grp * 64;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                uint32_t v[32];
                tmem_ld32(lane_base + st::T_STATE + grp * 64 + h2 * 32, v);  // every lane loads; rows >= 80 are not stored
                if (i < NV) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst + h2 * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        d4[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                            __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, st::TMEM_COLS);
    }
}

}  // namespace hedgehog

cudaError_t launch_hedgehog(const HedgehogParams &p, cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        if ((err = cudaFuncSetAttribute(hedgehog::hedgehog_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        hedgehog::SMEM_ALLOC)) != cudaSuccess)
            return err;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.BH * p.n_seg), 1, 1);
    cfg.blockDim = dim3(hedgehog::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = hedgehog::SMEM_ALLOC;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, hedgehog::hedgehog_kernel, p);
}

// The segment-state pass (n_seg > 1): one CTA per (head, segment) but the last.
cudaError_t launch_hedgehog_states(const HedgehogParams &p, cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        if ((err = cudaFuncSetAttribute(hedgehog::hedgehog_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        hedgehog::st::SMEM_ALLOC)) != cudaSuccess)
            return err;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.BH * (p.n_seg - 1)), 1, 1);
    cfg.blockDim = dim3(hedgehog::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = hedgehog::st::SMEM_ALLOC;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, hedgehog::hedgehog_state_kernel, p);
}

cudaError_t read_and_clear_hedgehog_status(uint32_t *status, uint32_t *detail) {
    unsigned int vals[2] = {0, 0};
    cudaError_t err = cudaMemcpyFromSymbol(&vals[0], g_status, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(&vals[1], g_detail, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero[1] = {0};
    if ((err = cudaMemcpyToSymbol(g_status, zero, sizeof(unsigned int))) != cudaSuccess) return err;
    if ((err = cudaMemcpyToSymbol(g_detail, zero, sizeof(unsigned int))) != cudaSuccess) return err;
    *status = vals[0];
    *detail = vals[1];
    return cudaSuccess;
}

}  // namespace tk
