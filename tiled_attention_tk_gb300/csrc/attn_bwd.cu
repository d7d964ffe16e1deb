// attn_bwd.cu -- attention backward for sm_103a (GB300).
//
// Gradients of L = sum(O * dO) for O = softmax(scale * Q K^T [+ causal]) V,
// using the forward's saved row log-sum-exp to recompute the weights:
//
//   P_ij  = exp(scale <Q_i, K_j> - LSE_i)          (0 for masked keys)
//   Delta_i = <dO_i, O_i>                           (= sum_j P_ij dP_ij)
//   dP_ij = <dO_i, V_j>
//   dS_ij = scale * P_ij (dP_ij - Delta_i)
//   dV_j  = sum_i P_ij dO_i,  dK_j = sum_i dS_ij Q_i,  dQ_i = sum_j dS_ij K_j
//
// The pages list attention backwards among the kernels built with the same
// tiles (groovesquid.com summary of the ThunderKittens paper); this is the
// standard chain rule through the online-softmax forward, written for the
// tcgen05 tensor cores.
//
// Three kernels on the caller's stream:
//   bwd_prep_kernel    Delta_i = <dO_i, O_i> (fp32) and a zeroed fp32 dQ
//                      accumulator, one warp per row.
//   attn_bwd_kernel<D> one CTA per (head, 128-key tile).  K_j and V_j stay in
//                      shared memory; for every 128-row query tile that sees
//                      the keys, the MMA warp forms S = Q K^T and dP = dO V^T
//                      in TMEM, four compute warps turn them into P and dS
//                      (bf16, written to 128-byte-swizzled shared memory),
//                      and the MMA warp accumulates dV += P^T dO and
//                      dK += dS^T Q in TMEM and forms dQ_part = dS K, which
//                      the compute warps add into the fp32 dQ accumulator
//                      (vector reductions).  At the end dK and dV are written
//                      as bf16.
//   bwd_dq_kernel      dQ = bf16(accumulator).
// The same shared-memory tiles serve as K-major and MN-major MMA operands
// through different descriptors (e.g. P for dV as P^T, dS as both).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "tk_attn.h"
#include "tk_attn_internal.h"
#include "tk_ptx.cuh"
#include "tk_sync.cuh"

namespace tk {

namespace bwd {

constexpr int BT = 128;             // rows per query tile and per key tile
constexpr int NUM_THREADS = 192;    // 4 compute warps, TMA warp, MMA warp
constexpr int WARP_TMA = 4;
constexpr int WARP_MMA = 5;
constexpr uint32_t TMEM_COLS = 512;

template <int D>
struct Layout {
    static constexpr int KATOMS = D / 64;
    static constexpr uint32_t BOX = 128 * 64 * 2;        // one 128-row x 64-column bf16 box
    static constexpr uint32_t TILE = BT * D * 2;         // a 128 x D tile
    static constexpr uint32_t K_OFF = 0;
    static constexpr uint32_t V_OFF = K_OFF + TILE;
    static constexpr uint32_t Q_OFF = V_OFF + TILE;
    static constexpr uint32_t DO_OFF = Q_OFF + TILE;
    static constexpr uint32_t P_OFF = DO_OFF + TILE;      // 128 queries x 128 keys bf16 (2 boxes)
    static constexpr uint32_t DS_OFF = P_OFF + 2 * BOX;
    static constexpr uint32_t BAR_OFF = DS_OFF + 2 * BOX;
    static constexpr int B_KVFULL = 0;
    static constexpr int B_QFULL = 1;
    static constexpr int B_SFULL = 2;      // S and dP in TMEM (MMA commit)
    static constexpr int B_PREADY = 3;     // P and dS in shared memory (compute warps, 4)
    static constexpr int B_GDONE = 4;      // dV, dK, dQ_part MMAs done (MMA commit)
    static constexpr int B_DQREAD = 5;     // dQ_part read out of TMEM (compute warps, 4)
    static constexpr int B_MMADONE = 6;
    static constexpr int NUM_BARS = 7;
    static constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
    static constexpr uint32_t SMEM_ALLOC =
        SMEM_USED + 1024 > 116u * 1024u ? SMEM_USED + 1024 : 116u * 1024u;  // one CTA per SM
    static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");
    // TMEM columns
    static constexpr uint32_t T_S = 0;           // S, then dQ_part (D columns)
    static constexpr uint32_t T_DP = 128;        // dP
    static constexpr uint32_t T_DV = 256;        // dV accumulator (D columns)
    static constexpr uint32_t T_DK = 256 + D;    // dK accumulator (D columns)
};

// Adds four floats to global memory with one vector reduction.
__device__ __forceinline__ void red_add_v4(float *addr, float a, float b, float c, float d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// Shared-memory address of 16-byte chunk `c` (0..7) of row `r` in a
// 128-byte-swizzled box (the layout TMA writes with the 128-byte swizzle).
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t box, int r, int c) {
    return box + r * 128 + ((c ^ (r & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
    using L = Layout<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + L::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    // Work: key tile kt of head bh; key tile 0 first (it sees the most query
    // tiles under the causal mask).
    const int kt = blockIdx.x / p.BH;
    const int bh = blockIdx.x % p.BH;
    const int qt_first = p.causal ? kt : 0;
    const int n_q = p.n_tiles - qt_first;

    if (warp == WARP_MMA) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(L::B_KVFULL), 1);
        mbar_init(bar(L::B_QFULL), 1);
        mbar_init(bar(L::B_SFULL), 1);
        mbar_init(bar(L::B_PREADY), 4);
        mbar_init(bar(L::B_GDONE), 1);
        mbar_init(bar(L::B_DQREAD), 4);
        mbar_init(bar(L::B_MMADONE), 1);
        *abort_flag = 0;
        fence_barrier_init();
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
            tma_prefetch_desc(&p.tmDO);
            mbar_arrive_expect_tx(bar(L::B_KVFULL), 2 * L::TILE);
            for (int c = 0; c < L::KATOMS; ++c) {
                tma_load_3d(sbase + L::K_OFF + c * L::BOX, &p.tmK, bar(L::B_KVFULL), c * 64, kt * BT, bh);
                tma_load_3d(sbase + L::V_OFF + c * L::BOX, &p.tmV, bar(L::B_KVFULL), c * 64, kt * BT, bh);
            }
            int issued = 0;
            for (int it = 0; it < n_q; ++it) {
                // Q, dO, P and dS of the previous query tile are free once its
                // gradient MMAs have completed.
                if (it > 0 && !wait_bounded(bar(L::B_GDONE), (it - 1) & 1, abort_flag,
                                            (ROLE_BWD_PRODUCER << 24) | (L::B_GDONE << 16) | it)) {
                    // Let the copies in flight land before the CTA exits.
                    const uint64_t t0 = global_timer_ns();
                    while (!(mbar_try_wait(bar(L::B_KVFULL), 0) && mbar_try_wait(bar(L::B_QFULL), (issued - 1) & 1)) &&
                           global_timer_ns() - t0 < kDrainLimitNs) {
                    }
                    break;
                }
                ++issued;
                const int qt = qt_first + it;
                mbar_arrive_expect_tx(bar(L::B_QFULL), 2 * L::TILE);
                for (int c = 0; c < L::KATOMS; ++c) {
                    tma_load_3d(sbase + L::Q_OFF + c * L::BOX, &p.tmQ, bar(L::B_QFULL), c * 64, qt * BT, bh);
                    tma_load_3d(sbase + L::DO_OFF + c * L::BOX, &p.tmDO, bar(L::B_QFULL), c * 64, qt * BT, bh);
                }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_KK = idesc_bf16_f32(BT, BT, 0, 0);  // S, dP: K-major A and B
            constexpr uint32_t IDESC_MM = idesc_bf16_f32(BT, D, 1, 1);   // dV, dK: MN-major A and B
            constexpr uint32_t IDESC_KM = idesc_bf16_f32(BT, D, 0, 1);   // dQ: K-major A, MN-major B
            bool ok = wait_bounded(bar(L::B_KVFULL), 0, abort_flag, (ROLE_BWD_MMA << 24) | (L::B_KVFULL << 16));
            for (int it = 0; ok && it < n_q; ++it) {
                if (!(ok = wait_bounded(bar(L::B_QFULL), it & 1, abort_flag,
                                        (ROLE_BWD_MMA << 24) | (L::B_QFULL << 16) | it)))
                    break;
                // S / dQ_part columns are free once the previous dQ_part was read.
                if (it > 0 && !(ok = wait_bounded(bar(L::B_DQREAD), (it - 1) & 1, abort_flag,
                                                  (ROLE_BWD_MMA << 24) | (L::B_DQREAD << 16) | it)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k / 4) * L::BOX + (k % 4) * 32;
                    umma_ss(tmem + L::T_S, smem_desc_sw128(sbase + L::Q_OFF + off, 16, 1024),
                            smem_desc_sw128(sbase + L::K_OFF + off, 16, 1024), IDESC_KK, k > 0);
                    umma_ss(tmem + L::T_DP, smem_desc_sw128(sbase + L::DO_OFF + off, 16, 1024),
                            smem_desc_sw128(sbase + L::V_OFF + off, 16, 1024), IDESC_KK, k > 0);
                }
                umma_commit(bar(L::B_SFULL));
                if (!(ok = wait_bounded(bar(L::B_PREADY), it & 1, abort_flag,
                                        (ROLE_BWD_MMA << 24) | (L::B_PREADY << 16) | it)))
                    break;
                tc_fence_after_sync();
                // 16 queries per step: P / dS (MN-major, rows = queries) and
                // dO / Q (MN-major, rows = queries) advance by 16 rows.
#pragma unroll
                for (int k = 0; k < BT / 16; ++k) {
                    const uint32_t roff = k * 2048;
                    const uint32_t acc = (it > 0 || k > 0) ? 1u : 0u;
                    umma_ss(tmem + L::T_DV, smem_desc_sw128(sbase + L::P_OFF + roff, L::BOX, 1024),
                            smem_desc_sw128(sbase + L::DO_OFF + roff, L::BOX, 1024), IDESC_MM, acc);
                    umma_ss(tmem + L::T_DK, smem_desc_sw128(sbase + L::DS_OFF + roff, L::BOX, 1024),
                            smem_desc_sw128(sbase + L::Q_OFF + roff, L::BOX, 1024), IDESC_MM, acc);
                }
                // dQ_part = dS K: 16 keys per step; dS K-major, K MN-major.
#pragma unroll
                for (int k = 0; k < BT / 16; ++k) {
                    const uint32_t aoff = (k / 4) * L::BOX + (k % 4) * 32;
                    umma_ss(tmem + L::T_S, smem_desc_sw128(sbase + L::DS_OFF + aoff, 16, 1024),
                            smem_desc_sw128(sbase + L::K_OFF + k * 2048, L::BOX, 1024), IDESC_KM, k > 0);
                }
                umma_commit(bar(L::B_GDONE));
            }
            umma_commit(bar(L::B_MMADONE));
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar(L::B_MMADONE), 0) &&
                   global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ compute warps: P, dS, dQ reduction
        const int t = threadIdx.x;  // row of the query tile == TMEM lane (S, dP, dQ_part),
                                    // row of the key tile for dK, dV
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const float c = p.scale_log2e;
        const size_t head_rows = static_cast<size_t>(bh) * p.N;
        bool ok = true;
        for (int it = 0; it < n_q; ++it) {
            const int qt = qt_first + it;
            const int row = qt * BT + t;
            const bool valid_row = row < p.N;
            // Rows past N: P = exp2(-inf) = 0 and Delta = 0, so they add nothing.
            const float lse2 = valid_row ? p.LSE[head_rows + row] * 1.4426950408889634f : INFINITY;
            const float delta = valid_row ? p.delta[head_rows + row] : 0.0f;
            // keys the row may see in this key tile: [0, kmax)
            int kmax = p.N - kt * BT;
            if (p.causal) kmax = min(kmax, row - kt * BT + 1);
            if (!(ok = wait_bounded(bar(L::B_SFULL), it & 1, abort_flag,
                                    (ROLE_BWD_COMPUTE << 24) | (L::B_SFULL << 16) | it)))
                break;
            tc_fence_after_sync();
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // 32 keys at a time
                uint32_t sr[32], dr[32];
                tmem_ld32(lane_base + L::T_S + q * 32, sr);
                tmem_ld32(lane_base + L::T_DP + q * 32, dr);
                uint32_t pp[16], ds[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    float pv[2], dv[2];
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int key = q * 32 + 2 * e + h;
                        const float x = fmaf(__uint_as_float(sr[2 * e + h]), c, -lse2);
                        pv[h] = key < kmax ? ex2(x) : 0.0f;
                        dv[h] = p.scale * pv[h] * (__uint_as_float(dr[2 * e + h]) - delta);
                    }
                    pp[e] = pack_bf16x2(pv[0], pv[1]);
                    ds[e] = pack_bf16x2(dv[0], dv[1]);
                }
                // keys q*32 .. q*32+31 = chunks 4(q%2) .. 4(q%2)+3 of box q/2, row t
                const uint32_t pbox = sbase + L::P_OFF + (q / 2) * L::BOX;
                const uint32_t dbox = sbase + L::DS_OFF + (q / 2) * L::BOX;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const int chunk = (q % 2) * 4 + v;
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw128_chunk(pbox, t, chunk)),
                                 "r"(pp[4 * v]), "r"(pp[4 * v + 1]), "r"(pp[4 * v + 2]), "r"(pp[4 * v + 3])
                                 : "memory");
                    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(sw128_chunk(dbox, t, chunk)),
                                 "r"(ds[4 * v]), "r"(ds[4 * v + 1]), "r"(ds[4 * v + 2]), "r"(ds[4 * v + 3])
                                 : "memory");
                }
            }
            fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
            tc_fence_before_sync();
            warp_arrive(bar(L::B_PREADY), lane);
            if (!(ok = wait_bounded(bar(L::B_GDONE), it & 1, abort_flag,
                                    (ROLE_BWD_COMPUTE << 24) | (L::B_GDONE << 16) | it)))
                break;
            tc_fence_after_sync();
            float *dq = p.dq_acc + (head_rows + (valid_row ? row : 0)) * D;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t r[32];
                tmem_ld32(lane_base + L::T_S + q * 32, r);
                if (valid_row) {
#pragma unroll
                    for (int v = 0; v < 8; ++v)
                        red_add_v4(dq + q * 32 + 4 * v, __uint_as_float(r[4 * v]), __uint_as_float(r[4 * v + 1]),
                                   __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3]));
                }
            }
            tc_fence_before_sync();
            warp_arrive(bar(L::B_DQREAD), lane);
        }
        if (ok) {
            // dK, dV of this key tile: TMEM lane t = key kt*128 + t.  The last
            // GDONE wait above covers every gradient MMA.
            const int key = kt * BT + t;
            const bool store = key < p.N;
            __nv_bfloat16 *dkrow = static_cast<__nv_bfloat16 *>(p.dK) + (head_rows + (store ? key : 0)) * D;
            __nv_bfloat16 *dvrow = static_cast<__nv_bfloat16 *>(p.dV) + (head_rows + (store ? key : 0)) * D;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                // every lane takes part in the TMEM loads; only the stores are guarded
                uint32_t rk[32], rv[32];
                tmem_ld32(lane_base + L::T_DK + q * 32, rk);
                tmem_ld32(lane_base + L::T_DV + q * 32, rv);
                if (store) {
                    uint32_t pk[16], pv[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        pk[e] = pack_bf16x2(__uint_as_float(rk[2 * e]), __uint_as_float(rk[2 * e + 1]));
                        pv[e] = pack_bf16x2(__uint_as_float(rv[2 * e]), __uint_as_float(rv[2 * e + 1]));
                    }
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        reinterpret_cast<uint4 *>(dkrow + q * 32)[v] =
                            make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                        reinterpret_cast<uint4 *>(dvrow + q * 32)[v] =
                            make_uint4(pv[4 * v], pv[4 * v + 1], pv[4 * v + 2], pv[4 * v + 3]);
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Delta_i = <dO_i, O_i> in fp32 and a zeroed fp32 dQ accumulator row; one
// warp per row, rows = B*H*N.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ O,
                                                      const __nv_bfloat16 *__restrict__ dO,
                                                      float *__restrict__ delta, float *__restrict__ dq_acc,
                                                      int64_t rows) {
    const int64_t row = static_cast<int64_t>(blockIdx.x) * 8 + threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    if (row >= rows) return;
    constexpr int PER = D / 32;  // elements per lane: 4 (D=128) or 2 (D=64)
    const __nv_bfloat16 *o = O + row * D + lane * PER;
    const __nv_bfloat16 *g = dO + row * D + lane * PER;
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < PER; ++e) s = fmaf(__bfloat162float(o[e]), __bfloat162float(g[e]), s);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
    if (lane == 0) delta[row] = s;
    float *acc = dq_acc + row * D + lane * PER;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.0f;
}

// dQ = bf16(dq_acc), eight elements per thread.
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dQ,
                                                     int64_t n8) {
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const float4 a = reinterpret_cast<const float4 *>(dq_acc)[2 * i];
        const float4 b = reinterpret_cast<const float4 *>(dq_acc)[2 * i + 1];
        reinterpret_cast<uint4 *>(dQ)[i] =
            make_uint4(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w), pack_bf16x2(b.x, b.y), pack_bf16x2(b.z, b.w));
    }
}

template <int D>
static cudaError_t launch_d(const BwdParams &p, int num_sms, cudaStream_t stream) {
    using L = Layout<D>;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        err = cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_ALLOC);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    const int64_t rows = static_cast<int64_t>(p.BH) * p.N;
    bwd_prep_kernel<D><<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(p.O), static_cast<const __nv_bfloat16 *>(p.dO), p.delta, p.dq_acc, rows);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(p.n_tiles) * p.BH), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_ALLOC;
    cfg.stream = stream;
    if ((err = cudaLaunchKernelEx(&cfg, attn_bwd_kernel<D>, p)) != cudaSuccess) return err;

    const int64_t n8 = rows * D / 8;
    int64_t blocks = (n8 + 255) / 256;
    if (blocks > 8LL * num_sms) blocks = 8LL * num_sms;
    bwd_dq_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p.dq_acc, static_cast<__nv_bfloat16 *>(p.dQ), n8);
    return cudaGetLastError();
}

}  // namespace bwd

cudaError_t launch_attn_bwd(int D, const BwdParams &p, int num_sms, cudaStream_t stream) {
    if (num_sms < 1) return cudaErrorInvalidValue;
    if (D == 64) return bwd::launch_d<64>(p, num_sms, stream);
    if (D == 128) return bwd::launch_d<128>(p, num_sms, stream);
    return cudaErrorInvalidValue;
}

// ------------------------------------------------------------------ fixed workspace
// A workspace that lives in the library itself, for tk_attn_bwd_noalloc:
// callers that cannot allocate device memory still get a backward pass for
// problems whose workspace fits.  Every device that loads the library holds
// this array until the process exits; every call on a device shares it.
static __device__ __align__(256) unsigned char g_noalloc_workspace[kNoAllocWorkspaceBytes];

// The device address of the array on the current device.  Host code cannot
// use the symbol itself (on the host it names a host-side stand-in), so the
// address is looked up once per device, with that device current, and
// cached.
cudaError_t noalloc_workspace(void **ptr) {
    static std::mutex mu;
    static void *cached[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cached[dev]) {
        void *addr = nullptr;
        err = cudaGetSymbolAddress(&addr, g_noalloc_workspace);
        if (err != cudaSuccess) return err;
        cached[dev] = addr;
    }
    *ptr = cached[dev];
    return cudaSuccess;
}

cudaError_t read_and_clear_bwd_status(uint32_t *status, uint32_t *detail) {
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
