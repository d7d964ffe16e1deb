// attn_fwd.cu -- fused attention forward for sm_103a (GB300).
//
// Computes, per (batch, head), O = softmax(scale * Q K^T [+ causal mask]) V
// and the natural-log row LSE, with the online softmax of the
// "ThunderKittens" attention kernel (10100.com/article/71410160, section
// "writing a kernel with TK", attn_fwd_template: consumer::compute keeps a
// running row max m and row sum l in the exp2 domain, with scale*log2(e)
// folded into one factor, rescales the partial output by exp2(c*(m_old -
// m_new)) before adding P V, and rounds P to bf16 for the second
// contraction; consumer::finish divides by l once) and the -inf fill of the
// ragged key tail from alanwu.xyz/posts/thunderkittens (attention inner loop).
//
// The Hopper design on that page (three consumer warpgroups of 64-row Q
// tiles, register accumulators, wgmma, two pipeline stages) is replaced by
// the Blackwell one:
//   warp 4      TMA producer: Q once, then K/V tiles through a STAGES-deep
//               shared-memory ring (full/empty mbarriers).
//   warp 5      MMA issuer: S = Q K^T (tcgen05.mma, smem x smem -> TMEM fp32)
//               into one of two S buffers, O += P V (P read from TMEM, V from
//               smem) into the O accumulator in TMEM.  Also owns TMEM.
//   warps 0-3   softmax + correction + epilogue: thread t owns query row t of
//               the 128-row tile (TMEM lane t); reads its S row with
//               tcgen05.ld, masks, updates m and l, writes P as bf16 over the
//               S columns, rescales its O row in TMEM, and at the end writes
//               O / l (bf16) and LSE.
// One CTA handles one 128-row Q tile of one head; CTAs are ordered heaviest
// (causal) tile first.
//
// Every wait on an mbarrier is bounded in time: if it gives up, the CTA
// records TK_ERR_DEVICE_TIMEOUT in a device status word, lets in-flight
// copies and MMAs drain (again bounded), frees its TMEM and returns.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tk_attn.h"
#include "tk_attn_internal.h"
#include "tk_ptx.cuh"

namespace tk {

// ------------------------------------------------------------------ status

__device__ unsigned int g_status;  // 0 or TK_ERR_DEVICE_TIMEOUT
__device__ unsigned int g_detail;  // where the first wait gave up

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s: far above any legitimate wait
constexpr uint64_t kDrainLimitNs = 50000000ull;   // 50 ms for draining after an abort

enum : uint32_t { ROLE_PRODUCER = 1, ROLE_MMA = 2, ROLE_SOFTMAX = 3, ROLE_SELFTEST = 4 };

__device__ __forceinline__ void record_timeout(uint32_t where) {
    if (atomicCAS(&g_status, 0u, (unsigned)TK_ERR_DEVICE_TIMEOUT) == 0u) atomicExch(&g_detail, where);
}

// Waits for the phase `parity` of `bar`.  Returns false (and raises the
// CTA's abort flag) if the wait exceeds `limit_ns`, or if another thread of
// the CTA has raised the abort flag.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                             uint32_t where, uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((spin & 63u) == 0u) {
            if (*abort_flag) return false;
            if (global_timer_ns() - t0 > limit_ns || spin > 0x7FFFFFF0u) {
                *abort_flag = 1;
                record_timeout(where);
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ layout

constexpr int BM = 128;          // query rows per tile (one TMEM lane each)
constexpr int BN = 128;          // keys per tile
constexpr int NUM_THREADS = 192; // 4 softmax warps + TMA warp + MMA warp
constexpr int WARP_TMA = 4;
constexpr int WARP_MMA = 5;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t TMEM_S0 = 0;    // S / P buffer 0: 128 fp32 columns
constexpr uint32_t TMEM_S1 = 128;  // S / P buffer 1
constexpr uint32_t TMEM_O = 256;   // O accumulator: D fp32 columns

template <int D>
struct Layout {
    static constexpr int KATOMS = D / 64;                 // 128-byte swizzle atoms along D
    static constexpr int STAGES = 2;                      // K/V ring depth
    static constexpr uint32_t BOX_BYTES = 128 * 64 * 2;   // one TMA box: 128 rows x 64 bf16
    static constexpr uint32_t TILE_BYTES = BM * D * 2;    // one 128-row tile
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t KV_OFF = TILE_BYTES;        // stage s: K, then V
    static constexpr uint32_t STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr uint32_t BAR_OFF = KV_OFF + STAGES * STAGE_BYTES;
    // barriers
    static constexpr int B_QFULL = 0;
    static constexpr int B_KVFULL = 1;                    // + stage
    static constexpr int B_KVEMPTY = B_KVFULL + STAGES;   // + stage
    static constexpr int B_SFULL = B_KVEMPTY + STAGES;    // + buffer (2)
    static constexpr int B_PFULL = B_SFULL + 2;
    static constexpr int B_ODONE = B_PFULL + 1;
    static constexpr int B_MMADONE = B_ODONE + 1;
    static constexpr int NUM_BARS = B_MMADONE + 1;
    static constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
    // +1024: slack for 1024-byte alignment.  At least 116 KB so that only one
    // CTA is resident per SM: each CTA allocates all 512 TMEM columns.
    static constexpr uint32_t SMEM_ALLOC =
        SMEM_USED + 1024 > 116u * 1024u ? SMEM_USED + 1024 : 116u * 1024u;
};

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
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

    // Work unit: heaviest query tiles first (matters under the causal mask),
    // consecutive CTAs on different heads.
    const int rank = blockIdx.x / p.BH;
    const int bh = blockIdx.x % p.BH;
    const int qt = p.n_qtiles - 1 - rank;
    const int n_kv = p.causal ? min(qt + 1, p.n_kvtiles) : p.n_kvtiles;

    if (warp == WARP_MMA) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(L::B_QFULL), 1);
        for (int s = 0; s < L::STAGES; ++s) {
            mbar_init(bar(L::B_KVFULL + s), 1);
            mbar_init(bar(L::B_KVEMPTY + s), 1);
        }
        mbar_init(bar(L::B_SFULL + 0), 1);
        mbar_init(bar(L::B_SFULL + 1), 1);
        mbar_init(bar(L::B_PFULL), BM);
        mbar_init(bar(L::B_ODONE), 1);
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
            mbar_arrive_expect_tx(bar(L::B_QFULL), L::TILE_BYTES);
            for (int c = 0; c < L::KATOMS; ++c)
                tma_load_3d(sbase + L::Q_OFF + c * L::BOX_BYTES, &p.tmQ, bar(L::B_QFULL), c * 64,
                            qt * BM, bh);
            int issued = 0;
            bool ok = true;
            for (int j = 0; j < n_kv; ++j) {
                const int s = j % L::STAGES;
                if (j >= L::STAGES &&
                    !wait_bounded(bar(L::B_KVEMPTY + s), ((j / L::STAGES) - 1) & 1, abort_flag,
                                  (ROLE_PRODUCER << 24) | (L::B_KVEMPTY << 16) | j)) {
                    ok = false;
                    break;
                }
                const uint32_t kdst = sbase + L::KV_OFF + s * L::STAGE_BYTES;
                mbar_arrive_expect_tx(bar(L::B_KVFULL + s), 2 * L::TILE_BYTES);
                for (int c = 0; c < L::KATOMS; ++c)
                    tma_load_3d(kdst + c * L::BOX_BYTES, &p.tmK, bar(L::B_KVFULL + s), c * 64, j * BN, bh);
                for (int c = 0; c < L::KATOMS; ++c)
                    tma_load_3d(kdst + L::TILE_BYTES + c * L::BOX_BYTES, &p.tmV, bar(L::B_KVFULL + s),
                                c * 64, j * BN, bh);
                ++issued;
            }
            if (!ok) {
                // Let the copies already in flight land before the CTA exits.
                for (int j = issued - L::STAGES < 0 ? 0 : issued - L::STAGES; j < issued; ++j) {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(bar(L::B_KVFULL + j % L::STAGES), (j / L::STAGES) & 1) &&
                           global_timer_ns() - t0 < kDrainLimitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);  // K-major Q and K
            constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 0, 1);   // P from TMEM, V MN-major
            bool ok = wait_bounded(bar(L::B_QFULL), 0, abort_flag, (ROLE_MMA << 24) | (L::B_QFULL << 16));

            auto issue_s = [&](int j) -> bool {
                const int s = j % L::STAGES;
                if (!wait_bounded(bar(L::B_KVFULL + s), (j / L::STAGES) & 1, abort_flag,
                                  (ROLE_MMA << 24) | (L::B_KVFULL << 16) | j))
                    return false;
                tc_fence_after_sync();
                const uint32_t kbase = sbase + L::KV_OFF + s * L::STAGE_BYTES;
                const uint32_t dcol = tmem + ((j & 1) ? TMEM_S1 : TMEM_S0);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k / 4) * L::BOX_BYTES + (k % 4) * 32;
                    umma_ss(dcol, smem_desc_sw128(sbase + L::Q_OFF + off, 16, 1024),
                            smem_desc_sw128(kbase + off, 16, 1024), IDESC_S, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(L::B_SFULL + (j & 1)));
                return true;
            };

            if (ok) ok = issue_s(0);
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) {
                    // S buffer (j+1)&1 last held P_{j-1}: PV_{j-1} must be done.
                    if (j >= 1 && !wait_bounded(bar(L::B_ODONE), (j - 1) & 1, abort_flag,
                                                (ROLE_MMA << 24) | (L::B_ODONE << 16) | j)) {
                        ok = false;
                        break;
                    }
                    if (!issue_s(j + 1)) {
                        ok = false;
                        break;
                    }
                }
                if (!wait_bounded(bar(L::B_PFULL), j & 1, abort_flag,
                                  (ROLE_MMA << 24) | (L::B_PFULL << 16) | j)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const int s = j % L::STAGES;
                const uint32_t vbase = sbase + L::KV_OFF + s * L::STAGE_BYTES + L::TILE_BYTES;
                const uint32_t pcol = tmem + ((j & 1) ? TMEM_S1 : TMEM_S0);
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) {
                    // 16 keys per step: P columns advance by 8 (two bf16 per
                    // 32-bit column), V rows by 16 * 128 bytes.
                    umma_ts(tmem + TMEM_O, pcol + k * 8,
                            smem_desc_sw128(vbase + k * 2048, L::BOX_BYTES, 1024), IDESC_O,
                            (j > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(bar(L::B_KVEMPTY + s));
                umma_commit(bar(L::B_ODONE));
            }
            // Every MMA issued so far has completed before TMEM is released.
            umma_commit(bar(L::B_MMADONE));
            {
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar(L::B_MMADONE), 0) &&
                       global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax / correction / epilogue
        const int t = threadIdx.x;  // row within the tile == TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const int row = qt * BM + t;
        const float c = p.scale_log2e;
        float m = -INFINITY;  // running max of raw scores
        float l = 0.0f;       // running sum of exp2(c*(s - m))
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            const uint32_t sbuf = lane_base + ((j & 1) ? TMEM_S1 : TMEM_S0);
            if (!wait_bounded(bar(L::B_SFULL + (j & 1)), (j >> 1) & 1, abort_flag,
                              (ROLE_SOFTMAX << 24) | (L::B_SFULL << 16) | j)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            float s[BN];
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) {
                uint32_t r[32];
                tmem_ld32(sbuf + q * 32, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[q * 32 + i] = __uint_as_float(r[i]);
            }
            if (j == n_kv - 1) {
                // Last key tile: the ragged tail (keys >= N) and, under the
                // causal mask, the diagonal (keys > row) take -inf.
                const int limit = p.causal ? min(row + 1, p.N) : p.N;
                const int kmax = limit - j * BN;
#pragma unroll
                for (int i = 0; i < BN; ++i) s[i] = (i < kmax) ? s[i] : -INFINITY;
            }
            float mx = m;
#pragma unroll
            for (int i = 0; i < BN; ++i) mx = fmaxf(mx, s[i]);
            const float ms = (mx == -INFINITY) ? 0.0f : mx * c;
            const float alpha = ex2(m * c - ms);
            float sum = 0.0f;
#pragma unroll
            for (int q = 0; q < BN / 32; ++q) {
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float p0 = ex2(fmaf(s[q * 32 + 2 * i], c, -ms));
                    const float p1 = ex2(fmaf(s[q * 32 + 2 * i + 1], c, -ms));
                    sum += p0 + p1;
                    pk[i] = pack_bf16x2(p0, p1);
                }
                tmem_st16(sbuf + q * 16, pk);  // P (bf16) over the first 64 S columns
            }
            l = l * alpha + sum;
            m = mx;
            if (j > 0) {
                // O holds PV_0..PV_{j-1}; it must be complete before rescaling.
                if (!wait_bounded(bar(L::B_ODONE), (j - 1) & 1, abort_flag,
                                  (ROLE_SOFTMAX << 24) | (L::B_ODONE << 16) | j)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll
                for (int q = 0; q < D / 32; ++q) {
                    uint32_t r[32];
                    tmem_ld32(lane_base + TMEM_O + q * 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                    tmem_st32(lane_base + TMEM_O + q * 32, r);
                }
            }
            tmem_st_wait();
            tc_fence_before_sync();
            mbar_arrive(bar(L::B_PFULL));
        }
        if (ok && wait_bounded(bar(L::B_ODONE), (n_kv - 1) & 1, abort_flag,
                               (ROLE_SOFTMAX << 24) | (L::B_ODONE << 16) | 0xFFFF)) {
            tc_fence_after_sync();
            const float inv_l = 1.0f / l;
            const bool store = row < p.N;
            __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.O) +
                                  (static_cast<size_t>(bh) * p.N + (store ? row : 0)) * D;
#pragma unroll
            for (int q = 0; q < D / 32; ++q) {
                uint32_t r[32];
                tmem_ld32(lane_base + TMEM_O + q * 32, r);
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    pk[i] = pack_bf16x2(__uint_as_float(r[2 * i]) * inv_l,
                                        __uint_as_float(r[2 * i + 1]) * inv_l);
                if (store) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + q * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
            if (store) p.LSE[static_cast<size_t>(bh) * p.N + row] = m * p.scale + logf(l);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ self test

// One CTA waits on a barrier nothing arrives on; the bounded wait gives up,
// records the timeout and the kernel returns normally.
__global__ void selftest_timeout_kernel(uint64_t limit_ns) {
    __shared__ uint64_t b;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_addr(&b), 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        wait_bounded(smem_addr(&b), 0, &abort_flag, (ROLE_SELFTEST << 24), limit_ns);
    __syncthreads();
}

// ------------------------------------------------------------------ host side

template <int D>
static cudaError_t launch_d(const AttnParams &p, cudaStream_t stream) {
    using L = Layout<D>;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        err = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   L::SMEM_ALLOC);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    const long long blocks = static_cast<long long>(p.n_qtiles) * p.BH;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_ALLOC;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D>, p);
}

cudaError_t launch_attn_fwd(int D, const AttnParams &p, int /*num_sms*/, cudaStream_t stream) {
    if (D == 64) return launch_d<64>(p, stream);
    if (D == 128) return launch_d<128>(p, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_selftest_timeout(uint64_t limit_ns, cudaStream_t stream) {
    selftest_timeout_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

cudaError_t read_and_clear_status(cudaStream_t stream, uint32_t *status, uint32_t *detail) {
    cudaError_t err = cudaStreamSynchronize(stream);
    if (err != cudaSuccess) return err;
    unsigned int vals[2] = {0, 0};
    err = cudaMemcpyFromSymbol(&vals[0], g_status, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    err = cudaMemcpyFromSymbol(&vals[1], g_detail, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    const unsigned int zero[1] = {0};
    err = cudaMemcpyToSymbol(g_status, zero, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    err = cudaMemcpyToSymbol(g_detail, zero, sizeof(unsigned int));
    if (err != cudaSuccess) return err;
    *status = vals[0];
    *detail = vals[1];
    return cudaSuccess;
}

}  // namespace tk
