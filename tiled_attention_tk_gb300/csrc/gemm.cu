// gemm.cu -- C = A op(B) on the attention kernels' pipeline (sm_103a, GB300).
//
// The pages single out GEMM as the workload the tile abstractions are built
// around, and name the two grid-level problems of a GEMM and their usual
// cures: a low L2 hit rate (threadblock swizzle) and wave quantisation
// (persistent grid + stream-K) (10100.com/article/71410160, section on
// grid-level abstraction).  This kernel is that GEMM written with the same
// TMA + tcgen05 + TMEM machinery as the attention kernels:
//
//   A  bf16 [M, K] row-major          C  bf16 [M, N] row-major
//   B  bf16 [N, K] row-major (C = A B^T, "b_kmajor")  or  [K, N] (C = A B)
//   fp32 accumulation in TMEM, C rounded to bf16 (round to nearest even).
//
// Two kernels.  Large problems run on CTA pairs (gemm_pair_kernel, below:
// 256 x 256 tiles, M = 256 products shared by two SMs, each loading half of
// the operand tiles).  The rest run on single CTAs (gemm_kernel): one
// persistent CTA per SM, 192 threads: a TMA producer warp, an MMA warp and
// four epilogue warps (one per 32 TMEM lanes).  Output tiles are 128 x 256
// (tcgen05 M = 128, N = 256), the K loop runs in steps of 64 through a
// four-stage shared-memory ring, and the accumulator is double-buffered in
// TMEM (2 x 256 columns) so the epilogue of one tile overlaps the main loop of
// the next.  The pair kernel keeps the same roles, tile order and epilogue.
//
// Schedule (single CTAs).  Tiles are numbered in groups of group_m tile
// rows, column by column inside a group, so the CTAs running at the same
// time share rows of A and columns of B in L2 (the threadblock swizzle).  The first dp_tiles
// tiles are handed out whole, round-robin over the CTAs (data-parallel
// waves).  When the tile count is not a multiple of the CTA count, the last
// sk_tiles tiles (the partial wave plus one full wave) are split in K: their
// K iterations, laid end to end, are cut into equal ranges, one per CTA
// (stream-K).  A CTA whose range starts inside a tile writes its fp32
// partial accumulator to a workspace slot of its own and publishes it on the
// tile's counter; the CTA that holds the tile's first K iteration (it reaches
// that tile last) waits for the counter, adds the partials in CTA order and
// writes C.  The order of the additions is fixed, so C is deterministic.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tk_attn.h"
#include "tk_attn_internal.h"
#include "tk_ptx.cuh"
#include "tk_ptx_pair.cuh"
#include "tk_sync.cuh"

namespace tk {
namespace gemm {

constexpr int BM = 128;            // output tile rows (TMEM lanes)
constexpr int BN = 256;            // output tile columns (TMEM columns)
constexpr int BK = 64;             // K per stage: one 128-byte swizzle atom of bf16
constexpr int STAGES = 4;
constexpr int NUM_THREADS = 192;   // producer, MMA, four epilogue warps
constexpr int WARP_TMA = 0;
constexpr int WARP_MMA = 1;
constexpr int WARP_EPI = 2;        // epilogue warps 2..5 (TMEM lane quarters 2, 3, 0, 1)
constexpr uint32_t TMEM_COLS = 512;
// Role tags of the device status word's `where` field (see tk_sync.cuh).
constexpr uint32_t ROLE_GEMM_PRODUCER = 9;
constexpr uint32_t ROLE_GEMM_MMA = 10;
constexpr uint32_t ROLE_GEMM_EPILOGUE = 11;

constexpr uint32_t A_BYTES = BM * BK * 2;              // 16 KB
constexpr uint32_t B_BYTES = BN * BK * 2;              // 32 KB
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t STAGE_OFF = 0;
constexpr uint32_t C_BOX_BYTES = 32 * 64 * 2;          // one warp's 32 rows x 64 columns of C
constexpr uint32_t CSTAGE_OFF = STAGE_OFF + STAGES * STAGE_BYTES;  // 2 boxes per epilogue warp
constexpr uint32_t BAR_OFF = CSTAGE_OFF + 4 * 2 * C_BOX_BYTES;
constexpr int B_FULL = 0;          // + stage
constexpr int B_EMPTY = STAGES;    // + stage
constexpr int B_ACC_FULL = 2 * STAGES;      // + accumulator (2)
constexpr int B_ACC_EMPTY = 2 * STAGES + 2; // + accumulator (2), four epilogue warps
constexpr int B_MMADONE = 2 * STAGES + 4;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;      // slack to align the ring to 1024 bytes
static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");

// One unit of work: K iterations [kb, ke) of output tile `tile`.
struct Item {
    int tile, kb, ke;
};

// Walks the work of worker `cta` of `grid` (a CTA, or on the pair path a pair
// of CTAs): its data-parallel tiles, then its stream-K range.  Every role of
// the worker walks the same sequence.
struct Schedule {
    const GemmParams &p;
    int cta, grid;
    int dp_next;       // next data-parallel tile of this CTA
    int64_t sk_pos, sk_end;
    __device__ Schedule(const GemmParams &pp, int c, int g) : p(pp), cta(c), grid(g), dp_next(c) {
        const int64_t total = static_cast<int64_t>(p.sk_tiles) * p.k_iters;
        sk_pos = static_cast<int64_t>(c) * p.sk_iters_per_cta;
        sk_end = sk_pos + p.sk_iters_per_cta;
        if (sk_pos > total) sk_pos = total;
        if (sk_end > total) sk_end = total;
    }
    __device__ bool next(Item &it) {
        if (dp_next < p.dp_tiles) {
            it = {dp_next, 0, p.k_iters};
            dp_next += grid;
            return true;
        }
        if (sk_pos >= sk_end) return false;
        const int t = static_cast<int>(sk_pos / p.k_iters);
        const int kb = static_cast<int>(sk_pos % p.k_iters);
        const int64_t left = sk_end - sk_pos;
        const int ke = left < p.k_iters - kb ? kb + static_cast<int>(left) : p.k_iters;
        it = {p.dp_tiles + t, kb, ke};
        sk_pos += ke - kb;
        return true;
    }
};

// Tile id -> (tile row, tile column): groups of group_m tile rows, column by
// column inside a group.
__device__ __forceinline__ void tile_coords(int tile, const GemmParams &p, int &tm, int &tn) {
    const int per_group = p.group_m * p.tiles_n;
    const int g = tile / per_group;
    const int first = g * p.group_m;
    const int rows = min(p.group_m, p.tiles_m - first);
    const int r = tile % per_group;
    tm = first + r % rows;
    tn = r / rows;
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const unsigned *p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

template <bool KMAJOR_B>
__global__ void __launch_bounds__(NUM_THREADS, 1) gemm_kernel(const __grid_constant__ GemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    if (warp == WARP_MMA) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(B_FULL + s), 1);
            mbar_init(bar(B_EMPTY + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(B_ACC_FULL + a), 1);
            mbar_init(bar(B_ACC_EMPTY + a), 4);
        }
        mbar_init(bar(B_MMADONE), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    Schedule sched(p, blockIdx.x, gridDim.x);
    Item it;

    if (warp == WARP_TMA) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&p.tmA);
            tma_prefetch_desc(&p.tmB);
            uint32_t n = 0;  // stages filled so far
            bool ok = true;
            while (ok && sched.next(it)) {
                int tm, tn;
                tile_coords(it.tile, p, tm, tn);
                for (int k = it.kb; k < it.ke; ++k, ++n) {
                    const uint32_t s = n % STAGES;
                    if (n >= STAGES &&
                        !(ok = wait_bounded(bar(B_EMPTY + s), ((n / STAGES) - 1) & 1, abort_flag,
                                            (ROLE_GEMM_PRODUCER << 24) | ((B_EMPTY + s) << 16) | (n & 0xFFFF))))
                        break;
                    const uint32_t a_dst = sbase + STAGE_OFF + s * STAGE_BYTES;
                    const uint32_t b_dst = a_dst + A_BYTES;
                    mbar_arrive_expect_tx(bar(B_FULL + s), STAGE_BYTES);
                    tma_load_3d(a_dst, &p.tmA, bar(B_FULL + s), k * BK, tm * BM, 0);
                    if (KMAJOR_B) {
                        tma_load_3d(b_dst, &p.tmB, bar(B_FULL + s), k * BK, tn * BN, 0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load_3d(b_dst + j * (64 * BK * 2), &p.tmB, bar(B_FULL + s), tn * BN + j * 64,
                                        k * BK, 0);
                    }
                }
            }
            if (!ok) {
                // let the copies in flight land before the CTA exits
                const uint64_t t0 = global_timer_ns();
                const uint32_t first = n > STAGES ? n - STAGES : 0;
                for (uint32_t j = first; j < n; ++j)
                    while (!mbar_try_wait(bar(B_FULL + j % STAGES), (j / STAGES) & 1) &&
                           global_timer_ns() - t0 < kDrainLimitNs) {
                    }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the loop (operands stay warp-uniform); one
        // elected lane sends each stage's MMAs and each commit.
        {
            constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, 0, KMAJOR_B ? 0 : 1);
            uint32_t n = 0;     // stages consumed
            uint32_t items = 0; // accumulators used
            bool ok = true;
            while (ok && sched.next(it)) {
                const uint32_t acc = items & 1;
                // the epilogue has read this accumulator's previous tile
                if (items >= 2 &&
                    !(ok = wait_bounded(bar(B_ACC_EMPTY + acc), ((items >> 1) - 1) & 1, abort_flag,
                                        (ROLE_GEMM_MMA << 24) | ((B_ACC_EMPTY + acc) << 16) | (items & 0xFFFF))))
                    break;
                tc_fence_after_sync();
                const uint32_t d = tmem + acc * BN;
                for (int k = it.kb; k < it.ke; ++k, ++n) {
                    const uint32_t s = n % STAGES;
                    if (!(ok = wait_bounded(bar(B_FULL + s), (n / STAGES) & 1, abort_flag,
                                            (ROLE_GEMM_MMA << 24) | ((B_FULL + s) << 16) | (n & 0xFFFF))))
                        break;
                    tc_fence_after_sync();
                    const uint32_t a_src = sbase + STAGE_OFF + s * STAGE_BYTES;
                    const uint32_t b_src = a_src + A_BYTES;
                    const uint64_t ad = smem_desc_sw128(a_src, 16, 1024);
                    const uint64_t bd = KMAJOR_B ? smem_desc_sw128(b_src, 16, 1024)
                                                 : smem_desc_sw128(b_src, 64 * BK * 2, 1024);
                    uint32_t av[BK / 16], bv[BK / 16];
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        av[kk] = static_cast<uint32_t>(ad) + ((kk * 32) >> 4);
                        bv[kk] = static_cast<uint32_t>(bd) + ((KMAJOR_B ? kk * 32 : kk * 2048) >> 4);
                    }
                    if (elect_one()) {
                        umma_ss_steps<BK / 16>(d, av, static_cast<uint32_t>(ad >> 32), bv, static_cast<uint32_t>(bd >> 32),
                                               IDESC, k > it.kb ? 1u : 0u);
                        umma_commit(bar(B_EMPTY + s));  // the stage is free once these MMAs are done
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (elect_one()) umma_commit(bar(B_ACC_FULL + acc));
                __syncwarp();
                ++items;
            }
            if (elect_one()) umma_commit(bar(B_MMADONE));
            __syncwarp();
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar(B_MMADONE), 0) &&
                   global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps
        const int q = warp % 4;           // TMEM lane quarter
        const int r = q * 32 + lane;      // row of the tile
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t cstage = sbase + CSTAGE_OFF + (warp - WARP_EPI) * 2 * C_BOX_BYTES;
        uint8_t *cstage_ptr = smem + CSTAGE_OFF + (warp - WARP_EPI) * 2 * C_BOX_BYTES;
        uint32_t items = 0, boxes = 0;
        bool ok = true;
        while (ok && sched.next(it)) {
            const uint32_t acc = items & 1;
            if (!(ok = wait_bounded(bar(B_ACC_FULL + acc), (items >> 1) & 1, abort_flag,
                                    (ROLE_GEMM_EPILOGUE << 24) | ((B_ACC_FULL + acc) << 16) | (items & 0xFFFF))))
                break;
            tc_fence_after_sync();
            ++items;
            const uint32_t d = lane_base + acc * BN;
            int tm, tn;
            tile_coords(it.tile, p, tm, tn);
            const bool whole = it.kb == 0 && it.ke == p.k_iters;
            if (it.kb > 0) {
                // --- stream-K partial: fp32 to this CTA's slot, [64 column
                // groups][128 rows][4], so a warp's vector store is 512
                // contiguous bytes; then publish it on the tile's counter.
                float4 *slot = reinterpret_cast<float4 *>(p.partials) + static_cast<size_t>(blockIdx.x) * (BM * BN / 4);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(d + c * 32, v);
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        __stcg(slot + (c * 8 + g) * BM + r,
                               make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                           __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3])));
                }
                tc_fence_before_sync();
                warp_arrive(bar(B_ACC_EMPTY + acc), lane);
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(p.counters + (it.tile - p.dp_tiles), 1u);
                continue;
            }
            // --- the tile's result: this accumulator plus, for a stream-K
            // tile, the partials of the CTAs that hold its later K ranges.
            int first_peer = 0, last_peer = -1;
            if (!whole) {
                const int64_t start = static_cast<int64_t>(it.tile - p.dp_tiles) * p.k_iters;
                const int64_t end = start + p.k_iters;
                first_peer = blockIdx.x + 1;
                last_peer = static_cast<int>((end - 1) / p.sk_iters_per_cta);
                const uint32_t want = 4u * static_cast<uint32_t>(last_peer - blockIdx.x);
                if (lane == 0) {
                    const unsigned *ctr = p.counters + (it.tile - p.dp_tiles);
                    const uint64_t t0 = global_timer_ns();
                    while (ld_acquire_u32(ctr) < want) {
                        if (*abort_flag) { ok = false; break; }
                        if (global_timer_ns() - t0 > kWaitLimitNs) {
                            *abort_flag = 1;
                            record_timeout((ROLE_GEMM_EPILOGUE << 24) | (0xFFu << 16) | (it.tile & 0xFFFF));
                            ok = false;
                            break;
                        }
                    }
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
                __threadfence();
            }
#pragma unroll 1
            for (int h = 0; h < BN / 64; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int c = 2 * h + c2;
                    uint32_t v[32];
                    tmem_ld32(d + c * 32, v);
                    if (h == BN / 64 - 1 && c2 == 1) {
                        tc_fence_before_sync();
                        warp_arrive(bar(B_ACC_EMPTY + acc), lane);  // accumulator free for the MMA warp
                    }
                    float f[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]);
                    for (int peer = first_peer; ok && peer <= last_peer; ++peer) {
                        const float4 *slot =
                            reinterpret_cast<const float4 *>(p.partials) + static_cast<size_t>(peer) * (BM * BN / 4);
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            const float4 x = __ldcg(slot + (c * 8 + g) * BM + r);
                            f[4 * g] += x.x;
                            f[4 * g + 1] += x.y;
                            f[4 * g + 2] += x.z;
                            f[4 * g + 3] += x.w;
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[c2 * 16 + e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
                }
                // 32 rows x 64 columns of C through a 128-byte-swizzled box
                const uint32_t b = boxes & 1;
                ++boxes;
                if (lane == 0) tma_store_wait_read_all();  // box b free again
                __syncwarp();
                uint8_t *box = cstage_ptr + b * C_BOX_BYTES;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(box + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&p.tmC, cstage + b * C_BOX_BYTES, tn * BN + h * 64, tm * BM + q * 32, 0);
                    tma_store_commit();
                }
            }
        }
        if (lane == 0) tma_store_wait_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ CTA pairs
// The same GEMM on pairs of CTAs (a cluster of two, tcgen05 cta_group::2):
// a pair computes a 256 x 256 output tile with M = 256 MMAs.  Each CTA loads
// its own 128 rows of A and its own 128 rows (K-major B) or columns (B
// [K, N]) of B into its shared memory, so every CTA reads half as much B per
// MMA as a single CTA does on a 128 x 256 tile; the leader (cluster rank 0)
// issues each MMA over both CTAs' operands, and each CTA's TMEM holds its 128
// rows of the accumulator.  The peer's TMA loads complete on the leader's
// stage barrier (which expects both CTAs' bytes); the leader's commits
// arrive on the barriers of both CTAs, one commit per CTA; the epilogue warps
// of both CTAs free an accumulator on the leader's barrier.  The schedule is
// the single-CTA kernel's with pairs in place of CTAs: whole tiles round-robin
// over the pairs, then, when the tiles do not fill whole waves, the partial
// wave plus one full wave split in K over all pairs (stream-K; a pair's
// partial goes to its own 256 x 256 slot, each CTA its 128 rows, and each of
// the pair's eight epilogue warps counts it on the tile's counter).
namespace pair {

constexpr int BM = 128;            // output rows per CTA (256 per pair)
constexpr int BN = 256;            // output tile columns
constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr uint32_t A_BYTES = BM * BK * 2;           // 16 KB
constexpr uint32_t B_BYTES = (BN / 2) * BK * 2;     // 16 KB: this CTA's half of B
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t STAGE_OFF = 0;
constexpr uint32_t CSTAGE_OFF = STAGE_OFF + STAGES * STAGE_BYTES;
constexpr uint32_t BAR_OFF = CSTAGE_OFF + 4 * 2 * C_BOX_BYTES;
constexpr int B_FULL = 0;                       // + stage (leader): both CTAs' operands landed
constexpr int B_EMPTY = STAGES;                 // + stage (each CTA): the pair's MMAs have read it
constexpr int B_ACC_FULL = 2 * STAGES;          // + accumulator (each CTA)
constexpr int B_ACC_EMPTY = 2 * STAGES + 2;     // + accumulator (leader): 4 epilogue warps x 2 CTAs
constexpr int B_MMADONE = 2 * STAGES + 4;
constexpr int NUM_BARS = 2 * STAGES + 5;
constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");

}  // namespace pair

template <bool KMAJOR_B>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    gemm_pair_kernel(const __grid_constant__ GemmParams p) {
    // this kernel's layout (shadows the single-CTA kernel's constants)
    constexpr int BM = pair::BM, BN = pair::BN, BK = pair::BK, STAGES = pair::STAGES;
    constexpr uint32_t A_BYTES = pair::A_BYTES, STAGE_BYTES = pair::STAGE_BYTES, STAGE_OFF = pair::STAGE_OFF,
                       CSTAGE_OFF = pair::CSTAGE_OFF, BAR_OFF = pair::BAR_OFF;
    constexpr int B_FULL = pair::B_FULL, B_EMPTY = pair::B_EMPTY, B_ACC_FULL = pair::B_ACC_FULL,
                  B_ACC_EMPTY = pair::B_ACC_EMPTY, B_MMADONE = pair::B_MMADONE, NUM_BARS = pair::NUM_BARS;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_addr(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    // The same barrier in the leader's and in this pair's other CTA.
    auto lead_bar = [&](int i) { return cluster_addr(bar(i), 0); };
    auto rank_bar = [&](int i, uint32_t r) { return cluster_addr(bar(i), r); };

    if (warp == WARP_MMA) {
        tmem_alloc_pair(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(B_FULL + s), 1);
            mbar_init(bar(B_EMPTY + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(B_ACC_FULL + a), 1);
            mbar_init(bar(B_ACC_EMPTY + a), 8);
        }
        mbar_init(bar(B_MMADONE), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers exist before either signals the other's
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const int pair_id = static_cast<int>(blockIdx.x) / 2;
    const int n_pairs = static_cast<int>(gridDim.x) / 2;

    if (warp == WARP_TMA) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&p.tmA);
            tma_prefetch_desc(&p.tmB);
            uint32_t n = 0;  // stages filled so far
            bool ok = true;
            Schedule sched(p, pair_id, n_pairs);
            Item it;
            while (ok && sched.next(it)) {
                int tm, tn;
                tile_coords(it.tile, p, tm, tn);
                for (int k = it.kb; k < it.ke; ++k, ++n) {
                    const uint32_t s = n % STAGES;
                    if (n >= STAGES &&
                        !(ok = wait_bounded(bar(B_EMPTY + s), ((n / STAGES) - 1) & 1, abort_flag,
                                            (ROLE_GEMM_PRODUCER << 24) | ((B_EMPTY + s) << 16) | (n & 0xFFFF))))
                        break;
                    const uint32_t a_dst = sbase + STAGE_OFF + s * STAGE_BYTES;
                    const uint32_t b_dst = a_dst + A_BYTES;
                    const uint32_t full = lead_bar(B_FULL + s);
                    if (leader) mbar_arrive_expect_tx(bar(B_FULL + s), 2 * STAGE_BYTES);
                    tma_load_3d_pair(a_dst, &p.tmA, full, k * BK, tm * (2 * BM) + static_cast<int>(rank) * BM, 0);
                    const int n0 = tn * BN + static_cast<int>(rank) * (BN / 2);
                    if (KMAJOR_B) {
                        tma_load_3d_pair(b_dst, &p.tmB, full, k * BK, n0, 0);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 2 / 64; ++j)
                            tma_load_3d_pair(b_dst + j * (64 * BK * 2), &p.tmB, full, n0 + j * 64, k * BK, 0);
                    }
                }
            }
            if (!ok && leader) {
                // let the copies in flight (both CTAs' land on the leader's
                // barriers) arrive before the pair exits
                const uint64_t t0 = global_timer_ns();
                const uint32_t first = n > STAGES ? n - STAGES : 0;
                for (uint32_t j = first; j < n; ++j)
                    while (!mbar_try_wait_cluster(bar(B_FULL + j % STAGES), (j / STAGES) & 1) &&
                           global_timer_ns() - t0 < kDrainLimitNs) {
                    }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------ MMA issuer (the leader)
        if (leader) {
            constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, BN, 0, KMAJOR_B ? 0 : 1);
            uint32_t n = 0;      // stages consumed
            uint32_t items = 0;  // accumulators used
            bool ok = true;
            Schedule sched(p, pair_id, n_pairs);
            Item it;
            while (ok && sched.next(it)) {
                const uint32_t acc = items & 1;
                // both CTAs' epilogues have read this accumulator's previous tile
                if (items >= 2) {
                    const uint32_t ph = ((items >> 1) - 1) & 1;
                    bool done = mbar_try_wait_cluster(bar(B_ACC_EMPTY + acc), ph);
                    const uint64_t t0 = global_timer_ns();
                    while (!done) {
                        done = mbar_try_wait_cluster(bar(B_ACC_EMPTY + acc), ph);
                        if (!done && (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs)) {
                            if (!*abort_flag) record_timeout((ROLE_GEMM_MMA << 24) | ((B_ACC_EMPTY + acc) << 16) |
                                                             (items & 0xFFFF));
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                }
                tc_fence_after_sync();
                const uint32_t d = tmem + acc * BN;
                for (int k = it.kb; k < it.ke; ++k, ++n) {
                    const uint32_t s = n % STAGES;
                    if (!(ok = wait_bounded(bar(B_FULL + s), (n / STAGES) & 1, abort_flag,
                                            (ROLE_GEMM_MMA << 24) | ((B_FULL + s) << 16) | (n & 0xFFFF))))
                        break;
                    tc_fence_after_sync();
                    const uint32_t a_src = sbase + STAGE_OFF + s * STAGE_BYTES;
                    const uint32_t b_src = a_src + A_BYTES;
                    const uint64_t ad = smem_desc_sw128(a_src, 16, 1024);
                    const uint64_t bd = KMAJOR_B ? smem_desc_sw128(b_src, 16, 1024)
                                                 : smem_desc_sw128(b_src, 64 * BK * 2, 1024);
                    uint32_t av[BK / 16], bv[BK / 16];
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        av[kk] = static_cast<uint32_t>(ad) + ((kk * 32) >> 4);
                        bv[kk] = static_cast<uint32_t>(bd) + ((KMAJOR_B ? kk * 32 : kk * 2048) >> 4);
                    }
                    if (elect_one()) {
                        umma_ss_x4_pair(d, av, static_cast<uint32_t>(ad >> 32), bv, static_cast<uint32_t>(bd >> 32),
                                        IDESC, k > it.kb ? 1u : 0u);
                        // the stage is free in both CTAs once these MMAs are done
                        umma_commit_pair(rank_bar(B_EMPTY + s, 0));
                        umma_commit_pair(rank_bar(B_EMPTY + s, 1));
                    }
                    __syncwarp();
                }
                if (!ok) break;
                if (elect_one()) {
                    umma_commit_pair(rank_bar(B_ACC_FULL + acc, 0));
                    umma_commit_pair(rank_bar(B_ACC_FULL + acc, 1));
                }
                __syncwarp();
                ++items;
            }
            if (elect_one()) umma_commit_pair(rank_bar(B_MMADONE, 0));
            __syncwarp();
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar(B_MMADONE), 0) &&
                   global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue warps (both CTAs)
        const int q = warp % 4;           // TMEM lane quarter
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const uint32_t cstage = sbase + CSTAGE_OFF + (warp - WARP_EPI) * 2 * C_BOX_BYTES;
        uint8_t *cstage_ptr = smem + CSTAGE_OFF + (warp - WARP_EPI) * 2 * C_BOX_BYTES;
        const int row = static_cast<int>(rank) * BM + q * 32 + lane;  // row of the pair's 256-row tile
        // this CTA's accumulator is free again for the leader's MMAs
        auto free_acc = [&](uint32_t acc) {
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(lead_bar(B_ACC_EMPTY + acc));
        };
        uint32_t items = 0, boxes = 0;
        bool ok = true;
        Schedule sched(p, pair_id, n_pairs);
        Item it;
        while (ok && sched.next(it)) {
            const uint32_t acc = items & 1;
            const uint32_t ph = (items >> 1) & 1;
            bool done = mbar_try_wait_cluster(bar(B_ACC_FULL + acc), ph);
            const uint64_t t0 = global_timer_ns();
            while (!done) {
                done = mbar_try_wait_cluster(bar(B_ACC_FULL + acc), ph);
                if (!done && (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs)) {
                    if (!*abort_flag)
                        record_timeout((ROLE_GEMM_EPILOGUE << 24) | ((B_ACC_FULL + acc) << 16) | (items & 0xFFFF));
                    *abort_flag = 1;
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            tc_fence_after_sync();
            ++items;
            const uint32_t d = lane_base + acc * BN;
            int tm, tn;
            tile_coords(it.tile, p, tm, tn);
            if (it.kb > 0) {
                // --- stream-K partial: fp32 into the pair's slot, [64 column
                // groups][256 rows][4] (each CTA its 128 rows), then counted
                // on the tile's counter by each of the pair's eight warps.
                float4 *slot = reinterpret_cast<float4 *>(p.partials) + static_cast<size_t>(pair_id) * (2 * BM * BN / 4);
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(d + c * 32, v);
#pragma unroll
                    for (int g = 0; g < 8; ++g)
                        __stcg(slot + (c * 8 + g) * (2 * BM) + row,
                               make_float4(__uint_as_float(v[4 * g]), __uint_as_float(v[4 * g + 1]),
                                           __uint_as_float(v[4 * g + 2]), __uint_as_float(v[4 * g + 3])));
                }
                free_acc(acc);
                __threadfence();
                __syncwarp();
                if (lane == 0) atomicAdd(p.counters + (it.tile - p.dp_tiles), 1u);
                continue;
            }
            // --- the tile's result: this accumulator plus, for a stream-K
            // tile, the partials of the pairs that hold its later K ranges.
            int first_peer = 0, last_peer = -1;
            if (it.ke < p.k_iters) {
                const int64_t start = static_cast<int64_t>(it.tile - p.dp_tiles) * p.k_iters;
                const int64_t end = start + p.k_iters;
                first_peer = pair_id + 1;
                last_peer = static_cast<int>((end - 1) / p.sk_iters_per_cta);
                const uint32_t want = 8u * static_cast<uint32_t>(last_peer - pair_id);
                if (lane == 0) {
                    const unsigned *ctr = p.counters + (it.tile - p.dp_tiles);
                    const uint64_t tw = global_timer_ns();
                    while (ld_acquire_u32(ctr) < want) {
                        if (*abort_flag) { ok = false; break; }
                        if (global_timer_ns() - tw > kWaitLimitNs) {
                            *abort_flag = 1;
                            record_timeout((ROLE_GEMM_EPILOGUE << 24) | (0xFFu << 16) | (it.tile & 0xFFFF));
                            ok = false;
                            break;
                        }
                    }
                }
                ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
                __threadfence();
            }
#pragma unroll 1
            for (int h = 0; h < BN / 64; ++h) {
                uint32_t pk[32];
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int c = 2 * h + c2;
                    uint32_t v[32];
                    tmem_ld32(d + c * 32, v);
                    if (h == BN / 64 - 1 && c2 == 1) free_acc(acc);
                    float f[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]);
                    for (int peer = first_peer; ok && peer <= last_peer; ++peer) {
                        const float4 *slot =
                            reinterpret_cast<const float4 *>(p.partials) + static_cast<size_t>(peer) * (2 * BM * BN / 4);
#pragma unroll
                        for (int g = 0; g < 8; ++g) {
                            const float4 x = __ldcg(slot + (c * 8 + g) * (2 * BM) + row);
                            f[4 * g] += x.x;
                            f[4 * g + 1] += x.y;
                            f[4 * g + 2] += x.z;
                            f[4 * g + 3] += x.w;
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) pk[c2 * 16 + e] = pack_bf16x2(f[2 * e], f[2 * e + 1]);
                }
                const uint32_t b = boxes & 1;
                ++boxes;
                if (lane == 0) tma_store_wait_read_all();  // box b free again
                __syncwarp();
                uint8_t *box = cstage_ptr + b * C_BOX_BYTES;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    *reinterpret_cast<uint4 *>(box + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                        make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&p.tmC, cstage + b * C_BOX_BYTES, tn * BN + h * 64,
                                 tm * (2 * BM) + static_cast<int>(rank) * BM + q * 32, 0);
                    tma_store_commit();
                }
            }
        }
        if (lane == 0) tma_store_wait_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    cluster_sync();  // neither CTA leaves while the other may still signal or read it
    if (warp == WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

}  // namespace gemm

// Pairs of CTAs of the pair kernel that can be resident at once on the
// current device (a GPC with an odd number of free SMs holds one pair fewer
// than half its SMs); cached per device.
cudaError_t gemm_pair_capacity(int *pairs) {
    static thread_local int cached_device = -1, cached_pairs = 0;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (cached_device != dev) {
        for (auto kern : {gemm::gemm_pair_kernel<true>, gemm::gemm_pair_kernel<false>})
            if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            gemm::pair::SMEM_ALLOC)) != cudaSuccess)
                return err;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(gemm::NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = gemm::pair::SMEM_ALLOC;
        int n = 0;
        if ((err = cudaOccupancyMaxActiveClusters(&n, gemm::gemm_pair_kernel<true>, &cfg)) != cudaSuccess)
            return err;
        cached_pairs = n;
        cached_device = dev;
    }
    *pairs = cached_pairs;
    return cudaSuccess;
}

cudaError_t launch_gemm(const GemmParams &p, int grid, cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        if ((err = cudaFuncSetAttribute(gemm::gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        gemm::SMEM_ALLOC)) != cudaSuccess)
            return err;
        if ((err = cudaFuncSetAttribute(gemm::gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        gemm::SMEM_ALLOC)) != cudaSuccess)
            return err;
        if ((err = cudaFuncSetAttribute(gemm::gemm_pair_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        gemm::pair::SMEM_ALLOC)) != cudaSuccess)
            return err;
        if ((err = cudaFuncSetAttribute(gemm::gemm_pair_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        gemm::pair::SMEM_ALLOC)) != cudaSuccess)
            return err;
        configured_device = dev;
    }
    if (p.pair) {
        // The pairs are persistent and the stream-K ranges were planned for
        // this many of them: all must be resident at once.
        int max_pairs = 0;
        if ((err = gemm_pair_capacity(&max_pairs)) != cudaSuccess) return err;
        if (grid < 2 || grid % 2 != 0 || grid / 2 > max_pairs) return cudaErrorInvalidConfiguration;
        if (p.sk_tiles > 0) {
            err = cudaMemsetAsync(p.counters, 0, static_cast<size_t>(p.sk_tiles) * sizeof(unsigned), stream);
            if (err != cudaSuccess) return err;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);  // clusters of two (compile-time dims)
        cfg.blockDim = dim3(gemm::NUM_THREADS, 1, 1);
        cfg.dynamicSmemBytes = gemm::pair::SMEM_ALLOC;
        cfg.stream = stream;
        return p.b_kmajor ? cudaLaunchKernelEx(&cfg, gemm::gemm_pair_kernel<true>, p)
                          : cudaLaunchKernelEx(&cfg, gemm::gemm_pair_kernel<false>, p);
    }
    if (p.sk_tiles > 0) {
        err = cudaMemsetAsync(p.counters, 0, static_cast<size_t>(p.sk_tiles) * sizeof(unsigned), stream);
        if (err != cudaSuccess) return err;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(gemm::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = gemm::SMEM_ALLOC;
    cfg.stream = stream;
    return p.b_kmajor ? cudaLaunchKernelEx(&cfg, gemm::gemm_kernel<true>, p)
                      : cudaLaunchKernelEx(&cfg, gemm::gemm_kernel<false>, p);
}

cudaError_t read_and_clear_gemm_status(uint32_t *status, uint32_t *detail) {
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
