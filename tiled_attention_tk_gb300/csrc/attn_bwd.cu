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
//   bwd_prep_kernel    -Delta_i = -<dO_i, O_i> (fp32) and -LSE_i * log2(e)
//                      per padded query row; zeroes the fp32 dQ accumulator.
//   attn_bwd_kernel<D> one CTA per (head, 128-key tile).  K_j and V_j stay in
//                      shared memory; Q_i of the query tiles that see the
//                      keys streams through two buffers, dO_i through two
//                      (D = 64) or one (D = 128).  The MMA
//                      warp forms S^T = K Q^T and dP^T = V dO^T in TMEM (one
//                      key per TMEM lane); two groups of four compute warps
//                      turn them into P^T and then dS^T, 32 queries at a
//                      time, written back over them as bf16 (dS^T also into
//                      128-byte-swizzled shared memory).  The MMA warp
//                      accumulates dV += P^T dO and dK += dS^T Q chunk by
//                      chunk with P^T and dS^T read from TMEM, then forms
//                      dQ_part = dS K, which four dQ warps add into the fp32
//                      accumulator (at D = 64 staged in shared memory, one bulk
//                      reduction per tile; at D = 128 half staged for one bulk
//                      reduction, half as vector reductions); at the end they
//                      write dK and dV as bf16.
//   bwd_dq_kernel      dQ = bf16(scale * accumulator).
// The same shared-memory tiles serve as K-major and MN-major MMA operands
// through different descriptors (Q and dO are K-major B operands of S^T and
// dP^T and MN-major B operands of dK and dV).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <type_traits>

#include "tk_attn.h"
#include "tk_attn_internal.h"
#include "tk_ptx.cuh"
#include "tk_sync.cuh"

namespace tk {

namespace bwd {

constexpr int BT = 128;             // rows per query tile and per key tile
constexpr int NUM_THREADS = 512;    // 8 compute warps, 4 dQ warps, TMA warp, MMA warp, 2 set-up warps
constexpr int WARP_DQ = 8;          // first of the four dQ warps
constexpr int WARP_TMA = 12;
constexpr int WARP_MMA = 13;
constexpr uint32_t TMEM_COLS = 512;
// Registers per thread and warpgroup: the compute warpgroups keep the launch
// budget, the dQ warpgroup takes what the control warpgroup (TMA, MMA and two
// set-up warps) gives up, so that it can hold a whole dQ_part row (128 fp32)
// before its reductions.  The shares add up to the launch budget (checked on
// the host against the compiled kernel), else the growing warpgroup would wait.
constexpr int LAUNCH_REGS = 128;
constexpr uint32_t REGS_DQ = 160;
constexpr uint32_t REGS_CTRL = 96;
static_assert(2 * LAUNCH_REGS + REGS_DQ + REGS_CTRL == 4 * LAUNCH_REGS, "register split = launch budget");
static_assert(NUM_THREADS == 512, "four whole warpgroups");

template <int D>
struct Layout {
    static constexpr int KATOMS = D / 64;
    static constexpr uint32_t BOX = 128 * 64 * 2;        // one 128-row x 64-column bf16 box
    static constexpr uint32_t TILE = BT * D * 2;         // a 128 x D tile
    static constexpr uint32_t K_OFF = 0;
    static constexpr uint32_t V_OFF = K_OFF + TILE;
    // Q and dO of a query tile.  At D = 64 both are double-buffered: buffer b
    // holds Q at QB_OFF + b * 2 * TILE and dO right after it.  At D = 128 Q is
    // double-buffered and dO single: the dV products are the last to read a
    // tile's dO, and the next tile's dO is first read by its dP^T, after the dK
    // and dQ_part products; the tile this frees stages half a dQ_part block.
    static constexpr uint32_t QB_OFF = V_OFF + TILE;
    static constexpr bool DO_SINGLE = D == 128;
    __host__ __device__ static constexpr uint32_t q_off(int b) {
        return DO_SINGLE ? QB_OFF + b * TILE : QB_OFF + b * 2 * TILE;
    }
    __host__ __device__ static constexpr uint32_t do_off(int b) {
        return DO_SINGLE ? QB_OFF + 2 * TILE : QB_OFF + b * 2 * TILE + TILE;
    }
    static constexpr uint32_t DS_OFF = QB_OFF + 4 * TILE;   // dS^T: 128 keys x 128 queries bf16 (2 boxes)
    // Per Q buffer b, the query tile's row values: -LSE*log2(e) at
    // RB_OFF + b * 1024 and -Delta 512 bytes further (128 floats each).
    static constexpr uint32_t RB_OFF = DS_OFF + 2 * BOX;
    // D = 64 leaves room for two fp32 staging copies of dQ_part, laid out like
    // an accumulator tile ([D/4][128 rows][4]); each goes out as one bulk
    // reduction (the TMA unit adds it into L2) instead of the dQ warps'
    // vector reductions.  D = 128 has room for one half (below); the other
    // half goes out as vector reductions.
    static constexpr bool DQ_BULK = D == 64;
    // D = 128 stages half of dQ_part (64 columns, 32 KB, the size of a bf16
    // tile) in the tile the single dO buffer leaves free.
    static constexpr uint32_t DQST_BYTES = DO_SINGLE ? BT * 64 * 4 : BT * D * 4;
    static constexpr uint32_t DQST_OFF = DO_SINGLE ? QB_OFF + 3 * TILE : RB_OFF + 2048;
    static_assert(!DO_SINGLE || DQST_BYTES == TILE, "the staged half fills the freed tile");
    static constexpr uint32_t BAR_OFF = RB_OFF + 2048 + (DQ_BULK ? 2 * DQST_BYTES : 0);
    static constexpr int B_KVFULL = 0;
    static constexpr int B_QFULL = 1;      // + buffer (2): Q and dO loaded
    static constexpr int B_QEMPTY = 3;     // + buffer (2): the products that read them are done (MMA commit)
    static constexpr int B_SFULL = 5;      // S^T in TMEM (MMA commit)
    static constexpr int B_DPFULL = 6;     // dP^T in TMEM (MMA commit)
    static constexpr int B_PRDY = 7;       // + chunk (4): 32 queries of P^T in TMEM (a compute group, 4)
    static constexpr int B_DSRDY = 11;     // + chunk (4): 32 queries of dS^T in TMEM and smem (a compute group, 4)
    static constexpr int B_GDONE = 15;     // dQ_part product done (MMA commit)
    static constexpr int B_DQREAD = 16;    // dQ_part read out of TMEM (dQ warps, 4)
    static constexpr int B_MMADONE = 17;
    static constexpr int B_STAGED = 18;    // + buffer (2): dQ_part staged (dQ warps, 4)
    static constexpr int B_STAGEFREE = 20; // + buffer (2): its bulk reduction has read it (one thread)
    static constexpr int B_KVFREE = 22;    // a unit's K and V are no longer read (MMA commit)
    static constexpr int B_DKVREAD = 23;   // a unit's dK and dV have left TMEM (dQ warps, 4)
    static constexpr int B_DOFULL = 24;    // dO loaded (single buffer)
    static constexpr int B_DOEMPTY = 25;   // the dV products that read dO are done (MMA commit)
    static constexpr int NUM_BARS = 26;
    static constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
    // No alignment slack: the dynamic shared memory of a kernel without
    // static shared memory starts 1024-byte aligned (the kernel checks).
    static constexpr uint32_t SMEM_ALLOC = SMEM_USED > 116u * 1024u ? SMEM_USED : 116u * 1024u;  // one CTA per SM
    static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");
    // TMEM columns; lane = key of this CTA's key tile, except dQ_part
    // (lane = query of the current query tile).
    static constexpr uint32_t T_S = 0;           // S^T, then bf16 P^T (see pcol)
    static constexpr uint32_t T_DP = 128;        // dP^T, then bf16 dS^T (see pcol); then dQ_part at D = 128
    // dQ_part (D columns): at D = 64 in columns of its own (the next dP^T need
    // not wait for it to be read), at D = 128 over the dP^T block
    static constexpr bool DQ_OWN = D == 64;
    static constexpr uint32_t T_DQ = DQ_OWN ? 384 : T_DP + 128 - D;
    static constexpr uint32_t T_DV = 256;        // dV accumulator (D columns)
    static constexpr uint32_t T_DK = 256 + D;    // dK accumulator (D columns)
    // Column (within the S^T / dP^T block) of the bf16 results of query
    // chunk c (32 queries, 16 columns): each compute group writes only over
    // its own inputs (group 0: columns 0..63, group 1: 64..127), after
    // reading them.
    __host__ __device__ static constexpr uint32_t pcol(int c) { return c < 2 ? 16 * c : 64 + 16 * (c - 2); }
};

// Shared-memory address of 16-byte chunk `c` (0..7) of row `r` in a
// 128-byte-swizzled box (the layout TMA writes with the 128-byte swizzle).
__device__ __forceinline__ uint32_t sw128_chunk(uint32_t box, int r, int c) {
    return box + r * 128 + ((c ^ (r & 7)) << 4);
}

// Adds four floats to global memory with one vector reduction.
__device__ __forceinline__ void red_add_v4(float *addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(__uint_as_float(a)),
                 "f"(__uint_as_float(b)), "f"(__uint_as_float(c)), "f"(__uint_as_float(d))
                 : "memory");
}

// Adds `bytes` (a multiple of 16) of fp32 from shared memory into global
// memory with the bulk-copy unit, in the current bulk group.
__device__ __forceinline__ void bulk_reduce_add_f32(float *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
}

// Waits until every bulk group but the newest has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// The two floats of a packed bf16 pair (low half first).
__device__ __forceinline__ float2 unpack_bf16x2(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

__device__ __forceinline__ uint32_t pack2(float2 v) { return pack_bf16x2(v.x, v.y); }

// Work units: key tile kt of head bh.  The grid is persistent (at most one
// CTA per SM), and a CTA starts its next unit while its last one finishes.
// Without the mask every unit costs the same: CTA c takes the head-major
// units c, c + grid, ..., so the CTAs running together hold a few heads' key
// tiles and share their Q and dO through L2.  Under the mask key tile kt sees
// n_tiles - kt query tiles; see bwd_sched.
struct BwdUnit {
    int kt, bh;
};

__device__ __forceinline__ int bwd_slot_index(int round, int cta, int grid) {
    return round * grid + ((round & 1) ? grid - 1 - cta : cta);
}

// The schedule under the mask: slots, one per CTA per round, odd rounds in
// reverse CTA order (snake).  The first heads run their key tiles in mirrored
// pairs (key tile i, which sees n_tiles - i query tiles, then key tile
// n_tiles-1-i, which sees i + 1: n_tiles + 1 together, whatever i is), head by
// head, so these slots are balanced as they come and the CTAs running together
// share a few heads' Q and dO; the heads left once fewer than two rounds of
// pairs would remain run one key tile per slot, heaviest first, which evens
// out the last rounds.  Odd tile counts run that way throughout.
struct BwdSched {
    int heads_paired, pair_slots, slots;
};

__device__ __forceinline__ BwdSched bwd_sched(const BwdParams &p) {
    BwdSched s{0, 0, p.BH * p.n_tiles};
    if (p.causal && p.n_tiles % 2 == 0) {
        const int hp = p.n_tiles / 2;
        s.heads_paired = max(0, (p.BH * hp - 2 * static_cast<int>(gridDim.x)) / hp);
        s.pair_slots = s.heads_paired * hp;
        s.slots = s.pair_slots + (p.BH - s.heads_paired) * p.n_tiles;
    }
    return s;
}

// Units this CTA runs (two per slot of a mirrored pair).
__device__ __forceinline__ int bwd_units_of_cta(const BwdParams &p) {
    const int grid = gridDim.x;
    if (!p.causal) {
        const int total = p.BH * p.n_tiles;
        return (total - static_cast<int>(blockIdx.x) + grid - 1) / grid;
    }
    const BwdSched s = bwd_sched(p);
    const int rounds = (s.slots + grid - 1) / grid;
    const int r0 = s.pair_slots / grid;
    const int pair_rounds = r0 + (bwd_slot_index(r0, blockIdx.x, grid) < s.pair_slots ? 1 : 0);
    return rounds - (bwd_slot_index(rounds - 1, blockIdx.x, grid) >= s.slots ? 1 : 0) + pair_rounds;
}

// The k-th unit of this CTA (k < bwd_units_of_cta).
__device__ __forceinline__ BwdUnit bwd_unit(int k, const BwdParams &p) {
    const int grid = gridDim.x;
    if (!p.causal) {
        const int idx = static_cast<int>(blockIdx.x) + k * grid;
        return {idx % p.n_tiles, idx / p.n_tiles};
    }
    const BwdSched s = bwd_sched(p);
    const int r0 = s.pair_slots / grid;
    const int pair_rounds = r0 + (bwd_slot_index(r0, blockIdx.x, grid) < s.pair_slots ? 1 : 0);
    const int idx = k < 2 * pair_rounds ? bwd_slot_index(k >> 1, blockIdx.x, grid)
                                        : bwd_slot_index(k - pair_rounds, blockIdx.x, grid);
    if (idx < s.pair_slots) {
        const int hp = p.n_tiles / 2, i = idx % hp;
        return {(k < 2 * pair_rounds && (k & 1)) ? p.n_tiles - 1 - i : i, idx / hp};
    }
    const int j = idx - s.pair_slots, left = p.BH - s.heads_paired;
    return {j / left, s.heads_paired + j % left};
}

// Keys sit on the TMEM lanes: the MMA warp forms S^T = K Q^T and
// dP^T = V dO^T, so that each key row of the tile belongs to one TMEM lane.
// Two groups of four compute warps (queries 0..63 and 64..127) write P^T
// and then dS^T back over S^T and dP^T as bf16, 32 queries at a time, and
// the MMA warp consumes each chunk as soon as it is ready: dV += P^T dO and
// dK += dS^T Q read P^T and dS^T from TMEM.  dS^T also goes to shared
// memory, where it is the MN-major A operand of dQ_part = dS K.  The next
// query tile's S^T is issued before this tile's dQ_part, so the compute
// warps start on it while the tensor core finishes this tile; four dQ warps
// add dQ_part into the fp32 accumulator and write dK and dV at the end.
//
// The unscaled dS' = P (dP - Delta) is what the products see; dK and dQ are
// multiplied by `scale` when they are rounded to bf16.
template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1) attn_bwd_kernel(const __grid_constant__ BwdParams p) {
    using L = Layout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    if (sbase & 1023u) {  // the 128-byte-swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) record_timeout(ROLE_BWD_LAYOUT << 24);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + L::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int my_units = bwd_units_of_cta(p);

    if (warp == WARP_MMA) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(L::B_KVFULL), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::B_QFULL + b), 1);
            mbar_init(bar(L::B_QEMPTY + b), 1);
        }
        mbar_init(bar(L::B_SFULL), 1);
        mbar_init(bar(L::B_DPFULL), 1);
        for (int c = 0; c < 4; ++c) {
            mbar_init(bar(L::B_PRDY + c), 4);
            mbar_init(bar(L::B_DSRDY + c), 4);
        }
        mbar_init(bar(L::B_GDONE), 1);
        mbar_init(bar(L::B_DQREAD), 4);
        mbar_init(bar(L::B_MMADONE), 1);
        mbar_init(bar(L::B_KVFREE), 1);
        mbar_init(bar(L::B_DKVREAD), 4);
        mbar_init(bar(L::B_DOFULL), 1);
        mbar_init(bar(L::B_DOEMPTY), 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::B_STAGED + b), 4);
            mbar_init(bar(L::B_STAGEFREE + b), 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp >= WARP_TMA) {
        regs_dealloc<REGS_CTRL>();
        if (warp == WARP_TMA) {
            // ------------------------------------------------ TMA producer
            if (lane == 0) {
                tma_prefetch_desc(&p.tmQ);
                tma_prefetch_desc(&p.tmK);
                tma_prefetch_desc(&p.tmV);
                tma_prefetch_desc(&p.tmDO);
                uint32_t g = 0;          // query tiles loaded (all units of the CTA)
                uint32_t kv_loads = 0;   // units whose K and V were loaded
                uint32_t do_loads = 0;   // dO loads into the single buffer
                bool ok = true;
                auto load_kv = [&](const BwdUnit &u) {
                    mbar_arrive_expect_tx(bar(L::B_KVFULL), 2 * L::TILE);
                    for (int c = 0; c < L::KATOMS; ++c) {
                        tma_load_3d(sbase + L::K_OFF + c * L::BOX, &p.tmK, bar(L::B_KVFULL), c * 64, u.kt * BT, u.bh);
                        tma_load_3d(sbase + L::V_OFF + c * L::BOX, &p.tmV, bar(L::B_KVFULL), c * 64, u.kt * BT, u.bh);
                    }
                    ++kv_loads;
                };
                for (int k = 0; ok && k < my_units; ++k) {
                    const BwdUnit u = bwd_unit(k, p);
                    const int qt_first = p.causal ? u.kt : 0;
                    const int n_q = p.n_tiles - qt_first;
                    const size_t head_tiles = static_cast<size_t>(u.bh) * p.n_tiles;
                    if (k == 0) load_kv(u);  // the first unit's K and V lead
                    for (int it = 0; it < n_q; ++it) {
                        const int b = g & 1;
                        // Buffer b was last used by query tile g-2.
                        if (g >= 2 && !(ok = wait_bounded(bar(L::B_QEMPTY + b), ((g >> 1) - 1) & 1, abort_flag,
                                                          (ROLE_BWD_PRODUCER << 24) | ((L::B_QEMPTY + b) << 16) | (g & 0xFFFF))))
                            break;
                        const int qt = qt_first + it;
                        const uint32_t qb = sbase + L::q_off(b), dob = sbase + L::do_off(b);
                        const uint32_t rb = sbase + L::RB_OFF + b * 1024;
                        const size_t row0 = (head_tiles + qt) * BT;
                        mbar_arrive_expect_tx(bar(L::B_QFULL + b), (L::DO_SINGLE ? 1 : 2) * L::TILE + 1024);
                        for (int c = 0; c < L::KATOMS; ++c)
                            tma_load_3d(qb + c * L::BOX, &p.tmQ, bar(L::B_QFULL + b), c * 64, qt * BT, u.bh);
                        bulk_load(rb, p.neg_lse2 + row0, 512, bar(L::B_QFULL + b));
                        bulk_load(rb + 512, p.neg_delta + row0, 512, bar(L::B_QFULL + b));
                        if constexpr (L::DO_SINGLE) {
                            ++g;  // counted before the wait below, so that the drain covers Q
                            // the single dO buffer, once the previous tile's dV products are done
                            if (g >= 2 && !(ok = wait_bounded(bar(L::B_DOEMPTY), (g - 2) & 1, abort_flag,
                                                              (ROLE_BWD_PRODUCER << 24) | (L::B_DOEMPTY << 16) | (g & 0xFFFF))))
                                break;
                            mbar_arrive_expect_tx(bar(L::B_DOFULL), L::TILE);
                            for (int c = 0; c < L::KATOMS; ++c)
                                tma_load_3d(dob + c * L::BOX, &p.tmDO, bar(L::B_DOFULL), c * 64, qt * BT, u.bh);
                            ++do_loads;
                        } else {
                            for (int c = 0; c < L::KATOMS; ++c)
                                tma_load_3d(dob + c * L::BOX, &p.tmDO, bar(L::B_QFULL + b), c * 64, qt * BT, u.bh);
                            ++g;
                        }
                        if (it == 0 && k > 0) {
                            // a later unit's K and V, once the unit before no longer reads
                            // them (its first Q and dO went ahead into the free buffer)
                            if (!(ok = wait_bounded(bar(L::B_KVFREE), (k - 1) & 1, abort_flag,
                                                    (ROLE_BWD_PRODUCER << 24) | (L::B_KVFREE << 16) | k)))
                                break;
                            load_kv(u);
                        }
                    }
                }
                if (!ok) {
                    // Let the copies in flight land before the CTA exits.
                    const uint64_t t0 = global_timer_ns();
                    for (uint32_t j = g >= 2 ? g - 2 : 0; j < g; ++j)
                        while (!mbar_try_wait(bar(L::B_QFULL + (j & 1)), (j >> 1) & 1) &&
                               global_timer_ns() - t0 < kDrainLimitNs) {
                        }
                    if (kv_loads > 0)
                        while (!mbar_try_wait(bar(L::B_KVFULL), (kv_loads - 1) & 1) && global_timer_ns() - t0 < kDrainLimitNs) {
                        }
                    if (do_loads > 0)
                        while (!mbar_try_wait(bar(L::B_DOFULL), (do_loads - 1) & 1) && global_timer_ns() - t0 < kDrainLimitNs) {
                        }
                }
            }
            __syncwarp();
        } else if (warp == WARP_MMA) {
            // ------------------------------------------------ MMA issuer
            // Per query tile i: dV(i) chunk by chunk, S^T(i+1), dK(i) chunk by
            // chunk, dQ_part(i), then dP^T(i+1) once dQ_part(i) has been read.
            // Each product that overwrites TMEM columns an earlier product reads
            // (S^T over P^T, dQ_part over dS^T) is issued after it; the tensor core
            // runs one thread's products in issue order.  The whole warp runs
            // the loop (operands stay warp-uniform); one elected lane sends each
            // block of products and each commit.
            {
                constexpr uint32_t IDESC_KK = idesc_bf16_f32(BT, BT, 0, 0);  // S^T, dP^T: K-major A and B
                constexpr uint32_t IDESC_TS = idesc_bf16_f32(BT, D, 0, 1);   // dV, dK: A from TMEM, B MN-major
                constexpr uint32_t IDESC_MM = idesc_bf16_f32(BT, D, 1, 1);   // dQ_part: MN-major A and B
                // Descriptors are formed once per operand tile; a k step adds its
                // compile-time offset to the start-address field, which cannot
                // carry out of its 14 bits (shared memory is below 256 KB).
                auto commit = [&](int b) {
                    if (elect_one()) umma_commit(bar(b));
                    __syncwarp();
                };
                // A = (K or V) x B = (Q or dO), both K-major over D, into `dst`.
                auto issue_kmajor = [&](uint32_t dst, uint32_t a_tile, uint32_t b_tile, int done_bar) {
                    const uint64_t ad = smem_desc_sw128(a_tile, 16, 1024), bd = smem_desc_sw128(b_tile, 16, 1024);
                    const uint32_t hi = static_cast<uint32_t>(ad >> 32);
                    uint32_t av[D / 16], bv[D / 16];
    #pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = ((k / 4) * L::BOX + (k % 4) * 32) >> 4;
                        av[k] = static_cast<uint32_t>(ad) + off;
                        bv[k] = static_cast<uint32_t>(bd) + off;
                    }
                    if (elect_one()) {
                        umma_ss_steps<D / 16>(dst, av, hi, bv, hi, IDESC_KK, 0u);
                        umma_commit(bar(done_bar));
                    }
                    __syncwarp();
                };
                auto issue_s = [&](uint32_t qb) { issue_kmajor(tmem + L::T_S, sbase + L::K_OFF, qb, L::B_SFULL); };     // S^T = K Q^T
                auto issue_dp = [&](uint32_t dob) { issue_kmajor(tmem + L::T_DP, sbase + L::V_OFF, dob, L::B_DPFULL); };  // dP^T = V dO^T
                uint32_t g = 0;  // query tiles (all units of the CTA)
                bool ok = true;
                for (int k = 0; ok && k < my_units; ++k) {
                    const int n_q = p.n_tiles - (p.causal ? bwd_unit(k, p).kt : 0);
                    // The unit's first S^T and dP^T: its K and V loaded, its first Q and dO
                    // loaded, and (dP^T lies over dQ_part) the previous tile's dQ_part read.
                    {
                        const uint32_t q0 = sbase + L::q_off(g & 1);
                        if (!(ok = wait_bounded(bar(L::B_KVFULL), k & 1, abort_flag,
                                                (ROLE_BWD_MMA << 24) | (L::B_KVFULL << 16) | k) &&
                                   wait_bounded(bar(L::B_QFULL + (g & 1)), (g >> 1) & 1, abort_flag,
                                                (ROLE_BWD_MMA << 24) | ((L::B_QFULL + (g & 1)) << 16) | (g & 0xFFFF))))
                            break;
                        tc_fence_after_sync();
                        issue_s(q0);
                        if (!L::DQ_OWN && g > 0 && !(ok = wait_bounded(bar(L::B_DQREAD), (g - 1) & 1, abort_flag,
                                                         (ROLE_BWD_MMA << 24) | (L::B_DQREAD << 16) | (g & 0xFFFF))))
                            break;
                        if (L::DO_SINGLE && !(ok = wait_bounded(bar(L::B_DOFULL), g & 1, abort_flag,
                                                                (ROLE_BWD_MMA << 24) | (L::B_DOFULL << 16) | (g & 0xFFFF))))
                            break;
                        tc_fence_after_sync();
                        issue_dp(sbase + L::do_off(g & 1));
                    }
                    for (int it = 0; ok && it < n_q; ++it, ++g) {
                        const int b = g & 1;
                        const uint32_t ph = g & 1;
                        const uint32_t qb = sbase + L::q_off(b);
                        const uint32_t dob = sbase + L::do_off(b);
                        const uint64_t qb_mn = smem_desc_sw128(qb, L::BOX, 1024), dob_mn = smem_desc_sw128(dob, L::BOX, 1024);
                        const uint32_t mn_hi = static_cast<uint32_t>(qb_mn >> 32);
                        // The unit's first dV and dK products start the accumulators
                        // over: the previous unit's dK and dV must have left TMEM.
                        if (it == 0 && k > 0 &&
                            !(ok = wait_bounded(bar(L::B_DKVREAD), (k - 1) & 1, abort_flag,
                                                (ROLE_BWD_MMA << 24) | (L::B_DKVREAD << 16) | k)))
                            break;
                        // dV += P^T dO as the P^T chunks arrive: 16 queries per step,
                        // 8 TMEM columns of P^T, dO rows advance by 16 * 128 bytes.
                        for (int c = 0; ok && c < 4; ++c) {
                            if (!(ok = wait_bounded(bar(L::B_PRDY + c), ph, abort_flag,
                                                    (ROLE_BWD_MMA << 24) | ((L::B_PRDY + c) << 16) | (g & 0xFFFF))))
                                break;
                            tc_fence_after_sync();
                            const uint32_t b0 = static_cast<uint32_t>(dob_mn) + ((2 * c * 2048) >> 4), b1 = b0 + (2048 >> 4);
                            if (elect_one()) {
                                umma_ts_lo(tmem + L::T_DV, tmem + L::T_S + L::pcol(c), b0, mn_hi, IDESC_TS, (it > 0 || c > 0) ? 1u : 0u);
                                umma_ts_lo(tmem + L::T_DV, tmem + L::T_S + L::pcol(c) + 8, b1, mn_hi, IDESC_TS, 1u);
                            }
                            __syncwarp();
                        }
                        if (!ok) break;
                        if constexpr (L::DO_SINGLE) commit(L::B_DOEMPTY);  // the single dO buffer may be reloaded
                        // S^T of the next query tile over P^T: the dV products above
                        // were the last to read P^T (the compute warps keep their own
                        // copy for dS^T), so the next P^T pass can start as soon as
                        // this tile's dS^T pass ends.
                        const bool has_next = it + 1 < n_q;
                        const uint32_t qn = sbase + L::q_off(b ^ 1);
                        if (has_next) {
                            if (!(ok = wait_bounded(bar(L::B_QFULL + (b ^ 1)), ((g + 1) >> 1) & 1, abort_flag,
                                                    (ROLE_BWD_MMA << 24) | ((L::B_QFULL + (b ^ 1)) << 16) | (g & 0xFFFF))))
                                break;
                            tc_fence_after_sync();
                            issue_s(qn);
                        }
                        // dK += dS'^T Q likewise.
                        for (int c = 0; ok && c < 4; ++c) {
                            if (!(ok = wait_bounded(bar(L::B_DSRDY + c), ph, abort_flag,
                                                    (ROLE_BWD_MMA << 24) | ((L::B_DSRDY + c) << 16) | (g & 0xFFFF))))
                                break;
                            tc_fence_after_sync();
                            const uint32_t b0 = static_cast<uint32_t>(qb_mn) + ((2 * c * 2048) >> 4), b1 = b0 + (2048 >> 4);
                            if (elect_one()) {
                                umma_ts_lo(tmem + L::T_DK, tmem + L::T_DP + L::pcol(c), b0, mn_hi, IDESC_TS, (it > 0 || c > 0) ? 1u : 0u);
                                umma_ts_lo(tmem + L::T_DK, tmem + L::T_DP + L::pcol(c) + 8, b1, mn_hi, IDESC_TS, 1u);
                            }
                            __syncwarp();
                        }
                        if (!ok) break;
                        commit(L::B_QEMPTY + b);  // Q, dO of this tile are no longer read
                        // with its own columns, the previous tile's dQ_part must have been read first
                        if (L::DQ_OWN && g > 0 && !(ok = wait_bounded(bar(L::B_DQREAD), (g - 1) & 1, abort_flag,
                                                                      (ROLE_BWD_MMA << 24) | (L::B_DQREAD << 16) | (g & 0xFFFF))))
                            break;
                        // dQ_part = dS' K (lane = query), 16 keys per step, dS' from
                        // the dS^T buffer (MN-major A) and K MN-major.
                        {
                            const uint64_t dsd = smem_desc_sw128(sbase + L::DS_OFF, L::BOX, 1024),
                                           kmd = smem_desc_sw128(sbase + L::K_OFF, L::BOX, 1024);
                            const uint32_t hi = static_cast<uint32_t>(dsd >> 32);
                            uint32_t av[BT / 16], bv[BT / 16];
    #pragma unroll
                            for (int kk = 0; kk < BT / 16; ++kk) {
                                av[kk] = static_cast<uint32_t>(dsd) + ((kk * 2048) >> 4);
                                bv[kk] = static_cast<uint32_t>(kmd) + ((kk * 2048) >> 4);
                            }
                            if (elect_one()) {
                                umma_ss_steps<BT / 16>(tmem + L::T_DQ, av, hi, bv, hi, IDESC_MM, 0u);
                                umma_commit(bar(L::B_GDONE));
                                if (!has_next) umma_commit(bar(L::B_KVFREE));  // the unit's K and V are no longer read
                            }
                            __syncwarp();
                        }
                        if (has_next) {
                            if (!L::DQ_OWN && !(ok = wait_bounded(bar(L::B_DQREAD), ph, abort_flag,
                                                    (ROLE_BWD_MMA << 24) | (L::B_DQREAD << 16) | (g & 0xFFFF))))
                                break;
                            if (L::DO_SINGLE && !(ok = wait_bounded(bar(L::B_DOFULL), (g + 1) & 1, abort_flag,
                                                                    (ROLE_BWD_MMA << 24) | (L::B_DOFULL << 16) | (g & 0xFFFF))))
                                break;
                            tc_fence_after_sync();
                            issue_dp(sbase + L::do_off(b ^ 1));
                        }
                    }
                }
                commit(L::B_MMADONE);
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar(L::B_MMADONE), 0) &&
                       global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
                }
            }
            __syncwarp();
        }
    } else if (warp < WARP_DQ) {
        // ------------------------------------------------ compute warps
        const int grp = warp / 4;              // queries 64*grp .. 64*grp + 63
        const int t = (warp % 4) * 32 + lane;  // TMEM lane: key row t of the key tile
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
        const float2 c2 = make_float2(p.scale_log2e, p.scale_log2e);
        bool ok = true;
        uint32_t g = 0;  // query tiles (all units of the CTA)
        for (int k = 0; ok && k < my_units; ++k) {
        const BwdUnit u = bwd_unit(k, p);
        const int n_q = p.n_tiles - (p.causal ? u.kt : 0);
        const bool key_out = u.kt * BT + t >= p.N;  // this lane's key is past N
        const bool ragged = u.kt * BT + BT > p.N;   // the key tile holds keys past N
        for (int it = 0; it < n_q; ++it, ++g) {
            const uint32_t ph = g & 1;
            // -LSE*log2(e) and -Delta of this group's 64 queries, loaded with
            // Q and dO (padded rows: -inf and 0, so their weights and
            // gradients are 0)
            const float *rows = reinterpret_cast<const float *>(smem + L::RB_OFF + (g & 1) * 1024) + grp * 64;
            const float4 *nl4 = reinterpret_cast<const float4 *>(rows);
            const float4 *dl4 = reinterpret_cast<const float4 *>(rows + 128);
            // At D = 64 the row values are requested before the TMEM loads they
            // go with (and both chunks of S^T at once), so their shared-memory
            // latency overlaps the TMEM latency; at D = 128 this measured no
            // faster and the values are read where they are used.
            constexpr bool kEarlyRows = D == 64;
            // Only the causal diagonal tile (a unit's first query tile under
            // the mask) and a ragged last key tile hold weights to zero: the
            // queries below qmin do not see this key (keys past N are seen by
            // none).
            const bool diag = p.causal && it == 0;
            const bool masked = diag || ragged;
            const int qmin = key_out ? BT : (diag ? t : 0);

            // P^T = exp2(S^T c - LSE log2 e), bf16, 32 queries per chunk
            // The row values of a chunk come from `lv`: shared memory, or (see
            // kEarlyRows) registers loaded before the chunk's TMEM load.
            auto p_chunk = [&](const uint32_t(&sr)[32], const float4 *lv, int cc, uint32_t(&pp)[16],
                               auto mask_tag) {
                const int q0 = (2 * grp + cc) * 32;
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 l4 = lv[e4];
                    float2 x0 = __ffma2_rn(make_float2(__uint_as_float(sr[4 * e4]), __uint_as_float(sr[4 * e4 + 1])),
                                           c2, make_float2(l4.x, l4.y));
                    float2 x1 = __ffma2_rn(
                        make_float2(__uint_as_float(sr[4 * e4 + 2]), __uint_as_float(sr[4 * e4 + 3])), c2,
                        make_float2(l4.z, l4.w));
                    float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
                    float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
                    if constexpr (decltype(mask_tag)::value) {
                        const int q = q0 + 4 * e4;
                        if (q + 0 < qmin) p0.x = 0.0f;
                        if (q + 1 < qmin) p0.y = 0.0f;
                        if (q + 2 < qmin) p1.x = 0.0f;
                        if (q + 3 < qmin) p1.y = 0.0f;
                    }
                    pp[2 * e4] = pack2(p0);
                    pp[2 * e4 + 1] = pack2(p1);
                }
            };
            // dS' = P (dP - Delta), bf16
            auto ds_chunk = [&](const uint32_t(&dr)[32], const uint32_t(&pr)[16], const float4 *dv,
                                uint32_t(&ds)[16]) {
#pragma unroll
                for (int e4 = 0; e4 < 8; ++e4) {
                    const float4 d4 = dv[e4];
                    const float2 g0 = __fadd2_rn(
                        make_float2(__uint_as_float(dr[4 * e4]), __uint_as_float(dr[4 * e4 + 1])),
                        make_float2(d4.x, d4.y));
                    const float2 g1 = __fadd2_rn(
                        make_float2(__uint_as_float(dr[4 * e4 + 2]), __uint_as_float(dr[4 * e4 + 3])),
                        make_float2(d4.z, d4.w));
                    ds[2 * e4] = pack2(__fmul2_rn(unpack_bf16x2(pr[2 * e4]), g0));
                    ds[2 * e4 + 1] = pack2(__fmul2_rn(unpack_bf16x2(pr[2 * e4 + 1]), g1));
                }
            };

            if (!(ok = wait_bounded(bar(L::B_SFULL), ph, abort_flag,
                                    (ROLE_BWD_COMPUTE << 24) | (L::B_SFULL << 16) | (g & 0xFFFF))))
                break;
            tc_fence_after_sync();
            // This group's two chunks of bf16 P^T, kept for dS^T (the next S^T
            // overwrites them in TMEM once the dV products have read them).
            uint32_t ppa[16], ppb[16];
            {
                const int ca = 2 * grp, cb = 2 * grp + 1;
                uint32_t sr[32];
                if constexpr (kEarlyRows) {
                    // both chunks of S^T and the first chunk's row values at once
                    uint32_t sr2[32];
                    float4 lv[8];
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) lv[e4] = nl4[e4];
                    tmem_ld32_async(lane_base + L::T_S + ca * 32, sr);
                    tmem_ld32_async(lane_base + L::T_S + cb * 32, sr2);
                    tmem_ld_wait();
                    reg_fence(sr);
                    reg_fence(sr2);
                    if (masked) p_chunk(sr, lv, 0, ppa, std::true_type());
                    else p_chunk(sr, lv, 0, ppa, std::false_type());
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) lv[e4] = nl4[8 + e4];
                    tmem_st16(lane_base + L::T_S + L::pcol(ca), ppa);
                    if (masked) p_chunk(sr2, lv, 1, ppb, std::true_type());
                    else p_chunk(sr2, lv, 1, ppb, std::false_type());
                } else {
                    tmem_ld32(lane_base + L::T_S + ca * 32, sr);
                    if (masked) p_chunk(sr, nl4, 0, ppa, std::true_type());
                    else p_chunk(sr, nl4, 0, ppa, std::false_type());
                    tmem_st16(lane_base + L::T_S + L::pcol(ca), ppa);
                    tmem_ld32(lane_base + L::T_S + cb * 32, sr);
                    if (masked) p_chunk(sr, nl4 + 8, 1, ppb, std::true_type());
                    else p_chunk(sr, nl4 + 8, 1, ppb, std::false_type());
                }
                tmem_st16(lane_base + L::T_S + L::pcol(cb), ppb);
                tmem_st_wait();
                tc_fence_before_sync();
                warp_arrive(bar(L::B_PRDY + ca), lane);
                warp_arrive(bar(L::B_PRDY + cb), lane);
            }

            if (!(ok = wait_bounded(bar(L::B_DPFULL), ph, abort_flag,
                                    (ROLE_BWD_COMPUTE << 24) | (L::B_DPFULL << 16) | (g & 0xFFFF))))
                break;
            tc_fence_after_sync();
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int ch = 2 * grp + cc;
                uint32_t dr[32], ds[16];
                const uint32_t(&pr)[16] = cc == 0 ? ppa : ppb;
                float4 dv[8];
                if constexpr (kEarlyRows) {
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4) dv[e4] = dl4[cc * 8 + e4];
                }
                tmem_ld32_async(lane_base + L::T_DP + ch * 32, dr);
                tmem_ld_wait();
                reg_fence(dr);
                ds_chunk(dr, pr, kEarlyRows ? dv : dl4 + cc * 8, ds);
                tmem_st16(lane_base + L::T_DP + L::pcol(ch), ds);
                // dS'^T row t (key), queries ch*32 .. ch*32+31 = pieces 4cc.. of box grp
                const uint32_t dbox = sbase + L::DS_OFF + grp * L::BOX;
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    st_shared_v4(sw128_chunk(dbox, t, cc * 4 + v), ds[4 * v], ds[4 * v + 1], ds[4 * v + 2],
                                 ds[4 * v + 3]);
            }
            tmem_st_wait();
            fence_proxy_async_smem();  // generic-proxy writes -> visible to the tensor core
            tc_fence_before_sync();
            warp_arrive(bar(L::B_DSRDY + 2 * grp), lane);
            warp_arrive(bar(L::B_DSRDY + 2 * grp + 1), lane);
        }
        }
    } else {
        // ------------------------------------------------ dQ warps
        regs_alloc<REGS_DQ>();
        const int t = (warp - WARP_DQ) * 32 + lane;  // TMEM lane: query row t (dQ_part), key row t (dK, dV)
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp - WARP_DQ) * 32) << 16);
        const bool issuer = warp == WARP_DQ && lane == 0;  // issues the bulk reductions
        int bulk_issued = 0;
        bool ok = true;
        uint32_t g = 0;  // query tiles (all units of the CTA)
        for (int k = 0; ok && k < my_units; ++k) {
            const BwdUnit u = bwd_unit(k, p);
            const int qt_first = p.causal ? u.kt : 0;
            const int n_q = p.n_tiles - qt_first;
            // the accumulator tile of the unit's first query tile
            float *const dq_first = p.dq_acc + (static_cast<size_t>(u.bh) * p.n_tiles + qt_first) * BT * D;
            for (int it = 0; it < n_q; ++it, ++g) {
                if (!(ok = wait_bounded(bar(L::B_GDONE), g & 1, abort_flag,
                                        (ROLE_BWD_COMPUTE << 24) | (L::B_GDONE << 16) | (g & 0xFFFF))))
                    break;
                tc_fence_after_sync();
                if constexpr (L::DQ_BULK) {
                    // dQ_part into staging buffer g & 1 ([D/4][128 rows][4], the
                    // accumulator's layout), then one bulk reduction of the tile.
                    uint32_t r0[32], r1[32];
                    tmem_ld32_async(lane_base + L::T_DQ, r0);
                    tmem_ld32_async(lane_base + L::T_DQ + 32, r1);
                    tmem_ld_wait();
                    reg_fence(r0);
                    reg_fence(r1);
                    tc_fence_before_sync();
                    warp_arrive(bar(L::B_DQREAD), lane);
                    const int b = g & 1;
                    if (g >= 2 && !(ok = wait_bounded(bar(L::B_STAGEFREE + b), ((g >> 1) - 1) & 1, abort_flag,
                                                      (ROLE_BWD_COMPUTE << 24) | ((L::B_STAGEFREE + b) << 16) |
                                                          (g & 0xFFFF))))
                        break;
                    const uint32_t stage = sbase + L::DQST_OFF + b * L::DQST_BYTES + t * 16;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stage + j * BT * 16, r0[4 * j], r0[4 * j + 1], r0[4 * j + 2], r0[4 * j + 3]);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stage + (8 + j) * BT * 16, r1[4 * j], r1[4 * j + 1], r1[4 * j + 2], r1[4 * j + 3]);
                    fence_proxy_async_smem();  // generic-proxy writes -> visible to the bulk-copy unit
                    warp_arrive(bar(L::B_STAGED + b), lane);
                    if (issuer) {
                        if ((ok = wait_bounded(bar(L::B_STAGED + b), (g >> 1) & 1, abort_flag,
                                               (ROLE_BWD_COMPUTE << 24) | ((L::B_STAGED + b) << 16) | (g & 0xFFFF)))) {
                            bulk_reduce_add_f32(dq_first + static_cast<size_t>(it) * BT * D,
                                                sbase + L::DQST_OFF + b * L::DQST_BYTES, L::DQST_BYTES);
                            tma_store_commit();
                            ++bulk_issued;
                            if (g >= 1) {
                                // the previous tile's reduction has read its buffer
                                bulk_wait_read_all_but_one();
                                mbar_arrive(bar(L::B_STAGEFREE + (b ^ 1)));
                            }
                        }
                    }
                    __syncwarp();
                    ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;  // the issuer's verdict holds for its warp
                    if (!ok) break;
                } else {
                    // The next dP^T waits for dQ_part to leave TMEM: the whole row
                    // is read (the dQ warpgroup's larger register share) and TMEM
                    // released first.  Then columns 0..63 go through the staging tile,
                    // laid out like the accumulator ([16 column groups][128 rows][4]),
                    // as one bulk reduction by the TMA unit, and columns 64..127 as
                    // vector reductions from the SM: the two paths share the traffic.
                    static_assert(D == 128, "the split reduction runs at D = 128");
                    uint32_t ra[32], rb[32], rc[32], rd[32];
                    tmem_ld32_async(lane_base + L::T_DQ, ra);
                    tmem_ld32_async(lane_base + L::T_DQ + 32, rb);
                    tmem_ld32_async(lane_base + L::T_DQ + 64, rc);
                    tmem_ld32_async(lane_base + L::T_DQ + 96, rd);
                    tmem_ld_wait();
                    reg_fence(ra);
                    reg_fence(rb);
                    reg_fence(rc);
                    reg_fence(rd);
                    tc_fence_before_sync();
                    warp_arrive(bar(L::B_DQREAD), lane);
                    float *const dq_tile = dq_first + static_cast<size_t>(it) * BT * D;
                    // the staging tile is free once the previous tile's bulk reduction has read it
                    if (g >= 1 && !(ok = wait_bounded(bar(L::B_STAGEFREE), (g - 1) & 1, abort_flag,
                                                      (ROLE_BWD_COMPUTE << 24) | (L::B_STAGEFREE << 16) | (g & 0xFFFF))))
                        break;
                    const uint32_t stage = sbase + L::DQST_OFF + t * 16;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stage + j * BT * 16, ra[4 * j], ra[4 * j + 1], ra[4 * j + 2], ra[4 * j + 3]);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        st_shared_v4(stage + (8 + j) * BT * 16, rb[4 * j], rb[4 * j + 1], rb[4 * j + 2], rb[4 * j + 3]);
                    fence_proxy_async_smem();  // generic-proxy writes -> visible to the bulk-copy unit
                    warp_arrive(bar(L::B_STAGED), lane);
                    if (issuer) {
                        if ((ok = wait_bounded(bar(L::B_STAGED), g & 1, abort_flag,
                                               (ROLE_BWD_COMPUTE << 24) | (L::B_STAGED << 16) | (g & 0xFFFF)))) {
                            bulk_reduce_add_f32(dq_tile, sbase + L::DQST_OFF, L::DQST_BYTES);
                            tma_store_commit();
                            ++bulk_issued;
                            tma_store_wait_read_all();  // the staging tile may be rewritten
                            mbar_arrive(bar(L::B_STAGEFREE));
                        }
                    }
                    __syncwarp();
                    ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;  // the issuer's verdict holds for its warp
                    if (!ok) break;
                    float *const dq_row = dq_tile + t * 4;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        red_add_v4(dq_row + (16 + j) * BT * 4, rc[4 * j], rc[4 * j + 1], rc[4 * j + 2], rc[4 * j + 3]);
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        red_add_v4(dq_row + (24 + j) * BT * 4, rd[4 * j], rd[4 * j + 1], rd[4 * j + 2], rd[4 * j + 3]);
                }
            }
            if (!ok) break;
            // dK = scale * (dS'^T Q), dV of this key tile (lane t = key).  The
            // unit's last GDONE wait covers every product; once both are read
            // the next unit's products may start them over.
            const int key = u.kt * BT + t;
            const bool valid_key = key < p.N;
            const float scale = p.scale;
            const size_t head_rows = static_cast<size_t>(u.bh) * p.N;
            // rows of the tensors' head dim p.D (32 and 96 run on the 64- and
            // 128-column kernel: the columns past p.D are not stored)
            __nv_bfloat16 *dkrow = static_cast<__nv_bfloat16 *>(p.dK) + (head_rows + (valid_key ? key : 0)) * p.D;
            __nv_bfloat16 *dvrow = static_cast<__nv_bfloat16 *>(p.dV) + (head_rows + (valid_key ? key : 0)) * p.D;
            // dK then dV, 32 columns at a time (one set of registers at once)
#pragma unroll 1
            for (int q = 0; q < 2 * (D / 32); ++q) {
                const bool is_v = q >= D / 32;
                const int c = is_v ? q - D / 32 : q;
                const float f = is_v ? 1.0f : scale;
                // every lane takes part in the TMEM loads; only the stores are guarded
                uint32_t r[32];
                tmem_ld32(lane_base + (is_v ? L::T_DV : L::T_DK) + c * 32, r);
                if (q == 2 * (D / 32) - 1) {
                    tc_fence_before_sync();
                    warp_arrive(bar(L::B_DKVREAD), lane);
                }
                if (valid_key && c * 32 < p.D) {
                    uint32_t pk[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        pk[e] = pack_bf16x2(f * __uint_as_float(r[2 * e]), f * __uint_as_float(r[2 * e + 1]));
                    __nv_bfloat16 *dst = (is_v ? dvrow : dkrow) + c * 32;
#pragma unroll
                    for (int v = 0; v < 4; ++v)
                        reinterpret_cast<uint4 *>(dst)[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
                }
            }
        }
        // The bulk reductions complete before the CTA (and its shared memory) goes away.
        if (issuer && bulk_issued > 0) tma_store_wait_all();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Per padded query row (n_tiles * 128 rows per head): -Delta = -<dO, O> in
// fp32 and -LSE * log2(e); rows past N get 0 and -inf.  D/8 lanes share a
// row (D the kernel's head dim), 16 bytes of O and of dO each, the lanes
// past the tensors' head dim d reading nothing.  Also zeroes the dQ
// accumulator (acc_vec4 float4s, grid-stride).
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ O,
                                                      const __nv_bfloat16 *__restrict__ dO,
                                                      const float *__restrict__ LSE, float *__restrict__ neg_delta,
                                                      float *__restrict__ neg_lse2, float *__restrict__ dq_acc,
                                                      int64_t padded_rows, int N, int d, int n_tiles,
                                                      int64_t acc_vec4) {
    constexpr int LPR = D / 8;            // lanes per row
    constexpr int RPB = 256 / LPR;        // rows per block
    const int64_t prow = static_cast<int64_t>(blockIdx.x) * RPB + threadIdx.x / LPR;
    const int sub = threadIdx.x % LPR;
    const bool live = prow < padded_rows;
    const int64_t bh = prow / (static_cast<int64_t>(n_tiles) * BT);
    const int n = static_cast<int>(prow % (static_cast<int64_t>(n_tiles) * BT));
    float s = 0.0f;
    if (live && n < N && sub * 8 < d) {
        const int64_t row = bh * N + n;
        const uint4 o = reinterpret_cast<const uint4 *>(O + row * d)[sub];
        const uint4 g = reinterpret_cast<const uint4 *>(dO + row * d)[sub];
        const uint32_t ow[4] = {o.x, o.y, o.z, o.w}, gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 a = unpack_bf16x2(ow[e]), c = unpack_bf16x2(gw[e]);
            s = fmaf(a.x, c.x, s);
            s = fmaf(a.y, c.y, s);
        }
    }
    // every lane of the warp takes part in the reduction
#pragma unroll
    for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
    if (live && sub == 0) {
        neg_delta[prow] = -s;
        neg_lse2[prow] = n < N ? -LSE[bh * N + n] * 1.4426950408889634f : -INFINITY;
    }
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < acc_vec4;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        reinterpret_cast<float4 *>(dq_acc)[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
}

// dQ = bf16(scale * accumulator), one 128-row query tile per block.  The
// accumulator of a tile is [D/4][128 rows][4 floats] (the layout the main
// kernel's reductions add into; D the kernel's head dim): its first d
// columns (the tensors' head dim) are read with consecutive threads on
// consecutive rows, turned into bf16 rows in shared memory, and written out
// row by row, so both sides are coalesced.
template <int D>
__global__ void __launch_bounds__(256) bwd_dq_kernel(const float *__restrict__ dq_acc, __nv_bfloat16 *__restrict__ dQ,
                                                     int N, int d, int n_tiles, float scale) {
    constexpr int STRIDE = D / 2 + 1;  // 32-bit words per staged row (odd: no bank conflicts)
    __shared__ uint32_t rows[BT * STRIDE];
    const int64_t tile = blockIdx.x;   // bh * n_tiles + qt
    const float4 *acc = reinterpret_cast<const float4 *>(dq_acc + tile * BT * D);
    // Fixed trip counts for the 256-thread block: every load of a thread is in
    // flight before the first is used.  Column groups past the tensors' head
    // dim d (96 on the 128-column kernel) are not read.
    constexpr int LOADS = BT * (D / 4) / 256;
    static_assert(LOADS * 256 == BT * (D / 4), "whole loads per thread");
    float4 a[LOADS];
#pragma unroll
    for (int k = 0; k < LOADS; ++k) {
        const int i = static_cast<int>(threadIdx.x) + k * 256;
        a[k] = i / BT < d / 4 ? acc[i] : make_float4(0.f, 0.f, 0.f, 0.f);  // columns 4*grp .. of row t
    }
#pragma unroll
    for (int k = 0; k < LOADS; ++k) {
        const int i = static_cast<int>(threadIdx.x) + k * 256;
        const int t = i % BT, grp = i / BT;
        rows[t * STRIDE + 2 * grp] = pack_bf16x2(scale * a[k].x, scale * a[k].y);
        rows[t * STRIDE + 2 * grp + 1] = pack_bf16x2(scale * a[k].z, scale * a[k].w);
    }
    __syncthreads();
    const int qt = static_cast<int>(tile % n_tiles);
    const int64_t bh = tile / n_tiles;
    constexpr int STORES = BT * (D / 8) / 256;
    static_assert(STORES * 256 == BT * (D / 8), "whole stores per thread");
#pragma unroll
    for (int k = 0; k < STORES; ++k) {
        const int i = static_cast<int>(threadIdx.x) + k * 256;
        const int t = i / (D / 8), g = i % (D / 8);
        const int n = qt * BT + t;
        if (n >= N || g >= d / 8) continue;
        const uint32_t *r = rows + t * STRIDE + 4 * g;
        reinterpret_cast<uint4 *>(dQ + (bh * N + n) * d)[g] = make_uint4(r[0], r[1], r[2], r[3]);
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
        // The warpgroups' register shares add up to a launch budget of 128 per
        // thread; a build compiled to fewer would leave the dQ warpgroup
        // waiting for registers, so it is refused here.
        cudaFuncAttributes attr;
        err = cudaFuncGetAttributes(&attr, attn_bwd_kernel<D>);
        if (err != cudaSuccess) return err;
        if (attr.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        err = cudaFuncSetAttribute(attn_bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::SMEM_ALLOC);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    const int64_t padded_rows = static_cast<int64_t>(p.BH) * p.n_tiles * BT;
    const int64_t acc_vec4 = padded_rows * D / 4;
    constexpr int RPB = 256 / (D / 8);  // rows per prep block
    bwd_prep_kernel<D><<<static_cast<unsigned>((padded_rows + RPB - 1) / RPB), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16 *>(p.O), static_cast<const __nv_bfloat16 *>(p.dO), p.LSE, p.neg_delta,
        p.neg_lse2, p.dq_acc, padded_rows, p.N, p.D, p.n_tiles, acc_vec4);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;

    // A persistent grid: at most one CTA per SM (the units' order is the kernel's).
    const int64_t units = static_cast<int64_t>(p.BH) * p.n_tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(units < num_sms ? units : num_sms), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_ALLOC;
    cfg.stream = stream;
    err = cudaLaunchKernelEx(&cfg, attn_bwd_kernel<D>, p);
    if (err != cudaSuccess) return err;

    bwd_dq_kernel<D><<<static_cast<unsigned>(static_cast<int64_t>(p.BH) * p.n_tiles), 256, 0, stream>>>(
        p.dq_acc, static_cast<__nv_bfloat16 *>(p.dQ), p.N, p.D, p.n_tiles, p.scale);
    return cudaGetLastError();
}

}  // namespace bwd

cudaError_t launch_attn_bwd(int D, const BwdParams &p, int num_sms, cudaStream_t stream) {
    if (num_sms < 1) return cudaErrorInvalidValue;
    if (D == 64 && p.D <= 64) return bwd::launch_d<64>(p, num_sms, stream);
    if (D == 128 && p.D > 64 && p.D <= 128) return bwd::launch_d<128>(p, num_sms, stream);
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
