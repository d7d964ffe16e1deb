// attn_fwd256.cu -- fused attention forward at head dim 256 for sm_103a (GB300).
//
// The computation of attn_fwd.cu -- O = softmax(scale * Q K^T [+ causal
// mask]) V and the natural-log row LSE, with the online softmax of the
// "ThunderKittens" attention kernel (10100.com/article/71410160, section
// "writing a kernel with TK", attn_fwd_template: running row max and sum in
// the exp2 domain, the partial output rescaled when the max moves, P rounded
// to bf16 for the second product, one division at the end) -- laid out for
// D = 256.  A Q tile's fp32 O now takes 256 of the 512 TMEM columns, so a
// work unit is one head and ONE 128-row Q tile, and the other 256 columns
// hold two S slots: the tensor core forms S of key tile j+1 while the softmax
// works on key tile j.  Roles (192 threads):
//   warp 5     TMA producer: Q once per unit (four 64-column boxes, 64 KB),
//              then 64 KB K and V tiles through two shared-memory slots in
//              the order the products use them: K0, K1, V0, K2, V1, K3, ...
//   warp 4     MMA issuer (one thread): S0, S1, then per key tile j:
//              O += P_j V_j and S_{j+2} (over P_j's slot, after the product
//              that reads P_j).  Also owns TMEM.
//   warps 0-3  softmax warpgroup: thread t owns query row t (TMEM lane t):
//              masks the tiles some row does not see in full, takes the row
//              max, writes P = exp2(c*s - c*m_ref) as bf16 over the S slot,
//              rescales O lazily (only when the row max has grown by more
//              than 2^24 since the reference was set; O and l keep the same
//              reference, so O / l is exact), and at the end of the unit
//              writes O / l (bf16) through a staging box and TMA stores, and
//              the LSE.
// Every mbarrier wait is bounded (tk_sync.cuh).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tk_attn.h"
#include "tk_attn_internal.h"
#include "tk_ptx.cuh"
#include "tk_sync.cuh"

namespace tk {
namespace fwd256 {

constexpr int BM = 128;            // query rows per unit (one TMEM lane each)
constexpr int BN = 128;            // keys per key tile
constexpr int NUM_THREADS = 192;   // softmax warpgroup, MMA warp, TMA warp
constexpr int WARP_MMA = 4;
constexpr int WARP_TMA = 5;
constexpr uint32_t TMEM_COLS = 512;
constexpr float kRescaleLog2 = 24.0f;  // as attn_fwd.cu: P < 2^24 between rescales
constexpr uint32_t BOX_BYTES = 128 * 64 * 2;  // one TMA box: 128 rows x 64 bf16

template <int D>
struct Layout {
    static constexpr int KATOMS = D / 64;                  // 64-column boxes along D
    static constexpr uint32_t TILE_BYTES = KATOMS * BOX_BYTES;  // a 128 x D tile
    static constexpr int NSLOTS = D == 256 ? 2 : 4;        // K/V slots
    static constexpr uint32_t Q_OFF = 0;
    static constexpr uint32_t SLOT_OFF = TILE_BYTES;
    static constexpr uint32_t STAGE_OFF = SLOT_OFF + NSLOTS * TILE_BYTES;  // O staging: one 128 x 64 box
    static constexpr uint32_t BAR_OFF = STAGE_OFF + BOX_BYTES;
    static constexpr int B_QFULL = 0;
    static constexpr int B_QEMPTY = 1;                     // the unit's last S product is done
    static constexpr int B_SLOTFULL = 2;                   // + slot
    static constexpr int B_SLOTEMPTY = B_SLOTFULL + NSLOTS;  // + slot: the product reading it is done
    static constexpr int B_SFULL = B_SLOTEMPTY + NSLOTS;   // + S slot (2)
    static constexpr int B_PFULL = B_SFULL + 2;            // + S slot (2): P in the slot (4 warps)
    static constexpr int B_PVDONE = B_PFULL + 2;           // O += P V done
    static constexpr int B_OFREE = B_PVDONE + 1;           // O read out by the epilogue (4 warps)
    static constexpr int B_MMADONE = B_OFREE + 1;
    static constexpr int NUM_BARS = B_MMADONE + 1;
    static constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
    static constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;  // slack for 1024-byte alignment
    // Built for 256.  At 128 the same plan (four K/V slots) measured 11 %
    // slower than attn_fwd.cu's two Q tiles per unit: with one softmax
    // warpgroup the softmax, not the tensor core, then sets the pace.
    static_assert(D == 128 || D == 256, "head dim 128 or 256");
    static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");
    static_assert(SMEM_ALLOC > 116u * 1024u, "one CTA per SM: each CTA holds all 512 TMEM columns");
};
// TMEM columns: S slot s at 128 s, O at 256 (D columns)
__host__ __device__ constexpr uint32_t tmem_s(uint32_t s) { return s * 128u; }
constexpr uint32_t T_O = 256;

struct Unit {
    int bh;
    int qt;
};

// Odd rounds run in reverse CTA order (snake).
__device__ __forceinline__ int unit_index(int round, int cta, int grid) {
    return round * grid + ((round & 1) ? grid - 1 - cta : cta);
}

// Units sit in slots, one slot per CTA per round.  Without the mask a slot is
// one Q tile, the tiles of a head adjacent, so CTAs running together share
// that head's K/V in L2.  Under the causal mask, with an even number of Q
// tiles, the first heads run in mirrored pairs: a slot holds a head's Q tile
// n-1-i and then its tile i, which together visit n+1 key tiles whatever i
// is, so these slots are balanced as they come and lie head by head (CTAs
// running together then read the K/V of a few heads, not of every head).  The
// heads left once fewer than a round of pairs would remain run one tile per
// slot, heaviest first (their last tiles, then the ones before ...), which
// evens out the last rounds.  Odd tile counts run that way throughout.
struct Sched {
    int heads_paired;  // heads whose tiles run in pairs (the first ones)
    int pair_slots;    // heads_paired * n_qtiles / 2
    int slots;
};

template <bool CAUSAL>
__device__ __forceinline__ Sched schedule(const AttnParams &p, int grid) {
    Sched s{0, 0, p.BH * p.n_qtiles};
    if (CAUSAL && p.n_qtiles % 2 == 0) {
        const int hp = p.n_qtiles / 2;
        s.heads_paired = max(0, (p.BH * hp - grid) / hp);
        s.pair_slots = s.heads_paired * hp;
        s.slots = s.pair_slots + (p.BH - s.heads_paired) * p.n_qtiles;
    }
    return s;
}

// Unit `h` (0 or 1) of slot `idx`.
template <bool CAUSAL>
__device__ __forceinline__ Unit slot_unit(int idx, int h, const Sched &s, const AttnParams &p) {
    if (CAUSAL && idx < s.pair_slots) {
        const int hp = p.n_qtiles / 2, i = idx % hp;
        return {idx / hp, h ? i : p.n_qtiles - 1 - i};
    }
    if (CAUSAL) {
        const int j = idx - s.pair_slots, left = p.BH - s.heads_paired;
        return {s.heads_paired + j % left, p.n_qtiles - 1 - j / left};
    }
    return {idx / p.n_qtiles, idx % p.n_qtiles};
}

// Slots of this CTA that hold pairs: every round before the first round with
// single units, and that round's slot if it is still a pair.
__device__ __forceinline__ int pair_rounds_of_cta(const Sched &s, int grid) {
    const int r0 = s.pair_slots / grid;
    return r0 + (unit_index(r0, blockIdx.x, grid) < s.pair_slots ? 1 : 0);
}

// Units this CTA runs: two per pair slot, one per other slot (the last round
// may hold no slot for it).
__device__ __forceinline__ int units_of_cta(const Sched &s, int grid) {
    const int rounds = (s.slots + grid - 1) / grid;
    const int mine = rounds - (unit_index(rounds - 1, blockIdx.x, grid) >= s.slots ? 1 : 0);
    return mine + pair_rounds_of_cta(s, grid);
}

// The k-th unit of this CTA (k < units_of_cta).
template <bool CAUSAL>
__device__ __forceinline__ Unit cta_unit(int k, const Sched &s, int pair_rounds, const AttnParams &p) {
    const int grid = gridDim.x;
    if (CAUSAL && k < 2 * pair_rounds) return slot_unit<CAUSAL>(unit_index(k >> 1, blockIdx.x, grid), k & 1, s, p);
    return slot_unit<CAUSAL>(unit_index(k - pair_rounds, blockIdx.x, grid), 0, s, p);
}

template <bool CAUSAL>
__device__ __forceinline__ int kv_tiles(int qt, const AttnParams &p) {
    if (!CAUSAL) return p.n_kvtiles;
    const int last_key = min(qt * BM + BM, p.Nq) - 1 + p.offset;
    return min(last_key / BN + 1, p.n_kvtiles);
}

// CAUSAL is p.causal: each mask has its own instantiation.
template <int D, bool CAUSAL>
__global__ void __launch_bounds__(NUM_THREADS, 1) attn_fwd256_kernel(const __grid_constant__ AttnParams p) {
    using L = Layout<D>;
    constexpr int KATOMS = L::KATOMS, NSLOTS = L::NSLOTS;
    constexpr uint32_t TILE_BYTES = L::TILE_BYTES, Q_OFF = L::Q_OFF, SLOT_OFF = L::SLOT_OFF,
                       STAGE_OFF = L::STAGE_OFF, BAR_OFF = L::BAR_OFF;
    constexpr int B_QFULL = L::B_QFULL, B_QEMPTY = L::B_QEMPTY, B_SLOTFULL = L::B_SLOTFULL,
                  B_SLOTEMPTY = L::B_SLOTEMPTY, B_SFULL = L::B_SFULL, B_PFULL = L::B_PFULL,
                  B_PVDONE = L::B_PVDONE, B_OFREE = L::B_OFREE, B_MMADONE = L::B_MMADONE,
                  NUM_BARS = L::NUM_BARS;
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
    const int grid = gridDim.x;
    const Sched sched = schedule<CAUSAL>(p, grid);
    const int pair_rounds = pair_rounds_of_cta(sched, grid);
    const int my_units = units_of_cta(sched, grid);

    if (warp == WARP_MMA) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        mbar_init(bar(B_QFULL), 1);
        mbar_init(bar(B_QEMPTY), 1);
        for (int s = 0; s < NSLOTS; ++s) {
            mbar_init(bar(B_SLOTFULL + s), 1);
            mbar_init(bar(B_SLOTEMPTY + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_SFULL + s), 1);
            mbar_init(bar(B_PFULL + s), 4);
        }
        mbar_init(bar(B_PVDONE), 1);
        mbar_init(bar(B_OFREE), 4);
        mbar_init(bar(B_MMADONE), 1);
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
            uint32_t loads = 0;  // K/V tiles loaded, in the order the products use them
            uint32_t q_loads = 0;
            int k_unit = 0;
            bool ok = true;
            for (int k = 0; ok && k < my_units; ++k) {
                const Unit u = cta_unit<CAUSAL>(k, sched, pair_rounds, p);
                const int n_kv = kv_tiles<CAUSAL>(u.qt, p);
                auto load_kv = [&](int j, bool v) -> bool {
                    const int s = loads % NSLOTS;
                    if (loads >= static_cast<uint32_t>(NSLOTS) &&
                        !wait_bounded(bar(B_SLOTEMPTY + s), ((loads / NSLOTS) - 1) & 1, abort_flag,
                                      (ROLE_PRODUCER << 24) | ((B_SLOTEMPTY + s) << 16) | (j & 0xFFFF)))
                        return false;
                    const uint32_t dst = sbase + SLOT_OFF + s * TILE_BYTES;
                    mbar_arrive_expect_tx(bar(B_SLOTFULL + s), TILE_BYTES);
                    for (int c = 0; c < KATOMS; ++c)
                        tma_load_3d(dst + c * BOX_BYTES, v ? &p.tmV : &p.tmK, bar(B_SLOTFULL + s), c * 64, j * BN,
                                    u.bh);
                    ++loads;
                    return true;
                };
                // K_0 only needs a free slot: start it before waiting for the
                // previous unit to release Q.
                if (!(ok = load_kv(0, false))) break;
                if (k_unit > 0 && !(ok = wait_bounded(bar(B_QEMPTY), (k_unit - 1) & 1, abort_flag,
                                                      (ROLE_PRODUCER << 24) | (B_QEMPTY << 16) | k_unit)))
                    break;
                mbar_arrive_expect_tx(bar(B_QFULL), TILE_BYTES);
                for (int c = 0; c < KATOMS; ++c)
                    tma_load_3d(sbase + Q_OFF + c * BOX_BYTES, &p.tmQ, bar(B_QFULL), c * 64, u.qt * BM, u.bh);
                ++q_loads;
                if (n_kv > 1 && !(ok = load_kv(1, false))) break;
                for (int j = 0; ok && j < n_kv; ++j) {
                    ok = load_kv(j, true);
                    if (ok && j + 2 < n_kv) ok = load_kv(j + 2, false);
                }
                ++k_unit;
            }
            if (!ok) {
                // Let the copies in flight land before the CTA exits.
                const uint32_t first = loads > static_cast<uint32_t>(NSLOTS) ? loads - NSLOTS : 0;
                for (uint32_t n = first; n < loads; ++n) {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(bar(B_SLOTFULL + n % NSLOTS), (n / NSLOTS) & 1) &&
                           global_timer_ns() - t0 < kDrainLimitNs) {
                    }
                }
                if (q_loads > 0) {  // the latest Q load
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(bar(B_QFULL), (q_loads - 1) & 1) && global_timer_ns() - t0 < kDrainLimitNs) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        // ------------------------------------------------ MMA issuer
        // The whole warp runs the loop (operands stay warp-uniform); one
        // elected lane sends each block of MMAs and each commit.
        {
            constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);  // K-major Q and K
            constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 0, 1);   // P from TMEM, V MN-major
            uint32_t taken = 0;   // K/V tiles consumed, in load order
            uint32_t g = 0;       // S products issued (all units): S number g uses slot g & 1
            bool ok = true;
            int k_unit = 0;
            auto take_slot = [&](uint32_t &slot) -> bool {
                slot = taken % NSLOTS;
                const bool r = wait_bounded(bar(B_SLOTFULL + slot), (taken / NSLOTS) & 1, abort_flag,
                                            (ROLE_MMA << 24) | ((B_SLOTFULL + slot) << 16) | (taken & 0xFFFF));
                ++taken;
                return r;
            };
            // Descriptors are formed once per operand tile; a k step adds its
            // compile-time offset to the start-address field (no carry:
            // shared memory is below 256 KB).
            const uint64_t qd = smem_desc_sw128(sbase + Q_OFF, 16, 1024);
            const uint32_t q_lo = static_cast<uint32_t>(qd), d_hi = static_cast<uint32_t>(qd >> 32);
            auto commit = [&](int b) {
                if (elect_one()) umma_commit(bar(b));
                __syncwarp();
            };
            auto issue_s = [&](uint32_t s, uint32_t kslot) {  // S = Q K^T into S slot s
                const uint32_t k_lo =
                    static_cast<uint32_t>(smem_desc_sw128(sbase + SLOT_OFF + kslot * TILE_BYTES, 16, 1024));
                uint32_t a[D / 16], b[D / 16];
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = ((k / 4) * BOX_BYTES + (k % 4) * 32) >> 4;
                    a[k] = q_lo + off;
                    b[k] = k_lo + off;
                }
                if (elect_one()) {
                    umma_ss_steps<D / 16>(tmem + tmem_s(s), a, d_hi, b, d_hi, IDESC_S, 0u);
                    umma_commit(bar(B_SFULL + s));
                    umma_commit(bar(B_SLOTEMPTY + kslot));
                }
                __syncwarp();
            };
            auto issue_pv = [&](uint32_t s, uint32_t vslot, bool accumulate) {  // O += P V, P in S slot s
                const uint64_t vd = smem_desc_sw128(sbase + SLOT_OFF + vslot * TILE_BYTES, BOX_BYTES, 1024);
                const uint32_t v_lo = static_cast<uint32_t>(vd), v_hi = static_cast<uint32_t>(vd >> 32);
                uint32_t b[BN / 16];
#pragma unroll
                for (int k = 0; k < BN / 16; ++k) b[k] = v_lo + ((k * 2048) >> 4);
                if (elect_one()) {
                    // 16 keys per step: P advances 8 TMEM columns (two bf16 each)
                    umma_ts_steps<BN / 16, 8>(tmem + T_O, tmem + tmem_s(s), b, v_hi, IDESC_O, accumulate ? 1u : 0u);
                    umma_commit(bar(B_PVDONE));
                    umma_commit(bar(B_SLOTEMPTY + vslot));
                }
                __syncwarp();
            };

            for (int k = 0; ok && k < my_units; ++k) {
                const Unit u = cta_unit<CAUSAL>(k, sched, pair_rounds, p);
                const int n_kv = kv_tiles<CAUSAL>(u.qt, p);
                const uint32_t g0 = g;  // S number of key tile 0 of this unit
                uint32_t ks = 0, vs = 0;
                if (!(ok = wait_bounded(bar(B_QFULL), k_unit & 1, abort_flag,
                                        (ROLE_MMA << 24) | (B_QFULL << 16) | k_unit)))
                    break;
                tc_fence_after_sync();
                for (int j = 0; ok && j < 2 && j < n_kv; ++j) {
                    if (!(ok = take_slot(ks))) break;  // K_j
                    tc_fence_after_sync();
                    issue_s(g & 1, ks);
                    ++g;
                    if (j == n_kv - 1) commit(B_QEMPTY);  // the unit's last S
                }
                for (int j = 0; ok && j < n_kv; ++j) {
                    const uint32_t gj = g0 + j, s = gj & 1;
                    if (!(ok = take_slot(vs))) break;  // V_j
                    if (!(ok = wait_bounded(bar(B_PFULL + s), (gj >> 1) & 1, abort_flag,
                                            (ROLE_MMA << 24) | ((B_PFULL + s) << 16) | (j & 0xFFFF))))
                        break;
                    if (j == 0 && k_unit > 0 &&
                        !(ok = wait_bounded(bar(B_OFREE), (k_unit - 1) & 1, abort_flag,
                                            (ROLE_MMA << 24) | (B_OFREE << 16) | k_unit)))
                        break;
                    tc_fence_after_sync();
                    issue_pv(s, vs, j > 0);
                    if (j + 2 < n_kv) {
                        if (!(ok = take_slot(ks))) break;  // K_{j+2}
                        tc_fence_after_sync();
                        issue_s(s, ks);  // over P_j, after the product that reads it
                        ++g;
                        if (j + 2 == n_kv - 1) commit(B_QEMPTY);
                    }
                }
                if (!ok) break;
                ++k_unit;
            }
            // Every MMA issued so far has completed before TMEM is released.
            commit(B_MMADONE);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar(B_MMADONE), 0) &&
                   global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax / correction / epilogue
        const int t = threadIdx.x;  // row within the Q tile == TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        const uint32_t o_addr = lane_base + T_O;
        const float c = p.scale_log2e;
        uint32_t g = 0;         // S hand-offs consumed (all units)
        uint32_t pv_base = 0;   // O += P V products of earlier units
        bool ok = true;
        for (int k = 0; ok && k < my_units; ++k) {
            const Unit u = cta_unit<CAUSAL>(k, sched, pair_rounds, p);
            const int qt = u.qt;
            const int row = qt * BM + t;
            const int n_kv = kv_tiles<CAUSAL>(qt, p);
            float m_ref = -INFINITY;  // reference max of raw scores (lazy)
            float l = 0.0f;           // sum of exp2(c * (s - m_ref))
            for (int j = 0; j < n_kv; ++j) {
                const uint32_t s = g & 1;
                if (!(ok = wait_bounded(bar(B_SFULL + s), (g >> 1) & 1, abort_flag,
                                        (ROLE_SOFTMAX << 24) | ((B_SFULL + s) << 16) | (j & 0xFFFF))))
                    break;
                ++g;
                tc_fence_after_sync();
                const uint32_t s_addr = lane_base + tmem_s(s);
                uint32_t sr[BN];
                tmem_ld128(s_addr, sr);
                float sv[BN];
#pragma unroll
                for (int i = 0; i < BN; ++i) sv[i] = __uint_as_float(sr[i]);
                if ((j + 1) * BN > p.Nkv || (CAUSAL && (j + 1) * BN > qt * BM + p.offset + 1)) {
                    // the ragged tail (keys >= Nkv) and, under the causal mask,
                    // keys past row + offset take -inf
                    const int limit = CAUSAL ? min(row + 1 + p.offset, p.Nkv) : p.Nkv;
                    const int kmax = limit - j * BN;
#pragma unroll
                    for (int i = 0; i < BN; ++i) sv[i] = (i < kmax) ? sv[i] : -INFINITY;
                }
                // Row max: eight independent chains of three-input maxima.
                float mx8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    float a = sv[k];
#pragma unroll
                    for (int q = 1; q < 15; q += 2) a = fmax3(a, sv[k + 8 * q], sv[k + 8 * (q + 1)]);
                    mx8[k] = fmaxf(a, sv[k + 120]);
                }
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmax3(mx8[6], mx8[7], m_ref));
                const bool need = (mx - m_ref) * c > kRescaleLog2;  // true when m_ref = -inf
                const float new_ref = need ? mx : m_ref;
                const float alpha = need ? ex2((m_ref - mx) * c) : 1.0f;
                const float neg = (new_ref == -INFINITY) ? 0.0f : -new_ref * c;
                const float2 c2 = make_float2(c, c);
                const float2 n2 = make_float2(neg, neg);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = h * 64 + 2 * i;
                        const float2 x = __ffma2_rn(make_float2(sv[e], sv[e + 1]), c2, n2);
                        const float p0 = ex2(x.x);
                        const float p1 = ex2(x.y);
                        acc[i % 4] = __fadd2_rn(acc[i % 4], make_float2(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(s_addr + h * 32, pk);  // P (bf16) over the first 64 columns of the slot
                }
                const float2 a = __fadd2_rn(__fadd2_rn(acc[0], acc[1]), __fadd2_rn(acc[2], acc[3]));
                l = l * alpha + (a.x + a.y);
                m_ref = new_ref;
                if (j > 0 && __any_sync(0xFFFFFFFFu, need)) {
                    // O holds P_0 V_0 .. P_{j-1} V_{j-1} of this unit; it must be
                    // complete.  P_{j-2} V_{j-2} already is (S_j, just read, was
                    // issued after it), so this parity wait is unambiguous.
                    if (!(ok = wait_bounded(bar(B_PVDONE), (pv_base + j - 1) & 1, abort_flag,
                                            (ROLE_SOFTMAX << 24) | (B_PVDONE << 16) | (j & 0xFFFF))))
                        break;
                    tc_fence_after_sync();
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t rr[32];
                        tmem_ld32(o_addr + q * 32, rr);
#pragma unroll
                        for (int i = 0; i < 32; ++i) rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha);
                        tmem_st32(o_addr + q * 32, rr);
                    }
                }
                tmem_st_wait();
                tc_fence_before_sync();
                warp_arrive(bar(B_PFULL + s), lane);
            }
            if (!ok) break;
            // ---- epilogue: O / l in bf16, LSE in fp32
            // The products of key tiles n-2 and n-1 may both be in flight here
            // (S of tile n-1 has its own slot, so it does not follow P_{n-2} V);
            // their completions are waited for in order, so that a parity wait
            // never runs two phases ahead of the barrier.
            for (int j = n_kv >= 2 ? n_kv - 2 : 0; ok && j < n_kv; ++j)
                ok = wait_bounded(bar(B_PVDONE), (pv_base + j) & 1, abort_flag,
                                  (ROLE_SOFTMAX << 24) | (B_PVDONE << 16) | 0xFF00 | (j & 0xFF));
            if (!ok) break;
            pv_base += n_kv;
            tc_fence_after_sync();
            const float inv_l = 1.0f / l;
            // O / l as bf16 through shared memory to TMA stores, 64 columns at
            // a time: each warp stages its own 32 rows in a 32 x 64 box (4 KB
            // of the staging area) and issues its own store, so the warps never
            // wait for one another; rows past N are clipped by the tensor map.
            uint8_t *wstage = smem + STAGE_OFF + warp * 4096;
            const uint32_t wstage_addr = sbase + STAGE_OFF + warp * 4096;
#pragma unroll 1
            for (int h = 0; h < KATOMS; ++h) {
                uint32_t ob[32];
                {
                    uint32_t rr[64];
                    tmem_ld64(o_addr + h * 64, rr);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        ob[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * inv_l, __uint_as_float(rr[2 * i + 1]) * inv_l);
                }
                if (h == KATOMS - 1) {
                    tc_fence_before_sync();
                    warp_arrive(bar(B_OFREE), lane);  // O may be overwritten
                }
                if (lane == 0) tma_store_wait_read_all();  // this warp's box is free again
                __syncwarp();
                // row `lane` of a 32-row box, 128-byte swizzle
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    *reinterpret_cast<uint4 *>(wstage + lane * 128 + ((q ^ (lane & 7)) << 4)) =
                        make_uint4(ob[4 * q], ob[4 * q + 1], ob[4 * q + 2], ob[4 * q + 3]);
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&p.tmO32, wstage_addr, h * 64, qt * BM + warp * 32, u.bh);
                    tma_store_commit();
                }
            }
            if (row < p.Nq) p.LSE[static_cast<size_t>(u.bh) * p.Nq + row] = m_ref * p.scale + logf(l);
        }
        if (lane == 0) tma_store_wait_all();  // every store of this warp has landed
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

template <int D>
static cudaError_t launch_d(const AttnParams &p, int num_sms, cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        for (auto kern : {attn_fwd256_kernel<D, false>, attn_fwd256_kernel<D, true>}) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Layout<D>::SMEM_ALLOC);
            if (err != cudaSuccess) return err;
        }
        configured_device = dev;
    }
    const long long units = static_cast<long long>(p.n_qtiles) * p.BH;
    const long long blocks = units < num_sms ? units : num_sms;  // persistent: <= one CTA per SM
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = Layout<D>::SMEM_ALLOC;
    cfg.stream = stream;
    return p.causal ? cudaLaunchKernelEx(&cfg, attn_fwd256_kernel<D, true>, p)
                    : cudaLaunchKernelEx(&cfg, attn_fwd256_kernel<D, false>, p);
}

}  // namespace fwd256

cudaError_t launch_attn_fwd256(const AttnParams &p, int num_sms, cudaStream_t stream) {
    if (num_sms < 1) return cudaErrorInvalidValue;
    return fwd256::launch_d<256>(p, num_sms, stream);
}

cudaError_t read_and_clear_fwd256_status(uint32_t *status, uint32_t *detail) {
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
