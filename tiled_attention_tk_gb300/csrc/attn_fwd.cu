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
// tiles, register accumulators, wgmma, two pipeline stages, one CTA per Q
// block) is replaced by a Blackwell one.  A persistent CTA per SM walks a
// list of work units; a unit is one head and a pair of consecutive 128-row Q
// tiles, Q0 and Q1.  Roles (512 threads, registers reallocated per
// warpgroup):
//   warp 13     TMA producer: Q0 and Q1 once per unit (each reloaded as soon
//               as the unit's last S of that tile is done), then K_j and V_j
//               into separate slots of a shared-memory ring (full/empty
//               mbarriers).
//   warp 12     MMA issuer: S_i = Q_i K_j^T (tcgen05.mma, smem x smem -> TMEM
//               fp32) and O_i += P_i V_j (P_i read from TMEM, V from smem)
//               into O_i in TMEM, ordered S0, S1, PV0, S0', PV1, S1', ... so
//               the tensor core works on one Q tile while the other tile's
//               softmax runs.  The order runs on across units: a unit's last
//               P V of a tile is followed by the next unit's first S of it.
//               Also owns TMEM.
//   warps 0-3   softmax warpgroup of Q0, warps 4-7 of Q1: thread t owns query
//               row t of its tile (TMEM lane t); reads its S row with
//               tcgen05.ld, masks the key tiles its rows see in part, takes
//               the row max, writes P = exp2(c*s - c*m_ref) as bf16 over the
//               S columns, updates l, rescales its O row only when the row
//               max has grown by more than 2^24 since the reference max was
//               set (lazy rescale; O and l always share the same reference,
//               so the result is exact), and at the end of a unit hands m_ref
//               and l to the epilogue and goes on to the next unit.
//   warps 8-11  epilogue: once a unit's last P V of a tile is done, O / l
//               (bf16) through shared memory to TMA stores, and LSE.
// TMEM (512 columns): S0/P0, S1/P1 (128 each), O0, O1 (D each).
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
#include "tk_sync.cuh"

namespace tk {


// ------------------------------------------------------------------ layout

constexpr int BM = 128;            // query rows per Q tile (one TMEM lane each)
constexpr int BN = 128;            // keys per key tile
constexpr int NUM_THREADS = 512;   // 2 softmax warpgroups, epilogue warpgroup, control warpgroup
constexpr int WARP_EPI = 8;        // warps 8..11: epilogue (warp 8 + q reads TMEM lanes 32q..32q+31)
constexpr int WARP_MMA = 12;
constexpr int WARP_TMA = 13;       // warps 14 and 15 only take part in set-up and tear-down
constexpr uint32_t TMEM_COLS = 512;
// Registers per thread after the split.  The CTA is launched with 128 per
// thread (512 threads fill the 64 K register file); the split hands the
// control and epilogue warpgroups' spare registers to the softmax warps and
// adds up to exactly the launch budget.
constexpr uint32_t REGS_SOFTMAX = 184;
constexpr uint32_t REGS_EPI = 80;
constexpr uint32_t REGS_CTRL = 64;
constexpr int LAUNCH_REGS = 128;
static_assert(2 * REGS_SOFTMAX + REGS_EPI + REGS_CTRL == 4 * LAUNCH_REGS, "register split = launch budget");
// Lazy rescale: the reference max of a row is moved (and O, l rescaled) only
// when the new row max exceeds it by more than this many powers of two.  P
// then stays below 2^24 (fine for bf16 P and fp32 l and O: the product of
// N, 2^24 and max|V| stays far from the fp32 limit for any bf16 V below
// 2^64), and O and l always share the reference, so O / l is exact.
constexpr float kRescaleLog2 = 24.0f;

template <int D>
struct Layout {
    // 128-byte swizzle atoms (TMA boxes of 64 columns) along D; for D = 32
    // and 96 the last box is half full (TMA fills the columns past D with 0).
    static constexpr int KATOMS = (D + 63) / 64;
    static constexpr uint32_t BOX_BYTES = 128 * 64 * 2;   // one TMA box: 128 rows x 64 bf16
    static constexpr uint32_t TILE_BYTES = KATOMS * BOX_BYTES;  // one 128-row tile, whole boxes
    static constexpr int NSLOTS = D > 64 ? 4 : 8;         // K/V ring slots (K_j, V_j alternate)
    static_assert(D % 32 == 0 && D >= 32 && D <= 128, "head dim 32, 64, 96 or 128");
    static constexpr uint32_t Q_OFF = 0;                  // Q tile i at Q_OFF + i * TILE_BYTES
    static constexpr uint32_t SLOT_OFF = 2 * TILE_BYTES;
    // O staging for the TMA stores: per epilogue warp, one 32-row x 64-column
    // box (4 KB) per 64 columns of D.
    static constexpr uint32_t STAGE_BOX = 32 * 64 * 2;
    static constexpr uint32_t STAGE_WARP = KATOMS * STAGE_BOX;
    static constexpr uint32_t STAGE_OFF = SLOT_OFF + NSLOTS * TILE_BYTES;
    // Row statistics (reference max, row sum) handed from a softmax
    // warpgroup to the epilogue at the end of each unit: [tile][row][2].
    static constexpr uint32_t STATS_OFF = STAGE_OFF + 4 * STAGE_WARP;
    static constexpr uint32_t BAR_OFF = STATS_OFF + 2 * BM * 8;
    // barriers
    static constexpr int B_QFULL = 0;                     // + Q tile (2)
    static constexpr int B_QEMPTY = 2;                    // + Q tile
    static constexpr int B_SLOTFULL = 4;                  // + slot
    static constexpr int B_SLOTEMPTY = B_SLOTFULL + NSLOTS;
    static constexpr int B_SFULL = B_SLOTEMPTY + NSLOTS;  // + Q tile: S in TMEM
    static constexpr int B_PFULL = B_SFULL + 2;           // + Q tile: P in TMEM (softmax -> MMA)
    static constexpr int B_ODONE = B_PFULL + 2;           // + Q tile: a unit's last P V is done
    static constexpr int B_OFREE = B_ODONE + 2;           // + Q tile: the epilogue has read O
    static constexpr int B_STFULL = B_OFREE + 2;          // + Q tile: row statistics written
    static constexpr int B_STEMPTY = B_STFULL + 2;        // + Q tile: row statistics read
    static constexpr int B_MMADONE = B_STEMPTY + 2;
    static constexpr int B_MERGE = B_MMADONE + 1;         // + epilogue warp: the other piece's block fetched
    static constexpr int NUM_BARS = B_MERGE + 4;
    // A split piece's merge fetches up to 8 blocks of 32 rows x (D + 1) fp32
    // (per Q tile and epilogue warp) into the Q and K/V buffers.
    static_assert(8u * 32u * (D + 1) * 4u <= STAGE_OFF - Q_OFF, "merge blocks fit the Q and K/V buffers");
    // No alignment slack: the dynamic shared memory of a kernel without
    // static shared memory starts 1024-byte aligned (the kernel checks).
    static constexpr uint32_t SMEM_ALLOC = BAR_OFF + NUM_BARS * 8 + 16;
    static_assert(STAGE_OFF % 1024 == 0 && STAGE_BOX % 1024 == 0, "swizzled staging boxes");
    static_assert(SMEM_ALLOC > 116u * 1024u, "one CTA per SM: each CTA holds all 512 TMEM columns");
    static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");
    // TMEM columns: S / P of Q tile i, O of Q tile i
    __host__ __device__ static constexpr uint32_t tmem_s(int i) { return static_cast<uint32_t>(i) * 128u; }
    __host__ __device__ static constexpr uint32_t tmem_o(int i) { return 256u + static_cast<uint32_t>(i) * D; }
};

// Work unit = (head bh, pair of consecutive 128-row Q tiles).  Units are
// handed to the persistent CTAs round by round; odd rounds run in reverse
// CTA order (snake) so that no CTA always gets the heaviest unit of a round.
// Without the causal mask, when the last round is less than half full its
// units are split in two pieces by key tiles (kv0 .. kv0 + nkv - 1), one
// piece per CTA, so that the last round takes half a unit's time.
struct Unit {
    int bh;
    int pair;
    int kv0;    // first key tile
    int nkv;    // key tiles of a piece (0 for a whole unit)
    int piece;  // -1: a whole unit; 0 / 1: the first / second key range of tail unit `tail`
    int tail;
};

__device__ __forceinline__ Unit unit_at(int idx, const AttnParams &p) {
    if (p.causal) {
        // Heaviest first: the last pair of every head, then the one before...
        const int r = idx / p.BH;
        return {idx % p.BH, p.n_pairs - 1 - r, 0, 0, -1, 0};
    }
    // Equal cost: the pairs of one head are adjacent, so CTAs running at
    // the same time share that head's K/V in L2.
    return {idx / p.n_pairs, idx % p.n_pairs, 0, 0, -1, 0};
}

__device__ __forceinline__ int unit_index(int round, int cta, int grid) {
    return round * grid + ((round & 1) ? grid - 1 - cta : cta);
}

// The k-th unit of this CTA (k < units_of_cta).
__device__ __forceinline__ Unit cta_unit(int k, const AttnParams &p) {
    if (p.split_pieces > 0 && k == p.split_round) {
        const int t = static_cast<int>(blockIdx.x) / 2, piece = static_cast<int>(blockIdx.x) % 2;
        Unit u = unit_at(p.split_round * static_cast<int>(gridDim.x) + t, p);
        u.kv0 = piece ? p.split_kv : 0;
        u.nkv = piece ? p.n_kvtiles - p.split_kv : p.split_kv;
        u.piece = piece;
        u.tail = t;
        return u;
    }
    return unit_at(unit_index(k, blockIdx.x, gridDim.x), p);
}

// Units this CTA runs: one per round, except that the last round may have
// none for it.
__device__ __forceinline__ int units_of_cta(const AttnParams &p) {
    if (p.split_pieces > 0) return p.split_round + (static_cast<int>(blockIdx.x) < p.split_pieces ? 1 : 0);
    const int total = p.BH * p.n_pairs;
    const int grid = gridDim.x;
    const int rounds = (total + grid - 1) / grid;
    return rounds - (unit_index(rounds - 1, blockIdx.x, grid) >= total ? 1 : 0);
}

// Key tiles Q tile `qt` of unit `u` must visit: the piece's, all of them,
// or under the causal mask those up to the last key its last row sees
// (row + offset).
__device__ __forceinline__ int kv_tiles(const Unit &u, int qt, const AttnParams &p) {
    if (u.piece >= 0) return u.nkv;
    if (!p.causal) return p.n_kvtiles;
    const int last_key = min(qt * BM + BM, p.Nq) - 1 + p.offset;
    return min(last_key / BN + 1, p.n_kvtiles);
}

// ------------------------------------------------------------------ kernel

template <int D>
__global__ void __launch_bounds__(NUM_THREADS, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
    using L = Layout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sbase = smem_addr(smem);
    if (sbase & 1023u) {  // the 128-byte-swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0) record_timeout(ROLE_LAYOUT << 24);
        return;
    }
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR_OFF);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + L::NUM_BARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float2 *stats = reinterpret_cast<float2 *>(smem + L::STATS_OFF);
    auto bar = [&](int i) { return smem_addr(&bars[i]); };

    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;
    const int my_units = units_of_cta(p);

    if (warp == WARP_MMA) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(L::B_QFULL + i), 1);
            mbar_init(bar(L::B_QEMPTY + i), 1);
            mbar_init(bar(L::B_SFULL + i), 1);
            // hand-offs from a warpgroup: one arrival per warp (after __syncwarp)
            mbar_init(bar(L::B_PFULL + i), 4);
            mbar_init(bar(L::B_ODONE + i), 1);
            mbar_init(bar(L::B_OFREE + i), 4);
            mbar_init(bar(L::B_STFULL + i), 4);
            mbar_init(bar(L::B_STEMPTY + i), 4);
        }
        for (int s = 0; s < L::NSLOTS; ++s) {
            mbar_init(bar(L::B_SLOTFULL + s), 1);
            mbar_init(bar(L::B_SLOTEMPTY + s), 1);
        }
        mbar_init(bar(L::B_MMADONE), 1);
        for (int q = 0; q < 4; ++q) mbar_init(bar(L::B_MERGE + q), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp >= WARP_MMA) {
        regs_dealloc<REGS_CTRL>();
        if (warp == WARP_TMA && lane == 0) {
            // ------------------------------------------------ TMA producer
            // Loads in the order the MMA warp consumes them: per unit K_0,
            // V_0, then Q0 and Q1 (each once the previous unit's last S of
            // that tile has completed), then K_j, V_j.
            tma_prefetch_desc(&p.tmQ);
            tma_prefetch_desc(&p.tmK);
            tma_prefetch_desc(&p.tmV);
            uint32_t loads = 0;  // K/V slot loads issued
            bool ok = true;
            for (int k = 0; ok && k < my_units; ++k) {
                const Unit u = cta_unit(k, p);
                const int n_kv = kv_tiles(u, 2 * u.pair + 1, p);
                if (k + 1 < my_units) {
                    // the next unit's Q tiles into L2: they are read once, from
                    // HBM, and the next unit's first S waits for them
                    const Unit un = cta_unit(k + 1, p);
                    for (int i = 0; i < 2 && (2 * un.pair + i) * BM < p.Nq; ++i)
                        for (int c = 0; c < L::KATOMS; ++c)
                            tma_prefetch_l2_3d(&p.tmQ, c * 64, (2 * un.pair + i) * BM, un.bh);
                }
                auto load_kv = [&](int j, int kv) -> bool {
                    const int s = loads % L::NSLOTS;
                    if (loads >= static_cast<uint32_t>(L::NSLOTS) &&
                        !wait_bounded(bar(L::B_SLOTEMPTY + s), ((loads / L::NSLOTS) - 1) & 1, abort_flag,
                                      (ROLE_PRODUCER << 24) | ((L::B_SLOTEMPTY + s) << 16) | (j & 0xFFFF)))
                        return false;
                    const uint32_t dst = sbase + L::SLOT_OFF + s * L::TILE_BYTES;
                    mbar_arrive_expect_tx(bar(L::B_SLOTFULL + s), L::TILE_BYTES);
                    for (int c = 0; c < L::KATOMS; ++c)
                        tma_load_3d(dst + c * L::BOX_BYTES, kv ? &p.tmV : &p.tmK, bar(L::B_SLOTFULL + s),
                                    c * 64, (u.kv0 + j) * BN, u.bh);
                    ++loads;
                    return true;
                };
                if (!(ok = load_kv(0, 0) && load_kv(0, 1))) break;
                for (int i = 0; ok && i < 2; ++i) {
                    if (k > 0 && !(ok = wait_bounded(bar(L::B_QEMPTY + i), (k - 1) & 1, abort_flag,
                                                     (ROLE_PRODUCER << 24) | ((L::B_QEMPTY + i) << 16) | k)))
                        break;
                    mbar_arrive_expect_tx(bar(L::B_QFULL + i), L::TILE_BYTES);
                    for (int c = 0; c < L::KATOMS; ++c)
                        tma_load_3d(sbase + L::Q_OFF + i * L::TILE_BYTES + c * L::BOX_BYTES, &p.tmQ,
                                    bar(L::B_QFULL + i), c * 64, (2 * u.pair + i) * BM, u.bh);
                }
                for (int j = 1; ok && j < n_kv; ++j) ok = load_kv(j, 0) && load_kv(j, 1);
            }
            if (!ok) {
                // Let the copies in flight land before the CTA exits.
                const uint32_t first = loads > static_cast<uint32_t>(L::NSLOTS) ? loads - L::NSLOTS : 0;
                for (uint32_t n = first; n < loads; ++n) {
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(bar(L::B_SLOTFULL + n % L::NSLOTS), (n / L::NSLOTS) & 1) &&
                           global_timer_ns() - t0 < kDrainLimitNs) {
                    }
                }
            }
        } else if (warp == WARP_MMA) {
            // ------------------------------------------------ MMA issuer
            // The whole warp runs the loop: waits and operand arithmetic are
            // warp-uniform, and one elected lane sends each block of MMAs and
            // each commit.  The stream does not stop between units: the last
            // key tile of a unit is followed at once by the next unit's first
            // S of each Q tile.  S of key tile j+1 of a Q tile is issued after
            // P V of key tile j of that tile, so its "S ready" commit also
            // tells the softmax that every earlier P V of the tile is done.
            constexpr uint32_t IDESC_S = idesc_bf16_f32(BM, BN, 0, 0);  // K-major Q and K
            constexpr uint32_t IDESC_O = idesc_bf16_f32(BM, D, 0, 1);   // P from TMEM, V MN-major
            constexpr int KS = D / 16;     // k steps of S = Q K^T
            uint32_t taken = 0;            // K/V slots consumed, in load order
            uint32_t p_seen[2] = {0, 0};   // P hand-offs consumed per Q tile
            bool ok = true;

            auto commit = [&](int b) {
                if (elect_one()) umma_commit(bar(b));
                __syncwarp();
            };
            auto take_slot = [&](uint32_t &slot) -> bool {
                slot = taken % L::NSLOTS;
                const bool r = wait_bounded(bar(L::B_SLOTFULL + slot), (taken / L::NSLOTS) & 1, abort_flag,
                                            (ROLE_MMA << 24) | ((L::B_SLOTFULL + slot) << 16) | (taken & 0xFFFF));
                ++taken;
                return r;
            };
            // S_i = Q_i K^T, then "S ready".  A k step moves 32 bytes along a
            // 128-byte swizzled row; every four steps the next 64-column box.
            auto issue_s = [&](int i, uint32_t kslot) {
                const uint64_t qd = smem_desc_sw128(sbase + L::Q_OFF + i * L::TILE_BYTES, 16, 1024);
                const uint64_t kd = smem_desc_sw128(sbase + L::SLOT_OFF + kslot * L::TILE_BYTES, 16, 1024);
                const uint32_t hi = static_cast<uint32_t>(qd >> 32);  // the same for Q and K
                uint32_t a[KS], b[KS];
#pragma unroll
                for (int k = 0; k < KS; ++k) {
                    const uint32_t off = ((k / 4) * L::BOX_BYTES + (k % 4) * 32) >> 4;
                    a[k] = static_cast<uint32_t>(qd) + off;
                    b[k] = static_cast<uint32_t>(kd) + off;
                }
                const uint32_t dst = tmem + L::tmem_s(i);
                if (elect_one()) {
                    umma_ss_steps<KS>(dst, a, hi, b, hi, IDESC_S, 0u);
                    umma_commit(bar(L::B_SFULL + i));
                }
                __syncwarp();
            };
            // O_i += P_i V over 128 keys in 8 k steps; P from the S columns
            // of TMEM (two bf16 per column), V MN-major from the slot.
            auto issue_pv = [&](int i, uint32_t vslot, bool accumulate) {
                const uint64_t vd = smem_desc_sw128(sbase + L::SLOT_OFF + vslot * L::TILE_BYTES, L::BOX_BYTES, 1024);
                const uint32_t v_lo = static_cast<uint32_t>(vd), v_hi = static_cast<uint32_t>(vd >> 32);
                if (elect_one())
                    umma_ts_x8(tmem + L::tmem_o(i), tmem + L::tmem_s(i), v_lo, v_hi, IDESC_O, accumulate ? 1u : 0u);
                __syncwarp();
            };
            auto wait_bar = [&](int b, uint32_t parity, uint32_t step) -> bool {
                return wait_bounded(bar(b), parity & 1, abort_flag, (ROLE_MMA << 24) | (b << 16) | (step & 0xFFFF));
            };
            auto wait_p = [&](int i, int j) -> bool {
                const bool r = wait_bar(L::B_PFULL + i, p_seen[i], j);
                ++p_seen[i];
                return r;
            };

            if (my_units > 0) {
                const Unit u0 = cta_unit(0, p);
                int n0 = kv_tiles(u0, 2 * u0.pair, p);
                int n1 = kv_tiles(u0, 2 * u0.pair + 1, p);  // n1 >= n0 >= 1
                uint32_t ks = 0, vs = 0;
                // The first unit's S of both Q tiles.
                ok = wait_bar(L::B_QFULL, 0, 0) && take_slot(ks);
                if (ok) {
                    tc_fence_after_sync();
                    issue_s(0, ks);
                    if (n0 == 1) commit(L::B_QEMPTY);
                    ok = wait_bar(L::B_QFULL + 1, 0, 0);
                }
                if (ok) {
                    tc_fence_after_sync();
                    issue_s(1, ks);
                    commit(L::B_SLOTEMPTY + ks);
                    if (n1 == 1) commit(L::B_QEMPTY + 1);
                }
                for (int k = 0; ok && k < my_units; ++k) {
                    const bool has_next = k + 1 < my_units;
                    int m0 = 0, m1 = 0;
                    if (has_next) {
                        const Unit un = cta_unit(k + 1, p);
                        m0 = kv_tiles(un, 2 * un.pair, p);
                        m1 = kv_tiles(un, 2 * un.pair + 1, p);
                    }
                    for (int j = 0; j < n1; ++j) {
                        const bool last = j + 1 == n1;
                        if (!(ok = take_slot(vs))) break;  // V_j
                        if (j < n0) {
                            if (!(ok = wait_p(0, j))) break;
                            // O of Q tile 0 is overwritten by the unit's first
                            // P V: the epilogue must have read the previous one.
                            if (j == 0 && k > 0 && !(ok = wait_bar(L::B_OFREE, k - 1, k))) break;
                            tc_fence_after_sync();
                            issue_pv(0, vs, j > 0);
                            if (j == n0 - 1) commit(L::B_ODONE);
                        }
                        // The next S of Q tile 0: key tile j+1 of this unit, or
                        // the next unit's first key tile.
                        if (!last) {
                            if (!(ok = take_slot(ks))) break;  // K_{j+1}
                            if (j + 1 < n0) {
                                tc_fence_after_sync();
                                issue_s(0, ks);
                                if (j + 2 == n0) commit(L::B_QEMPTY);
                            }
                        } else if (has_next) {
                            if (!(ok = take_slot(ks) && wait_bar(L::B_QFULL, k + 1, k + 1))) break;
                            tc_fence_after_sync();
                            issue_s(0, ks);
                            if (m0 == 1) commit(L::B_QEMPTY);
                        }
                        if (!(ok = wait_p(1, j))) break;
                        if (j == 0 && k > 0 && !(ok = wait_bar(L::B_OFREE + 1, k - 1, k))) break;
                        tc_fence_after_sync();
                        issue_pv(1, vs, j > 0);
                        commit(L::B_SLOTEMPTY + vs);
                        if (last) commit(L::B_ODONE + 1);
                        if (!last) {
                            issue_s(1, ks);
                            commit(L::B_SLOTEMPTY + ks);
                            if (j + 2 == n1) commit(L::B_QEMPTY + 1);
                        } else if (has_next) {
                            if (!(ok = wait_bar(L::B_QFULL + 1, k + 1, k + 1))) break;
                            tc_fence_after_sync();
                            issue_s(1, ks);
                            commit(L::B_SLOTEMPTY + ks);
                            if (m1 == 1) commit(L::B_QEMPTY + 1);
                        }
                    }
                    n0 = m0;
                    n1 = m1;
                }
            }
            // Every MMA issued so far has completed before TMEM is released.
            commit(L::B_MMADONE);
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar(L::B_MMADONE), 0) &&
                   global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
            }
        }
        __syncwarp();
    } else if (warp >= WARP_EPI) {
        // ------------------------------------------------ epilogue
        // Per unit and Q tile: O / l as bf16 through this warp's staging
        // boxes to TMA stores of its 32 rows, and LSE.  Runs while the
        // softmax warps are already on the next unit.
        regs_dealloc<REGS_EPI>();
        const int quarter = warp - WARP_EPI;           // TMEM lanes 32 * quarter ...
        const int r = quarter * 32 + lane;             // row within the Q tile
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        uint8_t *stage = smem + L::STAGE_OFF + quarter * L::STAGE_WARP;
        const uint32_t stage_addr = sbase + L::STAGE_OFF + quarter * L::STAGE_WARP;
        bool ok = true;
        auto wait_bar = [&](int b, uint32_t parity, uint32_t step) -> bool {
            return wait_bounded(bar(b), parity & 1, abort_flag, (ROLE_EPILOGUE << 24) | (b << 16) | (step & 0xFFFF));
        };
        // O / l (bf16) of this warp's 32 rows of Q tile `qt` of head `bh`,
        // from TMEM at o_addr, through its staging boxes (row `lane` of a
        // 32-row box, 128-byte swizzle) to one TMA store per 64 columns, and
        // LSE; "O free" once O has left TMEM.
        auto store_tile = [&](int tile, int qt, int bh, float inv_l, float lse) {
            // the staging boxes of this warp's previous stores are free
            if (lane == 0) tma_store_wait_read_all();
            __syncwarp();
            const uint32_t o_addr = lane_base + L::tmem_o(tile);
#pragma unroll
            for (int h = 0; h < L::KATOMS; ++h) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    if (h * 64 + half * 32 >= D) continue;  // D = 32, 96: the store clips at D
                    uint32_t rr[32];
                    tmem_ld32(o_addr + h * 64 + half * 32, rr);
                    uint32_t ob[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        ob[i] = pack_bf16x2(__uint_as_float(rr[2 * i]) * inv_l, __uint_as_float(rr[2 * i + 1]) * inv_l);
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int chunk = half * 4 + c;
                        *reinterpret_cast<uint4 *>(stage + h * L::STAGE_BOX + lane * 128 + ((chunk ^ (lane & 7)) << 4)) =
                            make_uint4(ob[4 * c], ob[4 * c + 1], ob[4 * c + 2], ob[4 * c + 3]);
                    }
                }
            }
            // All of O has left TMEM: the next unit's first P V may overwrite it.
            tc_fence_before_sync();
            warp_arrive(bar(L::B_OFREE + tile), lane);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
#pragma unroll
                for (int h = 0; h < L::KATOMS; ++h)
                    tma_store_3d(&p.tmO32, stage_addr + h * L::STAGE_BOX, h * 64, qt * BM + quarter * 32, bh);
                tma_store_commit();
            }
            const int row = qt * BM + r;
            if (row < p.Nq) p.LSE[static_cast<size_t>(bh) * p.Nq + row] = lse;
        };
        // Whole units; a split piece is always a CTA's last unit (below).
        const bool has_piece = p.split_pieces > 0 && my_units > p.split_round;
        const int n_whole = my_units - (has_piece ? 1 : 0);
        for (int k = 0; ok && k < n_whole; ++k) {
            const Unit u = cta_unit(k, p);
            for (int tile = 0; tile < 2; ++tile) {
                if (!(ok = wait_bar(L::B_STFULL + tile, k, k))) break;
                const float2 st = stats[tile * BM + r];     // (reference max, row sum)
                warp_arrive(bar(L::B_STEMPTY + tile), lane);
                if (!(ok = wait_bar(L::B_ODONE + tile, k, k))) break;
                tc_fence_after_sync();
                store_tile(tile, 2 * u.pair + tile, u.bh, 1.0f / st.y, st.x * p.scale + logf(st.y));
            }
        }
        if (ok && has_piece) {
            // ---- a piece of a split unit: both Q tiles at once.  Publish
            // O / l and LSE of this warp's rows (column-major [D][32] then 32
            // LSE, 128 contiguous bytes per column); the piece that publishes
            // second fetches the other piece's block with one bulk copy into
            // the Q / K / V buffers (idle once every MMA is done), merges into
            // its own O in TMEM (weights exp(LSE - max), unfused products and
            // sums: the same bits whichever piece merges) and alone stores O
            // and LSE.
            const int k = n_whole;
            const Unit u = cta_unit(k, p);
            constexpr uint32_t BLOCK = 32 * (D + 1);  // floats per warp block
            float2 st0 = make_float2(0.f, 1.f), st1 = make_float2(0.f, 1.f);
            ok = wait_bar(L::B_STFULL, k, k);
            if (ok) {
                st0 = stats[r];
                warp_arrive(bar(L::B_STEMPTY), lane);
                ok = wait_bar(L::B_STFULL + 1, k, k);
            }
            if (ok) {
                st1 = stats[BM + r];
                warp_arrive(bar(L::B_STEMPTY + 1), lane);
                ok = wait_bar(L::B_ODONE, k, k) && wait_bar(L::B_ODONE + 1, k, k);
            }
            unsigned merge_mask = 0;  // bit t: this warp merges Q tile t
            if (ok) {
                tc_fence_after_sync();
                float *mine = p.part + static_cast<size_t>((u.tail * 2 + u.piece) * 8 + quarter) * BLOCK + lane;
#pragma unroll 1
                for (int tile = 0; tile < 2; ++tile) {
                    const float2 st = tile ? st1 : st0;
                    const float inv_l = 1.0f / st.y;
                    float *blk = mine + tile * 4 * BLOCK;
                    const uint32_t o_addr = lane_base + L::tmem_o(tile);
#pragma unroll 1
                    for (int c = 0; c < D / 16; ++c) {
                        uint32_t rr[16];
                        tmem_ld16(o_addr + c * 16, rr);
#pragma unroll
                        for (int i = 0; i < 16; ++i) blk[(c * 16 + i) * 32] = __fmul_rn(__uint_as_float(rr[i]), inv_l);
                    }
                    blk[D * 32] = st.x * p.scale + logf(st.y);
                }
                __threadfence();
                __syncwarp();
                if (lane == 0) {
#pragma unroll 1
                    for (int tile = 0; tile < 2; ++tile)
                        if (atomicExch(p.ctr + (u.tail * 2 + tile) * 4 + quarter, p.epoch) == p.epoch)
                            merge_mask |= 1u << tile;
                }
                merge_mask = __shfl_sync(0xFFFFFFFFu, merge_mask, 0);
            }
            if (ok && merge_mask) {
                __threadfence();
                if (lane == 0) {
                    fence_proxy_async_global();
                    const uint32_t mb = bar(L::B_MERGE + quarter);
                    mbar_arrive_expect_tx(mb, __popc(merge_mask) * BLOCK * 4);
                    // the other piece's blocks: tile t at + t * 4 * BLOCK floats
                    const float *src = p.part + static_cast<size_t>((u.tail * 2 + 1 - u.piece) * 8 + quarter) * BLOCK;
#pragma unroll 1
                    for (int tile = 0; tile < 2; ++tile)
                        if (merge_mask & (1u << tile))
                            bulk_load(sbase + L::Q_OFF + (tile * 4 + quarter) * BLOCK * 4, src + tile * 4 * BLOCK,
                                      BLOCK * 4, mb);
                }
                __syncwarp();
                ok = wait_bar(L::B_MERGE + quarter, 0, k);
            }
#pragma unroll 1
            for (int tile = 0; ok && tile < 2; ++tile) {
                if (!(merge_mask & (1u << tile))) {
                    tc_fence_before_sync();
                    warp_arrive(bar(L::B_OFREE + tile), lane);
                    continue;
                }
                const float2 st = tile ? st1 : st0;
                const float *oth =
                    reinterpret_cast<const float *>(smem + L::Q_OFF + (tile * 4 + quarter) * BLOCK * 4) + lane;
                const float lse_own = st.x * p.scale + logf(st.y), lse_oth = oth[D * 32];
                const float m = fmaxf(lse_own, lse_oth);
                const float w_own = expf(lse_own - m), w_oth = expf(lse_oth - m);
                const float inv_w = 1.0f / (w_own + w_oth), inv_l = 1.0f / st.y;
                const uint32_t o_addr = lane_base + L::tmem_o(tile);
#pragma unroll 1
                for (int c = 0; c < D / 16; ++c) {
                    uint32_t rr[16];
                    tmem_ld16(o_addr + c * 16, rr);
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        rr[i] = __float_as_uint(__fmul_rn(
                            __fadd_rn(__fmul_rn(w_own, __fmul_rn(__uint_as_float(rr[i]), inv_l)),
                                      __fmul_rn(w_oth, oth[(c * 16 + i) * 32])),
                            inv_w));
                    tmem_st16(o_addr + c * 16, rr);
                }
                tmem_st_wait();
                // TMEM now holds the merged, normalised O
                store_tile(tile, 2 * u.pair + tile, u.bh, 1.0f, m + logf(w_own + w_oth));
            }
        }
        if (lane == 0) tma_store_wait_all();  // every store of this warp has landed
        __syncwarp();
    } else {
        // ------------------------------------------------ softmax / correction
        regs_alloc<REGS_SOFTMAX>();
        const int tile = warp / 4;                 // which Q tile of the unit this warpgroup owns
        const int t = threadIdx.x % 128;           // row within the tile == TMEM lane
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
        const uint32_t s_addr = lane_base + L::tmem_s(tile);
        const uint32_t o_addr = lane_base + L::tmem_o(tile);
        const float c = p.scale_log2e;
        uint32_t s_seen = 0;    // S hand-offs consumed
        bool ok = true;
        for (int k = 0; ok && k < my_units; ++k) {
            const Unit u = cta_unit(k, p);
            const int qt = 2 * u.pair + tile;
            const int row = qt * BM + t;
            const int n_kv = kv_tiles(u, qt, p);
            float m_ref = -INFINITY;  // reference max of raw scores (lazy)
            float l = 0.0f;           // sum of exp2(c * (s - m_ref))
            for (int j = 0; j < n_kv; ++j) {
                if (!(ok = wait_bounded(bar(L::B_SFULL + tile), s_seen & 1, abort_flag,
                                        (ROLE_SOFTMAX << 24) | ((L::B_SFULL + tile) << 16) | (j & 0xFFFF))))
                    break;
                ++s_seen;
                tc_fence_after_sync();
                // The whole S row: two 64-column TMEM loads, one wait.
                uint32_t sr[BN];
                tmem_ld64_async(s_addr, sr);
                tmem_ld64_async(s_addr + 64, sr + 64);
                tmem_ld_wait();
                reg_fence(sr);
                float s[BN];
#pragma unroll
                for (int i = 0; i < BN; ++i) s[i] = __uint_as_float(sr[i]);
                const int jg = u.kv0 + j;  // key tile within the head
                if ((jg + 1) * BN > p.Nkv || (p.causal && (jg + 1) * BN > qt * BM + p.offset + 1)) {
                    // A key tile that some row of this Q tile does not see in
                    // full: the ragged tail (keys >= Nkv) and, under the
                    // causal mask, keys past row + offset take -inf.
                    const int limit = p.causal ? min(row + 1 + p.offset, p.Nkv) : p.Nkv;
                    const int kmax = limit - jg * BN;
#pragma unroll
                    for (int i = 0; i < BN; ++i) s[i] = (i < kmax) ? s[i] : -INFINITY;
                }
                // Row max: eight independent chains of three-input maxima.
                float mx8[8];
#pragma unroll
                for (int k8 = 0; k8 < 8; ++k8) {
                    float a = s[k8];
#pragma unroll
                    for (int t2 = 1; t2 < 15; t2 += 2) a = fmax3(a, s[k8 + 8 * t2], s[k8 + 8 * (t2 + 1)]);
                    mx8[k8] = fmaxf(a, s[k8 + 120]);
                }
                const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]),
                                       fmax3(mx8[6], mx8[7], m_ref));
                const bool need = (mx - m_ref) * c > kRescaleLog2;  // true when m_ref = -inf
                const float new_ref = need ? mx : m_ref;
                const float alpha = need ? ex2((m_ref - mx) * c) : 1.0f;
                const float neg = (new_ref == -INFINITY) ? 0.0f : -new_ref * c;
                // P = exp2(c*s - c*m_ref): packed FMA for the argument, MUFU
                // ex2, packed adds for the row sum, bf16x2 packing for TMEM.
                const float2 c2 = make_float2(c, c);
                const float2 n2 = make_float2(neg, neg);
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // two halves keep the register peak low
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int e = h * 64 + 2 * i;
                        const float2 x = __ffma2_rn(make_float2(s[e], s[e + 1]), c2, n2);
                        const float p0 = ex2(x.x);
                        const float p1 = ex2(x.y);
                        acc[i % 4] = __fadd2_rn(acc[i % 4], make_float2(p0, p1));
                        pk[i] = pack_bf16x2(p0, p1);
                    }
                    tmem_st32(s_addr + h * 32, pk);  // P (bf16) over the first 64 S columns
                }
                const float2 a01 = __fadd2_rn(acc[0], acc[1]);
                const float2 a23 = __fadd2_rn(acc[2], acc[3]);
                const float2 a = __fadd2_rn(a01, a23);
                l = l * alpha + (a.x + a.y);
                m_ref = new_ref;
                if (j > 0 && __any_sync(0xFFFFFFFFu, need)) {
                    // S_j was issued after P V of key tile j-1: O is complete.
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
                warp_arrive(bar(L::B_PFULL + tile), lane);
            }
            if (!ok) break;
            // Row statistics to the epilogue (once it has read the last ones).
            if (k > 0 && !(ok = wait_bounded(bar(L::B_STEMPTY + tile), (k - 1) & 1, abort_flag,
                                             (ROLE_SOFTMAX << 24) | ((L::B_STEMPTY + tile) << 16) | (k & 0xFFFF))))
                break;
            stats[tile * BM + t] = make_float2(m_ref, l);
            warp_arrive(bar(L::B_STFULL + tile), lane);
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
static cudaError_t launch_d(const AttnParams &p, int num_sms, cudaStream_t stream) {
    using L = Layout<D>;
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        // The register split of the kernel's warpgroups adds up to the
        // launch budget of 128 registers per thread; a build that launched
        // with fewer would leave the growing warpgroup waiting, so it is
        // refused here instead.
        cudaFuncAttributes attr;
        err = cudaFuncGetAttributes(&attr, attn_fwd_kernel<D>);
        if (err != cudaSuccess) return err;
        if (attr.numRegs != LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        err = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   L::SMEM_ALLOC);
        if (err != cudaSuccess) return err;
        configured_device = dev;
    }
    const long long units = static_cast<long long>(p.n_pairs) * p.BH;
    const long long blocks = units < num_sms ? units : num_sms;  // persistent: <= one CTA per SM
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM_ALLOC;
    cfg.stream = stream;
    cfg.attrs = nullptr;
    cfg.numAttrs = 0;
    return cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D>, p);
}

cudaError_t launch_attn_fwd(int D, const AttnParams &p, int num_sms, cudaStream_t stream) {
    if (num_sms < 1) return cudaErrorInvalidValue;
    if (D == 32) return launch_d<32>(p, num_sms, stream);
    if (D == 64) return launch_d<64>(p, num_sms, stream);
    if (D == 96) return launch_d<96>(p, num_sms, stream);
    if (D == 128) return launch_d<128>(p, num_sms, stream);
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
