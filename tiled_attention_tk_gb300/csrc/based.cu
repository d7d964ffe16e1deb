// based.cu -- causal Based linear attention on tcgen05 (sm_103a, GB300).
//
// The pages list "Based Linear Attention" among the kernels built with the
// same tiles (thebeat.tech "ThunderKittens 2.0", New Kernels) without a
// formula.  The reading taken is the Based feature map, the second-order
// Taylor expansion of exp, on query/key features of dimension 16:
//
//   w_ij  = 1 + s_ij + s_ij^2 / 2,  s_ij = scale <q_i, k_j>   (= phi(q_i) . phi(k_j))
//   O_i   = sum_{j<=i} w_ij v_j / DEN_i,   DEN_i = sum_{j<=i} w_ij      (v_j in R^64)
//
// with phi(x) = [1, sqrt(scale) x, scale/sqrt(2) x_a^2, scale x_a x_b (a < b)]
// (153 features, padded with zeros to F = 160).  The kernel runs the chunked
// linear form: one CTA per (batch, head) walks the sequence in chunks of 128
// rows and keeps the running state
//
//   S^T = sum_j [v_j | 1] phi(k_j)^T      (65 live rows x 160 features, fp32 in TMEM)
//
// so that per chunk c, for the rows i of the chunk:
//   intra:  [num | den]_i  = sum_{j in c, j<=i} w_ij [v_j | 1]     (tensor core: P [V | 1])
//   inter:  [num | den]_i += phi(q_i) . S_{<c}                      (tensor core: phi(Q) S)
//   state:  S^T += [V | 1]^T phi(K)                                 (tensor core)
//   O_i = num_i / den_i.
//
// 512 threads: two compute warpgroups over the same 128 rows (row i of the
// chunk = TMEM lane i; they split the columns of every step), an epilogue
// warpgroup that writes O and DEN, a TMA warp and an MMA warp (and two warps
// that only take part in set-up).  The tensor core forms chunk c+1's Q K^T right after chunk
// c's P [V|1], so the compute warps form P of c+1 while the rest of chunk c's
// products run.  Q and K arrive as 128 x 64 boxes of which the first
// 16 columns are the tensor (the rest zero-filled by TMA), so the same
// 128-byte-swizzled layouts and descriptors as the attention kernels serve
// every operand.  The "1" column is a constant shared-memory box.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "tk_attn.h"
#include "tk_attn_internal.h"
#include "tk_ptx.cuh"
#include "tk_sync.cuh"

namespace tk {
namespace based {

constexpr int C = 128;             // rows per chunk
constexpr int DQK = 16;
constexpr int DV = 64;
constexpr int F = 160;             // feature columns (153 live; ten 16-feature steps)
constexpr int NV = 80;             // [num | den] columns (64 + 1, padded to a multiple of 16)
constexpr int NUM_THREADS = 320;   // the segment-state kernel: 8 compute warps, TMA warp, MMA warp
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
// The main kernel: 8 compute warps, an epilogue warpgroup that writes O, and a
// control warpgroup (TMA warp, MMA warp, two set-up warps).  Registers per
// thread and warpgroup (setmaxnreg) add up to the launch budget of 128: the
// host refuses a build compiled to any other count, else the growing
// warpgroups would wait for registers.
constexpr int MAIN_THREADS = 512;
constexpr int M_WARP_EPI = 8;
constexpr int M_WARP_TMA = 12;
constexpr int M_WARP_MMA = 13;
constexpr int LAUNCH_REGS = 128;
constexpr uint32_t REGS_COMPUTE = 168;
constexpr uint32_t REGS_EPI = 88;
constexpr uint32_t REGS_CTRL = 88;
static_assert(2 * REGS_COMPUTE + REGS_EPI + REGS_CTRL == 4 * LAUNCH_REGS, "register split = launch budget");
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ROLE_BASED_PRODUCER = 12;
constexpr uint32_t ROLE_BASED_MMA = 13;
constexpr uint32_t ROLE_BASED_COMPUTE = 14;

constexpr uint32_t BOX = 128 * 128;                   // 128 rows x 128 bytes
constexpr uint32_t QK_OFF = 0;                        // buffer b: Q, K boxes at + b * 2 * BOX
constexpr uint32_t V_OFF = QK_OFF + 4 * BOX;          // buffer b: V box at + b * BOX
constexpr uint32_t ONES_OFF = V_OFF + 2 * BOX;        // [row][col]: 1 in column 0
constexpr uint32_t PHIK_OFF = ONES_OFF + BOX;         // phi(K): 128 rows x 160 features (3 boxes, the last half used)
constexpr uint32_t SBOX = NV * 128;                   // 80 rows x 128 bytes
constexpr uint32_t SPREV_OFF = PHIK_OFF + 3 * BOX;    // S (bf16, K-major): 80 rows x 160 features (3 boxes, the last half used)
constexpr uint32_t OBOX = 32 * DV;                    // 32 rows x 64 bytes: one warp's O columns
constexpr uint32_t OST_OFF = SPREV_OFF + 3 * SBOX;    // O staging: two 32 x 32 boxes per epilogue warp
constexpr uint32_t BAR_OFF = OST_OFF + 8 * OBOX;
constexpr int B_QKFULL = 0;        // + buffer (2): Q, K of a chunk loaded
constexpr int B_QKEMPTY = 2;       // + buffer (2): its Q K^T and feature maps formed (8 warps)
constexpr int B_VFULL = 4;         // + buffer (2): V of a chunk loaded
constexpr int B_VEMPTY = 6;        // + buffer (2): its P [V|1] and state products done
constexpr int B_SFULL = 8;         // Q K^T in TMEM
constexpr int B_SREAD = 9;         // both groups hold their half of S in registers (8 warps)
constexpr int B_PREADY = 10;       // P in TMEM (8 warps)
constexpr int B_PHIQREADY = 11;    // phi(Q) in TMEM, the bf16 state of the chunks before in smem (8 warps)
constexpr int B_PHIKREADY = 12;    // phi(K) in smem (8 warps)
constexpr int B_ODONE = 13;        // [num | den] of the chunk complete
constexpr int B_STDONE = 14;       // state product done
constexpr int B_MMADONE = 15;
constexpr int B_OFREE = 16;        // [num | den] of the chunk read out (epilogue, 4)
constexpr int NUM_BARS = 17;
constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");
static_assert(SBOX % 1024 == 0 && SPREV_OFF % 1024 == 0 && OST_OFF % 1024 == 0,
              "swizzled boxes need 1024-byte alignment");

constexpr uint32_t T_S = 0;        // Q K^T (fp32, 128 cols)
constexpr uint32_t T_PHIQ = 128;   // phi(Q) bf16: 80 cols
constexpr uint32_t T_O = 208;      // [num | den] fp32: 80 cols
constexpr uint32_t T_ST = 288;     // S^T fp32: 160 cols (lane = value column, 64 = the "1" row)
constexpr uint32_t T_P = 448;      // P bf16: 64 cols, apart from S so the next S can be formed early
static_assert(T_P + 64 <= TMEM_COLS, "TMEM plan");

__device__ __forceinline__ uint32_t sw128(uint32_t box, int r, int c) { return box + r * 128 + ((c ^ (r & 7)) << 4); }

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Two bf16 products in one instruction (each rounded to nearest even).
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// phi(x) as 80 packed bf16 pairs, from x as 8 packed bf16 pairs
// w[n] = (x_2n, x_2n+1).  The order of the features is the kernel's own
// (phi(q) . phi(k) does not depend on it, and every phi here comes from this
// function):
//   word 0        (1, 0)
//   words 1..8    r (x_2n, x_2n+1)
//   words 9..16   h (x_2n^2, x_2n+1^2)
//   words 17..20  g (x_4n x_4n+1, x_4n+2 x_4n+3)
//   words 21..76  g x_a (x_2m, x_2m+1) for a = 0..13 and every m with 2m > a,
//                 a-major: the 112 products x_a x_b (a < b) not above
//   words 77..79  0
// The first 21 words are formed in fp32 and rounded once.  Each of the other
// 56 is one bf16x2 multiply of bf16(g x_a), broadcast to both halves, by the
// input pair w[m], so those features carry two roundings.  Every index is a
// compile-time constant once the loops are unrolled.
__device__ __forceinline__ void phi_words(const uint32_t (&w)[DQK / 2], float r, float h, float g,
                                          uint32_t (&pk)[F / 2]) {
    float x[DQK];
#pragma unroll
    for (int n = 0; n < DQK / 2; ++n) {
        x[2 * n] = __uint_as_float(w[n] << 16);
        x[2 * n + 1] = __uint_as_float(w[n] & 0xFFFF0000u);
    }
    pk[0] = pack_bf16x2(1.0f, 0.0f);
    const float2 r2 = make_float2(r, r), h2 = make_float2(h, h), g2 = make_float2(g, g);
    float y[DQK];  // g x_a in fp32
#pragma unroll
    for (int n = 0; n < DQK / 2; ++n) {
        const float2 xp = make_float2(x[2 * n], x[2 * n + 1]);
        const float2 lin = __fmul2_rn(r2, xp);
        const float2 sq = __fmul2_rn(__fmul2_rn(h2, xp), xp);
        const float2 yp = __fmul2_rn(g2, xp);
        pk[1 + n] = pack_bf16x2(lin.x, lin.y);
        pk[9 + n] = pack_bf16x2(sq.x, sq.y);
        y[2 * n] = yp.x;
        y[2 * n + 1] = yp.y;
    }
#pragma unroll
    for (int n = 0; n < DQK / 4; ++n) {
        const float2 u = __fmul2_rn(make_float2(y[4 * n], y[4 * n + 2]), make_float2(x[4 * n + 1], x[4 * n + 3]));
        pk[17 + n] = pack_bf16x2(u.x, u.y);
    }
    int k = 21;
#pragma unroll
    for (int a = 0; a < DQK - 2; ++a) {
        const uint32_t ya = pack_bf16x2(y[a], y[a]);
#pragma unroll
        for (int m = a / 2 + 1; m < DQK / 2; ++m) pk[k++] = mul_bf16x2(ya, w[m]);
    }
#pragma unroll
    for (; k < F / 2; ++k) pk[k] = 0u;
}

// phi of one row (16 features from a swizzled box) into the feature parts of
// PARTS (bit k = features 64k .. 64k+63; part 2 holds 128..159): into TMEM as
// the A operand of the inter product, or into row r of the phi(K) boxes.
// `live` false zeroes the row (a key past N, the constant feature included).
template <int PARTS, bool TO_TMEM>
__device__ __forceinline__ void phi_store(uint32_t box16, int r, bool live, float rs, float hs, float gs,
                                          uint32_t dst) {
    const uint4 lo = ld_shared_v4(sw128(box16, r, 0));
    const uint4 hi = ld_shared_v4(sw128(box16, r, 1));
    uint32_t w[DQK / 2] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    if (!live) {
#pragma unroll
        for (int n = 0; n < DQK / 2; ++n) w[n] = 0u;
    }
    uint32_t pk[F / 2];
    phi_words(w, rs, hs, gs, pk);
    if (!live) pk[0] = 0u;
#pragma unroll
    for (int part = 0; part < 3; ++part) {
        if (!(PARTS & (1 << part))) continue;
        if constexpr (TO_TMEM) {
            if (part < 2)
                tmem_st32(dst + part * 32, *reinterpret_cast<const uint32_t(*)[32]>(pk + 32 * part));
            else
                tmem_st16(dst + 64, *reinterpret_cast<const uint32_t(*)[16]>(pk + 64));
        } else {
            const uint32_t box = dst + part * BOX;
#pragma unroll
            for (int q = 0; q < (part < 2 ? 8 : 4); ++q)
                st_shared_v4(sw128(box, r, q), pk[32 * part + 4 * q], pk[32 * part + 4 * q + 1],
                             pk[32 * part + 4 * q + 2], pk[32 * part + 4 * q + 3]);
        }
    }
}

// O_i = num_i / den_i for the warp's 32 rows and its group's 32 columns of
// the [num | den] accumulator: bf16 into the warp's staging box (64-byte
// swizzle), then one TMA store by lane 0 (rows past N are clipped).  DEN is
// written when `den_out` is set.
__device__ __forceinline__ void write_o(uint32_t lane_taddr, int grp, int lane, uint32_t obox, const CUtensorMap *tmO,
                                        int row0, int bh, int N, float *den_out) {
    uint32_t o[32], d[16];
    tmem_ld32(lane_taddr + T_O + grp * 32, o);
    tmem_ld16(lane_taddr + T_O + 64, d);
    const float den = __uint_as_float(d[0]);
    const float inv = 1.0f / den;
    const float2 inv2 = make_float2(inv, inv);
    if (lane == 0) tma_store_wait_read_all();  // this warp's previous store has read the box
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const float2 v =
                __fmul2_rn(make_float2(__uint_as_float(o[8 * q + 2 * t]), __uint_as_float(o[8 * q + 2 * t + 1])), inv2);
            w[t] = pack_bf16x2(v.x, v.y);
        }
        // 64-byte swizzle: 16-byte chunk q of row `lane` at chunk q ^ ((lane >> 1) & 3)
        st_shared_v4(obox + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4), w[0], w[1], w[2], w[3]);
    }
    if (den_out && row0 + lane < N) *den_out = den;
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0 && row0 < N) {
        tma_store_3d(tmO, obox, grp * 32, row0, bh);
        tma_store_commit();
    }
}

// A piece of work: chunks c0 .. c0 + n - 1 of head bh, starting from no
// state, from the sum of the partial states of the segments before it
// (carry 1, from the segment-state pass), or from the state another CTA
// published for the chunks before c0 (carry 2); `publish` stores the state
// after the piece's last chunk for the CTA that walks the rest of the head.
struct Piece {
    int bh, c0, n, carry, publish, seg;
};

// MODE 0: one CTA per head.  MODE 1: one CTA per segment, after the
// segment-state pass.  MODE 2 (balanced): the heads' chunks, laid end to end,
// are cut into one run per CTA (at least a head long, so a run holds the end
// of one head, whole heads and the start of another); a CTA walks the start
// of the head it ends in first and publishes that state, then its whole
// heads, then the end of the head it starts in, from the state the CTA before
// it published.  Compiled apart, so the whole-head kernel carries none of the
// bookkeeping.
template <int MODE>
__global__ void __launch_bounds__(MAIN_THREADS, 1) based_kernel(const __grid_constant__ BasedParams p) {
    constexpr bool SEG = MODE == 1;
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
    // This CTA's pieces, in the order it walks them.  Chunk indices inside a
    // piece are local to it; the barriers' phases run on over all pieces
    // (g = chunks of earlier pieces + c).
    const int n_ch = (p.N + C - 1) / C;
    long long run_s = 0, run_e = 0;
    if (MODE == 2) {
        const long long total = static_cast<long long>(p.BH) * n_ch;
        run_s = static_cast<long long>(blockIdx.x) * total / gridDim.x;
        run_e = static_cast<long long>(blockIdx.x + 1) * total / gridDim.x;
    }
    const int hs = static_cast<int>(run_s / n_ch), cs = static_cast<int>(run_s % n_ch);
    const int he = static_cast<int>(run_e / n_ch), ce = static_cast<int>(run_e % n_ch);
    const int h_first = cs != 0 ? hs + 1 : hs;  // first whole head
    const int n_pieces = MODE == 2 ? (ce != 0) + (he - h_first) + (cs != 0) : 1;
    auto piece = [&](int k) -> Piece {
        if (MODE == 0) return {static_cast<int>(blockIdx.x), 0, n_ch, 0, 0, 0};
        if (MODE == 1) {
            const int seg = static_cast<int>(blockIdx.x) % p.n_seg;
            const int c0 = seg * p.seg_chunks;
            return {static_cast<int>(blockIdx.x) / p.n_seg, c0, min(p.seg_chunks, n_ch - c0), seg > 0 ? 1 : 0, 0, seg};
        }
        if (ce != 0 && k == 0) return {he, 0, ce, 0, 1, 0};  // the start of the head the run ends in
        const int kk = k - (ce != 0);
        if (kk < he - h_first) return {h_first + kk, 0, n_ch, 0, 0, 0};
        return {hs, cs, n_ch - cs, 2, 0, 0};  // the end of the head the run starts in
    };

    if (warp == M_WARP_MMA) {
        tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(B_QKFULL + b), 1);
            mbar_init(bar(B_QKEMPTY + b), 8);
            mbar_init(bar(B_VFULL + b), 1);
            mbar_init(bar(B_VEMPTY + b), 1);
        }
        mbar_init(bar(B_SFULL), 1);
        mbar_init(bar(B_SREAD), 8);
        mbar_init(bar(B_PREADY), 8);
        mbar_init(bar(B_PHIQREADY), 8);
        mbar_init(bar(B_PHIKREADY), 8);
        mbar_init(bar(B_ODONE), 1);
        mbar_init(bar(B_STDONE), 1);
        mbar_init(bar(B_MMADONE), 1);
        mbar_init(bar(B_OFREE), 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp < 4) {
        // the constant box: 1 in column 0 of every row, 0 elsewhere
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

    if (warp >= M_WARP_TMA) {
        regs_dealloc<REGS_CTRL>();
        if (warp == M_WARP_TMA) {
            // ------------------------------------------------ TMA producer
            if (lane == 0) {
                tma_prefetch_desc(&p.tmQ);
                tma_prefetch_desc(&p.tmK);
                tma_prefetch_desc(&p.tmV);
                // Q, K of chunk c into buffer c & 1 once chunk c-2's Q K^T and
                // feature maps are formed (early, so the next S never waits on
                // HBM); V of chunk c once chunk c-2's products are done.
                int qk_issued = 0, v_issued = 0;
                bool ok = true;
                int g0 = 0;  // chunks of earlier pieces
                for (int k = 0; ok && k < n_pieces; ++k) {
                const Piece pc = piece(k);
                for (int c = 0; c < pc.n; ++c) {
                    const int g = g0 + c;
                    const int b = g & 1;
                    if (g >= 2 && !(ok = wait_bounded(bar(B_QKEMPTY + b), ((g >> 1) - 1) & 1, abort_flag,
                                                      (ROLE_BASED_PRODUCER << 24) | ((B_QKEMPTY + b) << 16) | (g & 0xFFFF))))
                        break;
                    // Q and K boxes carry 16 real columns; TMA fills the rest with 0
                    // but still counts the full box.
                    const uint32_t dst = sbase + QK_OFF + b * 2 * BOX;
                    mbar_arrive_expect_tx(bar(B_QKFULL + b), 2 * BOX);
                    tma_load_3d(dst, &p.tmQ, bar(B_QKFULL + b), 0, (pc.c0 + c) * C, pc.bh);
                    tma_load_3d(dst + BOX, &p.tmK, bar(B_QKFULL + b), 0, (pc.c0 + c) * C, pc.bh);
                    ++qk_issued;
                    if (g >= 2 && !(ok = wait_bounded(bar(B_VEMPTY + b), ((g >> 1) - 1) & 1, abort_flag,
                                                      (ROLE_BASED_PRODUCER << 24) | ((B_VEMPTY + b) << 16) | (g & 0xFFFF))))
                        break;
                    mbar_arrive_expect_tx(bar(B_VFULL + b), BOX);
                    tma_load_3d(sbase + V_OFF + b * BOX, &p.tmV, bar(B_VFULL + b), 0, (pc.c0 + c) * C, pc.bh);
                    ++v_issued;
                }
                g0 += pc.n;
                }
                if (!ok) {
                    // let the loads in flight land before the CTA's shared memory goes away
                    const uint64_t t0 = global_timer_ns();
                    for (int j = qk_issued - 2 < 0 ? 0 : qk_issued - 2; j < qk_issued; ++j)
                        while (!mbar_try_wait(bar(B_QKFULL + (j & 1)), (j >> 1) & 1) && global_timer_ns() - t0 < kDrainLimitNs) {
                        }
                    for (int j = v_issued - 2 < 0 ? 0 : v_issued - 2; j < v_issued; ++j)
                        while (!mbar_try_wait(bar(B_VFULL + (j & 1)), (j >> 1) & 1) && global_timer_ns() - t0 < kDrainLimitNs) {
                        }
                }
            }
            __syncwarp();
        } else if (warp == M_WARP_MMA) {
            // ------------------------------------------------ MMA issuer
            // The whole warp runs the loop (operands stay warp-uniform); one
            // elected lane sends each block of products and each commit.
            {
                constexpr uint32_t ID_S = idesc_bf16_f32(C, C, 0, 0);       // Q K^T
                constexpr uint32_t ID_INTRA = idesc_bf16_f32(C, NV, 0, 1);  // P [V | 1]: A in TMEM, B MN-major
                constexpr uint32_t ID_INTER = idesc_bf16_f32(C, NV, 0, 0);  // phi(Q) S: A in TMEM, B K-major
                constexpr uint32_t ID_STATE = idesc_bf16_f32(C, F, 1, 1);   // [V | 1]^T phi(K): both MN-major
                // Per chunk c: Q K^T of chunk c+1 as soon as both groups hold S of
                // chunk c in registers; then P [V|1], phi(Q) S_{<c} and the state
                // update, each once its operands are in place.
                auto issue_s = [&](int c) {
                    const uint32_t qb = sbase + QK_OFF + (c & 1) * 2 * BOX;
                    const uint64_t qd = smem_desc_sw128(qb, 16, 1024), kd = smem_desc_sw128(qb + BOX, 16, 1024);
                    if (elect_one()) {
                        umma_ss(tmem + T_S, qd, kd, ID_S, 0);
                        umma_commit(bar(B_SFULL));
                    }
                    __syncwarp();
                };
                bool ok = true;
                int g0 = 0;  // chunks of earlier pieces
                for (int k = 0; ok && k < n_pieces; ++k) {
                const Piece pc = piece(k);
                const bool has_prev = pc.carry != 0;
                if (k == 0) {  // the first S (a later piece's was issued during the piece before it)
                    ok = wait_bounded(bar(B_QKFULL + (g0 & 1)), (g0 >> 1) & 1, abort_flag,
                                      (ROLE_BASED_MMA << 24) | ((B_QKFULL + (g0 & 1)) << 16) | (g0 & 0xFFFF));
                    if (ok) {
                        tc_fence_after_sync();
                        issue_s(g0);
                    }
                }
                for (int c = 0; ok && c < pc.n; ++c) {
                    const int g = g0 + c;
                    const int b = g & 1;
                    const uint32_t ph = g & 1;
                    const uint32_t vb = sbase + V_OFF + b * BOX;
                    if (!(ok = wait_bounded(bar(B_SREAD), ph, abort_flag,
                                            (ROLE_BASED_MMA << 24) | (B_SREAD << 16) | (g & 0xFFFF))))
                        break;
                    if (c + 1 < pc.n || k + 1 < n_pieces) {  // S of the next chunk, in this piece or the next
                        if (!(ok = wait_bounded(bar(B_QKFULL + (b ^ 1)), ((g + 1) >> 1) & 1, abort_flag,
                                                (ROLE_BASED_MMA << 24) | ((B_QKFULL + (b ^ 1)) << 16) | ((g + 1) & 0xFFFF))))
                            break;
                        tc_fence_after_sync();
                        issue_s(g + 1);
                    }
                    if (!(ok = wait_bounded(bar(B_PREADY), ph, abort_flag,
                                            (ROLE_BASED_MMA << 24) | (B_PREADY << 16) | (g & 0xFFFF))))
                        break;
                    if (!(ok = wait_bounded(bar(B_VFULL + b), (g >> 1) & 1, abort_flag,
                                            (ROLE_BASED_MMA << 24) | ((B_VFULL + b) << 16) | (g & 0xFFFF))))
                        break;
                    // the epilogue has read the previous chunk's [num | den]
                    if (g > 0 && !(ok = wait_bounded(bar(B_OFREE), (g - 1) & 1, abort_flag,
                                                     (ROLE_BASED_MMA << 24) | (B_OFREE << 16) | (g & 0xFFFF))))
                        break;
                    tc_fence_after_sync();
                    // intra: [num | den] = P [V | 1]; 16 chunk rows per step.  Descriptors
                    // are formed once per operand; a k step adds its compile-time
                    // offset to the start-address field (no carry: smem < 256 KB).
                    const uint64_t v1d = smem_desc_sw128(vb, ONES_OFF - (vb - sbase), 1024);
                    const uint32_t v1_lo = static_cast<uint32_t>(v1d), hi = static_cast<uint32_t>(v1d >> 32);
                    uint32_t v1v[C / 16];
    #pragma unroll
                    for (int k = 0; k < C / 16; ++k) v1v[k] = v1_lo + ((k * 2048) >> 4);
                    if (elect_one()) umma_ts_steps<C / 16, 8>(tmem + T_O, tmem + T_P, v1v, hi, ID_INTRA, 0u);
                    __syncwarp();
                    // inter: [num | den] += phi(Q) S_{<c}; 16 features per step
                    if (!(ok = wait_bounded(bar(B_PHIQREADY), ph, abort_flag,
                                            (ROLE_BASED_MMA << 24) | (B_PHIQREADY << 16) | (g & 0xFFFF))))
                        break;
                    tc_fence_after_sync();
                    const uint32_t s_lo = static_cast<uint32_t>(smem_desc_sw128(sbase + SPREV_OFF, 16, 1024));
                    uint32_t sv[F / 16];
    #pragma unroll
                    for (int k = 0; k < F / 16; ++k) sv[k] = s_lo + (((k / 4) * SBOX + (k % 4) * 32) >> 4);
                    if (elect_one()) {
                        if (c > 0 || has_prev) umma_ts_steps<F / 16, 8>(tmem + T_O, tmem + T_PHIQ, sv, hi, ID_INTER, 1u);
                        umma_commit(bar(B_ODONE));
                    }
                    __syncwarp();
                    // state: S^T += [V | 1]^T phi(K); 16 chunk rows per step
                    if (!(ok = wait_bounded(bar(B_PHIKREADY), ph, abort_flag,
                                            (ROLE_BASED_MMA << 24) | (B_PHIKREADY << 16) | (g & 0xFFFF))))
                        break;
                    tc_fence_after_sync();
                    const uint32_t pk_lo = static_cast<uint32_t>(smem_desc_sw128(sbase + PHIK_OFF, BOX, 1024));
                    uint32_t pkv[C / 16];
    #pragma unroll
                    for (int k = 0; k < C / 16; ++k) pkv[k] = pk_lo + ((k * 2048) >> 4);
                    if (elect_one()) {
                        umma_ss_steps<C / 16>(tmem + T_ST, v1v, hi, pkv, hi, ID_STATE, (c > 0 || has_prev) ? 1u : 0u);
                        umma_commit(bar(B_STDONE));
                        umma_commit(bar(B_VEMPTY + b));
                    }
                    __syncwarp();
                }
                g0 += pc.n;
                }
                if (elect_one()) umma_commit(bar(B_MMADONE));
                __syncwarp();
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(bar(B_MMADONE), 0) && global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
                }
            }
            __syncwarp();
        }
    } else if (warp >= M_WARP_EPI) {
        // ------------------------------------------------ epilogue warps
        // O = num / den and DEN of every chunk, once its [num | den] is
        // complete: warp w writes rows 32w .. 32w + 31 of the chunk, both
        // 32-column halves, and releases the accumulator for the next chunk's
        // first product.
        regs_dealloc<REGS_EPI>();
        const int ew = warp - M_WARP_EPI;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(ew * 32) << 16);
        const uint32_t obox0 = sbase + OST_OFF + (2 * ew) * OBOX, obox1 = obox0 + OBOX;
        bool ok = true;
        int g0 = 0;  // chunks of earlier pieces
        for (int k = 0; ok && k < n_pieces; ++k) {
            const Piece pc = piece(k);
            for (int c = 0; c < pc.n; ++c) {
                const int gc = g0 + c;
                if (!(ok = wait_bounded(bar(B_ODONE), gc & 1, abort_flag,
                                        (ROLE_BASED_COMPUTE << 24) | (B_ODONE << 16) | (gc & 0xFFFF))))
                    break;
                tc_fence_after_sync();
                const int row0 = (pc.c0 + c) * C + ew * 32;  // this warp's first row in the head
                write_o(lane_base, 0, lane, obox0, &p.tmO, row0, pc.bh, p.N,
                        p.DEN + static_cast<size_t>(pc.bh) * p.N + row0 + lane);
                write_o(lane_base, 1, lane, obox1, &p.tmO, row0, pc.bh, p.N, nullptr);
                tc_fence_before_sync();
                warp_arrive(bar(B_OFREE), lane);
            }
            g0 += pc.n;
        }
        if (lane == 0) tma_store_wait_all();
    } else {
        // ------------------------------------------------ compute warps
        regs_alloc<REGS_COMPUTE>();
        // Two warpgroups over the same 128 rows (warp w reads TMEM lanes
        // 32 (w % 4) ..); each takes half of every step.  Per chunk c: S(c)
        // into registers (the tensor core may then form S(c+1)); P(c) once
        // chunk c-1's [num | den] is complete; PREADY; the bf16 state copy of
        // chunk c-1 and phi(Q) of chunk c; PHIQREADY; phi(K) of chunk c;
        // PHIKREADY.  The epilogue warps write O.
        const int i = threadIdx.x % 128;  // row of the chunk = TMEM lane; also row i of S^T
        const int grp = warp / 4;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
        const float scale = p.scale;
        const float r = sqrtf(scale), h = scale * 0.70710678118654752f, g = scale;
        const int col0 = grp == 0 ? 0 : 64, ncol = grp == 0 ? 64 : F - 64;  // this group's state columns
        bool ok = true;
        int g0 = 0;  // chunks of earlier pieces
        // The chunk before the current one (possibly the previous piece's
        // last): its O is written while the current chunk's products run.
        int prev_bh = 0, prev_publish = 0, pc_prev_bh = 0;
        // --- this warp's rows and columns of S^T (fp32), once a piece's last
        // state product is done, for the CTA that walks the rest of the head;
        // then this warp's flag
        auto publish = [&](int pbh) {
            for (int blk = 0; blk < ncol; blk += 16) {
                uint32_t u[16];
                tmem_ld16(lane_base + T_ST + col0 + blk, u);
                if (i < NV) {
                    float4 *dst = reinterpret_cast<float4 *>(p.carry + (static_cast<size_t>(pbh) * NV + i) * F + col0 + blk);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_float4(__uint_as_float(u[4 * q]), __uint_as_float(u[4 * q + 1]),
                                             __uint_as_float(u[4 * q + 2]), __uint_as_float(u[4 * q + 3]));
                }
            }
            __threadfence();
            __syncwarp();
            if (lane == 0) atomicExch(p.flags + static_cast<size_t>(pbh) * 8 + warp, p.epoch);
        };
        for (int kp = 0; ok && kp < n_pieces; ++kp) {
        const Piece pc = piece(kp);
        const int bh = pc.bh, c0 = pc.c0, n_chunks = pc.n;
        const bool has_prev = pc.carry != 0;
        if (MODE == 2 && pc.carry == 2) {
            // --- the state of the head's chunks before c0, published by the
            // CTA that walked them: this warp's rows and columns of S^T, which
            // the same warp of that CTA wrote (rows >= 80 are 0).  S^T is
            // free once the previous piece's last state product is done (and
            // published, if that piece is the start of a head).
            if (kp > 0) {
                if (!(ok = wait_bounded(bar(B_STDONE), (g0 - 1) & 1, abort_flag,
                                        (ROLE_BASED_COMPUTE << 24) | (B_STDONE << 16) | ((g0 - 1) & 0xFFFF))))
                    break;
                tc_fence_after_sync();
                if (prev_publish) publish(prev_bh);
                prev_publish = 0;
            }
            if (lane == 0) {
                const volatile unsigned long long *flag = p.flags + static_cast<size_t>(bh) * 8 + warp;
                const uint64_t t0 = global_timer_ns();
                while (*flag != p.epoch) {
                    if (*abort_flag || global_timer_ns() - t0 > kWaitLimitNs) {
                        if (!*abort_flag) {
                            *abort_flag = 1;
                            record_timeout((ROLE_BASED_COMPUTE << 24) | (0xFF << 16) | (bh & 0xFFFF));
                        }
                        ok = false;
                        break;
                    }
                }
                __threadfence();
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            // all of this thread's 96 columns in flight at once (group 0 uses
            // the first 64), then into TMEM
            float4 v[24];
            const float4 *src = reinterpret_cast<const float4 *>(p.carry + (static_cast<size_t>(bh) * NV + i) * F + col0);
#pragma unroll
            for (int q = 0; q < 24; ++q) v[q] = i < NV ? __ldcg(src + q) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int blk = 0; blk < 6; ++blk) {
                if (blk * 16 >= ncol) break;
                uint32_t u[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    u[4 * q] = __float_as_uint(v[4 * blk + q].x);
                    u[4 * q + 1] = __float_as_uint(v[4 * blk + q].y);
                    u[4 * q + 2] = __float_as_uint(v[4 * blk + q].z);
                    u[4 * q + 3] = __float_as_uint(v[4 * blk + q].w);
                }
                tmem_st16(lane_base + T_ST + col0 + blk * 16, u);
            }
            tmem_st_wait();
        }
        if (SEG && has_prev) {
            // --- the state of the segments before this one: the sum of their
            // fp32 partial states, into the group's columns of S^T (rows >= 65 are 0)
            const int seg = pc.seg;
            for (int blk = 0; blk < ncol; blk += 16) {
                float acc[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[e] = 0.0f;
                if (i < NV) {
                    for (int sp = 0; sp < seg; ++sp) {
                        const float4 *src = reinterpret_cast<const float4 *>(
                            p.ws + ((static_cast<size_t>(bh) * p.n_seg + sp) * NV + i) * F + col0 + blk);
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
                tmem_st16(lane_base + T_ST + col0 + blk, u);
            }
            tmem_st_wait();
        }
        for (int c = 0; c < n_chunks; ++c) {
            const int gc = g0 + c;
            const int b = gc & 1;
            const uint32_t ph = gc & 1;
            const uint32_t qb = sbase + QK_OFF + b * 2 * BOX, kb = qb + BOX;
            const int row = (c0 + c) * C + i;  // sequence position of this thread's query and key
            if (!(ok = wait_bounded(bar(B_SFULL), ph, abort_flag,
                                    (ROLE_BASED_COMPUTE << 24) | (B_SFULL << 16) | (gc & 0xFFFF))))
                break;
            tc_fence_after_sync();
            // --- P: w_ij = 1 + s + s^2/2 for keys j <= i of the chunk (and j < N), this group's 64 keys
            uint32_t pk[32];
            if (grp == 1 && warp % 4 < 2) {
                // rows 0..63 see none of keys 64..127: nothing to read
                tc_fence_before_sync();
                warp_arrive(bar(B_SREAD), lane);
#pragma unroll
                for (int e = 0; e < 32; ++e) pk[e] = 0u;
            } else {
                const int jmax = min(i, p.N - 1 - (c0 + c) * C);  // last key of the chunk this row sees
                uint32_t sr[64];
                tmem_ld64(lane_base + T_S + grp * 64, sr);
                tc_fence_before_sync();
                warp_arrive(bar(B_SREAD), lane);
                // w = 1 + c t + (c^2 / 2) t^2 for the raw score t, in Horner form:
                // two packed FMAs per pair of keys
                const float2 sc2 = make_float2(scale, scale), one2 = make_float2(1.0f, 1.0f),
                             hc2 = make_float2(0.5f * scale * scale, 0.5f * scale * scale);
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int j0 = grp * 64 + 2 * e;
                    const float2 t2 = make_float2(__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1]));
                    const float2 w2 = __ffma2_rn(t2, __ffma2_rn(t2, hc2, sc2), one2);
                    pk[e] = pack_bf16x2(j0 <= jmax ? w2.x : 0.0f, j0 + 1 <= jmax ? w2.y : 0.0f);
                }
            }
            if (gc > 0) {
                // the previous chunk's P [V|1] and phi(Q) S are done: T_P, T_O and T_PHIQ are free
                if (!(ok = wait_bounded(bar(B_ODONE), ph ^ 1, abort_flag,
                                        (ROLE_BASED_COMPUTE << 24) | (B_ODONE << 16) | (gc & 0xFFFF))))
                    break;
                tc_fence_after_sync();
            }
            tmem_st32(lane_base + T_P + grp * 32, pk);
            prev_bh = bh;
            tmem_st_wait();
            tc_fence_before_sync();
            warp_arrive(bar(B_PREADY), lane);
            if (c > 0 || has_prev) {
                // --- bf16 copy of the state S_{<c} (rows 0..79 of S^T): 32-feature blocks
                // {0, 1} (group 0) and {2, 3, 4} (group 1) of the 160 (at a
                // segment's first chunk: the state the group itself stored above)
                if (c > 0 && !(ok = wait_bounded(bar(B_STDONE), ph ^ 1, abort_flag,
                                                 (ROLE_BASED_COMPUTE << 24) | (B_STDONE << 16) | (gc & 0xFFFF))))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int blk = 0; blk < 3; ++blk) {
                    if (grp == 0 && blk == 2) break;
                    const int col = grp == 0 ? blk * 32 : 64 + blk * 32;
                    uint32_t sv[32];
                    tmem_ld32(lane_base + T_ST + col, sv);  // every lane loads; rows >= 80 are not stored
                    if (i < NV) {
                        const uint32_t box = sbase + SPREV_OFF + (col / 64) * SBOX;
                        const int q0 = (col % 64) / 8;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            st_shared_v4(sw128(box, i, q0 + q),
                                         pack_bf16x2(__uint_as_float(sv[8 * q]), __uint_as_float(sv[8 * q + 1])),
                                         pack_bf16x2(__uint_as_float(sv[8 * q + 2]), __uint_as_float(sv[8 * q + 3])),
                                         pack_bf16x2(__uint_as_float(sv[8 * q + 4]), __uint_as_float(sv[8 * q + 5])),
                                         pack_bf16x2(__uint_as_float(sv[8 * q + 6]), __uint_as_float(sv[8 * q + 7])));
                    }
                }
            } else if (MODE == 2 && kp > 0) {
                // a later piece's first chunk from no state: the previous
                // piece's last state product must be done before phi(K) is
                // written again (and publish S^T if that piece was the start
                // of a head)
                if (!(ok = wait_bounded(bar(B_STDONE), ph ^ 1, abort_flag,
                                        (ROLE_BASED_COMPUTE << 24) | (B_STDONE << 16) | (gc & 0xFFFF))))
                    break;
                tc_fence_after_sync();
                if (prev_publish) publish(pc_prev_bh);
                prev_publish = 0;
            }
            // --- phi(Q) of chunk c into TMEM (group 0: features 0..63; group 1: 64..159)
            if (grp == 0)
                phi_store<1, true>(qb, i, true, r, h, g, lane_base + T_PHIQ);
            else
                phi_store<6, true>(qb, i, true, r, h, g, lane_base + T_PHIQ);
            tmem_st_wait();
            fence_proxy_async_smem();
            tc_fence_before_sync();
            warp_arrive(bar(B_PHIQREADY), lane);
            // --- phi(K) of chunk c into smem, 0 for keys past N (group 0: features 64..159;
            // group 1: 0..63); its last reader, chunk c-1's state product, is done
            if (grp == 0)
                phi_store<6, false>(kb, i, row < p.N, r, h, g, sbase + PHIK_OFF);
            else
                phi_store<1, false>(kb, i, row < p.N, r, h, g, sbase + PHIK_OFF);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            warp_arrive(bar(B_PHIKREADY), lane);
            warp_arrive(bar(B_QKEMPTY + b), lane);  // this chunk's Q and K are no longer read here
        }
        if (!ok) break;
        prev_publish = pc.publish;
        pc_prev_bh = bh;
        g0 += n_chunks;
        }
        // --- O of the last chunk (and the state, if that piece is the start
        // of a head)
        if (ok && g0 > 0) {
            const int g_last = g0 - 1;
            if (MODE == 2 && prev_publish &&
                (ok = wait_bounded(bar(B_STDONE), g_last & 1, abort_flag,
                                   (ROLE_BASED_COMPUTE << 24) | (B_STDONE << 16) | (g_last & 0xFFFF)))) {
                tc_fence_after_sync();
                publish(pc_prev_bh);
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == M_WARP_MMA) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}


// ------------------------------------------------------------------ segment states
//
// For a head split into segments, the state each segment starts from is the
// sum of the partial states of the segments before it.  This pass forms, per
// (head, segment) except the last, the segment's partial state
//   dS^T = sum over its rows of [v_j | 1] phi(k_j)^T      (fp32, 65 live rows x 160)
// with the same feature map and product as the main kernel's state update,
// and stores it to ws[bh][seg] (rows 65..79 are zero).
namespace st {
constexpr uint32_t K_OFF = 0;                         // K box of chunk c at + (c & 1) * BOX
constexpr uint32_t V_OFF = K_OFF + 2 * BOX;           // V box likewise
constexpr uint32_t ONES_OFF = V_OFF + 2 * BOX;
constexpr uint32_t PHIK_OFF = ONES_OFF + BOX;         // phi(K) of chunk c at + (c & 1) * 3 * BOX
constexpr uint32_t BAR_OFF = PHIK_OFF + 6 * BOX;
constexpr int B_FULL = 0;          // + buffer (2): K, V loaded
constexpr int B_FREE = 2;          // + buffer (2): the state product of the chunk in it is done
constexpr int B_PHIKREADY = 4;     // + buffer (2): phi(K) in smem (8 warps)
constexpr int B_STDONE = 6;
constexpr int B_MMADONE = 7;
constexpr int NUM_BARS = 8;
constexpr uint32_t SMEM_USED = BAR_OFF + NUM_BARS * 8 + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
constexpr uint32_t TMEM_COLS = 256;
static_assert(SMEM_ALLOC <= 227u * 1024u, "shared memory per CTA");
}  // namespace st

__global__ void __launch_bounds__(NUM_THREADS, 1) based_state_kernel(const __grid_constant__ BasedParams p) {
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
            mbar_init(bar(st::B_PHIKREADY + b), 8);
        }
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
            int issued = 0;
            bool ok = true;
            for (int c = 0; c < n_chunks; ++c) {
                const int b = c & 1;
                if (c >= 2 && !(ok = wait_bounded(bar(st::B_FREE + b), ((c >> 1) - 1) & 1, abort_flag,
                                                  (ROLE_BASED_PRODUCER << 24) | ((st::B_FREE + b) << 16) | c)))
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
            }
        }
        __syncwarp();
    } else if (warp == WARP_MMA) {
        if (lane == 0) {
            constexpr uint32_t ID_STATE = idesc_bf16_f32(C, F, 1, 1);  // [V | 1]^T phi(K): both MN-major
            bool ok = true;
            for (int c = 0; ok && c < n_chunks; ++c) {
                const int b = c & 1;
                const uint32_t vb = sbase + st::V_OFF + b * BOX;
                if (!(ok = wait_bounded(bar(st::B_FULL + b), (c >> 1) & 1, abort_flag,
                                        (ROLE_BASED_MMA << 24) | ((st::B_FULL + b) << 16) | c)))
                    break;
                if (!(ok = wait_bounded(bar(st::B_PHIKREADY + b), (c >> 1) & 1, abort_flag,
                                        (ROLE_BASED_MMA << 24) | ((st::B_PHIKREADY + b) << 16) | c)))
                    break;
                tc_fence_after_sync();
#pragma unroll
                for (int k = 0; k < C / 16; ++k)
                    umma_ss(tmem, smem_desc_sw128(vb + k * 2048, st::ONES_OFF - (vb - sbase), 1024),
                            smem_desc_sw128(sbase + st::PHIK_OFF + b * 3 * BOX + k * 2048, BOX, 1024), ID_STATE,
                            (c > 0 || k > 0) ? 1u : 0u);
                umma_commit(bar(st::B_FREE + b));
            }
            if (ok) umma_commit(bar(st::B_STDONE));
            umma_commit(bar(st::B_MMADONE));
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(bar(st::B_MMADONE), 0) && global_timer_ns() - t0 < (ok ? kWaitLimitNs : kDrainLimitNs)) {
            }
        }
        __syncwarp();
    } else {
        const int i = threadIdx.x % 128;
        const int grp = warp / 4;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp % 4) * 32) << 16);
        const float scale = p.scale;
        const float r = sqrtf(scale), h = scale * 0.70710678118654752f, g = scale;
        bool ok = true;
        for (int c = 0; c < n_chunks; ++c) {
            const int b = c & 1;
            if (!(ok = wait_bounded(bar(st::B_FULL + b), (c >> 1) & 1, abort_flag,
                                    (ROLE_BASED_COMPUTE << 24) | ((st::B_FULL + b) << 16) | c)))
                break;
            if (c >= 2 && !(ok = wait_bounded(bar(st::B_FREE + b), ((c >> 1) - 1) & 1, abort_flag,
                                              (ROLE_BASED_COMPUTE << 24) | ((st::B_FREE + b) << 16) | c)))
                break;
            const uint32_t kb = sbase + st::K_OFF + b * BOX, dst = sbase + st::PHIK_OFF + b * 3 * BOX;
            const bool live = (c0 + c) * C + i < p.N;
            if (grp == 0)
                phi_store<6, false>(kb, i, live, r, h, g, dst);
            else
                phi_store<1, false>(kb, i, live, r, h, g, dst);
            fence_proxy_async_smem();
            tc_fence_before_sync();
            warp_arrive(bar(st::B_PHIKREADY + b), lane);
        }
        if (ok && wait_bounded(bar(st::B_STDONE), 0, abort_flag, (ROLE_BASED_COMPUTE << 24) | (st::B_STDONE << 16))) {
            tc_fence_after_sync();
            // rows 0..79 of the partial state: group 0 columns 0..63, group 1 64..159
            const int col0 = grp == 0 ? 0 : 64, ncol = grp == 0 ? 64 : F - 64;
            float *dst = p.ws + ((static_cast<size_t>(bh) * p.n_seg + seg) * NV + i) * F;
            for (int blk = 0; blk < ncol; blk += 32) {
                uint32_t v[32];
                tmem_ld32(lane_base + col0 + blk, v);  // every lane loads; rows >= 80 are not stored
                if (i < NV) {
                    float4 *d4 = reinterpret_cast<float4 *>(dst + col0 + blk);
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

}  // namespace based

cudaError_t launch_based(const BasedParams &p, cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        if ((err = cudaFuncSetAttribute(based::based_kernel<0>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        based::SMEM_ALLOC)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(based::based_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        based::SMEM_ALLOC)) != cudaSuccess ||
            (err = cudaFuncSetAttribute(based::based_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        based::SMEM_ALLOC)) != cudaSuccess)
            return err;
        for (auto kern : {based::based_kernel<0>, based::based_kernel<1>, based::based_kernel<2>}) {
            cudaFuncAttributes attr;
            if ((err = cudaFuncGetAttributes(&attr, kern)) != cudaSuccess) return err;
            if (attr.numRegs != based::LAUNCH_REGS) return cudaErrorInvalidConfiguration;
        }
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(based::MAIN_THREADS, 1, 1);
    cfg.dynamicSmemBytes = based::SMEM_ALLOC;
    cfg.stream = stream;
    if (p.balanced) {
        // One CTA per SM, all resident at once (a CTA may wait for the state
        // another publishes), which a cooperative launch guarantees.
        int sms = 0;
        if ((err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return err;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.gridDim = dim3(static_cast<unsigned>(sms), 1, 1);
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        return cudaLaunchKernelEx(&cfg, based::based_kernel<2>, p);
    }
    cfg.gridDim = dim3(static_cast<unsigned>(p.BH * p.n_seg), 1, 1);
    return p.n_seg > 1 ? cudaLaunchKernelEx(&cfg, based::based_kernel<1>, p)
                       : cudaLaunchKernelEx(&cfg, based::based_kernel<0>, p);
}

// The segment-state pass (n_seg > 1): one CTA per (head, segment) but the last.
cudaError_t launch_based_states(const BasedParams &p, cudaStream_t stream) {
    static thread_local int configured_device = -1;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (configured_device != dev) {
        if ((err = cudaFuncSetAttribute(based::based_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        based::st::SMEM_ALLOC)) != cudaSuccess)
            return err;
        configured_device = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.BH * (p.n_seg - 1)), 1, 1);
    cfg.blockDim = dim3(based::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = based::st::SMEM_ALLOC;
    cfg.stream = stream;
    return cudaLaunchKernelEx(&cfg, based::based_state_kernel, p);
}

cudaError_t read_and_clear_based_status(uint32_t *status, uint32_t *detail) {
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
