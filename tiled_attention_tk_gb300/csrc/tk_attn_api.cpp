// tk_attn_api.cpp -- the C ABI declared in include/tk_attn.h: argument
// validation, TMA tensor-map encoding, per-device caches and the launch.
//
// The call sequence follows the launcher idiom of the ThunderKittens blog
// post (alanwu.xyz/posts/thunderkittens, run_add_kernel: launch, then read
// cudaGetLastError and report it), minus the synchronisation: the launch is
// asynchronous on the caller's stream and errors come back as status codes.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "tk_attn.h"
#include "tk_attn_internal.h"

namespace {

constexpr int kVersionMajor = 0;
constexpr int kVersionMinor = 2;
constexpr int kMaxDevices = 64;

thread_local int t_last_cuda_error = 0;

int fail_cuda(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return TK_ERR_CUDA;
}

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the
// library does not link libcuda directly.
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;
cudaError_t g_encode_err = cudaSuccess;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        g_encode_err = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                        cudaEnableDefault, &q);
        if (g_encode_err == cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else if (g_encode_err == cudaSuccess)
            g_encode_err = cudaErrorSymbolNotFound;
    });
    return g_encode;
}

struct DeviceInfo {
    bool checked = false;
    bool supported = false;
    int num_sms = 0;
};
DeviceInfo g_devices[kMaxDevices];
std::mutex g_devices_mu;

// Checks (once per device) that the current device is compute capability
// 10.3, the only target the kernels are compiled for.
int current_device(int *num_sms) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e);
    if (dev < 0 || dev >= kMaxDevices) return TK_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_devices_mu);
    DeviceInfo &info = g_devices[dev];
    if (!info.checked) {
        int major = 0, minor = 0, sms = 0;
        if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return fail_cuda(e);
        info.supported = (major == 10 && minor == 3);
        info.num_sms = sms;
        info.checked = true;
    }
    if (!info.supported) return TK_ERR_UNSUPPORTED_DEVICE;
    *num_sms = info.num_sms;
    return TK_OK;
}

bool overlaps(const void *a, uint64_t na, const void *b, uint64_t nb) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + nb && b0 < a0 + na;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_device_memory(const void *p) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();  // clear the sticky-free error state of this query
        return TK_ERR_NOT_DEVICE_MEMORY;
    }
    if (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)
        return TK_ERR_NOT_DEVICE_MEMORY;
    return TK_OK;
}

// 3-D view {D, N, B*H} of a contiguous [B,H,N,D] bf16 tensor, moved as
// 128-row x 64-column boxes with the 128-byte swizzle; loads read rows past
// N as 0, stores skip them.
int encode_qkv_map(CUtensorMap *map, const void *ptr, int64_t N, int64_t D, int64_t BH,
                   uint32_t box_rows = 128) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail_cuda(g_encode_err);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                   static_cast<cuuint64_t>(N) * static_cast<cuuint64_t>(D) * 2};
    const cuuint32_t box[3] = {64, box_rows, 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                     box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);
    return TK_OK;
}

// 3-D view {d0, d1, 1} of a contiguous row-major [d1, d0] bf16 matrix, moved
// as box0 x box1 boxes with the 128-byte swizzle (box0 * 2 = 128 bytes).
int encode_matrix_map(CUtensorMap *map, const void *ptr, int64_t d0, int64_t d1, uint32_t box0, uint32_t box1) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail_cuda(g_encode_err);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d0), static_cast<cuuint64_t>(d1), 1};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d0) * 2,
                                   static_cast<cuuint64_t>(d0) * static_cast<cuuint64_t>(d1) * 2};
    const cuuint32_t box[3] = {box0, box1, 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides,
                     box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);
    return TK_OK;
}

// 3-D view {64, N, BH} of a contiguous [BH, N, 64] bf16 output, stored as
// 32 x 32 boxes (one warp's half rows) with the 64-byte swizzle.
int encode_out32_map(CUtensorMap *map, const void *ptr, int64_t N, int64_t BH) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail_cuda(g_encode_err);
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {64 * 2, static_cast<cuuint64_t>(N) * 64 * 2};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
                     elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);
    return TK_OK;
}

// Shape checks of the backward entry points.
int check_shape(int64_t B, int64_t H, int64_t N, int64_t D) {
    if (B < 1 || H < 1 || N < 1) return TK_ERR_BAD_SHAPE;
    if (D != 32 && D != 64 && D != 96 && D != 128) return TK_ERR_UNSUPPORTED_D;
    // TMA coordinates and the launch grid are 32-bit.
    if (N > INT32_MAX || B > INT32_MAX / H) return TK_ERR_BAD_SHAPE;
    const int64_t BH = B * H;
    if (BH > INT64_MAX / N / D / 4) return TK_ERR_BAD_SHAPE;
    const int64_t n_tiles = (N + 127) / 128;
    if (n_tiles * BH > INT32_MAX) return TK_ERR_BAD_SHAPE;
    return TK_OK;
}

constexpr uint64_t kWorkspaceAlign = 256;

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

}  // namespace

extern "C" {

// The backward kernel's head dim: 32 and 96 run on the 64- and 128-column
// kernels (their tensor maps read the missing columns as zeros).
static int64_t bwd_kernel_dim(int64_t D) { return D <= 64 ? 64 : 128; }

// The fp32 dQ accumulator covers whole 128-row query tiles of every head, in
// the kernel's head dim.
static uint64_t dq_acc_bytes(int64_t B, int64_t H, int64_t N, int64_t D) {
    const uint64_t tiles = (static_cast<uint64_t>(N) + 127) / 128;
    return static_cast<uint64_t>(B) * H * tiles * 128 * bwd_kernel_dim(D) * 4;
}

// One fp32 value per query row, over whole 128-row tiles of every head.
static uint64_t row_bytes(int64_t B, int64_t H, int64_t N) {
    return static_cast<uint64_t>(B) * H * ((static_cast<uint64_t>(N) + 127) / 128) * 128 * 4;
}

size_t tk_attn_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N, int64_t D) {
    if (check_shape(B, H, N, D) != TK_OK) return 0;
    return static_cast<size_t>(round_up(dq_acc_bytes(B, H, N, D), kWorkspaceAlign) +
                               2 * round_up(row_bytes(B, H, N), kWorkspaceAlign));
}

int tk_attn_bwd(const void *Q, const void *K, const void *V, const void *O, const void *dO, const float *LSE,
                void *dQ, void *dK, void *dV, void *workspace, size_t workspace_bytes, int64_t B, int64_t H,
                int64_t N, int64_t D, int causal, float scale, cudaStream_t stream) {
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV || !workspace) return TK_ERR_NULL_PTR;
    int rc = check_shape(B, H, N, D);
    if (rc != TK_OK) return rc;
    if (causal != 0 && causal != 1) return TK_ERR_BAD_FLAG;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return TK_ERR_BAD_SCALE;
    const void *tensors[8] = {Q, K, V, O, dO, dQ, dK, dV};
    for (const void *t : tensors)
        if (!aligned(t, 16)) return TK_ERR_MISALIGNED;
    if (!aligned(LSE, 4)) return TK_ERR_MISALIGNED;
    const uint64_t need = tk_attn_bwd_workspace_bytes(B, H, N, D);
    if (!aligned(workspace, kWorkspaceAlign) || workspace_bytes < need) return TK_ERR_WORKSPACE;
    const int64_t BH = B * H;
    const uint64_t tb = static_cast<uint64_t>(BH) * N * D * 2;
    const uint64_t lb = static_cast<uint64_t>(BH) * N * 4;
    // Outputs (dQ, dK, dV, workspace) must not overlap any input or each other.
    const void *outs[4] = {dQ, dK, dV, workspace};
    const uint64_t out_bytes[4] = {tb, tb, tb, need};
    const void *ins[6] = {Q, K, V, O, dO, LSE};
    const uint64_t in_bytes[6] = {tb, tb, tb, tb, tb, lb};
    for (int a = 0; a < 4; ++a) {
        for (int b = 0; b < 6; ++b)
            if (overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b])) return TK_ERR_ALIAS;
        for (int b = a + 1; b < 4; ++b)
            if (overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b])) return TK_ERR_ALIAS;
    }
    int num_sms = 0;
    if ((rc = current_device(&num_sms)) != TK_OK) return rc;
    const void *ptrs[11] = {Q, K, V, O, dO, LSE, dQ, dK, dV, workspace, nullptr};
    for (int i = 0; i < 10; ++i)
        if ((rc = check_device_memory(ptrs[i])) != TK_OK) return rc;

    tk::BwdParams p;
    if ((rc = encode_qkv_map(&p.tmQ, Q, N, D, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmK, K, N, D, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmV, V, N, D, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmDO, dO, N, D, BH)) != TK_OK) return rc;
    p.O = O;
    p.dO = dO;
    p.LSE = LSE;
    p.dq_acc = static_cast<float *>(workspace);
    char *ws = static_cast<char *>(workspace);
    p.neg_delta = reinterpret_cast<float *>(ws + round_up(dq_acc_bytes(B, H, N, D), kWorkspaceAlign));
    p.neg_lse2 = reinterpret_cast<float *>(ws + round_up(dq_acc_bytes(B, H, N, D), kWorkspaceAlign) +
                                           round_up(row_bytes(B, H, N), kWorkspaceAlign));
    p.dQ = dQ;
    p.dK = dK;
    p.dV = dV;
    p.N = static_cast<int>(N);
    p.D = static_cast<int>(D);
    p.BH = static_cast<int>(BH);
    p.causal = causal;
    p.n_tiles = static_cast<int>((N + 127) / 128);
    p.scale = scale;
    p.scale_log2e = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    cudaError_t e = tk::launch_attn_bwd(static_cast<int>(bwd_kernel_dim(D)), p, num_sms, stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return TK_OK;
}

namespace {

int fwd_shape(int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D, int causal) {
    if (B < 1 || H < 1 || Nq < 1 || Nkv < 1) return TK_ERR_BAD_SHAPE;
    if (D != 32 && D != 64 && D != 96 && D != 128 && D != 256) return TK_ERR_UNSUPPORTED_D;
    // TMA coordinates and the launch grid are 32-bit.
    if (Nq > INT32_MAX || Nkv > INT32_MAX || B > INT32_MAX / H) return TK_ERR_BAD_SHAPE;
    const int64_t BH = B * H;
    const int64_t Nmax = Nq > Nkv ? Nq : Nkv;
    if (BH > INT64_MAX / Nmax / D / 2) return TK_ERR_BAD_SHAPE;
    if ((Nq + 127) / 128 * BH > INT32_MAX) return TK_ERR_BAD_SHAPE;
    if (causal != 0 && causal != 1) return TK_ERR_BAD_FLAG;
    // Causal queries stand at the end of the key sequence; each must see a key.
    if (causal && Nkv < Nq) return TK_ERR_BAD_SHAPE;
    return TK_OK;
}

// The forward's tail split.  Without the causal mask every unit costs the
// same, so the last round of units is the only imbalance: when it is at most
// half full, each of its units runs as two pieces (the first half of the key
// tiles and the rest) on two CTAs, and the round takes half a unit's time.
// Each piece leaves O / l and LSE in the workspace; the second to publish
// merges.  The workspace holds, per piece and Q tile, 128 x D + 128 floats,
// then one 8-byte counter per tail unit, Q tile and 32-row quarter.
struct FwdSplit {
    int round, pieces, kv_first;
    uint64_t part_bytes, workspace;
};

constexpr int64_t kFwdSplitMinKvTiles = 4;  // each piece gets at least two key tiles

FwdSplit plan_fwd_split(int64_t BH, int64_t Nq, int64_t Nkv, int64_t D, int causal, int num_sms) {
    FwdSplit f = {0, 0, 0, 0, 0};
    const int64_t n_kvtiles = (Nkv + 127) / 128;
    if (causal || D == 256 || n_kvtiles < kFwdSplitMinKvTiles) return f;
    const int64_t units = BH * (((Nq + 127) / 128 + 1) / 2);
    if (units <= num_sms) return f;
    const int64_t tail = units % num_sms;
    if (tail == 0 || 2 * tail > num_sms) return f;
    f.round = static_cast<int>(units / num_sms);
    f.pieces = static_cast<int>(2 * tail);
    f.kv_first = static_cast<int>((n_kvtiles + 1) / 2);
    f.part_bytes = round_up(static_cast<uint64_t>(f.pieces) * 2 * 128 * (D + 1) * 4, kWorkspaceAlign);
    f.workspace = f.part_bytes + round_up(static_cast<uint64_t>(tail) * 2 * 4 * 8, kWorkspaceAlign);
    return f;
}

// Tags the launches whose CTAs hand results to one another through a caller
// workspace (the forward's tail split, Based's balanced schedule): a counter
// or flag holds the tag of the last launch that wrote it, so no launch needs
// them cleared.
std::atomic<unsigned long long> g_launch_epoch{0};

}  // namespace

size_t tk_attn_fwd_workspace_bytes(int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D, int causal) {
    if (fwd_shape(B, H, Nq, Nkv, D, causal) != TK_OK) return 0;
    int num_sms = 0;
    if (current_device(&num_sms) != TK_OK) return 0;
    return static_cast<size_t>(plan_fwd_split(B * H, Nq, Nkv, D, causal, num_sms).workspace);
}

// The forward behind every entry point; `allow_split` is false for the
// entry points that take no workspace.
static int attn_fwd_impl(const void *Q, const void *K, const void *V, void *O, float *LSE, void *workspace,
                         size_t workspace_bytes, int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D,
                         int causal, float scale, bool allow_split, cudaStream_t stream) {
    // ---- host-side validation: nothing is enqueued unless all of it passes
    if (!Q || !K || !V || !O || !LSE) return TK_ERR_NULL_PTR;
    int rc = fwd_shape(B, H, Nq, Nkv, D, causal);
    if (rc != TK_OK) return rc;
    const int64_t BH = B * H;
    const int64_t n_qtiles = (Nq + 127) / 128;
    const int64_t n_kvtiles = (Nkv + 127) / 128;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return TK_ERR_BAD_SCALE;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(LSE, 4))
        return TK_ERR_MISALIGNED;
    const uint64_t q_bytes = static_cast<uint64_t>(BH) * Nq * D * 2;
    const uint64_t kv_bytes = static_cast<uint64_t>(BH) * Nkv * D * 2;
    const uint64_t lse_bytes = static_cast<uint64_t>(BH) * Nq * 4;
    if (overlaps(O, q_bytes, Q, q_bytes) || overlaps(O, q_bytes, K, kv_bytes) ||
        overlaps(O, q_bytes, V, kv_bytes) || overlaps(LSE, lse_bytes, Q, q_bytes) ||
        overlaps(LSE, lse_bytes, K, kv_bytes) || overlaps(LSE, lse_bytes, V, kv_bytes) ||
        overlaps(LSE, lse_bytes, O, q_bytes))
        return TK_ERR_ALIAS;

    int num_sms = 0;
    if ((rc = current_device(&num_sms)) != TK_OK) return rc;
    const FwdSplit f = allow_split ? plan_fwd_split(BH, Nq, Nkv, D, causal, num_sms) : FwdSplit{0, 0, 0, 0, 0};
    if (f.workspace > 0) {
        if (!workspace) return TK_ERR_NULL_PTR;
        if (!aligned(workspace, kWorkspaceAlign) || workspace_bytes < f.workspace) return TK_ERR_WORKSPACE;
        if (overlaps(workspace, f.workspace, Q, q_bytes) || overlaps(workspace, f.workspace, K, kv_bytes) ||
            overlaps(workspace, f.workspace, V, kv_bytes) || overlaps(workspace, f.workspace, O, q_bytes) ||
            overlaps(workspace, f.workspace, LSE, lse_bytes))
            return TK_ERR_ALIAS;
    }
    const void *ptrs[6] = {Q, K, V, O, LSE, f.workspace > 0 ? workspace : Q};
    for (const void *ptr : ptrs)
        if ((rc = check_device_memory(ptr)) != TK_OK) return rc;

    tk::AttnParams p;
    if ((rc = encode_qkv_map(&p.tmQ, Q, Nq, D, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmK, K, Nkv, D, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmV, V, Nkv, D, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmO, O, Nq, D, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmO32, O, Nq, D, BH, 32)) != TK_OK) return rc;
    p.O = O;
    p.LSE = LSE;
    p.Nq = static_cast<int>(Nq);
    p.Nkv = static_cast<int>(Nkv);
    p.offset = static_cast<int>(Nkv - Nq);
    p.BH = static_cast<int>(BH);
    p.causal = causal;
    p.n_qtiles = static_cast<int>(n_qtiles);
    p.n_kvtiles = static_cast<int>(n_kvtiles);
    p.n_pairs = static_cast<int>((n_qtiles + 1) / 2);
    p.scale = scale;
    p.scale_log2e = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
    p.split_round = f.round;
    p.split_pieces = f.pieces;
    p.split_kv = f.kv_first;
    char *ws = static_cast<char *>(workspace);
    p.part = f.pieces > 0 ? reinterpret_cast<float *>(ws) : nullptr;
    p.ctr = f.pieces > 0 ? reinterpret_cast<unsigned long long *>(ws + f.part_bytes) : nullptr;
    p.epoch = f.pieces > 0 ? ++g_launch_epoch : 0;

    cudaError_t e = D == 256 ? tk::launch_attn_fwd256(p, num_sms, stream)
                             : tk::launch_attn_fwd(static_cast<int>(D), p, num_sms, stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return TK_OK;
}

int tk_attn_fwd_ws(const void *Q, const void *K, const void *V, void *O, float *LSE, void *workspace,
                   size_t workspace_bytes, int64_t B, int64_t H, int64_t Nq, int64_t Nkv, int64_t D,
                   int causal, float scale, cudaStream_t stream) {
    return attn_fwd_impl(Q, K, V, O, LSE, workspace, workspace_bytes, B, H, Nq, Nkv, D, causal, scale, true,
                         stream);
}

int tk_attn_fwd_kv(const void *Q, const void *K, const void *V, void *O, float *LSE, int64_t B,
                   int64_t H, int64_t Nq, int64_t Nkv, int64_t D, int causal, float scale,
                   cudaStream_t stream) {
    return attn_fwd_impl(Q, K, V, O, LSE, nullptr, 0, B, H, Nq, Nkv, D, causal, scale, false, stream);
}

int tk_attn_fwd(const void *Q, const void *K, const void *V, void *O, float *LSE, int64_t B,
                int64_t H, int64_t N, int64_t D, int causal, float scale, cudaStream_t stream) {
    return tk_attn_fwd_kv(Q, K, V, O, LSE, B, H, N, N, D, causal, scale, stream);
}

int tk_attn_bwd_noalloc(const void *Q, const void *K, const void *V, const void *O, const void *dO,
                        const float *LSE, void *dQ, void *dK, void *dV, int64_t B, int64_t H, int64_t N,
                        int64_t D, int causal, float scale, cudaStream_t stream) {
    // The problem must fit the fixed workspace; this is decided on the host,
    // before anything touches the device.
    int rc = check_shape(B, H, N, D);
    if (rc != TK_OK) return rc;
    if (tk_attn_bwd_workspace_bytes(B, H, N, D) > tk::kNoAllocWorkspaceBytes) return TK_ERR_NOALLOC_TOO_LARGE;
    int num_sms = 0;
    if ((rc = current_device(&num_sms)) != TK_OK) return rc;
    void *ws = nullptr;
    const cudaError_t e = tk::noalloc_workspace(&ws);
    if (e != cudaSuccess) return fail_cuda(e);
    return tk_attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, ws, tk::kNoAllocWorkspaceBytes, B, H, N, D, causal,
                       scale, stream);
}

// ------------------------------------------------------------------ GEMM

namespace {

constexpr int kGemmBM = 128, kGemmBN = 256, kGemmBK = 64, kGemmGroupM = 8;
constexpr int kGemmMinSkIters = 4;  // K iterations per stream-K range at least
// Stream-K pays only when a tile's K loop is long against the fp32 partial
// it writes and the finisher reads (128 KB each way): measured on the GB300,
// it gains about 8% at K = 4096 over 3.2 waves and loses at K = 1024 and
// when there are fewer tiles than SMs, where one tile's partials are summed
// by a single CTA.
constexpr int kGemmSkMinKIters = 48;
constexpr uint64_t kGemmSlotBytes = static_cast<uint64_t>(kGemmBM) * kGemmBN * 4;

struct GemmPlan {
    int tiles_m, tiles_n, k_iters, grid, dp_tiles, sk_tiles, sk_iters_per_cta;
    uint64_t workspace;  // bytes: partial slots, then the counters
    int pair;            // CTA pairs on 256 x 256 tiles
};

int gemm_shape(int64_t M, int64_t N, int64_t K) {
    if (M < 1 || N < 1 || K < 1) return TK_ERR_BAD_SHAPE;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return TK_ERR_BAD_SHAPE;
    // Row strides of A, B and C must be multiples of 16 bytes (TMA).
    if (K % 8 != 0 || N % 8 != 0) return TK_ERR_BAD_SHAPE;
    return TK_OK;
}

// CTA pairs (cta_group::2, 256 x 256 tiles) take a problem with at least a
// full wave of pair tiles and K >= 768: per tile they ran 11-27 % faster than
// single CTAs on the GB300 (8192^3, 6144^3, 16384^3, 8192 x 8192 x 1024 and
// x 768, 2048 x 8192 x 2048), lost with fewer tiles than pairs (2048 x 2048 x
// 4096) and at shorter K (8192 x 8192 x 512: -5 %; x 256: -13 %).  `pairs` is
// the number of pairs that can be resident at once.
bool use_pairs(int64_t M, int64_t N, int64_t K, int64_t pairs) {
    const int64_t t2 = ((M + 2 * kGemmBM - 1) / (2 * kGemmBM)) * ((N + kGemmBN - 1) / kGemmBN);
    return pairs >= 1 && K >= 12 * kGemmBK && t2 >= pairs;
}

// The pairs the device can hold at once (0 if the query fails: single CTAs).
int64_t resident_pairs(int num_sms) {
    int n = 0;
    if (tk::gemm_pair_capacity(&n) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n < num_sms / 2 ? n : num_sms / 2;
}

// Data-parallel waves of whole tiles; when the tiles do not fill the last
// wave (and there is more than one wave), the last partial wave plus one full
// wave are split in K over all workers (stream-K): every worker gets at least
// one tile's worth of K iterations, so a tile has at most two K segments.  A
// worker is a CTA, or a pair of CTAs on the pair path (256 x 256 tiles, a
// 256 x 256 partial slot per pair).  Pairs split only below four waves: there
// stream-K gained (3000 x 5120 x 4096, 3.2 waves: 1474 -> 1581 TFLOP/s against
// single CTAs with stream-K), beyond it the partials cost what the last wave
// loses (8192^3, 13.5 waves: 1894 vs 1885; 6144^3, 7.6 waves: 1886 vs 1856).
GemmPlan plan_gemm(int64_t M, int64_t N, int64_t K, int num_sms, int stream_k) {
    GemmPlan g = {};
    const int64_t pairs = resident_pairs(num_sms);
    g.pair = use_pairs(M, N, K, pairs) ? 1 : 0;
    const int64_t bm = g.pair ? 2 * kGemmBM : kGemmBM;
    g.tiles_m = static_cast<int>((M + bm - 1) / bm);
    g.tiles_n = static_cast<int>((N + kGemmBN - 1) / kGemmBN);
    g.k_iters = static_cast<int>((K + kGemmBK - 1) / kGemmBK);
    const int64_t T = static_cast<int64_t>(g.tiles_m) * g.tiles_n;
    const int64_t P = g.pair ? pairs : num_sms;  // workers
    const int per_worker = g.pair ? 2 : 1;       // CTAs per worker
    if (!stream_k || g.k_iters < kGemmSkMinKIters || T <= P || T % P == 0 || (g.pair && T >= 4 * P)) {
        g.dp_tiles = static_cast<int>(T);
        g.grid = static_cast<int>(per_worker * (T < P ? T : P));
        return g;
    }
    g.sk_tiles = static_cast<int>(P + T % P);  // the partial wave plus one full wave
    g.dp_tiles = static_cast<int>(T - g.sk_tiles);
    const int64_t total = static_cast<int64_t>(g.sk_tiles) * g.k_iters;
    int64_t L = (total + P - 1) / P;
    if (L < kGemmMinSkIters) L = kGemmMinSkIters;
    g.sk_iters_per_cta = static_cast<int>(L);
    g.grid = static_cast<int>(per_worker * P);
    // one 128 x 256 fp32 slot per CTA (a pair's 256 x 256 slot is its two CTAs' slots)
    g.workspace = round_up(static_cast<uint64_t>(g.grid) * kGemmSlotBytes, kWorkspaceAlign) +
                  round_up(static_cast<uint64_t>(g.sk_tiles) * 4, kWorkspaceAlign);
    return g;
}

}  // namespace

size_t tk_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, int stream_k) {
    if (gemm_shape(M, N, K) != TK_OK || (stream_k != 0 && stream_k != 1)) return 0;
    int num_sms = 0;
    if (current_device(&num_sms) != TK_OK) return 0;
    return static_cast<size_t>(plan_gemm(M, N, K, num_sms, stream_k).workspace);
}

int tk_gemm_uses_pairs(int64_t M, int64_t N, int64_t K, int stream_k) {
    if (gemm_shape(M, N, K) != TK_OK || (stream_k != 0 && stream_k != 1)) return 0;
    int num_sms = 0;
    if (current_device(&num_sms) != TK_OK) return 0;
    return plan_gemm(M, N, K, num_sms, stream_k).pair;
}

int tk_gemm(const void *A, const void *B, void *C, void *workspace, size_t workspace_bytes, int64_t M,
            int64_t N, int64_t K, int b_kmajor, int stream_k, cudaStream_t stream) {
    if (!A || !B || !C) return TK_ERR_NULL_PTR;
    int rc = gemm_shape(M, N, K);
    if (rc != TK_OK) return rc;
    if ((b_kmajor != 0 && b_kmajor != 1) || (stream_k != 0 && stream_k != 1)) return TK_ERR_BAD_FLAG;
    if (!aligned(A, 16) || !aligned(B, 16) || !aligned(C, 16)) return TK_ERR_MISALIGNED;
    const uint64_t a_bytes = static_cast<uint64_t>(M) * K * 2, b_bytes = static_cast<uint64_t>(N) * K * 2,
                   c_bytes = static_cast<uint64_t>(M) * N * 2;
    if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, B, b_bytes)) return TK_ERR_ALIAS;
    int num_sms = 0;
    if ((rc = current_device(&num_sms)) != TK_OK) return rc;
    const GemmPlan g = plan_gemm(M, N, K, num_sms, stream_k);
    if (g.workspace > 0) {
        if (!workspace) return TK_ERR_NULL_PTR;
        if (!aligned(workspace, kWorkspaceAlign) || workspace_bytes < g.workspace) return TK_ERR_WORKSPACE;
        if (overlaps(workspace, g.workspace, A, a_bytes) || overlaps(workspace, g.workspace, B, b_bytes) ||
            overlaps(workspace, g.workspace, C, c_bytes))
            return TK_ERR_ALIAS;
    }
    const void *ptrs[4] = {A, B, C, g.workspace > 0 ? workspace : C};
    for (const void *ptr : ptrs)
        if ((rc = check_device_memory(ptr)) != TK_OK) return rc;

    tk::GemmParams p;
    if ((rc = encode_matrix_map(&p.tmA, A, K, M, 64, 128)) != TK_OK) return rc;
    if (b_kmajor) {
        if ((rc = encode_matrix_map(&p.tmB, B, K, N, 64, g.pair ? 128 : 256)) != TK_OK) return rc;
    } else {
        if ((rc = encode_matrix_map(&p.tmB, B, N, K, 64, 64)) != TK_OK) return rc;
    }
    if ((rc = encode_matrix_map(&p.tmC, C, N, M, 64, 32)) != TK_OK) return rc;
    char *ws = static_cast<char *>(workspace);
    p.partials = g.workspace > 0 ? reinterpret_cast<float *>(ws) : nullptr;
    p.counters = g.workspace > 0
                     ? reinterpret_cast<unsigned *>(ws + round_up(static_cast<uint64_t>(g.grid) * kGemmSlotBytes,
                                                                  kWorkspaceAlign))
                     : nullptr;
    p.M = static_cast<int>(M);
    p.N = static_cast<int>(N);
    p.K = static_cast<int>(K);
    p.b_kmajor = b_kmajor;
    p.tiles_m = g.tiles_m;
    p.tiles_n = g.tiles_n;
    p.k_iters = g.k_iters;
    p.group_m = kGemmGroupM;
    p.dp_tiles = g.dp_tiles;
    p.sk_tiles = g.sk_tiles;
    p.sk_iters_per_cta = g.sk_iters_per_cta;
    p.pair = g.pair;
    cudaError_t e = tk::launch_gemm(p, g.grid, stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return TK_OK;
}

// ------------------------------------------------------------------ Based linear attention

namespace {

// Segments per head for Based: one CTA per head leaves SMs idle when the
// heads are fewer than the SMs; a head's chunks are then split into
// segments (at least 4 chunks each), one CTA per segment, after a pass that
// forms each segment's partial state.
struct BasedPlan {
    int n_seg;
    int seg_chunks;
    uint64_t workspace;
    int balanced;  // Based only: the balanced schedule (more heads than SMs, not a multiple)
};

constexpr int kBasedMinSegChunks = 4;
constexpr uint64_t kBasedSegStateBytes = 80ull * 160ull * 4ull;     // one segment's state, fp32
constexpr uint64_t kHedgehogSegStateBytes = 80ull * 128ull * 4ull;  // likewise for Hedgehog

BasedPlan plan_segments(int64_t BH, int64_t N, int num_sms, uint64_t seg_state_bytes) {
    const int64_t n_chunks = (N + 127) / 128;
    BasedPlan pl{1, static_cast<int>(n_chunks), 0, 0};
    if (BH >= num_sms) return pl;
    int64_t n_seg = std::min<int64_t>(num_sms / BH, n_chunks / kBasedMinSegChunks);
    if (n_seg < 2) return pl;
    const int64_t seg_chunks = (n_chunks + n_seg - 1) / n_seg;
    n_seg = (n_chunks + seg_chunks - 1) / seg_chunks;  // no empty segment
    if (n_seg < 2) return pl;
    pl.n_seg = static_cast<int>(n_seg);
    pl.seg_chunks = static_cast<int>(seg_chunks);
    pl.workspace = round_up(static_cast<uint64_t>(BH) * n_seg * seg_state_bytes, kWorkspaceAlign);
    return pl;
}

// More heads than SMs, not a multiple of them: one CTA per head leaves SMs
// idle in the last wave.  When those idle SM-chunks, (waves * SMs - heads) *
// chunks, come to more than eight chunks per SM, the heads' chunks are cut
// into one equal run per CTA instead (balanced schedule); a head split between
// two CTAs passes its state through the workspace (80 x 160 fp32 per head,
// then eight 8-byte flags per head).  The balanced runs cost a CTA about five
// to nine chunks of its own (measured at 8 to 64 chunks per head), so below
// that margin one CTA per head is kept.
BasedPlan plan_based(int64_t BH, int64_t N, int num_sms) {
    const int64_t n_chunks = (N + 127) / 128;
    const int64_t waves = (BH + num_sms - 1) / num_sms;
    const int64_t idle = (waves * num_sms - BH) * n_chunks;  // SM-chunks one CTA per head leaves idle
    if (BH > num_sms && idle > 8 * static_cast<int64_t>(num_sms)) {
        BasedPlan pl{1, static_cast<int>(n_chunks), 0, 1};
        pl.workspace = round_up(static_cast<uint64_t>(BH) * kBasedSegStateBytes, kWorkspaceAlign) +
                       round_up(static_cast<uint64_t>(BH) * 8 * 8, kWorkspaceAlign);
        return pl;
    }
    return plan_segments(BH, N, num_sms, kBasedSegStateBytes);
}

int based_checks(const void *Q, const void *K, const void *V, void *O, float *DEN, int64_t B, int64_t H, int64_t N,
                 int64_t Dqk, int64_t Dv, float scale) {
    if (!Q || !K || !V || !O || !DEN) return TK_ERR_NULL_PTR;
    if (B < 1 || H < 1 || N < 1) return TK_ERR_BAD_SHAPE;
    if (Dqk != 16 || Dv != 64) return TK_ERR_UNSUPPORTED_D;
    if (N > INT32_MAX || B > INT32_MAX / H || B * H > INT32_MAX) return TK_ERR_BAD_SHAPE;
    const int64_t BH = B * H;
    if (BH > INT64_MAX / N / 64 / 2) return TK_ERR_BAD_SHAPE;
    if (!std::isfinite(scale) || !(scale > 0.0f)) return TK_ERR_BAD_SCALE;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(O, 16) || !aligned(DEN, 4))
        return TK_ERR_MISALIGNED;
    const uint64_t qk_bytes = static_cast<uint64_t>(BH) * N * 16 * 2, v_bytes = static_cast<uint64_t>(BH) * N * 64 * 2,
                   den_bytes = static_cast<uint64_t>(BH) * N * 4;
    const void *ins[3] = {Q, K, V};
    const uint64_t in_bytes[3] = {qk_bytes, qk_bytes, v_bytes};
    for (int a = 0; a < 3; ++a)
        if (overlaps(O, v_bytes, ins[a], in_bytes[a]) || overlaps(DEN, den_bytes, ins[a], in_bytes[a]))
            return TK_ERR_ALIAS;
    if (overlaps(O, v_bytes, DEN, den_bytes)) return TK_ERR_ALIAS;
    return TK_OK;
}

int based_launch(const void *Q, const void *K, const void *V, void *O, float *DEN, int64_t BH, int64_t N,
                 float scale, const BasedPlan &pl, void *workspace, cudaStream_t stream) {
    int rc;
    tk::BasedParams p;
    if ((rc = encode_qkv_map(&p.tmQ, Q, N, 16, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmK, K, N, 16, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmV, V, N, 64, BH)) != TK_OK) return rc;
    if ((rc = encode_out32_map(&p.tmO, O, N, BH)) != TK_OK) return rc;
    p.O = O;
    p.DEN = DEN;
    p.ws = static_cast<float *>(workspace);
    p.N = static_cast<int>(N);
    p.BH = static_cast<int>(BH);
    p.n_seg = pl.n_seg;
    p.seg_chunks = pl.seg_chunks;
    p.scale = scale;
    p.balanced = pl.balanced;
    p.carry = pl.balanced ? static_cast<float *>(workspace) : nullptr;
    p.flags = pl.balanced ? reinterpret_cast<unsigned long long *>(
                                static_cast<char *>(workspace) +
                                round_up(static_cast<uint64_t>(BH) * kBasedSegStateBytes, kWorkspaceAlign))
                          : nullptr;
    p.epoch = pl.balanced ? ++g_launch_epoch : 0;
    cudaError_t e = cudaSuccess;
    if (pl.n_seg > 1) e = tk::launch_based_states(p, stream);
    if (e == cudaSuccess) e = tk::launch_based(p, stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return TK_OK;
}

}  // namespace

int tk_based_fwd(const void *Q, const void *K, const void *V, void *O, float *DEN, int64_t B, int64_t H, int64_t N,
                 int64_t Dqk, int64_t Dv, float scale, cudaStream_t stream) {
    int rc = based_checks(Q, K, V, O, DEN, B, H, N, Dqk, Dv, scale);
    if (rc != TK_OK) return rc;
    int num_sms = 0;
    if ((rc = current_device(&num_sms)) != TK_OK) return rc;
    const void *ptrs[5] = {Q, K, V, O, DEN};
    for (const void *ptr : ptrs)
        if ((rc = check_device_memory(ptr)) != TK_OK) return rc;
    const BasedPlan whole{1, static_cast<int>((N + 127) / 128), 0, 0};
    return based_launch(Q, K, V, O, DEN, B * H, N, scale, whole, nullptr, stream);
}

size_t tk_based_workspace_bytes(int64_t B, int64_t H, int64_t N) {
    if (B < 1 || H < 1 || N < 1 || N > INT32_MAX || B > INT32_MAX / H) return 0;
    int num_sms = 0;
    if (current_device(&num_sms) != TK_OK) return 0;
    return static_cast<size_t>(plan_based(B * H, N, num_sms).workspace);
}

int tk_based_fwd_ws(const void *Q, const void *K, const void *V, void *O, float *DEN, void *workspace,
                    size_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t Dqk, int64_t Dv, float scale,
                    cudaStream_t stream) {
    int rc = based_checks(Q, K, V, O, DEN, B, H, N, Dqk, Dv, scale);
    if (rc != TK_OK) return rc;
    int num_sms = 0;
    if ((rc = current_device(&num_sms)) != TK_OK) return rc;
    const BasedPlan pl = plan_based(B * H, N, num_sms);
    if (pl.workspace > 0) {
        if (!workspace) return TK_ERR_NULL_PTR;
        if (!aligned(workspace, kWorkspaceAlign) || workspace_bytes < pl.workspace) return TK_ERR_WORKSPACE;
        const int64_t BH = B * H;
        const uint64_t qk_bytes = static_cast<uint64_t>(BH) * N * 16 * 2, v_bytes = static_cast<uint64_t>(BH) * N * 64 * 2,
                       den_bytes = static_cast<uint64_t>(BH) * N * 4;
        const void *bufs[5] = {Q, K, V, O, DEN};
        const uint64_t bytes[5] = {qk_bytes, qk_bytes, v_bytes, v_bytes, den_bytes};
        for (int a = 0; a < 5; ++a)
            if (overlaps(workspace, pl.workspace, bufs[a], bytes[a])) return TK_ERR_ALIAS;
    }
    const void *ptrs[6] = {Q, K, V, O, DEN, pl.workspace > 0 ? workspace : Q};
    for (const void *ptr : ptrs)
        if ((rc = check_device_memory(ptr)) != TK_OK) return rc;
    return based_launch(Q, K, V, O, DEN, B * H, N, scale, pl, pl.workspace > 0 ? workspace : nullptr, stream);
}

// ------------------------------------------------------------------ Hedgehog linear attention

// 3-D view {c, r, n} of a contiguous [n, r, c] bf16 tensor, moved as
// box_c x box_r x 1 boxes with the 128-byte swizzle.
int encode_batched_map(CUtensorMap *map, const void *ptr, int64_t c, int64_t r, int64_t n, uint32_t box_c,
                       uint32_t box_r) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return fail_cuda(g_encode_err);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(c), static_cast<cuuint64_t>(r), static_cast<cuuint64_t>(n)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(c) * 2, static_cast<cuuint64_t>(c) * r * 2};
    const cuuint32_t box[3] = {box_c, box_r, 1};
    const cuuint32_t elem_strides[3] = {1, 1, 1};
    CUresult res = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
                       elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (res != CUDA_SUCCESS) return fail_cuda(cudaErrorInvalidValue);
    return TK_OK;
}

namespace {

int hedgehog_checks(const void *Q, const void *K, const void *V, const void *Wq, const void *Wk, void *O, float *DEN,
                    int64_t B, int64_t H, int64_t N, int64_t Dqk, int64_t F, int64_t Dv) {
    if (!Q || !K || !V || !Wq || !Wk || !O || !DEN) return TK_ERR_NULL_PTR;
    if (B < 1 || H < 1 || N < 1) return TK_ERR_BAD_SHAPE;
    if (Dqk != 64 || F != 64 || Dv != 64) return TK_ERR_UNSUPPORTED_D;
    if (N > INT32_MAX || B > INT32_MAX / H || B * H > INT32_MAX) return TK_ERR_BAD_SHAPE;
    const int64_t BH = B * H;
    if (BH > INT64_MAX / N / 64 / 2) return TK_ERR_BAD_SHAPE;
    if (!aligned(Q, 16) || !aligned(K, 16) || !aligned(V, 16) || !aligned(Wq, 16) || !aligned(Wk, 16) ||
        !aligned(O, 16) || !aligned(DEN, 4))
        return TK_ERR_MISALIGNED;
    const uint64_t t_bytes = static_cast<uint64_t>(BH) * N * 64 * 2, w_bytes = static_cast<uint64_t>(H) * 64 * 64 * 2,
                   den_bytes = static_cast<uint64_t>(BH) * N * 4;
    const void *ins[5] = {Q, K, V, Wq, Wk};
    const uint64_t in_bytes[5] = {t_bytes, t_bytes, t_bytes, w_bytes, w_bytes};
    for (int a = 0; a < 5; ++a)
        if (overlaps(O, t_bytes, ins[a], in_bytes[a]) || overlaps(DEN, den_bytes, ins[a], in_bytes[a]))
            return TK_ERR_ALIAS;
    if (overlaps(O, t_bytes, DEN, den_bytes)) return TK_ERR_ALIAS;
    return TK_OK;
}

int hedgehog_launch(const void *Q, const void *K, const void *V, const void *Wq, const void *Wk, void *O, float *DEN,
                    int64_t H, int64_t BH, int64_t N, const BasedPlan &pl, void *workspace, cudaStream_t stream) {
    int rc;
    tk::HedgehogParams p;
    if ((rc = encode_qkv_map(&p.tmQ, Q, N, 64, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmK, K, N, 64, BH)) != TK_OK) return rc;
    if ((rc = encode_qkv_map(&p.tmV, V, N, 64, BH)) != TK_OK) return rc;
    if ((rc = encode_batched_map(&p.tmWq, Wq, 64, 64, H, 64, 64)) != TK_OK) return rc;
    if ((rc = encode_batched_map(&p.tmWk, Wk, 64, 64, H, 64, 64)) != TK_OK) return rc;
    if ((rc = encode_out32_map(&p.tmO, O, N, BH)) != TK_OK) return rc;
    p.O = O;
    p.DEN = DEN;
    p.ws = static_cast<float *>(workspace);
    p.N = static_cast<int>(N);
    p.H = static_cast<int>(H);
    p.BH = static_cast<int>(BH);
    p.n_seg = pl.n_seg;
    p.seg_chunks = pl.seg_chunks;
    cudaError_t e = cudaSuccess;
    if (pl.n_seg > 1) e = tk::launch_hedgehog_states(p, stream);
    if (e == cudaSuccess) e = tk::launch_hedgehog(p, stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return TK_OK;
}

}  // namespace

int tk_hedgehog_fwd(const void *Q, const void *K, const void *V, const void *Wq, const void *Wk, void *O, float *DEN,
                    int64_t B, int64_t H, int64_t N, int64_t Dqk, int64_t F, int64_t Dv, cudaStream_t stream) {
    int rc = hedgehog_checks(Q, K, V, Wq, Wk, O, DEN, B, H, N, Dqk, F, Dv);
    if (rc != TK_OK) return rc;
    int num_sms = 0;
    if ((rc = current_device(&num_sms)) != TK_OK) return rc;
    const void *ptrs[7] = {Q, K, V, Wq, Wk, O, DEN};
    for (const void *ptr : ptrs)
        if ((rc = check_device_memory(ptr)) != TK_OK) return rc;
    const BasedPlan whole{1, static_cast<int>((N + 127) / 128), 0, 0};
    return hedgehog_launch(Q, K, V, Wq, Wk, O, DEN, H, B * H, N, whole, nullptr, stream);
}

size_t tk_hedgehog_workspace_bytes(int64_t B, int64_t H, int64_t N) {
    if (B < 1 || H < 1 || N < 1 || N > INT32_MAX || B > INT32_MAX / H) return 0;
    int num_sms = 0;
    if (current_device(&num_sms) != TK_OK) return 0;
    return static_cast<size_t>(plan_segments(B * H, N, num_sms, kHedgehogSegStateBytes).workspace);
}

int tk_hedgehog_fwd_ws(const void *Q, const void *K, const void *V, const void *Wq, const void *Wk, void *O,
                       float *DEN, void *workspace, size_t workspace_bytes, int64_t B, int64_t H, int64_t N,
                       int64_t Dqk, int64_t F, int64_t Dv, cudaStream_t stream) {
    int rc = hedgehog_checks(Q, K, V, Wq, Wk, O, DEN, B, H, N, Dqk, F, Dv);
    if (rc != TK_OK) return rc;
    int num_sms = 0;
    if ((rc = current_device(&num_sms)) != TK_OK) return rc;
    const BasedPlan pl = plan_segments(B * H, N, num_sms, kHedgehogSegStateBytes);
    if (pl.workspace > 0) {
        if (!workspace) return TK_ERR_NULL_PTR;
        if (!aligned(workspace, kWorkspaceAlign) || workspace_bytes < pl.workspace) return TK_ERR_WORKSPACE;
        const int64_t BH = B * H;
        const uint64_t t_bytes = static_cast<uint64_t>(BH) * N * 64 * 2, w_bytes = static_cast<uint64_t>(H) * 64 * 64 * 2,
                       den_bytes = static_cast<uint64_t>(BH) * N * 4;
        const void *bufs[7] = {Q, K, V, Wq, Wk, O, DEN};
        const uint64_t bytes[7] = {t_bytes, t_bytes, t_bytes, w_bytes, w_bytes, t_bytes, den_bytes};
        for (int a = 0; a < 7; ++a)
            if (overlaps(workspace, pl.workspace, bufs[a], bytes[a])) return TK_ERR_ALIAS;
    }
    const void *ptrs[8] = {Q, K, V, Wq, Wk, O, DEN, pl.workspace > 0 ? workspace : Q};
    for (const void *ptr : ptrs)
        if ((rc = check_device_memory(ptr)) != TK_OK) return rc;
    return hedgehog_launch(Q, K, V, Wq, Wk, O, DEN, H, B * H, N, pl, pl.workspace > 0 ? workspace : nullptr, stream);
}

int tk_attn_device_status(cudaStream_t stream, uint32_t *detail) {
    uint32_t status = 0, where = 0, status_b = 0, where_b = 0, status_g = 0, where_g = 0;
    cudaError_t e = tk::read_and_clear_status(stream, &status, &where);  // synchronises the stream
    if (e != cudaSuccess) return fail_cuda(e);
    e = tk::read_and_clear_bwd_status(&status_b, &where_b);
    if (e != cudaSuccess) return fail_cuda(e);
    e = tk::read_and_clear_gemm_status(&status_g, &where_g);
    if (e != cudaSuccess) return fail_cuda(e);
    uint32_t status_l = 0, where_l = 0, status_h = 0, where_h = 0;
    e = tk::read_and_clear_based_status(&status_l, &where_l);
    if (e != cudaSuccess) return fail_cuda(e);
    e = tk::read_and_clear_hedgehog_status(&status_h, &where_h);
    if (e != cudaSuccess) return fail_cuda(e);
    uint32_t status_w = 0, where_w = 0;
    e = tk::read_and_clear_fwd256_status(&status_w, &where_w);
    if (e != cudaSuccess) return fail_cuda(e);
    if (detail)
        *detail = status     ? where
                  : status_b ? where_b
                  : status_g ? where_g
                  : status_l ? where_l
                  : status_h ? where_h
                             : where_w;
    return (status == 0 && status_b == 0 && status_g == 0 && status_l == 0 && status_h == 0 && status_w == 0)
               ? TK_OK
               : TK_ERR_DEVICE_TIMEOUT;
}

int tk_attn_selftest_timeout(uint64_t limit_ns, cudaStream_t stream) {
    if (limit_ns < 1000ull) limit_ns = 1000ull;
    if (limit_ns > 5000000000ull) limit_ns = 5000000000ull;
    int num_sms = 0;
    int rc = current_device(&num_sms);
    if (rc != TK_OK) return rc;
    cudaError_t e = tk::launch_selftest_timeout(limit_ns, stream);
    if (e != cudaSuccess) return fail_cuda(e);
    return TK_OK;
}

const char *tk_attn_strerror(int code) {
    switch (code) {
        case TK_OK: return "success";
        case TK_ERR_NULL_PTR: return "a required pointer is NULL";
        case TK_ERR_BAD_SHAPE: return "invalid shape (B, H, N must be >= 1 and sizes must fit)";
        case TK_ERR_UNSUPPORTED_D:
            return "unsupported head dimension (forward: 32, 64, 96, 128; backward: 64, 128; Based: 16 / 64; "
                   "Hedgehog: 64 / 64 / 64)";
        case TK_ERR_MISALIGNED: return "misaligned pointer (Q, K, V, O: 16 bytes; LSE: 4 bytes)";
        case TK_ERR_BAD_SCALE: return "scale must be finite and > 0";
        case TK_ERR_ALIAS: return "outputs overlap inputs or each other";
        case TK_ERR_BAD_FLAG: return "causal must be 0 or 1";
        case TK_ERR_UNSUPPORTED_DEVICE: return "current device is not compute capability 10.3 (sm_103a)";
        case TK_ERR_CUDA: return "a CUDA call or the kernel launch failed";
        case TK_ERR_DEVICE_TIMEOUT: return "a bounded wait inside a kernel gave up";
        case TK_ERR_NOT_DEVICE_MEMORY: return "a pointer is not device or managed memory";
        case TK_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
        case TK_ERR_NOALLOC_TOO_LARGE:
            return "problem needs more workspace than the 32 MiB built into tk_attn_bwd_noalloc";
        default: return "unknown status code";
    }
}

int tk_attn_last_cuda_error(void) { return t_last_cuda_error; }

int tk_attn_version(void) { return (kVersionMajor << 16) | kVersionMinor; }

}  // extern "C"
