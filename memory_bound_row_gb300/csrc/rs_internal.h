// Internal contract between the C-ABI layer (rowsoftmax_api.cu), the
// planner and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "rowsoftmax.h"

namespace rs {

// Per-thread unit counts instantiated for RS_PATH_ROWS.  A unit is one
// 16-byte access (4 fp32 or 8 fp16/bf16 elements) or, for the element-wise
// kernels, one element.  The planner picks only from these lists and the
// launchers dispatch over exactly the same lists.
#define RS_VPT_VEC_F32 1, 2, 3, 4, 5, 6, 8, 10, 12, 16
#define RS_VPT_VEC_16 1, 2, 3, 4, 5, 6, 8
#define RS_VPT_SCALAR 1, 2, 4, 8, 16

constexpr int kVptVecF32[] = {RS_VPT_VEC_F32};
constexpr int kVptVec16[] = {RS_VPT_VEC_16};
constexpr int kVptScalar[] = {RS_VPT_SCALAR};

// The normalisations (RMSNorm, LayerNorm) are instantiated for fewer counts.
#define RS_VPT_NORM_VEC 1, 2, 3, 4, 5, 6, 8
#define RS_VPT_NORM_SCALAR 1, 2, 4, 8, 16
constexpr int kVptNormVec[] = {RS_VPT_NORM_VEC};
constexpr int kVptNormScalar[] = {RS_VPT_NORM_SCALAR};

// The one-CTA-per-row streaming normalisation kernel: threads per CTA, and
// CTAs per SM in the grid (few, so that the rows being re-read stay in L2).
constexpr int kNormStreamThreads = 512;
constexpr int kNormStreamCtasPerSm = 2;

// Upper bound on fp32 values a thread holds in RS_PATH_ROWS (register budget).
constexpr int kRowsMaxValuesPerThread = 64;
constexpr int kRowsMaxThreads = 1024;

// Largest CTA an RS_PATH_ROWS instance is compiled for.  1024 threads leave
// 64 registers a thread, enough for up to 8 units and 32 values; larger
// instances are compiled for 512 threads (128 registers) so they do not spill.
constexpr int rows_block_limit(int vpt, int vec) { return (vpt <= 8 && vpt * vec <= 32) ? 1024 : 512; }

// RS_PATH_RING instances that re-read shared memory are compiled for at most
// kRingRereadThreads threads and kRingRereadMinCtas resident CTAs of that size,
// which caps them at 40 registers a thread.
constexpr int kRingRereadThreads = 512;
constexpr int kRingRereadMinCtas = 3;
constexpr int kRingRereadRegs = 40;

// Persistent ring kernel (RS_PATH_RING).
constexpr int kRingMaxStages = 8;
constexpr size_t kRingStaticSmem = 1024;  // upper bound of the kernel's static shared memory

// Cluster kernels (RS_PATH_CLUSTER / RS_PATH_STREAM).
constexpr int kWideThreads = 256;      // threads per CTA
constexpr int kWideUnitsPerThread = 4; // units per thread per stage
constexpr int kWideUnitsPerStage = kWideThreads * kWideUnitsPerThread;
constexpr int kWideMaxStages = 16;     // mbarriers per CTA
constexpr int kMaxClusterPortable = 8;
constexpr int kMaxCluster = 16;        // needs the non-portable cluster-size opt-in
constexpr size_t kWideStaticSmem = 1024;  // upper bound of the kernel's static shared memory
constexpr int kWideHoldThreads = 512;     // max threads per CTA of the register-holding cluster kernel
constexpr int kWideHoldMaxVpt = 8;        // units per thread it is instantiated for: 1, 2, 4, 8 (8: 256 threads)
constexpr int kWideHoldMaxSlots = 4;      // shared-memory landing slots per CTA of that kernel

// Per-call parameters of a row operation: the normalisations' weight and
// bias vectors (N stored values each, or null) and eps; zero for the softmax.
// A causal mask (the softmax only): row r keeps its first
// min(N, max(0, (r mod mask_period) + 1 + mask_offset)) elements; the rest is
// -inf, never read, and written as 0.  mask_period 0: no mask.
struct RowArgs {
    const void* w;
    const void* b;
    float eps;
    int64_t mask_period;
    int64_t mask_offset;
    uint64_t mask_magic;  // 2^64 / mask_period rounded up (mod 2^64), for rows and periods below 2^32
};

// The reciprocal constant of the remainder by direct computation (Lemire,
// Kaser and Kurz, "Faster Remainder by Direct Computation", 2019): for
// 32-bit n and d >= 1, n mod d = high64((c * n mod 2^64) * d) with
// c = floor((2^64 - 1) / d) + 1 (mod 2^64).
inline uint64_t remainder_magic(uint64_t d) { return d ? ~0ull / d + 1 : 0; }

// Launch of `kern` with the programmatic-dependent-launch attribute (unless
// `strict`), and a cluster dimension when cluster > 0.  The kernels wait for
// the previous grid of the stream before touching global memory (see
// wait_prior_grid), so the attribute only overlaps launch and setup.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem, cudaStream_t s,
                          int cluster, bool strict, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(block, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (!strict) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster > 0) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    cudaError_t err = cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        return err;
    }
    return cudaGetLastError();
}

// Launchers.  Each returns the CUDA error of the launch (cudaSuccess if it
// was enqueued).  Arguments were validated and planned by the caller.
// Normalisations: plan.op selects RMSNorm or LayerNorm; plan.path RS_PATH_ROWS,
// RS_PATH_RING, RS_PATH_CLUSTER (register-holding clusters) or RS_PATH_STREAM
// (one CTA per row, reads the row 2 or 3 times).
cudaError_t launch_norm_f32(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                            int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_norm_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                            int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_norm_bf16(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                             int64_t ldo, cudaStream_t s, const RowArgs& a);
// The softmax launchers take the mask in `a` (weight, bias and eps unused).
cudaError_t launch_rows_f32(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                            int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_rows_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                            int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_rows_bf16(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                             int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_ring_f32(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                            int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_ring_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                            int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_ring_bf16(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                             int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_wide(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                        int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a);

// Number of clusters of the planned wide kernel that fit on the device at
// once (0: the cluster shape cannot be scheduled).
cudaError_t wide_max_active_clusters(const rs_plan& p, int* n);

// Device status words, one per translation unit with bounded waits; each
// ORs its word into *flags (and clears it when asked).
cudaError_t read_status_f32(unsigned int* flags, bool clear);
cudaError_t read_status_f16(unsigned int* flags, bool clear);
cudaError_t read_status_bf16(unsigned int* flags, bool clear);
cudaError_t read_status_wide(unsigned int* flags, bool clear);
// The softmax under a causal mask (a.mask_period > 0): plan.path RS_PATH_ROWS,
// RS_PATH_RING (rows held in registers) or RS_PATH_CLUSTER (register-holding).
cudaError_t launch_causal_f32(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                              int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_causal_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                              int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_causal_bf16(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                               int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t causal_max_clusters_f32(const rs_plan& p, int* n);
cudaError_t causal_max_clusters_f16(const rs_plan& p, int* n);
cudaError_t causal_max_clusters_bf16(const rs_plan& p, int* n);
cudaError_t read_status_causal_f32(unsigned int* flags, bool clear);
cudaError_t read_status_causal_f16(unsigned int* flags, bool clear);
cudaError_t read_status_causal_bf16(unsigned int* flags, bool clear);
// Which LayerNorm row operation serves a planned shape on the register rows or
// the ring: 1 = OpLayerNormWarp (rows inside one warp), 2 = OpLayerNormWhole
// (vectorised rows that fill their threads exactly over a power-of-two number
// of warps), 3 = OpLayerNormWholeHeld (kind 2 on the ring with at most 32
// values a thread and kHeldThreads threads a CTA: the weight and bias held in
// registers, kHeldRegs a thread), 4 = OpLayerNormHeld (other fp32 rows of
// 2 to 8 warps on the ring at 8 units a thread, weight and bias held),
// 0 = OpLayerNorm (the others, and the other paths).
constexpr int kHeldThreads = 256;
constexpr int kHeldRegs = 128;
inline int layernorm_merge_kind(const rs_plan& p, int64_t N, int vec_full) {
    if (p.path != RS_PATH_ROWS && p.path != RS_PATH_RING) return 0;
    const int tpr = p.threads_per_row;
    if (tpr <= 32) return 1;
    const bool ring_held = p.path == RS_PATH_RING && p.vec_elems == vec_full &&
                           p.vec_per_thread * p.vec_elems <= 32 && p.block_threads <= kHeldThreads;
    const int wpr = tpr / 32;
    if (p.vec_elems == vec_full && (wpr & (wpr - 1)) == 0 &&
        N == (int64_t)tpr * p.vec_per_thread * p.vec_elems)
        return ring_held ? 3 : 2;
    if (ring_held && vec_full == 4 && p.vec_per_thread == 8) return 4;
    return 0;
}
// RMSNorm on the ring with the weight held in registers (OpRmsNormHeld): rows
// of at least 4 warps at up to 4 units a thread in kHeldThreads-thread CTAs
// (measured 3.9 % faster on 8192-value bf16 rows, no change on rows of 2 warps).
inline bool rmsnorm_ring_held(const rs_plan& p, int vec_full) {
    return p.path == RS_PATH_RING && p.vec_elems == vec_full && p.vec_per_thread <= 4 &&
           p.block_threads <= kHeldThreads && p.threads_per_row >= 128;
}
// LayerNorm instances with one merge of per-lane moments (kinds 1, 2 and 3 above).
cudaError_t launch_lnmerge_f32(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                               int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_lnmerge_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                               int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t launch_lnmerge_bf16(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                                int64_t ldo, cudaStream_t s, const RowArgs& a);
cudaError_t read_status_lnmerge_f32(unsigned int* flags, bool clear);
cudaError_t read_status_lnmerge_f16(unsigned int* flags, bool clear);
cudaError_t read_status_lnmerge_bf16(unsigned int* flags, bool clear);

// cudaOccupancyMaxActiveClusters of a planned register-holding cluster launch
// of a normalisation (plan.op).
cudaError_t norm_max_clusters_f32(const rs_plan& p, int* n);
cudaError_t norm_max_clusters_f16(const rs_plan& p, int* n);
cudaError_t norm_max_clusters_bf16(const rs_plan& p, int* n);
cudaError_t read_status_norm_f32(unsigned int* flags, bool clear);
cudaError_t read_status_norm_f16(unsigned int* flags, bool clear);
cudaError_t read_status_norm_bf16(unsigned int* flags, bool clear);

// The softmax of rows split by columns (rs_split.cu).  Pairs are float2
// {m, l}; the kernels use programmatic dependent launch unless `strict`.
struct SplitLaunch {
    int sm_count;
    int vec;      // elements per access: the 16-byte width, or 1 (element-wise)
    bool strict;  // launch in strict stream order
};
// ml[r * S + b] = the pair of columns [b * B, min(N, (b + 1) * B)) of row r.
cudaError_t launch_split_partial(const SplitLaunch& L, int dtype, const void* in, float2* ml, int64_t M, int N,
                                 int64_t ldi, int S, int B, cudaStream_t s);
// out[r] = the merge of the R pairs ml[r * sr + s * ss], s = 0 .. R - 1.
cudaError_t launch_split_merge(const SplitLaunch& L, const float2* ml, float2* out, int64_t R, int64_t sr, int64_t ss,
                               int64_t M, cudaStream_t s);
// y = exp(x - m) / l with (m, l) the merge of row r's R pairs as above.
cudaError_t launch_split_finish(const SplitLaunch& L, int dtype, const void* in, void* out, const float2* ml,
                                int64_t R, int64_t sr, int64_t ss, int64_t M, int N, int64_t ldi, int64_t ldo,
                                cudaStream_t s);
// Device address of the fixed scratch buffer (RS_SPLIT_NOALLOC_MAX_BYTES) of
// rowsoftmax_split_fwd_noalloc on the current device (rs_split.cu).
cudaError_t split_noalloc_scratch(void** ptr);

}  // namespace rs
