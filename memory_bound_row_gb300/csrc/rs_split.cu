// The softmax of rows split by columns into blocks (shards), in three steps:
//
//   partial  each (row, block) item reduces its columns to a pair (m, l):
//            m the max, l the sum of exp(x - m);
//   merge    the R pairs of a row are combined with the online normaliser of
//            the mohakchugh.is-a.dev post ("How Flash Attention Uses Triton"):
//            m = max(m1, m2), l = l1 exp(m1 - m) + l2 exp(m2 - m);
//   finish   every column of the row becomes exp(x - m) / l.
//
// The shards may live on different devices (the vocabulary-parallel softmax:
// each device reduces its block of columns, the pairs are exchanged, each
// device finishes its block), or be blocks of a few very wide rows on one
// device, so that every multiprocessor takes part (rowsoftmax_split_fwd).
// Pairs are float2 {m, l} in the natural-log domain: m + log(l) is the log of
// the sum of exp over the shard.
//
// Conventions (those of the row kernels): exp(x - m) is taken against
// safe_max(m), so a block whose entries are all -inf (or that has no column)
// gives the starting pair (-inf, 0); a pair whose max is -inf enters a merge
// with weight 0 times its sum (a NaN sum still propagates); NaN entries never
// win the max and make the sum NaN; a row whose merged max is -inf finishes
// as NaN, the plain formula's all -inf row.  Arithmetic is fp32, the
// exponential the hardware base-2 one on (x - m) log2 e.
#include <cuda_runtime.h>

#include <mutex>

#include "rs_common.cuh"
#include "rs_internal.h"

namespace rs {

namespace {

constexpr int kSplitThreads = 256;  // threads per CTA of every kernel here
constexpr int kPartialBatch = 4;    // units a thread loads before it reduces them
constexpr int kFinishUnits = 4;     // units a lane of a finishing warp holds

// A unit of a block, read so that it stays in L2 for a finish that follows
// (the read-only path with the default eviction priority); -inf past n.
template <int DT, int VEC>
__device__ __forceinline__ void load_unit_keep(const typename Traits<DT>::storage* row, int base, int n, float* v) {
    using T = Traits<DT>;
    if (VEC == T::kVec && base + VEC <= n) {
        T::unpack(__ldg(reinterpret_cast<const uint4*>(row + base)), v);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[e] = base + e < n ? load_param1<DT>(row + base + e) : kNegInf;
    }
}

// (m, l) absorbs (m2, l2): the online normaliser's step.
__device__ __forceinline__ void absorb(float& m, float& l, float m2, float l2) {
    const float mn = fmaxf(m, m2);
    const float ms = safe_max(mn);
    l = l * rescale(m, ms) + l2 * rescale(m2, ms);
    m = mn;
}

// The merged pair of row r from its R pairs at ml[r * sr + s * ss], the same
// in every lane of the warp.
__device__ __forceinline__ float2 warp_merged_pair(const float2* ml, int64_t r, int64_t R, int64_t sr, int64_t ss,
                                                   int lane) {
    if (R == 1) return ml[r * sr];
    float m = kNegInf, l = 0.0f;
    for (int64_t s = lane; s < R; s += 32) {
        const float2 p = ml[r * sr + s * ss];
        absorb(m, l, p.x, p.y);
    }
    group_merge(m, l, 32);
    return make_float2(m, l);
}

// Sum of a batch's values as a tree (short rounding chains).
template <int B, int VEC>
__device__ __forceinline__ float batch_sum(const float (&v)[B][VEC]) {
    float u[B];
#pragma unroll
    for (int k = 0; k < B; ++k) {
        float w[VEC];
#pragma unroll
        for (int e = 0; e < VEC; ++e) w[e] = v[k][e];
#pragma unroll
        for (int h = VEC / 2; h > 0; h /= 2)
#pragma unroll
            for (int e = 0; e < h; ++e) w[e] += w[e + h];
        u[k] = w[0];
    }
#pragma unroll
    for (int h = B / 2; h > 0; h /= 2)
#pragma unroll
        for (int k = 0; k < h; ++k) u[k] += u[k + h];
    return u[0];
}

// One pair per (row, block) item: item q = r * S + b covers columns
// [b * B, min(N, (b + 1) * B)) of row r and writes ml[q].  TPI threads serve
// an item (256 / TPI items a CTA at a time); each thread takes units t,
// t + TPI, ... of the item, kPartialBatch at a time, and keeps a running
// (m, l): a batch's max raises m (rescaling l once), then the batch's exps,
// summed as a tree, are added to l with compensated (Kahan) summation, so
// that a thread's long run of batches adds no more than a few roundings.
template <int DT, int VEC, int TPI>
__global__ void __launch_bounds__(kSplitThreads)
partial_kernel(const void* in_, float2* ml, int64_t M, int N, int64_t ldi, int S, int B) {
    using T = Traits<DT>;
    using St = typename T::storage;
    constexpr int kIpc = kSplitThreads / TPI;  // items a CTA serves at once
    constexpr int kWpi = TPI / 32;             // warps of an item
    const St* in = static_cast<const St*>(in_);
    __shared__ float2 part[2][kSplitThreads / 32];

    const int sub = threadIdx.x / TPI;
    const int t = threadIdx.x - sub * TPI;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int64_t items = M * (int64_t)S;
    wait_prior_grid();

    int it = 0;
    for (int64_t g = blockIdx.x; g * kIpc < items; g += gridDim.x, ++it) {
        const int64_t q = g * kIpc + sub;
        float m = kNegInf, l = 0.0f;
        float comp = 0.0f;  // the compensation of l's running sum
        if (q < items) {
            const int64_t r = q / S;
            const int64_t c0 = (q - r * S) * (int64_t)B;
            const int len = c0 >= N ? 0 : (int)(c0 + B < N ? B : N - c0);
            const St* x = in + r * ldi + c0;
            const int units = (len + VEC - 1) / VEC;
            for (int u0 = t; u0 < units; u0 += kPartialBatch * TPI) {
                float v[kPartialBatch][VEC];
#pragma unroll
                for (int k = 0; k < kPartialBatch; ++k) {
                    const int u = u0 + k * TPI;
                    if (u < units) {
                        load_unit_keep<DT, VEC>(x, u * VEC, len, v[k]);
                    } else {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) v[k][e] = kNegInf;
                    }
                }
                float bm = kNegInf;
#pragma unroll
                for (int k = 0; k < kPartialBatch; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) bm = fmaxf(bm, v[k][e]);
                if (bm > m) {
                    const float f = rescale(m, bm);
                    l *= f;
                    comp *= f;
                    m = bm;
                }
                const float ms = safe_max(m);
#pragma unroll
                for (int k = 0; k < kPartialBatch; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[k][e] = exp_diff(v[k][e], ms);
                const float y = batch_sum<kPartialBatch, VEC>(v) - comp;
                const float sum = l + y;
                comp = (sum - l) - y;
                l = sum;
            }
        }
        group_merge(m, l, 32);
        if constexpr (kWpi > 1) {
            float2* p = part[it & 1];
            if (lane == 0) p[warp] = make_float2(m, l);
            __syncthreads();
            const int w0 = (warp / kWpi) * kWpi;
            float pm = kNegInf, pl = 0.0f;
            if (lane < kWpi) {
                const float2 pr = p[w0 + lane];
                pm = pr.x;
                pl = pr.y;
            }
            group_merge(pm, pl, kWpi);
            m = pm;
            l = pl;
        }
        if (t == 0 && q < items) ml[q] = make_float2(m, l);
    }
    allow_next_grid();
}

// One CTA per row: out[r] = the merge of the R pairs ml[r * sr + s * ss]
// (R / 256 a thread, then warp butterflies and the CTA's warps: a tree).
__global__ void __launch_bounds__(kSplitThreads)
merge_kernel(const float2* ml, float2* out, int64_t R, int64_t sr, int64_t ss, int64_t M) {
    __shared__ float2 part[2][kSplitThreads / 32];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    wait_prior_grid();
    int it = 0;
    for (int64_t r = blockIdx.x; r < M; r += gridDim.x, ++it) {
        float m = kNegInf, l = 0.0f;
        for (int64_t s = threadIdx.x; s < R; s += kSplitThreads) {
            const float2 p = ml[r * sr + s * ss];
            absorb(m, l, p.x, p.y);
        }
        group_merge(m, l, 32);
        if (lane == 0) part[it & 1][warp] = make_float2(m, l);
        __syncthreads();
        if (warp == 0) {
            float pm = kNegInf, pl = 0.0f;
            if (lane < kSplitThreads / 32) {
                const float2 p = part[it & 1][lane];
                pm = p.x;
                pl = p.y;
            }
            group_merge(pm, pl, kSplitThreads / 32);
            if (lane == 0) out[r] = make_float2(pm, pl);
        }
    }
    allow_next_grid();
}

// y = exp(x - m) / l.  A warp item is 32 * kFinishUnits consecutive units of
// one row (lane j holds units j, j + 32, ...); every warp merges its row's R
// pairs itself (shuffles, no CTA barrier).
template <int DT, int VEC>
__global__ void __launch_bounds__(kSplitThreads)
finish_kernel(const void* in_, void* out_, const float2* ml, int64_t R, int64_t sr, int64_t ss, int64_t M, int N,
              int64_t ldi, int64_t ldo) {
    using T = Traits<DT>;
    using St = typename T::storage;
    const St* in = static_cast<const St*>(in_);
    St* out = static_cast<St*>(out_);
    const int lane = threadIdx.x & 31;
    const int upr = (N + VEC - 1) / VEC;
    const int cpr = (upr + 32 * kFinishUnits - 1) / (32 * kFinishUnits);  // warp items a row
    const int64_t items = M * (int64_t)cpr;
    const int64_t warps = (int64_t)gridDim.x * (kSplitThreads / 32);
    wait_prior_grid();
    for (int64_t w = (int64_t)blockIdx.x * (kSplitThreads / 32) + (threadIdx.x >> 5); w < items; w += warps) {
        const int64_t r = w / cpr;
        const int c = (int)(w - r * cpr);
        const float2 p = warp_merged_pair(ml, r, R, sr, ss, lane);
        const float ms = safe_max(p.x);
        const float inv = 1.0f / p.y;
        const St* x = in + r * ldi;
        St* y = out + r * ldo;
        const int ub = c * 32 * kFinishUnits + lane;
        float v[kFinishUnits][VEC];
#pragma unroll
        for (int k = 0; k < kFinishUnits; ++k) {
            const int u = ub + k * 32;
            if (u < upr) {
                load_unit<DT, VEC>(x, u * VEC, N, v[k]);
            } else {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = kNegInf;
            }
        }
#pragma unroll
        for (int k = 0; k < kFinishUnits; ++k) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[k][e] = exp_diff(v[k][e], ms) * inv;
            const int u = ub + k * 32;
            if (u < upr) store_unit<DT, VEC>(y, u * VEC, N, v[k]);
        }
    }
    allow_next_grid();
}

// CTAs of `kern` resident on one multiprocessor, queried once per device.
template <typename K>
int resident_ctas(K kern) {
    static std::mutex mu;
    static int known[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return 1;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!known[dev]) {
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kSplitThreads, 0) != cudaSuccess || n < 1) {
            (void)cudaGetLastError();
            n = 1;
        }
        known[dev] = n;
    }
    return known[dev];
}

// A grid-stride launch: `work` CTAs' worth of items, at most one wave of
// resident CTAs.
template <typename K>
unsigned grid_of(K kern, int64_t work, int sm_count) {
    const int64_t cap = (int64_t)sm_count * resident_ctas(kern);
    return (unsigned)(work < cap ? (work < 1 ? 1 : work) : cap);
}

template <int DT, int VEC>
cudaError_t launch_partial_vec(const SplitLaunch& L, const void* in, float2* ml, int64_t M, int N, int64_t ldi, int S,
                               int B, cudaStream_t s) {
    const int units = (B + VEC - 1) / VEC;
    const int64_t items = M * (int64_t)S;
    if (units <= 256) {
        return launch_kernel(partial_kernel<DT, VEC, 32>, grid_of(partial_kernel<DT, VEC, 32>, (items + 7) / 8, L.sm_count),
                             kSplitThreads, 0, s, 0, L.strict, in, ml, M, N, ldi, S, B);
    }
    if (units <= 512) {
        return launch_kernel(partial_kernel<DT, VEC, 64>, grid_of(partial_kernel<DT, VEC, 64>, (items + 3) / 4, L.sm_count),
                             kSplitThreads, 0, s, 0, L.strict, in, ml, M, N, ldi, S, B);
    }
    if (units <= 1024) {
        return launch_kernel(partial_kernel<DT, VEC, 128>, grid_of(partial_kernel<DT, VEC, 128>, (items + 1) / 2, L.sm_count),
                             kSplitThreads, 0, s, 0, L.strict, in, ml, M, N, ldi, S, B);
    }
    return launch_kernel(partial_kernel<DT, VEC, 256>, grid_of(partial_kernel<DT, VEC, 256>, items, L.sm_count),
                         kSplitThreads, 0, s,
                         0, L.strict, in, ml, M, N, ldi, S, B);
}

template <int DT>
cudaError_t launch_partial_dt(const SplitLaunch& L, const void* in, float2* ml, int64_t M, int N, int64_t ldi, int S,
                              int B, cudaStream_t s) {
    if (L.vec > 1) return launch_partial_vec<DT, Traits<DT>::kVec>(L, in, ml, M, N, ldi, S, B, s);
    return launch_partial_vec<DT, 1>(L, in, ml, M, N, ldi, S, B, s);
}

template <int DT, int VEC>
cudaError_t launch_finish_vec(const SplitLaunch& L, const void* in, void* out, const float2* ml, int64_t R,
                              int64_t sr, int64_t ss, int64_t M, int N, int64_t ldi, int64_t ldo, cudaStream_t s) {
    const int64_t upr = (N + VEC - 1) / VEC;
    const int64_t items = M * ((upr + 32 * kFinishUnits - 1) / (32 * kFinishUnits));
    return launch_kernel(finish_kernel<DT, VEC>, grid_of(finish_kernel<DT, VEC>, (items + 7) / 8, L.sm_count),
                         kSplitThreads, 0, s, 0, L.strict, in, out, ml, R, sr, ss, M, N, ldi, ldo);
}

template <int DT>
cudaError_t launch_finish_dt(const SplitLaunch& L, const void* in, void* out, const float2* ml, int64_t R,
                             int64_t sr, int64_t ss, int64_t M, int N, int64_t ldi, int64_t ldo, cudaStream_t s) {
    if (L.vec > 1) return launch_finish_vec<DT, Traits<DT>::kVec>(L, in, out, ml, R, sr, ss, M, N, ldi, ldo, s);
    return launch_finish_vec<DT, 1>(L, in, out, ml, R, sr, ss, M, N, ldi, ldo, s);
}

// Scratch of rowsoftmax_split_fwd_noalloc: a fixed device buffer that every
// GPU which loads this library holds until the process exits, for callers
// that cannot allocate device memory.
static __device__ __align__(256) unsigned char g_split_noalloc_scratch[RS_SPLIT_NOALLOC_MAX_BYTES];

}  // namespace

// The device address of the fixed scratch buffer on the current device.  The
// name of a __device__ array in host code is only a host-side stand-in, so the
// address is looked up with cudaGetSymbolAddress, once per device, with that
// device current, and kept.
cudaError_t split_noalloc_scratch(void** ptr) {
    static std::mutex mu;
    static void* addr[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        err = cudaGetSymbolAddress(&p, g_split_noalloc_scratch);
        if (err != cudaSuccess) return err;
        addr[dev] = p;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

cudaError_t launch_split_partial(const SplitLaunch& L, int dtype, const void* in, float2* ml, int64_t M, int N,
                                 int64_t ldi, int S, int B, cudaStream_t s) {
    switch (dtype) {
        case RS_F32: return launch_partial_dt<RS_F32>(L, in, ml, M, N, ldi, S, B, s);
        case RS_F16: return launch_partial_dt<RS_F16>(L, in, ml, M, N, ldi, S, B, s);
        default: return launch_partial_dt<RS_BF16>(L, in, ml, M, N, ldi, S, B, s);
    }
}

cudaError_t launch_split_merge(const SplitLaunch& L, const float2* ml, float2* out, int64_t R, int64_t sr, int64_t ss,
                               int64_t M, cudaStream_t s) {
    return launch_kernel(merge_kernel, grid_of(merge_kernel, M, L.sm_count), kSplitThreads, 0, s, 0, L.strict,
                         ml, out, R, sr, ss, M);
}

cudaError_t launch_split_finish(const SplitLaunch& L, int dtype, const void* in, void* out, const float2* ml,
                                int64_t R, int64_t sr, int64_t ss, int64_t M, int N, int64_t ldi, int64_t ldo,
                                cudaStream_t s) {
    switch (dtype) {
        case RS_F32: return launch_finish_dt<RS_F32>(L, in, out, ml, R, sr, ss, M, N, ldi, ldo, s);
        case RS_F16: return launch_finish_dt<RS_F16>(L, in, out, ml, R, sr, ss, M, N, ldi, ldo, s);
        default: return launch_finish_dt<RS_BF16>(L, in, out, ml, R, sr, ss, M, N, ldi, ldo, s);
    }
}

}  // namespace rs
