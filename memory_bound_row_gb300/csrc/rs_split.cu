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

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>

#include "rs_common.cuh"
#include "rs_internal.h"

namespace rs {

namespace {

constexpr int kSplitThreads = 256;  // threads per CTA of every kernel here
constexpr int kUnits = 8;           // 16-byte units a thread holds per pass (packed, unpacked one at a time)

// A unit's values as fp32: from the packed 16-byte word `raw` when it is a
// whole unit of the block (u < full), else read element by element (the
// ragged last unit), -inf past the block.  The block's reads use the
// read-only path with the default eviction priority, so that they stay in L2
// for a finish that follows.
template <int DT, int VEC>
__device__ __forceinline__ void unit_values(const uint4& raw, const typename Traits<DT>::storage* x, int u, int full,
                                            int len, float* f) {
    using T = Traits<DT>;
    if (VEC == T::kVec && u < full) {
        T::unpack(raw, f);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int j = u * VEC + e;
            f[e] = j < len ? load_param1<DT>(x + j) : kNegInf;
        }
    }
}

// -inf in both halves of a packed pair of 16-bit values.
template <int DT>
constexpr uint32_t neg_inf_pair() { return DT == RS_BF16 ? 0xFF80FF80u : 0xFC00FC00u; }

// Elementwise max of two packed pairs of 16-bit values (a NaN loses to the
// other operand, as in fmaxf).
template <int DT>
__device__ __forceinline__ uint32_t hmax_pair(uint32_t a, uint32_t b) {
    if constexpr (DT == RS_BF16) {
        const __nv_bfloat162 r =
            __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a), *reinterpret_cast<const __nv_bfloat162*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    } else {
        const __half2 r = __hmax2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
        return *reinterpret_cast<const uint32_t*>(&r);
    }
}

// Tree sum of a unit's values.
template <int VEC>
__device__ __forceinline__ float unit_sum(float (&f)[VEC]) {
#pragma unroll
    for (int h = VEC / 2; h > 0; h /= 2)
#pragma unroll
        for (int e = 0; e < h; ++e) f[e] += f[e + h];
    return f[0];
}

// (m, l) absorbs (m2, l2): the online normaliser's step.
__device__ __forceinline__ void absorb(float& m, float& l, float m2, float l2) {
    const float mn = fmaxf(m, m2);
    const float ms = safe_max(mn);
    l = l * rescale(m, ms) + l2 * rescale(m2, ms);
    m = mn;
}

// One pair per (row, block) item: item q = r * S + b covers columns
// [b * B, min(N, (b + 1) * B)) of row r and writes ml[q].  A group of TPI
// threads serves an item (TPI from 4 lanes to 8 warps, by the item's width);
// each thread takes units t, t + TPI, ... of the item, kUnits at a time: the
// loads of a pass are issued together and kept packed, then the pass's max
// raises the running m (rescaling l once) and its exponentials, summed as a
// tree, are added to l with compensated (Kahan) summation.
template <int DT, int VEC, int TPI>
__global__ void __launch_bounds__(kSplitThreads)
partial_kernel(const void* in_, float2* ml, int64_t M, int N, int64_t ldi, int S, int B) {
    using T = Traits<DT>;
    using St = typename T::storage;
    constexpr int kIpc = kSplitThreads / TPI;  // items a CTA serves at once
    constexpr int kWpi = TPI / 32;             // warps of an item (0: several items a warp)
    constexpr int kWidth = TPI < 32 ? TPI : 32;
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
            const int full = VEC == T::kVec ? len / VEC : 0;  // whole 16-byte units
            constexpr bool kPacked = VEC == T::kVec && DT != RS_F32;  // 16-bit words: the max on packed pairs
            constexpr uint32_t kFillWord = kPacked ? neg_inf_pair<DT>() : 0u;
            for (int u0 = t; u0 < units; u0 += kUnits * TPI) {
                uint4 raw[kUnits];
#pragma unroll
                for (int k = 0; k < kUnits; ++k) {
                    const int u = u0 + k * TPI;
                    raw[k] = u < full ? __ldg(reinterpret_cast<const uint4*>(x + u * VEC))
                                      : make_uint4(kFillWord, kFillWord, kFillWord, kFillWord);
                }
                float bm = kNegInf;
                if constexpr (kPacked) {
                    // whole units on packed pairs (the others hold -inf), then the
                    // item's ragged last unit, if this thread has it, element by element
                    uint32_t acc = neg_inf_pair<DT>();
#pragma unroll
                    for (int k = 0; k < kUnits; ++k) {
                        acc = hmax_pair<DT>(acc, raw[k].x);
                        acc = hmax_pair<DT>(acc, raw[k].y);
                        acc = hmax_pair<DT>(acc, raw[k].z);
                        acc = hmax_pair<DT>(acc, raw[k].w);
                    }
                    float two[2];
                    T::unpack2(acc, two);
                    bm = fmaxf(two[0], two[1]);
#pragma unroll
                    for (int k = 0; k < kUnits; ++k) {
                        const int u = u0 + k * TPI;
                        if (u >= full && u < units) {
                            float f[VEC];
                            unit_values<DT, VEC>(raw[k], x, u, full, len, f);
#pragma unroll
                            for (int e = 0; e < VEC; ++e) bm = fmaxf(bm, f[e]);
                        }
                    }
                } else {
#pragma unroll
                    for (int k = 0; k < kUnits; ++k) {
                        float f[VEC];
                        unit_values<DT, VEC>(raw[k], x, u0 + k * TPI, full, len, f);
#pragma unroll
                        for (int e = 0; e < VEC; ++e) bm = fmaxf(bm, f[e]);
                    }
                }
                if (bm > m) {
                    const float fac = rescale(m, bm);
                    l *= fac;
                    comp *= fac;
                    m = bm;
                }
                const float ms = safe_max(m);
                float us[kUnits];
#pragma unroll
                for (int k = 0; k < kUnits; ++k) {
                    float f[VEC];
                    unit_values<DT, VEC>(raw[k], x, u0 + k * TPI, full, len, f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) f[e] = exp_diff(f[e], ms);
                    us[k] = unit_sum<VEC>(f);
                }
#pragma unroll
                for (int h = kUnits / 2; h > 0; h /= 2)
#pragma unroll
                    for (int k = 0; k < h; ++k) us[k] += us[k + h];
                const float y = us[0] - comp;
                const float sum = l + y;
                comp = (sum - l) - y;
                l = sum;
            }
        }
        group_merge(m, l, kWidth);
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

// y = exp(x - m) / l.  A group of G lanes (4 to 32, by the row's width)
// serves one item, G * kUnits consecutive units of one row (lane j of the
// group holds units j, j + G, ...); the group merges its row's R pairs itself
// (G-lane butterflies, no CTA barrier), loads its units together, keeps them
// packed, and scales and stores them one at a time.
template <int DT, int VEC, int G>
__global__ void __launch_bounds__(kSplitThreads)
finish_kernel(const void* in_, void* out_, const float2* ml, int64_t R, int64_t sr, int64_t ss, int64_t M, int N,
              int64_t ldi, int64_t ldo) {
    using T = Traits<DT>;
    using St = typename T::storage;
    constexpr int kGpw = 32 / G;  // groups a warp
    const St* in = static_cast<const St*>(in_);
    St* out = static_cast<St*>(out_);
    const int lane = threadIdx.x & 31;
    const int t = lane % G;
    const int upr = (N + VEC - 1) / VEC;
    const int full = VEC == T::kVec ? N / VEC : 0;
    const int cpr = (upr + G * kUnits - 1) / (G * kUnits);  // items a row
    const int64_t items = M * (int64_t)cpr;
    const int64_t warps = (int64_t)gridDim.x * (kSplitThreads / 32);
    wait_prior_grid();
    for (int64_t wbase = ((int64_t)blockIdx.x * (kSplitThreads / 32) + (threadIdx.x >> 5)) * kGpw; wbase < items;
         wbase += warps * kGpw) {
        const int64_t gi = wbase + lane / G;
        const bool active = gi < items;
        const int64_t r = active ? gi / cpr : 0;
        const int c = active ? (int)(gi - r * cpr) : 0;
        float m = kNegInf, l = 0.0f;
        if (R == 1) {
            if (active) {
                const float2 p = ml[r * sr];
                m = p.x;
                l = p.y;
            }
        } else {
            if (active)
                for (int64_t s = t; s < R; s += G) {
                    const float2 p = ml[r * sr + s * ss];
                    absorb(m, l, p.x, p.y);
                }
            group_merge(m, l, G);
        }
        const float ms = safe_max(m);
        const float inv = 1.0f / l;
        const St* x = in + r * ldi;
        St* y = out + r * ldo;
        const int ub = c * G * kUnits + t;
        uint4 raw[kUnits];
#pragma unroll
        for (int k = 0; k < kUnits; ++k) {
            const int u = ub + k * G;
            raw[k] = active && u < full ? __ldcs(reinterpret_cast<const uint4*>(x + u * VEC)) : make_uint4(0, 0, 0, 0);
        }
        if (!active) continue;
#pragma unroll
        for (int k = 0; k < kUnits; ++k) {
            const int u = ub + k * G;
            if (u >= upr) break;
            float f[VEC];
            if (VEC == T::kVec && u < full) {
                T::unpack(raw[k], f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) f[e] = exp_diff(f[e], ms) * inv;
                __stcs(reinterpret_cast<uint4*>(y + u * VEC), T::pack(f));
            } else {
                load_unit<DT, VEC>(x, u * VEC, N, f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) f[e] = exp_diff(f[e], ms) * inv;
                store_unit<DT, VEC>(y, u * VEC, N, f);
            }
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

template <int DT, int VEC, int TPI>
cudaError_t launch_partial_one(const SplitLaunch& L, const void* in, float2* ml, int64_t M, int N, int64_t ldi, int S,
                               int B, cudaStream_t s) {
    constexpr int kIpc = kSplitThreads / TPI;
    const int64_t items = M * (int64_t)S;
    return launch_kernel(partial_kernel<DT, VEC, TPI>, grid_of(partial_kernel<DT, VEC, TPI>, (items + kIpc - 1) / kIpc,
                                                               L.sm_count),
                         kSplitThreads, 0, s, 0, L.strict, in, ml, M, N, ldi, S, B);
}

// Threads an item: enough for one pass of kUnits units a thread, 4 to 256.
template <int DT, int VEC>
cudaError_t launch_partial_vec(const SplitLaunch& L, const void* in, float2* ml, int64_t M, int N, int64_t ldi, int S,
                               int B, cudaStream_t s) {
    const int units = (B + VEC - 1) / VEC;
    if (units <= 4 * kUnits) return launch_partial_one<DT, VEC, 4>(L, in, ml, M, N, ldi, S, B, s);
    if (units <= 8 * kUnits) return launch_partial_one<DT, VEC, 8>(L, in, ml, M, N, ldi, S, B, s);
    if (units <= 16 * kUnits) return launch_partial_one<DT, VEC, 16>(L, in, ml, M, N, ldi, S, B, s);
    if (units <= 32 * kUnits) return launch_partial_one<DT, VEC, 32>(L, in, ml, M, N, ldi, S, B, s);
    if (units <= 64 * kUnits) return launch_partial_one<DT, VEC, 64>(L, in, ml, M, N, ldi, S, B, s);
    if (units <= 128 * kUnits) return launch_partial_one<DT, VEC, 128>(L, in, ml, M, N, ldi, S, B, s);
    return launch_partial_one<DT, VEC, 256>(L, in, ml, M, N, ldi, S, B, s);
}

template <int DT>
cudaError_t launch_partial_dt(const SplitLaunch& L, const void* in, float2* ml, int64_t M, int N, int64_t ldi, int S,
                              int B, cudaStream_t s) {
    if (L.vec > 1) return launch_partial_vec<DT, Traits<DT>::kVec>(L, in, ml, M, N, ldi, S, B, s);
    return launch_partial_vec<DT, 1>(L, in, ml, M, N, ldi, S, B, s);
}

template <int DT, int VEC, int G>
cudaError_t launch_finish_one(const SplitLaunch& L, const void* in, void* out, const float2* ml, int64_t R, int64_t sr,
                              int64_t ss, int64_t M, int N, int64_t ldi, int64_t ldo, cudaStream_t s) {
    const int64_t upr = (N + VEC - 1) / VEC;
    const int64_t items = M * ((upr + G * kUnits - 1) / (G * kUnits));
    const int64_t per_cta = (kSplitThreads / 32) * (32 / G);
    return launch_kernel(finish_kernel<DT, VEC, G>,
                         grid_of(finish_kernel<DT, VEC, G>, (items + per_cta - 1) / per_cta, L.sm_count),
                         kSplitThreads, 0, s, 0, L.strict, in, out, ml, R, sr, ss, M, N, ldi, ldo);
}

// Lanes an item: enough for one pass of kUnits units a lane over the row, 4 to 32.
template <int DT, int VEC>
cudaError_t launch_finish_vec(const SplitLaunch& L, const void* in, void* out, const float2* ml, int64_t R,
                              int64_t sr, int64_t ss, int64_t M, int N, int64_t ldi, int64_t ldo, cudaStream_t s) {
    const int64_t upr = (N + VEC - 1) / VEC;
    if (upr <= 4 * kUnits) return launch_finish_one<DT, VEC, 4>(L, in, out, ml, R, sr, ss, M, N, ldi, ldo, s);
    if (upr <= 8 * kUnits) return launch_finish_one<DT, VEC, 8>(L, in, out, ml, R, sr, ss, M, N, ldi, ldo, s);
    if (upr <= 16 * kUnits) return launch_finish_one<DT, VEC, 16>(L, in, out, ml, R, sr, ss, M, N, ldi, ldo, s);
    return launch_finish_one<DT, VEC, 32>(L, in, out, ml, R, sr, ss, M, N, ldi, ldo, s);
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
