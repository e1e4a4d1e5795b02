// The per-row arithmetic shared by RS_PATH_ROWS and RS_PATH_RING: a row is
// held in registers by the `tpr` threads of a row group, as VPT units of
// VEC fp32 values per thread (a fill value where the row has no element).
// The softmax below; RMSNorm and LayerNorm at the end, as row operations of
// the same engine.
//
// Three-level reduction as in the nano-triton post ("Reductions and
// broadcasting"): registers, then __shfl_xor_sync butterflies inside the
// warp, then (rows wider than a warp) one pair per warp through shared
// memory.  Each warp exponentiates against its own max m_w, and the warps'
// pairs (m_w, l_w) are merged with the online normaliser (mohakchugh.is-a.dev
// post, "How Flash Attention Uses Triton"): m = max m_w,
// l = sum l_w * exp(m_w - m).  The stored value is then exp(x - m_w) * c with
// c = exp(m_w - m) / l, i.e. exp(x - m) / l.
#pragma once

#include "rs_common.cuh"
#include "rs_internal.h"

namespace rs {

// Elements of row `row` that a causal mask keeps (N without a mask).  The
// remainder uses the host's reciprocal constant when row and period fit 32
// bits (two multiplications instead of a 64-bit division).
__device__ __forceinline__ int row_keep(const RowArgs& a, int64_t row, int N) {
    if (a.mask_period <= 0) return N;
    int64_t rm;
    if (((uint64_t)row >> 32) == 0 && ((uint64_t)a.mask_period >> 32) == 0)
        rm = (int64_t)__umul64hi(a.mask_magic * (uint64_t)row, (uint64_t)a.mask_period);
    else
        rm = row % a.mask_period;
    const int64_t L = rm + 1 + a.mask_offset;
    return L < 0 ? 0 : (L > N ? N : (int)L);
}

// Replaces v by exp(v - m_w) and returns the factor c with y = v * c.
// `part` is a per-iteration shared buffer of at least (blockDim.x / 32)
// pairs; rows wider than a warp synchronise the CTA once.
template <int VPT, int VEC>
__device__ __forceinline__ float row_exp_and_scale(float (&v)[VPT][VEC], int tpr, float2* part) {
    const int width = tpr < 32 ? tpr : 32;
    float m = kNegInf;
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
    m = group_max(m, width);
    const float ms = safe_max(m);

    float l = 0.0f;
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            v[k][e] = exp_diff(v[k][e], ms);
            l += v[k][e];
        }
    l = group_sum(l, width);
    if (tpr <= 32) return 1.0f / l;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wpr = tpr >> 5;  // warps of this row
    if (lane == 0) part[warp] = make_float2(m, l);
    __syncthreads();
    const int w0 = (warp / wpr) * wpr;
    const int ww = pow2_ceil(wpr);  // lanes 0..ww-1 merge the row's warp pairs
    float pm = kNegInf, pl = 0.0f;
    if (lane < wpr) {
        const float2 q = part[w0 + lane];
        pm = q.x;
        pl = q.y;
    }
    const float mrow = __shfl_sync(0xffffffffu, group_max(pm, ww), 0);
    const float mrs = safe_max(mrow);
    const float srow = __shfl_sync(0xffffffffu, group_sum(pl * rescale(pm, mrs), ww), 0);
    return rescale(m, mrs) / srow;
}

// Loads the thread's units t, t + tpr, ... of a row from global memory
// (16-byte units when VEC is the 16-byte width, else single elements);
// whole units take the branch-free path; `fill` stands for absent elements.
template <int DT, int VEC, int VPT>
__device__ __forceinline__ void load_row_units(const typename Traits<DT>::storage* row, int t, int tpr, int n,
                                               bool active, float (&v)[VPT][VEC], float fill = kNegInf) {
    if (active && (t + (VPT - 1) * tpr + 1) * VEC <= n) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (VEC == Traits<DT>::kVec) {
                Traits<DT>::unpack(__ldcs(reinterpret_cast<const uint4*>(row + (t + k * tpr) * VEC)), v[k]);
            } else {
                v[k][0] = Traits<DT>::load1(row + t + k * tpr);
            }
        }
    } else if (active) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) load_unit<DT, VEC>(row, (t + k * tpr) * VEC, n, v[k], fill);
    } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[k][e] = fill;
    }
}

// Stores v to the thread's units of a row (rounded to the storage type).
template <int DT, int VEC, int VPT>
__device__ __forceinline__ void store_row_units(typename Traits<DT>::storage* row, int t, int tpr, int n,
                                                const float (&v)[VPT][VEC]) {
    if ((t + (VPT - 1) * tpr + 1) * VEC <= n) {
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            if (VEC == Traits<DT>::kVec) {
                __stcs(reinterpret_cast<uint4*>(row + (t + k * tpr) * VEC), Traits<DT>::pack(v[k]));
            } else {
                Traits<DT>::store1(row + t + k * tpr, v[k][0]);
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k) store_unit<DT, VEC>(row, (t + k * tpr) * VEC, n, v[k]);
    }
}

// Stores v * c (the softmax's scaled values).
template <int DT, int VEC, int VPT>
__device__ __forceinline__ void store_row_units(typename Traits<DT>::storage* row, int t, int tpr, int n,
                                                float (&v)[VPT][VEC], float c) {
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[k][e] *= c;
    store_row_units<DT, VEC, VPT>(row, t, tpr, n, v);
}

// ---------------------------------------------------------------------------
// Row operations.  Each turns the thread's loaded units v (with kFill where the
// row has no element) into the values to store, cooperating with the other
// threads of the row through warp butterflies and, for rows wider than a warp,
// the per-warp pairs `part` (one CTA barrier per reduction).
// ---------------------------------------------------------------------------
// Sum over the threads of a row; SLOT picks the half of the per-warp pair.
template <int SLOT>
__device__ __forceinline__ float row_sum(float s, int tpr, float2* part) {
    const int width = tpr < 32 ? tpr : 32;
    s = group_sum(s, width);
    if (tpr <= 32) return s;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wpr = tpr >> 5;
    if (lane == 0) {
        if (SLOT == 0) part[warp].x = s; else part[warp].y = s;
    }
    __syncthreads();
    const int w0 = (warp / wpr) * wpr;
    float p = 0.0f;
    if (lane < wpr) p = SLOT == 0 ? part[w0 + lane].x : part[w0 + lane].y;
    return __shfl_sync(0xffffffffu, group_sum(p, pow2_ceil(wpr)), 0);
}

// Sum over the thread's values of acc' = f(acc, x, k, e), spread over up to
// eight independent accumulators (short dependency chains: the additions of
// different accumulators overlap in the pipeline), then added as a tree.
template <int VPT, int VEC, typename F>
__device__ __forceinline__ float thread_sum(const float (&v)[VPT][VEC], F f) {
    constexpr int n = VPT * VEC;
    constexpr int A = n >= 8 ? 8 : n >= 4 ? 4 : n >= 2 ? 2 : 1;
    float acc[A];
#pragma unroll
    for (int i = 0; i < A; ++i) acc[i] = 0.0f;
#pragma unroll
    for (int i = 0; i < n; ++i) acc[i % A] = f(acc[i % A], v[i / VEC][i % VEC], i / VEC, i % VEC);
#pragma unroll
    for (int h = A / 2; h > 0; h /= 2)
#pragma unroll
        for (int i = 0; i < h; ++i) acc[i] += acc[i + h];
    return acc[0];
}

// Where a normalisation reads its weight and bias units.  GlobalParams: the
// caller's vectors in global memory (read-only cache), with 1 and 0 for a
// null vector or past n.  SharedParams: copies staged once per CTA in shared
// memory by a persistent kernel, padded to whole 16-byte units with 1 and 0,
// read at unit offsets relative to the staged range.  HeldParams (below): a
// thread's own units in registers, read by unit index.
struct GlobalParams {
    const void* w;
    const void* b;
    float eps;
    int n;
    int offset;  // element of the vectors that unit offset 0 refers to
    template <int DT, int VEC>
    __device__ __forceinline__ void w_unit(int base, float* f) const {
        load_param_unit<DT, VEC>(w, offset + base, n, f, 1.0f);
    }
    template <int DT, int VEC>
    __device__ __forceinline__ void b_unit(int base, float* f) const {
        load_param_unit<DT, VEC>(b, offset + base, n, f, 0.0f);
    }
    template <int DT, int VEC>
    __device__ __forceinline__ void w_unit_k(int, int base, float* f) const { w_unit<DT, VEC>(base, f); }
    template <int DT, int VEC>
    __device__ __forceinline__ void b_unit_k(int, int base, float* f) const { b_unit<DT, VEC>(base, f); }
};

// The weight and bias units of a thread's VPT units held in registers as fp32
// (a persistent kernel whose threads serve the same columns of every row),
// read by unit index k.
template <int VPT, int VEC>
struct HeldParams {
    float w[VPT][VEC];
    float b[VPT][VEC];
    float eps;
    template <int DT, int V>
    __device__ __forceinline__ void w_unit_k(int k, int, float* f) const {
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] = w[k][e];
    }
    template <int DT, int V>
    __device__ __forceinline__ void b_unit_k(int k, int, float* f) const {
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] = b[k][e];
    }
};

template <int DT>
struct SharedParams {
    using S = typename Traits<DT>::storage;
    const S* w;  // shared memory, or null for weight 1
    const S* b;  // shared memory, or null for bias 0
    float eps;
    int padded;  // staged elements; units at or past it read 1 and 0
    template <int DT2, int VEC>
    __device__ __forceinline__ void w_unit(int base, float* f) const {
        static_assert(VEC == Traits<DT>::kVec, "staged parameters are read in whole units");
        if (w && base < padded) {
            Traits<DT>::unpack(*reinterpret_cast<const uint4*>(w + base), f);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) f[e] = 1.0f;
        }
    }
    template <int DT2, int VEC>
    __device__ __forceinline__ void b_unit(int base, float* f) const {
        static_assert(VEC == Traits<DT>::kVec, "staged parameters are read in whole units");
        if (b && base < padded) {
            Traits<DT>::unpack(*reinterpret_cast<const uint4*>(b + base), f);
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e) f[e] = 0.0f;
        }
    }
    template <int DT2, int VEC>
    __device__ __forceinline__ void w_unit_k(int, int base, float* f) const { w_unit<DT2, VEC>(base, f); }
    template <int DT2, int VEC>
    __device__ __forceinline__ void b_unit_k(int, int base, float* f) const { b_unit<DT2, VEC>(base, f); }
};

// Whether a row operation's weight and bias already sit in registers (then the
// LayerNorm epilogue stays scalar: packing held vectors into register pairs
// measured 10 % slower on bf16 32768 x 8192, by spills).
template <typename P> struct ParamsInRegisters { static constexpr bool value = false; };
template <int VPT, int VEC> struct ParamsInRegisters<HeldParams<VPT, VEC>> { static constexpr bool value = true; };

// Copies the elements [c0, c0 + len) of a parameter vector into shared memory
// `dst`, padded with `pad` up to `padded` elements (all threads of the CTA;
// the caller synchronises before reading).  A null source stages nothing.
template <int DT>
__device__ __forceinline__ void stage_param(typename Traits<DT>::storage* dst, const void* src, int c0, int len,
                                            int padded, float pad) {
    using S = typename Traits<DT>::storage;
    const S* q = static_cast<const S*>(src) + c0;
    S padv;
    if constexpr (DT == RS_F32) padv = pad;
    else if constexpr (DT == RS_BF16) padv = __float2bfloat16_rn(pad);
    else padv = __float2half_rn(pad);
    for (int i = threadIdx.x; i < padded; i += blockDim.x) dst[i] = i < len ? q[i] : padv;
}

struct OpSoftmax {
    static constexpr bool kHeldParams = false;
    static constexpr int kOp = RS_OP_SOFTMAX;
    static constexpr bool kMasked = false;
    static constexpr float kFill = kNegInf;
    template <int DT, int VEC, int VPT, typename P>
    __device__ static __forceinline__ void apply(float (&v)[VPT][VEC], int, int tpr, int, bool, const P&,
                                                 float2* part) {
        const float c = row_exp_and_scale<VPT, VEC>(v, tpr, part);
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[k][e] *= c;
    }
};

// Two fp32 lanes in one instruction (sub.rn.f32x2 and mul.rn.f32x2 on a
// 64-bit register pair, sm_100 and later): each lane rounds as the scalar
// instruction does, so the results are those of exp_diff and of v * c, at
// half the issue slots -- what the causal softmax's rows of one warp, bound
// by instruction issue rather than memory, gain from (bf16 1048576 x 2048
// causal scores: 1215 -> 1132 us).
__device__ __forceinline__ void pair_exp_diff(float& a, float& b, float ms) {
    float d0, d1;
    asm("{\n\t.reg .b64 x, y, r;\n\tmov.b64 x, {%2, %3};\n\tmov.b64 y, {%4, %4};\n\t"
        "sub.rn.f32x2 r, x, y;\n\tmov.b64 y, {%5, %5};\n\tmul.rn.f32x2 r, r, y;\n\tmov.b64 {%0, %1}, r;\n\t}"
        : "=f"(d0), "=f"(d1) : "f"(a), "f"(b), "f"(ms), "f"(kLog2e));
    a = ex2_approx(d0);
    b = ex2_approx(d1);
}
__device__ __forceinline__ void pair_mul(float& a, float& b, float c) {
    asm("{\n\t.reg .b64 x, y;\n\tmov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %2};\n\t"
        "mul.rn.f32x2 x, x, y;\n\tmov.b64 {%0, %1}, x;\n\t}"
        : "+f"(a), "+f"(b) : "f"(c));
}
// The normalisations' epilogues on a unit, in fp32 pairs (each lane rounds
// as the scalar expression does): RMSNorm (x r) w, LayerNorm
// fma(fma(x, r, nmr), w, b) with nmr = -mean r.  Measured against the scalar
// loops (same call): LayerNorm bf16 1048576 x 2048 +2.5 %, fp16 512 x 131072
// +3.2 %, RMSNorm +0.9 to +1.8 %, the rest unchanged.
__device__ __forceinline__ unsigned long long f2(float a, float b) {
    unsigned long long p;
    asm("mov.b64 %0, {%1, %2};" : "=l"(p) : "f"(a), "f"(b));
    return p;
}
__device__ __forceinline__ void f2_split(unsigned long long p, float& a, float& b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(p));
}
template <int VEC>
__device__ __forceinline__ void unit_rms(float (&f)[VEC], float r, const float (&w)[VEC]) {
    const unsigned long long rr = f2(r, r);
#pragma unroll
    for (int e = 0; e + 1 < VEC; e += 2) {
        unsigned long long x = f2(f[e], f[e + 1]);
        asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(x) : "l"(rr));
        asm("mul.rn.f32x2 %0, %0, %1;" : "+l"(x) : "l"(f2(w[e], w[e + 1])));
        f2_split(x, f[e], f[e + 1]);
    }
    if constexpr (VEC % 2 != 0) f[VEC - 1] = f[VEC - 1] * r * w[VEC - 1];
}
template <int VEC>
__device__ __forceinline__ void unit_ln(float (&f)[VEC], float r, float nmr, const float (&w)[VEC],
                                        const float (&b)[VEC]) {
    const unsigned long long rr = f2(r, r), nn = f2(nmr, nmr);
#pragma unroll
    for (int e = 0; e + 1 < VEC; e += 2) {
        unsigned long long x = f2(f[e], f[e + 1]);
        asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x) : "l"(rr), "l"(nn));
        asm("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x) : "l"(f2(w[e], w[e + 1])), "l"(f2(b[e], b[e + 1])));
        f2_split(x, f[e], f[e + 1]);
    }
    if constexpr (VEC % 2 != 0) f[VEC - 1] = fmaf(fmaf(f[VEC - 1], r, nmr), w[VEC - 1], b[VEC - 1]);
}

// A unit's values through exp_diff, and times c, in pairs (an odd last value alone).
template <int VEC>
__device__ __forceinline__ void unit_exp_diff(float (&f)[VEC], float ms) {
#pragma unroll
    for (int e = 0; e + 1 < VEC; e += 2) pair_exp_diff(f[e], f[e + 1], ms);
    if constexpr (VEC % 2 != 0) f[VEC - 1] = exp_diff(f[VEC - 1], ms);
}
template <int VEC>
__device__ __forceinline__ void unit_mul(float (&f)[VEC], float c) {
#pragma unroll
    for (int e = 0; e + 1 < VEC; e += 2) pair_mul(f[e], f[e + 1], c);
    if constexpr (VEC % 2 != 0) f[VEC - 1] *= c;
}

// The softmax under a causal mask (RowArgs::mask_period > 0): each row keeps
// a prefix (row_keep); the kernels copy and read only that prefix, and the rest
// of the row comes out as exactly 0 (NaN for a row that keeps nothing: an all
// -inf row).  `n` is the row's kept length.  Slot k of the row's threads
// covers elements [k tpr VEC, (k + 1) tpr VEC); the slots past the kept
// prefix hold only the fill, so their max, exponentials, sum and scaling are
// skipped (about half the arithmetic of a causal attention row), and only the
// last kept slot is masked element by element.  A separate type so that the
// unmasked kernels carry no mask code.
struct OpSoftmaxCausal : OpSoftmax {
    static constexpr bool kMasked = true;
    // The row's max and sum: leaves exp(x - m_w) in the kept slots (the fill
    // -inf elsewhere) and returns the scale c (finish applies it; a kernel may
    // fuse the scaling into its stores instead).
    template <int DT, int VEC, int VPT>
    __device__ static __forceinline__ float reduce(float (&v)[VPT][VEC], int tpr, int n, float2* part) {
        const int kk = (n + tpr * VEC - 1) / (tpr * VEC);  // slots holding a kept element
        const int width = tpr < 32 ? tpr : 32;
        float m = kNegInf;  // (the fill past the prefix is -inf: no effect on the max)
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
        m = group_max(m, width);
        const float ms = safe_max(m);
        float l = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
            if (k < kk) {
                unit_exp_diff<VEC>(v[k], ms);
#pragma unroll
                for (int e = 0; e < VEC; ++e) l += v[k][e];
            }
        l = group_sum(l, width);
        float c;
        if (tpr <= 32) {
            c = 1.0f / l;
        } else {
            const int warp = threadIdx.x >> 5;
            const int lane = threadIdx.x & 31;
            const int wpr = tpr >> 5;
            if (lane == 0) part[warp] = make_float2(m, l);
            __syncthreads();
            const int w0 = (warp / wpr) * wpr;
            const int ww = pow2_ceil(wpr);
            float pm = kNegInf, pl = 0.0f;
            if (lane < wpr) {
                const float2 q = part[w0 + lane];
                pm = q.x;
                pl = q.y;
            }
            const float mrow = __shfl_sync(0xffffffffu, group_max(pm, ww), 0);
            const float mrs = safe_max(mrow);
            const float srow = __shfl_sync(0xffffffffu, group_sum(pl * rescale(pm, mrs), ww), 0);
            c = rescale(m, mrs) / srow;
        }
        return c;
    }
    template <int DT, int VEC, int VPT>
    __device__ static __forceinline__ void finish(float (&v)[VPT][VEC], int t, int tpr, int n, float c) {
        const int kk = (n + tpr * VEC - 1) / (tpr * VEC);
        if (isfinite(c)) {
            // kept slots: exp(x - m) * c, which is 0 for the fill inside the
            // last kept slot; skipped slots: 0
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                unit_mul<VEC>(v[k], c);
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = k < kk ? v[k][e] : 0.0f;
            }
        } else {
            // a NaN or +inf in the prefix, or an empty prefix (rare): the kept
            // part as the formula gives it, the rest 0 (NaN without a prefix)
            const float masked = n > 0 ? 0.0f : __int_as_float(0x7fffffff);
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = (t + k * tpr) * VEC + e < n ? v[k][e] * c : masked;
        }
    }
    template <int DT, int VEC, int VPT, typename P>
    __device__ static __forceinline__ void apply(float (&v)[VPT][VEC], int t, int tpr, int n, bool, const P&,
                                                 float2* part) {
        finish<DT, VEC, VPT>(v, t, tpr, n, reduce<DT, VEC, VPT>(v, tpr, n, part));
    }
};

// RMSNorm ("Reference Kernel: RMSNorm", Hugging Face "triton-kernels" skill
// page): y = x * rsqrt(sum(x^2)/N + eps) * w, accumulated in fp32.
struct OpRmsNorm {
    static constexpr bool kHeldParams = false;
    static constexpr int kOp = RS_OP_RMSNORM;
    static constexpr bool kMasked = false;
    static constexpr float kFill = 0.0f;  // absent elements add nothing to the sum of squares
    template <int DT, int VEC, int VPT, typename P>
    __device__ static __forceinline__ void apply(float (&v)[VPT][VEC], int t, int tpr, int n, bool,
                                                 const P& a, float2* part) {
        float s = thread_sum<VPT, VEC>(v, [](float acc, float x, int, int) { return fmaf(x, x, acc); });
        s = row_sum<0>(s, tpr, part);
        const float r = 1.0f / sqrtf(s / (float)n + a.eps);
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            float w[VEC];
            a.template w_unit_k<DT, VEC>(k, (t + k * tpr) * VEC, w);
            unit_rms<VEC>(v[k], r, w);
        }
    }
};

// LayerNorm: y = (x - mean) * rsqrt(var + eps) * w + b, population variance,
// the two moments reduced one after the other (two passes over registers);
// the output is formed as ((x * r) - mean * r) * w + b with two FMAs.
struct OpLayerNorm {
    static constexpr bool kHeldParams = false;
    static constexpr int kOp = RS_OP_LAYERNORM;
    static constexpr bool kMasked = false;
    static constexpr float kFill = 0.0f;
    template <int DT, int VEC, int VPT, typename P>
    __device__ static __forceinline__ void apply(float (&v)[VPT][VEC], int t, int tpr, int n, bool whole,
                                                 const P& a, float2* part) {
        float s = thread_sum<VPT, VEC>(v, [](float acc, float x, int, int) { return acc + x; });
        const float mean = row_sum<0>(s, tpr, part) / (float)n;
        float d;
        if (whole) {
            d = thread_sum<VPT, VEC>(v, [mean](float acc, float x, int, int) {
                const float c = x - mean;
                return fmaf(c, c, acc);
            });
        } else {  // absent elements hold 0, not the mean: leave them out
            d = thread_sum<VPT, VEC>(v, [mean, t, tpr, n](float acc, float x, int k, int e) {
                const float c = x - mean;
                return (t + k * tpr) * VEC + e < n ? fmaf(c, c, acc) : acc;
            });
        }
        const float var = row_sum<1>(d, tpr, part) / (float)n;
        const float r = 1.0f / sqrtf(var + a.eps);
        const float nmr = -mean * r;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            float w[VEC], b[VEC];
            a.template w_unit_k<DT, VEC>(k, (t + k * tpr) * VEC, w);
            a.template b_unit_k<DT, VEC>(k, (t + k * tpr) * VEC, b);
            if constexpr (ParamsInRegisters<P>::value) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = fmaf(fmaf(v[k][e], r, nmr), w[e], b[e]);
            } else {
                unit_ln<VEC>(v[k], r, nmr, w, b);
            }
        }
    }
};

// Moments of a set of row values: count c, sum s and the sum q of squared
// deviations from the set's own mean s / c.  Two disjoint sets merge into
// their union by the parallel-variance identity (Chan, Golub and LeVeque,
// "Updating formulae and a pairwise algorithm for computing sample
// variances"):
//   q = q_a + q_b + (s_b c_a - s_a c_b)^2 / (c_a c_b (c_a + c_b)).
// The expression is symmetric in a and b to the bit (products rounded
// separately, then subtracted), so both lanes of a butterfly step agree.
__device__ __forceinline__ void merge_moments(float& c, float& s, float& q, float co, float so, float qo) {
    const float cross = __fmul_rn(so, c) - __fmul_rn(s, co);
    const float cc = __fmul_rn(c, co);
    const float t = cc > 0.0f ? __fdividef(__fmul_rn(cross, cross), __fmul_rn(cc, c + co)) : 0.0f;
    q = (q + qo) + t;
    s = s + so;
    c = c + co;
}

// Butterfly over aligned groups of `width` lanes (a power of two, at most 32)
// whose lanes' sets all hold the same count c: each step's correction is
// (s_b - s_a)^2 / (2c), with k = 1 / (2c) on entry, halved as c doubles.
__device__ __forceinline__ void equal_moments(float& s, float& q, float k, int width) {
    for (int o = 1; o < width; o <<= 1) {
        const float so = __shfl_xor_sync(0xffffffffu, s, o);
        const float qo = __shfl_xor_sync(0xffffffffu, q, o);
        const float d = so - s;
        q = fmaf(__fmul_rn(d, d), k, q + qo);
        s = s + so;
        k *= 0.5f;
    }
}

// Moments (s, q) of a row held by an aligned group of `width` lanes (a power
// of two, at most 32) from each lane's (c, s, q): the equal-count butterfly
// when every lane holds VPT * VEC values, else the general merge.
template <int VPT, int VEC>
__device__ __forceinline__ void group_moments(float& s, float& q, float c, int width) {
    if (__all_sync(0xffffffffu, c == (float)(VPT * VEC))) {
        equal_moments(s, q, 0.5f / (float)(VPT * VEC), width);
    } else {
        for (int o = 1; o < width; o <<= 1) {
            const float co = __shfl_xor_sync(0xffffffffu, c, o);
            const float so = __shfl_xor_sync(0xffffffffu, s, o);
            const float qo = __shfl_xor_sync(0xffffffffu, q, o);
            merge_moments(c, s, q, co, so, qo);
        }
    }
}

// The LayerNorm output from the row's moments: ((x * r) - mean * r) * w + b.
template <int DT, int VEC, int VPT, typename P>
__device__ __forceinline__ void layernorm_out(float (&v)[VPT][VEC], int t, int tpr, int n, float s, float q,
                                              const P& a) {
    const float mean = s / (float)n;
    const float r = 1.0f / sqrtf(q / (float)n + a.eps);
    const float nmr = -mean * r;
#pragma unroll
    for (int k = 0; k < VPT; ++k) {
        float w[VEC], b[VEC];
        a.template w_unit_k<DT, VEC>(k, (t + k * tpr) * VEC, w);
        a.template b_unit_k<DT, VEC>(k, (t + k * tpr) * VEC, b);
        if constexpr (ParamsInRegisters<P>::value) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[k][e] = fmaf(fmaf(v[k][e], r, nmr), w[e], b[e]);
        } else {
            unit_ln<VEC>(v[k], r, nmr, w, b);
        }
    }
}

// A lane's moments about its own mean when all VPT * VEC of its values lie in
// the row.
template <int VPT, int VEC>
__device__ __forceinline__ float whole_deviations(const float (&v)[VPT][VEC], float s) {
    const float mt = s * (1.0f / (float)(VPT * VEC));
    return thread_sum<VPT, VEC>(v, [mt](float acc, float x, int, int) {
        const float d = x - mt;
        return fmaf(d, d, acc);
    });
}

// LayerNorm for rows held inside one warp (tpr a power of two, at most 32):
// each lane takes the moments of its own values about its own mean, with no
// communication, and one butterfly merges them (OpLayerNorm reduces the mean
// first and then the deviations from it: two dependent reductions a row).
struct OpLayerNormWarp {
    static constexpr bool kHeldParams = false;
    static constexpr int kOp = RS_OP_LAYERNORM;
    static constexpr bool kMasked = false;
    static constexpr float kFill = 0.0f;
    template <int DT, int VEC, int VPT, typename P>
    __device__ static __forceinline__ void apply(float (&v)[VPT][VEC], int t, int tpr, int n, bool whole,
                                                 const P& a, float2*) {
        float s = thread_sum<VPT, VEC>(v, [](float acc, float x, int, int) { return acc + x; });
        float c, q;
        if (whole) {
            c = (float)(VPT * VEC);
            q = whole_deviations<VPT, VEC>(v, s);
        } else {  // absent elements hold 0, not the mean: leave them out
            // U whole units, the partial one (n mod VEC elements) held by lane
            // U mod tpr; lane t holds U / tpr whole units, one more if t < U mod tpr.
            const int U = n / VEC;
            const int rem = n - U * VEC;
            const int r = U & (tpr - 1);
            c = (float)(VEC * ((U >> (__popc(tpr - 1))) + (t < r ? 1 : 0)) + (t == r ? rem : 0));
            const float mt = c > 0.0f ? __fdividef(s, c) : 0.0f;
            q = thread_sum<VPT, VEC>(v, [mt, t, tpr, n](float acc, float x, int k, int e) {
                const float d = x - mt;
                return (t + k * tpr) * VEC + e < n ? fmaf(d, d, acc) : acc;
            });
        }
        group_moments<VPT, VEC>(s, q, c, tpr);
        layernorm_out<DT, VEC, VPT>(v, t, tpr, n, s, q, a);
    }
};

// LayerNorm for rows that fill their threads exactly (n = tpr * VPT * VEC)
// over a power-of-two number of warps: every lane, and every warp, holds the
// same count, so the lanes' moments merge in the equal-count butterfly inside
// each warp and again across the row's warps (one CTA barrier a row).
struct OpLayerNormWhole {
    static constexpr bool kHeldParams = false;
    static constexpr int kOp = RS_OP_LAYERNORM;
    static constexpr bool kMasked = false;
    static constexpr float kFill = 0.0f;
    template <int DT, int VEC, int VPT, typename P>
    __device__ static __forceinline__ void apply(float (&v)[VPT][VEC], int t, int tpr, int n, bool,
                                                 const P& a, float2* part) {
        float s = thread_sum<VPT, VEC>(v, [](float acc, float x, int, int) { return acc + x; });
        float q = whole_deviations<VPT, VEC>(v, s);
        equal_moments(s, q, 0.5f / (float)(VPT * VEC), 32);
        const int warp = threadIdx.x >> 5;
        const int lane = threadIdx.x & 31;
        const int wpr = tpr >> 5;
        if (lane == 0) part[warp] = make_float2(s, q);
        __syncthreads();
        const float2 p = lane < wpr ? part[(warp / wpr) * wpr + lane] : make_float2(0.0f, 0.0f);
        float sj = p.x, qj = p.y;
        equal_moments(sj, qj, 0.5f / (float)(32 * VPT * VEC), wpr);
        s = __shfl_sync(0xffffffffu, sj, 0);
        q = __shfl_sync(0xffffffffu, qj, 0);
        layernorm_out<DT, VEC, VPT>(v, t, tpr, n, s, q, a);
    }
};

// OpLayerNorm reading its weight and bias from registers (HeldParams).
struct OpLayerNormHeld : OpLayerNorm {
    static constexpr bool kHeldParams = true;
};

// OpRmsNorm reading its weight from registers (HeldParams).
struct OpRmsNormHeld : OpRmsNorm {
    static constexpr bool kHeldParams = true;
};

// OpLayerNormWhole reading its weight and bias from registers (HeldParams).
struct OpLayerNormWholeHeld : OpLayerNormWhole {
    static constexpr bool kHeldParams = true;
};

}  // namespace rs
