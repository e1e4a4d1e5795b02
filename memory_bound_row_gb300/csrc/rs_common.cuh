// Device-side building blocks shared by the row-softmax kernels:
// storage-type traits, 16-byte and element-wise global accesses, the
// "safe max" used in every exp(x - m), and the warp reductions.
//
// Arithmetic is fp32 for every storage type (the "fp32 Accumulation" rule,
// Hugging Face "triton-kernels" skill page, "Numerics").
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "rowsoftmax.h"

namespace rs {

constexpr float kNegInf = -__builtin_inff();

// ---------------------------------------------------------------------------
// Storage traits.  kVec is the number of elements in one 16-byte access.
// ---------------------------------------------------------------------------
template <int DT> struct Traits;

template <> struct Traits<RS_F32> {
    using storage = float;
    static constexpr int kVec = 4;
    __device__ static __forceinline__ float load1(const storage* p) { return __ldcs(p); }
    __device__ static __forceinline__ void store1(storage* p, float v) { __stcs(p, v); }
    __device__ static __forceinline__ void unpack(const uint4& u, float* v) {
        v[0] = __uint_as_float(u.x); v[1] = __uint_as_float(u.y);
        v[2] = __uint_as_float(u.z); v[3] = __uint_as_float(u.w);
    }
    __device__ static __forceinline__ uint4 pack(const float* v) {
        return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                          __float_as_uint(v[2]), __float_as_uint(v[3]));
    }
};

template <> struct Traits<RS_BF16> {
    using storage = __nv_bfloat16;
    static constexpr int kVec = 8;
    // bf16 is the upper half of an fp32 bit pattern: widening is a shift.
    __device__ static __forceinline__ float widen(unsigned short b) {
        return __uint_as_float(((unsigned int)b) << 16);
    }
    __device__ static __forceinline__ float load1(const storage* p) {
        return widen(__ldcs(reinterpret_cast<const unsigned short*>(p)));
    }
    __device__ static __forceinline__ void store1(storage* p, float v) {
        __nv_bfloat16 b = __float2bfloat16_rn(v);
        __stcs(reinterpret_cast<unsigned short*>(p), *reinterpret_cast<unsigned short*>(&b));
    }
    __device__ static __forceinline__ void unpack2(unsigned int w, float* v) {
        v[0] = __uint_as_float(w << 16);
        v[1] = __uint_as_float(w & 0xffff0000u);
    }
    __device__ static __forceinline__ unsigned int pack2(float a, float b) {
        __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<unsigned int*>(&h);
    }
    __device__ static __forceinline__ void unpack(const uint4& u, float* v) {
        unpack2(u.x, v); unpack2(u.y, v + 2); unpack2(u.z, v + 4); unpack2(u.w, v + 6);
    }
    __device__ static __forceinline__ uint4 pack(const float* v) {
        return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
    }
};

template <> struct Traits<RS_F16> {
    using storage = __half;
    static constexpr int kVec = 8;
    __device__ static __forceinline__ float load1(const storage* p) {
        unsigned short b = __ldcs(reinterpret_cast<const unsigned short*>(p));
        return __half2float(*reinterpret_cast<__half*>(&b));
    }
    __device__ static __forceinline__ void store1(storage* p, float v) {
        __half h = __float2half_rn(v);
        __stcs(reinterpret_cast<unsigned short*>(p), *reinterpret_cast<unsigned short*>(&h));
    }
    __device__ static __forceinline__ void unpack2(unsigned int w, float* v) {
        float2 f = __half22float2(*reinterpret_cast<__half2*>(&w));
        v[0] = f.x; v[1] = f.y;
    }
    __device__ static __forceinline__ unsigned int pack2(float a, float b) {
        __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<unsigned int*>(&h);
    }
    __device__ static __forceinline__ void unpack(const uint4& u, float* v) {
        unpack2(u.x, v); unpack2(u.y, v + 2); unpack2(u.z, v + 4); unpack2(u.w, v + 6);
    }
    __device__ static __forceinline__ uint4 pack(const float* v) {
        return make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
    }
};

// ---------------------------------------------------------------------------
// Access of one "unit" of VEC elements starting at element `base` of a row:
// VEC == Traits::kVec is one 16-byte access (the caller guarantees alignment),
// VEC == 1 is one element.  Units that run past n are filled with `fill`
// (-inf for the softmax max, 0 for sums) on load and clipped on store,
// element by element (masked tail).
// ---------------------------------------------------------------------------
template <int DT, int VEC>
__device__ __forceinline__ void load_unit(const typename Traits<DT>::storage* row, int base, int n,
                                          float* v, float fill = kNegInf) {
    using T = Traits<DT>;
    if (VEC == T::kVec && base + VEC <= n) {
        T::unpack(__ldcs(reinterpret_cast<const uint4*>(row + base)), v);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[e] = (base + e < n) ? T::load1(row + base + e) : fill;
    }
}

// One element of a read-only parameter vector (a weight or a bias), kept in
// the caches: every row reads the same vector.
template <int DT>
__device__ __forceinline__ float load_param1(const typename Traits<DT>::storage* p) {
    if constexpr (DT == RS_F32) {
        return __ldg(p);
    } else if constexpr (DT == RS_BF16) {
        return __uint_as_float(((unsigned int)__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
    } else {
        unsigned short b = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __half2float(*reinterpret_cast<__half*>(&b));
    }
}

// The unit [base, base + VEC) of a parameter vector of n values; `dflt` for
// a null vector and past n.
template <int DT, int VEC>
__device__ __forceinline__ void load_param_unit(const void* vec, int base, int n, float* f, float dflt) {
    using T = Traits<DT>;
    using S = typename T::storage;
    if (!vec) {
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] = dflt;
        return;
    }
    const S* q = static_cast<const S*>(vec);
    if (VEC == T::kVec && base + VEC <= n) {
        T::unpack(__ldg(reinterpret_cast<const uint4*>(q + base)), f);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] = (base + e < n) ? load_param1<DT>(q + base + e) : dflt;
    }
}

template <int DT, int VEC>
__device__ __forceinline__ void store_unit(typename Traits<DT>::storage* row, int base, int n,
                                           const float* v) {
    using T = Traits<DT>;
    if (VEC == T::kVec && base + VEC <= n) {
        __stcs(reinterpret_cast<uint4*>(row + base), T::pack(v));
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (base + e < n) T::store1(row + base + e, v[e]);
    }
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel of this library is launched so
// that it may begin (be scheduled, set up shared memory and barriers) while
// the previous kernel of its stream is still finishing.  Before its first
// access to global memory it waits for that kernel to complete and for its
// writes to be visible, which keeps the stream's order; it then allows the
// next programmatically launched kernel of the stream to begin its own setup.
// Kernels launched without the attribute, or first in their stream, pass the
// wait at once.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void wait_prior_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_next_grid() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// exp(x - m) is always taken against safe(m): a max of -inf (a row, or part
// of one, with no finite entry) is replaced by 0 so that -inf entries give
// exp(-inf) = 0 instead of (-inf) - (-inf) = NaN.  Partial sums that belong
// to a -inf max carry weight 0 in a merge (0 * NaN stays NaN, so a NaN input
// still reaches the result).  A row with no finite entry ends with a zero
// sum, and 0 * (1/0) gives the NaN row that the plain formula gives.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float safe_max(float m) { return m == kNegInf ? 0.0f : m; }

// log2(e): exp(d) = 2^(d * log2(e)).
constexpr float kLog2e = 1.4426950408889634f;

// 2^y with the hardware base-2 exponential (PTX ex2.approx.ftz.f32: relative
// error about 2^-22; results below the smallest normal flush to zero, which
// is below every tolerance of this library).  2^(-inf) = 0, 2^NaN = NaN.
__device__ __forceinline__ float ex2_approx(float y) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

// exp(x - ms): the difference is formed first (exact when x is near ms),
// then scaled into base 2.
__device__ __forceinline__ float exp_diff(float x, float ms) { return ex2_approx((x - ms) * kLog2e); }

// Exponentials against a rounded base-2 offset (the register-holding kernels):
// with m a set's max, o = rn(m log2 e) and exp(x - m) taken as
// 2^fma(x, log2 e, -o) -- one FMA and one ex2 an element.  The values come
// out as exp(x - m) 2^r with r = m log2 e - o, the rounding residual of the
// offset, shared by the set.  The set's sum times 2^-r is its plain sum of
// exp(x - m), so sets merge as ordinary (m, l) pairs, and with M and L the
// row's merged pair the set's values scale by exp(m - M) 2^-r / L
// (rescale_res).  r is at most half a unit in the last place of o, which
// stays below 1/2 only while |m| < 2^23 (|o| < 2^24); past that (and for an
// infinite or NaN max) the set takes the difference form exp_diff, r = 0.
constexpr float kOffsetFormLimit = 8388608.0f;  // 2^23
__device__ __forceinline__ bool offset_form(float m) { return fabsf(m) < kOffsetFormLimit; }
__device__ __forceinline__ float exp_off(float x, float o) { return ex2_approx(fmaf(x, kLog2e, -o)); }
// The offset of a set with max m (offset_form(m) true) and its residual.
__device__ __forceinline__ float offset_of(float m) { return m * kLog2e; }
__device__ __forceinline__ float residual_of(float m, float o) { return fmaf(m, kLog2e, -o); }
// Weight of a set with max m and residual r inside a row whose merged max is
// ms (safe_max applied): exp(m - ms) 2^-r, 0 for a set with no mass.
__device__ __forceinline__ float rescale_res(float m, float ms, float r) {
    return m == kNegInf ? 0.0f : ex2_approx(fmaf(m - ms, kLog2e, -r));
}

// Weight of a partial sum taken against max m when the merged max is ms.
__device__ __forceinline__ float rescale(float m, float ms) {
    return m == kNegInf ? 0.0f : exp_diff(m, ms);
}

// Smallest power of two >= n (n in 1..32).
__device__ __forceinline__ int pow2_ceil(int n) { return n <= 1 ? 1 : 1 << (32 - __clz(n - 1)); }

// Reductions over aligned groups of `width` lanes (width a power of two, <= 32).
__device__ __forceinline__ float group_max(float v, int width) {
    for (int o = width >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float group_sum(float v, int width) {
    for (int o = width >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Online-normaliser merge of the (m, l) pairs of aligned groups of `width`
// lanes: m = max_i m_i, l = sum_i l_i * exp(m_i - m).  The max is reduced
// first, so each lane takes one exp rather than two per butterfly step.
__device__ __forceinline__ void group_merge(float& m, float& l, int width) {
    const float mm = group_max(m, width);
    l = group_sum(l * rescale(m, safe_max(mm)), width);
    m = mm;
}

}  // namespace rs
