// The per-row arithmetic shared by RS_PATH_ROWS and RS_PATH_RING: a row is
// held in registers by the `tpr` threads of a row group, as VPT units of
// VEC fp32 values per thread (-inf where the row has no element).
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

namespace rs {

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
// whole units take the branch-free path.
template <int DT, int VEC, int VPT>
__device__ __forceinline__ void load_row_units(const typename Traits<DT>::storage* row, int t, int tpr, int n,
                                               bool active, float (&v)[VPT][VEC]) {
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
        for (int k = 0; k < VPT; ++k) load_unit<DT, VEC>(row, (t + k * tpr) * VEC, n, v[k]);
    } else {
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) v[k][e] = kNegInf;
    }
}

// Stores v * c to the thread's units of a row.
template <int DT, int VEC, int VPT>
__device__ __forceinline__ void store_row_units(typename Traits<DT>::storage* row, int t, int tpr, int n,
                                                float (&v)[VPT][VEC], float c) {
#pragma unroll
    for (int k = 0; k < VPT; ++k)
#pragma unroll
        for (int e = 0; e < VEC; ++e) v[k][e] *= c;
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

}  // namespace rs
