// RS_PATH_ROWS: single-pass row softmax with the whole row in registers.
//
// This is the fused kernel of "stanleyjacob.dev: Triton", Part II, "Worked
// example: fused softmax" (one pass: load the row with -inf in masked lanes,
// max, subtract, exp, sum, divide, store) laid out for the hardware by hand:
//  - a row is served by `tpr` threads (1..32 lanes of a warp, or 1..32 whole
//    warps); several rows share a CTA when tpr is small;
//  - thread t of a row holds units t, t + tpr, t + 2*tpr, ... of it, a unit
//    being one 16-byte access (the group-cyclic layout of the nano-triton post,
//    "The register layout"), so every warp access is contiguous;
//  - reductions are three-level as in the nano-triton post ("Reductions and
//    broadcasting"): registers, then __shfl_xor_sync butterflies, then, for
//    rows wider than a warp, one (m, l) pair per warp through shared memory.
//    Each warp exponentiates against its own max m_w, and the warps' pairs
//    merge with the online normaliser (mohakchugh.is-a.dev post, "How Flash
//    Attention Uses Triton"), so a row costs one CTA barrier and one exp per
//    element; the per-warp factor exp(m_w - m) / l scales the stored values.
#pragma once

#include "rs_common.cuh"
#include "rs_internal.h"

namespace rs {

template <int DT, int VEC, int VPT>
__global__ void __launch_bounds__(rows_block_limit(VPT, VEC))
rows_kernel(const void* in_, void* out_, int64_t M, int N, int64_t ldi, int64_t ldo, int tpr) {
    using T = Traits<DT>;
    using S = typename T::storage;
    const S* in = static_cast<const S*>(in_);
    S* out = static_cast<S*>(out_);
    __shared__ float2 part[2][32];  // per-warp (m, l), double-buffered over row iterations

    const int rows_per_cta = blockDim.x / tpr;
    const int grp = threadIdx.x / tpr;
    const int t = threadIdx.x - grp * tpr;
    const int width = tpr < 32 ? tpr : 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wpr = tpr >> 5;  // warps per row (0 when a row is narrower than a warp)

    int it = 0;
    for (int64_t rb = blockIdx.x; rb * rows_per_cta < M; rb += gridDim.x, ++it) {
        const int64_t row = rb * rows_per_cta + grp;
        const bool active = row < M;

        float v[VPT][VEC];
        if (active) {
            const S* xr = in + row * ldi;
#pragma unroll
            for (int k = 0; k < VPT; ++k) load_unit<DT, VEC>(xr, (t + k * tpr) * VEC, N, v[k]);
        } else {
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] = kNegInf;
        }

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
                v[k][e] = __expf(v[k][e] - ms);
                l += v[k][e];
            }
        l = group_sum(l, width);

        float c;  // y = exp(x - m_w) * c
        if (tpr <= 32) {
            c = 1.0f / l;
        } else {
            float2* p = part[it & 1];
            if (lane == 0) p[warp] = make_float2(m, l);
            __syncthreads();
            const int w0 = (warp / wpr) * wpr;
            float pm = kNegInf, pl = 0.0f;
            if (lane < wpr) {
                const float2 q = p[w0 + lane];
                pm = q.x;
                pl = q.y;
            }
            const float mrow = group_max(pm, 32);
            const float mrs = safe_max(mrow);
            const float srow = group_sum(pl * rescale(pm, mrs), 32);
            c = rescale(m, mrs) / srow;
        }

        if (active) {
            S* yr = out + row * ldo;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) v[k][e] *= c;
                store_unit<DT, VEC>(yr, (t + k * tpr) * VEC, N, v[k]);
            }
        }
    }
}

template <int DT, int VEC, int VPT>
cudaError_t launch_rows_one(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                            int64_t ldi, int64_t ldo, cudaStream_t s) {
    rows_kernel<DT, VEC, VPT><<<(unsigned)p.grid, p.block_threads, 0, s>>>(in, out, M, N, ldi, ldo,
                                                                         p.threads_per_row);
    return cudaGetLastError();
}

template <int DT, int VEC, int... Vs>
struct RowsDispatch;

template <int DT, int VEC>
struct RowsDispatch<DT, VEC> {
    static cudaError_t go(const rs_plan&, const void*, void*, int64_t, int, int64_t, int64_t,
                          cudaStream_t) {
        return cudaErrorInvalidConfiguration;
    }
};

template <int DT, int VEC, int V0, int... Vs>
struct RowsDispatch<DT, VEC, V0, Vs...> {
    static cudaError_t go(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                          int64_t ldi, int64_t ldo, cudaStream_t s) {
        if (p.vec_per_thread == V0) return launch_rows_one<DT, VEC, V0>(p, in, out, M, N, ldi, ldo, s);
        return RowsDispatch<DT, VEC, Vs...>::go(p, in, out, M, N, ldi, ldo, s);
    }
};

}  // namespace rs
