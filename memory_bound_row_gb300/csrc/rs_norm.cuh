// Normalisations of rows wider than the register and ring kernels hold
// (RS_PATH_STREAM for RMSNorm and LayerNorm): one CTA per row, a grid of a
// few CTAs per SM looping over the rows; the CTA streams the row from global
// memory once per moment and once more to write it: RMSNorm reads it twice
// (sum of squares, then normalise), LayerNorm three times (mean, then squared
// deviations, then normalise).  With few rows in progress at a time the
// later reads mostly hit the L2.
#pragma once

#include "rs_common.cuh"
#include "rs_internal.h"
#include "rs_rowmath.cuh"

namespace rs {

// Sum over the CTA; `red` holds one float per warp plus the broadcast slot.
__device__ __forceinline__ float block_sum(float x, float* red) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    x = group_sum(x, 32);
    if (lane == 0) red[warp] = x;
    __syncthreads();
    if (warp == 0) {
        float y = lane < nw ? red[lane] : 0.0f;
        y = group_sum(y, 32);
        if (lane == 0) red[32] = y;
    }
    __syncthreads();
    const float total = red[32];
    __syncthreads();  // red is reused by the next call
    return total;
}

// Calls f(u, v) for the thread's units u = threadIdx.x + i * blockDim.x of a
// row of `units` units, v the unit's values (0 past N), keeping U loads in
// flight.  KEEP reads with the default cache policy (the row is read again),
// else as streaming loads (last read).
template <int DT, int VEC, bool KEEP, int U = 4, typename F>
__device__ __forceinline__ void for_units(const typename Traits<DT>::storage* xr, int N, int units, F&& f) {
    const int step = blockDim.x;
    int u = threadIdx.x;
    for (; u + (U - 1) * step < units; u += U * step) {
        float v[U][VEC];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (KEEP) load_param_unit<DT, VEC>(xr, (u + k * step) * VEC, N, v[k], 0.0f);
            else load_unit<DT, VEC>(xr, (u + k * step) * VEC, N, v[k], 0.0f);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) f(u + k * step, v[k]);
    }
    for (; u < units; u += step) {
        float v[VEC];
        if (KEEP) load_param_unit<DT, VEC>(xr, u * VEC, N, v, 0.0f);
        else load_unit<DT, VEC>(xr, u * VEC, N, v, 0.0f);
        f(u, v);
    }
}

template <int DT, int VEC, typename OP>
__global__ void __launch_bounds__(kNormStreamThreads)
norm_stream_kernel(const void* in_, void* out_, int64_t M, int N, int64_t ldi, int64_t ldo, RowArgs a) {
    using S = typename Traits<DT>::storage;
    const S* in = static_cast<const S*>(in_);
    S* out = static_cast<S*>(out_);
    __shared__ float red[33];
    const int units = (N + VEC - 1) / VEC;
    wait_prior_grid();
    for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
        const S* xr = in + row * ldi;
        S* yr = out + row * ldo;
        float nmr = 0.0f, r;  // y = (x * r + nmr) * w + b, nmr = -mean * r (0 for RMSNorm)
        float acc[VEC];
        auto reset = [&]() {
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[e] = 0.0f;
        };
        auto total = [&]() {
#pragma unroll
            for (int h = VEC / 2; h > 0; h /= 2)
#pragma unroll
                for (int e = 0; e < h; ++e) acc[e] += acc[e + h];
            return acc[0];
        };
        if constexpr (OP::kOp == RS_OP_RMSNORM) {
            reset();
            for_units<DT, VEC, true>(xr, N, units, [&](int, const float* v) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] = fmaf(v[e], v[e], acc[e]);
            });
            r = 1.0f / sqrtf(block_sum(total(), red) / (float)N + a.eps);
        } else {
            reset();
            for_units<DT, VEC, true>(xr, N, units, [&](int, const float* v) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[e] += v[e];
            });
            const float mean = block_sum(total(), red) / (float)N;
            reset();
            for_units<DT, VEC, true>(xr, N, units, [&](int u, const float* v) {
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const float x = v[e] - mean;
                    if (u * VEC + e < N) acc[e] = fmaf(x, x, acc[e]);
                }
            });
            r = 1.0f / sqrtf(block_sum(total(), red) / (float)N + a.eps);
            nmr = -mean * r;
        }
        // The writing pass holds weight and bias units too: fewer in flight
        // for 16-byte units of 16-bit values (no spills at 128 registers).
        for_units<DT, VEC, false, (VEC == 8 ? 2 : 4)>(xr, N, units, [&](int u, const float* v) {
            float w[VEC], b[VEC], y[VEC];
            load_param_unit<DT, VEC>(a.w, u * VEC, N, w, 1.0f);
            load_param_unit<DT, VEC>(a.b, u * VEC, N, b, 0.0f);
#pragma unroll
            for (int e = 0; e < VEC; ++e) y[e] = fmaf(fmaf(v[e], r, nmr), w[e], b[e]);
            store_unit<DT, VEC>(yr, u * VEC, N, y);
        });
    }
    allow_next_grid();  // a grid that loops over rows: the next kernel may begin once this CTA is done
}

template <int DT, int VEC, typename OP>
cudaError_t launch_norm_stream(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                               int64_t ldo, cudaStream_t s, const RowArgs& a) {
    return launch_kernel(norm_stream_kernel<DT, VEC, OP>, (unsigned)p.grid, (unsigned)kNormStreamThreads, 0, s, 0,
                         p.strict_order != 0, in, out, M, N, ldi, ldo, a);
}

}  // namespace rs
