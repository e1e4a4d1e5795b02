// RS_PATH_ROWS: single-pass row operation (softmax, RMSNorm, LayerNorm) with
// the whole row in registers.
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
#include "rs_rowmath.cuh"

namespace rs {

template <int DT, int VEC, int VPT, typename OP>
__global__ void __launch_bounds__(rows_block_limit(VPT, VEC))
rows_kernel(const void* in_, void* out_, int64_t M, int N, int64_t ldi, int64_t ldo, int tpr, RowArgs args) {
    using S = typename Traits<DT>::storage;
    const S* in = static_cast<const S*>(in_);
    S* out = static_cast<S*>(out_);
    __shared__ float2 part[2][32];  // per-warp partials, double-buffered over row iterations

    const int rows_per_cta = blockDim.x / tpr;
    const int grp = threadIdx.x / tpr;
    const int t = threadIdx.x - grp * tpr;
    const bool whole = (t + (VPT - 1) * tpr + 1) * VEC <= N;  // all of this thread's units lie in the row
    wait_prior_grid();
    allow_next_grid();

    int it = 0;
    for (int64_t rb = blockIdx.x; rb * rows_per_cta < M; rb += gridDim.x, ++it) {
        const int64_t row = rb * rows_per_cta + grp;
        const bool active = row < M;
        float v[VPT][VEC];
        // A causal mask keeps a prefix: the rest reads as the fill (-inf) and is never loaded.
        int keep = N;
        if constexpr (OP::kMasked) keep = row_keep(args, active ? row : 0, N);
        load_row_units<DT, VEC, VPT>(in + (active ? row : 0) * ldi, t, tpr, keep, active, v, OP::kFill);
        OP::template apply<DT, VEC, VPT>(v, t, tpr, OP::kMasked ? keep : N, whole,
                                         GlobalParams{args.w, args.b, args.eps, N, 0}, part[it & 1]);
        if (active) store_row_units<DT, VEC, VPT>(out + row * ldo, t, tpr, N, v);
    }
}

template <int DT, int VEC, int VPT, typename OP>
cudaError_t launch_rows_one(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                            int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a) {
    return launch_kernel(rows_kernel<DT, VEC, VPT, OP>, (unsigned)p.grid, (unsigned)p.block_threads, 0, s, 0,
                         p.strict_order != 0, in, out, M, N, ldi, ldo, p.threads_per_row, a);
}

template <int DT, int VEC, typename OP, int... Vs>
struct RowsDispatch;

template <int DT, int VEC, typename OP>
struct RowsDispatch<DT, VEC, OP> {
    static cudaError_t go(const rs_plan&, const void*, void*, int64_t, int, int64_t, int64_t, cudaStream_t,
                          const RowArgs&) {
        return cudaErrorInvalidConfiguration;
    }
};

template <int DT, int VEC, typename OP, int V0, int... Vs>
struct RowsDispatch<DT, VEC, OP, V0, Vs...> {
    static cudaError_t go(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                          int64_t ldo, cudaStream_t s, const RowArgs& a) {
        if (p.vec_per_thread == V0) return launch_rows_one<DT, VEC, V0, OP>(p, in, out, M, N, ldi, ldo, s, a);
        return RowsDispatch<DT, VEC, OP, Vs...>::go(p, in, out, M, N, ldi, ldo, s, a);
    }
};

}  // namespace rs
