// RS_PATH_RING for the causal softmax with per-thread asynchronous copies
// (RS_RING_THREAD_COPIES).
//
// The ring of rs_ring.cuh stages whole rows with one bulk copy (TMA engine)
// per row; under a causal mask that reads the masked part too, and copying
// only each row's kept prefix by bulk copies measured far slower.  Here every
// thread copies, with 16-byte cp.async (global -> shared, no register held
// while the bytes are in flight), exactly the units of its own row that hold
// kept elements -- the units it will later read -- into a shared-memory
// stage.  Each thread waits only for its own copies (cp.async.wait_group), so
// no mbarrier and no barrier guard the stages: a thread never reads what
// another thread copied, and it refills a stage only after the values it read
// from it have been used (so its reads are complete).
// The arithmetic and the layout are those of the ring (one group of tpr
// threads a row, units t, t + tpr, ... of the row, the row's causal operation
// on registers); a persistent grid of CTAs loops over row groups with STAGES
// groups of copies in flight a thread.
//
// Measured on the causal scores [16, 32, 2048, 2048] (bf16): 1.222 ms against
// 1.320 ms for the bulk-copy ring in the same call.  Slower and not kept:
// three stages (1.295 ms); three buffers with two groups in flight and the
// refill issued as soon as a stage is loaded (1.238 ms); four (1.897 ms, one
// CTA an SM); re-reading the stage in three passes with two exponentials a
// kept element and 70 registers (1.513 ms); branches per slot that skip the
// masked slots' loads and arithmetic (1.377 and 1.419 ms).
// The rows of one warp are bound by instruction issue, not memory; three
// changes that each issue fewer instructions a row, kept (in one call, every
// step bitwise equal to the plain softmax of the same scores): the exponent's
// subtraction and scaling and the final scaling in fp32 pairs (1215 -> 1132
// us); the fill of the masked units selected on the 16-byte words before the
// unpack (-> 1067 us); the scaling fused into the stores, the masked slots
// selected to zero words after the rounding (-> 1033 us).
#pragma once

#include <mutex>

#include "rs_async.cuh"
#include "rs_common.cuh"
#include "rs_internal.h"
#include "rs_rowmath.cuh"

namespace rs {

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int PENDING>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
}

template <int DT, int VPT, int STAGES, typename OP>
__global__ void __launch_bounds__(rows_block_limit(VPT, Traits<DT>::kVec), 1)
ring_cp_kernel(const void* in_, void* out_, int64_t M, int N, int64_t ldi, int64_t ldo, int tpr, RowArgs args) {
    static_assert(OP::kOp == RS_OP_SOFTMAX && OP::kMasked, "the causal softmax only");
    using T = Traits<DT>;
    using S = typename T::storage;
    constexpr int VEC = T::kVec;
    const S* in = static_cast<const S*>(in_);
    S* out = static_cast<S*>(out_);

    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ float2 part[2][32];

    const int rpg = blockDim.x / tpr;  // rows per group (one group per stage)
    const int grp = threadIdx.x / tpr;
    const int t = threadIdx.x - grp * tpr;
    const int units_full = N / VEC;  // whole 16-byte units a row
    const size_t slot = (size_t)units_full * 16;
    const size_t stage_bytes = slot * rpg;
    const int64_t groups = (M + rpg - 1) / rpg;

    // This thread's kept whole units of its row of group g into stage s, as one
    // commit group (empty past the last group, so that every iteration commits).
    auto issue = [&](int s, int64_t g) {
        const int64_t row = g * rpg + grp;
        if (g < groups && row < M) {
            const int cu = (row_keep(args, row, N) + VEC - 1) / VEC;
            const int copy_units = cu < units_full ? cu : units_full;
            unsigned char* dst = ring + (size_t)s * stage_bytes + (size_t)grp * slot;
            const S* src = in + row * ldi;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int u = t + k * tpr;
                if (u < copy_units) cp_async16(dst + (size_t)u * 16, src + (size_t)u * VEC);
            }
        }
        cp_async_commit();
    };

    wait_prior_grid();
#pragma unroll
    for (int j = 0; j < STAGES; ++j) issue(j, blockIdx.x + (int64_t)j * gridDim.x);

    int s = 0;
    int64_t it = 0;
    for (int64_t g = blockIdx.x; g < groups; g += gridDim.x, ++it) {
        cp_async_wait<STAGES - 1>();  // this thread's copies of the oldest group have landed
        const int64_t row = g * rpg + grp;
        const bool active = row < M;
        const unsigned char* srow = ring + (size_t)s * stage_bytes + (size_t)grp * slot;
        const S* grow = in + (active ? row : 0) * ldi;

        // Fully kept units from the stage, the rest the fill (-inf); then the
        // one unit that holds the end of the kept prefix (staged, or the row's
        // ragged tail read from global memory), if this thread has it.
        // (The fill is selected on the 16-byte words, -inf pairs, before the
        // unpack: one select a word rather than one move a value.)
        float v[VPT][VEC];
        const int keep = row_keep(args, active ? row : 0, N);
        const int whole_units = keep / VEC;
        constexpr uint32_t kNegPair = DT == RS_BF16 ? 0xFF80FF80u : 0xFC00FC00u;
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            const int u = t + k * tpr;
            uint4 wv = make_uint4(kNegPair, kNegPair, kNegPair, kNegPair);
            if (active && u < whole_units) wv = *reinterpret_cast<const uint4*>(srow + (size_t)u * 16);
            T::unpack(wv, v[k]);
        }
        const int us = whole_units;
        if (active && keep % VEC && t <= us && us <= t + (VPT - 1) * tpr) {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                if (t + k * tpr != us) continue;
                if (us < units_full) {
                    T::unpack(*reinterpret_cast<const uint4*>(srow + (size_t)us * 16), v[k]);
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        if (us * VEC + e >= keep) v[k][e] = OP::kFill;
                } else {
                    load_unit<DT, VEC>(grow, us * VEC, keep, v[k], OP::kFill);
                }
            }
        }
        const float c = OP::template reduce<DT, VEC, VPT>(v, tpr, keep, part[it & 1]);
        // The row's values have been used (the stage's reads are complete):
        // refill the stage with the group STAGES iterations ahead, then store.
        issue(s, g + (int64_t)STAGES * gridDim.x);
        if (active) {
            S* yr = out + row * ldo;
            if (isfinite(c) && (t + (VPT - 1) * tpr + 1) * VEC <= N) {
                // Scale, round, and store each unit; the slots past the prefix
                // are selected to zero words after the rounding.
                const int kk = (keep + tpr * VEC - 1) / (tpr * VEC);
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    unit_mul<VEC>(v[k], c);
                    uint4 w = T::pack(v[k]);
                    if (k >= kk) w = make_uint4(0u, 0u, 0u, 0u);
                    __stcs(reinterpret_cast<uint4*>(yr + (size_t)(t + k * tpr) * VEC), w);
                }
            } else {
                OP::template finish<DT, VEC, VPT>(v, t, tpr, keep, c);
                store_row_units<DT, VEC, VPT>(yr, t, tpr, N, v);
            }
        }
        if (++s == STAGES) s = 0;
    }
    cp_async_wait<0>();  // no copy outlives the CTA
    allow_next_grid();
}

template <int DT, int VPT, int STAGES, typename OP>
cudaError_t launch_ring_cp_one(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                               int64_t ldo, cudaStream_t s, const RowArgs& a) {
    auto kern = ring_cp_kernel<DT, VPT, STAGES, OP>;
    static std::mutex mu;
    static bool ready[64] = {};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!ready[dev]) {
            int optin = 0;
            err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
            if (err != cudaSuccess) return err;
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       optin - (int)kRingStaticSmem);
            if (err != cudaSuccess) return err;
            ready[dev] = true;
        }
    }
    return launch_kernel(kern, (unsigned)p.grid, (unsigned)p.block_threads, p.smem_bytes, s, 0, p.strict_order != 0,
                         in, out, M, N, ldi, ldo, p.threads_per_row, a);
}

template <int DT, typename OP, int... Vs>
struct RingCpDispatch;

template <int DT, typename OP>
struct RingCpDispatch<DT, OP> {
    static cudaError_t go(const rs_plan&, const void*, void*, int64_t, int, int64_t, int64_t, cudaStream_t,
                          const RowArgs&) {
        return cudaErrorInvalidConfiguration;
    }
};

template <int DT, typename OP, int V0, int... Vs>
struct RingCpDispatch<DT, OP, V0, Vs...> {
    static cudaError_t go(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi, int64_t ldo,
                          cudaStream_t s, const RowArgs& a) {
        if (p.vec_per_thread == V0) {
            if (p.stages == 2) return launch_ring_cp_one<DT, V0, 2, OP>(p, in, out, M, N, ldi, ldo, s, a);
            if (p.stages == 3) return launch_ring_cp_one<DT, V0, 3, OP>(p, in, out, M, N, ldi, ldo, s, a);
            return cudaErrorInvalidConfiguration;
        }
        return RingCpDispatch<DT, OP, Vs...>::go(p, in, out, M, N, ldi, ldo, s, a);
    }
};

}  // namespace rs
