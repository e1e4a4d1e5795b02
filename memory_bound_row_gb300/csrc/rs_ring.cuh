// RS_PATH_RING: persistent single-pass row operation (softmax, RMSNorm,
// LayerNorm) whose input rows are staged through a ring of shared-memory
// stages by bulk asynchronous copies.
//
// The arithmetic is that of RS_PATH_ROWS (rs_rows.cuh): one group of `tpr`
// threads per row, the row in registers as 16-byte group-cyclic units, a
// warp-local max, one exp per element, per-warp (m, l) pairs merged with the
// online normaliser.  What changes is where the bytes in flight live.  A
// register-resident row costs registers for every byte being fetched, which
// caps the bytes in flight per SM well below what HBM needs to stay busy.
// Here each CTA keeps `stages` groups of rows in flight in shared memory:
// one thread issues a cp.async.bulk (TMA engine) copy per row into the next
// free stage, with completion counted on that stage's mbarrier, while all
// threads compute on the oldest stage.  Each CTA loops over row groups
// blockIdx.x, blockIdx.x + gridDim.x, ... (a persistent grid sized to the
// resident CTAs), so copies for later groups overlap the compute and the
// stores of the current one.  The multi-stage ring with deferred consumption
// is the scheme the nano-triton post describes for its matmul ("Version 2: a
// cp.async pipeline"), applied to rows and carried by the bulk-copy engine.
//
// The last partial 16-byte unit of a row (N not a multiple of 16 bytes) is
// read straight from global memory.  Waits are bounded (rs_async.cuh); a thread
// whose wait runs out flags the device status word and writes nothing more;
// the CTA lets its copies in flight land (bounded again) and stops.
#pragma once

#include <mutex>
#include <type_traits>

#include "rs_async.cuh"
#include "rs_common.cuh"
#include "rs_internal.h"
#include "rs_rowmath.cuh"

namespace rs {

// HOLD = true keeps the thread's units in registers as fp32 (one exp per
// element).  HOLD = false keeps only the staged copy in shared memory and
// reads it once per pass (max, sum of exps, normalise-and-store), taking the
// exp twice per element: fewer registers, so more CTAs and warps per SM.
template <int DT, int VPT, bool HOLD>
__device__ __forceinline__ void ring_unit(const unsigned char* srow, const typename Traits<DT>::storage* grow,
                                          int u, int units_full, int N, bool active, float* f,
                                          float fill = kNegInf) {
    constexpr int VEC = Traits<DT>::kVec;
    if (active && u < units_full) {
        Traits<DT>::unpack(*reinterpret_cast<const uint4*>(srow + (size_t)u * 16), f);
    } else if (active && u * VEC < N) {
        load_unit<DT, VEC>(grow, u * VEC, N, f, fill);
    } else {
#pragma unroll
        for (int e = 0; e < VEC; ++e) f[e] = fill;
    }
}

template <int DT, int VPT, bool HOLD, typename OP>
__global__ void __launch_bounds__(HOLD ? (OP::kHeldParams ? kHeldThreads : rows_block_limit(VPT, Traits<DT>::kVec))
                                       : kRingRereadThreads,
                                  HOLD ? (OP::kHeldParams ? 65536 / (kHeldThreads * kHeldRegs) : 1)
                                       : kRingRereadMinCtas)
ring_kernel(const void* in_, void* out_, int64_t M, int N, int64_t ldi, int64_t ldo, int tpr, int stages,
            uint64_t wait_ns, int withhold, RowArgs args) {
    static_assert(HOLD || (OP::kOp == RS_OP_SOFTMAX && !OP::kMasked), "the re-read variant is the softmax's only");
    using T = Traits<DT>;
    using S = typename T::storage;
    constexpr int VEC = T::kVec;
    const S* in = static_cast<const S*>(in_);
    S* out = static_cast<S*>(out_);

    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kRingMaxStages];
    __shared__ float2 part[2][32];

    const int rpg = blockDim.x / tpr;  // rows per group (one group per stage)
    const int grp = threadIdx.x / tpr;
    const int t = threadIdx.x - grp * tpr;
    const int width = tpr < 32 ? tpr : 32;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int wpr = tpr >> 5;

    const int units_full = N / VEC;                  // whole 16-byte units per row (bulk-copied)
    const uint32_t slot = (uint32_t)units_full * 16u;  // bytes of one row in a stage
    const size_t stage_bytes = (size_t)slot * rpg;
    const int64_t groups = (M + rpg - 1) / rpg;

    // Thread 0: fill stage s with row group g.
    auto issue = [&](int s, int64_t g) {
        const int64_t r0 = g * rpg;
        const int nrows = (int)(M - r0 < rpg ? M - r0 : rpg);
        if (slot == 0) {
            mbar_arrive(&full[s]);
            return;
        }
        mbar_arrive_expect_tx(&full[s], slot * (uint32_t)nrows);
        if (withhold) return;  // failure-path test: the awaited bytes never come
        unsigned char* dst = ring + (size_t)s * stage_bytes;
        for (int k = 0; k < nrows; ++k) bulk_load(dst + (size_t)k * slot, in + (r0 + k) * ldi, slot, &full[s]);
    };

    // Causal mask: the ring still stages whole rows and the masked part of a
    // row is never used.  Copying only each row's kept prefix moved fewer
    // bytes but measured slower on the causal attention workload [16, 32,
    // 2048, 2048]: 2.25 against 1.32 ms with the masked arithmetic skipped
    // (1.46 against 1.29 ms before), and 2.29-2.31 ms with the prefix copies
    // rounded up to 128 B, 512 B or 2 KB -- not the copy granularity: the
    // partial-row copies, all starting at the row heads, keep HBM far less
    // busy than whole rows.

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    wait_prior_grid();
    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            const int64_t g = blockIdx.x + (int64_t)s * gridDim.x;
            if (g < groups) issue(s, g);
        }
    }
    // Where the normalisations read their vectors.  Held instances
    // (OP::kHeldParams): each thread keeps the weight and bias of its units as
    // fp32 in registers for the whole loop (it serves the same columns of every
    // row).  Otherwise LayerNorm stages both vectors once per CTA in shared
    // memory after the ring stages (every row of the CTA reads them; measured
    // 33 % faster on 2048-value bf16 rows than the read-only cache), and
    // RMSNorm reads its one vector through the read-only cache (staging it cost
    // more in resident CTAs than it saved).
    constexpr bool kHeld = OP::kHeldParams;
    constexpr bool kStage = OP::kOp == RS_OP_LAYERNORM && !kHeld;
    using Params = typename std::conditional<
        kHeld, HeldParams<VPT, VEC>,
        typename std::conditional<kStage, SharedParams<DT>, GlobalParams>::type>::type;
    Params prm;
    if constexpr (kHeld) {
        const GlobalParams g{args.w, args.b, args.eps, N, 0};
#pragma unroll
        for (int k = 0; k < VPT; ++k) {
            g.template w_unit<DT, VEC>((t + k * tpr) * VEC, prm.w[k]);
            if constexpr (OP::kOp == RS_OP_LAYERNORM) g.template b_unit<DT, VEC>((t + k * tpr) * VEC, prm.b[k]);
        }
        prm.eps = args.eps;
    } else if constexpr (kStage) {
        const int npad = ((N + VEC - 1) / VEC) * VEC;
        S* sw = nullptr;
        S* sb = nullptr;
        unsigned char* pbase = ring + (size_t)stages * stage_bytes;
        if (args.w) {
            sw = reinterpret_cast<S*>(pbase);
            stage_param<DT>(sw, args.w, 0, N, npad, 1.0f);
            pbase += (size_t)npad * sizeof(S);
        }
        if (args.b) {
            sb = reinterpret_cast<S*>(pbase);
            stage_param<DT>(sb, args.b, 0, N, npad, 0.0f);
        }
        __syncthreads();
        prm = Params{sw, sb, args.eps, npad};
    } else {
        prm = Params{args.w, args.b, args.eps, N, 0};
    }

    bool abort = false;
    int s = 0;
    uint32_t parity = 0;
    int64_t it = 0;
    for (int64_t g = blockIdx.x; g < groups; g += gridDim.x, ++it) {
        if (!abort && !mbar_wait_bounded(&full[s], parity, wait_ns)) {
            abort = true;
            flag_timeout();
        }
        const int64_t row = g * rpg + grp;
        const bool active = row < M;
        const unsigned char* srow = ring + (size_t)s * stage_bytes + (size_t)grp * slot;
        const S* grow = in + (active ? row : 0) * ldi;

        if constexpr (HOLD && OP::kMasked) {
            // Fully kept units from the stage, the rest the fill (-inf); then
            // the one unit that holds the end of the kept prefix (staged, or
            // the row's ragged tail), if this thread has it.
            float v[VPT][VEC];
            const int keep = row_keep(args, active ? row : 0, N);
            const int whole_units = keep / VEC;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int u = t + k * tpr;
                if (active && u < whole_units) {
                    T::unpack(*reinterpret_cast<const uint4*>(srow + (size_t)u * 16), v[k]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[k][e] = OP::kFill;
                }
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
            OP::template apply<DT, VEC, VPT>(v, t, tpr, keep, false, prm, part[it & 1]);
            if (active && !abort) store_row_units<DT, VEC, VPT>(out + row * ldo, t, tpr, N, v);
        } else if constexpr (HOLD) {
            float v[VPT][VEC];
            if (active && (t + (VPT - 1) * tpr) < units_full) {
#pragma unroll
                for (int k = 0; k < VPT; ++k)
                    T::unpack(*reinterpret_cast<const uint4*>(srow + (size_t)(t + k * tpr) * 16), v[k]);
            } else {
#pragma unroll
                for (int k = 0; k < VPT; ++k)
                    ring_unit<DT, VPT, HOLD>(srow, grow, t + k * tpr, units_full, N, active, v[k], OP::kFill);
            }
            const bool whole = (t + (VPT - 1) * tpr + 1) * VEC <= N;
            OP::template apply<DT, VEC, VPT>(v, t, tpr, N, whole, prm, part[it & 1]);
            if (active && !abort) store_row_units<DT, VEC, VPT>(out + row * ldo, t, tpr, N, v);
        } else {
            float f[VEC];
            float m = kNegInf;
#pragma unroll 1
            for (int k = 0; k < VPT; ++k) {
                ring_unit<DT, VPT, HOLD>(srow, grow, t + k * tpr, units_full, N, active, f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) m = fmaxf(m, f[e]);
            }
            m = group_max(m, width);
            const float ms = safe_max(m);

            float l = 0.0f;
            asm volatile("" ::: "memory");  // re-read the stage, do not keep it in registers
#pragma unroll 1
            for (int k = 0; k < VPT; ++k) {
                ring_unit<DT, VPT, HOLD>(srow, grow, t + k * tpr, units_full, N, active, f);
#pragma unroll
                for (int e = 0; e < VEC; ++e) l += exp_diff(f[e], ms);
            }
            l = group_sum(l, width);

            float c;
            if (tpr <= 32) {
                c = 1.0f / l;
            } else {
                float2* p = part[it & 1];
                if (lane == 0) p[warp] = make_float2(m, l);
                __syncthreads();
                const int w0 = (warp / wpr) * wpr;
                const int ww = pow2_ceil(wpr);
                float pm = kNegInf, pl = 0.0f;
                if (lane < wpr) {
                    const float2 q = p[w0 + lane];
                    pm = q.x;
                    pl = q.y;
                }
                const float mrow = __shfl_sync(0xffffffffu, group_max(pm, ww), 0);
                const float mrs = safe_max(mrow);
                const float srow_sum = __shfl_sync(0xffffffffu, group_sum(pl * rescale(pm, mrs), ww), 0);
                c = rescale(m, mrs) / srow_sum;
            }

            if (active && !abort) {
                S* yr = out + row * ldo;
                asm volatile("" ::: "memory");
#pragma unroll 1
                for (int k = 0; k < VPT; ++k) {
                    ring_unit<DT, VPT, HOLD>(srow, grow, t + k * tpr, units_full, N, active, f);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) f[e] = exp_diff(f[e], ms) * c;
                    store_unit<DT, VEC>(yr, (t + k * tpr) * VEC, N, f);
                }
            }
        }

        // Every thread is done with stage s; refill it with the group
        // `stages` iterations ahead.
        if (__syncthreads_or(abort)) {
            abort = true;
            break;
        }
        if (threadIdx.x == 0) {
            const int64_t gn = g + (int64_t)stages * gridDim.x;
            if (gn < groups) {
                fence_proxy_async_smem();
                issue(s, gn);
            }
        }
        if (++s == stages) {
            s = 0;
            parity ^= 1u;
        }
    }

    // Persistent grid: the next kernel of the stream may begin its launch once
    // this CTA has no more rows (earlier, its waiting CTAs would share the SMs
    // with this grid's work).
    allow_next_grid();
    if (abort && threadIdx.x == 0) {
        // Let the copies of iterations it .. it + stages - 1 land before the
        // shared memory is released (iteration j used stage j % stages with
        // parity (j / stages) & 1).
        for (int64_t j = it; j < it + stages; ++j) {
            const int64_t gj = blockIdx.x + j * gridDim.x;
            if (gj >= groups) break;
            (void)mbar_wait_bounded(&full[j % stages], (uint32_t)((j / stages) & 1), wait_ns);
        }
    }
}

template <int DT, int VPT, bool HOLD, typename OP>
cudaError_t launch_ring_one(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                            int64_t ldo, cudaStream_t s, const RowArgs& a) {
    auto kern = ring_kernel<DT, VPT, HOLD, OP>;
    // The dynamic shared-memory ceiling is a per-device attribute: raise it to
    // the device maximum once per device for this instance.
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
    const uint64_t wait_ns = p.wait_limit_us > 0 ? (uint64_t)p.wait_limit_us * 1000ull : kWaitLimitNs;
    return launch_kernel(kern, (unsigned)p.grid, (unsigned)p.block_threads, p.smem_bytes, s, 0, p.strict_order != 0,
                         in, out, M, N, ldi, ldo, p.threads_per_row, p.stages, wait_ns, p.withhold_copies, a);
}

template <int DT, typename OP, int... Vs>
struct RingDispatch;

template <int DT, typename OP>
struct RingDispatch<DT, OP> {
    static cudaError_t go(const rs_plan&, const void*, void*, int64_t, int, int64_t, int64_t, cudaStream_t,
                          const RowArgs&) {
        return cudaErrorInvalidConfiguration;
    }
};

template <int DT, typename OP, int V0, int... Vs>
struct RingDispatch<DT, OP, V0, Vs...> {
    static cudaError_t go(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                          int64_t ldo, cudaStream_t s, const RowArgs& a) {
        if (p.vec_per_thread == V0) {
            if constexpr (OP::kOp == RS_OP_SOFTMAX && !OP::kMasked) {
                if (p.ring_values == RS_RING_REREAD)
                    return launch_ring_one<DT, V0, false, OP>(p, in, out, M, N, ldi, ldo, s, a);
            }
            if constexpr (OP::kMasked) {
                if (p.ring_values == RS_RING_REREAD) return cudaErrorInvalidConfiguration;
            }
            return launch_ring_one<DT, V0, true, OP>(p, in, out, M, N, ldi, ldo, s, a);
        }
        return RingDispatch<DT, OP, Vs...>::go(p, in, out, M, N, ldi, ldo, s, a);
    }
};

}  // namespace rs
