// RS_PATH_CLUSTER with the slice held in registers (RS_RING_REGISTERS), for
// every row operation of the engine (softmax, RMSNorm, LayerNorm).
//
// Persistent clusters; CTA `rank` of a cluster serves slice
// [rank * chunk, rank * chunk + len) of rows cluster_id, cluster_id +
// n_clusters, ...  Each CTA has `nslots` shared-memory slots filled by bulk
// copies.  A slot is only a landing buffer: the CTA copies its slice from the
// slot into registers (VPT 16-byte units per thread, fp32), releases the slot
// at once -- thread 0 immediately issues the copy of a later row into it --
// and then reduces and writes from registers, so the next rows' bytes stream
// in while this row is reduced and stored.  Each input byte crosses HBM once
// and each output byte once.
//
// Merges go warps -> CTA through shared memory and CTAs -> cluster through
// distributed shared memory: every CTA pushes one pair of floats into a slot
// of every CTA of its cluster (st.async, counted on the receivers' mbarrier)
// and combines the cluster's pairs itself.  The pair of a slice is
//   softmax    (m, l): its max and its sum of exp(x - m); pairs merge with
//              the online normaliser of the mohakchugh.is-a.dev post ("How
//              Flash Attention Uses Triton"): m = max m_c,
//              l = sum l_c exp(m_c - m).  Each warp takes its exponentials
//              as 2^fma(x, log2 e, -o) against its offset o = rn(m_w log2 e)
//              while |m_w| < 2^23, and folds the offset's rounding residual r
//              into its sum (times 2^-r) and into its final scale (rescale_res);
//              past that magnitude it takes exp_diff;
//   RMSNorm    (sum of x^2, 0): sums add;
//   LayerNorm  (S_c, Q_c): the slice's sum and its sum of squared deviations
//              from the slice's own mean mu_c = S_c / n_c; slices combine with
//              the textbook parallel-variance identity (Chan, Golub and
//              LeVeque): mu = sum S_c / N,
//              sum (x - mu)^2 = sum_c [Q_c + n_c (mu_c - mu)^2],
//              so the variance is exact algebra of slice moments and no global
//              E[x^2] - mu^2 cancellation occurs.  A slice's own (S_c, Q_c)
//              come the same way from its threads' moments about their own
//              means, merged over warps and then over the CTA's warps (one
//              CTA barrier a row).
//
// Waits are bounded by %globaltimer.  A copy wait that runs out sets bit 0 of
// the device status word; the CTA stops issuing copies and storing rows but
// keeps taking part in the exchange (it still pushes a pair per row and waits
// for its peers' pairs, under a limit three times the copy wait's, since a
// peer may itself be waiting out a copy), so its peers' rows complete; at the
// end it waits, bounded again, for its copies in flight.  A receive barrier is
// re-armed only after the phase it armed has completed; if a receive wait
// itself runs out (a peer stalled for longer than its own copy waits allow,
// which bounded waits exclude), the CTA stops waiting on and re-arming its
// receive barriers.  Rows of a call that reported a timeout are undefined.
#pragma once

#include <cooperative_groups.h>

#include <mutex>

#include "rs_async.cuh"
#include "rs_common.cuh"
#include "rs_internal.h"
#include "rs_rowmath.cuh"

namespace rs {

namespace hold_cg = cooperative_groups;

// Length of the slice of CTA `rank` (0 past the row).
__device__ __forceinline__ int hold_slice_len(int rank, int chunk, int N) {
    const int64_t c0 = (int64_t)rank * chunk;
    if (c0 >= N) return 0;
    return (int)(c0 + chunk < N ? chunk : N - c0);
}

template <int DT, int VPT, typename OP>
__global__ void __launch_bounds__(VPT <= 4 ? kWideHoldThreads : kWideHoldThreads / 2, 2)
wide_hold_kernel(const void* in_, void* out_, int64_t M, int N, int64_t ldi, int64_t ldo, int chunk, int nslots,
                 uint64_t wait_ns, int withhold, RowArgs args) {
    using T = Traits<DT>;
    using S = typename T::storage;
    constexpr int VEC = T::kVec;
    constexpr bool kSoftmax = OP::kOp == RS_OP_SOFTMAX;
    const S* in = static_cast<const S*>(in_);
    S* out = static_cast<S*>(out_);
    hold_cg::cluster_group cluster = hold_cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();

    extern __shared__ __align__(128) unsigned char slots[];
    __shared__ __align__(8) uint64_t bars[kWideHoldMaxSlots];  // slot filled
    __shared__ __align__(8) uint64_t recv_bar[2];  // all CTAs' pairs of a row received
    __shared__ __align__(8) float2 recv[2][kMaxCluster];
    __shared__ float2 warp_part[2][kWideHoldThreads / 32];
    __shared__ int exchange_broken;  // a receive wait ran out: stop waiting on and re-arming recv_bar

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int tpr = blockDim.x;

    const int64_t c0l = (int64_t)rank * chunk < N ? (int64_t)rank * chunk : (int64_t)N;
    const int c0 = (int)c0l;
    const int len = (int)((c0l + chunk < N ? c0l + chunk : (int64_t)N) - c0l);
    const int full = len / VEC;                        // whole units, bulk-copied
    const uint32_t slice_bytes = (uint32_t)full * 16u;
    const size_t slot_stride = ((size_t)chunk * sizeof(S) + 15) & ~(size_t)15;
    const uint32_t pair_bytes = (uint32_t)cs * (uint32_t)sizeof(float2);
    const bool whole = (tid + (VPT - 1) * tpr + 1) * VEC <= len;  // all of this thread's units in the slice

    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;

    // Causal mask: the elements of this CTA's slice that row `row` keeps (the
    // part of the kept prefix that falls in the slice); only the whole units
    // that hold them are copied.
    auto slice_keep = [&](int64_t row) {
        const int keep = row_keep(args, row, N) - c0;
        return keep < 0 ? 0 : (keep > len ? len : keep);
    };
    auto issue = [&](int64_t row, int slot) {
        uint32_t bytes = slice_bytes;
        if constexpr (OP::kMasked) {
            const int cu = (slice_keep(row) + VEC - 1) / VEC;
            bytes = (uint32_t)(cu < full ? cu : full) * 16u;
        }
        if (bytes == 0) {
            mbar_arrive(&bars[slot]);
            return;
        }
        mbar_arrive_expect_tx(&bars[slot], bytes);
        if (withhold) return;  // failure-path test: the awaited bytes never come
        bulk_load(slots + (size_t)slot * slot_stride, in + row * ldi + c0, bytes, &bars[slot]);
    };

    if (tid == 0) {
        for (int j = 0; j < nslots; ++j) mbar_init(&bars[j], 1);
        mbar_init(&recv_bar[0], 1);
        mbar_init(&recv_bar[1], 1);
        mbar_arrive_expect_tx(&recv_bar[0], pair_bytes);  // armed for rows 0 and 1 of this cluster
        mbar_arrive_expect_tx(&recv_bar[1], pair_bytes);
        fence_mbar_init();
        exchange_broken = 0;
    }
    __syncthreads();
    wait_prior_grid();
    if (tid == 0) {
        for (int j = 0; j < nslots; ++j)
            if (cluster_id + j * n_clusters < M) issue(cluster_id + j * n_clusters, j);
    }
    // Normalisations read their weight and bias units through the read-only
    // cache (staging the slice in shared memory measured no faster and cost
    // resident CTAs).
    const GlobalParams prm{args.w, args.b, args.eps, N, c0};
    cluster.sync();  // every CTA's receive barriers are armed before any pair is sent

    bool abort = false;
    int64_t abort_it = -1;
    int64_t it = 0;
    for (int64_t row = cluster_id; row < M; row += n_clusters, ++it) {
        const int slot = (int)(it % nslots);
        const uint32_t parity = (uint32_t)((it / nslots) & 1);
        if (!abort && !mbar_wait_bounded(&bars[slot], parity, wait_ns)) {
            abort = true;
            flag_timeout();
        }
        const unsigned char* buf = slots + (size_t)slot * slot_stride;
        const S* xr = in + row * ldi + c0;

        float v[VPT][VEC];
        if constexpr (OP::kMasked) {
            // Fully kept units from the slot, the rest the fill; then the one
            // partly kept unit (in the slot, or the slice's ragged tail), if
            // this thread holds it.
            const int lv = slice_keep(row);
            const int whole_units = lv / VEC;
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int u = tid + k * tpr;
                if (u < whole_units) {
                    T::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)u * 16), v[k]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[k][e] = OP::kFill;
                }
            }
            const int us = whole_units;
            if (lv % VEC && tid <= us && us <= tid + (VPT - 1) * tpr) {
#pragma unroll
                for (int k = 0; k < VPT; ++k) {
                    if (tid + k * tpr != us) continue;
                    if (us < full) {
                        T::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)us * 16), v[k]);
#pragma unroll
                        for (int e = 0; e < VEC; ++e)
                            if (us * VEC + e >= lv) v[k][e] = OP::kFill;
                    } else {
                        load_unit<DT, VEC>(xr, us * VEC, lv, v[k], OP::kFill);
                    }
                }
            }
        } else if ((tid + (VPT - 1) * tpr) < full) {
#pragma unroll
            for (int k = 0; k < VPT; ++k)
                T::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)(tid + k * tpr) * 16), v[k]);
        } else {
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int u = tid + k * tpr;
                if (u < full) {
                    T::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)u * 16), v[k]);
                } else {
                    load_unit<DT, VEC>(xr, u * VEC, len, v[k], OP::kFill);  // ragged tail, or fill past the slice
                }
            }
        }

        // This thread's contribution, reduced over the warp.
        float m = kNegInf;  // softmax: the warp's max
        float a0 = 0.0f;    // softmax: l; norms: sum of x^2 or sum of x
        float res = 0.0f;   // softmax: the residual of the warp's offset
        if constexpr (kSoftmax) {
#pragma unroll
            for (int k = 0; k < VPT; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
            m = group_max(m, 32);
            if (offset_form(m)) {
                const float o = offset_of(m);
                res = residual_of(m, o);
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        v[k][e] = exp_off(v[k][e], o);
                        a0 += v[k][e];
                    }
            } else {
                const float ms = safe_max(m);
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        v[k][e] = exp_diff(v[k][e], ms);
                        a0 += v[k][e];
                    }
            }
        } else if constexpr (OP::kOp == RS_OP_RMSNORM) {
            a0 = thread_sum<VPT, VEC>(v, [](float acc, float x, int, int) { return fmaf(x, x, acc); });
        } else {
            // LayerNorm: this thread's sum and squared deviations about its own
            // mean, merged over the warp (m carries the deviations).
            a0 = thread_sum<VPT, VEC>(v, [](float acc, float x, int, int) { return acc + x; });
            float c, q;
            if (whole) {
                c = (float)(VPT * VEC);
                q = whole_deviations<VPT, VEC>(v, a0);
            } else {  // absent elements hold 0: leave them out
                const int U = len / VEC;
                const int r = U & (tpr - 1);
                c = (float)(VEC * ((U >> __popc(tpr - 1)) + (tid < r ? 1 : 0)) + (tid == r ? len - U * VEC : 0));
                const float mt = c > 0.0f ? __fdividef(a0, c) : 0.0f;
                q = thread_sum<VPT, VEC>(v, [mt, tid, tpr, len](float acc, float x, int k, int e) {
                    const float d = x - mt;
                    return (tid + k * tpr) * VEC + e < len ? fmaf(d, d, acc) : acc;
                });
            }
            group_moments<VPT, VEC>(a0, q, c, 32);
            m = q;
        }
        if constexpr (OP::kOp != RS_OP_LAYERNORM) a0 = group_sum(a0, 32);
        if constexpr (kSoftmax) a0 *= ex2_approx(-res);  // the warp's plain sum of exp(x - m)

        // CTA merge of the warps' partials.  The barrier also ends every read
        // of the slot, which is then handed to the copy of a later row.
        if (lane == 0) warp_part[it & 1][warp] = make_float2(m, a0);
        abort = __syncthreads_or(abort) != 0;
        if (abort && abort_it < 0) abort_it = it;
        if (tid == 0 && !abort && row + nslots * n_clusters < M) {
            fence_proxy_async_smem();
            issue(row + nslots * n_clusters, slot);
        }
        float pm = kNegInf, pl = 0.0f;
        if (lane < nwarps) {
            const float2 q = warp_part[it & 1][lane];
            pm = q.x;
            pl = q.y;
        }
        if constexpr (kSoftmax) {
            group_merge(pm, pl, pow2_ceil(nwarps));  // lanes 0..nwarps-1 hold the CTA's pair
            pm = __shfl_sync(0xffffffffu, pm, 0);
            pl = __shfl_sync(0xffffffffu, pl, 0);
        } else if constexpr (OP::kOp == RS_OP_RMSNORM) {
            pm = __shfl_sync(0xffffffffu, group_sum(pl, pow2_ceil(nwarps)), 0);  // the slice's sum of squares
            pl = 0.0f;
        } else {
            // The warps' moments (lanes 0..nwarps-1: deviations, sum) merged into
            // the slice's sum and squared deviations from its own mean: equal
            // counts when the slice fills the CTA, else each warp's count.
            float sj = pl, qj = lane < nwarps ? pm : 0.0f;
            if (len == tpr * VPT * VEC) {
                equal_moments(sj, qj, 0.5f / (float)(32 * VPT * VEC), nwarps);
            } else {
                float cj = 0.0f;
                if (lane < nwarps) {
                    const int U = len / VEC;
                    const int rem = len - U * VEC;
                    const int qq = U >> __popc(tpr - 1);
                    const int r = U & (tpr - 1);
                    const int a = lane * 32;
                    const int lo = r - a < 0 ? 0 : (r - a > 32 ? 32 : r - a);
                    cj = (float)(VEC * (32 * qq + lo) + ((rem != 0 && r >= a && r < a + 32) ? rem : 0));
                }
                for (int o = 1; o < pow2_ceil(nwarps); o <<= 1) {
                    const float co = __shfl_xor_sync(0xffffffffu, cj, o);
                    const float so = __shfl_xor_sync(0xffffffffu, sj, o);
                    const float qo = __shfl_xor_sync(0xffffffffu, qj, o);
                    merge_moments(cj, sj, qj, co, so, qo);
                }
            }
            pm = __shfl_sync(0xffffffffu, sj, 0);
            pl = __shfl_sync(0xffffffffu, qj, 0);
        }

        // Cluster merge: warp 0 pushes this CTA's pair into slot `rank` of
        // every CTA's receive buffer (st.async, counted on their barrier); all
        // threads wait for the cs pairs of this row on their own barrier.
        const int rb = (int)(it & 1);
        if (warp == 0 && lane < cs) {
            const uint32_t dst = map_to_rank(smem_addr(&recv[rb][rank]), (uint32_t)lane);
            const uint32_t dbar = map_to_rank(smem_addr(&recv_bar[rb]), (uint32_t)lane);
            st_async_pair(dst, pm, pl, dbar);
        }
        // Waited for even after an abort (the phase must complete before it is
        // re-armed, and the peers' pairs must land before this CTA exits).
        bool received = false;
        if (!*reinterpret_cast<volatile int*>(&exchange_broken)) {
            received = mbar_wait_cluster_bounded(&recv_bar[rb], (uint32_t)((it >> 1) & 1), 3 * wait_ns);
            if (!received) {
                *reinterpret_cast<volatile int*>(&exchange_broken) = 1;
                abort = true;
                flag_timeout();
            }
        }
        float qa = kSoftmax ? kNegInf : 0.0f, qb = 0.0f;
        if (lane < cs) {
            const float2 q = recv[rb][lane];
            qa = q.x;
            qb = q.y;
        }
        if constexpr (kSoftmax) {
            group_merge(qa, qb, pow2_ceil(cs));
            qa = __shfl_sync(0xffffffffu, qa, 0);
            qb = __shfl_sync(0xffffffffu, qb, 0);
            const float c = rescale_res(m, safe_max(qa), res) / qb;
            __syncwarp();
            if (tid == 0 && received) mbar_arrive_expect_tx(&recv_bar[rb], pair_bytes);  // re-armed for row it + 2
            if (OP::kMasked && !isfinite(c)) {
                // a NaN or +inf in the kept prefix, or an empty prefix: past the
                // prefix exactly 0 (NaN when the row keeps nothing); elsewhere the
                // fill's exp(-inf) = 0 times a finite c is already 0
                const int lv = slice_keep(row);
                const float masked = row_keep(args, row, N) > 0 ? 0.0f : __int_as_float(0x7fffffff);
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e)
                        v[k][e] = (tid + k * tpr) * VEC + e < lv ? v[k][e] * c : masked;
            } else {
#pragma unroll
                for (int k = 0; k < VPT; ++k)
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[k][e] *= c;
            }
        } else {
            float r, nmr = 0.0f;
            if constexpr (OP::kOp == RS_OP_RMSNORM) {
                const float ss = __shfl_sync(0xffffffffu, group_sum(qa, pow2_ceil(cs)), 0);
                r = 1.0f / sqrtf(ss / (float)N + args.eps);
            } else {
                const float mean = __shfl_sync(0xffffffffu, group_sum(qa, pow2_ceil(cs)), 0) / (float)N;
                const int nl = lane < cs ? hold_slice_len(lane, chunk, N) : 0;
                float term = 0.0f;
                if (nl > 0) {
                    const float dm = qa / (float)nl - mean;
                    term = fmaf((float)nl * dm, dm, qb);
                }
                const float m2 = __shfl_sync(0xffffffffu, group_sum(term, pow2_ceil(cs)), 0);
                r = 1.0f / sqrtf(m2 / (float)N + args.eps);
                nmr = -mean * r;
            }
            __syncwarp();
            if (tid == 0 && received) mbar_arrive_expect_tx(&recv_bar[rb], pair_bytes);  // re-armed for row it + 2
#pragma unroll
            for (int k = 0; k < VPT; ++k) {
                const int base = (tid + k * tpr) * VEC;  // within the slice
                float w[VEC], b[VEC];
                prm.template w_unit<DT, VEC>(base, w);
                if constexpr (OP::kOp == RS_OP_LAYERNORM) prm.template b_unit<DT, VEC>(base, b);
                if constexpr (OP::kOp == RS_OP_RMSNORM) unit_rms<VEC>(v[k], r, w);
                else unit_ln<VEC>(v[k], r, nmr, w, b);
            }
        }

        if (!abort) store_row_units<DT, VEC, VPT>(out + row * ldo + c0, tid, tpr, len, v);
    }

    allow_next_grid();  // persistent grid: the next kernel may begin once this CTA is done
    if (abort && tid == 0 && abort_it >= 0) {
        for (int64_t j = abort_it; j < abort_it + nslots; ++j) {
            if (cluster_id + j * n_clusters >= M) break;
            (void)mbar_wait_bounded(&bars[j % nslots], (uint32_t)((j / nslots) & 1), wait_ns);
        }
    }
    cluster.sync();  // no CTA leaves while a peer's pair may still be in flight to it
}

// The dynamic shared-memory ceiling is raised to the device maximum and the
// non-portable cluster sizes are allowed, once per device and instance.
template <int DT, int VPT, typename OP>
cudaError_t ensure_hold_attributes() {
    static std::mutex mu;
    static bool done[64] = {};
    auto kern = wide_hold_kernel<DT, VPT, OP>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev]) return cudaSuccess;
    int optin = 0;
    err = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (err != cudaSuccess) return err;
    const int dyn = optin - (int)kWideStaticSmem;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn > 0 ? dyn : 0);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
    done[dev] = true;
    return cudaSuccess;
}

template <int DT, int VPT, typename OP>
cudaError_t launch_hold_one(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                            int64_t ldo, cudaStream_t s, const RowArgs& a) {
    cudaError_t err = ensure_hold_attributes<DT, VPT, OP>();
    if (err != cudaSuccess) return err;
    // Cluster grids are launched in strict stream order: with programmatic
    // dependent launch the persistent clusters measured about 10 % slower.
    const uint64_t wait_ns = p.wait_limit_us > 0 ? (uint64_t)p.wait_limit_us * 1000ull : kWaitLimitNs;
    return launch_kernel(wide_hold_kernel<DT, VPT, OP>, (unsigned)p.grid, (unsigned)p.block_threads, p.smem_bytes,
                         s, p.cluster_size, true, in, out, M, N, ldi, ldo, (int)p.chunk_elems, p.stages, wait_ns,
                         p.withhold_copies, a);
}

template <int DT, typename OP>
cudaError_t launch_hold(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi, int64_t ldo,
                        cudaStream_t s, const RowArgs& a) {
    if (p.vec_elems != Traits<DT>::kVec) return cudaErrorInvalidConfiguration;
    switch (p.vec_per_thread) {
        case 1: return launch_hold_one<DT, 1, OP>(p, in, out, M, N, ldi, ldo, s, a);
        case 2: return launch_hold_one<DT, 2, OP>(p, in, out, M, N, ldi, ldo, s, a);
        case 4: return launch_hold_one<DT, 4, OP>(p, in, out, M, N, ldi, ldo, s, a);
        case 8: return launch_hold_one<DT, 8, OP>(p, in, out, M, N, ldi, ldo, s, a);
        default: return cudaErrorInvalidConfiguration;
    }
}

template <int DT, int VPT, typename OP>
cudaError_t max_clusters_hold_one(const rs_plan& p, int* n) {
    cudaError_t err = ensure_hold_attributes<DT, VPT, OP>();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.cluster_size, 1, 1);
    cfg.blockDim = dim3((unsigned)p.block_threads, 1, 1);
    cfg.dynamicSmemBytes = p.smem_bytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.cluster_size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, wide_hold_kernel<DT, VPT, OP>, &cfg);
}

template <int DT, typename OP>
cudaError_t max_clusters_hold(const rs_plan& p, int* n) {
    switch (p.vec_per_thread) {
        case 1: return max_clusters_hold_one<DT, 1, OP>(p, n);
        case 2: return max_clusters_hold_one<DT, 2, OP>(p, n);
        case 4: return max_clusters_hold_one<DT, 4, OP>(p, n);
        case 8: return max_clusters_hold_one<DT, 8, OP>(p, n);
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace rs
