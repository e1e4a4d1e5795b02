// Wide rows: a thread-block cluster per row.
//
// RS_PATH_CLUSTER (STAGED = true).  The row is cut into one contiguous slice
// per CTA of the cluster.  Each CTA pulls its slice into shared memory with
// bulk asynchronous copies (cp.async.bulk, the TMA engine; one mbarrier per
// stage) issued all at once by one thread, and folds every stage into a
// running pair (m, l) as soon as it lands -- the online normaliser of
// Milakov and Gimelshein as written in the mohakchugh.is-a.dev post ("How
// Flash Attention Uses Triton"): m' = max(m, max(block)),
// l' = l * exp(m - m') + sum(exp(block - m')).  The CTAs of the cluster then
// exchange their pairs through distributed shared memory (a few bytes per
// CTA; no multicast) and every CTA normalises its slice from shared memory
// and writes it.  Each input byte crosses HBM once and each output byte once,
// the fused-softmax traffic of the Hugging Face "triton-kernels" skill page
// ("Reference Kernel: Softmax": one DRAM read, one DRAM write per row), for
// rows far wider than one SM can hold.
//
// RS_PATH_STREAM (STAGED = false).  Same cluster split and merge, but the
// slice is read from global memory twice (once for (m, l), once to
// normalise).  It serves rows wider than the clusters' shared memory and rows
// whose pointers or strides forbid 16-byte bulk copies.
//
// Waits.  Every mbarrier wait is bounded by %globaltimer; a wait that runs
// out sets bit 0 of the device status word, the CTA stops issuing copies,
// gives its copies in flight a second bounded wait, and keeps taking part in
// the cluster barriers (which every CTA of a cluster reaches the same number
// of times, so they cannot wait forever) without writing its slice.
#include <cooperative_groups.h>

#include <mutex>

#include "rs_async.cuh"
#include "rs_common.cuh"
#include "rs_internal.h"
#include "rs_rowmath.cuh"

namespace cg = cooperative_groups;

namespace rs {

template <int DT, int VEC, bool STAGED>
__global__ void __launch_bounds__(kWideThreads)
wide_kernel(const void* in_, void* out_, int64_t M, int N, int64_t ldi, int64_t ldo, int chunk, int nslots) {
    using T = Traits<DT>;
    using S = typename T::storage;
    const S* in = static_cast<const S*>(in_);
    S* out = static_cast<S*>(out_);
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();

    // STAGED: `nslots` (1 or 2) slots, each holding this CTA's slice of one
    // row; with two, the slice of the next row is in flight while the current
    // one is computed (persistent grids, where a cluster serves many rows).
    extern __shared__ __align__(128) unsigned char stage_buf[];
    __shared__ __align__(8) uint64_t bars[2][kWideMaxStages];
    __shared__ float2 warp_part[2][kWideThreads / 32];
    __shared__ float2 cta_part[2];

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    constexpr int kWarps = kWideThreads / 32;

    // This CTA's slice [c0, c0 + len) of every row it serves.
    const int64_t c0l = (int64_t)rank * chunk < N ? (int64_t)rank * chunk : (int64_t)N;
    const int c0 = (int)c0l;
    const int len = (int)((c0l + chunk < N ? c0l + chunk : (int64_t)N) - c0l);
    const int units = (len + VEC - 1) / VEC;  // the last unit may be partial
    const int full = len / VEC;               // whole 16-byte units (bulk-copied when STAGED)
    const int stages = (units + kWideUnitsPerStage - 1) / kWideUnitsPerStage;
    const size_t slot_bytes = ((size_t)chunk * sizeof(S) + 15) & ~(size_t)15;

    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;

    // Thread 0: bulk-copy the slice of `row` into `slot`, one mbarrier per stage.
    auto issue = [&](int64_t row, int slot) {
        const S* src = in + row * ldi + c0;
        unsigned char* dst = stage_buf + (size_t)slot * slot_bytes;
        for (int s = 0; s < stages; ++s) {
            const int u0 = s * kWideUnitsPerStage;
            const int u1 = min(full, u0 + kWideUnitsPerStage);
            if (u1 > u0) {
                const uint32_t bytes = (uint32_t)(u1 - u0) * 16u;
                mbar_arrive_expect_tx(&bars[slot][s], bytes);
                bulk_load(dst + (size_t)u0 * 16, src + (size_t)u0 * VEC, bytes, &bars[slot][s]);
            } else {
                mbar_arrive(&bars[slot][s]);
            }
        }
    };

    wait_prior_grid();
    if (STAGED) {
        if (tid == 0) {
            for (int s = 0; s < kWideMaxStages; ++s) {
                mbar_init(&bars[0][s], 1);
                mbar_init(&bars[1][s], 1);
            }
            fence_mbar_init();
        }
        __syncthreads();
        if (tid == 0) {
            for (int j = 0; j < nslots; ++j)
                if (cluster_id + j * n_clusters < M) issue(cluster_id + j * n_clusters, j);
        }
    }

    bool abort = false;
    int64_t abort_it = -1;  // iteration in which the CTA gave up
    int64_t it = 0;
    for (int64_t row = cluster_id; row < M; row += n_clusters, ++it) {
        const S* xr = in + row * ldi + c0;
        S* yr = out + row * ldo + c0;
        const int slot = (int)(it % nslots);
        const uint32_t parity = (uint32_t)((it / nslots) & 1);
        const unsigned char* buf = stage_buf + (size_t)slot * slot_bytes;

        // Pass 1: online (m, l) over the slice, one stage at a time.
        float m = kNegInf, l = 0.0f;
        for (int s = 0; s < stages; ++s) {
            if (STAGED && !abort && !mbar_wait_bounded(&bars[slot][s], parity)) {
                abort = true;
                flag_timeout();
            }
            float v[kWideUnitsPerThread][VEC];
#pragma unroll
            for (int k = 0; k < kWideUnitsPerThread; ++k) {
                const int u = s * kWideUnitsPerStage + k * kWideThreads + tid;
                if (STAGED && u < full) {
                    T::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)u * 16), v[k]);
                } else if (u < units) {
                    load_unit<DT, VEC>(xr, u * VEC, len, v[k]);
                } else {
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[k][e] = kNegInf;
                }
            }
            float mb = kNegInf;
#pragma unroll
            for (int k = 0; k < kWideUnitsPerThread; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) mb = fmaxf(mb, v[k][e]);
            const float mn = fmaxf(m, mb);
            const float ms = safe_max(mn);
            float lb = 0.0f;
#pragma unroll
            for (int k = 0; k < kWideUnitsPerThread; ++k)
#pragma unroll
                for (int e = 0; e < VEC; ++e) lb += exp_diff(v[k][e], ms);
            l = l * rescale(m, ms) + lb;
            m = mn;
        }

        // CTA merge: warps, then the warps' pairs through shared memory.
        group_merge(m, l, 32);
        if (lane == 0) warp_part[it & 1][warp] = make_float2(m, l);
        abort = __syncthreads_or(abort) != 0;
        if (abort && abort_it < 0) abort_it = it;
        {
            float pm = kNegInf, pl = 0.0f;
            if (lane < kWarps) {
                const float2 q = warp_part[it & 1][lane];
                pm = q.x;
                pl = q.y;
            }
            group_merge(pm, pl, 32);
            m = pm;
            l = pl;
        }

        // Cluster merge through distributed shared memory.
        if (tid == 0) cta_part[it & 1] = make_float2(m, l);
        cluster.sync();
        {
            float pm = kNegInf, pl = 0.0f;
            if (lane < cs) {
                const float2* peer = cluster.map_shared_rank(&cta_part[it & 1], lane);
                const float2 q = *peer;
                pm = q.x;
                pl = q.y;
            }
            group_merge(pm, pl, 32);
            m = pm;
            l = pl;
        }

        // Pass 2: normalise the slice and write it.
        if (!abort) {
            const float ms = safe_max(m);
            const float inv = 1.0f / l;
            for (int s = 0; s < stages; ++s) {
#pragma unroll
                for (int k = 0; k < kWideUnitsPerThread; ++k) {
                    const int u = s * kWideUnitsPerStage + k * kWideThreads + tid;
                    if (u >= units) continue;
                    float v[VEC];
                    if (STAGED && u < full) {
                        T::unpack(*reinterpret_cast<const uint4*>(buf + (size_t)u * 16), v);
                    } else {
                        load_unit<DT, VEC>(xr, u * VEC, len, v);
                    }
#pragma unroll
                    for (int e = 0; e < VEC; ++e) v[e] = exp_diff(v[e], ms) * inv;
                    store_unit<DT, VEC>(yr, u * VEC, len, v);
                }
            }
        }
        if (STAGED) {
            __syncthreads();  // the slot is free
            if (tid == 0 && !abort && row + nslots * n_clusters < M) {
                fence_proxy_async_smem();  // earlier generic reads of the slot precede the copies
                issue(row + nslots * n_clusters, slot);
            }
        }
    }

    if (STAGED && abort && tid == 0) {
        // Let the copies that were in flight when the CTA gave up (that row's
        // and the next row's slices) land before the shared memory is released.
        for (int64_t j = abort_it; j < abort_it + nslots; ++j) {
            if (cluster_id + j * n_clusters >= M) break;
            for (int s = 0; s < stages; ++s)
                (void)mbar_wait_bounded(&bars[j % nslots][s], (uint32_t)((j / nslots) & 1));
        }
    }
    allow_next_grid();  // persistent grid: the next kernel may begin once this CTA is done
    cluster.sync();  // peers may still be reading cta_part
}

// RS_PATH_CLUSTER with the slice held in registers (RS_RING_REGISTERS).
//
// Persistent clusters; CTA `rank` of a cluster serves slice
// [rank * chunk, rank * chunk + len) of rows cluster_id, cluster_id +
// n_clusters, ...  Each CTA has `nslots` shared-memory slots filled by bulk
// copies.  A slot is only a landing buffer: the CTA copies its slice from the
// slot into registers (VPT 16-byte units per thread, fp32), releases the slot
// at once -- thread 0 immediately issues the copy of a later row into it --
// and then reduces and normalises from registers with one exp per element, so
// the next rows' bytes stream in while this row is reduced and stored.
// Merges: warps -> CTA through shared memory, CTAs -> cluster through
// distributed shared memory, all with the (m, l) operator.
template <int DT, int VPT>
__global__ void __launch_bounds__(VPT <= 4 ? kWideHoldThreads : kWideHoldThreads / 2, 2)
wide_hold_kernel(const void* in_, void* out_, int64_t M, int N, int64_t ldi, int64_t ldo, int chunk, int nslots) {
    using T = Traits<DT>;
    using S = typename T::storage;
    constexpr int VEC = T::kVec;
    const S* in = static_cast<const S*>(in_);
    S* out = static_cast<S*>(out_);
    cg::cluster_group cluster = cg::this_cluster();
    const int cs = (int)cluster.num_blocks();
    const int rank = (int)cluster.block_rank();

    extern __shared__ __align__(128) unsigned char slots[];
    __shared__ __align__(8) uint64_t bars[2];      // slot filled
    __shared__ __align__(8) uint64_t recv_bar[2];  // all CTAs' pairs of a row received
    __shared__ __align__(8) float2 recv[2][kMaxCluster];
    __shared__ float2 warp_part[2][kWideHoldThreads / 32];

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

    const int64_t cluster_id = blockIdx.x / cs;
    const int64_t n_clusters = gridDim.x / cs;

    auto issue = [&](int64_t row, int slot) {
        if (slice_bytes == 0) {
            mbar_arrive(&bars[slot]);
            return;
        }
        mbar_arrive_expect_tx(&bars[slot], slice_bytes);
        bulk_load(slots + (size_t)slot * slot_stride, in + row * ldi + c0, slice_bytes, &bars[slot]);
    };

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&recv_bar[0], 1);
        mbar_init(&recv_bar[1], 1);
        mbar_arrive_expect_tx(&recv_bar[0], pair_bytes);  // armed for rows 0 and 1 of this cluster
        mbar_arrive_expect_tx(&recv_bar[1], pair_bytes);
        fence_mbar_init();
    }
    __syncthreads();
    wait_prior_grid();
    if (tid == 0) {
        for (int j = 0; j < nslots; ++j)
            if (cluster_id + j * n_clusters < M) issue(cluster_id + j * n_clusters, j);
    }
    cluster.sync();  // every CTA's receive barriers are armed before any pair is sent

    bool abort = false;
    int64_t abort_it = -1;
    int64_t it = 0;
    for (int64_t row = cluster_id; row < M; row += n_clusters, ++it) {
        const int slot = (int)(it % nslots);
        const uint32_t parity = (uint32_t)((it / nslots) & 1);
        if (!abort && !mbar_wait_bounded(&bars[slot], parity)) {
            abort = true;
            flag_timeout();
        }
        const unsigned char* buf = slots + (size_t)slot * slot_stride;
        const S* xr = in + row * ldi + c0;

        float v[VPT][VEC];
        if ((tid + (VPT - 1) * tpr) < full) {
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
                    load_unit<DT, VEC>(xr, u * VEC, len, v[k]);  // ragged tail, or -inf past the slice
                }
            }
        }

        float m = kNegInf;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) m = fmaxf(m, v[k][e]);
        m = group_max(m, 32);
        const float ms = safe_max(m);
        float l = 0.0f;
#pragma unroll
        for (int k = 0; k < VPT; ++k)
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                v[k][e] = exp_diff(v[k][e], ms);
                l += v[k][e];
            }
        l = group_sum(l, 32);

        // CTA merge of the warps' pairs.  The barrier also ends every read of
        // the slot, which is then handed to the copy of a later row.
        if (lane == 0) warp_part[it & 1][warp] = make_float2(m, l);
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
        group_merge(pm, pl, pow2_ceil(nwarps));  // lanes 0..nwarps-1 hold the CTA's pair
        pm = __shfl_sync(0xffffffffu, pm, 0);
        pl = __shfl_sync(0xffffffffu, pl, 0);

        // Cluster merge: warp 0 pushes this CTA's pair into slot `rank` of
        // every CTA's receive buffer (st.async, counted on their barrier); all
        // threads wait for the cs pairs of this row on their own barrier.
        const int rb = (int)(it & 1);
        if (warp == 0 && lane < cs) {
            const uint32_t dst = map_to_rank(smem_addr(&recv[rb][rank]), (uint32_t)lane);
            const uint32_t dbar = map_to_rank(smem_addr(&recv_bar[rb]), (uint32_t)lane);
            st_async_pair(dst, pm, pl, dbar);
        }
        if (!abort && !mbar_wait_cluster_bounded(&recv_bar[rb], (uint32_t)((it >> 1) & 1))) {
            abort = true;
            flag_timeout();
        }
        float qm = kNegInf, ql = 0.0f;
        if (lane < cs) {
            const float2 q = recv[rb][lane];
            qm = q.x;
            ql = q.y;
        }
        group_merge(qm, ql, pow2_ceil(cs));
        qm = __shfl_sync(0xffffffffu, qm, 0);
        ql = __shfl_sync(0xffffffffu, ql, 0);
        const float c = rescale(m, safe_max(qm)) / ql;
        __syncwarp();
        if (tid == 0) mbar_arrive_expect_tx(&recv_bar[rb], pair_bytes);  // re-armed for row it + 2

        if (!abort) store_row_units<DT, VEC, VPT>(out + row * ldo + c0, tid, tpr, len, v, c);
    }

    allow_next_grid();  // persistent grid: the next kernel may begin once this CTA is done
    if (abort && tid == 0 && abort_it >= 0) {
        for (int64_t j = abort_it; j < abort_it + nslots; ++j) {
            if (cluster_id + j * n_clusters >= M) break;
            (void)mbar_wait_bounded(&bars[j % nslots], (uint32_t)((j / nslots) & 1));
        }
    }
    cluster.sync();  // no CTA leaves while a peer's pair may still be in flight to it
}

// Kernel attributes are per device: the dynamic shared-memory ceiling is
// raised to the device maximum and the non-portable cluster sizes are
// allowed, once per device and kernel instance.  Nothing ever lowers them.
template <typename Kern>
static cudaError_t set_wide_attributes(Kern kern, std::mutex& mu, bool* done) {
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

template <int DT, int VEC, bool STAGED>
static cudaError_t ensure_wide_attributes() {
    static std::mutex mu;
    static bool done[64] = {};
    return set_wide_attributes(wide_kernel<DT, VEC, STAGED>, mu, done);
}

template <int DT, int VPT>
static cudaError_t ensure_hold_attributes() {
    static std::mutex mu;
    static bool done[64] = {};
    return set_wide_attributes(wide_hold_kernel<DT, VPT>, mu, done);
}

template <int DT, int VPT>
static cudaError_t launch_hold_one(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                                   int64_t ldo, cudaStream_t s) {
    cudaError_t err = ensure_hold_attributes<DT, VPT>();
    if (err != cudaSuccess) return err;
    // Cluster grids are launched in strict stream order: with programmatic
    // dependent launch the persistent clusters measured about 10 % slower.
    return launch_kernel(wide_hold_kernel<DT, VPT>, (unsigned)p.grid, (unsigned)p.block_threads, p.smem_bytes, s,
                         p.cluster_size, true, in, out, M, N, ldi, ldo, (int)p.chunk_elems, p.stages);
}

template <int DT, int VEC, bool STAGED>
static cudaError_t launch_wide_one(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                                   int64_t ldi, int64_t ldo, cudaStream_t s) {
    auto kern = wide_kernel<DT, VEC, STAGED>;
    cudaError_t err = ensure_wide_attributes<DT, VEC, STAGED>();
    if (err != cudaSuccess) return err;
    const int nslots = (STAGED && p.grid / p.cluster_size < M) ? 2 : 1;
    return launch_kernel(kern, (unsigned)p.grid, (unsigned)kWideThreads, STAGED ? p.smem_bytes : 0, s,
                         p.cluster_size, true, in, out, M, N, ldi, ldo, (int)p.chunk_elems, nslots);
}

template <int DT>
static cudaError_t launch_wide_dt(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                                  int64_t ldi, int64_t ldo, cudaStream_t s) {
    constexpr int KV = Traits<DT>::kVec;
    if (p.path == RS_PATH_CLUSTER && p.vec_elems == KV && p.ring_values == RS_RING_REGISTERS) {
        switch (p.vec_per_thread) {
            case 1: return launch_hold_one<DT, 1>(p, in, out, M, N, ldi, ldo, s);
            case 2: return launch_hold_one<DT, 2>(p, in, out, M, N, ldi, ldo, s);
            case 4: return launch_hold_one<DT, 4>(p, in, out, M, N, ldi, ldo, s);
            case 8: return launch_hold_one<DT, 8>(p, in, out, M, N, ldi, ldo, s);
            default: return cudaErrorInvalidConfiguration;
        }
    }
    if (p.path == RS_PATH_CLUSTER && p.vec_elems == KV)
        return launch_wide_one<DT, KV, true>(p, in, out, M, N, ldi, ldo, s);
    if (p.path == RS_PATH_STREAM && p.vec_elems == KV)
        return launch_wide_one<DT, KV, false>(p, in, out, M, N, ldi, ldo, s);
    if (p.path == RS_PATH_STREAM && p.vec_elems == 1)
        return launch_wide_one<DT, 1, false>(p, in, out, M, N, ldi, ldo, s);
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_wide(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                        int64_t ldo, cudaStream_t s) {
    switch (p.dtype) {
        case RS_F32: return launch_wide_dt<RS_F32>(p, in, out, M, N, ldi, ldo, s);
        case RS_F16: return launch_wide_dt<RS_F16>(p, in, out, M, N, ldi, ldo, s);
        case RS_BF16: return launch_wide_dt<RS_BF16>(p, in, out, M, N, ldi, ldo, s);
        default: return cudaErrorInvalidValue;
    }
}

template <int DT, int VEC, bool STAGED>
static cudaError_t max_clusters_one(const rs_plan& p, int* n) {
    auto kern = wide_kernel<DT, VEC, STAGED>;
    cudaError_t err = ensure_wide_attributes<DT, VEC, STAGED>();
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.cluster_size, 1, 1);
    cfg.blockDim = dim3(kWideThreads, 1, 1);
    cfg.dynamicSmemBytes = STAGED ? p.smem_bytes : 0;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.cluster_size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(n, kern, &cfg);
}

template <int DT, int VPT>
static cudaError_t max_clusters_hold(const rs_plan& p, int* n) {
    cudaError_t err = ensure_hold_attributes<DT, VPT>();
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
    return cudaOccupancyMaxActiveClusters(n, wide_hold_kernel<DT, VPT>, &cfg);
}

template <int DT>
static cudaError_t max_clusters_dt(const rs_plan& p, int* n) {
    constexpr int KV = Traits<DT>::kVec;
    if (p.path == RS_PATH_CLUSTER && p.ring_values == RS_RING_REGISTERS) {
        switch (p.vec_per_thread) {
            case 1: return max_clusters_hold<DT, 1>(p, n);
            case 2: return max_clusters_hold<DT, 2>(p, n);
            case 4: return max_clusters_hold<DT, 4>(p, n);
            case 8: return max_clusters_hold<DT, 8>(p, n);
            default: return cudaErrorInvalidConfiguration;
        }
    }
    if (p.path == RS_PATH_CLUSTER) return max_clusters_one<DT, KV, true>(p, n);
    if (p.vec_elems == KV) return max_clusters_one<DT, KV, false>(p, n);
    return max_clusters_one<DT, 1, false>(p, n);
}

cudaError_t wide_max_active_clusters(const rs_plan& p, int* n) {
    switch (p.dtype) {
        case RS_F32: return max_clusters_dt<RS_F32>(p, n);
        case RS_F16: return max_clusters_dt<RS_F16>(p, n);
        case RS_BF16: return max_clusters_dt<RS_BF16>(p, n);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t read_status_wide(unsigned int* flags, bool clear) { return read_unit_status(flags, clear); }

}  // namespace rs
