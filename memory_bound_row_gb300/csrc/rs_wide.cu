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
// The register-holding variant of RS_PATH_CLUSTER (RS_RING_REGISTERS, the
// default for slices that fit a CTA's registers) is in rs_hold.cuh.
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
#include "rs_hold.cuh"
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
                                  int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a) {
    constexpr int KV = Traits<DT>::kVec;
    if (p.path == RS_PATH_CLUSTER && p.vec_elems == KV && p.ring_values == RS_RING_REGISTERS) {
        return launch_hold<DT, OpSoftmax>(p, in, out, M, N, ldi, ldo, s, a);
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
                        int64_t ldo, cudaStream_t s, const RowArgs& a) {
    if (a.mask_period > 0) return cudaErrorInvalidConfiguration;  // the causal mask has its own instances
    switch (p.dtype) {
        case RS_F32: return launch_wide_dt<RS_F32>(p, in, out, M, N, ldi, ldo, s, a);
        case RS_F16: return launch_wide_dt<RS_F16>(p, in, out, M, N, ldi, ldo, s, a);
        case RS_BF16: return launch_wide_dt<RS_BF16>(p, in, out, M, N, ldi, ldo, s, a);
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

template <int DT>
static cudaError_t max_clusters_dt(const rs_plan& p, int* n) {
    constexpr int KV = Traits<DT>::kVec;
    if (p.path == RS_PATH_CLUSTER && p.ring_values == RS_RING_REGISTERS) {
        return max_clusters_hold<DT, OpSoftmax>(p, n);
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
