// RMSNorm and LayerNorm instances (register rows, ring, register-holding
// clusters, one-CTA-per-row streaming) for f16 storage: RS_PATH_ROWS,
// RS_PATH_RING and the one-CTA-per-row streaming kernel (rs_norm.cuh).
#include "rs_hold.cuh"
#include "rs_norm.cuh"
#include "rs_ring.cuh"
#include "rs_rows.cuh"

namespace rs {

template <typename OP>
static cudaError_t launch_norm_op(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                                  int64_t ldo, cudaStream_t s, const RowArgs& a) {
    constexpr int KV = Traits<RS_F16>::kVec;
    switch (p.path) {
        case RS_PATH_ROWS:
            if (p.vec_elems == KV)
                return RowsDispatch<RS_F16, KV, OP, RS_VPT_NORM_VEC>::go(p, in, out, M, N, ldi, ldo, s, a);
            if (p.vec_elems == 1)
                return RowsDispatch<RS_F16, 1, OP, RS_VPT_NORM_SCALAR>::go(p, in, out, M, N, ldi, ldo, s, a);
            return cudaErrorInvalidConfiguration;
        case RS_PATH_RING:
            if (p.vec_elems != KV) return cudaErrorInvalidConfiguration;
            return RingDispatch<RS_F16, OP, RS_VPT_NORM_VEC>::go(p, in, out, M, N, ldi, ldo, s, a);
        case RS_PATH_CLUSTER:
            return launch_hold<RS_F16, OP>(p, in, out, M, N, ldi, ldo, s, a);
        case RS_PATH_STREAM:
            if (p.vec_elems == KV) return launch_norm_stream<RS_F16, KV, OP>(p, in, out, M, N, ldi, ldo, s, a);
            if (p.vec_elems == 1) return launch_norm_stream<RS_F16, 1, OP>(p, in, out, M, N, ldi, ldo, s, a);
            return cudaErrorInvalidConfiguration;
        default:
            return cudaErrorInvalidConfiguration;
    }
}

cudaError_t launch_norm_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                            int64_t ldo, cudaStream_t s, const RowArgs& a) {
    if (p.op == RS_OP_RMSNORM && rmsnorm_ring_held(p, Traits<RS_F16>::kVec))
        return RingDispatch<RS_F16, OpRmsNormHeld, 1, 2, 3, 4>::go(p, in, out, M, N, ldi, ldo, s, a);
    if (p.op == RS_OP_RMSNORM) return launch_norm_op<OpRmsNorm>(p, in, out, M, N, ldi, ldo, s, a);
    if (p.op == RS_OP_LAYERNORM && layernorm_merge_kind(p, N, Traits<RS_F16>::kVec) != 0)
        return launch_lnmerge_f16(p, in, out, M, N, ldi, ldo, s, a);
    if (p.op == RS_OP_LAYERNORM) return launch_norm_op<OpLayerNorm>(p, in, out, M, N, ldi, ldo, s, a);
    return cudaErrorInvalidConfiguration;
}

cudaError_t norm_max_clusters_f16(const rs_plan& p, int* n) {
    if (p.op == RS_OP_RMSNORM) return max_clusters_hold<RS_F16, OpRmsNorm>(p, n);
    if (p.op == RS_OP_LAYERNORM) return max_clusters_hold<RS_F16, OpLayerNorm>(p, n);
    return cudaErrorInvalidConfiguration;
}

cudaError_t read_status_norm_f16(unsigned int* flags, bool clear) { return read_unit_status(flags, clear); }

}  // namespace rs
