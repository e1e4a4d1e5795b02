// LayerNorm on rows held inside one warp (OpLayerNormWarp: each lane's
// moments about its own mean, merged in one butterfly) for fp32 storage:
// the register rows and the ring.  Wider rows take OpLayerNorm (rs_norm_f32.cu).
#include "rs_ring.cuh"
#include "rs_rows.cuh"

namespace rs {

cudaError_t launch_lnwarp_f32(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                              int64_t ldo, cudaStream_t s, const RowArgs& a) {
    constexpr int KV = Traits<RS_F32>::kVec;
    if (p.threads_per_row > 32) return cudaErrorInvalidConfiguration;
    switch (p.path) {
        case RS_PATH_ROWS:
            if (p.vec_elems == KV)
                return RowsDispatch<RS_F32, KV, OpLayerNormWarp, RS_VPT_NORM_VEC>::go(p, in, out, M, N, ldi, ldo, s, a);
            if (p.vec_elems == 1)
                return RowsDispatch<RS_F32, 1, OpLayerNormWarp, RS_VPT_NORM_SCALAR>::go(p, in, out, M, N, ldi, ldo, s,
                                                                                      a);
            return cudaErrorInvalidConfiguration;
        case RS_PATH_RING:
            if (p.vec_elems != KV) return cudaErrorInvalidConfiguration;
            return RingDispatch<RS_F32, OpLayerNormWarp, RS_VPT_NORM_VEC>::go(p, in, out, M, N, ldi, ldo, s, a);
        default:
            return cudaErrorInvalidConfiguration;
    }
}

cudaError_t read_status_lnwarp_f32(unsigned int* flags, bool clear) { return read_unit_status(flags, clear); }

}  // namespace rs
