// RS_PATH_ROWS and RS_PATH_RING instances for f16 storage.
#include "rs_ring.cuh"
#include "rs_rows.cuh"

namespace rs {

cudaError_t launch_rows_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                            int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a) {
    if (p.vec_elems == Traits<RS_F16>::kVec)
        return RowsDispatch<RS_F16, Traits<RS_F16>::kVec, OpSoftmax, RS_VPT_VEC_16>::go(p, in, out, M, N, ldi, ldo, s, a);
    if (p.vec_elems == 1)
        return RowsDispatch<RS_F16, 1, OpSoftmax, RS_VPT_SCALAR>::go(p, in, out, M, N, ldi, ldo, s, a);
    return cudaErrorInvalidConfiguration;
}

cudaError_t launch_ring_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N,
                            int64_t ldi, int64_t ldo, cudaStream_t s, const RowArgs& a) {
    if (p.vec_elems != Traits<RS_F16>::kVec) return cudaErrorInvalidConfiguration;
    return RingDispatch<RS_F16, OpSoftmax, RS_VPT_VEC_16>::go(p, in, out, M, N, ldi, ldo, s, a);
}

cudaError_t read_status_f16(unsigned int* flags, bool clear) { return read_unit_status(flags, clear); }

}  // namespace rs
