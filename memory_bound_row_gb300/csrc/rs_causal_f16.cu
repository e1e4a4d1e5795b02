// Softmax under a causal mask (rowsoftmax_causal_fwd) for f16 storage: the
// register rows, the ring and the register-holding clusters instantiated
// with OpSoftmaxCausal, which copy and read only each row's kept prefix (the
// ring by per-thread asynchronous copies, rs_ring_cp.cuh; the bulk-copy ring
// when forced, which stages whole rows).
#include "rs_hold.cuh"
#include "rs_ring.cuh"
#include "rs_ring_cp.cuh"
#include "rs_rows.cuh"

namespace rs {

cudaError_t launch_causal_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                            int64_t ldo, cudaStream_t s, const RowArgs& a) {
    constexpr int KV = Traits<RS_F16>::kVec;
    switch (p.path) {
        case RS_PATH_ROWS:
            if (p.vec_elems == KV)
                return RowsDispatch<RS_F16, KV, OpSoftmaxCausal, RS_VPT_VEC_16>::go(p, in, out, M, N, ldi, ldo, s, a);
            if (p.vec_elems == 1)
                return RowsDispatch<RS_F16, 1, OpSoftmaxCausal, RS_VPT_SCALAR>::go(p, in, out, M, N, ldi, ldo, s, a);
            return cudaErrorInvalidConfiguration;
        case RS_PATH_RING:
            if (p.vec_elems != KV) return cudaErrorInvalidConfiguration;
            if (p.ring_values == RS_RING_THREAD_COPIES)
                return RingCpDispatch<RS_F16, OpSoftmaxCausal, RS_VPT_VEC_16>::go(p, in, out, M, N, ldi, ldo, s, a);
            return RingDispatch<RS_F16, OpSoftmaxCausal, RS_VPT_VEC_16>::go(p, in, out, M, N, ldi, ldo, s, a);
        case RS_PATH_CLUSTER:
            if (p.ring_values != RS_RING_REGISTERS) return cudaErrorInvalidConfiguration;
            return launch_hold<RS_F16, OpSoftmaxCausal>(p, in, out, M, N, ldi, ldo, s, a);
        default:
            return cudaErrorInvalidConfiguration;
    }
}

cudaError_t causal_max_clusters_f16(const rs_plan& p, int* n) { return max_clusters_hold<RS_F16, OpSoftmaxCausal>(p, n); }

cudaError_t read_status_causal_f16(unsigned int* flags, bool clear) { return read_unit_status(flags, clear); }

}  // namespace rs
