// LayerNorm instances that merge per-lane moments once (rs_rowmath.cuh) for
// fp16 storage, on the register rows and the ring: OpLayerNormWarp for rows
// inside one warp, OpLayerNormWhole for vectorised rows that fill their
// threads exactly over a power-of-two number of warps (on the ring with at most
// 32 values a thread: OpLayerNormWholeHeld, weight and bias in registers;
// other fp32 ring rows at 8 units a thread: OpLayerNormHeld).  The other
// shapes take OpLayerNorm (rs_norm_f16.cu).
#include "rs_ring.cuh"
#include "rs_rows.cuh"

namespace rs {

cudaError_t launch_lnmerge_f16(const rs_plan& p, const void* in, void* out, int64_t M, int N, int64_t ldi,
                               int64_t ldo, cudaStream_t s, const RowArgs& a) {
    constexpr int KV = Traits<RS_F16>::kVec;
    const int kind = layernorm_merge_kind(p, N, KV);
    if (kind == 1) {
        if (p.path == RS_PATH_RING) {
            if (p.vec_elems != KV) return cudaErrorInvalidConfiguration;
            return RingDispatch<RS_F16, OpLayerNormWarp, RS_VPT_NORM_VEC>::go(p, in, out, M, N, ldi, ldo, s, a);
        }
        if (p.vec_elems == KV)
            return RowsDispatch<RS_F16, KV, OpLayerNormWarp, RS_VPT_NORM_VEC>::go(p, in, out, M, N, ldi, ldo, s, a);
        if (p.vec_elems == 1)
            return RowsDispatch<RS_F16, 1, OpLayerNormWarp, RS_VPT_NORM_SCALAR>::go(p, in, out, M, N, ldi, ldo, s, a);
        return cudaErrorInvalidConfiguration;
    }
    if (kind == 3)
        return RingDispatch<RS_F16, OpLayerNormWholeHeld, 1, 2, 3, 4>::go(p, in, out, M, N, ldi, ldo, s, a);
    if (kind == 2) {
        if (p.path == RS_PATH_RING)
            return RingDispatch<RS_F16, OpLayerNormWhole, RS_VPT_NORM_VEC>::go(p, in, out, M, N, ldi, ldo, s, a);
        return RowsDispatch<RS_F16, KV, OpLayerNormWhole, RS_VPT_NORM_VEC>::go(p, in, out, M, N, ldi, ldo, s, a);
    }
    return cudaErrorInvalidConfiguration;
}

cudaError_t read_status_lnmerge_f16(unsigned int* flags, bool clear) { return read_unit_status(flags, clear); }

}  // namespace rs
