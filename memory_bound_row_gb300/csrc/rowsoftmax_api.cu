// The C ABI of include/rowsoftmax.h: argument validation, the planner that
// picks a kernel family and launch shape, and the dispatch onto the
// caller's stream.  Host code only; the kernels live in rs_rows_*.cu and
// rs_wide.cu.
#include <cuda_runtime.h>

#include <limits.h>
#include <stdint.h>
#include <string.h>

#include <initializer_list>
#include <mutex>

#include "rowsoftmax.h"
#include "rs_internal.h"

namespace {

thread_local int t_last_cuda_error = 0;

int fail_cuda(cudaError_t e) {
    t_last_cuda_error = (int)e;
    return RS_ERR_CUDA;
}

int elem_size(int dtype) { return dtype == RS_F32 ? 4 : 2; }

// Largest accepted N: keeps every in-kernel element index (which may run a
// 16-byte unit past N) inside int.
constexpr int64_t kMaxN = (int64_t)INT_MAX - 64;
constexpr int64_t kMaxGrid = (int64_t)INT_MAX;
constexpr int64_t kMaxMaskOffset = (int64_t)1 << 62;  // keeps (r mod P) + 1 + offset inside int64

// Auto-planner knobs.
constexpr int kRowsTargetValues = 32;             // fp32 values a thread holds (auto)
constexpr int kRowsTargetValuesLn16 = 64;         // ... for LayerNorm on 16-bit rows up to 8192 values (measured faster)
constexpr int kRowsMaxSingleWarpValues = 64;      // ... up to this many when it keeps a row in one warp
constexpr int64_t kRowsMaxRowBytes = 32 * 1024;   // auto: rows up to this go to RS_PATH_ROWS
constexpr int64_t kRowsMaxRowBytesF32 = 64 * 1024;  // ... fp32 softmax rows (measured: rows beat clusters to 64 KB)
constexpr int64_t kClusterTargetSlice = 64 * 1024;  // auto: bytes of row slice per CTA
constexpr int64_t kRingMinRowBytes = 512;           // auto: shorter rows stay on RS_PATH_ROWS
constexpr int64_t kRingMaxRowBytesSoftmax16 = 64 * 1024;  // auto: the ring's limit for wide 16-bit softmax rows
constexpr int kClusterThinValues = 16;                // ... taken when the cluster's CTAs hold at most this a thread
constexpr int kLnHeldMinThreadsF32 = 128;            // auto: fp32 LayerNorm rows not filling a power-of-two
                                                      // number of warps, of 128..256 threads at 8 units a
                                                      // thread, take the ring with held weight and bias ...
constexpr int kLnHeldMinWarpsF32 = 14;               // ... when this many warps of it fit an SM
constexpr int kRingDefaultStages = 2;               // auto: more stages cost resident CTAs (measured)
constexpr int kRingCopyMaxStages = 3;               // stages the per-thread-copy ring is instantiated for

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

bool valid_tpr(int tpr) {
    if (tpr >= 1 && tpr <= 32) return (tpr & (tpr - 1)) == 0;
    return tpr > 32 && tpr <= rs::kRowsMaxThreads && tpr % 32 == 0;
}

// The per-thread unit counts instantiated for (op, dtype, vec) and their number.
const int* vpt_table(int op, int dtype, int vec, int* n) {
    if (op != RS_OP_SOFTMAX) {
        if (vec == 1) {
            *n = (int)(sizeof(rs::kVptNormScalar) / sizeof(int));
            return rs::kVptNormScalar;
        }
        *n = (int)(sizeof(rs::kVptNormVec) / sizeof(int));
        return rs::kVptNormVec;
    }
    if (vec == 1) {
        *n = (int)(sizeof(rs::kVptScalar) / sizeof(int));
        return rs::kVptScalar;
    }
    if (dtype == RS_F32) {
        *n = (int)(sizeof(rs::kVptVecF32) / sizeof(int));
        return rs::kVptVecF32;
    }
    *n = (int)(sizeof(rs::kVptVec16) / sizeof(int));
    return rs::kVptVec16;
}

bool vpt_instantiated(int op, int dtype, int vec, int vpt) {
    int n = 0;
    const int* t = vpt_table(op, dtype, vec, &n);
    for (int i = 0; i < n; ++i)
        if (t[i] == vpt) return true;
    return false;
}

// Smallest instantiated count >= want, or 0.
int vpt_at_least(int op, int dtype, int vec, int64_t want) {
    int n = 0;
    const int* t = vpt_table(op, dtype, vec, &n);
    for (int i = 0; i < n; ++i)
        if (t[i] >= want) return t[i];
    return 0;
}

int plan_rows(int dtype, int vec, int64_t M, int64_t units, const rs_options& o, rs_plan* p,
              bool registers_hold_row = true, int sm_count = 0) {
    int tpr = o.threads_per_row;
    int vpt = o.vec_per_thread;
    if (tpr && !valid_tpr(tpr)) return RS_ERR_INVALID_ARG;
    if (vpt && !vpt_instantiated(p->op, dtype, vec, vpt)) return RS_ERR_NO_PATH;
    if (!tpr) {
        if (vpt) {
            const int64_t need = ceil_div(units, vpt);
            if (need <= 32) {
                tpr = 1;
                while (tpr < need) tpr <<= 1;
            } else {
                tpr = (int)round_up(need, 32);
            }
        } else {
            int n_inst = 0;
            const int* inst = vpt_table(p->op, dtype, vec, &n_inst);
            // (LayerNorm on 16-bit rows over 8192 values: 32 values a thread,
            // measured 7-19 % faster than 64.)
            const int target = p->op == RS_OP_LAYERNORM && dtype != RS_F32 && vec > 1 && units * vec <= 8192
                                   ? kRowsTargetValuesLn16
                                   : kRowsTargetValues;
            int vt = target / vec > 0 ? target / vec : 1;
            if (vt > inst[n_inst - 1]) vt = inst[n_inst - 1];
            // 16-bit rows that one warp can hold at up to 64 values a thread
            // stay in one warp: no CTA barrier per row (measured faster).
            if (dtype != RS_F32 && vec > 1 && units > 32 * vt && units <= 32 * (kRowsMaxSingleWarpValues / vec))
                vt = (int)ceil_div(units, 32);
            const int64_t need = ceil_div(units, vt);
            if (need <= 32) {
                tpr = 1;
                while (tpr < need) tpr <<= 1;
            } else {
                tpr = (int)round_up(need, 32);
            }
        }
        if (tpr > rs::kRowsMaxThreads) return RS_ERR_NO_PATH;
    }
    if (!vpt) {
        vpt = vpt_at_least(p->op, dtype, vec, ceil_div(units, tpr));
        if (!vpt) return RS_ERR_NO_PATH;
    }
    if ((int64_t)tpr * vpt < units) return RS_ERR_NO_PATH;
    if (vpt * vec > rs::kRowsMaxValuesPerThread) return RS_ERR_NO_PATH;
    const int block_limit = registers_hold_row ? rs::rows_block_limit(vpt, vec) : rs::kRingRereadThreads;
    if (tpr > block_limit) return RS_ERR_NO_PATH;

    int block = o.block_threads;
    if (block) {
        if (block % tpr != 0 || block % 32 != 0) return RS_ERR_INVALID_ARG;
        if (block > block_limit) return RS_ERR_NO_PATH;
    } else {
        // fp32 softmax rows of one or two warps: 128-thread CTAs (measured on
        // M = 4096, N = 768 .. 2048: +1 % at one warp a row, +6 to +10 % at two,
        // against 256-thread CTAs); others 256.
        const int cta = p->op == RS_OP_SOFTMAX && dtype == RS_F32 && vec > 1 && (tpr == 32 || tpr == 64) ? 128 : 256;
        int rpc = tpr >= cta ? 1 : cta / tpr;
        // Few rows: fewer rows a CTA, so that at least two CTAs reach each SM.
        if (sm_count > 0 && rpc > 1) {
            const int64_t fit = M / (2 * (int64_t)sm_count);
            if (fit < rpc) rpc = fit < 1 ? 1 : (int)fit;
            while ((tpr * rpc) % 32) ++rpc;  // whole warps
        }
        block = tpr * rpc;
    }
    const int rows_per_cta = block / tpr;
    int64_t grid = ceil_div(M, rows_per_cta);
    if (o.grid_limit > 0 && grid > o.grid_limit) grid = o.grid_limit;
    if (grid > kMaxGrid) grid = kMaxGrid;

    p->path = RS_PATH_ROWS;
    p->vec_elems = vec;
    p->threads_per_row = tpr;
    p->vec_per_thread = vpt;
    p->rows_per_cta = rows_per_cta;
    p->block_threads = block;
    p->cluster_size = 1;
    p->stages = 0;
    p->chunk_elems = 0;
    p->grid = grid;
    p->smem_bytes = 0;
    return RS_OK;
}

// Resident CTAs of one SM for a kernel of `block` threads and `smem` dynamic
// bytes, assuming the register budget its launch bound allows.
int64_t ctas_per_sm(const rs_device_info& dev, int block, size_t smem, int regs_per_thread) {
    int64_t by_threads = dev.max_threads_per_sm > 0 ? dev.max_threads_per_sm / block : 1;
    int64_t by_regs = 65536 / ((int64_t)block * regs_per_thread);
    int64_t by_smem = dev.max_smem_per_sm > 0 ? (int64_t)dev.max_smem_per_sm / (int64_t)(smem + 2048) : 1;
    int64_t n = by_threads;
    if (by_regs < n) n = by_regs;
    if (by_smem < n) n = by_smem;
    if (n > 32) n = 32;
    return n < 1 ? 1 : n;
}

// Ring shapes measured for 16-bit softmax rows of 257 to 4096 16-byte units
// (bf16, 2^28 / N to 2^29 / N rows, graph-replayed, against the 4-unit shape
// planned otherwise and, from 16384 values, the clusters):
//  - a multiple of 256 units: 8 units a thread, three stages (N = 4096 +9 %,
//    6144 +8 %, 8192 +7.8 %, 12288 +13 %, 16384 +12 %, 20480 +4.4 %, 24576
//    +3.5 %, 28672 +16 %, 32768 +8.3 %); several rows a CTA where they fill
//    448 to 512 threads (4096, 6144, 8192, 16384), else one row a CTA (12288:
//    two rows in 384 threads measured 7 % slower);
//  - else 5 units a thread where they fill whole warps exactly, or 6 where
//    they do and 4 do not: one row a CTA, two stages (2560 +34 %, 4608 +25 %,
//    5120 +7.6 %; 6 units at 3072, where 4 fill exactly, -1 to -4 %);
//  - else 8 units a thread on whole warps: rows of up to 768 units one row a
//    CTA and two stages (3584 +10 %, 5632 +17 %), wider rows as the first case.
// Given 4 row groups an SM at least, so that every CTA loops over its stages.
struct RingShape {
    int tpr, vpt, block, stages;
};
int ring16_block(int tpr) {
    const int filled = (512 / tpr) * tpr;
    return tpr <= 256 && filled >= 448 ? filled : tpr;
}
bool ring16_softmax_shape(int64_t units, int64_t M, int sm_count, RingShape* shape) {
    if (units <= 256 || units > 4096) return false;
    const auto exact = [units](int v) { return units % v == 0 && (units / v) % 32 == 0; };
    RingShape r{};
    if (units % 256 == 0) {
        r.tpr = (int)(units / 8);
        r.vpt = 8;
        r.stages = 3;
        r.block = ring16_block(r.tpr);
    } else if (exact(5)) {
        r = {(int)(units / 5), 5, (int)(units / 5), 2};
    } else if (exact(6) && !exact(4)) {
        r = {(int)(units / 6), 6, (int)(units / 6), 2};
    } else if (exact(4) && units <= 768) {
        return false;  // the planned 4-unit shape
    } else {
        r.tpr = (int)round_up(ceil_div(units, 8), 32);
        r.vpt = 8;
        if (units <= 768) {
            r.block = r.tpr;
            r.stages = 2;
        } else {
            r.block = ring16_block(r.tpr);
            r.stages = 3;
        }
    }
    if (M < (int64_t)(r.block / r.tpr) * 4 * sm_count) return false;
    *shape = r;
    return true;
}

// The causal mask's 16-bit rows of 257 to 4096 units (2049 to 32768 values)
// on its copy ring: 8 units a thread on whole warps (or 5 or 6 where they
// fill whole warps exactly and 8 do not), one row a CTA, two stages (bf16,
// period = N, 2^28 / N rows, against the 4-unit shape and the clusters
// planned otherwise: 4096 +36 %, 6000 +19 %, 6144 +33 %, 8192 +31 %, 12288
// +17 %, 16384 +21 %, 32768 +22 %), given 4 rows an SM at least.
bool causal16_ring(int64_t units, int64_t M, int sm_count) {
    return units > 256 && units <= 4096 && M >= 4 * (int64_t)sm_count;
}

// The causal mask's 16-bit rows of 32 to 256 units (256 to 2048 values) on
// its copy ring: the fewest lanes (a power of two, at least 4) that hold the
// row at up to 8 units a thread, 512-thread CTAs, two stages (bf16, period =
// N, 2^28 / N rows, against the 4-unit shape planned otherwise: 256 +21 %, 512
// +27 %, 768 +37 %, 1024 +25 %; 1280, 1536 and 2048 keep 32 lanes), given 4
// row groups an SM.
bool causal16_narrow(int64_t units, int64_t M, int sm_count, int* tpr, int* vpt) {
    if (units < 32 || units > 256) return false;
    int t = 4;
    while (t * 8 < units) t <<= 1;
    const int64_t need = ceil_div(units, t);
    const int v = need <= 2 ? 2 : need <= 3 ? 3 : need <= 4 ? 4 : need <= 5 ? 5 : need <= 6 ? 6 : 8;
    if (M < (int64_t)(512 / t) * 4 * sm_count) return false;
    *tpr = t;
    *vpt = v;
    return true;
}

// Shapes measured for the ring's 16-bit rows, against the first-guess plan
// (about 32 values a thread, 256-thread CTAs, two stages) and, where they
// were planned, the clusters: bf16 rows, 2^13 to 2^20 of them, graph-replayed
// in one call, every shape checked against the oracle first.  `want` gets the
// threads a row, units a thread, CTA size and stages to take (0: as planned);
// false where the first guess stands.
//
// softmax      rows of one warp at 4 or 8 units a thread: 512-thread CTAs
//              (2048 values +3.3 %; at 5 or 6 units 256-thread CTAs measured
//              4-12 % faster); rows that 16 lanes fill exactly at 4-8 units:
//              16 lanes, 512-thread CTAs at 4 or 8 units, else 256 (512 +9 %,
//              768 +2.9 %, 1024 +6 %); rows of 257 to 4096 units:
//              ring16_softmax_shape (+4 to +34 % from 2560 to 32768 values);
// causal mask  rows of 32 to 256 units: causal16_narrow (+21 to +37 %); of 257
//              to 4096 units: its copy ring at 8 units a thread (5 or 6 where
//              they fill whole warps exactly and 8 do not; 5 or 6 where they
//              fill 16 warps exactly: 20480 +5.7 %, 24576 +1.9 % against 8
//              units, 10240 -18 %, 12288 -0.6 % at 8 warps), one row a CTA, two
//              stages (+15 to +47 % from 2560 to 32768 values);
// LayerNorm    rows of 32 to 128 units: about 4 units a thread on the fewest
//              lanes that hold them (+3 to +24 %); rows of one warp: 128-thread
//              CTAs (2048 +5.8 %); 257 to 768 units: 6 (else 5, else 4) units
//              a thread, one row a CTA where they fill whole warps exactly (at
//              5 units at least 128 threads a CTA), else 4 units (+3 to +45 %;
//              5 units: 2560 +40 %, 5120 +12 %); 1536 and 3072 units: 6 units a
//              thread on 8 or 16 warps, one row a CTA (12288 +9.1 %, 24576
//              +8.6 %; on 6, 9, 10, 12 and 14 warps -4 to -19 %); 1537 to 2048
//              units: 8 units a thread, 512-thread CTAs (16384 +24 %); other
//              rows of 769 to 2560 units that 5 units fill exactly: 5 units,
//              one row a CTA (10240 +13 %, 20480 +12 %);
// RMSNorm      rows of one warp at 8 units: 512-thread CTAs (+0.8 %); 4 warps at
//              4 units: one row a 128-thread CTA (4096 +6.1 %); 5 to 7 warps at
//              4 units: three stages (+3 to +8 %); 8 warps at 4 units: four
//              stages (8192 +8.3 %); 2049 to 3072 units that 6 units a thread
//              fill whole warps exactly: 6 units, one row a CTA (18432 +6.9 %,
//              21504 +9.9 %, 24576 +11.1 % against 4 units on 18 to 24 warps;
//              at 1536 to 1920 units, where 4 units take at most 15 warps, -1
//              to -25 %); other rows of 129 to 2560 units that 5 units fill on
//              whole warps and 4 units do not within 512 threads: 5 units, one
//              row a CTA, 128-thread CTAs for rows of one warp (1280 +31 %,
//              2560 +21 %, 20480 +12 %; where 4 units fill 5 or 10 warps, 5120
//              and 10240, 5 units measured 8 and 2.5 % slower).
// The rules other than the causal and the wide softmax ones apply from 64
// rows an SM, so that every CTA loops over its stages.
struct ShapeWant {
    int tpr, vpt, block, stages;
};
bool measured_ring_shape(const rs_plan& p, int64_t units, int64_t M, int sm_count, ShapeWant* w) {
    const int tpr = p.threads_per_row, vpt = p.vec_per_thread;
    const auto fills = [units](int lanes, int v) { return units % v == 0 && (units / v) % lanes == 0; };
    *w = ShapeWant{0, 0, 0, 0};
    if (p.op == RS_OP_SOFTMAX && !p.masked) {
        RingShape r{};
        if (ring16_softmax_shape(units, M, sm_count, &r)) {
            *w = ShapeWant{r.tpr, r.vpt, r.block, r.stages};
            return true;
        }
    } else if (p.op == RS_OP_SOFTMAX && causal16_ring(units, M, sm_count)) {
        const int v = fills(512, 5) ? 5 : fills(512, 6) ? 6 : fills(32, 8) ? 8 : fills(32, 5) ? 5 : fills(32, 6) ? 6 : 8;
        const int t = (int)round_up(ceil_div(units, v), 32);
        *w = ShapeWant{t, v, t, 2};
        return true;
    } else if (p.op == RS_OP_SOFTMAX) {
        int t = 0, v = 0;
        if (causal16_narrow(units, M, sm_count, &t, &v)) {
            *w = ShapeWant{t, v, 512, 2};
            return true;
        }
    }
    if (M < (int64_t)64 * sm_count) return false;
    if (p.op == RS_OP_SOFTMAX) {
        const int v16 = !p.masked && units >= 64 && units <= 128 && units % 16 == 0 ? (int)(units / 16) : 0;
        if (v16 == 4 || v16 == 5 || v16 == 6 || v16 == 8) {
            *w = ShapeWant{16, v16, v16 == 4 || v16 == 8 ? 512 : 256, 0};
            return true;
        }
        if (tpr == 32 && (vpt == 4 || vpt == 8)) {
            *w = ShapeWant{0, 0, 512, 0};
            return true;
        }
        return false;
    }
    if (p.op == RS_OP_LAYERNORM) {
        if (units >= 32 && units <= 128) {
            int t = 8;
            while (t < 32 && t * 4 < units) t <<= 1;
            *w = ShapeWant{t, (int)ceil_div(units, t), 256, 0};
            return true;
        }
        if (tpr == 32) {
            *w = ShapeWant{0, 0, 128, 0};
            return true;
        }
        if (units > 256 && units <= 768) {
            const bool e6 = fills(32, 6), e5 = fills(32, 5), e4 = fills(32, 4);
            const int v = e6 ? 6 : e5 ? 5 : 4;
            const int t = (int)round_up(ceil_div(units, v), 32);
            *w = ShapeWant{t, v, v == 5 ? (t < 128 ? 128 / t * t : t) : e6 || e4 ? t : 0, 0};
            return true;
        }
        if (units >= 1536 && units <= 3072 && fills(256, 6)) {
            *w = ShapeWant{(int)(units / 6), 6, (int)(units / 6), 0};
            return true;
        }
        if (units > 1536 && units <= 2048) {
            *w = ShapeWant{256, 8, 512, 0};
            return true;
        }
        if (units > 768 && units <= 2560 && fills(32, 5)) {
            *w = ShapeWant{(int)(units / 5), 5, (int)(units / 5), 0};
            return true;
        }
        return false;
    }
    // RMSNorm
    const bool e4 = fills(32, 4) && units / 4 <= 512;
    if (units > 2048 && units <= 3072 && fills(32, 6)) *w = ShapeWant{(int)(units / 6), 6, (int)(units / 6), 0};
    else if (units > 128 && units <= 2560 && fills(32, 5) && !e4)
        *w = ShapeWant{(int)(units / 5), 5, units == 160 ? 128 : (int)(units / 5), 0};
    else if (tpr == 32 && vpt == 8) *w = ShapeWant{0, 0, 512, 0};
    else if (tpr == 128 && vpt <= 4) *w = ShapeWant{0, 0, 128, 0};
    else if (tpr == 256 && vpt <= 4) *w = ShapeWant{0, 0, 0, 4};
    else if (tpr > 128 && tpr < 256 && vpt <= 4) *w = ShapeWant{0, 0, 0, 3};
    else return false;
    return true;
}

// RS_PATH_RING.  `nparams` parameter vectors (LayerNorm's weight and bias)
// are staged in shared memory after the stages, padded to whole units, unless
// the plan takes a held-parameter instance (vectors in registers).
int plan_ring(int dtype, int vec, int64_t M, int64_t N, int64_t units, const rs_options& o,
              const rs_device_info& dev, rs_plan* p, int nparams = 0) {
    if (vec == 1) return RS_ERR_NO_PATH;  // bulk copies need 16-byte units
    if (o.stages && (o.stages < 2 || o.stages > rs::kRingMaxStages)) return RS_ERR_INVALID_ARG;
    if (o.ring_values < RS_RING_AUTO || o.ring_values > RS_RING_THREAD_COPIES) return RS_ERR_INVALID_ARG;
    // The causal softmax on 16-bit rows copies only the kept units, thread by
    // thread (measured 1.222 against 1.320 ms on bf16 1048576 x 2048 causal
    // scores with the bulk-copied whole rows).
    const bool copies_ok = p->masked && dtype != RS_F32 && !o.withhold_copies;
    const int values = o.ring_values != RS_RING_AUTO ? o.ring_values
                       : copies_ok && (!o.stages || o.stages <= kRingCopyMaxStages) ? RS_RING_THREAD_COPIES
                                                                                      : RS_RING_REGISTERS;
    if (values == RS_RING_REREAD && (p->op != RS_OP_SOFTMAX || p->masked)) return RS_ERR_NO_PATH;
    if (values == RS_RING_THREAD_COPIES && (!copies_ok || (o.stages && o.stages > kRingCopyMaxStages)))
        return RS_ERR_NO_PATH;
    rs_options ro = o;
    ro.grid_limit = 0;
    // LayerNorm on 16-bit rows that fill 4 or 8 warps at 4 units a thread takes
    // the instance that holds the weight and bias in registers (measured 7-16 %
    // faster than 8 units a thread with the vectors staged in shared memory;
    // slower on rows of 2 warps).
    if (p->op == RS_OP_LAYERNORM && !p->masked && dtype != RS_F32 && values == RS_RING_REGISTERS &&
        !o.vec_per_thread && !o.threads_per_row && !o.block_threads && N == units * vec && units % 4 == 0 &&
        (units / 4 == 128 || units / 4 == 256))
        ro.vec_per_thread = 4;
    int rc = plan_rows(dtype, vec, M, units, ro, p, values != RS_RING_REREAD);
    if (rc != RS_OK) return rc;
    // The shapes measured for 16-bit rows (measured_ring_shape), unless the
    // caller forced one.
    int def_stages = kRingDefaultStages;
    ShapeWant want{};
    if (dtype != RS_F32 && values != RS_RING_REREAD && !o.block_threads && !o.threads_per_row &&
        !o.vec_per_thread && measured_ring_shape(*p, units, M, dev.sm_count, &want)) {
        const int tpr = p->threads_per_row, vpt = p->vec_per_thread;
        rs_options rb = ro;
        if (want.tpr) rb.threads_per_row = want.tpr;
        if (want.vpt) rb.vec_per_thread = want.vpt;
        if (want.block) rb.block_threads = want.block;
        bool ok = true;
        if ((want.block && want.block != p->block_threads) || (want.tpr && want.tpr != tpr) ||
            (want.vpt && want.vpt != vpt)) {
            const rs_plan keep = *p;
            if (plan_rows(dtype, vec, M, units, rb, p, true) != RS_OK ||
                p->threads_per_row != (want.tpr ? want.tpr : tpr) || p->vec_per_thread != (want.vpt ? want.vpt : vpt)) {
                *p = keep;
                ok = false;
            }
        }
        if (ok && want.stages) def_stages = want.stages;
    }
    p->path = RS_PATH_RING;  // (the LayerNorm kind depends on the path)
    const int lkind = p->op == RS_OP_LAYERNORM ? rs::layernorm_merge_kind(*p, N, vec) : 0;
    const bool held = lkind == 3 || lkind == 4 || (p->op == RS_OP_RMSNORM && rs::rmsnorm_ring_held(*p, vec));
    const int64_t slot = (N / vec) * 16;
    const int64_t stage = slot * p->rows_per_cta;
    if (stage <= 0) return RS_ERR_NO_PATH;
    const int64_t max_dyn = (int64_t)dev.max_smem_per_block_optin - (int64_t)rs::kRingStaticSmem;
    int stages = o.stages ? o.stages : def_stages;
    int64_t smem = stage * stages + (int64_t)(held ? 0 : nparams) * round_up(N, vec) * elem_size(dtype);
    if (!o.stages && stages > kRingDefaultStages && smem > max_dyn) {  // a measured stage count that does not fit
        stages = kRingDefaultStages;
        smem = stage * stages + (int64_t)(held ? 0 : nparams) * round_up(N, vec) * elem_size(dtype);
    }
    if (smem > max_dyn || stage >= (1 << 20)) return RS_ERR_NO_PATH;  // mbarrier tx count < 2^20
    const int regs = values == RS_RING_REREAD ? rs::kRingRereadRegs
                     : held ? rs::kHeldRegs
                            : (rs::rows_block_limit(p->vec_per_thread, vec) == 1024 ? 64 : 128);
    const int64_t groups = ceil_div(M, p->rows_per_cta);
    int64_t grid = (int64_t)dev.sm_count * ctas_per_sm(dev, p->block_threads, (size_t)smem, regs);
    if (grid > groups) grid = groups;
    if (o.grid_limit > 0 && grid > o.grid_limit) grid = o.grid_limit;
    p->path = RS_PATH_RING;
    p->ring_values = values;
    p->stages = stages;
    p->smem_bytes = (size_t)smem;
    p->grid = grid;
    return RS_OK;
}

// RS_PATH_CLUSTER with the slice in registers: a persistent grid of clusters,
// each CTA holding VPT (1, 2 or 4) 16-byte units a thread of its slice.
int plan_cluster_hold(int dtype, int vec, int64_t M, int64_t N, const rs_options& o, const rs_device_info& dev,
                      rs_plan* p) {
    const int es = elem_size(dtype);
    const int64_t max_dyn = (int64_t)dev.max_smem_per_block_optin - (int64_t)rs::kWideStaticSmem;
    if (o.stages && (o.stages < 1 || o.stages > rs::kWideHoldMaxSlots)) return RS_ERR_INVALID_ARG;
    if (o.ring_values == RS_RING_THREAD_COPIES) return RS_ERR_NO_PATH;  // the ring's only
    int cs = o.cluster_size;
    int block = 0, vpt = 0;
    int64_t chunk = 0;
    // Candidate (threads, units a thread) shapes, in order of preference among
    // equally tight fits: the softmax holds most values a thread, the
    // normalisations (more per-row instructions after the exchange) prefer more
    // threads (both measured); 8 units a thread are compiled for 256-thread
    // CTAs only.
    static const int kShapesSoftmax[][2] = {{256, 8}, {512, 4}, {256, 4}, {512, 2}, {256, 2}, {512, 1}, {256, 1}};
    static const int kShapesNorm[][2] = {{512, 4}, {256, 8}, {512, 2}, {256, 4}, {512, 1}, {256, 2}, {256, 1}};
    const auto& kShapes = p->op == RS_OP_SOFTMAX ? kShapesSoftmax : kShapesNorm;
    // Cluster size: the smallest whose slices fill a CTA shape to at least 7/8
    // (idle lanes cost as much as busy ones on a latency-bound row), else the
    // best fill; any size 1..16, not only powers of two (measured: bf16 rows of
    // 24576 at 3 CTAs fill 256 x 4 exactly).
    double best_fill = 0.0;
    int best_c = 0;
    for (int c = cs ? cs : 1; c <= (cs ? cs : rs::kMaxCluster); ++c) {
        const int64_t ch = round_up(ceil_div(N, c), vec);
        const int64_t units = ch / vec;
        int b = 0, v = 0;
        int64_t best_cap = 0;
        for (const auto& sh : kShapes) {
            if (o.block_threads && sh[0] != o.block_threads) continue;
            if (o.vec_per_thread && sh[1] != o.vec_per_thread) continue;
            const int64_t cap = (int64_t)sh[0] * sh[1];
            if (cap < units) continue;
            if (!v || cap < best_cap) {  // the tightest fit; ties keep the earlier shape
                b = sh[0];
                v = sh[1];
                best_cap = cap;
            }
        }
        if (!v) continue;
        const double fill = (double)units / (double)best_cap;
        if (fill > best_fill + 1e-9) {
            best_fill = fill;
            block = b;
            vpt = v;
            chunk = ch;
            best_c = c;
        }
        if (fill >= 0.875) break;
    }
    if (!vpt) return RS_ERR_NO_PATH;
    cs = best_c;
    const size_t slot = (size_t)round_up(chunk * es, 16);
    const int64_t resident_ctas = (int64_t)dev.sm_count * ctas_per_sm(dev, block, 2 * slot, vpt == 8 ? 128 : 64);
    int64_t clusters = resident_ctas / cs;
    if (clusters < 1) clusters = 1;
    if (clusters > M) clusters = M;
    if (o.grid_limit > 0 && clusters * cs > o.grid_limit) clusters = o.grid_limit / cs > 0 ? o.grid_limit / cs : 1;
    if (clusters * cs > kMaxGrid) clusters = kMaxGrid / cs;
    const int slots = o.stages ? o.stages : (clusters < M ? 2 : 1);
    if ((int64_t)(slots * slot) > max_dyn) return RS_ERR_NO_PATH;
    p->path = RS_PATH_CLUSTER;
    p->ring_values = RS_RING_REGISTERS;
    p->vec_elems = vec;
    p->threads_per_row = block;
    p->vec_per_thread = vpt;
    p->rows_per_cta = 1;
    p->block_threads = block;
    p->cluster_size = cs;
    p->stages = slots;
    p->chunk_elems = chunk;
    p->grid = clusters * cs;
    p->smem_bytes = slots * slot;
    return RS_OK;
}

int plan_wide(int dtype, int path, int vec, int64_t M, int64_t N, const rs_options& o,
              const rs_device_info& dev, rs_plan* p) {
    if (path == RS_PATH_CLUSTER && vec > 1 &&
        (o.ring_values == RS_RING_REGISTERS || o.ring_values == RS_RING_AUTO)) {
        const int rc = plan_cluster_hold(dtype, vec, M, N, o, dev, p);
        if (rc == RS_OK || o.ring_values == RS_RING_REGISTERS) return rc;
    }
    if (o.withhold_copies) return RS_ERR_NO_PATH;  // only the register-holding clusters implement it
    if (o.ring_values < RS_RING_AUTO || o.ring_values > RS_RING_THREAD_COPIES) return RS_ERR_INVALID_ARG;
    if (o.ring_values == RS_RING_THREAD_COPIES) return RS_ERR_NO_PATH;  // the ring's only
    const int es = elem_size(dtype);
    const int64_t max_dyn = (int64_t)dev.max_smem_per_block_optin - (int64_t)rs::kWideStaticSmem;
    int cs = o.cluster_size;
    if (cs && (cs < 1 || cs > rs::kMaxCluster)) return RS_ERR_INVALID_ARG;
    if (path == RS_PATH_CLUSTER) {
        if (vec == 1) return RS_ERR_NO_PATH;  // bulk copies need 16-byte units
        if (!cs) {
            for (int c = 1; c <= rs::kMaxCluster; c <<= 1) {
                const int64_t slice = round_up(ceil_div(N, c), vec) * es;
                if (slice <= kClusterTargetSlice || (c == rs::kMaxCluster && slice <= max_dyn)) {
                    cs = c;
                    break;
                }
                if (c == rs::kMaxCluster) break;
            }
            if (!cs) return RS_ERR_NO_PATH;
        }
    } else if (!cs) {
        // Streaming: enough CTAs to cover the machine, at most kMaxClusterPortable per row.
        cs = 1;
        while (cs < rs::kMaxClusterPortable && M * cs < 2 * (int64_t)dev.sm_count) cs <<= 1;
    }
    const int64_t chunk = round_up(ceil_div(N, cs), vec);
    if (chunk > kMaxN) return RS_ERR_NO_PATH;
    int stages = 0;
    size_t smem = 0;
    int64_t clusters = M;
    if (o.grid_limit > 0 && clusters * cs > o.grid_limit) clusters = o.grid_limit / cs > 0 ? o.grid_limit / cs : 1;
    if (clusters * cs > kMaxGrid) clusters = kMaxGrid / cs;
    if (path == RS_PATH_CLUSTER) {
        // One slot per CTA when every cluster serves one row; two (the next
        // row's slice in flight) when clusters loop over rows.
        const int slots = clusters < M ? 2 : 1;
        smem = slots * (size_t)round_up(chunk * es, 16);
        if ((int64_t)smem > max_dyn) return RS_ERR_NO_PATH;
        stages = (int)ceil_div(ceil_div(chunk, vec), rs::kWideUnitsPerStage);
        if (stages > rs::kWideMaxStages) return RS_ERR_NO_PATH;
    }

    p->path = path;
    p->ring_values = path == RS_PATH_CLUSTER ? RS_RING_REREAD : RS_RING_AUTO;
    p->vec_elems = vec;
    p->threads_per_row = 0;
    p->vec_per_thread = 0;
    p->rows_per_cta = 1;
    p->block_threads = rs::kWideThreads;
    p->cluster_size = cs;
    p->stages = stages;
    p->chunk_elems = chunk;
    p->grid = clusters * cs;
    p->smem_bytes = smem;
    return RS_OK;
}

// RS_PATH_STREAM for the normalisations: one CTA per row, a grid of a few
// CTAs per SM looping over the rows.
int plan_norm_stream(int vec, int64_t M, const rs_options& o, const rs_device_info& dev, rs_plan* p) {
    if (o.cluster_size > 1 || o.threads_per_row || o.vec_per_thread) return RS_ERR_NO_PATH;
    if (o.block_threads && o.block_threads != rs::kNormStreamThreads) return RS_ERR_NO_PATH;
    int64_t grid = (int64_t)dev.sm_count * rs::kNormStreamCtasPerSm;
    if (grid > M) grid = M;
    if (o.grid_limit > 0 && grid > o.grid_limit) grid = o.grid_limit;
    p->path = RS_PATH_STREAM;
    p->vec_elems = vec;
    p->threads_per_row = rs::kNormStreamThreads;
    p->rows_per_cta = 1;
    p->block_threads = rs::kNormStreamThreads;
    p->cluster_size = 1;
    p->grid = grid;
    return RS_OK;
}

// Byte range [lo, lo + bytes) of `q` overlaps [r, r + rbytes)?
bool ranges_overlap(uintptr_t q, uint64_t bytes, uintptr_t r, uint64_t rbytes) {
    return q < r + rbytes && r < q + bytes;
}

// mask_period > 0: the softmax under a causal mask (row r keeps its first
// min(N, max(0, (r mod mask_period) + 1 + mask_offset)) elements).
int validate_and_plan_op(int op, const void* in, const void* out, const void* w, const void* b, int64_t M,
                         int64_t N, int64_t ldi, int64_t ldo, double eps, int dtype, const rs_options* opts,
                         const rs_device_info* dev, rs_plan* p, int64_t mask_period = 0,
                         int64_t mask_offset = 0) {
    memset(p, 0, sizeof(*p));
    p->dtype = dtype;
    p->op = op;
    if (mask_period < 0 || (mask_period > 0 && op != RS_OP_SOFTMAX)) return RS_ERR_INVALID_ARG;
    if (mask_offset < -kMaxMaskOffset || mask_offset > kMaxMaskOffset) return RS_ERR_INVALID_ARG;
    const bool masked = mask_period > 0;
    p->masked = masked ? 1 : 0;
    if (op != RS_OP_SOFTMAX && op != RS_OP_RMSNORM && op != RS_OP_LAYERNORM) return RS_ERR_INVALID_ARG;
    if (dtype != RS_F32 && dtype != RS_F16 && dtype != RS_BF16) return RS_ERR_UNSUPPORTED_DTYPE;
    if (M < 0 || N < 0) return RS_ERR_INVALID_ARG;
    if (op == RS_OP_SOFTMAX && (w || b)) return RS_ERR_INVALID_ARG;
    if (op == RS_OP_RMSNORM && b) return RS_ERR_INVALID_ARG;
    // eps enters the kernels as a float: finite, >= 0, representable.
    if (op != RS_OP_SOFTMAX && !(eps >= 0.0 && eps <= (double)3.402823466e38f)) return RS_ERR_INVALID_ARG;
    rs_options o;
    memset(&o, 0, sizeof(o));
    if (opts) o = *opts;
    if (o.path < RS_PATH_AUTO || o.path > RS_PATH_RING || o.grid_limit < 0 || o.vec_per_thread < 0 ||
        o.threads_per_row < 0 || o.block_threads < 0 || o.cluster_size < 0 || o.stages < 0 ||
        o.wait_limit_us < 0 || o.withhold_copies < 0 || o.withhold_copies > 1 || o.strict_order < 0 ||
        o.strict_order > 1)
        return RS_ERR_INVALID_ARG;
    // Withholding copies is only defined for the ring and the register-holding
    // clusters, and needs a short wait limit.
    if (o.withhold_copies && ((o.path != RS_PATH_RING && o.path != RS_PATH_CLUSTER) || o.wait_limit_us <= 0 ||
                              o.wait_limit_us > 1000000))
        return RS_ERR_INVALID_ARG;
    p->wait_limit_us = o.wait_limit_us;
    p->withhold_copies = o.withhold_copies;
    p->strict_order = o.strict_order;
    if (M == 0 || N == 0) return RS_OK;  // nothing to do, nothing launched
    if (N > kMaxN) return RS_ERR_INVALID_ARG;
    if (!in || !out) return RS_ERR_INVALID_ARG;
    if (ldi < N || ldo < N) return RS_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    const uintptr_t ai = (uintptr_t)in, ao = (uintptr_t)out, aw = (uintptr_t)w, ab = (uintptr_t)b;
    if (ai % es || ao % es || aw % es || ab % es) return RS_ERR_INVALID_ARG;
    // Byte extent of each tensor: ((M-1)*ld + N) * es, checked for overflow.
    if ((M - 1) > (INT64_MAX / es - N) / ldi || (M - 1) > (INT64_MAX / es - N) / ldo)
        return RS_ERR_INVALID_ARG;
    const uint64_t ext_i = (uint64_t)(((M - 1) * ldi + N) * es);
    const uint64_t ext_o = (uint64_t)(((M - 1) * ldo + N) * es);
    const uint64_t ext_v = (uint64_t)(N * es);  // a weight or bias vector
    if (ai > UINTPTR_MAX - ext_i || ao > UINTPTR_MAX - ext_o) return RS_ERR_INVALID_ARG;
    if ((w && aw > UINTPTR_MAX - ext_v) || (b && ab > UINTPTR_MAX - ext_v)) return RS_ERR_INVALID_ARG;
    if (ranges_overlap(ai, ext_i, ao, ext_o) && !(ai == ao && ldi == ldo)) return RS_ERR_OVERLAP;
    if ((w && ranges_overlap(aw, ext_v, ao, ext_o)) || (b && ranges_overlap(ab, ext_v, ao, ext_o)))
        return RS_ERR_OVERLAP;
    if (!dev || dev->sm_count <= 0 || dev->max_smem_per_block_optin <= 0) return RS_ERR_INVALID_ARG;

    const int kvec = 16 / es;
    const bool strides_ok = M == 1 || (((ldi * es) % 16) == 0 && ((ldo * es) % 16) == 0);
    const bool vec_ok = !o.force_scalar && ai % 16 == 0 && ao % 16 == 0 && aw % 16 == 0 && ab % 16 == 0 &&
                        strides_ok;
    const int vec = vec_ok ? kvec : 1;
    const int64_t units = ceil_div(N, vec);
    const bool norm = op != RS_OP_SOFTMAX;
    // Parameter vectors the ring kernel stages in shared memory (LayerNorm's).
    const int nparams = op == RS_OP_LAYERNORM ? (w ? 1 : 0) + (b ? 1 : 0) : 0;

    int path = o.path;
    if (path == RS_PATH_AUTO) {
        int rc = RS_ERR_NO_PATH;
        // 16-bit rows: the ring (bytes in flight in shared memory, not in
        // registers); fp32 rows: the register kernel, whose fp32 values cost
        // no more registers than the bytes they came from.  The normalisations
        // take the ring wherever its stages fit (measured 5-185 % faster than
        // the clusters on rows of 32-64 KB); the softmax below 32 KB, and up to
        // 64 KB where the cluster plan would spread a row thin (at most
        // kClusterThinValues values a thread: 3278 -> 5327 GB/s on 40 KB rows;
        // with fuller cluster shapes the clusters measured as fast or faster).
        RingShape shape16{};
        bool ring = dtype != RS_F32 && vec_ok && N * es >= kRingMinRowBytes &&
                    (norm || N * es < kRowsMaxRowBytes ||
                     (!masked && ring16_softmax_shape(units, M, dev->sm_count, &shape16)) ||
                     (masked && causal16_ring(units, M, dev->sm_count)));
        if (!ring && !norm && dtype != RS_F32 && vec_ok && N * es < kRingMaxRowBytesSoftmax16) {
            rs_plan cp = *p;
            ring = plan_wide(dtype, RS_PATH_CLUSTER, vec, M, N, o, *dev, &cp) != RS_OK ||
                   cp.vec_per_thread * cp.vec_elems <= kClusterThinValues;
        }
        // LayerNorm on fp32 rows that would take two reductions on the register
        // rows (ragged, or not a power-of-two number of warps) and span 4 to 8
        // warps at 8 units a thread: the ring, whose CTAs hold the weight and
        // bias in registers across their rows, where at least kLnHeldMinWarpsF32
        // warps fit an SM (measured +8.6 to +10 % on 4100-, 5000- and 7000-value
        // rows; 6000-value rows, 192-thread CTAs of which 2 fit an SM, -8.7 %;
        // rows that fill their warps, and rows of 2 warps, faster on the register
        // rows).
        rs_options ro = o;
        if (op == RS_OP_LAYERNORM && dtype == RS_F32 && vec_ok && !o.vec_per_thread && !o.threads_per_row &&
            !o.block_threads) {
            const int64_t t8 = round_up(ceil_div(units, 8), 32);
            const int64_t w8 = t8 / 32;
            const bool filled = N == t8 * 32 && (w8 & (w8 - 1)) == 0;
            const int64_t warps_per_sm = (65536 / (t8 * rs::kHeldRegs)) * w8;
            if (t8 >= kLnHeldMinThreadsF32 && t8 <= rs::kHeldThreads && !filled &&
                warps_per_sm >= kLnHeldMinWarpsF32) {
                ring = true;
                ro.vec_per_thread = 8;
            }
        }
        if (ring) rc = plan_ring(dtype, vec, M, N, units, ro, *dev, p, nparams);
        if (rc == RS_OK) return RS_OK;
        if (rc != RS_ERR_NO_PATH) return rc;
        const int64_t rows_max = dtype == RS_F32 && !norm ? kRowsMaxRowBytesF32
                                 : dtype != RS_F32 && !norm && vec_ok ? kRowsMaxRowBytes - 1
                                                                      : kRowsMaxRowBytes;
        if (N * es <= rows_max) rc = plan_rows(dtype, vec, M, units, o, p, true, dev->sm_count);
        if (rc == RS_OK) return RS_OK;
        if (rc != RS_ERR_NO_PATH) return rc;
        if (norm || masked) {
            if (vec_ok) {
                rc = plan_cluster_hold(dtype, vec, M, N, o, *dev, p);
                if (rc == RS_OK) return RS_OK;
                if (rc != RS_ERR_NO_PATH) return rc;
            }
            // The causal mask is served by the register rows, the ring and the
            // register-holding clusters only.
            return norm ? plan_norm_stream(vec, M, o, *dev, p) : RS_ERR_NO_PATH;
        }
        if (vec_ok) {
            rc = plan_wide(dtype, RS_PATH_CLUSTER, vec, M, N, o, *dev, p);
            if (rc == RS_OK) return RS_OK;
            if (rc != RS_ERR_NO_PATH) return rc;
        }
        return plan_wide(dtype, RS_PATH_STREAM, vec, M, N, o, *dev, p);
    }
    if (path == RS_PATH_ROWS) return plan_rows(dtype, vec, M, units, o, p, true, dev->sm_count);
    if (path == RS_PATH_RING) return plan_ring(dtype, vec, M, N, units, o, *dev, p, nparams);
    if (norm || masked) {
        if (path == RS_PATH_STREAM) return norm ? plan_norm_stream(vec, M, o, *dev, p) : RS_ERR_NO_PATH;
        // Clusters serve the normalisations and the causal mask with the slice in
        // registers only.
        if (vec == 1 || o.ring_values == RS_RING_REREAD || o.ring_values == RS_RING_THREAD_COPIES)
            return RS_ERR_NO_PATH;
        return plan_cluster_hold(dtype, vec, M, N, o, *dev, p);
    }
    return plan_wide(dtype, path, vec, M, N, o, *dev, p);
}

int validate_and_plan(const void* in, const void* out, int64_t M, int64_t N, int64_t ldi, int64_t ldo,
                      int dtype, const rs_options* opts, const rs_device_info* dev, rs_plan* p) {
    return validate_and_plan_op(RS_OP_SOFTMAX, in, out, nullptr, nullptr, M, N, ldi, ldo, 0.0, dtype, opts, dev,
                                p);
}

std::mutex g_dev_mu;
bool g_dev_known[64];
rs_device_info g_dev[64];

int query_device(int dev, rs_device_info* info) {
    memset(info, 0, sizeof(*info));
    cudaError_t e;
    if ((e = cudaDeviceGetAttribute(&info->sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&info->max_smem_per_block_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                    dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&info->max_smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&info->max_threads_per_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev)) !=
            cudaSuccess ||
        (e = cudaDeviceGetAttribute(&info->cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&info->cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess) {
        (void)cudaGetLastError();
        return fail_cuda(e);
    }
    return RS_OK;
}

int current_device(int* dev, rs_device_info* info) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail_cuda(e);
    }
    if (*dev < 0 || *dev >= 64) return fail_cuda(cudaErrorInvalidDevice);
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_dev_known[*dev]) {
        int rc = query_device(*dev, &g_dev[*dev]);
        if (rc != RS_OK) return rc;
        g_dev_known[*dev] = true;
    }
    *info = g_dev[*dev];
    return RS_OK;
}

// cudaOccupancyMaxActiveClusters for a planned cluster launch, cached by
// device and launch shape (the query costs far more than a launch).
struct ClusterKey {
    int dev, op, masked, dtype, path, values, vec, vpt, block, cs;
    size_t smem;
    bool operator==(const ClusterKey& o) const {
        return dev == o.dev && op == o.op && masked == o.masked && dtype == o.dtype && path == o.path &&
               values == o.values &&
               vec == o.vec && vpt == o.vpt && block == o.block && cs == o.cs && smem == o.smem;
    }
};
std::mutex g_cluster_mu;
ClusterKey g_cluster_keys[64];
int g_cluster_vals[64];
int g_cluster_n = 0;

cudaError_t max_active_clusters_cached(int dev, const rs_plan& p, int* n) {
    const ClusterKey k{dev, p.op, p.masked, p.dtype, p.path, p.ring_values, p.vec_elems, p.vec_per_thread,
                       p.block_threads, p.cluster_size, p.smem_bytes};
    {
        std::lock_guard<std::mutex> lock(g_cluster_mu);
        for (int i = 0; i < g_cluster_n; ++i)
            if (g_cluster_keys[i] == k) {
                *n = g_cluster_vals[i];
                return cudaSuccess;
            }
    }
    cudaError_t e;
    if (p.op == RS_OP_SOFTMAX && p.masked) {
        e = p.dtype == RS_F32 ? rs::causal_max_clusters_f32(p, n)
            : p.dtype == RS_F16 ? rs::causal_max_clusters_f16(p, n) : rs::causal_max_clusters_bf16(p, n);
    } else if (p.op == RS_OP_SOFTMAX) e = rs::wide_max_active_clusters(p, n);
    else if (p.dtype == RS_F32) e = rs::norm_max_clusters_f32(p, n);
    else if (p.dtype == RS_F16) e = rs::norm_max_clusters_f16(p, n);
    else e = rs::norm_max_clusters_bf16(p, n);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(g_cluster_mu);
    const int slot = g_cluster_n < 64 ? g_cluster_n++ : (int)(k.smem % 64);
    g_cluster_keys[slot] = k;
    g_cluster_vals[slot] = *n;
    return cudaSuccess;
}

// The kernels dereference `p` directly: it must be memory the current
// device can address at that same address.
int check_device_pointer(const void* p, int dev) {
    cudaPointerAttributes a;
    cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return RS_ERR_NOT_DEVICE_MEMORY;
    }
    switch (a.type) {
        case cudaMemoryTypeDevice:
            return a.device == dev ? RS_OK : RS_ERR_NOT_DEVICE_MEMORY;
        case cudaMemoryTypeManaged:
            return RS_OK;
        case cudaMemoryTypeHost:
            return a.devicePointer != nullptr && (uintptr_t)a.devicePointer == (uintptr_t)p
                       ? RS_OK
                       : RS_ERR_NOT_DEVICE_MEMORY;
        default:
            return RS_ERR_NOT_DEVICE_MEMORY;
    }
}

}  // namespace

extern "C" {

int rowsoftmax_plan(const void* in, const void* out, int64_t M, int64_t N, int64_t in_row_stride,
                    int64_t out_row_stride, int dtype, const rs_options* opts, const rs_device_info* dev,
                    rs_plan* plan) {
    if (!plan) return RS_ERR_INVALID_ARG;
    return validate_and_plan(in, out, M, N, in_row_stride, out_row_stride, dtype, opts, dev, plan);
}

int rownorm_plan(int op, const void* in, const void* out, const void* weight, const void* bias, int64_t M,
                 int64_t N, int64_t in_row_stride, int64_t out_row_stride, double eps, int dtype,
                 const rs_options* opts, const rs_device_info* dev, rs_plan* plan) {
    if (!plan) return RS_ERR_INVALID_ARG;
    if (op != RS_OP_RMSNORM && op != RS_OP_LAYERNORM) {
        memset(plan, 0, sizeof(*plan));
        return RS_ERR_INVALID_ARG;
    }
    return validate_and_plan_op(op, in, out, weight, bias, M, N, in_row_stride, out_row_stride, eps, dtype, opts,
                                dev, plan);
}

}  // extern "C"

namespace {

// Validate, plan on the current device and launch one row operation.
int run_op(int op, const void* in, void* out, const void* w, const void* b, int64_t M, int64_t N, int64_t ldi,
           int64_t ldo, double eps, int dtype, cudaStream_t stream, const rs_options* opts,
           int64_t mask_period = 0, int64_t mask_offset = 0) {
    // Shape and argument errors first: they need no device.
    rs_device_info probe;
    memset(&probe, 0, sizeof(probe));
    probe.sm_count = 1;
    probe.max_smem_per_block_optin = 1;
    rs_plan plan;
    int rc = validate_and_plan_op(op, in, out, w, b, M, N, ldi, ldo, eps, dtype, nullptr, &probe, &plan, mask_period,
                                  mask_offset);
    if (rc != RS_OK && rc != RS_ERR_NO_PATH) return rc;
    if (M == 0 || N == 0) return RS_OK;

    int dev = 0;
    rs_device_info info;
    rc = current_device(&dev, &info);
    if (rc != RS_OK) return rc;
    if ((rc = check_device_pointer(in, dev)) != RS_OK) return rc;
    if ((rc = check_device_pointer(out, dev)) != RS_OK) return rc;
    if (w && (rc = check_device_pointer(w, dev)) != RS_OK) return rc;
    if (b && (rc = check_device_pointer(b, dev)) != RS_OK) return rc;
    rc = validate_and_plan_op(op, in, out, w, b, M, N, ldi, ldo, eps, dtype, opts, &info, &plan, mask_period,
                              mask_offset);
    if (rc != RS_OK) return rc;

    const bool persistent_cluster = plan.path == RS_PATH_CLUSTER && plan.ring_values == RS_RING_REGISTERS;
    if ((op == RS_OP_SOFTMAX || plan.path == RS_PATH_CLUSTER) &&
        (plan.path == RS_PATH_CLUSTER || plan.path == RS_PATH_STREAM) &&
        (plan.cluster_size > rs::kMaxClusterPortable || persistent_cluster)) {
        int n = 0;
        cudaError_t e = max_active_clusters_cached(dev, plan, &n);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return fail_cuda(e);
        }
        if (n < 1) return RS_ERR_NO_PATH;
        // A persistent grid larger than what is co-resident would leave its
        // last clusters to run after the others, each with many rows.
        if (persistent_cluster && plan.grid / plan.cluster_size > n) plan.grid = (int64_t)n * plan.cluster_size;
    }

    cudaError_t e = cudaSuccess;
    const int n = (int)N;
    if (op != RS_OP_SOFTMAX) {
        const rs::RowArgs a{w, b, (float)eps, 0, 0, 0};
        switch (dtype) {
            case RS_F32: e = rs::launch_norm_f32(plan, in, out, M, n, ldi, ldo, stream, a); break;
            case RS_F16: e = rs::launch_norm_f16(plan, in, out, M, n, ldi, ldo, stream, a); break;
            default: e = rs::launch_norm_bf16(plan, in, out, M, n, ldi, ldo, stream, a); break;
        }
    } else if (mask_period > 0) {
        const rs::RowArgs a{nullptr, nullptr, 0.0f, mask_period, mask_offset,
                            rs::remainder_magic((uint64_t)mask_period)};
        switch (dtype) {
            case RS_F32: e = rs::launch_causal_f32(plan, in, out, M, n, ldi, ldo, stream, a); break;
            case RS_F16: e = rs::launch_causal_f16(plan, in, out, M, n, ldi, ldo, stream, a); break;
            default: e = rs::launch_causal_bf16(plan, in, out, M, n, ldi, ldo, stream, a); break;
        }
    } else {
        const rs::RowArgs a{nullptr, nullptr, 0.0f, 0, 0, 0};
        if (plan.path == RS_PATH_ROWS) {
            switch (dtype) {
                case RS_F32: e = rs::launch_rows_f32(plan, in, out, M, n, ldi, ldo, stream, a); break;
                case RS_F16: e = rs::launch_rows_f16(plan, in, out, M, n, ldi, ldo, stream, a); break;
                default: e = rs::launch_rows_bf16(plan, in, out, M, n, ldi, ldo, stream, a); break;
            }
        } else if (plan.path == RS_PATH_RING) {
            switch (dtype) {
                case RS_F32: e = rs::launch_ring_f32(plan, in, out, M, n, ldi, ldo, stream, a); break;
                case RS_F16: e = rs::launch_ring_f16(plan, in, out, M, n, ldi, ldo, stream, a); break;
                default: e = rs::launch_ring_bf16(plan, in, out, M, n, ldi, ldo, stream, a); break;
            }
        } else {
            e = rs::launch_wide(plan, in, out, M, n, ldi, ldo, stream, a);
        }
    }
    if (e != cudaSuccess) return fail_cuda(e);
    return RS_OK;
}

}  // namespace

extern "C" {

int rowsoftmax_fwd_ex(const void* in, void* out, int64_t M, int64_t N, int64_t in_row_stride,
                      int64_t out_row_stride, int dtype, cudaStream_t stream, const rs_options* opts) {
    return run_op(RS_OP_SOFTMAX, in, out, nullptr, nullptr, M, N, in_row_stride, out_row_stride, 0.0, dtype,
                  stream, opts);
}

int rowsoftmax_causal_fwd_ex(const void* in, void* out, int64_t M, int64_t N, int64_t in_row_stride,
                             int64_t out_row_stride, int64_t period, int64_t diag_offset, int dtype,
                             cudaStream_t stream, const rs_options* opts) {
    if (period < 1) return RS_ERR_INVALID_ARG;
    return run_op(RS_OP_SOFTMAX, in, out, nullptr, nullptr, M, N, in_row_stride, out_row_stride, 0.0, dtype, stream,
                  opts, period, diag_offset);
}

int rowsoftmax_causal_fwd(const void* in, void* out, int64_t M, int64_t N, int64_t in_row_stride,
                          int64_t out_row_stride, int64_t period, int64_t diag_offset, int dtype,
                          cudaStream_t stream) {
    return rowsoftmax_causal_fwd_ex(in, out, M, N, in_row_stride, out_row_stride, period, diag_offset, dtype,
                                    stream, nullptr);
}

int rowsoftmax_causal_plan(const void* in, const void* out, int64_t M, int64_t N, int64_t in_row_stride,
                           int64_t out_row_stride, int64_t period, int64_t diag_offset, int dtype,
                           const rs_options* opts, const rs_device_info* dev, rs_plan* plan) {
    if (!plan) return RS_ERR_INVALID_ARG;
    if (period < 1) {
        memset(plan, 0, sizeof(*plan));
        return RS_ERR_INVALID_ARG;
    }
    return validate_and_plan_op(RS_OP_SOFTMAX, in, out, nullptr, nullptr, M, N, in_row_stride, out_row_stride, 0.0,
                                dtype, opts, dev, plan, period, diag_offset);
}

int rownorm_fwd_ex(int op, const void* in, void* out, const void* weight, const void* bias, int64_t M,
                   int64_t N, int64_t in_row_stride, int64_t out_row_stride, double eps, int dtype,
                   cudaStream_t stream, const rs_options* opts) {
    if (op != RS_OP_RMSNORM && op != RS_OP_LAYERNORM) return RS_ERR_INVALID_ARG;
    return run_op(op, in, out, weight, bias, M, N, in_row_stride, out_row_stride, eps, dtype, stream, opts);
}

int rmsnorm_fwd(const void* in, void* out, const void* weight, int64_t M, int64_t N, int64_t in_row_stride,
                int64_t out_row_stride, double eps, int dtype, cudaStream_t stream) {
    return rownorm_fwd_ex(RS_OP_RMSNORM, in, out, weight, nullptr, M, N, in_row_stride, out_row_stride, eps,
                          dtype, stream, nullptr);
}

int layernorm_fwd(const void* in, void* out, const void* weight, const void* bias, int64_t M, int64_t N,
                  int64_t in_row_stride, int64_t out_row_stride, double eps, int dtype, cudaStream_t stream) {
    return rownorm_fwd_ex(RS_OP_LAYERNORM, in, out, weight, bias, M, N, in_row_stride, out_row_stride, eps,
                          dtype, stream, nullptr);
}

int rowsoftmax_fwd(const void* in, void* out, int64_t M, int64_t N, int64_t in_row_stride,
                   int64_t out_row_stride, int dtype, cudaStream_t stream) {
    return rowsoftmax_fwd_ex(in, out, M, N, in_row_stride, out_row_stride, dtype, stream, nullptr);
}

int rowsoftmax_device_info(rs_device_info* dev) {
    if (!dev) return RS_ERR_INVALID_ARG;
    int d = 0;
    return current_device(&d, dev);
}

const char* rowsoftmax_status_string(int status) {
    switch (status) {
        case RS_OK: return "ok";
        case RS_ERR_INVALID_ARG: return "invalid argument";
        case RS_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case RS_ERR_OVERLAP: return "input and output overlap (only exact in-place is allowed)";
        case RS_ERR_CUDA: return "CUDA error";
        case RS_ERR_NOT_DEVICE_MEMORY: return "pointer is not addressable by the current device";
        case RS_ERR_NO_PATH: return "no kernel configuration serves this shape with these options";
        default: return "unknown status";
    }
}

int rowsoftmax_last_cuda_error(void) {
    const int e = t_last_cuda_error;
    t_last_cuda_error = 0;
    return e;
}

int rowsoftmax_device_status(unsigned int* flags, int clear) {
    if (!flags) return RS_ERR_INVALID_ARG;
    *flags = 0;
    cudaError_t e = rs::read_status_wide(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_f32(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_f16(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_bf16(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_norm_f32(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_norm_f16(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_norm_bf16(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_causal_f32(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_causal_f16(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_causal_bf16(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_lnmerge_f32(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_lnmerge_f16(flags, clear != 0);
    if (e == cudaSuccess) e = rs::read_status_lnmerge_bf16(flags, clear != 0);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail_cuda(e);
    }
    return RS_OK;
}

int rowsoftmax_layout_owner(int64_t j, int threads, int vec, int* thread, int64_t* slot) {
    if (j < 0 || threads < 1 || vec < 1 || !thread || !slot) return RS_ERR_INVALID_ARG;
    *thread = (int)((j / vec) % threads);
    *slot = (j / ((int64_t)threads * vec)) * vec + j % vec;
    return RS_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// The softmax of rows split by columns: partial pairs, their merge, the finish,
// and the one-device split of few wide rows (kernels in rs_split.cu).
// ---------------------------------------------------------------------------
namespace {

constexpr int64_t kSplitTargetItems = 4096;     // (row, block) items a split call aims for
constexpr int64_t kSplitMinBlockUnits = 2048;   // 16-byte units of the narrowest block (32 KB)
constexpr int64_t kPairBytes = 8;               // one float2 {m, l}

// Row-major tensor of M rows x N elements of size es at `p`, row stride ld:
// pointer, alignment and extent checks; *ext = its byte extent.
int check_tensor(const void* p, int64_t M, int64_t N, int64_t ld, int es, uint64_t* ext) {
    *ext = 0;
    if (M == 0 || N == 0) return RS_OK;
    if (!p) return RS_ERR_INVALID_ARG;
    if ((uintptr_t)p % es) return RS_ERR_INVALID_ARG;
    if (ld < N) return RS_ERR_INVALID_ARG;
    if ((M - 1) > (INT64_MAX / es - N) / ld) return RS_ERR_INVALID_ARG;
    *ext = (uint64_t)(((M - 1) * ld + N) * es);
    if ((uintptr_t)p > UINTPTR_MAX - *ext) return RS_ERR_INVALID_ARG;
    return RS_OK;
}

// n float2 pairs at p: non-null, 8-byte aligned, no address overflow.
int check_pairs(const void* p, int64_t n, uint64_t* ext) {
    *ext = 0;
    if (n == 0) return RS_OK;
    if (!p || (uintptr_t)p % kPairBytes) return RS_ERR_INVALID_ARG;
    if (n > INT64_MAX / kPairBytes) return RS_ERR_INVALID_ARG;
    *ext = (uint64_t)(n * kPairBytes);
    if ((uintptr_t)p > UINTPTR_MAX - *ext) return RS_ERR_INVALID_ARG;
    return RS_OK;
}

int split_vec(const void* in, const void* out, int64_t M, int64_t ldi, int64_t ldo, int dtype) {
    const int es = elem_size(dtype);
    const bool strides = M == 1 || ((ldi * es) % 16 == 0 && (ldo * es) % 16 == 0);
    return (uintptr_t)in % 16 == 0 && (uintptr_t)out % 16 == 0 && strides ? 16 / es : 1;
}

// Blocks per row (S) and their width (B) of a one-device split: about
// kSplitTargetItems items, blocks of at least kSplitMinBlockUnits units,
// widths a whole number of 16-byte units.
void split_shape(int64_t M, int64_t N, int dtype, int64_t* S, int64_t* B) {
    const int64_t kvec = 16 / elem_size(dtype);
    const int64_t units = ceil_div(N, kvec);
    int64_t s = ceil_div(kSplitTargetItems, M);
    const int64_t smax = ceil_div(units, kSplitMinBlockUnits);
    if (s > smax) s = smax;
    if (s < 1) s = 1;
    const int64_t b = round_up(ceil_div(N, s), kvec);
    *B = b;
    *S = ceil_div(N, b);
}

// Current device, its facts, and device-pointer checks of the non-null pointers.
int split_device(rs::SplitLaunch* L, std::initializer_list<const void*> ptrs) {
    int dev = 0;
    rs_device_info info;
    int rc = current_device(&dev, &info);
    if (rc != RS_OK) return rc;
    for (const void* p : ptrs)
        if (p && (rc = check_device_pointer(p, dev)) != RS_OK) return rc;
    L->sm_count = info.sm_count;
    L->strict = false;
    return RS_OK;
}

}  // namespace

extern "C" {

int rowsoftmax_partial_fwd(const void* in, void* ml, int64_t M, int64_t N, int64_t in_row_stride, int dtype,
                           cudaStream_t stream) {
    if (dtype != RS_F32 && dtype != RS_F16 && dtype != RS_BF16) return RS_ERR_UNSUPPORTED_DTYPE;
    if (M < 0 || N < 0 || N > kMaxN) return RS_ERR_INVALID_ARG;
    if (M == 0) return RS_OK;
    const int es = elem_size(dtype);
    uint64_t ext_i = 0, ext_p = 0;
    int rc = check_tensor(in, M, N, in_row_stride, es, &ext_i);
    if (rc != RS_OK) return rc;
    if ((rc = check_pairs(ml, M, &ext_p)) != RS_OK) return rc;
    if (N > 0 && ranges_overlap((uintptr_t)in, ext_i, (uintptr_t)ml, ext_p)) return RS_ERR_OVERLAP;
    rs::SplitLaunch L;
    if ((rc = split_device(&L, {N > 0 ? in : nullptr, ml})) != RS_OK) return rc;
    const int64_t ldi = N > 0 ? in_row_stride : 0;
    L.vec = N > 0 ? split_vec(in, in, M, ldi, ldi, dtype) : 1;
    const cudaError_t e =
        rs::launch_split_partial(L, dtype, in, static_cast<float2*>(ml), M, (int)N, ldi, 1, (int)N, stream);
    return e == cudaSuccess ? RS_OK : fail_cuda(e);
}

int rowsoftmax_merge_ml(const void* ml_in, void* ml_out, int64_t R, int64_t M, cudaStream_t stream) {
    if (R < 0 || M < 0) return RS_ERR_INVALID_ARG;
    if (M == 0) return RS_OK;
    if (R > 0 && M > INT64_MAX / R) return RS_ERR_INVALID_ARG;
    uint64_t ext_in = 0, ext_out = 0;
    int rc = check_pairs(ml_in, R * M, &ext_in);
    if (rc != RS_OK) return rc;
    if ((rc = check_pairs(ml_out, M, &ext_out)) != RS_OK) return rc;
    if (R > 0 && ranges_overlap((uintptr_t)ml_in, ext_in, (uintptr_t)ml_out, ext_out)) return RS_ERR_OVERLAP;
    rs::SplitLaunch L;
    if ((rc = split_device(&L, {R > 0 ? ml_in : nullptr, ml_out})) != RS_OK) return rc;
    L.vec = 1;
    const cudaError_t e = rs::launch_split_merge(L, static_cast<const float2*>(ml_in), static_cast<float2*>(ml_out),
                                                 R, 1, M, M, stream);
    return e == cudaSuccess ? RS_OK : fail_cuda(e);
}

int rowsoftmax_finish_fwd(const void* in, void* out, const void* ml, int64_t R, int64_t M, int64_t N,
                          int64_t in_row_stride, int64_t out_row_stride, int dtype, cudaStream_t stream) {
    if (dtype != RS_F32 && dtype != RS_F16 && dtype != RS_BF16) return RS_ERR_UNSUPPORTED_DTYPE;
    if (M < 0 || N < 0 || R < 1 || N > kMaxN) return RS_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return RS_OK;
    if (M > INT64_MAX / R) return RS_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    uint64_t ext_i = 0, ext_o = 0, ext_p = 0;
    int rc = check_tensor(in, M, N, in_row_stride, es, &ext_i);
    if (rc != RS_OK) return rc;
    if ((rc = check_tensor(out, M, N, out_row_stride, es, &ext_o)) != RS_OK) return rc;
    if ((rc = check_pairs(ml, R * M, &ext_p)) != RS_OK) return rc;
    if (ranges_overlap((uintptr_t)in, ext_i, (uintptr_t)out, ext_o) &&
        !(in == out && in_row_stride == out_row_stride))
        return RS_ERR_OVERLAP;
    if (ranges_overlap((uintptr_t)ml, ext_p, (uintptr_t)out, ext_o)) return RS_ERR_OVERLAP;
    rs::SplitLaunch L;
    if ((rc = split_device(&L, {in, out, ml})) != RS_OK) return rc;
    L.vec = split_vec(in, out, M, in_row_stride, out_row_stride, dtype);
    const cudaError_t e = rs::launch_split_finish(L, dtype, in, out, static_cast<const float2*>(ml), R, 1, M, M,
                                                  (int)N, in_row_stride, out_row_stride, stream);
    return e == cudaSuccess ? RS_OK : fail_cuda(e);
}

int rowsoftmax_split_workspace_size(int64_t M, int64_t N, int dtype, size_t* bytes) {
    if (!bytes) return RS_ERR_INVALID_ARG;
    *bytes = 0;
    if (dtype != RS_F32 && dtype != RS_F16 && dtype != RS_BF16) return RS_ERR_UNSUPPORTED_DTYPE;
    if (M < 0 || N < 0 || N > kMaxN) return RS_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return RS_OK;
    int64_t S = 0, B = 0;
    split_shape(M, N, dtype, &S, &B);
    if (M > (INT64_MAX / kPairBytes) / (S + 1)) return RS_ERR_INVALID_ARG;
    *bytes = (size_t)(M * (S + 1) * kPairBytes);
    return RS_OK;
}

int rowsoftmax_split_fwd(const void* in, void* out, int64_t M, int64_t N, int64_t in_row_stride,
                         int64_t out_row_stride, int dtype, void* workspace, size_t workspace_bytes,
                         cudaStream_t stream) {
    size_t need = 0;
    int rc = rowsoftmax_split_workspace_size(M, N, dtype, &need);
    if (rc != RS_OK) return rc;
    if (M == 0 || N == 0) return RS_OK;
    const int es = elem_size(dtype);
    uint64_t ext_i = 0, ext_o = 0, ext_w = 0;
    if ((rc = check_tensor(in, M, N, in_row_stride, es, &ext_i)) != RS_OK) return rc;
    if ((rc = check_tensor(out, M, N, out_row_stride, es, &ext_o)) != RS_OK) return rc;
    if (workspace_bytes < need) return RS_ERR_INVALID_ARG;
    if ((rc = check_pairs(workspace, (int64_t)(need / kPairBytes), &ext_w)) != RS_OK) return rc;
    if (ranges_overlap((uintptr_t)in, ext_i, (uintptr_t)out, ext_o) &&
        !(in == out && in_row_stride == out_row_stride))
        return RS_ERR_OVERLAP;
    if (ranges_overlap((uintptr_t)workspace, ext_w, (uintptr_t)in, ext_i) ||
        ranges_overlap((uintptr_t)workspace, ext_w, (uintptr_t)out, ext_o))
        return RS_ERR_OVERLAP;
    rs::SplitLaunch L;
    if ((rc = split_device(&L, {in, out, workspace})) != RS_OK) return rc;
    int64_t S = 0, B = 0;
    split_shape(M, N, dtype, &S, &B);
    L.vec = split_vec(in, out, M, in_row_stride, out_row_stride, dtype);
    float2* parts = static_cast<float2*>(workspace);  // M x S pairs, row-major
    float2* merged = parts + M * S;                   // M pairs
    cudaError_t e = rs::launch_split_partial(L, dtype, in, parts, M, (int)N, in_row_stride, (int)S, (int)B, stream);
    // Up to 32 pairs a row are merged by each finishing warp itself; more are
    // merged once per row first.
    if (e == cudaSuccess && S > 32) e = rs::launch_split_merge(L, parts, merged, S, S, 1, M, stream);
    if (e == cudaSuccess) {
        e = S > 32 ? rs::launch_split_finish(L, dtype, in, out, merged, 1, 1, 0, M, (int)N, in_row_stride,
                                             out_row_stride, stream)
                   : rs::launch_split_finish(L, dtype, in, out, parts, S, S, 1, M, (int)N, in_row_stride,
                                             out_row_stride, stream);
    }
    return e == cudaSuccess ? RS_OK : fail_cuda(e);
}

}  // extern "C"

extern "C" {

// rowsoftmax_split_fwd with its workspace in the library's fixed device
// buffer instead of the caller's (see the header for who needs this).
int rowsoftmax_split_fwd_noalloc(const void* in, void* out, int64_t M, int64_t N, int64_t in_row_stride,
                                 int64_t out_row_stride, int dtype, cudaStream_t stream) {
    size_t need = 0;
    int rc = rowsoftmax_split_workspace_size(M, N, dtype, &need);
    if (rc != RS_OK) return rc;
    if (M == 0 || N == 0) return RS_OK;
    if (need > (size_t)RS_SPLIT_NOALLOC_MAX_BYTES) return RS_ERR_INVALID_ARG;
    void* scratch = nullptr;
    const cudaError_t e = rs::split_noalloc_scratch(&scratch);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return fail_cuda(e);
    }
    return rowsoftmax_split_fwd(in, out, M, N, in_row_stride, out_row_stride, dtype, scratch,
                                (size_t)RS_SPLIT_NOALLOC_MAX_BYTES, stream);
}

}  // extern "C"
