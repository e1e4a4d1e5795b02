/*
 * rowsoftmax -- fused row-wise softmax for NVIDIA GB300 (sm_103a), C ABI.
 *
 * The operation is the fused row softmax of "stanleyjacob.dev: Triton",
 * Part II, "Worked example: fused softmax": for every row r of a row-major
 * 2-D tensor, load the row once, find its max m_r, and write
 *
 *     y[r][j] = exp(x[r][j] - m_r) / sum_k exp(x[r][k] - m_r),   0 <= j < N,
 *
 * once.  Arithmetic is fp32 whatever the storage type (the "fp32
 * Accumulation" rule of the Hugging Face "triton-kernels" skill page,
 * "Numerics"); the output is rounded to the storage type with
 * round-to-nearest-even.  Rows longer than one thread block can hold are
 * split over a thread-block cluster and combined with the online
 * normaliser of Milakov and Gimelshein (mohakchugh.is-a.dev "Triton: Block-
 * Level GPU Programming Without CUDA", "How Flash Attention Uses Triton"):
 * partial pairs (m, l) merge as m = max(m1, m2),
 * l = l1 * exp(m1 - m) + l2 * exp(m2 - m).
 *
 * Data model (the Triton tutorial's kernel arguments in_row_stride,
 * out_row_stride and n_cols, taken from x.stride(0)):
 *  - `in` and `out` are DEVICE pointers (memory the current CUDA device can
 *    address: cudaMalloc, managed, or mapped pinned host memory), owned by the
 *    caller, who keeps them alive until the work on `stream` is done;
 *  - element (r, j) is at base + r * row_stride + j, in elements; the column
 *    stride is 1; row strides are >= N; padding columns are never read or
 *    written;
 *  - `in` and `out` have the same storage type `dtype` (rs_dtype);
 *  - in == out with equal strides (exact in-place) is allowed; any other
 *    overlap of the two address ranges is rejected with RS_ERR_OVERLAP;
 *  - pointers only need the alignment of one element; 16-byte aligned
 *    pointers and strides unlock 16-byte vector accesses, anything else is
 *    served by an element-wise kernel (no error).
 *
 * Special values follow the formula under IEEE rules: -inf entries give 0,
 * a row that is all -inf gives NaN, a NaN or +inf anywhere in a row gives a
 * NaN row.
 *
 * Execution: every call is asynchronous on `stream` (0 = legacy default
 * stream), allocates no device memory, and never synchronises.  Errors in
 * the arguments are reported before anything is launched.  Calls are safe
 * from several host threads.  The kernels that are not cluster launches
 * (RS_PATH_ROWS, RS_PATH_RING, and RS_PATH_STREAM of the normalisations) use
 * programmatic dependent launch: such a kernel may be scheduled and set up
 * while the previous kernel of the stream finishes, but reads and writes no
 * global memory before that kernel has completed, so stream order is kept;
 * back-to-back calls overlap their launch latency.  rs_options.strict_order
 * turns this off.
 */
#ifndef ROWSOFTMAX_H
#define ROWSOFTMAX_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define RS_API __attribute__((visibility("default")))
#else
#define RS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Storage types.  Input and output share one. */
typedef enum { RS_F32 = 0, RS_F16 = 1, RS_BF16 = 2 } rs_dtype;

/* Return codes of every entry point. */
typedef enum {
    RS_OK = 0,
    RS_ERR_INVALID_ARG = 1,        /* negative size, stride < N, null or mis-typed pointer, size overflow */
    RS_ERR_UNSUPPORTED_DTYPE = 2,  /* dtype is not an rs_dtype */
    RS_ERR_OVERLAP = 3,            /* in/out ranges overlap and the call is not exact in-place */
    RS_ERR_CUDA = 4,               /* a CUDA runtime call or the launch failed */
    RS_ERR_NOT_DEVICE_MEMORY = 5,  /* a pointer is not addressable by the current device */
    RS_ERR_NO_PATH = 6             /* the forced options cannot serve this shape */
} rs_status;

/* Row operations served by the same row engine (rs_plan.op). */
typedef enum {
    RS_OP_SOFTMAX = 0,   /* rowsoftmax_fwd */
    RS_OP_RMSNORM = 1,   /* rmsnorm_fwd */
    RS_OP_LAYERNORM = 2  /* layernorm_fwd */
} rs_op;

/* Kernel families (see rs_plan). */
typedef enum {
    RS_PATH_AUTO = 0,     /* let the library choose (the default) */
    RS_PATH_ROWS = 1,     /* single pass, the row held in registers; 1..1024 threads per row */
    RS_PATH_CLUSTER = 2,  /* wide rows: a cluster of CTAs per row, each CTA stages its slice in
                             shared memory with bulk asynchronous copies (TMA engine), online (m, l),
                             partial pairs merged over distributed shared memory; reads HBM once */
    RS_PATH_STREAM = 3,   /* any row: a cluster per row streams its slice twice from global memory
                             (online (m, l) on the first read, normalise on the second); reads 2x.
                             Normalisations: one CTA per row, reading it once per moment and
                             once to write (RMSNorm 2x, LayerNorm 3x) */
    RS_PATH_RING = 4      /* single pass as RS_PATH_ROWS, but a persistent grid whose CTAs stage the
                             next row groups in a ring of shared-memory stages filled by bulk
                             asynchronous copies (TMA engine); 16-byte aligned data only */
} rs_path;

/* Where RS_PATH_RING keeps a row between its passes. */
typedef enum {
    RS_RING_AUTO = 0,
    RS_RING_REGISTERS = 1,  /* fp32 copies in registers: one exp per element */
    RS_RING_REREAD = 2,     /* re-read the staged row from shared memory in each pass: two exps per
                               element, far fewer registers, more resident warps */
    RS_RING_THREAD_COPIES = 3  /* the causal softmax on 16-bit rows (the default there): each thread
                                  copies the units of its row that hold kept elements into the stage
                                  with 16-byte asynchronous copies and holds them in registers as fp32;
                                  the masked part is never copied; 2 or 3 stages */
} rs_ring_values;

/*
 * Forcing options for tests and tuning.  Zero fields mean "choose".  A NULL
 * rs_options pointer is the same as all zeros, i.e. rowsoftmax_fwd.
 */
typedef struct {
    int path;             /* rs_path */
    int threads_per_row;  /* RS_PATH_ROWS: 1,2,4,8,16,32 or a multiple of 32 up to 1024 */
    int vec_per_thread;   /* RS_PATH_ROWS: 16-byte vectors (or elements, when scalar) per thread */
    int block_threads;    /* threads per CTA (RS_PATH_ROWS: multiple of threads_per_row) */
    int cluster_size;     /* RS_PATH_CLUSTER / RS_PATH_STREAM: CTAs per row, 1..16 */
    int stages;           /* RS_PATH_RING: shared-memory stages per CTA, 2..8; register-holding
                             RS_PATH_CLUSTER: landing slots per CTA, 1..4 */
    int ring_values;      /* RS_PATH_RING: rs_ring_values */
    int force_scalar;     /* 1: element-wise accesses even when 16-byte vectors would be legal */
    int64_t grid_limit;   /* >0: cap on CTAs (rows loop inside the kernel); 0: one launch slot per row group */
    int64_t wait_limit_us;  /* RS_PATH_RING and the register-holding RS_PATH_CLUSTER kernel: >0 bounds
                               each wait for a bulk copy (default 4 s; the cluster's waits for its
                               peers' pairs take three times this limit) */
    int withhold_copies;  /* RS_PATH_RING or RS_PATH_CLUSTER (register-holding), failure-path tests
                             only: post the expected bytes of every stage or slot but never issue
                             the copies, so each copy wait runs out after wait_limit_us (which must be
                             set, at most 1 s), bit 0 of the device status word is set and the rows
                             whose waits ran out are left unwritten (the ring's other rows of the
                             same iteration may be partly written); no fault, trap or unbounded wait
                             is involved.  A plan on another kernel returns RS_ERR_NO_PATH */
    int strict_order;     /* 1: launch without programmatic dependent launch (see "Execution") */
} rs_options;

/* What a call would launch (filled by rowsoftmax_plan). */
typedef struct {
    int path;             /* rs_path actually chosen */
    int dtype;
    int vec_elems;        /* elements per access: 16/elem_size, or 1 for the element-wise kernels */
    int threads_per_row;  /* RS_PATH_ROWS / RS_PATH_RING */
    int vec_per_thread;   /* RS_PATH_ROWS / RS_PATH_RING */
    int rows_per_cta;     /* RS_PATH_ROWS; rows per stage for RS_PATH_RING */
    int block_threads;
    int cluster_size;     /* CTAs per row (1 for RS_PATH_ROWS / RS_PATH_RING) */
    int stages;           /* RS_PATH_CLUSTER: bulk-copy stages per CTA; RS_PATH_RING: ring depth */
    int ring_values;      /* RS_PATH_RING: RS_RING_REGISTERS, RS_RING_REREAD or RS_RING_THREAD_COPIES */
    int64_t chunk_elems;  /* RS_PATH_CLUSTER / RS_PATH_STREAM: row slice per CTA */
    int64_t grid;         /* CTAs launched */
    size_t smem_bytes;    /* dynamic shared memory per CTA */
    int64_t wait_limit_us;  /* copied from rs_options */
    int withhold_copies;  /* copied from rs_options */
    int op;               /* rs_op the plan serves */
    int strict_order;     /* copied from rs_options */
    int masked;           /* 1 for rowsoftmax_causal_* plans */
} rs_plan;

/* Device facts the planner needs; rowsoftmax_plan takes them explicitly so
 * the heuristics can be inspected without a GPU. */
typedef struct {
    int sm_count;                  /* multiprocessors */
    int max_smem_per_block_optin;  /* bytes, cudaDevAttrMaxSharedMemoryPerBlockOptin */
    int max_smem_per_sm;           /* bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor */
    int max_threads_per_sm;
    int cc_major, cc_minor;
} rs_device_info;

/*
 * y = softmax over each of the M rows of x (N columns).
 *   in, out          device pointers to x and y (see the data model above)
 *   M, N             rows and columns, >= 0; M == 0 or N == 0 is a no-op
 *                    returning RS_OK; N < 2^31
 *   in_row_stride    elements between the starts of consecutive rows of x, >= N
 *   out_row_stride   the same for y, >= N
 *   dtype            rs_dtype of both tensors
 *   stream           CUDA stream the kernel is enqueued on
 * Returns an rs_status.  RS_ERR_CUDA carries the CUDA error of the failing
 * call, readable (and cleared) with rowsoftmax_last_cuda_error.
 */
RS_API int rowsoftmax_fwd(const void* in, void* out, int64_t M, int64_t N,
                   int64_t in_row_stride, int64_t out_row_stride,
                   int dtype, cudaStream_t stream);

/* rowsoftmax_fwd with forcing options (tests, tuning sweeps).  The
 * semantics and error behaviour are those of rowsoftmax_fwd; a forced
 * configuration that cannot serve the shape returns RS_ERR_NO_PATH. */
RS_API int rowsoftmax_fwd_ex(const void* in, void* out, int64_t M, int64_t N,
                      int64_t in_row_stride, int64_t out_row_stride,
                      int dtype, cudaStream_t stream, const rs_options* opts);

/* Host-only: validate the arguments exactly as rowsoftmax_fwd_ex does and
 * describe the launch it would make on a device described by `dev` (no CUDA
 * call is made; pointers are only inspected for alignment and overlap).
 * Returns an rs_status; `plan` is filled on RS_OK (path 0 and grid 0 for an
 * empty problem). */
RS_API int rowsoftmax_plan(const void* in, const void* out, int64_t M, int64_t N,
                    int64_t in_row_stride, int64_t out_row_stride, int dtype,
                    const rs_options* opts, const rs_device_info* dev, rs_plan* plan);

/*
 * Row softmax under a causal mask, without reading the masked part: the
 * attention-score softmax that skips the fully masked causal region (the
 * mohakchugh.is-a.dev post, "How Flash Attention Uses Triton").  Row r keeps
 * its first
 *
 *     L_r = min(N, max(0, (r mod period) + 1 + diag_offset))
 *
 * elements: y[r][j] is the softmax of those L_r values for j < L_r and exactly
 * 0 for j >= L_r.  Elements at j >= L_r are never used (they may hold
 * anything, NaN included): the register rows, the ring on 16-bit rows
 * (RS_RING_THREAD_COPIES, the default there) and the clusters do not load
 * them, the bulk-copy ring (forced RS_RING_REGISTERS) stages whole rows and
 * ignores them; every output element is written.  For attention
 * scores [B, H, S_q, S_k] stored as (B*H*S_q) x S_k rows: period = S_q and
 * diag_offset = S_k - S_q.  L_r == 0 is an all -inf row: NaN.  Data model,
 * ownership, asynchrony and errors are those of rowsoftmax_fwd; period < 1 or
 * |diag_offset| > 2^62 is RS_ERR_INVALID_ARG.  The register-row, ring and
 * register-holding cluster kernels implement the mask; a shape that only the
 * streaming kernels could serve (rows wider than the clusters hold, or wide
 * rows without 16-byte alignment) returns RS_ERR_NO_PATH.
 */
RS_API int rowsoftmax_causal_fwd(const void* in, void* out, int64_t M, int64_t N,
                                 int64_t in_row_stride, int64_t out_row_stride, int64_t period,
                                 int64_t diag_offset, int dtype, cudaStream_t stream);

/* rowsoftmax_causal_fwd with forcing options (RS_PATH_STREAM and
 * RS_RING_REREAD, ring or cluster, return RS_ERR_NO_PATH). */
RS_API int rowsoftmax_causal_fwd_ex(const void* in, void* out, int64_t M, int64_t N,
                                    int64_t in_row_stride, int64_t out_row_stride, int64_t period,
                                    int64_t diag_offset, int dtype, cudaStream_t stream,
                                    const rs_options* opts);

/* Host-only planner of rowsoftmax_causal_fwd_ex (plan.masked = 1). */
RS_API int rowsoftmax_causal_plan(const void* in, const void* out, int64_t M, int64_t N,
                                  int64_t in_row_stride, int64_t out_row_stride, int64_t period,
                                  int64_t diag_offset, int dtype, const rs_options* opts,
                                  const rs_device_info* dev, rs_plan* plan);

/*
 * Row normalisations on the same engine (one read of x, one write of y for
 * every row that the register and ring kernels hold; RS_PATH_STREAM re-reads
 * wider rows).  Data model, ownership, in-place rule, asynchrony and error
 * behaviour are those of rowsoftmax_fwd; `weight` and `bias` are further
 * DEVICE pointers to N values of the same storage type `dtype` (contiguous,
 * read only, element-aligned; 16-byte alignment of both, as of x and y, lets
 * the vector kernels run), and may be NULL (weight 1, bias 0).  They must not
 * overlap `out` (RS_ERR_OVERLAP).  `eps` must be finite and >= 0
 * (RS_ERR_INVALID_ARG otherwise); the kernels compute in fp32 and round the
 * result to `dtype` with round-to-nearest-even.
 *
 * RMSNorm, after the "Reference Kernel: RMSNorm" of the Hugging Face
 * "triton-kernels" skill page (fp32 accumulation, masked lanes read as 0):
 *
 *     y[r][j] = x[r][j] / sqrt(sum_k x[r][k]^2 / N + eps) * w[j].
 */
RS_API int rmsnorm_fwd(const void* in, void* out, const void* weight, int64_t M, int64_t N,
                       int64_t in_row_stride, int64_t out_row_stride, double eps, int dtype,
                       cudaStream_t stream);

/*
 * LayerNorm, which the nano-triton post ("Rebuilding Triton and Helion from
 * Scratch", the opening and "deuteron: the autotuning layer") names beside
 * softmax as a memory-bound row kernel, without a formula; the plain
 * definition is taken, population variance and eps inside the square root:
 *
 *     mu_r  = sum_k x[r][k] / N,   var_r = sum_k (x[r][k] - mu_r)^2 / N,
 *     y[r][j] = (x[r][j] - mu_r) / sqrt(var_r + eps) * w[j] + b[j].
 *
 * Arguments as rmsnorm_fwd, plus `bias`.
 */
RS_API int layernorm_fwd(const void* in, void* out, const void* weight, const void* bias, int64_t M,
                         int64_t N, int64_t in_row_stride, int64_t out_row_stride, double eps,
                         int dtype, cudaStream_t stream);

/* rmsnorm_fwd (op RS_OP_RMSNORM, bias must be NULL) or layernorm_fwd (op
 * RS_OP_LAYERNORM) with forcing options.  Paths RS_PATH_ROWS, RS_PATH_RING
 * and RS_PATH_STREAM serve the normalisations; RS_PATH_CLUSTER and
 * RS_RING_REREAD return RS_ERR_NO_PATH.  An op that is not RS_OP_RMSNORM or
 * RS_OP_LAYERNORM is RS_ERR_INVALID_ARG. */
RS_API int rownorm_fwd_ex(int op, const void* in, void* out, const void* weight, const void* bias,
                          int64_t M, int64_t N, int64_t in_row_stride, int64_t out_row_stride,
                          double eps, int dtype, cudaStream_t stream, const rs_options* opts);

/* Host-only planner of rownorm_fwd_ex, as rowsoftmax_plan is of
 * rowsoftmax_fwd_ex. */
RS_API int rownorm_plan(int op, const void* in, const void* out, const void* weight, const void* bias,
                        int64_t M, int64_t N, int64_t in_row_stride, int64_t out_row_stride,
                        double eps, int dtype, const rs_options* opts, const rs_device_info* dev,
                        rs_plan* plan);

/*
 * The softmax of rows split by columns into shards: the vocabulary-parallel
 * softmax, where each device holds a block of columns of every row (logits
 * over a vocabulary sharded across devices), and, on one device, the split
 * of a few very wide rows into blocks so that every multiprocessor works on
 * them.  The steps are those of the online normaliser of the
 * mohakchugh.is-a.dev post ("How Flash Attention Uses Triton"): each shard
 * reduces its columns of a row to a pair (m, l) -- m the max, l the sum of
 * exp(x - m) -- the pairs of a row are merged as
 *     m = max(m1, m2),   l = l1 exp(m1 - m) + l2 exp(m2 - m),
 * from (-inf, 0), and each shard writes exp(x - m) / l with the merged pair.
 * In exact arithmetic the result is the row softmax of the whole row.
 *
 * Pairs are stored as two fp32 values {m, l} per row (8 bytes, 8-byte aligned
 * device memory), m in the units of x (so m + log(l) is the log of the sum of
 * exp over the shard).  A shard whose columns of a row are all -inf, or that
 * has no column, gives (-inf, 0); NaN entries make l NaN; a row whose merged
 * max is -inf finishes as NaN (the whole row was -inf).  Data model, device
 * pointers, asynchrony and error codes are those of rowsoftmax_fwd; a pair
 * array that overlaps a tensor it is read or written with is RS_ERR_OVERLAP.
 * Typical use on R devices, each holding x[:, c_s : c_s + N_s]:
 *     rowsoftmax_partial_fwd(x_s, pairs_s, M, N_s, ...);
 *     all-gather pairs_s over the devices into R x M pairs (shard-major);
 *     rowsoftmax_finish_fwd(x_s, y_s, all_pairs, R, M, N_s, ...);
 */

/* ml[r] = (m, l) of row r over its N columns (one shard).  N may be 0 (the
 * pairs are then (-inf, 0) and `in` is not read).  `ml` holds M pairs. */
RS_API int rowsoftmax_partial_fwd(const void* in, void* ml, int64_t M, int64_t N, int64_t in_row_stride, int dtype,
                                  cudaStream_t stream);

/* ml_out[r] = the merge of the R pairs ml_in[s * M + r], s = 0 .. R - 1 (R x M
 * pairs, shard-major: the layout of an all-gather of the shards' pair
 * arrays).  R == 0 gives (-inf, 0).  The two arrays must not overlap. */
RS_API int rowsoftmax_merge_ml(const void* ml_in, void* ml_out, int64_t R, int64_t M, cudaStream_t stream);

/* y[r][j] = exp(x[r][j] - m_r) / l_r for the N columns of this shard, with
 * (m_r, l_r) the merge of the R >= 1 pairs ml[s * M + r] (R == 1: an already
 * merged pair array).  In place (in == out, equal strides) is allowed; `ml`
 * must not overlap `out`.  R < 1 is RS_ERR_INVALID_ARG. */
RS_API int rowsoftmax_finish_fwd(const void* in, void* out, const void* ml, int64_t R, int64_t M, int64_t N,
                                 int64_t in_row_stride, int64_t out_row_stride, int dtype, cudaStream_t stream);

/* Host-only: the workspace bytes rowsoftmax_split_fwd needs for M rows of N
 * columns (0 for an empty problem): M * (S + 1) pairs, S the blocks a row is
 * split into (about 4096 (row, block) items in all, blocks of at least 32 KB). */
RS_API int rowsoftmax_split_workspace_size(int64_t M, int64_t N, int dtype, size_t* bytes);

/* The row softmax of rowsoftmax_fwd computed as above on one device: each row
 * is split into S blocks, one pair per (row, block) is written to
 * `workspace`, the pairs are merged and every block finishes.  x is read
 * twice (the second read mostly from L2 when the input fits there) and y
 * written once.  For rows too few to fill the device and too wide for the
 * cluster kernels (a few rows of millions of values); with many rows
 * rowsoftmax_fwd, which reads x once, is faster.  `workspace` is caller-owned
 * device memory of at least rowsoftmax_split_workspace_size bytes, 8-byte
 * aligned, not overlapping x or y (RS_ERR_INVALID_ARG when too small);
 * its contents on entry do not matter and are undefined afterwards.
 * In place (in == out, equal strides) is allowed. */
RS_API int rowsoftmax_split_fwd(const void* in, void* out, int64_t M, int64_t N, int64_t in_row_stride,
                                int64_t out_row_stride, int dtype, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/*
 * rowsoftmax_split_fwd for callers that cannot allocate device memory.  The
 * pages have no counterpart: this is an interface choice of this library.
 * Some callers may not call cudaMalloc around a softmax: a serving loop whose
 * device memory is all reserved up front by another allocator (a framework's
 * caching allocator or memory pool owns it, and memory taken behind its back
 * can make its own later allocations fail), or code on a latency-critical
 * path where cudaMalloc, which can synchronise the device, is not allowed.
 * This entry point needs no workspace argument: the split's pairs go to a
 * buffer of RS_SPLIT_NOALLOC_MAX_BYTES (1 MiB) that the library defines in
 * device memory, which every GPU that loads the library holds until the
 * process exits.  It calls no cudaMalloc, cudaFree or other allocating
 * routine.  The caller still passes `in` and `out`; everything else is as
 * rowsoftmax_split_fwd.
 *   - Problems whose workspace (rowsoftmax_split_workspace_size) exceeds
 *     RS_SPLIT_NOALLOC_MAX_BYTES return RS_ERR_INVALID_ARG before anything
 *     is launched (up to 65536 rows fit, whatever N).
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it; make that
 *     first call before any stream capture.
 *   - Every call shares the one buffer, and the buffer keeps the last call's
 *     contents.  Nothing in it has to start at zero: each call writes every
 *     pair it later reads.  Calls whose kernels overlap on the GPU (on
 *     different streams, or from different host threads, without ordering
 *     between them) race on the buffer and give undefined results: order
 *     them, for instance on one stream.
 */
#define RS_SPLIT_NOALLOC_MAX_BYTES (1u << 20)
RS_API int rowsoftmax_split_fwd_noalloc(const void* in, void* out, int64_t M, int64_t N, int64_t in_row_stride,
                                        int64_t out_row_stride, int dtype, cudaStream_t stream);

/* Host-only: fill `dev` for the current CUDA device.  Returns RS_OK or
 * RS_ERR_CUDA. */
RS_API int rowsoftmax_device_info(rs_device_info* dev);

/* Static text for an rs_status value ("unknown status" otherwise). */
RS_API const char* rowsoftmax_status_string(int status);

/* The cudaError_t of the last RS_ERR_CUDA returned on this host thread (0 if
 * none); reading it clears it. */
RS_API int rowsoftmax_last_cuda_error(void);

/*
 * Device-side status word of the current device.  The ring and cluster
 * kernels bound every wait on an mbarrier; a wait that runs out sets bit 0
 * and its CTA abandons the rows it was serving: the output of a call that
 * reported a timeout is undefined (unwritten, or partly written) in those
 * rows, and in the ring's other rows of the same row group.  Reads the word
 * (synchronously, with cudaMemcpyFromSymbol) into *flags and clears it when
 * `clear` is nonzero.  Returns RS_OK or RS_ERR_CUDA.
 */
RS_API int rowsoftmax_device_status(unsigned int* flags, int clear);

/*
 * Host-only description of the register layout of RS_PATH_ROWS: element j of
 * a row lives in thread (j / vec) mod threads, slot
 * (j / (threads * vec)) * vec + j mod vec of that thread -- the group-cyclic
 * layout of the nano-triton post ("The register layout"): consecutive 16-byte
 * groups are dealt to the threads round robin, so a warp's accesses are
 * adjacent and each thread's group is one 16-byte access.  Returns RS_OK, or
 * RS_ERR_INVALID_ARG for j < 0, threads < 1 or vec < 1.
 */
RS_API int rowsoftmax_layout_owner(int64_t j, int threads, int vec, int* thread, int64_t* slot);

#ifdef __cplusplus
}
#endif

#endif /* ROWSOFTMAX_H */
