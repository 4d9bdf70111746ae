/*
 * gemm.h -- C ABI of libgemm, a dense GEMM for one NVIDIA GB300 (sm_103a).
 *
 * The operation (every entry point below computes it):
 *
 *     C[m][n] = sum_{k=0}^{K-1} A(m,k) * B(n,k),   0 <= m < M, 0 <= n < N
 *
 * A is M x K and B is N x K, so C = A * B^T in storage terms. This is the
 * product of the CuTe DSL Ampere SGEMM example (its module docstring: A is
 * MxK, B is NxK, C is MxN, each with a selectable major mode; its reference
 * check contracts "mk,nk->mn") and of the CK Tile practice GEMM ("Problem
 * Size Configuration": A M x K, B N x K, C M x N). The Gluon Multi-CTA
 * tutorial's matmul_multicta stores B as K x N row-major, which is the
 * N-major B here. Accumulation is fp32 for every type; C is overwritten
 * (beta = 0).
 *
 * Layout. Leading dimensions are in ELEMENTS. "major" names the contiguous
 * dimension (the CuTe SGEMM example's a_major "k"|"m", b_major "k"|"n",
 * c_major "n"|"m"):
 *
 *     A K-major  (GEMM_MAJOR_K)  : A(m,k) = A[m*lda + k],  lda >= K
 *     A M-major  (GEMM_MAJOR_MN) : A(m,k) = A[k*lda + m],  lda >= M
 *     B K-major  (GEMM_MAJOR_K)  : B(n,k) = B[n*ldb + k],  ldb >= K
 *     B N-major  (GEMM_MAJOR_MN) : B(n,k) = B[k*ldb + n],  ldb >= N
 *     C N-major  (GEMM_MAJOR_MN) : C(m,n) = C[m*ldc + n],  ldc >= N  (row-major)
 *     C M-major  (GEMM_MAJOR_K)  : C(m,n) = C[n*ldc + m],  ldc >= M  (column-major)
 *
 * For C the enum slot GEMM_MAJOR_K means "M contiguous" (C has no K mode).
 * Any leading dimension and any base address aligned to the element size is
 * accepted (the pages' kernels need 16-byte aligned contiguous dimensions;
 * this library repacks misaligned 16-bit A/B into 16-byte aligned scratch,
 * may transpose large K-major fp32 A/B into MN-major scratch, and stores
 * misaligned C with predicated scalar stores).
 *
 * Types (dtype argument):
 *
 *     GEMM_F32       A, B, C fp32.       FP32 FFMA (SIMT) kernel.
 *     GEMM_F16_F32   A, B fp16, C fp32.  tcgen05 tensor-core kernel.
 *     GEMM_BF16_F32  A, B bf16, C fp32.  tcgen05 tensor-core kernel.
 *     GEMM_F16_F16   A, B fp16, C fp16.  tcgen05; C rounded to nearest even.
 *     GEMM_BF16_BF16 A, B bf16, C bf16.  tcgen05; C rounded to nearest even.
 *
 * Degenerate sizes: M == 0 or N == 0 is a no-op (returns GEMM_OK, launches
 * nothing); K == 0 writes C = 0. Negative sizes are GEMM_ERR_INVALID_ARG.
 *
 * Execution and ownership: the caller owns A, B and C. gemm() takes DEVICE
 * pointers of the current device -- memory from cudaMalloc, cudaMallocAsync
 * or a device memory pool of that device (cudaPointerGetAttributes reports
 * type device and the current ordinal). Host memory (pinned or pageable),
 * managed memory and other GPUs' memory are GEMM_ERR_INVALID_ARG, checked
 * before any launch: the library runs on one GPU and no kernel of it ever
 * addresses another GPU's memory. gemm() is asynchronous on `stream` (a
 * cudaStream_t of the current device; NULL = legacy default stream) and never
 * synchronises. C overlapping A or B is undefined
 * and not checked. Scratch for repacking misaligned operands comes from a
 * library-private, stream-ordered memory pool (cudaMallocAsync on `stream`,
 * freed on the same stream after use), so concurrent calls on different
 * streams do not share scratch. C++ exceptions never cross this ABI.
 *
 * Errors: every entry point returns GEMM_OK (0) or a negative status:
 *     GEMM_ERR_INVALID_ARG  bad size, pointer, leading dimension, enum or
 *                           alignment, or an operand that is not device
 *                           memory of the current device; checked on the
 *                           host before any launch
 *     GEMM_ERR_UNSUPPORTED  no usable device, or the device is not sm_103
 *     GEMM_ERR_CUDA         a CUDA runtime call failed (allocation, copy,
 *                           tensor-map encode, launch)
 *     GEMM_ERR_TIMEOUT      (from gemm_check_device_error) a kernel gave up
 *                           waiting on a pipeline barrier after its time
 *                           limit and wrote no trustworthy C
 * Device-side timeouts are reported asynchronously: a kernel that times out
 * records it in a per-device error word and returns without a trustworthy C;
 * gemm_check_device_error reads and clears that word. Every launch carries a
 * generation number of its own and gives up early only on a timeout of its
 * own generation, so a timeout does not spill over into later launches: a
 * GEMM launched after another one timed out, before anyone called
 * gemm_check_device_error, still runs to completion and is correct.
 */
#ifndef LIBGEMM_GEMM_H
#define LIBGEMM_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum gemm_major { GEMM_MAJOR_K = 0, GEMM_MAJOR_MN = 1 };

enum gemm_dtype {
    GEMM_F32 = 0,
    GEMM_F16_F32 = 1,
    GEMM_BF16_F32 = 2,
    GEMM_F16_F16 = 3,
    GEMM_BF16_BF16 = 4
};

enum gemm_status {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = -1,
    GEMM_ERR_UNSUPPORTED = -2,
    GEMM_ERR_CUDA = -3,
    GEMM_ERR_TIMEOUT = -4
};

/*
 * gemm -- C = A * B^T on the current CUDA device, asynchronously on `stream`.
 * A, B, C are device pointers laid out as described above. The fp32 type runs
 * the FFMA kernel modelled on the CuTe DSL Ampere SGEMM example (multistage
 * smem pipeline, register double buffer, predicated tails); the 16-bit types
 * run the tcgen05 kernel modelled on the Gluon Multi-CTA tutorial's "fast
 * matmul kernel" (TMA -> mbarrier ring -> 2-CTA tcgen05.mma into TMEM ->
 * epilogue warps), re-designed for sm_103a.
 */
int gemm(int64_t M, int64_t N, int64_t K,
         const void *A, int64_t lda, int a_major,
         const void *B, int64_t ldb, int b_major,
         void *C, int64_t ldc, int c_major,
         int dtype, void *stream);

/* Activations of the fused epilogue. */
enum gemm_activation {
    GEMM_ACT_NONE = 0,
    GEMM_ACT_RELU = 1, /* max(x, 0) */
    GEMM_ACT_GELU = 2  /* x * Phi(x) = x / 2 * (1 + erf(x / sqrt(2))) */
};

/* Fused epilogue of gemm_ex: D = act(alpha * (A * B^T) + beta * C + bias). */
typedef struct gemm_epilogue {
    float alpha;      /* scale of the product */
    float beta;       /* scale of the incoming C; 0 = C is not read */
    const void *bias; /* NULL, or a DEVICE vector of C's element type with one
                         entry per column of C (index n), 16-bit aligned */
    int activation;   /* enum gemm_activation */
} gemm_epilogue;

/*
 * gemm_ex -- C = act(alpha * A * B^T + beta * C + bias[n]) in one pass: the
 * accumulator (fp32) goes through the epilogue in fp32 registers before C is
 * rounded to its type and stored. This is the CuTe DSL Ampere SGEMM example's
 * `epilogue_op` hook (applied to the accumulator before the store), with
 * scaling, bias and activation. `epi` == NULL, or alpha 1 / beta 0 / no bias
 * / no activation, is exactly gemm(). With beta != 0, C is read before it is
 * overwritten (it must hold valid data). K == 0 gives act(beta * C + bias).
 * Arguments, layouts, status codes and asynchrony are those of gemm(); an
 * unknown activation or a misaligned bias is GEMM_ERR_INVALID_ARG.
 */
int gemm_ex(int64_t M, int64_t N, int64_t K,
            const void *A, int64_t lda, int a_major,
            const void *B, int64_t ldb, int b_major,
            void *C, int64_t ldc, int c_major,
            int dtype, const gemm_epilogue *epi, void *stream);

/*
 * gemm_host -- the same product with HOST buffers (pinned or pageable).
 * On `stream`: takes device buffers from the library's scratch pool (row
 * pitches rounded up to 16 bytes), copies the addressed elements of A and B
 * to them (2-D copies, so padding between rows is neither read nor written),
 * runs the same kernels as gemm(), copies C back into the addressed elements
 * of the host C and returns the buffers to the pool; the call returns once
 * the work is enqueued. The host buffers must stay valid and unmodified until
 * the stream has completed (synchronise before reading C). With pageable host
 * memory the copies are synchronous with respect to the host. Same status
 * codes and degenerate-size rules as gemm().
 */
int gemm_host(int64_t M, int64_t N, int64_t K,
              const void *A, int64_t lda, int a_major,
              const void *B, int64_t ldb, int b_major,
              void *C, int64_t ldc, int c_major,
              int dtype, void *stream);

/*
 * gemm_noalloc -- the same product for the 16-bit types (GEMM_F16_F32,
 * GEMM_BF16_F32, GEMM_F16_F16, GEMM_BF16_BF16) without allocating any device
 * memory. This entry point has no counterpart in the pages; it exists for
 * callers that cannot allocate: a program whose own allocator has already
 * reserved the device memory, or a latency-critical loop in which a device
 * allocation (and the synchronisation it may bring) is not acceptable.
 *
 * Where gemm() would repack an operand whose rows are not 16-byte aligned
 * into pool scratch, gemm_noalloc() repacks it into a fixed 32 MiB array
 * inside the library's device image, which every GPU that loads the library
 * holds until the process exits. Limit: the repacked operands together must
 * fit in 32 MiB (each takes rows x (contiguous extent rounded up to 8
 * elements) x 2 bytes, rounded up to 256 bytes; operands that are already
 * aligned take nothing); a larger problem returns GEMM_ERR_INVALID_ARG and
 * launches nothing. GEMM_F32 returns GEMM_ERR_UNSUPPORTED.
 *
 * All calls share the array and it keeps the last call's contents; nothing in
 * it needs to start at zero (each call rewrites every element its kernel
 * reads). Calls whose work overlaps on the GPU -- on different streams, or on
 * different threads without ordering -- race on the array; order them on one
 * stream. The first call on a device looks the array up on that device
 * (cudaGetSymbolAddress) and caches the address; make that first call before
 * any stream capture. It runs the kernel configuration gemm() would run for
 * the same problem (options, then a gemm_tune entry, then the default).
 * Otherwise arguments, layouts, status codes and asynchrony are those of
 * gemm().
 */
int gemm_noalloc(int64_t M, int64_t N, int64_t K,
                 const void *A, int64_t lda, int a_major,
                 const void *B, int64_t ldb, int b_major,
                 void *C, int64_t ldc, int c_major,
                 int dtype, void *stream);

/* A kernel configuration chosen by gemm_tune (the option values it stands
   for; see enum gemm_option). */
typedef struct gemm_tuning {
    int simt_config;    /* fp32: FFMA tile configuration 1..9 */
    int simt_transpose; /* fp32: 1 = run K-major operands as they are,
                           2 = transpose them to MN-major first */
    int tc_cta_group;   /* 16-bit: 1 or 2 CTAs per tile */
    int tc_multicast;   /* 16-bit: 1 off, 2 B multicast across two pairs */
    int tc_store;       /* 16-bit: 0 TMA store where possible, 1 st.global */
    float ms;           /* measured time per call of the chosen configuration */
    int candidates;     /* configurations measured */
    int tc_scheduler;   /* 16-bit: 1 static persistent, 2 cluster launch control */
} gemm_tuning;

/*
 * gemm_tune -- per-problem configuration selection (the pages' autotune
 * utilities, CuTe DSL `tune`/`autotune_jit`, done natively): runs every
 * kernel configuration valid for this problem on the caller's buffers and
 * stream (one warm-up call and `iterations` timed calls each, CUDA events;
 * the operand-multicast variant is never a candidate),
 * records the fastest in a process-wide table keyed by (M, N, K, dtype,
 * majors, 16-byte alignment of A, B and C) and writes it to *out (may be
 * NULL). Later gemm(), gemm_ex() and gemm_host() calls on a matching problem
 * use the recorded configuration for every option left at 0 (automatic).
 * C is overwritten with the product. Synchronises `stream`. iterations <= 0
 * means 5. A problem with nothing to run (M, N or K zero) records nothing
 * and returns GEMM_OK with out->candidates == 0. Status codes as gemm().
 */
int gemm_tune(int64_t M, int64_t N, int64_t K,
              const void *A, int64_t lda, int a_major,
              const void *B, int64_t ldb, int b_major,
              void *C, int64_t ldc, int c_major,
              int dtype, int iterations, void *stream, gemm_tuning *out);

/* gemm_tune_reset -- forget every configuration gemm_tune recorded. */
void gemm_tune_reset(void);

/*
 * softmax_rows -- y[m][n] = exp(x[m][n] - max_j x[m][j]) / sum_j exp(x[m][j] -
 * max_j x[m][j]) for every row m < M of an fp32 matrix (row pitches ldx and
 * ldy in elements, >= N; 4-byte aligned device pointers). The multi-CTA row
 * softmax of the Gluon Multi-CTA tutorial: rows up to 1024 columns take one
 * warp each, rows up to 16384 one CTA, longer rows a thread-block cluster of
 * up to 16 CTAs that combine their partial maxima and sums through
 * distributed shared memory, so x is read once and y written once. A
 * cluster's CTAs take 16384 columns each for aligned rows (x and y 16-byte
 * aligned, ldx and ldy multiples of 4, N <= 262144), else 32768. N up to
 * 524288; longer rows return GEMM_ERR_UNSUPPORTED. y may be x itself (ldy == ldx); other overlaps are
 * undefined. Asynchronous on `stream`; status codes as gemm(). The aligned
 * cluster layout's wait for its peers' partials is bounded by
 * GEMM_OPT_WAIT_LIMIT_NS; one that runs out is reported by
 * gemm_check_device_error() as GEMM_ERR_TIMEOUT.
 */
int softmax_rows(int64_t M, int64_t N, const float *x, int64_t ldx, float *y, int64_t ldy,
                 void *stream);

/* gemm_strerror -- a static, NUL-terminated description of a status code. */
const char *gemm_strerror(int status);

/*
 * gemm_check_device_error -- synchronises `stream`, then reads and clears the
 * current device's error word. Returns GEMM_OK, GEMM_ERR_TIMEOUT (a kernel
 * gave up on a barrier wait) or GEMM_ERR_CUDA (the synchronisation failed).
 */
int gemm_check_device_error(void *stream);

/*
 * gemm_device_checks -- debug builds only (the library compiled with
 * LIBGEMM_DEVICE_CHECKS): synchronises `stream`, then reads and clears the
 * current device's device-check word into *first: 0 when every device-side
 * check passed since the last call, else (code << 56 | detail) of the first
 * that failed (codes: 1 a tensor-core work unit outside the tile grid, 2 a
 * TMA coordinate not 16-byte aligned, 3 a tensor-core epilogue store outside
 * C, 4 an FFMA tile or K-slice outside the problem, 5 an FFMA store outside
 * C); the failed access itself was skipped. Returns GEMM_OK, GEMM_ERR_CUDA,
 * GEMM_ERR_INVALID_ARG (first == NULL), or GEMM_ERR_UNSUPPORTED in a library
 * built without the checks (*first = 0).
 */
int gemm_device_checks(void *stream, uint64_t *first);

/*
 * gemm_release_workspace -- synchronises every device the library has used
 * and returns its cached scratch memory (the per-stream repack and split
 * buffers, and what its pools keep of repack buffers and gemm_host() copies)
 * to the driver. Call it when no other thread is inside a gemm* call.
 */
void gemm_release_workspace(void);

/*
 * gemm_launch_count -- number of kernels this library has launched in this
 * process (all devices). Lets a caller count the launches of a timed region.
 */
uint64_t gemm_launch_count(void);

/* Options (process-wide; read at each call). */
enum gemm_option {
    /* Time limit of every pipeline barrier wait in the tensor-core kernel,
       the TMA-fed FFMA kernel (GEMM_OPT_SIMT_CONFIG 9) and the clustered
       softmax, in nanoseconds (default 1000000000; 0 restores the default).
       A wait that runs past it records GEMM_ERR_TIMEOUT in the device error
       word and the kernel winds down without further writes to C. */
    GEMM_OPT_WAIT_LIMIT_NS = 1,
    /* Tensor-core kernel variant: 0 = automatic (the 2-CTA pair kernel, or
       one CTA per tile for problems with fewer 256 x 256 tiles than a quarter
       of the SMs; see GEMM_OPT_TC_TILE_N),
       1 = one CTA per tile (cta_group::1, 128-row tiles),
       2 = CTA pair per tile (cta_group::2, 256-row tiles). */
    GEMM_OPT_TC_CTA_GROUP = 2,
    /* Test hook for the timeout path: 1 makes the tensor-core kernel's
       epilogue wait on a barrier that nothing completes, so every call times
       out (after GEMM_OPT_WAIT_LIMIT_NS) and reports GEMM_ERR_TIMEOUT through
       gemm_check_device_error. 0 (default) = off. */
    GEMM_OPT_TC_FAULT_INJECT = 3,
    /* Tile configuration of the fp32 FFMA kernel (all 128 x 128 CTA tiles),
       as (k-depth, ring stages, FMA form, CTAs per SM the registers are
       sized for, outputs per thread): 0 = automatic (9, the fastest
       measured at 8192^3),
       1 = (16, 4, packed, 2, 8 x 8), 2 = (16, 4, scalar, 2, 8 x 8),
       3 = (32, 3, packed, 2, 8 x 8), 4 = (8, 3, packed, 2, 8 x 8) -- the CuTe
       Ampere example's 128 x 128 x 8 with 3 stages --,
       5 = (16, 4, packed, 1, 8 x 8), 6 = (32, 4, packed, 1, 8 x 8),
       7 = (16, 4, packed, 2, 8 x 16), 8 = (32, 3, packed, 2, 8 x 16),
       9 = (16, 6, packed, 2, 8 x 16) with shared memory filled by TMA
       tensor copies and per-stage mbarriers instead of cp.async and a CTA
       barrier, when A and B (after any transpose) are MN-major with 16-byte
       aligned bases and row pitches; 7 otherwise.
       8 x 8 runs 256 threads per CTA, 8 x 16 runs 128. "Packed" is the
       two-lane fma.rn.f32x2. Every configuration rounds each multiply-add
       once (IEEE fma) and sums k in the same order. */
    GEMM_OPT_SIMT_CONFIG = 4,
    /* K-major fp32 operands: 0 = automatic (an operand is first transposed
       into an MN-major copy in pool scratch when the other output dimension
       is >= 512 and M*N*K >= 2^31; the FFMA kernel reads MN-major tiles with
       16-byte copies), 1 = never transpose (transposing 4-byte copies into
       shared memory instead), 2 = always transpose. */
    GEMM_OPT_SIMT_TRANSPOSE = 5,
    /* How the tensor-core kernel writes C: 0 = automatic (a TMA tensor store
       of each 32 x 32 chunk that lies entirely inside C when C's base and
       row pitch are 16-byte aligned; row-coalesced st.global for the other
       chunks), 1 = always st.global. */
    GEMM_OPT_TC_STORE = 6,
    /* Operand multicast in the 2-CTA tensor-core kernel: 0 = automatic
       (off; gemm_tune never selects it), 1 = off, 2 = on: clusters of two CTA
       pairs compute vertically adjacent 256 x 256 tiles and each half of the
       shared B tile is loaded once per cluster and multicast by TMA to both
       pairs. The multicast copies only ever address memory of the current
       device: every operand is checked to be this GPU's memory first. */
    GEMM_OPT_TC_MULTICAST = 7,
    /* Test hook for softmax_rows' timeout path: 1 makes the first CTA of the
       first row's cluster (aligned rows of 16385..262144 columns) withhold
       its partial, so that row's CTAs wait out GEMM_OPT_WAIT_LIMIT_NS and
       report GEMM_ERR_TIMEOUT through gemm_check_device_error; the row's y
       is then undefined. 0 (default) = off. */
    GEMM_OPT_SOFTMAX_FAULT_INJECT = 8,
    /* Wave tail of the fp32 FFMA kernel: 0 = automatic (the tiles left over
       after the last full round of 128 x 128 tiles over the SMs are split
       along K into 2-8 slices, computed by separate CTAs into pool scratch
       and summed in slice order by a fixup kernel before the epilogue, when
       a per-SM model predicts a saving of at least 10%, every slice keeps at
       least 32 k-tiles, and there is no full round or at least two; with
       exactly one full round and at most 1.8 rounds' worth of tiles, the
       TMA-fed kernel instead runs one whole tile per SM and shares the rest
       of the tiles' k-iterations evenly over one more CTA per SM (stream-K),
       whose partial tiles a fixup kernel adds in k order), 1 = never split,
       2 = always split the last wave of resident CTAs into 2-4 slices (every
       tile when there is less than one wave; tests), 3 = always stream-K in
       the TMA-fed kernel (a third of the tiles whole; tests). A split changes
       the order of the k-sum, never the per-product rounding. */
    GEMM_OPT_SIMT_SPLIT_TAIL = 9,
    /* Tile scheduler of the tensor-core kernel (the Gluon Multi-CTA
       tutorial's CLC-scheduled matmul): 0 = automatic (currently static),
       1 = static persistent (as many CTA pairs as fit, each walking every
       n-th tile of the raster order), 2 = cluster launch control (one
       cluster per tile is launched; running clusters take over tiles of
       clusters that have not started with clusterlaunchcontrol.try_cancel,
       a scheduler warp multicasting each response to both CTAs of the pair).
       The operand-multicast variant always uses the static schedule. */
    GEMM_OPT_TC_SCHEDULER = 10,
    /* Test hook for the TMA-fed FFMA kernel's timeout path: 1 makes its
       first CTA skip the copy of its second k-tile, so that CTA's waits run
       out after GEMM_OPT_WAIT_LIMIT_NS and gemm_check_device_error reports
       GEMM_ERR_TIMEOUT; C is then undefined. 0 (default) = off. */
    GEMM_OPT_SIMT_FAULT_INJECT = 11,
    /* Tile width of the tensor-core kernel in columns of C: 0 = automatic
       (256; a problem with fewer 256 x 256 tiles than a quarter of the SMs
       runs one CTA per tile, in the narrowest of 64 / 128 / 256 columns that
       still fits every tile into one round over the SMs), or 64, 128, 256
       (at least 64 per CTA: a CTA pair needs 128 or 256). Operand multicast
       always uses 256. */
    GEMM_OPT_TC_TILE_N = 12,
    /* Last round of the tensor-core kernel: 0 = automatic (when a launch
       takes at least two rounds of tiles over its resident clusters and the
       last round is at most half full, each of its tiles runs as two work
       units of half the width, so that round takes half as long), 1 = never,
       2 = always split the last round's tiles (tests). */
    GEMM_OPT_TC_SPLIT_TAIL = 13
};

/* gemm_set_option -- set an option; GEMM_OK or GEMM_ERR_INVALID_ARG. */
int gemm_set_option(int option, int64_t value);

/* gemm_get_option -- current value of an option, -1 for an unknown option. */
int64_t gemm_get_option(int option);

#ifdef __cplusplus
}
#endif

#endif /* LIBGEMM_GEMM_H */
