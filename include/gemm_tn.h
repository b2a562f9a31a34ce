/*
 * gemm_tn.h — C ABI of the GB300 (sm_103a) dense BF16 TN GEMM library.
 *
 * Operation (all entry points):
 *
 *     D = alpha * A * B^T + beta * C
 *
 *   A  M x K bf16, row-major with leading dimension lda >= K (K contiguous)
 *   B  N x K bf16, row-major with leading dimension ldb >= K (K contiguous)
 *   C  M x N, same element type as D, row-major, ldc >= N; not read when
 *      beta == 0 (it may then be NULL and NaN/Inf in it do not propagate)
 *   D  M x N bf16 or fp32 (out_dtype), row-major, ldd >= N
 *
 * Both operands are K-major — the "TN" convention of the
 * SM80_16x8x16_F32F16F16F32_TN atom named on the FlashAttention SM80 kernel
 * page (section on the SM80 mainloop).  Products are accumulated in fp32 on
 * the tensor cores (the GEMM whose work the H100 Nsight Compute page counts
 * as F = 2MNK, section 7); the epilogue computes alpha*acc + beta*c in fp32
 * and rounds once to bf16 (round-to-nearest-even) or stores fp32.  The
 * summation order over K is unspecified.
 *
 * Memory: every pointer is a DEVICE pointer owned by the caller.  A, B, C
 * and D must be 16-byte aligned and lda*2, ldb*2, ldc*esize, ldd*esize must
 * be multiples of 16 bytes (tensor-memory-accelerator addressing rules);
 * otherwise GEMM_ERR_MISALIGNED.  D may be the same buffer as C with
 * ldc == ldd (in-place beta); D must not overlap A or B.
 *
 * Asynchrony: calls enqueue work on `stream` (a cudaStream_t, NULL = the
 * legacy default stream) and return.  The return value covers argument
 * validation and the launch only.  A device-side failure (a bounded wait
 * that gave up) is recorded in a per-device status word that
 * gemm_get_status() reads.
 *
 * Degenerate shapes: M == 0 or N == 0 returns GEMM_OK with no launch;
 * K == 0 gives D = beta * C (or zeros).
 *
 * Library-owned memory: the skinny path (M <= 256) and the tiled k-split
 * use an fp32 partial-sum workspace and arrival counters, allocated (or
 * grown) on the first call for a (device, stream) pair that needs them and
 * kept until gemm_shutdown().  A skinny call that would allocate or grow it
 * during stream capture returns an error; a tiled call runs unsplit
 * instead.  Calls on different streams use different workspaces.
 *
 * Launch: kernels are launched with programmatic stream serialisation, so
 * their set-up (barrier initialisation, Tensor Memory allocation) may overlap
 * the tail of the previous kernel on the stream.  Each kernel waits for the
 * previous kernel's completion (griddepcontrol.wait) before its first global
 * memory access, so stream order is preserved for inputs and outputs.  The
 * one exception is opt-in: with gemm_tn_config.b_static the skinny kernel
 * loads its first ring of B before that wait.
 *
 * Thread safety: calls may come from several host threads; the last-error
 * string is per thread.
 *
 * Requires a compute capability 10.3 device (sm_103); anything else returns
 * GEMM_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef GEMM_TN_H_
#define GEMM_TN_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GEMM_OUT_BF16 = 0,
  GEMM_OUT_F32 = 1
} gemm_out_dtype;

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_VALUE = -1,      /* bad size, stride, dtype or NULL pointer */
  GEMM_ERR_MISALIGNED = -2,         /* pointer or stride breaks the 16-byte rule */
  GEMM_ERR_UNSUPPORTED_DEVICE = -3, /* current device is not sm_103 */
  GEMM_ERR_LAUNCH = -4,             /* CUDA launch or tensor-map encoding failed */
  GEMM_ERR_TIMEOUT = -5,            /* device: a bounded wait gave up */
  GEMM_ERR_NOT_IMPLEMENTED = -6,    /* requested path cannot run this shape */
  GEMM_ERR_OUT_OF_MEMORY = -7,      /* workspace allocation failed */
  GEMM_ERR_CUDA = -8                /* another CUDA runtime error */
} gemm_status;

typedef enum {
  GEMM_FP8_E4M3 = 0,  /* 1 sign, 4 exponent (bias 7), 3 mantissa bits; max 448; no infinities */
  GEMM_FP8_E5M2 = 1   /* 1 sign, 5 exponent (bias 15), 2 mantissa bits; max 57344; IEEE inf/NaN */
} gemm_fp8_format;

typedef enum {
  GEMM_ACT_NONE = 0,
  GEMM_ACT_RELU = 1,       /* max(x, 0) */
  GEMM_ACT_GELU = 2,       /* x * Phi(x) = 0.5 x (1 + erf(x / sqrt 2)) */
  GEMM_ACT_GELU_TANH = 3,  /* 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))) */
  GEMM_ACT_SILU = 4        /* x / (1 + exp(-x)) */
} gemm_activation;

typedef enum {
  GEMM_PATH_AUTO = 0,   /* choose by shape */
  GEMM_PATH_1SM = 1,    /* persistent tiled kernel, 128x256 tile, one CTA per SM */
  GEMM_PATH_2SM = 2,    /* persistent tiled kernel, 256x256 tile per CTA pair */
  GEMM_PATH_SKINNY = 3  /* M <= 256: swap-AB stream-K HBM streaming of B (the tokens are MMA N).
                           AUTO, with kb = K's k-blocks (64 bf16 or 128 fp8 elements), "B large"
                           = B (N x K) of at least 32 MiB, and "parts" = the equal k-parts per
                           tile the streaming kernel would use (0 where it would take stream-K
                           ranges instead):
                           - M <= 32: SKINNY, except 1SM for kb <= 16 with 1024 <= N <= 4096;
                           - 32 < M <= 64, parts >= 1: SKINNY when B is large with parts <= 2
                             (but not for N <= 4096 with kb >= 64), or when kb >= 64 and
                             N > 4096;
                           - 64 < M <= 128: SKINNY when B is large, 1 <= parts <= 2,
                             4096 < N <= 8192, and kb >= 64 (kb >= 32 up to M = 96);
                           - otherwise 2SM when M > 128 and B is large or the 128x256 tiles
                             number more than 64, or when M <= 128, B is large, those tiles
                             fill at most half of the SMs and kb > 32; else 1SM */
} gemm_path;

/* Overrides for gemm_bf16_tn_ex (benchmarks, ablations, tests).
 * Zero-initialise and set only what is needed; 0 means "library default". */
typedef struct gemm_tn_config {
  int path;                 /* gemm_path */
  int grid;                 /* persistent grid size in CTAs (tiled paths), 0 = auto */
  int raster_group;         /* tiled paths: tiles along M per raster strip, 0 = auto */
  int skinny_grid;          /* skinny path: number of CTAs (stream-K ranges), 0 = auto */
  uint64_t wait_timeout_ns; /* device-side wait limit, 0 = default (2 s, or env GEMM_WAIT_TIMEOUT_NS) */
  int test_fault;           /* tests only: 1 = the producer of CTA 0 drops one stage's loads,
                               so the consumer's bounded wait must expire (GEMM_ERR_TIMEOUT) */
  int disable_pdl;          /* 1 = launch without programmatic dependent launch (see below) */
  int skinny_skew_kb;       /* skinny path, equal-split mode: k-blocks (of 64 bf16 or 128 fp8 elements)
                               moved to the part that finishes each tile, rounded up to whole k-groups;
                               0 = default (8, or M rounded up to 16 divided by 4 when
                               that is larger), < 0 = none */
  int scheduler;            /* tiled paths: GEMM_SCHED_* (0 = the default) */
  int skinny_bm;            /* skinny path: rows of B per tile (MMA M), 64 or 128; 0 = auto: 64 where
                               64-row tiles fit one wave and M > 32 (or M > 16 and 128-row tiles would
                               be split into 4 or more k-parts), else 128 */
  int skinny_kgroup;        /* skinny path: k-blocks per ring stage, loaded as one TMA box per operand:
                               1, 2 or 4; 0 = auto (the largest of 4, 2, 1 that leaves at least 3
                               ring stages and does not exceed K's k-blocks; 1 for 128-row tiles
                               with more than 64 tokens).  Values
                               above 1 apply only when K is a whole number of k-blocks (64 bf16 or
                               128 fp8 elements); otherwise the path uses 1 */
  int tiled_k_parts;        /* tiled paths, single problem, static scheduler: k-parts per tile, 0..4;
                               0 = auto (4 when the tiles times 4 fit one round of clusters and K holds
                               at least 64 k-blocks, else 2 when the tiles times 2 fit and K holds at
                               least 128, else 1), 1 = no split.  Capped at launch
                               so that every part has a co-resident cluster and at K's k-blocks;
                               ignored with CLC or a grid override.  The fused-epilogue calls
                               (gemm_bf16_tn_bias_act, gemm_fp8_tn_bias_act), which take no
                               config, keep the automatic choice only when it is four parts
                               and K holds at least 128 k-blocks, and run unsplit otherwise.
                               Inside a stream capture that
                               would have to grow the stream's split workspace, the call runs
                               unsplit (the skinny path returns an error there instead) */
  int l2_hints;             /* tiled paths, single problem: L2 eviction priorities of the kernel's
                               copies, a sum of 1 (A loads evict-last: A rows are re-read by every
                               tile of their raster strip), 2 (B loads evict-first) and 4 (D stores
                               evict-first); 0 = library default, -1 = none */
  int cluster_pref;         /* 2-SM path, static scheduler, single problem: preferred cluster size,
                               4 or 8 CTAs (two or four pairs), with pairs (2 CTAs) as the fallback
                               where a cluster of SMs has no room for the larger size; 0 = pairs only.
                               Applied only when it divides the grid */
  int b_static;             /* skinny path: 1 = the caller promises that no work still running on the
                               GPU when this call starts writes B (B holds weights, written long
                               before); the kernel then loads its first ring of B before it waits for
                               the preceding kernel on the stream to finish, so that the weight
                               stream starts during that kernel's tail.  A, C and D keep the
                               stream order.  0 = B is loaded only after that wait */
  int skinny_pair;          /* skinny path: 2 = the pair form, clusters of two CTAs on tiles of 256 rows
                               of B (cta_group::2 MMAs, M = 256) with the tokens split between the two
                               CTAs, so that each MMA instruction consumes twice the weight rows and each
                               CTA loads half the token bytes; 1 = one CTA per tile; 0 = library
                               default (one CTA per tile) */
  int tail_slices;          /* tiled paths, single problem, static scheduler, no k-split: the tiles of
                               the last, partial round of the persistent grid (all tiles when they
                               fill less than one round) are each computed as 2 or 4 slices of
                               128 or 64 columns, one cluster per slice, so that the round uses
                               more of the GPU; 0 = auto (when the tiles fill less than one
                               round: the most slices, up to 4, that still fit it), 1 = none,
                               2 or 4 = that many where the round's tiles times the count fit one
                               round, at any number of rounds, else none */
} gemm_tn_config;

/* Tile schedulers of the tiled paths.
 * STATIC: a persistent grid of as many CTAs (pairs) as fit on the GPU at
 *   once; CTA c takes tiles c, c + grid, c + 2 grid, ...
 * CLC: one CTA (pair) per tile is launched; each running CTA, while it works
 *   on a tile, asks the hardware (cluster launch control) to cancel a CTA
 *   that has not started yet and then takes that CTA's tile.  CTAs stay
 *   resident as long as there is work, as in STATIC, but the split of tiles
 *   follows the SMs actually available (other kernels on the GPU, uneven
 *   tiles).  This is the dynamic persistent scheduling with cluster launch
 *   control that the SemiAnalysis Blackwell page lists among the new
 *   features ("Blackwell architecture features"). */
typedef enum { GEMM_SCHED_DEFAULT = 0, GEMM_SCHED_STATIC = 1, GEMM_SCHED_CLC = 2 } gemm_scheduler;

/* What the last successful launch on this host thread ran. */
typedef struct gemm_launch_info {
  int path;          /* gemm_path actually used (0 if no launch) */
  int grid;          /* CTAs launched */
  int cluster;       /* CTAs per cluster */
  int block;         /* threads per CTA */
  int tile_m;        /* output rows per tile (pair tile for the 2-SM path; skinny: rows of B, 64 or 128) */
  int tile_n;        /* output columns per tile (skinny: padded M) */
  int stages;        /* shared-memory ring depth */
  int smem_bytes;    /* dynamic shared memory per CTA */
  const char *kernel;/* kernel name (static string) */
  int scheduler;     /* tiled paths: GEMM_SCHED_STATIC or GEMM_SCHED_CLC; 0 otherwise */
  int k_parts;       /* k-parts per tile: tiled split (1 = none) or skinny equal split; 0 = skinny
                        stream-K ranges */
  int cluster_pref;  /* preferred cluster size requested for the launch (gemm_tn_config.cluster_pref),
                        0 = none */
  int tail_slices;   /* tiled paths: slices per tile of the last round (1 = none) */
} gemm_launch_info;

/* D = alpha * A * B^T + beta * C (see the file comment for every argument).
 * Returns a gemm_status. */
int gemm_bf16_tn(int64_t M, int64_t N, int64_t K,
                 const void *A, int64_t lda,
                 const void *B, int64_t ldb,
                 const void *C, int64_t ldc,
                 void *D, int64_t ldd,
                 float alpha, float beta, int out_dtype, void *stream);

/* Same operation with explicit overrides; cfg may be NULL (= gemm_bf16_tn).
 * A forced path that cannot run the shape returns GEMM_ERR_NOT_IMPLEMENTED
 * (GEMM_PATH_SKINNY needs 1 <= M <= 256 and K > 0). */
int gemm_bf16_tn_ex(int64_t M, int64_t N, int64_t K,
                    const void *A, int64_t lda,
                    const void *B, int64_t ldb,
                    const void *C, int64_t ldc,
                    void *D, int64_t ldd,
                    float alpha, float beta, int out_dtype, void *stream,
                    const gemm_tn_config *cfg);

/* Fused epilogue for MLP layers:
 *
 *     D = act(alpha * A * B^T + beta * C + bias)
 *
 * bias holds N values (one per output column, i.e. per row of B), in bf16
 * (bias_dtype 0) or fp32 (bias_dtype 1), device memory, aligned to its
 * element size; NULL means no bias.  activation is a gemm_activation; it is
 * evaluated in fp32 before the single rounding to out_dtype.  Every other
 * argument, and the error behaviour, are those of gemm_bf16_tn.  It fuses
 * the step after the GEMM in an MLP up-projection (the epilogue fusion the
 * H100 Nsight Compute page lists among GEMM optimisations, section 7). */
int gemm_bf16_tn_bias_act(int64_t M, int64_t N, int64_t K,
                          const void *A, int64_t lda,
                          const void *B, int64_t ldb,
                          const void *C, int64_t ldc,
                          void *D, int64_t ldd,
                          float alpha, float beta, int out_dtype,
                          const void *bias, int bias_dtype, int activation, void *stream);

/* FP8 TN GEMM with per-tensor scales:
 *
 *     D = alpha * (scale_a * scale_b) * A * B^T + beta * C
 *
 * A (M x K) and B (N x K) hold one-byte fp8 values of the same format
 * (fp8_format: GEMM_FP8_E4M3 or GEMM_FP8_E5M2), K contiguous; lda and ldb
 * count elements (bytes) and must be multiples of 16.  Products accumulate in
 * fp32 on the tensor cores (tcgen05.mma kind::f8f6f4, twice the bf16 rate);
 * C, D, out_dtype, the paths and the error behaviour are those of
 * gemm_bf16_tn.  FP8 with per-tensor scaling is the reduced-precision
 * variant the Ampere-to-Hopper page discusses for Ada and Hopper (sections on
 * FP8 and the Transformer Engine); it halves the bytes a decode GEMM
 * streams. */
int gemm_fp8_tn(int64_t M, int64_t N, int64_t K,
                const void *A, int64_t lda,
                const void *B, int64_t ldb,
                int fp8_format, float scale_a, float scale_b,
                const void *C, int64_t ldc,
                void *D, int64_t ldd,
                float alpha, float beta, int out_dtype, void *stream);

/* FP8 TN GEMM with the fused epilogue of gemm_bf16_tn_bias_act:
 *
 *     D = act(alpha * (scale_a * scale_b) * A * B^T + beta * C + bias[n])
 *
 * Operands and scales as gemm_fp8_tn; bias, bias_dtype and activation as
 * gemm_bf16_tn_bias_act.  The fp8 MLP up-projection with its bias and
 * activation in one pass (the FP8 variant of the Ampere-to-Hopper page and
 * the epilogue fusion of the H100 Nsight Compute page, section 7). */
int gemm_fp8_tn_bias_act(int64_t M, int64_t N, int64_t K,
                         const void *A, int64_t lda,
                         const void *B, int64_t ldb,
                         int fp8_format, float scale_a, float scale_b,
                         const void *C, int64_t ldc,
                         void *D, int64_t ldd,
                         float alpha, float beta, int out_dtype,
                         const void *bias, int bias_dtype, int activation, void *stream);

/* What a call would run, computed on the host without any device access:
 * for capacity planning, and so that the automatic choices can be tested
 * without a GPU.  The fields describe the path and, for the skinny path, its
 * geometry and work split; gemm_last_launch_info reports the same values
 * after a real launch. */
typedef struct gemm_plan_info {
  int path;           /* gemm_path the call would take (0 if M or N is 0: no launch) */
  int tile_m;         /* skinny: rows of B per tile (64 or 128); tiled: 128 (1SM) or 256 (2SM pair) */
  int tile_n;         /* skinny: M rounded up to 16 (MMA N); tiled: 256 */
  int skinny_kgroup;  /* skinny: k-blocks per ring stage (one TMA box per operand); else 0 */
  int skinny_stages;  /* skinny: ring stages; else 0 */
  int skinny_grid;    /* skinny: CTAs; else 0 */
  int k_parts;        /* k-parts per tile: tiled split (1 = none; capped at launch to co-resident
                         clusters) or skinny equal split; 0 = skinny stream-K ranges */
  int skinny_skew;    /* skinny, equal split: k-groups moved to the part that finishes each tile */
  int tail_slices;    /* tiled: slices per tile of the last round (gemm_tn_config.tail_slices; 1 = none) */
} gemm_plan_info;

/* Plan D = A * B^T for M x N x K on a GPU with num_sms SMs (152 on a
 * GB300), with bf16 (fp8_inputs = 0) or fp8 (fp8_inputs = 1) operands and
 * the overrides in cfg (may be NULL).  Writes *out and returns GEMM_OK;
 * GEMM_ERR_INVALID_VALUE for negative sizes, num_sms < 1, out == NULL or an
 * invalid cfg; GEMM_ERR_NOT_IMPLEMENTED where the launch would refuse the
 * forced path. */
int gemm_plan(int64_t M, int64_t N, int64_t K, int fp8_inputs, int num_sms, const gemm_tn_config *cfg,
              gemm_plan_info *out);

/* gemm_fp8_tn with explicit overrides (gemm_tn_config, as for
 * gemm_bf16_tn_ex); cfg may be NULL (= gemm_fp8_tn).  Skew and k-groups count
 * k-blocks of 128 fp8 elements. */
int gemm_fp8_tn_ex(int64_t M, int64_t N, int64_t K,
                   const void *A, int64_t lda,
                   const void *B, int64_t ldb,
                   int fp8_format, float scale_a, float scale_b,
                   const void *C, int64_t ldc,
                   void *D, int64_t ldd,
                   float alpha, float beta, int out_dtype, void *stream,
                   const gemm_tn_config *cfg);

/* One GEMM of a grouped call: D = alpha * A * B^T + beta * C with this
 * problem's own sizes, pointers and leading dimensions (the rules of
 * gemm_bf16_tn apply to each; M or N = 0 makes it a no-op). */
typedef struct gemm_problem {
  int64_t M, N, K;
  const void *A; int64_t lda;
  const void *B; int64_t ldb;
  const void *C; int64_t ldc;
  void *D; int64_t ldd;
} gemm_problem;

/* Grouped GEMM: num_problems independent BF16 TN GEMMs of any shapes,
 * sharing alpha, beta and out_dtype, run by the tiled kernels over one linear
 * order of all the problems' tiles, so that many small GEMMs fill the GPU
 * together instead of one launch each.  Grouping, batching and persistent
 * kernels are the remedies the Ampere-to-Hopper page lists for small GEMMs
 * that cannot fill the GPU ("why some operators improve a lot and others
 * hardly at all").
 *
 * `problems` is a host array, read during the call only.  Up to 56 non-empty
 * problems go into one launch (their tensor maps travel in the kernel's
 * parameters); larger groups take several launches on `stream`, which may
 * run at the same time, so the problems must be independent: no problem's D
 * may overlap another problem's A, B, C or D.  Pair tiles
 * (256 x 256) are used if some problem has M > 128 and the problems need
 * more 128 x 256 tiles than the GPU has SMs, else 128 x 256 tiles; M <=
 * 64 problems run on the tiled kernels too.  Errors: the codes of
 * gemm_bf16_tn, with the failing problem's index in gemm_last_error_string;
 * nothing is launched if any problem is invalid. */
int gemm_bf16_tn_grouped(int num_problems, const gemm_problem *problems,
                         float alpha, float beta, int out_dtype, void *stream);

/* Strided batched GEMM: for b in [0, batch),
 *   D_b = alpha * A_b * B_b^T + beta * C_b,  X_b = X + b * stride_x
 * (strides in elements), all problems M x N x K.  One launch reads every
 * problem through 3D tensor maps whose third coordinate is b.  Each stride
 * must be at least rows * ld of its matrix (problems do not overlap), and a
 * multiple of 16 bytes; strides are ignored when batch == 1.  Otherwise the
 * rules and errors of gemm_bf16_tn apply to every problem. */
int gemm_bf16_tn_batched(int64_t batch, int64_t M, int64_t N, int64_t K,
                         const void *A, int64_t lda, int64_t stride_a,
                         const void *B, int64_t ldb, int64_t stride_b,
                         const void *C, int64_t ldc, int64_t stride_c,
                         void *D, int64_t ldd, int64_t stride_d,
                         float alpha, float beta, int out_dtype, void *stream);

/* Synchronises `stream`, then returns and clears the current device's status
 * word: GEMM_OK, or GEMM_ERR_TIMEOUT if a kernel's bounded wait gave up since
 * the last call (its output is then undefined).  A CUDA error from the
 * synchronisation is returned as GEMM_ERR_CUDA. */
int gemm_get_status(void *stream);

/* Detail word of the last device error: (role << 24) | block index, with
 * role 1 = producer, 2 = MMA issuer, 3 = epilogue, 4 = skinny-path wait for
 * the other parts of a split tile.  0 if none. */
int gemm_get_status_detail(void);

/* Human-readable text for the last error on this host thread ("" if none). */
const char *gemm_last_error_string(void);

/* Launch details of the last successful call on this host thread. */
int gemm_last_launch_info(gemm_launch_info *out);

/* Frees library-owned device memory (skinny workspaces).  Call only when no
 * GEMM is in flight. */
void gemm_shutdown(void);

/* Library version, major * 10000 + minor * 100 + patch. */
int gemm_version(void);

/* Measurement kernel: the read ceiling of the skinny path's weight stream.
 *
 * Follows the Ampere-to-Hopper page, section "not reaching peak": a kernel
 * is judged against ceilings measured on the same machine.  Reads the
 * rows x row_bytes bytes at src (row-major, rows contiguous, device memory
 * owned by the caller) through TMA boxes of box_rows rows x kgroup
 * consecutive 128-byte chunks, as the skinny kernel loads its B operand,
 * into a shared-memory ring of up to 216 KiB (at most 64 boxes) per CTA, and discards them.
 * grid CTAs (0 = one per SM) each stream a contiguous range of boxes, in the
 * skinny kernel's order (k-chunks fastest within a tile of box_rows rows).
 * Nothing is written to global memory.
 *
 * box_rows is 32, 64, 128 or 256; kgroup 1, 2 or 4; rows a multiple of
 * box_rows; row_bytes a multiple of 128 * kgroup; src 16-byte aligned.
 * Otherwise GEMM_ERR_INVALID_VALUE or GEMM_ERR_MISALIGNED.  Asynchronous on
 * stream, launched with programmatic stream serialisation like the GEMM
 * kernels; device-side waits are bounded like theirs (gemm_get_status). */
int gemm_stream_read(const void *src, int64_t rows, int64_t row_bytes, int box_rows, int kgroup, int grid,
                     void *stream);

/* Measurement kernel: the tcgen05.mma rate at the skinny path's shapes.
 *
 * grid CTAs (cta_group = 1) or grid / 2 CTA pairs (cta_group = 2) each issue
 * reps groups of four tcgen05.mma instructions (kind::f16 with bf16 operands,
 * or kind::f8f6f4 with e4m3 when fp8 != 0; K = one 128-byte atom per group)
 * with M = 128 rows per CTA and N = n columns (the pair splits the n rows of
 * its second operand between its CTAs), on zeroed shared-memory operands,
 * accumulating in Tensor Memory; then they commit and wait.  out_ns (device
 * memory, two unsigned 64-bit words, owned by the caller) receives from the
 * first CTA: [0] the nanoseconds from the first issue to the completion of
 * all MMAs, [1] those of the issue loop alone.  It is the per-instruction
 * cost the skinny kernel pays for every stage it consumes (the SemiAnalysis
 * Blackwell page, section "5th-generation tensor core MMA", measures the
 * same instruction's throughput against its shape).
 *
 * n is a multiple of 16 in [16, 256], cta_group 1 or 2, 1 <= reps <= 2^24,
 * grid a multiple of cta_group up to 1024; else GEMM_ERR_INVALID_VALUE.
 * Asynchronous on stream; waits are bounded (gemm_get_status). */
int gemm_mma_rate(int n, int cta_group, int fp8, int reps, int grid, unsigned long long *out_ns, void *stream);

/* The skinny path (1 <= M <= 64) without any allocation at call time.
 *
 * The pages have no counterpart to this entry point; it exists for callers
 * that cannot allocate device memory when they call a GEMM: code that runs
 * under a memory budget reserved up front (a serving process that owns all
 * of HBM through its own pool), latency-critical code that cannot afford
 * cudaMalloc's implicit device synchronisation, and plug-ins whose host
 * framework owns every allocation.  gemm_bf16_tn allocates the skinny
 * path's workspace on first use; this entry point calls no cudaMalloc,
 * cudaFree or other allocating routine.
 *
 * Same operation and argument rules as gemm_bf16_tn, restricted to
 * 1 <= M <= 64, 1 <= N <= 131072 and K >= 1; larger sizes return
 * GEMM_ERR_INVALID_VALUE (text in gemm_last_error_string).  Its scratch (fp32
 * partial sums and arrival counters, about 10 MiB) is a fixed device array
 * inside the library, held by every device that loads the library until the
 * process exits.  The first call on a device looks up that array's device
 * address (cudaGetSymbolAddress) with the device current; make that first
 * call before any stream capture.  Every call on a device shares the array:
 * each call clears the counters on its stream before its kernel, so calls
 * ordered in one stream are safe, but calls whose kernels overlap on the GPU
 * (unordered streams) race and give wrong results.  Device-side waits give
 * up after GEMM_WAIT_TIMEOUT_NS nanoseconds (2 s when unset), as those of
 * gemm_bf16_tn do; timeouts are reported by gemm_get_status. */
int gemm_bf16_tn_skinny_noalloc(int64_t M, int64_t N, int64_t K,
                                const void *A, int64_t lda,
                                const void *B, int64_t ldb,
                                const void *C, int64_t ldc,
                                void *D, int64_t ldd,
                                float alpha, float beta, int out_dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_TN_H_ */
