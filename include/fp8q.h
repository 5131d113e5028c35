/*
 * fp8q -- FP8 scaled quantization and scaled GEMM for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libfp8q.so.  Every entry point takes plain pointers and sizes; a
 * "device" pointer is CUDA global memory of the current device, a "host"
 * pointer is ordinary process memory.  `stream` is a cudaStream_t passed as
 * void* (NULL = the legacy default stream).  All work is enqueued on that
 * stream and returns without synchronising, except where a function says
 * otherwise.  Host-side argument errors are returned before anything is
 * enqueued; FP8Q_ERR_CUDA reports a failed launch or CUDA call.
 *
 * The method is FP8 training's quantize-then-scaled-GEMM as described by the
 * web pages "2025 FP8 quantized-training guide" (blog.gitcode.com; cited as
 * [guide]), bjdmk.com.cn/news/5220490 ([essay]) and "mastering FP8 LLM
 * training 1.5x speedup" (nmedialink.com; [nemo]).
 *
 * Number formats ([guide] sec. 1.1; [essay] sec. 2):
 *   FP8Q_E4M3  1 sign, 4 exponent (bias 7), 3 mantissa bits; max 448,
 *              subnormals down to 2^-9, no Inf, NaN = S.1111.111
 *              (torch.float8_e4m3fn).
 *   FP8Q_E5M2  1/5/2 bits, bias 15; max 57344, subnormals down to 2^-16
 *              (torch.float8_e5m2).
 * The cast is saturating round-to-nearest-even: ties go to the even code,
 * finite overflow and +-Inf clamp to +-max, NaN stays NaN.
 *
 * Layouts: every matrix is row-major.  x is bf16 [rows][cols].  The row-wise
 * copy is uint8 [rows][cols]; the column-wise copy is the quantized transpose,
 * uint8 [cols][rows].  Each copy carries scales in the layout of its own
 * logical matrix (a copy of logical shape [R][C] with blocks along C):
 *
 *   kind                     scale buffer of a copy [R][C]            dequant
 *   PERTENSOR_CURRENT/DELAYED none (scalar *scale / *scale_inv)         s_inv
 *   BLOCK_1x128              fp32 [ceil(C/128)][Rp], Rp = R up to 128, d
 *                            pad rows 1.0 (K-block-major)
 *   BLOCK_128x128            fp32 [ceil(R/128)][ceil(C/128)]           d
 *   MXFP8_1x32               E8M0 bytes in 128x4 tiles: tile (i, j) of  2^(code-127)
 *                            512 B at (i * ceil(C/128) + j) * 512 holds
 *                            rows 128i.., scale columns 4j..; row r,
 *                            column k at (r%32)*16 + (r%128/32)*4 + k%4;
 *                            pad entries 127
 *   PERCHANNEL_CURRENT       fp32 [Rp], Rp = R up to 128: row r's       s_inv[r]
 *                            fp32(1 / s_r); pad entries 1.0 (the rule
 *                            for an all-zero row)
 *   BLOCK_GENERIC 1 x b      fp32 [ceil(C/b)][Rp], as BLOCK_1x128       d
 *   BLOCK_GENERIC b x b      fp32 [ceil(R/b)][ceil(C/b)], as 128x128    d
 *
 * The column-wise copy of BLOCK_1x128, MXFP8_1x32, PERCHANNEL_CURRENT and a
 * 1 x b BLOCK_GENERIC re-quantizes x^T with its blocks along the rows of x
 * (the contraction dimension of the wgrad GEMM; per channel: one factor per
 * column of x); for per-tensor, 128x128 and b x b kinds it is the byte
 * transpose of the row-wise copy with the same (transposed) scales.
 */
#ifndef FP8Q_H
#define FP8Q_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8Q_API __attribute__((visibility("default")))
#else
#define FP8Q_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8Q_OK = 0,
    FP8Q_ERR_ARG = 1,          /* NULL pointer, bad enum, bad flag combination */
    FP8Q_ERR_SHAPE = 2,        /* negative or inconsistent sizes, size limits */
    FP8Q_ERR_ALIGN = 3,        /* pointer or row pitch not 16-byte aligned */
    FP8Q_ERR_DTYPE = 4,        /* format / recipe combination not allowed */
    FP8Q_ERR_UNSUPPORTED = 5,  /* valid request this library does not implement */
    FP8Q_ERR_CUDA = 6,         /* a CUDA call or kernel launch failed */
    FP8Q_ERR_TIMEOUT = 7,      /* a bounded device wait gave up (see fp8q_device_errors) */
    FP8Q_WARN_NONFINITE = 8    /* reserved: nonfinite inputs are reported via counters */
} fp8q_status;

typedef enum { FP8Q_E4M3 = 0, FP8Q_E5M2 = 1 } fp8q_format;

/* Recipes: [guide] sec. 2.1-2.3, [nemo] scaling strategies 1-4. */
typedef enum {
    FP8Q_PERTENSOR_CURRENT = 0,  /* s = fmax / amax(x) of this tensor; q = sat_rne(x * s) */
    FP8Q_PERTENSOR_DELAYED = 1,  /* s from the max of an amax history of past steps */
    FP8Q_BLOCK_1x128 = 2,        /* d = amax / fmax per 1x128 block; q = sat_rne(x / d) */
    FP8Q_BLOCK_128x128 = 3,      /* same per 128x128 tile (weights) */
    FP8Q_MXFP8_1x32 = 4,         /* e = floor(log2 amax) - emax_elem per 1x32 block,
                                    E8M0 code e + 127, q = sat_rne(x * 2^-e) */
    FP8Q_PERCHANNEL_CURRENT = 5, /* [nemo] Figure 1 (channel-wise scaling, one factor
                                    per row / column): the per-tensor current rule
                                    per row of the copy, s_r = fmax / amax(row r),
                                    q = sat_rne(x * s_r) */
    FP8Q_BLOCK_GENERIC = 6       /* [nemo] scaling strategy 3 (sub-channel blocks of
                                    user-set dimensions): the blockwise rule of
                                    BLOCK_1x128 on blocks of block_rows x block_cols,
                                    either 1 x b or b x b with b in {32, 64, 128, 256} */
} fp8q_recipe_kind;

typedef struct {
    int kind;           /* fp8q_recipe_kind */
    int fmt;            /* fp8q_format of the quantized data */
    int want_rowwise;   /* 1: write data_row (+ scale_row) */
    int want_colwise;   /* 1: write data_col (+ scale_col) */
    int block_rows;     /* BLOCK_GENERIC only: 1 or b */
    int block_cols;     /* BLOCK_GENERIC only: b in {32, 64, 128, 256} */
} fp8q_recipe;

/*
 * Output of one quantize call.  All pointers are device memory owned by the
 * caller; unused ones may be NULL.
 *   data_row   uint8 [rows][cols]      (want_rowwise)
 *   data_col   uint8 [cols][rows]      (want_colwise)
 *   scale_row  scales of data_row      (block / MX kinds; size: fp8q_scale_bytes)
 *   scale_col  scales of data_col
 *   amax       fp32[1]  per-tensor kinds: max |x| over finite elements
 *   scale      fp32[1]  per-tensor kinds: the multiplier s the cast used
 *   scale_inv  fp32[1]  per-tensor kinds: fp32(1 / s), the GEMM's dequant scale
 *   counters   uint64[3], always required: [0] elements of the row-wise cast
 *              whose scaled fp32 value exceeded fmax (saturated), [1] the same
 *              for a re-quantized column-wise copy (0 when the column-wise
 *              copy is a byte transpose), [2] NaN / Inf elements of x.
 * rows / cols / fmt / kind (and, for BLOCK_GENERIC, block_rows / block_cols)
 * are filled in by fp8q_quantize and read by fp8q_scaled_gemm.
 */
typedef struct {
    void* data_row;
    void* data_col;
    void* scale_row;
    void* scale_col;
    float* amax;
    float* scale;
    float* scale_inv;
    unsigned long long* counters;
    int64_t rows;
    int64_t cols;
    int fmt;
    int kind;
    int block_rows;   /* BLOCK_GENERIC: the recipe's block shape (else 0) */
    int block_cols;
} fp8q_tensor;

/* Opaque per-tensor delayed-scaling state, owned by the library: an amax ring
 * of history_len fp32 entries, its head index, and the current s / s_inv, all
 * in device memory of the device current at creation. */
typedef struct fp8q_delayed_state fp8q_delayed_state;

/* Version of this ABI (major * 100 + minor). */
FP8Q_API int fp8q_version(void);

/* Human-readable name of a status code (static string). */
FP8Q_API const char* fp8q_status_str(fp8q_status s);

/*
 * Bytes of the scale buffers of a quantize call with this recipe and x shape
 * [rows][cols]: *row_bytes for scale_row, *col_bytes for scale_col (0 for
 * per-tensor kinds).  Either output pointer may be NULL.  Host only.  The
 * sizes are those of the layouts above, one scale per block of [guide]
 * sec. 2.2-2.3 or per channel of [nemo] Figure 1.
 */
FP8Q_API fp8q_status fp8q_scale_bytes(const fp8q_recipe* recipe, int64_t rows, int64_t cols,
                             size_t* row_bytes, size_t* col_bytes);

/*
 * Quantize x (device, bf16 [rows][cols]) with `recipe` into `out` (host
 * struct whose pointers are device buffers).  Sources: [guide] sec. 2.1
 * (per-tensor current / delayed), 2.2 (blockwise), 2.3 (MXFP8); [nemo]
 * strategies 1-4; [essay] sec. 3.3 (DelayedScaling margin / interval 1).
 *
 * Constraints: cols % 16 == 0; rows % 16 == 0 when want_colwise; x and every
 * data / scale pointer 16-byte aligned; rows * cols < 2^40.  rows or cols 0
 * is allowed (nothing but the per-tensor scalars and counters is written).
 *
 * Per-tensor current: amax over x first, then s = fmax / amax (amax 0 -> 1,
 * +Inf -> FLT_MAX), scale_inv = 1 / s.  Per-tensor delayed: `st` (required,
 * same fmt) supplies s; the call writes amax / scale / scale_inv / counters,
 * then records amax in st's history and derives the next step's scale
 * (st is left unchanged when x held a NaN / Inf).  Blockwise d = amax / fmax
 * (amax 0 -> 1).  Per-channel current: a pass over x first takes every
 * row's and every column's amax (into the scale buffers, as scratch), then
 * s = fmax / amax per row (row-wise copy) or per column (column-wise copy)
 * as for per-tensor current, and the scale buffers end holding fp32(1 / s).
 * Amax always excludes NaN / Inf.  Counters are overwritten.  BLOCK_GENERIC:
 * recipe->block_rows x block_cols must be 1 x b or b x b, b in {32, 64, 128,
 * 256} (else FP8Q_ERR_UNSUPPORTED); 1 x 128 and 128 x 128 run exactly as
 * BLOCK_1x128 and BLOCK_128x128; b = 32 and 64 take one pass over x; b = 256
 * takes a pass over x that leaves every block's amax in the scale buffers (as
 * scratch), then the cast.  The scale buffers end holding d.
 */
FP8Q_API fp8q_status fp8q_quantize(const fp8q_recipe* recipe, const void* x, int64_t rows, int64_t cols,
                          fp8q_delayed_state* st, fp8q_tensor* out, void* stream);

/*
 * Quantizes rows row0 .. row0 + rows - 1 of a tensor of total_rows x cols
 * whose rows arrive in blocks (a weight streamed in from the host, say): x is
 * the block (device bf16 [rows][cols]); out describes the WHOLE tensor's
 * buffers as fp8q_quantize would fill them for [total_rows][cols], and the
 * call writes the block's part: its rows of data_row, its columns of data_col,
 * and the scales of its 128-row groups.  Quantizing every block once gives
 * exactly what fp8q_quantize on the whole tensor writes, because these
 * recipes' scales never span two 128-row groups (no counterpart on the pages;
 * their block recipes read tile by tile).  Kinds: BLOCK_1x128, BLOCK_128x128,
 * MXFP8_1x32 (either copy), PERCHANNEL_CURRENT (row-wise copy only); others
 * FP8Q_ERR_DTYPE.  row0 % 128 == 0, and rows % 128 == 0 unless the block
 * ends the tensor; total_rows % 16 == 0 with a column copy; cols % 16 == 0.
 * Counters are ADDED to (zero them before the first block); out->rows is set
 * to total_rows.
 */
FP8Q_API fp8q_status fp8q_quantize_rows(const fp8q_recipe* recipe, const void* x, int64_t row0, int64_t rows,
                               int64_t total_rows, int64_t cols, fp8q_tensor* out, void* stream);

/*
 * Several quantize calls as one: the same outputs as fp8q_quantize on each
 * job in order (no counterpart on the pages; a launch arrangement), but the
 * jobs' tile passes run side by side, their resident CTAs shared out in
 * proportion to each job's 128x128 tiles, so that a small tensor does not
 * leave SMs idle while its kernel fills and drains (the Llama-3-8B
 * up-projection quantizes X of 1024 tiles and W of 3584).  Every job is
 * checked as fp8q_quantize checks its arguments before anything is enqueued;
 * 1 <= n <= FP8Q_MULTI_MAX (n = 0 does nothing); no two jobs may share an
 * output struct or a delayed state.  The work is ordered after what `stream`
 * holds and before what is enqueued on it later: the call records an event on
 * `stream`, runs each job on a library-owned stream of the current device
 * that waits for it, and makes `stream` wait for each job's end (so a CUDA
 * graph capture of `stream` takes the fork and join in).  Calls from several
 * host threads are serialised.
 */
#define FP8Q_MULTI_MAX 16
typedef struct {
    fp8q_recipe recipe;
    const void* x;             /* bf16 [rows][cols], device */
    int64_t rows, cols;
    fp8q_delayed_state* state; /* delayed recipe only, else NULL */
    fp8q_tensor* out;          /* host struct of device buffers, as for fp8q_quantize */
} fp8q_quantize_job;
FP8Q_API fp8q_status fp8q_quantize_multi(const fp8q_quantize_job* jobs, int n, void* stream);

/*
 * Creates a delayed-scaling state on the current device: history_len in
 * [1, 4096] (the [guide] sec. 2.1 history; 16 by default in the tests),
 * margin in [0, 64] (s = fmax / max(history) * 2^-margin; [essay] sec. 3.3
 * uses 0; an s below the smallest normal fp32, which a large margin on a
 * large history maximum can give, is raised to it so that scale_inv = 1 / s
 * stays finite).  The history starts all zero, so the first step casts with
 * s = 1.  Allocates device memory (cudaMalloc) and synchronises.  *out
 * receives the handle; free it with fp8q_delayed_destroy.
 */
FP8Q_API fp8q_status fp8q_delayed_create(int history_len, int fmt, int margin, fp8q_delayed_state** out);

/*
 * Records amax (device fp32[1]) as this step's amax and derives the next
 * scale, on `stream`.  nonfinite (device uint64[1], may be NULL) nonzero
 * leaves the state unchanged.  fp8q_quantize does this itself for the
 * delayed kind; this entry point serves callers that combine amax values
 * from elsewhere (e.g. a max over data-parallel replicas).  FP8Q_ERR_ARG when
 * the current device is not the one the state was created on.
 */
FP8Q_API fp8q_status fp8q_delayed_update(fp8q_delayed_state* st, const float* amax,
                                const unsigned long long* nonfinite, void* stream);

/*
 * Checkpoint: copies the state to host memory.  hist (host fp32
 * [history_len]), head, scale and scale_inv may each be NULL.  Synchronises
 * the device.  (The state is [guide] sec. 2.1's history; saving and restoring
 * it has no counterpart on the pages.)  FP8Q_ERR_ARG when the current device
 * is not the state's.
 */
FP8Q_API fp8q_status fp8q_delayed_get(const fp8q_delayed_state* st, float* hist, int* head,
                             float* scale, float* scale_inv);

/* Restore: overwrites history (host fp32 [history_len]), head, and the scale
 * pair from host memory.  Synchronises the device.  FP8Q_ERR_ARG when the
 * current device is not the state's. */
FP8Q_API fp8q_status fp8q_delayed_set(fp8q_delayed_state* st, const float* hist, int head,
                             float scale, float scale_inv);

/* History length of a state (host). */
FP8Q_API int fp8q_delayed_history_len(const fp8q_delayed_state* st);

/* Frees a state (NULL is ignored). */
FP8Q_API void fp8q_delayed_destroy(fp8q_delayed_state* st);

/*
 * Scaled FP8 GEMM, D[M][N] = A_q . B_q^T with fp32 accumulation ([guide]
 * sec. 3.1: the fprop, dgrad and wgrad GEMMs take quantized inputs and keep
 * BF16/FP32 outputs).  A_q is A's row-wise copy (a_use_col = 0, logical
 * [A->rows][A->cols]) or column-wise copy (a_use_col = 1, logical
 * [A->cols][A->rows]) and must be [M][K]; B_q likewise [N][K].  With a
 * layer's X [T][H], W [F][H], dY [T][F]:
 *   fprop  Y  = X . W^T     : A = X row,  B = W row   (M=T, N=F, K=H)
 *   dgrad  dX = dY . W      : A = dY row, B = W col   (M=T, N=H, K=F)
 *   wgrad  dW = dY^T . X    : A = dY col, B = X col   (M=F, N=H, K=T)
 * Recipe pairs: both per-tensor (current or delayed, E4M3 / E5M2 in any
 * mix): D = s_inv_A * s_inv_B * (q_A . q_B^T).  A BLOCK_1x128 with B
 * BLOCK_128x128 or BLOCK_1x128 (E4M3 or E5M2): partial sums over each
 * 128-wide K block are scaled by d_A[m][kb] * d_B[n(/128)][kb] and summed in
 * fp32.  Both MXFP8_1x32: every 32-wide K block scaled by 2^(eA + eB) in the
 * tensor core.  Both PERCHANNEL_CURRENT: D[m][n] = fp32(s_inv_A[m] *
 * s_inv_B[n]) * (q_A . q_B^T)[m][n] (runs on the SM-pair kernel whatever
 * fp8q_gemm_set_variant selects).
 * out_dtype 0 = bf16 (RNE), 1 = fp32; D is device [M][N] row-major, 16-byte
 * aligned, N % 8 == 0.  M, N, K >= 1; K % 16 == 0.  D is fully overwritten.
 * A bounded wait inside the kernel that gives up records FP8Q_ERR_TIMEOUT in
 * the word read by fp8q_device_errors and the kernel exits early.
 */
FP8Q_API fp8q_status fp8q_scaled_gemm(const fp8q_tensor* A, int a_use_col, const fp8q_tensor* B, int b_use_col,
                             void* D, int out_dtype, int64_t M, int64_t N, int64_t K, void* stream);

/*
 * fp8q_scaled_gemm with the next quantize fused into its epilogue: the GEMM's
 * bf16 output (as fp8q_scaled_gemm would store it) is also quantized with the
 * MXFP8 1x32 recipe along its rows ([guide] sec. 2.3 and 3.1: a GEMM's output
 * is the next layer's input; [nemo] strategy 4), so that Dq->data_row,
 * Dq->scale_row and Dq->counters ([0] saturated, [1] 0, [2] NaN / Inf) equal
 * what fp8q_quantize(MXFP8_1x32, fmt, row-wise only) of that bf16 D writes.
 * With Dq->data_col non-NULL the column-wise copy is written as well (codes
 * uint8 [N][M] in Dq->data_col, blocks of 32 along M, E8M0 tiles in
 * Dq->scale_col, its saturation count in counters[1]), equal to what
 * fp8q_quantize(MXFP8_1x32, fmt, row-wise and column-wise) of D writes: the
 * copy the next wgrad reads; it needs M % 16 == 0 and Dq->scale_col.
 * D (bf16 [M][N]) may be NULL: then only the quantized output is written.
 * Dq is caller-owned: data_row uint8 [M][N], scale_row (and scale_col) of
 * fp8q_scale_bytes(MXFP8_1x32, M, N) bytes, counters uint64[3]; its rows /
 * cols / fmt / kind are filled in (amax / scale / scale_inv are not used).
 * Constraints as fp8q_scaled_gemm plus N % 32 == 0 and 16-byte aligned Dq
 * buffers.  Runs on the SM-pair kernel whatever
 * fp8q_gemm_set_variant chose.  This entry point has no counterpart on the
 * pages: they describe the quantize and the GEMM as separate steps.
 */
FP8Q_API fp8q_status fp8q_scaled_gemm_mxq(const fp8q_tensor* A, int a_use_col, const fp8q_tensor* B, int b_use_col,
                                 void* D, int fmt, fp8q_tensor* Dq, int64_t M, int64_t N, int64_t K,
                                 void* stream);

/*
 * The same fusion for either row-wise recipe the next GEMM takes: out_kind
 * FP8Q_MXFP8_1x32 (exactly fp8q_scaled_gemm_mxq) or FP8Q_BLOCK_1x128 ([guide]
 * sec. 2.2: activations and gradients in 1x128 blocks; here blocks of 128
 * columns of D).  For 1x128, Dq->data_row, Dq->scale_row (fp32
 * [ceil(N/128)][ceil(M/128) * 128], K-block-major, pads 1.0) and Dq->counters
 * equal what fp8q_quantize(BLOCK_1x128, fmt, row-wise only) of the bf16 D
 * writes; N % 16 == 0; with Dq->data_col the column-wise copy too (blocks of
 * 128 rows of one column, fp32 scales [ceil(M/128)][ceil(N/128) * 128] in
 * Dq->scale_col; M % 16 == 0), as fp8q_quantize(BLOCK_1x128, fmt, both
 * copies) writes it.  Other kinds: FP8Q_ERR_UNSUPPORTED.  Same buffers,
 * constraints and kernel otherwise.  No counterpart on the pages (a fusion of
 * two steps they describe separately).
 */
FP8Q_API fp8q_status fp8q_scaled_gemm_q(const fp8q_tensor* A, int a_use_col, const fp8q_tensor* B, int b_use_col,
                                        void* D, int out_kind, int fmt, fp8q_tensor* Dq, int64_t M, int64_t N,
                                        int64_t K, void* stream);

/*
 * Chooses the GEMM kernel for subsequent fp8q_scaled_gemm calls (process
 * wide): 0 automatic (default: SM pairs once the problem has at least 64
 * tiles of 256 x 256 and, for blockwise scales, both scale arrays are
 * 16-byte aligned; else one SM per tile), 1 always one SM per 128-row tile
 * (tcgen05.mma.cta_group::1, M = 128), 2 always SM pairs
 * (tcgen05.mma.cta_group::2, M = 256, launched as clusters of two CTAs;
 * blockwise scale arrays must then be 16-byte aligned, else the GEMM returns
 * FP8Q_ERR_ARG).  Both compute the same D up to fp32 summation order.  Host
 * only.  No counterpart on the pages: a choice between two tilings of the
 * same GEMM.
 */
FP8Q_API fp8q_status fp8q_gemm_set_variant(int variant);

/*
 * Reads and clears the library's device error words on the current device
 * (bit 0: a GEMM pipeline wait timed out, bit 1: a quantize tile-load wait
 * timed out) into *flags.  Synchronises `stream`.  Returns FP8Q_ERR_TIMEOUT
 * when a bit was set, FP8Q_OK when none was.  No counterpart on the pages:
 * the library's own failure detection.
 */
FP8Q_API fp8q_status fp8q_device_errors(unsigned int* flags, void* stream);

/*
 * Failure-detection settings (host only, process wide; no counterpart on the
 * pages).  Every wait inside the quantize tile kernel and the GEMM kernels
 * (on a pipeline stage, an accumulator, a scale tile) is bounded: past the
 * limit it sets the error word that fp8q_device_errors reads, the CTA drains
 * what it has in flight (bounded), frees its TMEM and exits, and the device
 * stays usable.  fp8q_set_wait_limit sets that limit in nanoseconds for
 * launches made afterwards (0 restores the default, one second).
 * fp8q_stall_next(n) makes the next n quantize-tile or GEMM launches run
 * stalled: their producers issue no loads, so their first pipeline waits run
 * out and the launches end through the path above (their outputs are left
 * unwritten).  It exists to test that path; n = 0 cancels.
 */
FP8Q_API fp8q_status fp8q_set_wait_limit(uint64_t ns);
FP8Q_API fp8q_status fp8q_stall_next(int n);

/*
 * The saturating RNE cast on its own ([guide] sec. 1.1 formats, the cast
 * rule stated at the top of this header): out[i] = cast(float with bit
 * pattern start + i) for i < count (device uint8 out).  Serves exhaustive
 * checks of the device conversion over all 2^32 fp32 inputs.
 */
FP8Q_API fp8q_status fp8q_cast_f32_bits(uint32_t start, uint64_t count, int fmt, void* out, void* stream);

/*
 * Self-test of the blockwise recipes' division.  The quantize kernels compute
 * x / d (d = amax / fmax, [guide] sec. 2.2) as q = RN(x * r) with r = RN(1/d),
 * then one FMA residual correction, which yields the correctly rounded
 * quotient for d in [2^-80, 2^128) and quotients in [2^-24, 2^126) (smaller d
 * takes the IEEE division; quantization's quotients never exceed
 * fmax (1 + 2^-23); below 2^-24, where the residual of a tiny x can leave the
 * normal range, every quotient encodes to an FP8 zero).  This entry point
 * compares that computation (scalar, and the two-lane form with negated
 * lanes the tile kernel runs, on x and -x) with the IEEE quotient for every finite bf16 x
 * and every d[j] (device fp32 [nd]) whose quotient is below 2^126 and writes
 * the mismatch counts to mismatches (device uint64[2]: [0] FP8 codes of
 * format fmt over all those pairs, [1] fp32 bits where the IEEE quotient is
 * at least 2^-24).  Both must be 0.
 */
FP8Q_API fp8q_status fp8q_selftest_division(const float* d, int64_t nd, int fmt, unsigned long long* mismatches,
                                            void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8Q_H */
