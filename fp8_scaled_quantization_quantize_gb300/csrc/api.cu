// C-ABI entry points of libfp8q: argument validation, scale-buffer sizing,
// the delayed-scaling state, and dispatch to the kernels.
#include <stdlib.h>
#include <string.h>

#include <atomic>

#include "fp8q_internal.cuh"

struct fp8q_delayed_state {
    fp8q::DelayedDev* dev;
    int H;
    int fmt;
    int margin;
    int device;
};

using namespace fp8q;

namespace {

constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // one second
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_stall{0};

}  // namespace

namespace fp8q {

uint64_t wait_limit_ns() { return g_wait_ns.load(std::memory_order_relaxed); }

int take_stall() {
    int n = g_stall.load(std::memory_order_relaxed);
    while (n > 0 && !g_stall.compare_exchange_weak(n, n - 1, std::memory_order_relaxed)) {
    }
    return n > 0 ? 1 : 0;
}

}  // namespace fp8q

namespace {

constexpr int64_t kMaxElems = (int64_t)1 << 40;

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool valid_fmt(int f) { return f == FP8Q_E4M3 || f == FP8Q_E5M2; }

bool valid_kind(int k) { return k >= FP8Q_PERTENSOR_CURRENT && k <= FP8Q_BLOCK_GENERIC; }

// Block shapes of the generic kind: 1 x b or b x b, b in {32, 64, 128, 256}.
bool valid_generic(int br, int bc) {
    return (bc == 32 || bc == 64 || bc == 128 || bc == 256) && (br == 1 || br == bc);
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool is_pertensor(int k) { return k == FP8Q_PERTENSOR_CURRENT || k == FP8Q_PERTENSOR_DELAYED; }

// A blockwise copy as (block rows, block cols): 1x128 / 128x128 kinds and
// the generic kind's shape; (0, 0) for other kinds.
void block_shape(const fp8q_tensor* t, int& br, int& bc) {
    br = bc = 0;
    if (t->kind == FP8Q_BLOCK_1x128) br = 1, bc = 128;
    if (t->kind == FP8Q_BLOCK_128x128) br = bc = 128;
    if (t->kind == FP8Q_BLOCK_GENERIC) br = t->block_rows, bc = t->block_cols;
}

// Recipe pairs of the scaled GEMM: both per-tensor (current / delayed in any
// mix), both MXFP8, both per-channel, or blockwise A of 1 x b blocks with B of
// 1 x b or b x b blocks (b the same: the K block of the promotion).
bool gemm_kinds_ok(const fp8q_tensor* A, const fp8q_tensor* B) {
    const int ka = A->kind, kb = B->kind;
    if (is_pertensor(ka) || is_pertensor(kb)) return is_pertensor(ka) && is_pertensor(kb);
    if (ka == FP8Q_MXFP8_1x32 || kb == FP8Q_MXFP8_1x32 || ka == FP8Q_PERCHANNEL_CURRENT ||
        kb == FP8Q_PERCHANNEL_CURRENT)
        return ka == kb;
    int abr, abc, bbr, bbc;
    block_shape(A, abr, abc);
    block_shape(B, bbr, bbc);
    return abr == 1 && abc > 0 && bbc == abc && (bbr == 1 || bbr == bbc);
}

// Scale bytes of one copy with logical shape [R][C] (blocks along C; br x bc
// blocks for the generic kind).
size_t copy_scale_bytes(int kind, int64_t R, int64_t C, int br = 0, int bc = 0) {
    switch (kind) {
        case FP8Q_BLOCK_GENERIC:
            if (br == 1) return (size_t)(cdiv(C, bc) * cdiv(R, 128) * 128) * sizeof(float);
            return (size_t)(cdiv(R, br) * cdiv(C, bc)) * sizeof(float);
        case FP8Q_BLOCK_1x128:
            return (size_t)(cdiv(C, 128) * cdiv(R, 128) * 128) * sizeof(float);
        case FP8Q_BLOCK_128x128:
            return (size_t)(cdiv(R, 128) * cdiv(C, 128)) * sizeof(float);
        case FP8Q_MXFP8_1x32:
            return (size_t)(cdiv(R, 128) * cdiv(C, 128)) * 512u;
        case FP8Q_PERCHANNEL_CURRENT:
            return (size_t)(cdiv(R, 128) * 128) * sizeof(float);
        default:
            return 0;
    }
}

// Checks one quantize call's arguments (fp8q_quantize's contract) and fills
// the kernels' arguments; writes nothing.
fp8q_status prepare_quantize(const fp8q_recipe* rc, const void* x, int64_t rows, int64_t cols,
                             const fp8q_delayed_state* st, const fp8q_tensor* out, QuantArgs& a) {
    if (!rc || !out) return FP8Q_ERR_ARG;
    if (!valid_kind(rc->kind) || !valid_fmt(rc->fmt)) return FP8Q_ERR_ARG;
    if (rc->kind == FP8Q_BLOCK_GENERIC && !valid_generic(rc->block_rows, rc->block_cols))
        return FP8Q_ERR_UNSUPPORTED;
    const bool row = rc->want_rowwise != 0, col = rc->want_colwise != 0;
    if (!row && !col) return FP8Q_ERR_ARG;
    if (rows < 0 || cols < 0) return FP8Q_ERR_SHAPE;
    if (rows > 0 && cols > 0 && rows > kMaxElems / cols) return FP8Q_ERR_SHAPE;
    if (cols % 16 != 0) return FP8Q_ERR_SHAPE;
    if (col && rows % 16 != 0) return FP8Q_ERR_SHAPE;
    const bool empty = rows == 0 || cols == 0;
    const bool per_tensor = is_pertensor(rc->kind);
    if (!out->counters) return FP8Q_ERR_ARG;
    if (((uintptr_t)out->counters & 7u) != 0) return FP8Q_ERR_ALIGN;
    if (!empty) {
        if (!x || (row && !out->data_row) || (col && !out->data_col)) return FP8Q_ERR_ARG;
        if (!aligned16(x) || (row && !aligned16(out->data_row)) || (col && !aligned16(out->data_col)))
            return FP8Q_ERR_ALIGN;
    }
    if (per_tensor) {
        if (!out->amax || !out->scale || !out->scale_inv) return FP8Q_ERR_ARG;
        if (((uintptr_t)out->amax | (uintptr_t)out->scale | (uintptr_t)out->scale_inv) & 3u) return FP8Q_ERR_ALIGN;
    } else if (!empty) {
        if ((row && !out->scale_row) || (col && !out->scale_col)) return FP8Q_ERR_ARG;
        if ((row && !aligned16(out->scale_row)) || (col && !aligned16(out->scale_col))) return FP8Q_ERR_ALIGN;
    }
    if (rc->kind == FP8Q_PERTENSOR_DELAYED) {
        if (!st) return FP8Q_ERR_ARG;
        if (st->fmt != rc->fmt) return FP8Q_ERR_DTYPE;
        int dev = -1;
        cudaGetDevice(&dev);
        if (dev != st->device) return FP8Q_ERR_ARG;
    }
    memset(&a, 0, sizeof(a));
    a.x = (const uint16_t*)x;
    a.R = rows;
    a.C = cols;
    a.q_row = row ? (uint8_t*)out->data_row : nullptr;
    a.q_col = col ? (uint8_t*)out->data_col : nullptr;
    a.s_row = row ? out->scale_row : nullptr;
    a.s_col = col ? out->scale_col : nullptr;
    a.amax = out->amax;
    a.scale = out->scale;
    a.scale_inv = out->scale_inv;
    a.counters = out->counters;
    a.st = (rc->kind == FP8Q_PERTENSOR_DELAYED && st) ? st->dev : nullptr;
    a.tiles_r = empty ? 0 : cdiv(rows, 128);
    a.tiles_c = empty ? 0 : cdiv(cols, 128);
    a.row0 = 0;  // the whole tensor
    a.R_total = rows;
    a.tiles_r_total = a.tiles_r;
    a.wait_ns = wait_limit_ns();
    a.br = rc->kind == FP8Q_BLOCK_GENERIC ? rc->block_rows : 0;
    a.bc = rc->kind == FP8Q_BLOCK_GENERIC ? rc->block_cols : 0;
    return FP8Q_OK;
}

// The two GEMM operands of D[M][N] = A_q . B_q^T from the chosen copies:
// recipes, formats and the copies' logical shapes checked, the data and the
// scales each recipe needs present and 16-byte aligned.
fp8q_status prepare_operands(const fp8q_tensor* A, int a_use_col, const fp8q_tensor* B, int b_use_col, int64_t M,
                             int64_t N, int64_t K, GemmOperand& ga, GemmOperand& gb) {
    if (!valid_kind(A->kind) || !valid_kind(B->kind) || !valid_fmt(A->fmt) || !valid_fmt(B->fmt)) return FP8Q_ERR_ARG;
    // logical shapes of the chosen copies
    const int64_t am = a_use_col ? A->cols : A->rows, ak = a_use_col ? A->rows : A->cols;
    const int64_t bn = b_use_col ? B->cols : B->rows, bk = b_use_col ? B->rows : B->cols;
    if (am != M || ak != K || bn != N || bk != K) return FP8Q_ERR_SHAPE;
    if (!gemm_kinds_ok(A, B)) return FP8Q_ERR_DTYPE;
    const bool pt = is_pertensor(A->kind);
    ga.data = (const uint8_t*)(a_use_col ? A->data_col : A->data_row);
    ga.scale = a_use_col ? A->scale_col : A->scale_row;
    ga.scale_inv = A->scale_inv;
    ga.rows = M;
    ga.kind = A->kind;
    ga.fmt = A->fmt;
    gb.data = (const uint8_t*)(b_use_col ? B->data_col : B->data_row);
    gb.scale = b_use_col ? B->scale_col : B->scale_row;
    gb.scale_inv = B->scale_inv;
    gb.rows = N;
    gb.kind = B->kind;
    gb.fmt = B->fmt;
    // blockwise operands by block shape: the specialised kinds and the
    // generic 1 x 128 / 128 x 128 shapes are the same GEMM
    int abr, abc, bbr, bbc;
    block_shape(A, abr, abc);
    block_shape(B, bbr, bbc);
    ga.kblock = gb.kblock = abc;
    if (abc > 0) {
        ga.kind = FP8Q_BLOCK_1x128;
        gb.kind = bbr == 1 ? FP8Q_BLOCK_1x128 : FP8Q_BLOCK_128x128;
    }
    if (!ga.data || !gb.data) return FP8Q_ERR_ARG;
    if (pt ? !ga.scale_inv || !gb.scale_inv : !ga.scale || !gb.scale) return FP8Q_ERR_ARG;
    if (!aligned16(ga.data) || !aligned16(gb.data)) return FP8Q_ERR_ALIGN;
    if (!pt && (!aligned16(ga.scale) || !aligned16(gb.scale))) return FP8Q_ERR_ALIGN;
    return FP8Q_OK;
}

// The state's memory and its kernels belong to the device it was created on;
// a call made while another device is current would run them there.
bool on_state_device(const fp8q_delayed_state* st) {
    int dev = -1;
    return cudaGetDevice(&dev) == cudaSuccess && dev == st->device;
}

void set_meta(const fp8q_recipe* rc, int64_t rows, int64_t cols, fp8q_tensor* out) {
    out->rows = rows;
    out->cols = cols;
    out->fmt = rc->fmt;
    out->kind = rc->kind;
    out->block_rows = rc->kind == FP8Q_BLOCK_GENERIC ? rc->block_rows : 0;
    out->block_cols = rc->kind == FP8Q_BLOCK_GENERIC ? rc->block_cols : 0;
}

}  // namespace

extern "C" {

int fp8q_version(void) { return 100; }

const char* fp8q_status_str(fp8q_status s) {
    switch (s) {
        case FP8Q_OK: return "ok";
        case FP8Q_ERR_ARG: return "invalid argument";
        case FP8Q_ERR_SHAPE: return "invalid shape";
        case FP8Q_ERR_ALIGN: return "misaligned pointer or row pitch";
        case FP8Q_ERR_DTYPE: return "format / recipe combination not allowed";
        case FP8Q_ERR_UNSUPPORTED: return "not supported by this library";
        case FP8Q_ERR_CUDA: return "CUDA error";
        case FP8Q_ERR_TIMEOUT: return "device wait timed out";
        case FP8Q_WARN_NONFINITE: return "nonfinite input";
    }
    return "unknown status";
}

fp8q_status fp8q_scale_bytes(const fp8q_recipe* rc, int64_t rows, int64_t cols, size_t* row_bytes,
                             size_t* col_bytes) {
    if (!rc || !valid_kind(rc->kind)) return FP8Q_ERR_ARG;
    if (rc->kind == FP8Q_BLOCK_GENERIC && !valid_generic(rc->block_rows, rc->block_cols))
        return FP8Q_ERR_UNSUPPORTED;
    if (rows < 0 || cols < 0) return FP8Q_ERR_SHAPE;
    const int br = rc->block_rows, bc = rc->block_cols;
    if (row_bytes) *row_bytes = rc->want_rowwise ? copy_scale_bytes(rc->kind, rows, cols, br, bc) : 0;
    if (col_bytes) *col_bytes = rc->want_colwise ? copy_scale_bytes(rc->kind, cols, rows, br, bc) : 0;
    return FP8Q_OK;
}

fp8q_status fp8q_quantize(const fp8q_recipe* rc, const void* x, int64_t rows, int64_t cols,
                          fp8q_delayed_state* st, fp8q_tensor* out, void* stream) {
    QuantArgs a;
    const fp8q_status v = prepare_quantize(rc, x, rows, cols, st, out, a);
    if (v != FP8Q_OK) return v;
    set_meta(rc, rows, cols, out);
    return launch_quantize(rc, a, st ? st->dev : nullptr, (cudaStream_t)stream);
}

fp8q_status fp8q_quantize_rows(const fp8q_recipe* rc, const void* x, int64_t row0, int64_t rows, int64_t total_rows,
                               int64_t cols, fp8q_tensor* out, void* stream) {
    if (!rc || !out) return FP8Q_ERR_ARG;
    if (is_pertensor(rc->kind) || (rc->kind == FP8Q_PERCHANNEL_CURRENT && rc->want_colwise) ||
        rc->kind == FP8Q_BLOCK_GENERIC)
        return FP8Q_ERR_DTYPE;  // their scales need the whole tensor (or whole columns / other row groups)
    if (row0 < 0 || rows < 0 || total_rows < 0 || row0 + rows > total_rows) return FP8Q_ERR_SHAPE;
    if (row0 % 128 != 0 || (rows % 128 != 0 && row0 + rows != total_rows)) return FP8Q_ERR_SHAPE;
    if (rc->want_colwise && total_rows % 16 != 0) return FP8Q_ERR_SHAPE;
    if (total_rows > 0 && cols > 0 && total_rows > kMaxElems / cols) return FP8Q_ERR_SHAPE;
    QuantArgs a;
    const fp8q_status v = prepare_quantize(rc, x, rows, cols, nullptr, out, a);
    if (v != FP8Q_OK) return v;
    set_meta(rc, total_rows, cols, out);
    if (rows == 0 || cols == 0) return FP8Q_OK;
    a.row0 = row0;
    a.R_total = total_rows;
    a.tiles_r_total = cdiv(total_rows, 128);
    a.add_counters = 1;
    return launch_quantize(rc, a, nullptr, (cudaStream_t)stream);
}

fp8q_status fp8q_quantize_multi(const fp8q_quantize_job* jobs, int n, void* stream) {
    if (n < 0 || n > FP8Q_MULTI_MAX || (n > 0 && !jobs)) return FP8Q_ERR_ARG;
    QuantArgs a[FP8Q_MULTI_MAX];
    const fp8q_recipe* rcs[FP8Q_MULTI_MAX];
    DelayedDev* sts[FP8Q_MULTI_MAX];
    for (int i = 0; i < n; ++i) {  // every job is checked before anything is enqueued
        const fp8q_quantize_job& j = jobs[i];
        const fp8q_status v = prepare_quantize(&j.recipe, j.x, j.rows, j.cols, j.state, j.out, a[i]);
        if (v != FP8Q_OK) return v;
        for (int k = 0; k < i; ++k)
            if (jobs[k].out == j.out || (jobs[k].state && jobs[k].state == j.state)) return FP8Q_ERR_ARG;
        rcs[i] = &j.recipe;
        sts[i] = j.state ? j.state->dev : nullptr;
    }
    for (int i = 0; i < n; ++i) set_meta(&jobs[i].recipe, jobs[i].rows, jobs[i].cols, jobs[i].out);
    return launch_quantize_multi(n, rcs, a, sts, (cudaStream_t)stream);
}

fp8q_status fp8q_delayed_create(int history_len, int fmt, int margin, fp8q_delayed_state** out) {
    if (!out || !valid_fmt(fmt)) return FP8Q_ERR_ARG;
    if (history_len < 1 || history_len > 4096 || margin < 0 || margin > 64) return FP8Q_ERR_ARG;
    *out = nullptr;
    const size_t bytes = sizeof(DelayedDev) + sizeof(float) * (size_t)history_len;
    DelayedDev* dev = nullptr;
    if (cudaMalloc(&dev, bytes) != cudaSuccess) return FP8Q_ERR_CUDA;
    DelayedDev* host = (DelayedDev*)calloc(1, bytes);
    if (!host) {
        cudaFree(dev);
        return FP8Q_ERR_ARG;
    }
    host->scale = 1.0f;
    host->scale_inv = 1.0f;
    host->head = 0;
    host->H = history_len;
    host->fmt = fmt;
    host->margin = margin;
    const cudaError_t e = cudaMemcpy(dev, host, bytes, cudaMemcpyHostToDevice);
    free(host);
    if (e != cudaSuccess) {
        cudaFree(dev);
        return FP8Q_ERR_CUDA;
    }
    fp8q_delayed_state* st = (fp8q_delayed_state*)calloc(1, sizeof(fp8q_delayed_state));
    if (!st) {
        cudaFree(dev);
        return FP8Q_ERR_ARG;
    }
    st->dev = dev;
    st->H = history_len;
    st->fmt = fmt;
    st->margin = margin;
    cudaGetDevice(&st->device);
    *out = st;
    return FP8Q_OK;
}

fp8q_status fp8q_delayed_update(fp8q_delayed_state* st, const float* amax, const unsigned long long* nonfinite,
                                void* stream) {
    if (!st || !amax) return FP8Q_ERR_ARG;
    if (!on_state_device(st)) return FP8Q_ERR_ARG;
    return launch_delayed_update(st->dev, amax, nonfinite, (cudaStream_t)stream);
}

fp8q_status fp8q_delayed_get(const fp8q_delayed_state* st, float* hist, int* head, float* scale,
                             float* scale_inv) {
    if (!st) return FP8Q_ERR_ARG;
    if (!on_state_device(st)) return FP8Q_ERR_ARG;
    const size_t bytes = sizeof(DelayedDev) + sizeof(float) * (size_t)st->H;
    DelayedDev* host = (DelayedDev*)malloc(bytes);
    if (!host) return FP8Q_ERR_ARG;
    if (cudaDeviceSynchronize() != cudaSuccess || cudaMemcpy(host, st->dev, bytes, cudaMemcpyDeviceToHost) != cudaSuccess) {
        free(host);
        return FP8Q_ERR_CUDA;
    }
    if (hist) memcpy(hist, host->hist, sizeof(float) * (size_t)st->H);
    if (head) *head = host->head;
    if (scale) *scale = host->scale;
    if (scale_inv) *scale_inv = host->scale_inv;
    free(host);
    return FP8Q_OK;
}

fp8q_status fp8q_delayed_set(fp8q_delayed_state* st, const float* hist, int head, float scale, float scale_inv) {
    if (!st || !hist) return FP8Q_ERR_ARG;
    if (head < 0 || head >= st->H) return FP8Q_ERR_ARG;
    if (!on_state_device(st)) return FP8Q_ERR_ARG;
    const size_t bytes = sizeof(DelayedDev) + sizeof(float) * (size_t)st->H;
    DelayedDev* host = (DelayedDev*)calloc(1, bytes);
    if (!host) return FP8Q_ERR_ARG;
    host->scale = scale;
    host->scale_inv = scale_inv;
    host->head = head;
    host->H = st->H;
    host->fmt = st->fmt;
    host->margin = st->margin;
    memcpy(host->hist, hist, sizeof(float) * (size_t)st->H);
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(st->dev, host, bytes, cudaMemcpyHostToDevice);
    free(host);
    return e == cudaSuccess ? FP8Q_OK : FP8Q_ERR_CUDA;
}

int fp8q_delayed_history_len(const fp8q_delayed_state* st) { return st ? st->H : 0; }

void fp8q_delayed_destroy(fp8q_delayed_state* st) {
    if (!st) return;
    cudaFree(st->dev);
    free(st);
}

fp8q_status fp8q_scaled_gemm(const fp8q_tensor* A, int a_use_col, const fp8q_tensor* B, int b_use_col, void* D,
                             int out_dtype, int64_t M, int64_t N, int64_t K, void* stream) {
    if (!A || !B || !D) return FP8Q_ERR_ARG;
    if (out_dtype != 0 && out_dtype != 1) return FP8Q_ERR_ARG;
    if (M < 1 || N < 1 || K < 1) return FP8Q_ERR_SHAPE;
    if (K % 16 != 0 || N % 8 != 0) return FP8Q_ERR_SHAPE;
    GemmOperand ga, gb;
    const fp8q_status v = prepare_operands(A, a_use_col, B, b_use_col, M, N, K, ga, gb);
    if (v != FP8Q_OK) return v;
    if (!aligned16(D)) return FP8Q_ERR_ALIGN;
    return launch_gemm(ga, gb, D, out_dtype, M, N, K, (cudaStream_t)stream);
}

fp8q_status fp8q_scaled_gemm_q(const fp8q_tensor* A, int a_use_col, const fp8q_tensor* B, int b_use_col, void* D,
                               int out_kind, int fmt, fp8q_tensor* Dq, int64_t M, int64_t N, int64_t K,
                               void* stream) {
    if (!A || !B || !Dq || !valid_fmt(fmt)) return FP8Q_ERR_ARG;
    if (out_kind != FP8Q_MXFP8_1x32 && out_kind != FP8Q_BLOCK_1x128) return FP8Q_ERR_UNSUPPORTED;
    if (M < 1 || N < 1 || K < 1) return FP8Q_ERR_SHAPE;
    if (K % 16 != 0 || N % (out_kind == FP8Q_MXFP8_1x32 ? 32 : 16) != 0) return FP8Q_ERR_SHAPE;
    if (!Dq->data_row || !Dq->scale_row || !Dq->counters) return FP8Q_ERR_ARG;
    if (!aligned16(Dq->data_row) || !aligned16(Dq->scale_row) || (D && !aligned16(D))) return FP8Q_ERR_ALIGN;
    if (((uintptr_t)Dq->counters & 7u) != 0) return FP8Q_ERR_ALIGN;
    const bool col = Dq->data_col != nullptr;  // the column-wise copy too
    if (col) {
        if (!Dq->scale_col) return FP8Q_ERR_ARG;
        if (M % 16 != 0) return FP8Q_ERR_SHAPE;  // rows of the [N][M] copy are 16-byte multiples
        if (!aligned16(Dq->data_col) || !aligned16(Dq->scale_col)) return FP8Q_ERR_ALIGN;
    }
    GemmOperand ga, gb;
    const fp8q_status v = prepare_operands(A, a_use_col, B, b_use_col, M, N, K, ga, gb);
    if (v != FP8Q_OK) return v;
    Dq->rows = M;
    Dq->cols = N;
    Dq->fmt = fmt;
    Dq->kind = out_kind;
    return launch_gemm_pair(ga, gb, D, 0, M, N, K, (cudaStream_t)stream, out_kind, fmt, Dq->data_row, Dq->scale_row,
                            Dq->counters, col ? Dq->data_col : nullptr, col ? Dq->scale_col : nullptr);
}

fp8q_status fp8q_scaled_gemm_mxq(const fp8q_tensor* A, int a_use_col, const fp8q_tensor* B, int b_use_col, void* D,
                                 int fmt, fp8q_tensor* Dq, int64_t M, int64_t N, int64_t K, void* stream) {
    return fp8q_scaled_gemm_q(A, a_use_col, B, b_use_col, D, FP8Q_MXFP8_1x32, fmt, Dq, M, N, K, stream);
}

fp8q_status fp8q_gemm_set_variant(int variant) {
    if (variant < 0 || variant > 2) return FP8Q_ERR_ARG;
    g_gemm_variant = variant;
    return FP8Q_OK;
}

fp8q_status fp8q_device_errors(unsigned int* flags, void* stream) {
    if (!flags) return FP8Q_ERR_ARG;
    fp8q_status st = read_device_errors(flags, (cudaStream_t)stream);
    if (st != FP8Q_OK) return st;
    st = read_device_errors2(flags);
    if (st != FP8Q_OK) return st;
    st = read_quant_errors(flags);
    if (st != FP8Q_OK) return st;
    return *flags ? FP8Q_ERR_TIMEOUT : FP8Q_OK;
}

fp8q_status fp8q_set_wait_limit(uint64_t ns) {
    g_wait_ns.store(ns ? ns : kDefaultWaitNs, std::memory_order_relaxed);
    return FP8Q_OK;
}

fp8q_status fp8q_stall_next(int n) {
    if (n < 0) return FP8Q_ERR_ARG;
    g_stall.store(n, std::memory_order_relaxed);
    return FP8Q_OK;
}

fp8q_status fp8q_selftest_division(const float* d, int64_t nd, int fmt, unsigned long long* mismatches,
                                   void* stream) {
    if (!valid_fmt(fmt) || !mismatches || nd < 0 || (nd > 0 && !d)) return FP8Q_ERR_ARG;
    if (((uintptr_t)mismatches & 7u) != 0 || ((uintptr_t)d & 3u) != 0) return FP8Q_ERR_ALIGN;
    return launch_div_selftest(d, nd, fmt, mismatches, (cudaStream_t)stream);
}

fp8q_status fp8q_cast_f32_bits(uint32_t start, uint64_t count, int fmt, void* out, void* stream) {
    if (!valid_fmt(fmt)) return FP8Q_ERR_ARG;
    if (count > 0 && !out) return FP8Q_ERR_ARG;
    if (count > ((uint64_t)1 << 32)) return FP8Q_ERR_SHAPE;
    if (!aligned16(out)) return FP8Q_ERR_ALIGN;
    return launch_cast_bits(start, count, fmt, (uint8_t*)out, (cudaStream_t)stream);
}

}  // extern "C"
