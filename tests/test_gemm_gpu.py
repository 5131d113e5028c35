"""Parity of the tcgen05 scaled GEMM with the oracle's fp64 dequantize-and-sum
GEMM.  The oracle's operands are its own quantization of the same bf16
inputs (every GPU copy is checked equal to it on the way), so nothing the
oracle computes comes from the CUDA path.  Bar: normwise relative error
||D - D64||_F / ||D64||_F <= 2e-3 (bf16 output rounding alone gives about
1.5e-3), plus a per-element bound for fp32 output."""
import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 2e-3


def _api():
    from fp8_scaled_quantization_quantize_gb300 import api
    return api


def _quant(api, x, kind, fmt, rowwise=True, colwise=False):
    """api.quantize on the GPU, remembering the bf16 input for the oracle."""
    qt = api.quantize(x, kind, fmt, rowwise, colwise)
    qt.src = x.cpu()
    return qt


def _operand(api, qt, use_col):
    """The oracle's quantization of qt's input (codes and plain-layout
    dequantization scales of the chosen copy), after checking that the GPU's
    copy holds the same codes."""
    parent = getattr(qt, "src_parent", None)
    if parent is not None:   # api.row_block of a quantized tensor: its rows of the whole tensor's operand
        pq, r0, r1 = parent
        data, fmt, s, bm, bk = _operand(api, pq, False)
        data = data[r0:r1]
        if s.shape[0] > 1:
            s = s[r0 // bm: -(-r1 // bm)]
        assert np.array_equal(qt.data_row.cpu().numpy(), data)
        return data, fmt, s, bm, bk
    ref = getattr(qt, "src_ref", None)
    if ref is None:
        ref = O.quantize(qt.kind, qt.fmt, inputs.bf16_bits(qt.src), qt.rowwise, qt.colwise)
        qt.src_ref = ref
    which = "col" if use_col else "row"
    R, C = (qt.cols, qt.rows) if use_col else (qt.rows, qt.cols)
    data = ref["data_" + which]
    got = (qt.data_col if use_col else qt.data_row).cpu().numpy()
    assert np.array_equal(got, data), f"GPU {which} copy differs from the oracle's quantization"
    s, bm, bk = O.dequant_scales(qt.kind, ref, which, R, C)
    return data, qt.fmt, s, max(bm, 1), max(bk, 1)


def _check(api, qa, ac, qb, bc, out_dtype=torch.bfloat16, sample=None, ctx=""):
    D = api.scaled_gemm(qa, ac, qb, bc, out_dtype)
    torch.cuda.synchronize()
    A, fa, sa, abm, abk = _operand(api, qa, ac)
    B, fb, sbb, bbn, bbk = _operand(api, qb, bc)
    M, N = A.shape[0], B.shape[0]
    if sample is None:
        pm, pn = [g.ravel() for g in np.meshgrid(np.arange(M), np.arange(N), indexing="ij")]
    else:
        pm, pn = sample(M, N)
    ref = O.gemm_points(A, fa, sa, abm, abk, B, fb, sbb, bbn, bbk, pm, pn)
    got = D.float().cpu().numpy()[pm, pn].astype(np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert np.all(np.isfinite(got)), f"{ctx}: nonfinite outputs"
    assert rel <= TOL, f"{ctx}: normwise relative error {rel:.3e} > {TOL}"
    if out_dtype == torch.float32:
        # fp32 accumulation over K products: |err| <= K * 2^-22 * sum |a b| is
        # far looser than what a correct kernel shows; use a relative bound
        assert rel <= 1e-4, f"{ctx}: fp32-output normwise error {rel:.3e}"
    return rel


def _layer(T, H, F, seed):
    X = inputs.normal_bf16((T, H), seed)
    W = inputs.normal_bf16((F, H), seed + 1, 0.02)
    dY = inputs.normal_bf16((T, F), seed + 2, 1e-4)
    return X, W, dY


RECIPES = [
    # name, kind X, kind W, kind dY, fmt X, fmt W, fmt dY
    ("pertensor_e4m3", 0, 0, 0, O.E4M3, O.E4M3, O.E4M3),
    ("pertensor_hybrid", 0, 0, 0, O.E4M3, O.E4M3, O.E5M2),
    ("mxfp8", 4, 4, 4, O.E4M3, O.E4M3, O.E4M3),
    ("block_1x128_128x128", 2, 3, 2, O.E4M3, O.E4M3, O.E4M3),
    ("perchannel_hybrid", 5, 5, 5, O.E4M3, O.E4M3, O.E5M2),
]


@pytest.fixture(params=[1, 2], ids=["sm1", "sm2"])
def variant(request):
    """Runs the test on the one-SM (M = 128) and the SM-pair (M = 256) kernel."""
    api = _api()
    api.gemm_set_variant(request.param)
    yield request.param
    api.gemm_set_variant(0)


@pytest.mark.parametrize("name,kx,kw,kd,fx,fw,fd", RECIPES, ids=[r[0] for r in RECIPES])
@pytest.mark.parametrize("T,H,F", [(256, 256, 512), (208, 272, 400), (384, 640, 528)])
@pytest.mark.parametrize("out", [torch.bfloat16, torch.float32])
def test_fprop_dgrad_wgrad(name, kx, kw, kd, fx, fw, fd, T, H, F, out, variant):
    api = _api()
    X, W, dY = _layer(T, H, F, 40 + T)
    qx = _quant(api, X.cuda(), kx, fx, True, True)
    qw = _quant(api, W.cuda(), kw, fw, True, True)
    qd = _quant(api, dY.cuda(), kd, fd, True, True)
    _check(api, qx, False, qw, False, out, ctx=f"{name} fprop")      # Y  = X . W^T
    _check(api, qd, False, qw, True, out, ctx=f"{name} dgrad")       # dX = dY . W
    if kx == 2:   # blockwise wgrad: 1x128 x 1x128 along the token dim
        _check(api, qd, True, qx, True, out, ctx=f"{name} wgrad")
    else:
        _check(api, qd, True, qx, True, out, ctx=f"{name} wgrad")    # dW = dY^T . X


def test_gemm_k_sweep_and_ragged_k(variant):
    api = _api()
    for K in (16, 48, 128, 144, 1040):
        a = inputs.normal_bf16((130, K), K)
        b = inputs.normal_bf16((264, K), K + 1)
        for kind in (0, 4, 5):
            qa = _quant(api, a.cuda(), kind, O.E4M3, True, False)
            qb = _quant(api, b.cuda(), kind, O.E4M3, True, False)
            _check(api, qa, False, qb, False, ctx=f"K={K} kind={kind}")
        qa = _quant(api, a.cuda(), 2, O.E4M3, True, False)
        qb = _quant(api, b.cuda(), 3, O.E4M3, True, False)
        _check(api, qa, False, qb, False, ctx=f"K={K} block")


def test_gemm_outlier_columns_blockwise(variant):
    """1% outlier input channels x100 (the blockwise workload's activation)."""
    api = _api()
    x = inputs.to_bf16(inputs.with_outlier_columns(inputs.normal_f32((512, 1024), 3), 0.01, 100.0, 2))
    w = inputs.normal_bf16((768, 1024), 4, 0.02)
    qx = _quant(api, x.cuda(), 2, O.E4M3, True, False)
    qw = _quant(api, w.cuda(), 3, O.E4M3, True, False)
    _check(api, qx, False, qw, False, ctx="outliers")


def _edge_sample(k):
    def f(M, N):
        g = np.random.default_rng(M * 7 + N)
        rows = np.unique(np.concatenate([[0, M - 1], g.choice(M, k, replace=False)]))
        cols = np.unique(np.concatenate([[0, N - 1], g.choice(N, k, replace=False)]))
        pm1, pn1 = [a.ravel() for a in np.meshgrid(rows, np.arange(N), indexing="ij")]
        pm2, pn2 = [a.ravel() for a in np.meshgrid(np.arange(M), cols, indexing="ij")]
        return np.concatenate([pm1, pm2]), np.concatenate([pn1, pn2])
    return f


def test_full_config_pertensor_256():
    api = _api()
    A, B = inputs.pertensor_256()
    qa = _quant(api, A.cuda(), 0, O.E4M3, True, False)
    qb = _quant(api, B.cuda(), 0, O.E4M3, True, False)
    _check(api, qa, False, qb, False, ctx="per-tensor 256 full")


def test_full_config_blockwise_llama8b_up_proj(variant):
    api = _api()
    X, W = inputs.llama8b_up_proj()
    qx = _quant(api, X.cuda(), 2, O.E4M3, True, False)
    qw = _quant(api, W.cuda(), 3, O.E4M3, True, False)
    if variant == 2:   # SM pairs, the bench's kernel: every one of the 4096 x 14336 outputs
        _check(api, qx, False, qw, False, ctx="up-proj fprop, full output")
    else:
        _check(api, qx, False, qw, False, sample=_edge_sample(254), ctx="up-proj fprop (256 rows + 256 cols)")


def test_full_config_perchannel_llama8b_up_proj():
    """Per-channel current scaling at the Llama-3-8B up-projection (X with its
    1% outlier columns): fprop, and GEMMs through both column copies."""
    api = _api()
    X, W = inputs.llama8b_up_proj()
    qx = _quant(api, X.cuda(), 5, O.E4M3, True, True)
    qw = _quant(api, W.cuda(), 5, O.E4M3, True, True)
    s = _edge_sample(254)
    _check(api, qx, False, qw, False, sample=s, ctx="perchannel fprop")
    # the column copies (per-column factors): W^T W (K = 14336) and X^T X (K = 4096)
    _check(api, qw, True, qw, True, sample=s, ctx="perchannel W^T . W")
    _check(api, qx, True, qx, True, sample=s, ctx="perchannel X^T . X")


def test_full_config_mxfp8_llama8b_mlp(variant):
    api = _api()
    X, W, dY = inputs.llama8b_mlp()
    qx = _quant(api, X.cuda(), 4, O.E4M3, True, True)
    qw = _quant(api, W.cuda(), 4, O.E4M3, True, True)
    qd = _quant(api, dY.cuda(), 4, O.E4M3, True, True)
    s = _edge_sample(254)   # 256 rows x every column and every row x 256 columns
    _check(api, qx, False, qw, False, sample=s, ctx="MXFP8 MLP fprop")
    _check(api, qd, False, qw, True, sample=s, ctx="MXFP8 MLP dgrad")
    _check(api, qd, True, qx, True, sample=s, ctx="MXFP8 MLP wgrad")


@pytest.mark.parametrize("recipe", ["blockwise", "mxfp8"])
def test_full_config_405b_fprop(recipe):
    """The Llama-3.1-405B fprop of the roofline sweep (8192 x 53248 x 16384)
    on the kernel the sweep times (the automatic choice: SM pairs): 256 rows
    x every column and every row x 256 columns against the oracle's fp64
    sums on its own quantization of the same bf16 inputs."""
    api = _api()
    X = inputs.normal_bf16((8192, 16384), 405)
    W = inputs.normal_bf16((53248, 16384), 406, 0.02)
    ka, kb = (2, 3) if recipe == "blockwise" else (4, 4)
    qx = _quant(api, X.cuda(), ka, O.E4M3, True, False)
    qw = _quant(api, W.cuda(), kb, O.E4M3, True, False)
    _check(api, qx, False, qw, False, sample=_edge_sample(254), ctx=f"405B fprop {recipe}")


@pytest.mark.parametrize("ka,kb", [(2, 3), (4, 4), (0, 0), (5, 5)], ids=["blockwise", "mxfp8", "pertensor", "perchannel"])
def test_gemm_on_row_blocks_of_b(ka, kb):
    """D = A . B^T computed on row blocks of B (api.row_block: the weight in
    column shards of D) equals the matching columns of the whole GEMM bit for
    bit on the same kernel, and the oracle."""
    api = _api()
    # K = 512: a 128-row block of 128x128 scales is 16 bytes, so every block's
    # scales start 16-byte aligned, as the SM-pair kernel's bulk copies need
    a = inputs.normal_bf16((512, 512), 31)
    b = inputs.normal_bf16((1152, 512), 32, 0.02)
    qa = _quant(api, a.cuda(), ka, O.E4M3, True, False)
    qb = _quant(api, b.cuda(), kb, O.E4M3, True, False)
    api.gemm_set_variant(2)
    try:
        D = api.scaled_gemm(qa, False, qb, False)
        for r0, r1 in ((0, 384), (384, 1024), (1024, 1152)):
            blk = api.row_block(qb, r0, r1)
            blk.src_parent = (qb, r0, r1)
            Dc = api.scaled_gemm(qa, False, blk, False)
            torch.cuda.synchronize()
            assert torch.equal(Dc.view(torch.int16), D[:, r0:r1].contiguous().view(torch.int16)), (r0, r1)
            _check(api, qa, False, blk, False, ctx=f"row block {r0}:{r1}")
    finally:
        api.gemm_set_variant(0)
    assert api.device_errors() == 0


@pytest.mark.parametrize("M,N,K", [(4096, 4096, 640), (4096, 4096, 1024), (4096, 4096, 1152), (8192, 8192, 1024)])
def test_mxfp8_short_k_many_tiles_per_pair(M, N, K):
    """MXFP8 on the SM-pair kernel with few K blocks (5 to 9) and several
    tiles per SM pair: the scale-tile movers run up to four K blocks into
    the next tile, past the stage ring's length, so every landing-barrier wait
    must be exact (sampled rows and columns against the oracle)."""
    api = _api()
    a = inputs.normal_bf16((M, K), 70 + K)
    b = inputs.normal_bf16((N, K), 71 + K, 0.02)
    qa = _quant(api, a.cuda(), 4, O.E4M3, True, False)
    qb = _quant(api, b.cuda(), 4, O.E4M3, True, False)
    api.gemm_set_variant(2)
    try:
        _check(api, qa, False, qb, False, sample=_edge_sample(12), ctx=f"mx {M}x{N}x{K}")
    finally:
        api.gemm_set_variant(0)
    assert api.device_errors() == 0
