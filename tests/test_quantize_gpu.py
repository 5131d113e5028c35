"""Parity of the CUDA quantize kernels with the oracle: every byte of every
row-wise / column-wise copy, every scale (in the library's packed layout),
the per-tensor scalars and the saturation / nonfinite counters bit-exact, on
seeded inputs that span several 128x128 tiles with ragged edges, on the edge
cases of each recipe, and at the full workload shapes."""
import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs
from tests._helpers import assert_quant_equal, bits_of, gpu_outputs

pytestmark = pytest.mark.gpu

KINDS = [O.PERTENSOR_CURRENT, O.BLOCK_1x128, O.BLOCK_128x128, O.MXFP8_1x32, O.PERCHANNEL_CURRENT]
COPIES = [(True, False), (False, True), (True, True)]


def _api():
    from fp8_scaled_quantization_quantize_gb300 import api
    return api


def _run(kind, fmt, x, rowwise, colwise, state=None, ostate=None, ctx=""):
    api = _api()
    qt = api.quantize(x.cuda(), kind, fmt, rowwise, colwise, state=state)
    got = gpu_outputs(qt)
    ref = O.quantize(kind, fmt, bits_of(x), rowwise, colwise, state=ostate)
    assert_quant_equal(kind, got, ref, rowwise, colwise, ctx)
    return qt, got, ref


def _mixed(shape, seed):
    """N(0,1) with 1% outliers x1000, a zeroed stripe, tiny subnormal-range
    values and a few exact block-max ties."""
    x = inputs.normal_f32(shape, seed)
    x = inputs.with_outlier_elements(x, 0.01, 1000.0, seed + 7)
    x[: min(3, shape[0]), :] = 0.0
    g = np.random.default_rng(seed)
    idx = g.choice(x.size, size=max(1, x.size // 200), replace=False)
    x.reshape(-1)[idx] *= np.float32(2.0 ** -120)
    return inputs.to_bf16(x)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
@pytest.mark.parametrize("rowwise,colwise", COPIES)
@pytest.mark.parametrize("shape", [(272, 400), (128, 128), (16, 16), (400, 1040)])
def test_quantize_matches_oracle(kind, fmt, rowwise, colwise, shape):
    x = _mixed(shape, 11 + shape[0])
    _run(kind, fmt, x, rowwise, colwise, ctx=f"{kind} {fmt} {shape}")


@pytest.mark.parametrize("kind", KINDS)
def test_quantize_special_values(kind):
    """NaN (both signs), +-Inf, -0, bf16 subnormals, bf16 max, all-zero blocks."""
    x = inputs.normal_f32((256, 384), 3)
    x[5, :] = 0.0
    x[:, 200:232] = 0.0
    x[7, 9] = np.inf
    x[8, 10] = -np.inf
    x[9, 11] = -0.0
    x[10, 12:20] = np.float32(2.0 ** -130)
    x[11, 300] = np.float32(3.3895e38)
    xb = inputs.to_bf16(x)
    xb[12, 13] = float("nan")          # torch stores 0x7FC0
    bits = bits_of(xb).copy()
    bits[13, 14] = 0xFFC1               # negative NaN with a payload
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16)
    for fmt in (O.E4M3, O.E5M2):
        _run(kind, fmt, xb, True, True, ctx=f"special {kind} {fmt}")


@pytest.mark.parametrize("kind", KINDS)
def test_quantize_all_zero_and_empty(kind):
    _run(kind, O.E4M3, torch.zeros((144, 160), dtype=torch.bfloat16), True, True, ctx="zeros")
    api = _api()
    for shape in ((0, 64), (32, 0), (0, 0)):
        qt = api.quantize(torch.zeros(shape, dtype=torch.bfloat16, device="cuda"), kind, O.E4M3, True, True)
        got = gpu_outputs(qt)
        assert got["nonfinite"] == 0 and got["sat_row"] == 0
        if kind == O.PERTENSOR_CURRENT:
            assert got["scale"] == 1.0 and got["scale_inv"] == 1.0 and got["amax"] == 0.0


def test_delayed_steps_and_checkpoint():
    """32 steps of per-tensor delayed scaling (history 16, E5M2 as for dY)
    against the oracle state machine, a spike and a NaN step included; then a
    checkpoint restore replays steps 16..31 bit-exactly."""
    api = _api()
    mags = inputs.delayed_magnitudes(32)
    st = api.DelayedState(16, O.E5M2, 0)
    ost = O.Delayed(16, O.E5M2, 0)
    saved = None
    outs = []
    xs = []
    for t in range(32):
        x = inputs.normal_bf16((96, 160), 500 + t, 1e-4 * float(mags[t, 2]))
        if t == 25:
            x[3, 3] = float("nan")
        xs.append(x)
        if t == 16:
            saved = st.get()
            osaved = (ost.hist.copy(), ost.head, ost.scale, ost.scale_inv)
        _, got, ref = _run(O.PERTENSOR_DELAYED, O.E5M2, x, True, True, state=st, ostate=ost, ctx=f"step {t}")
        outs.append(got)
        hist, head, s, si = st.get()
        assert head == ost.head and np.array_equal(np.float32(hist), ost.hist)
        assert np.float32(s) == ost.scale and np.float32(si) == ost.scale_inv
    assert osaved[1] == saved[1]
    # restore and replay
    st.set(*saved)
    for t in range(16, 32):
        qt = api.quantize(xs[t].cuda(), O.PERTENSOR_DELAYED, O.E5M2, True, True, state=st)
        got = gpu_outputs(qt)
        assert np.array_equal(got["data_row"], outs[t]["data_row"]) and got["scale"] == outs[t]["scale"]


def test_delayed_update_entry_point():
    api = _api()
    st = api.DelayedState(4, O.E4M3, 1)
    ost = O.Delayed(4, O.E4M3, 1)
    for a in (3.0, 0.0, 17.5, 2.0, 1.0, 0.25):
        st.update(torch.tensor([a], dtype=torch.float32, device="cuda"))
        ost.update(a)
        hist, head, s, si = st.get()
        assert np.float32(s) == ost.scale and head == ost.head
    nf = torch.tensor([1], dtype=torch.int64, device="cuda")
    st.update(torch.tensor([1e6], dtype=torch.float32, device="cuda"), nf)
    assert np.float32(st.get()[2]) == ost.scale


CONFIG_SHAPES = [
    # (name, kind, fmt, shape, rowwise, colwise, maker)
    ("per-tensor 256 A", O.PERTENSOR_CURRENT, O.E4M3, None, True, True, lambda: inputs.pertensor_256()[0]),
    ("up-proj X", O.BLOCK_1x128, O.E4M3, None, True, True, lambda: inputs.llama8b_up_proj()[0]),
    ("up-proj W", O.BLOCK_128x128, O.E4M3, None, True, True, lambda: inputs.llama8b_up_proj()[1]),
    ("MXFP8 MLP X", O.MXFP8_1x32, O.E4M3, None, True, True, lambda: inputs.llama8b_mlp()[0]),
    ("perchannel X", O.PERCHANNEL_CURRENT, O.E4M3, None, True, True, lambda: inputs.llama8b_up_proj()[0]),
    ("perchannel W", O.PERCHANNEL_CURRENT, O.E4M3, None, True, True, lambda: inputs.llama8b_up_proj()[1]),
]


@pytest.mark.parametrize("name,kind,fmt,shape,rowwise,colwise,maker", CONFIG_SHAPES, ids=[c[0] for c in CONFIG_SHAPES])
def test_quantize_full_config_shapes(name, kind, fmt, shape, rowwise, colwise, maker):
    _run(kind, fmt, maker(), rowwise, colwise, ctx=name)


def test_quantize_full_mx_dy_and_w():
    X, W, dY = inputs.llama8b_mlp()
    del X
    _run(O.MXFP8_1x32, O.E4M3, W, True, True, ctx="MXFP8 MLP W")
    _run(O.MXFP8_1x32, O.E4M3, dY, True, True, ctx="MXFP8 MLP dY")


def test_quantize_sweep_tensor_pertensor_and_mx():
    x = inputs.sweep_tensor(64)
    _run(O.PERTENSOR_CURRENT, O.E4M3, x, True, False, ctx="sweep 64MiB current")
    _run(O.MXFP8_1x32, O.E4M3, x, True, False, ctx="sweep 64MiB mx")


def test_rejects_bad_arguments():
    api = _api()
    x = torch.zeros((32, 40), dtype=torch.bfloat16, device="cuda")   # cols % 16 != 0
    with pytest.raises(api.Fp8qError) as e:
        api.quantize(x, O.MXFP8_1x32, O.E4M3, True, False)
    assert e.value.status == 2
    x = torch.zeros((40, 32), dtype=torch.bfloat16, device="cuda")   # rows % 16 != 0 with colwise
    with pytest.raises(api.Fp8qError):
        api.quantize(x, O.BLOCK_1x128, O.E4M3, True, True)
    with pytest.raises(api.Fp8qError):                                 # delayed without a state
        api.quantize(torch.zeros((32, 32), dtype=torch.bfloat16, device="cuda"), O.PERTENSOR_DELAYED)


def test_quantize_multi_matches_separate_calls_and_oracle():
    """fp8q_quantize_multi over one job of every recipe (mixed shapes, both
    formats, a delayed state): every output equals the oracle's and what
    separate fp8q_quantize calls write, and the delayed state advances once."""
    api = _api()
    specs = [  # kind, fmt, shape, rowwise, colwise
        (O.BLOCK_1x128, O.E4M3, (400, 1040), True, True),
        (O.BLOCK_128x128, O.E4M3, (1040, 400), True, True),
        (O.PERTENSOR_CURRENT, O.E5M2, (272, 400), True, True),
        (O.PERTENSOR_DELAYED, O.E4M3, (256, 384), True, True),
        (O.MXFP8_1x32, O.E4M3, (208, 288), True, True),
        (O.PERCHANNEL_CURRENT, O.E5M2, (336, 528), True, False),
    ]
    xs = [_mixed(sh, 90 + i) for i, (_, _, sh, _, _) in enumerate(specs)]
    st, st2 = api.DelayedState(16, O.E4M3, 0), api.DelayedState(16, O.E4M3, 0)
    ost = O.Delayed(16, O.E4M3, 0)
    for s in (st, st2):     # one earlier step, so the multi call casts with a real history scale
        s.update(torch.tensor([3.5], dtype=torch.float32, device="cuda"))
    ost.update(3.5)
    qts = [api.alloc(k, f, *sh, r, c, "cuda") for k, f, sh, r, c in specs]
    xd = [x.cuda() for x in xs]
    jobs = [(x, q, st) if k == O.PERTENSOR_DELAYED else (x, q) for x, q, (k, *_) in zip(xd, qts, specs)]
    api.quantize_multi(jobs)
    for (k, f, sh, r, c), x, q, xdev in zip(specs, xs, qts, xd):
        got = gpu_outputs(q)
        ref = O.quantize(k, f, bits_of(x), r, c, state=ost if k == O.PERTENSOR_DELAYED else None)
        assert_quant_equal(k, got, ref, r, c, ctx=f"multi kind {k}")
        one = gpu_outputs(api.quantize(xdev, k, f, r, c, state=st2 if k == O.PERTENSOR_DELAYED else None))
        assert [got[kk] for kk in ("sat_row", "sat_col", "nonfinite")] == \
            [one[kk] for kk in ("sat_row", "sat_col", "nonfinite")], k
        for key in ("data_row", "data_col", "scale_row_bytes", "scale_col_bytes"):
            if key in one:
                assert np.array_equal(got[key], one[key]), (k, key)
    h, head, s, si = st.get()
    assert head == ost.head and np.float32(s) == ost.scale
    assert api.device_errors() == 0


def test_quantize_multi_in_a_cuda_graph():
    """The multi call's fork and join are captured into a CUDA graph with the
    stream: replays on new inputs give the outputs of direct calls."""
    api = _api()
    X = inputs.normal_bf16((512, 1024), 7).cuda()
    W = inputs.normal_bf16((1536, 1024), 8, 0.02).cuda()
    qx = api.alloc(O.BLOCK_1x128, O.E4M3, 512, 1024, True, True, "cuda")
    qw = api.alloc(O.BLOCK_128x128, O.E4M3, 1536, 1024, True, True, "cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        api.quantize_multi([(X, qx), (W, qw)])      # warm-up: creates the library's streams
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        api.quantize_multi([(X, qx), (W, qw)])
    X.copy_(inputs.normal_bf16((512, 1024), 17).cuda())
    W.copy_(inputs.normal_bf16((1536, 1024), 18, 0.02).cuda())
    g.replay()
    torch.cuda.synchronize()
    gx, gw = gpu_outputs(qx), gpu_outputs(qw)
    rx = gpu_outputs(api.quantize(X, O.BLOCK_1x128, O.E4M3, True, True))
    rw = gpu_outputs(api.quantize(W, O.BLOCK_128x128, O.E4M3, True, True))
    for got, ref in ((gx, rx), (gw, rw)):
        for key in ("data_row", "data_col", "scale_row_bytes", "scale_col_bytes"):
            assert np.array_equal(got[key], ref[key]), key
    assert api.device_errors() == 0


@pytest.mark.parametrize("kind,fmt,rowwise,colwise", [
    (O.BLOCK_1x128, O.E4M3, True, True), (O.BLOCK_128x128, O.E5M2, True, True),
    (O.MXFP8_1x32, O.E4M3, True, True), (O.MXFP8_1x32, O.E4M3, False, True),
    (O.PERCHANNEL_CURRENT, O.E4M3, True, False)])
def test_quantize_rows_blocks_equal_whole(kind, fmt, rowwise, colwise):
    """fp8q_quantize_rows over blocks [0, 256), [256, 640), [640, 720) of a
    720-row tensor writes every byte the whole-tensor call writes (buffers
    poisoned first), the counters add up to its counters, and both match the
    oracle."""
    api = _api()
    x = _mixed((720, 400), 123)
    xd = x.cuda()
    whole = gpu_outputs(api.quantize(xd, kind, fmt, rowwise, colwise))
    qt = api.alloc(kind, fmt, 720, 400, rowwise, colwise, "cuda")
    for t in (qt.data_row, qt.data_col, qt.scale_row, qt.scale_col):
        if t is not None:
            t.fill_(0xA5)
    qt.counters.zero_()
    for r0, r1 in ((0, 256), (256, 640), (640, 720)):
        api.quantize_rows_into(xd[r0:r1].contiguous(), qt, r0)
    got = gpu_outputs(qt)
    for key in ("data_row", "data_col", "scale_row_bytes", "scale_col_bytes"):
        if key in whole:
            assert np.array_equal(got[key], whole[key]), key
    assert [got[k] for k in ("sat_row", "sat_col", "nonfinite")] == [whole[k] for k in ("sat_row", "sat_col", "nonfinite")]
    ref = O.quantize(kind, fmt, bits_of(x), rowwise, colwise)
    assert_quant_equal(kind, got, ref, rowwise, colwise, ctx="rows")
    assert api.device_errors() == 0


def test_quantize_multi_and_rows_edge_cases():
    """An empty job among others, a single job, an empty block: the same bytes
    as the plain calls, nothing written for the empty ones."""
    api = _api()
    x = _mixed((272, 400), 5).cuda()
    empty = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    q1 = api.alloc(O.MXFP8_1x32, O.E4M3, 272, 400, True, True, "cuda")
    q0 = api.alloc(O.BLOCK_1x128, O.E4M3, 0, 64, True, True, "cuda")
    api.quantize_multi([(x, q1), (empty, q0)])
    ref = gpu_outputs(api.quantize(x, O.MXFP8_1x32, O.E4M3, True, True))
    got = gpu_outputs(q1)
    for key in ("data_row", "data_col", "scale_row_bytes", "scale_col_bytes"):
        assert np.array_equal(got[key], ref[key]), key
    assert gpu_outputs(q0)["nonfinite"] == 0
    q2 = api.alloc(O.BLOCK_128x128, O.E5M2, 272, 400, True, True, "cuda")
    api.quantize_multi([(x, q2)])                        # one job: the plain path
    one = gpu_outputs(api.quantize(x, O.BLOCK_128x128, O.E5M2, True, True))
    g2 = gpu_outputs(q2)
    for key in ("data_row", "data_col", "scale_row_bytes", "scale_col_bytes"):
        assert np.array_equal(g2[key], one[key]), key
    # an empty block of rows writes nothing, and E5M2 1x128 row-only blocks match the whole call
    q3 = api.alloc(O.BLOCK_1x128, O.E5M2, 272, 400, True, False, "cuda")
    q3.data_row.fill_(0x5A)
    q3.counters.zero_()
    api.quantize_rows_into(x[256:256].contiguous(), q3, 256)
    torch.cuda.synchronize()
    assert bool((q3.data_row == 0x5A).all())
    for r0, r1 in ((0, 128), (128, 272)):
        api.quantize_rows_into(x[r0:r1].contiguous(), q3, r0)
    whole = gpu_outputs(api.quantize(x, O.BLOCK_1x128, O.E5M2, True, False))
    g3 = gpu_outputs(q3)
    assert np.array_equal(g3["data_row"], whole["data_row"])
    assert np.array_equal(g3["scale_row_bytes"], whole["scale_row_bytes"])
    assert g3["sat_row"] == whole["sat_row"]
    assert api.device_errors() == 0


def test_bench_step_as_timed_matches_oracle():
    """The benchmark's step in the launch arrangement it is timed in: X
    (1x128) and W (128x128) of the Llama-3-8B up-projection, both copies, in
    one fp8q_quantize_multi call, then the fprop GEMM with the automatic
    kernel choice.  Every byte, scale and counter of both tensors equals the
    oracle's; the GEMM matches the oracle's fp64 sum on every output of 256
    rows and of 256 columns (the first and last of each among them)."""
    api = _api()
    X, W = inputs.llama8b_up_proj()
    T, H = X.shape
    F = W.shape[0]
    qx = api.alloc(O.BLOCK_1x128, O.E4M3, T, H, True, True, "cuda")
    qw = api.alloc(O.BLOCK_128x128, O.E4M3, F, H, True, True, "cuda")
    Xd, Wd = X.cuda(), W.cuda()
    api.quantize_multi([(Xd, qx), (Wd, qw)])
    refs = {}
    for name, kind, x, q in (("X", O.BLOCK_1x128, X, qx), ("W", O.BLOCK_128x128, W, qw)):
        refs[name] = O.quantize(kind, O.E4M3, bits_of(x), True, True)
        assert_quant_equal(kind, gpu_outputs(q), refs[name], True, True, ctx=f"bench step {name}")
    Y = api.scaled_gemm(qx, False, qw, False)
    torch.cuda.synchronize()
    g = np.random.default_rng(2024)
    rows = np.unique(np.concatenate([[0, T - 1], g.choice(np.arange(1, T - 1), 254, replace=False)]))
    cols = np.unique(np.concatenate([[0, F - 1], g.choice(np.arange(1, F - 1), 254, replace=False)]))
    pm1, pn1 = [a.ravel() for a in np.meshgrid(rows, np.arange(F), indexing="ij")]
    pm2, pn2 = [a.ravel() for a in np.meshgrid(np.arange(T), cols, indexing="ij")]
    pm, pn = np.concatenate([pm1, pm2]), np.concatenate([pn1, pn2])
    sx, xbm, xbk = O.dequant_scales(O.BLOCK_1x128, refs["X"], "row", T, H)
    sw, wbn, wbk = O.dequant_scales(O.BLOCK_128x128, refs["W"], "row", F, H)
    ref = O.gemm_points(refs["X"]["data_row"], O.E4M3, sx, xbm, xbk, refs["W"]["data_row"], O.E4M3, sw, wbn, wbk,
                        pm, pn)
    got = Y.float().cpu().numpy()[pm, pn].astype(np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert np.all(np.isfinite(got)) and rel <= 2e-3, rel
    assert api.device_errors() == 0


BAND = 256          # canary bytes on each side of every output buffer (keeps 16-byte alignment)
CANARY = 0xA5


def _guarded(nbytes, device):
    """nbytes of uint8 inside a buffer with BAND canary bytes on each side:
    (the inner view, the whole buffer)."""
    whole = torch.full((BAND + nbytes + BAND,), CANARY, dtype=torch.uint8, device=device)
    return whole[BAND:BAND + nbytes], whole


def _guarded_qtensor(api, kind, fmt, rows, cols, rowwise, colwise, device):
    """A QTensor whose every buffer sits between canary bands, sized as
    api.alloc sizes them."""
    rb, cb = api.scale_bytes(kind, rows, cols, rowwise, colwise)
    wholes = []

    def buf(n):
        v, w = _guarded(n, device)
        wholes.append((w, n))
        return v

    data_row = buf(rows * cols).view(rows, cols) if rowwise else None
    data_col = buf(rows * cols).view(cols, rows) if colwise else None
    scale_row = buf(max(rb, 16)) if rowwise and rb else None
    scale_col = buf(max(cb, 16)) if colwise and cb else None
    amax, scale, scale_inv = (buf(4).view(torch.float32) for _ in range(3))
    counters = buf(24).view(torch.int64)
    scale.fill_(1.0)
    scale_inv.fill_(1.0)
    counters.zero_()
    qt = api.QTensor(kind, fmt, rows, cols, data_row, data_col, scale_row, scale_col, amax, scale, scale_inv,
                     counters)
    return qt, wholes


def _bands_intact(wholes):
    for w, n in wholes:
        h = w.cpu().numpy()
        if not (np.all(h[:BAND] == CANARY) and np.all(h[BAND + n:] == CANARY)):
            return False
    return True


@pytest.mark.parametrize("kind", KINDS)
def test_outputs_stay_inside_their_buffers(kind):
    """Guard bands: every quantize output buffer (codes, scales, scalars,
    counters), the GEMM's D and the fused quantize's outputs are placed
    between canary bytes at ragged shapes (288 x 400: 128-row and 128-column
    tails); after the calls the canaries are intact and the quantize outputs
    still equal the oracle's."""
    api = _api()
    rows, cols = 288, 400
    x = _mixed((rows, cols), 77)
    qt, wholes = _guarded_qtensor(api, kind, O.E4M3, rows, cols, True, True, "cuda")
    api.quantize_into(x.cuda(), qt)
    ref = O.quantize(kind, O.E4M3, bits_of(x), True, True)
    assert_quant_equal(kind, gpu_outputs(qt), ref, True, True, ctx=f"guarded {kind}")
    assert _bands_intact(wholes), f"quantize kind {kind} wrote outside a buffer"
    # D = A . qt^T (M = N = 288, K = 400) into a guarded bf16 buffer; a 128x128
    # copy pairs with a 1x128 A operand, every other kind with itself
    qa = api.quantize(x.cuda(), O.BLOCK_1x128, O.E4M3, True, False) if kind == O.BLOCK_128x128 else qt
    d, dw = _guarded(rows * rows * 2, "cuda")
    api.scaled_gemm(qa, False, qt, False, out=d.view(torch.bfloat16).view(rows, rows))
    torch.cuda.synchronize()
    assert _bands_intact([(dw, rows * rows * 2)]), f"GEMM kind {kind} wrote outside D"
    if kind == O.MXFP8_1x32:
        # the fused MXFP8 quantize of D (N = 288, a multiple of 32)
        qy, yw = _guarded_qtensor(api, O.MXFP8_1x32, O.E4M3, rows, rows, True, False, "cuda")
        dy, dyw = _guarded(rows * rows * 2, "cuda")
        api.scaled_gemm_mxq(qt, False, qt, False, O.E4M3, want_d=True, out=qy,
                            d_out=dy.view(torch.bfloat16).view(rows, rows))
        torch.cuda.synchronize()
        assert _bands_intact(yw + [(dyw, rows * rows * 2)]), "fused quantize wrote outside its buffers"
    assert api.device_errors() == 0
