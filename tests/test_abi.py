"""CPU checks of the C ABI: the library loads, exports every entry point that
include/fp8q.h declares, sizes scale buffers per the documented layouts, and
rejects bad arguments before touching the GPU."""
import ctypes
import os
import re

import pytest

from fp8_scaled_quantization_quantize_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8q.h")


@pytest.fixture(scope="module")
def lib():
    from fp8_scaled_quantization_quantize_gb300 import build
    build.build()
    return L.load()


def declared():
    src = open(HEADER).read()
    return re.findall(r"FP8Q_API\s+[\w\s\*]+?\b(fp8q_\w+)\s*\(", src)


def test_header_declares_the_boundary():
    names = set(declared())
    assert {"fp8q_quantize", "fp8q_scaled_gemm", "fp8q_delayed_create", "fp8q_delayed_update",
            "fp8q_delayed_get", "fp8q_delayed_set", "fp8q_delayed_destroy", "fp8q_scale_bytes"} <= names
    assert names == set(L.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared():
        assert hasattr(lib, name), name


def test_version_and_status_strings(lib):
    assert lib.fp8q_version() == 100
    assert L.status_str(L.OK) == "ok"
    assert L.status_str(L.ERR_SHAPE) == "invalid shape"


def _sb(lib, kind, rows, cols, row=True, col=True):
    rc = L.Recipe(kind, L.E4M3, int(row), int(col))
    rb, cb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    st = lib.fp8q_scale_bytes(ctypes.byref(rc), rows, cols, ctypes.byref(rb), ctypes.byref(cb))
    return st, rb.value, cb.value


def test_scale_bytes(lib):
    assert _sb(lib, L.PERTENSOR_CURRENT, 256, 256) == (L.OK, 0, 0)
    # 1x128: [ceil(C/128)][R up to 128] fp32, and the column copy [ceil(R/128)][C up to 128]
    assert _sb(lib, L.BLOCK_1x128, 4096, 4096) == (L.OK, 32 * 4096 * 4, 32 * 4096 * 4)
    assert _sb(lib, L.BLOCK_1x128, 200, 272) == (L.OK, 3 * 256 * 4, 2 * 384 * 4)
    # 128x128: [ceil(R/128)][ceil(C/128)] fp32
    assert _sb(lib, L.BLOCK_128x128, 14336, 4096) == (L.OK, 112 * 32 * 4, 32 * 112 * 4)
    # MX: 512-byte tiles of 128 rows x 4 scale columns
    assert _sb(lib, L.MXFP8_1x32, 8192, 4096) == (L.OK, 64 * 32 * 512, 32 * 64 * 512)
    assert _sb(lib, L.MXFP8_1x32, 130, 48, True, False) == (L.OK, 2 * 1 * 512, 0)
    # per-channel: one fp32 per row of the copy, padded to 128
    assert _sb(lib, L.PERCHANNEL_CURRENT, 4096, 14336) == (L.OK, 4096 * 4, 14336 * 4)
    assert _sb(lib, L.PERCHANNEL_CURRENT, 200, 272) == (L.OK, 256 * 4, 384 * 4)
    assert _sb(lib, 9, 16, 16)[0] == L.ERR_ARG
    assert _sb(lib, L.MXFP8_1x32, -1, 16)[0] == L.ERR_SHAPE


def _q(lib, kind=L.MXFP8_1x32, fmt=L.E4M3, rows=32, cols=32, row=True, col=False, x=16, t=None, st=None):
    rc = L.Recipe(kind, fmt, int(row), int(col))
    if t is None:
        t = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 0, 0, 0, 0)
    return lib.fp8q_quantize(ctypes.byref(rc), x, rows, cols, st, ctypes.byref(t), None)


def test_quantize_validation_without_gpu(lib):
    assert _q(lib, cols=40) == L.ERR_SHAPE                  # cols % 16
    assert _q(lib, rows=40, col=True) == L.ERR_SHAPE        # rows % 16 with a column copy
    assert _q(lib, rows=-16) == L.ERR_SHAPE
    assert _q(lib, kind=7) == L.ERR_ARG
    assert _q(lib, fmt=3) == L.ERR_ARG
    assert _q(lib, row=False, col=False) == L.ERR_ARG
    assert _q(lib, x=24) == L.ERR_ALIGN                     # x not 16-byte aligned
    assert _q(lib, x=0) == L.ERR_ARG                        # NULL x
    t = L.Tensor(16, 32, 64, 128, 256, 272, 288, 0, 0, 0, 0, 0)
    assert _q(lib, t=t) == L.ERR_ARG                        # NULL counters
    t = L.Tensor(16, 32, 64 + 4, 128, 256, 272, 288, 512, 0, 0, 0, 0)
    assert _q(lib, t=t) == L.ERR_ALIGN                      # misaligned scale buffer
    assert _q(lib, kind=L.PERTENSOR_DELAYED) == L.ERR_ARG   # delayed needs a state
    assert _q(lib, rows=1 << 30, cols=1 << 11) == L.ERR_SHAPE


def test_quantize_multi_validation_without_gpu(lib):
    """Every job is checked before anything is enqueued; the same checks as
    fp8q_quantize, plus the job count and no shared outputs or states."""
    t1 = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 0, 0, 0, 0)
    t2 = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 0, 0, 0, 0)

    def jobs(*specs):
        arr = (L.QuantizeJob * max(len(specs), 1))()
        for i, (kind, rows, cols, x, t) in enumerate(specs):
            arr[i].recipe = L.Recipe(kind, L.E4M3, 1, 0)
            arr[i].x, arr[i].rows, arr[i].cols, arr[i].state = x, rows, cols, None
            arr[i].out = ctypes.pointer(t)
        return arr

    m = lambda arr, n: lib.fp8q_quantize_multi(arr, n, None)
    assert m(jobs(), 0) == L.OK                                              # nothing to do
    assert m(jobs(), -1) == L.ERR_ARG
    assert m(jobs(), L.MULTI_MAX + 1) == L.ERR_ARG
    assert m(jobs((L.MXFP8_1x32, 32, 32, 16, t1), (L.MXFP8_1x32, 32, 40, 16, t2)), 2) == L.ERR_SHAPE
    assert m(jobs((L.MXFP8_1x32, 32, 32, 16, t1), (L.BLOCK_1x128, 32, 32, 24, t2)), 2) == L.ERR_ALIGN
    assert m(jobs((L.MXFP8_1x32, 32, 32, 16, t1), (L.PERTENSOR_DELAYED, 32, 32, 16, t2)), 2) == L.ERR_ARG
    assert m(jobs((L.MXFP8_1x32, 32, 32, 16, t1), (L.BLOCK_1x128, 32, 32, 16, t1)), 2) == L.ERR_ARG  # same out


def test_quantize_rows_validation_without_gpu(lib):
    t = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 0, 0, 0, 0)

    def qr(kind, row0, rows, total, cols=32, col=False, x=16):
        rc = L.Recipe(kind, L.E4M3, 1, int(col))
        return lib.fp8q_quantize_rows(ctypes.byref(rc), x, row0, rows, total, cols, ctypes.byref(t), None)

    assert qr(L.PERTENSOR_CURRENT, 0, 128, 256) == L.ERR_DTYPE        # the scale needs the whole tensor
    assert qr(L.PERCHANNEL_CURRENT, 0, 128, 256, col=True) == L.ERR_DTYPE
    assert qr(L.BLOCK_128x128, 64, 128, 256) == L.ERR_SHAPE            # row0 off a 128-row group
    assert qr(L.BLOCK_128x128, 0, 100, 256) == L.ERR_SHAPE             # a partial block that does not end it
    assert qr(L.BLOCK_128x128, 128, 256, 256) == L.ERR_SHAPE           # past the end
    assert qr(L.MXFP8_1x32, 0, 128, 200, col=True) == L.ERR_SHAPE      # total rows % 16 with a column copy
    assert qr(L.BLOCK_1x128, 0, 128, 256, cols=40) == L.ERR_SHAPE
    assert qr(L.BLOCK_1x128, 0, 128, 256, x=24) == L.ERR_ALIGN


def test_gemm_validation_without_gpu(lib):
    a = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 64, 128, L.E4M3, L.MXFP8_1x32)
    b = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 96, 128, L.E4M3, L.MXFP8_1x32)
    g = lambda M, N, K, od=0, ac=0, bc=0, A=a, B=b, D=1024: lib.fp8q_scaled_gemm(
        ctypes.byref(A), ac, ctypes.byref(B), bc, D, od, M, N, K, None)
    assert g(64, 96, 64) == L.ERR_SHAPE                     # K mismatch with the operands
    assert g(64, 96, 128, od=2) == L.ERR_ARG
    assert g(0, 96, 128) == L.ERR_SHAPE
    assert g(64, 96, 128, D=1032) == L.ERR_ALIGN
    pt = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 96, 128, L.E4M3, L.PERTENSOR_CURRENT)
    assert g(64, 96, 128, B=pt) == L.ERR_DTYPE              # MX with per-tensor
    blk = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 64, 128, L.E4M3, L.BLOCK_128x128)
    blkb = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 96, 128, L.E4M3, L.BLOCK_128x128)
    assert g(64, 96, 128, A=blk, B=blkb) == L.ERR_DTYPE     # blockwise A must be 1x128


def test_fused_gemm_validation_without_gpu(lib):
    """fp8q_scaled_gemm_q refuses, before any launch, a column-wise output copy
    it cannot write: M % 16 != 0 (the [N][M] copy's rows must be 16-byte
    multiples), no column scale buffer, a misaligned column buffer; and an
    output kind it does not fuse."""
    a = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 72, 128, L.E4M3, L.MXFP8_1x32)
    b = L.Tensor(16, 32, 64, 128, 256, 272, 288, 512, 96, 128, L.E4M3, L.MXFP8_1x32)

    def g(M, kind=L.MXFP8_1x32, col=4096, scol=8192):
        dq = L.Tensor(1024, col, 2048, scol, 0, 0, 0, 3072, 0, 0, 0, 0)
        return lib.fp8q_scaled_gemm_q(ctypes.byref(a), 0, ctypes.byref(b), 0, None, kind, L.E4M3,
                                      ctypes.byref(dq), M, 96, 128, None)
    assert g(72) == L.ERR_SHAPE                      # column copy with M % 16 != 0
    assert g(64, scol=0) == L.ERR_ARG                # column copy without its scales
    assert g(64, col=4104) == L.ERR_ALIGN            # misaligned column codes
    assert g(64, kind=L.BLOCK_128x128) == L.ERR_UNSUPPORTED


def test_delayed_validation_without_gpu(lib):
    h = ctypes.c_void_p(0)
    assert lib.fp8q_delayed_create(0, L.E4M3, 0, ctypes.byref(h)) == L.ERR_ARG
    assert lib.fp8q_delayed_create(16, 5, 0, ctypes.byref(h)) == L.ERR_ARG
    assert lib.fp8q_delayed_create(16, L.E4M3, -1, ctypes.byref(h)) == L.ERR_ARG
    assert lib.fp8q_delayed_update(None, None, None, None) == L.ERR_ARG
    assert lib.fp8q_cast_f32_bits(0, 16, 9, 16, None) == L.ERR_ARG


def test_row_block_views():
    """api.row_block: views of the row copy and of its scales for a block of
    128-row groups (host buffers; no GPU needed)."""
    torch = pytest.importorskip("torch")
    from fp8_scaled_quantization_quantize_gb300 import api
    R, C = 1000, 384
    for kind, per_block in ((L.BLOCK_128x128, 3 * 4), (L.MXFP8_1x32, 3 * 512), (L.PERCHANNEL_CURRENT, 128 * 4)):
        qt = api.alloc(kind, L.E4M3, R, C, True, False, device="cpu")
        qt.data_row.copy_(torch.arange(R * C, dtype=torch.int64).reshape(R, C).to(torch.uint8))
        qt.scale_row.copy_(torch.arange(qt.scale_row.numel(), dtype=torch.int64).to(torch.uint8))
        b = api.row_block(qt, 256, 1000)
        assert (b.rows, b.cols, b.kind) == (744, C, kind)
        assert torch.equal(b.data_row, qt.data_row[256:1000])
        assert b.scale_row.numel() == 6 * per_block             # 128-row groups 2..7 (the last one partial)
        assert torch.equal(b.scale_row, qt.scale_row[2 * per_block:8 * per_block])
    qt = api.alloc(L.BLOCK_1x128, L.E4M3, R, C, True, False, device="cpu")
    with pytest.raises(ValueError):
        api.row_block(qt, 0, 128)                                # K-block-major scales
    qt = api.alloc(L.PERTENSOR_CURRENT, L.E4M3, R, C, True, False, device="cpu")
    with pytest.raises(ValueError):
        api.row_block(qt, 64, 512)                               # not a 128-row boundary
    assert api.row_block(qt, 896, 1000).rows == 104


def test_missing_library_raises(monkeypatch, tmp_path):
    """Without the built library the binding raises at the first call; there
    is no other implementation to fall back on."""
    from fp8_scaled_quantization_quantize_gb300 import _lib, api
    missing = str(tmp_path / "libfp8q.so")
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib.load, "__defaults__", (missing,))
    with pytest.raises(ImportError, match="not built"):
        _lib.load()
    with pytest.raises(ImportError, match="not built"):
        api.scale_bytes(api.BLOCK_1x128, 256, 256, True, True)


def test_binding_rejects_mismatched_or_host_buffers():
    """The binding refuses, before the library is called, tensors that would
    reach the kernels as out-of-range or host addresses: an input of another
    shape than its output buffers, host tensors, a wrong GEMM output."""
    torch = pytest.importorskip("torch")
    from fp8_scaled_quantization_quantize_gb300 import api
    qt = api.alloc(L.BLOCK_1x128, L.E4M3, 256, 128, True, True, device="cpu")
    x = torch.zeros((256, 128), dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="shape"):
        api.quantize_into(torch.zeros((512, 128), dtype=torch.bfloat16), qt)
    with pytest.raises(ValueError, match="shape"):
        api.quantize_multi([(torch.zeros((256, 256), dtype=torch.bfloat16), qt)])
    with pytest.raises(ValueError, match="shape"):
        api.quantize_rows_into(torch.zeros((128, 64), dtype=torch.bfloat16), qt, 0)
    with pytest.raises(ValueError, match="CUDA device"):
        api.quantize_into(x, qt)
    with pytest.raises(ValueError, match="CUDA device"):
        api.quantize_multi([(x, qt)])
    with pytest.raises(ValueError, match="CUDA device"):
        api.quantize_rows_into(x[:128], qt, 0)
    with pytest.raises(ValueError, match="contiguous 2-D bf16"):
        api.quantize_into(x.float(), qt)
    qb = api.alloc(L.BLOCK_128x128, L.E4M3, 384, 128, True, False, device="cpu")
    with pytest.raises(ValueError, match="CUDA device"):
        api.scaled_gemm(qt, False, qb, False)
    with pytest.raises(ValueError, match="CUDA device"):
        api.scaled_gemm_mxq(qt, False, qb, False)
    with pytest.raises(ValueError, match="uint8"):
        api.cast_f32_bits(0, 16, L.E4M3, torch.empty(16, dtype=torch.uint8))
    with pytest.raises(ValueError, match="fp32"):
        api.selftest_division(torch.ones(4), L.E4M3)
