"""The library's failure detection on a GPU, without a GPU fault: a launch run
stalled (fp8q_stall_next: its producers issue no loads, so no pipeline stage
ever fills) with a short wait limit (fp8q_set_wait_limit, 20 us) must give up
its waits, report the timeout in the error words (fp8q_device_errors returns
FP8Q_ERR_TIMEOUT with bit 0 for a GEMM, bit 1 for a quantize) and leave the
device usable: the very next launch of the same kind, with the default limit,
matches the oracle and reports no error.  Covers the quantize tile kernel and
both GEMM kernels (one SM per tile, SM pairs) on the per-tensor, blockwise and
MXFP8 pipelines, whose waits differ (accumulator, K-block partials and scale
ring, scale tiles)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import _lib as L
from fp8_scaled_quantization_quantize_gb300 import inputs
from tests._helpers import assert_quant_equal, bits_of, gpu_outputs

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000


def _api():
    from fp8_scaled_quantization_quantize_gb300 import api
    return api


def _errors():
    """(status, flags) of fp8q_device_errors (synchronises the stream)."""
    api = _api()
    v = ctypes.c_uint(0)
    st = L.load().fp8q_device_errors(ctypes.byref(v), api._stream(None))
    return st, v.value


@pytest.fixture(autouse=True)
def _clean():
    api = _api()
    api.stall_next(0)
    api.set_wait_limit(0)
    api.gemm_set_variant(0)
    _errors()
    yield
    api.stall_next(0)
    api.set_wait_limit(0)
    api.gemm_set_variant(0)


def test_stalled_quantize_times_out_and_the_next_call_is_exact():
    api = _api()
    x = inputs.normal_bf16((400, 1040), 41)
    api.set_wait_limit(LIMIT_NS)
    api.stall_next(1)
    api.quantize(x.cuda(), O.BLOCK_1x128, O.E4M3, True, True)
    st, flags = _errors()
    assert st == L.ERR_TIMEOUT and flags == 2, (st, flags)
    api.set_wait_limit(0)
    qt = api.quantize(x.cuda(), O.BLOCK_1x128, O.E4M3, True, True)
    ref = O.quantize(O.BLOCK_1x128, O.E4M3, bits_of(x), True, True)
    assert_quant_equal(O.BLOCK_1x128, gpu_outputs(qt), ref, True, True, "after a stalled launch")
    assert _errors() == (L.OK, 0)


def test_stall_counts_launches():
    """stall_next(2): the next two tile launches stall, the third does not."""
    api = _api()
    x = inputs.normal_bf16((256, 256), 42)
    api.set_wait_limit(LIMIT_NS)
    api.stall_next(2)
    for _ in range(2):
        api.quantize(x.cuda(), O.MXFP8_1x32, O.E4M3, True, False)
        assert _errors() == (L.ERR_TIMEOUT, 2)
    qt = api.quantize(x.cuda(), O.MXFP8_1x32, O.E4M3, True, False)
    ref = O.quantize(O.MXFP8_1x32, O.E4M3, bits_of(x), True, False)
    assert_quant_equal(O.MXFP8_1x32, gpu_outputs(qt), ref, True, False, "third launch")
    assert _errors() == (L.OK, 0)


RECIPES = {"pertensor": (O.PERTENSOR_CURRENT, O.PERTENSOR_CURRENT), "blockwise": (O.BLOCK_1x128, O.BLOCK_128x128),
           "mxfp8": (O.MXFP8_1x32, O.MXFP8_1x32)}


@pytest.mark.parametrize("variant", [1, 2], ids=["one_sm", "sm_pairs"])
@pytest.mark.parametrize("recipe", list(RECIPES))
def test_stalled_gemm_times_out_and_the_next_call_is_right(variant, recipe):
    api = _api()
    ka, kb = RECIPES[recipe]
    M, N, K = 512, 512, 640
    a = inputs.normal_bf16((M, K), 43)
    b = inputs.normal_bf16((N, K), 44, 0.02)
    qa = api.quantize(a.cuda(), ka, O.E4M3, True, False)
    qb = api.quantize(b.cuda(), kb, O.E4M3, True, False)
    api.gemm_set_variant(variant)
    api.set_wait_limit(LIMIT_NS)
    api.stall_next(1)
    api.scaled_gemm(qa, False, qb, False)
    st, flags = _errors()
    assert st == L.ERR_TIMEOUT and flags == 1, (st, flags)
    api.set_wait_limit(0)
    D = api.scaled_gemm(qa, False, qb, False)
    torch.cuda.synchronize()
    ra = O.quantize(ka, O.E4M3, bits_of(a), True, False)
    rb = O.quantize(kb, O.E4M3, bits_of(b), True, False)
    sa, abm, abk = O.dequant_scales(ka, ra, "row", M, K)
    sb, bbn, bbk = O.dequant_scales(kb, rb, "row", N, K)
    ref = O.gemm_full(ra["data_row"], O.E4M3, sa, abm, abk, rb["data_row"], O.E4M3, sb, bbn, bbk)
    got = D.float().cpu().numpy().astype(np.float64)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 2e-3, rel
    assert _errors() == (L.OK, 0)


@pytest.mark.parametrize("out_kind", [O.MXFP8_1x32, O.BLOCK_1x128], ids=["mxfp8_out", "1x128_out"])
def test_stalled_fused_both_copies_times_out_and_the_next_call_is_exact(out_kind):
    """The fused output quantize with both copies (whose 1x128 column path
    adds an exchange between warps on a bounded mbarrier), stalled: every
    wait gives up, the timeout is reported, and the next call's two copies
    equal the oracle's quantize of its D."""
    api = _api()
    M, N, K = 512, 512, 384
    a = inputs.normal_bf16((M, K), 45)
    b = inputs.normal_bf16((N, K), 46, 0.02)
    qa = api.quantize(a.cuda(), O.BLOCK_1x128, O.E4M3, True, False)
    qb = api.quantize(b.cuda(), O.BLOCK_128x128, O.E4M3, True, False)
    api.set_wait_limit(LIMIT_NS)
    api.stall_next(1)
    api.scaled_gemm_q(qa, False, qb, False, out_kind, O.E4M3, want_d=False, colwise=True)
    st, flags = _errors()
    assert st == L.ERR_TIMEOUT and flags == 1, (st, flags)
    api.set_wait_limit(0)
    D, Dq = api.scaled_gemm_q(qa, False, qb, False, out_kind, O.E4M3, want_d=True, colwise=True)
    torch.cuda.synchronize()
    ref = O.quantize(out_kind, O.E4M3, inputs.bf16_bits(D.cpu()), True, True)
    assert_quant_equal(out_kind, gpu_outputs(Dq), ref, True, True, "after a stalled fused launch")
    assert _errors() == (L.OK, 0)
