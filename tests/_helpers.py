"""Shared test helpers: run the CUDA path through the C ABI and put its
outputs next to the oracle's in a comparable form."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs

KIND_NAMES = {0: "pertensor_current", 1: "pertensor_delayed", 2: "block_1x128", 3: "block_128x128", 4: "mxfp8_1x32",
              5: "perchannel_current"}


def bits_of(x: torch.Tensor) -> np.ndarray:
    return inputs.bf16_bits(x)


def to_np_u8(t: torch.Tensor | None):
    return None if t is None else t.cpu().numpy()


def gpu_outputs(qt) -> dict:
    """Host copies of a QTensor's buffers."""
    torch.cuda.synchronize()
    c = qt.counters.cpu().numpy().astype(np.uint64)
    out = dict(sat_row=int(c[0]), sat_col=int(c[1]), nonfinite=int(c[2]),
               amax=np.float32(qt.amax.item()), scale=np.float32(qt.scale.item()),
               scale_inv=np.float32(qt.scale_inv.item()))
    if qt.data_row is not None:
        out["data_row"] = qt.data_row.cpu().numpy()
    if qt.data_col is not None:
        out["data_col"] = qt.data_col.cpu().numpy()
    if qt.scale_row is not None:
        out["scale_row_bytes"] = qt.scale_row.cpu().numpy()
    if qt.scale_col is not None:
        out["scale_col_bytes"] = qt.scale_col.cpu().numpy()
    return out


def expected_scale_bytes(kind: int, ref: dict, which: str) -> np.ndarray | None:
    """The oracle's scale buffer of a copy in the library's byte layout."""
    if kind == O.BLOCK_1x128:
        return ref["scale_" + which + "_packed"].astype(np.float32).view(np.uint8).ravel()
    if kind == O.BLOCK_128x128:
        return np.ascontiguousarray(ref["scale_" + which], dtype=np.float32).view(np.uint8).ravel()
    if kind == O.MXFP8_1x32:
        return ref["scale_" + which + "_packed"].ravel()
    if kind in (O.PERCHANNEL_CURRENT, O.BLOCK_GENERIC):
        return np.ascontiguousarray(ref["scale_" + which + "_packed"], dtype=np.float32).view(np.uint8).ravel()
    return None


def assert_quant_equal(kind: int, got: dict, ref: dict, rowwise: bool, colwise: bool, ctx=""):
    """Bit-exact comparison of every byte, scale and counter."""
    def diff_msg(a, b, name):
        bad = np.flatnonzero(a.ravel() != b.ravel())
        i = bad[0]
        return f"{ctx} {name}: {bad.size} mismatches, first at flat {i}: got {a.ravel()[i]!r} want {b.ravel()[i]!r}"

    if rowwise:
        assert got["data_row"].shape == ref["data_row"].shape
        assert np.array_equal(got["data_row"], ref["data_row"]), diff_msg(got["data_row"], ref["data_row"], "data_row")
    if colwise:
        assert got["data_col"].shape == ref["data_col"].shape
        assert np.array_equal(got["data_col"], ref["data_col"]), diff_msg(got["data_col"], ref["data_col"], "data_col")
    for which, on in (("row", rowwise), ("col", colwise)):
        if not on:
            continue
        exp = expected_scale_bytes(kind, ref, which)
        if exp is None:
            continue
        g = got["scale_" + which + "_bytes"][:exp.size]
        assert g.size == exp.size, f"{ctx} scale_{which} size {g.size} vs {exp.size}"
        assert np.array_equal(g, exp), diff_msg(g, exp, "scale_" + which)
    if kind in (O.PERTENSOR_CURRENT, O.PERTENSOR_DELAYED):
        for k in ("amax", "scale", "scale_inv"):
            assert np.float32(got[k]).view(np.uint32) == np.float32(ref[k]).view(np.uint32), \
                f"{ctx} {k}: got {got[k]!r} want {ref[k]!r}"
    assert got["nonfinite"] == ref["nonfinite"], f"{ctx} nonfinite {got['nonfinite']} vs {ref['nonfinite']}"
    assert got["sat_row"] == ref["sat_row"], f"{ctx} sat_row {got['sat_row']} vs {ref['sat_row']}"
    assert got["sat_col"] == ref["sat_col"], f"{ctx} sat_col {got['sat_col']} vs {ref['sat_col']}"
