"""The device's saturating round-to-nearest-even fp32 -> FP8 conversion against
the oracle's bit-level encoder on all 2^32 fp32 bit patterns, both formats
(E4M3 / E5M2 layouts: "2025 FP8 quantized-training guide", sec. 1.1)."""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

import oracle as O

pytestmark = pytest.mark.gpu

CHUNK = 1 << 28


def _oracle_chunk(start: int, count: int, fmt: int, pool) -> np.ndarray:
    parts = 32
    step = count // parts
    futs = [pool.submit(O.encode_bits_range, start + i * step, step, fmt) for i in range(parts)]
    return np.concatenate([f.result() for f in futs])


@pytest.mark.parametrize("fmt", [O.E4M3, O.E5M2])
def test_cast_all_fp32_bit_patterns(fmt):
    from fp8_scaled_quantization_quantize_gb300 import api
    O.lib()
    out = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    host = torch.empty(CHUNK, dtype=torch.uint8, pin_memory=True)
    with cf.ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as pool:
        for c in range((1 << 32) // CHUNK):
            start = c * CHUNK
            api.cast_f32_bits(start, CHUNK, fmt, out)
            host.copy_(out)
            torch.cuda.synchronize()
            ref = _oracle_chunk(start, CHUNK, fmt, pool)
            got = host.numpy()
            if not np.array_equal(got, ref):
                bad = np.flatnonzero(got != ref)
                i = bad[0]
                raise AssertionError(f"{bad.size} mismatches in chunk {c}; first bits 0x{start + i:08x}: "
                                     f"got 0x{got[i]:02x} want 0x{ref[i]:02x}")
