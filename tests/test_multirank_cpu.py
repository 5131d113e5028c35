"""The path's cross-replica exchanges, on CPU ranks (gloo, world size 2).

When a per-tensor recipe's tensor is sharded across data-parallel ranks
(rows split), every rank must quantize with the same scale: the shard amaxes
are combined by a max-allreduce before the delayed-scaling history update
("2025 FP8 quantized-training guide", sec. 2.1: the scale comes from the
amax history of the tensor).  Each rank computes its shard's amax with the
oracle, all-reduces the max, updates its own copy of the state, and casts its
shard; the states and the concatenated codes must equal the single-process
oracle run on the whole tensor.  Blockwise / MX recipes need no exchange:
their blocks never straddle a row split at a multiple of the block height,
so ranks that quantize row shards and all-gather the FP8 codes and scales
(tensor parallelism's gather, in FP8) hold what one process quantizing the
whole tensor would.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O
from fp8_scaled_quantization_quantize_gb300 import inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _steps():
    mags = inputs.delayed_magnitudes(24)
    return [inputs.bf16_bits(inputs.normal_bf16((64, 96), 700 + t, float(mags[t, 0]))) for t in range(24)]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    st = O.Delayed(16, O.E4M3, 0)
    codes, scales = [], []
    for x in _steps():
        shard = np.ascontiguousarray(np.array_split(x, world, axis=0)[rank])
        s = st.scale
        q, amax, sat, nf = O.cast_scaled(shard, s, O.E4M3)
        t = torch.tensor([amax, float(nf)], dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        st.update(float(t[0]), int(t[1]))
        codes.append(q)
        scales.append(float(s))
    gathered = [None] * world
    dist.all_gather_object(gathered, (codes, scales, st.hist.tolist(), st.head))
    if rank == 0:
        out.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_sharded_delayed_scaling_matches_single_process():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    gathered = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ref = O.Delayed(16, O.E4M3, 0)
    for t, x in enumerate(_steps()):
        s = ref.scale
        qfull, amax, sat, nf = O.cast_scaled(x, s, O.E4M3)
        ref.update(amax, nf)
        for r in range(world):
            assert gathered[r][1][t] == float(s)
        assert np.array_equal(np.concatenate([gathered[r][0][t] for r in range(world)]), qfull)
    for r in range(world):
        assert gathered[r][2] == ref.hist.tolist() and gathered[r][3] == ref.head


def _gather_worker(rank, world, port, out):
    """Each rank quantizes its row shard (row-wise copy; shard edges on
    128-row boundaries) and the ranks all-gather the FP8 codes and their
    block scales: the exchange a tensor-parallel layer makes when it gathers
    an activation or a gradient in FP8 instead of bf16."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x = inputs.bf16_bits(inputs.normal_bf16((512, 384), 900, 1e-3))
    shard = np.ascontiguousarray(np.split(x, world, axis=0)[rank])
    mine = {}
    for name, kind, fmt in (("activation mx e4m3", O.MXFP8_1x32, O.E4M3),
                            ("gradient 1x128 e5m2", O.BLOCK_1x128, O.E5M2)):
        q = O.quantize(kind, fmt, shard, True, False)
        mine[name] = (q["data_row"], q["scale_row"], q["sat_row"])
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    if rank == 0:
        out.put(gathered)
    dist.barrier()
    dist.destroy_process_group()


def test_fp8_allgather_of_row_shards_equals_whole_tensor_quantize():
    """Gathering per-rank FP8 shards (codes + 1x32 / 1x128 scales) gives what
    quantizing the whole tensor gives: these blocks never cross a row
    boundary, so sharding rows needs no scale exchange ("2025 FP8
    quantized-training guide", sec. 4.1: quantize locally, then all-gather the
    FP8 bytes; E5M2 for the gradients)."""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_gather_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    gathered = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    x = inputs.bf16_bits(inputs.normal_bf16((512, 384), 900, 1e-3))
    for name, kind, fmt in (("activation mx e4m3", O.MXFP8_1x32, O.E4M3),
                            ("gradient 1x128 e5m2", O.BLOCK_1x128, O.E5M2)):
        whole = O.quantize(kind, fmt, x, True, False)
        codes = np.concatenate([g[name][0] for g in gathered])
        scales = np.concatenate([g[name][1] for g in gathered])
        assert np.array_equal(codes, whole["data_row"]), name
        assert np.array_equal(scales, whole["scale_row"]), name
        assert sum(g[name][2] for g in gathered) == whole["sat_row"], name
