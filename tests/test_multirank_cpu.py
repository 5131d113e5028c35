"""The path's one cross-replica exchange, on CPU ranks (gloo, world size 2).

When a per-tensor recipe's tensor is sharded across data-parallel ranks
(rows split), every rank must quantize with the same scale: the shard amaxes
are combined by a max-allreduce before the delayed-scaling history update
("2025 FP8 quantized-training guide", sec. 2.1: the scale comes from the
amax history of the tensor).  Each rank computes its shard's amax with the
oracle, all-reduces the max, updates its own copy of the state, and casts its
shard; the states and the concatenated codes must equal the single-process
oracle run on the whole tensor.  Blockwise / MX recipes need no exchange:
their blocks never straddle a row split at a multiple of the block height.
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
