"""The path's sharding, emulated on gloo ranks on the CPU (world size 2).

The block-scaled linear layer shards with no exchange except two: the NVFP4 /
MOSS tensor amax (one max over shards) and the token-split weight gradient (one
sum of dW partials).  CTA-local NVFP4 needs no amax exchange at all.  Each rank runs the oracle on its shard; the combined
result must equal the unsharded oracle.  The benchmark's max-over-ranks timing
helper is checked the same way.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle as orc
        import workloads
        import bench

        def bits(t):
            return t.contiguous().view(torch.int16).numpy().view(np.uint16)

        # 1) tensor amax: max over row shards, then each shard quantized with the global amax
        X = workloads.draw("student_t3", (256, 512), 5)
        rows = slice(rank * 128, (rank + 1) * 128)
        local = torch.tensor([orc.amax_bf16(bits(X[rows]))], dtype=torch.float32)
        dist.all_reduce(local, op=dist.ReduceOp.MAX)
        full = orc.quantize(bits(X), "nvfp4")
        assert float(local) == full.amax
        part = orc.quantize(bits(X[rows]), "nvfp4", amax_in=float(local))
        assert np.array_equal(part.codes, full.codes[rows]) and np.array_equal(part.sf_logical, full.sf_logical[rows])
        assert part.tensor_scale == full.tensor_scale

        # 2) weight gradient split along tokens: sum of per-shard dW partials
        dY = workloads.draw("student_t3", (512, 384), 6, 1e-3)
        Xw = workloads.draw("normal", (512, 256), 7)
        toks = slice(rank * 256, (rank + 1) * 256)
        for fmt in ("mxfp8", "mxfp4"):
            pa = orc.quantize(bits(dY[toks]), fmt, "col")
            pb = orc.quantize(bits(Xw[toks]), fmt, "col")
            c, _ = orc.gemm(pa, pb)
            t = torch.from_numpy(c)
            dist.all_reduce(t, op=dist.ReduceOp.SUM)
            ref, _ = orc.gemm(orc.quantize(bits(dY), fmt, "col"), orc.quantize(bits(Xw), fmt, "col"))
            assert np.allclose(t.numpy(), ref, rtol=1e-12, atol=1e-300)

        # 3) CTA-local NVFP4: row shards aligned to the 128-row regions need no
        #    exchange at all; each rank's result is its slice of the unsharded one
        Xl = workloads.draw("student_t3", (512, 256), 8)
        rows4 = slice(rank * 256, (rank + 1) * 256)
        fullq = orc.quantize(bits(Xl), "nvfp4_local")
        partq = orc.quantize(bits(Xl[rows4]), "nvfp4_local")
        assert np.array_equal(partq.codes, fullq.codes[rows4])
        assert np.array_equal(partq.sf_logical, fullq.sf_logical[rows4])
        assert np.array_equal(partq.tensor_scale, fullq.tensor_scale[rank * 2:(rank + 1) * 2])

        # 4) the benchmark's job time is the slowest rank's
        assert bench.reduce_max(10.0 + rank, world) == 10.0 + world - 1
        q.put((rank, "ok"))
    except Exception as e:  # report to the parent instead of hanging the group
        q.put((rank, repr(e)))
    finally:
        dist.destroy_process_group()


def test_sharded_oracle_matches_unsharded_on_two_gloo_ranks():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=240)
    results = dict(q.get(timeout=5) for _ in procs)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert results == {0: "ok", 1: "ok"}, results
