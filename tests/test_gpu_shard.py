"""Row sharding on one GPU: the outputs of a matrix's row shards, each packed
and multiplied on its own, concatenate to the unsharded product bit for bit
(bankML "docs/modules/gpu.md", "Limitations": a share of every matrix's rows
per card keeps each output element one card's exact dot product).  The
multi-card gather is tested on CPU (tests/test_shard_cpu.py); this run has one
GPU, so the sharded class is checked at world size 1."""
import os
import socket

import numpy as np
import pytest
import torch

import oracle
from decode_q1_gemv_gb300 import binding, synth
from decode_q1_gemv_gb300.shard import ShardedQ1Linear, row_ranges

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("rows,n,nvec", [(4096, 4096, 1), (14336, 4096, 1), (1000, 14336, 1), (4096, 4096, 16),
                                         (14336, 4096, 64)])
@pytest.mark.parametrize("world", [2, 3, 5])
def test_shard_outputs_concatenate_to_unsharded(rows, n, nvec, world):
    rng = synth.rng_for(910, rows, n, nvec)
    blocks = synth.weight_blocks(rng, rows, n, "lognormal")
    x = synth.activations(rng, nvec, n)
    q, d = binding.quantize(dev(x))
    full = binding.gemm_small(binding.pack(dev(blocks), rows, n), rows, n, q, d) if nvec > 1 else \
        binding.gemv(binding.pack(dev(blocks), rows, n), rows, n, q[0], d[0])[None, :]
    parts = []
    for r0, r1 in row_ranges(rows, world):
        if r1 == r0:
            continue
        packed = binding.pack(dev(blocks[r0:r1]), r1 - r0, n)
        parts.append(binding.gemm_small(packed, r1 - r0, n, q, d) if nvec > 1 else
                     binding.gemv(packed, r1 - r0, n, q[0], d[0])[None, :])
    got = torch.cat(parts, dim=1).cpu().numpy()
    want = full.cpu().numpy()
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    if nvec == 1:
        wq, wd = oracle.q8_quantize(x)
        assert np.array_equal(got[0].view(np.uint32), oracle.gemm_threaded(blocks, wq, wd)[0].view(np.uint32))


def test_sharded_linear_world_one():
    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        rows, n = 3000, 2048
        rng = synth.rng_for(911)
        blocks = synth.weight_blocks(rng, rows, n)
        lin = ShardedQ1Linear(torch.from_numpy(blocks))
        q, d = binding.quantize(dev(synth.activations(rng, 4, n)))
        want = binding.gemm_small(binding.pack(dev(blocks), rows, n), rows, n, q, d)
        got = lin(q, d)
        assert torch.equal(got.view(torch.int32), want.view(torch.int32))
    finally:
        dist.destroy_process_group()
