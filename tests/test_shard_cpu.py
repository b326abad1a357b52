"""Row sharding across ranks (bankML "docs/modules/gpu.md", "Limitations": each
card takes a share of every matrix's rows, so each output element stays one
card's exact dot product): the row split, and the all-gather that assembles the
full output, on CPU with gloo at world sizes 2 and 3.  Each rank computes its
rows with the oracle; the gathered vector must equal the unsharded oracle
output bit for bit."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

from decode_q1_gemv_gb300.shard import ROW_ALIGN, row_ranges  # noqa: E402


@pytest.mark.parametrize("rows", [1, 255, 256, 257, 1000, 4096, 14336, 128256])
@pytest.mark.parametrize("world", [1, 2, 3, 4, 8])
def test_row_ranges_cover_in_aligned_balanced_pieces(rows, world):
    rr = row_ranges(rows, world)
    assert len(rr) == world
    assert rr[0][0] == 0 and rr[-1][1] == rows
    for (a0, a1), (b0, b1) in zip(rr, rr[1:]):
        assert a1 == b0 and a0 <= a1
    for a, b in rr:
        assert a % ROW_ALIGN == 0 or a == rows
    sizes = [(b - a + ROW_ALIGN - 1) // ROW_ALIGN for a, b in rr]
    assert max(sizes) - min(sizes) <= 1


def test_row_ranges_rejects_bad_arguments():
    for args in ((0, 2), (10, 0), (10, 2, 0)):
        with pytest.raises(ValueError):
            row_ranges(*args)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q, rows, n, nvec):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import oracle
    from decode_q1_gemv_gb300 import synth
    from decode_q1_gemv_gb300.shard import gather_rows, row_ranges
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = synth.rng_for(900, rows, n)
    blocks = synth.weight_blocks(rng, rows, n, "lognormal")        # every rank draws the same matrix
    qq, d = synth.raw_quants(rng, nvec, n, scale="lognormal", m128_frac=0.02)
    ranges = row_ranges(rows, world)
    r0, r1 = ranges[rank]
    local = oracle.gemm(blocks[r0:r1], qq, d) if r1 > r0 else np.zeros((nvec, 0), np.float32)
    full = gather_rows(torch.from_numpy(np.ascontiguousarray(local)), ranges).numpy()
    want = oracle.gemm(blocks, qq, d)
    ok = full.shape == want.shape and np.array_equal(full.view(np.uint32), want.view(np.uint32))
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, bool(ok)))


@pytest.mark.parametrize("world,rows,n,nvec", [(2, 700, 384, 3), (3, 300, 256, 1), (2, 100, 128, 2)])
def test_gather_rows_gloo(world, rows, n, nvec):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, rows, n, nvec)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    res = dict(q.get(timeout=10) for _ in range(world))
    assert all(res.values()) and len(res) == world
