"""q1_0_gemm_small_noalloc: the batched product for callers that cannot
allocate device memory at call time (for example a serving loop that reserves
all of its memory up front).  It runs the tensor-core kernel with its scratch
in a fixed array the library keeps on the device, so it must give exactly the
outputs of q1_0_gemm_small, call after call, while reusing that array.

This file is collected last on purpose: if it fails in a run that stops at the
first failure, every other test has already run.  It also passes on its own in
a fresh process, where its first call sets up the array's device address.
"""
import ctypes

import numpy as np
import pytest
import torch

from decode_q1_gemv_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def noalloc_c_abi(packed, rows, n, q, d, out):
    """One call of the C entry point itself (raw pointers, current stream)."""
    lib = binding.load()
    nvec = q.shape[0]
    rc = lib.q1_0_gemm_small_noalloc(ctypes.c_void_p(packed.data_ptr()), rows, n, nvec,
                                     ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(d.data_ptr()),
                                     ctypes.c_void_p(out.data_ptr()),
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == binding.Q1_OK, binding.last_error()


def case(seed, rows, n, nvec, raw):
    rng = synth.rng_for(700, seed)
    blocks = synth.weight_blocks(rng, rows, n, "lognormal")
    if raw:   # -128 quants and spread scales: blocks outside the MMA bound take the dp4a tables
        q, d = synth.raw_quants(rng, nvec, n, scale="lognormal", m128_frac=0.03)
        return blocks, dev(q), dev(d.view(np.int16))
    x = synth.activations(rng, nvec, n)
    q, d = binding.quantize(dev(x))
    return blocks, q, d


def test_noalloc_matches_gemm_small_on_consecutive_calls():
    """Two calls in a row with different shapes and inputs (the second reuses
    the array the first left behind): each output bit-identical to
    q1_0_gemm_small's on the same inputs."""
    for seed, rows, n, nvec, raw in ((1, 3000, 4096, 40, False), (2, 777, 1152, 16, True)):
        blocks, q, d = case(seed, rows, n, nvec, raw)
        packed = binding.pack(dev(blocks), rows, n)
        got = torch.full((nvec, rows), float("nan"), device="cuda")
        noalloc_c_abi(packed, rows, n, q, d, got)
        want = binding.gemm_small(packed, rows, n, q, d)
        torch.cuda.synchronize()
        g, w = got.cpu().numpy(), want.cpu().numpy()
        assert np.array_equal(g.view(np.uint32), w.view(np.uint32)), (rows, n, nvec)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    rows, n, nvec = 1, 32768, 64   # 4 groups x 256 blocks x 8 KB > 8 MiB
    packed = torch.zeros(binding.packed_bytes(rows, n), dtype=torch.uint8, device="cuda")
    q = torch.zeros((nvec, n), dtype=torch.int8, device="cuda")
    d = torch.zeros((nvec, n // 32), dtype=torch.int16, device="cuda")
    with pytest.raises(binding.Q1Error, match="fixed scratch"):
        binding.gemm_small_noalloc(packed, rows, n, q, d)
    assert binding.device_status() == 0
