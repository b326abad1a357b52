"""The tensor-core kernel of the batched product against the dp4a kernel and the
CPU oracle, through the C ABI.

q1_0_gemm_small runs one of two kernels; q1_gemm_small_kernel forces either.
The tensor-core kernel takes a block's per-lane sub-block chain from one f16
MMA accumulator when an activation-only bound shows every partial sum of the
chain is exact in f32, and the dp4a chain of the other kernel for the rest of
the blocks (a -128 quant, scales 512 or more, or the bound failing).  Every
case here runs both kernels on the same inputs: their outputs must be
bit-identical to each other and to the oracle (bankML "docs/modules/gpu.md",
"kernels.rs -- the Q1_0 kernels", first and second bullets; "How it is
verified": every row of every shape).
"""
import numpy as np
import pytest
import torch

import oracle
from decode_q1_gemv_gb300 import binding, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()
    oracle.build()
    yield
    binding.gemm_small_kernel("auto")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits_equal(got, want):
    got = np.asarray(got, dtype=np.float32)
    want = np.asarray(want, dtype=np.float32)
    assert got.shape == want.shape
    diff = np.argwhere(got.view(np.uint32) != want.view(np.uint32))
    assert diff.size == 0, f"{len(diff)} outputs differ; first (vector, row) {diff[:5].tolist()}"


def both_kernels(blocks, q, d):
    rows, nb, _ = blocks.shape
    n = nb * 128
    packed = binding.pack(dev(blocks), rows, n)
    qd, dd = dev(q), dev(d.view(np.int16))
    outs = {}
    for k in ("dp4a", "tensor"):
        binding.gemm_small_kernel(k)
        outs[k] = binding.gemm_small(packed, rows, n, qd, dd).cpu().numpy()
    binding.gemm_small_kernel("auto")
    return outs["dp4a"], outs["tensor"]


def lane_bound(q, d):
    """Per (vector, block) the largest lane value of the exactness bound,
    sum_k (m_k << (e_k - e_min)) * sum_i |q|, computed here from the fp16
    fields; -1 where a -128 quant or a scale >= 512 rules the block out."""
    nvec, n = q.shape
    nb = n // 128
    qb = q.astype(np.int64).reshape(nvec, nb, 4, 8, 4)
    h = d.astype(np.int64).reshape(nvec, nb, 4)
    E = (h >> 10) & 31
    m = np.where(E > 0, 1024 | (h & 1023), h & 1023)
    e = np.maximum(E, 1)
    c = m << (e - e.min(axis=2, keepdims=True))
    S = np.abs(qb).sum(axis=4)                       # [v, b, k, lane]
    T = (c[..., None] * S).sum(axis=2).max(axis=2)   # [v, b]
    bad = (qb == -128).any(axis=(2, 3, 4)) | (E > 23).any(axis=2)
    return np.where(bad, -1, T)


def activations_q(rng, nvec, n, regime):
    if regime == "raw":
        return synth.raw_quants(rng, nvec, n, scale="lognormal", m128_frac=0.03)
    x = synth.activations(rng, nvec, n)
    if regime == "layer":      # scales spread per 32 values: most blocks outside the bound
        x *= np.exp(rng.standard_normal((nvec, n // 32))).repeat(32, axis=1).astype(np.float32)
    elif regime == "mixed":    # every other block spread, one -128 planted below
        f = np.exp(2.0 * rng.standard_normal((nvec, n // 32))).astype(np.float32)
        f[:, (np.arange(n // 32) // 4) % 2 == 0] = 1.0
        x *= f.repeat(32, axis=1)
    q, d = oracle.q8_quantize(x)
    if regime == "mixed":
        q[nvec // 2, 3 * 128 + 17] = -128
    return q, d


@pytest.mark.parametrize("rows,n,nvec,regime", [
    (300, 1152, 16, "raw"),
    (1000, 1024, 33, "quantized"),
    (131, 384, 8, "quantized"),
    (4096, 4096, 64, "quantized"),
    (777, 2048, 16, "layer"),
    (2000, 4096, 20, "mixed"),
    (1, 128, 17, "quantized"),
    (260, 1408, 16, "quantized"),   # 11 blocks: the issuers' last round holds five
])
def test_tensor_kernel_equals_dp4a_and_oracle(rows, n, nvec, regime):
    rng = synth.rng_for(601, rows, n, nvec, len(regime))
    blocks = synth.weight_blocks(rng, rows, n, "lognormal" if rows % 2 else "halfnormal")
    q, d = activations_q(rng, nvec, n, regime)
    T = lane_bound(q, d)
    if regime == "quantized":
        assert (T >= 0).all() and (T <= 1 << 22).all()     # every block on the MMA path
    if regime == "mixed":
        assert (T < 0).any() and (T > 1 << 22).any() and ((T >= 0) & (T <= 1 << 22)).any()
    got_dp4a, got_tc = both_kernels(blocks, q, d)
    want = oracle.gemm_threaded(blocks, q, d)
    bits_equal(got_tc, want)
    bits_equal(got_dp4a, want)


def test_tensor_kernel_many_units_per_cta():
    """More 128-row x 16-vector units than CTAs: the persistent CTAs carry
    their pipelines across units."""
    rows, n, nvec = 128256, 512, 64
    rng = synth.rng_for(602)
    blocks = synth.weight_blocks(rng, rows, n, "lognormal")
    q, d = activations_q(rng, nvec, n, "quantized")
    _, got = both_kernels(blocks, q, d)
    bits_equal(got, oracle.gemm_threaded(blocks, q, d))


def test_tensor_kernel_at_the_exactness_bound():
    """Activations built so the bound lands on both sides of 2^22 in many
    blocks (fp16 scales one to two binades apart within a block, quants near
    the largest): the blocks just inside use the single-accumulator MMA, the
    ones just outside the dp4a chain, and both give the oracle's bits."""
    rng = synth.rng_for(603)
    rows, n, nvec = 512, 8192, 16
    nb = n // 128
    mant = rng.integers(900, 1024, size=(nvec, nb, 4))
    expo = 8 + rng.integers(0, 3, size=(nvec, nb, 4))          # 2^-7 .. 2^-5
    d = ((expo << 10) | mant).astype(np.uint16)
    mag = rng.integers(60, 128, size=(nvec, n))
    q = (mag * np.where(rng.integers(0, 2, size=(nvec, n)) == 1, 1, -1)).astype(np.int8)
    # scale each block's quants so the bound spreads around 2^22
    T = lane_bound(q, d.reshape(nvec, -1))
    target = rng.uniform(0.8, 1.25, size=(nvec, nb)) * (1 << 22)
    f = np.clip(target / np.maximum(T, 1), 0.05, 1.0)
    q = np.clip(np.round(q.astype(np.float64).reshape(nvec, nb, 128) * f[..., None]), -127, 127).astype(np.int8)
    q = q.reshape(nvec, n)
    d = d.reshape(nvec, -1)
    T = lane_bound(q, d)
    near = np.abs(np.log2(np.maximum(T, 1)) - 22) < 0.2
    assert ((T <= 1 << 22) & near).sum() > 20 and ((T > 1 << 22) & near).sum() > 20
    blocks = synth.weight_blocks(rng, rows, n, "lognormal")
    got_dp4a, got_tc = both_kernels(blocks, q, d)
    want = oracle.gemm_threaded(blocks, q, d)
    bits_equal(got_tc, want)
    bits_equal(got_dp4a, want)


def test_kernel_choice_knob():
    assert binding.gemm_small_kernel("tensor") == "auto"
    assert binding.gemm_small_kernel("dp4a") == "tensor"
    assert binding.gemm_small_kernel("auto") == "dp4a"
    with pytest.raises(binding.Q1Error):
        binding._check(binding.load().q1_gemm_small_kernel(3), "q1_gemm_small_kernel")


def test_tensor_kernel_rejects_oversized_scratch():
    """Forced onto the tensor core, a shape whose scratch would exceed the
    limit is refused before anything is launched."""
    rows, n, nvec = 1, 1 << 20, 64
    packed = torch.zeros(binding.packed_bytes(rows, n), dtype=torch.uint8, device="cuda")
    q = torch.zeros((nvec, n), dtype=torch.int8, device="cuda")
    d = torch.zeros((nvec, n // 32), dtype=torch.int16, device="cuda")
    binding.gemm_small_kernel("tensor")
    try:
        with pytest.raises(binding.Q1Error, match="scratch"):
            binding.gemm_small(packed, rows, n, q, d)
    finally:
        binding.gemm_small_kernel("auto")


@pytest.mark.parametrize("kernel", ["dp4a", "tensor"])
def test_outputs_written_once_and_guard_untouched(kernel):
    """Ragged rows (the last 128-row tile holds 44) and a ragged vector group
    (19 vectors: the second group of 16 holds 3): every output is written
    with the oracle's bits and nothing past the output array changes."""
    rows, n, nvec = 300, 1024, 19
    rng = synth.rng_for(606)
    blocks = synth.weight_blocks(rng, rows, n, "lognormal")
    q, d = activations_q(rng, nvec, n, "quantized")
    packed = binding.pack(dev(blocks), rows, n)
    guard = 512
    buf = torch.full((nvec * rows + guard,), float("nan"), device="cuda")
    prev = binding.gemm_small_kernel(kernel)
    try:
        binding.gemm_small(packed, rows, n, dev(q), dev(d.view(np.int16)), out=buf[:nvec * rows])
    finally:
        binding.gemm_small_kernel(prev)
    host = buf.cpu().numpy()
    assert not np.any(np.isnan(host[:nvec * rows]))
    assert np.all(np.isnan(host[nvec * rows:]))
    bits_equal(host[:nvec * rows].reshape(nvec, rows), oracle.gemm_threaded(blocks, q, d))


def test_device_status_clean():
    assert binding.device_status() == 0
