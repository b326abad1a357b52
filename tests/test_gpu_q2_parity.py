"""Parity of the Q2_0 (ternary) CUDA path with the CPU oracle, through the C ABI.

The format and its row product are this library's reading of the pages'
Q2_0 (bankML "docs/modules/gpu.md", "Advantages and efficiency" and
"Limitations" name it without defining it): 34-byte blocks of an fp16 scale
and 2-bit codes 0/1/2 = -1/0/+1, and the Q1_0 chain over ternary lane sums.
Every output is compared bit for bit with oracle.q2_gemv / q2_gemv_threaded.
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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits_equal(got, want):
    got = np.asarray(got, dtype=np.float32)
    want = np.asarray(want, dtype=np.float32)
    assert got.shape == want.shape
    diff = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
    assert diff.size == 0, (f"{diff.size} of {got.size} outputs differ; first at {diff[:5]}: "
                            f"gpu {got.ravel()[diff[:5]]} oracle {want.ravel()[diff[:5]]}")


@pytest.mark.parametrize("rows,n", [(1, 128), (33, 384), (256, 512), (300, 1152), (4097, 640)])
def test_pack_unpack_round_trip(rows, n):
    tb = synth.ternary_blocks(synth.rng_for(401, rows), rows, n)
    packed = binding.q2_pack(dev(tb), rows, n)
    assert packed.numel() == binding.q2_packed_bytes(rows, n) == (-(-rows // 256) * 256) * (-(-(n // 128) // 4) * 4) * 34
    back = binding.q2_unpack(packed, rows, n)
    assert np.array_equal(back.cpu().numpy(), tb)


def test_pack_rejects_code_three():
    rows, n = 40, 256
    tb = synth.ternary_blocks(synth.rng_for(402), rows, n)
    tb[7, 1, 5] |= 0x30  # element 4*3+2 = 14 of block 1 of row 7 gets code 3
    tb[30, 0, 9] |= 0x0C
    with pytest.raises(binding.Q1Error, match="row 7 block 1 holds the code 3"):
        binding.q2_pack(dev(tb), rows, n)
    ok = synth.ternary_blocks(synth.rng_for(403), rows, n)
    binding.q2_pack(dev(ok), rows, n)  # the rejection does not stick to the next call


def test_pack_rejects_non_finite_scale():
    rows, n = 40, 256
    tb = synth.ternary_blocks(synth.rng_for(404), rows, n)
    tb[12, 1, 0], tb[12, 1, 1] = 0x00, 0xFE   # NaN
    with pytest.raises(binding.Q1Error, match="row 12 block 1: the fp16 weight scale is not finite"):
        binding.q2_pack(dev(tb), rows, n)


@pytest.mark.parametrize("rows,n", [(1, 128), (7, 256), (33, 384), (300, 1024), (1000, 4096), (513, 14336),
                                    (70, 17408), (2600, 20480)])
@pytest.mark.parametrize("regime", ["halfnormal", "lognormal"])
def test_gemv_parity(rows, n, regime):
    """n above 16384 builds the activation table in chunks inside the tile loop."""
    rng = synth.rng_for(410, rows, n, len(regime))
    tb = synth.ternary_blocks(rng, rows, n, regime)
    q, d = synth.raw_quants(rng, 1, n, scale=regime, m128_frac=0.03)
    out = binding.q2_gemv(binding.q2_pack(dev(tb), rows, n), rows, n, dev(q[0]), dev(d[0].view(np.int16)))
    bits_equal(out.cpu().numpy(), oracle.q2_gemv(tb, q[0], d[0]))


@pytest.mark.parametrize("p_zero", [0.0, 0.5, 0.95, 1.0])
def test_gemv_zero_fractions(p_zero):
    rows, n = 700, 2048
    rng = synth.rng_for(411, int(p_zero * 100))
    tb = synth.ternary_blocks(rng, rows, n, "lognormal", p_zero=p_zero)
    x = synth.activations(rng, 1, n, outliers=0.01)
    q, d = oracle.q8_quantize(x)
    out = binding.q2_gemv(binding.q2_pack(dev(tb), rows, n), rows, n, dev(q[0]), dev(d[0].view(np.int16)))
    want = oracle.q2_gemv(tb, q[0], d[0])
    bits_equal(out.cpu().numpy(), want)
    if p_zero == 1.0:
        assert np.array_equal(want.view(np.uint32), np.zeros(rows, dtype=np.uint32))


def test_no_zero_weights_equal_q1_0_kernel():
    """Codes 0/2 only: the Q2_0 kernel and the Q1_0 kernel on the same signs
    give the same bits (both against their oracles as well)."""
    rows, n = 1024, 4096
    rng = synth.rng_for(412)
    nb = n // 128
    bits = rng.integers(0, 2, size=(rows, nb, 128)).astype(np.uint8)
    scales = synth.block_scales(rng, (rows, nb), "lognormal")
    tb = synth.assemble_ternary_blocks(scales, 2 * bits)
    b1 = synth.assemble_blocks(scales, synth.sign_bytes_from_bits(bits))
    x = synth.activations(rng, 1, n)
    q, d = oracle.q8_quantize(x)
    qd, dd = dev(q[0]), dev(d[0].view(np.int16))
    a = binding.q2_gemv(binding.q2_pack(dev(tb), rows, n), rows, n, qd, dd)
    b = binding.gemv(binding.pack(dev(b1), rows, n), rows, n, qd, dd)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("size", ["small", "large"])
def test_gemv_multi_products(size):
    """Several Q2_0 products in one launch, f32 activations (quantized in the
    kernel) and q8_0 ones mixed; 'large' has enough rows for the big-launch
    rows per thread and host-placed CTA ranges."""
    rng0 = np.random.default_rng(420 if size == "small" else 421)
    if size == "small":
        shapes = [(int(rng0.integers(1, 2500)), 128 * int(rng0.choice([1, 3, 8, 32, 112]))) for _ in range(11)]
    else:
        shapes = [(int(rng0.choice([4096, 8192, 16384])), 128 * int(rng0.choice([1, 2, 4, 9]))) for _ in range(12)]
    items, want = [], []
    for i, (rows, n) in enumerate(shapes):
        rng = synth.rng_for(422, i)
        tb = synth.ternary_blocks(rng, rows, n, "lognormal" if i % 2 else "halfnormal")
        out = torch.full((rows,), float("nan"), device="cuda")
        packed = binding.q2_pack(dev(tb), rows, n)
        if i % 3 == 2:
            q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.03)
            items.append((packed, rows, n, None, dev(q[0]), dev(d[0].view(np.int16)), out))
        else:
            x = synth.activations(rng, 1, n, outliers=0.01)
            q, d = oracle.q8_quantize(x)
            items.append((packed, rows, n, dev(x[0]), None, None, out))
        want.append(oracle.q2_gemv(tb, q[0], d[0]))
    binding.q2_gemv_multi(items)
    torch.cuda.synchronize()
    for item, w in zip(items, want):
        bits_equal(item[-1].cpu().numpy(), w)


@pytest.mark.parametrize("rows,n", [(14336, 4096), (4096, 14336), (128256, 4096)])
def test_full_size(rows, n):
    """Llama-3-8B shapes in Q2_0 as the set benchmark draws them: every row
    against the threaded oracle."""
    rng = synth.rng_for(430, rows, n)
    tb = synth.ternary_blocks_fast(rng, rows, n)
    x = synth.activations(rng, 1, n)
    q, d = oracle.q8_quantize(x)
    packed = binding.q2_pack(dev(tb), rows, n)
    out = torch.empty(rows, device="cuda")
    binding.q2_gemv_multi([(packed, rows, n, dev(x[0]), None, None, out)])
    bits_equal(out.cpu().numpy(), oracle.q2_gemv_threaded(tb, q[0], d[0]))


def test_q2_decode_set_full():
    """The 225-product decode set with Q2_0 weights in one launch, as the
    benchmark times it (CUDA graph): every output of every product against the
    threaded oracle."""
    from decode_q1_gemv_gb300.decode_set import DecodeSet
    ds = DecodeSet(seed=3, fmt="q2")
    g = ds.capture("set")
    ds.out_all.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    got_all = ds.out_all.cpu().numpy()
    for i, (name, rows, n) in enumerate(ds.shapes):
        q, d = oracle.q8_quantize(ds.host_x(i)[None, :])
        want = oracle.q2_gemv_threaded(ds.host_blocks(i), q[0], d[0])
        bits_equal(got_all[ds.out_off[i]:ds.out_off[i] + rows], want)
    del ds, g
    torch.cuda.empty_cache()


def test_device_status_clean():
    assert binding.device_status() == 0
