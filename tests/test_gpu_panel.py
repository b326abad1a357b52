"""The one-product panel kernel (one CTA per 32-row panel, its warps sharing
out the panel's block quads) against the CPU oracle and against the streaming
kernel, through the C ABI.

A single product of few rows goes to the panel kernel; the same product
launched together with one whose row is too long for it goes to the
streaming kernel.  Both must
give the oracle's bits: every output of the two launches is compared with the
other, and every output with the (threaded) oracle.  The shapes cover every warp
count (16, 8, 4) with quad and half-quad work units, fewer units than warps,
warps with several units, ragged rows, the longest row the kernel takes
(156 blocks), and CTAs that take several consecutive panels of a product
(5 and 7, with a last CTA of fewer), whose table is built once by the CTA.
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
                            f"got {got.ravel()[diff[:5]]} want {want.ravel()[diff[:5]]}")


# (rows, n, Q1_0 warps per CTA, blocks per work unit and panels per CTA on a
# 152-SM GB300); the test also requires that the launcher on the device it
# runs on picks the panel kernel.
SHAPES = [(1, 128, 4, 2, 1), (33, 384, 4, 2, 1), (256, 1024, 4, 2, 1), (300, 1536, 8, 2, 1),
          (3000, 2048, 8, 2, 1), (1000, 640, 4, 2, 1), (1024, 4096, 16, 2, 1), (4096, 4096, 16, 2, 1),
          (14336, 4096, 8, 4, 1), (18000, 4096, 4, 4, 1), (8192, 8192, 8, 4, 1), (9000, 2048, 8, 2, 1),
          (22000, 4096, 16, 2, 5), (30000, 1024, 16, 4, 7), (4096, 14336, 16, 4, 1), (300, 19968, 16, 2, 1)]


def _run(fmt, packed, rows, n, x, q, d):
    """(panel-kernel output, streaming-kernel output) of one product: paired
    with a product whose row is too long for the panel kernel, the launch
    takes the streaming kernel."""
    alone = torch.full((rows,), float("nan"), device="cuda")
    paired = torch.full((rows,), float("nan"), device="cuda")
    dummy_rows, dummy_n = 32, 20096
    if fmt == "q1":
        dummy = binding.pack(dev(synth.weight_blocks(synth.rng_for(999), dummy_rows, dummy_n)), dummy_rows, dummy_n)
        multi = binding.gemv_multi
    else:
        dummy = binding.q2_pack(dev(synth.ternary_blocks(synth.rng_for(999), dummy_rows, dummy_n)), dummy_rows,
                                dummy_n)
        multi = binding.q2_gemv_multi
    dx = torch.zeros(dummy_n, device="cuda")
    dout = torch.empty(dummy_rows, device="cuda")
    multi([(packed, rows, n, x, q, d, alone)])
    multi([(packed, rows, n, x, q, d, paired), (dummy, dummy_rows, dummy_n, dx, None, None, dout)])
    torch.cuda.synchronize()
    return alone.cpu().numpy(), paired.cpu().numpy()


@pytest.mark.parametrize("rows,n,warps,unit,ppc", SHAPES)
@pytest.mark.parametrize("act", ["f32", "q8"])
def test_panel_q1_equals_streaming_and_oracle(rows, n, warps, unit, ppc, act):
    plan = binding.multi_plan([(rows, n)], sms=152)
    assert (plan["panel_warps"], plan["panel_unit_blocks"], plan["panel_panels"]) == (warps, unit, ppc)
    assert binding.multi_plan([(rows, n)])["panel_warps"] > 0, "this device's launcher takes the streaming kernel"
    rng = synth.rng_for(501, rows, n, len(act))
    blocks = synth.weight_blocks(rng, rows, n, "lognormal" if rows % 2 else "halfnormal")
    packed = binding.pack(dev(blocks), rows, n)
    if act == "f32":
        xh = synth.activations(rng, 1, n, outliers=0.01)
        q, d = oracle.q8_quantize(xh)
        args = (dev(xh[0]), None, None)
    else:
        q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.03)
        args = (None, dev(q[0]), dev(d[0].view(np.int16)))
    alone, paired = _run("q1", packed, rows, n, *args)
    bits_equal(alone, paired)
    bits_equal(alone, oracle.gemm_threaded(blocks, q, d)[0])


@pytest.mark.parametrize("rows,n,warps,unit,ppc", [s for s in SHAPES if s[0] * s[1] <= 4096 * 14336])
@pytest.mark.parametrize("act", ["f32", "q8"])
def test_panel_q2_equals_streaming_and_oracle(rows, n, warps, unit, ppc, act):
    """Q2_0 keeps up to 128 registers a thread, so its warp counts can be
    lower than Q1_0's; every shape here stays within its one-wave limit."""
    assert binding.multi_plan([(rows, n)], fmt="q2")["panel_warps"] > 0
    rng = synth.rng_for(502, rows, n)
    if rows * n > 4096 * 4096:
        tb = synth.ternary_blocks_fast(rng, rows, n)
    else:
        tb = synth.ternary_blocks(rng, rows, n, "lognormal")
    packed = binding.q2_pack(dev(tb), rows, n)
    if act == "f32":
        xh = synth.activations(rng, 1, n, outliers=0.01)
        q, d = oracle.q8_quantize(xh)
        args = (dev(xh[0]), None, None)
    else:
        q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.03)
        args = (None, dev(q[0]), dev(d[0].view(np.int16)))
    alone, paired = _run("q2", packed, rows, n, *args)
    bits_equal(alone, paired)
    bits_equal(alone, oracle.q2_gemv_threaded(tb, q[0], d[0]))


def test_panel_in_graph_with_dependent_launches():
    """Back-to-back panel launches in a CUDA graph, each reading the previous
    one's output as its activation (programmatic dependent launch), against
    the oracle run of the same chain."""
    rows = n = 4096
    rng = synth.rng_for(503)
    blocks = [synth.weight_blocks(rng, rows, n, "halfnormal") for _ in range(3)]
    packed = [binding.pack(dev(b), rows, n) for b in blocks]
    x0 = synth.activations(rng, 1, n)[0]
    bufs = [dev(x0)] + [torch.empty(rows, device="cuda") for _ in range(3)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(3):
            binding.gemv_multi([(packed[i], rows, n, bufs[i], None, None, bufs[i + 1])], stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    for b in bufs[1:]:
        b.fill_(float("nan"))
    with torch.cuda.graph(g):
        for i in range(3):
            binding.gemv_multi([(packed[i], rows, n, bufs[i], None, None, bufs[i + 1])])
    g.replay()
    torch.cuda.synchronize()
    x = x0
    for i in range(3):
        q, d = oracle.q8_quantize(x[None, :])
        want = oracle.gemv(blocks[i], q[0], d[0])
        bits_equal(bufs[i + 1].cpu().numpy(), want)
        x = want


@pytest.mark.parametrize("shapes", [
    [(4096, 4096), (1024, 4096), (1024, 4096)],  # q, k, v
    [(14336, 4096), (14336, 4096)],              # gate and up: six panels a CTA
    [(14336, 4096), (6000, 2048)],               # five a CTA, products of different n
    [(20000, 1024), (20000, 1024)],              # one panel a CTA, two waves
    [(2048, 4096), (1000, 14336), (33, 128)],
    [(300, 1024), (7, 384), (256, 1152), (1, 128), (100, 2048), (32, 640), (500, 1024), (64, 4096)]])
def test_panel_product_lists(shapes):
    """Several products in one panel launch (one CTA per panel of each, in
    one wave or two, or one CTA per several consecutive panels of a product),
    f32 and q8_0 activations mixed: every output against the oracle and
    against the same products launched one at a time."""
    plan = binding.multi_plan(shapes)
    assert plan["panel_warps"] > 0
    items, want, alone = [], [], []
    for i, (rows, n) in enumerate(shapes):
        rng = synth.rng_for(504, i, rows, n)
        blocks = synth.weight_blocks(rng, rows, n, "lognormal" if i % 2 else "halfnormal")
        packed = binding.pack(dev(blocks), rows, n)
        out = torch.full((rows,), float("nan"), device="cuda")
        if i % 3 == 1:
            q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.03)
            item = (packed, rows, n, None, dev(q[0]), dev(d[0].view(np.int16)), out)
        else:
            xh = synth.activations(rng, 1, n, outliers=0.01)
            q, d = oracle.q8_quantize(xh)
            item = (packed, rows, n, dev(xh[0]), None, None, out)
        items.append(item)
        want.append(oracle.gemv(blocks, q[0], d[0]))
        one = torch.full((rows,), float("nan"), device="cuda")
        binding.gemv_multi([item[:-1] + (one,)])
        alone.append(one)
    binding.gemv_multi(items)
    torch.cuda.synchronize()
    for item, w, one in zip(items, want, alone):
        bits_equal(item[-1].cpu().numpy(), w)
        bits_equal(one.cpu().numpy(), w)


def test_panel_q2_list_several_panels_a_cta():
    """Two Q2_0 products of 752 panels in all: five consecutive panels a CTA,
    152 CTAs, with Q2_0's two sign planes; every output against the oracle."""
    shapes = [(12000, 2048), (12000, 2048)]
    assert binding.multi_plan(shapes, sms=152, fmt="q2")["panel_panels"] == 5
    assert binding.multi_plan(shapes, fmt="q2")["panel_warps"] > 0
    items, want = [], []
    for i, (rows, n) in enumerate(shapes):
        rng = synth.rng_for(505, i)
        tb = synth.ternary_blocks(rng, rows, n, "lognormal")
        xh = synth.activations(rng, 1, n, outliers=0.01)
        q, d = oracle.q8_quantize(xh)
        out = torch.full((rows,), float("nan"), device="cuda")
        items.append((binding.q2_pack(dev(tb), rows, n), rows, n, dev(xh[0]), None, None, out))
        want.append(oracle.q2_gemv(tb, q[0], d[0]))
    binding.q2_gemv_multi(items)
    torch.cuda.synchronize()
    for item, w in zip(items, want):
        bits_equal(item[-1].cpu().numpy(), w)
