"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Every comparison is element by element on the same seeded inputs: int8 quants
and fp16 scale bits byte for byte, f32 outputs bit for bit (the definition has
exactly one correct f32 per row; the tolerance is zero).  Small and ragged
shapes are compared in full; full-size workloads are compared on sampled rows
that the oracle computes one by one, in the launch configuration the benchmark
times.
"""
import numpy as np
import pytest
import torch

import oracle
from decode_q1_gemv_gb300 import binding, synth
from tests.golden.cases import load_cases

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    binding.load()
    oracle.build()


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bits_equal(got: np.ndarray, want: np.ndarray):
    got = np.asarray(got, dtype=np.float32)
    want = np.asarray(want, dtype=np.float32)
    assert got.shape == want.shape
    diff = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
    assert diff.size == 0, (f"{diff.size} of {got.size} outputs differ; first at {diff[:5]}: "
                            f"gpu {got.ravel()[diff[:5]]} oracle {want.ravel()[diff[:5]]}")


def gpu_gemv(blocks: np.ndarray, q: np.ndarray, d: np.ndarray) -> np.ndarray:
    rows, nb, _ = blocks.shape
    n = nb * 128
    packed = binding.pack(dev(blocks), rows, n)
    out = binding.gemv(packed, rows, n, dev(q.astype(np.int8)), dev(d.view(np.int16)))
    return out.cpu().numpy()


def gpu_gemm(blocks: np.ndarray, q: np.ndarray, d: np.ndarray) -> np.ndarray:
    rows, nb, _ = blocks.shape
    n = nb * 128
    packed = binding.pack(dev(blocks), rows, n)
    out = binding.gemm_small(packed, rows, n, dev(q.astype(np.int8)), dev(d.view(np.int16)))
    return out.cpu().numpy()


# ------------------------------------------------------------ self-check --
def test_library_self_check():
    rc, report = binding.verify(quick=False)
    assert rc == binding.Q1_OK, report
    lines = report.strip().splitlines()
    # first the exhaustive check of the kernels' quantizer rounding (all floats |t| < 2^22)
    assert lines[0] == "q8 rounding by adds: all 2499805184 floats with |t| < 2^22 equal roundf", report
    lines = lines[1:]
    assert len(lines) == 17 and all(line.endswith("bit-exact") for line in lines), report
    # both matrix-vector kernels: the last two shapes have too many rows for the panel kernel
    assert binding.multi_plan([(40000, 256)])["panel_warps"] == 0
    assert binding.multi_plan([(40000, 256)], fmt="q2")["panel_warps"] == 0
    assert binding.multi_plan([(9999, 1152)])["panel_warps"] > 0
    for kernel in ("q1_0_gemv ", "q1_0_gemm_small ", "q1_0_gemm_small_noalloc ", "q2_0_gemv "):
        assert any(line.startswith(kernel) for line in lines), (kernel, report)


def test_library_self_check_negative_control():
    """A corrupted packed buffer (one row's scales doubled after packing) must
    fail the self-check, and the report must name that row as the first that
    differs, case by case."""
    import re
    rc, report = binding.verify(quick=False, corrupt=True)
    assert rc == binding.Q1_MISMATCH, report
    corrupted = re.findall(r"^(\S+) (\d+)x(\d+): scales of row (\d+) doubled", report, re.M)
    differs = re.findall(r"^(\S+) (\d+)x(\d+) nvec=1 \S+: row (\d+) differs", report, re.M)
    assert len(corrupted) == 12 and corrupted == differs, report
    assert "nvec=16" in report and "bit-exact" in report  # the batched cases are left intact


def test_bounded_wait_gives_up_and_device_stays_usable():
    """The wait every product kernel uses, on a barrier nothing completes, gives
    up after its limit; the status is read on the host, and the product cases
    run right after it are bit-exact."""
    rc, report = binding.verify(quick=True, wait_probe=True)
    assert rc == binding.Q1_OK, report
    assert "gave up after" in report and report.count("bit-exact") == 3, report
    assert binding.device_status() == 0


# --------------------------------------------------------------- packing --
@pytest.mark.parametrize("rows,n", [(1, 128), (31, 384), (33, 1024), (100, 1152), (257, 4096), (64, 14336)])
def test_pack_unpack_round_trip(rows, n):
    blocks = synth.weight_blocks(synth.rng_for(101, rows, n), rows, n, "signed")
    packed = binding.pack(dev(blocks), rows, n)
    assert packed.numel() == binding.packed_bytes(rows, n)
    back = binding.unpack(packed, rows, n).cpu().numpy()
    assert np.array_equal(back, blocks)


@pytest.mark.parametrize("bad", [0x7C00, 0xFC00, 0x7E00, 0x7C01])
def test_pack_rejects_non_finite_scale(bad):
    """A block whose fp16 scale is +Inf, -Inf or NaN is rejected with an
    error naming the first such row and block (in row-major block order)."""
    rows, n = 300, 1024
    blocks = synth.weight_blocks(synth.rng_for(103), rows, n)
    for r, b in ((211, 5), (17, 6), (17, 2)):
        blocks[r, b, 0], blocks[r, b, 1] = bad & 0xFF, bad >> 8
    with pytest.raises(binding.Q1Error, match="row 17 block 2: the fp16 weight scale is not finite"):
        binding.pack(dev(blocks), rows, n)
    # the rejection belongs to that call only
    ok = synth.weight_blocks(synth.rng_for(104), rows, n)
    binding.pack(dev(ok), rows, n)


def test_pack_rejections_stay_per_call_across_streams():
    """Packs of a bad and a good matrix issued from two streams at once: the
    bad one is rejected and the good one is not."""
    rows, n = 4096, 4096
    bad = synth.weight_blocks(synth.rng_for(105), rows, n)
    bad[4000, 31, 1] = 0x7C
    bad[4000, 31, 0] = 0x00
    good = synth.weight_blocks(synth.rng_for(106), rows, n)
    bd, gd = dev(bad), dev(good)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with pytest.raises(binding.Q1Error, match="row 4000 block 31"):
            binding.pack(bd, rows, n, stream=s1)
        packed = binding.pack(gd, rows, n, stream=s2)
        assert np.array_equal(binding.unpack(packed, rows, n).cpu().numpy(), good)


# ---------------------------------------------------------- quantization --
QUANT_CASES = ["normal", "outliers", "tiny", "large", "zeros", "ties"]


def quant_case_activations(rng, case, nvec, n):
    """f32 activations of the named quantizer regime."""
    if case == "normal":
        x = synth.activations(rng, nvec, n)
    elif case == "outliers":
        x = synth.activations(rng, nvec, n, outliers=0.01)
    elif case == "tiny":
        x = synth.activations(rng, nvec, n) * np.float32(1e-6)
    elif case == "large":
        x = synth.activations(rng, nvec, n) * np.float32(3e4)
    elif case == "zeros":
        x = synth.activations(rng, nvec, n)
        x[:, 64:128] = 0.0
        if nvec > 1:
            x[1, :] = 0.0
    else:  # values whose scaled magnitude is exactly k + 0.5 when amax = 127
        x = np.zeros((nvec, n), dtype=np.float32)
        x[:, ::32] = 127.0
        x[:, 1::32] = (rng.integers(-126, 126, size=(nvec, n // 32)) + 0.5).astype(np.float32)
    return x


@pytest.mark.parametrize("case", QUANT_CASES)
def test_quantize_parity(case):
    rng = synth.rng_for(102, len(case))
    nvec, n = 3, 4096
    x = quant_case_activations(rng, case, nvec, n)
    q, d = binding.quantize(dev(x))
    want_q, want_d = oracle.q8_quantize(x)
    assert np.array_equal(q.cpu().numpy(), want_q)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), want_d)


@pytest.mark.parametrize("nvec,n", [(5, 1184), (1, 96), (2, 32 * 33), (5, 32 * 3333)])
def test_quantize_ragged_block_counts_guard_untouched(nvec, n):
    """Block counts that are not a multiple of a warp's four blocks or a CTA's
    32 (185, 3, 66 and 16665): every block quantized, nothing written past the
    end."""
    rng = synth.rng_for(103, nvec, n)
    x = synth.activations(rng, nvec, n, outliers=0.01)
    q_big = torch.full((nvec * n + 512,), 77, dtype=torch.int8, device="cuda")
    d_big = torch.full((nvec * (n // 32) + 256,), 0x7E00, dtype=torch.int16, device="cuda")
    binding.quantize(dev(x), q_big[:nvec * n], d_big[:nvec * (n // 32)])
    want_q, want_d = oracle.q8_quantize(x)
    got_q, got_d = q_big.cpu().numpy(), d_big.cpu().numpy().view(np.uint16)
    assert np.array_equal(got_q[:nvec * n].reshape(nvec, n), want_q)
    assert np.array_equal(got_d[:nvec * (n // 32)].reshape(nvec, n // 32), want_d)
    assert np.all(got_q[nvec * n:] == 77) and np.all(got_d[nvec * (n // 32):] == 0x7E00)


@pytest.mark.parametrize("nvec,n", [(2, 14336), (40, 16384)])
def test_quantize_from_pinned_host_activations(nvec, n):
    """x in pinned host memory, read by the kernel over the host link; q and d
    on the device and, in a second call, in pinned host memory too (one
    activation, and 40 side by side)."""
    rng = synth.rng_for(104, nvec)
    x = synth.activations(rng, nvec, n, outliers=0.01)
    hx = torch.from_numpy(x).pin_memory()
    want_q, want_d = oracle.q8_quantize(x)
    q, d = binding.quantize(hx)
    torch.cuda.synchronize()
    assert q.is_cuda and np.array_equal(q.cpu().numpy(), want_q)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), want_d)
    hq = torch.empty((nvec, n), dtype=torch.int8).pin_memory()
    hd = torch.empty((nvec, n // 32), dtype=torch.int16).pin_memory()
    binding.quantize(hx, hq, hd)
    torch.cuda.synchronize()
    assert np.array_equal(hq.numpy(), want_q) and np.array_equal(hd.numpy().view(np.uint16), want_d)


def test_quantize_hand_derived_fixture():
    import json
    import os
    spec = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "q8_hand_derived.json")))
    for c in spec["cases"]:
        xb = np.full(32, int(c["x_fill_hex"], 16), dtype=np.uint32)
        for k, v in c["x_hex"].items():
            xb[int(k)] = int(v, 16)
        q, d = binding.quantize(dev(xb.view(np.float32)[None, :]))
        want = np.full(32, c["expected_q_fill"], dtype=np.int64)
        for k, v in c["expected_q"].items():
            want[int(k)] = v
        assert np.array_equal(q.cpu().numpy()[0].astype(np.int64), want)
        assert int(d.cpu().numpy().view(np.uint16)[0, 0]) == int(c["expected_d_hex"], 16)


# ------------------------------------------------------ golden fixtures ----
@pytest.mark.parametrize("case", load_cases(), ids=lambda c: c[0])
def test_gemv_hand_derived(case):
    name, blocks, q, d1, expected = case
    got = gpu_gemv(blocks, q, d1)
    assert got.view(np.uint32)[0] == np.float32(expected).view(np.uint32), (name, got, expected)
    got_b = gpu_gemm(blocks, np.stack([q, q, q]), np.stack([d1, d1, d1]))
    assert np.all(got_b.view(np.uint32) == np.float32(expected).view(np.uint32))


# ------------------------------------------------------------ gemv: small --
SHAPES = [(1, 128), (7, 256), (31, 384), (32, 1024), (33, 1152), (100, 2048), (255, 4096),
          (300, 1024), (1000, 512), (64, 14336), (5, 16384), (3, 17408)]


@pytest.mark.parametrize("rows,n", SHAPES)
@pytest.mark.parametrize("regime", ["quantized", "raw_m128", "halfnormal_subnormal"])
def test_gemv_parity(rows, n, regime):
    rng = synth.rng_for(103, rows, n, len(regime))
    if regime == "quantized":
        blocks = synth.weight_blocks(rng, rows, n, "halfnormal")
        q, d = oracle.q8_quantize(synth.activations(rng, 1, n, outliers=0.01))
    elif regime == "raw_m128":
        blocks = synth.weight_blocks(rng, rows, n, "lognormal")
        q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.05)
    else:
        blocks = synth.weight_blocks(rng, rows, n, "halfnormal")
        q, d = synth.raw_quants(rng, 1, n, scale="halfnormal", m128_frac=0.01)
        d[0, ::7] = rng.integers(1, 0x400, size=d[0, ::7].shape)  # binary16 subnormal scales
    got = gpu_gemv(blocks, q[0], d[0])
    bits_equal(got, oracle.gemv(blocks, q[0], d[0]))


@pytest.mark.parametrize("rows,n", [(40000, 256), (20000, 512), (9999, 1152)])
def test_gemv_parity_many_rows(rows, n):
    """Row counts that select 4, 2 and 1 rows per thread in the launcher."""
    rng = synth.rng_for(104, rows, n)
    blocks = synth.weight_blocks(rng, rows, n, "lognormal")
    q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.02)
    bits_equal(gpu_gemv(blocks, q[0], d[0]), oracle.gemv(blocks, q[0], d[0]))


def test_config_single_256x1024():
    """W 256x1024, Bernoulli(0.5) signs, |N(0,0.02)| block scales, N(0,1) input."""
    rng = synth.rng_for(1, 0, 0)
    blocks = synth.weight_blocks(rng, 256, 1024, "halfnormal")
    x = synth.activations(synth.rng_for(1, 0, 1), 1, 1024)
    q, d = binding.quantize(dev(x))
    want_q, want_d = oracle.q8_quantize(x)
    assert np.array_equal(q.cpu().numpy(), want_q) and np.array_equal(d.cpu().numpy().view(np.uint16), want_d)
    packed = binding.pack(dev(blocks), 256, 1024)
    out = binding.gemv(packed, 256, 1024, q[0], d[0]).cpu().numpy()
    bits_equal(out, oracle.gemv(blocks, want_q[0], want_d[0]))


def test_config_4096x4096_outliers_full():
    """W 4096x4096, input N(0,1) with 1 % outliers at 20: every row compared."""
    rng = synth.rng_for(2, 0, 0)
    blocks = synth.weight_blocks(rng, 4096, 4096, "halfnormal")
    x = synth.activations(synth.rng_for(2, 0, 1), 1, 4096, outliers=0.01)
    q, d = binding.quantize(dev(x))
    packed = binding.pack(dev(blocks), 4096, 4096)
    out = binding.gemv(packed, 4096, 4096, q[0], d[0]).cpu().numpy()
    want_q, want_d = oracle.q8_quantize(x)
    bits_equal(out, oracle.gemv(blocks, want_q[0], want_d[0]))


# ------------------------------------------------------- batched products --
@pytest.mark.parametrize("nvec", [1, 2, 3, 4, 5, 8, 9, 16, 33, 64])
def test_gemm_small_parity(nvec):
    rows, n = 300, 1152
    rng = synth.rng_for(105, nvec)
    blocks = synth.weight_blocks(rng, rows, n, "lognormal")
    q, d = synth.raw_quants(rng, nvec, n, scale="lognormal", m128_frac=0.03)
    got = gpu_gemm(blocks, q, d)
    bits_equal(got, oracle.gemm(blocks, q, d))


def test_gemm_small_columns_equal_gemv():
    rows, n, nvec = 777, 4096, 16
    rng = synth.rng_for(106)
    blocks = synth.weight_blocks(rng, rows, n, "halfnormal")
    x = synth.activations(rng, nvec, n)
    q, d = binding.quantize(dev(x))
    packed = binding.pack(dev(blocks), rows, n)
    outb = binding.gemm_small(packed, rows, n, q, d).cpu().numpy()
    for v in range(nvec):
        outv = binding.gemv(packed, rows, n, q[v], d[v]).cpu().numpy()
        assert np.array_equal(outb[v].view(np.uint32), outv.view(np.uint32))


@pytest.mark.parametrize("rows,n,nvec,scale", [
    (14336, 4096, 16, "halfnormal"),
    (4096, 14336, 16, "halfnormal"),
    (128256, 4096, 64, "lognormal"),
    (4096, 14336, 64, "lognormal"),
])
def test_batched_full_size(rows, n, nvec, scale):
    """Multi-sequence (16 vectors) and prefill-chunk (64 vectors, log-normal
    block scales) products at full size: every output against the threaded
    oracle (gpu.md, "How it is verified": every row of every shape)."""
    rng = synth.rng_for(4 if nvec == 16 else 5, rows, n)
    blocks = synth.weight_blocks(rng, rows, n, scale)
    x = synth.activations(rng, nvec, n)
    q, d = binding.quantize(dev(x))
    packed = binding.pack(dev(blocks), rows, n)
    out = binding.gemm_small(packed, rows, n, q, d).cpu().numpy()
    qh, dh = q.cpu().numpy(), d.cpu().numpy().view(np.uint16)
    want_q, want_d = oracle.q8_quantize(x)
    assert np.array_equal(qh, want_q) and np.array_equal(dh, want_d)
    bits_equal(out, oracle.gemm_threaded(blocks, want_q, want_d))


# ----------------------------------------------------- multi-product call --
def test_gemv_multi_mixed_products():
    """One q1_0_gemv_multi launch over products of different shapes, some with
    f32 activations (quantized in the kernel) and some already quantized."""
    shapes = [(1, 128), (33, 384), (300, 1024), (4096, 4096), (1024, 4096), (64, 14336), (7, 17408), (2000, 1152)]
    items, want = [], []
    for i, (rows, n) in enumerate(shapes):
        rng = synth.rng_for(110, i)
        blocks = synth.weight_blocks(rng, rows, n, "lognormal" if i % 2 else "halfnormal")
        packed = binding.pack(dev(blocks), rows, n)
        out = torch.full((rows,), float("nan"), device="cuda")
        if i % 3 == 2:
            q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.03)
            items.append((packed, rows, n, None, dev(q[0]), dev(d[0].view(np.int16)), out))
        else:
            x = synth.activations(rng, 1, n, outliers=0.01)
            q, d = oracle.q8_quantize(x)
            items.append((packed, rows, n, dev(x[0]), None, None, out))
        want.append(oracle.gemv(blocks, q[0], d[0]))
    binding.gemv_multi(items)
    torch.cuda.synchronize()
    for (packed, rows, n, x, q, d, out), w in zip(items, want):
        bits_equal(out.cpu().numpy(), w)


@pytest.mark.parametrize("size", ["small", "large"])
def test_gemv_multi_many_products_balanced(size):
    """More than 8 products of unequal tile costs, so the launcher places the
    CTA range boundaries itself: every output of every product is compared.
    'large' has enough rows for eight rows per thread."""
    rng0 = np.random.default_rng(131 if size == "small" else 132)
    if size == "small":
        shapes = [(int(rng0.integers(1, 3000)), 128 * int(rng0.choice([1, 3, 8, 32, 112]))) for _ in range(20)]
    else:
        shapes = [(int(rng0.choice([4096, 6144, 8192, 16384])), 128 * int(rng0.choice([1, 2, 4, 9, 16])))
                  for _ in range(14)]
    plan = binding.multi_plan(shapes)
    if size == "large":
        assert plan["rows_per_thread"] == 8
    assert plan["max_range_cost"] < plan["total_cost"]
    items, want = [], []
    for i, (rows, n) in enumerate(shapes):
        rng = synth.rng_for(130, i)
        blocks = synth.weight_blocks(rng, rows, n, "lognormal" if i % 2 else "halfnormal")
        x = synth.activations(rng, 1, n, outliers=0.01)
        q, d = oracle.q8_quantize(x)
        out = torch.full((rows,), float("nan"), device="cuda")
        items.append((binding.pack(dev(blocks), rows, n), rows, n, dev(x[0]), None, None, out))
        want.append(oracle.gemv(blocks, q[0], d[0]))
    binding.gemv_multi(items)
    torch.cuda.synchronize()
    for item, w in zip(items, want):
        bits_equal(item[-1].cpu().numpy(), w)


@pytest.mark.parametrize("act", ["f32", "q8"])
@pytest.mark.parametrize("shapes", [
    [(2600, 20480)],
    [(300, 1024), (2600, 20480), (64, 24576), (1000, 4096), (5000, 16512), (7, 17408), (256, 384),
     (4096, 4096), (1, 128), (999, 20608)],
    [(128256, 16512)],
])
def test_streaming_kernel_long_rows_table_chunks(shapes, act):
    """Rows longer than the streaming kernel's one-chunk activation table
    (more than 128 blocks): the table is rebuilt chunk by chunk inside every
    tile, from f32 input (quantized on the way) or from q8_0 input, for one
    product and for a list of more than eight; every output against the
    oracle.  The lm_head-sized row count takes eight rows per thread."""
    plan = binding.multi_plan(shapes)
    assert plan["panel_warps"] == 0
    if shapes[0][0] == 128256:
        assert plan["rows_per_thread"] == 8
    items, want = [], []
    for i, (rows, n) in enumerate(shapes):
        rng = synth.rng_for(140, i, len(shapes), len(act))
        blocks = synth.weight_blocks(rng, rows, n, "lognormal" if i % 2 else "halfnormal")
        out = torch.full((rows,), float("nan"), device="cuda")
        packed = binding.pack(dev(blocks), rows, n)
        if act == "f32":
            x = synth.activations(rng, 1, n, outliers=0.01)
            q, d = oracle.q8_quantize(x)
            items.append((packed, rows, n, dev(x[0]), None, None, out))
        else:
            q, d = synth.raw_quants(rng, 1, n, scale="lognormal", m128_frac=0.03)
            items.append((packed, rows, n, None, dev(q[0]), dev(d[0].view(np.int16)), out))
        want.append(oracle.gemm_threaded(blocks, q, d)[0])
    binding.gemv_multi(items)
    torch.cuda.synchronize()
    for item, w in zip(items, want):
        bits_equal(item[-1].cpu().numpy(), w)


def test_gemv_multi_fused_equals_quantize_then_gemv():
    rows, n = 4096, 14336
    rng = synth.rng_for(111)
    blocks = synth.weight_blocks(rng, rows, n)
    x = dev(synth.activations(rng, 1, n, outliers=0.01)[0])
    packed = binding.pack(dev(blocks), rows, n)
    q, d = binding.quantize(x)
    a = binding.gemv(packed, rows, n, q, d)
    b = torch.empty(rows, device="cuda")
    binding.gemv_multi([(packed, rows, n, x, None, None, b)])
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("fmt,rows", [("q1", 1000), ("q1", 40000), ("q2", 1000), ("q2", 40000)])
@pytest.mark.parametrize("case", QUANT_CASES + ["fixture"])
def test_fused_quantization_every_regime(fmt, rows, case):
    """The product kernels quantize an f32 activation themselves while they
    build their tables (two words of a sub-block per thread, rounding with
    adds instead of conversions).  Every regime of the quantizer test, and the
    hand-derived q8 block, gives the oracle's quantize-then-product bits, in
    the panel kernel (1000 rows) and in the streaming kernel (40000 rows)."""
    import json
    import os
    n = 4096
    rng = synth.rng_for(112, rows, len(case), len(fmt))
    if case == "fixture":
        spec = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "q8_hand_derived.json")))
        blocks32 = []
        for c in spec["cases"]:
            xb = np.full(32, int(c["x_fill_hex"], 16), dtype=np.uint32)
            for k, v in c["x_hex"].items():
                xb[int(k)] = int(v, 16)
            blocks32.append(xb.view(np.float32))
        x = np.resize(np.concatenate(blocks32), n)[None, :].astype(np.float32)
    else:
        x = quant_case_activations(rng, case, 1, n)
    plan = binding.multi_plan([(rows, n)], fmt=fmt)
    assert (plan["panel_warps"] > 0) == (rows == 1000)
    wq, wd = oracle.q8_quantize(x)
    out = torch.empty(rows, device="cuda")
    if fmt == "q1":
        blocks = synth.weight_blocks(rng, rows, n, "lognormal")
        binding.gemv_multi([(binding.pack(dev(blocks), rows, n), rows, n, dev(x[0]), None, None, out)])
        want = oracle.gemm_threaded(blocks, wq, wd)[0]
    else:
        tb = synth.ternary_blocks_fast(rng, rows, n)
        binding.q2_gemv_multi([(binding.q2_pack(dev(tb), rows, n), rows, n, dev(x[0]), None, None, out)])
        want = oracle.q2_gemv_threaded(tb, wq[0], wd[0])
    bits_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("fmt,rows", [("q1", 1000), ("q1", 40000), ("q2", 1000), ("q2", 40000)])
def test_gemv_multi_prefetch_same_bits(fmt, rows):
    """q1_0_gemv_multi_prefetch / q2_0_gemv_multi_prefetch give the bits of the
    plain call, with the prefetched ranges another product's packed weights, a
    ragged byte count (rounded down inside the range), empty ranges, or
    several ranges (weights and the activation itself)."""
    n = 2048
    rng = synth.rng_for(113, rows, len(fmt))
    x = dev(synth.activations(rng, 1, n)[0])
    if fmt == "q1":
        blocks = synth.weight_blocks(rng, rows, n)
        packed, other = binding.pack(dev(blocks), rows, n), binding.pack(dev(blocks[:777]), 777, n)
        run = binding.gemv_multi
    else:
        tb = synth.ternary_blocks_fast(rng, rows, n)
        packed, other = binding.q2_pack(dev(tb), rows, n), binding.q2_pack(dev(tb[:777]), 777, n)
        run = binding.q2_gemv_multi
    base = torch.empty(rows, device="cuda")
    run([(packed, rows, n, x, None, None, base)])
    for pf in (other, (other.data_ptr(), other.numel() - 5), (other.data_ptr(), 0), (0, 0), [other, x],
               [(0, 0)] * 4, []):
        out = torch.full((rows,), float("nan"), device="cuda")
        run([(packed, rows, n, x, None, None, out)], prefetch=pf)
        assert torch.equal(out.view(torch.int32), base.view(torch.int32))


def test_gemv_multi_prefetch_rejects_bad_ranges():
    rows, n = 256, 1024
    packed = binding.pack(dev(synth.weight_blocks(synth.rng_for(114), rows, n)), rows, n)
    x = torch.zeros(n, device="cuda")
    out = torch.empty(rows, device="cuda")
    for pf in ((packed.data_ptr() + 8, 64), (packed.data_ptr(), -16), (0, 64), [packed] * 5,
               [x, (packed.data_ptr() + 4, 16)]):
        with pytest.raises(binding.Q1Error, match="prefetch"):
            binding.gemv_multi([(packed, rows, n, x, None, None, out)], prefetch=pf)


def test_gemv_multi_host_activations_and_outputs():
    """Activations and outputs in pinned host memory, read and written by the
    kernel directly: the same bits as device buffers."""
    shapes = [(4096, 4096), (1024, 4096), (300, 14336)]
    items_dev, items_host = [], []
    for i, (rows, n) in enumerate(shapes):
        rng = synth.rng_for(140, i)
        blocks = synth.weight_blocks(rng, rows, n)
        packed = binding.pack(dev(blocks), rows, n)
        x = synth.activations(rng, 1, n)[0]
        items_dev.append((packed, rows, n, dev(x), None, None, torch.empty(rows, device="cuda")))
        hx = torch.from_numpy(x).pin_memory()
        items_host.append((packed, rows, n, hx, None, None, torch.full((rows,), float("nan")).pin_memory()))
    binding.gemv_multi(items_dev)
    binding.gemv_multi(items_host)
    torch.cuda.synchronize()
    for a, b in zip(items_dev, items_host):
        assert torch.equal(a[-1].cpu().view(torch.int32), b[-1].view(torch.int32))
    with pytest.raises(ValueError):
        binding.product_array([(items_dev[0][0], 4096, 4096, torch.zeros(4096), None, None, items_dev[0][-1])])


def test_gemv_multi_rejects_bad_lists():
    rows, n = 32, 128
    packed = torch.empty(binding.packed_bytes(rows, n), dtype=torch.uint8, device="cuda")
    out = torch.empty(rows, device="cuda")
    with pytest.raises(ValueError):
        binding.product_array([(packed, rows, n, None, None, None, out)])
    arr = (binding.Product * 0)()
    with pytest.raises(binding.Q1Error):
        binding.gemv_multi(array=arr)


# ------------------------------------------------------- decode set (graph) --
@pytest.fixture(scope="module")
def decode_set():
    from decode_q1_gemv_gb300.decode_set import DecodeSet
    return DecodeSet(seed=3)


@pytest.fixture(scope="module")
def decode_set_expected(decode_set):
    """Every output of the decode set from the threaded oracle, with the q8_0
    quants and scales of every activation: per product (out, q, d)."""
    ds = decode_set
    exp = []
    for i in range(len(ds.shapes)):
        want_q, want_d = oracle.q8_quantize(ds.host_x(i)[None, :])
        want = oracle.gemm_threaded(ds.host_blocks(i), want_q, want_d)[0]
        exp.append((want, want_q[0], want_d[0]))
    return exp


@pytest.mark.parametrize("schedule", ["set", "grouped", "decode", "separate"])
def test_decode_set_graph_full(decode_set, decode_set_expected, schedule):
    """The full 225-product Llama-3-8B-shaped decode set, run exactly as the
    benchmark runs it (one CUDA graph per schedule, programmatic dependent
    launch): every output of every product against the oracle, bit for bit
    (gpu.md, "How it is verified": every row of every shape)."""
    ds = decode_set
    g = ds.capture(schedule)
    ds.out_all.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    got_all = ds.out_all.cpu().numpy()
    for i, (name, rows, n) in enumerate(ds.shapes):
        want, want_q, want_d = decode_set_expected[i]
        got = got_all[ds.out_off[i]:ds.out_off[i] + rows]
        assert not np.any(np.isnan(got)), name
        bits_equal(got, want)
        if schedule == "separate":
            assert np.array_equal(ds.q[i].cpu().numpy(), want_q), name
            assert np.array_equal(ds.d[i].cpu().numpy().view(np.uint16), want_d), name


# ---------------------------------------------------- edge and error cases --
def test_outputs_written_once_and_guard_untouched():
    rows, n = 77, 512
    rng = synth.rng_for(107)
    blocks = synth.weight_blocks(rng, rows, n)
    q, d = synth.raw_quants(rng, 1, n)
    packed = binding.pack(dev(blocks), rows, n)
    buf = torch.full((rows + 64,), float("nan"), device="cuda")
    binding.gemv(packed, rows, n, dev(q[0]), dev(d[0].view(np.int16)), out=buf[:rows])
    host = buf.cpu().numpy()
    assert not np.any(np.isnan(host[:rows]))
    assert np.all(np.isnan(host[rows:]))
    bits_equal(host[:rows], oracle.gemv(blocks, q[0], d[0]))


def test_deterministic_and_stream_independent():
    rows, n = 5000, 4096
    rng = synth.rng_for(108)
    blocks = synth.weight_blocks(rng, rows, n, "lognormal")
    q, d = synth.raw_quants(rng, 1, n, scale="lognormal")
    packed = binding.pack(dev(blocks), rows, n)
    qd, dd = dev(q[0]), dev(d[0].view(np.int16))
    a = binding.gemv(packed, rows, n, qd, dd).cpu().numpy()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = binding.gemv(packed, rows, n, qd, dd)
    s.synchronize()
    assert np.array_equal(a.view(np.uint32), b.cpu().numpy().view(np.uint32))


def test_bad_arguments_raise():
    packed = torch.empty(binding.packed_bytes(64, 256), dtype=torch.uint8, device="cuda")
    q = torch.zeros(256, dtype=torch.int8, device="cuda")
    d = torch.zeros(8, dtype=torch.int16, device="cuda")
    with pytest.raises(binding.Q1Error):
        binding.load()  # noqa: B018 - the library loads
        rc = binding.load().q1_0_gemv(packed.data_ptr(), 64, 200, q.data_ptr(), d.data_ptr(),
                                      torch.empty(64, device="cuda").data_ptr(), None)
        binding._check(rc, "q1_0_gemv")
    with pytest.raises(TypeError):
        binding.gemv(packed, 64, 256, q.float(), d)
    with pytest.raises(ValueError):
        binding.gemv(packed, 64, 256, q.cpu(), d)


def test_device_status_clean_after_suite():
    """No kernel gave up a bounded wait during the parity runs."""
    assert binding.device_status(clear=True) == 0


def test_bench_json_line_contract():
    """bench.py prints one JSON line with the keys the benchmark contract needs."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, "bench.py", "--layers", "1", "--steps", "3", "--warmup", "3",
                        "--no-cpu-baseline", "--schedules", "grouped"], cwd=root, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "e2e", "gpu_launches", "clocks"):
        assert key in d, key
    assert d["roofline"]["bound"] == "hbm" and d["roofline"]["peak"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["gpu_launches"] == 3 and d["value"] > 0
