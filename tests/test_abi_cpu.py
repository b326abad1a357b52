"""Host-side checks of the C-ABI library: it builds, loads, exports every
symbol include/q1gemv.h declares, and rejects bad arguments before touching a
device.  No call here launches a kernel (no GPU needed)."""
import ctypes
import os
import re

import pytest
import torch

from decode_q1_gemv_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q1gemv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z][a-z0-9_]*)\s*\(", text)) - {"defined"})


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    assert set(binding.EXPORTS) == set(names), names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_library_exports_are_c_symbols():
    """nm -D shows the entry points unmangled (extern "C")."""
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in syms, name


@pytest.mark.parametrize("rows,n,expect", [
    (1, 128, 256 * 4 * 18),           # rows pad to a 256-row panel group, blocks to 4
    (32, 1024, 256 * 8 * 18),
    (257, 1024, 512 * 8 * 18),
    (4096, 4096, 4096 * 32 * 18),     # exactly 18 bytes per 128 weights
    (4096, 14336, 4096 * 112 * 18),
    (128256, 4096, 128256 * 32 * 18),
    (100, 640, 256 * 8 * 18),         # 5 blocks pad to 8
])
def test_packed_bytes(lib, rows, n, expect):
    assert binding.packed_bytes(rows, n) == expect


@pytest.mark.parametrize("rows,n", [(0, 128), (-1, 128), (1, 0), (1, 64), (1, 200), (1, 1 << 25), (1 << 27, 128)])
def test_packed_bytes_rejects_bad_shapes(lib, rows, n):
    with pytest.raises(binding.Q1Error):
        binding.packed_bytes(rows, n)
    assert "bad shape" in binding.last_error()


def test_null_pointers_rejected_on_host(lib):
    """Argument checks run on the host and return Q1_ERR_ARG with a message."""
    assert lib.q1_0_pack(None, 4, 128, None, None) == binding.Q1_ERR_ARG
    assert "q1_0_pack" in binding.last_error()
    assert lib.q1_0_gemv(None, 4, 128, None, None, None, None) == binding.Q1_ERR_ARG
    assert "q1_0_gemv" in binding.last_error()
    assert lib.q1_0_gemm_small(None, 4, 128, 3, None, None, None, None) == binding.Q1_ERR_ARG
    assert lib.q8_quantize_act(None, 1, 128, None, None, None) == binding.Q1_ERR_ARG
    assert lib.q1_0_unpack(None, 4, 128, None, None) == binding.Q1_ERR_ARG


def test_shape_limits_rejected_on_host(lib):
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the shape check fails first
    assert lib.q1_0_gemv(fake, 4, 100, fake, fake, fake, None) == binding.Q1_ERR_ARG
    assert lib.q1_0_gemm_small(fake, 4, 128, 0, fake, fake, fake, None) == binding.Q1_ERR_ARG
    assert lib.q1_0_gemm_small(fake, 4, 128, 65, fake, fake, fake, None) == binding.Q1_ERR_ARG
    assert "nvec" in binding.last_error()
    assert lib.q8_quantize_act(fake, 1, 48, fake, fake, None) == binding.Q1_ERR_ARG


def test_kernel_choice_knob_rejects_bad_values_and_round_trips(lib):
    """The batched product's kernel choice is a host setting: a bad value is
    refused with a message, a good one returns the previous choice."""
    assert lib.q1_gemm_small_kernel(3) == binding.Q1_ERR_ARG
    assert "choice" in binding.last_error()
    assert lib.q1_gemm_small_kernel(-1) == binding.Q1_ERR_ARG
    assert binding.gemm_small_kernel("tensor") == "auto"
    assert binding.gemm_small_kernel("dp4a") == "tensor"
    assert binding.gemm_small_kernel("auto") == "dp4a"
    with pytest.raises(ValueError):
        binding.gemm_small_kernel("cuda")


def test_misaligned_pointers_rejected_on_host(lib):
    ok = ctypes.c_void_p(0x10000)
    bad = ctypes.c_void_p(0x10004)
    assert lib.q1_0_gemv(bad, 4, 128, ok, ok, ok, None) == binding.Q1_ERR_ARG
    assert "aligned" in binding.last_error()
    assert lib.q1_0_gemv(ok, 4, 128, ok, ok, bad, None) == binding.Q1_ERR_ARG
    assert lib.q1_0_pack(ctypes.c_void_p(0x10001), 4, 128, ok, None) == binding.Q1_ERR_ARG


@pytest.mark.parametrize("fn", ["q1_0_gemv_multi_prefetch", "q2_0_gemv_multi_prefetch"])
def test_prefetch_ranges_rejected_on_host(lib, fn):
    """Bad prefetch ranges are refused before anything is launched."""
    ok = 0x10000
    prods = (binding.Product * 1)(binding.Product(ok, 4, 128, ok, None, None, ok))
    call = getattr(lib, fn)

    def ranges(*rs):
        arr = (binding.Range * max(len(rs), 1))()
        for i, (p, b) in enumerate(rs):
            arr[i] = binding.Range(p, b)
        return arr, len(rs)

    for rs in ([(ok + 8, 64)], [(ok, -16)], [(None, 64)], [(ok, 1 << 41)], [(ok, 16)] * 5):
        arr, nr = ranges(*rs)
        assert call(prods, 1, arr, nr, None) == binding.Q1_ERR_ARG
        assert "prefetch" in binding.last_error()
    assert call(prods, 1, None, 2, None) == binding.Q1_ERR_ARG
    assert call(prods, 1, None, -1, None) == binding.Q1_ERR_ARG


def test_oracle_and_library_share_no_code():
    """The library sources never include or name the oracle, and vice versa."""
    csrc = os.path.join(ROOT, "decode_q1_gemv_gb300", "csrc")
    for fn in os.listdir(csrc):
        text = open(os.path.join(csrc, fn)).read()
        assert "oracle" not in text.lower(), fn
        assert "q1o_" not in text, fn
    pkg = os.path.join(ROOT, "decode_q1_gemv_gb300")
    for fn in os.listdir(pkg):
        if fn.endswith(".py"):
            text = open(os.path.join(pkg, fn)).read()
            assert "import oracle" not in text and "from oracle" not in text, fn
    otext = open(os.path.join(ROOT, "oracle", "q1_oracle.c")).read()
    assert "#include \"" not in otext
    otext_py = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
    assert "import decode_q1_gemv_gb300" not in otext_py and "from decode_q1_gemv_gb300" not in otext_py


# ------------------------------------------------- multi-product work split --
# q1_0_gemv_multi_plan reports the launcher's split without launching; these
# checks hold it to what the header promises, using only the shapes.
def _tiles(shapes, rows_per_thread):
    """(tiles, cost per tile) per product: a tile is rows_per_thread x 32 rows
    (two panel slots below 8 rows per thread), its cost the quad-padded
    blocks per row."""
    panels_per_tile = 8 if rows_per_thread == 8 else 2 * rows_per_thread
    out = []
    for rows, n in shapes:
        panels = -(-rows // 256) * 8
        nbp = -(-(n // 128) // 4) * 4
        out.append((panels // panels_per_tile, nbp))
    return out


def _tile_starts(tiles):
    starts, pos = [], 0
    for t, c in tiles:
        for _ in range(t):
            starts.append(pos)
            pos += c
    return starts, pos


def _check_partition(plan, tiles):
    starts, total = _tile_starts(tiles)
    cuts = plan["cuts"]
    assert plan["total_cost"] == total
    assert len(cuts) == plan["grid"] + 1 and cuts[0] == 0 and cuts[-1] == total
    assert all(a <= b for a, b in zip(cuts, cuts[1:]))
    boundaries = set(starts) | {total}
    # every CTA range starts on a tile boundary (or is empty at the end), so each
    # tile belongs to exactly one CTA and the range cost is the cut difference
    assert all(c in boundaries for c in cuts)
    assert max(b - a for a, b in zip(cuts, cuts[1:])) == plan["max_range_cost"]


def _best_max_range(tiles, ctas):
    """Smallest possible largest range over contiguous splits into at most
    `ctas` ranges at tile boundaries, by exhaustive search over the cut points
    (tiny inputs only)."""
    import itertools
    costs = [c for t, c in tiles for _ in range(t)]
    n = len(costs)
    best = sum(costs)
    for k in range(0, min(ctas - 1, n - 1) + 1):
        for cut in itertools.combinations(range(1, n), k):
            edges = (0,) + cut + (n,)
            best = min(best, max(sum(costs[a:b]) for a, b in zip(edges, edges[1:])))
    return best


def test_multi_plan_decode_set_is_balanced(lib):
    from decode_q1_gemv_gb300 import synth
    shapes = [(rows, n) for _, rows, n in synth.decode_set_shapes()]
    plan = binding.multi_plan(shapes, sms=152)
    assert plan["rows_per_thread"] == 8 and 0 < plan["grid"] <= 304
    tiles = _tiles(shapes, 8)
    _check_partition(plan, tiles)
    # an even split rounded to whole tiles: the largest range it leaves
    starts, total = _tile_starts(tiles)
    even = [0] * 304
    for s0, (t, c) in zip(starts, [(1, c) for t, c in tiles for _ in range(t)]):
        even[min(b for b in range(304) if total * (b + 1) // 304 > s0)] += c
    share = -(-total // 304)
    assert share <= plan["max_range_cost"] <= share + 112
    assert plan["max_range_cost"] < max(even)


def test_multi_plan_small_lists_split_evenly(lib):
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096)]
    plan = binding.multi_plan(shapes, sms=16)  # too many panels for one wave of the panel kernel
    assert plan["panel_warps"] == 0
    tiles = _tiles(shapes, plan["rows_per_thread"])
    starts, total = _tile_starts(tiles)
    g = plan["grid"]
    assert plan["cuts"] == [total * b // g for b in range(g + 1)]


@pytest.mark.parametrize("seed", range(6))
def test_multi_plan_matches_exhaustive_optimum(lib, seed):
    """More than 8 products, few tiles: the split's largest range equals the
    exhaustive optimum over all contiguous splits."""
    import random
    rnd = random.Random(seed)
    shapes = [(rnd.choice([32, 64, 96, 256]), 128 * rnd.choice([1, 4, 8, 28, 40])) for _ in range(rnd.randint(9, 11))]
    plan = binding.multi_plan(shapes, sms=1)
    tiles = _tiles(shapes, plan["rows_per_thread"])
    _check_partition(plan, tiles)
    assert plan["max_range_cost"] == _best_max_range(tiles, min(sum(t for t, _ in tiles), 2))
    plan3 = binding.multi_plan(shapes, sms=2)
    tiles3 = _tiles(shapes, plan3["rows_per_thread"])
    _check_partition(plan3, tiles3)
    ctas = min(sum(t for t, _ in tiles3), 4)  # at most two CTAs per SM
    assert plan3["grid"] <= ctas
    assert plan3["max_range_cost"] == _best_max_range(tiles3, ctas)


def _panel_per_sm(warps, nbp, regs):
    return min(65536 // (regs * 32 * warps), 2048 // (32 * warps), 233472 // (nbp * 1472 + 1024))


def _busiest(nbp, warps, unit):
    """Half quads of work of the busiest warp."""
    return -(-(nbp // unit) // warps) * (unit // 2)


SMEM_MAX = 233472 - 1024  # a CTA's dynamic shared memory at most


def _panel_smem(nbp, ppc):
    return nbp * 320 + ppc * nbp * 1152


def _expected_ppc(panel_counts, nbp, sms=152):
    """The panels-per-CTA rule, for lists that no one-panel shape runs in one
    wave: the smallest P >= ceil(panels / SMs) (at most 8) whose grid of
    ceil(panels_j / P) CTAs is one CTA per SM and whose shared memory fits;
    then 16 warps, and half-quad units when they lower the busiest warp's
    work.  None when no P qualifies."""
    total = sum(panel_counts)
    for P in range(-(-total // sms), 9):
        if _panel_smem(nbp, P) > SMEM_MAX:
            return None
        if sum(-(-c // P) for c in panel_counts) <= sms:
            b4 = -(-(P * nbp // 4) // 16) * 2
            b2 = -(-(P * nbp // 2) // 16)
            return 16, (2 if b2 < b4 else 4), P
    return None


def _one_wave_widths(panels, nbp, regs):
    return [w for w in (4, 8, 16) if panels <= max(1, min(_panel_per_sm(w, nbp, regs), 2048 // (32 * w))) * 152]


def _check_panel_choice(plan, rows, n, regs):
    warps, unit = plan["panel_warps"], plan["panel_unit_blocks"]
    panels = -(-rows // 256) * 8
    nbp = -(-(n // 128) // 4) * 4
    exp = None if _one_wave_widths(panels, nbp, regs) else _expected_ppc([panels], nbp)
    if exp:
        assert (warps, unit, plan["panel_panels"]) == exp
        assert plan["grid"] == -(-panels // exp[2]) <= 152 and plan["rows_per_thread"] == 4
        return
    assert plan["panel_panels"] == 1
    assert plan["grid"] == panels and plan["rows_per_thread"] == 4 and plan["cuts"] == []
    assert panels <= _panel_per_sm(warps, nbp, regs) * 152 and nbp <= 156
    # no other (warps, unit) that fits one wave gives the busiest warp less work
    # with at most 16 warps and no more warps than needed
    for w2 in (4, 8, 16):
        for u2 in (4, 2):
            if panels <= _panel_per_sm(w2, nbp, regs) * 152 and w2 <= max(4, 2 * nbp // 4):
                assert _busiest(nbp, warps, unit) <= _busiest(nbp, w2, u2)


@pytest.mark.parametrize("rows,n,warps,unit,ppc", [
    (4096, 4096, 16, 2, 1), (1024, 4096, 16, 2, 1), (4096, 14336, 16, 4, 1), (14336, 4096, 8, 4, 1),
    (256, 1024, 4, 2, 1), (1, 128, 4, 2, 1), (300, 384, 4, 2, 1), (300, 1536, 8, 2, 1), (8192, 8192, 8, 4, 1),
    (18000, 4096, 4, 4, 1), (20000, 256, 4, 2, 1), (22000, 4096, 16, 2, 5), (30000, 1024, 16, 4, 7),
    (4096, 19968, 16, 2, 1), (5000, 19968, 0, 0, 0), (4096, 20096, 0, 0, 0), (128256, 4096, 0, 0, 0),
    (40000, 256, 0, 0, 0)])
def test_multi_plan_one_product_kernel(lib, rows, n, warps, unit, ppc):
    """A single product of few rows goes to the panel kernel: W = 16, 8 or 4
    warps sharing out the panel's blocks in quads or half quads, the grid of
    one CTA per panel one wave (80 registers a thread, 2048 threads, 228 KB of
    shared memory at 1472 bytes per block plus 1 KB per CTA), n at most 156
    blocks, and the busiest warp as lightly loaded as those limits allow; or,
    when no such grid fits one wave, one CTA of 16 warps per SM taking several
    consecutive panels (at most 8)."""
    plan = binding.multi_plan([(rows, n)], sms=152)
    assert (plan["panel_warps"], plan["panel_unit_blocks"], plan["panel_panels"]) == (warps, unit, ppc)
    if warps:
        _check_panel_choice(plan, rows, n, 80 if warps < 16 else 128)
    else:
        assert plan["grid"] > 0 and len(plan["cuts"]) == plan["grid"] + 1
    # a second product with a row too long for the panel kernel sends the pair to the streaming kernel
    assert binding.multi_plan([(rows, n), (32, 20096)], sms=152)["panel_warps"] == 0


@pytest.mark.parametrize("rows,n,warps,unit,ppc", [
    (4096, 4096, 16, 2, 1), (1024, 4096, 16, 2, 1), (4096, 14336, 16, 4, 1), (14336, 4096, 4, 4, 1),
    (1, 128, 4, 2, 1), (8192, 8192, 8, 4, 1), (18000, 4096, 4, 4, 1), (20000, 4096, 16, 2, 5),
    (40000, 4096, 0, 0, 0), (4096, 20096, 0, 0, 0)])
def test_q2_multi_plan_one_product_kernel(lib, rows, n, warps, unit, ppc):
    """The Q2_0 panel kernel keeps up to 128 registers a thread: 4 CTAs of
    4 warps, 2 of 8 or 1 of 16 an SM by registers; several panels a CTA as for
    Q1_0."""
    plan = binding.multi_plan([(rows, n)], sms=152, fmt="q2")
    assert (plan["panel_warps"], plan["panel_unit_blocks"], plan["panel_panels"]) == (warps, unit, ppc)
    if warps:
        _check_panel_choice(plan, rows, n, 128)
    q1 = binding.multi_plan([(rows, n), (32, 20096)], sms=152)
    q2 = binding.multi_plan([(rows, n), (32, 20096)], sms=152, fmt="q2")
    assert q2 == q1 and q1["panel_warps"] == 0  # the streaming split depends on the shapes only


@pytest.mark.parametrize("shapes,warps,unit,ppc", [
    ([(4096, 4096), (1024, 4096), (1024, 4096)], 8, 4, 1),   # q, k, v of one layer: 192 panels
    ([(2048, 4096), (1000, 14336), (33, 128)], 16, 4, 1),   # unequal rows and n
    ([(300, 1024)] * 8, 4, 2, 1),                            # eight products
    ([(14336, 4096), (14336, 4096)], 16, 4, 6),              # gate and up: 896 panels, 6 a CTA
    ([(20000, 1024), (20000, 1024)], 4, 4, 1),               # 1264 panels: two waves
    ([(14336, 4096)] * 3, 0, 0, 0),                          # more than 8 panels a CTA, two waves
    ([(32, 128)] * 9, 0, 0, 0),                              # more than eight products
    ([(64, 4096), (32, 20096)], 0, 0, 0)])                   # a row longer than 156 blocks
def test_multi_plan_panel_lists(lib, shapes, warps, unit, ppc):
    """Lists of up to 8 products whose panels together fit one wave, or that
    several panels a CTA fit in one wave of one CTA per SM, or two waves when
    neither does, take the panel kernel, sized by the longest row and the
    total panels."""
    plan = binding.multi_plan(shapes, sms=152)
    assert (plan["panel_warps"], plan["panel_unit_blocks"], plan["panel_panels"]) == (warps, unit, ppc)
    if ppc > 1:
        assert plan["grid"] == sum(-(-(-(-r // 256) * 8) // ppc) for r, _ in shapes) <= 152
    elif warps:
        panels = sum(-(-r // 256) * 8 for r, _ in shapes)
        nbp = max(-(-(n // 128) // 4) * 4 for _, n in shapes)
        waves = 1 if panels <= _panel_per_sm(4, nbp, 80) * 152 else 2
        assert plan["grid"] == panels <= waves * _panel_per_sm(warps, nbp, 80 if warps < 16 else 128) * 152


@pytest.mark.parametrize("fmt,regs", [("q1", 80), ("q2", 128)])
@pytest.mark.parametrize("seed", range(4))
def test_multi_plan_panel_rules_random_lists(lib, fmt, regs, seed):
    """Random lists of 1-10 products: the launcher's kernel choice follows its
    stated rules.  The panel kernel only for at most 8 products with rows of at
    most 156 blocks; several panels a CTA when one CTA per panel would put two
    or more on an SM and some P fits; else one wave when any shape fits one
    (the busiest warp then no more loaded than under any other one-wave
    shape); two waves only for lists of two or more that fit no shape in one;
    the streaming kernel otherwise."""
    import random
    rnd = random.Random(1000 + seed)
    for _ in range(60):
        count = rnd.randint(1, 10)
        shapes = [(rnd.choice([1, 33, 256, 1024, 4096, 6000, 14336, 20000]),
                   128 * rnd.choice([1, 3, 8, 16, 32, 112, 156, 157])) for _ in range(count)]
        plan = binding.multi_plan(shapes, sms=152, fmt=fmt)
        panels = sum(-(-r // 256) * 8 for r, _ in shapes)
        nbp = max(-(-(n // 128) // 4) * 4 for _, n in shapes)
        per_sm = lambda w: min(max(1, 65536 // (regs * 32 * w)), 2048 // (32 * w), 233472 // (nbp * 1472 + 1024))
        one_wave = [w for w in (4, 8, 16) if panels <= per_sm(w) * 152]
        two_wave = [w for w in (4, 8, 16) if panels <= 2 * per_sm(w) * 152]
        eligible = count <= 8 and nbp <= 156
        exp = _expected_ppc([-(-r // 256) * 8 for r, _ in shapes], nbp) if eligible and not one_wave else None
        if exp:
            assert (plan["panel_warps"], plan["panel_unit_blocks"], plan["panel_panels"]) == exp, (shapes, plan)
            assert plan["grid"] == sum(-(-(-(-r // 256) * 8) // exp[2]) for r, _ in shapes) <= 152
            continue
        if not eligible or (not one_wave and (count < 2 or not two_wave)):
            assert plan["panel_warps"] == 0, (shapes, plan)
            continue
        assert plan["panel_warps"] in (4, 8, 16) and plan["grid"] == panels, (shapes, plan)
        assert plan["panel_panels"] == 1, (shapes, plan)
        w, u = plan["panel_warps"], plan["panel_unit_blocks"]
        if one_wave:
            assert panels <= per_sm(w) * 152
            best = min(_busiest(nbp, w2, u2) for w2 in one_wave for u2 in (4, 2))
            assert _busiest(nbp, w, u) == best, (shapes, plan)
        else:
            assert count >= 2 and u == 4 and panels <= 2 * per_sm(w) * 152, (shapes, plan)


def test_multi_plan_rejects_bad_arguments(lib):
    with pytest.raises(binding.Q1Error):
        binding.multi_plan([(0, 128)], sms=4)
    with pytest.raises(binding.Q1Error):
        binding.multi_plan([(32, 100)], sms=4)
    with pytest.raises(binding.Q1Error):
        binding.multi_plan([(32, 128)], sms=-1)


# ----------------------------------------------------------- Q2_0 sizes --
@pytest.mark.parametrize("rows,n,expect", [
    (1, 128, 256 * 4 * 34),
    (257, 1024, 512 * 8 * 34),
    (4096, 14336, 4096 * 112 * 34),
    (100, 640, 256 * 8 * 34),
])
def test_q2_packed_bytes(lib, rows, n, expect):
    assert binding.q2_packed_bytes(rows, n) == expect


@pytest.mark.parametrize("rows,n", [(0, 128), (1, 100), (1, 0), (1 << 27, 128)])
def test_q2_packed_bytes_rejects_bad_shapes(lib, rows, n):
    with pytest.raises(binding.Q1Error):
        binding.q2_packed_bytes(rows, n)


def test_q2_null_pointers_rejected_on_host(lib):
    assert lib.q2_0_pack(None, 32, 128, None, None) == binding.Q1_ERR_ARG
    assert lib.q2_0_gemv(None, 32, 128, None, None, None, None) == binding.Q1_ERR_ARG
    assert lib.q2_0_gemv_multi(None, 1, None) == binding.Q1_ERR_ARG


# ------------------------------------- binding: packed sizes checked first --
def _short(nbytes):
    return torch.empty(nbytes - 1, dtype=torch.uint8)


@pytest.mark.parametrize("call", ["gemv", "q2_gemv", "gemm_small", "unpack", "q2_unpack", "multi_q1", "multi_q2"])
def test_binding_rejects_short_packed_buffers_before_launch(lib, call):
    """Every binding call that takes a packed weight buffer checks its size
    against the format's packed size for (rows, n) before anything reaches the
    library: the kernels would read past a short buffer."""

    rows, n = 300, 1024
    q = torch.zeros(n, dtype=torch.int8)
    d = torch.zeros(n // 32, dtype=torch.int16)
    out = torch.zeros(rows)
    p1 = _short(binding.packed_bytes(rows, n))
    p2 = _short(binding.q2_packed_bytes(rows, n))
    with pytest.raises(ValueError, match="needs"):
        if call == "gemv":
            binding.gemv(p1, rows, n, q, d, out)
        elif call == "q2_gemv":
            binding.q2_gemv(p2, rows, n, q, d, out)
        elif call == "gemm_small":
            binding.gemm_small(p1, rows, n, q[None, :], d[None, :], out[None, :])
        elif call == "unpack":
            binding.unpack(p1, rows, n, torch.zeros((rows, n // 128, 18), dtype=torch.uint8))
        elif call == "q2_unpack":
            binding.q2_unpack(p2, rows, n, torch.zeros((rows, n // 128, 34), dtype=torch.uint8))
        elif call == "multi_q1":
            binding.product_array([(p1, rows, n, None, q, d, out)])
        else:
            binding.product_array([(p2, rows, n, None, q, d, out)], fmt="q2")


def test_binding_rejects_q1_buffer_for_q2_products(lib):
    """A Q1_0-packed buffer is about half the Q2_0 size: a Q2_0 product list
    naming it is refused on the host."""

    rows, n = 4096, 4096
    p1 = torch.empty(binding.packed_bytes(rows, n), dtype=torch.uint8)
    q = torch.zeros(n, dtype=torch.int8)
    d = torch.zeros(n // 32, dtype=torch.int16)
    with pytest.raises(ValueError, match="Q2_0"):
        binding.product_array([(p1, rows, n, None, q, d, torch.zeros(rows))], fmt="q2")
    with pytest.raises(ValueError, match="fmt"):
        binding.product_array([(p1, rows, n, None, q, d, torch.zeros(rows))], fmt="q3")
