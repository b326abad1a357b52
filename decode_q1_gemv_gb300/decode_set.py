"""The Llama-3-8B-shaped 1-bit decode matmul set on one GPU.

One decode step = for each of the 225 products (32 layers x q, k, v, o, gate,
up, down, then lm_head): q8_0-quantize the product's f32 activation and run
the Q1_0 matrix-vector product.  All weights are packed once and stay
resident; inputs are seeded synthetic data (``synth``), one activation vector
per product.  Schedules of the same work:

  "set"       one q1_0_gemv_multi launch for all 225 products (the products of
              this workload are independent: each has its own input vector)
  "grouped"   the launches a real decode step's data dependencies allow: per
              layer {q, k, v}, {o}, {gate, up}, {down}, then {lm_head}: 129
              dependent q1_0_gemv_multi launches
  "decode"    one launch per product in decode order: 225 dependent launches
  "separate"  q8_quantize_act then q1_0_gemv per product: 450 launches

Every schedule can be captured once as a CUDA graph and replayed; the kernels
use programmatic dependent launch, so each launch's weight streaming begins
while the previous kernel drains.  In "grouped" and "decode" each launch also
pulls the packed weights and the activations of the launch after it into L2
(q1_0_gemv_multi_prefetch; prefetch_next=False turns that off).  Weights do
not depend on the chain; in a real decode step the activation is the output
of the kernel just before, already in L2, while here every product reads its
own stored vector, so prefetching it gives a launch the inputs a real step's
launch finds in L2.

fmt="q2" builds the same set with Q2_0 (ternary) weights (q2_0_* calls,
34 bytes per 128 weights, synth.ternary_blocks_fast).
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding, synth

ALIGN = 256


def _round_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


class DecodeSet:
    def __init__(self, seed: int = 3, device: str = "cuda", shapes=None, scale: str = "halfnormal",
                 outliers: float = 0.0, fmt: str = "q1", prefetch_next: bool = True):
        if fmt not in ("q1", "q2"):
            raise ValueError(f"unknown weight format {fmt!r}")
        self.fmt = fmt
        self.block_bytes = synth.BLOCK_BYTES if fmt == "q1" else synth.Q2_BLOCK_BYTES
        self._packed_bytes = binding.packed_bytes if fmt == "q1" else binding.q2_packed_bytes
        self._pack = binding.pack if fmt == "q1" else binding.q2_pack
        self._gemv = binding.gemv if fmt == "q1" else binding.q2_gemv
        self._gemv_multi = binding.gemv_multi if fmt == "q1" else binding.q2_gemv_multi
        self.seed = seed
        self.prefetch_next = prefetch_next
        self.device = torch.device(device)
        self.shapes = list(shapes) if shapes is not None else synth.decode_set_shapes()
        self.scale = scale
        self.outliers = outliers
        # One resident buffer for all packed weights.
        self.offsets = []
        total = 0
        for _, rows, n in self.shapes:
            self.offsets.append(total)
            total += _round_up(self._packed_bytes(rows, n), ALIGN)
        self.packed = torch.empty(total, dtype=torch.uint8, device=self.device)
        self.weight_bytes = sum(rows * n * self.block_bytes // 128 for _, rows, n in self.shapes)
        for i, (_, rows, n) in enumerate(self.shapes):
            blocks = torch.from_numpy(self.host_blocks(i)).to(self.device)
            nbytes = self._packed_bytes(rows, n)
            view = self.packed[self.offsets[i]:self.offsets[i] + nbytes]
            self._pack(blocks, rows, n, view)
            del blocks
        # Activations (f32 inputs), their q8_0 form, and outputs: one contiguous
        # buffer each (so a host round trip is one copy in and one copy out),
        # with a view per product; input offsets are multiples of 256 elements
        # (so every scale view starts 16-byte aligned), output offsets of 64.
        self.x_off, self.out_off = [], []
        nx = nout = 0
        for _, rows, n in self.shapes:
            self.x_off.append(nx)
            self.out_off.append(nout)
            nx += _round_up(n, 256)
            nout += _round_up(rows, 64)
        self.x_all = torch.zeros(nx, dtype=torch.float32, device=self.device)  # padding stays 0
        self.q_all = torch.empty(nx, dtype=torch.int8, device=self.device)
        self.d_all = torch.empty(nx // 32, dtype=torch.int16, device=self.device)
        self.out_all = torch.empty(nout, dtype=torch.float32, device=self.device)
        self.x, self.q, self.d, self.out = [], [], [], []
        for i, (_, rows, n) in enumerate(self.shapes):
            o, oo = self.x_off[i], self.out_off[i]
            self.x.append(self.x_all[o:o + n])
            self.q.append(self.q_all[o:o + n])
            self.d.append(self.d_all[o // 32:(o + n) // 32])
            self.out.append(self.out_all[oo:oo + rows])
            self.x[i].copy_(torch.from_numpy(self.host_x(i)))
        torch.cuda.synchronize(self.device)
        self.graph = None

    # -------------------------------------------------------- host inputs --
    def host_blocks(self, i: int) -> np.ndarray:
        _, rows, n = self.shapes[i]
        if self.fmt == "q2":
            return synth.ternary_blocks_fast(synth.rng_for(self.seed, i, 0, 2), rows, n, self.scale)
        return synth.weight_blocks(synth.rng_for(self.seed, i, 0), rows, n, self.scale)

    def host_x(self, i: int) -> np.ndarray:
        _, rows, n = self.shapes[i]
        return synth.activations(synth.rng_for(self.seed, i, 1), 1, n, outliers=self.outliers)[0]

    # ------------------------------------------------------------ compute --
    def packed_view(self, i: int) -> torch.Tensor:
        _, rows, n = self.shapes[i]
        return self.packed[self.offsets[i]:self.offsets[i] + self._packed_bytes(rows, n)]

    SCHEDULES = ("set", "grouped", "decode", "separate")

    def _item(self, i, fused=True):
        _, rows, n = self.shapes[i]
        if fused:
            return (self.packed_view(i), rows, n, self.x[i], None, None, self.out[i])
        return (self.packed_view(i), rows, n, None, self.q[i], self.d[i], self.out[i])

    def groups(self, schedule: str):
        """Lists of product indices, one list per launch, in launch order."""
        idx = list(range(len(self.shapes)))
        if schedule == "set":
            return [idx]
        if schedule == "decode":
            return [[i] for i in idx]
        if schedule == "grouped":
            out, i = [], 0
            names = [name.split(".")[-1] for name, _, _ in self.shapes]
            while i < len(idx):
                nm = names[i]
                if nm == "q" and names[i + 1:i + 3] == ["k", "v"]:
                    out.append([i, i + 1, i + 2])
                    i += 3
                elif nm == "gate" and i + 1 < len(idx) and names[i + 1] == "up":
                    out.append([i, i + 1])
                    i += 2
                else:
                    out.append([i])
                    i += 1
            return out
        raise ValueError(schedule)

    def _arrays(self, schedule):
        key = "_arr_" + schedule
        if not hasattr(self, key):
            setattr(self, key, [binding.product_array([self._item(i) for i in g], fmt=self.fmt)
                                for g in self.groups(schedule)])
        return getattr(self, key)

    def weights_view(self, first: int, last: int) -> torch.Tensor:
        """The packed weights of products first..last (contiguous in the
        resident buffer, in product order)."""
        _, rows, n = self.shapes[last]
        return self.packed[self.offsets[first]:self.offsets[last] + self._packed_bytes(rows, n)]

    def activations_view(self, first: int, last: int) -> torch.Tensor:
        """The f32 activations of products first..last (contiguous)."""
        _, rows, n = self.shapes[last]
        return self.x_all[self.x_off[first]:self.x_off[last] + n]

    def _prefetches(self, schedule):
        """Per launch of the schedule: the next launch's packed weights and
        activations as a prebuilt range array, or None."""
        gs = self.groups(schedule)
        if not self.prefetch_next or schedule == "set":
            return [None] * len(gs)
        key = "_pf_" + schedule
        if not hasattr(self, key):
            setattr(self, key, [binding.prefetch_ranges([self.weights_view(gs[k + 1][0], gs[k + 1][-1]),
                                                         self.activations_view(gs[k + 1][0], gs[k + 1][-1])])
                                if k + 1 < len(gs) else None for k in range(len(gs))])
        return getattr(self, key)

    def launches(self, schedule: str) -> int:
        return 2 * len(self.shapes) if schedule == "separate" else len(self.groups(schedule))

    def step(self, stream=None, schedule: str = "set"):
        """Enqueue one decode step with the given schedule."""
        if schedule == "separate":
            for i, (_, rows, n) in enumerate(self.shapes):
                binding.quantize(self.x[i], self.q[i], self.d[i], stream=stream)
                self._gemv(self.packed_view(i), rows, n, self.q[i], self.d[i], self.out[i], stream=stream)
            return
        for arr, pf in zip(self._arrays(schedule), self._prefetches(schedule)):
            self._gemv_multi(array=arr, stream=stream, prefetch=pf)

    def products(self, stream=None):
        """Enqueue the products alone (activations already quantized)."""
        for i, (_, rows, n) in enumerate(self.shapes):
            self._gemv(self.packed_view(i), rows, n, self.q[i], self.d[i], self.out[i], stream=stream)

    def _capture(self, fn):
        s = torch.cuda.Stream(self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize(self.device)
        return g

    def capture(self, schedule: str = "set"):
        """Capture one step as a CUDA graph (after a warm-up on a side stream)."""
        self.graph = self._capture(lambda: self.step(schedule=schedule))
        return self.graph

    def capture_products(self):
        """Capture the 225 products alone as a CUDA graph."""
        return self._capture(self.products)

    def replay(self):
        if self.graph is None:
            self.capture()
        self.graph.replay()


    @property
    def activation_bytes(self) -> int:
        return sum(n * 4 for _, _, n in self.shapes)

    @property
    def output_bytes(self) -> int:
        return sum(rows * 4 for _, rows, _ in self.shapes)
