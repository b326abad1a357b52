"""The Llama-3-8B-shaped 1-bit decode matmul set on one GPU.

One decode step = for each of the 225 products (32 layers x q, k, v, o, gate,
up, down, then lm_head), in that order: quantize the product's f32 activation
(q8_quantize_act), then run the Q1_0 matrix-vector product (q1_0_gemv).  All
weights are packed once and stay resident; inputs are seeded synthetic data
(``synth``).  The step can be captured once as a CUDA graph and replayed; the
kernels use programmatic dependent launch, so inside the graph each product's
weight streaming can begin while the previous kernel drains.
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
                 outliers: float = 0.0):
        self.seed = seed
        self.device = torch.device(device)
        self.shapes = list(shapes) if shapes is not None else synth.decode_set_shapes()
        self.scale = scale
        self.outliers = outliers
        # One resident buffer for all packed weights.
        self.offsets = []
        total = 0
        for _, rows, n in self.shapes:
            self.offsets.append(total)
            total += _round_up(binding.packed_bytes(rows, n), ALIGN)
        self.packed = torch.empty(total, dtype=torch.uint8, device=self.device)
        self.weight_bytes = sum(rows * n * 18 // 128 for _, rows, n in self.shapes)
        for i, (_, rows, n) in enumerate(self.shapes):
            blocks = torch.from_numpy(self.host_blocks(i)).to(self.device)
            nbytes = binding.packed_bytes(rows, n)
            view = self.packed[self.offsets[i]:self.offsets[i] + nbytes]
            binding.pack(blocks, rows, n, view)
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
        self.x_all = torch.empty(nx, dtype=torch.float32, device=self.device)
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
        return synth.weight_blocks(synth.rng_for(self.seed, i, 0), rows, n, self.scale)

    def host_x(self, i: int) -> np.ndarray:
        _, rows, n = self.shapes[i]
        return synth.activations(synth.rng_for(self.seed, i, 1), 1, n, outliers=self.outliers)[0]

    # ------------------------------------------------------------ compute --
    def packed_view(self, i: int) -> torch.Tensor:
        _, rows, n = self.shapes[i]
        return self.packed[self.offsets[i]:self.offsets[i] + binding.packed_bytes(rows, n)]

    def step(self, stream=None):
        """Enqueue one decode step (quantize + product for every matmul)."""
        for i, (_, rows, n) in enumerate(self.shapes):
            binding.quantize(self.x[i], self.q[i], self.d[i], stream=stream)
            binding.gemv(self.packed_view(i), rows, n, self.q[i], self.d[i], self.out[i], stream=stream)

    def products(self, stream=None):
        """Enqueue the products alone (activations already quantized)."""
        for i, (_, rows, n) in enumerate(self.shapes):
            binding.gemv(self.packed_view(i), rows, n, self.q[i], self.d[i], self.out[i], stream=stream)

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

    def capture(self):
        """Capture one step as a CUDA graph (after a warm-up on a side stream)."""
        self.graph = self._capture(self.step)
        return self.graph

    def capture_products(self):
        """Capture the 225 products alone as a CUDA graph."""
        return self._capture(self.products)

    def replay(self):
        if self.graph is None:
            self.capture()
        self.graph.replay()

    @property
    def launches_per_step(self) -> int:
        return 2 * len(self.shapes)

    @property
    def activation_bytes(self) -> int:
        return sum(n * 4 for _, _, n in self.shapes)

    @property
    def output_bytes(self) -> int:
        return sum(rows * 4 for _, rows, _ in self.shapes)
