"""Row sharding of Q1_0 products across GPUs, with an all-gather of the outputs.

bankML "docs/modules/gpu.md" ("Limitations", and "Advantages and efficiency"
on several cards): each card takes a share of every matrix's rows, so every
output element stays one card's exact dot product and nothing is reduced
across devices; the consumer that needs the whole output vector gathers the
shares.  Here each rank packs only its own rows (the packed layout pads rows
to multiples of 256, so the split is in whole 256-row groups where the rows
allow), runs the ordinary one-GPU product on them, and the full vector is
assembled with one all-gather of f32 outputs (4 bytes per row).

Host logic only: the product on each rank is q1_0_gemv / q1_0_gemm_small of
the library on its own packed rows.
"""
from __future__ import annotations

import torch

ROW_ALIGN = 256  # rows of a panel group of the packed layout


def row_ranges(rows: int, world: int, align: int = ROW_ALIGN):
    """Contiguous [r0, r1) per rank covering 0..rows: whole `align`-row groups
    spread as evenly as possible, the ragged tail with the last non-empty
    share.  Ranks past the end get empty ranges."""
    if rows < 1 or world < 1 or align < 1:
        raise ValueError("rows, world and align must be positive")
    groups = (rows + align - 1) // align
    base, extra = divmod(groups, world)
    out, g0 = [], 0
    for r in range(world):
        g1 = g0 + base + (1 if r < extra else 0)
        out.append((min(g0 * align, rows), min(g1 * align, rows)))
        g0 = g1
    return out


def gather_rows(local: torch.Tensor, ranges, group=None) -> torch.Tensor:
    """All-gather of row-sharded outputs.  `local` is this rank's
    [..., r1 - r0] block of a [..., rows] output (the last axis is rows);
    returns the full [..., rows] tensor on every rank, each share copied
    unchanged (bit for bit) into place.  Works with any torch.distributed
    backend (NCCL on GPUs, gloo on CPU)."""
    import torch.distributed as dist

    world = dist.get_world_size(group)
    if len(ranges) != world:
        raise ValueError("one range per rank")
    rank = dist.get_rank(group)
    r0, r1 = ranges[rank]
    if local.shape[-1] != r1 - r0:
        raise ValueError(f"rank {rank}: local output has {local.shape[-1]} rows, its range {r1 - r0}")
    if world == 1:
        return local
    width = max(b - a for a, b in ranges)
    lead = local.shape[:-1]
    padded = torch.zeros(lead + (width,), dtype=local.dtype, device=local.device)
    padded[..., :r1 - r0] = local
    parts = [torch.empty_like(padded) for _ in range(world)]
    dist.all_gather(parts, padded.contiguous(), group=group)
    return torch.cat([p[..., :b - a] for p, (a, b) in zip(parts, ranges)], dim=-1)


class ShardedQ1Linear:
    """A Q1_0 matrix whose rows are split across the ranks of a process group:
    this rank packs and keeps only its own rows on its GPU.

    ``ShardedQ1Linear(blocks, group)`` takes the full [rows, n/128, 18] blocks
    (on the host or any device; only this rank's rows are copied to the GPU);
    ``__call__(q, d)`` runs the product on the local rows and returns the full
    output, gathered from all ranks."""

    def __init__(self, blocks: torch.Tensor, group=None, device=None):
        import torch.distributed as dist

        from . import binding

        if blocks.dim() != 3 or blocks.shape[2] != 18:
            raise ValueError("blocks must be uint8 [rows, n/128, 18]")
        self.group = group
        self.rows = int(blocks.shape[0])
        self.n = int(blocks.shape[1]) * 128
        self.ranges = row_ranges(self.rows, dist.get_world_size(group))
        self.r0, self.r1 = self.ranges[dist.get_rank(group)]
        self.device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
        self.local_rows = self.r1 - self.r0
        self.packed = None
        if self.local_rows:
            mine = blocks[self.r0:self.r1].contiguous().to(self.device)
            self.packed = binding.pack(mine, self.local_rows, self.n)

    def __call__(self, q: torch.Tensor, d: torch.Tensor) -> torch.Tensor:
        from . import binding

        nvec = q.numel() // self.n
        local = torch.empty((nvec, self.local_rows), dtype=torch.float32, device=self.device)
        if self.local_rows:
            if nvec == 1:
                binding.gemv(self.packed, self.local_rows, self.n, q, d, local[0])
            else:
                binding.gemm_small(self.packed, self.local_rows, self.n, q, d, local)
        full = gather_rows(local, self.ranges, self.group)
        return full[0] if nvec == 1 and q.dim() == 1 else full
