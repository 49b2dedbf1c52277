"""Traffic and operation counts for star stencils (used for rooflines and reports).

Compulsory (algorithmic) bytes of one sweep: every input point is read once and every
interior output point is written once, fp32. For the fused wave step the input ``u`` is
read once over the whole grid and ``u_prev``, ``v2dt2``, ``eta`` are read and ``u_next``
written only at interior points.

The tiled-reuse model follows "Thread Coarsening 與 Register Tiling" (the quantitative
ratios table and the exam table): a 7-point update costs 13 flops (7 multiplies and 6
adds with a distinct weight per term), a T^3 input tile yields (T-2)^3 outputs, and a
z-coarsened T x T block sweeping C planes loads T*T*(C+2) inputs for (T-2)^2*C
outputs. These helpers generalise the same counting to radius R.
"""
from __future__ import annotations

F32 = 4


def interior_points(nx: int, ny: int, nz: int, radius: int) -> int:
    """Points at least ``radius`` away from every face."""
    d = [n - 2 * radius for n in (nx, ny, nz)]
    return 0 if min(d) <= 0 else d[0] * d[1] * d[2]


def apply_bytes(nx: int, ny: int, nz: int, radius: int) -> int:
    """Compulsory DRAM bytes of one stencil sweep: read all of ``in``, write the interior."""
    return F32 * nx * ny * nz + F32 * interior_points(nx, ny, nz, radius)


def wave_bytes(nx: int, ny: int, nz: int, radius: int) -> int:
    """Compulsory DRAM bytes of one fused wave step (u whole grid; 3 reads + 1 write per interior point)."""
    return F32 * nx * ny * nz + 4 * F32 * interior_points(nx, ny, nz, radius)


def flops_per_point(radius: int, distinct_weights: bool = False) -> int:
    """Floating-point operations per output point.

    ``distinct_weights``: one multiply per term and adds between them (6R+1 terms ->
    12R+1 flops; 13 for the 7-point case). Otherwise the symmetric form: 6R adds plus
    R+1 multiplies (7R+1).
    """
    terms = 6 * radius + 1
    return 2 * terms - 1 if distinct_weights else 6 * radius + radius + 1


def naive_op_per_byte(radius: int = 1) -> float:
    """One thread per point, every term read from global memory: flops / (4 * terms)."""
    return flops_per_point(radius, True) / (F32 * (6 * radius + 1))


def tiled_op_per_byte(tile: int, radius: int = 1) -> float:
    """T^3 input tile per block, (T-2R)^3 outputs, each input read once."""
    out = (tile - 2 * radius) ** 3
    return flops_per_point(radius, True) * out / (F32 * tile ** 3)


def tiled_op_per_byte_limit(radius: int = 1) -> float:
    """Limit of ``tiled_op_per_byte`` as the tile grows."""
    return flops_per_point(radius, True) / F32


def halo_fraction(tile: int, radius: int = 1) -> float:
    """Fraction of a T^3 input tile that is halo (inputs producing no output)."""
    return 1.0 - ((tile - 2 * radius) / tile) ** 3


def coarsened_tile_counts(tile: int, planes: int, radius: int = 1):
    """(inputs, outputs, op/byte) of a T x T block sweeping ``planes`` output planes."""
    inputs = tile * tile * (planes + 2 * radius)
    outputs = (tile - 2 * radius) ** 2 * planes
    return inputs, outputs, flops_per_point(radius, True) * outputs / (F32 * inputs)


def shared_bytes_plane_buffers(tile: int, planes_in_shared: int) -> int:
    """Shared memory of ``planes_in_shared`` T x T fp32 planes."""
    return planes_in_shared * tile * tile * F32
