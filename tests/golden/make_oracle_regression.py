"""Write oracle_regression.txt: oracle outputs at fixed points of small seeded grids.

Calls only the CPU oracle and the seeded input generator. Rerun only when a change to
the oracle's arithmetic is justified by the stencil definition; the commit that changes
the file says why.
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from seismic_wave_propagation_gb300 import synth  # noqa: E402

CASES = [
    ("apply", 1, "average7", (20, 18, 16)),
    ("apply", 1, "laplacian2", (20, 18, 16)),
    ("apply", 4, "laplacian8", (24, 20, 18)),
    ("wave", 4, "laplacian8", (24, 20, 18)),
]


def case_values(kind, R, cname, dims):
    nx, ny, nz = dims
    c = synth.coeffs_for(cname).astype(np.float32)
    u = synth.uniform_field(nx, ny, nz)
    m = np.zeros((nz, ny, nx), bool)
    m[R:nz - R, R:ny - R, R:nx - R] = True
    idx = np.flatnonzero(m.ravel())[::53]
    if kind == "apply":
        vals = oracle.apply_points(u, c, R, idx)
    else:
        up = synth.uniform_field(nx, ny, nz, seed=synth.DEFAULT_SEED + 1)
        s = synth.layered_v2dt2(nx, ny, nz)
        e = synth.sponge_eta(nx, ny, nz, width=6)
        vals = oracle.wave_points(up, u, s, e, c, R, idx)
    return idx, vals


def main():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.txt")
    with open(path, "w") as f:
        f.write("# kind radius coeffs nx ny nz flat_index value_fp32_hex  (written by make_oracle_regression.py)\n")
        for kind, R, cname, dims in CASES:
            idx, vals = case_values(kind, R, cname, dims)
            for i, v in zip(idx, vals):
                f.write(f"{kind} {R} {cname} {dims[0]} {dims[1]} {dims[2]} {int(i)} "
                        f"{np.float32(v).view(np.uint32):08x}\n")


if __name__ == "__main__":
    main()
