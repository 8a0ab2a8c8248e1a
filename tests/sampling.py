"""Voxel samples for full-size parity tests, stratified by the launch plan.

A full-size call is checked against the oracle on a voxel subset (voxels are
independent, so any subset is a valid check).  A uniform subset of a few
hundred voxels misses most CTAs of a launch with a thousand or more output
blocks, so a fault confined to one block could pass.  These helpers instead
take voxels from EVERY output block a launch assigns to a CTA, at seeded
positions inside each block, plus the edges (first and last voxel, the last
row, the last column, the corners of the grid).
"""

import numpy as np


def _edges_general(N):
    return [0, N - 1]


def gather_blocks(N, voxels_per_cta, seed, per=1):
    """General gather: CTA b owns voxels [b*voxels_per_cta, (b+1)*voxels_per_cta).
    `per` distinct voxels from each block (fewer if the block is smaller)."""
    rng = np.random.default_rng(seed)
    nblocks = -(-N // voxels_per_cta)
    out = []
    for b in range(nblocks):
        lo = b * voxels_per_cta
        hi = min(N, lo + voxels_per_cta)
        k = min(per, hi - lo)
        out.extend(lo + rng.choice(hi - lo, size=k, replace=False))
    out.extend(_edges_general(N))
    out.append((nblocks - 1) * voxels_per_cta)            # first voxel of the last block
    return np.unique(np.asarray(out, np.int64))


def grid_blocks(nx, ny, nz, rows_per_cta, seed, per=1, cols=128):
    """Grid path: voxel n = row*nx + ix with row = iz*ny + iy; a CTA owns
    rows_per_cta consecutive rows and one block of `cols` columns.  `per`
    voxels from each (row block, column block), spread over `per` equal
    strata of the block's rows, each at a seeded row and column."""
    rng = np.random.default_rng(seed)
    rows = ny * nz
    nrb = -(-rows // rows_per_cta)
    ncb = -(-nx // cols)
    out = []
    for rb in range(nrb):
        r0 = rb * rows_per_cta
        r1 = min(rows, r0 + rows_per_cta)
        for cb in range(ncb):
            c0 = cb * cols
            c1 = min(nx, c0 + cols)
            k = min(per, r1 - r0)
            bounds = np.linspace(r0, r1, k + 1).astype(np.int64)
            for j in range(k):
                lo, hi = int(bounds[j]), int(max(bounds[j + 1], bounds[j] + 1))
                row = int(rng.integers(lo, hi))
                col = int(rng.integers(c0, c1))
                out.append(row * nx + col)
    last_row = rows - 1
    out.extend([0, nx - 1, (rows - 1) * nx, rows * nx - 1])  # corners of the row x column plane
    out.extend(last_row * nx + rng.integers(0, nx, size=4))  # the last row
    out.extend(rng.integers(0, rows, size=4) * nx + nx - 1)  # the last column
    return np.unique(np.asarray(out, np.int64))
