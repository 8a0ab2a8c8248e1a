"""Seeded synthetic inputs for the F^H D / Q gather.

This module only draws inputs: trajectories, voxel grids and per-sample values.
It computes nothing of the reconstruction itself (no Mu, no phase, no sum), so
both the CUDA path and the CPU oracle can take their inputs from it without
sharing any of the method's arithmetic.

Every array is float32, structure-of-arrays, as the gather kernel of the
"Iterative MRI reconstruction" chapter (section 17.3, Fig. 17.10/17.11) indexes
them: k-space coordinates kx, ky, kz and weights rPhi, iPhi, rD, iD per sample
m < M; voxel coordinates x, y, z per voxel n < N.  k is in cycles per voxel
unit and voxels sit at integer coordinates, matching the 2*PI*(k.x) phase of the
printed register-promoted kernel.

Random numbers come from numpy's PCG64 (``default_rng(seed)``).  Draw order:
k first (only when k itself is random), then rPhi, iPhi, rD, iD.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

F32 = np.float32


# --------------------------------------------------------------------------
# voxel grids
# --------------------------------------------------------------------------

def voxel_grid(L: int, Ly: int | None = None, Lz: int | None = None):
    """Integer voxel coordinates -L/2 .. L/2-1 per axis, x fastest.

    Voxel n = (iz*Ly + iy)*Lx + ix sits at (ix - Lx/2, iy - Ly/2, iz - Lz/2).
    Returns float32 arrays x, y, z of length Lx*Ly*Lz.
    """
    Lx = L
    Ly = L if Ly is None else Ly
    Lz = L if Lz is None else Lz
    ix = np.arange(Lx) - Lx // 2
    iy = np.arange(Ly) - Ly // 2
    iz = np.arange(Lz) - Lz // 2
    z, y, x = np.meshgrid(iz, iy, ix, indexing="ij")
    return (x.reshape(-1).astype(F32), y.reshape(-1).astype(F32),
            z.reshape(-1).astype(F32))


def grid_axes(L: int, Ly: int | None = None, Lz: int | None = None):
    """The axes of voxel_grid: xs, ys, zs with voxel_grid = xs x ys x zs, x fastest."""
    Ly = L if Ly is None else Ly
    Lz = L if Lz is None else Lz
    return tuple((np.arange(n) - n // 2).astype(F32) for n in (L, Ly, Lz))


def voxel_subset(N: int, count: int, seed: int) -> np.ndarray:
    """Sorted, distinct voxel indices (int64) drawn uniformly from range(N)."""
    count = min(count, N)
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(N, size=count, replace=False)).astype(np.int64)


# --------------------------------------------------------------------------
# trajectories
# --------------------------------------------------------------------------

def traj_uniform_random(M: int, rng: np.random.Generator):
    """M samples i.i.d. uniform in [-0.5, 0.5)^3 cycles/voxel."""
    k = rng.random((3, M)) - 0.5
    return k[0].astype(F32), k[1].astype(F32), k[2].astype(F32)


def traj_stack_of_spirals(planes: int, interleaves: int, points: int,
                          turns: float):
    """Stack of Archimedean spirals inside the ball |k| <= 0.5.

    Plane p sits at kz_p = -0.5 + (p + 0.5)/planes and has radius
    R_p = sqrt(0.25 - kz_p^2).  Interleave i of that plane is the spiral
    r_s = R_p * s/(points-1), angle_s = 2*pi*turns*s/(points-1) + 2*pi*i/interleaves
    for s < points.  Sample order: plane-major, then interleave, then point.
    """
    p = np.arange(planes, dtype=np.float64)
    kz_p = -0.5 + (p + 0.5) / planes
    R_p = np.sqrt(np.maximum(0.25 - kz_p * kz_p, 0.0))
    s = np.arange(points, dtype=np.float64) / (points - 1)
    i = np.arange(interleaves, dtype=np.float64)
    ang = (2.0 * math.pi * turns * s[None, :]
           + 2.0 * math.pi * i[:, None] / interleaves)          # [I, S]
    r = R_p[:, None, None] * s[None, None, :]                    # [P, 1, S]
    kx = r * np.cos(ang)[None, :, :]
    ky = r * np.sin(ang)[None, :, :]
    kz = np.broadcast_to(kz_p[:, None, None], kx.shape)
    return (kx.reshape(-1).astype(F32), ky.reshape(-1).astype(F32),
            np.ascontiguousarray(kz).reshape(-1).astype(F32))


def traj_radial_fibonacci(lines: int, points: int):
    """3D radial lines through the origin on Fibonacci-sphere directions.

    Direction i: z_i = 1 - (2i+1)/lines, azimuth i*pi*(3 - sqrt 5).  Point j on
    a line sits at t_j = (j - (points-1)/2)/(points-1), so t covers
    [-0.5, 0.5] and no point lands exactly on k = 0.  Sample order: line-major.
    """
    i = np.arange(lines, dtype=np.float64)
    zi = 1.0 - (2.0 * i + 1.0) / lines
    phi = i * math.pi * (3.0 - math.sqrt(5.0))
    rho = np.sqrt(np.maximum(1.0 - zi * zi, 0.0))
    d = np.stack([rho * np.cos(phi), rho * np.sin(phi), zi])     # [3, lines]
    j = np.arange(points, dtype=np.float64)
    t = (j - (points - 1) / 2.0) / (points - 1)
    k = d[:, :, None] * t[None, None, :]                         # [3, lines, pts]
    return (k[0].reshape(-1).astype(F32), k[1].reshape(-1).astype(F32),
            k[2].reshape(-1).astype(F32))


def traj_cartesian(Lx: int, Ly: int, Lz: int):
    """Uniform Cartesian k-grid k_d = j/L_d, j = -L_d/2 .. L_d/2-1, kx fastest."""
    jx = (np.arange(Lx) - Lx // 2) / Lx
    jy = (np.arange(Ly) - Ly // 2) / Ly
    jz = (np.arange(Lz) - Lz // 2) / Lz
    kz, ky, kx = np.meshgrid(jz, jy, jx, indexing="ij")
    return (kx.reshape(-1).astype(F32), ky.reshape(-1).astype(F32),
            kz.reshape(-1).astype(F32))


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------

@dataclass
class Workload:
    name: str
    kind: str                     # "fhd", "q" or "fhd_batched"
    L: int
    kx: np.ndarray
    ky: np.ndarray
    kz: np.ndarray
    x: np.ndarray
    y: np.ndarray
    z: np.ndarray
    rPhi: np.ndarray
    iPhi: np.ndarray
    rD: np.ndarray | None = None  # [M] or [B, M] (coil-major) for batched
    iD: np.ndarray | None = None
    B: int = 1
    meta: dict = field(default_factory=dict)

    @property
    def M(self) -> int:
        return int(self.kx.shape[0])

    @property
    def N(self) -> int:
        return int(self.x.shape[0])

    @property
    def pairs(self) -> int:
        return self.M * self.N

    def axes(self):
        """xs, ys, zs of the workload's voxel grid, read from its coordinates
        (voxel n = (iz L + iy) L + ix), so a shifted slab keeps its shift."""
        L = self.L
        return (np.ascontiguousarray(self.x[:L]), np.ascontiguousarray(self.y[0:L * L:L]),
                np.ascontiguousarray(self.z[0::L * L]))


WORKLOADS = {
    "fhd_tiny": "FHD tiny: 16^3 voxels, M=2048 uniform random k, seed 0",
    "fhd_64": "FHD 64^3 voxels, M=32,768 stack of spirals (32 planes x 4 interleaves x 256)",
    "fhd_128_radial": "FHD 128^3 voxels, M=262,144 3D radial (1024 Fibonacci lines x 256)",
    "q_128": "Q 128^3 voxels, M=1,048,576 stack of spirals (128 planes x 16 interleaves x 512)",
    "fhd_batched_128": "Batched FHD, 8 coils, 128^3 voxels, M=524,288 stack of spirals (64 x 16 x 512)",
}


def _normal(rng, shape):
    return rng.standard_normal(shape).astype(F32)


def make_workload(name: str, seed: int | None = None, L: int | None = None) -> Workload:
    """Build one of the named workloads.

    ``L`` overrides the voxel-grid edge (the trajectory is unchanged) so tests
    can run a workload's trajectory against a small grid.
    """
    if name == "fhd_tiny":
        seed = 0 if seed is None else seed
        rng = np.random.default_rng(seed)
        kx, ky, kz = traj_uniform_random(2048, rng)
        M = kx.shape[0]
        rPhi, iPhi, rD, iD = (_normal(rng, M) for _ in range(4))
        L = 16 if L is None else L
        x, y, z = voxel_grid(L)
        return Workload(name, "fhd", L, kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD)

    if name == "fhd_64":
        seed = 1 if seed is None else seed
        rng = np.random.default_rng(seed)
        kx, ky, kz = traj_stack_of_spirals(32, 4, 256, turns=64 / (2 * 4))
        M = kx.shape[0]
        rPhi, iPhi, rD, iD = (_normal(rng, M) for _ in range(4))
        L = 64 if L is None else L
        x, y, z = voxel_grid(L)
        return Workload(name, "fhd", L, kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD)

    if name == "fhd_128_radial":
        seed = 2 if seed is None else seed
        rng = np.random.default_rng(seed)
        kx, ky, kz = traj_radial_fibonacci(1024, 256)
        M = kx.shape[0]
        rPhi, iPhi, rD, iD = (_normal(rng, M) for _ in range(4))
        kabs = np.sqrt(kx.astype(np.float64) ** 2 + ky.astype(np.float64) ** 2
                       + kz.astype(np.float64) ** 2)
        scale = 1.0 / (1.0 + kabs / 0.05)
        rD = (rD * scale).astype(F32)
        iD = (iD * scale).astype(F32)
        L = 128 if L is None else L
        x, y, z = voxel_grid(L)
        return Workload(name, "fhd", L, kx, ky, kz, x, y, z, rPhi, iPhi, rD, iD)

    if name == "q_128":
        seed = 3 if seed is None else seed
        rng = np.random.default_rng(seed)
        kx, ky, kz = traj_stack_of_spirals(128, 16, 512, turns=128 / (2 * 16))
        M = kx.shape[0]
        rPhi, iPhi = _normal(rng, M), _normal(rng, M)
        L = 128 if L is None else L
        x, y, z = voxel_grid(L)
        return Workload(name, "q", L, kx, ky, kz, x, y, z, rPhi, iPhi)

    if name == "fhd_batched_128":
        seed = 4 if seed is None else seed
        rng = np.random.default_rng(seed)
        kx, ky, kz = traj_stack_of_spirals(64, 16, 512, turns=128 / (2 * 16))
        M = kx.shape[0]
        B = 8
        rPhi, iPhi = _normal(rng, M), _normal(rng, M)
        rD = rng.standard_normal((B, M))
        iD = rng.standard_normal((B, M))
        k = np.stack([kx, ky, kz]).astype(np.float64)            # [3, M]
        b = np.arange(B)
        kb = 0.2 * np.stack([np.cos(2 * math.pi * b / B),
                             np.sin(2 * math.pi * b / B), np.zeros(B)])  # [3, B]
        d2 = ((k[:, None, :] - kb[:, :, None]) ** 2).sum(axis=0)  # [B, M]
        g = np.exp(-d2 / (2 * 0.25 ** 2))
        rD = (rD * g).astype(F32)
        iD = (iD * g).astype(F32)
        L = 128 if L is None else L
        x, y, z = voxel_grid(L)
        return Workload(name, "fhd_batched", L, kx, ky, kz, x, y, z, rPhi, iPhi,
                        rD, iD, B=B)

    raise KeyError(f"unknown workload {name!r}; known: {sorted(WORKLOADS)}")


def random_fhd_inputs(M: int, N: int, seed: int, kmax: float = 0.5,
                      coord_max: float = 64.0, B: int | None = None):
    """Free-form random inputs for edge-case and tail tests.

    k ~ U[-kmax, kmax)^3, voxel coordinates ~ U[-coord_max, coord_max)^3 (not
    restricted to integers), Phi and D ~ N(0,1); D is [B, M] when B is given.
    """
    rng = np.random.default_rng(seed)
    k = ((rng.random((3, M)) * 2.0 - 1.0) * kmax).astype(F32)
    xyz = ((rng.random((3, N)) * 2.0 - 1.0) * coord_max).astype(F32)
    rPhi, iPhi = _normal(rng, M), _normal(rng, M)
    shape = M if B is None else (B, M)
    rD, iD = _normal(rng, shape), _normal(rng, shape)
    return dict(kx=k[0], ky=k[1], kz=k[2], x=xyz[0], y=xyz[1], z=xyz[2],
                rPhi=rPhi, iPhi=iPhi, rD=rD, iD=iD)
