"""The multi-rank benchmark path on CPU: two gloo ranks.

With N GPUs every rank works on its own voxel slab (z shifted by rank * L)
against the same trajectory; no data moves between ranks, only the barrier and
the max over ranks of the step time.  Here each rank computes its slab with
the oracle; the slabs together must equal one computation over the stacked
volume, and the timing reduction must return the maximum on every rank.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from non_cartesian_mri_gb300 import workloads as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    d = bench.Dist(world, rank, torch.device("cpu"))
    try:
        w = bench.slab(wl.make_workload("fhd_tiny", L=6), rank)
        f = oracle.fhd(w.kx, w.ky, w.kz, w.x, w.y, w.z, w.rPhi, w.iPhi, w.rD, w.iD)
        d.barrier()
        got = d.max(1.5 + rank)
        parts = [torch.zeros(2 * f.size, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(parts, torch.from_numpy(np.concatenate([f.real, f.imag])))
        if rank == 0:
            full = np.concatenate([p.numpy()[:f.size] + 1j * p.numpy()[f.size:] for p in parts])
            np.save(os.path.join(outdir, "gathered.npy"), full)
        np.save(os.path.join(outdir, f"max{rank}.npy"), np.array([got]))
        np.save(os.path.join(outdir, f"z{rank}.npy"), w.z)
        np.save(os.path.join(outdir, f"zs{rank}.npy"), w.axes()[2])
    finally:
        d.close()


@pytest.mark.parametrize("world", [2])
def test_two_rank_slabs_equal_the_stacked_volume(tmp_path, world):
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    w = wl.make_workload("fhd_tiny", L=6)
    xs = np.concatenate([w.x] * world)
    ys = np.concatenate([w.y] * world)
    zs = np.concatenate([w.z + np.float32(r * w.L) for r in range(world)]).astype(np.float32)
    ref = oracle.fhd(w.kx, w.ky, w.kz, xs, ys, zs, w.rPhi, w.iPhi, w.rD, w.iD)
    got = np.load(tmp_path / "gathered.npy")
    np.testing.assert_array_equal(got, ref)
    for r in range(world):
        assert float(np.load(tmp_path / f"max{r}.npy")[0]) == 1.5 + world - 1
    z0, z1 = np.load(tmp_path / "z0.npy"), np.load(tmp_path / "z1.npy")
    np.testing.assert_array_equal(z1 - z0, np.full_like(z0, w.L))
    # the grid entry points get each slab's own z axis
    zs0, zs1 = np.load(tmp_path / "zs0.npy"), np.load(tmp_path / "zs1.npy")
    np.testing.assert_array_equal(zs1 - zs0, np.full_like(zs0, w.L))


def test_slab_axes_expand_to_its_coordinates():
    import bench
    for rank in (0, 1, 3):
        w = bench.slab(wl.make_workload("fhd_tiny", L=6), rank)
        xs, ys, zs = w.axes()
        z, y, x = np.meshgrid(zs, ys, xs, indexing="ij")
        np.testing.assert_array_equal(x.reshape(-1), w.x)
        np.testing.assert_array_equal(y.reshape(-1), w.y)
        np.testing.assert_array_equal(z.reshape(-1), w.z)


def test_single_rank_dist_is_a_no_op():
    import bench
    d = bench.Dist(1, 0, torch.device("cpu"))
    d.barrier()
    assert d.max(3.25) == 3.25
    d.close()
