"""GB300-native hot path of iterative non-Cartesian MRI reconstruction.

Public API (torch tensors in, torch tensors out; see ``binding``):
    mu, fhd, q, fhd_batched, forward and their grid forms; fft3,
    toeplitz_kernel, toeplitz_apply, cg_solve (find rho); gridding; plan,
    device_errors, microbench
The CUDA library is built with ``non_cartesian_mri_gb300.build.build()``.
``workloads`` holds the seeded synthetic input generators.
"""

_API = ("mu", "fhd", "q", "fhd_batched", "forward", "forward_grid", "fhd_grid", "q_grid", "fhd_batched_grid", "plan",
        "plan_grid", "plan_grid_batched",
        "device_errors", "microbench", "mma_probe", "wait_selftest",
        "fft3", "toeplitz_kernel", "toeplitz_apply", "cg_solve", "gridding",
        "status_string", "MriError", "load", "lib_path", "TRIG", "gather_timing")


def __getattr__(name):
    if name in _API:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(f"module {__name__!r} has no attribute {name!r}")


__all__ = list(_API)
