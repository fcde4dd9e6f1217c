"""Seeded synthetic inputs for the emulated-DGEMM and INT8-GEMM workloads.

This module holds no arithmetic of the method: it only draws random matrices.
Both the CUDA-path tests/bench and the CPU oracle take their inputs from here.

The five workloads (shapes and value distributions of the emulation papers'
cases; all data synthetic, seeded with numpy's default_rng):

* dgemm_256_uniform   M=N=K=256, A, B ~ U(-1, 1), seed 1
* igemm_s8_4096       M=N=K=4096, int8 uniform in [-128, 127], seed 2
* dgemm_8192_wide     M=N=K=8192, entries u 2^e, u ~ U(-1, 1), e uniform
                      integer in [-10, 10] per entry, seed 3
* dgemv_16384_n{1,8}  A 16384 x 16384 ~ N(0, 1), B 16384 x n, seed 4
* dgemm_4096_k65536   M=N=4096, K=65536, A, B ~ N(0, 1), seed 5

and the INT4 x INT8 product of the four-product encoding (a sub-record of
the measurement, not a metric workload): igemm_s4s8_4096, M=N=K=4096, A
uniform in [-8, 7] (one value per int8), B uniform int8, seed 6.
"""

import numpy as np

WORKLOADS = {
    "dgemm_256_uniform": dict(kind="dgemm", m=256, n=256, k=256, seed=1, dist="uniform", r=13),
    "igemm_s8_4096": dict(kind="igemm", m=4096, n=4096, k=4096, seed=2, dist="int8"),
    "dgemm_8192_wide": dict(kind="dgemm", m=8192, n=8192, k=8192, seed=3, dist="wide", r=13),
    "dgemv_16384_n1": dict(kind="dgemm", m=16384, n=1, k=16384, seed=4, dist="normal", r=12),
    "dgemv_16384_n8": dict(kind="dgemm", m=16384, n=8, k=16384, seed=4, dist="normal", r=12),
    "dgemm_4096_k65536": dict(kind="dgemm", m=4096, n=4096, k=65536, seed=5, dist="normal", r=11),
}


def draw(rng, shape, dist):
    """One matrix of the given distribution."""
    if dist == "uniform":
        return rng.uniform(-1.0, 1.0, size=shape)
    if dist == "normal":
        return rng.standard_normal(size=shape)
    if dist == "wide":
        u = rng.uniform(-1.0, 1.0, size=shape)
        e = rng.integers(-10, 11, size=shape)
        return np.ldexp(u, e)
    if dist == "int8":
        return rng.integers(-128, 128, size=shape, dtype=np.int8)
    raise ValueError("unknown distribution %r" % dist)


def make_pair(m, n, k, seed, dist):
    """(A, B) with A m x k and B k x n, row-major, drawn from one generator
    (dist "int4_int8": A in [-8, 7] and B in [-128, 127], both int8)."""
    rng = np.random.default_rng(seed)
    if dist == "int4_int8":
        A = rng.integers(-8, 8, size=(m, k), dtype=np.int8)
        B = rng.integers(-128, 128, size=(k, n), dtype=np.int8)
        return A, B
    A = np.ascontiguousarray(draw(rng, (m, k), dist))
    B = np.ascontiguousarray(draw(rng, (k, n), dist))
    return A, B


def workload_inputs(name):
    """(A, B, spec) for a named workload."""
    spec = WORKLOADS[name]
    A, B = make_pair(spec["m"], spec["n"], spec["k"], spec["seed"], spec["dist"])
    return A, B, spec


def sample_indices(n, count, seed):
    """Sorted distinct indices in [0, n) for sampled checks."""
    rng = np.random.default_rng(seed)
    count = min(count, n)
    return np.sort(rng.choice(n, size=count, replace=False))
