"""Randomized parity sweep of the fused step against the oracle.

Each case draws a world size W (1..64), a sharding factor F dividing W, an
owned rank range, a tensor split of 1..5 tensors (empty tensors allowed), a
step counter, and whether the state shards are separate buffers or views of
one flat buffer (misaligned slices). Every output must be bit-identical.
"""
import numpy as np
import pytest

from test_gpu_parity import run_step_case

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _case(seed):
    rng = np.random.default_rng(seed)
    W = int(rng.choice([1, 2, 3, 4, 5, 6, 8, 12, 16, 24, 32, 64]))
    F = int(rng.choice([f for f in range(1, W + 1) if W % f == 0]))
    n_t = int(rng.integers(1, 6))
    numels = [int(x) for x in rng.integers(0, 6000, size=n_t)]
    if sum(numels) == 0:
        numels[0] = 1
    rb = int(rng.integers(0, W))
    re = int(rng.integers(rb + 1, W + 1))
    step = int(rng.integers(1, 100))
    views = bool(rng.integers(0, 2))
    return W, F, numels, rb, re, step, views


@pytest.mark.parametrize("seed", range(40))
def test_random_case(ora, seed):
    W, F, numels, rb, re, step, views = _case(seed)
    run_step_case(ora, W, F, numels, rb, re, step=step, state_views=views, key_base=50000 + seed)
