"""The bench's CPU-baseline helpers on the host: the oracle on one core and on
every core (threads, each on its own copy of the state), and the CPU model."""
import numpy as np

import bench
import oracle


def _sample(W=4, n_s=4096, rank=1, seed=0):
    rng = np.random.default_rng(seed)
    grads = np.zeros((W, W * n_s), np.uint16)
    for k in range(W):
        grads[k, rank * n_s:(rank + 1) * n_s] = (
            rng.standard_normal(n_s).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    master = rng.standard_normal(n_s).astype(np.float32) * 0.02
    m = np.abs(rng.standard_normal(n_s).astype(np.float32)) * 1e-4
    v = np.abs(rng.standard_normal(n_s).astype(np.float32)) * 1e-4
    others = [None if k == rank else rng.integers(0, 1 << 15, n_s).astype(np.uint16) for k in range(W)]
    return grads, master, m, v, others, rank, n_s


def test_all_core_baseline_uses_every_core_and_leaves_the_sample_unchanged():
    ora = oracle.load()
    grads, master, m, v, others, rank, n_s = _sample()
    before = master.copy(), m.copy(), v.copy()
    per = (6 * grads.shape[0] + 22) * n_s
    res = bench.cpu_baseline_all_cores(ora, grads, master, m, v, others, rank, n_s, per, seconds=0.2)
    assert res["cores"] == bench.host_cores() >= 1
    assert res["value"] > 0 and res["unit"] == bench.UNIT
    # each thread stepped its own copy of the state
    for a, b in zip((master, m, v), before):
        assert np.array_equal(a, b)


def test_thread_results_equal_a_single_oracle_step():
    # the threads run the unchanged oracle: one step from the sample equals the oracle's own
    ora = oracle.load()
    grads, master, m, v, others, rank, n_s = _sample(seed=3)
    a = master.copy(), m.copy(), v.copy()
    b = master.copy(), m.copy(), v.copy()
    bench.run_oracle_step(ora, grads, *a, others, rank, n_s, 1)
    bench.run_oracle_step(ora, grads, *b, others, rank, n_s, 1)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert not np.array_equal(a[0], master)


def test_cpu_model_is_named():
    name = bench.cpu_model()
    assert isinstance(name, str) and name
