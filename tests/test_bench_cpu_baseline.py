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


def _hybrid_units(W=8, F=4, P=8 * 1000 + 3, seed=0):
    import torch
    import fully_sharded_gb300 as fs
    lay, _ = fs.fsdp_flatten_layout([P], W, F)
    S, padded, R = lay.shard_numel, lay.padded_numel, W // F
    gen = torch.Generator().manual_seed(seed)
    g = (torch.randn((W, padded), generator=gen) * 1e-3).to(torch.bfloat16).view(torch.int16)
    st = [torch.randn((R, padded), generator=gen).abs() * 1e-4 for _ in range(3)]
    view = lambda a, r: a[r // F, (r % F) * S:(r % F + 1) * S]  # noqa: E731
    return [dict(layout=lay, grads=[g[k] for k in range(W)], master=[view(st[0], r) for r in range(W)],
                 exp_avg=[view(st[1], r) for r in range(W)], exp_avg_sq=[view(st[2], r) for r in range(W)],
                 other_shards=None, full_out=[torch.zeros(padded, dtype=torch.int16) for _ in range(R)])], g, st


def test_all_ranks_sample_takes_the_head_of_every_position():
    units, g, st = _hybrid_units()
    lay = units[0]["layout"]
    S = lay.shard_numel
    grads, (master, m, v), W, F, n_s = bench.oracle_sample_all_ranks(units, 100)
    assert (W, F, n_s) == (8, 4, 100) and grads.shape == (8, 400)
    gn = g.numpy().view(np.uint16)
    for k in range(W):
        for p in range(F):
            assert np.array_equal(grads[k, p * 100:(p + 1) * 100], gn[k, p * S:p * S + 100])
    for r in range(W):
        assert np.array_equal(master[r], st[0][r // F, (r % F) * S:(r % F) * S + 100].numpy())
        assert np.array_equal(v[r], st[2][r // F, (r % F) * S:(r % F) * S + 100].numpy())


def test_all_ranks_baseline_times_the_oracle_and_leaves_the_units_unchanged():
    import torch
    units, g, st = _hybrid_units(seed=1)
    before = [t.clone() for t in st]
    res = bench.cpu_baseline_all_ranks(units, torch, seconds=0.2, elems=4096)
    assert res["value"] > 0 and res["unit"] == bench.UNIT and res["cores"] == 1 and res["kind"] == "oracle"
    assert "F=4" in res["sample"]
    for a, b in zip(st, before):
        assert torch.equal(a, b)


def test_cpu_model_is_named():
    name = bench.cpu_model()
    assert isinstance(name, str) and name


def _info(W=8, elems=842301952, bytes_per_elem=70, units=33):
    return dict(W=W, units=units, params=6738415616, elems_per_step=elems, bytes_per_step=bytes_per_elem * elems,
                mode="local-rank", shard_elems=elems)


def test_bench_line_carries_the_contract_keys_and_its_arithmetic():
    info = _info()
    clocks = {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 14}
    line = bench.bench_line(info, "llama7b_local_rank", 1, 100, 5, 8.6, 860.0, 1, 1, 129e6, clocks,
                            peak=(6786.2, "measured"))
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
              "scaling", "vs_baseline", "dtype", "data", "config", "roofline", "gpu_launches", "clocks"):
        assert k in line, k
    assert line["config"]["workload"] == "llama7b_local_rank"
    assert line["higher_is_better"] is True and line["scaling"] == "weak" and line["vs_baseline"] is None
    gbs = 70 * 842301952 / 8.6e-3 / 1e9
    assert abs(line["value"] - gbs) < 0.01
    r = line["roofline"]
    assert set(r) >= {"bound", "achieved", "peak", "unit", "frac", "traffic"}
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 6786.2
    assert abs(r["achieved"] - gbs) < 0.01 and abs(r["frac"] - gbs / 6786.2) < 1e-4
    assert r["kernel"] == "fsdp::tma_kernel<8>"
    assert line["gpu_launches"] == 100 and line["clocks"] is clocks
    assert "inputs larger than L2" in line["config"]["l2"]


def test_bench_line_aggregates_ranks_and_names_the_ldg_form():
    # two GPU processes, the slowest 10 ms per step; this rank's launches took 9 ms on average;
    # two launches per step, none in the TMA form
    info = _info(W=4, elems=10 ** 6, bytes_per_elem=2 * 4 + 26, units=1)
    line = bench.bench_line(info, "sweep_1000000_W4", 2, 10, 3, 10.0, 180.0, 2, 0, 129e6, None,
                            peak=(6800.0, "fallback"))
    per_rank = 34 * 10 ** 6
    assert abs(line["value"] - 2 * per_rank / 10e-3 / 1e9) < 0.01  # rounded to 2 decimals
    assert abs(line["roofline"]["achieved"] - per_rank / 2 / 9e-3 / 1e9) < 0.01
    assert line["roofline"]["kernel"] == "fsdp::segment_kernel<4>" and line["roofline"]["peak_source"] == "fallback"
    assert line["gpu_launches"] == 20 and line["n_gpus"] == 2
    assert "L2-resident" in line["config"]["l2"]


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) runs without a GPU."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--steps", "2",
                          "--warmup", "3", "--ref-sample", "65536"], capture_output=True, text=True, timeout=300,
                         cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == bench.UNIT and d["metric"] == bench.METRIC
    assert d["config"]["workload"] == "llama7b_local_rank" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_loads_only_the_oracle():
    """The reference arm is the oracle alone: the CUDA library's package is never imported
    and its shared object is never mapped into the process."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    probe = ("import runpy, sys\n"
             "sys.argv = ['bench.py', '--impl', 'reference', '--steps', '1', '--warmup', '3', '--ref-sample', '4096']\n"
             "runpy.run_path('bench.py', run_name='__main__')\n"
             "maps = open('/proc/self/maps').read()\n"
             "print('PACKAGE', 'fully_sharded_gb300' in sys.modules)\n"
             "print('LIBRARY', 'libfsdp_gb300' in maps)\n"
             "print('ORACLE', 'libfsdp_oracle' in maps)\n")
    out = subprocess.run([sys.executable, "-c", probe], capture_output=True, text=True, timeout=300, cwd=root)
    assert out.returncode == 0, out.stderr[-2000:]
    assert "PACKAGE False" in out.stdout and "LIBRARY False" in out.stdout and "ORACLE True" in out.stdout


def test_bench_refuses_a_gpu_count_it_was_not_launched_with():
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2"], capture_output=True,
                         text=True, timeout=120, cwd=root)
    assert out.returncode != 0 and "nproc-per-node" in out.stderr


def test_oracle_parts_baseline_times_every_separate_call():
    res = bench.oracle_parts_baseline(4, 4096, seconds=0.05)
    for key in ("reduce_scatter_GB_per_s", "adam_GB_per_s", "all_gather_GB_per_s", "gather_state_f32_GB_per_s",
                "pack_f32_GB_per_s", "unpack_f32_GB_per_s"):
        assert res[key] > 0, key
    assert res["cores"] == 1 and res["kind"] == "oracle" and res["unit"] == bench.UNIT


def test_e2e_reports_unavailable_when_pinned_buffers_fail(monkeypatch):
    """A failed page-locked allocation makes the e2e record say so (no crash, no timing)."""
    import argparse

    def fail(*a, **k):
        raise RuntimeError("CUDA error: out of memory\nmore lines")

    monkeypatch.setattr(bench, "pipeline_setup", fail)
    args = argparse.Namespace(steps=4, e2e_steps=4, warmup=3)
    info = dict(W=8, shard_elems=1000, bytes_per_step=70 * 1000)
    e = bench.e2e_local_rank(args, None, None, None, None, [], info, None, 0, None, 1, None)
    assert e["value"] is None and e["unit"] == bench.UNIT
    assert e["h2d_bytes_per_step"] == 16 * 1000 and e["d2h_bytes_per_step"] == 2 * 1000
    assert "could not be allocated" in e["unavailable"] and "out of memory" in e["unavailable"]
    assert "more lines" not in e["unavailable"]
