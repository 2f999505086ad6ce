"""The library's launches inside CUDA graphs: a grouped step (the TMA form), a
pipelined step over two streams and a staged offload step over three are captured
once and replayed; every replay equals the same call made directly, bit for bit.
The last cases capture the first library call of a fresh process."""
import os
import subprocess
import sys

import pytest

import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")
bench = pytest.importorskip("bench")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _warm(torch, W=8):
    """One eager call first: the library's per-device sizing queries stay outside the capture."""
    units = bench.build_all_ranks(bench.sweep_workload(4096, W), W, torch, fs, synth)[0]
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(1))
    torch.cuda.synchronize()


def _outputs(units):
    outs = []
    for u in units:
        for name in ("master", "exp_avg", "exp_avg_sq", "full_out"):
            outs += [t.clone() for t in u[name]]
    return outs


def test_grouped_step_replays_from_a_graph():
    torch = gu.torch()
    n, W = 40_000_000, 8  # 19,536 chunks: the TMA form on a 152-SM GB300
    direct = bench.build_all_ranks(bench.sweep_workload(n, W), W, torch, fs, synth)[0]
    graphed = bench.build_all_ranks(bench.sweep_workload(n, W), W, torch, fs, synth)[0]
    hp = gu.adam_hyper(3)
    s = torch.cuda.Stream()
    _warm(torch)
    batch = fs.UnitBatch(graphed)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fs.fsdp_shard_step_grouped(batch, 0, W, hp, stream=torch.cuda.current_stream())
    for _ in range(3):
        g.replay()
        fs.fsdp_shard_step_grouped(direct, 0, W, hp, stream=s)
    torch.cuda.synchronize()
    for a, b in zip(_outputs(direct), _outputs(graphed)):
        assert torch.equal(a.view(torch.int8), b.view(torch.int8))


@pytest.mark.parametrize("shard", [300_000, 4_300_000])
def test_pipelined_step_replays_from_a_graph(shard):
    """Copies on one stream, steps on another, ordered by events: captured as one graph
    (a unit of 4.3 M shard elements moves in pieces, with 2D copies)."""
    torch = gu.torch()
    _warm(torch)
    wl = bench.sweep_workload(8 * shard + 3, 8)
    units, info, bufs = bench.build_local_rank(wl, 2, torch, fs, synth)
    units2, _, _ = bench.build_local_rank(wl, 2, torch, fs, synth)
    batch, staging, slot, keep = bench.pipeline_setup(torch, fs, units, info, 2, 2)
    batch2, staging2, slot2, keep2 = bench.pipeline_setup(torch, fs, units2, info, 2, 2)
    hp = gu.adam_hyper(5)
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=compute):
        fs.fsdp_pipeline_step(batch2, 2, staging2, slot2, 2, hp, compute=torch.cuda.current_stream(), copy=copy)
    for _ in range(2):
        g.replay()
        fs.fsdp_pipeline_step(batch, 2, staging, slot, 2, hp, compute=compute, copy=copy)
    torch.cuda.synchronize()
    for u, v in zip(units, units2):
        for name in ("master", "exp_avg", "exp_avg_sq", "full_out"):
            assert torch.equal(u[name][0].view(torch.int8), v[name][0].view(torch.int8)), name
    assert torch.equal(keep[1], keep2[1])  # the bf16 shard read back to host memory


def test_staged_offload_replays_from_a_graph():
    """Copies in, steps and copies back on three streams, captured from the compute stream."""
    torch = gu.torch()
    _warm(torch)
    wl = bench.sweep_workload(8 * 200_000 + 5, 8)
    sets = []
    for _ in range(2):
        units, info, bufs = bench.build_local_rank(wl, 1, torch, fs, synth)
        host = {n: bufs[n].cpu().pin_memory() for n in ("master", "exp_avg", "exp_avg_sq")}
        so = 0
        off = []
        for u in units:
            S = u["layout"].shard_numel
            off.append(dict(layout=u["layout"], grads=u["grads"], master=host["master"][so:so + S],
                            exp_avg=host["exp_avg"][so:so + S], exp_avg_sq=host["exp_avg_sq"][so:so + S],
                            other_shards=u["other_shards"], full_out=u["full_out"][0]))
            so += S
        slot = (max(u["layout"].shard_numel for u in units) + 3) // 4 * 4
        staging = torch.empty(3 * 3 * slot, device="cuda")
        sets.append((units, host, fs.OffloadBatch(off), staging, slot))
    hp = gu.adam_hyper(2)
    compute, h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    direct, graphed = sets
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=compute):
        fs.fsdp_offload_step(graphed[2], 1, graphed[3], graphed[4], 3, hp, compute=torch.cuda.current_stream(),
                             h2d=h2d, d2h=d2h)
    for _ in range(2):
        g.replay()
        fs.fsdp_offload_step(direct[2], 1, direct[3], direct[4], 3, hp, compute=compute, h2d=h2d, d2h=d2h)
    torch.cuda.synchronize()
    for n in ("master", "exp_avg", "exp_avg_sq"):
        assert torch.equal(direct[1][n].view(torch.int32), graphed[1][n].view(torch.int32)), n
    for u, v in zip(direct[0], graphed[0]):
        assert torch.equal(u["full_out"][0], v["full_out"][0])


_FIRST_CALL = r"""
import sys
import torch
sys.path[:0] = [sys.argv[1], sys.argv[2]]
import bench, fully_sharded_gb300 as fs, gpu_util as gu, synth
torch.cuda.set_device(0)
case = sys.argv[3]
W = 8 if case in ("tma", "pipeline") else 4
s = torch.cuda.Stream()
g = torch.cuda.CUDAGraph()
if case == "pipeline":
    wl = bench.sweep_workload(W * 300_000 + 3, W)
    sets = []
    for _ in range(2):
        units, info, bufs = bench.build_local_rank(wl, 2, torch, fs, synth)
        sets.append((units, bench.pipeline_setup(torch, fs, units, info, 2, 2)))
    (u1, (b1, st1, sl1, k1)), (u2, (b2, st2, sl2, k2)) = sets
    copy = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        fs.fsdp_pipeline_step(b2, 2, st2, sl2, 2, gu.adam_hyper(5), compute=torch.cuda.current_stream(), copy=copy)
    g.replay()
    fs.fsdp_pipeline_step(b1, 2, st1, sl1, 2, gu.adam_hyper(5), compute=s, copy=copy)
    pairs = [(a[n][0], b[n][0]) for a, b in zip(u1, u2) for n in ("master", "exp_avg", "exp_avg_sq", "full_out")]
else:
    wl = bench.sweep_workload(40_000_000 if case == "tma" else 4_000_003, W)
    direct = bench.build_all_ranks(wl, W, torch, fs, synth)[0]
    graphed = bench.build_all_ranks(wl, W, torch, fs, synth)[0]
    batch = fs.UnitBatch(graphed)
    with torch.cuda.graph(g, stream=s):
        fs.fsdp_shard_step_grouped(batch, 0, W, gu.adam_hyper(3), stream=torch.cuda.current_stream())
    g.replay()
    fs.fsdp_shard_step_grouped(direct, 0, W, gu.adam_hyper(3), stream=s)
    pairs = [(a[n][i], b[n][i]) for a, b in zip(direct, graphed)
             for n in ("master", "exp_avg", "exp_avg_sq", "full_out") for i in range(len(a[n]))]
torch.cuda.synchronize()
assert all(torch.equal(x.view(torch.int8), y.view(torch.int8)) for x, y in pairs)
code = fs.fsdp_device_status()
assert code == 0, code
print("same bits")
"""


@pytest.mark.parametrize("case", ["tma", "ldg", "pipeline"])
def test_first_call_of_a_process_inside_a_capture(case):
    """A fresh process whose first library call is made while a stream is being captured
    (the per-device sizing queries then run inside the capture): the replay equals the
    same call made directly, bit for bit. One process per case, so nothing is cached."""
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    r = subprocess.run([sys.executable, "-c", _FIRST_CALL, root, here, case], capture_output=True, text=True,
                       timeout=600, cwd=root)
    assert r.returncode == 0 and "same bits" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
