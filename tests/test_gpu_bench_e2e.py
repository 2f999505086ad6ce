"""The bench's end-to-end measurement (the pipelined call with host buffers) on a small
local-rank workload: the keys of its record, the bytes it counts per step, the
per-step distribution it reports beside the block-timed value, and the placement of
its pinned buffers and the host memory's bandwidth recorded beside the link rates."""
import argparse

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


def test_e2e_record():
    torch = gu.torch()
    wl = bench.sweep_workload(8 * 1_000_000 + 5, 8)
    rank = 3
    units, info, bufs = bench.build_local_rank(wl, rank, torch, fs, synth)
    args = argparse.Namespace(steps=4, e2e_steps=4, warmup=2)
    stream = torch.cuda.Stream()
    e = bench.e2e_local_rank(args, torch, fs, synth, wl, units, info, bufs, rank, stream, 1, None)
    S_tot = info["shard_elems"]
    assert e["unit"] == bench.UNIT and e["value"] > 0 and e["steps"] == 4
    assert e["h2d_bytes_per_step"] == 2 * 8 * S_tot and e["d2h_bytes_per_step"] == 2 * S_tot
    # value: the algorithmic bytes of one step over the block-timed step time
    assert abs(e["value"] - info["bytes_per_step"] / (e["ms_per_step"] * 1e-3) / 1e9) <= 0.01 * e["value"] + 0.05
    assert len(e["blocks_ms"]) == 3 and abs(min(e["blocks_ms"]) - e["ms_per_step"]) < 0.002
    p = e["per_step_ms"]
    assert 0 < p["min"] <= p["median"] <= p["max"]
    link = e["host_link"]
    assert link["h2d_GB_per_s"] > 0 and link["d2h_GB_per_s"] > 0
    assert abs(link["floor_ms"] - e["h2d_bytes_per_step"] / (link["h2d_GB_per_s"] * 1e9) * 1e3) < 0.02
    r_both = link["both_ways_GB_per_s_total"] / 2 * 1e9
    floor2 = (e["d2h_bytes_per_step"] / r_both
              + (e["h2d_bytes_per_step"] - e["d2h_bytes_per_step"]) / (link["h2d_GB_per_s"] * 1e9)) * 1e3
    assert abs(link["floor_two_way_ms"] - floor2) < 0.02
    # where the pinned buffers live, as the OS reports it: every page of the mappings
    # that hold them is on some NUMA node of this host, and the GPU's node is one of them
    place = link["placement"]
    assert place["numa_nodes"] and set(place["buffers"]) == {"grad_slices", "shard_out"}
    for name, b in place["buffers"].items():
        assert b["bytes"] > 0 and b["mapping_bytes"] >= b["bytes"], name
        pages = sum(b["mapping_pages_per_node"].values())
        assert pages * min(b["page_kB"]) * 1024 >= b["bytes"], name
        assert all(k[1:] in {n[4:] for n in place["numa_nodes"]} for k in b["mapping_pages_per_node"]), name
    if place["gpu_numa_node"] is not None and place["gpu_numa_node"] >= 0:
        assert "node%d" % place["gpu_numa_node"] in place["numa_nodes"]
    mem = link["host_memory"]
    assert mem["read_GB_per_s"] > 0 and mem["write_GB_per_s"] > 0 and mem["copy_GB_per_s"] > 0 and mem["threads"] >= 1
    assert fs.fsdp_device_status() == 0
