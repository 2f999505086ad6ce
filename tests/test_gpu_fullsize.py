"""Full-size workloads, in the launch configuration the benchmark times.

Inputs are filled on the device by the seeded generator. Every workload of the
benchmark's configurations is compared with the oracle on every element
(tests/full_parity.py runs the oracle on all host cores): the Llama block and
the GPT-2 units (TMA form), the Llama-7B local-rank headline (TMA form with
interleaved copies; all 33 units), the 1e9-element sweep at W = 2, 4, 8, 16 and
the hybrid workload at F = 16 and F = 4, whose every F also gives bit-identical
state and parameters in every replica group (so F = 1 matches too), and two
FlatParameters of more than 2^31 elements.
"""
import pytest

import full_parity
import gpu_util as gu
import synth
from synth import workloads as wls

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")
bench = pytest.importorskip("bench")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.empty_cache()


def every_element(ora, wl, units, rb, re, step, what, piece=1 << 20):
    """full_parity.check_unit_every_element on every unit of a launch."""
    for u, unit in enumerate(units):
        lay = unit["layout"]
        regen = full_parity.state_regen(wl, u, lay.numel)(lay.shard_numel, lay.shard_factor)
        done = full_parity.check_unit_every_element(ora, unit, rb, re, step, regen, "%s unit %d" % (what, u),
                                                    piece=piece)
        assert done == lay.shard_numel


def test_llama_block_all_ranks(ora):
    """Config 2 as the benchmark launches it (TMA form, one copy per array): every element."""
    torch = gu.torch()
    wl = wls.LLAMA_BLOCK
    units, info, keep = bench.build_all_ranks(wl, wl.world_size, torch, fs, synth)
    assert fs.fsdp_shard_step_grouped_plan(units, 0, 8, interleaved=True) == (1, 1, 0)
    fs.fsdp_shard_step_grouped(units, 0, wl.world_size, gu.adam_hyper(1))
    torch.cuda.synchronize()
    every_element(ora, wl, units, 0, 8, 1, "llama block")
    del units, keep


def test_gpt2_small_grouped(ora):
    """Config 3: 13 units in one launch of the TMA form; every element of every unit."""
    torch = gu.torch()
    wl = wls.GPT2_SMALL
    units, info, keep = bench.build_all_ranks(wl, wl.world_size, torch, fs, synth)
    assert info["params"] == 124439808
    assert fs.fsdp_shard_step_grouped_plan(units, 0, 8) == (1, 1)
    fs.fsdp_shard_step_grouped(units, 0, wl.world_size, gu.adam_hyper(1))
    torch.cuda.synchronize()
    every_element(ora, wl, units, 0, 8, 1, "gpt2")
    del units, keep


@pytest.mark.parametrize("W", [2, 4, 8, 16])
def test_sweep_1e9_every_element(ora, W):
    """One FlatParameter of 1e9 elements stepped for all W ranks in one launch, as the size
    sweep times it: the LDG form at W = 2 (split mapping) and 4, the TMA form with
    interleaved copies at W = 8 and the W = 16 TMA form at W = 16 (the gradient rows are
    2 GB apart). Every element of every
    rank's master, exp_avg, exp_avg_sq and of the full bf16 buffer equals the oracle's
    shard_step; the fp32 state of all ranks is one flat array whose 2 GiB boundaries the
    comparison crosses."""
    torch = gu.torch()
    n = 1_000_000_000
    wl = bench.sweep_workload(n, W)
    units, info, keep = bench.build_all_ranks(wl, W, torch, fs, synth)
    # the TMA form at W = 8 (interleaved copies: rows 3 GiB or more apart) and at W = 16 (rows
    # 2e9 bytes apart, not a multiple of 2 KB), the LDG form at W = 2 and 4
    tma, interleaved = (1 if W in (8, 16) else 0), (1 if W == 8 else 0)
    assert fs.fsdp_shard_step_grouped_plan(units, 0, W, interleaved=True) == (1, tma, interleaved)
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(2))
    torch.cuda.synchronize()
    assert fs.fsdp_device_status() == 0
    every_element(ora, wl, units, 0, W, 2, "sweep 1e9 W=%d" % W, piece=1 << 19)
    del units, keep
    torch.cuda.empty_cache()


def test_hybrid_full_size_identical_across_F(ora):
    """Config 4 (W = 16, one Llama block): F = 16 and F = 4 are compared with the oracle on
    every element of every replica; every F gives bit-identical master, exp_avg, exp_avg_sq
    and full buffers in every replica group, so F = 1 (16 replicas) equals the oracle too."""
    torch = gu.torch()
    wl = wls.HYBRID
    ref = None
    for F in (16, 4, 1):
        units, info, keep = bench.build_all_ranks(wl, F, torch, fs, synth)
        fs.fsdp_shard_step_grouped(units, 0, wl.world_size, gu.adam_hyper(1))
        torch.cuda.synchronize()
        grads, st, full = keep[0]
        R = wl.world_size // F
        if ref is None:
            ref = [x[0].clone() for x in st] + [full[0].clone()]
        if F in (16, 4):
            every_element(ora, wl, units, 0, 16, 1, "hybrid F=%d" % F)
        for g in range(R):
            for name, x, want in zip(("master", "exp_avg", "exp_avg_sq"), st, ref):
                assert torch.equal(x[g].view(torch.int32), want.view(torch.int32)), "%s F=%d g=%d" % (name, F, g)
            assert torch.equal(full[g], ref[3]), "full F=%d g=%d" % (F, g)
        del units, keep, grads, st, full
        torch.cuda.empty_cache()


@pytest.mark.parametrize("W,F,S", [(2, 1, (1 << 31) + 4112), (8, 8, (1 << 28) + 520)])
def test_flat_parameter_beyond_2_to_the_31_elements(ora, W, F, S):
    """One FlatParameter of more than 2^31 elements, every rank stepped in one launch.
    W = 2, F = 1 (the LDG form, two replicas): each shard is the whole padded buffer, so
    the kernel's element index itself passes 2^31. W = 8, F = 8 (the TMA form): the
    shards start beyond 2^31 elements of the gradient rows and the full buffer. Both
    have a ragged last chunk (S mod 2048 != 0) and padding at the end; every element of
    every replica is compared with the oracle."""
    torch = gu.torch()
    padded = F * S
    n = padded - (1 if W == 2 else 5)
    assert padded > (1 << 31) and S % 8 == 0 and S % 2048 != 0 and padded % W == 0
    wl = bench.sweep_workload(n, W)
    units, info, keep = bench.build_all_ranks(wl, F, torch, fs, synth)
    lay = units[0]["layout"]
    assert (lay.numel, lay.padded_numel, lay.shard_numel) == (n, padded, S)
    launches, tma = fs.fsdp_shard_step_grouped_plan(units, 0, W)
    assert (launches, tma) == (1, 1 if W == 8 else 0)
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(1))
    torch.cuda.synchronize()
    every_element(ora, wl, units, 0, W, 1, "beyond 2^31, W=%d F=%d" % (W, F))
    del units, keep
    torch.cuda.empty_cache()


def test_llama7b_local_rank_every_element(ora):
    """The benchmark's headline workload and launch: one grouped launch over 33 units, rank 0,
    on the TMA form with interleaved copies (every unit's step, then every gather). For every
    unit, the 32 blocks and the root unit, every element of the rank's master, exp_avg,
    exp_avg_sq, its own bf16 slice and the seven gathered slices equals the oracle's
    shard_step."""
    torch = gu.torch()
    wl = wls.LLAMA7B
    rank = 0
    units, info, bufs = bench.build_local_rank(wl, rank, torch, fs, synth)
    assert info["params"] == 6738415616 and info["shard_elems"] == 842301952
    assert fs.fsdp_shard_step_grouped_plan(units, rank, rank + 1, interleaved=True) == (1, 1, 1)
    fs.fsdp_shard_step_grouped(units, rank, rank + 1, gu.adam_hyper(1))
    torch.cuda.synchronize()
    assert fs.fsdp_device_status() == 0
    for u in range(len(units)):
        lay = units[u]["layout"]
        S = lay.shard_numel
        regen = full_parity.state_regen(wl, u, lay.numel)(S, lay.shard_factor)
        done = full_parity.check_unit_every_element(ora, units[u], rank, rank + 1, 1, regen,
                                                    "llama7b unit %d" % u)
        assert done == S
    del units, bufs
    torch.cuda.empty_cache()
