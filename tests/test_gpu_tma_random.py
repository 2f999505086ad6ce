"""Random launches of the TMA form against the oracle, on every element.

Each case draws a set of units (thousands to millions of elements in multiples
of 8 W, then a few small units of odd sizes whose shards lie off 16-byte
alignment, which the TMA form leaves to its unstaged path), a mode (every rank stepped, or one
rank stepped with the other ranks' shards gathered), a step counter and Adam
hyper-parameters. Units are added until the launch holds enough chunks for the
library to choose the TMA form (checked with the plan). Inputs are filled on
the device by the seeded generator, and every output of every unit is compared
with the oracle's shard_step bit for bit (tests/full_parity.py). Two more
local-rank cases space the gradient rows widely enough for the library to pick
the interleaved-copy staging, and a 45-unit launch splits over a TMA-form and
an LDG-form descriptor table.
"""
import numpy as np
import pytest

import full_parity
import gpu_util as gu
import synth
from synth import workloads as wls

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")
bench = pytest.importorskip("bench")

W = 8


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _chunks(P, local):
    S = -(-P // W)
    return (-(-S // 2048) + (W - 1) * -(-2 * S // 16384)) if local else W * -(-S // 2048)


def _draw_units(rng, local, need_chunks):
    """Units for one launch: at most 18 of them (a launch's descriptor table holds 40 units
    of the local-rank step and 21 of the all-ranks step). Their sizes are multiples of 8 W
    (shards of whole 16-byte rows) up to a last one that brings the launch to
    `need_chunks`; then one to three small units of odd sizes, whose shards (and, in the
    local-rank mode, the state views after them) lie off alignment. Launches made mostly
    of such segments take the LDG form instead (tests/test_gpu_realigned.py)."""
    units, chunks = [], 0
    while chunks < need_chunks and len(units) < 14:
        kind = int(rng.integers(0, 3))
        P = int([rng.integers(6000, 2_000_000), rng.integers(2_000_000, 9_000_000),
                 W * 2048 * rng.integers(1, 300)][kind])
        P = -(-P // (8 * W)) * 8 * W
        units.append([(P,)])
        chunks += _chunks(P, local)
    if chunks < need_chunks:  # one more unit with the chunks still missing
        per_elem = 22 / 16384 / W if local else 1 / 2048
        P = -(-int((need_chunks - chunks) / per_elem * 1.05) // (8 * W)) * 8 * W
        units.append([(P,)])
    for _ in range(int(rng.integers(1, 4))):
        units.append([(int(rng.integers(1, 6000)) | 1,)])
    if local:
        # one more tiny unit, so that the odd units' shard lengths sum to a multiple of 8:
        # the other ranks' shards are rows of one (W, sum of S) buffer, which stay 16-byte
        # aligned for the aligned units (else every gather lies off alignment, and the
        # launch takes the LDG form)
        odd = sum(-(-u[0][0] // W) for u in units if u[0][0] % (8 * W))
        if odd % 8:
            units.append([(W * (8 - odd % 8) - 1,)])
    return units


@pytest.mark.parametrize("seed", range(6))
def test_random_tma_launch(ora, seed):
    _check_random_launch(ora, seed, seed % 2 == 0)


@pytest.mark.parametrize("seed", (6, 7))
def test_random_tma_launch_wide_rows(ora, seed):
    """Local-rank launches whose gradient rows sit 2^28 elements apart (a 3.5 GiB span
    over the eight rows): the library stages their step chunks in interleaved
    quarter-chunk copies, the form the 7B step runs."""
    _check_random_launch(ora, seed, True, row_numel=1 << 28)


def _every_unit(ora, wl, units, rb, re, step, hp, what):
    for u, unit in enumerate(units):
        lay = unit["layout"]
        regen = full_parity.state_regen(wl, u, lay.numel)(lay.shard_numel, lay.shard_factor)
        assert full_parity.check_unit_every_element(ora, unit, rb, re, step, regen, "%s unit %d" % (what, u),
                                                    hp=hp) == lay.shard_numel


def _check_random_launch(ora, seed, local, row_numel=0):
    torch = gu.torch()
    rng = np.random.default_rng(900 + seed)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wl = wls.Workload("tma_random_%d" % seed, 7, _draw_units(rng, local, 130 * sms), W, sigma_state=1e-4)
    hp = dict(lr=float(10 ** rng.uniform(-4, -2)), beta1=float(rng.uniform(0.8, 0.95)),
              beta2=float(rng.uniform(0.95, 0.9999)), eps=float(10 ** rng.uniform(-10, -6)))
    step = int(rng.integers(1, 5000))
    rank = int(rng.integers(0, W))
    if local:
        units, info, bufs = bench.build_local_rank(wl, rank, torch, fs, synth, row_numel)
        rb, re = rank, rank + 1
    else:
        units, info, bufs = bench.build_all_ranks(wl, W, torch, fs, synth)
        rb, re = 0, W
    launches, tma, interleaved = fs.fsdp_shard_step_grouped_plan(units, rb, re, interleaved=True)
    assert tma >= 1, (launches, tma)
    assert interleaved == (tma if row_numel >= (1 << 28) else 0), (launches, tma, interleaved)
    fs.fsdp_shard_step_grouped(units, rb, re, fs.AdamHyper(step=step, **hp))
    torch.cuda.synchronize()
    _every_unit(ora, wl, units, rb, re, step, hp, "seed %d" % seed)
    del units, bufs
    torch.cuda.empty_cache()


def test_grouped_launch_split_over_both_forms(ora):
    """45 local-rank units of 4 M elements: the grouped step needs two descriptor tables
    (320 segments fit one); the first (every unit's step, then 275 gathers) holds enough
    chunks for the TMA form, the second (the other 40 gathers) runs on the LDG form.
    Every element of every unit matches."""
    torch = gu.torch()
    rng = np.random.default_rng(990)
    sizes = [4_000_000 + 64 * int(rng.integers(0, 64)) for _ in range(45)]
    wl = wls.Workload("tma_split", 7, [[(P,)] for P in sizes], W, sigma_state=1e-4)
    rank, step = 5, 77
    units, info, bufs = bench.build_local_rank(wl, rank, torch, fs, synth)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    launches, tma = fs.fsdp_shard_step_grouped_plan(units, rank, rank + 1)
    assert launches == 2
    if sms <= 152:
        assert tma == 1
    fs.fsdp_shard_step_grouped(units, rank, rank + 1, gu.adam_hyper(step))
    torch.cuda.synchronize()
    _every_unit(ora, wl, units, rank, rank + 1, step, gu.HP, "split launch")
    del units, bufs
    torch.cuda.empty_cache()
