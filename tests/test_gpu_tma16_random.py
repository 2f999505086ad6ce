"""Random launches of the W = 16 TMA form against the oracle, on every element.

The W = 16 instantiation of the TMA form (two 88 KB stages, one bulk copy per
array) runs single-replica W = 16 launches whose gradient rows are not all a
multiple of 2 KB apart. Each case draws units of random sizes (multiples of
8 W, then one or two small units of odd sizes whose shards lie off alignment and
take the form's unstaged path), a mode (every rank stepped, or one rank stepped
with the other 15 shards gathered), a step counter and Adam hyper-parameters;
units are added until the launch holds enough chunks for the form. The rows are
laid out off the 2 KB grain: in the all-ranks mode the first unit's padded
length is an odd multiple of 128 (its rows, one per rank in a (16, padded)
buffer, are a multiple of 256 bytes apart but not of 2 KB), in the local-rank
mode the gradient pool's rows are an odd multiple of 1 KB apart.
Inputs are filled on the device by the seeded generator; every output of every
unit is compared with the oracle's shard_step bit for bit (tests/full_parity.py).
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

W = 16


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.empty_cache()


def _chunks(P, local):
    S = -(-P // W)
    return (-(-S // 2048) + (W - 1) * -(-2 * S // 16384)) if local else W * -(-S // 2048)


def _draw_units(rng, local, need_chunks):
    """Units for one launch. Sizes are multiples of 8 W (shards of whole 16-byte rows), the
    first one an odd multiple of 128 (its padded length is not a multiple of 1024: its
    rows, one per rank in a (16, padded) buffer, are off the 2 KB grain), the last of them
    sized so that the launch reaches `need_chunks`; then one or two small units of odd
    sizes (shards off alignment). A launch's descriptor table holds 20 units of the
    local-rank step and 6 of the all-ranks step (16 segments of 20 pointers each) at
    W = 16: at most 16 and 6 units are drawn."""
    k = int(rng.integers(100, 20_000)) | 1
    units, chunks = [[(128 * k,)]], _chunks(128 * k, local)
    while chunks < need_chunks and len(units) < (12 if local else 3):
        kind = int(rng.integers(0, 3))
        P = int([rng.integers(6000, 2_000_000), rng.integers(2_000_000, 9_000_000),
                 W * 2048 * rng.integers(1, 150)][kind])
        P = -(-P // (8 * W)) * 8 * W
        units.append([(P,)])
        chunks += _chunks(P, local)
    if chunks < need_chunks:  # one more unit with the chunks still missing
        per_elem = (1 / 2048 + (W - 1) * 2 / 16384) / W if local else 1 / 2048
        P = -(-int((need_chunks - chunks) / per_elem * 1.05) // (8 * W)) * 8 * W
        units.append([(P,)])
    for _ in range(int(rng.integers(1, 3))):
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


@pytest.mark.parametrize("seed", range(4))
def test_random_tma16_launch(ora, seed):
    torch = gu.torch()
    local = seed % 2 == 0
    rng = np.random.default_rng(1600 + seed)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    wl = wls.Workload("tma16_random_%d" % seed, 7, _draw_units(rng, local, 130 * sms), W, sigma_state=1e-4)
    hp = dict(lr=float(10 ** rng.uniform(-4, -2)), beta1=float(rng.uniform(0.8, 0.95)),
              beta2=float(rng.uniform(0.95, 0.9999)), eps=float(10 ** rng.uniform(-10, -6)))
    step = int(rng.integers(1, 5000))
    rank = int(rng.integers(0, W))
    if local:
        maxpad = max(fs.fsdp_flatten_layout(wls.numels(u), W)[0].padded_numel for u in wl.units)
        row = -(-maxpad // 1024) * 1024 + 512  # rows an odd multiple of 1 KB apart
        units, info, bufs = bench.build_local_rank(wl, rank, torch, fs, synth, row)
        rb, re = rank, rank + 1
    else:
        units, info, bufs = bench.build_all_ranks(wl, W, torch, fs, synth)
        rb, re = 0, W
    launches, tma, interleaved = fs.fsdp_shard_step_grouped_plan(units, rb, re, interleaved=True)
    assert tma >= 1 and interleaved == 0, (launches, tma, interleaved)
    fs.fsdp_device_status(clear=True)
    fs.fsdp_shard_step_grouped(units, rb, re, fs.AdamHyper(step=step, **hp))
    torch.cuda.synchronize()
    assert fs.fsdp_device_status() == 0
    for u, unit in enumerate(units):
        lay = unit["layout"]
        regen = full_parity.state_regen(wl, u, lay.numel)(lay.shard_numel, lay.shard_factor)
        assert full_parity.check_unit_every_element(ora, unit, rb, re, step, regen, "seed %d unit %d" % (seed, u),
                                                    hp=hp) == lay.shard_numel
    del units, bufs
    torch.cuda.empty_cache()
