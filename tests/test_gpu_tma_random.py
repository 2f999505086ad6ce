"""Random launches of the TMA form against the oracle, on sampled outputs.

Each case draws a set of units (from a few elements to millions; odd sizes put
the state views and gathered shards of later units off 16-byte alignment, which
the TMA form leaves to its unstaged path), a mode (every rank stepped, or one
rank stepped with the other ranks' shards gathered), a step counter and Adam
hyper-parameters. Units are added until the launch holds enough chunks for the
library to choose the TMA form (checked with the plan). Inputs are filled on
the device by the seeded generator; the host regenerates them at sampled
positions (the ends of every shard, chunk boundaries, random positions), the
oracle computes those outputs, and they must equal the device's bit for bit.
Two more local-rank cases space the gradient rows widely enough for the
library to pick the interleaved-copy staging; those are compared on every
element.
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


def _positions(n, rng, k=48):
    pts = set(range(min(n, 9))) | set(range(max(0, n - 9), n))
    for b in (2047, 2048, 2049):
        if b < n:
            pts.add(b)
    pts |= set(rng.integers(0, n, size=min(k, n)).tolist())
    return np.array(sorted(pts), dtype=np.int64)


def _gather(t, idx):
    torch = gu.torch()
    return gu.to_host(t[torch.from_numpy(idx).cuda()])


def _chunks(P, local):
    S = -(-P // W)
    return (-(-S // 2048) + (W - 1) * -(-2 * S // 16384)) if local else W * -(-S // 2048)


def _draw_units(rng, local, need_chunks):
    """Units for one launch: at most 18 of them (a launch's descriptor table holds 40 units
    of the local-rank step and 21 of the all-ranks step), the last one sized so the
    launch reaches `need_chunks`."""
    units, chunks = [], 0
    while chunks < need_chunks and len(units) < 17:
        kind = int(rng.integers(0, 4))
        P = int([rng.integers(1, 6000), rng.integers(6000, 2_000_000), rng.integers(2_000_000, 9_000_000),
                 W * 2048 * rng.integers(1, 300)][kind])
        units.append([(P,)])
        chunks += _chunks(P, local)
    if chunks < need_chunks:  # one more unit, of an odd size, with the chunks still missing
        per_elem = 22 / 16384 / W if local else 1 / 2048
        P = int((need_chunks - chunks) / per_elem * 1.05) | 1
        units.append([(P,)])
    return units


@pytest.mark.parametrize("seed", range(6))
def test_random_tma_launch(ora, seed):
    _check_random_launch(ora, seed, seed % 2 == 0)


@pytest.mark.parametrize("seed", (6, 7))
def test_random_tma_launch_wide_rows(ora, seed):
    """Local-rank launches whose gradient rows sit 2^28 elements apart (a 3.5 GiB span
    over the eight rows): the library stages their step chunks in interleaved
    quarter-chunk copies, the form the 7B step runs. Every element of every unit is
    compared with the oracle."""
    _check_random_launch(ora, seed, True, row_numel=1 << 28, every_element=True)


def _check_random_launch(ora, seed, local, row_numel=0, every_element=False):
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
    if every_element:
        for u, unit in enumerate(units):
            lay = unit["layout"]
            regen = full_parity.state_regen(wl, u, lay.numel)(lay.shard_numel, lay.shard_factor)
            assert full_parity.check_unit_every_element(
                ora, unit, rb, re, step, regen, "seed %d unit %d" % (seed, u), hp=hp) == lay.shard_numel
        del units, bufs
        torch.cuda.empty_cache()
        return

    def oracle(rows, master, m, v):
        g = ora.fold_mean(rows)
        p, mm, vv = master.copy(), m.copy(), v.copy()
        bf = ora.adam(p, mm, vv, g, step=step, **hp)
        return p, mm, vv, bf

    for u, unit in enumerate(units):
        lay = unit["layout"]
        S, P = lay.shard_numel, lay.numel
        owned = [rank] if local else list(range(W))
        for r in owned:
            j = _positions(S, rng)
            i = r * S + j
            if local:  # the builder's gradient pool: units alternate over two sets of rows, no pad zeroing
                rows = [synth.normal_bf16_at(wls.key_grad(wl, u % 2, k, 0), i, wl.sigma_grad) for k in range(W)]
            else:
                rows = [synth.normal_bf16_at(wls.key_grad(wl, u, k, 0), i, wl.sigma_grad, n_valid=P)
                        for k in range(W)]
            master = synth.normal_f32_at(wls.key_master(wl, u), i, wl.sigma_master, n_valid=P)
            m = synth.normal_f32_at(wls.key_exp_avg(wl, u), i, wl.sigma_state, absval=True, n_valid=P)
            v = synth.normal_f32_at(wls.key_exp_avg_sq(wl, u), i, wl.sigma_state, absval=True, n_valid=P)
            op, om, ov, obf = oracle(rows, master, m, v)
            o = 0 if local else r
            what = "seed %d unit %d rank %d" % (seed, u, r)
            gu.assert_same_bits(_gather(unit["master"][o], j), op, "master " + what)
            gu.assert_same_bits(_gather(unit["exp_avg"][o], j), om, "exp_avg " + what)
            gu.assert_same_bits(_gather(unit["exp_avg_sq"][o], j), ov, "exp_avg_sq " + what)
            gu.assert_same_bits(_gather(unit["full_out"][0], i), obf, "bf16 " + what)
        if local:  # the other ranks' slices of the full buffer are copies of their shards
            for k in (0, W - 1):
                if k == rank:
                    continue
                jk = _positions(S, rng, k=24)
                want = synth.normal_bf16_at(wls.key_shard(wl, u), k * S + jk, wl.sigma_master, n_valid=P)
                gu.assert_same_bits(_gather(unit["full_out"][0], k * S + jk), want, "gathered unit %d k %d" % (u, k))
    del units, bufs
    torch.cuda.empty_cache()


def test_grouped_launch_split_over_both_forms(ora):
    """45 local-rank units of 4 M elements: the grouped step needs two descriptor tables
    (40 units of 8 segments each fit one); the first holds enough chunks for the TMA form,
    the second (5 units) runs on the LDG form. Every unit's sampled outputs match."""
    torch = gu.torch()
    rng = np.random.default_rng(990)
    sizes = [4_000_000 + int(rng.integers(0, 64)) for _ in range(45)]  # odd sizes: mixed alignment
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
    for u in (0, 1, 39, 40, 44):  # both sides of the split
        unit = units[u]
        S, P = unit["layout"].shard_numel, unit["layout"].numel
        j = _positions(S, rng)
        i = rank * S + j
        rows = [synth.normal_bf16_at(wls.key_grad(wl, u % 2, k, 0), i, wl.sigma_grad) for k in range(W)]
        master = synth.normal_f32_at(wls.key_master(wl, u), i, wl.sigma_master, n_valid=P)
        m = synth.normal_f32_at(wls.key_exp_avg(wl, u), i, wl.sigma_state, absval=True, n_valid=P)
        v = synth.normal_f32_at(wls.key_exp_avg_sq(wl, u), i, wl.sigma_state, absval=True, n_valid=P)
        g = ora.fold_mean(rows)
        op, om, ov = master.copy(), m.copy(), v.copy()
        obf = ora.adam(op, om, ov, g, step=step, **gu.HP)
        gu.assert_same_bits(_gather(unit["master"][0], j), op, "master unit %d" % u)
        gu.assert_same_bits(_gather(unit["exp_avg"][0], j), om, "exp_avg unit %d" % u)
        gu.assert_same_bits(_gather(unit["exp_avg_sq"][0], j), ov, "exp_avg_sq unit %d" % u)
        gu.assert_same_bits(_gather(unit["full_out"][0], i), obf, "bf16 unit %d" % u)
        jk = _positions(S, rng, k=24)
        want = synth.normal_bf16_at(wls.key_shard(wl, u), 0 * S + jk, wl.sigma_master, n_valid=P)
        gu.assert_same_bits(_gather(unit["full_out"][0], jk), want, "gathered unit %d" % u)
    del units, bufs
    torch.cuda.empty_cache()
