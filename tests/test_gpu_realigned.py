"""Steps whose rows and outputs, or state, lie off 16-byte alignment by a common
phase, against the oracle on every element.

When a shard length S is not a multiple of 8 elements, position p's slice of
every gradient row and of the gathered buffer starts 2pS bytes past a 16-byte
boundary (mod 16), and a rank's state views start 4pS bytes past one when they
are views of one buffer. The library gives such a step segment a width code
with the two phases, and the LDG form reads its rows as aligned 16-byte blocks
shifted into place and its state as aligned blocks shifted by whole words,
instead of falling back to one element per thread. Cases: all ranks at W = 2,
4, 8, 16 with the bench's buffers (rows of one (W, padded) buffer, state of one
(R, padded) buffer per quantity), hybrid groups, the local-rank mode over units
of odd sizes, special values with every state phase (0, 4, 8, 12 bytes), and
the one-launch reduce-scatter and grouped Adam on arrays at their own phases,
copies (pack, unpack, all-gather) whose sources and destinations start at
their own byte phases, and grouped launches (local-rank and all-ranks) split
into a TMA launch of their aligned segments and an LDG launch of the others.
"""
import numpy as np
import pytest

import full_parity
import gpu_util as gu
import synth
from synth import workloads as wls
from test_gpu_special_values import _same_or_both_nan, _same_or_both_nan_bf16, _special_inputs

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


def _every_element(ora, wl, units, rb, re, step, what):
    for u, unit in enumerate(units):
        lay = unit["layout"]
        regen = full_parity.state_regen(wl, u, lay.numel)(lay.shard_numel, lay.shard_factor)
        assert full_parity.check_unit_every_element(ora, unit, rb, re, step, regen, "%s unit %d" % (what, u)) \
            == lay.shard_numel


@pytest.mark.parametrize("W,F", [(2, 2), (4, 4), (8, 8), (16, 16), (16, 4), (8, 2)])
def test_odd_shards_all_ranks(ora, W, F):
    """One FlatParameter whose shards are an odd number of elements long, every rank stepped
    in one launch (the LDG form: the TMA form leaves launches made mostly of such segments)."""
    torch = gu.torch()
    # S odd; with groups (F < W) the padded length is a multiple of W, so S is a
    # multiple of W / F: 4 times an odd number here
    S = 300_001 if F == W else 4 * 75_001
    n = F * S - 1
    wl = bench.sweep_workload(n, W) if F == W else wls.Workload("odd_hybrid", 9, [[(n,)]], W, shard_factors=(F,),
                                                                    sigma_state=1e-4)
    units, info, keep = bench.build_all_ranks(wl, F, torch, fs, synth)
    lay = units[0]["layout"]
    assert lay.shard_numel == S and S % 8 != 0
    launches, tma = fs.fsdp_shard_step_grouped_plan(units, 0, W)
    assert (launches, tma) == (1, 0)
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(2))
    torch.cuda.synchronize()
    _every_element(ora, wl, units, 0, W, 2, "odd S, W=%d F=%d" % (W, F))
    del units, keep


@pytest.mark.parametrize("W", [2, 4])
def test_odd_shards_with_next_chunk_prefetch(ora, W):
    """At W = 2 and 4 the realigned step requests its block's next chunk into L2 before its
    loads; shards of about 1e6 elements give every block a next chunk in the same segment
    (the grid holds 3 blocks per SM), so the requests are issued. Every element."""
    torch = gu.torch()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S = 2048 * 3 * sms * 2 + 1  # two rounds of the grid per rank, odd
    n = W * S - 1
    wl = bench.sweep_workload(n, W)
    units, info, keep = bench.build_all_ranks(wl, W, torch, fs, synth)
    assert units[0]["layout"].shard_numel == S
    assert fs.fsdp_shard_step_grouped_plan(units, 0, W) == (1, 0)
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(6))
    torch.cuda.synchronize()
    _every_element(ora, wl, units, 0, W, 6, "odd S with prefetch, W=%d" % W)
    del units, keep


def test_odd_units_local_rank(ora):
    """The local-rank mode over units of odd sizes: each unit's rows, gathered slices and
    state views (one buffer per quantity) start at their own phases."""
    torch = gu.torch()
    W, rank = 8, 5
    sizes = [8 * 120_001 - 3, 8 * 200_003, 8 * 77_777 - 7, 8 * 300_000, 8 * 99_999 - 1]
    wl = wls.Workload("odd_local", 7, [[(P,)] for P in sizes], W, sigma_state=1e-4)
    units, info, bufs = bench.build_local_rank(wl, rank, torch, fs, synth)
    fs.fsdp_shard_step_grouped(units, rank, rank + 1, gu.adam_hyper(7))
    torch.cuda.synchronize()
    _every_element(ora, wl, units, rank, rank + 1, 7, "odd local")
    del units, bufs


@pytest.mark.parametrize("state_off", [0, 1, 2, 3])
def test_realigned_special_values(ora, state_off):
    """Special values (infinities, NaN, subnormals, signed zeros, extreme masters) through the
    realigned path, with every state phase: the state views start state_off elements (4 bytes
    each) into their buffers; S is odd, so most positions' rows lie off alignment too."""
    torch = gu.torch()
    W = 4
    S = 8193
    P = W * S - 2
    lay, _ = fs.fsdp_flatten_layout([P], W)
    padded = lay.padded_numel
    assert lay.shard_numel == S
    grads, master, m, v = _special_inputs(np.random.default_rng(700 + state_off), W, P, padded)
    sl = lambda a, r: a[r * S:(r + 1) * S].copy()  # noqa: E731
    rows = torch.zeros((W, padded), dtype=torch.int16, device="cuda")
    for k in range(W):
        rows[k] = gu.to_dev(grads[k])
    md = [gu.to_dev_at(sl(master, r), state_off) for r in range(W)]
    ed = [gu.to_dev_at(sl(m, r), state_off) for r in range(W)]
    vd = [gu.to_dev_at(sl(v, r), state_off) for r in range(W)]
    full = torch.zeros(padded, dtype=torch.int16, device="cuda")
    fs.fsdp_shard_step([rows[k] for k in range(W)], lay, 0, W, md, ed, vd, None, [full], gu.adam_hyper(3))
    torch.cuda.synchronize()
    om, oe, ov = [sl(master, r) for r in range(W)], [sl(m, r) for r in range(W)], [sl(v, r) for r in range(W)]
    ofull = [np.zeros(padded, np.uint16)]
    ora.shard_step(grads, W, 0, W, om, oe, ov, None, ofull, step=3, **gu.HP)
    for r in range(W):
        _same_or_both_nan(gu.to_host(md[r]), om[r], "master r%d" % r)
        _same_or_both_nan(gu.to_host(ed[r]), oe[r], "exp_avg r%d" % r)
        _same_or_both_nan(gu.to_host(vd[r]), ov[r], "exp_avg_sq r%d" % r)
    _same_or_both_nan_bf16(gu.to_host(full), ofull[0], "full")


@pytest.mark.parametrize("W", [4, 8, 16])
def test_realigned_reduce_scatter(ora, W):
    """Every rank's reduce-scatter in one launch with an odd S: each rank's slice of the rows
    and its fp32 output (views of one buffer, at r S elements) lie at their own phases."""
    torch = gu.torch()
    S = 70_001
    P = W * S - 1
    lay, _ = fs.fsdp_flatten_layout([P], W)
    padded = lay.padded_numel
    assert lay.shard_numel == S
    rng = np.random.default_rng(800 + W)
    grads = [((rng.standard_normal(padded, dtype=np.float32) * 1e-2).view(np.uint32) >> 16).astype(np.uint16)
             for _ in range(W)]
    for g in grads:
        g[P:] = 0
    rows = torch.zeros((W, padded), dtype=torch.int16, device="cuda")
    for k in range(W):
        rows[k] = gu.to_dev(grads[k])
    outs = torch.full((W * S,), float("nan"), device="cuda")
    fs.fsdp_reduce_scatter_ranks([rows[k] for k in range(W)], lay, 0, W, [outs[r * S:(r + 1) * S] for r in range(W)])
    torch.cuda.synchronize()
    got = gu.to_host(outs)
    for r in range(W):
        gu.assert_same_bits(got[r * S:(r + 1) * S], ora.reduce_scatter(grads, W, r), "reduce-scatter r%d" % r)


@pytest.mark.parametrize("offs", [(1, 2, 3, 1, 0), (0, 0, 0, 0, 1), (3, 1, 2, 2, 3)])
def test_realigned_adam_grouped(ora, offs):
    """Adam alone over shards whose gradient, state and bf16 output start at their own offsets
    (elements) into their buffers, with special values: every non-NaN output bit-identical."""
    torch = gu.torch()
    rng = np.random.default_rng(900 + sum(offs))
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-40, -1e-40, 3.3e38, -3.3e38, 1e-3],
                        dtype=np.float32)
    shards, want = [], []
    for n in (100_003, 65_536 + 5, 2_000_003):  # the last gives blocks a next chunk (prefetched)
        g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
        idx = rng.choice(n, size=n // 16, replace=False)
        g[idx] = rng.choice(specials, size=idx.size)
        p = (rng.standard_normal(n) * 0.02).astype(np.float32)
        m = np.abs(rng.standard_normal(n) * 1e-4).astype(np.float32)
        v = np.abs(rng.standard_normal(n) * 1e-4).astype(np.float32)
        v[rng.choice(n, size=n // 32, replace=False)] = 0.0
        op, om, ov = p.copy(), m.copy(), v.copy()
        obf = ora.adam(op, om, ov, g, step=4, **gu.HP)
        want.append((op, om, ov, obf))
        out_buf = torch.zeros(n + offs[4], dtype=torch.int16, device="cuda")
        shards.append(dict(master=gu.to_dev_at(p, offs[0]), exp_avg=gu.to_dev_at(m, offs[1]),
                           exp_avg_sq=gu.to_dev_at(v, offs[2]), grad_shard=gu.to_dev_at(g, offs[3]),
                           bf16_shard_out=out_buf[offs[4]:], n=n))
    fs.fsdp_adam_shard_step_grouped(shards, gu.adam_hyper(4))
    torch.cuda.synchronize()
    for i, (s, (op, om, ov, obf)) in enumerate(zip(shards, want)):
        _same_or_both_nan(gu.to_host(s["master"]), op, "master %d" % i)
        _same_or_both_nan(gu.to_host(s["exp_avg"]), om, "exp_avg %d" % i)
        _same_or_both_nan(gu.to_host(s["exp_avg_sq"]), ov, "exp_avg_sq %d" % i)
        _same_or_both_nan_bf16(gu.to_host(s["bf16_shard_out"]), obf, "bf16 %d" % i)


def _at(torch, h, off, dtype, pattern):
    """A device copy of `h` that starts `off` elements into a buffer filled with `pattern`
    (8 canary elements after it); returns (buffer, view)."""
    buf = torch.full((off + h.size + 8,), pattern, dtype=dtype, device="cuda")
    view = buf[off:off + h.size]
    if h.size:
        view.copy_(torch.from_numpy(np.ascontiguousarray(h).view(np.int16 if dtype == torch.int16 else np.float32)))
    return buf, view


def _canaries(buf, off, n, pattern):
    h = buf.cpu()
    return bool((h[:off] == pattern).all() and (h[off + n:] == pattern).all())


@pytest.mark.parametrize("seed", range(3))
def test_realigned_copies(ora, seed):
    """Pack, unpack and all-gather of bf16 tensors whose sources and destinations start at
    their own byte phases (element offsets 0..7 into their buffers): the copy segments go
    to the realigned copy path (aligned 16-byte stores, sources shifted into place, the
    bytes around them one at a time), the padding's zero fill too. Sizes from one element
    to several chunks; canaries around every destination catch stray writes."""
    torch = gu.torch()
    rng = np.random.default_rng(1000 + seed)
    numels = [1, 7, 15, 8191, 100_003, 3 * 8192 + 5, 0, 12_345, int(rng.integers(1, 40_000))]
    W = 8
    lay, offs = fs.fsdp_flatten_layout(numels, W)
    hs = [rng.integers(0, 1 << 16, size=n, dtype=np.uint16) for n in numels]
    src = [_at(torch, h, int(rng.integers(0, 8)), torch.int16, 5) for h in hs]
    fo = int(rng.integers(1, 8))
    fbuf, flat = _at(torch, np.zeros(lay.padded_numel, np.uint16), fo, torch.int16, 77)
    flat.fill_(77)
    fs.fsdp_pack_flat([v for _, v in src], lay, offs, flat)
    gu.assert_same_bits(gu.to_host(flat), ora.pack(hs, lay.padded_numel), "pack")
    assert _canaries(fbuf, fo, lay.padded_numel, 77), "write outside the flat buffer"
    outs = [_at(torch, np.zeros(n, np.uint16), int(rng.integers(0, 8)), torch.int16, 9) for n in numels]
    for _, v in outs:
        v.fill_(9)
    fs.fsdp_unpack_flat(flat, lay, offs, [v for _, v in outs])
    for (b, v), h in zip(outs, hs):
        gu.assert_same_bits(gu.to_host(v), h, "unpack of %d elements" % h.size)
        assert _canaries(b, b.numel() - 8 - h.size, h.size, 9), "write outside an unpacked tensor"
    # all-gather: odd shard length, each shard at its own offset, the full buffer at another
    S = 50_001 + 2 * int(rng.integers(0, 1000))
    glay, _ = fs.fsdp_flatten_layout([W * S], W)
    shards = [rng.integers(0, 1 << 16, size=S, dtype=np.uint16) for _ in range(W)]
    sd = [_at(torch, s, int(rng.integers(0, 8)), torch.int16, 3)[1] for s in shards]
    go = int(rng.integers(0, 8))
    gbuf, full = _at(torch, np.zeros(W * S, np.uint16), go, torch.int16, 11)
    full.fill_(11)
    fs.fsdp_all_gather(sd, glay, full)
    gu.assert_same_bits(gu.to_host(full), ora.all_gather(shards), "all-gather")
    assert _canaries(gbuf, go, W * S, 11), "write outside the full buffer"


def test_mixed_launch_split(ora):
    """A local-rank launch of four aligned units and two with odd shard lengths (their sum a
    multiple of 8, so that the other ranks' shards, rows of one (W, sum of S) buffer, stay
    aligned for the aligned units), large enough that the aligned segments alone make a
    TMA launch of at least 256 chunks per SM while the whole holds too many segments off
    alignment for it: the library splits it into a TMA launch of the aligned segments and
    an LDG launch of the others. Every element of every unit."""
    torch = gu.torch()
    W, rank = 8, 6
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S_al = 7_400_000 * max(1, -(-sms // 152))
    sizes = [8 * S_al] * 4 + [8 * 3_000_001 - 3, 8 * 2_000_007 - 5]
    wl = wls.Workload("mixed_local", 11, [[(P,)] for P in sizes], W, sigma_state=1e-4)
    units, info, bufs = bench.build_local_rank(wl, rank, torch, fs, synth)
    assert [u["layout"].shard_numel % 2 for u in units] == [0] * 4 + [1, 1]
    assert fs.fsdp_shard_step_grouped_plan(units, rank, rank + 1) == (2, 1)
    assert fs.fsdp_shard_step_grouped_plan(units[4:], rank, rank + 1) == (1, 0)
    fs.fsdp_device_status(clear=True)
    fs.fsdp_shard_step_grouped(units, rank, rank + 1, gu.adam_hyper(5))
    torch.cuda.synchronize()
    assert fs.fsdp_device_status() == 0
    _every_element(ora, wl, units, rank, rank + 1, 5, "mixed local")
    del units, bufs


def test_mixed_all_ranks_launch_split(ora):
    """The all-ranks step of three aligned units and one with an odd shard length (every
    rank's slice but rank 0's off alignment): split into a TMA launch of the aligned
    segments (rank 0's slice of the odd unit included) and an LDG launch of the others.
    Every element of every rank of every unit."""
    torch = gu.torch()
    W = 8
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S_al = 4_000_000 * max(1, -(-sms // 152))
    sizes = [8 * S_al] * 3 + [8 * 4_000_001 - 1]
    wl = wls.Workload("mixed_all_ranks", 13, [[(P,)] for P in sizes], W, sigma_state=1e-4)
    units, info, keep = bench.build_all_ranks(wl, W, torch, fs, synth)
    assert units[-1]["layout"].shard_numel % 2 == 1
    assert fs.fsdp_shard_step_grouped_plan(units, 0, W) == (2, 1)
    fs.fsdp_device_status(clear=True)
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(8))
    torch.cuda.synchronize()
    assert fs.fsdp_device_status() == 0
    _every_element(ora, wl, units, 0, W, 8, "mixed all ranks")
    del units, keep
