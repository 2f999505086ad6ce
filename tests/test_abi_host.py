"""C ABI host logic without a GPU: exported symbols, layout, accountant, argument checks.

Every GPU entry point called here is given arguments that the host-side
validation rejects, so no kernel is ever launched (the pointers are fake).
"""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import fully_sharded_gb300 as fs
import oracle_pins as pins
from fully_sharded_gb300 import FsdpError

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(fsdp_\w+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_symbol():
    names = declared_functions()
    assert len(names) >= 10
    lib = ctypes.CDLL(fs.library_path())
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_layout_matches_oracle_brute(ora):
    rng = np.random.default_rng(0)
    for W in range(1, 17):
        for P in list(range(0, 40)) + [1000, 1000003]:
            numels = [P] if P < 3 else np.diff(
                np.concatenate([[0], np.sort(rng.integers(0, P + 1, size=3)), [P]])).tolist()
            for F in [f for f in range(1, W + 1) if W % f == 0]:
                lay, offs = fs.fsdp_flatten_layout(numels, W, F)
                o_offs, oP, opad, oS = ora.flatten_layout(numels, W, F)
                assert offs == o_offs.tolist()
                assert (lay.numel, lay.padded_numel, lay.shard_numel) == (oP, opad, oS)
                assert (lay.world_size, lay.shard_factor, lay.n_tensors) == (W, F, len(numels))


def test_layout_golden_workloads():
    for c in pins.golden("workload_layouts.json")["cases"]:
        lay, offs = fs.fsdp_flatten_layout(c["numels"], c["W"], c["F"])
        assert (lay.numel, lay.padded_numel, lay.shard_numel) == (c["P"], c["padded"], c["S"])
        if c["offsets"] is not None:
            assert offs == c["offsets"]


@pytest.mark.parametrize("args", [
    ([], 4, 4),          # no tensors
    ([5], 0, 1),         # W < 1
    ([5], 65, 65),       # W > 64
    ([5], 8, 3),         # F does not divide W
    ([5], 8, 0),         # F < 1
    ([5, -1], 4, 4),     # negative numel
    ([2**62, 2**62], 4, 4),  # overflow
])
def test_layout_rejects(args):
    with pytest.raises(FsdpError) as e:
        fs.fsdp_flatten_layout(*args)
    assert e.value.status == fs.FSDP_EINVAL


def test_account_matches_oracle(ora):
    for P in (0.0, 1.0, 7e9, 124439808.0, 6738415616.0):
        for N in (1, 2, 8, 16, 64):
            for F in [f for f in range(1, N + 1) if N % f == 0]:
                for pf in (0, 1, 2):
                    a = fs.fsdp_account(P, P / 32, N, F, pf)
                    b = ora.account(P, P / 32, N, F, pf)
                    for k in b:
                        assert a[k] == pytest.approx(b[k], rel=1e-13, abs=1e-6), (P, N, F, pf, k)


def test_account_worked_example():
    g = pins.golden("worked_example_7b.json")
    i, e = g["inputs"], g["expected"]
    a = fs.fsdp_account(i["P"], i["unit_params_printed"], i["N"], i["N"], i["prefetch"])
    assert a["persistent_bytes"] == e["persistent_bytes"]
    assert a["ddp_persistent_bytes"] == e["ddp_state_bytes"]
    assert round(a["transient_bytes"] / 1e9, 1) == e["transient_bytes_1dec_gb"]
    assert round(a["peak_bytes"] / 1e9) == e["peak_bytes_int_gb"]
    assert a["comm_bytes"] == e["fsdp_comm_bytes"] and a["ddp_comm_bytes"] == e["ddp_comm_bytes"]


def test_account_rejects():
    for args in ((1e9, 1e8, 0, 1), (1e9, 1e8, 8, 3), (-1.0, 1.0, 8, 8), (1e9, 1e8, 8, 0)):
        with pytest.raises(FsdpError):
            fs.fsdp_account(*args)


def test_status_strings():
    assert fs.fsdp_status_string(0) == "ok"
    for s in (fs.FSDP_EINVAL, fs.FSDP_EALIAS, fs.FSDP_ECUDA, fs.FSDP_ENOSPACE):
        assert fs.fsdp_status_string(s) not in ("ok", "unknown status")


def test_noalloc_capacity_agrees_across_header_binding_and_message():
    """The allocation-free entry point's capacity has one definition (the header's macro):
    the binding's constant and the FSDP_ENOSPACE text both follow it."""
    text = open(os.path.join(ROOT, "include", "fsdp.h")).read()
    m = re.search(r"#define\s+FSDP_NOALLOC_STAGING_BYTES\s+\((\d+)ll\s*<<\s*(\d+)\)", text)
    assert m, "FSDP_NOALLOC_STAGING_BYTES not found in the header"
    assert int(m.group(1)) << int(m.group(2)) == fs.NOALLOC_STAGING_BYTES
    assert "%d MiB" % (fs.NOALLOC_STAGING_BYTES >> 20) in fs.fsdp_status_string(fs.FSDP_ENOSPACE)


def test_diagnostic_call_is_declared_apart_from_the_method():
    """The bounded-wait self-test is exported but declared in the diagnostic header only."""
    def decls(name):
        t = re.sub(r"/\*.*?\*/", "", open(os.path.join(ROOT, "include", name)).read(), flags=re.S)
        return set(re.findall(r"\b(fsdp_\w+)\s*\(", t))
    assert "fsdp_selftest_wait_timeout" in decls("fsdp_test.h")
    assert "fsdp_selftest_wait_timeout" not in decls("fsdp.h")
    assert hasattr(ctypes.CDLL(fs.library_path()), "fsdp_selftest_wait_timeout")


# ---------------------------------------------- GPU entry points, rejected

BASE = 1 << 40  # fake device addresses; every call below fails validation first
HP = fs.AdamHyper()


def _lay(P, W, F=None):
    return fs.fsdp_flatten_layout([P], W, F)[0]


def _expect(status, fn, *a, **k):
    with pytest.raises(FsdpError) as e:
        fn(*a, stream=0, **k)
    assert e.value.status == status


def _addr(i, size=1 << 24):
    return BASE + i * size


def test_shard_step_rejects_bad_arguments():
    W = 4
    lay = _lay(1024, W)
    g = [_addr(k) for k in range(W)]
    st = lambda j: [_addr(10 + 3 * r + j) for r in range(W)]  # noqa: E731
    full = [_addr(40)]
    ok = dict(grads=g, layout=lay, rank_begin=0, rank_end=W, master=st(0), exp_avg=st(1),
              exp_avg_sq=st(2), other_shards=None, full_out=full)

    def call(status, **over):
        a = dict(ok)
        a.update(over)
        _expect(status, fs.fsdp_shard_step, a["grads"], a["layout"], a["rank_begin"],
                a["rank_end"], a["master"], a["exp_avg"], a["exp_avg_sq"], a["other_shards"],
                a["full_out"], over.get("adam", HP))

    call(fs.FSDP_EINVAL, rank_begin=2, rank_end=2)
    call(fs.FSDP_EINVAL, rank_begin=-1)
    call(fs.FSDP_EINVAL, rank_end=W + 1)
    call(fs.FSDP_EINVAL, grads=g[:3] + [None])
    call(fs.FSDP_EINVAL, master=st(0)[:3] + [None])
    call(fs.FSDP_EINVAL, full_out=[None])
    call(fs.FSDP_EINVAL, adam=fs.AdamHyper(step=0))
    call(fs.FSDP_EINVAL, adam=fs.AdamHyper(weight_decay=0.01))
    call(fs.FSDP_EINVAL, adam=fs.AdamHyper(beta1=1.0))
    call(fs.FSDP_EINVAL, adam=fs.AdamHyper(beta2=-0.1))
    call(fs.FSDP_EINVAL, adam=fs.AdamHyper(eps=-1.0))
    call(fs.FSDP_EINVAL, adam=fs.AdamHyper(lr=float("nan")))
    bad = fs.Layout(lay.numel, lay.padded_numel + W, lay.shard_numel, W, W, 1)
    call(fs.FSDP_EINVAL, layout=bad)
    bad = fs.Layout(lay.numel, lay.padded_numel, lay.shard_numel, W, 3, 1)
    call(fs.FSDP_EINVAL, layout=bad)
    # local-rank mode without the other shards
    call(fs.FSDP_EINVAL, rank_begin=1, rank_end=2, master=st(0)[:1], exp_avg=st(1)[:1],
         exp_avg_sq=st(2)[:1])
    # outputs overlapping inputs or each other
    call(fs.FSDP_EALIAS, master=[g[0]] + st(0)[1:])
    call(fs.FSDP_EALIAS, exp_avg=st(0))
    call(fs.FSDP_EALIAS, full_out=[g[3] + 2])
    call(fs.FSDP_EALIAS, master=st(0)[:3] + [st(0)[2] + 4])


def test_unfused_entry_points_reject_bad_arguments():
    W = 4
    lay = _lay(1000, W)
    g = [_addr(k) for k in range(W)]
    _expect(fs.FSDP_EINVAL, fs.fsdp_reduce_scatter, g, lay, W, _addr(20))
    _expect(fs.FSDP_EINVAL, fs.fsdp_reduce_scatter, g, lay, -1, _addr(20))
    _expect(fs.FSDP_EINVAL, fs.fsdp_reduce_scatter, g[:3] + [None], lay, 0, _addr(20))
    _expect(fs.FSDP_EALIAS, fs.fsdp_reduce_scatter, g, lay, 0, g[1] + 100)
    a = [_addr(30 + j) for j in range(5)]
    _expect(fs.FSDP_EINVAL, fs.fsdp_adam_shard_step, a[0], a[1], a[2], a[3], fs.AdamHyper(step=0), n=10)
    _expect(fs.FSDP_EINVAL, fs.fsdp_adam_shard_step, a[0], a[1], a[2], a[3], HP, n=-1)
    _expect(fs.FSDP_EINVAL, fs.fsdp_adam_shard_step, a[0], a[1], None, a[3], HP, n=10)
    _expect(fs.FSDP_EALIAS, fs.fsdp_adam_shard_step, a[0], a[0] + 8, a[2], a[3], HP, n=10)
    _expect(fs.FSDP_EALIAS, fs.fsdp_adam_shard_step, a[0], a[1], a[2], a[2] + 4, HP, n=10)
    _expect(fs.FSDP_EALIAS, fs.fsdp_adam_shard_step, a[0], a[1], a[2], a[3], HP,
            bf16_shard_out=a[0] + 16, n=10)
    sh = [_addr(50 + k) for k in range(W)]
    _expect(fs.FSDP_EINVAL, fs.fsdp_all_gather, sh[:3] + [None], lay, _addr(60))
    _expect(fs.FSDP_EALIAS, fs.fsdp_all_gather, sh[:3] + [_addr(60) + 2], lay, _addr(60))


def test_rank_range_and_grouped_parts_reject_bad_arguments():
    W = 4
    lay = _lay(1000, W)
    S = lay.shard_numel
    g = [_addr(k) for k in range(W)]
    outs = [_addr(20 + r) for r in range(W)]
    _expect(fs.FSDP_EINVAL, fs.fsdp_reduce_scatter_ranks, g, lay, 0, W + 1, outs + [_addr(25)])
    _expect(fs.FSDP_EINVAL, fs.fsdp_reduce_scatter_ranks, g, lay, 2, 2, outs)
    _expect(fs.FSDP_EINVAL, fs.fsdp_reduce_scatter_ranks, g, lay, -1, 2, outs)
    _expect(fs.FSDP_EINVAL, fs.fsdp_reduce_scatter_ranks, g, lay, 0, 2, [outs[0], None])
    _expect(fs.FSDP_EINVAL, fs.fsdp_reduce_scatter_ranks, g[:3] + [None], lay, 0, 2, outs[:2])
    _expect(fs.FSDP_EALIAS, fs.fsdp_reduce_scatter_ranks, g, lay, 0, 2, [outs[0], g[2] + 64])
    _expect(fs.FSDP_EALIAS, fs.fsdp_reduce_scatter_ranks, g, lay, 0, 2, [outs[0], outs[0] + 4 * (S - 1)])
    a = lambda i: _addr(30 + i)  # noqa: E731
    shard = lambda b, n=10, **k: dict(master=a(b), exp_avg=a(b + 1), exp_avg_sq=a(b + 2),  # noqa: E731
                                      grad_shard=a(b + 3), n=n, **k)
    grouped = fs.fsdp_adam_shard_step_grouped
    _expect(fs.FSDP_EINVAL, grouped, [shard(0)], fs.AdamHyper(step=0))
    _expect(fs.FSDP_EINVAL, grouped, [shard(0), shard(5, n=-1)], HP)
    _expect(fs.FSDP_EINVAL, grouped, [shard(0), dict(shard(5), exp_avg=None)], HP)
    _expect(fs.FSDP_EALIAS, grouped, [shard(0), dict(shard(5), master=a(0) + 36)], HP)  # state of shard 0
    _expect(fs.FSDP_EALIAS, grouped, [shard(0), dict(shard(5), grad_shard=a(2) + 8)], HP)
    _expect(fs.FSDP_EALIAS, grouped, [shard(0), shard(5, bf16_shard_out=a(1) + 2)], HP)
    # empty shards and no shards are no-ops, whatever their pointers
    grouped([dict(master=None, exp_avg=None, exp_avg_sq=None, grad_shard=None, n=0)], HP, stream=0)
    grouped([], HP, stream=0)


def _plan_with_rows(W, F, stride_bytes, S, base=BASE):
    """The plan of one all-ranks unit whose W gradient rows start stride_bytes apart (fake
    device addresses: the plan reads no memory)."""
    lay = fs.fsdp_flatten_layout([F * S], W, F)[0]
    assert lay.shard_numel == S
    padded = lay.padded_numel
    assert stride_bytes >= 2 * padded
    grads = [base + k * stride_bytes for k in range(W)]
    top = base + W * stride_bytes + (1 << 30)
    state = [top + i * S * 4 for i in range(3 * W)]
    full = [top + 3 * W * S * 4 + g * padded * 2 for g in range(W // F)]
    unit = dict(layout=lay, grads=grads, master=state[:W], exp_avg=state[W:2 * W], exp_avg_sq=state[2 * W:],
                other_shards=None, full_out=full)
    return fs.fsdp_shard_step_grouped_plan([unit], 0, W, interleaved=True)


def test_w16_tma_form_follows_row_alignment():
    """W = 16 single-replica launches large enough for the TMA form take it exactly when their
    gradient rows do not all lie a multiple of 2 KB apart, whatever the rows' span; W = 8
    launches take it either way, and replicated W = 16 launches never."""
    S = 152 * 130 * 2048 // 16 + 8  # above 128 chunks per SM on a 152-SM GPU
    row = 2 * 16 * S
    grain = -(-row // 2048) * 2048
    for stride, want in ((grain, (1, 0, 0)), (grain + 1024, (1, 1, 0)), (grain + 512, (1, 1, 0)),
                         (grain + 4096, (1, 0, 0)), (grain + (30 << 30) // 15 // 2048 * 2048, (1, 0, 0)),
                         (2_000_000_000, (1, 1, 0))):
        assert _plan_with_rows(16, 16, stride, S) == want, stride
    assert _plan_with_rows(8, 8, grain, 2 * S)[:2] == (1, 1)
    assert _plan_with_rows(8, 8, grain + 1024, 2 * S)[:2] == (1, 1)
    assert _plan_with_rows(16, 8, grain + 1024, S // 2 // 8 * 8) == (1, 0, 0)


def _local_units(sizes, rank, W=8, base=BASE):
    """Units of the local-rank step laid out as the bench lays them out (fake addresses): a
    pool of W gradient rows as long as the largest padded unit, state and the other ranks'
    shards as views of one buffer per quantity (rows of W x sum of S), one full buffer."""
    lays = [fs.fsdp_flatten_layout([P], W)[0] for P in sizes]
    S_tot, maxpad = sum(l.shard_numel for l in lays), max(l.padded_numel for l in lays)
    region = 1 << 36
    master, exp_avg, exp_avg_sq, others, full = (base + (i + 1) * region for i in range(5))
    units, so, po = [], 0, 0
    for lay in lays:
        units.append(dict(layout=lay, grads=[base + 2 * k * maxpad for k in range(W)],
                          master=[master + 4 * so], exp_avg=[exp_avg + 4 * so], exp_avg_sq=[exp_avg_sq + 4 * so],
                          other_shards=[None if k == rank else others + 2 * (k * S_tot + so) for k in range(W)],
                          full_out=[full + 2 * po]))
        so += lay.shard_numel
        po += lay.padded_numel
    return units


def test_mixed_launch_splits_off_the_segments_off_alignment():
    """A grouped local-rank launch whose segments off 16-byte alignment (odd shard lengths) are
    too many for the TMA form is split in two when its aligned segments alone make a TMA
    launch of at least 256 chunks per SM (152 SMs without a GPU); otherwise it stays one
    launch (few such segments: one TMA launch; too few aligned chunks: one LDG launch)."""
    big, odd = [8 * 7_400_000] * 4, [8 * 3_000_001 - 3, 8 * 2_000_007 - 5]
    assert fs.fsdp_shard_step_grouped_plan(_local_units(big + odd, 6), 6, 7) == (2, 1)
    assert fs.fsdp_shard_step_grouped_plan(_local_units(big, 6), 6, 7) == (1, 1)
    assert fs.fsdp_shard_step_grouped_plan(_local_units(odd, 6), 6, 7) == (1, 0)
    # a small odd unit among the aligned ones rides in the one TMA launch
    assert fs.fsdp_shard_step_grouped_plan(_local_units(big + [8 * 1001 - 1, 8 * 1007 - 3], 6), 6, 7) == (1, 1)
    # aligned segments of about 90 chunks per SM: one LDG launch (the second launch would cost more)
    small = [8 * 2_600_000] * 4
    assert fs.fsdp_shard_step_grouped_plan(_local_units(small, 6), 6, 7) == (1, 1)
    assert fs.fsdp_shard_step_grouped_plan(_local_units(small + odd, 6), 6, 7) == (1, 0)


def _all_ranks_units(sizes, W=8, base=BASE):
    """All-ranks units laid out as the bench lays them out (fake addresses): per unit a
    (W, padded) gradient buffer, one (W, S) buffer per state quantity, one full buffer."""
    units, addr = [], base
    for P in sizes:
        lay = fs.fsdp_flatten_layout([P], W)[0]
        S, padded = lay.shard_numel, lay.padded_numel
        grads = [addr + 2 * k * padded for k in range(W)]
        addr += -(-2 * W * padded // 4096) * 4096
        state = []
        for _ in range(3):
            state.append([addr + 4 * r * S for r in range(W)])
            addr += -(-4 * W * S // 4096) * 4096
        units.append(dict(layout=lay, grads=grads, master=state[0], exp_avg=state[1], exp_avg_sq=state[2],
                          other_shards=None, full_out=[addr]))
        addr += -(-2 * padded // 4096) * 4096
    return units


def test_mixed_all_ranks_launch_splits_too():
    """The same split for the all-ranks step: a unit with an odd shard length has every rank's
    slice but rank 0's off alignment; beside three large aligned units it sends the whole
    launch to the LDG form, so the aligned segments (rank 0's slice included) go first on
    the TMA form."""
    big, odd = [8 * 4_000_000] * 3, [8 * 4_000_001 - 1]
    assert fs.fsdp_shard_step_grouped_plan(_all_ranks_units(big + odd), 0, 8) == (2, 1)
    assert fs.fsdp_shard_step_grouped_plan(_all_ranks_units(big), 0, 8) == (1, 1)
    assert fs.fsdp_shard_step_grouped_plan(_all_ranks_units(odd), 0, 8) == (1, 0)
    assert fs.fsdp_shard_step_grouped_plan(_all_ranks_units(big[:1] + odd), 0, 8) == (1, 0)


def test_pack_unpack_reject_bad_arguments():
    lay, offs = fs.fsdp_flatten_layout([10, 20, 30], 4)
    ts = [_addr(k) for k in range(3)]
    lib = fs._lib

    def pack(tensors, offsets, flat_addr, dtype=fs.FSDP_DTYPE_F32):
        return lib.fsdp_pack_flat(fs._parray(tensors), ctypes.byref(lay), fs._offsets(offsets),
                                  dtype, flat_addr, None)

    def unpack(flat_addr, offsets, tensors, dtype=fs.FSDP_DTYPE_F32):
        return lib.fsdp_unpack_flat(flat_addr, ctypes.byref(lay), fs._offsets(offsets), dtype,
                                    fs._parray(tensors), None)

    assert pack(ts, offs, _addr(9), dtype=7) == fs.FSDP_EINVAL
    assert pack(ts, [1] + offs[1:], _addr(9)) == fs.FSDP_EINVAL
    assert pack(ts, offs[:-1] + [offs[-1] + 1], _addr(9)) == fs.FSDP_EINVAL
    assert pack(ts, [0, 20, 10, 60], _addr(9)) == fs.FSDP_EINVAL
    assert pack(ts[:2] + [None], offs, _addr(9)) == fs.FSDP_EINVAL
    assert pack(ts, offs, ts[1] + 8) == fs.FSDP_EALIAS
    assert unpack(_addr(9), offs, ts[:2] + [None]) == fs.FSDP_EINVAL
    assert unpack(_addr(9), offs, [ts[0], ts[0] + 4, ts[2]]) == fs.FSDP_EALIAS
    assert unpack(_addr(9), offs, [ts[0], _addr(9) + 4, ts[2]]) == fs.FSDP_EALIAS


def test_grouped_rejects_mixed_layouts():
    l4 = _lay(1024, 4)
    l8 = _lay(1024, 8)
    u = lambda lay, i: dict(layout=lay, grads=[_addr(i * 100 + k) for k in range(lay.world_size)],  # noqa: E731
                            master=[_addr(i * 100 + 20 + r) for r in range(lay.world_size)],
                            exp_avg=[_addr(i * 100 + 40 + r) for r in range(lay.world_size)],
                            exp_avg_sq=[_addr(i * 100 + 60 + r) for r in range(lay.world_size)],
                            other_shards=None, full_out=[_addr(i * 100 + 90)])
    _expect(fs.FSDP_EINVAL, fs.fsdp_shard_step_grouped, [u(l4, 0), u(l8, 1)], 0, 4, HP)
    a, b = u(l4, 0), u(l4, 1)
    b["full_out"] = [a["full_out"][0] + 64]  # two units writing the same full buffer
    _expect(fs.FSDP_EALIAS, fs.fsdp_shard_step_grouped, [a, b], 0, 4, HP)


def test_pipeline_rejects_bad_arguments():
    W, S = 4, 256
    lay = _lay(W * S, W)
    unit = dict(layout=lay, grad_slices=_addr(1), master=_addr(2), exp_avg=_addr(3), exp_avg_sq=_addr(4),
                other_shards=[_addr(5 + k) for k in range(W)], full_out=_addr(10), shard_out=None)

    def call(status, units=None, rank=0, staging=_addr(20), slot=W * S, n_slots=2, adam=HP):
        with pytest.raises(FsdpError) as e:
            fs.fsdp_pipeline_step([unit] if units is None else units, rank, staging, slot, n_slots, adam,
                                  compute=0, copy=0)
        assert e.value.status == status

    call(fs.FSDP_EINVAL, n_slots=0)
    call(fs.FSDP_EINVAL, n_slots=9)
    call(fs.FSDP_EINVAL, slot=W * S - 1)
    call(fs.FSDP_EINVAL, rank=W)
    hybrid = dict(unit, layout=_lay(W * S, W, 2))
    call(fs.FSDP_EINVAL, units=[hybrid])
    call(fs.FSDP_EINVAL, units=[dict(unit, master=None)])
    call(fs.FSDP_EINVAL, units=[dict(unit, other_shards=[_addr(5), None, _addr(7), _addr(8)])])
    call(fs.FSDP_EALIAS, staging=_addr(2))                       # pool overlaps the master shard
    call(fs.FSDP_EALIAS, units=[dict(unit, shard_out=_addr(10) + 64)])
    call(fs.FSDP_EALIAS, units=[unit, dict(unit, grad_slices=_addr(30))])  # two units, same outputs


def test_offload_rejects_bad_arguments():
    W, S = 4, 256
    lay = _lay(W * S, W)
    unit = dict(layout=lay, grads=[_addr(1 + k) for k in range(W)], master=_addr(10), exp_avg=_addr(11),
                exp_avg_sq=_addr(12), other_shards=[_addr(20 + k) for k in range(W)], full_out=_addr(30))

    def call(status, units=None, rank=0, staging=_addr(40), slot=S, n_slots=2, adam=HP):
        with pytest.raises(FsdpError) as e:
            fs.fsdp_offload_step([unit] if units is None else units, rank, staging, slot, n_slots, adam,
                                 compute=0, h2d=0, d2h=0)
        assert e.value.status == status

    call(fs.FSDP_EINVAL, n_slots=0)
    call(fs.FSDP_EINVAL, n_slots=9)
    call(fs.FSDP_EINVAL, slot=S - 1)
    call(fs.FSDP_EINVAL, rank=W)
    call(fs.FSDP_EINVAL, rank=-1)
    call(fs.FSDP_EINVAL, units=[dict(unit, layout=_lay(W * S, W, 2))])     # hybrid layout
    call(fs.FSDP_EINVAL, units=[dict(unit, master=None)])
    call(fs.FSDP_EINVAL, units=[dict(unit, grads=unit["grads"][:3] + [None])])
    call(fs.FSDP_EINVAL, units=[dict(unit, other_shards=[_addr(20), None, _addr(22), _addr(23)])])
    call(fs.FSDP_EINVAL, units=[unit, dict(unit, layout=_lay(8 * S, 8))])  # another W
    call(fs.FSDP_EALIAS, staging=_addr(10))                                # staging over the master shard
    call(fs.FSDP_EALIAS, units=[dict(unit, exp_avg=_addr(10) + 512)])      # m overlapping master
    call(fs.FSDP_EALIAS, units=[dict(unit, full_out=_addr(2) + 16)])       # full_out over a gradient row
    call(fs.FSDP_EALIAS, units=[unit, dict(unit, grads=[_addr(50 + k) for k in range(W)])])  # same outputs


def test_account_zero_matches_oracle_and_golden(ora):
    for P in (0.0, 1.0, 7e9, 124439808.0):
        for N in (1, 2, 8, 64):
            for stage in range(4):
                a, b = fs.fsdp_account_zero(P, N, stage), ora.account_zero(P, N, stage)
                for k in b:
                    assert a[k] == pytest.approx(b[k], rel=1e-13, abs=1e-9), (P, N, stage, k)
    g = pins.golden("zero_stages.json")
    for st, want in g["total_bytes"].items():
        assert fs.fsdp_account_zero(g["P"], g["N"], int(st))["total_bytes"] == want
    for args in ((1e9, 0, 1), (1e9, 8, 4), (1e9, 8, -1), (-1.0, 8, 1)):
        with pytest.raises(FsdpError):
            fs.fsdp_account_zero(*args)


def test_state_entry_points_reject_bad_arguments():
    W = 4
    lay = _lay(1024, W)
    lib = fs._lib
    sh = fs._parray([_addr(k) for k in range(W)])
    assert lib.fsdp_all_gather_state(sh, ctypes.byref(lay), 9, _addr(9), None) == fs.FSDP_EINVAL
    assert lib.fsdp_all_gather_state(sh, ctypes.byref(lay), fs.FSDP_DTYPE_F32, _addr(2) + 8, None) == fs.FSDP_EALIAS
    g = [_addr(k) for k in range(W)]
    oth = [_addr(20 + k) for k in range(W)]

    def z1(status, **over):
        a = dict(grads=g, layout=lay, rank=1, avg=_addr(10), master=_addr(11), m=_addr(12), v=_addr(13),
                 others=oth, full=_addr(14), adam=HP)
        a.update(over)
        _expect(status, fs.fsdp_zero1_step, a["grads"], a["layout"], a["rank"], a["avg"], a["master"], a["m"],
                a["v"], a["others"], a["full"], a["adam"])

    z1(fs.FSDP_EINVAL, layout=_lay(1024, W, 2))
    z1(fs.FSDP_EINVAL, rank=4)
    z1(fs.FSDP_EINVAL, avg=None)
    z1(fs.FSDP_EINVAL, others=[oth[0], oth[1], None, oth[3]])
    z1(fs.FSDP_EINVAL, adam=fs.AdamHyper(step=0))
    z1(fs.FSDP_EALIAS, avg=_addr(11))
    z1(fs.FSDP_EALIAS, full=g[2] + 2)


def test_import_fails_loudly_without_the_cuda_library(tmp_path):
    """No fallback: with the library missing, importing the package raises."""
    import subprocess
    import sys
    env = dict(os.environ, FSDP_GB300_LIB=str(tmp_path / "missing.so"))
    r = subprocess.run([sys.executable, "-c", "import fully_sharded_gb300"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "ImportError" in r.stderr
