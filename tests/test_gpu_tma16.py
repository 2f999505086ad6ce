"""The TMA form for W = 16 against the oracle, on every element.

The library stages W = 16 single-replica steps through the TMA form (two
88 KB stages) when the gradient rows of some step segment of the launch do not
all lie a multiple of 2 KB apart. Here the 16 rows are views into one buffer,
an odd multiple of 1 KB apart. Cases: every rank stepped with aligned and with
ragged shards (and state views 16 bytes off 32-byte alignment, which the
consumers store as two float4 instead of one 32-byte store), one rank stepped with the other shards gathered and special
values (infinities, NaN, subnormals, signed zeros), each as a small unit beside
a zero filler unit whose rows bring the launch to the form, and the plan's
choice on both sides of the rule (tests/test_abi_host.py checks the rule on
the host alone, spans of many GiB included).
"""
import numpy as np
import pytest

import gpu_util as gu
from test_gpu_special_values import _same_or_both_nan, _same_or_both_nan_bf16, _special_inputs

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")

W = 16


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    yield
    torch.cuda.empty_cache()


def _rows(n, on_grain=False):
    """16 views of n bf16 elements in one buffer, 16-byte aligned, consecutive rows an odd
    multiple of 1 KB apart (off the 2 KB grain), or a multiple of 2 KB apart."""
    torch = gu.torch()
    stride = -(-n // 1024) * 1024 + (0 if on_grain else 512)  # elements: 2 bytes each
    buf = torch.empty(W * stride, dtype=torch.int16, device="cuda")
    views = [buf[k * stride:k * stride + n] for k in range(W)]
    assert all(v.numel() == n for v in views)
    assert ((views[1].data_ptr() - views[0].data_ptr()) % 2048 == 0) == on_grain
    return views


def _rows_from(grads):
    """The host rows copied into off-grain views."""
    torch = gu.torch()
    rows = _rows(grads[0].size)
    for view, g in zip(rows, grads):
        view.copy_(torch.from_numpy(g.view(np.int16)))
    return rows


def _filler(owned, local):
    """A zero-filled unit with off-grain rows whose chunks bring the launch to the TMA form's
    threshold (and to its W = 16 instantiation)."""
    torch = gu.torch()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    need = 130 * sms
    # local rank: 4 step chunks and 15 gather chunks of 16 KB per 8192 shard elements
    S = 8192 * -(-need // (4 + W - 1)) if local else 2048 * -(-need // W)
    lay, _ = fs.fsdp_flatten_layout([W * S], W)
    rows = _rows(W * S)
    for r in rows:
        r.zero_()
    z = lambda n, dt: torch.zeros(n, dtype=dt, device="cuda")  # noqa: E731
    return dict(layout=lay, grads=rows, master=[z(S, torch.float32) for _ in owned],
                exp_avg=[z(S, torch.float32) for _ in owned], exp_avg_sq=[z(S, torch.float32) for _ in owned],
                other_shards=[None if k in owned else z(S, torch.int16) for k in range(W)] if local else None,
                full_out=[z(W * S, torch.int16)])


def _shard_len(align8):
    torch = gu.torch()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S = -(-(130 * sms * 2048) // W)  # comfortably above 128 chunks per SM over the 16 positions
    return S - S % 8 + (0 if align8 else 3)


def _inputs(seed, P):
    rng = np.random.default_rng(seed)
    grads = [((rng.standard_normal(P, dtype=np.float32) * 1e-2).view(np.uint32) >> 16).astype(np.uint16)
             for _ in range(W)]
    master = rng.standard_normal(P, dtype=np.float32) * 0.02
    m = np.abs(rng.standard_normal(P, dtype=np.float32) * 1e-4)
    v = np.abs(rng.standard_normal(P, dtype=np.float32) * 1e-4)
    return grads, master, m, v


# state_off 4: the state views 16 bytes past 32-byte alignment (two float4 stores per array)
@pytest.mark.parametrize("align8,state_off", [(False, 0), (True, 0), (True, 4)])
def test_tma16_all_ranks_matches_oracle(ora, align8, state_off):
    torch = gu.torch()
    S = _shard_len(align8)
    P = W * S
    lay, _ = fs.fsdp_flatten_layout([P], W)
    assert lay.shard_numel == S
    grads, master, m, v = _inputs(160 + align8, P)
    sl = lambda a, r: a[r * S:(r + 1) * S]  # noqa: E731
    units = [dict(layout=lay, grads=_rows_from(grads),
                  master=[gu.to_dev_at(sl(master, r), state_off) for r in range(W)],
                  exp_avg=[gu.to_dev_at(sl(m, r), state_off) for r in range(W)],
                  exp_avg_sq=[gu.to_dev_at(sl(v, r), state_off) for r in range(W)],
                  other_shards=None, full_out=[torch.zeros(P, dtype=torch.int16, device="cuda")])]
    assert all(t.data_ptr() % 32 == 4 * state_off for t in units[0]["exp_avg_sq"])
    # S = 3 mod 8: fifteen of the sixteen positions' rows lie 2-14 bytes off
    # alignment, and the launch takes the LDG form's realigned path instead
    assert fs.fsdp_shard_step_grouped_plan(units, 0, W, interleaved=True) == (1, 1 if align8 else 0, 0)
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(4))
    torch.cuda.synchronize()
    assert fs.fsdp_device_status() == 0
    om, oe, ov = [sl(master, r).copy() for r in range(W)], [sl(m, r).copy() for r in range(W)], \
        [sl(v, r).copy() for r in range(W)]
    ofull = [np.zeros(P, np.uint16)]
    ora.shard_step(grads, W, 0, W, om, oe, ov, None, ofull, step=4, **gu.HP)
    u = units[0]
    for r in range(W):
        gu.assert_same_bits(gu.to_host(u["master"][r]), om[r], "master r%d" % r)
        gu.assert_same_bits(gu.to_host(u["exp_avg"][r]), oe[r], "exp_avg r%d" % r)
        gu.assert_same_bits(gu.to_host(u["exp_avg_sq"][r]), ov[r], "exp_avg_sq r%d" % r)
    gu.assert_same_bits(gu.to_host(u["full_out"][0]), ofull[0], "full")


def test_tma16_local_rank_matches_oracle(ora):
    """One rank stepped and the other 15 shards gathered (copy chunks through the same form),
    a ragged unit beside the filler."""
    torch = gu.torch()
    rank = 11
    P = W * 300_001 - 5
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S, padded = lay.shard_numel, lay.padded_numel
    grads, master, m, v = _inputs(170, padded)
    for a in (master, m, v):
        a[P:] = 0
    rng = np.random.default_rng(171)
    others = [((rng.standard_normal(S, dtype=np.float32) * 0.02).view(np.uint32) >> 16).astype(np.uint16)
              for _ in range(W)]
    sl = lambda a: a[rank * S:(rank + 1) * S]  # noqa: E731
    unit = dict(layout=lay, grads=[gu.to_dev(g) for g in grads], master=[gu.to_dev(sl(master))],
                exp_avg=[gu.to_dev(sl(m))], exp_avg_sq=[gu.to_dev(sl(v))],
                other_shards=[None if k == rank else gu.to_dev(others[k]) for k in range(W)],
                full_out=[torch.zeros(padded, dtype=torch.int16, device="cuda")])
    units = [unit, _filler([rank], True)]
    assert fs.fsdp_shard_step_grouped_plan(units, rank, rank + 1, interleaved=True) == (1, 1, 0)
    fs.fsdp_shard_step_grouped(units, rank, rank + 1, gu.adam_hyper(9))
    torch.cuda.synchronize()
    assert fs.fsdp_device_status() == 0
    om, oe, ov = [sl(master).copy()], [sl(m).copy()], [sl(v).copy()]
    ofull = [np.zeros(padded, np.uint16)]
    ora.shard_step(grads, W, rank, rank + 1, om, oe, ov, [None if k == rank else others[k] for k in range(W)],
                   ofull, step=9, **gu.HP)
    gu.assert_same_bits(gu.to_host(unit["master"][0]), om[0], "master")
    gu.assert_same_bits(gu.to_host(unit["exp_avg"][0]), oe[0], "exp_avg")
    gu.assert_same_bits(gu.to_host(unit["exp_avg_sq"][0]), ov[0], "exp_avg_sq")
    gu.assert_same_bits(gu.to_host(unit["full_out"][0]), ofull[0], "full (own slice and 15 gathered)")


@pytest.mark.parametrize("local", [False, True])
def test_tma16_special_values(ora, local):
    """Infinities, NaN, subnormal and signed-zero gradients and extreme masters through the
    W = 16 TMA form: every non-NaN output bit-identical, NaN exactly where the oracle has NaN."""
    torch = gu.torch()
    P = W * 8192 - 3  # shards of 8192 elements (16-byte aligned), a ragged last shard
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S, padded = lay.shard_numel, lay.padded_numel
    grads, master, m, v = _special_inputs(np.random.default_rng(180 + local), W, P, padded)
    rank = 6
    owned = [rank] if local else list(range(W))
    rng = np.random.default_rng(182)
    others = [((rng.standard_normal(S, dtype=np.float32) * 0.02).view(np.uint32) >> 16).astype(np.uint16)
              for _ in range(W)]
    sl = lambda a, r: a[r * S:(r + 1) * S]  # noqa: E731
    unit = dict(layout=lay, grads=[gu.to_dev(g) for g in grads],
                master=[gu.to_dev(sl(master, r)) for r in owned],
                exp_avg=[gu.to_dev(sl(m, r)) for r in owned],
                exp_avg_sq=[gu.to_dev(sl(v, r)) for r in owned],
                other_shards=[None if k in owned else gu.to_dev(others[k]) for k in range(W)] if local else None,
                full_out=[torch.zeros(padded, dtype=torch.int16, device="cuda")])
    units = [unit, _filler(owned, local)]
    assert fs.fsdp_shard_step_grouped_plan(units, owned[0], owned[-1] + 1, interleaved=True) == (1, 1, 0)
    fs.fsdp_shard_step_grouped(units, owned[0], owned[-1] + 1, gu.adam_hyper(3))
    torch.cuda.synchronize()
    om = [sl(master, r).copy() for r in owned]
    oe = [sl(m, r).copy() for r in owned]
    ov = [sl(v, r).copy() for r in owned]
    ofull = [np.zeros(padded, np.uint16)]
    ora.shard_step(grads, W, owned[0], owned[-1] + 1, om, oe, ov, others if local else None, ofull, step=3,
                   **gu.HP)
    nan_seen = 0
    for i, r in enumerate(owned):
        _same_or_both_nan(gu.to_host(unit["master"][i]), om[i], "master r%d" % r)
        _same_or_both_nan(gu.to_host(unit["exp_avg"][i]), oe[i], "exp_avg r%d" % r)
        _same_or_both_nan(gu.to_host(unit["exp_avg_sq"][i]), ov[i], "exp_avg_sq r%d" % r)
        nan_seen += int(np.isnan(om[i]).sum())
    got = gu.to_host(unit["full_out"][0])
    if local:  # the gathered shards are byte copies: every element, NaN or not
        for k in range(W):
            if k != rank:
                gu.assert_same_bits(got[k * S:(k + 1) * S], ofull[0][k * S:(k + 1) * S], "gathered k%d" % k)
        got, want = got[rank * S:(rank + 1) * S], ofull[0][rank * S:(rank + 1) * S]
    else:
        want = ofull[0]
    _same_or_both_nan_bf16(got, want, "full")
    assert nan_seen > 0


def test_tma16_rule_follows_row_alignment():
    """The same W = 16 unit runs on the LDG form when its rows lie a multiple of 2 KB apart,
    and on the TMA form when they do not (the plan, no launch)."""
    torch = gu.torch()
    S = _shard_len(True)
    P = W * S
    lay, _ = fs.fsdp_flatten_layout([P], W)
    state = [torch.empty(S, device="cuda") for _ in range(3 * W)]
    unit = dict(layout=lay, master=state[:W], exp_avg=state[W:2 * W], exp_avg_sq=state[2 * W:],
                other_shards=None, full_out=[torch.empty(P, dtype=torch.int16, device="cuda")])
    assert fs.fsdp_shard_step_grouped_plan([dict(unit, grads=_rows(P, on_grain=True))], 0, W) == (1, 0)
    assert fs.fsdp_shard_step_grouped_plan([dict(unit, grads=_rows(P))], 0, W) == (1, 1)
