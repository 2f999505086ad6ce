"""Special values through the fused step: +-inf, NaN, subnormal and signed-zero gradients,
huge and subnormal parameters. Non-NaN outputs must equal the oracle bit for bit; NaN must
appear exactly where the oracle has NaN (NaN payloads are not specified). The first cases
run on the LDG form (one small unit; W = 4 with the consecutive element mapping, and W = 2,
and W = 4 and 16 with replicas, with the split one), then Adam alone over two shards (split
mapping); the last put the same kind of unit at W = 8 into a grouped launch with a
zero-filled unit large enough for the library to choose the TMA form, all ranks and one rank
with its gather (tests/test_gpu_tma16.py does the same for the W = 16 TMA form)."""
import numpy as np
import pytest

import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _bf16(vals):
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _same_or_both_nan(got, want, what):
    g = np.asarray(got, np.float32)
    w = np.asarray(want, np.float32)
    gn, wn = np.isnan(g), np.isnan(w)
    assert np.array_equal(gn, wn), "%s: NaN positions differ" % what
    gu.assert_same_bits(g[~gn], w[~wn], what)


def _same_or_both_nan_bf16(got, want, what):
    f = lambda h: (np.asarray(h, np.uint32) << 16).view(np.float32)  # noqa: E731
    _same_or_both_nan(f(got), f(want), what)


@pytest.mark.parametrize("W,F", [(4, 4), (2, 2), (4, 1), (16, 2)])
def test_special_values_match_oracle(ora, W, F):
    """The LDG form with the consecutive element mapping (W = 4, F = 4) and with the split
    one (W = 2; W = 4 with four replicas per position; W = 16 with eight)."""
    torch = gu.torch()
    P = W * 4096
    lay, _ = fs.fsdp_flatten_layout([P], W, F)
    S, R = lay.shard_numel, W // F
    rng = np.random.default_rng(3 + W + F)
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-40, -1e-40, 3.3e38, -3.3e38, 1e-3],
                        dtype=np.float32)
    grads = []
    for k in range(W):
        x = (rng.standard_normal(P) * 1e-2).astype(np.float32)
        idx = rng.choice(P, size=P // 16, replace=False)
        x[idx] = rng.choice(specials, size=idx.size)
        grads.append(_bf16(x))
    master = synth.normal_f32(synth.stream_key(77, 1), P, 0.02)
    idx = rng.choice(P, size=P // 16, replace=False)
    master[idx] = rng.choice(np.array([0.0, -0.0, 1e-40, 3e38, -3e38, 1.0], np.float32), size=idx.size)
    m = np.abs(synth.normal_f32(synth.stream_key(77, 2), P, 1e-4))
    v = np.abs(synth.normal_f32(synth.stream_key(77, 3), P, 1e-4))
    v[rng.choice(P, size=P // 32, replace=False)] = 0.0
    sl = lambda a, r: a[(r % F) * S:(r % F + 1) * S].copy()  # noqa: E731
    om, oe, ov = [sl(master, r) for r in range(W)], [sl(m, r) for r in range(W)], [sl(v, r) for r in range(W)]
    ofull = [np.zeros(P, np.uint16) for _ in range(R)]
    ora.shard_step(grads, F, 0, W, om, oe, ov, None, ofull, step=2, **gu.HP)
    md = [gu.to_dev(sl(master, r)) for r in range(W)]
    ed = [gu.to_dev(sl(m, r)) for r in range(W)]
    vd = [gu.to_dev(sl(v, r)) for r in range(W)]
    full = [torch.zeros(P, dtype=torch.int16, device="cuda") for _ in range(R)]
    fs.fsdp_shard_step([gu.to_dev(g) for g in grads], lay, 0, W, md, ed, vd, None, full, gu.adam_hyper(2))
    torch.cuda.synchronize()
    nan_seen = 0
    for r in range(W):
        _same_or_both_nan(gu.to_host(md[r]), om[r], "master r%d" % r)
        _same_or_both_nan(gu.to_host(ed[r]), oe[r], "exp_avg r%d" % r)
        _same_or_both_nan(gu.to_host(vd[r]), ov[r], "exp_avg_sq r%d" % r)
        nan_seen += int(np.isnan(om[r]).sum())
    for g in range(R):
        _same_or_both_nan_bf16(gu.to_host(full[g]), ofull[g], "full g%d" % g)
    assert nan_seen > 0  # the case does reach the NaN paths


def test_special_values_grouped_adam(ora):
    """Adam alone (split element mapping) on special gradients and masters, two shards of one
    launch, one of them ragged."""
    torch = gu.torch()
    rng = np.random.default_rng(33)
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-40, -1e-40, 3.3e38, -3.3e38, 1e-3],
                        dtype=np.float32)
    shards, want = [], []
    for n in (8192, 5003):
        g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
        idx = rng.choice(n, size=n // 16, replace=False)
        g[idx] = rng.choice(specials, size=idx.size)
        p = (rng.standard_normal(n) * 0.02).astype(np.float32)
        idx = rng.choice(n, size=n // 16, replace=False)
        p[idx] = rng.choice(np.array([0.0, -0.0, 1e-40, 3e38, -3e38, 1.0], np.float32), size=idx.size)
        m = np.abs(rng.standard_normal(n) * 1e-4).astype(np.float32)
        v = np.abs(rng.standard_normal(n) * 1e-4).astype(np.float32)
        v[rng.choice(n, size=n // 32, replace=False)] = 0.0
        op, om, ov = p.copy(), m.copy(), v.copy()
        obf = ora.adam(op, om, ov, g, step=5, **gu.HP)
        want.append((op, om, ov, obf))
        shards.append(dict(master=gu.to_dev(p), exp_avg=gu.to_dev(m), exp_avg_sq=gu.to_dev(v),
                           grad_shard=gu.to_dev(g), bf16_shard_out=torch.zeros(n, dtype=torch.int16, device="cuda")))
    fs.fsdp_adam_shard_step_grouped(shards, gu.adam_hyper(5))
    torch.cuda.synchronize()
    nan_seen = 0
    for i, (s, (op, om, ov, obf)) in enumerate(zip(shards, want)):
        _same_or_both_nan(gu.to_host(s["master"]), op, "master %d" % i)
        _same_or_both_nan(gu.to_host(s["exp_avg"]), om, "exp_avg %d" % i)
        _same_or_both_nan(gu.to_host(s["exp_avg_sq"]), ov, "exp_avg_sq %d" % i)
        _same_or_both_nan_bf16(gu.to_host(s["bf16_shard_out"]), obf, "bf16 %d" % i)
        nan_seen += int(np.isnan(op).sum())
    assert nan_seen > 0


def _special_inputs(rng, W, P, padded):
    """Host inputs of one unit: W bf16 gradient rows and fp32 master/m/v over the padded
    FlatParameter (the pad stays zero), sprinkled with special values."""
    specials = np.array([np.inf, -np.inf, np.nan, 0.0, -0.0, 1e-40, -1e-40, 3.3e38, -3.3e38, 1e-3],
                        dtype=np.float32)
    grads = []
    for k in range(W):
        x = np.zeros(padded, np.float32)
        x[:P] = rng.standard_normal(P) * 1e-2
        idx = rng.choice(P, size=P // 16, replace=False)
        x[idx] = rng.choice(specials, size=idx.size)
        grads.append(_bf16(x))
    master = np.zeros(padded, np.float32)
    master[:P] = rng.standard_normal(P) * 0.02
    idx = rng.choice(P, size=P // 16, replace=False)
    master[idx] = rng.choice(np.array([0.0, -0.0, 1e-40, 3e38, -3e38, 1.0], np.float32), size=idx.size)
    m = np.zeros(padded, np.float32)
    v = np.zeros(padded, np.float32)
    m[:P] = np.abs(rng.standard_normal(P) * 1e-4)
    v[:P] = np.abs(rng.standard_normal(P) * 1e-4)
    v[rng.choice(P, size=P // 32, replace=False)] = 0.0
    return grads, master, m, v


def _filler_unit(torch, W, owned, chunks_needed, local):
    """A zero-filled unit whose chunks bring the launch to the TMA form's threshold."""
    if local:  # a step chunk of 2048 elements plus W - 1 gather chunks of 16 KB per 8192 elements
        S = 8192 * -(-chunks_needed // (4 + W - 1))
    else:
        S = 2048 * -(-chunks_needed // W)
    lay, _ = fs.fsdp_flatten_layout([W * S], W)
    z = lambda n, dt: torch.zeros(n, dtype=dt, device="cuda")  # noqa: E731
    return dict(layout=lay, grads=[z(W * S, torch.int16) for _ in range(W)],
                master=[z(S, torch.float32) for _ in owned], exp_avg=[z(S, torch.float32) for _ in owned],
                exp_avg_sq=[z(S, torch.float32) for _ in owned],
                other_shards=[None if k in owned else z(S, torch.int16) for k in range(W)] if local else None,
                full_out=[z(W * S, torch.int16)])


@pytest.mark.parametrize("local", [False, True])
def test_special_values_tma_form(ora, local):
    torch = gu.torch()
    W, P = 8, 8 * 8192 - 3  # shards of 8192 elements (16-byte aligned), a ragged last shard
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S, padded = lay.shard_numel, lay.padded_numel
    grads, master, m, v = _special_inputs(np.random.default_rng(40 + local), W, P, padded)
    rank = 5
    owned = [rank] if local else list(range(W))
    others = [gu.host_normal(synth.stream_key(78, 5), S, 0.02, idx0=k * S, bf16=True) for k in range(W)]
    om = [master[r * S:(r + 1) * S].copy() for r in owned]
    oe = [m[r * S:(r + 1) * S].copy() for r in owned]
    ov = [v[r * S:(r + 1) * S].copy() for r in owned]
    ofull = [np.zeros(padded, np.uint16)]
    ora.shard_step(grads, W, owned[0], owned[-1] + 1, om, oe, ov, others if local else None, ofull,
                   step=3, **gu.HP)
    unit = dict(layout=lay, grads=[gu.to_dev(g) for g in grads],
                master=[gu.to_dev(master[r * S:(r + 1) * S]) for r in owned],
                exp_avg=[gu.to_dev(m[r * S:(r + 1) * S]) for r in owned],
                exp_avg_sq=[gu.to_dev(v[r * S:(r + 1) * S]) for r in owned],
                other_shards=[None if k in owned else gu.to_dev(others[k]) for k in range(W)] if local else None,
                full_out=[torch.zeros(padded, dtype=torch.int16, device="cuda")])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    units = [unit, _filler_unit(torch, W, owned, 130 * sms, local)]
    launches, tma = fs.fsdp_shard_step_grouped_plan(units, owned[0], owned[-1] + 1)
    assert (launches, tma) == (1, 1), (launches, tma)
    fs.fsdp_shard_step_grouped(units, owned[0], owned[-1] + 1, gu.adam_hyper(3))
    torch.cuda.synchronize()
    nan_seen = 0
    for i, r in enumerate(owned):
        _same_or_both_nan(gu.to_host(unit["master"][i]), om[i], "master r%d" % r)
        _same_or_both_nan(gu.to_host(unit["exp_avg"][i]), oe[i], "exp_avg r%d" % r)
        _same_or_both_nan(gu.to_host(unit["exp_avg_sq"][i]), ov[i], "exp_avg_sq r%d" % r)
        nan_seen += int(np.isnan(om[i]).sum())
    got = gu.to_host(unit["full_out"][0])
    if local:  # the gathered shards are byte copies: compare every element, NaN or not
        for k in range(W):
            if k != rank:
                gu.assert_same_bits(got[k * S:(k + 1) * S], ofull[0][k * S:(k + 1) * S], "gathered k%d" % k)
        got, want = got[rank * S:(rank + 1) * S], ofull[0][rank * S:(rank + 1) * S]
    else:
        want = ofull[0]
    _same_or_both_nan_bf16(got, want, "full")
    assert nan_seen > 0


# Hyper-parameters at the edges the library accepts: lr = 0 (the master keeps its value
# except where the update is inf or NaN: 0 * inf), beta1 = beta2 = 0 (bias corrections of
# exactly 1: m = g, v = g^2), eps = 0 (0 / 0 where v and g are both 0), beta2 one step
# from 1 with t = 1 (a bias correction of about 1e-7), and a step count so large that
# both bias corrections round to 1.
HYPER_EDGES = [
    (dict(lr=0.0, beta1=0.9, beta2=0.999, eps=1e-8), 3),
    (dict(lr=1e-3, beta1=0.0, beta2=0.0, eps=1e-8), 1),
    (dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=0.0), 2),
    (dict(lr=1e-2, beta1=0.5, beta2=0.9999999, eps=1e-12), 1),
    (dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8), 10 ** 9),
]


@pytest.mark.parametrize("W", [4, 2])
@pytest.mark.parametrize("case", range(len(HYPER_EDGES)))
def test_hyper_parameter_edges(ora, W, case):
    """Every rank stepped, one small unit, on both element mappings of the LDG form (W = 4:
    consecutive, W = 2: split); gradients with zeros and special values, v with zeros."""
    torch = gu.torch()
    hp, step = HYPER_EDGES[case]
    P = W * 4096 - 1
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S, padded = lay.shard_numel, lay.padded_numel
    grads, master, m, v = _special_inputs(np.random.default_rng(500 + 7 * case + W), W, P, padded)
    for g in grads:  # zero gradients beside the zero v's: 0 / 0 when eps = 0
        g[: padded // 8] = 0
    v[: padded // 16] = 0.0
    sl = lambda a, r: a[r * S:(r + 1) * S].copy()  # noqa: E731
    om, oe, ov = [sl(master, r) for r in range(W)], [sl(m, r) for r in range(W)], [sl(v, r) for r in range(W)]
    ofull = [np.zeros(padded, np.uint16)]
    ora.shard_step(grads, W, 0, W, om, oe, ov, None, ofull, step=step, **hp)
    md = [gu.to_dev(sl(master, r)) for r in range(W)]
    ed = [gu.to_dev(sl(m, r)) for r in range(W)]
    vd = [gu.to_dev(sl(v, r)) for r in range(W)]
    full = [torch.zeros(padded, dtype=torch.int16, device="cuda")]
    fs.fsdp_shard_step([gu.to_dev(g) for g in grads], lay, 0, W, md, ed, vd, None, full,
                       fs.AdamHyper(step=step, **hp))
    torch.cuda.synchronize()
    for r in range(W):
        _same_or_both_nan(gu.to_host(md[r]), om[r], "master r%d" % r)
        _same_or_both_nan(gu.to_host(ed[r]), oe[r], "exp_avg r%d" % r)
        _same_or_both_nan(gu.to_host(vd[r]), ov[r], "exp_avg_sq r%d" % r)
    _same_or_both_nan_bf16(gu.to_host(full[0]), ofull[0], "full")
    if case == 0:  # lr = 0: every finite update leaves a nonzero master bit for bit as it was
        before = np.concatenate([sl(master, r) for r in range(W)])
        after = np.concatenate(om)
        fin = np.isfinite(after) & np.isfinite(before) & (before != 0)
        assert np.array_equal(after[fin].view(np.uint32), before[fin].view(np.uint32))
