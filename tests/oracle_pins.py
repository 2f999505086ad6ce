"""Pins of the CPU oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` takes a loaded oracle and raises AssertionError on a mismatch.
The values checked never come from the oracle's own formulas: they are the
pages' worked example, hand-derived IEEE results, exact rational arithmetic,
brute force over tiny cases, and library routines (torch.optim.Adam, torch's
bf16 conversion) on cases the method reduces to. tests/test_oracle_pins.py
runs them on the oracle; tests/test_oracle_mutants.py runs them on copies of
the oracle with one planted mistake each and expects at least one to fail.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

ADAM = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def f32_bits_to_bf16_exact(x) -> np.ndarray:
    """bf16 bits of fp32 values that are exactly representable in bf16."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(h) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint32) << 16).view(np.float32)


# ----------------------------------------------------------------- a1 layout

def pin_layout_brute(ora, seed=0):
    """All W in 1..16, P in 1..64, every F | W: the definition of an even split."""
    rng = np.random.default_rng(seed)
    for W in range(1, 17):
        for P in range(1, 65):
            cuts = np.sort(rng.integers(0, P + 1, size=rng.integers(0, 4)))
            numels = np.diff(np.concatenate([[0], cuts, [P]])).tolist()
            for F in [f for f in range(1, W + 1) if W % f == 0]:
                offs, P_, padded, S = ora.flatten_layout(numels, W, F)
                assert P_ == P
                # tensors occupy consecutive disjoint ranges in the listed order
                owner = np.full(P, -1)
                for i, n in enumerate(numels):
                    assert offs[i + 1] - offs[i] == n
                    assert np.all(owner[offs[i]:offs[i] + n] == -1)
                    owner[offs[i]:offs[i] + n] = i
                assert np.all(owner >= 0) and np.all(np.diff(owner) >= 0)
                # smallest multiple of W that holds P
                assert padded % W == 0 and P <= padded < P + W
                # F equal contiguous slices partition [0, padded)
                assert S * F == padded
                cover = np.zeros(padded, dtype=int)
                for p in range(F):
                    cover[p * S:(p + 1) * S] += 1
                assert np.all(cover == 1)


def pin_layout_golden(ora):
    g = golden("workload_layouts.json")
    for c in g["cases"]:
        offs, P, padded, S = ora.flatten_layout(c["numels"], c["W"], c["F"])
        assert (P, padded, S) == (c["P"], c["padded"], c["S"]), c["name"]
        if c["offsets"] is not None:
            assert offs.tolist() == c["offsets"], c["name"]


def pin_pack_roundtrip(ora, seed=1):
    """unflatten(flatten(x)) == x bit-exactly; pad is zero; gather(scatter) == flat."""
    rng = np.random.default_rng(seed)
    for W in (1, 2, 3, 4, 5, 8, 16):
        shapes = [(int(rng.integers(1, 9)), int(rng.integers(1, 9))) for _ in range(int(rng.integers(1, 5)))]
        for dt in (np.float32, np.uint16):
            ts = [rng.integers(0, 2**16, size=s).astype(dt) if dt is np.uint16
                  else rng.standard_normal(s).astype(np.float32) for s in shapes]
            numels = [int(np.prod(s)) for s in shapes]
            offs, P, padded, S = ora.flatten_layout(numels, W, W)
            flat = ora.pack(ts, padded)
            assert flat.size == padded
            assert not np.any(flat[P:].view(np.uint8 if dt is np.float32 else np.uint16))
            for t, o, n in zip(ts, offs[:-1], numels):
                assert flat[o:o + n].tobytes() == t.reshape(-1).tobytes()
            back = ora.unpack(flat, shapes)
            for a, b in zip(ts, back):
                assert a.tobytes() == b.tobytes()
            if dt is np.uint16:
                for F in [f for f in range(1, W + 1) if W % f == 0]:
                    s = padded // F
                    shards = [flat[p * s:(p + 1) * s].copy() for p in range(F)]
                    assert ora.all_gather(shards).tobytes() == flat.tobytes()


# ------------------------------------------------------- a3 reduce-scatter

def pin_rs_identical_rows(ora, seed=2):
    """W identical bf16 rows g: k*g needs <= 13 significand bits, so the sum is exact and the mean is g."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal(257) * 1e-2).astype(np.float32)
    g = ora_independent_bf16(x)
    for W in range(1, 17):
        out = ora.fold_mean([g] * W)
        assert out.tobytes() == bf16_bits_to_f32(g).tobytes(), W


def ora_independent_bf16(x):
    """bf16 bits by truncation toward zero: any bf16 value works as a test input."""
    return (np.asarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def pin_rs_marker_slices(ora):
    """g_k[i] = (i mod 16) + 16k: each rank must keep exactly slice p = r mod F of the mean."""
    for W in (1, 2, 4, 8, 16):
        P = 16 * W + 3
        padded = -(-P // W) * W
        i = np.arange(padded)
        grads = [f32_bits_to_bf16_exact(((i % 16) + 16 * k).astype(np.float32)) for k in range(W)]
        for F in [f for f in range(1, W + 1) if W % f == 0]:
            S = padded // F
            for r in range(W):
                p = r % F
                out = ora.reduce_scatter(grads, F, r)
                want = ((np.arange(p * S, (p + 1) * S) % 16) + 8 * (W - 1)).astype(np.float32)
                assert out.tobytes() == want.tobytes(), (W, F, r)


def _nearest_f32_ok(r: np.float32, q: Fraction) -> bool:
    """r is a nearest binary32 value to the rational q."""
    r = np.float32(r)
    d = abs(Fraction(float(r)) - q)
    for nb in (np.nextafter(r, np.float32(np.inf)), np.nextafter(r, np.float32(-np.inf))):
        if abs(Fraction(float(nb)) - q) < d:
            return False
    return True


def pin_rs_exact_rational(ora, seed=3):
    """Small-integer * 2^-e gradients: the fp32 fold is exact, the mean is the correctly rounded quotient."""
    rng = np.random.default_rng(seed)
    for W in range(1, 17):
        n = 64
        ints = rng.integers(-128, 128, size=(W, n))
        e = int(rng.integers(0, 20))
        rows = [f32_bits_to_bf16_exact((ints[k] * 2.0 ** -e).astype(np.float32)) for k in range(W)]
        out = ora.fold_mean(rows)
        for j in range(n):
            q = Fraction(int(ints[:, j].sum()), 2 ** e) / W
            assert _nearest_f32_ok(out[j], q), (W, j)


def pin_rs_fold_order(ora):
    """Hand-derived IEEE cases where the rank order of the fp32 fold changes the sum."""
    for c in golden("fold_order.json")["cases"]:
        rows = [f32_bits_to_bf16_exact(np.array([v], dtype=np.float32)) for v in c["rows_f32"]]
        W = len(rows)
        out = ora.fold_mean(rows)[0]
        q = Fraction(c["left_fold_sum"]) / W
        assert _nearest_f32_ok(out, q), c


def pin_rs_ddp_endpoint(ora, seed=4):
    """F = W slice r equals slice r of the F = 1 (DDP all-reduce average) result."""
    rng = np.random.default_rng(seed)
    for W in (2, 3, 4, 8):
        padded = W * 37
        grads = [ora_independent_bf16(rng.standard_normal(padded).astype(np.float32) * 1e-2)
                 for _ in range(W)]
        full = ora.reduce_scatter(grads, 1, 0)
        assert full.size == padded
        S = padded // W
        for r in range(W):
            assert ora.reduce_scatter(grads, W, r).tobytes() == full[r * S:(r + 1) * S].tobytes()


# ---------------------------------------------------------------- a4 Adam

def _torch_adam_steps(p0, m0, v0, grads, t0, hp):
    """Reference from torch.optim.Adam (CPU, fp32, single-tensor path)."""
    import torch
    p = torch.nn.Parameter(torch.from_numpy(p0.copy()))
    opt = torch.optim.Adam([p], lr=hp["lr"], betas=(hp["beta1"], hp["beta2"]), eps=hp["eps"],
                           weight_decay=0.0, foreach=False, fused=False)
    p.grad = torch.zeros_like(p)
    opt.step()  # creates the state; overwritten below
    with torch.no_grad():
        p.copy_(torch.from_numpy(p0))
    st = opt.state[p]
    st["exp_avg"].copy_(torch.from_numpy(m0))
    st["exp_avg_sq"].copy_(torch.from_numpy(v0))
    st["step"].fill_(float(t0 - 1))
    for g in grads:
        p.grad = torch.from_numpy(g.copy())
        opt.step()
    return (p.detach().numpy().copy(), st["exp_avg"].numpy().copy(), st["exp_avg_sq"].numpy().copy())


def _close(a, b, rel=1e-6):
    floor = rel * float(np.max(np.abs(b))) if b.size else 0.0
    return bool(np.all(np.abs(a.astype(np.float64) - b.astype(np.float64))
                       <= rel * np.abs(b.astype(np.float64)) + floor))


def pin_adam_torch(ora, seed=5):
    """Three steps against torch.optim.Adam, zero and non-zero initial state, several grad scales."""
    rng = np.random.default_rng(seed)
    n = 4096
    for gscale, t0, nonzero in ((1e-2, 1, False), (1e-3, 1, True), (1e-5, 1, False),
                                (1e-3, 7, True), (1e-6, 3, True)):
        p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
        m0 = (np.abs(rng.standard_normal(n)) * 1e-4).astype(np.float32) if nonzero else np.zeros(n, np.float32)
        v0 = (np.abs(rng.standard_normal(n)) * 1e-4).astype(np.float32) if nonzero else np.zeros(n, np.float32)
        grads = [(rng.standard_normal(n) * gscale).astype(np.float32) for _ in range(3)]
        tp, tm, tv = _torch_adam_steps(p0, m0, v0, grads, t0, ADAM)
        p, m, v = p0.copy(), m0.copy(), v0.copy()
        for k, g in enumerate(grads):
            ora.adam(p, m, v, g, step=t0 + k, **ADAM)
        assert _close(p, tp) and _close(m, tm) and _close(v, tv), (gscale, t0, nonzero)


def pin_adam_torch_hyper(ora, seed=12):
    """Against torch.optim.Adam at large step counters (bias corrections near 1, where a
    wrong power of beta still shows) and with other hyper-parameters."""
    rng = np.random.default_rng(seed)
    n = 4096
    other = dict(lr=1e-2, beta1=0.8, beta2=0.95, eps=1e-6)
    for hp, t0 in ((ADAM, 1000), (ADAM, 1_000_000), (other, 1), (other, 50), (other, 20_000)):
        p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
        m0 = (rng.standard_normal(n) * 1e-4).astype(np.float32)
        v0 = (np.abs(rng.standard_normal(n)) * 1e-4).astype(np.float32)
        grads = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(3)]
        tp, tm, tv = _torch_adam_steps(p0, m0, v0, grads, t0, hp)
        p, m, v = p0.copy(), m0.copy(), v0.copy()
        for k, g in enumerate(grads):
            ora.adam(p, m, v, g, step=t0 + k, **hp)
        assert _close(p, tp) and _close(m, tm) and _close(v, tv), (hp, t0)


def pin_adam_first_step(ora, seed=6):
    """From m = v = 0 at t = 1: mhat = g and vhat = g^2, so p' = p - lr g / (|g| + eps)."""
    rng = np.random.default_rng(seed)
    n = 4096
    p = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    want = p.astype(np.float64) - ADAM["lr"] * g.astype(np.float64) / (
        np.abs(g.astype(np.float64)) + ADAM["eps"])
    out = p.copy()
    ora.adam(out, m, v, g, step=1, **ADAM)
    # error budget: the update lr*q with q = mhat/(sqrt(vhat)+eps) ~ 1 carries a few
    # fp32 roundings (relative 2^-23 each, so ~8 * 2^-23 * lr absolute), plus one
    # rounding of the final subtraction (1 ulp of the result).
    ulp = np.spacing(np.abs(want).astype(np.float32)).astype(np.float64)
    assert np.all(np.abs(out - want) <= ulp + 8 * 2.0 ** -23 * ADAM["lr"])
    assert np.all(np.sign(p - out) == np.sign(g))


def pin_adam_zero_grad(ora):
    """g = 0 from m = v = 0 leaves every parameter bit pattern unchanged (any t)."""
    x = np.array([0.0, -0.0, 1.0, -3.5e-3, 1e-30, 3e38, -np.inf, np.inf], dtype=np.float32)
    for t in (1, 2, 1000):
        p = x.copy()
        m = np.zeros_like(x)
        v = np.zeros_like(x)
        bf = ora.adam(p, m, v, np.zeros_like(x), step=t, **ADAM)
        assert p.tobytes() == x.tobytes() and not np.any(m) and not np.any(v)
        assert bf.tobytes() == f32_to_bf16_torch(x).tobytes()


# ------------------------------------------------------------------ a5 cast

def cast_patterns(seed=7, n_random=1 << 20):
    hi = np.arange(1 << 16, dtype=np.uint32) << 16
    lows = np.array([0, 1, 0x3FFF, 0x7FFF, 0x8000, 0x8001, 0xBFFF, 0xFFFF], dtype=np.uint32)
    structured = (hi[:, None] | lows[None, :]).reshape(-1)
    rnd = np.random.default_rng(seed).integers(0, 1 << 32, size=n_random, dtype=np.uint64).astype(np.uint32)
    return np.concatenate([structured, rnd])


def pin_cast_torch(ora):
    """fp32 -> bf16 equals torch's round-to-nearest-even conversion on every non-NaN pattern tried."""
    import torch
    u = cast_patterns()
    x = u.view(np.float32)
    nan = np.isnan(x)
    got = ora.bf16_rne(x)
    want = torch.from_numpy(x[~nan].copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert got[~nan].tobytes() == want.tobytes()
    gn = got[nan].astype(np.uint32) << 16
    assert np.all(np.isnan(gn.view(np.float32)))


# ---------------------------------------------------- a7/a8 composite step

def _exact_int_grads(rng, W, padded, e=14):
    ints = rng.integers(-64, 65, size=(W, padded))
    return [f32_bits_to_bf16_exact((ints[k] * 2.0 ** -e).astype(np.float32)) for k in range(W)], ints, e


def pin_step_ddp_torch(ora, seed=8):
    """F = 1 (DDP): every replica ends equal to torch Adam applied to the exact all-reduce average.

    Integer * 2^-14 gradients make the fp32 sum exact and the mean exactly
    representable (W a power of two), so the average is known without the oracle.
    """
    rng = np.random.default_rng(seed)
    for W in (2, 4, 8):
        P = 61 * W - 3
        padded = -(-P // W) * W
        grads, ints, e = _exact_int_grads(rng, W, padded)
        mean = (ints.sum(axis=0) * 2.0 ** -e / W).astype(np.float32)
        assert np.all(mean.astype(np.float64) == ints.sum(axis=0) * 2.0 ** -e / W)
        p0 = (rng.standard_normal(padded) * 0.02).astype(np.float32)
        m0 = (np.abs(rng.standard_normal(padded)) * 1e-4).astype(np.float32)
        v0 = (np.abs(rng.standard_normal(padded)) * 1e-4).astype(np.float32)
        tp, tm, tv = _torch_adam_steps(p0, m0, v0, [mean], 1, ADAM)
        masters = [p0.copy() for _ in range(W)]
        ms = [m0.copy() for _ in range(W)]
        vs = [v0.copy() for _ in range(W)]
        fulls = [np.zeros(padded, np.uint16) for _ in range(W)]
        ora.shard_step(grads, 1, 0, W, masters, ms, vs, None, fulls, step=1, **ADAM)
        for r in range(W):
            assert _close(masters[r], tp) and _close(ms[r], tm) and _close(vs[r], tv), (W, r)
            assert fulls[r].tobytes() == fulls[0].tobytes()
        tb = f32_to_bf16_torch(tp)
        diff = np.abs(fulls[0].astype(np.int32) - tb.astype(np.int32))
        assert np.all(diff <= 1)


def f32_to_bf16_torch(x):
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def pin_step_f_continuum(ora, seed=9):
    """Every sharding factor F | W gives the same updated parameters (bit-identical) and
    the full bf16 buffer equals the bf16 of the updated flat master."""
    rng = np.random.default_rng(seed)
    for W in (4, 6, 8):
        P = 23 * W + 1
        padded = -(-P // W) * W
        grads = [ora_independent_bf16(rng.standard_normal(padded).astype(np.float32) * 1e-2)
                 for _ in range(W)]
        p0 = (rng.standard_normal(padded) * 0.02).astype(np.float32)
        m0 = (np.abs(rng.standard_normal(padded)) * 1e-4).astype(np.float32)
        v0 = (np.abs(rng.standard_normal(padded)) * 1e-4).astype(np.float32)
        ref = None
        for F in [f for f in range(1, W + 1) if W % f == 0]:
            S = padded // F
            R = W // F
            masters = [p0[(r % F) * S:(r % F + 1) * S].copy() for r in range(W)]
            ms = [m0[(r % F) * S:(r % F + 1) * S].copy() for r in range(W)]
            vs = [v0[(r % F) * S:(r % F + 1) * S].copy() for r in range(W)]
            fulls = [np.zeros(padded, np.uint16) for _ in range(R)]
            ora.shard_step(grads, F, 0, W, masters, ms, vs, None, fulls, step=3, **ADAM)
            flat = np.concatenate(masters[:F])
            for r in range(W):
                assert masters[r].tobytes() == flat[(r % F) * S:(r % F + 1) * S].tobytes()
            for g in range(R):
                assert fulls[g].tobytes() == f32_to_bf16_torch(flat).tobytes()
            if ref is None:
                ref = flat
            assert flat.tobytes() == ref.tobytes(), (W, F)


def pin_step_local_rank(ora, seed=10):
    """Local-rank mode: the owned slice equals the all-ranks result; other slices are copied bit-exactly."""
    rng = np.random.default_rng(seed)
    W = 4
    padded = 4 * 53
    S = padded // W
    grads = [ora_independent_bf16(rng.standard_normal(padded).astype(np.float32) * 1e-2) for _ in range(W)]
    p0 = (rng.standard_normal(padded) * 0.02).astype(np.float32)
    z = np.zeros(padded, np.float32)
    masters = [p0[r * S:(r + 1) * S].copy() for r in range(W)]
    full_all = np.zeros(padded, np.uint16)
    ora.shard_step(grads, W, 0, W, masters, [z[:S].copy() for _ in range(W)],
                   [z[:S].copy() for _ in range(W)], None, [full_all], step=1, **ADAM)
    for r in range(W):
        others = [rng.integers(0, 1 << 16, size=S).astype(np.uint16) for _ in range(W)]
        mr = [p0[r * S:(r + 1) * S].copy()]
        full = np.zeros(padded, np.uint16)
        ora.shard_step(grads, W, r, r + 1, mr, [z[:S].copy()], [z[:S].copy()], others, [full],
                       step=1, **ADAM)
        assert mr[0].tobytes() == masters[r].tobytes()
        for k in range(W):
            want = full_all[k * S:(k + 1) * S] if k == r else others[k]
            assert full[k * S:(k + 1) * S].tobytes() == want.tobytes()


# ------------------------------------------------------------ a9 accountant

def pin_account_worked_example(ora):
    g = golden("worked_example_7b.json")
    i, e = g["inputs"], g["expected"]
    P, N = i["P"], i["N"]
    U_exact = P / i["blocks"]
    a = ora.account(P, i["unit_params_printed"], N, N, i["prefetch"])
    assert a["ddp_persistent_bytes"] == e["ddp_state_bytes"]
    assert a["persistent_bytes"] == e["persistent_bytes"]
    assert float("%.2g" % U_exact) == e["unit_params_2sig"]
    assert round(a["transient_bytes"] / 1e9, 1) == e["transient_bytes_1dec_gb"]
    ax = ora.account(P, U_exact, N, N, i["prefetch"])
    assert 0.85e9 <= ax["transient_bytes"] <= 0.95e9
    assert round(a["peak_bytes"] / 1e9) == e["peak_bytes_int_gb"]
    assert i["gpu_bytes"] / 1e9 - round(a["peak_bytes"] / 1e9) == e["headroom_int_gb"]
    one = ora.account(P, P, N, N, 0)
    assert one["transient_bytes"] == e["single_unit_transient_bytes"]
    assert a["comm_bytes"] == e["fsdp_comm_bytes"] == 3 * e["per_collective_bytes"]
    assert a["ddp_comm_bytes"] == e["ddp_comm_bytes"]
    assert a["comm_bytes"] / a["ddp_comm_bytes"] == e["comm_ratio_vs_ddp"]


def _ring_reduce_scatter(bufs):
    """Ring reduce-scatter on integer data; returns (per-rank reduced chunk, elements sent by rank 0)."""
    n = len(bufs)
    chunks = [np.array_split(b.copy(), n) for b in bufs]
    sent0 = 0
    for s in range(n - 1):
        msgs = [(r, (r - s) % n, chunks[r][(r - s) % n].copy()) for r in range(n)]
        for r, c, payload in msgs:
            if r == 0:
                sent0 += payload.size
            chunks[(r + 1) % n][c] += payload
    owned = [chunks[r][(r + 1) % n] for r in range(n)]
    return owned, sent0


def _ring_all_gather(pieces):
    """Ring all-gather: rank r starts with piece r; returns (full buffers, elements sent by rank 0)."""
    n = len(pieces)
    have = [{r: pieces[r].copy()} for r in range(n)]
    sent0 = 0
    for s in range(n - 1):
        msgs = [(r, (r - s) % n) for r in range(n)]
        for r, c in msgs:
            payload = have[r][c]
            if r == 0:
                sent0 += payload.size
            have[(r + 1) % n][c] = payload.copy()
    fulls = [np.concatenate([h[c] for c in range(n)]) for h in have]
    return fulls, sent0


def ring_volume_sim(n_ranks: int, numel: int, kind: str) -> int:
    """Elements one rank sends in a ring all-gather / reduce-scatter / all-reduce of
    `numel` elements, measured by running the ring schedule on integer data (and
    checking that it computes the collective)."""
    if n_ranks == 1:
        return 0
    rng = np.random.default_rng(numel + n_ranks)
    bufs = [rng.integers(-5, 6, size=numel) for _ in range(n_ranks)]
    total = np.sum(bufs, axis=0)
    ref_chunks = np.array_split(total, n_ranks)
    if kind == "ag":
        pieces = np.array_split(bufs[0], n_ranks)
        fulls, sent = _ring_all_gather(pieces)
        assert all(np.array_equal(f, bufs[0]) for f in fulls)
        return sent
    owned, sent_rs = _ring_reduce_scatter(bufs)
    for r in range(n_ranks):
        assert np.array_equal(owned[r], ref_chunks[(r + 1) % n_ranks])
    if kind == "rs":
        return sent_rs
    ordered = [owned[(c - 1) % n_ranks] for c in range(n_ranks)]
    fulls, sent_ag = _ring_all_gather(ordered)
    assert all(np.array_equal(f, total) for f in fulls)
    return sent_rs + sent_ag


def pin_account_ring(ora):
    """The ring form equals a simulated ring schedule: 3 collectives in the group, all-reduce across groups."""
    P = 16 * 16 * 3  # divisible by every F*R below, so chunks are equal
    for N in (1, 2, 4, 8, 16):
        for F in [f for f in range(1, N + 1) if N % f == 0]:
            R = N // F
            a = ora.account(P, 0, N, F, 0)
            want = (2 * ring_volume_sim(F, P, "ag") + ring_volume_sim(F, P, "rs")
                    + ring_volume_sim(R, P // F, "ar"))
            assert abs(a["comm_elems_ring"] - want) <= 1e-9 * P, (N, F)
            assert a["persistent_bytes"] == 16 * P / F
        d = ora.account(P, 0, N, 1, 0)
        assert abs(d["ddp_comm_elems_ring"] - ring_volume_sim(N, P, "ar")) <= 1e-9 * P
        assert d["ddp_comm_elems"] == 2 * P


def pin_account_zero(ora):
    """ZeRO stages: the worked example's 7e9/8 totals per stage, the 4x / 8x limits, 8x at N = 8."""
    g = golden("zero_stages.json")
    for st, want in g["total_bytes"].items():
        a = ora.account_zero(g["P"], g["N"], int(st))
        assert a["total_bytes"] == want, st
        assert a["comm_elems"] == g["comm_elems_per_P"][st] * g["P"], st
    for st, want in g["large_N_reduction"].items():
        r = ora.account_zero(g["P"], g["large_N"], int(st))["reduction_vs_ddp"]
        assert abs(r - want) < 1e-3 * want, st
    assert ora.account_zero(g["P"], 8, 3)["reduction_vs_ddp"] == g["stage3_reduction_at_N8"]
    assert ora.account_zero(g["P"], 8, 3)["total_bytes"] == ora.account(g["P"], 0, 8, 8, 0)["persistent_bytes"]


ALL_PINS = [
    pin_layout_brute, pin_layout_golden, pin_pack_roundtrip,
    pin_rs_identical_rows, pin_rs_marker_slices, pin_rs_exact_rational, pin_rs_fold_order,
    pin_rs_ddp_endpoint,
    pin_adam_torch, pin_adam_first_step, pin_adam_zero_grad,
    pin_cast_torch,
    pin_step_ddp_torch, pin_step_f_continuum, pin_step_local_rank,
    pin_account_worked_example, pin_account_ring, pin_account_zero, pin_adam_torch_hyper,
]
