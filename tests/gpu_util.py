"""Helpers for the GPU parity tests: seeded inputs on host and device, comparisons."""
from __future__ import annotations

import numpy as np

import synth

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)


def torch():
    import torch as t
    return t


def to_dev(a: np.ndarray):
    t = torch()
    if a.dtype == np.uint16:
        return t.from_numpy(a.view(np.int16).copy()).cuda()
    return t.from_numpy(a.copy()).cuda()


def to_dev_at(a: np.ndarray, off: int):
    """A device copy of fp32 `a` that starts `off` elements into its own allocation
    (off = 4: 16 bytes past the allocation's alignment)."""
    if off == 0:
        return to_dev(a)
    t = torch()
    buf = t.zeros(off + len(a), dtype=t.float32, device="cuda")
    buf[off:] = to_dev(a)
    return buf[off:]


def to_host(x) -> np.ndarray:
    t = torch()
    a = x.detach().cpu()
    if a.dtype in (t.int16, t.bfloat16, t.uint16):
        return a.view(t.int16).numpy().view(np.uint16).copy()
    return a.numpy().copy()


def adam_hyper(step, **over):
    import fully_sharded_gb300 as fs
    h = dict(HP)
    h.update(over)
    return fs.AdamHyper(step=step, **h)


def assert_f32_close(got, want, what, rel=1e-6):
    """fp32 tolerance of the method: |a - b| <= rel |b| + rel max|b| (floor for cancellation)."""
    got = np.asarray(got, np.float32)
    want = np.asarray(want, np.float32)
    assert got.shape == want.shape, what
    floor = rel * float(np.max(np.abs(want))) if want.size else 0.0
    d = np.abs(got.astype(np.float64) - want.astype(np.float64))
    bad = d > rel * np.abs(want.astype(np.float64)) + floor
    assert not np.any(bad), "%s: %d of %d outside tolerance (first at %d: %r vs %r)" % (
        what, int(bad.sum()), bad.size, int(np.argmax(bad)), got[np.argmax(bad)], want[np.argmax(bad)])


def bf16_ulp_diff(a, b) -> np.ndarray:
    """Distance in bf16 ulps between two arrays of bf16 bit patterns (sign-magnitude aware)."""
    def ordered(x):
        x = np.asarray(x, np.uint16).astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def assert_bf16_close(got, want, what, ulps=1):
    d = bf16_ulp_diff(got, want)
    assert np.all(d <= ulps), "%s: %d bf16 values more than %d ulp apart" % (what, int((d > ulps).sum()), ulps)


def assert_same_bits(got, want, what):
    got = np.ascontiguousarray(got)
    want = np.ascontiguousarray(want)
    if got.tobytes() != want.tobytes():
        g = got.view(np.uint8) if got.dtype != np.uint8 else got
        w = want.view(np.uint8) if want.dtype != np.uint8 else want
        n = min(g.size, w.size)
        first = int(np.argmax(g[:n] != w[:n])) if n else 0
        raise AssertionError("%s: bit mismatch (sizes %d/%d, first differing byte %d)"
                             % (what, g.size, w.size, first))


def host_normal(key, n, sigma, idx0=0, absval=False, n_valid=None, bf16=False):
    if sigma == 0.0:
        return np.zeros(n, np.uint16 if bf16 else np.float32)
    f = synth.normal_bf16 if bf16 else synth.normal_f32
    return f(key, n, sigma, idx0=idx0, absval=absval, n_valid=n_valid)


def dev_normal(key, n, sigma, idx0=0, absval=False, n_valid=None, bf16=False):
    t = torch()
    x = t.empty(n, dtype=t.int16 if bf16 else t.float32, device="cuda")
    if sigma == 0.0:
        x.zero_()
    else:
        synth.fill_(x, key, sigma, idx0=idx0, absval=absval, n_valid=n_valid)
    return x


def guarded(n, dtype, pattern, guard=4096):
    """A CUDA buffer with `guard` canary elements on both sides; returns (whole, view)."""
    t = torch()
    whole = t.empty(n + 2 * guard, dtype=dtype, device="cuda")
    whole.fill_(pattern)
    return whole, whole[guard:guard + n]


def canaries_intact(whole, n, pattern, guard=4096) -> bool:
    h = whole.detach().cpu()
    return bool((h[:guard] == pattern).all() and (h[guard + n:] == pattern).all())
