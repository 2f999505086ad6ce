"""Special values through the fused step: +-inf, NaN, subnormal and signed-zero gradients,
huge and subnormal parameters. Non-NaN outputs must equal the oracle bit for bit; NaN must
appear exactly where the oracle has NaN (NaN payloads are not specified)."""
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


def test_special_values_match_oracle(ora):
    torch = gu.torch()
    W, P = 4, 4 * 4096
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S = lay.shard_numel
    rng = np.random.default_rng(3)
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
    om = [master[r * S:(r + 1) * S].copy() for r in range(W)]
    oe = [m[r * S:(r + 1) * S].copy() for r in range(W)]
    ov = [v[r * S:(r + 1) * S].copy() for r in range(W)]
    ofull = [np.zeros(P, np.uint16)]
    ora.shard_step(grads, W, 0, W, om, oe, ov, None, ofull, step=2, **gu.HP)
    md = [gu.to_dev(master[r * S:(r + 1) * S]) for r in range(W)]
    ed = [gu.to_dev(m[r * S:(r + 1) * S]) for r in range(W)]
    vd = [gu.to_dev(v[r * S:(r + 1) * S]) for r in range(W)]
    full = torch.zeros(P, dtype=torch.int16, device="cuda")
    fs.fsdp_shard_step([gu.to_dev(g) for g in grads], lay, 0, W, md, ed, vd, None, [full], gu.adam_hyper(2))
    torch.cuda.synchronize()
    nan_seen = 0
    for r in range(W):
        _same_or_both_nan(gu.to_host(md[r]), om[r], "master r%d" % r)
        _same_or_both_nan(gu.to_host(ed[r]), oe[r], "exp_avg r%d" % r)
        _same_or_both_nan(gu.to_host(vd[r]), ov[r], "exp_avg_sq r%d" % r)
        nan_seen += int(np.isnan(om[r]).sum())
    _same_or_both_nan_bf16(gu.to_host(full), ofull[0], "full")
    assert nan_seen > 0  # the case does reach the NaN paths
