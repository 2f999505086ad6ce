"""Full state dict, sharded resume and the ZeRO stage 1 step on the GPU, against the oracle."""
import numpy as np
import pytest

import gpu_util as gu
import synth
from synth import workloads as wls

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


SHAPES = [(64, 32), (32,), (32, 16), (16,), (1000, 3)]  # the tiny MLP plus a ragged tensor
W = 4


def _all_ranks_setup(base):
    torch = gu.torch()
    numels = wls.numels(SHAPES)
    lay, offs = fs.fsdp_flatten_layout(numels, W)
    P, padded, S = lay.numel, lay.padded_numel, lay.shard_numel
    master = synth.normal_f32(synth.stream_key(base, 1), padded, 0.02, n_valid=P)
    state = dict(master=[gu.to_dev(master[r * S:(r + 1) * S]) for r in range(W)],
                 exp_avg=[torch.zeros(S, device="cuda") for _ in range(W)],
                 exp_avg_sq=[torch.zeros(S, device="cuda") for _ in range(W)])
    return lay, offs, master, state


def _step(lay, state, base, step, full):
    P, padded = lay.numel, lay.padded_numel
    grads = [synth.normal_bf16(synth.stream_key(base, 4, k, step), padded, 1e-2, n_valid=P) for k in range(W)]
    fs.fsdp_shard_step([gu.to_dev(g) for g in grads], lay, 0, W, state["master"], state["exp_avg"],
                       state["exp_avg_sq"], None, [full], gu.adam_hyper(step))
    return grads


def test_full_state_dict_matches_oracle(ora):
    torch = gu.torch()
    lay, offs, master, state = _all_ranks_setup(11)
    S, padded = lay.shard_numel, lay.padded_numel
    full = torch.zeros(padded, dtype=torch.int16, device="cuda")
    grads = _step(lay, state, 11, 1, full)
    om = [master[r * S:(r + 1) * S].copy() for r in range(W)]
    z = [np.zeros(S, np.float32) for _ in range(W)]
    ora.shard_step(grads, W, 0, W, om, [x.copy() for x in z], [x.copy() for x in z], None,
                   [np.zeros(padded, np.uint16)], step=1, **gu.HP)
    from fully_sharded_gb300 import checkpoint as ck
    tensors = ck.full_state_dict(state["master"], lay, offs, SHAPES)
    want = ora.unpack(np.concatenate(om), SHAPES)
    for got, w in zip(tensors, want):
        assert tuple(got.shape) == w.shape
        gu.assert_same_bits(gu.to_host(got), w, "full state tensor")
    # bf16 parameters gathered the same way equal the fused step's full buffer
    flat = torch.empty(padded, dtype=torch.int16, device="cuda")
    fs.fsdp_all_gather_state([full[r * S:(r + 1) * S].clone() for r in range(W)], lay, flat)
    torch.cuda.synchronize()
    assert torch.equal(flat, full)


def test_sharded_resume_is_bit_exact(tmp_path):
    torch = gu.torch()
    from fully_sharded_gb300 import checkpoint as ck
    lay, offs, master, a = _all_ranks_setup(12)
    _, _, _, b = _all_ranks_setup(12)
    padded = lay.padded_numel
    fa = torch.zeros(padded, dtype=torch.int16, device="cuda")
    fb = torch.zeros(padded, dtype=torch.int16, device="cuda")
    for t in (1, 2, 3):
        _step(lay, a, 12, t, fa)
    _step(lay, b, 12, 1, fb)
    for r in range(W):
        ck.save_sharded(str(tmp_path), r, [dict(layout=lay, master=b["master"][r], exp_avg=b["exp_avg"][r],
                                                exp_avg_sq=b["exp_avg_sq"][r])], step=1)
    _, _, _, c = _all_ranks_setup(999)  # fresh buffers with other contents
    steps = [ck.load_sharded(str(tmp_path), r, [dict(layout=lay, master=c["master"][r], exp_avg=c["exp_avg"][r],
                                                     exp_avg_sq=c["exp_avg_sq"][r])]) for r in range(W)]
    assert steps == [1] * W
    fc = torch.zeros(padded, dtype=torch.int16, device="cuda")
    for t in (2, 3):
        _step(lay, c, 12, t, fc)
    torch.cuda.synchronize()
    for r in range(W):
        for name in ("master", "exp_avg", "exp_avg_sq"):
            assert torch.equal(a[name][r].view(torch.int32), c[name][r].view(torch.int32)), (name, r)
    assert torch.equal(fa, fc)


@pytest.mark.parametrize("rank", [0, 5])
def test_zero1_step_matches_oracle(ora, rank):
    torch = gu.torch()
    Wz, P = 8, 8 * 9001 + 5
    lay, _ = fs.fsdp_flatten_layout([P], Wz)
    S, padded = lay.shard_numel, lay.padded_numel
    base = 300 + rank
    grads = [synth.normal_bf16(synth.stream_key(base, 4, k), padded, 1e-2, n_valid=P) for k in range(Wz)]
    master = synth.normal_f32(synth.stream_key(base, 1), S, 0.02, idx0=rank * S, n_valid=P)
    m = synth.normal_f32(synth.stream_key(base, 2), S, 1e-4, idx0=rank * S, absval=True, n_valid=P)
    v = synth.normal_f32(synth.stream_key(base, 3), S, 1e-4, idx0=rank * S, absval=True, n_valid=P)
    others = [synth.normal_bf16(synth.stream_key(base, 5), S, 0.02, idx0=k * S, n_valid=P) for k in range(Wz)]
    avg = torch.empty(padded, device="cuda")
    md, ed, vd = gu.to_dev(master), gu.to_dev(m), gu.to_dev(v)
    full = torch.zeros(padded, dtype=torch.int16, device="cuda")
    fs.fsdp_zero1_step([gu.to_dev(g) for g in grads], lay, rank, avg, md, ed, vd,
                       [None if k == rank else gu.to_dev(o) for k, o in enumerate(others)], full, gu.adam_hyper(1))
    torch.cuda.synchronize()
    # the all-reduce average is the F = 1 reduce-scatter; the update is the local-rank step
    gu.assert_same_bits(gu.to_host(avg), ora.reduce_scatter(grads, 1, 0), "all-reduce average")
    om, oe, ov = master.copy(), m.copy(), v.copy()
    ofull = [np.zeros(padded, np.uint16)]
    ora.shard_step(grads, Wz, rank, rank + 1, [om], [oe], [ov], others, ofull, step=1, **gu.HP)
    gu.assert_same_bits(gu.to_host(md), om, "master")
    gu.assert_same_bits(gu.to_host(ed), oe, "exp_avg")
    gu.assert_same_bits(gu.to_host(vd), ov, "exp_avg_sq")
    gu.assert_same_bits(gu.to_host(full), ofull[0], "full")
