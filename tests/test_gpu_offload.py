"""Optimizer-state offload: master, m and v in mapped page-locked host memory, same results."""
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


@pytest.mark.parametrize("W,P,rank", [(8, 8 * 20000 + 3, None), (8, 8 * 30000, 2)])
def test_state_in_host_memory_matches_oracle(ora, W, P, rank):
    torch = gu.torch()
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S, padded = lay.shard_numel, lay.padded_numel
    ranks = list(range(W)) if rank is None else [rank]
    base = 4400 + W + (rank or 0)
    master = synth.normal_f32(synth.stream_key(base, 1), padded, 0.02, n_valid=P)
    m = synth.normal_f32(synth.stream_key(base, 2), padded, 1e-4, absval=True, n_valid=P)
    v = synth.normal_f32(synth.stream_key(base, 3), padded, 1e-4, absval=True, n_valid=P)
    grads = [synth.normal_bf16(synth.stream_key(base, 4, k), padded, 1e-2, n_valid=P) for k in range(W)]
    others = [synth.normal_bf16(synth.stream_key(base, 5), S, 0.02, idx0=k * S) for k in range(W)]
    sl = lambda a, r: np.ascontiguousarray(a[r * S:(r + 1) * S])  # noqa: E731
    pin = lambda a: torch.from_numpy(a.copy()).pin_memory()  # noqa: E731
    hm = [pin(sl(master, r)) for r in ranks]
    he = [pin(sl(m, r)) for r in ranks]
    hv = [pin(sl(v, r)) for r in ranks]
    full = torch.zeros(padded, dtype=torch.int16, device="cuda")
    local = rank is not None
    fs.fsdp_shard_step([gu.to_dev(g) for g in grads], lay, ranks[0], ranks[-1] + 1,
                       [t.data_ptr() for t in hm], [t.data_ptr() for t in he], [t.data_ptr() for t in hv],
                       [gu.to_dev(o) for o in others] if local else None, [full], gu.adam_hyper(3))
    torch.cuda.synchronize()
    om = [sl(master, r).copy() for r in ranks]
    oe = [sl(m, r).copy() for r in ranks]
    ov = [sl(v, r).copy() for r in ranks]
    ofull = [np.zeros(padded, np.uint16)]
    ora.shard_step(grads, W, ranks[0], ranks[-1] + 1, om, oe, ov, others if local else None, ofull,
                   step=3, **gu.HP)
    for i in range(len(ranks)):
        gu.assert_same_bits(hm[i].numpy(), om[i], "master")
        gu.assert_same_bits(he[i].numpy(), oe[i], "exp_avg")
        gu.assert_same_bits(hv[i].numpy(), ov[i], "exp_avg_sq")
    gu.assert_same_bits(gu.to_host(full), ofull[0], "full")
