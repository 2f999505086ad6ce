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


@pytest.mark.parametrize("W,rank,n_slots,same_stream,odd_slot", [
    (8, 5, 1, False, False), (8, 5, 2, False, False), (8, 5, 3, False, False), (8, 5, 2, True, False),
    (8, 5, 2, False, True), (3, 1, 2, False, False)])
def test_staged_offload_matches_oracle(ora, W, rank, n_slots, same_stream, odd_slot):
    """fsdp_offload_step over four units (a ragged one, whole chunks, a larger one, a tiny
    one), two steps in a row with fresh gradients: the host state and every full buffer
    equal the oracle's bit for bit. odd_slot: slot arrays not 16-byte aligned (the scalar
    path); W = 3: shards of odd length, misaligned views (the scalar path as well)."""
    torch = gu.torch()
    sizes = [8 * 40000 + 5, 8 * 2048 * 3, 8 * 100000, 17]
    lays = [fs.fsdp_flatten_layout([P], W)[0] for P in sizes]
    pin = lambda a: torch.from_numpy(a.copy()).pin_memory()  # noqa: E731
    units, oracle_units = [], []
    for u, (P, lay) in enumerate(zip(sizes, lays)):
        S, padded = lay.shard_numel, lay.padded_numel
        base = 4500 + 10 * W + u
        sl = lambda a: np.ascontiguousarray(a[rank * S:(rank + 1) * S])  # noqa: E731
        master = synth.normal_f32(synth.stream_key(base, 1), padded, 0.02, n_valid=P)
        m = synth.normal_f32(synth.stream_key(base, 2), padded, 1e-4, absval=True, n_valid=P)
        v = synth.normal_f32(synth.stream_key(base, 3), padded, 1e-4, absval=True, n_valid=P)
        others = [synth.normal_bf16(synth.stream_key(base, 5), S, 0.02, idx0=k * S) for k in range(W)]
        units.append(dict(layout=lay, master=pin(sl(master)), exp_avg=pin(sl(m)), exp_avg_sq=pin(sl(v)),
                          other_shards=[gu.to_dev(o) for o in others],
                          full_out=torch.zeros(padded, dtype=torch.int16, device="cuda")))
        oracle_units.append(dict(master=sl(master).copy(), m=sl(m).copy(), v=sl(v).copy(), others=others,
                                 full=np.zeros(padded, np.uint16), base=base, P=P, padded=padded))
    slot = max(l.shard_numel for l in lays)
    slot = slot + (1 if slot % 4 == 0 else 0) if odd_slot else (slot + 3) // 4 * 4
    staging = torch.empty(n_slots * 3 * slot, device="cuda")
    streams = [torch.cuda.Stream()] * 3 if same_stream else [torch.cuda.Stream() for _ in range(3)]
    for step in (1, 2):
        for u, o in zip(units, oracle_units):
            g = [synth.normal_bf16(synth.stream_key(o["base"], 4, k, step), o["padded"], 1e-2, n_valid=o["P"])
                 for k in range(W)]
            u["grads"] = [gu.to_dev(x) for x in g]
            o["grads"] = g
        fs.fsdp_offload_step(units, rank, staging, slot, n_slots, gu.adam_hyper(step),
                             compute=streams[0], h2d=streams[1], d2h=streams[2])
        streams[0].synchronize()  # ordered after every copy back
        for o in oracle_units:
            ora.shard_step(o["grads"], W, rank, rank + 1, [o["master"]], [o["m"]], [o["v"]], o["others"],
                           [o["full"]], step=step, **gu.HP)
        for i, (u, o) in enumerate(zip(units, oracle_units)):
            gu.assert_same_bits(u["master"].numpy(), o["master"], "master u%d step %d" % (i, step))
            gu.assert_same_bits(u["exp_avg"].numpy(), o["m"], "exp_avg u%d step %d" % (i, step))
            gu.assert_same_bits(u["exp_avg_sq"].numpy(), o["v"], "exp_avg_sq u%d step %d" % (i, step))
            gu.assert_same_bits(gu.to_host(u["full_out"]), o["full"], "full u%d step %d" % (i, step))
