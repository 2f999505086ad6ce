"""The pipelined multi-unit step against the oracle (prefetch depth 0, 1, 2).

Each unit's W gradient slices come from pinned host memory (or device
memory) through a bounded pool of staging slots; the result must be
bit-identical to the oracle's local-rank step of every unit, over two
consecutive steps that reuse the pool.
"""
import numpy as np
import pytest

import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")

W, RANK = 8, 3
SIZES = [8 * 4096, 8 * 1000 + 5, 8 * 30000, 64, 8 * 2048 * 3 + 1]


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def make_units(base):
    torch = gu.torch()
    units, host = [], []
    for u, P in enumerate(SIZES):
        lay, _ = fs.fsdp_flatten_layout([P], W)
        S, padded = lay.shard_numel, lay.padded_numel
        k = lambda *f: synth.stream_key(base, u, *f)  # noqa: E731
        master = synth.normal_f32(k(1), S, 0.02, idx0=RANK * S, n_valid=P)
        m = synth.normal_f32(k(2), S, 1e-4, idx0=RANK * S, absval=True, n_valid=P)
        v = synth.normal_f32(k(3), S, 1e-4, idx0=RANK * S, absval=True, n_valid=P)
        others = [synth.normal_bf16(k(5), S, 0.02, idx0=j * S, n_valid=P) for j in range(W)]
        units.append(dict(layout=lay, master=gu.to_dev(master), exp_avg=gu.to_dev(m), exp_avg_sq=gu.to_dev(v),
                          other_shards=[None if j == RANK else gu.to_dev(others[j]) for j in range(W)],
                          full_out=torch.zeros(padded, dtype=torch.int16, device="cuda"),
                          shard_out=torch.zeros(S, dtype=torch.int16).pin_memory()))
        host.append(dict(lay=lay, master=master, m=m, v=v, others=others))
    return units, host


def grads_for(base, step, host_units):
    out = []
    for u, h in enumerate(host_units):
        lay = h["lay"]
        S, P = lay.shard_numel, lay.numel
        rows = [synth.normal_bf16(synth.stream_key(base, u, 4, k, step), S, 1e-2, idx0=RANK * S, n_valid=P)
                for k in range(W)]
        out.append(np.stack(rows))
    return out


def oracle_step(ora, h, slices, step):
    lay = h["lay"]
    S, padded = lay.shard_numel, lay.padded_numel
    rows = []
    for k in range(W):
        r = np.zeros(padded, np.uint16)
        r[RANK * S:(RANK + 1) * S] = slices[k]
        rows.append(r)
    full = [np.zeros(padded, np.uint16)]
    ora.shard_step(rows, W, RANK, RANK + 1, [h["master"]], [h["m"]], [h["v"]], h["others"], full,
                   step=step, **gu.HP)
    return full[0]


@pytest.mark.parametrize("n_slots,source,same_stream", [
    (1, "host", False), (2, "host", False), (3, "host", False), (2, "device", False), (2, "host", True)])
def test_pipeline_matches_oracle(ora, n_slots, source, same_stream):
    torch = gu.torch()
    base = 7000 + 10 * n_slots + (source == "device") + 2 * same_stream
    units, host = make_units(base)
    slot = max(u["layout"].padded_numel for u in units)
    staging = torch.empty(n_slots * slot, dtype=torch.int16, device="cuda")
    compute = torch.cuda.Stream()
    copy = compute if same_stream else torch.cuda.Stream()
    for step in (1, 2):
        g = grads_for(base, step, host)
        for u, gs in zip(units, g):
            t = torch.from_numpy(gs.view(np.int16).copy())
            u["grad_slices"] = t.pin_memory() if source == "host" else t.cuda()
        fs.fsdp_pipeline_step(units, RANK, staging, slot, n_slots, gu.adam_hyper(step), compute=compute, copy=copy)
        torch.cuda.synchronize()
        for u, h, gs in zip(units, host, g):
            want_full = oracle_step(ora, h, gs, step)
            S = h["lay"].shard_numel
            gu.assert_same_bits(gu.to_host(u["master"]), h["master"], "master t%d" % step)
            gu.assert_same_bits(gu.to_host(u["exp_avg"]), h["m"], "exp_avg t%d" % step)
            gu.assert_same_bits(gu.to_host(u["exp_avg_sq"]), h["v"], "exp_avg_sq t%d" % step)
            gu.assert_same_bits(gu.to_host(u["full_out"]), want_full, "full t%d" % step)
            gu.assert_same_bits(u["shard_out"].numpy().view(np.uint16), want_full[RANK * S:(RANK + 1) * S],
                                "shard_out t%d" % step)


def test_pipeline_equals_grouped_step():
    """Same values through the grouped single launch and through the pipeline: identical bits."""
    torch = gu.torch()
    base = 7500
    units, host = make_units(base)
    g = grads_for(base, 1, host)
    # grouped: full-length gradient rows with the owned slice filled
    grouped = []
    for u, h, gs in zip(units, host, g):
        lay = h["lay"]
        S = lay.shard_numel
        rows = torch.zeros((W, lay.padded_numel), dtype=torch.int16, device="cuda")
        rows[:, RANK * S:(RANK + 1) * S] = torch.from_numpy(gs.view(np.int16)).cuda()
        grouped.append(dict(layout=lay, grads=[rows[k] for k in range(W)], master=[u["master"].clone()],
                            exp_avg=[u["exp_avg"].clone()], exp_avg_sq=[u["exp_avg_sq"].clone()],
                            other_shards=u["other_shards"], full_out=[u["full_out"].clone()]))
        u["grad_slices"] = torch.from_numpy(gs.view(np.int16).copy()).pin_memory()
    fs.fsdp_shard_step_grouped(grouped, RANK, RANK + 1, gu.adam_hyper(1))
    slot = max(u["layout"].padded_numel for u in units)
    staging = torch.empty(2 * slot, dtype=torch.int16, device="cuda")
    fs.fsdp_pipeline_step(units, RANK, staging, slot, 2, gu.adam_hyper(1))
    torch.cuda.synchronize()
    for u, gr in zip(units, grouped):
        assert torch.equal(u["master"], gr["master"][0]) and torch.equal(u["full_out"], gr["full_out"][0])
        assert torch.equal(u["exp_avg"], gr["exp_avg"][0]) and torch.equal(u["exp_avg_sq"], gr["exp_avg_sq"][0])


def _bf16_bits(x):
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_edge_units_in_pieces_match_oracle(ora):
    """First and last units above 4 M shard elements (odd lengths: ragged last pieces, an
    odd own-slice offset), a short unit between them: the pipeline moves the edge units in
    pieces; every output equals the oracle's local-rank step of each unit bit for bit."""
    torch = gu.torch()
    rng = np.random.default_rng(7700)
    sizes = [8 * (4194304 + 6149), 8 * 100000 + 5, 8 * (4194304 + 2 * 2048 + 3)]
    units, host = [], []
    for P in sizes:
        lay, _ = fs.fsdp_flatten_layout([P], W)
        S, padded = lay.shard_numel, lay.padded_numel
        valid = max(0, min(S, P - RANK * S))
        master = np.zeros(S, np.float32)
        master[:valid] = rng.standard_normal(valid) * 0.02
        m = np.abs(rng.standard_normal(S)).astype(np.float32) * 1e-4
        v = np.abs(rng.standard_normal(S)).astype(np.float32) * 1e-4
        others = [_bf16_bits(rng.standard_normal(S) * 0.02) for _ in range(W)]
        slices = np.stack([_bf16_bits(rng.standard_normal(S) * 1e-2) for _ in range(W)])
        units.append(dict(layout=lay, master=gu.to_dev(master), exp_avg=gu.to_dev(m), exp_avg_sq=gu.to_dev(v),
                          other_shards=[None if j == RANK else gu.to_dev(others[j]) for j in range(W)],
                          full_out=torch.zeros(padded, dtype=torch.int16, device="cuda"),
                          shard_out=torch.zeros(S, dtype=torch.int16).pin_memory(),
                          grad_slices=torch.from_numpy(slices.view(np.int16).copy()).pin_memory()))
        host.append(dict(lay=lay, master=master, m=m, v=v, others=others, slices=slices))
    slot = max(u["layout"].padded_numel for u in units)
    staging = torch.empty(2 * slot, dtype=torch.int16, device="cuda")
    fs.fsdp_pipeline_step(units, RANK, staging, slot, 2, gu.adam_hyper(4), compute=torch.cuda.Stream(),
                          copy=torch.cuda.Stream())
    torch.cuda.synchronize()
    for i, (u, h) in enumerate(zip(units, host)):
        want_full = oracle_step(ora, h, h["slices"], 4)
        S = h["lay"].shard_numel
        gu.assert_same_bits(gu.to_host(u["master"]), h["master"], "master unit %d" % i)
        gu.assert_same_bits(gu.to_host(u["exp_avg"]), h["m"], "exp_avg unit %d" % i)
        gu.assert_same_bits(gu.to_host(u["exp_avg_sq"]), h["v"], "exp_avg_sq unit %d" % i)
        gu.assert_same_bits(gu.to_host(u["full_out"]), want_full, "full unit %d" % i)
        gu.assert_same_bits(u["shard_out"].numpy().view(np.uint16), want_full[RANK * S:(RANK + 1) * S],
                            "shard_out unit %d" % i)
    assert fs.fsdp_device_status() == 0
