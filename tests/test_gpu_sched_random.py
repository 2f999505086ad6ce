"""Random draws of the two schedulers against the grouped single launch (itself checked
against the oracle elsewhere): the pipelined step (gradients from pinned host memory
through a pool of staging slots; units above 4 M shard elements at either end move in
pieces) and the staged offload step (optimizer state in pinned host memory). Each case
draws W, the rank, the number of slots and the unit sizes (odd sizes included); the
scheduler's outputs must equal the grouped step's on the same inputs, bit for bit."""
import numpy as np
import pytest

import gpu_util as gu

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _draw(rng, big_ends):
    W = int(rng.choice([2, 4, 8]))
    n = int(rng.integers(1, 5))
    sizes = []
    for u in range(n):
        if big_ends and u in (0, n - 1):
            S = int(rng.integers(4_194_305, 6_000_000))
        else:
            S = int(rng.integers(1, 600_000))
        sizes.append(W * S - int(rng.integers(0, W)))  # the last shard a little short: padding
    return W, int(rng.integers(0, W)), int(rng.integers(1, 4)), [max(1, P) for P in sizes]


def _units(torch, gen, W, rank, sizes):
    """Device state, gathered shards and full rows with the rank's slice filled (the grouped
    step's view), plus the rank's W gradient slices (the schedulers' view)."""
    out = []
    for P in sizes:
        lay, _ = fs.fsdp_flatten_layout([P], W)
        S, padded = lay.shard_numel, lay.padded_numel
        bf = lambda n: (torch.randn(n, device="cuda", generator=gen) * 1e-2).to(torch.bfloat16).view(torch.int16)  # noqa: E731
        slices = bf(W * S).view(W, S)
        rows = torch.zeros((W, padded), dtype=torch.int16, device="cuda")
        rows[:, rank * S:(rank + 1) * S] = slices
        out.append(dict(layout=lay, S=S, padded=padded, slices=slices, rows=rows,
                        master=torch.randn(S, device="cuda", generator=gen) * 0.02,
                        exp_avg=torch.randn(S, device="cuda", generator=gen).abs() * 1e-4,
                        exp_avg_sq=torch.randn(S, device="cuda", generator=gen).abs() * 1e-4,
                        others=[None if k == rank else bf(S) for k in range(W)]))
    return out


def _grouped(torch, units, rank, step):
    g = []
    for u in units:
        g.append(dict(layout=u["layout"], grads=[u["rows"][k] for k in range(u["rows"].shape[0])],
                      master=[u["master"].clone()], exp_avg=[u["exp_avg"].clone()],
                      exp_avg_sq=[u["exp_avg_sq"].clone()], other_shards=u["others"],
                      full_out=[torch.zeros(u["padded"], dtype=torch.int16, device="cuda")]))
    fs.fsdp_shard_step_grouped(g, rank, rank + 1, gu.adam_hyper(step))
    return g


@pytest.mark.parametrize("seed", range(6))
def test_random_pipeline_equals_grouped(seed):
    torch = gu.torch()
    rng = np.random.default_rng(3100 + seed)
    W, rank, n_slots, sizes = _draw(rng, big_ends=seed % 2 == 0)
    gen = torch.Generator("cuda").manual_seed(seed)
    units = _units(torch, gen, W, rank, sizes)
    step = int(rng.integers(1, 1000))
    want = _grouped(torch, units, rank, step)
    punits = []
    for u in units:
        punits.append(dict(layout=u["layout"], grad_slices=u["slices"].cpu().pin_memory(), master=u["master"],
                           exp_avg=u["exp_avg"], exp_avg_sq=u["exp_avg_sq"], other_shards=u["others"],
                           full_out=torch.zeros(u["padded"], dtype=torch.int16, device="cuda"),
                           shard_out=torch.zeros(u["S"], dtype=torch.int16).pin_memory()))
    slot = max(u["padded"] for u in units)
    staging = torch.empty(n_slots * slot, dtype=torch.int16, device="cuda")
    fs.fsdp_pipeline_step(punits, rank, staging, slot, n_slots, gu.adam_hyper(step), compute=torch.cuda.Stream(),
                          copy=torch.cuda.Stream())
    torch.cuda.synchronize()
    what = "W %d rank %d slots %d sizes %s" % (W, rank, n_slots, sizes)
    for p, g in zip(punits, want):
        for name in ("master", "exp_avg", "exp_avg_sq"):
            assert torch.equal(p[name].view(torch.int32), g[name][0].view(torch.int32)), name + " " + what
        assert torch.equal(p["full_out"], g["full_out"][0]), "full_out " + what
        S = p["layout"].shard_numel
        assert torch.equal(p["shard_out"], g["full_out"][0][rank * S:(rank + 1) * S].cpu()), "shard_out " + what
    assert fs.fsdp_device_status() == 0


@pytest.mark.parametrize("seed", range(4))
def test_random_offload_equals_grouped(seed):
    torch = gu.torch()
    rng = np.random.default_rng(3200 + seed)
    W, rank, n_slots, sizes = _draw(rng, big_ends=seed % 2 == 1)
    gen = torch.Generator("cuda").manual_seed(100 + seed)
    units = _units(torch, gen, W, rank, sizes)
    step = int(rng.integers(1, 1000))
    want = _grouped(torch, units, rank, step)
    ounits, host = [], []
    for u in units:
        h = {n: u[n].cpu().pin_memory() for n in ("master", "exp_avg", "exp_avg_sq")}
        host.append(h)
        ounits.append(dict(layout=u["layout"], grads=[u["rows"][k] for k in range(W)], master=h["master"],
                           exp_avg=h["exp_avg"], exp_avg_sq=h["exp_avg_sq"], other_shards=u["others"],
                           full_out=torch.zeros(u["padded"], dtype=torch.int16, device="cuda")))
    slot = (max(u["S"] for u in units) + 3) // 4 * 4
    staging = torch.empty(n_slots * 3 * slot, device="cuda")
    fs.fsdp_offload_step(ounits, rank, staging, slot, n_slots, gu.adam_hyper(step), compute=torch.cuda.Stream(),
                         h2d=torch.cuda.Stream(), d2h=torch.cuda.Stream())
    torch.cuda.synchronize()
    what = "W %d rank %d slots %d sizes %s" % (W, rank, n_slots, sizes)
    for o, h, g in zip(ounits, host, want):
        for name in ("master", "exp_avg", "exp_avg_sq"):
            assert torch.equal(h[name].view(torch.int32), g[name][0].cpu().view(torch.int32)), name + " " + what
        assert torch.equal(o["full_out"], g["full_out"][0]), "full_out " + what
    assert fs.fsdp_device_status() == 0
