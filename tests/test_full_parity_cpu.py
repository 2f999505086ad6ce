"""The full-size comparison harness (tests/full_parity.py) checked on the CPU.

The harness runs the oracle on pieces of a unit's slices. Here the "device"
outputs are the oracle's own step over the whole unit, held in CPU tensors:
the piecewise comparison must accept them on every element, in local-rank and
all-ranks mode, with ragged pieces; and one flipped bit in any output must be
reported.
"""
import numpy as np
import pytest
import torch

import full_parity
import gpu_util as gu

HP = gu.HP


def _unit(ora, W, rank_begin, rank_end, P, step, seed):
    rng = np.random.default_rng(seed)
    offs, _, padded, S = ora.flatten_layout([P], W)
    bf = lambda x: ora.bf16_rne(x.astype(np.float32))  # noqa: E731
    grads = [bf(rng.standard_normal(padded) * 1e-3) for _ in range(W)]
    owned = list(range(rank_begin, rank_end))
    pre = {name: [(np.abs(rng.standard_normal(S)) * 1e-4 if name != "master" else rng.standard_normal(S) * 0.02)
                  .astype(np.float32) for _ in owned] for name in ("master", "exp_avg", "exp_avg_sq")}
    local = rank_end - rank_begin < W
    others = [None if r in owned else bf(rng.standard_normal(S) * 0.02) for r in range(W)] if local else None
    post = {name: [x.copy() for x in pre[name]] for name in pre}
    full = [np.zeros(padded, np.uint16)]
    ora.shard_step(grads, W, rank_begin, rank_end, post["master"], post["exp_avg"], post["exp_avg_sq"],
                   others, full, step=step, **HP)

    class Lay:
        world_size, shard_factor, shard_numel = W, W, S

    t16 = lambda a: torch.from_numpy(a.view(np.int16).copy())  # noqa: E731
    unit = dict(layout=Lay, grads=[t16(g) for g in grads],
                master=[torch.from_numpy(x) for x in post["master"]],
                exp_avg=[torch.from_numpy(x) for x in post["exp_avg"]],
                exp_avg_sq=[torch.from_numpy(x) for x in post["exp_avg_sq"]],
                other_shards=None if others is None else [None if o is None else t16(o) for o in others],
                full_out=[t16(full[0])])

    def regen(name, r, a, n):
        return torch.from_numpy(pre[name][owned.index(r)][a:a + n].copy())

    return unit, regen, S


@pytest.mark.parametrize("W,rb,re", [(8, 3, 4), (4, 0, 4), (8, 0, 8)])
def test_pieces_equal_the_whole_unit(ora, W, rb, re):
    unit, regen, S = _unit(ora, W, rb, re, W * 5000 + 3, step=2, seed=W + rb)
    assert full_parity.check_unit_every_element(ora, unit, rb, re, 2, regen, "cpu", piece=700) == S


@pytest.mark.parametrize("where", ["master", "exp_avg_sq", "own_slice", "gathered_slice", "last_element"])
def test_a_flipped_bit_is_reported(ora, where):
    W, rb, re = 8, 3, 4
    unit, regen, S = _unit(ora, W, rb, re, W * 5000 + 3, step=1, seed=7)
    if where in ("master", "exp_avg_sq"):
        unit[where][0].view(torch.int32)[1234] ^= 1
    elif where == "own_slice":
        unit["full_out"][0][rb * S + 4321] ^= 1
    elif where == "gathered_slice":
        unit["full_out"][0][6 * S + 17] ^= 1 << 14
    else:
        unit["full_out"][0][W * S - 1] ^= 1
    with pytest.raises(AssertionError):
        full_parity.check_unit_every_element(ora, unit, rb, re, 1, regen, "cpu", piece=700)
