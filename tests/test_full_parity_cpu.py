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


def _unit(ora, W, rank_begin, rank_end, P, step, seed, F=None):
    F = W if F is None else F
    R = W // F
    rng = np.random.default_rng(seed)
    offs, _, padded, S = ora.flatten_layout([P], W, F)
    bf = lambda x: ora.bf16_rne(x.astype(np.float32))  # noqa: E731
    grads = [bf(rng.standard_normal(padded) * 1e-3) for _ in range(W)]
    owned = list(range(rank_begin, rank_end))
    pre = {name: [(np.abs(rng.standard_normal(S)) * 1e-4 if name != "master" else rng.standard_normal(S) * 0.02)
                  .astype(np.float32) for _ in owned] for name in ("master", "exp_avg", "exp_avg_sq")}
    groups = {r // F for r in owned}
    local = any(g * F + p not in owned for g in groups for p in range(F))
    others = [None if r in owned else bf(rng.standard_normal(S) * 0.02) for r in range(W)] if local else None
    post = {name: [x.copy() for x in pre[name]] for name in pre}
    full = [np.zeros(padded, np.uint16) for _ in range(R)]
    ora.shard_step(grads, F, rank_begin, rank_end, post["master"], post["exp_avg"], post["exp_avg_sq"],
                   others, full, step=step, **HP)

    class Lay:
        world_size, shard_factor, shard_numel = W, F, S

    t16 = lambda a: torch.from_numpy(a.view(np.int16).copy())  # noqa: E731
    unit = dict(layout=Lay, grads=[t16(g) for g in grads],
                master=[torch.from_numpy(x) for x in post["master"]],
                exp_avg=[torch.from_numpy(x) for x in post["exp_avg"]],
                exp_avg_sq=[torch.from_numpy(x) for x in post["exp_avg_sq"]],
                other_shards=None if others is None else [None if o is None else t16(o) for o in others],
                full_out=[t16(f) for f in full])

    def regen(name, r, a, n):
        return torch.from_numpy(pre[name][owned.index(r)][a:a + n].copy())

    return unit, regen, S


@pytest.mark.parametrize("W,F,rb,re", [(8, 8, 3, 4), (4, 4, 0, 4), (8, 8, 0, 8), (8, 2, 0, 8), (16, 4, 0, 16),
                                        (8, 2, 2, 5), (16, 1, 5, 6)])
def test_pieces_equal_the_whole_unit(ora, W, F, rb, re):
    """Full sharding and hybrid groups, all ranks and local rank ranges; pieces of 700
    elements (rounded down to a multiple of W / F) leave a shorter last piece."""
    unit, regen, S = _unit(ora, W, rb, re, W * 5000 + 3, step=2, seed=W + rb + 100 * F, F=F)
    assert full_parity.check_unit_every_element(ora, unit, rb, re, 2, regen, "cpu", piece=700) == S


def test_a_flipped_bit_in_a_second_replica_group_is_reported(ora):
    W, F = 8, 2
    unit, regen, S = _unit(ora, W, 0, W, W * 5000 + 3, step=1, seed=8, F=F)
    unit["full_out"][3][S + 99] ^= 1  # group 3, position 1
    with pytest.raises(AssertionError):
        full_parity.check_unit_every_element(ora, unit, 0, W, 1, regen, "cpu", piece=700)
    unit["full_out"][3][S + 99] ^= 1
    unit["exp_avg"][5].view(torch.int32)[S - 1] ^= 1 << 30  # rank 5: group 2, position 1, last element
    with pytest.raises(AssertionError):
        full_parity.check_unit_every_element(ora, unit, 0, W, 1, regen, "cpu", piece=700)


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
