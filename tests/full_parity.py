"""Every output of a full-size unit against the oracle, on all host cores.

The oracle's shard_step is the plain definition of one unit's step. A piece
of n elements taken at the same offset from every position's slice is itself
a unit step of padded length F * n with the same W and F (the fold, Adam and
the cast are elementwise; the gather is a copy), so the oracle runs on pieces,
one host thread per core (the C oracle holds no interpreter lock), and every
element of every output of the device step is compared with it bit for bit.

Inputs come from the seeded generator only: the gradient rows and the other
ranks' shards are inputs the step does not modify, so they are read back from
the device; the optimizer state the step updated in place is drawn again by
the device generator (`regen`) at the same positions.
"""
from __future__ import annotations

import concurrent.futures as cf
import os

import numpy as np

import gpu_util as gu


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def _h16(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def _h32(t) -> np.ndarray:
    return t.cpu().numpy()


def state_regen(wl, u, P):
    """regen for the workload builders' state of unit u (bench.build_local_rank and
    build_all_ranks): element a of rank r's slice is flat position r * S + a of each stream."""
    import torch

    import synth
    from synth import workloads as wls

    S = None

    def regen(name, r, a, n):
        t = torch.empty(n, device="cuda")
        idx0 = r * S + a
        if name == "master":
            synth.fill_(t, wls.key_master(wl, u), wl.sigma_master, idx0=idx0, n_valid=P)
        elif wl.sigma_state:
            key = wls.key_exp_avg(wl, u) if name == "exp_avg" else wls.key_exp_avg_sq(wl, u)
            synth.fill_(t, key, wl.sigma_state, idx0=idx0, absval=True, n_valid=P)
        else:
            t.zero_()
        return t

    def bind(shard_numel):
        nonlocal S
        S = shard_numel
        return regen

    return bind


def check_unit_every_element(ora, unit, rank_begin, rank_end, step, regen, what, piece=1 << 20, hp=None):
    """Compares every element a fused step wrote for one unit (F = W, owned ranks
    [rank_begin, rank_end), group 0) with the oracle's shard_step.

    unit:  the device arguments of the step (layout, grads, master / exp_avg / exp_avg_sq
           per owned rank, other_shards by rank or None, full_out per group).
    regen: regen(name, r, a, n) -> a CUDA fp32 tensor holding the pre-step value of state
           `name` ("master", "exp_avg", "exp_avg_sq") of rank r at shard elements [a, a + n).
    hp:    the Adam hyper-parameters of the step (lr, beta1, beta2, eps), gpu_util.HP if None.
    Returns the number of elements compared."""
    lay = unit["layout"]
    W, F, S = lay.world_size, lay.shard_factor, lay.shard_numel
    assert F == W, "pieces of F = W steps only"
    owned = list(range(rank_begin, rank_end))
    hp = dict(gu.HP if hp is None else hp)
    cores = host_cores()
    batch = cores * piece  # shard elements per round of host work
    compared = 0
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        for a0 in range(0, S, batch):
            nb = min(batch, S - a0)
            # inputs: gradient rows at every position's slice, state drawn again, other shards
            # (a rank's step reads only its own position's slice of the rows)
            g = [{r: _h16(unit["grads"][k][r * S + a0:r * S + a0 + nb]) for r in owned} for k in range(W)]
            st0 = {name: [_h32(regen(name, r, a0, nb)) for r in owned]
                   for name in ("master", "exp_avg", "exp_avg_sq")}
            oth = [None if (r in owned or unit["other_shards"] is None) else
                   _h16(unit["other_shards"][r][a0:a0 + nb]) for r in range(W)]
            # outputs of the device step
            got = {name: [_h32(unit[name][i][a0:a0 + nb]) for i in range(len(owned))]
                   for name in ("master", "exp_avg", "exp_avg_sq")}
            full = unit["full_out"][0]
            got_full = [_h16(full[p * S + a0:p * S + a0 + nb]) for p in range(F)]

            def oracle_piece(i0):
                n = min(piece, nb - i0)
                rows = np.zeros((W, F * n), np.uint16)  # slices of non-owned positions stay unread
                for k in range(W):
                    for r in owned:
                        rows[k, r * n:(r + 1) * n] = g[k][r][i0:i0 + n]
                st = {name: [x[i0:i0 + n].copy() for x in st0[name]] for name in st0}
                others = [None if o is None else o[i0:i0 + n].copy() for o in oth]
                out = [np.zeros(F * n, np.uint16)]
                ora.shard_step(list(rows), F, rank_begin, rank_end, st["master"], st["exp_avg"],
                               st["exp_avg_sq"], others if unit["other_shards"] is not None else None,
                               out, step=step, **hp)
                return i0, n, st, out[0]

            for i0, n, st, out in pool.map(oracle_piece, range(0, nb, piece)):
                at = "%s, shard elements [%d, %d)" % (what, a0 + i0, a0 + i0 + n)
                for name in ("master", "exp_avg", "exp_avg_sq"):
                    for i, r in enumerate(owned):
                        gu.assert_same_bits(got[name][i][i0:i0 + n], st[name][i], "%s rank %d %s" % (name, r, at))
                for p in range(F):
                    gu.assert_same_bits(got_full[p][i0:i0 + n], out[p * n:(p + 1) * n],
                                        "full slice %d %s" % (p, at))
            compared += nb
    return compared
