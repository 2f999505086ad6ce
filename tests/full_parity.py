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
    build_all_ranks), bound to the unit's S and F: element a of the slice at position
    p = r mod F is flat position p * S + a of each stream (every replica of a position
    holds the same draws)."""
    import torch

    import synth
    from synth import workloads as wls

    def bind(S, F):
        def regen(name, r, a, n):
            t = torch.empty(n, device="cuda")
            idx0 = (r % F) * S + a
            if name == "master":
                synth.fill_(t, wls.key_master(wl, u), wl.sigma_master, idx0=idx0, n_valid=P)
            elif wl.sigma_state:
                key = wls.key_exp_avg(wl, u) if name == "exp_avg" else wls.key_exp_avg_sq(wl, u)
                synth.fill_(t, key, wl.sigma_state, idx0=idx0, absval=True, n_valid=P)
            else:
                t.zero_()
            return t
        return regen

    return bind


def check_unit_every_element(ora, unit, rank_begin, rank_end, step, regen, what, piece=1 << 20, hp=None):
    """Compares every element a fused step wrote for one unit (owned ranks
    [rank_begin, rank_end); F | W, R = W / F groups) with the oracle's shard_step.

    unit:  the device arguments of the step (layout, grads, master / exp_avg / exp_avg_sq
           per owned rank, other_shards by rank or None, full_out per group).
    regen: regen(name, r, a, n) -> a CUDA fp32 tensor holding the pre-step value of state
           `name` ("master", "exp_avg", "exp_avg_sq") of rank r at shard elements [a, a + n).
    piece: elements per oracle call, rounded down to a multiple of R (a piece's length
           F * n must split evenly over the W ranks; S is a multiple of R too).
    hp:    the Adam hyper-parameters of the step (lr, beta1, beta2, eps), gpu_util.HP if None.
    Returns the number of shard elements compared."""
    lay = unit["layout"]
    W, F, S = lay.world_size, lay.shard_factor, lay.shard_numel
    R = W // F
    owned = list(range(rank_begin, rank_end))
    positions = sorted({r % F for r in owned})
    groups = sorted({r // F for r in owned})
    local = unit["other_shards"] is not None
    piece = max(R, piece // R * R)
    hp = dict(gu.HP if hp is None else hp)
    cores = host_cores()
    batch = cores * piece  # shard elements per round of host work
    compared = 0
    with cf.ThreadPoolExecutor(max_workers=cores) as pool:
        for a0 in range(0, S, batch):
            nb = min(batch, S - a0)
            # inputs: the gradient rows at every owned position's slice (a step reads no
            # other slice of them), the state drawn again, the other ranks' shards
            g = [{p: _h16(unit["grads"][k][p * S + a0:p * S + a0 + nb]) for p in positions} for k in range(W)]
            st0 = {name: [_h32(regen(name, r, a0, nb)) for r in owned]
                   for name in ("master", "exp_avg", "exp_avg_sq")}
            oth = [None] * W
            if local:
                for grp in groups:
                    for p in range(F):
                        r = grp * F + p
                        if r not in owned:
                            oth[r] = _h16(unit["other_shards"][r][a0:a0 + nb])
            # outputs of the device step
            got = {name: [_h32(unit[name][i][a0:a0 + nb]) for i in range(len(owned))]
                   for name in ("master", "exp_avg", "exp_avg_sq")}
            got_full = {grp: [_h16(unit["full_out"][grp][p * S + a0:p * S + a0 + nb]) for p in range(F)]
                        for grp in groups}

            def oracle_piece(i0):
                # S and the piece length are multiples of R, so every piece is one too
                n = min(piece, nb - i0)
                assert n % R == 0
                rows = np.zeros((W, F * n), np.uint16)  # slices of non-owned positions stay unread
                for k in range(W):
                    for p in positions:
                        rows[k, p * n:(p + 1) * n] = g[k][p][i0:i0 + n]
                st = {name: [x[i0:i0 + n].copy() for x in st0[name]] for name in st0}
                others = [None if o is None else o[i0:i0 + n].copy() for o in oth] if local else None
                out = [np.zeros(F * n, np.uint16) for _ in range(R)]
                ora.shard_step(list(rows), F, rank_begin, rank_end, st["master"], st["exp_avg"],
                               st["exp_avg_sq"], others, out, step=step, **hp)
                return i0, n, st, out

            for i0, n, st, out in pool.map(oracle_piece, range(0, nb, piece)):
                at = "%s, shard elements [%d, %d)" % (what, a0 + i0, a0 + i0 + n)
                for name in ("master", "exp_avg", "exp_avg_sq"):
                    for i, r in enumerate(owned):
                        gu.assert_same_bits(got[name][i][i0:i0 + n], st[name][i], "%s rank %d %s" % (name, r, at))
                for grp in groups:
                    for p in range(F):
                        gu.assert_same_bits(got_full[grp][p][i0:i0 + n], out[grp][p * n:(p + 1) * n],
                                            "full group %d slice %d %s" % (grp, p, at))
            compared += nb
    return compared
