"""GPU parity of every entry point against the CPU oracle, element by element.

Inputs are seeded draws made on the host (synth), uploaded, and given to both
sides. Sizes span several 2048-element chunks plus ragged tails; odd world
sizes and shard lengths exercise the misaligned (scalar) path. The method's
tolerance is asserted (fp32 within 1e-6 relative, bf16 within 1 ulp; layout,
pack, reduce-scatter and all-gather bit-exact), and on top of it the design
target that every output is bit-identical.
"""
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


def _inputs(key_base, W, F, P, padded, sigma_state, step=1, sigma_grad=1e-2):
    S = padded // F
    master = gu.host_normal(synth.stream_key(key_base, 1), padded, 0.02, n_valid=P)
    m = gu.host_normal(synth.stream_key(key_base, 2), padded, sigma_state, absval=True, n_valid=P)
    v = gu.host_normal(synth.stream_key(key_base, 3), padded, sigma_state, absval=True, n_valid=P)
    grads = [gu.host_normal(synth.stream_key(key_base, 4, k, step), padded, sigma_grad, n_valid=P,
                            bf16=True) for k in range(W)]
    others = [gu.host_normal(synth.stream_key(key_base, 5), S, 0.02, idx0=(r % F) * S, bf16=True)
              for r in range(W)]
    return master, m, v, grads, others


def run_step_case(ora, W, F, numels, rank_begin, rank_end, sigma_state=1e-4, step=1,
                  state_views=False, key_base=0, check_guard=True):
    torch = gu.torch()
    lay, offs = fs.fsdp_flatten_layout(numels, W, F)
    o_offs, P, padded, S = ora.flatten_layout(numels, W, F)
    assert offs == o_offs.tolist() and (lay.padded_numel, lay.shard_numel) == (padded, S)
    R = W // F
    master, m, v, grads, others = _inputs(key_base, W, F, P, padded, sigma_state, step)
    owned = list(range(rank_begin, rank_end))
    groups = sorted({r // F for r in owned})
    local = any(g * F + p not in owned for g in groups for p in range(F))
    # ---- oracle
    sl = lambda a, r: a[(r % F) * S:(r % F + 1) * S].copy()  # noqa: E731
    om = [sl(master, r) for r in owned]
    oe = [sl(m, r) for r in owned]
    ov = [sl(v, r) for r in owned]
    ofull = [np.zeros(padded, np.uint16) for _ in range(R)]
    ora.shard_step(grads, F, rank_begin, rank_end, om, oe, ov, others if local else None, ofull,
                   step=step, **gu.HP)
    # ---- device
    g_d = [gu.to_dev(g) for g in grads]
    if state_views:
        # one flat buffer per replica; a rank's state is a view at its position
        flat = {}
        for r in owned:
            g = r // F
            if g not in flat:
                flat[g] = (gu.to_dev(master), gu.to_dev(m), gu.to_dev(v))
        md = [flat[r // F][0][(r % F) * S:(r % F + 1) * S] for r in owned]
        ed = [flat[r // F][1][(r % F) * S:(r % F + 1) * S] for r in owned]
        vd = [flat[r // F][2][(r % F) * S:(r % F + 1) * S] for r in owned]
    else:
        md = [gu.to_dev(sl(master, r)) for r in owned]
        ed = [gu.to_dev(sl(m, r)) for r in owned]
        vd = [gu.to_dev(sl(v, r)) for r in owned]
    guard = 4096
    full_whole = [gu.guarded(padded, torch.int16, 0x5A5A, guard) for _ in range(R)]
    full_d = [fw[1] for fw in full_whole]
    oth_d = [gu.to_dev(o) for o in others] if local else None
    fs.fsdp_shard_step(g_d, lay, rank_begin, rank_end, md, ed, vd, oth_d, full_d,
                       gu.adam_hyper(step))
    torch.cuda.synchronize()
    for i, r in enumerate(owned):
        for got, want, what in ((md[i], om[i], "master"), (ed[i], oe[i], "exp_avg"),
                                (vd[i], ov[i], "exp_avg_sq")):
            g = gu.to_host(got)
            gu.assert_f32_close(g, want, "%s rank %d" % (what, r))
            gu.assert_same_bits(g, want, "%s rank %d" % (what, r))
    for g in groups:
        got = gu.to_host(full_d[g])
        gu.assert_bf16_close(got, ofull[g], "full group %d" % g)
        gu.assert_same_bits(got, ofull[g], "full group %d" % g)
        if check_guard:
            assert gu.canaries_intact(full_whole[g][0], padded, 0x5A5A, guard), "write outside full_out"
    return lay


# ----------------------------------------------------------------- tiny MLP

def test_tiny_mlp_three_steps(ora):
    """Tiny MLP unit, W = 4, three steps t = 1..3 from m = v = 0 with fresh grads each step."""
    torch = gu.torch()
    wl = wls.TINY_MLP
    W = wl.world_size
    numels = wls.numels(wl.units[0])
    lay, offs = fs.fsdp_flatten_layout(numels, W)
    padded, S, P = lay.padded_numel, lay.shard_numel, lay.numel
    # flatten the four tensors on the device (a2) and check against the oracle's pack
    tensors = [synth.normal_f32(synth.stream_key(0, 1, synth.KIND_TENSOR, i), n, wl.sigma_master)
               for i, n in enumerate(numels)]
    flat_d = torch.empty(padded, device="cuda")
    fs.fsdp_pack_flat([gu.to_dev(t) for t in tensors], lay, offs, flat_d)
    flat_o = ora.pack(tensors, padded)
    gu.assert_same_bits(gu.to_host(flat_d), flat_o, "packed master")
    md = [flat_d[r * S:(r + 1) * S] for r in range(W)]  # shards as views of the flat master
    ed = [torch.zeros(S, device="cuda") for _ in range(W)]
    vd = [torch.zeros(S, device="cuda") for _ in range(W)]
    full_d = torch.zeros(padded, dtype=torch.int16, device="cuda")
    om = [flat_o[r * S:(r + 1) * S].copy() for r in range(W)]
    oe = [np.zeros(S, np.float32) for _ in range(W)]
    ov = [np.zeros(S, np.float32) for _ in range(W)]
    for step in range(1, wl.steps + 1):
        grads = [synth.normal_bf16(wls.key_grad(wl, 0, k, step), padded, wl.sigma_grad, n_valid=P)
                 for k in range(W)]
        ofull = [np.zeros(padded, np.uint16)]
        ora.shard_step(grads, W, 0, W, om, oe, ov, None, ofull, step=step, **gu.HP)
        fs.fsdp_shard_step([gu.to_dev(g) for g in grads], lay, 0, W, md, ed, vd, None, [full_d],
                           gu.adam_hyper(step))
        torch.cuda.synchronize()
        for r in range(W):
            gu.assert_same_bits(gu.to_host(md[r]), om[r], "master r%d t%d" % (r, step))
            gu.assert_same_bits(gu.to_host(ed[r]), oe[r], "exp_avg r%d t%d" % (r, step))
            gu.assert_same_bits(gu.to_host(vd[r]), ov[r], "exp_avg_sq r%d t%d" % (r, step))
        gu.assert_same_bits(gu.to_host(full_d), ofull[0], "full t%d" % step)
    # unflatten the updated master back into tensors (a2 inverse)
    outs = [torch.empty(n, device="cuda") for n in numels]
    fs.fsdp_unpack_flat(flat_d, lay, offs, outs)
    back = ora.unpack(np.concatenate(om), [(n,) for n in numels])
    for a, b in zip(outs, back):
        gu.assert_same_bits(gu.to_host(a), b, "unpacked tensor")


# ------------------------------------------------------ ragged / misaligned

@pytest.mark.parametrize("W", [1, 2, 3, 4, 5, 7, 8, 16])
@pytest.mark.parametrize("P", [1, 13, 2047, 2049, 40961])
def test_all_ranks_ragged(ora, W, P):
    run_step_case(ora, W, W, [P], 0, W, step=2, key_base=W * 100000 + P)


@pytest.mark.parametrize("W,P", [(4, 2608), (3, 9001), (8, 65539), (16, 33333)])
def test_all_ranks_state_views(ora, W, P):
    """Shards as views of one flat master: misaligned slices take the scalar path."""
    numels = [P // 3, P - P // 3 - 5, 5]
    run_step_case(ora, W, W, numels, 0, W, state_views=True, key_base=7 + P)


def test_max_world_size(ora):
    run_step_case(ora, 64, 64, [64 * 300 + 17], 0, 64, key_base=64)


def test_large_step_count(ora):
    run_step_case(ora, 8, 8, [8 * 2048 * 3 + 5], 0, 8, step=1000000, key_base=99)


# ---------------------------------------------------------- local-rank mode

@pytest.mark.parametrize("rank", [0, 3, 7])
def test_local_rank(ora, rank):
    run_step_case(ora, 8, 8, [8 * 5000 + 3], rank, rank + 1, key_base=500 + rank)


def test_local_rank_range(ora):
    run_step_case(ora, 8, 8, [8 * 4096], 2, 6, key_base=600)


# ------------------------------------------------------------------ hybrid

@pytest.mark.parametrize("F", [1, 2, 4, 8, 16])
def test_hybrid_all_ranks(ora, F):
    run_step_case(ora, 16, F, [16 * 3000 + 9], 0, 16, key_base=700)


@pytest.mark.parametrize("W,F,P", [(4, 2, 4 * 5000 + 3), (4, 1, 4 * 2048 * 3 + 1), (8, 2, 8 * 3001 + 5),
                                   (8, 1, 8 * 2048 + 7), (3, 1, 3 * 4097 + 2), (5, 1, 5 * 777),
                                   (64, 2, 64 * 129 + 63), (2, 2, 2 * 2048 * 5)])
def test_split_mapping_launches(ora, W, F, P):
    """Launches the host runs with the split element mapping (2 x replicas per position
    >= W): every fixed-W instantiation and the generic one, ragged last chunks included."""
    assert 2 * (W // F) >= W
    run_step_case(ora, W, F, [P], 0, W, step=3, key_base=1100 + 10 * W + F)


@pytest.mark.parametrize("W,F", [(2, 2), (8, 2), (3, 1)])
def test_split_mapping_state_views(ora, W, F):
    """The split mapping on shards that are views of one flat master (misaligned ones take
    the scalar path beside aligned ones)."""
    P = W * 3000 + 1  # S = W * 3001 / F: odd positions of the views start off 16-byte alignment
    run_step_case(ora, W, F, [P // 3, P - P // 3 - 5, 5], 0, W, state_views=True, key_base=1200 + W + F)


@pytest.mark.parametrize("F,rb,re", [(4, 5, 6), (4, 4, 8), (2, 0, 3), (8, 6, 10)])
def test_hybrid_local(ora, F, rb, re):
    run_step_case(ora, 16, F, [16 * 2500 + 1], rb, re, key_base=800 + F)


def test_hybrid_identical_across_F():
    """All F give bit-identical updated parameters (global-order fold)."""
    torch = gu.torch()
    W, P = 16, 16 * 4099
    lay0, _ = fs.fsdp_flatten_layout([P], W, W)
    padded = lay0.padded_numel
    master, m, v, grads, _ = _inputs(900, W, W, P, padded, 1e-4)
    g_d = [gu.to_dev(g) for g in grads]
    results = {}
    for F in (1, 2, 4, 8, 16):
        lay, _ = fs.fsdp_flatten_layout([P], W, F)
        S = lay.shard_numel
        R = W // F
        md = [gu.to_dev(master[(r % F) * S:(r % F + 1) * S]) for r in range(W)]
        ed = [gu.to_dev(m[(r % F) * S:(r % F + 1) * S]) for r in range(W)]
        vd = [gu.to_dev(v[(r % F) * S:(r % F + 1) * S]) for r in range(W)]
        full = [torch.zeros(padded, dtype=torch.int16, device="cuda") for _ in range(R)]
        fs.fsdp_shard_step(g_d, lay, 0, W, md, ed, vd, None, full, gu.adam_hyper(1))
        torch.cuda.synchronize()
        flat = np.concatenate([gu.to_host(x) for x in md[:F]])
        for r in range(W):
            gu.assert_same_bits(gu.to_host(md[r]), flat[(r % F) * S:(r % F + 1) * S], "replica")
        for g in range(R):
            gu.assert_same_bits(gu.to_host(full[g]), gu.to_host(full[0]), "group full buffers")
        results[F] = (flat, gu.to_host(full[0]))
    for F in results:
        gu.assert_same_bits(results[F][0], results[16][0], "master F=%d vs F=16" % F)
        gu.assert_same_bits(results[F][1], results[16][1], "full F=%d vs F=16" % F)


# ------------------------------------------------------------- unfused path

@pytest.mark.parametrize("W,F,P", [(4, 4, 2608), (8, 8, 70000), (5, 5, 12345), (16, 4, 16 * 999)])
def test_unfused_matches_oracle_and_fused(ora, W, F, P):
    torch = gu.torch()
    lay, _ = fs.fsdp_flatten_layout([P], W, F)
    padded, S = lay.padded_numel, lay.shard_numel
    master, m, v, grads, _ = _inputs(1000 + P, W, F, P, padded, 1e-4)
    g_d = [gu.to_dev(g) for g in grads]
    shards = []
    for p in range(F):
        # a3
        gs = torch.empty(S, device="cuda")
        fs.fsdp_reduce_scatter(g_d, lay, p, gs)
        want = ora.reduce_scatter(grads, F, p)
        gu.assert_same_bits(gu.to_host(gs), want, "reduce_scatter position %d" % p)
        # a4 + a5
        sl = slice(p * S, (p + 1) * S)
        md, ed, vd = gu.to_dev(master[sl]), gu.to_dev(m[sl]), gu.to_dev(v[sl])
        bf = torch.empty(S, dtype=torch.int16, device="cuda")
        fs.fsdp_adam_shard_step(md, ed, vd, gs, gu.adam_hyper(1), bf)
        om, oe, ov = master[sl].copy(), m[sl].copy(), v[sl].copy()
        obf = ora.adam(om, oe, ov, want, step=1, **gu.HP)
        gu.assert_f32_close(gu.to_host(md), om, "adam master")
        gu.assert_same_bits(gu.to_host(md), om, "adam master")
        gu.assert_same_bits(gu.to_host(ed), oe, "adam exp_avg")
        gu.assert_same_bits(gu.to_host(vd), ov, "adam exp_avg_sq")
        gu.assert_same_bits(gu.to_host(bf), obf, "adam bf16")
        shards.append(bf)
    # a6
    full = torch.zeros(padded, dtype=torch.int16, device="cuda")
    fs.fsdp_all_gather(shards, lay, full)
    want_full = ora.all_gather([gu.to_host(s) for s in shards])
    gu.assert_same_bits(gu.to_host(full), want_full, "all_gather")
    # fused equals the three unfused launches
    md = [gu.to_dev(master[(r % F) * S:(r % F + 1) * S]) for r in range(W)]
    ed = [gu.to_dev(m[(r % F) * S:(r % F + 1) * S]) for r in range(W)]
    vd = [gu.to_dev(v[(r % F) * S:(r % F + 1) * S]) for r in range(W)]
    fulls = [torch.zeros(padded, dtype=torch.int16, device="cuda") for _ in range(W // F)]
    fs.fsdp_shard_step(g_d, lay, 0, W, md, ed, vd, None, fulls, gu.adam_hyper(1))
    gu.assert_same_bits(gu.to_host(fulls[0]), want_full, "fused vs unfused")


def test_all_gather_in_place_views(ora):
    """Shards that already are views of the full buffer are left in place."""
    torch = gu.torch()
    W, P = 8, 8 * 1001
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S = lay.shard_numel
    host = synth.normal_bf16(synth.stream_key(3, 3), lay.padded_numel, 0.02)
    full = gu.to_dev(host)
    shards = [full[k * S:(k + 1) * S] for k in range(W)]
    fs.fsdp_all_gather(shards, lay, full)
    torch.cuda.synchronize()
    gu.assert_same_bits(gu.to_host(full), host, "in-place gather")


# ------------------------------------------------------------ pack / unpack

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_pack_unpack_ragged(ora, dtype):
    torch = gu.torch()
    numels = [3, 5, 1000, 7, 4096, 1, 0, 33333]
    for W in (1, 3, 8):
        lay, offs = fs.fsdp_flatten_layout(numels, W)
        if dtype == "f32":
            hs = [synth.normal_f32(synth.stream_key(4, i), n, 1.0) for i, n in enumerate(numels)]
            tdt = torch.float32
        else:
            hs = [synth.normal_bf16(synth.stream_key(4, i), n, 1.0) for i, n in enumerate(numels)]
            tdt = torch.int16
        ds = [gu.to_dev(h) if h.size else torch.empty(0, dtype=tdt, device="cuda") for h in hs]
        whole, flat = gu.guarded(lay.padded_numel, tdt, 77)
        fs.fsdp_pack_flat(ds, lay, offs, flat)
        want = ora.pack(hs, lay.padded_numel)
        gu.assert_same_bits(gu.to_host(flat), want, "pack W=%d" % W)
        assert gu.canaries_intact(whole, lay.padded_numel, 77)
        outs = [torch.full((n,), 5, dtype=tdt, device="cuda") for n in numels]
        fs.fsdp_unpack_flat(flat, lay, offs, outs)
        for a, b in zip(outs, hs):
            gu.assert_same_bits(gu.to_host(a), b, "unpack")


# --------------------------------------------------------------- grouped

def test_grouped_scaled_gpt2(ora):
    """Several units of different sizes in one grouped launch == the oracle per unit."""
    torch = gu.torch()
    W = 8
    block = [(64,), (64,), (64, 192), (192,), (64, 64), (64,), (64,), (64,), (64, 256), (256,),
             (256, 64), (64,)]
    root = [(1000, 64), (128, 64), (64,), (64,)]
    units_shapes = [block] * 12 + [root]
    units, checks = [], []
    for u, shapes in enumerate(units_shapes):
        numels = wls.numels(shapes)
        lay, _ = fs.fsdp_flatten_layout(numels, W)
        P, padded, S = lay.numel, lay.padded_numel, lay.shard_numel
        master, m, v, grads, _ = _inputs(2000 + u, W, W, P, padded, 1e-4)
        om = [master[r * S:(r + 1) * S].copy() for r in range(W)]
        oe = [m[r * S:(r + 1) * S].copy() for r in range(W)]
        ov = [v[r * S:(r + 1) * S].copy() for r in range(W)]
        ofull = [np.zeros(padded, np.uint16)]
        ora.shard_step(grads, W, 0, W, om, oe, ov, None, ofull, step=1, **gu.HP)
        d = dict(layout=lay, grads=[gu.to_dev(g) for g in grads],
                 master=[gu.to_dev(master[r * S:(r + 1) * S]) for r in range(W)],
                 exp_avg=[gu.to_dev(m[r * S:(r + 1) * S]) for r in range(W)],
                 exp_avg_sq=[gu.to_dev(v[r * S:(r + 1) * S]) for r in range(W)],
                 other_shards=None,
                 full_out=[torch.zeros(padded, dtype=torch.int16, device="cuda")])
        units.append(d)
        checks.append((om, oe, ov, ofull[0]))
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(1))
    torch.cuda.synchronize()
    for d, (om, oe, ov, of) in zip(units, checks):
        for r in range(W):
            gu.assert_same_bits(gu.to_host(d["master"][r]), om[r], "grouped master")
            gu.assert_same_bits(gu.to_host(d["exp_avg"][r]), oe[r], "grouped exp_avg")
            gu.assert_same_bits(gu.to_host(d["exp_avg_sq"][r]), ov[r], "grouped exp_avg_sq")
        gu.assert_same_bits(gu.to_host(d["full_out"][0]), of, "grouped full")


def test_grouped_many_units_split_launches(ora):
    """More units than one descriptor table holds: split into several launches, same result."""
    torch = gu.torch()
    W = 16
    units, checks = [], []
    for u in range(40):  # 40 units x 16 positions = 640 segments > one table
        P = 16 * 64 + u
        lay, _ = fs.fsdp_flatten_layout([P], W)
        padded, S = lay.padded_numel, lay.shard_numel
        master, m, v, grads, _ = _inputs(3000 + u, W, W, P, padded, 0.0)
        om = [master[r * S:(r + 1) * S].copy() for r in range(W)]
        oe = [m[r * S:(r + 1) * S].copy() for r in range(W)]
        ov = [v[r * S:(r + 1) * S].copy() for r in range(W)]
        ofull = [np.zeros(padded, np.uint16)]
        ora.shard_step(grads, W, 0, W, om, oe, ov, None, ofull, step=1, **gu.HP)
        units.append(dict(layout=lay, grads=[gu.to_dev(g) for g in grads],
                          master=[gu.to_dev(x) for x in (master[r * S:(r + 1) * S] for r in range(W))],
                          exp_avg=[torch.zeros(S, device="cuda") for _ in range(W)],
                          exp_avg_sq=[torch.zeros(S, device="cuda") for _ in range(W)],
                          full_out=[torch.zeros(padded, dtype=torch.int16, device="cuda")]))
        checks.append((om, ofull[0]))
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(1))
    torch.cuda.synchronize()
    for d, (om, of) in zip(units, checks):
        for r in range(W):
            gu.assert_same_bits(gu.to_host(d["master"][r]), om[r], "split master")
        gu.assert_same_bits(gu.to_host(d["full_out"][0]), of, "split full")


# ------------------------------------------------------------- edge cases

def test_empty_unit_is_noop():
    torch = gu.torch()
    lay, _ = fs.fsdp_flatten_layout([0], 4)
    assert lay.padded_numel == 0
    full = torch.full((8,), 3, dtype=torch.int16, device="cuda")
    e = torch.empty(0, device="cuda")
    g = [torch.empty(0, dtype=torch.int16, device="cuda")] * 4
    fs.fsdp_shard_step(g, lay, 0, 4, [e] * 4, [e] * 4, [e] * 4, None, [full], gu.adam_hyper(1))
    fs.fsdp_shard_step_grouped([], 0, 4, gu.adam_hyper(1))
    fs.fsdp_adam_shard_step(e, e, e, e, gu.adam_hyper(1), n=0)
    torch.cuda.synchronize()
    assert (full.cpu() == 3).all()


def test_deterministic_repeat(ora):
    torch = gu.torch()
    W, P = 8, 8 * 20000 + 3
    lay, _ = fs.fsdp_flatten_layout([P], W)
    padded, S = lay.padded_numel, lay.shard_numel
    master, m, v, grads, _ = _inputs(4000, W, W, P, padded, 1e-4)
    g_d = [gu.to_dev(g) for g in grads]
    outs = []
    for _ in range(2):
        md = [gu.to_dev(master[r * S:(r + 1) * S]) for r in range(W)]
        ed = [gu.to_dev(m[r * S:(r + 1) * S]) for r in range(W)]
        vd = [gu.to_dev(v[r * S:(r + 1) * S]) for r in range(W)]
        full = torch.zeros(padded, dtype=torch.int16, device="cuda")
        fs.fsdp_shard_step(g_d, lay, 0, W, md, ed, vd, None, [full], gu.adam_hyper(5))
        outs.append((torch.cat(md).cpu(), full.cpu()))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


def test_device_aliasing_rejected():
    torch = gu.torch()
    W, P = 4, 4 * 512
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S = lay.shard_numel
    g = [torch.zeros(P, dtype=torch.int16, device="cuda") for _ in range(W)]
    st = [torch.zeros(S, device="cuda") for _ in range(3 * W)]
    full = torch.zeros(P, dtype=torch.int16, device="cuda")
    with pytest.raises(fs.FsdpError) as e:
        fs.fsdp_shard_step(g, lay, 0, W, st[:W], st[:W], st[2 * W:], None, [full], gu.adam_hyper(1))
    assert e.value.status == fs.FSDP_EALIAS
    with pytest.raises(fs.FsdpError) as e:
        fs.fsdp_shard_step(g, lay, 0, W, st[:W], st[W:2 * W], st[2 * W:], None, [g[1]],
                           gu.adam_hyper(1))
    assert e.value.status == fs.FSDP_EALIAS


# ------------------------------------------------------------------ cast

def test_cast_all_fp32_patterns(ora):
    """a5 over every fp32 bit pattern: Adam with g = m = v = 0 leaves p unchanged, so the
    bf16 output is the cast of p. Non-NaN patterns match the oracle bit for bit; NaN stays NaN."""
    torch = gu.torch()
    n = 1 << 27
    g = torch.zeros(n, device="cuda")
    mm = torch.zeros(n, device="cuda")
    vv = torch.zeros(n, device="cuda")
    bf = torch.empty(n, dtype=torch.int16, device="cuda")
    base = torch.arange(n, dtype=torch.int64, device="cuda")
    for part in range(1 << 5):
        bits = (base + part * n).to(torch.int64)
        p = (bits - ((bits >> 31) << 32)).to(torch.int32).view(torch.float32)  # wrap to int32
        mm.zero_()
        vv.zero_()
        fs.fsdp_adam_shard_step(p, mm, vv, g, gu.adam_hyper(1), bf)
        host_p = p.cpu().numpy()
        got = bf.cpu().numpy().view(np.uint16)
        want = ora.bf16_rne(host_p)
        nan = np.isnan(host_p)
        assert got[~nan].tobytes() == want[~nan].tobytes(), "cast part %d" % part
        assert np.all(np.isnan((got[nan].astype(np.uint32) << 16).view(np.float32)))
