"""The one-launch forms of the unfused parts against the oracle.

fsdp_reduce_scatter_ranks reduces the slices of a range of owned ranks in one
launch; fsdp_adam_shard_step_grouped updates several shards in one launch.
Every output must equal the oracle's reduce_scatter / adam of that rank or
shard bit for bit (and so the single-rank, single-shard calls). The cases
cover full sharding, hybrid groups (several ranks at one position), ragged
shard ends, shards that start off 16-byte alignment, and Adam launches (which
run the split element mapping of the LDG form) with and without the bf16
output.
"""
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


@pytest.mark.parametrize("W,F,rb,re,P", [(8, 8, 0, 8, 70000), (16, 4, 2, 11, 16 * 999 + 5), (5, 5, 1, 4, 12345),
                                         (2, 1, 0, 2, 2 * 40961), (3, 3, 2, 3, 2049 * 3 + 1)])
def test_reduce_scatter_ranks_matches_oracle(ora, W, F, rb, re, P):
    torch = gu.torch()
    lay, _ = fs.fsdp_flatten_layout([P], W, F)
    padded, S = lay.padded_numel, lay.shard_numel
    grads = [gu.host_normal(synth.stream_key(7100 + W, 4, k), padded, 1e-2, n_valid=P, bf16=True) for k in range(W)]
    g_d = [gu.to_dev(g) for g in grads]
    outs = [torch.full((S,), float("nan"), device="cuda") for _ in range(rb, re)]
    fs.fsdp_reduce_scatter_ranks(g_d, lay, rb, re, outs)
    one = torch.empty(S, device="cuda")
    for i, r in enumerate(range(rb, re)):
        want = ora.reduce_scatter(grads, F, r)
        gu.assert_same_bits(gu.to_host(outs[i]), want, "rank %d" % r)
        fs.fsdp_reduce_scatter(g_d, lay, r, one)
        gu.assert_same_bits(gu.to_host(one), want, "single-rank call, rank %d" % r)


def test_adam_grouped_matches_oracle(ora):
    """Shards of 1 to 400,003 elements in one launch; odd starting offsets put some of them
    off 16-byte alignment (the scalar path) beside aligned ones (the vector path with ragged
    last chunks); step 3 on non-zero state."""
    torch = gu.torch()
    sizes = [1, 7, 2047, 2048, 2049, 65536 + 3, 400003, 1024 + 5]
    offsets = [0, 1, 0, 3, 0, 0, 2, 0]  # elements into each buffer: non-zero offsets misalign the shard
    with_bf16 = [True, True, False, True, True, True, True, False]
    step = 3
    hp = dict(gu.HP)
    shards, want = [], []
    keep = []
    for i, (n, o) in enumerate(zip(sizes, offsets)):
        key = lambda f: synth.stream_key(7300 + i, f)  # noqa: E731
        p = gu.host_normal(key(1), n, 0.02)
        m = gu.host_normal(key(2), n, 1e-4, absval=True)
        v = gu.host_normal(key(3), n, 1e-4, absval=True)
        g = gu.host_normal(key(4), n, 1e-3)
        bufs = [torch.zeros(n + o, device="cuda") for _ in range(4)]
        for b, x in zip(bufs, (p, m, v, g)):
            b[o:].copy_(torch.from_numpy(x))
        bf = torch.zeros(n + o, dtype=torch.int16, device="cuda") if with_bf16[i] else None
        keep.append((bufs, bf))
        shards.append(dict(master=bufs[0][o:], exp_avg=bufs[1][o:], exp_avg_sq=bufs[2][o:], grad_shard=bufs[3][o:],
                           bf16_shard_out=None if bf is None else bf[o:]))
        op, om, ov = p.copy(), m.copy(), v.copy()
        obf = ora.adam(op, om, ov, g, step=step, **hp)
        want.append((op, om, ov, obf))
    fs.fsdp_adam_shard_step_grouped(shards, gu.adam_hyper(step))
    torch.cuda.synchronize()
    for i, (s, (op, om, ov, obf)) in enumerate(zip(shards, want)):
        what = "shard %d (n=%d, offset %d)" % (i, sizes[i], offsets[i])
        gu.assert_f32_close(gu.to_host(s["master"]), op, "master " + what)
        gu.assert_same_bits(gu.to_host(s["master"]), op, "master " + what)
        gu.assert_same_bits(gu.to_host(s["exp_avg"]), om, "exp_avg " + what)
        gu.assert_same_bits(gu.to_host(s["exp_avg_sq"]), ov, "exp_avg_sq " + what)
        if s["bf16_shard_out"] is not None:
            gu.assert_same_bits(gu.to_host(s["bf16_shard_out"]), obf, "bf16 " + what)
        gu.assert_same_bits(gu.to_host(s["grad_shard"]), np.ascontiguousarray(
            gu.host_normal(synth.stream_key(7300 + i, 4), sizes[i], 1e-3)), "gradient unchanged " + what)
    assert fs.fsdp_device_status() == 0
