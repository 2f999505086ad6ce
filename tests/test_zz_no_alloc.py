"""The allocation-free pipelined step against the ordinary one.

fsdp_pipeline_step_noalloc serves callers that cannot allocate device memory
when they step the optimizer (their memory belongs to another allocator, or
a cudaMalloc there could synchronize the device). It must give the same
results as fsdp_pipeline_step with a caller-owned staging pool, call after
call, since every call reuses the library's fixed staging array. This file is
collected last so that a run stopping at its first failure has run every
other test before it; it also passes when run on its own.

The cases vary the world size and the number of slots: W = 8 with two slots;
W = 2 with one slot and a first unit of more than 4 M shard elements, which
moves through the shared array in pieces; W = 4 with three slots, where the
largest unit's padded length is not a multiple of 8 elements and a smaller,
aligned unit lands in slot 1.
"""
import pytest

import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")

CASES = {
    # name: (W, rank, n_slots, unit sizes P)
    "w8_two_slots": (8, 5, 2, [7087872, 8 * 100003, 8 * 4096 + 3]),
    "w2_one_slot_pieces": (2, 1, 1, [2 * 5_000_001, 2 * 65536]),
    "w4_three_slots_ragged": (4, 2, 3, [4 * 1_000_001, 4 * 65536, 4 * 3001 + 1]),
}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _units(W, rank, sizes, base):
    torch = gu.torch()
    units = []
    for u, P in enumerate(sizes):
        lay, _ = fs.fsdp_flatten_layout([P], W)
        S, padded = lay.shard_numel, lay.padded_numel
        key = lambda *f: synth.stream_key(base, u, *f)  # noqa: E731
        units.append(dict(
            layout=lay,
            master=gu.dev_normal(key(1), S, 0.02, idx0=rank * S, n_valid=P),
            exp_avg=gu.dev_normal(key(2), S, 1e-4, idx0=rank * S, absval=True, n_valid=P),
            exp_avg_sq=gu.dev_normal(key(3), S, 1e-4, idx0=rank * S, absval=True, n_valid=P),
            other_shards=[None if k == rank else gu.dev_normal(key(5), S, 0.02, idx0=k * S, n_valid=P, bf16=True)
                          for k in range(W)],
            full_out=torch.zeros(padded, dtype=torch.int16, device="cuda"),
            shard_out=torch.zeros(S, dtype=torch.int16).pin_memory()))
    return units


def _set_grads(units, W, rank, base, step):
    """The step's gradient slices, drawn by the device generator into pinned host memory."""
    torch = gu.torch()
    for u, unit in enumerate(units):
        lay = unit["layout"]
        S, P = lay.shard_numel, lay.numel
        rows = torch.empty((W, S), dtype=torch.int16, device="cuda")
        for k in range(W):
            synth.fill_(rows[k], synth.stream_key(base, u, 4, k, step), 1e-2, idx0=rank * S, n_valid=P)
        host = torch.empty((W, S), dtype=torch.int16).pin_memory()
        host.copy_(rows)
        unit["grad_slices"] = host
    torch.cuda.synchronize()


def _copy_units(units):
    out = []
    for unit in units:
        c = dict(unit)
        for name in ("master", "exp_avg", "exp_avg_sq", "full_out"):
            c[name] = unit[name].clone()
        c["shard_out"] = unit["shard_out"].clone().pin_memory()
        out.append(c)
    return out


@pytest.mark.parametrize("case", list(CASES))
def test_noalloc_matches_pipeline_on_two_calls(case):
    torch = gu.torch()
    W, rank, n_slots, sizes = CASES[case]
    base = 9100 + 10 * list(CASES).index(case)
    ref = _units(W, rank, sizes, base)
    got = _copy_units(ref)
    slot = max(u["layout"].padded_numel for u in ref)
    slot = (slot + 7) // 8 * 8  # the caller-owned pool gets the same aligned slots
    assert n_slots * slot * 2 <= fs.NOALLOC_STAGING_BYTES
    staging = torch.empty(n_slots * slot, dtype=torch.int16, device="cuda")
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    for step in (1, 2):
        _set_grads(ref, W, rank, base, step)
        for g, r in zip(got, ref):
            g["grad_slices"] = r["grad_slices"]
        hp = gu.adam_hyper(step)
        fs.fsdp_pipeline_step(ref, rank, staging, slot, n_slots, hp, compute=compute, copy=copy)
        fs.fsdp_pipeline_step_noalloc(got, rank, n_slots, hp, compute=compute, copy=copy)
        torch.cuda.synchronize()
        for u, (g, r) in enumerate(zip(got, ref)):
            for name in ("master", "exp_avg", "exp_avg_sq"):
                a, b = gu.to_host(g[name]), gu.to_host(r[name])
                gu.assert_f32_close(a, b, "%s unit %d step %d" % (name, u, step))
                gu.assert_same_bits(a, b, "%s unit %d step %d" % (name, u, step))
            gu.assert_bf16_close(gu.to_host(g["full_out"]), gu.to_host(r["full_out"]),
                                 "full unit %d step %d" % (u, step))
            gu.assert_same_bits(g["shard_out"].numpy(), r["shard_out"].numpy(),
                                "shard_out unit %d step %d" % (u, step))


def test_noalloc_rejects_work_beyond_its_capacity():
    torch = gu.torch()
    W, rank, n_slots = 8, 5, 2
    P = fs.NOALLOC_STAGING_BYTES // 2 // n_slots + 8  # one slot's worth too large for two slots
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S = lay.shard_numel
    small = torch.zeros(8, device="cuda")
    unit = dict(layout=lay, grad_slices=small.data_ptr(), master=small.data_ptr(), exp_avg=small.data_ptr(),
                exp_avg_sq=small.data_ptr(), other_shards=[small.data_ptr()] * W, full_out=small.data_ptr(),
                shard_out=None)
    assert S > 0
    with pytest.raises(fs.FsdpError) as e:
        fs.fsdp_pipeline_step_noalloc([unit], rank, n_slots, gu.adam_hyper(1))
    assert e.value.status == fs.FSDP_ENOSPACE
    assert "%d MiB" % (fs.NOALLOC_STAGING_BYTES >> 20) in fs.fsdp_status_string(fs.FSDP_ENOSPACE)
