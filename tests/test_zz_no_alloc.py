"""The allocation-free pipelined step against the ordinary one.

fsdp_pipeline_step_noalloc serves callers that cannot allocate device memory
when they step the optimizer (their memory belongs to another allocator, or
a cudaMalloc there could synchronize the device). It must give the same
results as fsdp_pipeline_step with a caller-owned staging pool, call after
call, since every call reuses the library's fixed staging array. This file is
collected last so that a run stopping at its first failure has run every
other test before it; it also passes when run on its own.
"""
import numpy as np
import pytest

import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")

W, RANK, N_SLOTS = 8, 5, 2
SIZES = [7087872, 8 * 100003, 8 * 4096 + 3]  # a GPT-2-small block, a ragged unit, a small one


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _units(base):
    torch = gu.torch()
    units = []
    for u, P in enumerate(SIZES):
        lay, _ = fs.fsdp_flatten_layout([P], W)
        S, padded = lay.shard_numel, lay.padded_numel
        key = lambda *f: synth.stream_key(base, u, *f)  # noqa: E731
        units.append(dict(
            layout=lay,
            master=gu.dev_normal(key(1), S, 0.02, idx0=RANK * S, n_valid=P),
            exp_avg=gu.dev_normal(key(2), S, 1e-4, idx0=RANK * S, absval=True, n_valid=P),
            exp_avg_sq=gu.dev_normal(key(3), S, 1e-4, idx0=RANK * S, absval=True, n_valid=P),
            other_shards=[None if k == RANK else gu.dev_normal(key(5), S, 0.02, idx0=k * S, n_valid=P, bf16=True)
                          for k in range(W)],
            full_out=torch.zeros(padded, dtype=torch.int16, device="cuda"),
            shard_out=torch.zeros(S, dtype=torch.int16).pin_memory()))
    return units


def _set_grads(units, base, step):
    torch = gu.torch()
    for u, unit in enumerate(units):
        lay = unit["layout"]
        S, P = lay.shard_numel, lay.numel
        rows = [synth.normal_bf16(synth.stream_key(base, u, 4, k, step), S, 1e-2, idx0=RANK * S, n_valid=P)
                for k in range(W)]
        unit["grad_slices"] = torch.from_numpy(np.stack(rows).view(np.int16)).pin_memory()


def _copy_units(units):
    out = []
    for unit in units:
        c = dict(unit)
        for name in ("master", "exp_avg", "exp_avg_sq", "full_out"):
            c[name] = unit[name].clone()
        c["shard_out"] = unit["shard_out"].clone().pin_memory()
        out.append(c)
    return out


def test_noalloc_matches_pipeline_on_two_calls():
    torch = gu.torch()
    base = 9100
    ref = _units(base)
    got = _copy_units(ref)
    slot = max(u["layout"].padded_numel for u in ref)
    staging = torch.empty(N_SLOTS * slot, dtype=torch.int16, device="cuda")
    compute, copy = torch.cuda.Stream(), torch.cuda.Stream()
    for step in (1, 2):
        _set_grads(ref, base, step)
        for g, r in zip(got, ref):
            g["grad_slices"] = r["grad_slices"]
        hp = gu.adam_hyper(step)
        fs.fsdp_pipeline_step(ref, RANK, staging, slot, N_SLOTS, hp, compute=compute, copy=copy)
        fs.fsdp_pipeline_step_noalloc(got, RANK, N_SLOTS, hp, compute=compute, copy=copy)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            for name in ("master", "exp_avg", "exp_avg_sq"):
                a, b = gu.to_host(g[name]), gu.to_host(r[name])
                gu.assert_f32_close(a, b, "%s step %d" % (name, step))
                gu.assert_same_bits(a, b, "%s step %d" % (name, step))
            gu.assert_bf16_close(gu.to_host(g["full_out"]), gu.to_host(r["full_out"]), "full step %d" % step)
            gu.assert_same_bits(g["shard_out"].numpy(), r["shard_out"].numpy(), "shard_out step %d" % step)


def test_noalloc_rejects_work_beyond_its_capacity():
    torch = gu.torch()
    P = fs.NOALLOC_STAGING_BYTES // 2 // N_SLOTS + 8  # one slot's worth too large for two slots
    lay, _ = fs.fsdp_flatten_layout([P], W)
    S = lay.shard_numel
    small = torch.zeros(8, device="cuda")
    unit = dict(layout=lay, grad_slices=small.data_ptr(), master=small.data_ptr(), exp_avg=small.data_ptr(),
                exp_avg_sq=small.data_ptr(), other_shards=[small.data_ptr()] * W, full_out=small.data_ptr(),
                shard_out=None)
    assert S > 0
    with pytest.raises(fs.FsdpError) as e:
        fs.fsdp_pipeline_step_noalloc([unit], RANK, N_SLOTS, gu.adam_hyper(1))
    assert e.value.status == fs.FSDP_ENOSPACE
    assert "64 MiB" in fs.fsdp_status_string(fs.FSDP_ENOSPACE)
