"""The TMA form of the kernel: oracle parity, the status word, and its bounded waits.

The form is chosen by the library for W = 8 single-replica launches with
enough chunks per SM; the cases here are sized from the GPU's SM count so the
planner picks it. Inputs come from numpy's generator (any bf16/fp32 values
serve), compared element by element with the oracle.
"""
import time

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


def _tma_shard_len(align8):
    torch = gu.torch()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    S = -(-(130 * sms * 2048) // 8)  # comfortably above 128 chunks per SM over the 8 positions
    return S - S % 8 + (0 if align8 else 3)


# (align8, state_off): S a multiple of 8 or not; the state views 32-byte aligned
# (state_off 0: the consumers store a thread's 8 fp32 of an array as one 32-byte
# sector) or 16 bytes past that (4: two float4 each). With S = 3 mod 8 the rows
# of seven of the eight positions lie 2-14 bytes off alignment: the launch then
# takes the LDG form's realigned path instead (checked the same way).
@pytest.mark.parametrize("align8,state_off", [(False, 0), (True, 0), (True, 4)])
def test_tma_form_matches_oracle(ora, align8, state_off):
    torch = gu.torch()
    W = 8
    S = _tma_shard_len(align8)
    P = W * S
    lay, _ = fs.fsdp_flatten_layout([P], W)
    assert lay.shard_numel == S
    rng = np.random.default_rng(11 + align8)
    grads = [((rng.standard_normal(P, dtype=np.float32) * 1e-2).view(np.uint32) >> 16).astype(np.uint16)
             for _ in range(W)]
    master = (rng.standard_normal(P, dtype=np.float32) * 0.02)
    m = np.abs(rng.standard_normal(P, dtype=np.float32) * 1e-4)
    v = np.abs(rng.standard_normal(P, dtype=np.float32) * 1e-4)
    units = [dict(layout=lay, grads=[gu.to_dev(g) for g in grads],
                  master=[gu.to_dev_at(master[r * S:(r + 1) * S], state_off) for r in range(W)],
                  exp_avg=[gu.to_dev_at(m[r * S:(r + 1) * S], state_off) for r in range(W)],
                  exp_avg_sq=[gu.to_dev_at(v[r * S:(r + 1) * S], state_off) for r in range(W)],
                  other_shards=None, full_out=[torch.zeros(P, dtype=torch.int16, device="cuda")])]
    assert all(t.data_ptr() % 32 == 4 * state_off for t in units[0]["master"])
    assert fs.fsdp_shard_step_grouped_plan(units, 0, W) == (1, 1 if align8 else 0)
    fs.fsdp_device_status(clear=True)
    fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(4))
    torch.cuda.synchronize()
    assert fs.fsdp_device_status() == 0
    om = [master[r * S:(r + 1) * S].copy() for r in range(W)]
    oe = [m[r * S:(r + 1) * S].copy() for r in range(W)]
    ov = [v[r * S:(r + 1) * S].copy() for r in range(W)]
    ofull = [np.zeros(P, np.uint16)]
    ora.shard_step(grads, W, 0, W, om, oe, ov, None, ofull, step=4, **gu.HP)
    u = units[0]
    for r in range(W):
        gu.assert_same_bits(gu.to_host(u["master"][r]), om[r], "master r%d" % r)
        gu.assert_same_bits(gu.to_host(u["exp_avg"][r]), oe[r], "exp_avg r%d" % r)
        gu.assert_same_bits(gu.to_host(u["exp_avg_sq"][r]), ov[r], "exp_avg_sq r%d" % r)
    gu.assert_same_bits(gu.to_host(u["full_out"][0]), ofull[0], "full")


def test_bounded_wait_runs_out_and_the_context_stays_usable(ora):
    """A stage that waits for 16 bytes no copy delivers: the block gives up after the
    limit, records it in the status word and returns; later calls work normally."""
    torch = gu.torch()
    src = torch.arange(1 << 15, dtype=torch.int32, device="cuda")
    dst = torch.zeros_like(src)
    fs.fsdp_device_status(clear=True)
    t0 = time.perf_counter()
    status = fs.fsdp_selftest_wait_timeout(src, dst, 50_000_000)  # 50 ms limit
    elapsed = time.perf_counter() - t0
    assert status == 1
    assert 0.04 < elapsed < 5.0
    assert fs.fsdp_device_status() == 0  # the self-test cleared it
    # the context is intact: an ordinary step still matches the oracle
    from test_gpu_parity import run_step_case
    run_step_case(ora, 8, 8, [8 * 3000 + 1], 0, 8, key_base=31337)
    assert fs.fsdp_device_status() == 0
