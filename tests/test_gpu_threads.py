"""Host-side thread safety of the library: several threads drive it at once, each
on its own stream and buffers (the LDG form, a hybrid launch and the TMA form),
while another thread calls the host-only entry points. Every result must equal
the same calls made one after another, bit for bit."""
import threading

import pytest

import gpu_util as gu
import synth

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")
bench = pytest.importorskip("bench")

# (elements, W, F): 1472 chunks at W = 8 (LDG form), a two-replica hybrid launch,
# and 19,536 chunks at W = 8 (TMA form on a 152-SM GB300)
CASES = [(3_000_001, 8, 8), (5_000_003, 4, 2), (40_000_000, 8, 8)]
STEPS = 5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _build(n, W, F):
    torch = gu.torch()
    return bench.build_all_ranks(bench.sweep_workload(n, W), F, torch, fs, synth)


def _outputs(units):
    outs = []
    for u in units:
        for name in ("master", "exp_avg", "exp_avg_sq", "full_out"):
            outs += [t.clone() for t in u[name]]
    return outs


def _steps(units, W, stream):
    for t in range(1, STEPS + 1):
        fs.fsdp_shard_step_grouped(units, 0, W, gu.adam_hyper(t), stream=stream)


def test_concurrent_threads_match_sequential_calls():
    torch = gu.torch()
    seq = [_build(*c) for c in CASES]
    thr = [_build(*c) for c in CASES]
    streams = [torch.cuda.Stream() for _ in CASES]
    if CASES[2][1] == 8 and torch.cuda.get_device_properties(0).multi_processor_count <= 152:
        assert fs.fsdp_shard_step_grouped_plan(thr[2][0], 0, 8)[1] == 1  # the TMA form is exercised
    # one after another
    for (units, info, keep), (n, W, F), s in zip(seq, CASES, streams):
        _steps(units, W, s)
        s.synchronize()
    # all at once
    start = threading.Barrier(len(CASES) + 1)
    errors = []

    def gpu_worker(i):
        try:
            torch.cuda.set_device(0)
            start.wait()
            _steps(thr[i][0], CASES[i][1], streams[i])
            streams[i].synchronize()
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    def host_worker():
        try:
            start.wait()
            for _ in range(2000):
                lay, offs = fs.fsdp_flatten_layout([4096 * 4096, 4096, 11008 * 4096], 8)
                assert lay.padded_numel == 16781312 + 45088768 and offs[-1] == lay.numel
                acc = fs.fsdp_account(7e9, 7e9 / 32, 8, 8, 1)
                assert abs(acc["persistent_bytes"] - 14e9) < 1
        except Exception as e:
            errors.append(e)

    threads = [threading.Thread(target=gpu_worker, args=(i,)) for i in range(len(CASES))]
    threads.append(threading.Thread(target=host_worker))
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    for (a, _, _), (b, _, _), c in zip(seq, thr, CASES):
        for x, y in zip(_outputs(a), _outputs(b)):
            assert torch.equal(x.view(torch.int8), y.view(torch.int8)), "case %r" % (c,)
