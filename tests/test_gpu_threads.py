"""Host-side thread safety of the library: several threads drive it at once, each
on its own stream and buffers (the LDG form, a hybrid launch and the TMA form;
then the pipelined and offload schedulers and copy-only launches), while another
thread calls the host-only entry points. Every result must equal the same calls
made one after another, bit for bit."""
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


def _pipeline_set(torch, shard):
    wl = bench.sweep_workload(8 * shard + 3, 8)
    units, info, bufs = bench.build_local_rank(wl, 2, torch, fs, synth)
    batch, staging, slot, keep = bench.pipeline_setup(torch, fs, units, info, 2, 2)
    return units, batch, staging, slot, keep


def _offload_set(torch, shard):
    wl = bench.sweep_workload(8 * shard + 5, 8)
    units, info, bufs = bench.build_local_rank(wl, 1, torch, fs, synth)
    host = {n: bufs[n].cpu().pin_memory() for n in ("master", "exp_avg", "exp_avg_sq")}
    off, so = [], 0
    for u in units:
        S = u["layout"].shard_numel
        off.append(dict(layout=u["layout"], grads=u["grads"], master=host["master"][so:so + S],
                        exp_avg=host["exp_avg"][so:so + S], exp_avg_sq=host["exp_avg_sq"][so:so + S],
                        other_shards=u["other_shards"], full_out=u["full_out"][0]))
        so += S
    slot = (max(u["layout"].shard_numel for u in units) + 3) // 4 * 4
    return units, host, fs.OffloadBatch(off), torch.empty(3 * 3 * slot, device="cuda"), slot


def test_concurrent_schedulers_match_sequential_calls():
    """A pipelined step (its unit moving in pieces), a staged offload step and copy-only
    TMA-form launches (pack) from three threads at once, each with its own streams and
    buffers, equal the same calls made one after another."""
    torch = gu.torch()
    sets = []
    for _ in range(2):  # [0]: one after another, [1]: all at once
        pipe = _pipeline_set(torch, 4_300_000)
        off = _offload_set(torch, 1_000_000)
        numels = [45_000_001, 3, 45_000_005]  # 22,000 copy chunks: the TMA form on 152 SMs
        lay, offs = fs.fsdp_flatten_layout(numels, 8)
        tens = [torch.randn(n, device="cuda", generator=torch.Generator("cuda").manual_seed(i)) for i, n in
                enumerate(numels)]
        flat = torch.empty(lay.padded_numel, device="cuda")
        sets.append((pipe, off, (tens, lay, offs, flat)))
    torch.cuda.synchronize()
    streams = [[torch.cuda.Stream() for _ in range(3)] for _ in range(3)]

    def run_pipe(s, st):
        units, batch, staging, slot, keep = s
        for t in range(1, 4):
            fs.fsdp_pipeline_step(batch, 2, staging, slot, 2, gu.adam_hyper(t), compute=st[0], copy=st[1])
        st[0].synchronize()

    def run_off(s, st):
        units, host, batch, staging, slot = s
        for t in range(1, 4):
            fs.fsdp_offload_step(batch, 1, staging, slot, 3, gu.adam_hyper(t), compute=st[0], h2d=st[1], d2h=st[2])
        st[0].synchronize()

    def run_pack(s, st):
        tens, lay, offs, flat = s
        for _ in range(3):
            fs.fsdp_pack_flat(tens, lay, offs, flat, stream=st[0])
        st[0].synchronize()

    runs = (run_pipe, run_off, run_pack)
    for k, fn in enumerate(runs):
        fn(sets[0][k], streams[k])
    start = threading.Barrier(3)
    errors = []

    def worker(k):
        try:
            torch.cuda.set_device(0)
            start.wait()
            runs[k](sets[1][k], streams[k])
        except Exception as e:  # reported below, on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(3)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    (pa, oa, ka), (pb, ob, kb) = sets
    for u, v in zip(pa[0], pb[0]):
        for name in ("master", "exp_avg", "exp_avg_sq", "full_out"):
            assert torch.equal(u[name][0].view(torch.int8), v[name][0].view(torch.int8)), "pipeline " + name
    assert torch.equal(pa[4][1], pb[4][1]), "pipeline shard_out"
    for n in ("master", "exp_avg", "exp_avg_sq"):
        assert torch.equal(oa[1][n].view(torch.int32), ob[1][n].view(torch.int32)), "offload " + n
    for u, v in zip(oa[0], ob[0]):
        assert torch.equal(u["full_out"][0], v["full_out"][0]), "offload full_out"
    assert torch.equal(ka[3].view(torch.int32), kb[3].view(torch.int32)), "pack"
    assert fs.fsdp_device_status() == 0
