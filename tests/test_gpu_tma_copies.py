"""Copy launches large enough for the TMA form: pack, unpack, all-gather and the
state gather, each moving over 130 copy chunks of 16 KB per SM, against the
oracle bit for bit.

The inputs are random bit patterns (NaN and subnormal encodings included: a copy
moves bytes, not values). Tensor and shard sizes are odd, so some segments of each
launch start off a 16-byte boundary; the TMA form stages the aligned segments
through shared memory and copies the others from global memory, and both kinds
are checked. Guard canaries around every destination catch stray writes.
"""
import numpy as np
import pytest

import gpu_util as gu

pytestmark = pytest.mark.gpu

fs = pytest.importorskip("fully_sharded_gb300")

W = 8
COPY_CHUNK = 16384  # bytes per copy chunk


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _bytes_needed():
    sms = gu.torch().cuda.get_device_properties(0).multi_processor_count
    return 130 * sms * COPY_CHUNK


def _bits(rng, n, es):
    if es == 4:
        return rng.integers(0, 1 << 32, size=n, dtype=np.uint32).view(np.float32)
    return rng.integers(0, 1 << 16, size=n, dtype=np.uint16)


def _tdt(es):
    torch = gu.torch()
    return torch.float32 if es == 4 else torch.int16


@pytest.mark.parametrize("es", [4, 2])
def test_pack_unpack(ora, es):
    torch = gu.torch()
    rng = np.random.default_rng(600 + es)
    half = _bytes_needed() // es // 2
    numels = [half + 1, 3, half + 5, 0, 7]  # later tensors start off 16-byte boundaries
    lay, offs = fs.fsdp_flatten_layout(numels, W)
    hs = [_bits(rng, n, es) for n in numels]
    ds = [gu.to_dev(h) if h.size else torch.empty(0, dtype=_tdt(es), device="cuda") for h in hs]
    whole, flat = gu.guarded(lay.padded_numel, _tdt(es), 77)
    fs.fsdp_pack_flat(ds, lay, offs, flat)
    want = ora.pack(hs, lay.padded_numel)
    gu.assert_same_bits(gu.to_host(flat), want, "pack")
    assert gu.canaries_intact(whole, lay.padded_numel, 77), "write outside the flat buffer"
    outs = [gu.guarded(n, _tdt(es), 5) for n in numels]
    fs.fsdp_unpack_flat(flat, lay, offs, [o[1] for o in outs])
    for (w, o), h, n in zip(outs, hs, numels):
        gu.assert_same_bits(gu.to_host(o), h, "unpack of %d elements" % n)
        assert gu.canaries_intact(w, n, 5), "write outside an unpacked tensor"


@pytest.mark.parametrize("es", [2, 4])
def test_all_gather(ora, es):
    """bf16 parameters through fsdp_all_gather, fp32 state through fsdp_all_gather_state;
    an odd shard length puts every other destination off a 16-byte boundary."""
    torch = gu.torch()
    rng = np.random.default_rng(700 + es)
    S = (_bytes_needed() // es // W) | 1
    lay, _ = fs.fsdp_flatten_layout([W * S], W)
    assert lay.shard_numel == S
    shards = [_bits(rng, S, es) for _ in range(W)]
    whole, full = gu.guarded(W * S, _tdt(es), 9)
    if es == 2:
        fs.fsdp_all_gather([gu.to_dev(s) for s in shards], lay, full)
    else:
        fs.fsdp_all_gather_state([gu.to_dev(s) for s in shards], lay, full)
    # a copy of 4-byte elements is the copy of their bytes: gather the 2-byte halves
    want = ora.all_gather([np.ascontiguousarray(s).view(np.uint16) for s in shards])
    gu.assert_same_bits(gu.to_host(full).view(np.uint16), want, "all-gather, %d-byte elements" % es)
    assert gu.canaries_intact(whole, W * S, 9), "write outside the full buffer"
