"""Sharded checkpoint files on the host: round trip, layout and corruption checks."""
import os

import pytest
import torch

import fully_sharded_gb300 as fs
from fully_sharded_gb300 import checkpoint as ck


def _units(seed):
    g = torch.Generator().manual_seed(seed)
    out = []
    for P in (1000, 4096 + 3):
        lay, _ = fs.fsdp_flatten_layout([P], 4)
        S = lay.shard_numel
        out.append(dict(layout=lay, master=torch.randn(S, generator=g), exp_avg=torch.randn(S, generator=g),
                        exp_avg_sq=torch.rand(S, generator=g)))
    return out


def test_round_trip_is_bit_exact(tmp_path):
    a = _units(0)
    ck.save_sharded(str(tmp_path), 2, a, step=7)
    b = _units(1)
    assert ck.load_sharded(str(tmp_path), 2, b) == 7
    for x, y in zip(a, b):
        for name in ck.STATE_NAMES:
            assert torch.equal(x[name].view(torch.int32), y[name].view(torch.int32))


def test_detects_layout_mismatch_and_corruption(tmp_path):
    a = _units(0)
    ck.save_sharded(str(tmp_path), 0, a, step=1)
    other = _units(0)
    other[1]["layout"] = fs.fsdp_flatten_layout([4096 + 3], 8)[0]
    with pytest.raises(ValueError):
        ck.load_sharded(str(tmp_path), 0, other)
    path = os.path.join(str(tmp_path), "rank0", "unit1_exp_avg.bin")
    raw = bytearray(open(path, "rb").read())
    raw[10] ^= 1
    open(path, "wb").write(bytes(raw))
    with pytest.raises(ValueError):
        ck.load_sharded(str(tmp_path), 0, _units(0))
    with pytest.raises(FileNotFoundError):
        ck.load_sharded(str(tmp_path), 3, _units(0))
