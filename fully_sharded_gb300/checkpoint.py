"""Sharded checkpoint / resume and the rank-0 full state dict.

Glossary entry "fully sharded data parallel fsdp", "Checkpoint/Resume": a
FULL_STATE_DICT gathers the full model (on rank 0) instead of saving one piece
per rank. Both forms are here:

* ``save_sharded`` / ``load_sharded``: each rank writes its own fp32 master,
  exp_avg and exp_avg_sq shards of every unit plus the step counter; loading
  them back into fresh buffers resumes bit-exactly.
* ``full_state_dict``: gathers the W fp32 shards of one unit on the device
  (``fsdp_all_gather_state``) and unflattens them into the unit's tensors
  (``fsdp_unpack_flat``), padding dropped.

Files: ``<dir>/rank<r>/manifest.json`` (layouts, step, CRC-32 of every
array) and one raw little-endian ``.bin`` per array. Tensors may live on the
GPU or the CPU; the bytes go through host memory.
"""
from __future__ import annotations

import json
import os
import zlib

import numpy as np

from . import FSDP_DTYPE_F32, Layout, fsdp_all_gather_state, fsdp_unpack_flat

STATE_NAMES = ("master", "exp_avg", "exp_avg_sq")
FORMAT = "fsdp-gb300-sharded-v1"


def _host_bytes(t) -> bytes:
    return t.detach().contiguous().cpu().numpy().tobytes()


def _layout_dict(lay: Layout) -> dict:
    return dict(numel=lay.numel, padded_numel=lay.padded_numel, shard_numel=lay.shard_numel,
                world_size=lay.world_size, shard_factor=lay.shard_factor, n_tensors=lay.n_tensors)


def save_sharded(directory: str, rank: int, units, step: int) -> str:
    """Write rank `rank`'s shards. `units`: list of dicts with `layout` and the fp32 tensors
    `master`, `exp_avg`, `exp_avg_sq` (the rank's [S] shards). `step`: last completed step."""
    d = os.path.join(directory, "rank%d" % rank)
    os.makedirs(d, exist_ok=True)
    manifest = dict(format=FORMAT, rank=rank, step=int(step), units=[])
    for u, unit in enumerate(units):
        entry = dict(layout=_layout_dict(unit["layout"]), arrays={})
        for name in STATE_NAMES:
            raw = _host_bytes(unit[name])
            fname = "unit%d_%s.bin" % (u, name)
            with open(os.path.join(d, fname), "wb") as f:
                f.write(raw)
            entry["arrays"][name] = dict(file=fname, nbytes=len(raw), crc32=zlib.crc32(raw))
        manifest["units"].append(entry)
    tmp = os.path.join(d, "manifest.json.tmp")
    with open(tmp, "w") as f:
        json.dump(manifest, f, indent=1)
    os.replace(tmp, os.path.join(d, "manifest.json"))  # the manifest appears last
    return d


def load_sharded(directory: str, rank: int, units) -> int:
    """Read rank `rank`'s shards into the given tensors (same layouts); returns the step.
    Raises ValueError on a layout, size or checksum mismatch."""
    import torch
    d = os.path.join(directory, "rank%d" % rank)
    with open(os.path.join(d, "manifest.json")) as f:
        manifest = json.load(f)
    if manifest.get("format") != FORMAT or manifest.get("rank") != rank:
        raise ValueError("not a rank-%d checkpoint of this format: %s" % (rank, d))
    if len(manifest["units"]) != len(units):
        raise ValueError("checkpoint has %d units, expected %d" % (len(manifest["units"]), len(units)))
    for entry, unit in zip(manifest["units"], units):
        if entry["layout"] != _layout_dict(unit["layout"]):
            raise ValueError("layout mismatch: %r vs %r" % (entry["layout"], _layout_dict(unit["layout"])))
        for name in STATE_NAMES:
            a = entry["arrays"][name]
            with open(os.path.join(d, a["file"]), "rb") as f:
                raw = f.read()
            if len(raw) != a["nbytes"] or zlib.crc32(raw) != a["crc32"]:
                raise ValueError("corrupt array %s in %s" % (a["file"], d))
            dst = unit[name]
            if dst.numel() * dst.element_size() != len(raw):
                raise ValueError("size mismatch for %s" % a["file"])
            src = torch.from_numpy(np.frombuffer(raw, dtype=np.float32).copy())
            dst.copy_(src.view(dst.shape))
    return int(manifest["step"])


def full_state_dict(shards, layout: Layout, offsets, shapes, stream=None):
    """Full fp32 tensors of one unit from its F fp32 shards (device tensors): gather into
    a flat buffer on the device, then unflatten into new tensors of `shapes`."""
    import torch
    dev = shards[0].device
    flat = torch.empty(layout.padded_numel, dtype=torch.float32, device=dev)
    fsdp_all_gather_state(shards, layout, flat, stream=stream)
    outs = [torch.empty(s, dtype=torch.float32, device=dev) for s in shapes]
    fsdp_unpack_flat(flat, layout, offsets, outs, stream=stream)
    return outs


__all__ = ["save_sharded", "load_sharded", "full_state_dict", "FSDP_DTYPE_F32"]
