"""GB300-native FSDP FlatParameter shard step.

Python binding of the C ABI in ``include/fsdp.h`` (libfsdp_gb300.so, built
for sm_103a by ``fully_sharded_gb300.build``). The functions below have the
ABI's names and only marshal arguments: tensors become device pointers, lists
become host pointer arrays, the status code becomes an exception. Every step
of the path runs in the CUDA library; there is no other implementation, and
importing this package fails when the library is missing.

Tensors are torch CUDA tensors (contiguous) or raw integer device addresses.
bf16 buffers may be torch.bfloat16, torch.int16 or torch.uint16 (bit patterns).
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

from . import build as _build_mod

__all__ = [
    "FsdpError", "Layout", "AdamHyper", "Account", "library_path",
    "fsdp_flatten_layout", "fsdp_pack_flat", "fsdp_unpack_flat", "fsdp_reduce_scatter",
    "fsdp_adam_shard_step", "fsdp_all_gather", "fsdp_shard_step", "fsdp_shard_step_grouped",
    "fsdp_account", "fsdp_status_string", "UnitArgs", "UnitBatch",
    "fsdp_shard_step_grouped_launches", "fsdp_pipeline_step", "PipelineUnit", "PipelineBatch",
    "fsdp_pipeline_step_noalloc", "fsdp_all_gather_state", "fsdp_zero1_step", "fsdp_account_zero",
    "fsdp_shard_step_grouped_plan", "fsdp_device_status", "fsdp_selftest_wait_timeout",
    "fsdp_offload_step", "OffloadUnit", "OffloadBatch", "fsdp_reduce_scatter_ranks",
    "fsdp_adam_shard_step_grouped", "AdamShard",
]

FSDP_OK = 0
FSDP_EINVAL = -1
FSDP_EALIAS = -2
FSDP_ECUDA = -3
FSDP_ENOSPACE = -4
NOALLOC_STAGING_BYTES = 64 << 20  # FSDP_NOALLOC_STAGING_BYTES of include/fsdp.h
FSDP_DTYPE_F32 = 0
FSDP_DTYPE_BF16 = 1
MAX_WORLD = 64

_c_i32, _c_i64, _c_dbl, _c_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p


class Layout(ctypes.Structure):
    _fields_ = [("numel", _c_i64), ("padded_numel", _c_i64), ("shard_numel", _c_i64),
                ("world_size", _c_i32), ("shard_factor", _c_i32), ("n_tensors", _c_i32)]

    def __repr__(self):
        return ("Layout(numel=%d, padded_numel=%d, shard_numel=%d, world_size=%d, shard_factor=%d, "
                "n_tensors=%d)" % (self.numel, self.padded_numel, self.shard_numel, self.world_size,
                                   self.shard_factor, self.n_tensors))


class AdamHyper(ctypes.Structure):
    _fields_ = [("lr", _c_dbl), ("beta1", _c_dbl), ("beta2", _c_dbl), ("eps", _c_dbl),
                ("weight_decay", _c_dbl), ("step", _c_i64)]

    def __init__(self, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.0, step=1):
        super().__init__(lr, beta1, beta2, eps, weight_decay, step)


class UnitArgs(ctypes.Structure):
    _fields_ = [("layout", ctypes.POINTER(Layout)), ("grads", _c_p), ("master", _c_p),
                ("exp_avg", _c_p), ("exp_avg_sq", _c_p), ("other_shards", _c_p),
                ("full_out", _c_p)]


class PipelineUnit(ctypes.Structure):
    _fields_ = [("layout", ctypes.POINTER(Layout)), ("grad_slices", _c_p), ("master", _c_p),
                ("exp_avg", _c_p), ("exp_avg_sq", _c_p), ("other_shards", _c_p), ("full_out", _c_p),
                ("shard_out", _c_p)]


class OffloadUnit(ctypes.Structure):
    _fields_ = [("layout", ctypes.POINTER(Layout)), ("grads", _c_p), ("master", _c_p), ("exp_avg", _c_p),
                ("exp_avg_sq", _c_p), ("other_shards", _c_p), ("full_out", _c_p)]


class AdamShard(ctypes.Structure):
    _fields_ = [("master", _c_p), ("exp_avg", _c_p), ("exp_avg_sq", _c_p), ("grad_shard", _c_p),
                ("bf16_shard_out", _c_p), ("n", _c_i64)]


class ZeroAccount(ctypes.Structure):
    _fields_ = [(n, _c_dbl) for n in ("weights_bytes", "grads_bytes", "optimizer_bytes", "total_bytes",
                                      "reduction_vs_ddp", "comm_elems")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class Account(ctypes.Structure):
    _fields_ = [(n, _c_dbl) for n in (
        "persistent_bytes", "ddp_persistent_bytes", "transient_bytes", "peak_bytes", "comm_elems",
        "comm_elems_ring", "ddp_comm_elems", "ddp_comm_elems_ring", "comm_bytes", "ddp_comm_bytes")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


class FsdpError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__("%s: %s (status %d)" % (fn, fsdp_status_string(status), status))
        self.status = status


def library_path() -> str:
    """The in-tree library, or the file named by FSDP_GB300_LIB (an alternative build)."""
    return os.environ.get("FSDP_GB300_LIB") or _build_mod.SO


def _load():
    so = library_path()
    if not os.path.exists(so):
        raise ImportError("fully_sharded_gb300: CUDA library %s is not built; run "
                          "`python fully_sharded_gb300/build.py` (needs nvcc)" % so)
    lib = ctypes.CDLL(so)
    P = _c_p
    sigs = {
        "fsdp_flatten_layout": [P, _c_i32, _c_i32, _c_i32, P, ctypes.POINTER(Layout)],
        "fsdp_pack_flat": [P, ctypes.POINTER(Layout), P, _c_i32, P, P],
        "fsdp_unpack_flat": [P, ctypes.POINTER(Layout), P, _c_i32, P, P],
        "fsdp_reduce_scatter": [P, ctypes.POINTER(Layout), _c_i32, P, P],
        "fsdp_adam_shard_step": [P, P, P, P, _c_i64, ctypes.POINTER(AdamHyper), P, P],
        "fsdp_reduce_scatter_ranks": [P, ctypes.POINTER(Layout), _c_i32, _c_i32, P, P],
        "fsdp_adam_shard_step_grouped": [ctypes.POINTER(AdamShard), _c_i32, ctypes.POINTER(AdamHyper), P],
        "fsdp_all_gather": [P, ctypes.POINTER(Layout), P, P],
        "fsdp_shard_step": [P, ctypes.POINTER(Layout), _c_i32, _c_i32, P, P, P, P, P,
                            ctypes.POINTER(AdamHyper), P],
        "fsdp_shard_step_grouped": [ctypes.POINTER(UnitArgs), _c_i32, _c_i32, _c_i32,
                                    ctypes.POINTER(AdamHyper), P],
        "fsdp_shard_step_grouped_launches": [ctypes.POINTER(UnitArgs), _c_i32, _c_i32, _c_i32,
                                             ctypes.POINTER(_c_i32)],
        "fsdp_account": [_c_dbl, _c_dbl, _c_i32, _c_i32, _c_i32, ctypes.POINTER(Account)],
        "fsdp_pipeline_step": [ctypes.POINTER(PipelineUnit), _c_i32, _c_i32, P, _c_i64, _c_i32,
                               ctypes.POINTER(AdamHyper), P, P],
        "fsdp_pipeline_step_noalloc": [ctypes.POINTER(PipelineUnit), _c_i32, _c_i32, _c_i32,
                                       ctypes.POINTER(AdamHyper), P, P],
        "fsdp_all_gather_state": [P, ctypes.POINTER(Layout), _c_i32, P, P],
        "fsdp_zero1_step": [P, ctypes.POINTER(Layout), _c_i32, P, P, P, P, P, P, ctypes.POINTER(AdamHyper), P],
        "fsdp_account_zero": [_c_dbl, _c_i32, _c_i32, ctypes.POINTER(ZeroAccount)],
        "fsdp_shard_step_grouped_plan": [ctypes.POINTER(UnitArgs), _c_i32, _c_i32, _c_i32,
                                         ctypes.POINTER(_c_i32), ctypes.POINTER(_c_i32),
                                         ctypes.POINTER(_c_i32)],
        "fsdp_device_status": [_c_i32, ctypes.POINTER(ctypes.c_uint32)],
        "fsdp_selftest_wait_timeout": [P, P, _c_i64, _c_i64, P, ctypes.POINTER(ctypes.c_uint32)],
        "fsdp_offload_step": [ctypes.POINTER(OffloadUnit), _c_i32, _c_i32, P, _c_i64, _c_i32,
                              ctypes.POINTER(AdamHyper), P, P, P],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.fsdp_status_string.argtypes = [ctypes.c_int]
    lib.fsdp_status_string.restype = ctypes.c_char_p
    return lib


_lib = _load()


# ------------------------------------------------------------- marshalling

def _dptr(x, itemsize: int | None = None) -> int | None:
    """Device address of a contiguous CUDA tensor (or an int address, or None)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if not x.is_cuda:
        raise ValueError("expected a CUDA tensor, got one on %s" % x.device)
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if itemsize is not None and x.element_size() != itemsize:
        raise ValueError("expected %d-byte elements, got %s" % (itemsize, x.dtype))
    return x.data_ptr()


def _parray(xs, itemsize=None):
    if xs is None:
        return None
    arr = (_c_p * max(1, len(xs)))()
    for i, x in enumerate(xs):
        arr[i] = _dptr(x, itemsize)
    return arr


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != FSDP_OK:
        raise FsdpError(fn, status)


def fsdp_status_string(status: int) -> str:
    return _lib.fsdp_status_string(status).decode()


# -------------------------------------------------------------- the calls

def fsdp_flatten_layout(numels: Sequence[int], world_size: int, shard_factor: int | None = None):
    """a1: returns (Layout, offsets list of n+1 ints)."""
    n = len(numels)
    nums = (_c_i64 * max(1, n))(*numels)
    offs = (_c_i64 * (n + 1))()
    lay = Layout()
    F = world_size if shard_factor is None else shard_factor
    _check("fsdp_flatten_layout",
           _lib.fsdp_flatten_layout(nums, n, world_size, F, offs, ctypes.byref(lay)))
    return lay, list(offs)


def _offsets(offsets):
    return (_c_i64 * len(offsets))(*offsets)


def _dtype_of(t) -> int:
    size = t.element_size()
    return FSDP_DTYPE_F32 if size == 4 else FSDP_DTYPE_BF16


def fsdp_pack_flat(tensors, layout: Layout, offsets, flat_out, stream=None):
    """a2: flat_out[offsets[i]:offsets[i+1]] = tensors[i]; pad zeroed."""
    es = flat_out.element_size()
    _check("fsdp_pack_flat", _lib.fsdp_pack_flat(_parray(tensors, es), ctypes.byref(layout),
                                                 _offsets(offsets), _dtype_of(flat_out),
                                                 _dptr(flat_out), _stream(stream)))


def fsdp_unpack_flat(flat, layout: Layout, offsets, tensors_out, stream=None):
    es = flat.element_size()
    _check("fsdp_unpack_flat", _lib.fsdp_unpack_flat(_dptr(flat), ctypes.byref(layout),
                                                     _offsets(offsets), _dtype_of(flat),
                                                     _parray(tensors_out, es), _stream(stream)))


def fsdp_reduce_scatter(grads, layout: Layout, rank: int, grad_shard_out, stream=None):
    """a3: grad_shard_out (fp32 [S]) = fixed-order fp32 mean of the W bf16 rows at rank's slice."""
    _check("fsdp_reduce_scatter", _lib.fsdp_reduce_scatter(
        _parray(grads, 2), ctypes.byref(layout), rank, _dptr(grad_shard_out, 4), _stream(stream)))


def fsdp_adam_shard_step(master, exp_avg, exp_avg_sq, grad_shard, adam: AdamHyper,
                         bf16_shard_out=None, stream=None, n: int | None = None):
    """a4+a5: Adam in place on the fp32 shard; optional bf16 cast out."""
    if n is None:
        n = master.numel()
    _check("fsdp_adam_shard_step", _lib.fsdp_adam_shard_step(
        _dptr(master, 4), _dptr(exp_avg, 4), _dptr(exp_avg_sq, 4), _dptr(grad_shard, 4), n,
        ctypes.byref(adam), _dptr(bf16_shard_out, 2), _stream(stream)))


def fsdp_reduce_scatter_ranks(grads, layout: Layout, rank_begin: int, rank_end: int, grad_shards_out,
                              stream=None):
    """a3 for ranks [rank_begin, rank_end) in one launch: grad_shards_out[r - rank_begin] (fp32 [S])
    receives rank r's reduce-scatter."""
    _check("fsdp_reduce_scatter_ranks", _lib.fsdp_reduce_scatter_ranks(
        _parray(grads, 2), ctypes.byref(layout), rank_begin, rank_end, _parray(grad_shards_out, 4),
        _stream(stream)))


class AdamShardBatch:
    """Marshalled shards for fsdp_adam_shard_step_grouped."""

    def __init__(self, shards):
        self.n = len(shards)
        self.array = (AdamShard * max(1, self.n))()
        for i, s in enumerate(shards):
            a = self.array[i]
            a.master = _dptr(s["master"], 4)
            a.exp_avg = _dptr(s["exp_avg"], 4)
            a.exp_avg_sq = _dptr(s["exp_avg_sq"], 4)
            a.grad_shard = _dptr(s["grad_shard"], 4)
            a.bf16_shard_out = _dptr(s.get("bf16_shard_out"), 2)
            a.n = s["n"] if "n" in s else s["master"].numel()


def fsdp_adam_shard_step_grouped(shards, adam: AdamHyper, stream=None):
    """a4+a5 over several shards in one launch. `shards`: dicts (master, exp_avg, exp_avg_sq,
    grad_shard, optional bf16_shard_out and n) or a prepared AdamShardBatch."""
    batch = shards if isinstance(shards, AdamShardBatch) else AdamShardBatch(shards)
    _check("fsdp_adam_shard_step_grouped", _lib.fsdp_adam_shard_step_grouped(
        batch.array, batch.n, ctypes.byref(adam), _stream(stream)))


def fsdp_all_gather(shards, layout: Layout, full_out, stream=None):
    """a6: full_out[k*S:(k+1)*S] = shards[k]."""
    _check("fsdp_all_gather", _lib.fsdp_all_gather(_parray(shards, 2), ctypes.byref(layout),
                                                   _dptr(full_out, 2), _stream(stream)))


def fsdp_shard_step(grads, layout: Layout, rank_begin: int, rank_end: int, master, exp_avg,
                    exp_avg_sq, other_shards, full_out, adam: AdamHyper, stream=None):
    """a7/a8: fused reduce-scatter -> Adam -> bf16 -> all-gather for ranks [rank_begin, rank_end)."""
    _check("fsdp_shard_step", _lib.fsdp_shard_step(
        _parray(grads, 2), ctypes.byref(layout), rank_begin, rank_end, _parray(master, 4),
        _parray(exp_avg, 4), _parray(exp_avg_sq, 4), _parray(other_shards, 2),
        _parray(full_out, 2), ctypes.byref(adam), _stream(stream)))


class UnitBatch:
    """Marshalled arguments of several units for fsdp_shard_step_grouped (kept alive together)."""

    def __init__(self, units):
        self._keep = []
        self.array = (UnitArgs * max(1, len(units)))()
        self.n = len(units)
        for i, u in enumerate(units):
            lay = u["layout"]
            arrs = dict(grads=_parray(u["grads"], 2), master=_parray(u["master"], 4),
                        exp_avg=_parray(u["exp_avg"], 4), exp_avg_sq=_parray(u["exp_avg_sq"], 4),
                        other_shards=_parray(u.get("other_shards"), 2),
                        full_out=_parray(u["full_out"], 2))
            self._keep.append((lay, arrs))
            a = self.array[i]
            a.layout = ctypes.pointer(lay)
            for k, v in arrs.items():
                setattr(a, k, ctypes.cast(v, _c_p) if v is not None else None)


def fsdp_shard_step_grouped(units, rank_begin: int, rank_end: int, adam: AdamHyper, stream=None):
    """a7 over several units in one launch. `units`: list of dicts (layout, grads, master,
    exp_avg, exp_avg_sq, other_shards, full_out) or a prepared UnitBatch."""
    batch = units if isinstance(units, UnitBatch) else UnitBatch(units)
    _check("fsdp_shard_step_grouped", _lib.fsdp_shard_step_grouped(
        batch.array, batch.n, rank_begin, rank_end, ctypes.byref(adam), _stream(stream)))


def fsdp_shard_step_grouped_launches(units, rank_begin: int, rank_end: int) -> int:
    """Host only: how many kernel launches fsdp_shard_step_grouped makes for these units."""
    batch = units if isinstance(units, UnitBatch) else UnitBatch(units)
    n = _c_i32(0)
    _check("fsdp_shard_step_grouped_launches", _lib.fsdp_shard_step_grouped_launches(
        batch.array, batch.n, rank_begin, rank_end, ctypes.byref(n)))
    return n.value


def _addr(x) -> int | None:
    """Address of a tensor in device or (pinned) host memory, or an int address."""
    if x is None or isinstance(x, int):
        return x
    if not x.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return x.data_ptr()


class PipelineBatch:
    """Marshalled units for fsdp_pipeline_step (kept alive together)."""

    def __init__(self, units):
        self._keep = []
        self.array = (PipelineUnit * max(1, len(units)))()
        self.n = len(units)
        for i, u in enumerate(units):
            lay = u["layout"]
            oth = _parray(u["other_shards"], 2)
            self._keep.append((lay, oth))
            a = self.array[i]
            a.layout = ctypes.pointer(lay)
            a.grad_slices = _addr(u["grad_slices"])
            a.master = _dptr(u["master"], 4)
            a.exp_avg = _dptr(u["exp_avg"], 4)
            a.exp_avg_sq = _dptr(u["exp_avg_sq"], 4)
            a.other_shards = ctypes.cast(oth, _c_p)
            a.full_out = _dptr(u["full_out"], 2)
            a.shard_out = _addr(u.get("shard_out"))


def fsdp_pipeline_step(units, rank: int, staging, slot_numel: int, n_slots: int, adam: AdamHyper,
                       compute=None, copy=None):
    """Pipelined step of one rank over many units (prefetch = n_slots - 1). `units`: list of
    dicts (layout, grad_slices, master, exp_avg, exp_avg_sq, other_shards, full_out,
    shard_out) or a PipelineBatch; `staging`: device bf16 buffer of n_slots * slot_numel."""
    batch = units if isinstance(units, PipelineBatch) else PipelineBatch(units)
    _check("fsdp_pipeline_step", _lib.fsdp_pipeline_step(
        batch.array, batch.n, rank, _dptr(staging, 2), slot_numel, n_slots, ctypes.byref(adam),
        _stream(compute), _stream(copy)))


class OffloadBatch:
    """Marshalled units for fsdp_offload_step (kept alive together)."""

    def __init__(self, units):
        self._keep = []
        self.array = (OffloadUnit * max(1, len(units)))()
        self.n = len(units)
        for i, u in enumerate(units):
            lay = u["layout"]
            g = _parray(u["grads"], 2)
            oth = _parray(u["other_shards"], 2)
            self._keep.append((lay, g, oth))
            a = self.array[i]
            a.layout = ctypes.pointer(lay)
            a.grads = ctypes.cast(g, _c_p)
            for name in ("master", "exp_avg", "exp_avg_sq"):
                x = u[name]
                if x is not None and not isinstance(x, int) and x.element_size() != 4:
                    raise ValueError("%s: expected fp32, got %s" % (name, x.dtype))
                setattr(a, name, _addr(x))
            a.other_shards = ctypes.cast(oth, _c_p)
            a.full_out = _dptr(u["full_out"], 2)


def fsdp_offload_step(units, rank: int, staging, slot_numel: int, n_slots: int, adam: AdamHyper,
                      compute=None, h2d=None, d2h=None):
    """Staged optimizer-state offload over many units: `units` are dicts (layout, grads,
    master, exp_avg, exp_avg_sq, other_shards, full_out) with master/exp_avg/exp_avg_sq in
    (pinned) host memory, or an OffloadBatch; `staging`: device fp32 buffer of
    n_slots * 3 * slot_numel."""
    batch = units if isinstance(units, OffloadBatch) else OffloadBatch(units)
    _check("fsdp_offload_step", _lib.fsdp_offload_step(
        batch.array, batch.n, rank, _dptr(staging, 4), slot_numel, n_slots, ctypes.byref(adam),
        _stream(compute), _stream(h2d), _stream(d2h)))


def fsdp_pipeline_step_noalloc(units, rank: int, n_slots: int, adam: AdamHyper, compute=None,
                               copy=None):
    """fsdp_pipeline_step without a staging argument, for callers that cannot allocate
    device memory when they step: the pool is a fixed array of NOALLOC_STAGING_BYTES
    inside the library (FsdpError with status FSDP_ENOSPACE if n_slots times the largest
    unit, rounded up to 8 elements, does not fit). Calls on one device share that array,
    so their GPU work must not overlap."""
    batch = units if isinstance(units, PipelineBatch) else PipelineBatch(units)
    _check("fsdp_pipeline_step_noalloc", _lib.fsdp_pipeline_step_noalloc(
        batch.array, batch.n, rank, n_slots, ctypes.byref(adam), _stream(compute), _stream(copy)))


def fsdp_all_gather_state(shards, layout: Layout, full_out, stream=None):
    """Gather per-rank state (fp32 master/m/v, or bf16) into the full flat buffer of a group."""
    es = full_out.element_size()
    _check("fsdp_all_gather_state", _lib.fsdp_all_gather_state(
        _parray(shards, es), ctypes.byref(layout), _dtype_of(full_out), _dptr(full_out), _stream(stream)))


def fsdp_zero1_step(grads, layout: Layout, rank: int, avg_grad_out, master, exp_avg, exp_avg_sq, other_shards,
                    full_out, adam: AdamHyper, stream=None):
    """ZeRO stage 1 step of one rank: full all-reduce average into avg_grad_out, Adam on the
    rank's slice, bf16 shard and gather into full_out."""
    _check("fsdp_zero1_step", _lib.fsdp_zero1_step(
        _parray(grads, 2), ctypes.byref(layout), rank, _dptr(avg_grad_out, 4), _dptr(master, 4),
        _dptr(exp_avg, 4), _dptr(exp_avg_sq, 4), _parray(other_shards, 2), _dptr(full_out, 2),
        ctypes.byref(adam), _stream(stream)))


def fsdp_account_zero(P: float, N: int, stage: int) -> dict:
    """Per-GPU bytes of ZeRO stage 0 (DDP) .. 3 (FSDP) and the communication per step (host only)."""
    out = ZeroAccount()
    _check("fsdp_account_zero", _lib.fsdp_account_zero(float(P), N, stage, ctypes.byref(out)))
    return out.as_dict()


def fsdp_shard_step_grouped_plan(units, rank_begin: int, rank_end: int, interleaved: bool = False):
    """Host only: (launches, launches in the TMA form) of fsdp_shard_step_grouped for these
    units; with interleaved=True also the number of TMA launches that stage their step
    chunks in interleaved quarter-chunk copies."""
    batch = units if isinstance(units, UnitBatch) else UnitBatch(units)
    n, t, i = _c_i32(0), _c_i32(0), _c_i32(0)
    _check("fsdp_shard_step_grouped_plan", _lib.fsdp_shard_step_grouped_plan(
        batch.array, batch.n, rank_begin, rank_end, ctypes.byref(n), ctypes.byref(t), ctypes.byref(i)))
    return (n.value, t.value, i.value) if interleaved else (n.value, t.value)


def fsdp_device_status(clear: bool = False) -> int:
    """The current device's sticky status word (bit 0: a bounded wait of the TMA form ran out)."""
    v = ctypes.c_uint32(0)
    _check("fsdp_device_status", _lib.fsdp_device_status(1 if clear else 0, ctypes.byref(v)))
    return v.value


def fsdp_selftest_wait_timeout(src, dst, wait_limit_ns: int, stream=None) -> int:
    """Diagnostic call of include/fsdp_test.h (not part of the method's interface):
    provokes one bounded-wait timeout on a copy of src into dst; returns the status word seen."""
    v = ctypes.c_uint32(0)
    nbytes = src.numel() * src.element_size()
    _check("fsdp_selftest_wait_timeout", _lib.fsdp_selftest_wait_timeout(
        _dptr(src), _dptr(dst), nbytes, int(wait_limit_ns), _stream(stream), ctypes.byref(v)))
    return v.value


def fsdp_account(P: float, U: float, N: int, F: int | None = None, prefetch: int = 1) -> dict:
    """a9: closed-form memory and communication budget (host only)."""
    out = Account()
    _check("fsdp_account", _lib.fsdp_account(float(P), float(U), N, N if F is None else F,
                                             prefetch, ctypes.byref(out)))
    return out.as_dict()
