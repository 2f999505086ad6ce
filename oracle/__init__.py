"""CPU oracle of the FSDP FlatParameter shard step (test infrastructure only).

Thin numpy/ctypes wrapper around ``oracle/fsdp_oracle.c``, the plain,
single-threaded, fp32-exact definition of every step (layout, pack, reduce-
scatter, Adam, bf16 cast, all-gather, the composite unit step, hybrid
sharding and the memory/communication accountant). Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import this package; the
CUDA library never does, and it shares no code with it.

Parity status of each function is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against values fixed by the pages and by
mathematics (worked example, closed forms, brute force, library routines).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "fsdp_oracle.c")
SO = os.path.join(_HERE, "_build", "libfsdp_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC"]

_P = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_f64 = ctypes.c_double


def compile_oracle(src: str, out: str, extra: Sequence[str] = ()) -> str:
    """Compile an oracle C source into a shared library (used by build() and tests)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cc = os.environ.get("CC", "gcc")
    subprocess.run([cc, *CFLAGS, *extra, "-o", tmp, src, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    if not force and os.path.exists(SO) and os.path.getmtime(SO) >= os.path.getmtime(SRC):
        return SO
    return compile_oracle(SRC, SO)


class Oracle:
    """One loaded copy of the oracle library (tests may load altered copies)."""

    def __init__(self, so_path: str):
        lib = ctypes.CDLL(so_path)
        sig = {
            "ora_flatten_layout": (_i32, [_P, _i32, _i32, _i32, _P, _P]),
            "ora_pack": (None, [_P, _P, _i32, _i32, _i64, _P]),
            "ora_unpack": (None, [_P, _P, _i32, _i32, _P]),
            "ora_bf16_rne": (ctypes.c_uint16, [_f32]),
            "ora_bf16_rne_array": (None, [_P, _i64, _P]),
            "ora_fold_mean": (None, [_P, _i32, _i64, _P]),
            "ora_reduce_scatter": (_i32, [_P, _i32, _i32, _i64, _i32, _P]),
            "ora_adam": (None, [_P, _P, _P, _P, _i64, _f64, _f64, _f64, _f64, _i64, _P]),
            "ora_all_gather": (None, [_P, _i32, _i64, _P]),
            "ora_shard_step": (_i32, [_P, _i32, _i32, _i64, _i32, _i32, _P, _P, _P, _P, _P,
                                      _f64, _f64, _f64, _f64, _i64]),
            "ora_account": (_i32, [_f64, _f64, _i32, _i32, _i32, _P]),
            "ora_account_zero": (_i32, [_f64, _i32, _i32, _P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        self.lib = lib

    # -- helpers ------------------------------------------------------------
    @staticmethod
    def _ptr(a: np.ndarray) -> int:
        assert a.flags.c_contiguous
        return a.ctypes.data

    @classmethod
    def _ptrs(cls, arrs) -> ctypes.Array:
        arr = (ctypes.c_void_p * max(1, len(arrs)))()
        for i, a in enumerate(arrs):
            arr[i] = None if a is None else cls._ptr(a)
        return arr

    # -- a1 -----------------------------------------------------------------
    def flatten_layout(self, numels: Sequence[int], world_size: int, shard_factor: int | None = None):
        """Returns (offsets[n+1], P, padded, S)."""
        F = world_size if shard_factor is None else shard_factor
        n = len(numels)
        nums = np.asarray(numels, dtype=np.int64)
        offs = np.zeros(n + 1, dtype=np.int64)
        sizes = np.zeros(3, dtype=np.int64)
        rc = self.lib.ora_flatten_layout(self._ptr(nums) if n else None, n, world_size, F,
                                         self._ptr(offs), self._ptr(sizes))
        if rc != 0:
            raise ValueError("oracle layout rejected the arguments (%d)" % rc)
        return offs, int(sizes[0]), int(sizes[1]), int(sizes[2])

    # -- a2 -----------------------------------------------------------------
    def pack(self, tensors: Sequence[np.ndarray], padded_numel: int) -> np.ndarray:
        ts = [np.ascontiguousarray(t).reshape(-1) for t in tensors]
        dt = ts[0].dtype
        assert all(t.dtype == dt for t in ts)
        nums = np.asarray([t.size for t in ts], dtype=np.int64)
        flat = np.empty(padded_numel, dtype=dt)
        self.lib.ora_pack(self._ptrs(ts), self._ptr(nums), len(ts), dt.itemsize, padded_numel,
                          self._ptr(flat))
        return flat

    def unpack(self, flat: np.ndarray, shapes: Sequence[tuple]) -> list:
        flat = np.ascontiguousarray(flat)
        outs = [np.empty(s, dtype=flat.dtype) for s in shapes]
        nums = np.asarray([o.size for o in outs], dtype=np.int64)
        self.lib.ora_unpack(self._ptr(flat), self._ptr(nums), len(outs), flat.dtype.itemsize,
                            self._ptrs(outs))
        return outs

    # -- a5 -----------------------------------------------------------------
    def bf16_rne(self, x: np.ndarray) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, dtype=np.uint16)
        self.lib.ora_bf16_rne_array(self._ptr(x), x.size, self._ptr(out))
        return out

    # -- a3 -----------------------------------------------------------------
    def fold_mean(self, rows: Sequence[np.ndarray]) -> np.ndarray:
        rows = [np.ascontiguousarray(r, dtype=np.uint16) for r in rows]
        n = rows[0].size
        out = np.empty(n, dtype=np.float32)
        self.lib.ora_fold_mean(self._ptrs(rows), len(rows), n, self._ptr(out))
        return out

    def reduce_scatter(self, grads: Sequence[np.ndarray], shard_factor: int, rank: int) -> np.ndarray:
        grads = [np.ascontiguousarray(g, dtype=np.uint16) for g in grads]
        W = len(grads)
        padded = grads[0].size
        S = padded // shard_factor
        out = np.empty(S, dtype=np.float32)
        rc = self.lib.ora_reduce_scatter(self._ptrs(grads), W, shard_factor, padded, rank,
                                         self._ptr(out))
        if rc != 0:
            raise ValueError("oracle reduce_scatter rejected the arguments (%d)" % rc)
        return out

    # -- a4/a5 --------------------------------------------------------------
    def adam(self, param, exp_avg, exp_avg_sq, grad, lr, beta1, beta2, eps, step, with_bf16=True):
        """In-place on the three state arrays; returns the bf16 bits (or None)."""
        n = param.size
        for a in (param, exp_avg, exp_avg_sq, grad):
            assert a.dtype == np.float32 and a.flags.c_contiguous and a.size == n
        out = np.empty(n, dtype=np.uint16) if with_bf16 else None
        self.lib.ora_adam(self._ptr(param), self._ptr(exp_avg), self._ptr(exp_avg_sq),
                          self._ptr(grad), n, lr, beta1, beta2, eps, step,
                          self._ptr(out) if with_bf16 else None)
        return out

    # -- a6 -----------------------------------------------------------------
    def all_gather(self, shards: Sequence[np.ndarray]) -> np.ndarray:
        shards = [np.ascontiguousarray(s, dtype=np.uint16) for s in shards]
        S = shards[0].size
        full = np.empty(S * len(shards), dtype=np.uint16)
        self.lib.ora_all_gather(self._ptrs(shards), len(shards), S, self._ptr(full))
        return full

    # -- a7/a8 --------------------------------------------------------------
    def shard_step(self, grads, shard_factor, rank_begin, rank_end, master, exp_avg, exp_avg_sq,
                   other_shards, full_out, lr, beta1, beta2, eps, step):
        """In place on master/exp_avg/exp_avg_sq (lists per owned rank) and full_out (per group)."""
        W = len(grads)
        padded = grads[0].size
        rc = self.lib.ora_shard_step(
            self._ptrs(grads), W, shard_factor, padded, rank_begin, rank_end,
            self._ptrs(master), self._ptrs(exp_avg), self._ptrs(exp_avg_sq),
            self._ptrs(other_shards) if other_shards is not None else None,
            self._ptrs(full_out), lr, beta1, beta2, eps, step)
        if rc != 0:
            raise ValueError("oracle shard_step rejected the arguments (%d)" % rc)

    # -- a9 -----------------------------------------------------------------
    ACCOUNT_FIELDS = ("persistent_bytes", "ddp_persistent_bytes", "transient_bytes", "peak_bytes",
                      "comm_elems", "comm_elems_ring", "ddp_comm_elems", "ddp_comm_elems_ring",
                      "comm_bytes", "ddp_comm_bytes")

    def account(self, P, U, N, F=None, prefetch=1) -> dict:
        F = N if F is None else F
        out = np.zeros(len(self.ACCOUNT_FIELDS), dtype=np.float64)
        rc = self.lib.ora_account(float(P), float(U), N, F, prefetch, self._ptr(out))
        if rc != 0:
            raise ValueError("oracle account rejected the arguments (%d)" % rc)
        return dict(zip(self.ACCOUNT_FIELDS, out.tolist()))


def _account_zero(self, P, N, stage) -> dict:
    out = np.zeros(6, dtype=np.float64)
    rc = self.lib.ora_account_zero(float(P), N, stage, self._ptr(out))
    if rc != 0:
        raise ValueError("oracle account_zero rejected the arguments (%d)" % rc)
    return dict(zip(("weights_bytes", "grads_bytes", "optimizer_bytes", "total_bytes", "reduction_vs_ddp",
                     "comm_elems"), out.tolist()))


Oracle.account_zero = _account_zero

_default: Oracle | None = None


def load() -> Oracle:
    """Build (if stale) and load the oracle library."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default
