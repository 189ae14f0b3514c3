"""TEST INFRASTRUCTURE ONLY: ctypes binding of the plain C++ parity oracle.

The oracle (``zero_oracle.cpp``) is a single-threaded CPU definition of the
per-shard mixed-precision ZeRO optimizer step.  Only the test-suite, the smoke
check and the benchmark's CPU-baseline leg may import this package; the
product library never does, and it shares no code with it.  This module only
marshals numpy arrays into the C functions; all arithmetic is in the C++ file.

``Oracle(path)`` binds one compiled copy of the oracle (the mutation tests
load deliberately broken copies); the module-level functions use the default
build in this directory.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "zero_oracle.cpp")
HEADER = os.path.join(_HERE, "zero_oracle.h")
LIB_PATH = os.path.join(_HERE, "liborc.so")

FP16 = 0
BF16 = 1

CXXFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c++17",
            "-fPIC", "-shared", "-Wall", "-Wextra"]


def compile_source(src: str, out_path: str) -> str:
    """Compile one copy of the oracle source to a shared library."""
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out_path))
    os.close(fd)
    cmd = ["g++", *CXXFLAGS, "-I", _HERE, "-o", tmp, src]
    try:
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, out_path)
    except subprocess.CalledProcessError as e:
        os.unlink(tmp)
        raise RuntimeError("oracle build failed:\n" + e.stderr) from e
    return out_path


def build(force: bool = False) -> str:
    """Compile the oracle in place unless the library is newer than its source."""
    newest = max(os.path.getmtime(SOURCE), os.path.getmtime(HEADER))
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= newest):
        return LIB_PATH
    return compile_source(SOURCE, LIB_PATH)


class Hparams(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_double), ("beta1", ctypes.c_double),
                ("beta2", ctypes.c_double), ("eps", ctypes.c_double),
                ("weight_decay", ctypes.c_double),
                ("max_grad_norm", ctypes.c_double),
                ("bias_correction", ctypes.c_int32),
                ("dynamic_scale", ctypes.c_int32),
                ("min_scale", ctypes.c_double),
                ("scale_factor", ctypes.c_double),
                ("scale_window", ctypes.c_int64),
                ("hysteresis", ctypes.c_int64),
                ("warmup_min_lr", ctypes.c_double),
                ("warmup_max_lr", ctypes.c_double),
                ("warmup_num_steps", ctypes.c_int64)]


class Scaler(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("last_skipped", ctypes.c_int32),
                ("clean", ctypes.c_int64), ("t", ctypes.c_int64),
                ("skipped_total", ctypes.c_int64), ("overflows", ctypes.c_int32),
                ("pad_", ctypes.c_int32)]

    def as_tuple(self):
        """(scale, clean, t, skipped_total, last_skipped)."""
        return (float(self.scale), int(self.clean), int(self.t),
                int(self.skipped_total), int(self.last_skipped))


class Stats(ctypes.Structure):
    _fields_ = [("sumsq", ctypes.c_double), ("nonfinite", ctypes.c_int32),
                ("pad_", ctypes.c_int32)]


class Decision(ctypes.Structure):
    _fields_ = [("skip", ctypes.c_int32), ("coef", ctypes.c_float),
                ("norm", ctypes.c_double), ("inv", ctypes.c_double),
                ("scale_used", ctypes.c_float),
                ("step_size", ctypes.c_float), ("isb2", ctypes.c_float),
                ("decay", ctypes.c_float), ("b1", ctypes.c_float),
                ("omb1", ctypes.c_float), ("b2", ctypes.c_float),
                ("omb2", ctypes.c_float), ("eps", ctypes.c_float),
                ("lr", ctypes.c_double)]


_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def hparams(lr=1e-3, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.0,
            max_grad_norm=0.0, bias_correction=True, dynamic_scale=False,
            min_scale=1.0, scale_factor=2.0, scale_window=1000, hysteresis=1,
            warmup=(0.0, 0.0, 0)) -> Hparams:
    """`warmup` = (warmup_min_lr, warmup_max_lr, warmup_num_steps); 0 steps
    keeps lr constant."""
    return Hparams(lr, betas[0], betas[1], eps, weight_decay, max_grad_norm,
                   int(bias_correction), int(dynamic_scale), min_scale,
                   scale_factor, scale_window, hysteresis, warmup[0], warmup[1],
                   warmup[2])


def scaler(scale: float = 1.0) -> Scaler:
    return Scaler(scale, 0, 0, 0, 0, 0, 0)


def _ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be contiguous"
    return a.ctypes.data


def _ptr_array(bufs):
    arr = (ctypes.c_void_p * len(bufs))()
    for i, b in enumerate(bufs):
        arr[i] = _ptr(b)
    return arr


class Oracle:
    """One loaded copy of the oracle library."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        L.orc_shard_bounds.argtypes = [_I64, _I32, _I32, ctypes.POINTER(_I64)]
        L.orc_shard_bounds.restype = ctypes.c_int
        L.orc_memory_bytes.argtypes = [_I64, _I32, _I32]
        L.orc_memory_bytes.restype = _I64
        L.orc_f32_to_16.argtypes = [ctypes.c_float, _I32]
        L.orc_f32_to_16.restype = ctypes.c_uint16
        L.orc_16_to_f32.argtypes = [ctypes.c_uint16, _I32]
        L.orc_16_to_f32.restype = ctypes.c_float
        L.orc_cast_f32_to_16.argtypes = [_P, _P, _I64, _I32]
        L.orc_cast_16_to_f32.argtypes = [_P, _P, _I64, _I32]
        L.orc_reduce.argtypes = [_P, _I32, _I64, _I32, _P]
        L.orc_stats_of.argtypes = [_P, _I64]
        L.orc_stats_of.restype = Stats
        L.orc_fold_stats.argtypes = [_P, _I32]
        L.orc_fold_stats.restype = Stats
        L.orc_decide.argtypes = [ctypes.POINTER(Hparams), ctypes.POINTER(Scaler),
                                 Stats, ctypes.c_double, ctypes.POINTER(Decision)]
        L.orc_update.argtypes = [ctypes.POINTER(Decision), _P, _P, _P, _P, _P,
                                 _I64, _I32]
        L.orc_step.argtypes = [ctypes.POINTER(Hparams), ctypes.POINTER(Scaler),
                               _P, _I32, _I32, _I64, ctypes.c_double,
                               _P, _P, _P, _P, _I32,
                               ctypes.POINTER(Stats), ctypes.POINTER(Stats),
                               ctypes.POINTER(Decision)]
        L.orc_step.restype = ctypes.c_int
        L.orc_consolidate.argtypes = [_P, _I32, _I64, _P]
        self.L = L
        self.path = path

    # a0 and the closed forms -------------------------------------------------
    def shard_bounds(self, numel: int, world: int, rank: int):
        """(begin, real_end, shard_len, padded_numel)."""
        out = (_I64 * 4)()
        if self.L.orc_shard_bounds(numel, world, rank, out) != 0:
            raise ValueError("invalid shard request")
        return tuple(int(x) for x in out)

    def memory_bytes(self, numel: int, world: int, stage: int) -> int:
        return int(self.L.orc_memory_bytes(numel, world, stage))

    # casts -------------------------------------------------------------------
    def f32_to_16(self, x, dtype: int) -> np.ndarray:
        x = np.ascontiguousarray(x, dtype=np.float32)
        out = np.empty(x.shape, dtype=np.uint16)
        self.L.orc_cast_f32_to_16(_ptr(x), _ptr(out), x.size, dtype)
        return out

    def f16_to_f32(self, h, dtype: int) -> np.ndarray:
        h = np.ascontiguousarray(h, dtype=np.uint16)
        out = np.empty(h.shape, dtype=np.float32)
        self.L.orc_cast_16_to_f32(_ptr(h), _ptr(out), h.size, dtype)
        return out

    # a1..a7 ------------------------------------------------------------------
    def reduce(self, bufs, dtype: int) -> np.ndarray:
        n = bufs[0].size
        for b in bufs:
            assert b.dtype == np.uint16 and b.size == n
        s = np.empty(n, dtype=np.float32)
        self.L.orc_reduce(ctypes.cast(_ptr_array(bufs), _P), len(bufs), n, dtype,
                          _ptr(s))
        return s

    def stats_of(self, s) -> Stats:
        s = np.ascontiguousarray(s, dtype=np.float32)
        return self.L.orc_stats_of(_ptr(s), s.size)

    def fold_stats(self, per_rank) -> Stats:
        arr = (Stats * len(per_rank))(*per_rank)
        return self.L.orc_fold_stats(ctypes.cast(arr, _P), len(per_rank))

    def decide(self, hp: Hparams, st: Scaler, global_stats: Stats,
               divisor: float) -> Decision:
        d = Decision()
        self.L.orc_decide(ctypes.byref(hp), ctypes.byref(st), global_stats,
                          divisor, ctypes.byref(d))
        return d

    def update(self, d: Decision, s, master, m, v, p16, pdtype: int) -> None:
        """master None: p16 is the master weight (low-precision masters)."""
        n = m.size
        assert master is not None or p16 is not None
        for a in (s, master, m, v):
            assert a is None or (a.size == n and a.dtype == np.float32)
        if p16 is not None:
            assert p16.size == n and p16.dtype == np.uint16
        self.L.orc_update(ctypes.byref(d), _ptr(s), _ptr(master), _ptr(m),
                          _ptr(v), _ptr(p16), n, pdtype)

    def step(self, hp: Hparams, st: Scaler, grads, gdtype: int, master, m, v,
             p16, pdtype: int, divisor: float, global_stats: Stats | None = None):
        """One shard step in place; returns (own stats, decision).  master
        None: p16 is the master weight (low-precision masters)."""
        n = m.size
        assert master is not None or p16 is not None
        for g in grads:
            assert g.dtype == np.uint16 and g.size == n and g.flags["C_CONTIGUOUS"]
        for a in (master, m, v):
            assert a is None or (a.dtype == np.float32 and a.size == n and a.flags["C_CONTIGUOUS"])
        if p16 is not None:
            assert p16.dtype == np.uint16 and p16.size == n
        own = Stats()
        dec = Decision()
        arr = _ptr_array(grads)
        gs = ctypes.byref(global_stats) if global_stats is not None else None
        rc = self.L.orc_step(ctypes.byref(hp), ctypes.byref(st),
                             ctypes.cast(arr, _P), len(grads), gdtype, n, divisor,
                             _ptr(master), _ptr(m), _ptr(v), _ptr(p16), pdtype,
                             gs, ctypes.byref(own), ctypes.byref(dec))
        if rc != 0:
            raise ValueError("oracle step rejected its arguments")
        return own, dec


    def consolidate(self, shard_masters, numel: int) -> np.ndarray:
        """Full fp32 weights from the N shards' master arrays (rank order)."""
        arrs = [np.ascontiguousarray(a, np.float32) for a in shard_masters]
        ptrs = _ptr_array(arrs)
        out = np.empty(numel, np.float32)
        self.L.orc_consolidate(ctypes.cast(ptrs, _P), len(arrs), numel, _ptr(out))
        return out


_default: Oracle | None = None


def default() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def __getattr__(name):
    # Module-level shortcuts: oracle.step(...), oracle.shard_bounds(...), ...
    if name in ("shard_bounds", "memory_bytes", "f32_to_16", "f16_to_f32",
                "reduce", "stats_of", "fold_stats", "decide", "update", "step",
                "consolidate"):
        return getattr(default(), name)
    raise AttributeError(name)
