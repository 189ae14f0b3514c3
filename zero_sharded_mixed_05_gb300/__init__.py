"""GB300 per-shard mixed-precision ZeRO optimizer step.

A thin ctypes binding of the C ABI in ``include/zero_opt.h``: the functions
here carry the same names as the C entry points and only marshal arguments
(torch tensors become device pointers, the current torch stream becomes the
``cudaStream_t``).  Every step of the computation runs in the library's CUDA
kernels (``csrc/``); there is no Python or CPU fallback, and importing this
package fails loudly when the compiled library is missing.

Build the library with ``zero_sharded_mixed_05_gb300._build.build()`` (or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

from . import _build

FP16 = 0
BF16 = 1

ZERO_OK, ZERO_EINVAL, ZERO_ERANGE, ZERO_ENOMEM, ZERO_ECUDA, ZERO_ENOTSUP = range(6)

_i32, _i64, _f32, _f64, _vp = (ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                              ctypes.c_double, ctypes.c_void_p)


class zero_opt_config(ctypes.Structure):
    _fields_ = [("numel", _i64), ("world", _i32), ("grad_dtype", _i32),
                ("param_dtype", _i32), ("bias_correction", _i32),
                ("lr", _f64), ("beta1", _f64), ("beta2", _f64), ("eps", _f64),
                ("weight_decay", _f64), ("max_grad_norm", _f64),
                ("dynamic_scale", _i32), ("hysteresis", _i32),
                ("init_scale", _f64), ("min_scale", _f64), ("scale_factor", _f64),
                ("scale_window", _i64), ("warmup_min_lr", _f64), ("warmup_max_lr", _f64),
                ("warmup_num_steps", _i64), ("master16", _i32), ("table_kib", _i32)]


class zero_opt_buffers(ctypes.Structure):
    _fields_ = [("master", _vp), ("m", _vp), ("v", _vp), ("param16", _vp),
                ("grads", ctypes.POINTER(_vp)), ("n_ranks", _i32), ("n_micro", _i32),
                ("grads_shard_local", _i32), ("param16_shard_local", _i32),
                ("divisor", _f64), ("stash", _vp)]


class zero_opt_tensor(ctypes.Structure):
    _fields_ = [("numel", _i64), ("master", _vp), ("m", _vp), ("v", _vp),
                ("param16", _vp), ("grads", ctypes.POINTER(_vp))]


class zero_opt_tensor_list(ctypes.Structure):
    _fields_ = [("tensors", ctypes.POINTER(zero_opt_tensor)), ("n_tensors", _i32),
                ("n_ranks", _i32), ("n_micro", _i32), ("divisor", _f64),
                ("stash", _vp)]


class zero_opt_stats(ctypes.Structure):
    _fields_ = [("sumsq", _f64), ("nonfinite", _i32), ("reserved", _i32)]


class zero_opt_step_info(ctypes.Structure):
    _fields_ = [("sumsq", _f64), ("norm", _f64), ("coef", _f32), ("scale_used", _f32),
                ("skipped", _i32), ("nonfinite", _i32), ("t", _i64), ("fault", _i32),
                ("reserved", _i32)]


class zero_opt_scaler_state(ctypes.Structure):
    _fields_ = [("scale", _f32), ("last_skipped", _i32), ("clean_steps", _i64),
                ("t", _i64), ("skipped_total", _i64), ("overflows", _i32),
                ("reserved", _i32)]

    def as_tuple(self):
        """(scale, clean_steps, t, skipped_total, last_skipped)."""
        return (float(self.scale), int(self.clean_steps), int(self.t),
                int(self.skipped_total), int(self.last_skipped))


class zero_opt_counters(ctypes.Structure):
    _fields_ = [("launches", _i64), ("table_uploads", _i64), ("table_waits", _i64),
                ("device_allocs", _i64), ("device_frees", _i64), ("tables_cached", _i64),
                ("tables_pinned", _i64), ("table_bytes", _i64)]

    def as_dict(self):
        return {name: int(getattr(self, name)) for name, _ in self._fields_}


class zero_opt_ckpt_info(ctypes.Structure):
    _fields_ = [("numel", _i64), ("world", _i32), ("rank", _i32), ("begin", _i64),
                ("real_len", _i64), ("scaler", zero_opt_scaler_state)]


class ZeroOptError(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        super().__init__(f"{where}: status {status}: {message}")
        self.status = status


# ---------------------------------------------------------------- loading

LIB_PATH = _build.LIB

# (name, restype, argtypes) of every entry point in include/zero_opt.h
_P = ctypes.POINTER
SIGNATURES = [
    ("zero_opt_config_default", _i32, [_P(zero_opt_config)]),
    ("zero_opt_create", _i32, [_P(zero_opt_config), _P(_vp)]),
    ("zero_opt_destroy", _i32, [_vp]),
    ("zero_opt_shard_bounds", _i32, [_vp, _i32, _P(_i64), _P(_i64), _P(_i64), _P(_i64)]),
    ("zero_opt_memory_bytes", _i32, [_i64, _i32, _i32, _P(_i64)]),
    ("zero_opt_grad_stats", _i32, [_vp, _i32, _P(zero_opt_buffers), _vp, _P(zero_opt_stats)]),
    ("zero_opt_fold_stats", _i32, [_P(zero_opt_stats), _i32, _P(zero_opt_stats)]),
    ("zero_opt_step", _i32, [_vp, _i32, _P(zero_opt_buffers), _vp, _P(zero_opt_stats)]),
    ("zero_opt_grad_stats_async", _i32, [_vp, _i32, _P(zero_opt_buffers), _vp, _vp]),
    ("zero_opt_step_folded", _i32, [_vp, _i32, _P(zero_opt_buffers), _vp, _vp, _i32]),
    ("zero_opt_grad_stats_tensors", _i32,
     [_vp, _i32, _P(zero_opt_tensor_list), _vp, _P(zero_opt_stats)]),
    ("zero_opt_step_tensors", _i32,
     [_vp, _i32, _P(zero_opt_tensor_list), _vp, _P(zero_opt_stats)]),
    ("zero_opt_loss_scale", _i32, [_vp, _i32, _vp, _P(zero_opt_scaler_state)]),
    ("zero_opt_set_loss_scale", _i32, [_vp, _i32, _vp, _P(zero_opt_scaler_state)]),
    ("zero_opt_set_lr", _i32, [_vp, _f64]),
    ("zero_opt_last_step", _i32, [_vp, _vp, _P(zero_opt_step_info)]),
    ("zero_opt_set_events", _i32, [_vp, _vp, _vp, _vp]),
    ("zero_opt_inject_wait_fault", _i32, [_vp]),
    ("zero_opt_launch_count", _i32, [_vp, _P(_i64)]),
    ("zero_opt_get_counters", _i32, [_vp, _P(zero_opt_counters)]),
    ("zero_opt_ckpt_write", _i32, [ctypes.c_char_p, _P(zero_opt_ckpt_info), _vp, _vp, _vp]),
    ("zero_opt_ckpt_read", _i32, [ctypes.c_char_p, _P(zero_opt_ckpt_info), _vp, _vp, _vp]),
    ("zero_opt_save_shard", _i32, [_vp, _i32, _vp, _vp, _vp, _vp, ctypes.c_char_p]),
    ("zero_opt_save_shard16", _i32, [_vp, _i32, _vp, _i32, _vp, _vp, _vp, ctypes.c_char_p]),
    ("zero_opt_load_shard", _i32, [_vp, _i32, _vp, _vp, _vp, _vp, _i32, _vp, ctypes.c_char_p]),
    ("zero_opt_consolidate_fp32", _i32, [_P(ctypes.c_char_p), _i32, _i64, _vp]),
    ("zero_opt_grad_stats_noalloc", _i32, [_P(_vp), _i32, _i32, _i64, _vp, _vp]),
    ("zero_host_create", _i32, [_P(zero_opt_config), _i32, _P(_vp)]),
    ("zero_host_destroy", _i32, [_vp]),
    ("zero_host_threads", _i32, [_vp, _P(_i32)]),
    ("zero_host_grad_stats", _i32, [_vp, _i32, _P(zero_opt_buffers), _P(zero_opt_stats)]),
    ("zero_host_step", _i32, [_vp, _i32, _P(zero_opt_buffers), _P(zero_opt_stats)]),
    ("zero_host_grad_stats_tensors", _i32,
     [_vp, _i32, _P(zero_opt_tensor_list), _P(zero_opt_stats)]),
    ("zero_host_step_tensors", _i32, [_vp, _i32, _P(zero_opt_tensor_list), _P(zero_opt_stats)]),
    ("zero_host_loss_scale", _i32, [_vp, _i32, _P(zero_opt_scaler_state)]),
    ("zero_host_set_loss_scale", _i32, [_vp, _i32, _P(zero_opt_scaler_state)]),
    ("zero_host_last_step", _i32, [_vp, _P(zero_opt_step_info)]),
    ("zero_opt_status_string", ctypes.c_char_p, [_i32]),
    ("zero_opt_last_error", ctypes.c_char_p, []),
]

_lib = None


def lib():
    """The loaded CUDA library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: the CUDA library must be built first "
                "(zero_sharded_mixed_05_gb300._build.build()); there is no fallback")
        L = ctypes.CDLL(LIB_PATH)
        for name, res, args in SIGNATURES:
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def _check(status: int, where: str) -> None:
    if status != ZERO_OK:
        msg = lib().zero_opt_last_error().decode(errors="replace")
        raise ZeroOptError(status, where, msg)


def _ptr(x):
    """Address of a torch tensor or numpy array (or an int address)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return x.ctypes.data


def current_stream(device=None) -> int:
    import torch
    return torch.cuda.current_stream(device).cuda_stream


def _stream(s):
    if s is None:
        import torch
        if torch.cuda.is_available():
            return current_stream()
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def dtype_code(torch_dtype) -> int:
    import torch
    if torch_dtype == torch.float16:
        return FP16
    if torch_dtype == torch.bfloat16:
        return BF16
    raise ValueError(f"unsupported 16-bit dtype {torch_dtype}")


# ---------------------------------------------------------------- descriptors

def make_config(numel=0, world=1, grad_dtype=FP16, param_dtype=None, lr=2e-5,
                betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01, max_grad_norm=0.0,
                bias_correction=True, dynamic_scale=True, init_scale=65536.0,
                min_scale=1.0, scale_factor=2.0, scale_window=1000,
                hysteresis=1, warmup=(0.0, 0.0, 0), master16=False,
                table_kib=0) -> zero_opt_config:
    """`warmup` = (warmup_min_lr, warmup_max_lr, warmup_num_steps); 0 steps
    keeps lr constant.  `master16`: the 16-bit parameters are the master
    weights (no fp32 master array).  `table_kib`: KiB of the handle's
    run-table arena (0: 1024)."""
    cfg = zero_opt_config()
    _check(lib().zero_opt_config_default(ctypes.byref(cfg)), "zero_opt_config_default")
    cfg.numel = numel
    cfg.world = world
    cfg.grad_dtype = grad_dtype
    cfg.param_dtype = grad_dtype if param_dtype is None else param_dtype
    cfg.lr = lr
    cfg.beta1, cfg.beta2 = betas
    cfg.eps = eps
    cfg.weight_decay = weight_decay
    cfg.max_grad_norm = max_grad_norm
    cfg.bias_correction = int(bias_correction)
    cfg.dynamic_scale = int(dynamic_scale)
    cfg.init_scale = init_scale
    cfg.min_scale = min_scale
    cfg.scale_factor = scale_factor
    cfg.scale_window = scale_window
    cfg.hysteresis = hysteresis
    cfg.warmup_min_lr, cfg.warmup_max_lr, cfg.warmup_num_steps = warmup
    cfg.master16 = int(master16)
    cfg.table_kib = int(table_kib)
    return cfg


def _ptr_array(items):
    arr = (_vp * max(len(items), 1))()
    for i, g in enumerate(items):
        arr[i] = _ptr(g)
    return arr


def make_buffers(master, m, v, param16, grads, n_ranks=None, n_micro=1,
                 grads_shard_local=False, param16_shard_local=False, divisor=0.0,
                 stash=None) -> zero_opt_buffers:
    """Flat-shard buffers; `grads` lists the R*K gradient buffers rank-major."""
    grads = list(grads)
    if n_ranks is None:
        n_ranks = len(grads) // n_micro
    arr = _ptr_array(grads)
    b = zero_opt_buffers(_ptr(master), _ptr(m), _ptr(v), _ptr(param16),
                         ctypes.cast(arr, _P(_vp)), n_ranks, n_micro,
                         int(grads_shard_local), int(param16_shard_local),
                         float(divisor), _ptr(stash))
    b._keep = (arr, grads, master, m, v, param16, stash)
    return b


def make_tensor_list(tensors, n_ranks=1, n_micro=1, divisor=0.0,
                     stash=None) -> zero_opt_tensor_list:
    """Per-tensor list; each item is a dict with numel (optional), master, m, v,
    param16 and grads (R*K tensors, rank-major)."""
    items = (zero_opt_tensor * max(len(tensors), 1))()
    keep = []
    for i, t in enumerate(tensors):
        garr = _ptr_array(t["grads"])
        keep.append((garr, t))
        numel = t["numel"] if "numel" in t else t["master"].numel()
        items[i] = zero_opt_tensor(numel, _ptr(t["master"]), _ptr(t["m"]), _ptr(t["v"]),
                                   _ptr(t["param16"]), ctypes.cast(garr, _P(_vp)))
    lst = zero_opt_tensor_list(ctypes.cast(items, _P(zero_opt_tensor)), len(tensors),
                               n_ranks, n_micro, float(divisor), _ptr(stash))
    lst._keep = (items, keep, stash)
    return lst


# ---------------------------------------------------------------- entry points

def zero_opt_config_default() -> zero_opt_config:
    cfg = zero_opt_config()
    _check(lib().zero_opt_config_default(ctypes.byref(cfg)), "zero_opt_config_default")
    return cfg


def zero_opt_create(cfg: zero_opt_config) -> int:
    h = _vp()
    _check(lib().zero_opt_create(ctypes.byref(cfg), ctypes.byref(h)), "zero_opt_create")
    return h.value


def zero_opt_destroy(h) -> None:
    _check(lib().zero_opt_destroy(h), "zero_opt_destroy")


def zero_opt_shard_bounds(h, rank: int):
    """(begin, real_end, shard_len, padded_numel)."""
    out = [_i64() for _ in range(4)]
    _check(lib().zero_opt_shard_bounds(h, rank, *[ctypes.byref(o) for o in out]),
           "zero_opt_shard_bounds")
    return tuple(o.value for o in out)


def zero_opt_memory_bytes(numel: int, world: int, stage: int) -> int:
    out = _i64()
    _check(lib().zero_opt_memory_bytes(numel, world, stage, ctypes.byref(out)),
           "zero_opt_memory_bytes")
    return out.value


def zero_opt_grad_stats(h, rank: int, bufs: zero_opt_buffers, stream=None) -> zero_opt_stats:
    out = zero_opt_stats()
    _check(lib().zero_opt_grad_stats(h, rank, ctypes.byref(bufs), _stream(stream),
                                     ctypes.byref(out)), "zero_opt_grad_stats")
    return out


def zero_opt_step(h, rank: int, bufs: zero_opt_buffers, stream=None,
                  global_stats: zero_opt_stats | None = None) -> None:
    gs = ctypes.byref(global_stats) if global_stats is not None else None
    _check(lib().zero_opt_step(h, rank, ctypes.byref(bufs), _stream(stream), gs),
           "zero_opt_step")


def zero_opt_grad_stats_async(h, rank: int, bufs: zero_opt_buffers, out_dev,
                              stream=None) -> None:
    """Shard statistics into `out_dev`, a device buffer of 16 bytes (one
    zero_opt_stats), without synchronizing."""
    _check(lib().zero_opt_grad_stats_async(h, rank, ctypes.byref(bufs), _stream(stream),
                                           _ptr(out_dev)), "zero_opt_grad_stats_async")


def zero_opt_step_folded(h, rank: int, bufs: zero_opt_buffers, per_rank_dev, n: int,
                         stream=None) -> None:
    """Step with the global statistics folded on the device from `n` per-rank
    zero_opt_stats records at `per_rank_dev` (device, rank order)."""
    _check(lib().zero_opt_step_folded(h, rank, ctypes.byref(bufs), _stream(stream),
                                      _ptr(per_rank_dev), n), "zero_opt_step_folded")


def zero_opt_grad_stats_tensors(h, rank: int, lst: zero_opt_tensor_list,
                                stream=None) -> zero_opt_stats:
    out = zero_opt_stats()
    _check(lib().zero_opt_grad_stats_tensors(h, rank, ctypes.byref(lst), _stream(stream),
                                             ctypes.byref(out)),
           "zero_opt_grad_stats_tensors")
    return out


def zero_opt_step_tensors(h, rank: int, lst: zero_opt_tensor_list, stream=None,
                          global_stats: zero_opt_stats | None = None) -> None:
    gs = ctypes.byref(global_stats) if global_stats is not None else None
    _check(lib().zero_opt_step_tensors(h, rank, ctypes.byref(lst), _stream(stream), gs),
           "zero_opt_step_tensors")


def zero_opt_loss_scale(h, rank: int, stream=None) -> zero_opt_scaler_state:
    out = zero_opt_scaler_state()
    _check(lib().zero_opt_loss_scale(h, rank, _stream(stream), ctypes.byref(out)),
           "zero_opt_loss_scale")
    return out


def zero_opt_set_loss_scale(h, rank: int, state: zero_opt_scaler_state, stream=None) -> None:
    _check(lib().zero_opt_set_loss_scale(h, rank, _stream(stream), ctypes.byref(state)),
           "zero_opt_set_loss_scale")


def zero_opt_set_lr(h, lr: float) -> None:
    _check(lib().zero_opt_set_lr(h, lr), "zero_opt_set_lr")


def zero_opt_last_step(h, stream=None) -> zero_opt_step_info:
    out = zero_opt_step_info()
    _check(lib().zero_opt_last_step(h, _stream(stream), ctypes.byref(out)),
           "zero_opt_last_step")
    return out


def zero_opt_set_events(h, ev_start=None, ev_mid=None, ev_end=None) -> None:
    """Record torch.cuda.Event objects (or raw cudaEvent_t ints) around the
    passes of subsequent steps; no arguments turns the hook off."""
    def raw(e):
        if e is None or isinstance(e, int):
            return e
        return e.cuda_event
    _check(lib().zero_opt_set_events(h, raw(ev_start), raw(ev_mid), raw(ev_end)),
           "zero_opt_set_events")


def zero_opt_inject_wait_fault(h) -> None:
    """Arm the failure-detection test hook for the next statistics pass."""
    _check(lib().zero_opt_inject_wait_fault(h), "zero_opt_inject_wait_fault")


def zero_opt_launch_count(h) -> int:
    out = _i64()
    _check(lib().zero_opt_launch_count(h, ctypes.byref(out)), "zero_opt_launch_count")
    return out.value


def zero_opt_get_counters(h) -> zero_opt_counters:
    """Launches, run-table uploads and waits, and allocations after creation."""
    out = zero_opt_counters()
    _check(lib().zero_opt_get_counters(h, ctypes.byref(out)), "zero_opt_get_counters")
    return out


def zero_opt_status_string(status: int) -> str:
    return lib().zero_opt_status_string(status).decode()


def zero_opt_fold_stats(per_rank) -> zero_opt_stats:
    """The scalar all-reduce of per-rank statistics, folded in rank order."""
    per_rank = list(per_rank)
    arr = (zero_opt_stats * max(len(per_rank), 1))(*per_rank)
    out = zero_opt_stats()
    _check(lib().zero_opt_fold_stats(arr, len(per_rank), ctypes.byref(out)),
           "zero_opt_fold_stats")
    return out


def allgather_fold(own: zero_opt_stats, group=None) -> zero_opt_stats:
    """The scalar all-reduce of a multi-process run: every rank contributes its
    shard's statistics, all ranks receive all of them (torch.distributed
    all_gather on a tiny tensor) and fold them in rank order with
    zero_opt_fold_stats, so every rank gets bit-identical totals."""
    import torch
    import torch.distributed as dist
    ws = dist.get_world_size(group)
    mine = torch.tensor([own.sumsq, float(own.nonfinite)], dtype=torch.float64)
    if dist.get_backend(group) == "nccl":
        mine = mine.cuda()
    parts = [torch.empty_like(mine) for _ in range(ws)]
    dist.all_gather(parts, mine, group=group)
    per = [zero_opt_stats(float(p[0]), int(p[1]), 0) for p in (q.cpu() for q in parts)]
    return zero_opt_fold_stats(per)


# ---------------------------------------------------------------- checkpoints

def _np_ptr(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"] and a.dtype.itemsize == 4
    return a.ctypes.data


def zero_opt_ckpt_write(path: str, info: zero_opt_ckpt_info, master, m, v) -> None:
    """Write one shard file from host float32 numpy arrays."""
    _check(lib().zero_opt_ckpt_write(os.fsencode(path), ctypes.byref(info), _np_ptr(master),
                                     _np_ptr(m), _np_ptr(v)), "zero_opt_ckpt_write")


def zero_opt_ckpt_read(path: str, with_payload: bool = True):
    """(info, master, m, v) of a shard file, arrays as host numpy float32."""
    import numpy as np
    info = zero_opt_ckpt_info()
    _check(lib().zero_opt_ckpt_read(os.fsencode(path), ctypes.byref(info), None, None, None),
           "zero_opt_ckpt_read")
    if not with_payload:
        return info, None, None, None
    arrs = [np.empty(info.real_len, np.float32) for _ in range(3)]
    _check(lib().zero_opt_ckpt_read(os.fsencode(path), ctypes.byref(info),
                                    *[_np_ptr(a) for a in arrs]), "zero_opt_ckpt_read")
    return (info, *arrs)


def zero_opt_save_shard(h, rank: int, master, m, v, path: str, stream=None) -> None:
    _check(lib().zero_opt_save_shard(h, rank, _ptr(master), _ptr(m), _ptr(v), _stream(stream),
                                     os.fsencode(path)), "zero_opt_save_shard")


def zero_opt_save_shard16(h, rank: int, param16, m, v, path: str,
                          param16_shard_local: bool = False, stream=None) -> None:
    """Shard file of a master16 handle: its 16-bit masters (widened exactly), m, v
    and loss-scaler replica."""
    _check(lib().zero_opt_save_shard16(h, rank, _ptr(param16), int(param16_shard_local),
                                       _ptr(m), _ptr(v), _stream(stream), os.fsencode(path)),
           "zero_opt_save_shard16")


def zero_opt_load_shard(h, rank: int, master, m, v, path: str, param16=None,
                        param16_shard_local: bool = False, stream=None) -> None:
    _check(lib().zero_opt_load_shard(h, rank, _ptr(master), _ptr(m), _ptr(v), _ptr(param16),
                                     int(param16_shard_local), _stream(stream),
                                     os.fsencode(path)), "zero_opt_load_shard")


def zero_opt_consolidate_fp32(paths, numel: int):
    """Full fp32 master weights (numpy) merged from one checkpoint's shard files."""
    import numpy as np
    arr = (ctypes.c_char_p * len(paths))(*[os.fsencode(p) for p in paths])
    out = np.empty(numel, np.float32)
    _check(lib().zero_opt_consolidate_fp32(arr, len(paths), numel, _np_ptr(out)),
           "zero_opt_consolidate_fp32")
    return out


def zero_opt_grad_stats_noalloc(grads, grad_dtype: int, n: int, out, stream=None) -> None:
    """Statistics of the sum of `grads` (device tensors) written into `out`, a
    device buffer of at least 16 bytes holding one zero_opt_stats; allocates
    nothing on the device.

    The C entry point receives bare pointers and cannot check them, so this
    binding does: every gradient must be a contiguous CUDA tensor of the
    current device with the dtype `grad_dtype` names and at least `n`
    elements, and `out` a contiguous CUDA tensor of the current device of at
    least 16 bytes.  Anything else raises ValueError before a launch."""
    import torch
    want = {FP16: torch.float16, BF16: torch.bfloat16}.get(grad_dtype)
    if want is None:
        raise ValueError(f"grad_dtype must be FP16 or BF16, not {grad_dtype}")
    grads = list(grads)
    dev = torch.cuda.current_device()

    def on_device(t):
        return isinstance(t, torch.Tensor) and t.is_cuda and t.device.index == dev \
            and t.is_contiguous()
    for i, g in enumerate(grads):
        if not on_device(g):
            raise ValueError(f"grads[{i}] must be a contiguous CUDA tensor on device {dev}")
        if g.dtype != want:
            raise ValueError(f"grads[{i}] is {g.dtype}, grad_dtype names {want}")
        if g.numel() < n:
            raise ValueError(f"grads[{i}] holds {g.numel()} elements, fewer than n = {n}")
    if not on_device(out) or out.numel() * out.element_size() < 16:
        raise ValueError(f"out must be a contiguous CUDA tensor on device {dev} of at least "
                         "16 bytes (one zero_opt_stats)")
    arr = _ptr_array(grads)
    _check(lib().zero_opt_grad_stats_noalloc(ctypes.cast(arr, _P(_vp)), len(grads), grad_dtype,
                                             n, _stream(stream), _ptr(out)),
           "zero_opt_grad_stats_noalloc")


# ---------------------------------------------------------------- offloaded (host) step
# Same calls on host-resident buffers (numpy arrays or CPU tensors); no GPU.

def zero_host_create(cfg: zero_opt_config, n_threads: int = 0) -> int:
    h = _vp()
    _check(lib().zero_host_create(ctypes.byref(cfg), n_threads, ctypes.byref(h)),
           "zero_host_create")
    return h.value


def zero_host_destroy(h) -> None:
    _check(lib().zero_host_destroy(h), "zero_host_destroy")


def zero_host_threads(h) -> int:
    n = _i32()
    _check(lib().zero_host_threads(h, ctypes.byref(n)), "zero_host_threads")
    return n.value


def zero_host_grad_stats(h, rank: int, bufs: zero_opt_buffers) -> zero_opt_stats:
    out = zero_opt_stats()
    _check(lib().zero_host_grad_stats(h, rank, ctypes.byref(bufs), ctypes.byref(out)),
           "zero_host_grad_stats")
    return out


def zero_host_step(h, rank: int, bufs: zero_opt_buffers, global_stats=None) -> None:
    gs = ctypes.byref(global_stats) if global_stats is not None else None
    _check(lib().zero_host_step(h, rank, ctypes.byref(bufs), gs), "zero_host_step")


def zero_host_grad_stats_tensors(h, rank: int, lst: zero_opt_tensor_list) -> zero_opt_stats:
    out = zero_opt_stats()
    _check(lib().zero_host_grad_stats_tensors(h, rank, ctypes.byref(lst), ctypes.byref(out)),
           "zero_host_grad_stats_tensors")
    return out


def zero_host_step_tensors(h, rank: int, lst: zero_opt_tensor_list, global_stats=None) -> None:
    gs = ctypes.byref(global_stats) if global_stats is not None else None
    _check(lib().zero_host_step_tensors(h, rank, ctypes.byref(lst), gs), "zero_host_step_tensors")


def zero_host_loss_scale(h, rank: int) -> zero_opt_scaler_state:
    out = zero_opt_scaler_state()
    _check(lib().zero_host_loss_scale(h, rank, ctypes.byref(out)), "zero_host_loss_scale")
    return out


def zero_host_set_loss_scale(h, rank: int, state: zero_opt_scaler_state) -> None:
    _check(lib().zero_host_set_loss_scale(h, rank, ctypes.byref(state)),
           "zero_host_set_loss_scale")


def zero_host_last_step(h) -> zero_opt_step_info:
    out = zero_opt_step_info()
    _check(lib().zero_host_last_step(h, ctypes.byref(out)), "zero_host_last_step")
    return out
