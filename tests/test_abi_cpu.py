"""The C ABI on the host: exported symbols, argument validation and the
host-only calls (shard bounds, memory forms, statistics fold) against the
oracle.  No test here launches a kernel."""
import ctypes
import glob
import os
import re

import numpy as np
import pytest

import oracle as O

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def z():
    from zero_sharded_mixed_05_gb300 import _build
    _build.build()
    import zero_sharded_mixed_05_gb300 as z
    z.lib()
    return z


def _declared_functions():
    names = []
    for hdr in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(hdr).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:zero_status|const\s+char\s*\*)\s*(\w+)\s*\(", text, re.M)
    return names


def test_every_declared_symbol_is_exported(z):
    names = _declared_functions()
    assert len(names) == len(z.SIGNATURES)
    lib = ctypes.CDLL(z.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    bound = {s[0] for s in z.SIGNATURES}
    assert set(names) <= bound, set(names) - bound


def test_config_default_is_the_ds_config(z):
    c = z.zero_opt_config_default()
    assert (c.lr, c.beta1, c.beta2, c.eps, c.weight_decay) == (2e-5, 0.9, 0.999, 1e-8, 0.01)
    assert c.init_scale == 2.0 ** 16 and c.scale_window == 1000 and c.min_scale == 1.0
    assert c.dynamic_scale == 1 and c.hysteresis == 2 and c.bias_correction == 1
    assert c.warmup_num_steps == 0


@pytest.mark.parametrize("field,value,status", [
    ("numel", -1, 1), ("world", 0, 1), ("grad_dtype", 7, 1), ("param_dtype", -1, 1),
    ("lr", -1e-3, 1), ("beta1", 1.0, 1), ("beta2", -0.1, 1), ("eps", 0.0, 1),
    ("weight_decay", -0.5, 1), ("init_scale", 0.0, 1), ("min_scale", -1.0, 1),
    ("scale_factor", 0.5, 1), ("scale_window", 0, 1), ("bias_correction", 2, 1),
    ("hysteresis", 0, 1), ("max_grad_norm", float("nan"), 1), ("warmup_num_steps", -1, 1),
    ("warmup_max_lr", -1e-3, 1), ("table_kib", -1, 1), ("table_kib", (1 << 20) + 1, 1),
])
def test_create_rejects_bad_config(z, field, value, status):
    cfg = z.make_config(numel=100, world=2)
    setattr(cfg, field, value)
    h = ctypes.c_void_p(123)
    rc = z.lib().zero_opt_create(ctypes.byref(cfg), ctypes.byref(h))
    assert rc == status
    assert h.value is None
    assert z.lib().zero_opt_last_error()


def test_null_arguments(z):
    L = z.lib()
    assert L.zero_opt_create(None, None) == z.ZERO_EINVAL
    assert L.zero_opt_shard_bounds(None, 0, None, None, None, None) == z.ZERO_EINVAL
    assert L.zero_opt_memory_bytes(10, 1, 0, None) == z.ZERO_EINVAL
    assert L.zero_opt_step(None, 0, None, None, None) == z.ZERO_EINVAL
    assert L.zero_opt_fold_stats(None, 1, None) == z.ZERO_EINVAL
    assert L.zero_opt_destroy(None) == z.ZERO_OK
    assert z.zero_opt_status_string(4).startswith("ZERO_ECUDA")


@pytest.fixture()
def handle(z):
    h = z.zero_opt_create(z.make_config(numel=1_000_003, world=4))
    yield h
    z.zero_opt_destroy(h)


def test_shard_bounds_match_oracle(z):
    for numel in [0, 1, 3, 4, 5, 1_000_003, 124_439_808, 8_030_261_248]:
        for world in [1, 2, 3, 4, 8, 7]:
            h = z.zero_opt_create(z.make_config(numel=numel, world=world))
            try:
                for r in range(world):
                    assert z.zero_opt_shard_bounds(h, r) == O.shard_bounds(numel, world, r)
            finally:
                z.zero_opt_destroy(h)


def test_shard_bounds_rank_range(z, handle):
    with pytest.raises(z.ZeroOptError) as e:
        z.zero_opt_shard_bounds(handle, 4)
    assert e.value.status == z.ZERO_ERANGE
    with pytest.raises(z.ZeroOptError):
        z.zero_opt_shard_bounds(handle, -1)


def test_memory_bytes_match_oracle(z):
    for numel in [0, 1, 7, 1_000_003, 7_000_000_000, 8_030_261_248]:
        for world in [1, 2, 3, 8, 64]:
            for stage in range(4):
                assert z.zero_opt_memory_bytes(numel, world, stage) == O.memory_bytes(numel, world, stage)
    with pytest.raises(z.ZeroOptError) as e:
        z.zero_opt_memory_bytes(10, 1, 4)
    assert e.value.status == z.ZERO_ERANGE


def test_fold_matches_oracle(z):
    rng = np.random.default_rng(3)
    vals = rng.random(9) * 10.0 ** rng.integers(-5, 5, 9)
    flags = [0, 0, 1, 0, 0, 0, 0, 0, 0]
    ours = z.zero_opt_fold_stats([z.zero_opt_stats(v, f, 0) for v, f in zip(vals, flags)])
    ref = O.fold_stats([O.Stats(v, f, 0) for v, f in zip(vals, flags)])
    assert ours.sumsq == ref.sumsq and ours.nonfinite == ref.nonfinite == 1
    assert z.zero_opt_fold_stats([]).sumsq == 0.0


def _fake(addr):
    return addr  # a pointer value that is never dereferenced by validation


@pytest.mark.parametrize("case,status", [
    ("grads_null", 1), ("rk_zero", 1), ("rk_too_many", 1), ("master_null", 1),
    ("grad_entry_null", 1), ("rank_range", 2),
])
def test_step_validation(z, handle, case, status):
    grads = [_fake(0x1000 * (i + 1)) for i in range(4)]
    b = z.make_buffers(0x10000, 0x20000, 0x30000, 0x40000, grads)
    rank = 0
    if case == "grads_null":
        b.grads = None
    elif case == "rk_zero":
        b.n_ranks = 0
    elif case == "rk_too_many":
        b.n_ranks, b.n_micro = 64, 17
    elif case == "master_null":
        b.master = None
    elif case == "grad_entry_null":
        b._keep[0][2] = None
    elif case == "rank_range":
        rank = 9
    L = z.lib()
    assert L.zero_opt_step(handle, rank, ctypes.byref(b), None, None) == status
    out = z.zero_opt_stats()
    assert L.zero_opt_grad_stats(handle, rank, ctypes.byref(b), None, ctypes.byref(out)) == status


def test_tensor_list_validation(z, handle):
    t = [dict(numel=10, master=0x10, m=0x20, v=0x30, param16=None, grads=[0x40])]
    lst = z.make_tensor_list(t)
    assert z.lib().zero_opt_step_tensors(handle, 0, ctypes.byref(lst), None, None) == z.ZERO_EINVAL
    t[0]["numel"] = -1
    lst = z.make_tensor_list(t)
    assert z.lib().zero_opt_step_tensors(handle, 0, ctypes.byref(lst), None, None) == z.ZERO_EINVAL


def test_valid_step_without_device_is_a_cuda_error(z, handle):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a CUDA device is present")
    grads = [0x1000 * (i + 1) for i in range(4)]
    b = z.make_buffers(0x10000, 0x20000, 0x30000, 0x40000, grads)
    assert z.lib().zero_opt_step(handle, 1, ctypes.byref(b), None, None) == z.ZERO_ECUDA
    st = z.zero_opt_scaler_state()
    assert z.lib().zero_opt_loss_scale(handle, 0, None, ctypes.byref(st)) == z.ZERO_ECUDA


def test_set_lr_validation(z, handle):
    z.zero_opt_set_lr(handle, 1e-4)
    with pytest.raises(z.ZeroOptError):
        z.zero_opt_set_lr(handle, -1.0)


def test_counters_of_a_fresh_handle(z, handle):
    """zero_opt_get_counters: nothing launched, uploaded or allocated after
    creation; NULL arguments are rejected."""
    c = z.zero_opt_get_counters(handle)
    assert c.as_dict() == {"launches": 0, "table_uploads": 0, "table_waits": 0,
                           "device_allocs": 0, "device_frees": 0, "tables_cached": 0,
                           "tables_pinned": 0, "table_bytes": c.table_bytes}
    assert z.lib().zero_opt_get_counters(None, ctypes.byref(c)) == z.ZERO_EINVAL
    assert z.lib().zero_opt_get_counters(handle, None) == z.ZERO_EINVAL
