import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)

GOLDEN = os.path.join(HERE, "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")
    config.addinivalue_line("markers", "slow: long-running test")


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()


def read_golden(name):
    """Rows of a whitespace-separated fixture, comments dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def spawn_bounded(fn, args, nprocs, seconds=300):
    """torch.multiprocessing.spawn with a time limit: children still running
    after `seconds` are terminated (SIGTERM), and any that are still alive
    after a short grace period -- e.g. blocked inside a CUDA or NCCL call that
    does not return to the interpreter -- are killed (SIGKILL); the test then
    fails instead of waiting."""
    import time

    import torch.multiprocessing as tmp
    ctx = tmp.spawn(fn, args=args, nprocs=nprocs, join=False)
    deadline = time.time() + seconds
    while not ctx.join(timeout=5):
        if time.time() > deadline:
            for p in ctx.processes:
                if p.is_alive():
                    p.terminate()
            for p in ctx.processes:
                p.join(timeout=10)
            for p in ctx.processes:
                if p.is_alive():
                    p.kill()
                    p.join(timeout=10)
            raise AssertionError(f"spawned ranks did not finish within {seconds} s")
