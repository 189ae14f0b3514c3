"""Run tables live in the handle's arena: no allocation, free or device sync
after zero_opt_create.

Each call describes its buffers to the kernels in a run table.  A training loop
whose gradient buffers move from step to step (a caching allocator, views into
bucket buffers, fresh buffers per micro-batch) makes a new table every step;
these tests step such loops against the oracle and read the handle's counters:
no device or page-locked allocation and no free happen after creation, every
new buffer set costs one table copy, and the device memory in use does not
change.  They also drive the arena's placement (a tiny arena that wraps on
every step), its size limit, and the tables kept for captured CUDA graphs.
"""
import numpy as np
import pytest

import oracle as O
import synth
from harness import assert_state, to_np16, ulp16_diff

pytestmark = pytest.mark.gpu

SEED = 0x5EED0501


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)


class Loop:
    """A flat shard stepped on the GPU and by the oracle side by side, with
    the gradients of each step written into one of `pool` preallocated device
    buffers (so that consecutive steps pass different gradient pointers)."""

    def __init__(self, n, pool, table_kib=0, clip=0.5, scale=256.0):
        import torch

        import zero_sharded_mixed_05_gb300 as z
        self.z, self.torch, self.n = z, torch, n
        dev = torch.device("cuda:0")
        self.cfg = dict(lr=1e-3, weight_decay=0.01, max_grad_norm=clip, dynamic_scale=True,
                        init_scale=scale, scale_window=20)
        self.h = z.zero_opt_create(z.make_config(numel=n, world=1, grad_dtype=z.BF16,
                                                 table_kib=table_kib, **self.cfg))
        p0 = synth.normal_np(SEED, 0, 0, n, 0.02, synth.F32)
        self.state = [torch.from_numpy(p0).to(dev), torch.zeros(n, device=dev),
                      torch.zeros(n, device=dev), torch.zeros(n, dtype=torch.bfloat16, device=dev)]
        self.pool = [torch.empty(n, dtype=torch.bfloat16, device=dev) for _ in range(pool)]
        self.orc = O.default()
        self.hp = O.hparams(lr=1e-3, weight_decay=0.01, max_grad_norm=clip, dynamic_scale=True,
                            scale_window=20)
        self.sc = O.scaler(scale)
        self.ref = (p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32),
                    np.zeros(n, np.uint16))
        self.skips = []

    def grads_np(self, step, inject):
        g = synth.normal_np(SEED, 1, step * self.n, self.n, 1e-3 * self.sc.scale, synth.BF16)
        if inject:
            g[(step * 7919) % self.n] = 0x7F80            # +inf
        return g

    def step(self, step, slot, inject=False, stream=None):
        torch = self.torch
        g = self.grads_np(step, inject)
        buf = self.pool[slot]
        buf.copy_(torch.from_numpy(g.view(np.int16)).view(torch.bfloat16))
        bufs = self.z.make_buffers(*self.state, [buf])
        self.z.zero_opt_step(self.h, 0, bufs, stream)
        _, d = self.orc.step(self.hp, self.sc, [g], O.BF16, *self.ref, O.BF16, 1.0)
        self.skips.append(int(d.skip))
        return bufs

    def check(self):
        torch = self.torch
        torch.cuda.synchronize()
        master, m, v, p16 = self.state
        assert_state("master", master.cpu().numpy(), self.ref[0])
        assert_state("m", m.cpu().numpy(), self.ref[1])
        assert_state("v", v.cpu().numpy(), self.ref[2])
        assert ulp16_diff(to_np16(p16), self.ref[3]) <= 1
        assert self.z.zero_opt_loss_scale(self.h, 0).as_tuple() == self.sc.as_tuple()

    def close(self):
        self.z.zero_opt_destroy(self.h)


def test_fresh_gradient_buffers_every_step_allocate_nothing():
    """200 steps, each with gradients in a different buffer of a pool of 80
    (more than the 64 tables the arena keeps, so every step copies a new
    table and drops the least recently used one), with overflows on steps 50
    and 150: the state matches the oracle, the counters show one table copy
    per step and no allocation or free, and free device memory is unchanged."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    loop = Loop(300_007, pool=80)
    try:
        c0 = z.zero_opt_get_counters(loop.h)
        assert c0.device_allocs == 0 and c0.device_frees == 0 and c0.table_uploads == 0
        loop.step(1, 0)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        for step in range(2, 201):
            loop.step(step, step % 80, inject=step in (50, 150))
            if step % 40 == 0:
                loop.check()
        loop.check()
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        c = z.zero_opt_get_counters(loop.h)
        assert c.device_allocs == 0 and c.device_frees == 0, c.as_dict()
        assert c.table_uploads == 200, c.as_dict()
        assert c.tables_cached == 64 and c.tables_pinned == 0, c.as_dict()
        assert c.launches == 400, c.as_dict()
        assert free1 == free0, (free0, free1)
        assert [i + 1 for i, s in enumerate(loop.skips) if s] == [50, 150]
    finally:
        loop.close()


def test_a_buffer_set_seen_before_copies_no_table():
    """The same four buffer sets in turn: four table copies in all."""
    import zero_sharded_mixed_05_gb300 as z
    loop = Loop(100_003, pool=4)
    try:
        for step in range(1, 41):
            loop.step(step, step % 4)
        loop.check()
        c = z.zero_opt_get_counters(loop.h)
        assert c.table_uploads == 4 and c.tables_cached == 4, c.as_dict()
        assert c.device_allocs == 0 and c.device_frees == 0
    finally:
        loop.close()


def test_tiny_arena_wraps_on_every_step():
    """A 1 KiB arena holds four 256-byte tables; eight buffer sets in turn
    make every step place its table over an older one.  The results still
    match the oracle, and nothing is allocated."""
    import zero_sharded_mixed_05_gb300 as z
    loop = Loop(200_003, pool=8, table_kib=1)
    try:
        for step in range(1, 61):
            loop.step(step, step % 8, inject=step == 30)
        loop.check()
        c = z.zero_opt_get_counters(loop.h)
        assert c.table_bytes == 1024 and c.table_uploads == 60, c.as_dict()
        assert c.tables_cached <= 4
        assert c.device_allocs == 0 and c.device_frees == 0
    finally:
        loop.close()


def test_table_larger_than_the_arena_is_refused_before_any_launch():
    """A list of 20 tensors needs 20 x 80 bytes of table: more than a 1 KiB
    arena.  The step fails with ZERO_ERANGE and launches nothing."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    dev = torch.device("cuda:0")
    h = z.zero_opt_create(z.make_config(numel=20 * 1000, world=1, grad_dtype=z.BF16,
                                        table_kib=1))
    try:
        items = [dict(numel=1000, master=torch.zeros(1000, device=dev),
                      m=torch.zeros(1000, device=dev), v=torch.zeros(1000, device=dev),
                      param16=torch.zeros(1000, dtype=torch.bfloat16, device=dev),
                      grads=[torch.zeros(1000, dtype=torch.bfloat16, device=dev)])
                 for _ in range(20)]
        with pytest.raises(z.ZeroOptError) as e:
            z.zero_opt_step_tensors(h, 0, z.make_tensor_list(items))
        assert e.value.status == z.ZERO_ERANGE
        assert b"arena" in z.lib().zero_opt_last_error()
        assert z.zero_opt_get_counters(h).launches == 0
        # twelve tensors fit (960 bytes)
        z.zero_opt_step_tensors(h, 0, z.make_tensor_list(items[:12]))
        torch.cuda.synchronize()
        assert z.zero_opt_get_counters(h).launches == 2
    finally:
        z.zero_opt_destroy(h)


def test_captured_table_is_kept_through_later_evictions():
    """A step captured into a CUDA graph keeps its table for the handle's
    life: after 70 eager steps on other buffer sets (which drop every other
    table), replaying the graph still steps the captured buffers, and the
    state after the whole sequence matches the oracle.  A new buffer set is
    refused under capture, before any work is enqueued."""
    import torch

    import zero_sharded_mixed_05_gb300 as z
    loop = Loop(150_001, pool=72)
    s = torch.cuda.Stream()
    try:
        with torch.cuda.stream(s):
            loop.step(1, 0, stream=s)                    # slot 0's table copied in
        s.synchronize()
        bufs0 = z.make_buffers(*loop.state, [loop.pool[0]])
        fresh = torch.empty(loop.n, dtype=torch.bfloat16, device="cuda:0")
        bufs_new = z.make_buffers(*loop.state, [fresh])
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            z.zero_opt_step(loop.h, 0, bufs0, s)
            with pytest.raises(z.ZeroOptError) as e:
                z.zero_opt_step(loop.h, 0, bufs_new, s)
        assert e.value.status == z.ZERO_ECUDA
        c = z.zero_opt_get_counters(loop.h)
        # the eager first step and the captured one launched two kernels each
        assert c.tables_pinned == 1 and c.launches == 4, c.as_dict()
        with torch.cuda.stream(s):
            for step in range(2, 72):
                loop.step(step, step - 1, stream=s)      # slots 1..70
            # the graph's step, on slot 0's buffer
            g = loop.grads_np(72, False)
            loop.pool[0].copy_(torch.from_numpy(g.view(np.int16)).view(torch.bfloat16))
            graph.replay()
        _, d = loop.orc.step(loop.hp, loop.sc, [g], O.BF16, *loop.ref, O.BF16, 1.0)
        loop.check()
        c = z.zero_opt_get_counters(loop.h)
        assert c.tables_pinned == 1 and c.table_uploads == 71, c.as_dict()
        assert c.device_allocs == 0 and c.device_frees == 0
    finally:
        s.synchronize()
        loop.close()
