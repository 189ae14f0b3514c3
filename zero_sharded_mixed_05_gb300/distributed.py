"""The ZeRO-2 data-parallel step across processes: the exchanges around the
per-shard step.

Sources: "DeepSpeed framework interview answer" (algomooc.com), "ZeRO 三阶段",
and "LLM-train tutorials ch01" (jwzheng96.github.io) §1.2 stage table: the
gradients are reduce-scattered so that each rank holds the reduced gradient of
its own shard, each rank updates only its shard of the optimizer state, and the
updated 16-bit parameters are all-gathered.  Every rank also needs the global
overflow flag and gradient norm, a two-scalar all-reduce.

How the exchanges are done here:

- Reduce-scatter is split into its two halves.  The transport half is an
  all-to-all of the raw 16-bit bytes: rank r receives, from every rank j, rank
  j's gradient values of shard r (for every micro-step).  The reduction half is
  this library's kernel: the owner sums the N ranks' x K micro-steps' buffers
  in binary32, rank-major, exactly as the one-process step sums N simulated
  ranks.  A collective that reduces in transit would add 16-bit values in an
  order and precision of its own choosing; this way the result is bit-identical
  to the one-process step and to the oracle.  Each rank sends and receives
  (N-1)/N of its gradient bytes, the same volume as a ring reduce-scatter.
- The scalar all-reduce: every rank's 16-byte statistics record goes to every
  rank, and each folds them in rank order, so every rank takes identical
  decisions.  On the device back end this stays on the GPU
  (zero_opt_grad_stats_async, an all-gather of the records,
  zero_opt_step_folded), so a step never waits for the host; the host back
  end uses ``allgather_fold``.
- The all-gather of the updated 16-bit shards is ``all_gather_into_tensor``
  on their bytes.

Both back ends run the same exchanges: ``"device"`` steps with the CUDA kernels
on tensors of the current CUDA device (NCCL process group), ``"host"`` with the
offloaded CPU step on CPU tensors (gloo process group).
"""
from __future__ import annotations

from . import (allgather_fold, make_buffers, zero_host_create, zero_host_destroy,
               zero_host_grad_stats, zero_host_last_step, zero_host_step, zero_opt_create,
               zero_opt_destroy, zero_opt_grad_stats_async, zero_opt_last_step,
               zero_opt_shard_bounds, zero_opt_step_folded)


def _bytes(t):
    """A contiguous tensor's storage as uint8 (the collectives move bits)."""
    import torch
    return t.contiguous().view(torch.uint8)


class Zero2Step:
    """One rank's view of a ZeRO-2 data-parallel optimizer step.

    `cfg` is the zero_opt_config of the whole flat buffer (numel = Ψ, world =
    N = the process group's size).  Per step the rank passes its own local
    gradients: K full padded buffers (P = N*S elements, one per micro-step), and
    its shard's master, m and v (S elements; master None with cfg.master16),
    and the full padded 16-bit parameter buffer, whose every shard is updated
    on return (this rank's by the step, the others by the all-gather).
    """

    def __init__(self, cfg, group=None, backend="device", threads=0):
        import torch.distributed as dist
        if backend not in ("device", "host"):
            raise ValueError("backend must be 'device' or 'host'")
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        if cfg.world != self.world:
            raise ValueError(f"cfg.world = {cfg.world} but the process group has {self.world} ranks")
        self.backend = backend
        self.cfg = cfg
        self.S = -(-cfg.numel // cfg.world)
        self.P = self.S * cfg.world
        self._stats = None   # device: every rank's statistics record (16 bytes each)
        self._recv = None    # all-to-all receive buffers, one per micro-step
        if backend == "device":
            self.h = zero_opt_create(cfg)
            b, e, S, P = zero_opt_shard_bounds(self.h, self.rank)
            assert (S, P) == (self.S, self.P)
        else:
            self.h = zero_host_create(cfg, threads)

    def close(self):
        if self.h is not None:
            (zero_opt_destroy if self.backend == "device" else zero_host_destroy)(self.h)
            self.h = None

    def exchange_gradients(self, grads):
        """All-to-all of the K local gradient buffers: returns, rank-major, the
        N*K shard-local buffers (S elements) of this rank's shard."""
        import torch
        import torch.distributed as dist
        S, N = self.S, self.world
        K = len(grads)
        # receive buffers are kept from step to step (no allocation per step)
        if (self._recv is None or len(self._recv) != K or self._recv[0].dtype != grads[0].dtype
                or self._recv[0].device != grads[0].device):
            self._recv = [torch.empty_like(g) for g in grads]
        for g, out in zip(grads, self._recv):
            if g.numel() != self.P:
                raise ValueError(f"gradient buffers must hold P = {self.P} elements")
            dist.all_to_all_single(_bytes(out), _bytes(g), group=self.group)
        return [self._recv[k][j * S:(j + 1) * S] for j in range(N) for k in range(K)]

    def gather_params(self, param16):
        """All-gather of the 16-bit shards into the full padded buffer."""
        import torch.distributed as dist
        if not param16.is_contiguous():
            raise ValueError("param16 must be contiguous (it is gathered in place)")
        S, r = self.S, self.rank
        out = _bytes(param16)
        if dist.get_backend(self.group) == "nccl":
            # in place: the rank's own shard already sits at its offset
            dist.all_gather_into_tensor(out, out[r * S * 2:(r + 1) * S * 2], group=self.group)
        else:
            mine = param16[r * S:(r + 1) * S].clone()
            dist.all_gather_into_tensor(out, _bytes(mine), group=self.group)

    def step(self, grads, master, m, v, param16, stream=None):
        """Exchange, statistics, fold, step, all-gather.  On the device back
        end every part is enqueued on the stream and nothing waits for the
        host; last_step() reads the decision."""
        K = len(grads)
        mine = self.exchange_gradients(grads)
        bufs = make_buffers(master, m, v, param16, mine, n_ranks=self.world, n_micro=K,
                            grads_shard_local=True)
        if self.backend == "device":
            import torch
            import torch.distributed as dist
            if self._stats is None:
                self._stats = torch.zeros(16 * self.world, dtype=torch.uint8,
                                          device=mine[0].device)
            own = self._stats[16 * self.rank:16 * (self.rank + 1)]
            zero_opt_grad_stats_async(self.h, self.rank, bufs, own, stream)
            if dist.get_backend(self.group) == "nccl":
                dist.all_gather_into_tensor(self._stats, own, group=self.group)
            else:
                dist.all_gather_into_tensor(self._stats, own.clone(), group=self.group)
            zero_opt_step_folded(self.h, self.rank, bufs, self._stats, self.world, stream)
        else:
            own = zero_host_grad_stats(self.h, self.rank, bufs)
            G = allgather_fold(own, self.group)
            zero_host_step(self.h, self.rank, bufs, global_stats=G)
        self.gather_params(param16)

    def last_step(self, stream=None):
        """zero_opt_step_info of the last step (identical on every rank);
        synchronizes the stream on the device back end."""
        if self.backend == "device":
            return zero_opt_last_step(self.h, stream)
        return zero_host_last_step(self.h)
