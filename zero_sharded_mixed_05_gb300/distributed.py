"""The ZeRO-2 and ZeRO-3 data-parallel steps across processes: the exchanges
around the per-shard step.

Sources: "DeepSpeed framework interview answer" (algomooc.com), "ZeRO 三阶段",
and "LLM-train tutorials ch01" (jwzheng96.github.io) §1.2 stage table: the
gradients are reduce-scattered so that each rank holds the reduced gradient of
its own shard, each rank updates only its shard of the optimizer state, and
under ZeRO-2 the updated 16-bit parameters are all-gathered.  Under ZeRO-3 the
16-bit parameters are sharded too: each rank keeps only its shard, the step
updates it in place and gathers nothing, and the full parameters are
all-gathered again when a forward or backward pass needs them (the stage
table's "每次 forward / backward 再 all-gather").  Every rank also needs the
global overflow flag and gradient norm, a two-scalar all-reduce.

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
- The all-gather of the updated 16-bit shards (ZeRO-2, after every step;
  ZeRO-3, only when the caller asks for the full parameters with
  ``gather_params``) is ``all_gather_into_tensor`` on their bytes.

Device-memory traffic of the owner's step: the all-to-all lands N x K
shard-local buffers, and the statistics pass and the update pass each read
all of them, so a step reads 2 x 2NK bytes of gradients per parameter plus
the 26 bytes of optimizer state and 16-bit copy: 4NK + 26 (58 at N = 8,
K = 1), against 30 for one pre-reduced buffer.  That is the price of the
binary32 rank-order reduction.

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


class ZeroStep:
    """One rank's view of a ZeRO-2 or ZeRO-3 data-parallel optimizer step.

    `cfg` is the zero_opt_config of the whole flat buffer (numel = Ψ, world =
    N = the process group's size).  Per step the rank passes its own local
    gradients: K full padded buffers (P = N*S elements, one per micro-step), and
    its shard's master, m and v (S elements; master None with cfg.master16),
    and its 16-bit parameters: under ZeRO-2 (`stage` 2) the full padded buffer,
    whose every shard is updated on return (this rank's by the step, the others
    by the all-gather); under ZeRO-3 (`stage` 3) its own shard only (S
    elements), updated in place, with no gather (``gather_params`` builds the
    full buffer when a forward or backward pass needs it).
    """

    stage = 2

    def __init__(self, cfg, group=None, backend="device", threads=0, stage=None):
        import torch.distributed as dist
        if backend not in ("device", "host"):
            raise ValueError("backend must be 'device' or 'host'")
        if stage is not None:
            if stage not in (2, 3):
                raise ValueError("stage must be 2 or 3")
            self.stage = stage
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

    def gather_params(self, param16, out=None):
        """All-gather of the 16-bit shards.  ZeRO-2: `param16` is the full
        padded buffer, gathered in place.  ZeRO-3: `param16` is this rank's
        shard (S elements) and the full padded buffer is written to `out`
        (P elements, allocated when None) and returned."""
        import torch
        import torch.distributed as dist
        S, r = self.S, self.rank
        if not param16.is_contiguous():
            raise ValueError("param16 must be contiguous")
        if self.stage == 3:
            if param16.numel() != S:
                raise ValueError(f"a ZeRO-3 shard holds S = {S} elements")
            if out is None:
                out = torch.empty(self.P, dtype=param16.dtype, device=param16.device)
            if out.numel() != self.P or not out.is_contiguous():
                raise ValueError(f"out must be a contiguous buffer of P = {self.P} elements")
            dist.all_gather_into_tensor(_bytes(out), _bytes(param16), group=self.group)
            return out
        out = _bytes(param16)
        if dist.get_backend(self.group) == "nccl":
            # in place: the rank's own shard already sits at its offset
            dist.all_gather_into_tensor(out, out[r * S * 2:(r + 1) * S * 2], group=self.group)
        else:
            mine = param16[r * S:(r + 1) * S].clone()
            dist.all_gather_into_tensor(out, _bytes(mine), group=self.group)
        return param16

    def step(self, grads, master, m, v, param16, stream=None):
        """Exchange, statistics, fold, step and, under ZeRO-2, the all-gather.
        On the device back end every part is enqueued on the stream and
        nothing waits for the host; last_step() reads the decision."""
        K = len(grads)
        if self.stage == 3 and param16.numel() != self.S:
            raise ValueError(f"a ZeRO-3 step takes this rank's shard of S = {self.S} "
                             "16-bit parameters")
        if self.stage == 2 and param16.numel() != self.P:
            raise ValueError(f"a ZeRO-2 step takes the full padded buffer of P = {self.P} "
                             "16-bit parameters")
        mine = self.exchange_gradients(grads)
        bufs = make_buffers(master, m, v, param16, mine, n_ranks=self.world, n_micro=K,
                            grads_shard_local=True, param16_shard_local=self.stage == 3)
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
        if self.stage == 2:
            self.gather_params(param16)

    def last_step(self, stream=None):
        """zero_opt_step_info of the last step (identical on every rank);
        synchronizes the stream on the device back end."""
        if self.backend == "device":
            return zero_opt_last_step(self.h, stream)
        return zero_host_last_step(self.h)


class Zero2Step(ZeroStep):
    """ZeRO-2: optimizer state and gradients sharded, 16-bit parameters
    replicated (all-gathered after every step)."""

    stage = 2


class Zero3Step(ZeroStep):
    """ZeRO-3: optimizer state, gradients and 16-bit parameters sharded; the
    step updates the rank's parameter shard in place and gathers nothing."""

    stage = 3
