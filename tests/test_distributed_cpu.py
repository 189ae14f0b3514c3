"""The ZeRO-2 and ZeRO-3 steps across two processes (gloo, CPU, the host back
end): all-to-all of the raw 16-bit gradient slices, local binary32 reduction in
rank order, the two-scalar fold, the shard step and, under ZeRO-2, the
all-gather of the 16-bit parameters (under ZeRO-3 each rank keeps only its
parameter shard; the full buffer is gathered on request).  Every rank's shard
state and parameters must be bit-identical to the oracle's one-process step
over the same gradients (each rank's K micro-step buffers, rank-major),
including a step whose overflow sits on the other rank's gradient.  No GPU is
touched."""
import os
import socket

import numpy as np
import pytest

from conftest import spawn_bounded

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NUMEL = 100_003          # odd: the last shard has padding
WORLD = 2
K = 2
STEPS = 5
SEED = 0x5EED0201


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _local_grads(rank, step, scale, P, code):
    """Rank `rank`'s K full padded gradient buffers of one step (uint16)."""
    import synth
    out = []
    for k in range(K):
        g = np.zeros(P, np.uint16)
        g[:NUMEL] = synth.normal_np(SEED, 1 + rank * K + k, step * NUMEL, NUMEL, 2e-3 * scale,
                                    synth.F16 if code == 0 else synth.BF16)
        if step == 3 and rank == 1 and k == 0:
            g[54_321] = 0x7C00 if code == 0 else 0x7F80     # overflow on the other shard
        out.append(g)
    return out


def _cfg_kwargs(master16):
    return dict(numel=NUMEL, world=WORLD, lr=1e-3, weight_decay=0.01, max_grad_norm=0.3,
                dynamic_scale=True, init_scale=64.0, scale_window=1000, master16=master16)


def _worker(rank, port, out_dir, code, master16, stage=2):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle as O
    import synth
    import zero_sharded_mixed_05_gb300 as z
    from zero_sharded_mixed_05_gb300.distributed import Zero2Step, Zero3Step
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    cfg = z.make_config(grad_dtype=code, **_cfg_kwargs(master16))
    zs = (Zero2Step if stage == 2 else Zero3Step)(cfg, backend="host", threads=2)
    b, e, S, P = O.shard_bounds(NUMEL, WORLD, rank)
    p0 = synth.normal_np(SEED, 0, 0, NUMEL, 0.02, synth.F32)
    tdt = torch.float16 if code == 0 else torch.bfloat16
    master = torch.zeros(S)
    master[:e - b] = torch.from_numpy(p0[b:e])
    m, v = torch.zeros(S), torch.zeros(S)
    q0 = O.f32_to_16(p0, code)
    p16 = torch.zeros(P, dtype=torch.int16)
    p16[:NUMEL] = torch.from_numpy(q0.view(np.int16)) if master16 else 0
    p16 = p16.view(tdt)
    if stage == 3:
        p16 = p16[b:b + S].clone()          # ZeRO-3: this rank's shard only
    scale = 64.0
    infos = []
    for step in range(1, STEPS + 1):
        grads = [torch.from_numpy(g.view(np.int16)).view(tdt)
                 for g in _local_grads(rank, step, scale, P, code)]
        zs.step(grads, None if master16 else master, m, v, p16)
        info = zs.last_step()
        infos.append((info.skipped, info.scale_used, info.t, info.coef))
        scale = z.zero_host_loss_scale(zs.h, rank).scale
    shard16 = p16.view(torch.int16).numpy().view(np.uint16).copy()
    if stage == 3:
        p16 = zs.gather_params(p16)          # the full buffer, for a forward pass
    np.savez(os.path.join(out_dir, f"r{rank}.npz"), master=master.numpy(), m=m.numpy(),
             v=v.numpy(), p16=p16.view(torch.int16).numpy().view(np.uint16),
             shard16=shard16, infos=np.array(infos, dtype=np.float64))
    zs.close()
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("code,master16,stage",
                         [(0, False, 2), (1, True, 2), (0, False, 3), (1, True, 3)],
                         ids=["fp16", "bf16-master16", "zero3-fp16", "zero3-bf16-master16"])
def test_two_rank_zero_step_matches_the_oracle(tmp_path, code, master16, stage):
    from zero_sharded_mixed_05_gb300 import _build
    _build.build()
    import oracle as O
    import synth
    spawn_bounded(_worker, (_free_port(), str(tmp_path), code, master16, stage), WORLD)
    res = [np.load(os.path.join(tmp_path, f"r{r}.npz")) for r in range(WORLD)]
    # the oracle: the one-process step of every shard with R = WORLD ranks' K buffers each
    orc = O.default()
    hp = O.hparams(lr=1e-3, weight_decay=0.01, max_grad_norm=0.3, dynamic_scale=True,
                   scale_window=1000)
    p0 = synth.normal_np(SEED, 0, 0, NUMEL, 0.02, synth.F32)
    q0 = orc.f32_to_16(p0, code)
    bounds = [orc.shard_bounds(NUMEL, WORLD, r) for r in range(WORLD)]
    P = bounds[0][3]
    st, sc = [], []
    for r, (b, e, _, _) in enumerate(bounds):
        st.append([None if master16 else p0[b:e].copy(), np.zeros(e - b, np.float32),
                   np.zeros(e - b, np.float32),
                   q0[b:e].copy() if master16 else np.zeros(e - b, np.uint16)])
        sc.append(O.scaler(64.0))
    decisions = []
    for step in range(1, STEPS + 1):
        allg = [_local_grads(j, step, sc[0].scale, P, code) for j in range(WORLD)]
        flat = [allg[j][k] for j in range(WORLD) for k in range(K)]      # rank-major
        per = [orc.stats_of(orc.reduce([g[b:e].copy() for g in flat], code))
               for (b, e, _, _) in bounds]
        G = orc.fold_stats(per)
        for r, (b, e, _, _) in enumerate(bounds):
            _, d = orc.step(hp, sc[r], [g[b:e].copy() for g in flat], code, *st[r], code,
                            float(WORLD * K), G)
        decisions.append((d.skip, d.scale_used, sc[0].t, d.coef))
    assert [d[0] for d in decisions] == [0, 0, 1, 0, 0]
    for r, (b, e, _, _) in enumerate(bounds):
        got = res[r]
        assert [tuple(x) for x in got["infos"]] == [tuple(np.float64(y) for y in d)
                                                   for d in decisions]
        if not master16:
            assert (got["master"][:e - b].view(np.uint32) == st[r][0].view(np.uint32)).all()
        assert (got["m"][:e - b].view(np.uint32) == st[r][1].view(np.uint32)).all()
        assert (got["v"][:e - b].view(np.uint32) == st[r][2].view(np.uint32)).all()
        # the rank's own 16-bit shard (the ZeRO-3 step's whole output), and
        # the gathered buffer (ZeRO-2 after every step; ZeRO-3 on request)
        assert (got["shard16"][b - (b if stage == 3 else 0):][:e - b] == st[r][3]).all()
        for j, (bj, ej, _, _) in enumerate(bounds):
            assert (got["p16"][bj:ej] == st[j][3]).all(), (r, j)
        assert not got["p16"][NUMEL:].any()
