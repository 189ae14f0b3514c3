"""The ZeRO-2 and ZeRO-3 steps' device back end (CUDA kernels, NCCL process
group) in one process on one GPU.  With one rank the exchanges are copies, so
this checks the device path's plumbing: byte-view collectives on device
tensors, stream order between the collectives and the kernels, the fold, the
in-place gather (ZeRO-2) and the shard-local 16-bit parameters (ZeRO-3).  The state must match the oracle's one-process step bit for
bit (no clipping, so the coefficient does not depend on the norm's last
bits).  The exchange logic across ranks is covered on the CPU by
test_distributed_cpu.py."""
import os
import socket

import numpy as np
import pytest

from conftest import spawn_bounded

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NUMEL = 50_001
K = 2
STEPS = 3
SEED = 0x5EED0301


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _grads(step, scale):
    import synth
    out = []
    for k in range(K):
        g = synth.normal_np(SEED, 1 + k, step * NUMEL, NUMEL, 1e-3 * scale, synth.F16)
        if step == 2 and k == 1:
            g[31_337] = 0x7C00
        out.append(g)
    return out


def _worker(rank, port, out_path, stage=2):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import synth
    import zero_sharded_mixed_05_gb300 as z
    from zero_sharded_mixed_05_gb300.distributed import ZeroStep
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    torch.cuda.set_device(0)
    dist.init_process_group("nccl", rank=0, world_size=1, device_id=torch.device("cuda", 0))
    cfg = z.make_config(numel=NUMEL, world=1, grad_dtype=z.FP16, lr=1e-3, weight_decay=0.01,
                        dynamic_scale=True, init_scale=128.0)
    zs = ZeroStep(cfg, backend="device", stage=stage)
    dev = torch.device("cuda", 0)
    master = torch.from_numpy(synth.normal_np(SEED, 0, 0, NUMEL, 0.02, synth.F32)).to(dev)
    m, v = torch.zeros(NUMEL, device=dev), torch.zeros(NUMEL, device=dev)
    p16 = torch.zeros(NUMEL, dtype=torch.float16, device=dev)
    scale, infos = 128.0, []
    for step in range(1, STEPS + 1):
        grads = [torch.from_numpy(g.view(np.int16)).view(torch.float16).to(dev)
                 for g in _grads(step, scale)]
        zs.step(grads, master, m, v, p16)
        info = zs.last_step()
        infos.append((info.skipped, info.scale_used, info.t))
        scale = z.zero_opt_loss_scale(zs.h, 0).scale
    torch.cuda.synchronize()
    np.savez(out_path, master=master.cpu().numpy(), m=m.cpu().numpy(), v=v.cpu().numpy(),
             p16=p16.cpu().view(torch.int16).numpy().view(np.uint16), infos=np.array(infos))
    zs.close()
    dist.destroy_process_group()


@pytest.mark.parametrize("stage", [2, 3])
def test_one_rank_device_zero_step(tmp_path, stage):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    import oracle as O
    import synth
    out = os.path.join(tmp_path, "r0.npz")
    spawn_bounded(_worker, (_free_port(), out, stage), 1)
    got = np.load(out)
    orc = O.default()
    hp = O.hparams(lr=1e-3, weight_decay=0.01, dynamic_scale=True, scale_window=1000)
    sc = O.scaler(128.0)
    master = synth.normal_np(SEED, 0, 0, NUMEL, 0.02, synth.F32)
    m, v = np.zeros(NUMEL, np.float32), np.zeros(NUMEL, np.float32)
    p16 = np.zeros(NUMEL, np.uint16)
    infos = []
    for step in range(1, STEPS + 1):
        _, d = orc.step(hp, sc, _grads(step, sc.scale), O.FP16, master, m, v, p16, O.FP16,
                        float(K))
        infos.append((d.skip, d.scale_used, sc.t))
    assert [tuple(x) for x in got["infos"]] == [tuple(float(y) for y in i) for i in infos]
    assert [i[0] for i in infos] == [0, 1, 0]
    for name, ref in (("master", master), ("m", m), ("v", v)):
        assert (got[name].view(np.uint32) == ref.view(np.uint32)).all(), name
    assert (got["p16"] == p16).all()
