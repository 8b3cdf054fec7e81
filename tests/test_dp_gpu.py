"""The data-parallel step on the GPU: dp.fused_step -- the timed step of bench.py
for N > 1 -- through a one-rank NCCL process group, so its device-side count, its
NCCL all-reduce of that count, the fused kernel reading the total from device
memory, and the all-reduce of the partial loss all run on the device.  With one
rank the sums are the rank's own values, so the result must equal the plain
fused call bit for bit (the per-token mean of the LossAccelerationPlugin,
fms-hf-tuning PR #280, "Early Version Of This Plugin", reduced to one rank).
"""
import os
import socket

import numpy as np
import pytest
import torch

import workloads as wl
from ce_helpers import bits, to_device

pytestmark = pytest.mark.gpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_fused_step_one_rank_nccl(cuda_lib):
    import torch.distributed as dist

    from cross_entropy_loss_gb300 import dp

    if not dist.is_available() or not dist.is_nccl_available():
        pytest.skip("torch.distributed with NCCL is not available")
    ce = cuda_lib
    cfg = wl.mistral()
    x, y, V = cfg["logits"], cfg["labels"], cfg["V"]
    yd = torch.from_numpy(y).cuda()
    ref_t = to_device(x, wl.BF16)
    ref = ce.foak_ce_fwd_bwd(ref_t, yd)
    t = to_device(x, wl.BF16)
    cnt = torch.empty(1, dtype=torch.int64, device="cuda")
    ws = ce.workspace(x.shape[0], torch.device("cuda"))
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            device_id=torch.device("cuda", torch.cuda.current_device()))
    try:
        out = dp.fused_step(lambda yy: ce.foak_ce_count_valid(yy, V, out=cnt),
                            lambda xx, yy, d: ce.foak_ce_fwd_bwd_devdenom(xx, yy, d, workspace_tensor=ws), t, yd)
        torch.cuda.synchronize()
    finally:
        dist.destroy_process_group()
    assert int(out["denom"].item()) == int(ref["n_valid"].item()) == 4092
    assert out["loss"].item() == ref["loss"].item()
    assert out["err"].item() == 0
    np.testing.assert_array_equal(bits(t), bits(ref_t))
