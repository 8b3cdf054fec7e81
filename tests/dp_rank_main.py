"""One rank of the world-size-2 gloo run in tests/test_dp_gloo.py (started by the
same launcher bench.py uses for --gpus N).  Each rank takes its row shard of a small
batch and runs the data-parallel step of the per-token mean (count, all-reduced
denominator, fused forward+backward, summed partial losses) with the CPU oracle in
place of the kernels, then writes what it got for the test to check."""
import importlib.util
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import oracle  # noqa: E402
import workloads as wl  # noqa: E402


def _dp():
    spec = importlib.util.spec_from_file_location("_foak_dp", os.path.join(ROOT, "cross_entropy_loss_gb300", "dp.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def case():
    N, V = 37, 211
    x = wl.normal_matrix(N, V, seed=77, sigma=2.0, dtype=wl.F32)
    y = wl.uniform_labels(N, V, seed=77)
    y[[0, 5, 6, 30]] = -100
    return x, y, V


def main(out_dir):
    dp = _dp()
    rank, world, _ = dp.rank_env()
    dist.init_process_group("gloo")
    x, y, V = case()
    b, e = dp.shard_rows(x.shape[0], rank, world)
    grads = {}

    def count_fn(labels):
        return torch.tensor([oracle.count(labels.numpy(), V)[0]], dtype=torch.int64)

    def fused_fn(logits, labels, denom_count):
        r = oracle.ce(logits, labels.numpy(), V, denom=float(denom_count.item()))
        grads["g"] = r["grad"]
        return {"loss": torch.tensor([r["loss"]], dtype=torch.float64)}

    out = dp.fused_step(count_fn, fused_fn, x[b:e], torch.from_numpy(y[b:e].copy()))
    np.save(os.path.join(out_dir, f"grad{rank}.npy"), grads["g"])
    with open(os.path.join(out_dir, f"res{rank}.txt"), "w") as f:
        f.write(f"{b} {e} {int(out['denom'].item())} {float(out['loss'].item())!r} {world}\n")
    dist.destroy_process_group()


if __name__ == "__main__":
    main(sys.argv[1])
