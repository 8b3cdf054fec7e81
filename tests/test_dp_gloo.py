"""World-size-2 gloo run of the data-parallel host path (CPU, no GPU).

Each rank takes its row shard, counts its valid tokens, all-reduces the global
denominator, computes its shard (the oracle stands in for the kernels here), and
the ranks' partial losses and gradient rows must reproduce the whole batch --
the per-token mean across GPUs of the LossAccelerationPlugin
(fms-hf-tuning PR #280, "Early Version Of This Plugin").
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _dp():
    import importlib.util

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("_foak_dp", os.path.join(root, "cross_entropy_loss_gb300", "dp.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case():
    import workloads as wl

    N, V = 37, 211
    x = wl.normal_matrix(N, V, seed=77, sigma=2.0, dtype=wl.F32)
    y = wl.uniform_labels(N, V, seed=77)
    y[[0, 5, 6, 30]] = -100
    return x, y, V


def _rank_main(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import oracle

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dp = _dp()
    x, y, V = _case()
    b, e = dp.shard_rows(x.shape[0], rank, world)
    n_local, _ = oracle.count(y[b:e], V)
    denom = dp.global_denominator(n_local)
    r = oracle.ce(x[b:e], y[b:e], V, denom=denom)
    total = dp.global_loss(r["loss"])
    slowest = dp.max_over_ranks(float(rank + 1))
    np.save(os.path.join(out_dir, f"grad{rank}.npy"), r["grad"])
    with open(os.path.join(out_dir, f"res{rank}.txt"), "w") as f:
        f.write(f"{b} {e} {denom} {total!r} {slowest}\n")
    dist.destroy_process_group()


def test_shard_rows_partition():
    dp = _dp()
    for n in (0, 1, 7, 37, 4096):
        for w in (1, 2, 3, 8):
            spans = [dp.shard_rows(n, r, w) for r in range(w)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            assert all(spans[i][1] == spans[i + 1][0] for i in range(w - 1))
            sizes = [e - b for b, e in spans]
            assert max(sizes) - min(sizes) <= 1


def test_launcher_command_line():
    dp = _dp()
    argv = dp.launch_argv(4, "/x/bench.py", ["--gpus", "4", "--steps", "3"], 29512, python="py")
    assert argv == ["py", "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=4", "--master-addr",
                    "127.0.0.1", "--master-port=29512", "/x/bench.py", "--gpus", "4", "--steps", "3"]
    with pytest.raises(ValueError):
        dp.launch_argv(0, "b.py", [], 1)


def test_rank_env(monkeypatch):
    dp = _dp()
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert dp.rank_env() == (0, 1, 0)
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("LOCAL_RANK", "3")
    assert dp.rank_env() == (3, 4, 3)
    monkeypatch.setenv("RANK", "4")
    with pytest.raises(ValueError):
        dp.rank_env()


def test_launched_ranks_run_the_data_parallel_step(tmp_path):
    """Two gloo ranks started by the bench's launcher run dp.fused_step -- the bench's
    timed step for N > 1 -- on their row shards: the all-reduced denominator is the
    batch's n_valid, the summed partial losses are the batch's mean loss on both ranks,
    and the shards' gradients are the whole batch's."""
    import subprocess
    import sys

    import oracle

    dp = _dp()
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = os.path.join(root, "tests", "dp_rank_main.py")
    env = dict(os.environ)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT"):
        env.pop(k, None)
    r = subprocess.run(dp.launch_argv(2, script, [str(tmp_path)], _free_port()), env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    sys.path.insert(0, os.path.join(root, "tests"))
    import dp_rank_main

    x, y, V = dp_rank_main.case()
    whole = oracle.ce(x, y, V)
    grads = []
    for rank in range(2):
        b, e, denom, loss, world = open(tmp_path / f"res{rank}.txt").read().split()
        assert int(world) == 2 and int(denom) == whole["n_valid"]
        assert float(loss) == pytest.approx(whole["loss"], rel=1e-13)
        assert (int(b), int(e)) == dp.shard_rows(x.shape[0], rank, 2)
        grads.append(np.load(tmp_path / f"grad{rank}.npy"))
    np.testing.assert_allclose(np.concatenate(grads), whole["grad"], rtol=1e-13, atol=1e-18)


def test_two_ranks_reproduce_whole_batch(tmp_path):
    import oracle

    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    x, y, V = _case()
    whole = oracle.ce(x, y, V)
    grads, totals = [], set()
    for r in range(world):
        b, e, denom, total, slowest = open(tmp_path / f"res{r}.txt").read().split()
        assert float(denom) == whole["n_valid"]
        assert float(slowest) == world
        totals.add(float(total))
        grads.append(np.load(tmp_path / f"grad{r}.npy"))
    assert len(totals) == 1
    assert totals.pop() == pytest.approx(whole["loss"], rel=1e-13)
    np.testing.assert_allclose(np.concatenate(grads), whole["grad"], rtol=1e-13, atol=1e-18)
