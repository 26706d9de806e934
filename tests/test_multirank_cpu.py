"""The N > 1 path on CPU: two `gloo` ranks in separate processes.

The packed projection shards by tokens (data parallelism): each rank runs the
whole step on its own batch, with no exchange inside the step.  What the ranks
share is (a) the benchmark's job-level figures, the slowest rank's time and the
whole job's tokens, and (b) for a data-parallel optimizer, the dW that is the
sum of the ranks' dW over their token shards.  Both are checked here with real
processes and a real process group, on the CPU."""

import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
import synth


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # (a) rank r took 1.5 + r ms: the job takes the slowest
        ms = bench.max_over_ranks(1.5 + rank, world, torch.device("cpu"))
        tput = bench.job_tokens_per_s(1000, world, ms)
        # (b) dW over this rank's token shard, from the oracle; summed over ranks
        s = synth.Shape(T=64, D=128, H=1, d_qk=96, d_v=128, seq_len=64)
        inp = synth.forward_inputs(s, seed=11)
        g = synth.backward_inputs(s, seed=11)
        f32 = synth.to_numpy_f32
        pos = inp["pos"].numpy()
        W8, _, s_w = oracle.quantize_bank(f32(inp["Wq"]), f32(inp["Wk"]), f32(inp["Wv"]))
        fw = oracle.forward(f32(inp["x"]), W8, s_w, pos, s.H, s.d_qk, s.d_v)
        bw = oracle.backward(f32(g["dq"]), f32(g["dk"]), f32(g["dv"]), fw["q"], fw["k"], fw["rstd"], pos, W8, s_w,
                             fw["x8"], fw["x_scale"], s.H, s.d_qk, s.d_v)
        lo, hi = rank * s.T // world, (rank + 1) * s.T // world
        _, dW_shard = oracle.grad_gemms(bw["dY8"][lo:hi], bw["dy_scale"], W8, s_w, fw["x8"][lo:hi], fw["x_scale"])
        t = torch.from_numpy(np.ascontiguousarray(dW_shard, dtype=np.float64))
        dist.all_reduce(t)
        if rank == 0:
            np.save(os.path.join(out_dir, "dW_sum.npy"), t.numpy())
            np.save(os.path.join(out_dir, "dW_full.npy"), np.asarray(bw["dW"], dtype=np.float64))
            with open(os.path.join(out_dir, "job.txt"), "w") as f:
                f.write(f"{ms} {tput}\n")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    ms, tput = map(float, open(tmp_path / "job.txt").read().split())
    assert ms == 2.5                                    # the slowest rank's time
    assert abs(tput - 2 * 1000 / 2.5e-3) < 1e-6         # both ranks' tokens over it
    dW_sum, dW_full = np.load(tmp_path / "dW_sum.npy"), np.load(tmp_path / "dW_full.npy")
    np.testing.assert_allclose(dW_sum, dW_full, rtol=1e-12, atol=1e-12 * np.abs(dW_full).max())
