"""Worker functions for the multi-process (gloo, CPU) tests of the benchmark's
multi-rank host logic.  They live in an importable module so that
torch.multiprocessing's spawn start method can run them in child processes."""
import os


def max_over_ranks_worker(rank: int, world: int, port: int, out_dir: str) -> None:
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        # every rank times a different amount of work; the job is as slow as
        # its slowest rank
        t = bench.max_over_ranks(1.5 + rank, "cpu")
        bench.barrier()
        rate = bench.whole_job_rate(1000.0, world, 10, t)
        with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
            f.write(f"{t} {rate}\n")
    finally:
        dist.destroy_process_group()
