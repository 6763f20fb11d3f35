"""One rank of the replica plumbing test (tests/test_bench_host.py), started
by bench.spawn_ranks through torch.distributed.run: joins a gloo group,
reports made-up per-rank work through bench.replica_glups and, on rank 0,
prints the whole-job figure as one JSON line. No GPU."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def main():
    import torch.distributed as dist
    world, rank, _ = bench.dist_env()
    dist.init_process_group("gloo")
    # rank k: (k + 1) * 1e9 lattice updates in 0.5 + k seconds
    value = bench.replica_glups(1e9 * (rank + 1), 0.5 + rank)
    if rank == 0:
        print(json.dumps({"n_gpus": world, "value": value}), flush=True)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
