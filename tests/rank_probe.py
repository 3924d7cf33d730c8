"""A stand-in rank for the launcher test: started by bench.py's torchrun command on CPU, it joins
a gloo process group, reports a rank-dependent time and byte count through bench.py's reduction,
and rank 0 prints one JSON line as the benchmark would (n_gpus = the world size it joined)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    rank, world, local = bench.dist_env()
    dist.init_process_group("gloo")
    try:
        bench.barrier()
        t, b = bench.reduce_max_sum(10.0 + 5.0 * rank, 1000.0 * (rank + 1))
        if rank == 0:
            print(json.dumps({"n_gpus": world, "max_ms": t, "bytes": b,
                              "args": sys.argv[1:]}), flush=True)
        bench.barrier()
    finally:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
