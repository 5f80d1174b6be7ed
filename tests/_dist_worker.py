"""One rank of the two-rank CPU check of the bench's multi-process path (gloo): rank discovery from the
environment, the barrier, the max-over-ranks reduction of the step time and the per-rank shard seed. Prints
one JSON line."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    dist.init_process_group("gloo", init_method="env://")
    world, rank, local = bench._dist()
    bench._barrier(world)
    ms = bench._max_over_ranks(1.5 * (rank + 1), world, "cpu")
    case = bench.shard_case("tiny_decode_4k_b1_h16", rank)
    bench._barrier(world)
    print(json.dumps({"rank": rank, "world": world, "local": local, "max_ms": ms, "seed": case.seed}), flush=True)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
