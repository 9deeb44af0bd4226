"""One rank of the two-rank CPU check of bench.py's distributed context (run
under torch.distributed.run by test_bench_ranks.py): barrier, then the
max-over-ranks reduction that bench.py applies to each rank's timed
milliseconds.  Each rank writes its result as JSON to <out dir>/rank<r>.json
(the directory is the first argument)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import bench  # noqa: E402


def main():
    ctx = bench.DistCtx(torch)
    try:
        ctx.barrier()
        mine = 10.0 + 7.5 * ctx.rank  # rank 1 is the slow one
        res = {"rank": ctx.rank, "world": ctx.world, "mine": mine, "max": ctx.max(mine),
               "backend": ctx.dist.get_backend() if ctx.dist else None}
        with open(os.path.join(sys.argv[1], f"rank{ctx.rank}.json"), "w") as f:
            json.dump(res, f)
        ctx.barrier()
    finally:
        ctx.close()


if __name__ == "__main__":
    main()
