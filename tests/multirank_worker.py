"""One rank of the two-rank CPU check of bench.py's multi-rank path (gloo).

Run by tests/test_multirank.py as `python multirank_worker.py RANK WORLD PORT`;
prints one JSON line with what this rank saw.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def main():
    rank, world, port = (int(x) for x in sys.argv[1:4])
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from latent_query_split_gb300 import workloads
    w = workloads.CONFIGS["c1_fp32_small"]
    wr = bench.replica_workload(w, rank)
    inp = workloads.make_inputs(wr, device="cpu")
    slowest = bench.max_over_ranks(1.5 + rank, world)        # this rank's "time"
    dist.barrier()
    print(json.dumps({"rank": rank, "slowest": slowest, "seed": wr.seed,
                      "k_sum": float(inp["K"].double().sum()),
                      "offsets": inp["offsets"]}), flush=True)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
