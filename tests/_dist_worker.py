"""One rank of the two-process CPU check of the sharded layout (run by
test_sharding_multiproc.py with RANK / WORLD_SIZE / MASTER_* set)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def main():
    import numpy as np
    import torch.distributed as dist
    rank, world = int(os.environ['RANK']), int(os.environ['WORLD_SIZE'])
    dist.init_process_group('gloo', rank=rank, world_size=world)
    from rank_state_compression_head_b300 import sharding
    import synth
    w = synth.GDN_BATCHED
    mine = sharding.shard(w, rank, world)
    # this rank's first decode step inputs for two heads (host generator)
    d = synth.decode_inputs(mine, 0, heads=np.arange(2))
    t_ms = [3.0, 5.0, 4.0, 1.0][rank]                 # a made-up per-rank time
    sharding.barrier()
    t_max = sharding.max_over_ranks(t_ms)
    out = dict(rank=rank, seed=mine.seed, name=mine.name, n_heads=mine.n_heads, t_max=t_max,
               job_heads=sharding.job_heads(mine.n_heads, world), reports=sharding.reports(rank),
               k0=float(d['k'][0, 0]))
    print(json.dumps(out), flush=True)
    dist.destroy_process_group()


if __name__ == '__main__':
    main()
