"""The data-parallel layout with two ranks on CPU (gloo): every rank gets an
independent batch of requests of the workload's shapes, the job's time is the
slowest rank's, the job's heads are all ranks' heads, and only rank 0 reports."""
import json
import os
import socket
import subprocess
import sys

import pytest

import synth
from rank_state_compression_head_b300 import sharding

HERE = os.path.dirname(os.path.abspath(__file__))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(('127.0.0.1', 0))
        return s.getsockname()[1]


def _run_ranks(world: int):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                   MASTER_ADDR='127.0.0.1', MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES='')
        procs.append(subprocess.Popen([sys.executable, os.path.join(HERE, '_dist_worker.py')], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        try:
            o, e = p.communicate(timeout=180)
        except subprocess.TimeoutExpired:
            p.kill()
            raise
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    return sorted(outs, key=lambda r: r['rank'])


@pytest.mark.parametrize('world', [2])
def test_two_ranks_gloo(world):
    res = _run_ranks(world)
    w = synth.GDN_BATCHED
    assert [r['rank'] for r in res] == list(range(world))
    assert res[0]['seed'] == w.seed                          # one GPU runs exactly the named workload
    assert len({r['seed'] for r in res}) == world            # independent batches
    assert len({r['k0'] for r in res}) == world              # ... with different inputs
    assert all(r['name'] == w.name and r['n_heads'] == w.n_heads for r in res)
    assert all(r['t_max'] == 5.0 for r in res)               # max over ranks, seen by every rank
    assert all(r['job_heads'] == world * w.n_heads for r in res)
    assert [r['reports'] for r in res] == [True] + [False] * (world - 1)


def test_shard_single_rank_is_identity():
    w = synth.MAMBA2_BATCHED
    assert sharding.shard(w, 0, 1) is w
    assert sharding.max_over_ranks(2.5) == 2.5
    with pytest.raises(ValueError):
        sharding.shard(w, 2, 2)
