"""The N>1 host logic of bench.py on CPU with world_size-2 gloo ranks.

Each rank runs its own emulated ZeRO group (N independent replicas, no
cross-GPU data path); the only thing ranks share is the timing
reduction (max over ranks) and rank 0 alone printing the JSON line.
"""
import io
import os
import socket
import sys
from contextlib import redirect_stdout

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    got = bench.max_over_ranks(10.0 + rank * 3.5)
    # the end-to-end leg: when one rank sees too little host memory, every
    # rank skips it (rank 1 sees 10 GB available, rank 0 plenty)
    bench._mem_available_bytes = (lambda: 10 ** 12) if rank == 0 else (lambda: 10 * 10 ** 9)
    fits_small, _ = bench.e2e_fits_host(5 * 10 ** 9)       # 5 GB < 0.6 * 10 GB on both ranks
    fits_large, _ = bench.e2e_fits_host(8 * 10 ** 9)       # 8 GB > 6 GB on rank 1 only
    dist.barrier()
    dist.destroy_process_group()
    # reference arm under a multi-rank launch: rank 0 prints, the others exit 0 silently
    buf = io.StringIO()
    sys.argv = ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                "--workload", "flat:R=2,M=1,N=4096"]
    with redirect_stdout(buf):
        rc = bench.main()
    out[rank] = (got, rc, buf.getvalue(), fits_small, fits_large)


def test_two_gloo_ranks_max_and_single_printer():
    world = 2
    port = _free_port()
    manager = mp.get_context("spawn").Manager()      # no fork of a threaded process
    out = manager.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert out[0][0] == out[1][0] == 13.5
    assert out[0][1] == out[1][1] == 0
    assert out[0][2].strip().startswith("{") and '"impl": "reference"' in out[0][2]
    assert out[1][2] == ""
    assert out[0][3] and out[1][3]                     # both ranks pin
    assert not out[0][4] and not out[1][4]             # both ranks skip together
    import json
    line = json.loads(out[0][2])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
