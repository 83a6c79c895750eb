"""Host logic of bench.py without a GPU: replica aggregation over gloo ranks,
the workload configuration and the shape derivation."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, ws, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo")
    bench.barrier(ws)
    v = bench.reduce_max(10.0 + rank * 5.0, ws)
    out.put((rank, v))
    dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 15.0, 1: 15.0}


def test_reduce_max_single_process():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5


def test_shapes_match_oracle_derivation():
    from nvfp4_precision_transformer_gb300.shapes import LayerConfig, layer_gemms, layer_flops
    from oracle.gemm import linear_shapes
    cfg = LayerConfig()
    assert cfg.tokens == 15872
    ours = [(g.linear, g.pass_, g.M, g.N, g.K) for g in layer_gemms(cfg)]
    assert ours == list(linear_shapes(4096, 16384, 15872))
    assert abs(layer_flops(cfg) / 1e12 - 19.17) < 0.01


def test_reference_arm_prints_contract_line():
    env = dict(os.environ, WORLD_SIZE="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0", "--tokens", "512", "--hidden", "512", "--ffn", "1024"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "ms/layer" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
