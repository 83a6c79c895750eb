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


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_per_gemm_table_rates_and_fractions():
    bench = _bench()
    pk = {"bf16_tflops_sustained": 1000.0}
    M, N, K = 1024, 2048, 4096
    per_g = {("fp8_current", "autocast", "qkv", "fprop", M, N, K): [1.0, 3.0],     # mean 2 ms
             ("nvfp4", "prequant", "mlp_up", "wgrad", M, N, K): [0.5]}
    t = bench.per_gemm_table(per_g, pk)
    assert t["fields"] == bench.PER_GEMM_FIELDS
    rows = {(r[0], r[3]): r for r in t["rows"]}
    fl = 2.0 * M * N * K
    r = rows[("fp8_current", "fprop")]
    assert r[7] == 2.0 and r[8] == round(fl / 2e-3 / 1e12, 1)
    assert r[9] == round(fl / 2e-3 / 1e12 / 2000.0, 4)          # FP8: 2 x the bf16 peak
    r = rows[("nvfp4", "wgrad")]
    assert r[9] == round(fl / 0.5e-3 / 1e12 / 6000.0, 4)        # NVFP4: 6 x the bf16 peak


def test_nvfp4_over_bf16_ratios():
    bench = _bench()
    per = {"bf16/autocast": {"ms_per_layer": 12.0, "gemm_ms_per_layer": 11.0},
           "nvfp4/autocast": {"ms_per_layer": 6.0, "gemm_ms_per_layer": 4.0},
           "nvfp4/prequant": {"ms_per_layer": 4.0, "gemm_ms_per_layer": 3.5}}
    r = bench.nvfp4_over_bf16(per)
    assert r["autocast"] == 2.0 and r["prequant_kernel_only"] == round(11.0 / 3.5, 3)
    assert bench.nvfp4_over_bf16({"bf16/autocast": per["bf16/autocast"]}) is None


def test_fp8_gemm_traffic_follows_the_kernel_source(tmp_path, monkeypatch):
    """The committed DRAM figures are reported only for the GEMM source they were measured on."""
    bench = _bench()
    prof = os.path.join(ROOT, "profiles", "gemm_fp8_dram_traffic_codonfm_layer.json")
    d = json.load(open(prof))
    assert d["traffic_bytes_per_launch"] > d["algorithmic_bytes_per_launch"] > 0
    assert len(d["per_shape"]) == 12
    mean = sum(p["dram_read"] + p["dram_write"] for p in d["per_shape"]) // 12
    assert abs(mean - d["traffic_bytes_per_launch"]) <= 1
    # a copy of the tree: unchanged sources give the figure, an edited kernel gives none
    import hashlib
    csrc = tmp_path / "nvfp4_precision_transformer_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    h = hashlib.sha256()
    for name in ("gemm.cu", "common.cuh"):
        src = open(os.path.join(ROOT, "nvfp4_precision_transformer_gb300", "csrc", name), "rb").read()
        (csrc / name).write_bytes(src)
        h.update(src)
    # the figures keyed to the copied sources (the committed ones may predate the latest edit)
    d["kernel_source_sha256_prefix"] = h.hexdigest()[:16]
    (tmp_path / "profiles" / "gemm_fp8_dram_traffic_codonfm_layer.json").write_text(json.dumps(d))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    traffic, alg, note = bench.fp8_gemm_traffic()
    assert (traffic, alg) == (d["traffic_bytes_per_launch"], d["algorithmic_bytes_per_launch"]), note
    (csrc / "gemm.cu").write_bytes((csrc / "gemm.cu").read_bytes() + b"\n// edited\n")
    traffic, alg, note = bench.fp8_gemm_traffic()
    assert traffic is None and alg == d["algorithmic_bytes_per_launch"] and "changed" in note


def test_roofline_by_kind_uses_prequant_runs_and_dtype_peaks():
    bench = _bench()
    pk = {"bf16_tflops_sustained": 1000.0}
    agg = {("bf16", "autocast"): {"gemm_ms": 2.0, "gemm_flops": 2.0e12},
           ("nvfp4", "prequant"): {"gemm_ms": 1.0, "gemm_flops": 3.0e12},
           ("nvfp4", "autocast"): {"gemm_ms": 9.0, "gemm_flops": 3.0e12},
           ("fp8_current", "prequant"): {"gemm_ms": 1.0, "gemm_flops": 1.5e12}}
    r = bench.roofline_by_kind(agg, pk)
    assert set(r) == {"bf16", "nvfp4", "fp8_current"}
    assert r["bf16"]["achieved"] == 1000.0 and r["bf16"]["frac"] == 1.0
    assert r["nvfp4"]["achieved"] == 3000.0 and r["nvfp4"]["peak"] == 6000.0 and r["nvfp4"]["frac"] == 0.5
    assert r["fp8_current"]["peak"] == 2000.0 and r["fp8_current"]["frac"] == 0.75


def test_e2e_runs_as_many_steps_as_the_timed_region():
    sys.path.insert(0, ROOT)
    import bench
    old = sys.argv
    try:
        for argv, want in ((["bench.py"], None), (["bench.py", "--steps", "20"], 20), (["bench.py", "--steps", "2"], 5),
                           (["bench.py", "--steps", "20", "--e2e-steps", "3"], 3)):
            sys.argv = argv
            args = bench.parse()
            got = bench.e2e_steps(args)
            assert got == (want if want is not None else max(5, args.steps))
    finally:
        sys.argv = old
