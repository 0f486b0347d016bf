"""Host-side bookkeeping of bench.py on CPU: the slowest-rank time and the
whole-job throughput across two Gloo ranks, and the rule that a measured DRAM
traffic figure is reported only while the kernel source it was taken on is
unchanged."""

import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [2.5, 4.0][rank]
    got = bench.max_over_ranks(ms, world)
    out_q.put((rank, got, bench.job_throughput(2048, world, got)))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out_q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out_q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, value in res:
        assert ms == 4.0, f"rank {rank} saw {ms}"
        assert abs(value - 2 * 2048 / 4.0e-3) < 1e-6


def test_single_process_is_its_own_max():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_throughput(64, 1, 0.5) == 128000.0


def test_ncu_traffic_only_while_the_kernel_source_is_unchanged(monkeypatch):
    import bench
    key = ("qwen3_0.6b_layer_prefill2048", 2, "gemm_lm_head")
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, (1.0e6, "k_gemm.cu", bench.source_hash("k_gemm.cu")))
    assert bench.ncu_traffic(*key) == 1.0e6
    monkeypatch.setitem(bench.NCU_TRAFFIC, key, (1.0e6, "k_gemm.cu", "0" * 16))
    assert bench.ncu_traffic(*key) is None
    assert bench.ncu_traffic("no such workload", 2, "gemm_lm_head") is None


def test_source_hash_counts_code_not_comments(tmp_path, monkeypatch):
    """The hash that ties a traffic capture to a kernel ignores line comments and
    blank lines and follows any change to the code itself."""
    import shutil
    import bench
    src = os.path.join(bench.ROOT, "tensor_transformer_forward_gb300", "csrc")
    dst = tmp_path / "tensor_transformer_forward_gb300" / "csrc"
    shutil.copytree(src, dst)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.source_hash("k_gemm.cu")
    p = dst / "k_gemm.cu"
    text = p.read_text()
    p.write_text(text.replace("\n", "\n// a comment line\n\n", 1))
    assert bench.source_hash("k_gemm.cu") == h0
    p.write_text(text.replace("namespace tpk {", "namespace tpk {\nconstexpr int kAnotherConstant = 1;", 1))
    assert bench.source_hash("k_gemm.cu") != h0


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one JSON
    line with the keys the driver reads, on the tiny workload, without a GPU."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "tiny_prefill8",
                          "--steps", "1", "--warmup", "3"], cwd=root, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == "tiny_prefill8"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_algorithmic_work_matches_the_closed_forms():
    """The per-launch work bench.py divides by the measured time: GEMM and attention
    flops of the 0.6B prefill layer and the KV bytes of the 0.6B decode layer, as
    computed by hand from the shapes (2 T H N per projection, causal 4 hd nq T(T+1)/2,
    K and V rows of every cached key)."""
    import bench
    import synth
    pre = synth.WORKLOADS["qwen3_0.6b_layer_prefill2048"]
    T, H = 2048, 1024
    gemm = sum(bench.kernel_work(k, pre, 2)[0] for k in ("gemm_qkv", "gemm_o", "gemm_gate_up", "gemm_down"))
    assert gemm == 2 * T * H * (4096 + 2048 + 6144) + 2 * T * 3072 * H      # 64.42 GFLOP
    assert bench.kernel_work("attn_prefill", pre, 2)[0] == 4 * 128 * 16 * T * (T + 1) / 2
    dec = synth.WORKLOADS["qwen3_0.6b_layer_decode64x4096"]
    for n in (1, 2, 4):
        assert bench.kernel_work("attn_decode", dec, n)[1] == 64 * 4097 * 8 * 128 * 2 * 2  # 1074.0 MB
    # 32B at tp 16: kv heads replicated on two ranks, so 16 cached heads per key
    d32 = synth.WORKLOADS["qwen3_32b_layer_tp16_decode32x2048"]
    assert bench.kernel_work("attn_decode", d32, 16)[1] == 32 * 2049 * 16 * 128 * 2 * 2
    assert bench.kernel_work("gemm_lm_head", d32, 16)[1] == 151936 * 5120 * 2 + 32 * 5120 * 2
    pk = {"bf16_tflops_sustained": 1772.4, "hbm_gbs": 6682.2}
    r = bench.kernel_roofline("attn_decode", dec, 2, 1.0, pk)     # 1.074 GB in 1 ms
    assert r["bound"] == "hbm" and abs(r["achieved"] - 1074.0) < 0.1
    r = bench.kernel_roofline("gemm_gate_up", pre, 2, 1.0, pk)    # 25.77 GFLOP in 1 ms
    assert r["bound"] == "tensor" and abs(r["achieved"] - 25.77) < 0.01
    # a decode GEMM streams its weights: HBM-bound
    assert bench.kernel_roofline("gemm_gate_up", dec, 2, 1.0, pk)["bound"] == "hbm"
