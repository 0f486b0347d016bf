#!/usr/bin/env python
"""Throughput of one tensor-parallel forward step on GB300.

A step is one pass of the whole hot path over one batch: vocab-parallel
embedding of the step's token ids, the decoder layer(s) (every rank shard of
the tensor-parallel layer, rank-sums in the row-parallel GEMM epilogues), the
final norm, the vocab-parallel LM head and the argmax.  Default workload: the
full 28-layer Qwen3-0.6B-shaped model on a mixed batch (4 prefill sequences of
512 tokens + 128 decode sequences at 2048 cached tokens), tp_size 2 emulated on
one GPU.  Prints one JSON line; its "workloads" key holds the same measurement
(step time, tokens/s, each kernel's roofline fraction) for the other
configurations, taken in the same run.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--tp N]

--impl reference times the CPU oracle (fp64, plain torch) on the host cores on
a bounded sample of the same workload.  Under torchrun (N > 1) every rank runs
an independent replica (the tensor-parallel ranks are emulated inside one GPU);
rank 0 prints.
"""

from __future__ import annotations

import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import synth  # noqa: E402

DEFAULT_WORKLOAD = "qwen3_0.6b_model_mixed"
DEFAULT_TP = 2
# measured in the same run as the main line, one after another (each frees its
# buffers before the next is built)
# (workload, tp_size, page size of a paged KV cache or 0 for the contiguous one)
SUB_RECORDS = (("qwen3_0.6b_layer_prefill2048", 1, 0), ("qwen3_0.6b_layer_prefill2048", 2, 0),
               ("qwen3_0.6b_layer_decode64x4096", 1, 0), ("qwen3_0.6b_layer_decode64x4096", 2, 0),
               ("qwen3_0.6b_layer_decode64x4096", 4, 0), ("qwen3_0.6b_layer_decode64x4096", 2, 128),
               ("qwen3_32b_layer_tp16_decode32x2048", 16, 0), ("qwen3_32b_layer_tp16_prefill1024", 16, 0),
               ("qwen3_0.6b_model_mixed", 1, 0), ("qwen3_0.6b_model_mixed", 4, 0))
METRIC = "tokens/sec per layer-forward (prefill & decode) on 1 GB300; % HBM BW / % TC peak"
L2_FLUSH_BYTES = 256 << 20
# tensor-core operands fp16 (weights converted from bf16 at shard time) and bf16
# (KV cache, prefill q split into bf16 high + low parts); fp32 accumulators and
# fp32 residual stream
DTYPE = "f16/bf16 operands, f32 accumulate"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d["bf16_tflops_sustained"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def workload_config(w: synth.Workload, n: int) -> dict:
    s = w.shape
    return {"workload": w.name,
            "shape": f"hidden {s.hidden}, {s.num_q_heads} q / {s.num_kv_heads} kv heads, head_dim {s.head_dim}, "
                     f"intermediate {s.intermediate}, vocab {s.vocab}, {w.layers_run} layer(s)",
            "batch": f"{len(w.prefill)} prefill seqs {[q for q, _ in w.prefill]} + {len(w.decode)} decode seqs",
            "tokens_per_step": w.num_tokens, "tp_size": n, "tp_emulated_on_one_gpu": True,
            "step": "embed(ids) + decoder layer(s) + final norm + LM head + argmax",
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MB written, then another "
                  f"{L2_FLUSH_BYTES >> 20} MB read so the written lines are evicted; outside the step events)"}


# ---------------------------------------------------------------------------
# algorithmic work per launch of each kernel kind (emulated TP: all ranks' work)
# ---------------------------------------------------------------------------

# DRAM bytes (read + write) per launch from one ncu capture of the kernel,
# keyed by (workload, tp_size, kernel); each entry records a hash of the kernel's
# source at capture time and is reported only while the source is unchanged.
# The summaries of those captures are under profiles/.
NCU_TRAFFIC = {
    # one layer of the mixed step (bench.py --quick --layers 1): the same decode
    # attention as each of the 28 layers' (128 sequences x 2049 keys, tp 2); the
    # main and the side launch of the layer summed (serialised under ncu, the main
    # launch finds every item)
    ("qwen3_0.6b_model_mixed", 2, "attn_decode"): (1082750720 + 3527424 + 71168, "k_attention.cu", "bae1123ac46e89e3"),
    ("qwen3_0.6b_layer_prefill2048", 2, "gemm_lm_head"): (311223040 + 3034624, "k_gemm.cu", "baf27ff4fbfd0bf7"),
    ("qwen3_0.6b_layer_decode64x4096", 2, "attn_decode"): (1078377984 + 3269376, "k_attention.cu", "bae1123ac46e89e3"),
    ("qwen3_32b_layer_tp16_decode32x2048", 16, "gemm_lm_head"): (1558449920 + 3330048, "k_gemm.cu", "baf27ff4fbfd0bf7"),
}
KERNEL_HEADERS = ("kernels.h", "sm100.cuh", "common.cuh")


def source_hash(cu_file: str) -> str:
    """Hash of the kernel source and the headers it includes, code only: line
    comments and blank lines do not change a kernel, so they do not count."""
    import hashlib
    import re
    d = os.path.join(ROOT, "tensor_transformer_forward_gb300", "csrc")
    m = hashlib.sha256()
    for f in (cu_file,) + KERNEL_HEADERS:
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            for line in fh:
                code = re.sub(r"(^|\s)//.*$", "", line.rstrip("\n")).rstrip()
                if code:
                    m.update(code.encode() + b"\n")
    return m.hexdigest()[:16]


def ncu_traffic(workload: str, n: int, kernel: str):
    """Measured DRAM bytes per launch, or None (no capture, or the kernel changed since)."""
    e = NCU_TRAFFIC.get((workload, n, kernel))
    if e is None or source_hash(e[1]) != e[2]:
        return None
    return e[0]


def kernel_work(kind: str, w: synth.Workload, n: int):
    """(flops, bytes) of one launch of a kernel kind: the algorithmic work of all
    emulated ranks (weights fp16, residual stream fp32, fp16 operand rows with their
    32-column sums of squares, bf16 KV cache)."""
    s = w.shape
    T, H, hd, I, V = w.num_tokens, s.hidden, s.head_dim, s.intermediate, s.vocab
    nq_l = s.num_q_heads // n
    nkv_l = s.num_kv_heads // n if s.num_kv_heads >= n else 1
    B = w.num_seqs
    nqkv = n * (nq_l + 2 * nkv_l) * hd   # merged QKV outputs of all ranks (replicated kv heads counted)
    nqo = s.num_q_heads * hd
    rows_in = T * H * 2 + T * (H // 32) * 4            # fp16 operand rows + their sums of squares
    resid = T * H * (4 + 4 + 2) + T * (H // 32) * 4    # residual read + write, next fp16 rows + sums
    if kind == "gemm_qkv":
        return 2.0 * T * H * nqkv, float(nqkv * H * 2 + rows_in + T * nqkv * 2)
    if kind == "gemm_o":
        return 2.0 * T * nqo * H, float(H * nqo * 2 + T * nqo * 2 + resid)
    if kind == "gemm_gate_up":
        return 2.0 * T * H * 2 * I, float(2 * I * H * 2 + rows_in + T * I * 2)
    if kind == "gemm_down":
        return 2.0 * T * I * H, float(H * I * 2 + T * I * 2 + resid)
    if kind == "attn_prefill":
        f, by = 0.0, 0.0
        for q, c in w.prefill:
            f += 4.0 * hd * s.num_q_heads * (q * c + q * (q + 1) / 2)
            by += q * nqo * (2 + 2 + 2) + (c + q) * n * nkv_l * hd * 2 * 2   # q hi/lo + out; K and V
        return f, by
    if kind == "attn_decode":
        keys = float(sum(c + 1 for c in w.decode))
        return 4.0 * hd * s.num_q_heads * keys, keys * n * nkv_l * hd * 2 * 2
    if kind == "gemm_lm_head":
        return 2.0 * B * V * H, float(V) * H * 2 + B * H * 2
    if kind == "embed":  # bf16 table row in; fp32 residual row and its fp16 copy out
        return 0.0, float(T) * H * (2 + 4 + 2)
    if kind == "rmsnorm":  # fp32 residual row in; fp16 row and sums out
        return 0.0, float(T) * H * (4 + 2)
    if kind == "final_norm":
        return 0.0, float(B) * H * (4 + 2)
    return 0.0, 0.0


def kernel_roofline(kind: str, w: synth.Workload, n: int, ms_per_launch: float, pk: dict) -> dict:
    """The kernel's bound (the larger of its tensor-core time at the sustained bf16 peak
    and its HBM time at the measured copy bandwidth), the rate it achieved against
    that bound and the fraction of the peak."""
    flops, by = kernel_work(kind, w, n)
    t_tc = flops / (pk["bf16_tflops_sustained"] * 1e12)
    t_hbm = by / (pk["hbm_gbs"] * 1e9)
    sec = ms_per_launch / 1e3
    if t_tc >= t_hbm and flops > 0:
        ach = flops / sec / 1e12
        return {"bound": "tensor", "achieved": round(ach, 2), "unit": "TFLOP/s",
                "frac": round(ach / pk["bf16_tflops_sustained"], 4), "roofline_us": round(t_tc * 1e6, 2)}
    ach = by / sec / 1e9 if sec > 0 else 0.0
    return {"bound": "hbm", "achieved": round(ach, 2), "unit": "GB/s", "frac": round(ach / pk["hbm_gbs"], 4),
            "roofline_us": round(t_hbm * 1e6, 2)}


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.f.read().splitlines():
            p = [x.strip() for x in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
            except ValueError:
                continue
            n += 1
            for name, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        os.unlink(self.f.name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": n}


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------

class OracleStep:
    """The CPU oracle (fp64, unsharded) on single sequences of the workload's
    step, each with its own cached context: a bounded sample of the same
    workload.  A prefill sequence may be cut to a causal prefix of its tokens."""

    def __init__(self, w: synth.Workload):
        from oracle import forward as of
        from oracle import inputs as oi
        self.of, self.oi, self.w = of, oi, w
        s = w.shape
        self.shape = oi.shape_of(s)
        self.layers = [oi.layer_weights(s, li) for li in range(w.layers_run)]
        self.head = oi.head_weights(s)
        self.cores = torch.get_num_threads()
        self._seq = (None, None)

    def order(self, k: int = 4):
        """A sample of the step's sequences: up to k/2 prefill sequences and up to
        k/2 decode sequences (all of one kind if the step has only one kind)."""
        pre = list(range(len(self.w.prefill)))
        dec = list(range(len(self.w.prefill), self.w.num_seqs))
        if not pre or not dec:
            return (pre or dec)[:k]
        return pre[: k // 2] + dec[: k - k // 2]

    def q_len(self, b: int) -> int:
        return self.w.q_lens[b]

    def run(self, b: int, tokens: int) -> float:
        """Seconds of oracle time for the first `tokens` new tokens of sequence b
        (its inputs and cache are generated outside the timing)."""
        if self._seq[0] != b:
            self._seq = (b, self.oi.workload_seq_inputs(self.w, [b], range(self.w.layers_run))[0])
        seq = self._seq[1]
        part = self.of.SeqInput(hidden=None if seq.hidden is None else seq.hidden[:tokens],
                                ids=None if seq.ids is None else seq.ids[:tokens],
                                k_cache=seq.k_cache, v_cache=seq.v_cache)
        t0 = time.perf_counter()
        self.of.run_sequence(part, self.layers, self.head, self.shape, n=0)
        return time.perf_counter() - t0


def _sample_desc(w: synth.Workload, runs: int, seqs: set, max_tokens: int, secs: float) -> str:
    what = []
    if w.prefill:
        what.append(f"causal prefixes of up to {max_tokens} tokens of prefill sequences")
    if w.decode:
        what.append("decode tokens with their cached context")
    what = " and ".join(what)
    return (f"{runs} runs of the fp64 oracle (embed + {w.layers_run} layer(s) + head) over {len(seqs)} of the "
            f"step's {w.num_seqs} sequences: {what}; {secs:.1f} s of oracle time")


def cpu_baseline(w: synth.Workload, budget_s: float = 15.0) -> dict:
    o = OracleStep(w)
    order = o.order()
    share = budget_s / len(order)
    total_t, total_tok, runs, top = 0.0, 0, 0, 0
    for b in order:
        tokens, spent = min(64, o.q_len(b)), 0.0
        while spent < share:
            dt = o.run(b, tokens)
            spent += dt
            total_tok += tokens
            runs += 1
            top = max(top, tokens)
            if dt < share / 4 and tokens < o.q_len(b):
                tokens = min(o.q_len(b), tokens * 2)
        total_t += spent
    return {"value": total_tok / total_t, "unit": "tokens/s", "cores": o.cores, "kind": "oracle",
            "sample": _sample_desc(w, runs, set(order), top, total_t)}


def run_reference(args, w: synth.Workload, n: int) -> dict:
    """One step = the oracle on one sequence of the step (a causal prefix of a
    prefill sequence sized to keep the whole run within a few minutes, or one
    decode token with its cached context), cycling through the step's sequences."""
    o = OracleStep(w)
    order = o.order()
    b0 = order[0]
    t_probe = o.run(b0, min(16, o.q_len(b0)))
    per_step = 150.0 / max(1, args.steps + args.warmup)
    tokens = max(1, min(o.q_len(b0), int(min(16, o.q_len(b0)) * per_step / max(t_probe, 1e-6))))
    for k in range(args.warmup):
        b = order[k % len(order)]
        o.run(b, min(tokens, o.q_len(b)))
    total_t, total_tok, seen = 0.0, 0, set()
    for k in range(args.steps):
        b = order[k % len(order)]
        tk = min(tokens, o.q_len(b))
        total_t += o.run(b, tk)
        total_tok += tk
        seen.add(b)
    value = total_tok / total_t
    sample = _sample_desc(w, args.steps, seen, tokens, total_t)
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": total_t * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded counter generator)",
            "config": workload_config(w, n), "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": o.cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def max_over_ranks(ms: float, world: int) -> float:
    """The slowest rank's per-step time (every rank calls this)."""
    if world <= 1:
        return ms
    on_gpu = dist.get_backend() == "nccl"
    t = torch.tensor([ms], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_step: int, world: int, ms_per_step: float) -> float:
    """Whole-job tokens/s: every rank runs its own replica of the step."""
    return world * tokens_per_step / (ms_per_step / 1e3)


def build_runner(w: synth.Workload, n: int, page_size: int = 0):
    import synth.device as sd
    from tensor_transformer_forward_gb300 import ModelConfig
    from tensor_transformer_forward_gb300.runner import TPRunner
    s = w.shape
    cfg = ModelConfig(s.hidden, s.num_q_heads, s.num_kv_heads, s.head_dim, s.intermediate, s.vocab, s.num_layers,
                      s.rms_eps, s.rope_theta, n, s.tie_word_embeddings)
    q, c = w.q_lens, w.ctx_lens
    cap = (max(a + b for a, b in zip(q, c)) + 63) // 64 * 64
    r = TPRunner(cfg, w.layers_run, w.num_seqs, cap, w.num_tokens, page_size=page_size)
    for li in range(w.layers_run):
        full = sd.layer_weights(s, li)
        r.load_layer(li, full)
        del full
    r.load_head(sd.head_weights(s))
    hmap = r.kv_head_map()
    fill = max(c)
    contig = None
    for li in range(w.layers_run):
        if fill > 0:
            if page_size:  # generated in the contiguous layout, then copied into the pages
                if contig is None:
                    contig = torch.zeros(r.ctx.kv_cache_bytes(w.num_seqs, cap), dtype=torch.uint8, device="cuda")
                sd.fill_kv_cache(contig, n, w.num_seqs, r.nkv_l, cap, s.head_dim, hmap, s.num_kv_heads, li,
                                 w.num_seqs, fill)
                r.load_kv_contiguous(li, contig)
            else:
                sd.fill_kv_cache(r.kv[li], n, w.num_seqs, r.nkv_l, cap, s.head_dim, hmap, s.num_kv_heads, li,
                                 w.num_seqs, fill)
    del contig
    batch = r.make_batch(q, c, list(range(w.num_seqs)), num_prefill=len(w.prefill))
    ids = sd.token_ids(w.num_tokens, s.vocab)
    return r, batch, ids


class L2Flush:
    """Between timed steps: write a buffer larger than L2, then read another one, so
    that the dirty lines of the write are evicted (their write-back lands here,
    outside the timed step) and L2 holds only data the step never uses."""

    def __init__(self):
        self.dst = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.src = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")

    def __call__(self):
        self.dst.zero_()
        self.src.sum()


def kernel_table(prof: dict, steps: int, w: synth.Workload, n: int, pk: dict) -> dict:
    """Per kernel kind: device time per step and per launch and its roofline."""
    out = {}
    for k, (ms, cnt) in sorted(prof.items(), key=lambda kv: -kv[1][0]):
        per_launch = ms / max(cnt, 1)
        rec = {"us_per_step": round(ms / steps * 1e3, 2), "launches_per_step": round(cnt / steps, 2),
               "us_per_launch": round(per_launch * 1e3, 2)}
        rec.update(kernel_roofline(k, w, n, per_launch, pk))
        out[k] = rec
    return out


def step_roofline_us(w: synth.Workload, n: int, launches: dict, pk: dict) -> float:
    """Sum over the step's kernels of max(flops / tensor peak, bytes / HBM bandwidth)."""
    t = 0.0
    for k, per_step in launches.items():
        flops, by = kernel_work(k, w, n)
        t += per_step * max(flops / (pk["bf16_tflops_sustained"] * 1e12), by / (pk["hbm_gbs"] * 1e9))
    return t * 1e6


def sub_record(name: str, n: int, pk: dict, flush, page_size: int = 0) -> dict:
    """One configuration measured the way the main line is: L2 flushed between
    steps, CUDA events around each step (no per-kernel events), then a second pass
    with events around every launch for the per-kernel table."""
    w = synth.WORKLOADS[name]
    r, batch, ids = build_runner(w, n, page_size)
    T, B = w.num_tokens, w.num_seqs
    hidden = torch.empty(T, w.shape.hidden, dtype=torch.float32, device="cuda")
    out_ids = torch.empty(B, dtype=torch.int32, device="cuda")

    def step():
        r.step(batch, ids=ids, hidden=hidden, out_ids=out_ids)

    step()
    torch.cuda.synchronize()
    r.check_status()
    t0 = time.perf_counter()
    for _ in range(3):
        flush()
        step()
    torch.cuda.synchronize()
    est = (time.perf_counter() - t0) / 3
    steps = max(10, min(200, int(0.15 / max(est, 1e-6))))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        flush()
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    times = sorted(a.elapsed_time(b) for a, b in ev)
    ms = sum(times) / steps
    psteps = min(steps, 20)
    r.ctx.profile_begin(list(__import__("tensor_transformer_forward_gb300").binding.KERNELS))
    for _ in range(psteps):
        flush()
        step()
    prof = r.ctx.profile_end()
    r.check_status()
    table = kernel_table(prof, psteps, w, n, pk)
    roof = step_roofline_us(w, n, {k: v["launches_per_step"] for k, v in table.items()}, pk)
    rec = {"workload": name, "tp_size": n, "kv_cache": f"paged, {page_size}-position pages" if page_size else "contiguous",
           "tokens_per_step": T, "steps": steps, "ms_per_step": round(ms, 5),
           "tokens_per_s": round(T / (ms / 1e3), 1),
           "step_ms_p10_p50_p90": [round(times[len(times) // 10], 5), round(times[len(times) // 2], 5),
                                   round(times[9 * len(times) // 10], 5)],
           "step_roofline_us": round(roof, 2), "step_roofline_frac": round(roof / (ms * 1e3), 4),
           "dominant": next(iter(table)), "kernels": table}
    del r, batch, ids, hidden, out_ids
    torch.cuda.empty_cache()
    return rec


def run_ours(args, w: synth.Workload, n: int, rank: int, world: int) -> dict:
    dev = torch.cuda.current_device()
    pk = peaks()
    flush_l2 = L2Flush()
    r, batch, ids = build_runner(w, n)
    ctx = r.ctx
    T, H, B = w.num_tokens, w.shape.hidden, w.num_seqs
    hidden = torch.empty(T, H, dtype=torch.float32, device="cuda")
    out_ids = torch.empty(B, dtype=torch.int32, device="cuda")

    def step():
        r.step(batch, ids=ids, hidden=hidden, out_ids=out_ids)

    # untimed: which kernel dominates the step, and every kernel's share
    step()
    torch.cuda.synchronize()
    r.check_status()
    ctx.profile_begin(list(__import__("tensor_transformer_forward_gb300").binding.KERNELS))
    for _ in range(5):
        flush_l2()
        step()
    prof = ctx.profile_end()
    dominant = max(prof, key=lambda k: prof[k][0])
    table = kernel_table(prof, 5, w, n, pk)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    launches0 = ctx.launch_count()
    wall0 = time.perf_counter()
    for i in range(args.steps):
        flush_l2()
        starts[i].record()
        step()
        ends[i].record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    launches = ctx.launch_count() - launches0
    # second timed pass over the same steps, with events around each launch of the
    # dominant kernel: events between two kernels split their programmatic-launch
    # overlap, so the step times above are taken without them
    ctx.profile_begin([dominant], max_launches=max(64, 64 * args.steps))
    for i in range(args.steps):
        flush_l2()
        step()
    torch.cuda.synchronize()
    dom = ctx.profile_end()
    r.check_status()
    step_ms = sorted(s.elapsed_time(e) for s, e in zip(starts, ends))
    ms = sum(step_ms) / args.steps
    ms_max = max_over_ranks(ms, world)

    # roofline of the dominant kernel, timed live in the timed region
    dms, dcount = dom.get(dominant, (0.0, 0))
    avg_ms = dms / max(dcount, 1)
    dr = kernel_roofline(dominant, w, n, avg_ms, pk)
    flops, by = kernel_work(dominant, w, n)
    roofline = {"bound": dr["bound"], "kernel": dominant, "achieved": dr["achieved"],
                "peak": pk["bf16_tflops_sustained"] if dr["bound"] == "tensor" else pk["hbm_gbs"], "unit": dr["unit"],
                "frac": dr["frac"], "traffic": ncu_traffic(w.name, n, dominant),
                "peak_source": f"{pk['source']} ({'sustained bf16' if dr['bound'] == 'tensor' else 'copy'})",
                "algorithmic_per_launch": flops if dr["bound"] == "tensor" else by,
                "avg_launch_ms": round(avg_ms, 4), "launches_timed": dcount,
                "launch_timing": "CUDA events around each launch, in a second timed pass of the same steps"}

    # end to end through the public API, every step: the step's ids from page-locked
    # host memory and its next ids back into page-locked host memory.  The embedding
    # kernel reads the ids and the LM head writes the result over the host link
    # (NVLink-C2C on GB300) inside the timed region, with no separate copy operations.
    ids_host = ids.cpu().pin_memory()
    out_host = torch.full((B,), -1, dtype=torch.int32).pin_memory()
    e2e_steps = min(args.steps, 200)
    e_s = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    e_e = [torch.cuda.Event(enable_timing=True) for _ in range(e2e_steps)]
    for i in range(e2e_steps):
        flush_l2()
        e_s[i].record()
        r.step(batch, ids=ids_host, hidden=hidden, out_ids=out_host)
        e_e[i].record()
    torch.cuda.synchronize()
    wall_all = time.perf_counter() - wall0
    clk = clocks.stop()
    clk["window"] = (f"the timed steps, the dominant kernel's timed pass and the e2e pass "
                     f"({2 * args.steps + e2e_steps} steps, {wall_all:.2f} s)")
    r.check_status()
    if not torch.equal(out_host, out_ids.cpu()):
        raise RuntimeError("the ids written to host memory differ from the device run's")
    e2e_ms = sum(s.elapsed_time(e) for s, e in zip(e_s, e_e)) / e2e_steps
    roof_us = step_roofline_us(w, n, {k: v["launches_per_step"] for k, v in table.items()}, pk)
    del r, batch, ids, hidden, out_ids
    torch.cuda.empty_cache()

    config = workload_config(w, n)
    if w.layers_run > 1:
        config["tokens_x_layers_per_s"] = round(T * w.layers_run / (ms_max / 1e3), 1)
    line = {"metric": METRIC, "value": job_throughput(T, world, ms_max), "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
            "data": "synthetic (seeded counter generator; random-init weights of the named shape)",
            "config": config, "roofline": roofline,
            "e2e": {"value": job_throughput(T, world, max_over_ranks(e2e_ms, world)), "unit": "tokens/s",
                    "h2d_bytes_per_step": T * 4, "d2h_bytes_per_step": B * 4,
                    "transfer": "ids read from / next ids written to page-locked host memory by the kernels"},
            "gpu_launches": launches, "clocks": clk,
            "step_roofline_us": round(roof_us, 2), "step_roofline_frac": round(roof_us / (ms_max * 1e3), 4),
            "kernels": table, "wall_s_timed_region": round(wall, 3),
            "step_ms_p10_p50_p90": [round(step_ms[len(step_ms) // 10], 4), round(step_ms[len(step_ms) // 2], 4),
                                    round(step_ms[9 * len(step_ms) // 10], 4)]}
    if not args.no_sub and world == 1:
        line["workloads"] = [sub_record(name, tp, pk, flush_l2, ps) for name, tp, ps in SUB_RECORDS
                             if not (name == w.name and tp == n and ps == 0)]
    return line


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--tp", type=int, default=None)
    ap.add_argument("--quick", action="store_true",
                    help="only warm-up + timed steps (no kernel breakdown, e2e or CPU baseline): for profilers")
    ap.add_argument("--no-sub", action="store_true", help="skip the other configurations' records")
    ap.add_argument("--layers", type=int, default=None,
                    help="with --quick: run only the first LAYERS layers of the workload (each layer's launches "
                         "unchanged, less memory held): for profilers")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = synth.WORKLOADS[args.workload]
    if args.layers is not None:
        if not args.quick or not 1 <= args.layers <= w.layers_run:
            ap.error("--layers needs --quick and 1 <= LAYERS <= the workload's layers")
        w = dataclasses.replace(w, layers_run=args.layers)
    if args.tp is not None:
        n = args.tp
    elif w.name == DEFAULT_WORKLOAD:
        n = DEFAULT_TP
    else:
        n = max(w.tp_sizes)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, w, n)), flush=True)
        return
    if world > 1:
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    if args.quick:
        r, batch, ids = build_runner(w, n)
        hidden = torch.empty(w.num_tokens, w.shape.hidden, dtype=torch.float32, device="cuda")
        out_ids = torch.empty(w.num_seqs, dtype=torch.int32, device="cuda")
        for _ in range(args.warmup + args.steps):
            r.step(batch, ids=ids, hidden=hidden, out_ids=out_ids)
        torch.cuda.synchronize()
        r.check_status()
        print(json.dumps({"quick": True, "workload": w.name, "tp": n, "steps": args.steps,
                          "launches": r.ctx.launch_count()}), flush=True)
        return
    line = run_ours(args, w, n, rank, world)
    if rank == 0:
        if world == 1:
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
