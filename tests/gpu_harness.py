"""Shared set-up for the GPU parity tests: one workload step through the C ABI
(inputs from the device generator) and the same sequences through the CPU
oracle (inputs from the host generator, bit-identical)."""

from __future__ import annotations

import functools
from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np
import torch

import synth
import synth.device as sd
from oracle import forward as of
from oracle import inputs as oi

TOL = 2e-2  # max |err| <= TOL * RMS(reference), per tensor
MARGIN = 0.05  # greedy ids compared where the reference top-2 margin exceeds this
# the workloads' KV cache is bf16: the oracle's cache stores bf16 too (its arithmetic
# stays fp64), and attention reads what the cache holds
KV_DTYPE = torch.bfloat16


def model_config(s: synth.ModelShape, n: int):
    from tensor_transformer_forward_gb300 import ModelConfig
    return ModelConfig(s.hidden, s.num_q_heads, s.num_kv_heads, s.head_dim, s.intermediate, s.vocab, s.num_layers,
                       s.rms_eps, s.rope_theta, n, s.tie_word_embeddings)


def rel_err(got: torch.Tensor, ref: torch.Tensor) -> float:
    got = got.to(torch.float64).cpu()
    ref = ref.to(torch.float64).cpu()
    rms = float(ref.pow(2).mean().sqrt())
    return float((got - ref).abs().max()) / max(rms, 1e-30)


def assert_close(got, ref, what: str, tol: float = TOL) -> float:
    e = rel_err(got, ref)
    assert e <= tol, f"{what}: max|err|/RMS(ref) = {e:.3e} > {tol}"
    return e


@functools.lru_cache(maxsize=64)
def oracle_layer(s: synth.ModelShape, layer: int, perturbed: bool) -> of.LayerWeights:
    return oi.layer_weights(s, layer, perturbed_norms=perturbed)


@functools.lru_cache(maxsize=4)
def oracle_head(s: synth.ModelShape, perturbed: bool, need_embed: bool = True) -> of.HeadWeights:
    return oi.head_weights(s, perturbed_norms=perturbed, need_embed=need_embed)


class GpuStep:
    """Runs one step of a workload on the GPU and keeps what the tests compare."""

    def __init__(self, w: synth.Workload, n: int, layers: Optional[int] = None, perturbed: bool = False,
                 head: bool = True, logits: bool = True, capacity: Optional[int] = None,
                 keep_intermediates: bool = False, q_norm_scale: float = 1.0, page_size: int = 0):
        from tensor_transformer_forward_gb300.runner import TPRunner
        self.w, self.n, self.perturbed = w, n, perturbed
        s = w.shape
        self.L = w.layers_run if layers is None else layers
        q, c = w.q_lens, w.ctx_lens
        max_kv = max(a + b for a, b in zip(q, c))
        self.capacity = capacity or ((max_kv + 63) // 64 * 64)
        self.runner = TPRunner(model_config(s, n), self.L, w.num_seqs, self.capacity, w.num_tokens,
                               page_size=page_size, spare_pages=3 if page_size else 0)
        r = self.runner
        if keep_intermediates:
            r.ctx.keep_intermediates()
        for li in range(self.L):
            full = sd.layer_weights(s, li, perturbed)
            if q_norm_scale != 1.0:  # a power of two keeps the bf16 weights exact
                full["q_norm"].mul_(q_norm_scale)
            r.load_layer(li, full)
            del full
        if head or w.input_from_ids:
            r.load_head(sd.head_weights(s, perturbed))
        fill = max(c) if c else 0
        hmap = r.kv_head_map()
        contig = None
        for li in range(self.L):
            r.kv[li].zero_()
            if fill > 0:
                if page_size:  # filled in the contiguous layout, then copied into the pages
                    if contig is None:
                        contig = torch.zeros(r.ctx.kv_cache_bytes(w.num_seqs, self.capacity), dtype=torch.uint8,
                                             device="cuda")
                    contig.zero_()
                    sd.fill_kv_cache(contig, n, w.num_seqs, r.nkv_l, self.capacity, s.head_dim, hmap,
                                     s.num_kv_heads, li, w.num_seqs, fill)
                    r.load_kv_contiguous(li, contig)
                else:
                    sd.fill_kv_cache(r.kv[li], n, w.num_seqs, r.nkv_l, self.capacity, s.head_dim, hmap,
                                     s.num_kv_heads, li, w.num_seqs, fill)
        del contig
        self.batch = r.make_batch(q, c, list(range(w.num_seqs)), num_prefill=len(w.prefill))
        T = w.num_tokens
        self.ids = sd.token_ids(T, s.vocab) if w.input_from_ids else None
        self.hidden_in = None if w.input_from_ids else sd.hidden(T, s.hidden)
        self.out_ids = torch.full((w.num_seqs,), -1, dtype=torch.int32, device="cuda")
        self.logits = torch.empty(w.num_seqs, s.vocab, dtype=torch.float32, device="cuda") if (head and logits) else None
        hidden = None if self.hidden_in is None else self.hidden_in.float()
        self.hidden = r.step(self.batch, ids=self.ids, hidden=hidden, out_ids=self.out_ids, out_logits=self.logits,
                             layers=self.L, run_head=head)
        torch.cuda.synchronize()
        r.check_status()
        self.head_map = hmap

    def seq_rows(self, b: int) -> Tuple[int, int]:
        cu = np.concatenate([[0], np.cumsum(self.w.q_lens)])
        return int(cu[b]), int(cu[b + 1])

    def new_kv(self, layer: int, b: int) -> Tuple[torch.Tensor, torch.Tensor]:
        """The positions this step wrote, gathered to global kv heads [nkv, q_len, hd]
        (the first rank holding a head supplies it); also checks replicas agree."""
        s = self.w.shape
        c0 = self.w.ctx_lens[b]
        t0, t1 = self.seq_rows(b)
        q = t1 - t0
        got: Dict[int, Tuple[torch.Tensor, torch.Tensor]] = {}
        nkv_l = self.runner.nkv_l
        pos = self.runner.kv_positions(layer, b, c0, c0 + q)  # [n, 2, nkv_l, q, hd]
        for r in range(self.n):
            for j in range(nkv_l):
                g = self.head_map[r * nkv_l + j]
                k = pos[r, 0, j].float().cpu()
                v = pos[r, 1, j].float().cpu()
                if g in got:
                    assert torch.equal(got[g][0], k) and torch.equal(got[g][1], v), "replicated kv heads differ"
                else:
                    got[g] = (k, v)
        K = torch.stack([got[g][0] for g in range(s.num_kv_heads)])
        V = torch.stack([got[g][1] for g in range(s.num_kv_heads)])
        return K, V


def oracle_run(w: synth.Workload, seqs: Sequence[int], layers: int, perturbed: bool = False, head: bool = True):
    s = w.shape
    shape = oi.shape_of(s)
    lw = [oracle_layer(s, li, perturbed) for li in range(layers)]
    hw = oracle_head(s, perturbed, w.input_from_ids) if (head or w.input_from_ids) else None
    ins = oi.workload_seq_inputs(w, seqs, range(layers))
    outs = [of.run_sequence(seq, lw, hw, shape, n=0, head=head, kv_dtype=KV_DTYPE) for seq in ins]
    return outs, ins


def oracle_run_sp(w: synth.Workload, seq: int, layers: int, n: int, perturbed: bool = False, head: bool = True):
    """One sequence through the oracle's tensor + sequence parallel form."""
    s = w.shape
    lw = [oracle_layer(s, li, perturbed) for li in range(layers)]
    hw = oracle_head(s, perturbed) if (head or w.input_from_ids) else None
    ins = oi.workload_seq_inputs(w, [seq], range(layers))
    return of.run_sequence_sp(ins[0], lw, hw, oi.shape_of(s), n, head=head, kv_dtype=KV_DTYPE)


def check_step(g: GpuStep, seqs: Sequence[int], head: bool = True, layers: Optional[int] = None) -> Dict[str, float]:
    """Compare the chosen sequences of a GPU step against the oracle."""
    L = g.L if layers is None else layers
    outs, ins = oracle_run(g.w, seqs, L, g.perturbed, head)
    errs = {}
    for b, o, i in zip(seqs, outs, ins):
        t0, t1 = g.seq_rows(b)
        errs[f"hidden[{b}]"] = assert_close(g.hidden[t0:t1].float().cpu(), o.hidden, f"hidden of seq {b}")
        # the new positions' K / V, stored bf16 on the GPU, against the oracle's values
        # before its cache stored them: the bar includes the bf16 rounding
        K, V = g.new_kv(L - 1, b)
        errs[f"k[{b}]"] = assert_close(K, o.k_new[L - 1], f"new K of seq {b}")
        errs[f"v[{b}]"] = assert_close(V, o.v_new[L - 1], f"new V of seq {b}")
        if head:
            if g.logits is not None:
                errs[f"logits[{b}]"] = assert_close(g.logits[b].cpu(), o.logits, f"logits of seq {b}")
            top2 = torch.topk(o.logits, 2).values
            if float(top2[0] - top2[1]) > MARGIN:
                assert int(g.out_ids[b]) == o.next_id, f"greedy id of seq {b}: {int(g.out_ids[b])} != {o.next_id}"
            elif g.logits is not None:
                # several ids are correct: the GPU's pick must be a maximiser of its own logits
                lg = g.logits[b].cpu()
                assert float(lg[int(g.out_ids[b])]) == float(lg.max())
    print(f"\n{g.w.name} tp {g.n}: " + ", ".join(f"{k} {v:.2e}" for k, v in errs.items()))
    return errs
