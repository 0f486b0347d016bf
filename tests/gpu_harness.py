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


def assert_close_bf16_stored(got, ref, what: str, tol: float = TOL) -> float:
    """For outputs the method stores as bf16 (the KV cache): the bound applies on
    top of the format's own rounding, half a bf16 ulp of each reference value
    (bf16 keeps 8 significant bits, so the half-ulp of x is 2^(floor(log2|x|) - 8))."""
    got = got.to(torch.float64).cpu()
    ref = ref.to(torch.float64).cpu()
    mag = ref.abs().clamp_min(1e-30)
    half_ulp = torch.exp2(torch.floor(torch.log2(mag)) - 8)
    excess = ((got - ref).abs() - half_ulp).clamp_min(0.0)
    e = float(excess.max()) / max(float(ref.pow(2).mean().sqrt()), 1e-30)
    assert e <= tol, f"{what}: max(|err| - half bf16 ulp)/RMS(ref) = {e:.3e} > {tol}"
    return e


@functools.lru_cache(maxsize=64)
def oracle_layer(s: synth.ModelShape, layer: int, perturbed: bool) -> of.LayerWeights:
    return oi.layer_weights(s, layer, perturbed_norms=perturbed)


@functools.lru_cache(maxsize=4)
def oracle_head(s: synth.ModelShape, perturbed: bool) -> of.HeadWeights:
    return oi.head_weights(s, perturbed_norms=perturbed)


class GpuStep:
    """Runs one step of a workload on the GPU and keeps what the tests compare."""

    def __init__(self, w: synth.Workload, n: int, layers: Optional[int] = None, perturbed: bool = False,
                 head: bool = True, logits: bool = True, capacity: Optional[int] = None,
                 keep_intermediates: bool = False, q_norm_scale: float = 1.0):
        from tensor_transformer_forward_gb300.runner import TPRunner
        self.w, self.n, self.perturbed = w, n, perturbed
        s = w.shape
        self.L = w.layers_run if layers is None else layers
        q, c = w.q_lens, w.ctx_lens
        max_kv = max(a + b for a, b in zip(q, c))
        self.capacity = capacity or ((max_kv + 63) // 64 * 64)
        self.runner = TPRunner(model_config(s, n), self.L, w.num_seqs, self.capacity, w.num_tokens)
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
        for li in range(self.L):
            r.kv[li].zero_()
            if fill > 0:
                sd.fill_kv_cache(r.kv[li], n, w.num_seqs, r.nkv_l, self.capacity, s.head_dim, hmap, s.num_kv_heads,
                                 li, w.num_seqs, fill)
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
        view = self.runner.kv_view(layer)
        c0 = self.w.ctx_lens[b]
        t0, t1 = self.seq_rows(b)
        q = t1 - t0
        got: Dict[int, Tuple[torch.Tensor, torch.Tensor]] = {}
        nkv_l = self.runner.nkv_l
        for r in range(self.n):
            for j in range(nkv_l):
                g = self.head_map[r * nkv_l + j]
                k = view[r, 0, b, j, c0:c0 + q].float().cpu()
                v = view[r, 1, b, j, c0:c0 + q].float().cpu()
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
    hw = oracle_head(s, perturbed) if (head or w.input_from_ids) else None
    ins = oi.workload_seq_inputs(w, seqs, range(layers))
    outs = [of.run_sequence(seq, lw, hw, shape, n=0, head=head) for seq in ins]
    return outs, ins


def oracle_run_sp(w: synth.Workload, seq: int, layers: int, n: int, perturbed: bool = False, head: bool = True):
    """One sequence through the oracle's tensor + sequence parallel form."""
    s = w.shape
    lw = [oracle_layer(s, li, perturbed) for li in range(layers)]
    hw = oracle_head(s, perturbed) if (head or w.input_from_ids) else None
    ins = oi.workload_seq_inputs(w, [seq], range(layers))
    return of.run_sequence_sp(ins[0], lw, hw, oi.shape_of(s), n, head=head)


def check_step(g: GpuStep, seqs: Sequence[int], head: bool = True, layers: Optional[int] = None) -> Dict[str, float]:
    """Compare the chosen sequences of a GPU step against the oracle."""
    L = g.L if layers is None else layers
    outs, ins = oracle_run(g.w, seqs, L, g.perturbed, head)
    errs = {}
    for b, o, i in zip(seqs, outs, ins):
        t0, t1 = g.seq_rows(b)
        errs[f"hidden[{b}]"] = assert_close(g.hidden[t0:t1].float().cpu(), o.hidden, f"hidden of seq {b}")
        c0 = g.w.ctx_lens[b]
        K, V = g.new_kv(L - 1, b)
        errs[f"k[{b}]"] = assert_close_bf16_stored(K, o.k_cache[L - 1][:, c0:], f"new K of seq {b}")
        errs[f"v[{b}]"] = assert_close_bf16_stored(V, o.v_cache[L - 1][:, c0:], f"new V of seq {b}")
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
    return errs
