"""The oracle's emulated collectives against real ones: two CPU processes over
Gloo, one rank each, the way tp.py runs ("Tensor parallelism from scratch",
section "Implementation").  Rank 0 compares with the single-process emulation."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import forward as of

D = torch.float64
SHAPE = of.Shape(hidden=48, num_q_heads=4, num_kv_heads=2, head_dim=12, intermediate=64, vocab=91,
                 num_layers=2, tie_word_embeddings=True)


def _inputs():
    g = torch.Generator().manual_seed(21)
    H, nq, nkv, hd, I = SHAPE.hidden, SHAPE.num_q_heads, SHAPE.num_kv_heads, SHAPE.head_dim, SHAPE.intermediate
    r = lambda *s: torch.randn(*s, dtype=D, generator=g) * 0.2  # noqa: E731
    layers = [of.LayerWeights(q=r(nq * hd, H), k=r(nkv * hd, H), v=r(nkv * hd, H), o=r(H, nq * hd),
                              gate=r(I, H), up=r(I, H), down=r(H, I), in_norm=1 + r(H), post_norm=1 + r(H),
                              q_norm=1 + r(hd), k_norm=1 + r(hd)) for _ in range(2)]
    emb = torch.randn(SHAPE.vocab, H, dtype=D, generator=g)
    hw = of.HeadWeights(embed=emb, lm_head=emb, final_norm=1 + r(H))
    ids = torch.randint(0, SHAPE.vocab, (6,), generator=g)
    return layers, hw, ids


def _all_reduce(x, counter):
    counter[0] += 1
    dist.all_reduce(x)
    return x


def _rank_forward(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        layers, hw, ids = _inputs()
        n, r, hd, eps = world, rank, SHAPE.head_dim, SHAPE.rms_eps
        cnt = [0]
        start, end = of.vocab_range(SHAPE.vocab, n, r)
        e_r = of.shard_tensor("embed", hw.embed, SHAPE, n, r)
        outside = (ids < start) | (ids >= end)
        x = _all_reduce(e_r[(ids - start).masked_fill(outside, 0)].masked_fill(outside[:, None], 0.0), cnt)
        T = ids.shape[0]
        pos = torch.arange(T)
        for w in layers:
            rl = of.shard_layer(w, SHAPE, n, r)
            h = of.rms_norm(x, rl.in_norm, eps)
            qkv = h @ rl.qkv.T
            nqw, nkw = rl.nq_l * hd, rl.nkv_l * hd
            q = qkv[:, :nqw].reshape(T, rl.nq_l, hd).transpose(0, 1)
            k = qkv[:, nqw:nqw + nkw].reshape(T, rl.nkv_l, hd).transpose(0, 1)
            v = qkv[:, nqw + nkw:].reshape(T, rl.nkv_l, hd).transpose(0, 1)
            q = of.apply_rope(of.rms_norm(q, rl.q_norm, eps), pos, SHAPE.rope_theta)
            k = of.apply_rope(of.rms_norm(k, rl.k_norm, eps), pos, SHAPE.rope_theta)
            o = of.causal_gqa_attention(q, k, v).transpose(0, 1).reshape(T, nqw)
            x = x + _all_reduce(o @ rl.o.T, cnt)
            h2 = of.rms_norm(x, rl.post_norm, eps)
            gu = h2 @ rl.gate_up.T
            x = x + _all_reduce((of.silu(gu[:, :rl.i_l]) * gu[:, rl.i_l:]) @ rl.down.T, cnt)
        z = of.rms_norm(x[-1:], hw.final_norm, eps)
        local = z @ of.shard_tensor("lm_head", hw.lm_head, SHAPE, n, r).T
        per = of.div_ceil(SHAPE.vocab, n)
        if local.shape[-1] < per:
            local = torch.cat([local, torch.zeros(1, per - local.shape[-1], dtype=D)], dim=-1)
        parts = [torch.empty_like(local) for _ in range(n)]
        dist.all_gather(parts, local)
        logits = torch.cat(parts, dim=-1)[0, : SHAPE.vocab]
        if rank == 0:
            out_q.put((logits, cnt[0]))
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_gloo_ranks_match_emulation_and_single_process():
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_forward, args=(r, 2, port, out_q)) for r in range(2)]
    for p in procs:
        p.start()
    logits, count = out_q.get(timeout=90)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    layers, hw, ids = _inputs()
    seq = of.SeqInput(hidden=None, ids=ids, k_cache=[torch.zeros(2, 0, 12, dtype=D)] * 2,
                      v_cache=[torch.zeros(2, 0, 12, dtype=D)] * 2)
    emu = of.run_sequence(seq, layers, hw, SHAPE, n=2)
    single = of.run_sequence(seq, layers, hw, SHAPE, n=0)
    assert count == 2 * SHAPE.num_layers + 1
    assert torch.allclose(logits, emu.logits, rtol=1e-12, atol=1e-12)
    assert torch.allclose(logits, single.logits, rtol=1e-12, atol=1e-12)
