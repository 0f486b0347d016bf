"""Sequence parallelism in the oracle ("Tensor parallelism from scratch", section
"Exercises", exercise 1), pinned on the CPU: the token-chunked forward equals the
unsharded forward (itself pinned against brute force) and the all-reduce TP
emulation; each layer swaps its two all-reduces for two reduce-scatters and two
all-gathers; every rank normalizes only its own tokens; the emulated collectives
equal real Gloo ones on two processes, uneven chunks included; planted slips in
the chunked arithmetic are caught."""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import forward as of

D = torch.float64
SHAPE = of.Shape(hidden=48, num_q_heads=4, num_kv_heads=2, head_dim=12, intermediate=64, vocab=91,
                 num_layers=2, tie_word_embeddings=False)


def _weights(seed: int = 41):
    g = torch.Generator().manual_seed(seed)
    H, nq, nkv, hd, I = SHAPE.hidden, SHAPE.num_q_heads, SHAPE.num_kv_heads, SHAPE.head_dim, SHAPE.intermediate
    r = lambda *s: torch.randn(*s, dtype=D, generator=g) * 0.2  # noqa: E731
    layers = [of.LayerWeights(q=r(nq * hd, H), k=r(nkv * hd, H), v=r(nkv * hd, H), o=r(H, nq * hd),
                              gate=r(I, H), up=r(I, H), down=r(H, I), in_norm=1 + r(H), post_norm=1 + r(H),
                              q_norm=1 + r(hd), k_norm=1 + r(hd)) for _ in range(2)]
    hw = of.HeadWeights(embed=torch.randn(SHAPE.vocab, H, dtype=D, generator=g),
                        lm_head=torch.randn(SHAPE.vocab, H, dtype=D, generator=g), final_norm=1 + r(H))
    return layers, hw


def _seq(T: int, ctx: int, seed: int = 42) -> of.SeqInput:
    g = torch.Generator().manual_seed(seed)
    shp = (SHAPE.num_kv_heads, ctx, SHAPE.head_dim)
    return of.SeqInput(hidden=None, ids=torch.randint(0, SHAPE.vocab, (T,), generator=g),
                       k_cache=[torch.randn(*shp, dtype=D, generator=g) for _ in range(2)],
                       v_cache=[torch.randn(*shp, dtype=D, generator=g) for _ in range(2)])


def _close(a, b, tol=1e-12):
    scale = max(float(b.abs().max()), 1.0) if b.numel() else 1.0
    return a.shape == b.shape and (a.numel() == 0 or float((a - b).abs().max()) <= tol * scale)


def _sp_agrees(n: int = 2, T: int = 7, ctx: int = 5) -> bool:
    layers, hw = _weights()
    seq = _seq(T, ctx)
    sp = of.run_sequence_sp(seq, layers, hw, SHAPE, n)
    ref = of.run_sequence(seq, layers, hw, SHAPE, n=0)
    return (_close(torch.cat(sp.hidden_chunks), ref.hidden) and _close(sp.logits, ref.logits)
            and all(_close(a, b) for a, b in zip(sp.k_cache + sp.v_cache, ref.k_cache + ref.v_cache)))


def test_token_chunks_partition_the_tokens():
    for T in range(0, 12):
        for n in (1, 2, 3, 4):
            ch = [of.token_chunk(T, n, r) for r in range(n)]
            assert ch[0][0] == 0 and ch[-1][1] == T
            assert all(ch[r][1] == ch[r + 1][0] for r in range(n - 1))
            sizes = [b - a for a, b in ch]
            assert max(sizes) - min(sizes) <= 1 and sizes == sorted(sizes, reverse=True)


@pytest.mark.parametrize("n", [2, 4])
@pytest.mark.parametrize("T,ctx", [(1, 0), (3, 5), (8, 0), (13, 9)])
def test_sp_equals_unsharded_and_all_reduce_tp(n, T, ctx):
    """n = 4 replicates each kv head on two ranks; T < n leaves ranks without tokens."""
    layers, hw = _weights()
    seq = _seq(T, ctx)
    sp = of.run_sequence_sp(seq, layers, hw, SHAPE, n)
    tp = of.run_sequence(seq, layers, hw, SHAPE, n=n)
    ref = of.run_sequence(seq, layers, hw, SHAPE, n=0)
    got = torch.cat(sp.hidden_chunks)
    for r, x in enumerate(sp.hidden_chunks):
        assert x.shape[0] == of.token_chunk(T, n, r)[1] - of.token_chunk(T, n, r)[0]
    assert _close(got, ref.hidden) and _close(got, tp.hidden)
    assert _close(sp.logits, ref.logits) and sp.next_id == ref.next_id == tp.next_id
    for a, b in zip(sp.k_cache + sp.v_cache, ref.k_cache + ref.v_cache):
        assert _close(a, b)


def test_sp_hidden_rows_as_input():
    layers, hw = _weights()
    g = torch.Generator().manual_seed(7)
    x = torch.randn(6, SHAPE.hidden, dtype=D, generator=g)
    empty = [torch.zeros(SHAPE.num_kv_heads, 0, SHAPE.head_dim, dtype=D)] * 2
    seq = of.SeqInput(hidden=x, ids=None, k_cache=empty, v_cache=empty)
    sp = of.run_sequence_sp(seq, layers, hw, SHAPE, 4)
    ref = of.run_sequence(seq, layers, hw, SHAPE, n=0)
    assert _close(torch.cat(sp.hidden_chunks), ref.hidden) and _close(sp.logits, ref.logits)


def test_collectives_and_per_rank_norm_rows(monkeypatch):
    """Per layer two reduce-scatters and two all-gathers replace the two
    all-reduces; the hidden-size RMSNorms touch T rows in all instead of n x T."""
    layers, hw = _weights()
    n, T = 4, 10
    seq = _seq(T, 3)
    rows = {"count": 0}
    plain = of.rms_norm

    def counting(x, w, eps):
        if x.shape[-1] == SHAPE.hidden:
            rows["count"] += x.shape[0] if x.dim() == 2 else 1
        return plain(x, w, eps)

    monkeypatch.setattr(of, "rms_norm", counting)
    comm = of.Comm()
    of.run_sequence_sp(seq, layers, hw, SHAPE, n, comm=comm)
    L = len(layers)
    assert comm.num_all_reduce == 0
    assert comm.num_reduce_scatter == 2 * L + 1  # two per layer and the embedding's
    assert comm.num_all_gather_rows == 2 * L + 1  # two per layer and the final norm's
    assert comm.num_all_gather == 1  # the logits
    assert rows["count"] == 2 * L * T + T
    rows["count"] = 0
    tcomm = of.Comm()
    of.run_sequence(seq, layers, hw, SHAPE, n=n, comm=tcomm)
    assert tcomm.num_all_reduce == 2 * L + 1
    assert rows["count"] == 2 * L * n * T + 1  # every rank normalizes every token; the head's last row


# ---- planted slips (each must break the agreement above) ----

def _rs_no_sum(self, partials):
    self.num_reduce_scatter += 1
    T, n = partials[0].shape[0], len(partials)
    return [partials[r][slice(*of.token_chunk(T, n, r))].clone() for r in range(n)]


def _ag_reversed(self, chunks):
    self.num_all_gather_rows += 1
    return torch.cat(list(chunks)[::-1], dim=0)


def test_unmodified_sp_agrees():
    assert _sp_agrees()


@pytest.mark.parametrize("name,patch", [("reduce_scatter", _rs_no_sum), ("all_gather_rows", _ag_reversed)])
def test_planted_collective_slip_is_caught(monkeypatch, name, patch):
    monkeypatch.setattr(of.Comm, name, patch)
    assert not _sp_agrees()


def test_planted_residual_on_the_wrong_chunk_is_caught(monkeypatch):
    original = of.Comm.reduce_scatter

    def rotated(self, partials):
        out = original(self, partials)
        return out[1:] + out[:1]

    monkeypatch.setattr(of.Comm, "reduce_scatter", rotated)
    try:
        ok = _sp_agrees(n=2, T=8)  # equal chunks: shapes still fit, values land on the wrong tokens
    except RuntimeError:
        ok = False
    assert not ok


# ---- real collectives: two Gloo processes ----

def _rank_sp(rank, world, port, T, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        layers, hw = _weights()
        seq = _seq(T, 4)
        n, r, eps = world, rank, SHAPE.rms_eps
        chunks = [of.token_chunk(T, n, q) for q in range(n)]
        a, b = chunks[r]
        width = max(e - s for s, e in chunks)

        def reduce_scatter(full):  # full: this rank's [T, H] partial
            out = torch.empty(b - a, full.shape[1], dtype=D)
            dist.reduce_scatter(out, [full[s:e].contiguous() for s, e in chunks])
            return out

        def all_gather_rows(mine):  # Gloo gathers equal sizes: pad to the widest chunk
            pad = torch.zeros(width, mine.shape[1], dtype=D)
            pad[: mine.shape[0]] = mine
            parts = [torch.empty_like(pad) for _ in range(n)]
            dist.all_gather(parts, pad)
            return torch.cat([p[: e - s] for p, (s, e) in zip(parts, chunks)])

        start, end = of.vocab_range(SHAPE.vocab, n, r)
        e_r = of.shard_tensor("embed", hw.embed, SHAPE, n, r)
        ids = seq.ids
        outside = (ids < start) | (ids >= end)
        x = reduce_scatter(e_r[(ids - start).masked_fill(outside, 0)].masked_fill(outside[:, None], 0.0))
        for li, w in enumerate(layers):
            rl = of.shard_layer(w, SHAPE, n, r)
            kc = of.split_kv_by_rank(seq.k_cache[li], SHAPE, n)[r]
            vc = of.split_kv_by_rank(seq.v_cache[li], SHAPE, n)[r]
            h = all_gather_rows(of.rms_norm(x, rl.in_norm, eps))
            hd, ctx = SHAPE.head_dim, kc.shape[1]
            pos = torch.arange(ctx, ctx + T)
            qkv = h @ rl.qkv.T
            nqw, nkw = rl.nq_l * hd, rl.nkv_l * hd
            q = qkv[:, :nqw].reshape(T, rl.nq_l, hd).transpose(0, 1)
            k = qkv[:, nqw:nqw + nkw].reshape(T, rl.nkv_l, hd).transpose(0, 1)
            v = qkv[:, nqw + nkw:].reshape(T, rl.nkv_l, hd).transpose(0, 1)
            q = of.apply_rope(of.rms_norm(q, rl.q_norm, eps), pos, SHAPE.rope_theta)
            k = of.apply_rope(of.rms_norm(k, rl.k_norm, eps), pos, SHAPE.rope_theta)
            o = of.causal_gqa_attention(q, torch.cat([kc, k], 1), torch.cat([vc, v], 1))
            x = x + reduce_scatter(o.transpose(0, 1).reshape(T, nqw) @ rl.o.T)
            h2 = all_gather_rows(of.rms_norm(x, rl.post_norm, eps))
            gu = h2 @ rl.gate_up.T
            x = x + reduce_scatter((of.silu(gu[:, :rl.i_l]) * gu[:, rl.i_l:]) @ rl.down.T)
        final = all_gather_rows(x)
        if rank == 0:
            out_q.put(final)
    finally:
        dist.destroy_process_group()


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("T", [7, 1])
def test_two_gloo_ranks_match_the_sp_emulation(T):
    """T = 7: chunks of 4 and 3 tokens; T = 1: rank 1 holds no token."""
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_sp, args=(r, 2, port, T, out_q)) for r in range(2)]
    for p in procs:
        p.start()
    got = out_q.get(timeout=90)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    layers, hw = _weights()
    emu = of.run_sequence_sp(_seq(T, 4), layers, hw, SHAPE, 2, head=False)
    assert _close(got, torch.cat(emu.hidden_chunks))
