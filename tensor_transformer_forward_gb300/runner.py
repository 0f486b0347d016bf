"""A whole step through the C ABI: vocab-parallel embedding (or given hidden
states), the decoder layers, and the vocab-parallel LM head with argmax.

The runner owns (as torch device buffers) every rank's weight shards, one KV
cache per layer, the workspace and the device status word; each method is one
or a few C-ABI calls on the current stream.
"""

from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import torch

from .binding import (WEIGHTS_HEAD, WEIGHTS_LAYER, Batch, Context, ModelConfig, TP_OK, TPError,
                      tp_decode_advance, tp_decoder_layer_forward, tp_embed_vocab_parallel, tp_lm_head_argmax,
                      tp_read_status, tp_shard_weights)


class TPRunner:
    """page_size == 0: one contiguous cache slot of ``capacity`` positions per
    sequence.  page_size > 0 (a multiple of 128): a paged cache of
    max_seqs * ceil(capacity / page_size) pages (+ ``spare_pages``), each sequence
    slot owning the pages of one row of a page table drawn as a seeded random
    permutation, so that no sequence's pages are contiguous or in order."""

    def __init__(self, cfg: ModelConfig, num_layers: int, max_seqs: int, capacity: int, max_tokens: int,
                 page_size: int = 0, spare_pages: int = 0, page_seed: int = 0):
        self.cfg = cfg
        self.ctx = Context(cfg)
        self.num_layers = num_layers
        self.max_seqs = max_seqs
        self.capacity = capacity
        self.max_tokens = max_tokens
        self.page_size = page_size
        self.layer_shards: List[Optional[torch.Tensor]] = [None] * num_layers
        self.head_shards: Optional[torch.Tensor] = None
        if page_size > 0:
            self.pages_per_seq = -(-capacity // page_size)
            self.num_pages = max_seqs * self.pages_per_seq + spare_pages
            g = torch.Generator().manual_seed(page_seed)
            perm = torch.randperm(self.num_pages, generator=g)[: max_seqs * self.pages_per_seq]
            self.page_table = perm.view(max_seqs, self.pages_per_seq).to(torch.int32)  # host copy
            self.kv_blocks, self.kv_block_len = self.num_pages, page_size
        else:
            self.page_table = None
            self.kv_blocks, self.kv_block_len = max_seqs, capacity
        self.kv: List[torch.Tensor] = [self.ctx.alloc_kv_cache(self.kv_blocks, self.kv_block_len)
                                       for _ in range(num_layers)]
        self.workspace = self.ctx.init_workspace(max_tokens, max(max_seqs, 1), capacity)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        n = cfg.tp_size
        self.nkv_l = cfg.num_kv_heads // n if cfg.num_kv_heads >= n else 1

    # ---- weights ----
    def load_layer(self, layer: int, full: Dict[str, torch.Tensor]) -> None:
        dst = self.ctx.alloc_layer_shards()
        tp_shard_weights(self.ctx, dst, layer=full, status=self.status)
        self.layer_shards[layer] = dst

    def load_head(self, full: Dict[str, torch.Tensor]) -> None:
        dst = self.ctx.alloc_head_shards()
        tp_shard_weights(self.ctx, dst, head=full, status=self.status)
        self.head_shards = dst

    def kv_head_map(self) -> List[int]:
        """Global kv head stored at each (rank, local head) of the caches."""
        hd = self.cfg.head_dim
        out = []
        for r in range(self.cfg.tp_size):
            _, rows = self.ctx.shard_index_map("k", r)
            out.extend(rows[j * hd] // hd for j in range(len(rows) // hd))
        return out

    def kv_view(self, layer: int) -> torch.Tensor:
        """[n, 2, blocks, nkv_l, block_len, hd] bf16 view of a layer cache (blocks =
        slots of `capacity` positions, or pages of `page_size`)."""
        c = self.cfg
        return self.kv[layer].view(torch.bfloat16).view(c.tp_size, 2, self.kv_blocks, self.nkv_l,
                                                        self.kv_block_len, c.head_dim)

    def kv_positions(self, layer: int, slot: int, p0: int, p1: int) -> torch.Tensor:
        """Positions [p0, p1) of sequence slot `slot`: [n, 2, nkv_l, p1 - p0, hd] (either layout)."""
        v = self.kv_view(layer)
        if self.page_table is None:
            return v[:, :, slot, :, p0:p1]
        ps = self.page_size
        parts = []
        p = p0
        while p < p1:
            e = min(p1, (p // ps + 1) * ps)
            parts.append(v[:, :, int(self.page_table[slot, p // ps]), :, p % ps:p % ps + (e - p)])
            p = e
        return torch.cat(parts, dim=3)

    def load_kv_contiguous(self, layer: int, contig: torch.Tensor) -> None:
        """Copies a cache given in the contiguous layout [n][2][max_seqs][nkv_l][capacity][hd]
        (bf16 elements) into this runner's layout (setup, not a step)."""
        c = self.cfg
        src = contig.view(torch.bfloat16).view(c.tp_size, 2, self.max_seqs, self.nkv_l, self.capacity, c.head_dim)
        if self.page_table is None:
            self.kv_view(layer).copy_(src)
            return
        ps, P = self.page_size, self.pages_per_seq
        pad = P * ps - self.capacity
        if pad:
            src = torch.nn.functional.pad(src, (0, 0, 0, pad))
        blocks = src.reshape(c.tp_size, 2, self.max_seqs, self.nkv_l, P, ps, c.head_dim).permute(0, 1, 2, 4, 3, 5, 6)
        blocks = blocks.reshape(c.tp_size, 2, self.max_seqs * P, self.nkv_l, ps, c.head_dim)
        dst = self.kv_view(layer)
        dst[:, :, self.page_table.flatten().long().to(dst.device)] = blocks

    # ---- one step ----
    def make_batch(self, q_lens: Sequence[int], ctx_lens: Sequence[int], slots: Optional[Sequence[int]] = None,
                   num_prefill: Optional[int] = None, max_kv_len: Optional[int] = None) -> Batch:
        if slots is None:
            slots = list(range(len(q_lens)))
        if num_prefill is None:
            num_prefill = sum(1 for q in q_lens if q > 1)
        if self.page_table is not None:  # each sequence takes its slot's row of the page table
            rows = self.page_table[torch.as_tensor(list(slots), dtype=torch.long)]
            return Batch(q_lens, ctx_lens, slots, num_prefill, max_kv_len=max_kv_len, page_table=rows,
                         page_size=self.page_size)
        return Batch(q_lens, ctx_lens, slots, num_prefill, max_kv_len=max_kv_len)

    def embed(self, ids: torch.Tensor, hidden_out: torch.Tensor) -> None:
        tp_embed_vocab_parallel(self.ctx, self.head_shards, ids, hidden_out, self.status)

    def layer(self, layer: int, batch: Batch, hidden: torch.Tensor) -> None:
        tp_decoder_layer_forward(self.ctx, self.layer_shards[layer], batch, hidden, self.kv[layer], self.kv_blocks,
                                 self.kv_block_len, self.status)

    def head(self, batch: Batch, hidden: torch.Tensor, out_ids: torch.Tensor,
             out_logits: Optional[torch.Tensor] = None) -> None:
        tp_lm_head_argmax(self.ctx, self.head_shards, batch, hidden, out_ids, self.status, out_logits)

    def step(self, batch: Batch, ids: Optional[torch.Tensor] = None, hidden: Optional[torch.Tensor] = None,
             out_ids: Optional[torch.Tensor] = None, out_logits: Optional[torch.Tensor] = None,
             layers: Optional[int] = None, run_head: bool = True) -> torch.Tensor:
        """Embedding (when ids are given) -> layers -> head; returns the fp32 residual stream [T, H]."""
        if hidden is None:
            hidden = torch.empty(batch.num_tokens, self.cfg.hidden, dtype=torch.float32, device="cuda")
            self.embed(ids, hidden)
        elif ids is not None:
            self.embed(ids, hidden)
        else:
            self.ctx.hidden_written()  # rows from the caller: the first layer derives its norm inputs
        for li in range(self.num_layers if layers is None else layers):
            self.layer(li, batch, hidden)
        if run_head:
            self.head(batch, hidden, out_ids, out_logits)
        return hidden

    # ---- greedy generation ----
    def generate(self, prompts: Sequence[Sequence[int]], steps: int, graph: bool = True,
                 slots: Optional[Sequence[int]] = None) -> Tuple[List[List[int]], torch.Tensor]:
        """Greedy generation as the pages' tp.py main does it: one prefill forward
        over the prompts, then ``steps`` one-token forwards, each fed the argmax of
        the previous one; returns the ``steps`` chosen ids per sequence and the fp32
        logits [B, V] of the last forward.  The decode forward (embedding, layers,
        head, then tp_decode_advance) is captured once in a CUDA graph and replayed
        (graph=False launches it eagerly every step; both give the same ids)."""
        B = len(prompts)
        lens = [len(p) for p in prompts]
        if B == 0 or min(lens) < 1 or steps < 1:
            raise ValueError("generate needs at least one non-empty prompt and one step")
        if max(lens) + steps > self.capacity:
            raise ValueError("prompt + steps exceed the KV cache capacity")
        slots = list(range(B)) if slots is None else list(slots)
        H, V = self.cfg.hidden, self.cfg.vocab
        dev = "cuda"
        cur = torch.empty(B, dtype=torch.int32, device=dev)  # argmax ids out, next embedding input in
        history = torch.full((steps + 1, B), -1, dtype=torch.int32, device=dev)
        logits = torch.empty(B, V, dtype=torch.float32, device=dev)
        step_ctr = torch.ones(1, dtype=torch.int32, device=dev)  # row 0 holds the prefill's ids
        # prefill forward
        ids = torch.tensor([t for p in prompts for t in p], dtype=torch.int32, device=dev)
        pb = self.make_batch(lens, [0] * B, slots, num_prefill=B)
        hidden_p = torch.empty(sum(lens), H, dtype=torch.float32, device=dev)
        self.step(pb, ids=ids, hidden=hidden_p, out_ids=cur)
        history[0].copy_(cur)
        # decode forwards: positions lens[b], lens[b] + 1, ...; launches planned for the last
        db = self.make_batch([1] * B, lens, slots, num_prefill=0, max_kv_len=max(lens) + steps)
        hidden_d = torch.empty(B, H, dtype=torch.float32, device=dev)

        def decode() -> None:
            self.step(db, ids=cur, hidden=hidden_d, out_ids=cur, out_logits=logits)
            tp_decode_advance(self.ctx, db, cur, history, step_ctr, self.status)

        decode()  # eager: also makes every kernel variant ready before a capture
        if graph and steps > 1:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                decode()
            for _ in range(steps - 1):
                g.replay()
        else:
            for _ in range(steps - 1):
                decode()
        torch.cuda.synchronize()
        self.check_status()
        got = history[:steps].t().cpu().tolist()
        return got, logits

    def check_status(self) -> None:
        st = tp_read_status(self.status)
        if st != TP_OK:
            raise TPError(st, "device status")
