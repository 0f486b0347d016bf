"""ctypes binding of the C ABI in ``include/tpfwd.h``.

Argument marshalling only: torch tensors become raw device pointers, the
current torch stream becomes the ``cudaStream_t``; every step of the forward
runs in the library's CUDA kernels.  There is no fallback: if the library is
missing this module raises on import.
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Dict, List, Optional, Sequence

import torch

from . import _build

TP_OK = 0
TP_ERR_INVALID_ARG = 1
TP_ERR_HEADS_NOT_DIVISIBLE = 2
TP_ERR_KV_HEADS = 3
TP_ERR_INTERMEDIATE = 4
TP_ERR_VOCAB = 5
TP_ERR_UNSUPPORTED = 6
TP_ERR_CUDA = 7
TP_ERR_BAD_TOKEN = 8
TP_ERR_TIMEOUT = 9
TP_ERR_SATURATED = 10

PARAM = dict(q=0, k=1, v=2, o=3, gate=4, up=5, down=6, embed=7, lm_head=8, norm=9)
PART = dict(qkv=0, o=1, gate_up=2, down=3, in_norm=4, post_norm=5, q_norm=6, k_norm=7,
            embed=8, lm_head=9, final_norm=10)
WEIGHTS_LAYER, WEIGHTS_HEAD = 0, 1
WS_PART = dict(normed=0, qkv=1, attn=2, act=3)


class TPError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {_lib.tp_status_string(status).decode()} (status {status})"
        if status == TP_ERR_CUDA:
            msg += f" [{_lib.tp_last_cuda_error().decode()}]"
        super().__init__(msg)


class TPConfig(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("num_q_heads", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("num_layers", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
                ("tp_size", ctypes.c_int32), ("tie_word_embeddings", ctypes.c_int32)]


class TPBatch(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("num_prefill", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("max_q_len", ctypes.c_int32), ("max_kv_len", ctypes.c_int32),
                ("cu_q", ctypes.c_void_p), ("ctx_len", ctypes.c_void_p), ("slot", ctypes.c_void_p),
                ("page_table", ctypes.c_void_p), ("page_size", ctypes.c_int32), ("max_pages_per_seq", ctypes.c_int32)]


class TPLayerFull(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in ("q", "k", "v", "o", "gate", "up", "down",
                                                 "in_norm", "post_norm", "q_norm", "k_norm")]


class TPHeadFull(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in ("embed", "lm_head", "final_norm")]


def _load() -> ctypes.CDLL:
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    P, I32, I64, SZ, F32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
    pSZ, pI64, pI32 = ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_int32)
    sig = {
        "tp_create": ([ctypes.POINTER(TPConfig), ctypes.POINTER(P)], I32),
        "tp_destroy": ([P], I32),
        "tp_status_string": ([I32], ctypes.c_char_p),
        "tp_last_cuda_error": ([], ctypes.c_char_p),
        "tp_shard_index_map": ([P, I32, I32, P, pI64, pI32], I32),
        "tp_weights_bytes": ([P, I32, pSZ], I32),
        "tp_weights_part": ([P, I32, pSZ, pSZ], I32),
        "tp_shard_weights": ([P, ctypes.POINTER(TPLayerFull), ctypes.POINTER(TPHeadFull), P, P, P], I32),
        "tp_kv_cache_bytes": ([P, I32, I32, pSZ], I32),
        "tp_workspace_bytes": ([P, I32, I32, I32, pSZ], I32),
        "tp_workspace_init": ([P, P, SZ, I32, I32, I32, P], I32),
        "tp_embed_vocab_parallel": ([P, P, P, I32, P, P, P], I32),
        "tp_decoder_layer_forward": ([P, P, ctypes.POINTER(TPBatch), P, P, I32, I32, P, P], I32),
        "tp_lm_head_argmax": ([P, P, ctypes.POINTER(TPBatch), P, P, P, P, P], I32),
        "tp_lm_head_argmax_static": ([P, P, ctypes.POINTER(TPBatch), P, P, P, P, P], I32),
        "tp_read_status": ([P, P], I32),
        "tp_rank_sum_count": ([P, pI64], I32),
        "tp_workspace_part": ([P, I32, pSZ, pSZ], I32),
        "tp_keep_intermediates": ([P, I32], I32),
        "tp_decode_advance": ([P, P, P, P, I32, P, P, P], I32),
        "tp_hidden_written": ([P], I32),
        "tp_launch_count": ([P, pI64], I32),
        "tp_profile_begin": ([P, ctypes.c_uint32, I32], I32),
        "tp_profile_end": ([P, ctypes.POINTER(F32), pI32], I32),
        "tp_debug_wait_probe": ([P, P, I64, P], I32),
        "tp_debug_decode_plan": ([I32, I32, I32, I32, I32, I32, pI32, pI32], I32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()
EXPORTED = ("tp_create", "tp_destroy", "tp_status_string", "tp_last_cuda_error", "tp_shard_index_map",
            "tp_weights_bytes", "tp_weights_part", "tp_shard_weights", "tp_kv_cache_bytes", "tp_workspace_bytes",
            "tp_workspace_init", "tp_embed_vocab_parallel", "tp_decoder_layer_forward", "tp_lm_head_argmax",
            "tp_read_status", "tp_rank_sum_count", "tp_debug_wait_probe", "tp_workspace_part", "tp_launch_count",
            "tp_profile_begin", "tp_profile_end", "tp_lm_head_argmax_static", "tp_keep_intermediates",
            "tp_decode_advance", "tp_hidden_written", "tp_debug_decode_plan")
KERNELS = ("embed", "rmsnorm", "gemm_qkv", "rope", "attn_prefill", "attn_decode", "gemm_o", "gemm_gate_up",
           "gemm_down", "final_norm", "gemm_lm_head", "argmax", "decode_advance")


def lib() -> ctypes.CDLL:
    return _lib


def _check(st: int, what: str) -> None:
    if st != TP_OK:
        raise TPError(st, what)


def _stream(stream: Optional[torch.cuda.Stream] = None) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype: Optional[torch.dtype] = None) -> ctypes.c_void_p:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _dev_or_pinned(t: torch.Tensor, name: str, dtype: Optional[torch.dtype] = None) -> ctypes.c_void_p:
    """A CUDA tensor, or a page-locked CPU tensor that the kernel reads or writes over
    the host link itself."""
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or a page-locked (pinned) CPU tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if dtype is not None and t.dtype != dtype:
            raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
        return ctypes.c_void_p(t.data_ptr())
    return _dev(t, name, dtype)


@dataclasses.dataclass(frozen=True)
class ModelConfig:
    hidden: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    num_layers: int
    rms_eps: float
    rope_theta: float
    tp_size: int
    tie_word_embeddings: bool

    def c(self) -> TPConfig:
        return TPConfig(self.hidden, self.num_q_heads, self.num_kv_heads, self.head_dim, self.intermediate,
                        self.vocab, self.num_layers, self.rms_eps, self.rope_theta, self.tp_size,
                        int(self.tie_word_embeddings))


class Context:
    """Owns one ``tp_ctx`` (host-side plan); device buffers belong to the caller."""

    def __init__(self, cfg: ModelConfig):
        self.cfg = cfg
        self._c = cfg.c()
        h = ctypes.c_void_p()
        _check(_lib.tp_create(ctypes.byref(self._c), ctypes.byref(h)), "tp_create")
        self.handle = h
        self.workspace: Optional[torch.Tensor] = None

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            _lib.tp_destroy(h)
            self.handle = None

    # ---- host-only queries ----
    def shard_index_map(self, kind: str, rank: int):
        n, d = ctypes.c_int64(), ctypes.c_int32()
        _check(_lib.tp_shard_index_map(self.handle, PARAM[kind], rank, None, ctypes.byref(n), ctypes.byref(d)),
               "tp_shard_index_map")
        buf = (ctypes.c_int64 * max(1, n.value))()
        _check(_lib.tp_shard_index_map(self.handle, PARAM[kind], rank, buf, ctypes.byref(n), ctypes.byref(d)),
               "tp_shard_index_map")
        return {0: "rows", 1: "cols", -1: "all"}[d.value], list(buf)[: n.value]

    def weights_bytes(self, which: int) -> int:
        b = ctypes.c_size_t()
        _check(_lib.tp_weights_bytes(self.handle, which, ctypes.byref(b)), "tp_weights_bytes")
        return b.value

    def weights_part(self, part: str):
        o, b = ctypes.c_size_t(), ctypes.c_size_t()
        _check(_lib.tp_weights_part(self.handle, PART[part], ctypes.byref(o), ctypes.byref(b)), "tp_weights_part")
        return o.value, b.value

    def kv_cache_bytes(self, max_seqs: int, capacity: int) -> int:
        b = ctypes.c_size_t()
        _check(_lib.tp_kv_cache_bytes(self.handle, max_seqs, capacity, ctypes.byref(b)), "tp_kv_cache_bytes")
        return b.value

    def workspace_bytes(self, max_tokens: int, max_seqs: int, max_positions: int) -> int:
        b = ctypes.c_size_t()
        _check(_lib.tp_workspace_bytes(self.handle, max_tokens, max_seqs, max_positions, ctypes.byref(b)),
               "tp_workspace_bytes")
        return b.value

    def launch_count(self) -> int:
        c = ctypes.c_int64()
        _check(_lib.tp_launch_count(self.handle, ctypes.byref(c)), "tp_launch_count")
        return c.value

    def profile_begin(self, kinds: Sequence[str], max_launches: int = 65536) -> None:
        mask = 0
        for k in kinds:
            mask |= 1 << KERNELS.index(k)
        _check(_lib.tp_profile_begin(self.handle, mask, max_launches), "tp_profile_begin")

    def profile_end(self) -> Dict[str, tuple]:
        """{kernel: (total device ms, timed launches)} since profile_begin."""
        ms = (ctypes.c_float * len(KERNELS))()
        cnt = (ctypes.c_int32 * len(KERNELS))()
        _check(_lib.tp_profile_end(self.handle, ms, cnt), "tp_profile_end")
        return {k: (ms[i], cnt[i]) for i, k in enumerate(KERNELS) if cnt[i] > 0}

    def rank_sum_count(self) -> int:
        c = ctypes.c_int64()
        _check(_lib.tp_rank_sum_count(self.handle, ctypes.byref(c)), "tp_rank_sum_count")
        return c.value

    # ---- device buffers owned by torch ----
    def alloc_layer_shards(self) -> torch.Tensor:
        return torch.empty(self.weights_bytes(WEIGHTS_LAYER), dtype=torch.uint8, device="cuda")

    def alloc_head_shards(self) -> torch.Tensor:
        return torch.empty(self.weights_bytes(WEIGHTS_HEAD), dtype=torch.uint8, device="cuda")

    def alloc_kv_cache(self, max_seqs: int, capacity: int) -> torch.Tensor:
        # zeroed: attention tiles read whole 128-key blocks, so the unused tail of a
        # slot must hold finite values (masked scores are 0, and 0 * NaN is NaN)
        return torch.zeros(self.kv_cache_bytes(max_seqs, capacity), dtype=torch.uint8, device="cuda")

    def init_workspace(self, max_tokens: int, max_seqs: int, max_positions: int) -> torch.Tensor:
        nbytes = self.workspace_bytes(max_tokens, max_seqs, max_positions)
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        _check(_lib.tp_workspace_init(self.handle, _dev(ws, "workspace"), nbytes, max_tokens, max_seqs,
                                      max_positions, _stream()), "tp_workspace_init")
        self.workspace = ws
        return ws

    def hidden_written(self) -> None:
        """The caller wrote the residual stream itself: the next layer call recomputes
        the deferred norm's inputs (see tp_hidden_written)."""
        _check(_lib.tp_hidden_written(self.handle), "tp_hidden_written")

    def keep_intermediates(self, keep: bool = True) -> None:
        """Leave the layer's intermediates readable after each call (debugging)."""
        _check(_lib.tp_keep_intermediates(self.handle, 1 if keep else 0), "tp_keep_intermediates")

    def workspace_view(self, part: str, rows: int, cols: int, dtype=torch.float16) -> torch.Tensor:
        """[rows, cols] view of an intermediate of the last layer call (fp16; the q
        heads of the QKV buffer hold bf16); needs keep_intermediates()."""
        o, b = ctypes.c_size_t(), ctypes.c_size_t()
        _check(_lib.tp_workspace_part(self.handle, WS_PART[part], ctypes.byref(o), ctypes.byref(b)),
               "tp_workspace_part")
        assert rows * cols * 2 <= b.value
        return self.workspace[o.value:o.value + rows * cols * 2].view(dtype).view(rows, cols)

    def part_view(self, shards: torch.Tensor, part: str, shape: Sequence[int], dtype=torch.bfloat16) -> torch.Tensor:
        off, nbytes = self.weights_part(part)
        numel = 1
        for s in shape:
            numel *= s
        esz = torch.tensor([], dtype=dtype).element_size()
        assert numel * esz <= nbytes
        return shards[off:off + numel * esz].view(dtype).view(*shape)


class Batch:
    """Device arrays of one step plus the host summary the launches need.

    A contiguous cache takes ``slots`` (the cache slot of each sequence).  A paged
    cache takes ``page_table`` ([num_seqs][max_pages_per_seq] page ids, a list of
    lists or an int32 tensor) and ``page_size`` (a multiple of 128); ``slots`` is
    then unused (it may be None)."""

    def __init__(self, q_lens: Sequence[int], ctx_lens: Sequence[int], slots: Optional[Sequence[int]],
                 num_prefill: int, max_kv_len: Optional[int] = None, page_table=None, page_size: int = 0):
        cu = [0]
        for q in q_lens:
            cu.append(cu[-1] + int(q))
        self.q_lens, self.ctx_lens = list(q_lens), list(ctx_lens)
        self.slots = None if slots is None else list(slots)
        self.num_prefill = num_prefill
        self.cu_q = torch.tensor(cu, dtype=torch.int32, device="cuda")
        self.ctx_len = torch.tensor(list(ctx_lens), dtype=torch.int32, device="cuda")
        self.slot = None if slots is None else torch.tensor(list(slots), dtype=torch.int32, device="cuda")
        self.page_table = None
        pages = 0
        if page_table is not None:
            pt = page_table if isinstance(page_table, torch.Tensor) else torch.tensor(page_table, dtype=torch.int32)
            if pt.dim() != 2 or pt.shape[0] != len(q_lens) or page_size <= 0:
                raise ValueError("page_table must be [num_seqs][max_pages_per_seq] with a page_size > 0")
            self.page_table = pt.to(device="cuda", dtype=torch.int32).contiguous()
            pages = int(pt.shape[1])
        elif slots is None:
            raise ValueError("a batch needs slots (contiguous cache) or a page_table (paged cache)")
        self.page_size = int(page_size) if page_table is not None else 0
        pre = list(q_lens[:num_prefill])
        # max_kv_len plans the launches; a batch whose device ctx_len grows between
        # forwards (greedy decoding, one graph for every step) plans for its last one
        kv = max(int(c) + int(q) for c, q in zip(ctx_lens, q_lens))
        if max_kv_len is not None:
            if max_kv_len < kv:
                raise ValueError("max_kv_len below the batch's current kv length")
            kv = int(max_kv_len)
        self.c = TPBatch(len(q_lens), num_prefill, cu[-1], max(pre) if pre else 0, kv,
                         self.cu_q.data_ptr(), self.ctx_len.data_ptr(),
                         self.slot.data_ptr() if self.slot is not None else None,
                         self.page_table.data_ptr() if self.page_table is not None else None,
                         self.page_size, pages)

    @property
    def num_tokens(self) -> int:
        return self.c.num_tokens

    @property
    def num_seqs(self) -> int:
        return self.c.num_seqs


# ---------------------------------------------------------------------------
# The entry points, by the C names
# ---------------------------------------------------------------------------

def tp_shard_weights(ctx: Context, dst: torch.Tensor, layer: Optional[Dict[str, torch.Tensor]] = None,
                     head: Optional[Dict[str, torch.Tensor]] = None, status: Optional[torch.Tensor] = None) -> None:
    """A1: shard then merge full bf16 tensors (dict by name) into ``dst``; ``status``
    (device int32, optional) receives the saturation flag when a weight is outside
    the fp16 range of the tensor-core copies."""
    lp = hp = None
    keep: List[torch.Tensor] = []
    if layer is not None:
        f = TPLayerFull()
        for k, _ in TPLayerFull._fields_:
            t = layer[k]
            keep.append(t)
            setattr(f, k, _dev(t, k, torch.bfloat16).value)
        lp = ctypes.byref(f)
    if head is not None:
        f2 = TPHeadFull()
        for k, _ in TPHeadFull._fields_:
            t = head.get(k)
            if t is None:
                continue
            keep.append(t)
            setattr(f2, k, _dev(t, k, torch.bfloat16).value)
        hp = ctypes.byref(f2)
    st = _dev(status, "status", torch.int32) if status is not None else None
    _check(_lib.tp_shard_weights(ctx.handle, lp, hp, _dev(dst, "dst"), st, _stream()), "tp_shard_weights")


def tp_embed_vocab_parallel(ctx: Context, head_shards: torch.Tensor, ids: torch.Tensor, hidden_out: torch.Tensor,
                            status: torch.Tensor) -> None:
    _check(_lib.tp_embed_vocab_parallel(ctx.handle, _dev(head_shards, "head_shards"),
                                        _dev_or_pinned(ids, "ids", torch.int32), ids.numel(),
                                        _dev(hidden_out, "hidden_out", torch.float32),
                                        _dev(status, "status", torch.int32), _stream()), "tp_embed_vocab_parallel")


def tp_decoder_layer_forward(ctx: Context, layer_shards: torch.Tensor, batch: Batch, hidden: torch.Tensor,
                             kv_cache: torch.Tensor, kv_max_seqs: int, kv_capacity: int,
                             status: torch.Tensor) -> None:
    _check(_lib.tp_decoder_layer_forward(ctx.handle, _dev(layer_shards, "layer_shards"), ctypes.byref(batch.c),
                                         _dev(hidden, "hidden", torch.float32), _dev(kv_cache, "kv_cache"),
                                         kv_max_seqs, kv_capacity, _dev(status, "status", torch.int32), _stream()),
           "tp_decoder_layer_forward")


def tp_lm_head_argmax(ctx: Context, head_shards: torch.Tensor, batch: Batch, hidden: torch.Tensor,
                      out_ids: torch.Tensor, status: torch.Tensor, out_logits: Optional[torch.Tensor] = None) -> None:
    lg = _dev_or_pinned(out_logits, "out_logits", torch.float32) if out_logits is not None else None
    _check(_lib.tp_lm_head_argmax(ctx.handle, _dev(head_shards, "head_shards"), ctypes.byref(batch.c),
                                  _dev(hidden, "hidden", torch.float32),
                                  _dev_or_pinned(out_ids, "out_ids", torch.int32), lg,
                                  _dev(status, "status", torch.int32), _stream()), "tp_lm_head_argmax")


def tp_lm_head_argmax_static(ctx: Context, head_shards: torch.Tensor, batch: Batch, hidden: torch.Tensor,
                             out_ids: torch.Tensor, status: torch.Tensor,
                             out_logits: Optional[torch.Tensor] = None) -> None:
    """tp_lm_head_argmax without a workspace: for callers that cannot allocate
    device memory; its scratch is a fixed array inside the library (see tpfwd.h)."""
    lg = _dev_or_pinned(out_logits, "out_logits", torch.float32) if out_logits is not None else None
    _check(_lib.tp_lm_head_argmax_static(ctx.handle, _dev(head_shards, "head_shards"), ctypes.byref(batch.c),
                                         _dev(hidden, "hidden", torch.float32),
                                         _dev_or_pinned(out_ids, "out_ids", torch.int32),
                                         lg, _dev(status, "status", torch.int32), _stream()),
           "tp_lm_head_argmax_static")


def tp_decode_advance(ctx: Context, batch: Batch, ids: torch.Tensor, history: torch.Tensor, step: torch.Tensor,
                      status: torch.Tensor) -> None:
    """Greedy decoding bookkeeping after a decode forward: ctx_len += 1 on the
    device, the forward's ids to row ``step`` of ``history`` [rows, B], step += 1."""
    _check(_lib.tp_decode_advance(ctx.handle, ctypes.byref(batch.c), _dev(ids, "ids", torch.int32),
                                  _dev(history, "history", torch.int32), int(history.shape[0]),
                                  _dev(step, "step", torch.int32), _dev(status, "status", torch.int32), _stream()),
           "tp_decode_advance")


def tp_read_status(status: torch.Tensor) -> int:
    """Synchronises the current stream and returns the device status (TP_OK,
    TP_ERR_BAD_TOKEN, TP_ERR_TIMEOUT or TP_ERR_SATURATED)."""
    return _lib.tp_read_status(_dev(status, "status", torch.int32), _stream())


def tp_debug_wait_probe(flag: torch.Tensor, status: torch.Tensor, limit_ns: int) -> None:
    _check(_lib.tp_debug_wait_probe(_dev(flag, "flag", torch.int32), _dev(status, "status", torch.int32),
                                    int(limit_ns), _stream()), "tp_debug_wait_probe")


def tp_debug_decode_plan(max_kv_len: int, num_units: int, num_sms: int, head_dim: int, group: int,
                         max_splits: int):
    """The decode attention's split plan (host only): ([units per level], [splits per level])."""
    units = (ctypes.c_int32 * 4)()
    splits = (ctypes.c_int32 * 4)()
    _check(_lib.tp_debug_decode_plan(int(max_kv_len), int(num_units), int(num_sms), int(head_dim), int(group),
                                     int(max_splits), units, splits), "tp_debug_decode_plan")
    return list(units), list(splits)
