"""GB300-native tensor-parallel forward of a Qwen3-style decoder layer and its
vocab-parallel embedding / LM head (tp_size > 1 emulated as rank shards on
one GPU).  The compute runs in the C-ABI library ``_lib/libtpfwd.so``
(``include/tpfwd.h``); this package is its thin ctypes binding."""

from .binding import (  # noqa: F401
    PARAM, PART, TP_ERR_BAD_TOKEN, TP_ERR_CUDA, TP_ERR_HEADS_NOT_DIVISIBLE, TP_ERR_INTERMEDIATE, TP_ERR_INVALID_ARG,
    TP_ERR_KV_HEADS, TP_ERR_SATURATED, TP_ERR_TIMEOUT, TP_ERR_UNSUPPORTED, TP_ERR_VOCAB, TP_OK, WEIGHTS_HEAD, WEIGHTS_LAYER, Batch,
    Context, ModelConfig, TPError, tp_debug_wait_probe, tp_decoder_layer_forward, tp_embed_vocab_parallel,
    tp_lm_head_argmax, tp_read_status, tp_shard_weights)
from .binding import lib  # noqa: F401
