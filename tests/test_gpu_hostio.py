"""Ids in and out through page-locked host memory: the embedding kernel reads the
step's ids and the LM head writes the chosen ids over the host link, with the same
results as device buffers; memory the GPU cannot address is refused before any
launch."""

import ctypes

import numpy as np
import pytest
import torch

import synth
from tensor_transformer_forward_gb300 import binding
from tests.gpu_harness import GpuStep

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wl", ["prefill", "decode"])
def test_pinned_host_ids_match_device_ids(wl):
    if wl == "prefill":
        w = synth.Workload("hostio_pf", synth.QWEN3_06B, (2,), ((300, 0), (41, 7)), (), 1, True)
    else:
        w = synth.Workload("hostio_dec", synth.QWEN3_06B, (2,), (), (5, 130, 999), 1, True)
    g = GpuStep(w, 2, logits=False)
    r, batch = g.runner, g.batch
    dev_out = g.out_ids.clone()
    hidden_dev = g.hidden.clone()
    # the same step again with host buffers (the cache positions are rewritten with the same values)
    ids_host = g.ids.cpu().pin_memory()
    out_host = torch.full((w.num_seqs,), -1, dtype=torch.int32).pin_memory()
    hidden = torch.empty_like(g.hidden)
    r.step(batch, ids=ids_host, hidden=hidden, out_ids=out_host)
    torch.cuda.synchronize()
    r.check_status()
    assert torch.equal(out_host, dev_out.cpu())
    assert torch.equal(hidden, hidden_dev)


def test_pageable_host_memory_is_refused():
    w = synth.Workload("hostio_bad", synth.QWEN3_06B, (1,), (), (3,), 1, True)
    g = GpuStep(w, 1, logits=False)
    with pytest.raises(ValueError):
        binding.tp_embed_vocab_parallel(g.runner.ctx, g.runner.head_shards, torch.zeros(1, dtype=torch.int32),
                                        g.hidden, g.runner.status)
    # straight through the C ABI: a pageable host address gives TP_ERR_INVALID_ARG, nothing launched
    arr = np.zeros(1, dtype=np.int32)
    n0 = g.runner.ctx.launch_count()
    rc = binding._lib.tp_embed_vocab_parallel(g.runner.ctx.handle, ctypes.c_void_p(g.runner.head_shards.data_ptr()),
                                              ctypes.c_void_p(arr.ctypes.data), 1, ctypes.c_void_p(g.hidden.data_ptr()),
                                              ctypes.c_void_p(g.runner.status.data_ptr()), None)
    assert rc == binding.TP_ERR_INVALID_ARG
    assert g.runner.ctx.launch_count() == n0
