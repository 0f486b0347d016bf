/*
 * tpfwd -- GB300 (sm_103a) tensor-parallel forward of a Qwen3-style decoder
 * layer and its vocab-parallel embedding / LM head, with every tp_size > 1
 * run emulated as rank shards on one GPU.
 *
 * Plain C ABI: opaque host context, device pointers and sizes, int32 status
 * codes.  No call throws.  All device buffers are allocated by the caller
 * (e.g. PyTorch); the library owns only the host-side tp_ctx.  Every device
 * call is asynchronous on the given CUDA stream (void* = cudaStream_t).
 *
 * Sources ("the pages"):
 *  [TP]  ai-infra-handbooks, "Tensor parallelism from scratch": sections
 *        "Two ways to split", "Implementation" (tp.py: ColumnParallelLinear,
 *        RowParallelLinear, VocabParallelEmbedding, TPAttention, TPMLP,
 *        TPTransformer), "KV heads and the limit on TP".
 *  [SHD] jaehun.me, "mini-sglang 08: How several ranks share one ledger",
 *        section "Weights are cut by name" (models/weight.py:13-14, 34-52;
 *        layers/linear.py:102-106).
 *  [CH9] zero-to-sglang, "Chapter 9 Multi-process and Tensor Parallelism",
 *        section 3.3 "Loading Weights and Model State" (shard then merge;
 *        VocabParallelEmbedding / ParallelLMHead).
 *
 * Notation: H hidden, nq / nkv query / kv heads, hd head_dim, I intermediate,
 * V vocab, n tp_size.  Per rank: nq_l = nq/n, nkv_l = max(1, nkv/n),
 * I_l = I/n, V_l = ceil(V/n).  Weights are nn.Linear layout [out, in], bf16.
 */
#ifndef TPFWD_H
#define TPFWD_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t tp_status;

/* Status codes (returned by every call; host errors are returned before any launch). */
#define TP_OK 0
#define TP_ERR_INVALID_ARG 1          /* null pointer, bad size, buffer too small, T > planned maximum */
#define TP_ERR_HEADS_NOT_DIVISIBLE 2  /* nq % n != 0 ([TP] "KV heads and the limit on TP") */
#define TP_ERR_KV_HEADS 3             /* nkv >= n with nkv % n != 0, or nkv < n with n % nkv != 0 */
#define TP_ERR_INTERMEDIATE 4         /* I % n != 0 */
#define TP_ERR_VOCAB 5                /* some rank's div_ceil vocab slice would be empty */
#define TP_ERR_UNSUPPORTED 6          /* shape outside the kernels' range (hd not 64/128, H % 64, ...) */
#define TP_ERR_CUDA 7                 /* a CUDA runtime call or launch failed */
#define TP_ERR_BAD_TOKEN 8            /* device: a token id outside [0, V) or a position outside the cache */
#define TP_ERR_TIMEOUT 9              /* device: a bounded wait inside a kernel gave up */
#define TP_ERR_SATURATED 10           /* device: a value converted to an fp16 operand (a weight, a residual
                                         row, an attention output, SiLU*up, a decode q) was outside the fp16
                                         range and was clamped to +-65504; the results are not trustworthy */

typedef struct {
  int32_t hidden, num_q_heads, num_kv_heads, head_dim, intermediate, vocab, num_layers;
  float rms_eps, rope_theta;
  int32_t tp_size;
  int32_t tie_word_embeddings; /* 1: the LM head is the embedding table ([TP] TPTransformer) */
} tp_config;

typedef struct tp_ctx tp_ctx; /* opaque host-side plan */

/* Create a context; validates the shard rules for cfg->tp_size ([TP] "KV heads
 * and the limit on TP"; [SHD] weight.py:34-52 with uneven splits read as
 * errors).  *out receives the context (NULL on error). */
tp_status tp_create(const tp_config* cfg, tp_ctx** out);
tp_status tp_destroy(tp_ctx* ctx);
const char* tp_status_string(tp_status s);

/* ---------------- shard rules (host only) ----------------
 * Parameter kinds for index maps. */
#define TP_PARAM_Q 0
#define TP_PARAM_K 1
#define TP_PARAM_V 2
#define TP_PARAM_O 3
#define TP_PARAM_GATE 4
#define TP_PARAM_UP 5
#define TP_PARAM_DOWN 6
#define TP_PARAM_EMBED 7
#define TP_PARAM_LM_HEAD 8
#define TP_PARAM_NORM 9

/* Source indices of rank `rank`'s shard of a full tensor ([SHD] weight.py:34-52):
 * q/gate/up take an even chunk of rows; k/v take an even chunk of rows, or the
 * rows of head rank*nkv/n when nkv < n (replication); o/down take an even chunk
 * of columns; embed/lm_head take rows [rank*V_l, min((rank+1)*V_l, V)); norms
 * are kept whole.  *dim = 0 rows, 1 columns, -1 whole tensor.  *len receives
 * the index count; src_idx (host, may be NULL) receives the indices. */
tp_status tp_shard_index_map(const tp_ctx* ctx, int32_t kind, int32_t rank, int64_t* src_idx, int64_t* len,
                             int32_t* dim);

/* ---------------- device weight layout ----------------
 * A layer's shards live in one caller-allocated buffer of tp_weights_bytes(TP_WEIGHTS_LAYER)
 * bytes; the embedding / LM head / final norm in one of tp_weights_bytes(TP_WEIGHTS_HEAD).
 * Parts (byte offsets from tp_weights_part, each 1024-byte aligned):
 *  TP_PART_QKV      [n][(nq_l + 2 nkv_l) hd][H]: per rank cat(q_r, k_r, v_r) rows ([CH9] 3.3 merge)
 *  TP_PART_O        [n][H][nq_l hd]           : per rank the o_proj column slice
 *  TP_PART_GATE_UP  [n][I_p/64][2][64][H]     : per rank gate_r and up_r rows interleaved in
 *                                              blocks of 64 (I_p = I_l rounded up to 64, zero rows)
 *  TP_PART_DOWN     [n][H][I_p]               : per rank the down_proj column slice (zero padded)
 *  TP_PART_IN_NORM, TP_PART_POST_NORM [H]; TP_PART_Q_NORM, TP_PART_K_NORM [hd] (one copy,
 *                                              identical on every rank)
 *  TP_PART_EMBED    [n][V_l][H]               : per rank its vocab rows, zero padded to V_l
 *  TP_PART_LM_HEAD  [n][V_l][H]               : same layout; the embedding's rows when tied
 *  TP_PART_FINAL_NORM [H]
 * The projection parts (QKV, O, GATE_UP, DOWN) and the LM head are tensor-core operands and
 * are stored fp16 (converted from the bf16 inputs: exact for magnitudes in [2^-14, 65504],
 * smaller ones rounded to fp16's subnormal grid, larger ones saturated); embedding rows and
 * norm weights stay bf16.  QKV and GATE_UP hold their columns multiplied by the RMSNorm
 * weight that precedes them (input norm, post-attention norm): W[r][c] * w[c], the exact
 * bf16 x bf16 product rounded once to fp16.  The norms themselves are deferred: the layer
 * scales each output row by rsqrt(mean(x^2) + eps) of its input row.
 */
#define TP_WEIGHTS_LAYER 0
#define TP_WEIGHTS_HEAD 1
#define TP_PART_QKV 0
#define TP_PART_O 1
#define TP_PART_GATE_UP 2
#define TP_PART_DOWN 3
#define TP_PART_IN_NORM 4
#define TP_PART_POST_NORM 5
#define TP_PART_Q_NORM 6
#define TP_PART_K_NORM 7
#define TP_PART_EMBED 8
#define TP_PART_LM_HEAD 9
#define TP_PART_FINAL_NORM 10

tp_status tp_weights_bytes(const tp_ctx* ctx, int32_t which, size_t* bytes);
tp_status tp_weights_part(const tp_ctx* ctx, int32_t part, size_t* offset, size_t* bytes);

/* Full (unsharded) tensors, device pointers, bf16, nn.Linear layout, contiguous. */
typedef struct {
  const void *q, *k, *v, *o, *gate, *up, *down;     /* [nq hd, H] [nkv hd, H] x2 [H, nq hd] [I, H] x2 [H, I] */
  const void *in_norm, *post_norm, *q_norm, *k_norm; /* [H] [H] [hd] [hd] */
} tp_layer_full;
typedef struct {
  const void *embed, *lm_head, *final_norm; /* [V, H], [V, H] (ignored when tied), [H] */
} tp_head_full;

/* A1: shard then merge ([SHD] weight.py:34-52; [CH9] 3.3).  Exactly one of layer / head is
 * non-NULL; dst (device, tp_weights_bytes of that kind) receives every rank's shards in the
 * layout above.  Reads src only; asynchronous on stream.  dev_status (device int32, sticky,
 * may be NULL) receives TP_ERR_SATURATED's flag when a weight (times its folded norm weight)
 * is outside the fp16 range of the tensor-core copies. */
tp_status tp_shard_weights(tp_ctx* ctx, const tp_layer_full* layer, const tp_head_full* head, void* dst,
                           int32_t* dev_status, void* stream);

/* ---------------- KV cache and workspace ----------------
 * KV cache of one layer: [n][2 (K, V)][blocks][nkv_l][block_len][hd] bf16; rank r keeps its
 * own kv heads (replicated heads stored once per holding rank, [TP] "KV heads ...").
 * Contiguous cache: a block is a sequence slot of `capacity` positions (blocks = max_seqs,
 * block_len = capacity), chosen per sequence by tp_batch.slot.
 * Paged cache (zero-to-sglang "Chapter 9", section 3.3: the engine sets up the KV cache and
 * its page table): a block is a page of page_size positions (blocks = the number of pages);
 * tp_batch.page_table maps (sequence, position / page_size) to a page, so a sequence's
 * pages need be neither contiguous nor in order, and sequences may share none.
 * tp_kv_cache_bytes(ctx, blocks, block_len) sizes either. */
tp_status tp_kv_cache_bytes(const tp_ctx* ctx, int32_t max_seqs, int32_t capacity, size_t* bytes);

/* Workspace for steps of at most max_tokens tokens and max_seqs sequences and positions
 * < max_positions (it also holds the RoPE cos/sin table).  One workspace per context:
 * tp_workspace_init records it, zeroes its counters and fills the RoPE table (fp64 on the
 * host, stored fp32); it is synchronous. */
tp_status tp_workspace_bytes(const tp_ctx* ctx, int32_t max_tokens, int32_t max_seqs, int32_t max_positions,
                             size_t* bytes);
tp_status tp_workspace_init(tp_ctx* ctx, void* ws, size_t ws_bytes, int32_t max_tokens, int32_t max_seqs,
                            int32_t max_positions, void* stream);

/* Intermediates of the last tp_decoder_layer_forward, inside the workspace (for tests and
 * debugging; valid until the next call, and only while tp_keep_intermediates(ctx, 1) is set:
 * by default the calls drop each intermediate from L2 without writing it back once its last
 * reader has run, so that dead data costs no HBM write traffic): byte offset and size of
 *  TP_WS_NORMED  fp16 [T, H]                  the layer's output rows (the residual stream in fp16),
 *                                              which the next layer's deferred input norm reads (the
 *                                              norms are deferred into the next projection's epilogue,
 *                                              which scales row t by rsqrt(mean(x_t^2) + eps))
 *  TP_WS_QKV     [T, n, (nq_l+2nkv_l) hd]     merged projection; its q heads hold post-RoPE q
 *                                              as bf16 (k and v go straight to the cache)
 *  TP_WS_ATTN    fp16 [T, n * nq_l * hd]      attention output (o_proj input)
 *  TP_WS_ACT     fp16 [T, n * I_p]            SiLU(gate) * up (down_proj input) */
#define TP_WS_NORMED 0
#define TP_WS_QKV 1
#define TP_WS_ATTN 2
#define TP_WS_ACT 3
tp_status tp_workspace_part(const tp_ctx* ctx, int32_t part, size_t* offset, size_t* bytes);
/* The deferred RMSNorms read an fp16 copy of the residual rows and their 32-column sums of
 * squares, which tp_embed_vocab_parallel and each tp_decoder_layer_forward leave in the
 * workspace for the hidden buffer they wrote; the next layer call on the same buffer and
 * token count reuses them, any other buffer gets them recomputed.  A caller that writes
 * hidden itself between two such calls tells the context with this (the pages have no
 * counterpart: the norms there are separate passes). */
tp_status tp_hidden_written(tp_ctx* ctx);

/* keep != 0: leave the intermediates above readable after each call (no L2 discards).
 * The pages have no counterpart; this is a debugging switch. */
tp_status tp_keep_intermediates(tp_ctx* ctx, int32_t keep);

/* A step's batch.  Sequences [0, num_prefill) may have several new tokens; sequences
 * [num_prefill, num_seqs) have exactly one.  Tokens are packed per sequence in order. */
typedef struct {
  int32_t num_seqs;
  int32_t num_prefill;
  int32_t num_tokens;  /* T = cu_q[num_seqs] */
  int32_t max_q_len;   /* max new tokens over the prefill sequences */
  int32_t max_kv_len;  /* max over sequences of ctx_len + q_len */
  const int32_t* cu_q;    /* device [num_seqs + 1]: first packed token of each sequence */
  const int32_t* ctx_len; /* device [num_seqs]: cached tokens = position of the first new token */
  const int32_t* slot;    /* device [num_seqs]: cache slot (< max_seqs of the cache); contiguous cache only */
  /* Paged cache (page_table != NULL; slot is then ignored and may be NULL):
   * page_table: device int32 [num_seqs][max_pages_per_seq]; entry [b][i] is the page that
   *   holds positions [i * page_size, (i + 1) * page_size) of sequence b (the entries a
   *   step reads or writes must be pages of the cache, else the device flags TP_ERR_BAD_TOKEN
   *   and that part of the step is skipped);
   * page_size: positions per page, a positive multiple of 128 (every 128-key tile of the
   *   attention kernels then lies in one page);
   * max_pages_per_seq: the table's row length; max_kv_len <= max_pages_per_seq * page_size. */
  const int32_t* page_table;
  int32_t page_size;
  int32_t max_pages_per_seq;
} tp_batch;

/* A2: vocab-parallel embedding ([TP] VocabParallelEmbedding): per rank, ids inside its slice
 * are looked up and the others give 0; the rank outputs are summed (fixed rank order).
 * ids: int32 [T] in device memory or in page-locked host memory (cudaHostAlloc / registered),
 * which the kernel then reads over the host link itself (no separate copy; the buffer must
 * stay unchanged until the kernel has run); other host memory is rejected with
 * TP_ERR_INVALID_ARG.  hidden_out: device fp32 [T, H] (the residual stream is fp32; GEMM
 * operands are fp16; attention runs on bf16 q and the bf16 KV cache).  Ids outside [0, V) give zero rows
 * and set TP_ERR_BAD_TOKEN in *dev_status (device int32, sticky, read by tp_read_status). */
tp_status tp_embed_vocab_parallel(tp_ctx* ctx, const void* head_shards, const int32_t* ids, int32_t num_tokens,
                                  void* hidden_out, int32_t* dev_status, void* stream);

/* A3-A10: one decoder layer under tensor parallelism, all ranks ([TP] TPTransformer.forward loop
 * body, TPAttention, TPMLP): RMSNorm -> merged QKV (column) -> q/k RMSNorm + RoPE + KV write ->
 * per-rank GQA attention -> o_proj (row) + rank-sum + residual -> RMSNorm -> gate/up (column) with
 * SiLU*up -> down (row) + rank-sum + residual.  hidden: device fp32 [T, H] residual stream,
 * updated in place.
 * kv_cache: this layer's cache (tp_kv_cache_bytes(kv_max_seqs, kv_capacity)): for a contiguous
 * cache kv_max_seqs slots of kv_capacity positions, for a paged one (batch->page_table set)
 * kv_max_seqs pages of kv_capacity = batch->page_size positions; positions
 * [ctx_len, ctx_len + q_len) of each sequence are written.  Exactly two rank-sums. */
tp_status tp_decoder_layer_forward(tp_ctx* ctx, const void* layer_shards, const tp_batch* batch, void* hidden,
                                   void* kv_cache, int32_t kv_max_seqs, int32_t kv_capacity, int32_t* dev_status,
                                   void* stream);

/* A11-A13: final RMSNorm of each sequence's last token, vocab-parallel logits (all ranks'
 * slices, padded columns masked) with a fused (max, first index) epilogue, and the argmax
 * reduction that replaces the all-gather ([TP] TPTransformer.forward; [CH9] ParallelLMHead).
 * hidden: device fp32 [T, H].  out_ids: int32 [num_seqs], in device memory or in page-locked
 * host memory, which the kernel then writes over the host link itself (complete when the
 * stream reaches this call's end); other host memory is rejected with TP_ERR_INVALID_ARG.
 * out_logits: fp32 [num_seqs, V] or NULL, under the same memory rule as out_ids. */
tp_status tp_lm_head_argmax(tp_ctx* ctx, const void* head_shards, const tp_batch* batch, const void* hidden,
                            int32_t* out_ids, float* out_logits, int32_t* dev_status, void* stream);

/* Same computation and results as tp_lm_head_argmax, for callers that cannot allocate device
 * memory (and so cannot provide the workspace): code that must not call cudaMalloc at that
 * point -- it can synchronise the device, or the process's device memory is owned by another
 * allocator -- or a caller holding only the weights, its inputs and its outputs.  The pages have
 * no counterpart; this is an interface convenience.
 * Scratch lives in one fixed array compiled into the library (about 1 MiB, held on every GPU
 * that loads the library until the process exits); no context workspace is needed and nothing
 * is allocated.  Limits: num_seqs <= TP_STATIC_SCRATCH_MAX_SEQS and hidden <=
 * TP_STATIC_SCRATCH_MAX_HIDDEN, else TP_ERR_INVALID_ARG before any launch.
 * The first call on a device looks up the array's device address (with that device current);
 * make that first call before any stream capture.  All calls share the array: calls that
 * overlap on the GPU race and must not be issued; each call clears the part that must start
 * at zero. */
#define TP_STATIC_SCRATCH_MAX_SEQS 64
#define TP_STATIC_SCRATCH_MAX_HIDDEN 8192
tp_status tp_lm_head_argmax_static(tp_ctx* ctx, const void* head_shards, const tp_batch* batch, const void* hidden,
                                   int32_t* out_ids, float* out_logits, int32_t* dev_status, void* stream);

/* Greedy generation between two forwards ([TP] tp.py main: the argmax of the last logits is
 * appended and fed back as the next one-token input).  batch: a decode batch (num_prefill
 * == 0, one token per sequence) whose forward (tp_decoder_layer_forward for every layer, then
 * tp_lm_head_argmax) has just run; its device ctx_len[b] grows by one (the token that
 * forward wrote to the cache; the array is written although tp_batch declares it const).
 * ids: device int32 [num_seqs], that forward's argmax ids; they are copied to row *step of
 * history (device int32 [max_rows][num_seqs]) and *step (device int32) grows by one.  All
 * state is on the device, so a CUDA graph of one decode forward plus this call can be
 * replayed unchanged step after step; the ids buffer can be the next forward's embedding
 * input.  A row outside [0, max_rows) is not written and sets TP_ERR_BAD_TOKEN in
 * *dev_status; a position beyond the cache is flagged by the next forward.
 * TP_ERR_INVALID_ARG for a null pointer, max_rows <= 0 or a batch with prefill sequences. */
tp_status tp_decode_advance(tp_ctx* ctx, const tp_batch* batch, const int32_t* ids, int32_t* history,
                            int32_t max_rows, int32_t* step, int32_t* dev_status, void* stream);

/* Synchronises the stream, reads the device status word and returns TP_OK, TP_ERR_TIMEOUT,
 * TP_ERR_BAD_TOKEN or TP_ERR_SATURATED (in that order of precedence; the word is not cleared).
 * Every device call ORs its flags into the caller's word: an fp16 conversion that clamps sets
 * the saturation flag, so a clamp is never silent.  After TP_ERR_TIMEOUT the context's
 * workspace counters are still consistent (every kernel counts itself in on its way out), but
 * that step's outputs are not valid. */
tp_status tp_read_status(const int32_t* dev_status, void* stream);

/* Rank-sums (emulated all-reduces) issued through this context so far: one per embedding,
 * two per layer ([TP] prints 57 = 28 x 2 + 1 for a 28-layer prefill). */
tp_status tp_rank_sum_count(const tp_ctx* ctx, int64_t* count);

/* ---------------- measurement hooks ----------------
 * Kernel kinds for per-kernel timing. */
#define TP_K_EMBED 0
#define TP_K_RMSNORM 1
#define TP_K_GEMM_QKV 2
#define TP_K_ROPE 3 /* q/k norm + RoPE + KV write: fused into TP_K_GEMM_QKV, never launched */
#define TP_K_ATTN_PREFILL 4
#define TP_K_ATTN_DECODE 5
#define TP_K_GEMM_O 6
#define TP_K_GEMM_GATE_UP 7
#define TP_K_GEMM_DOWN 8
#define TP_K_FINAL_NORM 9
#define TP_K_GEMM_LM_HEAD 10
#define TP_K_ARGMAX 11
#define TP_K_DECODE_ADVANCE 12
#define TP_K_COUNT 13

/* Kernels this context has launched so far (every kernel counts once). */
tp_status tp_launch_count(const tp_ctx* ctx, int64_t* count);
/* Start timing: from now on each launch of a kind whose bit is set in kind_mask is
 * bracketed by two CUDA events recorded on its stream (at most max_launches launches;
 * later ones are not timed).  Restarts the totals. */
tp_status tp_profile_begin(tp_ctx* ctx, uint32_t kind_mask, int32_t max_launches);
/* Stop timing, wait for the recorded events, and return per kind the summed device
 * time in ms (total_ms[TP_K_COUNT]) and the number of timed launches (launches[TP_K_COUNT]). */
tp_status tp_profile_end(tp_ctx* ctx, float* total_ms, int32_t* launches);

/* Text of the last CUDA error seen by a call on this thread ("" if none). */
const char* tp_last_cuda_error(void);

/* Test hook for the bounded waits: one kernel waits on a barrier nothing completes unless
 * *flag (device int32) is non-zero, gives up after limit_ns and sets TP_ERR_TIMEOUT. */
tp_status tp_debug_wait_probe(const int32_t* flag, int32_t* dev_status, int64_t limit_ns, void* stream);

/* The decode attention's split plan, as tp_decoder_layer_forward makes it for the decode
 * sequences of a step; host only, nothing is launched ("Tensor parallelism from scratch",
 * "The cost of communication", bounds a decode step below by the time to read memory; the
 * decode attention reads the KV cache, so its units of work are cut to keep every SM
 * streaming to the end).  The step's num_units (sequence,
 * rank, kv head) units go in up to four levels taken in order: level l holds units_out[l]
 * units whose keys are split in splits_out[l] parts; on 128-dim heads every split is
 * whole 128-key tiles and later levels are split finer (guided self-scheduling: the items
 * get smaller as the work left runs out).  max_kv_len: the step's longest context
 * (tp_batch.max_kv_len); num_sms: the device's SMs; head_dim: 64 or 128; group: q heads
 * per kv head (1, 2, 4 or 8); max_splits: the most splits the workspace holds partials
 * for.  units_out, splits_out: host int32[4].  TP_ERR_INVALID_ARG on a null pointer or a
 * value out of range (max_kv_len, num_units, num_sms, max_splits < 1).  Without a GPU the
 * occupancy query behind the first level's split count gives way to one CTA per SM. */
tp_status tp_debug_decode_plan(int32_t max_kv_len, int32_t num_units, int32_t num_sms, int32_t head_dim,
                               int32_t group, int32_t max_splits, int32_t* units_out, int32_t* splits_out);

#ifdef __cplusplus
}
#endif

#endif /* TPFWD_H */
