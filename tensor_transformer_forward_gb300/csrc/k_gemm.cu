// tcgen05 / TMEM / TMA GEMM with the tensor-parallel epilogues.
//
// Computes, for every token row t and feature f,
//     Y[t, f] = sum_r  X[t, r-th K segment] . W[r-th row block + f, :]
// where the segments r are the tensor-parallel ranks of a row-split layer
// (o_proj, down_proj) or a single segment for column-split layers (merged QKV,
// merged gate/up, LM head with all ranks' vocab slices stacked).
// ("Tensor parallelism from scratch", section "Two ways to split": a column
// split gives each rank a slice of the output, a row split gives each rank a
// partial sum that the all-reduce adds up; mini-SGLang linear.py:102-106.)
//
// Each rank's partial is accumulated by the tensor core in its own TMEM
// accumulator (fp32) and the partials are added in fixed rank order in the
// epilogue -- the all-reduce of the pages, done on one GPU.
//
// Structure: persistent, warp-specialised, 64 + 32 * EW threads per CTA
// (EW = 4 or 8 epilogue warps, GemmCfg::EW).
//   warp 0      TMA producer: X and W tiles (64-wide K blocks, 128-byte
//               swizzle) into a STAGES-deep shared-memory ring.
//   warp 1      TMEM allocator + MMA issuer (one thread): tcgen05.mma
//               M=128 x N=BN x K=16, two TMEM accumulators so the epilogue of
//               one segment overlaps the main loop of the next.
//   warps 2..   epilogue: tcgen05.ld of the accumulator (one TMEM lane = one
//               row of the MMA's M side per thread), then the fused epilogue;
//               with 8 warps (320 threads) the two warps of a TMEM lane
//               quarter take the two halves of the tile's columns.
// Orientation: tokens on the M side (tiles of 128 tokens x BN features), or,
// for a handful of tokens against a long weight (the LM head), weights on the
// M side (tiles of 128 features x BN tokens) so no shared-memory traffic is
// spent on padding rows.
// Split-K (for small token counts): a tile's K range is split over several
// CTAs; each writes an fp32 partial, the last to arrive (atomic counter, no
// spin-wait) adds the partials in split order and runs the epilogue.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cstdio>

#include "kernels.h"
#include "sm100.cuh"

namespace tpk {

struct GemmParams {
  int T, N, n_seg, kb_seg, x_k_seg, w_row_seg;
  int tiles_t, tiles_f, splits, total_kb;
  void* out;
  int ldo, out_cols;
  float* partials;
  int* counters;
  float* amax_val;
  int* amax_idx;
  int amax_ld;
  float* logits;
  int ld_logits, vocab;
  int32_t* out_ids;
  int* done_counter;   // CTAs finished (weight-streaming argmax)
  int* sched_counter;  // tiles handed out beyond the first wave (weight-streaming argmax)
  unsigned long long* amax_keys;  // [T] per-token argmax keys, zero between launches
  QkvEpi qkv;
  int* status;
  const void* discard[2];
  int64_t discard_lines[2];
  const float* row_ss;  // deferred RMSNorm: per-row 32-column sums of squares, or null
  int row_groups;
  float row_inv_k, row_eps;
  // residual epilogues: also leave the next norm's inputs (fp16 rows through tmO2,
  // 32-column sums of squares), reading the old residual instead of a reduce-add
  float* row_ss_out;
  int row_ss_out_groups;
  __half* row_out16;  // the fp16 rows (weights-on-M path writes them directly; ld = out_cols)
};

// PAIR: a cluster of two CTAs computes 256-token x BN tiles with one
// tcgen05.mma.cta_group::2 (M = 256): each CTA loads its own 128 token rows and
// half of the BN weight rows (BN / 2), so a K block moves 32 KB (BN = 256) into
// and out of each SM's shared memory instead of 48 KB; each CTA's epilogue
// handles its 128 rows from its own TMEM.
// XCH: a cluster of two such pairs on one 256 x 256 residual tile, each pair over
// one half of the K range (a rank segment at tp 2); each CTA sends the columns it
// does not finish to the other pair's CTA of the same rows through distributed
// shared memory and finishes the other 128 columns, adding the two halves in
// split order.
template <int BN, int EPI = EPI_STORE, bool ACC = false, bool SWAP = false, bool PAIR = false, bool XCH = false>
struct GemmCfg {
  static_assert(!XCH || (PAIR && EPI == EPI_RESID && BN == 256), "the exchange: residual 256-wide pair tiles");
  static constexpr int CL = XCH ? 4 : (PAIR ? 2 : 1);  // CTAs per cluster
  // epilogue warps: 8 (two per TMEM lane quarter, splitting the columns) where the
  // columns split into independent halves, else 4
  static constexpr int EW =
      (!SWAP && (EPI == EPI_STORE || EPI == EPI_RESID || (EPI == EPI_SILU && BN >= 256) ||
                 (EPI == EPI_QKV && !ACC && BN >= 256)))
          ? 8
          : 4;
  static constexpr int THREADS = 64 + 32 * EW;
  static constexpr int A_BYTES = 128 * 128;  // 128 rows x 64 fp16
  static constexpr int B_BYTES = (PAIR ? BN / 2 : BN) * 128;  // this CTA's weight rows x 64 fp16
  static constexpr int TM_T = SWAP ? BN : (PAIR ? 256 : 128);  // tokens per tile (both CTAs of a pair)
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // as many stages as fit in ~200 KB (narrow tiles stream weights: more bytes in flight)
  // QKV with two warps per lane quarter (see QKV_PAIR below) keeps 3 stages: its
  // row staging takes the room of the fourth
  static constexpr bool QKV_PAIR = EPI == EPI_QKV && !SWAP && !ACC && EW == 8;
  // token-tile residual epilogues also stage fp16 rows (one 32 x 32 box of 2 KB per
  // epilogue warp next to its fp32 box)
  static constexpr bool RESID_ROWS = !SWAP && EPI == EPI_RESID;
  // ... and prefetch the old residual of their first NXB 32-column chunks into
  // extra fp32 boxes while the MMA runs (one box per chunk)
  static constexpr int NXB = RESID_ROWS ? ((BN / (EW / 4)) / 32 < 2 ? (BN / (EW / 4)) / 32 : 2) : 1;
  static constexpr int ROW16_BYTES = RESID_ROWS ? EW * (2048 + (NXB - 1) * 4096) : 0;
  static constexpr int STAGES =
      QKV_PAIR ? (PAIR ? 4 : 3)
      : ((204800 - ROW16_BYTES - ((SWAP && EPI != EPI_ARGMAX) ? BN * 512 : 0)) / STAGE_BYTES) > 12
          ? 12
          : ((204800 - ROW16_BYTES - ((SWAP && EPI != EPI_ARGMAX) ? BN * 512 : 0)) / STAGE_BYTES);
  // two accumulators of BN columns, each starting at a multiple of TM_STRIDE (the
  // allocation is a power of two of at least 32 columns)
  static constexpr int TMEM_COLS = 2 * BN <= 32 ? 32 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
  static constexpr int TM_STRIDE = TMEM_COLS / 2;
  static constexpr int QUEUE = 4;  // tile queue depth (weight-streaming argmax)
  // weight-streaming argmax: tiles from a dynamic queue; other swapped (few-token)
  // GEMMs: static round-robin over tiles x K splits
  static constexpr bool DYN = SWAP && EPI == EPI_ARGMAX;
  // swapped epilogues other than the argmax stage the summed tile token-major in
  // fp32 ([BN tokens][128 features]) and write whole token rows from there
  static constexpr int TROW_BYTES = (SWAP && EPI != EPI_ARGMAX) ? BN * 128 * 4 : 0;
  static constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * QUEUE + 1 + 2;  // ... PRO, XRDY, XFULL
  // outputs leave through TMA stores (fp16) / TMA reduce-adds (fp32 residual) from one
  // 32-row x 128-byte staging box per epilogue warp
  static constexpr bool TMA_OUT = !SWAP && (EPI == EPI_STORE || EPI == EPI_SILU || EPI == EPI_RESID);
  static constexpr int OUT_BYTES = (TMA_OUT ? EW * 4096 : 0) + ROW16_BYTES;
  // QKV with two warps per lane quarter: q/k norm weights [2][128] fp32, the
  // per-row partial sums of squares [2 parities][2 warps][BN/64 heads at most][128]
  // and each warp's row staging [2 outputs][32 rows][128 bytes at most]
  static constexpr int QKV_BYTES = QKV_PAIR ? 128 + 256 * 4 + 2 * 2 * (BN / 64) * 128 * 4 + EW * 2 * 32 * 128 : 0;
  // small area after the barriers: TMEM address and flags (64 B), the argmax
  // epilogue's per-warp partials (2 x 512 B) and per-token running best (2 x BEST
  // entries: up to 256 tokens on the weight-streaming argmax path, else 64; the
  // other swapped epilogues use the same area for their token table)
  static constexpr int BEST = (SWAP && EPI == EPI_ARGMAX) ? 256 : 64;
  // the weight-streaming argmax keeps 64-bit keys instead: [4 warps][BN] column
  // maxima of a tile and [BN] per-token running maxima
  // and, per epilogue warp, a 32 x 33 word buffer that transposes a 32 x 32 block of keys
  static constexpr int SMALL_BYTES = 64 + ((SWAP && EPI == EPI_ARGMAX) ? 40 * BN + 4 * 32 * 33 * 4 : 1024 + 8 * BEST);
  static constexpr int SMEM =
      1024 + STAGES * STAGE_BYTES + OUT_BYTES + TROW_BYTES + NUM_BARS * 8 + SMALL_BYTES + 128 + QKV_BYTES;
  static_assert(SMEM <= 232448, "shared memory per block");
};

struct Unit {
  int tt, tf, split, g0, g1;
};

__device__ __forceinline__ Unit unit_of(const GemmParams& p, int u) {
  Unit un;
  un.split = u % p.splits;
  const int tile = u / p.splits;
  un.tf = tile % p.tiles_f;
  un.tt = tile / p.tiles_f;
  un.g0 = static_cast<int>((static_cast<long long>(un.split) * p.total_kb) / p.splits);
  un.g1 = static_cast<int>((static_cast<long long>(un.split + 1) * p.total_kb) / p.splits);
  return un;
}

// After a wait gave up (TP_DEVFLAG_TIMEOUT is set, the results are not valid):
// counts unit u and every later unit of this CTA in on their split-K tile
// counters, so that each counter still returns to zero (the last to arrive
// clears it) and the next launch starts clean.  One thread.  A CTA pair keeps
// one counter per CTA of a tile (its 128 rows): counter 2 * tile + crank.
__device__ __forceinline__ void drain_split_counters(const GemmParams& p, int u, int units, int ustep, int per_tile,
                                                     int crank) {
  if (p.splits <= 1) return;
  for (; u < units; u += ustep) {
    const int tile = (u / p.splits) * per_tile + crank;
    if (atomicAdd(p.counters + tile, 1) == p.splits - 1) p.counters[tile] = 0;
  }
}

// Deferred RMSNorm of input row t: rsqrt(mean of squares + eps) from the
// row's 32-column sums of squares ("Tensor parallelism from scratch", the
// RMSNorm before each projection; its weight is folded into W), 1 without them.
__device__ __forceinline__ float row_scale(const GemmParams& p, int t) {
  if (p.row_ss == nullptr) return 1.0f;
  const float* g = p.row_ss + static_cast<size_t>(t) * p.row_groups;
  float s0 = 0.0f, s1 = 0.0f;
  int i = 0;
  if ((p.row_groups & 3) == 0) {
    for (; i < p.row_groups; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(g + i);
      s0 += v.x + v.y;
      s1 += v.z + v.w;
    }
  } else {
    for (; i < p.row_groups; ++i) s0 += g[i];
  }
  return rsqrtf((s0 + s1) * p.row_inv_k + p.row_eps);
}

// fast divide: the result is rounded to fp16 (11 bits) next, far coarser than its ~2 ulp fp32 error;
// for g very negative the divisor overflows to inf and the quotient is 0, the correct limit
__device__ __forceinline__ float silu_f(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

// (value, index) order of torch.argmax (larger value first, NaN above all, then
// the lower index) as one unsigned 64-bit key (larger = better): the value's bits
// made monotone in the high word (NaN above everything, -0 taken as +0), the
// complemented index in the low word (lower index wins a tie).  Every key is
// above 0, the cleared state.
__device__ __forceinline__ unsigned long long amax_key(float v, int i) {
  uint32_t hi;
  if (v != v) {
    hi = 0xffffffffu;
  } else {
    const uint32_t b = __float_as_uint(v == 0.0f ? 0.0f : v);
    hi = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  }
  return (static_cast<unsigned long long>(hi) << 32) | static_cast<unsigned long long>(~static_cast<uint32_t>(i));
}

// 8 consecutive values as bf16 (the KV cache) or fp16 (GEMM / attention operands)
__device__ __forceinline__ void store8(__nv_bfloat16* dst, const float* x) {
  uint4 w;
  w.x = pack_bf16x2(x[0], x[1]);
  w.y = pack_bf16x2(x[2], x[3]);
  w.z = pack_bf16x2(x[4], x[5]);
  w.w = pack_bf16x2(x[6], x[7]);
  *reinterpret_cast<uint4*>(dst) = w;
}
__device__ __forceinline__ void store8(__half* dst, const float* x, uint32_t& sat) {
  uint4 w;
  w.x = pack_f16x2(x[0], x[1], sat);
  w.y = pack_f16x2(x[2], x[3], sat);
  w.z = pack_f16x2(x[4], x[5], sat);
  w.w = pack_f16x2(x[6], x[7], sat);
  *reinterpret_cast<uint4*>(dst) = w;
}

// ---- TMA-store staging: one thread = one row of a 32-row x 128-byte box, written
// with the 128-byte swizzle the tensor map declares (16-byte chunk c of row r at
// chunk c ^ (r & 7)), so the 8 rows of a bank group never collide.
__device__ __forceinline__ void stage_f32x32(uint8_t* box, int r, const float* v) {
  uint8_t* rowp = box + r * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<float4*>(rowp + ((c ^ (r & 7)) << 4)) = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
}
__device__ __forceinline__ void stage_f16x64(uint8_t* box, int r, const float* v, uint32_t& sat) {
  uint8_t* rowp = box + r * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    uint4 w;
    w.x = pack_f16x2(v[8 * c + 0], v[8 * c + 1], sat);
    w.y = pack_f16x2(v[8 * c + 2], v[8 * c + 3], sat);
    w.z = pack_f16x2(v[8 * c + 4], v[8 * c + 5], sat);
    w.w = pack_f16x2(v[8 * c + 6], v[8 * c + 7], sat);
    *reinterpret_cast<uint4*>(rowp + ((c ^ (r & 7)) << 4)) = w;
  }
}
// One row of a 32-row x 64-byte fp16 box (tensor map without swizzle).
__device__ __forceinline__ void stage_f16x32(uint8_t* box, int r, const float* v, uint32_t& sat) {
  uint4* rowp = reinterpret_cast<uint4*>(box + r * 64);
#pragma unroll
  for (int c = 0; c < 4; ++c)
    rowp[c] = make_uint4(pack_f16x2(v[8 * c], v[8 * c + 1], sat), pack_f16x2(v[8 * c + 2], v[8 * c + 3], sat),
                         pack_f16x2(v[8 * c + 4], v[8 * c + 5], sat), pack_f16x2(v[8 * c + 6], v[8 * c + 7], sat));
}
// Whole warp: wait until the box's previous store has read it.
__device__ __forceinline__ void box_acquire(int lane) {
  if (lane == 0) bulk_wait_read();
  __syncwarp();
}
// Whole warp, after every lane staged its row: hand the box to the TMA unit.
__device__ __forceinline__ void box_release(const CUtensorMap* map, uint8_t* box, int x, int y, bool reduce_add,
                                            int lane) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    if (reduce_add) tma_reduce_add_2d(map, smem_u32(box), x, y);
    else tma_store_2d(map, smem_u32(box), x, y);
    bulk_commit();
  }
}

// Per-thread asynchronous copies (cp.async, 16 bytes each) and their waits.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// The old residual of this row's 32 columns from col, copied asynchronously into
// row `lane` of an fp32 staging box (in the swizzled layout stage_f32x32 writes).
__device__ __forceinline__ void prefetch_rows32(const GemmParams& p, uint8_t* xbox, int t, bool row_ok, int col,
                                                int lane) {
  if (row_ok && col < p.out_cols) {
    const float* src = reinterpret_cast<const float*>(p.out) + static_cast<size_t>(t) * p.ldo + col;
#pragma unroll
    for (int c = 0; c < 8; ++c) cp_async16(smem_u32(xbox + lane * 128 + ((c ^ (lane & 7)) << 4)), src + 4 * c);
  }
  cp_async_commit();
}

// Residual epilogue with the next norm's inputs: v (32 columns of this row's
// rank-summed tile, starting at column col) += the old residual; the new
// residual leaves through the fp32 box (plain TMA store), its fp16 copy through
// the fp16 box, and the group's sum of squares goes to row_ss_out.  Whole warp.
// With prefetched (box already holds the old residual, copied by prefetch_rows32
// and waited for) the old values come from the box, else from global memory.
template <typename Cfg>
__device__ __forceinline__ void resid_rows32(const GemmParams& p, const CUtensorMap* tmO, const CUtensorMap* tmO2,
                                             uint8_t* box, uint8_t* box16, int t, bool row_ok, int col, int tbox,
                                             int lane, float* v, bool prefetched, uint32_t& sat) {
  float s = 0.0f;
  if (row_ok && col < p.out_cols) {  // out_cols % 32 == 0: a group is wholly inside or outside
    const float4* x = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.out) +
                                                      static_cast<size_t>(t) * p.ldo + col);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float4 o = prefetched ? *reinterpret_cast<const float4*>(box + lane * 128 + ((i ^ (lane & 7)) << 4))
                                  : x[i];
      v[4 * i] += o.x;
      v[4 * i + 1] += o.y;
      v[4 * i + 2] += o.z;
      v[4 * i + 3] += o.w;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) s += v[i] * v[i];
    p.row_ss_out[static_cast<size_t>(t) * p.row_ss_out_groups + col / 32] = s;
  }
  box_acquire(lane);  // the fp16 box (and a reused fp32 box) of the previous chunk has been read
  stage_f32x32(box, lane, v);
  stage_f16x32(box16, lane, v, sat);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmO, smem_u32(box), col, tbox);
    tma_store_2d(tmO2, smem_u32(box16), col, tbox);
    bulk_commit();
  }
}

__device__ __forceinline__ void argmax_scan(const GemmParams& p, int t, int f, const float* v, float& best,
                                            int& bi) {
  float* lg = p.logits ? p.logits + static_cast<size_t>(t) * p.ld_logits : nullptr;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int fi = f + i;
    if (fi < p.vocab) {
      const float x = v[i];
      if (lg) lg[fi] = x;
      const bool take = (bi < 0) || (x > best) || (x != x && best == best);
      if (take) {
        best = x;
        bi = fi;
      }
    }
  }
}

// Token row t -> its position and where its K / V go in the cache: block (slot
// or page) and row in the block (binary search over cu_q for prefill tokens).
struct TokPos {
  int pos, blk, brow;
  bool ok, prefill;
};
__device__ __forceinline__ TokPos token_position(const QkvEpi& q, int t) {
  // decode sequences (one token each) follow the prefill ones: direct index;
  // a prefill token searches the prefill sequences only
  int lo;
  const int t_dec = q.num_prefill < q.B ? q.cu_q[q.num_prefill] : INT_MAX;
  if (t >= t_dec) {
    lo = q.num_prefill + (t - t_dec);
    if (lo >= q.B) {  // a "decode" sequence with more than one token: reject, stay in bounds
      TokPos bad{0, 0, 0, false, false};
      return bad;
    }
  } else {
    lo = 0;
    int hi = q.num_prefill - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (q.cu_q[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
  }
  TokPos tp;
  tp.pos = q.ctx_len[lo] + (t - q.cu_q[lo]);
  const int blk = tp.pos < q.max_pos ? kv_block(q.kvm, lo, tp.pos) : -1;
  tp.ok = blk >= 0;
  tp.blk = tp.ok ? blk : 0;
  tp.brow = tp.ok ? tp.pos % q.kvm.block_len : 0;
  tp.prefill = lo < q.num_prefill;
  return tp;
}

// One head of the merged QKV row of token t (fp32, straight from the
// accumulator): q and k get RMSNorm over head_dim and rotate-half RoPE at the
// token's position; q goes back to the QKV buffer, k and v to the rank's cache
// (post-RoPE K, raw V).  ("Tensor parallelism from scratch", tp.py
// TPAttention.forward: q_norm / k_norm, apply_rope, cache.update.)
template <int HD>
__device__ __forceinline__ void qkv_head(const GemmParams& p, int t, const TokPos& tp, int col0, const float* h,
                                         uint32_t& sat) {
  const QkvEpi& q = p.qkv;
  constexpr int HALF = HD / 2;
  const int r = col0 / q.w_rank;
  const int sh = (col0 - r * q.w_rank) / HD;
  __nv_bfloat16* kv = reinterpret_cast<__nv_bfloat16*>(q.kv);
  if (sh >= q.nq_l + q.nkv_l) {  // v: raw into the cache
    const int g = sh - q.nq_l - q.nkv_l;
    __nv_bfloat16* dst = kv + kv_row(q.kvm, q.nkv_l, r, 1, tp.blk, g, tp.brow) * HD;
#pragma unroll
    for (int j = 0; j < HD / 8; ++j) store8(dst + j * 8, h + j * 8);
    return;
  }
  const bool is_q = sh < q.nq_l;
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < HD; ++i) ss += h[i] * h[i];
  const float inv = rsqrtf(ss / static_cast<float>(HD) + q.eps);
  const __nv_bfloat16* nw = reinterpret_cast<const __nv_bfloat16*>(is_q ? q.q_norm : q.k_norm);
  // (cos, sin) pairs of d and d+1 for this position: one float4 every 32 (positions side by side)
  const float4* cs4 = reinterpret_cast<const float4*>(q.rope) + static_cast<size_t>(tp.pos >> 5) * (HALF / 2) * 32 +
                      (tp.pos & 31);
  // q of a prefill token: bf16 high part in the QKV buffer and the bf16 low part
  // q - bf16(q) in q_lo (the tensor-core attention multiplies both with the bf16
  // keys); q of a decode token: fp16 in the QKV buffer (fp32 attention math).
  __nv_bfloat16* qhi = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(t) * p.ldo + col0;
  __half* q16 = reinterpret_cast<__half*>(qhi);
  __nv_bfloat16* qlo = reinterpret_cast<__nv_bfloat16*>(q.q_lo) +
                       static_cast<size_t>(t) * q.n * q.nq_l * HD + (static_cast<size_t>(r) * q.nq_l + sh) * HD;
  __nv_bfloat16* kdst = kv + kv_row(q.kvm, q.nkv_l, r, 0, tp.blk, sh - q.nq_l, tp.brow) * HD;  // k: bf16 cache
#pragma unroll
  for (int j = 0; j < HALF / 8; ++j) {
    // 16-byte loads: 8 norm weights of each half, 8 (cos, sin) pairs
    const uint4 w0 = *reinterpret_cast<const uint4*>(nw + j * 8);
    const uint4 w1 = *reinterpret_cast<const uint4*>(nw + HALF + j * 8);
    const float wa[8] = {bf16lo(w0.x), bf16hi(w0.x), bf16lo(w0.y), bf16hi(w0.y),
                         bf16lo(w0.z), bf16hi(w0.z), bf16lo(w0.w), bf16hi(w0.w)};
    const float wb[8] = {bf16lo(w1.x), bf16hi(w1.x), bf16lo(w1.y), bf16hi(w1.y),
                         bf16lo(w1.z), bf16hi(w1.z), bf16lo(w1.w), bf16hi(w1.w)};
    float4 c4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c4[i] = __ldg(cs4 + (j * 4 + i) * 32);
    const float cx[8] = {c4[0].x, c4[0].z, c4[1].x, c4[1].z, c4[2].x, c4[2].z, c4[3].x, c4[3].z};
    const float sy[8] = {c4[0].y, c4[0].w, c4[1].y, c4[1].w, c4[2].y, c4[2].w, c4[3].y, c4[3].w};
    float y0[8], y1[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int d = j * 8 + i;
      const float u0 = h[d] * inv * wa[i];
      const float u1 = h[d + HALF] * inv * wb[i];
      y0[i] = u0 * cx[i] - u1 * sy[i];
      y1[i] = u1 * cx[i] + u0 * sy[i];
    }
    if (!is_q) {
      store8(kdst + j * 8, y0);
      store8(kdst + HALF + j * 8, y1);
    } else if (!tp.prefill) {
      store8(q16 + j * 8, y0, sat);
      store8(q16 + HALF + j * 8, y1, sat);
    } else {
      float l0[8], l1[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        l0[i] = y0[i] - bf2f(f2bf(y0[i]));
        l1[i] = y1[i] - bf2f(f2bf(y1[i]));
      }
      store8(qhi + j * 8, y0);
      store8(qhi + HALF + j * 8, y1);
      store8(qlo + j * 8, l0);
      store8(qlo + HALF + j * 8, l1);
    }
  }
}

// Each thread of the warp reads 8 consecutive fp32 columns of its TMEM lane.
__device__ __forceinline__ void tc_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}

// QKV tile epilogue with two warps per TMEM lane quarter (tokens on the M side).
// Warp w of the pair takes rotation pairs [w*QP, (w+1)*QP) of every head in the
// tile, i.e. dims d and d + hd/2 of those pairs; a q/k head's sum of squares is
// completed across the pair through shared memory (ss, double-buffered by tile
// parity).  The (cos, sin) values of the thread's token and pairs are loaded
// before the accumulator is ready, so their latency hides behind the MMA, and
// they serve every q/k head of the tile; the q/k norm weights sit in shared
// memory (nw: [2][128] fp32, q then k).  Same arithmetic as qkv_head, after the
// deferred input norm's row scale rinv.
// Each thread stages its row's results in the warp's staging (stg: [2 outputs:
// high / k / v, q low][2 segments: the pairs' first and second halves][32 rows]
// [QP bf16]).  q rows leave through TMA stores of those 32-row boxes (tmQ: the
// QKV buffer, tmQlo: the q low part); so do k and v rows when the warp's 32
// tokens are one sequence at consecutive positions (32 consecutive rows of the
// cache seen as [rows][hd], tmKV); otherwise each row goes to its token's cache
// position, written by the warp as whole row segments.
// Returns false (on both warps of the pair) when the accumulator wait failed.
template <int BN, int HD>
__device__ __forceinline__ bool qkv_pair_tile(const GemmParams& p, const CUtensorMap* tmQ, const CUtensorMap* tmQlo,
                                              const CUtensorMap* tmKV, uint32_t tfull, uint32_t use, volatile int* abort_flag, uint32_t ta,
                                              int t, const TokPos& tp, int f0, bool row_ok, int w, int q, int row,
                                              int par, const float* nw, float* ss, uint8_t* stg, float rinv,
                                              uint32_t& sat) {
  constexpr int HALF = HD / 2, QP = HALF / 2, NR = QP / 2, HPT = BN / HD;
  constexpr int SEGB = QP * 2;        // bytes of one row segment (QP bf16)
  constexpr int NC = SEGB / 16;       // 16-byte chunks per row segment
  constexpr int OUTB = 2 * 32 * SEGB; // bytes per output
  const int lane = threadIdx.x & 31;
  const int tbox = t - lane;          // first row of this warp's 32 rows
  const QkvEpi& e = p.qkv;
  int kind[HPT];  // per head of the tile: 0 q, 1 k, 2 v, -1 past the last column (warp-uniform)
  bool any_rot = false;
#pragma unroll
  for (int hb = 0; hb < HPT; ++hb) {
    const int col0 = f0 + hb * HD;
    if (col0 >= p.N) {
      kind[hb] = -1;
    } else {
      const int sh = (col0 - (col0 / e.w_rank) * e.w_rank) / HD;
      kind[hb] = sh < e.nq_l ? 0 : (sh < e.nq_l + e.nkv_l ? 1 : 2);
      any_rot |= kind[hb] < 2;
    }
  }
  const bool live = row_ok && tp.ok;
  float4 rc[NR];
  if (any_rot && live) {
    const float4* cs4 = reinterpret_cast<const float4*>(e.rope) + static_cast<size_t>(tp.pos >> 5) * (HALF / 2) * 32 +
                        (tp.pos & 31) + w * NR * 32;
#pragma unroll
    for (int i = 0; i < NR; ++i) rc[i] = __ldg(cs4 + i * 32);
  } else {
#pragma unroll
    for (int i = 0; i < NR; ++i) rc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const bool ok = mbar_wait(tfull, use, abort_flag, p.status);
  if (!named_bar_and(2 + q, 64, ok)) return false;
  tc_fence_after();
  float inv[HPT];
#pragma unroll
  for (int hb = 0; hb < HPT; ++hb) inv[hb] = 0.0f;
  if (any_rot) {
    float* mine = ss + (par * 2 + w) * (HPT * 128);
    const float* other = ss + (par * 2 + (1 - w)) * (HPT * 128);
#pragma unroll
    for (int hb = 0; hb < HPT; ++hb) {
      if (kind[hb] < 0 || kind[hb] == 2) continue;
      float s = 0.0f;
#pragma unroll
      for (int c = 0; c < QP / 16; ++c) {
        float a[16], b[16];
        tc_ld16(ta + hb * HD + w * QP + c * 16, a);
        tc_ld16(ta + hb * HD + HALF + w * QP + c * 16, b);
#pragma unroll
        for (int i = 0; i < 16; ++i) s += a[i] * a[i] + b[i] * b[i];
      }
      mine[hb * 128 + row] = s;
      inv[hb] = s;
    }
    named_bar_sync(2 + q, 64);
#pragma unroll
    for (int hb = 0; hb < HPT; ++hb)
      if (kind[hb] == 0 || kind[hb] == 1)
        inv[hb] = rsqrtf((inv[hb] + other[hb * 128 + row]) * (rinv * rinv) / static_cast<float>(HD) + e.eps);
  }
  __nv_bfloat16* kv = reinterpret_cast<__nv_bfloat16*>(e.kv);
#pragma unroll
  for (int hb = 0; hb < HPT; ++hb) {
    if (kind[hb] < 0) continue;
    const int col0 = f0 + hb * HD;
    const int r = col0 / e.w_rank;
    const int sh = (col0 - r * e.w_rank) / HD;
    const bool lo_out = kind[hb] == 0 && tp.prefill;  // per row
    const float* w8 = nw + (kind[hb] == 1 ? 128 : 0);
    // the staging's previous TMA stores have read it
    if (lane == 0) bulk_wait_read();
    __syncwarp();
#pragma unroll
    for (int c2 = 0; c2 < QP / 16; ++c2) {
      float a[16], b[16];
      tc_ld16(ta + hb * HD + w * QP + c2 * 16, a);
      tc_ld16(ta + hb * HD + HALF + w * QP + c2 * 16, b);
#pragma unroll
      for (int hc = 0; hc < 2; ++hc) {  // 8 pairs per staged chunk
        const int c = c2 * 2 + hc;       // chunk within the row segment
        const int d0 = w * QP + c * 8;
        float x0[8], x1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {  // deferred RMSNorm of the input row
          x0[i] = a[hc * 8 + i] * rinv;
          x1[i] = b[hc * 8 + i] * rinv;
        }
        uint8_t* s0 = stg + lane * SEGB + c * 16;                 // output 0, segment 0
        uint8_t* s1 = stg + 32 * SEGB + lane * SEGB + c * 16;     // output 0, segment 1
        if (kind[hb] == 2) {  // v: raw
          *reinterpret_cast<uint4*>(s0) = make_uint4(pack_bf16x2(x0[0], x0[1]), pack_bf16x2(x0[2], x0[3]),
                                                     pack_bf16x2(x0[4], x0[5]), pack_bf16x2(x0[6], x0[7]));
          *reinterpret_cast<uint4*>(s1) = make_uint4(pack_bf16x2(x1[0], x1[1]), pack_bf16x2(x1[2], x1[3]),
                                                     pack_bf16x2(x1[4], x1[5]), pack_bf16x2(x1[6], x1[7]));
          continue;
        }
        float y0[8], y1[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 cc = rc[(c * 8 + i) >> 1];
          const float cs = (i & 1) ? cc.z : cc.x;
          const float sn = (i & 1) ? cc.w : cc.y;
          const float u0 = x0[i] * inv[hb] * w8[d0 + i];
          const float u1 = x1[i] * inv[hb] * w8[HALF + d0 + i];
          y0[i] = u0 * cs - u1 * sn;
          y1[i] = u1 * cs + u0 * sn;
        }
        if (kind[hb] == 0 && !tp.prefill) {  // decode q: fp16
          *reinterpret_cast<uint4*>(s0) = make_uint4(pack_f16x2(y0[0], y0[1], sat), pack_f16x2(y0[2], y0[3], sat),
                                                     pack_f16x2(y0[4], y0[5], sat), pack_f16x2(y0[6], y0[7], sat));
          *reinterpret_cast<uint4*>(s1) = make_uint4(pack_f16x2(y1[0], y1[1], sat), pack_f16x2(y1[2], y1[3], sat),
                                                     pack_f16x2(y1[4], y1[5], sat), pack_f16x2(y1[6], y1[7], sat));
        } else {  // k, prefill q high part: bf16
          *reinterpret_cast<uint4*>(s0) = make_uint4(pack_bf16x2(y0[0], y0[1]), pack_bf16x2(y0[2], y0[3]),
                                                     pack_bf16x2(y0[4], y0[5]), pack_bf16x2(y0[6], y0[7]));
          *reinterpret_cast<uint4*>(s1) = make_uint4(pack_bf16x2(y1[0], y1[1]), pack_bf16x2(y1[2], y1[3]),
                                                     pack_bf16x2(y1[4], y1[5]), pack_bf16x2(y1[6], y1[7]));
          if (lo_out) {  // q - bf16(q)
            float l0[8], l1[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              l0[i] = y0[i] - bf2f(f2bf(y0[i]));
              l1[i] = y1[i] - bf2f(f2bf(y1[i]));
            }
            *reinterpret_cast<uint4*>(s0 + OUTB) =
                make_uint4(pack_bf16x2(l0[0], l0[1]), pack_bf16x2(l0[2], l0[3]), pack_bf16x2(l0[4], l0[5]),
                           pack_bf16x2(l0[6], l0[7]));
            *reinterpret_cast<uint4*>(s1 + OUTB) =
                make_uint4(pack_bf16x2(l1[0], l1[1]), pack_bf16x2(l1[2], l1[3]), pack_bf16x2(l1[4], l1[5]),
                           pack_bf16x2(l1[6], l1[7]));
          }
        }
      }
    }
    if (kind[hb] == 0) {
      // q: 32-row boxes to the QKV buffer (and the low part), rows past the last
      // token clipped by the tensor maps
      const bool any_lo = __any_sync(0xffffffffu, live && lo_out);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int lo_col = (r * e.nq_l + sh) * HD;
#pragma unroll
        for (int sg = 0; sg < 2; ++sg) {
          tma_store_2d(tmQ, smem_u32(stg + sg * 32 * SEGB), col0 + sg * HALF + w * QP, tbox);
          if (any_lo) tma_store_2d(tmQlo, smem_u32(stg + OUTB + sg * 32 * SEGB), lo_col + sg * HALF + w * QP, tbox);
        }
        bulk_commit();
      }
      continue;
    }
    const int g = kind[hb] == 1 ? sh - e.nq_l : sh - e.nq_l - e.nkv_l;
    {
      // k / v of 32 tokens at consecutive rows of one cache block (one sequence at
      // consecutive positions, not crossing a page): 32 consecutive cache rows
      const int blk0 = __shfl_sync(0xffffffffu, tp.blk, 0);
      const int brow0 = __shfl_sync(0xffffffffu, tp.brow, 0);
      if (__all_sync(0xffffffffu, live && tp.blk == blk0 && tp.brow == brow0 + lane)) {
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          const int crow = static_cast<int>(kv_row(e.kvm, e.nkv_l, r, kind[hb] == 2 ? 1 : 0, blk0, g, brow0));
#pragma unroll
          for (int sg = 0; sg < 2; ++sg) tma_store_2d(tmKV, smem_u32(stg + sg * 32 * SEGB), sg * HALF + w * QP, crow);
          bulk_commit();
        }
        continue;
      }
    }
    __syncwarp();
    // k / v: lane -> (row rr, segment sg, chunk k) of the staged rows; row rr's
    // cache row comes from its owner lane
    const unsigned long long my_dst =
        live ? reinterpret_cast<unsigned long long>(
                   kv + kv_row(e.kvm, e.nkv_l, r, kind[hb] == 2 ? 1 : 0, tp.blk, g, tp.brow) * HD)
             : 0ull;
#pragma unroll
    for (int i = 0; i < 2 * NC; ++i) {
      const int idx = i * 32 + lane;
      const int rr = idx / (2 * NC), rem = idx % (2 * NC), sg = rem / NC, k = rem % NC;
      const unsigned long long dd = __shfl_sync(0xffffffffu, my_dst, rr);
      if (dd) *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(dd) + sg * HALF + w * QP + k * 8) =
          *reinterpret_cast<const uint4*>(stg + sg * 32 * SEGB + rr * SEGB + k * 16);
    }
    __syncwarp();  // the staging rows are rewritten by the next head
  }
  return true;
}

// Streams the heads of one accumulator tile (tokens on the M side) through qkv_head.
template <int BN, int HD>
__device__ __forceinline__ void qkv_stream(const GemmParams& p, uint32_t ta, int t, const TokPos& tp, int f0,
                                           bool row_ok, int c_begin, int c_end, float rinv, uint32_t& sat) {
#pragma unroll 1
  for (int hb = c_begin / HD; hb < c_end / HD; ++hb) {
    const int col0 = f0 + hb * HD;
    if (col0 >= p.N) break;  // warp-uniform
    float h[HD];
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      float v[32];
      tc_ld32(ta + hb * HD + c * 32, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) h[c * 32 + i] = v[i] * rinv;
    }
    if (row_ok && tp.ok) qkv_head<HD>(p, t, tp, col0, h, sat);
  }
}

// ---- few-token GEMMs with the weights on the MMA's M side ----
// The accumulator tile is 128 features (TMEM lanes) x BN tokens (columns).  Each
// epilogue thread owns one feature row: it adds the rank segments of its unit in
// rank order, the K splits are added in split order (last CTA to arrive), and
// the sum is staged token-major in shared memory.  Each warp then writes whole
// token rows: lane l holds features 4l .. 4l+3 of the tile.

// q/k RMSNorm + rotate-half RoPE for one token row of one head spread over a
// group of G lanes (G = HD / 4; lane i of the group holds dims 4i .. 4i+3), then
// the q / k / v row written out.  ("Tensor parallelism from scratch", tp.py
// TPAttention.forward: q_norm / k_norm, apply_rope, cache.update.)
template <int HD>
__device__ __forceinline__ void qkv_row_group(const GemmParams& p, int t, const TokPos& tp, int col0, int gl,
                                              float4 v, uint32_t& sat) {
  const QkvEpi& q = p.qkv;
  constexpr int G = HD / 4;  // lanes per head
  constexpr int HALF = HD / 2;
  const int r = col0 / q.w_rank;
  const int sh = (col0 - r * q.w_rank) / HD;
  const int d0 = 4 * gl;  // first dim of this lane
  __nv_bfloat16* kv = reinterpret_cast<__nv_bfloat16*>(q.kv);
  float y[4] = {v.x, v.y, v.z, v.w};
  const bool is_v = sh >= q.nq_l + q.nkv_l, is_q = sh < q.nq_l;
  {  // every lane runs the shuffles (the two heads of a 64-dim pair may be of different kinds)
    float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv = rsqrtf(ss / static_cast<float>(HD) + q.eps);
    const __nv_bfloat16* nw = reinterpret_cast<const __nv_bfloat16*>(is_q ? q.q_norm : q.k_norm);
    const uint2 wv = *reinterpret_cast<const uint2*>(nw + d0);
    const float w4[4] = {bf16lo(wv.x), bf16hi(wv.x), bf16lo(wv.y), bf16hi(wv.y)};
    float u[4], o4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) u[i] = y[i] * inv * w4[i];
#pragma unroll
    for (int i = 0; i < 4; ++i) o4[i] = __shfl_xor_sync(0xffffffffu, u[i], G / 2);  // the dim HALF away
    const bool lower = d0 < HALF;
    const int dr = lower ? d0 : d0 - HALF;  // rotation index of dims dr .. dr+3
    const float4* cs4 = reinterpret_cast<const float4*>(q.rope) +
                        (static_cast<size_t>(tp.pos >> 5) * (HALF / 2) + dr / 2) * 32 + (tp.pos & 31);
    const float4 c01 = __ldg(cs4), c23 = __ldg(cs4 + 32);
    const float cx[4] = {c01.x, c01.z, c23.x, c23.z};
    const float sy[4] = {c01.y, c01.w, c23.y, c23.w};
    if (!is_v) {  // v is cached raw
#pragma unroll
      for (int i = 0; i < 4; ++i) y[i] = lower ? u[i] * cx[i] - o4[i] * sy[i] : u[i] * cx[i] + o4[i] * sy[i];
    }
  }
  if (col0 >= p.N) return;  // a 64-dim head past the last feature (its weights were zero fill)
  if (is_q) {
    if (tp.prefill) {  // bf16 high part to the QKV buffer, bf16 low part to q_lo
      __nv_bfloat16* qhi = reinterpret_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(t) * p.ldo + col0 + d0;
      __nv_bfloat16* qlo = reinterpret_cast<__nv_bfloat16*>(q.q_lo) + static_cast<size_t>(t) * q.n * q.nq_l * HD +
                           (static_cast<size_t>(r) * q.nq_l + sh) * HD + d0;
      float lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) lo[i] = y[i] - bf2f(f2bf(y[i]));
      *reinterpret_cast<uint2*>(qhi) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
      *reinterpret_cast<uint2*>(qlo) = make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
    } else {  // fp16 (decode attention runs in fp32)
      __half* q16 = reinterpret_cast<__half*>(p.out) + static_cast<size_t>(t) * p.ldo + col0 + d0;
      *reinterpret_cast<uint2*>(q16) = make_uint2(pack_f16x2(y[0], y[1], sat), pack_f16x2(y[2], y[3], sat));
    }
    return;
  }
  const int g = is_v ? sh - q.nq_l - q.nkv_l : sh - q.nq_l;
  __nv_bfloat16* dst = kv + kv_row(q.kvm, q.nkv_l, r, is_v ? 1 : 0, tp.blk, g, tp.brow) * HD + d0;
  *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
}

// One token row t of a swapped tile (features f0 .. f0+127; this lane: f0 + 4 lane ..).
template <int EPI>
__device__ __forceinline__ void swap_row(const GemmParams& p, int t, int f0, int lane, float4 v, uint32_t& sat) {
  if constexpr (EPI == EPI_RESID) {  // residual += row (fp32, in place)
    const int f = f0 + 4 * lane;
    float* o = reinterpret_cast<float*>(p.out) + static_cast<size_t>(t) * p.ldo + f;
    if (f + 4 <= p.out_cols) {
      float4 x = *reinterpret_cast<float4*>(o);
      x.x += v.x; x.y += v.y; x.z += v.z; x.w += v.w;
      *reinterpret_cast<float4*>(o) = x;
    } else {
      const float vv[4] = {v.x, v.y, v.z, v.w};
      for (int i = 0; i < 4; ++i)
        if (f + i < p.out_cols) o[i] += vv[i];
    }
  } else if constexpr (EPI == EPI_STORE) {
    const int f = f0 + 4 * lane;
    __half* o = reinterpret_cast<__half*>(p.out) + static_cast<size_t>(t) * p.ldo + f;
    if (f + 4 <= p.out_cols) {
      *reinterpret_cast<uint2*>(o) = make_uint2(pack_f16x2(v.x, v.y, sat), pack_f16x2(v.z, v.w, sat));
    } else {
      const float vv[4] = {v.x, v.y, v.z, v.w};
      for (int i = 0; i < 4; ++i)
        if (f + i < p.out_cols) o[i] = to_f16(vv[i], sat);
    }
  } else if constexpr (EPI == EPI_SILU) {
    // tile rows 0..63 are gate rows, 64..127 the matching up rows: lane l < 16 pairs
    // with lane l + 16 and writes 4 of the 64 outputs
    float4 u;
    u.x = __shfl_xor_sync(0xffffffffu, v.x, 16);
    u.y = __shfl_xor_sync(0xffffffffu, v.y, 16);
    u.z = __shfl_xor_sync(0xffffffffu, v.z, 16);
    u.w = __shfl_xor_sync(0xffffffffu, v.w, 16);
    if (lane < 16) {
      const int fo = f0 / 2 + 4 * lane;
      __half* o = reinterpret_cast<__half*>(p.out) + static_cast<size_t>(t) * p.ldo + fo;
      const float a0 = silu_f(v.x) * u.x, a1 = silu_f(v.y) * u.y, a2 = silu_f(v.z) * u.z, a3 = silu_f(v.w) * u.w;
      if (fo + 4 <= p.out_cols) {
        *reinterpret_cast<uint2*>(o) = make_uint2(pack_f16x2(a0, a1, sat), pack_f16x2(a2, a3, sat));
      } else {
        const float aa[4] = {a0, a1, a2, a3};
        for (int i = 0; i < 4; ++i)
          if (fo + i < p.out_cols) o[i] = to_f16(aa[i], sat);
      }
    }
  }
}

// The q/k/v heads of one token row of a swapped QKV tile (warp-uniform token).
__device__ __forceinline__ void swap_qkv_row(const GemmParams& p, int t, const TokPos& tp, int f0, int lane,
                                             float4 v, uint32_t& sat) {
  if (f0 >= p.N) return;
  if (p.qkv.hd == 128) {
    qkv_row_group<128>(p, t, tp, f0, lane, v, sat);
  } else {  // two 64-dim heads per tile: lanes 0..15 and 16..31
    qkv_row_group<64>(p, t, tp, f0 + (lane >> 4) * 64, lane & 15, v, sat);
  }
}

template <int BN, int EPI>
__device__ __forceinline__ void swap_epilogue(const GemmParams& p, uint32_t tmem, int warp, int lane, int units,
                                              volatile int* abort_flag, volatile int* last_flag, float* sRow,
                                              int* sPos, uint32_t bar0, int stages) {
  const int q = warp & 3;         // TMEM lane quarter
  const int wq = warp - 2;        // 0..3 for the token rows
  const int row = q * 32 + lane;  // feature row of the tile
  const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
  const uint32_t tfull0 = bar0 + 8u * (2 * stages), tempty0 = bar0 + 8u * (2 * stages + 2);
  uint32_t sat = 0;  // an fp16 output clamped to the fp16 range (reported at the end)
  // every unit covers the same tokens (one token tile): their deferred-RMSNorm
  // row scales once (sInv: [BN], after the [4][BN] position table)
  float* sInv = reinterpret_cast<float*>(sPos + 256);
  if constexpr (EPI == EPI_QKV || EPI == EPI_SILU) {
    const int et = threadIdx.x - 64;
    if (et < BN) sInv[et] = et < p.T ? row_scale(p, et) : 0.0f;
    if constexpr (EPI == EPI_SILU) named_bar_sync(1, 128);
  }
  if constexpr (EPI == EPI_QKV) {
    // every unit covers the same tokens (one token tile): their positions once, in
    // parallel (sPos: [BN] position, [BN] cache block, [BN] row in the block, [BN]
    // flags 1 = valid, 2 = prefill)
    const int et = threadIdx.x - 64;
    if (et < BN) {
      TokPos tp{0, 0, 0, false, false};
      if (et < p.T) {
        tp = token_position(p.qkv, et);
        if (!tp.ok) raise_flag(p.status, TP_DEVFLAG_BAD_TOKEN);
      }
      sPos[et] = tp.pos;
      sPos[BN + et] = tp.blk;
      sPos[2 * BN + et] = tp.brow;
      sPos[3 * BN + et] = (tp.ok ? 1 : 0) | (tp.prefill ? 2 : 0);
    }
    named_bar_sync(1, 128);
  }
  int seg = 0;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const Unit un = unit_of(p, u);
    const int f0 = un.tf * 128;
    float acc[BN];
#pragma unroll
    for (int i = 0; i < BN; ++i) acc[i] = 0.0f;
    bool ok = true;
    for (int g = un.g0; g < un.g1;) {  // one accumulator use per rank segment, in rank order
      g = min(un.g1, (g / p.kb_seg + 1) * p.kb_seg);
      const int b = seg & 1;
      const uint32_t use = (seg >> 1) & 1;
      if (!warp_all(mbar_wait(tfull0 + 8u * b, use, abort_flag, p.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t ta = lane_addr + static_cast<uint32_t>(b * GemmCfg<BN, EPI, true, true>::TM_STRIDE);
      if constexpr (BN == 16) {
        float v[16];
        tc_ld16(ta, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] += v[i];
      } else {
#pragma unroll
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tc_ld32(ta + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[c * 32 + i] += v[i];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty0 + 8u * b);
      ++seg;
    }
    // every epilogue thread takes the same path from here (named barriers follow)
    if (!named_bar_and(1, 128, ok)) {
      if (threadIdx.x == 64) drain_split_counters(p, u, units, gridDim.x, 1, 0);
      break;
    }
    if (p.splits > 1) {
      const int tile = un.tt * p.tiles_f + un.tf;
      float* part = p.partials + (static_cast<size_t>(tile) * p.splits + un.split) * (BN * 128);
#pragma unroll
      for (int t = 0; t < BN; ++t) part[t * 128 + row] = acc[t];
      __threadfence();
      named_bar_sync(1, 128);
      if (threadIdx.x == 64) {
        const int old = atomicAdd(p.counters + tile, 1);
        *last_flag = (old == p.splits - 1) ? 1 : 0;
      }
      named_bar_sync(1, 128);
      if (*last_flag == 0) continue;
      __threadfence();
      const float* base = p.partials + static_cast<size_t>(tile) * p.splits * (BN * 128);
#pragma unroll
      for (int t = 0; t < BN; ++t) acc[t] = __ldcg(base + t * 128 + row);
      for (int sp = 1; sp < p.splits; ++sp) {
        const float* ps = base + static_cast<size_t>(sp) * (BN * 128);
#pragma unroll
        for (int t = 0; t < BN; ++t) acc[t] += __ldcg(ps + t * 128 + row);
      }
      if (threadIdx.x == 64) p.counters[tile] = 0;
    }
#pragma unroll
    for (int t = 0; t < BN; ++t) sRow[t * 128 + row] = acc[t];
    named_bar_sync(1, 128);
    const int nt = min(BN, p.T - un.tt * BN);
    if constexpr (EPI == EPI_RESID) {
      // residual rows: all of this warp's loads first, then the adds and stores
      // (with row_ss_out: also the fp16 row and the 32-column sums of squares the
      // next norm reads; lanes 8g .. 8g+7 hold the 32 features of group g)
      constexpr int TPW = BN / 4;
      const int f = f0 + 4 * lane;
      const bool stats = p.row_ss_out != nullptr;
      if (f0 + 128 <= p.out_cols) {  // uniform: the whole feature tile is inside
        float4 x[TPW];
#pragma unroll
        for (int k = 0; k < TPW; ++k) {
          const int t = wq + 4 * k;
          if (t < nt) x[k] = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.out) +
                                                              static_cast<size_t>(un.tt * BN + t) * p.ldo + f);
        }
#pragma unroll
        for (int k = 0; k < TPW; ++k) {
          const int t = wq + 4 * k;
          if (t < nt) {  // uniform over the warp
            const float4 v = *reinterpret_cast<const float4*>(sRow + t * 128 + 4 * lane);
            float4 y = x[k];
            y.x += v.x; y.y += v.y; y.z += v.z; y.w += v.w;
            const size_t tok = static_cast<size_t>(un.tt * BN + t);
            *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + tok * p.ldo + f) = y;
            if (stats) {
              *reinterpret_cast<uint2*>(p.row_out16 + tok * p.out_cols + f) =
                  make_uint2(pack_f16x2(y.x, y.y, sat), pack_f16x2(y.z, y.w, sat));
              float s = y.x * y.x + y.y * y.y + y.z * y.z + y.w * y.w;
              s += __shfl_xor_sync(0xffffffffu, s, 1);
              s += __shfl_xor_sync(0xffffffffu, s, 2);
              s += __shfl_xor_sync(0xffffffffu, s, 4);
              if ((lane & 7) == 0) p.row_ss_out[tok * p.row_ss_out_groups + f / 32] = s;
            }
          }
        }
      } else {  // the last, partial feature tile
        for (int t = wq; t < nt; t += 4) {
          const float4 v = *reinterpret_cast<const float4*>(sRow + t * 128 + 4 * lane);
          const float vv[4] = {v.x, v.y, v.z, v.w};
          const size_t tok = static_cast<size_t>(un.tt * BN + t);
          float* o = reinterpret_cast<float*>(p.out) + tok * p.ldo;
          float s = 0.0f;
          for (int i = 0; i < 4; ++i) {
            if (f + i < p.out_cols) {
              const float y = o[f + i] + vv[i];
              o[f + i] = y;
              if (stats) {
                p.row_out16[tok * p.out_cols + f + i] = to_f16(y, sat);
                s += y * y;
              }
            }
          }
          if (stats) {  // uniform
            s += __shfl_xor_sync(0xffffffffu, s, 1);
            s += __shfl_xor_sync(0xffffffffu, s, 2);
            s += __shfl_xor_sync(0xffffffffu, s, 4);
            if ((lane & 7) == 0 && f < p.out_cols) p.row_ss_out[tok * p.row_ss_out_groups + f / 32] = s;
          }
        }
      }
    } else {
      for (int t = wq; t < nt; t += 4) {
        float4 v = *reinterpret_cast<const float4*>(sRow + t * 128 + 4 * lane);
        if constexpr (EPI == EPI_QKV || EPI == EPI_SILU) {
          const float ri = sInv[t];
          v.x *= ri;
          v.y *= ri;
          v.z *= ri;
          v.w *= ri;
        }
        if constexpr (EPI == EPI_QKV) {
          const int fl = sPos[3 * BN + t];
          TokPos tp;
          tp.pos = sPos[t];
          tp.blk = sPos[BN + t];
          tp.brow = sPos[2 * BN + t];
          tp.ok = (fl & 1) != 0;
          tp.prefill = (fl & 2) != 0;
          if (tp.ok) swap_qkv_row(p, un.tt * BN + t, tp, f0, lane, v, sat);
        } else {
          swap_row<EPI>(p, un.tt * BN + t, f0, lane, v, sat);
        }
      }
    }
    named_bar_sync(1, 128);  // the staging rows are reused by the next unit
  }
  report_sat(p.status, sat);
}

template <int BN, int EPI, bool ACC, bool SWAP, bool PAIR, bool XCH>
__global__ void __launch_bounds__(GemmCfg<BN, EPI, ACC, SWAP, PAIR, XCH>::THREADS, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const __grid_constant__ CUtensorMap tmO, const __grid_constant__ CUtensorMap tmO2,
                   const __grid_constant__ CUtensorMap tmKV, const GemmParams p) {
  using C = GemmCfg<BN, EPI, ACC, SWAP, PAIR, XCH>;
  constexpr int STAGES = C::STAGES;
  static_assert(!PAIR || (!SWAP && EPI != EPI_ARGMAX), "CTA pairs: token tiles only");
  // rank in the cluster; a pair is ranks 2k and 2k + 1, the even one (its leader)
  // issuing the MMAs for both; 0 without pairs
  const uint32_t crank = PAIR ? cluster_ctarank() : 0u;
  const uint32_t prank = crank & 1u, lead = crank & ~1u;
  // a pair takes every unit its cluster index selects (both CTAs the same units);
  // with the exchange, pair k of a cluster takes split k of the cluster's tile
  const int u0 = XCH ? static_cast<int>(blockIdx.x) / 4 * 2 + static_cast<int>(crank >> 1)
                     : static_cast<int>(blockIdx.x) / C::CL;
  const int ustep = XCH ? static_cast<int>(gridDim.x) / 4 * 2 : static_cast<int>(gridDim.x) / C::CL;
  const uint16_t pmask = static_cast<uint16_t>(3u << lead);  // this pair's CTAs (multicast commits)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * C::A_BYTES;
  uint8_t* sOut = smem + STAGES * C::STAGE_BYTES;  // [EW][4096] output staging boxes, then [EW][2048] fp16 boxes
  float* sRow = reinterpret_cast<float*>(sOut + C::OUT_BYTES);  // [BN][128] token rows (swapped epilogues)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + C::OUT_BYTES + C::TROW_BYTES);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::NUM_BARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  // small area: the swapped epilogues' token table (red_v, reused as sPos / sInv),
  // or the weight-streaming argmax's 64-bit keys: [4 warps][BN] per-tile column
  // maxima (wkey) and [BN] per-token running maxima (bestk)
  uint8_t* small = reinterpret_cast<uint8_t*>(tmem_slot + 16);
  float* red_v = reinterpret_cast<float*>(small);
  unsigned long long* wkey = reinterpret_cast<unsigned long long*>(small);
  unsigned long long* bestk = wkey + 4 * BN;
  uint32_t* transp = reinterpret_cast<uint32_t*>(bestk + BN);  // [4 warps][32][33]
  // QKV_PAIR: [2][128] q/k norm weights, 128-byte aligned (the staging rows below take 16-byte accesses)
  float* sNw = reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(small + (C::SMALL_BYTES - 64)) + 127) &
                                        ~uintptr_t(127));
  float* sSS = sNw + 256;                                    // QKV_PAIR: partial sums of squares
  uint8_t* sStg = reinterpret_cast<uint8_t*>(sSS + 2 * 2 * (BN / 64) * 128);  // QKV_PAIR: [EW][2][32][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t bar0 = smem_u32(bars);
#define FULL(s) (bar0 + 8u * (s))
#define EMPTY(s) (bar0 + 8u * (STAGES + (s)))
#define TFULL(b) (bar0 + 8u * (2 * STAGES + (b)))
#define TEMPTY(b) (bar0 + 8u * (2 * STAGES + 2 + (b)))
#define DRAIN (bar0 + 8u * (2 * STAGES + 4))
#define QFULL(k) (bar0 + 8u * (2 * STAGES + 5 + (k)))
#define QEMPTY(k) (bar0 + 8u * (2 * STAGES + 5 + C::QUEUE + (k)))
#define PRO (bar0 + 8u * (2 * STAGES + 5 + 2 * C::QUEUE))
#define XRDY (bar0 + 8u * (2 * STAGES + 6 + 2 * C::QUEUE))
#define XFULL (bar0 + 8u * (2 * STAGES + 7 + 2 * C::QUEUE))
  volatile int* queue = reinterpret_cast<volatile int*>(tmem_slot + 4);  // [QUEUE] tile ids
  // an epilogue warp hands an accumulator back to the MMA issuer (a pair's leader)
  auto tempty_arrive = [&](uint32_t bar) {
    if constexpr (PAIR) mbar_arrive_cluster(mapa_shared(bar, lead));
    else mbar_arrive(bar);
  };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(TFULL(b), 1);
      mbar_init(TEMPTY(b), PAIR ? 2 * C::EW : C::EW);  // a pair's leader counts both CTAs' epilogue warps
    }
    mbar_init(DRAIN, 1);
    for (int k = 0; k < C::QUEUE; ++k) {
      mbar_init(QFULL(k), 1);
      mbar_init(QEMPTY(k), 5);  // the MMA thread and the 4 epilogue warps
    }
    mbar_init(PRO, 1);
    mbar_init(XRDY, 1);                  // the other pair's CTA: its stage memory is free
    mbar_init(XFULL, XCH ? 32 * C::EW : 1);  // its epilogue threads: their columns are here
    *abort_flag = 0;
    *last_flag = 0;
    fence_barrier_init();
  }
  if (SWAP && EPI == EPI_ARGMAX && threadIdx.x >= 64)
    for (int i = threadIdx.x - 64; i < BN; i += blockDim.x - 64) bestk[i] = 0ull;  // below every key
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  // a pair's barriers are initialised in both CTAs before either signals the other's
  if constexpr (PAIR) cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int units = p.tiles_t * p.tiles_f * p.splits;
  // The set-up above overlaps the previous kernel; inputs, counters and outputs
  // come after it.  The producer waits on its own, after issuing its first weight
  // tiles (constant data), so their latency hides behind the previous kernel.
  if (warp != 0) {
    griddep_wait();
    griddep_launch();
  }
  if (threadIdx.x >= 64) {  // dead intermediates out of L2, no write-back
    // after the producer's first loads are out (the discards would queue ahead of them)
    if (mbar_wait(PRO, 0, abort_flag, p.status)) {
      const int64_t nthr = static_cast<int64_t>(gridDim.x) * (blockDim.x - 64);
      const int64_t me = static_cast<int64_t>(blockIdx.x) * (blockDim.x - 64) + (threadIdx.x - 64);
      for (int k = 0; k < 2; ++k)
        for (int64_t i = me; i < p.discard_lines[k]; i += nthr) l2_discard(static_cast<const char*>(p.discard[k]) + i * 128);
    }
  }
  // tile extents on the token and feature sides
  constexpr int TM_T = C::TM_T;         // tokens per tile
  constexpr int TM_F = SWAP ? 128 : BN;  // features per tile

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      // Weight-streaming path: tiles are handed out dynamically (first wave by
      // CTA index, then an atomic counter), so SMs that stream faster take more
      // tiles; each tile id goes through a small queue to the MMA and epilogue
      // warps, -1 ends it.  Otherwise a static round-robin over the tiles.
      int qk = 0;
      // one K block of unit un into stage s: the X part, the W part or both
      auto load = [&](const Unit& un, int g, int s, bool x_part, bool w_part) {
        const int r = g / p.kb_seg, kb = g - r * p.kb_seg;
        // this CTA's token rows and (pairs) its half of the tile's weight rows
        const int t0 = un.tt * TM_T + static_cast<int>(prank) * 128;
        const int f0 = un.tf * TM_F + static_cast<int>(prank) * (BN / 2);
        const uint32_t xdst = smem_u32(SWAP ? sB + s * C::B_BYTES : sA + s * C::A_BYTES);
        const uint32_t wdst = smem_u32(SWAP ? sA + s * C::A_BYTES : sB + s * C::B_BYTES);
        if constexpr (PAIR) {
          // both CTAs' loads complete on the leader's full barrier, which expects both
          const uint32_t cbar = mapa_shared(FULL(s), lead);
          if (x_part) tma_load_2d_pair(xdst, &tmX, cbar, r * p.x_k_seg + kb * 64, t0);
          if (w_part) tma_load_2d_pair(wdst, &tmW, cbar, kb * 64, r * p.w_row_seg + f0);
        } else {
          if (x_part) tma_load_2d(xdst, &tmX, FULL(s), r * p.x_k_seg + kb * 64, t0);
          if (w_part) tma_load_2d(wdst, &tmW, FULL(s), kb * 64, r * p.w_row_seg + f0);
        }
      };
      auto expect = [&](int s) {
        if constexpr (PAIR) {
          if (prank == 0) mbar_arrive_expect_tx(FULL(s), 2 * C::STAGE_BYTES);
        } else {
          mbar_arrive_expect_tx(FULL(s), C::STAGE_BYTES);
        }
      };
      // The first unit's first stages (all free): weight tiles before the previous
      // kernel has finished, the X tiles once its outputs are visible.
      int npre = 0;
      Unit un0{};
      if (u0 < units) {
        un0 = unit_of(p, u0);
        npre = min(STAGES, un0.g1 - un0.g0);
        for (int i = 0; i < npre; ++i) {
          expect(i);
          load(un0, un0.g0 + i, i, false, true);
        }
      }
      griddep_wait();
      griddep_launch();
      for (int i = 0; i < npre; ++i) load(un0, un0.g0 + i, i, true, false);
      mbar_arrive(PRO);
      for (int u = u0; ok && (C::DYN || u < units);) {
        if constexpr (C::DYN) {
          const int id = u < units ? u : -1;
          if (!mbar_wait(QEMPTY(qk % C::QUEUE), ((qk / C::QUEUE) & 1) ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          queue[qk % C::QUEUE] = id;
          mbar_arrive(QFULL(qk % C::QUEUE));
          ++qk;
          if (id < 0) break;
        }
        const Unit un = unit_of(p, u);
        for (int g = un.g0; g < un.g1; ++g) {
          if (it >= npre) {  // the first npre K blocks (of unit u0) were issued above
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            if (!mbar_wait(EMPTY(s), ph ^ 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            expect(s);
            load(un, g, s, true, true);
          }
          ++it;
        }
        if constexpr (C::DYN) u = static_cast<int>(gridDim.x) + atomicAdd(p.sched_counter, 1);
        else u += ustep;
      }
      // every load issued has landed before the CTA may exit (a pair's loads land on
      // the leader's barriers: the leader waits for both CTAs', and the peer stays
      // until the final cluster barrier, which the leader reaches after this)
      if (prank == 0)
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
          mbar_wait(FULL(j % STAGES), (j / STAGES) & 1, nullptr, p.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer (a pair's leader issues for both CTAs) ----------------
    if (lane == 0 && prank == 0) {
      const uint32_t idesc = idesc_f16_f32(PAIR ? 256 : 128, BN);
      int it = 0, seg = 0, qk = 0;
      bool ok = true;
      for (int u = u0; ok && (C::DYN || u < units); u += ustep) {
        if constexpr (C::DYN) {
          if (!mbar_wait(QFULL(qk % C::QUEUE), (qk / C::QUEUE) & 1, abort_flag, p.status)) break;
          u = queue[qk % C::QUEUE];
          mbar_arrive(QEMPTY(qk % C::QUEUE));
          ++qk;
          if (u < 0) break;
        }
        const Unit un = unit_of(p, u);
        for (int g = un.g0; ok && g < un.g1;) {
          const int gend = min(un.g1, (g / p.kb_seg + 1) * p.kb_seg);
          const int b = seg & 1;
          const uint32_t use = (seg >> 1) & 1;
          if (!mbar_wait(TEMPTY(b), use ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d = tmem + static_cast<uint32_t>(b * C::TM_STRIDE);
          const int gs = g;
          for (; g < gend; ++g) {
            const int s = it % STAGES;
            const uint32_t ph = (it / STAGES) & 1;
            if (!mbar_wait(FULL(s), ph, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t ad = sdesc_k_sw128(smem_u32(sA + s * C::A_BYTES));
            const uint64_t bd = sdesc_k_sw128(smem_u32(sB + s * C::B_BYTES));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
            {
              if constexpr (PAIR) tc_mma_f16_pair(d, ad + 2ull * kk, bd + 2ull * kk, idesc, (g > gs || kk > 0) ? 1u : 0u);
              else tc_mma_f16(d, ad + 2ull * kk, bd + 2ull * kk, idesc, (g > gs || kk > 0) ? 1u : 0u);
            }
            if constexpr (PAIR) tc_commit_pair_mc(EMPTY(s), pmask);  // frees the stage in both CTAs
            else tc_commit(EMPTY(s));
            ++it;
          }
          if (!ok) break;
          if constexpr (PAIR) tc_commit_pair_mc(TFULL(b), pmask);  // both CTAs' epilogues
          else tc_commit(TFULL(b));
          ++seg;
        }
      }
      if constexpr (PAIR) tc_commit_pair_local(DRAIN);
      else tc_commit(DRAIN);
      mbar_wait(DRAIN, 0, nullptr, p.status);
    }
  } else if constexpr (SWAP && EPI != EPI_ARGMAX) {
    // ---------------- epilogue, weights on the M side, few tokens ----------------
    // token positions: the argmax scratch area is free here (3 x 64 ints)
    swap_epilogue<BN, EPI>(p, tmem, warp, lane, units, abort_flag, last_flag, sRow, reinterpret_cast<int*>(red_v),
                           bar0, STAGES);
  } else if constexpr (SWAP) {
    // ---------------- epilogue, weights on the M side: argmax over features ----------------
    static_assert(EPI == EPI_ARGMAX && !ACC, "weight-streaming path implements the argmax epilogue");
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int et = threadIdx.x - 64;  // epilogue thread 0..127
    int seg = 0, qk = 0;
    bool ok = true;
    for (;;) {
      ok = mbar_wait(QFULL(qk % C::QUEUE), (qk / C::QUEUE) & 1, abort_flag, p.status);
      if (!named_bar_and(1, 128, ok)) break;
      const int u = queue[qk % C::QUEUE];
      __syncwarp();
      if (lane == 0) mbar_arrive(QEMPTY(qk % C::QUEUE));
      ++qk;
      if (u < 0) break;  // uniform: every epilogue thread read the same id
      const Unit un = unit_of(p, u);
      const int f = un.tf * 128 + row;
      const int t0 = un.tt * BN;
      const bool f_ok = f < p.vocab;
      const int b = seg & 1;
      const uint32_t use = (seg >> 1) & 1;
      ok = mbar_wait(TFULL(b), use, abort_flag, p.status);
      if (!named_bar_and(1, 128, ok)) break;
      tc_fence_after();
      // Each warp reduces every token column of the tile over its 32 vocab rows.
      // A 32 x 32 block (rows = lanes, columns = tokens) of order-preserving keys
      // (amax_key's high word) goes through a padded shared-memory buffer, so that
      // lane l then scans column c0 + l down the 32 rows (strictly greater keeps
      // the lowest row, the lowest vocab index, on ties).  No barrier inside the
      // tile: the 4 warps meet once, after the accumulator has been handed back.
      uint32_t* tb = transp + q * (32 * 33);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        if constexpr (BN == 16) {
          float v16[16];
          tc_ld16(lane_addr + static_cast<uint32_t>(b * C::TM_STRIDE), v16);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = i < 16 ? v16[i] : 0.0f;
        } else {
          tc_ld32(lane_addr + static_cast<uint32_t>(b * C::TM_STRIDE + c0), v);
        }
        const int ncol = min(min(32, BN), p.T - (t0 + c0));  // valid token columns (warp-uniform)
        if (p.logits && f_ok) {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i < ncol) p.logits[static_cast<size_t>(t0 + c0 + i) * p.ld_logits + f] = v[i];
        }
#pragma unroll
        for (int i = 0; i < (BN < 32 ? BN : 32); ++i)  // 0: no row (every key of a row is above 0)
          tb[i * 33 + lane] = f_ok ? static_cast<uint32_t>(amax_key(v[i], 0) >> 32) : 0u;
        __syncwarp();
        uint32_t mkey = 0u, mlane = 0u;
#pragma unroll
        for (int r = 0; r < 32; ++r) {
          const uint32_t k = tb[lane * 33 + r];
          if (k > mkey) {
            mkey = k;
            mlane = static_cast<uint32_t>(r);
          }
        }
        __syncwarp();  // the buffer is rewritten by the next block
        if (c0 + lane < BN) {
          const uint32_t fw = static_cast<uint32_t>(un.tf * 128 + q * 32) + mlane;
          wkey[q * BN + c0 + lane] =
              mkey == 0u ? 0ull : ((static_cast<unsigned long long>(mkey) << 32) | static_cast<unsigned long long>(~fw));
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(TEMPTY(b));
      ++seg;
      named_bar_sync(1, 128);
      for (int c = et; c < BN && t0 + c < p.T; c += 128) {
        unsigned long long k = bestk[c];
#pragma unroll
        for (int w = 0; w < 4; ++w) k = max(k, wkey[w * BN + c]);
        bestk[c] = k;
      }
      named_bar_sync(1, 128);  // wkey is rewritten by the next tile
    }
    // Each CTA folds its per-token best into one 64-bit key per token with
    // atomicMax (key order = torch.argmax order); the last CTA to finish reads the
    // keys back, writes the ids and clears the keys for the next launch.  A CTA
    // whose wait gave up (TP_DEVFLAG_TIMEOUT is set, the ids are not valid) adds
    // no key but still counts itself in, so the counters and keys always return
    // to zero for the next launch.
    {
      const bool all_ok = named_bar_and(1, 128, ok);
      if (all_ok)
        for (int t = et; t < p.T; t += 128)
          if (bestk[t] != 0ull) atomicMax(p.amax_keys + t, bestk[t]);
      __threadfence();
      named_bar_sync(1, 128);
      if (et == 0) *last_flag = (atomicAdd(p.done_counter, 1) == static_cast<int>(gridDim.x) - 1) ? 1 : 0;
      named_bar_sync(1, 128);
      if (*last_flag) {
        __threadfence();
        for (int t = et; t < p.T; t += 128) {
          const unsigned long long k = atomicExch(p.amax_keys + t, 0ull);
          p.out_ids[t] = static_cast<int>(~static_cast<uint32_t>(k & 0xffffffffull));
        }
        if (et == 0) {  // every CTA has taken its last tile id: ready for the next launch
          *p.done_counter = 0;
          *p.sched_counter = 0;
        }
      }
    }
  } else if constexpr (XCH) {
    // ---------------- epilogue of the K-split exchange (warps 2..9) ----------------
    // This CTA's 128 rows of the 256 x 256 tile, its split's K half complete in
    // TMEM buffer 0.  Split `me` finishes columns [128 me, 128 me + 128) and sends
    // the other 128 to the other pair's CTA of the same rows (cluster rank ^ 2),
    // into that CTA's stage memory once the MMAs reading it are done: fp32,
    // [32 column groups of 4][128 rows][4], so a warp's 16-byte stores and loads
    // are contiguous.  The two warps of a lane quarter take 64 columns each.
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int ws = (warp - 2) >> 2;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    uint8_t* box = sOut + (warp - 2) * (C::NXB * 4096 + 2048);
    uint8_t* box16 = box + C::NXB * 4096;
    uint32_t sat = 0;
    const int me = static_cast<int>(crank >> 1);
    const uint32_t peer = crank ^ 2u;
    const int fin = me * 128 + ws * 64;        // this thread's finished columns
    const int snd = (1 - me) * 128 + ws * 64;  // and the ones it sends
    const uint32_t rbuf = smem_u32(smem);
    if (u0 < units) {
      const Unit un = unit_of(p, u0);
      const int t = un.tt * C::TM_T + static_cast<int>(prank) * 128 + row;
      const int tbox = un.tt * C::TM_T + static_cast<int>(prank) * 128 + q * 32;
      const int f0 = un.tf * BN;
      const bool row_ok = t < p.T;
      if (p.row_ss_out != nullptr) {  // old residual of the first finished chunks, while the MMA runs
#pragma unroll
        for (int k = 0; k < C::NXB; ++k) prefetch_rows32(p, box + k * 4096, t, row_ok, f0 + fin + 32 * k, lane);
      }
      bool ok = warp_all(mbar_wait(TFULL(0), 0, abort_flag, p.status));
      // this pair's MMAs are done: this CTA's stage memory may take the peer's columns
      if (ok && threadIdx.x == 64) mbar_arrive_cluster(mapa_shared(XRDY, peer));
      ok = ok && warp_all(mbar_wait_cl(XRDY, 0, abort_flag, p.status));
      tc_fence_after();
      if (ok) {
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          float v[32];
          tc_ld32(lane_addr + static_cast<uint32_t>(snd + 32 * c), v);
          const int cg0 = (ws * 64 + 32 * c) >> 2;  // the peer's column group of v[0]
#pragma unroll
          for (int k = 0; k < 8; ++k)
            st_cluster_v4(mapa_shared(rbuf + static_cast<uint32_t>(((cg0 + k) * 128 + row) * 16), peer), v[4 * k],
                          v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
      }
      // every epilogue thread arrives (after a failure too, so that the peer's bounded wait ends)
      mbar_arrive_cluster(mapa_shared(XFULL, peer));
      ok = ok && warp_all(mbar_wait_cl(XFULL, 0, abort_flag, p.status));
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          float v[32];
          tc_ld32(lane_addr + static_cast<uint32_t>(fin + 32 * c), v);
          const int cg0 = (ws * 64 + 32 * c) >> 2;
          const float* rb = reinterpret_cast<const float*>(smem);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 o = *reinterpret_cast<const float4*>(rb + ((cg0 + k) * 128 + row) * 4);
            // split 0's half plus split 1's (the rank order at tp 2)
            v[4 * k] = me == 0 ? v[4 * k] + o.x : o.x + v[4 * k];
            v[4 * k + 1] = me == 0 ? v[4 * k + 1] + o.y : o.y + v[4 * k + 1];
            v[4 * k + 2] = me == 0 ? v[4 * k + 2] + o.z : o.z + v[4 * k + 2];
            v[4 * k + 3] = me == 0 ? v[4 * k + 3] + o.w : o.w + v[4 * k + 3];
          }
          if (p.row_ss_out != nullptr) {  // uniform: read-add-store and the next norm's inputs
            if (c == 0) cp_async_wait_all();
            resid_rows32<C>(p, &tmO, &tmO2, c < C::NXB ? box + c * 4096 : box, box16, t, row_ok, f0 + fin + 32 * c,
                            tbox, lane, v, c < C::NXB, sat);
          } else {
            box_acquire(lane);
            stage_f32x32(box, lane, v);
            box_release(&tmO, box, f0 + fin + 32 * c, tbox, true, lane);
          }
        }
      }
    }
    report_sat(p.status, sat);
    cp_async_wait_all();  // no copy into the staging outlives the CTA
    if (lane == 0) bulk_wait_read();
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..), tokens on the M side ----------------
    // A warp reads TMEM lanes 32*(warp % 4) .. +31 (one token row per thread);
    // with 8 epilogue warps the two warps of a lane quarter take the two halves
    // of the tile's columns (contiguous ranges that hold whole heads / whole
    // gate-up blocks), so the epilogue keeps pace with the MMA.
    constexpr int NSPLIT = C::EW / 4;
    constexpr int BNH = BN / NSPLIT;  // accumulator columns per thread
    const int q = warp & 3;
    const int cbase = ((warp - 2) >> 2) * BNH;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    // this warp's output staging box (TMA_OUT); with RESID_ROWS its NXB fp32 boxes
    // (the first is `box`) and then its fp16 row box
    uint8_t* box = sOut + (warp - 2) * (C::RESID_ROWS ? C::NXB * 4096 + 2048 : 4096);
    uint8_t* box16 = box + C::NXB * 4096;
    uint32_t sat = 0;  // an fp16 output clamped to the fp16 range (reported at the end)
    if constexpr (C::QKV_PAIR) {
      const int e = threadIdx.x - 64;
      if (e < p.qkv.hd) {
        sNw[e] = bf2f(reinterpret_cast<const __nv_bfloat16*>(p.qkv.q_norm)[e]);
        sNw[128 + e] = bf2f(reinterpret_cast<const __nv_bfloat16*>(p.qkv.k_norm)[e]);
      }
      named_bar_sync(1, 32 * C::EW);
    }
    int seg = 0;
    for (int u = u0; u < units; u += ustep) {
      const Unit un = unit_of(p, u);
      const int t = un.tt * C::TM_T + static_cast<int>(prank) * 128 + row;
      const int tbox = un.tt * C::TM_T + static_cast<int>(prank) * 128 + q * 32;  // first row of this warp's boxes
      const int f0 = un.tf * BN;
      const bool row_ok = t < p.T;
      float rinv = 1.0f;  // deferred RMSNorm of the input row (QKV, gate_up)
      if constexpr (EPI == EPI_QKV || EPI == EPI_SILU) rinv = row_ok ? row_scale(p, t) : 0.0f;
      if constexpr (C::RESID_ROWS) {  // old residual of the first chunks, copied while the MMA runs
        if (p.row_ss_out != nullptr) {
          cp_async_wait_all();  // copies of a unit this CTA did not finish (a non-last split)
          box_acquire(lane);    // the boxes' previous stores have read them
#pragma unroll
          for (int k = 0; k < C::NXB; ++k) prefetch_rows32(p, box + k * 4096, t, row_ok, f0 + cbase + 32 * k, lane);
        }
      }
      TokPos tp{0, 0, 0, false, false};
      if constexpr (EPI == EPI_QKV) {
        if (row_ok) {
          tp = token_position(p.qkv, t);
          if (!tp.ok && cbase == 0) raise_flag(p.status, TP_DEVFLAG_BAD_TOKEN);
        }
      }
      if constexpr (C::QKV_PAIR) {
        const int b = seg & 1;
        const uint32_t use = (seg >> 1) & 1;
        const uint32_t ta = lane_addr + static_cast<uint32_t>(b * C::TM_STRIDE);
        const int w = (warp - 2) >> 2;
        uint8_t* stg = sStg + (warp - 2) * (2 * 32 * 128);
        const bool ok = p.qkv.hd == 128
                            ? qkv_pair_tile<BN, 128>(p, &tmO, &tmO2, &tmKV, TFULL(b), use, abort_flag, ta, t, tp, f0,
                                                     row_ok, w, q, row, seg & 1, sNw, sSS, stg, rinv, sat)
                            : qkv_pair_tile<BN, 64>(p, &tmO, &tmO2, &tmKV, TFULL(b), use, abort_flag, ta, t, tp, f0,
                                                    row_ok, w, q, row, seg & 1, sNw, sSS, stg, rinv, sat);
        if (!ok) break;
        tc_fence_before();
        __syncwarp();
        if (lane == 0) tempty_arrive(TEMPTY(b));
        ++seg;
      } else if constexpr (!ACC) {
        const int b = seg & 1;
        const uint32_t use = (seg >> 1) & 1;
        if (!warp_all(mbar_wait(TFULL(b), use, abort_flag, p.status))) break;
        tc_fence_after();
        const uint32_t ta = lane_addr + static_cast<uint32_t>(b * C::TM_STRIDE);
        if constexpr (EPI == EPI_QKV) {
          if (BN >= 128 && p.qkv.hd == 128) {
            qkv_stream<BN, (BN >= 128 ? 128 : 64)>(p, ta, t, tp, f0, row_ok, cbase, cbase + BNH, rinv, sat);
          } else {
            qkv_stream<BN, 64>(p, ta, t, tp, f0, row_ok, cbase, cbase + BNH, rinv, sat);
          }
        } else if constexpr (EPI == EPI_SILU) {
          // gate/up interleaved in 64-column blocks: 128 accumulator columns = 64 outputs
#pragma unroll 1
          for (int qb = cbase / 128; qb < (cbase + BNH) / 128; ++qb) {
            float o[64];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              float gv[32], uv[32];
              tc_ld32(ta + qb * 128 + h * 32, gv);
              tc_ld32(ta + qb * 128 + 64 + h * 32, uv);
#pragma unroll
              for (int i = 0; i < 32; ++i) o[h * 32 + i] = silu_f(gv[i] * rinv) * (uv[i] * rinv);
            }
            box_acquire(lane);
            stage_f16x64(box, lane, o, sat);
            box_release(&tmO, box, f0 / 2 + qb * 64, tbox, false, lane);
          }
        } else if constexpr (EPI == EPI_ARGMAX) {
          float best = -INFINITY;
          int bi = -1;
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            float v[32];
            tc_ld32(ta + c * 32, v);
            if (row_ok) argmax_scan(p, t, f0 + c * 32, v, best, bi);
          }
          if (row_ok) {
            p.amax_val[static_cast<size_t>(un.tf) * p.amax_ld + t] = best;
            p.amax_idx[static_cast<size_t>(un.tf) * p.amax_ld + t] = bi < 0 ? INT_MAX : bi;
          }
        } else if constexpr (EPI == EPI_RESID) {
          // residual += this tile: TMA reduce-add of fp32 boxes (one add per element in L2)
#pragma unroll 1
          for (int c = cbase / 32; c < (cbase + BNH) / 32; ++c) {
            float v[32];
            tc_ld32(ta + c * 32, v);
            if (p.row_ss_out != nullptr) {  // uniform: read-add-store and the next norm's inputs
              const int k = c - cbase / 32;
              if (k == 0) cp_async_wait_all();
              resid_rows32<C>(p, &tmO, &tmO2, k < C::NXB ? box + k * 4096 : box, box16, t, row_ok, f0 + c * 32,
                              tbox, lane, v, k < C::NXB, sat);
            } else {
              box_acquire(lane);
              stage_f32x32(box, lane, v);
              box_release(&tmO, box, f0 + c * 32, tbox, true, lane);
            }
          }
        } else {
#pragma unroll 1
          for (int c = cbase / 64; c < (cbase + BNH) / 64; ++c) {
            float v[64];
            tc_ld32(ta + c * 64, *reinterpret_cast<float(*)[32]>(v));
            tc_ld32(ta + c * 64 + 32, *reinterpret_cast<float(*)[32]>(v + 32));
            box_acquire(lane);
            stage_f16x64(box, lane, v, sat);
            box_release(&tmO, box, f0 + c * 64, tbox, false, lane);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) tempty_arrive(TEMPTY(b));
        ++seg;
      } else {
        float acc[BNH];  // this thread's columns cbase .. cbase + BNH
#pragma unroll
        for (int i = 0; i < BNH; ++i) acc[i] = 0.0f;
        bool ok = true;
        for (int g = un.g0; g < un.g1;) {
          g = min(un.g1, (g / p.kb_seg + 1) * p.kb_seg);
          const int b = seg & 1;
          const uint32_t use = (seg >> 1) & 1;
          if (!warp_all(mbar_wait(TFULL(b), use, abort_flag, p.status))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ta = lane_addr + static_cast<uint32_t>(b * C::TM_STRIDE + cbase);
#pragma unroll
          for (int c = 0; c < BNH / 32; ++c) {
            float v[32];
            tc_ld32(ta + c * 32, v);
#pragma unroll
            for (int i = 0; i < 32; ++i) acc[c * 32 + i] += v[i];
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) tempty_arrive(TEMPTY(b));
          ++seg;
        }
        // every epilogue thread takes the same path from here (named barriers follow)
        if (!named_bar_and(1, 32 * C::EW, ok)) {
          if (threadIdx.x == 64) drain_split_counters(p, u, units, ustep, PAIR ? 2 : 1, static_cast<int>(prank));
          break;
        }
        if (p.splits > 1) {
          // a pair's CTAs each sum their own 128 rows: one partial set per CTA of the tile
          const int tile = (un.tt * p.tiles_f + un.tf) * (PAIR ? 2 : 1) + static_cast<int>(prank);
          float* part = p.partials + (static_cast<size_t>(tile) * p.splits + un.split) * (BN * 128);
          if (row_ok) {  // rows past the last token are never read
#pragma unroll
            for (int c = 0; c < BNH; ++c) part[(cbase + c) * 128 + row] = acc[c];
          }
          __threadfence();
          named_bar_sync(1, 32 * C::EW);
          if (threadIdx.x == 64) {
            const int old = atomicAdd(p.counters + tile, 1);
            *last_flag = (old == p.splits - 1) ? 1 : 0;
          }
          named_bar_sync(1, 32 * C::EW);
          const bool last = *last_flag != 0;
          if (!last) continue;
          __threadfence();
          const float* base = p.partials + static_cast<size_t>(tile) * p.splits * (BN * 128);
          if (row_ok) {
#pragma unroll
            for (int c = 0; c < BNH; ++c) acc[c] = __ldcg(base + (cbase + c) * 128 + row);
            for (int s = 1; s < p.splits; ++s) {
              const float* ps = base + static_cast<size_t>(s) * (BN * 128);
#pragma unroll
              for (int c = 0; c < BNH; ++c) acc[c] += __ldcg(ps + (cbase + c) * 128 + row);
            }
          }
          // the counter is cleared after every thread of this CTA has passed the
          // second barrier above (it is read once per tile, by thread 64)
          if (threadIdx.x == 64) p.counters[tile] = 0;
        }
        if constexpr (EPI == EPI_QKV || EPI == EPI_SILU) {
#pragma unroll
          for (int c = 0; c < BNH; ++c) acc[c] *= rinv;
        }
        if constexpr (C::TMA_OUT) {  // whole warp (rows past the last token are clipped by the TMA unit)
          if constexpr (EPI == EPI_SILU) {
#pragma unroll
            for (int qb = 0; qb < BNH / 128; ++qb) {
              float o[64];
#pragma unroll
              for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 32; ++i) o[h * 32 + i] = silu_f(acc[qb * 128 + h * 32 + i]) * acc[qb * 128 + 64 + h * 32 + i];
              box_acquire(lane);
              stage_f16x64(box, lane, o, sat);
              box_release(&tmO, box, f0 / 2 + (cbase / 128 + qb) * 64, tbox, false, lane);
            }
          } else if constexpr (EPI == EPI_RESID) {
#pragma unroll
            for (int c = 0; c < BNH / 32; ++c) {
              if (p.row_ss_out != nullptr) {  // uniform: read-add-store and the next norm's inputs
                if (c == 0) cp_async_wait_all();
                resid_rows32<C>(p, &tmO, &tmO2, c < C::NXB ? box + c * 4096 : box, box16, t, row_ok,
                                f0 + cbase + c * 32, tbox, lane, acc + c * 32, c < C::NXB, sat);
              } else {
                box_acquire(lane);
                stage_f32x32(box, lane, acc + c * 32);
                box_release(&tmO, box, f0 + cbase + c * 32, tbox, true, lane);
              }
            }
          } else {
#pragma unroll
            for (int c = 0; c < BNH / 64; ++c) {
              box_acquire(lane);
              stage_f16x64(box, lane, acc + c * 64, sat);
              box_release(&tmO, box, f0 + cbase + c * 64, tbox, false, lane);
            }
          }
        } else if (row_ok) {
          if constexpr (EPI == EPI_QKV) {
            static_assert(!ACC || C::EW == 4, "split-K QKV keeps whole heads in one thread");
            if (tp.ok) {
              if constexpr (BN >= 128) {
                if (p.qkv.hd == 128) {
#pragma unroll
                  for (int hb = 0; hb < BN / 128; ++hb)
                    if (f0 + hb * 128 < p.N) qkv_head<128>(p, t, tp, f0 + hb * 128, acc + hb * 128, sat);
                }
              }
              if (p.qkv.hd == 64) {
#pragma unroll
                for (int hb = 0; hb < BN / 64; ++hb)
                  if (f0 + hb * 64 < p.N) qkv_head<64>(p, t, tp, f0 + hb * 64, acc + hb * 64, sat);
              }
            }
          } else if constexpr (EPI == EPI_ARGMAX) {
            static_assert(C::EW == 4, "argmax keeps a whole tile row in one thread");
            float best = -INFINITY;
            int bi = -1;
#pragma unroll
            for (int c = 0; c < BN / 32; ++c) argmax_scan(p, t, f0 + c * 32, acc + c * 32, best, bi);
            p.amax_val[static_cast<size_t>(un.tf) * p.amax_ld + t] = best;
            p.amax_idx[static_cast<size_t>(un.tf) * p.amax_ld + t] = bi < 0 ? INT_MAX : bi;
          }
        }
      }
    }
    report_sat(p.status, sat);
    if constexpr (C::RESID_ROWS) cp_async_wait_all();  // no copy into the staging outlives the CTA
    // every store has read its staging before the CTA (and its shared memory) goes
    // away; the writes themselves complete on their own and are covered by the next
    // kernel's wait on this grid
    if constexpr (C::TMA_OUT || C::QKV_PAIR) {
      if (lane == 0) bulk_wait_read();
      __syncwarp();
    }
  }
#undef FULL
#undef EMPTY
#undef TFULL
#undef TEMPTY
#undef DRAIN
#undef QFULL
#undef QEMPTY
#undef PRO
#undef XRDY
#undef XFULL
  tc_fence_before();
  __syncthreads();
  // a pair: the leader's MMAs into this CTA's TMEM and shared memory, and the
  // peer's arrivals on the leader's barriers, are all done before either leaves
  if constexpr (PAIR) cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2D 16-bit row-major tensor [rows, cols] (row stride ld elements), box 64 x box_rows, 128 B swizzle.
bool make_tmap_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows, bool bf16) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * 2)};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

static bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows) {
  return make_tmap_2d(m, base, rows, cols, ld, box_rows, false);
}

// Output tensor [rows, cols] (row stride ld elements) written by the epilogue's
// TMA stores: boxes of 128 bytes x 32 rows, 128-byte swizzle.
static bool make_map_out(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld,
                         CUtensorMapDataType type, int elem_bytes) {
  auto fn = encode_fn();
  if (!fn || !base || rows <= 0 || cols <= 0) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (ld * elem_bytes) % 16) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld * elem_bytes)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elem_bytes), 32u};
  cuuint32_t estr[2] = {1u, 1u};
  return fn(m, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 16-bit [rows][cols] row-major, box box_cols columns x 32 rows, no swizzle.
static bool make_map_rows16(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int box_cols = 32) {
  auto fn = encode_fn();
  if (!fn || !base || rows <= 0 || cols <= 0) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (cols * 2) % 16) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * 2)};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), 32u};
  cuuint32_t estr[2] = {1u, 1u};
  if ((box_cols * 2) % 16) return false;
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static inline int cdiv(long long a, long long b) { return static_cast<int>((a + b - 1) / b); }

// tile width of a CTA pair (TMEM: two accumulators of BN columns per CTA): 256,
// or 128 for the rank-sum epilogue (its running sums in registers hold BN at 128)
constexpr int kPairMaxBN = 256;

// 4-CTA clusters of the exchange kernel resident at once on the current device
// (cluster placement follows the GPU's SM groups, so fewer than SMs / 4 can fit);
// 0 when the query fails.
static int xch_max_clusters() {
  static PerDevice pd;
  int dev = -1, n = 0;
  if (per_device_ready(pd, &dev, &n)) return n;
  auto kern = gemm_tc_kernel<256, EPI_RESID, true, false, true, true>;
  using Cfg = GemmCfg<256, EPI_RESID, true, false, true, true>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(4 * 64);
  cfg.blockDim = dim3(Cfg::THREADS);
  cfg.dynamicSmemBytes = Cfg::SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 4;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  per_device_mark(pd, dev, n);
  return n;
}

GemmPlan plan_gemm(const GemmProblem& pr, int num_sms) {
  GemmPlan pl{};
  const int total_kb = pr.n_seg * (pr.k_seg / 64);
  if (pr.epi == EPI_ARGMAX && pr.T <= 256) {
    // up to 256 tokens against the whole vocab: weights on the M side, tokens as N,
    // so the weights stream from HBM once
    pl.swap = true;
    pl.BN = pr.T <= 16 ? 16
            : pr.T <= 32 ? 32
            : pr.T <= 64 ? 64
            : pr.T <= 128 ? 128
            : pr.T <= 160 ? 160
            : pr.T <= 192 ? 192
                          : 256;
    pl.tiles_t = 1;
    pl.tiles_f = cdiv(pr.N, 128);
    pl.splits = 1;
    pl.acc = false;
    const int units = pl.tiles_f;
    pl.grid = units < num_sms ? units : num_sms;
    pl.partial_floats = 0;
    return pl;
  }
  const double weight_bytes = static_cast<double>(pr.N) * total_kb * 64 * 2;
  if (pr.T <= 64 && pr.epi != EPI_ARGMAX && (weight_bytes >= 24e6 || (pr.T <= 16 && weight_bytes >= 4e6))) {
    // few tokens (decode) against a large weight: weights on the M side (128-feature
    // tiles), tokens as N, K split so that tiles x splits fill the GPU; its stages
    // carry mostly weights (a token tile's carry 128 mostly empty token rows).  Up
    // to 16 tokens this wins from 4 MB of weights on (0.6B layer, one sequence:
    // 475 -> 412 us per 8-layer token); with 17-64 tokens and small weights the
    // token tiles do (their epilogues write whole rows; measured).
    pl.swap = true;
    pl.BN = pr.T <= 32 ? 32 : 64;
    pl.tiles_t = 1;
    pl.tiles_f = cdiv(pr.N, 128);
    // at least 8 K blocks per split (the last CTA of a tile adds every split's
    // partial serially) and at most 8 splits
    int splits = num_sms / pl.tiles_f;
    if (splits > total_kb / 8) splits = total_kb / 8;
    if (splits > 8) splits = 8;
    if (splits < 1) splits = 1;
    pl.splits = splits;
    pl.acc = true;
    const int units = pl.tiles_f * splits;
    pl.grid = units < num_sms ? units : num_sms;
    pl.partial_floats = splits > 1 ? static_cast<size_t>(pl.tiles_f) * splits * pl.BN * 128 : 0;
    return pl;
  }
  pl.tiles_t = cdiv(pr.T, 128);
  // tile width: wide tiles while there are enough of them to fill the GPU
  int BN;
  const int min_bn = pr.epi == EPI_QKV ? pr.qkv.hd : 64;
  if (pr.epi == EPI_ARGMAX) {
    BN = 64;  // weight streaming: small units balance the HBM-bound LM head
  } else if (pr.epi == EPI_SILU) {
    BN = (pl.tiles_t * cdiv(pr.N, 256) >= num_sms) ? 256 : 128;
  } else if (pr.n_seg == 1 && pl.tiles_t * cdiv(pr.N, 256) >= num_sms) {
    BN = 256;
  } else if (pl.tiles_t * cdiv(pr.N, 128) >= num_sms / 2) {
    BN = 128;
  } else {
    BN = 64;
  }
  if (BN < min_bn) BN = min_bn;
  pl.BN = BN;
  pl.tiles_f = cdiv(pr.N, BN);
  const int tiles = pl.tiles_t * pl.tiles_f;
  int splits = 1;
  // K splits fill the GPU when tiles are few, but each split costs a partial
  // written and re-read; a few-token GEMM with at least 32 feature tiles (QKV,
  // gate_up at decode) streams its weights faster unsplit (measured, 0.6B decode)
  const bool few_tokens_wide = pr.T <= 64 && tiles >= 32 && pr.n_seg == 1;
  if (pr.epi != EPI_ARGMAX && tiles < num_sms && !few_tokens_wide) {
    splits = num_sms / tiles;
    if (splits > total_kb / 2) splits = total_kb / 2;
    if (splits < 1) splits = 1;
  }
  // few-token row-parallel GEMMs (o_proj, down at decode): at most 4 K splits (a
  // sweep of 2 / 4 / 6 / 9 on the 0.6B layer found 4 best: fewer partials to add)
  if (pr.T <= 64 && pr.n_seg > 1 && splits > 4) splits = 4;
  pl.splits = splits;
  pl.acc = (pr.n_seg > 1) || (splits > 1);
  if (pl.acc && BN > 128) {  // running sums need BN <= 128
    pl.BN = 128;
    pl.tiles_f = cdiv(pr.N, 128);
  }
  // Residual GEMMs with one or two rank segments whose 256 x 256 tiles fit one
  // wave of 4-CTA clusters: the two pairs of a cluster take one K half each (a
  // rank segment at tp 2) and meet through distributed shared memory, no
  // partials in global memory.  A 256-wide pair tile moves its operands at
  // ~390 ns per K block against ~330 ns for the 128-wide one with the whole K.
  if (pl.splits == 1 && pr.epi == EPI_RESID && pr.T >= 256 && pr.n_seg <= 2 && total_kb % 2 == 0 &&
      total_kb >= 16) {
    const int tt2 = cdiv(pr.T, 256), tf2 = cdiv(pr.N, 256);
    const int tiles2 = tt2 * tf2;
    if (4 * tiles2 >= num_sms / 2 && tiles2 <= xch_max_clusters()) {
      pl.pair = true;
      pl.xch = true;
      pl.BN = 256;
      pl.acc = true;
      pl.splits = 2;
      pl.tiles_t = tt2;
      pl.tiles_f = tf2;
      pl.grid = 4 * tiles2;
      pl.partial_floats = 0;
      return pl;
    }
  }
  // Long-K residual (row-parallel) GEMMs on CTA pairs with 256-wide tiles and the
  // K range (the rank segments) split in two: a 256-wide pair tile moves its
  // operands at ~390 ns per K block against ~330 ns for a 128-wide one with half
  // the MMA work, and the rank-sum's running sums cap the unsplit residual tiles
  // at 128 columns.  The two halves meet in split-K partials (per CTA of the
  // pair), the last to arrive adds them in split order.  Measured: 32B down_proj
  // (1024 tokens, 400 K blocks) 370 -> 279 us; with 32 or 48 K blocks (0.6B
  // o_proj / down_proj at 2176 tokens) the partials cost more than the main loop
  // saves (22.8 -> 35.2 and 27.0 -> 37.1 us), so those keep 128-wide tiles.
  if (pl.splits == 1 && pr.epi == EPI_RESID && pr.T >= 256 && total_kb >= 256) {
    const int tt2 = cdiv(pr.T, 256), tf2 = cdiv(pr.N, 256);
    if (tt2 * tf2 * 2 >= num_sms / 4) {
      pl.pair = true;
      pl.BN = 256;
      pl.acc = true;
      pl.splits = 2;
      pl.tiles_t = tt2;
      pl.tiles_f = tf2;
      const int units = tt2 * tf2 * 2;
      const int pairs = units < num_sms / 2 ? units : num_sms / 2;
      pl.grid = 2 * pairs;
      pl.partial_floats = static_cast<size_t>(tt2) * tf2 * 2 * pl.splits * 256 * 128;
      return pl;
    }
  }
  // CTA pairs (256-token tiles, cta_group::2): unsplit token tiles with enough
  // pair tiles to keep at least half of the SM pairs busy
  if (pl.splits == 1 && (pr.epi == EPI_STORE || pr.epi == EPI_SILU || pr.epi == EPI_QKV || pr.epi == EPI_RESID) &&
      pr.T >= 256) {
    const int bn = (pl.acc || pr.epi == EPI_RESID) ? 128 : kPairMaxBN;  // the pair variants instantiated
    const int tt2 = cdiv(pr.T, 256), tf2 = cdiv(pr.N, bn);
    if (tt2 * tf2 >= num_sms / 4) {
      pl.pair = true;
      pl.BN = bn;
      pl.tiles_t = tt2;
      pl.tiles_f = tf2;
      const int pairs = tt2 * tf2 < num_sms / 2 ? tt2 * tf2 : num_sms / 2;
      pl.grid = 2 * pairs;
      pl.partial_floats = 0;
      return pl;
    }
  }
  const int units = pl.tiles_t * pl.tiles_f * pl.splits;
  pl.grid = units < num_sms ? units : num_sms;
  pl.partial_floats = pl.splits > 1 ? static_cast<size_t>(pl.tiles_t) * pl.tiles_f * pl.splits * pl.BN * 128 : 0;
  return pl;
}

int gemm_num_tiles_f(const GemmProblem& pr, const GemmPlan& plan) { return plan.tiles_f; }

template <int BN, int EPI, bool ACC, bool SWAP, bool PAIR = false, bool XCH = false>
static cudaError_t launch_variant(const CUtensorMap& mx, const CUtensorMap& mw, const GemmProblem& pr,
                                  const GemmParams& gp, int grid, cudaStream_t s) {
  auto kern = gemm_tc_kernel<BN, EPI, ACC, SWAP, PAIR, XCH>;
  using Cfg = GemmCfg<BN, EPI, ACC, SWAP, PAIR, XCH>;
  constexpr int smem = Cfg::SMEM;
  static PerDevice attr;  // per instantiation and device
  {
    const cudaError_t e = smem_attr_per_device(attr, kern, smem);
    if (e != cudaSuccess) return e;
  }
  CUtensorMap mo = mx;  // unused unless the outputs leave through TMA
  CUtensorMap mo2 = mx;  // fp16 residual rows of the residual epilogues (row_ss_out set)
  CUtensorMap mkv = mx;  // the KV cache as [rows][hd] (paired QKV epilogue)
  if constexpr (Cfg::TMA_OUT) {
    const bool ok = EPI == EPI_RESID
                        ? make_map_out(&mo, pr.out, pr.T, pr.out_cols, pr.ldo, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4)
                        : make_map_out(&mo, pr.out, pr.T, pr.out_cols, pr.ldo, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2);
    if (!ok) return cudaErrorInvalidValue;
  }
  if constexpr (Cfg::RESID_ROWS) {
    if (gp.row_ss_out && !make_map_rows16(&mo2, pr.row_out16, pr.T, pr.out_cols)) return cudaErrorInvalidValue;
  }
  if constexpr (Cfg::QKV_PAIR) {  // q rows (high / fp16 part, low part) leave through TMA
    const int qp = pr.qkv.hd / 4;
    const int64_t kv_rows =
        static_cast<int64_t>(pr.qkv.n) * 2 * pr.qkv.kvm.blocks * pr.qkv.nkv_l * static_cast<int64_t>(pr.qkv.kvm.block_len);
    if (pr.ldo != pr.out_cols || !pr.qkv.q_lo || kv_rows >= (int64_t(1) << 31) ||
        !make_map_rows16(&mo, pr.out, pr.T, pr.ldo, qp) ||
        !make_map_rows16(&mo2, pr.qkv.q_lo, pr.T, static_cast<int64_t>(pr.qkv.n) * pr.qkv.nq_l * pr.qkv.hd, qp) ||
        !make_map_rows16(&mkv, pr.qkv.kv, kv_rows, pr.qkv.hd, qp))
      return cudaErrorInvalidValue;
  }
  if constexpr (PAIR)
    return launch_pdl_cluster(kern, Cfg::CL, dim3(grid), dim3(Cfg::THREADS), smem, s, mx, mw, mo, mo2, mkv, gp);
  return launch_pdl(kern, dim3(grid), dim3(Cfg::THREADS), smem, s, mx, mw, mo, mo2, mkv, gp);
}

cudaError_t launch_gemm(const GemmProblem& pr, const GemmPlan& pl, float* partials, int* counters, int* status,
                        cudaStream_t stream) {
  if (pr.T <= 0) return cudaSuccess;
  if (pr.k_seg % 64 || pr.ldo % 8) return cudaErrorInvalidValue;
  CUtensorMap mx, mw;
  if (!make_map(&mx, pr.x, pr.x_rows, pr.x_cols, pr.x_ld, pl.swap ? pl.BN : 128)) return cudaErrorInvalidValue;
  if (!make_map(&mw, pr.w, pr.w_rows, pr.w_cols, pr.w_ld, pl.swap ? 128 : (pl.pair ? pl.BN / 2 : pl.BN)))
    return cudaErrorInvalidValue;
  GemmParams gp{};
  gp.T = pr.T;
  gp.N = pr.N;
  gp.n_seg = pr.n_seg;
  gp.kb_seg = pr.k_seg / 64;
  gp.x_k_seg = pr.x_k_seg;
  gp.w_row_seg = pr.w_row_seg;
  gp.tiles_t = pl.tiles_t;
  gp.tiles_f = pl.tiles_f;
  gp.splits = pl.splits;
  gp.total_kb = pr.n_seg * gp.kb_seg;
  gp.out = pr.out;
  gp.ldo = pr.ldo;
  gp.out_cols = pr.out_cols;
  gp.partials = partials;
  gp.counters = counters;
  gp.amax_val = pr.amax_val;
  gp.amax_idx = pr.amax_idx;
  gp.amax_ld = pr.amax_ld;
  gp.logits = pr.logits;
  gp.ld_logits = pr.ld_logits;
  gp.vocab = pr.vocab;
  gp.out_ids = pr.out_ids;
  gp.done_counter = counters;
  gp.sched_counter = counters + 1;
  gp.amax_keys = reinterpret_cast<unsigned long long*>(counters + kArgmaxKeyOffset);
  gp.qkv = pr.qkv;
  for (int k = 0; k < 2; ++k) {
    gp.discard[k] = pr.discard[k];
    gp.discard_lines[k] = pr.discard[k] ? pr.discard_lines[k] : 0;
  }
  gp.row_ss_out = pr.row_ss_out;
  gp.row_ss_out_groups = pr.out_cols / 32;
  gp.row_out16 = static_cast<__half*>(pr.row_out16);
  if (pr.row_ss_out && (pr.epi != EPI_RESID || !pr.row_out16 || pr.out_cols % 32 || pr.ldo % 4)) return cudaErrorInvalidValue;
  gp.row_ss = pr.row_ss;
  gp.row_groups = pr.row_groups;
  gp.row_inv_k = pr.row_ss ? 1.0f / static_cast<float>(pr.k_seg) : 0.0f;
  gp.row_eps = pr.row_eps;
  if (pr.row_ss && (pr.n_seg != 1 || pr.row_groups * 32 != pr.k_seg || (pr.epi != EPI_QKV && pr.epi != EPI_SILU)))
    return cudaErrorInvalidValue;
  gp.status = status;
  const int g = pl.grid;
#define TP_V(BN_, EPI_, ACC_, SW_)                                                           \
  if (pl.BN == BN_ && pr.epi == EPI_ && pl.acc == ACC_ && pl.swap == SW_ && !pl.pair)         \
    return launch_variant<BN_, EPI_, ACC_, SW_>(mx, mw, pr, gp, g, stream);
#define TP_VP(BN_, EPI_, ACC_)                                                               \
  if (pl.BN == BN_ && pr.epi == EPI_ && pl.acc == ACC_ && !pl.swap && pl.pair && !pl.xch)    \
    return launch_variant<BN_, EPI_, ACC_, false, true>(mx, mw, pr, gp, g, stream);
  if (pl.xch) {
    if (pl.BN != 256 || pr.epi != EPI_RESID || !pl.pair || pl.splits != 2 || g != 4 * pl.tiles_t * pl.tiles_f)
      return cudaErrorInvalidValue;
    return launch_variant<256, EPI_RESID, true, false, true, true>(mx, mw, pr, gp, g, stream);
  }
  TP_VP(256, EPI_STORE, false)
  TP_VP(256, EPI_SILU, false)
  TP_VP(256, EPI_QKV, false)
  TP_VP(128, EPI_RESID, false)
  TP_VP(128, EPI_RESID, true)
  TP_VP(256, EPI_RESID, true)
  TP_V(256, EPI_STORE, false, false)
  TP_V(128, EPI_STORE, false, false)
  TP_V(64, EPI_STORE, false, false)
  TP_V(128, EPI_STORE, true, false)
  TP_V(64, EPI_STORE, true, false)
  TP_V(256, EPI_QKV, false, false)
  TP_V(128, EPI_QKV, false, false)
  TP_V(64, EPI_QKV, false, false)
  TP_V(128, EPI_QKV, true, false)
  TP_V(64, EPI_QKV, true, false)
  TP_V(256, EPI_SILU, false, false)
  TP_V(128, EPI_SILU, false, false)
  TP_V(128, EPI_SILU, true, false)
  TP_V(256, EPI_RESID, false, false)
  TP_V(128, EPI_RESID, false, false)
  TP_V(64, EPI_RESID, false, false)
  TP_V(128, EPI_RESID, true, false)
  TP_V(64, EPI_RESID, true, false)
  TP_V(32, EPI_STORE, true, true)
  TP_V(64, EPI_STORE, true, true)
  TP_V(32, EPI_QKV, true, true)
  TP_V(64, EPI_QKV, true, true)
  TP_V(32, EPI_SILU, true, true)
  TP_V(64, EPI_SILU, true, true)
  TP_V(32, EPI_RESID, true, true)
  TP_V(64, EPI_RESID, true, true)
  TP_V(64, EPI_ARGMAX, false, false)
  TP_V(16, EPI_ARGMAX, false, true)
  TP_V(32, EPI_ARGMAX, false, true)
  TP_V(64, EPI_ARGMAX, false, true)
  TP_V(128, EPI_ARGMAX, false, true)
  TP_V(160, EPI_ARGMAX, false, true)
  TP_V(192, EPI_ARGMAX, false, true)
  TP_V(256, EPI_ARGMAX, false, true)
#undef TP_V
#undef TP_VP
  return cudaErrorNotSupported;
}

}  // namespace tpk
