// Bandwidth-bound kernels of the tensor-parallel forward: vocab-parallel
// embedding with its rank-sum, RMSNorm, q/k RMSNorm + RoPE + KV-cache write,
// final RMSNorm of each sequence's last token, and the argmax reduction that
// replaces the logits all-gather.  Plain coalesced 16-byte loads; no tensor
// cores (none of this is a contraction).
#include <climits>

#include "kernels.h"
#include "sm100.cuh"

namespace tpk {

// ---------------------------------------------------------------------------
// Vocab-parallel embedding ("Tensor parallelism from scratch", tp.py
// VocabParallelEmbedding; mini-SGLang layers/embedding.py:42): every rank r
// looks up ids inside its slice [r*V_l, min((r+1)*V_l, V)) of the table and
// writes 0 for the others; the all-reduce sums the rank outputs.  Emulated
// rank by rank in fixed order (exactly one term is non-zero, so the sum is
// the table row, bit for bit).  Ids outside [0, V) give a zero row and raise
// TP_DEVFLAG_BAD_TOKEN.
// One CTA per token; each thread owns 8 consecutive hidden elements.
// ---------------------------------------------------------------------------
__global__ void embed_vocab_parallel_kernel(const int32_t* __restrict__ ids, const uint4* __restrict__ table,
                                            int n, int64_t v_local, int64_t vocab, int H,
                                            uint4* __restrict__ out, int* status) {
  const int t = blockIdx.x;
  const int id = ids[t];
  if (threadIdx.x == 0 && (id < 0 || id >= vocab)) raise_flag(status, TP_DEVFLAG_BAD_TOKEN);
  const int chunks = H / 8;
  for (int c = threadIdx.x; c < chunks; c += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int r = 0; r < n; ++r) {
      const int64_t start = r * v_local;
      const int64_t end = min(start + v_local, vocab);
      if (id >= start && id < end) {  // this rank's slice holds the id
        const uint4 w = table[((static_cast<int64_t>(r) * v_local + (id - start)) * H) / 8 + c];
        acc[0] += bf16lo(w.x); acc[1] += bf16hi(w.x);
        acc[2] += bf16lo(w.y); acc[3] += bf16hi(w.y);
        acc[4] += bf16lo(w.z); acc[5] += bf16hi(w.z);
        acc[6] += bf16lo(w.w); acc[7] += bf16hi(w.w);
      }
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    out[static_cast<int64_t>(t) * chunks + c] = o;
  }
}

cudaError_t launch_embed(const int32_t* ids, int T, const void* embed_stacked, int n, int64_t v_local,
                         int64_t vocab, int H, void* out, int* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int threads = H / 8 < 128 ? 32 * ((H / 8 + 31) / 32) : 128;
  embed_vocab_parallel_kernel<<<T, threads, 0, s>>>(ids, reinterpret_cast<const uint4*>(embed_stacked), n, v_local,
                                                    vocab, H, reinterpret_cast<uint4*>(out), status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// RMSNorm over the hidden dimension, fp32 math: y = x * rsqrt(mean(x^2)+eps) * w.
// One warp per row; row_index (optional) picks the source row of each output row.
// ---------------------------------------------------------------------------
template <int VPL>  // 16-byte vectors per lane
__global__ void rmsnorm_kernel(const uint4* __restrict__ x, int64_t rows, int H, const uint4* __restrict__ w,
                               float eps, uint4* __restrict__ out, const int32_t* __restrict__ row_index) {
  const int warps = blockDim.x / 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int64_t src = row_index ? row_index[row] : row;
  const int chunks = H / 8;
  const uint4* xr = x + src * chunks;
  float v[VPL][8];
  float ss = 0.0f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int c = lane + 32 * j;
    if (c < chunks) {
      const uint4 u = xr[c];
      v[j][0] = bf16lo(u.x); v[j][1] = bf16hi(u.x);
      v[j][2] = bf16lo(u.y); v[j][3] = bf16hi(u.y);
      v[j][4] = bf16lo(u.z); v[j][5] = bf16hi(u.z);
      v[j][6] = bf16lo(u.w); v[j][7] = bf16hi(u.w);
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += v[j][i] * v[j][i];
    }
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / static_cast<float>(H) + eps);
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int c = lane + 32 * j;
    if (c < chunks) {
      const uint4 wu = w[c];
      const float wf[8] = {bf16lo(wu.x), bf16hi(wu.x), bf16lo(wu.y), bf16hi(wu.y),
                           bf16lo(wu.z), bf16hi(wu.z), bf16lo(wu.w), bf16hi(wu.w)};
      uint4 o;
      o.x = pack_bf16x2(v[j][0] * inv * wf[0], v[j][1] * inv * wf[1]);
      o.y = pack_bf16x2(v[j][2] * inv * wf[2], v[j][3] * inv * wf[3]);
      o.z = pack_bf16x2(v[j][4] * inv * wf[4], v[j][5] * inv * wf[5]);
      o.w = pack_bf16x2(v[j][6] * inv * wf[6], v[j][7] * inv * wf[7]);
      out[row * chunks + c] = o;
    }
  }
}

// Wide rows (H > 2048): one warp per row, two passes (the second re-reads the row from L1/L2).
__global__ void rmsnorm_wide_kernel(const uint4* __restrict__ x, int64_t rows, int H, const uint4* __restrict__ w,
                                    float eps, uint4* __restrict__ out, const int32_t* __restrict__ row_index) {
  const int warps = blockDim.x / 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int64_t src = row_index ? row_index[row] : row;
  const int chunks = H / 8;
  const uint4* xr = x + src * chunks;
  float ss = 0.0f;
  for (int c = lane; c < chunks; c += 32) {
    const uint4 u = xr[c];
    const float f[8] = {bf16lo(u.x), bf16hi(u.x), bf16lo(u.y), bf16hi(u.y),
                        bf16lo(u.z), bf16hi(u.z), bf16lo(u.w), bf16hi(u.w)};
#pragma unroll
    for (int i = 0; i < 8; ++i) ss += f[i] * f[i];
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / static_cast<float>(H) + eps);
  for (int c = lane; c < chunks; c += 32) {
    const uint4 u = xr[c];
    const uint4 wu = w[c];
    uint4 o;
    o.x = pack_bf16x2(bf16lo(u.x) * inv * bf16lo(wu.x), bf16hi(u.x) * inv * bf16hi(wu.x));
    o.y = pack_bf16x2(bf16lo(u.y) * inv * bf16lo(wu.y), bf16hi(u.y) * inv * bf16hi(wu.y));
    o.z = pack_bf16x2(bf16lo(u.z) * inv * bf16lo(wu.z), bf16hi(u.z) * inv * bf16hi(wu.z));
    o.w = pack_bf16x2(bf16lo(u.w) * inv * bf16lo(wu.w), bf16hi(u.w) * inv * bf16hi(wu.w));
    out[row * chunks + c] = o;
  }
}

cudaError_t launch_rmsnorm(const void* x, int64_t rows, int H, const void* w, float eps, void* out,
                           const int32_t* row_index, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int vpl = (H / 8 + 31) / 32;
  const int warps = 4;
  const unsigned grid = static_cast<unsigned>((rows + warps - 1) / warps);
  auto X = reinterpret_cast<const uint4*>(x);
  auto W = reinterpret_cast<const uint4*>(w);
  auto O = reinterpret_cast<uint4*>(out);
  if (vpl <= 1) rmsnorm_kernel<1><<<grid, 32 * warps, 0, s>>>(X, rows, H, W, eps, O, row_index);
  else if (vpl <= 2) rmsnorm_kernel<2><<<grid, 32 * warps, 0, s>>>(X, rows, H, W, eps, O, row_index);
  else if (vpl <= 4) rmsnorm_kernel<4><<<grid, 32 * warps, 0, s>>>(X, rows, H, W, eps, O, row_index);
  else if (vpl <= 8) rmsnorm_kernel<8><<<grid, 32 * warps, 0, s>>>(X, rows, H, W, eps, O, row_index);
  else rmsnorm_wide_kernel<<<grid, 32 * warps, 0, s>>>(X, rows, H, W, eps, O, row_index);
  return cudaGetLastError();
}

// Last token of each sequence (cu_q[b+1]-1), then RMSNorm with the final norm weight.
__global__ void last_token_index_kernel(const int32_t* cu_q, int B, int32_t* idx) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b < B) idx[b] = cu_q[b + 1] - 1;
}

cudaError_t launch_final_norm_select(const void* hidden, int H, const int32_t* cu_q, int B, const void* w,
                                     float eps, void* out, int32_t* idx, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  last_token_index_kernel<<<(B + 127) / 128, 128, 0, s>>>(cu_q, B, idx);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_rmsnorm(hidden, B, H, w, eps, out, idx, s);
}

// ---------------------------------------------------------------------------
// q/k RMSNorm per head over head_dim, rotate-half RoPE at each token's
// position, then K and V written to the rank's cache (post-RoPE K, raw V);
// q is rewritten in place for the attention kernel.
// ("Tensor parallelism from scratch", tp.py TPAttention.forward: q_norm/k_norm,
// apply_rope at positions start..start+T, cache.update.)
// One warp per (token, rank, head slot); the slot enumerates nq_l q heads,
// nkv_l k heads and nkv_l v heads of the rank.
// ---------------------------------------------------------------------------
template <int HD>
__global__ void qk_norm_rope_kernel(RopeArgs a) {
  constexpr int HALF = HD / 2;
  constexpr int PER = HALF / 32;  // elements per lane in each half
  const int warps = blockDim.x / 32;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  const int slots = a.nq_l + 2 * a.nkv_l;
  const int64_t total = static_cast<int64_t>(a.T) * a.n * slots;
  if (wid >= total) return;
  const int slot_h = static_cast<int>(wid % slots);
  const int r = static_cast<int>((wid / slots) % a.n);
  const int t = static_cast<int>(wid / (static_cast<int64_t>(slots) * a.n));
  // sequence of token t: largest b with cu_q[b] <= t
  int lo = 0, hi = a.B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.cu_q[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  const int b = lo;
  const int pos = a.ctx_len[b] + (t - a.cu_q[b]);
  if (pos < 0 || pos >= a.cap || pos >= a.max_pos) {
    if (lane == 0) raise_flag(a.status, TP_DEVFLAG_BAD_TOKEN);
    return;
  }
  __nv_bfloat16* row = reinterpret_cast<__nv_bfloat16*>(a.qkv) + static_cast<int64_t>(t) * a.n * a.w_rank +
                       static_cast<int64_t>(r) * a.w_rank + static_cast<int64_t>(slot_h) * HD;
  float x0[PER], x1[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    x0[i] = bf2f(row[lane + 32 * i]);
    x1[i] = bf2f(row[HALF + lane + 32 * i]);
  }
  const int seq_slot = a.slot[b];
  const size_t plane = static_cast<size_t>(a.max_seqs) * a.nkv_l * a.cap * HD;  // one of K or V for one rank
  if (slot_h >= a.nq_l + a.nkv_l) {  // v: raw copy into the cache
    const int g = slot_h - a.nq_l - a.nkv_l;
    __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(a.kv) + (2 * static_cast<size_t>(r) + 1) * plane +
                         ((static_cast<size_t>(seq_slot) * a.nkv_l + g) * a.cap + pos) * HD;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
      dst[lane + 32 * i] = f2bf(x0[i]);
      dst[HALF + lane + 32 * i] = f2bf(x1[i]);
    }
    return;
  }
  const bool is_q = slot_h < a.nq_l;
  const __nv_bfloat16* nw = reinterpret_cast<const __nv_bfloat16*>(is_q ? a.q_norm : a.k_norm);
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < PER; ++i) ss += x0[i] * x0[i] + x1[i] * x1[i];
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / static_cast<float>(HD) + a.eps);
  const float2* cs = a.rope + static_cast<size_t>(pos) * HALF;
  float y0[PER], y1[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int d = lane + 32 * i;
    const float u0 = x0[i] * inv * bf2f(nw[d]);
    const float u1 = x1[i] * inv * bf2f(nw[HALF + d]);
    const float2 c = cs[d];
    y0[i] = u0 * c.x - u1 * c.y;
    y1[i] = u1 * c.x + u0 * c.y;
  }
  __nv_bfloat16* dst;
  if (is_q) {
    dst = row;
  } else {
    const int g = slot_h - a.nq_l;
    dst = reinterpret_cast<__nv_bfloat16*>(a.kv) + (2 * static_cast<size_t>(r)) * plane +
          ((static_cast<size_t>(seq_slot) * a.nkv_l + g) * a.cap + pos) * HD;
  }
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    dst[lane + 32 * i] = f2bf(y0[i]);
    dst[HALF + lane + 32 * i] = f2bf(y1[i]);
  }
}

cudaError_t launch_qk_norm_rope(const RopeArgs& a, cudaStream_t s) {
  if (a.T <= 0) return cudaSuccess;
  const int64_t warps = static_cast<int64_t>(a.T) * a.n * (a.nq_l + 2 * a.nkv_l);
  const unsigned grid = static_cast<unsigned>((warps + 7) / 8);
  if (a.hd == 128) qk_norm_rope_kernel<128><<<grid, 256, 0, s>>>(a);
  else if (a.hd == 64) qk_norm_rope_kernel<64><<<grid, 256, 0, s>>>(a);
  else return cudaErrorInvalidValue;
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Argmax over the per-tile (max, first index) partials of the LM-head epilogue,
// in vocab order: the global first maximal id (NaN counts as the maximum),
// torch.argmax semantics.  Replaces the all-gather of the vocab-parallel
// logits ("Tensor parallelism from scratch", tp.py forward: all_gather, then
// logits[0, -1].argmax()).  One warp per sequence.
// ---------------------------------------------------------------------------
__device__ __forceinline__ bool amax_better(float v, int i, float bv, int bi) {
  const bool vn = v != v, bn = bv != bv;
  if (vn != bn) return vn;
  if (!vn && v != bv) return v > bv;
  return i < bi;
}

__global__ void argmax_reduce_kernel(const float* __restrict__ val, const int* __restrict__ idx, int tiles, int ld,
                                     int B, int32_t* __restrict__ out) {
  const int b = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (b >= B) return;
  float bv = -INFINITY;
  int bi = INT_MAX;
  for (int k = lane; k < tiles; k += 32) {
    const float v = val[static_cast<size_t>(k) * ld + b];
    const int i = idx[static_cast<size_t>(k) * ld + b];
    if (amax_better(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    if (amax_better(ov, oi, bv, bi)) {
      bv = ov;
      bi = oi;
    }
  }
  if (lane == 0) out[b] = bi;
}

cudaError_t launch_argmax_reduce(const float* val, const int* idx, int tiles, int ld, int B, int32_t* out,
                                 cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  argmax_reduce_kernel<<<(B + 3) / 4, 128, 0, s>>>(val, idx, tiles, ld, B, out);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Bounded-wait probe: waits on an mbarrier that nothing completes (and on a
// global flag the caller never sets), with the same bounded wait the GEMM
// uses; must return with TP_DEVFLAG_TIMEOUT set instead of hanging.
// ---------------------------------------------------------------------------
__global__ void wait_probe_kernel(const int* flag, int* status, long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const volatile int* f = flag;
    if (*f == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, static_cast<uint64_t>(limit_ns));
  }
  __syncthreads();
}

cudaError_t launch_wait_probe(const int* flag, int* status, long long limit_ns, cudaStream_t s) {
  wait_probe_kernel<<<1, 32, 0, s>>>(flag, status, limit_ns);
  return cudaGetLastError();
}

}  // namespace tpk
