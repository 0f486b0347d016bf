// Bandwidth-bound kernels of the tensor-parallel forward: vocab-parallel
// embedding with its rank-sum, RMSNorm, the final RMSNorm of each sequence's
// last token, and the argmax reduction that replaces the logits all-gather.
// (q/k RMSNorm + RoPE + KV-cache write run in the QKV GEMM epilogue.)  Plain coalesced 16-byte loads; no tensor
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
// One CTA per token; each thread owns 8 consecutive hidden elements.  Also the
// first layer's deferred-RMSNorm inputs: the row in fp16 (xh) and the sums of
// squares of its 32-column groups (ss), or neither when xh is null.
// ---------------------------------------------------------------------------
__global__ void embed_vocab_parallel_kernel(const int32_t* __restrict__ ids, const uint4* __restrict__ table,
                                            int n, int64_t v_local, int64_t vocab, int H,
                                            float4* __restrict__ out, uint4* __restrict__ xh,
                                            float* __restrict__ ss, int* status) {
  griddep_wait();  // the ids may come from the previous step's argmax
  griddep_launch();
  const int t = blockIdx.x;
  // one read per warp (the ids may live in host memory, read over the host link)
  int id = 0;
  if ((threadIdx.x & 31) == 0) id = ids[t];
  id = __shfl_sync(0xffffffffu, id, 0);
  if (threadIdx.x == 0 && (id < 0 || id >= vocab)) raise_flag(status, TP_DEVFLAG_BAD_TOKEN);
  const int chunks = H / 8;
  const int trips = (chunks + blockDim.x - 1) / blockDim.x;  // the same on every lane (group shuffles)
  uint32_t sat = 0;  // an fp16 row element clamped to the fp16 range
  for (int k = 0; k < trips; ++k) {
    const int c = threadIdx.x + k * blockDim.x;
    const bool live = c < chunks;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
    for (int r = 0; r < n && live; ++r) {
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
    if (live) {
      out[(static_cast<int64_t>(t) * chunks + c) * 2] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      out[(static_cast<int64_t>(t) * chunks + c) * 2 + 1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    if (xh != nullptr) {  // uniform
      float s = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) s += acc[i] * acc[i];
      s += __shfl_xor_sync(0xffffffffu, s, 1);  // the 4 chunks of a 32-column group
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      if (live) {
        uint4 o;
        o.x = pack_f16x2(acc[0], acc[1], sat);
        o.y = pack_f16x2(acc[2], acc[3], sat);
        o.z = pack_f16x2(acc[4], acc[5], sat);
        o.w = pack_f16x2(acc[6], acc[7], sat);
        xh[static_cast<int64_t>(t) * chunks + c] = o;
        if ((c & 3) == 0) ss[static_cast<int64_t>(t) * (H / 32) + c / 4] = s;
      }
    }
  }
  report_sat(status, sat);
}

cudaError_t launch_embed(const int32_t* ids, int T, const void* embed_stacked, int n, int64_t v_local,
                         int64_t vocab, int H, void* out, void* xh, float* ss, int* status, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (H % 32) return cudaErrorInvalidValue;
  // enough threads that a row takes one or two chunks per thread (the loads overlap)
  const int threads = H / 8 < 512 ? 32 * ((H / 8 + 31) / 32) : 512;
  return launch_pdl(embed_vocab_parallel_kernel, dim3(T), dim3(threads), 0, s, ids,
                    reinterpret_cast<const uint4*>(embed_stacked), n, v_local, vocab, H, reinterpret_cast<float4*>(out),
                    reinterpret_cast<uint4*>(xh), ss, status);
}

// two bf16 ones: the norm weight of a norm whose weight is folded into the next GEMM
constexpr uint32_t kOnes2 = 0x3F803F80u;

// ---------------------------------------------------------------------------
// RMSNorm over the hidden dimension of the fp32 residual stream, fp32 math:
// y = x * rsqrt(mean(x^2) + eps) * w, written as fp16 (the next GEMM's operand);
// w null: ones (the weight is folded into that GEMM's weights).
// One warp per row; row_index (optional) picks the source row of each output row.
// ---------------------------------------------------------------------------
template <int VPL>  // 8-element groups per lane kept in registers
__global__ void rmsnorm_kernel(const float4* __restrict__ x, int64_t rows, int H, const uint4* __restrict__ w,
                               float eps, uint4* __restrict__ out, const int32_t* __restrict__ cu_last, int* status) {
  griddep_wait();
  griddep_launch();
  const int warps = blockDim.x / 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int64_t src = cu_last ? cu_last[row + 1] - 1 : row;
  const int chunks = H / 8;
  const float4* xr = x + src * (H / 4);
  float v[VPL][8];
  float ss = 0.0f;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int c = lane + 32 * j;
    if (c < chunks) {
      const float4 a = xr[2 * c], b = xr[2 * c + 1];
      v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
      v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += v[j][i] * v[j][i];
    }
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / static_cast<float>(H) + eps);
  uint32_t sat = 0;
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int c = lane + 32 * j;
    if (c < chunks) {
      const uint4 wu = w ? w[c] : make_uint4(kOnes2, kOnes2, kOnes2, kOnes2);
      const float wf[8] = {bf16lo(wu.x), bf16hi(wu.x), bf16lo(wu.y), bf16hi(wu.y),
                           bf16lo(wu.z), bf16hi(wu.z), bf16lo(wu.w), bf16hi(wu.w)};
      uint4 o;
      o.x = pack_f16x2(v[j][0] * inv * wf[0], v[j][1] * inv * wf[1], sat);
      o.y = pack_f16x2(v[j][2] * inv * wf[2], v[j][3] * inv * wf[3], sat);
      o.z = pack_f16x2(v[j][4] * inv * wf[4], v[j][5] * inv * wf[5], sat);
      o.w = pack_f16x2(v[j][6] * inv * wf[6], v[j][7] * inv * wf[7], sat);
      out[row * chunks + c] = o;
    }
  }
  report_sat(status, sat);
}

// Wide rows (H > 2048): one warp per row, two passes (the second re-reads the row from L1/L2).
__global__ void rmsnorm_wide_kernel(const float4* __restrict__ x, int64_t rows, int H, const uint4* __restrict__ w,
                                    float eps, uint4* __restrict__ out, const int32_t* __restrict__ cu_last,
                                    int* status) {
  griddep_wait();
  griddep_launch();
  const int warps = blockDim.x / 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int64_t src = cu_last ? cu_last[row + 1] - 1 : row;
  const int chunks = H / 8;
  const float4* xr = x + src * (H / 4);
  float ss = 0.0f;
  for (int c = lane; c < chunks; c += 32) {
    const float4 a = xr[2 * c], b = xr[2 * c + 1];
    ss += a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
  }
  ss = warp_sum(ss);
  const float inv = rsqrtf(ss / static_cast<float>(H) + eps);
  uint32_t sat = 0;
  for (int c = lane; c < chunks; c += 32) {
    const float4 a = xr[2 * c], b = xr[2 * c + 1];
    const uint4 wu = w ? w[c] : make_uint4(kOnes2, kOnes2, kOnes2, kOnes2);
    uint4 o;
    o.x = pack_f16x2(a.x * inv * bf16lo(wu.x), a.y * inv * bf16hi(wu.x), sat);
    o.y = pack_f16x2(a.z * inv * bf16lo(wu.y), a.w * inv * bf16hi(wu.y), sat);
    o.z = pack_f16x2(b.x * inv * bf16lo(wu.z), b.y * inv * bf16hi(wu.z), sat);
    o.w = pack_f16x2(b.z * inv * bf16lo(wu.w), b.w * inv * bf16hi(wu.w), sat);
    out[row * chunks + c] = o;
  }
  report_sat(status, sat);
}

// Few long rows (decode): one 256-thread block per row, every 8-element chunk of
// the row loaded at once (CPT chunks per thread), one block-wide sum of squares.
template <int CPT>
__global__ void __launch_bounds__(256) rmsnorm_row_block_kernel(const float4* __restrict__ x, int64_t rows, int H,
                                                                 const uint4* __restrict__ w, float eps,
                                                                 uint4* __restrict__ out,
                                                                 const int32_t* __restrict__ cu_last, int* status) {
  griddep_wait();
  griddep_launch();
  __shared__ float red[8];
  const int64_t row = blockIdx.x;
  const int64_t src = cu_last ? cu_last[row + 1] - 1 : row;
  const int chunks = H / 8;
  const float4* xr = x + src * (H / 4);
  float v[CPT][8];
  float ss = 0.0f;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + 256 * j;
    if (c < chunks) {
      const float4 a = xr[2 * c], b = xr[2 * c + 1];
      v[j][0] = a.x; v[j][1] = a.y; v[j][2] = a.z; v[j][3] = a.w;
      v[j][4] = b.x; v[j][5] = b.y; v[j][6] = b.z; v[j][7] = b.w;
#pragma unroll
      for (int i = 0; i < 8; ++i) ss += v[j][i] * v[j][i];
    }
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += red[i];
  const float inv = rsqrtf(tot / static_cast<float>(H) + eps);
  uint32_t sat = 0;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = threadIdx.x + 256 * j;
    if (c < chunks) {
      const uint4 wu = w ? w[c] : make_uint4(kOnes2, kOnes2, kOnes2, kOnes2);
      const float wf[8] = {bf16lo(wu.x), bf16hi(wu.x), bf16lo(wu.y), bf16hi(wu.y),
                           bf16lo(wu.z), bf16hi(wu.z), bf16lo(wu.w), bf16hi(wu.w)};
      uint4 o;
      o.x = pack_f16x2(v[j][0] * inv * wf[0], v[j][1] * inv * wf[1], sat);
      o.y = pack_f16x2(v[j][2] * inv * wf[2], v[j][3] * inv * wf[3], sat);
      o.z = pack_f16x2(v[j][4] * inv * wf[4], v[j][5] * inv * wf[5], sat);
      o.w = pack_f16x2(v[j][6] * inv * wf[6], v[j][7] * inv * wf[7], sat);
      out[row * chunks + c] = o;
    }
  }
  report_sat(status, sat);
}

static cudaError_t rmsnorm_rows(const void* x, int64_t rows, int H, const void* w, float eps, void* out,
                                const int32_t* cu_last, int* status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int chunks = H / 8;
  if (rows <= 256 && chunks > 128 && chunks <= 4 * 256) {  // few long rows: a block per row
    auto X = reinterpret_cast<const float4*>(x);
    auto W = reinterpret_cast<const uint4*>(w);
    auto O = reinterpret_cast<uint4*>(out);
    const dim3 grid(static_cast<unsigned>(rows)), block(256);
    if (chunks <= 256) return launch_pdl(rmsnorm_row_block_kernel<1>, grid, block, 0, s, X, rows, H, W, eps, O, cu_last, status);
    if (chunks <= 512) return launch_pdl(rmsnorm_row_block_kernel<2>, grid, block, 0, s, X, rows, H, W, eps, O, cu_last, status);
    return launch_pdl(rmsnorm_row_block_kernel<4>, grid, block, 0, s, X, rows, H, W, eps, O, cu_last, status);
  }
  const int vpl = (H / 8 + 31) / 32;
  const int warps = 4;
  const dim3 grid(static_cast<unsigned>((rows + warps - 1) / warps)), block(32 * warps);
  auto X = reinterpret_cast<const float4*>(x);
  auto W = reinterpret_cast<const uint4*>(w);
  auto O = reinterpret_cast<uint4*>(out);
  if (vpl <= 1) return launch_pdl(rmsnorm_kernel<1>, grid, block, 0, s, X, rows, H, W, eps, O, cu_last, status);
  if (vpl <= 2) return launch_pdl(rmsnorm_kernel<2>, grid, block, 0, s, X, rows, H, W, eps, O, cu_last, status);
  if (vpl <= 4) return launch_pdl(rmsnorm_kernel<4>, grid, block, 0, s, X, rows, H, W, eps, O, cu_last, status);
  if (vpl <= 8) return launch_pdl(rmsnorm_kernel<8>, grid, block, 0, s, X, rows, H, W, eps, O, cu_last, status);
  return launch_pdl(rmsnorm_wide_kernel, grid, block, 0, s, X, rows, H, W, eps, O, cu_last, status);
}

// Row statistics for a deferred RMSNorm (the norm itself happens in the next
// GEMM's epilogue, its weight folded into that GEMM's weights): fp16 copy of
// each fp32 residual row and the sum of squares of each 32-column group.  One
// warp per row; lane l takes 8-column chunks l, l + 32, ...; the 4 lanes of a
// 32-column group add their sums with two shuffles.
__global__ void row_stats_kernel(const float4* __restrict__ x, int64_t rows, int H, uint4* __restrict__ xh,
                                 float* __restrict__ ss, int* status) {
  griddep_wait();
  griddep_launch();
  const int warps = blockDim.x / 32;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * warps + threadIdx.x / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;  // warp-uniform
  const int chunks = H / 8, groups = H / 32;
  const float4* xr = x + row * (H / 4);
  uint32_t sat = 0;
  for (int c0 = 0; c0 < chunks; c0 += 32) {  // same trip count on every lane
    const int c = c0 + lane;
    float s = 0.0f;
    if (c < chunks) {
      const float4 a = xr[2 * c], b = xr[2 * c + 1];
      s = a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
      uint4 o;
      o.x = pack_f16x2(a.x, a.y, sat);
      o.y = pack_f16x2(a.z, a.w, sat);
      o.z = pack_f16x2(b.x, b.y, sat);
      o.w = pack_f16x2(b.z, b.w, sat);
      xh[row * chunks + c] = o;
    }
    s += __shfl_xor_sync(0xffffffffu, s, 1);
    s += __shfl_xor_sync(0xffffffffu, s, 2);
    if ((lane & 3) == 0 && c < chunks) ss[row * groups + c / 4] = s;
  }
  report_sat(status, sat);
}

cudaError_t launch_row_stats(const void* x, int64_t rows, int H, void* xh, float* ss, int* status,
                             cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  if (H % 32) return cudaErrorInvalidValue;
  const int warps = 4;
  return launch_pdl(row_stats_kernel, dim3(static_cast<unsigned>((rows + warps - 1) / warps)), dim3(32 * warps), 0,
                    s, reinterpret_cast<const float4*>(x), rows, H, reinterpret_cast<uint4*>(xh), ss, status);
}

cudaError_t launch_rmsnorm(const void* x, int64_t rows, int H, const void* w, float eps, void* out, int* status,
                           cudaStream_t s) {
  return rmsnorm_rows(x, rows, H, w, eps, out, nullptr, status, s);
}

// Final RMSNorm of each sequence's last token (row cu_q[b+1] - 1 of the residual stream).
cudaError_t launch_final_norm_select(const void* hidden, int H, const int32_t* cu_q, int B, const void* w,
                                     float eps, void* out, int* status, cudaStream_t s) {
  return rmsnorm_rows(hidden, B, H, w, eps, out, cu_q, status, s);
}

// ---------------------------------------------------------------------------
// bf16 -> fp16, in place (weight shards used as tensor-core operands).  Exact
// for magnitudes in fp16's normal range [2^-14, 65504]; smaller magnitudes
// round to fp16's subnormal grid (absolute error <= 2^-25), larger ones
// saturate.
// ---------------------------------------------------------------------------
__global__ void bf16_to_f16_kernel(uint32_t* __restrict__ w, size_t n_pairs, int* status) {
  uint32_t sat = 0;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n_pairs;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint32_t v = w[i];
    w[i] = pack_f16x2(bf16lo(v), bf16hi(v), sat);
  }
  report_sat(status, sat);
}

// W[r][c] * norm[c] -> fp16, in place ([rows][cols] bf16 in, fp16 out): an
// RMSNorm weight folded into the projection that reads the normed rows
// (xn W^T = (x * inv) (W * diag(w))^T).  The bf16 x bf16 product is exact in
// fp32, so the only rounding is the one to fp16.
__global__ void fold_norm_f16_kernel(uint32_t* __restrict__ w, size_t n_pairs, int cols,
                                     const __nv_bfloat16* __restrict__ norm, int* status) {
  uint32_t sat = 0;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n_pairs;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const uint32_t v = w[i];
    const int c = static_cast<int>((2 * i) % static_cast<size_t>(cols));  // cols is even
    w[i] = pack_f16x2(bf16lo(v) * bf2f(norm[c]), bf16hi(v) * bf2f(norm[c + 1]), sat);
  }
  report_sat(status, sat);
}

cudaError_t launch_fold_norm_f16(void* w, size_t rows, int cols, const void* norm, int* status, cudaStream_t s) {
  const size_t pairs = rows * static_cast<size_t>(cols) / 2;
  if (pairs == 0) return cudaSuccess;
  if (cols % 2) return cudaErrorInvalidValue;
  const size_t blocks = (pairs + 255) / 256;
  fold_norm_f16_kernel<<<static_cast<unsigned>(blocks < 65536 ? blocks : 65536), 256, 0, s>>>(
      reinterpret_cast<uint32_t*>(w), pairs, cols, reinterpret_cast<const __nv_bfloat16*>(norm), status);
  return cudaGetLastError();
}

cudaError_t launch_bf16_to_f16(void* w, size_t elems, int* status, cudaStream_t s) {
  if (elems == 0) return cudaSuccess;
  const size_t pairs = elems / 2;
  const size_t blocks = (pairs + 255) / 256;
  bf16_to_f16_kernel<<<static_cast<unsigned>(blocks < 65536 ? blocks : 65536), 256, 0, s>>>(
      reinterpret_cast<uint32_t*>(w), pairs, status);
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
  griddep_wait();
  griddep_launch();
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
  return launch_pdl(argmax_reduce_kernel, dim3((B + 3) / 4), dim3(128), 0, s, val, idx, tiles, ld, B, out);
}

// ---------------------------------------------------------------------------
// Greedy decoding between two forwards ("Tensor parallelism from scratch", tp.py
// main: the argmax of the last logits is appended and fed back as the next
// single-token input): each sequence's cached length grows by the token the
// forward just wrote, and the forward's argmax ids go to row *step of the
// history.  One block; the step counter lives on the device so that a captured
// graph of the decode forward + this kernel can be replayed unchanged.
// ---------------------------------------------------------------------------
__global__ void decode_advance_kernel(int32_t* ctx_len, int B, const int32_t* ids, int32_t* history, int max_rows,
                                      int32_t* step, int32_t* status) {
  griddep_wait();
  griddep_launch();
  __shared__ int row;
  if (threadIdx.x == 0) row = *step;
  __syncthreads();
  const bool in = row >= 0 && row < max_rows;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    ctx_len[b] += 1;
    if (in) history[static_cast<size_t>(row) * B + b] = ids[b];
  }
  if (threadIdx.x == 0) {
    if (!in) raise_flag(status, TP_DEVFLAG_BAD_TOKEN);
    *step = row + 1;
  }
}

cudaError_t launch_decode_advance(int32_t* ctx_len, int B, const int32_t* ids, int32_t* history, int max_rows,
                                  int32_t* step, int32_t* status, cudaStream_t s) {
  if (B <= 0) return cudaSuccess;
  return launch_pdl(decode_advance_kernel, dim3(1), dim3(B < 1024 ? ((B + 31) / 32) * 32 : 1024), 0, s, ctx_len, B,
                    ids, history, max_rows, step, status);
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
