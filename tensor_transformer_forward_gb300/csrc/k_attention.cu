// Per-rank GQA attention over the rank's KV cache ("Tensor parallelism from
// scratch", tp.py TPAttention.forward and section "KV heads and the limit on
// TP"): each rank attends with its nq_l query heads over its nkv_l kv heads;
// local q head h reads local kv head h / (nq_l / nkv_l) (repeat_interleave);
// scores are scaled by 1/sqrt(hd); new token j of a sequence with ctx cached
// tokens sees keys 0 .. ctx + j.  Softmax in fp32 (base-2, max-subtracted).
//
// Cache layout (per layer): [n][2 (K, V)][max_seqs][nkv_l][cap][hd] bf16.
// q comes from the merged QKV buffer (fp16).  Output layout: [T][n * nq_l * hd]
// fp16 (rank-major heads, the row-split o_proj operand).
#include <climits>

#include "kernels.h"
#include "sm100.cuh"

namespace tpk {

// ---------------------------------------------------------------------------
// Decode (one new token per sequence): flash-decoding split over the keys.
// One CTA = (sequence, rank, local kv head, key split), 4 warps; the G query
// heads of the kv group share every K/V load.  Lanes split head_dim in 16-byte
// pieces (hd/8 lanes per key), so one warp load covers 32/(hd/8) keys.
// Splits combine through an fp32 workspace; the last CTA of a (seq, rank,
// head) to finish (atomic counter, no waiting) merges them in split order.
// ---------------------------------------------------------------------------
template <int HD, int G>
__global__ void __launch_bounds__(128) attn_decode_kernel(AttnArgs a) {
  constexpr int LPK = HD / 8;        // lanes per key
  constexpr int KPI = 32 / LPK;      // keys per warp instruction
  constexpr int U = 4;               // key groups in flight per lane
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ks = lane / LPK, dc = lane % LPK;
  const int per_seq = a.n * a.nkv_l;
  const int unit = blockIdx.x;
  const int b = a.seq_begin + unit / per_seq;
  const int r = (unit % per_seq) / a.nkv_l;
  const int g = unit % a.nkv_l;
  const int split = blockIdx.y;
  const int t = a.cu_q[b];
  const int L = a.ctx_len[b] + 1;
  const int chunk = (L + a.splits - 1) / a.splits;
  const int k0 = split * chunk;
  const int k1 = min(L, k0 + chunk);

  const size_t plane = static_cast<size_t>(a.max_seqs) * a.nkv_l * a.cap * HD;
  const size_t head_off = (static_cast<size_t>(a.slot[b]) * a.nkv_l + g) * a.cap * HD;
  const uint4* Kc = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.kv) +
                                                   (2 * static_cast<size_t>(r)) * plane + head_off);
  const uint4* Vc = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(a.kv) +
                                                   (2 * static_cast<size_t>(r) + 1) * plane + head_off);

  // this lane's 8 dims of each query head, pre-scaled into the exp2 domain
  float q[G][8];
  const __half* qrow = reinterpret_cast<const __half*>(a.qkv) + static_cast<size_t>(t) * a.n * a.w_rank +
                       static_cast<size_t>(r) * a.w_rank;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint4 u = *reinterpret_cast<const uint4*>(qrow + (g * G + h) * HD + dc * 8);
    q[h][0] = f16lo(u.x); q[h][1] = f16hi(u.x); q[h][2] = f16lo(u.y); q[h][3] = f16hi(u.y);
    q[h][4] = f16lo(u.z); q[h][5] = f16hi(u.z); q[h][6] = f16lo(u.w); q[h][7] = f16hi(u.w);
#pragma unroll
    for (int i = 0; i < 8; ++i) q[h][i] *= a.scale_log2;
  }
  float m[G], l[G], acc[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[h][i] = 0.0f;
  }

  constexpr int STEP = 4 * KPI;  // keys covered by one pass of all warps
  // the loop bound is warp-uniform (shuffles inside); each lane adds its key offset ks
  for (int wb = k0 + warp * KPI; wb < k1; wb += STEP * U) {
    const int base = wb + ks;
    uint4 kv_k[U], kv_v[U];
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int key = base + j * STEP;
      if (key < k1) {
        kv_k[j] = __ldcs(Kc + static_cast<size_t>(key) * LPK + dc);
        kv_v[j] = __ldcs(Vc + static_cast<size_t>(key) * LPK + dc);
      }
    }
#pragma unroll
    for (int j = 0; j < U; ++j) {
      const int key = base + j * STEP;
      const bool valid = key < k1;  // uniform across the LPK lanes of this key
      float kf[8], vf[8];
      kf[0] = bf16lo(kv_k[j].x); kf[1] = bf16hi(kv_k[j].x); kf[2] = bf16lo(kv_k[j].y); kf[3] = bf16hi(kv_k[j].y);
      kf[4] = bf16lo(kv_k[j].z); kf[5] = bf16hi(kv_k[j].z); kf[6] = bf16lo(kv_k[j].w); kf[7] = bf16hi(kv_k[j].w);
      vf[0] = bf16lo(kv_v[j].x); vf[1] = bf16hi(kv_v[j].x); vf[2] = bf16lo(kv_v[j].y); vf[3] = bf16hi(kv_v[j].y);
      vf[4] = bf16lo(kv_v[j].z); vf[5] = bf16hi(kv_v[j].z); vf[6] = bf16lo(kv_v[j].w); vf[7] = bf16hi(kv_v[j].w);
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s += q[h][i] * kf[i];
#pragma unroll
        for (int o = LPK / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (valid) {
          const float mn = fmaxf(m[h], s);
          const float corr = exp2f(m[h] - mn);
          const float p = exp2f(s - mn);
          l[h] = l[h] * corr + p;
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[h][i] = acc[h][i] * corr + p * vf[i];
          m[h] = mn;
        }
      }
    }
  }

  // merge the KPI key groups of this warp (lanes with the same dims)
#pragma unroll
  for (int h = 0; h < G; ++h) {
#pragma unroll
    for (int o = LPK; o < 32; o <<= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m[h], o);
      const float l2 = __shfl_xor_sync(0xffffffffu, l[h], o);
      float a2[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a2[i] = __shfl_xor_sync(0xffffffffu, acc[h][i], o);
      const float mn = fmaxf(m[h], m2);
      if (mn != -INFINITY) {
        const float c1 = exp2f(m[h] - mn), c2 = exp2f(m2 - mn);
        l[h] = l[h] * c1 + l2 * c2;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[h][i] = acc[h][i] * c1 + a2[i] * c2;
        m[h] = mn;
      }
    }
  }
  // merge the 4 warps through shared memory: [warp][h][HD + 2]
  __shared__ float red[4][G][HD + 2];
  __shared__ int last_flag;
  if (ks == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int i = 0; i < 8; ++i) red[warp][h][dc * 8 + i] = acc[h][i];
      if (dc == 0) {
        red[warp][h][HD] = m[h];
        red[warp][h][HD + 1] = l[h];
      }
    }
  }
  __syncthreads();
  // thread x handles (h, d) pairs; merged state of this split
  const int unit_heads = G * HD;
  float* part = a.part + (static_cast<size_t>(unit) * a.splits + split) * G * (HD + 2);
  for (int e = threadIdx.x; e < unit_heads; e += blockDim.x) {
    const int h = e / HD, d = e % HD;
    float mm = -INFINITY, ll = 0.0f, aa = 0.0f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float m2 = red[w][h][HD], l2 = red[w][h][HD + 1], a2 = red[w][h][d];
      const float mn = fmaxf(mm, m2);
      if (mn != -INFINITY) {
        const float c1 = exp2f(mm - mn), c2 = exp2f(m2 - mn);
        ll = ll * c1 + l2 * c2;
        aa = aa * c1 + a2 * c2;
        mm = mn;
      }
    }
    if (a.splits == 1) {
      __half* o = reinterpret_cast<__half*>(a.out) + static_cast<size_t>(t) * a.n * a.nq_l * HD +
                  (static_cast<size_t>(r) * a.nq_l + g * G + h) * HD + d;
      *o = __float2half_rn(sat_f16(aa / ll));
    } else {
      part[h * (HD + 2) + d] = aa;
      if (d == 0) {
        part[h * (HD + 2) + HD] = mm;
        part[h * (HD + 2) + HD + 1] = ll;
      }
    }
  }
  if (a.splits == 1) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(a.counters + unit, 1);
    last_flag = (old == a.splits - 1);
  }
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  const float* base = a.part + static_cast<size_t>(unit) * a.splits * G * (HD + 2);
  for (int e = threadIdx.x; e < unit_heads; e += blockDim.x) {
    const int h = e / HD, d = e % HD;
    float mm = -INFINITY, ll = 0.0f, aa = 0.0f;
    for (int s = 0; s < a.splits; ++s) {
      const float* ps = base + (static_cast<size_t>(s) * G + h) * (HD + 2);
      const float m2 = __ldcg(ps + HD), l2 = __ldcg(ps + HD + 1), a2 = __ldcg(ps + d);
      const float mn = fmaxf(mm, m2);
      if (mn != -INFINITY) {
        const float c1 = exp2f(mm - mn), c2 = exp2f(m2 - mn);
        ll = ll * c1 + l2 * c2;
        aa = aa * c1 + a2 * c2;
        mm = mn;
      }
    }
    __half* o = reinterpret_cast<__half*>(a.out) + static_cast<size_t>(t) * a.n * a.nq_l * HD +
                (static_cast<size_t>(r) * a.nq_l + g * G + h) * HD + d;
    *o = __float2half_rn(sat_f16(aa / ll));
  }
  if (threadIdx.x == 0) a.counters[unit] = 0;
}

int decode_splits(int max_kv_len, int num_units, int num_sms) {
  int by_len = (max_kv_len + 511) / 512;
  int by_fill = (4 * num_sms + num_units - 1) / (num_units > 0 ? num_units : 1);
  int s = by_len < by_fill ? by_len : by_fill;
  if (s < 1) s = 1;
  if (s > 64) s = 64;
  return s;
}

cudaError_t launch_attention_decode(const AttnArgs& a, cudaStream_t s) {
  const int seqs = a.seq_end - a.seq_begin;
  if (seqs <= 0) return cudaSuccess;
  const int G = a.nq_l / a.nkv_l;
  dim3 grid(seqs * a.n * a.nkv_l, a.splits);
#define TP_DEC(HD_, G_) \
  if (a.hd == HD_ && G == G_) { attn_decode_kernel<HD_, G_><<<grid, 128, 0, s>>>(a); return cudaGetLastError(); }
  TP_DEC(128, 1) TP_DEC(128, 2) TP_DEC(128, 4) TP_DEC(128, 8)
  TP_DEC(64, 1) TP_DEC(64, 2) TP_DEC(64, 4) TP_DEC(64, 8)
#undef TP_DEC
  return cudaErrorNotSupported;
}

// ---------------------------------------------------------------------------
// Prefill (several new tokens per sequence, causal with cache offset):
// flash-attention style on the tensor cores with m16n8k16 fp16 MMA (fp32
// accumulate).  One CTA = 64 queries of one (sequence, rank, q head), 4 warps
// x 16 query rows; K/V blocks of 64 keys double-buffered in shared memory by
// cp.async (rows beyond the sequence zero-filled), converted from the bf16
// cache to fp16 in place (exact in fp16's normal range).
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int HD>
struct PrefillCfg {
  static constexpr int BQ = 64, BK = 64;
  static constexpr int LD = HD + 8;  // padded smem row (elements): conflict-free ldmatrix
  static constexpr int TILE = BK * LD;
  static constexpr int SMEM = (BQ * LD + 4 * TILE) * 2;
};

template <int HD>
__global__ void __launch_bounds__(128) attn_prefill_kernel(AttnArgs a) {
  using C = PrefillCfg<HD>;
  constexpr int BQ = C::BQ, BK = C::BK, LD = C::LD;
  constexpr int KSTEPS = HD / 16;  // k-steps of the QK^T product
  constexpr int NT_O = HD / 8;     // n-tiles of the output
  extern __shared__ __align__(16) __half sm[];
  __half* sQ = sm;
  __half* sK = sm + BQ * LD;          // [2][BK][LD]
  __half* sV = sK + 2 * C::TILE;      // [2][BK][LD]

  const int b = a.seq_begin + blockIdx.z;
  const int qlen = a.cu_q[b + 1] - a.cu_q[b];
  const int q0 = (gridDim.x - 1 - blockIdx.x) * BQ;  // heaviest blocks first
  if (q0 >= qlen) return;
  const int hg = blockIdx.y;
  const int r = hg / a.nq_l, h = hg % a.nq_l;
  const int G = a.nq_l / a.nkv_l;
  const int g = h / G;
  const int ctx = a.ctx_len[b];
  const int tbase = a.cu_q[b];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const size_t plane = static_cast<size_t>(a.max_seqs) * a.nkv_l * a.cap * HD;
  const size_t head_off = (static_cast<size_t>(a.slot[b]) * a.nkv_l + g) * a.cap * HD;
  const __nv_bfloat16* Kc = reinterpret_cast<const __nv_bfloat16*>(a.kv) + (2 * static_cast<size_t>(r)) * plane + head_off;
  const __nv_bfloat16* Vc = reinterpret_cast<const __nv_bfloat16*>(a.kv) + (2 * static_cast<size_t>(r) + 1) * plane + head_off;

  // Q tile
  constexpr int CPR = HD / 8;  // 16-byte chunks per row
  for (int c = threadIdx.x; c < BQ * CPR; c += 128) {
    const int row = c / CPR, col = (c % CPR) * 8;
    const int qi = q0 + row;
    const __half* src = reinterpret_cast<const __half*>(a.qkv) +
                        static_cast<size_t>(tbase + min(qi, qlen - 1)) * a.n * a.w_rank +
                        static_cast<size_t>(r) * a.w_rank + h * HD + col;
    cp_async16(smem_u32(sQ + row * LD + col), src, qi < qlen);
  }
  const int kend = ctx + min(q0 + BQ, qlen);  // keys needed by this CTA
  const int nblocks = (kend + BK - 1) / BK;
  auto load_kv = [&](int blk, int buf) {
    for (int c = threadIdx.x; c < BK * CPR; c += 128) {
      const int row = c / CPR, col = (c % CPR) * 8;
      const int key = blk * BK + row;
      const bool ok = key < kend;
      const size_t off = static_cast<size_t>(ok ? key : 0) * HD + col;
      cp_async16(smem_u32(sK + buf * C::TILE + row * LD + col), Kc + off, ok);
      cp_async16(smem_u32(sV + buf * C::TILE + row * LD + col), Vc + off, ok);
    }
  };
  // the chunks this thread loaded, turned from bf16 into fp16 in place once they landed
  auto convert_kv = [&](int buf) {
    for (int c = threadIdx.x; c < BK * CPR; c += 128) {
      const int row = c / CPR, col = (c % CPR) * 8;
      uint4* pk = reinterpret_cast<uint4*>(sK + buf * C::TILE + row * LD + col);
      uint4* pv = reinterpret_cast<uint4*>(sV + buf * C::TILE + row * LD + col);
      uint4 k = *pk, v = *pv;
      k.x = pack_f16x2(bf16lo(k.x), bf16hi(k.x)); k.y = pack_f16x2(bf16lo(k.y), bf16hi(k.y));
      k.z = pack_f16x2(bf16lo(k.z), bf16hi(k.z)); k.w = pack_f16x2(bf16lo(k.w), bf16hi(k.w));
      v.x = pack_f16x2(bf16lo(v.x), bf16hi(v.x)); v.y = pack_f16x2(bf16lo(v.y), bf16hi(v.y));
      v.z = pack_f16x2(bf16lo(v.z), bf16hi(v.z)); v.w = pack_f16x2(bf16lo(v.w), bf16hi(v.w));
      *pk = k;
      *pv = v;
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  float o[NT_O][4];
#pragma unroll
  for (int i = 0; i < NT_O; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.0f, 0.0f};
  uint32_t qa[KSTEPS][4];
  const int qrow0 = q0 + warp * 16 + (lane >> 2);  // query index of c0/c1; +8 for c2/c3

  for (int blk = 0; blk < nblocks; ++blk) {
    const int buf = blk & 1;
    if (blk + 1 < nblocks) load_kv(blk + 1, buf ^ 1);
    cp_async_commit();
    cp_async_wait<1>();
    convert_kv(buf);
    __syncthreads();
    if (blk == 0) {
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const uint32_t addr = smem_u32(sQ + (warp * 16 + (lane & 15)) * LD + kk * 16 + (lane >> 4) * 8);
        ldsm_x4(addr, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
    }
    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
    const __half* kt = sK + buf * C::TILE;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int kk = 0; kk < KSTEPS; kk += 2) {
        uint32_t b0, b1, b2, b3;
        const uint32_t addr = smem_u32(kt + (j * 8 + (lane & 7)) * LD + kk * 16 + (lane >> 3) * 8);
        ldsm_x4(addr, b0, b1, b2, b3);
        mma16816(s[j], qa[kk], b0, b1);
        mma16816(s[j], qa[kk + 1], b2, b3);
      }
    }
    // scale, mask, online softmax (exp2 domain)
    float bmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = blk * BK + j * 8 + (lane & 3) * 2 + (e & 1);
        const int qi = qrow0 + (e >> 1) * 8;
        const bool vis = (qi < qlen) && (key <= ctx + qi);
        const float v = vis ? s[j][e] * a.scale_log2 : -INFINITY;
        s[j][e] = v;
        bmax[e >> 1] = fmaxf(bmax[e >> 1], v);
      }
    }
    float corr[2], mbase[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      bmax[i] = fmaxf(bmax[i], __shfl_xor_sync(0xffffffffu, bmax[i], 1));
      bmax[i] = fmaxf(bmax[i], __shfl_xor_sync(0xffffffffu, bmax[i], 2));
      const float mn = fmaxf(mrow[i], bmax[i]);
      mbase[i] = (mn == -INFINITY) ? 0.0f : mn;
      corr[i] = exp2f(mrow[i] - mbase[i]);
      mrow[i] = mn;
    }
    float psum[2] = {0.0f, 0.0f};
    uint32_t pa[4][4];  // P as A fragments: 4 k-steps of 16 keys
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float p0 = exp2f(s[j][0] - mbase[0]), p1 = exp2f(s[j][1] - mbase[0]);
      const float p2 = exp2f(s[j][2] - mbase[1]), p3 = exp2f(s[j][3] - mbase[1]);
      psum[0] += p0 + p1;
      psum[1] += p2 + p3;
      __half2 h01 = __floats2half2_rn(p0, p1), h23 = __floats2half2_rn(p2, p3);  // P in [0, 1]
      pa[j >> 1][(j & 1) * 2 + 0] = *reinterpret_cast<uint32_t*>(&h01);
      pa[j >> 1][(j & 1) * 2 + 1] = *reinterpret_cast<uint32_t*>(&h23);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      psum[i] += __shfl_xor_sync(0xffffffffu, psum[i], 1);
      psum[i] += __shfl_xor_sync(0xffffffffu, psum[i], 2);
      lrow[i] = lrow[i] * corr[i] + psum[i];
    }
#pragma unroll
    for (int i = 0; i < NT_O; ++i) {
      o[i][0] *= corr[0];
      o[i][1] *= corr[0];
      o[i][2] *= corr[1];
      o[i][3] *= corr[1];
    }
    // O += P V
    const __half* vt = sV + buf * C::TILE;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t afr[4] = {pa[kk][0], pa[kk][1], pa[kk][2], pa[kk][3]};
#pragma unroll
      for (int nt = 0; nt < NT_O; nt += 2) {
        uint32_t b0, b1, b2, b3;
        const uint32_t addr =
            smem_u32(vt + (kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + nt * 8 + (lane >> 4) * 8);
        ldsm_x4_t(addr, b0, b1, b2, b3);
        mma16816(o[nt], afr, b0, b1);
        mma16816(o[nt + 1], afr, b2, b3);
      }
    }
    __syncthreads();
  }
  // normalise and store
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int qi = qrow0 + i * 8;
    if (qi >= qlen) continue;
    const float inv = 1.0f / lrow[i];
    __half* orow = reinterpret_cast<__half*>(a.out) + static_cast<size_t>(tbase + qi) * a.n * a.nq_l * HD +
                   (static_cast<size_t>(r) * a.nq_l + h) * HD;
#pragma unroll
    for (int nt = 0; nt < NT_O; ++nt) {
      const int d = nt * 8 + (lane & 3) * 2;
      *reinterpret_cast<uint32_t*>(orow + d) = pack_f16x2(o[nt][i * 2] * inv, o[nt][i * 2 + 1] * inv);
    }
  }
}

cudaError_t launch_attention_prefill(const AttnArgs& a, cudaStream_t s) {
  const int seqs = a.seq_end - a.seq_begin;
  if (seqs <= 0 || a.max_q_len <= 0) return cudaSuccess;
  dim3 grid((a.max_q_len + 63) / 64, a.n * a.nq_l, seqs);
  if (a.hd == 128) {
    constexpr int smem = PrefillCfg<128>::SMEM;
    static bool attr = false;
    if (!attr) {
      cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      attr = true;
    }
    attn_prefill_kernel<128><<<grid, 128, smem, s>>>(a);
  } else if (a.hd == 64) {
    constexpr int smem = PrefillCfg<64>::SMEM;
    static bool attr = false;
    if (!attr) {
      cudaError_t e = cudaFuncSetAttribute(attn_prefill_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      attr = true;
    }
    attn_prefill_kernel<64><<<grid, 128, smem, s>>>(a);
  } else {
    return cudaErrorNotSupported;
  }
  return cudaGetLastError();
}

}  // namespace tpk
