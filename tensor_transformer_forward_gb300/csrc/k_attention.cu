// Per-rank GQA attention over the rank's KV cache ("Tensor parallelism from
// scratch", tp.py TPAttention.forward and section "KV heads and the limit on
// TP"): each rank attends with its nq_l query heads over its nkv_l kv heads;
// local q head h reads local kv head h / (nq_l / nkv_l) (repeat_interleave);
// scores are scaled by 1/sqrt(hd); new token j of a sequence with ctx cached
// tokens sees keys 0 .. ctx + j.  Softmax in fp32 (base-2, max-subtracted).
//
// Cache layout (per layer): [n][2 (K, V)][blocks][nkv_l][block_len][hd] bf16, a
// block being a sequence slot of a contiguous cache or a page of a paged one (the
// batch's block table maps (sequence, position / block_len) to a block).  q comes
// from the merged QKV buffer: fp16 for decode tokens (fp32 math), bf16 high +
// low parts for prefill tokens (bf16 tensor-core operands next to the bf16
// cache).  Output layout: [T][n * nq_l * hd] fp16 (rank-major heads, the
// row-split o_proj operand).
#include <climits>

#include "kernels.h"
#include "sm100.cuh"

namespace tpk {

// 2^x for the softmax numerators (hardware approximation, results below 2^-126
// flush to zero: such terms are far below the bf16 rounding of P)
__device__ __forceinline__ float ex2_ftz(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// paired fp32 arithmetic (two lanes of one 64-bit register)
__device__ __forceinline__ uint64_t f32x2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// Item i of a decode launch: its (sequence, rank, kv head) unit, its key split
// and the unit's split count, walking the plan's levels in order (a unit's
// items are consecutive).
struct DecCta {
  int unit, split, nsplit;
};
__device__ __forceinline__ DecCta dec_cta(const AttnArgs& a, int i) {
  DecCta c{0, 0, 1};
  int u0 = 0;
#pragma unroll
  for (int l = 0; l < kDecLevels; ++l) {
    const int s = a.plan.splits[l], n = a.plan.units[l] * s;
    if (i < n) {
      c.unit = u0 + i / s;
      c.split = i % s;
      c.nsplit = s;
      return c;
    }
    i -= n;
    u0 += a.plan.units[l];
  }
  return c;
}
// partials per unit in the split workspace
__device__ __forceinline__ int dec_part_stride(const AttnArgs& a) { return plan_max_splits(a.plan); }

// ---------------------------------------------------------------------------
// Decode (one new token per sequence): flash-decoding split over the keys.
// One CTA = (sequence, rank, local kv head, key split).  Warp 4 streams the
// split's K and V rows (contiguous in the cache) into a 4-stage shared-memory
// ring with bulk copies; warps 0-3 compute from shared memory.  The G query
// heads of the kv group share every K/V row.  Lanes split head_dim in 16-byte
// pieces (hd/8 lanes per key); each half-warp-sized lane group takes one key,
// a warp covers 32/(hd/8) keys per step, and the online-softmax correction is
// applied once per 4 such steps.  Splits combine through an fp32 workspace;
// the last CTA of a (seq, rank, head) to finish (atomic counter, no waiting)
// merges them in split order.
// ---------------------------------------------------------------------------
template <int HD>
struct DecCfg {
  static constexpr int CK = HD == 128 ? 32 : 64;      // keys per ring stage (16 KB of K + V)
  static constexpr int STAGES = 4;
  static constexpr int ROW = HD * 2;                  // bytes per key row
  static constexpr int STAGE_BYTES = 2 * CK * ROW;    // K then V
  static constexpr int SMEM = STAGES * STAGE_BYTES + 128;
};

template <int HD, int G>
__global__ void __launch_bounds__(160) attn_decode_kernel(AttnArgs a) {
  using C = DecCfg<HD>;
  constexpr int LPK = HD / 8;        // lanes per key
  constexpr int KPI = 32 / LPK;      // keys per warp step
  constexpr int U = 4;               // warp steps per softmax correction
  extern __shared__ __align__(128) uint8_t dsm[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(dsm + C::STAGES * C::STAGE_BYTES);  // full[4], empty[4]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * C::STAGES);
  const uint32_t bar0 = smem_u32(bars);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int ks = lane / LPK, dc = lane % LPK;
  const int per_seq = a.n * a.nkv_l;
  const DecCta cta = dec_cta(a, blockIdx.x);
  const int unit = cta.unit, split = cta.split, nsplit = cta.nsplit, pstride = dec_part_stride(a);
  const int b = a.seq_begin + unit / per_seq;
  const int r = (unit % per_seq) / a.nkv_l;
  const int g = unit % a.nkv_l;
  const int t = a.cu_q[b];
  const int L = a.ctx_len[b] + 1;
  // splits start on kKeyAlign-key boundaries (pages hold whole chunks)
  const int chunk = ((L + nsplit - 1) / nsplit + kKeyAlign - 1) / kKeyAlign * kKeyAlign;
  const int k0 = split * chunk;
  const int k1n = min(L, k0 + chunk);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar0 + 8u * s, 1);
      mbar_init(bar0 + 8u * (C::STAGES + s), 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  // a split whose keys lie (partly) outside the cache reads nothing (zero output)
  // and flags the batch
  const bool bad = __syncthreads_or(L < 1 || kv_blocks_bad(a.kvm, b, k0, k1n, threadIdx.x, blockDim.x));
  const int k1 = bad ? k0 : k1n;
  const int nchunks = k1 > k0 ? (k1 - k0 + C::CK - 1) / C::CK : 0;
  const __nv_bfloat16* kvb = reinterpret_cast<const __nv_bfloat16*>(a.kv);
  // the batch arrays are the host's; q and the cache come from earlier kernels
  griddep_wait();
  griddep_launch();
  if (bad && threadIdx.x == 0) raise_flag(a.status, TP_DEVFLAG_BAD_TOKEN);

  // per-lane state for the warp's keys: G heads x (m, l, acc[8])
  float m[G], l[G], acc[G][8];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[h][i] = 0.0f;
  }

  if (warp == 4) {
    // ---------------- bulk-copy producer ----------------
    if (lane == 0) {
      int issued = 0;
      // block of the next chunk, looked up one chunk ahead (its load overlaps the wait)
      int blk_next = nchunks > 0 ? kv_block_checked(a.kvm, b, k0) : 0;
      for (int c = 0; c < nchunks; ++c) {
        const int s = c % C::STAGES;
        const int key = k0 + c * C::CK;
        const int blk = blk_next;
        if (c + 1 < nchunks) blk_next = kv_block_checked(a.kvm, b, key + C::CK);
        if (!mbar_wait(bar0 + 8u * (C::STAGES + s), ((c / C::STAGES) & 1) ^ 1u, abort_flag, a.status)) break;
        const uint32_t bytes = static_cast<uint32_t>(min(C::CK, k1 - key)) * C::ROW;
        const uint32_t full = bar0 + 8u * s;
        mbar_arrive_expect_tx(full, 2 * bytes);
        uint8_t* st = dsm + s * C::STAGE_BYTES;
        const int brow = key % a.kvm.block_len;
        bulk_load(smem_u32(st), kvb + kv_row(a.kvm, a.nkv_l, r, 0, blk, g, brow) * HD, bytes, full);
        bulk_load(smem_u32(st + C::CK * C::ROW), kvb + kv_row(a.kvm, a.nkv_l, r, 1, blk, g, brow) * HD, bytes, full);
        issued = c + 1;
      }
      for (int c = (issued > C::STAGES ? issued - C::STAGES : 0); c < issued; ++c)
        mbar_wait(bar0 + 8u * (c % C::STAGES), (c / C::STAGES) & 1, nullptr, a.status);
    }
  } else {
    // ---------------- compute warps 0..3 ----------------
    // this lane's 8 dims of each query head (fp16 q), pre-scaled into the exp2 domain
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
    for (int c = 0; c < nchunks; ++c) {
      const int s = c % C::STAGES;
      if (!mbar_wait(bar0 + 8u * s, (c / C::STAGES) & 1, abort_flag, a.status)) break;
      const uint8_t* st = dsm + s * C::STAGE_BYTES;
      const int nk = min(C::CK, k1 - (k0 + c * C::CK));
      // this warp's keys of the chunk: warp * (CK/4) .. + CK/4, KPI per step, U steps per correction
      constexpr int KW = C::CK / 4;
      static_assert(KW % (KPI * U) == 0, "a warp's share of a chunk is whole correction groups");
      for (int base = warp * KW; base < warp * KW + KW; base += KPI * U) {
        float sc[G][U];
        uint4 vv[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int kk = base + u * KPI + ks;
          const bool valid = kk < nk;  // uniform across the LPK lanes of this key
          const uint4 kr = *reinterpret_cast<const uint4*>(st + kk * C::ROW + dc * 16);
          // rows past the chunk's end hold stale bytes: V is zeroed so 0 * NaN cannot occur
          vv[u] = valid ? *reinterpret_cast<const uint4*>(st + C::CK * C::ROW + kk * C::ROW + dc * 16)
                        : make_uint4(0u, 0u, 0u, 0u);
          const float kf[8] = {bf16lo(kr.x), bf16hi(kr.x), bf16lo(kr.y), bf16hi(kr.y),
                               bf16lo(kr.z), bf16hi(kr.z), bf16lo(kr.w), bf16hi(kr.w)};
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float d = 0.0f;
#pragma unroll
            for (int i = 0; i < 8; ++i) d += q[h][i] * kf[i];
#pragma unroll
            for (int o = LPK / 2; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            sc[h][u] = valid ? d : -INFINITY;
          }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float mx = sc[h][0];
#pragma unroll
          for (int u = 1; u < U; ++u) mx = fmaxf(mx, sc[h][u]);
          const float mn = fmaxf(m[h], mx);
          if (mn == -INFINITY) continue;  // nothing valid yet
          const float corr = exp2f(m[h] - mn);
          l[h] *= corr;
#pragma unroll
          for (int i = 0; i < 8; ++i) acc[h][i] *= corr;
#pragma unroll
          for (int u = 0; u < U; ++u) {
            const float pu = exp2f(sc[h][u] - mn);
            l[h] += pu;
            const float vf[8] = {bf16lo(vv[u].x), bf16hi(vv[u].x), bf16lo(vv[u].y), bf16hi(vv[u].y),
                                 bf16lo(vv[u].z), bf16hi(vv[u].z), bf16lo(vv[u].w), bf16hi(vv[u].w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[h][i] += pu * vf[i];
          }
          m[h] = mn;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar0 + 8u * (C::STAGES + s));
    }
  }

  // merge the KPI key groups of each compute warp (lanes with the same dims)
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
  // merge the 4 compute warps through shared memory (reusing the ring): [warp][h][HD + 2]
  __syncthreads();
  float (*red)[G][HD + 2] = reinterpret_cast<float (*)[G][HD + 2]>(dsm);
  __shared__ int last_flag;
  if (warp < 4 && ks == 0) {
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
  const int unit_heads = G * HD;
  float* part = a.part + (static_cast<size_t>(unit) * pstride + split) * G * (HD + 2);
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
    if (nsplit == 1) {
      __half* o = reinterpret_cast<__half*>(a.out) + static_cast<size_t>(t) * a.n * a.nq_l * HD +
                  (static_cast<size_t>(r) * a.nq_l + g * G + h) * HD + d;
      uint32_t sat = 0;
      *o = to_f16(ll > 0.0f ? aa / ll : 0.0f, sat);
      report_sat(a.status, sat);
    } else {
      part[h * (HD + 2) + d] = aa;
      if (d == 0) {
        part[h * (HD + 2) + HD] = mm;
        part[h * (HD + 2) + HD + 1] = ll;
      }
    }
  }
  if (nsplit == 1) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int old = atomicAdd(a.counters + unit, 1);
    last_flag = (old == nsplit - 1);
  }
  __syncthreads();
  if (!last_flag) return;
  __threadfence();
  const float* pbase = a.part + static_cast<size_t>(unit) * pstride * G * (HD + 2);
  for (int e = threadIdx.x; e < unit_heads; e += blockDim.x) {
    const int h = e / HD, d = e % HD;
    float mm = -INFINITY, ll = 0.0f, aa = 0.0f;
    for (int sp = 0; sp < nsplit; ++sp) {
      const float* ps = pbase + (static_cast<size_t>(sp) * G + h) * (HD + 2);
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
    uint32_t sat = 0;
    *o = to_f16(ll > 0.0f ? aa / ll : 0.0f, sat);
    report_sat(a.status, sat);
  }
  if (threadIdx.x == 0) a.counters[unit] = 0;
}

template <int HD, int G>
static cudaError_t prepare_decode(int* ctas_per_sm) {
  static PerDevice pd;  // the attribute and the occupancy, once per device
  int dev = -1, occ = 0;
  if (!per_device_ready(pd, &dev, &occ)) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DecCfg<HD>::SMEM);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_decode_kernel<HD, G>, 160, DecCfg<HD>::SMEM);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    per_device_mark(pd, dev, occ);
  }
  *ctas_per_sm = occ;
  return cudaSuccess;
}

template <int HD, int G>
static cudaError_t launch_decode_tc_hd(const AttnArgs& a, cudaStream_t s);
static cudaError_t decode_tc_ctas_per_sm(int G, int* per_sm);

// Key splits per (sequence, rank, kv head).  CUDA-core kernel (64-dim heads): the
// count that minimises waves(units * s / resident CTAs) * (keys per split + fixed
// cost), so that the grid fills whole waves.  Tensor-core kernel (128-dim heads),
// which streams K and V at the HBM rate: a wave of c CTAs takes as long as
// max(c, nsat) CTAs' shares of the bytes, nsat being the CTAs that keep HBM
// saturated, and each CTA adds about 1.25 key tiles of fixed work (set-up, the split
// merge); minimised over s is
//   sum over waves of (key tiles per split + 1.25) * max(CTAs in the wave, nsat).
// nsat = 0.36 x the resident CTAs (one per SM here, by the occupancy query) and the
// 1.25 tiles fit split sweeps of 64 sequences x 4097 keys (tp 2) and 32 x 2049
// (tp 16), 512 units each: 1 split was best in both, 161 / 91 us against 177 / 109 us
// with 2 and more with 3, 4 or 6.  Ties go to fewer splits.
static int decode_splits(int max_kv_len, int num_units, int num_sms, int hd, int G, int max_splits) {
  int per_sm = 1;
  cudaError_t e = cudaErrorNotSupported;
#define TP_OCC(HD_, G_) \
  if (hd == HD_ && G == G_) e = prepare_decode<HD_, G_>(&per_sm);
  TP_OCC(128, 1) TP_OCC(128, 2) TP_OCC(128, 4) TP_OCC(128, 8)
  TP_OCC(64, 1) TP_OCC(64, 2) TP_OCC(64, 4) TP_OCC(64, 8)
#undef TP_OCC
  // 128-dim heads run on the tensor-core kernel, with its own occupancy
  if (hd == 128) e = decode_tc_ctas_per_sm(G, &per_sm);
  const int gran = 1, fixed = 96;
  if (e != cudaSuccess) per_sm = 1;
  const long long resident = static_cast<long long>(num_sms) * per_sm;
  const int units = num_units > 0 ? num_units : 1;
  int limit = max_kv_len / 32;
  if (limit > max_splits) limit = max_splits;
  if (limit > 64) limit = 64;
  if (limit < 1) limit = 1;
  int best = 1;
  long long best_cost = -1;
  if (hd == 128) {
    const long long tiles = (static_cast<long long>(max_kv_len) + 127) / 128;
    if (limit > tiles) limit = static_cast<int>(tiles);  // every split holds a key tile
    if (limit < 1) limit = 1;
    long long nsat = resident * 36 / 100;
    if (nsat < 1) nsat = 1;
    for (int s = 1; s <= limit; ++s) {
      const long long t = ((max_kv_len + s - 1) / s + 127) / 128;  // key tiles per split
      const long long ctas = static_cast<long long>(units) * s;
      const long long full = ctas / resident, rem = ctas % resident;
      const long long weight = full * (resident > nsat ? resident : nsat) + (rem > 0 ? (rem > nsat ? rem : nsat) : 0);
      const long long cost = (4 * t + 5) * weight;  // (tiles + 1.25) * weight, x4
      if (best_cost < 0 || cost < best_cost) {
        best_cost = cost;
        best = s;
      }
    }
    return best;
  }
  for (int s = 1; s <= limit; ++s) {
    const long long waves = (static_cast<long long>(units) * s + resident - 1) / resident;
    const long long per_split = ((max_kv_len + s - 1) / s + gran - 1) / gran * gran;
    const long long cost = waves * (per_split + fixed);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

template <int HD, int G>
static cudaError_t launch_decode_hd(const AttnArgs& a, dim3 grid, cudaStream_t s) {
  int per_sm = 0;
  cudaError_t e = prepare_decode<HD, G>(&per_sm);  // sets the shared-memory attribute once
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_decode_kernel<HD, G>, grid, dim3(160), DecCfg<HD>::SMEM, s, a);
}

cudaError_t launch_attention_decode(const AttnArgs& a, cudaStream_t s) {
  const int seqs = a.seq_end - a.seq_begin;
  if (seqs <= 0) return cudaSuccess;
  const int G = a.nq_l / a.nkv_l;
  const int units = seqs * a.n * a.nkv_l;
  for (int l = 0; l < kDecLevels; ++l)
    if (a.plan.units[l] < 0 || a.plan.splits[l] < 1) return cudaErrorInvalidValue;
  if (plan_units(a.plan) != units) return cudaErrorInvalidValue;
  dim3 grid(plan_items(a.plan));
#define TP_DEC_TC(HD_, G_) \
  if (a.hd == HD_ && G == G_) return launch_decode_tc_hd<HD_, G_>(a, s);
#define TP_DEC(HD_, G_) \
  if (a.hd == HD_ && G == G_) return launch_decode_hd<HD_, G_>(a, grid, s);
  TP_DEC_TC(128, 1) TP_DEC_TC(128, 2) TP_DEC_TC(128, 4) TP_DEC_TC(128, 8)
  TP_DEC(64, 1) TP_DEC(64, 2) TP_DEC(64, 4) TP_DEC(64, 8)
#undef TP_DEC
#undef TP_DEC_TC
  return cudaErrorNotSupported;
}

// ---------------------------------------------------------------------------
// Decode on the tensor cores, persistent.  Work items are the (sequence, rank,
// local kv head, key split) pieces of dec_cta, handed out in order from a ticket
// counter; each CTA keeps drawing items until none are left, and its K / V
// streams, MMAs and softmax run on from one item into the next without draining
// (a CTA per item left every SM idle while one pair of CTAs ended and the next
// started, and a last partial wave of items ran on part of the GPU).  One CTA
// per SM (its shared memory fills the SM, so a launch can leave whole SMs to
// another kernel), 512 threads: two independent pipelines of 8 warps, each
// drawing its own items.  A pipeline's warps:
//   warp 0    scheduler: draws the next ticket three K tiles before the current
//             item's K stream ends, checks the item's cache blocks, publishes
//             it in a 4-entry item ring, loads its query into registers and
//             writes it as Q^T (bf16 high and low parts, the MMA's B operand)
//             once the previous item's S MMAs are done
//   warp 1    (pipeline 0: TMEM allocation for both) one MMA-issuing thread
//   warps 2-5 softmax, one thread per key of a 128-key tile; at the end of an
//             item, O (one TMEM row per output dim) into a staging buffer
//   warp 6    lane 0 streams K, lane 1 V through rings of 16 KB slots (two
//             per tile; see DtcCfg)
//   warp 7    writer: the staged output as fp16, or a split's partial and, for
//             the last split of a unit to arrive, the merge of its splits in
//             split order (so the softmax never waits on global memory)
//   S^T = K Q^T   M = 128 keys, N = 16, K = head_dim: the B operand holds the
//                 G query heads of the kv group as bf16 high parts (rows 0..G-1)
//                 and bf16 low parts (rows G..2G-1), so S = S_hi + S_lo carries q
//                 to ~16 significant bits against the bf16 cache
//   O^T += V^T P^T   M = head_dim (V read MN-major from its TMA tile), N = 16,
//                 K = 128 keys; P^T ([head][key]) written by the softmax as bf16
//                 high parts (rows 0..G-1) and low parts (rows G..2G-1), summed
//                 at the end, so P also keeps ~16 significant bits
// S^T and P^T are double-buffered; the output is rescaled only when a head's
// running max grows by more than 2^8.  Ring phases count tiles and items over
// the whole launch, so every role sees the same sequence of phases.  The result
// does not depend on which CTA takes an item: an item's arithmetic is fixed, and
// splits merge in split order.
// ---------------------------------------------------------------------------
template <int HD, int G>
struct DtcCfg {
  static constexpr int BK = 128;                   // keys per tile
  static constexpr int NSUB = HD / 64;             // 64-dim sub-tiles
  static constexpr int SUB_BYTES = BK * 128;       // [128 keys][64 dims] bf16
  static constexpr int KT_BYTES = NSUB * SUB_BYTES;
  static constexpr int QSUB = 16 * 128;            // [16 rows][64 dims] bf16
  static constexpr int QT_BYTES = NSUB * QSUB;
  static constexpr int PT_BYTES = 2 * QSUB;        // [16 heads][128 keys] bf16 (two 64-key sub-tiles)
  // K and V stream through rings of 16 KB slots: a K tile is two slots of 64
  // head dims ([128 keys][64 dims]), a V tile two slots of 64 keys ([64 keys]
  // [2 x 64 dims]).  Three slots per ring (where both pipelines' share fits: up
  // to 4 heads per kv group) keep 1.5 tiles of each in flight per pipeline, so a
  // pipeline does not wait a whole load latency per tile for the V slot its
  // last PV MMA frees.
  static constexpr int SLOT = 16384;
  static constexpr int VSUB = 8192;                // [64 keys][64 dims] of a V slot
  static constexpr int KSLOTS = G <= 4 ? 3 : 2;
  static constexpr int VSLOTS = G <= 4 ? 3 : 2;
  // a pipeline's operand tiles (1024-byte aligned: 128-byte swizzle atoms)
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = K_OFF + KSLOTS * SLOT;
  static constexpr int Q_OFF = V_OFF + VSLOTS * SLOT;   // Q^T
  static constexpr int P_OFF = Q_OFF + QT_BYTES;   // two P^T buffers
  static constexpr int BIG = P_OFF + 2 * PT_BYTES;
  // the rest of a pipeline's share, after both pipelines' operand tiles
  static constexpr int ST_BYTES = (G * (HD + 2) * 4 + 15) / 16 * 16;  // staged output of the G heads
  static constexpr int RED_OFF = 0;                // max then sum: [2][4 warps][8 heads] fp32 each
  static constexpr int ST_OFF = RED_OFF + 512;     // two staging buffers
  static constexpr int RING_OFF = ST_OFF + 2 * ST_BYTES;  // item ring: 4 x 32 bytes
  static constexpr int BAR_OFF = RING_OFF + 128;
  static constexpr int NBARS = 23 + 2 * KSLOTS + 2 * VSLOTS;
  static constexpr int SMALL = (BAR_OFF + NBARS * 8 + 8 + 15) / 16 * 16;  // + TMEM address, abort flag
  static constexpr int SMEM = 1024 + 2 * BIG + 2 * SMALL;
  static_assert(SMEM <= 232448, "two pipelines fit one SM's shared memory");
  static constexpr int S_COL = 0, O_COL = 32, PIPE_COLS = 64, TMEM_COLS = 128;
  static constexpr int THREADS = 512;  // two pipelines of 8 warps
};

// An item of the decode ring: its unit and split, the split's keys [k0, k1) and
// tile count (k1 = k0 when its cache blocks failed the check), its sequence and
// the token row of its query.
struct DecItem {
  int unit, split, nsplit, k0, k1, ntiles, b, t;
};

template <int HD, int G>
__global__ void __launch_bounds__(512, 1) attn_decode_tc_kernel(const __grid_constant__ CUtensorMap tmKV,
                                                                const __grid_constant__ CUtensorMap tmKV64,
                                                                const __grid_constant__ CUtensorMap tmKV16,
                                                                const AttnArgs a) {
  using C = DtcCfg<HD, G>;
  static_assert(2 * G <= 16, "hi and lo rows of the kv group fit N = 16");
  static_assert(HD == 128, "a K tile is two 64-dim slots");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem0 = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int pipe = threadIdx.x >> 8;  // warps 0-7 pipeline 0, warps 8-15 pipeline 1
  uint8_t* smem = smem0 + pipe * C::BIG;                       // operand tiles
  uint8_t* sm2 = smem0 + 2 * C::BIG + pipe * C::SMALL;          // the rest
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm2 + C::BAR_OFF);
  // barriers: 0-3 item full | 4-7 item empty | 8 q full | 9 q empty | 10,11 s full | 12,13 p full |
  // 14 pv done | 15 item's o done | 16,17 staging full | 18,19 staging empty | 20 next-item request |
  // 21 drain | 22 item's o read | then full and empty per K slot, per V slot
  // the TMEM address and the abort flag live in pipeline 0's share (one per CTA)
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(reinterpret_cast<uint64_t*>(smem0 + 2 * C::BIG + C::BAR_OFF) + C::NBARS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* red = reinterpret_cast<float*>(sm2 + C::RED_OFF);
  uint8_t* ring = sm2 + C::RING_OFF;
  const uint32_t bar0 = smem_u32(bars);
#define D_IF(s) (bar0 + 8u * (s))
#define D_IE(s) (bar0 + 8u * (4 + (s)))
#define D_QF (bar0 + 8u * 8)
#define D_QE (bar0 + 8u * 9)
#define D_SF(b) (bar0 + 8u * (10 + (b)))
#define D_PF(b) (bar0 + 8u * (12 + (b)))
#define D_OD (bar0 + 8u * 14)
#define D_OF (bar0 + 8u * 15)
#define D_STF(b) (bar0 + 8u * (16 + (b)))
#define D_STE(b) (bar0 + 8u * (18 + (b)))
#define D_NREQ (bar0 + 8u * 20)
#define D_DR (bar0 + 8u * 21)
#define D_OE (bar0 + 8u * 22)
#define D_KF(s) (bar0 + 8u * (23 + (s)))
#define D_KE(s) (bar0 + 8u * (23 + C::KSLOTS + (s)))
#define D_VF(s) (bar0 + 8u * (23 + 2 * C::KSLOTS + (s)))
#define D_VE(s) (bar0 + 8u * (23 + 2 * C::KSLOTS + C::VSLOTS + (s)))
  const int warp = (threadIdx.x >> 5) & 7, lane = threadIdx.x & 31;  // warp within the pipeline
  const int per_seq = a.n * a.nkv_l;
  const int units = (a.seq_end - a.seq_begin) * per_seq;
  const int items = plan_items(a.plan);
  const int pstride = dec_part_stride(a);

  if ((threadIdx.x & 255) == 0) {
    for (int i = 0; i < 4; ++i) {
      mbar_init(D_IF(i), 1);
      mbar_init(D_IE(i), 8);  // MMA, 4 softmax warps, K lane, V lane, writer
    }
    for (int i = 0; i < C::KSLOTS; ++i) {
      mbar_init(D_KF(i), 1);
      mbar_init(D_KE(i), 1);
    }
    for (int i = 0; i < C::VSLOTS; ++i) {
      mbar_init(D_VF(i), 1);
      mbar_init(D_VE(i), 1);
    }
    mbar_init(D_QF, 32);
    mbar_init(D_QE, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(D_SF(i), 1);
      mbar_init(D_PF(i), 4);
      mbar_init(D_STF(i), 128);
      mbar_init(D_STE(i), 32);
    }
    mbar_init(D_OD, 1);
    mbar_init(D_OF, 1);
    mbar_init(D_NREQ, 1);
    mbar_init(D_DR, 1);
    mbar_init(D_OE, 4);
    if (pipe == 0) *abort_flag = 0;
    fence_barrier_init();
  }
  if (threadIdx.x >> 5 == 1) {  // both pipelines' columns, 64 each
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  // Zero the V slots and Q^T: rows 2G..15 of Q^T stay zero, and a short tile
  // (at most 16 keys) loads 16 V rows only, so a first item of one short tile
  // would leave unwritten rows (their P is 0, and 0 * NaN would not vanish);
  // later short tiles find earlier tiles' rows there, which are finite cache values.
  for (int i = threadIdx.x & 255; i < (C::VSLOTS * C::SLOT + C::QT_BYTES) / 16; i += 256)
    *reinterpret_cast<uint4*>(smem + C::V_OFF + i * 16) = make_uint4(0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot + pipe * C::PIPE_COLS;
  const int nbar = 1 + pipe;  // the pipeline's named barrier for its softmax warps

  if (warp == 0) {
    // ---------------- scheduler: items, cache checks, query rows ----------------
    // The first item is drawn and checked before the dependency wait (the batch
    // tables do not come from the QKV GEMM); its query rows only after it.
    int tk = 0;
    if (lane == 0) tk = atomicAdd(a.sched, 1);
    tk = __shfl_sync(0xffffffffu, tk, 0);
    bool waited = false;
    for (int it = 0;; ++it) {
      DecItem e{-1, 0, 1, 0, 0, 0, 0, 0};
      bool bad_l = false;
      if (tk < items) {
        const DecCta c = dec_cta(a, tk);
        e.unit = c.unit;
        e.split = c.split;
        e.nsplit = c.nsplit;
        e.b = a.seq_begin + c.unit / per_seq;
        e.t = a.cu_q[e.b];
        const int L = a.ctx_len[e.b] + 1;
        // splits start on kKeyAlign-key boundaries (a page holds whole key tiles)
        const int chunk = ((L + e.nsplit - 1) / e.nsplit + kKeyAlign - 1) / kKeyAlign * kKeyAlign;
        e.k0 = e.split * chunk;
        e.k1 = min(L, e.k0 + chunk);
        // a split whose keys lie (partly) outside the cache reads nothing and flags the batch
        bad_l = L < 1 || kv_blocks_bad(a.kvm, e.b, e.k0, e.k1, lane, 32);
      }
      const bool bad = __any_sync(0xffffffffu, bad_l);
      if (bad || e.k1 < e.k0) e.k1 = e.k0;
      e.ntiles = (e.k1 - e.k0 + C::BK - 1) / C::BK;
      const int slot = it & 3;
      if (it >= 4 && !warp_all(mbar_wait(D_IE(slot), ((it >> 2) - 1) & 1, abort_flag, a.status))) break;
      if (lane == 0) {
        *reinterpret_cast<DecItem*>(ring + slot * 32) = e;
        mbar_arrive(D_IF(slot));
      }
      if (!waited) {
        griddep_wait();  // q and the cache come from the QKV GEMM
        griddep_launch();
        waited = true;
      }
      if (bad && lane == 0) raise_flag(a.status, TP_DEVFLAG_BAD_TOKEN);
      if (e.unit < 0) break;
      // the item's query into registers at once, into Q^T once the previous
      // item's S MMAs are done: rows 0..G-1 = bf16(q_h), rows G..2G-1 =
      // bf16(q_h - bf16(q_h)); 16-byte chunks in the 128-byte-swizzled K-major
      // layout of the MMA's B operand
      {
        constexpr int NQC = (G * (HD / 8) + 31) / 32;  // 8-dim chunks per lane
        const int r = (e.unit % per_seq) / a.nkv_l, g = e.unit % a.nkv_l;
        const __half* qrow = reinterpret_cast<const __half*>(a.qkv) + static_cast<size_t>(e.t) * a.n * a.w_rank +
                             static_cast<size_t>(r) * a.w_rank + static_cast<size_t>(g) * G * HD;
        uint4 qv[NQC];
#pragma unroll
        for (int k = 0; k < NQC; ++k) {
          const int i = lane + 32 * k;
          qv[k] = i < G * (HD / 8) ? __ldcg(reinterpret_cast<const uint4*>(qrow + i * 8)) : make_uint4(0u, 0u, 0u, 0u);
        }
        if (it >= 1 && !warp_all(mbar_wait(D_QE, (it - 1) & 1, abort_flag, a.status))) break;
        uint8_t* qt = smem + C::Q_OFF;
#pragma unroll
        for (int k = 0; k < NQC; ++k) {
          const int i = lane + 32 * k;
          if (i < G * (HD / 8)) {
            const int h = i / (HD / 8), c = i % (HD / 8);  // head, 8-dim chunk
            const uint4 u = qv[k];
            const float x[8] = {f16lo(u.x), f16hi(u.x), f16lo(u.y), f16hi(u.y),
                                f16lo(u.z), f16hi(u.z), f16lo(u.w), f16hi(u.w)};
            float lo[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) lo[j] = x[j] - bf2f(f2bf(x[j]));
            uint4 w;
            w.x = pack_bf16x2(x[0], x[1]); w.y = pack_bf16x2(x[2], x[3]);
            w.z = pack_bf16x2(x[4], x[5]); w.w = pack_bf16x2(x[6], x[7]);
            const int rl = G + h;
            *reinterpret_cast<uint4*>(qt + (c >> 3) * C::QSUB + h * 128 + (((c & 7) ^ (h & 7)) << 4)) = w;
            w.x = pack_bf16x2(lo[0], lo[1]); w.y = pack_bf16x2(lo[2], lo[3]);
            w.z = pack_bf16x2(lo[4], lo[5]); w.w = pack_bf16x2(lo[6], lo[7]);
            *reinterpret_cast<uint4*>(qt + (c >> 3) * C::QSUB + rl * 128 + (((c & 7) ^ (rl & 7)) << 4)) = w;
          }
        }
        fence_proxy_async_smem();
        mbar_arrive(D_QF);
      }
      // the next ticket a few K tiles before the item's K stream ends: late enough
      // that the items left go to whichever pipelines free up first, early enough
      // that the next item's first K tile follows the last one without a gap
      if (!warp_all(mbar_wait(D_NREQ, it & 1, abort_flag, a.status))) break;
      if (lane == 0) tk = atomicAdd(a.sched, 1);
      tk = __shfl_sync(0xffffffffu, tk, 0);
    }
    if (!waited) {
      griddep_wait();
      griddep_launch();
    }
  } else if (warp == 1) {
    griddep_wait();
    griddep_launch();
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, 16);                 // K (K-major) x Q^T (K-major)
      const uint32_t id_o = idesc_bf16_f32(128, 16, false, true);    // V^T (MN-major) x P^T (K-major)
      const uint32_t kt = smem_u32(smem + C::K_OFF), vt = smem_u32(smem + C::V_OFF);
      auto pv = [&](int g, bool first) -> bool {  // O^T (+)= V(g)^T P(g)^T, g counting tiles over the launch
        const int pb = g & 1;
        const int v0 = (2 * g) % C::VSLOTS, v1 = (2 * g + 1) % C::VSLOTS;  // the tile's two key halves
        if (!mbar_wait(D_PF(pb), (g >> 1) & 1, abort_flag, a.status)) return false;
        const uint32_t pt = smem_u32(smem + C::P_OFF + pb * C::PT_BYTES);
        // each key half as soon as it has landed; its slot frees when its MMAs are done
        for (int h = 0; h < 2; ++h) {
          const int vs = h ? v1 : v0;
          if (!mbar_wait(D_VF(vs), ((2 * g + h) / C::VSLOTS) & 1, abort_flag, a.status)) return false;
          tc_fence_after();
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4) {
            const int kk = 4 * h + k4;
            const uint64_t ad = sdesc_mn_sw128(vt + vs * C::SLOT + k4 * 16 * 128, C::VSUB, 1024);
            const uint64_t bd = sdesc_k_sw128(pt + h * C::QSUB) + 2ull * k4;
            tc_mma_f16(tmem + C::O_COL, ad, bd, id_o, (!first || kk > 0) ? 1u : 0u);
          }
          tc_commit(D_VE(vs));
        }
        tc_commit(D_OD);
        return true;
      };
      int jt = 0;  // tiles of the items before this one
      for (int it = 0;; ++it) {
        const int slot = it & 3;
        if (!mbar_wait(D_IF(slot), (it >> 2) & 1, abort_flag, a.status)) break;
        const DecItem e = *reinterpret_cast<const DecItem*>(ring + slot * 32);
        mbar_arrive(D_IE(slot));
        if (e.unit < 0) break;
        if (!mbar_wait(D_QF, it & 1, abort_flag, a.status)) break;
        tc_fence_after();
        const uint32_t qt = smem_u32(smem + C::Q_OFF);
        bool ok = true;
        for (int j = 0; j < e.ntiles; ++j) {
          const int g = jt + j, sb = g & 1;
          const int k0s = (2 * g) % C::KSLOTS, k1s = (2 * g + 1) % C::KSLOTS;  // the tile's two dim halves
          // score buffer sb last held S(g-2), read by the softmax before P(g-2) was ready;
          // each head-dim half as soon as it has landed, its slot free when its MMAs are done
          for (int h = 0; h < 2 && ok; ++h) {
            const int ks = h ? k1s : k0s;
            if (!mbar_wait(D_KF(ks), ((2 * g + h) / C::KSLOTS) & 1, abort_flag, a.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const int kk = 4 * h + k4;
              const uint64_t ad = sdesc_k_sw128(kt + ks * C::SLOT) + 2ull * k4;
              const uint64_t bd = sdesc_k_sw128(qt + h * C::QSUB) + 2ull * k4;
              tc_mma_f16(tmem + C::S_COL + sb * 16, ad, bd, id_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(D_KE(ks));
          }
          if (!ok) break;
          tc_commit(D_SF(sb));
          if (j == e.ntiles - 1) tc_commit(D_QE);  // Q^T is free once the item's last S is done
          if (j > 0 && !pv(g - 1, j == 1)) { ok = false; break; }
        }
        if (!ok) break;
        if (e.ntiles == 0) tc_commit(D_QE);  // no S MMAs: arrives once the earlier MMAs are done
        if (e.ntiles > 0 && !pv(jt + e.ntiles - 1, e.ntiles == 1)) break;
        // the softmax has read the previous item's output: without this an item
        // with no key tiles would complete the barrier a second time before the
        // softmax waited for the first (a parity wait cannot tell them apart)
        if (it > 0 && !mbar_wait(D_OE, (it - 1) & 1, abort_flag, a.status)) break;
        tc_commit(D_OF);      // the item's output is complete in TMEM
        jt += e.ntiles;
      }
      tc_commit(D_DR);  // completes after every MMA above
      mbar_wait(D_DR, 0, nullptr, a.status);
    }
  } else if (warp <= 5) {
    griddep_wait();
    griddep_launch();
    // ---------------- softmax, one thread per key of the tile (warps 2..5) ----------------
    const int q = (threadIdx.x >> 5) & 3;  // TMEM lane quarter (warps 2-5 and 10-13 cover all four)
    const int row = q * 32 + lane;    // key of the tile / output dim
    const int wq = warp - 2;          // 0..3 for the cross-warp reductions
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    int jt = 0;
    for (int it = 0;; ++it) {
      const int slot = it & 3;
      // the barrier also agrees on failed waits (named barriers have no time limit)
      const bool got = warp_all(mbar_wait(D_IF(slot), (it >> 2) & 1, abort_flag, a.status));
      if (!named_bar_and(nbar, 128, got)) break;
      const DecItem e = *reinterpret_cast<const DecItem*>(ring + slot * 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(D_IE(slot));
      if (e.unit < 0) break;
      float m[G], l[G];  // running max (exp2 domain) and sum per head: the same in every softmax thread
#pragma unroll
      for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.0f;
      }
      bool ok = true;
      for (int j = 0; j < e.ntiles; ++j) {
        const int g = jt + j, sb = g & 1;
        if (!warp_all(mbar_wait(D_SF(sb), (g >> 1) & 1, abort_flag, a.status))) ok = false;
        tc_fence_after();
        float sv[16];
        tc_ld16(lane_addr + C::S_COL + sb * 16, sv);
        const bool valid = e.k0 + j * C::BK + row < e.k1;
        float sc[G], mw[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          sc[h] = valid ? (sv[h] + sv[G + h]) * a.scale_log2 : -INFINITY;
          mw[h] = warp_max(sc[h]);
        }
        float* rmax = red + sb * 32;  // [4 warps][8 heads], alternating buffers
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) rmax[wq * 8 + h] = mw[h];
        }
        if (!named_bar_and(nbar, 128, ok)) { ok = false; break; }
        float mt[G], corr[G];
        bool rescale = false;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          mt[h] = fmaxf(fmaxf(rmax[h], rmax[8 + h]), fmaxf(rmax[16 + h], rmax[24 + h]));
          corr[h] = 1.0f;
          if (mt[h] > m[h] + 8.0f) {  // uniform across the block
            corr[h] = m[h] == -INFINITY ? 0.0f : exp2f(m[h] - mt[h]);
            m[h] = mt[h];
            rescale = true;
          }
        }
        float p[G], pw[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
          p[h] = exp2f(sc[h] - (m[h] == -INFINITY ? 0.0f : m[h]));
          pw[h] = warp_sum(p[h]);
        }
        float* rsum = red + 64 + sb * 32;  // the same for the sums
        if (lane == 0) {
#pragma unroll
          for (int h = 0; h < G; ++h) rsum[wq * 8 + h] = pw[h];
        }
        // P^T(g): key `row` of head h at row h, column row of the [16][128] tile
        uint8_t* pt = smem + C::P_OFF + sb * C::PT_BYTES + (row >> 6) * C::QSUB;
#pragma unroll
        for (int h = 0; h < G; ++h) {  // bf16 high part in row h, bf16 low part in row G + h
          const __nv_bfloat16 hi = f2bf(p[h]);
          const __nv_bfloat16 lo = f2bf(p[h] - bf2f(hi));
          const int rl = G + h;
          *reinterpret_cast<__nv_bfloat16*>(pt + h * 128 + ((((row & 63) >> 3) ^ (h & 7)) << 4) + (row & 7) * 2) = hi;
          *reinterpret_cast<__nv_bfloat16*>(pt + rl * 128 + ((((row & 63) >> 3) ^ (rl & 7)) << 4) + (row & 7) * 2) = lo;
        }
        named_bar_sync(nbar, 128);
#pragma unroll
        for (int h = 0; h < G; ++h) l[h] = l[h] * corr[h] + (rsum[h] + rsum[8 + h] + rsum[16 + h] + rsum[24 + h]);
        if (rescale && j > 0) {
          // O^T columns of the rescaled heads, once O += P(g-1) V(g-1) has completed
          // (S(g) done implies PV(g-2) done: the barrier is at phase g-1 or g)
          if (!warp_all(mbar_wait(D_OD, (g - 1) & 1, abort_flag, a.status))) ok = false;
          if (ok) {
            tc_fence_after();
            float ov[16];
            tc_ld16(lane_addr + C::O_COL, ov);
#pragma unroll
            for (int h = 0; h < G; ++h) {
              ov[h] *= corr[h];
              ov[G + h] *= corr[h];
            }
            tc_st16(lane_addr + C::O_COL, ov);
          }
        }
        if (!ok) continue;
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(D_PF(sb));
      }
      jt += e.ntiles;
      // the item's output (one O^T row per output dim) into staging buffer it & 1,
      // once the writer has emptied it (item it - 2)
      const int ob = it & 1;
      bool w = ok && warp_all(mbar_wait(D_OF, it & 1, abort_flag, a.status));
      if (w && it >= 2) w = warp_all(mbar_wait(D_STE(ob), ((it >> 1) - 1) & 1, abort_flag, a.status));
      if (!named_bar_and(nbar, 128, w)) break;
      tc_fence_after();
      float ov[16];
      tc_ld16(lane_addr + C::O_COL, ov);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(D_OE);
      float* st = reinterpret_cast<float*>(sm2 + C::ST_OFF + ob * C::ST_BYTES);
      if (row < HD) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float o = e.ntiles > 0 ? ov[h] + ov[G + h] : 0.0f;  // P V = P_hi V + P_lo V
          st[h * (HD + 2) + row] = e.nsplit == 1 ? (l[h] > 0.0f ? o / l[h] : 0.0f) : o;
          if (row == 0) {
            st[h * (HD + 2) + HD] = m[h];
            st[h * (HD + 2) + HD + 1] = l[h];
          }
        }
      }
      mbar_arrive(D_STF(ob));
    }
  } else if (warp == 6) {
    griddep_wait();
    griddep_launch();
    // ---------------- TMA: lane 0 streams K tiles, lane 1 V tiles ----------------
    if (lane < 2) {
      const bool is_k = lane == 0;
      tma_prefetch_desc(is_k ? &tmKV : &tmKV64);
      tma_prefetch_desc(&tmKV16);
      const int nsl = is_k ? C::KSLOTS : C::VSLOTS;
      int issued = 0;  // slots filled over the launch (two per tile)
      for (int it = 0;; ++it) {
        const int slot = it & 3;
        if (!mbar_wait(D_IF(slot), (it >> 2) & 1, abort_flag, a.status)) break;
        const DecItem e = *reinterpret_cast<const DecItem*>(ring + slot * 32);
        mbar_arrive(D_IE(slot));
        if (e.unit < 0) break;
        const int r = (e.unit % per_seq) / a.nkv_l, g = e.unit % a.nkv_l;
        bool ok = true;
        // block of the next tile, looked up one tile ahead (its load overlaps the wait)
        int blk_next = e.ntiles > 0 ? kv_block_checked(a.kvm, e.b, e.k0) : 0;
        for (int j = 0; j < e.ntiles; ++j) {
          const int key = e.k0 + j * C::BK;
          const int blk = blk_next;
          if (j + 1 < e.ntiles) blk_next = kv_block_checked(a.kvm, e.b, key + C::BK);
          // a last tile of at most 16 keys loads 16 rows (the typical ctx + 1 tail)
          const bool short_tail = j == e.ntiles - 1 && e.k1 - key <= 16;
          const int krow = static_cast<int>(kv_row(a.kvm, a.nkv_l, r, is_k ? 0 : 1, blk, g, key % a.kvm.block_len));
          // K: slot h = head dims [64h, 64h + 64) of the 128 keys; V: slot h = keys
          // [64h, 64h + 64) with both dim halves (a short tile fills half 0 only)
          for (int h = 0; h < 2; ++h) {
            const int sl = issued % nsl;
            const uint32_t full = is_k ? D_KF(sl) : D_VF(sl), empty = is_k ? D_KE(sl) : D_VE(sl);
            uint8_t* dst = smem + (is_k ? C::K_OFF : C::V_OFF) + sl * C::SLOT;
            if (!mbar_wait(empty, ((issued / nsl) & 1) ^ 1u, abort_flag, a.status)) { ok = false; break; }
            ++issued;
            if (is_k) {
              mbar_arrive_expect_tx(full, short_tail ? C::SLOT / 8 : C::SLOT);
              tma_load_2d(smem_u32(dst), short_tail ? &tmKV16 : &tmKV, full, h * 64, krow);
            } else if (!short_tail) {
              mbar_arrive_expect_tx(full, C::SLOT);
              for (int sub = 0; sub < 2; ++sub)
                tma_load_2d(smem_u32(dst + sub * C::VSUB), &tmKV64, full, sub * 64, krow + 64 * h);
            } else if (h == 0) {
              mbar_arrive_expect_tx(full, C::SLOT / 4);
              for (int sub = 0; sub < 2; ++sub)
                tma_load_2d(smem_u32(dst + sub * C::VSUB), &tmKV16, full, sub * 64, krow);
            } else {
              mbar_arrive(full);  // keys 64..127 of a short tile: none (P is 0 there)
            }
          }
          if (!ok) break;
          // the scheduler may draw the next item three tiles before this one's K
          // stream ends (drawing, decoding and checking it takes about as long)
          if (is_k && j == (e.ntiles > 3 ? e.ntiles - 3 : 0)) mbar_arrive(D_NREQ);
        }
        if (!ok) break;
        if (is_k && e.ntiles == 0) mbar_arrive(D_NREQ);
      }
      // every slot's last load has landed before the CTA may exit (a consumer that
      // gave up early leaves them unwaited)
      for (int q = issued > nsl ? issued - nsl : 0; q < issued; ++q)
        mbar_wait(is_k ? D_KF(q % nsl) : D_VF(q % nsl), (q / nsl) & 1, nullptr, a.status);
    }
  } else {
    griddep_wait();
    griddep_launch();
    // ---------------- writer: outputs, split partials and merges (warp 7) ----------------
    for (int it = 0;; ++it) {
      const int slot = it & 3;
      if (!warp_all(mbar_wait(D_IF(slot), (it >> 2) & 1, abort_flag, a.status))) break;
      const DecItem e = *reinterpret_cast<const DecItem*>(ring + slot * 32);
      __syncwarp();
      if (lane == 0) mbar_arrive(D_IE(slot));
      if (e.unit < 0) break;
      const int ob = it & 1;
      if (!warp_all(mbar_wait(D_STF(ob), (it >> 1) & 1, abort_flag, a.status))) break;
      const float* st = reinterpret_cast<const float*>(sm2 + C::ST_OFF + ob * C::ST_BYTES);
      const int r = (e.unit % per_seq) / a.nkv_l, g = e.unit % a.nkv_l;
      __half* obase = reinterpret_cast<__half*>(a.out) + static_cast<size_t>(e.t) * a.n * a.nq_l * HD +
                      (static_cast<size_t>(r) * a.nq_l + g * G) * HD;
      if (e.nsplit == 1) {
        uint32_t sat = 0;
        for (int i = lane; i < G * HD / 8; i += 32) {
          const int h = i / (HD / 8), c = i % (HD / 8);
          const float* s8 = st + h * (HD + 2) + c * 8;
          uint4 w;
          w.x = pack_f16x2(s8[0], s8[1], sat); w.y = pack_f16x2(s8[2], s8[3], sat);
          w.z = pack_f16x2(s8[4], s8[5], sat); w.w = pack_f16x2(s8[6], s8[7], sat);
          *reinterpret_cast<uint4*>(obase + h * HD + c * 8) = w;
        }
        report_sat(a.status, sat);
        mbar_arrive(D_STE(ob));
        continue;
      }
      // a split: its partial (unnormalised O, m, l per head), then the last split
      // of the unit to arrive (atomic counter, no waiting) merges them in split order
      float* part = a.part + (static_cast<size_t>(e.unit) * pstride + e.split) * G * (HD + 2);
      for (int i = lane; i < G * (HD + 2) / 2; i += 32)
        reinterpret_cast<float2*>(part)[i] = reinterpret_cast<const float2*>(st)[i];
      mbar_arrive(D_STE(ob));
      __threadfence();
      __syncwarp();
      int last = 0;
      if (lane == 0) last = atomicAdd(a.counters + e.unit, 1) == e.nsplit - 1 ? 1 : 0;
      last = __shfl_sync(0xffffffffu, last, 0);
      if (!last) continue;
      __threadfence();
      const float* pbase = a.part + static_cast<size_t>(e.unit) * pstride * G * (HD + 2);
      uint32_t sat = 0;
      for (int i = lane; i < G * HD / 8; i += 32) {
        const int h = i / (HD / 8), c = i % (HD / 8);
        float mm = -INFINITY, ll = 0.0f, acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
        // four splits' partials loaded at once (one L2 round trip), then added in split order
        for (int s0 = 0; s0 < e.nsplit; s0 += 4) {
          float m2[4], l2[4], a2[4][8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            m2[q] = -INFINITY;
            l2[q] = 0.0f;
            if (s0 + q < e.nsplit) {
              const float* ps = pbase + (static_cast<size_t>(s0 + q) * G + h) * (HD + 2);
              m2[q] = __ldcg(ps + HD);
              l2[q] = __ldcg(ps + HD + 1);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 v = __ldcg(reinterpret_cast<const float2*>(ps + c * 8) + k);
                a2[q][2 * k] = v.x;
                a2[q][2 * k + 1] = v.y;
              }
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (s0 + q >= e.nsplit) break;
            const float mn = fmaxf(mm, m2[q]);
            if (mn != -INFINITY) {
              const float c1 = exp2f(mm - mn), c2 = exp2f(m2[q] - mn);
              ll = ll * c1 + l2[q] * c2;
#pragma unroll
              for (int k = 0; k < 8; ++k) acc[k] = acc[k] * c1 + a2[q][k] * c2;
              mm = mn;
            }
          }
        }
        float o[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = ll > 0.0f ? acc[k] / ll : 0.0f;
        uint4 w;
        w.x = pack_f16x2(o[0], o[1], sat); w.y = pack_f16x2(o[2], o[3], sat);
        w.z = pack_f16x2(o[4], o[5], sat); w.w = pack_f16x2(o[6], o[7], sat);
        *reinterpret_cast<uint4*>(obase + h * HD + c * 8) = w;
      }
      report_sat(a.status, sat);
      if (lane == 0) a.counters[e.unit] = 0;
    }
  }
#undef D_IF
#undef D_IE
#undef D_QF
#undef D_QE
#undef D_KF
#undef D_KE
#undef D_VF
#undef D_VE
#undef D_SF
#undef D_PF
#undef D_OD
#undef D_OF
#undef D_STF
#undef D_STE
#undef D_NREQ
#undef D_DR
#undef D_OE
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x >> 5 == 1) {
    tc_fence_after();
    tmem_dealloc(*tmem_slot, C::TMEM_COLS);
  }
  // the last CTA to finish, over every launch drawing from the counter, resets it
  // for the next step (every CTA has drawn its last tickets before it counts itself)
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.sched + 1, 1) == a.sched_ctas - 1) {
      atomicExch(a.sched, 0);
      atomicExch(a.sched + 1, 0);
    }
  }
}

template <int HD, int G>
static cudaError_t prepare_decode_tc(int* ctas_per_sm) {
  static PerDevice pd;  // the attributes and the occupancy, once per device
  int dev = -1, occ = 0;
  if (!per_device_ready(pd, &dev, &occ)) {
    cudaError_t e = cudaFuncSetAttribute(attn_decode_tc_kernel<HD, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DtcCfg<HD, G>::SMEM);
    if (e != cudaSuccess) return e;
    // all of the unified L1 / shared storage as shared memory, so that two CTAs fit per SM
    e = cudaFuncSetAttribute(attn_decode_tc_kernel<HD, G>, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, attn_decode_tc_kernel<HD, G>, DtcCfg<HD, G>::THREADS,
                                                      DtcCfg<HD, G>::SMEM);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    per_device_mark(pd, dev, occ);
  }
  *ctas_per_sm = occ;
  return cudaSuccess;
}

static cudaError_t decode_tc_ctas_per_sm(int G, int* per_sm) {
  if (G == 1) return prepare_decode_tc<128, 1>(per_sm);
  if (G == 2) return prepare_decode_tc<128, 2>(per_sm);
  if (G == 4) return prepare_decode_tc<128, 4>(per_sm);
  if (G == 8) return prepare_decode_tc<128, 8>(per_sm);
  return cudaErrorNotSupported;
}

template <int HD, int G>
static cudaError_t launch_decode_tc_hd(const AttnArgs& a, cudaStream_t s) {
  using C = DtcCfg<HD, G>;
  int per_sm = 0;
  cudaError_t e0 = prepare_decode_tc<HD, G>(&per_sm);  // sets the shared-memory attributes once
  if (e0 != cudaSuccess) return e0;
  // persistent: a.ctas CTAs (one per SM: their shared memory fills it), each
  // running two pipelines; CTAs that start late, e.g. on SMs another stream's
  // kernel held, take whatever items are left
  if (!a.sched || a.ctas < 1 || a.sched_ctas < a.ctas) return cudaErrorInvalidValue;
  const int64_t kv_rows = static_cast<int64_t>(a.n) * 2 * a.kvm.blocks * a.nkv_l * a.kvm.block_len;
  if (kv_rows >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  CUtensorMap mkv, mkv64, mkv16;  // boxes of 128, 64 and 16 rows x 64 dims
  if (!make_tmap_2d(&mkv, a.kv, kv_rows, HD, HD, 128, true)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&mkv64, a.kv, kv_rows, HD, HD, 64, true)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&mkv16, a.kv, kv_rows, HD, HD, 16, true)) return cudaErrorInvalidValue;
  return launch_pdl(attn_decode_tc_kernel<HD, G>, dim3(a.ctas), dim3(C::THREADS), C::SMEM, s, mkv, mkv64, mkv16, a);
}

// The decode split plan.  A few units: every unit in decode_splits parts (one
// level).  Otherwise, on the persistent tensor-core kernel, the units in levels
// of 1, 2, 4 and 8 splits, sized by guided self-scheduling: items of a level are
// handed out while the work left is at least kDecodeGuide x (pipelines) x (item
// size), so that the items still to come when a pipeline runs dry are small
// against the work left, and the pipelines end close together.  Split counts
// are rounded so that every split of a full-length unit holds whole key tiles
// (17 tiles in 8 parts of 3 tiles: 6 splits).
constexpr double kDecodeGuide = 0.5;
DecodeSplit decode_split_plan(int max_kv_len, int num_units, int num_sms, int hd, int G, int max_splits) {
  DecodeSplit d{};
  for (int l = 0; l < kDecLevels; ++l) d.splits[l] = 1;
  d.splits[0] = decode_splits(max_kv_len, num_units, num_sms, hd, G, max_splits);
  d.units[0] = num_units > 0 ? num_units : 0;
  if (hd != 128 || d.splits[0] != 1 || num_units <= 0) return d;
  const int nt = (max_kv_len + 127) / 128;  // key tiles of a full-length unit
  const double pipes = 2.0 * num_sms;       // decode pipelines: two per CTA, one CTA per SM
  double left = static_cast<double>(num_units) * nt;
  int u = 0;
  const int want[kDecLevels] = {1, 2, 4, 8};
  for (int l = 0; l < kDecLevels; ++l) {
    int f = want[l] < max_splits ? want[l] : max_splits;
    if (f > nt) f = nt;
    if (f < 1) f = 1;
    const int chunk = (nt + f - 1) / f;  // tiles per split
    const int ns = (nt + chunk - 1) / chunk;
    d.splits[l] = ns;
    int n = num_units - u;
    if (l + 1 < kDecLevels) {
      const double stop = kDecodeGuide * pipes * chunk;  // work left when this level's items get too big
      const double fit = (left - stop) / nt;
      n = fit <= 0.0 ? 0 : (fit >= n ? n : static_cast<int>(fit + 0.999999));
    }
    d.units[l] = n;
    u += n;
    left -= static_cast<double>(n) * nt;
  }
  return d;
}

// ---------------------------------------------------------------------------
// Prefill (several new tokens per sequence, causal with cache offset):
// flash attention on the tcgen05 tensor cores.  One CTA = 128 queries of one
// (sequence, rank, q head); 320 threads:
//   warp 0      TMA: the Q tiles once (bf16 high and low parts), then K and V
//               blocks of 128 keys from the rank's bf16 cache into separate
//               2-stage rings (one lane each): a K stage frees as soon as its S
//               MMA is done, a V stage when its PV MMA is.
//   warp 1      TMEM allocation + one MMA-issuing thread: S(j) = Q K(j)^T
//               (as Q_hi K^T + Q_lo K^T, so q keeps ~16 significant bits) into
//               one of two TMEM score buffers, then O += P(j) V(j) into the TMEM
//               output accumulator (P read from tensor memory, V as an MN-major
//               operand straight from the TMA tile).  S(j+1) is issued before
//               O += P(j) V(j), so the scores of the next block are computed
//               while the softmax of this one runs.
//   warps 2-9   softmax: two threads per query row (its TMEM lane), one per
//               64-key half -- scale, causal mask, row max, exp2, row sum;
//               P(j) (bf16) written back over its own scores in TMEM, so the
//               two score buffers double as two P buffers; the running output
//               is rescaled only when the row max has grown by more than 2^8
//               (otherwise P may exceed 1 by at most 2^8, exactly compensated by
//               the row sum); final O / l written as fp16.
// Ordering: tcgen05 operations of the MMA thread complete in issue order, so
// S(j+2) (issued after O += P(j) V(j)) never overwrites P(j) before it is read,
// and the completion of S(j) implies that of O += P(j-2) V(j-2).
// All waits are bounded (TP_WAIT_LIMIT_NS) and end in TP_DEVFLAG_TIMEOUT.
// Cache positions never written must hold finite values (the runner zeroes the
// cache once): keys past the sequence get P = 0, but 0 * NaN would not vanish.
// ---------------------------------------------------------------------------
template <int HD>
struct FaCfg {
  static constexpr int BQ = 128, BKV = 128;
  static constexpr int NSUB = HD / 64;            // 64-column (128-byte) sub-tiles per row
  static constexpr int SUB_BYTES = 128 * 128;     // one [128 rows][64] bf16 sub-tile
  static constexpr int TILE_BYTES = NSUB * SUB_BYTES;
  static constexpr int STAGES = 2;
  static constexpr int Q_OFF = 0;                                  // [hi | lo]
  static constexpr int KV_OFF = 2 * TILE_BYTES;                    // K ring [stage], then V ring [stage]
  static constexpr int BAR_OFF = KV_OFF + STAGES * 2 * TILE_BYTES;
  static constexpr int SMEM = 1024 + BAR_OFF + 256;
  static constexpr int S_COL = 0;      // two score buffers: columns [0,128) and [128,256); P(j) (bf16
                                       // pairs) overwrites the first 64 columns of its score buffer
  static constexpr int O_COL = 256;    // output accumulator: columns [256, 256+HD)
};

template <int HD>
__global__ void __launch_bounds__(320, 1)
    attn_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmQlo,
                           const __grid_constant__ CUtensorMap tmKV, const AttnArgs a) {
  using C = FaCfg<HD>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  // barriers: q_full | k_full[S] | k_empty[S] | v_full[S] | v_empty[S] | s_full[2] | p_full[2] | o_done |
  //           drain | q_free | o_read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 9 + 4 * STAGES);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t bar0 = smem_u32(bars);
#define B_Q (bar0)
#define B_KF(s) (bar0 + 8u * (1 + (s)))
#define B_KE(s) (bar0 + 8u * (1 + STAGES + (s)))
#define B_VF(s) (bar0 + 8u * (1 + 2 * STAGES + (s)))
#define B_VE(s) (bar0 + 8u * (1 + 3 * STAGES + (s)))
#define B_SF(b) (bar0 + 8u * (1 + 4 * STAGES + (b)))
#define B_PF(b) (bar0 + 8u * (3 + 4 * STAGES + (b)))
#define B_OD (bar0 + 8u * (5 + 4 * STAGES))
#define B_DR (bar0 + 8u * (6 + 4 * STAGES))
#define B_QE (bar0 + 8u * (7 + 4 * STAGES))
#define B_OE (bar0 + 8u * (8 + 4 * STAGES))

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Work items: (query block, sequence, rank, q head), heaviest first (the query
  // block index from the last varies slowest); CTA c takes items c, c + grid, ...
  // Every role walks the same items and skips the same ones.
  const int heads = a.n * a.nq_l;
  const int nseq = a.seq_end - a.seq_begin;
  const int qblocks = (a.max_q_len + C::BQ - 1) / C::BQ;
  const int n_items = qblocks * heads * nseq;
  struct Item {
    int b, r, h, g, qlen, q0, ctx, tbase, nblk;
    bool bad;
  };
  // false: no queries in this block; bad: a cache block of the sequence's keys
  // [0, ctx + qlen) lies outside the cache (the item is skipped and flagged)
  auto item_at = [&](int i, Item& x) -> bool {
    const int rest = i % (heads * nseq);
    x.b = a.seq_begin + rest / heads;
    const int hg = rest % heads;
    x.qlen = a.cu_q[x.b + 1] - a.cu_q[x.b];
    x.q0 = (qblocks - 1 - i / (heads * nseq)) * C::BQ;
    if (x.q0 >= x.qlen) return false;
    x.r = hg / a.nq_l;
    x.h = hg % a.nq_l;
    x.g = x.h / (a.nq_l / a.nkv_l);
    x.ctx = a.ctx_len[x.b];
    x.tbase = a.cu_q[x.b];
    x.bad = x.ctx < 0 || kv_blocks_bad(a.kvm, x.b, 0, x.ctx + x.qlen, 0, 1);
    const int kend = x.ctx + min(x.q0 + C::BQ, x.qlen);  // keys the item needs: [0, kend)
    x.nblk = (kend + C::BKV - 1) / C::BKV;
    return true;
  };

  if (threadIdx.x == 0) {
    mbar_init(B_Q, 1);
    mbar_init(B_QE, 1);
    mbar_init(B_OE, 8);  // one arrival per softmax warp once it has read the output
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(B_KF(s), 1);
      mbar_init(B_KE(s), 1);
      mbar_init(B_VF(s), 1);
      mbar_init(B_VE(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(B_SF(i), 1);
      mbar_init(B_PF(i), 8);
    }
    mbar_init(B_OD, 1);
    mbar_init(B_DR, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_wait();  // q and the cache come from the QKV GEMM
  griddep_launch();

  if (warp == 0) {
    // ---------------- TMA producers: lane 0 streams Q then K, lane 1 streams V ----------------
    // The K / V rings and the Q tile run on across the CTA's items (jb counts
    // every key block the CTA has streamed, it every item).
    if (lane < 2) {
      const bool is_k = lane == 0;
      if (is_k) {
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmQlo);
        tma_prefetch_desc(&tmKV);
      }
      uint8_t* ring = smem + C::KV_OFF + (is_k ? 0 : STAGES * C::TILE_BYTES);
      int jb = 0, it = 0;
      bool ok = true;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
        Item x;
        if (!item_at(i, x)) continue;
        if (x.bad) {
          if (is_k) raise_flag(a.status, TP_DEVFLAG_BAD_TOKEN);
          continue;
        }
        if (is_k) {
          // this item's q once the previous item's score MMAs have read the last one
          if (!mbar_wait(B_QE, (it & 1) ^ 1u, abort_flag, a.status)) break;
          const int qcol = x.r * a.w_rank + x.h * HD;
          const int qlo_col = (x.r * a.nq_l + x.h) * HD;
          mbar_arrive_expect_tx(B_Q, 2 * C::TILE_BYTES);
          for (int s = 0; s < C::NSUB; ++s) {
            tma_load_2d(smem_u32(smem + C::Q_OFF + s * C::SUB_BYTES), &tmQ, B_Q, qcol + s * 64, x.tbase + x.q0);
            tma_load_2d(smem_u32(smem + C::Q_OFF + C::TILE_BYTES + s * C::SUB_BYTES), &tmQlo, B_Q,
                        qlo_col + s * 64, x.tbase + x.q0);
          }
        }
        // block of the next key block, looked up one block ahead (its load overlaps the wait)
        int blk_next = kv_block_checked(a.kvm, x.b, 0);
        for (int j = 0; j < x.nblk; ++j, ++jb) {
          const int st = jb % STAGES;
          const uint32_t full = is_k ? B_KF(st) : B_VF(st);
          const uint32_t empty = is_k ? B_KE(st) : B_VE(st);
          const int blk = blk_next;
          if (j + 1 < x.nblk) blk_next = kv_block_checked(a.kvm, x.b, (j + 1) * C::BKV);
          if (!mbar_wait(empty, ((jb / STAGES) & 1) ^ 1u, abort_flag, a.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full, C::TILE_BYTES);
          const int row = static_cast<int>(
              kv_row(a.kvm, a.nkv_l, x.r, is_k ? 0 : 1, blk, x.g, (j * C::BKV) % a.kvm.block_len));
          for (int s = 0; s < C::NSUB; ++s)
            tma_load_2d(smem_u32(ring + st * C::TILE_BYTES + s * C::SUB_BYTES), &tmKV, full, s * 64, row);
        }
        ++it;
      }
      // every load issued has landed before the CTA may exit
      if (is_k && it > 0) mbar_wait(B_Q, (it - 1) & 1, nullptr, a.status);
      for (int j = (jb > STAGES ? jb - STAGES : 0); j < jb; ++j)
        mbar_wait(is_k ? B_KF(j % STAGES) : B_VF(j % STAGES), (j / STAGES) & 1, nullptr, a.status);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, C::BKV);      // S = Q K^T: both K-major
      const uint32_t id_o = idesc_bf16_f32(128, HD, true);    // O += P V: V MN-major
      bool ok = true;
      int jb = 0, it = 0, drains = 0;
      for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
      Item x;
      if (!item_at(i, x) || x.bad) continue;
      const int nblk = x.nblk;
      const int jb0 = jb;
      ok = mbar_wait(B_Q, it & 1, abort_flag, a.status);
      tc_fence_after();
      // O += P(j) V(j), P(j) from TMEM (score buffer of the CTA's key block jb0 + j);
      // the first one overwrites O, so it waits until the previous item's output was read
      auto pv = [&](int j) -> bool {
        const int gj = jb0 + j;
        const int st = gj % STAGES, sb = gj & 1;
        if (j == 0 && !mbar_wait(B_OE, (it & 1) ^ 1u, abort_flag, a.status)) return false;
        if (!mbar_wait(B_PF(sb), (gj >> 1) & 1, abort_flag, a.status)) return false;
        if (!mbar_wait(B_VF(st), (gj / STAGES) & 1, abort_flag, a.status)) return false;
        tc_fence_after();
        const uint32_t vt = smem_u32(smem + C::KV_OFF + (STAGES + st) * C::TILE_BYTES);
        const uint32_t pa = tmem + C::S_COL + sb * 128;
#pragma unroll
        for (int kk = 0; kk < C::BKV / 16; ++kk) {
          const uint64_t bd = sdesc_mn_sw128(vt + kk * 16 * 128, C::SUB_BYTES, 1024);
          tc_mma_f16_ts(tmem + C::O_COL, pa + kk * 8, bd, id_o, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(B_OD);
        tc_commit(B_VE(st));
        return true;
      };
      for (int j = 0; ok && j < nblk; ++j) {
        const int gj = jb0 + j;
        const int st = gj % STAGES, sb = gj & 1;
        // score buffer sb last held P(gj-2), whose PV MMA was issued before this point
        if (!mbar_wait(B_KF(st), (gj / STAGES) & 1, abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t qt = smem_u32(smem + C::Q_OFF);
        const uint32_t kt = smem_u32(smem + C::KV_OFF + st * C::TILE_BYTES);
#pragma unroll
        for (int part = 0; part < 2; ++part) {  // S = Q_hi K^T + Q_lo K^T
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint64_t ad = sdesc_k_sw128(qt + part * C::TILE_BYTES + (kk >> 2) * C::SUB_BYTES) + 2ull * (kk & 3);
            const uint64_t bd = sdesc_k_sw128(kt + (kk >> 2) * C::SUB_BYTES) + 2ull * (kk & 3);
            tc_mma_f16(tmem + C::S_COL + sb * 128, ad, bd, id_s, (part > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc_commit(B_SF(sb));
        tc_commit(B_KE(st));                 // the K stage is free once S(j) is done
        if (j == nblk - 1) tc_commit(B_QE);  // and the Q tile once the item's last S is
        if (j > 0 && !pv(j - 1)) { ok = false; break; }
      }
      if (ok && !pv(nblk - 1)) ok = false;
      tc_commit(B_DR);  // the item's output: completes after every MMA above
      ++drains;
      jb = jb0 + nblk;
      ++it;
      }
      if (drains > 0) mbar_wait(B_DR, (drains - 1) & 1, nullptr, a.status);  // every MMA has completed
    }
  } else {
    // ---------------- softmax / output (warps 2..9) ----------------
    // Two warps per query row: warps 2-5 take keys [0, 64) of each block and
    // output dims [0, HD/2), warps 6-9 the other halves (both see the same TMEM
    // lanes).  The halves exchange their row maxima through two spare TMEM
    // columns and agree on every rescale decision.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    constexpr int OH = HD / 2;                  // output dims per half
    bool ok = true;
    int jb = 0, it = 0;
    for (int i = blockIdx.x; ok && i < n_items; i += gridDim.x) {
    Item x;
    if (!item_at(i, x) || x.bad) continue;
    const int nblk = x.nblk, q0 = x.q0, qlen = x.qlen, ctx = x.ctx, tbase = x.tbase, r = x.r, h = x.h;
    const int qi = q0 + row;                    // query index within the sequence
    const bool row_ok = qi < qlen;
    const int last_key = ctx + qi;              // keys <= last_key are visible
    float m_used = -INFINITY, l = 0.0f;
    for (int j = 0; j < nblk; ++j) {
      const int gj = jb + j;
      const int sb = gj & 1;
      if (!mbar_wait(B_SF(sb), (gj >> 1) & 1, abort_flag, a.status)) ok = false;
      if (!named_bar_and(1, 256, ok)) { ok = false; break; }
      tc_fence_after();
      float sv[64];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        float v[32];
        tc_ld32(lane_addr + C::S_COL + sb * 128 + half * 64 + c * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) sv[c * 32 + i] = v[i];
      }
      const int key0 = j * C::BKV + half * 64;
      const bool need_mask = (key0 + 63 > ctx + q0) || !row_ok;  // diagonal blocks and padding rows only
      if (need_mask) {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (!row_ok || key0 + i > last_key) sv[i] = -INFINITY;
      }
      // row max in four independent three-input chains (short dependency chains)
      float mc[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        mc[c] = sv[16 * c];
#pragma unroll
        for (int i = 1; i < 15; i += 2) mc[c] = max3f(mc[c], sv[16 * c + i], sv[16 * c + i + 1]);
        mc[c] = fmaxf(mc[c], sv[16 * c + 15]);
      }
      float mx = max3f(mc[0], mc[1], fmaxf(mc[2], mc[3]));
      mx *= a.scale_log2;  // the scale is positive: max of the scaled scores
      // row max over both halves (TMEM columns 384 + 2 * (j & 1) + half); past this
      // barrier both halves have read their scores, so P may overwrite them
      tc_st1(lane_addr + 384 + 2 * (gj & 1) + half, mx);
      tc_fence_before();
      named_bar_sync(1, 256);
      tc_fence_after();
      mx = fmaxf(mx, tc_ld1(lane_addr + 384 + 2 * (gj & 1) + (half ^ 1)));
      const bool rescale = mx > m_used + 8.0f;
      const float m_new = rescale ? mx : m_used;
      const float mb = m_new == -INFINITY ? 0.0f : m_new;
      // p = 2^(s * scale - m): one paired FMA, two ex2, one paired add per two keys;
      // P(j) as bf16 pairs (keys 2c, 2c+1 in column c)
      uint32_t pw[32];
      float psum;
      {
        const uint64_t sc2 = f32x2(a.scale_log2, a.scale_log2), nb2 = f32x2(-mb, -mb);
        uint64_t acc2[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) acc2[k] = f32x2(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x0, x1;
          unpack_f32x2(fma_f32x2(f32x2(sv[2 * c], sv[2 * c + 1]), sc2, nb2), x0, x1);
          const float p0 = ex2_ftz(x0), p1 = ex2_ftz(x1);
          acc2[c & 3] = add_f32x2(acc2[c & 3], f32x2(p0, p1));
          pw[c] = pack_bf16x2(p0, p1);
        }
        float s0, s1, s2, s3;
        unpack_f32x2(add_f32x2(acc2[0], acc2[1]), s0, s1);
        unpack_f32x2(add_f32x2(acc2[2], acc2[3]), s2, s3);
        psum = (s0 + s1) + (s2 + s3);
      }
      // A rescale of O waits for the previous block's PV MMA (S(j) done implies
      // PV(j-2) done, so the output barrier is at phase j-1 or j here).  A failed
      // wait only marks the thread; every softmax thread leaves together at the
      // next agreement point (named barriers have no time limit).
      // The rescale is decided per row (lane) but the O update is warp-collective
      // (tcgen05.ld/st): when any row of the warp needs it, every lane waits for
      // the output barrier and loads and stores its O row, the others with a
      // factor of 1.
      const bool touch_o = rescale && j > 0 && m_used != -INFINITY;
      const bool warp_touch = __any_sync(0xffffffffu, touch_o);
      if (warp_touch && !warp_all(mbar_wait(B_OD, (gj - 1) & 1, abort_flag, a.status))) ok = false;
      if (!ok) continue;  // warp-uniform here
      if (warp_touch) {
        tc_fence_after();
        const float corr = exp2f(touch_o ? m_used - m_new : 0.0f);  // no branch before the collectives
        l *= corr;
#pragma unroll
        for (int c = 0; c < OH / 32; ++c) {
          float v[32];
          tc_ld32(lane_addr + C::O_COL + half * OH + c * 32, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= corr;
          tc_st32(lane_addr + C::O_COL + half * OH + c * 32, v);
        }
      }
      if (rescale) m_used = m_new;
      l += psum;
      tc_st32u(lane_addr + C::S_COL + sb * 128 + half * 32, pw);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(B_PF(sb));
    }
    // the MMA thread commits the drain barrier after the item's last PV
    if (ok) ok = mbar_wait(B_DR, it & 1, abort_flag, a.status);
    if (named_bar_and(1, 256, ok)) {
      tc_fence_after();
      // row sum over both halves (TMEM columns 388 + half)
      tc_st1(lane_addr + 388 + half, l);
      tc_fence_before();
      named_bar_sync(1, 256);
      tc_fence_after();
      l += tc_ld1(lane_addr + 388 + (half ^ 1));
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      __half* orow = reinterpret_cast<__half*>(a.out) + static_cast<size_t>(tbase + (row_ok ? qi : 0)) * a.n * a.nq_l * HD +
                     (static_cast<size_t>(r) * a.nq_l + h) * HD + half * OH;
      uint32_t sat = 0;
#pragma unroll
      for (int c = 0; c < OH / 32; ++c) {
        float v[32];
        tc_ld32(lane_addr + C::O_COL + half * OH + c * 32, v);
        if (row_ok) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            uint4 w;
            w.x = pack_f16x2(v[k * 8 + 0] * inv, v[k * 8 + 1] * inv, sat);
            w.y = pack_f16x2(v[k * 8 + 2] * inv, v[k * 8 + 3] * inv, sat);
            w.z = pack_f16x2(v[k * 8 + 4] * inv, v[k * 8 + 5] * inv, sat);
            w.w = pack_f16x2(v[k * 8 + 6] * inv, v[k * 8 + 7] * inv, sat);
            *reinterpret_cast<uint4*>(orow + c * 32 + k * 8) = w;
          }
        }
      }
      report_sat(a.status, sat);
    } else {
      ok = false;
    }
    // O has been read: the next item's first PV may overwrite it
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(B_OE);
    jb += nblk;
    ++it;
    }
  }
#undef B_QE
#undef B_OE
#undef B_Q
#undef B_KF
#undef B_KE
#undef B_VF
#undef B_VE
#undef B_SF
#undef B_PF
#undef B_OD
#undef B_DR
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int HD>
static cudaError_t launch_prefill_hd(const AttnArgs& a, cudaStream_t s) {
  using C = FaCfg<HD>;
  const int64_t w_cols = static_cast<int64_t>(a.n) * a.w_rank;
  const int64_t kv_rows = static_cast<int64_t>(a.n) * 2 * a.kvm.blocks * a.nkv_l * a.kvm.block_len;
  if (kv_rows >= (int64_t(1) << 31)) return cudaErrorInvalidValue;
  const int64_t q_cols = static_cast<int64_t>(a.n) * a.nq_l * HD;
  CUtensorMap mq, mqlo, mkv;
  if (!make_tmap_2d(&mq, a.qkv, a.T, w_cols, w_cols, 128, true)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&mqlo, a.q_lo, a.T, q_cols, q_cols, 128, true)) return cudaErrorInvalidValue;
  if (!make_tmap_2d(&mkv, a.kv, kv_rows, HD, HD, 128, true)) return cudaErrorInvalidValue;
  static PerDevice attr;  // per device
  {
    const cudaError_t e = smem_attr_per_device(attr, attn_prefill_tc_kernel<HD>, C::SMEM);
    if (e != cudaSuccess) return e;
  }
  // persistent: a.ctas CTAs walk the items (one per SM at most, fewer while a decode
  // attention launch shares the GPU)
  const int items = (a.max_q_len + C::BQ - 1) / C::BQ * a.n * a.nq_l * (a.seq_end - a.seq_begin);
  const int ctas = a.ctas < items ? a.ctas : items;
  if (ctas < 1) return cudaErrorInvalidValue;
  return launch_pdl(attn_prefill_tc_kernel<HD>, dim3(ctas), dim3(320), C::SMEM, s, mq, mqlo, mkv, a);
}

cudaError_t launch_attention_prefill(const AttnArgs& a, cudaStream_t s) {
  const int seqs = a.seq_end - a.seq_begin;
  if (seqs <= 0 || a.max_q_len <= 0) return cudaSuccess;
  if (a.hd == 128) return launch_prefill_hd<128>(a, s);
  if (a.hd == 64) return launch_prefill_hd<64>(a, s);
  return cudaErrorNotSupported;
}

}  // namespace tpk
