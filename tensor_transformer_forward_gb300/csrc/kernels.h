// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
// Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

struct tp_ctx;

namespace tpk {

// One-time per-device set-up of a kernel (cudaFuncSetAttribute applies to the
// current device only): bit d of `done` is set once device d is prepared, and
// `value[d]` keeps a per-device result (an occupancy).  Devices >= 64 are
// prepared on every call.  Two threads may both prepare a device; the calls are
// idempotent.
struct PerDevice {
  std::atomic<uint64_t> done{0};
  int value[64] = {};
};
inline bool per_device_ready(PerDevice& pd, int* dev, int* value) {
  if (cudaGetDevice(dev) != cudaSuccess) *dev = -1;
  if (*dev < 0 || *dev >= 64) return false;
  if (!(pd.done.load(std::memory_order_acquire) >> *dev & 1u)) return false;
  if (value) *value = pd.value[*dev];
  return true;
}
inline void per_device_mark(PerDevice& pd, int dev, int value) {
  if (dev < 0 || dev >= 64) return;
  pd.value[dev] = value;
  pd.done.fetch_or(uint64_t(1) << dev, std::memory_order_release);
}
// The kernel's dynamic shared-memory limit raised to smem bytes on the current device.
template <typename K>
inline cudaError_t smem_attr_per_device(PerDevice& pd, K kern, int smem) {
  int dev = -1;
  if (per_device_ready(pd, &dev, nullptr)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess) per_device_mark(pd, dev, 1);
  return e;
}

// The address a kernel uses for p: device (or managed) memory as it is, page-locked
// host memory through its device mapping; null for memory the GPU cannot address.
template <typename T>
T* gpu_view(T* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();
    return nullptr;
  }
  if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return p;
  if (a.type == cudaMemoryTypeHost) return static_cast<T*>(a.devicePointer);
  return nullptr;
}

// What the LM-head call needs to know about a context (filled by api.cu).
struct HeadView {
  int H, n, vocab, num_sms;
  int64_t v_l;
  size_t lm_head_off, final_norm_off;
  float eps;
};
int ctx_head_view(tp_ctx* ctx, HeadView* out);  // returns a tp_status
int ctx_hidden_size(const tp_ctx* ctx);          // H, without touching the device (0 for null)

// Launch with programmatic stream serialization: the kernel may begin (up to its
// griddep_wait()) while the previous kernel on the stream is still running.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// The same, as clusters of `cluster` CTAs along x (2: a CTA pair sharing tcgen05
// cta_group::2 MMAs); grid.x must be a multiple of the cluster size.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kern)(KArgs...), int cluster, dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------- KV cache addressing ----------------
// A layer's cache is [n][2 (K, V)][blocks][nkv_l][block_len][hd] bf16.  Position p
// of sequence b lives in block table[b * stride + p / block_len], at row
// p % block_len.  A contiguous cache is the case of one block per sequence slot
// (table = the batch's slot array, stride 1, block_len = the capacity); a paged
// cache has pages of block_len positions and a page table of stride entries per
// sequence.
struct KvMap {
  const int32_t* table;
  int stride;     // table entries per sequence
  int block_len;  // positions per block
  int blocks;     // blocks in the cache
};
// The block holding position p of sequence b, or -1 when p or the table entry is
// outside the cache.
__device__ __forceinline__ int kv_block(const KvMap& m, int b, int p) {
  if (p < 0) return -1;
  const int i = p / m.block_len;
  if (i >= m.stride) return -1;
  const int blk = m.table[static_cast<int64_t>(b) * m.stride + i];
  return (blk >= 0 && blk < m.blocks) ? blk : -1;
}
// The block of position p of sequence b once the range it is in has been checked.
__device__ __forceinline__ int kv_block_checked(const KvMap& m, int b, int p) {
  return m.table[static_cast<int64_t>(b) * m.stride + p / m.block_len];
}
// This thread's share of the check that every block holding keys [k0, k1) of
// sequence b (k0 >= 0) is inside the cache: threads tid, tid + nthr, ... take one
// block each; the CTA combines the answers (__syncthreads_or).
__device__ __forceinline__ bool kv_blocks_bad(const KvMap& m, int b, int k0, int k1, int tid, int nthr) {
  if (k1 <= k0) return false;
  const int ib0 = k0 / m.block_len, ib1 = (k1 - 1) / m.block_len;
  bool bad = false;
  for (int ib = ib0 + tid; ib <= ib1; ib += nthr) bad |= kv_block(m, b, ib * m.block_len) < 0;
  return bad;
}
// Key splits of the decode kernels start on multiples of this many keys, so that a
// page of a paged cache (a multiple of it) holds whole key tiles of a split.
constexpr int kKeyAlign = 128;
// Row (of hd elements) of (rank r, K or V, block, local kv head g, row in block).
__device__ __forceinline__ int64_t kv_row(const KvMap& m, int nkv_l, int r, int kv, int blk, int g, int row) {
  return ((((static_cast<int64_t>(r) * 2 + kv) * m.blocks + blk) * nkv_l + g) * m.block_len) + row;
}

// ---------------- GEMM (tcgen05) ----------------
enum GemmEpi : int { EPI_STORE = 0, EPI_SILU = 1, EPI_RESID = 2, EPI_ARGMAX = 3, EPI_QKV = 4 };

// Extra inputs of the merged-QKV epilogue: per-head RMSNorm of q and k, RoPE at
// each token's position, K/V written to the rank's cache.
struct QkvEpi {
  int n, nq_l, nkv_l, hd, w_rank;
  const void* q_norm;        // [hd] bf16
  const void* k_norm;
  float eps;
  const float2* rope;        // (cos, sin) per (position, d < hd/2), blocked by 32 positions (see api.cu)
  int max_pos;
  const int32_t* cu_q;       // [B+1]
  const int32_t* ctx_len;    // [B]
  int B;
  void* kv;                  // cache [n][2][blocks][nkv_l][block_len][hd]
  KvMap kvm;
  int num_prefill;           // sequences [0, num_prefill): q as bf16 hi + lo parts; later ones: q as fp16
  void* q_lo;                // bf16 [T, n * nq_l * hd]: q - bf16(q) of prefill tokens
};

// Y[t, f] = sum over rank segments r of X[t, r*x_k_seg : +K_seg] . W[r*w_row_seg + f, 0 : K_seg]
// X: [T, x_cols] bf16 row-major; W: [w_rows, K_seg] bf16 row-major ([out, in]).
struct GemmProblem {
  const void* x;
  int64_t x_rows, x_cols, x_ld;   // elements
  const void* w;
  int64_t w_rows, w_cols, w_ld;
  int T;            // valid token rows
  int N;            // output features computed per segment (tile space, before SiLU folding)
  int n_seg;        // rank segments along K (1 = column-parallel)
  int k_seg;        // K per segment (multiple of 64)
  int x_k_seg;      // X column offset between segments
  int w_row_seg;    // W row offset between segments
  int epi;          // GemmEpi
  void* out;        // bf16 [T, ldo]
  int ldo;
  int out_cols;     // valid output columns
  // argmax epilogue
  float* amax_val;  // [tiles_f, amax_ld]
  int* amax_idx;
  int amax_ld;
  float* logits;    // optional fp32 [T, ld_logits]
  int ld_logits;
  int vocab;        // features >= vocab are masked out of the argmax
  int32_t* out_ids; // argmax result per token (weight-streaming path: reduced in the kernel)
  QkvEpi qkv;       // EPI_QKV only
  // dead workspace ranges (their last reader has completed) dropped from L2 without
  // write-back by the epilogue warps at the start (128-byte aligned, whole lines)
  const void* discard[2];
  int64_t discard_lines[2];
  // deferred RMSNorm of the input rows (QKV, gate_up): X holds the raw residual
  // rows (fp16), the norm weight is folded into W, and the epilogue scales row t
  // by rsqrt(sum(row_ss[t][0 .. row_groups)) / K + eps); null: no scaling
  const float* row_ss;  // [T][row_groups] sums of squares of 32-column groups
  int row_groups;
  float row_eps;
  // residual epilogue (EPI_RESID) that also leaves the next deferred norm's inputs:
  // the new residual rows in fp16 (row_out16, [T][out_cols]) and their 32-column
  // sums of squares (row_ss_out, [T][out_cols / 32]); null: plain reduce-add
  void* row_out16;
  float* row_ss_out;
};

struct GemmPlan {
  int BN;
  bool swap;        // weights on the MMA's M side (few tokens): tiles of 128 features x BN tokens
  bool pair;        // CTA pairs (clusters of 2): tiles of 256 tokens x BN features, cta_group::2 MMAs
  bool acc;         // running sum in registers (multi-segment or split-K)
  bool xch;         // residual pair tiles, K in two halves on two pairs of a 4-CTA cluster
                    // exchanging partials through distributed shared memory
  int tiles_t, tiles_f, splits;
  int grid;
  size_t partial_floats;  // workspace floats for split-K partials
};

GemmPlan plan_gemm(const GemmProblem& pr, int num_sms);
// TMA descriptor of a 2D 16-bit row-major tensor, box 64 columns x box_rows, 128-byte swizzle.
bool make_tmap_2d(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t ld, int box_rows,
                  bool bf16);
// workspace: partials (fp32) and per-tile counters (int, zeroed once, self-resetting)
// counters (launch_gemm): split-K tile counters from index 0 (fewer than 256 tiles
// are ever split); the weight-streaming argmax uses [0] and [1] and, from int
// index kArgmaxKeyOffset, one 64-bit key per token (at most kArgmaxMaxTokens).
// All zero between launches; the kernels leave them zero.
constexpr int kArgmaxKeyOffset = 2048;
constexpr int kArgmaxMaxTokens = 256;
constexpr int kGemmCounterInts = kArgmaxKeyOffset + 2 * kArgmaxMaxTokens;
cudaError_t launch_gemm(const GemmProblem& pr, const GemmPlan& plan, float* partials, int* counters,
                        int* status, cudaStream_t stream);
int gemm_num_tiles_f(const GemmProblem& pr, const GemmPlan& plan);

// ---------------- small kernels ----------------
cudaError_t launch_embed(const int32_t* ids, int T, const void* embed_stacked, int n, int64_t v_local,
                         int64_t vocab, int H, void* out, void* xh, float* ss, int* status, cudaStream_t s);
cudaError_t launch_rmsnorm(const void* x, int64_t rows, int H, const void* w, float eps, void* out, int* status,
                           cudaStream_t s);
// Row statistics for a deferred RMSNorm: fp16 copy of x [rows][H] and the sums of
// squares of each 32-column group, ss [rows][H / 32].
cudaError_t launch_row_stats(const void* x, int64_t rows, int H, void* xh, float* ss, int* status,
                             cudaStream_t s);


// Decode split plan: the units (sequence, rank, kv head) in consecutive levels,
// level l holding units[l] units whose keys are split in splits[l] parts each (a
// split covers whole 128-key tiles); items are handed out level by level, so
// the pieces get smaller as the work runs out.
constexpr int kDecLevels = 4;
struct DecodeSplit {
  int units[kDecLevels];
  int splits[kDecLevels];
};
__host__ __device__ inline int plan_items(const DecodeSplit& d) {
  int n = 0;
  for (int l = 0; l < kDecLevels; ++l) n += d.units[l] * d.splits[l];
  return n;
}
__host__ __device__ inline int plan_units(const DecodeSplit& d) {
  int n = 0;
  for (int l = 0; l < kDecLevels; ++l) n += d.units[l];
  return n;
}
// the largest split count of a level that holds units (partials per unit in the workspace)
__host__ __device__ inline int plan_max_splits(const DecodeSplit& d) {
  int m = 1;
  for (int l = 0; l < kDecLevels; ++l)
    if (d.units[l] > 0 && d.splits[l] > m) m = d.splits[l];
  return m;
}
struct AttnArgs {
  const void* qkv;           // [T, n * w_rank] (q post-RoPE: bf16 high part for prefill tokens, fp16 for decode)
  const void* q_lo;          // [T, n * nq_l * hd] bf16 low part of q (prefill tokens)
  int T;                     // rows of qkv
  int n, nq_l, nkv_l, hd, w_rank;
  const void* kv;            // cache [n][2][blocks][nkv_l][block_len][hd]
  KvMap kvm;
  const int32_t* cu_q;
  const int32_t* ctx_len;
  int seq_begin, seq_end;    // sequences handled by this launch
  int max_q_len, max_kv_len;
  void* out;                 // [T, n * nq_l * hd]
  float scale_log2;          // log2(e) / sqrt(hd)
  float* part;               // split-KV partials (decode)
  int* counters;
  DecodeSplit plan;          // decode: the units' key splits
  int ctas;                  // CTAs of a persistent launch (each walks work items)
  int* sched;                // decode: 2 ints (next ticket, CTAs done), zero between steps
  int sched_ctas;            // decode: CTAs of all the launches that draw from sched
  int* status;
};
cudaError_t launch_attention_prefill(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_attention_decode(const AttnArgs& a, cudaStream_t s);
DecodeSplit decode_split_plan(int max_kv_len, int num_units, int num_sms, int hd, int G, int max_splits);

cudaError_t launch_final_norm_select(const void* hidden, int H, const int32_t* cu_q, int B, const void* w,
                                     float eps, void* out, int* status, cudaStream_t s);
cudaError_t launch_argmax_reduce(const float* val, const int* idx, int tiles, int ld, int B, int32_t* out,
                                 cudaStream_t s);
cudaError_t launch_wait_probe(const int* flag, int* status, long long limit_ns, cudaStream_t s);
cudaError_t launch_decode_advance(int32_t* ctx_len, int B, const int32_t* ids, int32_t* history, int max_rows,
                                  int32_t* step, int32_t* status, cudaStream_t s);
// Weight conversions at shard time; status (device int32, may be null) receives
// TP_DEVFLAG_SATURATED when a weight is outside the fp16 range.
cudaError_t launch_bf16_to_f16(void* w, size_t elems, int* status, cudaStream_t s);
cudaError_t launch_fold_norm_f16(void* w, size_t rows, int cols, const void* norm, int* status, cudaStream_t s);

}  // namespace tpk
