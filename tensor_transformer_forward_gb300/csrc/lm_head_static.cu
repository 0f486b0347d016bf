// LM head + greedy argmax for callers that cannot allocate device memory.
//
// tp_lm_head_argmax needs a caller-allocated workspace (from
// tp_workspace_init) for its scratch: the normalised last-token rows, counters
// (CTA arrivals, tiles handed out) and the per-token argmax keys.  Some callers
// cannot hand one over: code that must not call cudaMalloc at that point (it
// can synchronise the device, or the process's device memory belongs to
// another allocator), or a caller that only holds the model weights and its
// inputs and outputs.  tp_lm_head_argmax_static runs the same kernels with that
// scratch in a fixed-size array compiled into this library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it until the process exits, and every call on a device shares
// it (it keeps the previous call's contents).  The counters and keys are
// cleared on the stream at the start of each call; the other scratch is
// overwritten before it is read.  Two calls that overlap on the GPU (other streams) race on
// the array and must not be issued.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/tpfwd.h"
#include "common.cuh"
#include "kernels.h"

namespace {
constexpr int kMaxSeqs = TP_STATIC_SCRATCH_MAX_SEQS;
constexpr int kMaxHidden = TP_STATIC_SCRATCH_MAX_HIDDEN;
constexpr int kMaxDevices = 64;

// byte layout of the scratch array
constexpr size_t kZOff = 0;                                              // fp16 [kMaxSeqs][kMaxHidden]
constexpr size_t kCntOff = kZOff + size_t(kMaxSeqs) * kMaxHidden * 2;    // GEMM counters and argmax keys
constexpr size_t kCntBytes = size_t(tpk::kGemmCounterInts) * 4;
constexpr size_t kScratchBytes = kCntOff + kCntBytes;
}  // namespace

// The scratch (about 1 MiB).  Host code only ever sees a host-side stand-in
// for this name; kernels get its device address from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_lm_head_scratch[kScratchBytes];

namespace {

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
tp_status scratch_address(char** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return TP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return TP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_lm_head_scratch);
    if (e != cudaSuccess || !p) return TP_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = static_cast<char*>(g_scratch_addr[dev]);
  return TP_OK;
}

}  // namespace

extern "C" tp_status tp_lm_head_argmax_static(tp_ctx* ctx, const void* head_shards, const tp_batch* b,
                                              const void* hidden, int32_t* out_ids, float* out_logits,
                                              int32_t* dev_status, void* stream) {
  if (!ctx || !head_shards || !b || !hidden || !out_ids || !dev_status) return TP_ERR_INVALID_ARG;
  if (!b->cu_q || b->num_seqs <= 0 || b->num_tokens < b->num_seqs) return TP_ERR_INVALID_ARG;
  // the array's limits, checked before any CUDA call
  if (b->num_seqs > kMaxSeqs) return TP_ERR_INVALID_ARG;
  if (tpk::ctx_hidden_size(ctx) > kMaxHidden) return TP_ERR_INVALID_ARG;
  // outputs: device memory, or page-locked host memory through its device mapping,
  // as tp_lm_head_argmax accepts them; anything else is refused before a launch
  out_ids = tpk::gpu_view(out_ids);
  if (!out_ids) return TP_ERR_INVALID_ARG;
  if (out_logits) {
    out_logits = tpk::gpu_view(out_logits);
    if (!out_logits) return TP_ERR_INVALID_ARG;
  }
  tpk::HeadView hv{};
  tp_status st = static_cast<tp_status>(tpk::ctx_head_view(ctx, &hv));
  if (st != TP_OK) return st;
  char* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != TP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char* w = static_cast<const char*>(head_shards);
  const int B = b->num_seqs;
  void* z = scratch + kZOff;
  // the final norm's weight is folded into the LM head copy: normalize with ones
  cudaError_t e = tpk::launch_final_norm_select(hidden, hv.H, b->cu_q, B, nullptr, hv.eps, z, dev_status, s);
  if (e != cudaSuccess) return TP_ERR_CUDA;
  tpk::GemmProblem g{};
  g.x = z; g.x_rows = B; g.x_cols = hv.H; g.x_ld = hv.H;
  g.w = w + hv.lm_head_off; g.w_rows = static_cast<int64_t>(hv.n) * hv.v_l; g.w_cols = hv.H; g.w_ld = hv.H;
  g.T = B; g.N = static_cast<int>(static_cast<int64_t>(hv.n) * hv.v_l); g.n_seg = 1; g.k_seg = hv.H;
  g.epi = tpk::EPI_ARGMAX; g.out = nullptr; g.ldo = 8; g.out_cols = 0;
  g.amax_val = nullptr;  // per-tile partials: only the many-token path uses them
  g.amax_idx = nullptr;
  g.amax_ld = B; g.logits = out_logits; g.ld_logits = hv.vocab; g.vocab = hv.vocab; g.out_ids = out_ids;
  const tpk::GemmPlan pl = tpk::plan_gemm(g, hv.num_sms);
  if (!pl.swap) return TP_ERR_UNSUPPORTED;
  int* counter = reinterpret_cast<int*>(scratch + kCntOff);
  e = cudaMemsetAsync(counter, 0, kCntBytes, s);  // counters and argmax keys start at zero
  if (e != cudaSuccess) return TP_ERR_CUDA;
  e = tpk::launch_gemm(g, pl, nullptr, counter, dev_status, s);
  return e == cudaSuccess ? TP_OK : TP_ERR_CUDA;
}
