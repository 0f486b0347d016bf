// C-ABI of the tensor-parallel forward (declared in include/tpfwd.h): shard
// rules, device layouts, workspace planning and the launch sequence of each
// call.  Host code only; the arithmetic runs in the kernels of k_*.cu.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/tpfwd.h"
#include "common.cuh"
#include "kernels.h"

namespace {

constexpr size_t kAlign = 1024;
constexpr int kMaxSms = 256;            // bound used to size split-K partials
constexpr int kGemmCounters = 4096;
static_assert(kGemmCounters >= tpk::kGemmCounterInts, "GEMM counter region too small");
constexpr int kMaxDecodeSplits = 64;

thread_local char g_last_cuda_error[256] = "";

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

tp_status cuda_fail(cudaError_t e) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return TP_ERR_CUDA;
}
#define TP_CUDA(call)                        \
  do {                                       \
    cudaError_t e_ = (call);                 \
    if (e_ != cudaSuccess) return cuda_fail(e_); \
  } while (0)

struct Region {
  size_t off = 0, bytes = 0;
};

}  // namespace

struct tp_ctx {
  tp_config c;
  int n, nq_l, nkv_l, i_l, i_p, hd, H;
  int64_t v_l;
  int w_rank;  // merged qkv rows per rank
  int k_r;     // o_proj input columns per rank
  // layer weight parts
  Region qkv, o, gate_up, down, in_norm, post_norm, q_norm, k_norm;
  size_t layer_bytes = 0;
  // head weight parts
  Region embed, lm_head, final_norm;
  size_t head_bytes = 0;
  // workspace
  char* ws = nullptr;
  size_t ws_bytes = 0;
  int ws_tokens = 0, ws_seqs = 0, ws_pos = 0;
  Region r_rope, r_xn, r_qkv, r_qlo, r_attn, r_act, r_gpart, r_gcnt, r_apart, r_acnt, r_amax_v, r_amax_i, r_z, r_ss;
  bool keep_intermediates = false;  // leave dead intermediates in L2 (to read them after a call)
  // the workspace's fp16 residual rows and row sums of squares (the deferred
  // RMSNorm's inputs) belong to this hidden buffer with this many rows, or to none
  const void* stats_for = nullptr;
  int stats_T = -1;
  int lm_tiles_max = 0;
  int num_sms = 0;
  int64_t rank_sums = 0;
  int64_t launches = 0;
  // per-kernel event timing (tp_profile_begin / tp_profile_end)
  bool prof_on = false;
  uint32_t prof_mask = 0;
  std::vector<cudaEvent_t> prof_ev;  // pairs
  std::vector<int> prof_kind;
  int prof_used = 0;
  // a second, higher-priority stream for the prefill attention of a mixed batch
  // (runs beside the decode attention), with the events that fork and join it
  cudaStream_t side = nullptr;
  cudaEvent_t fork_ev = nullptr, join_ev = nullptr;
  ~tp_ctx() {
    for (cudaEvent_t e : prof_ev) cudaEventDestroy(e);
    if (fork_ev) cudaEventDestroy(fork_ev);
    if (join_ev) cudaEventDestroy(join_ev);
    if (side) cudaStreamDestroy(side);
  }
};

namespace {

int64_t div_ceil64(int64_t a, int64_t b) { return (a + b - 1) / b; }

tp_status validate(const tp_config& c) {
  if (c.hidden <= 0 || c.num_q_heads <= 0 || c.num_kv_heads <= 0 || c.head_dim <= 0 || c.intermediate <= 0 ||
      c.vocab <= 0 || c.num_layers < 0 || c.tp_size <= 0 || !(c.rms_eps >= 0.0f) || !(c.rope_theta > 0.0f))
    return TP_ERR_INVALID_ARG;
  const int n = c.tp_size;
  if (c.num_q_heads % c.num_kv_heads) return TP_ERR_INVALID_ARG;
  if (c.num_q_heads % n) return TP_ERR_HEADS_NOT_DIVISIBLE;
  if (c.num_kv_heads >= n && c.num_kv_heads % n) return TP_ERR_KV_HEADS;
  if (c.num_kv_heads < n && n % c.num_kv_heads) return TP_ERR_KV_HEADS;
  if (c.intermediate % n) return TP_ERR_INTERMEDIATE;
  const int64_t per = div_ceil64(c.vocab, n);
  if (static_cast<int64_t>(n - 1) * per >= c.vocab) return TP_ERR_VOCAB;
  // kernel coverage
  if (c.head_dim != 64 && c.head_dim != 128) return TP_ERR_UNSUPPORTED;
  if (c.hidden % 64) return TP_ERR_UNSUPPORTED;
  const int nq_l = c.num_q_heads / n;
  const int nkv_l = c.num_kv_heads >= n ? c.num_kv_heads / n : 1;
  const int G = nq_l / nkv_l;
  if (nq_l % nkv_l || (G != 1 && G != 2 && G != 4 && G != 8)) return TP_ERR_UNSUPPORTED;
  return TP_OK;
}

// kv heads held by rank r ([SHD] weight.py:38-41: head r*nkv/n when nkv < n)
void kv_heads_of_rank(const tp_ctx* x, int r, std::vector<int>& heads) {
  heads.clear();
  const int nkv = x->c.num_kv_heads, n = x->n;
  if (nkv < n) {
    heads.push_back(r * nkv / n);
  } else {
    for (int g = r * (nkv / n); g < (r + 1) * (nkv / n); ++g) heads.push_back(g);
  }
}

void lay_out(tp_ctx* x) {
  size_t off = 0;
  auto take = [&](Region& r, size_t bytes) {
    r.off = off;
    r.bytes = bytes;
    off = align_up(off + bytes);
  };
  const size_t H = x->H, n = x->n;
  take(x->qkv, n * x->w_rank * H * 2);
  take(x->o, n * H * x->k_r * 2);
  take(x->gate_up, n * 2 * static_cast<size_t>(x->i_p) * H * 2);
  take(x->down, n * H * x->i_p * 2);
  take(x->in_norm, H * 2);
  take(x->post_norm, H * 2);
  take(x->q_norm, x->hd * 2);
  take(x->k_norm, x->hd * 2);
  x->layer_bytes = off;
  off = 0;
  take(x->embed, n * x->v_l * H * 2);
  take(x->lm_head, n * x->v_l * H * 2);  // fp16 operand copy, also when tied
  take(x->final_norm, H * 2);
  x->head_bytes = off;
}

struct WsPlan {
  Region rope, xn, qkv, qlo, attn, act, gpart, gcnt, apart, acnt, amax_v, amax_i, z, ss;
  size_t total = 0;
  int lm_tiles = 0;
};

WsPlan plan_ws(const tp_ctx* x, int64_t T, int64_t B, int64_t P) {
  WsPlan w;
  size_t off = 0;
  auto take = [&](Region& r, size_t bytes) {
    r.off = off;
    r.bytes = bytes;
    off = align_up(off + std::max<size_t>(bytes, 16));
  };
  const size_t H = x->H, n = x->n;
  take(w.rope, static_cast<size_t>((P + 31) / 32 * 32) * (x->hd / 2) * 8);
  take(w.xn, T * H * 2);
  take(w.qkv, T * n * x->w_rank * 2);
  take(w.qlo, T * n * x->nq_l * x->hd * 2);
  take(w.attn, T * n * x->nq_l * x->hd * 2);
  take(w.act, T * n * x->i_p * 2);
  // split-K partials: 128 x 128 fp32 per SM, or the residual GEMMs' pair tiles (256
  // tokens x 256 features, two K halves) over all tokens and the hidden size
  const size_t pair_parts = static_cast<size_t>((T + 255) / 256) * ((H + 255) / 256) * 2 * 2 * 256 * 128 * 4;
  take(w.gpart, std::max<size_t>(static_cast<size_t>(kMaxSms) * 128 * 128 * 4, pair_parts));
  take(w.gcnt, kGemmCounters * 4);
  const int64_t splits = std::min<int64_t>(kMaxDecodeSplits, std::max<int64_t>(1, (P + 255) / 256));
  take(w.apart, static_cast<size_t>(B) * n * x->nq_l * (x->hd + 2) * splits * 4);
  take(w.acnt, (static_cast<size_t>(B) * n * x->nkv_l + 2) * 4);  // split counters, then the decode tickets
  w.lm_tiles = static_cast<int>(div_ceil64(n * x->v_l, 64));
  take(w.amax_v, static_cast<size_t>(w.lm_tiles) * B * 4);
  take(w.amax_i, static_cast<size_t>(w.lm_tiles) * B * 4);
  take(w.z, B * H * 2);
  take(w.ss, T * (H / 32) * 4);  // deferred RMSNorm: sums of squares of 32-column groups
  w.total = off;
  return w;
}

tp_status ensure_device(tp_ctx* x) {
  if (x->num_sms > 0) return TP_OK;
  int dev = 0;
  TP_CUDA(cudaGetDevice(&dev));
  int sms = 0;
  TP_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
  if (sms <= 0 || sms > kMaxSms) return TP_ERR_UNSUPPORTED;
  x->num_sms = sms;
  return TP_OK;
}

template <typename T>
T* at(const void* base, const Region& r) {
  return reinterpret_cast<T*>(const_cast<char*>(reinterpret_cast<const char*>(base)) + r.off);
}

tp_status check_batch(const tp_ctx* x, const tp_batch* b) {
  if (!b || !b->cu_q || !b->ctx_len || (!b->slot && !b->page_table)) return TP_ERR_INVALID_ARG;
  if (b->page_table) {  // paged cache: pages hold whole 128-key tiles
    if (b->page_size <= 0 || b->page_size % tpk::kKeyAlign || b->max_pages_per_seq <= 0) return TP_ERR_INVALID_ARG;
    if (static_cast<int64_t>(b->max_kv_len) > static_cast<int64_t>(b->max_pages_per_seq) * b->page_size)
      return TP_ERR_INVALID_ARG;
  }
  if (b->num_seqs <= 0 || b->num_seqs > x->ws_seqs) return TP_ERR_INVALID_ARG;
  if (b->num_prefill < 0 || b->num_prefill > b->num_seqs) return TP_ERR_INVALID_ARG;
  if (b->num_tokens < b->num_seqs || b->num_tokens > x->ws_tokens) return TP_ERR_INVALID_ARG;
  if (b->max_kv_len <= 0 || b->max_kv_len > x->ws_pos) return TP_ERR_INVALID_ARG;
  if (b->num_prefill > 0 && (b->max_q_len <= 0 || b->max_q_len > b->num_tokens)) return TP_ERR_INVALID_ARG;
  return TP_OK;
}

// Brackets one launch site with profiling events when its kind is selected.
struct Timed {
  tp_ctx* x;
  cudaStream_t s;
  int slot = -1;
  Timed(tp_ctx* x_, int kind, cudaStream_t s_, int kernels = 1) : x(x_), s(s_) {
    x->launches += kernels;
    if (x->prof_on && (x->prof_mask >> kind & 1u) && 2 * (x->prof_used + 1) <= static_cast<int>(x->prof_ev.size())) {
      slot = x->prof_used++;
      x->prof_kind[slot] = kind;
      cudaEventRecord(x->prof_ev[2 * slot], s);
    }
  }
  ~Timed() {
    if (slot >= 0) cudaEventRecord(x->prof_ev[2 * slot + 1], s);
  }
};

// Whole 128-byte lines of [p, p + bytes) for a GEMM's L2 discard list (p is
// 256-byte aligned: workspace regions are).
void set_discard(const tp_ctx* x, tpk::GemmProblem& g, int k, const void* p, size_t bytes) {
  if (x->keep_intermediates) return;
  g.discard[k] = p;
  g.discard_lines[k] = static_cast<int64_t>(bytes / 128);
}

tp_status gemm(tp_ctx* x, int kind, const tpk::GemmProblem& pr, int32_t* dev_status, cudaStream_t s) {
  tpk::GemmPlan pl = tpk::plan_gemm(pr, x->num_sms);
  if (pl.partial_floats * 4 > x->r_gpart.bytes) return TP_ERR_UNSUPPORTED;
  if (pl.splits > 1 && (pl.pair ? 2 : 1) * pl.tiles_t * pl.tiles_f > tpk::kArgmaxKeyOffset) return TP_ERR_UNSUPPORTED;
  Timed tm(x, kind, s);
  cudaError_t e = tpk::launch_gemm(pr, pl, at<float>(x->ws, x->r_gpart), at<int>(x->ws, x->r_gcnt), dev_status, s);
  if (e != cudaSuccess) return cuda_fail(e);
  return TP_OK;
}

}  // namespace

int tpk::ctx_hidden_size(const tp_ctx* x) { return x ? x->H : 0; }

int tpk::ctx_head_view(tp_ctx* x, tpk::HeadView* out) {
  if (!x || !out) return TP_ERR_INVALID_ARG;
  const tp_status st = ensure_device(x);
  if (st != TP_OK) return st;
  out->H = x->H;
  out->n = x->n;
  out->vocab = x->c.vocab;
  out->num_sms = x->num_sms;
  out->v_l = x->v_l;
  out->lm_head_off = x->lm_head.off;
  out->final_norm_off = x->final_norm.off;
  out->eps = x->c.rms_eps;
  return TP_OK;
}

extern "C" {

const char* tp_last_cuda_error(void) { return g_last_cuda_error; }

const char* tp_status_string(tp_status s) {
  switch (s) {
    case TP_OK: return "ok";
    case TP_ERR_INVALID_ARG: return "invalid argument";
    case TP_ERR_HEADS_NOT_DIVISIBLE: return "query heads not divisible by tp_size";
    case TP_ERR_KV_HEADS: return "kv heads neither divisible by nor dividing tp_size";
    case TP_ERR_INTERMEDIATE: return "intermediate size not divisible by tp_size";
    case TP_ERR_VOCAB: return "a rank's vocab slice would be empty";
    case TP_ERR_UNSUPPORTED: return "shape not supported by the kernels";
    case TP_ERR_CUDA: return "CUDA error";
    case TP_ERR_BAD_TOKEN: return "token id or position out of range";
    case TP_ERR_TIMEOUT: return "bounded wait timed out in a kernel";
    case TP_ERR_SATURATED: return "an fp16 operand exceeded the fp16 range and was clamped";
    default: return "unknown status";
  }
}

tp_status tp_create(const tp_config* cfg, tp_ctx** out) {
  if (!cfg || !out) return TP_ERR_INVALID_ARG;
  *out = nullptr;
  tp_status st = validate(*cfg);
  if (st != TP_OK) return st;
  tp_ctx* x = new (std::nothrow) tp_ctx();
  if (!x) return TP_ERR_INVALID_ARG;
  x->c = *cfg;
  x->n = cfg->tp_size;
  x->H = cfg->hidden;
  x->hd = cfg->head_dim;
  x->nq_l = cfg->num_q_heads / x->n;
  x->nkv_l = cfg->num_kv_heads >= x->n ? cfg->num_kv_heads / x->n : 1;
  x->i_l = cfg->intermediate / x->n;
  x->i_p = (x->i_l + 63) / 64 * 64;
  x->v_l = div_ceil64(cfg->vocab, x->n);
  x->w_rank = (x->nq_l + 2 * x->nkv_l) * x->hd;
  x->k_r = x->nq_l * x->hd;
  lay_out(x);
  *out = x;
  return TP_OK;
}

tp_status tp_destroy(tp_ctx* ctx) {
  delete ctx;
  return TP_OK;
}

tp_status tp_shard_index_map(const tp_ctx* x, int32_t kind, int32_t rank, int64_t* src_idx, int64_t* len,
                             int32_t* dim) {
  if (!x || !len || !dim || rank < 0 || rank >= x->n) return TP_ERR_INVALID_ARG;
  std::vector<int64_t> idx;
  auto range = [&](int64_t a, int64_t b) {
    for (int64_t i = a; i < b; ++i) idx.push_back(i);
  };
  const int64_t hd = x->hd, n = x->n;
  switch (kind) {
    case TP_PARAM_Q: {
      const int64_t per = x->c.num_q_heads * hd / n;
      range(rank * per, (rank + 1) * per);
      *dim = 0;
      break;
    }
    case TP_PARAM_K:
    case TP_PARAM_V: {
      std::vector<int> heads;
      kv_heads_of_rank(x, rank, heads);
      for (int g : heads) range(g * hd, (g + 1) * hd);
      *dim = 0;
      break;
    }
    case TP_PARAM_GATE:
    case TP_PARAM_UP:
      range(static_cast<int64_t>(rank) * x->i_l, static_cast<int64_t>(rank + 1) * x->i_l);
      *dim = 0;
      break;
    case TP_PARAM_O: {
      const int64_t per = x->c.num_q_heads * hd / n;
      range(rank * per, (rank + 1) * per);
      *dim = 1;
      break;
    }
    case TP_PARAM_DOWN:
      range(static_cast<int64_t>(rank) * x->i_l, static_cast<int64_t>(rank + 1) * x->i_l);
      *dim = 1;
      break;
    case TP_PARAM_EMBED:
    case TP_PARAM_LM_HEAD:
      range(rank * x->v_l, std::min<int64_t>((rank + 1) * x->v_l, x->c.vocab));
      *dim = 0;
      break;
    case TP_PARAM_NORM:
      range(0, x->H);
      *dim = -1;
      break;
    default:
      return TP_ERR_INVALID_ARG;
  }
  *len = static_cast<int64_t>(idx.size());
  if (src_idx) std::memcpy(src_idx, idx.data(), idx.size() * sizeof(int64_t));
  return TP_OK;
}

tp_status tp_weights_bytes(const tp_ctx* x, int32_t which, size_t* bytes) {
  if (!x || !bytes) return TP_ERR_INVALID_ARG;
  if (which == TP_WEIGHTS_LAYER) *bytes = x->layer_bytes;
  else if (which == TP_WEIGHTS_HEAD) *bytes = x->head_bytes;
  else return TP_ERR_INVALID_ARG;
  return TP_OK;
}

tp_status tp_weights_part(const tp_ctx* x, int32_t part, size_t* offset, size_t* bytes) {
  if (!x || !offset || !bytes) return TP_ERR_INVALID_ARG;
  const Region* r = nullptr;
  switch (part) {
    case TP_PART_QKV: r = &x->qkv; break;
    case TP_PART_O: r = &x->o; break;
    case TP_PART_GATE_UP: r = &x->gate_up; break;
    case TP_PART_DOWN: r = &x->down; break;
    case TP_PART_IN_NORM: r = &x->in_norm; break;
    case TP_PART_POST_NORM: r = &x->post_norm; break;
    case TP_PART_Q_NORM: r = &x->q_norm; break;
    case TP_PART_K_NORM: r = &x->k_norm; break;
    case TP_PART_EMBED: r = &x->embed; break;
    case TP_PART_LM_HEAD: r = &x->lm_head; break;
    case TP_PART_FINAL_NORM: r = &x->final_norm; break;
    default: return TP_ERR_INVALID_ARG;
  }
  *offset = r->off;
  *bytes = r->bytes;
  return TP_OK;
}

tp_status tp_shard_weights(tp_ctx* x, const tp_layer_full* L, const tp_head_full* Hd, void* dst, int32_t* dev_status,
                           void* stream) {
  if (!x || !dst || (L == nullptr) == (Hd == nullptr)) return TP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* d = static_cast<char*>(dst);
  const size_t H = x->H, hd = x->hd, row = H * 2;
  const int n = x->n;
  if (L) {
    if (!L->q || !L->k || !L->v || !L->o || !L->gate || !L->up || !L->down || !L->in_norm || !L->post_norm ||
        !L->q_norm || !L->k_norm)
      return TP_ERR_INVALID_ARG;
    TP_CUDA(cudaMemsetAsync(d, 0, x->layer_bytes, s));
    std::vector<int> heads;
    const size_t q_rows = static_cast<size_t>(x->nq_l) * hd;
    for (int r = 0; r < n; ++r) {
      // merged qkv: [q_r; k_r; v_r]  ([CH9] 3.3: shard first, then merge)
      char* blk = d + x->qkv.off + static_cast<size_t>(r) * x->w_rank * row;
      TP_CUDA(cudaMemcpyAsync(blk, static_cast<const char*>(L->q) + r * q_rows * row, q_rows * row,
                              cudaMemcpyDeviceToDevice, s));
      kv_heads_of_rank(x, r, heads);
      size_t kr = q_rows;
      for (int g : heads) {
        TP_CUDA(cudaMemcpyAsync(blk + kr * row, static_cast<const char*>(L->k) + g * hd * row, hd * row,
                                cudaMemcpyDeviceToDevice, s));
        kr += hd;
      }
      for (int g : heads) {
        TP_CUDA(cudaMemcpyAsync(blk + kr * row, static_cast<const char*>(L->v) + g * hd * row, hd * row,
                                cudaMemcpyDeviceToDevice, s));
        kr += hd;
      }
      // o_proj columns [r*k_r, (r+1)*k_r) of [H, nq*hd]
      const size_t o_ld = static_cast<size_t>(x->c.num_q_heads) * hd * 2;
      TP_CUDA(cudaMemcpy2DAsync(d + x->o.off + static_cast<size_t>(r) * H * x->k_r * 2, x->k_r * 2,
                                static_cast<const char*>(L->o) + static_cast<size_t>(r) * x->k_r * 2, o_ld,
                                x->k_r * 2, H, cudaMemcpyDeviceToDevice, s));
      // gate/up rows [r*i_l, (r+1)*i_l), interleaved in blocks of 64 rows
      for (int j = 0; j * 64 < x->i_l; ++j) {
        const size_t rows = std::min(64, x->i_l - j * 64);
        const size_t src_row = static_cast<size_t>(r) * x->i_l + j * 64;
        char* gdst = d + x->gate_up.off + ((static_cast<size_t>(r) * (x->i_p / 64) + j) * 128) * row;
        TP_CUDA(cudaMemcpyAsync(gdst, static_cast<const char*>(L->gate) + src_row * row, rows * row,
                                cudaMemcpyDeviceToDevice, s));
        TP_CUDA(cudaMemcpyAsync(gdst + 64 * row, static_cast<const char*>(L->up) + src_row * row, rows * row,
                                cudaMemcpyDeviceToDevice, s));
      }
      // down columns [r*i_l, (r+1)*i_l) of [H, I] into [H, i_p]
      TP_CUDA(cudaMemcpy2DAsync(d + x->down.off + static_cast<size_t>(r) * H * x->i_p * 2,
                                static_cast<size_t>(x->i_p) * 2,
                                static_cast<const char*>(L->down) + static_cast<size_t>(r) * x->i_l * 2,
                                static_cast<size_t>(x->c.intermediate) * 2, static_cast<size_t>(x->i_l) * 2, H,
                                cudaMemcpyDeviceToDevice, s));
    }
    TP_CUDA(cudaMemcpyAsync(d + x->in_norm.off, L->in_norm, row, cudaMemcpyDeviceToDevice, s));
    TP_CUDA(cudaMemcpyAsync(d + x->post_norm.off, L->post_norm, row, cudaMemcpyDeviceToDevice, s));
    TP_CUDA(cudaMemcpyAsync(d + x->q_norm.off, L->q_norm, hd * 2, cudaMemcpyDeviceToDevice, s));
    TP_CUDA(cudaMemcpyAsync(d + x->k_norm.off, L->k_norm, hd * 2, cudaMemcpyDeviceToDevice, s));
    // the projection shards are tensor-core operands: stored fp16; the RMSNorm
    // weights that precede QKV and gate_up are folded into their columns
    // (x_n W^T = (x inv) (W diag(w))^T, the row scale inv applied in the epilogue)
    {
      cudaError_t e = tpk::launch_fold_norm_f16(d + x->qkv.off, static_cast<size_t>(n) * x->w_rank, x->H,
                                                d + x->in_norm.off, dev_status, s);
      if (e == cudaSuccess)
        e = tpk::launch_fold_norm_f16(d + x->gate_up.off, static_cast<size_t>(n) * 2 * x->i_p, x->H,
                                      d + x->post_norm.off, dev_status, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    for (const Region* r : {&x->o, &x->down}) {
      cudaError_t e = tpk::launch_bf16_to_f16(d + r->off, r->bytes / 2, dev_status, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    return TP_OK;
  }
  if (!Hd->embed || !Hd->final_norm || (!x->c.tie_word_embeddings && !Hd->lm_head)) return TP_ERR_INVALID_ARG;
  TP_CUDA(cudaMemsetAsync(d, 0, x->head_bytes, s));
  for (int r = 0; r < n; ++r) {
    const int64_t a = r * x->v_l, b = std::min<int64_t>((r + 1) * x->v_l, x->c.vocab);
    TP_CUDA(cudaMemcpyAsync(d + x->embed.off + static_cast<size_t>(r) * x->v_l * row,
                            static_cast<const char*>(Hd->embed) + a * row, (b - a) * row, cudaMemcpyDeviceToDevice,
                            s));
    const void* lm = x->c.tie_word_embeddings ? Hd->embed : Hd->lm_head;
    TP_CUDA(cudaMemcpyAsync(d + x->lm_head.off + static_cast<size_t>(r) * x->v_l * row,
                            static_cast<const char*>(lm) + a * row, (b - a) * row, cudaMemcpyDeviceToDevice, s));
  }
  TP_CUDA(cudaMemcpyAsync(d + x->final_norm.off, Hd->final_norm, row, cudaMemcpyDeviceToDevice, s));
  {
    // the LM head's fp16 copy carries the final RMSNorm weight in its columns (the
    // norm's row scale is applied to the logits, or dropped for the argmax alone)
    cudaError_t e = tpk::launch_fold_norm_f16(d + x->lm_head.off, static_cast<size_t>(n) * x->v_l, x->H,
                                              d + x->final_norm.off, dev_status, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  return TP_OK;
}

tp_status tp_kv_cache_bytes(const tp_ctx* x, int32_t max_seqs, int32_t capacity, size_t* bytes) {
  if (!x || !bytes || max_seqs <= 0 || capacity <= 0) return TP_ERR_INVALID_ARG;
  *bytes = static_cast<size_t>(x->n) * 2 * max_seqs * x->nkv_l * capacity * x->hd * 2;
  return TP_OK;
}

tp_status tp_workspace_bytes(const tp_ctx* x, int32_t max_tokens, int32_t max_seqs, int32_t max_positions,
                             size_t* bytes) {
  if (!x || !bytes || max_tokens <= 0 || max_seqs <= 0 || max_positions <= 0) return TP_ERR_INVALID_ARG;
  *bytes = plan_ws(x, max_tokens, max_seqs, max_positions).total;
  return TP_OK;
}

tp_status tp_workspace_init(tp_ctx* x, void* ws, size_t ws_bytes, int32_t max_tokens, int32_t max_seqs,
                            int32_t max_positions, void* stream) {
  if (!x || !ws || max_tokens <= 0 || max_seqs <= 0 || max_positions <= 0) return TP_ERR_INVALID_ARG;
  const WsPlan w = plan_ws(x, max_tokens, max_seqs, max_positions);
  if (ws_bytes < w.total) return TP_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(ws) % 256) return TP_ERR_INVALID_ARG;
  tp_status st = ensure_device(x);
  if (st != TP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  x->ws = static_cast<char*>(ws);
  x->ws_bytes = ws_bytes;
  x->ws_tokens = max_tokens;
  x->ws_seqs = max_seqs;
  x->ws_pos = max_positions;
  x->r_rope = w.rope; x->r_xn = w.xn; x->r_qkv = w.qkv; x->r_qlo = w.qlo; x->r_attn = w.attn; x->r_act = w.act;
  x->r_gpart = w.gpart; x->r_gcnt = w.gcnt; x->r_apart = w.apart; x->r_acnt = w.acnt;
  x->r_amax_v = w.amax_v; x->r_amax_i = w.amax_i; x->r_z = w.z; x->r_ss = w.ss;
  x->lm_tiles_max = w.lm_tiles;
  TP_CUDA(cudaMemsetAsync(x->ws + w.gcnt.off, 0, w.gcnt.bytes, s));
  TP_CUDA(cudaMemsetAsync(x->ws + w.acnt.off, 0, w.acnt.bytes, s));
  // RoPE table: angle(p, d) = p * theta^(-2d/hd), rotate-half pairs (d, d + hd/2); fp64, stored
  // fp32 as (cos, sin).  Blocked by 32 positions so that the 32 consecutive positions a warp
  // reads side by side are adjacent: float4 (cos_d, sin_d, cos_d+1, sin_d+1) of position p at
  // index ((p / 32) * (hd / 4) + d / 2) * 32 + p % 32.
  const int half = x->hd / 2;
  const int P32 = (max_positions + 31) / 32 * 32;
  std::vector<float> tab(static_cast<size_t>(P32) * half * 2, 0.0f);
  for (int d = 0; d < half; ++d) {
    const double inv_freq = std::pow(static_cast<double>(x->c.rope_theta), -2.0 * d / x->hd);
    for (int p = 0; p < max_positions; ++p) {
      const double ang = static_cast<double>(p) * inv_freq;
      const size_t f4 = (static_cast<size_t>(p / 32) * (half / 2) + d / 2) * 32 + p % 32;
      tab[f4 * 4 + (d % 2) * 2] = static_cast<float>(std::cos(ang));
      tab[f4 * 4 + (d % 2) * 2 + 1] = static_cast<float>(std::sin(ang));
    }
  }
  TP_CUDA(cudaMemcpyAsync(x->ws + w.rope.off, tab.data(), tab.size() * 4, cudaMemcpyHostToDevice, s));
  TP_CUDA(cudaStreamSynchronize(s));
  return TP_OK;
}

tp_status tp_embed_vocab_parallel(tp_ctx* x, const void* head_shards, const int32_t* ids, int32_t T,
                                  void* hidden_out, int32_t* dev_status, void* stream) {
  if (!x || !head_shards || !ids || !hidden_out || !dev_status || T <= 0) return TP_ERR_INVALID_ARG;
  ids = tpk::gpu_view(ids);  // page-locked host ids are read by the kernel over the host link
  if (!ids) return TP_ERR_INVALID_ARG;
  cudaError_t e;
  // with a workspace large enough, also the first layer's deferred-norm inputs
  const bool stats = x->ws != nullptr && T <= x->ws_tokens;
  x->stats_for = nullptr;
  {
    Timed tm(x, TP_K_EMBED, static_cast<cudaStream_t>(stream));
    e = tpk::launch_embed(ids, T, static_cast<const char*>(head_shards) + x->embed.off, x->n, x->v_l, x->c.vocab,
                          x->H, hidden_out, stats ? x->ws + x->r_xn.off : nullptr,
                          stats ? reinterpret_cast<float*>(x->ws + x->r_ss.off) : nullptr, dev_status,
                          static_cast<cudaStream_t>(stream));
  }
  if (e != cudaSuccess) return cuda_fail(e);
  if (stats) {
    x->stats_for = hidden_out;
    x->stats_T = T;
  }
  x->rank_sums += 1;
  return TP_OK;
}

tp_status tp_decoder_layer_forward(tp_ctx* x, const void* shards, const tp_batch* b, void* hidden, void* kv,
                                   int32_t kv_max_seqs, int32_t kv_cap, int32_t* dev_status, void* stream) {
  if (!x || !shards || !hidden || !kv || !dev_status || !x->ws) return TP_ERR_INVALID_ARG;
  tp_status st = check_batch(x, b);
  if (st != TP_OK) return st;
  if (kv_max_seqs <= 0 || kv_cap <= 0) return TP_ERR_INVALID_ARG;
  if (b->page_table ? kv_cap != b->page_size : kv_cap < b->max_kv_len) return TP_ERR_INVALID_ARG;
  // the cache's blocks: slots of a contiguous cache, or pages
  tpk::KvMap kvm;
  if (b->page_table) {
    kvm.table = b->page_table; kvm.stride = b->max_pages_per_seq; kvm.block_len = b->page_size;
  } else {
    kvm.table = b->slot; kvm.stride = 1; kvm.block_len = kv_cap;
  }
  kvm.blocks = kv_max_seqs;
  st = ensure_device(x);
  if (st != TP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char* w = static_cast<const char*>(shards);
  const int T = b->num_tokens, H = x->H, n = x->n;
  void* xn = x->ws + x->r_xn.off;
  void* qkv = x->ws + x->r_qkv.off;
  void* attn = x->ws + x->r_attn.off;
  void* act = x->ws + x->r_act.off;
  cudaError_t e;

  float* ss = reinterpret_cast<float*>(x->ws + x->r_ss.off);

  // A3: input RMSNorm, deferred: w_in is folded into the QKV weights and each row's
  // rsqrt(mean + eps) scales its accumulators in the QKV epilogue.  Its inputs (the
  // fp16 residual rows and their 32-column sums of squares) are left in the
  // workspace by the embedding or the previous layer's down_proj epilogue; computed
  // here only when hidden came from elsewhere.
  const bool have_stats = x->stats_for == hidden && x->stats_T == T;
  x->stats_for = nullptr;  // until this call completes
  if (!have_stats) {
    Timed tm(x, TP_K_RMSNORM, s);
    e = tpk::launch_row_stats(hidden, T, H, xn, ss, dev_status, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }

  // A4 + A5: merged QKV of all ranks (column split: no exchange), with q/k RMSNorm,
  // RoPE and the K/V cache write fused into the epilogue (fp32, no intermediate rounding)
  tpk::GemmProblem g{};
  g.x = xn; g.x_rows = T; g.x_cols = H; g.x_ld = H;
  g.w = w + x->qkv.off; g.w_rows = static_cast<int64_t>(n) * x->w_rank; g.w_cols = H; g.w_ld = H;
  g.T = T; g.N = n * x->w_rank; g.n_seg = 1; g.k_seg = H; g.x_k_seg = 0; g.w_row_seg = 0;
  g.epi = tpk::EPI_QKV; g.out = qkv; g.ldo = n * x->w_rank; g.out_cols = n * x->w_rank;
  g.qkv.n = n; g.qkv.nq_l = x->nq_l; g.qkv.nkv_l = x->nkv_l; g.qkv.hd = x->hd; g.qkv.w_rank = x->w_rank;
  g.qkv.q_norm = w + x->q_norm.off; g.qkv.k_norm = w + x->k_norm.off; g.qkv.eps = x->c.rms_eps;
  g.qkv.rope = reinterpret_cast<const float2*>(x->ws + x->r_rope.off); g.qkv.max_pos = x->ws_pos;
  g.qkv.cu_q = b->cu_q; g.qkv.ctx_len = b->ctx_len; g.qkv.B = b->num_seqs;
  g.qkv.kv = kv; g.qkv.kvm = kvm;
  g.qkv.num_prefill = b->num_prefill; g.qkv.q_lo = x->ws + x->r_qlo.off;
  g.row_ss = ss; g.row_groups = H / 32; g.row_eps = x->c.rms_eps;
  // dead by now: the SiLU*up rows of the previous layer (read by its down_proj)
  set_discard(x, g, 0, act, static_cast<size_t>(T) * n * x->i_p * 2);
  st = gemm(x, TP_K_GEMM_QKV, g, dev_status, s);
  if (st != TP_OK) return st;

  // A6: per-rank attention
  tpk::AttnArgs aa{};
  aa.qkv = qkv; aa.q_lo = x->ws + x->r_qlo.off; aa.T = T; aa.n = n; aa.nq_l = x->nq_l; aa.nkv_l = x->nkv_l; aa.hd = x->hd; aa.w_rank = x->w_rank;
  aa.kv = kv; aa.kvm = kvm;
  aa.cu_q = b->cu_q; aa.ctx_len = b->ctx_len;
  aa.max_q_len = b->max_q_len; aa.max_kv_len = b->max_kv_len; aa.out = attn;
  aa.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(x->hd)));
  aa.part = reinterpret_cast<float*>(x->ws + x->r_apart.off);
  aa.counters = reinterpret_cast<int*>(x->ws + x->r_acnt.off);
  aa.sched = aa.counters + static_cast<size_t>(x->ws_seqs) * n * x->nkv_l;
  aa.status = dev_status;
  // A mixed batch runs its two attention kernels side by side: the prefill
  // attention (tensor cores, a few persistent CTAs) on a second, higher-priority
  // stream forked after the QKV GEMM and joined before o_proj, the decode attention
  // (HBM-bound, which keeps HBM saturated on the remaining SMs) on the caller's stream.
  const bool has_decode = b->num_prefill < b->num_seqs;
  const bool side_by_side = b->num_prefill > 0 && has_decode;
  cudaStream_t ps = s;
  const int pre_ctas = std::max(8, x->num_sms * 3 / 8);  // the prefill attention's CTAs beside the decode
  if (side_by_side) {
    if (!x->side) {
      int least = 0, greatest = 0;
      TP_CUDA(cudaDeviceGetStreamPriorityRange(&least, &greatest));
      TP_CUDA(cudaStreamCreateWithPriority(&x->side, cudaStreamNonBlocking, greatest));
      TP_CUDA(cudaEventCreateWithFlags(&x->fork_ev, cudaEventDisableTiming));
      TP_CUDA(cudaEventCreateWithFlags(&x->join_ev, cudaEventDisableTiming));
    }
    TP_CUDA(cudaEventRecord(x->fork_ev, s));
    TP_CUDA(cudaStreamWaitEvent(x->side, x->fork_ev, 0));
    ps = x->side;
  }
  if (b->num_prefill > 0) {
    aa.seq_begin = 0; aa.seq_end = b->num_prefill;
    // beside the decode attention 3/8 of the SMs walk the work items (measured on
    // the 28-layer mixed step, 128 decode + 4 x 512 prefill tokens, beside the
    // persistent decode kernel: 16 / 24 / 30 / 38 / 48 / 57 / 76 CTAs gave 7.61 /
    // 7.51 / 7.48 / 7.45 / 7.42 / 7.42 / 7.44 ms); alone, one CTA per item, which
    // the hardware hands to SMs as they free up (heaviest items first)
    aa.ctas = side_by_side ? pre_ctas : INT_MAX;
    Timed tm(x, TP_K_ATTN_PREFILL, ps);
    e = tpk::launch_attention_prefill(aa, ps);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  if (has_decode) {
    aa.seq_begin = b->num_prefill; aa.seq_end = b->num_seqs;
    const int units = (b->num_seqs - b->num_prefill) * n * x->nkv_l;
    // split partials must fit the workspace region planned for them
    const int64_t per_split = static_cast<int64_t>(b->num_seqs - b->num_prefill) * n * x->nq_l * (x->hd + 2) * 4;
    const int max_splits = static_cast<int>(std::min<int64_t>(64, static_cast<int64_t>(x->r_apart.bytes) / per_split));
    const tpk::DecodeSplit ds =
        tpk::decode_split_plan(b->max_kv_len, units, x->num_sms, x->hd, x->nq_l / x->nkv_l, std::max(1, max_splits));
    aa.plan = ds;
    // the persistent decode kernel: one CTA per SM (two pipelines each) drawing
    // items from a ticket counter.  Beside a prefill attention it leaves that
    // kernel's SMs free, and a second launch on the prefill's stream takes them
    // over once the prefill ends, drawing from the same counter.
    const int items = tpk::plan_items(ds);
    const int want = std::max(1, std::min(x->num_sms, (items + 1) / 2));
    const bool persistent = x->hd == 128;  // the tensor-core kernel (64-dim heads: a CTA per item)
    const int side_ctas =
        side_by_side && persistent ? std::min(pre_ctas, std::max(0, want - (x->num_sms - pre_ctas))) : 0;
    aa.ctas = want - side_ctas;
    aa.sched_ctas = want;
    {
      Timed tm(x, TP_K_ATTN_DECODE, s);
      e = tpk::launch_attention_decode(aa, s);
      if (e != cudaSuccess) return cuda_fail(e);
    }
    if (side_ctas > 0) {
      aa.ctas = side_ctas;
      x->launches += 1;  // counted, not timed: it runs inside the timed launch above
      e = tpk::launch_attention_decode(aa, ps);
      if (e != cudaSuccess) return cuda_fail(e);
    }
  }
  if (side_by_side) {
    TP_CUDA(cudaEventRecord(x->join_ev, x->side));
    TP_CUDA(cudaStreamWaitEvent(s, x->join_ev, 0));
  }

  // A7: o_proj (row split) per rank, rank-sum in fixed order + residual, in place on hidden
  g = tpk::GemmProblem{};
  g.x = attn; g.x_rows = T; g.x_cols = static_cast<int64_t>(n) * x->k_r; g.x_ld = g.x_cols;
  g.w = w + x->o.off; g.w_rows = static_cast<int64_t>(n) * H; g.w_cols = x->k_r; g.w_ld = x->k_r;
  g.T = T; g.N = H; g.n_seg = n; g.k_seg = x->k_r; g.x_k_seg = x->k_r; g.w_row_seg = H;
  g.epi = tpk::EPI_RESID; g.out = hidden; g.ldo = H; g.out_cols = H;
  // A8 (post-attention RMSNorm, deferred into gate_up): its inputs from this epilogue
  g.row_out16 = xn; g.row_ss_out = ss;
  // dead by now: q (high part / decode q) and its low part, read by the attention
  set_discard(x, g, 0, qkv, static_cast<size_t>(T) * n * x->w_rank * 2);
  set_discard(x, g, 1, x->ws + x->r_qlo.off, static_cast<size_t>(T) * n * x->nq_l * x->hd * 2);
  st = gemm(x, TP_K_GEMM_O, g, dev_status, s);
  if (st != TP_OK) return st;
  x->rank_sums += 1;

  // A8: post-attention RMSNorm, deferred as A3 (w_post folded into gate_up; its
  // inputs came from the o_proj epilogue)

  // A9: merged gate/up of all ranks (column split) with SiLU(gate) * up
  g = tpk::GemmProblem{};
  g.x = xn; g.x_rows = T; g.x_cols = H; g.x_ld = H;
  g.w = w + x->gate_up.off; g.w_rows = static_cast<int64_t>(n) * 2 * x->i_p; g.w_cols = H; g.w_ld = H;
  g.T = T; g.N = n * 2 * x->i_p; g.n_seg = 1; g.k_seg = H;
  g.epi = tpk::EPI_SILU; g.out = act; g.ldo = n * x->i_p; g.out_cols = n * x->i_p;
  g.row_ss = ss; g.row_groups = H / 32; g.row_eps = x->c.rms_eps;
  // dead by now: the attention output, read by o_proj
  set_discard(x, g, 0, attn, static_cast<size_t>(T) * n * x->nq_l * x->hd * 2);
  st = gemm(x, TP_K_GEMM_GATE_UP, g, dev_status, s);
  if (st != TP_OK) return st;

  // A10: down_proj (row split) per rank, rank-sum + residual
  g = tpk::GemmProblem{};
  g.x = act; g.x_rows = T; g.x_cols = static_cast<int64_t>(n) * x->i_p; g.x_ld = g.x_cols;
  g.w = w + x->down.off; g.w_rows = static_cast<int64_t>(n) * H; g.w_cols = x->i_p; g.w_ld = x->i_p;
  g.T = T; g.N = H; g.n_seg = n; g.k_seg = x->i_p; g.x_k_seg = x->i_p; g.w_row_seg = H;
  g.epi = tpk::EPI_RESID; g.out = hidden; g.ldo = H; g.out_cols = H;
  // the next layer's deferred input norm: its inputs from this epilogue
  g.row_out16 = xn; g.row_ss_out = ss;
  st = gemm(x, TP_K_GEMM_DOWN, g, dev_status, s);
  if (st != TP_OK) return st;
  x->rank_sums += 1;
  x->stats_for = hidden;
  x->stats_T = T;
  return TP_OK;
}

tp_status tp_lm_head_argmax(tp_ctx* x, const void* head_shards, const tp_batch* b, const void* hidden,
                            int32_t* out_ids, float* out_logits, int32_t* dev_status, void* stream) {
  if (!x || !head_shards || !hidden || !out_ids || !dev_status || !x->ws) return TP_ERR_INVALID_ARG;
  out_ids = tpk::gpu_view(out_ids);  // page-locked host ids are written by the kernel over the host link
  if (!out_ids) return TP_ERR_INVALID_ARG;
  if (out_logits) {  // the same rule for the logits
    out_logits = tpk::gpu_view(out_logits);
    if (!out_logits) return TP_ERR_INVALID_ARG;
  }
  tp_status st = check_batch(x, b);
  if (st != TP_OK) return st;
  st = ensure_device(x);
  if (st != TP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char* w = static_cast<const char*>(head_shards);
  const int B = b->num_seqs, H = x->H;
  void* z = x->ws + x->r_z.off;
  cudaError_t e;
  // A11.  The final norm's weight is folded into the LM head copy, and its row scale
  // rsqrt(mean(x^2) + eps) > 0 does not move the argmax: when only the ids are asked
  // for and the last tokens' fp16 rows (left by the last down_proj) are contiguous
  // (one sequence, or one token per sequence), the head reads them directly;
  // otherwise the select kernel gathers and normalizes the rows (ones for weight).
  const bool contiguous = B == 1 || (b->num_prefill == 0 && b->num_tokens == B);
  const bool direct = out_logits == nullptr && contiguous && x->stats_for == hidden && x->stats_T == b->num_tokens;
  const void* zin = z;
  if (direct) {
    zin = x->ws + x->r_xn.off + static_cast<size_t>(B == 1 ? b->num_tokens - 1 : 0) * H * 2;
  } else {
    Timed tm(x, TP_K_FINAL_NORM, s);
    e = tpk::launch_final_norm_select(hidden, H, b->cu_q, B, nullptr, x->c.rms_eps, z, dev_status, s);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  tpk::GemmProblem g{};
  g.x = zin; g.x_rows = B; g.x_cols = H; g.x_ld = H;
  g.w = w + x->lm_head.off; g.w_rows = static_cast<int64_t>(x->n) * x->v_l; g.w_cols = H; g.w_ld = H;
  g.T = B; g.N = static_cast<int>(static_cast<int64_t>(x->n) * x->v_l); g.n_seg = 1; g.k_seg = H;
  g.epi = tpk::EPI_ARGMAX; g.out = nullptr; g.ldo = 8; g.out_cols = 0;
  g.amax_val = reinterpret_cast<float*>(x->ws + x->r_amax_v.off);
  g.amax_idx = reinterpret_cast<int*>(x->ws + x->r_amax_i.off);
  g.amax_ld = B; g.logits = out_logits; g.ld_logits = x->c.vocab; g.vocab = x->c.vocab; g.out_ids = out_ids;
  // dead by now: the last layer's SiLU*up rows (the weights stream next, through L2)
  // and, when the head does not read them, the fp16 rows its down_proj left for a
  // next layer (a later layer call on this hidden then recomputes them)
  set_discard(x, g, 0, x->ws + x->r_act.off, static_cast<size_t>(b->num_tokens) * x->n * x->i_p * 2);
  if (!direct && !x->keep_intermediates) {
    set_discard(x, g, 1, x->ws + x->r_xn.off, static_cast<size_t>(b->num_tokens) * H * 2);
    x->stats_for = nullptr;
  }
  tpk::GemmPlan pl = tpk::plan_gemm(g, x->num_sms);
  if (pl.tiles_f > x->lm_tiles_max || pl.splits != 1 || (pl.swap && pl.grid > x->lm_tiles_max)) return TP_ERR_UNSUPPORTED;
  {
    // few sequences: weights stream through the M side and the argmax over all
    // ranks' vocab slices finishes inside the kernel (last CTA to arrive)
    Timed tm(x, TP_K_GEMM_LM_HEAD, s);
    e = tpk::launch_gemm(g, pl, nullptr, at<int>(x->ws, x->r_gcnt), dev_status, s);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  if (!pl.swap) {
    Timed tm(x, TP_K_ARGMAX, s);
    e = tpk::launch_argmax_reduce(g.amax_val, g.amax_idx, pl.tiles_f, B, B, out_ids, s);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return TP_OK;
}

tp_status tp_decode_advance(tp_ctx* x, const tp_batch* b, const int32_t* ids, int32_t* history, int32_t max_rows,
                            int32_t* step, int32_t* dev_status, void* stream) {
  if (!x || !ids || !history || !step || !dev_status || max_rows <= 0) return TP_ERR_INVALID_ARG;
  tp_status st = check_batch(x, b);
  if (st != TP_OK) return st;
  if (b->num_prefill != 0 || b->num_tokens != b->num_seqs) return TP_ERR_INVALID_ARG;  // decode batches only
  st = ensure_device(x);
  if (st != TP_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  {
    Timed tm(x, TP_K_DECODE_ADVANCE, s);
    e = tpk::launch_decode_advance(const_cast<int32_t*>(b->ctx_len), b->num_seqs, ids, history, max_rows, step,
                                   dev_status, s);
  }
  if (e != cudaSuccess) return cuda_fail(e);
  return TP_OK;
}

tp_status tp_hidden_written(tp_ctx* x) {
  if (!x) return TP_ERR_INVALID_ARG;
  x->stats_for = nullptr;
  return TP_OK;
}

tp_status tp_keep_intermediates(tp_ctx* x, int32_t keep) {
  if (!x) return TP_ERR_INVALID_ARG;
  x->keep_intermediates = keep != 0;
  return TP_OK;
}

tp_status tp_read_status(const int32_t* dev_status, void* stream) {
  if (!dev_status) return TP_ERR_INVALID_ARG;
  TP_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  int32_t v = 0;
  TP_CUDA(cudaMemcpy(&v, dev_status, 4, cudaMemcpyDeviceToHost));
  if (v & TP_DEVFLAG_TIMEOUT) return TP_ERR_TIMEOUT;
  if (v & TP_DEVFLAG_BAD_TOKEN) return TP_ERR_BAD_TOKEN;
  if (v & TP_DEVFLAG_SATURATED) return TP_ERR_SATURATED;
  return TP_OK;
}

tp_status tp_workspace_part(const tp_ctx* x, int32_t part, size_t* offset, size_t* bytes) {
  if (!x || !offset || !bytes || !x->ws) return TP_ERR_INVALID_ARG;
  const Region* r = nullptr;
  switch (part) {
    case TP_WS_NORMED: r = &x->r_xn; break;
    case TP_WS_QKV: r = &x->r_qkv; break;
    case TP_WS_ATTN: r = &x->r_attn; break;
    case TP_WS_ACT: r = &x->r_act; break;
    default: return TP_ERR_INVALID_ARG;
  }
  *offset = r->off;
  *bytes = r->bytes;
  return TP_OK;
}

tp_status tp_launch_count(const tp_ctx* x, int64_t* count) {
  if (!x || !count) return TP_ERR_INVALID_ARG;
  *count = x->launches;
  return TP_OK;
}

tp_status tp_profile_begin(tp_ctx* x, uint32_t kind_mask, int32_t max_launches) {
  if (!x || max_launches <= 0 || max_launches > (1 << 20)) return TP_ERR_INVALID_ARG;
  const size_t need = 2 * static_cast<size_t>(max_launches);
  while (x->prof_ev.size() < need) {
    cudaEvent_t e;
    TP_CUDA(cudaEventCreate(&e));
    x->prof_ev.push_back(e);
  }
  x->prof_kind.assign(max_launches, -1);
  x->prof_used = 0;
  x->prof_mask = kind_mask;
  x->prof_on = true;
  return TP_OK;
}

tp_status tp_profile_end(tp_ctx* x, float* total_ms, int32_t* launches) {
  if (!x || !total_ms || !launches) return TP_ERR_INVALID_ARG;
  x->prof_on = false;
  for (int k = 0; k < TP_K_COUNT; ++k) {
    total_ms[k] = 0.0f;
    launches[k] = 0;
  }
  for (int i = 0; i < x->prof_used; ++i) {
    TP_CUDA(cudaEventSynchronize(x->prof_ev[2 * i + 1]));
    float ms = 0.0f;
    TP_CUDA(cudaEventElapsedTime(&ms, x->prof_ev[2 * i], x->prof_ev[2 * i + 1]));
    const int k = x->prof_kind[i];
    if (k >= 0 && k < TP_K_COUNT) {
      total_ms[k] += ms;
      launches[k] += 1;
    }
  }
  x->prof_used = 0;
  return TP_OK;
}

tp_status tp_rank_sum_count(const tp_ctx* x, int64_t* count) {
  if (!x || !count) return TP_ERR_INVALID_ARG;
  *count = x->rank_sums;
  return TP_OK;
}

tp_status tp_debug_wait_probe(const int32_t* flag, int32_t* dev_status, int64_t limit_ns, void* stream) {
  if (!flag || !dev_status || limit_ns <= 0 || limit_ns > 10000000000LL) return TP_ERR_INVALID_ARG;
  cudaError_t e = tpk::launch_wait_probe(flag, dev_status, limit_ns, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return TP_OK;
}

tp_status tp_debug_decode_plan(int32_t max_kv_len, int32_t num_units, int32_t num_sms, int32_t head_dim,
                               int32_t group, int32_t max_splits, int32_t* units_out, int32_t* splits_out) {
  static_assert(tpk::kDecLevels == 4, "the header promises four levels");
  if (!units_out || !splits_out || max_kv_len < 1 || num_units < 1 || num_sms < 1 || max_splits < 1 ||
      (head_dim != 64 && head_dim != 128) || (group != 1 && group != 2 && group != 4 && group != 8))
    return TP_ERR_INVALID_ARG;
  const tpk::DecodeSplit d = tpk::decode_split_plan(max_kv_len, num_units, num_sms, head_dim, group, max_splits);
  for (int l = 0; l < tpk::kDecLevels; ++l) {
    units_out[l] = d.units[l];
    splits_out[l] = d.splits[l];
  }
  return TP_OK;
}

}  // extern "C"
