// Device half of the seeded generator in synth/__init__.py (same definition,
// bit for bit): SplitMix64 counter draws, 4-lane Irwin-Hall normal samples
// scaled in fp32 and rounded to bf16, uniform token ids.  Used to fill large
// device buffers (weights, KV caches) without a host round trip.  Contains no
// arithmetic of the transformer.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__host__ __device__ __forceinline__ uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

__device__ __forceinline__ __nv_bfloat16 normal_bf16(uint64_t key, uint64_t idx, float scale, float sigma,
                                                     int has_mean, float mean) {
  const uint64_t u = mix64(key + (idx + 1) * kGolden);
  const int64_t s = static_cast<int64_t>((u & 0xFFFF) + ((u >> 16) & 0xFFFF) + ((u >> 32) & 0xFFFF) + (u >> 48));
  const float x = __fmul_rn(static_cast<float>(s - 131070), scale);
  float y = __fmul_rn(x, sigma);
  if (has_mean) y = __fadd_rn(y, mean);
  return __float2bfloat16_rn(y);
}

__global__ void fill_normal_kernel(__nv_bfloat16* dst, uint64_t count, uint64_t key, uint64_t start, float scale,
                                   float sigma, int has_mean, float mean) {
  for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < count;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x)
    dst[i] = normal_bf16(key, start + i, scale, sigma, has_mean, mean);
}

struct HeadMap {
  int g[256];
};

// cache [n][2][max_seqs][nkv_l][cap][hd]; element (r, kv, slot, gl, pos, d) for slot < num_slots,
// pos < fill_len takes draw ((slot*2 + kv)*nkv + head[r*nkv_l + gl]) * pos_stride + pos) * hd + d.
__global__ void fill_kv_kernel(__nv_bfloat16* cache, int n, int max_seqs, int nkv_l, int cap, int hd, HeadMap map,
                               int nkv, uint64_t key, int num_slots, int fill_len, uint64_t pos_stride,
                               float scale) {
  const uint64_t per_rank_kv = static_cast<uint64_t>(num_slots) * nkv_l * fill_len * hd;
  const uint64_t total = static_cast<uint64_t>(n) * 2 * per_rank_kv;
  for (uint64_t e = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    uint64_t rem = e;
    const int d = static_cast<int>(rem % hd); rem /= hd;
    const int pos = static_cast<int>(rem % fill_len); rem /= fill_len;
    const int gl = static_cast<int>(rem % nkv_l); rem /= nkv_l;
    const int slot = static_cast<int>(rem % num_slots); rem /= num_slots;
    const int kv = static_cast<int>(rem % 2); rem /= 2;
    const int r = static_cast<int>(rem);
    const int g = map.g[r * nkv_l + gl];
    const uint64_t idx = ((static_cast<uint64_t>(slot) * 2 + kv) * nkv + g) * pos_stride * hd +
                         static_cast<uint64_t>(pos) * hd + d;
    const size_t dst = ((((static_cast<size_t>(r) * 2 + kv) * max_seqs + slot) * nkv_l + gl) * cap + pos) * hd + d;
    cache[dst] = normal_bf16(key, idx, scale, 1.0f, 0, 0.0f);
  }
}

__global__ void fill_ids_kernel(int32_t* dst, uint64_t count, uint64_t key, uint64_t start, uint64_t vocab) {
  for (uint64_t i = blockIdx.x * static_cast<uint64_t>(blockDim.x) + threadIdx.x; i < count;
       i += static_cast<uint64_t>(gridDim.x) * blockDim.x) {
    const uint64_t u = mix64(key + (start + i + 1) * kGolden);
    dst[i] = static_cast<int32_t>(((u >> 32) * vocab) >> 32);
  }
}

uint64_t stream_key(uint64_t seed, uint64_t stream) { return mix64(seed * kGolden + stream); }
float ih_scale() { return static_cast<float>(1.7320508075688772935 / 65536.0); }

}  // namespace

extern "C" {

int synth_fill_normal_bf16(void* dst, uint64_t count, uint64_t seed, uint64_t stream, uint64_t start, float sigma,
                           int has_mean, float mean, void* cuda_stream) {
  if (!dst) return 1;
  if (count == 0) return 0;
  const uint64_t blocks = (count + 255) / 256;
  const unsigned grid = static_cast<unsigned>(blocks < 65536 ? blocks : 65536);
  fill_normal_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      static_cast<__nv_bfloat16*>(dst), count, stream_key(seed, stream), start, ih_scale(), sigma, has_mean, mean);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

int synth_fill_kv(void* cache, int n, int max_seqs, int nkv_l, int cap, int hd, const int32_t* head_map, int nkv,
                  uint64_t seed, uint64_t layer, int num_slots, int fill_len, uint64_t pos_stride,
                  void* cuda_stream) {
  if (!cache || !head_map || n * nkv_l > 256 || num_slots > max_seqs || fill_len > cap) return 1;
  if (num_slots <= 0 || fill_len <= 0) return 0;
  HeadMap m{};
  for (int i = 0; i < n * nkv_l; ++i) m.g[i] = head_map[i];
  fill_kv_kernel<<<65536, 256, 0, static_cast<cudaStream_t>(cuda_stream)>>>(
      static_cast<__nv_bfloat16*>(cache), n, max_seqs, nkv_l, cap, hd, m, nkv, stream_key(seed, layer), num_slots,
      fill_len, pos_stride, ih_scale());
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

int synth_fill_token_ids(int32_t* dst, uint64_t count, uint64_t vocab, uint64_t seed, uint64_t stream,
                         uint64_t start, void* cuda_stream) {
  if (!dst) return 1;
  if (count == 0) return 0;
  const uint64_t blocks = (count + 255) / 256;
  fill_ids_kernel<<<static_cast<unsigned>(blocks < 65536 ? blocks : 65536), 256, 0,
                    static_cast<cudaStream_t>(cuda_stream)>>>(dst, count, stream_key(seed, stream), start, vocab);
  return cudaGetLastError() == cudaSuccess ? 0 : 2;
}

}  // extern "C"
