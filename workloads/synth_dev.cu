// Device twin of synth_host.c: the synthetic target's row filler, the per-node
// row parameters of a flattened tree, and the closed-loop request advance.
// Input generation only (no Graft arithmetic).  Every operation matches the
// host definition bit for bit: SplitMix64 counter hashing, the exact
// Irwin-Hall(12) normal, one IEEE add for the planted bias, and
// round-to-nearest-even to bf16.  Built with -fmad=false.
#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t SALT_NOISE = 0x6E6F697365ull;
constexpr uint64_t SALT_HIT = 0x486974ull;
constexpr uint64_t SALT_BIGRAM = 0x4269677261ull;
constexpr uint64_t SALT_TRI = 0x547269ull;
constexpr uint64_t SALT_REQ = 0x526571ull;
constexpr uint64_t CTX_MUL = 0xD1B54A32D192ED03ull;

__device__ __forceinline__ uint64_t sm64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}
__device__ __forceinline__ uint64_t h2(uint64_t a, uint64_t b) { return sm64(sm64(a) ^ b); }
__device__ __forceinline__ uint64_t h3(uint64_t a, uint64_t b, uint64_t c) { return sm64(h2(a, b) ^ c); }
__device__ __forceinline__ uint64_t ctx_push(uint64_t ctx, int32_t t) {
  return sm64(ctx ^ (CTX_MUL * ((uint64_t)(uint32_t)t + 1ull)));
}

struct Target {
  int32_t V, kind, hit_all;
  uint32_t hit_num;
  float bias;
  uint64_t seed;
  const int32_t* table;
};

__device__ int32_t succ_of(const Target& tg, int32_t b, int32_t prev, int32_t t) {
  uint64_t V = (uint64_t)tg.V;
  switch (tg.kind) {
    case 1: return (int32_t)(h3(tg.seed ^ SALT_TRI, (uint64_t)(uint32_t)prev, (uint64_t)(uint32_t)t) % V);
    case 2: return (int32_t)(h3(tg.seed ^ SALT_REQ, (uint64_t)(uint32_t)b, (uint64_t)(uint32_t)t) % V);
    case 3:
      if (tg.table && tg.table[t] >= 0) return tg.table[t];
      // fall through
    default: return (int32_t)(h2(tg.seed ^ SALT_BIGRAM, (uint64_t)(uint32_t)t) % V);
  }
}
__device__ bool hit_of(const Target& tg, uint64_t ctx) {
  if (tg.hit_all) return true;
  return (uint32_t)(sm64(ctx ^ SALT_HIT) >> 32) < tg.hit_num;
}

__device__ __forceinline__ float noise_z(uint64_t rowkey, int64_t v) {
  uint64_t c = rowkey + 3ull * (uint64_t)v;
  uint32_t s = 0;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    uint64_t h = sm64(c + (uint64_t)j);
    s += (uint32_t)(h & 0xFFFF) + (uint32_t)((h >> 16) & 0xFFFF) + (uint32_t)((h >> 32) & 0xFFFF) +
         (uint32_t)(h >> 48);
  }
  int32_t num = 2 * (int32_t)s - 12 * 65535;
  return __fmul_rn(__int2float_rn(num), 1.0f / 131072.0f);
}
__device__ __forceinline__ uint16_t bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

constexpr int FILL_T = 256, FILL_E = 8;

__global__ void k_fill(const uint64_t* __restrict__ rk, const int32_t* __restrict__ pl,
                       const float* __restrict__ bi, int64_t n, int32_t V, int32_t dtype, void* out,
                       int64_t stride) {
  for (int64_t r = blockIdx.y; r < n; r += gridDim.y) {
    const uint64_t key = rk[r];
    const int32_t p = pl[r];
    const float bias = bi[r];
    for (int64_t base = (int64_t)blockIdx.x * FILL_T * FILL_E; base < V; base += (int64_t)gridDim.x * FILL_T * FILL_E) {
#pragma unroll
      for (int k = 0; k < FILL_E; ++k) {
        int64_t v = base + threadIdx.x + (int64_t)k * FILL_T;
        if (v >= V) break;
        float x;
        if (p == -2) {
          x = __uint_as_float(0x7FC00000u);
        } else {
          x = noise_z(key, v);
          if (v == p) x = __fadd_rn(x, bias);
        }
        if (dtype == 0)
          ((float*)out)[r * stride + v] = x;
        else
          ((uint16_t*)out)[r * stride + v] = (p == -2) ? (uint16_t)0x7FC0 : bf16_rne(x);
      }
    }
  }
}

__global__ void k_tree_rowparams(Target tg, int32_t B, int32_t S, const int32_t* tok, const int8_t* parent,
                                 const uint64_t* root_ctx, const int32_t* root_prev, uint64_t* rowkey,
                                 int32_t* planted, float* bias) {
  int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  uint64_t ctx[64];
  for (int32_t i = 0; i < S; ++i) {
    int64_t k = (int64_t)b * S + i;
    int32_t t = tok[k];
    if (t < 0) { rowkey[k] = 0; planted[k] = -2; bias[k] = 0.f; continue; }
    int32_t prev;
    if (i == 0) { ctx[i] = root_ctx[b]; prev = root_prev[b]; }
    else {
      int p = parent[k];
      if (p < 0 || p >= i) { rowkey[k] = 0; planted[k] = -2; bias[k] = 0.f; continue; }  // malformed: pad
      ctx[i] = ctx_push(ctx[p], t);
      prev = tok[(int64_t)b * S + p];
    }
    rowkey[k] = sm64(ctx[i] ^ SALT_NOISE);
    planted[k] = hit_of(tg, ctx[i]) ? succ_of(tg, b, prev, t) : -1;
    bias[k] = tg.bias;
  }
}

__global__ void k_advance(int32_t B, int32_t S, const int32_t* out_tokens, const int32_t* accept_len,
                          int32_t* root, int32_t* prev, uint64_t* ctx) {
  int32_t b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  int32_t cnt = accept_len[b] + 1;
  int32_t r = root[b], p = prev[b];
  uint64_t c = ctx[b];
  for (int32_t j = 0; j < cnt && j < S; ++j) {
    int32_t t = out_tokens[(int64_t)b * S + j];
    p = r; r = t; c = ctx_push(c, t);
  }
  root[b] = r; prev[b] = p; ctx[b] = c;
}

}  // namespace

extern "C" {

int synd_fill_rows(const uint64_t* rk, const int32_t* pl, const float* bi, int64_t n, int32_t V, int32_t dtype,
                   void* out, int64_t stride, void* stream) {
  if (n <= 0) return 0;
  int gx = (int)((V + FILL_T * FILL_E - 1) / (FILL_T * FILL_E));
  if (gx > 1024) gx = 1024;
  int gy = n < 65535 ? (int)n : 65535;
  k_fill<<<dim3(gx, gy), FILL_T, 0, (cudaStream_t)stream>>>(rk, pl, bi, n, V, dtype, out, stride);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int synd_tree_rowparams(int32_t V, int32_t kind, int32_t hit_all, uint32_t hit_num, float bias, uint64_t seed,
                        const int32_t* table, int32_t B, int32_t S, const int32_t* tok, const int8_t* parent,
                        const uint64_t* root_ctx, const int32_t* root_prev, uint64_t* rowkey, int32_t* planted,
                        float* biasv, void* stream) {
  if (S > 64 || B <= 0) return -1;
  Target tg{V, kind, hit_all, hit_num, bias, seed, table};
  k_tree_rowparams<<<(B + 63) / 64, 64, 0, (cudaStream_t)stream>>>(tg, B, S, tok, parent, root_ctx, root_prev,
                                                                   rowkey, planted, biasv);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

int synd_advance(int32_t B, int32_t S, const int32_t* out_tokens, const int32_t* accept_len, int32_t* root,
                 int32_t* prev, uint64_t* ctx, void* stream) {
  if (B <= 0) return -1;
  k_advance<<<(B + 63) / 64, 64, 0, (cudaStream_t)stream>>>(B, S, out_tokens, accept_len, root, prev, ctx);
  return cudaGetLastError() == cudaSuccess ? 0 : -3;
}

}  // extern "C"
