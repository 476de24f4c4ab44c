// graft_coverage's kernel: the coverage gain of the retrieval graft
// (popular-science article on arXiv 2605.20104, section 三).
//
// At the prune boundary the retrieved candidates add target probability mass
// that the pruned tree does not cover.  For each request (checkpoint or tail
// mode, where the retrieved slots follow the kept draft slots), every retrieved
// slot whose parent is a kept slot (the root, or the last kept block token) is
// a boundary candidate; its token is new unless a kept draft child of the same
// parent carries it.  The gain is the sum, over the new tokens, of their
// softmax probability in the parent's logits row.  A diagnostic off the hot
// path: one CTA per request streams each boundary parent's row once.
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;

constexpr int CT = 256;

// CTA-wide (max, sum of exp(x - max)) of one logits row.
template <int DT>
__device__ void row_lse(const char* rowp, int V, float* s_m, float* s_s, float& m_out, float& s_out) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float m = -INFINITY, sum = 0.f;
  for (int v = t; v < V; v += CT) {
    const float x = load_scalar<DT>(rowp, v);
    if (x > m) {
      sum = sum * expf(m - x) + 1.f;
      m = x;
    } else if (x != -INFINITY) {
      sum += expf(x - m);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(FULL, m, o), s2 = __shfl_xor_sync(FULL, sum, o);
    const float mm = fmaxf(m, m2);
    sum = (mm == -INFINITY) ? 0.f : sum * expf(m - mm) + s2 * expf(m2 - mm);
    m = mm;
  }
  if (lane == 0) { s_m[warp] = m; s_s[warp] = sum; }
  __syncthreads();
  if (t == 0) {
    float M = -INFINITY, Ssum = 0.f;
    for (int w = 0; w < CT / 32; ++w) {
      const float mm = fmaxf(M, s_m[w]);
      Ssum = (mm == -INFINITY) ? 0.f : Ssum * expf(M - mm) + s_s[w] * expf(s_m[w] - mm);
      M = mm;
    }
    s_m[0] = M;
    s_s[0] = Ssum;
  }
  __syncthreads();
  m_out = s_m[0];
  s_out = s_s[0];
  __syncthreads();
}

template <int DT>
__global__ __launch_bounds__(CT) void k_coverage(VerifyArgs a, const int32_t* info, float* gain) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  __shared__ float s_m[CT / 32], s_s[CT / 32];
  __shared__ int32_t s_tok[MAX_S], s_par[MAX_S];
  const int b = blockIdx.x, t = threadIdx.x, S = a.S;
  const int n_draft = info[(int64_t)b * 4 + 1], n_retr = info[(int64_t)b * 4 + 2];
  const int r0 = min(max(1 + n_draft, 1), S), r1 = min(r0 + max(n_retr, 0), S);
  if (t < S) {
    s_tok[t] = a.tree_tok[(int64_t)b * S + t];
    s_par[t] = a.tree_parent[(int64_t)b * S + t];
  }
  __syncthreads();
  float total = 0.f;  // thread 0's running sum
  // boundary parents in slot order (a kept slot with a retrieved child)
  for (int p = 0; p < r0 && p < S; ++p) {
    bool has = false;
    for (int j = r0; j < r1; ++j) has |= s_par[j] == p;
    if (!has || s_tok[p] < 0 || s_tok[p] >= a.g.V) continue;  // (uniform: shared values)
    const char* rowp = reinterpret_cast<const char*>(a.logits) + ((size_t)b * S + p) * (size_t)a.g.stride * ES;
    float M, Z;
    row_lse<DT>(rowp, a.g.V, s_m, s_s, M, Z);
    if (t == 0 && Z > 0.f) {
      for (int j = r0; j < r1; ++j) {
        const int32_t tk = s_tok[j];
        if (s_par[j] != p || tk < 0 || tk >= a.g.V) continue;
        bool dup = false;  // a kept draft child of p with the same token is not new
        for (int q = 1; q < r0; ++q) dup |= s_par[q] == p && s_tok[q] == tk;
        if (!dup) total += expf(load_scalar<DT>(rowp, tk) - M) / Z;
      }
    }
  }
  if (t == 0) gain[b] = total;
}

template <int DT>
cudaError_t coverage_impl(const VerifyArgs& a, const int32_t* info, float* gain, cudaStream_t s) {
  k_coverage<DT><<<a.batch, CT, 0, s>>>(a, info, gain);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_coverage(const VerifyArgs& a, const int32_t* info, float* gain, int dtype, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? coverage_impl<GRAFT_BF16>(a, info, gain, s) : coverage_impl<GRAFT_F32>(a, info, gain, s);
}

}  // namespace graft
