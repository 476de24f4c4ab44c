// Block-wide softmax statistics of one logits row, for the kernels that need
// target probabilities (stochastic verification, the coverage diagnostic).
//
// Thread t of the CTA owns the contiguous chunk [t*ch, min((t+1)*ch, V)) of
// the row (ch a multiple of the vector width when the row is 16-byte aligned,
// so the chunk is read with 16-byte loads) and keeps an online (max, sum of
// exp2((x - max) * k2)) over it; k2 = log2(e) / temperature.  The chunks'
// pairs stay in shared memory, so an inverse-CDF draw over the row can locate
// its chunk without another pass.  All threads of the CTA must call.
#pragma once
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "scan_common.cuh"

namespace graft {
namespace softmax {
using namespace scan;

template <int NT>
struct RowStats {
  float m[NT];  // chunk maxima
  float s[NT];  // chunk sums of exp2((x - m[t]) * k2)
  float M, W;   // row maximum and sum of exp2((x - M) * k2)
  int ch;       // elements per chunk
};

// (m, s) <- online update with element x.
__device__ __forceinline__ void online_add(float& m, float& s, float x, float k2) {
  if (x > m) {
    s = s * exp2f((m - x) * k2) + 1.f;
    m = x;
  } else if (x != -INFINITY) {
    s += exp2f((x - m) * k2);
  }
}

// Chunk size: V / NT rounded up to a multiple of `epl` (the elements of one
// 16-byte load on the vector path, else 1).
template <int NT>
__device__ __forceinline__ int chunk_size(int V, int epl) {
  int ch = (V + NT - 1) / NT;
  return (ch + epl - 1) / epl * epl;
}

template <int DT, int NT>
__device__ void row_stats(const char* rowp, int V, bool vec, float k2, RowStats<NT>& st) {
  const int t = threadIdx.x;
  constexpr int EPL = Vec16<DT>::EPL;
  const int ch = chunk_size<NT>(V, vec ? EPL : 1);
  const int v0 = min(t * ch, V), v1 = min(v0 + ch, V);
  float m = -INFINITY, s = 0.f;
  if (vec) {
    const uint4* p = reinterpret_cast<const uint4*>(rowp);
    const int full = v0 + (v1 - v0) / EPL * EPL;  // whole vectors of the chunk
#pragma unroll 4
    for (int v = v0; v < full; v += EPL) {
      Vec16<DT> x;
      x.r = p[v / EPL];
      const float vm = x.vmax();
      if (vm > m) { s *= exp2f((m - vm) * k2); m = vm; }  // one rescale per vector
      if (m != -INFINITY) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) s += exp2f((x.elem(e) - m) * k2);
      }
    }
    for (int v = full; v < v1; ++v) online_add(m, s, load_scalar<DT>(rowp, v), k2);
  } else {
    for (int v = v0; v < v1; ++v) online_add(m, s, load_scalar<DT>(rowp, v), k2);
  }
  st.m[t] = m;
  st.s[t] = s;
  __syncthreads();
  if (t < 32) {
    float M = -INFINITY;
    for (int i = t; i < NT; i += 32) M = fmaxf(M, st.m[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
    float W = 0.f;
    if (M != -INFINITY)
      for (int i = t; i < NT; i += 32) W += st.m[i] == -INFINITY ? 0.f : st.s[i] * exp2f((st.m[i] - M) * k2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) W += __shfl_xor_sync(FULL, W, o);
    if (t == 0) { st.M = M; st.W = W; st.ch = ch; }
  }
  __syncthreads();
}

}  // namespace softmax
}  // namespace graft
