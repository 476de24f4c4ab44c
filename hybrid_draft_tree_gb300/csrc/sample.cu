// graft_verify_update_sample's acceptance kernel: lossless stochastic tree
// verification (popular-science article on arXiv 2605.20104, section 二 third
// gear: the output distribution equals sampling from the target model).
//
// The candidates are deterministic (draft top-k and retrieved tokens), so at a
// node n with target distribution p = softmax(row_n / T) the children are
// tested one by one in slot order: child c is accepted when
// u[c] * rem < p(tok_c), rem being the mass not yet rejected at n; a rejected
// token's mass leaves rem (a repeated token has none left).  Acceptance
// descends into c; when every child is rejected (or n is a leaf) the last
// token is drawn from p restricted to the unrejected tokens by inverse CDF
// with u_res.  Every emitted token is then distributed exactly as p.  The
// uniforms are inputs.  One CTA per request walks the accepted path, reading
// each node's row once for its normaliser and the last one again for the
// draw; the top-8 and matrix update come from the scan kernels as in greedy
// verification.
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;

constexpr int PT = 256;
constexpr int PW = PT / 32;

// CTA-wide max and sum of exp((x - max) * inv_t) over one row.
template <int DT>
__device__ void row_norm(const char* rowp, int V, float inv_t, float* s_a, float* s_b, float& m_out, float& w_out) {
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  float m = -INFINITY;
  for (int v = t; v < V; v += PT) m = fmaxf(m, load_scalar<DT>(rowp, v));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
  if (lane == 0) s_a[warp] = m;
  __syncthreads();
  m = s_a[0];
  for (int w = 1; w < PW; ++w) m = fmaxf(m, s_a[w]);
  float sum = 0.f;
  if (m > -INFINITY)
    for (int v = t; v < V; v += PT) sum += expf((load_scalar<DT>(rowp, v) - m) * inv_t);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
  if (lane == 0) s_b[warp] = sum;
  __syncthreads();
  float total = 0.f;
  for (int w = 0; w < PW; ++w) total += s_b[w];
  m_out = m;
  w_out = total;
  __syncthreads();
}

template <int DT>
__global__ __launch_bounds__(PT) void k_sample(VerifyArgs a) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  __shared__ int32_t s_tok[MAX_S], s_par[MAX_S], s_rej[MAX_S];
  __shared__ float s_a[PW], s_b[PW], s_chunk[PT];
  __shared__ int s_acc, s_nrej, s_pick;
  const int b = blockIdx.x, t = threadIdx.x, S = a.S, V = a.g.V;
  const float inv_t = a.inv_temp;
  if (t < S) {
    s_tok[t] = a.tree_tok[(int64_t)b * S + t];
    s_par[t] = a.tree_parent[(int64_t)b * S + t];
  }
  __syncthreads();
  int32_t* out = a.out_tokens + (int64_t)b * S;
  if (s_tok[0] < 0 || s_tok[0] >= V) {  // no valid root: nothing accepted, nothing emitted
    if (t < S) out[t] = -1;
    if (t == 0) a.accept_len[b] = 0;
    return;
  }
  int node = 0, len = 0;
  for (int depth = 0; depth < S; ++depth) {  // the path has fewer than S nodes
    const char* rowp = reinterpret_cast<const char*>(a.logits) + ((size_t)b * S + node) * (size_t)a.g.stride * ES;
    float M, W;
    row_norm<DT>(rowp, V, inv_t, s_a, s_b, M, W);
    if (t == 0) {
      float rem = 1.f;
      int acc = -1, nrej = 0;
      for (int j = node + 1; j < S && acc < 0; ++j) {
        const int32_t tk = s_tok[j];
        if (s_par[j] != node || tk < 0 || tk >= V) continue;
        bool seen = false;
        for (int q = 0; q < nrej; ++q) seen |= s_rej[q] == tk;
        if (seen) continue;  // a repeated token: its mass is gone
        const float pc = expf((load_scalar<DT>(rowp, tk) - M) * inv_t) / W;
        if (a.u_accept[(int64_t)b * S + j] * rem < pc) acc = j;
        else { rem -= pc; s_rej[nrej++] = tk; }
      }
      s_acc = acc;
      s_nrej = nrej;
    }
    __syncthreads();
    const int acc = s_acc;
    if (acc >= 0) {
      if (t == 0) out[len] = s_tok[acc];
      ++len;
      node = acc;
      __syncthreads();
      continue;
    }
    // every child rejected (or a leaf): draw from the unrejected tokens,
    // weights exp((x - M) / T), by inverse CDF over contiguous chunks
    const int nrej = s_nrej;
    const int ch = (V + PT - 1) / PT;
    const int v0 = min(t * ch, V), v1 = min(v0 + ch, V);
    float local = 0.f;
    for (int v = v0; v < v1; ++v) local += expf((load_scalar<DT>(rowp, v) - M) * inv_t);
    for (int q = 0; q < nrej; ++q) {
      const int32_t r = s_rej[q];
      if (r >= v0 && r < v1) local -= expf((load_scalar<DT>(rowp, r) - M) * inv_t);
    }
    s_chunk[t] = fmaxf(local, 0.f);
    if (t == 0) s_pick = -1;
    __syncthreads();
    if (t == 0) {
      // exclusive prefix over the chunks (sequential: 256 values), then the chunk holding the target
      float total = 0.f;
      for (int i = 0; i < PT; ++i) total += s_chunk[i];
      const float target = a.u_resid[b] * total;
      float acc_sum = 0.f;
      int pick_chunk = -1;
      for (int i = 0; i < PT; ++i) {
        if (s_chunk[i] > 0.f && acc_sum + s_chunk[i] > target) { pick_chunk = i; break; }
        acc_sum += s_chunk[i];
      }
      if (pick_chunk < 0)  // rounding put the target at the very end: the last chunk with mass
        for (int i = PT - 1; i >= 0 && pick_chunk < 0; --i)
          if (s_chunk[i] > 0.f) pick_chunk = i;
      int pick = -1;
      if (pick_chunk >= 0) {
        const int c0 = min(pick_chunk * ch, V), c1 = min(c0 + ch, V);
        float run = acc_sum;
        int last = -1;
        for (int v = c0; v < c1 && pick < 0; ++v) {
          bool rej = false;
          for (int q = 0; q < nrej; ++q) rej |= s_rej[q] == v;
          if (rej) continue;
          const float wv = expf((load_scalar<DT>(rowp, v) - M) * inv_t);
          if (wv <= 0.f) continue;
          last = v;
          run += wv;
          if (run > target) pick = v;
        }
        if (pick < 0) pick = last;
      }
      s_pick = pick;
    }
    __syncthreads();
    if (t == 0) {
      out[len] = s_pick;
      a.accept_len[b] = len;
    }
    for (int j = len + 1 + t; j < S; j += PT) out[j] = -1;
    return;
  }
}

template <int DT>
cudaError_t sample_impl(const VerifyArgs& a, cudaStream_t s) {
  k_sample<DT><<<a.batch, PT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sample(const VerifyArgs& a, int dtype, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? sample_impl<GRAFT_BF16>(a, s) : sample_impl<GRAFT_F32>(a, s);
}

}  // namespace graft
