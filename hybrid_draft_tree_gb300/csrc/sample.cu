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
// uniforms are inputs.
//
// One CTA per request walks the accepted path.  Each node's row is read once
// (row_softmax.cuh: per-thread contiguous chunks with their online max and sum
// of exponentials); the final draw finds its chunk from the chunks' sums and
// one warp scans that chunk, so no second pass over the row is needed.  The
// top-8 and matrix update come from the scan kernels as in greedy
// verification.
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "row_softmax.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;
using namespace softmax;

constexpr int PT = 1024;  // threads per CTA: one row per CTA, so memory parallelism comes from the threads
constexpr float LOG2E = 1.4426950408889634f;

template <int DT>
__global__ __launch_bounds__(PT) void k_sample(VerifyArgs a) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  __shared__ RowStats<PT> st;
  __shared__ int32_t s_tok[MAX_S], s_par[MAX_S], s_rej[MAX_S];
  __shared__ float s_x[MAX_S];         // logits of the node's children, by slot
  __shared__ float s_u[MAX_S];         // the request's acceptance uniforms, by slot
  __shared__ float s_cw[PT];           // chunk weights of the final draw
  __shared__ int s_acc, s_nrej, s_chunk, s_pick;
  __shared__ float s_target, s_before;
  const int b = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5, S = a.S, V = a.g.V;
  const float k2 = a.inv_temp * LOG2E;
  if (t < S) {
    s_tok[t] = a.tree_tok[(int64_t)b * S + t];
    s_par[t] = a.tree_parent[(int64_t)b * S + t];
    s_u[t] = a.u_accept[(int64_t)b * S + t];
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
    // the children's logits, fetched beside the row pass
    if (t < S) {
      const int32_t tk = s_tok[t];
      s_x[t] = (t > node && s_par[t] == node && tk >= 0 && tk < V) ? load_scalar<DT>(rowp, tk) : 0.f;
    }
    row_stats<DT, PT>(rowp, V, a.g.vec != 0, k2, st);
    const float M = st.M, W = st.W;
    if (t == 0) {
      float rem = 1.f;
      int acc = -1, nrej = 0;
      for (int j = node + 1; j < S && acc < 0; ++j) {
        const int32_t tk = s_tok[j];
        if (s_par[j] != node || tk < 0 || tk >= V) continue;
        bool seen = false;
        for (int q = 0; q < nrej; ++q) seen |= s_rej[q] == tk;
        if (seen) continue;  // a repeated token: its mass is gone
        const float pc = exp2f((s_x[j] - M) * k2) / W;
        if (s_u[j] * rem < pc) acc = j;
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
      continue;
    }
    // every child rejected (or a leaf): draw from the unrejected tokens.
    // 1. chunk weights relative to M, minus the rejected tokens in the chunk
    const int nrej = s_nrej;
    const int ch = st.ch;
    const int c0 = min(t * ch, V), c1 = min(c0 + ch, V);
    float cw = st.m[t] == -INFINITY ? 0.f : st.s[t] * exp2f((st.m[t] - M) * k2);
    for (int q = 0; q < nrej; ++q) {
      const int32_t r = s_rej[q];
      if (r >= c0 && r < c1) cw -= exp2f((load_scalar<DT>(rowp, r) - M) * k2);
    }
    cw = fmaxf(cw, 0.f);
    s_cw[t] = cw;
    // 2. the chunk holding the target (warp 0): lane l sums chunks 8l..8l+7 in
    //    order, a warp scan orders the lanes; a fixed summation order
    __syncthreads();
    if (warp == 0) {
      constexpr int CPL = PT / 32;
      float w8[CPL];
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) { w8[i] = s_cw[lane * CPL + i]; lsum += w8[i]; }
      float incl = lsum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(FULL, incl, o);
        if (lane >= o) incl += y;
      }
      const float total = __shfl_sync(FULL, incl, 31);
      const float target = a.u_resid[b] * total;
      float run = incl - lsum;  // weight before this lane's chunks
      int c = -1, last = -1;
      float cb = 0.f, last_before = 0.f;
#pragma unroll
      for (int i = 0; i < CPL; ++i) {
        if (w8[i] > 0.f) {
          if (c < 0 && run + w8[i] > target) { c = lane * CPL + i; cb = run; }
          last = lane * CPL + i;
          last_before = run;
        }
        run += w8[i];
      }
      const unsigned hit = __ballot_sync(FULL, c >= 0);
      const unsigned any = __ballot_sync(FULL, last >= 0);
      const int src = hit ? __ffs(hit) - 1 : (any ? 31 - __clz(any) : 0);  // else rounding: the last chunk with weight
      const int cc = __shfl_sync(FULL, hit ? c : last, src);
      const float bb = __shfl_sync(FULL, hit ? cb : last_before, src);
      if (lane == 0) {
        s_chunk = (hit | any) ? cc : -1;
        s_before = bb;
        s_target = target;
      }
    }
    __syncthreads();
    // 3. warp 0 scans the chunk: per-lane sub-ranges, a warp prefix, then the
    //    lane holding the target walks its elements
    if (warp == 0) {
      const int c = s_chunk;
      int pick = -1;
      if (c >= 0) {
        const int lo = min(c * ch, V), hi = min(lo + ch, V);
        const float bef = s_before;  // weight of the chunks before c
        const int sub = (hi - lo + 31) / 32;
        const int l0 = min(lo + lane * sub, hi), l1 = min(l0 + sub, hi);
        float ls = 0.f;
        int last = -1;
        for (int v = l0; v < l1; ++v) {
          bool rej = false;
          for (int q = 0; q < nrej; ++q) rej |= s_rej[q] == v;
          if (rej) continue;
          const float wv = exp2f((load_scalar<DT>(rowp, v) - M) * k2);
          if (wv > 0.f) { ls += wv; last = v; }
        }
        float li = ls;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(FULL, li, o);
          if (lane >= o) li += y;
        }
        const float tgt = s_target;
        const float lb = bef + li - ls;  // weight before this lane's sub-range
        const bool mine = ls > 0.f && lb <= tgt && tgt < lb + ls;
        const unsigned who = __ballot_sync(FULL, mine);
        int lpick = -1;
        if (who != 0 && lane == __ffs(who) - 1) {
          float run = lb;
          for (int v = l0; v < l1 && lpick < 0; ++v) {
            bool rej = false;
            for (int q = 0; q < nrej; ++q) rej |= s_rej[q] == v;
            if (rej) continue;
            const float wv = exp2f((load_scalar<DT>(rowp, v) - M) * k2);
            if (wv <= 0.f) continue;
            run += wv;
            if (run > tgt) lpick = v;
          }
          if (lpick < 0) lpick = last;
        }
        pick = __shfl_sync(FULL, lpick, who != 0 ? __ffs(who) - 1 : 0);
        if (who == 0) {  // rounding: the chunk's last element with weight
          const unsigned has = __ballot_sync(FULL, last >= 0);
          pick = has ? __shfl_sync(FULL, last, 31 - __clz(has)) : -1;
        }
      }
      if (lane == 0) s_pick = pick;
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
