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
// path: one CTA per request streams each boundary parent's row once
// (row_softmax.cuh).
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "row_softmax.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;
using namespace softmax;

constexpr int CT = 1024;  // threads per CTA: one row per CTA, so memory parallelism comes from the threads

constexpr float LOG2E = 1.4426950408889634f;

template <int DT>
__global__ __launch_bounds__(CT) void k_coverage(VerifyArgs a, const int32_t* info, float* gain) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  __shared__ RowStats<CT> st;
  __shared__ int32_t s_tok[MAX_S], s_par[MAX_S];
  __shared__ float s_x[MAX_S];  // a boundary candidate's logit in its parent's row, by slot
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
    if (t >= r0 && t < r1 && s_par[t] == p && s_tok[t] >= 0 && s_tok[t] < a.g.V)
      s_x[t] = load_scalar<DT>(rowp, s_tok[t]);  // fetched beside the row pass
    row_stats<DT, CT>(rowp, a.g.V, a.g.vec != 0, LOG2E, st);
    const float M = st.M, Z = st.W;
    if (t == 0 && Z > 0.f) {
      for (int j = r0; j < r1; ++j) {
        const int32_t tk = s_tok[j];
        if (s_par[j] != p || tk < 0 || tk >= a.g.V) continue;
        bool dup = false;  // a kept draft child of p with the same token is not new
        for (int q = 1; q < r0; ++q) dup |= s_par[q] == p && s_tok[q] == tk;
        if (!dup) total += exp2f((s_x[j] - M) * LOG2E) / Z;
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
