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
// path: one thread-block cluster of CL CTAs per request streams each boundary
// parent's row once, split over the cluster's SMs (row_softmax.cuh; aligned
// rows whose eighth fits STAGE_MAX arrive by bulk copies into shared memory).
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "row_softmax.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;
using namespace softmax;

constexpr int CT = 256;  // threads per CTA (CL CTAs per request)
constexpr int STAGE_MAX = 160 * 1024;  // shared memory for a CTA's eighth of a row (bulk staging)

constexpr float LOG2E = 1.4426950408889634f;

// BULK: each row pass stages the CTA's eighth of the row by bulk copies;
// otherwise the threads load their chunks.
template <int DT, bool BULK>
__global__ __launch_bounds__(CT, 4) void k_coverage(VerifyArgs a, const int32_t* info, float* gain) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  extern __shared__ __align__(16) char s_stage[];  // BULK: this CTA's range of the current row
  __shared__ unsigned long long s_bar;
  __shared__ ClusterRow<CT> st;
  __shared__ int32_t s_tok[MAX_S], s_par[MAX_S];
  __shared__ float s_x[MAX_S];  // a boundary candidate's logit in its parent's row, by slot
  const cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / CL, t = threadIdx.x, S = a.S, warp = t >> 5, lane = t & 31;
  const int n_draft = info[(int64_t)b * 4 + 1], n_retr = info[(int64_t)b * 4 + 2];
  const int r0 = min(max(1 + n_draft, 1), S), r1 = min(r0 + max(n_retr, 0), S);
  if (t < S) {
    s_tok[t] = a.tree_tok[(int64_t)b * S + t];
    s_par[t] = a.tree_parent[(int64_t)b * S + t];
  }
  if (BULK && t == 0) {
    bulk::mbar_init(&s_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster_started_arrive();
  __syncthreads();
  // boundary parents (a kept slot with a retrieved child), in slot order
  __shared__ unsigned long long s_bmask;
  if (t == 0) s_bmask = 0ull;
  __syncthreads();
  if (t >= r0 && t < r1) {
    const int p = s_par[t];
    if (p >= 0 && p < r0) atomicOr(&s_bmask, 1ull << p);
  }
  __syncthreads();
  uint64_t bmask = s_bmask;
  float total = 0.f;  // lane 0 of warp 0's running sum (used in CTA 0)
  int pass = 0;
  while (bmask != 0ull) {  // (uniform: the same values in every CTA)
    const int p = __ffsll((long long)bmask) - 1;
    bmask &= bmask - 1ull;
    if (s_tok[p] < 0 || s_tok[p] >= a.g.V) continue;
    const char* rowp = reinterpret_cast<const char*>(a.logits) + ((size_t)b * S + p) * (size_t)a.g.stride * ES;
    {  // the candidates' logits, fetched beside the row pass by the CTA's last two warps
      const int j = t - (CT - 64);
      if (j >= r0 && j < r1 && s_par[j] == p && s_tok[j] >= 0 && s_tok[j] < a.g.V)
        s_x[j] = load_scalar<DT>(rowp, s_tok[j]);
    }
    cluster_row_stats<DT, CT, BULK>(cluster, rowp, a.g.V, a.g.vec != 0, LOG2E, st, pass++, BULK ? s_stage : nullptr,
                                    &s_bar, a.err, a.wait_polls);
    const float M = st.M, Z = st.W;
    if (warp == 0 && rank == 0 && Z > 0.f) {
      // the kept draft children of p; a candidate with one of their tokens is not new
      uint64_t kept = 0ull;
      for (int base = 0; base < r0; base += 32) {
        const int q = base + lane;
        kept |= (uint64_t)__ballot_sync(FULL, q >= 1 && q < r0 && s_par[q] == p) << base;
      }
      float g = 0.f;
      for (int j = r0 + lane; j < r1; j += 32) {
        const int32_t tk = s_tok[j];
        if (s_par[j] != p || tk < 0 || tk >= a.g.V) continue;
        bool dup = false;
        for (uint64_t km = kept; km != 0ull; km &= km - 1ull) dup |= s_tok[__ffsll((long long)km) - 1] == tk;
        if (!dup) g += exp2f((s_x[j] - M) * LOG2E) / Z;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) g += __shfl_xor_sync(FULL, g, o);
      total += g;
    }
    __syncthreads();  // s_x is read before the next parent's loads
  }
  if (t == 0 && rank == 0) gain[b] = total;
  if (pass == 0) cluster_started_wait();  // (no pass: the start barrier still completes)
}

template <int DT, bool BULK>
cudaError_t coverage_launch(const VerifyArgs& a, const int32_t* info, float* gain, int bytes, cudaStream_t s) {
  if (BULK && bytes > 48 * 1024) {  // above the default limit the kernel must opt in (per device: set it each time)
    const cudaError_t e =
        cudaFuncSetAttribute(k_coverage<DT, BULK>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.batch * CL);
  cfg.blockDim = dim3(CT);
  cfg.dynamicSmemBytes = BULK ? bytes : 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_coverage<DT, BULK>, a, info, gain);
}

template <int DT>
cudaError_t coverage_impl(const VerifyArgs& a, const int32_t* info, float* gain, cudaStream_t s) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int bytes = stage_bytes(a.g.V, ES);
  return a.g.vec && bytes <= STAGE_MAX ? coverage_launch<DT, true>(a, info, gain, bytes, s)
                                       : coverage_launch<DT, false>(a, info, gain, bytes, s);
}

}  // namespace

cudaError_t launch_coverage(const VerifyArgs& a, const int32_t* info, float* gain, int dtype, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? coverage_impl<GRAFT_BF16>(a, info, gain, s) : coverage_impl<GRAFT_F32>(a, info, gain, s);
}

}  // namespace graft
