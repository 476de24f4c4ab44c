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
// One thread-block cluster of CL CTAs per request walks the accepted path
// (row_softmax.cuh: each node's row is read once, split over the cluster's
// SMs, each CTA keeping its range in shared memory).  Every CTA takes the same
// decisions from the same statistics, so the walk needs no further exchange;
// for the final draw every CTA derives every CTA's weight from the exchanged
// (max, sum) pairs, so all agree on the CTA holding the target without another
// exchange, and that CTA finds its chunk and one warp scans it in shared
// memory, so no second pass over the row is needed.  The top-8 and matrix update come
// from the scan kernels as in greedy verification; this kernel reads only the
// logits and the trees, so it is launched as a programmatic dependent of the
// update kernel and runs beside it (it waits for that kernel only before it
// exits, so its completion still implies theirs).
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "row_softmax.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;
using namespace softmax;

constexpr int PT = 256;  // threads per CTA (CL CTAs per request)
constexpr int STAGE_MAX = 160 * 1024;  // shared memory for a CTA's range of the row; larger rows read it again
constexpr float LOG2E = 1.4426950408889634f;

// BULK: the rows are staged by bulk copies (aligned rows whose CTA range fits
// the stage); otherwise by the threads' loads, or read again (staged = 0).
template <int DT, bool BULK>
__global__ __launch_bounds__(PT, 4) void k_sample(VerifyArgs a, int staged) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  extern __shared__ __align__(16) char s_stage[];  // this CTA's range of the current row (when staged)
  __shared__ ClusterRow<PT> st;
  __shared__ int32_t s_tok[MAX_S], s_par[MAX_S], s_rej[MAX_S];
  __shared__ float s_rejx[MAX_S];      // the rejected tokens' logits
  __shared__ float s_x[MAX_S];         // logits of the node's children, by slot
  __shared__ float s_u[MAX_S];         // the request's acceptance uniforms, by slot
  __shared__ float s_cw[PT];           // chunk weights of the final draw
  __shared__ int s_acc, s_nrej, s_chunk, s_pick, s_owner;
  __shared__ float s_target, s_before, s_ures, s_cbefore;
  __shared__ unsigned long long s_bar;  // the row staging's bulk copies
  const cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.x / CL, t = threadIdx.x, lane = t & 31, warp = t >> 5, S = a.S, V = a.g.V;
  const float k2 = a.inv_temp * LOG2E;
  if (t < S) {
    s_tok[t] = a.tree_tok[(int64_t)b * S + t];
    s_par[t] = a.tree_parent[(int64_t)b * S + t];
    s_u[t] = a.u_accept[(int64_t)b * S + t];
  }
  if (t == 0) {
    s_ures = a.u_resid[b];
    bulk::mbar_init(&s_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  cluster_started_arrive();
  char* stage = staged ? s_stage : nullptr;
  __syncthreads();
  int32_t* out = a.out_tokens + (int64_t)b * S;
  if (s_tok[0] < 0 || s_tok[0] >= V) {  // no valid root: nothing accepted, nothing emitted (uniform in the cluster)
    if (rank == 0 && t < S) out[t] = -1;
    if (rank == 0 && t == 0) a.accept_len[b] = 0;
    cluster_started_wait();
    grid_dependency_wait();
    return;
  }
  int node = 0, len = 0;
  for (int depth = 0; depth < S; ++depth) {  // the path has fewer than S nodes
    const char* rowp = reinterpret_cast<const char*>(a.logits) + ((size_t)b * S + node) * (size_t)a.g.stride * ES;
    // the children's logits, fetched beside the row pass by the CTA's last
    // two warps (the first ones start the row's loads without waiting)
    {
      const int j = t - (PT - 64);
      if (j >= 0 && j < S) {
        const int32_t tk = s_tok[j];
        s_x[j] = (j > node && s_par[j] == node && tk >= 0 && tk < V) ? load_scalar<DT>(rowp, tk) : 0.f;
      }
    }
    cluster_row_stats<DT, PT, BULK>(cluster, rowp, V, a.g.vec != 0, k2, st, depth, stage, &s_bar, a.err,
                                    a.wait_polls);
    const float M = st.M, W = st.W;
    if (warp == 0) {  // the same decisions in every CTA of the cluster
      // the node's children in slot order, found by the whole warp; then one
      // lane tests them in that order (each test depends on the ones before)
      uint64_t kids = 0ull;
      for (int base = 0; base < S; base += 32) {
        const int j = base + lane;
        const bool c = j > node && j < S && s_par[j] == node && s_tok[j] >= 0 && s_tok[j] < V;
        kids |= (uint64_t)__ballot_sync(FULL, c) << base;
      }
      if (lane == 0) {
        float rem = 1.f;
        int acc = -1, nrej = 0;
        while (kids != 0ull && acc < 0) {
          const int j = __ffsll((long long)kids) - 1;
          kids &= kids - 1ull;
          const int32_t tk = s_tok[j];
          bool seen = false;
          for (int q = 0; q < nrej; ++q) seen |= s_rej[q] == tk;
          if (seen) continue;  // a repeated token: its mass is gone
          const float pc = exp2f((s_x[j] - M) * k2) / W;
          if (s_u[j] * rem < pc) acc = j;
          else { rem -= pc; s_rejx[nrej] = s_x[j]; s_rej[nrej++] = tk; }
        }
        s_acc = acc;
        s_nrej = nrej;
      }
    }
    __syncthreads();
    const int acc = s_acc;
    if (acc >= 0) {
      if (rank == 0 && t == 0) out[len] = s_tok[acc];
      ++len;
      node = acc;
      continue;
    }
    // every child rejected (or a leaf): draw from the unrejected tokens.
    // 1. every CTA's weight relative to M, from the pairs the statistics
    //    exchanged, minus the rejected tokens in its range: the same values in
    //    every CTA, so each finds the CTA holding the target by itself
    const int nrej = s_nrej;
    if (warp == 0) {
      float wr = 0.f;
      if (lane < CL) {
        const float cmr = st.em[lane], csr = st.es[lane];
        wr = cmr == -INFINITY ? 0.f : csr * exp2f((cmr - M) * k2);
        int rlo, rhi;
        cta_range(V, a.g.vec ? Vec16<DT>::EPL : 1, lane, rlo, rhi);
        for (int q = 0; q < nrej; ++q) {
          const int32_t r = s_rej[q];
          if (r >= rlo && r < rhi) wr -= exp2f((s_rejx[q] - M) * k2);
        }
        wr = fmaxf(wr, 0.f);
      }
      float ci = wr;  // inclusive scan over the ranks (lanes 0 .. CL - 1)
#pragma unroll
      for (int o = 1; o < CL; o <<= 1) {
        const float y = __shfl_up_sync(FULL, ci, o);
        if (lane >= o) ci += y;
      }
      const float total = __shfl_sync(FULL, ci, CL - 1);
      const float target = s_ures * total;
      const unsigned hit = __ballot_sync(FULL, lane < CL && wr > 0.f && ci > target);
      const unsigned any = __ballot_sync(FULL, lane < CL && wr > 0.f);
      const int own = hit ? __ffs(hit) - 1 : (any ? 31 - __clz(any) : -1);  // else rounding: the last CTA with weight
      const float bc = __shfl_sync(FULL, ci - wr, own >= 0 ? own : 0);
      if (lane == 0) {
        s_owner = own;
        s_cbefore = bc;
        s_target = target;
      }
    }
    __syncthreads();
    const int owner = s_owner;
    if (owner < 0 && rank == 0 && t == 0) s_pick = -1;  // no token has weight
    const int ch = st.ch, lo = st.lo, hi = st.hi;
    // element v of this CTA's range
    auto elem = [&](int v) { return stage ? stage_elem<DT>(stage, v - lo) : load_scalar<DT>(rowp, v); };
    constexpr int CPL = PT / 32;
    float w8[CPL];
    float lsum = 0.f, incl = 0.f;
    if (owner == rank) {
      // 2. this CTA holds the target: its chunk weights, minus the rejected
      //    tokens in each chunk; warp 0's lane l sums chunks CPL*l ..
      //    CPL*l + CPL-1 in order and a warp scan orders the lanes
      const int c0 = min(lo + t * ch, hi), c1 = min(c0 + ch, hi);
      float cw = st.m[t] == -INFINITY ? 0.f : st.s[t] * exp2f((st.m[t] - M) * k2);
      for (int q = 0; q < nrej; ++q) {
        const int32_t r = s_rej[q];
        if (r >= c0 && r < c1) cw -= exp2f((elem(r) - M) * k2);
      }
      cw = fmaxf(cw, 0.f);
      s_cw[t] = cw;
      __syncthreads();  // (uniform in the CTA)
      if (warp == 0) {
#pragma unroll
        for (int i = 0; i < CPL; ++i) { w8[i] = s_cw[lane * CPL + i]; lsum += w8[i]; }
        incl = lsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(FULL, incl, o);
          if (lane >= o) incl += y;
        }
      }
    }
    const float before_cta = s_cbefore, target = s_target;
    if (warp == 0 && owner == rank) {
      // 3. its chunk, from the lanes' sums
      float run = before_cta + incl - lsum;  // weight before this lane's chunks
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
      __syncwarp();
      // 4. the chunk: per-lane sub-ranges, a warp prefix, then the lane
      //    holding the target walks its elements
      const int cidx = s_chunk;
      int pick = -1;
      if (cidx >= 0) {
        const int clo = min(lo + cidx * ch, hi), chi = min(clo + ch, hi);
        const float bef = s_before;  // weight of everything before chunk cidx
        const int sub = (chi - clo + 31) / 32;
        const int l0 = min(clo + lane * sub, chi), l1 = min(l0 + sub, chi);
        float ls = 0.f;
        int lastv = -1;
        for (int v = l0; v < l1; ++v) {
          bool rej = false;
          for (int q = 0; q < nrej; ++q) rej |= s_rej[q] == v;
          if (rej) continue;
          const float wv = exp2f((elem(v) - M) * k2);
          if (wv > 0.f) { ls += wv; lastv = v; }
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
          float rr = lb;
          for (int v = l0; v < l1 && lpick < 0; ++v) {
            bool rej = false;
            for (int q = 0; q < nrej; ++q) rej |= s_rej[q] == v;
            if (rej) continue;
            const float wv = exp2f((elem(v) - M) * k2);
            if (wv <= 0.f) continue;
            rr += wv;
            if (rr > tgt) lpick = v;
          }
          if (lpick < 0) lpick = lastv;
        }
        pick = __shfl_sync(FULL, lpick, who != 0 ? __ffs(who) - 1 : 0);
        if (who == 0) {  // rounding: the chunk's last element with weight
          const unsigned has = __ballot_sync(FULL, lastv >= 0);
          pick = has ? __shfl_sync(FULL, lastv, 31 - __clz(has)) : -1;
        }
      }
      if (lane == 0) s_pick = pick;
    }
    // thread 0 (warp 0, which holds `owner`) of the owning CTA (of CTA 0 when
    // no token has weight) writes the drawn token and the accepted length
    if (t == 0 && (owner >= 0 ? owner == rank : rank == 0)) {
      out[len] = s_pick;
      a.accept_len[b] = len;
    }
    if (rank == 0)
      for (int j = len + 1 + t; j < S; j += PT) out[j] = -1;
    grid_dependency_wait();
    return;
  }
  grid_dependency_wait();
}

template <int DT, bool BULK>
cudaError_t sample_launch(const VerifyArgs& a, int staged, int bytes, cudaStream_t s) {
  if (staged && bytes > 48 * 1024) {  // above the default limit the kernel must opt in (per device: set it each time)
    const cudaError_t e =
        cudaFuncSetAttribute(k_sample<DT, BULK>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.batch * CL);
  cfg.blockDim = dim3(PT);
  cfg.dynamicSmemBytes = staged ? bytes : 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // the walk reads only the logits and the trees: it may start while the
  // update kernel ahead of it runs (it waits for it only before exiting)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_sample<DT, BULK>, a, staged);
}

template <int DT>
cudaError_t sample_impl(const VerifyArgs& a, cudaStream_t s) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int bytes = stage_bytes(a.g.V, ES);
  const int staged = bytes <= STAGE_MAX ? 1 : 0;
  return staged && a.g.vec ? sample_launch<DT, true>(a, staged, bytes, s) : sample_launch<DT, false>(a, staged, bytes, s);
}

}  // namespace

cudaError_t launch_sample(const VerifyArgs& a, int dtype, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? sample_impl<GRAFT_BF16>(a, s) : sample_impl<GRAFT_F32>(a, s);
}

}  // namespace graft
