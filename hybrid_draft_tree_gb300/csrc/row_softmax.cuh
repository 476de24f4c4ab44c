// Softmax statistics of one logits row, computed by a thread-block cluster,
// for the kernels that need target probabilities (stochastic verification,
// the coverage diagnostic).
//
// One request's row is read by a cluster of CL CTAs (CL SMs): CTA r of the
// cluster owns a contiguous range of the row, and thread t of the CTA owns a
// contiguous chunk of that range (lengths multiples of the vector width when
// the row is 16-byte aligned, so chunks are read with 16-byte loads).  Each
// thread keeps a (max, sum of exp2((x - max) * k2)) over its chunk (online
// while reading the row, or the maximum first when the chunk is staged),
// k2 = log2(e) / temperature; warp 0 folds them into the CTA's pair, and each
// CTA writes its pair into every CTA of the cluster (distributed shared
// memory), each then folding the CL pairs in rank order, so every CTA of the
// cluster holds the same row maximum and sum.  The chunks' pairs stay in shared memory, so an inverse-CDF
// draw over the row can locate its CTA and its chunk without another pass;
// given a staging buffer, the CTA also keeps its range of the row in shared
// memory, so the draw reads no global memory at all.
// All threads of every CTA of the cluster must call.
#pragma once
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "bulk_copy.cuh"
#include "graft_internal.cuh"
#include "scan_common.cuh"

namespace graft {
namespace softmax {
using namespace scan;
namespace cg = cooperative_groups;

constexpr int CL = 8;  // CTAs per row: one portable thread-block cluster

template <int NT>
struct ClusterRow {
  float m[NT];        // chunk maxima
  float s[NT];        // chunk sums of exp2((x - m[t]) * k2)
  float pm[2][CL], ps[2][CL];  // every CTA's (max, sum) by pass parity and rank, written by that CTA
  float em[CL], es[CL];        // every CTA's (max, sum) of the last pass, by rank
  float M, W;         // row maximum and sum of exp2((x - M) * k2), the same in every CTA of the cluster
  int lo, hi, ch;     // this CTA's element range and its chunk length
};

// The cluster's start barrier, split: every thread of every CTA arrives once
// at the start of the kernel (cluster_started_arrive) and waits before its
// first write into another CTA's shared memory (cluster_started_wait, called by
// the first pass of cluster_row_stats; a kernel that makes no pass calls it
// before it exits), so no CTA is written to before it runs.
__device__ __forceinline__ void cluster_started_arrive() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_started_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// 16 bytes of shared memory at shared-space address a.  The stage reaches the
// statistics as a generic pointer (it may be null in the kernels), so its
// loads are made explicit shared-memory loads.
__device__ __forceinline__ uint4 lds16(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}

// (m, s) <- online update with element x.
__device__ __forceinline__ void online_add(float& m, float& s, float x, float k2) {
  if (x > m) {
    s = s * exp2f((m - x) * k2) + 1.f;
    m = x;
  } else if (x != -INFINITY) {
    s += exp2f((x - m) * k2);
  }
}

// Element i of a staged range (the row's own type), and its store.
template <int DT>
__device__ __forceinline__ float stage_elem(const char* stage, int i) {
  if (DT == GRAFT_BF16) return __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(stage)[i] << 16);
  return reinterpret_cast<const float*>(stage)[i];
}
template <int DT>
__device__ __forceinline__ void store_elem(char* stage, int i, float x) {
  if (DT == GRAFT_BF16) reinterpret_cast<unsigned short*>(stage)[i] = (unsigned short)(__float_as_uint(x) >> 16);
  else reinterpret_cast<float*>(stage)[i] = x;
}

// Element range [lo, hi) of cluster rank `rank` in a V-element row: ranges of
// ceil(V / CL) rounded up to a multiple of `epl`.
__device__ __forceinline__ void cta_range(int V, int epl, int rank, int& lo, int& hi) {
  int per = (V + CL - 1) / CL;
  per = (per + epl - 1) / epl * epl;
  lo = min(rank * per, V);
  hi = min(lo + per, V);
}

// Bytes of shared memory that hold one CTA's range of a V-element row.
__device__ __host__ __forceinline__ int stage_bytes(int V, int esize) {
  const int epl = 16 / esize;
  int per = (V + CL - 1) / CL;
  per = (per + epl - 1) / epl * epl;
  return per * esize;
}

// One pass over row `rowp` (pass index `pass`, from 0: consecutive passes
// alternate the exchange slots, so a CTA never overwrites a pair another CTA
// may still be reading; the kernel must have called cluster_started_arrive).
// On return st.M, st.W hold the row's statistics in every CTA; st.m / st.s /
// st.lo / st.hi / st.ch describe this CTA's chunks and st.em / st.es every
// CTA's pair.  With `stage` (stage_bytes(V, esize) bytes of shared memory,
// 16-byte aligned), element v of this CTA's range is left at stage[v - lo].
// With BULK (a stage, an aligned row and `bar`, an initialised mbarrier; pass
// p waits for its phase p & 1, so every call must stage), the range arrives
// by bulk copies issued by one thread (the wait bounded by `polls`, a timeout
// flagged in `err` and drained before the stage is read) and the threads then
// read their chunks from shared memory; the chunks then hold an odd number of
// 16-byte vectors, so the threads of a warp read distinct banks.
template <int DT, int NT, bool BULK = false>
__device__ void cluster_row_stats(const cg::cluster_group& cluster, const char* rowp, int V, bool vec, float k2,
                                  ClusterRow<NT>& st, int pass, char* stage = nullptr,
                                  unsigned long long* bar = nullptr, uint32_t* err = nullptr, uint32_t polls = 0) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int t = threadIdx.x;
  constexpr int EPL = Vec16<DT>::EPL;
  constexpr int UNR = 8;  // 16-byte loads in flight per thread
  const int epl = vec ? EPL : 1;
  const bool bulk = BULK;  // the caller guarantees a stage, an aligned row and a barrier
  int lo, hi;
  cta_range(V, epl, (int)cluster.block_rank(), lo, hi);
  int ch = (hi - lo + NT - 1) / NT;
  ch = (ch + epl - 1) / epl * epl;
  if (bulk && ((ch / EPL) & 1) == 0) ch += EPL;  // an odd number of vectors per chunk
  const int v0 = min(lo + t * ch, hi), v1 = min(v0 + ch, hi);
  float m = -INFINITY, s = 0.f;
  if (bulk) {
    const uint32_t bytes = (uint32_t)((hi - lo) / EPL) * 16u;  // the range's whole vectors
    const uint32_t parity = (uint32_t)pass & 1u;
    if (t == 0 && bytes > 0) {
      bulk::mbar_expect_tx(bar, bytes);
      for (uint32_t off = 0; off < bytes; off += 32768u)
        bulk::bulk_g2s(stage + off, rowp + (size_t)lo * ES + off, min(32768u, bytes - off), bar);
    }
    for (int v = lo + (int)(bytes / ES) + t; v < hi; v += NT) store_elem<DT>(stage, v - lo, load_scalar<DT>(rowp, v));
    if (t < 32 && bytes > 0) {
      const bool ok = bulk::mbar_poll_warp(bar, parity, polls ? polls : bulk::SPIN);
      if (!ok && t == 0) {
        atomicOr(err, GRAFT_ERR_TIMEOUT);  // the step's results are not valid
        bulk::mbar_wait_drain(bar, parity);  // the copies land before the stage is read or rewritten
      }
    }
    __syncthreads();
    if (bytes > 0) (void)bulk::mbar_test_wait(bar, parity);  // each thread observes the completed phase itself
    // the chunk is in shared memory, so it is read twice: its maximum first
    // (four independent maxima), then its exponentials into eight independent
    // partial sums, with no rescaling between them
    const uint32_t sp = bulk::smem_u32(stage) + (uint32_t)(v0 - lo) * ES;  // the chunk, 16-byte aligned
    const int nvec = (v1 - v0) / EPL;
    float m0 = -INFINITY, m1 = -INFINITY, m2 = -INFINITY, m3 = -INFINITY;
    int i = 0;
    for (; i + 4 <= nvec; i += 4) {
      Vec16<DT> x0, x1, x2, x3;
      x0.r = lds16(sp + 16u * i);
      x1.r = lds16(sp + 16u * (i + 1));
      x2.r = lds16(sp + 16u * (i + 2));
      x3.r = lds16(sp + 16u * (i + 3));
      m0 = fmaxf(m0, x0.vmax_drop_nan());
      m1 = fmaxf(m1, x1.vmax_drop_nan());
      m2 = fmaxf(m2, x2.vmax_drop_nan());
      m3 = fmaxf(m3, x3.vmax_drop_nan());
    }
    for (; i < nvec; ++i) {
      Vec16<DT> x0;
      x0.r = lds16(sp + 16u * i);
      m0 = fmaxf(m0, x0.vmax_drop_nan());
    }
    for (int v = v0 + nvec * EPL; v < v1; ++v) m1 = fmaxf(m1, stage_elem<DT>(stage, v - lo));
    m = fmaxf(fmaxf(m0, m1), fmaxf(m2, m3));
    if (m != -INFINITY) {
      // exp2(x * k2 - m * k2): one fused multiply-add per element
      const float mk = m * k2;
      float qa[4] = {0.f, 0.f, 0.f, 0.f}, qb[4] = {0.f, 0.f, 0.f, 0.f};
      for (i = 0; i + 2 <= nvec; i += 2) {
        Vec16<DT> x0, x1;
        x0.r = lds16(sp + 16u * i);
        x1.r = lds16(sp + 16u * (i + 1));
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          qa[e & 3] += exp2f(fmaf(x0.elem(e), k2, -mk));
          qb[e & 3] += exp2f(fmaf(x1.elem(e), k2, -mk));
        }
      }
      if (i < nvec) {
        Vec16<DT> x0;
        x0.r = lds16(sp + 16u * i);
#pragma unroll
        for (int e = 0; e < EPL; ++e) qa[e & 3] += exp2f(fmaf(x0.elem(e), k2, -mk));
      }
      for (int v = v0 + nvec * EPL; v < v1; ++v) qb[v & 3] += exp2f((stage_elem<DT>(stage, v - lo) - m) * k2);
      s = ((qa[0] + qa[1]) + (qa[2] + qa[3])) + ((qb[0] + qb[1]) + (qb[2] + qb[3]));
    }
  } else if (!BULK && vec) {
    const uint4* p = reinterpret_cast<const uint4*>(rowp) + v0 / EPL;
    const int nvec = (v1 - v0) / EPL;  // whole vectors of the chunk (only the row's last chunk has a rest)
    uint4* sp = stage ? reinterpret_cast<uint4*>(stage + (size_t)(v0 - lo) * ES) : nullptr;
    for (int base = 0; base < nvec; base += UNR) {
      Vec16<DT> x[UNR];
#pragma unroll
      for (int u = 0; u < UNR; ++u)
        if (base + u < nvec) x[u].r = __ldcs(p + base + u);
      // the batch's maximum first (one rescale per batch), then its
      // exponentials into four independent partial sums
      float bm = -INFINITY;
#pragma unroll
      for (int u = 0; u < UNR; ++u) {
        if (base + u >= nvec) break;
        if (sp) sp[base + u] = x[u].r;
        bm = fmaxf(bm, x[u].vmax());
      }
      if (bm > m) { s *= exp2f((m - bm) * k2); m = bm; }
      if (m != -INFINITY) {
        float q[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int u = 0; u < UNR; ++u) {
          if (base + u >= nvec) break;
#pragma unroll
          for (int e = 0; e < EPL; ++e) q[e & 3] += exp2f((x[u].elem(e) - m) * k2);
        }
        s += (q[0] + q[1]) + (q[2] + q[3]);
      }
    }
    for (int v = v0 + nvec * EPL; v < v1; ++v) {
      const float x = load_scalar<DT>(rowp, v);
      if (stage) store_elem<DT>(stage, v - lo, x);
      online_add(m, s, x, k2);
    }
  } else {
    for (int v = v0; v < v1; ++v) {
      const float x = load_scalar<DT>(rowp, v);
      if (stage) store_elem<DT>(stage, v - lo, x);
      online_add(m, s, x, k2);
    }
  }
  st.m[t] = m;
  st.s[t] = s;
  if (t == 0) { st.lo = lo; st.hi = hi; st.ch = ch; }
  __syncthreads();
  const int slot = pass & 1;
  if (pass == 0) cluster_started_wait();
  if (t < 32) {
    float cm = -INFINITY;
    for (int i = t; i < NT; i += 32) cm = fmaxf(cm, st.m[i]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(FULL, cm, o));
    float cs = 0.f;
    if (cm != -INFINITY)
      for (int i = t; i < NT; i += 32) cs += st.m[i] == -INFINITY ? 0.f : st.s[i] * exp2f((st.m[i] - cm) * k2);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) cs += __shfl_xor_sync(FULL, cs, o);
    if (t < CL) {  // this CTA's pair, written into every CTA of the cluster
      const int rank = (int)cluster.block_rank();
      *cluster.map_shared_rank(&st.pm[slot][rank], t) = cm;
      *cluster.map_shared_rank(&st.ps[slot][rank], t) = cs;
    }
  }
  // every CTA's pair of this pass is in every CTA; no CTA reads another's
  // shared memory, so a CTA may exit after its last pass
  cluster.sync();
  if (t < 32) {
    // lane r folds CTA r's pair; the same butterflies over the same values in
    // every CTA give every CTA the same (M, W)
    float mr = -INFINITY, sr = 0.f;
    if (t < CL) {
      mr = st.pm[slot][t];
      sr = st.ps[slot][t];
      st.em[t] = mr;
      st.es[t] = sr;
    }
    // (the CL = 8 pairs sit in lanes 0..7: three butterfly steps fold them)
    static_assert(CL == 8, "the fold below covers 8 lanes");
    float M = mr;
#pragma unroll
    for (int o = CL / 2; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(FULL, M, o));
    float W = (mr == -INFINITY) ? 0.f : sr * exp2f((mr - M) * k2);
#pragma unroll
    for (int o = CL / 2; o > 0; o >>= 1) W += __shfl_xor_sync(FULL, W, o);
    if (t == 0) { st.M = M; st.W = W; }
  }
  __syncthreads();
}

}  // namespace softmax
}  // namespace graft
