// The verify + update pass of a Graft step (popular-science article on arXiv
// 2605.20104, section 二 third gear) for small steps: few verified rows, each
// small enough to sit in the shared memory of one thread-block cluster.
//
// With few rows (a single request's tree: 61 rows) the two-pass scan is all
// latency: two launches, a stream of a few MB, then pass 2's chain of unit
// maxima, a candidate reload and the request ticket.  Here one cluster of CL
// CTAs takes one row: each CTA stages its range of the row in shared memory
// (the row's only read: bulk copies into shared memory), then every thread
// takes the maximum of its elements, each warp the two largest of its
// threads' maxima, and the CTA takes T, the 8th largest of those 16.  Eight
// distinct elements of the range reach T (each is its thread's maximum), so
// every element of the range's top-8 is >= T; the CTA lists its elements >= T from
// shared memory and sorts them into its exact top-8 (value desc, id asc).  The row's top-8 is among the 8
// CTAs' top-8s: CTA 0 of the cluster merges the 64 keys through distributed
// shared memory, writes the row's share of the update and, for the row
// completing a request, runs its acceptance from the request's tree arrays,
// which it staged in shared memory at the start.  A range with fewer than 8
// finite values among the 16, or with more than RCAP elements >= T (heavy ties),
// takes its exact top-8 by repeated maxima over the staged range instead.
#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include <climits>

#include "bulk_copy.cuh"
#include "graft_internal.cuh"
#include "row_softmax.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;
using namespace bulk;
namespace cg = cooperative_groups;
using softmax::CL;

constexpr int RT = 256;     // threads per CTA
constexpr int RW = RT / 32;
constexpr int RCAP = 128;   // elements >= T one CTA may list before its exact pass
constexpr int UNR = 8;      // 16-byte loads in flight per thread while staging (unaligned rows)
constexpr uint32_t BULK = 32768;  // bytes per bulk copy

// Lanes 16g .. 16g + 15 hold two descending runs of 8 keys (lanes 16g ..
// 16g + 7 and 16g + 8 .. 16g + 15); lanes 16g .. 16g + 7 get the 8 largest of
// the 16, descending.  The second run reversed makes the 16 a bitonic
// sequence, which four compare-exchange stages sort.
__device__ __forceinline__ u64 top8_of_two_runs(u64 key, int lane) {
  const u64 r = __shfl_xor_sync(FULL, key, 7);
  if (lane & 8) key = r;
#pragma unroll
  for (int j = 8; j > 0; j >>= 1) {
    const u64 o = __shfl_xor_sync(FULL, key, j);
    key = (lane & j) == 0 ? (key > o ? key : o) : (key < o ? key : o);
  }
  return key;
}

template <int DT>
__global__ void __launch_bounds__(RT, 8) k_cluster_select(VerifyArgs a, int32_t* C) {
  extern __shared__ __align__(16) char stage[];
  __shared__ int32_t stok[CLUSTER_MAX_ROWS];
  __shared__ uint64_t smask[MAX_S];  // CTA 0: the tree arrays of this row's request
  __shared__ int32_t spos[MAX_S];
  __shared__ int8_t spar[MAX_S];
  __shared__ int32_t wmax[2 * RW];   // each warp's two largest thread maxima
  __shared__ u64 s_list[RCAP];       // this CTA's elements >= T
  __shared__ u64 s_top[K];           // this CTA's top-8 keys (read by CTA 0)
  __shared__ u64 s_wbest[RW];
  __shared__ int s_nc, s_T;
  __shared__ unsigned long long s_bar;  // the staging copies' barrier
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  constexpr int EPL = Vec16<DT>::EPL;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
  const int row = blockIdx.x / CL;
  const int rows = a.batch * a.S;  // the host keeps rows <= CLUSTER_MAX_ROWS
  const int V = a.g.V;
  grid_dependents_launch();  // the stochastic walk may be scheduled as SMs free up; it waits for this grid

  for (int r = t; r < rows; r += RT) stok[r] = __ldcg(a.tree_tok + r);
  const int b = row / a.S;
  if (rank == 0)
    for (int i = t; i < a.S; i += RT) {
      const size_t q = (size_t)b * a.S + i;
      spar[i] = __ldcg(a.tree_parent + q);
      spos[i] = __ldcg(a.tree_pos + q);
      smask[i] = __ldcg(reinterpret_cast<const unsigned long long*>(a.tree_mask) + q);
    }
  if (t == 0) {
    s_nc = 0;
    mbar_init(&s_bar, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const int32_t tok = stok[row];
  // a request with no valid slot has no row to finish it: its first row's cluster does
  if (rank == 0 && warp == 0 && !a.sample && row == b * a.S && request_valid(a, stok, b, lane) == 0)
    accept_request(a, b, lane, stok);
  if (rank == 0 && t == 0 && tok >= V) atomicOr(a.err, GRAFT_ERR_TOKEN);  // such a slot is skipped
  if (tok < 0 || tok >= V) return;  // the whole cluster (one row) leaves before any exchange

  // 1. stage this CTA's range of the row; every thread keeps the maximum of
  //    its elements.  Thread t owns the range's whole 16-byte vectors t,
  //    t + RT, ... and its other elements t, t + RT, ... after them: a warp's
  //    shared-memory reads are then consecutive (no bank conflicts), and any
  //    split of the elements among the threads serves the threshold argument
  const bool vec = a.g.vec;
  const int epl = vec ? EPL : 1;
  int lo, hi;
  softmax::cta_range(V, epl, rank, lo, hi);
  const int nv = vec ? (hi - lo) / EPL : 0;  // whole vectors of the range
  const int rest0 = lo + nv * EPL;            // its first element after them
  const char* rowp = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)a.g.stride * ES;
  const uint4* sv = reinterpret_cast<const uint4*>(stage);
  float tm = -INFINITY;  // NaN elements are flagged and left out
  bool nan = false;
  if (vec) {
    // the whole vectors in bulk copies issued by one thread (the row and the
    // stage are 16-byte aligned), the rest with plain loads
    const uint32_t bytes = (uint32_t)nv * 16u;
    if (t == 0 && bytes > 0) {
      mbar_expect_tx(&s_bar, bytes);
      for (uint32_t off = 0; off < bytes; off += BULK)
        bulk_g2s(stage + off, rowp + (size_t)lo * ES + off, min(BULK, bytes - off), &s_bar);
    }
    for (int v = rest0 + t; v < hi; v += RT) softmax::store_elem<DT>(stage, v - lo, load_scalar<DT>(rowp, v));
    if (warp == 0 && bytes > 0) {
      const bool ok = mbar_poll_warp(&s_bar, 0, a.wait_polls ? a.wait_polls : SPIN);
      if (!ok && lane == 0) {
        atomicOr(a.err, GRAFT_ERR_TIMEOUT);  // the step's results are not valid
        mbar_wait_drain(&s_bar, 0);          // the copies land before this CTA reads on or exits
      }
    }
    __syncthreads();
    if (bytes > 0) (void)mbar_test_wait(&s_bar, 0);  // each thread observes the completed phase itself
    if (DT == GRAFT_BF16) {
      // a NaN-propagating running maximum of bf16 pairs (four pair
      // operations per vector); a NaN in it sends the thread through its
      // vectors again with NaN left out
      const __nv_bfloat162 ninf = __float2bfloat162_rn(-INFINITY);
      __nv_bfloat162 acc = ninf;
      for (int q = t; q < nv; q += RT) {
        const uint4 r = sv[q];
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
        const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
        acc = __hmax2_nan(acc, __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d)));
      }
      const uint32_t u = *reinterpret_cast<const uint32_t*>(&acc);
      const float lo = __uint_as_float(u << 16), hi = __uint_as_float(u & 0xFFFF0000u);
      if (lo != lo || hi != hi) {
        nan = true;
        for (int q = t; q < nv; q += RT) {
          Vec16<DT> x;
          x.r = sv[q];
#pragma unroll
          for (int e = 0; e < EPL; ++e) tm = fmaxf(tm, x.elem(e));  // fmaxf drops NaN
        }
      } else {
        tm = fmaxf(lo, hi);
      }
    } else {
      for (int q = t; q < nv; q += RT) {
        Vec16<DT> x;
        x.r = sv[q];
        const float m = x.vmax();
        if (m != m) {
          nan = true;
#pragma unroll
          for (int e = 0; e < EPL; ++e) tm = fmaxf(tm, x.elem(e));  // fmaxf drops NaN
        } else {
          tm = fmaxf(tm, m);
        }
      }
    }
  }
  // elements after the whole vectors (every element when the row is not
  // 16-byte aligned: staged here with plain loads)
  for (int base = rest0 + t; base < hi; base += RT * UNR) {
    float x[UNR];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int v = base + u * RT;
      x[u] = v < hi ? (vec ? softmax::stage_elem<DT>(stage, v - lo) : load_scalar<DT>(rowp, v)) : -INFINITY;
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const int v = base + u * RT;
      if (v >= hi) break;
      if (!vec) softmax::store_elem<DT>(stage, v - lo, x[u]);
      if (x[u] != x[u]) nan = true;
      tm = fmaxf(tm, x[u]);
    }
  }
  if (nan) atomicOr(a.err, GRAFT_ERR_NAN);

  // 2. T = the 8th largest of the warps' two largest thread maxima (16
  //    values from 16 threads: 16 distinct elements)
  {
    const int32_t k1 = ord_int(tm);
    const int32_t m1 = __reduce_max_sync(FULL, k1);
    const int lead = __ffs(__ballot_sync(FULL, k1 == m1)) - 1;
    const int32_t m2 = __reduce_max_sync(FULL, lane == lead ? INT_MIN : k1);
    if (lane == 0) { wmax[2 * warp] = m1; wmax[2 * warp + 1] = m2; }
  }
  __syncthreads();
  if (warp == 0) {
    // lane l < 16 counts the values above its own (ties by position); the
    // lane with 7 above holds the 8th largest
    const int32_t v = lane < 2 * RW ? wmax[lane] : INT_MIN;
    int above = 0;
#pragma unroll
    for (int i = 0; i < 2 * RW; ++i) {
      const int32_t x = wmax[i];
      above += (x > v) || (x == v && i < lane);
    }
    const unsigned at8 = __ballot_sync(FULL, lane < 2 * RW && above == K - 1);
    if (lane == __ffs(at8) - 1) s_T = v;
  }
  __syncthreads();
  const int32_t Ti = s_T;
  const float T = from_ord_int(Ti);
  bool exact = !(Ti != INT_MIN && T > -INFINITY);  // fewer than 8 finite values

  // 3. this CTA's elements >= T, from shared memory, then its top-8
  if (!exact) {
    for (int q = t; q < nv; q += RT) {
      Vec16<DT> x;
      x.r = sv[q];
      unsigned m = x.ge_mask(T);
      while (m) {
        const int e = __ffs(m) - 1;
        m &= m - 1;
        const int pos = atomicAdd(&s_nc, 1);
        if (pos < RCAP) s_list[pos] = make_key(x.elem(e), lo + q * EPL + e);
      }
    }
    for (int v = rest0 + t; v < hi; v += RT) {
      const float x = softmax::stage_elem<DT>(stage, v - lo);
      if (x >= T) {
        const int pos = atomicAdd(&s_nc, 1);
        if (pos < RCAP) s_list[pos] = make_key(x, v);
      }
    }
    __syncthreads();
    exact = s_nc > RCAP;  // heavy ties: the list overflowed
    if (!exact && warp == 0) {
      // up to 32 candidates: one bitonic sort of them (of 16 when they fit);
      // more: chunks merged into a running top-8
      const int nc = s_nc;
      u64 top;
      if (nc <= 16) top = bitonic_desc<16>(lane < nc ? s_list[lane] : 0ull, lane);
      else if (nc <= 32) top = bitonic_desc<32>(lane < nc ? s_list[lane] : 0ull, lane);
      else top = warp_merge(0ull, s_list, nc, lane);
      if (lane < K) s_top[lane] = top;
    }
  }
  if (exact) {
    // exact pass: 8 rounds of block-wide maxima below the last
    u64 prev = ~0ull;
    for (int r = 0; r < K; ++r) {
      u64 best = 0ull;
      for (int q = t; q < nv; q += RT) {
        Vec16<DT> x;
        x.r = sv[q];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const u64 key = make_key(x.elem(e), lo + q * EPL + e);
          if (key < prev && key > best) best = key;
        }
      }
      for (int v = rest0 + t; v < hi; v += RT) {
        const u64 key = make_key(softmax::stage_elem<DT>(stage, v - lo), v);
        if (key < prev && key > best) best = key;
      }
      best = warp_max_u64(best);
      if (lane == 0) s_wbest[warp] = best;
      __syncthreads();
      u64 cb = lane < RW ? s_wbest[lane] : 0ull;
      cb = warp_max_u64(cb);
      if (t == 0) s_top[r] = cb;  // 0 (no key) once the range runs out
      prev = cb;
      __syncthreads();
    }
  }
  cluster.sync();  // every CTA's top-8 is written

  // 4. CTA 0 merges the 8 CTAs' top-8s (lane l reads keys l and l + 32 of the 64)
  u64 top = 0ull;
  if (rank == 0 && warp == 0) {
    // a tournament of bitonic merges over the 8 descending lists: CTAs
    // (0, 1), (2, 3), (4, 5), (6, 7), then the pairs' winners, then the halves'
    u64 k0 = *cluster.map_shared_rank(&s_top[lane & 7], lane >> 3);
    u64 k1 = *cluster.map_shared_rank(&s_top[lane & 7], 4 + (lane >> 3));
    k0 = top8_of_two_runs(k0, lane);  // lanes 0..7: CTAs 0, 1; lanes 16..23: CTAs 2, 3
    k1 = top8_of_two_runs(k1, lane);  // the same for CTAs 4 .. 7
    const int down = (lane & 7) | ((lane & 8) << 1);  // lanes 8..15 take lanes 16..23
    k0 = top8_of_two_runs(__shfl_sync(FULL, k0, down), lane);  // lanes 0..7: CTAs 0 .. 3
    k1 = top8_of_two_runs(__shfl_sync(FULL, k1, down), lane);  // lanes 0..7: CTAs 4 .. 7
    const u64 k1d = __shfl_sync(FULL, k1, lane & 7);
    top = top8_of_two_runs((lane & 8) ? k1d : k0, lane);        // lanes 0..7: the row's top-8
  }
  cluster.sync();  // CTA 0 has read the keys: the other CTAs may leave
  if (rank != 0 || warp != 0) return;
  const int32_t id = key_id(top);
  if (lane < K) a.topk[(size_t)row * K + lane] = id;
  // the matrix row of the token: written unless a later row in (request,
  // slot) order carries the same token
  bool later = false;
  for (int r = row + 1 + lane; r < rows; r += 32) later |= stok[r] == tok;
  later = __any_sync(FULL, later);
  if (!later && lane < K) st_keep(C + (size_t)tok * K + lane, id, l2_keep_policy());
  if (a.sample) return;  // stochastic verification accepts in its own kernel
  // the warp that completes the request's last valid row runs acceptance
  const int nvalid = request_valid(a, stok, b, lane);
  __syncwarp();
  int tk = 0;
  if (lane == 0) tk = ticket_acq_rel(&a.req_ticket[b]);
  tk = __shfl_sync(FULL, tk, 0);
  if (tk == nvalid - 1) {
    if (lane == 0) a.req_ticket[b] = 0;
    __syncwarp();
    accept_staged(a, b, lane, stok, spar, spos, smask);
  }
}

// Clusters of this kernel that fit on the device at once with V-element rows
// (0 when the rows do not fit the kernel, or on any error).
template <int DT>
int cluster_select_max_active_impl(int V) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int bytes = softmax::stage_bytes(V, ES);
  if (bytes > CLUSTER_STAGE_MAX) return 0;
  if (bytes > 48 * 1024 &&
      cudaFuncSetAttribute(k_cluster_select<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(CL);
  cfg.blockDim = dim3(RT);
  cfg.dynamicSmemBytes = bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, k_cluster_select<DT>, &cfg) != cudaSuccess) return 0;
  return n;
}

template <int DT>
cudaError_t cluster_select_impl(const VerifyArgs& a, int32_t* C, cudaStream_t s) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int bytes = softmax::stage_bytes(a.g.V, ES);
  if (bytes > 48 * 1024) {  // above the default limit the kernel must opt in (per device: set it each time)
    const cudaError_t e = cudaFuncSetAttribute(k_cluster_select<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(a.batch * a.S * CL);
  cfg.blockDim = dim3(RT);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_cluster_select<DT>, a, C);
}

}  // namespace

bool cluster_select_fits(int rows, int V, int esize) {
  return rows <= CLUSTER_MAX_ROWS && softmax::stage_bytes(V, esize) <= CLUSTER_STAGE_MAX;
}

int cluster_select_max_active(int V, int dtype) {
  const int n = dtype == GRAFT_BF16 ? cluster_select_max_active_impl<GRAFT_BF16>(V)
                                    : cluster_select_max_active_impl<GRAFT_F32>(V);
  cudaGetLastError();  // a failed query leaves no error behind
  return n;
}

// Measured on GB300 (verify_update, L2 flushed), one request of 61 rows:
// 32000 fp32 (16 KB per CTA) 14.3-15.0 us against 17.1-18.8 us on the
// two-pass scan; 128256 bf16 (32 KB) 16.4 against 18.9; 151936 bf16 (38 KB)
// 18.4 against 19.3-20.5; two requests of 32000 fp32 (122 clusters, all
// resident) 18.4 against 19.1.  Once the clusters no longer fit at once
// (three requests of 32000 fp32; two of 151936 bf16, 5 CTAs per SM by shared
// memory) each further wave makes it slower than the two-pass scan.
bool cluster_select_auto(int rows, int V, int esize, int max_active) {
  return rows <= max_active && rows <= CLUSTER_AUTO_ROWS && softmax::stage_bytes(V, esize) <= CLUSTER_AUTO_STAGE;
}

cudaError_t launch_cluster_select(const VerifyArgs& a, int dtype, int32_t* C, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? cluster_select_impl<GRAFT_BF16>(a, C, s) : cluster_select_impl<GRAFT_F32>(a, C, s);
}

}  // namespace graft
