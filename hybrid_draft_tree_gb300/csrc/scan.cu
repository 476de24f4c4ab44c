// Streaming kernels of graft_verify_update and graft_warmup.
//
// The hot loop of a Graft step is the read of every verified slot's logits
// row (popular-science article on arXiv 2605.20104, section 二 third gear:
// verify the flattened tree in one pass, then update the continuation-matrix
// row of every verified position with the target's most likely successors).
// Greedy verification needs each row's argmax and the update needs its
// top-8, so one pass computes the top-8 and element 0 serves as the argmax.
//
// Per CTA and round every thread holds NV 16-byte vectors in registers (all
// loads in flight at once), then
//   pass 1: per-thread max -> per-warp max; T = min over the 8 warp maxima is
//           a value that at least 8 elements of the round reach, and the 8th
//           best value seen by the CTA so far is another; the larger of the
//           two bounds the combined top-8 from below;
//   pass 2: elements >= T (a few dozen of ~16K) go to a shared-memory
//           candidate list; warp 0 merges them into the running top-8 with a
//           32-lane bitonic sort on 64-bit keys (value desc, id asc).
// If the candidate list overflows (e.g. a row of equal values) the CTA falls
// back to an exact 8-round selection over its registers.
// A row split over several CTAs hands partial top-8s to the last CTA of the
// row (atomic ticket, no waiting); the last row of a request runs the
// acceptance walk on bit masks.  Nothing ever spins.
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {

using namespace scan;
constexpr int ST = 256;
constexpr int SW = ST / 32;
constexpr int NV = 8;
constexpr int CAND_CAP = 512;

// ---- load slots ------------------------------------------------------------
// A slot is 16 bytes (8 bf16 / 4 fp32) on the vector path, one element on the
// scalar path (rows not 16-byte aligned).
template <int DT, bool VEC> struct Slot;

template <int DT> struct Slot<DT, true> : Vec16<DT> {
  __device__ __forceinline__ void load(const char* row, int64_t s) {
    this->r = __ldcs(reinterpret_cast<const uint4*>(row) + s);
  }
};
template <> struct Slot<GRAFT_BF16, false> {
  uint32_t r;
  static constexpr int EPL = 1;
  __device__ __forceinline__ void load(const char* row, int64_t s) {
    r = (uint32_t)__ldcs(reinterpret_cast<const unsigned short*>(row) + s) << 16;
  }
  __device__ __forceinline__ float vmax() const { return __uint_as_float(r); }
  __device__ __forceinline__ float elem(int) const { return __uint_as_float(r); }
};
template <> struct Slot<GRAFT_F32, false> {
  uint32_t r;
  static constexpr int EPL = 1;
  __device__ __forceinline__ void load(const char* row, int64_t s) {
    r = __float_as_uint(__ldcs(reinterpret_cast<const float*>(row) + s));
  }
  __device__ __forceinline__ float vmax() const { return __uint_as_float(r); }
  __device__ __forceinline__ float elem(int) const { return __uint_as_float(r); }
};

// Shared state of one CTA's running top-8.
struct ScanSmem {
  u64 top[K];
  u64 cand[CAND_CAP];
  u64 wbest[SW];
  u64 sel[K];
  int32_t wmax[SW];
  int32_t cnt;
  float thr;     // value of the 8th best key so far (-inf while fewer than 8)
  int32_t flag;
};

// Warp 0: top <- top-8 of (top U cand[0..cnt)).  Requires cnt <= CAND_CAP.
__device__ __forceinline__ void warp_merge_candidates(ScanSmem& sm, int cnt, int lane) {
  u64 key = lane < K ? sm.top[lane] : 0ull;
  int base = 0;
  do {
    if (lane >= K) {
      const int c = base + lane - K;
      key = c < cnt ? sm.cand[c] : 0ull;
    }
    key = bitonic32_desc(key, lane);
    base += 32 - K;
  } while (base < cnt);
  if (lane < K) sm.top[lane] = key;
  const u64 k8 = __shfl_sync(FULL, key, K - 1);
  if (lane == 0) sm.thr = k8 ? key_val(k8) : -INFINITY;
}

// Scan slots [s0, s1) of one row (plus the scalar tail elements [tail0, V)
// when tail_n > 0) into sm.top.  Called by all ST threads; sm.top/thr must be
// initialised.  Element ids are row-relative.
template <int DT, bool VEC>
__device__ void scan_range(const char* row, int64_t s0, int64_t s1, int64_t tail0, int tail_n, ScanSmem& sm,
                           uint32_t* err) {
  using SlotT = Slot<DT, VEC>;
  constexpr int EPL = SlotT::EPL;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n = s1 > s0 ? s1 - s0 : 0;
  int64_t rounds = (n + (int64_t)ST * NV - 1) / ((int64_t)ST * NV);
  if (rounds == 0 && tail_n > 0) rounds = 1;
  const int64_t per_round = rounds ? (n + rounds - 1) / rounds : 0;

  for (int64_t r = 0; r < rounds; ++r) {
    const int64_t rb = s0 + r * per_round;
    const int64_t re = min(rb + per_round, s1);
    const bool last = (r == rounds - 1);

    SlotT v[NV];
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t s = rb + tid + (int64_t)k * ST;
      if (s < re) v[k].load(row, s);
    }
    const bool has_tail = last && tid < tail_n;
    const float tv = has_tail ? load_scalar<DT>(row, tail0 + tid) : -INFINITY;

    // pass 1: slot maxima, thread max, warp max
    float vm[NV];
    float tmax = tv;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      const int64_t s = rb + tid + (int64_t)k * ST;
      vm[k] = (s < re) ? v[k].vmax() : -INFINITY;
      tmax = max_nan(tmax, vm[k]);
    }
    if (tmax != tmax) atomicOr(err, GRAFT_ERR_NAN);
    const int32_t wm = __reduce_max_sync(FULL, ord_int(tmax));
    if (lane == 0) sm.wmax[warp] = wm;
    __syncthreads();
    int32_t tmin = sm.wmax[0];
#pragma unroll
    for (int w = 1; w < SW; ++w) tmin = min(tmin, sm.wmax[w]);
    const float T = fmaxf(from_ord_int(tmin), sm.thr);

    // pass 2: candidates >= T
#pragma unroll
    for (int k = 0; k < NV; ++k) {
      if (vm[k] >= T) {
        const int64_t s = rb + tid + (int64_t)k * ST;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const float x = v[k].elem(e);
          if (x >= T) {
            const int c = atomicAdd(&sm.cnt, 1);
            if (c < CAND_CAP) sm.cand[c] = make_key(x, (int32_t)(s * EPL + e));
          }
        }
      }
    }
    if (has_tail && tv >= T) {
      const int c = atomicAdd(&sm.cnt, 1);
      if (c < CAND_CAP) sm.cand[c] = make_key(tv, (int32_t)(tail0 + tid));
    }
    __syncthreads();
    const int cnt = sm.cnt;

    if (cnt <= CAND_CAP) {
      if (warp == 0 && cnt > 0) warp_merge_candidates(sm, cnt, lane);
    } else {
      // exact fallback: 8 selections of the largest key below the previous one
      u64 prev = ~0ull;
      for (int q = 0; q < K; ++q) {
        u64 best = 0ull;
#pragma unroll
        for (int k = 0; k < NV; ++k) {
          const int64_t s = rb + tid + (int64_t)k * ST;
          if (s < re) {
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
              const u64 kk = make_key(v[k].elem(e), (int32_t)(s * EPL + e));
              if (kk < prev && kk > best) best = kk;
            }
          }
        }
        if (has_tail) {
          const u64 kk = make_key(tv, (int32_t)(tail0 + tid));
          if (kk < prev && kk > best) best = kk;
        }
        if (tid < K) {
          const u64 kk = sm.top[tid];
          if (kk < prev && kk > best) best = kk;
        }
        best = warp_max_u64(best);
        if (lane == 0) sm.wbest[warp] = best;
        __syncthreads();
        u64 m = sm.wbest[0];
#pragma unroll
        for (int w = 1; w < SW; ++w) m = sm.wbest[w] > m ? sm.wbest[w] : m;
        if (tid == 0) sm.sel[q] = m;
        prev = m;
        __syncthreads();
      }
      if (tid < K) sm.top[tid] = sm.sel[tid];
      if (tid == 0) sm.thr = sm.sel[K - 1] ? key_val(sm.sel[K - 1]) : -INFINITY;
    }
    if (tid == 0) sm.cnt = 0;
    __syncthreads();
  }
}

__device__ __forceinline__ void init_top(ScanSmem& sm) {
  if (threadIdx.x < K) sm.top[threadIdx.x] = 0ull;
  if (threadIdx.x == 0) { sm.thr = -INFINITY; sm.cnt = 0; }
}

// ---- verify + update scan ----------------------------------------------------
template <int DT, bool VEC>
__global__ __launch_bounds__(ST) void k_verify(VerifyArgs a) {
  __shared__ ScanSmem sm;
  const int split = blockIdx.x;
  const int row = blockIdx.y;
  const int S = a.S;
  const int b = row / S;
  const int tid = threadIdx.x, lane = tid & 31;
  const int esize = DT == GRAFT_BF16 ? 2 : 4;
  const ScanGeom& g = a.g;

  const int32_t tok = a.tree_tok[row];
  const bool valid = tok >= 0 && tok < g.V;
  if (tid == 0 && split == 0 && tok >= g.V) atomicOr(a.err, GRAFT_ERR_TOKEN);

  init_top(sm);
  __syncthreads();
  if (valid) {
    const char* rowp = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)g.stride * esize;
    const int64_t s0 = (int64_t)split * g.per_cta;
    const int64_t s1 = min(s0 + g.per_cta, g.nslot);
    const bool owns_tail = split == g.nsplit - 1 && g.tail > 0;
    scan_range<DT, VEC>(rowp, s0, s1, g.nslot * g.epl, owns_tail ? g.tail : 0, sm, a.err);
  }

  if (g.nsplit > 1) {
    if (valid && tid < K) a.part[((size_t)row * MAX_SPLIT + split) * K + tid] = sm.top[tid];
    __threadfence();
    __syncthreads();
    if (tid == 0) {
      const int t = atomicAdd(&a.row_ticket[row], 1);
      sm.flag = (t == g.nsplit - 1);
      if (sm.flag) a.row_ticket[row] = 0;
    }
    __syncthreads();
    if (!sm.flag) return;
    __threadfence();
    if (valid && tid < 32) {
      // merge the row's nsplit partial top-8s (<= 128 keys)
      const u64* p = a.part + (size_t)row * MAX_SPLIT * K;
      const int cnt = g.nsplit * K;
      u64 key = 0ull;
      int base = 0;
      bool first = true;
      do {
        if (first || lane >= K) {
          const int c = first ? lane : base + lane - K;
          key = c < cnt ? __ldcg(p + c) : 0ull;
        }
        key = bitonic32_desc(key, lane);
        base = first ? 32 : base + (32 - K);
        first = false;
      } while (base < cnt);
      if (lane < K) sm.top[lane] = key;
    }
    __syncthreads();
  }

  // this CTA finishes the row: stage its top-8 and claim the matrix row
  if (valid) {
    if (tid < K) a.topk[(size_t)row * K + tid] = key_id(sm.top[tid]);
    if (tid == 0) atomicMax(&a.winner[tok], row + 1);
  }
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int t = atomicAdd(&a.req_ticket[b], 1);
    sm.flag = (t == S - 1);
    if (sm.flag) a.req_ticket[b] = 0;
  }
  __syncthreads();
  if (!sm.flag || tid >= 32) return;
  __threadfence();

  accept_request(a, b, lane);
}

// ---- last-writer scatter into the matrix -------------------------------------
constexpr int XT = 1024;
__global__ __launch_bounds__(XT) void k_scatter(ScatterArgs a) {
  for (int r = threadIdx.x; r < a.rows; r += XT) {
    const int32_t t = a.tree_tok[r];
    if (t >= 0 && t < a.V && a.winner[t] == r + 1) {
      const int4* src = reinterpret_cast<const int4*>(a.topk + (size_t)r * K);
      int4* dst = reinterpret_cast<int4*>(a.C + (size_t)t * K);
      dst[0] = src[0];
      dst[1] = src[1];
    }
  }
  __syncthreads();
  for (int r = threadIdx.x; r < a.rows; r += XT) {
    const int32_t t = a.tree_tok[r];
    if (t >= 0 && t < a.V) a.winner[t] = 0;
  }
}

// ---- warm-up -----------------------------------------------------------------------
__global__ void k_warm_mark(WarmArgs a) {
  const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= a.n_rows) return;
  const int32_t t = a.tokens[n];
  if (t < 0 || t >= a.g.V) { atomicOr(a.err, GRAFT_ERR_TOKEN); return; }
  atomicMax(&a.winner[t], (int32_t)(n + 1));
}
__global__ void k_warm_list(WarmArgs a) {
  const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= a.n_rows) return;
  const int32_t t = a.tokens[n];
  if (t < 0 || t >= a.g.V) return;
  if (a.winner[t] == (int32_t)(n + 1)) a.list[atomicAdd(a.count, 1)] = (int32_t)n;
}
template <int DT, bool VEC>
__global__ __launch_bounds__(ST) void k_warm_scan(WarmArgs a) {
  __shared__ ScanSmem sm;
  const int esize = DT == GRAFT_BF16 ? 2 : 4;
  const int count = __ldcg(a.count);
  for (int e = blockIdx.x; e < count; e += gridDim.x) {
    const int32_t n = __ldcg(a.list + e);
    const int32_t t = a.tokens[n];
    init_top(sm);
    __syncthreads();
    const char* rowp = reinterpret_cast<const char*>(a.logits) + (size_t)n * (size_t)a.g.stride * esize;
    scan_range<DT, VEC>(rowp, 0, a.g.nslot, a.g.nslot * a.g.epl, a.g.tail, sm, a.err);
    if (threadIdx.x < K) a.C[(size_t)t * K + threadIdx.x] = key_id(sm.top[threadIdx.x]);
    __syncthreads();
  }
}
__global__ void k_warm_reset(WarmArgs a) {
  const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (n == 0) *a.count = 0;
  if (n >= a.n_rows) return;
  const int32_t t = a.tokens[n];
  if (t >= 0 && t < a.g.V) a.winner[t] = 0;
}

template <int DT, bool VEC>
cudaError_t verify_impl(const VerifyArgs& a, cudaStream_t s) {
  dim3 grid(a.g.nsplit, a.batch * a.S);
  k_verify<DT, VEC><<<grid, ST, 0, s>>>(a);
  return cudaGetLastError();
}
template <int DT, bool VEC>
cudaError_t warm_impl(const WarmArgs& a, int grid_ctas, cudaStream_t s) {
  const int t = 256;
  const unsigned g = (unsigned)((a.n_rows + t - 1) / t);
  k_warm_mark<<<g, t, 0, s>>>(a);
  k_warm_list<<<g, t, 0, s>>>(a);
  k_warm_scan<DT, VEC><<<grid_ctas, ST, 0, s>>>(a);
  k_warm_reset<<<g, t, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_verify(const VerifyArgs& a, int dtype, cudaStream_t s) {
  if (dtype == GRAFT_BF16) return a.g.vec ? verify_impl<GRAFT_BF16, true>(a, s) : verify_impl<GRAFT_BF16, false>(a, s);
  return a.g.vec ? verify_impl<GRAFT_F32, true>(a, s) : verify_impl<GRAFT_F32, false>(a, s);
}
cudaError_t launch_scatter(const ScatterArgs& a, cudaStream_t s) {
  k_scatter<<<1, XT, 0, s>>>(a);
  return cudaGetLastError();
}
cudaError_t launch_warmup(const WarmArgs& a, int dtype, int grid_ctas, cudaStream_t s) {
  if (dtype == GRAFT_BF16)
    return a.g.vec ? warm_impl<GRAFT_BF16, true>(a, grid_ctas, s) : warm_impl<GRAFT_BF16, false>(a, grid_ctas, s);
  return a.g.vec ? warm_impl<GRAFT_F32, true>(a, grid_ctas, s) : warm_impl<GRAFT_F32, false>(a, grid_ctas, s);
}

}  // namespace graft
