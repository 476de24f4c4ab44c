// Pass 2 of the two-pass verify scan: exact top-8 of every verified row from
// the unit maxima of pass 1 (umax.cu), then the row's share of the update and
// the request's acceptance.
//
// One warp per row reads the row's unit maxima.  T0, the 8th largest of the
// 32 lanes' maxima, is reached by 8 distinct elements, so every element of the
// row's top-8 is >= T0 and lies in a unit whose maximum is >= T0.  The warp
// re-reads only those units (about 9 of 594 for V = 151936 bf16), keeps the
// elements >= T0 and sorts them (64-bit keys, value desc, id asc).  Then
// (popular-science article on arXiv 2605.20104, section 二 third gear): a row
// writes C[its token] when no later row in (request, slot) order carries the
// same token, and the warp that completes the last valid row of a request
// (atomic ticket) runs its greedy acceptance.
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;

constexpr int CCAP = 256;          // shared 64-bit words per warp
constexpr int ECAP = 192;          // candidate elements per row
constexpr int UCAP = 2 * (CCAP - ECAP);  // candidate units per row (int ids after the keys)
constexpr int UB = 16;             // candidate units loaded at once per lane

constexpr int SW = 8;  // pass-2 warps per CTA

constexpr int NQ = TWO_PASS_MAX_UNITS / 128;  // float4 unit-maxima loads per lane, all in flight

// Unit maxima of one row into registers: lane l holds units 4i..4i+3 for
// i = l, l + 32, ...; units past the row's last and NaN maxima (flagged by
// pass 1) read as -inf.  Returns the lane's maximum.
__device__ __forceinline__ float load_unit_maxima(const float4* um4, int upr, bool live, int lane, float4 (&y)[NQ]) {
  const int n4 = (upr + 3) >> 2;
  float lmax = -INFINITY;
#pragma unroll
  for (int k = 0; k < NQ; ++k) {
    const int i4 = k * 32 + lane;
    y[k] = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    if (live && i4 < n4) y[k] = __ldcg(um4 + i4);
  }
#pragma unroll
  for (int k = 0; k < NQ; ++k) {
    const int u = 4 * (k * 32 + lane);
    y[k].x = (y[k].x == y[k].x) ? y[k].x : -INFINITY;
    y[k].y = (y[k].y == y[k].y && u + 1 < upr) ? y[k].y : -INFINITY;
    y[k].z = (y[k].z == y[k].z && u + 2 < upr) ? y[k].z : -INFINITY;
    y[k].w = (y[k].w == y[k].w && u + 3 < upr) ? y[k].w : -INFINITY;
    lmax = fmaxf(lmax, fmaxf(fmaxf(y[k].x, y[k].y), fmaxf(y[k].z, y[k].w)));
  }
  return lmax;
}

// Exact top-8 of one row (one warp; lanes 0..7 return its keys, descending)
// from the row's unit maxima y / lane maximum lmax:
//   1. T0 = the 8th largest lane maximum.  Eight distinct elements (one per
//      lane holding such a maximum) reach T0, so every element of the row's
//      top-8 is >= T0 and lies in a unit whose maximum is >= T0;
//   2. those units are listed in shared memory (`list`: CCAP words);
//   3. they are read again (UB loads in flight per lane) and every element
//      >= T0 is appended: per-lane bit masks, one warp scan for the offsets,
//      then each lane writes its own (about one element per candidate unit);
//   4. the candidates are sorted (64-bit keys, value desc, id asc).
// With the units' second largest elements and maxima positions (pass 1 with
// top2: um / us / up, the row's unit records), a candidate unit whose second
// largest element is below T0 holds exactly one element >= T0, its maximum,
// whose key comes from the records; only the other candidates are read again.
// Heavy ties at the top (more candidates than the list holds) and rows of
// fewer than eight finite unit maxima take the exact rescan.  `overlap()` is
// called exactly once: while the candidate loads are in flight, or before the
// rescan.
template <int DT, class F>
__device__ __forceinline__ u64 select_top8(const float4 (&y)[NQ], float lmax, const uint4* rowv, const char* rowp,
                                           int64_t nslot, int tail, u64* list, int lane, uint32_t* err,
                                           const float* um, const float* us, const uint8_t* up, F&& overlap) {
  constexpr int EPL = Vec16<DT>::EPL;
  const unsigned lt = (1u << lane) - 1u;
  bool overlapped = false;
  const float T0 = eighth_of_lanes(lmax, lane);
  bool overflow = !(T0 > -INFINITY);  // fewer than 8 finite unit maxima: tiny or -inf rows
  u64 top = 0ull;
  if (!overflow) {
    int* ulist = reinterpret_cast<int*>(list + ECAP);
    int cu = 0;
#pragma unroll
    for (int k = 0; k < NQ; ++k)
      cu += (y[k].x >= T0) + (y[k].y >= T0) + (y[k].z >= T0) + (y[k].w >= T0);
    int incl = cu;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int z = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += z;
    }
    const int nu = __shfl_sync(FULL, incl, 31);
    overflow = nu > UCAP;  // heavy ties at the top: exact rescan below
    if (!overflow && cu > 0) {
      int off = incl - cu;
#pragma unroll
      for (int k = 0; k < NQ; ++k) {
        const int u = 4 * (k * 32 + lane);
        if (y[k].x >= T0) ulist[off++] = u;
        if (y[k].y >= T0) ulist[off++] = u + 1;
        if (y[k].z >= T0) ulist[off++] = u + 2;
        if (y[k].w >= T0) ulist[off++] = u + 3;
      }
    }
    __syncwarp();
    int nc = 0;
    int nr = nu;  // units to read again
    if (us && !overflow) {
      // single-element units give their key from the records (units of 32
      // lanes x EPL elements); the others are compacted in place for the reload
      nr = 0;
      for (int base = 0; base < nu; base += 32) {
        const int q = base + lane;
        int u = 0;
        float mx = 0.f, sx = 0.f;
        int ps = 0;
        if (q < nu) {
          u = ulist[q];
          mx = __ldcg(um + u);
          sx = __ldcg(us + u);
          ps = __ldcg(up + u);
        }
        if (!overlapped) { overlap(); overlapped = true; }
        __syncwarp();
        const bool multi = q < nu && !(sx < T0);
        const bool single = q < nu && !multi;
        const unsigned bs = __ballot_sync(FULL, single), bm = __ballot_sync(FULL, multi);
        if (single) list[nc + __popc(bs & lt)] = make_key(mx, u * (32 * EPL) + ps);
        if (multi) ulist[nr + __popc(bm & lt)] = u;
        nc += __popc(bs);
        nr += __popc(bm);
        __syncwarp();
      }
    }
    for (int base = 0; base < nr && !overflow; base += UB) {
      Vec16<DT> v[UB];
      int32_t sl[UB];
      unsigned mq[UB];
#pragma unroll
      for (int q = 0; q < UB; ++q) {
        sl[q] = -1;
        if (base + q < nr) {
          const int32_t s = ulist[base + q] * 32 + lane;
          if (s < nslot) { sl[q] = s; v[q].r = __ldcg(rowv + s); }
        }
      }
      if (!overlapped) { overlap(); overlapped = true; }
      const int nq = min(UB, nr - base);  // candidates in this batch (warp-uniform)
      int cnt = 0;
#pragma unroll
      for (int q = 0; q < UB; ++q) {
        if (q >= nq) break;
        mq[q] = sl[q] >= 0 ? v[q].ge_mask(T0) : 0u;
        cnt += __popc(mq[q]);
      }
      int inc = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int z = __shfl_up_sync(FULL, inc, o);
        if (lane >= o) inc += z;
      }
      const int total = __shfl_sync(FULL, inc, 31);
      if (nc + total > ECAP) { overflow = true; break; }
      int off = nc + inc - cnt;
#pragma unroll
      for (int q = 0; q < UB; ++q) {
        if (q >= nq) break;
        unsigned m = mq[q];
        while (m) {
          const int e = __ffs(m) - 1;
          m &= m - 1;
          list[off++] = make_key(v[q].elem(e), sl[q] * EPL + e);
        }
      }
      nc += total;
    }
    if (!overflow) {
      // the row's last V % EPL elements are not in any unit
      bool c = false;
      float x = 0.f;
      const int32_t id = (int32_t)(nslot * EPL + lane);
      if (lane < tail) {
        x = load_scalar<DT>(rowp, id);
        if (x != x) atomicOr(err, GRAFT_ERR_NAN);
        else c = x >= T0;
      }
      const unsigned bm = __ballot_sync(FULL, c);
      const int pos = nc + __popc(bm & lt);
      if (c && pos < ECAP) list[pos] = make_key(x, id);
      nc += __popc(bm);
      overflow = nc > ECAP;
    }
    __syncwarp();
    if (!overflow) {
      if (nc <= 16) top = bitonic_desc<16>(lane < nc ? list[lane] : 0ull, lane);
      else if (nc <= 32) top = bitonic_desc<32>(lane < nc ? list[lane] : 0ull, lane);
      else top = warp_merge_ool(0ull, list, nc, lane);
    }
  }
  if (!overlapped) overlap();
  if (overflow) top = exact_row<DT>(rowv, nslot, rowp, tail, lane);  // ties, tiny rows: exact rescan
  return top;
}

template <int DT>
__global__ void __launch_bounds__(SW * 32) k_select(VerifyArgs a, int32_t* C) {
  __shared__ u64 cand[SW][CCAP];
  __shared__ int32_t stok[TWO_PASS_MAX_ROWS];
  __shared__ uint64_t smask[SW * MAX_S];  // tree arrays of the requests this CTA's rows belong to
  __shared__ int32_t spos[SW * MAX_S];
  __shared__ int8_t spar[SW * MAX_S];
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rows = a.batch * a.S;  // the host keeps rows <= TWO_PASS_MAX_ROWS
  const int row = blockIdx.x * SW + warp;
  const bool live = row < rows;
  const ScanGeom& g = a.g;
  const int64_t nslot = g.nslot;
  const int upr = a.upr;
  const char* rowp = reinterpret_cast<const char*>(a.logits) + (size_t)(live ? row : 0) * (size_t)g.stride * ES;
  const uint4* rowv = reinterpret_cast<const uint4*>(rowp);
  const float4* um4 = reinterpret_cast<const float4*>(a.umax + (size_t)(live ? row : 0) * a.ups);
  u64* list = cand[warp];
  // a dependent grid (the stochastic walk, which reads none of this kernel's
  // results) may be scheduled beside this one
  grid_dependents_launch();

  // the tree tokens of all rows (last-writer test, request sizes); written
  // before pass 1 started, so read before waiting for it
#pragma unroll 8
  for (int r = threadIdx.x; r < rows; r += SW * 32) stok[r] = __ldcg(a.tree_tok + r);
  // the other tree arrays of the (at most SW) requests this CTA's rows belong
  // to, for the acceptance of whichever of them completes here
  const int b_lo = min(blockIdx.x * SW, rows - 1) / a.S;
  const int b_hi = (min(blockIdx.x * SW + SW, rows) - 1) / a.S;
  {
    const int n_st = (b_hi - b_lo + 1) * a.S, r0 = b_lo * a.S;
    for (int i = threadIdx.x; i < n_st; i += SW * 32) {
      spar[i] = __ldcg(a.tree_parent + r0 + i);
      spos[i] = __ldcg(a.tree_pos + r0 + i);
      smask[i] = __ldcg(reinterpret_cast<const unsigned long long*>(a.tree_mask) + r0 + i);
    }
  }

  // the row's unit maxima (pass 1's results), then its exact top-8
  grid_dependency_wait();
  float4 y[NQ];
  const float lmax = load_unit_maxima(um4, upr, live, lane, y);
  __syncthreads();
  // requests with no valid slot have no row to finish them
  if (warp == 0 && !a.sample)
    for (int b = blockIdx.x; b < a.batch; b += gridDim.x)
      if (request_valid(a, stok, b, lane) == 0) accept_request(a, b, lane, stok);
  if (!live) return;
  const int32_t tok = stok[row];
  if (tok < 0 || tok >= g.V) return;

  // last-writer test and request size: shared-memory work, done while the
  // candidate units are in flight (or before the exact rescan)
  bool later = false;
  int nv = 0;
  auto writer_and_size = [&]() {
#pragma unroll 4
    for (int r = row + 1 + lane; r < rows; r += 32) later |= stok[r] == tok;
    later = __any_sync(FULL, later);
    nv = request_valid(a, stok, row / a.S, lane);
  };
  const size_t urow = (size_t)row * a.ups;
  const u64 top = select_top8<DT>(y, lmax, rowv, rowp, nslot, g.tail, list, lane, a.err, a.umax + urow,
                                  a.top2 ? a.usec + urow : nullptr, a.top2 ? a.upos + urow : nullptr,
                                  writer_and_size);
  const int32_t id = key_id(top);
  if (lane < K) a.topk[(size_t)row * K + lane] = id;

  // matrix update: this row is its token's last writer unless a later row
  //    (in (request, slot) order) carries the same token
  if (!later && lane < K) st_keep(C + (size_t)tok * K + lane, id, l2_keep_policy());

  // the warp that completes the request's last valid row runs acceptance:
  //    the warp's writes are released by lane 0's ticket increment, and the
  //    last incrementer acquires every other row's (stochastic verification
  //    accepts in its own kernel)
  if (a.sample) return;
  __syncwarp();
  const int b = row / a.S;
  int t = 0;
  if (lane == 0) t = ticket_acq_rel(&a.req_ticket[b]);
  t = __shfl_sync(FULL, t, 0);
  if (t == nv - 1) {
    if (lane == 0) a.req_ticket[b] = 0;
    __syncwarp();
    const int o = (b - b_lo) * a.S;
    accept_staged(a, b, lane, stok, spar + o, spos + o, smask + o);
  }
}

template <int DT>
cudaError_t select_impl(const VerifyArgs& a, int32_t* C, cudaStream_t s) {
  const int rows = a.batch * a.S;
  // programmatic dependent launch: pass 2's CTAs start as pass 1's leave the
  // SMs, load the tree tokens, then wait for pass 1's unit maxima
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((rows + SW - 1) / SW);
  cfg.blockDim = dim3(SW * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_select<DT>, a, C);
}

// Warm-up (article section 六): the rows named by the listing kernel (the
// last occurrence of each token, so at most one row per token) write their
// token's matrix row with their top-8; pass 1 stored their unit maxima by list
// position.  A persistent grid of warps walks the first min(*count, cap)
// entries.
template <int DT>
__global__ void __launch_bounds__(SW * 32) k_warm_select(VerifyArgs a, const int32_t* tokens, const int32_t* list,
                                                       const int32_t* count, int cap, int32_t* C) {
  __shared__ u64 cand[SW][CCAP];
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  u64* lst = cand[warp];
  grid_dependency_wait();  // the unit maxima come from pass 1 (the list from the kernels before it)
  const int n = min(__ldcg(count), cap);
  const uint64_t keep = l2_keep_policy();
  for (int k = blockIdx.x * SW + warp; k < n; k += gridDim.x * SW) {
    const int32_t row = __ldcg(list + k);
    const int32_t tok = __ldcg(tokens + row);
    const char* rowp = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)a.g.stride * ES;
    const float4* um4 = reinterpret_cast<const float4*>(a.umax + (size_t)k * a.ups);
    float4 y[NQ];
    const float lmax = load_unit_maxima(um4, a.upr, true, lane, y);
    const size_t urow = (size_t)k * a.ups;
    const u64 top = select_top8<DT>(y, lmax, reinterpret_cast<const uint4*>(rowp), rowp, a.g.nslot, a.g.tail, lst,
                                    lane, a.err, a.umax + urow, a.top2 ? a.usec + urow : nullptr,
                                    a.top2 ? a.upos + urow : nullptr, [] {});
    if (lane < K) st_keep(C + (size_t)tok * K + lane, key_id(top), keep);
    __syncwarp();  // the candidate list is reused by the warp's next row
  }
}

template <int DT>
cudaError_t warm_select_impl(const VerifyArgs& a, const int32_t* tokens, const int32_t* list, const int32_t* count,
                             int cap, int32_t* C, int grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(SW * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_warm_select<DT>, a, tokens, list, count, cap, C);
}

}  // namespace

cudaError_t launch_two_pass_select(const VerifyArgs& a, int dtype, int32_t* C, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? select_impl<GRAFT_BF16>(a, C, s) : select_impl<GRAFT_F32>(a, C, s);
}

cudaError_t launch_warm_select(const VerifyArgs& a, const int32_t* tokens, const int32_t* list, const int32_t* count,
                               int cap, int32_t* C, int dtype, int grid, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? warm_select_impl<GRAFT_BF16>(a, tokens, list, count, cap, C, grid, s)
                             : warm_select_impl<GRAFT_F32>(a, tokens, list, count, cap, C, grid, s);
}

}  // namespace graft
