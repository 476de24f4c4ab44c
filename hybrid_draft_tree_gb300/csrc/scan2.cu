// Two-pass verify scan for 16-byte aligned logits rows (the default path).
//
// The verify + update pass of a Graft step (popular-science article on arXiv
// 2605.20104, section 二 third gear) needs, for every verified slot, the top-8
// of its logits row (element 0 = the greedy argmax).  Selection work on the
// streaming path costs memory parallelism, so it is moved off it:
//
// Pass 1 (k_umax): a persistent grid streams the valid rows once, in equal
//   contiguous slices, with 16-byte evict-first loads, and writes only the
//   maximum of every 512-byte unit (32 lanes x 16 bytes): 1/128 of the bytes
//   read.  No shared state, no barriers on the stream.
// Pass 2 (k_select): one warp per row reads the row's unit maxima.  The 8th
//   largest of them, T, is reached by 8 distinct elements, so every element of
//   the row's top-8 is >= T and lies in a unit whose maximum is >= T.  The
//   warp re-reads only those units (about 8 of ~600 for V = 151936), keeps
//   the elements >= T and sorts them (64-bit keys, value desc, id asc).
// The request kernel (k_finish) then runs acceptance and the matrix update.
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;

constexpr int UT = 256;            // pass-1 threads per CTA
constexpr int UW = UT / 32;
constexpr int UNV = 4;             // units (one 16-byte load per lane each) per warp iteration
constexpr int UMAXROWS = 192;
constexpr int MPL = TWO_PASS_MAX_UNITS / 32;  // unit maxima per lane in pass 2
constexpr int CCAP = 256;          // candidate keys per warp in pass 2

__device__ __forceinline__ uint4 neg_inf_vec(int dt) {
  const uint32_t w = dt == GRAFT_BF16 ? 0xFF80FF80u : 0xFF800000u;
  return make_uint4(w, w, w, w);
}

// ---- pass 1: unit maxima -----------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(UT, 4) k_umax(VerifyArgs a) {
  __shared__ int warpsum[UW];
  __shared__ int rowlist[UMAXROWS];
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const ScanGeom& g = a.g;
  const int rows = a.batch * a.S;
  const int64_t nslot = g.nslot;
  const int64_t upr = a.upr;

  // compact the valid rows (same result in every CTA)
  const int per = (rows + UT - 1) / UT;
  const int r0 = min(tid * per, rows), r1 = min(r0 + per, rows);
  int cnt = 0;
  for (int r = r0; r < r1; ++r) {
    const int32_t t = a.tree_tok[r];
    cnt += (t >= 0 && t < g.V);
    if (t >= g.V && blockIdx.x == 0) atomicOr(a.err, GRAFT_ERR_TOKEN);  // such a slot is skipped
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warpsum[warp] = incl;
  __syncthreads();
  int wbase = 0, total = 0;
#pragma unroll
  for (int w = 0; w < UW; ++w) {
    const int x = warpsum[w];
    wbase += (w < warp) ? x : 0;
    total += x;
  }
  const int64_t NU = (int64_t)total * upr;
  if (NU == 0) return;
  const int Ge = (int)min((int64_t)gridDim.x, NU);
  const int c = blockIdx.x;
  if (c >= Ge) return;
  const int64_t u0 = (int64_t)c * NU / Ge, u1 = (int64_t)(c + 1) * NU / Ge;
  const int64_t k0 = u0 / upr, klast = (u1 - 1) / upr;
  if (klast - k0 + 1 > UMAXROWS) {  // the host keeps rows <= (UMAXROWS - 2) * grid
    if (tid == 0) atomicOr(a.err, GRAFT_ERR_TREE);
    return;
  }
  int64_t vidx = wbase + incl - cnt;
  for (int r = r0; r < r1; ++r) {
    const int32_t t = a.tree_tok[r];
    if (t >= 0 && t < g.V) {
      if (vidx >= k0 && vidx <= klast) rowlist[vidx - k0] = r;
      ++vidx;
    }
  }
  __syncthreads();

  for (int64_t k = k0; k <= klast; ++k) {
    const int row = rowlist[k - k0];
    const int64_t ulo = max(u0, k * upr) - k * upr, uhi = min(u1, (k + 1) * upr) - k * upr;
    const uint4* rowv = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(a.logits) +
                                                       (size_t)row * (size_t)g.stride * ES);
    float* um = a.umax + (size_t)row * upr;
    for (int64_t ub = ulo + (int64_t)warp * UNV; ub < uhi; ub += (int64_t)UW * UNV) {
      Vec16<DT> v[UNV];
      if (ub + UNV <= uhi && (ub + UNV) * 32 <= nslot) {
#pragma unroll
        for (int kk = 0; kk < UNV; ++kk) v[kk].r = __ldcs(rowv + (ub + kk) * 32 + lane);
      } else {
#pragma unroll
        for (int kk = 0; kk < UNV; ++kk) {
          const int64_t s = (ub + kk) * 32 + lane;
          v[kk].r = (ub + kk < uhi && s < nslot) ? __ldcs(rowv + s) : neg_inf_vec(DT);
        }
      }
#pragma unroll
      for (int kk = 0; kk < UNV; ++kk) {
        const float m = v[kk].vmax();
        if (m != m) atomicOr(a.err, GRAFT_ERR_NAN);
        const int32_t mi = __reduce_max_sync(FULL, ord_int(m));
        if (lane == kk && ub + kk < uhi) um[ub + kk] = from_ord_int(mi);
      }
    }
  }
}

// ---- pass 2: exact top-8 of each row from its candidate units ---------------------
template <int DT>
__device__ __noinline__ u64 exact_row(const uint4* rowv, int64_t nslot, const char* rowp, int tail, int lane) {
  constexpr int EPL = Vec16<DT>::EPL;
  u64 prev = ~0ull, out = 0ull;
  for (int r = 0; r < K; ++r) {
    u64 best = 0ull;
    for (int64_t s = lane; s < nslot; s += 32) {
      Vec16<DT> v;
      v.r = __ldcg(rowv + s);
#pragma unroll
      for (int e = 0; e < EPL; ++e) {
        const u64 key = make_key(v.elem(e), (int32_t)(s * EPL + e));
        if (key < prev && key > best) best = key;
      }
    }
    if (lane < tail) {
      const int32_t id = (int32_t)(nslot * EPL + lane);
      const u64 key = make_key(load_scalar<DT>(rowp, id), id);
      if (key < prev && key > best) best = key;
    }
    best = warp_max_u64(best);
    if (lane == r) out = best;
    prev = best;
  }
  return out;
}

constexpr int SW = 8;  // pass-2 warps per CTA

// Warp-aggregated append of this lane's keys (n of them, in keys[0..n)) to a
// per-warp list; returns the warp's total.  No atomics, no divergent loops.
__device__ __forceinline__ int warp_append(u64* list, int cap, int base, const u64* keys, int n, int lane) {
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += y;
  }
  const int off = base + incl - n;
  for (int i = 0; i < n; ++i)
    if (off + i < cap) list[off + i] = keys[i];
  return base + __shfl_sync(FULL, incl, 31);
}

template <int DT>
__global__ void __launch_bounds__(SW * 32) k_select(VerifyArgs a) {
  __shared__ u64 cand[SW][CCAP];
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  constexpr int EPL = Vec16<DT>::EPL;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * SW + warp;
  if (row >= a.batch * a.S) return;
  const int32_t tok = a.tree_tok[row];
  if (tok < 0 || tok >= a.g.V) return;
  const ScanGeom& g = a.g;
  const int64_t nslot = g.nslot;
  const int upr = a.upr;
  const char* rowp = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)g.stride * ES;
  const uint4* rowv = reinterpret_cast<const uint4*>(rowp);
  const float* um = a.umax + (size_t)row * upr;
  u64* list = cand[warp];

  // 1. unit maxima; T0 = 8th largest lane maximum: 8 distinct units reach it
  float m[MPL];
  float lmax = -INFINITY;
#pragma unroll
  for (int i = 0; i < MPL; ++i) {
    const int u = i * 32 + lane;
    const float x = u < upr ? __ldcg(um + u) : -INFINITY;
    m[i] = x == x ? x : -INFINITY;  // NaN rows were flagged by pass 1
    lmax = fmaxf(lmax, m[i]);
  }
  const float T0 = key_val(__shfl_sync(FULL, bitonic32_desc(make_key(lmax, lane), lane), K - 1));

  // 2. exact 8th largest unit maximum T, from the units >= T0 (value, unit) keys
  bool overflow = T0 == -INFINITY;  // fewer than 8 finite maxima
  u64 top = 0ull;
  int nu = 0;
  if (!overflow) {
    int n = 0, over = 0;
    u64 mine[K];
#pragma unroll
    for (int i = 0; i < MPL; ++i) {
      if (m[i] >= T0) {
        if (n < K) mine[n] = make_key(m[i], i * 32 + lane);
        n += 1;
      }
    }
    over = n > K;
    n = min(n, K);
    nu = warp_append(list, CCAP, 0, mine, n, lane);
    overflow = nu > CCAP || __any_sync(FULL, over);
  }
  float T = -INFINITY;
  if (!overflow) {
    __syncwarp();
    const u64 k8 = __shfl_sync(FULL, warp_merge_ool(0ull, list, nu, lane), K - 1);
    T = key_val(k8);
    // units with maximum >= T (the 8 largest and any tied with the 8th), as unit ids
    __syncwarp();
    int n = 0;
    int mine[4];
    for (int q = lane; q < nu && n < 4; q += 32) {
      const u64 key = list[q];
      if (key_val(key) >= T) mine[n++] = (int)(0xFFFFFFFFu - (uint32_t)key);
    }
    if (nu > 128) overflow = true;  // more than 4 candidate keys per lane: leave it to the exact rescan
    __syncwarp();
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += y;
    }
    const int nunits = __shfl_sync(FULL, incl, 31);
    int* ulist = reinterpret_cast<int*>(list + CCAP / 2);  // the upper half of the list is free now
    for (int i = 0; i < n; ++i) ulist[incl - n + i] = mine[i];
    __syncwarp();

    // 3. read those units (eight loads in flight per lane); keep elements >= T
    int nc = 0;
    for (int base = 0; base < nunits && !overflow; base += K) {
      Vec16<DT> v[K];
      int64_t sl[K];
#pragma unroll
      for (int q = 0; q < K; ++q) {
        sl[q] = -1;
        if (base + q < nunits) {
          const int64_t s = (int64_t)ulist[base + q] * 32 + lane;
          if (s < nslot) { sl[q] = s; v[q].r = __ldcg(rowv + s); }
        }
      }
#pragma unroll
      for (int q = 0; q < K; ++q) {
        u64 keys[EPL];
        int kn = 0;
        if (sl[q] >= 0 && v[q].vmax() >= T) {
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            const float x = v[q].elem(e);
            if (x >= T) keys[kn++] = make_key(x, (int32_t)(sl[q] * EPL + e));
          }
        }
        nc = warp_append(list, CCAP / 2, nc, keys, kn, lane);
      }
    }
    if (!overflow) {
      u64 keys[1];
      int kn = 0;
      if (lane < g.tail) {  // the row's last V % EPL elements
        const int32_t id = (int32_t)(nslot * EPL + lane);
        const float x = load_scalar<DT>(rowp, id);
        if (x != x) atomicOr(a.err, GRAFT_ERR_NAN);
        else if (x >= T) keys[kn++] = make_key(x, id);
      }
      nc = warp_append(list, CCAP / 2, nc, keys, kn, lane);
      __syncwarp();
      if (nc <= CCAP / 2) top = warp_merge_ool(0ull, list, nc, lane);
      else overflow = true;
    }
  }
  if (overflow) top = exact_row<DT>(rowv, nslot, rowp, g.tail, lane);  // ties, tiny rows: exact rescan
  if (lane < K) a.topk[(size_t)row * K + lane] = key_id(top);
}

template <int DT>
cudaError_t umax_impl(const VerifyArgs& a, int grid, cudaStream_t s) {
  k_umax<DT><<<grid, UT, 0, s>>>(a);
  return cudaGetLastError();
}
template <int DT>
cudaError_t select_impl(const VerifyArgs& a, cudaStream_t s) {
  const int rows = a.batch * a.S;
  k_select<DT><<<(rows + SW - 1) / SW, SW * 32, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int two_pass_ctas_per_sm() { return 4; }
int two_pass_max_rows(int grid) { return (UMAXROWS - 2) * grid; }

cudaError_t launch_two_pass_umax(const VerifyArgs& a, int dtype, int grid, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? umax_impl<GRAFT_BF16>(a, grid, s) : umax_impl<GRAFT_F32>(a, grid, s);
}
cudaError_t launch_two_pass_select(const VerifyArgs& a, int dtype, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? select_impl<GRAFT_BF16>(a, s) : select_impl<GRAFT_F32>(a, s);
}

}  // namespace graft
