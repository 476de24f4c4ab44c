// Pass 1 of the two-pass verify scan (the default path for 16-byte aligned
// rows): unit maxima.
//
// The verify + update pass of a Graft step (popular-science article on arXiv
// 2605.20104, section 二 third gear) needs the top-8 of every verified slot's
// logits row.  Selection work on the streaming path costs memory parallelism,
// so this kernel only streams: a persistent grid reads the valid rows once, in
// equal contiguous slices, with 16-byte evict-first loads, and writes the
// maximum of every 512-byte unit (32 lanes x 16 bytes), 1/128 of the bytes
// read.  No shared state and no barriers on the stream.  Pass 2 (select.cu)
// then finds each row's top-8 from its unit maxima.  The warm-up (article
// section 六) runs the same pass over the rows its listing kernel names: the
// last occurrence of each token.
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "scan_common.cuh"

namespace graft {
namespace {
using namespace scan;

constexpr int UT = 256;            // threads per CTA
constexpr int UMAXROWS = 192;      // rows one CTA's slice may touch
constexpr int UW = UT / 32;
constexpr int UNV = 8;             // units (one 16-byte load per lane each) per warp iteration

__device__ __forceinline__ uint4 neg_inf_vec(int dt) {
  const uint32_t w = dt == GRAFT_BF16 ? 0xFF80FF80u : 0xFF800000u;
  return make_uint4(w, w, w, w);
}

// LIST = false: the valid rows of the verified trees (token in [0, V)), unit
// records stored by row.  LIST = true (the warm-up): the first min(*count,
// cap) rows named by `list`, unit records stored by list position.
// TOP2 = true: besides its maximum, each unit records its second largest
// element (the largest of the others) and the position of its maximum in the
// unit (the lowest on ties), so pass 2 can take a unit with one element at or
// above its threshold without reading the unit again.
template <int DT, bool LIST, bool TOP2>
__global__ void __launch_bounds__(UT, 4) k_umax(VerifyArgs a, const int32_t* list, const int32_t* count, int cap) {
  __shared__ int warpsum[UW];
  __shared__ int rowlist[UMAXROWS];
  grid_dependents_launch();  // pass 2 may be scheduled as SMs free up; it waits for this grid's results
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const ScanGeom& g = a.g;
  const int rows = LIST ? 0 : a.batch * a.S;
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
  if (LIST) total = min(__ldcg(count), cap);
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
  if (LIST) {
    for (int64_t k = k0 + tid; k <= klast; k += UT) rowlist[k - k0] = __ldcg(list + k);
  } else {
    int64_t vidx = wbase + incl - cnt;
    for (int r = r0; r < r1; ++r) {
      const int32_t t = a.tree_tok[r];
      if (t >= 0 && t < g.V) {
        if (vidx >= k0 && vidx <= klast) rowlist[vidx - k0] = r;
        ++vidx;
      }
    }
  }
  __syncthreads();

  for (int64_t k = k0; k <= klast; ++k) {
    const int row = rowlist[k - k0];
    const int64_t ulo = max(u0, k * upr) - k * upr, uhi = min(u1, (k + 1) * upr) - k * upr;
    const uint4* rowv = reinterpret_cast<const uint4*>(reinterpret_cast<const char*>(a.logits) +
                                                       (size_t)row * (size_t)g.stride * ES);
    float* um = a.umax + (size_t)(LIST ? k : row) * a.ups;
    float* us = TOP2 ? a.usec + (size_t)(LIST ? k : row) * a.ups : nullptr;
    uint8_t* up = TOP2 ? a.upos + (size_t)(LIST ? k : row) * a.ups : nullptr;
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
      if (!TOP2) {
#pragma unroll
        for (int kk = 0; kk < UNV; ++kk) {
          const float m = v[kk].vmax();
          if (m != m) atomicOr(a.err, GRAFT_ERR_NAN);
          const int32_t mi = __reduce_max_sync(FULL, ord_int(m));
          if (lane == kk && ub + kk < uhi) um[ub + kk] = from_ord_int(mi);
        }
      } else {
        // per unit: the maximum (warp reduction), the lowest lane holding it,
        // the largest of everything else (that lane's second, the other
        // lanes' maxima), and that lane's 16 bytes, handed to lane kk
        float mk = 0.f, sk = 0.f;
        int wk = 0;
        Vec16<DT> ck;
        ck.r = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int kk = 0; kk < UNV; ++kk) {
          float m1, m2;
          v[kk].top2(m1, m2);
          if (m1 != m1) atomicOr(a.err, GRAFT_ERR_NAN);
          const int32_t k1 = ord_int(m1);
          const int32_t mi = __reduce_max_sync(FULL, k1);
          const unsigned wm = __ballot_sync(FULL, k1 == mi);
          const int w = __ffs(wm) - 1;
          const int32_t xi = __reduce_max_sync(FULL, lane == w ? ord_int(m2) : k1);
          uint4 r;
          r.x = __shfl_sync(FULL, v[kk].r.x, w);
          r.y = __shfl_sync(FULL, v[kk].r.y, w);
          r.z = __shfl_sync(FULL, v[kk].r.z, w);
          r.w = __shfl_sync(FULL, v[kk].r.w, w);
          if (lane == kk) {
            mk = from_ord_int(mi);
            sk = (wm & (wm - 1u)) ? mk : from_ord_int(xi);  // the maximum held by two lanes: it repeats
            wk = w;
            ck.r = r;
          }
        }
        if (lane < UNV && ub + lane < uhi) {
          const unsigned em = ck.ge_mask(mk);  // the maximum's elements in lane wk's 16 bytes
          um[ub + lane] = mk;
          us[ub + lane] = sk;
          up[ub + lane] = (uint8_t)(wk * Vec16<DT>::EPL + (em ? __ffs(em) - 1 : 0));
        }
      }
    }
  }
}

template <int DT, bool LIST>
cudaError_t umax_impl(const VerifyArgs& a, const int32_t* list, const int32_t* count, int cap, int grid,
                      cudaStream_t s) {
  if (a.top2) k_umax<DT, LIST, true><<<grid, UT, 0, s>>>(a, list, count, cap);
  else k_umax<DT, LIST, false><<<grid, UT, 0, s>>>(a, list, count, cap);
  return cudaGetLastError();
}

}  // namespace

int two_pass_ctas_per_sm() { return 4; }
int two_pass_max_rows(int grid) { return min(TWO_PASS_MAX_ROWS, (UMAXROWS - 2) * grid); }

cudaError_t launch_two_pass_umax(const VerifyArgs& a, int dtype, int grid, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? umax_impl<GRAFT_BF16, false>(a, nullptr, nullptr, 0, grid, s)
                             : umax_impl<GRAFT_F32, false>(a, nullptr, nullptr, 0, grid, s);
}

cudaError_t launch_warm_umax(const VerifyArgs& a, const int32_t* list, const int32_t* count, int cap, int dtype,
                             int grid, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? umax_impl<GRAFT_BF16, true>(a, list, count, cap, grid, s)
                             : umax_impl<GRAFT_F32, true>(a, list, count, cap, grid, s);
}

}  // namespace graft
