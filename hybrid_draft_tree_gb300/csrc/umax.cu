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
// then finds each row's top-8 from its unit maxima.
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

template <int DT>
__global__ void __launch_bounds__(UT, 4) k_umax(VerifyArgs a) {
  __shared__ int warpsum[UW];
  __shared__ int rowlist[UMAXROWS];
  grid_dependents_launch();  // pass 2 may be scheduled as SMs free up; it waits for this grid's results
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
    float* um = a.umax + (size_t)row * a.ups;
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

template <int DT>
cudaError_t umax_impl(const VerifyArgs& a, int grid, cudaStream_t s) {
  k_umax<DT><<<grid, UT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int two_pass_ctas_per_sm() { return 4; }
int two_pass_max_rows(int grid) { return min(TWO_PASS_MAX_ROWS, (UMAXROWS - 2) * grid); }

cudaError_t launch_two_pass_umax(const VerifyArgs& a, int dtype, int grid, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? umax_impl<GRAFT_BF16>(a, grid, s) : umax_impl<GRAFT_F32>(a, grid, s);
}

}  // namespace graft
