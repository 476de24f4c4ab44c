// Pass 1 of the two-pass verify scan (for 16-byte aligned rows): unit
// maxima.
//
// The verify + update pass of a Graft step (popular-science article on arXiv
// 2605.20104, section 二 third gear) needs the top-8 of every verified slot's
// logits row.  Selection work on the streaming path costs memory parallelism,
// so this kernel only streams: a persistent grid reads the valid rows once,
// in equal contiguous slices of units, with 16-byte evict-first loads, and
// writes the maximum of every 512-byte unit (32 lanes x 16 bytes), 1/128 of
// the bytes read.  No shared state and no barriers on the stream.
// Pass 2 (select.cu) then finds each row's top-8 from its unit maxima.  The
// warm-up (article section 六) runs the same pass over the rows its listing
// kernel names: the last occurrence of each token.
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

// This CTA's share: units [u0, u1) of the rows' NU = rows * upr units, which
// fall in compacted rows k0 .. klast (rowlist[k - k0] = the row behind k).
// NU <= 4096 rows x 1024 units (the warm-up's list: 4096 rows at most) fits
// in 32 bits.
struct Slice {
  int u0, u1, k0, klast;
  int live;  // 0: nothing to stream here (the whole CTA agrees)
};

constexpr int UCHUNKS = TWO_PASS_MAX_ROWS / UT;  // row chunks of UT, one row per thread each

// Thread 0's part: this CTA's slice of `total` compacted rows (equal shares
// of the units, the first NU % Ge CTAs one unit more).
__device__ __forceinline__ Slice slice_of(int total, int upr, const VerifyArgs& a) {
  Slice s{0, 0, 0, -1, 0};
  const int NU = total * upr;
  const int Ge = min((int)gridDim.x, NU);
  const int c = blockIdx.x;
  if (NU > 0 && c < Ge) {
    const int q = NU / Ge, rem = NU - q * Ge;
    s.u0 = c * q + min(c, rem);
    s.u1 = s.u0 + q + (c < rem ? 1 : 0);
    s.k0 = s.u0 / upr;
    s.klast = (s.u1 - 1) / upr;
    s.live = 1;
    if (s.klast - s.k0 + 1 > UMAXROWS) {  // the host keeps rows <= (UMAXROWS - 2) * grid
      atomicOr(a.err, GRAFT_ERR_TREE);
      s.live = 0;
    }
  }
  return s;
}

// Compacts the rows and fills `rowlist` for this CTA's slice (ends with a
// CTA barrier).  LIST = false: the valid tree rows, in row order: thread t
// tests rows t, t + UT, ... (all its loads issued at once), each warp counts
// its chunk's valid rows with a ballot, warp 0 scans the counts and thread 0
// takes the slice; a valid row's compacted index is its chunk-warp's prefix
// plus the valid lanes below it.  LIST = true: the first min(*count, cap)
// entries of `list`.  wpre: UCHUNKS * UW ints of shared memory.
template <bool LIST, int ES>
__device__ __forceinline__ Slice compact_rows(const VerifyArgs& a, const int32_t* list, const int32_t* count, int cap,
                                              int* rowlist, int* wpre, Slice* s_slice) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int upr = a.upr;
  if (LIST) {
    if (tid == 0) *s_slice = slice_of(min(__ldcg(count), cap), upr, a);
    __syncthreads();
    const Slice s = *s_slice;
    if (s.live)
      for (int k = s.k0 + tid; k <= s.klast; k += UT) rowlist[k - s.k0] = __ldcg(list + k);
    __syncthreads();
    return s;
  }
  const int rows = a.batch * a.S;  // <= TWO_PASS_MAX_ROWS on this path (the host checks)
  if (rows > TWO_PASS_MAX_ROWS) {
    if (tid == 0) atomicOr(a.err, GRAFT_ERR_TREE);
    return Slice{0, 0, 0, -1, 0};
  }
  const int V = a.g.V;
  const int nchunk = (rows + UT - 1) / UT;
  // the loops stop at nchunk (uniform): the loads still issue back to back
  int32_t tok[UCHUNKS];
#pragma unroll
  for (int i = 0; i < UCHUNKS; ++i) {
    if (i >= nchunk) break;
    tok[i] = i * UT + tid < rows ? a.tree_tok[i * UT + tid] : -1;
  }
  if (a.spec) {
    // every row expected valid (the compacted index is the row): while the
    // tree tokens are on their way, this warp's first group of the slice it
    // would then get is prefetched into L2 (a wrong guess costs one group of
    // reads per warp)
    const int NU = rows * upr, Ge = min((int)gridDim.x, NU), c = blockIdx.x;
    if (c < Ge) {
      const int q = NU / Ge, rem = NU - q * Ge;
      const int u0 = c * q + min(c, rem), u1 = u0 + q + (c < rem ? 1 : 0);
      const int u = u0 + warp * UNV;
      int row = u / upr, j = u - row * upr;
      const char* base = reinterpret_cast<const char*>(a.logits);
      const size_t rstride = (size_t)a.g.stride * ES;
#pragma unroll
      for (int kk = 0; kk < UNV; ++kk) {
        if (u + kk < u1) {
          const int64_t sl = (int64_t)j * 32 + lane;
          if (sl < a.g.nslot) prefetch_l2(base + (size_t)row * rstride + (size_t)sl * 16);
        }
        if (++j == upr) {
          j = 0;
          ++row;
        }
      }
    }
  }
  unsigned vm = 0;  // bit i: row i * UT + tid is valid
#pragma unroll
  for (int i = 0; i < UCHUNKS; ++i) {
    if (i >= nchunk) break;
    const bool ok = tok[i] >= 0 && tok[i] < V;
    if (tok[i] >= V && blockIdx.x == 0) atomicOr(a.err, GRAFT_ERR_TOKEN);  // such a slot is skipped
    const unsigned b = __ballot_sync(FULL, ok);
    if (lane == 0) wpre[i * UW + warp] = __popc(b);
    vm |= (ok ? 1u : 0u) << i;
  }
  __syncthreads();
  if (warp == 0) {
    // exclusive prefix of the nchunk * UW counts, 4 consecutive per lane
    const int n = nchunk * UW;
    int c4[4], sum = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      c4[q] = (lane * 4 + q < n) ? wpre[lane * 4 + q] : 0;
      sum += c4[q];
    }
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL, incl, o);
      if (lane >= o) incl += y;
    }
    int run = incl - sum;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (lane * 4 + q < n) wpre[lane * 4 + q] = run;
      run += c4[q];
    }
    const int total = __shfl_sync(FULL, incl, 31);
    if (lane == 0) *s_slice = slice_of(total, upr, a);
  }
  __syncthreads();
  const Slice s = *s_slice;
  if (s.live) {
    const unsigned below = (1u << lane) - 1u;
#pragma unroll 1
    for (int i = 0; i < nchunk; ++i) {
      const bool ok = (vm >> i) & 1u;
      const unsigned b = __ballot_sync(FULL, ok);
      const int vidx = wpre[i * UW + warp] + __popc(b & below);
      if (ok && vidx >= s.k0 && vidx <= s.klast) rowlist[vidx - s.k0] = i * UT + tid;
    }
  }
  __syncthreads();
  return s;
}

// Streams this CTA's slice.  The slice's units are dealt to the warps in
// groups of UNV as one flat sequence, across row boundaries: warp w takes
// groups w, w + UW, ..., so the warps' shares differ by one group at most
// (a loop per row would give each warp its own remainder at every row end).
// A group inside one row is read with straight loads; a group that crosses a
// row end (or the slice end) locates each unit on its own.  Unit records go
// to row `row` (LIST = false) or list position k (LIST = true) of a.umax
// (and, with TOP2, a.usec / a.upos: besides its maximum, each unit records
// its second largest element, the largest of the others, and the position of
// its maximum in the unit, the lowest on ties, so pass 2 can take a unit with
// one element at or above its threshold without reading the unit again).
template <int DT, bool LIST, bool TOP2>
__device__ __forceinline__ void stream_units(const VerifyArgs& a, const Slice& sl, const int* rowlist, int warp,
                                             int lane) {
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const ScanGeom& g = a.g;
  const int64_t nslot = g.nslot;
  const char* base = reinterpret_cast<const char*>(a.logits);
  const size_t rstride = (size_t)g.stride * ES;
  const int nu = sl.u1 - sl.u0;
  const int upr32 = a.upr;  // <= TWO_PASS_MAX_UNITS
  // the group's first unit as (compacted row k, unit j of that row), walked
  // forward from the slice's first unit
  int64_t k = sl.k0;
  int j = sl.u0 - sl.k0 * upr32 + warp * UNV;
  while (j >= upr32) {
    j -= upr32;
    ++k;
  }
  for (int g0 = warp * UNV; g0 < nu; g0 += UW * UNV) {
    const bool one_row = j + UNV <= upr32 && g0 + UNV <= nu;
    const int row0 = rowlist[k - sl.k0];
    // unit kk of the group: its compacted row kr, its row, its index jj in the row
    auto locate = [&](int kk, int64_t& kr, int& row, int64_t& jj) {
      if (one_row) {
        kr = k; row = row0; jj = j + kk;
      } else {
        kr = min(k + (j + kk) / upr32, (int64_t)sl.klast);  // units past the slice end are masked out
        jj = (j + kk) % upr32;
        row = rowlist[kr - sl.k0];
      }
    };
    Vec16<DT> v[UNV];
    if (one_row && (j + UNV) * 32 <= nslot) {
      const uint4* rowv = reinterpret_cast<const uint4*>(base + (size_t)row0 * rstride);
#pragma unroll
      for (int kk = 0; kk < UNV; ++kk) v[kk].r = __ldcs(rowv + (j + kk) * 32 + lane);
    } else {
#pragma unroll
      for (int kk = 0; kk < UNV; ++kk) {
        int64_t kr, jj;
        int row;
        locate(kk, kr, row, jj);
        const int64_t s = jj * 32 + lane;
        v[kk].r = (g0 + kk < nu && s < nslot)
                      ? __ldcs(reinterpret_cast<const uint4*>(base + (size_t)row * rstride) + s)
                      : neg_inf_vec(DT);
      }
    }
    // lane kk stores unit kk's records
    int64_t kr_l = 0, jj_l = 0;
    int row_l = 0;
    const bool st = lane < UNV && g0 + lane < nu;
    if (st) locate(lane, kr_l, row_l, jj_l);
    const size_t rec = (size_t)(LIST ? kr_l : row_l) * a.ups + jj_l;
    if (!TOP2) {
      float mk = 0.f;
#pragma unroll
      for (int kk = 0; kk < UNV; ++kk) {
        const float m = v[kk].vmax();
        if (m != m) atomicOr(a.err, GRAFT_ERR_NAN);
        const int32_t mi = __reduce_max_sync(FULL, ord_int(m));
        if (lane == kk) mk = from_ord_int(mi);
      }
      if (st) a.umax[rec] = mk;
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
      if (st) {
        const unsigned em = ck.ge_mask(mk);  // the maximum's elements in lane wk's 16 bytes
        a.umax[rec] = mk;
        a.usec[rec] = sk;
        a.upos[rec] = (uint8_t)(wk * Vec16<DT>::EPL + (em ? __ffs(em) - 1 : 0));
      }
    }
    j += UW * UNV;
    while (j >= upr32) {
      j -= upr32;
      ++k;
    }
  }
}


// LIST = false: the valid rows of the verified trees, unit records stored by
// row.  LIST = true (the warm-up): the first min(*count, cap) rows named by
// `list`, unit records stored by list position.  TOP2: units also record
// their second largest element and the position of their maximum.
template <int DT, bool LIST, bool TOP2>
__global__ void __launch_bounds__(UT, 4) k_umax(VerifyArgs a, const int32_t* list, const int32_t* count, int cap) {
  __shared__ int wpre[UCHUNKS * UW];
  __shared__ int rowlist[UMAXROWS];
  __shared__ Slice s_slice;
  grid_dependents_launch();  // pass 2 may be scheduled as SMs free up; it waits for this grid's results
  if (LIST) grid_dependency_wait();  // the warm-up's list comes from the kernel ahead
  const Slice sl = compact_rows<LIST, DT == GRAFT_BF16 ? 2 : 4>(a, list, count, cap, rowlist, wpre, &s_slice);
  if (!sl.live) return;
  stream_units<DT, LIST, TOP2>(a, sl, rowlist, threadIdx.x >> 5, threadIdx.x & 31);
}

template <int DT, bool LIST>
cudaError_t umax_impl(const VerifyArgs& a, const int32_t* list, const int32_t* count, int cap, int grid,
                      cudaStream_t s) {
  if (LIST)  // the warm-up: a programmatic dependent of its listing kernel
    return a.top2 ? launch_dependent(k_umax<DT, LIST, true>, dim3(grid), dim3(UT), 0, s, a, list, count, cap)
                  : launch_dependent(k_umax<DT, LIST, false>, dim3(grid), dim3(UT), 0, s, a, list, count, cap);
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
