// Persistent, TMA-pipelined verify scan for 16-byte aligned logits rows.
//
// The verify + update pass of a Graft step (popular-science article on arXiv
// 2605.20104, section 二 third gear) reads every verified slot's logits row
// once; this kernel streams those rows at HBM speed.
//
// Work: the valid rows are compacted in-kernel and cut into 32 KB chunks;
// CTA c of G (one per SM) owns the contiguous chunk range [cT/G, (c+1)T/G).
// Per CTA one producer thread issues cp.async.bulk copies (the 1-D TMA path)
// into a 6-stage shared-memory ring guarded by mbarriers (full: bytes landed;
// empty: all consumer warps done), keeping up to 192 KB in flight per SM.
// Each of the 8 consumer warps takes 1/8 of every chunk from shared memory
// and keeps its own running top-8 of the current row: elements below the
// warp's 8th best (or, while it has fewer than 8, below the 8th largest lane
// maximum of the chunk) are discarded with one compare per 16-byte vector;
// survivors are merged with a 32-lane bitonic sort on 64-bit keys (value
// desc, id asc).  At the end of a row segment the 8 warps' lists are merged;
// a row split over several CTAs is finished by the last of them (atomic
// ticket), which stages the row's top-8, claims the token's matrix row
// (atomicMax of row+1) and, if it completes its request, runs the acceptance
// walk.  Every wait is bounded: on expiry the kernel flags GRAFT_ERR_TIMEOUT,
// the producer stops issuing, waits for the copies it has in flight to land
// (a separate, far longer bound with a back-off: a bulk copy of 32 KB lands
// within microseconds) and the CTA finishes.  The consumers' and producer's
// poll limit is a launch argument, so a test can make the waits run out.
#include <cuda_bf16.h>

#include "graft_internal.cuh"
#include "scan_common.cuh"
#include "bulk_copy.cuh"

namespace graft {
namespace {
using namespace scan;
using namespace bulk;

constexpr int NCW = 8;                  // consumer warps
constexpr int NCT = NCW * 32;           // consumer threads
constexpr int TPB = NCT + 32;           // + one producer warp
constexpr int NSTAGE = 6;
constexpr int VPL = TMA_CHUNK / 16 / NCT;  // 16-byte vectors per consumer lane per chunk
constexpr int WCAP = 256;               // candidate keys per warp
constexpr int MAXROWS = 128;            // rows one CTA may touch

struct TmaSmem {
  u64 full[NSTAGE];
  u64 empty[NSTAGE];
  u64 wcand[NCW][WCAP];
  u64 segtop[2][NCW][K];
  int wcnt[NCW];
  int rowlist[MAXROWS];
  int warpsum[TPB / 32];
  int abort_flag;
};
constexpr size_t SMEM_BYTES = (size_t)NSTAGE * TMA_CHUNK + sizeof(TmaSmem);

__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(NCT) : "memory"); }

// CTA owning global chunk i when T chunks are split over G CTAs.
__device__ __forceinline__ int cta_of(int64_t i, int64_t T, int G) { return (int)(((i + 1) * G - 1) / T); }

template <int DT>
__device__ __forceinline__ u64 warp_exact_top8(const Vec16<DT>* v, int nvalid_mask, int64_t vbase, int vl0,
                                               bool has_tail, float tv, int32_t tail_id, u64 top, int lane) {
  constexpr int EPL = Vec16<DT>::EPL;
  u64 prev = ~0ull, out = 0ull;
  for (int r = 0; r < K; ++r) {
    u64 best = 0ull;
#pragma unroll
    for (int kk = 0; kk < VPL; ++kk) {
      if (nvalid_mask & (1 << kk)) {
        const int64_t vid = vbase + vl0 + kk * 32;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
          const u64 key = make_key(v[kk].elem(e), (int32_t)(vid * EPL + e));
          if (key < prev && key > best) best = key;
        }
      }
    }
    if (has_tail) {
      const u64 key = make_key(tv, tail_id);
      if (key < prev && key > best) best = key;
    }
    if (lane < K && top < prev && top > best) best = top;
    best = warp_max_u64(best);
    if (lane == r) out = best;
    prev = best;
  }
  return out;
}

template <int DT>
__global__ void __launch_bounds__(TPB, 1) k_verify_tma(VerifyArgs a) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* ring = smem_raw;
  TmaSmem& sm = *reinterpret_cast<TmaSmem*>(smem_raw + (size_t)NSTAGE * TMA_CHUNK);
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  constexpr int EPL = 16 / ES;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const ScanGeom& g = a.g;
  const uint32_t polls = a.wait_polls ? a.wait_polls : SPIN;
  const int S = a.S;
  const int rows = a.batch * S;
  const int G = gridDim.x, c = blockIdx.x;
  const int cpr = g.cpr;

  // ---- compact the valid rows (same result in every CTA) --------------------------
  const int per = (rows + TPB - 1) / TPB;
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
  if (lane == 31) sm.warpsum[warp] = incl;
  if (tid == 0) sm.abort_flag = 0;
  if (tid < NCW) sm.wcnt[tid] = 0;
  __syncthreads();
  int wbase = 0, total = 0;
#pragma unroll
  for (int w = 0; w < TPB / 32; ++w) {
    const int x = sm.warpsum[w];
    wbase += (w < warp) ? x : 0;
    total += x;
  }
  const int64_t T = (int64_t)total * cpr;
  const int64_t i0 = (int64_t)c * T / G, i1 = (int64_t)(c + 1) * T / G;
  const int64_t k0 = i0 / cpr;
  const int64_t klast = i1 > i0 ? (i1 - 1) / cpr : k0 - 1;
  int64_t vidx = wbase + incl - cnt;
  for (int r = r0; r < r1; ++r) {
    const int32_t t = a.tree_tok[r];
    if (t >= 0 && t < g.V) {
      if (vidx >= k0 && vidx <= klast && vidx - k0 < MAXROWS) sm.rowlist[vidx - k0] = r;
      ++vidx;
    }
  }
  if (tid == 0) {
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], NCW);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // requests without any valid slot have no row to finish them: CTA 0 does
  __syncthreads();
  if (i1 <= i0) return;
  if (klast - k0 + 1 > MAXROWS) {  // host keeps rows <= (MAXROWS - 2) * G, so this cannot happen
    if (tid == 0) atomicOr(a.err, GRAFT_ERR_TREE);
    return;
  }

  // ---- producer warp ------------------------------------------------------------
  if (warp == NCW) {
    if (lane == 0) {
      int64_t issued = 0;
      for (int64_t i = i0; i < i1; ++i) {
        const int64_t j = i - i0;
        const int s = (int)(j % NSTAGE);
        const uint32_t use = (uint32_t)(j / NSTAGE);
        if (use > 0 && !mbar_wait(&sm.empty[s], (use - 1) & 1, polls)) {
          atomicOr(a.err, GRAFT_ERR_TIMEOUT);
          *(volatile int*)&sm.abort_flag = 1;
          break;
        }
        if (*(volatile int*)&sm.abort_flag) break;
        const int64_t k = i / cpr;
        const int q = (int)(i % cpr);
        const int row = sm.rowlist[k - k0];
        const int64_t off = (int64_t)q * TMA_CHUNK;
        const uint32_t bytes = (uint32_t)min((int64_t)TMA_CHUNK, g.row_vec_bytes - off);
        const char* src = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)g.stride * ES + off;
        mbar_expect_tx(&sm.full[s], bytes);
        bulk_g2s(ring + (size_t)s * TMA_CHUNK, src, bytes, &sm.full[s]);
        ++issued;
      }
      // drain: every copy still in flight lands before this CTA may exit (the
      // stages of the last NSTAGE copies; a stage is reissued only after its
      // previous copy was consumed, or given up with the abort flag set first)
      for (int64_t j = issued > NSTAGE ? issued - NSTAGE : 0; j < issued; ++j)
        if (!mbar_wait_drain(&sm.full[j % NSTAGE], (uint32_t)(j / NSTAGE) & 1)) atomicOr(a.err, GRAFT_ERR_TIMEOUT);
    }
    return;
  }

  // ---- consumer warps -------------------------------------------------------------
  u64 top = 0ull;
  float thr = -INFINITY;
  int64_t cur_k = -1;
  int nseg_done = 0;
  bool dead = false;
  const int vl0 = warp * 32 * VPL + lane;

  auto finish_segment = [&](int64_t k) {
    const int par = nseg_done & 1;
    if (lane < K) sm.segtop[par][warp][lane] = top;
    consumers_sync();
    ++nseg_done;
    if (warp != 0) return;
    u64 key = warp_merge(0ull, &sm.segtop[par][0][0], NCW * K, lane);
    const int row = sm.rowlist[k - k0];
    // the row's segments: distinct owners of its chunks (owners never decrease;
    // CTAs with an empty range own nothing and are skipped)
    int nseg = 0, myseg = 0, prev_owner = -1;
    for (int qq = 0; qq < cpr; ++qq) {
      const int o = cta_of(k * cpr + qq, T, G);
      if (o != prev_owner) {
        if (o == c) myseg = nseg;
        ++nseg;
        prev_owner = o;
      }
    }
    if (lane < K) a.part[((size_t)row * MAX_SPLIT + myseg) * K + lane] = key;
    if (lane == 0 && myseg == 0) a.row_nseg[row] = nseg;
  };

  for (int64_t i = i0; i < i1; ++i) {
    const int64_t j = i - i0;
    const int s = (int)(j % NSTAGE);
    const uint32_t use = (uint32_t)(j / NSTAGE);
    const int64_t k = i / cpr;
    const int q = (int)(i % cpr);
    if (k != cur_k) {
      if (cur_k >= 0) finish_segment(cur_k);
      top = 0ull;
      thr = -INFINITY;
      cur_k = k;
    }
    if (!dead) dead = __any_sync(FULL, *(volatile int*)&sm.abort_flag != 0);
    if (!dead && !mbar_wait_warp(&sm.full[s], use & 1, polls)) {
      if (lane == 0) {
        atomicOr(a.err, GRAFT_ERR_TIMEOUT);
        *(volatile int*)&sm.abort_flag = 1;
      }
      dead = true;
    }
    if (!dead) {
      const int64_t off = (int64_t)q * TMA_CHUNK;
      const int nvec = (int)(min((int64_t)TMA_CHUNK, g.row_vec_bytes - off) / 16);
      const uint4* stage = reinterpret_cast<const uint4*>(ring + (size_t)s * TMA_CHUNK);
      Vec16<DT> v[VPL];
      float vm[VPL];
      int vmask = 0;
#pragma unroll
      for (int kk = 0; kk < VPL; ++kk) {
        const int vl = vl0 + kk * 32;
        if (vl < nvec) {
          v[kk].r = stage[vl];
          vm[kk] = v[kk].vmax();
          vmask |= 1 << kk;
        } else {
          vm[kk] = -INFINITY;
        }
      }
      const int row = sm.rowlist[k - k0];
      const bool has_tail = (q == cpr - 1) && warp == 0 && lane < g.tail;
      const int32_t tail_id = (int32_t)(g.nslot * EPL + lane);
      const float tv = has_tail
          ? load_scalar<DT>(reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)g.stride * ES, tail_id)
          : -INFINITY;
      float lmax = tv;
#pragma unroll
      for (int kk = 0; kk < VPL; ++kk) lmax = max_nan(lmax, vm[kk]);
      if (lmax != lmax) atomicOr(a.err, GRAFT_ERR_NAN);
      float T8 = thr;
      if (T8 == -INFINITY) {  // fewer than 8 kept: the 8th largest lane maximum bounds the top-8
        u64 lk = make_key(lmax, lane);
        lk = bitonic32_desc(lk, lane);
        const u64 k8 = __shfl_sync(FULL, lk, K - 1);
        T8 = key_val(k8);
      }
      const int64_t vbase = (int64_t)q * (TMA_CHUNK / 16);
#pragma unroll
      for (int kk = 0; kk < VPL; ++kk) {
        if (vm[kk] >= T8) {
          const int64_t vid = vbase + vl0 + kk * 32;
#pragma unroll
          for (int e = 0; e < EPL; ++e) {
            const float x = v[kk].elem(e);
            if (x >= T8) {
              const int idx = atomicAdd(&sm.wcnt[warp], 1);
              if (idx < WCAP) sm.wcand[warp][idx] = make_key(x, (int32_t)(vid * EPL + e));
            }
          }
        }
      }
      if (has_tail && tv >= T8) {
        const int idx = atomicAdd(&sm.wcnt[warp], 1);
        if (idx < WCAP) sm.wcand[warp][idx] = make_key(tv, tail_id);
      }
      __syncwarp();
      const int cw = *(volatile int*)&sm.wcnt[warp];
      if (cw > 0) {
        if (cw <= WCAP) top = warp_merge(top, sm.wcand[warp], cw, lane);
        else top = warp_exact_top8<DT>(v, vmask, vbase, vl0, has_tail, tv, tail_id, top, lane);
        const u64 k8 = __shfl_sync(FULL, top, K - 1);
        thr = k8 ? key_val(k8) : -INFINITY;
        __syncwarp();
        if (lane == 0) sm.wcnt[warp] = 0;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.empty[s]);
  }
  if (cur_k >= 0) finish_segment(cur_k);
}

template <int DT>
cudaError_t verify_tma_impl(const VerifyArgs& a, int grid, cudaStream_t s) {
  k_verify_tma<DT><<<grid, TPB, SMEM_BYTES, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t verify_tma_smem_bytes() { return SMEM_BYTES; }
int verify_tma_max_rows(int grid) { return (MAXROWS - 2) * grid; }

cudaError_t prepare_verify_tma() {
  cudaError_t e = cudaFuncSetAttribute(k_verify_tma<GRAFT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SMEM_BYTES);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(k_verify_tma<GRAFT_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  return e;
}

cudaError_t launch_verify_tma(const VerifyArgs& a, int dtype, int grid, cudaStream_t s) {
  return dtype == GRAFT_BF16 ? verify_tma_impl<GRAFT_BF16>(a, grid, s) : verify_tma_impl<GRAFT_F32>(a, grid, s);
}

}  // namespace graft
