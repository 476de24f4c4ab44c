// Single-pass verify scan, its finishing kernel, and the warm-up kernels.
//
// The hot loop of a Graft step is the read of every verified slot's logits
// row (popular-science article on arXiv 2605.20104, section 二 third gear:
// verify the flattened tree in one pass, then update the continuation-matrix
// row of every verified position with the target's most likely successors).
// Greedy verification needs each row's argmax and the update needs its
// top-8, so one pass computes the top-8 and element 0 serves as the argmax.
//
// The default path for 16-byte aligned rows is the two-pass scan (umax.cu,
// select.cu).  This file holds the single-pass scan, taken for rows that are
// not 16-byte aligned, for more rows than the two-pass scan takes, and by the
// allocation-free entry point: k_verify streams equal contiguous slices of
// the valid rows, keeps a lock-free running top-8 per row segment in shared
// memory, and hands each segment's top-8 to k_finish (one CTA per request),
// which merges a row's partials, runs the acceptance walk on bit masks and
// writes the matrix rows (the last writer wins).
//
// The warm-up kernels load the matrix from the last occurrence of each token;
// their row selection (scan_range) is CTA-wide: per round every thread holds
// NV 16-byte vectors (all loads in flight), then
//   pass 1: per-thread max -> per-warp max; T = min over the 8 warp maxima is
//           a value that at least 8 elements of the round reach, and the 8th
//           best value seen by the CTA so far is another; the larger of the
//           two bounds the combined top-8 from below;
//   pass 2: elements >= T (a few dozen of ~16K) go to a shared-memory
//           candidate list; warp 0 merges them into the running top-8 with a
//           32-lane bitonic sort on 64-bit keys (value desc, id asc).
// If the candidate list overflows (e.g. a row of equal values) the CTA falls
// back to an exact 8-round selection over its registers.  Nothing ever spins.
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
  __device__ __forceinline__ void set_neg_inf() {
    const uint32_t w = DT == GRAFT_BF16 ? 0xFF80FF80u : 0xFF800000u;
    this->r = make_uint4(w, w, w, w);
  }
  // the n < EPL elements after the last full vector; the rest read as -inf
  __device__ __forceinline__ void load_tail(const char* row, int64_t first, int n) {
    uint32_t w[4];
    if (DT == GRAFT_BF16) {
      const unsigned short* p = reinterpret_cast<const unsigned short*>(row) + first;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t lo = (2 * i < n) ? p[2 * i] : 0xFF80u;
        const uint32_t hi = (2 * i + 1 < n) ? p[2 * i + 1] : 0xFF80u;
        w[i] = lo | (hi << 16);
      }
    } else {
      const uint32_t* p = reinterpret_cast<const uint32_t*>(row) + first;
#pragma unroll
      for (int i = 0; i < 4; ++i) w[i] = (i < n) ? p[i] : 0xFF800000u;
    }
    this->r = make_uint4(w[0], w[1], w[2], w[3]);
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
  __device__ __forceinline__ void load_tail(const char*, int64_t, int) { r = 0xFF800000u; }
  __device__ __forceinline__ void set_neg_inf() { r = 0xFF800000u; }
};
template <> struct Slot<GRAFT_F32, false> {
  uint32_t r;
  static constexpr int EPL = 1;
  __device__ __forceinline__ void load(const char* row, int64_t s) {
    r = __float_as_uint(__ldcs(reinterpret_cast<const float*>(row) + s));
  }
  __device__ __forceinline__ float vmax() const { return __uint_as_float(r); }
  __device__ __forceinline__ float elem(int) const { return __uint_as_float(r); }
  __device__ __forceinline__ void load_tail(const char*, int64_t, int) { r = 0xFF800000u; }
  __device__ __forceinline__ void set_neg_inf() { r = 0xFF800000u; }
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

// ---- verify + update scan: plain loads, one running top-8 per warp ----------------
// A persistent grid (VCPS CTAs per SM) splits the concatenated valid rows into
// equal contiguous slices.  Within a row segment every warp takes units of 32
// x VNV load slots, keeps the next unit's loads in flight while it filters the
// current one against its own threshold, and merges the rare survivors into
// its own top-8; the CTA syncs once per row segment to merge its 8 warps.
constexpr int VT = 256;
constexpr int VW = VT / 32;
constexpr int VNV = 4;
constexpr int VUNIT = 32 * VNV;
constexpr int VMAXROWS = 192;
constexpr int VSEGS = 24;     // row segments streamed between two CTA barriers
#ifndef GRAFT_VERIFY_CTAS_PER_SM
#define GRAFT_VERIFY_CTAS_PER_SM 4
#endif
constexpr int VCPS = GRAFT_VERIFY_CTAS_PER_SM;

struct VSmem {
  u64 top8[VSEGS][K];  // the CTA's running top-8 of each row segment of the group
  u64 seed[2][VW][K];  // each warp's 8 largest lane maxima of its first unit (by segment parity)
  int warpsum[VW];
  int rowlist[VMAXROWS];
};

// Load one unit: slot s = base + kk*32 + lane for kk < VNV; slots at or past
// `end` (the segment end, never beyond the row's last full vector) read -inf.
// Full units (all but the last of a segment) take unconditional loads.
template <int DT, bool VEC>
__device__ __forceinline__ void load_unit(Slot<DT, VEC> (&v)[VNV], const char* row, int64_t base, int64_t end,
                                          int lane) {
  if (base + VUNIT <= end) {
#pragma unroll
    for (int kk = 0; kk < VNV; ++kk) v[kk].load(row, base + kk * 32 + lane);
  } else {
#pragma unroll
    for (int kk = 0; kk < VNV; ++kk) {
      const int64_t s = base + kk * 32 + lane;
      if (s < end) v[kk].load(row, s);
      else v[kk].set_neg_inf();
    }
  }
}

// ---- the CTA's running top-8 of a row segment ------------------------------------
// top8[0..8) in shared memory, descending, 0 = empty.  A key is inserted by
// offering it to slot 0 with atomicMax and carrying the smaller of (offered,
// previous) down to the next slot.  Slot 0 ends as the largest key ever
// offered, slot 1 as the largest of everything carried out of slot 0 (all keys
// but one), and so on: at any time the slots hold the exact top-8 of the keys
// inserted so far, lock-free.  Slot 7's value is the filter threshold every
// warp of the CTA reads.
// Slots only grow during a segment, so a slot already >= k would pass k on
// unchanged: the cascade may start at the first slot seen below k.
__device__ __forceinline__ void top8_insert(u64* top8, u64 k) {
  int i = 0;
#pragma unroll
  for (int j = K - 1; j >= 0; --j)
    if (*(volatile u64*)&top8[j] < k) i = j;
    else break;
  if (*(volatile u64*)&top8[K - 1] >= k) return;  // cannot enter
#pragma unroll 1
  for (; i < K && k; ++i) {
    const u64 old = atomicMax(&top8[i], k);
    if (old < k) k = old;
    if (k < *(volatile u64*)&top8[K - 1]) return;  // can no longer enter
  }
}

__device__ __forceinline__ float top8_threshold(const u64* top8) {
  const u64 k8 = *(volatile const u64*)&top8[K - 1];
  return k8 ? key_val(k8) : -INFINITY;
}

// Insert the elements of one slot that beat the CTA's current 8th key (rare).
template <int DT, bool VEC>
__device__ __noinline__ void insert_slot(Slot<DT, VEC> v, int64_t vid, float T, u64* top8) {
  constexpr int EPL = Slot<DT, VEC>::EPL;
#pragma unroll 1
  for (int e = 0; e < EPL; ++e) {
    const float x = v.elem(e);
    if (x >= T) {
      const u64 key = make_key(x, (int32_t)(vid * EPL + e));
      if (key > *(volatile u64*)&top8[K - 1]) top8_insert(top8, key);
    }
  }
}

// Filter one unit.  Common case: the vector maxima, one compare against the
// warp's cached threshold Treg and one vote (NaN also fails `lmax < Treg`).
// A stale Treg only lets more through: the CTA's threshold never decreases.
// Otherwise the threshold is refreshed from shared memory, read once and
// broadcast (lanes may arrive at different times after the inserts of an
// earlier unit, and all must take the same branches), and the survivors are
// inserted into the CTA's top-8.
template <int DT, bool VEC>
__device__ __forceinline__ void process_unit(const Slot<DT, VEC> (&v)[VNV], int64_t base, int64_t end, float& Treg,
                                             u64* top8, uint32_t* err, int lane) {
  float vm[VNV];
  float lmax = -INFINITY;
#pragma unroll
  for (int kk = 0; kk < VNV; ++kk) {
    vm[kk] = v[kk].vmax();
    lmax = max_nan(lmax, vm[kk]);
  }
  if (!__any_sync(FULL, !(lmax < Treg))) return;
  if (lmax != lmax) atomicOr(err, GRAFT_ERR_NAN);
  float T = __shfl_sync(FULL, top8_threshold(top8), 0);
  if (T == -INFINITY) T = (Treg != -INFINITY) ? Treg : eighth_lane_max(lmax, lane);  // top-8 not full yet
  Treg = T;
  if (!__any_sync(FULL, lmax >= T)) return;
#pragma unroll
  for (int kk = 0; kk < VNV; ++kk) {
    const int64_t sl = base + kk * 32 + lane;
    if (vm[kk] >= T && sl < end) insert_slot<DT, VEC>(v[kk], sl, T, top8);
  }
  __syncwarp();
}

__device__ __forceinline__ int owner_of(int64_t i, int64_t N, int G) { return (int)(((i + 1) * G - 1) / N); }

template <int DT, bool VEC>
__global__ void __launch_bounds__(VT, VCPS) k_verify(VerifyArgs a) {
  __shared__ VSmem sm;
  using SlotT = Slot<DT, VEC>;
  constexpr int ES = DT == GRAFT_BF16 ? 2 : 4;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const ScanGeom& g = a.g;
  const int rows = a.batch * a.S;
  const int64_t nslot = g.nslot;
  const int64_t npr = nslot + (g.tail > 0 ? 1 : 0);  // load slots per row (+1 for the tail)

  // compact the valid rows (same result in every CTA)
  const int per = (rows + VT - 1) / VT;
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
  __syncthreads();
  int wbase = 0, total = 0;
#pragma unroll
  for (int w = 0; w < VW; ++w) {
    const int x = sm.warpsum[w];
    wbase += (w < warp) ? x : 0;
    total += x;
  }
  const int64_t N = (int64_t)total * npr;
  if (N == 0) return;
  // effective grid: every CTA owns >= min_per slots, so a row spans <= MAX_SPLIT CTAs
  const int64_t min_per = (npr + MAX_SPLIT - 2) / (MAX_SPLIT - 1);
  const int Ge = (int)max((int64_t)1, min((int64_t)gridDim.x, N / min_per));
  const int c = blockIdx.x;
  if (c >= Ge) return;
  const int64_t s0 = (int64_t)c * N / Ge, s1 = (int64_t)(c + 1) * N / Ge;
  const int64_t k0 = s0 / npr, klast = (s1 - 1) / npr;
  if (klast - k0 + 1 > VMAXROWS) {  // the host keeps rows <= (VMAXROWS - 2) * grid
    if (tid == 0) atomicOr(a.err, GRAFT_ERR_TREE);
    return;
  }
  int64_t vidx = wbase + incl - cnt;
  for (int r = r0; r < r1; ++r) {
    const int32_t t = a.tree_tok[r];
    if (t >= 0 && t < g.V) {
      if (vidx >= k0 && vidx <= klast) sm.rowlist[vidx - k0] = r;
      ++vidx;
    }
  }
  __syncthreads();

  // Stream the CTA's row segments in groups of VSEGS.  Inside a group no warp
  // waits for another: each keeps its own top-8 per segment and filters
  // against the segment's shared threshold.  After the group, the segments
  // are finished by different warps in parallel.
  for (int64_t g0 = k0; g0 <= klast; g0 += VSEGS) {
    const int nsg = (int)min((int64_t)VSEGS, klast - g0 + 1);
    for (int i = tid; i < VSEGS * K; i += VT) (&sm.top8[0][0])[i] = 0ull;
    __syncthreads();
    for (int j = 0; j < nsg; ++j) {
      const int64_t k = g0 + j;
      const int row = sm.rowlist[k - k0];
      const int64_t lo = max(s0, k * npr) - k * npr, hi = min(s1, (k + 1) * npr) - k * npr;
      const char* rowp = reinterpret_cast<const char*>(a.logits) + (size_t)row * (size_t)g.stride * ES;
      u64* top8 = sm.top8[j];
      float Treg = -INFINITY;
      const int64_t vhi = min(hi, nslot);  // vector slots of this segment: [lo, vhi)
      const int64_t nunits = vhi > lo ? (vhi - lo + VUNIT - 1) / VUNIT : 0;
      // First round, cooperatively: every warp loads its first unit; the 8th
      // largest of the CTA's lane maxima (8 distinct elements reach it) seeds
      // the threshold, so the first round inserts a few keys instead of
      // every warp filling the top-8 against its own, weaker bound.
      {
        SlotT v[VNV];
        float lmax = -INFINITY;
        const bool has = warp < nunits;
        if (has) {
          load_unit<DT, VEC>(v, rowp, lo + warp * VUNIT, vhi, lane);
#pragma unroll
          for (int kk = 0; kk < VNV; ++kk) lmax = max_nan(lmax, v[kk].vmax());
        }
        const u64 lk = bitonic32_desc(make_key(lmax == lmax ? lmax : -INFINITY, lane), lane);
        if (lane < K) sm.seed[j & 1][warp][lane] = lk;
        __syncthreads();
        const u64 s8 = __shfl_sync(FULL, warp_merge_ool(0ull, &sm.seed[j & 1][0][0], VW * K, lane), K - 1);
        Treg = s8 ? key_val(s8) : -INFINITY;
        if (has) process_unit<DT, VEC>(v, lo + warp * VUNIT, vhi, Treg, top8, a.err, lane);
      }
      // steady state, double-buffered: the next unit's loads are in flight
      // while the current one is filtered (and, rarely, inserted)
      int64_t u = warp + VW;
      if (u < nunits) {
        SlotT va[VNV], vb[VNV];
        load_unit<DT, VEC>(va, rowp, lo + u * VUNIT, vhi, lane);
        while (true) {
          if (u + VW < nunits) load_unit<DT, VEC>(vb, rowp, lo + (u + VW) * VUNIT, vhi, lane);
          process_unit<DT, VEC>(va, lo + u * VUNIT, vhi, Treg, top8, a.err, lane);
          u += VW;
          if (u >= nunits) break;
          if (u + VW < nunits) load_unit<DT, VEC>(va, rowp, lo + (u + VW) * VUNIT, vhi, lane);
          process_unit<DT, VEC>(vb, lo + u * VUNIT, vhi, Treg, top8, a.err, lane);
          u += VW;
          if (u >= nunits) break;
        }
      }
      if (warp == VW - 1 && hi > nslot && lane < g.tail) {  // the row's last V % EPL elements
        constexpr int EPLc = SlotT::EPL;
        const int32_t id = (int32_t)(nslot * EPLc + lane);
        const float x = load_scalar<DT>(rowp, id);
        if (x != x) atomicOr(a.err, GRAFT_ERR_NAN);
        else top8_insert(top8, make_key(x, id));
      }
    }
    __syncthreads();
    // hand the segments' top-8s to the finishing kernel: partial `c - first`
    // of the row's `last - first + 1`
    for (int i = tid; i < nsg * K; i += VT) {
      const int j = i / K, e = i % K;
      const int64_t k = g0 + j;
      const int row = sm.rowlist[k - k0];
      const int first = owner_of(k * npr, N, Ge);
      a.part[((size_t)row * MAX_SPLIT + (c - first)) * K + e] = sm.top8[j][e];
      if (e == 0 && c == first) a.row_nseg[row] = owner_of(k * npr + npr - 1, N, Ge) - first + 1;
    }
    __syncthreads();
  }
}

// ---- finishing: one CTA per request ---------------------------------------------
// Warps merge the request's rows (each row's partial top-8s from the scan) and
// stage them; after one barrier warp 0 runs the acceptance walk; then every
// valid row writes its top-8 into the continuation matrix unless a later row
// (in (request, slot) order, any request) carries the same token: the last
// writer wins without a global winner table or a second kernel.
constexpr int FT = 1024;
constexpr int FW = FT / 32;
__global__ __launch_bounds__(FT) void k_finish(VerifyArgs a, int32_t* C) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int b = blockIdx.x, S = a.S;
  const int rows = a.batch * S;
  const uint64_t keep = l2_keep_policy();
  u64 keys[(MAX_S + FW - 1) / FW];
#pragma unroll
  for (int h = 0; h < (MAX_S + FW - 1) / FW; ++h) {
    const int i = warp + h * FW;
    keys[h] = 0ull;
    if (i >= S) continue;
    const int row = b * S + i;
    const int32_t t = a.tree_tok[row];
    if (t < 0 || t >= a.g.V) continue;
    const int nseg = min(max(a.row_nseg[row], 1), MAX_SPLIT);
    keys[h] = warp_merge_global(a.part + (size_t)row * MAX_SPLIT * K, nseg * K, lane);
    if (lane < K) a.topk[(size_t)row * K + lane] = key_id(keys[h]);
  }
  __syncthreads();
  if (warp == 0 && !a.sample) accept_request(a, b, lane);  // stochastic verification accepts in k_sample
#pragma unroll
  for (int h = 0; h < (MAX_S + FW - 1) / FW; ++h) {
    const int i = warp + h * FW;
    if (i >= S) continue;
    const int row = b * S + i;
    const int32_t t = a.tree_tok[row];
    if (t < 0 || t >= a.g.V) continue;
    bool later = false;
    for (int r = row + 1 + lane; r < rows; r += 32) later |= (a.tree_tok[r] == t);
    const int32_t id = key_id(keys[h]);
    if (!__any_sync(FULL, later) && lane < K) st_keep(C + (size_t)t * K + lane, id, keep);
  }
}

// ---- warm-up -----------------------------------------------------------------------
// The warm-up's kernels run as a chain of programmatic dependent launches:
// each may be scheduled as its predecessor's CTAs leave and waits for the
// predecessor's results (grid_dependency_wait) before reading them.
__global__ void k_warm_mark(WarmArgs a) {
  grid_dependents_launch();
  const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= a.n_rows) return;
  const int32_t t = a.tokens[n];
  if (t < 0 || t >= a.g.V) { atomicOr(a.err, GRAFT_ERR_TOKEN); return; }
  atomicMax(&a.winner[t], (int32_t)(n + 1));
}
__global__ void k_warm_list(WarmArgs a) {
  grid_dependents_launch();
  grid_dependency_wait();  // every mark is in
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
  for (int e = a.start + blockIdx.x; e < count; e += gridDim.x) {
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
  grid_dependency_wait();  // the kernels before it have read the list and the marks
  const int64_t n = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (n == 0) *a.count = 0;
  if (n >= a.n_rows) return;
  const int32_t t = a.tokens[n];
  if (t >= 0 && t < a.g.V) a.winner[t] = 0;
}

template <int DT, bool VEC>
cudaError_t verify_impl(const VerifyArgs& a, int grid, cudaStream_t s) {
  k_verify<DT, VEC><<<grid, VT, 0, s>>>(a);
  return cudaGetLastError();
}
template <int DT, bool VEC>
cudaError_t warm_scan_impl(const WarmArgs& a, int grid_ctas, cudaStream_t s) {
  k_warm_scan<DT, VEC><<<grid_ctas, ST, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

int verify_ctas_per_sm() { return VCPS; }
int verify_max_rows(int grid) { return (VMAXROWS - 2) * grid; }
cudaError_t launch_verify(const VerifyArgs& a, int dtype, int grid, cudaStream_t s) {
  if (dtype == GRAFT_BF16)
    return a.g.vec ? verify_impl<GRAFT_BF16, true>(a, grid, s) : verify_impl<GRAFT_BF16, false>(a, grid, s);
  return a.g.vec ? verify_impl<GRAFT_F32, true>(a, grid, s) : verify_impl<GRAFT_F32, false>(a, grid, s);
}
cudaError_t launch_finish(const VerifyArgs& a, int32_t* C, cudaStream_t s) {
  k_finish<<<a.batch, FT, 0, s>>>(a, C);
  return cudaGetLastError();
}
cudaError_t launch_warmup_begin(const WarmArgs& a, cudaStream_t s) {
  const int t = 256;
  const unsigned g = (unsigned)((a.n_rows + t - 1) / t);
  k_warm_mark<<<g, t, 0, s>>>(a);
  const cudaError_t e = cudaGetLastError();
  return e != cudaSuccess ? e : launch_dependent(k_warm_list, dim3(g), dim3(t), 0, s, a);
}
cudaError_t launch_warmup_scan(const WarmArgs& a, int dtype, int grid_ctas, cudaStream_t s) {
  if (dtype == GRAFT_BF16)
    return a.g.vec ? warm_scan_impl<GRAFT_BF16, true>(a, grid_ctas, s) : warm_scan_impl<GRAFT_BF16, false>(a, grid_ctas, s);
  return a.g.vec ? warm_scan_impl<GRAFT_F32, true>(a, grid_ctas, s) : warm_scan_impl<GRAFT_F32, false>(a, grid_ctas, s);
}
cudaError_t launch_warmup_end(const WarmArgs& a, cudaStream_t s) {
  const int t = 256;
  const unsigned g = (unsigned)((a.n_rows + t - 1) / t);
  return launch_dependent(k_warm_reset, dim3(g), dim3(t), 0, s, a);
}

}  // namespace graft
