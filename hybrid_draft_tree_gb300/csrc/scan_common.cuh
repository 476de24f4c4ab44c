// Device helpers shared by the verify-scan kernels: 64-bit sort keys
// (value descending, then token id ascending) and warp-level sorting.
#pragma once
#include <climits>

#include <cuda_bf16.h>
#include <stdint.h>

#include "graft_internal.cuh"

namespace graft {
namespace scan {

typedef unsigned long long u64;
constexpr unsigned FULL = 0xffffffffu;

// ---- keys ------------------------------------------------------------------
__device__ __forceinline__ uint32_t ord_bits(float f) {
  uint32_t u = __float_as_uint(f);
  if (u == 0x80000000u) u = 0u;  // -0 ties with +0
  return u ^ ((uint32_t)((int32_t)u >> 31) | 0x80000000u);
}
__device__ __forceinline__ u64 make_key(float v, int32_t id) {
  return ((u64)ord_bits(v) << 32) | (u64)(0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ int32_t key_id(u64 k) { return k ? (int32_t)(0xFFFFFFFFu - (uint32_t)k) : -1; }
__device__ __forceinline__ float key_val(u64 k) {
  const uint32_t o = (uint32_t)(k >> 32);
  return __uint_as_float((o & 0x80000000u) ? (o ^ 0x80000000u) : ~o);
}
// signed-int image of a float with the same order (for warp reductions)
__device__ __forceinline__ int32_t ord_int(float f) {
  const int32_t i = __float_as_int(f);
  return i ^ ((i >> 31) & 0x7FFFFFFF);
}
__device__ __forceinline__ float from_ord_int(int32_t i) { return __int_as_float(i ^ ((i >> 31) & 0x7FFFFFFF)); }

__device__ __forceinline__ float max_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// ---- warp helpers ------------------------------------------------------------
// Bitonic sort of the keys of each group of W lanes; lanes 0..W-1 end up
// descending (for W = 32: the whole warp).
template <int W>
__device__ __forceinline__ u64 bitonic_desc(u64 key, int lane) {
#pragma unroll
  for (int k = 2; k <= W; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const u64 o = __shfl_xor_sync(FULL, key, j);
      const bool desc = (lane & k) == 0;
      const bool low = (lane & j) == 0;
      key = (low == desc) ? (key > o ? key : o) : (key < o ? key : o);
    }
  }
  return key;
}
__device__ __forceinline__ u64 bitonic32_desc(u64 key, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const u64 o = __shfl_xor_sync(FULL, key, j);
      const bool desc = (lane & k) == 0;
      const bool low = (lane & j) == 0;
      key = (low == desc) ? (key > o ? key : o) : (key < o ? key : o);
    }
  }
  return key;
}
__device__ __forceinline__ u64 warp_max_u64(u64 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const u64 x = __shfl_xor_sync(FULL, v, o);
    v = x > v ? x : v;
  }
  return v;
}


// ---- a 16-byte vector of logits: 8 bf16 or 4 fp32 --------------------------------
template <int DT> struct Vec16;
template <> struct Vec16<GRAFT_BF16> {
  uint4 r;
  static constexpr int EPL = 8;
  __device__ __forceinline__ float vmax() const {  // NaN-propagating
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    const uint32_t u = *reinterpret_cast<const uint32_t*>(&m);
    return max_nan(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  }
  // the largest element, NaN left out (a NaN element is never the result
  // unless all eight are NaN): for callers that fold the result with fmaxf
  // anyway, one instruction per pair instead of the NaN-propagating form
  __device__ __forceinline__ float vmax_drop_nan() const {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmax2(__hmax2(a, b), __hmax2(c, d));
    const uint32_t u = *reinterpret_cast<const uint32_t*>(&m);
    return fmaxf(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
  }
  // the largest element (NaN-propagating) and the second largest of the eight
  // (the largest of the others; equal to m1 when the maximum repeats):
  // pairwise max/min of the even and of the odd halves, then their merge
  __device__ __forceinline__ void top2(float& m1, float& m2) const {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 hab = __hmax2_nan(a, b), lab = __hmin2(a, b);
    const __nv_bfloat162 hcd = __hmax2_nan(c, d), lcd = __hmin2(c, d);
    const __nv_bfloat162 h = __hmax2_nan(hab, hcd);                      // (max even, max odd)
    const __nv_bfloat162 l = __hmax2(__hmin2(hab, hcd), __hmax2(lab, lcd));  // (2nd even, 2nd odd)
    const uint32_t hu = *reinterpret_cast<const uint32_t*>(&h), lu = *reinterpret_cast<const uint32_t*>(&l);
    const float he = __uint_as_float(hu << 16), ho = __uint_as_float(hu & 0xFFFF0000u);
    const float le = __uint_as_float(lu << 16), lo = __uint_as_float(lu & 0xFFFF0000u);
    m1 = max_nan(he, ho);
    m2 = fmaxf(fminf(he, ho), fmaxf(le, lo));
  }
  __device__ __forceinline__ float elem(int e) const {
    const uint32_t w = (e < 2) ? r.x : (e < 4) ? r.y : (e < 6) ? r.z : r.w;
    return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
  }
  // bit e set iff elem(e) >= t; t must be a bf16 value (exact in bf16), NaN compares false
  __device__ __forceinline__ unsigned ge_mask(float t) const {
    const __nv_bfloat162 t2 = __float2bfloat162_rn(t);
    const unsigned m0 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&r.x), t2);
    const unsigned m1 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&r.y), t2);
    const unsigned m2 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&r.z), t2);
    const unsigned m3 = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&r.w), t2);
    // low halves (even elements) land on bits 0,2,4,6, high halves on 16,18,20,22
    const unsigned x = (m0 & 0x10001u) | ((m1 & 0x10001u) << 2) | ((m2 & 0x10001u) << 4) | ((m3 & 0x10001u) << 6);
    return (x & 0x55u) | ((x >> 15) & 0xAAu);
  }
};
template <> struct Vec16<GRAFT_F32> {
  uint4 r;
  static constexpr int EPL = 4;
  __device__ __forceinline__ float vmax() const {
    return max_nan(max_nan(__uint_as_float(r.x), __uint_as_float(r.y)),
                   max_nan(__uint_as_float(r.z), __uint_as_float(r.w)));
  }
  __device__ __forceinline__ float vmax_drop_nan() const {
    return fmaxf(fmaxf(__uint_as_float(r.x), __uint_as_float(r.y)), fmaxf(__uint_as_float(r.z), __uint_as_float(r.w)));
  }
  __device__ __forceinline__ float elem(int e) const {
    return __uint_as_float(e == 0 ? r.x : e == 1 ? r.y : e == 2 ? r.z : r.w);
  }
  // the largest element (NaN-propagating) and the second largest of the four
  __device__ __forceinline__ void top2(float& m1, float& m2) const {
    const float a = __uint_as_float(r.x), b = __uint_as_float(r.y);
    const float c = __uint_as_float(r.z), d = __uint_as_float(r.w);
    m1 = max_nan(max_nan(a, b), max_nan(c, d));
    m2 = fmaxf(fminf(fmaxf(a, b), fmaxf(c, d)), fmaxf(fminf(a, b), fminf(c, d)));
  }
  // bit e set iff elem(e) >= t (NaN compares false)
  __device__ __forceinline__ unsigned ge_mask(float t) const {
    return (unsigned)(__uint_as_float(r.x) >= t) | ((unsigned)(__uint_as_float(r.y) >= t) << 1) |
           ((unsigned)(__uint_as_float(r.z) >= t) << 2) | ((unsigned)(__uint_as_float(r.w) >= t) << 3);
  }
};

template <int DT>
__device__ __forceinline__ float load_scalar(const char* row, int64_t v) {
  if (DT == GRAFT_BF16) return __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(row)[v] << 16);
  return reinterpret_cast<const float*>(row)[v];
}

// Merge `cnt` candidate keys from shared memory into a warp's running top-8
// (lanes 0..7 hold it, descending; other lanes hold 0).  Returns the lane's
// new key.
__device__ __forceinline__ u64 warp_merge(u64 top, const u64* cand, int cnt, int lane) {
  u64 key = lane < K ? top : 0ull;
  int base = 0;
  do {
    if (lane >= K) {
      const int c = base + lane - K;
      key = c < cnt ? cand[c] : 0ull;
    }
    key = bitonic32_desc(key, lane);
    base += 32 - K;
  } while (base < cnt);
  return lane < K ? key : 0ull;
}

// Out-of-line copies for rare paths: keeps the hot loops small enough for the
// instruction cache.
static __device__ __noinline__ u64 warp_merge_ool(u64 top, const u64* cand, int cnt, int lane) {
  return warp_merge(top, cand, cnt, lane);
}
// Value of the 8th largest lane key (a lower bound that 8 distinct elements reach).
static __device__ __noinline__ float eighth_lane_max(float lmax, int lane) {
  const u64 lk = bitonic32_desc(make_key(lmax, lane), lane);
  return key_val(__shfl_sync(FULL, lk, K - 1));
}

// Merge `cnt` keys read from global memory (L2, bypassing L1) into a top-8.
__device__ __forceinline__ u64 warp_merge_global(const u64* src, int cnt, int lane) {
  u64 key = 0ull;
  int base = 0;
  bool first = true;
  do {
    if (first || lane >= K) {
      const int c = first ? lane : base + lane - K;
      key = c < cnt ? __ldcg(src + c) : 0ull;
    }
    key = bitonic32_desc(key, lane);
    base = first ? 32 : base + (32 - K);
    first = false;
  } while (base < cnt);
  return lane < K ? key : 0ull;
}

// ---- greedy acceptance of request b (one warp) -----------------------------------
// match(i): slot i is valid and is the root or carries its parent's argmax;
// accepted(i) <=> every ancestor-or-self of i matches <=> mask_i & ~match == 0.
// The winner is the accepted slot of greatest position (ties: lower slot);
// its path tokens after the root, then the bonus token argmax(winner), are
// emitted.
// stok: the tree tokens of all rows in shared memory, or nullptr to read them
// from global memory.
static __device__ void accept_request(const VerifyArgs& a, int b, int lane, const int32_t* stok = nullptr) {
  const int S = a.S;
  const size_t base = (size_t)b * S;
  int32_t tk[2], ps[2];
  uint64_t mk[2];
  bool ok[2], mt[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    ok[h] = false; mt[h] = false;
    tk[h] = -1; ps[h] = -1; mk[h] = 0ull;
    if (s < S) {
      tk[h] = stok ? stok[base + s] : a.tree_tok[base + s];
      if (tk[h] >= 0 && tk[h] < a.g.V) {
        ps[h] = a.tree_pos[base + s];
        mk[h] = a.tree_mask[base + s];
        if (s == 0) {
          ok[h] = ps[h] == 0;
          mt[h] = ok[h];
        } else {
          const int p = a.tree_parent[base + s];
          ok[h] = p >= 0 && p < s && (stok ? stok[base + p] : a.tree_tok[base + p]) >= 0 && ps[h] >= 1 && ps[h] < S;
          if (ok[h]) mt[h] = tk[h] == __ldcg(a.topk + (base + p) * K);
        }
        if (!ok[h]) atomicOr(a.err, GRAFT_ERR_TREE);
      }
    }
  }
  const uint64_t match = (uint64_t)__ballot_sync(FULL, mt[0]) | ((uint64_t)__ballot_sync(FULL, mt[1]) << 32);
  int wkey = -1;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    if (ok[h] && ((mk[h] >> s) & 1ull) && (mk[h] & ~match) == 0ull) wkey = max(wkey, (ps[h] << 8) | (255 - s));
  }
  wkey = __reduce_max_sync(FULL, wkey);
  int32_t* out = a.out_tokens + base;
  if (wkey < 0) {  // no valid root: nothing accepted, nothing emitted
    for (int j = lane; j < S; j += 32) out[j] = -1;
    if (lane == 0) a.accept_len[b] = 0;
    return;
  }
  const int w = 255 - (wkey & 255);
  const int L = wkey >> 8;
  const uint64_t mw = a.tree_mask[base + w];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    if (s > 0 && ok[h] && ((mw >> s) & 1ull) && ps[h] <= L) out[ps[h] - 1] = tk[h];
  }
  for (int j = lane; j < S; j += 32)
    if (j > L) out[j] = -1;
  if (lane == 0) {
    out[L] = __ldcg(a.topk + (base + w) * K);
    a.accept_len[b] = L;
  }
}

// Greedy acceptance of request b (one warp) from tree arrays staged in shared
// memory (sp/spos/smask indexed by slot): match(i) = slot i is valid and is the
// root or carries its parent's argmax; accepted(i) <=> mask_i & ~match == 0;
// the winner is the accepted slot of greatest position (ties: lower slot); its
// path tokens after the root, then the bonus token argmax(winner), are emitted.
// The argmax of every slot's row is fetched in one round trip to L2.
static __device__ __forceinline__ void accept_staged(const VerifyArgs& a, int b, int lane, const int32_t* stok,
                                           const int8_t* sp, const int32_t* spos, const uint64_t* smask) {
  const int S = a.S;
  const size_t base = (size_t)b * S;
  int32_t tk[2], ps[2], am[2], pp[2];
  uint64_t mk[2];
  bool ok[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    tk[h] = s < S ? stok[base + s] : -1;  // raw: a token >= V (flagged by pass 1) still counts as a node
    const bool v = tk[h] >= 0 && tk[h] < a.g.V;
    am[h] = v ? __ldcg(a.topk + (base + s) * K) : -1;
    ps[h] = v ? spos[s] : -1;
    mk[h] = v ? smask[s] : 0ull;
    pp[h] = v && s > 0 ? (int)sp[s] : -1;
  }
  bool mt[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    const int p = pp[h];
    const int q = p >= 0 ? p : 0;
    const int32_t pa0 = __shfl_sync(FULL, am[0], q & 31), pa1 = __shfl_sync(FULL, am[1], q & 31);
    const int32_t ptk0 = __shfl_sync(FULL, tk[0], q & 31), ptk1 = __shfl_sync(FULL, tk[1], q & 31);
    const int32_t pam = q < 32 ? pa0 : pa1, ptk = q < 32 ? ptk0 : ptk1;
    ok[h] = false;
    mt[h] = false;
    if (tk[h] >= 0 && tk[h] < a.g.V) {
      if (s == 0) {
        ok[h] = ps[h] == 0;
        mt[h] = ok[h];
      } else {
        ok[h] = p >= 0 && p < s && ptk >= 0 && ps[h] >= 1 && ps[h] < S;
        mt[h] = ok[h] && tk[h] == pam;
      }
      if (!ok[h]) atomicOr(a.err, GRAFT_ERR_TREE);
    }
  }
  const uint64_t match = (uint64_t)__ballot_sync(FULL, mt[0]) | ((uint64_t)__ballot_sync(FULL, mt[1]) << 32);
  int wkey = -1;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    if (ok[h] && ((mk[h] >> s) & 1ull) && (mk[h] & ~match) == 0ull) wkey = max(wkey, (ps[h] << 8) | (255 - s));
  }
  wkey = __reduce_max_sync(FULL, wkey);
  int32_t* out = a.out_tokens + base;
  if (wkey < 0) {  // no valid root: nothing accepted, nothing emitted
    for (int j = lane; j < S; j += 32) out[j] = -1;
    if (lane == 0) a.accept_len[b] = 0;
    return;
  }
  const int w = 255 - (wkey & 255);
  const int L = wkey >> 8;
  const uint64_t mw = smask[w];
  const int32_t bonus0 = __shfl_sync(FULL, am[0], w & 31), bonus1 = __shfl_sync(FULL, am[1], w & 31);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int s = lane + 32 * h;
    if (s > 0 && ok[h] && ((mw >> s) & 1ull) && ps[h] <= L) out[ps[h] - 1] = tk[h];
  }
  for (int j = lane; j < S; j += 32)
    if (j > L) out[j] = -1;
  if (lane == 0) {
    out[L] = w < 32 ? bonus0 : bonus1;
    a.accept_len[b] = L;
  }
}

// ---- pieces shared by the row-selection kernels ------------------------------------
template <int DT>
static __device__ __noinline__ u64 exact_row(const uint4* rowv, int64_t nslot, const char* rowp, int tail, int lane) {
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

// Value of the 8th largest of the 32 lanes' x: seven rounds remove the
// current maximum (one lane each, the lowest on ties), the eighth reads it.
// x must not be NaN.
static __device__ __forceinline__ float eighth_of_lanes(float x, int lane) {
  int32_t k = ord_int(x);
  int32_t m = 0;
#pragma unroll
  for (int r = 0; r < K; ++r) {
    m = __reduce_max_sync(FULL, k);
    if (r < K - 1) {
      const unsigned owner = __ffs(__ballot_sync(FULL, k == m)) - 1;
      if (lane == (int)owner) k = INT_MIN;
    }
  }
  return from_ord_int(m);
}

// *p += 1 with acquire-release semantics at GPU scope; returns the old value.
static __device__ __forceinline__ int ticket_acq_rel(int32_t* p) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(old) : "l"(p) : "memory");
  return old;
}

// Number of valid slots (0 <= token < V) of request b, from the shared tree
// tokens (one warp).
static __device__ __forceinline__ int request_valid(const VerifyArgs& a, const int32_t* stok, int b, int lane) {
  const int base = b * a.S;
  bool v0 = false, v1 = false;
  if (lane < a.S) { const int32_t t = stok[base + lane]; v0 = t >= 0 && t < a.g.V; }
  if (lane + 32 < a.S) { const int32_t t = stok[base + lane + 32]; v1 = t >= 0 && t < a.g.V; }
  return __popc(__ballot_sync(FULL, v0)) + __popc(__ballot_sync(FULL, v1));
}

}  // namespace scan
}  // namespace graft
