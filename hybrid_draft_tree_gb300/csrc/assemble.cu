// graft_assemble's kernel: steps 1-3 of a Graft decode step for one request
// per CTA (popular-science article on arXiv 2605.20104, section 二 gears 1-2
// and the flatten of gear 3; section 四 static trees; section 七 Graft-TAIL).
//
// Work per request is a few KB, so the kernel is latency-bound: everything
// lives in shared memory, one thread per draft node / template entry / slot,
// and the only global traffic is the draft input, at most `budget` 32-byte
// matrix rows gathered for retrieval, and the flattened tree written out.
#include <climits>

#include "graft_internal.cuh"

namespace graft {
namespace {

constexpr int AT = 256;  // threads per CTA (>= MAX_DRAFT, >= MAX_S)
constexpr int WALK = 8;  // ancestors a node walks for its path confidence (deeper trees: layer passes)

__device__ __forceinline__ void raise_err(uint32_t* err, uint32_t bit) { atomicOr(err, bit); }

// Bitonic sort of a warp's 64-bit keys, descending (lane 0 holds the largest).
__device__ __forceinline__ unsigned long long bitonic32_desc_u64(unsigned long long key, int lane) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long o = __shfl_xor_sync(0xffffffffu, key, j);
      const bool desc = (lane & k) == 0;
      const bool low = (lane & j) == 0;
      key = (low == desc) ? (key > o ? key : o) : (key < o ? key : o);
    }
  }
  return key;
}

// Block-wide exclusive prefix count of a predicate.  All threads must call.
__device__ __forceinline__ int block_excl_count(bool v, int* s_warp, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned m = __ballot_sync(0xffffffffu, v);
  const int pre = __popc(m & ((1u << lane) - 1u));
  if (lane == 0) s_warp[warp] = __popc(m);
  __syncthreads();
  int base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < AT / 32; ++w) {
    const int c = s_warp[w];
    base += (w < warp) ? c : 0;
    tot += c;
  }
  __syncthreads();
  total = tot;
  return base + pre;
}

// Path confidences conf(n) = conf(parent) * p(n) (fp32, root first) and
// layer depths of draft nodes 0..nn-1, for the whole CTA (every thread calls;
// thread t owns node t).  s_depth[t] must be -1 for t < nn on entry.  Each node
// walks up to WALK ancestors and multiplies their probabilities root first:
// the same products, in the same order, as computing one layer after the
// other.  Trees deeper than WALK take the layer-by-layer passes.  -0 (a -0.0
// probability) is stored as +0: keys and maxima use the bits, and the two
// compare equal as values.  Returns node t's depth (-1 for t >= nn).
__device__ int block_path_conf(int nn, int t, float prob, const int32_t* s_par, const float* s_prob, float* s_conf,
                               int32_t* s_depth) {
  int my_depth = -1;
  bool deep = false;
  if (t < nn) {
    float pr[WALK];  // pr[i]: probability of the ancestor i levels up (pr[0]: this node)
    int p = t, d = 0;
#pragma unroll
    for (int i = 0; i < WALK; ++i) {
      const bool in = p >= 0;
      const int q = in ? p : 0;
      pr[i] = in ? s_prob[q] : 1.f;
      d += in;
      p = in ? s_par[q] : -1;
    }
    deep = p >= 0;
    if (!deep) {
      float c = 0.f;
#pragma unroll
      for (int k = 0; k < WALK; ++k) {
        const int i = WALK - 1 - k;
        const float x = (i == d - 1) ? pr[i] : __fmul_rn(c, pr[i]);
        c = (i < d) ? (x == 0.f ? 0.f : x) : c;
      }
      s_conf[t] = c;
      my_depth = d - 1;
    }
  }
  // (uniform: every thread takes the passes or none does)
  const bool layered = __syncthreads_or(deep);
  if (layered) my_depth = -1;
  for (int pass = 0; layered && pass <= nn; ++pass) {
    float nc = 0.f;
    int nd = -1;
    if (t < nn && my_depth < 0) {
      const int p = s_par[t];
      if (p < 0) { nc = prob; nd = 0; }
      else {
        const int dp = s_depth[p];
        if (dp >= 0) { nc = __fmul_rn(s_conf[p], prob); nd = dp + 1; }
      }
    }
    __syncthreads();
    if (nd >= 0) { s_conf[t] = nc == 0.f ? 0.f : nc; s_depth[t] = nd; my_depth = nd; }
    if (!__syncthreads_or(t < nn && my_depth < 0)) break;
  }
  return my_depth;
}

__global__ __launch_bounds__(AT) void k_assemble(AssembleArgs a) {
  const int b = blockIdx.x;
  const int t = threadIdx.x;
  const int n = a.n;
  const int S = a.S;

  __shared__ int32_t s_tok[MAX_DRAFT];
  __shared__ int32_t s_par[MAX_DRAFT];
  __shared__ float s_conf[MAX_DRAFT];
  __shared__ float s_prob[MAX_DRAFT];
  __shared__ int s_cnt0[MAX_S];
  __shared__ int32_t s_depth[MAX_DRAFT];
  __shared__ int32_t s_slot[MAX_DRAFT];
  __shared__ __align__(16) unsigned long long s_key[MAX_DRAFT];
  __shared__ int32_t s_rtok[MAX_S];
  __shared__ int32_t s_rslot[MAX_S];
  __shared__ int32_t o_tok[MAX_S];
  __shared__ int32_t o_par[MAX_S];
  __shared__ int32_t o_pos[MAX_S];
  __shared__ int32_t o_rep[MAX_S];
  __shared__ int s_warp[AT / 32];
  __shared__ int s_bad, s_best[3], s_tcut, s_chain;

  const uint64_t keep = l2_keep_policy();
  if (t == 0) { s_bad = 0; s_tcut = n; s_chain = 0; }
  if (t < 3) s_best[t] = -1;
  if (t < MAX_S) {
    o_tok[t] = -1; o_par[t] = -1; o_pos[t] = -1; o_rep[t] = 0; s_rtok[t] = -1; s_rslot[t] = -1; s_cnt0[t] = 0;
  }
  __syncthreads();

  // ---- load and validate -------------------------------------------------
  const int32_t root = a.root_tok[b];
  float prob = 0.f;
  if (t < n) {
    const int64_t k = (int64_t)b * n + t;
    const int32_t tk = a.draft_tok[k];
    s_tok[t] = tk;
    if (tk < 0 || tk >= a.V) { raise_err(a.err, GRAFT_ERR_TOKEN); s_bad = 1; }
    else prefetch_keep(a.C + (int64_t)tk * K);  // matrix rows the first gathers may read
    prob = a.draft_aux[k];
    s_prob[t] = prob;
    if (a.mode != GRAFT_MODE_TAIL) {
      const int p = a.draft_parent[k];
      s_par[t] = p;
      if (p < -1 || p >= t) { raise_err(a.err, GRAFT_ERR_TREE); s_bad = 1; }
      if (!(prob >= 0.f && prob <= 1.f)) { raise_err(a.err, GRAFT_ERR_NAN); s_bad = 1; }
    } else {
      s_par[t] = t - 1;
      if (prob != prob) { raise_err(a.err, GRAFT_ERR_NAN); s_bad = 1; }
    }
    s_depth[t] = -1;
  }
  const bool root_ok = root >= 0 && root < a.V;
  if (t == 0 && !root_ok) raise_err(a.err, GRAFT_ERR_TOKEN);
  if (t == 0 && root_ok) prefetch_keep(a.C + (int64_t)root * K);
  __syncthreads();
  const bool bad = s_bad != 0 || !root_ok;
  const int nn = bad ? 0 : n;   // a request with bad input degrades to its root only

  int n_draft = 0, n_retr = 0, event = -1;
  int R = 0, anchor_slot = 0, anchor_pos = 0, rbase = 1;
  int32_t anchor_tok = root;

  if (a.mode != GRAFT_MODE_TAIL) {
    // ---- path confidence, root to leaf (gear 1) ---------------------------
    const int my_depth = block_path_conf(nn, t, prob, s_par, s_prob, s_conf, s_depth);

    // ---- checkpoints: best path confidence of layers 0, 1, 5 ---------------
    int D = a.budget, cut = INT_MAX;
    if (a.mode == GRAFT_MODE_CHECKPOINT && a.ablation == 2) {
      // ablation without adaptive pruning (section 五): the same split every step
      D = a.fixed_draft;
      R = a.budget - D;
    } else if (a.mode == GRAFT_MODE_CHECKPOINT) {
      if (a.event_in) {
        // incremental drafting: graft_check already evaluated the checkpoints
        // as the layers were drafted; its verdict stands for itself
        // (a request with bad input degrades to its root, as in graft_assemble)
        if (t < 3) s_best[t] = (!bad && a.event_in[b] == a.ckpt_depth[t]) ? 0 : -1;
        if (t == 0 && !bad && a.event_in[b] >= 0 && a.event_in[b] != a.ckpt_depth[0] &&
            a.event_in[b] != a.ckpt_depth[1] && a.event_in[b] != a.ckpt_depth[2])
          raise_err(a.err, GRAFT_ERR_TREE);  // not a checkpoint depth: treated as no firing
      } else if (t < nn) {
#pragma unroll
        for (int k = 0; k < 3; ++k)
          if (my_depth == a.ckpt_depth[k]) atomicMax(&s_best[k], __float_as_int(s_conf[t]));  // conf >= 0
      }
      __syncthreads();
      for (int k = 0; k < 3; ++k) {
        const int bi = s_best[k];
        if (a.event_in ? bi == 0 : (bi >= 0 && __int_as_float(bi) < a.ckpt_thr[k])) {
          event = a.ckpt_depth[k];
          D = min(max(a.ckpt_draft[k], 0), a.budget);
          R = a.budget - D;
          cut = a.ckpt_depth[k];
          break;
        }
      }
      if (a.ablation == 1) R = 0;  // ablation without retrieval (section 五): pruned slots stay empty
    }

    // ---- keep the top-D candidates by (confidence desc, index asc) --------
    // key = (conf bits << 32) | (~index) for candidates (conf >= 0, so its bits
    // order like the value), 0 otherwise; rank = number of larger keys.  Each
    // warp sorts its 32 keys (bitonic, in registers); a candidate's rank is
    // then the sum over the warps' sorted lists of the keys above its own,
    // found by binary search in each list.
    const unsigned long long mine =
        (t < nn && my_depth <= cut)
            ? (((unsigned long long)__float_as_uint(s_conf[t]) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)t))
            : 0ull;
    s_key[t] = bitonic32_desc_u64(mine, t & 31);
    __syncthreads();
    bool kept = false;
    if (mine != 0ull) {
      const int nw = (nn + 31) >> 5;  // warps holding candidates
      int rank = 0;
#pragma unroll
      for (int w = 0; w < AT / 32; ++w) {
        if (w < nw) {
          const unsigned long long* L = s_key + 32 * w;  // descending; zeros last
          int lo = 0;
#pragma unroll
          for (int step = 16; step > 0; step >>= 1)   // lo = number of keys above `mine`
            if (L[lo + step - 1] > mine) lo += step;
          rank += lo + (L[lo] > mine ? 1 : 0);
        }
      }
      kept = rank < D;
    }
    const int pre = block_excl_count(kept, s_warp, n_draft);
    if (t < MAX_DRAFT) s_slot[t] = kept ? 1 + pre : -1;
    __syncthreads();
    if (kept) {
      const int s = 1 + pre;
      const int p = s_par[t];
      int ps = 0;
      if (p >= 0) {
        ps = s_slot[p];
        if (ps < 0) { raise_err(a.err, GRAFT_ERR_TREE); ps = 0; }   // cannot happen for probabilities <= 1
      }
      o_tok[s] = s_tok[t];
      o_par[s] = ps;
      o_pos[s] = my_depth + 1;
      o_rep[s] = (a.mode == GRAFT_MODE_STATIC) && (s_conf[t] < a.static_thr);
    }
    if (t == 0) { o_tok[0] = root_ok ? root : -1; o_par[0] = -1; o_pos[0] = root_ok ? 0 : -1; }
    __syncthreads();
    rbase = 1 + n_draft;

    if (a.mode == GRAFT_MODE_STATIC) {
      // ---- in-place replacement, parents before children (section 四) -----
      // A replaced slot takes C[parent token][its rank among the parent's
      // replaced children]; with no candidate there it keeps its draft token,
      // so every request verifies the same number of slots.
      const int used = 1 + n_draft;
      const int nrep_local = (t >= 1 && t < used) ? o_rep[t] : 0;
      // rank of a replaced slot among its parent's replaced children (slot
      // order): lanes of one warp with the same parent match, and warp 1 adds
      // the count of warp 0 (all slots are in warps 0 and 1)
      int srank = 0;
      const bool rep_me = t >= 1 && t < used && o_rep[t] != 0;
      const int pkey = rep_me ? o_par[t] : -2 - t;  // replaced slots match on their parent
      if (t < MAX_S) {
        const unsigned same = __match_any_sync(0xffffffffu, pkey);
        srank = __popc(same & ((1u << (t & 31)) - 1u));
        if (t < 32 && rep_me && (same >> t) == 1u) s_cnt0[pkey] = __popc(same);  // the group's last lane
      }
      // gathers in passes by chain depth (the replaced slots on the path from
      // the slot up to its first kept ancestor): a chain's first slot reads
      // its kept parent's token, so every chain starts in the first pass
      // whatever its level, and pass r needs only pass r - 1's results
      int cdepth = 0;
      if (rep_me) {
        cdepth = 1;
        for (int p = o_par[t]; p >= 1 && o_rep[p]; p = o_par[p]) ++cdepth;
        atomicMax(&s_chain, cdepth);
      }
      __syncthreads();
      if (t >= 32 && rep_me) srank += s_cnt0[pkey];
      const int rounds = s_chain;
      for (int level = 1; level <= rounds; ++level) {
        if (t >= 1 && t < used && cdepth == level) {
          const int p = o_par[t];
          const int32_t ptok = o_tok[p];
          int32_t tk = -1;
          if (srank < K && ptok >= 0 && ptok < a.V) {
            tk = ld_keep(a.C + (int64_t)ptok * K + srank, keep);
            if (tk < -1 || tk >= a.V) { raise_err(a.err, GRAFT_ERR_TOKEN); tk = -1; }
          }
          if (tk >= 0) { o_tok[t] = tk; o_rep[t] = 2; }
        }
        __syncthreads();
      }
      const bool realised = t >= 1 && t < used && o_rep[t] == 2;
      const bool kept_draft = t >= 1 && t < used && o_rep[t] != 2;
      block_excl_count(kept_draft, s_warp, n_draft);
      block_excl_count(realised, s_warp, n_retr);
      event = __syncthreads_count(nrep_local != 0);
    }
  } else {
    // ---- tail mode: keep the confident prefix as a chain (section 七) -------
    if (t < nn && prob < a.tail_thr) atomicMin(&s_tcut, t);
    __syncthreads();
    const int tc = bad ? 0 : min(s_tcut, nn);
    if (t >= 1 && t <= tc) { o_tok[t] = s_tok[t - 1]; o_par[t] = t - 1; o_pos[t] = t; }
    if (t == 0) { o_tok[0] = root_ok ? root : -1; o_par[0] = -1; o_pos[0] = root_ok ? 0 : -1; }
    event = tc;
    n_draft = tc;
    R = bad ? 0 : a.budget - tc;
    anchor_slot = tc;
    anchor_pos = tc;
    anchor_tok = (tc == 0) ? root : s_tok[tc - 1];
    rbase = 1 + tc;
    __syncthreads();
  }

  if (a.mode != GRAFT_MODE_STATIC) {
    // ---- retrieval subtree: a pure gather along the template (gear 2) -----
    R = min(R, a.tpl.len);
    const int j = t;
    const bool mine = j < R;
    const int jd = mine ? a.tpl.depth[j] : 0;
    const int jq = mine ? a.tpl.parent[j] : -1;
    const int jr = mine ? a.tpl.rank[j] : 0;
    int maxd = a.tpl.maxdepth[R];  // the gather rounds
    if (a.rtok_in) {
      // incremental drafting: graft_retrieve gathered the entries already
      if (mine) {
        int32_t tk = a.rtok_in[(int64_t)b * a.budget + j];
        if (tk < -1 || tk >= a.V) { raise_err(a.err, GRAFT_ERR_TOKEN); tk = -1; }
        s_rtok[j] = tk;
      }
      __syncthreads();
      maxd = 0;
    }
    for (int level = 1; level <= maxd; ++level) {
      if (mine && jd == level) {
        const int32_t ptok = (jq < 0) ? anchor_tok : s_rtok[jq];
        int32_t tk = -1;
        if (ptok >= 0 && ptok < a.V) {
          tk = ld_keep(a.C + (int64_t)ptok * K + jr, keep);
          if (tk < -1 || tk >= a.V) { raise_err(a.err, GRAFT_ERR_TOKEN); tk = -1; }
        }
        s_rtok[j] = tk;
      }
      __syncthreads();
    }
    const bool realised = mine && s_rtok[j] >= 0;
    const int pre = block_excl_count(realised, s_warp, n_retr);
    if (realised) s_rslot[j] = rbase + pre;
    __syncthreads();
    if (realised) {
      const int s = rbase + pre;
      o_tok[s] = s_rtok[j];
      o_par[s] = (jq < 0) ? anchor_slot : s_rslot[jq];
      o_pos[s] = anchor_pos + jd;
    }
    __syncthreads();
  }

  // ---- positions are set; ancestor masks by walking parents (gear 3) ------
  if (t < S) {
    const int64_t k = (int64_t)b * S + t;
    const int32_t tk = o_tok[t];
    if (a.slot_src) {
      // where the slot's token came from: the root, the drafter, or the matrix
      // (retrieval slots follow the kept draft slots; in static mode the
      // in-place replacements)
      const bool retrieved = (a.mode == GRAFT_MODE_STATIC) ? o_rep[t] == 2 : t >= rbase;
      a.slot_src[k] = (int8_t)(tk < 0 ? -1 : t == 0 ? 0 : retrieved ? 2 : 1);
    }
    if (tk >= 0) {
      uint64_t m = 1ull << t;
      int p = o_par[t];
      for (int steps = 0; p >= 0 && steps < MAX_S; ++steps) { m |= 1ull << p; p = o_par[p]; }
      st_keep(a.tree_tok + k, tk, keep);
      st_keep(a.tree_parent + k, (int8_t)o_par[t], keep);
      st_keep(a.tree_pos + k, o_pos[t], keep);
      st_keep(a.tree_mask + k, m, keep);
    } else {
      st_keep(a.tree_tok + k, -1, keep);
      st_keep(a.tree_parent + k, (int8_t)-1, keep);
      st_keep(a.tree_pos + k, -1, keep);
      st_keep(a.tree_mask + k, 0ull, keep);
    }
  }
  const int valid = __syncthreads_count(t < S && o_tok[t] >= 0);
  if (t == 0) {
    int32_t* info = a.info + (int64_t)b * 4;
    info[0] = event;
    info[1] = n_draft;
    info[2] = n_retr;
    info[3] = valid;
  }
}

// ---- incremental drafting: checkpoint verdicts and early retrieval ---------------
// graft_check: for each request whose event is still -1, evaluate (in order)
// the checkpoints whose layer is complete (depth <= a.layer) on the draft so
// far; the first whose best path confidence is below its threshold fires and
// its depth becomes the request's event.  One CTA per request.
// With best_out set instead (graft_confidence), write the best path
// confidence of each checkpoint layer, -1 for an empty layer.
__global__ __launch_bounds__(AT) void k_check(AssembleArgs a, int32_t* event, float* best_out) {
  const int b = blockIdx.x, t = threadIdx.x, n = a.n;
  __shared__ int32_t s_par[MAX_DRAFT];
  __shared__ float s_prob[MAX_DRAFT];
  __shared__ float s_conf[MAX_DRAFT];
  __shared__ int32_t s_depth[MAX_DRAFT];
  __shared__ int s_bad, s_best[3];
  if (t == 0) s_bad = 0;
  if (t < 3) s_best[t] = -1;
  __syncthreads();
  float prob = 0.f;
  if (t < n) {
    const int64_t k = (int64_t)b * n + t;
    const int p = a.draft_parent[k];
    prob = a.draft_aux[k];
    s_par[t] = p;
    s_prob[t] = prob;
    s_depth[t] = -1;
    if (p < -1 || p >= t) { raise_err(a.err, GRAFT_ERR_TREE); s_bad = 1; }
    if (!(prob >= 0.f && prob <= 1.f)) { raise_err(a.err, GRAFT_ERR_NAN); s_bad = 1; }
  }
  __syncthreads();
  const int nn = s_bad ? 0 : n;  // bad input: nothing fires (assemble degrades the request)
  const int my_depth = block_path_conf(nn, t, prob, s_par, s_prob, s_conf, s_depth);
  if (t < nn) {
#pragma unroll
    for (int k = 0; k < 3; ++k)
      if (my_depth == a.ckpt_depth[k] && a.ckpt_depth[k] <= a.layer) atomicMax(&s_best[k], __float_as_int(s_conf[t]));
  }
  __syncthreads();
  if (best_out) {
    if (t < 3) best_out[(int64_t)b * 3 + t] = s_best[t] >= 0 ? __int_as_float(s_best[t]) : -1.f;
    return;
  }
  if (t == 0 && event[b] < 0) {
    for (int k = 0; k < 3; ++k) {
      const int bi = s_best[k];
      if (bi >= 0 && __int_as_float(bi) < a.ckpt_thr[k]) { event[b] = a.ckpt_depth[k]; break; }
    }
  }
}

// Retrieval slots of a request: budget - D(fired checkpoint), 0 when nothing
// fired or without retrieval, budget - fixed_draft under the fixed split.
__device__ __forceinline__ int retrieval_slots(const AssembleArgs& a, int ev) {
  if (a.ablation == 2) return a.budget - a.fixed_draft;
  if (a.ablation == 1 || ev < 0) return 0;
  for (int k = 0; k < 3; ++k)
    if (ev == a.ckpt_depth[k]) return a.budget - min(max(a.ckpt_draft[k], 0), a.budget);
  return 0;
}

// graft_retrieve: the retrieval subtree of every request that fired, gathered
// along the template from the matrix (gear 2), anchored at the root, in
// template order: out[b][j] = token of entry j, or -1 when the entry is not
// realised or beyond the request's retrieval slots.  One CTA per request.
__global__ __launch_bounds__(MAX_S) void k_retrieve(AssembleArgs a, const int32_t* event, int32_t* out) {
  const int b = blockIdx.x, j = threadIdx.x;
  __shared__ int32_t s_rtok[MAX_S];
  const uint64_t keep = l2_keep_policy();
  const int32_t root = a.root_tok[b];
  const bool root_ok = root >= 0 && root < a.V;
  const int R = root_ok ? min(retrieval_slots(a, event[b]), a.tpl.len) : 0;
  const bool mine = j < R;
  const int jd = mine ? a.tpl.depth[j] : 0;
  const int jq = mine ? a.tpl.parent[j] : -1;
  const int jr = mine ? a.tpl.rank[j] : 0;
  s_rtok[j] = -1;
  const int maxd = a.tpl.maxdepth[R];  // the gather rounds
  __syncthreads();
  for (int level = 1; level <= maxd; ++level) {
    if (mine && jd == level) {
      const int32_t ptok = (jq < 0) ? root : s_rtok[jq];
      int32_t tk = -1;
      if (ptok >= 0 && ptok < a.V) {
        tk = ld_keep(a.C + (int64_t)ptok * K + jr, keep);
        if (tk < -1 || tk >= a.V) { raise_err(a.err, GRAFT_ERR_TOKEN); tk = -1; }
      }
      s_rtok[j] = tk;
    }
    __syncthreads();
  }
  if (j < a.budget) out[(int64_t)b * a.budget + j] = mine ? s_rtok[j] : -1;
}

}  // namespace

cudaError_t launch_check(const AssembleArgs& a, int32_t* event, float* best_out, cudaStream_t s) {
  k_check<<<a.batch, AT, 0, s>>>(a, event, best_out);
  return cudaGetLastError();
}
cudaError_t launch_retrieve(const AssembleArgs& a, const int32_t* event, int32_t* out, cudaStream_t s) {
  k_retrieve<<<a.batch, MAX_S, 0, s>>>(a, event, out);
  return cudaGetLastError();
}

cudaError_t launch_assemble(const AssembleArgs& a, cudaStream_t s) {
  k_assemble<<<a.batch, AT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace graft
