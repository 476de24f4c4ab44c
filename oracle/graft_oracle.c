/*
 * Graft CPU oracle — TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded restatement of one Graft decode step
 * (prune-then-graft hybrid draft trees for lossless speculative decoding,
 * arXiv 2605.20104).  It exists to check the CUDA library; only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or constant generator with the CUDA
 * library: the retrieval template and the slot budget are derived here from
 * the stated rules, independently.
 *
 * Sources (the method is described in prose only; every step below follows
 * the text, in its order):
 *   [P1] Hugging Face paper page "精简草稿，增强检索：投机解码的混合树构建"
 *        (2605.20104), abstract: prune first, then graft retrieved tokens
 *        into the positions pruning opened; training-free and lossless.
 *   [P2] Popular-science article on arXiv 2605.20104, section 二 ("three
 *        gears"): gear 1 = calibrated pruning at draft depths 0/1/5 on the
 *        best path's cumulative confidence, slot split 8+52 / 24+36 / 40+20
 *        of a 60-slot budget; gear 2 = GPU-resident continuation matrix
 *        (top-k successors per token), retrieval rooted at the current token
 *        and expanded by an asymmetric template; gear 3 = flatten the hybrid
 *        tree, rebuild tree positions and mask, verify in one pass, then
 *        update the matrix row of every verified position, accepted or not.
 *        Section 四 (batched serving): fixed verify slots per request, low
 *        confidence draft nodes replaced in place by retrieval nodes.
 *        Section 五 (ablations): pruning without retrieval, and a fixed
 *        draft/retrieval split instead of the confidence checkpoints.
 *        Section 六: warm-up writes target distributions into the matrix.
 *        Section 七 (Graft-TAIL): keep a block draft's confident prefix and
 *        replace the low-confidence tail with retrieval at equal budget.
 *
 * Readings where the text is silent (each is stated where it is used):
 *   k = 8 successors per row; the root (last emitted token) occupies one
 *   verify slot in addition to the 60-slot budget; "depth d" is draft layer
 *   d (layer 0 = the root's children); a checkpoint fires on a strict "<";
 *   kept draft nodes are the top-D by path confidence (ties: lower BFS
 *   index); unused draft slots stay empty; the template is ordered by
 *   (sum of ranks, depth, rank path) and truncated to the retrieval budget;
 *   an empty (-1) matrix entry drops a template node and its subtree (in the
 *   static-tree mode the replaced node keeps its draft token); flatten order
 *   is root, kept draft (BFS), realised retrieval (template order); argmax
 *   and top-k ties go to the lower token id, -0 equals +0, NaN is an error;
 *   the last writer in (request, slot) order wins a matrix row.
 *
 * Parity unpinned: the pages fix no value or rule to check the following
 * against, so the tests pin the rule stated here and its invariants instead
 * of an external value: the template's order (or_template), the static
 * mode's replacement rank among replaced siblings, and the fixed split's
 * ratio in the ablation (a parameter).
 *
 * Floating point: path confidences are fp32 products taken root to leaf (the
 * same precision as the CUDA kernels, because they decide which nodes are
 * kept); logits are compared as doubles (exact for fp32 and bf16 inputs).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_K 8
#define OR_MAXS 64
#define OR_MAXN 1024
#define OR_MAXTPL 256

typedef struct {
  int32_t V, K, budget, S, mode;       /* mode 0 checkpoint, 1 static, 2 tail */
  int32_t ckpt_depth[3];
  float ckpt_thr[3];
  int32_t ckpt_draft[3];
  int32_t tpl_depth, tpl_width;
  float static_thr, tail_thr;
  int32_t ablation;     /* checkpoint mode [P2 §五]: 0 Graft, 1 pruning without retrieval, 2 fixed split */
  int32_t fixed_draft;  /* draft slots of the fixed split (ablation 2) */
} or_params;

enum { OR_OK = 0, OR_EINVAL = -1, OR_EDATA = -4 };

/* ------------------------------------------------------------------------
 * Retrieval template [P2 §二, gear 2]: rooted at the anchor token; the rank-r
 * successor of a node gets max(1, width >> r) children of its own, so top
 * ranks form a long chain and low ranks keep width; depth <= tpl_depth.
 * Entries are rank paths.  They are ordered by (sum of ranks, depth, rank
 * path lexicographically) and the first R are used.  Every path with rank
 * sum <= s is enumerated for s = 0, 1, 2, ... until at least R exist, so the
 * first R of the full ordering are exact.
 * ---------------------------------------------------------------------- */
typedef struct { int32_t len, sum; int8_t r[16]; } or_path;

static int fanout(int32_t width, int depth, const int8_t* r) {
  if (depth == 0) return width;                 /* the anchor */
  int f = width >> r[depth - 1];
  return f < 1 ? 1 : f;
}
static void enum_paths(or_path* cur, int32_t smax, int32_t dmax, int32_t width,
                       or_path* out, int32_t* n, int32_t cap) {
  int f = fanout(width, cur->len, cur->r);
  if (cur->len >= dmax) return;
  for (int rank = 0; rank < f && rank < OR_K; ++rank) {
    if (cur->sum + rank > smax) break;
    or_path nx = *cur;
    nx.r[nx.len++] = (int8_t)rank; nx.sum += rank;
    if (*n < cap) out[*n] = nx;
    ++*n;
    enum_paths(&nx, smax, dmax, width, out, n, cap);
  }
}
static int path_cmp(const void* a_, const void* b_) {
  const or_path* a = (const or_path*)a_; const or_path* b = (const or_path*)b_;
  if (a->sum != b->sum) return a->sum < b->sum ? -1 : 1;
  if (a->len != b->len) return a->len < b->len ? -1 : 1;
  for (int i = 0; i < a->len; ++i) if (a->r[i] != b->r[i]) return a->r[i] < b->r[i] ? -1 : 1;
  return 0;
}
/* Writes the first R entries: parent entry index (-1 = anchor), rank, depth.
 * Returns the number written (fewer than R if the template is smaller). */
int or_template(int32_t dmax, int32_t width, int32_t R, int32_t* parent, int32_t* rank, int32_t* depth) {
  if (R < 0 || R > OR_MAXTPL || dmax < 1 || dmax > 16 || width < 1) return OR_EINVAL;
  static or_path buf[1 << 16];
  int32_t n = 0, prev_n = -1;
  for (int32_t s = 0;; ++s) {
    or_path root; memset(&root, 0, sizeof root);
    n = 0;
    enum_paths(&root, s, dmax, width, buf, &n, 1 << 16);
    if (n > (1 << 16)) return OR_EINVAL;
    if (n >= R || n == prev_n) break;           /* enough, or nothing more exists */
    prev_n = n;
  }
  qsort(buf, (size_t)n, sizeof(or_path), path_cmp);
  int32_t m = n < R ? n : R;
  for (int32_t j = 0; j < m; ++j) {
    rank[j] = buf[j].r[buf[j].len - 1];
    depth[j] = buf[j].len;
    parent[j] = -1;
    if (buf[j].len > 1) {
      or_path pp = buf[j]; pp.len -= 1; pp.sum -= buf[j].r[buf[j].len - 1];
      for (int32_t q = 0; q < j; ++q) if (path_cmp(&buf[q], &pp) == 0) { parent[j] = q; break; }
    }
  }
  return m;
}

/* ------------------------------------------------------------------------
 * Top-8 of one logits row [P2 §二, gear 3: the matrix row records the most
 * probable successors].  Full scan, keeping a sorted list of the best eight
 * under "a before b iff value_a > value_b, or equal values and id_a < id_b".
 * ---------------------------------------------------------------------- */
static double load_val(const void* row, int32_t dtype, int64_t v) {
  if (dtype == 0) return (double)((const float*)row)[v];
  uint32_t u = (uint32_t)((const uint16_t*)row)[v] << 16;
  float f; memcpy(&f, &u, 4);
  return (double)f;
}
static int before(double va, int32_t ia, double vb, int32_t ib) {
  return va > vb || (va == vb && ia < ib);
}
int or_topk8_row(const void* row, int32_t dtype, int32_t V, int32_t* ids) {
  double bv[OR_K]; int32_t bi[OR_K]; int32_t cnt = 0;
  for (int64_t v = 0; v < V; ++v) {
    double x = load_val(row, dtype, v);
    if (x != x) return OR_EDATA;
    if (cnt == OR_K && !before(x, (int32_t)v, bv[OR_K - 1], bi[OR_K - 1])) continue;
    int32_t p = cnt < OR_K ? cnt++ : OR_K - 1;
    while (p > 0 && before(x, (int32_t)v, bv[p - 1], bi[p - 1])) { bv[p] = bv[p - 1]; bi[p] = bi[p - 1]; --p; }
    bv[p] = x; bi[p] = (int32_t)v;
  }
  for (int32_t k = 0; k < OR_K; ++k) ids[k] = k < cnt ? bi[k] : -1;
  return OR_OK;
}

/* ------------------------------------------------------------------------
 * Assembly helpers.
 * ---------------------------------------------------------------------- */
typedef struct { float conf; int32_t idx; } or_rank_item;
static int rank_cmp(const void* a_, const void* b_) {
  const or_rank_item* a = (const or_rank_item*)a_; const or_rank_item* b = (const or_rank_item*)b_;
  if (a->conf != b->conf) return a->conf > b->conf ? -1 : 1;
  return a->idx < b->idx ? -1 : (a->idx > b->idx);
}

/* Path confidence [P2 §二, gear 1: cumulative confidence along the path]:
 * conf(n) = conf(parent) * p(n) in fp32, conf(root) = 1; depth = layer. */
int or_path_conf(int32_t n, const int16_t* parent, const float* prob, float* conf, int32_t* depth) {
  for (int32_t i = 0; i < n; ++i) {
    int32_t p = parent[i];
    if (p >= i || p < -1) return OR_EINVAL;
    if (!(prob[i] >= 0.0f && prob[i] <= 1.0f)) return OR_EDATA;   /* NaN or not a probability */
    float pc = (p < 0) ? 1.0f : conf[p];
    volatile float prod = pc * prob[i];         /* one rounding, no contraction */
    conf[i] = prod;
    depth[i] = (p < 0) ? 0 : depth[p] + 1;
  }
  return OR_OK;
}

static void finish_tree(int32_t S, int32_t n_valid, int32_t* tok, int32_t* par, int32_t* pos, uint64_t* mask) {
  /* Tree position = depth (root 0); mask row = ancestors and self [P2 §二, gear 3]. */
  for (int32_t i = 0; i < S; ++i) {
    if (i >= n_valid || tok[i] < 0) { tok[i] = -1; par[i] = -1; pos[i] = -1; mask[i] = 0; continue; }
    if (i == 0) { par[0] = -1; pos[0] = 0; mask[0] = 1ull; continue; }
    pos[i] = pos[par[i]] + 1;
    mask[i] = mask[par[i]] | (1ull << i);
  }
}

static int check_tok(int32_t t, int32_t V) { return t >= 0 && t < V; }

/* ------------------------------------------------------------------------
 * Checkpoint mode, one request [P2 §二 gears 1-3].
 * info = {fired depth or -1, kept draft, realised retrieval, valid slots}.
 * ---------------------------------------------------------------------- */
int or_assemble_checkpoint(const or_params* P, int32_t root_tok, int32_t n, const int32_t* dtok,
                           const int16_t* dpar, const float* dprob, const int32_t* C,
                           int32_t* tok, int32_t* par, int32_t* pos, uint64_t* mask, int32_t* info) {
  if (n < 0 || n > OR_MAXN || P->S > OR_MAXS || P->S != P->budget + 1) return OR_EINVAL;
  if (P->ablation < 0 || P->ablation > 2 || (P->ablation == 2 && (P->fixed_draft < 0 || P->fixed_draft > P->budget)))
    return OR_EINVAL;
  if (!check_tok(root_tok, P->V)) return OR_EDATA;
  for (int32_t i = 0; i < n; ++i) if (!check_tok(dtok[i], P->V)) return OR_EDATA;
  float conf[OR_MAXN]; int32_t depth[OR_MAXN];
  int rc = or_path_conf(n, dpar, dprob, conf, depth);
  if (rc) return rc;

  /* Gear 1: checkpoints in order; the first whose best path confidence is
   * below its threshold fires and fixes the (draft, retrieval) split. */
  int32_t fired = -1, D = P->budget, R = 0, cut = 1 << 30;
  if (P->ablation == 2) {
    /* [P2 §五] ablation without adaptive pruning: the same (draft, retrieval)
     * split every step, whatever the confidences; the top-D nodes of the
     * whole tree are kept. */
    D = P->fixed_draft; R = P->budget - D;
  } else {
    for (int k = 0; k < 3; ++k) {
      int32_t d = P->ckpt_depth[k];
      int any = 0; float best = 0.f;
      for (int32_t i = 0; i < n; ++i) if (depth[i] == d) { if (!any || conf[i] > best) best = conf[i]; any = 1; }
      if (any && best < P->ckpt_thr[k]) { fired = d; D = P->ckpt_draft[k]; R = P->budget - D; cut = d; break; }
    }
    /* [P2 §五] ablation without retrieval: the pruned slots stay empty. */
    if (P->ablation == 1) R = 0;
  }

  /* Keep the top-D draft nodes of layers <= cut by confidence. */
  or_rank_item items[OR_MAXN]; int32_t m = 0;
  for (int32_t i = 0; i < n; ++i) if (depth[i] <= cut) { items[m].conf = conf[i]; items[m].idx = i; ++m; }
  qsort(items, (size_t)m, sizeof(or_rank_item), rank_cmp);
  int keep[OR_MAXN]; memset(keep, 0, sizeof keep);
  for (int32_t j = 0; j < m && j < D; ++j) keep[items[j].idx] = 1;

  /* Gear 3 flatten: root, kept draft nodes in BFS order ... */
  int32_t slot_of[OR_MAXN]; int32_t s = 0;
  tok[s] = root_tok; par[s] = -1; ++s;
  int32_t nd = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (!keep[i]) continue;
    if (dpar[i] >= 0 && !keep[dpar[i]]) return OR_EINVAL;   /* kept set must be a subtree */
    slot_of[i] = s; tok[s] = dtok[i]; par[s] = dpar[i] < 0 ? 0 : slot_of[dpar[i]]; ++s; ++nd;
  }

  /* Gear 2: retrieval subtree at the root ("the current token"), a pure
   * gather C[parent token][rank]; -1 drops the node and its subtree. */
  int32_t tp[OR_MAXTPL], tr[OR_MAXTPL], td[OR_MAXTPL];
  int32_t nt = or_template(P->tpl_depth, P->tpl_width, R, tp, tr, td);
  if (nt < 0) return OR_EINVAL;
  int32_t rtok[OR_MAXTPL], rslot[OR_MAXTPL]; int32_t nr = 0;
  for (int32_t j = 0; j < nt; ++j) {
    rtok[j] = -1; rslot[j] = -1;
    int32_t ptok = tp[j] < 0 ? root_tok : rtok[tp[j]];
    if (ptok < 0) continue;
    int32_t t = C[(int64_t)ptok * OR_K + tr[j]];
    if (t < -1 || t >= P->V) return OR_EDATA;
    if (t < 0) continue;
    rtok[j] = t;
    rslot[j] = s; tok[s] = t; par[s] = tp[j] < 0 ? 0 : rslot[tp[j]]; ++s; ++nr;
  }
  int32_t n_valid = s;
  for (; s < P->S; ++s) tok[s] = -1;
  finish_tree(P->S, n_valid, tok, par, pos, mask);
  info[0] = fired; info[1] = nd; info[2] = nr; info[3] = n_valid;
  return OR_OK;
}

/* ------------------------------------------------------------------------
 * Incremental drafting, one request [P2 §二, gears 1 and 2]: the checkpoints
 * are meant to stop the drafter, so they are evaluated as its layers complete,
 * and the retrieval gather can run beside the drafter.
 * or_check_layer: with layers 0..layer complete (the n nodes given), evaluate
 * in order every checkpoint whose layer is <= `layer`, unless *event already
 * holds a firing depth; the first that fires writes its depth to *event.
 * ---------------------------------------------------------------------- */
int or_check_layer(const or_params* P, int32_t n, const int16_t* dpar, const float* dprob, int32_t layer,
                   int32_t* event) {
  if (n < 0 || n > OR_MAXN || layer < 0) return OR_EINVAL;
  if (P->ablation == 2 || *event >= 0) return OR_OK;   /* the fixed split has no checkpoints */
  float conf[OR_MAXN]; int32_t depth[OR_MAXN];
  int rc = or_path_conf(n, dpar, dprob, conf, depth);
  if (rc) return rc;
  for (int k = 0; k < 3; ++k) {
    int32_t d = P->ckpt_depth[k];
    if (d > layer) continue;
    int any = 0; float best = 0.f;
    for (int32_t i = 0; i < n; ++i) if (depth[i] == d) { if (!any || conf[i] > best) best = conf[i]; any = 1; }
    if (any && best < P->ckpt_thr[k]) { *event = d; break; }
  }
  return OR_OK;
}

/* or_retrieve: the retrieval entries of one request in template order for
 * the split its event fixes (gear 2: a pure gather C[parent token][rank]
 * anchored at the root); out[j] = token, or -1 when entry j is not realised or
 * j is past the request's retrieval slots.  out has budget entries. */
int or_retrieve(const or_params* P, int32_t root_tok, int32_t event, const int32_t* C, int32_t* out) {
  int32_t R = 0;
  if (P->ablation == 2) R = P->budget - P->fixed_draft;
  else if (P->ablation == 0 && event >= 0)
    for (int k = 0; k < 3; ++k) if (P->ckpt_depth[k] == event) { R = P->budget - P->ckpt_draft[k]; break; }
  for (int32_t j = 0; j < P->budget; ++j) out[j] = -1;
  if (!check_tok(root_tok, P->V)) return OR_EDATA;
  int32_t tp[OR_MAXTPL], tr[OR_MAXTPL], td[OR_MAXTPL];
  int32_t nt = or_template(P->tpl_depth, P->tpl_width, R, tp, tr, td);
  if (nt < 0) return OR_EINVAL;
  for (int32_t j = 0; j < nt; ++j) {
    int32_t ptok = tp[j] < 0 ? root_tok : out[tp[j]];
    if (ptok < 0) continue;
    int32_t t = C[(int64_t)ptok * OR_K + tr[j]];
    if (t < -1 || t >= P->V) return OR_EDATA;
    out[j] = t;
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------
 * Static-tree mode, one request [P2 §四]: each request keeps a fixed number of
 * verify slots (the top-`budget` draft nodes by path confidence, plus the
 * root), and every kept node whose path confidence is below static_thr is
 * replaced in place by a retrieval node.  A replaced node j whose parent p
 * holds token t (after p's own replacement) takes C[t][s], s = j's rank among
 * p's replaced children in slot order.  When that entry is empty there is no
 * retrieval candidate to put there, so j keeps its draft token and the slot
 * count stays fixed.
 * info = {nodes marked for replacement, slots holding a draft token,
 *         slots holding a retrieved token, valid slots}.
 * ---------------------------------------------------------------------- */
int or_assemble_static(const or_params* P, int32_t root_tok, int32_t n, const int32_t* dtok,
                       const int16_t* dpar, const float* dprob, const int32_t* C,
                       int32_t* tok, int32_t* par, int32_t* pos, uint64_t* mask, int32_t* info) {
  if (n < 0 || n > OR_MAXN || P->S > OR_MAXS || P->S != P->budget + 1) return OR_EINVAL;
  if (P->ablation < 0 || P->ablation > 2 || (P->ablation == 2 && (P->fixed_draft < 0 || P->fixed_draft > P->budget)))
    return OR_EINVAL;
  if (!check_tok(root_tok, P->V)) return OR_EDATA;
  for (int32_t i = 0; i < n; ++i) if (!check_tok(dtok[i], P->V)) return OR_EDATA;
  float conf[OR_MAXN]; int32_t depth[OR_MAXN];
  int rc = or_path_conf(n, dpar, dprob, conf, depth);
  if (rc) return rc;
  or_rank_item items[OR_MAXN];
  for (int32_t i = 0; i < n; ++i) { items[i].conf = conf[i]; items[i].idx = i; }
  qsort(items, (size_t)n, sizeof(or_rank_item), rank_cmp);
  int keep[OR_MAXN]; memset(keep, 0, sizeof keep);
  for (int32_t j = 0; j < n && j < P->budget; ++j) keep[items[j].idx] = 1;

  int32_t slot_of[OR_MAXN], s = 1;
  int replaced[OR_MAXS]; memset(replaced, 0, sizeof replaced);
  tok[0] = root_tok; par[0] = -1;
  int32_t nrep = 0;
  for (int32_t i = 0; i < n; ++i) {
    if (!keep[i]) continue;
    if (dpar[i] >= 0 && !keep[dpar[i]]) return OR_EINVAL;
    slot_of[i] = s; tok[s] = dtok[i]; par[s] = dpar[i] < 0 ? 0 : slot_of[dpar[i]];
    replaced[s] = conf[i] < P->static_thr;
    nrep += replaced[s];
    ++s;
  }
  int32_t used = s;
  int32_t nd = 0, nr = 0;
  for (int32_t i = 1; i < used; ++i) {                    /* parents precede children */
    int32_t p = par[i];
    if (!replaced[i]) { ++nd; continue; }
    int32_t srank = 0;
    for (int32_t q = 1; q < i; ++q) if (par[q] == p && replaced[q]) ++srank;
    int32_t t = srank < OR_K ? C[(int64_t)tok[p] * OR_K + srank] : -1;
    if (t < -1 || t >= P->V) return OR_EDATA;
    if (t >= 0) { tok[i] = t; ++nr; }
    else ++nd;                                            /* no candidate: the draft token stays */
  }
  for (; s < P->S; ++s) tok[s] = -1;
  finish_tree(P->S, used, tok, par, pos, mask);
  info[0] = nrep; info[1] = nd; info[2] = nr; info[3] = used;
  return OR_OK;
}

/* ------------------------------------------------------------------------
 * Tail mode, one request [P2 §七, Graft-TAIL]: t = first block position whose
 * confidence is below tail_thr (n if none); the prefix block[0..t) is kept as
 * a chain under the root; the tail's budget - t slots go to the first
 * budget - t template entries anchored at block[t-1] (the root if t = 0).
 * info = {t, kept draft, realised retrieval, valid slots}.
 * ---------------------------------------------------------------------- */
int or_assemble_tail(const or_params* P, int32_t root_tok, int32_t n, const int32_t* btok,
                     const float* bconf, const int32_t* C,
                     int32_t* tok, int32_t* par, int32_t* pos, uint64_t* mask, int32_t* info) {
  if (n < 0 || n > P->budget || P->S > OR_MAXS || P->S != P->budget + 1) return OR_EINVAL;
  if (!check_tok(root_tok, P->V)) return OR_EDATA;
  for (int32_t i = 0; i < n; ++i) if (!check_tok(btok[i], P->V)) return OR_EDATA;
  for (int32_t i = 0; i < n; ++i) if (bconf[i] != bconf[i]) return OR_EDATA;
  int32_t t = n;
  for (int32_t i = 0; i < n; ++i) if (bconf[i] < P->tail_thr) { t = i; break; }
  int32_t s = 0;
  tok[s] = root_tok; par[s] = -1; ++s;
  for (int32_t i = 0; i < t; ++i) { tok[s] = btok[i]; par[s] = s - 1; ++s; }
  int32_t anchor = t;                                      /* slot of block[t-1], or the root */
  int32_t R = P->budget - t;
  int32_t tp[OR_MAXTPL], tr[OR_MAXTPL], td[OR_MAXTPL];
  int32_t nt = or_template(P->tpl_depth, P->tpl_width, R, tp, tr, td);
  if (nt < 0) return OR_EINVAL;
  int32_t rtok[OR_MAXTPL], rslot[OR_MAXTPL], nr = 0;
  for (int32_t j = 0; j < nt; ++j) {
    rtok[j] = -1; rslot[j] = -1;
    int32_t ptok = tp[j] < 0 ? tok[anchor] : rtok[tp[j]];
    if (ptok < 0) continue;
    int32_t x = C[(int64_t)ptok * OR_K + tr[j]];
    if (x < -1 || x >= P->V) return OR_EDATA;
    if (x < 0) continue;
    rtok[j] = x; rslot[j] = s; tok[s] = x; par[s] = tp[j] < 0 ? anchor : rslot[tp[j]]; ++s; ++nr;
  }
  int32_t n_valid = s;
  for (; s < P->S; ++s) tok[s] = -1;
  finish_tree(P->S, n_valid, tok, par, pos, mask);
  info[0] = t; info[1] = t; info[2] = nr; info[3] = n_valid;
  return OR_OK;
}

/* ------------------------------------------------------------------------
 * Greedy tree verification, one request [P2 §二 gear 3; §三 monotonicity]:
 * y_i = argmax of row i (ties: lower id).  Node i is accepted iff every
 * non-root node j on the root->i path carries the token the target chose at
 * j's parent (tok_j == y_parent(j)).  The accepted node of greatest depth
 * (ties: lower slot) is the winner; the emitted tokens are the path's tokens
 * after the root followed by the bonus token y_winner.
 * topk[i][0..8) receives the top-8 of every valid row (-1 rows for pads).
 * out_tokens[S]: emitted tokens then -1.
 * ---------------------------------------------------------------------- */
int or_verify(int32_t S, const int32_t* tok, const int32_t* par, const void* logits, int32_t dtype,
              int32_t V, int64_t stride, int32_t* topk, int32_t* accept_len, int32_t* out_tokens) {
  if (S <= 0 || S > OR_MAXS || tok[0] < 0) return OR_EINVAL;
  int32_t y[OR_MAXS];
  for (int32_t i = 0; i < S; ++i) {
    if (tok[i] < 0) { for (int k = 0; k < OR_K; ++k) topk[i * OR_K + k] = -1; y[i] = -1; continue; }
    if (tok[i] >= V || (i > 0 && (par[i] < 0 || par[i] >= i || tok[par[i]] < 0))) return OR_EINVAL;
    const char* row = (const char*)logits + (size_t)i * (size_t)stride * (dtype == 0 ? 4 : 2);
    int rc = or_topk8_row(row, dtype, V, &topk[i * OR_K]);
    if (rc) return rc;
    y[i] = topk[i * OR_K];
  }
  int32_t win = 0, win_depth = 0;
  for (int32_t i = 1; i < S; ++i) {
    if (tok[i] < 0) continue;
    int ok = 1, d = 0;
    for (int32_t j = i; j != 0; j = par[j]) { if (tok[j] != y[par[j]]) ok = 0; ++d; }
    if (ok && d > win_depth) { win = i; win_depth = d; }
  }
  int32_t path[OR_MAXS];
  for (int32_t j = win, d = win_depth; j != 0; j = par[j]) path[--d] = tok[j];
  for (int32_t i = 0; i < S; ++i) out_tokens[i] = -1;
  for (int32_t d = 0; d < win_depth; ++d) out_tokens[d] = path[d];
  out_tokens[win_depth] = y[win];
  *accept_len = win_depth;
  return OR_OK;
}

/* Online update [P2 §二 gear 3, §六]: every verified position (root,
 * accepted and rejected nodes) overwrites its token's row with the top-8 of
 * its logits row, in slot order. */
int or_update(int32_t* C, int32_t V, int32_t S, const int32_t* tok, const int32_t* topk) {
  for (int32_t i = 0; i < S; ++i) {
    if (tok[i] < 0) continue;
    if (tok[i] >= V) return OR_EINVAL;
    for (int k = 0; k < OR_K; ++k) C[(int64_t)tok[i] * OR_K + k] = topk[i * OR_K + k];
  }
  return OR_OK;
}

/* Warm-up bulk load [P2 §六]: rows in order, each overwrites its token's row
 * with its top-8. */
int or_warmup(int32_t* C, int32_t V, int64_t N, const int32_t* toks, const void* logits,
              int32_t dtype, int64_t stride) {
  int32_t ids[OR_K];
  for (int64_t n = 0; n < N; ++n) {
    if (toks[n] < 0 || toks[n] >= V) return OR_EDATA;
    const char* row = (const char*)logits + (size_t)n * (size_t)stride * (dtype == 0 ? 4 : 2);
    int rc = or_topk8_row(row, dtype, V, ids);
    if (rc) return rc;
    for (int k = 0; k < OR_K; ++k) C[(int64_t)toks[n] * OR_K + k] = ids[k];
  }
  return OR_OK;
}
