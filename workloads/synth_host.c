/*
 * Seeded synthetic inputs for the Graft hot path (host side).
 *
 * This file holds only input generation: counter-based random numbers,
 * synthetic draft trees, draft blocks, token histories and the synthetic
 * "target model" whose logits rows are a pure function of the token prefix.
 * It holds none of the method's arithmetic (no confidence check, no retrieval,
 * no flattening, no verification, no top-k).  Both the CPU oracle and the
 * CUDA library receive what this file produces; the device twin in
 * synth_dev.cu reproduces the row filler and the per-node row parameters
 * bit for bit.
 *
 * Random numbers: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) used as a counter-based hash.
 * Normal noise for logits: Irwin-Hall sum of twelve 16-bit uniforms,
 *   z = (2*sum - 12*65535) / 2^17,
 * which is exact in fp32 (|numerator| < 2^24) and needs no transcendental
 * function, so host and device agree to the bit.
 *
 * Build with -ffp-contract=off: every float expression below is a single
 * IEEE operation and must not be fused.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- salts: one per independent random stream ------------------------- */
#define SALT_NOISE  0x6E6F697365ull  /* "noise" */
#define SALT_HIT    0x486974ull
#define SALT_BIGRAM 0x4269677261ull
#define SALT_TRI    0x547269ull
#define SALT_REQ    0x526571ull
#define SALT_START  0x5374617274ull
#define SALT_PREV   0x50726576ull
#define SALT_CTX    0x437478ull
#define SALT_DRAFT  0x4472616674ull
#define SALT_BLOCK  0x426C6F636Bull
#define SALT_ACTIVE 0x416374ull
#define SALT_HIST   0x48697374ull
#define SALT_WARM   0x5761726Dull
#define SALT_NEXT   0x4E657874ull
#define CTX_MUL     0xD1B54A32D192ED03ull

uint64_t syn_sm64(uint64_t x) {
  x += 0x9E3779B97F4A7C15ull;
  x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
  x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
  return x ^ (x >> 31);
}
static uint64_t h2(uint64_t a, uint64_t b) { return syn_sm64(syn_sm64(a) ^ b); }
static uint64_t h3(uint64_t a, uint64_t b, uint64_t c) { return syn_sm64(h2(a, b) ^ c); }
static uint64_t h4(uint64_t a, uint64_t b, uint64_t c, uint64_t d) { return syn_sm64(h3(a, b, c) ^ d); }
static double u01(uint64_t h) { return (double)(h >> 11) * (1.0 / 9007199254740992.0); }

/* Prefix hash: the context after appending token t. */
uint64_t syn_ctx_push(uint64_t ctx, int32_t t) {
  return syn_sm64(ctx ^ (CTX_MUL * ((uint64_t)(uint32_t)t + 1ull)));
}

/* ---- the synthetic target ------------------------------------------------
 * kind 0: global bigram   succ = h(seed, t) mod V
 * kind 1: trigram         succ = h(seed, prev, t) mod V
 * kind 2: per-request     succ = h(seed, b, t) mod V
 * kind 3: table           succ = table[t] if >= 0 else the kind-0 value
 * The planted successor gets +bias when the context "hits":
 *   hit  <=>  hit_all || (uint32)(h(ctx) >> 32) < hit_num.
 */
typedef struct {
  int32_t V, kind, hit_all;
  uint32_t hit_num;
  float bias;
  uint64_t seed;
  const int32_t* table;
} syn_target;

static int32_t succ_of(const syn_target* tg, int32_t b, int32_t prev, int32_t t) {
  uint64_t V = (uint64_t)tg->V;
  switch (tg->kind) {
    case 1: return (int32_t)(h3(tg->seed ^ SALT_TRI, (uint64_t)(uint32_t)prev, (uint64_t)(uint32_t)t) % V);
    case 2: return (int32_t)(h3(tg->seed ^ SALT_REQ, (uint64_t)(uint32_t)b, (uint64_t)(uint32_t)t) % V);
    case 3:
      if (tg->table && tg->table[t] >= 0) return tg->table[t];
      /* fall through */
    default: return (int32_t)(h2(tg->seed ^ SALT_BIGRAM, (uint64_t)(uint32_t)t) % V);
  }
}
static int hit_of(const syn_target* tg, uint64_t ctx) {
  if (tg->hit_all) return 1;
  return (uint32_t)(syn_sm64(ctx ^ SALT_HIT) >> 32) < tg->hit_num;
}

static void mk_target(syn_target* tg, int32_t V, int32_t kind, int32_t hit_all, uint32_t hit_num,
                      float bias, uint64_t seed, const int32_t* table) {
  tg->V = V; tg->kind = kind; tg->hit_all = hit_all; tg->hit_num = hit_num;
  tg->bias = bias; tg->seed = seed; tg->table = table;
}

/* Planted successor of the context (prev, t) as seen by the target (exported
 * so the harness can build the draft's "correct" tokens and greedy targets). */
int32_t syn_succ(int32_t V, int32_t kind, uint64_t seed, const int32_t* table,
                 int32_t b, int32_t prev, int32_t t) {
  syn_target tg; mk_target(&tg, V, kind, 1, 0, 0.f, seed, table);
  return succ_of(&tg, b, prev, t);
}

/* ---- row filler ---------------------------------------------------------- */
static float noise_z(uint64_t rowkey, int64_t v) {
  uint64_t c = rowkey + 3ull * (uint64_t)v;
  uint32_t s = 0;
  for (int j = 0; j < 3; ++j) {
    uint64_t h = syn_sm64(c + (uint64_t)j);
    s += (uint32_t)(h & 0xFFFF) + (uint32_t)((h >> 16) & 0xFFFF) +
         (uint32_t)((h >> 32) & 0xFFFF) + (uint32_t)(h >> 48);
  }
  int32_t num = 2 * (int32_t)s - 12 * 65535;
  return (float)num * (1.0f / 131072.0f);
}
static uint16_t f32_to_bf16_rne(float f) {
  uint32_t u; memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0x7FC0;
  u += 0x7FFFu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Fill n rows of V logits. planted[r] = -1: noise only; -2: the row is a pad
 * and is filled with quiet NaN (the method must never read it).
 * dtype 0 = fp32, 1 = bf16.  out row r starts at r*stride elements. */
void syn_fill_rows(const uint64_t* rowkey, const int32_t* planted, const float* bias, int64_t n,
                   int32_t V, int32_t dtype, void* out, int64_t stride) {
  for (int64_t r = 0; r < n; ++r) {
    if (dtype == 0) {
      float* row = (float*)out + r * stride;
      if (planted[r] == -2) { uint32_t q = 0x7FC00000u; for (int64_t v = 0; v < V; ++v) memcpy(&row[v], &q, 4); continue; }
      for (int64_t v = 0; v < V; ++v) {
        float x = noise_z(rowkey[r], v);
        if (v == planted[r]) x = x + bias[r];
        row[v] = x;
      }
    } else {
      uint16_t* row = (uint16_t*)out + r * stride;
      if (planted[r] == -2) { for (int64_t v = 0; v < V; ++v) row[v] = 0x7FC0; continue; }
      for (int64_t v = 0; v < V; ++v) {
        float x = noise_z(rowkey[r], v);
        if (v == planted[r]) x = x + bias[r];
        row[v] = f32_to_bf16_rne(x);
      }
    }
  }
}

/* ---- per-node row parameters of a flattened tree ---------------------------
 * tok/parent are [B][S]; a slot with tok < 0 is a pad.  parent[i] < i.
 * The prefix of slot i is the committed sequence (ending in the root token,
 * whose context hash is root_ctx[b]) followed by the path root -> i. */
void syn_tree_rowparams(int32_t V, int32_t kind, int32_t hit_all, uint32_t hit_num, float bias_val,
                        uint64_t seed, const int32_t* table, int32_t B, int32_t S,
                        const int32_t* tok, const int8_t* parent, const uint64_t* root_ctx,
                        const int32_t* root_prev, uint64_t* rowkey, int32_t* planted, float* bias) {
  syn_target tg; mk_target(&tg, V, kind, hit_all, hit_num, bias_val, seed, table);
  uint64_t ctx[256];
  for (int32_t b = 0; b < B; ++b) {
    for (int32_t i = 0; i < S && i < 256; ++i) {
      int64_t k = (int64_t)b * S + i;
      int32_t t = tok[k];
      if (t < 0) { rowkey[k] = 0; planted[k] = -2; bias[k] = 0.f; continue; }
      int32_t prev;
      if (i == 0) { ctx[i] = root_ctx[b]; prev = root_prev[b]; }
      else {
        int p = parent[k];
        if (p < 0 || p >= i) { rowkey[k] = 0; planted[k] = -2; bias[k] = 0.f; continue; }
        ctx[i] = syn_ctx_push(ctx[p], t);
        prev = tok[(int64_t)b * S + p];
      }
      rowkey[k] = syn_sm64(ctx[i] ^ SALT_NOISE);
      planted[k] = hit_of(&tg, ctx[i]) ? succ_of(&tg, b, prev, t) : -1;
      bias[k] = bias_val;
    }
  }
}

/* Row parameters for one prefix given by (ctx, prev, t) — used for greedy
 * reference decoding and warm-up roll-outs. */
void syn_prefix_rowparams(int32_t V, int32_t kind, int32_t hit_all, uint32_t hit_num, float bias_val,
                          uint64_t seed, const int32_t* table, int32_t b, uint64_t ctx,
                          int32_t prev, int32_t t, uint64_t* rowkey, int32_t* planted, float* bias) {
  syn_target tg; mk_target(&tg, V, kind, hit_all, hit_num, bias_val, seed, table);
  *rowkey = syn_sm64(ctx ^ SALT_NOISE);
  *planted = hit_of(&tg, ctx) ? succ_of(&tg, b, prev, t) : -1;
  *bias = bias_val;
}

/* ---- closed-loop request state -------------------------------------------- */
void syn_init_state(uint64_t seed, int32_t V, int32_t B, int32_t* root, int32_t* prev, uint64_t* ctx) {
  for (int32_t b = 0; b < B; ++b) {
    prev[b] = (int32_t)(h2(seed ^ SALT_PREV, (uint64_t)b) % (uint64_t)V);
    root[b] = (int32_t)(h2(seed ^ SALT_START, (uint64_t)b) % (uint64_t)V);
    ctx[b] = syn_ctx_push(syn_ctx_push(h2(seed ^ SALT_CTX, (uint64_t)b), prev[b]), root[b]);
  }
}
/* Append the emitted tokens (emitted[b][0..count[b]) ) to each request. */
void syn_advance(int32_t B, int32_t S, const int32_t* emitted, const int32_t* count,
                 int32_t* root, int32_t* prev, uint64_t* ctx) {
  for (int32_t b = 0; b < B; ++b)
    for (int32_t j = 0; j < count[b]; ++j) {
      int32_t t = emitted[(int64_t)b * S + j];
      prev[b] = root[b]; root[b] = t; ctx[b] = syn_ctx_push(ctx[b], t);
    }
}

/* ---- synthetic draft tree ----------------------------------------------------
 * Full tree with per-layer branching br[0..L): the root has br[0] children,
 * every layer-d node has br[d+1] children.  BFS order, children grouped by
 * parent.  Per sibling group: logits ~ N(0, sigma^2), probabilities = fp32
 * softmax over the group, sorted descending.  One sibling, drawn with
 * probability equal to its own probability, carries the target's planted
 * successor of the parent's context; the others are distinct uniform tokens.
 * Returns the node count (<= cap) or -1. */
static float gauss(uint64_t h1, uint64_t h2_) {
  double u1 = u01(h1), u2 = u01(h2_);
  if (u1 < 1e-300) u1 = 1e-300;
  return (float)(sqrt(-2.0 * log(u1)) * cos(6.283185307179586 * u2));
}

int32_t syn_draft_tree(int32_t V, int32_t kind, uint64_t seed, const int32_t* table, float sigma,
                       int64_t step, int32_t b, int32_t root, int32_t prev, const int32_t* br, int32_t L,
                       int32_t cap, int32_t* tok, int16_t* parent, float* prob) {
  syn_target tg; mk_target(&tg, V, kind, 1, 0, 0.f, seed, table);
  int32_t n = 0, lay_lo = 0, lay_hi = 0;  /* previous layer range [lay_lo, lay_hi) */
  for (int32_t d = 0; d < L; ++d) {
    int32_t np = (d == 0) ? 1 : (lay_hi - lay_lo);
    int32_t start = n;
    for (int32_t q = 0; q < np; ++q) {
      int32_t pidx = (d == 0) ? -1 : lay_lo + q;
      int32_t ptok = (d == 0) ? root : tok[pidx];
      int32_t pprev = (d == 0) ? prev : (parent[pidx] < 0 ? root : tok[parent[pidx]]);
      int32_t g = br[d];
      if (n + g > cap || g > 16) return -1;
      float x[16], p[16];
      uint64_t base = h4(seed ^ SALT_DRAFT, (uint64_t)step, (uint64_t)b, (uint64_t)(pidx + 1));
      float m = -INFINITY;
      for (int32_t j = 0; j < g; ++j) {
        x[j] = sigma * gauss(h2(base, 2ull * j), h2(base, 2ull * j + 1));
        if (x[j] > m) m = x[j];
      }
      float s = 0.f;
      for (int32_t j = 0; j < g; ++j) { p[j] = expf(x[j] - m); s += p[j]; }
      for (int32_t j = 0; j < g; ++j) p[j] = p[j] / s;
      for (int32_t j = 1; j < g; ++j)  /* insertion sort, descending */
        for (int32_t k = j; k > 0 && p[k] > p[k - 1]; --k) { float t_ = p[k]; p[k] = p[k - 1]; p[k - 1] = t_; }
      double u = u01(h2(base, 1000)), cum = 0.0;
      int32_t c = g - 1;
      for (int32_t j = 0; j < g; ++j) { cum += p[j]; if (u < cum) { c = j; break; } }
      int32_t good = succ_of(&tg, b, pprev, ptok);
      for (int32_t j = 0; j < g; ++j) {
        int32_t t;
        if (j == c) t = good;
        else {
          uint64_t ctr = 0;
          for (;;) {
            t = (int32_t)(h3(base, 2000 + (uint64_t)j, ctr++) % (uint64_t)V);
            int clash = (t == good);
            for (int32_t k = 0; k < j; ++k) if (tok[n - j + k] == t) clash = 1;
            if (!clash) break;
          }
        }
        tok[n] = t; parent[n] = (int16_t)pidx; prob[n] = p[j]; ++n;
      }
    }
    lay_lo = start; lay_hi = n;
  }
  return n;
}

/* ---- synthetic draft block (block drafting, e.g. a diffusion drafter) ------
 * conf_i = 1 / (1 + exp(-(z_i - decay*i))), z_i ~ N(mu, sd^2).  Token i is the
 * planted successor of the chain context with probability conf_i, else a
 * uniform token. */
void syn_draft_block(int32_t V, int32_t kind, uint64_t seed, const int32_t* table, int64_t step,
                     int32_t b, int32_t root, int32_t prev, int32_t n, float mu, float sd, float decay,
                     int32_t* tok, float* conf) {
  syn_target tg; mk_target(&tg, V, kind, 1, 0, 0.f, seed, table);
  uint64_t base = h3(seed ^ SALT_BLOCK, (uint64_t)step, (uint64_t)b);
  int32_t p = prev, t = root;
  for (int32_t i = 0; i < n; ++i) {
    float z = mu + sd * gauss(h2(base, 3ull * i), h2(base, 3ull * i + 1));
    float c = 1.0f / (1.0f + expf(-(z - decay * (float)i)));
    int32_t good = succ_of(&tg, b, p, t);
    int32_t nt = (u01(h2(base, 3ull * i + 2)) < (double)c) ? good
               : (int32_t)(h2(base ^ SALT_NEXT, (uint64_t)i) % (uint64_t)V);
    tok[i] = nt; conf[i] = c;
    p = t; t = nt;
  }
}

/* ---- long-context history ---------------------------------------------------
 * N tokens drawn from `active` distinct ids.  The history is cut into spans of
 * length U[span_lo, span_hi]; each span, with probability copy_p, copies an
 * equal-length earlier window (when one exists), else draws i.i.d. Zipf(s)
 * over the active set (rank r has weight r^-s). */
int32_t syn_history(uint64_t seed, int32_t V, int32_t N, int32_t active, double zipf_s, double copy_p,
                    int32_t span_lo, int32_t span_hi, int32_t* hist, int32_t* active_ids) {
  if (active > V || active <= 0) return -1;
  uint8_t* used = (uint8_t*)calloc((size_t)V, 1);
  double* cdf = (double*)malloc(sizeof(double) * (size_t)active);
  if (!used || !cdf) { free(used); free(cdf); return -1; }
  for (int32_t i = 0, ctr = 0; i < active;) {
    int32_t t = (int32_t)(h2(seed ^ SALT_ACTIVE, (uint64_t)ctr++) % (uint64_t)V);
    if (!used[t]) { used[t] = 1; active_ids[i++] = t; }
  }
  double acc = 0.0;
  for (int32_t r = 0; r < active; ++r) { acc += pow((double)(r + 1), -zipf_s); cdf[r] = acc; }
  int32_t pos = 0; uint64_t span = 0;
  while (pos < N) {
    uint64_t hs = h2(seed ^ SALT_HIST, span++);
    int32_t len = span_lo + (int32_t)(h2(hs, 1) % (uint64_t)(span_hi - span_lo + 1));
    if (len > N - pos) len = N - pos;
    if (u01(h2(hs, 2)) < copy_p && pos >= len) {
      int32_t src = (int32_t)(h2(hs, 3) % (uint64_t)(pos - len + 1));
      for (int32_t j = 0; j < len; ++j) hist[pos + j] = hist[src + j];
    } else {
      for (int32_t j = 0; j < len; ++j) {
        double u = u01(h3(hs, 4, (uint64_t)j)) * acc;
        int32_t lo = 0, hi = active - 1;
        while (lo < hi) { int32_t mid = (lo + hi) / 2; if (cdf[mid] > u) hi = mid; else lo = mid + 1; }
        hist[pos + j] = active_ids[lo];
      }
    }
    pos += len;
  }
  free(used); free(cdf);
  return 0;
}

/* Warm-up rows from a history: row i is the target's row after hist[i];
 * its planted successor is hist[i+1] (none for the last row). */
void syn_history_rowparams(uint64_t seed, int32_t N, const int32_t* hist, float bias_val,
                           uint64_t* rowkey, int32_t* planted, float* bias) {
  for (int32_t i = 0; i < N; ++i) {
    rowkey[i] = syn_sm64(h2(seed ^ SALT_WARM, (uint64_t)i) ^ SALT_NOISE);
    planted[i] = (i + 1 < N) ? hist[i + 1] : -1;
    bias[i] = bias_val;
  }
}
/* Successor of each token's last occurrence in a history (-1 if none). */
void syn_history_successors(int32_t V, int32_t N, const int32_t* hist, int32_t* table) {
  for (int32_t t = 0; t < V; ++t) table[t] = -1;
  for (int32_t i = 0; i + 1 < N; ++i) table[hist[i]] = hist[i + 1];
}

/* Warm-up roll-outs: R roll-outs of P positions along the target's planted
 * chain (a context that misses its plant continues with a uniform token).
 * Writes tokens[R*P] and the row parameters of each position. */
void syn_rollouts(int32_t V, int32_t kind, int32_t hit_all, uint32_t hit_num, float bias_val,
                  uint64_t seed, const int32_t* table, int32_t R, int32_t P, int32_t* tokens,
                  uint64_t* rowkey, int32_t* planted, float* bias) {
  syn_target tg; mk_target(&tg, V, kind, hit_all, hit_num, bias_val, seed, table);
  for (int32_t r = 0; r < R; ++r) {
    uint64_t hb = h2(seed ^ SALT_WARM, 1000000ull + (uint64_t)r);
    int32_t prev = (int32_t)(h2(hb, 1) % (uint64_t)V);
    int32_t t = (int32_t)(h2(hb, 2) % (uint64_t)V);
    uint64_t ctx = syn_ctx_push(syn_ctx_push(h2(hb, 3), prev), t);
    for (int32_t i = 0; i < P; ++i) {
      int64_t k = (int64_t)r * P + i;
      tokens[k] = t;
      rowkey[k] = syn_sm64(ctx ^ SALT_NOISE);
      int32_t s = succ_of(&tg, 0, prev, t);
      int hit = hit_of(&tg, ctx);
      planted[k] = hit ? s : -1;
      bias[k] = bias_val;
      int32_t nt = hit ? s : (int32_t)(syn_sm64(ctx ^ SALT_NEXT) % (uint64_t)V);
      prev = t; t = nt; ctx = syn_ctx_push(ctx, t);
    }
  }
}
