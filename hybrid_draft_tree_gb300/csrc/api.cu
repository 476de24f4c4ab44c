// C ABI of libgraft: handle management, argument checking and launches.
// The method (popular-science article on arXiv 2605.20104, section 二) is
// described in include/graft.h; the kernels live in assemble.cu (assembly,
// incremental drafting, confidences), umax.cu + select.cu (the default verify
// scan), scan.cu (single-pass scan, finishing, warm-up), scan_tma.cu,
// sample.cu (stochastic verification), coverage.cu and noalloc.cu.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <queue>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "graft_internal.cuh"

struct graft_handle {
  graft_config cfg;
  int S = 0;
  int device = 0;
  int num_sms = 0;
  int cluster_max_active = 0;  // clusters of the cluster-per-row verify resident at once (0: not available)
  int warm_ctas = 0;        // resident CTAs of the warm-up scan
  int scan_ctas_target = 0; // CTAs wanted per verify launch
  bool tma_ready = false;   // the TMA scan's shared-memory opt-in succeeded
  int32_t* C = nullptr;           // [V][8]
  int32_t* winner = nullptr;      // [V]
  int32_t* tpl = nullptr;         // [3][tpl_len]: parent, rank, depth; then [tpl_len + 1]: depth maxima of prefixes
  int tpl_len = 0;
  unsigned long long* part = nullptr;  // [rows][MAX_SPLIT][8]
  int32_t* row_ticket = nullptr;  // [rows]
  int32_t* req_ticket = nullptr;  // [max_batch]
  int32_t* topk = nullptr;        // [rows][8]
  int32_t* row_nseg = nullptr;    // [rows]
  float* umax = nullptr;          // [rows][upr_max rounded up to 4] two-pass unit maxima
  float* usec = nullptr;          // [rows][same] second largest element of every unit (scan_kernel 4)
  uint8_t* upos = nullptr;        // [rows][same] position of every unit's maximum (scan_kernel 4)
  float* warm_umax = nullptr;     // [min(V, WARM_TWO_PASS_ROWS)][upr_max rounded up to 4] the warm-up's
  int warm_rows = 0;
  int upr_max = 0;
  int32_t* list = nullptr;        // [V] warm-up rows
  int32_t* count = nullptr;       // [1]
  uint32_t* err = nullptr;        // [1]
  int32_t last_launches = 0;
  uint32_t wait_polls = 0;        // TMA scan wait limit (0 = the kernel's default)
  char msg[256] = {0};
  // tracing: event pairs around kernels, read back by graft_profile_read
  static constexpr int kProfSlots = 64;
  bool profiling = false;
  cudaEvent_t prof_ev[2 * kProfSlots] = {};
  const char* prof_name[kProfSlots] = {};
  int prof_n = 0;
};

namespace {

int fail(graft_handle* h, int code, const char* fmt, ...) {
  if (h) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(h->msg, sizeof h->msg, fmt, ap);
    va_end(ap);
  }
  return code;
}

int cuda_fail(graft_handle* h, cudaError_t e, const char* what) {
  return fail(h, GRAFT_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Retrieval template (article §二, second gear): rank paths below the anchor;
// the rank-r successor of a node has max(1, width >> r) children, the anchor
// `width`; depth <= max_depth.  Entries are emitted in increasing
// (rank sum, depth, rank path) order by best-first expansion: a child's key
// is never smaller than its parent's, so popping the smallest key from a
// frontier seeded with the anchor's children yields the global order.
struct TplNode {
  int sum, depth;
  std::vector<int> path;
  int index;  // emitted index, set when popped
};
struct TplCmp {
  bool operator()(const TplNode& a, const TplNode& b) const {  // "a after b"
    if (a.sum != b.sum) return a.sum > b.sum;
    if (a.depth != b.depth) return a.depth > b.depth;
    return a.path > b.path;
  }
};

void build_template(int max_depth, int width, int len, std::vector<int32_t>& parent, std::vector<int32_t>& rank,
                    std::vector<int32_t>& depth) {
  std::priority_queue<TplNode, std::vector<TplNode>, TplCmp> frontier;
  // frontier entries carry their parent's emitted index in `index`
  for (int r = 0; r < width && r < graft::K; ++r) frontier.push(TplNode{r, 1, {r}, -1});
  while ((int)parent.size() < len && !frontier.empty()) {
    TplNode nd = frontier.top();
    frontier.pop();
    const int me = (int)parent.size();
    parent.push_back(nd.index);
    rank.push_back(nd.path.back());
    depth.push_back(nd.depth);
    if (nd.depth < max_depth) {
      int fan = width >> nd.path.back();
      if (fan < 1) fan = 1;
      for (int r = 0; r < fan && r < graft::K; ++r) {
        TplNode c{nd.sum + r, nd.depth + 1, nd.path, me};
        c.path.push_back(r);
        frontier.push(c);
      }
    }
  }
}

// A named NVTX range around one ABI call, for profilers that record NVTX
// (ncu --nvtx); header-only NVTX 3, a few nanoseconds when none is attached.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Bracket one kernel launch with profiling events when tracing is on.
struct ProfScope {
  graft_handle* h;
  cudaStream_t s;
  int slot = -1;
  ProfScope(graft_handle* h_, cudaStream_t s_, const char* name) : h(h_), s(s_) {
    if (h->profiling && h->prof_n < graft_handle::kProfSlots) {
      slot = h->prof_n++;
      h->prof_name[slot] = name;
      cudaEventRecord(h->prof_ev[2 * slot], s);
    }
  }
  ~ProfScope() {
    if (slot >= 0) cudaEventRecord(h->prof_ev[2 * slot + 1], s);
  }
};

template <typename T>
cudaError_t dalloc(T** p, size_t n) {
  return cudaMalloc(reinterpret_cast<void**>(p), n * sizeof(T) + 16);
}

void free_all(graft_handle* h) {
  for (auto& e : h->prof_ev)
    if (e) cudaEventDestroy(e);
  cudaFree(h->C); cudaFree(h->winner); cudaFree(h->tpl); cudaFree(h->part);
  cudaFree(h->row_ticket); cudaFree(h->req_ticket); cudaFree(h->topk); cudaFree(h->row_nseg); cudaFree(h->umax); cudaFree(h->usec); cudaFree(h->upos);
  cudaFree(h->warm_umax);
  cudaFree(h->list); cudaFree(h->count); cudaFree(h->err);
}

int check_cfg(const graft_config* c, graft_handle* h) {
  if (c->vocab < 1) return fail(h, GRAFT_EINVAL, "vocab must be >= 1");
  if (c->topk != graft::K) return fail(h, GRAFT_EINVAL, "topk must be 8");
  if (c->budget < 1 || c->budget + 1 > graft::MAX_S) return fail(h, GRAFT_EINVAL, "budget must be in [1, 63]");
  if (c->max_batch < 1 || (int64_t)c->max_batch * (c->budget + 1) > 65535)
    return fail(h, GRAFT_EINVAL, "max_batch * (budget + 1) must be in [1, 65535]");
  if (c->mode < GRAFT_MODE_CHECKPOINT || c->mode > GRAFT_MODE_TAIL) return fail(h, GRAFT_EINVAL, "bad mode");
  if (c->logits_dtype != GRAFT_F32 && c->logits_dtype != GRAFT_BF16) return fail(h, GRAFT_EINVAL, "bad logits dtype");
  if (c->mode == GRAFT_MODE_CHECKPOINT)
    for (int k = 0; k < 3; ++k)
      if (c->ckpt_draft[k] < 0 || c->ckpt_draft[k] > c->budget || c->ckpt_depth[k] < 0)
        return fail(h, GRAFT_EINVAL, "checkpoint %d: draft slots must be in [0, budget], depth >= 0", k);
  for (int k = 0; k < 3; ++k)
    if (!(c->ckpt_thr[k] >= 0.f && c->ckpt_thr[k] <= 1.f))
      return fail(h, GRAFT_EINVAL, "checkpoint threshold %d must be in [0, 1]", k);
  if (!(c->static_thr >= 0.f && c->static_thr <= 1.f) || !(c->tail_thr >= 0.f && c->tail_thr <= 1.f))
    return fail(h, GRAFT_EINVAL, "static and tail thresholds must be in [0, 1]");
  if (c->tpl_depth < 1 || c->tpl_depth > 16 || c->tpl_width < 1 || c->tpl_width > 64)
    return fail(h, GRAFT_EINVAL, "template depth must be in [1, 16] and width in [1, 64]");
  if (c->ablation < 0 || c->ablation > 2 || (c->ablation != 0 && c->mode != GRAFT_MODE_CHECKPOINT))
    return fail(h, GRAFT_EINVAL, "ablation must be 0, or 1 / 2 in checkpoint mode");
  if (c->ablation == 2 && (c->fixed_draft < 0 || c->fixed_draft > c->budget))
    return fail(h, GRAFT_EINVAL, "fixed_draft must be in [0, budget]");
  const int maxn = c->mode == GRAFT_MODE_TAIL ? c->budget : graft::MAX_DRAFT;
  if (c->max_draft_nodes < 0 || c->max_draft_nodes > maxn)
    return fail(h, GRAFT_EINVAL, "max_draft_nodes must be in [0, %d]", maxn);
  if (c->scan_kernel < 0 || c->scan_kernel > 5) return fail(h, GRAFT_EINVAL, "scan_kernel must be in [0, 5]");
  return GRAFT_OK;
}

// Geometry of a row scan: 16-byte vector loads when every row start is
// 16-byte aligned, scalar loads otherwise; `ctas_wanted` CTAs in total.
graft::ScanGeom scan_geom(const graft_handle* h, const void* logits, int64_t stride, int64_t rows,
                          int ctas_wanted) {
  graft::ScanGeom g{};
  const int es = h->cfg.logits_dtype == GRAFT_BF16 ? 2 : 4;
  g.V = h->cfg.vocab;
  g.stride = stride;
  g.vec = ((reinterpret_cast<uintptr_t>(logits) & 15) == 0) && ((stride * es) % 16 == 0);
  g.epl = g.vec ? 16 / es : 1;
  g.nslot = g.V / g.epl;
  g.tail = (int32_t)(g.V - g.nslot * g.epl);
  int64_t nsplit = rows > 0 ? (ctas_wanted + rows - 1) / rows : 1;
  const int64_t by_size = (g.nslot + 1023) / 1024;  // at least ~1024 slots per CTA
  if (nsplit > by_size) nsplit = by_size;
  if (nsplit > graft::MAX_SPLIT) nsplit = graft::MAX_SPLIT;
  if (nsplit < 1) nsplit = 1;
  g.nsplit = (int32_t)nsplit;
  g.per_cta = (g.nslot + nsplit - 1) / nsplit;
  g.row_vec_bytes = g.nslot * 16;
  g.cpr = (int32_t)((g.row_vec_bytes + graft::TMA_CHUNK - 1) / graft::TMA_CHUNK);
  return g;
}

}  // namespace

extern "C" {

void graft_default_config(graft_config* c, int32_t vocab, int32_t max_batch, int32_t mode, int32_t dtype) {
  std::memset(c, 0, sizeof *c);
  c->vocab = vocab;
  c->topk = graft::K;
  c->budget = mode == GRAFT_MODE_TAIL ? 16 : 60;
  c->max_batch = max_batch;
  c->mode = mode;
  c->logits_dtype = dtype;
  c->ckpt_depth[0] = 0; c->ckpt_depth[1] = 1; c->ckpt_depth[2] = 5;
  c->ckpt_thr[0] = 0.30f; c->ckpt_thr[1] = 0.20f; c->ckpt_thr[2] = 0.10f;
  c->ckpt_draft[0] = 8; c->ckpt_draft[1] = 24; c->ckpt_draft[2] = 40;
  c->tpl_depth = 8;
  c->tpl_width = 8;
  c->static_thr = 0.15f;
  c->tail_thr = 0.4f;
  c->max_draft_nodes = mode == GRAFT_MODE_TAIL ? 16 : 184;
  c->scan_kernel = 0;
  c->ablation = 0;
  c->fixed_draft = 40;
}

int graft_init(const graft_config* cfg, graft_handle** out) {
  if (!cfg || !out) return GRAFT_EINVAL;
  *out = nullptr;
  graft_handle* h = new (std::nothrow) graft_handle();
  if (!h) return GRAFT_ENOMEM;
  int rc = check_cfg(cfg, h);
  if (rc) { delete h; return rc; }
  h->cfg = *cfg;
  h->S = cfg->budget + 1;
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) { delete h; return GRAFT_ECUDA; }

  std::vector<int32_t> tp, tr, td;
  build_template(cfg->tpl_depth, cfg->tpl_width, cfg->budget, tp, tr, td);
  h->tpl_len = (int)tp.size();

  const size_t V = (size_t)cfg->vocab;
  const size_t rows = (size_t)cfg->max_batch * h->S;
  e = dalloc(&h->C, V * graft::K);
  if (e == cudaSuccess) e = dalloc(&h->winner, V);
  if (e == cudaSuccess) e = dalloc(&h->tpl, 4 * (size_t)h->tpl_len + 1);
  if (e == cudaSuccess) e = dalloc(&h->part, rows * graft::MAX_SPLIT * graft::K);
  if (e == cudaSuccess) e = dalloc(&h->row_ticket, rows);
  if (e == cudaSuccess) e = dalloc(&h->req_ticket, (size_t)cfg->max_batch);
  if (e == cudaSuccess) e = dalloc(&h->topk, rows * graft::K);
  if (e == cudaSuccess) e = dalloc(&h->row_nseg, rows);
  {
    const int64_t epl_min = cfg->logits_dtype == GRAFT_BF16 ? 8 : 4;  // two-pass runs on 16-byte aligned rows only
    const int64_t upr = (V / epl_min + 31) / 32;
    h->upr_max = (int)(upr <= graft::TWO_PASS_MAX_UNITS ? upr : 0);
    const size_t ups = (size_t)((h->upr_max + 3) & ~3);
    if (e == cudaSuccess && h->upr_max > 0) e = dalloc(&h->umax, rows * ups);
    if (e == cudaSuccess && h->upr_max > 0 && cfg->scan_kernel == 4) e = dalloc(&h->usec, rows * ups);
    if (e == cudaSuccess && h->upr_max > 0 && cfg->scan_kernel == 4) e = dalloc(&h->upos, rows * ups);
    h->warm_rows = (int)std::min<size_t>(V, graft::WARM_TWO_PASS_ROWS);
    if (e == cudaSuccess && h->upr_max > 0) e = dalloc(&h->warm_umax, (size_t)h->warm_rows * ups);
  }
  if (e == cudaSuccess) e = dalloc(&h->list, V);
  if (e == cudaSuccess) e = dalloc(&h->count, 1);
  if (e == cudaSuccess) e = dalloc(&h->err, 1);
  if (e != cudaSuccess) { free_all(h); delete h; return GRAFT_ENOMEM; }

  e = cudaMemset(h->C, 0xFF, V * graft::K * sizeof(int32_t));  // -1 = empty
  if (e == cudaSuccess) e = cudaMemset(h->winner, 0, V * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->row_ticket, 0, rows * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->req_ticket, 0, cfg->max_batch * sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->count, 0, sizeof(int32_t));
  if (e == cudaSuccess) e = cudaMemset(h->err, 0, sizeof(uint32_t));
  if (e == cudaSuccess) {
    std::vector<int32_t> all(tp);
    all.insert(all.end(), tr.begin(), tr.end());
    all.insert(all.end(), td.begin(), td.end());
    int32_t m = 0;  // depth maxima of the template's prefixes: the gather rounds a retrieval of R entries takes
    all.push_back(0);
    for (int32_t d : td) all.push_back(m = std::max(m, d));
    e = cudaMemcpy(h->tpl, all.data(), all.size() * sizeof(int32_t), cudaMemcpyHostToDevice);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) { free_all(h); delete h; return GRAFT_ECUDA; }
  h->warm_ctas = h->num_sms * 4;
  h->scan_ctas_target = h->num_sms * 8;
  h->tma_ready = graft::prepare_verify_tma() == cudaSuccess;
  h->cluster_max_active = graft::cluster_select_max_active(cfg->vocab, cfg->logits_dtype);
  cudaGetLastError();
  *out = h;
  return GRAFT_OK;
}

int graft_destroy(graft_handle* h) {
  if (!h) return GRAFT_EINVAL;
  cudaDeviceSynchronize();
  free_all(h);
  delete h;
  return GRAFT_OK;
}

int graft_warmup(graft_handle* h, const int32_t* d_tokens, const void* d_logits, int64_t n_rows, int64_t row_stride,
                 void* stream) {
  NvtxRange nvtx("graft_warmup");
  if (!h) return GRAFT_EINVAL;
  h->last_launches = 0;
  if (n_rows < 0 || n_rows >= 0x7FFFFFFF) return fail(h, GRAFT_EINVAL, "n_rows must be in [0, 2^31-1)");
  if (n_rows == 0) return GRAFT_OK;
  if (!d_tokens || !d_logits) return fail(h, GRAFT_EINVAL, "null pointer");
  if (row_stride < h->cfg.vocab) return fail(h, GRAFT_EINVAL, "row_stride < vocab");
  if (graft::misaligned(d_tokens, 4) || graft::misaligned(d_logits, h->cfg.logits_dtype == GRAFT_BF16 ? 2 : 4))
    return fail(h, GRAFT_EINVAL, "a buffer is not aligned to its element size");
  graft::WarmArgs a{};
  a.g = scan_geom(h, d_logits, row_stride, n_rows, 0);
  a.g.nsplit = 1;
  a.g.per_cta = a.g.nslot;
  a.n_rows = n_rows;
  a.logits = d_logits;
  a.tokens = d_tokens;
  a.winner = h->winner;
  a.list = h->list;
  a.count = h->count;
  a.C = h->C;
  a.err = h->err;
  // the last occurrence of each token (listed on the device) takes the
  // two-pass scan on aligned rows, up to warm_rows of them; any further rows
  // (and unaligned rows) take the single-pass scan
  const int32_t upr = (int32_t)((a.g.nslot + 31) / 32);
  const bool two_pass = a.g.vec && h->warm_umax && a.g.nslot > 0 && upr <= h->upr_max;
  a.start = two_pass ? h->warm_rows : 0;
  graft::VerifyArgs v{};
  v.g = a.g;
  v.logits = d_logits;
  v.umax = h->warm_umax;
  v.top2 = 0;
  v.upr = upr;
  v.ups = (upr + 3) & ~3;
  v.err = h->err;
  const int grid1 = h->num_sms * graft::two_pass_ctas_per_sm();
  const int dt = h->cfg.logits_dtype;
  cudaError_t e;
  {
    ProfScope ps(h, (cudaStream_t)stream, "warmup");
    e = graft::launch_warmup_begin(a, (cudaStream_t)stream);
    if (e == cudaSuccess && two_pass)
      e = graft::launch_warm_umax(v, h->list, h->count, h->warm_rows, dt, grid1, (cudaStream_t)stream);
    if (e == cudaSuccess && two_pass)
      e = graft::launch_warm_select(v, d_tokens, h->list, h->count, h->warm_rows, h->C, dt, h->num_sms * 2,
                                    (cudaStream_t)stream);
    if (e == cudaSuccess && n_rows > a.start)
      e = graft::launch_warmup_scan(a, dt, h->warm_ctas, (cudaStream_t)stream);
    if (e == cudaSuccess) e = graft::launch_warmup_end(a, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_warmup launch");
  h->last_launches = 3 + (two_pass ? 2 : 0) + (n_rows > a.start ? 1 : 0);
  return GRAFT_OK;
}

}  // extern "C"

namespace {

graft::AssembleArgs assemble_args(const graft_handle* h, int32_t batch, int32_t draft_nodes) {
  const graft_config& c = h->cfg;
  graft::AssembleArgs a{};
  a.mode = c.mode; a.V = c.vocab; a.budget = c.budget; a.S = h->S; a.n = draft_nodes; a.batch = batch;
  for (int k = 0; k < 3; ++k) {
    a.ckpt_depth[k] = c.ckpt_depth[k];
    a.ckpt_thr[k] = c.ckpt_thr[k];
    a.ckpt_draft[k] = c.ckpt_draft[k];
  }
  a.static_thr = c.static_thr;
  a.tail_thr = c.tail_thr;
  a.ablation = c.ablation;
  a.fixed_draft = c.fixed_draft;
  a.C = h->C;
  a.tpl.parent = h->tpl;
  a.tpl.rank = h->tpl + h->tpl_len;
  a.tpl.depth = h->tpl + 2 * h->tpl_len;
  a.tpl.maxdepth = h->tpl + 3 * h->tpl_len;
  a.tpl.len = h->tpl_len;
  a.err = h->err;
  return a;
}

int assemble_impl(graft_handle* h, int32_t batch, const int32_t* d_root_tok, const int32_t* d_draft_tok,
                  const int16_t* d_draft_parent, const float* d_draft_aux, int32_t draft_nodes,
                  const int32_t* d_event, const int32_t* d_retrieved, int32_t* d_tree_tok, int8_t* d_tree_parent,
                  int32_t* d_tree_pos, uint64_t* d_tree_mask, int32_t* d_info, int8_t* d_slot_src, void* stream) {
  if (!h) return GRAFT_EINVAL;
  h->last_launches = 0;
  const graft_config& c = h->cfg;
  if (batch < 0 || batch > c.max_batch) return fail(h, GRAFT_EINVAL, "batch %d outside [0, %d]", batch, c.max_batch);
  if (draft_nodes < 0 || draft_nodes > c.max_draft_nodes)
    return fail(h, GRAFT_EINVAL, "draft_nodes %d outside [0, %d]", draft_nodes, c.max_draft_nodes);
  if (batch == 0) return GRAFT_OK;
  if (!d_root_tok || !d_tree_tok || !d_tree_parent || !d_tree_pos || !d_tree_mask || !d_info)
    return fail(h, GRAFT_EINVAL, "null pointer");
  if (draft_nodes > 0 && (!d_draft_tok || !d_draft_aux || (c.mode != GRAFT_MODE_TAIL && !d_draft_parent)))
    return fail(h, GRAFT_EINVAL, "null draft pointer");
  if (graft::misaligned(d_root_tok, 4) || graft::misaligned(d_draft_tok, 4) || graft::misaligned(d_draft_parent, 2) ||
      graft::misaligned(d_draft_aux, 4) || graft::misaligned(d_event, 4) || graft::misaligned(d_retrieved, 4) ||
      graft::misaligned(d_tree_tok, 4) || graft::misaligned(d_tree_pos, 4) || graft::misaligned(d_tree_mask, 8) ||
      graft::misaligned(d_info, 4))
    return fail(h, GRAFT_EINVAL, "a buffer is not aligned to its element size");
  graft::AssembleArgs a = assemble_args(h, batch, draft_nodes);
  a.root_tok = d_root_tok; a.draft_tok = d_draft_tok; a.draft_parent = d_draft_parent; a.draft_aux = d_draft_aux;
  a.event_in = d_event;
  a.rtok_in = d_retrieved;
  a.tree_tok = d_tree_tok; a.tree_parent = d_tree_parent; a.tree_pos = d_tree_pos; a.tree_mask = d_tree_mask;
  a.info = d_info;
  a.slot_src = d_slot_src;
  cudaError_t e;
  {
    ProfScope ps(h, (cudaStream_t)stream, "k_assemble");
    e = graft::launch_assemble(a, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_assemble launch");
  h->last_launches = 1;
  return GRAFT_OK;
}

}  // namespace

extern "C" {

int graft_assemble(graft_handle* h, int32_t batch, const int32_t* d_root_tok, const int32_t* d_draft_tok,
                   const int16_t* d_draft_parent, const float* d_draft_aux, int32_t draft_nodes, int32_t* d_tree_tok,
                   int8_t* d_tree_parent, int32_t* d_tree_pos, uint64_t* d_tree_mask, int32_t* d_info, void* stream) {
  NvtxRange nvtx("graft_assemble");
  return assemble_impl(h, batch, d_root_tok, d_draft_tok, d_draft_parent, d_draft_aux, draft_nodes, nullptr, nullptr,
                       d_tree_tok, d_tree_parent, d_tree_pos, d_tree_mask, d_info, nullptr, stream);
}

int graft_assemble_src(graft_handle* h, int32_t batch, const int32_t* d_root_tok, const int32_t* d_draft_tok,
                       const int16_t* d_draft_parent, const float* d_draft_aux, int32_t draft_nodes,
                       int32_t* d_tree_tok, int8_t* d_tree_parent, int32_t* d_tree_pos, uint64_t* d_tree_mask,
                       int32_t* d_info, int8_t* d_slot_src, void* stream) {
  NvtxRange nvtx("graft_assemble_src");
  if (!h) return GRAFT_EINVAL;
  if (batch > 0 && !d_slot_src) return fail(h, GRAFT_EINVAL, "null pointer");
  return assemble_impl(h, batch, d_root_tok, d_draft_tok, d_draft_parent, d_draft_aux, draft_nodes, nullptr, nullptr,
                       d_tree_tok, d_tree_parent, d_tree_pos, d_tree_mask, d_info, d_slot_src, stream);
}

int graft_check(graft_handle* h, int32_t batch, const int16_t* d_draft_parent, const float* d_draft_prob,
                int32_t draft_nodes, int32_t layer, int32_t* d_event, void* stream) {
  NvtxRange nvtx("graft_check");
  if (!h) return GRAFT_EINVAL;
  h->last_launches = 0;
  const graft_config& c = h->cfg;
  if (c.mode != GRAFT_MODE_CHECKPOINT) return fail(h, GRAFT_EINVAL, "graft_check needs checkpoint mode");
  if (batch < 0 || batch > c.max_batch) return fail(h, GRAFT_EINVAL, "batch %d outside [0, %d]", batch, c.max_batch);
  if (draft_nodes < 0 || draft_nodes > c.max_draft_nodes)
    return fail(h, GRAFT_EINVAL, "draft_nodes %d outside [0, %d]", draft_nodes, c.max_draft_nodes);
  if (layer < 0) return fail(h, GRAFT_EINVAL, "layer must be >= 0");
  if (batch == 0) return GRAFT_OK;
  if (!d_event || (draft_nodes > 0 && (!d_draft_parent || !d_draft_prob))) return fail(h, GRAFT_EINVAL, "null pointer");
  if (graft::misaligned(d_event, 4) || graft::misaligned(d_draft_parent, 2) || graft::misaligned(d_draft_prob, 4))
    return fail(h, GRAFT_EINVAL, "a buffer is not aligned to its element size");
  if (c.ablation == 2) return GRAFT_OK;  // the fixed split has no checkpoints
  graft::AssembleArgs a = assemble_args(h, batch, draft_nodes);
  a.draft_parent = d_draft_parent; a.draft_aux = d_draft_prob; a.layer = layer;
  cudaError_t e;
  {
    ProfScope ps(h, (cudaStream_t)stream, "k_check");
    e = graft::launch_check(a, d_event, nullptr, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_check launch");
  h->last_launches = 1;
  return GRAFT_OK;
}

int graft_retrieve(graft_handle* h, int32_t batch, const int32_t* d_root_tok, const int32_t* d_event,
                   int32_t* d_retrieved, void* stream) {
  NvtxRange nvtx("graft_retrieve");
  if (!h) return GRAFT_EINVAL;
  h->last_launches = 0;
  const graft_config& c = h->cfg;
  if (c.mode != GRAFT_MODE_CHECKPOINT) return fail(h, GRAFT_EINVAL, "graft_retrieve needs checkpoint mode");
  if (batch < 0 || batch > c.max_batch) return fail(h, GRAFT_EINVAL, "batch %d outside [0, %d]", batch, c.max_batch);
  if (batch == 0) return GRAFT_OK;
  if (!d_root_tok || !d_event || !d_retrieved) return fail(h, GRAFT_EINVAL, "null pointer");
  if (graft::misaligned(d_root_tok, 4) || graft::misaligned(d_event, 4) || graft::misaligned(d_retrieved, 4))
    return fail(h, GRAFT_EINVAL, "a buffer is not aligned to its element size");
  graft::AssembleArgs a = assemble_args(h, batch, 0);
  a.root_tok = d_root_tok;
  cudaError_t e;
  {
    ProfScope ps(h, (cudaStream_t)stream, "k_retrieve");
    e = graft::launch_retrieve(a, d_event, d_retrieved, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_retrieve launch");
  h->last_launches = 1;
  return GRAFT_OK;
}

int graft_assemble_staged(graft_handle* h, int32_t batch, const int32_t* d_root_tok, const int32_t* d_draft_tok,
                          const int16_t* d_draft_parent, const float* d_draft_prob, int32_t draft_nodes,
                          const int32_t* d_event, const int32_t* d_retrieved, int32_t* d_tree_tok,
                          int8_t* d_tree_parent, int32_t* d_tree_pos, uint64_t* d_tree_mask, int32_t* d_info,
                          void* stream) {
  NvtxRange nvtx("graft_assemble_staged");
  if (!h) return GRAFT_EINVAL;
  if (h->cfg.mode != GRAFT_MODE_CHECKPOINT) return fail(h, GRAFT_EINVAL, "graft_assemble_staged needs checkpoint mode");
  if (batch > 0 && (!d_event || !d_retrieved)) return fail(h, GRAFT_EINVAL, "null pointer");
  return assemble_impl(h, batch, d_root_tok, d_draft_tok, d_draft_parent, d_draft_prob, draft_nodes, d_event,
                       d_retrieved, d_tree_tok, d_tree_parent, d_tree_pos, d_tree_mask, d_info, nullptr, stream);
}

int graft_confidence(graft_handle* h, int32_t batch, const int16_t* d_draft_parent, const float* d_draft_prob,
                     int32_t draft_nodes, float* d_best, void* stream) {
  NvtxRange nvtx("graft_confidence");
  if (!h) return GRAFT_EINVAL;
  h->last_launches = 0;
  const graft_config& c = h->cfg;
  if (c.mode == GRAFT_MODE_TAIL) return fail(h, GRAFT_EINVAL, "graft_confidence needs a draft tree");
  if (batch < 0 || batch > c.max_batch) return fail(h, GRAFT_EINVAL, "batch %d outside [0, %d]", batch, c.max_batch);
  if (draft_nodes < 0 || draft_nodes > c.max_draft_nodes)
    return fail(h, GRAFT_EINVAL, "draft_nodes %d outside [0, %d]", draft_nodes, c.max_draft_nodes);
  if (batch == 0) return GRAFT_OK;
  if (!d_best || (draft_nodes > 0 && (!d_draft_parent || !d_draft_prob))) return fail(h, GRAFT_EINVAL, "null pointer");
  if (graft::misaligned(d_best, 4) || graft::misaligned(d_draft_parent, 2) || graft::misaligned(d_draft_prob, 4))
    return fail(h, GRAFT_EINVAL, "a buffer is not aligned to its element size");
  graft::AssembleArgs a = assemble_args(h, batch, draft_nodes);
  a.draft_parent = d_draft_parent; a.draft_aux = d_draft_prob; a.layer = INT32_MAX;
  cudaError_t e;
  {
    ProfScope ps(h, (cudaStream_t)stream, "k_check");
    e = graft::launch_check(a, nullptr, d_best, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_confidence launch");
  h->last_launches = 1;
  return GRAFT_OK;
}

int graft_template(int32_t depth, int32_t width, int32_t len, int32_t* parent_out, int32_t* rank_out,
                   int32_t* depth_out) {
  if (depth < 1 || depth > 16 || width < 1 || width > 64 || len < 0 || len > 65536) return GRAFT_EINVAL;
  if (len > 0 && (!parent_out || !rank_out || !depth_out)) return GRAFT_EINVAL;
  std::vector<int32_t> tp, tr, td;
  try {
    build_template(depth, width, len, tp, tr, td);
  } catch (...) {
    return GRAFT_ENOMEM;
  }
  for (size_t j = 0; j < tp.size(); ++j) {
    parent_out[j] = tp[j];
    rank_out[j] = tr[j];
    depth_out[j] = td[j];
  }
  return (int)tp.size();
}

int graft_calibrate_thresholds(const float* best, int32_t n_rows, double quantile, float* thr_out) {
  if (!best || !thr_out || n_rows < 0 || !(quantile > 0.0 && quantile <= 1.0)) return GRAFT_EINVAL;
  for (int k = 0; k < 3; ++k) {
    std::vector<float> v;
    for (int32_t i = 0; i < n_rows; ++i) {
      const float x = best[(int64_t)i * 3 + k];
      if (x >= 0.f && x <= 1.f) v.push_back(x);  // -1 = the layer was empty
    }
    if (v.empty()) return GRAFT_EINVAL;
    std::sort(v.begin(), v.end());
    // nearest rank: the smallest sample value with at least `quantile` of the sample at or below it
    // (1e-9 absorbs the rounding of q * n when it is an integer in exact arithmetic)
    int64_t r = (int64_t)std::ceil(quantile * (double)v.size() - 1e-9);
    if (r < 1) r = 1;
    if (r > (int64_t)v.size()) r = (int64_t)v.size();
    thr_out[k] = v[(size_t)(r - 1)];
  }
  return GRAFT_OK;
}

int graft_set_thresholds(graft_handle* h, const float* thr) {
  if (!h || !thr) return GRAFT_EINVAL;
  for (int k = 0; k < 3; ++k)
    if (!(thr[k] >= 0.f && thr[k] <= 1.f)) return fail(h, GRAFT_EINVAL, "threshold %d must be in [0, 1]", k);
  for (int k = 0; k < 3; ++k) h->cfg.ckpt_thr[k] = thr[k];
  return GRAFT_OK;
}

int graft_coverage(graft_handle* h, int32_t batch, const int32_t* d_tree_tok, const int8_t* d_tree_parent,
                   const int32_t* d_info, const void* d_logits, int64_t row_stride, float* d_gain, void* stream) {
  NvtxRange nvtx("graft_coverage");
  if (!h) return GRAFT_EINVAL;
  h->last_launches = 0;
  const graft_config& c = h->cfg;
  if (c.mode == GRAFT_MODE_STATIC) return fail(h, GRAFT_EINVAL, "graft_coverage needs checkpoint or tail mode");
  if (batch < 0 || batch > c.max_batch) return fail(h, GRAFT_EINVAL, "batch %d outside [0, %d]", batch, c.max_batch);
  if (batch == 0) return GRAFT_OK;
  if (!d_tree_tok || !d_tree_parent || !d_info || !d_logits || !d_gain) return fail(h, GRAFT_EINVAL, "null pointer");
  if (row_stride < c.vocab) return fail(h, GRAFT_EINVAL, "row_stride < vocab");
  if (graft::misaligned(d_tree_tok, 4) || graft::misaligned(d_info, 4) || graft::misaligned(d_gain, 4) ||
      graft::misaligned(d_logits, c.logits_dtype == GRAFT_BF16 ? 2 : 4))
    return fail(h, GRAFT_EINVAL, "a buffer is not aligned to its element size");
  graft::VerifyArgs a{};
  a.g = scan_geom(h, d_logits, row_stride, (int64_t)batch * h->S, h->scan_ctas_target);  // 16-byte loads when aligned
  a.S = h->S; a.batch = batch; a.logits = d_logits;
  a.tree_tok = d_tree_tok; a.tree_parent = d_tree_parent;
  cudaError_t e;
  {
    ProfScope ps(h, (cudaStream_t)stream, "k_coverage");
    e = graft::launch_coverage(a, d_info, d_gain, c.logits_dtype, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_coverage launch");
  h->last_launches = 1;
  return GRAFT_OK;
}

}  // extern "C"

namespace {

int launch_sample_step(graft_handle* h, const graft::VerifyArgs& a, void* stream) {
  cudaError_t e;
  {
    ProfScope ps(h, (cudaStream_t)stream, "k_sample");
    e = graft::launch_sample(a, h->cfg.logits_dtype, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_verify_update_sample launch");
  h->last_launches += 1;
  return GRAFT_OK;
}

// Greedy (sample = false) or stochastic verification, and the update.
int verify_impl(graft_handle* h, int32_t batch, const int32_t* d_tree_tok, const int8_t* d_tree_parent,
                const int32_t* d_tree_pos, const uint64_t* d_tree_mask, const void* d_logits, int64_t row_stride,
                int32_t* d_accept_len, int32_t* d_out_tokens, bool sample, float temperature,
                const float* d_u_accept, const float* d_u_resid, void* stream) {
  if (!h) return GRAFT_EINVAL;
  h->last_launches = 0;
  const graft_config& c = h->cfg;
  if (batch < 0 || batch > c.max_batch) return fail(h, GRAFT_EINVAL, "batch %d outside [0, %d]", batch, c.max_batch);
  if (batch == 0) return GRAFT_OK;
  if (!d_tree_tok || !d_tree_parent || !d_tree_pos || !d_tree_mask || !d_logits || !d_accept_len || !d_out_tokens)
    return fail(h, GRAFT_EINVAL, "null pointer");
  if (row_stride < c.vocab) return fail(h, GRAFT_EINVAL, "row_stride < vocab");
  if (graft::misaligned(d_tree_tok, 4) || graft::misaligned(d_tree_pos, 4) || graft::misaligned(d_tree_mask, 8) ||
      graft::misaligned(d_logits, c.logits_dtype == GRAFT_BF16 ? 2 : 4) || graft::misaligned(d_accept_len, 4) ||
      graft::misaligned(d_out_tokens, 4) || graft::misaligned(d_u_accept, 4) || graft::misaligned(d_u_resid, 4))
    return fail(h, GRAFT_EINVAL, "a buffer is not aligned to its element size");
  const int64_t rows = (int64_t)batch * h->S;
  graft::VerifyArgs a{};
  a.g = scan_geom(h, d_logits, row_stride, rows, h->scan_ctas_target);
  a.S = h->S; a.batch = batch; a.logits = d_logits;
  a.tree_tok = d_tree_tok; a.tree_parent = d_tree_parent; a.tree_pos = d_tree_pos; a.tree_mask = d_tree_mask;
  a.accept_len = d_accept_len; a.out_tokens = d_out_tokens;
  a.part = h->part; a.row_ticket = h->row_ticket; a.req_ticket = h->req_ticket; a.topk = h->topk;
  a.winner = h->winner; a.err = h->err; a.row_nseg = h->row_nseg;
  a.sample = sample ? 1 : 0;
  a.inv_temp = sample ? 1.f / temperature : 1.f;
  a.u_accept = d_u_accept; a.u_resid = d_u_resid;
  const bool tma_fits = h->tma_ready && a.g.vec && a.g.row_vec_bytes >= graft::TMA_CHUNK &&
                        a.g.cpr <= graft::MAX_SPLIT && rows <= graft::verify_tma_max_rows(h->num_sms);
  a.upr = (int32_t)((a.g.nslot + 31) / 32);
  a.ups = (a.upr + 3) & ~3;
  const int grid2 = h->num_sms * graft::two_pass_ctas_per_sm();
  const bool two_pass_fits = a.g.vec && h->umax && a.g.nslot > 0 && a.upr <= h->upr_max &&
                             rows <= graft::two_pass_max_rows(grid2);
  const bool use_tma = tma_fits && c.scan_kernel == 2;
  // few rows, each staged in a cluster's shared memory: one launch, no reload
  const int esize = c.logits_dtype == GRAFT_BF16 ? 2 : 4;
  const bool use_cluster = graft::cluster_select_fits((int)rows, c.vocab, esize) &&
                           (c.scan_kernel == 5 ||
                            (c.scan_kernel == 0 &&
                             graft::cluster_select_auto((int)rows, c.vocab, esize, h->cluster_max_active)));
  const bool use_two_pass = !use_tma && two_pass_fits && (c.scan_kernel == 0 || c.scan_kernel >= 3);
  const int grid = h->num_sms * graft::verify_ctas_per_sm();
  if (!use_tma && !use_two_pass && rows > graft::verify_max_rows(grid))
    return fail(h, GRAFT_EINVAL, "batch * (budget + 1) = %lld rows exceeds %d on this GPU", (long long)rows,
                graft::verify_max_rows(grid));
  a.umax = h->umax;
  a.usec = h->usec;
  a.upos = h->upos;
  a.top2 = (c.scan_kernel == 4 && h->usec && h->upos) ? 1 : 0;
  a.spec = c.mode == GRAFT_MODE_STATIC ? 1 : 0;  // static trees fill every slot
  a.wait_polls = h->wait_polls;  // measured: the records slow pass 1 by more than they save
  cudaError_t e;
  if (use_cluster) {
    {
      ProfScope ps(h, (cudaStream_t)stream, "k_cluster_select");
      e = graft::launch_cluster_select(a, c.logits_dtype, h->C, (cudaStream_t)stream);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "graft_verify_update cluster launch");
    h->last_launches = 1;
    return sample ? launch_sample_step(h, a, stream) : GRAFT_OK;
  }
  if (use_two_pass) {
    {
      ProfScope ps(h, (cudaStream_t)stream, "k_umax");
      e = graft::launch_two_pass_umax(a, c.logits_dtype, grid2, (cudaStream_t)stream);
    }
    if (e == cudaSuccess) {
      ProfScope ps(h, (cudaStream_t)stream, "k_select");
      e = graft::launch_two_pass_select(a, c.logits_dtype, h->C, (cudaStream_t)stream);
    }
    if (e != cudaSuccess) return cuda_fail(h, e, "graft_verify_update two-pass launch");
    h->last_launches = 2;
    return sample ? launch_sample_step(h, a, stream) : GRAFT_OK;
  }
  {
    ProfScope ps(h, (cudaStream_t)stream, use_tma ? "k_verify_tma" : "k_verify");
    e = use_tma ? graft::launch_verify_tma(a, c.logits_dtype, h->num_sms, (cudaStream_t)stream)
                : graft::launch_verify(a, c.logits_dtype, grid, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_verify_update scan launch");
  {
    ProfScope ps(h, (cudaStream_t)stream, "k_finish");
    e = graft::launch_finish(a, h->C, (cudaStream_t)stream);
  }
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_verify_update finish launch");
  h->last_launches = 2;
  return sample ? launch_sample_step(h, a, stream) : GRAFT_OK;
}

}  // namespace

extern "C" {

int graft_verify_update(graft_handle* h, int32_t batch, const int32_t* d_tree_tok, const int8_t* d_tree_parent,
                        const int32_t* d_tree_pos, const uint64_t* d_tree_mask, const void* d_logits,
                        int64_t row_stride, int32_t* d_accept_len, int32_t* d_out_tokens, void* stream) {
  NvtxRange nvtx("graft_verify_update");
  return verify_impl(h, batch, d_tree_tok, d_tree_parent, d_tree_pos, d_tree_mask, d_logits, row_stride, d_accept_len,
                     d_out_tokens, false, 1.f, nullptr, nullptr, stream);
}

int graft_verify_update_sample(graft_handle* h, int32_t batch, const int32_t* d_tree_tok, const int8_t* d_tree_parent,
                               const int32_t* d_tree_pos, const uint64_t* d_tree_mask, const void* d_logits,
                               int64_t row_stride, float temperature, const float* d_u_accept,
                               const float* d_u_resid, int32_t* d_accept_len, int32_t* d_out_tokens, void* stream) {
  NvtxRange nvtx("graft_verify_update_sample");
  if (!h) return GRAFT_EINVAL;
  if (!(temperature > 0.f) || !std::isfinite(temperature) || !std::isfinite(1.f / temperature))
    return fail(h, GRAFT_EINVAL, "temperature must be finite and > 0, with a finite inverse");
  if (batch > 0 && (!d_u_accept || !d_u_resid)) return fail(h, GRAFT_EINVAL, "null pointer");
  return verify_impl(h, batch, d_tree_tok, d_tree_parent, d_tree_pos, d_tree_mask, d_logits, row_stride, d_accept_len,
                     d_out_tokens, true, temperature, d_u_accept, d_u_resid, stream);
}



int graft_get_matrix(graft_handle* h, int32_t* host_out, void* stream) {
  if (!h || !host_out) return fail(h, GRAFT_EINVAL, "null pointer");
  const size_t bytes = (size_t)h->cfg.vocab * graft::K * sizeof(int32_t);
  cudaError_t e = cudaMemcpyAsync(host_out, h->C, bytes, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  return e == cudaSuccess ? GRAFT_OK : cuda_fail(h, e, "graft_get_matrix");
}

int graft_set_matrix(graft_handle* h, const int32_t* host_in, void* stream) {
  if (!h || !host_in) return fail(h, GRAFT_EINVAL, "null pointer");
  const size_t bytes = (size_t)h->cfg.vocab * graft::K * sizeof(int32_t);
  cudaError_t e = cudaMemcpyAsync(h->C, host_in, bytes, cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
  return e == cudaSuccess ? GRAFT_OK : cuda_fail(h, e, "graft_set_matrix");
}

int32_t* graft_matrix_device_ptr(graft_handle* h) { return h ? h->C : nullptr; }

int graft_sync(graft_handle* h, void* stream, uint32_t* out_flags) {
  if (!h) return GRAFT_EINVAL;
  uint32_t flags = 0;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e == cudaSuccess) e = cudaMemcpy(&flags, h->err, sizeof flags, cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && flags) e = cudaMemset(h->err, 0, sizeof(uint32_t));
  if (out_flags) *out_flags = flags;
  if (e != cudaSuccess) return cuda_fail(h, e, "graft_sync");
  if (flags) return fail(h, GRAFT_EDEVICE, "device error flags 0x%x (token %d, nan %d, tree %d, timeout %d)", flags,
                         !!(flags & GRAFT_ERR_TOKEN), !!(flags & GRAFT_ERR_NAN), !!(flags & GRAFT_ERR_TREE),
                         !!(flags & GRAFT_ERR_TIMEOUT));
  return GRAFT_OK;
}

const char* graft_last_error(const graft_handle* h) { return h ? h->msg : "null handle"; }

int32_t graft_last_launch_count(const graft_handle* h) { return h ? h->last_launches : 0; }

int graft_set_wait_limit(graft_handle* h, uint32_t polls) {
  if (!h) return GRAFT_EINVAL;
  h->wait_polls = polls;
  return GRAFT_OK;
}

int graft_profile_enable(graft_handle* h, int32_t on) {
  if (!h) return GRAFT_EINVAL;
  if (on && !h->prof_ev[0]) {
    for (auto& e : h->prof_ev)
      if (cudaEventCreate(&e) != cudaSuccess) return cuda_fail(h, cudaGetLastError(), "graft_profile_enable");
  }
  h->profiling = on != 0;
  h->prof_n = 0;
  return GRAFT_OK;
}

int graft_profile_read(graft_handle* h, const char** names, float* ms, int32_t max) {
  if (!h || (max > 0 && (!names || !ms))) return GRAFT_EINVAL;
  if (cudaDeviceSynchronize() != cudaSuccess) return cuda_fail(h, cudaGetLastError(), "graft_profile_read");
  const int n = h->prof_n < max ? h->prof_n : max;
  for (int i = 0; i < n; ++i) {
    names[i] = h->prof_name[i];
    ms[i] = 0.f;
    cudaEventElapsedTime(&ms[i], h->prof_ev[2 * i], h->prof_ev[2 * i + 1]);
  }
  h->prof_n = 0;
  return n;
}

}  // extern "C"
