// Internal declarations shared by the CUDA translation units of libgraft.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "graft.h"

namespace graft {

constexpr int K = 8;            // successors per continuation-matrix row
constexpr int MAX_S = 64;       // slots per request (one uint64 mask row)
constexpr int MAX_DRAFT = 256;  // draft nodes per request in one assemble CTA
constexpr int MAX_SPLIT = 16;   // CTAs per logits row in the verify scan
constexpr int TMA_CHUNK = 32768; // bytes per pipeline stage of the TMA verify scan
constexpr int TWO_PASS_MAX_ROWS = 4096;   // verified rows per call on the two-pass scan
constexpr int TWO_PASS_MAX_UNITS = 1024;  // 512-byte units per row on the two-pass scan (512 KB rows)
constexpr int WARM_TWO_PASS_ROWS = 4096;  // warm-up rows per call on the two-pass scan (the rest: single pass)
constexpr int CLUSTER_MAX_ROWS = 256;     // verified rows per call on the cluster-per-row verify
constexpr int CLUSTER_STAGE_MAX = 200 * 1024;  // shared-memory bytes of one CTA's eighth of a row there
constexpr int CLUSTER_AUTO_ROWS = 256;    // the automatic choice takes the cluster-per-row verify up to here
constexpr int CLUSTER_AUTO_STAGE = 48 * 1024;  // ... and up to this many bytes of a row per CTA

// Template entry j (j < tpl_len): parent entry (-1 = anchor), rank, depth;
// maxdepth[R] = the largest depth among entries 0 .. R-1 (maxdepth[0] = 0).
struct TemplateDev {
  const int32_t* parent;
  const int32_t* rank;
  const int32_t* depth;
  const int32_t* maxdepth;
  int32_t len;
};

struct AssembleArgs {
  int32_t mode, V, budget, S, n, batch;
  int32_t ckpt_depth[3];
  float ckpt_thr[3];
  int32_t ckpt_draft[3];
  float static_thr, tail_thr;
  int32_t ablation, fixed_draft;
  int32_t layer;              // graft_check: deepest complete draft layer
  const int32_t* event_in;    // graft_assemble_staged: checkpoint verdicts, or nullptr
  const int32_t* rtok_in;     // graft_assemble_staged: gathered retrieval entries [batch][budget], or nullptr
  const int32_t* root_tok;
  const int32_t* draft_tok;
  const int16_t* draft_parent;
  const float* draft_aux;
  const int32_t* C;
  TemplateDev tpl;
  int32_t* tree_tok;
  int8_t* tree_parent;
  int32_t* tree_pos;
  uint64_t* tree_mask;
  int32_t* info;
  int8_t* slot_src;           // [batch][S] slot provenance (0 root, 1 draft, 2 retrieved, -1 pad), or nullptr
  uint32_t* err;
};

struct ScanGeom {
  int32_t V;          // elements per row
  int64_t stride;     // elements between row starts
  int32_t vec;        // 1 = 16-byte vector loads, 0 = scalar loads
  int32_t epl;        // elements per load slot (8 bf16 / 4 f32 when vec, else 1)
  int64_t nslot;      // load slots per row (full vectors only when vec)
  int32_t tail;       // elements after the last full vector (vec only)
  int32_t nsplit;     // CTAs per row
  int64_t per_cta;    // load slots per CTA
  int32_t cpr;        // TMA scan: 32 KB chunks per row
  int64_t row_vec_bytes;  // bytes of a row's full 16-byte vectors
};

// True when device pointer p is not aligned to a (a power of two) bytes;
// the ABI refuses such buffers (a null pointer counts as aligned: the null
// checks are separate).
inline bool misaligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; }

struct VerifyArgs {
  ScanGeom g;
  int32_t S, batch;
  const void* logits;
  const int32_t* tree_tok;
  const int8_t* tree_parent;
  const int32_t* tree_pos;
  const uint64_t* tree_mask;
  int32_t* accept_len;
  int32_t* out_tokens;
  unsigned long long* part;   // [rows][MAX_SPLIT][K] partial top-8 keys
  int32_t* row_ticket;        // [rows]
  int32_t* req_ticket;        // [batch]
  int32_t sample;             // 1: acceptance by stochastic verification (k_sample), not greedy
  float inv_temp;             // stochastic verification: 1 / temperature
  const float* u_accept;      // stochastic verification: [batch][S] uniforms, one per candidate slot
  const float* u_resid;       // stochastic verification: [batch] uniforms for the final draw
  int32_t* topk;              // [rows][K] staged top-8 ids
  int32_t* winner;            // [V] last-writer key (row + 1), 0 = none
  int32_t* row_nseg;          // [rows] number of partial top-8s the scan wrote for the row
  float* umax;                // two-pass scan: [rows][ups] maximum of every 512-byte unit
  float* usec;                // two-pass scan with top2: [rows][ups] second largest element of every unit
  uint8_t* upos;              // two-pass scan with top2: [rows][ups] position of the unit's maximum in the unit
  int32_t top2;               // two-pass scan: 1 = units record (max, second, position), 0 = max only
  int32_t spec;               // two-pass scan: 1 = every row is expected valid (static trees): pass 1 prefetches
                              // its first groups into L2 before the rows' validity is known
  uint32_t wait_polls;        // TMA scan: polls before an mbarrier wait gives up (0 = the kernel's default)
  int32_t upr;                // two-pass scan: units per row
  int32_t ups;                // two-pass scan: row stride of umax (upr rounded up to a multiple of 4)
  uint32_t* err;
};


struct WarmArgs {
  ScanGeom g;
  int64_t n_rows;
  int32_t start;      // the single-pass scan takes list entries from here on
  const void* logits;
  const int32_t* tokens;
  int32_t* winner;
  int32_t* list;
  int32_t* count;
  int32_t* C;
  uint32_t* err;
};

// L2 residency of the small, hot state (the continuation matrix and the
// flattened trees): evict-last cache policy on their loads and stores, while
// the logits stream through with evict-first loads.
// Programmatic dependent launch.  A kernel launched with programmatic stream
// serialization may begin before the kernel ahead of it in the stream ends;
// grid_dependency_wait() blocks until that kernel has finished and its
// writes are visible (a no-op for an ordinary launch).  The kernel ahead
// calls grid_dependents_launch() to let the dependent grid be scheduled.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Launch `kernel` as a programmatic dependent of the kernel ahead of it in
// the stream (it must call grid_dependency_wait() before reading that
// kernel's results).
template <class... P, class... A>
cudaError_t launch_dependent(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, A... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

__device__ __forceinline__ uint64_t l2_keep_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// Fetch the line holding ptr into L2 with the evict-last priority (no data returned).
__device__ __forceinline__ void prefetch_keep(const void* ptr) {
  asm volatile("prefetch.global.L2::evict_last [%0];" ::"l"(ptr));
}
// A plain prefetch of the 128-byte line holding ptr into L2.
__device__ __forceinline__ void prefetch_l2(const void* ptr) { asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr)); }
__device__ __forceinline__ int32_t ld_keep(const int32_t* ptr, uint64_t pol) {
  int32_t v;
  asm volatile("ld.global.L2::cache_hint.s32 %0, [%1], %2;" : "=r"(v) : "l"(ptr), "l"(pol) : "memory");
  return v;
}
__device__ __forceinline__ void st_keep(int32_t* ptr, int32_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.s32 [%0], %1, %2;" ::"l"(ptr), "r"(v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep(int8_t* ptr, int8_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b8 [%0], %1, %2;" ::"l"(ptr), "h"((short)v), "l"(pol) : "memory");
}
__device__ __forceinline__ void st_keep(uint64_t* ptr, uint64_t v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;" ::"l"(ptr), "l"(v), "l"(pol) : "memory");
}

// launchers (return cudaGetLastError())
cudaError_t launch_assemble(const AssembleArgs& a, cudaStream_t s);
cudaError_t launch_check(const AssembleArgs& a, int32_t* event, float* best_out, cudaStream_t s);
cudaError_t launch_coverage(const VerifyArgs& a, const int32_t* info, float* gain, int dtype, cudaStream_t s);
cudaError_t launch_sample(const VerifyArgs& a, int dtype, cudaStream_t s);
cudaError_t launch_retrieve(const AssembleArgs& a, const int32_t* event, int32_t* out, cudaStream_t s);
cudaError_t launch_verify(const VerifyArgs& a, int dtype, int grid, cudaStream_t s);
int verify_ctas_per_sm();
int verify_max_rows(int grid);
cudaError_t prepare_verify_tma();
cudaError_t launch_verify_tma(const VerifyArgs& a, int dtype, int grid, cudaStream_t s);
size_t verify_tma_smem_bytes();
int verify_tma_max_rows(int grid);
cudaError_t launch_finish(const VerifyArgs& a, int32_t* C, cudaStream_t s);
cudaError_t launch_two_pass_umax(const VerifyArgs& a, int dtype, int grid, cudaStream_t s);
cudaError_t launch_two_pass_select(const VerifyArgs& a, int dtype, int32_t* C, cudaStream_t s);
bool cluster_select_fits(int rows, int V, int esize);
bool cluster_select_auto(int rows, int V, int esize, int max_active);
int cluster_select_max_active(int V, int dtype);
cudaError_t launch_cluster_select(const VerifyArgs& a, int dtype, int32_t* C, cudaStream_t s);
int two_pass_ctas_per_sm();
int two_pass_max_rows(int grid);
cudaError_t launch_warmup_begin(const WarmArgs& a, cudaStream_t s);
cudaError_t launch_warmup_scan(const WarmArgs& a, int dtype, int grid_ctas, cudaStream_t s);
cudaError_t launch_warmup_end(const WarmArgs& a, cudaStream_t s);
cudaError_t launch_warm_umax(const VerifyArgs& a, const int32_t* list, const int32_t* count, int cap, int dtype,
                             int grid, cudaStream_t s);
cudaError_t launch_warm_select(const VerifyArgs& a, const int32_t* tokens, const int32_t* list, const int32_t* count,
                               int cap, int32_t* C, int dtype, int grid, cudaStream_t s);

}  // namespace graft
