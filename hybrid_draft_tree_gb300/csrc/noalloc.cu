// graft_verify_update_noalloc: the verify + update step without any device
// allocation, for callers that cannot call cudaMalloc.
//
// Who needs it: a serving engine that records its decode step into a CUDA
// graph cannot allocate while the stream is being captured, and engines that
// hand all device memory to their own pre-planned arena (or to another
// runtime's caching allocator) cannot take a stray cudaMalloc without failing
// or fragmenting it.  Such callers cannot create a graft_handle (graft_init
// allocates), so this entry point takes the continuation matrix as a caller
// buffer and keeps its scratch in a fixed device array in this file.
//
// The scratch (partial top-8s per row segment, segment counts, staged top-8s)
// lives in `g_scratch`, a file-scope __device__ array of GRAFT_NOALLOC_BYTES
// bytes.  Every GPU that loads this library holds it until the process exits.
// Host code may not use the array's name as a device address (in host code it
// names a host-side stand-in), so the device address is obtained once per
// device with cudaGetSymbolAddress, with that device current, on the first
// call made on it.  The address belongs to the device's context: it is kept
// with that context's id and looked up again when the current context is a
// different one (after cudaDeviceReset, or once the primary context was
// released and created anew).
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "graft_internal.cuh"

namespace {

constexpr int kMaxRows = GRAFT_NOALLOC_MAX_ROWS;
constexpr size_t kPartBytes = (size_t)kMaxRows * graft::MAX_SPLIT * graft::K * sizeof(unsigned long long);
constexpr size_t kNsegBytes = (size_t)kMaxRows * sizeof(int32_t);
constexpr size_t kTopkBytes = (size_t)kMaxRows * graft::K * sizeof(int32_t);
constexpr size_t kBytes = kPartBytes + kNsegBytes + kTopkBytes;
static_assert(kBytes == GRAFT_NOALLOC_BYTES, "scratch size mismatch with graft.h");

__device__ __align__(256) unsigned char g_scratch[kBytes];

constexpr int kMaxDevices = 64;
struct DeviceSetup {
  bool ready = false;
  unsigned long long ctx_id = 0;     // id of the context the address below belongs to
  unsigned char* scratch = nullptr;  // device address of g_scratch on this device
  int num_sms = 0;
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

// Driver entry points reached through the runtime (the library does not link
// the driver library itself).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Id of the calling thread's current context (unique for the process's
// lifetime: a context made after a reset gets a new id); 0 when the thread
// has no current context yet.  Call with the mutex held.
int current_context_id(unsigned long long* id) {
  *id = 0;
  if (!g_ctx_get_current || !g_ctx_get_id) {
    cudaDriverEntryPointQueryResult q1, q2;
    void* f1 = nullptr;
    void* f2 = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1) != cudaSuccess ||
        q1 != cudaDriverEntryPointSuccess || !f1)
      return GRAFT_ECUDA;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
        q2 != cudaDriverEntryPointSuccess || !f2)
      return GRAFT_ECUDA;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS) return GRAFT_ECUDA;
  if (ctx == nullptr) return GRAFT_OK;
  if (g_ctx_get_id(ctx, id) != CUDA_SUCCESS) return GRAFT_ECUDA;
  return GRAFT_OK;
}

// The scratch address and SM count of the current device, looked up on the
// first call made on it, and again whenever the current context is not the
// one the address was taken in.  `stream` must belong to the current device.
int setup_current_device(void* stream, DeviceSetup** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GRAFT_ECUDA;
  int sdev = -1;
  if (cudaStreamGetDevice((cudaStream_t)stream, &sdev) != cudaSuccess) return GRAFT_EINVAL;
  if (sdev != dev) return GRAFT_EINVAL;  // the stream (and so the buffers) of another device
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  unsigned long long ctx_id = 0;
  if (current_context_id(&ctx_id) != GRAFT_OK) return GRAFT_ECUDA;
  DeviceSetup& d = g_setup[dev];
  if (!d.ready || ctx_id == 0 || d.ctx_id != ctx_id) {
    d.ready = false;
    void* ptr = nullptr;
    // (makes the device's primary context current on this thread if it was not)
    if (cudaGetSymbolAddress(&ptr, g_scratch) != cudaSuccess || ptr == nullptr) return GRAFT_ECUDA;
    if (current_context_id(&ctx_id) != GRAFT_OK || ctx_id == 0) return GRAFT_ECUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
      return GRAFT_ECUDA;
    d.scratch = static_cast<unsigned char*>(ptr);
    d.num_sms = sms;
    d.ctx_id = ctx_id;
    d.ready = true;
  }
  *out = &d;
  return GRAFT_OK;
}

}  // namespace

extern "C" int graft_verify_update_noalloc(int32_t vocab, int32_t logits_dtype, int32_t batch, int32_t slots,
                                           const int32_t* d_tree_tok, const int8_t* d_tree_parent,
                                           const int32_t* d_tree_pos, const uint64_t* d_tree_mask,
                                           const void* d_logits, int64_t row_stride, int32_t* d_matrix,
                                           int32_t* d_accept_len, int32_t* d_out_tokens, uint32_t* d_err_flags,
                                           void* stream) {
  if (vocab < 1 || (logits_dtype != GRAFT_F32 && logits_dtype != GRAFT_BF16)) return GRAFT_EINVAL;
  if (slots < 1 || slots > graft::MAX_S || batch < 0) return GRAFT_EINVAL;
  if (batch == 0) return GRAFT_OK;
  const int64_t rows = (int64_t)batch * slots;
  if (rows > kMaxRows) return GRAFT_EINVAL;  // beyond the fixed scratch
  if (row_stride < vocab) return GRAFT_EINVAL;
  if (!d_tree_tok || !d_tree_parent || !d_tree_pos || !d_tree_mask || !d_logits || !d_matrix || !d_accept_len ||
      !d_out_tokens || !d_err_flags)
    return GRAFT_EINVAL;
  if (graft::misaligned(d_tree_tok, 4) || graft::misaligned(d_tree_pos, 4) || graft::misaligned(d_tree_mask, 8) ||
      graft::misaligned(d_logits, logits_dtype == GRAFT_BF16 ? 2 : 4) || graft::misaligned(d_matrix, 4) ||
      graft::misaligned(d_accept_len, 4) || graft::misaligned(d_out_tokens, 4) || graft::misaligned(d_err_flags, 4))
    return GRAFT_EINVAL;  // a buffer not aligned to its element size
  DeviceSetup* dev = nullptr;
  const int rc = setup_current_device(stream, &dev);
  if (rc != GRAFT_OK) return rc;
  const int grid = dev->num_sms * graft::verify_ctas_per_sm();
  if (rows > graft::verify_max_rows(grid)) return GRAFT_EINVAL;

  // scan geometry: 16-byte vector loads when every row start is 16-byte aligned
  graft::ScanGeom g{};
  const int es = logits_dtype == GRAFT_BF16 ? 2 : 4;
  g.V = vocab;
  g.stride = row_stride;
  g.vec = ((reinterpret_cast<uintptr_t>(d_logits) & 15) == 0) && ((row_stride * es) % 16 == 0);
  g.epl = g.vec ? 16 / es : 1;
  g.nslot = vocab / g.epl;
  g.tail = (int32_t)(vocab - g.nslot * g.epl);
  g.nsplit = 1;
  g.per_cta = g.nslot;
  g.row_vec_bytes = g.nslot * 16;
  g.cpr = 1;

  graft::VerifyArgs a{};
  a.g = g;
  a.S = slots;
  a.batch = batch;
  a.logits = d_logits;
  a.tree_tok = d_tree_tok;
  a.tree_parent = d_tree_parent;
  a.tree_pos = d_tree_pos;
  a.tree_mask = d_tree_mask;
  a.accept_len = d_accept_len;
  a.out_tokens = d_out_tokens;
  a.part = reinterpret_cast<unsigned long long*>(dev->scratch);
  a.row_nseg = reinterpret_cast<int32_t*>(dev->scratch + kPartBytes);
  a.topk = reinterpret_cast<int32_t*>(dev->scratch + kPartBytes + kNsegBytes);
  a.err = d_err_flags;
  // Every entry the kernels read is written earlier in the same call (segment
  // counts and partials by the scan, staged top-8s before acceptance reads
  // them), so nothing left by a previous call needs clearing.
  cudaError_t e = graft::launch_verify(a, logits_dtype, grid, (cudaStream_t)stream);
  if (e == cudaSuccess) e = graft::launch_finish(a, d_matrix, (cudaStream_t)stream);
  return e == cudaSuccess ? GRAFT_OK : GRAFT_ECUDA;
}
