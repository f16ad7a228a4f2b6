// fill_noalloc.cu -- ridgefill_fill_noalloc: the attention fill without a
// caller-provided workspace.
//
// Some callers have no way to obtain device memory on demand: a host engine
// that hands out every device buffer itself and offers plugins no allocator,
// or code that runs once the engine has divided up all of device memory.
// Such callers can still pass their inputs and outputs, but not a workspace.
// This entry point keeps its scratch (the predicted layer inputs of one row
// chunk and their sums of squares) in a fixed-size array in device global
// memory that belongs to the library.  Every GPU that loads the library holds
// that array until the process exits.
//
// Notes for callers:
//  - The array is shared by every call on a device and keeps the contents of
//    the last call.  Nothing in it has to start at zero: each chunk writes
//    every scratch element it later reads.  Two calls whose work overlaps on
//    the GPU (different streams without ordering, or different host threads)
//    race on the array; order them on one stream.
//  - The first call on a device looks up the array's device address (once per
//    device and context, with that device current); make that first call
//    before any stream capture.
//  - Host-memory maps (maps_on_host = 1) are not supported here: their three
//    map slots would not fit in the array.  Nor is a split state in host
//    memory (h_on_host = 1).
//  - The call itself allocates nothing: no cudaMalloc, cudaFree or allocating
//    library routine.
#include <mutex>

#include "abi_common.h"

namespace rf {
namespace {

static __device__ __align__(256) unsigned char g_fill_scratch[RF_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the context current on this thread (driver entry points looked up once).
rf_status current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (get_cur == nullptr || get_id == nullptr)
    return fail(RF_ERR_CUDA, "driver entry points cuCtxGetCurrent / cuCtxGetId unavailable");
  CUcontext ctx = nullptr;
  if (get_cur(&ctx) != CUDA_SUCCESS) return fail(RF_ERR_CUDA, "cuCtxGetCurrent failed");
  *id = 0;  // no context current yet
  if (ctx != nullptr && get_id(ctx, id) != CUDA_SUCCESS)
    return fail(RF_ERR_CUDA, "cuCtxGetId failed");
  return RF_OK;
}

// Device address of g_fill_scratch in the current device's context (host code must not
// use the symbol itself: on the host it only names a stand-in).  Looked up the first time
// a device is used and again whenever that device's context has changed since (a reset
// gives it a new context and the array a new address).
rf_status scratch_address(void** out) {
  static void* addr[kMaxDev] = {};
  static unsigned long long ctx_of[kMaxDev] = {};
  static std::mutex mu;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDev) return fail(RF_ERR_CUDA, "device index %d out of range", dev);
  unsigned long long ctx = 0;
  rf_status st = current_context_id(&ctx);
  if (st != RF_OK) return st;
  std::lock_guard<std::mutex> lk(mu);
  if (addr[dev] == nullptr || ctx == 0 || ctx_of[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fill_scratch);  // initialises the context if needed
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    if (ctx == 0 && (st = current_context_id(&ctx)) != RF_OK) return st;
    addr[dev] = p;
    ctx_of[dev] = ctx;
  }
  *out = addr[dev];
  return RF_OK;
}

}  // namespace
}  // namespace rf

using namespace rf;

extern "C" rf_status ridgefill_fill_noalloc(const rf_fill_args* a, void* stream) {
  if (a == nullptr) return fail(RF_ERR_ARG, "args is NULL");
  if (a->maps_on_host != 0)
    return fail(RF_ERR_ARG, "ridgefill_fill_noalloc does not stream host maps (maps_on_host = 1)");
  if (a->h_on_host != 0)
    return fail(RF_ERR_ARG, "ridgefill_fill_noalloc does not stream a host split state (h_on_host = 1)");
  rf_fill_args c = *a;
  // int8 maps: the codes are converted inside the map GEMM unless the caller asked for layer
  // groups (whose bf16 copies would take most of the fixed scratch)
  if (c.A_scale != nullptr && c.q8_group_layers == 0) c.q8_group_layers = -1;
  // largest chunk (multiple of 128 rows) whose workspace fits the static scratch
  const int64_t want = a->rows_per_chunk > 0 ? a->rows_per_chunk
                                             : ceil_div(a->rows > 0 ? a->rows : 1, kBM) * kBM;
  int64_t best = 0;
  for (int64_t r = kBM; r <= want; r += kBM) {
    c.rows_per_chunk = r;
    const size_t need = ridgefill_fill_workspace_size(&c);
    if (need == 0) return ridgefill_fill(&c, nullptr, 0, stream);  // reports the argument error
    if (need > RF_NOALLOC_SCRATCH_BYTES) break;
    best = r;
  }
  if (best == 0) {
    c.rows_per_chunk = kBM;
    return fail(RF_ERR_WORKSPACE,
                "ridgefill_fill_noalloc: one 128-row chunk needs %zu bytes of scratch but the "
                "static scratch holds %zu bytes (reduce n_layers * d_out or use ridgefill_fill)",
                ridgefill_fill_workspace_size(&c), static_cast<size_t>(RF_NOALLOC_SCRATCH_BYTES));
  }
  c.rows_per_chunk = best;
  void* scratch = nullptr;
  rf_status st = scratch_address(&scratch);
  if (st != RF_OK) return st;
  return ridgefill_fill(&c, scratch, RF_NOALLOC_SCRATCH_BYTES, stream);
}
