// abi_common.cu -- status handling, tensor-map encoding, per-device state,
// and the map-GEMM launch shared by the attention and GDN fills.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <mutex>
#include <string>

#include "abi_common.h"
#include "sm103_ptx.cuh"

namespace rf {

namespace {
thread_local std::string g_last_error;
constexpr int kMaxDevices = 64;
__device__ int g_device_error = 0;
constexpr int kTileCtrSlots = 1024;
__device__ int g_tile_ctr[kTileCtrSlots];
__device__ uint32_t g_probe_flag = 0;  // never written: the flag ridgefill_wait_selftest waits on

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
  });
  return fn;
}

int current_device() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}
}  // namespace

rf_status fail(rf_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

rf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(RF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

const char* last_error_cstr() { return g_last_error.c_str(); }
void clear_last_error() { g_last_error.clear(); }

int* device_error_word() {
  static int* ptr[kMaxDevices] = {};
  static std::mutex mu;
  const int d = current_device();
  if (d < 0) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
    ptr[d] = static_cast<int*>(p);
  }
  return ptr[d];
}

int* tile_counter_slot() {
  static int* base[kMaxDevices] = {};
  static std::atomic<unsigned> seq{0};
  static std::mutex mu;
  const int d = current_device();
  if (d < 0) return nullptr;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (base[d] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_tile_ctr) != cudaSuccess) return nullptr;
      base[d] = static_cast<int*>(p);
    }
  }
  return base[d] + (seq.fetch_add(1) % kTileCtrSlots);
}

bool make_tmap_4d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base,
                  const uint64_t (&dims)[4], const uint64_t (&strides)[3], const uint32_t (&box)[4],
                  CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
  cuuint32_t b[4] = {box[0], box[1], box[2], box[3]};
  cuuint32_t es[4] = {1, 1, 1, 1};
  CUresult r = fn(tm, dtype, 4, const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int sm_count() {
  static int cnt[kMaxDevices] = {};
  const int d = current_device();
  if (d < 0) return 0;
  if (cnt[d] == 0) {
    int c = 0;
    if (cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, d) != cudaSuccess) return 0;
    cnt[d] = c;
  }
  return cnt[d];
}

bool make_tmap_3d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base, uint64_t d0,
                  uint64_t d1, uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t box0,
                  uint32_t box1, CUtensorMapSwizzle swizzle) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  if (d2 <= 1) {
    d2 = 1;
    stride2 = stride1 * (d1 > 0 ? d1 : 1);
  }
  cuuint64_t dims[3] = {d0, d1, d2};
  cuuint64_t strides[2] = {stride1, stride2};
  cuuint32_t box[3] = {box0, box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(tm, dtype, 3, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

StreamWrite32 stream_write32() {
  static StreamWrite32 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &p, 11070, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<StreamWrite32>(p);
  });
  return fn;
}

std::mutex& host_stream_mutex() {
  static std::mutex mu;
  return mu;
}

size_t host_rows_bytes(int64_t rows, int d_in, size_t* flags_off) {
  const size_t data = align_up(static_cast<size_t>(rows) * d_in * 2, 256);
  *flags_off = data;
  return data + align_up(static_cast<size_t>(host_row_groups(rows)) * 4, 256);
}

rf_status stream_host_rows(HostStreamer* hs, const void* H, int64_t rows, int d_in, uint8_t* dev,
                           uint32_t* flags, cudaStream_t s, HostRows* out) {
  out->flags = flags;
  out->gen = ++hs->h_gen == 0 ? ++hs->h_gen : hs->h_gen;
  const int64_t groups = host_row_groups(rows);
  StreamWrite32 wr = stream_write32();
  out->overlap = wr != nullptr;
  // clear the flags, in order on `s` (one call: few API calls keep the host ahead of the GPU)
  cudaError_t e = cudaMemsetAsync(flags, 0, static_cast<size_t>(groups) * 4, s);
  const uint8_t* src = static_cast<const uint8_t*>(H);
  if (e == cudaSuccess) e = cudaEventRecord(hs->start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs->copy, hs->start, 0);
  for (int64_t g = 0; g < groups && e == cudaSuccess; ++g) {
    const int64_t r0 = g == 0 ? 0 : kHostFirstRows + (g - 1) * kHostRowGroup;
    const int64_t gr = g == 0 ? kHostFirstRows : kHostRowGroup;
    const int64_t nr = rows - r0 < gr ? rows - r0 : gr;
    const size_t off = static_cast<size_t>(r0) * d_in * 2;
    e = cudaMemcpyAsync(dev + off, src + off, static_cast<size_t>(nr) * d_in * 2,
                        cudaMemcpyHostToDevice, hs->copy);
    if (e == cudaSuccess && out->overlap &&
        wr(reinterpret_cast<CUstream>(hs->copy), reinterpret_cast<CUdeviceptr>(flags + g), out->gen,
           0) != CUDA_SUCCESS)
      e = cudaErrorUnknown;
  }
  if (e == cudaSuccess) e = cudaEventRecord(hs->h_done, hs->copy);
  if (e == cudaSuccess && !out->overlap) e = cudaStreamWaitEvent(s, hs->h_done, 0);
  if (e != cudaSuccess) return cuda_fail(e, "streaming the split state from host memory");
  out->base = dev;
  return RF_OK;
}

HostStreamer* host_streamer() {
  static HostStreamer hs[kMaxDevices];
  static std::mutex mu;
  const int d = current_device();
  if (d < 0) {
    fail(RF_ERR_CUDA, "no current CUDA device");
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  HostStreamer& h = hs[d];
  if (h.copy == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&h.copy, cudaStreamNonBlocking);
    for (int i = 0; i < kMapSlots && e == cudaSuccess; ++i) {
      e = cudaEventCreateWithFlags(&h.copied[i], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.freed[i], cudaEventDisableTiming);
    }
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&h.side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.side_start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.side_done, cudaEventDisableTiming);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i)
      e = cudaEventCreateWithFlags(&h.side_ev[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.start, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&h.h_done, cudaEventDisableTiming);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i)
      e = cudaEventCreateWithFlags(&h.staged[i], cudaEventDisableTiming);
    if (e != cudaSuccess) {
      cuda_fail(e, "creating the map-copy stream");
      h.copy = nullptr;
      return nullptr;
    }
  }
  return &h;
}

rf_status launch_map(const MapLaunch& m, cudaStream_t s) {
  GemmParams p{};
  p.mode = kModeMap;
  p.k_blocks = m.d_in / kBK;
  const bool single = m.slot_layer >= 0;
  const int slot_layers = m.slot_count > 0 ? m.slot_count : 1;
  const uint64_t brows = single ? static_cast<uint64_t>(slot_layers) * m.d_out
                                : static_cast<uint64_t>(m.n_layers) * m.d_out;
  const uint64_t in_row = static_cast<uint64_t>(m.d_in) * 2;
  const uint64_t out_row = static_cast<uint64_t>(m.d_out) * 2;
  const bool q8 = m.A_scale != nullptr;
  // bf16 maps: stages of two k-blocks, each operand's staged by one copy through a rank-4
  // view {64 k, rows, k-blocks, 1} whose third dimension steps 128 bytes
  const uint64_t kblocks = static_cast<uint64_t>(m.d_in / kBK);
  const uint64_t dh[4] = {kBK, static_cast<uint64_t>(m.rows), kblocks, 1};
  const uint64_t sh[3] = {in_row, 128, in_row * static_cast<uint64_t>(m.rows)};
  const uint32_t bh[4] = {kBK, kBM, 2, 1};
  bool ok = q8 ? make_tmap_3d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m.H, m.d_in, m.rows, 1,
                              in_row, 0, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B)
               : make_tmap_4d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m.H, dh, sh, bh,
                              CU_TENSOR_MAP_SWIZZLE_128B);
  // B boxes of bn / 2 rows: each CTA of a pair stages half of a tile's columns
  if (q8) {
    // codes {d_in, B rows} int8 in boxes {128, bn / 2} (two k-blocks, one scale group);
    // scales [layers, d_in / 128, d_out] bf16 in boxes {bn / 2} (one 128-weight group of a
    // half tile's rows)
    const uint64_t groups = static_cast<uint64_t>(m.d_in / kQ8Group);
    const uint64_t slayers = single ? static_cast<uint64_t>(slot_layers) : static_cast<uint64_t>(m.n_layers);
    ok = ok && make_tmap_3d(&p.tmB[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, m.A, m.d_in, brows, 1,
                            static_cast<uint64_t>(m.d_in), 0, 2 * kBK, m.bn / 2,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_tmap_3d(&p.tmB[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m.A_scale, m.d_out, groups,
                            slayers, out_row, out_row * groups, m.bn / 2, 1,
                            CU_TENSOR_MAP_SWIZZLE_NONE);
    p.q8 = static_cast<const int8_t*>(m.A);
    p.q8_scale = static_cast<const __nv_bfloat16*>(m.A_scale);
    p.q8_ld = m.d_in;
  } else {
    const uint64_t da[4] = {kBK, brows, kblocks, 1};
    const uint64_t sa[3] = {in_row, 128, in_row * brows};
    const uint32_t ba[4] = {kBK, static_cast<uint32_t>(m.bn / 2), 2, 1};
    ok = ok && make_tmap_4d(&p.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m.A, da, sa, ba,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    p.k2 = 1;
  }
  ok = ok && make_tmap_3d(&p.tmO[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, m.xhat, m.d_out, m.rows,
                          m.n_layers, out_row, out_row * m.R, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the map GEMM");
  p.m_tiles = static_cast<int32_t>(ceil_div(m.rows, kBM));
  p.n_tiles = static_cast<int32_t>(brows / m.bn);
  p.batches = 1;
  p.bn = m.bn;
  p.group_m = 32;
  p.rows = static_cast<int32_t>(m.rows);
  p.ss_stride = static_cast<int32_t>(m.R);
  p.d_out = m.d_out;
  p.layer_base = single ? m.slot_layer : 0;
  p.ss_tiles = m.d_out / m.bn;
  if (m.out_rows != nullptr) {
    p.map_rows = m.out_rows;
    p.map_out = static_cast<__nv_bfloat16*>(m.xhat);
    p.map_ld = m.R;
  }
  p.h_ready = m.h_ready;
  p.h_gen = m.h_gen;
  p.h_group_rows = kHostRowGroup;
  p.h_first_rows = kHostFirstRows;
  if (m.h_ready != nullptr) p.group_m0 = kHostFirstRows / kBM;  // first raster group: the first flag's rows
  p.h_row_base = static_cast<int32_t>(m.h_row_base);
  p.bias = m.bias;
  p.gain = static_cast<const __nv_bfloat16*>(m.gain);
  p.ss_part = m.ss;
  p.lim_a = static_cast<int64_t>(m.n_layers) * p.ss_tiles * m.R;
  p.lim_b = static_cast<int64_t>(m.n_layers) * m.R * m.d_out;
  p.err = device_error_word();
  if (p.err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  const int64_t tiles = static_cast<int64_t>((p.m_tiles + 1) / 2) * p.n_tiles;
  const int pairs = static_cast<int>(tiles < sm_count() / 2 ? tiles : sm_count() / 2);
  if (pairs <= 0) return RF_OK;
  cudaError_t e = q8 ? launch_gemm2_q8(p, pairs, s) : launch_gemm2(p, pairs, s);
  if (e != cudaSuccess) return cuda_fail(e, "map GEMM launch");
  return RF_OK;
}

rf_status launch_map_q8_groups(MapLaunch m, int group, void* dq, cudaStream_t s) {
  const void* codes = m.A;
  const void* scales = m.A_scale;
  const size_t lc = static_cast<size_t>(m.d_out) * m.d_in;         // codes per layer
  const size_t ls = static_cast<size_t>(m.d_in / kQ8Group) * m.d_out;  // scales per layer
  for (int l0 = 0; l0 < m.n_layers; l0 += group) {
    const int g = m.n_layers - l0 < group ? m.n_layers - l0 : group;
    const cudaError_t e = launch_dequant_maps(static_cast<const int8_t*>(codes) + l0 * lc,
                                              static_cast<const __nv_bfloat16*>(scales) + l0 * ls,
                                              g, m.d_out, m.d_in, dq, s);
    if (e != cudaSuccess) return cuda_fail(e, "int8 map dequantisation");
    m.A = dq;
    m.A_scale = nullptr;
    m.slot_layer = l0;
    m.slot_count = g;
    const rf_status st = launch_map(m, s);
    if (st != RF_OK) return st;
  }
  return RF_OK;
}

int q8_group(int option, bool q8, bool maps_on_host, int n_layers) {
  if (!q8 || maps_on_host || option < 0) return 0;
  const int k = option > 0 ? option : 4;
  return k < n_layers ? k : n_layers;
}

size_t map_slot_bytes(int d_out, int d_in, bool q8) {
  const size_t n = static_cast<size_t>(d_out) * d_in;
  if (!q8) return n * 2;
  return align_up(n, 256) + align_up(static_cast<size_t>(d_out) * (d_in / kQ8Group) * 2, 256);
}

cudaError_t copy_map_layer(uint8_t* slot, const void* A, const void* A_scale, int l, int d_out,
                           int d_in, cudaStream_t copy, const void** dA, const void** dS) {
  const size_t n = static_cast<size_t>(d_out) * d_in;
  if (A_scale == nullptr) {
    *dA = slot;
    *dS = nullptr;
    return cudaMemcpyAsync(slot, static_cast<const uint8_t*>(A) + l * n * 2, n * 2,
                           cudaMemcpyHostToDevice, copy);
  }
  const size_t sb = static_cast<size_t>(d_out) * (d_in / kQ8Group) * 2;  // [d_in / 128, d_out]
  uint8_t* sslot = slot + align_up(n, 256);
  *dA = slot;
  *dS = sslot;
  cudaError_t e = cudaMemcpyAsync(slot, static_cast<const uint8_t*>(A) + l * n, n,
                                  cudaMemcpyHostToDevice, copy);
  if (e != cudaSuccess) return e;
  return cudaMemcpyAsync(sslot, static_cast<const uint8_t*>(A_scale) + l * sb, sb,
                         cudaMemcpyHostToDevice, copy);
}

namespace {
constexpr uint32_t kGuardWord = 0x7FC0DEADu;  // a NaN pattern no kernel result repeats by chance

struct GuardSet {
  uint64_t off[kMaxGuards];
  int n;
};

__global__ void guard_kernel(uint8_t* ws, const __grid_constant__ GuardSet g, int check, int* err) {
  constexpr int kWords = static_cast<int>(kGuardBytes / 4);
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < g.n * kWords; i += gridDim.x * blockDim.x) {
    uint32_t* w = reinterpret_cast<uint32_t*>(ws + g.off[i / kWords]) + i % kWords;
    if (!check) *w = kGuardWord;
    else if (*w != kGuardWord) atomicCAS(err, 0, static_cast<int>(kErrGuard));
  }
}

rf_status guards_launch(void* ws, const Layout& lay, int check, cudaStream_t s) {
  if (!kDebug || lay.n == 0) return RF_OK;
  GuardSet g{};
  g.n = lay.n;
  for (int i = 0; i < lay.n; ++i) g.off[i] = lay.guard[i];
  int* err = device_error_word();
  if (err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  guard_kernel<<<32, 256, 0, s>>>(static_cast<uint8_t*>(ws), g, check, err);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? RF_OK : cuda_fail(e, "workspace guard launch");
}
}  // namespace

rf_status guards_fill(void* ws, const Layout& lay, cudaStream_t s) {
  return guards_launch(ws, lay, 0, s);
}
rf_status guards_check(void* ws, const Layout& lay, cudaStream_t s) {
  return guards_launch(ws, lay, 1, s);
}

rf_status check_pinned(const void* ptr, const char* what) {
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeHost) {
    cudaGetLastError();
    return fail(RF_ERR_NOT_PINNED, "maps_on_host set but %s is not page-locked host memory", what);
  }
  return RF_OK;
}

}  // namespace rf

// --------------------------------------------------------------- C ABI
namespace rf {
const char* last_error_cstr();
void clear_last_error();
}

extern "C" const char* ridgefill_status_string(rf_status s) {
  switch (s) {
    case RF_OK: return "ok";
    case RF_ERR_ARG: return "invalid argument";
    case RF_ERR_SHAPE: return "unsupported or inconsistent shape";
    case RF_ERR_ALIGN: return "pointer not 16-byte aligned";
    case RF_ERR_NOT_PINNED: return "host maps are not page-locked";
    case RF_ERR_CUDA: return "CUDA error";
    case RF_ERR_TIMEOUT: return "device wait timed out";
    case RF_ERR_NUMERIC: return "ridge system not positive definite";
    case RF_ERR_WORKSPACE: return "workspace missing or too small";
    case RF_ERR_SOURCE: return "the host map source reported an error";
    case RF_ERR_BOUNDS: return "debug build: out-of-bounds store or overwritten guard band";
  }
  return "unknown status";
}

extern "C" const char* ridgefill_last_error(void) { return rf::last_error_cstr(); }

extern "C" rf_status ridgefill_device_error(void* stream, int* code) {
  if (code == nullptr) return rf::fail(RF_ERR_ARG, "code is NULL");
  *code = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return rf::cuda_fail(e, "cudaStreamSynchronize");
  int* w = rf::device_error_word();
  if (w == nullptr) return rf::fail(RF_ERR_CUDA, "device error word unavailable");
  int v = 0;
  e = cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return rf::cuda_fail(e, "reading the device error word");
  if (v != 0) {
    const int zero = 0;
    e = cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return rf::cuda_fail(e, "clearing the device error word");
  }
  *code = v;
  if (v == 0) return RF_OK;
  if (v == rf::kErrNumeric) return rf::fail(RF_ERR_NUMERIC, "ridge system not positive definite");
  if (v == rf::kErrIndex) return rf::fail(RF_ERR_ARG, "a row index list entry was out of range");
  if (v == rf::kErrGuard) return rf::fail(RF_ERR_BOUNDS, "a workspace guard band was overwritten");
  if (v == rf::kErrBounds) return rf::fail(RF_ERR_BOUNDS, "a kernel store fell outside its buffer");
  return rf::fail(RF_ERR_TIMEOUT, "device wait ran out at site %d", v);
}

extern "C" double ridgefill_compute_share(int32_t split, int32_t n_layers, int64_t tail,
                                          int64_t prompt) {
  if (n_layers <= 0 || prompt <= 0) return 0.0;
  const double S = split, L = n_layers, T = static_cast<double>(tail),
               N = static_cast<double>(prompt);
  return (S * (N - T) + L * T) / (L * N);
}

namespace rf {
namespace {
// One warp; lane 0 waits, with the kernels' own bounded helpers, on an mbarrier that
// nothing arrives at (which = 0) or a device word that nothing sets (which = 1).
__global__ void wait_probe_kernel(int which, const uint32_t* word, int* err) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (which == 0) mbar_wait(&bar, 0, &abort_flag, err, kErrProbe);
    else flag_wait(word, 1u, &abort_flag, err, kErrProbe + 1);
  }
}
}  // namespace
}  // namespace rf

extern "C" rf_status ridgefill_wait_selftest(int32_t which, void* stream) {
  using namespace rf;
  if (which != 0 && which != 1) return fail(RF_ERR_ARG, "which must be 0 or 1");
  int* err = device_error_word();
  if (err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  void* flag = nullptr;
  if (cudaGetSymbolAddress(&flag, g_probe_flag) != cudaSuccess)
    return fail(RF_ERR_CUDA, "probe flag unavailable");
  wait_probe_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      which, static_cast<const uint32_t*>(flag), err);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test launch");
  return RF_OK;
}

extern "C" int32_t ridgefill_abi_version(void) { return 10; }

extern "C" size_t ridgefill_workspace_size(int32_t which, const void* args) {
  if (args == nullptr) {
    rf::fail(RF_ERR_ARG, "args is NULL");
    return 0;
  }
  switch (which) {
    case RF_CALL_FILL: return ridgefill_fill_workspace_size(static_cast<const rf_fill_args*>(args));
    case RF_CALL_FILL_GDN: return ridgefill_gdn_workspace_size(static_cast<const rf_gdn_args*>(args));
    case RF_CALL_FIT: return ridgefill_fit_workspace_size(static_cast<const rf_fit_args*>(args));
    case RF_CALL_RESCALE:
      return ridgefill_rescale_workspace_size(static_cast<const rf_rescale_args*>(args));
    default:
      rf::fail(RF_ERR_ARG, "unknown call %d", static_cast<int>(which));
      return 0;
  }
}
