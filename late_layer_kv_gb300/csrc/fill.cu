// fill.cu -- ridgefill_fill: the attention late-layer cache fill (RidgeFill,
// "Training-Free Late-Layer Cache Fill for Faster Prefill", sections 2.1-2.2).
//
// Per row chunk: one grouped map GEMM writes X_hat for every late layer, then
// one batched K/V GEMM writes the caches.  With maps in page-locked host
// memory the map GEMM runs one layer at a time while the next layer's map is
// copied into the other device slot on a side stream (paper section 4.2:
// maps held in VRAM or streamed from host, identical outputs).
#include <cmath>
#include <mutex>

#include "abi_common.h"

namespace rf {
namespace {

struct FillPlan {
  int bn_map = 0, bn_kv = 0;
  int64_t R = 0;  // rows per chunk
  size_t off_xhat = 0, off_ss = 0, off_slots = 0, total = 0;
};

rf_status validate_fill(const rf_fill_args* a) {
  if (a == nullptr) return fail(RF_ERR_ARG, "args is NULL");
  if (a->n_layers < 1) return fail(RF_ERR_SHAPE, "n_layers must be >= 1");
  if (a->d_in < 64 || a->d_in % 64 != 0) return fail(RF_ERR_SHAPE, "d_in must be a positive multiple of 64");
  if (a->d_out < 128 || a->d_out % 128 != 0)
    return fail(RF_ERR_SHAPE, "d_out must be a positive multiple of 128");
  if (a->head_dim != 64 && a->head_dim != 128) return fail(RF_ERR_SHAPE, "head_dim must be 64 or 128");
  if (a->n_kv_heads < 1) return fail(RF_ERR_SHAPE, "n_kv_heads must be >= 1");
  if ((static_cast<int64_t>(a->n_kv_heads) * a->head_dim) % 128 != 0)
    return fail(RF_ERR_SHAPE, "n_kv_heads * head_dim must be a multiple of 128");
  if (a->rows < 0 || a->pos0 < 0) return fail(RF_ERR_ARG, "rows and pos0 must be >= 0");
  if (a->cache_len < a->pos0 + a->rows) return fail(RF_ERR_SHAPE, "pos0 + rows exceeds cache_len");
  if (a->cache_len >= (int64_t(1) << 24)) return fail(RF_ERR_SHAPE, "cache_len must be < 2^24");
  if (a->rows_per_chunk < 0 || a->rows_per_chunk % 128 != 0)
    return fail(RF_ERR_SHAPE, "rows_per_chunk must be 0 or a multiple of 128");
  if (!(a->rope_theta > 0.0) || !(a->rms_eps >= 0.0)) return fail(RF_ERR_ARG, "bad rope_theta or rms_eps");
  if (static_cast<int64_t>(a->n_layers) * a->d_out >= (int64_t(1) << 31) ||
      static_cast<int64_t>(a->n_layers) * a->n_kv_heads >= (int64_t(1) << 31) ||
      a->rows >= (int64_t(1) << 31))
    return fail(RF_ERR_SHAPE, "sizes exceed the 32-bit tile indexing");
  if (a->maps_on_host != 0 && a->maps_on_host != 1) return fail(RF_ERR_ARG, "maps_on_host must be 0 or 1");
  return RF_OK;
}

void plan_fill(const rf_fill_args* a, FillPlan* pl) {
  pl->bn_map = (a->d_out % 256 == 0) ? 256 : 128;
  const int kvw = a->n_kv_heads * a->head_dim;
  pl->bn_kv = (kvw % 256 == 0) ? 256 : 128;
  const int64_t all = ceil_div(a->rows > 0 ? a->rows : 1, kBM) * kBM;
  pl->R = a->rows_per_chunk > 0 ? (a->rows_per_chunk < all ? a->rows_per_chunk : all) : all;
  const size_t L = a->n_layers, d = a->d_out;
  pl->off_xhat = 0;
  pl->off_ss = align_up(L * pl->R * d * 2, 256);
  pl->off_slots = align_up(pl->off_ss + L * (d / pl->bn_map) * pl->R * 4, 256);
  const size_t slots = a->maps_on_host ? kMapSlots * d * static_cast<size_t>(a->d_in) * 2 : 0;
  pl->total = align_up(pl->off_slots + slots, 256);
}

// K/V GEMM on CTA pairs (true) or single CTAs
constexpr bool kKvPairs = true;

rf_status launch_kv(const rf_fill_args* a, const FillPlan& pl, int64_t start, int64_t rc,
                    const void* xhat, const float* ss, cudaStream_t s) {
  GemmParams p{};
  p.mode = kModeKV;
  p.k_blocks = a->d_out / kBK;
  const int kvw = a->n_kv_heads * a->head_dim;
  const uint64_t drow = static_cast<uint64_t>(a->d_out) * 2;
  const uint64_t hd = a->head_dim;
  const uint64_t pos_end = static_cast<uint64_t>(a->pos0 + start + rc);
  bool ok = make_tmap_3d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xhat, a->d_out, rc,
                         a->n_layers, drow, drow * pl.R, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  // pair kernel: B boxes of bn / 2 rows (each CTA of a pair stages half of a tile's columns)
  const uint32_t bbox = kKvPairs ? pl.bn_kv / 2 : pl.bn_kv;
  ok = ok && make_tmap_3d(&p.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Wk, a->d_out, kvw,
                          a->n_layers, drow, drow * kvw, kBK, bbox, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_3d(&p.tmB[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Wv, a->d_out, kvw,
                          a->n_layers, drow, drow * kvw, kBK, bbox, CU_TENSOR_MAP_SWIZZLE_128B);
  const uint64_t planes = static_cast<uint64_t>(a->n_layers) * a->n_kv_heads;
  const uint64_t plane_bytes = static_cast<uint64_t>(a->cache_len) * hd * 2;
  ok = ok && make_tmap_3d(&p.tmO[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Kc, hd, pos_end, planes,
                          hd * 2, plane_bytes, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_3d(&p.tmO[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Vc, hd, pos_end, planes,
                          hd * 2, plane_bytes, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the K/V GEMM");
  p.m_tiles = static_cast<int32_t>(ceil_div(rc, kBM));
  p.n_k_tiles = kvw / pl.bn_kv;
  p.n_tiles = 2 * p.n_k_tiles;
  p.batches = a->n_layers;
  p.bn = pl.bn_kv;
  p.group_m = 16;
  p.rows = static_cast<int32_t>(rc);
  p.ss_stride = static_cast<int32_t>(pl.R);
  p.d_out = a->d_out;
  p.ss_tiles = a->d_out / pl.bn_map;
  p.ss_in = ss;
  p.n_kv = a->n_kv_heads;
  p.head_dim = a->head_dim;
  p.pos_base = static_cast<int32_t>(a->pos0 + start);
  p.inv_d = static_cast<float>(1.0 / a->d_out);
  p.eps = static_cast<float>(a->rms_eps);
  for (int i = 0; i < a->head_dim / 2; ++i) {
    const double f = std::pow(a->rope_theta, -2.0 * i / a->head_dim);
    p.inv_freq_hi[i] = static_cast<float>(f);
    p.inv_freq_lo[i] = static_cast<float>(f - static_cast<double>(p.inv_freq_hi[i]));
  }
  p.err = device_error_word();
  if (p.err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  cudaError_t e;
  if (kKvPairs) {
    const int64_t tiles = static_cast<int64_t>((p.m_tiles + 1) / 2) * p.n_tiles * p.batches;
    const int pairs = static_cast<int>(tiles < sm_count() / 2 ? tiles : sm_count() / 2);
    if (pairs <= 0) return RF_OK;
    e = launch_gemm2(p, pairs, s);
  } else {
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles * p.batches;
    const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
    if (grid <= 0) return RF_OK;
    e = launch_gemm(p, grid, s);
  }
  if (e != cudaSuccess) return cuda_fail(e, "K/V GEMM launch");
  return RF_OK;
}

std::mutex g_host_map_mu;

}  // namespace
}  // namespace rf

using namespace rf;

extern "C" size_t ridgefill_fill_workspace_size(const rf_fill_args* a) {
  if (validate_fill(a) != RF_OK) return 0;
  FillPlan pl;
  plan_fill(a, &pl);
  return pl.total;
}

extern "C" rf_status ridgefill_fill(const rf_fill_args* a, void* workspace, size_t ws_bytes,
                                    void* stream) {
  rf_status st = validate_fill(a);
  if (st != RF_OK) return st;
  if (a->rows == 0) return RF_OK;
  const void* req[] = {a->H, a->A, a->bias, a->Wk, a->Wv, a->Kc, a->Vc};
  for (const void* p : req)
    if (p == nullptr) return fail(RF_ERR_ARG, "a required pointer is NULL");
  const void* dev[] = {a->H, a->bias, a->gain, a->Wk, a->Wv, a->Kc, a->Vc, workspace};
  for (const void* p : dev)
    if (p != nullptr && !aligned16(p)) return fail(RF_ERR_ALIGN, "a device pointer is not 16-byte aligned");
  if (!aligned16(a->A)) return fail(RF_ERR_ALIGN, "A is not 16-byte aligned");
  if (a->maps_on_host) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, a->A);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      return fail(RF_ERR_NOT_PINNED, "maps_on_host set but A is not page-locked host memory");
    }
  }
  FillPlan pl;
  plan_fill(a, &pl);
  if (workspace == nullptr || ws_bytes < pl.total)
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes", pl.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* xhat = ws + pl.off_xhat;
  float* ss = reinterpret_cast<float*>(ws + pl.off_ss);
  const size_t map_bytes = static_cast<size_t>(a->d_out) * a->d_in * 2;

  HostStreamer* hs = nullptr;
  std::unique_lock<std::mutex> lk(g_host_map_mu, std::defer_lock);
  if (a->maps_on_host) {
    lk.lock();
    hs = host_streamer();
    if (hs == nullptr) return RF_ERR_CUDA;
    // the copy stream starts after work already queued on `s` (earlier users of the slots)
    cudaError_t e = cudaEventRecord(hs->start, s);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hs->copy, hs->start, 0);
    if (e != cudaSuccess) return cuda_fail(e, "ordering the map-copy stream");
  }

  cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(a->stage_events);
  auto mark = [&](int64_t start, int i) -> rf_status {
    if (ev == nullptr || start != 0) return RF_OK;
    cudaError_t e = cudaEventRecord(ev[i], s);
    return e == cudaSuccess ? RF_OK : cuda_fail(e, "recording a stage event");
  };
  for (int64_t start = 0; start < a->rows; start += pl.R) {
    if ((st = mark(start, 0)) != RF_OK) return st;
    const int64_t rc = (a->rows - start < pl.R) ? a->rows - start : pl.R;
    MapLaunch m{};
    m.H = static_cast<const uint8_t*>(a->H) + static_cast<size_t>(start) * a->d_in * 2;
    m.rows = rc;
    m.d_in = a->d_in;
    m.d_out = a->d_out;
    m.n_layers = a->n_layers;
    m.bn = pl.bn_map;
    m.R = pl.R;
    m.bias = a->bias;
    m.gain = a->gain;
    m.xhat = xhat;
    m.ss = ss;
    if (!a->maps_on_host) {
      m.A = a->A;
      m.slot_layer = -1;
      st = launch_map(m, s);
      if (st != RF_OK) return st;
    } else {
      for (int l = 0; l < a->n_layers; ++l) {
        const int k = l % kMapSlots;
        uint8_t* slot = ws + pl.off_slots + k * map_bytes;
        cudaError_t e = cudaSuccess;
        cudaEvent_t const* cev = reinterpret_cast<cudaEvent_t const*>(a->copy_events);
        if (start > 0 || l >= kMapSlots) e = cudaStreamWaitEvent(hs->copy, hs->freed[k], 0);
        if (e == cudaSuccess && cev != nullptr && start == 0) e = cudaEventRecord(cev[2 * l], hs->copy);
        if (e == cudaSuccess)
          e = cudaMemcpyAsync(slot, static_cast<const uint8_t*>(a->A) + l * map_bytes, map_bytes,
                              cudaMemcpyHostToDevice, hs->copy);
        if (e == cudaSuccess && cev != nullptr && start == 0)
          e = cudaEventRecord(cev[2 * l + 1], hs->copy);
        if (e == cudaSuccess) e = cudaEventRecord(hs->copied[k], hs->copy);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hs->copied[k], 0);
        if (e != cudaSuccess) return cuda_fail(e, "streaming a map from host memory");
        m.A = slot;
        m.slot_layer = l;
        st = launch_map(m, s);
        if (st != RF_OK) return st;
        e = cudaEventRecord(hs->freed[k], s);
        if (e != cudaSuccess) return cuda_fail(e, "recording a map slot release");
      }
    }
    if ((st = mark(start, 1)) != RF_OK) return st;
    st = launch_kv(a, pl, start, rc, xhat, ss, s);
    if (st != RF_OK) return st;
    if ((st = mark(start, 2)) != RF_OK) return st;
  }
  return RF_OK;
}
