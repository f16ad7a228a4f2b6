// fill.cu -- ridgefill_fill: the attention late-layer cache fill (RidgeFill,
// "Training-Free Late-Layer Cache Fill for Faster Prefill", sections 2.1-2.2).
//
// Per row chunk: one grouped map GEMM writes X_hat for every late layer, then
// one batched K/V GEMM writes the caches.  With maps in page-locked host
// memory the map GEMM runs one layer at a time while the next layer's map is
// copied into the other device slot on a side stream (paper section 4.2:
// maps held in VRAM or streamed from host, identical outputs).
#include <chrono>
#include <cmath>
#include <mutex>
#include <thread>

#include "abi_common.h"
#include "sm103_ptx.cuh"

namespace rf {
namespace {

struct FillPlan {
  int bn_map = 0, bn_kv = 0;
  int64_t R = 0;  // rows per chunk
  int dq_layers = 0;
  size_t off_dq = 0;
  size_t off_xhat = 0, off_ss = 0, off_slots = 0, off_gather = 0, off_hdev = 0, off_hflags = 0,
         off_rope = 0, total = 0;
  Layout lay;
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
  if (a->row_idx != nullptr) {
    if (a->h_rows < a->rows || a->h_rows >= (int64_t(1) << 31))
      return fail(RF_ERR_SHAPE, "with row_idx, h_rows must be >= rows and < 2^31");
    if (a->cache_len < a->pos0 + a->h_rows)
      return fail(RF_ERR_SHAPE, "pos0 + h_rows exceeds cache_len");
  }
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
  if (a->A_scale != nullptr && a->d_in % kQ8Group != 0)
    return fail(RF_ERR_SHAPE, "int8 maps need d_in to be a multiple of 128");
  if (a->q8_group_layers < -1) return fail(RF_ERR_ARG, "q8_group_layers must be >= -1");
  if (a->h_on_host != 0 && a->h_on_host != 1) return fail(RF_ERR_ARG, "h_on_host must be 0 or 1");
  if (a->h_on_host && a->row_idx != nullptr)
    return fail(RF_ERR_ARG, "h_on_host cannot be combined with row_idx");
  if (a->map_source != nullptr && a->maps_on_host != 1)
    return fail(RF_ERR_ARG, "map_source needs maps_on_host = 1");
  if (a->host_wait_ms < 0) return fail(RF_ERR_ARG, "host_wait_ms must be >= 0");
  return RF_OK;
}

using Clock = std::chrono::steady_clock;

// Bounded host wait for event `ev` (cudaEventQuery polling): RF_ERR_TIMEOUT after `ms`.
rf_status host_wait_event(cudaEvent_t ev, int ms, const char* what) {
  const auto t0 = Clock::now();
  for (;;) {
    const cudaError_t e = cudaEventQuery(ev);
    if (e == cudaSuccess) return RF_OK;
    if (e != cudaErrorNotReady) return cuda_fail(e, what);
    if (Clock::now() - t0 > std::chrono::milliseconds(ms))
      return fail(RF_ERR_TIMEOUT, "%s: still pending after %d ms", what, ms);
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
}

// Layer l's map from the caller's host source into staging half j, after the previous copy
// out of that half has finished; then its copy into the device slot on the copy stream.
rf_status source_map_layer(const rf_fill_args* a, HostStreamer* hs, int j, int l, uint8_t* slot,
                           size_t slot_bytes, const void** dA, const void** dS) {
  const int ms = a->host_wait_ms > 0 ? a->host_wait_ms : 10000;
  rf_status st = host_wait_event(hs->staged[j], ms, "copy out of a map staging half");
  if (st != RF_OK) return st;
  uint8_t* half = static_cast<uint8_t*>(a->map_staging) + j * slot_bytes;
  const auto t0 = Clock::now();
  const int32_t rc = a->map_source(a->map_source_user, l, half, slot_bytes);
  const auto took = std::chrono::duration_cast<std::chrono::milliseconds>(Clock::now() - t0).count();
  if (rc != 0) return fail(RF_ERR_SOURCE, "map_source returned %d for layer %d", rc, l);
  if (took > ms)
    return fail(RF_ERR_TIMEOUT, "map_source took %lld ms for layer %d (limit %d ms)",
                static_cast<long long>(took), l, ms);
  const size_t n = static_cast<size_t>(a->d_out) * a->d_in;
  const bool q8 = a->A_scale != nullptr;
  cudaError_t e = copy_map_layer(slot, half, q8 ? half + align_up(n, 256) : nullptr, 0, a->d_out,
                                 a->d_in, hs->copy, dA, dS);
  if (e == cudaSuccess) e = cudaEventRecord(hs->staged[j], hs->copy);
  return e == cudaSuccess ? RF_OK : cuda_fail(e, "copying a map out of its staging half");
}

void plan_fill(const rf_fill_args* a, FillPlan* pl) {
  pl->bn_map = (a->d_out % 256 == 0) ? 256 : 128;
  const int kvw = a->n_kv_heads * a->head_dim;
  pl->bn_kv = (kvw % 256 == 0) ? 256 : 128;
  const int64_t all = ceil_div(a->rows > 0 ? a->rows : 1, kBM) * kBM;
  pl->R = a->rows_per_chunk > 0 ? (a->rows_per_chunk < all ? a->rows_per_chunk : all) : all;
  const size_t L = a->n_layers, d = a->d_out;
  Layout& lay = pl->lay;
  pl->off_xhat = lay.take(L * pl->R * d * 2);
  pl->off_ss = lay.take(L * (d / pl->bn_map) * pl->R * 4);
  const size_t slots =
      a->maps_on_host ? kMapSlots * map_slot_bytes(a->d_out, a->d_in, a->A_scale != nullptr) : 0;
  pl->off_slots = lay.take(slots);
  const size_t gather = a->row_idx != nullptr ? static_cast<size_t>(pl->R) * a->d_in * 2 : 0;
  pl->off_gather = lay.take(gather);
  size_t hflags = 0;
  const size_t hbytes = a->h_on_host ? host_rows_bytes(a->rows, a->d_in, &hflags) : 0;
  pl->off_hdev = lay.take(hbytes);
  pl->off_hflags = pl->off_hdev + hflags;
  const size_t rope = static_cast<size_t>(a->head_dim / 2) * pl->R * 8;  // (cos, sin) f32 pairs
  pl->off_rope = lay.take(rope);
  pl->dq_layers = q8_group(a->q8_group_layers, a->A_scale != nullptr, a->maps_on_host != 0,
                           a->n_layers);
  pl->off_dq = lay.take(static_cast<size_t>(pl->dq_layers) * a->d_out * a->d_in * 2);
  pl->total = lay.off;
}

// RoPE angles of one row chunk (rotate-half pairs, frequency f_i = theta^(-2i/hd)):
// tab[i * ld + r] = (cos, sin) of (pos0 + position of row r) * f_i.  The angle is
// formed and reduced modulo 2 pi in f64, then its cos and sin taken in f32.
struct RopeFreqs {
  double f[64];
};

__global__ void rope_table_kernel(float2* tab, int64_t ld, int half, int64_t rc, int64_t pos0,
                                  int64_t start, const int32_t* row_idx, int64_t h_rows,
                                  const __grid_constant__ RopeFreqs fr) {
  const int64_t n = static_cast<int64_t>(half) * rc;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n;
       k += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int i = static_cast<int>(k / rc);
    const int64_t r = k - i * rc;
    int64_t pos = start + r;
    if (row_idx != nullptr) {
      const int64_t idx = row_idx[start + r];
      pos = idx >= 0 && idx < h_rows ? idx : 0;  // out-of-range rows are skipped anyway
    }
    constexpr double kTwoPiD = 6.283185307179586476925286766559;
    const double ang = static_cast<double>(pos0 + pos) * fr.f[i];
    const double q = rint(ang * (1.0 / kTwoPiD));
    const double red = fma(-q, kTwoPiD, ang);  // |red| <= pi, error ~ q * 2.4e-16
    float s, c;
    sincosf(static_cast<float>(red), &s, &c);
    tab[i * ld + r] = make_float2(c, s);
  }
}

// Exact prefix rows (section 2.4): the split states of the listed rows
// idx[0 .. rc) gathered into a dense [rc, d_in] block for the map GEMM; one
// warp per row, an entry outside [0, h_rows) gives a zero row and an error code.
__global__ void gather_rows_kernel(const __nv_bfloat16* H, const int32_t* idx, int64_t rc,
                                   int64_t h_rows, int d_in, __nv_bfloat16* out, int* err) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= rc) return;
  const int64_t src = idx[w];
  const bool ok = src >= 0 && src < h_rows;
  if (!ok && lane == 0) atomicCAS(err, 0, kErrIndex);
  const uint4* s = reinterpret_cast<const uint4*>(H + (ok ? src : 0) * d_in);
  uint4* d = reinterpret_cast<uint4*>(out + w * d_in);
  for (int j = lane; j < d_in / 8; j += 32) d[j] = ok ? s[j] : make_uint4(0, 0, 0, 0);
}

// `only`: 0 = keys and values, RF_RESCALE_KEYS / RF_RESCALE_VALUES = that half alone
rf_status launch_kv(const rf_fill_args* a, const FillPlan& pl, int64_t start, int64_t rc,
                    const void* xhat, const float* ss, cudaStream_t s, int only = 0,
                    const float2* rope_tab = nullptr) {
  GemmParams p{};
  p.mode = kModeKV;
  p.k_blocks = a->d_out / kBK;
  const int kvw = a->n_kv_heads * a->head_dim;
  const uint64_t drow = static_cast<uint64_t>(a->d_out) * 2;
  const uint64_t hd = a->head_dim;
  const uint64_t pos_end = static_cast<uint64_t>(a->pos0 + start + rc);
  // stages of two k-blocks: each operand staged by one copy through a rank-4 view
  // {64 k, rows, k-blocks, layers} whose third dimension steps 128 bytes; B boxes of bn / 2
  // rows (each CTA of a pair stages half of a tile's columns)
  const uint64_t kblocks = static_cast<uint64_t>(a->d_out / kBK);
  const uint64_t L = static_cast<uint64_t>(a->n_layers);
  const uint64_t dx[4] = {kBK, static_cast<uint64_t>(rc), kblocks, L};
  const uint64_t sx[3] = {drow, 128, drow * static_cast<uint64_t>(pl.R)};
  const uint32_t bx[4] = {kBK, kBM, 2, 1};
  bool ok = make_tmap_4d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xhat, dx, sx, bx,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  const uint64_t dw[4] = {kBK, static_cast<uint64_t>(kvw), kblocks, L};
  const uint64_t sw[3] = {drow, 128, drow * static_cast<uint64_t>(kvw)};
  const uint32_t bw[4] = {kBK, static_cast<uint32_t>(pl.bn_kv / 2), 2, 1};
  ok = ok && make_tmap_4d(&p.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Wk, dw, sw, bw,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_4d(&p.tmB[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Wv, dw, sw, bw,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  p.k2 = 1;
  const uint64_t planes = static_cast<uint64_t>(a->n_layers) * a->n_kv_heads;
  const uint64_t plane_bytes = static_cast<uint64_t>(a->cache_len) * hd * 2;
  ok = ok && make_tmap_3d(&p.tmO[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Kc, hd, pos_end, planes,
                          hd * 2, plane_bytes, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_3d(&p.tmO[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Vc, hd, pos_end, planes,
                          hd * 2, plane_bytes, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the K/V GEMM");
  p.m_tiles = static_cast<int32_t>(ceil_div(rc, kBM));
  p.n_k_tiles = only == RF_RESCALE_VALUES ? 0 : kvw / pl.bn_kv;
  p.n_tiles = only == 0 ? 2 * p.n_k_tiles : kvw / pl.bn_kv;
  p.batches = a->n_layers;
  p.bn = pl.bn_kv;
  // raster groups of one pair row tile: the pairs that take a row tile's column tiles
  // together share its first (DRAM) read of X_hat, and W_kv of the layer stays in L2
  p.group_m = 2;
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
  p.k_scale = a->k_scale;
  p.v_scale = a->v_scale;
  p.rope_tab = rope_tab;
  p.rope_ld = pl.R;
  if (a->row_idx != nullptr) {
    p.kv_rows = a->row_idx + start;
    p.kv_pos0 = static_cast<int32_t>(a->pos0);
    p.kv_hrows = static_cast<int32_t>(a->h_rows);
    p.kv_cache[0] = static_cast<__nv_bfloat16*>(a->Kc);
    p.kv_cache[1] = static_cast<__nv_bfloat16*>(a->Vc);
    p.cache_len = a->cache_len;
    p.lim_b = static_cast<int64_t>(a->n_layers) * a->n_kv_heads * a->cache_len * a->head_dim;
  }
  for (int i = 0; i < a->head_dim / 2; ++i) {
    const double f = std::pow(a->rope_theta, -2.0 * i / a->head_dim);
    p.inv_freq_hi[i] = static_cast<float>(f);
    p.inv_freq_lo[i] = static_cast<float>(f - static_cast<double>(p.inv_freq_hi[i]));
  }
  p.err = device_error_word();
  if (p.err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  const int64_t tiles = static_cast<int64_t>((p.m_tiles + 1) / 2) * p.n_tiles * p.batches;
  const int pairs = static_cast<int>(tiles < sm_count() / 2 ? tiles : sm_count() / 2);
  if (pairs <= 0) return RF_OK;
  const cudaError_t e = launch_gemm2(p, pairs, s);
  if (e != cudaSuccess) return cuda_fail(e, "K/V GEMM launch");
  return RF_OK;
}

}  // namespace

rf_status launch_gather_rows(const void* H, const int32_t* idx, int64_t rc, int64_t h_rows,
                             int d_in, void* out, cudaStream_t s) {
  if (rc <= 0) return RF_OK;
  gather_rows_kernel<<<static_cast<unsigned>((rc * 32 + 255) / 256), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(H), idx, rc, h_rows, d_in,
      static_cast<__nv_bfloat16*>(out), device_error_word());
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? RF_OK : cuda_fail(e, "row gather launch");
}

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
  const bool sourced = a->map_source != nullptr;
  const void* req[] = {a->H, sourced ? a->map_staging : a->A, a->bias, a->Wk, a->Wv, a->Kc, a->Vc};
  for (const void* p : req)
    if (p == nullptr) return fail(RF_ERR_ARG, "a required pointer is NULL");
  const void* dev[] = {a->H, a->bias, a->gain, a->Wk, a->Wv, a->Kc, a->Vc, workspace};
  for (const void* p : dev)
    if (p != nullptr && !aligned16(p)) return fail(RF_ERR_ALIGN, "a device pointer is not 16-byte aligned");
  if (!aligned16(a->A) || !aligned16(a->map_staging))
    return fail(RF_ERR_ALIGN, "A or map_staging is not 16-byte aligned");
  if (a->A_scale != nullptr && !sourced && !aligned16(a->A_scale))
    return fail(RF_ERR_ALIGN, "A_scale is not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(a->row_idx) & 3u) != 0)
    return fail(RF_ERR_ALIGN, "row_idx is not 4-byte aligned");
  if (sourced) {
    if ((st = check_pinned(a->map_staging, "map_staging")) != RF_OK) return st;
  } else if (a->maps_on_host) {
    if ((st = check_pinned(a->A, "A")) != RF_OK) return st;
    if (a->A_scale != nullptr && (st = check_pinned(a->A_scale, "A_scale")) != RF_OK) return st;
  }
  if (a->h_on_host && (st = check_pinned(a->H, "H")) != RF_OK) return st;
  FillPlan pl;
  plan_fill(a, &pl);
  if (workspace == nullptr || ws_bytes < pl.total)
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes", pl.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* xhat = ws + pl.off_xhat;
  float* ss = reinterpret_cast<float*>(ws + pl.off_ss);
  const size_t slot_bytes = map_slot_bytes(a->d_out, a->d_in, a->A_scale != nullptr);
  if ((st = guards_fill(ws, pl.lay, s)) != RF_OK) return st;

  HostStreamer* hs = nullptr;
  std::unique_lock<std::mutex> lk(host_stream_mutex(), std::defer_lock);
  if (a->maps_on_host || a->h_on_host) {
    lk.lock();
    hs = host_streamer();
    if (hs == nullptr) return RF_ERR_CUDA;
  }
  // split state in host memory: streamed in row groups, overlapped with the map GEMM
  const uint8_t* h_base = static_cast<const uint8_t*>(a->H);
  HostRows hr;
  if (a->h_on_host) {
    if ((st = stream_host_rows(hs, a->H, a->rows, a->d_in, ws + pl.off_hdev,
                               reinterpret_cast<uint32_t*>(ws + pl.off_hflags), s, &hr)) != RF_OK)
      return st;
    h_base = hr.base;
  }
  if (a->maps_on_host) {
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
    m.H = h_base + static_cast<size_t>(start) * a->d_in * 2;
    if (hr.overlap) {
      m.h_ready = hr.flags;
      m.h_gen = hr.gen;
      m.h_row_base = start;
    }
    if (a->row_idx != nullptr) {  // the chunk's listed rows, gathered
      void* hc = ws + pl.off_gather;
      if ((st = launch_gather_rows(a->H, a->row_idx + start, rc, a->h_rows, a->d_in, hc, s)) != RF_OK)
        return st;
      m.H = hc;
    }
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
    if (!a->maps_on_host && pl.dq_layers > 0) {
      // int8 maps: bf16(q s) of a few layers at a time, then the bf16 GEMM on them
      m.A = a->A;
      m.A_scale = a->A_scale;
      if ((st = launch_map_q8_groups(m, pl.dq_layers, ws + pl.off_dq, s)) != RF_OK) return st;
    } else if (!a->maps_on_host) {
      m.A = a->A;
      m.A_scale = a->A_scale;
      m.slot_layer = -1;
      st = launch_map(m, s);
      if (st != RF_OK) return st;
    } else {
      for (int l = 0; l < a->n_layers; ++l) {
        const int k = l % kMapSlots;
        uint8_t* slot = ws + pl.off_slots + k * slot_bytes;
        cudaError_t e = cudaSuccess;
        cudaEvent_t const* cev = reinterpret_cast<cudaEvent_t const*>(a->copy_events);
        if (start > 0 || l >= kMapSlots) e = cudaStreamWaitEvent(hs->copy, hs->freed[k], 0);
        if (e == cudaSuccess && cev != nullptr && start == 0) e = cudaEventRecord(cev[2 * l], hs->copy);
        if (e != cudaSuccess) return cuda_fail(e, "streaming a map from host memory");
        if (sourced) {
          const int j = static_cast<int>((start / pl.R * a->n_layers + l) & 1);
          if ((st = source_map_layer(a, hs, j, l, slot, slot_bytes, &m.A, &m.A_scale)) != RF_OK)
            return st;
        } else {
          e = copy_map_layer(slot, a->A, a->A_scale, l, a->d_out, a->d_in, hs->copy, &m.A,
                             &m.A_scale);
        }
        if (e == cudaSuccess && cev != nullptr && start == 0)
          e = cudaEventRecord(cev[2 * l + 1], hs->copy);
        if (e == cudaSuccess) e = cudaEventRecord(hs->copied[k], hs->copy);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hs->copied[k], 0);
        if (e != cudaSuccess) return cuda_fail(e, "streaming a map from host memory");
        m.slot_layer = l;
        st = launch_map(m, s);
        if (st != RF_OK) return st;
        e = cudaEventRecord(hs->freed[k], s);
        if (e != cudaSuccess) return cuda_fail(e, "recording a map slot release");
      }
    }
    if ((st = mark(start, 1)) != RF_OK) return st;
    // the chunk's RoPE angles, then the K/V GEMM
    float2* tab = reinterpret_cast<float2*>(ws + pl.off_rope);
    {
      RopeFreqs fr{};
      for (int i = 0; i < a->head_dim / 2; ++i) fr.f[i] = std::pow(a->rope_theta, -2.0 * i / a->head_dim);
      const int64_t n = static_cast<int64_t>(a->head_dim / 2) * rc;
      const int64_t blocks = (n + 255) / 256 < 4 * sm_count() ? (n + 255) / 256 : 4 * sm_count();
      rope_table_kernel<<<static_cast<unsigned>(blocks > 0 ? blocks : 1), 256, 0, s>>>(
          tab, pl.R, a->head_dim / 2, rc, a->pos0, start, a->row_idx, a->h_rows, fr);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "RoPE table launch");
    }
    st = launch_kv(a, pl, start, rc, xhat, ss, s, 0, tab);
    if (st != RF_OK) return st;
    if ((st = mark(start, 2)) != RF_OK) return st;
  }
  if (a->h_on_host) {  // later work on `s` (and the caller's reuse of H) follows the copy
    cudaError_t e = cudaStreamWaitEvent(s, hs->h_done, 0);
    if (e != cudaSuccess) return cuda_fail(e, "ordering after the split-state copy");
  }
  return guards_check(ws, pl.lay, s);
}

// ------------------------------------------------------------------ value / key rescale
// RidgeFill section 2.3 "Value rescale" and the key scale of section 6.6: the
// c tail rows are projected from the map's prediction (map GEMM + K/V GEMM into
// scratch caches) and from their true inputs (g * x and its sums of squares,
// then the same K/V GEMM); the per-head mean of the norm ratios scales the
// filled rows of the cache in place.
namespace rf {
namespace {

struct RescalePlan {
  FillPlan fp;     // fill plan of the c predicted rows (map tile widths)
  int64_t R2 = 0;  // rows of the stacked buffers: predicted rows [0, c), true rows [c, 2c)
  size_t off_x = 0, off_ss = 0, off_cache = 0, off_scale = 0, total = 0;
  Layout lay;
};

rf_status validate_rescale(const rf_rescale_args* a) {
  if (a == nullptr) return fail(RF_ERR_ARG, "args is NULL");
  if (a->which != RF_RESCALE_VALUES && a->which != RF_RESCALE_KEYS)
    return fail(RF_ERR_ARG, "which must be RF_RESCALE_VALUES or RF_RESCALE_KEYS");
  if (a->tail_rows < 1 || a->tail_rows >= (int64_t(1) << 23))
    return fail(RF_ERR_ARG, "tail_rows must be in [1, 2^23)");
  rf_fill_args f{};
  f.n_layers = a->n_layers;
  f.d_in = a->d_in;
  f.d_out = a->d_out;
  f.n_kv_heads = a->n_kv_heads;
  f.head_dim = a->head_dim;
  f.rows = a->rows;
  f.pos0 = a->pos0;
  f.cache_len = a->cache_len;
  f.rope_theta = 1e4;
  f.rms_eps = a->rms_eps;
  f.A_scale = a->A_scale;
  return validate_fill(&f);
}

void plan_rescale(const rf_rescale_args* a, RescalePlan* pl) {
  rf_fill_args f{};
  f.n_layers = a->n_layers;
  f.d_in = a->d_in;
  f.d_out = a->d_out;
  f.n_kv_heads = a->n_kv_heads;
  f.head_dim = a->head_dim;
  f.rows = a->tail_rows;
  plan_fill(&f, &pl->fp);
  pl->R2 = ceil_div(2 * a->tail_rows, kBM) * kBM;
  const size_t L = a->n_layers, d = a->d_out, R2 = pl->R2;
  Layout& lay = pl->lay;
  pl->off_x = lay.take(L * R2 * d * 2);
  pl->off_ss = lay.take(L * (d / pl->fp.bn_map) * R2 * 4);
  pl->off_cache = lay.take(L * a->n_kv_heads * R2 * a->head_dim * 2);
  pl->off_scale = lay.take(L * a->n_kv_heads * 4);
  pl->total = lay.off;
}

// One warp per (layer, true row r): X_hat row c + r = bf16(g x) and its sum of
// squares as the row's first partial (the other partials zero), in the layout
// the map GEMM gives the predicted rows.
__global__ void true_input_kernel(const __nv_bfloat16* X, const __nv_bfloat16* g, int L, int64_t c,
                                  int d, int64_t R2, int ss_tiles, __nv_bfloat16* xhat, float* ss) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<int64_t>(L) * c) return;
  const int l = static_cast<int>(w / c);
  const int64_t r = w % c;
  const __nv_bfloat16* src = X + (static_cast<size_t>(l) * c + r) * d;
  __nv_bfloat16* dst = xhat + (static_cast<size_t>(l) * R2 + c + r) * d;
  const __nv_bfloat16* gl = g != nullptr ? g + static_cast<size_t>(l) * d : nullptr;
  float acc = 0.f;
  for (int j = 8 * lane; j < d; j += 256) {
    const uint4 xv = *reinterpret_cast<const uint4*>(src + j);
    uint4 gv = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);  // bf16 1.0 pairs
    if (gl != nullptr) gv = *reinterpret_cast<const uint4*>(gl + j);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 x2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xw[e]));
      const float2 g2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[e]));
      acc = fmaf(x2.x, x2.x, acc);
      acc = fmaf(x2.y, x2.y, acc);
      out[e] = pack_bf16(x2.x * g2.x, x2.y * g2.y);
    }
    *reinterpret_cast<uint4*>(dst + j) = make_uint4(out[0], out[1], out[2], out[3]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  for (int t = lane; t < ss_tiles; t += 32)
    ss[(static_cast<size_t>(l) * ss_tiles + t) * R2 + c + r] = t == 0 ? acc : 0.f;
}

__device__ __forceinline__ float row_sq(const __nv_bfloat16* p, int hd) {
  float s = 0.f;
  for (int j = 0; j < hd; j += 8) {
    const uint4 v = *reinterpret_cast<const uint4*>(p + j);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      s = fmaf(f.x, f.x, s);
      s = fmaf(f.y, f.y, s);
    }
  }
  return s;
}

// One CTA per (layer, kv head) of the stacked projections (predicted rows
// [0, c), true rows [c, 2c)): the mean over rows of |true| / |predicted|.
__global__ void __launch_bounds__(256) rescale_ratio_kernel(const __nv_bfloat16* proj, int64_t R2,
                                                            int64_t c, int hd, float* scale_ws,
                                                            float* scale_out) {
  __shared__ float s_sum[256];
  __shared__ int s_cnt[256];
  const size_t plane = blockIdx.x;
  float sum = 0.f;
  int cnt = 0;
  for (int64_t r = threadIdx.x; r < c; r += blockDim.x) {
    const float np = row_sq(proj + (plane * R2 + r) * hd, hd);
    const float nt = row_sq(proj + (plane * R2 + c + r) * hd, hd);
    if (np > 0.f) {
      sum += sqrtf(nt) / sqrtf(np);
      ++cnt;
    }
  }
  s_sum[threadIdx.x] = sum;
  s_cnt[threadIdx.x] = cnt;
  __syncthreads();
  for (int o = blockDim.x / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      s_sum[threadIdx.x] += s_sum[threadIdx.x + o];
      s_cnt[threadIdx.x] += s_cnt[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const float sc = s_cnt[0] > 0 ? s_sum[0] / static_cast<float>(s_cnt[0]) : 1.f;
    scale_ws[plane] = sc;
    if (scale_out != nullptr) scale_out[plane] = sc;
  }
}

// cache[plane, pos0 + r, :] *= scale[plane] for r < rows (8 bf16 per thread step)
__global__ void rescale_apply_kernel(__nv_bfloat16* cache, const float* scale, int64_t planes,
                                     int64_t cache_len, int64_t pos0, int64_t rows, int hd) {
  const int64_t per_plane = rows * (hd / 8);
  const int64_t total = planes * per_plane;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t plane = i / per_plane, rem = i % per_plane;
    const int64_t r = rem / (hd / 8), c8 = rem % (hd / 8);
    uint4* p = reinterpret_cast<uint4*>(cache + (plane * cache_len + pos0 + r) * hd + 8 * c8);
    const float sc = scale[plane];
    uint4 v = *p;
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      w[e] = pack_bf16(f.x * sc, f.y * sc);
    }
    *p = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

}  // namespace
}  // namespace rf

extern "C" size_t ridgefill_rescale_workspace_size(const rf_rescale_args* a) {
  if (rf::validate_rescale(a) != RF_OK) return 0;
  rf::RescalePlan pl;
  rf::plan_rescale(a, &pl);
  return pl.total;
}

extern "C" rf_status ridgefill_rescale(const rf_rescale_args* a, void* workspace, size_t ws_bytes,
                                       void* stream) {
  using namespace rf;
  rf_status st = validate_rescale(a);
  if (st != RF_OK) return st;
  const void* req[] = {a->H_tail, a->X_true, a->A, a->bias, a->Wk, a->Wv, a->Kc, a->Vc};
  for (const void* p : req)
    if (p == nullptr) return fail(RF_ERR_ARG, "a required pointer is NULL");
  const void* dev[] = {a->H_tail, a->X_true, a->A,  a->A_scale, a->bias, a->gain,
                       a->Wk,     a->Wv,     a->Kc, a->Vc,      a->scale, workspace};
  for (const void* p : dev)
    if (p != nullptr && !aligned16(p)) return fail(RF_ERR_ALIGN, "a device pointer is not 16-byte aligned");
  RescalePlan pl;
  plan_rescale(a, &pl);
  if (workspace == nullptr || ws_bytes < pl.total)
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes", pl.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t c = a->tail_rows, R2 = pl.R2;
  const int ss_tiles = a->d_out / pl.fp.bn_map;
  float* ss = reinterpret_cast<float*>(ws + pl.off_ss);
  uint8_t* proj = ws + pl.off_cache;
  float* scale = reinterpret_cast<float*>(ws + pl.off_scale);
  if ((st = guards_fill(ws, pl.lay, s)) != RF_OK) return st;

  // predicted rows: the map GEMM writes X_hat rows [0, c) of every layer
  MapLaunch m{};
  m.H = a->H_tail;
  m.A = a->A;
  m.A_scale = a->A_scale;
  m.rows = c;
  m.d_in = a->d_in;
  m.d_out = a->d_out;
  m.n_layers = a->n_layers;
  m.slot_layer = -1;
  m.bn = pl.fp.bn_map;
  m.R = R2;
  m.bias = a->bias;
  m.gain = a->gain;
  m.xhat = ws + pl.off_x;
  m.ss = ss;
  if ((st = launch_map(m, s)) != RF_OK) return st;
  // true rows: rows [c, 2c) from g * x
  const int64_t warps = static_cast<int64_t>(a->n_layers) * c;
  true_input_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(a->X_true), static_cast<const __nv_bfloat16*>(a->gain),
      a->n_layers, c, a->d_out, R2, ss_tiles, reinterpret_cast<__nv_bfloat16*>(ws + pl.off_x), ss);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "true-input kernel launch");
  // one K/V GEMM over the 2c stacked rows, the scaled projection only, into scratch
  rf_fill_args f{};
  f.n_layers = a->n_layers;
  f.d_in = a->d_in;
  f.d_out = a->d_out;
  f.n_kv_heads = a->n_kv_heads;
  f.head_dim = a->head_dim;
  f.rows = 2 * c;
  f.pos0 = 0;
  f.cache_len = R2;
  f.rope_theta = 1e4;  // keys of both inputs rotate alike; the norms do not depend on it
  f.rms_eps = a->rms_eps;
  f.Wk = a->Wk;
  f.Wv = a->Wv;
  f.Kc = proj;
  f.Vc = proj;
  FillPlan fp2 = pl.fp;
  fp2.R = R2;  // row stride of the partial sums
  if ((st = launch_kv(&f, fp2, 0, 2 * c, ws + pl.off_x, ss, s, a->which)) != RF_OK) return st;

  // scales, then the filled rows of the cache in place
  const bool values = a->which == RF_RESCALE_VALUES;
  const int64_t planes = static_cast<int64_t>(a->n_layers) * a->n_kv_heads;
  rescale_ratio_kernel<<<static_cast<unsigned>(planes), 256, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(proj), R2, c, a->head_dim, scale, a->scale);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "rescale ratio launch");
  if (a->rows > 0) {
    const int64_t work = planes * a->rows * (a->head_dim / 8);
    const int64_t blocks = (work + 255) / 256 < 8 * sm_count() ? (work + 255) / 256 : 8 * sm_count();
    rescale_apply_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(
        static_cast<__nv_bfloat16*>(values ? a->Vc : a->Kc), scale, planes, a->cache_len, a->pos0,
        a->rows, a->head_dim);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "rescale apply launch");
  }
  return guards_check(ws, pl.lay, s);
}
