// gdn.cu -- ridgefill_fill_gdn: end-of-fill recurrent state of Gated DeltaNet
// late layers (RidgeFill, "Training-Free Late-Layer Cache Fill for Faster
// Prefill", section 2.3: every filled row updates the shared state from its
// predicted input).
//
// Per row chunk: the grouped map GEMM (X_hat for every GDN layer), the GDN
// projection GEMM (RMS scale, L2-normalised k per head, v, alpha, beta),
// then the state kernel, which carries S over the chunk's rows in order.
//
// State kernel.  For one head the recurrence
//   S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
// is, row by row of S (index i over d_v),
//   S_t[i,:] = alpha_t S_{t-1}[i,:] + c_t[i] k_t^T,
//   c_t[i]   = beta_t (v_t[i] - alpha_t S_{t-1}[i,:] . k_t),
// so the d_v rows of S evolve independently.  A CTA owns 64 rows of S of one
// (layer, head) in registers: each thread two rows and 32 columns, taken as
// every fourth 16-byte chunk so that the four threads of a row read k from
// distinct shared-memory banks.  The
// decay is applied lazily: the registers hold S / g, g being the product of
// the gates since the last renormalisation, so a prompt row costs one FMA per
// element for the dot product and one for the update.  k, v and the gates are
// staged through shared memory 16 prompt rows at a time with cp.async in a
// four-deep ring, so the loads run three stages ahead of the arithmetic.
#include <cmath>
#include <mutex>

#include "abi_common.h"
#include "sm103_ptx.cuh"

namespace rf {
namespace {

constexpr int kSRows = 64;      // rows of S (d_v) per CTA, two per thread
constexpr int kGdnThreads = 128;
constexpr int kStageRows = 16;  // prompt rows per staging buffer
constexpr int kBufs = 4;        // staging ring depth (loads run kBufs - 1 stages ahead)
constexpr int kDk = 128;
constexpr int kStateSmem = kBufs * (kStageRows * (kDk + kSRows) + 2 * kStageRows) * 4;
constexpr float kRenorm = 1e-20f;

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem)), "l"(gmem)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// d = a * b + c on two float lanes at once (one issued instruction)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

__global__ void __launch_bounds__(kGdnThreads) gdn_state_kernel(const GdnStateParams p) {
  extern __shared__ __align__(16) float smem_f[];
  float (*sk)[kStageRows][kDk] = reinterpret_cast<float (*)[kStageRows][kDk]>(smem_f);
  float (*sv)[kStageRows][kSRows] =
      reinterpret_cast<float (*)[kStageRows][kSRows]>(smem_f + kBufs * kStageRows * kDk);
  float (*sg)[2][kStageRows] = reinterpret_cast<float (*)[2][kStageRows]>(
      smem_f + kBufs * kStageRows * (kDk + kSRows));

  const int slice = blockIdx.x, h = blockIdx.y, l = blockIdx.z;
  const int tid = threadIdx.x;
  const int rp = tid >> 2;    // this thread owns S rows rp and rp + 32 of the slice
  const int part = tid & 3;   // and the 16-byte column chunks part, part + 4, ..., part + 28
  const int i0 = slice * kSRows + rp;
  const int H = p.heads;
  const size_t ra = static_cast<size_t>(p.rows_alloc);
  const int dv = p.dv;

  const float* kbase = p.k + (static_cast<size_t>(l) * H + h) * ra * kDk;
  const float* vbase = p.v + (static_cast<size_t>(l) * H + h) * ra * dv + slice * kSRows;
  const float* abase = p.gate + (static_cast<size_t>(l) * 2 * H + h) * ra;
  const float* bbase = p.gate + (static_cast<size_t>(l) * 2 * H + H + h) * ra;
  const size_t row0 = ((static_cast<size_t>(l) * H + h) * dv + i0) * kDk;
  const size_t row1 = row0 + static_cast<size_t>(32) * kDk;

  // S0, S1 hold columns 4 (part + 4 q) + e at pair 2 q + e / 2
  float2 S0[16], S1[16];
  const float* src = p.first ? p.S0 : p.S;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    float4 x0 = make_float4(0.f, 0.f, 0.f, 0.f), x1 = x0;
    if (src != nullptr) {
      x0 = *reinterpret_cast<const float4*>(src + row0 + 4 * (part + 4 * q));
      x1 = *reinterpret_cast<const float4*>(src + row1 + 4 * (part + 4 * q));
    }
    S0[2 * q] = make_float2(x0.x, x0.y); S0[2 * q + 1] = make_float2(x0.z, x0.w);
    S1[2 * q] = make_float2(x1.x, x1.y); S1[2 * q + 1] = make_float2(x1.z, x1.w);
  }
  float g = 1.f;

  const int nst = (p.rows + kStageRows - 1) / kStageRows;
  auto load = [&](int st, int buf) {
    const int t0 = st * kStageRows;
    const int n = min(kStageRows, p.rows - t0);
    for (int q = tid; q < n * (kDk / 4); q += kGdnThreads) {
      const int rr = q / (kDk / 4), cc = q % (kDk / 4);
      cp_async16(&sk[buf][rr][cc * 4], kbase + static_cast<size_t>(t0 + rr) * kDk + cc * 4);
    }
    for (int q = tid; q < n * (kSRows / 4); q += kGdnThreads) {
      const int rr = q / (kSRows / 4), cc = q % (kSRows / 4);
      cp_async16(&sv[buf][rr][cc * 4], vbase + static_cast<size_t>(t0 + rr) * dv + cc * 4);
    }
    if (tid < 2 * (kStageRows / 4)) {
      const int which = tid / (kStageRows / 4), cc = tid % (kStageRows / 4);
      if (cc * 4 < n)  // gate rows are padded to the 128-row allocation
        cp_async16(&sg[buf][which][cc * 4], (which ? bbase : abase) + t0 + cc * 4);
    }
    cp_async_commit();
  };

  // one cp.async group per stage (empty past the end) keeps the group count uniform
  for (int q = 0; q < kBufs - 1; ++q) {
    if (q < nst) load(q, q);
    else cp_async_commit();
  }
  for (int st = 0; st < nst; ++st) {
    const int buf = st % kBufs;
    const int ahead = st + kBufs - 1;
    if (ahead < nst) load(ahead, ahead % kBufs);
    else cp_async_commit();
    cp_async_wait<kBufs - 1>();
    __syncthreads();
    const int n = min(kStageRows, p.rows - st * kStageRows);
    for (int tt = 0; tt < n; ++tt) {
      const float a = sg[buf][0][tt];
      const float bt = sg[buf][1][tt];
      const float v0 = sv[buf][tt][rp], v1 = sv[buf][tt][rp + 32];
      float2 kk[16];
      const float4* k4 = reinterpret_cast<const float4*>(&sk[buf][tt][0]);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 x = k4[part + 4 * q];
        kk[2 * q] = make_float2(x.x, x.y);
        kk[2 * q + 1] = make_float2(x.z, x.w);
      }
      float2 e0a = make_float2(0.f, 0.f), e0b = e0a, e1a = e0a, e1b = e0a;
#pragma unroll
      for (int j = 0; j < 16; j += 2) {
        e0a = ffma2(S0[j], kk[j], e0a);
        e0b = ffma2(S0[j + 1], kk[j + 1], e0b);
        e1a = ffma2(S1[j], kk[j], e1a);
        e1b = ffma2(S1[j + 1], kk[j + 1], e1b);
      }
      float e0 = (e0a.x + e0a.y) + (e0b.x + e0b.y);
      float e1 = (e1a.x + e1a.y) + (e1b.x + e1b.y);
      e0 += __shfl_xor_sync(0xffffffffu, e0, 1);
      e1 += __shfl_xor_sync(0xffffffffu, e1, 1);
      e0 += __shfl_xor_sync(0xffffffffu, e0, 2);
      e1 += __shfl_xor_sync(0xffffffffu, e1, 2);
      // true S_{t-1}[i,:] k_t = g * e
      const float ag = a * g;
      const float c0 = bt * (v0 - ag * e0);
      const float c1 = bt * (v1 - ag * e1);
      if (ag >= kRenorm) {
        const float inv = 1.f / ag;
        const float2 s0 = make_float2(c0 * inv, c0 * inv), s1 = make_float2(c1 * inv, c1 * inv);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          S0[j] = ffma2(s0, kk[j], S0[j]);
          S1[j] = ffma2(s1, kk[j], S1[j]);
        }
        g = ag;
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          S0[j] = make_float2(fmaf(c0, kk[j].x, ag * S0[j].x), fmaf(c0, kk[j].y, ag * S0[j].y));
          S1[j] = make_float2(fmaf(c1, kk[j].x, ag * S1[j].x), fmaf(c1, kk[j].y, ag * S1[j].y));
        }
        g = 1.f;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    *reinterpret_cast<float4*>(p.S + row0 + 4 * (part + 4 * q)) =
        make_float4(g * S0[2 * q].x, g * S0[2 * q].y, g * S0[2 * q + 1].x, g * S0[2 * q + 1].y);
    *reinterpret_cast<float4*>(p.S + row1 + 4 * (part + 4 * q)) =
        make_float4(g * S1[2 * q].x, g * S1[2 * q].y, g * S1[2 * q + 1].x, g * S1[2 * q + 1].y);
  }
}

struct GdnPlan {
  int bn_map = 0;
  int64_t R = 0;
  size_t off_xhat = 0, off_ss = 0, off_k = 0, off_v = 0, off_gate = 0, off_slots = 0, total = 0;
};

rf_status validate_gdn(const rf_gdn_args* a) {
  if (a == nullptr) return fail(RF_ERR_ARG, "args is NULL");
  if (a->n_layers < 1) return fail(RF_ERR_SHAPE, "n_layers must be >= 1");
  if (a->d_in < 64 || a->d_in % 64 != 0) return fail(RF_ERR_SHAPE, "d_in must be a positive multiple of 64");
  if (a->d_out < 128 || a->d_out % 128 != 0)
    return fail(RF_ERR_SHAPE, "d_out must be a positive multiple of 128");
  if (a->d_k != kDk || a->d_v != kDk) return fail(RF_ERR_SHAPE, "d_k and d_v must be 128");
  if (a->n_heads < 8 || a->n_heads > 64 || a->n_heads % 8 != 0)
    return fail(RF_ERR_SHAPE, "n_heads must be a multiple of 8 in [8, 64]");
  if (a->chunk != 64) return fail(RF_ERR_SHAPE, "chunk must be 64");
  if (a->rows < 0) return fail(RF_ERR_ARG, "rows must be >= 0");
  if (a->rows_per_chunk < 0 || a->rows_per_chunk % 128 != 0)
    return fail(RF_ERR_SHAPE, "rows_per_chunk must be 0 or a multiple of 128");
  if (!(a->rms_eps >= 0.0) || !(a->l2_eps >= 0.0)) return fail(RF_ERR_ARG, "bad rms_eps or l2_eps");
  if (a->maps_on_host != 0 && a->maps_on_host != 1) return fail(RF_ERR_ARG, "maps_on_host must be 0 or 1");
  if (a->rows >= (int64_t(1) << 31) || static_cast<int64_t>(a->n_layers) * a->d_out >= (int64_t(1) << 31))
    return fail(RF_ERR_SHAPE, "sizes exceed the 32-bit tile indexing");
  return RF_OK;
}

void plan_gdn(const rf_gdn_args* a, GdnPlan* pl) {
  pl->bn_map = (a->d_out % 256 == 0) ? 256 : 128;
  const int64_t all = ceil_div(a->rows > 0 ? a->rows : 1, kBM) * kBM;
  pl->R = a->rows_per_chunk > 0 ? (a->rows_per_chunk < all ? a->rows_per_chunk : all) : all;
  const size_t L = a->n_layers, d = a->d_out, R = pl->R, H = a->n_heads;
  size_t off = 0;
  pl->off_xhat = off;  off = align_up(off + L * R * d * 2, 256);
  pl->off_ss = off;    off = align_up(off + L * (d / pl->bn_map) * R * 4, 256);
  pl->off_k = off;     off = align_up(off + L * H * R * kDk * 4, 256);
  pl->off_v = off;     off = align_up(off + L * H * R * kDk * 4, 256);
  pl->off_gate = off;  off = align_up(off + L * 2 * H * R * 4, 256);
  pl->off_slots = off; off = align_up(off + (a->maps_on_host ? kMapSlots * d * static_cast<size_t>(a->d_in) * 2 : 0), 256);
  pl->total = off;
}

rf_status launch_gdn_proj(const rf_gdn_args* a, const GdnPlan& pl, int64_t rc, const void* xhat,
                          const float* ss, float* kb, float* vb, float* gb, cudaStream_t s) {
  GemmParams p{};
  p.mode = kModeGdnProj;
  p.k_blocks = a->d_out / kBK;
  const int H = a->n_heads;
  const uint64_t drow = static_cast<uint64_t>(a->d_out) * 2;
  const uint64_t hk = static_cast<uint64_t>(H) * kDk;
  bool ok = make_tmap_3d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xhat, a->d_out, rc, a->n_layers,
                         drow, drow * pl.R, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_3d(&p.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Wk, a->d_out, hk,
                          a->n_layers, drow, drow * hk, kBK, 256, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_3d(&p.tmB[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Wv, a->d_out, hk,
                          a->n_layers, drow, drow * hk, kBK, 256, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_3d(&p.tmB[2], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Wa, a->d_out, H,
                          a->n_layers, drow, drow * H, kBK, H, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_3d(&p.tmB[3], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a->Wb, a->d_out, H,
                          a->n_layers, drow, drow * H, kBK, H, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the GDN projection GEMM");
  p.m_tiles = static_cast<int32_t>(ceil_div(rc, kBM));
  p.n_k_tiles = H / 2;
  p.n_v_tiles = H / 2;
  p.n_tiles = H + 1;
  p.batches = a->n_layers;
  p.bn = 256;
  p.group_m = 16;
  p.rows = static_cast<int32_t>(rc);
  p.ss_stride = static_cast<int32_t>(pl.R);
  p.d_out = a->d_out;
  p.ss_tiles = a->d_out / pl.bn_map;
  p.ss_in = ss;
  p.inv_d = static_cast<float>(1.0 / a->d_out);
  p.eps = static_cast<float>(a->rms_eps);
  p.gdn_k = kb;
  p.gdn_v = vb;
  p.gdn_gate = gb;
  p.gdn_heads = H;
  p.gdn_rows_alloc = static_cast<int32_t>(pl.R);
  p.l2_eps = static_cast<float>(a->l2_eps);
  p.err = device_error_word();
  if (p.err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles * p.batches;
  const int grid = static_cast<int>(tiles < sm_count() ? tiles : sm_count());
  if (grid <= 0) return RF_OK;
  cudaError_t e = launch_gemm(p, grid, s);
  if (e != cudaSuccess) return cuda_fail(e, "GDN projection GEMM launch");
  return RF_OK;
}

std::mutex g_gdn_host_map_mu;

}  // namespace

cudaError_t launch_gdn_state(const GdnStateParams& p, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(gdn_state_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kStateSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.dv / kSRows, p.heads, p.layers);
  gdn_state_kernel<<<grid, kGdnThreads, kStateSmem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace rf

using namespace rf;

extern "C" size_t ridgefill_gdn_workspace_size(const rf_gdn_args* a) {
  if (validate_gdn(a) != RF_OK) return 0;
  GdnPlan pl;
  plan_gdn(a, &pl);
  return pl.total;
}

extern "C" rf_status ridgefill_fill_gdn(const rf_gdn_args* a, void* workspace, size_t ws_bytes,
                                        void* stream) {
  rf_status st = validate_gdn(a);
  if (st != RF_OK) return st;
  if (a->S == nullptr) return fail(RF_ERR_ARG, "S is NULL");
  if (a->rows > 0) {
    const void* req[] = {a->H, a->A, a->bias, a->Wk, a->Wv, a->Wa, a->Wb};
    for (const void* q : req)
      if (q == nullptr) return fail(RF_ERR_ARG, "a required pointer is NULL");
  }
  const void* dev[] = {a->H, a->bias, a->gain, a->Wk, a->Wv, a->Wa, a->Wb, a->S0, a->S, workspace};
  for (const void* q : dev)
    if (q != nullptr && !aligned16(q)) return fail(RF_ERR_ALIGN, "a device pointer is not 16-byte aligned");
  if (a->A != nullptr && !aligned16(a->A)) return fail(RF_ERR_ALIGN, "A is not 16-byte aligned");
  if (a->maps_on_host && a->rows > 0) {
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, a->A);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeHost) {
      cudaGetLastError();
      return fail(RF_ERR_NOT_PINNED, "maps_on_host set but A is not page-locked host memory");
    }
  }
  GdnPlan pl;
  plan_gdn(a, &pl);
  if (workspace == nullptr || ws_bytes < pl.total)
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes", pl.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* xhat = ws + pl.off_xhat;
  float* ss = reinterpret_cast<float*>(ws + pl.off_ss);
  float* kb = reinterpret_cast<float*>(ws + pl.off_k);
  float* vb = reinterpret_cast<float*>(ws + pl.off_v);
  float* gb = reinterpret_cast<float*>(ws + pl.off_gate);

  GdnStateParams sp{};
  sp.k = kb;
  sp.v = vb;
  sp.gate = gb;
  sp.S0 = a->S0;
  sp.S = a->S;
  sp.layers = a->n_layers;
  sp.heads = a->n_heads;
  sp.dv = a->d_v;
  sp.rows_alloc = static_cast<int32_t>(pl.R);
  sp.chunk = a->chunk;
  sp.err = device_error_word();

  if (a->rows == 0) {  // the end-of-fill state is the initial state
    sp.rows = 0;
    sp.first = 1;
    cudaError_t e = launch_gdn_state(sp, s);
    return e == cudaSuccess ? RF_OK : cuda_fail(e, "GDN state launch");
  }

  HostStreamer* hs = nullptr;
  std::unique_lock<std::mutex> lk(g_gdn_host_map_mu, std::defer_lock);
  const size_t map_bytes = static_cast<size_t>(a->d_out) * a->d_in * 2;
  if (a->maps_on_host) {
    lk.lock();
    hs = host_streamer();
    if (hs == nullptr) return RF_ERR_CUDA;
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
    const int64_t rc = (a->rows - start < pl.R) ? a->rows - start : pl.R;
    if ((st = mark(start, 0)) != RF_OK) return st;
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
      if ((st = launch_map(m, s)) != RF_OK) return st;
    } else {
      for (int l = 0; l < a->n_layers; ++l) {
        const int k = l % kMapSlots;
        uint8_t* slot = ws + pl.off_slots + k * map_bytes;
        cudaError_t e = cudaSuccess;
        if (start > 0 || l >= kMapSlots) e = cudaStreamWaitEvent(hs->copy, hs->freed[k], 0);
        if (e == cudaSuccess)
          e = cudaMemcpyAsync(slot, static_cast<const uint8_t*>(a->A) + l * map_bytes, map_bytes,
                              cudaMemcpyHostToDevice, hs->copy);
        if (e == cudaSuccess) e = cudaEventRecord(hs->copied[k], hs->copy);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hs->copied[k], 0);
        if (e != cudaSuccess) return cuda_fail(e, "streaming a map from host memory");
        m.A = slot;
        m.slot_layer = l;
        if ((st = launch_map(m, s)) != RF_OK) return st;
        e = cudaEventRecord(hs->freed[k], s);
        if (e != cudaSuccess) return cuda_fail(e, "recording a map slot release");
      }
    }
    if ((st = mark(start, 1)) != RF_OK) return st;
    if ((st = launch_gdn_proj(a, pl, rc, xhat, ss, kb, vb, gb, s)) != RF_OK) return st;
    if ((st = mark(start, 2)) != RF_OK) return st;
    sp.rows = static_cast<int32_t>(rc);
    sp.first = start == 0 ? 1 : 0;
    cudaError_t e = launch_gdn_state(sp, s);
    if (e != cudaSuccess) return cuda_fail(e, "GDN state launch");
    if ((st = mark(start, 3)) != RF_OK) return st;
  }
  return RF_OK;
}
