// quant.cu -- ridgefill_quantize_maps: the int8 map format of RidgeFill,
// "Training-Free Late-Layer Cache Fill for Faster Prefill", section 2.2
// ("Size and cost") and section 4.2: int8 codes with one bf16 scale per 128
// consecutive weights of each map row.  HBM-bound: one read of the maps, one
// write of codes and scales.
#include "abi_common.h"
#include "sm103_ptx.cuh"

namespace rf {
namespace {

// One warp per group of 128 weights (lane i holds weights 4i .. 4i + 3):
// s = bf16(max|a| / 127), q = clamp(rint(a / s), -127, 127), both divisions in
// IEEE float32 (round to nearest), rint ties to even; a zero group gets s = q = 0.
// The scale of group gi of map row j in layer l is stored at [l, gi, j].
template <bool kBf16>
__global__ void __launch_bounds__(256) quantize_kernel(const void* A, uint32_t* q,
                                                       __nv_bfloat16* scale, int64_t groups,
                                                       int d_out, int G) {
  const int lane = threadIdx.x & 31;
  const int64_t nw = (static_cast<int64_t>(gridDim.x) * blockDim.x) >> 5;
  for (int64_t g = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; g < groups;
       g += nw) {
    float a[4];
    if (kBf16) {
      const uint2 v = __ldg(reinterpret_cast<const uint2*>(A) + g * 32 + lane);
      const float2 lo = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
      const float2 hi = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
      a[0] = lo.x; a[1] = lo.y; a[2] = hi.x; a[3] = hi.y;
    } else {
      const float4 v = __ldg(reinterpret_cast<const float4*>(A) + g * 32 + lane);
      a[0] = v.x; a[1] = v.y; a[2] = v.z; a[3] = v.w;
    }
    float m = fmaxf(fmaxf(fabsf(a[0]), fabsf(a[1])), fmaxf(fabsf(a[2]), fabsf(a[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const __nv_bfloat16 sb = __float2bfloat16_rn(__fdiv_rn(m, 127.f));
    const float s = __bfloat162float(sb);
    uint32_t packed = 0;
    if (s > 0.f) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int qi = static_cast<int>(rintf(__fdiv_rn(a[e], s)));
        qi = qi > 127 ? 127 : (qi < -127 ? -127 : qi);
        packed |= (static_cast<uint32_t>(qi) & 0xFFu) << (8 * e);
      }
    }
    q[g * 32 + lane] = packed;
    if (lane == 0) {
      const int64_t row = g / G, gi = g - row * G;  // row = l * d_out + j
      const int64_t l = row / d_out, j = row - l * d_out;
      scale[(l * G + gi) * d_out + j] = sb;
    }
  }
}

// bf16(q * s) of layers [0, layers) of int8 maps: 16 codes a thread (one 16-byte load, two
// 16-byte stores); q * s is exact in f32 (8 by 8 significant bits), so the one rounding gives
// the bf16 value the in-GEMM converters produce.
__global__ void __launch_bounds__(256) dequant_maps_kernel(const uint4* q, const __nv_bfloat16* scale,
                                                           int64_t n16, int d_out, int d_in,
                                                           uint4* out) {
  const int64_t per_row = d_in / 16;
  const int G = d_in / kQ8Group;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < n16;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = t / per_row;  // l * d_out + j
    const int i16 = static_cast<int>(t - row * per_row);
    const int64_t l = row / d_out, j = row - l * d_out;
    const float sc = __bfloat162float(scale[(l * G + (i16 * 16) / kQ8Group) * d_out + j]);
    const uint4 v = __ldg(q + t);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int b0 = static_cast<int8_t>(w[e] & 0xFFu), b1 = static_cast<int8_t>((w[e] >> 8) & 0xFFu);
      const int b2 = static_cast<int8_t>((w[e] >> 16) & 0xFFu), b3 = static_cast<int8_t>(w[e] >> 24);
      o[2 * e] = pack_bf16(static_cast<float>(b0) * sc, static_cast<float>(b1) * sc);
      o[2 * e + 1] = pack_bf16(static_cast<float>(b2) * sc, static_cast<float>(b3) * sc);
    }
    out[2 * t] = make_uint4(o[0], o[1], o[2], o[3]);
    out[2 * t + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

}  // namespace

cudaError_t launch_dequant_maps(const void* q, const void* scale, int layers, int d_out, int d_in,
                                void* out, cudaStream_t s) {
  const int64_t n16 = static_cast<int64_t>(layers) * d_out * (d_in / 16);
  const int64_t blocks = (n16 + 255) / 256 < 8 * sm_count() ? (n16 + 255) / 256 : 8 * sm_count();
  dequant_maps_kernel<<<static_cast<unsigned>(blocks > 0 ? blocks : 1), 256, 0, s>>>(
      static_cast<const uint4*>(q), static_cast<const __nv_bfloat16*>(scale), n16, d_out, d_in,
      static_cast<uint4*>(out));
  return cudaGetLastError();
}

}  // namespace rf

extern "C" rf_status ridgefill_quantize_maps(const rf_quantize_args* a, void* stream) {
  using namespace rf;
  if (a == nullptr) return fail(RF_ERR_ARG, "args is NULL");
  if (a->n_maps < 1 || a->d_out < 1 || a->d_in < kQ8Group || a->d_in % kQ8Group != 0)
    return fail(RF_ERR_SHAPE, "need n_maps, d_out >= 1 and d_in a positive multiple of 128");
  if (a->src_bf16 != 0 && a->src_bf16 != 1) return fail(RF_ERR_ARG, "src_bf16 must be 0 or 1");
  if (a->A == nullptr || a->q == nullptr || a->scale == nullptr)
    return fail(RF_ERR_ARG, "a required pointer is NULL");
  if (!aligned16(a->A) || !aligned16(a->q) || !aligned16(a->scale))
    return fail(RF_ERR_ALIGN, "a device pointer is not 16-byte aligned");
  const int64_t groups = static_cast<int64_t>(a->n_maps) * a->d_out * (a->d_in / kQ8Group);
  const int64_t blocks_needed = (groups + 7) / 8;  // eight warps per block
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  const unsigned blocks = static_cast<unsigned>(blocks_needed < cap ? blocks_needed : cap);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto* q = static_cast<uint32_t*>(a->q);
  auto* sc = static_cast<__nv_bfloat16*>(a->scale);
  const int G = a->d_in / kQ8Group;
  if (a->src_bf16) quantize_kernel<true><<<blocks, 256, 0, s>>>(a->A, q, sc, groups, a->d_out, G);
  else quantize_kernel<false><<<blocks, 256, 0, s>>>(a->A, q, sc, groups, a->d_out, G);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return RF_OK;
}
