// abi_common.h -- host helpers shared by the C-ABI translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include "../../include/ridgefill.h"
#include "rf_internal.h"

namespace rf {

// Record `msg` as the calling thread's last error and return `s`.
rf_status fail(rf_status s, const char* fmt, ...);
rf_status cuda_fail(cudaError_t e, const char* what);

// Device error word of the current device (address in device memory).
int* device_error_word();

// Number of SMs of the current device.
int sm_count();

// 3D tiled tensor map over a bf16 (or f32) array; dims innermost first,
// strides in bytes for dims 1 and 2.  Returns false on an encode error.
bool make_tmap_3d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base, uint64_t d0,
                  uint64_t d1, uint64_t d2, uint64_t stride1, uint64_t stride2, uint32_t box0,
                  uint32_t box1, CUtensorMapSwizzle swizzle);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Device slots for maps streamed from host memory: the copy of layer l + 2
// can run while layer l computes and layer l + 1 waits.
constexpr int kMapSlots = 3;

// Per-device side stream and events for streaming maps from host memory.
struct HostStreamer {
  cudaStream_t copy = nullptr;
  cudaEvent_t copied[kMapSlots] = {};
  cudaEvent_t freed[kMapSlots] = {};
  cudaEvent_t start = nullptr;
};
HostStreamer* host_streamer();  // nullptr on failure (error recorded)

// The map GEMM over `rows` split-state rows starting at H (grouped over all
// maps in A when `slot_layer` < 0, else the single layer `slot_layer` whose
// map is at A).  Writes X_hat [L, R, d_out] and the sums-of-squares partials.
struct MapLaunch {
  const void* H;
  const void* A;
  int64_t rows;
  int32_t d_in, d_out, n_layers;
  int32_t slot_layer;
  int32_t bn;
  int64_t R;  // allocated rows of X_hat / partial buffers
  const float* bias;
  const void* gain;
  void* xhat;
  float* ss;
};
rf_status launch_map(const MapLaunch& m, cudaStream_t s);

}  // namespace rf
