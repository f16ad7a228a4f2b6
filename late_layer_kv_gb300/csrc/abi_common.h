// abi_common.h -- host helpers shared by the C-ABI translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

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
// 4D tiled tensor map (dims innermost first, strides in bytes for dims 1-3, any order of
// magnitude: a dimension may step through memory more finely than the one before it).
bool make_tmap_4d(CUtensorMap* tm, CUtensorMapDataType dtype, const void* base,
                  const uint64_t (&dims)[4], const uint64_t (&strides)[3], const uint32_t (&box)[4],
                  CUtensorMapSwizzle swizzle);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Workspace layout: regions at 256-byte boundaries, in order.  A debug build follows every
// region with a guard band of kGuardBytes; guards_fill writes a pattern into the bands
// before a call's first launch and guards_check compares them after its last (a changed
// word sets kErrGuard in the device error word).  Release builds add no bands.
constexpr size_t kGuardBytes = 4096;
constexpr int kMaxGuards = 24;
struct Layout {
  size_t off = 0;
  int n = 0;
  size_t guard[kMaxGuards] = {};
  size_t take(size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    if (kDebug && n < kMaxGuards) {
      guard[n++] = off;
      off += kGuardBytes;
    }
    return o;
  }
};
rf_status guards_fill(void* ws, const Layout& lay, cudaStream_t s);
rf_status guards_check(void* ws, const Layout& lay, cudaStream_t s);

// Device slots for maps streamed from host memory: the copy of layer l + 2
// can run while layer l computes and layer l + 1 waits.
constexpr int kMapSlots = 3;

// Per-device side stream and events for streaming maps from host memory.
struct HostStreamer {
  cudaStream_t copy = nullptr;
  cudaStream_t side = nullptr;       // work beside a persistent GEMM (fit column sums, GDN projections)
  cudaEvent_t side_start = nullptr;
  cudaEvent_t side_done = nullptr;
  cudaEvent_t side_ev[2] = {};     // side-stream steps taken in turn (Cholesky trailing updates)
  cudaEvent_t copied[kMapSlots] = {};
  cudaEvent_t freed[kMapSlots] = {};
  cudaEvent_t start = nullptr;
  cudaEvent_t h_done = nullptr;  // split state copied from host memory
  uint32_t h_gen = 0;            // value that marks this call's row groups ready
  cudaEvent_t staged[2] = {};    // host map source: copy out of staging half j done
};

// Stream write of a 32-bit value by the GPU's front end, no SM involved: marks a
// host-to-device copy done for a kernel that is already running.  nullptr if the
// driver does not offer it.
using StreamWrite32 = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
StreamWrite32 stream_write32();

// Rows of split state per ready flag when H streams from host memory: a first group of
// kHostFirstRows (the height of the map GEMM's first raster group, so the GEMM starts once
// those rows have landed), then groups of kHostRowGroup (one raster group of the map GEMM);
// both multiples of the pair GEMM's 256-row tiles.
constexpr int kHostFirstRows = 1024;
constexpr int kHostRowGroup = 4096;
// Flag groups of `rows` streamed rows, and the group of row r.
inline int64_t host_row_groups(int64_t rows) {
  return rows <= kHostFirstRows ? 1 : 1 + (rows - kHostFirstRows + kHostRowGroup - 1) / kHostRowGroup;
}

// Split state in page-locked host memory, streamed into device memory `dev` in groups of
// kHostRowGroup rows on the copy stream.  Each group's flag (flags[g], in device memory)
// is set to `gen` by a stream write once its rows have landed, so a map GEMM given the
// flags can start on a group as soon as it is there; the flags are cleared on `s` first.
// Without stream writes `s` waits for the whole copy (overlap false).  hs->h_done is
// recorded after the last group.
struct HostRows {
  const uint8_t* base = nullptr;  // device copy of H
  uint32_t* flags = nullptr;
  uint32_t gen = 0;
  bool overlap = false;
};
rf_status stream_host_rows(HostStreamer* hs, const void* H, int64_t rows, int d_in, uint8_t* dev,
                           uint32_t* flags, cudaStream_t s, HostRows* out);
// Bytes of device memory stream_host_rows needs: rows and ready flags (offsets 0 and the
// returned flags offset).
size_t host_rows_bytes(int64_t rows, int d_in, size_t* flags_off);
HostStreamer* host_streamer();  // nullptr on failure (error recorded)
// Held by a call for as long as it enqueues work on the copy stream (maps or split state).
std::mutex& host_stream_mutex();

// The map GEMM over `rows` split-state rows starting at H (grouped over all
// maps in A when `slot_layer` < 0, else the single layer `slot_layer` whose
// map is at A).  Writes X_hat [L, R, d_out] and the sums-of-squares partials.
struct MapLaunch {
  const void* H;
  const void* A;        // bf16 maps, or int8 codes when A_scale is set
  const void* A_scale;  // bf16 [layers, d_in / 128, d_out] for int8 maps, else null
  int64_t rows;
  int32_t d_in, d_out, n_layers;
  int32_t slot_layer;
  int32_t slot_count;  // layers in the slot (0: one)
  int32_t bn;
  int64_t R;  // allocated rows of X_hat / partial buffers
  const int32_t* out_rows;  // X_hat row of each GEMM row (rows left out are not written), or null
  const uint32_t* h_ready;  // split state streamed from host memory: ready flags, or null
  uint32_t h_gen;
  int64_t h_row_base;       // row of H's first row in the flags' numbering
  const float* bias;
  const void* gain;
  void* xhat;
  float* ss;
};
rf_status launch_map(const MapLaunch& m, cudaStream_t s);
// bf16(q * s) of `layers` int8 maps (codes [layers, d_out, d_in], scales
// [layers, d_in / 128, d_out]) into out [layers, d_out, d_in]
cudaError_t launch_dequant_maps(const void* q, const void* scale, int layers, int d_out, int d_in,
                                void* out, cudaStream_t s);
// The map GEMM of resident int8 maps (m.A codes, m.A_scale scales, every layer) run as
// `group` layers at a time: their bf16(q * s) into `dq` (group * d_out * d_in bf16), then
// the bf16 GEMM of those layers
rf_status launch_map_q8_groups(MapLaunch m, int group, void* dq, cudaStream_t s);
// Layers per group of the resident int8 map GEMM for a q8_group_layers option (0 when the
// codes are converted inside the GEMM, or the maps are not int8 in device memory)
int q8_group(int option, bool q8, bool maps_on_host, int n_layers);

// Gather the split-state rows H[idx[0 .. rc)] ([h_rows, d_in] bf16) into a dense [rc, d_in]
// block; an index outside [0, h_rows) gives a zero row and a device error code.
rf_status launch_gather_rows(const void* H, const int32_t* idx, int64_t rc, int64_t h_rows,
                             int d_in, void* out, cudaStream_t s);

// One layer's map in a device slot: bf16 [d_out, d_in], or (q8) int8 codes
// followed at a 256-byte boundary by the bf16 scales [d_in / 128, d_out].
size_t map_slot_bytes(int d_out, int d_in, bool q8);
// Enqueue on `copy` the host-to-device copy of layer l's map (and scales) into
// `slot`; *dA and *dS receive the slot's code (or bf16) and scale pointers.
cudaError_t copy_map_layer(uint8_t* slot, const void* A, const void* A_scale, int l, int d_out,
                           int d_in, cudaStream_t copy, const void** dA, const void** dS);
// RF_OK if p is page-locked host memory, else RF_ERR_NOT_PINNED with `what` in the message.
rf_status check_pinned(const void* p, const char* what);

}  // namespace rf
