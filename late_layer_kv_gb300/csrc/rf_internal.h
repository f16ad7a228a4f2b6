// rf_internal.h -- shared declarations of the RidgeFill CUDA library (not ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

// Debug builds (RF_DEBUG=1, a separate library) check the index of every plain global
// store of the kernels against its buffer's extent, skip a store outside and record it,
// and put a guard band after every workspace region that each call fills with a pattern
// first and checks last.  Release builds compile none of this.
#ifndef RF_DEBUG
#define RF_DEBUG 0
#endif

namespace rf {

constexpr bool kDebug = RF_DEBUG != 0;

// ------------------------------------------------------------ GEMM tiling
constexpr int kBM = 128;           // rows per CTA (one TMEM lane per row)
constexpr int kBK = 64;            // K elements per stage (one 128-byte row)
constexpr int kBNMax = 256;        // max columns per tile (TMEM cols per accumulator)
constexpr int kGramWideCols = 512; // Gram tiles on CTA pairs: both accumulators, one tile
constexpr int kOutBoxBytes = 64 * 32 * 2;   // one 64-col x 32-row bf16 store box
constexpr int kOutWarpBytes = 2 * kOutBoxBytes;
constexpr int kGemmThreads = 256;  // warp 0 TMA, warp 1 MMA, warp 2 TMEM, warps 4-7 epilogue
constexpr int kGemmThreadsQ8 = 512;  // int8 maps: warps 8-15 convert the B operand
constexpr int kQ8Group = 128;        // map weights of a row that share one bf16 scale
// dynamic shared memory of the pair GEMM kernels (the stage rings, epilogue staging,
// barriers and 1 KB of alignment slack), within the 227 KB a CTA may use
constexpr int kGemmSmem = 1024 + 4 * (kBM * kBK * 2 + kBNMax * kBK * 2) + 4 * kOutWarpBytes + 256;

enum GemmMode : int {
  kModeMap = 0,      // X_hat = H A^T + b (times gain), row sums of squares
  kModeKV = 1,       // K/V projection, RMS scale, RoPE on K, cache store
  kModeGdnProj = 2,  // GDN projections: RMS scale, k L2-norm, v, sigmoid gates
  kModeGram = 3,     // fit sums: [X | Y_1 .. Y_L]^T X over rows, MN-major operands, f64 add
  kModeSolve = 4,    // fit solve: A = C~^T G^-1 (split bf16), column scale, f32/bf16 out
  kModeF32 = 5,      // plain product, f32 out: alpha acc (+ the stored value), batched or lower tiles
};

// Device error word sites (which wait ran out).
enum ErrSite : int {
  kErrProducer = 1,
  kErrMma = 2,
  kErrEpilogue = 3,
  kErrGdn = 4,
  kErrConvert = 5,   // int8-map converter warps
  kErrIndex = 6,     // a row index list entry was out of range (the row was skipped)
  kErrHostRows = 8,  // a split-state row group copied from host memory never arrived
  kErrProbe = 20,    // ridgefill_wait_selftest: + 0 mbarrier wait, + 1 flag wait
  kErrNumeric = 7,   // the ridge system was not positive definite (Cholesky pivot <= 0)
  kErrGuard = 9,     // debug builds: a workspace guard band was overwritten
  kErrBounds = 10,   // debug builds: a kernel store fell outside its buffer (skipped)
};

// True when element index i lies in [0, n).  Debug builds record a miss in the error
// word; release builds assume it (no check is compiled).
__device__ __forceinline__ bool in_bounds(int64_t i, int64_t n, int* err) {
#if RF_DEBUG
  if (i < 0 || i >= n) {
    atomicCAS(err, 0, static_cast<int>(kErrBounds));
    return false;
  }
#else
  (void)i;
  (void)n;
  (void)err;
#endif
  return true;
}

struct GemmParams {
  CUtensorMap tmA;     // A operand, K-major 3D {K, rows, batch}, box {64, 128, 1}
  CUtensorMap tmA2;    // gram mode: the Y operand, MN-major 3D {d_out, rows, L}, box {64, 64, 1}
  CUtensorMap tmB[4];  // B operand segments, K-major 3D {K, n, batch}, box {64, bn|16, 1}
  CUtensorMap tmO[2];  // outputs, 3D, box {64, 32, 1}
  int32_t mode;
  int32_t k_blocks;    // K / 64
  int32_t m_tiles;
  int32_t n_tiles;     // tiles along N per batch entry
  int32_t batches;     // batch entries (layers) the tile loop covers
  int32_t batch_base;  // batch entry of the first (a layer subset starts past 0)
  int32_t bn;          // MMA N of a tile
  int32_t group_m;     // raster group height
  int32_t group_m0;    // > 0: height of the first raster group (split state streaming in)
  int32_t rows;        // valid rows of this launch
  int32_t ss_stride;   // row stride of the sum-of-squares partials
  int32_t d_out;
  int32_t layer_base;  // map mode: layer of B row 0
  int32_t ss_tiles;    // partials per row per layer
  // int8 maps (map mode on CTA pairs): codes [B rows, q8_ld] and bf16 scales
  // [B rows, q8_ld / 128]; the converter warps write bf16(q * s) into the B stages
  const int8_t* q8;
  const __nv_bfloat16* q8_scale;
  int32_t q8_ld;
  // split state streamed from host memory (map mode): rows of group g (row < h_first_rows:
  // g = 0, else g = 1 + (row - h_first_rows) / h_group_rows; row counted from h_row_base)
  // may be read once h_ready[g] == h_gen
  const uint32_t* h_ready;
  uint32_t h_gen;
  int32_t h_group_rows;
  int32_t h_first_rows;  // rows of group 0 (the later groups have h_group_rows)
  int32_t h_row_base;
  // map epilogue; with map_rows set, tile row r is stored as X_hat row map_rows[r] (row by
  // row, straight from registers) into map_out [L, map_ld, d_out]
  const int32_t* map_rows;
  __nv_bfloat16* map_out;
  int64_t map_ld;
  const float* bias;
  const __nv_bfloat16* gain;
  float* ss_part;
  // K/V epilogue
  const float* ss_in;
  int32_t n_k_tiles;
  int32_t n_kv;
  int32_t head_dim;
  int32_t pos_base;
  float inv_d;
  float eps;
  const float* k_scale;  // [L, n_kv] per-head key scale, or null
  const float* v_scale;  // [L, n_kv] per-head value scale, or null
  // exact prefix rows: when kv_rows is set, tile row r goes to cache position
  // kv_pos0 + kv_rows[r] (kv_rows[r] in [0, kv_hrows)), stored row by row
  const int32_t* kv_rows;
  int32_t kv_pos0;
  int32_t kv_hrows;
  // RoPE angles of this launch's rows: rope_tab[i * rope_ld + row] = (cos, sin) of
  // frequency i at the row's position; null: computed in the epilogue
  const float2* rope_tab;
  int64_t rope_ld;
  __nv_bfloat16* kv_cache[2];  // K, V caches [L, n_kv, cache_len, head_dim]
  int64_t cache_len;
  // GDN projection epilogue
  __nv_bfloat16* gdn_k;  // [L, H, 2, rows_alloc, dk]: bf16 high part, then the low remainder
  __nv_bfloat16* gdn_v;  // [L, H, 2, rows_alloc, dv], same split
  float* gdn_gate;     // [L, 2, H, rows_alloc] f32 (alpha, beta)
  int32_t gdn_heads;
  int32_t gdn_rows_alloc;
  int32_t n_v_tiles;
  float l2_eps;
  // gram epilogue (MN-major operands; A = X for the first gram_x_tiles M tiles, else Y)
  int32_t gram_x_tiles;
  int32_t gram_y_tiles_per_layer;
  double* gram_G;      // [d_in, d_in]
  double* gram_C;      // [L, d_out, d_in]
  int32_t gram_ld;     // d_in
  // symmetric Gram product (with `lower`): G is stored, not added to, and each pair tile
  // below the diagonal also stores its transpose
  int32_t gram_sym;
  // solve epilogue
  const float* col_scale;   // [N]
  const float* mu_x;        // [N]
  float* out_f32;           // [M, N] or null
  __nv_bfloat16* out_bf16;  // [M, N] or null
  float* bias_part;         // [M, n_tiles]
  int32_t out_ld;
  // plain f32 epilogue: out_f32[b * out_bstride + row * out_ld + col] = alpha acc (plus the
  // stored value when beta_one) for rows < rows and cols < cols; with lower set the tiles
  // are the pair tiles on and below the diagonal of a square product (bn = 2 kBM, one batch)
  int64_t out_bstride;
  float alpha;
  int32_t beta_one;
  int32_t lower;
  int32_t cols;
  int* err;
  int* tile_ctr;  // this launch's tile counter (zeroed before the launch): tiles are taken in order
  // K-major bf16 map mode: stages of two k-blocks, each operand staged by one copy through a
  // rank-3 view {64 k, rows, k-blocks} (three stages in the space of six)
  int32_t k2;
  // elements of the buffers the epilogue writes with plain stores (checked by debug
  // builds): map mode ss_part, map_out; K/V mode with a row list the caches (per tensor);
  // GDN mode gdn_gate; Gram mode gram_G, gram_C; solve mode the outputs, bias_part; f32
  // mode out_f32 (lim_b)
  int64_t lim_a, lim_b;
  float inv_freq_hi[64];
  float inv_freq_lo[64];
};

// A zeroed-before-use counter for one pair-GEMM launch's dynamic tile order (a slot of a
// library-owned device array of the current device; slots rotate over launches)
int* tile_counter_slot();

// every mode on CTA pairs (B tensor maps with boxes of half a tile's columns); `pairs`
// clusters of 2.  With `ctr` set, the launch takes its tiles from that counter (zeroed by
// the caller before the first of the launches that share it) instead of a fresh one: two
// launches of the same tiles on one counter split the tiles between them.
cudaError_t launch_gemm2(const GemmParams& p, int pairs, cudaStream_t stream, int* ctr = nullptr);
// map mode on CTA pairs with int8 maps (p.q8, p.q8_scale); tmB unused
cudaError_t launch_gemm2_q8(const GemmParams& p, int pairs, cudaStream_t stream);

// ------------------------------------------------------------ GDN state
struct GdnStateParams {
  CUtensorMap tmK;     // k hi/lo, 3D {dk, rows, L*H*2}, box {64, 64, 1}, 128-byte swizzle
  CUtensorMap tmV;     // v hi/lo, same layout
  const float* gate;   // [L, 2, H, rows_alloc]: alpha, then beta
  const float* S0;     // [L, H, dv, dk] or null
  float* S;            // [L, H, dv, dk]
  int32_t layers;
  int32_t heads;
  int32_t rows;        // rows of this launch
  int32_t rows_alloc;
  int32_t first;       // 1 if S starts from S0/zero, 0 if it continues from S
  int32_t layer_base;  // layer of grid row 0 (a layer subset starts past 0)
  int* err;
};
cudaError_t launch_gdn_state(const GdnStateParams& p, cudaStream_t stream);

// ------------------------------------------------------------ fit
struct FitParams;  // defined in fit.cu

}  // namespace rf
