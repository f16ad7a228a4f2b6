// gdn.cu -- ridgefill_fill_gdn: end-of-fill recurrent state of Gated DeltaNet
// late layers (RidgeFill, "Training-Free Late-Layer Cache Fill for Faster
// Prefill", section 2.3: every filled row updates the shared state from its
// predicted input).
//
// Per row chunk: the grouped map GEMM (X_hat for every GDN layer), the GDN
// projection GEMM (RMS scale, L2-normalised k per head, v, alpha, beta; k and v
// stored as bf16 high parts plus bf16 remainders), then the state kernel.
//
// State kernel: the recurrence S_t = a_t S_{t-1} (I - b_t k_t k_t^T) + b_t v_t k_t^T
// in chunks of C = 64 rows on the tensor cores.  Inside a chunk, with the
// cumulative log gates G_t = sum_{s<=t} log a_s, g_t = e^{G_t}, the rows of
//   NEW = (I + B)^-1 (diag(b) V - diag(b g) K S_0^T),
//   B_ts = b_t e^{G_t - G_s} k_t.k_s for s < t (else 0)
// are the per-row innovations b_t (v_t - a_t S_{t-1} k_t), and
//   S_C = g_C S_0 + NEW^T diag(e^{G_C - G_t}) K.
// With T = (I + B)^-1, W = T diag(b g) K and U = T diag(b) V (the WY factors)
// this is NEW^T = U^T - S_0 W^T, which needs S_0 only in two products per chunk.
//
// One CTA per (layer, head) carries S through the chunks in TMEM (f32).  Its
// roles:
//   warp 9      TMA producers: lane 0 streams k (hi and lo) and the gates into
//               three chunk buffers, lane 1 streams v into one;
//   warp 8      MMA issuer (one thread) and TMEM owner;
//   warps 4-7   chunk-local work: B from P = K K^T (tensor cores), T = (I + B)^-1
//               by 16 x 16 diagonal blocks and a recursive 2 x 2 block inverse
//               (CUDA cores, in place), and the T operands of U^T, W^T;
//   warps 0-3   the serial part: the -W operand, NEW^T = U^T - S_0 W^T (tensor
//               cores, added to U^T in TMEM), its decay-weighted bf16 split,
//               S += NEW'^T K, and the bf16 split of the new S for the next chunk.
// The issuer sends P of the next chunk as soon as its keys have landed and the
// previous P has been read, so the chunk-local work of chunk c + 1 overlaps the
// serial part of chunk c.  Every product takes bf16 high and low parts of both
// operands (hi.hi + hi.lo + lo.hi, about 16 significant bits; P also lo.lo);
// S and NEW' are A operands read from TMEM, the rest come from
// 128-byte-swizzled shared-memory tiles.  Where the operand shared by two split
// terms allows, the terms are one N = 128 product whose two 64-column halves are
// summed afterwards.
#include <cmath>
#include <mutex>

#include "abi_common.h"
#include "sm103_ptx.cuh"

namespace rf {
namespace {

constexpr int kC = 64;         // rows per chunk
constexpr int kDk = 128;       // d_k = d_v
constexpr int kStateThreads = 320;
constexpr int kPreBar = 1;     // named barrier of warps 4-7

// shared memory, from a 1024-byte aligned base
constexpr uint32_t kBox = 8192;                     // one 64 x 64 bf16 swizzled box
constexpr uint32_t kKV = 4 * kBox;                  // hi, lo of columns 0-63, then of 64-127
constexpr int kKBufs = 3;                           // chunk buffers of k (and its gates)
constexpr uint32_t kOffK = 0;
constexpr uint32_t kOffV = kOffK + kKBufs * kKV;    // one chunk buffer of v
constexpr uint32_t kOffT = kOffV + kKV;             // T diag(b g) hi, lo; T diag(b) hi, lo
constexpr uint32_t kOffW = kOffT + 4 * kBox;        // -W hi, lo: [j][t] rows (MN-major B)
constexpr uint32_t kOffGateRaw = kOffW + 4 * kBox;  // per k buffer: alpha[64], beta[64]
constexpr uint32_t kOffGate = kOffGateRaw + kKBufs * 512;  // three slots: beta, b g, decay, G2
constexpr uint32_t kOffScr = kOffGate + 3 * 1024;          // B, then T in place: [64][68] f32
constexpr int kLd = 68;  // 16-byte rows; 8 consecutive rows cover all banks
constexpr uint32_t kOffBar = kOffScr + kC * kLd * 4;
constexpr uint32_t kStateSmem = kOffBar + 256 + 1024;
static_assert(kStateSmem <= 232448, "state kernel shared memory");

// TMEM columns
constexpr uint32_t kColS = 0;     // S (f32, 128)
constexpr uint32_t kColSh = 128;  // S bf16 high parts (64 columns = 128 values)
constexpr uint32_t kColSl = 192;  // S bf16 remainders
constexpr uint32_t kColN = 256;   // U^T, then NEW^T, as two 64-column parts to be summed
constexpr uint32_t kColNh = 256;  // NEW'^T bf16 high parts (32 columns, over the read NEW^T)
constexpr uint32_t kColNl = 320;  // NEW'^T remainders (over the read second part)
constexpr uint32_t kColP = 384;   // P = K K^T (f32, 64; rows 0-63)
constexpr uint32_t kColW = 448;   // W^T (f32, 64)

// barriers
enum : int {
  kBarKFull = 0,   // 3: k + gates of a chunk landed
  kBarKEmpty = 3,  // 3: the chunk's last product that reads k is done
  kBarVFull = 6,
  kBarVEmpty = 7,
  kBarP = 8,       // P done
  kBarUW = 9,      // U^T and W^T done
  kBarDA = 10,     // NEW^T done
  kBarDB = 11,     // S update done
  kBarTops = 12,   // T operands written (4 warp arrivals)
  kBarWop = 13,    // -W operand written (4 warp arrivals)
  kBarNop = 14,    // NEW' operand written (4 warp arrivals)
  kBarSops = 15,   // S operand written and S pre-scaled (4 warp arrivals)
  kBarFinal = 16,
  kBarPfree = 17,  // P read out of TMEM (4 warp arrivals)
  kNumBars = 18,
};

// gates are kept in log2 units; a gate below 2^-115 counts as 2^-115
constexpr float kMinLog2Gate = -115.f;

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// bf16 high parts and remainders of 8 values, packed two per word (lower index low)
__device__ __forceinline__ void split8(const float (&x)[8], uint4& hi, uint4& lo) {
  uint32_t h[4], r[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    h[e] = *reinterpret_cast<const uint32_t*>(&hv);
    r[e] = pack_bf16(x[2 * e] - __low2float(hv), x[2 * e + 1] - __high2float(hv));
  }
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(r[0], r[1], r[2], r[3]);
}
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 hv = __floats2bfloat162_rn(x0, x1);
  hi = *reinterpret_cast<const uint32_t*>(&hv);
  lo = pack_bf16(x0 - __low2float(hv), x1 - __high2float(hv));
}

// log2 of the chunk's total decay: warp-wide sum of log2 alpha over its n rows
__device__ __forceinline__ float chunk_log2_decay(const float* alpha, int n, int lane) {
  float s = 0.f;
  for (int t = lane; t < n; t += 32) s += fmaxf(log2f(alpha[t]), kMinLog2Gate);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ float4 fma4(float a, float4 b, float4 c) {
  return make_float4(fmaf(a, b.x, c.x), fmaf(a, b.y, c.y), fmaf(a, b.z, c.z), fmaf(a, b.w, c.w));
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// 2 x 4 tile (rows r and r + 8, columns 4 cg .. 4 cg + 3) of the product of
// the 16 x (16 n) row panel at A (stride kLd) and the (16 n) x 16 column panel at B.
template <int N>
__device__ __forceinline__ void tile_product(const float* A, const float* B, int r, int cg,
                                             float4& y0, float4& y1) {
  y0 = make_float4(0.f, 0.f, 0.f, 0.f);
  y1 = y0;
#pragma unroll 1
  for (int k = 0; k < 16 * N; k += 4) {
    const float4 a0 = ld4(A + r * kLd + k), a1 = ld4(A + (r + 8) * kLd + k);
    const float a0v[4] = {a0.x, a0.y, a0.z, a0.w}, a1v[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const float4 bv = ld4(B + (k + kk) * kLd + 4 * cg);
      y0 = fma4(a0v[kk], bv, y0);
      y1 = fma4(a1v[kk], bv, y1);
    }
  }
}

// P = K K^T of one chunk: 16 MMAs with A = [K_hi; K_lo] (128 K-major rows: a box of high
// parts and the box of remainders after it, `kd` its descriptor) and B = K_hi, then K_lo.
// Out of line: the MMA warp issues it from inside each of its waits.
__device__ __noinline__ void issue_p_mmas(uint32_t d_tmem, uint64_t kd, uint32_t id_p) {
#pragma unroll
  for (int g = 0; g < 2; ++g)
#pragma unroll
    for (int kblk = 0; kblk < 2; ++kblk)
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        const uint32_t o = (kblk * 2 * kBox + 32 * ks) >> 4;
        mma_bf16(d_tmem, kd + o, kd + o + (g == 1 ? kBox >> 4 : 0), id_p,
                 (g | kblk | ks) != 0 ? 1u : 0u);
      }
}

__global__ void __launch_bounds__(kStateThreads, 1)
    gdn_state_kernel(const __grid_constant__ GdnStateParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(sm);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + kNumBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tslot + 1);
  float* Bs = reinterpret_cast<float*>(sm + kOffScr);
  float* Xs = reinterpret_cast<float*>(sm + kOffT);  // scratch while T is formed

  const int h = blockIdx.x, l = blockIdx.y + p.layer_base;
  const int H = p.heads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int lh = l * H + h;
  const size_t ra = static_cast<size_t>(p.rows_alloc);
  const float* alpha_g = p.gate + (static_cast<size_t>(l) * 2 * H + h) * ra;
  const float* beta_g = p.gate + (static_cast<size_t>(l) * 2 * H + H + h) * ra;
  float* s_out = p.S + static_cast<size_t>(lh) * kDk * kDk;
  const float* s_in = p.first ? (p.S0 != nullptr ? p.S0 + static_cast<size_t>(lh) * kDk * kDk
                                                 : nullptr)
                              : s_out;
  const int nch = (p.rows + kC - 1) / kC;

  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) mbar_init(&bar[i], 1);
    mbar_init(&bar[kBarTops], 4);
    mbar_init(&bar[kBarWop], 4);
    mbar_init(&bar[kBarNop], 4);
    mbar_init(&bar[kBarSops], 4);
    mbar_init(&bar[kBarPfree], 4);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = *tslot;

  if (warp == 9) {
    // ---------------------------------------------------------------- producer
    // lane 0 streams k (and the gates), lane 1 streams v: k runs ahead by its
    // three buffers, v by one
    if (lane == 0 && nch > 0) {
      tma_prefetch(&p.tmK);
      int loaded = 0;
      bool ok = true;
      for (int c = 0; c < nch; ++c) {
        const int kb = c % kKBufs;
        if (c >= kKBufs &&
            !mbar_wait(&bar[kBarKEmpty + kb], ((c - kKBufs) / kKBufs) & 1, abort_flag, p.err, kErrGdn)) {
          ok = false;
          break;
        }
        uint64_t* kf = &bar[kBarKFull + kb];
        mbar_expect_tx(kf, kKV + 512);
        for (int part = 0; part < 2; ++part)
          for (int box = 0; box < 2; ++box)
            tma_load_3d(sb + kOffK + kb * kKV + box * 2 * kBox + part * kBox, &p.tmK, kf, 64 * box,
                        kC * c, 2 * lh + part);
        bulk_load(sb + kOffGateRaw + kb * 512, alpha_g + kC * c, 256, kf);
        bulk_load(sb + kOffGateRaw + kb * 512 + 256, beta_g + kC * c, 256, kf);
        loaded = c + 1;
      }
      if (!ok)  // let the copies already issued land before the CTA exits
        for (int c = loaded - kKBufs < 0 ? 0 : loaded - kKBufs; c < loaded; ++c)
          mbar_drain(&bar[kBarKFull + c % kKBufs], (c / kKBufs) & 1);
    } else if (lane == 1 && nch > 0) {
      tma_prefetch(&p.tmV);
      int loaded = 0;
      bool ok = true;
      for (int c = 0; c < nch; ++c) {
        if (c >= 1 && !mbar_wait(&bar[kBarVEmpty], (c - 1) & 1, abort_flag, p.err, kErrGdn)) {
          ok = false;
          break;
        }
        uint64_t* vf = &bar[kBarVFull];
        mbar_expect_tx(vf, kKV);
        for (int part = 0; part < 2; ++part)
          for (int box = 0; box < 2; ++box)
            tma_load_3d(sb + kOffV + box * 2 * kBox + part * kBox, &p.tmV, vf, 64 * box, kC * c,
                        2 * lh + part);
        loaded = c + 1;
      }
      if (!ok && loaded > 0) mbar_drain(&bar[kBarVFull], (loaded - 1) & 1);
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && nch > 0) {
      const uint32_t id_p = idesc_bf16_f32(128, 64);
      const uint32_t id_uw = idesc_bf16_f32(128, 64) | (1u << 15);
      const uint32_t id_u2 = idesc_bf16_f32(128, 128) | (1u << 15);
      const uint32_t id_da = idesc_bf16_f32(128, 64) | (1u << 16);
      const uint32_t id_da2 = idesc_bf16_f32(128, 128) | (1u << 16);
      const uint32_t id_db = idesc_bf16_f32(128, 128) | (1u << 16);
      // descriptors of shared-memory offset 0; an operand at byte offset `o` adds o >> 4
      const uint64_t dk = sdesc_kmajor_sw128(sb);
      const uint64_t dm = sdesc_mnmajor_sw128(sb, 2 * kBox);  // 64-column blocks 16 KB apart
      int p_next = 0;  // next chunk whose P = K K^T is still to be issued
      // P = K K^T with A = [K_hi; K_lo] (128 K-major rows: a box of high parts and
      // the box of remainders after it) and B = K_hi, then K_lo: rows 0-63 of the
      // result hold K_hi K^T, rows 64-127 K_lo K^T; their sum is P.
      auto issue_p = [&](int c) {
        issue_p_mmas(tb + kColP, dk + ((kOffK + (c % kKBufs) * kKV) >> 4), id_p);
        mma_commit(&bar[kBarP]);
      };
      // P of the next chunk needs only its keys and the P columns (free once the
      // previous P has been read out); it is issued while waiting for anything else.
      auto try_p = [&]() {
        if (p_next < nch && (p_next == 0 || mbar_poll(&bar[kBarPfree], (p_next - 1) & 1)) &&
            mbar_poll(&bar[kBarKFull + p_next % kKBufs], (p_next / kKBufs) & 1)) {
          tc_fence_after();
          issue_p(p_next);
          ++p_next;
        }
      };
      auto wait = [&](int b, uint32_t parity) -> bool {
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
          if (mbar_test_for(&bar[b], parity, 200)) break;
          try_p();
          if (*abort_flag) return false;
          if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort_flag = 1;
            atomicCAS(p.err, 0, kErrGdn);
            return false;
          }
        }
        tc_fence_after();
        return true;
      };
      // U^T = V^T (T diag(b))^T into two 64-column parts (V_hi [T_hi | T_lo]^T as one
      // N = 128 product, plus V_lo T_hi^T on the first part) and
      // W^T = K^T (T diag(b g))^T (three split terms)
      auto issue_uw = [&](int c) {
        const uint64_t vd = dm + (kOffV >> 4);
        const uint64_t kd = dm + ((kOffK + (c % kKBufs) * kKV) >> 4);
        const uint64_t tu = dk + ((kOffT + 2 * kBox) >> 4), tw = dk + (kOffT >> 4);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tb + kColN, vd + ((2048 * ks) >> 4), tu + ((32 * ks) >> 4), id_u2, ks != 0 ? 1u : 0u);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tb + kColN, vd + (kBox >> 4) + ((2048 * ks) >> 4), tu + ((32 * ks) >> 4), id_uw, 1u);
#pragma unroll
        for (int g = 0; g < 3; ++g) {
          const uint64_t ad = kd + (g == 2 ? kBox >> 4 : 0);
          const uint64_t bd = tw + (g == 1 ? kBox >> 4 : 0);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tb + kColW, ad + ((2048 * ks) >> 4), bd + ((32 * ks) >> 4), id_uw,
                     (g | ks) != 0 ? 1u : 0u);
        }
        mma_commit(&bar[kBarUW]);
        mma_commit(&bar[kBarVEmpty]);
      };
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        if (!wait(kBarTops, c & 1) || !wait(kBarVFull, c & 1)) break;
        issue_uw(c);
        if (!wait(kBarWop, c & 1) || !wait(kBarSops, c & 1)) break;
        {  // NEW^T += S_0 (-W)^T on U^T: S_hi [-W_hi | -W_lo]^T (N = 128) and S_lo (-W_hi)^T
          const uint64_t wd = dm + (kOffW >> 4);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_bf16_tmem_a(tb + kColN, tb + kColSh + 8 * ks, wd + ((2048 * ks) >> 4), id_da2, 1u);
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            mma_bf16_tmem_a(tb + kColN, tb + kColSl + 8 * ks, wd + ((2048 * ks) >> 4), id_da, 1u);
          mma_commit(&bar[kBarDA]);
        }
        if (!wait(kBarNop, c & 1)) break;
        {  // S += NEW'^T K
          const uint64_t kd = dm + ((kOffK + (c % kKBufs) * kKV) >> 4);
#pragma unroll
          for (int g = 0; g < 3; ++g) {
            const uint32_t at = tb + (g == 2 ? kColNl : kColNh);
            const uint64_t bd = kd + (g == 1 ? kBox >> 4 : 0);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16_tmem_a(tb + kColS, at + 8 * ks, bd + ((2048 * ks) >> 4), id_db, 1u);
          }
          mma_commit(&bar[kBarDB]);
          mma_commit(&bar[kBarKEmpty + c % kKBufs]);
        }
      }
      // every MMA issued has finished before TMEM is released
      mma_commit(&bar[kBarFinal]);
      mbar_drain(&bar[kBarFinal], 0);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- chunk-local work
    const int pt = tid - 128;  // 0..127, TMEM lane of this thread
    const int q = warp - 4;
    const uint32_t lrow = tb + (static_cast<uint32_t>(32 * q) << 16);
    // Software pipeline over chunks: the front of chunk c + 1 (gates, B, the
    // diagonal blocks of T) runs while the products U^T, W^T of chunk c are on
    // the tensor cores; the rest of T needs the T-operand tiles they read.
    auto gates = [&](int c, float* gs) {
      const float* ga = reinterpret_cast<const float*>(sm + kOffGateRaw + (c % kKBufs) * 512);
      const float* gbeta = ga + 64;
      const int n = min(kC, p.rows - kC * c);
      float la[2], be[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int t = 2 * lane + e;
        la[e] = t < n ? fmaxf(log2f(ga[t]), kMinLog2Gate) : 0.f;
        be[e] = t < n ? gbeta[t] : 0.f;
      }
      const float pair = la[0] + la[1];
      float incl = pair;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const float g0 = incl - la[1], g1 = incl;
      const float gC = __shfl_sync(0xffffffffu, incl, 31);
      gs[2 * lane] = be[0];
      gs[2 * lane + 1] = be[1];
      gs[64 + 2 * lane] = be[0] * exp2f(g0);
      gs[64 + 2 * lane + 1] = be[1] * exp2f(g1);
      gs[128 + 2 * lane] = exp2f(gC - g0);
      gs[128 + 2 * lane + 1] = exp2f(gC - g1);
      gs[192 + 2 * lane] = g0;
      gs[192 + 2 * lane + 1] = g1;
    };
    // gates, B and the diagonal blocks of T for chunk c
    auto front = [&](int c) -> bool {
      bool ok = mbar_wait(&bar[kBarKFull + c % kKBufs], (c / kKBufs) & 1, abort_flag, p.err, kErrGdn);
      if (!named_bar_all(kPreBar, 128, ok)) return false;
      float* gs = reinterpret_cast<float*>(sm + kOffGate + (c % 3) * 1024);  // beta, bg, dec, G2
      if (c == 0 && q == 0) gates(0, gs);  // later chunks: computed during the previous chunk
      ok = mbar_wait(&bar[kBarP], c & 1, abort_flag, p.err, kErrGdn);
      if (!named_bar_all(kPreBar, 128, ok)) return false;
      tc_fence_after();
      // B_ts = b_t 2^{G2_t - G2_s} P_ts below the diagonal.  Lane t < 64 holds
      // (K_hi K^T)[t], lane 64 + t (K_lo K^T)[t]: warps 4-5 finish columns 0-31 and
      // warps 6-7 columns 32-63, each first leaving the other half in B's row.
      {
        const int t = pt & 63;
        const bool lowq = q < 2;
        const int own = lowq ? 0 : 32;  // columns this thread finishes
        uint32_t r[2][32];
        tmem_ld32(lrow + kColP, r[0]);
        tmem_ld32(lrow + kColP + 32, r[1]);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kBarPfree]);
        uint32_t keep[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) keep[j] = lowq ? r[0][j] : r[1][j];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = __uint_as_float(lowq ? r[1][j + e] : r[0][j + e]);
          st4(Bs + t * kLd + (32 - own) + j, make_float4(v[0], v[1], v[2], v[3]));
        }
        named_bar_sync(kPreBar, 128);
        const float gt = gs[192 + t], bt = gs[t];
#pragma unroll
        for (int j = 0; j < 32; j += 4) {
          const int s0 = own + j;
          const float4 other = ld4(Bs + t * kLd + s0);
          const float4 gsv = ld4(gs + 192 + s0);
          const float ov[4] = {other.x, other.y, other.z, other.w};
          const float g4[4] = {gsv.x, gsv.y, gsv.z, gsv.w};
          float v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float pts = __uint_as_float(keep[j + e]) + ov[e];
            v[e] = s0 + e < t ? bt * ex2(gt - g4[e]) * pts : 0.f;
          }
          st4(Bs + t * kLd + s0, make_float4(v[0], v[1], v[2], v[3]));
        }
      }
      named_bar_sync(kPreBar, 128);
      // T = (I + B)^-1, unit lower triangular: the 16 x 16 diagonal blocks by substitution
      if (pt < 64) {
        const int b = pt >> 4, s = pt & 15, o = 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float brow[16];
#pragma unroll
          for (int k4 = 0; k4 < 16; k4 += 4) {
            const float4 v = ld4(Bs + (o + r) * kLd + o + k4);
            brow[k4] = v.x; brow[k4 + 1] = v.y; brow[k4 + 2] = v.z; brow[k4 + 3] = v.w;
          }
          float acc = r == s ? 1.f : 0.f;
#pragma unroll
          for (int k = 0; k < r; ++k) acc = fmaf(-brow[k], x[k], acc);
          x[r] = acc;
        }
        named_bar_sync(kPreBar + 1, 64);  // all columns are computed before B_bb is overwritten
#pragma unroll
        for (int r = 0; r < 16; ++r) Bs[(o + r) * kLd + o + s] = x[r];
      }
      named_bar_sync(kPreBar, 128);
      return true;
    };
    // the rest of T, then T diag(b g) and T diag(b) as bf16 hi/lo K-major tiles [t][s]
    auto back = [&](int c) -> bool {
      const float* gs = reinterpret_cast<const float*>(sm + kOffGate + (c % 3) * 1024);
      if (c > 0) {  // the T-operand area (scratch X here) is free once U^T, W^T of c - 1 are done
        const bool ok = mbar_wait(&bar[kBarUW], (c - 1) & 1, abort_flag, p.err, kErrGdn);
        if (!named_bar_all(kPreBar, 128, ok)) return false;
      }
      // warp 6, idle in the first block step below, prepares the next chunk's gates
      // (read again only after the next chunk's keys are waited for by every warp)
      if (q == 2 && c + 1 < nch &&
          mbar_wait(&bar[kBarKFull + (c + 1) % kKBufs], ((c + 1) / kKBufs) & 1, abort_flag, p.err,
                    kErrGdn))
        gates(c + 1, reinterpret_cast<float*>(sm + kOffGate + ((c + 1) % 3) * 1024));
      {
        // 32 x 32 halves: T_10 = -T_11 B_10 T_00 and T_32 = -T_33 B_32 T_22
        const int r = (pt & 31) >> 2, cg = pt & 3;
        const int a = pt < 32 ? 1 : 3, b = a - 1;
        float4 y0, y1;
        if (pt < 64) {
          tile_product<1>(Bs + (16 * a) * kLd + 16 * b, Bs + (16 * b) * kLd + 16 * b, r, cg, y0, y1);
          st4(Xs + (16 * a + r) * kLd + 16 * b + 4 * cg, y0);
          st4(Xs + (16 * a + r + 8) * kLd + 16 * b + 4 * cg, y1);
        }
        named_bar_sync(kPreBar, 128);
        if (pt < 64) {
          tile_product<1>(Bs + (16 * a) * kLd + 16 * a, Xs + (16 * a) * kLd + 16 * b, r, cg, y0, y1);
          st4(Bs + (16 * a + r) * kLd + 16 * b + 4 * cg, make_float4(-y0.x, -y0.y, -y0.z, -y0.w));
          st4(Bs + (16 * a + r + 8) * kLd + 16 * b + 4 * cg, make_float4(-y1.x, -y1.y, -y1.z, -y1.w));
        }
        named_bar_sync(kPreBar, 128);
        // the 64 x 64 whole: T[32:64, 0:32] = -T[32:64, 32:64] B[32:64, 0:32] T[0:32, 0:32]
        const int blk = pt >> 5, a2 = 2 + (blk >> 1), b2 = blk & 1;
        tile_product<2>(Bs + (16 * a2) * kLd, Bs + 16 * b2, r, cg, y0, y1);
        st4(Xs + (16 * a2 + r) * kLd + 16 * b2 + 4 * cg, y0);
        st4(Xs + (16 * a2 + r + 8) * kLd + 16 * b2 + 4 * cg, y1);
        named_bar_sync(kPreBar, 128);
        tile_product<2>(Bs + (16 * a2) * kLd + 32, Xs + 32 * kLd + 16 * b2, r, cg, y0, y1);
        st4(Bs + (16 * a2 + r) * kLd + 16 * b2 + 4 * cg, make_float4(-y0.x, -y0.y, -y0.z, -y0.w));
        st4(Bs + (16 * a2 + r + 8) * kLd + 16 * b2 + 4 * cg, make_float4(-y1.x, -y1.y, -y1.z, -y1.w));
        named_bar_sync(kPreBar, 128);
      }
#pragma unroll 1
      for (int m = 0; m < 4; ++m) {
        const int idx = pt + 128 * m;
        const int t = idx >> 3, ch = idx & 7;
        float w[8], u[8];
        {
          const float4 t0 = ld4(Bs + t * kLd + 8 * ch), t1 = ld4(Bs + t * kLd + 8 * ch + 4);
          const float4 w0 = ld4(gs + 64 + 8 * ch), w1 = ld4(gs + 64 + 8 * ch + 4);
          const float4 u0 = ld4(gs + 8 * ch), u1 = ld4(gs + 8 * ch + 4);
          const float tv[8] = {t0.x, t0.y, t0.z, t0.w, t1.x, t1.y, t1.z, t1.w};
          const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float v = 8 * ch + e <= t ? tv[e] : 0.f;
            w[e] = v * wv[e];
            u[e] = v * uv[e];
          }
        }
        uint4 hi, lo;
        const uint32_t off = swz(t, ch);
        split8(w, hi, lo);
        *reinterpret_cast<uint4*>(sm + kOffT + off) = hi;
        *reinterpret_cast<uint4*>(sm + kOffT + kBox + off) = lo;
        split8(u, hi, lo);
        *reinterpret_cast<uint4*>(sm + kOffT + 2 * kBox + off) = hi;
        *reinterpret_cast<uint4*>(sm + kOffT + 3 * kBox + off) = lo;
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarTops]);
      return true;
    };
    if (nch > 0 && front(0)) {
      for (int c = 0; c < nch; ++c) {
        if (!back(c)) break;
        if (c + 1 < nch && !front(c + 1)) break;
      }
    }
  } else {
    // ---------------------------------------------------------------- serial part
    const int i = tid;  // state row = TMEM lane
    const uint32_t lrow = tb + (static_cast<uint32_t>(32 * warp) << 16);
    const float* src = s_in != nullptr ? s_in + static_cast<size_t>(i) * kDk : nullptr;
    float* dst = s_out + static_cast<size_t>(i) * kDk;
    // 64 columns of S: the bf16 split (operand of the next chunk) and S times the
    // next chunk's total decay g (the accumulator the next update adds to)
    auto put_state = [&](uint32_t (&r)[2][32], int half, float g) {
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int m = 0; m < 16; ++m)
          split2(__uint_as_float(r[cc][2 * m]), __uint_as_float(r[cc][2 * m + 1]), hi[m], lo[m]);
        tmem_st16(lrow + kColSh + 32 * half + 16 * cc, hi);
        tmem_st16(lrow + kColSl + 32 * half + 16 * cc, lo);
#pragma unroll
        for (int j = 0; j < 32; ++j) r[cc][j] = __float_as_uint(g * __uint_as_float(r[cc][j]));
        tmem_st32(lrow + kColS + 64 * half + 32 * cc, r[cc]);
      }
    };
    bool ok = true;
    if (nch == 0) {
      for (int j = 0; j < kDk; j += 4)
        *reinterpret_cast<float4*>(dst + j) =
            src != nullptr ? *reinterpret_cast<const float4*>(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      ok = mbar_wait(&bar[kBarKFull], 0, abort_flag, p.err, kErrGdn);
      if (ok) {
        const float* ga = reinterpret_cast<const float*>(sm + kOffGateRaw);
        const float g = exp2f(chunk_log2_decay(ga, min(kC, p.rows), lane));
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t r[2][32];
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const float4 x = src != nullptr ? *reinterpret_cast<const float4*>(src + 64 * half + j)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
            r[j >> 5][j & 31] = __float_as_uint(x.x);
            r[j >> 5][(j & 31) + 1] = __float_as_uint(x.y);
            r[j >> 5][(j & 31) + 2] = __float_as_uint(x.z);
            r[j >> 5][(j & 31) + 3] = __float_as_uint(x.w);
          }
          put_state(r, half, g);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kBarSops]);
      }
    }
    for (int c = 0; c < nch && ok; ++c) {
      {  // -W as the MN-major B operand of NEW^T: row j holds W^T[j][0..63]
        if (!mbar_wait(&bar[kBarUW], c & 1, abort_flag, p.err, kErrGdn)) break;
        tc_fence_after();
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          uint32_t r[32];
          tmem_ld32(lrow + kColW + 32 * h, r);
          tmem_wait_ld();
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = -__uint_as_float(r[8 * c4 + e]);
            uint4 hi, lo;
            split8(x, hi, lo);
            const uint32_t off = swz(i, 4 * h + c4);
            *reinterpret_cast<uint4*>(sm + kOffW + off) = hi;
            *reinterpret_cast<uint4*>(sm + kOffW + 2 * kBox + off) = lo;
          }
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kBarWop]);
      }
      if (!mbar_wait(&bar[kBarDA], c & 1, abort_flag, p.err, kErrGdn)) break;
      tc_fence_after();
      {  // NEW'^T[i][t] = NEW^T[i][t] 2^{G2_C - G2_t}
        const float* dec = reinterpret_cast<const float*>(sm + kOffGate + (c % 3) * 1024) + 128;
        // t in [32 half, 32 half + 32): both parts are read before the split of the
        // same t range overwrites them
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t r0[32], r1[32];
          tmem_ld32(lrow + kColN + 32 * half, r0);
          tmem_ld32(lrow + kColN + 64 + 32 * half, r1);
          tmem_wait_ld();
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const int t = 32 * half + 2 * m;
            const float y0 = (__uint_as_float(r0[2 * m]) + __uint_as_float(r1[2 * m])) * dec[t];
            const float y1 = (__uint_as_float(r0[2 * m + 1]) + __uint_as_float(r1[2 * m + 1])) * dec[t + 1];
            split2(y0, y1, hi[m], lo[m]);
          }
          tmem_st16(lrow + kColNh + 16 * half, hi);
          tmem_st16(lrow + kColNl + 16 * half, lo);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarNop]);
      // the next chunk's total decay, while the update runs
      float g = 1.f;
      if (c + 1 < nch) {
        const int kn = (c + 1) % kKBufs;
        if (!mbar_wait(&bar[kBarKFull + kn], ((c + 1) / kKBufs) & 1, abort_flag, p.err, kErrGdn)) break;
        const float* ga = reinterpret_cast<const float*>(sm + kOffGateRaw + kn * 512);
        g = exp2f(chunk_log2_decay(ga, min(kC, p.rows - kC * (c + 1)), lane));
      }
      if (!mbar_wait(&bar[kBarDB], c & 1, abort_flag, p.err, kErrGdn)) break;
      tc_fence_after();
      if (c + 1 == nch) {
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t r[2][32];
          tmem_ld32(lrow + kColS + 64 * half, r[0]);
          tmem_ld32(lrow + kColS + 64 * half + 32, r[1]);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 64; j += 4)
            *reinterpret_cast<float4*>(dst + 64 * half + j) =
                make_float4(__uint_as_float(r[j >> 5][j & 31]), __uint_as_float(r[j >> 5][(j & 31) + 1]),
                            __uint_as_float(r[j >> 5][(j & 31) + 2]),
                            __uint_as_float(r[j >> 5][(j & 31) + 3]));
        }
      } else {
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          uint32_t r[2][32];
          tmem_ld32(lrow + kColS + 64 * half, r[0]);
          tmem_ld32(lrow + kColS + 64 * half + 32, r[1]);
          tmem_wait_ld();
          put_state(r, half, g);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kBarSops]);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

// ---------------------------------------------------------------- exact rows and rho
// Exact prefix rows (section 2.4): row exact_idx[e] takes its true input X_exact[l, e]
// in place of the map's prediction: bf16(g x) into X_hat and its sum of squares as the
// row's first partial (the others zero), after the map GEMM of the row's chunk.
__global__ void exact_input_kernel(const __nv_bfloat16* X, const __nv_bfloat16* g,
                                   const int32_t* idx, int64_t n_exact, int L, int d,
                                   int64_t start, int64_t rc, int64_t rows, int64_t R,
                                   int ss_tiles, __nv_bfloat16* xhat, float* ss, int* err) {
  const int64_t w = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= static_cast<int64_t>(L) * n_exact) return;
  const int l = static_cast<int>(w / n_exact);
  const int64_t e = w % n_exact;
  const int64_t t = idx[e];
  if (t < 0 || t >= rows) {
    if (lane == 0) atomicCAS(err, 0, kErrIndex);
    return;
  }
  if (t < start || t >= start + rc) return;
  const int64_t r = t - start;
  const __nv_bfloat16* src = X + (static_cast<size_t>(l) * n_exact + e) * d;
  __nv_bfloat16* dst = xhat + (static_cast<size_t>(l) * R + r) * d;
  const __nv_bfloat16* gl = g != nullptr ? g + static_cast<size_t>(l) * d : nullptr;
  float acc = 0.f;
  for (int j = 8 * lane; j < d; j += 256) {
    const uint4 xv = *reinterpret_cast<const uint4*>(src + j);
    uint4 gv = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);  // bf16 1.0 pairs
    if (gl != nullptr) gv = *reinterpret_cast<const uint4*>(gl + j);
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
    uint32_t out[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 x2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xw[q]));
      const float2 g2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gw[q]));
      acc = fmaf(x2.x, x2.x, acc);
      acc = fmaf(x2.y, x2.y, acc);
      out[q] = pack_bf16(x2.x * g2.x, x2.y * g2.y);
    }
    *reinterpret_cast<uint4*>(dst + j) = make_uint4(out[0], out[1], out[2], out[3]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  for (int j = lane; j < ss_tiles; j += 32)
    ss[(static_cast<size_t>(l) * ss_tiles + j) * R + r] = j == 0 ? acc : 0.f;
}

// The filled rows: the rows of [0, rows) not in exact_idx (ascending), in order.
// fill[t - #(exact rows before t)] = t for every filled row t.
__global__ void complement_kernel(const int32_t* exact_idx, int64_t n_exact, int64_t rows,
                                  int32_t* fill) {
  const int64_t n_fill = rows - n_exact;
  for (int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; t < rows;
       t += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    int64_t lo = 0, hi = n_exact;
    while (lo < hi) {
      const int64_t mid = (lo + hi) >> 1;
      if (exact_idx[mid] < t) lo = mid + 1;
      else hi = mid;
    }
    const bool exact = lo < n_exact && exact_idx[lo] == t;
    const int64_t k = t - lo;
    if (!exact && k >= 0 && k < n_fill) fill[k] = static_cast<int32_t>(t);
  }
}

// rho of section 2.3 (terminal-state correction), one CTA per (layer, head) and
// row chunk.  A row's weight in the state at the end of the rows is the product
// of the gates after it.  Each thread runs over a segment of rows with
//   den <- den * alpha_t + 1,  num <- num * alpha_t + [row t filled],  P <- P * alpha_t
// (weights relative to the segment's end), the segments combine in row order
// ((n, d, P)_a then (n, d, P)_b gives (n_a P_b + n_b, d_a P_b + d_b, P_a P_b)), and
// the chunk's result extends the sums carried from earlier chunks.  f64 throughout.
constexpr int kRhoThreads = 1024;

__global__ void __launch_bounds__(kRhoThreads) rho_chunk_kernel(
    const float* gate, int H, int64_t R, int64_t rc, int64_t start, const int32_t* exact_idx,
    int64_t n_exact, double* acc, int first) {
  __shared__ double s_n[kRhoThreads], s_d[kRhoThreads], s_p[kRhoThreads];
  const int lh = blockIdx.x;
  const int l = lh / H, h = lh - l * H;
  const float* alpha = gate + (static_cast<size_t>(l) * 2 * H + h) * R;  // alpha plane of (l, h)
  const int64_t seg = (rc + kRhoThreads - 1) / kRhoThreads;
  const int64_t a = threadIdx.x * seg;
  const int64_t b = a + seg < rc ? a + seg : rc;
  // first exact row at or after prompt row start + a (exact_idx ascending)
  int64_t lo = 0, hi = n_exact;
  while (lo < hi) {
    const int64_t mid = (lo + hi) >> 1;
    if (exact_idx[mid] < start + a) lo = mid + 1;
    else hi = mid;
  }
  double num = 0.0, den = 0.0, P = 1.0;
  for (int64_t t = a; t < b; ++t) {
    const double al = alpha[t];
    bool exact = false;
    if (lo < n_exact && exact_idx[lo] == start + t) {
      exact = true;
      ++lo;
    }
    den = fma(den, al, 1.0);
    num = fma(num, al, exact ? 0.0 : 1.0);
    P *= al;
  }
  s_n[threadIdx.x] = num;
  s_d[threadIdx.x] = den;
  s_p[threadIdx.x] = P;
  __syncthreads();
  for (int stride = 1; stride < kRhoThreads; stride <<= 1) {
    const int i = static_cast<int>(threadIdx.x);
    if ((i & (2 * stride - 1)) == 0) {
      const int j = i + stride;  // the later segment
      s_n[i] = fma(s_n[i], s_p[j], s_n[j]);
      s_d[i] = fma(s_d[i], s_p[j], s_d[j]);
      s_p[i] *= s_p[j];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    double* c = acc + 2 * static_cast<size_t>(lh);
    if (first) {
      c[0] = s_n[0];
      c[1] = s_d[0];
    } else {
      c[0] = fma(c[0], s_p[0], s_n[0]);
      c[1] = fma(c[1], s_p[0], s_d[0]);
    }
  }
}

// rho = filled / all weight (0 with no rows), written to `rho` if set; with
// delta_M set, the terminal-state correction S += rho * delta_M of the (layer, head).
__global__ void __launch_bounds__(256) rho_finish_kernel(const double* acc, int empty, float* rho,
                                                         const float* delta_M, float* S, int dvdk) {
  const size_t lh = blockIdx.x;
  const double d = acc != nullptr ? acc[2 * lh + 1] : 0.0;
  const float r = (empty || !(d > 0.0)) ? 0.f : static_cast<float>(acc[2 * lh] / d);
  if (rho != nullptr && threadIdx.x == 0) rho[lh] = r;
  if (delta_M == nullptr) return;
  float* s = S + lh * dvdk;
  const float* m = delta_M + lh * dvdk;
  for (int i = threadIdx.x; i < dvdk; i += blockDim.x) s[i] = fmaf(r, m[i], s[i]);
}

struct GdnPlan {
  int bn_map = 0;
  int64_t R = 0;
  size_t off_xhat = 0, off_ss = 0, off_k = 0, off_v = 0, off_gate = 0, off_slots = 0, off_rho = 0,
         off_fill = 0, off_hc = 0, off_hdev = 0, off_hflags = 0, off_dq = 0, total = 0;
  int dq_layers = 0;     // resident int8 maps: layers dequantised ahead of the bf16 GEMM
  bool compact = false;  // map only the filled rows (exact rows, one row chunk, bf16 GEMM)
  Layout lay;
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
  if (a->A_scale != nullptr && a->d_in % kQ8Group != 0)
    return fail(RF_ERR_SHAPE, "int8 maps need d_in to be a multiple of 128");
  if (a->n_exact < 0 || a->n_exact > a->rows) return fail(RF_ERR_ARG, "n_exact must be in [0, rows]");
  if (a->n_exact > 0 && (a->exact_idx == nullptr || a->X_exact == nullptr))
    return fail(RF_ERR_ARG, "n_exact > 0 needs exact_idx and X_exact");
  if (a->h_on_host != 0 && a->h_on_host != 1) return fail(RF_ERR_ARG, "h_on_host must be 0 or 1");
  if (a->q8_group_layers < -1) return fail(RF_ERR_ARG, "q8_group_layers must be >= -1");
  return RF_OK;
}

void plan_gdn(const rf_gdn_args* a, GdnPlan* pl) {
  pl->bn_map = (a->d_out % 256 == 0) ? 256 : 128;
  const int64_t all = ceil_div(a->rows > 0 ? a->rows : 1, kBM) * kBM;
  pl->R = a->rows_per_chunk > 0 ? (a->rows_per_chunk < all ? a->rows_per_chunk : all) : all;
  const size_t L = a->n_layers, d = a->d_out, R = pl->R, H = a->n_heads;
  Layout& lay = pl->lay;
  pl->off_xhat = lay.take(L * R * d * 2);
  pl->off_ss = lay.take(L * (d / pl->bn_map) * R * 4);
  pl->off_k = lay.take(L * H * R * kDk * 4);
  pl->off_v = lay.take(L * H * R * kDk * 4);
  pl->off_gate = lay.take(L * 2 * H * R * 4);
  pl->off_slots = lay.take(a->maps_on_host ? kMapSlots * map_slot_bytes(a->d_out, a->d_in, a->A_scale != nullptr) : 0);
  pl->off_rho = lay.take(L * H * 2 * sizeof(double));
  if (a->h_on_host) {
    size_t fo = 0;
    pl->off_hdev = lay.take(host_rows_bytes(a->rows, a->d_in, &fo));
    pl->off_hflags = pl->off_hdev + fo;
  }
  pl->dq_layers = q8_group(a->q8_group_layers, a->A_scale != nullptr, a->maps_on_host != 0,
                           a->n_layers);
  if (pl->dq_layers > 0)
    pl->off_dq = lay.take(static_cast<size_t>(pl->dq_layers) * a->d_out * a->d_in * 2);
  // the compacted map GEMM writes rows by index: the bf16 GEMM only (not the in-GEMM int8
  // conversion)
  pl->compact = a->n_exact > 0 && pl->R >= a->rows && (a->A_scale == nullptr || pl->dq_layers > 0);
  if (pl->compact) {
    const size_t n_fill = static_cast<size_t>(a->rows - a->n_exact);
    pl->off_fill = lay.take(static_cast<size_t>(a->rows) * 4);
    pl->off_hc = lay.take(n_fill * a->d_in * 2);
  }
  pl->total = lay.off;
}

// The projection GEMM of layers [l0, l0 + nl) of the chunk (all of them by default).
rf_status launch_gdn_proj(const rf_gdn_args* a, const GdnPlan& pl, int64_t rc, const void* xhat,
                          const float* ss, __nv_bfloat16* kb, __nv_bfloat16* vb, float* gb,
                          cudaStream_t s, int l0 = 0, int nl = -1, int max_pairs = 0,
                          int* ctr = nullptr) {
  GemmParams p{};
  p.mode = kModeGdnProj;
  p.k_blocks = a->d_out / kBK;
  const int H = a->n_heads;
  const uint64_t drow = static_cast<uint64_t>(a->d_out) * 2;
  const uint64_t hk = static_cast<uint64_t>(H) * kDk;
  // stages of two k-blocks: each operand staged by one copy through a rank-4 view
  // {64 k, rows, k-blocks, layers} whose third dimension steps 128 bytes.  B boxes of half
  // a tile's columns: each CTA of a pair stages one half (the gate tile's halves are the H
  // rows of w_a and of w_b)
  const uint64_t kblocks = static_cast<uint64_t>(a->d_out / kBK);
  const uint64_t L = static_cast<uint64_t>(a->n_layers);
  auto view = [&](CUtensorMap* tm, const void* base, uint64_t rows, uint64_t layer_stride,
                  uint32_t box_rows) {
    const uint64_t dims[4] = {kBK, rows, kblocks, L};
    const uint64_t strides[3] = {drow, 128, layer_stride};
    const uint32_t box[4] = {kBK, box_rows, 2, 1};
    return make_tmap_4d(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, dims, strides, box,
                        CU_TENSOR_MAP_SWIZZLE_128B);
  };
  bool ok = view(&p.tmA, xhat, static_cast<uint64_t>(rc), drow * pl.R, kBM);
  ok = ok && view(&p.tmB[0], a->Wk, hk, drow * hk, 128);
  ok = ok && view(&p.tmB[1], a->Wv, hk, drow * hk, 128);
  ok = ok && view(&p.tmB[2], a->Wa, H, drow * H, static_cast<uint32_t>(H));
  ok = ok && view(&p.tmB[3], a->Wb, H, drow * H, static_cast<uint32_t>(H));
  p.k2 = 1;
  // outputs: k and v planes {d_k, rows, L*H*2} (high part, then remainder, per layer and head)
  const uint64_t prow = static_cast<uint64_t>(kDk) * 2, pplane = prow * pl.R;
  const uint64_t planes = static_cast<uint64_t>(a->n_layers) * H * 2;
  ok = ok && make_tmap_3d(&p.tmO[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kb, kDk, rc, planes, prow,
                          pplane, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_3d(&p.tmO[1], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, vb, kDk, rc, planes, prow,
                          pplane, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the GDN projection GEMM");
  p.m_tiles = static_cast<int32_t>(ceil_div(rc, kBM));
  p.n_k_tiles = H / 2;
  p.n_v_tiles = H / 2;
  p.n_tiles = H + 1;
  p.batches = nl < 0 ? a->n_layers : nl;
  p.batch_base = l0;
  p.bn = 256;
  p.group_m = 2;  // one pair row tile per group: every column tile of a row panel in turn
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
  p.lim_a = static_cast<int64_t>(a->n_layers) * 2 * H * pl.R;
  p.l2_eps = static_cast<float>(a->l2_eps);
  p.err = device_error_word();
  if (p.err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  const int64_t tiles = static_cast<int64_t>((p.m_tiles + 1) / 2) * p.n_tiles * p.batches;
  int pairs = static_cast<int>(tiles < sm_count() / 2 ? tiles : sm_count() / 2);
  if (max_pairs > 0 && pairs > max_pairs) pairs = max_pairs;
  if (pairs <= 0) return RF_OK;
  cudaError_t e = launch_gemm2(p, pairs, s, ctr);
  if (e != cudaSuccess) return cuda_fail(e, "GDN projection GEMM launch");
  return RF_OK;
}


}  // namespace

cudaError_t launch_gdn_state(const GdnStateParams& p, cudaStream_t stream) {
  // set on every launch: the attribute belongs to the current device, and the call is
  // cheap next to the kernel
  cudaError_t e = cudaFuncSetAttribute(gdn_state_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kStateSmem);
  if (e != cudaSuccess) return e;
  dim3 grid(p.heads, p.layers);
  gdn_state_kernel<<<grid, kStateThreads, kStateSmem, stream>>>(p);
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
  if (a->A_scale != nullptr && !aligned16(a->A_scale))
    return fail(RF_ERR_ALIGN, "A_scale is not 16-byte aligned");
  const void* dev2[] = {a->X_exact, a->rho, a->delta_M};
  for (const void* q : dev2)
    if (q != nullptr && !aligned16(q)) return fail(RF_ERR_ALIGN, "a device pointer is not 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(a->exact_idx) & 3u) != 0)
    return fail(RF_ERR_ALIGN, "exact_idx is not 4-byte aligned");
  if (a->h_on_host && a->rows > 0 && (st = check_pinned(a->H, "H")) != RF_OK) return st;
  if (a->maps_on_host && a->rows > 0) {
    if ((st = check_pinned(a->A, "A")) != RF_OK) return st;
    if (a->A_scale != nullptr && (st = check_pinned(a->A_scale, "A_scale")) != RF_OK) return st;
  }
  GdnPlan pl;
  plan_gdn(a, &pl);
  if (workspace == nullptr || ws_bytes < pl.total)
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes", pl.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* xhat = ws + pl.off_xhat;
  float* ss = reinterpret_cast<float*>(ws + pl.off_ss);
  __nv_bfloat16* kb = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_k);
  __nv_bfloat16* vb = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_v);
  float* gb = reinterpret_cast<float*>(ws + pl.off_gate);
  if ((st = guards_fill(ws, pl.lay, s)) != RF_OK) return st;

  GdnStateParams sp{};
  sp.gate = gb;
  sp.S0 = a->S0;
  sp.S = a->S;
  sp.layers = a->n_layers;
  sp.heads = a->n_heads;
  sp.rows_alloc = static_cast<int32_t>(pl.R);
  sp.err = device_error_word();
  if (sp.err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  // k and v of one launch as {d_k, rows, L*H*2} (hi/lo planes of each layer and head)
  auto state_maps = [&](int64_t rc) -> bool {
    const uint64_t row_b = static_cast<uint64_t>(kDk) * 2;
    const uint64_t plane_b = row_b * pl.R;
    const uint64_t planes = static_cast<uint64_t>(a->n_layers) * a->n_heads * 2;
    return make_tmap_3d(&sp.tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, kb, kDk, rc, planes, row_b,
                        plane_b, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B) &&
           make_tmap_3d(&sp.tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, vb, kDk, rc, planes, row_b,
                        plane_b, 64, kC, CU_TENSOR_MAP_SWIZZLE_128B);
  };

  const int LH = a->n_layers * a->n_heads;
  const bool want_rho = a->rho != nullptr || a->delta_M != nullptr;
  double* rho_acc = reinterpret_cast<double*>(ws + pl.off_rho);
  if (a->rows == 0) {  // the end-of-fill state is the initial state; no filled rows: rho = 0
    sp.rows = 0;
    sp.first = 1;
    cudaError_t e = launch_gdn_state(sp, s);
    if (e != cudaSuccess) return cuda_fail(e, "GDN state launch");
    if (a->rho != nullptr) {
      rho_finish_kernel<<<LH, 256, 0, s>>>(nullptr, 1, a->rho, nullptr, a->S, kDk * kDk);
      if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "rho launch");
    }
    return guards_check(ws, pl.lay, s);
  }

  // With all rows in one chunk and more (layer, head) states than SMs, the states of the
  // first `la` layers run as soon as their projections are done, beside the projection GEMM
  // of the other layers: a first launch of it on the side stream holds only the SMs the
  // states leave, and a second one after the states, on the same tile counter, takes over
  // the freed SMs and shares the remaining tiles with it.  The last `L - la` layers' states
  // then fill one wave of the SMs.  Without the split the states of all layers run in two
  // waves, the second one on part of the GPU.
  int la = 0;
  {
    const int per_wave = sm_count() / a->n_heads;  // layers whose states fill one wave
    if (pl.R >= a->rows && per_wave > 0 && a->n_layers > per_wave) la = a->n_layers - per_wave;
  }
  HostStreamer* hs = nullptr;
  std::unique_lock<std::mutex> lk(host_stream_mutex(), std::defer_lock);
  const size_t slot_bytes = map_slot_bytes(a->d_out, a->d_in, a->A_scale != nullptr);
  if (a->maps_on_host || a->h_on_host || la > 0) {
    lk.lock();
    hs = host_streamer();
    if (hs == nullptr) return RF_ERR_CUDA;
  }
  // split state in host memory: streamed in row groups, overlapped with the map GEMM (with
  // exact rows compacted, the gather waits for the whole copy)
  const uint8_t* h_base = static_cast<const uint8_t*>(a->H);
  HostRows hr;
  if (a->h_on_host) {
    if ((st = stream_host_rows(hs, a->H, a->rows, a->d_in, ws + pl.off_hdev,
                               reinterpret_cast<uint32_t*>(ws + pl.off_hflags), s, &hr)) != RF_OK)
      return st;
    h_base = hr.base;
    if (pl.compact && hr.overlap) {
      cudaError_t e = cudaStreamWaitEvent(s, hs->h_done, 0);
      if (e != cudaSuccess) return cuda_fail(e, "ordering after the split-state copy");
    }
  }
  if (a->maps_on_host) {
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
    m.H = h_base + static_cast<size_t>(start) * a->d_in * 2;
    m.rows = rc;
    if (hr.overlap && !pl.compact) {
      m.h_ready = hr.flags;
      m.h_gen = hr.gen;
      m.h_row_base = start;
    }
    if (pl.compact) {  // map only the filled rows; their X_hat rows land at their positions
      int32_t* fill = reinterpret_cast<int32_t*>(ws + pl.off_fill);
      const int64_t blocks = (a->rows + 255) / 256 < 4 * sm_count() ? (a->rows + 255) / 256 : 4 * sm_count();
      complement_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a->exact_idx, a->n_exact,
                                                                    a->rows, fill);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "filled-row list launch");
      const int64_t n_fill = a->rows - a->n_exact;
      if ((st = launch_gather_rows(h_base, fill, n_fill, a->rows, a->d_in, ws + pl.off_hc, s)) != RF_OK)
        return st;
      m.H = ws + pl.off_hc;
      m.rows = n_fill;
      m.out_rows = fill;
    }
    m.d_in = a->d_in;
    m.d_out = a->d_out;
    m.n_layers = a->n_layers;
    m.bn = pl.bn_map;
    m.R = pl.R;
    m.bias = a->bias;
    m.gain = a->gain;
    m.xhat = xhat;
    m.ss = ss;
    if (m.rows == 0) {
      // every row of the chunk is exact: no map GEMM
    } else if (!a->maps_on_host && pl.dq_layers > 0) {
      m.A = a->A;
      m.A_scale = a->A_scale;
      if ((st = launch_map_q8_groups(m, pl.dq_layers, ws + pl.off_dq, s)) != RF_OK) return st;
    } else if (!a->maps_on_host) {
      m.A = a->A;
      m.A_scale = a->A_scale;
      m.slot_layer = -1;
      if ((st = launch_map(m, s)) != RF_OK) return st;
    } else {
      for (int l = 0; l < a->n_layers; ++l) {
        const int k = l % kMapSlots;
        uint8_t* slot = ws + pl.off_slots + k * slot_bytes;
        cudaError_t e = cudaSuccess;
        if (start > 0 || l >= kMapSlots) e = cudaStreamWaitEvent(hs->copy, hs->freed[k], 0);
        if (e == cudaSuccess)
          e = copy_map_layer(slot, a->A, a->A_scale, l, a->d_out, a->d_in, hs->copy, &m.A,
                             &m.A_scale);
        if (e == cudaSuccess) e = cudaEventRecord(hs->copied[k], hs->copy);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hs->copied[k], 0);
        if (e != cudaSuccess) return cuda_fail(e, "streaming a map from host memory");
        m.slot_layer = l;
        if ((st = launch_map(m, s)) != RF_OK) return st;
        e = cudaEventRecord(hs->freed[k], s);
        if (e != cudaSuccess) return cuda_fail(e, "recording a map slot release");
      }
    }
    if (a->n_exact > 0) {  // exact rows of this chunk take their true inputs
      const int64_t warps = static_cast<int64_t>(a->n_layers) * a->n_exact;
      exact_input_kernel<<<static_cast<unsigned>((warps * 32 + 255) / 256), 256, 0, s>>>(
          static_cast<const __nv_bfloat16*>(a->X_exact), static_cast<const __nv_bfloat16*>(a->gain),
          a->exact_idx, a->n_exact, a->n_layers, a->d_out, start, rc, a->rows, pl.R,
          a->d_out / pl.bn_map, static_cast<__nv_bfloat16*>(xhat), ss, device_error_word());
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "exact-row input launch");
    }
    if ((st = mark(start, 1)) != RF_OK) return st;
    sp.rows = static_cast<int32_t>(rc);
    sp.first = start == 0 ? 1 : 0;
    if (!state_maps(rc)) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the GDN state");
    if (la > 0) {
      // the first layers' projections; then their states on `s`, beside the others'
      // projections on the side stream limited to the SMs the states leave (whichever is
      // dispatched first, neither can take the other's SMs); then the others' projections
      // on every SM, sharing the side launch's tile counter
      if ((st = launch_gdn_proj(a, pl, rc, xhat, ss, kb, vb, gb, s, 0, la)) != RF_OK) return st;
      int* ctr = tile_counter_slot();
      if (ctr == nullptr) return fail(RF_ERR_CUDA, "tile counter unavailable");
      cudaError_t e = cudaMemsetAsync(ctr, 0, sizeof(int), s);
      if (e == cudaSuccess) e = cudaEventRecord(hs->side_start, s);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(hs->side, hs->side_start, 0);
      if (e != cudaSuccess) return cuda_fail(e, "ordering the other layers' projections");
      const int free_pairs = (sm_count() - la * a->n_heads) / 2;
      if (free_pairs > 0 &&
          (st = launch_gdn_proj(a, pl, rc, xhat, ss, kb, vb, gb, hs->side, la, a->n_layers - la,
                                free_pairs, ctr)) != RF_OK)
        return st;
      if ((e = cudaEventRecord(hs->side_done, hs->side)) != cudaSuccess)
        return cuda_fail(e, "recording the other layers' projections");
      GdnStateParams spa = sp;
      spa.layers = la;
      spa.layer_base = 0;
      if ((e = launch_gdn_state(spa, s)) != cudaSuccess) return cuda_fail(e, "GDN state launch");
      if ((st = launch_gdn_proj(a, pl, rc, xhat, ss, kb, vb, gb, s, la, a->n_layers - la, 0,
                                ctr)) != RF_OK)
        return st;
      if ((e = cudaStreamWaitEvent(s, hs->side_done, 0)) != cudaSuccess)
        return cuda_fail(e, "ordering after the other layers' projections");
    } else if ((st = launch_gdn_proj(a, pl, rc, xhat, ss, kb, vb, gb, s)) != RF_OK) {
      return st;
    }
    if (want_rho) {
      rho_chunk_kernel<<<LH, kRhoThreads, 0, s>>>(gb, a->n_heads, pl.R, rc, start, a->exact_idx,
                                                  a->n_exact, rho_acc, start == 0 ? 1 : 0);
      cudaError_t e = cudaGetLastError();
      if (e != cudaSuccess) return cuda_fail(e, "rho launch");
    }
    if ((st = mark(start, 2)) != RF_OK) return st;
    GdnStateParams spb = sp;
    spb.layers = a->n_layers - la;
    spb.layer_base = la;
    cudaError_t e = launch_gdn_state(spb, s);
    if (e != cudaSuccess) return cuda_fail(e, "GDN state launch");
    if ((st = mark(start, 3)) != RF_OK) return st;
  }
  if (a->h_on_host) {  // later work on `s` (and the caller's reuse of H) follows the copy
    cudaError_t e = cudaStreamWaitEvent(s, hs->h_done, 0);
    if (e != cudaSuccess) return cuda_fail(e, "ordering after the split-state copy");
  }
  if (want_rho) {  // rho, and the terminal-state correction on the final state
    rho_finish_kernel<<<LH, 256, 0, s>>>(rho_acc, 0, a->rho, a->delta_M, a->S, kDk * kDk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "rho launch");
  }
  return guards_check(ws, pl.lay, s);
}
