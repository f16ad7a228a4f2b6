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
//   warp 9      TMA producer: k, v (hi and lo) and the gates of each chunk;
//   warp 8      MMA issuer (one thread) and TMEM owner;
//   warps 4-7   chunk-local work for the chunk ahead: P = K K^T on the tensor
//               cores, T by blocked inversion on the CUDA cores, then
//               W^T = K^T (T diag(b g))^T and U^T = V^T (T diag(b))^T;
//   warps 0-3   the serial part: NEW^T = U^T - S_0 W^T (tensor cores, added to
//               U^T in TMEM), its decay-weighted bf16 split, S += NEW'^T K, and
//               the bf16 split of the new S for the next chunk.
// The chunk-local work of chunk c + 1 overlaps the serial part of chunk c.
// Every product takes bf16 high and low parts of both operands (hi.hi + hi.lo
// + lo.hi: about 16 significant bits); S and NEW' are A operands read from
// TMEM, the rest come from 128-byte-swizzled shared-memory tiles.
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
constexpr uint32_t kKV = 4 * kBox;                  // hi (2 boxes) then lo (2 boxes)
constexpr uint32_t kOffK = 0;                       // two chunk buffers of k
constexpr uint32_t kOffV = kOffK + 2 * kKV;         // one chunk buffer of v
constexpr uint32_t kOffT = kOffV + kKV;             // T diag(b g) hi, lo; T diag(b) hi, lo
constexpr uint32_t kOffW = kOffT + 4 * kBox;        // -W hi, lo: [j][t] rows (MN-major B)
constexpr uint32_t kOffGateRaw = kOffW + 4 * kBox;  // two buffers: alpha[64], beta[64]
constexpr uint32_t kOffGate = kOffGateRaw + 2 * 512;  // two slots: beta, b g, decay, G
constexpr uint32_t kOffScr = kOffGate + 2 * 1024;     // B, T: [64][65] f32 each
constexpr int kLd = 65;
constexpr uint32_t kOffBar = kOffScr + 2 * kC * kLd * 4;
constexpr uint32_t kStateSmem = kOffBar + 256 + 1024;
static_assert(kStateSmem <= 232448, "state kernel shared memory");

// TMEM columns
constexpr uint32_t kColS = 0;     // S (f32, 128)
constexpr uint32_t kColSh = 128;  // S bf16 high parts (64 columns = 128 values)
constexpr uint32_t kColSl = 192;  // S bf16 remainders
constexpr uint32_t kColN = 256;   // U^T, then NEW^T (f32, 64)
constexpr uint32_t kColNh = 320;  // NEW'^T bf16 high parts (32 columns)
constexpr uint32_t kColNl = 352;  // NEW'^T remainders
constexpr uint32_t kColP = 384;   // P = K K^T, then W^T (f32, 64)

// barriers
enum : int {
  kBarKFull = 0,   // 2: k + gates of a chunk landed
  kBarKEmpty = 2,  // 2: the chunk's last product that reads k is done
  kBarVFull = 4,
  kBarVEmpty = 5,
  kBarP = 6,       // P done
  kBarUW = 7,      // U^T and W^T done
  kBarDA = 8,      // NEW^T done
  kBarDB = 9,      // S update done
  kBarTops = 10,   // T operands written (4 warp arrivals)
  kBarWop = 11,    // -W operand written
  kBarNop = 12,    // NEW' operand written
  kBarSops = 13,   // S operand written and S pre-scaled
  kBarFinal = 14,
  kNumBars = 15,
};

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

// log of the chunk's total decay: warp-wide sum of log alpha over its n rows
__device__ __forceinline__ float chunk_log_decay(const float* alpha, int n, int lane) {
  float s = 0.f;
  for (int t = lane; t < n; t += 32) s += fmaxf(logf(alpha[t]), -80.f);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s;
}

// the three split terms of one product: hi.hi, hi.lo, lo.hi
struct Split {
  uint32_t a[3];
  uint32_t b[3];
};

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
  float* Ts = Bs + kC * kLd;
  float* Xs = reinterpret_cast<float*>(sm + kOffT);  // scratch while T is formed

  const int h = blockIdx.x, l = blockIdx.y;
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
    if (lane == 0 && nch > 0) {
      tma_prefetch(&p.tmK);
      tma_prefetch(&p.tmV);
      int loaded_k = 0, loaded_v = 0;
      bool ok = true;
      for (int c = 0; c < nch && ok; ++c) {
        const int kb = c & 1;
        if (c >= 2 && !mbar_wait(&bar[kBarKEmpty + kb], ((c - 2) >> 1) & 1, abort_flag, p.err, kErrGdn)) {
          ok = false;
          break;
        }
        uint64_t* kf = &bar[kBarKFull + kb];
        mbar_expect_tx(kf, kKV + 512);
        for (int part = 0; part < 2; ++part)
          for (int box = 0; box < 2; ++box)
            tma_load_3d(sb + kOffK + kb * kKV + part * 2 * kBox + box * kBox, &p.tmK, kf, 64 * box,
                        kC * c, 2 * lh + part);
        bulk_load(sb + kOffGateRaw + kb * 512, alpha_g + kC * c, 256, kf);
        bulk_load(sb + kOffGateRaw + kb * 512 + 256, beta_g + kC * c, 256, kf);
        loaded_k = c + 1;
        if (c >= 1 && !mbar_wait(&bar[kBarVEmpty], (c - 1) & 1, abort_flag, p.err, kErrGdn)) {
          ok = false;
          break;
        }
        uint64_t* vf = &bar[kBarVFull];
        mbar_expect_tx(vf, kKV);
        for (int part = 0; part < 2; ++part)
          for (int box = 0; box < 2; ++box)
            tma_load_3d(sb + kOffV + part * 2 * kBox + box * kBox, &p.tmV, vf, 64 * box, kC * c,
                        2 * lh + part);
        loaded_v = c + 1;
      }
      if (!ok) {  // let the copies already issued land before the CTA exits
        for (int c = loaded_k - 2 < 0 ? 0 : loaded_k - 2; c < loaded_k; ++c)
          mbar_drain(&bar[kBarKFull + (c & 1)], (c >> 1) & 1);
        if (loaded_v > 0) mbar_drain(&bar[kBarVFull], (loaded_v - 1) & 1);
      }
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0 && nch > 0) {
      const uint32_t id_p = idesc_bf16_f32(128, 64);
      const uint32_t id_uw = idesc_bf16_f32(128, 64) | (1u << 15);
      const uint32_t id_da = idesc_bf16_f32(128, 64) | (1u << 16);
      const uint32_t id_db = idesc_bf16_f32(128, 128) | (1u << 16);
      auto wait = [&](int b, uint32_t parity) -> bool {
        const bool ok = mbar_wait(&bar[b], parity, abort_flag, p.err, kErrGdn);
        tc_fence_after();
        return ok;
      };
      // P = K K^T: A = the k tile read as 128 K-major rows (rows 64-127 are not used)
      auto issue_p = [&](int c) {
        const uint32_t kt = sb + kOffK + (c & 1) * kKV;
        const uint32_t ah[3] = {kt, kt, kt + 2 * kBox};
        const uint32_t bh[3] = {kt, kt + 2 * kBox, kt};
        uint32_t acc = 0;
        for (int g = 0; g < 3; ++g)
          for (int kblk = 0; kblk < 2; ++kblk)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t ad = sdesc_kmajor_sw128(ah[g] + kblk * kBox + 32 * ks);
              const uint64_t bd = sdesc_kmajor_sw128(bh[g] + kblk * kBox + 32 * ks);
              mma_bf16(tb + kColP, ad, bd, id_p, acc);
              acc = 1;
            }
        mma_commit(&bar[kBarP]);
      };
      // U^T = V^T (T diag(b))^T and W^T = K^T (T diag(b g))^T
      auto issue_uw = [&](int c) {
        const uint32_t kt = sb + kOffK + (c & 1) * kKV, vt = sb + kOffV;
        const uint32_t tw = sb + kOffT, tu = sb + kOffT + 2 * kBox;
        for (int which = 0; which < 2; ++which) {
          const uint32_t at = which == 0 ? vt : kt;
          const uint32_t bt = which == 0 ? tu : tw;
          const uint32_t dcol = which == 0 ? kColN : kColP;
          const uint32_t ah[3] = {at, at, at + 2 * kBox};
          const uint32_t bh[3] = {bt, bt + kBox, bt};
          uint32_t acc = 0;
          for (int g = 0; g < 3; ++g)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t ad = sdesc_mnmajor_sw128(ah[g] + 2048 * ks, 8192);
              const uint64_t bd = sdesc_kmajor_sw128(bh[g] + 32 * ks);
              mma_bf16(tb + dcol, ad, bd, id_uw, acc);
              acc = 1;
            }
        }
        mma_commit(&bar[kBarUW]);
        mma_commit(&bar[kBarVEmpty]);
      };
      bool ok = wait(kBarKFull, 0);
      if (ok) issue_p(0);
      ok = ok && wait(kBarTops, 0) && wait(kBarVFull, 0);
      if (ok) issue_uw(0);
      for (int c = 0; c < nch && ok; ++c) {
        if (!wait(kBarWop, c & 1) || !wait(kBarSops, c & 1)) break;
        {  // NEW^T += S_0 (-W)^T, added to U^T
          const uint32_t wt = sb + kOffW;
          const uint32_t ah[3] = {tb + kColSh, tb + kColSh, tb + kColSl};
          const uint32_t bh[3] = {wt, wt + 2 * kBox, wt};
          for (int g = 0; g < 3; ++g)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              mma_bf16_tmem_a(tb + kColN, ah[g] + 8 * ks, sdesc_mnmajor_sw128(bh[g] + 2048 * ks, 8192),
                              id_da, 1u);
          mma_commit(&bar[kBarDA]);
        }
        if (c + 1 < nch) {
          if (!wait(kBarKFull + ((c + 1) & 1), ((c + 1) >> 1) & 1)) break;
          issue_p(c + 1);
        }
        if (!wait(kBarNop, c & 1)) break;
        {  // S += NEW'^T K
          const uint32_t kt = sb + kOffK + (c & 1) * kKV;
          const uint32_t ah[3] = {tb + kColNh, tb + kColNh, tb + kColNl};
          const uint32_t bh[3] = {kt, kt + 2 * kBox, kt};
          for (int g = 0; g < 3; ++g)
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
              mma_bf16_tmem_a(tb + kColS, ah[g] + 8 * ks, sdesc_mnmajor_sw128(bh[g] + 2048 * ks, 8192),
                              id_db, 1u);
          mma_commit(&bar[kBarDB]);
          mma_commit(&bar[kBarKEmpty + (c & 1)]);
        }
        if (c + 1 < nch) {
          if (!wait(kBarTops, (c + 1) & 1) || !wait(kBarVFull, (c + 1) & 1)) break;
          issue_uw(c + 1);
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
    for (int c = 0; c < nch; ++c) {
      const int kb = c & 1;
      bool ok = mbar_wait(&bar[kBarKFull + kb], (c >> 1) & 1, abort_flag, p.err, kErrGdn);
      if (!named_bar_all(kPreBar, 128, ok)) break;
      float* gs = reinterpret_cast<float*>(sm + kOffGate + kb * 1024);  // beta, bg, dec, G
      if (q == 0) {
        const float* ga = reinterpret_cast<const float*>(sm + kOffGateRaw + kb * 512);
        const float* gbeta = ga + 64;
        const int n = min(kC, p.rows - kC * c);
        float la[2], be[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int t = 2 * lane + e;
          la[e] = t < n ? fmaxf(logf(ga[t]), -80.f) : 0.f;
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
        gs[64 + 2 * lane] = be[0] * expf(g0);
        gs[64 + 2 * lane + 1] = be[1] * expf(g1);
        gs[128 + 2 * lane] = expf(gC - g0);
        gs[128 + 2 * lane + 1] = expf(gC - g1);
        gs[192 + 2 * lane] = g0;
        gs[192 + 2 * lane + 1] = g1;
      }
      ok = mbar_wait(&bar[kBarP], c & 1, abort_flag, p.err, kErrGdn);
      if (!named_bar_all(kPreBar, 128, ok)) break;
      tc_fence_after();
      // B_ts = b_t e^{G_t - G_s} P_ts below the diagonal
      if (q < 2) {
        const int t = pt;
        const float gt = gs[192 + t], bt = gs[t];
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          tmem_ld32(tb + (static_cast<uint32_t>(32 * q) << 16) + kColP + 32 * half, r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int s = 32 * half + j;
            Bs[t * kLd + s] = s < t ? bt * expf(gt - gs[192 + s]) * __uint_as_float(r[j]) : 0.f;
          }
        }
      }
      named_bar_sync(kPreBar, 128);
      // T = (I + B)^-1, unit lower triangular, by 16 x 16 blocks: diagonal blocks
      // by substitution, then block diagonals a - b = 1, 2, 3:
      //   T_ab = -T_aa sum_{c=b}^{a-1} B_ac T_cb
      if (pt < 64) {
        const int b = pt >> 4, s = pt & 15, o = 16 * b;
        float x[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          float acc = r == s ? 1.f : 0.f;
#pragma unroll
          for (int k = 0; k < r; ++k) acc = fmaf(-Bs[(o + r) * kLd + o + k], x[k], acc);
          x[r] = acc;
        }
#pragma unroll
        for (int r = 0; r < 16; ++r) Ts[(o + r) * kLd + o + s] = x[r];
      }
      named_bar_sync(kPreBar, 128);
      for (int d = 1; d < 4; ++d) {
        const int nel = (4 - d) * 256;
        for (int idx = pt; idx < nel; idx += 128) {
          const int b = idx >> 8, e = idx & 255, r = e >> 4, cc = e & 15, a = b + d;
          float acc = 0.f;
          for (int c2 = b; c2 < a; ++c2) {
            const float* brow = Bs + (16 * a + r) * kLd + 16 * c2;
            const float* tcol = Ts + (16 * c2) * kLd + 16 * b + cc;
#pragma unroll
            for (int k = 0; k < 16; ++k) acc = fmaf(brow[k], tcol[k * kLd], acc);
          }
          Xs[(16 * a + r) * kLd + 16 * b + cc] = acc;
        }
        named_bar_sync(kPreBar, 128);
        for (int idx = pt; idx < nel; idx += 128) {
          const int b = idx >> 8, e = idx & 255, r = e >> 4, cc = e & 15, a = b + d;
          const float* trow = Ts + (16 * a + r) * kLd + 16 * a;
          const float* xcol = Xs + (16 * a) * kLd + 16 * b + cc;
          float acc = 0.f;
#pragma unroll
          for (int k = 0; k < 16; ++k) acc = fmaf(trow[k], xcol[k * kLd], acc);
          Ts[(16 * a + r) * kLd + 16 * b + cc] = -acc;
        }
        named_bar_sync(kPreBar, 128);
      }
      // T diag(b g) and T diag(b) as bf16 hi/lo K-major tiles [t][s]
      for (int idx = pt; idx < kC * 8; idx += 128) {
        const int t = idx >> 3, ch = idx & 7;
        float w[8], u[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int s = 8 * ch + e;
          const float v = s <= t ? Ts[t * kLd + s] : 0.f;
          w[e] = v * gs[64 + s];
          u[e] = v * gs[s];
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
      // -W as the MN-major B operand: row j holds W^T[j][0..63]
      ok = mbar_wait(&bar[kBarUW], c & 1, abort_flag, p.err, kErrGdn);
      if (!named_bar_all(kPreBar, 128, ok)) break;
      tc_fence_after();
      {
        const int j = pt;
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          tmem_ld32(tb + (static_cast<uint32_t>(32 * q) << 16) + kColP + 32 * half, r);
          tmem_wait_ld();
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            float x[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = -__uint_as_float(r[8 * c8 + e]);
            uint4 hi, lo;
            split8(x, hi, lo);
            const uint32_t off = swz(j, 4 * half + c8);
            *reinterpret_cast<uint4*>(sm + kOffW + off) = hi;
            *reinterpret_cast<uint4*>(sm + kOffW + 2 * kBox + off) = lo;
          }
        }
      }
      fence_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarWop]);
    }
  } else {
    // ---------------------------------------------------------------- serial part
    const int i = tid;  // state row = TMEM lane
    const uint32_t lrow = tb + (static_cast<uint32_t>(32 * warp) << 16);
    const float* src = s_in != nullptr ? s_in + static_cast<size_t>(i) * kDk : nullptr;
    float* dst = s_out + static_cast<size_t>(i) * kDk;
    // S (f32, pre-scaled by the next chunk's decay g) and its bf16 split, 64 columns at a time
    auto put_state = [&](const float (&s)[64], int half, float g) {
      uint32_t r[32], hi[32], lo[32];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
#pragma unroll
        for (int j = 0; j < 32; ++j) r[j] = __float_as_uint(g * s[32 * cc + j]);
        tmem_st32(lrow + kColS + 64 * half + 32 * cc, r);
      }
#pragma unroll
      for (int m = 0; m < 32; ++m) split2(s[2 * m], s[2 * m + 1], hi[m], lo[m]);
      tmem_st32(lrow + kColSh + 32 * half, hi);
      tmem_st32(lrow + kColSl + 32 * half, lo);
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
        const float g = expf(chunk_log_decay(ga, min(kC, p.rows), lane));
        for (int half = 0; half < 2; ++half) {
          float s[64];
#pragma unroll
          for (int j = 0; j < 64; j += 4) {
            const float4 x = src != nullptr ? *reinterpret_cast<const float4*>(src + 64 * half + j)
                                            : make_float4(0.f, 0.f, 0.f, 0.f);
            s[j] = x.x; s[j + 1] = x.y; s[j + 2] = x.z; s[j + 3] = x.w;
          }
          put_state(s, half, g);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[kBarSops]);
      }
    }
    for (int c = 0; c < nch && ok; ++c) {
      const int kb = c & 1;
      if (!mbar_wait(&bar[kBarDA], c & 1, abort_flag, p.err, kErrGdn)) break;
      tc_fence_after();
      {  // NEW'^T[i][t] = NEW^T[i][t] e^{G_C - G_t}
        const float* dec = reinterpret_cast<const float*>(sm + kOffGate + kb * 1024) + 128;
        uint32_t hi[32], lo[32];
        for (int half = 0; half < 2; ++half) {
          uint32_t r[32];
          tmem_ld32(lrow + kColN + 32 * half, r);
          tmem_wait_ld();
#pragma unroll
          for (int m = 0; m < 16; ++m) {
            const int t = 32 * half + 2 * m;
            split2(__uint_as_float(r[2 * m]) * dec[t], __uint_as_float(r[2 * m + 1]) * dec[t + 1],
                   hi[16 * half + m], lo[16 * half + m]);
          }
        }
        tmem_st32(lrow + kColNh, hi);
        tmem_st32(lrow + kColNl, lo);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar[kBarNop]);
      if (!mbar_wait(&bar[kBarDB], c & 1, abort_flag, p.err, kErrGdn)) break;
      tc_fence_after();
      if (c + 1 == nch) {
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t r[32];
          tmem_ld32(lrow + kColS + 32 * cc, r);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + 32 * cc + j) =
                make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                            __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        }
      } else {
        const int kn = (c + 1) & 1;
        if (!mbar_wait(&bar[kBarKFull + kn], ((c + 1) >> 1) & 1, abort_flag, p.err, kErrGdn)) break;
        const float* ga = reinterpret_cast<const float*>(sm + kOffGateRaw + kn * 512);
        const float g = expf(chunk_log_decay(ga, min(kC, p.rows - kC * (c + 1)), lane));
        for (int half = 0; half < 2; ++half) {
          float s[64];
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            uint32_t r[32];
            tmem_ld32(lrow + kColS + 64 * half + 32 * cc, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) s[32 * cc + j] = __uint_as_float(r[j]);
          }
          put_state(s, half, g);
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
                          const float* ss, __nv_bfloat16* kb, __nv_bfloat16* vb, float* gb,
                          cudaStream_t s) {
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
  __nv_bfloat16* kb = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_k);
  __nv_bfloat16* vb = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_v);
  float* gb = reinterpret_cast<float*>(ws + pl.off_gate);

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
    if (!state_maps(rc)) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the GDN state");
    cudaError_t e = launch_gdn_state(sp, s);
    if (e != cudaSuccess) return cuda_fail(e, "GDN state launch");
    if ((st = mark(start, 3)) != RF_OK) return st;
  }
  return RF_OK;
}
