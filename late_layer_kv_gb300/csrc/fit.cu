// fit.cu -- ridgefill_fit: the closed-form ridge maps (RidgeFill, "Training-Free
// Late-Layer Cache Fill for Faster Prefill", section 2.2: "The ridge map",
// "Fitting", "The penalty").
//
// ACCUMULATE adds one batch of calibration pairs to caller-owned f64 running
// sums.  One tcgen05 GEMM forms [X^T X ; Y_1^T X ; ... ; Y_L^T X] over the
// batch's rows: X and Y are read in place as MN-major operands (their rows are
// the reduction dimension), products of bf16 inputs are exact in f32, the
// batch is summed in f32 in TMEM and each tile is added into the f64 sums.
// The column sums and the row count go the same way.
//
// SOLVE, from the sums:
//   mu_S = sx/n, mu_l = sy_l/n, G~ = G - n mu_S mu_S^T, C~_l = C_l - n mu_l mu_S^T
//   alpha = lambda * tr(G~) / d_in
//   s_i = (G~_ii + alpha)^(-1/2);  G^ = diag(s) (G~ + alpha I) diag(s)   (unit diagonal)
//   G^ = L L^T (blocked Cholesky, f32), X = L^-1 (blocked), G^-1 = X^T X
//   A_l[o, i] = s_i sum_k (s_k C~_l[o, k]) G^-1[k, i],  b_l = mu_l - A_l mu_S
// The last product is one tcgen05 GEMM over the split bf16 operands
// [c_hi | c_hi | c_lo] x [g_hi | g_lo | g_hi] (K = 3 d_in), which carries about
// 16 bits of each f32 operand.
#include <cmath>
#include <mutex>

#include "abi_common.h"
#include "sm103_ptx.cuh"

namespace rf {
namespace {

constexpr int kNB = 64;  // Cholesky / triangular-inverse block

// ------------------------------------------------------------ column sums
// Partial column sums of a [batches][rows, width] bf16 array over row slabs:
// part[slab][col_base + b*width + c] = sum of rows in the slab (f32 over 64-row
// runs, then f64), eight columns per thread so each load is 16 bytes.
__global__ void colsum_partial_kernel(const __nv_bfloat16* in, int64_t rows, int width,
                                      int batches, int64_t batch_stride, int64_t slab_rows,
                                      double* part, int64_t part_ld, int64_t col_base) {
  const int oct = width / 8;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= static_cast<int64_t>(oct) * batches) return;
  const int b = static_cast<int>(t / oct);
  const int c = static_cast<int>(t % oct) * 8;
  const int64_t r_lo = static_cast<int64_t>(blockIdx.y) * slab_rows;
  const int64_t r_hi = r_lo + slab_rows < rows ? r_lo + slab_rows : rows;
  const __nv_bfloat16* p = in + b * batch_stride + c;
  double acc[8] = {};
  for (int64_t r0 = r_lo; r0 < r_hi; r0 += 64) {
    const int64_t r1 = r0 + 64 < r_hi ? r0 + 64 : r_hi;
    float f[8] = {};
#pragma unroll 4
    for (int64_t r = r0; r < r1; ++r) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(p + r * width));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
        f[2 * e] += x.x;
        f[2 * e + 1] += x.y;
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += f[e];
  }
  double* dst = part + blockIdx.y * part_ld + col_base + static_cast<int64_t>(b) * width + c;
#pragma unroll
  for (int e = 0; e < 8; ++e) dst[e] = acc[e];
}

// out_x[c] += sum over slabs (c < nx), out_y[c - nx] += ... (fixed order).
__global__ void colsum_reduce_kernel(const double* part, int slabs, int64_t part_ld, int64_t nx,
                                     double* out_x, double* out_y) {
  const int64_t c = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (c >= part_ld) return;
  double s = 0.0;
  for (int k = 0; k < slabs; ++k) s += part[k * part_ld + c];
  if (c < nx) out_x[c] += s;
  else out_y[c - nx] += s;
}

__global__ void add_count_kernel(double* count, double rows) { *count += rows; }

// ------------------------------------------------------------ solve: centring
// One block: mu_x, alpha (trace of the centred Gram), the equilibration s.
constexpr int kPrepThreads = 1024;  // the diagonal reads are latency-bound: many in flight
__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const double* G, const double* sx,
                                                            const double* count, int d,
                            double lam, float* s_f32, float* mu_f32, double* mu_f64,
                            double* alpha_ws, double* alpha_out) {
  __shared__ double red[kPrepThreads];
  const double n = *count;
  double tr = 0.0;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const double mu = sx[i] / n;
    mu_f64[i] = mu;
    mu_f32[i] = static_cast<float>(mu);
    tr += G[static_cast<size_t>(i) * d + i] - n * mu * mu;
  }
  red[threadIdx.x] = tr;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  const double alpha = lam * red[0] / d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const double mu = sx[i] / n;
    const double dd = G[static_cast<size_t>(i) * d + i] - n * mu * mu + alpha;
    s_f32[i] = static_cast<float>(dd > 0.0 ? 1.0 / sqrt(dd) : 0.0);
  }
  if (threadIdx.x == 0) {
    *alpha_ws = alpha;
    if (alpha_out != nullptr) *alpha_out = alpha;
  }
}

// ------------------------------------------------------------ f64 inputs without f64 math
// This GPU's f64 pipe runs at a small fraction of its f32 rate, so kernels that read the
// f64 sums take each value apart with integer operations into a double-float pair
// (hi, lo): hi holds the 24 leading significant bits (truncated) and lo the next 23, so
// |v - (hi + lo)| < 2^-46 |v|.  Magnitudes below 2^-126 give hi = 0 (below 2^-103, lo = 0);
// magnitudes above the f32 range give hi = +-inf, and a NaN stays a NaN.  w0 and w1 are
// the low and high 32-bit words of the f64.
__device__ __forceinline__ float2 ff_of_bits(uint32_t w0, uint32_t w1) {
  const uint32_t sign = w1 & 0x80000000u;
  const int e = static_cast<int>((w1 >> 20) & 0x7ffu);  // biased f64 exponent
  float hi, lo = 0.f;
  if (e > 1150) {
    const bool nan = e == 2047 && ((w1 & 0xfffffu) | w0) != 0u;
    hi = __uint_as_float(sign | 0x7f800000u | (nan ? 0x400000u : 0u));
  } else if (e < 897) {
    hi = __uint_as_float(sign);
  } else {
    // same exponent, the top 23 of the 52 fraction bits
    hi = __uint_as_float(sign | (static_cast<uint32_t>(e - 896) << 23) | ((w1 & 0xfffffu) << 3) |
                         (w0 >> 29));
    if (e >= 920) {
      // the next 23 fraction bits r, worth r * 2^(E - 23) with 2^E = 2^-23 ulp(hi): written
      // as (1 + r 2^-23) 2^E - 2^E, a difference that f32 takes exactly
      const uint32_t base = sign | (static_cast<uint32_t>(e - 919) << 23);
      lo = __uint_as_float(base | ((w0 & 0x1fffffffu) >> 6)) - __uint_as_float(base);
    }
  }
  return make_float2(hi, lo);
}

__device__ __forceinline__ float2 ff_load(const double* p) {
  const uint2 w = *reinterpret_cast<const uint2*>(p);
  return ff_of_bits(w.x, w.y);
}

// a - b c for double-float a, b, c, rounded once to f32.  The product's high part and its
// exact error (fma), then an exact two-sum of the high parts; the low-order terms are
// carried to about 2^-46 of |a|, so a difference down to 2^-22 |a| still comes out within
// about one f32 ulp (f64 arithmetic rounded to f32 would hold down to about 2^-29 |a|).
__device__ __forceinline__ float ff_sub_mul(float2 a, float2 b, float2 c) {
  const float ph = __fmul_rn(b.x, c.x);  // kept apart from the subtraction below
  const float pl = fmaf(b.x, c.x, -ph) + fmaf(b.x, c.y, b.y * c.x);
  const float sh = __fsub_rn(a.x, ph);
  const float z = __fsub_rn(sh, a.x);
  const float se = __fadd_rn(__fsub_rn(a.x, __fsub_rn(sh, z)), __fsub_rn(-ph, z));
  return sh + (se + (a.y - pl));
}

constexpr int kCentreRows = 8;  // rows per thread of the centring kernels

// G^ = diag(s) (G - sx mu^T + alpha I) diag(s), f32 [d, d] (sx mu^T = n mu mu^T); eight
// consecutive columns of kCentreRows rows per thread (d is a multiple of 128)
__global__ void __launch_bounds__(256) equilibrate_kernel(const double* __restrict__ G,
                                                          const double* __restrict__ sx,
                                                          const double* __restrict__ mu,
                                                          const float* __restrict__ s,
                                                          const double* __restrict__ alpha, int d,
                                                          float* __restrict__ Gh) {
  const int g = d / 8;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int j0 = static_cast<int>(t % g) * 8;
  const int64_t i0 = t / g * kCentreRows;
  if (i0 >= d) return;
  float2 m[8];
  float sj[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    m[c] = ff_load(mu + j0 + c);
    sj[c] = s[j0 + c];
  }
  const float2 al = ff_load(alpha);
  const float a = al.x + al.y;
  for (int r = 0; r < kCentreRows && i0 + r < d; ++r) {
    const int64_t i = i0 + r;
    const float2 b = ff_load(sx + i);
    const float si = s[i];
    const uint4* src = reinterpret_cast<const uint4*>(G + i * d + j0);
    float v[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = src[q];
      v[2 * q] = ff_sub_mul(ff_of_bits(w.x, w.y), b, m[2 * q]);
      v[2 * q + 1] = ff_sub_mul(ff_of_bits(w.z, w.w), b, m[2 * q + 1]);
    }
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      if (i == j0 + c) v[c] += a;
      v[c] = v[c] * si * sj[c];
    }
    float4* dst = reinterpret_cast<float4*>(Gh + i * d + j0);
    dst[0] = make_float4(v[0], v[1], v[2], v[3]);
    dst[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}

// ------------------------------------------------------------ bf16 splits
__device__ __forceinline__ void split_bf16(float v, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(v);
  lo = __float2bfloat16_rn(v - __bfloat162float(hi));
}

__device__ __forceinline__ uint32_t bf16x2(__nv_bfloat16 a, __nv_bfloat16 b) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(a)) |
         (static_cast<uint32_t>(__bfloat16_as_ushort(b)) << 16);
}

// Products to about f32 precision on the bf16 tensor cores.  x = h + m + l with h = bf16(x),
// m = bf16(x - h), l = bf16(x - h - m) (both differences exact in f32).  A matrix is stored
// as seven K-wide bf16 planes [h, h, m, m, h, l, h] per row; planes 0-5 of one such split
// against planes 1-6 of another pair h h, h m, m m, m h, h l and l h, so one product over
// the stacked K (6 K) sums every term but m l, l m and l l, each within about 2^-24 of the
// result.
constexpr int kPlanes = 7;

__device__ __forceinline__ void split3_bf16(float x, __nv_bfloat16& h, __nv_bfloat16& m,
                                            __nv_bfloat16& l) {
  h = __float2bfloat16_rn(x);
  const float r = x - __bfloat162float(h);
  m = __float2bfloat16_rn(r);
  l = __float2bfloat16_rn(r - __bfloat162float(m));
}

// the seven planes of n consecutive values (n = 2 or 4 here) as bf16 words: w[plane][n / 2]
template <int N>
__device__ __forceinline__ void planes_of(const float (&x)[N], uint32_t (&w)[kPlanes][N / 2]) {
#pragma unroll
  for (int i = 0; i < N; i += 2) {
    __nv_bfloat16 h0, m0, l0, h1, m1, l1;
    split3_bf16(x[i], h0, m0, l0);
    split3_bf16(x[i + 1], h1, m1, l1);
    const uint32_t h = bf16x2(h0, h1), m = bf16x2(m0, m1), l = bf16x2(l0, l1);
    w[0][i / 2] = h; w[1][i / 2] = h; w[2][i / 2] = m; w[3][i / 2] = m;
    w[4][i / 2] = h; w[5][i / 2] = l; w[6][i / 2] = h;
  }
}

// Seven-plane split of a batch of row-major f32 matrices: output row r of batch entry bat,
// [kPlanes * K] bf16 at out + (bat * rows + r) * kPlanes * K, holds element (r, k) of the
// source, src[bat * sstride + r * ld + k], or, transposed (TR), src[bat * sstride + k * ld + r].
// One 64 x 64 tile per CTA through shared memory (grid K / 64, ceil(rows / 64), batches);
// K is a multiple of 64.
template <bool TR>
__global__ void __launch_bounds__(256) split7_kernel(const float* __restrict__ src, int64_t ld,
                                                     int64_t sstride, int rows, int K,
                                                     __nv_bfloat16* __restrict__ out) {
  __shared__ float t[64][65];
  const int k0 = blockIdx.x * 64, r0 = blockIdx.y * 64;
  const int64_t bat = blockIdx.z;
  const float* sb = src + bat * sstride;
  float v[16];  // all loads in flight before the shared-memory stores
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = threadIdx.x + 256 * q;
    const int i = e / 64, j = e % 64;  // i: source row in the tile, j: source column
    if (TR) v[q] = r0 + j < rows ? sb[static_cast<int64_t>(k0 + i) * ld + r0 + j] : 0.f;
    else v[q] = r0 + i < rows ? sb[static_cast<int64_t>(r0 + i) * ld + k0 + j] : 0.f;
  }
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = threadIdx.x + 256 * q;
    const int i = e / 64, j = e % 64;
    if (TR) t[j][i] = v[q];
    else t[i][j] = v[q];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 64 * 16; e += 256) {
    const int r = e / 16, kq = (e % 16) * 4;
    if (r0 + r >= rows) continue;
    const float x[4] = {t[r][kq], t[r][kq + 1], t[r][kq + 2], t[r][kq + 3]};
    uint32_t w[kPlanes][2];
    planes_of(x, w);
    __nv_bfloat16* o = out + (bat * rows + r0 + r) * static_cast<int64_t>(kPlanes) * K + k0 + kq;
#pragma unroll
    for (int pl = 0; pl < kPlanes; ++pl)
      *reinterpret_cast<uint2*>(o + static_cast<int64_t>(pl) * K) = make_uint2(w[pl][0], w[pl][1]);
  }
}

// Copies n held-back panel blocks (rows kb and kb + 1 of block column kb - 1) from `pst`
// into place (256 threads).
__device__ __forceinline__ void copy_held(float* A, int ld, int kb, const float* pst, int n) {
  for (int b = 0; b < n; ++b) {
    float* dst = A + static_cast<size_t>(kb + b) * kNB * ld + static_cast<size_t>(kb - 1) * kNB;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = 4 * (static_cast<int>(threadIdx.x) + 256 * q);  // four floats of one row
      *reinterpret_cast<float4*>(dst + static_cast<size_t>(e / kNB) * ld + e % kNB) =
          *reinterpret_cast<const float4*>(pst + b * kNB * kNB + e);
    }
  }
}

// ------------------------------------------------------------ Cholesky (f32)
// One 64x64 diagonal block: the lower factor L_kk and its inverse, both right-looking
// in one sweep over the
// columns j: the pivot, column j of L and row j of L^-1 scaled by its reciprocal,
// then the rank-1 updates a_ik -= l_ij l_kj and x_ic -= l_ij x_jc.  A pivot <= 0
// records kErrNumeric in the device error word and continues with pivot 1.
// 256 threads, ti = tid % 16, tk = tid / 16, all cells in registers: thread
// (ti, tk) keeps a_ik for rows i = ti + 16u and columns k = tk + 16v, and x_ic
// transposed, rows i = tk + 16v and columns c = ti + 16u, so column j of L and
// row j of L^-1 both sit in the sixteen threads tk = j % 16 (half a warp).  That
// half-warp reads the pivot a_jj from its lane ti = j % 16 by a shuffle, takes its
// root and reciprocal and publishes the column and the row through shared memory
// (double-buffered by the parity of j) with zeros outside i > j and c <= j.  The
// updates then need no masks: the zeros leave every other cell unchanged, and only
// the (never read) upper triangle of a takes stray updates.  One barrier a step.  The
// inverse L_kk^-1 (zeros above) goes to Linv [64, 64] and over the diagonal block: later
// steps read only the blocks below it, and the triangular inverse starts from it.  col and
// xrow are [2][64] floats of shared memory each.
__device__ void factor_diag(float* blk, int ld, int* err, float* Linv, float (*col)[kNB],
                            float (*xrow)[kNB]) {
  const int tid = threadIdx.x, ti = tid & 15, tk = tid >> 4;
  float a[4][4], x[4][4];
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      a[u][v] = blk[static_cast<size_t>(ti + 16 * u) * ld + tk + 16 * v];
      x[v][u] = (tk + 16 * v == ti + 16 * u) ? 1.f : 0.f;
    }
  const int hl = 16 * (tk & 1);                   // this half-warp's first lane
  const unsigned half = 0xffffu << hl;
  // j = 16 jw + jt with jw unrolled, so every register index below is static
#pragma unroll
  for (int jw = 0; jw < 4; ++jw) {
    for (int jt = 0; jt < 16; ++jt) {
      const int j = 16 * jw + jt, buf = j & 1;
      if (tk == jt) {  // column j of L (a[u][jw]) and row j of L^-1 (x[jw][u])
        float v = __shfl_sync(half, a[jw][jw], hl + jt);  // a_jj, from lane ti = jt
        if (!(v > 0.f)) {
          if (ti == 0) atomicCAS(err, 0, kErrNumeric);
          v = 1.f;
        }
        const float r = rsqrtf(v), p = v * r;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = ti + 16 * u;  // row of a, column of x
          float lv = 0.f, xv = 0.f;
          if (i > j) {
            a[u][jw] *= r;
            lv = a[u][jw];
          } else {
            if (i == j) a[u][jw] = p;
            x[jw][u] *= r;
            xv = x[jw][u];
          }
          col[buf][i] = lv;
          xrow[buf][i] = xv;
        }
      }
      __syncthreads();
      float ci[4], xr[4], ck[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        ci[u] = col[buf][ti + 16 * u];
        xr[u] = xrow[buf][ti + 16 * u];
        ck[u] = col[buf][tk + 16 * u];
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int v = 0; v < 4; ++v) {
          a[u][v] = fmaf(-ci[u], ck[v], a[u][v]);
          x[v][u] = fmaf(-ck[v], xr[u], x[v][u]);
        }
    }
  }
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      const int i = ti + 16 * u, k = tk + 16 * v;
      const float xv = i <= k ? x[v][u] : 0.f;  // x cell: row k, column i
      blk[static_cast<size_t>(k) * ld + i] = xv;
      Linv[k * kNB + i] = xv;
    }
}

// The first diagonal block (the later ones are factored by the panel launches).
__global__ void __launch_bounds__(256) potrf_diag_kernel(float* A, int ld, int* err, float* Linv) {
  __shared__ float col[2][kNB];   // l_ij for i > j, else 0
  __shared__ float xrow[2][kNB];  // x_jc for c <= j, else 0
  factor_diag(A, ld, err, Linv, col, xrow);
}

__global__ void __launch_bounds__(256) copy_held_kernel(float* A, int ld, int kb, const float* pst,
                                                        int n) {
  copy_held(A, ld, kb, pst, n);
}

// Panel of Cholesky step kb and its two look-ahead block columns, one 64-row block
// ib = kb + 1 + blockIdx.x per CTA (256 threads, 4 x 4 outputs each):
//   P_ib = A[ib, kb] L_kk^-T = A[ib, kb] Linv^T          (the block of L, written back)
//   A[ib, kb + 1] -= P_ib P_(kb+1)^T                      (step kb)
//   A[ib, kb + 2] -= L[ib, kb-1] L[kb+2, kb-1]^T + P_ib P_(kb+2)^T   (steps kb - 1, kb)
// Every CTA forms P_(kb+1) and P_(kb+2) itself rather than waiting for the CTAs that own
// them.  Column kb + 2 takes step kb - 1 here (not in the trailing update of step kb - 1),
// so the trailing update of step kb covers the columns from kb + 4 on and the panel of step
// kb needs only the trailing update of step kb - 2: one step of the factorisation runs
// between the two.  With `planes` set, the blocks ib >= kb + 4 also go there as seven-plane
// splits, row (ib - kb - 4) * 64 + r, for that trailing update on the tensor cores.
// CTA 0 (ib = kb + 1), whose block of column kb + 1 is the next diagonal block, then
// factors it (factor_diag, L_(kb+1)^-1 to Linv_out), so the launch chain of the
// factorisation is one launch per step.  The blocks of rows kb + 1 and kb + 2 of column kb
// are read unsolved by every CTA: they go to `pst` and the next launch's last CTA copies
// them into place (with `held` blocks of the previous step from `pst_prev`).
// Dynamic shared memory: Lt = Linv^T [64][68], then X (the block being solved, later
// L[ib, kb-1]), P1 = P_(kb+1), P2 = P_(kb+2), Pi = P_ib and Q = L[kb+2, kb-1], [64][65] each.
constexpr int kPanelSmem = (kNB * (kNB + 4) + 5 * kNB * (kNB + 1)) * 4;

__device__ __forceinline__ void load_block(const float* src, int ld, float (*dst)[kNB + 1]) {
  float v[16];  // all loads in flight before the shared-memory stores
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = threadIdx.x + 256 * q;
    v[q] = src[static_cast<size_t>(e / kNB) * ld + e % kNB];
  }
#pragma unroll
  for (int q = 0; q < 16; ++q) {
    const int e = threadIdx.x + 256 * q;
    dst[e / kNB][e % kNB] = v[q];
  }
}

// acc = X Linv^T for this thread's rows r0 + u and columns c0 + w (Linv[c][k] = 0 for k > c)
__device__ __forceinline__ void solve_block(const float (*X)[kNB + 1], const float (*Lt)[kNB + 4],
                                            int r0, int c0, float (&acc)[4][4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int w = 0; w < 4; ++w) acc[u][w] = 0.f;
  for (int k = 0; k < c0 + 4; ++k) {
    const float4 l = *reinterpret_cast<const float4*>(&Lt[k][c0]);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float xv = X[r0 + u][k];
      acc[u][0] = fmaf(xv, l.x, acc[u][0]);
      acc[u][1] = fmaf(xv, l.y, acc[u][1]);
      acc[u][2] = fmaf(xv, l.z, acc[u][2]);
      acc[u][3] = fmaf(xv, l.w, acc[u][3]);
    }
  }
}

__device__ __forceinline__ void store_tile(float (*dst)[kNB + 1], int r0, int c0,
                                           const float (&acc)[4][4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u)
#pragma unroll
    for (int w = 0; w < 4; ++w) dst[r0 + u][c0 + w] = acc[u][w];
}

// cv -= Lf Rf^T for this thread's rows r0 + u (rows of Lf) and columns c0 + w (rows of Rf)
__device__ __forceinline__ void sub_product(const float (*Lf)[kNB + 1], const float (*Rf)[kNB + 1],
                                            int r0, int c0, float (&cv)[4][4]) {
  for (int k = 0; k < kNB; ++k) {
    float pr[4], pc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      pr[u] = Lf[r0 + u][k];
      pc[u] = Rf[c0 + u][k];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int w = 0; w < 4; ++w) cv[u][w] = fmaf(-pr[u], pc[w], cv[u][w]);
  }
}

__device__ __forceinline__ void load_tile(const float* blk, int ld, int r0, int c0, float (&cv)[4][4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const float4 c4 = *reinterpret_cast<const float4*>(blk + static_cast<size_t>(r0 + u) * ld + c0);
    cv[u][0] = c4.x; cv[u][1] = c4.y; cv[u][2] = c4.z; cv[u][3] = c4.w;
  }
}

__device__ __forceinline__ void put_tile(float* blk, int ld, int r0, int c0, const float (&cv)[4][4]) {
#pragma unroll
  for (int u = 0; u < 4; ++u)
    *reinterpret_cast<float4*>(blk + static_cast<size_t>(r0 + u) * ld + c0) =
        make_float4(cv[u][0], cv[u][1], cv[u][2], cv[u][3]);
}

__global__ void __launch_bounds__(256) panel_ahead_kernel(float* A, int ld, int kb,
                                                          const float* Linv, float* Linv_out,
                                                          float* pst, const float* pst_prev,
                                                          int held, __nv_bfloat16* planes,
                                                          int* err) {
  extern __shared__ __align__(16) float psm[];
  typedef float Tile[kNB + 1];
  auto Lt = reinterpret_cast<float (*)[kNB + 4]>(psm);
  Tile* X = reinterpret_cast<Tile*>(psm + kNB * (kNB + 4));
  Tile* P1 = X + kNB;
  Tile* P2 = P1 + kNB;
  Tile* Pi = P2 + kNB;
  Tile* Q = Pi + kNB;
  const int ib = kb + 1 + blockIdx.x;
  const int tid = threadIdx.x;
  const int r0 = (tid / 16) * 4, c0 = (tid % 16) * 4;
  auto blk = [&](int bi, int bj) {
    return A + static_cast<size_t>(bi) * kNB * ld + static_cast<size_t>(bj) * kNB;
  };
  // the previous step's held-back blocks (rows kb, kb + 1 of column kb - 1): read by no
  // launch of the factorisation from here on
  if (held > 0 && blockIdx.x + 1 == gridDim.x) copy_held(A, ld, kb, pst_prev, held);
  {
    float lv[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) lv[q] = Linv[tid + 256 * q];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int e = tid + 256 * q;
      Lt[e % kNB][e / kNB] = lv[q];
    }
  }
  load_block(blk(kb + 1, kb), ld, X);
  __syncthreads();
  float acc[4][4];
  solve_block(X, Lt, r0, c0, acc);  // P_(kb+1)
  store_tile(P1, r0, c0, acc);
  if (ib >= kb + 2) {
    __syncthreads();  // X free
    load_block(blk(kb + 2, kb), ld, X);
    __syncthreads();
    solve_block(X, Lt, r0, c0, acc);  // P_(kb+2)
    store_tile(P2, r0, c0, acc);
    if (ib >= kb + 3) {
      __syncthreads();
      load_block(blk(ib, kb), ld, X);
      __syncthreads();
      solve_block(X, Lt, r0, c0, acc);  // P_ib
      store_tile(Pi, r0, c0, acc);
    }
  }
  const Tile* own = ib == kb + 1 ? P1 : (ib == kb + 2 ? P2 : Pi);
  // the blocks of rows kb + 1 and kb + 2 are still to be read (unsolved) by the other CTAs:
  // they go to `pst`, and the next diagonal-factor launch copies them into place
  if (ib <= kb + 2) put_tile(pst + (ib - kb - 1) * kNB * kNB, kNB, r0, c0, acc);
  else put_tile(blk(ib, kb), ld, r0, c0, acc);
  if (planes != nullptr && ib >= kb + 4) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      uint32_t w[kPlanes][2];
      planes_of(acc[u], w);
      __nv_bfloat16* o =
          planes + (static_cast<int64_t>(ib - kb - 4) * kNB + r0 + u) * kPlanes * kNB + c0;
#pragma unroll
      for (int pl = 0; pl < kPlanes; ++pl)
        *reinterpret_cast<uint2*>(o + pl * kNB) = make_uint2(w[pl][0], w[pl][1]);
    }
  }
  const bool prev = kb >= 1 && ib >= kb + 2;  // step kb - 1 on column kb + 2
  __syncthreads();  // every solve is done (X free); P1, P2 and Pi are complete
  if (prev) {
    load_block(blk(ib, kb - 1), ld, X);   // L[ib, kb - 1]
    load_block(blk(kb + 2, kb - 1), ld, Q);  // L[kb + 2, kb - 1]
  }
  float cv[4][4];
  load_tile(blk(ib, kb + 1), ld, r0, c0, cv);
  sub_product(own, P1, r0, c0, cv);
  put_tile(blk(ib, kb + 1), ld, r0, c0, cv);
  if (ib >= kb + 2) {
    load_tile(blk(ib, kb + 2), ld, r0, c0, cv);
    if (prev) {
      __syncthreads();  // X and Q complete
      sub_product(X, Q, r0, c0, cv);
    }
    sub_product(own, P2, r0, c0, cv);
    put_tile(blk(ib, kb + 2), ld, r0, c0, cv);
  }
  if (ib == kb + 1) {  // block (kb + 1, kb + 1) is complete: factor it
    __syncthreads();   // its rows, written above, are visible to the whole CTA
    factor_diag(blk(kb + 1, kb + 1), ld, err, Linv_out, reinterpret_cast<float (*)[kNB]>(&X[0][0]),
                reinterpret_cast<float (*)[kNB]>(&X[0][0] + 2 * kNB));
  }
}

// Zeros above the diagonal of the f32 [d, d] matrix, four columns per thread (d * d < 2^31)
__global__ void zero_upper_kernel(float* A, int d) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int q = d / 4;
  if (t >= d * q) return;
  const int r = t / q, c = (t - r * q) * 4;
  if (c + 3 <= r) return;  // on or below the diagonal
  float4* p = reinterpret_cast<float4*>(A) + t;
  if (c > r) {
    *p = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    float4 v = *p;
    if (c + 1 > r) v.y = 0.f;
    if (c + 2 > r) v.z = 0.f;
    if (c + 3 > r) v.w = 0.f;
    *p = v;
  }
}

// ------------------------------------------------------------ split operands


// B' [d, 2d] = [hi(G^-1) | lo(G^-1)] from the f64 inverse: hi = bf16(v_hi) and
// lo = bf16((v_hi - hi) + v_lo) of the double-float (v_hi, v_lo), the first difference
// exact; eight consecutive k per thread
__global__ void split_ginv_kernel(const double* __restrict__ Gi, int d, __nv_bfloat16* __restrict__ Bp) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int g = d / 8;
  if (t >= static_cast<int64_t>(d) * g) return;
  const int64_t i = t / g;
  const int k0 = static_cast<int>(t % g) * 8;
  const uint4* src = reinterpret_cast<const uint4*>(Gi + i * d + k0);
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 w = src[q];
    const float2 v0 = ff_of_bits(w.x, w.y), v1 = ff_of_bits(w.z, w.w);
    const __nv_bfloat16 h0 = __float2bfloat16_rn(v0.x), h1 = __float2bfloat16_rn(v1.x);
    const __nv_bfloat16 l0 = __float2bfloat16_rn((v0.x - __bfloat162float(h0)) + v0.y);
    const __nv_bfloat16 l1 = __float2bfloat16_rn((v1.x - __bfloat162float(h1)) + v1.y);
    hw[q] = bf16x2(h0, h1);
    lw[q] = bf16x2(l0, l1);
  }
  __nv_bfloat16* row = Bp + i * 2 * d;
  *reinterpret_cast<uint4*>(row + k0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  *reinterpret_cast<uint4*>(row + d + k0) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// X = L^-1 (f32, lower, n elements) split into the four bf16 planes [hi; lo; hi; hi] of n
// elements each: planes 0-2 against planes 1-3, summed over the stacked rows, give
// hi^T lo + lo^T hi + hi^T hi in one Gram product.  Eight elements per thread.
__global__ void split2_kernel(const float* __restrict__ X, int64_t n, __nv_bfloat16* __restrict__ P) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= n / 8) return;
  const float4* src = reinterpret_cast<const float4*>(X) + 2 * t;
  const float4 x0 = src[0], x1 = src[1];
  const float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    __nv_bfloat16 h0, l0, h1, l1;
    split_bf16(v[2 * q], h0, l0);
    split_bf16(v[2 * q + 1], h1, l1);
    hw[q] = bf16x2(h0, h1);
    lw[q] = bf16x2(l0, l1);
  }
  const uint4 h = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  uint4* dst = reinterpret_cast<uint4*>(P) + t;
  const int64_t plane = n / 8;  // uint4 per plane
  dst[0] = h;
  dst[plane] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  dst[2 * plane] = h;
  dst[3 * plane] = h;
}

// A' [L*d_out, 2d] = [hi(c) | lo(c)],  c[o, k] = s_k (C[o, k] - sy[o] mu_x[k])
// (sy[o] mu_x[k] = n mu_y[o] mu_x[k]), centred in double-float as above; eight consecutive
// k of kCentreRows rows per thread (d is a multiple of 128): 64-byte reads of C, 16-byte
// stores of each part
__global__ void __launch_bounds__(256) split_rhs_kernel(const double* __restrict__ C,
                                                        const double* __restrict__ sy,
                                                        const double* __restrict__ mu_x,
                                                        const float* __restrict__ s,
                                                        int64_t rows_out, int d,
                                                        __nv_bfloat16* __restrict__ Ap) {
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int g = d / 8;
  const int k0 = static_cast<int>(t % g) * 8;
  const int64_t o0 = t / g * kCentreRows;
  if (o0 >= rows_out) return;
  float2 m[8];
  float sk[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    m[c] = ff_load(mu_x + k0 + c);
    sk[c] = s[k0 + c];
  }
#pragma unroll 2
  for (int r = 0; r < kCentreRows; ++r) {
    const int64_t o = o0 + r;
    if (o >= rows_out) break;
    const float2 b = ff_load(sy + o);
    const uint4* src = reinterpret_cast<const uint4*>(C + o * d + k0);
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 w = src[q];
      const float v0 = ff_sub_mul(ff_of_bits(w.x, w.y), b, m[2 * q]) * sk[2 * q];
      const float v1 = ff_sub_mul(ff_of_bits(w.z, w.w), b, m[2 * q + 1]) * sk[2 * q + 1];
      __nv_bfloat16 h0, l0, h1, l1;
      split_bf16(v0, h0, l0);
      split_bf16(v1, h1, l1);
      hw[q] = bf16x2(h0, h1);
      lw[q] = bf16x2(l0, l1);
    }
    __nv_bfloat16* row = Ap + o * 2 * d;
    *reinterpret_cast<uint4*>(row + k0) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    *reinterpret_cast<uint4*>(row + d + k0) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  }
}

// b[o] = mu_y[o] - sum_t part[o, t]
__global__ void bias_kernel(const double* sy, const double* count, const float* part,
                            int n_tiles, int64_t rows_out, float* b) {
  const int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (o >= rows_out) return;
  double acc = 0.0;
  for (int t = 0; t < n_tiles; ++t) acc += part[o * n_tiles + t];
  b[o] = static_cast<float>(sy[o] / (*count) - acc);
}

// ------------------------------------------------------------ plan
struct FitPlan {
  size_t off_gh = 0, off_s = 0, off_mu32 = 0, off_mu64 = 0, off_alpha = 0,
         off_xs = 0, off_gi = 0, off_bp = 0, off_ap = 0, off_part = 0,
         off_cs = 0, off_linv = 0, off_pst = 0, total = 0;
  int bn = 0;
  int slabs = 0;
  int64_t slab_rows = 0;
  Layout lay;
};

rf_status validate_fit(const rf_fit_args* a) {
  if (a == nullptr) return fail(RF_ERR_ARG, "args is NULL");
  if (a->n_layers < 1) return fail(RF_ERR_SHAPE, "n_layers must be >= 1");
  if (a->d_in < 128 || a->d_in % 128 != 0 || a->d_in > 16384)
    return fail(RF_ERR_SHAPE, "d_in must be a multiple of 128 in [128, 16384]");
  if (a->d_out < 128 || a->d_out % 128 != 0) return fail(RF_ERR_SHAPE, "d_out must be a positive multiple of 128");
  if ((a->flags & ~(RF_FIT_ACCUMULATE | RF_FIT_SOLVE)) != 0 || a->flags == 0)
    return fail(RF_ERR_ARG, "flags must be RF_FIT_ACCUMULATE and/or RF_FIT_SOLVE");
  if (a->rows < 0 || a->rows >= (int64_t(1) << 31)) return fail(RF_ERR_ARG, "rows out of range");
  if (static_cast<int64_t>(a->n_layers) * a->d_out >= (int64_t(1) << 31) / 3)
    return fail(RF_ERR_SHAPE, "n_layers * d_out too large");
  if ((a->flags & RF_FIT_SOLVE) && !(a->lambda >= 0.0)) return fail(RF_ERR_ARG, "lambda must be >= 0");
  return RF_OK;
}

void plan_fit(const rf_fit_args* a, FitPlan* pl) {
  const size_t d = a->d_in, M = static_cast<size_t>(a->n_layers) * a->d_out;
  pl->bn = (a->d_in % 256 == 0) ? 256 : 128;
  Layout& lay = pl->lay;
  if (a->flags & RF_FIT_ACCUMULATE) {
    const int64_t rows = a->rows > 0 ? a->rows : 1;
    pl->slab_rows = ceil_div(ceil_div(rows, 64), 64) * 64;  // at most 64 slabs, 64-row runs
    pl->slabs = static_cast<int>(ceil_div(rows, pl->slab_rows));
    pl->off_cs = lay.take(static_cast<size_t>(pl->slabs) * (d + M) * 8);
  }
  if (a->flags & RF_FIT_SOLVE) {
    pl->off_gh = lay.take(d * d * 4);
    pl->off_s = lay.take(d * 4);
    pl->off_mu32 = lay.take(d * 4);
    pl->off_mu64 = lay.take(d * 8);
    pl->off_alpha = lay.take(8);
    pl->off_linv = lay.take(2 * kNB * kNB * 4);
    pl->off_pst = lay.take(4 * kNB * kNB * 4);
    pl->off_xs = lay.take(4 * d * d * 2);  // bf16 planes [hi; lo; hi; hi] of L^-1
    pl->off_gi = lay.take(d * d * 8);
    pl->off_bp = lay.take(d * 2 * d * 2);
    pl->off_ap = lay.take(M * 2 * d * 2);
    pl->off_part = lay.take(M * (d / pl->bn) * 4);
  }
  pl->total = lay.off;
}

// Gram-mode tcgen05 GEMM: out_G[m, n] += sum_k Xa[k, m] Xb[k, n] for the d-wide
// arrays Xa, Xb ([rows, d], MN-major), and, if Y is given, out_C[l, o, n] +=
// sum_k Y[l, k, o] Xb[k, n].
// Gram products on CTA pairs (M = 256: each CTA stages 128 columns of [X | Y] and half of
// the tile's X columns).

rf_status launch_gram(const void* Xa, const void* Xb, const void* Y, int L, int64_t rows, int d,
                      int dout, int bn, double* out_G, double* out_C, cudaStream_t s,
                      bool sym = false) {
  GemmParams p{};
  p.mode = kModeGram;
  p.k_blocks = static_cast<int32_t>(ceil_div(rows, kBK));
  const uint64_t xrow = static_cast<uint64_t>(d) * 2, yrow = static_cast<uint64_t>(dout) * 2;
  bool ok = make_tmap_3d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xa, d, rows, 1, xrow, 0, 64, 64,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_3d(&p.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xb, d, rows, 1, xrow, 0, 64,
                          64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (Y != nullptr)
    ok = ok && make_tmap_3d(&p.tmA2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, dout, rows, L, yrow,
                            yrow * rows, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the Gram GEMM");
  p.gram_x_tiles = d / kBM;
  p.gram_y_tiles_per_layer = dout / kBM;
  p.m_tiles = p.gram_x_tiles + (Y != nullptr ? L * p.gram_y_tiles_per_layer : 0);
  // pairs take 512-column tiles where d allows and the tiles fill eight waves: each A
  // stage then feeds two MMAs, which halves the A reads per flop
  const int64_t wide_tiles = static_cast<int64_t>((p.m_tiles + 1) / 2) * (d / kGramWideCols);
  sym = sym && Y == nullptr && bn == 2 * kBM;
  const bool wide = !sym && d % kGramWideCols == 0 && wide_tiles >= 8 * (sm_count() / 2);
  if (wide) {
    // wide tiles stage two 64-column blocks per copy: rank-4 views {64 columns, rows,
    // column blocks, layers} whose third dimension steps 128 bytes
    const uint64_t dx[4] = {64, static_cast<uint64_t>(rows), static_cast<uint64_t>(d / 64), 1};
    const uint64_t sx[3] = {xrow, 128, xrow * static_cast<uint64_t>(rows)};
    const uint32_t bx[4] = {64, 64, 2, 1};
    ok = make_tmap_4d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xa, dx, sx, bx,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    ok = ok && make_tmap_4d(&p.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Xb, dx, sx, bx,
                            CU_TENSOR_MAP_SWIZZLE_128B);
    if (Y != nullptr) {
      const uint64_t dy[4] = {64, static_cast<uint64_t>(rows), static_cast<uint64_t>(dout / 64),
                              static_cast<uint64_t>(L)};
      const uint64_t sy[3] = {yrow, 128, yrow * static_cast<uint64_t>(rows)};
      ok = ok && make_tmap_4d(&p.tmA2, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, dy, sy, bx,
                              CU_TENSOR_MAP_SWIZZLE_128B);
    }
    if (!ok) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the wide Gram GEMM");
  }
  p.bn = wide ? kGramWideCols : bn;
  p.n_tiles = d / p.bn;
  p.batches = 1;
  p.group_m = 16;
  p.d_out = dout;
  p.gram_G = out_G;
  p.gram_C = out_C;
  p.gram_ld = d;
  p.lim_a = static_cast<int64_t>(d) * d;
  p.lim_b = static_cast<int64_t>(L) * dout * d;
  p.err = device_error_word();
  if (p.err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  p.lower = sym ? 1 : 0;
  p.gram_sym = sym ? 1 : 0;
  const int64_t u = (p.m_tiles + 1) / 2;
  const int64_t tiles = sym ? u * (u + 1) / 2 : u * p.n_tiles;
  const int pairs = static_cast<int>(tiles < sm_count() / 2 ? tiles : sm_count() / 2);
  if (pairs <= 0) return RF_OK;
  const cudaError_t e = launch_gemm2(p, pairs, s);
  if (e != cudaSuccess) return cuda_fail(e, "Gram GEMM launch");
  return RF_OK;
}

// out_b = alpha A_b B_b^T (+ out_b when beta_one) on the tensor cores for b < batches, from
// the seven-plane splits of A_b [M, K] (Ap7) and B_b [N, K] (Bp7), each batch entry's rows
// following the previous entry's: planes 0-5 of A against planes 1-6 of B, K' = 6 K.
// out_b = out + b * out_bstride, rows out_ld apart; lower: one square product (M = N), only
// the pair tiles on and below the diagonal (the upper part of a diagonal tile is written
// too).  `lim` elements of out are in bounds (checked by debug builds).  max_pairs > 0
// caps the CTA pairs (the SMs the launch takes).
rf_status launch_f32_product(const __nv_bfloat16* Ap7, const __nv_bfloat16* Bp7, int M, int N,
                             int K, int batches, float* out, int64_t out_ld, int64_t out_bstride,
                             float alpha, bool beta_one, bool lower, int64_t lim, cudaStream_t s,
                             int max_pairs = 0) {
  if (M <= 0 || N <= 0 || batches <= 0) return RF_OK;
  GemmParams p{};
  p.mode = kModeF32;
  p.k_blocks = 6 * K / kBK;
  // stages of two k-blocks (6K / 64 is even), each operand staged by one copy through a
  // rank-4 view {64 k, rows, k-blocks, batches}
  const uint64_t row = static_cast<uint64_t>(kPlanes) * K * 2;
  const uint64_t kbl = static_cast<uint64_t>(6 * K / kBK), nb = static_cast<uint64_t>(batches);
  const uint64_t dA[4] = {kBK, static_cast<uint64_t>(M), kbl, nb};
  const uint64_t sA[3] = {row, 128, row * static_cast<uint64_t>(M)};
  const uint64_t dB[4] = {kBK, static_cast<uint64_t>(N), kbl, nb};
  const uint64_t sB[3] = {row, 128, row * static_cast<uint64_t>(N)};
  const uint32_t bx[4] = {kBK, 128, 2, 1};
  bool ok = make_tmap_4d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Ap7, dA, sA, bx,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  ok = ok && make_tmap_4d(&p.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Bp7 + K, dB, sB, bx,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  p.k2 = 1;
  if (!ok) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for an f32 product");
  p.m_tiles = static_cast<int32_t>(ceil_div(M, kBM));
  p.bn = 256;
  p.n_tiles = static_cast<int32_t>(ceil_div(N, 256));
  p.batches = lower ? 1 : batches;
  p.group_m = 16;
  p.rows = M;
  p.cols = N;
  p.out_f32 = out;
  p.out_ld = static_cast<int32_t>(out_ld);
  p.out_bstride = out_bstride;
  p.alpha = alpha;
  p.beta_one = beta_one ? 1 : 0;
  p.lower = lower ? 1 : 0;
  p.lim_b = lim;
  p.err = device_error_word();
  if (p.err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  const int64_t u = (p.m_tiles + 1) / 2;
  const int64_t tiles = lower ? u * (u + 1) / 2 : u * p.n_tiles * p.batches;
  int pairs = static_cast<int>(tiles < sm_count() / 2 ? tiles : sm_count() / 2);
  if (max_pairs > 0 && pairs > max_pairs) pairs = max_pairs;
  const cudaError_t e = launch_gemm2(p, pairs, s);
  if (e != cudaSuccess) return cuda_fail(e, "f32 product launch");
  return RF_OK;
}

rf_status accumulate(const rf_fit_args* a, const FitPlan& pl, uint8_t* ws, cudaStream_t s) {
  const int64_t rows = a->rows;
  if (rows == 0) return RF_OK;
  const int L = a->n_layers, din = a->d_in, dout = a->d_out;
  HostStreamer* hs = host_streamer();
  if (hs == nullptr) return RF_ERR_CUDA;
  // one caller at a time on the device's side stream and its events
  std::lock_guard<std::mutex> lk(host_stream_mutex());
  // the Gram products first, on `s`; the column sums, HBM-bound, then run beside them on the
  // side stream, in the few SMs (and the issue slots) the persistent GEMM leaves
  cudaError_t e = cudaEventRecord(hs->side_start, s);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(hs->side, hs->side_start, 0);
  if (e != cudaSuccess) return cuda_fail(e, "ordering the column sums");
  rf_status st = launch_gram(a->X, a->X, a->Y, L, rows, din, dout, pl.bn, a->G, a->C, s);
  if (st != RF_OK) return st;
  // column sums: slab partials, then a fixed-order reduction into the f64 sums
  cudaStream_t cs_stream = hs->side;
  double* cs = reinterpret_cast<double*>(ws + pl.off_cs);
  const int64_t ld = din + static_cast<int64_t>(L) * dout;
  const int64_t tx = din / 8, ty = static_cast<int64_t>(dout / 8) * L;
  colsum_partial_kernel<<<dim3(static_cast<unsigned>((tx + 127) / 128), pl.slabs), 128, 0,
                          cs_stream>>>(static_cast<const __nv_bfloat16*>(a->X), rows, din, 1, 0,
                                       pl.slab_rows, cs, ld, 0);
  colsum_partial_kernel<<<dim3(static_cast<unsigned>((ty + 127) / 128), pl.slabs), 128, 0,
                          cs_stream>>>(static_cast<const __nv_bfloat16*>(a->Y), rows, dout, L,
                                       rows * dout, pl.slab_rows, cs, ld, din);
  colsum_reduce_kernel<<<static_cast<unsigned>((ld + 255) / 256), 256, 0, cs_stream>>>(
      cs, pl.slabs, ld, din, a->sx, a->sy);
  add_count_kernel<<<1, 1, 0, cs_stream>>>(a->count, static_cast<double>(rows));
  e = cudaGetLastError();
  if (e == cudaSuccess) e = cudaEventRecord(hs->side_done, cs_stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(s, hs->side_done, 0);
  if (e != cudaSuccess) return cuda_fail(e, "column-sum launch");
  return RF_OK;
}

rf_status solve(const rf_fit_args* a, const FitPlan& pl, uint8_t* ws, cudaStream_t s) {
  const int d = a->d_in;
  const int64_t M = static_cast<int64_t>(a->n_layers) * a->d_out;
  float* Gh = reinterpret_cast<float*>(ws + pl.off_gh);
  float* sc = reinterpret_cast<float*>(ws + pl.off_s);
  float* mu32 = reinterpret_cast<float*>(ws + pl.off_mu32);
  double* mu64 = reinterpret_cast<double*>(ws + pl.off_mu64);
  double* alpha = reinterpret_cast<double*>(ws + pl.off_alpha);
  double* Gi = reinterpret_cast<double*>(ws + pl.off_gi);
  __nv_bfloat16* Xs = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_xs);
  __nv_bfloat16* Bp = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_bp);
  __nv_bfloat16* Ap = reinterpret_cast<__nv_bfloat16*>(ws + pl.off_ap);
  float* part = reinterpret_cast<float*>(ws + pl.off_part);
  int* err = device_error_word();
  if (err == nullptr) return fail(RF_ERR_CUDA, "device error word unavailable");
  const int64_t dd = static_cast<int64_t>(d) * d;

  prep_kernel<<<1, kPrepThreads, 0, s>>>(a->G, a->sx, a->count, d, a->lambda, sc, mu32, mu64, alpha,
                                a->alpha_out);
  const int64_t eq_threads = ceil_div(d, kCentreRows) * (d / 8);
  equilibrate_kernel<<<static_cast<unsigned>(ceil_div(eq_threads, 256)), 256, 0, s>>>(
      a->G, a->sx, mu64, sc, alpha, d, Gh);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "fit preparation launch");

  // blocked Cholesky, lower factor in place, right-looking with a look-ahead of two block
  // columns: the panel launch of step kb (on `s`) solves block column kb and applies step kb
  // to block column kb + 1 and steps kb - 1 and kb to block column kb + 2; the update of the
  // rest of the trailing matrix (the columns from kb + 4 on) by step kb runs on the side
  // stream, and the panel of step kb + 2 is the first launch that waits for it, so the
  // trailing updates leave the chain of panel launches; each panel launch also factors the
  // next diagonal block.  Concurrent launches write disjoint blocks, and every element takes
  // its updates in step order; the blocks above the diagonal are never read.  The diagonal
  // blocks receive L_kk^-1 (the first step of the inverse below); the panels read the
  // factor's copy in `linv` (two buffers, by step parity).
  const int nb = d / kNB;
  float* linv = reinterpret_cast<float*>(ws + pl.off_linv);
  float* pst = reinterpret_cast<float*>(ws + pl.off_pst);
  // seven-plane splits of the trailing updates' panels (one buffer per step parity) and of
  // the inverse's operands, in the area of the f64 inverse (8 d^2 bytes, free until the
  // G^-1 product)
  __nv_bfloat16* cplanes = reinterpret_cast<__nv_bfloat16*>(Gi);
  const int64_t plane_buf = static_cast<int64_t>(d) * kPlanes * kNB;
  HostStreamer* hs = host_streamer();
  if (hs == nullptr) return RF_ERR_CUDA;
  if ((e = cudaFuncSetAttribute(panel_ahead_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kPanelSmem)) != cudaSuccess)
    return cuda_fail(e, "Cholesky panel attributes");
  {
    // one caller at a time on the device's side stream and its events
    std::lock_guard<std::mutex> lk(host_stream_mutex());
    int last_trailing = -1, held = 0;
    constexpr int kBlk = kNB * kNB;
    potrf_diag_kernel<<<1, 256, 0, s>>>(Gh, d, err, linv);
    for (int kb = 0; kb + 1 < nb; ++kb) {
      // block column kb + 2 was last written by the trailing update of step kb - 2
      if (kb >= 2 && kb + 2 < nb && (e = cudaStreamWaitEvent(s, hs->side_ev[kb % 2], 0)) != cudaSuccess)
        return cuda_fail(e, "Cholesky look-ahead");
      __nv_bfloat16* planes = cplanes + (kb % 2) * plane_buf;
      // L_kk^-1 and the held-back blocks alternate between two buffers by step parity
      panel_ahead_kernel<<<nb - kb - 1, 256, kPanelSmem, s>>>(
          Gh, d, kb, linv + (kb % 2) * kBlk, linv + ((kb + 1) % 2) * kBlk, pst + (kb % 2) * 2 * kBlk,
          pst + ((kb + 1) % 2) * 2 * kBlk, held, planes, err);
      held = nb - kb - 1 < 2 ? nb - kb - 1 : 2;  // blocks of rows kb + 1, kb + 2 held back
      const int rem = d - (kb + 4) * kNB;
      if (rem > 0) {
        if ((e = cudaEventRecord(hs->side_start, s)) == cudaSuccess)
          e = cudaStreamWaitEvent(hs->side, hs->side_start, 0);
        if (e != cudaSuccess) return cuda_fail(e, "Cholesky look-ahead");
        // the next panel launch (nb - kb - 2 CTAs, one per SM) keeps its SMs
        const int pairs = (sm_count() - (nb - kb - 2)) / 2;
        const int64_t off = static_cast<int64_t>(kb + 4) * kNB * (d + 1);
        rf_status st = launch_f32_product(planes, planes, rem, rem, kNB, 1, Gh + off, d, 0, -1.f,
                                          true, true, dd - off, hs->side, pairs > 0 ? pairs : 1);
        if (st != RF_OK) return st;
        if ((e = cudaEventRecord(hs->side_ev[kb % 2], hs->side)) != cudaSuccess)
          return cuda_fail(e, "Cholesky look-ahead");
        last_trailing = kb;
      }
    }
    if (held > 0)  // the last step's held-back block
      copy_held_kernel<<<1, 256, 0, s>>>(Gh, d, nb - 1, pst + ((nb - 2) % 2) * 2 * kBlk, held);
    if (last_trailing >= 0 &&
        (e = cudaStreamWaitEvent(s, hs->side_ev[last_trailing % 2], 0)) != cudaSuccess)
      return cuda_fail(e, "Cholesky look-ahead");
  }
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "Cholesky launch");
  zero_upper_kernel<<<static_cast<unsigned>((dd / 4 + 255) / 256), 256, 0, s>>>(Gh, d);
  // X = L^-1 in place: the 64 x 64 diagonal blocks are inverted already; recursive
  // doubling: blocks [s1 | s2] of size s (already inverted) merge as
  //   T = L_21 X_11,  X_21 = -X_22 T,
  // every pair of a level in one batched f32 product on the tensor cores (the blocks above
  // the diagonal are zero, so the triangular operands are used whole).  T lives in the
  // area of the bf16 planes of X (free until the split below), the operands' seven-plane
  // splits in `cplanes`.
  float* T = reinterpret_cast<float*>(Xs);
  for (int sz = kNB; sz < d; sz *= 2) {
    const int full = d / (2 * sz);        // pairs with both halves of size sz
    const int rest = d - full * 2 * sz;   // a last pair [sz | rest - sz] if rest > sz
    for (int part = 0; part < 2; ++part) {
      const int cnt = part == 0 ? full : (rest > sz ? 1 : 0);
      if (cnt == 0) continue;
      const int b0 = part == 0 ? 0 : full * 2 * sz;
      const int s2 = part == 0 ? sz : rest - sz;
      const int64_t step = 2 * static_cast<int64_t>(sz) * (d + 1);
      const float* l21 = Gh + static_cast<size_t>(b0 + sz) * d + b0;
      const float* x11 = Gh + static_cast<size_t>(b0) * d + b0;
      const float* x22 = Gh + static_cast<size_t>(b0 + sz) * d + b0 + sz;
      float* x21 = Gh + static_cast<size_t>(b0 + sz) * d + b0;
      const int64_t tb = static_cast<int64_t>(s2) * sz;  // T entries per pair
      __nv_bfloat16* pa = cplanes;
      __nv_bfloat16* pb = cplanes + cnt * static_cast<int64_t>(s2) * kPlanes * sz;
      // T = L_21 X_11: A rows are the rows of L_21, B rows the columns of X_11
      split7_kernel<false><<<dim3(sz / 64, ceil_div(s2, 64), cnt), 256, 0, s>>>(l21, d, step, s2, sz, pa);
      split7_kernel<true><<<dim3(sz / 64, sz / 64, cnt), 256, 0, s>>>(x11, d, step, sz, sz, pb);
      if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "triangular inverse split");
      rf_status st = launch_f32_product(pa, pb, s2, sz, sz, cnt, T, sz, tb, 1.f, false, false,
                                        cnt * tb, s);
      if (st != RF_OK) return st;
      // X_21 = -X_22 T: A rows are the rows of X_22, B rows the columns of T
      pb = cplanes + cnt * static_cast<int64_t>(s2) * kPlanes * s2;
      split7_kernel<false><<<dim3(s2 / 64, ceil_div(s2, 64), cnt), 256, 0, s>>>(x22, d, step, s2, s2, pa);
      split7_kernel<true><<<dim3(s2 / 64, sz / 64, cnt), 256, 0, s>>>(T, sz, tb, sz, s2, pb);
      if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "triangular inverse split");
      st = launch_f32_product(pa, pb, s2, sz, s2, cnt, x21, d, step, -1.f, false, false,
                              dd - (static_cast<int64_t>(b0 + sz) * d + b0), s);
      if (st != RF_OK) return st;
    }
  }
  // G^-1 = X^T X on the tensor cores: one MN-major Gram product over the stacked bf16
  // planes, [hi; lo; hi] against [lo; hi; hi] (K = 3d, summed in f32 in TMEM).  With
  // 256-column tiles only the pair tiles on and below the diagonal are computed, each
  // stored with its transpose; otherwise every tile is added into the cleared inverse.
  split2_kernel<<<static_cast<unsigned>(ceil_div(dd / 8, 256)), 256, 0, s>>>(Gh, dd, Xs);
  const bool sym = pl.bn == 2 * kBM;
  if (!sym && (e = cudaMemsetAsync(Gi, 0, static_cast<size_t>(dd) * 8, s)) != cudaSuccess)
    return cuda_fail(e, "clearing the inverse");
  rf_status st;
  if ((st = launch_gram(Xs, Xs + dd, nullptr, 0, 3 * d, d, 128, pl.bn, Gi, nullptr, s, sym)) != RF_OK)
    return st;

  split_ginv_kernel<<<static_cast<unsigned>(ceil_div(dd / 8, 256)), 256, 0, s>>>(Gi, d, Bp);
  const int64_t rhs_threads = ceil_div(M, kCentreRows) * (d / 8);
  split_rhs_kernel<<<static_cast<unsigned>(ceil_div(rhs_threads, 256)), 256, 0, s>>>(
      a->C, a->sy, mu64, sc, M, d, Ap);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "operand split launch");

  GemmParams p{};
  p.mode = kModeSolve;
  // K = 3d over two-plane operands: the producer reads A' planes hi, hi, lo against B'
  // planes hi, lo, hi
  p.k_blocks = 3 * d / kBK;
  // stages of two k-blocks, each operand staged by one copy through a rank-4 view
  // {64 k, rows, k-blocks, 1}; on CTA pairs each CTA stages half of the tile's B rows
  const uint64_t krow = static_cast<uint64_t>(2 * d) * 2;
  const uint64_t kbl = static_cast<uint64_t>(2 * d / kBK);
  const uint64_t dA[4] = {kBK, static_cast<uint64_t>(M), kbl, 1};
  const uint64_t sA[3] = {krow, 128, krow * static_cast<uint64_t>(M)};
  const uint32_t bA[4] = {kBK, kBM, 2, 1};
  bool ok = make_tmap_4d(&p.tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Ap, dA, sA, bA,
                         CU_TENSOR_MAP_SWIZZLE_128B);
  const uint64_t dB[4] = {kBK, static_cast<uint64_t>(d), kbl, 1};
  const uint64_t sB[3] = {krow, 128, krow * static_cast<uint64_t>(d)};
  const uint32_t bB[4] = {kBK, static_cast<uint32_t>(pl.bn / 2), 2, 1};
  ok = ok && make_tmap_4d(&p.tmB[0], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Bp, dB, sB, bB,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  p.k2 = 1;
  if (!ok) return fail(RF_ERR_CUDA, "cuTensorMapEncodeTiled failed for the solve GEMM");
  p.m_tiles = static_cast<int32_t>(ceil_div(M, kBM));
  p.bn = pl.bn;
  p.n_tiles = d / pl.bn;
  p.batches = 1;
  p.group_m = 16;
  p.rows = static_cast<int32_t>(M);
  p.col_scale = sc;
  p.mu_x = mu32;
  p.out_f32 = a->A_out_f32;
  p.out_bf16 = static_cast<__nv_bfloat16*>(a->A_out);
  p.bias_part = part;
  p.out_ld = d;
  p.lim_a = M * p.n_tiles;
  p.lim_b = M * d;
  p.err = err;
  const int64_t tiles = static_cast<int64_t>((p.m_tiles + 1) / 2) * p.n_tiles;
  const int pairs = static_cast<int>(tiles < sm_count() / 2 ? tiles : sm_count() / 2);
  if ((e = launch_gemm2(p, pairs, s)) != cudaSuccess) return cuda_fail(e, "solve GEMM launch");
  bias_kernel<<<static_cast<unsigned>((M + 255) / 256), 256, 0, s>>>(a->sy, a->count, part,
                                                                     p.n_tiles, M, a->b_out);
  if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "offset launch");
  return RF_OK;
}

}  // namespace
}  // namespace rf

using namespace rf;

extern "C" size_t ridgefill_fit_workspace_size(const rf_fit_args* a) {
  if (validate_fit(a) != RF_OK) return 0;
  FitPlan pl;
  plan_fit(a, &pl);
  return pl.total > 0 ? pl.total : 256;
}

extern "C" rf_status ridgefill_fit(const rf_fit_args* a, void* workspace, size_t ws_bytes,
                                   void* stream) {
  rf_status st = validate_fit(a);
  if (st != RF_OK) return st;
  const void* sums[] = {a->G, a->C, a->sx, a->sy, a->count};
  for (const void* q : sums)
    if (q == nullptr) return fail(RF_ERR_ARG, "a running-sum pointer is NULL");
  if ((a->flags & RF_FIT_ACCUMULATE) && a->rows > 0 && (a->X == nullptr || a->Y == nullptr))
    return fail(RF_ERR_ARG, "X and Y are required to accumulate");
  if ((a->flags & RF_FIT_SOLVE) &&
      (a->b_out == nullptr || (a->A_out == nullptr && a->A_out_f32 == nullptr)))
    return fail(RF_ERR_ARG, "the solve needs b_out and A_out or A_out_f32");
  const void* dev[] = {a->X, a->Y, a->G, a->C, a->A_out, a->A_out_f32, a->b_out, workspace};
  for (const void* q : dev)
    if (q != nullptr && !aligned16(q)) return fail(RF_ERR_ALIGN, "a device pointer is not 16-byte aligned");
  FitPlan pl;
  plan_fit(a, &pl);
  if (pl.total > 0 && (workspace == nullptr || ws_bytes < pl.total))
    return fail(RF_ERR_WORKSPACE, "workspace needs %zu bytes", pl.total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((st = guards_fill(workspace, pl.lay, s)) != RF_OK) return st;
  if (a->flags & RF_FIT_ACCUMULATE) {
    if ((st = accumulate(a, pl, static_cast<uint8_t*>(workspace), s)) != RF_OK) return st;
  }
  if (a->flags & RF_FIT_SOLVE) {
    if ((st = solve(a, pl, static_cast<uint8_t*>(workspace), s)) != RF_OK) return st;
  }
  return guards_check(workspace, pl.lay, s);
}
