// fill_gemm.cu -- persistent, warp-specialised tcgen05 GEMM with the fill's
// epilogues (RidgeFill, "Training-Free Late-Layer Cache Fill for Faster
// Prefill", sections 2.2 and 2.3).
//
//   map mode : X_hat = H A^T + b for every late layer in one grouped GEMM over
//              the concatenated maps [A_1; ...; A_L] (B operand [L*d_out, d_in]);
//              the epilogue adds b, accumulates per-row sums of squares of the
//              f32 result (one partial per tile), multiplies by the RMSNorm gain
//              and stores bf16 X_hat [L, rows, d_out] through TMA.
//   kv mode  : per layer, X_hat_l W^T for the K and V weights; the epilogue
//              applies the per-row RMS scale rsqrt(ss/d + eps), RoPE on K, and
//              stores bf16 straight into the [layer, kv_head, pos, head_dim] cache.
//   gdn mode : per GDN layer, X_hat_l times [Wk; Wv; Wa|Wb]; the epilogue applies
//              the RMS scale, L2-normalises k per head, and writes f32 k, v and
//              the gates (alpha, beta) for the state kernel.
//
// Roles (256 threads, one CTA per SM): warp 0 issues TMA loads into a
// kStages-deep ring, warp 1 issues tcgen05.mma (M=128, N=bn, K=16) into one of
// two TMEM accumulators, warp 2 owns the TMEM allocation, warps 4-7 drain the
// accumulators (TMEM lane = tile row) while the next tile accumulates.
// Tiles are handed out in raster order by a launch-wide counter: CTA 0's producer takes
// the next tile and passes its index through a small ring in both CTAs' shared memory to
// the other roles, so the pairs that share an operand panel start its tiles together
// (with a fixed round-robin they drift apart over a long launch and re-read the panel).
// rf_gemm2_kernel runs the map, K/V and GDN modes on CTA pairs (M=256); its
// int8-map variant (section 2.2 "Size and cost") adds warp 3 loading int8 codes
// and scales and warps 8-15 dequantising them into the MMA stages.
#include "rf_internal.h"
#include "sm103_ptx.cuh"

namespace rf {

namespace {

constexpr double kTwoPi = 6.283185307179586476925286766559;
constexpr float kTwoPiHi = static_cast<float>(kTwoPi);
constexpr float kTwoPiLo = static_cast<float>(kTwoPi - static_cast<double>(kTwoPiHi));
constexpr float kInvTwoPi = static_cast<float>(1.0 / kTwoPi);

// cos/sin of pos * f where f = fhi + flo (a float pair of the double frequency).
// The product is carried exactly as hi + lo (FMA two-product), reduced by
// 2*pi split in two floats (Cody-Waite), then evaluated by sincosf.
__device__ __forceinline__ void rope_cs(float posf, float fhi, float flo, float& c, float& s) {
  const float ph = posf * fhi;
  const float pe = fmaf(posf, fhi, -ph);
  const float pl = fmaf(posf, flo, pe);
  const float k = rintf(ph * kInvTwoPi);
  float r = fmaf(-k, kTwoPiHi, ph);
  r = fmaf(-k, kTwoPiLo, r);
  r += pl;
  sincosf(r, &s, &c);
}


// Which B segment a tile reads and its MMA width.
struct TileB {
  int seg;   // tensor map index
  int nrow;  // first B row inside the segment
  int bn;    // MMA N
};

__device__ __forceinline__ TileB tile_b(const GemmParams& p, int n) {
  TileB t;
  if (p.mode == kModeMap || p.mode == kModeGram || p.mode == kModeSolve || p.mode == kModeF32) {
    t.seg = 0; t.nrow = n * p.bn; t.bn = p.bn;
  } else if (p.mode == kModeKV) {
    const bool v = n >= p.n_k_tiles;
    t.seg = v ? 1 : 0; t.nrow = (v ? n - p.n_k_tiles : n) * p.bn; t.bn = p.bn;
  } else {
    if (n < p.n_k_tiles) {
      t.seg = 0; t.nrow = n * p.bn; t.bn = p.bn;
    } else if (n < p.n_k_tiles + p.n_v_tiles) {
      t.seg = 1; t.nrow = (n - p.n_k_tiles) * p.bn; t.bn = p.bn;
    } else {
      t.seg = 2; t.nrow = 0; t.bn = 2 * p.gdn_heads;  // Wa rows then Wb rows
    }
  }
  return t;
}

// Write 32 consecutive bf16 of this lane's row into a 64-column, 32-row
// store box laid out with the 128-byte swizzle (16-byte chunk ^= row % 8).
__device__ __forceinline__ void stage32(uint8_t* box, int lane, int col, const uint32_t (&w)[16]) {
  const int ch0 = col >> 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ch = (ch0 + c) ^ (lane & 7);
    *reinterpret_cast<uint4*>(box + lane * 128 + ch * 16) =
        make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
  }
}

__device__ __forceinline__ float f32(uint32_t u) { return __uint_as_float(u); }

// 32 bf16 (16 words) of one row straight to global memory
__device__ __forceinline__ void store32(__nv_bfloat16* dst, const uint32_t (&w)[16]) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < 4; ++c) d[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
}


// ------------------------------------------------------------------ epilogues
__device__ __forceinline__ void map_half(const uint32_t (&r)[32], const float* bp,
                                         const __nv_bfloat16* gp, float& ss, uint32_t (&w)[16]) {
  const float4* b4 = reinterpret_cast<const float4*>(bp);
#pragma unroll
  for (int j = 0; j < 32; j += 4) {
    const float4 bb = __ldg(b4 + j / 4);
    float x0 = f32(r[j]) + bb.x, x1 = f32(r[j + 1]) + bb.y;
    float x2 = f32(r[j + 2]) + bb.z, x3 = f32(r[j + 3]) + bb.w;
    ss = fmaf(x0, x0, ss); ss = fmaf(x1, x1, ss);
    ss = fmaf(x2, x2, ss); ss = fmaf(x3, x3, ss);
    if (gp != nullptr) {
      const uint2 gg = __ldg(reinterpret_cast<const uint2*>(gp + j));
      const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gg.x));
      const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&gg.y));
      x0 *= g01.x; x1 *= g01.y; x2 *= g23.x; x3 *= g23.y;
    }
    w[j / 2] = pack_bf16(x0, x1);
    w[j / 2 + 1] = pack_bf16(x2, x3);
  }
}

// kBoxes: staging boxes per warp (2: double-buffered stores; 1 frees shared memory);
// kDirect: rows listed in p.map_rows, stored one by one (no staging)
template <int kBoxes = 2, bool kDirect = false>
__device__ void epilogue_map(const GemmParams& p, uint32_t tcol, uint8_t* stg, int q, int lane,
                             int m, int n, uint32_t tempty) {
  const int gcol = n * p.bn;
  const int l = p.layer_base + gcol / p.d_out;
  const int j0 = gcol % p.d_out;
  const int row = m * kBM + q * 32 + lane;
  const int nch = p.bn / 64;
  // rows listed by index (exact rows left out of the GEMM) are stored one by one
  constexpr bool direct = kDirect;
  const int orow = direct ? (row < p.rows ? p.map_rows[row] : -1) : row;
  float ss = 0.f;
  for (int c = 0; c < nch; ++c) {
    uint32_t r0[32], r1[32];
    tmem_ld32(tcol + c * 64, r0);
    tmem_ld32(tcol + c * 64 + 32, r1);
    tmem_wait_ld();
    if (c == nch - 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cl(tempty);
    }
    const int col = j0 + c * 64;
    const float* bp = p.bias + static_cast<size_t>(l) * p.d_out + col;
    const __nv_bfloat16* gp =
        p.gain != nullptr ? p.gain + static_cast<size_t>(l) * p.d_out + col : nullptr;
    uint32_t w0[16], w1[16];
    map_half(r0, bp, gp, ss, w0);
    map_half(r1, bp + 32, gp != nullptr ? gp + 32 : nullptr, ss, w1);
    if constexpr (direct) {
      const int64_t o = (static_cast<int64_t>(l) * p.map_ld + orow) * p.d_out + col;
      if (orow >= 0 && orow < p.map_ld && in_bounds(o + 63, p.lim_b, p.err)) {
        __nv_bfloat16* dst = p.map_out + o;
        store32(dst, w0);
        store32(dst + 32, w1);
      }
      continue;
    }
    uint8_t* box = stg + (c % kBoxes) * kOutBoxBytes;
    if (lane == 0) bulk_wait_read<kBoxes - 1>();
    __syncwarp();
    stage32(box, lane, 0, w0);
    stage32(box, lane, 32, w1);
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(&p.tmO[0], smem_u32(box), col, m * kBM + q * 32, l);
      bulk_commit();
    }
  }
  if (row < p.rows && orow >= 0 && (!direct || orow < p.map_ld)) {
    const int64_t o = (static_cast<int64_t>(l) * p.ss_tiles + j0 / p.bn) * p.ss_stride + orow;
    if (in_bounds(o, p.lim_a, p.err)) p.ss_part[o] = ss;
  }
}

__device__ __forceinline__ float row_rms_scale(const GemmParams& p, int l, int row) {
  float ssum = 0.f;
  if (row < p.rows) {
    const float* sp = p.ss_in + static_cast<size_t>(l) * p.ss_tiles * p.ss_stride + row;
    for (int t = 0; t < p.ss_tiles; ++t) ssum += sp[static_cast<size_t>(t) * p.ss_stride];
  }
  return rsqrtf(fmaf(ssum, p.inv_d, p.eps));
}

__device__ void epilogue_kv(const GemmParams& p, uint32_t tcol, uint8_t* stg, int q, int lane,
                            int m, int n, int l, float rs, uint32_t tempty) {
  const int row = m * kBM + q * 32 + lane;
  // rows listed by index (exact prefix rows skipped) are stored one by one
  const bool direct = p.kv_rows != nullptr;
  int pos = p.pos_base + row;
  bool keep = true;
  if (direct) {
    keep = row < p.rows;
    const int idx = keep ? p.kv_rows[row] : 0;
    if (keep && (idx < 0 || idx >= p.kv_hrows)) {
      keep = false;
      atomicCAS(p.err, 0, kErrIndex);
    }
    pos = p.kv_pos0 + idx;
  }
  const float posf = static_cast<float>(pos);
  const bool is_k = n < p.n_k_tiles;
  const int hd = p.head_dim;
  const int half = hd / 2;
  const int hpt = p.bn / hd;
  const int head0 = (is_k ? n : n - p.n_k_tiles) * hpt;
  const CUtensorMap* out = &p.tmO[is_k ? 0 : 1];
  const float* hscale = is_k ? p.k_scale : p.v_scale;
  for (int hh = 0; hh < hpt; ++hh) {
    const uint32_t hc = tcol + hh * hd;
    // the head's rescale factor folds into the row's RMS scale (both multiply the row)
    const float rh = hscale != nullptr ? rs * hscale[l * p.n_kv + head0 + hh] : rs;
    const int64_t drow_off = ((static_cast<int64_t>(l) * p.n_kv + head0 + hh) * p.cache_len + pos) * hd;
    __nv_bfloat16* drow = direct ? p.kv_cache[is_k ? 0 : 1] + drow_off : nullptr;
    const bool keep_h = keep && (!direct || in_bounds(drow_off + hd - 1, p.lim_b, p.err));
    if (!direct && lane == 0) bulk_wait_read<0>();
    __syncwarp();
    if (is_k) {
      for (int i0 = 0; i0 < half; i0 += 32) {
        uint32_t a[32], b[32];
        tmem_ld32(hc + i0, a);
        tmem_ld32(hc + half + i0, b);
        tmem_wait_ld();
        uint32_t w1[16], w2[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
          float c0, s0, c1, s1;
          if (p.rope_tab != nullptr) {  // frequency-major: a warp reads 32 consecutive rows
            const float2 t0 = p.rope_tab[(i0 + j) * p.rope_ld + row];
            const float2 t1 = p.rope_tab[(i0 + j + 1) * p.rope_ld + row];
            c0 = t0.x; s0 = t0.y; c1 = t1.x; s1 = t1.y;
          } else {
            rope_cs(posf, p.inv_freq_hi[i0 + j], p.inv_freq_lo[i0 + j], c0, s0);
            rope_cs(posf, p.inv_freq_hi[i0 + j + 1], p.inv_freq_lo[i0 + j + 1], c1, s1);
          }
          const float xa = f32(a[j]) * rh, ya = f32(b[j]) * rh;
          const float xb = f32(a[j + 1]) * rh, yb = f32(b[j + 1]) * rh;
          w1[j / 2] = pack_bf16(xa * c0 - ya * s0, xb * c1 - yb * s1);
          w2[j / 2] = pack_bf16(ya * c0 + xa * s0, yb * c1 + xb * s1);
        }
        if (direct) {
          if (keep_h) {
            store32(drow + i0, w1);
            store32(drow + half + i0, w2);
          }
        } else {
          stage32(stg + (i0 / 64) * kOutBoxBytes, lane, i0 % 64, w1);
          stage32(stg + ((half + i0) / 64) * kOutBoxBytes, lane, (half + i0) % 64, w2);
        }
      }
    } else {
      for (int c0 = 0; c0 < hd; c0 += 32) {
        uint32_t a[32];
        tmem_ld32(hc + c0, a);
        tmem_wait_ld();
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 32; j += 2) w[j / 2] = pack_bf16(f32(a[j]) * rh, f32(a[j + 1]) * rh);
        if (direct) {
          if (keep_h) store32(drow + c0, w);
        } else {
          stage32(stg + (c0 / 64) * kOutBoxBytes, lane, c0 % 64, w);
        }
      }
    }
    if (hh == hpt - 1) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cl(tempty);
    }
    if (direct) continue;
    fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      for (int bx = 0; bx < hd / 64; ++bx)
        tma_store_3d(out, smem_u32(stg + bx * kOutBoxBytes), bx * 64,
                     p.pos_base + m * kBM + q * 32, l * p.n_kv + head0 + hh);
      bulk_commit();
    }
  }
}

// GDN projections: k (L2-normalised per head) and v as bf16 high parts plus
// bf16 remainders, staged per 64-column half and stored by TMA into the
// [L, H, 2, rows, 128] planes; the gate tile stores sigmoid(alpha), sigmoid(beta).
__device__ void epilogue_gdn(const GemmParams& p, uint32_t tcol, uint8_t* stg, int q, int lane,
                             int m, int n, int l, float rs, uint32_t tempty) {
  const int row = m * kBM + q * 32 + lane;
  const int H = p.gdn_heads;
  if (n < p.n_k_tiles + p.n_v_tiles) {
    const bool is_k = n < p.n_k_tiles;
    const int hpt = p.bn / 128;
    const int head0 = (is_k ? n : n - p.n_k_tiles) * hpt;
    const CUtensorMap* out = &p.tmO[is_k ? 0 : 1];
    for (int hh = 0; hh < hpt; ++hh) {
      const uint32_t hc = tcol + hh * 128;
      float scale = rs;
      if (is_k) {
        float nrm = 0.f;
        for (int c0 = 0; c0 < 128; c0 += 64) {
          uint32_t a[32], b[32];
          tmem_ld32(hc + c0, a);
          tmem_ld32(hc + c0 + 32, b);
          tmem_wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float x = f32(a[j]) * rs, y = f32(b[j]) * rs;
            nrm = fmaf(x, x, nrm);
            nrm = fmaf(y, y, nrm);
          }
        }
        scale = rs * rsqrtf(nrm + p.l2_eps);
      }
      const int plane = (l * H + head0 + hh) * 2;
      for (int bx = 0; bx < 2; ++bx) {
        if (lane == 0) bulk_wait_read<0>();
        __syncwarp();
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t a[32];
          tmem_ld32(hc + 64 * bx + 32 * c, a);
          tmem_wait_ld();
          uint32_t wh[16], wl[16];
#pragma unroll
          for (int j = 0; j < 32; j += 2) {
            const float x0 = f32(a[j]) * scale, x1 = f32(a[j + 1]) * scale;
            const __nv_bfloat162 hv = __floats2bfloat162_rn(x0, x1);
            wh[j / 2] = *reinterpret_cast<const uint32_t*>(&hv);
            wl[j / 2] = pack_bf16(x0 - __low2float(hv), x1 - __high2float(hv));
          }
          stage32(stg, lane, 32 * c, wh);
          stage32(stg + kOutBoxBytes, lane, 32 * c, wl);
        }
        if (hh == hpt - 1 && bx == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cl(tempty);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_3d(out, smem_u32(stg), 64 * bx, m * kBM + q * 32, plane);
          tma_store_3d(out, smem_u32(stg + kOutBoxBytes), 64 * bx, m * kBM + q * 32, plane + 1);
          bulk_commit();
        }
      }
    }
  } else {
    const bool valid = row < p.rows;
    const size_t ra = static_cast<size_t>(p.gdn_rows_alloc);
    // gate tile: columns [0, H) are the alpha logits, [H, 2H) the beta logits
    for (int c0 = 0; c0 < 2 * H; c0 += 32) {
      uint32_t a[32];
      tmem_ld32(tcol + c0, a);  // columns past 2H are read but unused
      tmem_wait_ld();
      if (valid) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int c = c0 + j;
          if (c < 2 * H) {
            const float z = f32(a[j]) * rs;
            const bool is_a = c < H;
            // sigmoid(z): alpha for the first H columns, beta for the next H
            const float val = 1.f / (1.f + expf(-z));
            const int which = is_a ? 0 : 1;
            const int h = is_a ? c : c - H;
            const int64_t o = ((static_cast<int64_t>(l) * 2 + which) * H + h) * ra + row;
            if (in_bounds(o, p.lim_a, p.err)) p.gdn_gate[o] = val;
          }
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive_cl(tempty);
  }
}

// Fit sums: this tile of [X | Y_1 .. Y_L]^T X (f32, summed over the call's rows)
// is added into the caller's f64 sums, one output row per thread.
__device__ void epilogue_gram(const GemmParams& p, uint32_t tcol, int q, int lane, int m, int n,
                              uint32_t tempty) {
  const int r = q * 32 + lane;
  double* dst;
  int64_t o, lim;
  if (m < p.gram_x_tiles) {
    o = static_cast<int64_t>(m * kBM + r) * p.gram_ld + n * p.bn;
    dst = p.gram_G + o;
    lim = p.lim_a;
  } else {
    const int mm = m - p.gram_x_tiles;
    const int l = mm / p.gram_y_tiles_per_layer;
    const int oc = (mm % p.gram_y_tiles_per_layer) * kBM + r;
    o = (static_cast<int64_t>(l) * p.d_out + oc) * p.gram_ld + n * p.bn;
    dst = p.gram_C + o;
    lim = p.lim_b;
  }
  const bool ok = in_bounds(o + p.bn - 1, lim, p.err);
  // symmetric product: a pair tile below the diagonal (column tile n < pair row m / 2) also
  // writes its transpose, column c of this row to row c (lanes: consecutive addresses)
  const bool mirror = p.gram_sym && n != m / 2;
  const int64_t rg = static_cast<int64_t>(m) * kBM + r;
  const bool ok_t = !mirror || in_bounds(static_cast<int64_t>(n * p.bn + p.bn - 1) * p.gram_ld + rg,
                                         p.lim_a, p.err);
  for (int c0 = 0; c0 < p.bn; c0 += 32) {
    uint32_t a[32];
    tmem_ld32(tcol + c0, a);
    tmem_wait_ld();
    if (c0 + 32 == p.bn) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cl(tempty);
    }
    if (!ok) continue;
    double2* d2 = reinterpret_cast<double2*>(dst + c0);
    if (p.gram_sym) {
#pragma unroll
      for (int j = 0; j < 16; ++j)
        d2[j] = make_double2(static_cast<double>(f32(a[2 * j])), static_cast<double>(f32(a[2 * j + 1])));
      if (mirror && ok_t) {
        double* col = p.gram_G + static_cast<int64_t>(n * p.bn + c0) * p.gram_ld + rg;
#pragma unroll
        for (int j = 0; j < 32; ++j) col[static_cast<int64_t>(j) * p.gram_ld] = static_cast<double>(f32(a[j]));
      }
      continue;
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      double2 v = d2[j];
      v.x += static_cast<double>(f32(a[2 * j]));
      v.y += static_cast<double>(f32(a[2 * j + 1]));
      d2[j] = v;
    }
  }
}

// Fit solve: out[o, i] = s_i * acc[o, i] (f32 and/or bf16) and the partial
// sum over this tile's columns of out[o, i] * mu_x[i] (for the offsets).
__device__ void epilogue_solve(const GemmParams& p, uint32_t tcol, int q, int lane, int m, int n,
                               uint32_t tempty) {
  const int o = m * kBM + q * 32 + lane;
  const int c_base = n * p.bn;
  const bool valid = o < p.rows &&
                     in_bounds(static_cast<int64_t>(o) * p.out_ld + c_base + p.bn - 1, p.lim_b, p.err) &&
                     in_bounds(static_cast<int64_t>(o) * p.n_tiles + n, p.lim_a, p.err);
  float part = 0.f;
  for (int c0 = 0; c0 < p.bn; c0 += 32) {
    uint32_t a[32];
    tmem_ld32(tcol + c0, a);
    tmem_wait_ld();
    if (c0 + 32 == p.bn) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cl(tempty);
    }
    if (!valid) continue;
    const int c = c_base + c0;
    float v[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      v[j] = f32(a[j]) * __ldg(p.col_scale + c + j);
      part = fmaf(v[j], __ldg(p.mu_x + c + j), part);
    }
    if (p.out_f32 != nullptr) {
      float4* d4 = reinterpret_cast<float4*>(p.out_f32 + static_cast<size_t>(o) * p.out_ld + c);
#pragma unroll
      for (int j = 0; j < 8; ++j) d4[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    if (p.out_bf16 != nullptr) {
      uint4* d4 = reinterpret_cast<uint4*>(p.out_bf16 + static_cast<size_t>(o) * p.out_ld + c);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        d4[j] = make_uint4(pack_bf16(v[8 * j], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                           pack_bf16(v[8 * j + 4], v[8 * j + 5]), pack_bf16(v[8 * j + 6], v[8 * j + 7]));
    }
  }
  if (valid) p.bias_part[static_cast<size_t>(o) * p.n_tiles + n] = part;
}

// Plain f32 product: out[b, o, c] = alpha acc, plus the stored value when beta_one (rows
// below p.rows, columns below p.cols, a multiple of 32).  The stored values of the next
// 32 columns are loaded while the current ones are written, so two chunks of the row's
// read-modify-write are in flight at a time.
__device__ void epilogue_f32(const GemmParams& p, uint32_t tcol, int q, int lane, int m, int n,
                             int b, uint32_t tempty) {
  const int o = m * kBM + q * 32 + lane;
  const int c_base = n * p.bn;
  const int64_t row0 = static_cast<int64_t>(b) * p.out_bstride + static_cast<int64_t>(o) * p.out_ld;
  // chunk c0 of this row is stored when it lies inside the output (and, in debug builds,
  // inside the buffer)
  auto live = [&](int c0) {
    if (o >= p.rows || c_base + c0 >= p.cols) return false;
    const int64_t e0 = row0 + c_base + c0;
    return in_bounds(e0, p.lim_b, p.err) && in_bounds(e0 + 31, p.lim_b, p.err);
  };
  auto load_old = [&](int c0, bool ok, float4 (&v)[8]) {
    const float4* s4 = reinterpret_cast<const float4*>(p.out_f32 + row0 + c_base + c0);
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = (ok && p.beta_one) ? s4[j] : make_float4(0.f, 0.f, 0.f, 0.f);
  };
  bool ok = live(0);
  float4 cur[8];
  load_old(0, ok, cur);
  for (int c0 = 0; c0 < p.bn; c0 += 32) {
    uint32_t a[32];
    tmem_ld32(tcol + c0, a);
    const bool more = c0 + 32 < p.bn;
    const bool ok_next = more && live(c0 + 32);
    float4 nxt[8];
    load_old(c0 + 32, ok_next, nxt);
    tmem_wait_ld();
    if (!more) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cl(tempty);
    }
    if (ok) {
      float4* d4 = reinterpret_cast<float4*>(p.out_f32 + row0 + c_base + c0);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        d4[j] = make_float4(fmaf(p.alpha, f32(a[4 * j]), cur[j].x), fmaf(p.alpha, f32(a[4 * j + 1]), cur[j].y),
                            fmaf(p.alpha, f32(a[4 * j + 2]), cur[j].z), fmaf(p.alpha, f32(a[4 * j + 3]), cur[j].w));
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
    ok = ok_next;
  }
}

}  // namespace

// ------------------------------------------------------------------ CTA pairs
// Every mode runs on CTA pairs (clusters of 2): the pair computes a 256-row x
// bn-column tile with tcgen05.mma.cta_group::2.  Each CTA stages its 128 rows
// of A and its bn / 2 rows of B (up to 32 KB a stage, six stages); the MMA of CTA 0 reads
// both CTAs' halves and writes each CTA's 128 accumulator rows into its own
// TMEM.  Loads of both CTAs complete on CTA 0's `full` barrier; CTA 0's commits
// release both CTAs' stages and accumulators; both CTAs' epilogues release the
// accumulator on CTA 0's `tempty` barrier.
constexpr int kStages2 = 6;
constexpr int kRing = 4;  // tile ids handed from CTA 0's producer to every other role
constexpr int kHalfBytes = 128 * kBK * 2;  // 128 rows x 64 K of bf16
// Wide Gram tiles (bn = kGramWideCols): the pair accumulates 256 x 512 in both TMEM
// halves with two N = 256 MMAs per K step that share one A stage.  A stage then holds this CTA's A half and
// its two B quarters (48 KB), four stages in the space of the six narrow ones.
constexpr int kWideStageBytes = 3 * kHalfBytes;
constexpr int kStagesWide = 4;
static_assert(kStagesWide * kWideStageBytes <= kStages2 * 2 * kHalfBytes, "wide Gram stages");

namespace {

// Tile t of the pair grid: pair row tile mu (row tiles 2 mu and 2 mu + 1, one per CTA) of
// column tile n, in batch b; grouped raster over pair row tiles.
__device__ __forceinline__ int units_m(const GemmParams& p) { return (p.m_tiles + 1) / 2; }
// Tiles of one launch: pair row tiles x column tiles x batches, or the pair tiles on and below
// the diagonal (lower: n <= mu)
__device__ __forceinline__ int tiles_total(const GemmParams& p) {
  const int u = units_m(p);
  return p.lower ? u * (u + 1) / 2 : u * p.n_tiles * p.batches;
}
__device__ __forceinline__ void decode_unit(int t, const GemmParams& p, int& mu, int& n, int& b) {
  if (p.lower) {  // row-major over the lower triangle: t = mu (mu + 1) / 2 + n
    int r = static_cast<int>((sqrtf(8.f * static_cast<float>(t) + 1.f) - 1.f) * 0.5f);
    while ((r + 1) * (r + 2) / 2 <= t) ++r;
    while (r * (r + 1) / 2 > t) --r;
    mu = r;
    n = t - r * (r + 1) / 2;
    b = 0;
    return;
  }
  const int m_units = units_m(p);
  const int gp = p.group_m / 2 > 0 ? p.group_m / 2 : 1;
  const int per_b = m_units * p.n_tiles;
  b = t / per_b;
  int r = t - b * per_b;
  b += p.batch_base;
  // a shorter first group: the rows it needs land first when the split state streams in
  const int g0 = min(p.group_m0 / 2, m_units);
  if (g0 > 0) {
    if (r < g0 * p.n_tiles) {
      mu = r % g0;
      n = r / g0;
      return;
    }
    r -= g0 * p.n_tiles;
  }
  const int gsz = gp * p.n_tiles;
  const int g = r / gsz;
  const int first = g0 + g * gp;
  const int gm = min(m_units - first, gp);
  const int rr = r - g * gsz;
  mu = first + rr % gm;
  n = rr / gm;
}

// ---- int8 maps.  A third ring ("raw", kRawStages deep) holds this CTA's half of
// each B tile as int8 codes (box {64, bn / 2}, no swizzle: row r at r * 64 bytes)
// and the rows' bf16 scales of the stage's 128-weight group (box {bn / 2}); a
// producer thread (warp 3) fills it by TMA and the converter warps turn it into
// the bf16 stage the MMA reads.
constexpr int kRawK = 2;                  // k-blocks per raw stage (128-byte code rows)
constexpr int kRawRow = kRawK * kBK;      // bytes of one row of codes in a raw stage
constexpr int kRawBytes = 128 * kRawRow;  // int8 codes of a half tile, kRawK k-blocks
constexpr int kRawScaleBytes = 128 * 2;   // bf16 scales of its rows
constexpr int kStagesQ8 = 4;              // bf16 MMA stages with int8 maps
constexpr int kRawStages = 4;
constexpr int kOutBoxesQ8 = 1;            // one store box per epilogue warp (map mode)
constexpr int kConvGroups = 2;            // converter warp groups taking alternate stages
// scale ring padded so the epilogue's 128-byte-swizzled staging stays 1024-byte aligned
constexpr int kRawScaleRegion = (kRawStages * kRawScaleBytes + 1023) / 1024 * 1024;
static_assert(1024 + kStages2 * 2 * kHalfBytes + 4 * kOutWarpBytes + 8 * (2 * kStages2 + 5 + 2 * kRing) +
                      8 + 4 * kRing <=
                  kGemmSmem, "pair GEMM shared memory");
static_assert(1024 + kStagesQ8 * 2 * kHalfBytes + kRawStages * kRawBytes + kRawScaleRegion +
                      4 * kOutBoxesQ8 * kOutBoxBytes + 8 * (2 * kStagesQ8 + 5 + 2 * kRawStages) + 8 <=
                  kGemmSmem, "int8 pair GEMM shared memory");

// bf16(q * s) of 16 codes.  A byte permute turns u = b ^ 0x80 = q + 128 into the
// float 2^15 + u (bits 0x47 : 00 : u : 00); one FMA with c = -(2^15 + 128) s, which
// f32 holds exactly (9 x 8 significant bits), gives (2^15 + u) s + c = q s exactly
// before its rounding, and q s (at most 16 significant bits) survives it; the pack
// rounds once to bf16.
__device__ __forceinline__ void q8_dequant16(uint4 v, float sc, float c, uint32_t (&w)[8]) {
  const uint32_t x[4] = {v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u,
                         v.w ^ 0x80808080u};
  const float2 s2 = make_float2(sc, sc), c2 = make_float2(c, c);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 f01 = __ffma2_rn(make_float2(__uint_as_float(__byte_perm(x[e], 0x47000000u, 0x7504)),
                                              __uint_as_float(__byte_perm(x[e], 0x47000000u, 0x7514))),
                                  s2, c2);
    const float2 f23 = __ffma2_rn(make_float2(__uint_as_float(__byte_perm(x[e], 0x47000000u, 0x7524)),
                                              __uint_as_float(__byte_perm(x[e], 0x47000000u, 0x7534))),
                                  s2, c2);
    w[2 * e] = pack_bf16(f01.x, f01.y);
    w[2 * e + 1] = pack_bf16(f23.x, f23.y);
  }
}

// Converter thread (crow, cch): rows crow + 32 i (i < NR) of the half tile, the 16 codes
// of column chunk cch of the k-block at byte `sub` of each 128-byte code row (the raw
// stage is a 128-byte-swizzled box: chunk c of row r at c ^ (r % 8), so a warp's eight
// rows spread over all banks); writes them as bf16 in the same swizzled layout of a
// {64, rows} box.  All shared-memory loads are issued before any conversion.
template <int NR>
__device__ __forceinline__ void q8_convert(const uint8_t* raw, int sub, const uint8_t* rsc,
                                           uint8_t* sb, int crow, int cch) {
  uint4 v[NR];
  float sc[NR];
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int row = crow + 32 * i;
    v[i] = *reinterpret_cast<const uint4*>(raw + row * kRawRow +
                                           (((sub >> 4) + cch) ^ (row & 7)) * 16);
    sc[i] = __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(rsc + row * 2)) << 16);
  }
#pragma unroll
  for (int i = 0; i < NR; ++i) {
    const int row = crow + 32 * i;
    uint32_t w[8];
    q8_dequant16(v[i], sc[i], -32896.f * sc[i], w);
    uint8_t* rp = sb + row * 128;
    *reinterpret_cast<uint4*>(rp + (((2 * cch) ^ (row & 7)) * 16)) = make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(rp + (((2 * cch + 1) ^ (row & 7)) * 16)) =
        make_uint4(w[4], w[5], w[6], w[7]);
  }
}

}  // namespace

// kQ8: map mode with int8 maps (tmB[0]: codes {d_in, B rows, 1} uint8; tmB[1]: scales
// {d_out, d_in / 128, layers} bf16).  Warps 8-11 dequantise this CTA's B half of each
// stage into shared memory and arrive on CTA 0's `full` barrier (released at cluster
// scope; the MMA acquires at cluster scope before reading both halves).
template <bool kQ8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kQ8 ? kGemmThreadsQ8 : kGemmThreads, 1)
    rf_gemm2_kernel(const __grid_constant__ GemmParams p) {
  constexpr int kS = kQ8 ? kStagesQ8 : kStages2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem;
  uint8_t* sB = sA + kS * kHalfBytes;
  uint8_t* sRaw = sB + kS * kHalfBytes;                           // kQ8 only
  uint8_t* sRawScale = sRaw + (kQ8 ? kRawStages * kRawBytes : 0);  // kQ8 only
  uint8_t* stg_all = sRawScale + (kQ8 ? kRawScaleRegion : 0);
  constexpr int kStgWarpBytes = kQ8 ? kOutBoxesQ8 * kOutBoxBytes : kOutWarpBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(stg_all + 4 * kStgWarpBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + kS;
  uint64_t* tfull = bars + 2 * kS;
  uint64_t* tempty = tfull + 2;
  uint64_t* fin = tempty + 2;
  uint64_t* ring_full = fin + 1;                           // tile-id ring (both CTAs)
  uint64_t* ring_empty = ring_full + kRing;                // CTA 0's only
  uint64_t* raw_full = ring_empty + kRing;                 // kQ8 only
  uint64_t* raw_empty = raw_full + (kQ8 ? kRawStages : 0);  // kQ8 only
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(raw_empty + (kQ8 ? kRawStages : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* ring = reinterpret_cast<int*>(tmem_slot + 2);
  // tiles in the order a launch-wide counter hands them out (pairs that share an operand
  // panel then run its tiles together); the int8 kernel keeps the static order
  constexpr bool kDyn = !kQ8;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();  // position in the CTA pair
  const int cl = blockIdx.x / 2, ncl = gridDim.x / 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kS; ++s) {
      // both CTAs' producers (+ both CTAs' four converter warps)
      mbar_init(&full[s], kQ8 ? 10 : 2);
      mbar_init(&empty[s], 1);  // the commit of the pair's MMA CTA
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);  // four epilogue warps in each CTA
    }
    mbar_init(fin, 1);
    for (int r = 0; r < kRing; ++r) {
      mbar_init(&ring_full[r], 1);    // CTA 0's producer
      mbar_init(&ring_empty[r], 10);  // MMA, CTA 1's producer, four epilogue warps in each CTA
    }
    if (kQ8) {
      for (int s = 0; s < kRawStages; ++s) {
        mbar_init(&raw_full[s], 1);   // this CTA's raw producer (+ its copies' bytes)
        mbar_init(&raw_empty[s], 4 * kRawK);  // four converter warps per k-block of the stage
      }
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch(&p.tmA);
    tma_prefetch(&p.tmB[0]);
    if (!kQ8 && p.mode == kModeGram && p.m_tiles > p.gram_x_tiles) tma_prefetch(&p.tmA2);
    if (kQ8 || p.mode == kModeKV || p.mode == kModeGdnProj) tma_prefetch(&p.tmB[1]);
    if (!kQ8 && p.mode == kModeGdnProj) {
      tma_prefetch(&p.tmB[2]);
      tma_prefetch(&p.tmB[3]);
    }
  }
  if (warp == 2) {
    tmem_alloc_pair(tmem_slot, 512);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers are initialised and their TMEM allocated
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = tiles_total(p);
  const uint32_t full0 = cluster_addr(smem_u32(full), 0);
  const uint32_t tempty0 = cluster_addr(smem_u32(tempty), 0);
  const uint32_t ring_empty0 = cluster_addr(smem_u32(ring_empty), 0);
  // tile of the it-th turn of this pair: the static order, or the ring (every role but CTA
  // 0's producer, which fills it); -1 after the last tile, -2 when a wait gave up
  auto tile_of = [&](int it, bool all_lanes, int site) -> int {
    if constexpr (!kDyn) {
      const int t = cl + it * ncl;
      return t < total ? t : -1;
    } else {
      const int slot = it % kRing;
      if (!mbar_wait_acq_cluster(&ring_full[slot], static_cast<uint32_t>(it / kRing) & 1u,
                                 abort_flag, p.err, site))
        return -2;
      const int t = *reinterpret_cast<volatile int*>(&ring[slot]);
      if (all_lanes) __syncwarp();
      if (!all_lanes || lane == 0) {
        if (rank == 0) mbar_arrive(&ring_empty[slot]);
        else mbar_arrive_cl(ring_empty0 + 8 * slot);
      }
      return t;
    }
  };
  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer of this CTA's halves
      const bool wide = !kQ8 && p.mode == kModeGram && p.bn == kGramWideCols;
      const bool k2 = !kQ8 && p.k2 != 0;
      const uint32_t nst = wide ? kStagesWide : (k2 ? kS / 2 : kS);
      uint32_t stage = 0, phase = 0;
      int issued[kS];
      for (int s = 0; s < kS; ++s) issued[s] = -1;
      bool ok = true;
      int h_seen = -1;  // last split-state row group known to be in device memory
      for (int it = 0; ok; ++it) {
        int t;
        if (kDyn && rank == 0) {
          // take the next tile and hand it to the other roles of both CTAs
          const int slot = it % kRing;
          if (it >= kRing &&
              !mbar_wait_acq_cluster(&ring_empty[slot], (static_cast<uint32_t>(it / kRing) & 1u) ^ 1u,
                                     abort_flag, p.err, kErrProducer)) {
            ok = false;
            break;
          }
          t = atomicAdd(p.tile_ctr, 1);
          if (t >= total) t = -1;
          ring[slot] = t;
          st_cluster_u32(cluster_addr(smem_u32(&ring[slot]), 1), static_cast<uint32_t>(t));
          mbar_arrive(&ring_full[slot]);
          mbar_arrive_cl(cluster_addr(smem_u32(&ring_full[slot]), 1));
        } else {
          t = tile_of(it, false, kErrProducer);
        }
        if (t < 0) {
          if (t == -2) ok = false;
          break;
        }
        int mu, n, b;
        decode_unit(t, p, mu, n, b);
        const int m = 2 * mu + static_cast<int>(rank);
        const TileB tb = tile_b(p, n);
        if (p.h_ready != nullptr && m * kBM < p.rows) {
          const int hr = p.h_row_base + m * kBM;
          const int g = hr < p.h_first_rows ? 0 : 1 + (hr - p.h_first_rows) / p.h_group_rows;
          if (g != h_seen) {
            if (!flag_wait(p.h_ready + g, p.h_gen, abort_flag, p.err, kErrHostRows)) break;
            fence_acq_rel_gpu();
            h_seen = g;
          }
        }
        for (int kb = 0; kb < p.k_blocks; kb += k2 ? 2 : 1) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.err, kErrProducer)) {
            ok = false;
            break;
          }
          const uint32_t fb = full0 + 8 * stage;
          const int half = tb.bn / 2;  // B rows (tile columns) this CTA stages
          const uint32_t tx = kQ8 ? kHalfBytes : (k2 ? 2 : 1) * (kHalfBytes + half * kBK * 2);
          if (rank == 0) mbar_expect_tx(&full[stage], tx);
          else mbar_expect_tx_cl(fb, tx);
          if (k2) {
            // two k-blocks of A and of this CTA's B half, one copy each (rank-4 views
            // {64 k, rows, k-blocks, batch}); solve mode: K = 3 planes of d over two-plane
            // operands, A' hi, hi, lo against B' hi, lo, hi (k-block kb of the product reads
            // A' k-block ka, B' k-block kbb; d / 64 is even, so no pair straddles two planes)
            int ka = kb, kbb = kb;
            if (p.mode == kModeSolve) {
              const int np = p.k_blocks / 3;
              ka = kb >= np ? kb - np : kb;
              kbb = kb >= 2 * np ? kb - 2 * np : kb;
            }
            tma_load_4d_pair(smem_u32(sA + stage * 2 * kHalfBytes), &p.tmA, fb, 0, m * kBM, ka, b);
            if (tb.seg < 2)
              tma_load_4d_pair(smem_u32(sB + stage * 2 * kHalfBytes), &p.tmB[tb.seg], fb, 0,
                               tb.nrow + half * static_cast<int>(rank), kbb, b);
            else  // GDN gate tile: CTA 0 stages the alpha weights, CTA 1 the beta weights
              tma_load_4d_pair(smem_u32(sB + stage * 2 * kHalfBytes), &p.tmB[2 + rank], fb, 0, 0,
                               kb, b);
          } else if (!kQ8 && p.mode == kModeGram) {
            // MN-major operands: 64-wide column blocks of [rows, width] arrays, 64 rows of K;
            // A: this CTA's 128 columns of [X | Y_1 .. Y_L], B: its half of the X columns of
            // each N <= 256 MMA (a wide tile's second MMA starts 256 columns on)
            uint8_t* adst = wide ? sA + stage * kWideStageBytes : sA + stage * kHalfBytes;
            uint8_t* bdst = wide ? adst + kHalfBytes : sB + stage * kHalfBytes;
            const int nmma = tb.bn < 256 ? tb.bn : 256;
            const int bpm = nmma / 128;  // 64-column boxes per MMA in this CTA's half
            // (the empty second half of an odd last row tile reads past X: zero fill)
            if (wide) {
              // rank-4 views {64 columns, rows, column blocks, layers}: one copy stages two
              // 64-column blocks (16 KB), the A half in one, each MMA's B half in one
              if (m < p.gram_x_tiles || m >= p.m_tiles) {
                tma_load_4d_pair(smem_u32(adst), &p.tmA, fb, 0, kb * kBK, m * (kBM / 64), 0);
              } else {
                const int mm = m - p.gram_x_tiles;
                tma_load_4d_pair(smem_u32(adst), &p.tmA2, fb, 0, kb * kBK,
                                 (mm % p.gram_y_tiles_per_layer) * (kBM / 64),
                                 mm / p.gram_y_tiles_per_layer);
              }
              for (int jj = 0; jj < 2; ++jj)
                tma_load_4d_pair(smem_u32(bdst + jj * 16384), &p.tmB[0], fb, 0, kb * kBK,
                                 (tb.nrow + 256 * jj + 128 * static_cast<int>(rank)) / 64, 0);
            } else if (m < p.gram_x_tiles || m >= p.m_tiles) {
              for (int j = 0; j < kBM / 64; ++j)
                tma_load_3d_pair(smem_u32(adst + j * 8192), &p.tmA, fb, m * kBM + 64 * j,
                                 kb * kBK, 0);
            } else {
              const int mm = m - p.gram_x_tiles;
              const int l = mm / p.gram_y_tiles_per_layer;
              const int m0 = (mm % p.gram_y_tiles_per_layer) * kBM;
              for (int j = 0; j < kBM / 64; ++j)
                tma_load_3d_pair(smem_u32(adst + j * 8192), &p.tmA2, fb, m0 + 64 * j, kb * kBK, l);
            }
            for (int j = 0; j < (wide ? 0 : half / 64); ++j)
              tma_load_3d_pair(smem_u32(bdst + j * 8192), &p.tmB[0], fb,
                               tb.nrow + (j / bpm) * nmma + (nmma / 2) * static_cast<int>(rank) +
                                   64 * (j % bpm),
                               kb * kBK, 0);
          } else {
            // solve mode: K = 3 planes of d over two-plane operands, A' hi, hi, lo against
            // B' hi, lo, hi (k-block kb of the product reads A' k-block ka, B' k-block kbb)
            const int np = p.k_blocks / 3;
            const bool sv = !kQ8 && p.mode == kModeSolve;
            const int ka = sv && kb >= np ? kb - np : kb;
            tma_load_3d_pair(smem_u32(sA + stage * kHalfBytes), &p.tmA, fb, ka * kBK, m * kBM, b);
            if (sv) {
              const int kbb = kb >= 2 * np ? kb - 2 * np : kb;
              tma_load_3d_pair(smem_u32(sB + stage * kHalfBytes), &p.tmB[0], fb, kbb * kBK,
                               tb.nrow + half * static_cast<int>(rank), b);
            }
          }
          if (kQ8 || k2 || p.mode == kModeGram || p.mode == kModeSolve) {
            // B comes from the converter warps, or was loaded above
          } else if (tb.seg < 2)
            tma_load_3d_pair(smem_u32(sB + stage * kHalfBytes), &p.tmB[tb.seg], fb, kb * kBK,
                             tb.nrow + half * static_cast<int>(rank), b);
          else  // GDN gate tile: CTA 0 stages the alpha weights, CTA 1 the beta weights
            tma_load_3d_pair(smem_u32(sB + stage * kHalfBytes), &p.tmB[2 + rank], fb, kb * kBK, 0, b);
          issued[stage] = static_cast<int>(phase);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      if (!ok && rank == 0)  // let the copies counted on this CTA's barriers land
        for (int s = 0; s < kS; ++s)
          if (issued[s] >= 0) mbar_drain(&full[s], static_cast<uint32_t>(issued[s]));
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ---------------- MMA issuer (CTA 0 only)
      const bool wide = !kQ8 && p.mode == kModeGram && p.bn == kGramWideCols;
      const bool k2 = !kQ8 && p.k2 != 0;
      const uint32_t nst = wide ? kStagesWide : (k2 ? kS / 2 : kS);
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int it = 0; ok; ++it) {
        const int t = tile_of(it, false, kErrMma);
        if (t < 0) break;
        int mu, n, b;
        decode_unit(t, p, mu, n, b);
        const TileB tb = tile_b(p, n);
        const bool mn = !kQ8 && p.mode == kModeGram;
        const uint32_t idesc =
            idesc_bf16_f32(2 * kBM, wide ? 256 : tb.bn) | (mn ? (3u << 15) : 0u);
        // a wide tile takes both accumulators: one buffer, its phase flips every tile
        const int acc = wide ? 0 : it & 1;
        const uint32_t acc_phase = wide ? it & 1 : (it >> 1) & 1;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.err, kErrMma)) break;
        tc_fence_after();
        const uint32_t dt = tmem_base + acc * kBNMax;
        for (int kb = 0; kb < p.k_blocks; kb += k2 ? 2 : 1) {
          const bool got = kQ8 ? mbar_wait_acq_cluster(&full[stage], phase, abort_flag, p.err, kErrMma)
                               : mbar_wait(&full[stage], phase, abort_flag, p.err, kErrMma);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (k2) {
            // two k-blocks: A's 16 KB apart, B's (bn / 2 rows of 128 bytes) bn * 64 bytes apart
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sA + (2 * stage + h) * kHalfBytes));
              const uint64_t bd = sdesc_kmajor_sw128(
                  smem_u32(sB + 2 * stage * kHalfBytes + h * (tb.bn / 2) * 128));
#pragma unroll
              for (int k = 0; k < kBK / 16; ++k)
                mma_bf16_pair(dt, ad + 2 * k, bd + 2 * k, idesc, (kb | h | k) != 0 ? 1u : 0u);
            }
          } else if (!mn) {
            const uint64_t ad = sdesc_kmajor_sw128(smem_u32(sA + stage * kHalfBytes));
            const uint64_t bd = sdesc_kmajor_sw128(smem_u32(sB + stage * kHalfBytes));
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)
              mma_bf16_pair(dt, ad + 2 * k, bd + 2 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          } else if (!wide) {
            // MN-major: 64-element column blocks 8 KB apart, K rows 128 B apart
            const uint64_t ad = sdesc_mnmajor_sw128(smem_u32(sA + stage * kHalfBytes), 8192);
            const uint64_t bd = sdesc_mnmajor_sw128(smem_u32(sB + stage * kHalfBytes), 8192);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)  // advance 16 K rows (2048 B)
              mma_bf16_pair(dt, ad + 128 * k, bd + 128 * k, idesc, (kb | k) != 0 ? 1u : 0u);
          } else {
            // wide: the same A stage against the two B quarters, into TMEM columns 0-255
            // and 256-511
            const uint32_t sa = smem_u32(sA + stage * kWideStageBytes);
            const uint64_t ad = sdesc_mnmajor_sw128(sa, 8192);
            const uint64_t bd0 = sdesc_mnmajor_sw128(sa + kHalfBytes, 8192);
            const uint64_t bd1 = sdesc_mnmajor_sw128(sa + 2 * kHalfBytes, 8192);
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              const uint32_t accum = (kb | k) != 0 ? 1u : 0u;
              mma_bf16_pair(dt, ad + 128 * k, bd0 + 128 * k, idesc, accum);
              mma_bf16_pair(dt + 256, ad + 128 * k, bd1 + 128 * k, idesc, accum);
            }
          }
          // frees the stage in both CTAs
          mma_commit_pair(&empty[stage], 0x3);
          if (++stage == nst) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (ok) mma_commit_pair(&tfull[acc], 0x3);
      }
      // every MMA issued has finished before TMEM is released
      mma_commit_pair(fin, 0x1);
      mbar_drain(fin, 0);
    }
  } else if (kQ8 && warp == 3) {
    if (lane == 0) {
      // ---------------- int8 producer: this CTA's codes and scales of every stage
      uint32_t rs = 0, rphase = 0;
      int issued[kRawStages];
      for (int s = 0; s < kRawStages; ++s) issued[s] = -1;
      bool ok = true;
      for (int t = cl; t < total && ok; t += ncl) {
        int mu, n, b;
        decode_unit(t, p, mu, n, b);
        const TileB tb = tile_b(p, n);
        const int half = tb.bn / 2;
        const int brow0 = tb.nrow + half * static_cast<int>(rank);
        const int l = brow0 / p.d_out, j0 = brow0 - l * p.d_out;
        for (int kb = 0; kb < p.k_blocks; kb += kRawK) {  // k_blocks is even (d_in % 128 == 0)
          if (!mbar_wait(&raw_empty[rs], rphase ^ 1, abort_flag, p.err, kErrProducer)) {
            ok = false;
            break;
          }
          mbar_expect_tx(&raw_full[rs], half * (kRawRow + 2));
          tma_load_3d(smem_u32(sRaw + rs * kRawBytes), &p.tmB[0], &raw_full[rs], kb * kBK, brow0, 0);
          tma_load_3d(smem_u32(sRawScale + rs * kRawScaleBytes), &p.tmB[1], &raw_full[rs], j0,
                      (kb * kBK) / kQ8Group, l);
          issued[rs] = static_cast<int>(rphase);
          if (++rs == kRawStages) {
            rs = 0;
            rphase ^= 1;
          }
        }
      }
      if (!ok)
        for (int s = 0; s < kRawStages; ++s)
          if (issued[s] >= 0) mbar_drain(&raw_full[s], static_cast<uint32_t>(issued[s]));
    }
  } else if (warp >= 4 && warp < 8) {
    // ---------------- epilogue warpgroup (both CTAs)
    const int q = warp - 4;
    uint8_t* stg = stg_all + q * kStgWarpBytes;
    for (int it = 0;; ++it) {
      const int t = tile_of(it, true, kErrEpilogue);
      if (t < 0) break;
      int mu, n, b;
      decode_unit(t, p, mu, n, b);
      const int m = 2 * mu + static_cast<int>(rank);
      const bool wide = !kQ8 && p.mode == kModeGram && p.bn == kGramWideCols;
      const int acc = wide ? 0 : it & 1;
      const uint32_t acc_phase = wide ? it & 1 : (it >> 1) & 1;
      float rs = 1.f;
      if (!kQ8 && (p.mode == kModeKV || p.mode == kModeGdnProj))
        rs = row_rms_scale(p, b, m * kBM + q * 32 + lane);
      if (!mbar_wait(&tfull[acc], acc_phase, abort_flag, p.err, kErrEpilogue)) break;
      tc_fence_after();
      const uint32_t tcol = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kBNMax;
      if (m >= p.m_tiles) {  // the second half of a last, odd row tile: nothing to store
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cl(tempty0 + 8 * acc);
      } else if (kQ8) {
        epilogue_map<kOutBoxesQ8>(p, tcol, stg, q, lane, m, n, tempty0 + 8 * acc);
      } else if (p.mode == kModeMap) {
        if (p.map_rows != nullptr) epilogue_map<2, true>(p, tcol, stg, q, lane, m, n, tempty0 + 8 * acc);
        else epilogue_map(p, tcol, stg, q, lane, m, n, tempty0 + 8 * acc);
      } else if (p.mode == kModeKV) {
        epilogue_kv(p, tcol, stg, q, lane, m, n, b, rs, tempty0 + 8 * acc);
      } else if (p.mode == kModeGram) {
        epilogue_gram(p, tcol, q, lane, m, n, tempty0 + 8 * acc);
      } else if (p.mode == kModeSolve) {
        epilogue_solve(p, tcol, q, lane, m, n, tempty0 + 8 * acc);
      } else if (p.mode == kModeF32) {
        epilogue_f32(p, tcol, q, lane, m, n, b, tempty0 + 8 * acc);
      } else {
        epilogue_gdn(p, tcol, stg, q, lane, m, n, b, rs, tempty0 + 8 * acc);
      }
    }
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
  } else if (kQ8 && warp >= 8) {
    // ---------------- int8 converters: raw stage -> bf16 B stage of this CTA.  Two
    // groups of four warps take alternate stages, so one group's waits and fences
    // overlap the other's conversion.
    const int cg = (warp - 8) >> 2;
    const int ct = static_cast<int>(threadIdx.x) - 256 - 128 * cg;
    const int crow = ct >> 2, cch = ct & 3;
    const int nr = p.bn / 64;  // rows of the half tile / 32 (map mode: one tile width)
    const int my_tiles = cl < total ? (total - cl + ncl - 1) / ncl : 0;
    const int jobs = my_tiles * p.k_blocks;
    for (int j = cg; j < jobs; j += kConvGroups) {
      const uint32_t stage = static_cast<uint32_t>(j % kS), phase = static_cast<uint32_t>(j / kS) & 1u;
      const int rj = j / kRawK;  // raw stage job: kRawK consecutive k-blocks share one
      const uint32_t rs = static_cast<uint32_t>(rj % kRawStages);
      const uint32_t rphase = static_cast<uint32_t>(rj / kRawStages) & 1u;
      const int sub = (j % kRawK) * kBK;  // byte offset of this k-block inside each code row
      if (!mbar_wait(&raw_full[rs], rphase, abort_flag, p.err, kErrConvert) ||
          !mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.err, kErrConvert))
        break;
      if (nr == 4)
        q8_convert<4>(sRaw + rs * kRawBytes, sub, sRawScale + rs * kRawScaleBytes,
                      sB + stage * kHalfBytes, crow, cch);
      else
        q8_convert<2>(sRaw + rs * kRawBytes, sub, sRawScale + rs * kRawScaleBytes,
                      sB + stage * kHalfBytes, crow, cch);
      fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0) {
          mbar_arrive(&full[stage]);  // release at CTA scope; the MMA issuer is in this CTA
        } else {
          // this CTA's shared-memory writes, released to the peer's MMA issuer
          fence_release_smem_cluster();
          mbar_arrive_relaxed_cl(full0 + 8 * stage);
        }
        mbar_arrive(&raw_empty[rs]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no pair MMA, commit or remote arrival targets either CTA any more
  if (warp == 2) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, 512);
  }
}

cudaError_t launch_gemm2(const GemmParams& p, int pairs, cudaStream_t stream, int* ctr) {
  // set on every launch: the attribute belongs to the current device, and the call is
  // cheap next to the kernel
  cudaError_t e = cudaFuncSetAttribute(rf_gemm2_kernel<false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  GemmParams q = p;
  if (ctr != nullptr) {
    q.tile_ctr = ctr;
  } else {
    q.tile_ctr = tile_counter_slot();
    if (q.tile_ctr == nullptr) return cudaErrorInvalidSymbol;
    if ((e = cudaMemsetAsync(q.tile_ctr, 0, sizeof(int), stream)) != cudaSuccess) return e;
  }
  rf_gemm2_kernel<false><<<2 * pairs, kGemmThreads, kGemmSmem, stream>>>(q);
  return cudaGetLastError();
}

cudaError_t launch_gemm2_q8(const GemmParams& p, int pairs, cudaStream_t stream) {
  // set on every launch: the attribute belongs to the current device, and the call is
  // cheap next to the kernel
  cudaError_t e = cudaFuncSetAttribute(rf_gemm2_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  rf_gemm2_kernel<true><<<2 * pairs, kGemmThreadsQ8, kGemmSmem, stream>>>(p);
  return cudaGetLastError();
}


}  // namespace rf
