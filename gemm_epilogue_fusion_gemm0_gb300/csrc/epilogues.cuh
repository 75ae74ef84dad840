// epilogues.cuh -- the epilogue programs of the chain, one policy class each.
//
// Each thread owns one row of the 128 x 256 fp32 accumulator tile (its TMEM
// lane) and one 128-column half of it (TileCtx::half; two epilogue warps share
// each lane quadrant), walked in 32-column chunks (tcgen05.ld 32x32b.x32).  So
// every row reduction below is a plain per-thread sum that leaves one partial
// per (row, half tile): no shuffles, no atomics, and a fixed summation order
// (bit-reproducible results).  Partials are stored [2 * nt][M], index
// 2 * nb + half.
//
// The primitives used are the method's tile-local ones (CODA blog,
// blog.hotdry.top, section "五类 Epilogue 原语"): an elementwise map (residual
// add), a rank-1 vector broadcast (gamma, the per-row r), rank-2 tile loads and
// stores (z, h), and a partial tile reduction finished by a small pass
// (per-tile sums of squares / of grad_h2 * gamma * h).
#pragma once

#include <cuda_fp8.h>

#include "gemm.cuh"

namespace coda {

struct Chunk8 {
  uint32_t w[4];
};

// Column mapping of a policy: how many 256-column accumulator tiles cover the
// output, and where the producer fetches the j-th 64-column chunk (j = 0..3)
// of an MN-major B tile.  The default is the plain contiguous tiling.
struct EpiDefaultCols {
  static __host__ __device__ __forceinline__ int num_col_tiles(int N) { return (N + kBN - 1) / kBN; }
  static __device__ __forceinline__ int b_col(int nb, int j, int /*N*/) { return nb * kBN + 64 * j; }
};

// Loads the four 8-element groups [n0 + 8q, n0 + 8q + 8) of row `rowp` (q = 0..3);
// groups at or past `limit` (or all of them when !ok) read as zeros.  Issued for
// the next 32-column chunk before the current one is processed, so global-load
// latency overlaps the epilogue arithmetic.
__device__ __forceinline__ void ldg_chunk(const __nv_bfloat16* rowp, int n0, int limit, bool ok,
                                          Chunk8 (&out)[4]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int n = n0 + q * 8;
    if (ok && n < limit) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(rowp + n));
      out[q] = Chunk8{{v.x, v.y, v.z, v.w}};
    } else {
      out[q] = Chunk8{{0u, 0u, 0u, 0u}};
    }
  }
}

// r[m] = rsqrt(sum of the row's h^2 partials / d + eps), summed in the same
// order and with the same expression as the stand-alone row-reduction kernel,
// so the folded and the separate forms give bit-identical r.
struct FoldedRowReduce {
  const float* part;  // [n_part][M] partial sums of h^2; null: r is read from `r`
  int n_part;
  int d;
  float eps;
  float* r_out;       // written by the tiles of column block 0
};

__device__ __forceinline__ float folded_rsqrt(const FoldedRowReduce& f, int m, int M) {
  float s = 0.f;
  for (int t = 0; t < f.n_part; ++t) s += __ldcg(f.part + static_cast<size_t>(t) * M + m);
  return rsqrtf(s / static_cast<float>(f.d) + f.eps);
}

constexpr int kHalfCols = kBN / 2;        // accumulator columns per epilogue thread
constexpr int kHalfChunks = kHalfCols / 32;

__device__ __forceinline__ size_t partial_index(const TileCtx& c, int m) {
  return static_cast<size_t>(2 * c.nb + c.half) * c.M + m;
}

__device__ __forceinline__ Chunk8 ldg8(const __nv_bfloat16* p) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(p));
  return Chunk8{{v.x, v.y, v.z, v.w}};
}

__device__ __forceinline__ void stg8(__nv_bfloat16* p, const uint32_t (&w)[4]) {
  *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// ---------------------------------------------------------------------------
// GEMM0 epilogue (step 1 of the reparameterisation, CODA blog section
// "GEMM-Residual-RMSNorm-GEMM 重参数化"): residual add, gamma scaling and the
// tile-local partial sum of squares.
//   h  = acc + z                (fp32)          -> h_out  bf16
//   hg = h * gamma              (fp32)          -> hg_out bf16 (GEMM1's A operand)
//   part[2 nb + half][m] = sum over the half tile's columns of h^2 (fp32, before rounding)
// With hg_out == nullptr and part == nullptr it is the plain residual-add
// epilogue of the unfused reference sequence.
// ---------------------------------------------------------------------------
struct EpiResidualGammaSumsq : EpiDefaultCols {
  struct Params {
    const __nv_bfloat16* z;
    const __nv_bfloat16* gamma;
    __nv_bfloat16* h_out;
    __nv_bfloat16* hg_out;  // may be null (unfused sequence)
    float* part;            // [2 * nt][M], may be null (unfused sequence)
  };

  static __device__ __forceinline__ void apply(const Params& p, const WaitCtl&, const TileCtx& c) {
    const int m = c.mb * kBM + c.row;
    const bool row_ok = m < c.M;
    const size_t rowoff = static_cast<size_t>(row_ok ? m : 0) * c.N;
    const bool fused = p.hg_out != nullptr;
    float ss = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < kHalfChunks; ++ch) {
      const int col = c.half * kHalfCols + ch * 32;
      const int n0 = c.nb * kBN + col;
      uint32_t v[32];
      tmem_ld32(c.taddr + col, v);
      tmem_ld_wait(v);
      if (row_ok) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int n = n0 + g * 8;
          if (n < c.N) {
            const Chunk8 zz = ldg8(p.z + rowoff + n);
            const Chunk8 gg = ldg8(p.gamma + n);
            uint32_t hw[4], hgw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float h0 = __uint_as_float(v[g * 8 + 2 * e]) + bf16lo(zz.w[e]);
              const float h1 = __uint_as_float(v[g * 8 + 2 * e + 1]) + bf16hi(zz.w[e]);
              ss = fmaf(h0, h0, ss);
              ss = fmaf(h1, h1, ss);
              hw[e] = pack_bf16x2(h0, h1);
              hgw[e] = pack_bf16x2(h0 * bf16lo(gg.w[e]), h1 * bf16hi(gg.w[e]));
            }
            stg8(p.h_out + rowoff + n, hw);
            if (fused) stg8(p.hg_out + rowoff + n, hgw);
          }
        }
      }
    }
    if (row_ok && p.part != nullptr) p.part[partial_index(c, m)] = ss;
  }
};

// ---------------------------------------------------------------------------
// Plain fp32 store (weight gradients): out[m, n] = acc.
// ---------------------------------------------------------------------------
struct EpiStoreF32 : EpiDefaultCols {
  struct Params {
    float* out;  // [M, N] row-major
  };

  static __device__ __forceinline__ void apply(const Params& p, const WaitCtl&, const TileCtx& c) {
    const int m = c.mb * kBM + c.row;
    const bool row_ok = m < c.M;
    const size_t rowoff = static_cast<size_t>(row_ok ? m : 0) * c.N;
#pragma unroll 1
    for (int ch = 0; ch < kHalfChunks; ++ch) {
      const int col = c.half * kHalfCols + ch * 32;
      uint32_t v[32];
      tmem_ld32(c.taddr + col, v);
      tmem_ld_wait(v);
      const int n0 = c.nb * kBN + col;
      if (row_ok) {
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const int n = n0 + g * 4;
          if (n < c.N)
            *reinterpret_cast<uint4*>(p.out + rowoff + n) =
                make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// GEMM1 epilogue (step 3): y = r[m] * acc, the row scale applied after the
// second GEMM.  With r == nullptr it is the plain store of the unfused
// reference sequence.
// ---------------------------------------------------------------------------
struct EpiRowScale : EpiDefaultCols {
  struct Params {
    const float* r;  // [M], may be null (scale 1)
    __nv_bfloat16* y_out;
    FoldedRowReduce fold;  // fold.part != null: r computed here from the partials
  };

  static __device__ __forceinline__ void apply(const Params& p, const WaitCtl&, const TileCtx& c) {
    const int m = c.mb * kBM + c.row;
    const bool row_ok = m < c.M;
    const size_t rowoff = static_cast<size_t>(row_ok ? m : 0) * c.N;
    float rr = 1.f;
    if (row_ok && p.fold.part != nullptr) {
      rr = folded_rsqrt(p.fold, m, c.M);
      if (c.nb == 0 && c.half == 0) p.fold.r_out[m] = rr;
    } else if (row_ok && p.r != nullptr) {
      rr = __ldg(p.r + m);
    }
#pragma unroll 1
    for (int ch = 0; ch < kHalfChunks; ++ch) {
      const int col = c.half * kHalfCols + ch * 32;
      uint32_t v[32];
      tmem_ld32(c.taddr + col, v);
      tmem_ld_wait(v);
      const int n0 = c.nb * kBN + col;
      if (row_ok) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int n = n0 + g * 8;
          if (n < c.N) {
            uint32_t yw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              yw[e] = pack_bf16x2(rr * __uint_as_float(v[g * 8 + 2 * e]),
                                  rr * __uint_as_float(v[g * 8 + 2 * e + 1]));
            stg8(p.y_out + rowoff + n, yw);
          }
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// Data-gradient epilogue (CODA blog, section "反向传播的 GEMM-Epilogue 结构"):
// acc = grad_h2 = grad_y @ W1^T for this tile.
//   pass 1: qpart[2 nb + half][m] = sum over the half tile of acc * gamma * h;
//           publish it with a release flag carrying this call's token;
//   then:   wait until every column tile of this row block has published,
//           q[m] = sum of the row's 2 nt partials (fixed order), coef = r^3 q / d;
//   pass 2: grad_h = r * gamma * acc - coef * h   -> dh_out bf16.
// q * r = sum_j grad_h2 * h2 is the statistic s of the method.  The flag wait
// needs every block of the launch resident (cooperative launch) and tiles in
// row-major order with at most gridDim.x column tiles per row; then every wait
// depends only on tiles with smaller index and cannot deadlock.
// ---------------------------------------------------------------------------
struct EpiRmsNormBackward : EpiDefaultCols {
  struct Params {
    const __nv_bfloat16* h;
    const __nv_bfloat16* gamma;
    const float* r;
    __nv_bfloat16* dh_out;
    float* qpart;     // [2 * nt][M]
    uint64_t* flags;  // [mt][nt]
    uint64_t token;
    // Optional extras of the full backward (all null for the plain dgrad):
    const __nv_bfloat16* dh_res;  // [M, d] gradient reaching h through the residual; added to dh
    __nv_bfloat16* h2_out;        // [M, d] normalised activation r * h * gamma (dW1's operand)
    float* gpart;                 // [4 * slabs][d] per-warp column partials of dgamma
  };

  static __device__ __forceinline__ void apply(const Params& p, const WaitCtl& wc,
                                               const TileCtx& c) {
    const int m = c.mb * kBM + c.row;
    const bool row_ok = m < c.M;
    const size_t rowoff = static_cast<size_t>(row_ok ? m : 0) * c.N;

    float qp = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < kHalfChunks; ++ch) {
      const int col = c.half * kHalfCols + ch * 32;
      uint32_t v[32];
      tmem_ld32(c.taddr + col, v);
      tmem_ld_wait(v);
      const int n0 = c.nb * kBN + col;
      if (row_ok) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int n = n0 + g * 8;
          if (n < c.N) {
            const Chunk8 hh = ldg8(p.h + rowoff + n);
            const Chunk8 gg = ldg8(p.gamma + n);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              qp = fmaf(__uint_as_float(v[g * 8 + 2 * e]) * bf16lo(gg.w[e]), bf16lo(hh.w[e]), qp);
              qp = fmaf(__uint_as_float(v[g * 8 + 2 * e + 1]) * bf16hi(gg.w[e]), bf16hi(hh.w[e]),
                        qp);
            }
          }
        }
      }
    }
    if (row_ok) p.qpart[partial_index(c, m)] = qp;

    // Publish this tile's partials, then wait for the whole row block.
    named_bar_sync(1, kEpiThreads);
    uint64_t* row_flags = p.flags + static_cast<size_t>(c.mb) * c.nt;
    if (threadIdx.x == kEpiFirstThread) {
      __threadfence();
      st_release_gpu_u64(row_flags + c.nb, p.token);
      for (int j = 0; j < c.nt; ++j)
        if (!flag_wait(row_flags + j, p.token, wc, kSiteRowFlags)) break;
      __threadfence();
    }
    named_bar_sync(1, kEpiThreads);

    float q = 0.f;
    float rr = 0.f;
    if (row_ok) {
      for (int j = 0; j < 2 * c.nt; ++j) q += __ldcg(p.qpart + static_cast<size_t>(j) * c.M + m);
      rr = __ldg(p.r + m);
    }
    const float coef = rr * rr * rr * q / static_cast<float>(c.N);
    const bool extras = p.gpart != nullptr;

#pragma unroll 1
    for (int ch = 0; ch < kHalfChunks; ++ch) {
      const int col = c.half * kHalfCols + ch * 32;
      uint32_t v[32];
      tmem_ld32(c.taddr + col, v);
      tmem_ld_wait(v);
      const int n0 = c.nb * kBN + col;
      float t[32];  // r * h * grad_h2: this row's contribution to dgamma
#pragma unroll
      for (int i = 0; i < 32; ++i) t[i] = 0.f;
      if (row_ok) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int n = n0 + g * 8;
          if (n < c.N) {
            const Chunk8 hh = ldg8(p.h + rowoff + n);
            const Chunk8 gg = ldg8(p.gamma + n);
            Chunk8 rs = {{0u, 0u, 0u, 0u}};
            if (p.dh_res != nullptr) rs = ldg8(p.dh_res + rowoff + n);
            uint32_t dw[4], h2w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a0 = __uint_as_float(v[g * 8 + 2 * e]);
              const float a1 = __uint_as_float(v[g * 8 + 2 * e + 1]);
              const float h0 = bf16lo(hh.w[e]), h1 = bf16hi(hh.w[e]);
              const float g0 = bf16lo(gg.w[e]), g1 = bf16hi(gg.w[e]);
              const float d0 = rr * g0 * a0 - coef * h0 + bf16lo(rs.w[e]);
              const float d1 = rr * g1 * a1 - coef * h1 + bf16hi(rs.w[e]);
              dw[e] = pack_bf16x2(d0, d1);
              h2w[e] = pack_bf16x2(rr * h0 * g0, rr * h1 * g1);
              t[g * 8 + 2 * e] = rr * h0 * a0;
              t[g * 8 + 2 * e + 1] = rr * h1 * a1;
            }
            stg8(p.dh_out + rowoff + n, dw);
            if (p.h2_out != nullptr) stg8(p.h2_out + rowoff + n, h2w);
          }
        }
      }
      if (extras) {
        // Column sums over the warp's 32 rows: butterfly reduction; lane k ends
        // with the sum for column n0 + k.
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) {
          const bool upper = (lane & o) != 0;
#pragma unroll
          for (int j = 0; j < o; ++j) {
            const float send = upper ? t[j] : t[j + o];
            const float keep = upper ? t[j + o] : t[j];
            t[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
          }
        }
        const int slab_warp = c.mb * 4 + (c.row >> 5);
        if (n0 + lane < c.N) p.gpart[static_cast<size_t>(slab_warp) * c.N + n0 + lane] = t[0];
      }
    }
  }
};

// ---------------------------------------------------------------------------
// GEMM1 epilogue with the gated activation (CODA blog, SwiGLU gating among the
// section "五类 Epilogue 原语", and the pairing idea of section
// "成对激活的寄存器级融合").  W1 = [W_gate | W_up] ([d, N1], the usual layout);
// output tile nb covers gated columns [128 nb, 128 nb + 128): its B tile holds
// the 128 gate columns in accumulator columns 0..127 and the matching 128 up
// columns in 128..255.  Each thread owns a whole accumulator row in TMEM, so
// the pair (gate_j, up_j) is column j and j + 128 of the same thread; no
// weight interleaving and no shuffles are needed.
//   g = r[m] * acc[:, j], u = r[m] * acc[:, j + 128]
//   a[m, 128 nb + j] = silu(g) * u            -> a_out [M, N1/2] bf16
//   optionally y_out = [g | u] at their [gate | up] positions ([M, N1] bf16)
// ---------------------------------------------------------------------------
__device__ __forceinline__ float silu_f(float t) { return t / (1.0f + __expf(-t)); }

struct EpiRowScaleSwiGLU {
  struct Params {
    const float* r;         // [M]
    __nv_bfloat16* y_out;   // [M, N1] pre-activation, may be null
    __nv_bfloat16* a_out;   // [M, N1 / 2]
    FoldedRowReduce fold;   // fold.part != null: r computed here from the partials
  };

  static __host__ __device__ __forceinline__ int num_col_tiles(int N) { return (N / 2 + 127) / 128; }
  static __device__ __forceinline__ int b_col(int nb, int j, int N) {
    return (j < 2 ? 0 : N / 2) + nb * 128 + 64 * (j & 1);
  }

  static __device__ __forceinline__ void apply(const Params& p, const WaitCtl&, const TileCtx& c) {
    const int m = c.mb * kBM + c.row;
    const bool row_ok = m < c.M;
    const int half = c.N / 2;
    float rr = 0.f;
    if (row_ok && p.fold.part != nullptr) {
      rr = folded_rsqrt(p.fold, m, c.M);
      if (c.nb == 0 && c.half == 0) p.fold.r_out[m] = rr;
    } else if (row_ok) {
      rr = __ldg(p.r + m);
    }
    const size_t a_row = static_cast<size_t>(row_ok ? m : 0) * half;
    const size_t y_row = static_cast<size_t>(row_ok ? m : 0) * c.N;
#pragma unroll 1
    for (int ch = 0; ch < 2; ++ch) {  // this thread's 64 gated outputs of the tile
      const int col = c.half * 64 + ch * 32;
      uint32_t g[32], u[32];
      tmem_ld32(c.taddr + col, g);
      tmem_ld32(c.taddr + 128 + col, u);
      tmem_ld_wait(g);
      tmem_ld_wait(u);
      const int o0 = c.nb * 128 + col;
      if (row_ok) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int o = o0 + q * 8;
          if (o < half) {
            uint32_t aw[4], gw[4], uw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float g0 = rr * __uint_as_float(g[q * 8 + 2 * e]);
              const float g1 = rr * __uint_as_float(g[q * 8 + 2 * e + 1]);
              const float u0 = rr * __uint_as_float(u[q * 8 + 2 * e]);
              const float u1 = rr * __uint_as_float(u[q * 8 + 2 * e + 1]);
              aw[e] = pack_bf16x2(silu_f(g0) * u0, silu_f(g1) * u1);
              gw[e] = pack_bf16x2(g0, g1);
              uw[e] = pack_bf16x2(u0, u1);
            }
            stg8(p.a_out + a_row + o, aw);
            if (p.y_out != nullptr) {
              stg8(p.y_out + y_row + o, gw);
              stg8(p.y_out + y_row + half + o, uw);
            }
          }
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// SwiGLU backward epilogue with the row statistic formed upstream (CODA blog,
// section "反向传播的 GEMM-Epilogue 结构": s = sum_cols(grad_y * y) can be
// accumulated in the epilogue of the GEMM where grad_y and y meet).
// The GEMM is the down-projection data gradient: acc = da = dout @ W2^T, one
// 256-column tile of the N1/2 gated columns.  With the saved pre-activation
// y = [g | u] (bf16, [M, N1]) loaded as a rank-2 tile:
//   dg = da * u * silu'(g),  du = da * silu(g)      -> dy_out = [dg | du] bf16
//   spart[2 nb + half][m] = sum over the half tile of dg * g + du * u   (fp32)
// ---------------------------------------------------------------------------
struct EpiSwiGLUBackward : EpiDefaultCols {
  struct Params {
    const __nv_bfloat16* y;  // [M, 2 * half] saved pre-activation [g | u]
    __nv_bfloat16* dy_out;   // [M, 2 * half]
    float* spart;            // [2 * nt][M]
  };

  static __device__ __forceinline__ void apply(const Params& p, const WaitCtl&, const TileCtx& c) {
    const int m = c.mb * kBM + c.row;
    const bool row_ok = m < c.M;
    const int half = c.N;  // the GEMM's output width is the gated width
    const size_t rowoff = static_cast<size_t>(row_ok ? m : 0) * (2 * static_cast<size_t>(half));
    const __nv_bfloat16* grow = p.y + rowoff;
    const __nv_bfloat16* urow = p.y + rowoff + half;
    const int jbase = c.nb * kBN + c.half * kHalfCols;
    float ss = 0.f;
    Chunk8 gc[4], uc[4];
    ldg_chunk(grow, jbase, half, row_ok, gc);
    ldg_chunk(urow, jbase, half, row_ok, uc);
#pragma unroll
    for (int ch = 0; ch < kHalfChunks; ++ch) {
      const int col = c.half * kHalfCols + ch * 32;
      const int j0 = c.nb * kBN + col;
      uint32_t v[32];
      tmem_ld32(c.taddr + col, v);
      Chunk8 gn[4], un[4];
      if (ch + 1 < kHalfChunks) {
        ldg_chunk(grow, j0 + 32, half, row_ok, gn);
        ldg_chunk(urow, j0 + 32, half, row_ok, un);
      }
      tmem_ld_wait(v);
      if (row_ok) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int j = j0 + q * 8;
          if (j < half) {
            uint32_t dgw[4], duw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float dgv[2], duv[2];
#pragma unroll
              for (int k = 0; k < 2; ++k) {
                const float da = __uint_as_float(v[q * 8 + 2 * e + k]);
                const float g = k ? bf16hi(gc[q].w[e]) : bf16lo(gc[q].w[e]);
                const float u = k ? bf16hi(uc[q].w[e]) : bf16lo(uc[q].w[e]);
                const float sig = __fdividef(1.0f, 1.0f + __expf(-g));
                dgv[k] = da * u * sig * (1.0f + g * (1.0f - sig));
                duv[k] = da * g * sig;
                ss = fmaf(dgv[k], g, ss);
                ss = fmaf(duv[k], u, ss);
              }
              dgw[e] = pack_bf16x2(dgv[0], dgv[1]);
              duw[e] = pack_bf16x2(duv[0], duv[1]);
            }
            stg8(p.dy_out + rowoff + j, dgw);
            stg8(p.dy_out + rowoff + half + j, duw);
          }
        }
      }
      if (ch + 1 < kHalfChunks) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          gc[q] = gn[q];
          uc[q] = un[q];
        }
      }
    }
    if (row_ok) p.spart[partial_index(c, m)] = ss;
  }
};

// ---------------------------------------------------------------------------
// Data-gradient epilogue with the statistic given (formed upstream):
//   grad_h = r * gamma * acc - (r^2 * s / d) * h,  acc = grad_h2 = grad_y @ W1^T.
// Purely tile-local: no cross-tile exchange, any tile order.
// ---------------------------------------------------------------------------
struct EpiRmsNormBackwardGivenS : EpiDefaultCols {
  struct Params {
    const __nv_bfloat16* h;
    const __nv_bfloat16* gamma;
    const float* r;
    const float* s;
    __nv_bfloat16* dh_out;
  };

  static __device__ __forceinline__ void apply(const Params& p, const WaitCtl&, const TileCtx& c) {
    const int m = c.mb * kBM + c.row;
    const bool row_ok = m < c.M;
    const size_t rowoff = static_cast<size_t>(row_ok ? m : 0) * c.N;
    const float rr = row_ok ? __ldg(p.r + m) : 0.f;
    const float coef = row_ok ? rr * rr * __ldg(p.s + m) / static_cast<float>(c.N) : 0.f;
    const int nbase = c.nb * kBN + c.half * kHalfCols;
    Chunk8 hc[4], gc[4];
    ldg_chunk(p.h + rowoff, nbase, c.N, row_ok, hc);
    ldg_chunk(p.gamma, nbase, c.N, row_ok, gc);
#pragma unroll
    for (int ch = 0; ch < kHalfChunks; ++ch) {
      const int col = c.half * kHalfCols + ch * 32;
      const int n0 = c.nb * kBN + col;
      uint32_t v[32];
      tmem_ld32(c.taddr + col, v);
      Chunk8 hn[4], gn[4];
      if (ch + 1 < kHalfChunks) {
        ldg_chunk(p.h + rowoff, n0 + 32, c.N, row_ok, hn);
        ldg_chunk(p.gamma, n0 + 32, c.N, row_ok, gn);
      }
      tmem_ld_wait(v);
      if (row_ok) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int n = n0 + g * 8;
          if (n < c.N) {
            uint32_t dw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float d0 = rr * bf16lo(gc[g].w[e]) * __uint_as_float(v[g * 8 + 2 * e]) -
                               coef * bf16lo(hc[g].w[e]);
              const float d1 = rr * bf16hi(gc[g].w[e]) * __uint_as_float(v[g * 8 + 2 * e + 1]) -
                               coef * bf16hi(hc[g].w[e]);
              dw[e] = pack_bf16x2(d0, d1);
            }
            stg8(p.dh_out + rowoff + n, dw);
          }
        }
      }
      if (ch + 1 < kHalfChunks) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          hc[q] = hn[q];
          gc[q] = gn[q];
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// FP8 forward (E4M3 operands with per-tensor scales).
// GEMM0: h = acc * (sx * sW0) + z, partial sums of h^2 as in the bf16 path, and
//        GEMM1's operand quantised once: hq = e4m3_satfinite(h * gamma / s_hg).
// GEMM1: y = r * (s_hg * sW1) * acc.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return (lo & 0xFFFFu) | (hi << 16);
}

struct EpiResidualGammaSumsqFp8 : EpiDefaultCols {
  struct Params {
    const __nv_bfloat16* z;
    const __nv_bfloat16* gamma;
    __nv_bfloat16* h_out;
    uint8_t* hq_out;   // [M, d] E4M3 codes of h * gamma / s_hg
    float* part;       // [2 * nt][M]
    float acc_scale;   // sx * sW0
    float inv_s_hg;    // 1 / s_hg
  };

  static __device__ __forceinline__ void apply(const Params& p, const WaitCtl&, const TileCtx& c) {
    const int m = c.mb * kBM + c.row;
    const bool row_ok = m < c.M;
    const size_t rowoff = static_cast<size_t>(row_ok ? m : 0) * c.N;
    float ss = 0.f;
#pragma unroll 1
    for (int ch = 0; ch < kHalfChunks; ++ch) {
      const int col = c.half * kHalfCols + ch * 32;
      const int n0 = c.nb * kBN + col;
      uint32_t v[32];
      tmem_ld32(c.taddr + col, v);
      tmem_ld_wait(v);
      if (row_ok) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int n = n0 + g * 8;
          if (n < c.N) {
            const Chunk8 zz = ldg8(p.z + rowoff + n);
            const Chunk8 gg = ldg8(p.gamma + n);
            uint32_t hw[4];
            float q[8];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float h0 = __uint_as_float(v[g * 8 + 2 * e]) * p.acc_scale + bf16lo(zz.w[e]);
              const float h1 =
                  __uint_as_float(v[g * 8 + 2 * e + 1]) * p.acc_scale + bf16hi(zz.w[e]);
              ss = fmaf(h0, h0, ss);
              ss = fmaf(h1, h1, ss);
              hw[e] = pack_bf16x2(h0, h1);
              q[2 * e] = h0 * bf16lo(gg.w[e]) * p.inv_s_hg;
              q[2 * e + 1] = h1 * bf16hi(gg.w[e]) * p.inv_s_hg;
            }
            stg8(p.h_out + rowoff + n, hw);
            *reinterpret_cast<uint2*>(p.hq_out + rowoff + n) =
                make_uint2(pack_e4m3x4(q[0], q[1], q[2], q[3]), pack_e4m3x4(q[4], q[5], q[6], q[7]));
          }
        }
      }
    }
    if (row_ok) p.part[partial_index(c, m)] = ss;
  }
};

struct EpiRowScaleFp8 : EpiDefaultCols {
  struct Params {
    const float* r;  // [M]
    __nv_bfloat16* y_out;
    float scale;     // s_hg * sW1
  };

  static __device__ __forceinline__ void apply(const Params& p, const WaitCtl&, const TileCtx& c) {
    const int m = c.mb * kBM + c.row;
    const bool row_ok = m < c.M;
    const size_t rowoff = static_cast<size_t>(row_ok ? m : 0) * c.N;
    const float rr = row_ok ? __ldg(p.r + m) * p.scale : 0.f;
#pragma unroll 1
    for (int ch = 0; ch < kHalfChunks; ++ch) {
      const int col = c.half * kHalfCols + ch * 32;
      uint32_t v[32];
      tmem_ld32(c.taddr + col, v);
      tmem_ld_wait(v);
      const int n0 = c.nb * kBN + col;
      if (row_ok) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int n = n0 + g * 8;
          if (n < c.N) {
            uint32_t yw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              yw[e] = pack_bf16x2(rr * __uint_as_float(v[g * 8 + 2 * e]),
                                  rr * __uint_as_float(v[g * 8 + 2 * e + 1]));
            stg8(p.y_out + rowoff + n, yw);
          }
        }
      }
    }
  }
};

}  // namespace coda
