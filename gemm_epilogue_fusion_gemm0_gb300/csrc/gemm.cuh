// gemm.cuh -- persistent, warp-specialised tcgen05 GEMM with a programmable epilogue.
//
// The mainloop is fixed and the epilogue is a policy class, which is the
// split the method is built on (CODA blog, blog.hotdry.top, section
// "核心观察：Epilogue 是天然的融合点": a tiled MMA mainloop followed by an
// epilogue that works on the output tile while it is still on chip).
//
//   C[M, N] = A[M, K] @ B[K, N], bf16 operands, fp32 accumulation in TMEM.
//   A is K-major (row-major [M, K], activations) or MN-major (row-major
//   [K, M], i.e. the transpose of an activation: weight gradients, K = tokens).
//   B is MN-major (row-major [K, N], i.e. a weight stored [in, out], or an
//   activation gradient) or K-major (row-major [N, K], i.e. the transpose of
//   a weight stored [in, out]).
//
// Block = 320 threads, one block per SM, persistent over output tiles:
//   warp 0      TMA producer: 4-stage ring of A (128x64) + B (64x256) tiles,
//               128-byte swizzle, completion on mbarriers with expect-tx
//   warp 1      allocates 512 TMEM columns, one thread issues
//               tcgen05.mma (M=128, N=256, K=16) into one of two fp32
//               accumulators (2 x 256 columns), commits stage and tile barriers
//   warps 2..9  epilogue: drain the accumulator with tcgen05.ld (thread = row;
//               two warps per TMEM lane quadrant, one per 128-column half),
//               apply Epi, store; while they work the MMA warp fills the other
//               accumulator, so epilogue and mainloop overlap.
#pragma once

#include "ptx.cuh"

namespace coda {

__device__ uint32_t g_coda_status = 0;  // device status word (see WaitSite)

// ---------------------------------------------------------------------------
// Checked build (compiled with -DCODA_CHECKED, libcoda_checked.so): every
// staged load and store of a rank-2 tensor in the epilogues is checked against
// the extent of the tensor it belongs to (and every vector load of gamma
// against its length), every TMA box start against its tensor map's extent and
// the 16-byte alignment of its innermost coordinate, and every index into the
// workspace (partial sums, completion flags, split-tail slots) against the
// size the host gave it.  A failed check records 0x200 | site in the status
// word (first failure wins; coda_get_device_status reports
// CODA_ERR_DEVICE_BOUNDS) and skips the access; a failed TMA check also makes
// the producer leave its role like a wait that ran out.  Nothing traps.  In the
// normal build every check compiles to nothing.
// ---------------------------------------------------------------------------
#ifdef CODA_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

enum CheckSite : uint32_t {
  kChkTmaA = 1,        // A operand box start
  kChkTmaB = 2,        // B operand box start
  kChkLoad = 3,        // epilogue operand load (z, h, dh_res, saved y)
  kChkStore = 4,       // epilogue output store
  kChkPartial = 5,     // per-tile partial sum (sum of squares, q, s)
  kChkFlag = 6,        // row-block completion flag
  kChkSplitSlot = 7,   // split-tail partial slot or its flag
  kChkColPartial = 8,  // column partial of dgamma
};

__device__ __forceinline__ bool checked(bool ok, uint32_t site) {
  if (!kChecked || ok) return true;
  atomicCAS(&g_coda_status, 0u, 0x200u | site);
  return false;
}

// The bytes of one tensor, for the checked build's address checks (an empty
// span checks nothing).
struct Span {
  const char* base;
  size_t bytes;
};

__device__ __forceinline__ Span span(const void* base, int rows, size_t row_bytes) {
  return Span{static_cast<const char*>(base), static_cast<size_t>(rows) * row_bytes};
}

// [p, p + n) lies inside the span
__device__ __forceinline__ bool in_span(const Span& s, const void* p, size_t n) {
  const char* c = static_cast<const char*>(p);
  return s.base == nullptr || (c >= s.base && c + n <= s.base + s.bytes);
}

// A TMA box start: the innermost coordinate x (elements of `esize` bytes) on a
// 16-byte boundary, both coordinates non-negative and less than one tile (256)
// past their extent (a load may start past the edge; it reads the fill value).
__device__ __forceinline__ bool tma_start_ok(int x, int y, int x_ext, int y_ext, int esize) {
  return x >= 0 && y >= 0 && (x * esize) % 16 == 0 && x < x_ext + 256 && y < y_ext + 256;
}

constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kStages = 4;
constexpr int kThreads = 320;       // warp 0 TMA, warp 1 MMA, warps 2..9 epilogue
constexpr int kEpiThreads = 256;
constexpr int kEpiWarps = kEpiThreads / 32;
constexpr int kEpiFirstThread = 64;
constexpr uint32_t kAStageBytes = kBM * kBK * 2;   // 16 KB
constexpr uint32_t kBStageBytes = kBN * kBK * 2;   // 32 KB
constexpr uint32_t kBChunkBytes = 64 * kBK * 2;    // one 64-column MN-major chunk: 8 KB
constexpr uint32_t kStageBytes = kAStageBytes + kBStageBytes;
constexpr uint32_t kTmemCols = 2 * kBN;
constexpr uint32_t kSmemA = 0;
constexpr uint32_t kSmemB = kStages * kAStageBytes;
constexpr uint32_t kSmemBar = kSmemB + kStages * kBStageBytes;
// barriers: full[S] | empty[S] | tfull[2] | tempty[2] | drain, then the TMEM
// address holder and the abort flag right after them
constexpr uint32_t kBarBytes = 8u * (2 * kStages + 5);
constexpr uint32_t kSmemBytes = kSmemBar + 256 + 1024;  // barriers + 1 KB alignment slack

static_assert(kBarBytes + 8 <= 256, "barrier area overflows its reserved 256 bytes");

// Epilogue store staging: policies that stage their output stores through
// shared memory (Epi::kStageBytesPerWarp > 0) get that many bytes per epilogue
// warp right after the barrier area.
template <class Epi>
__host__ __device__ constexpr uint32_t cta_smem_bytes() {
  return kSmemBytes + kEpiWarps * Epi::kStageBytesPerWarp;
}

// Serpentine K order: on odd waves of a block's persistent tile loop the
// producer walks K backwards, so the next wave starts on the K slices that
// the previous wave left in L2 (the MMA order follows the producer's).
constexpr bool kSerpentineK = false;

static_assert(kBK * 2 == 128, "one K tile row must be exactly one 128-byte swizzle row");
static_assert(kSmemBytes <= 232448, "exceeds the 227 KB per-block shared memory limit");

// Tile order.  Tiles are visited in groups of `group_m` row blocks; inside a
// group the row block varies fastest, so the blocks working at the same time
// share a few column tiles of B and a few row blocks of A in L2.
// group_m = 1 gives plain row-major order (all column tiles of a row block
// are consecutive), which the cross-tile row statistic of the backward needs.
struct TileMap {
  int mt, nt, group_m;
  __device__ __forceinline__ void coords(int t, int& mb, int& nb) const {
    const int per_group = group_m * nt;
    const int g = t / per_group;
    const int w = t - g * per_group;
    const int rows = min(group_m, mt - g * group_m);
    mb = g * group_m + w % rows;
    nb = w / rows;
  }
};

// Epilogue context handed to the policy for one output tile.
struct TileCtx {
  uint32_t taddr;  // TMEM address of this thread's lane, column 0 of the tile
  int mb, nb;      // tile coordinates (nb: column tile index inside the row block)
  int n0, nend;    // the tile's output columns are [n0, nend); nend <= n0 + 256 and <= N
  int row;         // row inside the tile (0..127) owned by this thread
  int half;        // which 128-column half of the tile this thread drains (0, 1)
  int M, N;        // problem size (N = output columns)
  int nt;          // number of column tiles per row block
  uint32_t stage;  // this warp's store-staging buffer (shared address), if the policy has one
};

__device__ __forceinline__ bool epi_all(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 256, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(ok ? 1u : 0u)
      : "memory");
  return r != 0;
}

template <class Epi, bool kBMNMajor, bool kAMNMajor = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_epilogue_kernel(const __grid_constant__ CUtensorMap tmA,
                         const __grid_constant__ CUtensorMap tmB, int M, int N, int K, int group_m,
                         const typename Epi::Params ep, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms need 1 KB alignment
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sA = base + kSmemA;
  const uint32_t sB = base + kSmemB;
  const uint32_t bar0 = base + kSmemBar;
  // barrier layout: full[kStages] | empty[kStages] | tfull[2] | tempty[2] | drain
  const uint32_t bar_full = bar0;
  const uint32_t bar_empty = bar0 + 8u * kStages;
  const uint32_t bar_tfull = bar0 + 16u * kStages;
  const uint32_t bar_tempty = bar_tfull + 16u;
  const uint32_t bar_drain = bar_tempty + 16u;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kSmemBar + kBarBytes);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem + kSmemBar + kBarBytes + 4);

  static_assert(cta_smem_bytes<Epi>() <= 232448, "exceeds the 227 KB per-block shared memory limit");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int mt = (M + kBM - 1) / kBM;
  const int nt = Epi::num_col_tiles(N);
  const int nk = (K + kBK - 1) / kBK;
  const int num_tiles = mt * nt;
  const TileMap tmap{mt, nt, group_m};
  const WaitCtl wc{timeout_ns, &g_coda_status, abort_flag};

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full + 8u * s, 1);
      mbar_init(bar_empty + 8u * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8u * b, 1);
      mbar_init(bar_tempty + 8u * b, kEpiThreads);
    }
    mbar_init(bar_drain, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  griddep_launch_dependents();
  griddep_wait();  // prologue done: from here on the preceding kernel's output may be read

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued_mask = 0, last_par = 0;  // per stage: issued?, parity of last issue
      bool ok = true;
      uint32_t wave = 0;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++wave) {
        int mb, nb;
        tmap.coords(t, mb, nb);
        const bool reverse = kSerpentineK && (wave & 1u);
        for (int kbi = 0; kbi < nk; ++kbi) {
          const int kb = reverse ? nk - 1 - kbi : kbi;
          if (!bounded_wait(bar_empty + 8u * s, ph ^ 1u, wc, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t full = bar_full + 8u * s;
          if constexpr (kChecked) {
            const bool a_ok = kAMNMajor ? tma_start_ok(mb * kBM, kb * kBK, M, K, 2)
                                        : tma_start_ok(kb * kBK, mb * kBM, K, M, 2);
            bool b_ok = true;
            if constexpr (kBMNMajor) {
              for (int j = 0; j < kBN / 64; ++j)
                b_ok = b_ok && tma_start_ok(Epi::b_col(nb, j, N), kb * kBK, N, K, 2);
            } else {
              b_ok = tma_start_ok(kb * kBK, nb * kBN, K, N, 2);
            }
            if (!checked(a_ok, kChkTmaA) || !checked(b_ok, kChkTmaB)) {
              *wc.abort_flag = 1u;
              ok = false;
              break;
            }
          }
          mbar_arrive_expect_tx(full, kStageBytes);
          const uint32_t a_dst = sA + s * kAStageBytes;
          const uint32_t b_dst = sB + s * kBStageBytes;
          if constexpr (kAMNMajor) {
            tma_load_2d(a_dst, &tmA, full, mb * kBM, kb * kBK);
            tma_load_2d(a_dst + kBChunkBytes, &tmA, full, mb * kBM + 64, kb * kBK);
          } else {
            tma_load_2d(a_dst, &tmA, full, kb * kBK, mb * kBM);
          }
          if constexpr (kBMNMajor) {
#pragma unroll
            for (int j = 0; j < kBN / 64; ++j)
              tma_load_2d(b_dst + j * kBChunkBytes, &tmB, full, Epi::b_col(nb, j, N), kb * kBK);
          } else {
            tma_load_2d(b_dst, &tmB, full, kb * kBK, nb * kBN);
          }
          issued_mask |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every issued copy land before the block can exit.
        WaitCtl dwc = wc;
        for (int i = 0; i < kStages; ++i)
          if (issued_mask & (1u << i)) {
            const uint32_t p = (last_par >> i) & 1u;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar_full + 8u * i, p) &&
                   globaltimer_ns() - t0 < dwc.timeout_ns) {
            }
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN, kAMNMajor, kBMNMajor);
      int s = 0;
      uint32_t ph = 0;
      uint32_t it = 0;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; ok && t < num_tiles; t += gridDim.x, ++it) {
        const uint32_t b = it & 1u;
        const uint32_t aph = (it >> 1) & 1u;
        if (!bounded_wait(bar_tempty + 8u * b, aph ^ 1u, wc, kSiteMmaTmemEmpty)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * kBN;
        for (int kb = 0; kb < nk; ++kb) {
          if (!bounded_wait(bar_full + 8u * s, ph, wc, kSiteMmaFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sA + s * kAStageBytes;
          const uint32_t b0 = sB + s * kBStageBytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            const uint64_t ad = kAMNMajor ? sdesc_sw128(a0 + k * 2048, kBChunkBytes, 1024)
                                          : sdesc_sw128(a0 + k * 32, 16, 1024);
            const uint64_t bd = kBMNMajor ? sdesc_sw128(b0 + k * 2048, kBChunkBytes, 1024)
                                          : sdesc_sw128(b0 + k * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb | k) != 0 ? 1u : 0u);
          }
          issued = true;
          umma_commit(bar_empty + 8u * s);  // frees the smem stage when these MMAs finish
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(bar_tfull + 8u * b);  // accumulator b is complete
      }
      if (issued) {
        // All MMAs of this block must finish before TMEM is released.
        umma_commit(bar_drain);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(bar_drain, 0)) {
          if (globaltimer_ns() - t0 > timeout_ns) {
            record_failure(wc, kSiteDrain);
            break;
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;         // TMEM lane quadrant this warp may access
    const int half = (warp - 2) >> 2;  // warps 2..5: columns 0..127, warps 6..9: 128..255
    const int row = quad * 32 + lane;
    uint32_t it = 0;
    for (int t = blockIdx.x; t < num_tiles; t += gridDim.x, ++it) {
      const uint32_t b = it & 1u;
      const uint32_t aph = (it >> 1) & 1u;
      int mb, nb;
      tmap.coords(t, mb, nb);
      const bool ok = bounded_wait(bar_tfull + 8u * b, aph, wc, kSiteEpiTmemFull);
      if (!epi_all(ok)) break;  // all 128 epilogue threads leave together
      tc_fence_after();
      TileCtx c;
      c.taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + b * kBN;
      c.mb = mb;
      c.nb = nb;
      c.n0 = nb * kBN;
      c.nend = min(N, c.n0 + kBN);
      c.row = row;
      c.half = half;
      c.M = M;
      c.N = N;
      c.nt = nt;
      c.stage = base + kSmemBar + 256u + static_cast<uint32_t>(warp - 2) * Epi::kStageBytesPerWarp;
      Epi::apply(ep, wc, c);
      tc_fence_before();
      mbar_arrive(bar_tempty + 8u * b);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0) Epi::at_exit(ep);  // every thread of the block is done (barrier above)
}

}  // namespace coda
