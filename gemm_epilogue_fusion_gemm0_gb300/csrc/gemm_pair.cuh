// gemm_pair.cuh -- the GEMM-epilogue kernel on a CTA pair (tcgen05 .cta_group::2).
//
// Same contract and epilogue policies as gemm_epilogue_kernel (gemm.cuh), but a
// cluster of two CTAs on two SMs computes one 256 x 256 output tile:
//   - CTA r (r = 0, 1) loads rows [128 r, 128 r + 128) of the A tile and half
//     of the B tile (N columns [128 r, 128 r + 128)) into its own shared memory;
//   - one thread of CTA 0 issues tcgen05.mma.cta_group::2 (M = 256, N = 256,
//     K = 16), which reads both CTAs' operands and writes each CTA's 128
//     accumulator rows into that CTA's tensor memory;
//   - each CTA's epilogue drains its own 128 x 256 accumulator.
// Each SM therefore streams 32 KB per 64-deep K step instead of 48 KB, which
// leaves room for a 6-stage ring and halves the B traffic from L2.
//
// Barriers: the TMA of both CTAs completes on CTA 0's `full` barrier (CTA 0
// arms it with both CTAs' bytes); the MMA commit is multicast to the `empty`,
// `tfull` and `drain` barriers of both CTAs; each CTA's epilogue releases an
// accumulator by one arrive on CTA 0's `tempty` barrier (count 2).
//
// Work: the kernel is persistent; tile t goes to pair t mod (number of pairs),
// except that a launch may share its last tiles out along K (the split tail
// below) when whole tiles would leave the last wave of pairs mostly idle.
#pragma once

#include <type_traits>

#include "gemm.cuh"

namespace coda {

constexpr int kPairBM = 256;                         // tile rows per CTA pair
constexpr int kPairStages = 6;
constexpr uint32_t kPairAStageBytes = 128 * kBK * 2;  // 16 KB: this CTA's 128 rows
constexpr uint32_t kPairBStageBytes = 128 * kBK * 2;  // 16 KB: this CTA's half of B
constexpr uint32_t kPairStageBytes = kPairAStageBytes + kPairBStageBytes;
constexpr uint32_t kPairSmemA = 0;
constexpr uint32_t kPairSmemB = kPairStages * kPairAStageBytes;
constexpr uint32_t kPairSmemBar = kPairSmemB + kPairStages * kPairBStageBytes;
// barriers: full[S] | empty[S] | tfull[2] | tempty[2] | drain, then the TMEM
// address holder and the abort flag right after them
constexpr uint32_t kPairBarBytes = 8u * (2 * kPairStages + 5);
constexpr uint32_t kPairSmemBytes = kPairSmemBar + 256 + 1024;

static_assert(kPairBarBytes + 8 <= 256, "barrier area overflows its reserved 256 bytes");

static_assert(kPairSmemBytes <= 232448, "exceeds the 227 KB per-block shared memory limit");

// ---------------------------------------------------------------------------
// Stream-K tail.  With T tiles on U CTA pairs, T = W U + R (0 < R < U), plain
// round-robin leaves the last wave R/U full.  Instead:
//   - tiles [0, dp_tiles), dp_tiles = (W - 1) U, are whole work items, tile t
//     going to pair t mod U;
//   - the remaining S = U + R tiles are laid end to end along K (S * nk k-blocks
//     of kBK) and cut into U contiguous slices, pair i taking
//     [floor(i S nk / U), floor((i + 1) S nk / U)).
// Every pair then runs the same number of k-blocks, up to one.  A slice is at
// least nk long, so a tile is shared by at most two pairs: the owner, whose
// slice holds the tile's first k-block, and the next pair, whose slice starts
// inside the tile.  That pair's first item is the tile's tail: its epilogue
// warps write the fp32 accumulator to a partial slot and publish it with a
// release flag.  The owner's epilogue waits for the flag, adds the partial into
// its TMEM accumulator and runs the policy on the sum.  A partial is always its
// pair's first tail item and waits for nothing but its own data, so the owner's
// wait always ends.
// A flag holds (*epoch + 1) ^ salt, epoch being the launch counter at the start
// of the caller's workspace, which the last block of the launch to finish
// advances (launch_exit), and salt a random value the host draws for each call:
// flags of earlier launches on the counter never match and other contents match
// only by a 2^-64 coincidence, so the slots need no clearing and a launch
// replayed from a CUDA graph draws a fresh token.  The owner's wait needs the
// other pair resident, so such a launch is cooperative.
// Policies whose epilogue waits on other tiles (the data gradient's row flags)
// are launched without a split tail.
// ---------------------------------------------------------------------------
struct SkParams {
  int dp_tiles;     // tiles handed out whole; >= the tile count: no split tail
  float* part;      // [S][2 CTAs][128 x 256] fp32 partial accumulators
  uint64_t* flags;  // [S][2 CTAs]
  uint64_t* epoch;  // launch counter (any initial value); null when the tail is not split
  int slots;        // S, the partial slots the workspace holds
  uint64_t salt;    // this call's random value; a flag holds token ^ salt
  // Piece split (policies with kSplitTail = false, see PieceWork); 0: none
  int pieces;       // P, K pieces per tile past dp_tiles
  int lvl_first;    // pairs from lvl_first on take lvl pieces each before the others
  int lvl;
};

constexpr SkParams kNoSplitTail = {0x7fffffff, nullptr, nullptr, nullptr, 0, 0, 0, 0, 0};

// A policy opts out of the split tail (its epilogue waits on other tiles) with
// `static constexpr bool kSplitTail = false;`; the kernel then compiles without it.
template <class E, class = void>
struct SplitsTail : std::true_type {};
template <class E>
struct SplitsTail<E, std::void_t<decltype(E::kSplitTail)>> : std::bool_constant<E::kSplitTail> {};

constexpr int kItemWhole = 0;  // all nk k-blocks of the tile
constexpr int kItemOwner = 1;  // k-blocks [0, kb1): adds the partial, runs the epilogue
constexpr int kItemTail = 2;   // k-blocks [kb0, nk): writes the partial

struct WorkItem {
  int tile, kb0, kb1, kind;
  int piece = 0;  // the K piece of a pieced tile (PieceWork)
};

// The split items of one CTA pair, in order (the same sequence in the producer,
// MMA and epilogue roles, each of which first runs its whole tiles
// pair, pair + npairs, ... below dp_end).
struct SplitWork {
  int nk, sk_base;
  long long kpos, kend;
  __device__ __forceinline__ SplitWork(int pair, int npairs, int num_tiles, int dp_end, int nk_)
      : nk(nk_), sk_base(dp_end) {
    const long long tot = static_cast<long long>(num_tiles - dp_end) * nk_;
    kpos = tot * pair / npairs;
    kend = tot * (pair + 1) / npairs;
  }
  __device__ __forceinline__ bool next(WorkItem& w) {
    if (kpos >= kend) return false;
    const int s = static_cast<int>(kpos / nk);
    w.tile = sk_base + s;
    w.kb0 = static_cast<int>(kpos - static_cast<long long>(s) * nk);
    w.kb1 = static_cast<int>(min(static_cast<long long>(nk), w.kb0 + (kend - kpos)));
    w.kind = w.kb0 > 0 ? kItemTail : (w.kb1 < nk ? kItemOwner : kItemWhole);
    kpos += w.kb1 - w.kb0;
    return true;
  }
};

// ---------------------------------------------------------------------------
// Piece split, for policies whose epilogue waits on other tiles (the data
// gradient's row statistic: kSplitTail = false).  The stream-K tail above cuts
// each pair's share of the last tiles at a different K offset, so the pairs
// stop walking K in step and the long-K operands stop being shared in L2; and
// a split tile that waited on its row block while holding TMEM could block the
// pair's later items.  Instead, with R tiles past dp_tiles (whole row blocks,
// R <= pairs):
//   - every tile past dp_tiles is cut into P pieces along K, piece q holding
//     k-blocks [q nk / P, (q + 1) nk / P);
//   - the R P pieces are dealt in piece-major order (unit u = q R + tile): the
//     first (U - lvl_first) lvl units go, lvl at a time, to the pairs from
//     lvl_first on (those with one whole tile fewer), the rest round-robin to
//     pairs 0, 1, ...; so at any time only two or three piece indices are in
//     flight and the pairs of each walk K in step;
//   - piece P - 1 of a tile is its owner: the last R units, dealt last, so an
//     owner is the last item of its pair and no pair holds two; the host
//     keeps the levelled units clear of them.  Every other piece writes its
//     fp32 accumulator to a partial slot and publishes a flag; the owner waits
//     for its tile's P - 1 flags, adds the partials into its accumulator and
//     runs the policy (which may then wait on its row block's other owners).
// Pieces never wait and owners wait only on pieces and on other owners, all
// resident (a cooperative launch), so every wait ends.  Slots: tile
// dp_tiles + i, piece q < P - 1, CTA r is slot (i (P - 1) + q) 2 + r.
// ---------------------------------------------------------------------------
struct PieceWork {
  int R, P, nk, base, npairs, pair, lvl_first, lvl, lvl_units, rr_units;
  int i = 0, j = 0;
  __device__ __forceinline__ PieceWork(const SkParams& sk, int pair_, int npairs_, int num_tiles,
                                       int nk_)
      : R(num_tiles - sk.dp_tiles), P(sk.pieces), nk(nk_), base(sk.dp_tiles), npairs(npairs_),
        pair(pair_), lvl_first(sk.lvl_first), lvl(sk.lvl) {
    lvl_units = (npairs - lvl_first) * lvl;
    rr_units = R * P - lvl_units;
  }
  __device__ __forceinline__ bool next(WorkItem& w) {
    int u;
    if (pair >= lvl_first && i < lvl) {
      u = (pair - lvl_first) * lvl + i++;
    } else {
      const int v = pair + j * npairs;
      if (v >= rr_units) return false;
      ++j;
      u = lvl_units + v;
    }
    const int q = u / R;
    w.tile = base + (u - q * R);
    w.kb0 = static_cast<int>(static_cast<long long>(q) * nk / P);
    w.kb1 = static_cast<int>(static_cast<long long>(q + 1) * nk / P);
    w.kind = q == P - 1 ? kItemOwner : kItemTail;
    w.piece = q;
    return true;
  }
};

// Partial slot layout: the 128 x 256 fp32 block of one CTA in float4 units,
// stored so that a warp's 32 rows of one 16-byte column group are 512
// contiguous bytes.  Each epilogue thread owns one row and one 128-column half
// (4 chunks of 32 columns, 8 float4 each).
constexpr int kSkChunks = kBN / 2 / 32;
constexpr size_t kSkSlotFloats = 128 * kBN;
__device__ __forceinline__ size_t sk_part_index4(int half, int ch, int v, int row) {
  return static_cast<size_t>(((half * kSkChunks + ch) * 8 + v) * 128 + row);
}

// Tail item: this thread's row and half of the accumulator -> the partial slot.
__device__ __forceinline__ void sk_write_partial(uint32_t taddr, float4* slot, int half, int row) {
#pragma unroll 1
  for (int ch = 0; ch < kSkChunks; ++ch) {
    uint32_t v[32];
    tmem_ld32(taddr + half * (kBN / 2) + ch * 32, v);
    tmem_ld_wait(v);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      slot[sk_part_index4(half, ch, j, row)] =
          make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                      __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
  }
}

// Owner item: accumulator += partial, in place in TMEM.  The partial's loads
// are issued before the TMEM read of the same chunk so that the two latencies
// overlap.
__device__ __forceinline__ void sk_add_partial(uint32_t taddr, const float4* slot, int half,
                                               int row) {
#pragma unroll 1
  for (int ch = 0; ch < kSkChunks; ++ch) {
    const uint32_t col = taddr + half * (kBN / 2) + ch * 32;
    float4 q[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = __ldcg(slot + sk_part_index4(half, ch, j, row));
    uint32_t v[32];
    tmem_ld32(col, v);
    tmem_ld_wait(v);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + q[j].x);
      v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + q[j].y);
      v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + q[j].z);
      v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + q[j].w);
    }
    tmem_st32(col, v);
  }
  tmem_st_wait();
}

// The epilogue of a piece (PieceWork) for this thread's row and half: a piece
// writes its accumulator to its partial slot and publishes the slot's flag; the
// owner (the tile's last piece) waits for the tile's p1 flags and adds the
// partials into its accumulator.  Kept out of line so that the policies'
// epilogues keep their registers.
__device__ __noinline__ void piece_epilogue(float* part, uint64_t* flags, uint64_t* epoch,
                                           uint64_t salt, WaitCtl wc, uint32_t taddr, size_t first,
                                           int p1, int piece, bool is_piece, uint32_t rank, int half,
                                           int row) {
  if (is_piece) {
    const size_t slot = (first + piece) * 2 + rank;
    sk_write_partial(taddr, reinterpret_cast<float4*>(part + slot * kSkSlotFloats), half, row);
    __threadfence();
    named_bar_sync(1, kEpiThreads);
    if (threadIdx.x == kEpiFirstThread) st_release_gpu_u64(flags + slot, launch_tag(epoch, salt));
  } else {
    if (threadIdx.x == kEpiFirstThread) {
      const uint64_t tag = launch_tag(epoch, salt);
      for (int q = 0; q < p1; ++q)
        if (!flag_wait(flags + (first + q) * 2 + rank, tag, wc, kSitePieces)) break;
      __threadfence();
    }
    named_bar_sync(1, kEpiThreads);
    for (int q = 0; q < p1; ++q)
      sk_add_partial(taddr,
                     reinterpret_cast<const float4*>(part + ((first + q) * 2 + rank) * kSkSlotFloats),
                     half, row);
    tc_fence_before();
    named_bar_sync(1, kEpiThreads);
    tc_fence_after();
  }
}

// ---------------------------------------------------------------------------
// Column plan: tiles narrower than 256 columns, so that a launch's tiles spread
// evenly over the CTA pairs.  With 256-column tiles a row block of d columns has
// ceil(d / 256) tiles, and T tiles on U pairs leave the last wave (T mod U) / U
// full: at d = 4096 and 32 row blocks, 512 tiles run 6.74 waves in the time of
// 7.  A plan cuts every row block into nt tiles instead, nt - nl of them w
// columns wide and nl of them w + step (w and step multiples of 16, w + step at
// most 256), laid out from column 0 in tile order: tile j of row block mb is wide iff
// (j + mb * rot) mod nt < nl, so the wide tiles move to other pairs from one row
// block to the next (tile t goes to pair t mod U).  The MMA of a tile has that
// width (N of tcgen05.mma .cta_group::2 is any multiple of 16 up to 256), each
// CTA loads b_rows rows of B (half the widest tile) and the epilogue masks the
// columns past the tile.  Only for K-major B operands in bf16 (the data
// gradients: B = W1 read as [d, N1]).  nt == 0: the policy's own tiling.
// kserp (with or without nt) reverses the K order of every other wave of
// tiles: the pairs of one wave walk K in step, so the wave that follows starts
// on the K slices of B that the previous one read last, which the L2 may still
// hold.  Only the load order changes; the MMA accumulates the k-blocks in the
// order they arrive, so results differ only in fp32 summation order.
// ---------------------------------------------------------------------------
struct ColPlan {
  int nt;      // column tiles per row block (0: no plan)
  int w;       // width of a narrow tile (multiple of 16)
  int nl;      // wide tiles (w + step columns) per row block
  int rot;     // rotation of the wide tiles from one row block to the next
  int b_rows;  // rows of B each CTA loads per stage (the B tensor map's box)
  int step;    // a wide tile's extra columns (multiple of 16)
  int kserp;   // 1: tiles of odd waves (tile / pairs odd) load K backwards (any nt)
  // wide tiles among the positions [0, x) of the periodic pattern
  __host__ __device__ __forceinline__ int wide_before(int x) const {
    return (x / nt) * nl + min(x % nt, nl);
  }
  // first column and width of tile j of row block mb
  __host__ __device__ __forceinline__ void tile(int mb, int j, int& n0, int& width) const {
    const int s = static_cast<int>((static_cast<long long>(mb) * rot) % nt);
    width = ((j + s) % nt < nl) ? w + step : w;
    n0 = j * w + step * (wide_before(s + j) - wide_before(s));
  }
};

constexpr ColPlan kNoColPlan = {0, kBN, 0, 0, 128, 16, 0};

// plus the policy's store-staging buffers after the barrier area (see cta_smem_bytes)
template <class Epi>
__host__ __device__ constexpr uint32_t pair_smem_bytes() {
  return kPairSmemBytes + kEpiWarps * Epi::kStageBytesPerWarp;
}

// kFp8: E4M3 operands (tcgen05 kind::f8f6f4).  A 128-byte smem row then holds
// 128 K elements, so a stage covers K = 128 with the same bytes, each MMA
// consumes K = 32, and an MN-major B half-tile (128 columns) is one TMA box.
template <class Epi, bool kBMNMajor, bool kAMNMajor = false, bool kFp8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    gemm_pair_epilogue_kernel(const __grid_constant__ CUtensorMap tmA,
                              const __grid_constant__ CUtensorMap tmB, int M, int N, int K,
                              int group_m, const typename Epi::Params ep, const SkParams sk,
                              const ColPlan cplan, uint64_t timeout_ns) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sA = base + kPairSmemA;
  const uint32_t sB = base + kPairSmemB;
  const uint32_t bar0 = base + kPairSmemBar;
  // full[S] | empty[S] | tfull[2] | tempty[2] | drain
  const uint32_t bar_full = bar0;
  const uint32_t bar_empty = bar0 + 8u * kPairStages;
  const uint32_t bar_tfull = bar0 + 16u * kPairStages;
  const uint32_t bar_tempty = bar_tfull + 16u;
  const uint32_t bar_drain = bar_tempty + 16u;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + kPairSmemBar + kPairBarBytes);
  volatile uint32_t* abort_flag =
      reinterpret_cast<volatile uint32_t*>(smem + kPairSmemBar + kPairBarBytes + 4);

  static_assert(pair_smem_bytes<Epi>() <= 232448, "exceeds the 227 KB per-block shared memory limit");
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair = blockIdx.x >> 1;
  const int npairs = gridDim.x >> 1;
  const int mt = (M + kPairBM - 1) / kPairBM;
  // a column plan applies to bf16 K-major B without a split tail (see ColPlan)
  constexpr bool kPlanCapable = !kBMNMajor && !kAMNMajor && !kFp8 && !SplitsTail<Epi>::value;
  const bool planned = kPlanCapable && cplan.nt > 0;
  const int nt = planned ? cplan.nt : Epi::num_col_tiles(N);
  // first output column and width of tile (mb, nb)
  const auto geometry = [&](int mb, int nb, int& n0, int& width) {
    if (planned) {
      cplan.tile(mb, nb, n0, width);
    } else {
      n0 = nb * kBN;
      width = kBN;
    }
  };
  static_assert(!(kFp8 && kAMNMajor), "FP8 path: A must be K-major");
  constexpr int kKE = kFp8 ? 128 : kBK;  // K elements per stage (128-byte rows)
  const int nk = (K + kKE - 1) / kKE;
  const int num_tiles = mt * nt;
  const TileMap tmap{mt, nt, group_m};
  const WaitCtl wc{timeout_ns, &g_coda_status, abort_flag};
  constexpr bool kSplit = SplitsTail<Epi>::value;
  // whole tiles below dp_end; a split needs the slots (never planned without them)
  // tiles past dp_end cut into K pieces (PieceWork), for the policies without a split tail
  const bool pieced = kPlanCapable && !planned && sk.pieces > 1 && sk.part != nullptr;
  const int dp_end =
      ((kSplit && sk.part != nullptr) || pieced) ? min(sk.dp_tiles, num_tiles) : num_tiles;

  if (threadIdx.x == 0) {
    *abort_flag = 0u;
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(bar_full + 8u * s, 1);
      mbar_init(bar_empty + 8u * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_tfull + 8u * b, 1);
      mbar_init(bar_tempty + 8u * b, 2);
    }
    mbar_init(bar_drain, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync_all();  // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  griddep_launch_dependents();
  griddep_wait();  // prologue done: from here on the preceding kernel's output may be read

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int s = 0;
      uint32_t ph = 0;
      uint32_t issued_mask = 0, last_par = 0;
      bool ok = true;
      // bytes one CTA's copies bring per stage (a plan's B box has b_rows rows of 128 bytes)
      const uint32_t stage_bytes =
          planned ? kPairAStageBytes + static_cast<uint32_t>(cplan.b_rows) * 128u : kPairStageBytes;
      const auto loads = [&](const WorkItem& w) {
        int mb, nb;
        tmap.coords(w.tile, mb, nb);
        const int arow = mb * kPairBM + static_cast<int>(rank) * 128;
        int n0, width;
        geometry(mb, nb, n0, width);
        const int bcol = n0 + static_cast<int>(rank) * (width / 2);  // K-major B rows
        // serpentine K order: whole tiles of odd waves walk K backwards (see ColPlan)
        const bool rev = kPlanCapable && cplan.kserp != 0 && w.kind == kItemWhole &&
                         ((w.tile / npairs) & 1) != 0;
        for (int ki = w.kb0; ki < w.kb1; ++ki) {
          const int kb = rev ? w.kb0 + w.kb1 - 1 - ki : ki;
          if (!bounded_wait(bar_empty + 8u * s, ph ^ 1u, wc, kSiteProducerEmpty)) {
            ok = false;
            break;
          }
          const uint32_t full_local = bar_full + 8u * s;
          const uint32_t full_leader = mapa_shared(full_local, 0);
          if constexpr (kChecked) {
            constexpr int es = kFp8 ? 1 : 2;
            const bool a_ok = kAMNMajor ? tma_start_ok(arow, kb * kBK, M, K, es)
                                        : tma_start_ok(kb * kKE, arow, K, M, es);
            bool b_ok;
            if constexpr (kFp8 && kBMNMajor) {
              b_ok = tma_start_ok(Epi::b_col(nb, 2 * static_cast<int>(rank), N), kb * kKE, N, K, es);
            } else if constexpr (kBMNMajor) {
              const int j0 = 2 * static_cast<int>(rank);
              b_ok = tma_start_ok(Epi::b_col(nb, j0, N), kb * kBK, N, K, es) &&
                     tma_start_ok(Epi::b_col(nb, j0 + 1, N), kb * kBK, N, K, es);
            } else {
              b_ok = tma_start_ok(kb * kKE, bcol, K, N, es);
            }
            if (!checked(a_ok, kChkTmaA) || !checked(b_ok, kChkTmaB)) {
              *wc.abort_flag = 1u;
              ok = false;
              break;
            }
          }
          if (leader) mbar_arrive_expect_tx(full_local, 2u * stage_bytes);
          const uint32_t a_dst = sA + s * kPairAStageBytes;
          const uint32_t b_dst = sB + s * kPairBStageBytes;
          if constexpr (kAMNMajor) {
            tma_load_2d_pair(a_dst, &tmA, full_leader, arow, kb * kBK);
            tma_load_2d_pair(a_dst + kBChunkBytes, &tmA, full_leader, arow + 64, kb * kBK);
          } else {
            tma_load_2d_pair(a_dst, &tmA, full_leader, kb * kKE, arow);
          }
          if constexpr (kFp8 && kBMNMajor) {
            // this CTA's 128 B columns (chunks 2r, 2r+1 of the tile) in one 128 x 128 box
            tma_load_2d_pair(b_dst, &tmB, full_leader, Epi::b_col(nb, 2 * static_cast<int>(rank), N),
                             kb * kKE);
          } else if constexpr (kFp8) {
            tma_load_2d_pair(b_dst, &tmB, full_leader, kb * kKE, bcol);
          } else if constexpr (kBMNMajor) {
            const int j0 = 2 * static_cast<int>(rank);  // this CTA's two 64-column chunks
            tma_load_2d_pair(b_dst, &tmB, full_leader, Epi::b_col(nb, j0, N), kb * kBK);
            tma_load_2d_pair(b_dst + kBChunkBytes, &tmB, full_leader, Epi::b_col(nb, j0 + 1, N),
                             kb * kBK);
          } else {
            tma_load_2d_pair(b_dst, &tmB, full_leader, kb * kBK, bcol);
          }
          issued_mask |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
          if (++s == kPairStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      };
      for (int t = pair; ok && t < dp_end; t += npairs) loads(WorkItem{t, 0, nk, kItemWhole});
      if constexpr (kSplit) {
        SplitWork work(pair, npairs, num_tiles, dp_end, nk);
        WorkItem w;
        while (ok && work.next(w)) loads(w);
      }
      if (kPlanCapable && pieced) {
        PieceWork work(sk, pair, npairs, num_tiles, nk);
        WorkItem w;
        while (ok && work.next(w)) loads(w);
      }
      if (!ok && leader) {
        // Let every issued copy (of both CTAs) land before the pair can exit.
        for (int i = 0; i < kPairStages; ++i)
          if (issued_mask & (1u << i)) {
            const uint32_t p = (last_par >> i) & 1u;
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar_full + 8u * i, p) && globaltimer_ns() - t0 < timeout_ns) {
            }
          }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (CTA 0 only)
    if (lane == 0) {
      if (leader) {
        constexpr uint32_t idesc_full = kFp8 ? idesc_e4m3_f32(kPairBM, kBN, false, kBMNMajor)
                                             : idesc_bf16_f32(kPairBM, kBN, kAMNMajor, kBMNMajor);
        int s = 0;
        uint32_t ph = 0;
        uint32_t it = 0;
        bool ok = true;
        const auto mmas = [&](const WorkItem& w) {
          const uint32_t b = it & 1u;
          const uint32_t aph = (it >> 1) & 1u;
          if (!bounded_wait(bar_tempty + 8u * b, aph ^ 1u, wc, kSiteMmaTmemEmpty)) {
            ok = false;
            return;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + b * kBN;
          uint32_t idesc = idesc_full;
          if (planned) {  // N of the MMA = the tile's width
            int mb, nb, n0, width;
            tmap.coords(w.tile, mb, nb);
            geometry(mb, nb, n0, width);
            idesc = idesc_bf16_f32(kPairBM, width, kAMNMajor, kBMNMajor);
          }
          for (int kb = w.kb0; kb < w.kb1; ++kb) {
            if (!bounded_wait(bar_full + 8u * s, ph, wc, kSiteMmaFull)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t a0 = sA + s * kPairAStageBytes;
            const uint32_t b0 = sB + s * kPairBStageBytes;
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k) {
              // K-major: every MMA consumes 32 bytes of each 128-byte row (16 bf16 or
              // 32 FP8 elements).  MN-major: 16 (bf16) or 32 (FP8) K rows, i.e. 2 or 4
              // eight-row groups of 1024 bytes.
              const uint64_t ad = kAMNMajor ? sdesc_sw128(a0 + k * 2048, kBChunkBytes, 1024)
                                            : sdesc_sw128(a0 + k * 32, 16, 1024);
              const uint64_t bd =
                  kBMNMajor ? sdesc_sw128(b0 + k * (kFp8 ? 4096 : 2048), kFp8 ? 16384 : kBChunkBytes,
                                          1024)
                            : sdesc_sw128(b0 + k * 32, 16, 1024);
              if constexpr (kFp8)
                umma_f8_pair(d_tmem, ad, bd, idesc, (kb != w.kb0 || k != 0) ? 1u : 0u);
              else
                umma_bf16_pair(d_tmem, ad, bd, idesc, (kb != w.kb0 || k != 0) ? 1u : 0u);
            }
            umma_commit_pair_mc(bar_empty + 8u * s, 0x3);
            if (++s == kPairStages) {
              s = 0;
              ph ^= 1u;
            }
          }
          if (!ok) return;
          umma_commit_pair_mc(bar_tfull + 8u * b, 0x3);
        };
        for (int t = pair; ok && t < dp_end; t += npairs, ++it) mmas(WorkItem{t, 0, nk, kItemWhole});
        if constexpr (kSplit) {
          SplitWork work(pair, npairs, num_tiles, dp_end, nk);
          WorkItem w;
          for (; ok && work.next(w); ++it) mmas(w);
        }
        if (kPlanCapable && pieced) {
          PieceWork work(sk, pair, npairs, num_tiles, nk);
          WorkItem w;
          for (; ok && work.next(w); ++it) mmas(w);
        }
        // Always signal `drain` in both CTAs once every MMA issued here is done.
        umma_commit_pair_mc(bar_drain, 0x3);
      }
      // Both CTAs: no TMEM release while MMAs may still write it.
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar_drain, 0)) {
        if (globaltimer_ns() - t0 > timeout_ns) {
          record_failure(wc, kSiteDrain);
          break;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = quad * 32 + lane;
    uint32_t it = 0;
    const auto drain = [&](const WorkItem& w) -> bool {
      const uint32_t b = it & 1u;
      const uint32_t aph = (it >> 1) & 1u;
      int mb, nb;
      tmap.coords(w.tile, mb, nb);
      const bool ok = bounded_wait(bar_tfull + 8u * b, aph, wc, kSiteEpiTmemFull);
      if (!epi_all(ok)) return false;
      tc_fence_after();
      if (kSplit && w.kind != kItemWhole) {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + b * kBN;
        // split tile: this CTA's 128-row half of the tile's partial slot and flag
        const size_t slot = static_cast<size_t>(w.tile - sk.dp_tiles) * 2 + rank;
        float4* part = reinterpret_cast<float4*>(sk.part + slot * kSkSlotFloats);
        uint64_t* flag = sk.flags + slot;
        if constexpr (kChecked) {
          if (!epi_all(checked(sk.part != nullptr && w.tile >= sk.dp_tiles &&
                                   slot < 2 * static_cast<size_t>(sk.slots),
                               kChkSplitSlot)))
            return false;  // leave the role (every epilogue thread agrees)
        }
        if (w.kind == kItemTail) {
          sk_write_partial(taddr, part, half, row);
          __threadfence();
          named_bar_sync(1, kEpiThreads);
          if (threadIdx.x == kEpiFirstThread) {
            st_release_gpu_u64(flag, launch_tag(sk.epoch, sk.salt));
          }
        } else {
          if (threadIdx.x == kEpiFirstThread) {
            flag_wait(flag, launch_tag(sk.epoch, sk.salt), wc, kSiteSplitTail);
            __threadfence();
          }
          named_bar_sync(1, kEpiThreads);
          sk_add_partial(taddr, part, half, row);
          // a policy may read columns another thread just wrote (SwiGLU pairs
          // column j with j + 128): all stores land before any thread reads
          tc_fence_before();
          named_bar_sync(1, kEpiThreads);
          tc_fence_after();
        }
      }
      if (kPlanCapable && w.kind != kItemWhole) {
        const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + b * kBN;
        const int p1 = sk.pieces - 1;
        const size_t first = static_cast<size_t>(w.tile - sk.dp_tiles) * p1;  // the tile's slots
        if constexpr (kChecked) {
          if (!epi_all(checked(sk.part != nullptr && w.tile >= sk.dp_tiles &&
                                   (first + p1) * 2 <= 2 * static_cast<size_t>(sk.slots),
                               kChkSplitSlot)))
            return false;  // leave the role (every epilogue thread agrees)
        }
        piece_epilogue(sk.part, sk.flags, sk.epoch, sk.salt, wc, taddr, first, p1, w.piece,
                       w.kind == kItemTail, rank, half, row);
      }
      if (w.kind != kItemTail) {
        TileCtx c;
        c.taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) + b * kBN;
        c.mb = mb * 2 + static_cast<int>(rank);  // this CTA's 128-row slab
        c.nb = nb;
        int width;
        geometry(mb, nb, c.n0, width);
        c.nend = min(N, c.n0 + width);
        c.row = row;
        c.half = half;
        c.M = M;
        c.N = N;
        c.nt = nt;
        c.stage =
            base + kPairSmemBar + 256u + static_cast<uint32_t>(warp - 2) * Epi::kStageBytesPerWarp;
        Epi::apply(ep, wc, c);
      }
      tc_fence_before();
      named_bar_sync(1, kEpiThreads);
      if (threadIdx.x == kEpiFirstThread) mbar_arrive_cluster(mapa_shared(bar_tempty + 8u * b, 0));
      return true;
    };
    bool go = true;
    for (int t = pair; go && t < dp_end; t += npairs, ++it) go = drain(WorkItem{t, 0, nk, kItemWhole});
    if constexpr (kSplit) {
      SplitWork work(pair, npairs, num_tiles, dp_end, nk);
      WorkItem w;
      for (; go && work.next(w); ++it) go = drain(w);
    }
    if (kPlanCapable && pieced) {
      PieceWork work(sk, pair, npairs, num_tiles, nk);
      WorkItem w;
      for (; go && work.next(w); ++it) go = drain(w);
    }
  }

  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc_pair(tmem_base, kTmemCols);
  }
  // Both CTAs are past their last flag access (cluster barrier above): count
  // this block out of the launch (the last one advances the launch counter).
  if (threadIdx.x == 0) {
    if ((kSplit || pieced) && sk.epoch != nullptr)
      launch_exit(sk.epoch, sk.salt);  // the data gradient's own counter is this same slot
    else
      Epi::at_exit(ep);
  }
}

}  // namespace coda
