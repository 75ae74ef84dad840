// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA, tcgen05 (TMEM + MMA).
//
// Every wait of the kernels' own protocols (mbarrier phases, completion flags
// written by other blocks) goes through bounded_wait()/flag_wait(): it gives up
// after a host-set number of nanoseconds, records a code in the library's device
// status word and returns false, so a protocol bug ends the kernel instead of
// hanging the GPU.  The end of a launch is not a wait: each block counts itself
// out with one atomic and the last one advances the launch counter
// (launch_exit below).  The one wait not bounded here is
// griddepcontrol.wait (programmatic dependent launch), which ends when the
// preceding kernel in the stream completes; every kernel of this library
// completes because all its other waits are bounded.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

namespace coda {

// ---------------------------------------------------------------------------
// addresses, timers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// True once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Status codes written to the device status word (low byte = which wait).
enum WaitSite : uint32_t {
  kSiteProducerEmpty = 1,
  kSiteMmaTmemEmpty = 2,
  kSiteMmaFull = 3,
  kSiteEpiTmemFull = 4,
  kSiteRowFlags = 5,
  kSiteDrain = 6,
  kSiteSelftestBarrier = 7,
  kSiteSelftestFlag = 8,
  kSiteSplitTail = 9,  // owner of a split tile waiting for its partial
  kSitePieces = 10,    // owner of a tile cut into K pieces waiting for the pieces' partials
};

struct WaitCtl {
  uint64_t timeout_ns;
  uint32_t* status;                // device status word (first failure wins)
  volatile uint32_t* abort_flag;   // shared-memory flag: set once any role gave up
};

__device__ __forceinline__ void record_failure(const WaitCtl& c, uint32_t site) {
  atomicCAS(c.status, 0u, 0x100u | site);
  *c.abort_flag = 1u;
}

// Bounded wait on an mbarrier phase.  Returns false if it ran out (or another
// role of this block already gave up).
__device__ __forceinline__ bool bounded_wait(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                             uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*c.abort_flag) return false;
    if (globaltimer_ns() - t0 > c.timeout_ns) {
      record_failure(c, site);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// global-memory flags (cross-block completion within one cooperative launch)
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t ld_acquire_gpu_u64(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_gpu_u64(uint64_t* p, uint64_t v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Bounded wait until *p == token.
__device__ __forceinline__ bool flag_wait(const uint64_t* p, uint64_t token, const WaitCtl& c,
                                          uint32_t site) {
  if (ld_acquire_gpu_u64(p) == token) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(32);
    if (ld_acquire_gpu_u64(p) == token) return true;
    if (globaltimer_ns() - t0 > c.timeout_ns) {
      record_failure(c, site);
      return false;
    }
  }
}

// 128-bit compare-and-swap at GPU scope (acquire-release): {lo, hi} at p becomes
// {n_lo, n_hi} if it held {e_lo, e_hi}.  Returns true on success; `o_lo`,
// `o_hi` receive the value found.
__device__ __forceinline__ bool cas128_gpu(uint64_t* p, uint64_t e_lo, uint64_t e_hi,
                                           uint64_t n_lo, uint64_t n_hi, uint64_t& o_lo,
                                           uint64_t& o_hi) {
  asm volatile(
      "{\n\t.reg .b128 d, e, n;\n\t"
      "mov.b128 e, {%2, %3};\n\t"
      "mov.b128 n, {%4, %5};\n\t"
      "atom.acq_rel.gpu.global.cas.b128 d, [%6], e, n;\n\t"
      "mov.b128 {%0, %1}, d;\n\t}"
      : "=l"(o_lo), "=l"(o_hi)
      : "l"(e_lo), "l"(e_hi), "l"(n_lo), "l"(n_hi), "l"(p)
      : "memory");
  return o_lo == e_lo && o_hi == e_hi;
}

__device__ __forceinline__ uint64_t atom_add_acq_rel_gpu_u64(uint64_t* p, uint64_t v) {
  uint64_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v)
               : "memory");
  return old;
}

// End of a launch whose blocks exchange flags tagged with a token taken from a
// launch counter (the data gradient's row flags, the split tail's partial
// flags).  `slot` is the first 256 bytes of the caller's workspace (16-byte
// aligned, any initial contents); every workspace layout of this library keeps
// it there and never writes data into it, so one counter serves every call,
// shape and entry point that shares the buffer:
//   slot[0]           launch counter; this launch's token is slot[0] + 1
//   slot[1]           kSlotReady once slot[2] has been prepared by a launch
//   slot[2]           blocks of the current launch that have finished (0 at its start)
//   slot[4], slot[5]  {token ^ salt, blocks finished}: the count of a first launch
// A flag holds token ^ salt, `salt` being a random 64-bit value the host draws
// for each call (fixed across replays of a captured call, whose tokens the
// counter keeps distinct).  Flags left by other calls, other buffers or any
// earlier contents therefore match only by a 2^-64 coincidence.
// Called by one thread per block once every thread of the block is done with
// the launch's flags.  The block that completes the count (gridDim.x) prepares
// slot[2] for the next launch and stores the token as the new launch counter,
// after which no flag of this launch is read any more.  Nothing waits.  In
// steady state each block adds 1 to slot[2] (one atomic).  On a slot not yet
// prepared (a fresh workspace) the count goes through a 128-bit
// compare-and-swap on {token ^ salt, count} (a tag that does not match
// restarts the count); every failed compare-and-swap means another block got
// in, so that loop runs at most gridDim.x + 1 times.  Only the last block
// writes slot[1], after every block has read it, so all blocks of a launch take
// the same path.
constexpr uint64_t kSlotReady = 0xC0DA5107C0DA5107ull;

// The value a flag of this launch carries.
__device__ __forceinline__ uint64_t launch_tag(const uint64_t* slot, uint64_t salt) {
  return (*reinterpret_cast<const volatile uint64_t*>(slot) + 1) ^ salt;
}

__device__ __forceinline__ void launch_exit(uint64_t* slot, uint64_t salt) {
  volatile uint64_t* vs = reinterpret_cast<volatile uint64_t*>(slot);
  const uint64_t token = vs[0] + 1;
  bool last = false;
  if (vs[1] == kSlotReady) {
    last = atom_add_acq_rel_gpu_u64(slot + 2, 1) == gridDim.x - 1;
  } else {
    const uint64_t tag = token ^ salt;
    uint64_t e_lo = vs[4], e_hi = vs[5];
    for (uint32_t i = 0; i <= gridDim.x; ++i) {
      const uint64_t n_hi = (e_lo == tag) ? e_hi + 1 : 1;
      uint64_t o_lo, o_hi;
      if (cas128_gpu(slot + 4, e_lo, e_hi, tag, n_hi, o_lo, o_hi)) {
        last = n_hi == gridDim.x;
        break;
      }
      e_lo = o_lo;
      e_hi = o_hi;
    }
  }
  if (last) {
    vs[2] = 0;
    vs[1] = kSlotReady;
    st_release_gpu_u64(slot, token);
  }
}

// Named barrier over `count` threads (ids 1.. are free; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), 2-D tiles, completion on an mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// x = innermost coordinate (elements), y = outer coordinate (rows).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format):
//   bits  0-13 start address >> 4
//   bits 16-29 leading-dimension byte offset >> 4
//   bits 32-45 stride-dimension byte offset >> 4
//   bits 46-47 descriptor version (1)
//   bits 49-51 base offset (0: every swizzle atom is 1024-byte aligned)
//   bits 61-63 layout (2 = 128-byte swizzle)
// K-major operand (rows of 64 bf16 = 128 B): SBO = 1024 (next 8-row group),
//   LBO unused (1).  One MMA consumes K = 16 = 32 bytes of each row, so a K
//   step advances the start address by 32 bytes inside the swizzle atom.
// MN-major operand (rows = K, 64 contiguous bf16 of M/N per row):
//   LBO = byte distance between 64-element M/N chunks,
//   SBO = byte distance between 8-row K groups (1024).
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulator.
//   bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format (1 = bf16),
//   bit 15 A major (0 = K), bit 16 B major (1 = MN), bits 17-22 N >> 3, bits 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on `bar` when all previously issued MMAs of this thread complete.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets lane
// (base lane + i), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}

// Waits for outstanding tcgen05.ld; the registers are tied in so that no use
// of them can be scheduled before the wait.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&v)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]),
                 "+r"(v[6]), "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]),
                 "+r"(v[12]), "+r"(v[13]), "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]),
                 "+r"(v[18]), "+r"(v[19]), "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]),
                 "+r"(v[24]), "+r"(v[25]), "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]),
                 "+r"(v[30]), "+r"(v[31])
               :
               : "memory");
}

// The store twin of tmem_ld32: thread i of the warp writes lane (base lane + i),
// columns [col, col + 32).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Waits until this thread's earlier tcgen05.st have completed.
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------------------
// bf16 packing helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

}  // namespace coda

namespace coda {

// ---------------------------------------------------------------------------
// CTA-pair (cluster of 2) variants: tcgen05 with .cta_group::2
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Shared::cluster address of the variable at shared::cta address `addr` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
  return out;
}

// All threads of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

// Arrive on an mbarrier given by its shared::cluster address (own or peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialisation: it may start while the preceding kernel in
// the stream is finishing, runs its prologue (barriers, TMEM, descriptor
// prefetch; nothing that reads another kernel's output), then waits here until
// the preceding grid has completed and its writes are visible.  Both are no-ops
// for a launch without the attribute.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream start its own prologue (it still waits for
// this grid to complete before touching memory).
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// TMA load whose completion is signalled on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map,
                                                 uint32_t bar_cluster, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// D[tmem of both CTAs] (+)= A[smem of both CTAs] * B[smem of both CTAs]; M = 256 split by
// rows across the pair, B split by its N rows/columns; issued by one thread of CTA 0.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier at the same offset in every CTA of `cta_mask` when all
// previously issued MMAs of this thread complete.
__device__ __forceinline__ void umma_commit_pair_mc(uint32_t bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(bar),
      "h"(cta_mask)
      : "memory");
}

}  // namespace coda

namespace coda {

// D[tmem of both CTAs] (+)= A * B with FP8 operands (kind::f8f6f4; K = 32 per
// instruction); same operand split across the CTA pair as umma_bf16_pair.
__device__ __forceinline__ void umma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor for kind::f8f6f4 with E4M3 A/B (format code 0) and an
// fp32 accumulator; same field positions as idesc_bf16_f32.
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int m, int n, bool a_mn_major,
                                                      bool b_mn_major) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
         (static_cast<uint32_t>(m >> 4) << 24);
}

}  // namespace coda
