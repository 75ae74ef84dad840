// coda.cu -- libcoda.so: kernels of the GEMM -> residual -> RMSNorm -> GEMM chain
// and the C ABI declared in include/coda.h.
//
// Forward (CODA blog, blog.hotdry.top, section
// "GEMM-Residual-RMSNorm-GEMM 重参数化", its three steps):
//   launch 1  GEMM0 x @ W0 with EpiResidualGammaSumsq   -> h, hg = h*gamma, partial sum h^2
//   launch 2  rowreduce_rsqrt_kernel                    -> r = 1/sqrt(sum/d + eps)
//   launch 3  GEMM1 hg @ W1 with EpiRowScale            -> y = r * acc
// Backward data gradient (section "反向传播的 GEMM-Epilogue 结构"):
//   launch 1  GEMM dy @ W1^T with EpiRmsNormBackward    -> grad_h (cooperative launch)

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <random>
#include <tuple>
#include <vector>

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "coda.h"
#include "epilogues.cuh"
#include "gemm_pair.cuh"

namespace coda {

// ---------------------------------------------------------------------------
// auxiliary kernels
// ---------------------------------------------------------------------------

// Step 2 of the forward: the light auxiliary reduction over the per-tile
// partial sums of squares (fixed summation order over tiles).
__global__ void rowreduce_rsqrt_kernel(const float* __restrict__ part, int nt, int M, int d,
                                       float eps, float* __restrict__ r) {
  griddep_launch_dependents();
  griddep_wait();
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  float s = 0.f;
  for (int t = 0; t < nt; ++t) s += __ldg(part + static_cast<size_t>(t) * M + m);
  r[m] = rsqrtf(s / static_cast<float>(d) + eps);
}

// Auxiliary reduction of the backward statistic: s[m] = sum_t spart[t][m]
// (fixed summation order over tiles).
__global__ void rowsum_kernel(const float* __restrict__ part, int nt, int M, float* __restrict__ s) {
  griddep_launch_dependents();
  griddep_wait();
  const int m = blockIdx.x * blockDim.x + threadIdx.x;
  if (m >= M) return;
  float acc = 0.f;
  for (int t = 0; t < nt; ++t) acc += __ldg(part + static_cast<size_t>(t) * M + m);
  s[m] = acc;
}

// dgamma[j] = sum_i gpart[i][j] over the per-warp column partials (fixed order).
__global__ void colsum_kernel(const float* __restrict__ part, int nrows, int d,
                              float* __restrict__ out) {
  griddep_launch_dependents();
  griddep_wait();
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= d) return;
  float acc = 0.f;
  for (int i = 0; i < nrows; ++i) acc += __ldg(part + static_cast<size_t>(i) * d + j);
  out[j] = acc;
}

// Standalone RMSNorm of the unfused reference sequence: reads h, writes
// hn = bf16(r * h * gamma) and r.  One block of 256 threads per row.
__global__ void __launch_bounds__(256) rmsnorm_rows_kernel(const __nv_bfloat16* __restrict__ h,
                                                           const __nv_bfloat16* __restrict__ gamma,
                                                           float eps, int M, int d,
                                                           __nv_bfloat16* __restrict__ hn,
                                                           float* __restrict__ r) {
  __shared__ float warp_sums[8];
  griddep_launch_dependents();
  griddep_wait();
  const int m = blockIdx.x;
  if (m >= M) return;
  const __nv_bfloat16* row = h + static_cast<size_t>(m) * d;
  const int nchunks = d / 8;
  float ss = 0.f;
  for (int i = threadIdx.x; i < nchunks; i += blockDim.x) {
    const Chunk8 c = ldg8(row + 8 * i);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float a = bf16lo(c.w[e]), b = bf16hi(c.w[e]);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += warp_sums[w];
  const float rr = rsqrtf(tot / static_cast<float>(d) + eps);
  if (threadIdx.x == 0) r[m] = rr;
  __nv_bfloat16* out = hn + static_cast<size_t>(m) * d;
  for (int i = threadIdx.x; i < nchunks; i += blockDim.x) {
    const Chunk8 c = ldg8(row + 8 * i);
    const Chunk8 g = ldg8(gamma + 8 * i);
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = pack_bf16x2(rr * bf16lo(c.w[e]) * bf16lo(g.w[e]), rr * bf16hi(c.w[e]) * bf16hi(g.w[e]));
    stg8(out + 8 * i, w);
  }
}

__device__ uint64_t g_selftest_flag = 0;  // never written by anyone

// Watchdog self-test: both waits run out by construction.
__global__ void watchdog_selftest_kernel(uint64_t timeout_ns) {
  griddep_launch_dependents();
  griddep_wait();
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t abort_flag;
  if (threadIdx.x != 0) return;
  abort_flag = 0u;
  const uint32_t b = smem_u32(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  WaitCtl wc{timeout_ns, &g_coda_status, &abort_flag};
  bounded_wait(b, 0u, wc, kSiteSelftestBarrier);  // nobody arrives
  flag_wait(&g_selftest_flag, 1ull, wc, kSiteSelftestFlag);  // nobody sets it
}

static auto* const kGemm0 = &gemm_epilogue_kernel<EpiResidualGammaSumsq, true>;
static auto* const kGemm1 = &gemm_epilogue_kernel<EpiRowScale, true>;
static auto* const kDgrad = &gemm_epilogue_kernel<EpiRmsNormBackward, false>;
static auto* const kPairGemm0 = &gemm_pair_epilogue_kernel<EpiResidualGammaSumsq, true>;
static auto* const kPairGemm1 = &gemm_pair_epilogue_kernel<EpiRowScale, true>;
static auto* const kPairDgrad = &gemm_pair_epilogue_kernel<EpiRmsNormBackward, false>;
static auto* const kDgradFull = &gemm_epilogue_kernel<EpiRmsNormBackwardFull, false>;
static auto* const kPairDgradFull = &gemm_pair_epilogue_kernel<EpiRmsNormBackwardFull, false>;
static auto* const kGemm1Swiglu = &gemm_epilogue_kernel<EpiRowScaleSwiGLU, true>;
static auto* const kPairGemm1Swiglu = &gemm_pair_epilogue_kernel<EpiRowScaleSwiGLU, true>;
static auto* const kSwigluBwd = &gemm_epilogue_kernel<EpiSwiGLUBackward, false>;
static auto* const kWgrad = &gemm_epilogue_kernel<EpiStoreF32, true, true>;
static auto* const kPairGemm0F8 = &gemm_pair_epilogue_kernel<EpiResidualGammaSumsqFp8, true, false, true>;
static auto* const kPairGemm1F8 = &gemm_pair_epilogue_kernel<EpiRowScaleFp8, true, false, true>;
static auto* const kPairWgrad = &gemm_pair_epilogue_kernel<EpiStoreF32, true, true>;
static auto* const kXgrad = &gemm_epilogue_kernel<EpiRowScale, false>;
static auto* const kPairXgrad = &gemm_pair_epilogue_kernel<EpiRowScale, false>;
static auto* const kPairSwigluBwd = &gemm_pair_epilogue_kernel<EpiSwiGLUBackward, false>;
static auto* const kDgradGivenS = &gemm_epilogue_kernel<EpiRmsNormBackwardGivenS, false>;
static auto* const kPairDgradGivenS = &gemm_pair_epilogue_kernel<EpiRmsNormBackwardGivenS, false>;

// dynamic shared memory of each kernel (ring, barriers, the policy's staging buffers)
constexpr uint32_t kGemm0Smem = cta_smem_bytes<EpiResidualGammaSumsq>();
constexpr uint32_t kGemm1Smem = cta_smem_bytes<EpiRowScale>();
constexpr uint32_t kDgradSmem = cta_smem_bytes<EpiRmsNormBackward>();
constexpr uint32_t kPairGemm0Smem = pair_smem_bytes<EpiResidualGammaSumsq>();
constexpr uint32_t kPairGemm1Smem = pair_smem_bytes<EpiRowScale>();
constexpr uint32_t kPairDgradSmem = pair_smem_bytes<EpiRmsNormBackward>();
constexpr uint32_t kDgradFullSmem = cta_smem_bytes<EpiRmsNormBackwardFull>();
constexpr uint32_t kPairDgradFullSmem = pair_smem_bytes<EpiRmsNormBackwardFull>();
constexpr uint32_t kGemm1SwigluSmem = cta_smem_bytes<EpiRowScaleSwiGLU>();
constexpr uint32_t kPairGemm1SwigluSmem = pair_smem_bytes<EpiRowScaleSwiGLU>();
constexpr uint32_t kSwigluBwdSmem = cta_smem_bytes<EpiSwiGLUBackward>();
constexpr uint32_t kWgradSmem = cta_smem_bytes<EpiStoreF32>();
constexpr uint32_t kPairGemm0F8Smem = pair_smem_bytes<EpiResidualGammaSumsqFp8>();
constexpr uint32_t kPairGemm1F8Smem = pair_smem_bytes<EpiRowScaleFp8>();
constexpr uint32_t kPairWgradSmem = pair_smem_bytes<EpiStoreF32>();
constexpr uint32_t kXgradSmem = cta_smem_bytes<EpiRowScale>();
constexpr uint32_t kPairXgradSmem = pair_smem_bytes<EpiRowScale>();
constexpr uint32_t kPairSwigluBwdSmem = pair_smem_bytes<EpiSwiGLUBackward>();
constexpr uint32_t kDgradGivenSSmem = cta_smem_bytes<EpiRmsNormBackwardGivenS>();
constexpr uint32_t kPairDgradGivenSSmem = pair_smem_bytes<EpiRmsNormBackwardGivenS>();

}  // namespace coda

// ---------------------------------------------------------------------------
// Data gradient without any allocation: scratch in a static device array.
//
// Some callers cannot call cudaMalloc (or any allocating routine) at the
// point where they run the backward: code inside a custom allocator or
// memory-pool callback, runtimes that forbid allocation while a step is in
// flight because it could synchronise the device or fragment a pre-sized
// pool, and embedders whose device memory is fully reserved up front.  For
// them this entry point takes only inputs and outputs; the partial row
// statistics and completion flags that coda_bwd_dgrad keeps in the caller's
// workspace live instead in the fixed array below, which every GPU that
// loads this library holds until the process exits.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocPartials = 2 * CODA_NOALLOC_MAX_PARTIALS;  // fp32, two per (row, column tile)
constexpr size_t kNoAllocFlags = CODA_NOALLOC_MAX_TILES;        // u64 per output tile
constexpr size_t kNoAllocFlagOffset = kNoAllocPartials * sizeof(float);
constexpr size_t kNoAllocEpochOffset = kNoAllocFlagOffset + kNoAllocFlags * sizeof(uint64_t);
constexpr size_t kNoAllocBytes = kNoAllocEpochOffset + 256;

// 4 MiB of partials + 128 KiB of flags + a 256-byte slot with the launch
// counter and its arrival word.  The flags need no clearing: each launch
// publishes counter + 1 and its last block to finish advances the counter, so
// values left by an earlier call never match (the array starts zeroed).
static __device__ __align__(256) unsigned char g_noalloc_dgrad_scratch[kNoAllocBytes];

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

using namespace coda;

constexpr int kMaxDevices = 64;
constexpr int kGroupM = 16;     // 128-row blocks per L2 group (single-CTA tiles)
constexpr int kPairGroupM = 8;  // 256-row blocks per L2 group (CTA-pair tiles)

struct DevState {
  bool init = false;
  coda_status_t status = CODA_OK;
  int sms = 0;
  int max_pairs = 0;  // co-resident clusters of two for the CTA-pair kernels
  void* noalloc_scratch = nullptr;  // device address of g_noalloc_dgrad_scratch on this device
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::atomic<uint64_t> g_timeout_ns{1000000000ull};
std::atomic<int> g_fold_rowreduce{0};  // 1: r computed in GEMM1's epilogue (no separate launch)
std::atomic<int> g_split_tail{1};      // 1: split tails in the CTA-pair GEMMs that qualify
std::atomic<int> g_mma_mode{1};  // 0: single-CTA 128x256 tiles, 1: CTA-pair 256x256 tiles (default)
cudaEvent_t* g_launch_events = nullptr;  // measurement hook (coda_set_launch_events)
int g_launch_events_n = 0;

// Records the measurement-hook event that follows launch k, if one is set.
void after_launch(int k, cudaStream_t stream) {
  if (g_launch_events != nullptr && k < g_launch_events_n) cudaEventRecord(g_launch_events[k], stream);
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Every workspace starts with the 256-byte slot of the launch counter that the
// completion flags' tokens come from (launch_exit in ptx.cuh); no layout puts
// data there, so calls of any shape and entry point may share one buffer.
constexpr size_t kSlotBytes = 256;

// A fresh random 64-bit value per call, mixed into its completion flags: the
// SplitMix64 output function (Steele, Lea and Flood, "Fast splittable
// pseudorandom number generators", OOPSLA 2014) applied to a per-process seed
// plus a counter.
uint64_t next_salt() {
  static const uint64_t seed = [] {
    uint64_t v = static_cast<uint64_t>(
        std::chrono::steady_clock::now().time_since_epoch().count());
    v ^= reinterpret_cast<uintptr_t>(&v);  // differs between processes under ASLR
    try {
      std::random_device rd;
      v ^= (static_cast<uint64_t>(rd()) << 32) ^ rd();
    } catch (...) {
      // no entropy source: the clock and the address above still differ per process
    }
    return v;
  }();
  static std::atomic<uint64_t> counter{0};
  uint64_t z = seed + 0x9E3779B97F4A7C15ull * (counter.fetch_add(1) + 1);
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  return z ^ (z >> 31);
}

// First use of the library on the current device (once per device, under a
// lock): checks the device, sets the kernels' shared-memory limits (which loads
// the library's device code on this device, the static scratch array of the
// no-allocation entry point included) and looks up the device address of that
// array, so that whichever entry point runs first on a device does both.
coda_status_t device_setup(int* sms, int* max_pairs = nullptr, void** noalloc_scratch = nullptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();
    return CODA_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& s = g_dev[dev];
  if (!s.init) {
    int major = 0, minor = 0, count = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return CODA_ERR_NO_DEVICE;
    }
    s.sms = count;
    s.status = CODA_OK;
    if (major != 10 || minor != 3) {
      s.status = CODA_ERR_UNSUPPORTED_DEVICE;
    } else {
      bool ok = true;
      ok &= cudaFuncSetAttribute(kGemm0, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kGemm0Smem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kGemm1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kGemm1Smem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kDgrad, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDgradSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairGemm0, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairGemm0Smem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairGemm1, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairGemm1Smem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairDgrad, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairDgradSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kDgradFull, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDgradFullSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairDgradFull, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairDgradFullSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kGemm1Swiglu, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kGemm1SwigluSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairGemm1Swiglu, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairGemm1SwigluSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kSwigluBwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSwigluBwdSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kWgrad, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kWgradSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairGemm0F8, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairGemm0F8Smem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairGemm1F8, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairGemm1F8Smem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairWgrad, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairWgradSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kXgrad, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kXgradSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairXgrad, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairXgradSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairSwigluBwd, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairSwigluBwdSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kDgradGivenS, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kDgradGivenSSmem) == cudaSuccess;
      ok &= cudaFuncSetAttribute(kPairDgradGivenS, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kPairDgradGivenSSmem) == cudaSuccess;
      if (ok) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (count / 2));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kPairDgradSmem;
        int clusters = 0;
        if (cudaOccupancyMaxActiveClusters(&clusters, kPairDgrad, &cfg) == cudaSuccess)
          s.max_pairs = std::min(clusters, count / 2);
        else
          ok = false;
      }
      if (g_encode == nullptr) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess && fn != nullptr) {
          g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        } else {
          ok = false;
        }
      }
      if (ok) {
        // In host code the array's name is only a host-side stand-in: its device
        // address on this device comes from the runtime.
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_dgrad_scratch) == cudaSuccess && p != nullptr)
          s.noalloc_scratch = p;
        else
          ok = false;
      }
      if (!ok) {
        cudaGetLastError();
        s.status = CODA_ERR_LAUNCH;
      }
    }
    s.init = true;
  }
  *sms = s.sms;
  if (max_pairs) *max_pairs = s.max_pairs;
  if (noalloc_scratch) *noalloc_scratch = s.noalloc_scratch;
  return s.status;
}

// 2-D bf16 tensor map over a row-major [outer, inner] matrix, 128-byte swizzle.
bool tmap_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
             uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D tensor map over a row-major [outer, inner] matrix of 1-byte (FP8) codes,
// 128-byte swizzle.
bool tmap_2d_u8(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer,
                uint32_t box_inner, uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename... ExpT, typename... ActT>
cudaError_t launch(void (*kernel)(ExpT...), int grid, int block, size_t smem, cudaStream_t stream,
                   bool cooperative, ActT&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // programmatic dependent launch for every kernel (griddep_wait in ptx.cuh)
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = 1;
  ++na;
  if (cooperative) {
    attr[na].id = cudaLaunchAttributeCooperative;
    attr[na].val.cooperative = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<ActT>(args)...);
}

coda_status_t check_common(int64_t M, int64_t d, int64_t N1) {
  if (M < 0 || d <= 0 || N1 <= 0) return CODA_ERR_INVALID_ARG;
  if (d % 8 != 0 || N1 % 8 != 0) return CODA_ERR_UNSUPPORTED_SHAPE;
  const int64_t lim = (int64_t(1) << 31) - 256;
  if (M > lim || d > lim || N1 > lim) return CODA_ERR_UNSUPPORTED_SHAPE;
  return CODA_OK;
}

// ---------------------------------------------------------------------------
// Split-tail (stream-K) region of a workspace: partial accumulators, their
// flags and the launch counter that the flags' tokens come from.
// ---------------------------------------------------------------------------
constexpr int kSkMaxPairs = 80;  // no split tail for launches of more CTA pairs

// Partial slots for launches of up to `tiles` CTA-pair tiles: a split tail
// covers U + R <= 2 U - 1 tiles.
int64_t sk_slots(int64_t tiles) { return std::min<int64_t>(tiles, 2 * kSkMaxPairs); }

size_t sk_region_bytes(int64_t tiles) {
  const int64_t slots = sk_slots(tiles);
  return align256(static_cast<size_t>(slots) * 2 * kSkSlotFloats * 4) +
         align256(static_cast<size_t>(slots) * 2 * 8);
}

struct SkRegion {
  float* part = nullptr;
  uint64_t* flags = nullptr;
  uint64_t* epoch = nullptr;
  int64_t slots = 0;
};

// `slot`: the workspace's launch-counter slot (its first 256 bytes).
SkRegion sk_region(void* base, int64_t tiles, void* slot) {
  SkRegion r;
  r.slots = sk_slots(tiles);
  char* p = static_cast<char*>(base);
  r.part = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(r.slots) * 2 * kSkSlotFloats * 4);
  r.flags = reinterpret_cast<uint64_t*>(p);
  r.epoch = static_cast<uint64_t*>(slot);
  return r;
}

// Whole tiles for the first W - 1 waves, the last U + R tiles split along K
// (gemm_pair.cuh).  The split costs a cooperative launch (measured at 2-4 us
// when it still ended with a grid barrier) and, per pair, a partial written or
// added and sometimes a wait for
// a TMEM buffer; it gains the idle share of the last wave, (U - R) / U of a
// tile.  Measured on GB300 it pays for the llama7b and llama70b GEMM1 (R/U =
// 0.16, 64 and 128 k-blocks per tile) and loses when the last wave is mostly
// full (GEMM0 there, R/U = 0.74) or tiles are short (llama1b, 32 k-blocks).  So:
// split only when R <= U / 2 and a tile has at least 64 k-blocks, with at
// least two waves and enough slots.
SkParams plan_split_tail(const SkRegion& reg, int64_t num_tiles, int npairs, int64_t nk,
                         uint64_t salt) {
  SkParams sk = kNoSplitTail;
  if (g_split_tail.load() == 0 || reg.part == nullptr || npairs < 1 || npairs > kSkMaxPairs)
    return sk;
  const int64_t W = num_tiles / npairs, R = num_tiles % npairs;
  if (W < 2 || R == 0 || 2 * R > npairs || nk < 64 || npairs + R > reg.slots) return sk;
  sk.dp_tiles = static_cast<int>(num_tiles - (npairs + R));
  sk.part = reg.part;
  sk.flags = reg.flags;
  sk.epoch = reg.epoch;
  sk.slots = static_cast<int>(reg.slots);
  sk.salt = salt;
  return sk;
}

struct FwdWorkspace {
  __nv_bfloat16* act;  // hg (fused) or hn (unfused), [M, d]
  float* part;         // [nt0][M] (fused only)
  SkRegion sk;         // split tails of GEMM0 and GEMM1 (fused only)
};

// CTA-pair tiles of the forward's larger GEMM (sizes the split-tail region)
int64_t fwd_pair_tiles(int64_t M, int64_t d, int64_t N1) {
  return cdiv(M, kPairBM) * std::max(cdiv(d, kBN), cdiv(N1, kBN));
}

// [slot | act | partials | split-tail region]
size_t fwd_ws_bytes(int64_t M, int64_t d, int64_t N1, bool fused) {
  const size_t act = align256(static_cast<size_t>(M) * d * 2);
  const size_t part = fused ? align256(static_cast<size_t>(2 * cdiv(d, kBN)) * M * 4) : 0;
  const size_t sk = fused ? sk_region_bytes(fwd_pair_tiles(M, d, N1)) : 0;
  return kSlotBytes + act + part + sk;
}

enum class FwdKind { kFused, kUnfused, kFusedSwiGLU };

coda_status_t fwd_impl(FwdKind kind, const coda_bf16* x, const coda_bf16* W0, const coda_bf16* z,
                       const coda_bf16* gamma, const coda_bf16* W1, float eps, int64_t M, int64_t d,
                       int64_t N1, coda_bf16* h_out, float* r_out, coda_bf16* y_out,
                       coda_bf16* a_out, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
  const bool fused = kind != FwdKind::kUnfused;
  const bool swiglu = kind == FwdKind::kFusedSwiGLU;
  coda_status_t st = check_common(M, d, N1);
  if (st != CODA_OK) return st;
  if (swiglu && N1 % 16 != 0) return CODA_ERR_UNSUPPORTED_SHAPE;  // N1/2 rows of 16 bytes
  if (M == 0) return CODA_OK;
  if (!x || !W0 || !z || !gamma || !W1 || !h_out || !r_out || (swiglu ? !a_out : !y_out))
    return CODA_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return CODA_ERR_INVALID_ARG;
  const void* ptrs[] = {x, W0, z, gamma, W1, h_out, r_out, swiglu ? a_out : y_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CODA_ERR_MISALIGNED;
  if (swiglu && !aligned16(y_out)) return CODA_ERR_MISALIGNED;  // optional, may be null
  if (workspace == nullptr || workspace_bytes < fwd_ws_bytes(M, d, N1, fused))
    return CODA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return CODA_ERR_MISALIGNED;
  int sms = 0, max_pairs = 0;
  st = device_setup(&sms, &max_pairs);
  if (st != CODA_OK) return st;
  const bool pair = g_mma_mode.load() == 1;

  FwdWorkspace ws;
  char* const wsb = static_cast<char*>(workspace);
  ws.act = reinterpret_cast<__nv_bfloat16*>(wsb + kSlotBytes);
  ws.part = fused ? reinterpret_cast<float*>(wsb + kSlotBytes +
                                             align256(static_cast<size_t>(M) * d * 2))
                  : nullptr;
  if (fused)
    ws.sk = sk_region(wsb + kSlotBytes + align256(static_cast<size_t>(M) * d * 2) +
                          align256(static_cast<size_t>(2 * cdiv(d, kBN)) * M * 4),
                      fwd_pair_tiles(M, d, N1), wsb);
  const uint64_t salt = next_salt();

  CUtensorMap mA0, mB0, mA1, mB1;
  bool ok = tmap_2d(&mA0, x, d, M, kBK, kBM);           // x  [M, d]  K-major
  ok &= tmap_2d(&mB0, W0, d, d, 64, kBK);               // W0 [d(K), d(N)]  MN-major
  ok &= tmap_2d(&mA1, ws.act, d, M, kBK, kBM);          // hg [M, d]  K-major
  ok &= tmap_2d(&mB1, W1, N1, d, 64, kBK);              // W1 [d(K), N1(N)] MN-major
  if (!ok) return CODA_ERR_LAUNCH;

  const int mt = static_cast<int>(cdiv(M, kBM));
  const int nt0 = static_cast<int>(cdiv(d, kBN));
  const int nt1 = swiglu ? EpiRowScaleSwiGLU::num_col_tiles(static_cast<int>(N1))
                        : static_cast<int>(cdiv(N1, kBN));
  const int Mi = static_cast<int>(M), di = static_cast<int>(d), N1i = static_cast<int>(N1);
  const uint64_t tmo = g_timeout_ns.load();

  EpiResidualGammaSumsq::Params p0 = {};
  p0.z = reinterpret_cast<const __nv_bfloat16*>(z);
  p0.gamma = reinterpret_cast<const __nv_bfloat16*>(gamma);
  p0.h_out = reinterpret_cast<__nv_bfloat16*>(h_out);
  p0.hg_out = fused ? ws.act : nullptr;
  p0.part = ws.part;
  const int mtp = static_cast<int>(cdiv(M, kPairBM));
  const int64_t nkb = cdiv(d, kBK);  // k-blocks of both GEMMs (K = d)
  const int np0 = std::min(max_pairs, mtp * nt0), np1 = std::min(max_pairs, mtp * nt1);
  const SkParams sk0 = plan_split_tail(ws.sk, static_cast<int64_t>(mtp) * nt0, np0, nkb, salt);
  const SkParams sk1 = plan_split_tail(ws.sk, static_cast<int64_t>(mtp) * nt1, np1, nkb, salt);
  cudaError_t e =
      pair ? launch(kPairGemm0, 2 * np0, kThreads, kPairGemm0Smem, stream, sk0.epoch != nullptr,
                    mA0, mB0, Mi, di, di, kPairGroupM, p0, sk0, kNoColPlan, tmo)
           : launch(kGemm0, std::min(sms, mt * nt0), kThreads, kGemm0Smem, stream, false, mA0,
                    mB0, Mi, di, di, kGroupM, p0, tmo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(0, stream);
  int k_launch = 1;
  FoldedRowReduce fold = {};
  if (fused && g_fold_rowreduce.load() == 1) {
    fold.part = ws.part;
    fold.n_part = 2 * nt0;
    fold.d = di;
    fold.eps = eps;
    fold.r_out = r_out;
  } else if (fused) {
    e = launch(rowreduce_rsqrt_kernel, static_cast<int>(cdiv(M, 256)), 256, 0, stream, false,
               static_cast<const float*>(ws.part), 2 * nt0, Mi, di, eps, r_out);
  } else {
    e = launch(rmsnorm_rows_kernel, Mi, 256, 0, stream, false,
               static_cast<const __nv_bfloat16*>(p0.h_out), p0.gamma, eps, Mi, di, ws.act, r_out);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  if (fold.part == nullptr) after_launch(k_launch++, stream);
  if (swiglu) {
    EpiRowScaleSwiGLU::Params ps = {};
    ps.r = r_out;
    ps.fold = fold;
    ps.y_out = reinterpret_cast<__nv_bfloat16*>(y_out);
    ps.a_out = reinterpret_cast<__nv_bfloat16*>(a_out);
    e = pair ? launch(kPairGemm1Swiglu, 2 * np1, kThreads, kPairGemm1SwigluSmem, stream,
                      sk1.epoch != nullptr, mA1, mB1, Mi, N1i, di, kPairGroupM, ps, sk1, kNoColPlan, tmo)
             : launch(kGemm1Swiglu, std::min(sms, mt * nt1), kThreads, kGemm1SwigluSmem,
                      stream, false, mA1, mB1, Mi, N1i, di, kGroupM, ps, tmo);
  } else {
    EpiRowScale::Params p1 = {};
    p1.r = fused ? r_out : nullptr;
    p1.fold = fold;
    p1.y_out = reinterpret_cast<__nv_bfloat16*>(y_out);
    e = pair ? launch(kPairGemm1, 2 * np1, kThreads, kPairGemm1Smem, stream, sk1.epoch != nullptr,
                      mA1, mB1, Mi, N1i, di, kPairGroupM, p1, sk1, kNoColPlan, tmo)
             : launch(kGemm1, std::min(sms, mt * nt1), kThreads, kGemm1Smem, stream, false, mA1,
                      mB1, Mi, N1i, di, kGroupM, p1, tmo);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(k_launch, stream);
  return CODA_OK;
}

// ---------------------------------------------------------------------------
// Column plans for the CTA-pair data gradient (gemm_pair.cuh, ColPlan).
// ---------------------------------------------------------------------------
// 0: 256-column tiles; 1 (2): the data gradients may use narrower column tiles
// whose widths are multiples of 16 (of 64)
std::atomic<int> g_col_plan{0};
std::atomic<int> g_dgrad_kserp{0};  // 1: the data gradients load every other wave's K backwards

// Most column tiles per row block the data-gradient workspace is sized for.
int64_t dgrad_max_col_tiles(int64_t d) { return 2 * cdiv(d, kBN); }

// Partial slots (each two CTA halves of 128 x 256 fp32) the data-gradient
// workspace holds for the pieces of its last row blocks (PieceWork): three per
// 256 x 256 tile, at most 192 (48 MiB).
int64_t dgrad_piece_slots(int64_t M, int64_t d) {
  return std::min<int64_t>(3 * cdiv(M, kPairBM) * cdiv(d, kBN), 192);
}

// The data gradient's workspace: the 256-byte slot of the launch counter, qpart
// [2 * max tiles][M] fp32, flags [slabs][max tiles] (a launch uses the first
// slabs * nt), then the pieces' partial slots and their flags.
struct DgradWs {
  uint64_t* epoch;
  float* qpart;
  uint64_t* flags;
  float* ppart;      // [pslots][2 CTAs][128 x 256]
  uint64_t* pflags;  // [pslots][2 CTAs]
  int64_t pslots;
};

// [slot | qpart | flags | piece partials | piece flags]
size_t dgrad_ws_bytes(int64_t M, int64_t d) {
  const int64_t slabs = 2 * cdiv(M, kPairBM), nt = dgrad_max_col_tiles(d);
  const int64_t ps = dgrad_piece_slots(M, d);
  return kSlotBytes + align256(static_cast<size_t>(2 * nt) * M * 4) +
         align256(static_cast<size_t>(slabs) * nt * 8) +
         align256(static_cast<size_t>(ps) * 2 * kSkSlotFloats * 4) +
         align256(static_cast<size_t>(ps) * 2 * 8);
}

DgradWs dgrad_ws(void* base, int64_t M, int64_t d) {
  const int64_t slabs = 2 * cdiv(M, kPairBM), nt = dgrad_max_col_tiles(d);
  char* p = static_cast<char*>(base);
  DgradWs w;
  w.epoch = reinterpret_cast<uint64_t*>(p);
  p += kSlotBytes;
  w.qpart = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(2 * nt) * M * 4);
  w.flags = reinterpret_cast<uint64_t*>(p);
  p += align256(static_cast<size_t>(slabs) * nt * 8);
  w.pslots = dgrad_piece_slots(M, d);
  w.ppart = reinterpret_cast<float*>(p);
  p += align256(static_cast<size_t>(w.pslots) * 2 * kSkSlotFloats * 4);
  w.pflags = reinterpret_cast<uint64_t*>(p);
  return w;
}

// ---------------------------------------------------------------------------
// Piece split of the CTA-pair data gradient's last row blocks (gemm_pair.cuh,
// PieceWork).
// ---------------------------------------------------------------------------
std::atomic<int> g_dgrad_pieces{1};  // 1: the planner below may cut the last row blocks

struct PiecePlan {
  int dp_tiles = 0, pieces = 0, lvl_first = 0, lvl = 0;
};

// The k last row blocks (R = k nt tiles, R <= npairs) cut into P pieces of at
// least 16 k-blocks, dealt as PieceWork deals them.  The model counts each
// pair's work in tiles: a whole tile 1, a piece piece_cost / P (for the data
// gradient with the row statistic 1.5: pieces finish later than their share
// of K there, because a pair's last whole tile may wait, holding one of the
// two TMEM accumulators, for its row block's tiles in the next wave, which a
// short piece after it cannot cover; 1.5 fits the GB300 measurements of 14
// shapes, 0.88 to 1.08 of the whole-tile time), plus, for the owners that
// finish the launch, about 2 us per partial they add (a k-block takes about
// 0.33 us).  A plan is taken when it shortens the busiest pair's work by at
// least 3 %.
PiecePlan plan_dgrad_pieces(int mt, int nt, int npairs, int64_t nk, int64_t slots,
                            double piece_cost = 1.5, double min_gain = 0.03) {
  PiecePlan best;
  if (npairs < 2 || nt < 1 || nk < 32) return best;
  const int64_t total = static_cast<int64_t>(mt) * nt;
  const double whole = static_cast<double>((total + npairs - 1) / npairs);
  double best_t = (1.0 - min_gain) * whole;
  for (int k = 1; k <= mt && k * nt <= npairs; ++k) {
    const int64_t R = static_cast<int64_t>(k) * nt, dp = total - R;
    const int64_t W = dp / npairs, E = dp % npairs;
    for (int P = 2; P <= 8 && nk / P >= 16; ++P) {
      if (R * (P - 1) > slots) break;
      int lvl_first = npairs, lvl = 0;
      if (E > 0) {
        lvl_first = static_cast<int>(E);
        lvl = static_cast<int>(std::min<int64_t>(P, (P - 1) * R / (npairs - E)));
      }
      const int64_t rr = R * P - static_cast<int64_t>(npairs - lvl_first) * lvl;
      if (rr < R) continue;
      double mx = 0.0;
      for (int p = 0; p < npairs; ++p) {
        const int64_t pieces = (p >= lvl_first ? lvl : 0) + rr / npairs + (p < rr % npairs ? 1 : 0);
        mx = std::max(mx, static_cast<double>(W + (p < E ? 1 : 0)) + piece_cost * pieces / P);
      }
      const double t = mx + (P - 1) * 6.0 / static_cast<double>(nk);
      if (t < best_t) {
        best_t = t;
        best.dp_tiles = static_cast<int>(dp);
        best.pieces = P;
        best.lvl_first = lvl_first;
        best.lvl = lvl;
      }
    }
  }
  return best;
}

// The piece plan of a CTA-pair data gradient of the given shape on `npairs`
// pairs: the row-statistic launch cuts whole row blocks (a piece counting 1.5
// times its share of K, at least 3 % saved); the tile-local launch of the
// SwiGLU backward cuts any last tiles (a piece counting its share, at least 1 %).
PiecePlan piece_plan_for(int64_t M, int64_t d, int64_t N1, int npairs, bool tile_local) {
  const int mt = static_cast<int>(cdiv(M, kPairBM)), nt = static_cast<int>(cdiv(d, kBN));
  const int64_t nk = cdiv(N1, kBK), slots = dgrad_piece_slots(M, d);
  return tile_local ? plan_dgrad_pieces(mt * nt, 1, npairs, nk, slots, 1.0, 0.01)
                    : plan_dgrad_pieces(mt, nt, npairs, nk, slots);
}

// The piece split's parameters for a row-statistic launch on `npairs` pairs
// (kNoSplitTail when no plan pays or the switch is off).
SkParams dgrad_pieces(const DgradWs& dw, int64_t M, int64_t d, int64_t N1, int npairs,
                      uint64_t salt) {
  SkParams sk = kNoSplitTail;
  if (g_dgrad_pieces.load() == 0) return sk;
  const PiecePlan pp = piece_plan_for(M, d, N1, npairs, false);
  if (pp.pieces == 0) return sk;
  sk.dp_tiles = pp.dp_tiles;
  sk.part = dw.ppart;
  sk.flags = dw.pflags;
  sk.epoch = dw.epoch;
  sk.slots = static_cast<int>(dw.pslots);
  sk.salt = salt;
  sk.pieces = pp.pieces;
  sk.lvl_first = pp.lvl_first;
  sk.lvl = pp.lvl;
  return sk;
}

// Largest per-pair load of a plan with tiles handed out round-robin in
// row-major order, in units of one 256-column tile; `c` is the fixed cost of a
// tile in the same unit.
double plan_load(const ColPlan& cp, int mt, int npairs, double c, std::vector<double>& load) {
  load.assign(npairs, 0.0);
  int64_t t = 0;
  for (int mb = 0; mb < mt; ++mb)
    for (int j = 0; j < cp.nt; ++j, ++t) {
      int n0, width;
      cp.tile(mb, j, n0, width);
      load[t % npairs] += width / 256.0 + c;
    }
  return *std::max_element(load.begin(), load.end());
}

struct PlanKey {
  int64_t mt, d, K;
  int npairs;
  bool operator<(const PlanKey& o) const {
    return std::tie(mt, d, K, npairs) < std::tie(o.mt, o.d, o.K, o.npairs);
  }
};
std::mutex g_plan_mu;
std::map<PlanKey, ColPlan> g_plan_cache;

// The column plan for a data gradient of mt 256-row blocks, d output columns
// and K = N1 on `npairs` CTA pairs: among 256-column tiles and every tiling
// into nt tiles (ceil(d/256) <= nt <= 2 ceil(d/256), at most npairs, so that a
// row block's tiles can all be in flight at once) of widths w and w + step
// (step 16 or 64 as the switch says, w a multiple of step, 128 <= w,
// w + step <= 256), each with its best rotation, the one whose largest
// per-pair load is smallest.  A tile's fixed cost (pipeline fill, drain,
// epilogue not hidden) is taken as 2 us against a pair's 256-column tile time
// 2 * 256 * 256 * K / (25 TFLOP/s); a plan must beat the 256-column tiling by
// 0.5 % to be taken.  Memoised per shape, pair count and step.
ColPlan plan_dgrad_cols(int64_t mt, int64_t d, int64_t K, int npairs) {
  const int mode = g_col_plan.load();
  if (mode == 0 || npairs < 2) return kNoColPlan;
  const int step = mode == 2 ? 64 : 16;
  const PlanKey key{mt, d, K, npairs * 4 + mode};
  {
    std::lock_guard<std::mutex> lock(g_plan_mu);
    auto it = g_plan_cache.find(key);
    if (it != g_plan_cache.end()) return it->second;
  }
  const double c = 2e-6 / (2.0 * 256 * 256 * static_cast<double>(K) / 25e12);
  std::vector<double> load;
  const int nt0 = static_cast<int>(cdiv(d, kBN));
  ColPlan uni = {nt0, kBN, 0, 0, 128, step};
  const double base = plan_load(uni, static_cast<int>(mt), npairs, c, load);
  ColPlan best = kNoColPlan;
  double best_load = base * (1.0 - 0.005);
  const int nt_hi = static_cast<int>(std::min<int64_t>(dgrad_max_col_tiles(d), npairs));
  for (int nt = nt0; nt <= nt_hi; ++nt) {
    int w = static_cast<int>(d / nt) / step * step;
    int nl = static_cast<int>(cdiv(d - static_cast<int64_t>(nt) * w, step));
    if (nl >= nt) {
      w += step;
      nl = 0;
    }
    if (w < 128 || w + (nl > 0 ? step : 0) > kBN) continue;
    for (int rot = 0; rot < (nl > 0 ? nt : 1); ++rot) {
      const ColPlan cp = {nt, w, nl, rot, (w + (nl > 0 ? step : 0)) / 2, step};
      const double l = plan_load(cp, static_cast<int>(mt), npairs, c, load);
      if (l < best_load - 1e-9) {
        best_load = l;
        best = cp;
      }
    }
  }
  std::lock_guard<std::mutex> lock(g_plan_mu);
  g_plan_cache[key] = best;
  return best;
}

}  // namespace

extern "C" {

size_t coda_fwd_workspace_bytes(int64_t M, int64_t d, int64_t N1) {
  if (check_common(M, d, N1) != CODA_OK || M == 0) return 0;
  return fwd_ws_bytes(M, d, N1, true);
}

size_t coda_fwd_unfused_workspace_bytes(int64_t M, int64_t d, int64_t N1) {
  if (check_common(M, d, N1) != CODA_OK || M == 0) return 0;
  return fwd_ws_bytes(M, d, N1, false);
}

size_t coda_bwd_dgrad_workspace_bytes(int64_t M, int64_t d, int64_t N1) {
  if (check_common(M, d, N1) != CODA_OK || M == 0) return 0;
  // one flag per (128-row slab, column tile); CTA-pair tiles cover 2 * ceil(M/256) slabs
  // and a column plan cuts a row block into at most twice ceil(d/256) tiles; then the
  // launch counter's 256-byte slot
  return dgrad_ws_bytes(M, d);
}

coda_status_t coda_fwd(const coda_bf16* x, const coda_bf16* W0, const coda_bf16* z,
                       const coda_bf16* gamma, const coda_bf16* W1, float eps, int64_t M, int64_t d,
                       int64_t N1, coda_bf16* h_out, float* r_out, coda_bf16* y_out,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return fwd_impl(FwdKind::kFused, x, W0, z, gamma, W1, eps, M, d, N1, h_out, r_out, y_out,
                  nullptr, workspace, workspace_bytes, stream);
}

coda_status_t coda_fwd_swiglu(const coda_bf16* x, const coda_bf16* W0, const coda_bf16* z,
                              const coda_bf16* gamma, const coda_bf16* W1, float eps, int64_t M,
                              int64_t d, int64_t N1, coda_bf16* h_out, float* r_out,
                              coda_bf16* y_out, coda_bf16* a_out, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  return fwd_impl(FwdKind::kFusedSwiGLU, x, W0, z, gamma, W1, eps, M, d, N1, h_out, r_out, y_out,
                  a_out, workspace, workspace_bytes, stream);
}

coda_status_t coda_fwd_unfused(const coda_bf16* x, const coda_bf16* W0, const coda_bf16* z,
                               const coda_bf16* gamma, const coda_bf16* W1, float eps, int64_t M,
                               int64_t d, int64_t N1, coda_bf16* h_out, float* r_out,
                               coda_bf16* y_out, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream) {
  return fwd_impl(FwdKind::kUnfused, x, W0, z, gamma, W1, eps, M, d, N1, h_out, r_out, y_out,
                  nullptr, workspace, workspace_bytes, stream);
}

coda_status_t coda_bwd_dgrad(const coda_bf16* dy, const coda_bf16* W1, const coda_bf16* h,
                             const float* r, const coda_bf16* gamma, int64_t M, int64_t d,
                             int64_t N1, coda_bf16* dh_out, void* workspace, size_t workspace_bytes,
                             cudaStream_t stream) {
  coda_status_t st = check_common(M, d, N1);
  if (st != CODA_OK) return st;
  if (M == 0) return CODA_OK;
  if (!dy || !W1 || !h || !r || !gamma || !dh_out) return CODA_ERR_INVALID_ARG;
  const void* ptrs[] = {dy, W1, h, r, gamma, dh_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CODA_ERR_MISALIGNED;
  if (workspace == nullptr || workspace_bytes < coda_bwd_dgrad_workspace_bytes(M, d, N1))
    return CODA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return CODA_ERR_MISALIGNED;
  int sms = 0, max_pairs = 0;
  st = device_setup(&sms, &max_pairs);
  if (st != CODA_OK) return st;
  const bool pair = g_mma_mode.load() == 1;

  // Row-major tile order; every column tile of a row block must be in flight
  // at once (at most one wave per row block), see EpiRmsNormBackward.
  const int mt = static_cast<int>(cdiv(M, pair ? kPairBM : kBM));
  ColPlan cp = pair ? plan_dgrad_cols(mt, d, N1, max_pairs) : kNoColPlan;
  cp.kserp = g_dgrad_kserp.load();
  const int nt = cp.nt > 0 ? cp.nt : static_cast<int>(cdiv(d, kBN));
  int units = pair ? std::min(max_pairs, mt * nt) : std::min(sms, mt * nt);
  if (nt > units) return CODA_ERR_UNSUPPORTED_SHAPE;

  CUtensorMap mA, mB;
  bool ok = tmap_2d(&mA, dy, N1, M, kBK, kBM);                  // dy [M, N1] K-major (K = N1)
  ok &= tmap_2d(&mB, W1, N1, d, kBK, pair ? cp.b_rows : kBN);   // W1 [d(N), N1(K)] K-major
  if (!ok) return CODA_ERR_LAUNCH;

  const DgradWs dw = dgrad_ws(workspace, M, d);
  const uint64_t salt = next_salt();
  // the last row blocks cut into K pieces, when the planner finds it pays (every pair runs)
  const SkParams sk =
      (pair && cp.nt == 0) ? dgrad_pieces(dw, M, d, N1, max_pairs, salt) : kNoSplitTail;
  if (sk.pieces > 0) units = max_pairs;
  EpiRmsNormBackward::Params p = {};
  p.h = reinterpret_cast<const __nv_bfloat16*>(h);
  p.gamma = reinterpret_cast<const __nv_bfloat16*>(gamma);
  p.r = r;
  p.dh_out = reinterpret_cast<__nv_bfloat16*>(dh_out);
  p.qpart = dw.qpart;
  p.flags = dw.flags;
  p.epoch = dw.epoch;
  p.salt = salt;
  cudaError_t e =
      pair ? launch(kPairDgrad, 2 * units, kThreads, kPairDgradSmem, stream, true, mA, mB,
                    static_cast<int>(M), static_cast<int>(d), static_cast<int>(N1), 1, p, sk, cp,
                    g_timeout_ns.load())
           : launch(kDgrad, units, kThreads, kDgradSmem, stream, true, mA, mB,
                    static_cast<int>(M), static_cast<int>(d), static_cast<int>(N1), 1, p,
                    g_timeout_ns.load());
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(0, stream);
  return CODA_OK;
}

size_t coda_fwd_fp8_workspace_bytes(int64_t M, int64_t d, int64_t N1) {
  if (check_common(M, d, N1) != CODA_OK || M == 0) return 0;
  return kSlotBytes + align256(static_cast<size_t>(M) * d) +
         align256(static_cast<size_t>(2 * cdiv(d, kBN)) * M * 4);
}

coda_status_t coda_fwd_fp8(const uint8_t* x_q, float sx, const uint8_t* W0_q, float sW0,
                           const coda_bf16* z, const coda_bf16* gamma, const uint8_t* W1_q,
                           float sW1, float s_hg, float eps, int64_t M, int64_t d, int64_t N1,
                           coda_bf16* h_out, float* r_out, coda_bf16* y_out, void* workspace,
                           size_t workspace_bytes, cudaStream_t stream) {
  coda_status_t st = check_common(M, d, N1);
  if (st != CODA_OK) return st;
  if (d % 16 != 0 || N1 % 16 != 0) return CODA_ERR_UNSUPPORTED_SHAPE;  // 16-byte FP8 rows
  if (M == 0) return CODA_OK;
  if (!x_q || !W0_q || !z || !gamma || !W1_q || !h_out || !r_out || !y_out)
    return CODA_ERR_INVALID_ARG;
  const float scales[] = {sx, sW0, sW1, s_hg};
  for (float v : scales)
    if (!std::isfinite(v) || !(v > 0.f)) return CODA_ERR_INVALID_ARG;
  if (!std::isfinite(eps) || eps < 0.f) return CODA_ERR_INVALID_ARG;
  const void* ptrs[] = {x_q, W0_q, z, gamma, W1_q, h_out, r_out, y_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CODA_ERR_MISALIGNED;
  if (workspace == nullptr || workspace_bytes < coda_fwd_fp8_workspace_bytes(M, d, N1))
    return CODA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return CODA_ERR_MISALIGNED;
  int sms = 0, max_pairs = 0;
  st = device_setup(&sms, &max_pairs);
  if (st != CODA_OK) return st;
  const uint64_t tmo = g_timeout_ns.load();
  const int Mi = static_cast<int>(M), di = static_cast<int>(d), N1i = static_cast<int>(N1);
  uint8_t* hq = static_cast<uint8_t*>(workspace) + kSlotBytes;
  float* part = reinterpret_cast<float*>(static_cast<char*>(workspace) + kSlotBytes +
                                         align256(static_cast<size_t>(M) * d));

  CUtensorMap mA0, mB0, mA1, mB1;
  bool ok = tmap_2d_u8(&mA0, x_q, d, M, 128, 128);    // x  [M, d] codes, K-major
  ok &= tmap_2d_u8(&mB0, W0_q, d, d, 128, 128);       // W0 [d(K), d(N)], MN-major
  ok &= tmap_2d_u8(&mA1, hq, d, M, 128, 128);         // hq [M, d], K-major
  ok &= tmap_2d_u8(&mB1, W1_q, N1, d, 128, 128);      // W1 [d(K), N1(N)], MN-major
  if (!ok) return CODA_ERR_LAUNCH;

  const int mtp = static_cast<int>(cdiv(M, kPairBM));
  const int nt0 = static_cast<int>(cdiv(d, kBN));
  const int nt1 = static_cast<int>(cdiv(N1, kBN));
  EpiResidualGammaSumsqFp8::Params p0 = {};
  p0.z = reinterpret_cast<const __nv_bfloat16*>(z);
  p0.gamma = reinterpret_cast<const __nv_bfloat16*>(gamma);
  p0.h_out = reinterpret_cast<__nv_bfloat16*>(h_out);
  p0.hq_out = hq;
  p0.part = part;
  p0.acc_scale = sx * sW0;
  p0.inv_s_hg = 1.0f / s_hg;
  cudaError_t e = launch(kPairGemm0F8, 2 * std::min(max_pairs, mtp * nt0), kThreads,
                         kPairGemm0F8Smem, stream, false, mA0, mB0, Mi, di, di, kPairGroupM, p0, kNoSplitTail,
                         kNoColPlan, tmo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(0, stream);
  e = launch(rowreduce_rsqrt_kernel, static_cast<int>(cdiv(M, 256)), 256, 0, stream, false,
             static_cast<const float*>(part), 2 * nt0, Mi, di, eps, r_out);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(1, stream);
  EpiRowScaleFp8::Params p1 = {};
  p1.r = r_out;
  p1.y_out = reinterpret_cast<__nv_bfloat16*>(y_out);
  p1.scale = s_hg * sW1;
  e = launch(kPairGemm1F8, 2 * std::min(max_pairs, mtp * nt1), kThreads, kPairGemm1F8Smem, stream,
             false, mA1, mB1, Mi, N1i, di, kPairGroupM, p1, kNoSplitTail, kNoColPlan, tmo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(2, stream);
  return CODA_OK;
}

// CTA-pair tiles of the full backward's largest split-capable GEMM (dW1, dx or
// dW0), which sizes its split-tail region
int64_t bwd_pair_tiles(int64_t M, int64_t d, int64_t N1) {
  return std::max(cdiv(d, kPairBM) * cdiv(std::max(d, N1), kBN), cdiv(M, kPairBM) * cdiv(d, kBN));
}

size_t coda_bwd_workspace_bytes(int64_t M, int64_t d, int64_t N1) {
  if (check_common(M, d, N1) != CODA_OK || M == 0) return 0;
  const int64_t slabs = std::max(2 * cdiv(M, kPairBM), cdiv(M, kBM));
  return coda_bwd_dgrad_workspace_bytes(M, d, N1) + align256(static_cast<size_t>(M) * d * 2) +
         align256(static_cast<size_t>(4 * slabs) * d * 4) + sk_region_bytes(bwd_pair_tiles(M, d, N1));
}

coda_status_t coda_bwd(const coda_bf16* dy, const coda_bf16* x, const coda_bf16* W0,
                       const coda_bf16* W1, const coda_bf16* h, const float* r,
                       const coda_bf16* gamma, const coda_bf16* dh_res, int64_t M, int64_t d,
                       int64_t N1, coda_bf16* dh_out, coda_bf16* dx_out, float* dgamma_out,
                       float* dW0_out, float* dW1_out, void* workspace, size_t workspace_bytes,
                       cudaStream_t stream) {
  coda_status_t st = check_common(M, d, N1);
  if (st != CODA_OK) return st;
  if (M == 0) return CODA_OK;
  if (!dy || !x || !W0 || !W1 || !h || !r || !gamma || !dh_out || !dx_out || !dgamma_out ||
      !dW0_out || !dW1_out)
    return CODA_ERR_INVALID_ARG;
  const void* ptrs[] = {dy, x, W0, W1, h, r, gamma, dh_out, dx_out, dgamma_out, dW0_out, dW1_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CODA_ERR_MISALIGNED;
  if (dh_res != nullptr && !aligned16(dh_res)) return CODA_ERR_MISALIGNED;
  if (workspace == nullptr || workspace_bytes < coda_bwd_workspace_bytes(M, d, N1))
    return CODA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return CODA_ERR_MISALIGNED;
  int sms = 0, max_pairs = 0;
  st = device_setup(&sms, &max_pairs);
  if (st != CODA_OK) return st;
  const bool pair = g_mma_mode.load() == 1;
  const uint64_t tmo = g_timeout_ns.load();
  const int Mi = static_cast<int>(M), di = static_cast<int>(d), N1i = static_cast<int>(N1);

  const int nt = static_cast<int>(cdiv(d, kBN));  // 256-column tiles of the GEMMs with N = d
  const int mt = static_cast<int>(cdiv(M, pair ? kPairBM : kBM));
  // launch 1 (the data gradient) may cut its row blocks into a column plan's tiles
  ColPlan cp = pair ? plan_dgrad_cols(mt, d, N1, max_pairs) : kNoColPlan;
  cp.kserp = g_dgrad_kserp.load();
  const int nt1 = cp.nt > 0 ? cp.nt : nt;
  int units = pair ? std::min(max_pairs, mt * nt1) : std::min(sms, mt * nt1);
  if (nt1 > units) return CODA_ERR_UNSUPPORTED_SHAPE;
  const int slabs = pair ? 2 * mt : mt;

  char* ws = static_cast<char*>(workspace);
  const DgradWs dw = dgrad_ws(ws, M, d);
  char* rest = ws + coda_bwd_dgrad_workspace_bytes(M, d, N1);
  __nv_bfloat16* h2 = reinterpret_cast<__nv_bfloat16*>(rest);
  float* gpart = reinterpret_cast<float*>(rest + align256(static_cast<size_t>(M) * d * 2));
  const SkRegion skr =
      sk_region(rest + align256(static_cast<size_t>(M) * d * 2) +
                    align256(static_cast<size_t>(4 * std::max(2 * cdiv(M, kPairBM), cdiv(M, kBM))) *
                             d * 4),
                bwd_pair_tiles(M, d, N1), dw.epoch);
  const uint64_t salt = next_salt();

  const uint32_t bbox = pair ? 128 : kBN;
  CUtensorMap mDy, mW1, mH2, mDyMN, mDh, mW0, mX, mDhMN;
  bool ok = tmap_2d(&mDy, dy, N1, M, kBK, kBM);     // dy [M, N1] K-major (dgrad)
  ok &= tmap_2d(&mW1, W1, N1, d, kBK, pair ? cp.b_rows : kBN);  // W1 [d(N), N1(K)] K-major
  ok &= tmap_2d(&mH2, h2, d, M, 64, kBK);           // h2^T: [M(K), d(M)] MN-major A
  ok &= tmap_2d(&mDyMN, dy, N1, M, 64, kBK);        // dy: [M(K), N1(N)] MN-major B
  ok &= tmap_2d(&mDh, dh_out, d, M, kBK, kBM);      // dh [M, d] K-major A
  ok &= tmap_2d(&mW0, W0, d, d, kBK, bbox);         // W0 [d_in(N), d_out(K)] K-major B
  ok &= tmap_2d(&mX, x, d, M, 64, kBK);             // x^T: [M(K), d(M)] MN-major A
  ok &= tmap_2d(&mDhMN, dh_out, d, M, 64, kBK);     // dh: [M(K), d(N)] MN-major B
  if (!ok) return CODA_ERR_LAUNCH;

  // 1. dgrad + RMSNorm backward + residual gradient + h2 + dgamma partials
  EpiRmsNormBackwardFull::Params p = {};
  p.h = reinterpret_cast<const __nv_bfloat16*>(h);
  p.gamma = reinterpret_cast<const __nv_bfloat16*>(gamma);
  p.r = r;
  p.dh_out = reinterpret_cast<__nv_bfloat16*>(dh_out);
  p.qpart = dw.qpart;
  p.flags = dw.flags;
  p.epoch = dw.epoch;
  p.salt = salt;
  const SkParams skd =
      (pair && cp.nt == 0) ? dgrad_pieces(dw, M, d, N1, max_pairs, salt) : kNoSplitTail;
  if (skd.pieces > 0) units = max_pairs;
  p.dh_res = reinterpret_cast<const __nv_bfloat16*>(dh_res);
  p.h2_out = h2;
  p.gpart = gpart;
  cudaError_t e = pair ? launch(kPairDgradFull, 2 * units, kThreads, kPairDgradFullSmem, stream,
                                true, mDy, mW1, Mi, di, N1i, 1, p, skd, cp, tmo)
                       : launch(kDgradFull, units, kThreads, kDgradFullSmem, stream, true, mDy, mW1,
                                Mi, di, N1i, 1, p, tmo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(0, stream);
  // 2. dgamma = column sums of the partials
  e = launch(colsum_kernel, static_cast<int>(cdiv(d, 256)), 256, 0, stream, false,
             static_cast<const float*>(gpart), 4 * slabs, di, dgamma_out);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(1, stream);
  // 3. dW1 = h2^T dy   (K = tokens)
  EpiStoreF32::Params pw1 = {};
  pw1.out = dW1_out;
  const int mtw = static_cast<int>(cdiv(d, pair ? kPairBM : kBM));
  const int ntw1 = static_cast<int>(cdiv(N1, kBN));
  const int64_t nkw = cdiv(M, kBK);  // k-blocks of the weight gradients (K = tokens)
  const int npw1 = std::min(max_pairs, mtw * ntw1);
  const SkParams skw1 = plan_split_tail(skr, static_cast<int64_t>(mtw) * ntw1, npw1, nkw, salt);
  e = pair ? launch(kPairWgrad, 2 * npw1, kThreads, kPairWgradSmem, stream, skw1.epoch != nullptr,
                    mH2, mDyMN, di, N1i, Mi, kPairGroupM, pw1, skw1, kNoColPlan, tmo)
           : launch(kWgrad, std::min(sms, mtw * ntw1), kThreads, kWgradSmem, stream, false, mH2,
                    mDyMN, di, N1i, Mi, kGroupM, pw1, tmo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(2, stream);
  // 4. dx = dh W0^T
  EpiRowScale::Params px = {};
  px.r = nullptr;
  px.y_out = reinterpret_cast<__nv_bfloat16*>(dx_out);
  const int mtx = static_cast<int>(cdiv(M, pair ? kPairBM : kBM));
  const int npx = std::min(max_pairs, mtx * nt);
  const SkParams skx =
      plan_split_tail(skr, static_cast<int64_t>(mtx) * nt, npx, cdiv(d, kBK), salt);
  e = pair ? launch(kPairXgrad, 2 * npx, kThreads, kPairXgradSmem, stream, skx.epoch != nullptr,
                    mDh, mW0, Mi, di, di, kPairGroupM, px, skx, kNoColPlan, tmo)
           : launch(kXgrad, std::min(sms, mtx * nt), kThreads, kXgradSmem, stream, false, mDh,
                    mW0, Mi, di, di, kGroupM, px, tmo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(3, stream);
  // 5. dW0 = x^T dh   (K = tokens)
  EpiStoreF32::Params pw0 = {};
  pw0.out = dW0_out;
  const int npw0 = std::min(max_pairs, mtw * nt);
  const SkParams skw0 = plan_split_tail(skr, static_cast<int64_t>(mtw) * nt, npw0, nkw, salt);
  e = pair ? launch(kPairWgrad, 2 * npw0, kThreads, kPairWgradSmem, stream, skw0.epoch != nullptr,
                    mX, mDhMN, di, di, Mi, kPairGroupM, pw0, skw0, kNoColPlan, tmo)
           : launch(kWgrad, std::min(sms, mtw * nt), kThreads, kWgradSmem, stream, false, mX,
                    mDhMN, di, di, Mi, kGroupM, pw0, tmo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(4, stream);
  return CODA_OK;
}

// [slot | s-partials | piece partials | piece flags]: launch 3 (the tile-local
// data gradient) may cut its last tiles into K pieces, like the data gradient.
size_t swiglu_spart_bytes(int64_t M, int64_t N1) {
  return align256(static_cast<size_t>(2 * cdiv(N1 / 2, kBN)) * M * 4);
}

size_t coda_bwd_swiglu_dgrad_workspace_bytes(int64_t M, int64_t d, int64_t N1, int64_t Dout) {
  if (check_common(M, d, N1) != CODA_OK || Dout <= 0 || M == 0) return 0;
  const int64_t ps = dgrad_piece_slots(M, d);
  return kSlotBytes + swiglu_spart_bytes(M, N1) +
         align256(static_cast<size_t>(ps) * 2 * kSkSlotFloats * 4) +
         align256(static_cast<size_t>(ps) * 2 * 8);
}

coda_status_t coda_bwd_swiglu_dgrad(const coda_bf16* dout, const coda_bf16* W2, const coda_bf16* y,
                                    const coda_bf16* W1, const coda_bf16* h, const float* r,
                                    const coda_bf16* gamma, int64_t M, int64_t d, int64_t N1,
                                    int64_t Dout, coda_bf16* dy_out, float* s_out,
                                    coda_bf16* dh_out, void* workspace, size_t workspace_bytes,
                                    cudaStream_t stream) {
  coda_status_t st = check_common(M, d, N1);
  if (st != CODA_OK) return st;
  if (Dout <= 0) return CODA_ERR_INVALID_ARG;
  if (N1 % 16 != 0 || Dout % 8 != 0 || Dout > (int64_t(1) << 31) - 256)
    return CODA_ERR_UNSUPPORTED_SHAPE;
  if (M == 0) return CODA_OK;
  if (!dout || !W2 || !y || !W1 || !h || !r || !gamma || !dy_out || !s_out || !dh_out)
    return CODA_ERR_INVALID_ARG;
  const void* ptrs[] = {dout, W2, y, W1, h, r, gamma, dy_out, s_out, dh_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CODA_ERR_MISALIGNED;
  if (workspace == nullptr ||
      workspace_bytes < coda_bwd_swiglu_dgrad_workspace_bytes(M, d, N1, Dout))
    return CODA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned16(workspace)) return CODA_ERR_MISALIGNED;
  int sms = 0, max_pairs = 0;
  st = device_setup(&sms, &max_pairs);
  if (st != CODA_OK) return st;
  const bool pair = g_mma_mode.load() == 1;
  const int64_t half = N1 / 2;
  const int Mi = static_cast<int>(M), di = static_cast<int>(d), N1i = static_cast<int>(N1);
  const int halfi = static_cast<int>(half), Douti = static_cast<int>(Dout);
  const uint64_t tmo = g_timeout_ns.load();

  CUtensorMap mA0, mB0, mA1, mB1;
  const uint32_t bbox = pair ? 128 : kBN;
  bool ok = tmap_2d(&mA0, dout, Dout, M, kBK, kBM);   // dout [M, Dout]       K-major (K = Dout)
  ok &= tmap_2d(&mB0, W2, Dout, half, kBK, bbox);     // W2 [half(N), Dout(K)] K-major
  ok &= tmap_2d(&mA1, dy_out, N1, M, kBK, kBM);       // dy [M, N1]           K-major (K = N1)
  ok &= tmap_2d(&mB1, W1, N1, d, kBK, bbox);          // W1 [d(N), N1(K)]      K-major
  if (!ok) return CODA_ERR_LAUNCH;

  const int nts = static_cast<int>(cdiv(half, kBN));
  const int ntd = static_cast<int>(cdiv(d, kBN));
  const int mt = static_cast<int>(cdiv(M, kBM));
  const int mtp = static_cast<int>(cdiv(M, kPairBM));

  // 1. down-projection data gradient with the SwiGLU backward + partial s
  EpiSwiGLUBackward::Params p0 = {};
  p0.y = reinterpret_cast<const __nv_bfloat16*>(y);
  p0.dy_out = reinterpret_cast<__nv_bfloat16*>(dy_out);
  p0.spart = reinterpret_cast<float*>(static_cast<char*>(workspace) + kSlotBytes);
  cudaError_t e =
      pair ? launch(kPairSwigluBwd, 2 * std::min(max_pairs, mtp * nts), kThreads,
                    kPairSwigluBwdSmem, stream, false, mA0, mB0, Mi, halfi, Douti, kPairGroupM,
                    p0, kNoSplitTail, kNoColPlan, tmo)
           : launch(kSwigluBwd, std::min(sms, mt * nts), kThreads, kSwigluBwdSmem, stream, false,
                    mA0, mB0, Mi, halfi, Douti, kGroupM, p0, tmo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(0, stream);
  // 2. light auxiliary reduction of the statistic
  e = launch(rowsum_kernel, static_cast<int>(cdiv(M, 256)), 256, 0, stream, false,
             static_cast<const float*>(p0.spart), 2 * nts, Mi, s_out);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(1, stream);
  // 3. RMSNorm-branch data gradient, tile-local with s given; its last tiles may
  // be cut into K pieces (any tiles: no row statistic ties them together)
  EpiRmsNormBackwardGivenS::Params p1 = {};
  p1.h = reinterpret_cast<const __nv_bfloat16*>(h);
  p1.gamma = reinterpret_cast<const __nv_bfloat16*>(gamma);
  p1.r = r;
  p1.s = s_out;
  p1.dh_out = reinterpret_cast<__nv_bfloat16*>(dh_out);
  SkParams sk3 = kNoSplitTail;
  if (pair && g_dgrad_pieces.load() != 0) {
    const int64_t pslots = dgrad_piece_slots(M, d);
    const PiecePlan pp = piece_plan_for(M, d, N1, max_pairs, true);
    if (pp.pieces > 0) {
      char* pbase = static_cast<char*>(workspace) + kSlotBytes + swiglu_spart_bytes(M, N1);
      sk3.dp_tiles = pp.dp_tiles;
      sk3.part = reinterpret_cast<float*>(pbase);
      sk3.flags = reinterpret_cast<uint64_t*>(
          pbase + align256(static_cast<size_t>(pslots) * 2 * kSkSlotFloats * 4));
      sk3.epoch = static_cast<uint64_t*>(workspace);
      sk3.slots = static_cast<int>(pslots);
      sk3.salt = next_salt();
      sk3.pieces = pp.pieces;
      sk3.lvl_first = pp.lvl_first;
      sk3.lvl = pp.lvl;
    }
  }
  const int units3 = sk3.pieces > 0 ? max_pairs : std::min(max_pairs, mtp * ntd);
  e = pair ? launch(kPairDgradGivenS, 2 * units3, kThreads, kPairDgradGivenSSmem, stream,
                    sk3.pieces > 0, mA1, mB1, Mi, di, N1i, kPairGroupM, p1, sk3, kNoColPlan, tmo)
           : launch(kDgradGivenS, std::min(sms, mt * ntd), kThreads, kDgradGivenSSmem, stream,
                    false, mA1, mB1, Mi, di, N1i, kGroupM, p1, tmo);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  after_launch(2, stream);
  return CODA_OK;
}

coda_status_t coda_get_device_status(cudaStream_t stream, uint32_t* detail) {
  if (detail) *detail = 0;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_NO_DEVICE;
  }
  if (cudaStreamSynchronize(stream) != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  uint32_t v = 0;
  if (cudaMemcpyFromSymbol(&v, coda::g_coda_status, sizeof(v)) != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  if (v != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(coda::g_coda_status, &zero, sizeof(zero)) != cudaSuccess) {
      cudaGetLastError();
      return CODA_ERR_LAUNCH;
    }
  }
  if (detail) *detail = v;
  if (v == 0) return CODA_OK;
  return (v & 0x200u) ? CODA_ERR_DEVICE_BOUNDS : CODA_ERR_DEVICE_TIMEOUT;
}

void coda_set_launch_events(cudaEvent_t* events, int n) {
  g_launch_events = (n > 0) ? events : nullptr;
  g_launch_events_n = (n > 0) ? n : 0;
}

coda_status_t coda_set_mma_mode(int mode) {
  if (mode != 0 && mode != 1) return CODA_ERR_INVALID_ARG;
  g_mma_mode.store(mode);
  return CODA_OK;
}

int coda_get_mma_mode(void) { return g_mma_mode.load(); }

coda_status_t coda_set_split_tail(int enable) {
  if (enable != 0 && enable != 1) return CODA_ERR_INVALID_ARG;
  g_split_tail.store(enable);
  return CODA_OK;
}

coda_status_t coda_set_col_plan(int enable) {
  if (enable < 0 || enable > 2) return CODA_ERR_INVALID_ARG;
  g_col_plan.store(enable);
  return CODA_OK;
}

coda_status_t coda_set_serpentine_k(int enable) {
  if (enable != 0 && enable != 1) return CODA_ERR_INVALID_ARG;
  g_dgrad_kserp.store(enable);
  return CODA_OK;
}

int coda_get_serpentine_k(void) { return g_dgrad_kserp.load(); }

coda_status_t coda_set_dgrad_pieces(int enable) {
  if (enable != 0 && enable != 1) return CODA_ERR_INVALID_ARG;
  g_dgrad_pieces.store(enable);
  return CODA_OK;
}

int coda_get_dgrad_pieces(void) { return g_dgrad_pieces.load(); }

int coda_dgrad_piece_plan(int64_t M, int64_t d, int64_t N1, int npairs, int tile_local,
                          int32_t* plan) {
  if (plan == nullptr || npairs < 1 || check_common(M, d, N1) != CODA_OK || M == 0) return -1;
  const PiecePlan pp = piece_plan_for(M, d, N1, npairs, tile_local != 0);
  plan[0] = pp.dp_tiles;
  plan[1] = pp.pieces;
  plan[2] = pp.lvl_first;
  plan[3] = pp.lvl;
  return pp.pieces > 0 ? 1 : 0;
}

coda_status_t coda_set_fold_rowreduce(int enable) {
  if (enable != 0 && enable != 1) return CODA_ERR_INVALID_ARG;
  g_fold_rowreduce.store(enable);
  return CODA_OK;
}

void coda_set_wait_timeout_ns(uint64_t ns) { g_timeout_ns.store(ns == 0 ? 1 : ns); }

const char* coda_status_string(coda_status_t s) {
  switch (s) {
    case CODA_OK: return "CODA_OK";
    case CODA_ERR_INVALID_ARG: return "CODA_ERR_INVALID_ARG";
    case CODA_ERR_UNSUPPORTED_SHAPE: return "CODA_ERR_UNSUPPORTED_SHAPE";
    case CODA_ERR_MISALIGNED: return "CODA_ERR_MISALIGNED";
    case CODA_ERR_WORKSPACE_TOO_SMALL: return "CODA_ERR_WORKSPACE_TOO_SMALL";
    case CODA_ERR_LAUNCH: return "CODA_ERR_LAUNCH";
    case CODA_ERR_DEVICE_TIMEOUT: return "CODA_ERR_DEVICE_TIMEOUT";
    case CODA_ERR_NO_DEVICE: return "CODA_ERR_NO_DEVICE";
    case CODA_ERR_UNSUPPORTED_DEVICE: return "CODA_ERR_UNSUPPORTED_DEVICE";
    case CODA_ERR_DEVICE_BOUNDS: return "CODA_ERR_DEVICE_BOUNDS";
  }
  return "CODA_ERR_UNKNOWN";
}

coda_status_t coda_watchdog_selftest(uint64_t timeout_ns, cudaStream_t stream) {
  int sms = 0;
  coda_status_t st = device_setup(&sms);
  if (st != CODA_OK) return st;
  cudaError_t e = launch(coda::watchdog_selftest_kernel, 1, 32, 0, stream, false, timeout_ns);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  return CODA_OK;
}

}  // extern "C"

extern "C" coda_status_t coda_bwd_dgrad_noalloc(const coda_bf16* dy, const coda_bf16* W1,
                                                const coda_bf16* h, const float* r,
                                                const coda_bf16* gamma, int64_t M, int64_t d,
                                                int64_t N1, coda_bf16* dh_out,
                                                cudaStream_t stream) {
  coda_status_t st = check_common(M, d, N1);
  if (st != CODA_OK) return st;
  if (M == 0) return CODA_OK;
  if (!dy || !W1 || !h || !r || !gamma || !dh_out) return CODA_ERR_INVALID_ARG;
  const void* ptrs[] = {dy, W1, h, r, gamma, dh_out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return CODA_ERR_MISALIGNED;
  const int64_t mt64 = cdiv(M, kBM), nt64 = cdiv(d, kBN);
  if (2 * static_cast<uint64_t>(nt64) * static_cast<uint64_t>(M) > kNoAllocPartials ||
      static_cast<uint64_t>(mt64) * static_cast<uint64_t>(nt64) > kNoAllocFlags)
    return CODA_ERR_UNSUPPORTED_SHAPE;  // larger than the static scratch
  int sms = 0;
  void* scratch = nullptr;
  st = device_setup(&sms, nullptr, &scratch);
  if (st != CODA_OK) return st;

  const int mt = static_cast<int>(mt64);
  const int nt = static_cast<int>(nt64);
  const int grid = std::min(sms, mt * nt);
  if (nt > grid) return CODA_ERR_UNSUPPORTED_SHAPE;

  CUtensorMap mA, mB;
  bool ok = tmap_2d(&mA, dy, N1, M, kBK, kBM);
  ok &= tmap_2d(&mB, W1, N1, d, kBK, kBN);
  if (!ok) return CODA_ERR_LAUNCH;

  EpiRmsNormBackward::Params p = {};
  p.h = reinterpret_cast<const __nv_bfloat16*>(h);
  p.gamma = reinterpret_cast<const __nv_bfloat16*>(gamma);
  p.r = r;
  p.dh_out = reinterpret_cast<__nv_bfloat16*>(dh_out);
  p.qpart = reinterpret_cast<float*>(scratch);
  p.flags = reinterpret_cast<uint64_t*>(static_cast<unsigned char*>(scratch) + kNoAllocFlagOffset);
  p.epoch = reinterpret_cast<uint64_t*>(static_cast<unsigned char*>(scratch) + kNoAllocEpochOffset);
  p.salt = next_salt();
  cudaError_t e = launch(kDgrad, grid, kThreads, kDgradSmem, stream, true, mA, mB,
                         static_cast<int>(M), static_cast<int>(d), static_cast<int>(N1), 1, p,
                         g_timeout_ns.load());
  if (e != cudaSuccess) {
    cudaGetLastError();
    return CODA_ERR_LAUNCH;
  }
  return CODA_OK;
}
