// Latency probes for the stage-count rule of "第 6 课：Shared Memory 布局与异步流水"
// (section 4): S_min = ceil(T_copy / T_compute) + 1.  T_copy is the time from
// issuing one stage's TMA loads to its full barrier completing; T_compute is
// the time the tensor pipe spends on one k-block of MMAs.  Both are measured
// here in SM clock cycles with the same tile shapes the GEMM kernel uses.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "pipeline.cuh"
#include "gemm_tn_f16.h"

namespace gb300 {
namespace {

__device__ unsigned long long g_probe_cycles;
__device__ unsigned long long g_probe_samples;
__device__ unsigned int g_probe_fail;

constexpr uint64_t kProbeTimeoutNs = 200000000ull;  // 0.2 s per wait

// One thread per CTA issues a stage's loads (A box 64 x 128, B box 64 x bn)
// from rows of a [rows x 64] fp16 scratch tensor, waits for the bytes, and
// accumulates the cycles.  Only one stage is in flight per CTA, so this is a
// latency, not a bandwidth, measurement.
__global__ void __launch_bounds__(32, 1)
    probe_copy(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               int bn, int64_t rows, int reps) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(bn) * 128u;
  const uint32_t bar = base + stage_bytes;
  if (threadIdx.x != 0) return;
  mbar_init(bar, 1);
  fence_barrier_init();
  const int64_t span = 128 + bn;
  const int64_t slots = rows / span;
  unsigned long long total = 0, n = 0;
  for (int r = 0; r < reps; ++r) {
    // walk the footprint so consecutive loads touch fresh lines
    const int64_t slot = (static_cast<int64_t>(r) * gridDim.x + blockIdx.x) * 7919 % slots;
    const int32_t y = static_cast<int32_t>(slot * span);
    const uint64_t t0 = clock64();
    mbar_arrive_expect_tx(bar, stage_bytes);
    tma_load_2d(base, &tmA, bar, 0, y);
    tma_load_2d(base + kABytes, &tmB, bar, 0, y + 128);
    if (!wait_timed(bar, r & 1, kProbeTimeoutNs)) {
      atomicOr(&g_probe_fail, 1u);
      // the bytes may still be landing: give them one more bounded wait
      wait_timed(bar, r & 1, kProbeTimeoutNs);
      break;
    }
    const uint64_t t1 = clock64();
    if (r > 0) {  // first load also pays descriptor fetch
      total += t1 - t0;
      ++n;
    }
  }
  atomicAdd(&g_probe_cycles, total);
  atomicAdd(&g_probe_samples, n);
}

// One thread issues `reps` k-blocks (4 x tcgen05.mma 128 x bn x 16) back to
// back on a zeroed stage, then waits for the last to complete.
__global__ void __launch_bounds__(128, 1) probe_mma(int bn, uint32_t tmem_cols, int reps) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(bn) * 128u;
  const uint32_t bar = base + stage_bytes;
  uint32_t* slot = reinterpret_cast<uint32_t*>(smem_raw + (base - raw) + stage_bytes + 8);
  for (uint32_t off = threadIdx.x * 16u; off < stage_bytes; off += 128u * 16u)
    st_shared_v4(base + off, 0u, 0u, 0u, 0u);
  fence_proxy_async_smem();
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (warp == 0) {
    tmem_alloc(smem_u32(slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *slot;
  if (threadIdx.x == 0) {
    const uint32_t idesc = (1u << 4) | (static_cast<uint32_t>(bn >> 3) << 17) |
                           (static_cast<uint32_t>(kBM >> 4) << 24);
    const uint64_t a_desc = sw128_kmajor_desc(base);
    const uint64_t b_desc = sw128_kmajor_desc(base + kABytes);
    const uint64_t t0 = clock64();
    for (int r = 0; r < reps; ++r) {
#pragma unroll
      for (int k = 0; k < kBK / kUmmaK; ++k)
        umma_f16(tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, (r | k) != 0);
    }
    umma_commit(bar);
    const bool ok = wait_timed(bar, 0, kProbeTimeoutNs);
    const uint64_t t1 = clock64();
    if (!ok) atomicOr(&g_probe_fail, 1u);
    atomicAdd(&g_probe_cycles, static_cast<unsigned long long>(t1 - t0));
    atomicAdd(&g_probe_samples, static_cast<unsigned long long>(reps));
  }
  __syncwarp();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, tmem_cols);
  }
}

int reset_counters(cudaStream_t s) {
  const unsigned long long z = 0;
  const unsigned int zi = 0;
  if (cudaMemcpyToSymbolAsync(g_probe_cycles, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_probe_samples, &z, sizeof(z), 0, cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_probe_fail, &zi, sizeof(zi), 0, cudaMemcpyHostToDevice, s) !=
          cudaSuccess)
    return GEMM_ERR_CUDA;
  return GEMM_OK;
}

int read_counters(cudaStream_t s, double* per_sample) {
  unsigned long long c = 0, n = 0;
  unsigned int fail = 0;
  if (cudaMemcpyFromSymbolAsync(&c, g_probe_cycles, sizeof(c), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&n, g_probe_samples, sizeof(n), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&fail, g_probe_fail, sizeof(fail), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (fail) return GEMM_ERR_TIMEOUT;
  *per_sample = n ? static_cast<double>(c) / static_cast<double>(n) : 0.0;
  return GEMM_OK;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" int gemm_probe_latencies(int bn, int ctas, const void* scratch, int64_t footprint_bytes,
                                    int reps, double* copy_cycles, double* compute_cycles,
                                    void* stream) {
  if (bn < 32 || bn > 256 || (bn % 32) != 0 || ctas < 0 || reps < 2 || reps > (1 << 20) ||
      !scratch || !copy_cycles || !compute_cycles ||
      (reinterpret_cast<uintptr_t>(scratch) & 15) ||
      footprint_bytes < static_cast<int64_t>(128 + bn) * 128 * 4 || footprint_bytes > (1ll << 40))
    return GEMM_ERR_INVALID_VALUE;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;
  if (ctas == 0 || ctas > sms) ctas = sms;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || !fn)
    return GEMM_ERR_CUDA;
  const EncodeTiledFn encode = reinterpret_cast<EncodeTiledFn>(fn);
  const int64_t rows = footprint_bytes / 128;
  CUtensorMap tmA, tmB;
  const cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t estr[2] = {1, 1};
  const cuuint32_t boxA[2] = {64, 128};
  const cuuint32_t boxB[2] = {64, static_cast<cuuint32_t>(bn)};
  if (encode(&tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(scratch), dims, strides,
             boxA, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      encode(&tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(scratch), dims, strides,
             boxB, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return GEMM_ERR_INVALID_VALUE;

  const int smem = static_cast<int>(kABytes + bn * 128 + 64 + 1024);
  if (cudaFuncSetAttribute(probe_copy, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess ||
      cudaFuncSetAttribute(probe_mma, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
          cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  int rc = reset_counters(s);
  if (rc != GEMM_OK) return rc;
  probe_copy<<<ctas, 32, smem, s>>>(tmA, tmB, bn, rows, reps);
  if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
  if ((rc = read_counters(s, copy_cycles)) != GEMM_OK) return rc;

  if ((rc = reset_counters(s)) != GEMM_OK) return rc;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(bn)) cols <<= 1;
  probe_mma<<<1, 128, smem, s>>>(bn, cols, reps);
  if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
  return read_counters(s, compute_cycles);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of gemm_probe_latencies.
//
// Some callers cannot call cudaMalloc: a serving process whose memory pool
// has already reserved nearly all of HBM (a fresh allocation would fail or
// make the pool give memory back), or a latency-sensitive loop that must not
// allocate because cudaMalloc/cudaFree can synchronise the device.  For them
// the copy probe's load footprint lives in a fixed array in device memory
// that the library owns.  Every GPU that loads this library holds the array
// (kStaticProbeScratchBytes) until the process exits.
//
// In host code the array's name is only a host-side stand-in for the device
// symbol, never a device address.  The device address is fetched with
// cudaGetSymbolAddress, with the device current, once per device and CUDA
// context: the cache is keyed on the context's unique id, so a context that
// was torn down and re-created (cudaDeviceReset) gets a fresh lookup instead
// of a stale address.  That set-up runs inside the entry point's first call
// on a device (and its first call after such a reset).  Under lazy module
// loading, the CUDA default, the lookup may also load this file's device
// code, and with it allocate the array itself, so make that first call early
// -- while the device still has 16 MiB free, and before any stream capture
// on the device.  Later calls allocate nothing.
//
// All calls share the array and the probes' result counters.  The array's
// contents are never relied on (the probe only times loads of it), and the
// counters are cleared at the start of every call; two calls that overlap
// on the GPU (e.g. on different streams) race on the counters and report
// wrong numbers.
// ---------------------------------------------------------------------------
namespace gb300 {
namespace {

constexpr int64_t kStaticProbeScratchBytes = 16ll << 20;  // 16 MiB per device
static __device__ __align__(256) uint8_t g_probe_static_scratch[kStaticProbeScratchBytes];

std::mutex g_static_mu;
// Device address of the array per device, with the id of the CUDA context it
// was looked up in (ptr == nullptr: not set up).
struct StaticScratch {
  unsigned long long ctx_id;
  void* ptr;
};
StaticScratch g_static_scratch[64];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// Unique id of the CUDA context current on this thread (driver entry points
// fetched through the runtime, so nothing links libcuda).  Fails when no
// context is current yet.  Called with g_static_mu held.
bool current_context_id(unsigned long long* id) {
  if (!g_ctx_get_current || !g_ctx_get_id) {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &qa) !=
            cudaSuccess ||
        qa != cudaDriverEntryPointSuccess || !a ||
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
            cudaSuccess ||
        qb != cudaDriverEntryPointSuccess || !b) {
      cudaGetLastError();
      return false;
    }
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(a);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(b);
  }
  CUcontext ctx = nullptr;
  return g_ctx_get_current(&ctx) == CUDA_SUCCESS && ctx != nullptr &&
         g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}

// The array's device address on the current device, looked up once per
// device and context.
int static_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (dev < 0 || dev >= 64) return GEMM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_static_mu);
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  StaticScratch& e = g_static_scratch[dev];
  if (have_id && e.ptr && e.ctx_id == id) {
    *out = e.ptr;
    return GEMM_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_probe_static_scratch) != cudaSuccess || !p) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  // the lookup makes the runtime's context current if none was
  if (have_id || current_context_id(&id)) {
    e.ctx_id = id;
    e.ptr = p;
  }
  *out = p;
  return GEMM_OK;
}

}  // namespace
}  // namespace gb300

extern "C" int gemm_probe_latencies_static(int bn, int ctas, int64_t footprint_bytes, int reps,
                                           double* copy_cycles, double* compute_cycles,
                                           void* stream) {
  using namespace gb300;
  if (footprint_bytes > kStaticProbeScratchBytes) return GEMM_ERR_INVALID_VALUE;
  void* ptr = nullptr;
  const int rc = static_scratch_address(&ptr);
  if (rc != GEMM_OK) return rc;
  // Same probes, same checks (bn, ctas, reps, minimum footprint, device), on
  // the library-owned array instead of a caller-allocated region.
  return gemm_probe_latencies(bn, ctas, ptr, footprint_bytes, reps, copy_cycles, compute_cycles,
                              stream);
}
