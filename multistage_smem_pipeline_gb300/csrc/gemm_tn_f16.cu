// Host side of the C-ABI: argument checks, configuration choice, TMA
// descriptor encoding and the launch of the persistent kernel.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm_kernel.cuh"
#include "gemm_tn_f16.h"

namespace gb300 {
namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxDynSmem = 232448;  // 227 KiB opt-in limit per CTA on sm_100-class parts
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceState {
  bool init = false;
  int status = GEMM_OK;
  int sm_count = 0;
  int smem_attr = 0;  // dynamic smem size last granted to the kernel
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

int get_encoder() {
  if (g_encode) return GEMM_OK;
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return GEMM_ERR_CUDA;
  g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  return GEMM_OK;
}

// Current device, checked to be compute capability 10.3 (state cached).
int current_device(int* dev_out, DeviceState** st_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.init) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    st.init = true;
    st.sm_count = sms;
    st.status = (major == 10 && minor == 3) ? GEMM_OK : GEMM_ERR_UNSUPPORTED_DEVICE;
  }
  *dev_out = dev;
  *st_out = &st;
  return st.status;
}

int sm_count_or_default() {
  int dev = 0;
  DeviceState* st = nullptr;
  if (current_device(&dev, &st) == GEMM_OK) return st->sm_count;
  cudaGetLastError();
  return 148;
}

uint32_t pow2_at_least(uint32_t x) {
  uint32_t p = 32;
  while (p < x) p <<= 1;
  return p;
}

// tcgen05 instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B
// fp16 (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
uint32_t make_idesc(int m, int n) {
  return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}

int stages_that_fit(int bn) {
  const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(bn) * 128u;
  const uint32_t fixed = kEpiWarps * kEpiBufs * kEpiChunkBytes + 16 + 1024;
  int s = 2;
  while (s + 1 <= kMaxStages) {
    const uint32_t bars = 8u * (2 * (s + 1) + 5);
    if ((s + 1) * stage_bytes + fixed + bars > static_cast<uint32_t>(kMaxDynSmem)) break;
    ++s;
  }
  return s;
}

// Relative time of one k-block on one SM for a 128 x bn tile: the tensor
// pipe needs 2*bn cycles (128 x bn x 64 MACs at 8192 flop/clk), the operand
// reads from shared memory need (16 KiB + bn*128 B) / 128 B/clk.
double kblock_cost(int bn) { return std::max(2.0 * bn, 128.0 + bn); }

struct Plan {
  gemm_config_t cfg;
  GemmParams p;
};

int make_plan(int64_t M, int64_t N, int64_t K, const gemm_options_t* opt, int sms, Plan* out) {
  gemm_options_t o;
  std::memset(&o, 0, sizeof(o));
  if (opt) o = *opt;
  if (o.path < 0 || o.path > 2 || o.bn < 0 || o.bn > 256 || (o.bn % 32) != 0 || o.kstage < 0 ||
      o.kstage == 1 || o.kstage > kMaxStages || o.max_ctas < 0 || o.group_m < 0 || o.inject < 0 ||
      o.inject > 1)
    return GEMM_ERR_INVALID_VALUE;
  int path = o.path;
  if (path == GEMM_PATH_AUTO) path = (M <= kBM) ? GEMM_PATH_SKINNY : GEMM_PATH_SQUARE;
  if (path == GEMM_PATH_SKINNY && M > kBM) return GEMM_ERR_INVALID_VALUE;

  const int64_t num_m = (M + kBM - 1) / kBM;
  const int64_t num_k = (K + kBK - 1) / kBK;
  int bn = o.bn;
  if (bn == 0) {
    // Fewest waves x per-k-block cost; ties go to the wider tile (less L2 traffic).
    double best = 0;
    for (int cand = 256; cand >= 32; cand -= 32) {
      const int64_t tiles = num_m * ((N + cand - 1) / cand);
      const int64_t waves = (tiles + sms - 1) / sms;
      const double cost = static_cast<double>(waves) * kblock_cost(cand);
      if (bn == 0 || cost < best * (1.0 - 1e-9)) {
        best = cost;
        bn = cand;
      }
    }
  }
  const int64_t num_n = (N + bn - 1) / bn;
  const int64_t tiles = num_m * num_n;
  if (tiles > INT_MAX || num_k > INT_MAX) return GEMM_ERR_INVALID_VALUE;
  const int fit = stages_that_fit(bn);
  const int stages = o.kstage ? o.kstage : fit;
  if (stages > fit) return GEMM_ERR_INVALID_VALUE;
  int ctas = static_cast<int>(std::min<int64_t>(tiles, sms));
  if (o.max_ctas) ctas = std::min(ctas, o.max_ctas);
  const int group_m = o.group_m ? o.group_m : 16;

  const uint32_t stage_bytes = kABytes + static_cast<uint32_t>(bn) * 128u;
  const SmemLayout L = SmemLayout::make(stages, stage_bytes);

  Plan pl;
  std::memset(&pl, 0, sizeof(pl));
  pl.cfg.path = path;
  pl.cfg.bm = kBM;
  pl.cfg.bn = bn;
  pl.cfg.bk = kBK;
  pl.cfg.kstage = stages;
  pl.cfg.ctas = ctas;
  pl.cfg.group_m = group_m;
  pl.cfg.tiles = static_cast<int>(tiles);
  pl.cfg.smem_bytes = static_cast<int>(L.total + 1024);  // + alignment slack
  pl.cfg.tmem_cols = static_cast<int>(pow2_at_least(2u * bn));

  GemmParams& p = pl.p;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.bn = bn;
  p.stages = stages;
  p.num_m_blocks = static_cast<int32_t>(num_m);
  p.num_n_blocks = static_cast<int32_t>(num_n);
  p.num_k_blocks = static_cast<int32_t>(num_k);
  p.num_tiles = static_cast<int32_t>(tiles);
  p.group_m = group_m;
  p.idesc = make_idesc(kBM, bn);
  p.tmem_cols = pow2_at_least(2u * bn);
  p.stage_bytes = stage_bytes;
  p.l2_hints = (path == GEMM_PATH_SKINNY) ? 3u : 0u;
  p.timeout_ns = o.timeout_ns ? o.timeout_ns : kDefaultTimeoutNs;
  p.inject = o.inject;
  *out = pl;
  return GEMM_OK;
}

int encode_2d(CUtensorMap* map, const void* ptr, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer, CUtensorMapSwizzle swz) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};  // bytes between rows
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_INVALID_VALUE;
}

bool overlaps(const void* a, uint64_t abytes, const void* b, uint64_t bbytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bbytes && y < x + abytes;
}

int check_args(const void* D, const void* A, const void* B, int64_t M, int64_t N, int64_t K) {
  if (M < 0 || N < 0 || K < 0 || M > INT_MAX || N > INT_MAX || K > INT_MAX)
    return GEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!D || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_VALUE;
  if ((reinterpret_cast<uintptr_t>(D) & 15) || (reinterpret_cast<uintptr_t>(A) & 15) ||
      (reinterpret_cast<uintptr_t>(B) & 15) || (K % 8) != 0 || (N % 8) != 0)
    return GEMM_ERR_MISALIGNED;
  const uint64_t dbytes = static_cast<uint64_t>(M) * N * 2;
  if (K > 0 && (overlaps(D, dbytes, A, static_cast<uint64_t>(M) * K * 2) ||
                overlaps(D, dbytes, B, static_cast<uint64_t>(N) * K * 2)))
    return GEMM_ERR_INVALID_VALUE;
  return GEMM_OK;
}

int run(void* D, const void* A, const void* B, int64_t M, int64_t N, int64_t K,
        const gemm_options_t* opt, cudaStream_t stream) {
  int rc = check_args(D, A, B, M, N, K);
  if (rc != GEMM_OK) return rc;
  if (opt) {  // validate options even when there is nothing to compute
    Plan tmp;
    rc = make_plan(std::max<int64_t>(M, 1), std::max<int64_t>(N, 8), std::max<int64_t>(K, 8), opt,
                   148, &tmp);
    if (rc != GEMM_OK) return rc;
  }
  if (M == 0 || N == 0) return GEMM_OK;
  int dev = 0;
  DeviceState* st = nullptr;
  rc = current_device(&dev, &st);
  if (rc != GEMM_OK) return rc;
  if (K == 0) {
    if (cudaMemsetAsync(D, 0, static_cast<size_t>(M) * N * 2, stream) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
  }
  Plan pl;
  rc = make_plan(M, N, K, opt, st->sm_count, &pl);
  if (rc != GEMM_OK) return rc;
  if ((rc = get_encoder()) != GEMM_OK) return rc;

  CUtensorMap tmA, tmB, tmD;
  if (encode_2d(&tmA, A, K, M, kBK, kBM, CU_TENSOR_MAP_SWIZZLE_128B) != GEMM_OK ||
      encode_2d(&tmB, B, K, N, kBK, pl.cfg.bn, CU_TENSOR_MAP_SWIZZLE_128B) != GEMM_OK ||
      encode_2d(&tmD, D, N, M, kEpiCols, 32, CU_TENSOR_MAP_SWIZZLE_64B) != GEMM_OK)
    return GEMM_ERR_INVALID_VALUE;

  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (st->smem_attr < pl.cfg.smem_bytes) {
      if (cudaFuncSetAttribute(gemm_tn_f16_persistent, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               kMaxDynSmem) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_ERR_CUDA;
      }
      st->smem_attr = kMaxDynSmem;
    }
  }
  gemm_tn_f16_persistent<<<pl.cfg.ctas, kThreads, pl.cfg.smem_bytes, stream>>>(tmA, tmB, tmD,
                                                                               pl.p);
  if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
  return GEMM_OK;
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" int gemm_tn_f16(void* D, const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                           void* stream) {
  return run(D, A, B, M, N, K, nullptr, static_cast<cudaStream_t>(stream));
}

extern "C" int gemm_tn_f16_ex(void* D, const void* A, const void* B, int64_t M, int64_t N,
                              int64_t K, const gemm_options_t* opt, void* stream) {
  return run(D, A, B, M, N, K, opt, static_cast<cudaStream_t>(stream));
}

extern "C" int gemm_query_config(int64_t M, int64_t N, int64_t K, const gemm_options_t* opt,
                                 gemm_config_t* out) {
  if (!out || M <= 0 || N <= 0 || K <= 0 || M > INT_MAX || N > INT_MAX || K > INT_MAX)
    return GEMM_ERR_INVALID_VALUE;
  Plan pl;
  const int rc = make_plan(M, N, K, opt, sm_count_or_default(), &pl);
  if (rc == GEMM_OK) *out = pl.cfg;
  return rc;
}

extern "C" int gemm_get_device_error(void* stream, uint32_t* raw) {
  int dev = 0;
  DeviceState* st = nullptr;
  const int rc = current_device(&dev, &st);
  if (rc != GEMM_OK) return rc;
  unsigned int word = 0;
  const unsigned int zero = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&word, g_gemm_error, sizeof(word), 0, cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_gemm_error, &zero, sizeof(zero), 0, cudaMemcpyHostToDevice, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  if (raw) *raw = word;
  return static_cast<int>(word & 0xffu);
}

extern "C" int64_t gemm_minimum_stages(int64_t copy_cycles, int64_t compute_cycles) {
  if (copy_cycles <= 0 || compute_cycles <= 0) return -1;
  return copy_cycles / compute_cycles + (copy_cycles % compute_cycles != 0) + 1;
}

extern "C" const char* gemm_status_string(int status) {
  switch (status) {
    case GEMM_OK: return "GEMM_OK";
    case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE";
    case GEMM_ERR_MISALIGNED: return "GEMM_ERR_MISALIGNED";
    case GEMM_ERR_UNSUPPORTED_DEVICE: return "GEMM_ERR_UNSUPPORTED_DEVICE";
    case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH";
    case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
    case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
    default: return "GEMM_ERR_UNKNOWN";
  }
}
