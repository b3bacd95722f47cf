// Row repacking kernels for the padded GEMM entry point (declared in
// repack.cuh).  Both are plain HBM-bound copies: every thread moves one
// 16-byte chunk (8 fp16) per step of a grid-stride loop, consecutive threads
// taking consecutive chunks of a row, so a warp reads and writes 512
// contiguous bytes.  The unaligned side is accessed with the widest loads or
// stores its address allows (16, 4 or 2 bytes); rows that do not end on a
// chunk boundary handle their last chunk element by element.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "repack.cuh"

namespace gb300 {
namespace {

constexpr int kThreads = 256;
constexpr int kBlocksPerSm = 8;  // 8 x 256 threads: a full SM

// A thread's position (row r, chunk j) in the flat chunk order i = r * cpr + j,
// advanced by the grid stride (step_r rows + step_j chunks) without dividing.
struct Walk {
  int64_t r, j;
  __device__ __forceinline__ void advance(int64_t step_r, int64_t step_j, int64_t cpr) {
    r += step_r;
    j += step_j;
    if (j >= cpr) {
      j -= cpr;
      ++r;
    }
  }
};

__device__ __forceinline__ uint32_t pair16(uint32_t lo, uint32_t hi) { return lo | (hi << 16); }

__global__ void __launch_bounds__(kThreads)
    repack_rows_kernel(uint4* __restrict__ dst, const uint16_t* __restrict__ src, int64_t rows,
                       int64_t cols, int64_t cpr, int64_t step_r, int64_t step_j) {
  const int64_t total = rows * cpr;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (i >= total) return;
  Walk w{i / cpr, i % cpr};
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (; i < total; i += stride, w.advance(step_r, step_j, cpr)) {
    const int64_t c0 = 8 * w.j;
    const uint16_t* s = src + w.r * cols + c0;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(s);
    uint4 v;
    if (c0 + 8 <= cols) {
      if ((addr & 15) == 0) {
        v = __ldg(reinterpret_cast<const uint4*>(s));
      } else if ((addr & 3) == 0) {
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(s);
        v = make_uint4(__ldg(s32), __ldg(s32 + 1), __ldg(s32 + 2), __ldg(s32 + 3));
      } else {
        // s[0] and s[7] alone; s[1..6] as three aligned words
        const uint32_t* s32 = reinterpret_cast<const uint32_t*>(s + 1);
        const uint32_t x0 = __ldg(s32), x1 = __ldg(s32 + 1), x2 = __ldg(s32 + 2);
        const uint32_t h0 = __ldg(s), h7 = __ldg(s + 7);
        v = make_uint4(h0 | (x0 << 16), (x0 >> 16) | (x1 << 16), (x1 >> 16) | (x2 << 16),
                       (x2 >> 16) | (h7 << 16));
      }
    } else {
      uint32_t h[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) h[q] = (c0 + q < cols) ? static_cast<uint32_t>(__ldg(s + q)) : 0u;
      v = make_uint4(pair16(h[0], h[1]), pair16(h[2], h[3]), pair16(h[4], h[5]),
                     pair16(h[6], h[7]));
    }
    dst[i] = v;
  }
}

__global__ void __launch_bounds__(kThreads)
    unpack_rows_kernel(uint16_t* __restrict__ dst, const uint4* __restrict__ src, int64_t rows,
                       int64_t cols, int64_t cpr, int64_t step_r, int64_t step_j) {
  const int64_t total = rows * cpr;
  int64_t i = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
  if (i >= total) return;
  Walk w{i / cpr, i % cpr};
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  for (; i < total; i += stride, w.advance(step_r, step_j, cpr)) {
    const int64_t c0 = 8 * w.j;
    const uint4 v = __ldg(src + i);
    uint16_t* d = dst + w.r * cols + c0;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(d);
    if (c0 + 8 <= cols) {
      if ((addr & 15) == 0) {
        *reinterpret_cast<uint4*>(d) = v;
      } else if ((addr & 3) == 0) {
        uint32_t* d32 = reinterpret_cast<uint32_t*>(d);
        d32[0] = v.x;
        d32[1] = v.y;
        d32[2] = v.z;
        d32[3] = v.w;
      } else {
        uint32_t* d32 = reinterpret_cast<uint32_t*>(d + 1);
        d[0] = static_cast<uint16_t>(v.x);
        d32[0] = (v.x >> 16) | (v.y << 16);
        d32[1] = (v.y >> 16) | (v.z << 16);
        d32[2] = (v.z >> 16) | (v.w << 16);
        d[7] = static_cast<uint16_t>(v.w >> 16);
      }
    } else {
      const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (c0 + q < cols) d[q] = static_cast<uint16_t>(wv[q >> 1] >> (16 * (q & 1)));
    }
  }
}

struct Grid {
  int blocks;
  int64_t cpr, step_r, step_j;
};

Grid grid_for(int64_t rows, int64_t cols, int sm_count) {
  Grid g;
  g.cpr = padded_cols(cols) / 8;
  const int64_t total = rows * g.cpr;
  g.blocks = static_cast<int>(
      std::min<int64_t>((total + kThreads - 1) / kThreads,
                        static_cast<int64_t>(std::max(sm_count, 1)) * kBlocksPerSm));
  const int64_t stride = static_cast<int64_t>(g.blocks) * kThreads;
  g.step_r = stride / g.cpr;
  g.step_j = stride % g.cpr;
  return g;
}

}  // namespace

cudaError_t repack_rows(void* dst, const void* src, int64_t rows, int64_t cols, int sm_count,
                        cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const Grid g = grid_for(rows, cols, sm_count);
  repack_rows_kernel<<<g.blocks, kThreads, 0, stream>>>(static_cast<uint4*>(dst),
                                                        static_cast<const uint16_t*>(src), rows,
                                                        cols, g.cpr, g.step_r, g.step_j);
  return cudaGetLastError();
}

cudaError_t unpack_rows(void* dst, const void* src, int64_t rows, int64_t cols, int sm_count,
                        cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  const Grid g = grid_for(rows, cols, sm_count);
  unpack_rows_kernel<<<g.blocks, kThreads, 0, stream>>>(static_cast<uint16_t*>(dst),
                                                        static_cast<const uint4*>(src), rows,
                                                        cols, g.cpr, g.step_r, g.step_j);
  return cudaGetLastError();
}

}  // namespace gb300
