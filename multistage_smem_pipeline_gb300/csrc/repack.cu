// Row repacking kernels for the padded GEMM entry point (declared in
// repack.cuh).  Both are plain HBM-bound copies.  Rows of at least kRowMin
// elements go one warp per row, touching the unaligned side only in whole
// aligned 16-byte blocks (see the row kernels below).  Shorter rows go one
// 16-byte chunk (8 fp16) per thread per step of a grid-stride loop over all
// rows' chunks, accessing the unaligned side with the widest loads or stores
// its address allows (16, 4 or 2 bytes); a row's last partial chunk goes
// element by element.
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

// ---------------------------------------------------------------- row kernels
//
// One warp per row, for rows of at least kRowMin elements.  The unaligned
// side is accessed only as whole 16-byte-aligned blocks: lane l of step i
// owns aligned block 32 i + l, takes the block before it from lane l - 1
// (lane 0 from lane 31 of the previous step) and assembles its 16 output
// bytes by a byte shift that is the same for the whole row.  A block that
// holds at least one byte of the row lies in the same page as that byte, so
// reading it whole cannot fault; only the row's two end blocks are written
// element by element.  Each lane loads kUnroll blocks before it shuffles, so
// a warp keeps kUnroll x 512 bytes in flight.
constexpr int kRowMin = 128;
constexpr int kUnroll = 4;

// Bytes [shift, shift + 16) of the 32 bytes lo:hi (shift even, 0..16).
__device__ __forceinline__ uint4 window16(const uint4& lo, const uint4& hi, int shift) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t o[4];
  const bool half = (shift & 2) != 0;
#define GB300_WINDOW_CASE(Q)                                                          \
  case Q:                                                                            \
    _Pragma("unroll") for (int k = 0; k < 4; ++k) o[k] =                              \
        half ? __funnelshift_r(w[(Q) + k], w[((Q) + k + 1) & 7], 16) : w[(Q) + k];    \
    break;
  switch (shift >> 2) {
    GB300_WINDOW_CASE(0)
    GB300_WINDOW_CASE(1)
    GB300_WINDOW_CASE(2)
    GB300_WINDOW_CASE(3)
    default:  // shift == 16
      o[0] = w[4], o[1] = w[5], o[2] = w[6], o[3] = w[7];
  }
#undef GB300_WINDOW_CASE
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint4 shfl_up_u4(const uint4& v, int delta) {
  return make_uint4(__shfl_up_sync(0xffffffffu, v.x, delta), __shfl_up_sync(0xffffffffu, v.y, delta),
                    __shfl_up_sync(0xffffffffu, v.z, delta), __shfl_up_sync(0xffffffffu, v.w, delta));
}

__device__ __forceinline__ uint4 shfl_u4(const uint4& v, int lane) {
  return make_uint4(__shfl_sync(0xffffffffu, v.x, lane), __shfl_sync(0xffffffffu, v.y, lane),
                    __shfl_sync(0xffffffffu, v.z, lane), __shfl_sync(0xffffffffu, v.w, lane));
}

// dst (aligned, row stride cpr chunks) <- src rows of `cols` halves at any
// 2-byte alignment; the pad of each row's last chunk is written as +0.
__global__ void __launch_bounds__(kThreads)
    repack_rows_warp_kernel(uint4* __restrict__ dst, const uint16_t* __restrict__ src,
                            int64_t rows, int64_t cols, int64_t cpr) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5; r < rows;
       r += warps) {
    const uintptr_t s0 = reinterpret_cast<uintptr_t>(src + r * cols);
    const uintptr_t a0 = s0 & ~static_cast<uintptr_t>(15);
    const uintptr_t s_end = s0 + 2 * static_cast<uintptr_t>(cols);  // one past the row
    const int shift = static_cast<int>(s0 - a0);                    // even, 0..14
    uint4* drow = dst + r * cpr;
    // aligned source block b: zero unless it holds a byte of the row
    auto block = [&](int64_t b) {
      const uintptr_t at = a0 + 16 * static_cast<uintptr_t>(b);
      return at < s_end ? __ldg(reinterpret_cast<const uint4*>(at)) : make_uint4(0, 0, 0, 0);
    };
    uint4 carry = make_uint4(0, 0, 0, 0);  // block 32 i of step i, from lane 31 of step i - 1
    for (int64_t j1 = 0; j1 < cpr; j1 += 32 * kUnroll) {
      uint4 nexts[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) nexts[u] = block(j1 + 32 * u + lane + 1);
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t j0 = j1 + 32 * u;
        const int64_t j = j0 + lane;
        const uint4 next = nexts[u];               // chunk j is bytes of blocks j and j + 1
        uint4 cur = shfl_up_u4(next, 1);
        if (lane == 0) cur = (j0 == 0) ? block(0) : carry;
        carry = shfl_u4(next, 31);
        if (j < cpr) {
          uint4 v = window16(cur, next, shift);
          const int64_t c0 = 8 * j;
          if (c0 + 8 > cols) {  // the row's last chunk: +0 past the row
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (c0 + q >= cols) w[q >> 1] &= (q & 1) ? 0x0000ffffu : 0xffff0000u;
            v = make_uint4(w[0], w[1], w[2], w[3]);
          }
          drow[j] = v;
        }
      }
    }
  }
}

// dst rows of `cols` halves at any 2-byte alignment <- the first cols
// columns of src (aligned, row stride cpr chunks).
__global__ void __launch_bounds__(kThreads)
    unpack_rows_warp_kernel(uint16_t* __restrict__ dst, const uint4* __restrict__ src,
                            int64_t rows, int64_t cols, int64_t cpr) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kThreads / 32);
  for (int64_t r = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5; r < rows;
       r += warps) {
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst + r * cols);
    const uintptr_t a0 = d0 & ~static_cast<uintptr_t>(15);
    const uintptr_t d_end = d0 + 2 * static_cast<uintptr_t>(cols);
    const int lead = static_cast<int>(d0 - a0);  // bytes of block 0 before the row, even
    const int64_t nblocks = static_cast<int64_t>((d_end - a0 + 15) / 16);
    const uint4* srow = src + r * cpr;
    uint4 carry = make_uint4(0, 0, 0, 0);
    for (int64_t i1 = 0; i1 < nblocks; i1 += 32 * kUnroll) {
      uint4 curs[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i = i1 + 32 * u + lane;
        curs[u] = i < cpr ? __ldg(srow + i) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int64_t i0 = i1 + 32 * u;
        const int64_t i = i0 + lane;
        // output block i holds the row's bytes [16 i - lead, 16 i - lead + 16):
        // the tail of chunk i - 1 and the head of chunk i
        const uint4 cur = curs[u];
        uint4 prev = shfl_up_u4(cur, 1);
        if (lane == 0) prev = carry;
        carry = shfl_u4(cur, 31);
        if (i < nblocks) {
          const uint4 v = window16(prev, cur, 16 - lead);
          const uintptr_t at = a0 + 16 * static_cast<uintptr_t>(i);
          if (at >= d0 && at + 16 <= d_end) {
            *reinterpret_cast<uint4*>(at) = v;
          } else {  // the row's end blocks: only the row's own bytes
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const uintptr_t e = at + 2 * q;
              if (e >= d0 && e < d_end)
                *reinterpret_cast<uint16_t*>(e) =
                    static_cast<uint16_t>(w[q >> 1] >> (16 * (q & 1)));
            }
          }
        }
      }
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

int warp_grid(int64_t rows, int sm_count) {
  const int64_t blocks = (rows + (kThreads / 32) - 1) / (kThreads / 32);
  return static_cast<int>(
      std::min<int64_t>(blocks, static_cast<int64_t>(std::max(sm_count, 1)) * kBlocksPerSm));
}

cudaError_t repack_rows(void* dst, const void* src, int64_t rows, int64_t cols, int sm_count,
                        cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (cols >= kRowMin) {
    repack_rows_warp_kernel<<<warp_grid(rows, sm_count), kThreads, 0, stream>>>(
        static_cast<uint4*>(dst), static_cast<const uint16_t*>(src), rows, cols,
        padded_cols(cols) / 8);
    return cudaGetLastError();
  }
  const Grid g = grid_for(rows, cols, sm_count);
  repack_rows_kernel<<<g.blocks, kThreads, 0, stream>>>(static_cast<uint4*>(dst),
                                                        static_cast<const uint16_t*>(src), rows,
                                                        cols, g.cpr, g.step_r, g.step_j);
  return cudaGetLastError();
}

cudaError_t unpack_rows(void* dst, const void* src, int64_t rows, int64_t cols, int sm_count,
                        cudaStream_t stream) {
  if (rows <= 0 || cols <= 0) return cudaSuccess;
  if (cols >= kRowMin) {
    unpack_rows_warp_kernel<<<warp_grid(rows, sm_count), kThreads, 0, stream>>>(
        static_cast<uint16_t*>(dst), static_cast<const uint4*>(src), rows, cols,
        padded_cols(cols) / 8);
    return cudaGetLastError();
  }
  const Grid g = grid_for(rows, cols, sm_count);
  unpack_rows_kernel<<<g.blocks, kThreads, 0, stream>>>(static_cast<uint16_t*>(dst),
                                                        static_cast<const uint4*>(src), rows,
                                                        cols, g.cpr, g.step_r, g.step_j);
  return cudaGetLastError();
}

}  // namespace gb300
