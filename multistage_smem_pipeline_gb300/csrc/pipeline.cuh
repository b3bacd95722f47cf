// Constants, parameter block, shared-memory carve-up and small device helpers
// shared by the GEMM kernel and the latency probes.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace gb300 {

constexpr int kBM = 128;             // UMMA M: one TMEM lane per output row
constexpr int kBK = 64;              // 64 fp16 = 128 B = one 128-byte swizzle row
constexpr int kUmmaK = 16;           // K per tcgen05.mma (kind::f16)
// Epilogue warps per CTA: 4 (one per TMEM lane quadrant) or 8 (two per
// quadrant, taking alternate 32-column chunks).  The block is the producer
// warp, the MMA warp and the epilogue warps.
__host__ __device__ constexpr int threads_for(int epi_warps) { return 64 + 32 * epi_warps; }
constexpr int kEpiBufs = 2;          // store staging buffers per epilogue warp
constexpr int kEpiCols = 32;         // columns per epilogue chunk (one tcgen05.ld x32)
constexpr uint32_t kEpiChunkBytes = 32 * kEpiCols * 2;  // 32 rows x 32 fp16
constexpr uint32_t kABytes = kBM * kBK * 2;             // 16 KiB
constexpr int kMaxStages = 16;
constexpr uint32_t kErrTimeout = 5;    // == GEMM_ERR_TIMEOUT
constexpr uint32_t kErrInvariant = 7;  // == GEMM_ERR_INVARIANT

enum WaitSite : uint32_t { kSiteEmpty = 1, kSiteFull = 2, kSiteTmemEmpty = 3, kSiteTmemFull = 4 };
// Site of a failed invariant check: the ring slot the MMA thread consumed did
// not carry the sequence number of the fill it expected.
constexpr uint32_t kSiteRingSeq = 5;

// The misc area: the TMEM base address (+0), the CTA's abort flag (+4), the
// index of the error word its errors go to (+8), then from +16 one sequence
// word per ring slot for the invariant check, kMaxStages of them.
constexpr uint32_t kMiscBytes = 16 + 4 * 16;
constexpr uint32_t kMiscSlotSeq = 16;

// Error words per device: the host gives each stream its own (see
// error_slot), the kernels record their first error there.
constexpr int kErrorSlots = 64;

struct GemmParams {
  int32_t M, N, K;
  int32_t bn;            // tile width along N (multiple of 32, 32..256)
  int32_t stages;        // ring depth (2..kMaxStages)
  int32_t num_m_blocks, num_n_blocks, num_k_blocks, num_tiles;
  int32_t group_m;       // m-blocks per rasterisation group
  uint32_t idesc;        // tcgen05 instruction descriptor
  uint32_t tmem_cols;    // allocated TMEM columns (power of two >= 2*bn)
  uint32_t stage_bytes;  // katoms * (kABytes + b_atom_bytes)
  uint32_t b_atom_bytes; // B rows per CTA x 128 B: one 64-wide K atom of B
  int32_t katoms;        // 64-wide K atoms per stage (1 or 2); a k-block is 64 * katoms wide
  uint32_t l2_hints;     // bit 0: stream B with evict-first; bit 1: keep A with evict-last
  uint64_t timeout_ns;
  int32_t inject;
  int32_t k_rotate;      // 1: each tile starts its k loop at a tile-dependent k-block
  int32_t epi_warps;     // epilogue warps (4 or 8); must match the launched kernel
  int32_t b_kn;          // 1: B is K x N row-major (N contiguous): an MN-major operand
  int32_t scaled;        // 1: D = alpha * acc + beta * C instead of D = acc
  float alpha, beta;
  const uint16_t* C;     // M x N fp16, row stride ldc; read only when scaled and beta != 0
  int32_t acc_f16;       // 1: fp16 accumulator (low 16 bits of each TMEM column)
  int64_t ldc;           // elements between rows of C (a multiple of 8)
  int32_t b_resident;    // 1: all of B (one n-block, every k slice) is loaded once per CTA
                         //    into its own region; the ring then carries A only
  uint32_t bres_bytes;   // size of that region: num_k_blocks * katoms * b_atom_bytes (else 0)
  uint16_t* D;           // direct-store kernels only: D (rows not 16-byte aligned) ...
  int64_t ldd;           // ... and its row stride in elements
  int32_t check;         // 1: the MMA thread checks each ring slot's fill sequence number
  int32_t err_slot;      // index of the device error word this call's errors go to
};

// MN-major B: one 64-element N chunk per TMA box; chunks 8 KiB apart.
constexpr uint32_t kMnChunkBytes = 64 * 64 * 2;

// First k-block of tile t.  With rotation the tiles in flight start at
// evenly spread k offsets, so when every tile reads the same rows of A (one
// m-block) they do not all hit the same L2 lines at the same moment.  Only
// the order of the fp32 accumulation changes.
__device__ __forceinline__ int first_k_block(int t, const GemmParams& p) {
  if (!p.k_rotate) return 0;
  return static_cast<int>((static_cast<int64_t>(t) * p.num_k_blocks) / p.num_tiles) %
         p.num_k_blocks;
}

// Shared-memory carve-up, offsets from the 1024-aligned base: the ring, the
// resident B region (if any; 1024-aligned since stages are whole 16 KiB A
// slices), the epilogue staging buffers, then 2 * stages + 5 + bres_bars
// mbarriers (full, empty, 2 tmem-full, 2 tmem-empty, drain, then one per
// k-block of the resident B -- one slot at least).
struct SmemLayout {
  uint32_t ring, bres, epi, bars, misc, total;
  __host__ __device__ static SmemLayout make(int stages, uint32_t stage_bytes, int epi_warps,
                                             uint32_t bres_bytes = 0, int bres_bars = 1) {
    SmemLayout L;
    L.ring = 0;
    L.bres = stages * stage_bytes;
    L.epi = L.bres + bres_bytes;
    L.bars = L.epi + epi_warps * kEpiBufs * kEpiChunkBytes;
    L.misc = L.bars + 8 * (2 * stages + 5 + (bres_bars > 1 ? bres_bars : 1));
    L.total = L.misc + kMiscBytes;
    return L;
  }
};

// Chunks of 32 columns handled by one epilogue warp: `half` in [0, stride)
// picks every stride-th chunk; returns the last one (or -1 if none).
__device__ __forceinline__ int last_epi_chunk(int nchunks, int half, int stride) {
  const int top = nchunks - 1 - half;
  return top < 0 ? -1 : nchunks - 1 - (top % stride);
}

// Bounded wait that ignores the abort flag: used while draining.
__device__ __forceinline__ bool wait_timed(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0 && global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// Grouped rasterisation: consecutive tile ids walk down `group_m` m-blocks
// before moving to the next n-block, so the tiles in flight at once share
// their A rows and B rows in L2.
__device__ __forceinline__ void tile_coords(int t, const GemmParams& p, int& mb, int& nb) {
  const int group_tiles = p.group_m * p.num_n_blocks;
  const int g = t / group_tiles;
  const int first_m = g * p.group_m;
  const int gm = min(p.num_m_blocks - first_m, p.group_m);
  const int in = t - g * group_tiles;
  mb = first_m + in % gm;
  nb = in / gm;
}

// The pipeline invariant check (the kernels' kCheck instantiations, chosen
// for p.check): the producer stamps ring slot s
// with the sequence number of the fill it issues there (written before its
// arrive on the slot's full barrier, which orders it), and the MMA thread,
// once the slot is full, compares the stamp with the count of slots it has
// consumed.  A wrong stage index or phase that still lets the pipeline run
// shows up as a mismatch, recorded as GEMM_ERR_INVARIANT | site << 8 in the
// device error word; the kernel goes on (no trap).  inject == 2 plants one
// wrong stamp, to test the check.
template <bool kCheck>
__device__ __forceinline__ void stamp_slot(volatile uint32_t* seq, int stage, uint32_t issued,
                                           const GemmParams& p) {
  if (kCheck) seq[stage] = issued + ((p.inject == 2 && issued == 0) ? 1u : 0u);
}

__device__ __forceinline__ uint32_t pack_half2(uint32_t lo_bits, uint32_t hi_bits) {
  const __half2 h = __floats2half2_rn(__uint_as_float(lo_bits), __uint_as_float(hi_bits));
  return *reinterpret_cast<const uint32_t*>(&h);
}

// An fp16 accumulator occupies the low 16 bits of each 32-bit TMEM column;
// widen it to fp32 bits (exactly) so the rest of the epilogue is shared.
__device__ __forceinline__ void widen_f16_accumulator(uint32_t (&r)[32]) {
#pragma unroll
  for (int i = 0; i < 32; ++i)
    r[i] = __float_as_uint(__half2float(__ushort_as_half(static_cast<unsigned short>(r[i]))));
}

__device__ __forceinline__ uint16_t ld_shared_u16(uint32_t addr) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
  return v;
}

// The direct-store form of the epilogue's last step, for a D whose rows are
// not 16-byte aligned (no TMA store can describe them): the warp writes the
// 32 x 32 chunk it staged at `buf` (64-byte rows, piece j of row r at
// position j ^ ((r >> 1) & 3)) row by row, lane l taking column l, so each
// store instruction writes one row's 64 contiguous bytes.  Rows at or past M
// and columns at or past N are not written.
__device__ __forceinline__ void store_chunk_direct(uint32_t buf, uint16_t* D, int64_t ldd, int M,
                                                   int N, int m0, int n0, int lane) {
  const int col = n0 + lane;
  const uint32_t piece = static_cast<uint32_t>(lane) >> 3;
  const uint32_t within = (static_cast<uint32_t>(lane) & 7u) * 2u;
#pragma unroll 4
  for (int r = 0; r < 32; ++r) {
    const uint32_t sw = (static_cast<uint32_t>(r) >> 1) & 3u;
    const uint16_t v = ld_shared_u16(buf + static_cast<uint32_t>(r) * 64u + ((piece ^ sw) << 4) + within);
    const int row = m0 + r;
    if (row < M && col < N) D[static_cast<int64_t>(row) * ldd + col] = v;
  }
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

// The C term of the scaled epilogue for the warp's 32 x 32 chunk (rows
// [m0, m0 + 32), columns [col, col + 32)), copied into the warp's staging
// buffer `buf` (free to overwrite) with cp.async, in the layout of the
// epilogue's stores: 16-byte piece j of row r at j ^ ((r >> 1) & 3).  Copy i
// of a lane is row 8 i + lane / 4, piece lane % 4, so one warp-wide copy
// reads 64 contiguous bytes of each of 8 rows -- 8 whole lines of C, where
// one row per lane would touch 32 lines for 16 bytes each -- and no register
// holds C on the way.  Rows at or past M and pieces at or past N are
// zero-filled without reading C (nothing is stored there); a piece that
// straddles N reads up to the next multiple of 8, which the row stride ldc
// covers.  Returns once the chunk is in `buf` and visible to the warp.
// The copies alone, not committed: the caller commits and waits (the pair
// kernel's epilogue keeps the next chunk's copies in flight this way).
__device__ __forceinline__ void copy_c_chunk(const GemmParams& p, int m0, int col, int lane,
                                             uint32_t buf) {
  const uint32_t piece = static_cast<uint32_t>(lane) & 3u;
  const int c8 = col + 8 * static_cast<int>(piece);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t r = 8u * i + (static_cast<uint32_t>(lane) >> 2);
    const int row = m0 + static_cast<int>(r);
    const bool in = row < p.M && c8 < p.N;
    const uint16_t* src = in ? p.C + static_cast<size_t>(row) * p.ldc + c8 : p.C;
    cp_async_16(buf + r * 64u + ((piece ^ ((r >> 1) & 3u)) << 4), src, in ? 16u : 0u);
  }
}

__device__ __forceinline__ void stage_c_chunk(const GemmParams& p, int m0, int col, int lane,
                                              uint32_t buf) {
  copy_c_chunk(p, m0, col, lane, buf);
  cp_async_wait_all();
  __syncwarp();
}

// r (fp32 bits of row `lane` of the chunk) <- alpha * r, then + beta * C when
// stage_c_chunk has put the chunk's C in `buf`: each lane reads back its own
// row, the only row it later writes, so `buf` can then take the row's D
// values without another barrier.
__device__ __forceinline__ void apply_alpha_beta(uint32_t (&r)[32], const GemmParams& p,
                                                 bool with_c, uint32_t buf, int lane) {
#pragma unroll
  for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(p.alpha * __uint_as_float(r[i]));
  if (!with_c) return;
  const uint32_t sw = (static_cast<uint32_t>(lane) >> 1) & 3u;
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint4 c = ld_shared_v4(buf + static_cast<uint32_t>(lane) * 64u + ((g ^ sw) << 4));
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[q]);
      const float2 f = __half22float2(h);
      r[8 * g + 2 * q] = __float_as_uint(fmaf(p.beta, f.x, __uint_as_float(r[8 * g + 2 * q])));
      r[8 * g + 2 * q + 1] =
          __float_as_uint(fmaf(p.beta, f.y, __uint_as_float(r[8 * g + 2 * q + 1])));
    }
  }
}

}  // namespace gb300
