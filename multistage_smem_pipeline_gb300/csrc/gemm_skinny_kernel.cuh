// Small-M ("skinny") fp16 TN GEMM for sm_103a: M <= 128, one 128 x BN tile
// of D per CTA.
//
// D = A * B^T with one 128-row block of A against a long B (the skinny case:
// M = 128, N = 14336, K = 4096 reads 117 MB of B and 1 MiB of A).  Such a
// shape is bound by HBM, not by the tensor pipe ("第 6 课：Shared Memory 布局与
// 异步流水", section 1: the memory wall), and the page's stage rule (section
// 4) applies to the whole round trip of a stage: S_min = ceil(T_round /
// T_stage) + 1, where T_round is the load latency under load plus the time
// the MMA thread spends on the stage.  Traced on GB300 at the skinny shape:
// a stage of A and B (2 x 64-wide K slices, 56 KiB at BN = 96) takes about
// 2400 cycles to land once every SM is streaming -- A from L2 as slowly as B
// from HBM -- and its eight 128 x 96 x 16 MMAs take about 760 cycles to
// issue, so three stages in flight give one stage per ~1050 cycles and four
// would give one per ~790.  A CTA that also kept its epilogue's staging
// buffers (16 KiB) has room for three.
//
// This kernel is built for that case: every CTA computes exactly one tile
// (the grid is the number of n-tiles, at most one per SM), so once the
// tile's last MMA has completed nothing reads or fills the ring any more, and
// the epilogue stages its stores in the ring's first stage.  All the shared
// memory goes to the ring: four 56 KiB stages at BN = 96.  With one tile
// there is also no tile loop, no second accumulator and no TMEM-empty
// handshake: the pipeline is the page's prologue / mainloop / epilogue once.
//
// Roles: warp 0 (one thread) loads A and B with TMA into the ring (A with
// evict-last: every CTA reads the same rows; B with evict-first: read once);
// warp 1 (one thread) issues tcgen05.mma into one TMEM accumulator and
// commits each stage back to its producer; warps 2..5 read the accumulator's
// four lane quadrants, round to fp16 and store D (TMA, or plain stores for a
// D whose rows are not 16-byte aligned).  The read-after-write guard of
// "cute(9) multistage_gemm" (its cp_async_wait before the MMAs of a k-tile)
// is the stage's full barrier, the write-after-read guard its empty barrier.
// Each tile starts its k loop at a different k-block (CTAs then read
// different A slices at a time); the MMAs are those of the single-CTA kernel
// in the same order, so the results are bit-identical to it.  Every wait is
// bounded, as in the other kernels.
#pragma once
#include "gemm_kernel.cuh"

namespace gb300 {

constexpr int kSkinnyEpiWarps = 4;
constexpr int kSkinnyThreads = 64 + 32 * kSkinnyEpiWarps;  // producer, MMA, epilogue

// Shared-memory carve-up of the skinny kernel, offsets from the 1024-aligned
// base: the ring (whose first stage the epilogue reuses), then the mbarriers
// full[S], empty[S], tmem-full, drain.
struct SkinnyLayout {
  uint32_t ring, bars, misc, total;
  __host__ __device__ static SkinnyLayout make(int stages, uint32_t stage_bytes) {
    SkinnyLayout L;
    L.ring = 0;
    L.bars = stages * stage_bytes;
    L.misc = L.bars + 8 * (2 * stages + 2);
    L.total = L.misc + kMiscBytes;
    return L;
  }
};
// the epilogue's staging buffers fit in one ring stage
static_assert(kSkinnyEpiWarps * kEpiBufs * kEpiChunkBytes <= kABytes, "staging exceeds a stage");

// kCheck: the pipeline invariant check (as in gemm_tn_f16_persistent).
template <bool kDirectD, bool kCheck = false>
__global__ void __launch_bounds__(kSkinnyThreads, 1)
    gemm_tn_f16_skinny(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw);
  const int S = p.stages;
  const SkinnyLayout L = SkinnyLayout::make(S, p.stage_bytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x;  // this CTA's tile: n-block t of the one m-block
  const uint32_t bars = base + L.bars;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  const uint32_t tfull_bar = bars + 8u * (2 * S);
  const uint32_t drain_bar = bars + 8u * (2 * S + 1);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  volatile uint32_t* const slot_seq = reinterpret_cast<volatile uint32_t*>(smem + L.misc + kMiscSlotSeq);

  if (threadIdx.x == 0) {
    grid_launch_dependents();  // see gemm_tn_f16_persistent
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);   // producer's arrive.expect_tx; TMA bytes complete it
      mbar_init(empty_bar(s), 1);  // one tcgen05.commit per consumed stage
    }
    mbar_init(tfull_bar, 1);       // tcgen05.commit after the tile's last k-block
    mbar_init(drain_bar, 1);
    init_abort_state(abort_flag, p);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (!kDirectD) tma_prefetch_desc(&tmD);
    // The first ring of this CTA's operand boxes, fetched into L2 while the
    // previous grid finishes (see tma_prefetch_l2_2d).
    const int kf = first_k_block(t, p);
    for (int i = 0; i < p.num_k_blocks && i < S; ++i) {
      const int kb = (kf + i < p.num_k_blocks) ? kf + i : kf + i - p.num_k_blocks;
      for (int at = 0; at < p.katoms; ++at) {
        const int x = (kb * p.katoms + at) * kBK;
        tma_prefetch_l2_2d(&tmA, x, 0);
        if (p.b_kn) {
          for (int ch = 0; ch < p.bn / 64; ++ch) tma_prefetch_l2_2d(&tmB, t * p.bn + 64 * ch, x);
        } else {
          tma_prefetch_l2_2d(&tmB, x, t * p.bn);
        }
      }
    }
  }
  __syncwarp();
  __syncthreads();  // barriers initialised: the producer may start at once
  uint32_t tmem_base = 0;
  if (warp != 0) {
    if (warp == 1) {
      tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
      tmem_relinquish();
    }
    tc_fence_before_sync();
    named_barrier_sync(1, kSkinnyThreads - 32);
    tc_fence_after_sync();
    tmem_base = *tmem_slot;
  }
  uint64_t pol_a = 0, pol_b = 0;  // the producer's L2 policies (no memory access)
  if (warp == 0 && lane == 0) {
    pol_b = l2_policy_evict_first();
    pol_a = l2_policy_evict_last();
  }
  grid_dependency_wait();  // first global-memory access follows

  const int k0 = first_k_block(t, p);
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      for (int i = 0; i < p.num_k_blocks && !*abort_flag; ++i) {
        const int kb = (k0 + i < p.num_k_blocks) ? k0 + i : k0 + i - p.num_k_blocks;
        if (!wait_or_abort(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, kSiteEmpty))
          break;
        const uint32_t a_dst = base + L.ring + stage * p.stage_bytes;
        const uint32_t b_dst = a_dst + p.katoms * kABytes;
        stamp_slot<kCheck>(slot_seq, stage, issued, p);
        mbar_arrive_expect_tx(full_bar(stage), p.stage_bytes);
        if (!(p.inject == 1 && issued == 0)) {
          for (int at = 0; at < p.katoms; ++at) {
            const int x = (kb * p.katoms + at) * kBK;  // past K: the box reads zeros
            tma_load_2d_hint(a_dst + at * kABytes, &tmA, full_bar(stage), x, 0, pol_a);
            const uint32_t bd = b_dst + at * p.b_atom_bytes;
            if (p.b_kn) {  // B is K x N: one 64-column box per chunk of the tile
              for (int ch = 0; ch < p.bn / 64; ++ch)
                tma_load_2d(bd + ch * kMnChunkBytes, &tmB, full_bar(stage), t * p.bn + 64 * ch, x);
            } else {
              tma_load_2d_hint(bd, &tmB, full_bar(stage), x, t * p.bn, pol_b);
            }
          }
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // Drain: the loads of the last min(issued, S) stages must have landed
      // before the CTA (and its shared memory) goes away.
      const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0u;
      for (uint32_t i = first; i < issued; ++i)
        wait_timed(full_bar(i % S), (i / S) & 1u, p.timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t b_kstep = p.b_kn ? 128u : 2u;  // descriptor address units per K = 16
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; i < p.num_k_blocks; ++i) {
        if (!wait_or_abort(full_bar(stage), phase, p.timeout_ns, abort_flag, kSiteFull)) {
          ok = false;
          break;
        }
        check_slot<kCheck>(slot_seq, stage, static_cast<uint32_t>(i), abort_flag);
        tc_fence_after_sync();
        const uint32_t a_src = base + L.ring + stage * p.stage_bytes;
        const uint32_t b_src = a_src + p.katoms * kABytes;
        for (int at = 0; at < p.katoms; ++at) {
          const uint64_t a_desc = sw128_kmajor_desc(a_src + at * kABytes);
          const uint64_t b_desc =
              p.b_kn ? sw128_mnmajor_desc(b_src + at * p.b_atom_bytes, kMnChunkBytes)
                     : sw128_kmajor_desc(b_src + at * p.b_atom_bytes);
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k)
            umma_f16(tmem_base, a_desc + 2u * k, b_desc + b_kstep * k, p.idesc, (i | at | k) != 0);
        }
        umma_commit(empty_bar(stage));  // frees the stage once these MMAs have read it
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      // The accumulator is complete once every MMA has; a timed-out tile
      // signals nothing and the epilogue leaves on the abort flag.
      if (ok) umma_commit(tfull_bar);
      umma_commit(drain_bar);
      wait_timed(drain_bar, 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    // warp w reads TMEM lane quadrant w % 4 (the quadrant it may access) and
    // stores those 32 rows of every 32-column chunk of the tile.  Its two
    // staging buffers lie in the ring's first stage, free once the tile's
    // MMAs have completed: the producer has no later loads.
    const int q = warp & 3;
    const uint32_t my_bufs = base + L.ring + (warp - 2) * kEpiBufs * kEpiChunkBytes;
    const int m0 = q * 32;
    int ok = 0;
    if (lane == 0) ok = wait_or_abort(tfull_bar, 0, p.timeout_ns, abort_flag, kSiteTmemFull);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok && m0 < p.M) {
      tc_fence_after_sync();
      fence_proxy_async_smem();  // the ring's last async-proxy uses precede these writes
      const int n0 = t * p.bn;
      const int nchunks = (min(p.bn, p.N - n0) + kEpiCols - 1) / kEpiCols;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      for (int c = 0; c < nchunks; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * kEpiCols, r);
        tmem_ld_wait();
        if (p.acc_f16) widen_f16_accumulator(r);
        const uint32_t buf = my_bufs + (c % kEpiBufs) * kEpiChunkBytes;
        if (c >= kEpiBufs) {
          if (lane == 0) bulk_wait_group_read<kEpiBufs - 1>();  // buffer's last store has read it
          __syncwarp();
        }
        if (p.scaled) {  // C passes through the staging buffer on its way to the rows' lanes
          const bool with_c = p.beta != 0.0f;
          if (with_c) stage_c_chunk(p, m0, n0 + c * kEpiCols, lane, buf);
          apply_alpha_beta(r, p, with_c, buf, lane);
        }
        // row `lane` of the 32 x 32 chunk, placed with the 64-byte swizzle of
        // the TMA store (piece j of row r at j ^ ((r >> 1) & 3))
        const uint32_t row_addr = buf + lane * 64u;
        const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          st_shared_v4(row_addr + ((j ^ sw) << 4), pack_half2(r[8 * j + 0], r[8 * j + 1]),
                       pack_half2(r[8 * j + 2], r[8 * j + 3]),
                       pack_half2(r[8 * j + 4], r[8 * j + 5]),
                       pack_half2(r[8 * j + 6], r[8 * j + 7]));
        }
        if (kDirectD) {
          __syncwarp();
          store_chunk_direct(buf, p.D, p.ldd, p.M, p.N, m0, n0 + c * kEpiCols, lane);
          __syncwarp();
        } else {
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmD, buf, n0 + c * kEpiCols, m0);
            bulk_commit_group();
          }
        }
      }
    }
    // The staging buffers must have been read before the CTA's shared memory
    // is released; the stores themselves complete with the grid.
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }

  __syncwarp();  // single-lane roles rejoin their warps
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace gb300
