// Split-K fp16 TN GEMM over a CTA pair, for shapes whose k loops are short
// enough that each CTA's fill and MMA issue set the time (1024^3: one wave of
// 128 x 64 tiles, each CTA pulling 384 KiB through its SM for 8 k-blocks).
//
// A cluster of two CTAs owns one 128 x BN tile of D.  CTA r multiplies the
// r-th half of the k range into its own TMEM accumulator (the pipeline of
// "cute(9) multistage_gemm": a ring of K-tiles filled ahead of the MMAs,
// guarded by full and empty barriers, here TMA loads and tcgen05.mma).  Then
// each CTA finalises half of the tile's columns: CTA r keeps columns
// [r BN/2, (r+1) BN/2), sends its fp32 partial of the other half into the
// peer's shared memory (st.async), receives the peer's partial of
// its own half, adds the two, rounds to fp16 and stores D.  Per CTA that is
// half the k-blocks of a 128 x BN tile -- at 1024^3 with BN = 128, 256 KiB of
// operands and 32 MMAs per CTA instead of 384 KiB and 64 for a 128 x 64 tile
// over the whole k range -- for a 32 KiB exchange.
//
// The peer's partial lands in a region of its own after the ring
// (128 x BN/2 x 4 bytes), so a CTA may send as soon as its own MMAs are done,
// without waiting for the peer's.  Each epilogue warp loads its 32 x 32
// chunk of the peer's half from TMEM and stores it from registers into the
// peer's region with 16-byte remote stores whose bytes complete on the peer's
// receive barrier (one expect_tx of the whole half, made at set-up).  The
// epilogue's staging buffers for D reuse the ring, idle once the CTA's MMAs
// have completed (one tile per pair).  Eight epilogue warps, two per TMEM lane
// quadrant, each send and finish every other 32-column chunk.  The final
// value of an element is p0 + p1 in fp32 whichever CTA forms it, so the
// result does not depend on the pair's timing.  Every wait is bounded; both
// CTAs meet on a cluster barrier before either exits (a relaxed one: each has
// already seen the peer's partial land, so it need not wait for its stores).
#pragma once
#include "gemm_kernel.cuh"

namespace gb300 {

constexpr int kSplitEpiWarps = 8;
constexpr int kSplitThreads = 64 + 32 * kSplitEpiWarps;  // producer, MMA, epilogue
constexpr uint32_t kSplitStagingBytes = kSplitEpiWarps * kEpiBufs * kEpiChunkBytes;  // 32 KiB

// Bytes of ring the epilogue reuses: the staging buffers for D.
__host__ __device__ constexpr uint32_t splitk_ring_reuse_bytes(int /*bn*/) {
  return kSplitStagingBytes;
}

// Shared-memory carve-up, offsets from the 1024-aligned base: the ring (see
// splitk_ring_reuse_bytes), the peer's fp32 partial of this CTA's BN/2
// columns, then the mbarriers full[S], empty[S], tmem-full, drain, rx-full.
struct SplitLayout {
  uint32_t ring, rx, bars, misc, total;
  __host__ __device__ static SplitLayout make(int stages, uint32_t stage_bytes, int bn) {
    SplitLayout L;
    L.ring = 0;
    L.rx = stages * stage_bytes;
    L.bars = L.rx + static_cast<uint32_t>(bn) * 256u;
    L.misc = L.bars + 8 * (2 * stages + 3);
    L.total = L.misc + kMiscBytes;
    return L;
  }
};

// wait_or_abort with acquire at cluster scope (for barriers the peer arrives on).
__device__ __forceinline__ bool wait_cluster_or_abort(uint32_t bar, uint32_t parity,
                                                      uint64_t timeout_ns, volatile int* abort_flag,
                                                      uint32_t site) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > timeout_ns) {
        *abort_flag = 1;
        record_error(kErrTimeout, site, abort_flag);
        return false;
      }
    }
  }
}

// A partial of half a tile, 128 rows x BN/2 fp32 columns, as the epilogue
// warps hold it: chunk c (32 columns) of lane quadrant q is 4 KiB at
// (c * 4 + q) * 4096, in which 16-byte group g (columns 4g..4g+3) of row
// q * 32 + lane lies at g * 512 + lane * 16 -- one contiguous 4 KiB block
// per warp and chunk, and conflict-free 16-byte stores and loads across a warp.
__device__ __forceinline__ uint32_t splitk_chunk_offset(int c, int q) {
  return static_cast<uint32_t>(c * 4 + q) * 4096u;
}

// kCheck: the pipeline invariant check (as in gemm_tn_f16_persistent).
// kMcN, kMcM: 2 to put the next n-tile (m-tile) in the same cluster.  The CTAs
// of one k-half whose tiles share a block of A (same m-block) then each load
// half of its rows for both by TMA multicast, and likewise for B: each SM
// fetches half the bytes it receives.  Every CTA's ring slot is then written
// by its multicast partners too, so a slot is free only when every CTA that
// writes into it has consumed it: each MMA commit arrives on the empty
// barrier of the CTA itself and of its partners, and each empty barrier
// counts one arrival per CTA.  The host passes the grid of cluster tiles
// (kMcM x kMcN tiles each) in num_m_blocks and num_n_blocks.
template <bool kCheck = false, int kMcN = 1, int kMcM = 1>
__global__ void __launch_bounds__(kSplitThreads, 1)
    gemm_tn_f16_splitk(const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB,
                       const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw);
  const int S = p.stages;
  const SplitLayout L = SplitLayout::make(S, p.stage_bytes, p.bn);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  static_assert((kMcN == 1 || kMcN == 2) && (kMcM == 1 || kMcM == 2), "1 or 2 tiles per dimension");
  constexpr int kClusterCtas = 2 * kMcN * kMcM;
  constexpr bool kMc = kClusterCtas > 2;
  const uint32_t rank = cluster_ctarank();
  const uint32_t kr = rank & 1u;                           // this CTA's k-half
  const uint32_t peer = rank ^ 1u;                         // the other k-half of this tile
  const uint32_t a_mate = rank ^ 2u;                       // kMcN: same m-block, next n-block
  const uint32_t b_mate = rank ^ (kMcN == 2 ? 4u : 2u);    // kMcM: same n-block, next m-block
  const int jn = kMcN == 2 ? static_cast<int>((rank >> 1) & 1u) : 0;
  const int jm = kMcM == 2 ? static_cast<int>((rank >> (kMcN == 2 ? 2 : 1)) & 1u) : 0;
  const uint16_t a_mask = static_cast<uint16_t>((1u << rank) | (1u << a_mate));
  const uint16_t b_mask = static_cast<uint16_t>((1u << rank) | (1u << b_mate));
  const uint16_t commit_mask = static_cast<uint16_t>(
      (1u << rank) | (kMcN == 2 ? 1u << a_mate : 0u) | (kMcM == 2 ? 1u << b_mate : 0u));
  int mb, nb;
  tile_coords(static_cast<int>(blockIdx.x / kClusterCtas), p, mb, nb);
  mb = mb * kMcM + jm;
  nb = nb * kMcN + jn;
  // this CTA's k-blocks: the first ceil(nk/2) for k-half 0, the rest for k-half 1
  const int h0 = (p.num_k_blocks + 1) / 2;
  const int kb_lo = kr ? h0 : 0;
  const int nkb = kr ? p.num_k_blocks - h0 : h0;
  const uint32_t bars = base + L.bars;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  const uint32_t tfull_bar = bars + 8u * (2 * S);
  const uint32_t drain_bar = bars + 8u * (2 * S + 1);
  const uint32_t rx_full_bar = bars + 8u * (2 * S + 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  volatile uint32_t* const slot_seq = reinterpret_cast<volatile uint32_t*>(smem + L.misc + kMiscSlotSeq);

  if (threadIdx.x == 0) {
    grid_launch_dependents();  // see gemm_tn_f16_persistent
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1 + (kMcN == 2) + (kMcM == 2));  // one commit per writing CTA
    }
    mbar_init(tfull_bar, 1);
    mbar_init(drain_bar, 1);
    mbar_init(rx_full_bar, 1);
    // the peer's remote stores of this CTA's half complete these bytes
    mbar_arrive_expect_tx(rx_full_bar, static_cast<uint32_t>(p.bn) * 256u);
    init_abort_state(abort_flag, p);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tmD);
  }
  __syncwarp();
  cluster_sync();  // every CTA's barriers exist before any remote arrive or multicast
  uint32_t tmem_base = 0;
  if (warp != 0) {
    if (warp == 1) {
      tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
      tmem_relinquish();
    }
    tc_fence_before_sync();
    named_barrier_sync(1, kSplitThreads - 32);
    tc_fence_after_sync();
    tmem_base = *tmem_slot;
  }
  grid_dependency_wait();  // first global-memory access follows

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      for (int i = 0; i < nkb && !*abort_flag; ++i) {
        const int kb = kb_lo + i;
        if (!wait_or_abort(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, kSiteEmpty))
          break;
        const uint32_t a_dst = base + L.ring + stage * p.stage_bytes;
        const uint32_t b_dst = a_dst + p.katoms * kABytes;
        stamp_slot<kCheck>(slot_seq, stage, issued, p);
        mbar_arrive_expect_tx(full_bar(stage), p.stage_bytes);
        if (!(p.inject == 1 && issued == 0)) {
          for (int at = 0; at < p.katoms; ++at) {
            const int x = (kb * p.katoms + at) * kBK;  // past K (or M, N): the box reads zeros
            const uint32_t ad = a_dst + at * kABytes, bd = b_dst + at * p.b_atom_bytes;
            if (kMcN == 2)  // rows jn * 64 .. +64 of the A block, for this CTA and its a-mate
              tma_load_2d_mc(ad + jn * (kABytes / 2), &tmA, full_bar(stage), x,
                             mb * kBM + jn * (kBM / 2), a_mask);
            else
              tma_load_2d(ad, &tmA, full_bar(stage), x, mb * kBM);
            if (kMcM == 2)  // rows jm * BN/2 .. of the B block, for this CTA and its b-mate
              tma_load_2d_mc(bd + jm * (p.b_atom_bytes / 2), &tmB, full_bar(stage), x,
                             nb * p.bn + jm * (p.bn / 2), b_mask);
            else
              tma_load_2d(bd, &tmB, full_bar(stage), x, nb * p.bn);
          }
        }
        ++issued;
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0u;
      for (uint32_t i = first; i < issued; ++i)
        wait_timed(full_bar(i % S), (i / S) & 1u, p.timeout_ns);
      // The partners' commits on this CTA's empty barriers have landed before
      // the cluster's final barrier (their last phases complete).
      if (kMc)
        for (uint32_t i = first; i < issued; ++i)
          wait_timed(empty_bar(i % S), (i / S) & 1u, p.timeout_ns);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int i = 0; i < nkb; ++i) {
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
          const uint64_t b_desc = sw128_kmajor_desc(b_src + at * p.b_atom_bytes);
#pragma unroll
          for (int k = 0; k < kBK / kUmmaK; ++k)
            umma_f16(tmem_base, a_desc + 2u * k, b_desc + 2u * k, p.idesc, (i | at | k) != 0);
        }
        if (kMc)
          umma_commit_mc(empty_bar(stage), commit_mask);
        else
          umma_commit(empty_bar(stage));
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) umma_commit(tfull_bar);
      umma_commit(drain_bar);
      wait_timed(drain_bar, 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..9)
    const int q = warp & 3;            // TMEM lane quadrant this warp may access
    const int sel = (warp - 2) >> 2;   // which of every two 32-column chunks it takes
    const int m0 = mb * kBM + q * 32;
    const bool rows_live = m0 < p.M;
    const int half = p.bn / 2;  // a multiple of 32
    const uint32_t my_bufs = base + L.ring + (warp - 2) * kEpiBufs * kEpiChunkBytes;
    const uint32_t rx = base + L.rx;
    const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    int ok = 0;
    if (lane == 0) ok = wait_or_abort(tfull_bar, 0, p.timeout_ns, abort_flag, kSiteTmemFull);
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok) {
      tc_fence_after_sync();
      fence_proxy_async_smem();  // the ring's last async-proxy uses precede the writes below
      // 1. send this CTA's partial of the peer's half straight from registers
      // into the peer's region: 16-byte remote stores whose bytes complete on
      // the peer's receive barrier
      const uint32_t rx_peer = mapa_shared(rx, peer) + lane * 16u;
      const uint32_t rx_full_peer = mapa_shared(rx_full_bar, peer);
      for (int c = sel; c < half / kEpiCols; c += 2) {
        const uint32_t off = splitk_chunk_offset(c, q);
        uint32_t r[32];
        if (rows_live) {
          tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>((kr ^ 1u) * half + c * kEpiCols), r);
          tmem_ld_wait();
        } else {  // rows past M: the peer stores nothing there, but the bytes are counted
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
#pragma unroll
        for (int g = 0; g < 8; ++g)
          st_async_cluster_v4(rx_peer + off + g * 512u, r[4 * g], r[4 * g + 1], r[4 * g + 2],
                              r[4 * g + 3], rx_full_peer);
      }
      // 2. the peer's partial of this CTA's half: add, round, store (the warp
      // goes on only if every lane saw it land, so the tcgen05.ld below stays
      // warp-uniform)
      if (__all_sync(0xffffffffu, wait_cluster_or_abort(rx_full_bar, 0, p.timeout_ns, abort_flag,
                                                        kSiteTmemFull)) &&
          rows_live) {
        const int n0 = nb * p.bn + static_cast<int>(kr) * half;
        const int nchunks = (min(half, p.N - n0) + kEpiCols - 1) / kEpiCols;
        int seq = 0;
        for (int c = sel; c < nchunks; c += 2, ++seq) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(kr * half + c * kEpiCols), r);
          tmem_ld_wait();
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            const uint4 v = ld_shared_v4(rx + splitk_chunk_offset(c, q) + g * 512u + lane * 16u);
            r[4 * g] = __float_as_uint(__uint_as_float(r[4 * g]) + __uint_as_float(v.x));
            r[4 * g + 1] = __float_as_uint(__uint_as_float(r[4 * g + 1]) + __uint_as_float(v.y));
            r[4 * g + 2] = __float_as_uint(__uint_as_float(r[4 * g + 2]) + __uint_as_float(v.z));
            r[4 * g + 3] = __float_as_uint(__uint_as_float(r[4 * g + 3]) + __uint_as_float(v.w));
          }
          const uint32_t buf = my_bufs + (seq % kEpiBufs) * kEpiChunkBytes;
          if (seq >= kEpiBufs) {
            if (lane == 0) bulk_wait_group_read<kEpiBufs - 1>();
            __syncwarp();
          }
          if (p.scaled) {
            const bool with_c = p.beta != 0.0f;
            if (with_c) stage_c_chunk(p, m0, n0 + c * kEpiCols, lane, buf);
            apply_alpha_beta(r, p, with_c, buf, lane);
          }
          const uint32_t row_addr = buf + lane * 64u;
          const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_shared_v4(row_addr + ((j ^ sw) << 4), pack_half2(r[8 * j + 0], r[8 * j + 1]),
                         pack_half2(r[8 * j + 2], r[8 * j + 3]),
                         pack_half2(r[8 * j + 4], r[8 * j + 5]),
                         pack_half2(r[8 * j + 6], r[8 * j + 7]));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmD, buf, n0 + c * kEpiCols, m0);
            bulk_commit_group();
          }
        }
      }
    }
    if (lane == 0) bulk_wait_group_read<0>();
    // After a timeout the peer's copies into this CTA may still be landing:
    // give them a bounded wait before the shared memory is released (at once
    // when the partial has arrived).
    if (warp == 2 && lane == 0) wait_timed(rx_full_bar, 0, p.timeout_ns);
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before_sync();
  // Each CTA has seen the peer's partial land (rx-full), and with multicast
  // its partners' bytes (full) and commits (empty), before it gets here, so
  // nothing targets a CTA that has left; the arrive need not wait for the D
  // stores.
  cluster_sync_relaxed();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace gb300
