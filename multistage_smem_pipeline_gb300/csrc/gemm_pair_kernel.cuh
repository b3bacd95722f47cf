// Persistent fp16 TN GEMM over CTA pairs (cluster of 2, tcgen05 cta_group::2).
//
// A pair owns a 256 x BN output tile.  Each CTA loads its own 128 rows of A
// and its own half (BN/2 rows) of B for every k-block into its stage ring;
// one thread of the even CTA issues tcgen05.mma.cta_group::2 with M = 256,
// which reads A from each CTA's shared memory and the two halves of B from
// both, and accumulates each CTA's 128 x BN block of D in that CTA's TMEM.
// Per SM, a 64-wide K slice then costs 16 KiB of A + BN/2 x 128 B of B for
// 128 x BN x 64 MACs -- half the B bytes of a single-CTA tile of the same
// width.  The ring depth follows S_min = ceil(T_copy / T_compute) + 1 of
// "第 6 课：Shared Memory 布局与异步流水", section 4, with both latencies
// measured on the GPU with every SM loading: at BN = 256 the narrow tile
// holds three stages of two slices (64 KiB each), and the wide unit below
// four stages of one slice carrying both tiles' B halves (48 KiB each),
// which is S_min for its measured T_copy (about 2550 cycles from HBM)
// against T_compute (about 1030 cycles for the slice's MMAs on both tiles).
//
// Barriers (same shared-memory offsets in both CTAs):
//   full[s]      even CTA only, count 1: the even CTA's producer arrives
//                expecting both CTAs' bytes; both CTAs' TMA loads complete
//                them (the odd CTA's bytes may land first: the transaction
//                count may go below zero within a phase, and the phase cannot
//                complete before the even CTA's arrival).  The odd CTA makes
//                no remote arrive here: a release at cluster scope per k-block
//                would put a fence in the producer's loop;
//   empty[s]     both CTAs, count 1: the pair MMA's commit, multicast;
//   tfull[b]     both CTAs, count 1: commit after a tile's last k-block, multicast;
//   tempty[b]    even CTA only: one arrive per epilogue warp of both CTAs;
//   drain        even CTA: final commit before TMEM is freed.
// As in the single-CTA kernel, every wait is bounded and a timeout is
// reported through the device error word.  On that path the odd CTA cannot
// observe its own loads landing (they complete on the even CTA's barrier);
// the even CTA's bounded drain of the full barriers, which count both CTAs'
// bytes, plus the final cluster barrier cover them.
#pragma once
#include "gemm_kernel.cuh"

namespace gb300 {

// kDirectD: as in gemm_tn_f16_persistent.
// kScaled: the epilogue forms alpha * acc + beta * C (p.scaled); the plain
// GEMM's instantiation carries none of that code, so its epilogue keeps the
// registers.
// kNT: n-tiles per work unit.  With 2 (the "wide" unit), one unit is the
// 256 x 2*BN block of two adjacent n-tiles: every ring stage carries the A
// slice once and both tiles' B halves, the MMA thread issues both tiles'
// MMAs from it into the two TMEM accumulators, and the epilogue drains the
// first accumulator, then the second.  A k-slice's bytes then feed twice the
// MMA work, so the same shared memory holds a deeper ring (4 one-slice
// stages of 48 KiB instead of 3 two-slice stages of 64 KiB at BN = 256):
// more lookahead against the DRAM latency of a slice's first fetch.  The
// accumulators are no longer double-buffered across units: the next unit's
// MMAs wait until both are drained.  Each accumulator sees the same MMAs in
// the same order as with kNT = 1, so the results are bit-identical.
// kCheck: the pipeline invariant check (as in gemm_tn_f16_persistent).
template <int kEpiWarps, bool kDirectD, int kNT, bool kScaled, bool kCheck = false>
__global__ void __launch_bounds__(threads_for(kEpiWarps), 1)
    gemm_tn_f16_pair(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw);
  constexpr int kThreads = threads_for(kEpiWarps);
  constexpr int kChunkStride = kEpiWarps / 4;  // warps sharing a TMEM lane quadrant
  // TMEM chunks read per wait in the epilogue.  The plain epilogue rounds a
  // batch to fp16 as soon as it is in registers (64 registers live for four
  // chunks); the scaled one keeps fp32 until C is applied, and the direct
  // stores need registers of their own, so those read two chunks at a time
  // to stay within the 168 registers of an 8-warp CTA.
  constexpr int kEpiBatch = (kScaled || kDirectD) ? 2 : 4;
  const SmemLayout L = SmemLayout::make(p.stages, p.stage_bytes, kEpiWarps);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  const uint32_t rank = cluster_ctarank();  // 0 = even CTA (issues the MMAs), 1 = odd
  const int pair = blockIdx.x >> 1;
  const int num_pairs = gridDim.x >> 1;
  const int half_bn = p.bn >> 1;
  const uint32_t bars = base + L.bars;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bars + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bars + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * S + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  volatile uint32_t* const slot_seq = reinterpret_cast<volatile uint32_t*>(smem + L.misc + kMiscSlotSeq);

  if (threadIdx.x == 0) {
    grid_launch_dependents();  // see gemm_tn_f16_persistent
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * kEpiWarps);  // every epilogue warp of both CTAs
    }
    mbar_init(drain_bar, 1);
    init_abort_state(abort_flag, p);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (!kDirectD) tma_prefetch_desc(&tmD);
  }
  __syncwarp();
  // Both CTAs' barriers exist before any remote arrive or multicast commit,
  // and the peer is known to be running before the collective TMEM allocation.
  cluster_sync();
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), p.tmem_cols);  // one warp in each CTA of the pair
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem_base = *tmem_slot;
  uint64_t pol_a = 0, pol_b = 0;  // the producer's L2 policies (no memory access)
  if (warp == 0 && lane == 0) {
    pol_a = l2_policy_evict_last();
    pol_b = l2_policy_evict_first();
  }
  grid_dependency_wait();  // first global-memory access follows

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      for (int t = pair; t < p.num_tiles && !*abort_flag; t += num_pairs) {
        int mb, nb;
        tile_coords(t, p, mb, nb);           // mb counts 256-row pair blocks
        const int a_row = mb * (2 * kBM) + static_cast<int>(rank) * kBM;
        const int b_row = nb * kNT * p.bn + static_cast<int>(rank) * half_bn;
        bool ok = true;
        const int k0 = first_k_block(t, p);
        for (int i = 0; i < p.num_k_blocks; ++i) {
          const int kb = (k0 + i < p.num_k_blocks) ? k0 + i : k0 + i - p.num_k_blocks;
          if (!wait_or_abort(empty_bar(stage), phase ^ 1u, p.timeout_ns, abort_flag, kSiteEmpty)) {
            ok = false;
            break;
          }
          const uint32_t a_dst = base + L.ring + stage * p.stage_bytes;
          const uint32_t b_dst = a_dst + p.katoms * kABytes;
          const uint32_t leader_full = mapa_shared(full_bar(stage), 0);
          if (rank == 0) {  // the even CTA's barrier counts both CTAs' bytes
            stamp_slot<kCheck>(slot_seq, stage, issued, p);
            mbar_arrive_expect_tx(full_bar(stage), 2u * p.stage_bytes);
          }
          if (!(p.inject == 1 && issued == 0 && rank == 0)) {
            for (int at = 0; at < p.katoms; ++at) {
              const int x = (kb * p.katoms + at) * kBK;  // past K: the box reads zeros
              const uint32_t ad = a_dst + at * kABytes;
              if (p.l2_hints & 2u)
                tma_load_2d_pair_hint(ad, &tmA, leader_full, x, a_row, pol_a);
              else
                tma_load_2d_pair(ad, &tmA, leader_full, x, a_row);
#pragma unroll
              for (int j = 0; j < kNT; ++j) {  // tile j's B half (past N: the box reads zeros)
                const uint32_t bd = b_dst + (j * p.katoms + at) * p.b_atom_bytes;
                const int br = b_row + j * p.bn;
                if (p.b_kn) {  // B is K x N: one 64-column box per chunk of this CTA's half
                  for (int ch = 0; ch < half_bn / 64; ++ch)
                    tma_load_2d_pair(bd + ch * kMnChunkBytes, &tmB, leader_full, br + 64 * ch, x);
                } else if (p.l2_hints & 1u) {
                  tma_load_2d_pair_hint(bd, &tmB, leader_full, x, br, pol_b);
                } else {
                  tma_load_2d_pair(bd, &tmB, leader_full, x, br);
                }
              }
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (rank == 0) {  // the even CTA's full barriers count both CTAs' bytes
        const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0u;
        for (uint32_t i = first; i < issued; ++i)
          wait_timed(full_bar(i % S), (i / S) & 1u, p.timeout_ns);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      const uint64_t b_kstep = p.b_kn ? 128u : 2u;  // descriptor address units per K = 16
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      uint32_t consumed = 0;  // ring slots consumed (the invariant check)
      for (int t = pair; t < p.num_tiles; t += num_pairs) {
        bool drained = true;
        for (int j = 0; j < kNT && drained; ++j)
          drained = wait_or_abort(tempty_bar(acc + j), acc_phase ^ 1u, p.timeout_ns, abort_flag,
                                  kSiteTmemEmpty);
        if (!drained) break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.bn);
        bool ok = true;
        for (int i = 0; i < p.num_k_blocks; ++i) {
          if (!wait_or_abort(full_bar(stage), phase, p.timeout_ns, abort_flag, kSiteFull)) {
            ok = false;
            break;
          }
          check_slot<kCheck>(slot_seq, stage, consumed++, abort_flag);
          tc_fence_after_sync();
          const uint32_t a_src = base + L.ring + stage * p.stage_bytes;
          const uint32_t b_src = a_src + p.katoms * kABytes;
          for (int at = 0; at < p.katoms; ++at) {
            const uint64_t a_desc = sw128_kmajor_desc(a_src + at * kABytes);
            uint64_t b_desc[kNT];
#pragma unroll
            for (int j = 0; j < kNT; ++j) {
              const uint32_t bs = b_src + (j * p.katoms + at) * p.b_atom_bytes;
              b_desc[j] = p.b_kn ? sw128_mnmajor_desc(bs, kMnChunkBytes) : sw128_kmajor_desc(bs);
            }
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k)
#pragma unroll
              for (int j = 0; j < kNT; ++j)
                umma_f16_pair(d_tmem + static_cast<uint32_t>(j * p.bn), a_desc + 2u * k,
                              b_desc[j] + b_kstep * k, p.idesc, (i | at | k) != 0);
          }
          umma_commit_pair_mc(empty_bar(stage), 0x3);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair_mc(tfull_bar(acc), 0x3);
        if (kNT == 2 || ++acc == 2) {  // a wide unit uses both accumulators
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit_pair_mc(drain_bar, 0x1);
      wait_timed(drain_bar, 0, p.timeout_ns);
      // Every epilogue warp of both CTAs has released its last accumulator
      // (the two waits a next unit would make): their remote arrivals on this
      // CTA's barriers have all landed before the pair's final barrier.
      for (int j = 0; j < 2; ++j) {
        wait_timed(tempty_bar(acc), acc_phase ^ 1u, p.timeout_ns);
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // epilogue warps: lane quadrant warp % 4 (the quadrant a warp may access
    // in TMEM); with 8 warps, each takes every other 32-column chunk of it
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t my_bufs = base + L.epi + (warp - 2) * kEpiBufs * kEpiChunkBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t chunk_seq = 0;
    for (int t = pair; t < p.num_tiles; t += num_pairs) {
      int mb, nb;
      tile_coords(t, p, mb, nb);
      int ok = 0;
      if (lane == 0)
        ok = wait_or_abort(tfull_bar(acc), acc_phase, p.timeout_ns, abort_flag, kSiteTmemFull);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const int m0 = mb * (2 * kBM) + static_cast<int>(rank) * kBM + q * 32;
      const bool rows_live = m0 < p.M;
#pragma unroll 1
      for (int j = 0; j < kNT; ++j) {  // the unit's tiles, one accumulator each
        const int n0 = (nb * kNT + j) * p.bn;
        // <= 0 when the tile lies past N (the second tile of a ragged wide unit)
        const int nchunks = (min(p.bn, p.N - n0) + kEpiCols - 1) / kEpiCols;
        const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                               static_cast<uint32_t>((acc + j) * p.bn);
        const uint32_t leader_tempty = mapa_shared(tempty_bar(acc + j), 0);
        const int last_c = last_epi_chunk(nchunks, half, kChunkStride);
        // TMEM is read kEpiBatch chunks at a time with one wait, and the
        // accumulator is released as soon as its last chunk is in registers:
        // the conversion, the C update and the stores that follow no longer
        // hold up the next unit's MMAs.
        for (int c0 = half; c0 <= last_c && rows_live; c0 += kChunkStride * kEpiBatch) {
          uint32_t r[kEpiBatch][32];
          bool c_ahead = false;  // the scaled epilogue: this chunk's C was sent ahead
#pragma unroll
          for (int b = 0; b < kEpiBatch; ++b)
            if (c0 + b * kChunkStride <= last_c)
              tmem_ld_32x32b_x32(t_row + (c0 + b * kChunkStride) * kEpiCols, r[b]);
          tmem_ld_wait();
          if (c0 + (kEpiBatch - 1) * kChunkStride >= last_c) {  // the last chunk is in this batch
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(leader_tempty);
          }
          if (!kScaled) {
            // Round the batch to fp16 now, in place: r[b][i] holds columns 2i
            // and 2i + 1.  An fp16 accumulator's bits are taken as they are
            // (the low 16 bits of each TMEM column), which is exactly what
            // widening to fp32 and rounding back gives.
#pragma unroll
            for (int b = 0; b < kEpiBatch; ++b)
#pragma unroll
              for (int i = 0; i < 16; ++i)
                r[b][i] = p.acc_f16 ? ((r[b][2 * i] & 0xffffu) | (r[b][2 * i + 1] << 16))
                                    : pack_half2(r[b][2 * i], r[b][2 * i + 1]);
          }
#pragma unroll
          for (int b = 0; b < kEpiBatch; ++b) {
            const int c = c0 + b * kChunkStride;
            if (c > last_c) break;
            if (kScaled && p.acc_f16) widen_f16_accumulator(r[b]);
            const uint32_t buf = my_bufs + (chunk_seq % kEpiBufs) * kEpiChunkBytes;
            const bool with_c = kScaled && p.beta != 0.0f;
            if (!(with_c && c_ahead) && chunk_seq >= static_cast<uint32_t>(kEpiBufs)) {
              if (lane == 0) bulk_wait_group_read<kEpiBufs - 1>();
              __syncwarp();
            }
            if (kScaled) {  // C passes through the staging buffer on its way to the rows' lanes
              if (with_c) {
                // This chunk's C is already in flight when the previous chunk
                // of the batch sent it ahead; the next chunk's C goes into the
                // other buffer once that buffer's last store has read it, and
                // lands while this chunk is finished.
                if (!c_ahead) {
                  copy_c_chunk(p, m0, n0 + c * kEpiCols, lane, buf);
                  cp_async_commit();
                }
                const int cn = c + kChunkStride;
                c_ahead = b + 1 < kEpiBatch && cn <= last_c;
                if (c_ahead) {
                  if (lane == 0) bulk_wait_group_read<0>();
                  __syncwarp();
                  copy_c_chunk(p, m0, n0 + cn * kEpiCols, lane,
                               my_bufs + ((chunk_seq + 1) % kEpiBufs) * kEpiChunkBytes);
                  cp_async_commit();
                  cp_async_wait_pending<1>();
                } else {
                  cp_async_wait_pending<0>();
                }
                __syncwarp();
              }
              apply_alpha_beta(r[b], p, with_c, buf, lane);
            }
            const uint32_t row_addr = buf + lane * 64u;
            const uint32_t sw = (lane >> 1) & 3u;
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              if (kScaled)
                st_shared_v4(row_addr + ((v ^ sw) << 4),
                             pack_half2(r[b][8 * v + 0], r[b][8 * v + 1]),
                             pack_half2(r[b][8 * v + 2], r[b][8 * v + 3]),
                             pack_half2(r[b][8 * v + 4], r[b][8 * v + 5]),
                             pack_half2(r[b][8 * v + 6], r[b][8 * v + 7]));
              else
                st_shared_v4(row_addr + ((v ^ sw) << 4), r[b][4 * v], r[b][4 * v + 1],
                             r[b][4 * v + 2], r[b][4 * v + 3]);
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
            ++chunk_seq;
          }
        }
        if (!rows_live || last_c < 0) {
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(leader_tempty);
        }
      }
      if (kNT == 2 || ++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // The staging buffers must have been read before the CTA's shared memory
    // is released; the stores themselves complete with the grid.
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }

  __syncwarp();
  tc_fence_before_sync();
  // No remote arrive or commit still targets either CTA (the MMA thread has
  // seen the last ones land), so the arrive need not wait for the D stores.
  cluster_sync_relaxed();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem_base, p.tmem_cols);
  }
}

}  // namespace gb300
