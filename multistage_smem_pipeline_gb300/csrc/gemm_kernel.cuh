// Persistent, warp-specialised fp16 TN GEMM for sm_103a.
//
// One CTA per SM walks a list of 128 x BN output tiles.  Inside the CTA:
//   warp 0, one thread  -- producer: TMA loads of the A (128 x 64) and B
//                          (BN x 64) k-blocks into a `stages`-deep ring;
//   warp 1, one thread  -- MMA issuer: 4 x tcgen05.mma (K = 16 each) per
//                          k-block into an fp32 accumulator in TMEM;
//   warps 2..          -- epilogue (4 or 8 warps): TMEM -> registers -> fp16 ->
//                          swizzled shared memory -> TMA store, while the MMA
//                          thread already fills the second TMEM accumulator;
//                          with 8 warps two share each TMEM lane quadrant and
//                          take alternate 32-column chunks.
// With one n-block (N <= BN) every tile multiplies by the same B; in the
// resident-B mode the producer loads all of B (BN x K) once into its own
// shared-memory region, each k-block behind its own barrier and issued with
// the first tile's A stage that needs it, and the ring carries only A.
//
// This is the multistage pipeline of "cute(9) multistage_gemm" (sections 4-6:
// a ring of kStage K-tiles, a prologue that runs ahead, a mainloop that
// overlaps the copy of tile k+S-1 with the MMA of tile k) in Blackwell form.
// The page's cp_async_wait<kStage-2> + __syncthreads (the read-after-write
// guard) becomes a wait on the stage's "full" mbarrier, whose transaction
// count the TMA engine decrements as bytes land; the page's rule that a stage
// is overwritten only after all its reads (the write-after-read guard,
// "第 6 课：Shared Memory 布局与异步流水", section 3) becomes the "empty"
// mbarrier that tcgen05.commit arrives on once the MMAs reading the stage
// have completed.  The prologue's "fill kStage-1 stages" is implicit: the
// producer runs ahead until every empty barrier is taken.  The page's
// register double-buffer (ldmatrix of ik+1 during the MMA of ik) has no
// counterpart: tcgen05.mma reads its operands from shared memory directly.
// The page's Reg->Global epilogue is replaced by the Reg->Shared->Global form
// its section 7 recommends, using TMA stores.
//
// Every wait is bounded (a per-wait %globaltimer limit); on expiry the
// kernel records GEMM_ERR_TIMEOUT in a device error word, all roles leave
// their loops, in-flight copies and MMAs are drained with bounded waits, and
// TMEM is freed, so the context stays usable.
#pragma once
#include "pipeline.cuh"

namespace gb300 {

// The device error words: the first error of the kernels launched on a given
// stream (the host maps streams to words), 0 = none.
__device__ unsigned int g_gemm_error[kErrorSlots];

// `state` is the CTA's abort flag, followed by the index of its error word.
__device__ __forceinline__ void record_error(uint32_t code, uint32_t site,
                                             const volatile int* state) {
  atomicCAS(&g_gemm_error[static_cast<uint32_t>(state[1]) % kErrorSlots], 0u, code | (site << 8));
}

// The CTA's abort flag and error-word index, set by one thread at start-up.
__device__ __forceinline__ void init_abort_state(volatile int* state, const GemmParams& p) {
  state[0] = 0;
  state[1] = p.err_slot;
}

// The MMA thread's half of the invariant check (see stamp_slot).
template <bool kCheck>
__device__ __forceinline__ void check_slot(const volatile uint32_t* seq, int stage,
                                           uint32_t consumed, const volatile int* state) {
  if (kCheck && seq[stage] != consumed) record_error(kErrInvariant, kSiteRingSeq, state);
}

// Wait for phase `parity` of `bar`; give up when the CTA is aborting or after
// timeout_ns without completion (then record the error and start the abort).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, uint64_t timeout_ns,
                                              volatile int* abort_flag, uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
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

// kResident selects the resident-B mode at compile time (p.b_resident must
// agree), so the streaming kernel's loops carry none of its code.  kDirectD
// stores D with plain stores to p.D (row stride p.ldd) instead of TMA stores
// through tmD, which such kernels never touch.  kCheck adds the pipeline
// invariant check (p.check), at no cost to the kernels without it.
template <int kEpiWarps, bool kResident, bool kDirectD, bool kCheck = false>
__global__ void __launch_bounds__(threads_for(kEpiWarps), 1)
    gemm_tn_f16_persistent(const __grid_constant__ CUtensorMap tmA,
                           const __grid_constant__ CUtensorMap tmB,
                           const __grid_constant__ CUtensorMap tmD, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* const smem = smem_raw + (base - raw);
  constexpr int kThreads = threads_for(kEpiWarps);
  constexpr int kChunkStride = kEpiWarps / 4;  // warps sharing a TMEM lane quadrant
  const SmemLayout L =
      SmemLayout::make(p.stages, p.stage_bytes, kEpiWarps, kResident ? p.bres_bytes : 0u,
                       kResident ? p.num_k_blocks : 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int S = p.stages;
  const uint32_t bars = base + L.bars;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (S + s); };
  auto tfull_bar = [&](int b) { return bars + 8u * (2 * S + b); };
  auto tempty_bar = [&](int b) { return bars + 8u * (2 * S + 2 + b); };
  const uint32_t drain_bar = bars + 8u * (2 * S + 4);
  // k-block j of the resident B completes on its own barrier
  auto bres_bar = [&](int j) { return bars + 8u * (2 * S + 5 + j); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L.misc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.misc + 4);
  volatile uint32_t* const slot_seq = reinterpret_cast<volatile uint32_t*>(smem + L.misc + kMiscSlotSeq);

  if (threadIdx.x == 0) {
    // The next GEMM in the stream may start its own set-up on SMs this grid
    // frees; its griddepcontrol.wait still orders it after this grid.
    grid_launch_dependents();
    for (int s = 0; s < S; ++s) {
      mbar_init(full_bar(s), 1);   // producer's arrive.expect_tx; TMA bytes complete it
      mbar_init(empty_bar(s), 1);  // one tcgen05.commit per consumed stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);          // tcgen05.commit after a tile's last k-block
      mbar_init(tempty_bar(b), kEpiWarps); // one arrive per epilogue warp
    }
    mbar_init(drain_bar, 1);
    if (kResident)
      for (int j = 0; j < p.num_k_blocks; ++j)
        mbar_init(bres_bar(j), 1);  // producer's arrive.expect_tx for k-block j of B
    init_abort_state(abort_flag, p);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    if (!kDirectD) tma_prefetch_desc(&tmD);
    // The first ring of this CTA's first tile, fetched into L2 while the
    // previous grid finishes (see tma_prefetch_l2_2d).
    const int t0 = static_cast<int>(blockIdx.x);
    if (t0 < p.num_tiles) {
      int mb, nb;
      tile_coords(t0, p, mb, nb);
      const int kf = first_k_block(t0, p);
      for (int i = 0; i < p.num_k_blocks && i < S; ++i) {
        const int kb = (kf + i < p.num_k_blocks) ? kf + i : kf + i - p.num_k_blocks;
        for (int at = 0; at < p.katoms; ++at) {
          const int x = (kb * p.katoms + at) * kBK;
          tma_prefetch_l2_2d(&tmA, x, mb * kBM);
          if (p.b_kn) {
            for (int ch = 0; ch < p.bn / 64; ++ch) tma_prefetch_l2_2d(&tmB, nb * p.bn + 64 * ch, x);
          } else {
            tma_prefetch_l2_2d(&tmB, x, kResident ? static_cast<int>(blockIdx.x % p.num_n_blocks) * p.bn
                                                  : nb * p.bn);
          }
        }
      }
    }
  }
  __syncwarp();  // reconverge warp 0 before the aligned CTA barrier
  __syncthreads();  // barriers initialised: the producer may start loading at once
  uint32_t tmem_base = 0;
  if (warp != 0) {
    // TMEM is needed only by the MMA and epilogue warps (1..); they meet on
    // named barrier 1 while the producer already streams the first stages.
    if (warp == 1) {
      tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
      tmem_relinquish();
    }
    tc_fence_before_sync();
    named_barrier_sync(1, kThreads - 32);
    tc_fence_after_sync();
    tmem_base = *tmem_slot;
  }
  // The producer's L2 policies are made before the wait: they touch no
  // memory, and the first loads need not wait for them.
  uint64_t pol_a = 0, pol_b = 0;
  if (warp == 0 && lane == 0) {
    pol_b = l2_policy_evict_first();
    pol_a = l2_policy_evict_last();
  }
  // Set-up done without touching global memory; from here on the previous
  // kernel's results must be complete and visible.
  grid_dependency_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0;
      // Resident B: every tile of this CTA multiplies by the same n-block of
      // B (the host orders tiles n-fastest over a grid that is a multiple of
      // num_n).  Its k-blocks are loaded once, during the first tile, each
      // just before that tile's A stage for the same k-block and behind its
      // own barrier, so the first MMAs need not wait for all of B.
      const int n_row = static_cast<int>(blockIdx.x % p.num_n_blocks) * p.bn;
      int b_issued = 0;
      for (int t = blockIdx.x; t < p.num_tiles && !*abort_flag; t += gridDim.x) {
        int mb, nb;
        tile_coords(t, p, mb, nb);
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
          if (kResident && t == static_cast<int>(blockIdx.x)) {  // B's k-block kb, once
            mbar_arrive_expect_tx(bres_bar(kb), p.katoms * p.b_atom_bytes);
            for (int at = 0; at < p.katoms; ++at)
              tma_load_2d(base + L.bres + (kb * p.katoms + at) * p.b_atom_bytes, &tmB,
                          bres_bar(kb), (kb * p.katoms + at) * kBK, n_row);
            ++b_issued;
          }
          stamp_slot<kCheck>(slot_seq, stage, issued, p);
          mbar_arrive_expect_tx(full_bar(stage), p.stage_bytes);
          if (!(p.inject == 1 && issued == 0)) {
            for (int at = 0; at < p.katoms; ++at) {
              const int x = (kb * p.katoms + at) * kBK;  // past K: the box reads zeros
              const uint32_t ad = a_dst + at * kABytes, bd = b_dst + at * p.b_atom_bytes;
              if (p.l2_hints & 2u)
                tma_load_2d_hint(ad, &tmA, full_bar(stage), x, mb * kBM, pol_a);
              else
                tma_load_2d(ad, &tmA, full_bar(stage), x, mb * kBM);
              if (kResident) {
                // B is already in its own region
              } else if (p.b_kn) {  // B is K x N: one 64-column box per chunk of the tile
                for (int ch = 0; ch < p.bn / 64; ++ch)
                  tma_load_2d(bd + ch * kMnChunkBytes, &tmB, full_bar(stage), nb * p.bn + 64 * ch,
                              x);
              } else if (p.l2_hints & 1u) {
                tma_load_2d_hint(bd, &tmB, full_bar(stage), x, nb * p.bn, pol_b);
              } else {
                tma_load_2d(bd, &tmB, full_bar(stage), x, nb * p.bn);
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
      // Drain: the loads of the last min(issued, S) stages must have landed
      // before the CTA (and its shared memory) goes away.
      const uint32_t first = issued > static_cast<uint32_t>(S) ? issued - S : 0u;
      for (uint32_t i = first; i < issued; ++i)
        wait_timed(full_bar(i % S), (i / S) & 1u, p.timeout_ns);
      if (kResident) {
        const int kf = first_k_block(blockIdx.x, p);  // the first tile's k order
        for (int j = 0; j < b_issued; ++j) {
          const int kb = (kf + j < p.num_k_blocks) ? kf + j : kf + j - p.num_k_blocks;
          wait_timed(bres_bar(kb), 0, p.timeout_ns);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint64_t b_kstep = p.b_kn ? 128u : 2u;  // descriptor address units per K = 16
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool first_tile = true;  // resident B: its k-blocks are still landing
      uint32_t consumed = 0;   // ring slots consumed (the invariant check)
      for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
        if (!wait_or_abort(tempty_bar(acc), acc_phase ^ 1u, p.timeout_ns, abort_flag,
                           kSiteTmemEmpty))
          break;
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.bn);
        const int k0 = kResident ? first_k_block(t, p) : 0;
        bool ok = true;
        for (int i = 0; i < p.num_k_blocks; ++i) {
          if (!wait_or_abort(full_bar(stage), phase, p.timeout_ns, abort_flag, kSiteFull)) {
            ok = false;
            break;
          }
          check_slot<kCheck>(slot_seq, stage, consumed++, abort_flag);
          const uint32_t a_src = base + L.ring + stage * p.stage_bytes;
          uint32_t b_src = a_src + p.katoms * kABytes;
          if (kResident) {
            const int kb = (k0 + i < p.num_k_blocks) ? k0 + i : k0 + i - p.num_k_blocks;
            b_src = base + L.bres + kb * p.katoms * p.b_atom_bytes;
            if (first_tile &&
                !wait_or_abort(bres_bar(kb), 0, p.timeout_ns, abort_flag, kSiteFull)) {
              ok = false;
              break;
            }
          }
          tc_fence_after_sync();
          for (int at = 0; at < p.katoms; ++at) {
            const uint64_t a_desc = sw128_kmajor_desc(a_src + at * kABytes);
            const uint64_t b_desc =
                p.b_kn ? sw128_mnmajor_desc(b_src + at * p.b_atom_bytes, kMnChunkBytes)
                       : sw128_kmajor_desc(b_src + at * p.b_atom_bytes);
#pragma unroll
            for (int k = 0; k < kBK / kUmmaK; ++k) {
              // K-major: +32 bytes along K inside the 128-byte swizzle row = +2
              // in the descriptor's address field (16-byte units); MN-major:
              // +16 rows of 128 bytes = +128
              umma_f16(d_tmem, a_desc + 2u * k, b_desc + b_kstep * k, p.idesc, (i | at | k) != 0);
            }
          }
          umma_commit(empty_bar(stage));  // frees the stage once these MMAs have read it
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull_bar(acc));      // accumulator complete
        first_tile = false;
        if (++acc == 2) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // Drain: every MMA issued by this thread completes before TMEM is freed.
      umma_commit(drain_bar);
      wait_timed(drain_bar, 0, p.timeout_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // epilogue warps: lane quadrant warp % 4 (the quadrant a warp may access
    // in TMEM); with 8 warps, each takes every other 32-column chunk of it
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const uint32_t my_bufs = base + L.epi + (warp - 2) * kEpiBufs * kEpiChunkBytes;
    int acc = 0;
    uint32_t acc_phase = 0;
    uint32_t chunk_seq = 0;
    for (int t = blockIdx.x; t < p.num_tiles; t += gridDim.x) {
      int mb, nb;
      tile_coords(t, p, mb, nb);
      int ok = 0;
      if (lane == 0)
        ok = wait_or_abort(tfull_bar(acc), acc_phase, p.timeout_ns, abort_flag, kSiteTmemFull);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after_sync();
      const int m0 = mb * kBM + q * 32;
      const int n0 = nb * p.bn;
      const bool rows_live = m0 < p.M;
      const int nchunks = (min(p.bn, p.N - n0) + kEpiCols - 1) / kEpiCols;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * p.bn);
      const int last_c = last_epi_chunk(nchunks, half, kChunkStride);
      for (int c = half; c <= last_c && rows_live; c += kChunkStride) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * kEpiCols, r);
        tmem_ld_wait();
        if (c == last_c) {  // accumulator fully read: hand it back to the MMA thread
          tc_fence_before_sync();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty_bar(acc));
        }
        if (p.acc_f16) widen_f16_accumulator(r);
        const uint32_t buf = my_bufs + (chunk_seq % kEpiBufs) * kEpiChunkBytes;
        if (chunk_seq >= static_cast<uint32_t>(kEpiBufs)) {
          if (lane == 0) bulk_wait_group_read<kEpiBufs - 1>();  // buffer's last store has read it
          __syncwarp();
        }
        if (p.scaled) {  // C passes through the staging buffer on its way to the rows' lanes
          const bool with_c = p.beta != 0.0f;
          if (with_c) stage_c_chunk(p, m0, n0 + c * kEpiCols, lane, buf);
          apply_alpha_beta(r, p, with_c, buf, lane);
        }
        // Row `lane` of the 32 x 32 box, 64 bytes = four 16-byte pieces, placed
        // with the 64-byte swizzle the TMA store expects (piece j of row r at
        // position j ^ ((r >> 1) & 3)); conflict-free across the warp.
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
        ++chunk_seq;
      }
      if (!rows_live || last_c < 0) {  // nothing for this warp to store: release at once
        tc_fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty_bar(acc));
      }
      if (++acc == 2) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    // The staging buffers must have been read before the CTA's shared memory
    // is released; the stores themselves complete with the grid.
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
  }

  __syncwarp();  // single-lane roles rejoin their warps
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

}  // namespace gb300
