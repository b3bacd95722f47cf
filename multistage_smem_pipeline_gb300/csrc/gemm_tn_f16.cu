// Host side of the C-ABI: argument checks, configuration choice, TMA
// descriptor encoding and the launch of the persistent kernel.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm_pair_kernel.cuh"
#include "gemm_skinny_kernel.cuh"
#include "gemm_splitk_kernel.cuh"
#include "gemm_tn_f16.h"
#include "host.cuh"

namespace gb300 {

struct DeviceState {
  bool init = false;
  int status = GEMM_OK;
  int sm_count = 0;
  int smem_attr = 0;       // dynamic smem granted to the single-CTA kernel
  int pair_smem_attr = 0;  // ... and to the pair kernel
  int max_pairs = 0;       // co-resident 2-CTA clusters at full shared memory
  int max_quads = 0;       // ... 4-CTA clusters (split K with multicast)
  int max_octs = 0;        // ... 8-CTA clusters
};

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxDynSmem = 232448;  // 227 KiB opt-in limit per CTA on sm_100-class parts
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr int kMaxResidentN = 4;  // n-blocks a resident-B plan may have
constexpr int64_t kWideMinK = 4096;  // shortest k loop for which wide pair units are chosen
constexpr int kSkinnyKatoms = 2;     // K slices per stage of the small-M kernel's ring

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

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

// Deepest ring (at least 2) whose carve-up, plus 1 KiB of alignment slack,
// fits the dynamic shared memory limit; 1 if not even 2 stages fit.
int stages_that_fit(uint32_t stage_bytes, int epi_warps, uint32_t bres_bytes = 0,
                    int bres_bars = 1) {
  const auto fits = [&](int s) {
    return SmemLayout::make(s, stage_bytes, epi_warps, bres_bytes, bres_bars).total + 1024 <=
           static_cast<uint32_t>(kMaxDynSmem);
  };
  if (!fits(2)) return 1;
  int s = 2;
  while (s + 1 <= kMaxStages && fits(s + 1)) ++s;
  return s;
}

// Relative time of one k-block on one SM: the tensor pipe needs 2*n cycles
// for its 128 x n x 64 block (8192 flop/clk/SM), and the stage must be
// refilled at the rate the ring sustains with every SM loading -- about
// 60 B/clk per SM measured on GB300 with a 4-6 deep ring.
// With `mmas` > 0 the MMA side is also floored at kMmaIssueCycles per
// instruction: the issuing thread needs about that long per tcgen05.mma
// (measured issue to issue), so a 128 x n x 16 MMA with n/2 < 124 cycles of
// tensor work is issue-bound.  Applied to the pair path, where it decides
// between tile widths (measured: wide units at bn 160-192 ran at 0.7x of bn
// 256); the single-CTA plans for short k loops were measured without it.
constexpr double kMmaIssueCycles = 124.0;
double kblock_cost(int n_per_sm, uint32_t stage_bytes, int mmas = 0) {
  const double mma = std::max(2.0 * n_per_sm, mmas * kMmaIssueCycles);
  return std::max(mma, static_cast<double>(stage_bytes) / 60.0);
}

uint32_t b_atom_bytes_for(int path, int bn) {
  const int b_rows = (path == GEMM_PATH_PAIR) ? bn / 2 : bn;
  return static_cast<uint32_t>(b_rows) * 128u;
}

// nt: n-tiles sharing each A slice (2 for a wide pair unit)
uint32_t stage_bytes_for(int path, int bn, int katoms = 1, int nt = 1) {
  return static_cast<uint32_t>(katoms) * (kABytes + nt * b_atom_bytes_for(path, bn));
}

struct Plan {
  gemm_config_t cfg;
  GemmParams p;
  int mc_n, mc_m;  // split K: tiles per cluster along n and m (multicast operands)
};

int make_plan(int64_t M, int64_t N, int64_t K, const gemm_options_t* opt, int sms, int max_pairs,
              int max_quads, int max_octs, Plan* out, int b_kn = 0, bool direct_d = false) {
  gemm_options_t o;
  std::memset(&o, 0, sizeof(o));
  if (opt) o = *opt;
  if (o.path < 0 || o.path > 3 || o.bn < 0 || o.bn > 256 || (o.bn % 32) != 0 || o.kstage < 0 ||
      o.kstage == 1 || o.kstage > kMaxStages || o.max_ctas < 0 || o.group_m < 0 || o.inject < 0 ||
      o.inject > 2 || o.katoms < 0 || o.katoms > 2 || o.acc_f16 < 0 || o.acc_f16 > 1 ||
      o.b_resident < 0 || o.b_resident > 2 || o.pdl < 0 || o.pdl > 1 || o.wide < 0 ||
      o.wide > 2 || o.small_m < 0 || o.small_m > 2 || o.split_k < 0 || o.split_k > 2 ||
      o.check < 0 || o.check > 1 || o.multicast < 0 || o.multicast > 2 ||
      (o.epi_warps != 0 && o.epi_warps != 4 && o.epi_warps != 8))
    return GEMM_ERR_INVALID_VALUE;
  if (o.path == GEMM_PATH_SKINNY && M > kBM) return GEMM_ERR_INVALID_VALUE;
  if (max_pairs < 1) max_pairs = std::max(1, sms / 2);
  if (max_quads < 1) max_quads = std::max(1, sms / 4);
  if (max_octs < 1) max_octs = std::max(1, sms / 8);

  // Candidates: (path, bn, tiles per unit).  Cost = waves of units x
  // k-blocks x per-k-block cost; ties go to the pair path, then to wide
  // units, then to the wider tile (less L2 traffic).  Wide pair units (two
  // adjacent n-tiles sharing each A slice) are candidates only for long k
  // loops, where the ring's lookahead, not the per-unit drain, limits the pair.
  if (o.wide == 2 && o.path != GEMM_PATH_AUTO && o.path != GEMM_PATH_PAIR)
    return GEMM_ERR_INVALID_VALUE;
  int path = 0, bn = 0, nt = 1;
  double best = 0;
  for (int cp = 3; cp >= 1; --cp) {
    if (cp == GEMM_PATH_SKINNY) continue;
    int kind = cp;
    if (o.path != GEMM_PATH_AUTO || o.wide == 2) {  // wide units exist on the pair path only
      const int want = (o.wide == 2) ? GEMM_PATH_PAIR
                                     : (o.path == GEMM_PATH_SKINNY) ? GEMM_PATH_SQUARE : o.path;
      if (kind != want) continue;
    } else if (kind == GEMM_PATH_PAIR && (M <= kBM || K <= 1024)) {
      // M <= 128: a pair tile would be at least half empty.  K <= 1024: the
      // k loop per tile is short, so the pair's per-tile costs (2-CTA
      // handshakes, twice the TMEM drained per tile) outweigh its lower
      // operand traffic per k-block (measured: 256^3, 1024^3 and 81920x256x256
      // all faster on single-CTA tiles).
      continue;
    }
    for (int cand = 256; cand >= 32; cand -= 32) {
      if (o.bn && cand != o.bn) continue;
      // resident B: each CTA keeps one n-block, so few n-blocks, and at
      // least one CTA for each of them
      if (o.b_resident == 2 && ((N + cand - 1) / cand > kMaxResidentN ||
                                (o.max_ctas && (N + cand - 1) / cand > o.max_ctas)))
        continue;
      // a K x N B is loaded in 64-column boxes: each CTA's share of BN must be whole boxes
      if (b_kn && cand % (kind == GEMM_PATH_PAIR ? 128 : 64) != 0) continue;
      const int bm = (kind == GEMM_PATH_PAIR) ? 2 * kBM : kBM;
      const int64_t cand_n = (N + cand - 1) / cand;
      int64_t slots = (kind == GEMM_PATH_PAIR) ? max_pairs : sms;
      if (kind == GEMM_PATH_PAIR && o.max_ctas)
        slots = std::min<int64_t>(slots, std::max(1, o.max_ctas / 2));
      for (int cnt = 2; cnt >= 1; --cnt) {
        if (cnt == 2 && (kind != GEMM_PATH_PAIR || o.wide == 1 ||
                         (o.wide == 0 && (cand_n < 2 || K < kWideMinK))))
          continue;
        if (cnt == 1 && kind == GEMM_PATH_PAIR && o.wide == 2) continue;
        const int64_t units = ((M + bm - 1) / bm) * ((cand_n + cnt - 1) / cnt);
        const int64_t waves = (units + slots - 1) / slots;
        const double cost = static_cast<double>(waves) *
                            static_cast<double>((K + kBK - 1) / kBK) *
                            kblock_cost(cnt * cand, stage_bytes_for(kind, cand, 1, cnt),
                                        kind == GEMM_PATH_PAIR ? 4 * cnt : 0);
        if (bn == 0 || cost < best * (1.0 - 1e-9)) {
          best = cost;
          bn = cand;
          path = kind;
          nt = cnt;
        }
      }
    }
  }
  if (bn == 0) return GEMM_ERR_INVALID_VALUE;
  if (path == GEMM_PATH_SQUARE && M <= kBM && o.path != GEMM_PATH_SQUARE) path = GEMM_PATH_SKINNY;

  // Split K over a CTA pair: for short k loops whose 128 x bn tiles fit in
  // one wave of pairs, each CTA of a pair takes half the k-blocks and the two
  // exchange fp32 partials through distributed shared memory.  bn is the
  // narrowest multiple of 64 (each CTA keeps half the columns, whole 32-column
  // chunks) whose tiles fit the co-resident pairs; the ring must also hold the
  // exchange once the MMAs are done.  Chosen by itself for single-CTA plans of
  // one wave with 256 <= K <= 1024 (measured: 1024^3 and 256^3).
  const int64_t tiles_1 = ((M + kBM - 1) / kBM) * ((N + bn - 1) / bn);  // the unsplit plan's
  int split_bn = 0, split_katoms = 0, split_stages = 0;
  uint32_t split_stage_bytes = 0;
  {
    const bool kind_ok = !b_kn && !o.acc_f16 && !direct_d && o.b_resident != 2 && o.wide != 2 &&
                         o.small_m != 2 && (o.path == GEMM_PATH_AUTO || o.path == GEMM_PATH_SQUARE) &&
                         (o.epi_warps == 0 || o.epi_warps == kSplitEpiWarps);
    int64_t pair_cap = max_pairs;
    if (o.max_ctas) pair_cap = std::min<int64_t>(pair_cap, o.max_ctas / 2);
    for (int cand = 64; kind_ok && cand <= 256 && !split_bn; cand += 64) {
      if (o.bn && cand != o.bn) continue;
      const int64_t t = ((M + kBM - 1) / kBM) * ((N + cand - 1) / cand);
      if (t > pair_cap) continue;
      // K slices per stage: 2 when the ring still gets 3 stages, as elsewhere
      int ka = 0, fit = 0;
      uint32_t sb = 0;
      for (int k2 : {2, 1}) {
        if (ka || (o.katoms && k2 != o.katoms)) continue;
        const uint32_t b = static_cast<uint32_t>(k2) * (kABytes + static_cast<uint32_t>(cand) * 128u);
        int f = 1;
        while (f + 1 <= kMaxStages &&
               SplitLayout::make(f + 1, b, cand).total + 1024 <= static_cast<uint32_t>(kMaxDynSmem))
          ++f;
        if (k2 == 2 && !o.katoms && f < 3) continue;
        ka = k2;
        fit = f;
        sb = b;
      }
      // this is the tile width; the plan stands or falls with it
      if (!ka || (K + kBK * ka - 1) / (kBK * ka) < 2 ||  // a k-block for each CTA at least
          fit < 2 || fit * sb < splitk_ring_reuse_bytes(cand))
        break;
      split_bn = cand;
      split_katoms = ka;
      split_stages = fit;
      split_stage_bytes = sb;
    }
  }
  if (o.split_k == 2 && !split_bn) return GEMM_ERR_INVALID_VALUE;
  const bool split_k =
      split_bn && (o.split_k == 2 ||
                   (o.split_k == 0 && o.path == GEMM_PATH_AUTO && path == GEMM_PATH_SQUARE &&
                    o.b_resident == 0 && M > kBM && K >= 256 && K <= 1024 && tiles_1 <= sms));
  if (split_k) {
    bn = split_bn;
    path = GEMM_PATH_SQUARE;
    nt = 1;
    if (o.kstage) {  // a forced ring depth must fit this kernel's plan
      if (o.kstage > split_stages ||
          static_cast<uint32_t>(o.kstage) * split_stage_bytes < splitk_ring_reuse_bytes(bn))
        return GEMM_ERR_INVALID_VALUE;
      split_stages = o.kstage;
    }
  }

  const int bm = (path == GEMM_PATH_PAIR) ? 2 * kBM : kBM;
  const int64_t num_m = (M + bm - 1) / bm;
  const int64_t num_n = (N + bn - 1) / bn;
  const int64_t tiles = num_m * num_n;
  if (tiles > INT_MAX) return GEMM_ERR_INVALID_VALUE;
  // Split K with multicast operands: the cluster also holds the next n-tile
  // and/or m-tile, and the CTAs of a k-half that share a block of A (B) each
  // fetch half of it for both.  Every cluster must be resident at once (one
  // wave).  Chosen by itself only with partners on both sides (8 CTAs, A and
  // B both halved): 256^3 3.99 -> 3.85 us, 512^3 even; 1024^3 on 4-CTA
  // clusters (all that fit at once there) was 6.77 -> 6.85 us, same box.
  // With multicast = 2 a 4-CTA cluster is taken when 8 do not fit.
  int mc_n = 1, mc_m = 1;
  if (o.multicast == 2 && (!split_k || o.check)) return GEMM_ERR_INVALID_VALUE;
  if (split_k && o.multicast != 1 && !o.check) {
    const auto fits = [&](int cn, int cm) {
      const int size = 2 * cn * cm;
      int64_t cap = size == 8 ? max_octs : size == 4 ? max_quads : max_pairs;
      if (o.max_ctas) cap = std::min<int64_t>(cap, o.max_ctas / size);
      return ((num_m + cm - 1) / cm) * ((num_n + cn - 1) / cn) <= cap;
    };
    const int cn = num_n >= 2 ? 2 : 1, cm = num_m >= 2 ? 2 : 1;
    if (fits(cn, cm) && (o.multicast == 2 || cn * cm == 4)) {
      mc_n = cn;
      mc_m = cm;
    } else if (o.multicast == 2 && cn == 2 && fits(2, 1)) {
      mc_n = 2;
    } else if (o.multicast == 2 && cm == 2 && fits(1, 2)) {
      mc_m = 2;
    }
    if (o.multicast == 2 && mc_n * mc_m == 1) return GEMM_ERR_INVALID_VALUE;
  }
  const int64_t packed_m = (num_m + mc_m - 1) / mc_m, packed_n = (num_n + mc_n - 1) / mc_n;
  // Wide pair units: two adjacent n-tiles per unit share each A slice, so a
  // one-slice stage feeds twice the MMA work and the ring gets deeper (more
  // lookahead against DRAM latency) in the same shared memory.
  const bool wide = nt == 2;
  const int64_t units_n = (num_n + nt - 1) / nt;
  const int64_t units = num_m * units_n;
  // Eight epilogue warps drain a tile twice as fast; they pay off when the k
  // loop per tile is short (the epilogue is then the critical path), four
  // are enough -- and leave the MMA and producer warps their issue slots --
  // when it is long.
  // A wide unit releases each accumulator as soon as its chunks are in
  // registers; eight warps hold all of a quadrant's chunks at once.
  int epi_warps = o.epi_warps ? o.epi_warps : ((K <= 1024 || wide) ? 8 : 4);
  // Two 64-wide K slices per stage halve the issuing threads' per-byte
  // barrier/commit work (measured: +12 % at 8192^3); used whenever the ring
  // still gets at least 3 stages.
  int katoms = o.katoms ? o.katoms
                        : (stages_that_fit(stage_bytes_for(path, bn, 2, nt), epi_warps) >= 3 ? 2
                                                                                         : 1);
  // Resident B: a single-CTA kernel whose tiles all share one n-block holds
  // that n-block's B (BN x K) in shared memory and streams only A -- a third
  // of the bytes per 128 x 256 tile when K = N = 256.  With a few n-blocks,
  // tiles are ordered n-fastest (group_m = 1) over a grid that is a multiple
  // of num_n, so CTA c only ever meets n-block c % num_n.  Used when each CTA
  // has at least two tiles, the ring still gets 3 stages of A, and it keeps
  // more of A in flight than the streamed plan's ring would (A streams from
  // DRAM; B in shared memory takes room from A's ring) -- or as much, with
  // several n-blocks (with one, streamed B is an L2 hit for every tile).
  // Chosen by itself with the streamed plan's epilogue warps only (four
  // warps' deeper ring did not pay: 81920x256x256 18.31 against 18.25 us with
  // eight).  Measured, same box, resident against streamed: 81920x1024x128
  // 32.8 / 34.3 us (128 against 64 KiB of A in flight), 65536x128x512 20.5 /
  // 17.3 (64 against 96), 81920x512x256 27.1 / 27.4 (equal, 2 n-blocks),
  // 81920x256x256 18.25 / 18.12 (equal, 1 n-block).
  const uint32_t streamed_a_in_flight =
      static_cast<uint32_t>(stages_that_fit(stage_bytes_for(path, bn, katoms, nt), epi_warps)) *
      katoms * kABytes;
  bool b_resident = false;
  uint32_t bres_bytes = 0;
  int64_t ctas_1 = std::min<int64_t>(tiles, sms);
  if (o.max_ctas) ctas_1 = std::min<int64_t>(ctas_1, o.max_ctas);
  const int64_t ctas_res = ctas_1 / num_n * num_n;
  const bool res_possible = !split_k && path != GEMM_PATH_PAIR && !b_kn && num_n <= kMaxResidentN &&
                            ctas_res >= 1 && (num_n == 1 || o.group_m <= 1);
  if (o.b_resident == 2 && !res_possible) return GEMM_ERR_INVALID_VALUE;
  if (res_possible && (o.b_resident == 2 || (o.b_resident == 0 && tiles >= 2 * sms))) {
    const int min_stages = (o.b_resident == 2) ? 2 : 3;
    for (int ew : {epi_warps, 4}) {
      if (b_resident || (o.epi_warps && ew != o.epi_warps)) continue;
      for (int ka : {2, 1}) {
        if (b_resident || (o.katoms && ka != o.katoms)) continue;
        const int nk = static_cast<int>((K + kBK * ka - 1) / (kBK * ka));
        const uint32_t bres = static_cast<uint32_t>(nk) * ka * b_atom_bytes_for(path, bn);
        if (bres > static_cast<uint32_t>(kMaxDynSmem)) continue;
        const int f = stages_that_fit(static_cast<uint32_t>(ka) * kABytes, ew, bres, nk);
        const uint32_t a_in_flight = static_cast<uint32_t>(f) * ka * kABytes;
        const bool deeper = a_in_flight > streamed_a_in_flight ||
                            (a_in_flight == streamed_a_in_flight && num_n >= 2);
        if (f >= min_stages && (ka == 1 || o.katoms || f >= 3) &&
            (o.b_resident == 2 || (deeper && ew == epi_warps))) {
          b_resident = true;
          bres_bytes = bres;
          epi_warps = ew;
          katoms = ka;
        }
      }
    }
    if (o.b_resident == 2 && !b_resident) return GEMM_ERR_INVALID_VALUE;
  }
  // The small-M kernel on the skinny path: one tile per CTA (so at most one
  // n-tile per SM), its epilogue staged in the ring once the tile's MMAs are
  // done, so the whole shared memory holds the ring.  It has four epilogue
  // warps.
  int64_t ctas_cap = sms;
  if (o.max_ctas) ctas_cap = std::min<int64_t>(ctas_cap, o.max_ctas);
  const bool small_possible = !split_k && path == GEMM_PATH_SKINNY && !b_resident &&
                              num_n <= ctas_cap &&
                              (o.epi_warps == 0 || o.epi_warps == kSkinnyEpiWarps);
  if (o.small_m == 2 && !small_possible) return GEMM_ERR_INVALID_VALUE;
  const bool small_m = small_possible && o.small_m != 1;
  if (small_m) {
    epi_warps = kSkinnyEpiWarps;
    katoms = o.katoms ? o.katoms : kSkinnyKatoms;
  }
  if (split_k) {
    epi_warps = kSplitEpiWarps;
    katoms = split_katoms;
  }
  const int64_t num_k = (K + kBK * katoms - 1) / (kBK * katoms);
  uint32_t stage_bytes = b_resident ? static_cast<uint32_t>(katoms) * kABytes
                                    : stage_bytes_for(path, bn, katoms, nt);
  int stages = 0;
  uint32_t smem_total = 0;
  if (split_k) {
    stage_bytes = split_stage_bytes;
    stages = split_stages;
    smem_total = SplitLayout::make(stages, stage_bytes, bn).total + 1024;
  } else if (small_m) {
    const auto small_total = [&](int sc) { return SkinnyLayout::make(sc, stage_bytes).total + 1024; };
    int fit = 1;
    while (fit + 1 <= kMaxStages && small_total(fit + 1) <= static_cast<uint32_t>(kMaxDynSmem))
      ++fit;
    if (fit < 2) return GEMM_ERR_INVALID_VALUE;
    stages = o.kstage ? o.kstage : fit;
    if (stages > fit) return GEMM_ERR_INVALID_VALUE;
    smem_total = small_total(stages);
  } else {
    const int bres_bars = b_resident ? static_cast<int>(num_k) : 1;  // one per k-block of B
    const int fit = stages_that_fit(stage_bytes, epi_warps, bres_bytes, bres_bars);
    if (fit < 2) return GEMM_ERR_INVALID_VALUE;
    stages = o.kstage ? o.kstage : fit;
    if (stages > fit) return GEMM_ERR_INVALID_VALUE;
    smem_total = SmemLayout::make(stages, stage_bytes, epi_warps, bres_bytes, bres_bars).total + 1024;
  }
  // Balanced grids: as many CTAs (pairs) as the fewest waves need, so every
  // one gets the same number of tiles (units) to one.  An HBM-bound stream
  // then has no partial last wave (tall 81920 x 256 x 256: 640 tiles as 5 on
  // each of 128 CTAs instead of 4 or 5 on 152, 18.6 against 18.9 us back to
  // back, the same 20.8 us launched alone); on the tensor-bound pair path the
  // idle SMs leave the busy ones more of the power cap (4096^3: 128 units as
  // 2 on 64 pairs, 85.1 against 85.5 us).
  const auto balanced = [](int64_t work, int64_t slots, int64_t multiple) {
    const int64_t waves = (work + slots - 1) / slots;
    const int64_t even = (work + waves - 1) / waves;
    return std::min<int64_t>(slots, (even + multiple - 1) / multiple * multiple);
  };
  int ctas;
  if (split_k) {
    ctas = static_cast<int>(2 * mc_n * mc_m * packed_m * packed_n);  // a CTA pair for each tile
  } else if (small_m) {
    ctas = static_cast<int>(tiles);  // one tile each
  } else if (path == GEMM_PATH_PAIR) {
    int64_t pairs = std::min<int64_t>(units, max_pairs);
    if (o.max_ctas) pairs = std::min<int64_t>(pairs, std::max(1, o.max_ctas / 2));
    ctas = static_cast<int>(2 * balanced(units, pairs, 1));
  } else if (b_resident) {
    ctas = static_cast<int>(balanced(tiles, ctas_res, num_n));  // a multiple of num_n
  } else {
    ctas = static_cast<int>(balanced(tiles, ctas_1, 1));
  }
  const int group_m =
      o.group_m ? o.group_m
                : (path == GEMM_PATH_PAIR ? (wide ? 16 : 8) : (b_resident && num_n > 1 ? 1 : 16));

  Plan pl;
  std::memset(&pl, 0, sizeof(pl));
  pl.cfg.path = path;
  pl.cfg.bm = bm;
  pl.cfg.bn = bn;
  pl.cfg.bk = kBK * katoms;
  pl.cfg.katoms = katoms;
  pl.cfg.epi_warps = epi_warps;
  pl.cfg.kstage = stages;
  pl.cfg.ctas = ctas;
  pl.cfg.group_m = group_m;
  pl.cfg.tiles = static_cast<int>(tiles);
  pl.cfg.smem_bytes = static_cast<int>(smem_total);  // includes 1 KiB of alignment slack
  // two accumulators (consecutive tiles overlap), one in the small-M kernel
  pl.cfg.tmem_cols = static_cast<int>(pow2_at_least((small_m || split_k) ? bn : 2u * bn));
  pl.cfg.b_resident = b_resident ? 1 : 0;
  pl.cfg.pdl = o.pdl ? 0 : 1;
  pl.cfg.wide = wide ? 1 : 0;
  pl.cfg.small_m = small_m ? 1 : 0;
  pl.cfg.split_k = split_k ? 1 : 0;
  pl.cfg.cluster = split_k ? 2 * mc_n * mc_m : (path == GEMM_PATH_PAIR ? 2 : 1);
  pl.mc_n = mc_n;
  pl.mc_m = mc_m;

  GemmParams& p = pl.p;
  p.M = static_cast<int32_t>(M);
  p.N = static_cast<int32_t>(N);
  p.K = static_cast<int32_t>(K);
  p.bn = bn;
  p.stages = stages;
  // the kernel schedules units: with wide units, pairs of adjacent n-tiles;
  // with split K, clusters of mc_m x mc_n tiles
  p.num_m_blocks = static_cast<int32_t>(split_k ? packed_m : num_m);
  p.num_n_blocks = static_cast<int32_t>(split_k ? packed_n : units_n);
  p.num_k_blocks = static_cast<int32_t>(num_k);
  p.num_tiles = static_cast<int32_t>(split_k ? packed_m * packed_n : units);
  p.group_m = group_m;
  p.idesc = make_idesc(bm, bn) | (b_kn ? (1u << 16) : 0u);  // bit 16: B is MN-major
  if (o.acc_f16) p.idesc &= ~(3u << 4);                      // bits 4-5: D format F16
  p.acc_f16 = o.acc_f16;
  p.b_kn = b_kn;
  p.tmem_cols = static_cast<uint32_t>(pl.cfg.tmem_cols);
  p.stage_bytes = stage_bytes;
  p.b_atom_bytes = b_atom_bytes_for(path, bn);
  p.katoms = katoms;
  p.epi_warps = epi_warps;
  p.b_resident = b_resident ? 1 : 0;
  p.bres_bytes = bres_bytes;
  // One m-block: every tile reads the same rows of A (keep them in L2, stream
  // B through it once) and the k loops are rotated across tiles.
  p.l2_hints = (num_m == 1) ? 3u : 0u;
  p.k_rotate = (num_m == 1 && num_n > 1) ? 1 : 0;
  p.timeout_ns = o.timeout_ns ? o.timeout_ns : kDefaultTimeoutNs;
  p.inject = o.inject;
  p.check = o.check;
  *out = pl;
  return GEMM_OK;
}

int encode_2d(CUtensorMap* map, const View& v, uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swz) {
  const cuuint64_t dims[2] = {v.cols, v.rows};
  const cuuint64_t strides[1] = {v.ld * 2};  // bytes between rows
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(v.ptr),
                              dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GEMM_OK : GEMM_ERR_INVALID_VALUE;
}

template <typename Kernel>
bool grant_smem(Kernel k) {
  return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem) ==
         cudaSuccess;
}

// Every kernel instantiation: epilogue warps (4, 8) x resident B x direct D
// store for the single-CTA kernel, epilogue warps x direct D x tiles per unit
// x scaled epilogue for the pair.
template <bool kDirectD>
bool grant_all(bool ok) {
  return ok && grant_smem(gemm_tn_f16_skinny<kDirectD>) && grant_smem(gemm_tn_f16_splitk<>) &&
         grant_smem(gemm_tn_f16_splitk<false, 2, 1>) && grant_smem(gemm_tn_f16_splitk<false, 1, 2>) &&
         grant_smem(gemm_tn_f16_splitk<false, 2, 2>) &&
         grant_smem(gemm_tn_f16_persistent<4, false, kDirectD>) &&
         grant_smem(gemm_tn_f16_persistent<8, false, kDirectD>) &&
         grant_smem(gemm_tn_f16_persistent<4, true, kDirectD>) &&
         grant_smem(gemm_tn_f16_persistent<8, true, kDirectD>) &&
         grant_smem(gemm_tn_f16_pair<4, kDirectD, 1, false>) &&
         grant_smem(gemm_tn_f16_pair<8, kDirectD, 1, false>) &&
         grant_smem(gemm_tn_f16_pair<4, kDirectD, 2, false>) &&
         grant_smem(gemm_tn_f16_pair<8, kDirectD, 2, false>) &&
         grant_smem(gemm_tn_f16_pair<4, kDirectD, 1, true>) &&
         grant_smem(gemm_tn_f16_pair<8, kDirectD, 1, true>) &&
         grant_smem(gemm_tn_f16_pair<4, kDirectD, 2, true>) &&
         grant_smem(gemm_tn_f16_pair<8, kDirectD, 2, true>);
}

// The invariant-checking instantiations: the plain forms (D stored by TMA,
// no scaled epilogue) of every kernel.
bool grant_checked() {
  return grant_smem(gemm_tn_f16_skinny<false, true>) && grant_smem(gemm_tn_f16_splitk<true>) &&
         grant_smem(gemm_tn_f16_persistent<4, false, false, true>) &&
         grant_smem(gemm_tn_f16_persistent<8, false, false, true>) &&
         grant_smem(gemm_tn_f16_persistent<4, true, false, true>) &&
         grant_smem(gemm_tn_f16_persistent<8, true, false, true>) &&
         grant_smem(gemm_tn_f16_pair<4, false, 1, false, true>) &&
         grant_smem(gemm_tn_f16_pair<8, false, 1, false, true>) &&
         grant_smem(gemm_tn_f16_pair<4, false, 2, false, true>) &&
         grant_smem(gemm_tn_f16_pair<8, false, 2, false, true>);
}

cudaError_t launch_checked(const cudaLaunchConfig_t& cfg, bool pair, bool wide, bool resident,
                           bool small, bool split, int epi_warps, const CUtensorMap& a,
                           const CUtensorMap& b, const CUtensorMap& d, const GemmParams& p) {
  if (split) return cudaLaunchKernelEx(&cfg, gemm_tn_f16_splitk<true>, a, b, d, p);
  if (small) return cudaLaunchKernelEx(&cfg, gemm_tn_f16_skinny<false, true>, a, b, d, p);
  if (pair) {
    if (wide)
      return epi_warps == 8
                 ? cudaLaunchKernelEx(&cfg, gemm_tn_f16_pair<8, false, 2, false, true>, a, b, d, p)
                 : cudaLaunchKernelEx(&cfg, gemm_tn_f16_pair<4, false, 2, false, true>, a, b, d, p);
    return epi_warps == 8
               ? cudaLaunchKernelEx(&cfg, gemm_tn_f16_pair<8, false, 1, false, true>, a, b, d, p)
               : cudaLaunchKernelEx(&cfg, gemm_tn_f16_pair<4, false, 1, false, true>, a, b, d, p);
  }
  if (resident)
    return epi_warps == 8
               ? cudaLaunchKernelEx(&cfg, gemm_tn_f16_persistent<8, true, false, true>, a, b, d, p)
               : cudaLaunchKernelEx(&cfg, gemm_tn_f16_persistent<4, true, false, true>, a, b, d, p);
  return epi_warps == 8
             ? cudaLaunchKernelEx(&cfg, gemm_tn_f16_persistent<8, false, false, true>, a, b, d, p)
             : cudaLaunchKernelEx(&cfg, gemm_tn_f16_persistent<4, false, false, true>, a, b, d, p);
}

cudaError_t launch_splitk(const cudaLaunchConfig_t& cfg, int mc_n, int mc_m, const CUtensorMap& a,
                          const CUtensorMap& b, const CUtensorMap& d, const GemmParams& p) {
  if (mc_n == 2 && mc_m == 2)
    return cudaLaunchKernelEx(&cfg, gemm_tn_f16_splitk<false, 2, 2>, a, b, d, p);
  if (mc_n == 2) return cudaLaunchKernelEx(&cfg, gemm_tn_f16_splitk<false, 2, 1>, a, b, d, p);
  if (mc_m == 2) return cudaLaunchKernelEx(&cfg, gemm_tn_f16_splitk<false, 1, 2>, a, b, d, p);
  return cudaLaunchKernelEx(&cfg, gemm_tn_f16_splitk<>, a, b, d, p);
}

template <bool kDirectD, int kNT, bool kScaled>
cudaError_t launch_pair_as(const cudaLaunchConfig_t& cfg, int epi_warps, const CUtensorMap& a,
                           const CUtensorMap& b, const CUtensorMap& d, const GemmParams& p) {
  return epi_warps == 8
             ? cudaLaunchKernelEx(&cfg, gemm_tn_f16_pair<8, kDirectD, kNT, kScaled>, a, b, d, p)
             : cudaLaunchKernelEx(&cfg, gemm_tn_f16_pair<4, kDirectD, kNT, kScaled>, a, b, d, p);
}

template <bool kDirectD, int kNT>
cudaError_t launch_pair(const cudaLaunchConfig_t& cfg, int epi_warps, const CUtensorMap& a,
                        const CUtensorMap& b, const CUtensorMap& d, const GemmParams& p) {
  return p.scaled ? launch_pair_as<kDirectD, kNT, true>(cfg, epi_warps, a, b, d, p)
                  : launch_pair_as<kDirectD, kNT, false>(cfg, epi_warps, a, b, d, p);
}

template <bool kDirectD>
cudaError_t launch_kernel(const cudaLaunchConfig_t& cfg, bool pair, bool wide, bool resident,
                          bool small, int epi_warps, const CUtensorMap& a, const CUtensorMap& b,
                          const CUtensorMap& d, const GemmParams& p) {
  if (small) return cudaLaunchKernelEx(&cfg, gemm_tn_f16_skinny<kDirectD>, a, b, d, p);
  if (pair)
    return wide ? launch_pair<kDirectD, 2>(cfg, epi_warps, a, b, d, p)
                : launch_pair<kDirectD, 1>(cfg, epi_warps, a, b, d, p);
  if (resident)
    return epi_warps == 8
               ? cudaLaunchKernelEx(&cfg, gemm_tn_f16_persistent<8, true, kDirectD>, a, b, d, p)
               : cudaLaunchKernelEx(&cfg, gemm_tn_f16_persistent<4, true, kDirectD>, a, b, d, p);
  return epi_warps == 8
             ? cudaLaunchKernelEx(&cfg, gemm_tn_f16_persistent<8, false, kDirectD>, a, b, d, p)
             : cudaLaunchKernelEx(&cfg, gemm_tn_f16_persistent<4, false, kDirectD>, a, b, d, p);
}

// Grant every kernel the full dynamic shared memory and find how many
// 2-CTA clusters can be resident at once (the pair path's persistent grid).
int prepare_device(DeviceState* st) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (st->smem_attr == kMaxDynSmem && st->pair_smem_attr == kMaxDynSmem && st->max_pairs > 0)
    return GEMM_OK;
  if (!grant_all<true>(grant_all<false>(true)) || !grant_checked()) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  st->smem_attr = st->pair_smem_attr = kMaxDynSmem;
  // co-resident 2-CTA clusters, for the larger of the two block sizes
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * (st->sm_count / 2), 1, 1);
  cfg.blockDim = dim3(threads_for(8), 1, 1);
  cfg.dynamicSmemBytes = kMaxDynSmem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tn_f16_pair<8, false, 1, false>, &cfg) !=
          cudaSuccess ||
      clusters < 1) {
    cudaGetLastError();
    clusters = st->sm_count / 2;
  }
  st->max_pairs = std::min(clusters, st->sm_count / 2);
  // co-resident 4- and 8-CTA clusters of the split-K kernel
  cfg.blockDim = dim3(kSplitThreads, 1, 1);
  attr[0].val.clusterDim.x = 4;
  cfg.gridDim = dim3(4 * (st->sm_count / 4), 1, 1);
  if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tn_f16_splitk<false, 2, 1>, &cfg) !=
          cudaSuccess ||
      clusters < 0) {
    cudaGetLastError();
    clusters = 0;  // multicast split K then uses 2-CTA clusters only
  }
  st->max_quads = std::min(clusters, st->sm_count / 4);
  attr[0].val.clusterDim.x = 8;
  cfg.gridDim = dim3(8 * (st->sm_count / 8), 1, 1);
  if (cudaOccupancyMaxActiveClusters(&clusters, gemm_tn_f16_splitk<false, 2, 2>, &cfg) !=
          cudaSuccess ||
      clusters < 0) {
    cudaGetLastError();
    clusters = 0;
  }
  st->max_octs = std::min(clusters, st->sm_count / 8);
  return GEMM_OK;
}

// Device error words are per stream: the legacy default stream has word 0,
// the first 63 other streams a process uses get one each, and later streams
// share the remaining words by a hash of their handle.
std::mutex g_slot_mu;
uintptr_t g_slot_stream[kErrorSlots];
int g_slots_used = 1;

int error_slot(cudaStream_t s) {
  const uintptr_t h = reinterpret_cast<uintptr_t>(s);
  if (h == 0) return 0;
  std::lock_guard<std::mutex> lk(g_slot_mu);
  for (int i = 1; i < g_slots_used; ++i)
    if (g_slot_stream[i] == h) return i;
  if (g_slots_used < kErrorSlots) {
    g_slot_stream[g_slots_used] = h;
    return g_slots_used++;
  }
  return 1 + static_cast<int>((h >> 4) % static_cast<uintptr_t>(kErrorSlots - 1));
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

// D = beta * C elementwise: the scaled form with an empty k range.
__global__ void scale_c_kernel(uint16_t* D, const uint16_t* C, float beta, int64_t n) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float c = __half2float(__ushort_as_half(C[i]));
    D[i] = __half_as_ushort(__float2half_rn(beta * c));
  }
}

int check_scaled(const void* D, const Scaled& sc, int64_t M, int64_t N) {
  if (sc.b_kn != 0 && sc.b_kn != 1) return GEMM_ERR_INVALID_VALUE;
  if (!std::isfinite(sc.alpha) || !std::isfinite(sc.beta)) return GEMM_ERR_INVALID_VALUE;
  if (sc.beta == 0.0f || M == 0 || N == 0) return GEMM_OK;  // C is not read
  if (!sc.C) return GEMM_ERR_INVALID_VALUE;
  if (reinterpret_cast<uintptr_t>(sc.C) & 15) return GEMM_ERR_MISALIGNED;
  const uint64_t bytes = static_cast<uint64_t>(M) * N * 2;
  // C may be D exactly (in place: each element is read before the same CTA
  // writes it); any other overlap would read partly written values.
  if (sc.C != D && overlaps(sc.C, bytes, D, bytes)) return GEMM_ERR_INVALID_VALUE;
  return GEMM_OK;
}

}  // namespace

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

int device_sm_count(const DeviceState* st) { return st->sm_count; }

bool overlaps(const void* a, uint64_t abytes, const void* b, uint64_t bbytes) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bbytes && y < x + abytes;
}

int write_empty_sum(void* D, const void* C, float beta, int64_t n, int sm_count,
                    cudaStream_t stream) {
  if (C && beta != 0.0f) {
    const int blocks = static_cast<int>(std::min<int64_t>((n + 255) / 256, 8 * sm_count));
    scale_c_kernel<<<blocks, 256, 0, stream>>>(static_cast<uint16_t*>(D),
                                               static_cast<const uint16_t*>(C), beta, n);
    return cudaGetLastError() == cudaSuccess ? GEMM_OK : GEMM_ERR_LAUNCH;
  }
  if (cudaMemsetAsync(D, 0, static_cast<size_t>(n) * 2, stream) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  return GEMM_OK;
}

int launch_gemm(int64_t M, int64_t N, int64_t K, const View& a, const View& b, const View& d,
                int b_kn, const Scaled* sc, int64_t ldc, const gemm_options_t* opt,
                DeviceState* st, cudaStream_t stream, uint16_t* d_direct, int64_t ldd) {
  int rc;
  if ((rc = prepare_device(st)) != GEMM_OK) return rc;
  Plan pl;
  rc = make_plan(M, N, K, opt, st->sm_count, st->max_pairs, st->max_quads, st->max_octs, &pl, b_kn,
                 d_direct != nullptr);
  if (rc != GEMM_OK) return rc;
  if ((rc = get_encoder()) != GEMM_OK) return rc;
  pl.p.ldc = ldc;
  pl.p.err_slot = error_slot(stream);
  if (sc && !(sc->alpha == 1.0f && sc->beta == 0.0f)) {
    pl.p.scaled = 1;
    pl.p.alpha = sc->alpha;
    pl.p.beta = sc->beta;
    pl.p.C = static_cast<const uint16_t*>(sc->C);
  }

  const bool pair = pl.cfg.path == GEMM_PATH_PAIR;
  // a pair CTA loads half of B; a multicast split-K CTA half of the block it shares
  const uint32_t b_box_rows = (pair || pl.mc_m == 2) ? pl.cfg.bn / 2 : pl.cfg.bn;
  const uint32_t a_box_rows = pl.mc_n == 2 ? kBM / 2 : kBM;
  CUtensorMap tmA, tmB, tmD;
  const int b_rc = b_kn ? encode_2d(&tmB, b, 64, kBK, CU_TENSOR_MAP_SWIZZLE_128B)
                        : encode_2d(&tmB, b, kBK, b_box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
  if (encode_2d(&tmA, a, kBK, a_box_rows, CU_TENSOR_MAP_SWIZZLE_128B) != GEMM_OK ||
      b_rc != GEMM_OK)
    return GEMM_ERR_INVALID_VALUE;
  if (d_direct) {  // plain stores to D; the kernel never reads tmD
    pl.p.D = d_direct;
    pl.p.ldd = ldd;
    tmD = tmA;
  } else if (encode_2d(&tmD, d, kEpiCols, 32, CU_TENSOR_MAP_SWIZZLE_64B) != GEMM_OK) {
    return GEMM_ERR_INVALID_VALUE;
  }

  // Programmatic dependent launch: the kernel's set-up (barriers, TMEM)
  // may overlap the end of the previous kernel in the stream; the kernel
  // waits for that kernel before its first global-memory access.
  cudaLaunchConfig_t cfg;
  std::memset(&cfg, 0, sizeof(cfg));
  cudaLaunchAttribute attr[2];
  int nattr = 0;
  if (pl.cfg.pdl) {
    attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[nattr].val.programmaticStreamSerializationAllowed = 1;
    ++nattr;
  }
  if (pl.cfg.cluster > 1) {
    attr[nattr].id = cudaLaunchAttributeClusterDimension;
    attr[nattr].val.clusterDim.x = static_cast<unsigned>(pl.cfg.cluster);
    attr[nattr].val.clusterDim.y = 1;
    attr[nattr].val.clusterDim.z = 1;
    ++nattr;
  }
  cfg.gridDim = dim3(pl.cfg.ctas, 1, 1);
  cfg.blockDim = dim3(pl.cfg.small_m ? kSkinnyThreads : threads_for(pl.cfg.epi_warps), 1, 1);
  cfg.dynamicSmemBytes = pl.cfg.smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = nattr;
  const bool wide = pl.cfg.wide != 0, res = pl.p.b_resident != 0, small = pl.cfg.small_m != 0;
  // the invariant check exists for the plain forms only: D stored by TMA, no scaled epilogue
  if (pl.p.check && (d_direct || pl.p.scaled)) return GEMM_ERR_INVALID_VALUE;
  const cudaError_t e =
      pl.p.check ? launch_checked(cfg, pair, wide, res, small, pl.cfg.split_k != 0,
                                  pl.cfg.epi_warps, tmA, tmB, tmD, pl.p) :
      pl.cfg.split_k ? launch_splitk(cfg, pl.mc_n, pl.mc_m, tmA, tmB, tmD, pl.p) :
      d_direct ? launch_kernel<true>(cfg, pair, wide, res, small, pl.cfg.epi_warps, tmA, tmB, tmD,
                                     pl.p)
               : launch_kernel<false>(cfg, pair, wide, res, small, pl.cfg.epi_warps, tmA, tmB,
                                      tmD, pl.p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_LAUNCH;
  }
  if (cudaGetLastError() != cudaSuccess) return GEMM_ERR_LAUNCH;
  return GEMM_OK;
}

int check_options(const gemm_options_t* opt, int b_kn, int64_t M, int64_t N, int64_t K) {
  if (!opt) return GEMM_OK;
  Plan tmp;
  return make_plan(std::max<int64_t>(M, 1), std::max<int64_t>(N, 8), std::max<int64_t>(K, 8), opt,
                   148, 74, 37, 18, &tmp, b_kn);
}

namespace {

int run(void* D, const void* A, const void* B, int64_t M, int64_t N, int64_t K,
        const gemm_options_t* opt, cudaStream_t stream, const Scaled* sc = nullptr) {
  int rc = check_args(D, A, B, M, N, K);
  if (rc != GEMM_OK) return rc;
  const int b_kn = sc ? sc->b_kn : 0;
  if (sc && (rc = check_scaled(D, *sc, M, N)) != GEMM_OK) return rc;
  if ((rc = check_options(opt, b_kn, M, N, K)) != GEMM_OK) return rc;
  if (M == 0 || N == 0) return GEMM_OK;
  int dev = 0;
  DeviceState* st = nullptr;
  rc = current_device(&dev, &st);
  if (rc != GEMM_OK) return rc;
  if (K == 0)
    return write_empty_sum(D, sc ? sc->C : nullptr, sc ? sc->beta : 0.0f, M * N, st->sm_count,
                           stream);
  const uint64_t m = M, n = N, k = K;
  const View a{A, k, m, k};
  const View b = b_kn ? View{B, n, k, n} : View{B, k, n, k};
  const View d{D, n, m, n};
  return launch_gemm(M, N, K, a, b, d, b_kn, sc, N, opt, st, stream);
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" int gemm_tn_f16(void* D, const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                           void* stream) {
  return run(D, A, B, M, N, K, nullptr, static_cast<cudaStream_t>(stream));
}

extern "C" int gemm_f16_scaled(void* D, const void* C, const void* A, const void* B, int64_t M,
                               int64_t N, int64_t K, float alpha, float beta, int b_layout,
                               const gemm_options_t* opt, void* stream) {
  const Scaled sc{C, alpha, beta, b_layout};
  return run(D, A, B, M, N, K, opt, static_cast<cudaStream_t>(stream), &sc);
}

extern "C" int gemm_tn_f16_ex(void* D, const void* A, const void* B, int64_t M, int64_t N,
                              int64_t K, const gemm_options_t* opt, void* stream) {
  return run(D, A, B, M, N, K, opt, static_cast<cudaStream_t>(stream));
}

extern "C" int gemm_query_config(int64_t M, int64_t N, int64_t K, const gemm_options_t* opt,
                                 gemm_config_t* out) {
  if (!out || M <= 0 || N <= 0 || K <= 0 || M > INT_MAX || N > INT_MAX || K > INT_MAX)
    return GEMM_ERR_INVALID_VALUE;
  int sms = 148, pairs = 74, quads = 37, octs = 18, dev = 0;
  DeviceState* st = nullptr;
  if (current_device(&dev, &st) == GEMM_OK && prepare_device(st) == GEMM_OK) {
    sms = st->sm_count;
    pairs = st->max_pairs;
    quads = st->max_quads;
    octs = st->max_octs;
  } else {
    cudaGetLastError();
  }
  const int b_kn = opt ? opt->b_layout : 0;
  if (b_kn != 0 && b_kn != 1) return GEMM_ERR_INVALID_VALUE;
  Plan pl;
  const int rc = make_plan(M, N, K, opt, sms, pairs, quads, octs, &pl, b_kn);
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
  const size_t off = static_cast<size_t>(error_slot(s)) * sizeof(unsigned int);
  if (cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemcpyFromSymbolAsync(&word, g_gemm_error, sizeof(word), off, cudaMemcpyDeviceToHost,
                                s) != cudaSuccess ||
      cudaMemcpyToSymbolAsync(g_gemm_error, &zero, sizeof(zero), off, cudaMemcpyHostToDevice, s) !=
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
    case GEMM_ERR_INVARIANT: return "GEMM_ERR_INVARIANT";
    default: return "GEMM_ERR_UNKNOWN";
  }
}
