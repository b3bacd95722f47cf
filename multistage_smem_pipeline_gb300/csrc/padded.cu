// The padded entry point: gemm_f16_scaled for any K and N and any
// 2-byte-aligned operand.  Every operand the GEMM kernel reads whose base or
// row stride is not 16-byte aligned is first copied into a caller-owned
// workspace with rows padded to a multiple of 8 elements (+0 in the pad) and
// the GEMM runs on the aligned copies.  A D of that kind is stored by the
// kernel's epilogue with plain stores when C is not read; when C is read, C
// goes into a padded D that the GEMM updates in place and that is copied back
// afterwards.  This is the host wrapper of "CUDA 算子笔记 2" (GEMM section),
// which pads A, B and C to tile multiples before its kernel; here the pad is
// only what TMA needs.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "gemm_tn_f16.h"
#include "host.cuh"
#include "repack.cuh"

namespace gb300 {
namespace {

struct PadPlan {
  bool ok;              // false: a padded extent or the workspace size would overflow
  int64_t Kp, Np;
  bool pack_a, pack_b, pad_d;
  bool direct_d;        // pad_d and C not read: the GEMM stores D directly, no padded copy
  bool c_to_d;          // C copied into D (D aligned, C not); then C := D (in place)
  uint64_t off_a, off_b, off_d, total;
};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

uint64_t round_up(uint64_t x, uint64_t a) { return (x + a - 1) / a * a; }

// Which operands are repacked and where they go in the workspace.  The pure
// function of the arguments that both gemm_padded_workspace_bytes and
// gemm_f16_padded evaluate.
PadPlan plan_padding(const void* D, const void* C, const void* A, const void* B, int64_t M,
                     int64_t N, int64_t K, float beta, int b_kn) {
  PadPlan pp;
  std::memset(&pp, 0, sizeof(pp));
  pp.Kp = padded_cols(K);
  pp.Np = padded_cols(N);
  // the kernel's extents are int32: K and N rounded up to 8 must still fit
  pp.ok = pp.Kp <= INT_MAX && pp.Np <= INT_MAX;
  if (!pp.ok || M == 0 || N == 0 || K == 0) return pp;  // nothing reaches the GEMM kernel
  pp.pack_a = !aligned16(A) || K % 8 != 0;
  pp.pack_b = !aligned16(B) || (b_kn ? N % 8 != 0 : K % 8 != 0);
  pp.pad_d = !aligned16(D) || N % 8 != 0;
  pp.direct_d = pp.pad_d && beta == 0.0f;
  pp.c_to_d = !pp.pad_d && beta != 0.0f && !aligned16(C);
  // Each region is below 2^63 bytes (extents below 2^31); the sum of three
  // is kept below 2^63 too, or the plan is refused.
  constexpr uint64_t kRegionAlign = 256;
  constexpr uint64_t kLimit = uint64_t{1} << 63;
  uint64_t off = 0;
  const auto add = [&](uint64_t bytes) {
    const uint64_t r = round_up(bytes, kRegionAlign);
    if (r >= kLimit - off) pp.ok = false;
    else off += r;
  };
  if (pp.pack_a) {
    pp.off_a = off;
    add(static_cast<uint64_t>(M) * pp.Kp * 2);
  }
  if (pp.pack_b) {
    pp.off_b = off;
    add(b_kn ? static_cast<uint64_t>(K) * pp.Np * 2 : static_cast<uint64_t>(N) * pp.Kp * 2);
  }
  if (pp.pad_d && !pp.direct_d) {
    pp.off_d = off;
    add(static_cast<uint64_t>(M) * pp.Np * 2);
  }
  pp.total = off;
  return pp;
}

int check_padded_args(const void* D, const void* C, const void* A, const void* B, int64_t M,
                      int64_t N, int64_t K, float alpha, float beta, int b_kn) {
  if (M < 0 || N < 0 || K < 0 || M > INT_MAX || N > INT_MAX || K > INT_MAX)
    return GEMM_ERR_INVALID_VALUE;
  if (b_kn != 0 && b_kn != 1) return GEMM_ERR_INVALID_VALUE;
  if (!std::isfinite(alpha) || !std::isfinite(beta)) return GEMM_ERR_INVALID_VALUE;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!D || (K > 0 && (!A || !B)) || (beta != 0.0f && !C)) return GEMM_ERR_INVALID_VALUE;
  const auto odd = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 1) != 0; };
  if (odd(D) || (K > 0 && (odd(A) || odd(B))) || (beta != 0.0f && odd(C)))
    return GEMM_ERR_MISALIGNED;
  const uint64_t dbytes = static_cast<uint64_t>(M) * N * 2;
  if (K > 0 && (overlaps(D, dbytes, A, static_cast<uint64_t>(M) * K * 2) ||
                overlaps(D, dbytes, B, static_cast<uint64_t>(N) * K * 2)))
    return GEMM_ERR_INVALID_VALUE;
  if (beta != 0.0f && C != D && overlaps(C, dbytes, D, dbytes)) return GEMM_ERR_INVALID_VALUE;
  return GEMM_OK;
}

int run_padded(void* D, const void* C, const void* A, const void* B, int64_t M, int64_t N,
               int64_t K, float alpha, float beta, int b_kn, void* workspace,
               uint64_t workspace_bytes, const gemm_options_t* opt, cudaStream_t stream) {
  int rc = check_padded_args(D, C, A, B, M, N, K, alpha, beta, b_kn);
  if (rc != GEMM_OK) return rc;
  if ((rc = check_options(opt, b_kn, M, N, K)) != GEMM_OK) return rc;
  if (M == 0 || N == 0) return GEMM_OK;
  const PadPlan pp = plan_padding(D, C, A, B, M, N, K, beta, b_kn);
  if (!pp.ok) return GEMM_ERR_INVALID_VALUE;
  if (pp.total > 0) {
    if (!workspace || workspace_bytes < pp.total) return GEMM_ERR_INVALID_VALUE;
    if (!aligned16(workspace)) return GEMM_ERR_MISALIGNED;
    const uint64_t dbytes = static_cast<uint64_t>(M) * N * 2;
    if (overlaps(workspace, pp.total, D, dbytes) ||
        (beta != 0.0f && overlaps(workspace, pp.total, C, dbytes)) ||
        (K > 0 && (overlaps(workspace, pp.total, A, static_cast<uint64_t>(M) * K * 2) ||
                   overlaps(workspace, pp.total, B, static_cast<uint64_t>(N) * K * 2))))
      return GEMM_ERR_INVALID_VALUE;
  }
  int dev = 0;
  DeviceState* st = nullptr;
  if ((rc = current_device(&dev, &st)) != GEMM_OK) return rc;
  if (K == 0) return write_empty_sum(D, C, beta, M * N, device_sm_count(st), stream);

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int sms = device_sm_count(st);
  const auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (pp.pack_a && !ok(repack_rows(ws + pp.off_a, A, M, K, sms, stream))) return GEMM_ERR_LAUNCH;
  if (pp.pack_b && !ok(b_kn ? repack_rows(ws + pp.off_b, B, K, N, sms, stream)
                            : repack_rows(ws + pp.off_b, B, N, K, sms, stream)))
    return GEMM_ERR_LAUNCH;
  // Where C is read it ends up aligned with row stride ldc: in the padded D
  // (which the GEMM then updates in place), in D itself, or as given.
  const bool padded_copy = pp.pad_d && !pp.direct_d;
  void* d_eff = padded_copy ? static_cast<void*>(ws + pp.off_d) : D;
  const void* c_eff = C;
  if (beta != 0.0f && (padded_copy || pp.c_to_d)) {
    if (!ok(repack_rows(d_eff, C, M, N, sms, stream))) return GEMM_ERR_LAUNCH;
    c_eff = d_eff;
  }
  const uint64_t m = M, n = N, k = K, kp = pp.Kp, np = pp.Np;
  // With K padded, A's pad columns are +0 and the kernel iterates Kp; an
  // unpacked B (K x N) simply ends at row K and reads zeros past it.
  const View a = pp.pack_a ? View{ws + pp.off_a, kp, m, kp} : View{A, k, m, k};
  View b;
  if (b_kn)
    b = pp.pack_b ? View{ws + pp.off_b, np, k, np} : View{B, n, k, n};
  else
    b = pp.pack_b ? View{ws + pp.off_b, kp, n, kp} : View{B, k, n, k};
  const View d = padded_copy ? View{d_eff, np, m, np} : View{D, n, m, n};
  const Scaled sc{c_eff, alpha, beta, b_kn};
  rc = launch_gemm(M, N, pp.Kp, a, b, d, b_kn, &sc, padded_copy ? pp.Np : N, opt, st, stream,
                   pp.direct_d ? static_cast<uint16_t*>(D) : nullptr, N);
  if (rc != GEMM_OK) return rc;
  if (padded_copy && !ok(unpack_rows(D, d_eff, M, N, sms, stream))) return GEMM_ERR_LAUNCH;
  return GEMM_OK;
}

}  // namespace
}  // namespace gb300

using namespace gb300;

extern "C" int gemm_padded_workspace_bytes(const void* D, const void* C, const void* A,
                                           const void* B, int64_t M, int64_t N, int64_t K,
                                           float beta, int b_layout, uint64_t* bytes) {
  if (!bytes || M < 0 || N < 0 || K < 0 || M > INT_MAX || N > INT_MAX || K > INT_MAX ||
      (b_layout != 0 && b_layout != 1))
    return GEMM_ERR_INVALID_VALUE;
  const PadPlan pp = plan_padding(D, C, A, B, M, N, K, beta, b_layout);
  if (!pp.ok) return GEMM_ERR_INVALID_VALUE;
  *bytes = pp.total;
  return GEMM_OK;
}

extern "C" int gemm_f16_padded(void* D, const void* C, const void* A, const void* B, int64_t M,
                               int64_t N, int64_t K, float alpha, float beta, int b_layout,
                               void* workspace, uint64_t workspace_bytes,
                               const gemm_options_t* opt, void* stream) {
  return run_padded(D, C, A, B, M, N, K, alpha, beta, b_layout, workspace, workspace_bytes, opt,
                    static_cast<cudaStream_t>(stream));
}

