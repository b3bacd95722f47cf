// Host-side pieces shared by the library's C-ABI translation units: the
// per-device state, operand views, and the single GEMM launch that the plain,
// scaled and padded entry points all end in.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

#include "gemm_tn_f16.h"

namespace gb300 {

struct DeviceState;  // per-device cache: SM count, granted smem, co-resident pairs

// The current device, checked to be compute capability 10.3 (state cached
// per device); GEMM_ERR_CUDA or GEMM_ERR_UNSUPPORTED_DEVICE otherwise.
int current_device(int* dev_out, DeviceState** st_out);
int device_sm_count(const DeviceState* st);

// A row-major fp16 matrix as one TMA tensor map sees it: `cols` contiguous
// elements per row, `rows` rows, `ld` elements between row starts (ld * 2 a
// multiple of 16, the base 16-byte aligned).
struct View {
  const void* ptr;
  uint64_t cols, rows, ld;
};

// The scaled form D = alpha * A op(B) + beta * C (b_kn: B is K x N).
struct Scaled {
  const void* C;
  float alpha, beta;
  int b_kn;
};

// Byte ranges [a, a + abytes) and [b, b + bbytes) intersect.
bool overlaps(const void* a, uint64_t abytes, const void* b, uint64_t bbytes);

// D = beta * C (rounded to fp16), or D = 0 when C is null or beta == 0: the
// empty sum (K == 0).  Element by element, so any 2-byte alignment is fine.
int write_empty_sum(void* D, const void* C, float beta, int64_t n, int sm_count,
                    cudaStream_t stream);

// Options checked against the shape even when there is nothing to compute.
int check_options(const gemm_options_t* opt, int b_kn, int64_t M, int64_t N, int64_t K);

// One GEMM launch on aligned operands.  M, N, K are the extents the kernel
// tiles and iterates; the views give each operand's tensor-map extents and
// row stride (A: K x M, B: K x N for an N x K B or N x K for a K x N B,
// D: N x M, as cols x rows).  A view may be narrower than the iterated
// extent: the loads past its edge read zeros.  sc != nullptr selects the
// scaled epilogue, reading C with row stride ldc.  d_direct != nullptr
// stores D with plain stores there (row stride ldd, any 2-byte alignment)
// instead of TMA stores through the view d, which is then not used.
int launch_gemm(int64_t M, int64_t N, int64_t K, const View& a, const View& b, const View& d,
                int b_kn, const Scaled* sc, int64_t ldc, const gemm_options_t* opt,
                DeviceState* st, cudaStream_t stream, uint16_t* d_direct = nullptr,
                int64_t ldd = 0);

}  // namespace gb300
