// Row repacking between a caller's fp16 matrix (rows of `cols` elements,
// packed back to back, any 2-byte alignment) and a 16-byte-aligned copy whose
// rows are padded to a multiple of 8 elements -- the layout the TMA tensor
// maps of the GEMM need (row strides a multiple of 16 bytes).  This is the
// padding step of the host wrapper in "CUDA 算子笔记 2" (GEMM section), which
// copies A, B and C into zero-padded buffers before the kernel and copies C
// back after it; here the copies are kernels on the caller's stream and the
// padding is only to the next multiple of 8 elements.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>

namespace gb300 {

// Elements per padded row: cols rounded up to a multiple of 8.
inline int64_t padded_cols(int64_t cols) { return (cols + 7) / 8 * 8; }

// dst (16-byte aligned, rows x padded_cols(cols), row stride padded_cols(cols))
// <- src (rows x cols, row stride cols); the pad columns are written as +0.
// Returns a cudaError_t of the launch.
cudaError_t repack_rows(void* dst, const void* src, int64_t rows, int64_t cols, int sm_count,
                        cudaStream_t stream);

// dst (rows x cols, row stride cols, any 2-byte alignment) <- the first cols
// columns of src (16-byte aligned, row stride padded_cols(cols)).
cudaError_t unpack_rows(void* dst, const void* src, int64_t rows, int64_t cols, int sm_count,
                        cudaStream_t stream);

}  // namespace gb300
