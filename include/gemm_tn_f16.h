/*
 * gemm_tn_f16 -- multi-stage pipelined fp16 GEMM D = A * B^T for GB300 (sm_103a).
 *
 * The operation is the one computed by the kernel of "cute(9) multistage_gemm"
 * (code listing and section 11 "性能测试"): A is M x K row-major, B is N x K
 * row-major, D is M x N row-major, D = A @ B^T.  Here the products are
 * accumulated in fp32 (in tensor memory) and D is rounded to fp16 once,
 * round-to-nearest-even.  The page's pipeline -- a kStage ring of shared-memory
 * tiles filled ahead of the MMA (its sections 4-6) and guarded against
 * read-after-write and write-after-read hazards ("第 6 课：Shared Memory 布局与
 * 异步流水", section 3) -- is realised with TMA loads, full/empty mbarrier
 * pairs and tcgen05.mma issued by one thread.
 *
 * All entry points are plain C.  Pointers named D, A, B are DEVICE pointers
 * on the current CUDA device; `stream` is a cudaStream_t (NULL = legacy
 * default stream) of that device.  No call allocates device memory, with one
 * exception: the 16 MiB array behind gemm_probe_latencies_static, a static
 * device array of the library's probe code that a GPU holds from the moment
 * that code is loaded (at the first use of a probe under lazy module loading,
 * the CUDA default; at context creation under eager loading) until exit.
 * Every function returns a gemm_status_t value (0 = success) unless stated.
 */
#ifndef GEMM_TN_F16_H
#define GEMM_TN_F16_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_VALUE = 1,     /* negative or too-large size, NULL pointer, overlap, bad option */
  GEMM_ERR_MISALIGNED = 2,        /* pointer not 16-byte aligned, or K or N not a multiple of 8 */
  GEMM_ERR_UNSUPPORTED_DEVICE = 3,/* current device is not compute capability 10.3 */
  GEMM_ERR_LAUNCH = 4,            /* the kernel launch itself failed */
  GEMM_ERR_TIMEOUT = 5,           /* a pipeline wait in the kernel gave up (see gemm_get_device_error) */
  GEMM_ERR_CUDA = 6,              /* another CUDA runtime error (no device, memset failed, ...) */
  GEMM_ERR_INVARIANT = 7          /* a pipeline invariant check failed (opt->check; see
                                     gemm_get_device_error) */
} gemm_status_t;

/* Kernel paths. */
enum {
  GEMM_PATH_AUTO = 0,    /* choose from the shape */
  GEMM_PATH_SQUARE = 1,  /* persistent 128 x BN tiles, compute-bound shapes */
  GEMM_PATH_SKINNY = 2,  /* M <= 128: one M tile, N spread over every SM, B streamed once
                            (the small-M kernel; see gemm_options_t.small_m) */
  GEMM_PATH_PAIR = 3     /* persistent 256 x BN tiles over CTA pairs (tcgen05 cta_group::2) */
};

/*
 * gemm_tn_f16: D[i][j] = fp16_rn( sum_k A[i][k] * B[j][k] ), fp32 accumulation.
 *
 *   D  device, M*N fp16, row-major, leading dimension N.  Written only.
 *   A  device, M*K fp16, row-major, leading dimension K.  Read only.
 *   B  device, N*K fp16, row-major, leading dimension K.  Read only.
 *   M, N, K  0 <= M, N, K <= 2^31 - 1.
 *
 * Requirements (checked on the host before anything is launched):
 *   - A, B, D 16-byte aligned and K % 8 == 0, N % 8 == 0 (TMA strides are
 *     multiples of 16 bytes), else GEMM_ERR_MISALIGNED;
 *   - D must not overlap A or B, pointers non-NULL when M*N > 0,
 *     else GEMM_ERR_INVALID_VALUE;
 *   - current device of compute capability 10.3, else GEMM_ERR_UNSUPPORTED_DEVICE.
 * M, N, K need not be multiples of the tile sizes: loads past the edge read
 * zeros and stores past the edge are clipped.  M == 0 or N == 0 is a no-op;
 * K == 0 writes D = 0 (the empty sum).
 * The call is asynchronous on `stream`.  A launch failure returns
 * GEMM_ERR_LAUNCH; a pipeline wait that times out inside the kernel (no
 * progress for the timeout, 2 s by default) is reported by
 * gemm_get_device_error().  The caller owns all buffers.
 */
int gemm_tn_f16(void* D, const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                void* stream);

/* Options for gemm_tn_f16_ex.  Zero-initialise and set what you need. */
typedef struct {
  int path;            /* GEMM_PATH_*                                           */
  int bn;              /* tile width along N: 0 = choose, else 32..256, % 32 == 0
                          (GEMM_PATH_PAIR: the pair's width; each CTA loads bn/2 rows of B) */
  int kstage;          /* shared-memory ring depth: 0 = deepest that fits, else 2..16 */
  int max_ctas;        /* persistent CTAs at most: 0 = one per SM.  The grid is then
                          balanced: the fewest CTAs (pairs) that keep the fewest
                          waves of tiles (units), so each gets the same number to one */
  int group_m;         /* m-blocks per rasterisation group: 0 = choose           */
  uint64_t timeout_ns; /* per-wait limit inside the kernel: 0 = 2 s              */
  int inject;          /* test hooks: 1 = the producer announces its first stage
                          but never loads it, so the consumers' waits run out;
                          the kernel then reports GEMM_ERR_TIMEOUT and exits.
                          2 = the producer stamps its first ring slot with a
                          wrong sequence number (nothing else changes), which
                          `check` must report as GEMM_ERR_INVARIANT */
  int katoms;          /* 64-wide K slices per ring stage: 0 = choose, 1 or 2 (a
                          stage of 2 halves the per-byte barrier and commit work) */
  int epi_warps;       /* epilogue warps per CTA: 0 = choose, 4 or 8 (8 doubles the
                          TMEM -> global drain rate, for short k loops) */
  int b_layout;        /* gemm_query_config only: plan for this B layout (GEMM_B_*);
                          gemm_f16_scaled takes the layout as an argument */
  int acc_f16;         /* 0: fp32 accumulator (default); 1: fp16 accumulator, rounded
                          after every 16-deep K slice -- the arithmetic of the
                          F16F16F16F16 MMA atom of "cute(9) multistage_gemm" */
  int b_resident;      /* 0 = choose; 1 = never; 2 = always (else GEMM_ERR_INVALID_VALUE).
                          Resident B: on a single-CTA path with one n-block (N <= bn)
                          and an N x K B, each CTA loads all of B into shared memory
                          once and its ring streams only A (the tall shapes) */
  int pdl;             /* 0: launch with programmatic stream serialization (the
                          kernel's set-up overlaps the end of the previous kernel
                          in the stream; it waits for that kernel -- griddepcontrol
                          -- before touching global memory); 1: plain launch */
  int wide;            /* pair path: 0 = choose, 1 = never, 2 = always (on another
                          path GEMM_ERR_INVALID_VALUE).  A wide unit is two adjacent
                          n-tiles (a 256 x 2*bn block) sharing each A slice: the
                          ring carries A once per two B halves and both TMEM
                          accumulators hold the unit, so the same shared memory
                          holds a deeper ring.  Results are bit-identical. */
  int small_m;         /* skinny path (M <= 128): 0 = choose, 1 = never, 2 = always (else
                          GEMM_ERR_INVALID_VALUE).  The small-M kernel computes one
                          128 x bn tile per CTA (so at most one n-tile per SM) and
                          stages its epilogue in its ring once the tile's MMAs are
                          done, so the whole shared memory holds the ring (four
                          stages at bn = 96 where the single-CTA kernel fits three).
                          Otherwise the single-CTA kernel runs.  With the same
                          katoms the results are bit-identical. */
  int check;           /* 1: verify the pipeline's invariants in the kernel (debug):
                          the producer stamps every ring slot with the sequence
                          number of the fill it issues there, and the MMA thread
                          compares it, once the slot is full, with the count of
                          slots it has consumed -- a wrong stage index or phase
                          that still lets the pipeline run.  A mismatch records
                          GEMM_ERR_INVARIANT (site 5) in the device error word;
                          the kernel never traps and runs on.  Built for the plain
                          forms (D stored by TMA, alpha = 1, beta = 0); with a
                          scaled epilogue or a D stored directly (gemm_f16_padded
                          with unaligned D rows) it is GEMM_ERR_INVALID_VALUE.
                          0: off, at no cost: separate kernel instantiations */
  int split_k;         /* 0 = choose, 1 = never, 2 = always (else GEMM_ERR_INVALID_VALUE).
                          Split: a cluster of two CTAs computes each 128 x bn tile,
                          each CTA half of the k range; the two exchange their fp32
                          partials through distributed shared memory and each
                          rounds and stores half of the tile.  Chosen by itself
                          for 256 <= K <= 1024 when the unsplit tiles fit in one
                          wave and the split ones in one wave of CTA pairs
                          (1024^3, 256^3).  Needs
                          an N x K B, an fp32 accumulator and aligned D rows;
                          results differ from the unsplit sum only in fp32
                          rounding (bit-exact where the partial sums are). */
  int multicast;       /* split-K only: 0 = choose, 1 = never, 2 = always (else
                          GEMM_ERR_INVALID_VALUE).  The cluster then also holds
                          the next n-tile and/or m-tile (4 or 8 CTAs); the CTAs of
                          one k-half that share an A or B block each load half of
                          it for both by TMA multicast, so each SM fetches half the
                          operand bytes it receives.  Chosen by itself with
                          partners along both n and m (8 CTAs) when every cluster
                          fits on the GPU at once; asked for, a 4-CTA cluster is
                          taken when 8 do not fit.  Results are bit-identical to
                          the pair form.  Not combined with `check`. */
} gemm_options_t;

/* gemm_tn_f16 with an explicit configuration (sweeps, tests).  Same
 * arguments, ownership and errors as gemm_tn_f16; an option out of range
 * returns GEMM_ERR_INVALID_VALUE.  `opt` may be NULL (= all zero). */
int gemm_tn_f16_ex(void* D, const void* A, const void* B, int64_t M, int64_t N, int64_t K,
                   const gemm_options_t* opt, void* stream);

/* B operand layouts for gemm_f16_scaled. */
enum {
  GEMM_B_NK = 0,   /* B is N x K row-major (leading dimension K): D = alpha A B^T + beta C */
  GEMM_B_KN = 1    /* B is K x N row-major (leading dimension N): D = alpha A B + beta C   */
};

/*
 * gemm_f16_scaled: D = fp16_rn( alpha * A op(B) + beta * C ), fp32 accumulation
 * and fp32 alpha, beta -- the problem "CUDA 算子笔记 2" states in its GEMM
 * section (C = alpha A B + beta C with fp16 matrices and fp32 scalars; its
 * B is K x N, i.e. GEMM_B_KN).
 *
 *   D  device, M*N fp16, row-major, leading dimension N.  Written only.
 *   C  device, M*N fp16, row-major, leading dimension N.  Read only, and only
 *      when beta != 0 (it may then be NULL).  C may be D itself (in place:
 *      C = alpha A B + beta C); any other overlap of C and D is rejected.
 *   A  device, M*K fp16, row-major.
 *   B  device: N*K row-major for GEMM_B_NK, K*N row-major for GEMM_B_KN.
 *
 * Requirements and errors are those of gemm_tn_f16, plus: C 16-byte aligned
 * when read; alpha and beta finite; b_layout one of GEMM_B_*.  With
 * GEMM_B_KN the tile width is a multiple of 64 (128 on the pair path); an
 * explicit opt->bn that is not is GEMM_ERR_INVALID_VALUE.  K == 0 writes
 * D = beta * C (rounded to fp16).  opt may be NULL.  Asynchronous on stream.
 */
int gemm_f16_scaled(void* D, const void* C, const void* A, const void* B, int64_t M, int64_t N,
                    int64_t K, float alpha, float beta, int b_layout, const gemm_options_t* opt,
                    void* stream);

/*
 * gemm_f16_padded: gemm_f16_scaled for any K and N and any 2-byte-aligned
 * operand -- the general shapes the host wrapper of "CUDA 算子笔记 2" (GEMM
 * section) serves by copying A, B and C into zero-padded buffers before its
 * kernel and copying the result back.
 *
 * Same operation, layouts (leading dimensions K or N, rows packed back to
 * back) and ownership as gemm_f16_scaled.  Each operand the kernel reads
 * whose base address or row stride is not a multiple of 16 bytes is first
 * copied, on `stream`, into `workspace` with its rows padded to a multiple
 * of 8 elements (+0 in the pad); the GEMM kernel then runs on the aligned
 * copies.  A D of that kind is written by the kernel's epilogue with plain
 * stores when beta == 0; when beta != 0 the GEMM updates a padded copy of C
 * in place, which is then copied into D.  Operands already aligned are used
 * in place, so with K % 8 == 0, N % 8 == 0 and 16-byte-aligned pointers this
 * is exactly
 * gemm_f16_scaled and needs no workspace.  The results are those of the
 * unpadded problem: the pad contributes exact zeros.
 *
 *   workspace        device, caller-owned, 16-byte aligned, at least the
 *                    size gemm_padded_workspace_bytes returns for the same
 *                    D, C, A, B, M, N, K, beta and b_layout; it must not
 *                    overlap any operand.  Its contents on entry do not
 *                    matter and on return are unspecified.  It may be NULL
 *                    when that size is 0.  Calls in flight at once on
 *                    different streams need separate workspaces.
 *   workspace_bytes  its size in bytes.
 *
 * Errors: a pointer that is odd (not fp16-aligned) is GEMM_ERR_MISALIGNED;
 * a workspace that is too small or overlaps an operand is
 * GEMM_ERR_INVALID_VALUE, and a misaligned one GEMM_ERR_MISALIGNED; the
 * other checks are those of gemm_f16_scaled.  Nothing is launched when a
 * check fails.  Up to five kernels are launched (repack A, repack B, repack
 * C when C is read into a padded D, the GEMM, and then the copy back of that
 * D), all asynchronous on `stream`.
 */
int gemm_f16_padded(void* D, const void* C, const void* A, const void* B, int64_t M, int64_t N,
                    int64_t K, float alpha, float beta, int b_layout, void* workspace,
                    uint64_t workspace_bytes, const gemm_options_t* opt, void* stream);

/* Workspace bytes gemm_f16_padded needs for these arguments (0 when every
 * operand it reads or writes is already aligned).  It depends on the
 * pointers' alignment, so pass the pointers of the call (they are not
 * dereferenced).  Host only; returns GEMM_ERR_INVALID_VALUE for a negative
 * or too-large size (K or N above 2^31 - 8, or a workspace of 2^63 bytes or
 * more), a bad b_layout or a NULL `bytes`.  gemm_f16_padded refuses the same
 * sizes. */
int gemm_padded_workspace_bytes(const void* D, const void* C, const void* A, const void* B,
                                int64_t M, int64_t N, int64_t K, float beta, int b_layout,
                                uint64_t* bytes);

/* Chosen configuration for a shape (host only, no GPU work; needs a current
 * device only to read its SM count -- with no device, 148 SMs are assumed). */
typedef struct {
  int path, bm, bn, bk, kstage, ctas, group_m, tiles;
  int smem_bytes, tmem_cols;
  int katoms;          /* bk = 64 * katoms */
  int epi_warps;       /* threads per CTA = 64 + 32 * epi_warps */
  int b_resident;      /* 1: B is held in shared memory for the whole kernel */
  int pdl;             /* 1: launched with programmatic stream serialization */
  int wide;            /* 1: pair units of two adjacent n-tiles (tiles still counts
                          output tiles; the grid is sized by units) */
  int small_m;         /* 1: the small-M kernel (one tile per CTA) */
  int split_k;         /* 1: k split over a CTA pair (ctas = 2 x tiles) */
  int cluster;         /* CTAs per thread-block cluster: 1, 2 (pairs, split K), or 4
                          or 8 (split K with multicast operands) */
} gemm_config_t;
int gemm_query_config(int64_t M, int64_t N, int64_t K, const gemm_options_t* opt,
                      gemm_config_t* out);

/* Synchronises `stream`, then returns and clears the device error word of
 * `stream` on the current device: GEMM_OK, GEMM_ERR_TIMEOUT if a kernel
 * launched on it gave up waiting, or GEMM_ERR_INVARIANT if a call with
 * opt->check found a ring slot out of sequence (the first error is kept until
 * read).  Each stream has its own word: the legacy default stream (NULL) and
 * the first 63 other streams a process passes to this library; streams beyond
 * those share words by a hash of their handle, so a poll may then also report
 * (and clear) another stream's error.  A kernel captured in a CUDA graph
 * reports to the word of the stream it was captured on.
 * If `raw` is not NULL it receives the raw word (low byte = status, next byte
 * = the wait site that gave up: 1 producer/empty, 2 mma/full, 3 mma/tmem-empty,
 * 4 epilogue/tmem-full; or 5, the invariant check of a ring slot). */
int gemm_get_device_error(void* stream, uint32_t* raw);

/* Minimum ring depth that hides a copy latency behind compute:
 * S_min = ceil(copy_cycles / compute_cycles) + 1 ("第 6 课：Shared Memory 布局与
 * 异步流水", section 4: in-flight stages >= ceil(T_copy/T_compute), plus the one
 * being consumed).  Both arguments must be positive; otherwise returns -1.
 * Host only. */
int64_t gemm_minimum_stages(int64_t copy_cycles, int64_t compute_cycles);

/* Latency probes on the current device (the two inputs of S_min), in SM clock
 * cycles, averaged over `reps` measurements each:
 *   copy_cycles    -- one stage's TMA loads (A 128x64 + B bn x 64 fp16) from
 *                     issue to the full barrier completing, one stage in
 *                     flight per SM, `ctas` SMs loading at once (0 = all SMs),
 *                     addresses strided through a `footprint_bytes` region of
 *                     `scratch` (device, >= footprint_bytes, caller-owned) so
 *                     that loads miss L2 when the region exceeds it;
 *   compute_cycles -- one k-block of MMAs (4 x tcgen05.mma 128 x bn x 16)
 *                     issued back to back, per k-block.
 * Synchronous. */
int gemm_probe_latencies(int bn, int ctas, const void* scratch, int64_t footprint_bytes, int reps,
                         double* copy_cycles, double* compute_cycles, void* stream);

/* gemm_probe_latencies_static: the same probes as gemm_probe_latencies for
 * callers that cannot allocate device memory -- for example a serving process
 * whose memory pool already holds nearly all of HBM, or a loop that must not
 * call cudaMalloc/cudaFree because they can synchronise the device.  The
 * pages have no counterpart to this entry point; it exists only for such
 * callers.
 *   - The copy probe loads from a fixed 16 MiB array in device memory owned by
 *     the library (held on every GPU that loads it until the process exits);
 *     footprint_bytes above 16 MiB returns GEMM_ERR_INVALID_VALUE, other
 *     arguments are checked as in gemm_probe_latencies.  16 MiB fits in L2,
 *     so copy_cycles is the L2-resident latency.
 *   - Calls no allocating routine.  The first call on a device (and the first
 *     after the device's context was re-created, e.g. by cudaDeviceReset)
 *     looks up the array's device address with cudaGetSymbolAddress; under
 *     lazy module loading, the CUDA default, that lookup may load the
 *     library's device code and so allocate the 16 MiB array itself.  Make
 *     that first call early, while 16 MiB are free, and before any stream
 *     capture on the device; later calls allocate nothing.
 *   - All calls share the array and the result counters (cleared at the start
 *     of each call); calls that overlap on the GPU race and report wrong
 *     numbers.
 * Synchronous. */
int gemm_probe_latencies_static(int bn, int ctas, int64_t footprint_bytes, int reps,
                                double* copy_cycles, double* compute_cycles, void* stream);

/* Human-readable name of a status code (static string). */
const char* gemm_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_TN_F16_H */
