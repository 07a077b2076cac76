/*
 * fa_testing.h — C ABI of the TEST library libfa_gb300_testing.so.
 *
 * Not part of the attention library's contract (include/fa.h): these entry
 * points exercise single device primitives (the exponentials, one-tile
 * tcgen05 MMAs, TMA and tensor-memory round trips, a bounded wait that must
 * time out), run microbenchmarks of the GPU's units, and run the work
 * scheduler on the host. The tests use them to pin the building blocks the
 * attention kernels are made of; libfa_gb300.so contains none of them.
 *
 * Conventions as in fa.h: device pointers, status codes (fa_status), calls
 * asynchronous on `stream`. This library keeps its own device error word and
 * its own last-error text.
 */
#ifndef FA_GB300_TESTING_H
#define FA_GB300_TESTING_H

#include <stddef.h>

#if defined(__GNUC__)
#define FA_TEST_API __attribute__((visibility("default")))
#else
#define FA_TEST_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Thread-local detail of the last failing call into this library ("" if none). */
FA_TEST_API const char* fa_test_last_error(void);

/*
 * Synchronises the device and reads (optionally clears) this library's device
 * error word (the wait-site code a probe recorded; 0 if none).
 */
FA_TEST_API int fa_test_get_device_error(int* code, int clear);

/* y[i] = 2^x[i] on the device: mode 0 software polynomial, mode 1 MUFU ex2. */
FA_TEST_API int fa_test_exp2(const float* x, float* y, int n, int mode, void* stream);

/*
 * Microbenchmarks, one CTA per SM (`ctas` CTAs): each CTA writes two doubles to
 * out_dev[2*cta + {0, 1}]: its clock64 span and the operations it performed.
 *   kind 0: MUFU ex2 throughput, kind 1: software exp2 throughput (operations =
 *   exponentials, 256 threads per CTA); kinds 2-6: tcgen05 bf16 MMA throughput
 *   for M128 K16 and N = 256, 128, 64 with both operands in shared memory
 *   (kinds 2, 3, 4) or N = 128, 64 with A in TMEM (kinds 5, 6), issued by one
 *   thread; kinds 7-11: the same five shapes issued by an elected lane of a
 *   converged warp; kinds 12-27: SS N=128 MMAs in groups of 4 with extras
 *   after each group selected by the bits of (kind - 12): 1 tcgen05 fence, 2 a
 *   commit, 4 an mbarrier poll, 8 a runtime accumulate flag; kinds 28-30: SS
 *   N=128 MMAs with descriptors built next to each MMA from a loop-varying
 *   offset, issued by lane 0 (28) or an elected lane of the converged warp
 *   (29), or with hoisted descriptors (30); kinds 31-34: kind 28 plus, per group
 *   of 4 MMAs, a runtime accumulate flag (31), a tcgen05 fence (32), a commit
 *   (33), a bounded mbarrier wait on a completed phase (34), a bare try_wait
 *   loop (35) or a test_wait loop (36) on it, a named-barrier handshake with a
 *   second warp (37, warp-wide issue), a shared-memory flag read (38) or a
 *   global-memory read (39); kinds 40-51: latency of probes made by another warp
 *   while warp 0 streams MMAs or not: (kind-40)/4 selects the probe (0 TMEM
 *   load, 1 shared load, 2 mbarrier test_wait), bit 1 whether the probing warp
 *   shares warp 0's SM sub-partition, bit 0 whether MMAs run; operations =
 *   probes; operations =
 *   FLOPs. iters <= 2^24.
 */
FA_TEST_API int fa_micro(int kind, int iters, double* out_dev, int ctas, void* stream);

/* Host twin of the device polynomial exp2 (identical operation sequence). */
FA_TEST_API float fa_exp2_poly_host(float x);

/*
 * One-tile tcgen05 MMA probe (one CTA), fp32 result C[128][N], N in {64,128}:
 *   mode 0: C = A[128][128] * B[N][128]^T   mode 1: C = A * B[128][N] (A via TMEM)
 *   mode 2: C = A^T * B[128][N]   (A is read as [K=128][M=128])
 * A, B bf16 row-major device buffers.
 */
FA_TEST_API int fa_test_mma(const void* A, const void* B, float* C, int mode, int N, void* stream);

/*
 * One-tile e4m3 tcgen05 MMA probe (kind::f8f6f4, one CTA): fp32
 * C[128][N] = A[128][128] * B[N][128]^T, N in {64,128}; A and B are row-major
 * e4m3 codes (device). mode 0: A and B from shared memory; mode 1: A from
 * tensor memory.
 */
FA_TEST_API int fa_test_mma_fp8(const void* A, const void* B, float* C, int mode, int N, void* stream);

/*
 * Data-path round trips (one CTA): a 128-row x 64-column bf16 tile of src
 * (device, 16-byte aligned, row-major) is loaded into shared memory by TMA
 * (128-byte swizzle) and stored to dst by TMA; and each of 128 threads writes
 * the words r * 1000 + c (c < 32) to its tensor-memory lane and reads them back
 * into tmem_out[r][c] (device, 128 x 32 unsigned).
 */
FA_TEST_API int fa_test_roundtrip(const void* src, void* dst, unsigned* tmem_out, void* stream);

/*
 * CTA-pair (cta_group::2) tcgen05 MMA probe: a cluster of two CTAs computes
 * C[256][N] (fp32), N = 128, with M=256 MMAs issued by CTA 0; CTA r
 * holds A rows [128r, 128r+128) and B's N columns [r*N/2, (r+1)*N/2).
 *   mode 0: C = A[256][128] * B[N][128]^T   mode 1: C = A * B[128][N] (A via TMEM)
 * flags (device, 4 ints): [r] = 1 if CTA r saw the MMAs complete, [2+r] = its
 * TMEM base address (equal in both CTAs).
 */
FA_TEST_API int fa_test_mma_pair(const void* A, const void* B, float* C, int* flags, int mode, int N,
                            void* stream);

/*
 * Runs a kernel whose bounded wait can never complete; *status_dev (device
 * int) becomes 1 when the wait timed out as designed. Leaves the site code in
 * the device error word (clear it with fa_get_device_error(&c, 1)).
 */
FA_TEST_API int fa_test_wait_timeout(int* status_dev, double timeout_ms, void* stream);

/*
 * Host run of the work scheduler: writes, for CTA `cta` of a persistent grid
 * of `grid` CTAs, its units in execution order as 4 ints each
 * (sequence, row block, head, cost) into out (room for max_units units).
 * heads_per_group: heads per scheduler group (0 = the kernels' own choice: the
 * fewest heads whose units cover the grid).
 * kind 0 = forward (units of 256 query rows, cost = KV blocks of 128), kind 1
 * = one-pass backward (units of 128 keys, cost = query blocks of 64), kind 2 =
 * dK/dV pass of the two-pass backward (units of 128 keys, cost = query blocks
 * of 128), kind 3 = its dQ pass (units of 128 query rows, cost = KV blocks of
 * 128), kind 4 = the dK/dV pass on CTA pairs (units of 256 keys, cost =
 * query blocks of 128), kind 5 = the dQ pass for head dim 192 (units of 128
 * query rows, cost = KV blocks of 64; the dK/dV pass for head dim 192 is
 * kind 1). cu_seqlens_host
 * is a HOST array (or NULL for dense B x Sq/Sk). Returns the number of units
 * (may exceed max_units; only max_units are written), or -1 on bad arguments.
 */
FA_TEST_API int fa_sched_list(int kind, int B, const int* cu_seqlens_host, int Sq, int Sk, int heads,
                  int causal, int grid, int cta, int heads_per_group, int* out, int max_units);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_TESTING_H */
