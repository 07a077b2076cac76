// Device probes of the test library (libfa_gb300_testing.so, declared in
// include/fa_testing.h; not linked into the attention library):
//   * the device exponentials (software polynomial and MUFU ex2) over an array;
//   * a one-tile tcgen05 MMA probe that checks the shared-memory/instruction
//     descriptors, the TMEM load/store layout and the TMEM-A operand form
//     against a plain product computed by the test;
//   * a bounded-wait probe whose wait can never complete, which must end with
//     the timeout status instead of hanging.
#include "../exp2_poly.cuh"
#include "../internal.h"
#include "../ptx.cuh"

namespace fa {
using namespace ptx;

__global__ void exp2_probe_kernel(const float* x, float* y, int n, int mode) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) y[i] = mode == 0 ? exp2_poly(x[i]) : ex2_mufu(x[i]);
}

cudaError_t launch_exp2_probe(const float* x, float* y, int n, int mode, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  exp2_probe_kernel<<<(n + 255) / 256, 256, 0, st>>>(x, y, n, mode);
  return cudaGetLastError();
}

// Byte offset of element (r, c) of a rows x cols bf16 matrix stored as
// 128-byte-swizzled column chunks of 64 elements (the TMA SWIZZLE_128B image).
__device__ __forceinline__ uint32_t sw128_offset(int r, int c, int rows) {
  const int chunk = c >> 6;
  const int byte = (c & 63) * 2;
  const int unit = (byte >> 4) ^ (r & 7);
  return chunk * rows * 128 + r * 128 + unit * 16 + (byte & 15);
}

// mode 0: C[128][N] = A[128][128] * B[N][128]^T    (A, B K-major in shared memory)
// mode 1: C[128][N] = A[128][128] * B[128][N]      (A from TMEM, B MN-major)
// mode 2: C[128][N] = At[128][128]^T * B[128][N]   (A MN-major, B MN-major)
// A/At/B are row-major bf16 in global memory; C is fp32 row-major.
__global__ void __launch_bounds__(128, 1)
    mma_probe_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B, float* C, int mode, int N,
                     int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t a_s = base, b_s = base + 32768;
  const uint32_t bar = base + 65536;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 65536 + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 65536 + 72);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

  // stage A (128 x 128) and B into swizzled shared memory with plain stores
  for (int i = tid; i < 128 * 128; i += 128) {
    const int r = i >> 7, c = i & 127;
    *reinterpret_cast<__nv_bfloat16*>(smem + sw128_offset(r, c, 128)) = A[i];
  }
  const int b_rows = mode == 0 ? N : 128, b_cols = mode == 0 ? 128 : N;
  for (int i = tid; i < b_rows * b_cols; i += 128) {
    const int r = i / b_cols, c = i % b_cols;
    *reinterpret_cast<__nv_bfloat16*>(smem + 32768 + sw128_offset(r, c, b_rows)) = B[i];
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  if (mode == 1) {
    // thread r writes row r of A (bf16 pairs) into TMEM columns [0, 64)
    const int r = tid;
    uint32_t pk[32];
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = half * 64 + 2 * j;
        const float lo = __bfloat162float(A[r * 128 + c]);
        const float hi = __bfloat162float(A[r * 128 + c + 1]);
        pk[j] = pack_bf16x2(lo, hi);
      }
      tmem_st32(tmem + lane_off + half * 32, pk);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t d_tm = tmem + 256;
  if (tid == 0) {
    for (int kk = 0; kk < 8; ++kk) {
      if (mode == 0) {
        const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
        const uint32_t boff = (kk >> 2) * (N * 128) + (kk & 3) * 32;
        mma_ss(d_tm, sdesc_sw128(a_s + off, 128 * 128, 1024),
               sdesc_sw128(b_s + boff, N * 128, 1024), idesc_bf16(128, N, false, false),
               kk > 0);
      } else if (mode == 1) {
        mma_ts(d_tm, tmem + kk * 8, sdesc_sw128(b_s + kk * 2048, 128 * 128, 1024),
               idesc_bf16(128, N, false, true), kk > 0);
      } else {
        mma_ss(d_tm, sdesc_sw128(a_s + kk * 2048, 128 * 128, 1024),
               sdesc_sw128(b_s + kk * 2048, 128 * 128, 1024), idesc_bf16(128, N, true, true),
               kk > 0);
      }
    }
    tc_commit(bar);
  }
  const WaitCtl wc{err, abort_flag, 1000000000ull};
  const bool ok = mbar_wait(bar, 0, wc, SITE_TEST);
  tc_fence_after();
  if (ok) {
    for (int c = 0; c < N; c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + 256 + c, v);
      for (int i = 0; i < 32; ++i) C[tid * N + c + i] = __uint_as_float(v[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_mma_probe(const __nv_bfloat16* A, const __nv_bfloat16* B, float* C, int mode,
                             int N, cudaStream_t st) {
  const int smem = 65536 + 128 + 1024 + 65536;  // slack keeps any mis-decoded offset in bounds
  cudaError_t e = cudaFuncSetAttribute(mma_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mma_probe_kernel<<<1, 128, smem, st>>>(A, B, C, mode, N, device_error_word());
  return cudaGetLastError();
}

// 8-bit operands, K-major, 128-byte swizzle: rows of 128 one-byte elements.
__device__ __forceinline__ uint32_t sw128_offset8(int r, int c) {
  return r * 128 + ((((uint32_t)c >> 4) ^ (uint32_t)(r & 7)) << 4) + (c & 15);
}

// e4m3 (kind::f8f6f4) probe: C[128][N] = A[128][128] * B[N][128]^T, fp32.
// mode 0: A and B in shared memory; mode 1: A from TMEM (four codes per
// column), B in shared memory. A and B are row-major e4m3 codes.
__global__ void __launch_bounds__(128, 1)
    mma_fp8_probe_kernel(const uint8_t* A, const uint8_t* B, float* C, int mode, int N,
                         int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t a_s = base, b_s = base + 16384;
  const uint32_t bar = base + 32768;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 32768 + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 32768 + 72);
  const int warp = threadIdx.x >> 5;
  const int tid = threadIdx.x;
  for (int i = tid; i < 128 * 128; i += 128) smem[sw128_offset8(i >> 7, i & 127)] = A[i];
  for (int i = tid; i < N * 128; i += 128) smem[16384 + sw128_offset8(i >> 7, i & 127)] = B[i];
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  if (mode == 1) {
    uint32_t pk[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const uint8_t* a = A + tid * 128 + 4 * j;
      pk[j] = (uint32_t)a[0] | ((uint32_t)a[1] << 8) | ((uint32_t)a[2] << 16) |
              ((uint32_t)a[3] << 24);
    }
    tmem_st32(tmem + lane_off, pk);
    tmem_st_wait();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t d_tm = tmem + 256;
  if (tid == 0) {
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t bd = sdesc_sw128(b_s + kk * 32, 16384, 1024);
      if (mode == 0)
        mma_ss_f8(d_tm, sdesc_sw128(a_s + kk * 32, 16384, 1024), bd, idesc_e4m3(128, N), kk > 0);
      else
        mma_ts_f8(d_tm, tmem + kk * 8, bd, idesc_e4m3(128, N), kk > 0);
    }
    tc_commit(bar);
  }
  const WaitCtl wc{err, abort_flag, 1000000000ull};
  const bool ok = mbar_wait(bar, 0, wc, SITE_TEST);
  tc_fence_after();
  if (ok) {
    for (int c = 0; c < N; c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + 256 + c, v);
      for (int i = 0; i < 32; ++i) C[tid * N + c + i] = __uint_as_float(v[i]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_mma_fp8_probe(const uint8_t* A, const uint8_t* B, float* C, int mode, int N,
                                 cudaStream_t st) {
  const int smem = 32768 + 128 + 1024 + 32768;  // slack keeps any mis-decoded offset in bounds
  cudaError_t e = cudaFuncSetAttribute(mma_fp8_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mma_fp8_probe_kernel<<<1, 128, smem, st>>>(A, B, C, mode, N, device_error_word());
  return cudaGetLastError();
}

// Round trips through the data paths the kernels use, one CTA of 128 threads:
//   TMA: a 128-row x 64-column bf16 tile (128-byte swizzle) loaded from src
//        into shared memory and stored back to dst by TMA;
//   TMEM: thread r writes the words r * 1000 + c (c < 32) into its lane's
//        columns [0, 32) and reads them back into tmem_out[r][c].
struct RoundTrip {
  CUtensorMap src, dst;
  uint32_t* tmem_out;
  int* err;
};

__global__ void __launch_bounds__(128, 1) roundtrip_probe_kernel(const __grid_constant__ RoundTrip p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t tile = base, bar = base + 16384;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 16384 + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16384 + 72);
  const int warp = threadIdx.x >> 5, tid = threadIdx.x;
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtl wc{p.err, abort_flag, 1000000000ull};
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, 16384);
    tma_load_3d(tile, &p.src, bar, 0, 0, 0);
    if (mbar_wait(bar, 0, wc, SITE_TEST)) {
      tma_store_3d(&p.dst, tile, 0, 0, 0);
      tma_store_commit();
      tma_store_wait_all();
    }
  }
  __syncwarp();                       // warp 0 reconverges before the warp-wide TMEM ops
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  uint32_t v[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) v[c] = (uint32_t)tid * 1000u + (uint32_t)c;
  tmem_st32(tmem + lane_off, v);
  tmem_st_wait();
  uint32_t w[32];
  tmem_ld32(tmem + lane_off, w);
#pragma unroll
  for (int c = 0; c < 32; ++c) p.tmem_out[tid * 32 + c] = w[c];
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

cudaError_t launch_roundtrip_probe(const CUtensorMap& src, const CUtensorMap& dst,
                                   uint32_t* tmem_out, cudaStream_t st) {
  RoundTrip p;
  p.src = src;
  p.dst = dst;
  p.tmem_out = tmem_out;
  p.err = device_error_word();
  const int smem = 16384 + 128 + 1024;
  cudaError_t e = cudaFuncSetAttribute(roundtrip_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  roundtrip_probe_kernel<<<1, 128, smem, st>>>(p);
  return cudaGetLastError();
}

// CTA-pair (cta_group::2) MMA probe: a cluster of two CTAs computes
//   mode 0: C[256][N] = A[256][128] * B[N][128]^T   (A, B K-major in shared memory)
//   mode 1: C[256][N] = A[256][128] * B[128][N]     (A from TMEM, B MN-major)
// with M=256 MMAs issued by CTA 0. CTA r holds A rows [128r, 128r+128) and B's
// N columns [r*N/2, (r+1)*N/2); its TMEM receives C rows [128r, 128r+128).
// flags[r] = 1 if CTA r saw its MMAs complete; flags[2 + r] = its TMEM base.
// TMEM (256 columns): A in [0, 64) for mode 1, C in [128, 128 + N), N = 128.
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    mma_pair_probe_kernel(const __nv_bfloat16* A, const __nv_bfloat16* B, float* C, int* flags,
                          int mode, int N, int* err) {
  extern __shared__ __align__(1024) uint8_t smem_pp[];
  const uint32_t base = smem_u32(smem_pp);
  uint8_t* smem = smem_pp;
  const uint32_t a_s = base, b_s = base + 32768;
  const uint32_t bar = base + 65536;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 65536 + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 65536 + 72);
  const int warp = threadIdx.x >> 5, tid = threadIdx.x;
  const int rank = (int)cluster_ctarank();
  const int nh = N / 2;
  for (int i = tid; i < 128 * 128; i += 128) {
    const int r = i >> 7, c = i & 127;
    *reinterpret_cast<__nv_bfloat16*>(smem + sw128_offset(r, c, 128)) = A[(rank * 128 + r) * 128 + c];
  }
  if (mode == 0) {
    for (int i = tid; i < nh * 128; i += 128) {                 // B rows [rank*nh, +nh), K-major
      const int r = i >> 7, c = i & 127;
      *reinterpret_cast<__nv_bfloat16*>(smem + 32768 + sw128_offset(r, c, nh)) =
          B[(rank * nh + r) * 128 + c];
    }
  } else {
    for (int i = tid; i < 128 * nh; i += 128) {                 // B columns [rank*nh, +nh), MN-major
      const int r = i / nh, c = i % nh;
      *reinterpret_cast<__nv_bfloat16*>(smem + 32768 + sw128_offset(r, c, 128)) =
          B[r * N + rank * nh + c];
    }
  }
  if (tid == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc_pair(smem_u32(tmem_slot), 256);
    tmem_relinquish_pair();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  if (mode == 1) {                                              // A rows into TMEM columns [0, 64)
    uint32_t pk[32];
    for (int half = 0; half < 2; ++half) {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int c = half * 64 + 2 * j;
        const int row = rank * 128 + tid;
        pk[j] = pack_bf16x2(__bfloat162float(A[row * 128 + c]), __bfloat162float(A[row * 128 + c + 1]));
      }
      tmem_st32(tmem + lane_off + half * 32, pk);
    }
    tmem_st_wait();
  }
  tc_fence_before();
  cluster_sync_all();                                           // both CTAs' operands in place
  tc_fence_after();
  const uint32_t d_tm = tmem + 128;
  if (rank == 0 && tid == 0) {
    for (int kk = 0; kk < 8; ++kk) {
      if (mode == 0) {
        const uint32_t off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
        const uint32_t boff = (kk >> 2) * (nh * 128) + (kk & 3) * 32;
        mma_ss_pair(d_tm, sdesc_sw128(a_s + off, 128 * 128, 1024),
                    sdesc_sw128(b_s + boff, nh * 128, 1024), idesc_bf16(256, N, false, false),
                    kk > 0);
      } else {
        mma_ts_pair(d_tm, tmem + kk * 8, sdesc_sw128(b_s + kk * 2048, 128 * 128, 1024),
                    idesc_bf16(256, N, false, true), kk > 0);
      }
    }
    tc_commit_pair(bar, 0x3);
  }
  const WaitCtl wc{err, abort_flag, 1000000000ull};
  const bool ok = mbar_wait(bar, 0, wc, SITE_TEST);
  tc_fence_after();
  if (ok) {
    for (int c = 0; c < N; c += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_off + 128 + c, v);
      for (int i = 0; i < 32; ++i) C[(rank * 128 + tid) * N + c + i] = __uint_as_float(v[i]);
    }
  }
  if (tid == 0) {
    flags[rank] = ok ? 1 : 0;
    flags[2 + rank] = (int)tmem;
  }
  tc_fence_before();
  cluster_sync_all();                                           // no CTA frees TMEM its peer still uses
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 256);
  }
}

cudaError_t launch_mma_pair_probe(const __nv_bfloat16* A, const __nv_bfloat16* B, float* C,
                                  int* flags, int mode, int N, cudaStream_t st) {
  const int smem = 65536 + 128;
  cudaError_t e = cudaFuncSetAttribute(mma_pair_probe_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  mma_pair_probe_kernel<<<2, 128, smem, st>>>(A, B, C, flags, mode, N, device_error_word());
  return cudaGetLastError();
}

// A wait on a barrier that nothing ever arrives on: must return through the
// timeout path, recording SITE_TEST in the error word and `status[0] = 1`.
__global__ void wait_timeout_probe_kernel(int* status, int* err, unsigned long long timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{err, &abort_flag, timeout_ns};
  const bool ok = mbar_wait(smem_u32(&bar), 0, wc, SITE_TEST);
  if (threadIdx.x == 0) status[0] = ok ? 0 : 1;
}

cudaError_t launch_wait_timeout_probe(int* status, unsigned long long timeout_ns,
                                      cudaStream_t st) {
  wait_timeout_probe_kernel<<<1, 32, 0, st>>>(status, device_error_word(), timeout_ns);
  return cudaGetLastError();
}

}  // namespace fa

namespace fa {

// ---------------------------------------------------------------------------
// Microbenchmarks (one CTA per SM; each CTA writes its clock64 span and op
// count to out[2*blockIdx.x + {0,1}] as doubles).
//   kind 0: MUFU ex2.approx throughput      (ops = exponentials)
//   kind 1: software exp2 throughput        (ops = exponentials)
//   kind 2: tcgen05 bf16 MMA throughput, M128 N256 K16, smem operands (ops = FLOPs)
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256, 1) micro_exp_kernel(int iters, int poly, double* out,
                                                           float seed) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = -(seed + 0.001f * (threadIdx.x + i));
  __syncthreads();
  const long long t0 = clock64();
  for (int it = 0; it < iters; ++it) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float y = poly ? exp2_poly(a[i]) : ex2_mufu(a[i]);
      a[i] = -y - 0.5f;   // stays in (-1.5, -0.5): keeps a dependency chain per lane
    }
  }
  __syncthreads();
  const long long t1 = clock64();
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc += a[i];
  if (acc == 12345.f) out[0] = acc;   // keep the work
  if (threadIdx.x == 0) {
    out[2 * blockIdx.x] = (double)(t1 - t0);
    out[2 * blockIdx.x + 1] = (double)iters * 8.0 * blockDim.x;
  }
}

// tcgen05 MMA throughput for one instruction shape: M=128, N in {64,128,256},
// K=16, operands from shared memory (ts = 0) or A from TMEM (ts = 1).
template <int N, int TS>
__global__ void __launch_bounds__(128, 1) micro_mma_kernel(int iters, int style, double* out,
                                                           int* err) {
  constexpr int ts = TS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t bar = base + 65536;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 65536 + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 65536 + 72);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 65536 / 16; i += 128)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0x3c003c00u, 0, 0x3c003c00u, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t idesc = idesc_bf16(128, N, false, false);
  // D in columns [0, N); the TMEM A operand (ts) in columns [256, 320).
  // style 0: lane 0 alone runs the loop; style 1: the whole warp runs it and
  // one elected lane issues; both with the descriptors computed up front.
  uint64_t ad[4], bd[4];
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    ad[kk] = sdesc_sw128(base + kk * 32, 16384, 1024);
    bd[kk] = sdesc_sw128(base + 16384 + kk * 32, 32768, 1024);
  }
  long long t0 = 0, t1 = 0;
  if (style == 0) {
    if (threadIdx.x == 0) {
      t0 = clock64();
      for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          if constexpr (TS != 0)
            mma_ts(tmem, tmem + 256 + kk * 8, bd[kk], idesc, 1u);
          else
            mma_ss(tmem, ad[kk], bd[kk], idesc, 1u);
        }
      }
      tc_commit(bar);
    }
  } else if (warp == 0) {
    t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (elect_one()) {
          if constexpr (TS != 0)
            mma_ts(tmem, tmem + 256 + kk * 8, bd[kk], idesc, 1u);
          else
            mma_ss(tmem, ad[kk], bd[kk], idesc, 1u);
        }
        __syncwarp();
      }
    }
    if (elect_one()) tc_commit(bar);
    __syncwarp();
  }
  const WaitCtl wc{err, abort_flag, 2000000000ull};
  mbar_wait(bar, 0, wc, SITE_TEST);
  if (threadIdx.x == 0) {
    t1 = clock64();
    out[2 * blockIdx.x] = (double)(t1 - t0);
    out[2 * blockIdx.x + 1] = (double)iters * 4.0 * 2.0 * 128 * N * 16;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Issue-cost probe: SS N=128 MMAs in groups of 4, with optional extras after
// each group (mods bit 0: tcgen05 fence::after_thread_sync; bit 1: a commit to a
// spare mbarrier; bit 2: a try_wait on an already completed mbarrier; bit 3: a
// runtime accumulate flag on every MMA).
__global__ void __launch_bounds__(128, 1) micro_issue_kernel(int iters, int mods, double* out,
                                                             int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t bar = base + 65536, spare = bar + 8, done = bar + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 65536 + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 65536 + 72);
  const int warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < 65536 / 16; i += 128)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0x3c003c00u, 0, 0x3c003c00u, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(spare, 1);
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) mbar_arrive(done);   // phase 0 of `done` completes
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
  long long t0 = 0, t1 = 0;
  if (threadIdx.x == 0) {
    t0 = clock64();
    for (int it = 0; it < iters; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss(tmem, sdesc_sw128(base + kk * 32, 16384, 1024),
               sdesc_sw128(base + 16384 + kk * 32, 16384, 1024), idesc,
               (mods & 8) ? (uint32_t)(it > 0 || kk > 0) : 1u);
      if (mods & 1) tc_fence_after();
      if (mods & 2) tc_commit(spare);
      if (mods & 4) mbar_try_wait(done, 0);
    }
    tc_commit(bar);
  }
  const WaitCtl wc{err, abort_flag, 2000000000ull};
  mbar_wait(bar, 0, wc, SITE_TEST);
  if (threadIdx.x == 0) {
    t1 = clock64();
    out[2 * blockIdx.x] = (double)(t1 - t0);
    out[2 * blockIdx.x + 1] = (double)iters * 4.0 * 2.0 * 128 * 128 * 16;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Issue-style probe with the descriptors computed next to each MMA from a
// loop-varying stage offset (as the attention kernels do):
//   style 0: lane 0 alone runs the loop; 1: the converged warp runs it and an
//   elected lane issues; 2: lane 0, descriptors hoisted out of the loop.
template <int STYLE, int X>
__global__ void __launch_bounds__(128, 1) micro_style_kernel(int iters, double* out, int* err,
                                                             int one) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t bar = base + 65536, spare = bar + 8, done = bar + 16;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 65536 + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 65536 + 72);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 65536 / 16; i += 128)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0x3c003c00u, 0, 0x3c003c00u, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(spare, 1);
    mbar_init(done, 1);
    mbar_arrive(done);
    *abort_flag = 0;
    *reinterpret_cast<volatile int*>(smem + 65536 + 80) = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
  long long t0 = 0;
  if (warp == 0 && (STYLE == 1 || lane == 0 || X == 7)) {
    t0 = clock64();
    uint64_t ah[4], bh[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      ah[kk] = sdesc_sw128(base + kk * 32, 16384, 1024);
      bh[kk] = sdesc_sw128(base + 16384 + kk * 32, 16384, 1024);
    }
    for (int it = 0; it < iters; ++it) {
      const uint32_t stage = (it & 1) * 8192;   // loop-varying operand offset
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = STYLE == 2 ? ah[kk] : sdesc_sw128(base + stage + kk * 32, 16384, 1024);
        const uint64_t b =
            STYLE == 2 ? bh[kk] : sdesc_sw128(base + 16384 + stage + kk * 32, 16384, 1024);
        // X = 1: accumulate flag is a runtime value (always 1 here)
        const uint32_t acc = X == 1 ? (uint32_t)(one != 0) : 1u;
        if (STYLE == 1) {
          if (elect_one()) mma_ss(tmem, a, b, idesc, acc);
          __syncwarp();
        } else {
          mma_ss(tmem, a, b, idesc, acc);
        }
      }
      if (X == 2) tc_fence_after();
      if (X == 3) tc_commit(spare);
      if (X == 4) {
        const WaitCtl w2{err, abort_flag, 2000000000ull};
        mbar_wait(done, 0, w2, SITE_TEST);
      }
      if (X == 5) {   // bare try_wait on the completed phase
        while (!mbar_try_wait(done, 0)) {
        }
      }
      if (X == 6) {   // non-blocking test_wait on the completed phase
        while (!mbar_test_wait(done, 0)) {
        }
      }
      if (X == 7) {   // named-barrier handshake with warp 1
        asm volatile("bar.sync 1, 64;" ::: "memory");
      }
      if (X == 8) {   // plain shared-memory flag read
        while (*reinterpret_cast<volatile int*>(smem + 65536 + 80) != 0) {
        }
      }
      if (X == 9) {   // global-memory read
        while (*reinterpret_cast<volatile int*>(err) == 12345) {
        }
      }

    }
    if (STYLE == 1) {
      if (elect_one()) tc_commit(bar);
      __syncwarp();
    } else {
      tc_commit(bar);
    }
  }
  if (X == 7 && warp == 1) {
    for (int it = 0; it < iters; ++it) asm volatile("bar.sync 1, 64;" ::: "memory");
  }
  const WaitCtl wc{err, abort_flag, 2000000000ull};
  mbar_wait(bar, 0, wc, SITE_TEST);
  if (threadIdx.x == 0) {
    out[2 * blockIdx.x] = (double)(clock64() - t0);
    out[2 * blockIdx.x + 1] = (double)iters * 4.0 * 2.0 * 128 * 128 * 16;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Load latency seen by another warp while warp 0 streams MMAs (or not):
// OP 0 tcgen05.ld x32 (+wait), 1 ld.shared.v4, 2 mbarrier.test_wait; the probe
// warp is warp 4 (same SM sub-partition as warp 0) or warp 5 (another one).
template <int OP, int SAME, int MMA>
__global__ void __launch_bounds__(256, 1) micro_lat_kernel(int iters, double* out, int* err) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const uint32_t bar = base + 65536, done = bar + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 65536 + 64);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 65536 + 72);
  volatile int* stop = reinterpret_cast<volatile int*>(smem + 65536 + 76);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = threadIdx.x; i < 65536 / 16; i += 256)
    reinterpret_cast<uint4*>(smem)[i] = make_uint4(0x3c003c00u, 0, 0x3c003c00u, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    mbar_init(done, 1);
    mbar_arrive(done);
    *abort_flag = 0;
    *stop = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  constexpr uint32_t idesc = idesc_bf16(128, 256, false, false);
  const int probe_warp = SAME ? 4 : 5;
  if (warp == 0 && lane == 0 && MMA) {
    // stream MMAs (D in columns [0,256)) for a fixed number of groups
    for (int it = 0; it < iters * 4; ++it) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ss(tmem, sdesc_sw128(base + kk * 32, 16384, 1024),
               sdesc_sw128(base + 16384 + kk * 32, 32768, 1024), idesc, 1u);
    }
    tc_commit(bar);
  }
  if (warp == probe_warp) {
    // probes on TMEM columns [256, 288) of this warp's lane quarter
    const uint32_t taddr = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 256;
    uint32_t acc = 0;
    const long long t0 = clock64();
    for (int it = 0; it < iters; ++it) {
      if (OP == 0) {
        uint32_t r[32];
        tmem_ld32(taddr, r);
        acc += r[lane & 31];
      } else if (OP == 1) {
        uint32_t v;
        asm volatile("ld.volatile.shared.u32 %0, [%1];"
                     : "=r"(v)
                     : "r"(base + 40960 + ((it * 16 + lane * 16) & 8191))
                     : "memory");
        acc += v;
      } else {
        acc += mbar_test_wait(done, 0) ? 1u : 0u;
      }
    }
    const long long t1 = clock64();
    if (lane == 0) {
      out[2 * blockIdx.x] = (double)(t1 - t0);
      out[2 * blockIdx.x + 1] = (double)iters;   // "ops" = probes; rate = probes per clock
    }
    if (acc == 0xdeadbeef) out[0] = 0;
  }
  if (MMA) {
    const WaitCtl wc{err, abort_flag, 4000000000ull};
    mbar_wait(bar, 0, wc, SITE_TEST);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_micro(int kind, int iters, double* out, int ctas, cudaStream_t st) {
  if (kind >= 40 && kind <= 51) {
    const int k = kind - 40, op = k / 4, same = (k >> 1) & 1, mma = k & 1;
    void (*kern)(int, double*, int*) =
        op == 0 ? (same ? (mma ? micro_lat_kernel<0, 1, 1> : micro_lat_kernel<0, 1, 0>)
                        : (mma ? micro_lat_kernel<0, 0, 1> : micro_lat_kernel<0, 0, 0>))
      : op == 1 ? (same ? (mma ? micro_lat_kernel<1, 1, 1> : micro_lat_kernel<1, 1, 0>)
                        : (mma ? micro_lat_kernel<1, 0, 1> : micro_lat_kernel<1, 0, 0>))
                : (same ? (mma ? micro_lat_kernel<2, 1, 1> : micro_lat_kernel<2, 1, 0>)
                        : (mma ? micro_lat_kernel<2, 0, 1> : micro_lat_kernel<2, 0, 0>));
    const int smem = 65536 + 128 + 1024;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<ctas, 256, smem, st>>>(iters, out, device_error_word());
    return cudaGetLastError();
  }
  if (kind >= 28 && kind <= 39) {
    // 28-30: styles 0/1/2; 31-39: style 0 with extras X = 1..9 per group of 4
    const int smem = 65536 + 128 + 1024;
    void (*kern)(int, double*, int*, int) =
        kind == 28 ? micro_style_kernel<0, 0> : kind == 29 ? micro_style_kernel<1, 0>
        : kind == 30 ? micro_style_kernel<2, 0> : kind == 31 ? micro_style_kernel<0, 1>
        : kind == 32 ? micro_style_kernel<0, 2> : kind == 33 ? micro_style_kernel<0, 3>
        : kind == 34 ? micro_style_kernel<0, 4> : kind == 35 ? micro_style_kernel<0, 5>
        : kind == 36 ? micro_style_kernel<0, 6> : kind == 37 ? micro_style_kernel<1, 7>
        : kind == 38 ? micro_style_kernel<0, 8> : micro_style_kernel<0, 9>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<ctas, 128, smem, st>>>(iters, out, device_error_word(), 1);
    return cudaGetLastError();
  }
  if (kind >= 12 && kind <= 27) {
    const int smem = 65536 + 128 + 1024;
    cudaError_t e = cudaFuncSetAttribute(micro_issue_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    micro_issue_kernel<<<ctas, 128, smem, st>>>(iters, kind - 12, out, device_error_word());
    return cudaGetLastError();
  }
  if (kind == 0 || kind == 1) {
    micro_exp_kernel<<<ctas, 256, 0, st>>>(iters, kind, out, 0.37f);
    return cudaGetLastError();
  }
  if (kind >= 2 && kind <= 11) {
    // 2: N=256 SS, 3: N=128 SS, 4: N=64 SS, 5: N=128 A-in-TMEM, 6: N=64 A-in-TMEM;
    // 7-11: the same shapes issued by an elected lane of a converged warp
    const int style = kind >= 7 ? 1 : 0;
    const int k5 = (kind - 2) % 5;
    const int smem = 65536 + 128 + 1024;
    void (*kern)(int, int, double*, int*) =
        k5 == 0 ? micro_mma_kernel<256, 0> : k5 == 1 ? micro_mma_kernel<128, 0>
        : k5 == 2 ? micro_mma_kernel<64, 0> : k5 == 3 ? micro_mma_kernel<128, 1>
                                             : micro_mma_kernel<64, 1>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kern<<<ctas, 128, smem, st>>>(iters, style, out, device_error_word());
    return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
