// FP8 (e4m3) quantization of attention inputs for the FP8 forward.
//
// The FlashAttention-4 pages name the low-precision lineage only through the
// title of FlashAttention-3 ("Fast and Accurate Attention with Asynchrony and
// Low Precision", the pages' reference lists); the scaling granularity here is
// this library's reading:
//   Q, K: one scale per (sequence, head, block of 128 rows) over the block's
//         rows and all d columns; codes keep the [B, S, H, d] layout.
//   V:    one scale per (sequence, head) over all rows; codes are written
//         transposed, [B, H, d, S_pad] with the keys contiguous (S_pad = S
//         rounded up to 16, the pad holding zero codes), so that V^T is a
//         K-major operand of the P V product.
// scale = amax / 448 (the largest e4m3 value), 1 when amax = 0; code =
// e4m3(x * r) with r = 1 / scale (one float32 division per block, a multiply
// per element), rounded to nearest even with saturation, all in float32.
// HBM-bound: Q and K are read once and their codes written once; V is read
// twice (its per-head amax first) and its codes written once, transposed
// through shared memory.
#include "internal.h"

#include <cuda_fp8.h>

namespace fa {
namespace quant {

constexpr int ROWS = 128;       // rows (keys) per scale block / per transpose tile
constexpr int THREADS = 256;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ float amax8(const uint4& v) {
  float m = fmaxf(fabsf(bf16_lo(v.x)), fabsf(bf16_hi(v.x)));
  m = fmaxf(m, fmaxf(fabsf(bf16_lo(v.y)), fabsf(bf16_hi(v.y))));
  m = fmaxf(m, fmaxf(fabsf(bf16_lo(v.z)), fabsf(bf16_hi(v.z))));
  return fmaxf(m, fmaxf(fabsf(bf16_lo(v.w)), fabsf(bf16_hi(v.w))));
}

__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// eight bf16 values * rs -> eight e4m3 codes (first value in the lowest byte);
// __fmul_rn keeps each product a plain rounded multiply (never fused)
__device__ __forceinline__ uint2 quant8(const uint4& v, float rs) {
  uint2 r;
  r.x = e4m3x2(__fmul_rn(bf16_lo(v.x), rs), __fmul_rn(bf16_hi(v.x), rs)) |
        (e4m3x2(__fmul_rn(bf16_lo(v.y), rs), __fmul_rn(bf16_hi(v.y), rs)) << 16);
  r.y = e4m3x2(__fmul_rn(bf16_lo(v.z), rs), __fmul_rn(bf16_hi(v.z), rs)) |
        (e4m3x2(__fmul_rn(bf16_lo(v.w), rs), __fmul_rn(bf16_hi(v.w), rs)) << 16);
  return r;
}

__device__ __forceinline__ float block_max(float m, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  float r = red[0];
#pragma unroll
  for (int w = 1; w < THREADS / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float scale_of(float amax) { return amax > 0.f ? amax / 448.f : 1.f; }

// Q / K: grid (row blocks, H, B). Each thread keeps its share of the block's
// 16-byte vectors in registers between the two steps.
template <int D>
__global__ void __launch_bounds__(THREADS) quant_rows_kernel(const __nv_bfloat16* x, int S, int H,
                                                             uint8_t* codes, float* scales) {
  constexpr int VPR = D / 8;                               // vectors per row
  constexpr int PER = ROWS * VPR / THREADS;                // vectors per thread
  __shared__ float red[THREADS / 32];
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int r0 = blk * ROWS;
  const int nrows = S - r0 < ROWS ? S - r0 : ROWS;
  uint4 v[PER];
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = i * THREADS + threadIdx.x;
    const int r = idx / VPR, c = (idx % VPR) * 8;
    v[i] = make_uint4(0, 0, 0, 0);
    if (r < nrows) {
      v[i] = *reinterpret_cast<const uint4*>(x + (((long long)b * S + r0 + r) * H + h) * D + c);
      m = fmaxf(m, amax8(v[i]));
    }
  }
  const float s = scale_of(block_max(m, red));
  const float rs = 1.f / s;
  if (threadIdx.x == 0) scales[((long long)b * H + h) * gridDim.x + blk] = s;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = i * THREADS + threadIdx.x;
    const int r = idx / VPR, c = (idx % VPR) * 8;
    if (r < nrows)
      *reinterpret_cast<uint2*>(codes + (((long long)b * S + r0 + r) * H + h) * D + c) = quant8(v[i], rs);
  }
}

// V, step 1: per-(sequence, head) amax into vmax (zeroed beforehand) as the
// bits of a non-negative float, whose integer order is the float order.
template <int D>
__global__ void __launch_bounds__(THREADS) v_amax_kernel(const __nv_bfloat16* x, int S, int H,
                                                         unsigned* vmax) {
  constexpr int VPR = D / 8;
  constexpr int PER = ROWS * VPR / THREADS;
  __shared__ float red[THREADS / 32];
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int r0 = blk * ROWS;
  const int nrows = S - r0 < ROWS ? S - r0 : ROWS;
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = i * THREADS + threadIdx.x;
    const int r = idx / VPR, c = (idx % VPR) * 8;
    if (r < nrows)
      m = fmaxf(m, amax8(*reinterpret_cast<const uint4*>(x + (((long long)b * S + r0 + r) * H + h) * D + c)));
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) atomicMax(vmax + (long long)b * H + h, __float_as_uint(m));
}

// V, step 2: quantize a tile of 128 keys and write it transposed, keys
// contiguous; keys in [S, S_pad) get zero codes. grid (key tiles, H, B).
template <int D>
__global__ void __launch_bounds__(THREADS) v_quant_t_kernel(const __nv_bfloat16* x, int S, int H,
                                                            int S_pad, const unsigned* vmax,
                                                            uint8_t* codes_t) {
  constexpr int VPR = D / 8;
  constexpr int PER = ROWS * VPR / THREADS;
  constexpr int TS = ROWS + 16;                            // tile row stride (bytes), 16-aligned
  __shared__ __align__(16) uint8_t tile[D * TS];
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int k0 = blk * ROWS;
  const int nrows = S - k0 < ROWS ? S - k0 : ROWS;
  const float rs = 1.f / scale_of(__uint_as_float(vmax[(long long)b * H + h]));
  // lanes take consecutive keys of one 8-column group, so a warp's byte
  // writes into each tile row land in 32 consecutive bytes (no bank conflict)
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    const int idx = i * THREADS + threadIdx.x;
    const int r = idx % ROWS, c = (idx / ROWS) * 8;
    uint2 q = make_uint2(0, 0);
    if (r < nrows)
      q = quant8(*reinterpret_cast<const uint4*>(x + (((long long)b * S + k0 + r) * H + h) * D + c), rs);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      tile[(c + e) * TS + r] = (uint8_t)(((e < 4 ? q.x : q.y) >> (8 * (e & 3))) & 0xffu);
  }
  __syncthreads();
  // row c of the tile -> codes_t[b][h][c][k0 .. k0 + 128), 16 bytes at a time, up to S_pad
  const int nvec = (S_pad - k0 < ROWS ? S_pad - k0 : ROWS) / 16;
  uint8_t* dst = codes_t + (((long long)b * H + h) * D) * S_pad + k0;
  for (int i = threadIdx.x; i < D * (ROWS / 16); i += THREADS) {
    const int c = i / (ROWS / 16), vq = i % (ROWS / 16);
    if (vq < nvec)
      *reinterpret_cast<uint4*>(dst + (long long)c * S_pad + vq * 16) =
          *reinterpret_cast<const uint4*>(tile + c * TS + vq * 16);
  }
}

// V, step 3: amax -> scale, in place (after step 2 has read the amax values).
__global__ void v_scale_kernel(unsigned* vmax_scales, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    const float s = scale_of(__uint_as_float(vmax_scales[i]));
    reinterpret_cast<float*>(vmax_scales)[i] = s;
  }
}

template <int D>
cudaError_t launch_d(const __nv_bfloat16* x, int B, int S, int H, int layout, uint8_t* codes,
                     float* scales, cudaStream_t st) {
  const dim3 grid((S + ROWS - 1) / ROWS, H, B);
  if (layout == 0) {
    quant_rows_kernel<D><<<grid, THREADS, 0, st>>>(x, S, H, codes, scales);
    return cudaGetLastError();
  }
  unsigned* vmax = reinterpret_cast<unsigned*>(scales);
  cudaError_t e = cudaMemsetAsync(vmax, 0, (size_t)B * H * sizeof(unsigned), st);
  if (e != cudaSuccess) return e;
  v_amax_kernel<D><<<grid, THREADS, 0, st>>>(x, S, H, vmax);
  const int S_pad = (S + 15) / 16 * 16;
  v_quant_t_kernel<D><<<grid, THREADS, 0, st>>>(x, S, H, S_pad, vmax, codes);
  v_scale_kernel<<<(B * H + 255) / 256, 256, 0, st>>>(vmax, B * H);
  return cudaGetLastError();
}

}  // namespace quant

cudaError_t launch_quantize_fp8(const __nv_bfloat16* x, int B, int S, int H, int d, int layout,
                                uint8_t* codes, float* scales, cudaStream_t st) {
  if (B == 0 || S == 0) return cudaSuccess;
  if (d == 128) return quant::launch_d<128>(x, B, S, H, layout, codes, scales, st);
  if (d == 64) return quant::launch_d<64>(x, B, S, H, layout, codes, scales, st);
  return cudaErrorInvalidValue;
}

}  // namespace fa
