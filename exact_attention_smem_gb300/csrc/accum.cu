// Gradient accumulation across parts: a backward split over disjoint key
// shards (context parallelism) yields, per shard, partial dQ of the queries
// and the shard's own dK, dV; the gradients are their sums. This is the
// cross-shard counterpart of the accumulation of dQ over key blocks inside the
// backward ("FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", abstract item (3): the backward's dQ
// accumulation). Sums are kept in fp32; partials arrive in bf16 (the
// backward's output type). Memory-bound: 16-byte vectors, a grid-stride loop
// over groups of 8 elements.
#include "internal.h"
#include "ptx.cuh"

namespace fa {
using ptx::pack_bf16x2;

namespace {

constexpr int THREADS = 256;

__global__ void __launch_bounds__(THREADS)
    accumulate_kernel(float* __restrict__ acc, const __nv_bfloat16* __restrict__ x, long long n8) {
  for (long long i = (long long)blockIdx.x * THREADS + threadIdx.x; i < n8;
       i += (long long)gridDim.x * THREADS) {
    const uint4 v = reinterpret_cast<const uint4*>(x)[i];
    float4* a4 = reinterpret_cast<float4*>(acc) + 2 * i;
    float4 a = a4[0], b = a4[1];
    a.x += __uint_as_float(v.x << 16);
    a.y += __uint_as_float(v.x & 0xffff0000u);
    a.z += __uint_as_float(v.y << 16);
    a.w += __uint_as_float(v.y & 0xffff0000u);
    b.x += __uint_as_float(v.z << 16);
    b.y += __uint_as_float(v.z & 0xffff0000u);
    b.z += __uint_as_float(v.w << 16);
    b.w += __uint_as_float(v.w & 0xffff0000u);
    a4[0] = a;
    a4[1] = b;
  }
}

__global__ void __launch_bounds__(THREADS)
    to_bf16_kernel(__nv_bfloat16* __restrict__ out, const float* __restrict__ in, long long n8) {
  for (long long i = (long long)blockIdx.x * THREADS + threadIdx.x; i < n8;
       i += (long long)gridDim.x * THREADS) {
    const float4 a = reinterpret_cast<const float4*>(in)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(in)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16x2(a.x, a.y);
    o.y = pack_bf16x2(a.z, a.w);
    o.z = pack_bf16x2(b.x, b.y);
    o.w = pack_bf16x2(b.z, b.w);
    reinterpret_cast<uint4*>(out)[i] = o;
  }
}

int grid_for(long long n8) {
  const long long sms = num_sms() > 0 ? num_sms() : 152;
  long long g = (n8 + THREADS - 1) / THREADS;
  const long long cap = sms * 8;                       // a few waves of 256-thread blocks
  return (int)(g < cap ? (g > 0 ? g : 1) : cap);
}

}  // namespace

cudaError_t launch_accumulate(float* acc, const __nv_bfloat16* x, long long n,
                              cudaStream_t stream) {
  const long long n8 = n / 8;
  accumulate_kernel<<<grid_for(n8), THREADS, 0, stream>>>(acc, x, n8);
  return cudaGetLastError();
}

cudaError_t launch_to_bf16(__nv_bfloat16* out, const float* in, long long n, cudaStream_t stream) {
  const long long n8 = n / 8;
  to_bf16_kernel<<<grid_for(n8), THREADS, 0, stream>>>(out, in, n8);
  return cudaGetLastError();
}

}  // namespace fa
