// Merge of attention results computed over disjoint key sets for the same
// queries (the combine step of context parallelism: K/V split into shards,
// each shard's forward run separately). With part p's row result O_p and
// log-sum-exp LSE_p,
//     LSE = log sum_p exp(LSE_p),    O = sum_p exp(LSE_p - LSE) O_p,
// which is exactly the attention over the union of the key sets: the softmax
// normaliser of the union is the sum of the parts' normalisers. This is the
// same rescale-and-accumulate step the online softmax applies between KV
// blocks ("FlashAttention-4 Conquers Asymmetric GPU Hardware Scaling",
// episode description: tiling with an online softmax), applied across parts,
// as blockwise attention across devices does (the same page's source list,
// entry 14: Ring Attention with Blockwise Transformers).
// A row that saw no key in a part has LSE_p = +inf and O_p = 0 (the forward's
// convention) and counts zero; a row that saw no key in any part gets O = 0,
// LSE = +inf. Memory-bound: one warp per (row, head).
#include "internal.h"
#include "ptx.cuh"

#include <cmath>

namespace fa {

namespace {

constexpr int MAX_PARTS = 64;

__global__ void merge_kernel(const __nv_bfloat16* __restrict__ o_parts,
                             const float* __restrict__ lse_parts, int P, long long rows, int Hq,
                             int S, int d, int packed, __nv_bfloat16* __restrict__ o,
                             float* __restrict__ lse) {
  const int lane = threadIdx.x & 31;
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  const long long part_o = rows * Hq * d, part_l = rows * Hq;
  for (long long rh = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
       rh < rows * Hq; rh += warps) {
    const long long t = rh / Hq;
    const int h = (int)(rh % Hq);
    // the forward's LSE layout: dense [B][Hq][S], packed [Hq][T]
    const long long li = packed ? (long long)h * rows + t
                                : ((t / S) * Hq + h) * (long long)S + (t % S);
    float m = -INFINITY;
    for (int q = lane; q < P; q += 32) {
      const float l = lse_parts[q * part_l + li];
      if (l != INFINITY) m = fmaxf(m, l);
    }
    for (int sh = 16; sh > 0; sh >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, sh));
    __nv_bfloat16* orow = o + rh * d;
    if (m == -INFINITY) {                                // no key in any part
      for (int c = lane; c < d; c += 32) orow[c] = __float2bfloat16(0.f);
      if (lane == 0) lse[li] = INFINITY;
      continue;
    }
    float wsum = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // columns lane + 32e (d <= 256)
    for (int q = 0; q < P; ++q) {
      const float l = lse_parts[q * part_l + li];
      if (l == INFINITY) continue;
      const float wq = expf(l - m);
      wsum += wq;
      const __nv_bfloat16* prow = o_parts + q * part_o + rh * d;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int c = lane + 32 * e;
        if (c < d) acc[e] = fmaf(wq, __bfloat162float(prow[c]), acc[e]);
      }
    }
    const float inv = 1.0f / wsum;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int c = lane + 32 * e;
      if (c < d) orow[c] = __float2bfloat16(acc[e] * inv);
    }
    if (lane == 0) lse[li] = m + logf(wsum);
  }
}

}  // namespace

cudaError_t launch_merge(const __nv_bfloat16* o_parts, const float* lse_parts, int P,
                         long long rows, int Hq, int S, int d, int packed, __nv_bfloat16* o,
                         float* lse, cudaStream_t stream) {
  if (P < 1 || P > MAX_PARTS) return cudaErrorInvalidValue;
  const long long items = rows * Hq;
  if (items == 0) return cudaSuccess;
  const long long want = (items + 7) / 8;
  const int blocks = (int)(want < 152 * 32 ? want : 152 * 32);
  merge_kernel<<<blocks, 256, 0, stream>>>(o_parts, lse_parts, P, rows, Hq, S, d, packed, o, lse);
  return cudaGetLastError();
}

}  // namespace fa
