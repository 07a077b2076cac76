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
// LSE = +inf. Memory-bound: a group of d/8 lanes per (row, head), each lane
// moving 16 bytes per part; items run with the row index fastest, the order
// of both LSE layouts, so their LSE reads are contiguous.
#include "internal.h"
#include "ptx.cuh"

#include <cmath>

namespace fa {
using ptx::pack_bf16x2;

namespace {

constexpr int MAX_PARTS = 64;
constexpr int THREADS = 256;

__device__ __forceinline__ void add8(float (&acc)[8], float w, const uint4& v) {
  const uint32_t x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    acc[2 * i] = fmaf(w, __uint_as_float(x[i] << 16), acc[2 * i]);
    acc[2 * i + 1] = fmaf(w, __uint_as_float(x[i] & 0xffff0000u), acc[2 * i + 1]);
  }
}

// LPI lanes per item (a power of two >= d / 8); lane `sub` owns columns
// [8 sub, 8 sub + 8). Item i: dense (b, h, s) = (i / (Hq S), i / S % Hq, i % S),
// packed (h, t) = (i / T, i % T); its LSE entry is i in both layouts.
template <int LPI>
__global__ void __launch_bounds__(THREADS) merge_kernel(const __nv_bfloat16* __restrict__ o_parts,
                                                        const float* __restrict__ lse_parts, int P,
                                                        long long rows, int Hq, int S, int d,
                                                        int packed, __nv_bfloat16* __restrict__ o,
                                                        float* __restrict__ lse) {
  constexpr int IPB = THREADS / LPI;
  const int sub = threadIdx.x % LPI;
  const bool active = sub * 8 < d;
  const long long items = rows * Hq, part_o = rows * Hq * d;
  for (long long i = (long long)blockIdx.x * IPB + threadIdx.x / LPI; i < items;
       i += (long long)gridDim.x * IPB) {
    long long t;
    int h;
    if (packed) {
      h = (int)(i / rows);
      t = i - (long long)h * rows;
    } else {
      const long long bh = i / S;
      t = (bh / Hq) * S + (i - bh * S);
      h = (int)(bh % Hq);
    }
    float m = -INFINITY;
    for (int q = 0; q < P; ++q) {
      const float l = lse_parts[q * items + i];
      if (l != INFINITY) m = fmaxf(m, l);
    }
    const long long orow = (t * Hq + h) * d + sub * 8;
    if (m == -INFINITY) {                                // no key in any part
      if (active) *reinterpret_cast<uint4*>(o + orow) = make_uint4(0, 0, 0, 0);
      if (sub == 0) lse[i] = INFINITY;
      continue;
    }
    float wsum = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int q = 0;
    for (; q + 4 <= P; q += 4) {                         // four parts' loads in flight
      float w[4];
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const float l = lse_parts[(q + u) * items + i];
        w[u] = l == INFINITY ? 0.f : expf(l - m);
        v[u] = active && l != INFINITY
                   ? *reinterpret_cast<const uint4*>(o_parts + (q + u) * part_o + orow)
                   : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {                   // a part without keys adds 0 * 0
        wsum += w[u];
        add8(acc, w[u], v[u]);
      }
    }
    for (; q < P; ++q) {
      const float l = lse_parts[q * items + i];
      if (l == INFINITY) continue;
      const float w = expf(l - m);
      wsum += w;
      add8(acc, w, active ? *reinterpret_cast<const uint4*>(o_parts + q * part_o + orow)
                          : make_uint4(0, 0, 0, 0));
    }
    if (active) {
      const float inv = 1.0f / wsum;
      uint4 r;
      r.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      r.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
      r.z = pack_bf16x2(acc[4] * inv, acc[5] * inv);
      r.w = pack_bf16x2(acc[6] * inv, acc[7] * inv);
      *reinterpret_cast<uint4*>(o + orow) = r;
    }
    if (sub == 0) lse[i] = m + logf(wsum);
  }
}

template <int LPI>
cudaError_t launch_lpi(const __nv_bfloat16* o_parts, const float* lse_parts, int P,
                       long long rows, int Hq, int S, int d, int packed, __nv_bfloat16* o,
                       float* lse, cudaStream_t stream) {
  constexpr int IPB = THREADS / LPI;
  const long long items = rows * Hq;
  const long long want = (items + IPB - 1) / IPB;
  const int blocks = (int)(want < 152 * 16 ? want : 152 * 16);
  merge_kernel<LPI><<<blocks, THREADS, 0, stream>>>(o_parts, lse_parts, P, rows, Hq, S, d, packed,
                                                    o, lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge(const __nv_bfloat16* o_parts, const float* lse_parts, int P,
                         long long rows, int Hq, int S, int d, int packed, __nv_bfloat16* o,
                         float* lse, cudaStream_t stream) {
  if (P < 1 || P > MAX_PARTS || d % 64 != 0 || d > 256) return cudaErrorInvalidValue;
  if (rows * Hq == 0) return cudaSuccess;
  if (d == 64) return launch_lpi<8>(o_parts, lse_parts, P, rows, Hq, S, d, packed, o, lse, stream);
  if (d == 128) return launch_lpi<16>(o_parts, lse_parts, P, rows, Hq, S, d, packed, o, lse, stream);
  return launch_lpi<32>(o_parts, lse_parts, P, rows, Hq, S, d, packed, o, lse, stream);
}

}  // namespace fa
