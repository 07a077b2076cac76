// FP8 (e4m3) forward for sm_103a: O = softmax(scale * Q^ K^T [+ causal mask]) V^
// and the fp32 row log-sum-exp, where Q^, K^, V^ are the dequantized inputs
// (e4m3 codes times per-block scales, written by the quantize kernels).
//
// Same method and pipeline as the bf16 forward (FlashAttention-4 pages:
// "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for Asymmetric
// Hardware Scaling", abstract items (1) and (2); the low-precision lineage is
// named by the FlashAttention-3 title in the pages' reference lists): a
// persistent CTA per SM, a TMA producer warp, one MMA-issuing thread, two
// softmax warpgroups in ping-pong over two 128-row query tiles, an online
// softmax with rescaling and an LPT schedule. The differences:
//   * both products run as tcgen05 kind::f8f6f4 MMAs (32 K elements per
//     instruction, K-major operands only: V arrives transposed, keys
//     contiguous, so V^T is the K-major B operand of P V);
//   * the block scales enter the softmax: S_raw (the exact fp32 sum of code
//     products) times scale * log2(e) * q_scale(tile) * k_scale(block);
//   * P is written to TMEM as e4m3, four weights per column, as 2^7 * p
//     relative to the row's reference maximum: weights down to 2^-13 of it
//     keep three mantissa bits instead of falling into e4m3's subnormals,
//     and with the rescale threshold tau clamped to 1.5 (base 2) the largest
//     weight, 2^(7 + tau) <= 362, stays below e4m3's 448; the row sum l is
//     taken over the same fp32 weights, the LSE removes the factor, and
//     O = O_acc * v_scale / l.
// Head dim 128, dense [B, S, H, d] layouts (no packed sequences).
#include "exp2_poly.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

#include <cuda_fp8.h>

#include <cmath>

namespace fa {
using namespace ptx;

namespace fwd8 {

constexpr int D = 128;
constexpr int BM = 128;         // query rows per tile
constexpr int BN = 128;         // keys per KV block
constexpr int UNIT_ROWS = 2 * BM;
constexpr int NUM_THREADS = 384;
constexpr int MMA_WARP = 8;
constexpr int TMA_WARP = 9;
constexpr int REGS_SOFTMAX = 192;
constexpr int REGS_CONTROL = 112;
constexpr float P_LOG2_OFFSET = 7.f;  // weights stored as 2^7 * p
constexpr float TAU_MAX = 1.5f;       // 2^(7 + 1.5) = 362 < 448

struct Cfg {
  static constexpr int TILE_BYTES = 128 * 128;          // 128 rows x 128 one-byte elements
  static constexpr int NSTAGE = 8;
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = 2 * TILE_BYTES;
  static constexpr int BAR_OFF = KV_OFF + NSTAGE * TILE_BYTES;
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KVFULL = 2, B_KVEMPTY = 2 + NSTAGE,
                       B_SFULL = 2 + 2 * NSTAGE, B_PFULL = B_SFULL + 2, B_OFULL = B_PFULL + 2,
                       B_DRAIN = B_OFULL + 2, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  // O write-out staging (bf16, 128B swizzle): per softmax warpgroup its whole
  // tile, two 128-row x 64-column chunks
  static constexpr int OCHUNK_BYTES = 128 * 128;
  static constexpr int OCHUNKS = D / 64;
  static constexpr int STAGE_OFF = (MISC_OFF + 16 + 1023) & ~1023;
  static constexpr int SMEM_BYTES = STAGE_OFF + 2 * OCHUNKS * OCHUNK_BYTES + 1024;
  static_assert(SMEM_BYTES <= 232448, "FP8 forward shared memory");
  static constexpr uint32_t IDESC_S = idesc_e4m3(128, 128);
  static constexpr uint32_t IDESC_PV = idesc_e4m3(128, D);
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_O = 256;
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// S (TMEM, 128x128 fp32) = Q_tile (128 x 128 codes) * K_block^T; both K-major.
__device__ __forceinline__ void issue_s(uint32_t tm_s, uint32_t q_tile, uint32_t k_tile) {
#pragma unroll
  for (int kk = 0; kk < D / 32; ++kk)
    mma_ss_f8(tm_s, sdesc_sw128(q_tile + kk * 32, Cfg::TILE_BYTES, 1024),
              sdesc_sw128(k_tile + kk * 32, Cfg::TILE_BYTES, 1024), Cfg::IDESC_S, kk > 0 ? 1u : 0u);
}

// O (TMEM, 128 x D fp32) (+)= P (TMEM, 128 x 128 e4m3) * V_block, with the B
// operand V^T (D rows x 128 keys, K-major).
__device__ __forceinline__ void issue_pv(uint32_t tm_o, uint32_t tm_p, uint32_t vt_tile,
                                         bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < BN / 32; ++kk)
    mma_ts_f8(tm_o, tm_p + kk * 8, sdesc_sw128(vt_tile + kk * 32, Cfg::TILE_BYTES, 1024),
              Cfg::IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

template <int POLY8>
__global__ void __launch_bounds__(NUM_THREADS, 1) fwd_fp8_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t bars = base + C::BAR_OFF;
#define BAR(i) (bars + 8u * (uint32_t)(i))
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_QFULL), 1);
    mbar_init(BAR(C::B_QEMPTY), 1);
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(BAR(C::B_KVFULL + s), 1);
      mbar_init(BAR(C::B_KVEMPTY + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(C::B_SFULL + t), 1);
      mbar_init(BAR(C::B_PFULL + t), BM);
      mbar_init(BAR(C::B_OFULL + t), 1);
    }
    mbar_init(BAR(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
    tma_prefetch_desc(&p.tm_o);
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const SchedSpec spec{nullptr, p.nseq, p.Sq, p.Sk, p.Hq, p.causal, UNIT_ROWS, BN, 0, p.hblock};
  const WaitCtl wc{p.err, abort_flag, p.timeout_ns};
  const int G = gridDim.x;
  const int cta = blockIdx.x;
  const int group = p.Hq / p.Hkv;

  if (warp >= 8) {
    regs_dec<REGS_CONTROL>();
  if (warp >= 10) {
    // spare warps of the control warpgroup
  } else if (warp == TMA_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Walker w;
      w.init(spec);
      uint32_t kv_it = 0;
      int u_it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        const int n = u.cost;
        if (n == 0) continue;
        const int kvh = u.head / group;
        const int q_row = u.q_start + u.m * UNIT_ROWS;
        if (u_it > 0) {
          ok = mbar_wait(BAR(C::B_QEMPTY), (u_it - 1) & 1, wc, SITE_FWD_Q_EMPTY);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(BAR(C::B_QFULL), 2 * C::TILE_BYTES);
        for (int t = 0; t < 2; ++t)
          tma_load_3d(base + C::Q_OFF + t * C::TILE_BYTES, &p.tm_q, BAR(C::B_QFULL), 0, u.head,
                      q_row + t * BM);
        ++u_it;
        for (int j = 0; j < n && ok; ++j) {
          for (int which = 0; which < 2; ++which) {
            const int s = kv_it % C::NSTAGE;
            const uint32_t rnd = kv_it / C::NSTAGE;
            if (rnd > 0) {
              ok = mbar_wait(BAR(C::B_KVEMPTY + s), (rnd - 1) & 1, wc, SITE_FWD_KV_EMPTY);
              if (!ok) break;
            }
            mbar_arrive_expect_tx(BAR(C::B_KVFULL + s), C::TILE_BYTES);
            const uint32_t dst = base + C::KV_OFF + s * C::TILE_BYTES;
            if (which == 0)        // K rows [k_start + j*BN, +128) of KV head kvh
              tma_load_3d(dst, &p.tm_k, BAR(C::B_KVFULL + s), 0, kvh, u.k_start + j * BN);
            else                   // V^T: all D rows, keys [j*BN, +128) of (sequence, kvh)
              tma_load_3d(dst, &p.tm_v, BAR(C::B_KVFULL + s), j * BN, 0, u.seq * p.Hkv + kvh);
            ++kv_it;
          }
        }
      }
      if (!ok) {
        for (uint32_t i = kv_it > (uint32_t)C::NSTAGE ? kv_it - C::NSTAGE : 0; i < kv_it; ++i)
          drain_wait(BAR(C::B_KVFULL + i % C::NSTAGE), (i / C::NSTAGE) & 1, 100000000ull);
        if (u_it > 0) drain_wait(BAR(C::B_QFULL), (u_it - 1) & 1, 100000000ull);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      Walker w;
      w.init(spec);
      uint32_t kv_it = 0, sp_it = 0;
      int u_it = 0;
      bool ok = true;
      const uint32_t q0 = base + C::Q_OFF, q1 = q0 + C::TILE_BYTES, kvb = base + C::KV_OFF;
      const uint32_t tS0 = tmem + C::TM_S, tS1 = tS0 + 128;
      const uint32_t tO0 = tmem + C::TM_O, tO1 = tO0 + D;
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        const int n = u.cost;
        if (n == 0) continue;
        ok = mbar_wait(BAR(C::B_QFULL), u_it & 1, wc, SITE_FWD_Q_FULL);
        if (!ok) break;
        ++u_it;
        int sk = kv_it % C::NSTAGE;
        ok = mbar_wait(BAR(C::B_KVFULL + sk), (kv_it / C::NSTAGE) & 1, wc, SITE_FWD_KV_FULL);
        if (!ok) break;
        tc_fence_after();
        issue_s(tS0, q0, kvb + sk * C::TILE_BYTES);
        tc_commit(BAR(C::B_SFULL + 0));
        issue_s(tS1, q1, kvb + sk * C::TILE_BYTES);
        tc_commit(BAR(C::B_SFULL + 1));
        tc_commit(BAR(C::B_KVEMPTY + sk));
        ++kv_it;
        if (n == 1) tc_commit(BAR(C::B_QEMPTY));
        for (int j = 0; j < n; ++j) {
          // sync point 1: V_j, P_0(j) and (if any) K_{j+1}
          const int sv = kv_it % C::NSTAGE;
          const bool more = j + 1 < n;
          const int sk2 = (kv_it + 1) % C::NSTAGE;
          ok = mbar_wait3(BAR(C::B_KVFULL + sv), (kv_it / C::NSTAGE) & 1, SITE_FWD_KV_FULL,
                          BAR(C::B_PFULL + 0), sp_it & 1, SITE_FWD_P_FULL,
                          more ? BAR(C::B_KVFULL + sk2) : BAR(C::B_KVFULL + sv),
                          more ? ((kv_it + 1) / C::NSTAGE) & 1 : (kv_it / C::NSTAGE) & 1,
                          SITE_FWD_KV_FULL, wc);
          if (!ok) break;
          ++kv_it;
          tc_fence_after();
          issue_pv(tO0, tS0, kvb + sv * C::TILE_BYTES, j > 0);
          if (more) {
            issue_s(tS0, q0, kvb + sk2 * C::TILE_BYTES);
            tc_commit(BAR(C::B_SFULL + 0));
          } else {
            tc_commit(BAR(C::B_OFULL + 0));
          }
          // sync point 2: P_1(j)
          ok = mbar_wait(BAR(C::B_PFULL + 1), sp_it & 1, wc, SITE_FWD_P_FULL);
          if (!ok) break;
          tc_fence_after();
          issue_pv(tO1, tS1, kvb + sv * C::TILE_BYTES, j > 0);
          tc_commit(BAR(C::B_KVEMPTY + sv));
          if (more) {
            issue_s(tS1, q1, kvb + sk2 * C::TILE_BYTES);
            tc_commit(BAR(C::B_SFULL + 1));
            tc_commit(BAR(C::B_KVEMPTY + sk2));
            ++kv_it;
            if (j + 2 == n) tc_commit(BAR(C::B_QEMPTY));
          } else {
            tc_commit(BAR(C::B_OFULL + 1));
          }
          ++sp_it;
        }
      }
      if (!ok) {
        tc_commit(BAR(C::B_DRAIN));
        drain_wait(BAR(C::B_DRAIN), 0, 100000000ull);
      }
    }
  }
  } else {
    regs_inc<REGS_SOFTMAX>();
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;                 // Q tile of this warpgroup
    const int lg = warp & 3;                 // TMEM lane quarter
    const int r = lg * 32 + lane;            // row within the tile
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const uint32_t tS = tmem + lane_off + C::TM_S + t * 128;
    const uint32_t tO = tmem + lane_off + C::TM_O + t * D;
    const float tau = fminf(fmaxf(p.tau, 0.f), TAU_MAX);   // the host allows [0, 1.5]
    Walker w;
    w.init(spec);
    uint32_t sp_it = 0;
    int u_it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!w.seek(snake_index(k, G, cta), u)) break;
      const int n = u.cost;
      const int row = u.m * UNIT_ROWS + t * BM + r;
      const bool valid = row < u.q_len;
      const long long grow = (long long)u.q_start + row;
      const int kvh = u.head / group;
      float* lse_ptr = p.lse + (long long)u.seq * p.lse_seqstride +
                       (long long)u.head * p.lse_hstride + row;
      __nv_bfloat16* orow = p.o + (grow * p.Hq + u.head) * D;
      if (n == 0) {
        if (valid) {
          uint4 z = make_uint4(0, 0, 0, 0);
          for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = z;
          *lse_ptr = INFINITY;
        }
        continue;
      }
      // softmax scale * log2(e) * this tile's query scale; per block times k_scale
      // (a tile wholly past the last query row has no scale block; its rows
      // are not stored)
      const int qb = u.m * 2 + t;
      const float sl2q =
          p.scale_log2 * (qb < p.nqb ? p.q_scale[((long long)u.seq * p.Hq + u.head) * p.nqb + qb] : 1.f);
      const float* ksc = p.k_scale + ((long long)u.seq * p.Hkv + kvh) * p.nkb;
      int kv_lim = u.k_len;
      if (p.causal) {
        const int lim = row + 1 + (u.k_len - u.q_len);
        kv_lim = lim < kv_lim ? lim : kv_lim;
      }
      float m_ref = -INFINITY, l = 0.f;
      float kscale = ksc[0];
      for (int j = 0; j < n; ++j) {
        const float c_j = sl2q * kscale;
        if (j + 1 < n) kscale = ksc[j + 1];             // next block's scale, read early
        ok = mbar_wait(BAR(C::B_SFULL + t), sp_it & 1, wc, SITE_FWD_S_FULL);
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[BN];                       // S row, raw fp32 bits
        tmem_ld128(tS, sr);
        const int lim = kv_lim - j * BN;
        if (__any_sync(0xffffffffu, lim < BN)) {
#pragma unroll
          for (int c = 0; c < BN; ++c) sr[c] = c < lim ? sr[c] : f2u(-INFINITY);
        }
        float mx[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) mx[i] = u2f(sr[i]);
#pragma unroll
        for (int c = 4; c < BN - 4; c += 8)          // [4, BN - 4) in pairs of four
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[i] = fmax3(mx[i], u2f(sr[c + i]), u2f(sr[c + 4 + i]));
#pragma unroll
        for (int i = 0; i < 4; ++i) mx[i] = fmaxf(mx[i], u2f(sr[BN - 4 + i]));
        const float m_blk = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]) * c_j;
        if (j == 0) {
          m_ref = m_blk;
        } else if (__any_sync(0xffffffffu, m_blk > m_ref + tau)) {
          const bool need = m_blk > m_ref + tau;
          const float m_new = need ? m_blk : m_ref;
          const float alpha = need ? ex2_mufu(m_ref - m_new) : 1.0f;
          const uint64_t a2 = f2pack(alpha, alpha);
#pragma unroll 1
          for (int c = 0; c < D; c += 32) {
            uint32_t o[32];
            tmem_ld32(tO + c, o);
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              float x0, x1;
              f2unpack(fmul2(f2pack(u2f(o[i]), u2f(o[i + 1])), a2), x0, x1);
              o[i] = f2u(x0);
              o[i + 1] = f2u(x1);
            }
            tmem_st32(tO + c, o);
          }
          l *= alpha;
          m_ref = m_new;
        }
        // weights 2^7 * p = exp2(S * c_j - m + 7), summed in fp32 and packed as e4m3
        const float msub = (m_ref == -INFINITY ? 0.f : m_ref) - P_LOG2_OFFSET;
        const uint64_t c2 = f2pack(c_j, c_j), negm2 = f2pack(-msub, -msub);
        uint64_t la2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          float x0, x1, x2, x3;
          f2unpack(ffma2(f2pack(u2f(sr[4 * c]), u2f(sr[4 * c + 1])), c2, negm2), x0, x1);
          f2unpack(ffma2(f2pack(u2f(sr[4 * c + 2]), u2f(sr[4 * c + 3])), c2, negm2), x2, x3);
          // POLY8 of every 8 exponentials on the FMA pipe, the rest on MUFU
          const float p0 = ((4 * c) & 7) < POLY8 ? exp2_poly(x0) : ex2_mufu(x0);
          const float p1 = ((4 * c + 1) & 7) < POLY8 ? exp2_poly(x1) : ex2_mufu(x1);
          const float p2 = ((4 * c + 2) & 7) < POLY8 ? exp2_poly(x2) : ex2_mufu(x2);
          const float p3 = ((4 * c + 3) & 7) < POLY8 ? exp2_poly(x3) : ex2_mufu(x3);
          la2[c & 1] = fadd2(la2[c & 1], fadd2(f2pack(p0, p1), f2pack(p2, p3)));
          pk[c] = e4m3x4(p0, p1, p2, p3);
        }
        {
          float a0, a1;
          f2unpack(fadd2(la2[0], la2[1]), a0, a1);
          l += a0 + a1;
        }
        tmem_st32(tS, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(C::B_PFULL + t));
        ++sp_it;
      }
      if (!ok) break;
      ok = mbar_wait(BAR(C::B_OFULL + t), u_it & 1, wc, SITE_FWD_O_FULL);
      if (!ok) break;
      tc_fence_after();
      ++u_it;
      const float inv = l > 0.f ? p.v_scale[(long long)u.seq * p.Hkv + kvh] / l : 0.f;
      const int row0 = u.m * UNIT_ROWS + t * BM;         // the tile's first row in the sequence
      if (row0 + BM <= u.q_len) {
        // A whole tile of the sequence: out through this warpgroup's staging
        // buffer (the tensor map's 128B-swizzled layout) with TMA stores of
        // full 128-byte lines.
        const uint32_t stage = base + C::STAGE_OFF + t * C::OCHUNKS * C::OCHUNK_BYTES;
        uint8_t* stage_p = smem + C::STAGE_OFF + t * C::OCHUNKS * C::OCHUNK_BYTES + r * 128;
        if (r == 0) tma_store_wait_read();               // the previous tile's stores read it
        named_bar_sync(1 + t, BM);
#pragma unroll 1
        for (int ch = 0; ch < C::OCHUNKS; ++ch) {
          uint32_t o[64];
          tmem_ld64(tO + ch * 64, o);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            uint4 v;
            v.x = pack_bf16x2(u2f(o[8 * j]) * inv, u2f(o[8 * j + 1]) * inv);
            v.y = pack_bf16x2(u2f(o[8 * j + 2]) * inv, u2f(o[8 * j + 3]) * inv);
            v.z = pack_bf16x2(u2f(o[8 * j + 4]) * inv, u2f(o[8 * j + 5]) * inv);
            v.w = pack_bf16x2(u2f(o[8 * j + 6]) * inv, u2f(o[8 * j + 7]) * inv);
            *reinterpret_cast<uint4*>(stage_p + ch * C::OCHUNK_BYTES + ((j ^ (r & 7)) << 4)) = v;
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1 + t, BM);
        if (r == 0) {
          for (int ch = 0; ch < C::OCHUNKS; ++ch)
            tma_store_3d(&p.tm_o, stage + ch * C::OCHUNK_BYTES, ch * 64, u.head,
                         u.q_start + row0);
          tma_store_commit();
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          uint32_t q[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            q[i] = pack_bf16x2(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
            dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
            dst[2] = make_uint4(q[8], q[9], q[10], q[11]);
            dst[3] = make_uint4(q[12], q[13], q[14], q[15]);
          }
        }
      }
      if (valid)
        *lse_ptr = l > 0.f ? (m_ref + log2f(l) - P_LOG2_OFFSET) * 0.69314718055994530942f
                           : INFINITY;
    }
  }

  // the O stores complete before the CTA (and its shared memory) goes away
  if (warp < 8 && (threadIdx.x & (BM - 1)) == 0) tma_store_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
#undef BAR
}

}  // namespace fwd8

template <int POLY8>
static cudaError_t launch_fp8_one(const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = fwd8::fwd_fp8_kernel<POLY8>;
  const int smem = fwd8::Cfg::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, fwd8::NUM_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_fp8(const FwdParams& p, int grid, cudaStream_t stream, int poly8) {
  switch (poly8) {
    case 0: return launch_fp8_one<0>(p, grid, stream);
    case 2: return launch_fp8_one<2>(p, grid, stream);
    case 4: return launch_fp8_one<4>(p, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace fa
