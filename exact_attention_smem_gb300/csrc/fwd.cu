// Forward attention kernel for sm_103a: O = softmax(scale * Q K^T [+ causal mask]) V
// and the fp32 row log-sum-exp, by tiling with an online softmax.
//
// Method (FlashAttention-4 pages): "FlashAttention-4: Algorithm and Kernel
// Pipelining Co-Design for Asymmetric Hardware Scaling" — abstract items (1)
// and (2) and the daily.dev Summary: fully asynchronous MMAs with larger tiles,
// a ping-pong pipeline overlapping one tile's MMAs with the other tile's
// softmax, a software exp2 beside the MUFU unit, conditional rescaling, and a
// longest-processing-time-first scheduler. Tiling + online softmax itself is the
// lineage described in "FlashAttention-4 Conquers Asymmetric GPU Hardware
// Scaling" (episode description).
//
// One persistent CTA per SM, 12 warps (3 warpgroups):
//   warps 0-3  softmax for Q tile 0 (one thread per row = TMEM lane)
//   warps 4-7  softmax for Q tile 1
//   warp  8    TMEM allocation + MMA issue (one elected thread)
//   warp  9    TMA producer (one elected thread)
//   warps 10-11 idle (they complete the third warpgroup for the register split)
// Work unit: 2 x 128 query rows of one (sequence, query head). K/V blocks of 128
// keys stream through an mbarrier ring of shared-memory stages (K_j, V_j, ...).
// TMEM (512 columns): S_0 [0,128), S_1 [128,256), O_0 [256,256+d), O_1 after it;
// P_t (bf16) overwrites the first 64 columns of S_t and is the A operand of
// O_t += P_t V (A from TMEM, B = V from shared memory).
#include "exp2_poly.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

#include <cmath>

namespace fa {
using namespace ptx;

namespace fwdk {

constexpr int BM = 128;         // query rows per tile
constexpr int BN = 128;         // keys per KV block
constexpr int UNIT_ROWS = 2 * BM;
constexpr int NUM_THREADS = 384;   // 3 warpgroups: softmax 0, softmax 1, MMA/TMA (+2 idle warps)
constexpr int MMA_WARP = 8;
constexpr int TMA_WARP = 9;
// Register split: launch gives 168 per thread (65536 / 384, rounded down to 8);
// the MMA/TMA warpgroup gives back down to 112 and the softmax warpgroups take
// 192: 2*128*192 + 128*112 = 63488 <= 384*168 = 64512 (no spills either side).
constexpr int REGS_SOFTMAX = 192;
constexpr int REGS_CONTROL = 112;
constexpr int MAX_SEQ_SMEM = 256;   // packed boundaries kept in shared memory up to this

template <int D>
struct Cfg {
  static constexpr int CHUNKS = D / 64;                 // 128-byte column chunks per row
  static constexpr int CHUNK_BYTES = 128 * 128;         // 128 rows x 128 bytes
  static constexpr int TILE_BYTES = CHUNKS * CHUNK_BYTES;
  static constexpr int NSTAGE = D == 128 ? 4 : 8;
  static constexpr int Q_OFF = 0;
  static constexpr int KV_OFF = 2 * TILE_BYTES;
  static constexpr int BAR_OFF = KV_OFF + NSTAGE * TILE_BYTES;
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KVFULL = 2, B_KVEMPTY = 2 + NSTAGE,
                       B_SFULL = 2 + 2 * NSTAGE, B_PFULL = B_SFULL + 2, B_OFULL = B_PFULL + 2,
                       B_DRAIN = B_OFULL + 2,
                       // tile 1's own Q pair when the tiles load separately
                       // (B_QFULL / B_QEMPTY then serve tile 0 alone)
                       B_QFULL1 = B_DRAIN + 1, B_QEMPTY1 = B_DRAIN + 2, NBAR = B_DRAIN + 3;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int CU_OFF = MISC_OFF + 16;
  // O write-out staging: one 128-row x 64-column chunk (128B swizzle) per softmax warpgroup
  static constexpr int STAGE_OFF = (CU_OFF + (MAX_SEQ_SMEM + 1) * 4 + 1023) & ~1023;
  static constexpr int SMEM_BYTES = STAGE_OFF + 2 * CHUNK_BYTES + 1024;
  static_assert(SMEM_BYTES <= 232448, "forward shared memory");
  static constexpr uint32_t IDESC_S = idesc_bf16(128, 128, false, false);
  static constexpr uint32_t IDESC_PV = idesc_bf16(128, D, false, true);
  static constexpr uint32_t TM_S = 0;
  static constexpr uint32_t TM_O = 256;
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

// Wait that ignores the abort flag: used only to let in-flight async work land
// before an aborting CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// S (TMEM, 128x128 fp32) = Q_tile (128 x D) * K_block^T; both operands K-major.
template <int D>
__device__ __forceinline__ void issue_s(uint32_t tm_s, uint32_t q_tile, uint32_t k_tile) {
  using C = Cfg<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
    mma_ss(tm_s, sdesc_sw128(q_tile + off, C::CHUNK_BYTES, 1024),
           sdesc_sw128(k_tile + off, C::CHUNK_BYTES, 1024), C::IDESC_S, kk > 0 ? 1u : 0u);
  }
}

// O (TMEM, 128 x D fp32) (+)= P (TMEM, 128 x 128 bf16) * V_block (128 x D, MN-major B).
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tm_o, uint32_t tm_p, uint32_t v_tile,
                                         bool accumulate) {
  using C = Cfg<D>;
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    mma_ts(tm_o, tm_p + kk * 8, sdesc_sw128(v_tile + kk * 16 * 128, C::CHUNK_BYTES, 1024),
           C::IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int D, int POLY8>
__global__ void __launch_bounds__(NUM_THREADS, 1) fwd_kernel(const __grid_constant__ FwdParams p) {
  using C = Cfg<D>;
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
  int* cu_s = reinterpret_cast<int*>(smem + C::CU_OFF);

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_QFULL), 1);
    mbar_init(BAR(C::B_QEMPTY), 1);
    mbar_init(BAR(C::B_QFULL1), 1);
    mbar_init(BAR(C::B_QEMPTY1), 1);
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
  // packed boundaries in shared memory when they fit (query list, then key list)
  const int ncu = p.cu_k ? 2 * (p.nseq + 1) : p.nseq + 1;
  const bool cu_in_smem = p.cu != nullptr && ncu <= MAX_SEQ_SMEM + 1;
  if (cu_in_smem)
    for (int i = threadIdx.x; i < ncu; i += NUM_THREADS)
      cu_s[i] = i <= p.nseq ? p.cu[i] : p.cu_k[i - p.nseq - 1];
  const int* cu_k_spec = p.cu_k ? (cu_in_smem ? cu_s + p.nseq + 1 : p.cu_k) : nullptr;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const SchedSpec spec{cu_in_smem ? cu_s : p.cu, p.nseq, p.Sq, p.Sk, p.Hq, p.causal,
                       UNIT_ROWS, BN, 0, p.hblock, cu_k_spec};
  const WaitCtl wc{p.err, abort_flag, p.timeout_ns};
  const int G = gridDim.x;
  const int cta = blockIdx.x;
  const int group = p.Hq / p.Hkv;

  if (warp >= 8) {
    regs_dec<REGS_CONTROL>();
  if (warp >= 10) {
    // spare warps of the control warpgroup: nothing to do
  } else if (warp == TMA_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Walker w;
      w.init(spec);
      uint32_t kv_it = 0;
      int u_it = 0;
      uint32_t q_cnt[2] = {0, 0};           // Q loads issued on each Q pair
      const bool split = p.split_q != 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        const int n = u.cost;
        if (n == 0) continue;
        const int kvh = u.head / group;
        const int q_row = u.q_start + u.m * UNIT_ROWS;
        for (int t = 0; t < (split ? 2 : 1); ++t) {
          const uint32_t full = BAR(t ? C::B_QFULL1 : C::B_QFULL);
          if (u_it > 0) {
            ok = mbar_wait(BAR(t ? C::B_QEMPTY1 : C::B_QEMPTY), (u_it - 1) & 1, wc,
                           SITE_FWD_Q_EMPTY);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(full, split ? C::TILE_BYTES : 2 * C::TILE_BYTES);
          for (int tt = t; tt < (split ? t + 1 : 2); ++tt)
            for (int c = 0; c < C::CHUNKS; ++c)
              tma_load_3d(base + C::Q_OFF + tt * C::TILE_BYTES + c * C::CHUNK_BYTES, &p.tm_q,
                          full, c * 64, u.head, q_row + tt * BM);
          ++q_cnt[t];
        }
        if (!ok) break;
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
            const void* tm = which ? static_cast<const void*>(&p.tm_v)
                                   : static_cast<const void*>(&p.tm_k);
            for (int c = 0; c < C::CHUNKS; ++c)
              tma_load_3d(base + C::KV_OFF + s * C::TILE_BYTES + c * C::CHUNK_BYTES, tm,
                          BAR(C::B_KVFULL + s), c * 64, kvh, u.k_start + j * BN);
            ++kv_it;
          }
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA exits
        for (uint32_t i = kv_it > (uint32_t)C::NSTAGE ? kv_it - C::NSTAGE : 0; i < kv_it; ++i)
          drain_wait(BAR(C::B_KVFULL + i % C::NSTAGE), (i / C::NSTAGE) & 1, 100000000ull);
        for (int t = 0; t < 2; ++t)
          if (q_cnt[t] > 0)
            drain_wait(BAR(t ? C::B_QFULL1 : C::B_QFULL), (q_cnt[t] - 1) & 1, 100000000ull);
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
      const bool split = p.split_q != 0;
      // tile 1's Q empty barrier: its own pair when the tiles load separately
      const uint32_t q_empty1 = BAR(split ? C::B_QEMPTY1 : C::B_QEMPTY);
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        const int n = u.cost;
        if (n == 0) continue;
        int sk = kv_it % C::NSTAGE;
        if (split) {
          ok = mbar_wait3(BAR(C::B_QFULL), u_it & 1, SITE_FWD_Q_FULL, BAR(C::B_QFULL1),
                          u_it & 1, SITE_FWD_Q_FULL, BAR(C::B_KVFULL + sk),
                          (kv_it / C::NSTAGE) & 1, SITE_FWD_KV_FULL, wc);
          if (!ok) break;
        } else {
          ok = mbar_wait(BAR(C::B_QFULL), u_it & 1, wc, SITE_FWD_Q_FULL);
          if (!ok) break;
          ok = mbar_wait(BAR(C::B_KVFULL + sk), (kv_it / C::NSTAGE) & 1, wc, SITE_FWD_KV_FULL);
          if (!ok) break;
        }
        ++u_it;
        tc_fence_after();
        issue_s<D>(tS0, q0, kvb + sk * C::TILE_BYTES);
        tc_commit(BAR(C::B_SFULL + 0));
        if (split && n == 1) tc_commit(BAR(C::B_QEMPTY));
        issue_s<D>(tS1, q1, kvb + sk * C::TILE_BYTES);
        tc_commit(BAR(C::B_SFULL + 1));
        tc_commit(BAR(C::B_KVEMPTY + sk));
        ++kv_it;
        if (n == 1) tc_commit(q_empty1);
        for (int j = 0; j < n; ++j) {
          // sync point 1: V_j, P_0(j) and (if any) K_{j+1}, probed together
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
          issue_pv<D>(tO0, tS0, kvb + sv * C::TILE_BYTES, j > 0);
          if (more) {
            issue_s<D>(tS0, q0, kvb + sk2 * C::TILE_BYTES);
            tc_commit(BAR(C::B_SFULL + 0));
            if (split && j + 2 == n) tc_commit(BAR(C::B_QEMPTY));
          } else {
            tc_commit(BAR(C::B_OFULL + 0));
          }
          // sync point 2: P_1(j)
          ok = mbar_wait(BAR(C::B_PFULL + 1), sp_it & 1, wc, SITE_FWD_P_FULL);
          if (!ok) break;
          tc_fence_after();
          issue_pv<D>(tO1, tS1, kvb + sv * C::TILE_BYTES, j > 0);
          tc_commit(BAR(C::B_KVEMPTY + sv));
          if (more) {
            issue_s<D>(tS1, q1, kvb + sk2 * C::TILE_BYTES);
            tc_commit(BAR(C::B_SFULL + 1));
            tc_commit(BAR(C::B_KVEMPTY + sk2));
            ++kv_it;
            if (j + 2 == n) tc_commit(q_empty1);
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
    const float sl2 = p.scale_log2;
    const float tau = p.tau;
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
      float* lse_ptr = p.lse + (p.cu ? (long long)u.q_start : (long long)u.seq * p.lse_seqstride) +
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
      int kv_lim = u.k_len;
      if (p.causal) {
        const int lim = row + 1 + (u.k_len - u.q_len);
        kv_lim = lim < kv_lim ? lim : kv_lim;
      }
      float m_ref = -INFINITY, l = 0.f, lp = 0.f;
      for (int j = 0; j < n; ++j) {
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
        const float m_blk = fmaxf(fmax3(mx[0], mx[1], mx[2]), mx[3]) * sl2;
        if (j == 0) {
          m_ref = m_blk;
        } else {
          const bool need = m_blk > m_ref + tau;
          if (__any_sync(0xffffffffu, need)) {
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
            lp *= alpha;
            m_ref = m_new;
          }
        }
        const float msub = m_ref == -INFINITY ? 0.f : m_ref;
        // Two row sums: of the fp32 p (for the LSE) and of the bf16-rounded P
        // that the PV MMA actually multiplies (for normalising O, so that the
        // weights applied to V sum to one). Pairs use the f32x2 pipe.
        const uint64_t sl2x2 = f2pack(sl2, sl2), negm2 = f2pack(-msub, -msub);
        uint64_t la2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
        float lb4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float x0, x1;
          f2unpack(ffma2(f2pack(u2f(sr[2 * c]), u2f(sr[2 * c + 1])), sl2x2, negm2), x0, x1);
          const float p0 = ((2 * c) & 7) < POLY8 ? exp2_poly(x0) : ex2_mufu(x0);
          const float p1 = ((2 * c + 1) & 7) < POLY8 ? exp2_poly(x1) : ex2_mufu(x1);
          const uint32_t pb = pack_bf16x2(p0, p1);
          la2[c & 1] = fadd2(la2[c & 1], f2pack(p0, p1));
          add_bf16x2_f32(lb4[2 * (c & 1)], lb4[2 * (c & 1) + 1], pb);
          pk[c] = pb;
        }
        {
          float a0, a1, b0, b1;
          f2unpack(fadd2(la2[0], la2[1]), a0, a1);
          b0 = lb4[0] + lb4[2];
          b1 = lb4[1] + lb4[3];
          l += a0 + a1;
          lp += b0 + b1;
        }
        tmem_st64(tS, pk);
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
      const float inv = lp > 0.f ? 1.0f / lp : 0.f;
      const int row0 = u.m * UNIT_ROWS + t * BM;         // the tile's first row in the sequence
      if (row0 + BM <= u.q_len) {
        // A whole tile of the sequence: each 64-column chunk goes through this
        // warpgroup's staging buffer (rows in the 128B-swizzled layout the
        // tensor map uses) and out as one TMA store of full 128-byte lines.
        const uint32_t stage = base + C::STAGE_OFF + t * C::CHUNK_BYTES;
        uint8_t* stage_p = smem + C::STAGE_OFF + t * C::CHUNK_BYTES + r * 128;
#pragma unroll 1
        for (int ch = 0; ch < C::CHUNKS; ++ch) {
          uint32_t o[64];
          tmem_ld64(tO + ch * 64, o);
          uint32_t q[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) q[i] = pack_bf16x2(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
          // the previous store from this buffer has read it
          if (r == 0) tma_store_wait_read();
          named_bar_sync(1 + t, BM);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<uint4*>(stage_p + ((j ^ (r & 7)) << 4)) =
                make_uint4(q[4 * j], q[4 * j + 1], q[4 * j + 2], q[4 * j + 3]);
          fence_proxy_async_smem();
          named_bar_sync(1 + t, BM);
          if (r == 0) {
            tma_store_3d(&p.tm_o, stage, ch * 64, u.head, u.q_start + row0);
            tma_store_commit();
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t o[32];
          tmem_ld32(tO + c, o);
          uint32_t q[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) q[i] = pack_bf16x2(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
            dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
            dst[2] = make_uint4(q[8], q[9], q[10], q[11]);
            dst[3] = make_uint4(q[12], q[13], q[14], q[15]);
          }
        }
      }
      if (valid) *lse_ptr = l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994530942f : INFINITY;
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

}  // namespace fwdk

template <int D, int POLY8>
static cudaError_t launch_one(const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = fwdk::fwd_kernel<D, POLY8>;
  const int smem = fwdk::Cfg<D>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, fwdk::NUM_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd(const FwdParams& p, int d, int grid, cudaStream_t stream, int poly8) {
  if (d == 128) {
    switch (poly8) {
      case 0: return launch_one<128, 0>(p, grid, stream);
      case 2: return launch_one<128, 2>(p, grid, stream);
      case 4: return launch_one<128, 4>(p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (d == 64) {
    switch (poly8) {
      case 0: return launch_one<64, 0>(p, grid, stream);
      case 2: return launch_one<64, 2>(p, grid, stream);
      case 4: return launch_one<64, 4>(p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
