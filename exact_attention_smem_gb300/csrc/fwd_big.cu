// Forward attention for head dims 192 and 256 on sm_103a: O and the fp32 row
// log-sum-exp, by tiling with an online softmax, like the head-dim 64/128
// kernel (fwd.cu) but shaped for the larger head dim, which does not leave
// room for that kernel's two ping-pong query tiles: two 128-row O tiles of
// d = 256 alone would fill the 512 TMEM columns, and K/V blocks of 128 keys
// would leave no shared memory for a ring.
//
// Method: "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling", abstract items (1)-(2) and the Summary
// (asynchronous MMAs accumulating in tensor memory, conditional rescaling,
// longest-processing-time-first scheduling); tiling with an online softmax as
// in "FlashAttention-4 Conquers Asymmetric GPU Hardware Scaling" (episode
// description).
//
// One persistent CTA per SM, 8 warps: warps 0-3 run the softmax of one
// 128-row query tile (one thread per row = TMEM lane), warp 4 allocates TMEM
// and one of its threads issues the MMAs, warp 5 is the TMA producer, warps
// 6-7 are idle. A unit is 128 query rows of one (sequence, head); K/V blocks
// have 64 keys. TMEM: four S buffers of 64 columns [0,256) and O [256,256+d).
// S runs two blocks ahead of the softmax: at the sync point of block j the MMA
// thread issues O += P(j) V_j (P in bf16 over the first 32 columns of its S
// buffer, the TMEM A operand) and then S(j+2) = Q K_{j+2}^T. K and V have
// rings of their own (K is released once its S is done, V once its PV is).
#include "exp2_poly.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

#include <cmath>

namespace fa {
using namespace ptx;

namespace fwdb {

constexpr int BM = 128;            // query rows per unit
constexpr int BN = 64;             // keys per block
constexpr int NUM_THREADS = 256;
constexpr int MMA_WARP = 4;
constexpr int TMA_WARP = 5;
constexpr int NS = 4;              // S buffers
constexpr int LOOK = 2;            // S(j + LOOK) is issued at block j's sync point
constexpr int MAX_SEQ_SMEM = 256;
constexpr int SMEM_LIMIT = 232448;

template <int D>
struct Cfg {
  static constexpr int CHUNKS = D / 64;                // 128-byte column chunks per row
  static constexpr int Q_CHUNK = BM * 128;             // 128 rows x 128 bytes
  static constexpr int KV_CHUNK = BN * 128;            // 64 rows x 128 bytes
  static constexpr int Q_BYTES = CHUNKS * Q_CHUNK;
  static constexpr int KV_BYTES = CHUNKS * KV_CHUNK;
  static constexpr int NK = 2, NV = D == 256 ? 3 : 4;
  static constexpr int Q_OFF = 0, K_OFF = Q_BYTES, V_OFF = K_OFF + NK * KV_BYTES,
                       BAR_OFF = V_OFF + NV * KV_BYTES;
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KFULL = 2, B_KEMPTY = B_KFULL + NK,
                       B_VFULL = B_KEMPTY + NK, B_VEMPTY = B_VFULL + NV,
                       B_SFULL = B_VEMPTY + NV,    // [NS]
                       B_PFULL = B_SFULL + NS,     // [NS]: one per S buffer (see the MMA role)
                       B_OFULL = B_PFULL + NS, B_OSYNC = B_OFULL + 1, B_DRAIN = B_OSYNC + 1,
                       NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int CU_OFF = MISC_OFF + 16;
  static constexpr int SMEM_BYTES = CU_OFF + (MAX_SEQ_SMEM + 1) * 4 + 1024;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
  static constexpr uint32_t TM_S = 0, TM_O = NS * BN;
  static_assert(TM_O + D <= 512, "TMEM columns");
  static constexpr uint32_t IDESC_S = idesc_bf16(BM, BN, false, false);   // S = Q K^T
  static constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, false, true);    // O += P V
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// S (TMEM, 128 x 64 fp32) = Q tile (128 x D, K-major) * K block (64 x D, K-major)^T
template <int D>
__device__ __forceinline__ void issue_s(uint32_t tm_s, uint32_t q_tile, uint32_t k_tile) {
  using C = Cfg<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t c = (kk >> 2), w = (kk & 3) * 32;
    mma_ss(tm_s, sdesc_sw128(q_tile + c * C::Q_CHUNK + w, C::Q_CHUNK, 1024),
           sdesc_sw128(k_tile + c * C::KV_CHUNK + w, C::KV_CHUNK, 1024), C::IDESC_S,
           kk > 0 ? 1u : 0u);
  }
}

// O (TMEM, 128 x D) (+)= P (TMEM, 128 x 64 bf16 in the S buffer's first 32
// columns) * V block (64 x D, MN-major B)
template <int D>
__device__ __forceinline__ void issue_pv(uint32_t tm_o, uint32_t tm_p, uint32_t v_tile,
                                         bool accumulate) {
  using C = Cfg<D>;
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk)
    mma_ts(tm_o, tm_p + kk * 8, sdesc_sw128(v_tile + kk * 16 * 128, C::KV_CHUNK, 1024),
           C::IDESC_PV, (accumulate || kk > 0) ? 1u : 0u);
}

template <int D, int POLY8>
__global__ void __launch_bounds__(NUM_THREADS, 1) fwd_big_kernel(const __grid_constant__ FwdParams p) {
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
    for (int s = 0; s < C::NK; ++s) {
      mbar_init(BAR(C::B_KFULL + s), 1);
      mbar_init(BAR(C::B_KEMPTY + s), 1);
    }
    for (int s = 0; s < C::NV; ++s) {
      mbar_init(BAR(C::B_VFULL + s), 1);
      mbar_init(BAR(C::B_VEMPTY + s), 1);
    }
    for (int s = 0; s < NS; ++s) {
      mbar_init(BAR(C::B_SFULL + s), 1);
      mbar_init(BAR(C::B_PFULL + s), BM);
    }
    mbar_init(BAR(C::B_OFULL), 1);
    mbar_init(BAR(C::B_OSYNC), 1);
    mbar_init(BAR(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
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

  const SchedSpec spec{cu_in_smem ? cu_s : p.cu, p.nseq, p.Sq, p.Sk, p.Hq, p.causal, BM, BN, 0,
                       p.hblock, cu_k_spec};
  const WaitCtl wc{p.err, abort_flag, p.timeout_ns};
  const int G = gridDim.x;
  const int cta = blockIdx.x;
  const int group = p.Hq / p.Hkv;

  if (warp >= 4) {
  if (warp >= 6) {
    // idle warps
  } else if (warp == TMA_WARP) {
    // ------------------------------------------------------------ producer
    // Per unit: Q, then K_0 .. K_{LOOK-1}, then for each block b: V_b and
    // K_{b+LOOK}, the order the MMA thread consumes them in.
    if (lane == 0) {
      Walker w;
      w.init(spec);
      uint32_t nk = 0, nv = 0;
      int u_it = 0;
      bool ok = true;
      auto load_k = [&](int kvh, int krow) -> bool {
        const int s = nk % C::NK;
        if (nk >= (uint32_t)C::NK &&
            !mbar_wait(BAR(C::B_KEMPTY + s), ((nk / C::NK) - 1) & 1, wc, SITE_FWD_KV_EMPTY))
          return false;
        mbar_arrive_expect_tx(BAR(C::B_KFULL + s), C::KV_BYTES);
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(base + C::K_OFF + s * C::KV_BYTES + c * C::KV_CHUNK, &p.tm_k,
                      BAR(C::B_KFULL + s), c * 64, kvh, krow);
        ++nk;
        return true;
      };
      auto load_v = [&](int kvh, int krow) -> bool {
        const int s = nv % C::NV;
        if (nv >= (uint32_t)C::NV &&
            !mbar_wait(BAR(C::B_VEMPTY + s), ((nv / C::NV) - 1) & 1, wc, SITE_FWD_KV_EMPTY))
          return false;
        mbar_arrive_expect_tx(BAR(C::B_VFULL + s), C::KV_BYTES);
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(base + C::V_OFF + s * C::KV_BYTES + c * C::KV_CHUNK, &p.tm_v,
                      BAR(C::B_VFULL + s), c * 64, kvh, krow);
        ++nv;
        return true;
      };
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        const int n = u.cost;
        if (n == 0) continue;
        const int kvh = u.head / group;
        if (u_it > 0) {
          ok = mbar_wait(BAR(C::B_QEMPTY), (u_it - 1) & 1, wc, SITE_FWD_Q_EMPTY);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(BAR(C::B_QFULL), C::Q_BYTES);
        for (int c = 0; c < C::CHUNKS; ++c)
          tma_load_3d(base + C::Q_OFF + c * C::Q_CHUNK, &p.tm_q, BAR(C::B_QFULL), c * 64, u.head,
                      u.q_start + u.m * BM);
        ++u_it;
        for (int b = 0; b < LOOK && b < n && ok; ++b) ok = load_k(kvh, u.k_start + b * BN);
        for (int b = 0; b < n && ok; ++b) {
          ok = load_v(kvh, u.k_start + b * BN);
          if (ok && b + LOOK < n) ok = load_k(kvh, u.k_start + (b + LOOK) * BN);
        }
      }
      if (!ok) {
        for (uint32_t i = nk > (uint32_t)C::NK ? nk - C::NK : 0; i < nk; ++i)
          drain_wait(BAR(C::B_KFULL + i % C::NK), (i / C::NK) & 1, 100000000ull);
        for (uint32_t i = nv > (uint32_t)C::NV ? nv - C::NV : 0; i < nv; ++i)
          drain_wait(BAR(C::B_VFULL + i % C::NV), (i / C::NV) & 1, 100000000ull);
        if (u_it > 0) drain_wait(BAR(C::B_QFULL), (u_it - 1) & 1, 100000000ull);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    // One sync point per block: P(j) ready (+ V_j, K_{j+LOOK} loaded) ->
    // O += P(j) V_j, then S(j+LOOK) into the buffer of S(j+LOOK-NS), whose P
    // an earlier PV has read (MMAs of one thread execute in order). P ready
    // has one barrier per S buffer: the softmax may finish P(j+1) before this
    // thread waits for P(j), and a parity wait cannot tell phases two apart.
    // The softmax writes the previous unit's O out before it arrives for the
    // first block of this unit, which orders PV(0) (overwriting O) after it.
    if (lane == 0) {
      Walker w;
      w.init(spec);
      uint32_t nk = 0, nv = 0, sj = 0;
      int u_it = 0;
      bool ok = true;
      const uint32_t qt = base + C::Q_OFF;
      auto kslot = [&](uint32_t x) { return base + C::K_OFF + (x % C::NK) * C::KV_BYTES; };
      auto vslot = [&](uint32_t x) { return base + C::V_OFF + (x % C::NV) * C::KV_BYTES; };
      auto sbuf = [&](uint32_t x) { return tmem + C::TM_S + (x % NS) * BN; };
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        const int n = u.cost;
        if (n == 0) continue;
        // prologue: S(0) .. S(LOOK-1)
        for (int b = 0; b < LOOK && b < n && ok; ++b) {
          const uint32_t x = nk + b;
          ok = mbar_wait3(BAR(C::B_QFULL), u_it & 1, SITE_FWD_Q_FULL,
                          BAR(C::B_KFULL + x % C::NK), (x / C::NK) & 1, SITE_FWD_KV_FULL,
                          BAR(C::B_QFULL), u_it & 1, SITE_FWD_Q_FULL, wc);
          if (!ok) break;
          tc_fence_after();
          issue_s<D>(sbuf(sj + b), qt, kslot(x));
          tc_commit(BAR(C::B_SFULL + (sj + b) % NS));
          tc_commit(BAR(C::B_KEMPTY + x % C::NK));
          if (b + 1 == n) tc_commit(BAR(C::B_QEMPTY));
        }
        if (!ok) break;
        const uint32_t k0 = nk;
        nk += (uint32_t)(n < LOOK ? n : LOOK);
        for (int jb = 0; jb < n && ok; ++jb, ++sj) {
          const bool ahead = jb + LOOK < n;
          const uint32_t xk = k0 + jb + LOOK, xv = nv;
          ok = mbar_wait3(BAR(C::B_PFULL + sj % NS), (sj / NS) & 1, SITE_FWD_P_FULL,
                          BAR(C::B_VFULL + xv % C::NV), (xv / C::NV) & 1, SITE_FWD_KV_FULL,
                          ahead ? BAR(C::B_KFULL + xk % C::NK) : BAR(C::B_PFULL + sj % NS),
                          ahead ? (xk / C::NK) & 1 : (sj / NS) & 1, SITE_FWD_KV_FULL, wc);
          if (!ok) break;
          tc_fence_after();
          issue_pv<D>(tmem + C::TM_O, sbuf(sj), vslot(xv), jb > 0);
          tc_commit(BAR(C::B_OSYNC));                    // PV(sj) done: O may be rescaled
          tc_commit(BAR(C::B_VEMPTY + xv % C::NV));
          ++nv;
          if (ahead) {
            issue_s<D>(sbuf(sj + LOOK), qt, kslot(xk));
            tc_commit(BAR(C::B_SFULL + (sj + LOOK) % NS));
            tc_commit(BAR(C::B_KEMPTY + xk % C::NK));
            ++nk;
            if (jb + LOOK + 1 == n) tc_commit(BAR(C::B_QEMPTY));
          }
          if (jb + 1 == n) tc_commit(BAR(C::B_OFULL));
        }
        ++u_it;
      }
      if (!ok) {
        tc_commit(BAR(C::B_DRAIN));
        drain_wait(BAR(C::B_DRAIN), 0, 100000000ull);
      }
    }
  }
  } else {
    // ------------------------------------------------------------ softmax
    const int r = warp * 32 + lane;                      // row within the tile
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tmem + lane_off + C::TM_O;
    const float sl2 = p.scale_log2;
    const float tau = p.tau;
    Walker w;
    w.init(spec);
    uint32_t sj = 0;
    int u_it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!w.seek(snake_index(k, G, cta), u)) break;
      const int n = u.cost;
      const int row = u.m * BM + r;
      const bool valid = row < u.q_len;
      const long long grow = (long long)u.q_start + row;
      float* lse_ptr = p.lse + (p.cu ? (long long)u.q_start : (long long)u.seq * p.lse_seqstride) +
                       (long long)u.head * p.lse_hstride + row;
      __nv_bfloat16* orow = p.o + (grow * p.Hq + u.head) * D;
      if (n == 0) {
        if (valid) {
          for (int c = 0; c < D; c += 8) *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
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
      for (int jb = 0; jb < n; ++jb, ++sj) {
        ok = mbar_wait(BAR(C::B_SFULL + sj % NS), (sj / NS) & 1, wc, SITE_FWD_S_FULL);
        if (!ok) break;
        tc_fence_after();
        const uint32_t tS = tmem + lane_off + C::TM_S + (sj % NS) * BN;
        uint32_t sr[BN];
        tmem_ld64(tS, sr);
        const int lim = kv_lim - jb * BN;
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
        if (jb == 0) {
          m_ref = m_blk;
        } else {
          const bool need = m_blk > m_ref + tau;
          if (__any_sync(0xffffffffu, need)) {
            // S runs ahead of the PVs, so S(j) landing does not mean PV(j-1)
            // has: wait for it before O is rescaled. (PV(j) needs P(j), which
            // this thread has not produced yet, so the barrier cannot be two
            // phases ahead of this parity wait.)
            const float m_new = need ? m_blk : m_ref;
            const float alpha = need ? ex2_mufu(m_ref - m_new) : 1.0f;
            const uint64_t a2 = f2pack(alpha, alpha);
            ok = mbar_wait(BAR(C::B_OSYNC), (sj - 1) & 1, wc, SITE_FWD_O_FULL);
            if (!ok) break;
            tc_fence_after();
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
        const uint64_t sl2x2 = f2pack(sl2, sl2), negm2 = f2pack(-msub, -msub);
        uint64_t la2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
        float lb4[4] = {0.f, 0.f, 0.f, 0.f};
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) {
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
        tmem_st32(tS, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(C::B_PFULL + sj % NS));
      }
      if (!ok) break;
      ok = mbar_wait(BAR(C::B_OFULL), u_it & 1, wc, SITE_FWD_O_FULL);
      if (!ok) break;
      tc_fence_after();
      ++u_it;
      const float inv = lp > 0.f ? 1.0f / lp : 0.f;
      // one row per thread: 32-byte stores where the row is 32-byte aligned
      // (half the store instructions and line accesses), else 16-byte ones
      const bool wide = (reinterpret_cast<uintptr_t>(orow) & 31) == 0;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t o[32];
        tmem_ld32(tO + c, o);
        uint32_t q[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) q[i] = pack_bf16x2(u2f(o[2 * i]) * inv, u2f(o[2 * i + 1]) * inv);
        if (valid) {
          if (wide) {
            const uint32_t q0[8] = {q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]};
            const uint32_t q1[8] = {q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]};
            st_global_v8(orow + c, q0);
            st_global_v8(orow + c + 16, q1);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(orow + c);
            dst[0] = make_uint4(q[0], q[1], q[2], q[3]);
            dst[1] = make_uint4(q[4], q[5], q[6], q[7]);
            dst[2] = make_uint4(q[8], q[9], q[10], q[11]);
            dst[3] = make_uint4(q[12], q[13], q[14], q[15]);
          }
        }
      }
      if (valid) *lse_ptr = l > 0.f ? (m_ref + log2f(l)) * 0.69314718055994530942f : INFINITY;
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
#undef BAR
}

}  // namespace fwdb

template <int D, int POLY8>
static cudaError_t launch_big(const FwdParams& p, int grid, cudaStream_t stream) {
  auto kern = fwdb::fwd_big_kernel<D, POLY8>;
  const int smem = fwdb::Cfg<D>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, fwdb::NUM_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

// Head dims 192 and 256 (the tensor maps of K and V use 64-row boxes).
cudaError_t launch_fwd_big(const FwdParams& p, int d, int grid, cudaStream_t stream, int poly8) {
  if (d == 256) {
    switch (poly8) {
      case 0: return launch_big<256, 0>(p, grid, stream);
      case 2: return launch_big<256, 2>(p, grid, stream);
      case 4: return launch_big<256, 4>(p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  if (d == 192) {
    switch (poly8) {
      case 0: return launch_big<192, 0>(p, grid, stream);
      case 2: return launch_big<192, 2>(p, grid, stream);
      case 4: return launch_big<192, 4>(p, grid, stream);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace fa
