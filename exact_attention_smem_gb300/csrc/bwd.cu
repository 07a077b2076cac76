// Backward attention for sm_103a: dQ, dK, dV from Q, K, V, O, dO and LSE.
//
// Three kernels on one stream:
//   1. preprocess: -D_i = -sum_c dO_ic O_ic and -LSE_i * log2(e) into padded
//      row arrays (each sequence starts on a 128-row boundary so one 64- or
//      128-row block is one aligned bulk copy; stored negated so the main
//      kernels use them as FMA addends), padding rows get LSE = +inf and D = 0,
//      and the fp32 dQ accumulator (one-pass form) is zeroed;
//   2. main: one persistent CTA per SM walks (sequence, 128-key block, KV head)
//      units longest-first. For each query head of the KV group and each block
//      of 64 query rows that sees the keys it computes, with tcgen05 MMAs
//      accumulating in TMEM:
//         S^T  = K Q^T            P^T  = exp2(S^T * scale*log2e - LSE*log2e)
//         dP^T = V dO^T           dS^T = P^T o (dP^T - D)
//         dV  += P^T dO           dK  += dS^T Q        dQ^T = K^T dS^T
//      and adds dQ^T into the fp32 accumulator with atomic adds. dK and dV stay
//      in TMEM for the whole unit (summed over the GQA group) and are written
//      once, dK scaled by the softmax scale;
//   3. convert: dQ = bf16(scale * accumulator).
// The pages' backward keeps accumulators and the P/dS operands in tensor
// memory to cut shared-memory traffic ("FlashAttention-4: Algorithm and Kernel
// Pipelining Co-Design for Asymmetric Hardware Scaling", abstract item (3) and
// the Summary); here P^T and dS^T live in TMEM as the A operands of the dV/dK
// MMAs, and dS^T is also staged once in shared memory as the B operand of dQ^T.
//
// Warps: 0-3 P/dS (one thread per key row = TMEM lane), 4-7 dQ drain (one
// thread per head-dim row of dQ^T), 8 MMA issue + TMEM allocation, 9 TMA.
// TMEM columns: dV [0,d) dK [d,2d); S buffers [2d,2d+128) (two of 64 columns:
// S^T of a step, then its P^T in bf16); dP buffers [2d+128,2d+256) (dP^T, then
// dS^T in bf16, then the step's dQ^T once dK has read dS^T). Steps alternate
// buffers, so S^T runs two steps ahead of the P/dS warps and dP^T one.
#include "exp2_poly.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

#include <cmath>

namespace fa {
using namespace ptx;

namespace bwdk {

constexpr int BN = 128;   // keys per unit
constexpr int BMQ = 64;   // query rows per step
constexpr int NUM_THREADS = 384;   // 3 warpgroups: P/dS, dQ drain, MMA/TMA (+2 idle warps)
constexpr int MMA_WARP = 8;
constexpr int TMA_WARP = 9;
// Register split (launch: 168 per thread = 65536 / 384 rounded down to 8):
// 128 * (REGS_PDS + REGS_DRAIN + REGS_CONTROL) <= 384 * 168.
constexpr int REGS_PDS = 232;
constexpr int REGS_DRAIN = 120;
constexpr int REGS_CONTROL = 152;
constexpr int NSTAGE = 4;
constexpr int MAX_SEQ_SMEM = 1024;

template <int D>
struct Cfg {
  static constexpr int CHUNKS = D / 64;
  static constexpr int KV_CHUNK = 128 * 128;
  static constexpr int KV_TILE = CHUNKS * KV_CHUNK;
  static constexpr int Q_CHUNK = 64 * 128;
  static constexpr int Q_TILE = CHUNKS * Q_CHUNK;
  static constexpr int ST_LSE = 2 * Q_TILE;            // offsets inside a stage
  static constexpr int ST_D = ST_LSE + 256;
  static constexpr int STAGE_TX = 2 * Q_TILE + 512;
  static constexpr int STAGE_BYTES = (STAGE_TX + 1023) & ~1023;
  static constexpr int DS_BYTES = 128 * 128;            // dS^T [128 keys][64 q] bf16
  static constexpr int K_OFF = 0;
  static constexpr int V_OFF = KV_TILE;
  static constexpr int ST_OFF = 2 * KV_TILE;
  static constexpr int DS_OFF = ST_OFF + NSTAGE * STAGE_BYTES;
  static constexpr int BAR_OFF = DS_OFF + DS_BYTES;   // one dS^T staging buffer
  static constexpr int B_KVFULL = 0, B_KVEMPTY = 1, B_QDFULL = 2, B_QDEMPTY = 2 + NSTAGE,
                       B_SFULL = 2 + 2 * NSTAGE,  // [2]
                       B_DPFULL = B_SFULL + 2,    // [2]
                       // P/dS ready: one barrier per buffer. A single barrier
                       // could be arrived on for steps i and i+1 before the MMA
                       // thread waits on step i (S^T(i+1) is issued early), and
                       // a parity wait cannot tell phases two apart.
                       B_PREADY = B_DPFULL + 2,   // [2]
                       B_DSREADY = B_PREADY + 2,  // [2]
                       B_DQFULL = B_DSREADY + 2,  // [2]
                       B_DQEMPTY = B_DQFULL + 2,  // [2]
                       B_DSBEMPTY = B_DQEMPTY + 2,  // staging buffer free (once per step)
                       B_ACCFULL = B_DSBEMPTY + 1, B_ACCEMPTY = B_ACCFULL + 1,
                       B_DRAIN = B_ACCEMPTY + 1, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int CU_OFF = MISC_OFF + 16;
  static constexpr int SMEM_BYTES = CU_OFF + (MAX_SEQ_SMEM + 1) * 4 + 1024;
  // dV, dK accumulators; two S^T buffers (also P^T) and two dP^T buffers (also
  // dS^T, then dQ^T), so later steps' S^T/dP^T MMAs run during step i's math.
  static constexpr uint32_t TM_DV = 0, TM_DK = D, TM_SB = 2 * D, TM_DB = 2 * D + 128;
  static constexpr uint32_t IDESC_SDP = idesc_bf16(128, 64, false, false);  // S^T, dP^T
  static constexpr uint32_t IDESC_ACC = idesc_bf16(128, D, false, true);    // dV, dK (A in TMEM)
  static constexpr uint32_t IDESC_DQ = idesc_bf16(D, 64, true, true);       // dQ^T
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// X^T (TMEM, 128 keys x 64 q) = Kt (128 x D, K-major) * Qb (64 x D, K-major)^T
template <int D>
__device__ __forceinline__ void issue_kq(uint32_t tm, uint32_t kt, uint32_t qb) {
  using C = Cfg<D>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    mma_ss(tm, sdesc_sw128(kt + (kk >> 2) * C::KV_CHUNK + (kk & 3) * 32, C::KV_CHUNK, 1024),
           sdesc_sw128(qb + (kk >> 2) * C::Q_CHUNK + (kk & 3) * 32, C::Q_CHUNK, 1024),
           C::IDESC_SDP, kk > 0 ? 1u : 0u);
  }
}

// Acc (TMEM, 128 keys x D) (+)= A^T (TMEM, 128 keys x 64 q, bf16) * Xb (64 q x D, MN-major)
template <int D>
__device__ __forceinline__ void issue_acc(uint32_t tm_acc, uint32_t tm_a, uint32_t xb, bool acc) {
  using C = Cfg<D>;
#pragma unroll
  for (int kk = 0; kk < BMQ / 16; ++kk) {
    mma_ts(tm_acc, tm_a + kk * 8, sdesc_sw128(xb + kk * 2048, C::Q_CHUNK, 1024), C::IDESC_ACC,
           (acc || kk > 0) ? 1u : 0u);
  }
}

// dQ^T (TMEM, D x 64 q) = Kt^T (D x 128 keys, MN-major A) * dS^T (128 keys x 64 q, MN-major B)
template <int D>
__device__ __forceinline__ void issue_dq(uint32_t tm, uint32_t kt, uint32_t dsb) {
  using C = Cfg<D>;
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    mma_ss(tm, sdesc_sw128(kt + kk * 2048, C::KV_CHUNK, 1024),
           sdesc_sw128(dsb + kk * 2048, C::DS_BYTES, 1024), C::IDESC_DQ, kk > 0 ? 1u : 0u);
  }
}

// Role timeline for tuning (CTA 0 only, when a trace buffer is armed).
#define FA_TRACE(ev, step)                                                        \
  do {                                                                            \
    if (p.trace != nullptr && blockIdx.x == 0 && (step) < (uint32_t)TRACE_STEPS) \
      p.trace[(ev) * TRACE_STEPS + (step)] = clock64();                           \
  } while (0)

struct StepInfo {
  int h, m;
};

__device__ __forceinline__ StepInfo step_of(int i, int cost, int m_first, int g, int group) {
  StepInfo s;
  const int hh = i / cost;
  s.h = g * group + hh;
  s.m = m_first + (i - hh * cost);
  return s;
}

__device__ __forceinline__ int first_qblock(const Unit& u, int causal) {
  if (!causal) return 0;
  int r0 = u.m * BN - (u.k_len - u.q_len);
  r0 = r0 > 0 ? r0 : 0;
  return r0 / BMQ;
}

template <int D, int POLY8>
__global__ void __launch_bounds__(NUM_THREADS, 1) bwd_kernel(const __grid_constant__ BwdParams p) {
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
    mbar_init(BAR(C::B_KVFULL), 1);
    mbar_init(BAR(C::B_KVEMPTY), 1);
    for (int s = 0; s < NSTAGE; ++s) {
      mbar_init(BAR(C::B_QDFULL + s), 1);
      mbar_init(BAR(C::B_QDEMPTY + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(BAR(C::B_SFULL + b), 1);
      mbar_init(BAR(C::B_DPFULL + b), 1);
      mbar_init(BAR(C::B_DQFULL + b), 1);
      mbar_init(BAR(C::B_DQEMPTY + b), 128);
      mbar_init(BAR(C::B_PREADY + b), 128);
      mbar_init(BAR(C::B_DSREADY + b), 128);
    }
    mbar_init(BAR(C::B_DSBEMPTY), 1);
    mbar_init(BAR(C::B_ACCFULL), 1);
    mbar_init(BAR(C::B_ACCEMPTY), 128);
    mbar_init(BAR(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_do);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  // packed boundaries in shared memory when they fit (query list, then the key
  // list when it differs; the host stores the two back to back)
  const int ncu = p.k_off ? 2 * (p.nseq + 1) : p.nseq + 1;
  const bool cu_in_smem = p.cu != nullptr && ncu <= MAX_SEQ_SMEM + 1;
  if (cu_in_smem)
    for (int i = threadIdx.x; i < ncu; i += NUM_THREADS) cu_s[i] = p.cu[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const SchedSpec spec{cu_in_smem ? cu_s : p.cu, p.nseq, p.Sq, p.Sk, p.Hkv, p.causal, BN, BMQ, 1,
                       p.hblock, nullptr, p.k_off};
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
      uint32_t it = 0;
      int u_it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        if (u.cost == 0) continue;
        const int g = u.head;
        const int n = u.cost * group;
        const int m_first = first_qblock(u, p.causal);
        const long long pbase = pad_start(u.seq, u.q_start);
        if (u_it > 0) {
          ok = mbar_wait(BAR(C::B_KVEMPTY), (u_it - 1) & 1, wc, SITE_BWD_KV_EMPTY);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(BAR(C::B_KVFULL), 2 * C::KV_TILE);
        for (int c = 0; c < C::CHUNKS; ++c) {
          tma_load_3d(base + C::K_OFF + c * C::KV_CHUNK, &p.tm_k, BAR(C::B_KVFULL), c * 64, g,
                      u.k_start + u.m * BN);
          tma_load_3d(base + C::V_OFF + c * C::KV_CHUNK, &p.tm_v, BAR(C::B_KVFULL), c * 64, g,
                      u.k_start + u.m * BN);
        }
        ++u_it;
        for (int i = 0; i < n; ++i) {
          const StepInfo st = step_of(i, u.cost, m_first, g, group);
          const int s = it % NSTAGE;
          if (it >= (uint32_t)NSTAGE) {
            ok = mbar_wait(BAR(C::B_QDEMPTY + s), ((it / NSTAGE) - 1) & 1, wc, SITE_BWD_QD_EMPTY);
            if (!ok) break;
          }
          const uint32_t sb = base + C::ST_OFF + s * C::STAGE_BYTES;
          const uint32_t full = BAR(C::B_QDFULL + s);
          mbar_arrive_expect_tx(full, C::STAGE_TX);
          const int row = u.q_start + st.m * BMQ;
          for (int c = 0; c < C::CHUNKS; ++c) {
            tma_load_3d(sb + c * C::Q_CHUNK, &p.tm_q, full, c * 64, st.h, row);
            tma_load_3d(sb + C::Q_TILE + c * C::Q_CHUNK, &p.tm_do, full, c * 64, st.h, row);
          }
          const long long off = (long long)st.h * p.pad_hstride + pbase + (long long)st.m * BMQ;
          bulk_load(sb + C::ST_LSE, p.lse2 + off, 256, full);
          bulk_load(sb + C::ST_D, p.delta + off, 256, full);
          ++it;
        }
      }
      if (!ok) {
        for (uint32_t i = it > (uint32_t)NSTAGE ? it - NSTAGE : 0; i < it; ++i)
          drain_wait(BAR(C::B_QDFULL + i % NSTAGE), (i / NSTAGE) & 1, 100000000ull);
        if (u_it > 0) drain_wait(BAR(C::B_KVFULL), (u_it - 1) & 1, 100000000ull);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      Walker w;
      w.init(spec);
      uint32_t it = 0;
      int u_it = 0;
      bool ok = true;
      const uint32_t kt = base + C::K_OFF, vt = base + C::V_OFF;
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        if (u.cost == 0) continue;
        const int n = u.cost * group;
        // Two sync points per step, each probing all it needs at once:
        //   A(i): P(i) ready, Q(i+2) loaded, dQ^T(i-1) drained
        //         -> dV(i), S^T(i+2) (into the S buffer dV(i) has just read),
        //            dP^T(i+1) (into the dP buffer the drain has just emptied)
        //   B(i): dS(i) ready -> dK(i), dQ^T(i) (into the dP buffer of step i,
        //         after dK(i) has read its dS^T)
        // S^T runs two steps ahead of the P/dS warps and dP^T one. The unit
        // prologue issues S^T(0), S^T(1) and dP^T(0).
        for (int j = 0; j < 2 && j < n && ok; ++j) {
          const uint32_t st = it + j, b = st & 1;
          const bool dqe = j == 0 && st >= 2;            // dP buffer b last held dQ^T(st-2)
          ok = mbar_wait3(BAR(C::B_KVFULL), u_it & 1, SITE_BWD_KV_FULL,
                          BAR(C::B_QDFULL + st % NSTAGE), (st / NSTAGE) & 1, SITE_BWD_QD_FULL,
                          dqe ? BAR(C::B_DQEMPTY + b) : BAR(C::B_KVFULL),
                          dqe ? ((st >> 1) - 1) & 1 : u_it & 1, SITE_BWD_DQ_EMPTY, wc);
          if (!ok) break;
          tc_fence_after();
          const uint32_t sbj = base + C::ST_OFF + (st % NSTAGE) * C::STAGE_BYTES;
          issue_kq<D>(tmem + C::TM_SB + 64 * b, kt, sbj);
          tc_commit(BAR(C::B_SFULL + b));
          if (j == 0) {
            issue_kq<D>(tmem + C::TM_DB + 64 * b, vt, sbj + C::Q_TILE);
            tc_commit(BAR(C::B_DPFULL + b));
          }
        }
        for (int i = 0; i < n && ok; ++i, ++it) {
          const uint32_t b = it & 1, b1 = b ^ 1;
          const int s = it % NSTAGE;
          const uint32_t sb = base + C::ST_OFF + s * C::STAGE_BYTES;
          const bool more = i + 1 < n, more2 = i + 2 < n;
          const uint32_t st1 = it + 1, st2 = it + 2;
          const uint32_t sb1 = base + C::ST_OFF + (st1 % NSTAGE) * C::STAGE_BYTES;
          const uint32_t sb2 = base + C::ST_OFF + (st2 % NSTAGE) * C::STAGE_BYTES;
          // ---- sync point A(i)
          {
            const uint32_t bq = more2 ? BAR(C::B_QDFULL + st2 % NSTAGE) : BAR(C::B_PREADY + b);
            const uint32_t pq = more2 ? (st2 / NSTAGE) & 1 : (it >> 1) & 1;
            const bool dqe = more && st1 >= 2;           // dP buffer b1 last held dQ^T(it-1)
            const uint32_t bd = dqe ? BAR(C::B_DQEMPTY + b1) : BAR(C::B_PREADY + b);
            const uint32_t pd = dqe ? ((st1 >> 1) - 1) & 1 : (it >> 1) & 1;
            ok = mbar_wait3(BAR(C::B_PREADY + b), (it >> 1) & 1, SITE_BWD_P_READY, bq, pq,
                            SITE_BWD_QD_FULL, bd, pd, SITE_BWD_DQ_EMPTY, wc);
            if (!ok) break;
            FA_TRACE(TR_MMA_P, it);
            if (i == 0 && u_it > 0) {
              ok = mbar_wait(BAR(C::B_ACCEMPTY), (u_it - 1) & 1, wc, SITE_BWD_ACC_FULL);
              if (!ok) break;
            }
            tc_fence_after();
            issue_acc<D>(tmem + C::TM_DV, tmem + C::TM_SB + 64 * b, sb + C::Q_TILE, i > 0);
            if (more2) {
              issue_kq<D>(tmem + C::TM_SB + 64 * b, kt, sb2);                         // S^T(i+2)
              tc_commit(BAR(C::B_SFULL + b));
            }
            if (more) {
              issue_kq<D>(tmem + C::TM_DB + 64 * b1, vt, sb1 + C::Q_TILE);            // dP^T(i+1)
              tc_commit(BAR(C::B_DPFULL + b1));
            }
          }
          // ---- sync point B(i)
          ok = mbar_wait(BAR(C::B_DSREADY + b), (it >> 1) & 1, wc, SITE_BWD_DS_READY);
          if (!ok) break;
          FA_TRACE(TR_MMA_DS, it);
          tc_fence_after();
          issue_acc<D>(tmem + C::TM_DK, tmem + C::TM_DB + 64 * b, sb, i > 0);       // dK += dS^T Q
          issue_dq<D>(tmem + C::TM_DB + 64 * b, kt, base + C::DS_OFF);
          tc_commit(BAR(C::B_DQFULL + b));
          tc_commit(BAR(C::B_DSBEMPTY));
          tc_commit(BAR(C::B_QDEMPTY + s));
          if (!more) {
            tc_commit(BAR(C::B_ACCFULL));
            tc_commit(BAR(C::B_KVEMPTY));
          }
        }
        ++u_it;
      }
      if (!ok) {
        tc_commit(BAR(C::B_DRAIN));
        drain_wait(BAR(C::B_DRAIN), 0, 100000000ull);
      }
    }
  }
  } else if (warp < 4) {
    regs_inc<REGS_PDS>();
    // ------------------------------------------------------------ P^T / dS^T
    const int j = warp * 32 + lane;                       // key row within the block
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const float sl2 = p.scale_log2;
    Walker w;
    w.init(spec);
    uint32_t it = 0;
    int u_it = 0;
    bool ok = true;
    uint8_t* dsb_base = smem + C::DS_OFF;
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!w.seek(snake_index(k, G, cta), u)) break;
      const int g = u.head;
      const int key = u.m * BN + j;                       // key index within the sequence
      const bool key_ok = key < u.k_len;
      __nv_bfloat16* dk_row = p.dk + (((long long)u.k_start + key) * p.Hkv + g) * D;
      __nv_bfloat16* dv_row = p.dv + (((long long)u.k_start + key) * p.Hkv + g) * D;
      if (u.cost == 0) {                                   // keys no query sees
        if (key_ok) {
          for (int c = 0; c < D; c += 8) {
            *reinterpret_cast<uint4*>(dk_row + c) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(dv_row + c) = make_uint4(0, 0, 0, 0);
          }
        }
        continue;
      }
      const int n = u.cost * group;
      const int m_first = first_qblock(u, p.causal);
      // query q (within the sequence) sees this key iff q >= qmin
      const int qmin = p.causal ? key - (u.k_len - u.q_len) : -(1 << 30);
      for (int i = 0; i < n; ++i, ++it) {
        const StepInfo st = step_of(i, u.cost, m_first, g, group);
        const int s = it % NSTAGE;
        const uint8_t* stage = smem + C::ST_OFF + s * C::STAGE_BYTES;
        const float* nlse_s = reinterpret_cast<const float*>(stage + C::ST_LSE);  // -LSE*log2e
        const float* nd_s = reinterpret_cast<const float*>(stage + C::ST_D);      // -D
        ok = mbar_wait(BAR(C::B_QDFULL + s), (it / NSTAGE) & 1, wc, SITE_BWD_QD_FULL);
        if (!ok) break;
        const uint32_t b = it & 1;
        const uint32_t t_s = tmem + lane_off + C::TM_SB + 64 * b;
        const uint32_t t_dp = tmem + lane_off + C::TM_DB + 64 * b;
        // S^T(i) and dP^T(i) are both issued well ahead: load them in one TMEM
        // round trip (dP^T is ready no later than S^T in the MMA order).
        ok = mbar_wait3(BAR(C::B_SFULL + b), (it >> 1) & 1, SITE_BWD_S_FULL,
                        BAR(C::B_DPFULL + b), (it >> 1) & 1, SITE_BWD_DP_FULL,
                        BAR(C::B_SFULL + b), (it >> 1) & 1, SITE_BWD_S_FULL, wc);
        if (!ok) break;
        if (j == 0) FA_TRACE(TR_PDS_S, it);
        tc_fence_after();
        uint32_t sa[64], dpa[64];
        tmem_ld64x2(t_s, sa, t_dp, dpa);
        // The row arrays hold -LSE*log2(e) and -D, so both phases are packed
        // fp32 pairs: x = s*scale*log2e - LSE*log2e (one FFMA2 per pair) and
        // dS = P * (dP - D) (one FADD2 + one FMUL2 per pair).
        uint64_t p2[BMQ / 2];
        {
          // columns c with q0 + c < qmin are masked; a key past the sequence masks all
          const int cmin = key_ok ? qmin - st.m * BMQ : BMQ;
          const uint64_t sl2x2 = f2pack(sl2, sl2);
          const bool mask = __any_sync(0xffffffffu, cmin > 0);
#pragma unroll
          for (int c = 0; c < BMQ; c += 4) {
            const float4 l4 = *reinterpret_cast<const float4*>(nlse_s + c);
            float x[4];
            f2unpack(ffma2(f2pack(u2f(sa[c]), u2f(sa[c + 1])), sl2x2, f2pack(l4.x, l4.y)), x[0],
                     x[1]);
            f2unpack(ffma2(f2pack(u2f(sa[c + 2]), u2f(sa[c + 3])), sl2x2, f2pack(l4.z, l4.w)),
                     x[2], x[3]);
            float pe[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              pe[e] = ((c + e) & 7) < POLY8 ? exp2_poly(x[e]) : ex2_mufu(x[e]);
              if (mask) pe[e] = (c + e) < cmin ? 0.f : pe[e];
            }
            p2[c / 2] = f2pack(pe[0], pe[1]);
            p2[c / 2 + 1] = f2pack(pe[2], pe[3]);
          }
        }
        {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float lo, hi;
            f2unpack(p2[c], lo, hi);
            pk[c] = pack_bf16x2(lo, hi);
          }
          tmem_st32(t_s, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(C::B_PREADY + b));
        if (j == 0) FA_TRACE(TR_PDS_P, it);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < BMQ; c += 4) {
          const float4 d4 = *reinterpret_cast<const float4*>(nd_s + c);
          float d0, d1, d2, d3;
          f2unpack(fmul2(p2[c / 2], fadd2(f2pack(u2f(dpa[c]), u2f(dpa[c + 1])), f2pack(d4.x, d4.y))),
                   d0, d1);
          f2unpack(fmul2(p2[c / 2 + 1],
                         fadd2(f2pack(u2f(dpa[c + 2]), u2f(dpa[c + 3])), f2pack(d4.z, d4.w))),
                   d2, d3);
          pk[c / 2] = pack_bf16x2(d0, d1);
          pk[c / 2 + 1] = pack_bf16x2(d2, d3);
        }
        if (j == 0) FA_TRACE(TR_PDS_DP, it);
        if (it >= 1) {   // the staging buffer still feeds dQ^T(it-1) until that completes
          ok = mbar_wait(BAR(C::B_DSBEMPTY), (it - 1) & 1, wc, SITE_BWD_DS_READY);
          if (!ok) break;
        }
        tmem_st32(t_dp, pk);
        {
          // dS^T row j -> shared memory, [128 keys][64 q] with the 128-byte swizzle
          uint8_t* row = dsb_base + j * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *reinterpret_cast<uint4*>(row + ((c ^ (j & 7)) << 4)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(C::B_DSREADY + b));
        if (j == 0) FA_TRACE(TR_PDS_DS, it);
      }
      if (!ok) break;
      // unit epilogue: dV, dK rows of this key
      ok = mbar_wait(BAR(C::B_ACCFULL), u_it & 1, wc, SITE_BWD_ACC_FULL);
      if (!ok) break;
      tc_fence_after();
      ++u_it;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        const float mul = which ? p.scale : 1.0f;
        __nv_bfloat16* dst = which ? dk_row : dv_row;
        const uint32_t col = which ? C::TM_DK : C::TM_DV;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          uint32_t a[32];
          tmem_ld32(tmem + lane_off + col + c, a);
          uint32_t q[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) q[e] = pack_bf16x2(u2f(a[2 * e]) * mul, u2f(a[2 * e + 1]) * mul);
          if (key_ok) {
            uint4* o4 = reinterpret_cast<uint4*>(dst + c);
            o4[0] = make_uint4(q[0], q[1], q[2], q[3]);
            o4[1] = make_uint4(q[4], q[5], q[6], q[7]);
            o4[2] = make_uint4(q[8], q[9], q[10], q[11]);
            o4[3] = make_uint4(q[12], q[13], q[14], q[15]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(BAR(C::B_ACCEMPTY));
    }
  } else {
    regs_dec<REGS_DRAIN>();
    // ------------------------------------------------------------ dQ drain
    const int dd = (warp & 3) * 32 + lane;                // head-dim index = TMEM lane
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    Walker w;
    w.init(spec);
    uint32_t it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!w.seek(snake_index(k, G, cta), u)) break;
      if (u.cost == 0) continue;
      const int n = u.cost * group;
      const int m_first = first_qblock(u, p.causal);
      for (int i = 0; i < n; ++i, ++it) {
        const StepInfo st = step_of(i, u.cost, m_first, u.head, group);
        const uint32_t b = it & 1;
        ok = mbar_wait(BAR(C::B_DQFULL + b), (it >> 1) & 1, wc, SITE_BWD_DQ_FULL);
        if (!ok) break;
        if (dd == 0) FA_TRACE(TR_DRN_FULL, it);
        tc_fence_after();
        uint32_t a[64];
        tmem_ld64(tmem + lane_off + C::TM_DB + 64 * b, a);
        tc_fence_before();
        mbar_arrive(BAR(C::B_DQEMPTY + b));
        const int q0 = st.m * BMQ;
        const int nvalid = u.q_len - q0;
        float* dst = p.dq_acc + (((long long)u.q_start + q0) * p.Hq + st.h) * D + dd;
        const long long rstride = (long long)p.Hq * D;
        if (nvalid >= BMQ) {
#pragma unroll
          for (int c = 0; c < BMQ; ++c) atomicAdd(dst + c * rstride, u2f(a[c]));
        } else {
#pragma unroll
          for (int c = 0; c < BMQ; ++c)
            if (c < nvalid) atomicAdd(dst + c * rstride, u2f(a[c]));
        }
        if (dd == 0) FA_TRACE(TR_DRN_DONE, it);
      }
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

// -D and -LSE*log2e into the padded row arrays, and their padding rows; zero
// the dQ accumulator when there is one (one-pass kernel). A warp takes 32
// consecutive query rows of one head. Each row's O and dO are read by a group
// of lanes, 16 bytes (8 values) per lane: D/8 lanes rounded up to a power of
// two, so one pass of the warp covers 4, 2, 1 or 1 rows (D = 64, 128, 192,
// 256); the loads of eight passes go out together. The 32 results then go
// out as one coalesced store per array (the arrays are head-major). The
// remaining warps write the padding rows [q_len, round_up(q_len, 128)) of each
// (sequence, head): LSE = +inf, D = 0, so a block's padded query rows
// contribute exact zeros.
template <int D>
struct PreGroup {
  static constexpr int LANES = D / 8;                       // lanes with data
  static constexpr int G = LANES <= 8 ? 8 : LANES <= 16 ? 16 : 32;
  static constexpr int RPW = 32 / G;                        // rows per pass of a warp
  static constexpr int PASSES = 32 / RPW;                   // passes over 32 rows
  static constexpr int BATCH = PASSES < 8 ? PASSES : 8;     // passes loaded together
};

template <int D>
__global__ void bwd_pre_kernel(BwdParams p, BwdAux aux) {
  using PG = PreGroup<D>;
  const int T = p.total_q;
  const int nchunk = (T + 31) / 32;
  const long long nrowwarps = (long long)p.Hq * nchunk;
  const long long nwork = nrowwarps + (long long)p.Hq * p.nseq;
  const int lane = threadIdx.x & 31;
  const int gl = lane & (PG::G - 1);                         // lane within the row's group
  const int c = gl * 8;                                      // this lane's 8 columns
  const int sub = lane / PG::G;                              // row of the pass
  const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
  for (long long wi = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); wi < nwork;
       wi += warps) {
    if (wi < nrowwarps) {
      const int h = (int)(wi / nchunk), t0 = (int)(wi - (long long)h * nchunk) * 32;
      float mine = 0.f;                                      // lane L: D of row t0 + L
#pragma unroll 1
      for (int i0 = 0; i0 < PG::PASSES; i0 += PG::BATCH) {
        uint4 ov[PG::BATCH], gv[PG::BATCH];
#pragma unroll
        for (int b = 0; b < PG::BATCH; ++b) {
          const int t = t0 + (i0 + b) * PG::RPW + sub;
          ov[b] = gv[b] = make_uint4(0, 0, 0, 0);
          if (t < T && c < D) {
            const long long r = (long long)t * p.Hq + h;
            ov[b] = *reinterpret_cast<const uint4*>(aux.o + r * D + c);
            gv[b] = *reinterpret_cast<const uint4*>(aux.dout + r * D + c);
            if (p.dq_acc) {
              float4* zr = reinterpret_cast<float4*>(p.dq_acc + r * D + c);
              zr[0] = make_float4(0.f, 0.f, 0.f, 0.f);
              zr[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        }
#pragma unroll
        for (int b = 0; b < PG::BATCH; ++b) {
          const __nv_bfloat162* o2 = reinterpret_cast<const __nv_bfloat162*>(&ov[b]);
          const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&gv[b]);
          float acc = 0.f;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 of = __bfloat1622float2(o2[e]);
            const float2 gf = __bfloat1622float2(g2[e]);
            acc = fmaf(of.x, gf.x, acc);
            acc = fmaf(of.y, gf.y, acc);
          }
#pragma unroll
          for (int sh = PG::G / 2; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
#pragma unroll
          for (int j = 0; j < PG::RPW; ++j) {
            const float v = __shfl_sync(0xffffffffu, acc, j * PG::G);
            if (lane == (i0 + b) * PG::RPW + j) mine = v;
          }
        }
      }
      const int t = t0 + lane;
      if (t < T) {
        int seq, q_start;
        if (p.cu) {
          int lo = 0, hi = p.nseq;                           // last seq with cu[seq] <= t
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (p.cu[mid] <= t) lo = mid; else hi = mid;
          }
          seq = lo;
          q_start = p.cu[lo];
        } else {
          seq = t / p.Sq;
          q_start = seq * p.Sq;
        }
        const int row = t - q_start;
        const float lse = aux.lse[(p.cu ? 0ll : (long long)seq * aux.lse_seqstride) +
                                  (long long)h * aux.lse_hstride + (p.cu ? t : row)];
        const long long pi = (long long)h * p.pad_hstride + pad_start(seq, q_start) + row;
        const_cast<float*>(p.lse2)[pi] = -lse * 1.4426950408889634f;
        const_cast<float*>(p.delta)[pi] = -mine;
      }
    } else {
      const long long k = wi - nrowwarps;
      const int h = (int)(k / p.nseq), seq = (int)(k - (long long)h * p.nseq);
      int q_start, q_len;
      if (p.cu) {
        q_start = p.cu[seq];
        q_len = p.cu[seq + 1] - q_start;
      } else {
        q_start = seq * p.Sq;
        q_len = p.Sq;
      }
      const int end = (q_len + 127) & ~127;
      const long long base = (long long)h * p.pad_hstride + pad_start(seq, q_start);
      for (int row = q_len + lane; row < end; row += 32) {
        const_cast<float*>(p.lse2)[base + row] = -INFINITY;
        const_cast<float*>(p.delta)[base + row] = 0.f;
      }
    }
  }
}

__global__ void bwd_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                   long long n8, float scale) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (long long)gridDim.x * blockDim.x) {
    const float4 a = reinterpret_cast<const float4*>(acc)[2 * i];
    const float4 b = reinterpret_cast<const float4*>(acc)[2 * i + 1];
    uint4 o;
    o.x = pack_bf16x2(a.x * scale, a.y * scale);
    o.y = pack_bf16x2(a.z * scale, a.w * scale);
    o.z = pack_bf16x2(b.x * scale, b.y * scale);
    o.w = pack_bf16x2(b.z * scale, b.w * scale);
    reinterpret_cast<uint4*>(dq)[i] = o;
  }
}

}  // namespace bwdk

template <int D, int POLY8>
static cudaError_t launch_main(const BwdParams& p, int grid, cudaStream_t stream) {
  auto kern = bwdk::bwd_kernel<D, POLY8>;
  const int smem = bwdk::Cfg<D>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, bwdk::NUM_THREADS, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const BwdParams& p, const BwdAux& aux, int d, int grid, int grid_q,
                       cudaStream_t stream, int poly8, int mode, int pdl) {
  if (mode == 0 && d != 128) return cudaErrorNotSupported;
  if (d != 64 && d != 128 && d != 192 && d != 256) return cudaErrorNotSupported;
  const long long rows = (long long)p.total_q * p.Hq;
  if (rows > 0) {
    // 8 warps per block, RPW rows per warp
    // one warp per 32 rows of a head plus one per (sequence, head) for the
    // padding; 8 warps per block
    const long long work = (long long)p.Hq * ((p.total_q + 31) / 32 + p.nseq);
    const long long b = (work + 7) / 8;
    const int blocks = (int)(b < 65535ll * 8 ? b : 65535ll * 8);
    if (d == 128)
      bwdk::bwd_pre_kernel<128><<<blocks, 256, 0, stream>>>(p, aux);
    else if (d == 192)
      bwdk::bwd_pre_kernel<192><<<blocks, 256, 0, stream>>>(p, aux);
    else if (d == 256)
      bwdk::bwd_pre_kernel<256><<<blocks, 256, 0, stream>>>(p, aux);
    else
      bwdk::bwd_pre_kernel<64><<<blocks, 256, 0, stream>>>(p, aux);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (mode != 0) {
    cudaEvent_t ev0, ev1;
    take_events(1, &ev0, &ev1);
    if (ev0) cudaEventRecord(ev0, stream);
    const cudaError_t e =
        mode == 2 ? launch_bwd_pair(p, p.total_k > 0 ? grid : 0, p.total_q > 0 ? grid_q : 0,
                                    stream, poly8)
                  : launch_bwd_split(p, d, p.total_k > 0 ? grid : 0, p.total_q > 0 ? grid_q : 0,
                                     stream, poly8, pdl);
    if (ev1) cudaEventRecord(ev1, stream);
    return e;
  }
  if (p.total_k > 0) {
    cudaEvent_t ev0, ev1;
    take_events(1, &ev0, &ev1);
    if (ev0) cudaEventRecord(ev0, stream);
    cudaError_t e;
    switch (poly8) {
      case 0: e = launch_main<128, 0>(p, grid, stream); break;
      case 2: e = launch_main<128, 2>(p, grid, stream); break;
      case 4: e = launch_main<128, 4>(p, grid, stream); break;
      default: e = cudaErrorInvalidValue;
    }
    if (ev1) cudaEventRecord(ev1, stream);
    if (e != cudaSuccess) return e;
  }
  if (rows > 0) {
    const long long n8 = rows * d / 8;
    const int blocks = (int)(n8 / 256 + 1 < 152 * 16 ? n8 / 256 + 1 : 152 * 16);
    bwdk::bwd_convert_kernel<<<blocks, 256, 0, stream>>>(p.dq_acc, aux.dq, n8, p.scale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace fa
