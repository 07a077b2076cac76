// Backward attention for sm_103a in two passes, with every accumulator in
// tensor memory and no atomics:
//
//   dK/dV pass: one persistent CTA per SM walks (sequence, 128-key block, KV
//     head) units longest-first; for each query head of the KV group and each
//     block of 128 query rows that sees the keys:
//        S^T  = K Q^T            P^T  = exp2(S^T * scale*log2e - LSE*log2e)
//        dP^T = V dO^T           dS^T = P^T o (dP^T - D)
//        dV  += P^T dO           dK  += dS^T Q
//     dK and dV stay in TMEM for the whole unit and are written once.
//   dQ pass: one persistent CTA per SM walks (sequence, 128-query block, query
//     head) units longest-first; for each 128-key block the rows see:
//        S  = Q K^T              P  = exp2(S * scale*log2e - LSE*log2e)
//        dP = dO V^T             dS = P o (dP - D)
//        dQ += dS K
//     and writes dQ once, scaled, in bf16.
//
// The pages' backward ("FlashAttention-4: Algorithm and Kernel Pipelining
// Co-Design for Asymmetric Hardware Scaling", abstract item (3) and the
// Summary) keeps accumulators and the P/dS operands in tensor memory to cut
// shared-memory traffic and atomic adds, with dQ accumulated by atomics into an
// fp32 buffer. This form recomputes S and dP once more (seven 128x128xd MMAs
// per block pair instead of five) and in exchange: every MMA is a full-rate
// M=128, N=128 shape; P^T/dS^T (and dS) live only in TMEM as the A operand of
// the accumulating MMA, so shared memory carries nothing but TMA tiles; dQ
// needs no fp32 buffer, no atomics and no convert pass; and the result is
// deterministic.
//
// Both kernels: 12 warps. Warps 0-3 and 4-7 are two compute warpgroups that
// split the columns of each score tile (half each, one thread per TMEM lane =
// tile row); warp 8 allocates TMEM and one of its threads issues the MMAs;
// warp 9 is the TMA producer; warps 10-11 only complete the register split.
// A warpgroup writes its bf16 half of P^T/dS^T/dS over the first half of its
// own fp32 columns, so with 128-column tiles the A operand of the accumulating
// MMA sits in columns [0,32) and [64,96) of its buffer (64-column tiles:
// [0,16) and [32,48); 32-column tiles: [0,8) and [16,24)). Head dims 64 and
// 128 step over 128 query rows / 128 keys; 192 and 256 over smaller steps
// (kv_step_rows, q_block_keys below).
#include "exp2_poly.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "sched.cuh"

#include <cmath>

namespace fa {
using namespace ptx;

namespace bsplit {

constexpr int BN = 128;            // keys per block
constexpr int BM = 128;            // query rows per block
constexpr int NUM_THREADS = 384;
constexpr int MMA_WARP = 8;
constexpr int TMA_WARP = 9;
// Launch gives 168 registers per thread (65536 / 384 rounded down to 8);
// 128 * (2 * REGS_COMPUTE + REGS_CONTROL) <= 384 * 168.
constexpr int REGS_COMPUTE = 200;
constexpr int REGS_CONTROL = 104;
constexpr int SMEM_LIMIT = 232448;
constexpr int MAX_SEQ_SMEM = 200;  // packed boundaries kept in shared memory up to this

template <int D, int ROWS = 128>
struct Tile {
  static constexpr int CHUNKS = D / 64;        // 128-byte column chunks per row
  static constexpr int CHUNK = ROWS * 128;     // ROWS rows x 128 bytes, 128B swizzle
  static constexpr int BYTES = CHUNKS * CHUNK; // one tile of ROWS rows
};

// Step sizes by head dim. Up to 128: 128 query rows per dK/dV step, 128 keys
// per dQ block. 192: 64 and 64 (dK/dV pass: dV 192 + dK 192 + S^T 64 + dP^T 64
// = 512 TMEM columns, ~216 KB of tiles; dQ pass: S 2 x 64 + dP 64 + dQ 192
// columns, ~216 KB). 256: dV and dK alone would fill TMEM, so a dK/dV unit
// accumulates one 128-column half of them (S^T and dP^T are recomputed for
// each half) over 64-row steps, with 64 KB K and V tiles, two Q slots and one
// dO slot (~226 KB); the dQ pass takes 32-key blocks (S 2 x 32 + dP 32 + dQ
// 256 columns; Q and dO 64 KB each, five 16 KB K/V slots).
template <int D>
constexpr int kv_step_rows() { return D > 128 ? 64 : 128; }
template <int D>
constexpr int q_block_keys() { return D > 192 ? 32 : D > 128 ? 64 : 128; }
template <int D>
constexpr int acc_cols() { return D > 192 ? 128 : D; }   // dV/dK columns per dK/dV unit

// dK/dV pass layout. Q slots are held from S^T(i) to dK(i), the longest span,
// so Q gets three slots and dO two. The -LSE*log2(e) and -D values of a
// step's 128 query rows (one per score column) go through a two-slot ring of
// their own, filled by the producer and released by the compute warps. The
// layout leaves no room for aligning the dynamic shared memory by hand: the
// kernel requires (and checks) that it starts on a 1024-byte boundary.
template <int D>
struct CfgKV {
  using T = Tile<D>;
  static constexpr int BMS = kv_step_rows<D>();       // query rows per step
  static constexpr int DA = acc_cols<D>();             // accumulator columns (dV, dK)
  static constexpr int HALVES = D / DA;                // units per key block and KV head
  using QT = Tile<D, BMS>;                             // a Q or dO step tile
  static constexpr int NQ = D > 192 ? 2 : 3, NDO = D > 192 ? 1 : 2, NLD = 2;
  static constexpr int LD_BYTES = 2 * BMS * 4;        // [-LSE*log2e x BMS][-D x BMS]
  static constexpr int K_OFF = 0, V_OFF = T::BYTES, Q_OFF = 2 * T::BYTES,
                       DO_OFF = Q_OFF + NQ * QT::BYTES, LD_OFF = DO_OFF + NDO * QT::BYTES,
                       BAR_OFF = LD_OFF + NLD * LD_BYTES;
  static constexpr int B_KVFULL = 0, B_KVEMPTY = 1, B_QFULL = 2, B_QEMPTY = B_QFULL + NQ,
                       B_DOFULL = B_QEMPTY + NQ, B_DOEMPTY = B_DOFULL + NDO,
                       B_LDFULL = B_DOEMPTY + NDO, B_LDEMPTY = B_LDFULL + NLD,
                       B_SFULL = B_LDEMPTY + NLD, B_DPFULL = B_SFULL + 1,
                       B_PREADY = B_DPFULL + 1, B_DSREADY = B_PREADY + 1,
                       B_ACCFULL = B_DSREADY + 1, B_DRAIN = B_ACCFULL + 1, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int CU_OFF = MISC_OFF + 16;
  static constexpr int SMEM_BYTES = CU_OFF + (MAX_SEQ_SMEM + 1) * 4;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "dK/dV pass shared memory");
  // TMEM: dV [0,DA), dK [DA,2DA), S^T/P^T [2DA,2DA+BMS), dP^T/dS^T [2DA+BMS,2DA+2BMS)
  static constexpr uint32_t TM_DV = 0, TM_DK = DA, TM_SB = 2 * DA, TM_DB = 2 * DA + BMS;
  static_assert(2 * DA + 2 * BMS <= 512, "TMEM columns");
  static constexpr uint32_t IDESC_S = idesc_bf16(128, BMS, false, false);  // S^T, dP^T
  static constexpr uint32_t IDESC_ACC = idesc_bf16(128, DA, false, true);  // dV, dK
};

// dQ pass layout: Q and dO of the unit, and a ring of K/V tiles in the order
// K_0 V_0 K_1 V_1 ...; K_j is held from S(j) to dQ(j), two steps, so the ring
// has five slots.
template <int D>
struct CfgQ {
  using T = Tile<D>;
  static constexpr int BNS = q_block_keys<D>();       // keys per block
  using KT = Tile<D, BNS>;                             // a K or V block tile
  static constexpr int NKV = 5;
  static constexpr int Q_OFF = 0, DO_OFF = T::BYTES, KV_OFF = 2 * T::BYTES,
                       BAR_OFF = KV_OFF + NKV * KT::BYTES;
  static constexpr int B_QFULL = 0, B_QEMPTY = 1, B_KVFULL = 2, B_KVEMPTY = B_KVFULL + NKV,
                       B_SFULL = B_KVEMPTY + NKV,   // [2]
                       B_DPFULL = B_SFULL + 2, B_DSREADY = B_DPFULL + 1,
                       B_DQFULL = B_DSREADY + 1, B_DRAIN = B_DQFULL + 1, NBAR = B_DRAIN + 1;
  static constexpr int MISC_OFF = BAR_OFF + NBAR * 8;
  static constexpr int CU_OFF = MISC_OFF + 16;
  static constexpr int SMEM_BYTES = CU_OFF + (MAX_SEQ_SMEM + 1) * 4 + 1024;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "dQ pass shared memory");
  // TMEM: S/dS buffers [0,BNS) and [BNS,2BNS), dP [2BNS,3BNS), dQ [3BNS,3BNS+D)
  static constexpr uint32_t TM_S = 0, TM_DP = 2 * BNS, TM_DQ = 3 * BNS;
  static_assert(3 * BNS + D <= 512, "TMEM columns");
  static constexpr uint32_t IDESC_S = idesc_bf16(128, BNS, false, false);  // S, dP
  static constexpr uint32_t IDESC_DQ = idesc_bf16(128, D, false, true);    // dQ
};

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// Wait that ignores the abort flag: lets in-flight async work land before an
// aborting CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return;
  }
}

// X (TMEM, 128 x BROWS fp32) = A (128 rows x D) * B (BROWS rows x D)^T, both
// K-major tiles.
template <int D, uint32_t IDESC, int BROWS = 128>
__device__ __forceinline__ void mma_abt(uint32_t tm, uint32_t a, uint32_t b) {
  using TA = Tile<D>;
  using TB = Tile<D, BROWS>;
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint32_t k_off = (kk & 3) * 32;
    mma_ss(tm, sdesc_sw128(a + (kk >> 2) * TA::CHUNK + k_off, TA::CHUNK, 1024),
           sdesc_sw128(b + (kk >> 2) * TB::CHUNK + k_off, TB::CHUNK, 1024), IDESC,
           kk > 0 ? 1u : 0u);
  }
}

// Acc (TMEM, 128 x D) (+)= X (TMEM, 128 x KROWS bf16; each warpgroup's half of
//                          the K dimension packed into the first half of its
//                          KROWS/2 fp32 columns: [0, KROWS/4) and [KROWS/2, 3KROWS/4))
//                          * Y (KROWS rows x D tile, MN-major B)
template <int D, uint32_t IDESC, int KROWS = 128>
__device__ __forceinline__ void mma_acc(uint32_t tm_acc, uint32_t tm_x, uint32_t y, bool acc) {
  using TY = Tile<D, KROWS>;
  constexpr int KS = KROWS / 16;                  // K steps; half of them per warpgroup
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    const uint32_t ta = tm_x + (kk < KS / 2 ? kk * 8 : KROWS / 2 + (kk - KS / 2) * 8);
    mma_ts(tm_acc, ta, sdesc_sw128(y + kk * 2048, TY::CHUNK, 1024), IDESC,
           (acc || kk > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ uint32_t pack2(uint64_t v) {
  float lo, hi;
  f2unpack(v, lo, hi);
  return pack_bf16x2(lo, hi);
}

// COLS fp32 values (COLS/2 pairs) -> bf16 pairs stored over the first COLS/2 columns.
// TMEM row loads of a warpgroup's COLS columns (64, 32 or 16), and stores of
// COLS/2 columns (bf16 pairs over the first half of those columns).
template <int COLS>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[COLS]) {
  if constexpr (COLS == 64)
    tmem_ld64(taddr, r);
  else if constexpr (COLS == 32)
    tmem_ld32(taddr, r);
  else
    tmem_ld16(taddr, r);
}
template <int COLS>
__device__ __forceinline__ void tmem_st_half(uint32_t taddr, const uint32_t* r) {
  if constexpr (COLS == 64)
    tmem_st32(taddr, r);
  else if constexpr (COLS == 32)
    tmem_st16(taddr, r);
  else
    tmem_st8(taddr, r);
}

template <int COLS = 64>
__device__ __forceinline__ void store_bf16_half(uint32_t taddr, const uint64_t (&v2)[COLS / 2]) {
  uint32_t pk[COLS / 2];
#pragma unroll
  for (int c = 0; c < COLS / 2; ++c) pk[c] = pack2(v2[c]);
  tmem_st_half<COLS>(taddr, pk);
}

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

// First block of QROWS query rows that sees the unit's keys.
template <int QROWS = BM>
__device__ __forceinline__ int first_qblock(const Unit& u, int causal) {
  if (!causal) return 0;
  int r0 = u.m * BN - (u.k_len - u.q_len);
  r0 = r0 > 0 ? r0 : 0;
  return r0 / QROWS;
}

// Writes one warpgroup's half (D/2 columns) of a TMEM accumulator row to a bf16 row.
template <int D>
__device__ __forceinline__ void store_acc_half(uint32_t t_acc, __nv_bfloat16* dst, float mul,
                                               bool ok) {
  // 32-byte stores where the row allows (each thread writes its own row piece,
  // so a warp's store instruction touches 32 different lines: fewer, wider
  // stores halve those line accesses); 16-byte ones otherwise
  const bool wide = (reinterpret_cast<uintptr_t>(dst) & 31) == 0;
#pragma unroll 1
  for (int c = 0; c < D / 2; c += 32) {
    uint32_t a[32];
    tmem_ld32(t_acc + c, a);
    uint32_t q[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) q[e] = pack_bf16x2(u2f(a[2 * e]) * mul, u2f(a[2 * e + 1]) * mul);
    if (ok) {
      if (wide) {
        const uint32_t q0[8] = {q[0], q[1], q[2], q[3], q[4], q[5], q[6], q[7]};
        const uint32_t q1[8] = {q[8], q[9], q[10], q[11], q[12], q[13], q[14], q[15]};
        st_global_v8(dst + c, q0);
        st_global_v8(dst + c + 16, q1);
      } else {
        uint4* o4 = reinterpret_cast<uint4*>(dst + c);
        o4[0] = make_uint4(q[0], q[1], q[2], q[3]);
        o4[1] = make_uint4(q[4], q[5], q[6], q[7]);
        o4[2] = make_uint4(q[8], q[9], q[10], q[11]);
        o4[3] = make_uint4(q[12], q[13], q[14], q[15]);
      }
    }
  }
}

// Role timeline for tuning (CTA 0 only, when a trace buffer is armed).
#define FA_TRACE(ev, step)                                                        \
  do {                                                                            \
    if (p.trace != nullptr && blockIdx.x == 0 && (step) < (uint32_t)TRACE_STEPS) \
      p.trace[(ev) * TRACE_STEPS + (step)] = clock64();                           \
  } while (0)
#define FA_TRACE_VAL(ev, step, val)                                               \
  do {                                                                            \
    if (p.trace != nullptr && blockIdx.x == 0 && (step) < (uint32_t)TRACE_STEPS) \
      p.trace[(ev) * TRACE_STEPS + (step)] = (val);                               \
  } while (0)

template <int D>
__device__ __forceinline__ void zero_half(__nv_bfloat16* dst) {
#pragma unroll
  for (int c = 0; c < D / 2; c += 8) *reinterpret_cast<uint4*>(dst + c) = make_uint4(0, 0, 0, 0);
}

// ============================================================== dK/dV pass
template <int D, int POLY8>
__global__ void __launch_bounds__(NUM_THREADS, 1) dkdv_kernel(const __grid_constant__ BwdParams p) {
  using C = CfgKV<D>;
  using T = Tile<D>;
  using QT = typename C::QT;
  constexpr int BMS = C::BMS;                           // query rows per step
  constexpr int COLS = BMS / 2;                         // score columns per warpgroup
  constexpr int DA = C::DA, HALVES = C::HALVES;         // unit head = KV head * HALVES + half
  // a dQ pass launched as this grid's programmatic dependent may start
  // launching now; its CTAs take SMs as this grid's CTAs exit
  griddep_launch_dependents();
  extern __shared__ __align__(1024) uint8_t smem_al[];
  uint32_t base;                                        // opaque to the compiler: checked, not assumed
  asm volatile("{\n\t.reg .u64 t;\n\tcvta.to.shared.u64 t, %1;\n\tcvt.u32.u64 %0, t;\n\t}"
               : "=r"(base)
               : "l"(smem_al));
  if (base & 1023u) {                                   // 128B-swizzled tiles need 1024 B
    if (threadIdx.x == 0) atomicCAS(p.err, 0, SITE_SMEM_ALIGN);
    return;
  }
  uint8_t* smem = smem_al;
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
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(BAR(C::B_QFULL + s), 1);
      mbar_init(BAR(C::B_QEMPTY + s), 1);
    }
    for (int s = 0; s < C::NDO; ++s) {
      mbar_init(BAR(C::B_DOFULL + s), 1);
      mbar_init(BAR(C::B_DOEMPTY + s), 1);
    }
    for (int s = 0; s < C::NLD; ++s) {
      mbar_init(BAR(C::B_LDFULL + s), 1);
      mbar_init(BAR(C::B_LDEMPTY + s), 256);
    }
    mbar_init(BAR(C::B_SFULL), 1);
    mbar_init(BAR(C::B_DPFULL), 1);
    mbar_init(BAR(C::B_PREADY), 256);
    mbar_init(BAR(C::B_DSREADY), 256);
    mbar_init(BAR(C::B_ACCFULL), 1);
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

  const SchedSpec spec{cu_in_smem ? cu_s : p.cu, p.nseq, p.Sq, p.Sk, p.Hkv * HALVES, p.causal,
                       BN, BMS, 1, p.hblock * HALVES, nullptr, p.k_off};
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
      int u_it = 0;
      bool ok = true;
      uint32_t nq = 0, nd = 0, nl = 0;                    // Q / dO / row-value loads issued
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        if (u.cost == 0) continue;
        const int n = u.cost * group;
        const int m_first = first_qblock<BMS>(u, p.causal);
        // The first steps' Q/dO (as many as both rings hold) need only free
        // ring slots: they go out before the wait for the previous unit to
        // release K/V. More would wait for this unit's own dV/dK, which need
        // its K/V.
        constexpr int LEAD = C::NQ < C::NDO ? C::NQ : C::NDO;
        const int lead = n < LEAD ? n : LEAD;
        for (int i = 0; i <= n; ++i) {
          if (i == lead) {
            if (u_it > 0) {
              ok = mbar_wait(BAR(C::B_KVEMPTY), (u_it - 1) & 1, wc, SITE_DKDV_KV_EMPTY);
              if (!ok) break;
            }
            mbar_arrive_expect_tx(BAR(C::B_KVFULL), 2 * T::BYTES);
            FA_TRACE(TR_KV_KVLOAD, nq - (uint32_t)lead);
            const int krow = u.k_start + u.m * BN;
            for (int c = 0; c < T::CHUNKS; ++c) {
              tma_load_3d(base + C::K_OFF + c * T::CHUNK, &p.tm_k, BAR(C::B_KVFULL), c * 64,
                          u.head / HALVES, krow);
              tma_load_3d(base + C::V_OFF + c * T::CHUNK, &p.tm_v, BAR(C::B_KVFULL), c * 64,
                          u.head / HALVES, krow);
            }
            ++u_it;
          }
          if (i == n) break;
          // Q(s) goes into slot s % NQ once dK(s - NQ) is done, dO(s) into slot
          // s % NDO once dV(s - NDO) is done.
          const StepInfo st = step_of(i, u.cost, m_first, u.head / HALVES, group);
          const int row = u.q_start + st.m * BMS;
          const int sq = nq % C::NQ, sd = nd % C::NDO;
          if (nq >= (uint32_t)C::NQ) {
            ok = mbar_wait(BAR(C::B_QEMPTY + sq), ((nq / C::NQ) - 1) & 1, wc, SITE_DKDV_Q_EMPTY);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(BAR(C::B_QFULL + sq), QT::BYTES);
          for (int c = 0; c < QT::CHUNKS; ++c)
            tma_load_3d(base + C::Q_OFF + sq * QT::BYTES + c * QT::CHUNK, &p.tm_q,
                        BAR(C::B_QFULL + sq), c * 64, st.h, row);
          ++nq;
          if (nd >= (uint32_t)C::NDO) {
            ok = mbar_wait(BAR(C::B_DOEMPTY + sd), ((nd / C::NDO) - 1) & 1, wc,
                           SITE_DKDV_DO_EMPTY);
            if (!ok) break;
          }
          mbar_arrive_expect_tx(BAR(C::B_DOFULL + sd), QT::BYTES);
          for (int c = 0; c < QT::CHUNKS; ++c)
            tma_load_3d(base + C::DO_OFF + sd * QT::BYTES + c * QT::CHUNK, &p.tm_do,
                        BAR(C::B_DOFULL + sd), c * 64, st.h, row);
          ++nd;
          // the step's row values, released by the compute warps after dS
          const int sl = nl % C::NLD;
          if (nl >= (uint32_t)C::NLD) {
            ok = mbar_wait(BAR(C::B_LDEMPTY + sl), ((nl / C::NLD) - 1) & 1, wc,
                           SITE_DKDV_LD_EMPTY);
            if (!ok) break;
          }
          const long long off = (long long)st.h * p.pad_hstride + pad_start(u.seq, u.q_start) +
                                (long long)st.m * BMS;
          const uint32_t ld = base + C::LD_OFF + sl * C::LD_BYTES;
          mbar_arrive_expect_tx(BAR(C::B_LDFULL + sl), C::LD_BYTES);
          bulk_load(ld, p.lse2 + off, BMS * 4, BAR(C::B_LDFULL + sl));
          bulk_load(ld + BMS * 4, p.delta + off, BMS * 4, BAR(C::B_LDFULL + sl));
          ++nl;
        }
      }
      if (!ok) {
        // let the copies already issued land before the CTA exits
        for (uint32_t i = nq > (uint32_t)C::NQ ? nq - C::NQ : 0; i < nq; ++i)
          drain_wait(BAR(C::B_QFULL + i % C::NQ), (i / C::NQ) & 1, 100000000ull);
        for (uint32_t i = nd > (uint32_t)C::NDO ? nd - C::NDO : 0; i < nd; ++i)
          drain_wait(BAR(C::B_DOFULL + i % C::NDO), (i / C::NDO) & 1, 100000000ull);
        for (uint32_t i = nl > (uint32_t)C::NLD ? nl - C::NLD : 0; i < nl; ++i)
          drain_wait(BAR(C::B_LDFULL + i % C::NLD), (i / C::NLD) & 1, 100000000ull);
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
      const uint32_t tSB = tmem + C::TM_SB, tDB = tmem + C::TM_DB;
      auto qslot = [&](uint32_t s) { return base + C::Q_OFF + (s % C::NQ) * QT::BYTES; };
      auto dslot = [&](uint32_t s) { return base + C::DO_OFF + (s % C::NDO) * QT::BYTES; };
      uint32_t half_off = 0;                              // this unit's dV/dK columns in Q, dO
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        if (u.cost == 0) continue;
        const int n = u.cost * group;
        half_off = (uint32_t)(u.head % HALVES) * (DA / 64) * QT::CHUNK;
        // Per step two sync points, each probing everything it needs at once
        // (every memory access of this thread waits for the MMAs it has
        // queued, so the probes of a sync point go out together):
        //   A(i): P^T(i) ready (+ Q(i+1) loaded) -> dV(i), S^T(i+1)
        //   B(i): dS^T(i) ready (+ dO(i+1) loaded) -> dK(i), dP^T(i+1)
        // S^T(i+1) reuses the S buffer right after dV(i) has read P^T(i) from
        // it (MMAs of one thread execute in order); dP^T(i+1) likewise after
        // dK(i). The compute warps write the previous unit's dK/dV out before
        // they arrive for step 0 of this unit, so A(0) also orders dV(0)
        // (which overwrites the accumulator) after that read.
        ok = mbar_wait3(BAR(C::B_KVFULL), u_it & 1, SITE_DKDV_KV_FULL,
                        BAR(C::B_QFULL + it % C::NQ), (it / C::NQ) & 1, SITE_DKDV_Q_FULL,
                        BAR(C::B_DOFULL + it % C::NDO), (it / C::NDO) & 1, SITE_DKDV_DO_FULL, wc);
        if (!ok) break;
        FA_TRACE(TR_KV_PRO, it);
        tc_fence_after();
        mma_abt<D, C::IDESC_S, BMS>(tSB, kt, qslot(it));
        tc_commit(BAR(C::B_SFULL));
        mma_abt<D, C::IDESC_S, BMS>(tDB, vt, dslot(it));
        tc_commit(BAR(C::B_DPFULL));
        // K and V feed only S^T and dP^T: they are released once the unit's
        // last dP^T is issued, so the next unit's copy overlaps this one's tail
        if (n == 1) tc_commit(BAR(C::B_KVEMPTY));
        for (int i = 0; i < n && ok; ++i, ++it) {
          const bool more = i + 1 < n;
          const uint32_t it1 = it + 1;
          // ---- A(i)
          ok = mbar_wait3(BAR(C::B_PREADY), it & 1, SITE_DKDV_P_READY,
                          more ? BAR(C::B_QFULL + it1 % C::NQ) : BAR(C::B_PREADY),
                          more ? (it1 / C::NQ) & 1 : it & 1, SITE_DKDV_Q_FULL,
                          BAR(C::B_PREADY), it & 1, SITE_DKDV_P_READY, wc);
          if (!ok) break;
          FA_TRACE(TR_KV_A, it);
          tc_fence_after();
          mma_acc<D, C::IDESC_ACC, BMS>(tmem + C::TM_DV, tSB, dslot(it) + half_off, i > 0);
          tc_commit(BAR(C::B_DOEMPTY + it % C::NDO));
          if (more) {
            mma_abt<D, C::IDESC_S, BMS>(tSB, kt, qslot(it1));
            tc_commit(BAR(C::B_SFULL));
          }
          // ---- B(i)
          ok = mbar_wait3(BAR(C::B_DSREADY), it & 1, SITE_DKDV_DS_READY,
                          more ? BAR(C::B_DOFULL + it1 % C::NDO) : BAR(C::B_DSREADY),
                          more ? (it1 / C::NDO) & 1 : it & 1, SITE_DKDV_DO_FULL,
                          BAR(C::B_DSREADY), it & 1, SITE_DKDV_DS_READY, wc);
          if (!ok) break;
          FA_TRACE(TR_KV_B, it);
          tc_fence_after();
          mma_acc<D, C::IDESC_ACC, BMS>(tmem + C::TM_DK, tDB, qslot(it) + half_off, i > 0);
          tc_commit(BAR(C::B_QEMPTY + it % C::NQ));
          if (more) {
            mma_abt<D, C::IDESC_S, BMS>(tDB, vt, dslot(it1));
            tc_commit(BAR(C::B_DPFULL));
            if (i + 2 == n) tc_commit(BAR(C::B_KVEMPTY));
          } else {
            tc_commit(BAR(C::B_ACCFULL));
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
  } else {
    regs_inc<REGS_COMPUTE>();
    // ------------------------------------------------------------ P^T / dS^T
    const int wg = warp >> 2;                             // query-column half
    const int lg = warp & 3;
    const int j = lg * 32 + lane;                         // key row within the block
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int c0 = wg * COLS;
    const uint32_t t_s = tmem + lane_off + C::TM_SB + c0;
    const uint32_t t_dp = tmem + lane_off + C::TM_DB + c0;
    const float sl2 = p.scale_log2;
    Walker w;
    w.init(spec);
    uint32_t it = 0;
    int u_it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!w.seek(snake_index(k, G, cta), u)) break;
      const int g = u.head / HALVES;
      const int key = u.m * BN + j;                       // key index within the sequence
      const bool key_ok = key < u.k_len;
      const long long krow = ((long long)u.k_start + key) * p.Hkv + g;
      const int col0 = (u.head % HALVES) * DA + wg * (DA / 2);
      __nv_bfloat16* dk_row = p.dk + krow * D + col0;
      __nv_bfloat16* dv_row = p.dv + krow * D + col0;
      if (u.cost == 0) {                                   // keys no query sees
        if (key_ok) {
          zero_half<DA>(dk_row);
          zero_half<DA>(dv_row);
        }
        continue;
      }
      const int n = u.cost * group;
      const int m_first = first_qblock<BMS>(u, p.causal);
      // query q (within the sequence) sees this key iff q >= qmin
      const int qmin = p.causal ? key - (u.k_len - u.q_len) : -(1 << 30);
      for (int i = 0; i < n; ++i, ++it) {
        const StepInfo st = step_of(i, u.cost, m_first, g, group);
        // -LSE*log2(e) and -D of this warpgroup's 64 query rows (padding rows
        // hold -inf and 0, so they contribute exact zeros), from the ring
        const uint32_t sl = it % C::NLD;
        const float4* nl4 =
            reinterpret_cast<const float4*>(smem + C::LD_OFF + sl * C::LD_BYTES) + c0 / 4;
        const float4* nd4 = nl4 + BMS / 4;
        ok = mbar_wait(BAR(C::B_LDFULL + sl), (it / C::NLD) & 1, wc, SITE_DKDV_LD_FULL);
        if (!ok) break;
        // -LSE*log2(e) into registers while S^T is still on its way
        float4 l4r[COLS / 4];
#pragma unroll
        for (int c = 0; c < COLS / 4; ++c) l4r[c] = nl4[c];
        ok = mbar_wait(BAR(C::B_SFULL), it & 1, wc, SITE_DKDV_S_FULL);
        if (!ok) break;
        if (threadIdx.x == 0) FA_TRACE(TR_KV_S, it);
        tc_fence_after();
        uint32_t sa[COLS];
        tmem_ld_cols<COLS>(t_s, sa);
        // columns c with q0 + c < qmin are masked; a key past the sequence masks all
        const int cmin = key_ok ? qmin - (st.m * BMS + c0) : COLS;
        const bool mask = __any_sync(0xffffffffu, cmin > 0);
        uint64_t p2[COLS / 2];
        {
          const uint64_t sl2x2 = f2pack(sl2, sl2);
#pragma unroll
          for (int c = 0; c < COLS; c += 4) {
            const float4 l4 = l4r[c / 4];
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
        store_bf16_half<COLS>(t_s, p2);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(C::B_PREADY));
        if (threadIdx.x == 0) FA_TRACE(TR_KV_P, it);
        ok = mbar_wait(BAR(C::B_DPFULL), it & 1, wc, SITE_DKDV_DP_FULL);
        if (!ok) break;
        if (threadIdx.x == 0) FA_TRACE(TR_KV_DP, it);
        tc_fence_after();
        uint32_t dpa[COLS];
        tmem_ld_cols<COLS>(t_dp, dpa);
        uint32_t pk[COLS / 2];
#pragma unroll
        for (int c = 0; c < COLS; c += 4) {
          const float4 d4 = nd4[c / 4];
          pk[c / 2] = pack2(fmul2(p2[c / 2], fadd2(f2pack(u2f(dpa[c]), u2f(dpa[c + 1])),
                                                   f2pack(d4.x, d4.y))));
          pk[c / 2 + 1] = pack2(fmul2(p2[c / 2 + 1],
                                      fadd2(f2pack(u2f(dpa[c + 2]), u2f(dpa[c + 3])),
                                            f2pack(d4.z, d4.w))));
        }
        mbar_arrive(BAR(C::B_LDEMPTY + sl));
        tmem_st_half<COLS>(t_dp, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(C::B_DSREADY));
        if (threadIdx.x == 0) FA_TRACE(TR_KV_DS, it);
      }
      if (!ok) break;
      // unit epilogue: this warpgroup's half of the dV and dK rows of this key
      ok = mbar_wait(BAR(C::B_ACCFULL), u_it & 1, wc, SITE_DKDV_ACC_FULL);
      if (!ok) break;
      if (threadIdx.x == 0) FA_TRACE(TR_KV_EPI, it - 1);
      tc_fence_after();
      ++u_it;
      store_acc_half<DA>(tmem + lane_off + C::TM_DV + wg * (DA / 2), dv_row, 1.0f, key_ok);
      store_acc_half<DA>(tmem + lane_off + C::TM_DK + wg * (DA / 2), dk_row, p.scale, key_ok);
      if (threadIdx.x == 0) FA_TRACE(TR_KV_EPI_END, it - 1);
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

// ============================================================== dK/dV pass, CTA pairs
// The same pass with each unit's MMAs issued over a cluster of two CTAs
// (cta_group::2, M = 256). A unit is 256 keys; CTA r of the pair owns keys
// [128r, 128r+128): its K/V tiles, its TMEM accumulators and its P^T/dS^T
// columns. The step's Q and dO tiles are split the way each M=256 MMA takes
// its B operand: S^T and dP^T read query rows [64r, 64r+64) (all head-dim
// columns, K-major) from CTA r, dV and dK read head-dim columns [64r, 64r+64)
// of all 128 query rows (MN-major) from CTA r. Each CTA thus reads half of
// every B operand from its own shared memory, the traffic that bounds the
// one-CTA form. CTA 0 issues every MMA; CTA 1's TMA completions (forwarded
// by its warp 10) and its P^T/dS^T readiness reach CTA 0's barriers as remote
// arrivals, and CTA 0's commits are multicast to both CTAs.
// A Q/dO slot holds [rows half: two 64-row x 128-byte chunks][columns half:
// one 128-row x 128-byte chunk], 32 KB, the same size as in the one-CTA form.
constexpr int PAIR_BN = 256;     // keys per unit (two CTAs)

// X (TMEM, 256 keys x 128 q over the pair) = K/V tile (this CTA's 128 rows,
// K-major) * (64 rows of this CTA's half of B, K-major)^T
template <uint32_t IDESC>
__device__ __forceinline__ void mma_abt_pair(uint32_t tm, uint32_t a, uint32_t b) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t a_off = (kk >> 2) * (128 * 128) + (kk & 3) * 32;
    const uint32_t b_off = (kk >> 2) * (64 * 128) + (kk & 3) * 32;
    mma_ss_pair(tm, sdesc_sw128(a + a_off, 128 * 128, 1024), sdesc_sw128(b + b_off, 64 * 128, 1024),
                IDESC, kk > 0 ? 1u : 0u);
  }
}
// Acc (TMEM, 256 keys x 128 over the pair) (+)= X (TMEM bf16, columns [0,32)
// and [64,96)) * Y (128 q rows x this CTA's 64 head-dim columns, MN-major)
template <uint32_t IDESC>
__device__ __forceinline__ void mma_acc_pair(uint32_t tm_acc, uint32_t tm_x, uint32_t y, bool acc) {
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t ta = tm_x + (kk < 4 ? kk * 8 : 64 + (kk - 4) * 8);
    mma_ts_pair(tm_acc, ta, sdesc_sw128(y + kk * 2048, 128 * 128, 1024), IDESC,
                (acc || kk > 0) ? 1u : 0u);
  }
}

__device__ __forceinline__ int first_qblock_pair(const Unit& u, int causal) {
  if (!causal) return 0;
  int r0 = u.m * PAIR_BN - (u.k_len - u.q_len);
  r0 = r0 > 0 ? r0 : 0;
  return r0 / BM;
}

template <int POLY8>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    dkdv_pair_kernel(const __grid_constant__ BwdParams p) {
  constexpr int D = 128;
  using C = CfgKV<D>;
  using T = Tile<D>;
  constexpr uint32_t IDESC_S2 = idesc_bf16(256, 128, false, false);   // S^T, dP^T
  constexpr uint32_t IDESC_ACC2 = idesc_bf16(256, D, false, true);    // dV, dK
  constexpr uint32_t ROWS_HALF = 0, COLS_HALF = 2 * 64 * 128;         // offsets inside a slot
  extern __shared__ __align__(1024) uint8_t smem_al[];
  uint32_t base;                                        // opaque to the compiler: checked, not assumed
  asm volatile("{\n\t.reg .u64 t;\n\tcvta.to.shared.u64 t, %1;\n\tcvt.u32.u64 %0, t;\n\t}"
               : "=r"(base)
               : "l"(smem_al));
  if (base & 1023u) {                                   // same in both CTAs of the pair
    if (threadIdx.x == 0) atomicCAS(p.err, 0, SITE_SMEM_ALIGN);
    return;
  }
  uint8_t* smem = smem_al;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t bars = base + C::BAR_OFF;
#define BAR(i) (bars + 8u * (uint32_t)(i))
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::MISC_OFF + 4);
  int* cu_s = reinterpret_cast<int*>(smem + C::CU_OFF);

  if (threadIdx.x == 0) {
    // CTA 0's full barriers also count CTA 1's forwarded completion
    const uint32_t fulls = leader ? 2 : 1;
    mbar_init(BAR(C::B_KVFULL), fulls);
    mbar_init(BAR(C::B_KVEMPTY), 1);
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(BAR(C::B_QFULL + s), fulls);
      mbar_init(BAR(C::B_QEMPTY + s), 1);
    }
    for (int s = 0; s < C::NDO; ++s) {
      mbar_init(BAR(C::B_DOFULL + s), fulls);
      mbar_init(BAR(C::B_DOEMPTY + s), 1);
    }
    for (int s = 0; s < C::NLD; ++s) {
      mbar_init(BAR(C::B_LDFULL + s), 1);
      mbar_init(BAR(C::B_LDEMPTY + s), 256);
    }
    mbar_init(BAR(C::B_SFULL), 1);
    mbar_init(BAR(C::B_DPFULL), 1);
    mbar_init(BAR(C::B_PREADY), 512);                  // 16 warps of the pair, 32 each
    mbar_init(BAR(C::B_DSREADY), 512);
    mbar_init(BAR(C::B_ACCFULL), 1);
    mbar_init(BAR(C::B_DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == TMA_WARP && lane == 0) {
    tma_prefetch_desc(&p.tm_q);
    tma_prefetch_desc(&p.tm_q2);
    tma_prefetch_desc(&p.tm_do);
    tma_prefetch_desc(&p.tm_do2);
    tma_prefetch_desc(&p.tm_k);
    tma_prefetch_desc(&p.tm_v);
  }
  if (warp == MMA_WARP) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  // packed boundaries in shared memory when they fit (query list, then the key
  // list when it differs; the host stores the two back to back)
  const int ncu = p.k_off ? 2 * (p.nseq + 1) : p.nseq + 1;
  const bool cu_in_smem = p.cu != nullptr && ncu <= MAX_SEQ_SMEM + 1;
  if (cu_in_smem)
    for (int i = threadIdx.x; i < ncu; i += NUM_THREADS) cu_s[i] = p.cu[i];
  tc_fence_before();
  cluster_sync_all();                                   // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const SchedSpec spec{cu_in_smem ? cu_s : p.cu, p.nseq, p.Sq, p.Sk, p.Hkv, p.causal, PAIR_BN, BM,
                       1, p.hblock, nullptr, p.k_off};
  const WaitCtl wc{p.err, abort_flag, p.timeout_ns};
  const int G = gridDim.x / 2;                          // pairs
  const int cta = blockIdx.x / 2;                       // this pair
  const int group = p.Hq / p.Hkv;

  if (warp >= 8) {
    regs_dec<REGS_CONTROL>();
  if (warp == 11) {
    // spare warp of the control warpgroup
  } else if (warp == 10) {
    // ------------------------------------------------------------ forwarder
    // CTA 1: each of its K/V, Q and dO copies, once landed, counts on CTA 0's
    // barrier of the same slot (same order as the producer issues them).
    if (!leader && lane == 0) {
      Walker w;
      w.init(spec);
      int u_it = 0;
      bool ok = true;
      uint32_t nq = 0, nd = 0;
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        if (u.cost == 0) continue;
        const int n = u.cost * group;
        const int lead = n < 2 ? n : 2;
        for (int i = 0; i <= n; ++i) {
          if (i == lead) {
            ok = mbar_wait(BAR(C::B_KVFULL), u_it & 1, wc, SITE_DKDV_KV_FULL);
            if (!ok) break;
            mbar_arrive_cluster(BAR(C::B_KVFULL), 0, 1);
            ++u_it;
          }
          if (i == n) break;
          ok = mbar_wait(BAR(C::B_QFULL + nq % C::NQ), (nq / C::NQ) & 1, wc, SITE_DKDV_Q_FULL);
          if (!ok) break;
          mbar_arrive_cluster(BAR(C::B_QFULL + nq % C::NQ), 0, 1);
          ++nq;
          ok = mbar_wait(BAR(C::B_DOFULL + nd % C::NDO), (nd / C::NDO) & 1, wc, SITE_DKDV_DO_FULL);
          if (!ok) break;
          mbar_arrive_cluster(BAR(C::B_DOFULL + nd % C::NDO), 0, 1);
          ++nd;
        }
      }
    }
  } else if (warp == TMA_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      Walker w;
      w.init(spec);
      int u_it = 0;
      bool ok = true;
      uint32_t nq = 0, nd = 0, nl = 0;                    // Q / dO / row-value loads issued
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        if (u.cost == 0) continue;
        const int n = u.cost * group;
        const int m_first = first_qblock_pair(u, p.causal);
        const int lead = n < 2 ? n : 2;
        for (int i = 0; i <= n; ++i) {
          if (i == lead) {
            if (u_it > 0) {
              ok = mbar_wait_cl(BAR(C::B_KVEMPTY), (u_it - 1) & 1, wc, SITE_DKDV_KV_EMPTY);
              if (!ok) break;
            }
            mbar_arrive_expect_tx(BAR(C::B_KVFULL), 2 * T::BYTES);
            const int krow = u.k_start + u.m * PAIR_BN + 128 * (int)rank;
            for (int c = 0; c < T::CHUNKS; ++c) {
              tma_load_3d(base + C::K_OFF + c * T::CHUNK, &p.tm_k, BAR(C::B_KVFULL), c * 64,
                          u.head, krow);
              tma_load_3d(base + C::V_OFF + c * T::CHUNK, &p.tm_v, BAR(C::B_KVFULL), c * 64,
                          u.head, krow);
            }
            ++u_it;
          }
          if (i == n) break;
          const StepInfo st = step_of(i, u.cost, m_first, u.head, group);
          const int row = u.q_start + st.m * BM;
          const int sq = nq % C::NQ, sd = nd % C::NDO;
          if (nq >= (uint32_t)C::NQ) {
            ok = mbar_wait_cl(BAR(C::B_QEMPTY + sq), ((nq / C::NQ) - 1) & 1, wc, SITE_DKDV_Q_EMPTY);
            if (!ok) break;
          }
          {
            const uint32_t slot = base + C::Q_OFF + sq * T::BYTES, bq = BAR(C::B_QFULL + sq);
            mbar_arrive_expect_tx(bq, T::BYTES);
            for (int c = 0; c < 2; ++c)                   // rows [64r, 64r+64), all columns
              tma_load_3d(slot + ROWS_HALF + c * (64 * 128), &p.tm_q2, bq, c * 64, st.h,
                          row + 64 * (int)rank);
            tma_load_3d(slot + COLS_HALF, &p.tm_q, bq, 64 * (int)rank, st.h, row);  // columns half
          }
          ++nq;
          if (nd >= (uint32_t)C::NDO) {
            ok = mbar_wait_cl(BAR(C::B_DOEMPTY + sd), ((nd / C::NDO) - 1) & 1, wc,
                              SITE_DKDV_DO_EMPTY);
            if (!ok) break;
          }
          {
            const uint32_t slot = base + C::DO_OFF + sd * T::BYTES, bd = BAR(C::B_DOFULL + sd);
            mbar_arrive_expect_tx(bd, T::BYTES);
            for (int c = 0; c < 2; ++c)
              tma_load_3d(slot + ROWS_HALF + c * (64 * 128), &p.tm_do2, bd, c * 64, st.h,
                          row + 64 * (int)rank);
            tma_load_3d(slot + COLS_HALF, &p.tm_do, bd, 64 * (int)rank, st.h, row);
          }
          ++nd;
          const int sl = nl % C::NLD;
          if (nl >= (uint32_t)C::NLD) {
            ok = mbar_wait(BAR(C::B_LDEMPTY + sl), ((nl / C::NLD) - 1) & 1, wc,
                           SITE_DKDV_LD_EMPTY);
            if (!ok) break;
          }
          const long long off = (long long)st.h * p.pad_hstride + pad_start(u.seq, u.q_start) +
                                (long long)st.m * BM;
          const uint32_t ld = base + C::LD_OFF + sl * C::LD_BYTES;
          mbar_arrive_expect_tx(BAR(C::B_LDFULL + sl), C::LD_BYTES);
          bulk_load(ld, p.lse2 + off, BM * 4, BAR(C::B_LDFULL + sl));
          bulk_load(ld + BM * 4, p.delta + off, BM * 4, BAR(C::B_LDFULL + sl));
          ++nl;
        }
      }
      if (!ok) {
        for (uint32_t i = nq > (uint32_t)C::NQ ? nq - C::NQ : 0; i < nq; ++i)
          drain_wait(BAR(C::B_QFULL + i % C::NQ), (i / C::NQ) & 1, 100000000ull);
        for (uint32_t i = nd > (uint32_t)C::NDO ? nd - C::NDO : 0; i < nd; ++i)
          drain_wait(BAR(C::B_DOFULL + i % C::NDO), (i / C::NDO) & 1, 100000000ull);
        for (uint32_t i = nl > (uint32_t)C::NLD ? nl - C::NLD : 0; i < nl; ++i)
          drain_wait(BAR(C::B_LDFULL + i % C::NLD), (i / C::NLD) & 1, 100000000ull);
        if (u_it > 0) drain_wait(BAR(C::B_KVFULL), (u_it - 1) & 1, 100000000ull);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issue (CTA 0)
    if (leader && lane == 0) {
      Walker w;
      w.init(spec);
      uint32_t it = 0;
      int u_it = 0;
      bool ok = true;
      const uint32_t kt = base + C::K_OFF, vt = base + C::V_OFF;
      const uint32_t tSB = tmem + C::TM_SB, tDB = tmem + C::TM_DB;
      auto qslot = [&](uint32_t s) { return base + C::Q_OFF + (s % C::NQ) * T::BYTES; };
      auto dslot = [&](uint32_t s) { return base + C::DO_OFF + (s % C::NDO) * T::BYTES; };
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        if (u.cost == 0) continue;
        const int n = u.cost * group;
        // Same schedule as the one-CTA form (sync points A and B per step),
        // with pair MMAs and commits multicast to both CTAs.
        ok = mbar_wait3_cl(BAR(C::B_KVFULL), u_it & 1, SITE_DKDV_KV_FULL,
                           BAR(C::B_QFULL + it % C::NQ), (it / C::NQ) & 1, SITE_DKDV_Q_FULL,
                           BAR(C::B_DOFULL + it % C::NDO), (it / C::NDO) & 1, SITE_DKDV_DO_FULL,
                           wc);
        if (!ok) break;
        tc_fence_after();
        mma_abt_pair<IDESC_S2>(tSB, kt, qslot(it) + ROWS_HALF);
        tc_commit_pair(BAR(C::B_SFULL), 0x3);
        mma_abt_pair<IDESC_S2>(tDB, vt, dslot(it) + ROWS_HALF);
        tc_commit_pair(BAR(C::B_DPFULL), 0x3);
        if (n == 1) tc_commit_pair(BAR(C::B_KVEMPTY), 0x3);   // K/V: see the one-CTA form
        for (int i = 0; i < n && ok; ++i, ++it) {
          const bool more = i + 1 < n;
          const uint32_t it1 = it + 1;
          ok = mbar_wait3_cl(BAR(C::B_PREADY), it & 1, SITE_DKDV_P_READY,
                             more ? BAR(C::B_QFULL + it1 % C::NQ) : BAR(C::B_PREADY),
                             more ? (it1 / C::NQ) & 1 : it & 1, SITE_DKDV_Q_FULL,
                             BAR(C::B_PREADY), it & 1, SITE_DKDV_P_READY, wc);
          if (!ok) break;
          FA_TRACE(TR_KV_A, it);
          tc_fence_after();
          mma_acc_pair<IDESC_ACC2>(tmem + C::TM_DV, tSB, dslot(it) + COLS_HALF, i > 0);
          tc_commit_pair(BAR(C::B_DOEMPTY + it % C::NDO), 0x3);
          if (more) {
            mma_abt_pair<IDESC_S2>(tSB, kt, qslot(it1) + ROWS_HALF);
            tc_commit_pair(BAR(C::B_SFULL), 0x3);
          }
          ok = mbar_wait3_cl(BAR(C::B_DSREADY), it & 1, SITE_DKDV_DS_READY,
                             more ? BAR(C::B_DOFULL + it1 % C::NDO) : BAR(C::B_DSREADY),
                             more ? (it1 / C::NDO) & 1 : it & 1, SITE_DKDV_DO_FULL,
                             BAR(C::B_DSREADY), it & 1, SITE_DKDV_DS_READY, wc);
          if (!ok) break;
          FA_TRACE(TR_KV_B, it);
          tc_fence_after();
          mma_acc_pair<IDESC_ACC2>(tmem + C::TM_DK, tDB, qslot(it) + COLS_HALF, i > 0);
          tc_commit_pair(BAR(C::B_QEMPTY + it % C::NQ), 0x3);
          if (more) {
            mma_abt_pair<IDESC_S2>(tDB, vt, dslot(it1) + ROWS_HALF);
            tc_commit_pair(BAR(C::B_DPFULL), 0x3);
            if (i + 2 == n) tc_commit_pair(BAR(C::B_KVEMPTY), 0x3);
          } else {
            tc_commit_pair(BAR(C::B_ACCFULL), 0x3);
          }
        }
        ++u_it;
      }
      // every MMA of this CTA pair has landed before either CTA tears down
      tc_commit_pair(BAR(C::B_DRAIN), 0x3);
      drain_wait(BAR(C::B_DRAIN), 0, 100000000ull);
    }
  }
  } else {
    regs_inc<REGS_COMPUTE>();
    // ------------------------------------------------------------ P^T / dS^T
    const int wg = warp >> 2;                             // query-column half
    const int lg = warp & 3;
    const int j = lg * 32 + lane;                         // key row within this CTA's 128
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int c0 = wg * 64;
    const uint32_t t_s = tmem + lane_off + C::TM_SB + c0;
    const uint32_t t_dp = tmem + lane_off + C::TM_DB + c0;
    const float sl2 = p.scale_log2;
    Walker w;
    w.init(spec);
    uint32_t it = 0;
    int u_it = 0;
    bool ok = true;
    // a warp's 32 threads count once (32) on CTA 0's barrier
    auto ready = [&](uint32_t bar) {
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(bar, 0, 32);
    };
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!w.seek(snake_index(k, G, cta), u)) break;
      const int g = u.head;
      const int key = u.m * PAIR_BN + 128 * (int)rank + j;   // key index within the sequence
      const bool key_ok = key < u.k_len;
      const long long krow = ((long long)u.k_start + key) * p.Hkv + g;
      __nv_bfloat16* dk_row = p.dk + krow * D + wg * (D / 2);
      __nv_bfloat16* dv_row = p.dv + krow * D + wg * (D / 2);
      if (u.cost == 0) {
        if (key_ok) {
          zero_half<D>(dk_row);
          zero_half<D>(dv_row);
        }
        continue;
      }
      const int n = u.cost * group;
      const int m_first = first_qblock_pair(u, p.causal);
      const int qmin = p.causal ? key - (u.k_len - u.q_len) : -(1 << 30);
      for (int i = 0; i < n; ++i, ++it) {
        const StepInfo st = step_of(i, u.cost, m_first, g, group);
        const uint32_t sl = it % C::NLD;
        const float4* nl4 =
            reinterpret_cast<const float4*>(smem + C::LD_OFF + sl * C::LD_BYTES) + c0 / 4;
        const float4* nd4 = nl4 + BM / 4;
        ok = mbar_wait(BAR(C::B_LDFULL + sl), (it / C::NLD) & 1, wc, SITE_DKDV_LD_FULL);
        if (!ok) break;
        float4 l4r[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) l4r[c] = nl4[c];
        ok = mbar_wait_cl(BAR(C::B_SFULL), it & 1, wc, SITE_DKDV_S_FULL);
        if (!ok) break;
        if (threadIdx.x == 0) FA_TRACE(TR_KV_S, it);
        tc_fence_after();
        uint32_t sa[64];
        tmem_ld64(t_s, sa);
        const int cmin = key_ok ? qmin - (st.m * BM + c0) : 64;
        const bool mask = __any_sync(0xffffffffu, cmin > 0);
        uint64_t p2[32];
        {
          const uint64_t sl2x2 = f2pack(sl2, sl2);
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            const float4 l4 = l4r[c / 4];
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
        store_bf16_half(t_s, p2);
        tmem_st_wait();
        tc_fence_before();
        ready(BAR(C::B_PREADY));
        if (threadIdx.x == 0) FA_TRACE(TR_KV_P, it);
        ok = mbar_wait_cl(BAR(C::B_DPFULL), it & 1, wc, SITE_DKDV_DP_FULL);
        if (!ok) break;
        if (threadIdx.x == 0) FA_TRACE(TR_KV_DP, it);
        tc_fence_after();
        uint32_t dpa[64];
        tmem_ld64(t_dp, dpa);
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 64; c += 4) {
          const float4 d4 = nd4[c / 4];
          pk[c / 2] = pack2(fmul2(p2[c / 2], fadd2(f2pack(u2f(dpa[c]), u2f(dpa[c + 1])),
                                                   f2pack(d4.x, d4.y))));
          pk[c / 2 + 1] = pack2(fmul2(p2[c / 2 + 1],
                                      fadd2(f2pack(u2f(dpa[c + 2]), u2f(dpa[c + 3])),
                                            f2pack(d4.z, d4.w))));
        }
        mbar_arrive(BAR(C::B_LDEMPTY + sl));
        tmem_st32(t_dp, pk);
        tmem_st_wait();
        tc_fence_before();
        ready(BAR(C::B_DSREADY));
        if (threadIdx.x == 0) FA_TRACE(TR_KV_DS, it);
      }
      if (!ok) break;
      ok = mbar_wait_cl(BAR(C::B_ACCFULL), u_it & 1, wc, SITE_DKDV_ACC_FULL);
      if (!ok) break;
      tc_fence_after();
      ++u_it;
      store_acc_half<D>(tmem + lane_off + C::TM_DV + wg * (D / 2), dv_row, 1.0f, key_ok);
      store_acc_half<D>(tmem + lane_off + C::TM_DK + wg * (D / 2), dk_row, p.scale, key_ok);
      tc_fence_before();
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync_all();                                   // the peer no longer signals or reads this CTA
  if (warp == MMA_WARP) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
#undef BAR
}

// ============================================================== dQ pass
template <int D, int POLY8>
__global__ void __launch_bounds__(NUM_THREADS, 1) dq_kernel(const __grid_constant__ BwdParams p) {
  using C = CfgQ<D>;
  using T = Tile<D>;
  using KT = typename C::KT;
  constexpr int BNS = C::BNS;                           // keys per block
  constexpr int COLS = BNS / 2;                         // score columns per warpgroup
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
    for (int s = 0; s < C::NKV; ++s) {
      mbar_init(BAR(C::B_KVFULL + s), 1);
      mbar_init(BAR(C::B_KVEMPTY + s), 1);
    }
    mbar_init(BAR(C::B_SFULL + 0), 1);
    mbar_init(BAR(C::B_SFULL + 1), 1);
    mbar_init(BAR(C::B_DPFULL), 1);
    mbar_init(BAR(C::B_DSREADY), 256);
    mbar_init(BAR(C::B_DQFULL), 1);
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

  const SchedSpec spec{cu_in_smem ? cu_s : p.cu, p.nseq, p.Sq, p.Sk, p.Hq, p.causal, BM, BNS, 0,
                       p.hblock_q, nullptr, p.k_off};
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
      uint32_t r = 0;                                     // K/V ring position
      uint32_t pj = 0;                                    // steps loaded (trace index)
      int u_it = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        const int n = u.cost;
        if (n == 0) continue;
        const int kvh = u.head / group;
        const int row = u.q_start + u.m * BM;
        if (u_it > 0) {
          ok = mbar_wait(BAR(C::B_QEMPTY), (u_it - 1) & 1, wc, SITE_DQ_Q_EMPTY);
          if (!ok) break;
        }
        mbar_arrive_expect_tx(BAR(C::B_QFULL), 2 * T::BYTES);
        for (int c = 0; c < T::CHUNKS; ++c) {
          tma_load_3d(base + C::Q_OFF + c * T::CHUNK, &p.tm_q, BAR(C::B_QFULL), c * 64, u.head,
                      row);
          tma_load_3d(base + C::DO_OFF + c * T::CHUNK, &p.tm_do, BAR(C::B_QFULL), c * 64,
                      u.head, row);
        }
        ++u_it;
        for (int jb = 0; jb < n && ok; ++jb) {
          for (int which = 0; which < 2; ++which, ++r) {
            const int s = r % C::NKV;
            if (r >= (uint32_t)C::NKV) {
              ok = mbar_wait(BAR(C::B_KVEMPTY + s), ((r / C::NKV) - 1) & 1, wc, SITE_DQ_KV_EMPTY);
              if (!ok) break;
            }
            if (which == 0) FA_TRACE(TR_Q_KLOAD, pj);
            mbar_arrive_expect_tx(BAR(C::B_KVFULL + s), KT::BYTES);
            const void* tm = which ? static_cast<const void*>(&p.tm_v)
                                   : static_cast<const void*>(&p.tm_k);
            for (int c = 0; c < KT::CHUNKS; ++c)
              tma_load_3d(base + C::KV_OFF + s * KT::BYTES + c * KT::CHUNK, tm,
                          BAR(C::B_KVFULL + s), c * 64, kvh, u.k_start + jb * BNS);
          }
          ++pj;
        }
      }
      if (!ok) {
        for (uint32_t i = r > (uint32_t)C::NKV ? r - C::NKV : 0; i < r; ++i)
          drain_wait(BAR(C::B_KVFULL + i % C::NKV), (i / C::NKV) & 1, 100000000ull);
        if (u_it > 0) drain_wait(BAR(C::B_QFULL), (u_it - 1) & 1, 100000000ull);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      Walker w;
      w.init(spec);
      uint32_t r = 0, sj = 0;
      int u_it = 0;
      bool ok = true;
      const uint32_t qt = base + C::Q_OFF, dot = base + C::DO_OFF;
      auto kv = [&](uint32_t x) { return base + C::KV_OFF + (x % C::NKV) * KT::BYTES; };
      auto full = [&](uint32_t x) { return BAR(C::B_KVFULL + x % C::NKV); };
      auto empty = [&](uint32_t x) { return BAR(C::B_KVEMPTY + x % C::NKV); };
      auto ph = [&](uint32_t x) { return (x / C::NKV) & 1; };
      for (int k = 0; ok; ++k) {
        Unit u;
        if (!w.seek(snake_index(k, G, cta), u)) break;
        const int n = u.cost;
        if (n == 0) continue;
        // K_j sits at ring position r + 2j, V_j at r + 2j + 1. One sync point
        // per step: dS(j) ready (+ V_{j+1}, K_{j+2} loaded) -> dQ += dS(j) K_j,
        // dP(j+1), S(j+2) (into the buffer dQ(j) has just read). S runs two
        // steps ahead of the compute warps, dP one. The compute warps write
        // the previous unit's dQ before they arrive for step 0 of this unit,
        // which orders dQ(0) (overwriting the accumulator) after that read.
        ok = mbar_wait3(BAR(C::B_QFULL), u_it & 1, SITE_DQ_Q_FULL, full(r), ph(r),
                        SITE_DQ_KV_FULL, full(r + 1), ph(r + 1), SITE_DQ_KV_FULL, wc);
        if (!ok) break;
        tc_fence_after();
        mma_abt<D, C::IDESC_S, BNS>(tmem + C::TM_S + BNS * (sj & 1), qt, kv(r));
        tc_commit(BAR(C::B_SFULL + (sj & 1)));
        mma_abt<D, C::IDESC_S, BNS>(tmem + C::TM_DP, dot, kv(r + 1));
        tc_commit(BAR(C::B_DPFULL));
        tc_commit(empty(r + 1));
        if (n == 1) tc_commit(BAR(C::B_QEMPTY));
        if (n > 1) {
          ok = mbar_wait(full(r + 2), ph(r + 2), wc, SITE_DQ_KV_FULL);
          if (!ok) break;
          tc_fence_after();
          mma_abt<D, C::IDESC_S, BNS>(tmem + C::TM_S + BNS * ((sj + 1) & 1), qt, kv(r + 2));
          tc_commit(BAR(C::B_SFULL + ((sj + 1) & 1)));
        }
        for (int jb = 0; jb < n && ok; ++jb, ++sj) {
          const uint32_t b = sj & 1;
          const bool more = jb + 1 < n, more2 = jb + 2 < n;
          const uint32_t rk = r + 2 * jb, rv1 = rk + 3, rk2 = rk + 4;
          ok = mbar_wait3(BAR(C::B_DSREADY), sj & 1, SITE_DQ_DS_READY,
                          more ? full(rv1) : BAR(C::B_DSREADY), more ? ph(rv1) : sj & 1,
                          SITE_DQ_KV_FULL, more2 ? full(rk2) : BAR(C::B_DSREADY),
                          more2 ? ph(rk2) : sj & 1, SITE_DQ_KV_FULL, wc);
          if (!ok) break;
          FA_TRACE(TR_Q_SYNC, sj);
          tc_fence_after();
          mma_acc<D, C::IDESC_DQ, BNS>(tmem + C::TM_DQ, tmem + C::TM_S + BNS * b, kv(rk), jb > 0);
          tc_commit(empty(rk));
          if (more) {
            mma_abt<D, C::IDESC_S, BNS>(tmem + C::TM_DP, dot, kv(rv1));
            tc_commit(BAR(C::B_DPFULL));
            tc_commit(empty(rv1));
            if (jb + 2 == n) tc_commit(BAR(C::B_QEMPTY));
          } else {
            tc_commit(BAR(C::B_DQFULL));
          }
          if (more2) {
            mma_abt<D, C::IDESC_S, BNS>(tmem + C::TM_S + BNS * b, qt, kv(rk2));
            tc_commit(BAR(C::B_SFULL + b));
          }
        }
        r += 2 * n;
        ++u_it;
      }
      if (!ok) {
        tc_commit(BAR(C::B_DRAIN));
        drain_wait(BAR(C::B_DRAIN), 0, 100000000ull);
      }
    }
  }
  } else {
    regs_inc<REGS_COMPUTE>();
    // ------------------------------------------------------------ P / dS
    const int wg = warp >> 2;                             // key-column half
    const int lg = warp & 3;
    const int rr = lg * 32 + lane;                        // query row within the block
    const uint32_t lane_off = (uint32_t)(lg * 32) << 16;
    const int c0 = wg * COLS;
    const uint32_t t_s = tmem + lane_off + C::TM_S + c0;
    const uint32_t t_dp = tmem + lane_off + C::TM_DP + c0;
    const float sl2 = p.scale_log2;
    Walker w;
    w.init(spec);
    uint32_t sj = 0;
    int u_it = 0;
    bool ok = true;
    for (int k = 0; ok; ++k) {
      Unit u;
      if (!w.seek(snake_index(k, G, cta), u)) break;
      const int n = u.cost;
      const int row = u.m * BM + rr;
      const bool valid = row < u.q_len;
      __nv_bfloat16* dq_row =
          p.dq + (((long long)u.q_start + row) * p.Hq + u.head) * D + wg * (D / 2);
      if (n == 0) {                                        // rows that see no key
        if (valid) zero_half<D>(dq_row);
        continue;
      }
      const long long pi = (long long)u.head * p.pad_hstride + pad_start(u.seq, u.q_start) + row;
      const float nlse = p.lse2[pi];                      // -LSE*log2(e); -inf on padding rows
      const float nd = p.delta[pi];                       // -D
      int kv_lim = u.k_len;
      if (p.causal) {
        const int lim = row + 1 + (u.k_len - u.q_len);
        kv_lim = lim < kv_lim ? lim : kv_lim;
      }
      const uint64_t sl2x2 = f2pack(sl2, sl2), nl2 = f2pack(nlse, nlse), nd2 = f2pack(nd, nd);
      for (int jb = 0; jb < n; ++jb, ++sj) {
        const uint32_t b = sj & 1;
        ok = mbar_wait(BAR(C::B_SFULL + b), (sj >> 1) & 1, wc, SITE_DQ_S_FULL);
        if (!ok) break;
        if (threadIdx.x == 0) FA_TRACE(TR_Q_S, sj);
        tc_fence_after();
        uint32_t sa[COLS];
        tmem_ld_cols<COLS>(t_s + BNS * b, sa);
        const int lim = kv_lim - (jb * BNS + c0);         // columns c >= lim are masked
        const bool mask = __any_sync(0xffffffffu, lim < COLS);
        uint64_t p2[COLS / 2];
#pragma unroll
        for (int c = 0; c < COLS; c += 2) {
          float x0, x1;
          f2unpack(ffma2(f2pack(u2f(sa[c]), u2f(sa[c + 1])), sl2x2, nl2), x0, x1);
          float e0 = (c & 7) < POLY8 ? exp2_poly(x0) : ex2_mufu(x0);
          float e1 = ((c + 1) & 7) < POLY8 ? exp2_poly(x1) : ex2_mufu(x1);
          if (mask) {
            e0 = c < lim ? e0 : 0.f;
            e1 = c + 1 < lim ? e1 : 0.f;
          }
          p2[c / 2] = f2pack(e0, e1);
        }
        if (threadIdx.x == 0) FA_TRACE(TR_Q_P, sj);
        ok = mbar_wait(BAR(C::B_DPFULL), sj & 1, wc, SITE_DQ_DP_FULL);
        if (!ok) break;
        if (threadIdx.x == 0) FA_TRACE(TR_Q_DP, sj);
        tc_fence_after();
        uint32_t dpa[COLS];
        tmem_ld_cols<COLS>(t_dp, dpa);
        uint32_t pk[COLS / 2];
#pragma unroll
        for (int c = 0; c < COLS; c += 2)
          pk[c / 2] = pack2(fmul2(p2[c / 2], fadd2(f2pack(u2f(dpa[c]), u2f(dpa[c + 1])), nd2)));
        tmem_st_half<COLS>(t_s + BNS * b, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(BAR(C::B_DSREADY));
        if (threadIdx.x == 0) FA_TRACE(TR_Q_DS, sj);
      }
      if (!ok) break;
      ok = mbar_wait(BAR(C::B_DQFULL), u_it & 1, wc, SITE_DQ_DQ_FULL);
      if (!ok) break;
      tc_fence_after();
      ++u_it;
      store_acc_half<D>(tmem + lane_off + C::TM_DQ + wg * (D / 2), dq_row, p.scale, valid);
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
  // launched as the dK/dV pass's dependent: this grid completes only after
  // that one has (no wait at all when launched the ordinary way)
  if (threadIdx.x == 0) griddep_wait();
#undef BAR
}

}  // namespace bsplit

// The dK/dV pass runs with p_kv, the dQ pass with p_q (for head dim 192 the two
// passes read Q/dO and K/V through tensor maps with different box heights).
template <int D, int POLY8>
static cudaError_t launch_split_pair(const BwdParams& p_kv, const BwdParams& p_q, int grid_kv,
                                     int grid_q, cudaStream_t stream, int pdl) {
  auto kkv = bsplit::dkdv_kernel<D, POLY8>;
  auto kq = bsplit::dq_kernel<D, POLY8>;
  const int s_kv = bsplit::CfgKV<D>::SMEM_BYTES, s_q = bsplit::CfgQ<D>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, s_kv);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, s_q)) !=
      cudaSuccess)
    return e;
  if (grid_kv > 0) {
    kkv<<<grid_kv, bsplit::NUM_THREADS, s_kv, stream>>>(p_kv);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (grid_q > 0) {
    // After a dK/dV pass, as its programmatic dependent: the dQ pass reads only
    // what the preprocess wrote (complete before the dK/dV pass began) and
    // shares nothing with the dK/dV pass, so its CTAs may start on the SMs the
    // dK/dV CTAs leave; each dQ CTA waits for the dK/dV grid before it exits,
    // so the backward completes only once both passes have.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid_q, 1, 1);
    cfg.blockDim = dim3(bsplit::NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = s_q;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl && grid_kv > 0 ? 1 : 0;
    if ((e = cudaLaunchKernelEx(&cfg, kq, p_q)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// Most CTA pairs of the dK/dV pair kernel that can be resident at once (0 on error).
int dkdv_pair_max_clusters() {
  auto kern = bsplit::dkdv_pair_kernel<0>;
  const int smem = bsplit::CfgKV<128>::SMEM_BYTES;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(bsplit::NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, (void*)kern, &cfg) != cudaSuccess) return 0;
  return n;
}

template <int POLY8>
static cudaError_t launch_pair_then_dq(const BwdParams& p, int grid_pair, int grid_q,
                                       cudaStream_t stream) {
  auto kkv = bsplit::dkdv_pair_kernel<POLY8>;
  auto kq = bsplit::dq_kernel<128, POLY8>;
  const int s_kv = bsplit::CfgKV<128>::SMEM_BYTES, s_q = bsplit::CfgQ<128>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, s_kv);
  if (e != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, s_q)) !=
      cudaSuccess)
    return e;
  if (grid_pair > 0) {
    kkv<<<grid_pair, bsplit::NUM_THREADS, s_kv, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (grid_q > 0) {
    kq<<<grid_q, bsplit::NUM_THREADS, s_q, stream>>>(p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// The two-pass backward with the dK/dV pass on CTA pairs (head dim 128);
// grid_pair is even.
cudaError_t launch_bwd_pair(const BwdParams& p, int grid_pair, int grid_q, cudaStream_t stream,
                            int poly8) {
  switch (poly8) {
    case 0: return launch_pair_then_dq<0>(p, grid_pair, grid_q, stream);
    case 2: return launch_pair_then_dq<2>(p, grid_pair, grid_q, stream);
    case 4: return launch_pair_then_dq<4>(p, grid_pair, grid_q, stream);
    default: return cudaErrorInvalidValue;
  }
}

// The two passes of the split backward (after the preprocess pass of bwd.cu).
cudaError_t launch_bwd_split(const BwdParams& p, int d, int grid_kv, int grid_q,
                             cudaStream_t stream, int poly8, int pdl) {
  if (d == 128) {
    switch (poly8) {
      case 0: return launch_split_pair<128, 0>(p, p, grid_kv, grid_q, stream, pdl);
      case 2: return launch_split_pair<128, 2>(p, p, grid_kv, grid_q, stream, pdl);
      case 4: return launch_split_pair<128, 4>(p, p, grid_kv, grid_q, stream, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  if (d == 64) {
    switch (poly8) {
      case 0: return launch_split_pair<64, 0>(p, p, grid_kv, grid_q, stream, pdl);
      case 2: return launch_split_pair<64, 2>(p, p, grid_kv, grid_q, stream, pdl);
      case 4: return launch_split_pair<64, 4>(p, p, grid_kv, grid_q, stream, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  if (d == 192 || d == 256) {
    // dK/dV pass: 64-row Q/dO steps; dQ pass: 64-key (192) or 32-key (256) K/V blocks
    BwdParams p_kv = p, p_q = p;
    p_kv.tm_q = p.tm_q2;
    p_kv.tm_do = p.tm_do2;
    p_q.tm_k = p.tm_k2;
    p_q.tm_v = p.tm_v2;
    if (d == 256) {
      switch (poly8) {
        case 0: return launch_split_pair<256, 0>(p_kv, p_q, grid_kv, grid_q, stream, pdl);
        case 2: return launch_split_pair<256, 2>(p_kv, p_q, grid_kv, grid_q, stream, pdl);
        case 4: return launch_split_pair<256, 4>(p_kv, p_q, grid_kv, grid_q, stream, pdl);
        default: return cudaErrorInvalidValue;
      }
    }
    switch (poly8) {
      case 0: return launch_split_pair<192, 0>(p_kv, p_q, grid_kv, grid_q, stream, pdl);
      case 2: return launch_split_pair<192, 2>(p_kv, p_q, grid_kv, grid_q, stream, pdl);
      case 4: return launch_split_pair<192, 4>(p_kv, p_q, grid_kv, grid_q, stream, pdl);
      default: return cudaErrorInvalidValue;
    }
  }
  return cudaErrorNotSupported;
}

}  // namespace fa
