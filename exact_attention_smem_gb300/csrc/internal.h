// Host/device structures shared by the launchers and the kernels. Not part of
// the public ABI (include/fa.h is).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

namespace fa {

// Wait sites recorded in the device error word when a bounded wait expires.
enum WaitSite : int {
  SITE_FWD_Q_EMPTY = 101, SITE_FWD_KV_EMPTY, SITE_FWD_Q_FULL, SITE_FWD_KV_FULL,
  SITE_FWD_P_FULL, SITE_FWD_S_FULL, SITE_FWD_O_FULL,
  SITE_BWD_KV_FULL = 201, SITE_BWD_QD_EMPTY, SITE_BWD_QD_FULL, SITE_BWD_S_FULL,
  SITE_BWD_DP_FULL, SITE_BWD_P_READY, SITE_BWD_DS_READY, SITE_BWD_DQ_FULL,
  SITE_BWD_DQ_EMPTY, SITE_BWD_ACC_FULL, SITE_BWD_KV_EMPTY,
  SITE_DKDV_KV_FULL = 301, SITE_DKDV_KV_EMPTY, SITE_DKDV_Q_FULL, SITE_DKDV_Q_EMPTY,
  SITE_DKDV_DO_FULL, SITE_DKDV_DO_EMPTY, SITE_DKDV_S_FULL, SITE_DKDV_DP_FULL,
  SITE_DKDV_P_READY, SITE_DKDV_DS_READY, SITE_DKDV_ACC_FULL, SITE_DKDV_LD_FULL,
  SITE_DKDV_LD_EMPTY,
  SITE_DQ_Q_FULL = 401, SITE_DQ_Q_EMPTY, SITE_DQ_KV_FULL, SITE_DQ_KV_EMPTY, SITE_DQ_S_FULL,
  SITE_DQ_DP_FULL, SITE_DQ_DS_READY, SITE_DQ_DQ_FULL,
  SITE_SMEM_ALIGN = 801,         // dynamic shared memory not on a 1024-byte boundary
  SITE_TEST = 901,
};

// Runtime knobs (settable through fa_debug_set; defaults are the tuned values).
struct Knobs {
  float tau_log2 = 0.0f;         // rescale threshold, base-2 units
  float fp8_tau = 1.5f;          // the same for the FP8 forward (at most 1.5)
  int poly8 = 0;                 // eighths of the exponentials done by the polynomial (fwd)
  int bwd_poly8 = 0;             // same for the backward
  int fp8_poly8 = 0;             // same for the FP8 forward
  int bwd_mode = 1;              // 1: two-pass backward (dK/dV pass + dQ pass); 2: the same
                                 // with the dK/dV pass on CTA pairs (d = 128; d = 64 runs
                                 // mode 1); 0: one pass with dQ by fp32 atomics + convert
  long long timeout_ns = 2000000000LL;
  int grid_override = 0;         // >0: persistent grid size (schedule permutation tests)
  int fwd_hblock = 0;            // >0: forward heads per scheduler group (0: one group)
  int fwd_split_q = -1;          // forward Q barriers per tile: 1 on, 0 off, -1 automatic
  int bwd_hblock = 0;            // >0: dK/dV-pass KV heads per scheduler group (0: automatic)
  int bwd_hblock_q = 0;          // >0: dQ-pass query heads per scheduler group (0: automatic)
  int bwd_pdl = -1;              // dQ pass as the dK/dV pass's dependent: 1 on, 0 off, -1 auto
  cudaEvent_t ev[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};  // [fwd|bwd][start|stop]
  long long* trace = nullptr;    // device buffer for the backward role timeline
};
// Backward timeline: trace[event * TRACE_STEPS + step] = clock64 of CTA 0.
constexpr int TRACE_STEPS = 512;
enum TraceEvent : int {
  TR_MMA_P = 0, TR_MMA_DS, TR_MMA_QD2, TR_MMA_DQE,     // MMA thread: after each wait
  TR_PDS_S, TR_PDS_P, TR_PDS_DP, TR_PDS_DS,            // P/dS warps (thread 0)
  TR_DRN_FULL, TR_DRN_DONE,                            // dQ drain (thread 128)
  // two-pass form, dK/dV pass
  TR_KV_A, TR_KV_B,                                    // MMA thread after sync A / B
  TR_KV_S, TR_KV_P, TR_KV_DP, TR_KV_DS,                // compute thread 0
  // two-pass form, dQ pass
  TR_Q_SYNC,                                           // MMA thread after its sync
  TR_Q_S, TR_Q_P, TR_Q_DP, TR_Q_DS,                    // compute thread 0
  TR_Q_KLOAD,                                          // producer: K_j load issued
  // dK/dV pass unit boundaries, at the index of a unit's first step (EPI: of
  // the unit just finished, i.e. its last step)
  TR_KV_KVLOAD,                                        // producer: K/V of the unit issued
  TR_KV_PRO,                                           // MMA thread: S^T(0)/dP^T(0) issued
  TR_KV_EPI, TR_KV_EPI_END,                            // compute thread 0: dK/dV write-out
  TR_NUM
};
Knobs knobs_snapshot();
void take_events(int which, cudaEvent_t* start, cudaEvent_t* stop);  // one-shot timing events

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;  // [T, H, d] views, 64-column x 128-row boxes, 128B swizzle
  CUtensorMap tm_o;              // the output O, same view (bf16 forward, head dim <= 128)
  __nv_bfloat16* o;
  float* lse;
  const int* cu;                 // packed boundaries or nullptr
  const int* cu_k;               // packed key boundaries when they differ from cu, else nullptr
  int nseq, Hq, Hkv, Sq, Sk;     // dense per-sequence lengths (ignored when packed)
  int total_q;                   // rows of the packed/flattened query tensor
  int causal;
  int lse_hstride;               // LSE stride between heads (dense Sq, packed T)
  long long lse_seqstride;       // dense: Hq*Sq per batch entry; packed: unused (0)
  float scale_log2;              // softmax scale * log2(e)
  float tau;                     // rescale threshold (base 2)
  int hblock;                    // heads per scheduler group
  int split_q;                   // bf16 forward, d <= 128: one Q full/empty pair per tile
  int* err;
  unsigned long long timeout_ns;
  // FP8 forward only (else unused): e4m3 inputs with per-block scales
  const float* q_scale;          // [B, Hq, nqb]: per 128 query rows
  const float* k_scale;          // [B, Hkv, nkb]: per 128 keys
  const float* v_scale;          // [B, Hkv]
  int nqb, nkb;
};

struct BwdParams {
  CUtensorMap tm_q, tm_do;       // [T, Hq, d] views, 64-column boxes of 64 rows (one-pass
                                 // kernel) or 128 rows (two-pass kernels), 128B swizzle
  CUtensorMap tm_k, tm_v;        // [T, Hkv, d] views, 64-column x 128-row boxes
  CUtensorMap tm_q2, tm_do2;     // 64-column x 64-row boxes (CTA-pair dK/dV pass; head dim
                                 // 192: the dK/dV pass's 64-row steps)
  CUtensorMap tm_k2, tm_v2;      // 64-column x 64-row boxes (head dim 192: the dQ pass's
                                 // 64-key blocks)
  __nv_bfloat16 *dk, *dv;
  __nv_bfloat16* dq;             // bf16 [Tq, Hq, d] (written directly by the dQ pass)
  float* dq_acc;                 // fp32 [Tq, Hq, d] (one-pass kernel only; else nullptr)
  const float* lse2;             // fp32 [Hq][pad_hstride] padded per sequence: -LSE * log2(e)
  const float* delta;            // fp32 [Hq][pad_hstride] padded: -D_i = -sum_c dO_ic O_ic
  long long pad_hstride;         // floats per head in the padded row arrays
  const int* cu;                 // packed boundaries or nullptr: the query list, then (k_off > 0)
  int k_off;                     // the key list at cu[k_off..]; 0 when keys share the query list
  int nseq, Hq, Hkv, Sq, Sk, total_q, total_k, causal;
  float scale_log2, scale;
  int hblock;                    // KV heads per scheduler group (dK/dV units)
  int hblock_q;                  // query heads per scheduler group (dQ units)
  long long* trace;              // optional role timeline of CTA 0 (nullptr = off)
  int* err;
  unsigned long long timeout_ns;
};

// Padded per-sequence row arrays used by the backward: sequence i's rows start
// at a 128-float boundary (every 64- or 128-row block is an aligned copy) and
// are followed by at least 129 padding rows, so a block that starts inside the
// sequence never reaches the next sequence's rows.
__host__ __device__ __forceinline__ long long pad_start(int seq_i, int q_start) {
  return (long long)((q_start + 127) & ~127) + 256ll * seq_i;
}
__host__ __device__ __forceinline__ long long pad_hstride(long long T, int nseq) {
  return ((T + 127) & ~127ll) + 256ll * (nseq + 1);
}

// Launchers (fwd.cu / bwd.cu). Return a cudaError_t.
cudaError_t launch_fwd(const FwdParams& p, int d, int grid, cudaStream_t stream, int poly8);
cudaError_t launch_fwd_big(const FwdParams& p, int d, int grid, cudaStream_t stream, int poly8);
cudaError_t launch_fwd_fp8(const FwdParams& p, int grid, cudaStream_t stream, int poly8);
cudaError_t launch_quantize_fp8(const __nv_bfloat16* x, int B, int S, int H, int d, int layout,
                                uint8_t* codes, float* scales, cudaStream_t st);
int fwd_units_total(const FwdParams& p);
struct BwdAux {                  // inputs of the preprocess / convert passes
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;              // caller layout (dense [B][Hq][Sq], packed [Hq][T])
  int lse_hstride;
  long long lse_seqstride;
  __nv_bfloat16* dq;
};
// mode 1: preprocess, dK/dV pass (grid), dQ pass (grid_q); mode 0: preprocess,
// one-pass kernel (grid), convert.
// pdl: the two-pass form launches its dQ pass as a programmatic dependent of
// the dK/dV pass (the passes share no data), so dQ CTAs take SMs as dK/dV
// CTAs finish.
cudaError_t launch_bwd(const BwdParams& p, const BwdAux& aux, int d, int grid, int grid_q,
                       cudaStream_t stream, int poly8, int mode, int pdl);
cudaError_t launch_bwd_split(const BwdParams& p, int d, int grid_kv, int grid_q,
                             cudaStream_t stream, int poly8, int pdl);
cudaError_t launch_bwd_pair(const BwdParams& p, int grid_pair, int grid_q, cudaStream_t stream,
                            int poly8);
int dkdv_pair_max_clusters();
cudaError_t launch_merge(const __nv_bfloat16* o_parts, const float* lse_parts, int P,
                         long long rows, int Hq, int S, int d, int packed, __nv_bfloat16* o,
                         float* lse, cudaStream_t stream);

cudaError_t launch_accumulate(float* acc, const __nv_bfloat16* x, long long n,
                              cudaStream_t stream);
cudaError_t launch_to_bf16(__nv_bfloat16* out, const float* in, long long n, cudaStream_t stream);

int num_sms();
int* device_error_word();

}  // namespace fa
