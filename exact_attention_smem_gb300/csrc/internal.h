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
  SITE_TEST = 901,
};

// Runtime knobs (settable through fa_debug_set; defaults are the tuned values).
struct Knobs {
  float tau_log2 = 0.0f;         // rescale threshold, base-2 units
  int poly8 = 0;                 // eighths of the exponentials done by the polynomial (fwd)
  int bwd_poly8 = 0;             // same for the backward
  long long timeout_ns = 2000000000LL;
  int grid_override = 0;         // >0: persistent grid size (schedule permutation tests)
  cudaEvent_t ev[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};  // [fwd|bwd][start|stop]
  long long* trace = nullptr;    // device buffer for the backward role timeline
};
// Backward timeline: trace[event * TRACE_STEPS + step] = clock64 of CTA 0.
constexpr int TRACE_STEPS = 512;
enum TraceEvent : int {
  TR_MMA_P = 0, TR_MMA_DS, TR_MMA_QD2, TR_MMA_DQE,     // MMA thread: after each wait
  TR_PDS_S, TR_PDS_P, TR_PDS_DP, TR_PDS_DS,            // P/dS warps (thread 0)
  TR_DRN_FULL, TR_DRN_DONE,                            // dQ drain (thread 128)
  TR_NUM
};
Knobs knobs_snapshot();
void take_events(int which, cudaEvent_t* start, cudaEvent_t* stop);  // one-shot timing events

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;  // [T, H, d] views, 64-column x 128-row boxes, 128B swizzle
  __nv_bfloat16* o;
  float* lse;
  const int* cu;                 // packed boundaries or nullptr
  int nseq, Hq, Hkv, Sq, Sk;     // dense per-sequence lengths (ignored when packed)
  int total_q;                   // rows of the packed/flattened query tensor
  int causal;
  int lse_hstride;               // LSE stride between heads (dense Sq, packed T)
  long long lse_seqstride;       // dense: Hq*Sq per batch entry; packed: unused (0)
  float scale_log2;              // softmax scale * log2(e)
  float tau;                     // rescale threshold (base 2)
  int hblock;                    // heads per scheduler group
  int* err;
  unsigned long long timeout_ns;
};

struct BwdParams {
  CUtensorMap tm_q, tm_do;       // [T, Hq, d] views, 64-column x 64-row boxes, 128B swizzle
  CUtensorMap tm_k, tm_v;        // [T, Hkv, d] views, 64-column x 128-row boxes
  __nv_bfloat16 *dk, *dv;
  float* dq_acc;                 // fp32 [Tq, Hq, d]
  const float* lse2;             // fp32 [Hq][pad_hstride] padded per sequence: -LSE * log2(e)
  const float* delta;            // fp32 [Hq][pad_hstride] padded: -D_i = -sum_c dO_ic O_ic
  long long pad_hstride;         // floats per head in the padded row arrays
  const int* cu;
  int nseq, Hq, Hkv, Sq, Sk, total_q, total_k, causal;
  float scale_log2, scale;
  int hblock;                    // KV heads per scheduler group
  long long* trace;              // optional role timeline of CTA 0 (nullptr = off)
  int* err;
  unsigned long long timeout_ns;
};

// Padded per-sequence row arrays used by the backward: sequence i's rows start
// at a 64-float boundary, so every 64-row block is one aligned 256-byte copy.
__host__ __device__ __forceinline__ long long pad_start(int seq_i, int q_start) {
  return (long long)((q_start + 63) & ~63) + 128ll * seq_i;
}
__host__ __device__ __forceinline__ long long pad_hstride(long long T, int nseq) {
  return ((T + 63) & ~63ll) + 128ll * (nseq + 1);
}

// Launchers (fwd.cu / bwd.cu). Return a cudaError_t.
cudaError_t launch_fwd(const FwdParams& p, int d, int grid, cudaStream_t stream, int poly8);
int fwd_units_total(const FwdParams& p);
struct BwdAux {                  // inputs of the preprocess / convert passes
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;              // caller layout (dense [B][Hq][Sq], packed [Hq][T])
  int lse_hstride;
  long long lse_seqstride;
  __nv_bfloat16* dq;
};
cudaError_t launch_bwd(const BwdParams& p, const BwdAux& aux, int d, int grid,
                       cudaStream_t stream, int poly8);

int num_sms();
int* device_error_word();

}  // namespace fa
