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
};
Knobs knobs_snapshot();

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
  int* err;
  unsigned long long timeout_ns;
};

struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  __nv_bfloat16 *dk, *dv;
  float* dq_acc;                 // fp32 [T, Hq, d]
  const float* lse_log2;         // fp32 [Hq, T] (LSE * log2 e)
  const float* delta;            // fp32 [Hq, T]
  const int* cu;
  int nseq, Hq, Hkv, Sq, Sk, total_q, total_k, causal;
  float scale_log2, scale;
  int* err;
  unsigned long long timeout_ns;
};

// Launchers (fwd.cu / bwd.cu). Return a cudaError_t.
cudaError_t launch_fwd(const FwdParams& p, int d, int grid, cudaStream_t stream, int poly8);
int fwd_units_total(const FwdParams& p);
cudaError_t launch_bwd(const BwdParams& p, int d, int grid, cudaStream_t stream, int poly8,
                       const __nv_bfloat16* o, const __nv_bfloat16* dout, const float* lse,
                       __nv_bfloat16* dq, int lse_hstride, long long lse_seqstride);

int num_sms();
int* device_error_word();

}  // namespace fa
