// C ABI of the test library libfa_gb300_testing.so (include/fa_testing.h):
// single-primitive probes, microbenchmarks and a host run of the work
// scheduler, for the tests. The attention library (libfa_gb300.so) does not
// contain any of this.
#include "../../../include/fa.h"
#include "../../../include/fa_testing.h"
#include "../exp2_poly.cuh"
#include "../host_common.h"
#include "../internal.h"
#include "../sched.cuh"

#include <cstdint>

namespace fa {
cudaError_t launch_exp2_probe(const float* x, float* y, int n, int mode, cudaStream_t st);
cudaError_t launch_mma_probe(const __nv_bfloat16* A, const __nv_bfloat16* B, float* C, int mode,
                             int N, cudaStream_t st);
cudaError_t launch_wait_timeout_probe(int* status, unsigned long long timeout_ns,
                                      cudaStream_t st);
cudaError_t launch_mma_pair_probe(const __nv_bfloat16* A, const __nv_bfloat16* B, float* C,
                                  int* flags, int mode, int N, cudaStream_t st);
cudaError_t launch_micro(int kind, int iters, double* out, int ctas, cudaStream_t st);
cudaError_t launch_mma_fp8_probe(const uint8_t* A, const uint8_t* B, float* C, int mode, int N,
                                 cudaStream_t st);
cudaError_t launch_roundtrip_probe(const CUtensorMap& src, const CUtensorMap& dst,
                                   uint32_t* tmem_out, cudaStream_t st);
}  // namespace fa

using namespace fa;

extern "C" const char* fa_test_last_error(void) { return last_error(); }

extern "C" int fa_test_get_device_error(int* code, int clear) {
  return read_device_error(code, clear);
}

extern "C" int fa_test_exp2(const float* x, float* y, int n, int mode, void* stream) {
  if (!x || !y || n < 0 || (mode != 0 && mode != 1))
    return fail(FA_ERR_INVALID_ARG, "fa_test_exp2 arguments");
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_exp2_probe(x, y, n, mode, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "%s", cudaGetErrorString(e));
}

extern "C" float fa_exp2_poly_host(float x) { return fa::exp2_poly(x); }

extern "C" int fa_micro(int kind, int iters, double* out_dev, int ctas, void* stream) {
  if (kind < 0 || kind > 51 || iters <= 0 || iters > (1 << 24) || !out_dev || ctas <= 0 ||
      ctas > 4096)
    return fail(FA_ERR_INVALID_ARG, "fa_micro arguments");
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_micro(kind, iters, out_dev, ctas, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "%s", cudaGetErrorString(e));
}

extern "C" int fa_test_mma(const void* A, const void* B, float* C, int mode, int N,
                           void* stream) {
  if (!A || !B || !C || mode < 0 || mode > 2 || (N != 64 && N != 128))
    return fail(FA_ERR_INVALID_ARG, "fa_test_mma arguments");
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_mma_probe(static_cast<const __nv_bfloat16*>(A),
                                   static_cast<const __nv_bfloat16*>(B), C, mode, N,
                                   static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "%s", cudaGetErrorString(e));
}

extern "C" int fa_test_mma_pair(const void* A, const void* B, float* C, int* flags, int mode,
                                int N, void* stream) {
  if (!A || !B || !C || !flags || (mode != 0 && mode != 1) || N != 128)
    return fail(FA_ERR_INVALID_ARG, "fa_test_mma_pair arguments");
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_mma_pair_probe(static_cast<const __nv_bfloat16*>(A),
                                        static_cast<const __nv_bfloat16*>(B), C, flags, mode, N,
                                        static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "%s", cudaGetErrorString(e));
}

extern "C" int fa_test_mma_fp8(const void* A, const void* B, float* C, int mode, int N,
                               void* stream) {
  if (!A || !B || !C || (mode != 0 && mode != 1) || (N != 64 && N != 128))
    return fail(FA_ERR_INVALID_ARG, "fa_test_mma_fp8 arguments");
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_mma_fp8_probe(static_cast<const uint8_t*>(A),
                                       static_cast<const uint8_t*>(B), C, mode, N,
                                       static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "%s", cudaGetErrorString(e));
}

extern "C" int fa_test_roundtrip(const void* src, void* dst, unsigned* tmem_out, void* stream) {
  if (!src || !dst || !tmem_out || !aligned16(src) || !aligned16(dst))
    return fail(FA_ERR_INVALID_ARG, "fa_test_roundtrip arguments");
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  CUtensorMap ms, md;
  if ((st = encode_rows(&ms, src, 128, 1, 64)) != FA_OK) return st;   // one 128 x 64 tile
  if ((st = encode_rows(&md, dst, 128, 1, 64)) != FA_OK) return st;
  cudaError_t e = launch_roundtrip_probe(ms, md, tmem_out, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "%s", cudaGetErrorString(e));
}

extern "C" int fa_test_wait_timeout(int* status_dev, double timeout_ms, void* stream) {
  if (!status_dev || !(timeout_ms > 0 && timeout_ms <= 10000))
    return fail(FA_ERR_INVALID_ARG, "fa_test_wait_timeout arguments");
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_wait_timeout_probe(status_dev, (unsigned long long)(timeout_ms * 1e6),
                                            static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "%s", cudaGetErrorString(e));
}

extern "C" int fa_sched_list(int kind, int B, const int* cu_seqlens_host, int Sq, int Sk,
                             int heads, int causal, int grid, int cta, int heads_per_group,
                             int* out, int max_units) {
  if (kind < 0 || kind > 5 || B < 0 || Sq < 0 || Sk < 0 || heads <= 0 || grid <= 0 ||
      cta < 0 || cta >= grid || heads_per_group < 0 || max_units < 0 || (max_units > 0 && !out))
    return -1;
  // kind: 0 forward, 1 one-pass backward, 2 dK/dV pass, 3 dQ pass, 4 dK/dV pass on CTA pairs
  static const int kUnit[6] = {256, 128, 128, 128, 256, 128},
                   kInner[6] = {128, 64, 128, 128, 128, 64}, kList[6] = {0, 1, 1, 0, 1, 0};
  SchedSpec s{cu_seqlens_host, B, Sq, Sk, heads, causal ? 1 : 0, kUnit[kind], kInner[kind],
              kList[kind], heads_per_group};
  if (heads_per_group == 0) {
    long long per_head = 0;
    for (int i = 0; i < B; ++i) {
      int qs, ql, ks, kl;
      s.seq(i, qs, ql, ks, kl);
      per_head += s.nblocks(ql, kl);
    }
    s.hblock = pick_hblock(per_head, heads, grid);
  }
  Walker w;
  w.init(s);
  int count = 0;
  for (int k = 0;; ++k) {
    Unit u;
    if (!w.seek(snake_index(k, grid, cta), u)) break;
    if (count < max_units) {
      out[4 * count + 0] = u.seq;
      out[4 * count + 1] = u.m;
      out[4 * count + 2] = u.head;
      out[4 * count + 3] = u.cost;
    }
    ++count;
  }
  return count;
}
