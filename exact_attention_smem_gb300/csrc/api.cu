// C ABI (include/fa.h): argument validation, launch configuration and kernel
// launches (device properties and TMA encoding: host_common.cu). Nothing here allocates device memory.
#include "../../include/fa.h"
#include "host_common.h"
#include "internal.h"
#include "sched.cuh"

#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

namespace fa {
namespace {

std::mutex g_mu;
Knobs g_knobs;

struct Shape {
  long long Tq, Tk;  // rows of the flattened q / k tensors
  bool packed;
};

// Packed layouts: cu alone gives the boundaries of queries and keys (then
// Sq == Sk == T); with cu_k the keys have their own boundaries and Sq / Sk are
// the query / key row counts.
int validate_common(const void* const* ptrs, int nptrs, int B, int Hq, int Hkv, int Sq, int Sk,
                    int d, float scale, const int* cu, Shape* sh, const int* cu_k = nullptr) {
  for (int i = 0; i < nptrs; ++i) {
    if (!ptrs[i]) return fail(FA_ERR_INVALID_ARG, "tensor pointer %d is NULL", i);
    if (!aligned16(ptrs[i]))
      return fail(FA_ERR_INVALID_ARG, "tensor pointer %d is not 16-byte aligned", i);
  }
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0)
    return fail(FA_ERR_INVALID_ARG, "bad sizes B=%d Hq=%d Hkv=%d Sq=%d Sk=%d", B, Hq, Hkv, Sq, Sk);
  if (Hq % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "Hq (%d) %% Hkv (%d) != 0", Hq, Hkv);
  if (d != 64 && d != 128 && d != 192 && d != 256)
    return fail(FA_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128; forward also 192, 256)", d);
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (cu_k && !cu) return fail(FA_ERR_INVALID_ARG, "key boundaries without query boundaries");
  if (cu) {
    if (!cu_k && Sq != Sk)
      return fail(FA_ERR_INVALID_ARG, "packed layout: Sq and Sk must both equal the packed "
                  "row count T (got %d, %d)", Sq, Sk);
    sh->Tq = Sq;
    sh->Tk = Sk;
    sh->packed = true;
  } else {
    sh->Tq = (long long)B * Sq;
    sh->Tk = (long long)B * Sk;
    sh->packed = false;
  }
  if (sh->Tq > (1ll << 31) - 512 || sh->Tk > (1ll << 31) - 512)
    return fail(FA_ERR_INVALID_ARG, "too many rows");
  return FA_OK;
}

}  // namespace

Knobs knobs_snapshot() {
  std::lock_guard<std::mutex> lk(g_mu);
  return g_knobs;
}

void take_events(int which, cudaEvent_t* start, cudaEvent_t* stop) {
  std::lock_guard<std::mutex> lk(g_mu);
  *start = g_knobs.ev[which][0];
  *stop = g_knobs.ev[which][1];
  g_knobs.ev[which][0] = g_knobs.ev[which][1] = nullptr;
}

}  // namespace fa

using namespace fa;

namespace {
int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int Sq, int Sk, int d, int causal, float scale, const int* cu_seqlens,
             const int* cu_seqlens_k, void* stream) {
  clear_last_error();
  const void* ptrs[5] = {q, k, v, o, lse};
  Shape sh;
  int st = validate_common(ptrs, 5, B, Hq, Hkv, Sq, Sk, d, scale, cu_seqlens, &sh, cu_seqlens_k);
  if (st != FA_OK) return st;
  if (B == 0 || sh.Tq == 0) return FA_OK;
  DevInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  const Knobs kn = knobs_snapshot();

  FwdParams p;
  memset(&p, 0, sizeof(p));
  if ((st = encode_rows(&p.tm_q, q, sh.Tq, Hq, d)) != FA_OK) return st;
  const int kv_box = d > 128 ? 64 : 128;             // keys per K/V block of the kernel
  if (sh.Tk > 0) {
    if ((st = encode_rows(&p.tm_k, k, sh.Tk, Hkv, d, kv_box)) != FA_OK) return st;
    if ((st = encode_rows(&p.tm_v, v, sh.Tk, Hkv, d, kv_box)) != FA_OK) return st;
  } else {
    // no keys at all: every row is fully masked; maps are never used by the TMA
    if ((st = encode_rows(&p.tm_k, q, sh.Tq, Hq, d)) != FA_OK) return st;
    if ((st = encode_rows(&p.tm_v, q, sh.Tq, Hq, d)) != FA_OK) return st;
  }
  if (d <= 128 && (st = encode_rows(&p.tm_o, o, sh.Tq, Hq, d)) != FA_OK) return st;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.cu = cu_seqlens;
  p.cu_k = cu_seqlens_k;
  p.nseq = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.total_q = (int)sh.Tq;
  p.causal = causal ? 1 : 0;
  p.lse_hstride = sh.packed ? (int)sh.Tq : Sq;
  p.lse_seqstride = sh.packed ? 0 : (long long)Hq * Sq;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.tau = kn.tau_log2;
  p.err = di->err_word;
  p.timeout_ns = (unsigned long long)kn.timeout_ns;

  // persistent grid: one CTA per SM, capped by an upper bound on the unit count
  const int unit_rows = d > 128 ? 128 : 256;         // query rows per unit of the kernel
  const long long units_per_head =
      sh.packed ? (sh.Tq + unit_rows - 1) / unit_rows + B
                : (long long)B * ((Sq + unit_rows - 1) / unit_rows);
  const long long units = units_per_head * Hq;
  int grid = kn.grid_override > 0 ? kn.grid_override : di->sms;
  if (units < grid) grid = (int)units;
  if (grid < 1) grid = 1;
  // The forward keeps one group (pure LPT): its K/V traffic is far from the
  // DRAM roof, and static snake rounds balance best over a single LPT list.
  p.hblock = kn.fwd_hblock > 0 && kn.fwd_hblock < Hq ? kn.fwd_hblock : Hq;
  // Short key ranges (few blocks per unit, so unit changes weigh): tile 0's
  // next Q loads once tile 0's last S is done, not tile 1's. Measured on the
  // dense workloads: +3% at S = 2048 causal, -1% at S = 32768, so dense
  // layouts with at most 4096 keys only.
  p.split_q = kn.fwd_split_q >= 0 ? kn.fwd_split_q : (!sh.packed && Sk <= 4096 ? 1 : 0);
  cudaEvent_t ev0, ev1;
  take_events(0, &ev0, &ev1);
  if (ev0) cudaEventRecord(ev0, static_cast<cudaStream_t>(stream));
  cudaError_t e = d > 128 ? launch_fwd_big(p, d, grid, static_cast<cudaStream_t>(stream), kn.poly8)
                          : launch_fwd(p, d, grid, static_cast<cudaStream_t>(stream), kn.poly8);
  if (ev1) cudaEventRecord(ev1, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

}  // namespace

extern "C" int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                      const int* cu_seqlens, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, Hq, Hkv, Sq, Sk, d, causal, scale, cu_seqlens, nullptr,
                  stream);
}

extern "C" int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                             int nseq, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
                             float scale, const int* cu_seqlens_q, const int* cu_seqlens_k,
                             void* stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) {
    return fail(FA_ERR_INVALID_ARG, "fa_fwd_varlen needs both boundary lists");
  }
  return fwd_impl(q, k, v, o, lse, nseq, Hq, Hkv, Tq, Tk, d, causal, scale, cu_seqlens_q,
                  cu_seqlens_k, stream);
}

extern "C" int fa_quantize_fp8(const void* x, int B, int S, int H, int d, int layout, void* codes,
                               float* scales, void* stream) {
  clear_last_error();
  if (!x || !codes || !scales) return fail(FA_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(x) || !aligned16(codes))
    return fail(FA_ERR_INVALID_ARG, "x and codes must be 16-byte aligned");
  if (B < 0 || S < 0 || H <= 0) return fail(FA_ERR_INVALID_ARG, "bad sizes B=%d S=%d H=%d", B, S, H);
  if (layout != 0 && layout != 1) return fail(FA_ERR_INVALID_ARG, "layout must be 0 or 1");
  if (d != 64 && d != 128) return fail(FA_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128)", d);
  if ((long long)B * H > (1LL << 30) || (long long)S * H * d > (1LL << 40))
    return fail(FA_ERR_INVALID_ARG, "sizes too large");
  if (B == 0 || S == 0) return FA_OK;
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_quantize_fp8(static_cast<const __nv_bfloat16*>(x), B, S, H, d, layout,
                                      static_cast<uint8_t*>(codes), scales,
                                      static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "quantize launch: %s", cudaGetErrorString(e));
}

extern "C" int fa_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* q_scale,
                          const float* k_scale, const float* v_scale, void* o, float* lse, int B,
                          int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                          void* stream) {
  clear_last_error();
  const void* ptrs[8] = {q8, k8, vt8, q_scale, k_scale, v_scale, o, lse};
  for (int i = 0; i < 8; ++i)
    if (!ptrs[i]) return fail(FA_ERR_INVALID_ARG, "tensor pointer %d is NULL", i);
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o))
    return fail(FA_ERR_INVALID_ARG, "q8, k8, vt8 and o must be 16-byte aligned");
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Sq < 0 || Sk < 0)
    return fail(FA_ERR_INVALID_ARG, "bad sizes B=%d Hq=%d Hkv=%d Sq=%d Sk=%d", B, Hq, Hkv, Sq, Sk);
  if (Hq % Hkv != 0) return fail(FA_ERR_INVALID_ARG, "Hq (%d) %% Hkv (%d) != 0", Hq, Hkv);
  if (d != 128) return fail(FA_ERR_UNSUPPORTED, "FP8 forward head dim %d (supported: 128)", d);
  if (!std::isfinite(scale) || !(scale > 0.f))
    return fail(FA_ERR_INVALID_ARG, "scale must be finite and > 0");
  if ((long long)B * Sq > INT32_MAX / 2 || (long long)B * Sk > INT32_MAX / 2)
    return fail(FA_ERR_INVALID_ARG, "sizes too large");
  if (B == 0 || Sq == 0) return FA_OK;
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  const Knobs kn = knobs_snapshot();

  FwdParams p;
  memset(&p, 0, sizeof(p));
  const long long Tq = (long long)B * Sq;
  const long long S_pad = ((long long)Sk + 15) / 16 * 16;
  {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)Tq};
    const cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)Hq * d};
    const cuuint32_t box[3] = {128, 1, 128};
    if ((st = encode_u8(&p.tm_q, q8, dims, strides, box)) != FA_OK) return st;
  }
  if (Sk > 0) {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)Hkv, (cuuint64_t)B * Sk};
    const cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)Hkv * d};
    const cuuint32_t box[3] = {128, 1, 128};
    if ((st = encode_u8(&p.tm_k, k8, dims, strides, box)) != FA_OK) return st;
    const cuuint64_t vdims[3] = {(cuuint64_t)S_pad, (cuuint64_t)d, (cuuint64_t)B * Hkv};
    const cuuint64_t vstrides[2] = {(cuuint64_t)S_pad, (cuuint64_t)S_pad * d};
    const cuuint32_t vbox[3] = {128, 128, 1};
    if ((st = encode_u8(&p.tm_v, vt8, vdims, vstrides, vbox)) != FA_OK) return st;
  } else {
    // no keys: every row is fully masked and the maps are never used
    p.tm_k = p.tm_q;
    p.tm_v = p.tm_q;
  }
  if ((st = encode_rows(&p.tm_o, o, Tq, Hq, d)) != FA_OK) return st;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.nseq = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.total_q = (int)Tq;
  p.causal = causal ? 1 : 0;
  p.lse_hstride = Sq;
  p.lse_seqstride = (long long)Hq * Sq;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.err = di->err_word;
  p.timeout_ns = (unsigned long long)kn.timeout_ns;
  p.tau = kn.fp8_tau;
  p.q_scale = q_scale;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.nqb = (Sq + 127) / 128;
  p.nkb = (Sk + 127) / 128;
  const long long units = (long long)B * ((Sq + 255) / 256) * Hq;
  int grid = kn.grid_override > 0 ? kn.grid_override : di->sms;
  if (units < grid) grid = (int)units;
  if (grid < 1) grid = 1;
  p.hblock = Hq;
  cudaEvent_t ev0, ev1;
  take_events(0, &ev0, &ev1);
  if (ev0) cudaEventRecord(ev0, static_cast<cudaStream_t>(stream));
  cudaError_t e = launch_fwd_fp8(p, grid, static_cast<cudaStream_t>(stream), kn.fp8_poly8);
  if (ev1) cudaEventRecord(ev1, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "FP8 forward launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

extern "C" size_t fa_bwd_workspace_bytes(int B, int Hq, int Sq, int d, int total_q) {
  if (B < 0 || Hq <= 0 || Sq < 0 || d <= 0 || total_q < 0) return 0;
  const size_t T = total_q > 0 ? (size_t)total_q : (size_t)B * (size_t)Sq;
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  const size_t P = (size_t)pad_hstride((long long)T, B);
  // + the query and key boundary lists back to back (separate key boundaries)
  return up(T * Hq * d * sizeof(float)) + 2 * up(P * Hq * sizeof(float)) +
         up(2 * ((size_t)B + 1) * sizeof(int));
}

namespace {
int bwd_impl(const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Sq,
             int Sk, int d, int causal, float scale, const int* cu_seqlens,
             const int* cu_seqlens_k, void* workspace, size_t workspace_bytes, void* stream) {
  clear_last_error();
  const void* ptrs[9] = {q, k, v, o, lse, dout, dq, dk, dv};
  Shape sh;
  int st = validate_common(ptrs, 9, B, Hq, Hkv, Sq, Sk, d, scale, cu_seqlens, &sh, cu_seqlens_k);
  if (st != FA_OK) return st;
  if (B == 0 || (sh.Tq == 0 && sh.Tk == 0)) return FA_OK;
  const size_t need = fa_bwd_workspace_bytes(B, Hq, Sq, d, sh.packed ? (int)sh.Tq : 0);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return fail(FA_ERR_WORKSPACE, "workspace must be >= %zu bytes and 256-byte aligned", need);
  DevInfo* di = nullptr;
  if ((st = device_info(&di)) != FA_OK) return st;
  const Knobs kn = knobs_snapshot();

  const int mode = (kn.bwd_mode == 2 && d != 128) ? 1 : kn.bwd_mode;
  if (mode == 0 && d != 128)
    return fail(FA_ERR_UNSUPPORTED, "the one-pass backward supports head dim 128 only");
  BwdParams p;
  memset(&p, 0, sizeof(p));
  const long long Tq = sh.Tq > 0 ? sh.Tq : 1, Tk = sh.Tk > 0 ? sh.Tk : 1;
  const int qbox = mode == 0 ? 64 : 128;
  if ((st = encode_rows(&p.tm_q, sh.Tq > 0 ? q : k, sh.Tq > 0 ? Tq : Tk, sh.Tq > 0 ? Hq : Hkv,
                        d, qbox)) != FA_OK)
    return st;
  if ((st = encode_rows(&p.tm_do, sh.Tq > 0 ? dout : k, sh.Tq > 0 ? Tq : Tk,
                        sh.Tq > 0 ? Hq : Hkv, d, qbox)) != FA_OK)
    return st;
  if ((st = encode_rows(&p.tm_k, sh.Tk > 0 ? k : q, sh.Tk > 0 ? Tk : Tq, sh.Tk > 0 ? Hkv : Hq,
                        d)) != FA_OK)
    return st;
  if ((st = encode_rows(&p.tm_v, sh.Tk > 0 ? v : q, sh.Tk > 0 ? Tk : Tq, sh.Tk > 0 ? Hkv : Hq,
                        d)) != FA_OK)
    return st;
  if (mode == 2 || d > 128) {
    if ((st = encode_rows(&p.tm_q2, sh.Tq > 0 ? q : k, sh.Tq > 0 ? Tq : Tk, sh.Tq > 0 ? Hq : Hkv,
                          d, 64)) != FA_OK)
      return st;
    if ((st = encode_rows(&p.tm_do2, sh.Tq > 0 ? dout : k, sh.Tq > 0 ? Tq : Tk,
                          sh.Tq > 0 ? Hq : Hkv, d, 64)) != FA_OK)
      return st;
  }
  if (d > 128) {
    // the dQ pass's K/V blocks: 64 keys at head dim 192, 32 at 256
    const int kbox = d > 192 ? 32 : 64;
    if ((st = encode_rows(&p.tm_k2, sh.Tk > 0 ? k : q, sh.Tk > 0 ? Tk : Tq, sh.Tk > 0 ? Hkv : Hq,
                          d, kbox)) != FA_OK)
      return st;
    if ((st = encode_rows(&p.tm_v2, sh.Tk > 0 ? v : q, sh.Tk > 0 ? Tk : Tq, sh.Tk > 0 ? Hkv : Hq,
                          d, kbox)) != FA_OK)
      return st;
  }
  auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
  char* ws = static_cast<char*>(workspace);
  const size_t T = (size_t)sh.Tq;
  const size_t P = (size_t)pad_hstride((long long)T, B);
  p.dq_acc = mode == 0 ? reinterpret_cast<float*>(ws) : nullptr;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.lse2 = reinterpret_cast<float*>(ws + up(T * Hq * d * sizeof(float)));
  p.delta = reinterpret_cast<float*>(ws + up(T * Hq * d * sizeof(float)) + up(P * Hq * sizeof(float)));
  p.pad_hstride = (long long)P;
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.cu = cu_seqlens;
  p.k_off = 0;
  if (cu_seqlens_k) {
    // The kernels take one list: the query boundaries, then the key boundaries
    // (a single pointer keeps the scheduler's registers as in the one-list case).
    int* both = reinterpret_cast<int*>(ws + up(T * Hq * d * sizeof(float)) +
                                       2 * up(P * Hq * sizeof(float)));
    const size_t nb = ((size_t)B + 1) * sizeof(int);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t ce = cudaMemcpyAsync(both, cu_seqlens, nb, cudaMemcpyDeviceToDevice, s);
    if (ce == cudaSuccess)
      ce = cudaMemcpyAsync(both + B + 1, cu_seqlens_k, nb, cudaMemcpyDeviceToDevice, s);
    if (ce != cudaSuccess) return fail(FA_ERR_CUDA, "boundary copy: %s", cudaGetErrorString(ce));
    p.cu = both;
    p.k_off = B + 1;
  }
  p.nseq = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.Sq = Sq;
  p.Sk = Sk;
  p.total_q = (int)sh.Tq;
  p.total_k = (int)sh.Tk;
  p.causal = causal ? 1 : 0;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.scale = scale;
  p.err = di->err_word;
  p.timeout_ns = (unsigned long long)kn.timeout_ns;
  p.trace = kn.trace;
  BwdAux aux;
  aux.o = static_cast<const __nv_bfloat16*>(o);
  aux.dout = static_cast<const __nv_bfloat16*>(dout);
  aux.lse = lse;
  aux.lse_hstride = sh.packed ? (int)sh.Tq : Sq;
  aux.lse_seqstride = sh.packed ? 0 : (long long)Hq * Sq;
  aux.dq = static_cast<__nv_bfloat16*>(dq);
  int grid = kn.grid_override > 0 ? kn.grid_override : di->sms;
  // dK/dV units per KV head: one per 128-key block (two at head dim 256, one
  // per 128-column half of dV and dK)
  const long long kv_units_per_head =
      (sh.packed ? (sh.Tk + 127) / 128 + B : (long long)B * ((Sk + 127) / 128)) * (d > 192 ? 2 : 1);
  // Head groups keep the data concurrently running units share in L2. Packed
  // layouts use one group in the two-pass form: their scheduler walks the
  // list one (cost level, sequence) group at a time, so head groups of one
  // head would multiply that walk by the head count (dense layouts seek
  // directly and keep the L2-sized groups).
  // When Q and dO of all heads fit in L2 a dense layout also takes one group:
  // the L2-sized groups buy nothing there and deal the LPT list in lumps (mha
  // S=2048: per-CTA cost max/mean 1.24 against 1.01 with one group).
  // Otherwise at least two KV heads per group: one-head groups deal the GQA
  // workload (B=8, Hkv=8, S=8192) 1.10 max/mean and run its backward in 25.9
  // ms, two-head groups 25.3 ms (long causal S=32768: 23.7 ms either way).
  const double qdo_bytes = (double)sh.Tq * Hq * d * 4.0;
  int hb_auto = pick_hblock(kv_units_per_head, Hkv, grid);
  if (mode != 0 && hb_auto < 2) hb_auto = Hkv < 2 ? Hkv : 2;
  p.hblock = (mode != 0 && (sh.packed || qdo_bytes <= 96e6)) ? Hkv : hb_auto;
  if (kn.bwd_hblock > 0) p.hblock = kn.bwd_hblock < Hkv ? kn.bwd_hblock : Hkv;
  // dQ units (128 query rows of one head) stream the K/V of their head. When
  // the K/V of all heads would not stay in L2 (GB300: 129 MB) a dense layout
  // takes the fewest heads whose units cover the grid twice (one group over
  // 32 heads of S=32768 re-read K/V from DRAM about 14 times); otherwise, and
  // for packed layouts (see above), one group balances best.
  const long long q_units_per_head =
      sh.packed ? (sh.Tq + 127) / 128 + B : (long long)B * ((Sq + 127) / 128);
  const double kv_bytes = (double)sh.Tk * Hkv * d * 4.0;
  p.hblock_q = (sh.packed || kv_bytes <= 96e6) ? Hq : pick_hblock(q_units_per_head, Hq, 2 * grid);
  if (kn.bwd_hblock_q > 0) p.hblock_q = kn.bwd_hblock_q < Hq ? kn.bwd_hblock_q : Hq;
  int grid_q = kn.grid_override > 0 ? kn.grid_override : di->sms;
  if (mode != 0) {
    const long long kv_units = kv_units_per_head * Hkv, q_units = q_units_per_head * Hq;
    if (kv_units < grid) grid = (int)(kv_units > 0 ? kv_units : 1);
    if (q_units < grid_q) grid_q = (int)(q_units > 0 ? q_units : 1);
  }
  if (mode == 2) {
    // dK/dV units of 256 keys on CTA pairs: a grid of pairs that can all be
    // resident at once (a persistent grid must never wait for a pair slot)
    const long long pair_units_per_head =
        sh.packed ? (sh.Tk + 255) / 256 + B : (long long)B * ((Sk + 255) / 256);
    int pairs = (kn.grid_override > 0 ? kn.grid_override : di->sms) / 2;
    const int maxc = dkdv_pair_max_clusters();
    if (maxc <= 0) return fail(FA_ERR_CUDA, "no CTA pair of the dK/dV kernel fits on this GPU");
    if (pairs > maxc) pairs = maxc;
    const long long pair_units = pair_units_per_head * Hkv;
    if (pair_units < pairs) pairs = (int)(pair_units > 0 ? pair_units : 1);
    if (pairs < 1) pairs = 1;
    grid = 2 * pairs;
    p.hblock = sh.packed ? Hkv : pick_hblock(pair_units_per_head, Hkv, pairs);
  }
  // Short dense problems: the dQ pass may start on the SMs the dK/dV pass
  // leaves (+1.5-1.8% at S = 2048). Where units are long or L2-sized head
  // groups matter (GQA, packed) the staggered start measured 1.2-1.4% slower,
  // so dense layouts with at most 4096 keys only.
  const int pdl = kn.bwd_pdl >= 0 ? kn.bwd_pdl : (!sh.packed && Sk <= 4096 ? 1 : 0);
  cudaError_t e = launch_bwd(p, aux, d, grid, grid_q, static_cast<cudaStream_t>(stream),
                             kn.bwd_poly8, mode, pdl);
  if (e == cudaErrorNotSupported)
    return fail(FA_ERR_UNSUPPORTED, "backward head dim %d unsupported", d);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "backward launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

}  // namespace

extern "C" int fa_bwd(const void* q, const void* k, const void* v, const void* o,
                      const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                      int Hq, int Hkv, int Sq, int Sk, int d, int causal, float scale,
                      const int* cu_seqlens, void* workspace, size_t workspace_bytes,
                      void* stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale,
                  cu_seqlens, nullptr, workspace, workspace_bytes, stream);
}

extern "C" int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o,
                             const float* lse, const void* dout, void* dq, void* dk, void* dv,
                             int nseq, int Hq, int Hkv, int Tq, int Tk, int d, int causal,
                             float scale, const int* cu_seqlens_q, const int* cu_seqlens_k,
                             void* workspace, size_t workspace_bytes, void* stream) {
  if (!cu_seqlens_q || !cu_seqlens_k) {
    return fail(FA_ERR_INVALID_ARG, "fa_bwd_varlen needs both boundary lists");
  }
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, nseq, Hq, Hkv, Tq, Tk, d, causal, scale,
                  cu_seqlens_q, cu_seqlens_k, workspace, workspace_bytes, stream);
}

extern "C" int fa_merge(const void* o_parts, const float* lse_parts, int P, int B, int Hq, int S,
                        int d, int packed, void* o, float* lse, void* stream) {
  clear_last_error();
  const void* ptrs[4] = {o_parts, lse_parts, o, lse};
  for (int i = 0; i < 4; ++i)
    if (!ptrs[i]) return fail(FA_ERR_INVALID_ARG, "pointer %d is NULL", i);
  if (!aligned16(o_parts) || !aligned16(o))   // the kernel moves 16-byte vectors
    return fail(FA_ERR_INVALID_ARG, "o_parts and o must be 16-byte aligned");
  if (P < 1 || P > 64) return fail(FA_ERR_INVALID_ARG, "parts P=%d (1..64)", P);
  if (B < 0 || Hq <= 0 || S < 0) return fail(FA_ERR_INVALID_ARG, "bad sizes B=%d Hq=%d S=%d", B, Hq, S);
  if (d != 64 && d != 128 && d != 192 && d != 256)
    return fail(FA_ERR_UNSUPPORTED, "head dim %d (supported: 64, 128, 192, 256)", d);
  const long long rows = packed ? (long long)S : (long long)B * S;
  if (rows == 0) return FA_OK;
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_merge(static_cast<const __nv_bfloat16*>(o_parts), lse_parts, P, rows, Hq,
                               packed ? (int)rows : S, d, packed ? 1 : 0,
                               static_cast<__nv_bfloat16*>(o), lse,
                               static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "merge launch: %s", cudaGetErrorString(e));
  return FA_OK;
}

extern "C" int fa_accumulate(float* acc, const void* x, long long n, void* stream) {
  clear_last_error();
  if (!acc || !x) return fail(FA_ERR_INVALID_ARG, "acc and x must not be NULL");
  if (!aligned16(acc) || !aligned16(x))
    return fail(FA_ERR_INVALID_ARG, "acc and x must be 16-byte aligned");
  if (n < 0 || n % 8) return fail(FA_ERR_INVALID_ARG, "n=%lld must be >= 0 and a multiple of 8", n);
  if (n == 0) return FA_OK;
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_accumulate(acc, static_cast<const __nv_bfloat16*>(x), n,
                                    static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "accumulate launch: %s", cudaGetErrorString(e));
}

extern "C" int fa_to_bf16(void* out, const float* in, long long n, void* stream) {
  clear_last_error();
  if (!out || !in) return fail(FA_ERR_INVALID_ARG, "out and in must not be NULL");
  if (!aligned16(out) || !aligned16(in))
    return fail(FA_ERR_INVALID_ARG, "out and in must be 16-byte aligned");
  if (n < 0 || n % 8) return fail(FA_ERR_INVALID_ARG, "n=%lld must be >= 0 and a multiple of 8", n);
  if (n == 0) return FA_OK;
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = launch_to_bf16(static_cast<__nv_bfloat16*>(out), in, n,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : fail(FA_ERR_CUDA, "conversion launch: %s", cudaGetErrorString(e));
}

extern "C" const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported";
    case FA_ERR_ARCH: return "wrong GPU architecture (need sm_103a)";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_WORKSPACE: return "workspace missing or too small";
    case FA_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

extern "C" const char* fa_last_error(void) { return last_error(); }

extern "C" int fa_get_device_error(int* code, int clear) {
  return read_device_error(code, clear);
}

extern "C" int fa_debug_set(const char* key, double value) {
  if (!key) return fail(FA_ERR_INVALID_ARG, "key is NULL");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!strcmp(key, "tau")) {
    if (!(value >= 0.0 && value <= 16.0)) return fail(FA_ERR_INVALID_ARG, "tau in [0, 16]");
    g_knobs.tau_log2 = (float)value;
  } else if (!strcmp(key, "fp8_tau")) {
    if (!(value >= 0.0 && value <= 1.5)) return fail(FA_ERR_INVALID_ARG, "fp8_tau in [0, 1.5]");
    g_knobs.fp8_tau = (float)value;
  } else if (!strcmp(key, "poly8") || !strcmp(key, "bwd_poly8") || !strcmp(key, "fp8_poly8")) {
    const int v = (int)value;
    if (v != 0 && v != 2 && v != 4) return fail(FA_ERR_INVALID_ARG, "poly8 in {0, 2, 4}");
    (key[0] == 'p' ? g_knobs.poly8 : key[0] == 'b' ? g_knobs.bwd_poly8 : g_knobs.fp8_poly8) = v;
  } else if (!strcmp(key, "bwd_mode")) {
    if (value != 0.0 && value != 1.0 && value != 2.0)
      return fail(FA_ERR_INVALID_ARG, "bwd_mode in {0, 1, 2}");
    g_knobs.bwd_mode = (int)value;
  } else if (!strcmp(key, "bwd_pdl")) {
    if (value != -1.0 && value != 0.0 && value != 1.0)
      return fail(FA_ERR_INVALID_ARG, "bwd_pdl in {-1, 0, 1}");
    g_knobs.bwd_pdl = (int)value;
  } else if (!strcmp(key, "fwd_split_q")) {
    if (value != -1.0 && value != 0.0 && value != 1.0)
      return fail(FA_ERR_INVALID_ARG, "fwd_split_q in {-1, 0, 1}");
    g_knobs.fwd_split_q = (int)value;
  } else if (!strcmp(key, "fwd_hblock")) {
    if (!(value >= 0.0 && value <= 65536.0)) return fail(FA_ERR_INVALID_ARG, "fwd_hblock");
    g_knobs.fwd_hblock = (int)value;
  } else if (!strcmp(key, "bwd_hblock")) {
    if (!(value >= 0.0 && value <= 65536.0)) return fail(FA_ERR_INVALID_ARG, "bwd_hblock");
    g_knobs.bwd_hblock = (int)value;
  } else if (!strcmp(key, "bwd_hblock_q")) {
    if (!(value >= 0.0 && value <= 65536.0)) return fail(FA_ERR_INVALID_ARG, "bwd_hblock_q");
    g_knobs.bwd_hblock_q = (int)value;
  } else if (!strcmp(key, "timeout_ms")) {
    if (!(value >= 1.0 && value <= 60000.0)) return fail(FA_ERR_INVALID_ARG, "timeout_ms");
    g_knobs.timeout_ns = (long long)(value * 1e6);
  } else if (!strcmp(key, "grid")) {
    if (!(value >= 0.0 && value <= 100000.0)) return fail(FA_ERR_INVALID_ARG, "grid");
    g_knobs.grid_override = (int)value;
  } else {
    return fail(FA_ERR_INVALID_ARG, "unknown key '%s'", key);
  }
  return FA_OK;
}

extern "C" int fa_debug_set_events(int which, void* start, void* stop) {
  if (which != 0 && which != 1) return fail(FA_ERR_INVALID_ARG, "which must be 0 or 1");
  std::lock_guard<std::mutex> lk(g_mu);
  g_knobs.ev[which][0] = static_cast<cudaEvent_t>(start);
  g_knobs.ev[which][1] = static_cast<cudaEvent_t>(stop);
  return FA_OK;
}

extern "C" int fa_debug_set_trace(void* trace_dev, size_t bytes) {
  if (trace_dev && bytes < sizeof(long long) * TRACE_STEPS * TR_NUM)
    return fail(FA_ERR_INVALID_ARG, "trace buffer needs %zu bytes",
                sizeof(long long) * TRACE_STEPS * TR_NUM);
  std::lock_guard<std::mutex> lk(g_mu);
  g_knobs.trace = static_cast<long long*>(trace_dev);
  return FA_OK;
}
