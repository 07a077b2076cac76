// Host-side helpers shared by the C-ABI translation units (host_common.h).
#include "../../include/fa.h"
#include "host_common.h"
#include "internal.h"

#include <cudaTypedefs.h>

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

namespace fa {

__device__ int g_error_word;  // first expired bounded wait (site code), per device

namespace {
thread_local std::string t_last_error;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::mutex g_dev_mu;
DevInfo g_dev[64];
}  // namespace

void clear_last_error() { t_last_error.clear(); }
const char* last_error() { return t_last_error.c_str(); }

int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return status;
}

int device_info(DevInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return fail(FA_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& di = g_dev[dev];
  if (!di.init) {
    cudaDeviceProp prop;
    e = cudaGetDeviceProperties(&prop, dev);
    if (e != cudaSuccess)
      return fail(FA_ERR_CUDA, "cudaGetDeviceProperties: %s", cudaGetErrorString(e));
    di.sms = prop.multiProcessorCount;
    di.major = prop.major;
    di.minor = prop.minor;
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_error_word);
    if (e != cudaSuccess)
      return fail(FA_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    di.err_word = static_cast<int*>(p);
    if (!g_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    di.init = true;
  }
  if (di.major != 10 || di.minor != 3)
    return fail(FA_ERR_ARCH, "device compute capability %d.%d; this library is built for 10.3 "
                "(sm_103a)", di.major, di.minor);
  *out = &di;
  return FA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// [rows, heads, d] bf16 view, boxes of 64 columns x 1 head x box_rows rows, 128B swizzle.
int encode_rows(CUtensorMap* tm, const void* ptr, long long rows, int heads, int d,
                int box_rows) {
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)rows};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)heads * d * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)box_rows};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return FA_OK;
}

// e4m3 codes: a 3-D view (innermost first) with 128-byte rows of 128 codes.
int encode_u8(CUtensorMap* tm, const void* ptr, const cuuint64_t (&dims)[3],
              const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3]) {
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return FA_OK;
}

int read_device_error(int* code, int clear) {
  if (!code) return fail(FA_ERR_INVALID_ARG, "code is NULL");
  DevInfo* di = nullptr;
  int st = device_info(&di);
  if (st != FA_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpyFromSymbol(code, g_error_word, sizeof(int));
  if (e == cudaSuccess && clear) {
    int zero = 0;
    e = cudaMemcpyToSymbol(g_error_word, &zero, sizeof(int));
  }
  if (e != cudaSuccess) return fail(FA_ERR_CUDA, "error word read: %s", cudaGetErrorString(e));
  return FA_OK;
}

int num_sms() {
  DevInfo* di = nullptr;
  return device_info(&di) == FA_OK ? di->sms : 0;
}

int* device_error_word() {
  DevInfo* di = nullptr;
  return device_info(&di) == FA_OK ? di->err_word : nullptr;
}

}  // namespace fa
