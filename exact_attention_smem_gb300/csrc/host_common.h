// Host-side helpers shared by the C-ABI translation units: the thread's last
// error text, the per-device property cache (with the device error word), and
// TMA tensor-map encoding. Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

struct DevInfo {
  bool init = false;
  int sms = 0, major = 0, minor = 0;
  int* err_word = nullptr;       // device address of this library's error word
};

// Records a printf-style message as the thread's last error; returns status.
int fail(int status, const char* fmt, ...);
void clear_last_error();
const char* last_error();

// Properties of the current device (cached per device, thread-safe); fails with
// FA_ERR_ARCH unless the device is compute capability 10.3.
int device_info(DevInfo** out);

bool aligned16(const void* p);

// [rows, heads, d] bf16 view, boxes of 64 columns x 1 head x box_rows rows, 128B swizzle.
int encode_rows(CUtensorMap* tm, const void* ptr, long long rows, int heads, int d,
                int box_rows = 128);
// e4m3 codes: a 3-D view (innermost first) with 128-byte rows of 128 codes.
int encode_u8(CUtensorMap* tm, const void* ptr, const cuuint64_t (&dims)[3],
              const cuuint64_t (&strides)[2], const cuuint32_t (&box)[3]);

// Synchronises the device, reads (and optionally clears) the error word.
int read_device_error(int* code, int clear);

}  // namespace fa
