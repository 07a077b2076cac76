// fa_bwd_noalloc: the backward for callers that cannot allocate device memory.
//
// fa_bwd needs a scratch workspace (the fp32 dQ accumulator and two padded
// fp32 row arrays) that the caller allocates. Some callers cannot do that: a
// runtime whose device memory is entirely owned by its own pool allocator
// (a raw cudaMalloc would bypass its accounting), or code on a latency path
// where cudaMalloc is not allowed because it can synchronise the whole device.
// This entry point takes the same inputs and outputs as fa_bwd and uses a
// fixed scratch array that lives in the library itself instead.
//
// The scratch is a file-scope __device__ array of FA_BWD_NOALLOC_SCRATCH_BYTES
// bytes. Every GPU that loads this library holds it until the process exits.
// Host code cannot pass the array's name to a kernel (on the host it is only a
// stand-in symbol, not a device address), so the first call on each device
// looks the device address up with cudaGetSymbolAddress while that device is
// current and caches it; make that first call before any stream capture.
// All calls share the one array and it keeps the previous call's contents; the
// backward's preprocess pass zeroes the dQ accumulator and rewrites the row
// arrays on every call, so nothing stale is read. Calls whose work overlaps on
// the GPU (other streams, or other threads) race on the array and give wrong
// results: serialise them.
#include "../../include/fa.h"

#include <cuda_runtime.h>

#include <mutex>

namespace fa {
int report_error(int status, const char* fmt, ...);  // sets fa_last_error(); api.cu
}

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {nullptr};

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal,
                              float scale, const int* cu_seqlens, void* stream) {
  const size_t need =
      fa_bwd_workspace_bytes(B, Hq, Sq, d, cu_seqlens ? Sq : 0);
  if (need > (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES)
    return fa::report_error(FA_ERR_WORKSPACE,
                            "this backward needs %zu bytes of scratch but the built-in scratch of "
                            "fa_bwd_noalloc holds %zu bytes; call fa_bwd with a workspace instead",
                            need, (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return fa::report_error(FA_ERR_CUDA, "no current CUDA device");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
      if (e != cudaSuccess || !p)
        return fa::report_error(FA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s",
                                cudaGetErrorString(e));
      g_scratch_addr[dev] = p;
    }
    scratch = g_scratch_addr[dev];
  }
  return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale,
                cu_seqlens, scratch, (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES, stream);
}
