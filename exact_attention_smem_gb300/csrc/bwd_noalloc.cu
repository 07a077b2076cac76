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
// current and caches it; make that first call before any stream capture. The
// cached address is tied to the CUDA context it was looked up in: after a
// cudaDeviceReset (or any other replacement of the device's primary context)
// the next call sees a different current context and looks the address up
// again.
// All calls share the one array and it keeps the previous call's contents; the
// backward's preprocess pass zeroes the dQ accumulator and rewrites the row
// arrays on every call, so nothing stale is read. Calls whose work overlaps on
// the GPU (other streams, or other threads) race on the array and give wrong
// results: serialise them.
#include "../../include/fa.h"
#include "host_common.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_bwd_scratch[FA_BWD_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);

struct ScratchSlot {
  CUcontext ctx = nullptr;       // context the address was looked up in
  void* addr = nullptr;
};

std::mutex g_scratch_mu;
ScratchSlot g_scratch[64];
CtxGetCurrentFn g_ctx_get_current = nullptr;

CUcontext current_context() {
  if (!g_ctx_get_current) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  CUcontext c = nullptr;
  return g_ctx_get_current(&c) == CUDA_SUCCESS ? c : nullptr;
}

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int Hq, int Hkv, int Sq, int Sk, int d, int causal,
                              float scale, const int* cu_seqlens, void* stream) {
  const size_t need =
      fa_bwd_workspace_bytes(B, Hq, Sq, d, cu_seqlens ? Sq : 0);
  if (need > (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES)
    return fa::fail(FA_ERR_WORKSPACE,
                            "this backward needs %zu bytes of scratch but the built-in scratch of "
                            "fa_bwd_noalloc holds %zu bytes; call fa_bwd with a workspace instead",
                            need, (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return fa::fail(FA_ERR_CUDA, "no current CUDA device");
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    ScratchSlot& slot = g_scratch[dev];
    // A thread the runtime has not used yet may have no current context: the
    // lookup below makes the device's primary context current.
    CUcontext ctx = current_context();
    if (!slot.addr || !ctx || ctx != slot.ctx) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_bwd_scratch);
      if (e != cudaSuccess || !p)
        return fa::fail(FA_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
      slot.addr = p;
      slot.ctx = current_context();
    }
    scratch = slot.addr;
  }
  return fa_bwd(q, k, v, o, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Sk, d, causal, scale,
                cu_seqlens, scratch, (size_t)FA_BWD_NOALLOC_SCRATCH_BYTES, stream);
}
