// The LM head for callers that cannot allocate device memory.
//
// dllm_head_confidence() needs a caller-provided workspace. Some callers can
// neither call cudaMalloc nor keep a buffer of their own: a plugin whose host
// framework owns every byte of device memory and hands it no allocator, or a
// thread that must not block (cudaMalloc can synchronise the whole device).
// dllm_head_confidence_noalloc() serves them: it runs exactly the same
// kernels, with the scratch placed in the fixed array below, which the
// library's module reserves on every GPU that loads it, until the process
// exits.
//
// The array's name, in host code, is only a stand-in for the symbol, not a
// device address; its device address is looked up once per device with
// cudaGetSymbolAddress (the first call made on each device does this, so
// that first call should come before any stream capture), and again when
// the device's context has changed since (after cudaDeviceReset the module
// is loaded anew and the array may sit elsewhere). Every call shares
// the one array and leaves its contents behind; nothing in it needs to start
// at zero, because each call writes every scratch element it reads. Calls
// whose work overlaps on the GPU (two streams, two host threads) race on the
// array: serialise them.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace dllm {
namespace {

static __device__ __align__(256) unsigned char g_head_scratch[DLLM_HEAD_NOALLOC_SCRATCH_BYTES];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// The calling thread's current driver context (nullptr if none or if the
// query is unavailable), fetched through the runtime's entry-point query so
// that the library keeps no link-time driver dependency.
CUcontext current_context() {
  static CtxGetCurrentFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<CtxGetCurrentFn>(p);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct ScratchSlot {
  CUcontext ctx;
  void *ptr;
};
ScratchSlot g_slot[kMaxDevices] = {};

// Device address of the scratch array on the current device: looked up on
// the first call per device, and again whenever the current context is not
// the one the address was taken in. Returns nullptr on failure.
void *scratch_on_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchSlot &slot = g_slot[dev];
  if (!slot.ptr || !slot.ctx || slot.ctx != current_context()) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_head_scratch) != cudaSuccess) return nullptr;
    slot.ptr = p;
    slot.ctx = current_context();   // after the look-up, which makes the context current
  }
  return slot.ptr;
}

}  // namespace
}  // namespace dllm

extern "C" dllm_status dllm_head_confidence_noalloc(const dllm_bf16 *hidden, const dllm_bf16 *w_head,
                                                    const dllm_bf16 *emb, int R, int d, int V,
                                                    int32_t *argmax, float *conf, float *pe,
                                                    dllm_stream stream) {
  if (R < 0 || d < 1 || V < 1) return DLLM_ERR_INVALID_ARG;
  const size_t need = dllm_head_workspace(R, d, V, pe != nullptr);
  if (need > static_cast<size_t>(DLLM_HEAD_NOALLOC_SCRATCH_BYTES)) return DLLM_ERR_UNSUPPORTED;
  if (R == 0) return DLLM_OK;
  void *ws = dllm::scratch_on_current_device();
  if (!ws) return DLLM_ERR_CUDA;
  return dllm_head_confidence(hidden, w_head, emb, R, d, V, argmax, conf, pe, ws,
                              static_cast<size_t>(DLLM_HEAD_NOALLOC_SCRATCH_BYTES), stream);
}
