// Shared host/device helpers of the CUDA path (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "dllm.h"

namespace dllm {

// ---------------------------------------------------------------------------
// Device status word. Each translation unit owns one; dllm_get_device_status()
// ORs them together. Kernels set bits with atomicOr and never trap.
// ---------------------------------------------------------------------------
uint32_t status_attn(bool clear);
uint32_t status_head(bool clear);
uint32_t status_commit(bool clear);
uint32_t status_model(bool clear);
uint32_t status_moe(bool clear);

#define DLLM_DEFINE_STATUS(tag)                                              \
  static __device__ unsigned int g_status_##tag;                             \
  uint32_t status_##tag(bool clear) {                                        \
    unsigned int v = 0;                                                      \
    if (cudaMemcpyFromSymbol(&v, g_status_##tag, sizeof(v)) != cudaSuccess) \
      return 0x80000000u;                                                    \
    if (clear) {                                                             \
      unsigned int z = 0;                                                    \
      cudaMemcpyToSymbol(g_status_##tag, &z, sizeof(z));                     \
    }                                                                        \
    return v;                                                                \
  }

// Host-side count of kernel launches (dllm_launch_count).
void count_launches(unsigned n);

// CTAs of dllm_block_attn's main kernel without key splits:
// B * H * (query tiles of 128 rows).
int attn_base_ctas(int B, int H, int dh, int max_q);

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

inline bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15) == 0;
}

// Records the CUDA runtime error behind a failed call (per host thread, read
// by dllm_last_cuda_error) and returns DLLM_ERR_CUDA.
dllm_status cuda_error(cudaError_t e);

inline dllm_status launch_status(unsigned launches = 1) {
  count_launches(launches);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? DLLM_OK : cuda_error(e);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch: kernels are launched with the
// programmatic-serialisation attribute, so a kernel may start (and run its
// prologue) while the previous kernel in the stream finishes. Every kernel
// calls pdl_wait() before its first global-memory access, which blocks
// until the previous kernel has completed and its writes are visible, and
// pdl_trigger() to let the next kernel launch early.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Every kernel of the library prefers the largest shared-memory carveout:
// the tcgen05 kernels need it (up to 227 KB), and when a small kernel asked
// for a different L1/shared split, an SM would have to drain and
// reconfigure between it and its neighbours in the stream.
void prefer_max_shared(const void *kern);

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args) {
  prefer_max_shared(reinterpret_cast<const void *>(kern));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// The same for a kernel launched as two-CTA clusters (grid.x even): the CTA
// pairs of tcgen05.mma.cta_group::2.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_pairs(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                    Args &&...args) {
  prefer_max_shared(reinterpret_cast<const void *>(kern));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Device helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Round-to-nearest-even float -> bf16 bits (finite inputs).
__device__ __forceinline__ uint16_t f32_to_bf16(float f) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ uint4 pack8(const float *f) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = static_cast<uint32_t>(f32_to_bf16(f[2 * i])) |
           (static_cast<uint32_t>(f32_to_bf16(f[2 * i + 1])) << 16);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

}  // namespace dllm
