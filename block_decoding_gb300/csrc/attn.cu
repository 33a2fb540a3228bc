// K1: non-causal attention of the window queries over cached prefix + fresh
// window K/V (dInfer article, "vicinity KV refresh"; Sangam abstract:
// bidirectional attention).
//
// First correct version: one warp per query row, K/V tiles staged in shared
// memory, fp32 online softmax on the CUDA cores.
#include "common.cuh"

namespace dllm {

DLLM_DEFINE_STATUS(attn)

namespace {

constexpr int kWarps = 8;
constexpr int kKeyTile = 64;

template <int DH>
__global__ void __launch_bounds__(kWarps * 32)
attn_rows_kernel(const uint16_t *__restrict__ q, const uint16_t *__restrict__ k,
                 const uint16_t *__restrict__ v, void *__restrict__ out, int out_fp32,
                 const int32_t *__restrict__ q_off, const int32_t *__restrict__ kv_off,
                 int H, float scale) {
  constexpr int E = DH / 32;  // dims per lane
  __shared__ __align__(16) uint16_t Ks[kKeyTile][DH];
  __shared__ __align__(16) uint16_t Vs[kKeyTile][DH];

  const int i = blockIdx.z, h = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q0 = q_off[i], W = q_off[i + 1] - q0;
  const int k0 = kv_off[i], L = kv_off[i + 1] - k0;
  const int t0 = blockIdx.x * kWarps;
  if (t0 >= W) return;
  const int t = t0 + warp;
  const bool active = t < W;
  const size_t row_stride = static_cast<size_t>(H) * DH;

  float qr[E], o[E];
#pragma unroll
  for (int e = 0; e < E; ++e) { qr[e] = 0.f; o[e] = 0.f; }
  if (active) {
    const uint16_t *qp = q + (q0 + t) * row_stride + h * DH + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) qr[e] = bf16_to_f32(qp[e]) * scale;
  }
  float m = -INFINITY, l = 0.f;

  constexpr int kChunks = DH * 2 / 16;  // 16-byte chunks per row
  for (int u0 = 0; u0 < L; u0 += kKeyTile) {
    const int n = min(kKeyTile, L - u0);
    for (int c = threadIdx.x; c < n * kChunks; c += blockDim.x) {
      const int r = c / kChunks, cc = c - r * kChunks;
      const size_t g = (k0 + u0 + r) * row_stride + h * DH;
      reinterpret_cast<uint4 *>(&Ks[r][0])[cc] = reinterpret_cast<const uint4 *>(k + g)[cc];
      reinterpret_cast<uint4 *>(&Vs[r][0])[cc] = reinterpret_cast<const uint4 *>(v + g)[cc];
    }
    __syncthreads();
    if (active) {
      for (int u = 0; u < n; ++u) {
        float s = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) s = fmaf(qr[e], bf16_to_f32(Ks[u][lane * E + e]), s);
        s = warp_sum(s);
        const float mn = fmaxf(m, s);
        const float corr = __expf(m - mn);
        const float pu = __expf(s - mn);
        l = l * corr + pu;
#pragma unroll
        for (int e = 0; e < E; ++e) o[e] = fmaf(o[e], corr, pu * bf16_to_f32(Vs[u][lane * E + e]));
        m = mn;
      }
    }
    __syncthreads();
  }
  if (!active) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const size_t ob = (q0 + t) * row_stride + h * DH + lane * E;
  if (out_fp32) {
    float *op = static_cast<float *>(out) + ob;
#pragma unroll
    for (int e = 0; e < E; ++e) op[e] = o[e] * inv;
  } else {
    uint16_t *op = static_cast<uint16_t *>(out) + ob;
#pragma unroll
    for (int e = 0; e < E; ++e) op[e] = f32_to_bf16(o[e] * inv);
  }
}

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" size_t dllm_block_attn_workspace(int B, int H, int dh, int max_q, int max_kv) {
  (void)B; (void)H; (void)dh; (void)max_q; (void)max_kv;
  return 0;
}

extern "C" dllm_status dllm_block_attn(const dllm_bf16 *q, const dllm_bf16 *k,
                                       const dllm_bf16 *v, void *out, int out_fp32,
                                       const int32_t *q_off, const int32_t *kv_off,
                                       int B, int H, int dh, int max_q, int max_kv,
                                       float scale, void *ws, size_t ws_bytes,
                                       dllm_stream stream) {
  (void)ws; (void)ws_bytes;
  if (B < 0 || H < 1 || max_q < 0 || max_kv < 0) return DLLM_ERR_INVALID_ARG;
  if (dh != 64 && dh != 128) return DLLM_ERR_UNSUPPORTED;
  if (B > 4096 || H > 256) return DLLM_ERR_UNSUPPORTED;
  if (B == 0 || max_q == 0) return DLLM_OK;
  if (!q || !k || !v || !out || !q_off || !kv_off) return DLLM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return DLLM_ERR_INVALID_ARG;
  dim3 grid((max_q + kWarps - 1) / kWarps, H, B);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dh == 64)
    attn_rows_kernel<64><<<grid, kWarps * 32, 0, s>>>(q, k, v, out, out_fp32, q_off, kv_off, H, scale);
  else
    attn_rows_kernel<128><<<grid, kWarps * 32, 0, s>>>(q, k, v, out, out_fp32, q_off, kv_off, H, scale);
  return launch_status();
}
