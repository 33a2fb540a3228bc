// K2: LM head + online vocabulary softmax statistics + expected embedding
// (dInfer article: decoding problem 3 -- only the top token of each
// position is normally used -- and "iteration smoothing", which feeds the
// probability-weighted information of undecoded positions forward).
//
// First correct version on the CUDA cores:
//   head_logits : z[r][v] = <h[r], W[v]>              (fp32 scratch)
//   head_stats  : m, lowest argmax, l = sum exp(z-m), conf = 1/l per row
//   pe_partial  : sum over a vocab slice of exp(z-m)/l * E[v]
//   pe_combine  : sum of the slices
#include "common.cuh"

namespace dllm {

DLLM_DEFINE_STATUS(head)

namespace {

constexpr int kTV = 64, kTR = 64, kTK = 32;  // logits tile (vocab x rows x k)
constexpr int kPeSplits = 32;                // vocab slices of the P.E partials
constexpr int kPeRows = 32;                  // head rows per P.E CTA

__global__ void __launch_bounds__(256)
head_logits_kernel(const uint16_t *__restrict__ hid, const uint16_t *__restrict__ w,
                   float *__restrict__ z, int R, int d, int V) {
  __shared__ float Ws[kTK][kTV + 1];
  __shared__ float Hs[kTK][kTR + 1];
  const int v0 = blockIdx.x * kTV, r0 = blockIdx.y * kTR;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;  // 16 x 16 threads, 4x4 outputs each
  float acc[4][4] = {};
  for (int k0 = 0; k0 < d; k0 += kTK) {
    for (int e = threadIdx.x; e < kTV * kTK; e += 256) {
      const int rr = e / kTK, kk = e - rr * kTK;
      const int vv = v0 + rr, hr = r0 + rr;
      Ws[kk][rr] = vv < V ? bf16_to_f32(w[static_cast<size_t>(vv) * d + k0 + kk]) : 0.f;
      Hs[kk][rr] = hr < R ? bf16_to_f32(hid[static_cast<size_t>(hr) * d + k0 + kk]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kTK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) { a[x] = Ws[kk][tx + 16 * x]; b[x] = Hs[kk][ty + 16 * x]; }
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) acc[y][x] = fmaf(b[y], a[x], acc[y][x]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int y = 0; y < 4; ++y) {
    const int r = r0 + ty + 16 * y;
    if (r >= R) continue;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const int vv = v0 + tx + 16 * x;
      if (vv < V) z[static_cast<size_t>(r) * V + vv] = acc[y][x];
    }
  }
}

__global__ void __launch_bounds__(256)
head_stats_kernel(const float *__restrict__ z, int V, float *__restrict__ m_out,
                  float *__restrict__ l_out, int32_t *__restrict__ argmax,
                  float *__restrict__ conf) {
  const int r = blockIdx.x;
  const float *zr = z + static_cast<size_t>(r) * V;
  __shared__ float sm[8];
  __shared__ int sa[8];
  __shared__ float sl[8];
  float m = -INFINITY;
  int a = 0x7fffffff;
  for (int v = threadIdx.x; v < V; v += 256) {
    const float x = zr[v];
    if (x > m) { m = x; a = v; }   // ascending v: first maximum kept
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const int a2 = __shfl_xor_sync(0xffffffffu, a, o);
    if (m2 > m || (m2 == m && a2 < a)) { m = m2; a = a2; }
  }
  if (lane == 0) { sm[warp] = m; sa[warp] = a; }
  __syncthreads();
  m = sm[0]; a = sa[0];
  for (int w = 1; w < 8; ++w)
    if (sm[w] > m || (sm[w] == m && sa[w] < a)) { m = sm[w]; a = sa[w]; }
  float l = 0.f;
  for (int v = threadIdx.x; v < V; v += 256) l += expf(zr[v] - m);
  l = warp_sum(l);
  if (lane == 0) sl[warp] = l;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += sl[w];
    m_out[r] = m;
    l_out[r] = t;
    argmax[r] = a;
    conf[r] = 1.f / t;
  }
}

__global__ void __launch_bounds__(256)
pe_partial_kernel(const float *__restrict__ z, const float *__restrict__ m_in,
                  const float *__restrict__ l_in, const uint16_t *__restrict__ emb,
                  float *__restrict__ part, int R, int d, int V, int slice) {
  __shared__ float ps[kPeRows][33];
  const int col = blockIdx.x * 256 + threadIdx.x;
  const int s = blockIdx.y;
  const int r0 = blockIdx.z * kPeRows;
  const int nr = min(kPeRows, R - r0);
  const int vb = s * slice, ve = min(V, vb + slice);
  float acc[kPeRows];
#pragma unroll
  for (int x = 0; x < kPeRows; ++x) acc[x] = 0.f;
  for (int v0 = vb; v0 < ve; v0 += 32) {
    for (int e = threadIdx.x; e < kPeRows * 32; e += 256) {
      const int rr = e >> 5, vv = e & 31;
      const int v = v0 + vv;
      float p = 0.f;
      if (rr < nr && v < ve) {
        const int r = r0 + rr;
        p = expf(z[static_cast<size_t>(r) * V + v] - m_in[r]) / l_in[r];
      }
      ps[rr][vv] = p;
    }
    __syncthreads();
    if (col < d) {
      const int nv = min(32, ve - v0);
      for (int vv = 0; vv < nv; ++vv) {
        const float e = bf16_to_f32(emb[static_cast<size_t>(v0 + vv) * d + col]);
#pragma unroll
        for (int x = 0; x < kPeRows; ++x) acc[x] = fmaf(ps[x][vv], e, acc[x]);
      }
    }
    __syncthreads();
  }
  if (col < d)
    for (int x = 0; x < nr; ++x)
      part[(static_cast<size_t>(s) * R + r0 + x) * d + col] = acc[x];
}

__global__ void pe_combine_kernel(const float *__restrict__ part, float *__restrict__ pe,
                                  int R, int d, int splits) {
  const size_t n = static_cast<size_t>(R) * d;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; idx < n;
       idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float t = 0.f;
    for (int s = 0; s < splits; ++s) t += part[s * n + idx];
    pe[idx] = t;
  }
}

struct HeadWs {
  size_t z, m, l, part, total;
};

HeadWs head_ws_layout(int R, int d, int V, int with_pe) {
  HeadWs w{};
  size_t off = 0;
  w.z = off; off += align256(static_cast<size_t>(R) * V * sizeof(float));
  w.m = off; off += align256(static_cast<size_t>(R) * sizeof(float));
  w.l = off; off += align256(static_cast<size_t>(R) * sizeof(float));
  w.part = off;
  if (with_pe) off += align256(static_cast<size_t>(kPeSplits) * R * d * sizeof(float));
  w.total = off;
  return w;
}

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" size_t dllm_head_workspace(int R, int d, int V, int with_pe) {
  if (R < 0 || d < 0 || V < 0) return 0;
  return head_ws_layout(R, d, V, with_pe).total;
}

extern "C" dllm_status dllm_head_confidence(const dllm_bf16 *hidden, const dllm_bf16 *w_head,
                                            const dllm_bf16 *emb, int R, int d, int V,
                                            int32_t *argmax, float *conf, float *pe,
                                            void *ws, size_t ws_bytes, dllm_stream stream) {
  if (R < 0 || d < 1 || V < 1) return DLLM_ERR_INVALID_ARG;
  if (d % 64 != 0 || d > 16384 || R > 4096) return DLLM_ERR_UNSUPPORTED;
  if (R == 0) return DLLM_OK;
  if (!hidden || !w_head || !argmax || !conf) return DLLM_ERR_INVALID_ARG;
  if (pe && !emb) return DLLM_ERR_INVALID_ARG;
  const HeadWs L = head_ws_layout(R, d, V, pe != nullptr);
  if (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return DLLM_ERR_WORKSPACE;
  char *base = static_cast<char *>(ws);
  float *z = reinterpret_cast<float *>(base + L.z);
  float *m = reinterpret_cast<float *>(base + L.m);
  float *l = reinterpret_cast<float *>(base + L.l);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  dim3 g1((V + kTV - 1) / kTV, (R + kTR - 1) / kTR);
  head_logits_kernel<<<g1, 256, 0, s>>>(hidden, w_head, z, R, d, V);
  head_stats_kernel<<<R, 256, 0, s>>>(z, V, m, l, argmax, conf);
  if (pe) {
    float *part = reinterpret_cast<float *>(base + L.part);
    const int slice = (V + kPeSplits - 1) / kPeSplits;
    dim3 g2((d + 255) / 256, kPeSplits, (R + kPeRows - 1) / kPeRows);
    pe_partial_kernel<<<g2, 256, 0, s>>>(z, m, l, emb, part, R, d, V, slice);
    pe_combine_kernel<<<1024, 256, 0, s>>>(part, pe, R, d, kPeSplits);
  }
  return launch_status(pe ? 4 : 2);
}
