// The end-to-end pieces: a small bidirectional transformer run block by
// block with a prefix K/V cache (Sangam abstract: approximate caching with
// recurring per-block prefills; dInfer article, "vicinity KV refresh": each
// iteration recomputes only the block and its neighbourhood).
//
//   dllm_gemm_bf16      C = A W^T on tcgen05 (swap-AB: weight rows on M), with
//                       plain, residual-add or SwiGLU (gate/up) epilogues
//   dllm_model_forward  all layers over a window of rows whose keys are the
//                       cached prefix + the window: RMSNorm -> QKV GEMM ->
//                       RoPE + cache write -> attention -> O GEMM + residual
//                       -> RMSNorm -> gate/up GEMM + SwiGLU -> down GEMM +
//                       residual; final RMSNorm
//   dllm_decode_step    one whole step of the block decode loop: input rows
//                       (committed tokens, smoothed block rows, mask rows) ->
//                       forward -> head (+P.E) -> commit -> sequence write-back
#include "umma_gemm.cuh"

namespace dllm {

DLLM_DEFINE_STATUS(model)

// Programmatic-dependent launch of a kernel on the step chain (see common.cuh).
#define LAUNCH(kern, grid, block, stream, ...)                                                    \
  do {                                                                                           \
    if (launch_pdl(kern, dim3(grid), dim3(block), 0, stream, __VA_ARGS__) != cudaSuccess)        \
      return DLLM_ERR_CUDA;                                                                      \
  } while (0)

namespace {

// ---------------------------------------------------------------------------
// small ops
// ---------------------------------------------------------------------------
// y = x / sqrt(mean(x^2) + eps), one row per CTA, fp32 arithmetic. CTA 0
// also writes the step's small metadata (so that no separate launch does):
// the offsets of a one-request attention call, meta[0..4) = {0, n, 0, L},
// and the identity head-row map of a blk-position block, meta[4 + j] = 0,
// meta[4 + 64 + j] = j.
__global__ void __launch_bounds__(128)
rmsnorm_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ y, int d, float eps, int32_t *meta, int n,
               int L, int blk) {
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x;
  if (r == 0) {
    const int j = threadIdx.x;
    if (j == 0) { meta[0] = 0; meta[1] = n; meta[2] = 0; meta[3] = L; }
    if (j < blk) { meta[4 + j] = 0; meta[4 + 64 + j] = j; }
  }
  const uint4 *x4 = reinterpret_cast<const uint4 *>(x + static_cast<size_t>(r) * d);
  uint4 *y4 = reinterpret_cast<uint4 *>(y + static_cast<size_t>(r) * d);
  float ss = 0.f;
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) {
    float f[8];
    unpack8(x4[c], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
  }
  __shared__ float part[4];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  const float tot = part[0] + part[1] + part[2] + part[3];
  const float inv = rsqrtf(tot / d + eps);
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) {
    float f[8];
    unpack8(x4[c], f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] *= inv;
    y4[c] = pack8(f);
  }
}

// A decode step's first kernel: row t of the step gathers its input row
// into x -- the block's next-step row for a block position (window steps),
// else E[token], or E[mask_id] for a masked position -- then
// h = x / sqrt(mean(x^2) + eps) from the same registers (rmsnorm_kernel's
// arithmetic); CTA 0 also writes the step's metadata as rmsnorm_kernel does.
__global__ void __launch_bounds__(128)
embed_norm_kernel(uint16_t *__restrict__ x, uint16_t *__restrict__ h, int row0, int n,
                  const int32_t *__restrict__ tokens, const uint8_t *__restrict__ masked,
                  const uint16_t *__restrict__ block_emb, int b0, int blk, int use_block,
                  const uint16_t *__restrict__ emb, int V, int mask_id, int d, float eps, int32_t *meta, int L,
                  int meta_blk, unsigned int *status) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  if (t == 0) {
    const int j = threadIdx.x;
    if (j == 0) { meta[0] = 0; meta[1] = n; meta[2] = 0; meta[3] = L; }
    if (j < meta_blk) { meta[4 + j] = 0; meta[4 + 64 + j] = j; }
  }
  const int p = row0 + t;
  const uint16_t *src;
  if (use_block && p >= b0 && p < b0 + blk) {
    src = block_emb + static_cast<size_t>(p - b0) * d;
  } else {
    int id = masked[p] ? mask_id : tokens[p];
    if (id < 0 || id >= V) {
      if (threadIdx.x == 0) atomicOr(status, DLLM_DEV_ID_RANGE);
      id = mask_id;
    }
    src = emb + static_cast<size_t>(id) * d;
  }
  const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
  uint4 *x4 = reinterpret_cast<uint4 *>(x + static_cast<size_t>(t) * d);
  uint4 *h4 = reinterpret_cast<uint4 *>(h + static_cast<size_t>(t) * d);
  constexpr int kMaxChunks = 4;   // d / 8 / 128 (d <= 4096)
  uint4 keep[kMaxChunks];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = threadIdx.x + k * 128;
    if (c < d / 8) {
      keep[k] = s4[c];
      x4[c] = keep[k];
      float f[8];
      unpack8(keep[k], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
    }
  }
  __shared__ float part[4];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = ss;
  __syncthreads();
  const float inv = rsqrtf((part[0] + part[1] + part[2] + part[3]) / d + eps);
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = threadIdx.x + k * 128;
    if (c < d / 8) {
      float f[8];
      unpack8(keep[k], f);
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] *= inv;
      h4[c] = pack8(f);
    }
  }
}

__global__ void writeback_kernel(int32_t *tokens, uint8_t *masked, const int32_t *btok, const uint8_t *bmask,
                                 int b0, int blk) {
  pdl_trigger();
  pdl_wait();
  const int j = threadIdx.x;
  if (j < blk) {
    tokens[b0 + j] = btok[j];
    masked[b0 + j] = bmask[j];
  }
}

// ---------------------------------------------------------------------------
// GEMM: C[tokens][features] = X[tokens][K] . W[features][K]^T (swap-AB)
//
// A few window tokens leave each projection latency-bound: its CTAs stream
// a few tens of KB each, so the DRAM latency of the first loads dominates.
// Every projection therefore also prefetches the next projection's weights
// into L2 (they do not depend on its result; 129 MB of L2 hold a layer's
// 34 MB twice over), and the next one's loads hit L2.
// ---------------------------------------------------------------------------
struct L2Next {
  const void *p = nullptr;
  unsigned long long bytes = 0;
};

template <int BN, int EPI>
bool gemm_t(const uint16_t *X, const uint16_t *W, uint16_t *C, int M, int N, int K, int w_rows,
            const uint16_t *aux, int a1_row, cudaStream_t s, L2Next pf = {}) {
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_sw128(&ta, W, w_rows, K, K, 128)) return false;
  if (!make_tmap_bf16_sw128(&tb, X, M, K, K, BN)) return false;
  UmmaArgs a{};
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&a.status), g_status_model) != cudaSuccess) return false;
  a.m_tiles = (N + 127) / 128;
  a.n_blocks = (M + BN - 1) / BN;
  a.k_splits = 1;
  a.k_steps = K / 64;
  a.k_per_split = a.k_steps;
  a.M = N;
  a.N = M;
  a.ld = N;
  a.outb = C;
  a.aux = aux;
  a.a1_row = a1_row;
  a.pf = pf.p;
  a.pf_bytes = pf.bytes;
  return launch_umma_gemm<BN, false, EPI>(ta, tb, a, s);
}

// epilogue: 0 none, 1 residual (C = X W^T + aux), 2 SwiGLU (W = [2N][K]: gate rows then up rows)
bool gemm_bf16(const uint16_t *X, const uint16_t *W, uint16_t *C, int M, int N, int K, int epilogue,
               const uint16_t *aux, cudaStream_t s, L2Next pf = {}) {
  if (epilogue == 2) {
    if (M <= 16) return gemm_t<16, kEpiSwiGLU>(X, W, C, M, N, K, 2 * N, nullptr, N, s, pf);
    if (M <= 32) return gemm_t<32, kEpiSwiGLU>(X, W, C, M, N, K, 2 * N, nullptr, N, s, pf);
    if (M <= 64) return gemm_t<64, kEpiSwiGLU>(X, W, C, M, N, K, 2 * N, nullptr, N, s, pf);
    return gemm_t<128, kEpiSwiGLU>(X, W, C, M, N, K, 2 * N, nullptr, N, s, pf);
  }
  const uint16_t *ax = epilogue == 1 ? aux : nullptr;
  if (M <= 16) return gemm_t<16, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s, pf);
  if (M <= 32) return gemm_t<32, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s, pf);
  if (M <= 64) return gemm_t<64, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s, pf);
  if (M <= 128) return gemm_t<128, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s, pf);
  return gemm_t<256, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s, pf);
}

// ---------------------------------------------------------------------------
// Split-K for few tokens: with 96 window tokens a projection has only
// N/128 weight tiles (8..64), too few CTAs to stream the weights at full
// bandwidth. The K range is split so that about one unit runs per SM; fp32
// partials [split][tokens][N] (a few MB, mostly L2-resident) are reduced by
// one epilogue kernel that also applies the residual or SwiGLU.
// ---------------------------------------------------------------------------
// Splits so that the units (tiles x splits) fill the SMs in one wave: more
// would leave a second, mostly empty wave. The count is monotone in `sms`,
// so sizing scratch with the largest SM count covers every GPU.
int splitk_count(int n_feat, int tokens, int K, int sms = num_sms()) {
  const int m_tiles = (n_feat + 127) / 128;
  const int bn = tokens <= 16 ? 16 : tokens <= 32 ? 32 : tokens <= 64 ? 64 : tokens <= 128 ? 128 : 256;
  const int n_blocks = (tokens + bn - 1) / bn;
  const int base = m_tiles * n_blocks;
  const int k_steps = K / 64;
  if (2 * base > sms || k_steps < 2) return 1;
  int s = sms / base;
  if (s > k_steps) s = k_steps;
  return s;
}

// mode 0: C = sum; 1: C = sum + aux; 2: SwiGLU over [gate | up] halves of the
// n_in = 2 * n_out partial columns.
__global__ void __launch_bounds__(256)
splitk_epilogue_kernel(const float *__restrict__ part, int splits, int tokens, int n_in, int n_out, int mode,
                       const uint16_t *aux, uint16_t *out) {
  pdl_trigger();
  pdl_wait();
  const size_t per = static_cast<size_t>(tokens) * n_in;
  const int n4 = n_out / 4;
  for (size_t idx = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
       idx < static_cast<size_t>(tokens) * n4; idx += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int t = static_cast<int>(idx / n4);
    const int c = static_cast<int>(idx - static_cast<size_t>(t) * n4) * 4;
    float a[4] = {0.f, 0.f, 0.f, 0.f}, g[4] = {0.f, 0.f, 0.f, 0.f};
    for (int s = 0; s < splits; ++s) {
      const float *row = part + s * per + static_cast<size_t>(t) * n_in;
      const float4 x = *reinterpret_cast<const float4 *>(row + c);
      a[0] += x.x; a[1] += x.y; a[2] += x.z; a[3] += x.w;
      if (mode == 2) {
        const float4 u = *reinterpret_cast<const float4 *>(row + n_out + c);
        g[0] += u.x; g[1] += u.y; g[2] += u.z; g[3] += u.w;
      }
    }
    uint16_t *o = out + static_cast<size_t>(t) * n_out + c;
    float r[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      if (mode == 2) r[e] = a[e] / (1.f + __expf(-a[e])) * g[e];   // silu(gate) * up
      else r[e] = a[e] + (mode == 1 ? bf16_to_f32(aux[static_cast<size_t>(t) * n_out + c + e]) : 0.f);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] = f32_to_bf16(r[e]);
  }
}

// QKV projection finished from its fp32 partials: q, k, v of token t summed
// over the K splits, RoPE on q and k, q -> q_out [n][d], k, v -> cache row
// kv_row0 + t. One CTA per token.
__global__ void __launch_bounds__(256)
qkv_rope_epilogue_kernel(const float *__restrict__ part, int splits, int tokens, int H, int dh, int pos0,
                         float log2_base, uint16_t *__restrict__ q_out, uint16_t *__restrict__ kc,
                         uint16_t *__restrict__ vc, int kv_row0) {
  pdl_trigger();
  pdl_wait();
  // grid (token, section): section 0 = q, 1 = k (rotated), 2 = v
  const int t = blockIdx.x, sec = blockIdx.y;
  const int d = H * dh, half = dh / 2, n_in = 3 * d;
  const size_t per = static_cast<size_t>(tokens) * n_in;
  const float *row = part + static_cast<size_t>(t) * n_in + static_cast<size_t>(sec) * d;
  const float pos = static_cast<float>(pos0 + t);
  uint16_t *o = sec == 0 ? q_out + static_cast<size_t>(t) * d
                         : (sec == 1 ? kc : vc) + static_cast<size_t>(kv_row0 + t) * d;
  for (int idx = threadIdx.x; idx < H * half; idx += blockDim.x) {
    const int h = idx / half, i = idx - h * half;
    const int a = h * dh + i, b = a + half;
    float x1 = 0.f, x2 = 0.f;
#pragma unroll 4
    for (int s = 0; s < splits; ++s) {
      x1 += row[s * per + a];
      x2 += row[s * per + b];
    }
    if (sec == 2) {
      o[a] = f32_to_bf16(x1);
      o[b] = f32_to_bf16(x2);
      continue;
    }
    // activations are bf16 between kernels: round the projection first
    x1 = bf16_to_f32(f32_to_bf16(x1));
    x2 = bf16_to_f32(f32_to_bf16(x2));
    const float inv_freq = exp2f(-(2.f * i / dh) * log2_base);
    float sn, cs;
    sincosf(pos * inv_freq, &sn, &cs);
    o[a] = f32_to_bf16(x1 * cs - x2 * sn);
    o[b] = f32_to_bf16(x2 * cs + x1 * sn);
  }
}

// Residual projection finished from its fp32 partials, then the next
// RMSNorm: x[t] <- bf16(x[t] + sum_s part[s][t]); h[t] = x[t] / rms(x[t]).
// One CTA per token (d <= 4096: 128 threads x 8 x 4 values).
__global__ void __launch_bounds__(128)
residual_norm_epilogue_kernel(const float *__restrict__ part, int splits, int tokens, int d, uint16_t *x,
                              uint16_t *__restrict__ h, float eps) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  const size_t per = static_cast<size_t>(tokens) * d;
  uint4 *x4 = reinterpret_cast<uint4 *>(x + static_cast<size_t>(t) * d);
  uint4 *h4 = reinterpret_cast<uint4 *>(h + static_cast<size_t>(t) * d);
  constexpr int kMaxChunks = 4;  // d / 8 / 128
  float keep[kMaxChunks][8];
  float ss = 0.f;
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = threadIdx.x + k * 128;
    if (c >= d / 8) break;
    float f[8];
    unpack8(x4[c], f);
#pragma unroll 8
    for (int s = 0; s < splits; ++s) {
      const float4 *p = reinterpret_cast<const float4 *>(part + s * per + static_cast<size_t>(t) * d + c * 8);
      const float4 a = p[0], b = p[1];
      f[0] += a.x; f[1] += a.y; f[2] += a.z; f[3] += a.w; f[4] += b.x; f[5] += b.y; f[6] += b.z; f[7] += b.w;
    }
    const uint4 packed = pack8(f);
    x4[c] = packed;
    unpack8(packed, keep[k]);   // the stored (bf16) residual stream feeds the norm
#pragma unroll
    for (int e = 0; e < 8; ++e) ss = fmaf(keep[k][e], keep[k][e], ss);
  }
  __shared__ float red[4];
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  const float inv = rsqrtf((red[0] + red[1] + red[2] + red[3]) / d + eps);
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int c = threadIdx.x + k * 128;
    if (c >= d / 8) break;
    float f[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = keep[k][e] * inv;
    h4[c] = pack8(f);
  }
}

template <int BN>
bool gemm_partials(const uint16_t *X, const uint16_t *W, float *part, int M, int N, int K, int splits,
                   cudaStream_t s, L2Next pf = {}) {
  CUtensorMap ta, tb;
  if (!make_tmap_bf16_sw128(&ta, W, N, K, K, 128)) return false;
  if (!make_tmap_bf16_sw128(&tb, X, M, K, K, BN)) return false;
  UmmaArgs a{};
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&a.status), g_status_model) != cudaSuccess) return false;
  a.m_tiles = (N + 127) / 128;
  a.n_blocks = (M + BN - 1) / BN;
  a.k_steps = K / 64;
  a.k_per_split = (a.k_steps + splits - 1) / splits;
  a.k_splits = (a.k_steps + a.k_per_split - 1) / a.k_per_split;
  a.M = N;
  a.N = M;
  a.ld = N;
  a.out = part;
  a.pf = pf.p;
  a.pf_bytes = pf.bytes;
  return launch_umma_gemm<BN, false, kEpiStoreT>(ta, tb, a, s);
}

// C[M tokens][n_out] from X[M][K] and W: epilogue as in gemm_bf16; splits K
// when the weight tiles alone would leave most SMs idle. part: fp32 scratch
// of at least splitk_count(...) * M * (2 n_out for SwiGLU, else n_out) floats.
bool gemm_auto(const uint16_t *X, const uint16_t *W, uint16_t *C, int M, int n_out, int K, int epilogue,
               const uint16_t *aux, float *part, cudaStream_t s, L2Next pf = {}) {
  const int n_in = epilogue == 2 ? 2 * n_out : n_out;
  const int splits = splitk_count(n_in, M, K);
  if (splits <= 1) return gemm_bf16(X, W, C, M, n_out, K, epilogue, aux, s, pf);
  bool ok;
  if (M <= 16) ok = gemm_partials<16>(X, W, part, M, n_in, K, splits, s, pf);
  else if (M <= 32) ok = gemm_partials<32>(X, W, part, M, n_in, K, splits, s, pf);
  else if (M <= 64) ok = gemm_partials<64>(X, W, part, M, n_in, K, splits, s, pf);
  else if (M <= 128) ok = gemm_partials<128>(X, W, part, M, n_in, K, splits, s, pf);
  else ok = gemm_partials<256>(X, W, part, M, n_in, K, splits, s, pf);
  if (!ok) return false;
  const int k_steps = K / 64, per = (k_steps + splits - 1) / splits, real = (k_steps + per - 1) / per;
  const size_t items = static_cast<size_t>(M) * (n_out / 4);
  const int grid = static_cast<int>(items / 256 + 1 < 2048 ? items / 256 + 1 : 2048);
  if (launch_pdl(splitk_epilogue_kernel, dim3(grid), dim3(256), 0, s, static_cast<const float *>(part), real, M, n_in,
                 n_out, epilogue, aux, C) != cudaSuccess)
    return false;
  count_launches(1);
  return true;
}

// fp32 partials of X W^T in `part` ([splits][M][N]); returns the number of K
// splits written (>= 1), or 0 on a launch failure.
int gemm_to_partials(const uint16_t *X, const uint16_t *W, float *part, int M, int N, int K, cudaStream_t s,
                     L2Next pf = {}) {
  const int splits = splitk_count(N, M, K);
  bool ok;
  if (M <= 16) ok = gemm_partials<16>(X, W, part, M, N, K, splits, s, pf);
  else if (M <= 32) ok = gemm_partials<32>(X, W, part, M, N, K, splits, s, pf);
  else if (M <= 64) ok = gemm_partials<64>(X, W, part, M, N, K, splits, s, pf);
  else if (M <= 128) ok = gemm_partials<128>(X, W, part, M, N, K, splits, s, pf);
  else ok = gemm_partials<256>(X, W, part, M, N, K, splits, s, pf);
  if (!ok) return 0;
  const int k_steps = K / 64, per = (k_steps + splits - 1) / splits;
  return (k_steps + per - 1) / per;
}

size_t splitk_bytes(int n_feat, int tokens, int K) {
  return static_cast<size_t>(splitk_count(n_feat, tokens, K, 256)) * tokens * n_feat * 4;
}

bool model_ok(const dllm_model *m) {
  if (!m || m->layers < 1 || m->d < 64 || m->H < 1 || (m->dh != 64 && m->dh != 128) || m->H * m->dh != m->d)
    return false;
  if (m->d % 64 || m->d > 4096 || m->ffn % 64 || m->ffn < 64 || m->V < 2 || !m->emb || !m->w_head) return false;
  if (!m->wqkv || !m->wo || !m->wgu || !m->wdown) return false;
  for (int l = 0; l < m->layers; ++l)
    if (!m->wqkv[l] || !m->wo[l] || !m->wgu[l] || !m->wdown[l]) return false;
  return true;
}

struct FwdWs {
  size_t x, h, q, o, f, meta, part, attn, total;
};

FwdWs fwd_layout(const dllm_model *m, int n) {
  FwdWs w{};
  size_t off = 0;
  auto take = [&](size_t b) { const size_t o = off; off += align256(b); return o; };
  const size_t rd = static_cast<size_t>(n) * m->d * 2;
  w.x = take(rd);
  w.h = take(rd);
  w.q = take(rd);
  w.o = take(rd);
  w.f = take(static_cast<size_t>(n) * m->ffn * 2);
  w.meta = take(4 * 140);
  size_t pb = splitk_bytes(3 * m->d, n, m->d);
  const size_t cand[3] = {splitk_bytes(m->d, n, m->d), splitk_bytes(2 * m->ffn, n, m->d),
                          splitk_bytes(m->d, n, m->ffn)};
  for (size_t c : cand) pb = c > pb ? c : pb;
  w.part = take(pb > 0 ? pb : 256);
  w.attn = off;
  off += align256(dllm_block_attn_workspace(1, m->H, m->dh, n, m->max_seq));
  w.total = off;
  return w;
}

// All layers over n rows already in ws.x (positions pos0..), keys = cache
// rows [0, L); writes the final-normed rows to out.
dllm_status forward_rows(const dllm_model *m, char *base, const FwdWs &W, int n, int pos0, int L,
                         dllm_bf16 *const *k_cache, dllm_bf16 *const *v_cache, dllm_bf16 *out, cudaStream_t s,
                         int row_map_blk = 0, bool normed = false) {
  uint16_t *x = reinterpret_cast<uint16_t *>(base + W.x);
  uint16_t *h = reinterpret_cast<uint16_t *>(base + W.h);
  uint16_t *q = reinterpret_cast<uint16_t *>(base + W.q);
  uint16_t *o = reinterpret_cast<uint16_t *>(base + W.o);
  uint16_t *f = reinterpret_cast<uint16_t *>(base + W.f);
  int32_t *meta = reinterpret_cast<int32_t *>(base + W.meta);
  float *part = reinterpret_cast<float *>(base + W.part);
  const int d = m->d;
  // h = RMSNorm(x) for the first layer; afterwards every residual epilogue
  // writes the next norm (the last one the final norm into `out`). The same
  // launch writes the attention offsets and the commit's row map into meta.
  // normed: the caller's embed_norm_kernel has written x, h and meta
  unsigned launches = 0;
  if (!normed) {
    LAUNCH(rmsnorm_kernel, n, 128, s, x, h, d, m->rms_eps, meta, n, L, row_map_blk);
    launches = 1;
  }
  const unsigned long long dd = static_cast<unsigned long long>(d);
  const unsigned long long ffn = static_cast<unsigned long long>(m->ffn);
  for (int l = 0; l < m->layers; ++l) {
    // each projection warms L2 with the next projection's weights
    const L2Next next_o{m->wo[l], dd * dd * 2};
    const L2Next next_gu{m->wgu[l], 2 * ffn * dd * 2};
    const L2Next next_down{m->wdown[l], dd * ffn * 2};
    const L2Next next_qkv = l + 1 < m->layers ? L2Next{m->wqkv[l + 1], 3 * dd * dd * 2} : L2Next{};
    int sp = gemm_to_partials(h, m->wqkv[l], part, n, 3 * d, d, s, next_o);
    if (!sp) return DLLM_ERR_CUDA;
    LAUNCH(qkv_rope_epilogue_kernel, dim3(n, 3), 256, s, static_cast<const float *>(part), sp, n, m->H, m->dh, pos0,
           log2f(m->rope_base), q, k_cache[l], v_cache[l], pos0);
    const dllm_status st =
        dllm_block_attn(q, k_cache[l], v_cache[l], o, 0, meta, meta + 2, 1, m->H, m->dh, n, L, n, m->max_seq,
                        1.f / sqrtf(static_cast<float>(m->dh)), base + W.attn, W.total - W.attn, s);
    if (st != DLLM_OK) return st;
    sp = gemm_to_partials(o, m->wo[l], part, n, d, d, s, next_gu);
    if (!sp) return DLLM_ERR_CUDA;
    LAUNCH(residual_norm_epilogue_kernel, n, 128, s, static_cast<const float *>(part), sp, n, d, x, h,
           m->rms_eps);
    if (!gemm_auto(h, m->wgu[l], f, n, m->ffn, d, 2, nullptr, part, s, next_down)) return DLLM_ERR_CUDA;
    sp = gemm_to_partials(f, m->wdown[l], part, n, d, m->ffn, s, next_qkv);
    if (!sp) return DLLM_ERR_CUDA;
    uint16_t *next = (l + 1 == m->layers) ? out : h;
    LAUNCH(residual_norm_epilogue_kernel, n, 128, s, static_cast<const float *>(part), sp, n, d, x, next,
           m->rms_eps);
    launches += 7;
  }
  return launch_status(launches);
}

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" dllm_status dllm_gemm_bf16(const dllm_bf16 *A, const dllm_bf16 *W, dllm_bf16 *C, int M, int N, int K,
                                      int epilogue, const dllm_bf16 *aux, dllm_stream stream) {
  if (M < 0 || N < 1 || K < 1 || epilogue < 0 || epilogue > 2) return DLLM_ERR_INVALID_ARG;
  if (K % 64 || N % 16 || M > 65536 || (epilogue == 2 && N % 64)) return DLLM_ERR_UNSUPPORTED;
  if (M == 0) return DLLM_OK;
  if (!A || !W || !C || (epilogue == 1 && !aux)) return DLLM_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(W) || !aligned16(C)) return DLLM_ERR_INVALID_ARG;
  if (!gemm_bf16(A, W, C, M, N, K, epilogue, aux, static_cast<cudaStream_t>(stream))) return DLLM_ERR_CUDA;
  return launch_status(1);
}

extern "C" size_t dllm_model_forward_workspace(const dllm_model *m, int n) {
  if (!model_ok(m) || n < 1) return 0;
  return fwd_layout(m, n).total;
}

extern "C" dllm_status dllm_model_forward(const dllm_model *m, const dllm_bf16 *x_in, int n, int pos0,
                                          dllm_bf16 *const *k_cache, dllm_bf16 *const *v_cache,
                                          dllm_bf16 *hidden_out, void *ws, size_t ws_bytes, dllm_stream stream) {
  if (!model_ok(m)) return DLLM_ERR_INVALID_ARG;
  if (n < 1 || pos0 < 0 || pos0 + n > m->max_seq || !x_in || !hidden_out || !k_cache || !v_cache)
    return DLLM_ERR_INVALID_ARG;
  for (int l = 0; l < m->layers; ++l)
    if (!k_cache[l] || !v_cache[l]) return DLLM_ERR_INVALID_ARG;
  const FwdWs W = fwd_layout(m, n);
  if (!ws || ws_bytes < W.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return DLLM_ERR_WORKSPACE;
  char *base = static_cast<char *>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(base + W.x, x_in, static_cast<size_t>(n) * m->d * 2, cudaMemcpyDeviceToDevice, s) !=
      cudaSuccess)
    return DLLM_ERR_CUDA;
  return forward_rows(m, base, W, n, pos0, pos0 + n, k_cache, v_cache, hidden_out, s);
}

namespace {

struct StepWs {
  FwdWs fwd;
  size_t hid, head, ctl, total;
};

StepWs step_layout(const dllm_model *m, const dllm_decode_state *st) {
  StepWs w{};
  w.fwd = fwd_layout(m, st->T);
  size_t off = w.fwd.total;
  w.hid = off;
  off += align256(static_cast<size_t>(st->T) * m->d * 2);
  w.head = off;
  off += align256(dllm_head_workspace(st->blk, m->d, m->V, st->params.smoothing ? 1 : 0));
  w.ctl = off;  // decode-graph loop counter
  off += 256;
  w.total = off;
  return w;
}

bool state_ok(const dllm_model *m, const dllm_decode_state *st) {
  if (!st || st->T < 1 || st->T > m->max_seq || st->blk < 1 || st->blk > 64 || st->prompt_len < 0 ||
      st->vic < 0 || st->prompt_len + st->blk > st->T)
    return false;
  if (!st->tokens || !st->masked || !st->k_cache || !st->v_cache || !st->bmask || !st->btokens ||
      !st->bcredit || !st->bprev || !st->bnext_emb || !st->n_commit || !st->argmax || !st->conf)
    return false;
  if (st->params.smoothing && !st->pe) return false;
  for (int l = 0; l < m->layers; ++l)
    if (!st->k_cache[l] || !st->v_cache[l]) return false;
  return true;
}

}  // namespace

extern "C" size_t dllm_decode_step_workspace(const dllm_model *m, const dllm_decode_state *st) {
  if (!model_ok(m) || !st || st->T < 1) return 0;
  return step_layout(m, st).total;
}

extern "C" dllm_status dllm_decode_step(const dllm_model *m, const dllm_decode_state *st, int block, int refresh,
                                        void *ws, size_t ws_bytes, dllm_stream stream) {
  if (!model_ok(m) || !state_ok(m, st)) return DLLM_ERR_INVALID_ARG;
  const int b0 = st->prompt_len + block * st->blk;
  if (block < 0 || b0 + st->blk > st->T) return DLLM_ERR_INVALID_ARG;
  const StepWs W = step_layout(m, st);
  if (!ws || ws_bytes < W.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return DLLM_ERR_WORKSPACE;
  char *base = static_cast<char *>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int *status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status_model) != cudaSuccess) return DLLM_ERR_CUDA;

  // rows of this step: every position (refresh) or the window around the block
  const int row0 = refresh ? 0 : (b0 - st->vic > 0 ? b0 - st->vic : 0);
  const int row1 = refresh ? st->T : (b0 + st->blk + st->vic < st->T ? b0 + st->blk + st->vic : st->T);
  const int n = row1 - row0;
  // keys: the cache up to the window end, or the whole sequence when the
  // rows right of the window are kept from the refresh (dual cache)
  const int L = (refresh || st->dual_cache) ? st->T : row1;
  uint16_t *x = reinterpret_cast<uint16_t *>(base + W.fwd.x);
  uint16_t *h0 = reinterpret_cast<uint16_t *>(base + W.fwd.h);
  int32_t *meta0 = reinterpret_cast<int32_t *>(base + W.fwd.meta);
  LAUNCH(embed_norm_kernel, n, 128, s, x, h0, row0, n, st->tokens, st->masked, st->bnext_emb, b0, st->blk,
         refresh ? 0 : 1, m->emb, m->V, st->params.mask_id, m->d, m->rms_eps, meta0, L, st->blk, status);
  dllm_bf16 *hid = reinterpret_cast<dllm_bf16 *>(base + W.hid);
  dllm_status r = forward_rows(m, base, W.fwd, n, row0, L, st->k_cache, st->v_cache, hid, s, st->blk, true);
  if (r != DLLM_OK) return r;
  const dllm_bf16 *hb = hid + static_cast<size_t>(b0 - row0) * m->d;
  if (st->hidden)
    cudaMemcpyAsync(st->hidden, hb, static_cast<size_t>(st->blk) * m->d * 2, cudaMemcpyDeviceToDevice, s);
  r = dllm_head_confidence(hb, m->w_head, m->emb, st->blk, m->d, m->V, st->argmax, st->conf,
                           st->params.smoothing ? st->pe : nullptr, base + W.head, W.total - W.head, stream);
  if (r != DLLM_OK) return r;
  int32_t *meta = reinterpret_cast<int32_t *>(base + W.fwd.meta);   // row map written by forward_rows
  r = dllm_commit(st->argmax, st->conf, st->params.smoothing ? st->pe : nullptr, meta + 4, meta + 4 + 64, st->blk,
                  1, st->blk, st->bmask, st->btokens, st->bcredit, st->bprev, m->emb, m->V, m->d, st->bnext_emb,
                  st->n_commit, &st->params, stream);
  if (r != DLLM_OK) return r;
  LAUNCH(writeback_kernel, 1, 64, s, st->tokens, st->masked, st->btokens, st->bmask, b0, st->blk);
  return launch_status(2);   // embed_norm + writeback (the others count themselves)
}

// ---------------------------------------------------------------------------
// The whole decode loop of one request as one CUDA graph
// ---------------------------------------------------------------------------
namespace dllm {
namespace {

__global__ void reset_block_kernel(const int32_t *tokens, const uint8_t *masked, int b0, int blk, uint8_t *bmask,
                                   int32_t *btok, int32_t *bprev, float *bcredit, int32_t *ctl) {
  const int j = threadIdx.x;
  if (j < blk) {
    bmask[j] = masked[b0 + j];
    btok[j] = tokens[b0 + j];
    bprev[j] = -1;
    bcredit[j] = 0.f;
  }
  if (j == 0) ctl[0] = 0;
}

// Loop condition after a step: some position of the block is still masked,
// and fewer than blk steps ran (each step commits at least one position, so
// the cap is only reached if a step reported an error).
__global__ void while_cond_kernel(cudaGraphConditionalHandle h, const uint8_t *bmask, int blk, int32_t *ctl) {
  const int lane = threadIdx.x;
  const bool m0 = lane < blk && bmask[lane];
  const bool m1 = lane + 32 < blk && bmask[lane + 32];
  const unsigned any = __ballot_sync(0xffffffffu, m0 || m1);
  if (lane == 0) {
    const int it = ++ctl[0];
    cudaGraphSetConditional(h, (any != 0u && it < blk) ? 1u : 0u);
  }
}

// Block condition: no response position before b0 holds a committed EOS.
__global__ void eos_cond_kernel(cudaGraphConditionalHandle h, const int32_t *tokens, const uint8_t *masked, int p0,
                                int p1, int eos) {
  int found = 0;
  if (eos >= 0)
    for (int p = p0 + threadIdx.x; p < p1; p += blockDim.x)
      if (!masked[p] && tokens[p] == eos) found = 1;
  found = __syncthreads_or(found);
  if (threadIdx.x == 0) cudaGraphSetConditional(h, found ? 0u : 1u);
}

// Record what `fn` enqueues on a capture stream as a standalone graph.
template <typename F>
cudaError_t capture(cudaStream_t cs, cudaGraph_t *out, F fn) {
  cudaError_t e = cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed);
  if (e != cudaSuccess) return e;
  const dllm_status st = fn();
  e = cudaStreamEndCapture(cs, out);
  if (st != DLLM_OK && e == cudaSuccess) return cudaErrorUnknown;
  return e;
}

}  // namespace
}  // namespace dllm

struct dllm_decode_graph_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

extern "C" dllm_status dllm_decode_graph_destroy(dllm_decode_graph g) {
  if (!g) return DLLM_ERR_INVALID_ARG;
  if (g->exec) cudaGraphExecDestroy(g->exec);
  if (g->graph) cudaGraphDestroy(g->graph);
  delete g;
  return DLLM_OK;
}

extern "C" dllm_status dllm_decode_graph_create(const dllm_model *m, const dllm_decode_state *st, void *ws,
                                                size_t ws_bytes, dllm_decode_graph *out) {
  if (!out) return DLLM_ERR_INVALID_ARG;
  *out = nullptr;
  if (!model_ok(m) || !state_ok(m, st)) return DLLM_ERR_INVALID_ARG;
  const StepWs W = step_layout(m, st);
  if (!ws || ws_bytes < W.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return DLLM_ERR_WORKSPACE;
  const int nblocks = (st->T - st->prompt_len) / st->blk;
  if (nblocks < 1) return DLLM_ERR_INVALID_ARG;
  int32_t *ctl = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + W.ctl);
  cudaStream_t cs = nullptr;
  if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return DLLM_ERR_CUDA;
  dllm_decode_graph g = new dllm_decode_graph_s();
  bool ok = cudaGraphCreate(&g->graph, 0) == cudaSuccess;
  cudaGraphNode_t prev = nullptr;
  for (int b = 0; ok && b < nblocks; ++b) {
    const int b0 = st->prompt_len + b * st->blk;
    cudaGraphConditionalHandle hi = 0, hw = 0;
    cudaGraph_t seg = nullptr;
    cudaGraphNode_t e_node = nullptr, if_node = nullptr, c_node = nullptr, w_node = nullptr, b_node = nullptr;
    ok = cudaGraphConditionalHandleCreate(&hi, g->graph, 0, 0) == cudaSuccess;
    // eos check -> IF handle
    ok = ok && capture(cs, &seg, [&] {
      eos_cond_kernel<<<1, 256, 0, cs>>>(hi, st->tokens, st->masked, st->prompt_len, b0, st->eos_id);
      return launch_status(1);
    }) == cudaSuccess;
    ok = ok && cudaGraphAddChildGraphNode(&e_node, g->graph, prev ? &prev : nullptr, prev ? 1 : 0, seg) ==
                   cudaSuccess;
    if (seg) cudaGraphDestroy(seg), seg = nullptr;
    cudaGraphNodeParams ip = {};
    ip.type = cudaGraphNodeTypeConditional;
    ip.conditional.handle = hi;
    ip.conditional.type = cudaGraphCondTypeIf;
    ip.conditional.size = 1;
    ok = ok && cudaGraphAddNode(&if_node, g->graph, &e_node, nullptr, 1, &ip) == cudaSuccess;
    if (!ok) break;
    cudaGraph_t body_if = ip.conditional.phGraph_out[0];
    ok = cudaGraphConditionalHandleCreate(&hw, body_if, 0, 0) == cudaSuccess;
    // block reset + refresh step + loop condition
    ok = ok && capture(cs, &seg, [&] {
      reset_block_kernel<<<1, 64, 0, cs>>>(st->tokens, st->masked, b0, st->blk, st->bmask, st->btokens, st->bprev,
                                           st->bcredit, ctl);
      const dllm_status r = dllm_decode_step(m, st, b, 1, ws, ws_bytes, cs);
      if (r != DLLM_OK) return r;
      while_cond_kernel<<<1, 32, 0, cs>>>(hw, st->bmask, st->blk, ctl);
      return launch_status(2);
    }) == cudaSuccess;
    ok = ok && cudaGraphAddChildGraphNode(&c_node, body_if, nullptr, 0, seg) == cudaSuccess;
    if (seg) cudaGraphDestroy(seg), seg = nullptr;
    cudaGraphNodeParams wp = {};
    wp.type = cudaGraphNodeTypeConditional;
    wp.conditional.handle = hw;
    wp.conditional.type = cudaGraphCondTypeWhile;
    wp.conditional.size = 1;
    ok = ok && cudaGraphAddNode(&w_node, body_if, &c_node, nullptr, 1, &wp) == cudaSuccess;
    if (!ok) break;
    cudaGraph_t body_w = wp.conditional.phGraph_out[0];
    // window step + loop condition
    ok = capture(cs, &seg, [&] {
      const dllm_status r = dllm_decode_step(m, st, b, 0, ws, ws_bytes, cs);
      if (r != DLLM_OK) return r;
      while_cond_kernel<<<1, 32, 0, cs>>>(hw, st->bmask, st->blk, ctl);
      return launch_status(1);
    }) == cudaSuccess;
    ok = ok && cudaGraphAddChildGraphNode(&b_node, body_w, nullptr, 0, seg) == cudaSuccess;
    if (seg) cudaGraphDestroy(seg), seg = nullptr;
    prev = if_node;
  }
  ok = ok && cudaGraphInstantiate(&g->exec, g->graph, 0) == cudaSuccess;
  cudaStreamDestroy(cs);
  if (!ok) {
    cudaGetLastError();
    dllm_decode_graph_destroy(g);
    return DLLM_ERR_CUDA;
  }
  *out = g;
  return DLLM_OK;
}

extern "C" dllm_status dllm_decode_graph_launch(dllm_decode_graph g, dllm_stream stream) {
  if (!g || !g->exec) return DLLM_ERR_INVALID_ARG;
  return cudaGraphLaunch(g->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? DLLM_OK : DLLM_ERR_CUDA;
}
