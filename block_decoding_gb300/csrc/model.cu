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

namespace {

// ---------------------------------------------------------------------------
// small ops
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(128)
embed_rows_kernel(uint16_t *__restrict__ x, int row0, int n, const int32_t *__restrict__ tokens,
                  const uint8_t *__restrict__ masked, const uint16_t *__restrict__ block_emb, int b0, int blk,
                  int use_block, const uint16_t *__restrict__ emb, int V, int mask_id, int d,
                  unsigned int *status) {
  const int t = blockIdx.x;
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
  uint4 *d4 = reinterpret_cast<uint4 *>(x + static_cast<size_t>(t) * d);
  for (int c = threadIdx.x; c < d / 8; c += blockDim.x) d4[c] = s4[c];
}

// y = x / sqrt(mean(x^2) + eps), one row per CTA, fp32 arithmetic.
__global__ void __launch_bounds__(128)
rmsnorm_kernel(const uint16_t *__restrict__ x, uint16_t *__restrict__ y, int d, float eps) {
  const int r = blockIdx.x;
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

// RoPE (rotate-half pairs (i, i + dh/2), angle pos * base^(-2i/dh)) on the q
// and k parts of qkv [n][3d]; q -> q_out [n][d]; k, v -> cache rows
// kv_row0 + t of [T][d].
__global__ void __launch_bounds__(256)
rope_qkv_kernel(const uint16_t *__restrict__ qkv, int pos0, int H, int dh, float log2_base,
                uint16_t *__restrict__ q_out, uint16_t *__restrict__ kc, uint16_t *__restrict__ vc, int kv_row0) {
  const int t = blockIdx.x;
  const int d = H * dh, half = dh / 2;
  const float pos = static_cast<float>(pos0 + t);
  const uint16_t *row = qkv + static_cast<size_t>(t) * 3 * d;
  uint16_t *qo = q_out + static_cast<size_t>(t) * d;
  uint16_t *ko = kc + static_cast<size_t>(kv_row0 + t) * d;
  uint16_t *vo = vc + static_cast<size_t>(kv_row0 + t) * d;
  for (int idx = threadIdx.x; idx < H * half; idx += blockDim.x) {
    const int h = idx / half, i = idx - h * half;
    const float inv_freq = exp2f(-(2.f * i / dh) * log2_base);
    float sn, cs;
    sincosf(pos * inv_freq, &sn, &cs);
    const int a = h * dh + i, b = a + half;
    const float q1 = bf16_to_f32(row[a]), q2 = bf16_to_f32(row[b]);
    const float k1 = bf16_to_f32(row[d + a]), k2 = bf16_to_f32(row[d + b]);
    qo[a] = f32_to_bf16(q1 * cs - q2 * sn);
    qo[b] = f32_to_bf16(q2 * cs + q1 * sn);
    ko[a] = f32_to_bf16(k1 * cs - k2 * sn);
    ko[b] = f32_to_bf16(k2 * cs + k1 * sn);
    vo[a] = row[2 * d + a];
    vo[b] = row[2 * d + b];
  }
}

// Offsets of a one-request attention call and the identity head-row map.
__global__ void step_meta_kernel(int32_t *meta, int n, int L, int blk) {
  const int j = threadIdx.x;
  if (j == 0) { meta[0] = 0; meta[1] = n; meta[2] = 0; meta[3] = L; }
  if (j < blk) { meta[4 + j] = 0; meta[4 + 64 + j] = j; }
}

__global__ void writeback_kernel(int32_t *tokens, uint8_t *masked, const int32_t *btok, const uint8_t *bmask,
                                 int b0, int blk) {
  const int j = threadIdx.x;
  if (j < blk) {
    tokens[b0 + j] = btok[j];
    masked[b0 + j] = bmask[j];
  }
}

// ---------------------------------------------------------------------------
// GEMM: C[tokens][features] = X[tokens][K] . W[features][K]^T (swap-AB)
// ---------------------------------------------------------------------------
template <int BN, int EPI>
bool gemm_t(const uint16_t *X, const uint16_t *W, uint16_t *C, int M, int N, int K, int w_rows,
            const uint16_t *aux, int a1_row, cudaStream_t s) {
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
  return launch_umma_gemm<BN, false, EPI>(ta, tb, a, s);
}

// epilogue: 0 none, 1 residual (C = X W^T + aux), 2 SwiGLU (W = [2N][K]: gate rows then up rows)
bool gemm_bf16(const uint16_t *X, const uint16_t *W, uint16_t *C, int M, int N, int K, int epilogue,
               const uint16_t *aux, cudaStream_t s) {
  if (epilogue == 2) {
    if (M <= 16) return gemm_t<16, kEpiSwiGLU>(X, W, C, M, N, K, 2 * N, nullptr, N, s);
    if (M <= 32) return gemm_t<32, kEpiSwiGLU>(X, W, C, M, N, K, 2 * N, nullptr, N, s);
    if (M <= 64) return gemm_t<64, kEpiSwiGLU>(X, W, C, M, N, K, 2 * N, nullptr, N, s);
    return gemm_t<128, kEpiSwiGLU>(X, W, C, M, N, K, 2 * N, nullptr, N, s);
  }
  const uint16_t *ax = epilogue == 1 ? aux : nullptr;
  if (M <= 16) return gemm_t<16, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s);
  if (M <= 32) return gemm_t<32, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s);
  if (M <= 64) return gemm_t<64, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s);
  if (M <= 128) return gemm_t<128, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s);
  return gemm_t<256, kEpiBf16T>(X, W, C, M, N, K, N, ax, 0, s);
}

bool model_ok(const dllm_model *m) {
  if (!m || m->layers < 1 || m->d < 64 || m->H < 1 || (m->dh != 64 && m->dh != 128) || m->H * m->dh != m->d)
    return false;
  if (m->d % 64 || m->ffn % 64 || m->ffn < 64 || m->V < 2 || !m->emb || !m->w_head) return false;
  if (!m->wqkv || !m->wo || !m->wgu || !m->wdown) return false;
  for (int l = 0; l < m->layers; ++l)
    if (!m->wqkv[l] || !m->wo[l] || !m->wgu[l] || !m->wdown[l]) return false;
  return true;
}

struct FwdWs {
  size_t x, h, qkv, q, o, f, meta, attn, total;
};

FwdWs fwd_layout(const dllm_model *m, int n) {
  FwdWs w{};
  size_t off = 0;
  auto take = [&](size_t b) { const size_t o = off; off += align256(b); return o; };
  const size_t rd = static_cast<size_t>(n) * m->d * 2;
  w.x = take(rd);
  w.h = take(rd);
  w.qkv = take(3 * rd);
  w.q = take(rd);
  w.o = take(rd);
  w.f = take(static_cast<size_t>(n) * m->ffn * 2);
  w.meta = take(4 * 140);
  w.attn = off;
  off += align256(dllm_block_attn_workspace(1, m->H, m->dh, n, m->max_seq));
  w.total = off;
  return w;
}

// All layers over n rows already in ws.x (positions pos0..), keys = cache
// rows [0, L); writes the final-normed rows to out.
dllm_status forward_rows(const dllm_model *m, char *base, const FwdWs &W, int n, int pos0, int L,
                         dllm_bf16 *const *k_cache, dllm_bf16 *const *v_cache, dllm_bf16 *out, cudaStream_t s) {
  uint16_t *x = reinterpret_cast<uint16_t *>(base + W.x);
  uint16_t *h = reinterpret_cast<uint16_t *>(base + W.h);
  uint16_t *qkv = reinterpret_cast<uint16_t *>(base + W.qkv);
  uint16_t *q = reinterpret_cast<uint16_t *>(base + W.q);
  uint16_t *o = reinterpret_cast<uint16_t *>(base + W.o);
  uint16_t *f = reinterpret_cast<uint16_t *>(base + W.f);
  int32_t *meta = reinterpret_cast<int32_t *>(base + W.meta);
  const int d = m->d;
  step_meta_kernel<<<1, 64, 0, s>>>(meta, n, L, 0);
  unsigned launches = 1;
  for (int l = 0; l < m->layers; ++l) {
    rmsnorm_kernel<<<n, 128, 0, s>>>(x, h, d, m->rms_eps);
    if (!gemm_bf16(h, m->wqkv[l], qkv, n, 3 * d, d, 0, nullptr, s)) return DLLM_ERR_CUDA;
    rope_qkv_kernel<<<n, 256, 0, s>>>(qkv, pos0, m->H, m->dh, log2f(m->rope_base), q, k_cache[l], v_cache[l],
                                      pos0);
    launches += 3;
    const dllm_status st =
        dllm_block_attn(q, k_cache[l], v_cache[l], o, 0, meta, meta + 2, 1, m->H, m->dh, n, L, n, m->max_seq,
                        1.f / sqrtf(static_cast<float>(m->dh)), base + W.attn, W.total - W.attn, s);
    if (st != DLLM_OK) return st;
    if (!gemm_bf16(o, m->wo[l], x, n, d, d, 1, x, s)) return DLLM_ERR_CUDA;
    rmsnorm_kernel<<<n, 128, 0, s>>>(x, h, d, m->rms_eps);
    if (!gemm_bf16(h, m->wgu[l], f, n, m->ffn, d, 2, nullptr, s)) return DLLM_ERR_CUDA;
    if (!gemm_bf16(f, m->wdown[l], x, n, d, m->ffn, 1, x, s)) return DLLM_ERR_CUDA;
    launches += 4;
  }
  rmsnorm_kernel<<<n, 128, 0, s>>>(x, out, d, m->rms_eps);
  return launch_status(launches + 1);
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
  uint16_t *x = reinterpret_cast<uint16_t *>(base + W.fwd.x);
  embed_rows_kernel<<<n, 128, 0, s>>>(x, row0, n, st->tokens, st->masked, st->bnext_emb, b0, st->blk,
                                      refresh ? 0 : 1, m->emb, m->V, st->params.mask_id, m->d, status);
  dllm_bf16 *hid = reinterpret_cast<dllm_bf16 *>(base + W.hid);
  dllm_status r = forward_rows(m, base, W.fwd, n, row0, row1, st->k_cache, st->v_cache, hid, s);
  if (r != DLLM_OK) return r;
  const dllm_bf16 *hb = hid + static_cast<size_t>(b0 - row0) * m->d;
  if (st->hidden)
    cudaMemcpyAsync(st->hidden, hb, static_cast<size_t>(st->blk) * m->d * 2, cudaMemcpyDeviceToDevice, s);
  r = dllm_head_confidence(hb, m->w_head, m->emb, st->blk, m->d, m->V, st->argmax, st->conf,
                           st->params.smoothing ? st->pe : nullptr, base + W.head, W.total - W.head, stream);
  if (r != DLLM_OK) return r;
  int32_t *meta = reinterpret_cast<int32_t *>(base + W.fwd.meta);
  step_meta_kernel<<<1, 64, 0, s>>>(meta, n, row1, st->blk);
  r = dllm_commit(st->argmax, st->conf, st->params.smoothing ? st->pe : nullptr, meta + 4, meta + 4 + 64, st->blk,
                  1, st->blk, st->bmask, st->btokens, st->bcredit, st->bprev, m->emb, m->V, m->d, st->bnext_emb,
                  st->n_commit, &st->params, stream);
  if (r != DLLM_OK) return r;
  writeback_kernel<<<1, 64, 0, s>>>(st->tokens, st->masked, st->btokens, st->bmask, b0, st->blk);
  return launch_status(3);
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
