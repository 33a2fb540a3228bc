// K3: the parallel-decode commit of one denoise step.
//
// dInfer article, "the art of decoding": threshold parallel decoding, credit
// decoding (credit accumulates while a position's prediction is stable and
// lets it commit below the confidence threshold) and hierarchical decoding
// (recursive bisection, centre of each sub-region first); "iteration
// smoothing" gives the still-masked positions E[mask] + alpha * P.E as their
// next input. One CTA per request: the decision over <= 64 positions is a
// few hundred instructions. The next-step embedding rows (the bytes) are
// written by a second kernel with one CTA per block position.
#include "common.cuh"

namespace dllm {

DLLM_DEFINE_STATUS(commit)

namespace {

constexpr int kMaxBlk = 64;
constexpr int kThreads = 128;     // decision kernel
constexpr int kRowThreads = 128;  // row writer

struct Span {
  int8_t l, r, k;
};

__global__ void __launch_bounds__(kThreads)
commit_kernel(const int32_t *__restrict__ argmax, const float *__restrict__ conf,
              const float *__restrict__ pe, const int32_t *__restrict__ row_req,
              const int32_t *__restrict__ row_pos, int R, int B, int blk,
              uint8_t *__restrict__ mask, int32_t *__restrict__ tokens,
              float *__restrict__ credit, int32_t *__restrict__ prev,
              const uint16_t *__restrict__ emb, int V, int d,
              uint16_t *__restrict__ next_emb, int32_t *__restrict__ n_commit,
              dllm_params prm) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x;
  const int tid = threadIdx.x;

  __shared__ int row_of[kMaxBlk];
  __shared__ int s_bad;
  __shared__ float s_p[kMaxBlk];
  __shared__ float s_cr[kMaxBlk];
  __shared__ int s_a[kMaxBlk];
  __shared__ uint8_t s_masked[kMaxBlk];
  __shared__ uint8_t s_cand[kMaxBlk];
  __shared__ uint8_t s_sel[kMaxBlk];
  __shared__ Span stack[2 * kMaxBlk + 4];

  if (tid < blk) {
    row_of[tid] = -1;
    s_masked[tid] = mask[i * blk + tid] != 0;
    s_cand[tid] = 0;
    s_sel[tid] = 0;
  }
  if (tid == 0) s_bad = 0;
  __syncthreads();

  // Inverse row map of this request.
  for (int r = tid; r < R; r += blockDim.x) {
    const int ri = row_req[r];
    if (ri < 0 || ri >= B) { atomicOr(&s_bad, DLLM_DEV_ROW_RANGE); continue; }
    if (ri != i) continue;
    const int j = row_pos[r];
    if (j < 0 || j >= blk) { atomicOr(&s_bad, DLLM_DEV_ROW_RANGE); continue; }
    if (!s_masked[j]) continue;
    if (atomicCAS(&row_of[j], -1, r) != -1) atomicOr(&s_bad, DLLM_DEV_ROW_DUPLICATE);
  }
  __syncthreads();

  // 1-2. credit update and candidates (float32: a product, then a sum).
  if (tid < blk) {
    const int j = tid;
    if (s_masked[j]) {
      const int r = row_of[j];
      if (r < 0) {
        atomicOr(&s_bad, DLLM_DEV_ROW_MISSING);
      } else {
        const int a = argmax[r];
        const float p = conf[r];
        if (a < 0 || a >= V) atomicOr(&s_bad, DLLM_DEV_ID_RANGE);
        const float c0 = credit[i * blk + j];
        const float cr = (prev[i * blk + j] == a) ? __fadd_rn(__fmul_rn(prm.lambda_, c0), p) : p;
        s_p[j] = p;
        s_cr[j] = cr;
        s_a[j] = a;
        s_cand[j] = (p >= prm.tau) || (cr >= prm.kappa);
      }
    } else {
      const int t = tokens[i * blk + j];
      if (t < 0 || t >= V) atomicOr(&s_bad, DLLM_DEV_ID_RANGE);
    }
  }
  __syncthreads();
  if (s_bad) {
    // leave the request untouched; report on the status word
    if (tid == 0) {
      atomicOr(&g_status_commit, static_cast<unsigned>(s_bad));
      n_commit[i] = 0;
    }
    return;
  }

  // 3-4. selection (one thread: <= 64 positions, explicit stack)
  if (tid == 0) {
    int n = 0;
    if (prm.hierarchical) {
      int j = 0;
      while (j < blk) {
        if (!s_masked[j]) { ++j; continue; }
        const int l0 = j;
        while (j < blk && s_masked[j]) ++j;
        int top = 0;
        stack[top++] = Span{static_cast<int8_t>(l0), static_cast<int8_t>(j),
                            static_cast<int8_t>(prm.hier_levels > 100 ? 100 : prm.hier_levels)};
        while (top > 0) {
          const Span sp = stack[--top];
          if (sp.k <= 0 || sp.r <= sp.l) continue;
          const int c = sp.l + (sp.r - sp.l - 1) / 2;
          int best = -1, bd = 0;
          float bp = 0.f;
          for (int s = sp.l; s < sp.r; ++s) {
            if (!s_cand[s]) continue;
            const int ds = s > c ? s - c : c - s;
            if (best < 0 || ds < bd || (ds == bd && s_p[s] > bp)) { best = s; bd = ds; bp = s_p[s]; }
          }
          if (best < 0) continue;
          s_sel[best] = 1;
          ++n;
          stack[top++] = Span{sp.l, static_cast<int8_t>(best), static_cast<int8_t>(sp.k - 1)};
          stack[top++] = Span{static_cast<int8_t>(best + 1), sp.r, static_cast<int8_t>(sp.k - 1)};
        }
      }
    } else {
      for (int j = 0; j < blk; ++j)
        if (s_masked[j] && s_cand[j]) { s_sel[j] = 1; ++n; }
    }
    if (n == 0) {
      int best = -1;
      float bp = 0.f;
      for (int j = 0; j < blk; ++j)
        if (s_masked[j] && (best < 0 || s_p[j] > bp)) { best = j; bp = s_p[j]; }
      if (best >= 0) { s_sel[best] = 1; n = 1; }
    }
    n_commit[i] = n;
  }
  __syncthreads();

  // 5. state writes
  if (tid < blk) {
    const int j = tid;
    if (s_masked[j]) {
      if (s_sel[j]) {
        tokens[i * blk + j] = s_a[j];
        mask[i * blk + j] = 0;
        credit[i * blk + j] = 0.f;
        prev[i * blk + j] = -1;
      } else {
        credit[i * blk + j] = s_cr[j];
        prev[i * blk + j] = s_a[j];
      }
    }
  }
}

// Next-step input embedding of block position j of request i, derived from
// the state the decision kernel left: a committed position (mask 0) gets
// E[token]; a position still masked gets E[mask_id] (+ alpha * P.E of its
// head row when smoothing). One CTA per (position, request), so the rows of
// a block are copied by many SMs at once.
__global__ void __launch_bounds__(kRowThreads)
commit_rows_kernel(const float *__restrict__ pe, const int32_t *__restrict__ row_req,
                   const int32_t *__restrict__ row_pos, int R, int blk, const uint8_t *__restrict__ mask,
                   const int32_t *__restrict__ tokens, const uint16_t *__restrict__ emb, int V, int d,
                   uint16_t *__restrict__ next_emb, dllm_params prm) {
  pdl_trigger();
  pdl_wait();
  const int j = blockIdx.x, i = blockIdx.y;
  __shared__ int s_row;
  const bool masked = mask[i * blk + j] != 0;
  if (threadIdx.x == 0) s_row = 0x7fffffff;
  __syncthreads();
  if (masked && prm.smoothing)
    for (int r = threadIdx.x; r < R; r += blockDim.x)
      if (row_req[r] == i && row_pos[r] == j) atomicMin(&s_row, r);
  __syncthreads();
  const int d8 = d >> 3;
  const uint4 *E = reinterpret_cast<const uint4 *>(emb);
  uint4 *out = reinterpret_cast<uint4 *>(next_emb) + (static_cast<size_t>(i) * blk + j) * d8;
  int src = masked ? prm.mask_id : tokens[i * blk + j];
  if (src < 0 || src >= V) {
    if (threadIdx.x == 0) atomicOr(&g_status_commit, DLLM_DEV_ID_RANGE);
    src = prm.mask_id;
  }
  const uint4 *in = E + static_cast<size_t>(src) * d8;
  const bool smooth = masked && prm.smoothing && s_row != 0x7fffffff;
  const float4 *P = smooth ? reinterpret_cast<const float4 *>(pe + static_cast<size_t>(s_row) * d) : nullptr;
  for (int c = threadIdx.x; c < d8; c += blockDim.x) {
    if (!smooth) {
      out[c] = in[c];
    } else {
      float f[8];
      unpack8(in[c], f);
      const float4 a = P[2 * c], b = P[2 * c + 1];
      f[0] = fmaf(prm.alpha, a.x, f[0]); f[1] = fmaf(prm.alpha, a.y, f[1]);
      f[2] = fmaf(prm.alpha, a.z, f[2]); f[3] = fmaf(prm.alpha, a.w, f[3]);
      f[4] = fmaf(prm.alpha, b.x, f[4]); f[5] = fmaf(prm.alpha, b.y, f[5]);
      f[6] = fmaf(prm.alpha, b.z, f[6]); f[7] = fmaf(prm.alpha, b.w, f[7]);
      out[c] = pack8(f);
    }
  }
}

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" dllm_status dllm_commit(const int32_t *argmax, const float *conf,
                                   const float *pe, const int32_t *row_req,
                                   const int32_t *row_pos, int R, int B, int blk,
                                   uint8_t *mask, int32_t *tokens, float *credit,
                                   int32_t *prev_argmax, const dllm_bf16 *emb,
                                   int V, int d, dllm_bf16 *next_emb,
                                   int32_t *n_commit, const dllm_params *params,
                                   dllm_stream stream) {
  if (!params) return DLLM_ERR_INVALID_ARG;
  if (B < 0 || R < 0 || blk < 1 || V < 1 || d < 8) return DLLM_ERR_INVALID_ARG;
  if (blk > kMaxBlk || B > 4096 || d % 8 != 0) return DLLM_ERR_UNSUPPORTED;
  if (B == 0) return DLLM_OK;
  if (!mask || !tokens || !credit || !prev_argmax || !emb || !next_emb || !n_commit)
    return DLLM_ERR_INVALID_ARG;
  if (R > 0 && (!argmax || !conf || !row_req || !row_pos)) return DLLM_ERR_INVALID_ARG;
  const dllm_params p = *params;
  if (p.mask_id < 0 || p.mask_id >= V) return DLLM_ERR_INVALID_ARG;
  if (p.hierarchical && p.hier_levels < 1) return DLLM_ERR_INVALID_ARG;
  if (p.smoothing && R > 0 && (!pe || !aligned16(pe))) return DLLM_ERR_INVALID_ARG;
  if (!aligned16(emb) || !aligned16(next_emb)) return DLLM_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint16_t *e16 = emb;
  if (launch_pdl(commit_kernel, dim3(B), dim3(kThreads), 0, s, argmax, conf, pe, row_req, row_pos, R, B, blk,
                 mask, tokens, credit, prev_argmax, e16, V, d, next_emb, n_commit, p) != cudaSuccess)
    return DLLM_ERR_CUDA;
  if (launch_pdl(commit_rows_kernel, dim3(blk, B), dim3(kRowThreads), 0, s, pe, row_req, row_pos, R, blk,
                 static_cast<const uint8_t *>(mask), static_cast<const int32_t *>(tokens), e16, V, d, next_emb,
                 p) != cudaSuccess)
    return DLLM_ERR_CUDA;
  return launch_status(2);
}
