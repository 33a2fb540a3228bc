// K3: the parallel-decode commit of one denoise step.
//
// dInfer article, "the art of decoding": threshold parallel decoding, credit
// decoding (credit accumulates while a position's prediction is stable and
// lets it commit below the confidence threshold) and hierarchical decoding
// (recursive bisection, centre of each sub-region first); "iteration
// smoothing" gives the still-masked positions E[mask] + alpha * P.E as their
// next input. One launch: one CTA per block position, each taking its
// request's decision (one thread per position, the selection on 64-bit
// position masks) and writing its position's next-step embedding row.
#include <atomic>

#include "common.cuh"

namespace dllm {

DLLM_DEFINE_STATUS(commit)

namespace {

constexpr int kMaxBlk = 64;
constexpr int kThreads = 128;   // per CTA: threads 0..blk-1 decide their positions, all write the row
constexpr int kMaxB = 4096;
constexpr int kSlots = 32;      // arrival-count slots, one per call in turn

// Arrival counts of the CTAs of each request, per slot: zero at load, and
// zero again after every call (the last CTA of a request resets its count).
// Calls in flight at the same time take different slots as long as fewer
// than kSlots are in flight; a captured call keeps its slot at every replay.
__device__ unsigned int g_arrive[kSlots][kMaxB];

struct Span {
  int8_t l, r, k;
};

// Bits [lo, hi) of a 64-bit position mask (0 <= lo <= hi <= 64).
__device__ __forceinline__ uint64_t bits_between(int lo, int hi) {
  const uint64_t upto_hi = hi >= 64 ? ~0ull : ((1ull << hi) - 1ull);
  const uint64_t upto_lo = lo >= 64 ? ~0ull : ((1ull << lo) - 1ull);
  return upto_hi & ~upto_lo;
}

// One CTA per (block position jr, request i). Every CTA of request i takes
// the request's whole decision from the state as it was on entry (all of
// them read the same values and compute the same result), then writes
// next_emb of position jr. The state is written by the request's last CTA
// to finish its reads (an arrival count per request), so that no CTA reads
// a position's state after it changed; nothing waits on another CTA.
//
// Every global read of the decision is issued in one round: the position's
// state, and for every head row its request, position, argmax and
// confidence (the head outputs of rows of other requests are read and
// dropped, so that no read waits on the row map). Behind them, the rows a
// still-masked position jr usually needs (E[mask_id], and the P.E of head
// row i * blk + jr) are read speculatively; a committed position or another
// head row takes a second round. The selection works on 64-bit
// position masks in one thread.
__global__ void __launch_bounds__(kThreads)
commit_kernel(const int32_t *__restrict__ argmax, const float *__restrict__ conf, const float *__restrict__ pe,
              const int32_t *__restrict__ row_req, const int32_t *__restrict__ row_pos, int R, int B, int blk,
              uint8_t *__restrict__ mask, int32_t *__restrict__ tokens, float *__restrict__ credit,
              int32_t *__restrict__ prev, const uint16_t *__restrict__ emb, int V, int d,
              uint16_t *__restrict__ next_emb, int32_t *__restrict__ n_commit, unsigned int *__restrict__ arrive,
              dllm_params prm) {
  pdl_trigger();
  pdl_wait();
  const int jr = blockIdx.x, i = blockIdx.y;
  const int j = threadIdx.x;   // block position decided by this thread (j < blk)
  const bool pos = j < blk;
  const size_t g = static_cast<size_t>(i) * blk + j;

  __shared__ int row_of[kMaxBlk];
  __shared__ int s_bad, s_last;
  __shared__ uint8_t s_m[kMaxBlk];
  __shared__ float s_p[kMaxBlk];
  __shared__ int s_arg[kMaxBlk];
  __shared__ float s_conf[kMaxBlk];
  __shared__ int s_tok[kMaxBlk];
  __shared__ uint32_t s_ballot[2][2];   // [warp]: masked, candidate
  __shared__ uint64_t s_sel;
  __shared__ Span stack[2 * kMaxBlk + 4];

  // one round of decision reads: this position's state, and the head rows
  uint8_t m8 = 0;
  float c0 = 0.f;
  int32_t pv = -1, tk = 0;
  if (pos) {
    m8 = mask[g];
    c0 = credit[g];
    pv = prev[g];
    tk = tokens[g];
    row_of[j] = -1;
  }
  if (j == 0) s_bad = 0;
  constexpr int kRowBatch = 2;   // rows per thread whose reads are in flight together
  int rq[kRowBatch], rp[kRowBatch], ra[kRowBatch];
  float rc[kRowBatch];
  int r0 = 0;
  auto load_rows = [&](int base) {
#pragma unroll
    for (int u = 0; u < kRowBatch; ++u) {
      const int r = base + u * kThreads + j;
      rq[u] = -1;
      if (r < R) {
        rq[u] = row_req[r];
        rp[u] = row_pos[r];
        ra[u] = argmax[r];
        rc[u] = conf[r];
      }
    }
  };
  load_rows(0);
  // then, behind them, the speculative row reads for position jr
  const int d8 = d >> 3;
  const uint4 *E = reinterpret_cast<const uint4 *>(emb);
  constexpr int kPer = 4;   // uint4 (8 values) per thread: d <= 8 * kPer * kThreads
  const bool spec = d8 <= kPer * kThreads;
  const int guess = i * blk + jr;
  uint4 e_spec[kPer];
  float4 p_spec[2 * kPer];
  if (spec) {
    const uint4 *em = E + static_cast<size_t>(prm.mask_id) * d8;
    const float4 *pg = (prm.smoothing && guess < R) ? reinterpret_cast<const float4 *>(pe + static_cast<size_t>(guess) * d)
                                                    : nullptr;
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int c = j + u * kThreads;
      if (c < d8) {
        e_spec[u] = em[c];
        if (pg) {
          p_spec[2 * u] = pg[2 * c];
          p_spec[2 * u + 1] = pg[2 * c + 1];
        }
      }
    }
  }

  if (pos) {
    s_m[j] = m8 != 0;
    s_tok[j] = tk;
  }
  __syncthreads();
  const bool masked = pos && m8 != 0;
  // claim each masked position's row; its head outputs go with it
  for (;;) {
#pragma unroll
    for (int u = 0; u < kRowBatch; ++u) {
      const int r = r0 + u * kThreads + j;
      if (r >= R) continue;
      const int ri = rq[u], rj = rp[u];
      if (ri < 0 || ri >= B) { atomicOr(&s_bad, DLLM_DEV_ROW_RANGE); continue; }
      if (ri != i) continue;
      if (rj < 0 || rj >= blk) { atomicOr(&s_bad, DLLM_DEV_ROW_RANGE); continue; }
      if (!s_m[rj]) continue;   // rows of committed positions are ignored
      if (atomicCAS(&row_of[rj], -1, r) != -1) {
        atomicOr(&s_bad, DLLM_DEV_ROW_DUPLICATE);
      } else {
        s_arg[rj] = ra[u];
        s_conf[rj] = rc[u];
      }
    }
    r0 += kRowBatch * kThreads;
    if (r0 >= R) break;
    load_rows(r0);
  }
  __syncthreads();

  // credit and candidacy (float32: a product, then a sum)
  int a = 0;
  float p = 0.f, cr = 0.f;
  bool cand = false;
  if (masked) {
    const int r = row_of[j];
    if (r < 0) {
      atomicOr(&s_bad, DLLM_DEV_ROW_MISSING);
    } else {
      a = s_arg[j];
      p = s_conf[j];
      if (a < 0 || a >= V) atomicOr(&s_bad, DLLM_DEV_ID_RANGE);
      cr = (pv == a) ? __fadd_rn(__fmul_rn(prm.lambda_, c0), p) : p;
      cand = (p >= prm.tau) || (cr >= prm.kappa);
    }
    s_p[j] = p;
  } else if (pos && (tk < 0 || tk >= V)) {
    atomicOr(&s_bad, DLLM_DEV_ID_RANGE);
  }
  const uint32_t bm = __ballot_sync(0xffffffffu, masked), bc = __ballot_sync(0xffffffffu, cand);
  if ((j & 31) == 0 && j < kMaxBlk) {
    s_ballot[j >> 5][0] = bm;
    s_ballot[j >> 5][1] = bc;
  }
  __syncthreads();
  const int bad = s_bad;

  // 3-4. selection
  if (j == 0 && !bad) {
    const uint64_t M = static_cast<uint64_t>(s_ballot[0][0]) | (static_cast<uint64_t>(s_ballot[1][0]) << 32);
    const uint64_t C = static_cast<uint64_t>(s_ballot[0][1]) | (static_cast<uint64_t>(s_ballot[1][1]) << 32);
    uint64_t sel = 0;
    if (prm.hierarchical) {
      // every maximal run of masked positions is a region; in a span [l, r)
      // the candidate nearest the centre c = l + (r - l - 1) / 2 is taken
      // (at equal distance the one with the larger p, else the lower index),
      // then both sides recurse with one level less
      const int8_t k0 = static_cast<int8_t>(prm.hier_levels > 100 ? 100 : prm.hier_levels);
      uint64_t rest = M;
      while (rest) {
        const int l0 = __ffsll(static_cast<long long>(rest)) - 1;
        const uint64_t above = ~rest & ~bits_between(0, l0);   // unmasked positions past l0
        const int re = above ? __ffsll(static_cast<long long>(above)) - 1 : 64;
        rest &= ~bits_between(l0, re);
        const int r1 = re < blk ? re : blk;
        int top = 0;
        stack[top++] = Span{static_cast<int8_t>(l0), static_cast<int8_t>(r1), k0};
        while (top > 0) {
          const Span sp = stack[--top];
          if (sp.k <= 0 || sp.r <= sp.l) continue;
          const int c = sp.l + (sp.r - sp.l - 1) / 2;
          const uint64_t right = C & bits_between(c, sp.r), left = C & bits_between(sp.l, c);
          if (!right && !left) continue;
          const int br = right ? __ffsll(static_cast<long long>(right)) - 1 : -1;
          const int bl = left ? 63 - __clzll(static_cast<long long>(left)) : -1;
          int best;
          if (bl < 0) best = br;
          else if (br < 0) best = bl;
          else if (c - bl < br - c) best = bl;
          else if (br - c < c - bl) best = br;
          else best = s_p[br] > s_p[bl] ? br : bl;
          sel |= 1ull << best;
          stack[top++] = Span{sp.l, static_cast<int8_t>(best), static_cast<int8_t>(sp.k - 1)};
          stack[top++] = Span{static_cast<int8_t>(best + 1), sp.r, static_cast<int8_t>(sp.k - 1)};
        }
      }
    } else {
      sel = C;
    }
    if (sel == 0 && M) {
      // nothing passed: the masked position with the largest p (lowest index on ties)
      int best = -1;
      float bp = 0.f;
      for (uint64_t t = M; t; t &= t - 1) {
        const int q = __ffsll(static_cast<long long>(t)) - 1;
        if (best < 0 || s_p[q] > bp) { best = q; bp = s_p[q]; }
      }
      sel = 1ull << best;
    }
    s_sel = sel;
  }
  if (j == 0 && bad) s_sel = 0;   // the request is left unchanged
  __syncthreads();

  // this CTA's row: next_emb of position jr. Committed (now or before):
  // E[token]; still masked: E[mask_id] (+ alpha * P.E of its head row)
  {
    const bool was_masked = s_m[jr] != 0;
    const bool now = was_masked && ((s_sel >> jr) & 1ull);
    int src = !was_masked ? s_tok[jr] : (now ? s_arg[jr] : prm.mask_id);
    if (src < 0 || src >= V) src = prm.mask_id;   // reported above
    const int prow = was_masked && !now && prm.smoothing ? row_of[jr] : -1;
    uint4 *out = reinterpret_cast<uint4 *>(next_emb) + (static_cast<size_t>(i) * blk + jr) * d8;
    const float4 *P = prow >= 0 ? reinterpret_cast<const float4 *>(pe + static_cast<size_t>(prow) * d) : nullptr;
    auto emit = [&](int c, uint4 e, const float4 *pp) {
      if (!pp) {
        out[c] = e;
        return;
      }
      float f[8];
      unpack8(e, f);
      const float4 x = pp[0], y = pp[1];
      f[0] = fmaf(prm.alpha, x.x, f[0]); f[1] = fmaf(prm.alpha, x.y, f[1]);
      f[2] = fmaf(prm.alpha, x.z, f[2]); f[3] = fmaf(prm.alpha, x.w, f[3]);
      f[4] = fmaf(prm.alpha, y.x, f[4]); f[5] = fmaf(prm.alpha, y.y, f[5]);
      f[6] = fmaf(prm.alpha, y.z, f[6]); f[7] = fmaf(prm.alpha, y.w, f[7]);
      out[c] = pack8(f);
    };
    if (spec && src == prm.mask_id && (!P || prow == guess)) {
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int c = j + u * kThreads;
        if (c < d8) emit(c, e_spec[u], P ? &p_spec[2 * u] : nullptr);
      }
    } else {
      const uint4 *in = E + static_cast<size_t>(src) * d8;
      for (int c = j; c < d8; c += kThreads) emit(c, in[c], P ? &P[2 * c] : nullptr);
    }
  }

  // arrival: this CTA's reads of the state are complete (their values were
  // used above); the request's last CTA writes the state
  if (j == 0) {
    const unsigned int old = atomicAdd(&arrive[i], 1u);
    s_last = old + 1u == gridDim.x;
    if (s_last) atomicExch(&arrive[i], 0u);
  }
  __syncthreads();
  if (!s_last) return;
  if (bad) {
    if (j == 0) {
      atomicOr(&g_status_commit, static_cast<unsigned>(bad));
      n_commit[i] = 0;
    }
    return;
  }
  if (j == 0) n_commit[i] = __popcll(s_sel);
  // 5. state writes
  if (masked) {
    if ((s_sel >> j) & 1ull) {
      tokens[g] = a;
      mask[g] = 0;
      credit[g] = 0.f;
      prev[g] = -1;
    } else {
      credit[g] = cr;
      prev[g] = a;
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
  if (blk > kMaxBlk || B > kMaxB || d % 8 != 0) return DLLM_ERR_UNSUPPORTED;
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
  unsigned int *arrive = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&arrive), g_arrive) != cudaSuccess) return DLLM_ERR_CUDA;
  static std::atomic<unsigned int> next_slot{0};
  arrive += static_cast<size_t>(next_slot.fetch_add(1u, std::memory_order_relaxed) % kSlots) * kMaxB;
  const uint16_t *e16 = emb;
  if (launch_pdl(commit_kernel, dim3(blk, B), dim3(kThreads), 0, s, argmax, conf, pe, row_req, row_pos, R, B, blk,
                 mask, tokens, credit, prev_argmax, e16, V, d, next_emb, n_commit, arrive, p) != cudaSuccess)
    return DLLM_ERR_CUDA;
  return launch_status(1);
}
