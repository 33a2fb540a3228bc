// Mixture-of-experts SwiGLU FFN with top-k routing (the MoE block of the
// LLaDA-MoE family that dInfer serves -- dInfer abstract; MoE dLLMs --
// TIDE abstract):
//
//   router   logits z = h . W_r^T; per token the top-k experts by logit
//            (ties: lower index), weights softmax(z) over the chosen
//   scan     expert-sorted order of the n*k (token, rank) assignments:
//            segment offsets per expert, each assignment's row in it
//   gather   Xp[row] = h[token of row]
//   GEMM 1   per expert e, rows of its segment: A1 = silu(Xp W1_e^T) * (Xp W3_e^T)
//   GEMM 2   per expert e: Y = A1 W2_e^T (fp32)
//   combine  out[t] = sum_j w[t][j] * Y[row of (t, j)]
//
// The two grouped GEMMs are persistent tcgen05 kernels (TMA-fed, TMEM
// accumulators) whose work units are (expert, 128-row tile of the expert's
// weight, block of BN of the expert's tokens); every CTA derives the unit
// list from the segment offsets the scan kernel wrote, so the host never
// reads the routing. Decode-sized batches give each expert a handful of
// tokens, so the GEMMs stream every touched expert's weights once: they are
// HBM-bound on the expert weights.

#include <cfloat>
#include <climits>

#include "common.cuh"
#include "umma_gemm.cuh"

namespace dllm {

DLLM_DEFINE_STATUS(moe)

namespace {

constexpr int kMaxE = 256;
constexpr int kMaxTopk = 16;
constexpr int kMaxAssign = 1 << 16;

// ---------------------------------------------------------------------------
// router logits: one CTA per (8 tokens, 16 experts), one warp per pair of
// experts; each lane keeps 2 x 8 accumulators over its 8-element column
// slices. All ten 16-byte loads of a slice (two weight rows, eight token
// rows; ragged edges clamped to the last valid row) are issued before any
// is used, so a warp keeps ten or more loads in flight instead of one.
// ---------------------------------------------------------------------------
constexpr int kRouterTok = 8;
constexpr int kRouterExpPerWarp = 2;
constexpr int kRouterExpPerCta = 8 * kRouterExpPerWarp;

__global__ void __launch_bounds__(256) moe_logits_kernel(const uint16_t *__restrict__ h,
                                                         const uint16_t *__restrict__ wr, int n, int d, int E,
                                                         float *__restrict__ z) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = blockIdx.y * kRouterExpPerCta + warp * kRouterExpPerWarp;
  const int t0 = blockIdx.x * kRouterTok;
  if (e0 >= E) return;
  const uint16_t *wrow[kRouterExpPerWarp];
#pragma unroll
  for (int i = 0; i < kRouterExpPerWarp; ++i) wrow[i] = wr + static_cast<size_t>(min(e0 + i, E - 1)) * d;
  const uint16_t *hrow[kRouterTok];
#pragma unroll
  for (int j = 0; j < kRouterTok; ++j) hrow[j] = h + static_cast<size_t>(min(t0 + j, n - 1)) * d;
  float acc[kRouterExpPerWarp][kRouterTok];
#pragma unroll
  for (int i = 0; i < kRouterExpPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < kRouterTok; ++j) acc[i][j] = 0.f;
#pragma unroll 2
  for (int c = lane * 8; c < d; c += 256) {
    uint4 wv[kRouterExpPerWarp], hv[kRouterTok];
#pragma unroll
    for (int i = 0; i < kRouterExpPerWarp; ++i) wv[i] = *reinterpret_cast<const uint4 *>(wrow[i] + c);
#pragma unroll
    for (int j = 0; j < kRouterTok; ++j) hv[j] = *reinterpret_cast<const uint4 *>(hrow[j] + c);
#pragma unroll
    for (int i = 0; i < kRouterExpPerWarp; ++i) {
      float f[8];
      unpack8(wv[i], f);
#pragma unroll
      for (int j = 0; j < kRouterTok; ++j) {
        float x[8];
        unpack8(hv[j], x);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[i][j] = fmaf(f[q], x[q], acc[i][j]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kRouterExpPerWarp; ++i)
#pragma unroll
    for (int j = 0; j < kRouterTok; ++j) {
      const float v = warp_sum(acc[i][j]);
      if (lane == 0 && e0 + i < E && t0 + j < n) z[static_cast<size_t>(t0 + j) * E + e0 + i] = v;
    }
}

// ---------------------------------------------------------------------------
// top-k: one warp per token, 8 tokens per CTA: k rounds of a warp arg-max
// over the E logits (ties: lower index); weights exp(z - z_max) over the
// chosen, normalised
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) moe_topk_kernel(const float *__restrict__ z, int n, int E, int topk,
                                                       int32_t *__restrict__ ids, float *__restrict__ wts) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= n) return;
  float v[kMaxE / 32];
  bool taken[kMaxE / 32];
#pragma unroll
  for (int i = 0; i < kMaxE / 32; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? z[static_cast<size_t>(t) * E + e] : -FLT_MAX;
    taken[i] = e >= E;
  }
  float zmax = 0.f, den = 0.f, my_ez = 0.f;
  int my_id = 0;
  for (int j = 0; j < topk; ++j) {
    float bv = -FLT_MAX;
    int be = INT_MAX;
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i) {
      const int e = lane + 32 * i;
      if (!taken[i] && (v[i] > bv || (v[i] == bv && e < be))) {
        bv = v[i];
        be = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oe = __shfl_xor_sync(0xffffffffu, be, o);
      if (ov > bv || (ov == bv && oe < be)) {
        bv = ov;
        be = oe;
      }
    }
#pragma unroll
    for (int i = 0; i < kMaxE / 32; ++i)
      if (lane + 32 * i == be) taken[i] = true;
    if (j == 0) zmax = bv;
    const float ez = expf(bv - zmax);
    den += ez;
    if (lane == j) {
      my_id = be;
      my_ez = ez;
    }
  }
  if (lane < topk) {
    ids[static_cast<size_t>(t) * topk + lane] = my_id;
    wts[static_cast<size_t>(t) * topk + lane] = my_ez / den;
  }
}

// ---------------------------------------------------------------------------
// expert-sorted order: one CTA, a counting sort by expert. Pass 1 counts the
// assignments a = t*k + j per expert (shared-memory atomics), one warp turns
// the counts into segment offsets, pass 2 gives each assignment the next free
// row of its segment. The order inside a segment is the order in which the
// atomics land: no result depends on it, since every row of a grouped GEMM
// output is a function of that row's input alone and the combine sums a
// token's k rows in rank order. Each thread holds up to kScanBatch ids in
// registers, so both passes cost one read of the ids when A <= 8192.
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 1024;
constexpr int kScanBatch = 8;

__global__ void __launch_bounds__(kScanThreads) moe_scan_kernel(const int32_t *__restrict__ ids, int A, int topk,
                                                                int E, int32_t *__restrict__ offsets,
                                                                int32_t *__restrict__ perm_tok,
                                                                int32_t *__restrict__ pos_of) {
  pdl_trigger();
  pdl_wait();
  __shared__ int cnt[kMaxE];
  __shared__ int seg[kMaxE + 1];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += kScanThreads) cnt[e] = 0;
  __syncthreads();
  int ev[kScanBatch];
  auto load_batch = [&](int b0) {
#pragma unroll
    for (int i = 0; i < kScanBatch; ++i) {
      const int a = b0 + i * kScanThreads + static_cast<int>(threadIdx.x);
      const int e = a < A ? ids[a] : -1;
      ev[i] = e >= 0 && e < E ? e : -1;
    }
  };
  constexpr int kBatchSpan = kScanBatch * kScanThreads;
  for (int b0 = 0; b0 < A; b0 += kBatchSpan) {
    load_batch(b0);
#pragma unroll
    for (int i = 0; i < kScanBatch; ++i)
      if (ev[i] >= 0) atomicAdd(&cnt[ev[i]], 1);
  }
  __syncthreads();
  if (warp == 0) {   // exclusive scan of the counts
    int running = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      const int v = e < E ? cnt[e] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < E) {
        seg[e] = running + incl - v;
        cnt[e] = running + incl - v;   // next free row of the segment
      }
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) seg[E] = running;
  }
  __syncthreads();
  for (int e = threadIdx.x; e <= E; e += kScanThreads) offsets[e] = seg[e];
  for (int b0 = 0; b0 < A; b0 += kBatchSpan) {
    if (A > kBatchSpan) load_batch(b0);
#pragma unroll
    for (int i = 0; i < kScanBatch; ++i) {
      if (ev[i] < 0) continue;
      const int a = b0 + i * kScanThreads + static_cast<int>(threadIdx.x);
      const int p = atomicAdd(&cnt[ev[i]], 1);
      perm_tok[p] = a / topk;
      pos_of[a] = p;
    }
  }
}

__global__ void __launch_bounds__(128) moe_gather_kernel(const uint16_t *__restrict__ h,
                                                         const int32_t *__restrict__ perm_tok, int d,
                                                         uint16_t *__restrict__ xp) {
  pdl_wait();
  pdl_trigger();   // after the wait: the first grouped GEMM reads the scan's offsets before its own wait
  const int p = blockIdx.x;
  const uint4 *src = reinterpret_cast<const uint4 *>(h + static_cast<size_t>(perm_tok[p]) * d);
  uint4 *dst = reinterpret_cast<uint4 *>(xp + static_cast<size_t>(p) * d);
  for (int i = threadIdx.x; i < d / 8; i += blockDim.x) dst[i] = src[i];
}

__global__ void __launch_bounds__(256) moe_combine_kernel(const float *__restrict__ yp,
                                                          const int32_t *__restrict__ pos_of,
                                                          const float *__restrict__ wts, int d, int topk, int A,
                                                          void *__restrict__ out, int out_fp32) {
  pdl_trigger();
  pdl_wait();
  __shared__ int pos[kMaxTopk];
  __shared__ float w[kMaxTopk];
  const int t = blockIdx.x;
  if (threadIdx.x < topk) {
    // rows come from the scan of this call's own routing; the clamp only
    // keeps a corrupted index inside the buffer
    pos[threadIdx.x] = min(max(pos_of[static_cast<size_t>(t) * topk + threadIdx.x], 0), A - 1);
    w[threadIdx.x] = wts[static_cast<size_t>(t) * topk + threadIdx.x];
  }
  __syncthreads();
  for (int c = threadIdx.x * 4; c < d; c += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < topk; ++j) {
      const float4 y = *reinterpret_cast<const float4 *>(yp + static_cast<size_t>(pos[j]) * d + c);
      acc.x = fmaf(w[j], y.x, acc.x);
      acc.y = fmaf(w[j], y.y, acc.y);
      acc.z = fmaf(w[j], y.z, acc.z);
      acc.w = fmaf(w[j], y.w, acc.w);
    }
    const size_t o = static_cast<size_t>(t) * d + c;
    if (out_fp32) {
      *reinterpret_cast<float4 *>(static_cast<float *>(out) + o) = acc;
    } else {
      uint16_t *ob = static_cast<uint16_t *>(out) + o;
      const uint32_t lo = static_cast<uint32_t>(f32_to_bf16(acc.x)) | (static_cast<uint32_t>(f32_to_bf16(acc.y)) << 16);
      const uint32_t hi = static_cast<uint32_t>(f32_to_bf16(acc.z)) | (static_cast<uint32_t>(f32_to_bf16(acc.w)) << 16);
      *reinterpret_cast<uint2 *>(ob) = make_uint2(lo, hi);
    }
  }
}

// ---------------------------------------------------------------------------
// grouped GEMM over the experts' token segments
//
//   D[m][n] = sum_k A_e[m][k] * Xs[seg_e + n][k]
//
// A_e = rows [e * a_rows_per_e, +M_e) of the stacked expert weights (K-major),
// Xs = the expert-sorted activations (K-major). Same warp roles as the head's
// GEMM: warp 0 TMA producer, warp 1 TMEM owner + MMA issuer, warps 2..5
// epilogue. Work unit u of expert e covers (m tile, token block) with the
// token block varying fastest, so an expert's weight tile is read once and
// its reuse by the expert's other token blocks hits L2.
// ---------------------------------------------------------------------------
enum : int { kGrpSwiGLU = 0, kGrpStoreF32 = 1 };

struct GroupedArgs {
  const int32_t *offsets;  // [E + 1] segment starts of the expert-sorted rows
  int E;
  int rows;                // rows of Xs and of the output
  int m_tiles;             // per expert: output features / 128
  int a_rows_per_e;        // rows of A per expert (2F for W13, d for W2)
  int a1_row;              // SwiGLU: offset of the up rows inside an expert
  int k_steps;             // K / 64
  int stages;
  int ld;                  // output row stride (elements)
  void *out;               // bf16 (SwiGLU) or float
  unsigned int *status;
};

constexpr int kGrpMetaBytes = 2 * (kMaxE + 1) * 4 + 64;

template <int BN, int EPI>
constexpr int grp_stage_bytes() {
  return (EPI == kGrpSwiGLU ? 2 : 1) * kATileBytes + BN * 128;
}

struct GrpUnit {
  int e, mt, row0, valid;
};

template <int BN>
__device__ __forceinline__ GrpUnit grp_unit(const int *uprefix, const int *seg, int E, int u) {
  int lo = 0, hi = E - 1;  // the last expert whose first unit is <= u
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (uprefix[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  const int local = u - uprefix[lo];
  const int cnt = seg[lo + 1] - seg[lo];
  const int nblk = (cnt + BN - 1) / BN;
  const int nb = local % nblk;
  return GrpUnit{lo, local / nblk, seg[lo] + nb * BN, min(BN, cnt - nb * BN)};
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kUmmaThreads, 1)
moe_grouped_gemm_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                        const GroupedArgs args) {
  constexpr bool kDual = EPI == kGrpSwiGLU;
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 128, "N tile");
  constexpr int kNumA = kDual ? 2 : 1;
  constexpr int kStage = grp_stage_bytes<BN, EPI>();
  constexpr int kBOff = kNumA * kATileBytes;
  constexpr int kAccCols = kNumA * BN;
  constexpr int kBuffers = 2 * kAccCols <= 512 ? 2 : 1;
  constexpr int kC0 = kBuffers * kAccCols;
  constexpr uint32_t kCols = (kC0 <= 32) ? 32 : (kC0 <= 64) ? 64 : (kC0 <= 128) ? 128 : (kC0 <= 256) ? 256 : 512;
  constexpr uint32_t kIdesc = idesc_bf16(128, BN, 0, 0);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = args.stages;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * kStage);
  uint64_t *empty = full + S;
  uint64_t *tfull = empty + S;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *seg = reinterpret_cast<int *>(smem + static_cast<size_t>(S) * kStage + 256);
  int *uprefix = seg + kMaxE + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = args.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Segment offsets of the routing, clamped to [0, rows] and made monotone
  // so that no unit can address rows outside the buffers. They are read
  // before this grid's dependency wait: the scan that wrote them completed
  // before this grid could launch, because every kernel between the two
  // (the gather; for the second GEMM also the first) signals its dependents
  // only after its own wait has returned. (L2 loads: no stale L1 line.)
  for (int i = threadIdx.x; i <= E; i += blockDim.x) seg[i] = min(max(__ldcg(args.offsets + i), 0), args.rows);
  __syncthreads();
  if (threadIdx.x == 0) {
    uprefix[0] = 0;
    for (int e = 0; e < E; ++e) {
      if (seg[e + 1] < seg[e]) seg[e + 1] = seg[e];
      uprefix[e + 1] = uprefix[e] + args.m_tiles * ((seg[e + 1] - seg[e] + BN - 1) / BN);
    }
  }
  __syncthreads();
  const int units = uprefix[E];

  // The expert weights (A) depend on no earlier kernel: the producer fills the
  // A tiles of the first S stages (fresh stages: no wait for a free slot)
  // while the previous kernel is still finishing, and adds their B tiles (the
  // activations an earlier kernel wrote) once the dependency wait returns.
  const uint64_t pol = policy_evict_first();  // expert weights stream through once
  int pre = 0;
  if (warp == 0 && lane == 0) {
    int u = blockIdx.x, ks = 0;
    while (pre < S && u < units) {
      const GrpUnit g = grp_unit<BN>(uprefix, seg, E, u);
      const int arow = g.e * args.a_rows_per_e + g.mt * 128;
      mbar_arrive_expect_tx(&full[pre], kStage);
      uint8_t *dst = smem + static_cast<size_t>(pre) * kStage;
      tma_load_2d_hint(dst, &tma_a, &full[pre], ks * 64, arow, pol);
      if (kDual) tma_load_2d_hint(dst + kATileBytes, &tma_a, &full[pre], ks * 64, arow + args.a1_row, pol);
      ++pre;
      if (++ks == args.k_steps) {
        ks = 0;
        u += gridDim.x;
      }
    }
  }
  pdl_wait();
  pdl_trigger();   // after the wait: the next grouped GEMM reads the offsets before its own

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0, it = 0;
      uint32_t phase = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        const GrpUnit g = grp_unit<BN>(uprefix, seg, E, u);
        const int arow = g.e * args.a_rows_per_e + g.mt * 128;
        for (int ks = 0; ks < args.k_steps; ++ks, ++it) {
          uint8_t *dst = smem + static_cast<size_t>(stage) * kStage;
          if (it >= pre) {   // stage `it` < pre (phase 0) already holds its A tiles
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) goto producer_done;
            mbar_arrive_expect_tx(&full[stage], kStage);
            tma_load_2d_hint(dst, &tma_a, &full[stage], ks * 64, arow, pol);
            if (kDual) tma_load_2d_hint(dst + kATileBytes, &tma_a, &full[stage], ks * 64, arow + args.a1_row, pol);
          }
          tma_load_2d(dst + kBOff, &tma_b, &full[stage], ks * 64, g.row0);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag)) goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        for (int ks = 0; ks < args.k_steps; ++ks) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) goto mma_done;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + static_cast<size_t>(stage) * kStage);
          const uint32_t b_addr = a_addr + kBOff;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = sw128_desc(b_addr + kk * 32, 16, 1024);
#pragma unroll
            for (int k = 0; k < kNumA; ++k)
              umma_bf16(d_tmem + k * BN, sw128_desc(a_addr + k * kATileBytes + kk * 32, 16, 1024), bdesc, kIdesc,
                        (ks > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&empty[stage]);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        umma_commit(&tfull[acc]);
        if (kBuffers == 2) {
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1;
        } else {
          acc_phase ^= 1;
        }
      }
    mma_done:;
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const GrpUnit g = grp_unit<BN>(uprefix, seg, E, u);
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int m = g.mt * 128 + row;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * kAccCols);
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 16) {
        uint32_t r[16];
        float v[16], gt[16];
        tmem_ld16(taddr + c0, r);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
        if constexpr (kDual) {
#pragma unroll
          for (int j = 0; j < 16; ++j) gt[j] = v[j];
          tmem_ld16(taddr + BN + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c0 + j < g.valid) {
            const size_t o = static_cast<size_t>(g.row0 + c0 + j) * args.ld + m;
            if constexpr (kDual) {
              const float x = gt[j] / (1.f + __expf(-gt[j])) * v[j];   // silu(gate) * up
              static_cast<uint16_t *>(args.out)[o] = f32_to_bf16(x);
            } else {
              static_cast<float *>(args.out)[o] = v[j];
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (kBuffers == 2) {
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      } else {
        acc_phase ^= 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kCols);
  }
  if (threadIdx.x == 0 && *abort_flag && args.status) atomicOr(args.status, DLLM_DEV_WAIT_TIMEOUT);
}

template <int BN, int EPI>
bool launch_grouped(const CUtensorMap &ta, const CUtensorMap &tb, GroupedArgs a, int max_units, cudaStream_t s) {
  constexpr int kStage = grp_stage_bytes<BN, EPI>();
  int stages = (220 * 1024 - 1024 - 256 - kGrpMetaBytes) / kStage;
  if (stages > 12) stages = 12;
  if (stages < 2) return false;
  a.stages = stages;
  const size_t smem = 1024 + static_cast<size_t>(kStage) * stages + 256 + kGrpMetaBytes;
  auto kern = moe_grouped_gemm_kernel<BN, EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return false;
  const int grid = max_units < num_sms() ? max_units : num_sms();
  return launch_pdl(kern, dim3(grid > 0 ? grid : 1), dim3(kUmmaThreads), smem, s, ta, tb, a) == cudaSuccess;
}

template <int EPI>
bool launch_grouped_bn(int BN, const CUtensorMap &ta, const CUtensorMap &tb, const GroupedArgs &a, int max_units,
                       cudaStream_t s) {
  switch (BN) {
    case 16: return launch_grouped<16, EPI>(ta, tb, a, max_units, s);
    case 32: return launch_grouped<32, EPI>(ta, tb, a, max_units, s);
    case 64: return launch_grouped<64, EPI>(ta, tb, a, max_units, s);
    default: return launch_grouped<128, EPI>(ta, tb, a, max_units, s);
  }
}

// token-block size from the mean tokens per expert (any size is correct;
// this only sets the waste on the last block of each expert)
int moe_bn(int A, int E) {
  const int avg = (A + E - 1) / E;
  return avg <= 16 ? 16 : avg <= 32 ? 32 : avg <= 64 ? 64 : 128;
}

struct MoeWs {
  size_t offsets, z, perm, pos, ids, wts, xp, a1, yp, total;
};

MoeWs moe_layout(int n, int d, int E, int F, int topk) {
  const size_t A = static_cast<size_t>(n) * topk;
  MoeWs w{};
  size_t off = 0;
  w.offsets = off; off += align256((E + 1) * 4);
  w.z = off;       off += align256(static_cast<size_t>(n) * E * 4);
  w.perm = off;    off += align256(A * 4);
  w.pos = off;     off += align256(A * 4);
  w.ids = off;     off += align256(A * 4);
  w.wts = off;     off += align256(A * 4);
  w.xp = off;      off += align256(A * d * 2);
  w.a1 = off;      off += align256(A * F * 2);
  w.yp = off;      off += align256(A * d * 4);
  w.total = off;
  return w;
}

bool moe_args_ok(int n, int d, int E, int F, int topk) {
  return n >= 0 && d >= 128 && d % 128 == 0 && d <= 8192 && F >= 128 && F % 128 == 0 && E >= 1 && E <= kMaxE &&
         topk >= 1 && topk <= kMaxTopk && topk <= E && static_cast<long long>(n) * topk <= kMaxAssign &&
         static_cast<long long>(E) * 2 * F < INT_MAX && static_cast<long long>(E) * d < INT_MAX;
}

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" size_t dllm_moe_ffn_workspace(int n, int d, int E, int F, int topk) {
  if (!moe_args_ok(n, d, E, F, topk)) return 0;
  return moe_layout(n, d, E, F, topk).total;
}

extern "C" dllm_status dllm_moe_ffn(const dllm_bf16 *h, const dllm_bf16 *w_router, const dllm_bf16 *w13,
                                    const dllm_bf16 *w2, int n, int d, int E, int F, int topk, void *out,
                                    int out_fp32, int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes,
                                    dllm_stream stream) {
  if (!moe_args_ok(n, d, E, F, topk)) return DLLM_ERR_UNSUPPORTED;
  if (n == 0) return DLLM_OK;
  if (!h || !w_router || !w13 || !w2 || !out) return DLLM_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(w_router) || !aligned16(w13) || !aligned16(w2) || !aligned16(out))
    return DLLM_ERR_INVALID_ARG;
  const MoeWs W = moe_layout(n, d, E, F, topk);
  if (!ws || ws_bytes < W.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return DLLM_ERR_WORKSPACE;
  char *base = static_cast<char *>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int *status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status_moe) != cudaSuccess) return DLLM_ERR_CUDA;
  const int A = n * topk;
  int32_t *offsets = reinterpret_cast<int32_t *>(base + W.offsets);
  int32_t *perm = reinterpret_cast<int32_t *>(base + W.perm);
  int32_t *pos = reinterpret_cast<int32_t *>(base + W.pos);
  int32_t *ids = topk_ids ? topk_ids : reinterpret_cast<int32_t *>(base + W.ids);
  float *wts = topk_w ? topk_w : reinterpret_cast<float *>(base + W.wts);
  uint16_t *xp = reinterpret_cast<uint16_t *>(base + W.xp);
  uint16_t *a1 = reinterpret_cast<uint16_t *>(base + W.a1);
  float *yp = reinterpret_cast<float *>(base + W.yp);
  const int BN = moe_bn(A, E);

  CUtensorMap ta1, tb1, ta2, tb2;
  if (!make_tmap_bf16_sw128(&ta1, w13, static_cast<uint64_t>(E) * 2 * F, d, d, 128) ||
      !make_tmap_bf16_sw128(&tb1, xp, A, d, d, BN) ||
      !make_tmap_bf16_sw128(&ta2, w2, static_cast<uint64_t>(E) * d, F, F, 128) ||
      !make_tmap_bf16_sw128(&tb2, a1, A, F, F, BN))
    return DLLM_ERR_CUDA;

  const uint16_t *hb = reinterpret_cast<const uint16_t *>(h);
  float *z = reinterpret_cast<float *>(base + W.z);
  const int groups = (n + kRouterTok - 1) / kRouterTok;
  const dim3 router_grid(groups, (E + kRouterExpPerCta - 1) / kRouterExpPerCta);
  if (launch_pdl(moe_logits_kernel, router_grid, dim3(256), 0, s, hb, reinterpret_cast<const uint16_t *>(w_router),
                 n, d, E, z) != cudaSuccess)
    return DLLM_ERR_CUDA;
  if (launch_pdl(moe_topk_kernel, dim3(groups), dim3(256), 0, s, static_cast<const float *>(z), n, E, topk, ids,
                 wts) != cudaSuccess)
    return DLLM_ERR_CUDA;
  if (launch_pdl(moe_scan_kernel, dim3(1), dim3(kScanThreads), 0, s, static_cast<const int32_t *>(ids), A, topk, E, offsets,
                 perm, pos) != cudaSuccess)
    return DLLM_ERR_CUDA;
  if (launch_pdl(moe_gather_kernel, dim3(A), dim3(128), 0, s, hb, static_cast<const int32_t *>(perm), d, xp) !=
      cudaSuccess)
    return DLLM_ERR_CUDA;
  const int blocks = (A + BN - 1) / BN + E;   // bound on the token blocks over all experts
  GroupedArgs g1{offsets, E, A, F / 128, 2 * F, F, d / 64, 0, F, a1, status};
  if (!launch_grouped_bn<kGrpSwiGLU>(BN, ta1, tb1, g1, (F / 128) * blocks, s)) return DLLM_ERR_CUDA;
  GroupedArgs g2{offsets, E, A, d / 128, d, 0, F / 64, 0, d, yp, status};
  if (!launch_grouped_bn<kGrpStoreF32>(BN, ta2, tb2, g2, (d / 128) * blocks, s)) return DLLM_ERR_CUDA;
  if (launch_pdl(moe_combine_kernel, dim3(n), dim3(256), 0, s, static_cast<const float *>(yp),
                 static_cast<const int32_t *>(pos), static_cast<const float *>(wts), d, topk, A, out, out_fp32) !=
      cudaSuccess)
    return DLLM_ERR_CUDA;
  return launch_status(7);
}
