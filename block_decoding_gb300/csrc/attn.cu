// K1: non-causal attention of the window queries over cached prefix + fresh
// window K/V (dInfer article, "vicinity KV refresh": only the block and its
// neighbourhood are recomputed each iteration, the distant cache is reused;
// Sangam abstract: attention is bidirectional, so no causal mask).
//
// One CTA per (request, head, 128-query tile, key split). K and V arrive in
// tiles of 128 keys; TMEM holds three S buffers of 128 keys, so the scores of
// the next tiles are ready while the softmax works on one.
// Warp roles (224 threads):
//   warp 0      TMA: the query tile once, then K and V tiles (a ring each;
//               a K stage is free once the S that read it is done, a V stage
//               once its P.V is)
//   warp 1      S MMAs (one lane): S(j) = Q K_j^T into buffer j mod 3 once
//               P(j - 3) V is done
//   warps 2..5  softmax: one thread per query row (its TMEM lane) holds the
//               tile's 128 scores, so the row max needs no exchange;
//               P = exp2(S*c - m) against a reference max m that moves only
//               when the row max passes it by more than 2^8 (O is then
//               rescaled in TMEM, after the previous P.V); P goes back to TMEM
//               as bf16 pairs over S(j)
//   warp 6      P.V MMAs (one lane): O += P(j) V_j, P read from TMEM, once
//               P(j) is written
// The S and P.V MMAs are issued by two threads: one thread's issue, waits
// and commits were the step's critical path, and each tracks completion of
// its own MMAs through its own commits.
// TMEM (512 columns): S/P buffer b at 128 b, O at 384. With one key split the
// CTA writes O/l; otherwise (m, l, O) partials go to the workspace and
// attn_combine merges them.
#include "umma.cuh"

namespace dllm {

DLLM_DEFINE_STATUS(attn)

namespace {

constexpr int kAttnThreads = 32 * 7;    // TMA warp, S-MMA warp, softmax warpgroup, P.V-MMA warp
constexpr int kBox = 128 * 64 * 2;      // 16 KB: 128 rows x 64 bf16 (one swizzled TMA box)
constexpr int kSBuf = 3;                // S / P buffers in TMEM
constexpr uint32_t kColO = 384;         // TMEM column of O

static_assert(kSBuf == 3, "the stage / buffer barriers below assume three buffers");

template <int DH>
struct AttnSmem {
  static constexpr int kT = (DH / 64) * kBox;        // one tile of 128 rows (Q, K or V)
  // K and V ring stages: stage st of tile j is the buffer of tile j, so the
  // barrier that frees a stage is that buffer's s_full (K) / pv_done (V)
  static constexpr int kKSt = kSBuf;
  static constexpr int kVSt = kSBuf;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kT;
  static constexpr int kOffV = kOffK + kKSt * kT;
  static constexpr int kOffBar = kOffV + kVSt * kT;
  static constexpr int kBytes = kOffBar + 256;
};

struct AttnArgs {
  const int32_t *q_off, *kv_off;
  int H, q_tiles, kv_splits, tiles_per_split, max_q, max_kv, q_rows, kv_rows;
  float scale_log2;
  void *out;
  int out_fp32;
  float *part_o, *part_ml;
  unsigned int *status;
};

// Row ranges of request i, clipped to the buffers (an offset outside them
// sets DLLM_DEV_OFFSETS and is clipped, never dereferenced).
__device__ __forceinline__ void request_extent(const AttnArgs &a, int i, int &q0, int &W, int &k0, int &L,
                                               bool report) {
  q0 = a.q_off[i];
  W = a.q_off[i + 1] - q0;
  k0 = a.kv_off[i];
  L = a.kv_off[i + 1] - k0;
  bool bad = false;
  if (q0 < 0 || W < 0 || q0 > a.q_rows) { bad = true; q0 = 0; W = 0; }
  if (q0 + W > a.q_rows) { bad = true; W = a.q_rows - q0; }
  if (k0 < 0 || L < 0 || k0 > a.kv_rows) { bad = true; k0 = 0; L = 0; }
  if (k0 + L > a.kv_rows) { bad = true; L = a.kv_rows - k0; }
  // the host bounds size the grid and the split partials: never go past them
  if (W > a.max_q) { bad = true; W = a.max_q; }
  if (L > a.max_kv) { bad = true; L = a.max_kv; }
  if (bad && report && a.status) atomicOr(a.status, DLLM_DEV_OFFSETS);
}

// n values of a row (o[0..n)) times `inv` to the output (bf16 or fp32).
__device__ __forceinline__ void store_cols(void *out, int out_fp32, size_t base, const float *o, int n, float inv) {
  if (out_fp32) {
    float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(out) + base);
    for (int c = 0; c < n; c += 4) p[c / 4] = make_float4(o[c] * inv, o[c + 1] * inv, o[c + 2] * inv, o[c + 3] * inv);
  } else {
    uint4 *p = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + base);
    for (int c = 0; c < n; c += 8) {
      float f[8];
      for (int e = 0; e < 8; ++e) f[e] = o[c + e] * inv;
      p[c / 8] = pack8(f);
    }
  }
}

// Split partial row index of (key split sp, request i, query row lr, head h).
__device__ __forceinline__ size_t partial_row(const AttnArgs &a, int sp, int i, int lr, int h) {
  return (static_cast<size_t>(sp) * gridDim.z * a.max_q + static_cast<size_t>(i) * a.max_q + lr) * a.H + h;
}

template <int DH>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_umma_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const AttnArgs args) {
  using Lay = AttnSmem<DH>;
  constexpr int kKSt = Lay::kKSt, kVSt = Lay::kVSt;
  constexpr uint32_t kIdescS = idesc_bf16(128, 128, 0, 0);
  constexpr uint32_t kIdescO = idesc_bf16(128, DH, 0, 1);

  pdl_trigger();
  pdl_wait();   // offsets and Q/K/V may come from the previous kernel
  const int i = blockIdx.z, h = blockIdx.y;
  const int qt = blockIdx.x / args.kv_splits, sp = blockIdx.x % args.kv_splits;
  int q0, W, k0, L;
  request_extent(args, i, q0, W, k0, L, threadIdx.x == 0 && blockIdx.x == 0 && h == 0);
  const int H = args.H;
  if (qt * 128 >= W) return;
  const int n_tiles = (L + 127) / 128;
  const int t_begin = sp * args.tiles_per_split;
  const int t_end = min(n_tiles, t_begin + args.tiles_per_split);
  const int nT = t_end - t_begin;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (nT <= 0) {
    // no keys in this split: zeros (single split) or an empty partial
    if (warp >= 2 && warp < 6) {
      const int lr = qt * 128 + (warp & 3) * 32 + lane;
      if (lr < W) {
        if (args.kv_splits == 1) {
          float z[DH];
          for (int c = 0; c < DH; ++c) z[c] = 0.f;
          store_cols(args.out, args.out_fp32, (static_cast<size_t>(q0 + lr) * H + h) * DH, z, DH, 1.f);
        } else {
          const size_t pr = partial_row(args, sp, i, lr, h);
          args.part_ml[pr * 2] = -INFINITY;
          args.part_ml[pr * 2 + 1] = 0.f;
        }
      }
    }
    return;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kOffBar);
  uint64_t *q_full = bars;                 // 1
  uint64_t *k_full = bars + 1;             // kKSt
  uint64_t *v_full = k_full + kKSt;        // kVSt
  uint64_t *s_full = v_full + kVSt;        // [buffer]: S(j) done (also frees K stage j mod 3)
  uint64_t *p_full = s_full + kSBuf;       // [buffer]
  uint64_t *pv_done = p_full + kSBuf;      // [buffer]: P(j) V done (also frees V stage j mod 3)
  uint64_t *o_ready = pv_done + kSBuf;     // one phase, after the last P.V
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(o_ready + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    int act = 0;   // softmax warps that hold query rows
    for (int q = 0; q < 4; ++q) act += qt * 128 + q * 32 < W;
    mbar_init(q_full, 1);
    for (int s = 0; s < kKSt; ++s) mbar_init(&k_full[s], 1);
    for (int s = 0; s < kVSt; ++s) mbar_init(&v_full[s], 1);
    for (int b = 0; b < kSBuf; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&p_full[b], act);
      mbar_init(&pv_done[b], 1);
    }
    mbar_init(o_ready, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  uint8_t *sQ = smem + Lay::kOffQ;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, Lay::kT);
      for (int c = 0; c < DH / 64; ++c) tma_load_2d(sQ + c * kBox, &tm_q, q_full, h * DH + c * 64, q0 + qt * 128);
      // K runs at most kKSt - 1 tiles ahead of V: a K stage frees as soon as
      // its S has run, a V stage only after its P.V, so this order never
      // waits on a later event while an earlier load could go. The stage of
      // tile t frees with buffer t mod 3's barrier; that buffer's next S / P.V
      // needs the tile being loaded here, so the parity test is exact.
      int jk = 0, jv = 0;
      while (jv < nT) {
        if (jk < nT && jk <= jv + (kKSt - 1)) {
          const int st = jk % kKSt;
          if (jk >= kKSt && !mbar_wait(&s_full[st], ((jk - kKSt) / kKSt) & 1, abort_flag)) break;
          uint8_t *dst = smem + Lay::kOffK + st * Lay::kT;
          mbar_arrive_expect_tx(&k_full[st], Lay::kT);
          const int y = k0 + (t_begin + jk) * 128;
          for (int c = 0; c < DH / 64; ++c) tma_load_2d(dst + c * kBox, &tm_k, &k_full[st], h * DH + c * 64, y);
          ++jk;
        } else {
          const int st = jv % kVSt;
          if (jv >= kVSt && !mbar_wait(&pv_done[st], ((jv - kVSt) / kVSt) & 1, abort_flag)) break;
          uint8_t *dst = smem + Lay::kOffV + st * Lay::kT;
          mbar_arrive_expect_tx(&v_full[st], Lay::kT);
          const int y = k0 + (t_begin + jv) * 128;
          for (int c = 0; c < DH / 64; ++c) tma_load_2d(dst + c * kBox, &tm_v, &v_full[st], h * DH + c * 64, y);
          ++jv;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- S issuer
    // S(j) = Q K_j^T into buffer j mod 3, once P(j - 3) V (issued by the
    // P.V warp) is done: that buffer's barrier, whose next phase needs S(j),
    // so the parity test is exact. Descriptors: only the 14-bit start-address
    // field differs between the K steps of one operand.
    if (lane == 0) {
      const uint64_t dq = sw128_desc(smem_u32(sQ), 16, 1024);
      bool ok = mbar_wait(q_full, 0, abort_flag);
      for (int j = 0; ok && j < nT; ++j) {
        const int st = j % kKSt, b = j % kSBuf;
        if (!mbar_wait(&k_full[st], (j / kKSt) & 1, abort_flag)) break;
        if (j >= kSBuf && !mbar_wait(&pv_done[b], ((j - kSBuf) / kSBuf) & 1, abort_flag)) break;
        tc_fence_after();
        const uint64_t dk = sw128_desc(smem_u32(smem + Lay::kOffK + st * Lay::kT), 16, 1024);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kBox + (kk & 3) * 32) >> 4);
          umma_bf16(tmem + b * 128, dq + off, dk + off, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[b]);
      }
    }
  } else if (warp == 6) {
    // ------------------------------------------------------------- P.V issuer
    // O += P(j) V_j once the softmax has written P(j) over S(j).
    if (lane == 0) {
      for (int j = 0; j < nT; ++j) {
        const int st = j % kVSt, b = j % kSBuf;
        if (!mbar_wait(&p_full[b], (j / kSBuf) & 1, abort_flag)) break;
        if (!mbar_wait(&v_full[st], (j / kVSt) & 1, abort_flag)) break;
        tc_fence_after();
        const uint64_t dv = sw128_desc(smem_u32(smem + Lay::kOffV + st * Lay::kT), kBox, 1024);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          umma_bf16_tmem_a(tmem + kColO, tmem + b * 128 + kk * 8, dv + static_cast<uint64_t>((kk * 2048) >> 4),
                           kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&pv_done[b]);
        if (j + 1 == nT) umma_commit(o_ready);
      }
    }
  } else {
    // ------------------------------------------------------------- softmax
    const int quarter = warp & 3;               // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;        // query row in the tile = TMEM lane
    const int lr = qt * 128 + row;              // query row in the request
    const bool warp_rows = qt * 128 + quarter * 32 < W;   // any row of this warp is a query
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t t_o = lane_base + kColO;
    const float c2 = args.scale_log2;
    constexpr float kLazy = 8.f;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    // a warp without query rows takes no part (the P barriers count only the
    // warps that hold rows)
    for (int j = 0; warp_rows && j < nT; ++j) {
      const int b = j % kSBuf;
      const uint32_t t_s = lane_base + b * 128;
      int w = 1;
      if (lane == 0) w = mbar_wait(&s_full[b], (j / kSBuf) & 1, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
      if (!ok) break;
      tc_fence_after();
      const int key0 = (t_begin + j) * 128;
      const bool full = key0 + 128 <= L && c2 > 0.f;   // no key masking; max(S*c) = max(S)*c
      uint32_t sr[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, *reinterpret_cast<uint32_t(*)[32]>(sr + c * 32));
      tmem_ld_wait();
      float mx = -INFINITY;
      if (full) {
        // three-input maxima: two new scores per step and chain
        float a0 = fmaxf(__uint_as_float(sr[0]), __uint_as_float(sr[1]));
        float a1 = fmaxf(__uint_as_float(sr[2]), __uint_as_float(sr[3]));
#pragma unroll
        for (int e = 4; e < 128; e += 4) {
          a0 = fmaxf(a0, fmaxf(__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])));
          a1 = fmaxf(a1, fmaxf(__uint_as_float(sr[e + 2]), __uint_as_float(sr[e + 3])));
        }
        mx = fmaxf(a0, a1) * c2;
      } else {
#pragma unroll
        for (int e = 0; e < 128; ++e)
          if (key0 + e < L) mx = fmaxf(mx, __uint_as_float(sr[e]) * c2);
      }
      const bool move = mx > m + kLazy;   // always on the first tile (m = -inf)
      const float m_new = move ? mx : m;
      const float corr = move ? ex2_approx(m - m_new) : 1.f;
      // a moved reference rescales O, which must hold exactly P(< j) V: wait
      // for P(j - 1) V (its buffer's barrier; a commit completes only once
      // every earlier MMA has, and the buffer is reused only after this
      // softmax hands over P(j + 2), so the parity test is exact), then the
      // whole warp rescales (tcgen05.ld/st are warp-collective; corr = 1 for
      // rows that keep their reference)
      if (j > 0 && __any_sync(0xffffffffu, move)) {
        int w2 = 1;
        if (lane == 0) w2 = mbar_wait(&pv_done[(j - 1) % kSBuf], ((j - 1) / kSBuf) & 1, abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, w2, 0) != 0;
        if (!ok) break;
        tc_fence_after();
#pragma unroll 1
        for (int c0 = 0; c0 < DH; c0 += 32) {
          uint32_t r[32];
          tmem_ld32(t_o + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr);
          tmem_st32(t_o + c0, r);
        }
      }
      // P = exp2(S*c - m) as bf16 pairs over the buffer's first 64 columns
      // two scores per packed FMA (S*c - m) and per packed add (the row sum)
      float2 acc = make_float2(0.f, 0.f);
      const float2 c2v = make_float2(c2, c2), mv = make_float2(-m_new, -m_new);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const int k = c * 64 + e;
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), c2v, mv);
          float p0 = ex2_approx(x.x);
          float p1 = ex2_approx(x.y);
          if (!full) {
            if (key0 + k >= L) p0 = 0.f;
            if (key0 + k + 1 >= L) p1 = 0.f;
          }
          acc = __fadd2_rn(acc, make_float2(p0, p1));
          pk[e >> 1] = pack_bf16x2(p0, p1);
        }
        tmem_st32(t_s + c * 32, pk);
      }
      tmem_st_wait();
      l = l * corr + (acc.x + acc.y);
      m = m_new;
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full[b]);
    }
    // O is final once the last P.V is done
    if (ok && warp_rows) {
      int w = 1;
      if (lane == 0) w = mbar_wait(o_ready, 0, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
    }
    tc_fence_after();
    if (ok && warp_rows) {
      const bool single = args.kv_splits == 1;
      const size_t pr = single ? 0 : partial_row(args, sp, i, lr < W ? lr : 0, h);
#pragma unroll 1
      for (int c0 = 0; c0 < DH; c0 += 32) {
        uint32_t r[32];
        tmem_ld32(t_o + c0, r);
        tmem_ld_wait();
        if (lr < W) {
          float o[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __uint_as_float(r[e]);
          if (single) {
            store_cols(args.out, args.out_fp32, (static_cast<size_t>(q0 + lr) * H + h) * DH + c0, o, 32, 1.f / l);
          } else {
            float4 *po = reinterpret_cast<float4 *>(args.part_o + pr * DH + c0);
#pragma unroll
            for (int e = 0; e < 32; e += 4) po[e / 4] = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
          }
        }
      }
      if (!single && lr < W) {
        args.part_ml[pr * 2] = m;
        args.part_ml[pr * 2 + 1] = l;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag && args.status) atomicOr(args.status, DLLM_DEV_WAIT_TIMEOUT);
}

// Merge the key-split partials of every (query row, head).
template <int DH>
__global__ void __launch_bounds__(256)
attn_combine_kernel(const AttnArgs args, int B) {
  pdl_trigger();
  pdl_wait();
  const int lr = blockIdx.x, i = blockIdx.y;
  int q0, W, k0, L;
  request_extent(args, i, q0, W, k0, L, false);
  if (lr >= W) return;
  const int n_tiles = (L + 127) / 128;
  const int n_valid = (n_tiles + args.tiles_per_split - 1) / args.tiles_per_split;
  const int H = args.H;
  const size_t split_stride = static_cast<size_t>(B) * args.max_q * H;
  for (int idx = threadIdx.x; idx < H * (DH / 4); idx += blockDim.x) {
    const int h = idx / (DH / 4), c4 = idx - h * (DH / 4);
    const size_t pr0 = (static_cast<size_t>(i) * args.max_q + lr) * H + h;
    float M = -INFINITY;
    for (int s = 0; s < n_valid; ++s) M = fmaxf(M, args.part_ml[(s * split_stride + pr0) * 2]);
    float lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < n_valid; ++s) {
      const size_t pr = s * split_stride + pr0;
      const float ms = args.part_ml[pr * 2];
      if (ms == -INFINITY) continue;
      const float wgt = exp2f(ms - M);
      lsum += args.part_ml[pr * 2 + 1] * wgt;
      const float4 x = reinterpret_cast<const float4 *>(args.part_o + pr * DH)[c4];
      acc.x += x.x * wgt; acc.y += x.y * wgt; acc.z += x.z * wgt; acc.w += x.w * wgt;
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const size_t ob = (static_cast<size_t>(q0 + lr) * H + h) * DH + c4 * 4;
    if (args.out_fp32) {
      reinterpret_cast<float4 *>(static_cast<float *>(args.out) + ob)[0] =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      uint16_t *p = static_cast<uint16_t *>(args.out) + ob;
      p[0] = f32_to_bf16(acc.x * inv); p[1] = f32_to_bf16(acc.y * inv);
      p[2] = f32_to_bf16(acc.z * inv); p[3] = f32_to_bf16(acc.w * inv);
    }
  }
}

struct AttnPlan {
  int q_tiles, kv_splits, tiles_per_split;
  size_t part_o, part_ml, total;
};

constexpr long long kMaxSplitCtas = 256;

size_t partial_bytes(size_t rows, int dh) { return align256(rows * dh * 4) + align256(rows * 2 * 4); }

AttnPlan attn_plan(int B, int H, int dh, int max_q, int max_kv, int sms) {
  AttnPlan p{};
  p.q_tiles = (max_q + 127) / 128;
  const int max_tiles = (max_kv + 127) / 128;
  const long long base = static_cast<long long>(B) * H * p.q_tiles;
  // One CTA per SM (shared memory, TMEM). A CTA's time is about its key
  // tiles plus about two tiles of prologue / epilogue; the grid takes waves
  // of them, and a split plan adds the merge launch (about three tiles,
  // overlapped by PDL in part). Pick the split count with the least total
  // (ties: fewer splits). A split plan never has more than kMaxSplitCtas
  // CTAs, which bounds its partials by kMaxSplitCtas x 128 rows whatever
  // the shape.
  long long best_cost = -1;
  p.tiles_per_split = max_tiles > 0 ? max_tiles : 1;
  for (int s = 1; s <= (max_tiles > 0 ? max_tiles : 1); ++s) {
    const int tps = (max_tiles + s - 1) / s;
    const int s_eff = (max_tiles + tps - 1) / tps;
    const long long ctas = base * s_eff;
    if (s_eff > 1 && ctas > kMaxSplitCtas) break;
    const long long waves = (ctas + sms - 1) / sms;
    const long long cost = waves * (tps + 2) + (s_eff > 1 ? 3 : 0);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      p.tiles_per_split = tps;
    }
  }
  if (p.tiles_per_split < 1) p.tiles_per_split = 1;
  p.kv_splits = (max_tiles + p.tiles_per_split - 1) / p.tiles_per_split;
  if (p.kv_splits < 1) p.kv_splits = 1;
  if (p.kv_splits > 1) {
    const size_t rows = static_cast<size_t>(p.kv_splits) * B * max_q * H;
    p.part_o = 0;
    p.part_ml = align256(rows * dh * 4);
    p.total = partial_bytes(rows, dh);
  }
  return p;
}

template <int DH>
dllm_status launch_attn(const dllm_bf16 *q, const dllm_bf16 *k, const dllm_bf16 *v, void *out, int out_fp32,
                        const int32_t *q_off, const int32_t *kv_off, int B, int H, int max_q, int max_kv,
                        int q_rows, int kv_rows, float scale, void *ws, size_t ws_bytes, cudaStream_t s) {
  const AttnPlan p = attn_plan(B, H, DH, max_q, max_kv, sm_budget());
  if (p.total > 0 && (!ws || ws_bytes < p.total || (reinterpret_cast<uintptr_t>(ws) & 255)))
    return DLLM_ERR_WORKSPACE;
  CUtensorMap tq, tk, tv;
  const uint64_t d = static_cast<uint64_t>(H) * DH;
  if (!make_tmap_bf16_sw128(&tq, q, q_rows, d, d, 128) || !make_tmap_bf16_sw128(&tk, k, kv_rows, d, d, 128) ||
      !make_tmap_bf16_sw128(&tv, v, kv_rows, d, d, 128))
    return DLLM_ERR_CUDA;
  AttnArgs a{};
  a.q_off = q_off;
  a.kv_off = kv_off;
  a.H = H;
  a.q_tiles = p.q_tiles;
  a.kv_splits = p.kv_splits;
  a.tiles_per_split = p.tiles_per_split;
  a.max_q = max_q;
  a.max_kv = max_kv;
  a.q_rows = q_rows;
  a.kv_rows = kv_rows;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  a.out_fp32 = out_fp32;
  a.part_o = p.total ? reinterpret_cast<float *>(static_cast<char *>(ws) + p.part_o) : nullptr;
  a.part_ml = p.total ? reinterpret_cast<float *>(static_cast<char *>(ws) + p.part_ml) : nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(&a.status), g_status_attn);
  if (e != cudaSuccess) return cuda_error(e);
  const int smem = AttnSmem<DH>::kBytes + 1024;
  auto kern = attn_umma_kernel<DH>;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return cuda_error(e);
  dim3 grid(p.q_tiles * p.kv_splits, H, B);
  e = launch_pdl(kern, grid, dim3(kAttnThreads), smem, s, tq, tk, tv, a);
  if (e != cudaSuccess) return cuda_error(e);
  unsigned launches = 1;
  if (p.kv_splits > 1) {
    e = launch_pdl(attn_combine_kernel<DH>, dim3(max_q, B), dim3(256), 0, s, a, B);
    if (e != cudaSuccess) return cuda_error(e);
    launches = 2;
  }
  return launch_status(launches);
}

}  // namespace

int attn_base_ctas(int B, int H, int dh, int max_q) {
  if (B < 1 || H < 1 || max_q < 1 || (dh != 64 && dh != 128)) return 0;
  return B * H * ((max_q + 127) / 128);
}

}  // namespace dllm

using namespace dllm;

extern "C" size_t dllm_block_attn_workspace(int B, int H, int dh, int max_q, int max_kv) {
  if (B < 1 || H < 1 || max_q < 1 || max_kv < 1 || (dh != 64 && dh != 128)) return 0;
  // A split plan has kv_splits * B * max_q * H partial rows, with
  // kv_splits <= key tiles and (kv_splits * B * H * query tiles) <=
  // kMaxSplitCtas, hence at most kMaxSplitCtas * 128 rows: a bound for any
  // GPU, any SM budget and any call with smaller max_q or max_kv.
  const long long tiles = (max_kv + 127) / 128;
  if (tiles < 2) return 0;
  long long rows = tiles * B * static_cast<long long>(max_q) * H;
  if (rows > kMaxSplitCtas * 128) rows = kMaxSplitCtas * 128;
  return partial_bytes(static_cast<size_t>(rows), dh);
}

extern "C" dllm_status dllm_block_attn(const dllm_bf16 *q, const dllm_bf16 *k, const dllm_bf16 *v, void *out,
                                       int out_fp32, const int32_t *q_off, const int32_t *kv_off, int B,
                                       int H, int dh, int max_q, int max_kv, int q_rows, int kv_rows,
                                       float scale, void *ws, size_t ws_bytes, dllm_stream stream) {
  if (B < 0 || H < 1 || max_q < 0 || max_kv < 0 || q_rows < 0 || kv_rows < 0) return DLLM_ERR_INVALID_ARG;
  if (dh != 64 && dh != 128) return DLLM_ERR_UNSUPPORTED;
  if (B > 4096 || H > 256) return DLLM_ERR_UNSUPPORTED;
  if (B == 0 || max_q == 0 || q_rows == 0) return DLLM_OK;
  if (!q || !k || !v || !out || !q_off || !kv_off) return DLLM_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return DLLM_ERR_INVALID_ARG;
  // no keys anywhere: every request is clipped to L = 0 and gets zeros; the
  // tensor maps stay valid but are never used
  if (kv_rows == 0) kv_rows = 1;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dh == 64)
    return launch_attn<64>(q, k, v, out, out_fp32, q_off, kv_off, B, H, max_q, max_kv, q_rows, kv_rows, scale,
                           ws, ws_bytes, s);
  return launch_attn<128>(q, k, v, out, out_fp32, q_off, kv_off, B, H, max_q, max_kv, q_rows, kv_rows, scale,
                          ws, ws_bytes, s);
}
