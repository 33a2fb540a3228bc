// K1: non-causal attention of the window queries over cached prefix + fresh
// window K/V (dInfer article, "vicinity KV refresh": only the block and its
// neighbourhood are recomputed each iteration, the distant cache is reused;
// Sangam abstract: attention is bidirectional, so no causal mask).
//
// One CTA per (request, head, 128-query tile, key split). tcgen05 flash
// attention with TMEM accumulators:
//   warp 0      TMA: Q tile once, then K and V tiles of 128 keys (one stage
//               ring each, K one tile ahead)
//   warp 1      MMA: S_j = Q K_j^T (K-major x K-major, N = 128) into one of
//               two TMEM S buffers, issued one tile ahead; O += P_j V_j
//               (P K-major from shared memory, V MN-major) into the TMEM O
//               accumulator
//   warps 2..17 softmax, four warps per TMEM lane quarter (32 keys and a
//               quarter of O's columns each): row max over S_j (keys beyond the
//               request masked), P_j = exp2(S*c - m) packed in registers
//               against a reference max m that moves only when the row max
//               passes it by more than 2^8 (then O is rescaled in TMEM),
//               stored to shared memory (128-byte-swizzled K-major) once
//               P_{j-1} V_{j-1} is done
// With one key split the CTA writes O/l; otherwise (m, l, O) partials go to
// the workspace and attn_combine merges them.
#include "umma.cuh"

namespace dllm {

DLLM_DEFINE_STATUS(attn)

namespace {

constexpr int kSoftWarps = 16;      // four per TMEM lane quarter, 32 keys of a tile each
constexpr int kAttnThreads = 32 * (2 + kSoftWarps);  // TMA warp, MMA warp, softmax warps
constexpr int kBox = 128 * 64 * 2;  // 16 KB: 128 rows x 64 bf16 (one swizzled TMA box)

// K and V tiles have rings of their own: a K stage is free once S_j = Q K_j^T
// has run, long before P_j V_j frees the V stage, so the next K tiles are in
// flight while the softmax of tile j runs.
template <int DH>
struct AttnSmem {
  static constexpr int kQ = (DH / 64) * kBox;
  static constexpr int kT = (DH / 64) * kBox;   // one K or V tile of 128 keys
  static constexpr int kStages = DH == 128 ? 2 : 4;   // per ring
  static constexpr int kOffK = kQ;
  static constexpr int kOffV = kOffK + kStages * kT;
  static constexpr int kOffP = kOffV + kStages * kT;
  static constexpr int kOffRed = kOffP + 2 * kBox;          // row-max / l exchange, 3 x 4 x 128 floats
  static constexpr int kOffBar = kOffRed + 3 * 4 * 128 * 4;
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

__device__ __forceinline__ void store_row(void *out, int out_fp32, size_t base, const float *o, int DH,
                                          float inv) {
  if (out_fp32) {
    float4 *p = reinterpret_cast<float4 *>(static_cast<float *>(out) + base);
    for (int c = 0; c < DH; c += 4) p[c / 4] = make_float4(o[c] * inv, o[c + 1] * inv, o[c + 2] * inv, o[c + 3] * inv);
  } else {
    uint4 *p = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + base);
    for (int c = 0; c < DH; c += 8) {
      float f[8];
      for (int e = 0; e < 8; ++e) f[e] = o[c + e] * inv;
      p[c / 8] = pack8(f);
    }
  }
}

template <int DH>
__global__ void __launch_bounds__(kAttnThreads, 1)
attn_umma_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const AttnArgs args) {
  using Lay = AttnSmem<DH>;
  constexpr int kSt = Lay::kStages;
  constexpr uint32_t kIdescS = idesc_bf16(128, 128, 0, 0);
  constexpr uint32_t kIdescO = idesc_bf16(128, DH, 0, 1);
  constexpr uint32_t kColO = 256;

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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (t_begin >= t_end) {
    // no keys in this split: zeros (single split) or an empty partial
    if (warp >= 2 && warp < 6) {
      const int row = (warp & 3) * 32 + lane;
      const int lr = qt * 128 + row;
      if (lr < W) {
        if (args.kv_splits == 1) {
          float z[DH];
          for (int c = 0; c < DH; ++c) z[c] = 0.f;
          store_row(args.out, args.out_fp32, (static_cast<size_t>(q0 + lr) * H + h) * DH, z, DH, 1.f);
        } else {
          const size_t pr = (static_cast<size_t>(sp) * gridDim.z * args.max_q + static_cast<size_t>(i) * args.max_q + lr) * H + h;
          args.part_ml[pr * 2] = -INFINITY;
          args.part_ml[pr * 2 + 1] = 0.f;
        }
      }
    }
    return;
  }
  const int nT = t_end - t_begin;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::kOffBar);
  uint64_t *q_full = bars;                 // 1
  uint64_t *k_full = bars + 1;             // kSt
  uint64_t *k_empty = k_full + kSt;        // kSt
  uint64_t *v_full = k_empty + kSt;        // kSt
  uint64_t *v_empty = v_full + kSt;        // kSt
  uint64_t *s_full = v_empty + kSt;        // 2
  uint64_t *s_empty = s_full + 2;          // 2
  uint64_t *p_full = s_empty + 2;          // 1
  uint64_t *pv_done = p_full + 1;          // 1
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(pv_done + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kSt; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&v_full[s], 1);
      mbar_init(&v_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], kSoftWarps);
    }
    mbar_init(p_full, kSoftWarps);
    mbar_init(pv_done, 1);
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
  uint8_t *sQ = smem;
  uint8_t *sP = smem + Lay::kOffP;

  if (warp == 0) {
    // ------------------------------------------------------------- producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, Lay::kQ);
      for (int c = 0; c < DH / 64; ++c) tma_load_2d(sQ + c * kBox, &tm_q, q_full, h * DH + c * 64, q0 + qt * 128);
      // K runs one tile ahead of V: K_{j+2} (free once S_j has run), then
      // V_{j+1} (free once P_{j-1} V_{j-1} has run) -- the order in which
      // their stages come free, so the single issuing thread never waits on
      // a later event while an earlier load could go
      int jk = 0, jv = 0;
      while (jv < nT) {
        if (jk < nT && jk <= jv + 1) {
          const int s = jk % kSt;
          if (!mbar_wait(&k_empty[s], ((jk / kSt) & 1) ^ 1, abort_flag)) break;
          uint8_t *dst = smem + Lay::kOffK + s * Lay::kT;
          mbar_arrive_expect_tx(&k_full[s], Lay::kT);
          const int y = k0 + (t_begin + jk) * 128;
          for (int c = 0; c < DH / 64; ++c) tma_load_2d(dst + c * kBox, &tm_k, &k_full[s], h * DH + c * 64, y);
          ++jk;
        } else {
          const int s = jv % kSt;
          if (!mbar_wait(&v_empty[s], ((jv / kSt) & 1) ^ 1, abort_flag)) break;
          uint8_t *dst = smem + Lay::kOffV + s * Lay::kT;
          mbar_arrive_expect_tx(&v_full[s], Lay::kT);
          const int y = k0 + (t_begin + jv) * 128;
          for (int c = 0; c < DH / 64; ++c) tma_load_2d(dst + c * kBox, &tm_v, &v_full[s], h * DH + c * 64, y);
          ++jv;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      auto issue_s = [&](int j) -> bool {
        const int s = j % kSt, b = j & 1;
        if (!mbar_wait(&k_full[s], (j / kSt) & 1, abort_flag)) return false;
        if (!mbar_wait(&s_empty[b], ((j >> 1) & 1) ^ 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t a0 = smem_u32(sQ);
        const uint32_t b0 = smem_u32(smem + Lay::kOffK + s * Lay::kT);
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          umma_bf16(tmem + b * 128, sw128_desc(a0 + off, 16, 1024), sw128_desc(b0 + off, 16, 1024), kIdescS,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[b]);
        umma_commit(&k_empty[s]);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, abort_flag) && issue_s(0);
      for (int j = 0; ok && j < nT; ++j) {
        if (j + 1 < nT && !issue_s(j + 1)) break;
        const int s = j % kSt;
        if (!mbar_wait(p_full, j & 1, abort_flag)) break;
        if (!mbar_wait(&v_full[s], (j / kSt) & 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t pa = smem_u32(sP);
        const uint32_t vb = smem_u32(smem + Lay::kOffV + s * Lay::kT);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t ad = sw128_desc(pa + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sw128_desc(vb + kk * 2048, kBox, 1024);
          umma_bf16(tmem + kColO, ad, bd, kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(pv_done);
        umma_commit(&v_empty[s]);
      }
    }
  } else {
    // ------------------------------------------------------------- softmax
    // Four warps per TMEM lane quarter: group g (0..3) owns keys 32g..32g+31
    // of every tile and O columns [g DH/4, (g+1) DH/4). The four warps of a
    // quarter exchange their partial row max through shared memory (a
    // 128-thread named barrier per quarter).
    //
    // O accumulates in TMEM across the tiles (P_j V_j adds to it). m is a
    // reference maximum: P_j = exp2(S_j*c - m), and m moves only when a
    // tile's row max exceeds it by more than kLazy (so P < 2^kLazy); then O
    // (once P_{j-1} V_{j-1} has landed) and l are rescaled by exp2(m - m_new).
    // O / l is the same for any reference m; the final m, l and O go out.
    const int quarter = warp & 3;
    const int g = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;
    const uint32_t trow = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    constexpr int kOQ = DH / 4;
    const uint32_t t_o = trow + kColO + g * kOQ;   // this warp's O columns
    const uint32_t bar_id = 1 + quarter;
    float *red = reinterpret_cast<float *>(smem + Lay::kOffRed);   // [2 parity][4 groups][128 rows], then [4][128]
    const float c2 = args.scale_log2;
    constexpr float kLazy = 8.f;
    float m = -INFINITY, l = 0.f;
    // Every softmax warp executes exactly nT + 1 quarter barriers, whatever
    // happens: after a failed (bounded) wait it keeps walking the loop with
    // ok = false, doing no work, so the four warps of a quarter never pair
    // barriers from different places.
    bool ok = true;
    for (int j = 0; j < nT; ++j) {
      const int b = j & 1;
      int w = 1;
      if (ok) {
        if (lane == 0) w = mbar_wait(&s_full[b], (j >> 1) & 1, abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
      }
      const int key0 = (t_begin + j) * 128 + g * 32;
      // all 32 keys of this warp valid and a positive scale: no per-key
      // masking, and the max of the raw scores scales to the max of S*c
      const bool fast = key0 + 32 <= L && c2 > 0.f;
      // this warp's 32 scores, then the S buffer goes back to the MMA warp
      uint32_t sr[32];
      float mx = -INFINITY;
      if (ok) {
        tc_fence_after();
        tmem_ld32(trow + b * 128 + g * 32, sr);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_empty[b]);
        if (fast) {
          float a0 = __uint_as_float(sr[0]), a1 = __uint_as_float(sr[1]);
          float a2 = __uint_as_float(sr[2]), a3 = __uint_as_float(sr[3]);
#pragma unroll
          for (int e = 4; e < 32; e += 4) {
            a0 = fmaxf(a0, __uint_as_float(sr[e]));
            a1 = fmaxf(a1, __uint_as_float(sr[e + 1]));
            a2 = fmaxf(a2, __uint_as_float(sr[e + 2]));
            a3 = fmaxf(a3, __uint_as_float(sr[e + 3]));
          }
          mx = fmaxf(fmaxf(a0, a1), fmaxf(a2, a3)) * c2;
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (key0 + e < L) mx = fmaxf(mx, __uint_as_float(sr[e]) * c2);
        }
      }
      red[(b * 4 + g) * 128 + row] = mx;
      named_bar_sync(bar_id, 128);
      if (!ok) continue;
      // the same four values in the same order in all four warps
      mx = fmaxf(fmaxf(red[(b * 4) * 128 + row], red[(b * 4 + 1) * 128 + row]),
                 fmaxf(red[(b * 4 + 2) * 128 + row], red[(b * 4 + 3) * 128 + row]));
      const bool move = mx > m + kLazy;   // always on the first tile (m = -inf)
      const float m_new = move ? mx : m;
      const float corr = move ? ex2_approx(m - m_new) : 1.f;
      // P = exp2(S*c - m_new) for this warp's 32 keys, packed to bf16 in
      // registers while P_{j-1} V_{j-1} still runs
      float lsum = 0.f;
      uint32_t pk[16];
      {
        float p[32];
        if (fast) {
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            p[e] = ex2_approx(fmaf(__uint_as_float(sr[e]), c2, -m_new));
            p[e + 1] = ex2_approx(fmaf(__uint_as_float(sr[e + 1]), c2, -m_new));
            s0 += p[e];
            s1 += p[e + 1];
          }
          lsum = s0 + s1;
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            p[e] = (key0 + e < L) ? ex2_approx(fmaf(__uint_as_float(sr[e]), c2, -m_new)) : 0.f;
            lsum += p[e];
          }
        }
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(p[2 * e], p[2 * e + 1]);
      }
      // P_{j-1} V_{j-1} done: the P buffer is free and O holds tiles < j
      if (j >= 1) {
        if (lane == 0) w = mbar_wait(pv_done, (j - 1) & 1, abort_flag) ? 1 : 0;
        ok = __shfl_sync(0xffffffffu, w, 0) != 0;
        if (!ok) continue;
        // rescale this warp's columns of O in place: the whole warp or none
        // of it (tcgen05.ld/st are warp-collective), rows that keep their
        // reference max scaling by corr = 1
        if (__any_sync(0xffffffffu, move)) {
          tc_fence_after();
#pragma unroll
          for (int c0 = 0; c0 < kOQ; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(t_o + c0, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * corr);
            tmem_st16(t_o + c0, r);
          }
          tmem_st_wait();
        }
      }
      // P_j keys 32g..32g+31 -> P box g / 2, 16-byte chunks 4 (g & 1) .. +3
      // of the row (128-byte swizzled K-major), then P_j V_j may start
      uint8_t *box = sP + (g >> 1) * kBox + row * 128;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        const int c = (g & 1) * 4 + ch;
        *reinterpret_cast<uint4 *>(box + ((c ^ (row & 7)) << 4)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full);
      l = l * corr + lsum;
      m = m_new;
    }
    float o[kOQ];
    if (ok) {
      int w = 1;
      if (lane == 0) w = mbar_wait(pv_done, (nT - 1) & 1, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, w, 0) != 0;
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < kOQ; c0 += 16) {
          uint32_t r[16];
          tmem_ld16(t_o + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) o[c0 + e] = __uint_as_float(r[e]);
        }
      }
    }
    // total l of the row = the four groups' partial sums, in group order
    red[(8 + g) * 128 + row] = l;
    named_bar_sync(bar_id, 128);
    l = (red[8 * 128 + row] + red[9 * 128 + row]) + (red[10 * 128 + row] + red[11 * 128 + row]);
    const int lr = qt * 128 + row;
    if (ok && lr < W) {
      if (args.kv_splits == 1) {
        store_row(args.out, args.out_fp32, (static_cast<size_t>(q0 + lr) * H + h) * DH + g * kOQ, o, kOQ,
                  1.f / l);
      } else {
        const size_t pr = (static_cast<size_t>(sp) * gridDim.z * args.max_q + static_cast<size_t>(i) * args.max_q + lr) * H + h;
        float4 *po = reinterpret_cast<float4 *>(args.part_o + pr * DH + g * kOQ);
#pragma unroll
        for (int c = 0; c < kOQ; c += 4) po[c / 4] = make_float4(o[c], o[c + 1], o[c + 2], o[c + 3]);
        if (g == 0) {
          args.part_ml[pr * 2] = m;
          args.part_ml[pr * 2 + 1] = l;
        }
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
  // One CTA per SM (shared memory), so the time is about
  // waves x (tiles per CTA + one tile of prologue/epilogue), plus the merge
  // pass when the keys are split (a separate launch overlapped by PDL: about
  // two tile times, four when it merges the partials of more than 64 CTAs --
  // fitted to the measured steps): pick the split count that minimises it
  // (ties: fewer splits). A split plan never has more than kMaxSplitCtas
  // CTAs, which bounds its partials by kMaxSplitCtas x 128 rows whatever the
  // shape.
  long long best_cost = -1;
  p.tiles_per_split = max_tiles > 0 ? max_tiles : 1;
  for (int s = 1; s <= (max_tiles > 0 ? max_tiles : 1); ++s) {
    const int tps = (max_tiles + s - 1) / s;
    const int s_eff = (max_tiles + tps - 1) / tps;
    const long long ctas = base * s_eff;
    if (s_eff > 1 && ctas > kMaxSplitCtas) break;
    const long long waves = (ctas + sms - 1) / sms;
    const long long merge = s_eff > 1 ? (ctas > 64 ? 4 : 2) : 0;
    const long long cost = waves * (tps + 1) + merge;
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
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&a.status), g_status_attn) != cudaSuccess)
    return DLLM_ERR_CUDA;
  const int smem = AttnSmem<DH>::kBytes + 1024;
  auto kern = attn_umma_kernel<DH>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return DLLM_ERR_CUDA;
  dim3 grid(p.q_tiles * p.kv_splits, H, B);
  if (launch_pdl(kern, grid, dim3(kAttnThreads), smem, s, tq, tk, tv, a) != cudaSuccess) return DLLM_ERR_CUDA;
  unsigned launches = 1;
  if (p.kv_splits > 1) {
    if (launch_pdl(attn_combine_kernel<DH>, dim3(max_q, B), dim3(256), 0, s, a, B) != cudaSuccess)
      return DLLM_ERR_CUDA;
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
