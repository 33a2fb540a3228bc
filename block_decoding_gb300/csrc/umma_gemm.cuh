// Persistent tcgen05 GEMM for the vocabulary-sized contractions of the head.
//
//   D[m][n] = sum_k A[m][k] * B[n][k]      (bf16 in, fp32 accumulate in TMEM)
//
// M tile 128 (one TMEM lane per row), N tile BN (<= 256 TMEM columns), K in
// steps of 64 (one 128-byte swizzled TMA box). A is K-major ([m][k], e.g.
// the LM head W[v][d]) or MN-major ([k][m], e.g. the embedding table E[v][d]
// read as E^T for P.E); B is always K-major ([n][k]).
//
// Work unit = (m tile, n block, k split); CTAs (one per SM) walk the units.
// Warp roles (192 threads):
//   warp 0      TMA producer (one lane): stage ring of A/B boxes, full/empty
//               mbarriers with transaction counts;
//   warp 1      TMEM owner + MMA issuer (one lane): 4 x tcgen05.mma (K = 16)
//               per stage into one of two TMEM accumulators, tcgen05.commit
//               frees the stage and, after the last K step, hands the
//               accumulator to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, then the
//               kind-specific store (coalesced along m for a fixed n).
// Every wait is bounded (umma.cuh): a stuck pipeline sets the device status
// word and the kernel returns after releasing its TMEM.
#pragma once

#include "umma.cuh"

namespace dllm {

enum UmmaEpilogue : int {
  kEpiStoreT = 0,   // out[(split*N + n)*ld + m] = D                   (logits z[r][v])
  kEpiScaleT = 1,   // out[(split*N + n)*ld + m] = D * col_scale[n]    (P.E partials)
  kEpiBf16T = 2,    // outb[n*ld + m] = bf16(D (+ aux[n*ld + m]))      (projection, + residual)
  kEpiSwiGLU = 3,   // two A tiles (rows m and a1_row + m), two accumulators:
                    // outb[n*ld + m] = bf16(silu(D0) * D1)            (gate/up projection)
  kEpiRowStats = 4,  // CTA pairs only (umma_pair.cuh), rows on M (tokens), columns on N
                    // (vocabulary): per (row m, 32-column chunk q of n) max, lowest
                    // arg-max column and sum exp(D - max) over n < N ->
                    // st_m / st_a / st_l[m * st_ld + q]; outb[m * ld + n] = bf16(D - that
                    // max)                                         (logits + softmax stats)
};

struct UmmaArgs {
  int m_tiles, n_blocks, k_splits;
  int k_steps, k_per_split;
  int M, N;
  int stages;
  float *out;
  long long ld;
  const float *col_scale;
  unsigned int *status;
  uint16_t *outb;          // bf16 epilogues
  const uint16_t *aux;     // residual (may alias outb) or nullptr
  int a1_row;              // SwiGLU: row offset of the second A tile
  const void *pf;          // optional: L2 prefetch of [pf, pf + pf_bytes) (the
  unsigned long long pf_bytes;  // next GEMM's weights), split over the CTAs
  float *st_m, *st_l;      // kEpiRowStats: [M][st_ld] statistics of 32-column
  int *st_a;               // chunks, chunk q of row m at m * st_ld + q
  int st_ld;
  // Split tail (kEpiStoreT, one n block, no k split): units past full_units
  // are the two K halves of the M tiles tail_m0 .. m_tiles - 1; the first
  // half stores as usual, the second into out2[n * ld2 + m - 128 tail_m0].
  // Used when the last round of whole tiles would leave most CTAs idle.
  float *out2;             // nullptr: no split tail
  long long ld2;
  int full_units, tail_m0;
};

constexpr int kUmmaThreads = 192;
constexpr int kATileBytes = 128 * 64 * 2;  // 16 KB: 128 rows x 64 bf16

// A tiles per stage: two for SwiGLU (gate, up), else one.
template <int EPI>
constexpr int umma_num_a() {
  return EPI == kEpiSwiGLU ? 2 : 1;
}

template <int BN, int EPI = 0>
constexpr int umma_stage_bytes() {
  return umma_num_a<EPI>() * kATileBytes + BN * 64 * 2;
}

// TMEM accumulator buffers: two (epilogue overlaps the next unit) when they
// fit in the 512 columns, else one.
template <int BN, int EPI = 0>
constexpr int umma_acc_buffers() {
  return 2 * umma_num_a<EPI>() * BN <= 512 ? 2 : 1;
}

template <int BN, int EPI = 0>
constexpr uint32_t umma_tmem_cols() {
  constexpr int c = umma_acc_buffers<BN, EPI>() * umma_num_a<EPI>() * BN;
  return (c <= 32) ? 32 : (c <= 64) ? 64 : (c <= 128) ? 128 : (c <= 256) ? 256 : 512;
}

inline size_t umma_smem_bytes(int stage_bytes, int stages) {
  return 1024 + static_cast<size_t>(stage_bytes) * stages + 256;
}

// Work walk: CTA c takes units u = c, c + G, ... (G CTAs); a unit is one
// (m tile, n block, k split), or one K half of a split-tail tile.
struct UnitPos {
  int mt, nb, sp;
  int kb, ke;   // k-steps [kb, ke)
  bool half;    // the second K half of a split-tail tile
};

__device__ __forceinline__ int unit_count(const UmmaArgs &a) {
  return a.out2 ? a.full_units + 2 * (a.m_tiles - a.tail_m0) : a.m_tiles * a.n_blocks * a.k_splits;
}

// The n block varies fastest: the units of one A tile run on neighbouring
// CTAs at the same time, so A (the streamed weight) is read from HBM once
// and its other uses hit L2.
__device__ __forceinline__ UnitPos unit_pos(const UmmaArgs &a, int u) {
  if (a.out2 && u >= a.full_units) {
    const int t = u - a.full_units, kh = a.k_steps / 2;
    const int h = t & 1;
    return UnitPos{a.tail_m0 + (t >> 1), 0, 0, h ? kh : 0, h ? a.k_steps : kh, h != 0};
  }
  const int nb = u % a.n_blocks;
  const int rest = u / a.n_blocks;
  const int sp = rest / a.m_tiles;
  const int kb = sp * a.k_per_split;
  return UnitPos{rest % a.m_tiles, nb, sp, kb, min(a.k_steps, kb + a.k_per_split), false};
}

template <int BN, bool A_MN, int EPI>
__global__ void __launch_bounds__(kUmmaThreads, 1)
umma_gemm_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                 const UmmaArgs args) {
  static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "N tile");
  constexpr bool kDual = EPI == kEpiSwiGLU;
  static_assert(!kDual || (BN <= 128 && !A_MN), "dual accumulators: 4 x BN TMEM columns, K-major A");
  static_assert(EPI != kEpiRowStats, "statistics: the CTA-pair kernel (umma_pair.cuh)");
  constexpr int kNumA = umma_num_a<EPI>();
  constexpr int kStage = umma_stage_bytes<BN, EPI>();
  constexpr int kBOff = kNumA * kATileBytes;              // B tile offset inside a stage
  constexpr int kAccCols = kNumA * BN;                    // TMEM columns per accumulator buffer
  constexpr int kBuffers = umma_acc_buffers<BN, EPI>();
  constexpr uint32_t kCols = umma_tmem_cols<BN, EPI>();
  constexpr uint32_t kIdesc = idesc_bf16(128, BN, A_MN ? 1 : 0, 0);

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = args.stages;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * kStage);
  uint64_t *empty = full + S;
  uint64_t *tfull = empty + S;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cid = static_cast<int>(blockIdx.x), nctas = static_cast<int>(gridDim.x);
  const int units = unit_count(args);

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
  pdl_trigger();
  pdl_wait();   // the prologue above touches no global memory

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();  // A streams through once
      int stage = 0;
      uint32_t phase = 0;
      for (int u = cid; u < units; u += nctas) {
        const UnitPos up = unit_pos(args, u);
        const int mt = up.mt, nb = up.nb;
        const int kb = up.kb, ke = up.ke;
        for (int ks = kb; ks < ke; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) goto producer_done;
          mbar_arrive_expect_tx(&full[stage], kStage);
          uint8_t *a_dst = smem + static_cast<size_t>(stage) * kStage;
#pragma unroll
          for (int k = 0; k < kNumA; ++k) {
            uint8_t *ak = a_dst + k * kATileBytes;
            if (A_MN) {
              tma_load_2d_hint(ak, &tma_a, &full[stage], (mt + k) * 128, ks * 64, pol);
              tma_load_2d_hint(ak + kATileBytes / 2, &tma_a, &full[stage], (mt + k) * 128 + 64, ks * 64, pol);
            } else {
              const int row = kDual ? (k == 0 ? mt * 128 : args.a1_row + mt * 128) : (mt + k) * 128;
              tma_load_2d_hint(ak, &tma_a, &full[stage], ks * 64, row, pol);
            }
          }
          tma_load_2d(a_dst + kBOff, &tma_b, &full[stage], ks * 64, nb * BN);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      // every load of this CTA is issued: warm L2 with its share of the next
      // GEMM's weights, which do not depend on this GEMM's result
      l2_prefetch_share(args.pf, args.pf_bytes);
    producer_done:;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int u = cid; u < units; u += nctas) {
        const UnitPos up = unit_pos(args, u);
        const int kb = up.kb, ke = up.ke;
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag)) goto mma_done;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kAccCols);
        for (int ks = kb; ks < ke; ++ks) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) goto mma_done;
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + static_cast<size_t>(stage) * kStage);
          const uint32_t b_addr = a_addr + kBOff;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = sw128_desc(b_addr + kk * 32, 16, 1024);
#pragma unroll
            for (int k = 0; k < kNumA; ++k) {
              const uint32_t ak = a_addr + k * kATileBytes;
              const uint64_t adesc = A_MN ? sw128_desc(ak + kk * 2048, kATileBytes / 2, 1024)
                                          : sw128_desc(ak + kk * 32, 16, 1024);
              umma_bf16(d_tmem + k * BN, adesc, bdesc, kIdesc, (ks > kb || kk > 0) ? 1u : 0u);
            }
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
    for (int u = cid; u < units; u += nctas) {
      const UnitPos up = unit_pos(args, u);
      const int mt = up.mt, nb = up.nb, sp = up.sp;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int m = mt * 128 + row;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * kAccCols);
      // fp32 stores of this unit: out[(sp N + n) ld + m], or for the second K
      // half of a split-tail tile out2[n ld2 + m - 128 tail_m0] (chosen once
      // per unit, outside the store loop)
      const bool to2 = EPI == kEpiStoreT && up.half;
      float *ob = to2 ? args.out2 : args.out + static_cast<size_t>(sp) * args.N * args.ld;
      const long long ob_ld = to2 ? args.ld2 : args.ld;
      const int ob_m0 = to2 ? 128 * args.tail_m0 : 0;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += (BN >= 32 ? 32 : 16)) {
        float v[32];
        float g[32];  // SwiGLU: the gate accumulator (v holds the up accumulator)
        if constexpr (BN >= 32) {
          uint32_t r[32];
          tmem_ld32(taddr + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          if constexpr (kDual) {
#pragma unroll
            for (int j = 0; j < 32; ++j) g[j] = v[j];
            tmem_ld32(taddr + BN + c0, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          }
        } else {
          uint32_t r[16];
          tmem_ld16(taddr + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
          if constexpr (kDual) {
#pragma unroll
            for (int j = 0; j < 16; ++j) g[j] = v[j];
            tmem_ld16(taddr + BN + c0, r);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
          }
        }
        constexpr int kC = BN >= 32 ? 32 : 16;
        if (m < args.M) {
#pragma unroll
          for (int j = 0; j < kC; ++j) {
            const int n = nb * BN + c0 + j;
            if (n < args.N) {
              float x = v[j];
              if constexpr (EPI == kEpiStoreT || EPI == kEpiScaleT) {
                if (EPI == kEpiScaleT) x *= args.col_scale[n];
                ob[static_cast<size_t>(n) * ob_ld + (m - ob_m0)] = x;
              } else {
                const size_t o = static_cast<size_t>(n) * args.ld + m;
                if constexpr (kDual) x = g[j] / (1.f + __expf(-g[j])) * x;   // silu(gate) * up
                if (EPI == kEpiBf16T && args.aux) x += bf16_to_f32(args.aux[o]);
                args.outb[o] = f32_to_bf16(x);
              }
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

// Host launcher: returns false if the launch could not be configured.
template <int BN, bool A_MN, int EPI>
bool launch_umma_gemm(const CUtensorMap &ta, const CUtensorMap &tb, UmmaArgs args, cudaStream_t s) {
  constexpr int kStage = umma_stage_bytes<BN, EPI>();
  int stages = static_cast<int>((220 * 1024 - 1024 - 256) / kStage);
  if (stages > 12) stages = 12;
  if (stages < 2) return false;
  args.stages = stages;
  const size_t smem = umma_smem_bytes(kStage, stages);
  auto kern = umma_gemm_kernel<BN, A_MN, EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return false;
  const int units = args.out2 ? args.full_units + 2 * (args.m_tiles - args.tail_m0)
                              : args.m_tiles * args.n_blocks * args.k_splits;
  const int sms = sm_budget();
  const int ctas = units < sms ? units : sms;
  return launch_pdl(kern, dim3(ctas), dim3(kUmmaThreads), smem, s, ta, tb, args) == cudaSuccess;
}

}  // namespace dllm
