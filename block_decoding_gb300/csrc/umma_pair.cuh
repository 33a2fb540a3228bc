// The head GEMMs at many rows on CTA pairs (tcgen05.mma.cta_group::2).
//
//   D[m][n] = sum_k A[m][k] * B[n][k]      (bf16 in, fp32 accumulate in TMEM)
//
// A cluster of two CTAs on one TPC computes a 256 x BN tile: CTA r loads A
// rows 128 (2 t + r) .. +128 of M tile pair t and B rows BN/2 r .. +BN/2 of
// the n block into the same shared-memory offsets, and one pair MMA reads
// both halves of both operands. Per SM that is 16 KB of A and BN/2 x 128 B
// of B per K step of 64, a third less L2 -> SM traffic than the one-CTA
// tile of 128 x BN, for the same accumulator per SM (128 rows x BN in each
// CTA's TMEM, two buffers), so that the stage ring holds more K steps.
// The logits GEMM puts the rows (tokens) on M and the vocabulary on N
// (kEpiRowStats): each epilogue thread then holds one row and reduces its
// own 32-column chunks; the P.E GEMM keeps d on M and the rows on N.
//
// Roles (192 threads per CTA, as in umma_gemm.cuh):
//   warp 0      TMA producer of this CTA's halves; both CTAs' loads of a
//               stage signal the full barrier of rank 0, which expects the
//               bytes of both;
//   warp 1      TMEM allocation in both CTAs; in rank 0 one lane issues the
//               pair MMAs and commits each stage's release to the empty
//               barriers of both CTAs, and each finished accumulator to the
//               accumulator-full barriers of both;
//   warps 2..5  epilogue of this CTA's 128 rows; each warp's release of an
//               accumulator buffer arrives on rank 0's barrier (count 8).
// Every mbarrier wait is bounded. Before exiting, each producer waits until
// every stage it filled has been released (no MMA reads its shared memory
// and no commit still targets its barriers), and both CTAs meet at a
// cluster barrier that every thread reaches on every path.
#pragma once

#include <atomic>

#include "umma_gemm.cuh"

namespace dllm {

// This CTA's share of a stage: its A tile and half of the B tile.
template <int BN>
constexpr int pair_stage_bytes() {
  return kATileBytes + (BN / 2) * 64 * 2;
}

// Unit walk of the row-statistics GEMM (rows = tokens on M): the M tile pair
// varies fastest, so the pairs of one vocabulary tile run at the same time
// and share its HBM read; no K split.
__device__ __forceinline__ UnitPos unit_pos_mfast(const UmmaArgs &a, int u) {
  return UnitPos{u % a.m_tiles, u / a.m_tiles, 0, 0, a.k_steps, false};
}

// args.m_tiles counts 256-row M tile pairs. The row-statistics epilogue
// stores no fp32 D: it writes the statistics of each row's 32-column chunks
// and outb[m * ld + n] = bf16(D - max of D over n's chunk).
template <int BN, bool A_MN, int EPI>
__global__ void __launch_bounds__(kUmmaThreads, 1)
umma_pair_kernel(const __grid_constant__ CUtensorMap tma_a, const __grid_constant__ CUtensorMap tma_b,
                 const UmmaArgs args) {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "N tile");
  static_assert(EPI == kEpiStoreT || EPI == kEpiScaleT || EPI == kEpiRowStats, "fp32 and statistics epilogues");
  static_assert(EPI != kEpiRowStats || !A_MN, "statistics: plain K-major tiles");
  constexpr bool kRows = EPI == kEpiRowStats;
  constexpr int kHalfN = BN / 2;
  constexpr int kStage = pair_stage_bytes<BN>();
  constexpr int kBOff = kATileBytes;
  constexpr uint32_t kCols = umma_tmem_cols<BN, EPI>();
  constexpr uint32_t kIdesc = idesc_bf16(256, BN, A_MN ? 1 : 0, 0);
  static_assert(umma_acc_buffers<BN, EPI>() == 2, "two accumulator buffers");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = args.stages;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + static_cast<size_t>(S) * kStage);
  uint64_t *empty = full + S;
  uint64_t *tfull = empty + S;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pid = static_cast<int>(blockIdx.x >> 1), npairs = static_cast<int>(gridDim.x >> 1);
  const int units = unit_count(args);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);   // 4 epilogue warps x 2 CTAs (used in rank 0)
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tma_a);
    tma_prefetch_desc(&tma_b);
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_barrier();   // the peer's barriers are initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();
  pdl_wait();   // the prologue above touches no global memory

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int u = pid; ok && u < units; u += npairs) {
        const UnitPos up = kRows ? unit_pos_mfast(args, u) : unit_pos(args, u);
        const int mt = 2 * up.mt + static_cast<int>(rank);   // this CTA's 128-row M tile
        const int brow = up.nb * BN + static_cast<int>(rank) * kHalfN;
        for (int ks = up.kb; ks < up.ke; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * kStage);
          const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
          uint8_t *dst = smem + static_cast<size_t>(stage) * kStage;
          // both operands with the default L2 policy: the streamed one (A,
          // or B = W in the row-statistics GEMM) is read by two pairs that
          // sit on different GPCs and drift apart, and with evict-first the
          // later one missed it (read 1.37x from HBM)
          if (A_MN) {
            tma_load_2d_pair(dst, &tma_a, fb, mt * 128, ks * 64);
            tma_load_2d_pair(dst + kATileBytes / 2, &tma_a, fb, mt * 128 + 64, ks * 64);
          } else {
            tma_load_2d_pair(dst, &tma_a, fb, ks * 64, mt * 128);
          }
          tma_load_2d_pair(dst + kBOff, &tma_b, fb, ks * 64, brow);
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
      }
      // drain: every stage filled above has been released by the MMAs
      for (int i = 0; ok && i < S; ++i) {
        if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) break;
        if (++stage == S) { stage = 0; phase ^= 1; }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer (rank 0)
    if (leader && lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int u = pid; u < units; u += npairs) {
        const UnitPos up = kRows ? unit_pos_mfast(args, u) : unit_pos(args, u);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        bool ok = true;
        for (int ks = up.kb; ks < up.ke; ++ks) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + static_cast<size_t>(stage) * kStage);
          const uint32_t b_addr = a_addr + kBOff;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bdesc = sw128_desc(b_addr + kk * 32, 16, 1024);
            const uint64_t adesc = A_MN ? sw128_desc(a_addr + kk * 2048, kATileBytes / 2, 1024)
                                        : sw128_desc(a_addr + kk * 32, 16, 1024);
            umma_bf16_pair(d_tmem, adesc, bdesc, kIdesc, (ks > up.kb || kk > 0) ? 1u : 0u);
          }
          umma_commit_pair(smem_u32(&empty[stage]));
          umma_commit_pair(mapa_shared(smem_u32(&empty[stage]), 1));
          if (++stage == S) { stage = 0; phase ^= 1; }
        }
        if (!ok) break;
        umma_commit_pair(smem_u32(&tfull[acc]));
        umma_commit_pair(mapa_shared(smem_u32(&tfull[acc]), 1));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int u = pid; u < units; u += npairs) {
      const UnitPos up = kRows ? unit_pos_mfast(args, u) : unit_pos(args, u);
      const int mt = 2 * up.mt + static_cast<int>(rank), nb = up.nb;
      int ok = 1;
      if (lane == 0) ok = mbar_wait(&tfull[acc], acc_phase, abort_flag) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const int m = mt * 128 + row;
      const uint32_t taddr =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * BN);
      float *ob = args.out + static_cast<size_t>(up.sp) * args.N * args.ld;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float v[32];
        {
          uint32_t r[32];
          tmem_ld32(taddr + c0, r);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        }
        if (!kRows && m < args.M) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int n = nb * BN + c0 + j;
            if (n < args.N) {
              float x = v[j];
              if (EPI == kEpiScaleT) x *= args.col_scale[n];
              ob[static_cast<size_t>(n) * args.ld + m] = x;
            }
          }
        }
        if constexpr (kRows) {
          // this thread's row m over columns n0 .. n0 + 31 (one 32-column
          // chunk): max, its lowest column, sum of exp(D - max) over n < N,
          // then the row's bf16 D - max as four 16-byte stores
          const int n0 = nb * BN + c0;
          float mx = -INFINITY;
          int ar = 0x7fffffff;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n0 + j < args.N && v[j] > mx) { mx = v[j]; ar = j; }   // ascending: the first maximum
          float sum = 0.f;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (n0 + j < args.N) sum += __expf(v[j] - mx);
          if (m < args.M && n0 < args.N) {
            const size_t o = static_cast<size_t>(m) * args.st_ld + n0 / 32;
            args.st_m[o] = mx;
            args.st_l[o] = sum;
            args.st_a[o] = mx != -INFINITY ? n0 + ar : 0x7fffffff;   // no finite value: no argmax
            uint4 *dst = reinterpret_cast<uint4 *>(args.outb + static_cast<size_t>(m) * args.ld + n0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float f[8];
#pragma unroll
              for (int e = 0; e < 8; ++e) f[e] = v[8 * q + e] - mx;
              dst[q] = pack8(f);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty[acc]);
        else mbar_arrive_cluster_relaxed(mapa_shared(smem_u32(&tempty[acc]), 0));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_barrier();   // the peer's last arrivals on this CTA's barriers have landed
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kCols);
  }
  if (threadIdx.x == 0 && *abort_flag && args.status) atomicOr(args.status, DLLM_DEV_WAIT_TIMEOUT);
}

// CTA pairs that can be resident at once for this kernel (cached per
// instantiation and device); 0 if the query fails.
template <int BN, bool A_MN, int EPI>
int umma_pair_max_active(size_t smem) {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (const int c = cache[dev].load(std::memory_order_relaxed)) return c;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * 76);
  cfg.blockDim = dim3(kUmmaThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, umma_pair_kernel<BN, A_MN, EPI>, &cfg) != cudaSuccess || n <= 0) return 0;
  cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Host launcher (args.m_tiles = M tile pairs): returns false if the launch
// could not be configured.
template <int BN, bool A_MN, int EPI>
bool launch_umma_pair(const CUtensorMap &ta, const CUtensorMap &tb, UmmaArgs args, cudaStream_t s) {
  constexpr int kStage = pair_stage_bytes<BN>();
  int stages = static_cast<int>((220 * 1024 - 1024 - 256) / kStage);
  if (stages > 12) stages = 12;
  if (stages < 2) return false;
  args.stages = stages;
  args.out2 = nullptr;
  const size_t smem = umma_smem_bytes(kStage, stages);
  auto kern = umma_pair_kernel<BN, A_MN, EPI>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return false;
  const int units = args.m_tiles * args.n_blocks * args.k_splits;
  int pairs = sm_budget() / 2;
  const int resident = umma_pair_max_active<BN, A_MN, EPI>(smem);
  if (resident > 0 && resident < pairs) pairs = resident;
  if (units < pairs) pairs = units;
  if (pairs < 1) return false;
  return launch_pdl_pairs(kern, dim3(2 * pairs), dim3(kUmmaThreads), smem, s, ta, tb, args) == cudaSuccess;
}

}  // namespace dllm
