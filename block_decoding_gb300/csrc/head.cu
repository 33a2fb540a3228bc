// K2: LM head + vocabulary softmax statistics + expected embedding P.E.
//
// dInfer article: decoding problem 3 (a plain decoder keeps only the most
// confident token of each position) and "iteration smoothing" (the
// probability-weighted information of undecoded positions is carried into
// the next iteration). Per head row r:
//   z[r][v] = <h[r], W[v]>, m = max z, a = lowest argmax,
//   l = sum exp(z - m), conf = 1 / l, PE[r] = sum_v exp(z - m) / l * E[v].
//
// Kernels (one stream, no host sync):
//   1. umma_gemm<LOGITS>  z^T tile = W tile (128 vocab rows, K-major) x h^T,
//                         tcgen05 + TMA; the epilogue writes fp32 z and, per
//                         (vocab tile, row), max / lowest argmax / sum exp
//   2. stats_combine      per row: merge the tiles -> m, argmax, l, conf, 1/l
//   3. finalize_probs     P[r][v] = bf16(exp(z - m)) (zero in the 64-pad)
//   4. umma_gemm<PE>      PE^T partial = E^T tile (128 d rows, MN-major) x P^T
//                         over a vocab split, scaled by 1/l
//   5. pe_combine         sum of the vocab splits
// W and E, the two V x d streams, are each read once from HBM; z is written
// once and read once (by finalize_probs).
#include "umma_pair.cuh"

namespace dllm {

DLLM_DEFINE_STATUS(head)

namespace {

constexpr int kStatChunks = 32;   // vocab slices per row (P pass; few-row statistics)
// From this many head rows on, the logits GEMM computes the softmax
// statistics in its epilogue (one pass over the R x V logits saved); below,
// a separate pass over them is cheaper (measured: R = 32 step 360 vs
// 368 us, R = 512 head 0.90 vs 0.87 ms).
constexpr int kFusedStatsRows = 128;

// (m, l, a) <- (m, l, a) merged with (m2, l2, a2): running max, sum of
// exp(z - max) rescaled to it, lowest index among the maxima.
__device__ __forceinline__ void merge_stats(float &m, float &l, int &a, float m2, float l2, int a2) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) { m = m2; l = l2; a = a2; return; }
  if (m2 > m) {
    l = l * __expf(m - m2) + l2;
    m = m2;
    a = a2;
  } else {
    l += l2 * __expf(m2 - m);
    if (m2 == m && a2 < a) a = a2;
  }
}

// Per row: merge the logits GEMM's statistics of every 32-wide vocab slice
// (st_*[r][slice], slice order = vocab order) into m, the lowest argmax and
// l; write m, 1/l, argmax and conf = 1/l. One CTA of 256 threads per row.
__global__ void __launch_bounds__(256)
stats_combine_kernel(const float *__restrict__ st_m, const float *__restrict__ st_l, const int *__restrict__ st_a,
                     int slices, float *__restrict__ m_out, float *__restrict__ inv_l,
                     int32_t *__restrict__ argmax, float *__restrict__ conf) {
  pdl_trigger();
  pdl_wait();
  __shared__ float sm[8], sl[8];
  __shared__ int sa[8];
  const int r = blockIdx.x;
  const size_t row = static_cast<size_t>(r) * slices;
  float m = -INFINITY, l = 0.f;
  int a = 0x7fffffff;
  // up to 16 slices per thread per round, loaded together (independent
  // loads in flight), then reduced: max and its lowest index first, then the
  // rescaled sum
  for (int t0 = 0; t0 < slices; t0 += 16 * 256) {
    float xm[16], xl[16];
    int xa[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const int t = t0 + k * 256 + threadIdx.x;
      const bool in = t < slices;
      xm[k] = in ? st_m[row + t] : -INFINITY;
      xl[k] = in ? st_l[row + t] : 0.f;
      xa[k] = in ? st_a[row + t] : 0x7fffffff;
    }
    float mm = -INFINITY;
    int aa = 0x7fffffff;
#pragma unroll
    for (int k = 0; k < 16; ++k)
      if (xm[k] > mm || (xm[k] == mm && xa[k] < aa)) { mm = xm[k]; aa = xa[k]; }
    float ll = 0.f;
    if (mm != -INFINITY) {
#pragma unroll
      for (int k = 0; k < 16; ++k)
        if (xm[k] != -INFINITY) ll += xl[k] * __expf(xm[k] - mm);
    }
    merge_stats(m, l, a, mm, ll, aa);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    merge_stats(m, l, a, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o),
                __shfl_xor_sync(0xffffffffu, a, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    sm[warp] = m;
    sl[warp] = l;
    sa[warp] = a;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < 8; ++w) merge_stats(m, l, a, sm[w], sl[w], sa[w]);
    m_out[r] = m;
    inv_l[r] = 1.f / l;
    argmax[r] = a;
    conf[r] = 1.f / l;
  }
}

// Few rows (R < kFusedStatsRows): the logits are small enough (R x V fp32,
// 16 MB at R = 32) that one extra pass over them costs less than the
// statistics epilogue in the logits GEMM. Per (row, vocab chunk): max,
// lowest argmax, sum exp.
__global__ void __launch_bounds__(256)
stats_partial_kernel(const float *__restrict__ z, long long ldz, int V, int chunk,
                     float *__restrict__ pm, int *__restrict__ pa, float *__restrict__ pl,
                     const float *__restrict__ z2, long long ld2, int tail_v0) {
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x, r = blockIdx.y;
  const int v0 = c * chunk, v1 = min(V, v0 + chunk);
  const float *zr = z + static_cast<size_t>(r) * ldz;
  const float *z2r = z2 + static_cast<size_t>(r) * ld2;
  // a logit of the split tail is the sum of its two K halves
  auto zval = [&](int v) { return v >= tail_v0 ? zr[v] + z2r[v - tail_v0] : zr[v]; };
  __shared__ float sm[8];
  __shared__ int sa[8];
  __shared__ float sl[8];
  float m = -INFINITY;
  int a = 0x7fffffff;
  for (int v = v0 + threadIdx.x; v < v1; v += 256) {
    const float x = zval(v);
    if (x > m) { m = x; a = v; }  // ascending v per thread: first maximum kept
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
  m = sm[0];
  a = sa[0];
  for (int w = 1; w < 8; ++w)
    if (sm[w] > m || (sm[w] == m && sa[w] < a)) { m = sm[w]; a = sa[w]; }
  float l = 0.f;
  if (m > -INFINITY)
    for (int v = v0 + threadIdx.x; v < v1; v += 256) l += __expf(zval(v) - m);
  l = warp_sum(l);
  if (lane == 0) sl[warp] = l;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += sl[w];
    const int idx = r * gridDim.x + c;
    pm[idx] = m;
    pa[idx] = a;
    pl[idx] = t;
  }
}

// Few rows: per row, merge the chunk partials -> m, lowest argmax, l (one
// warp), then, when P is wanted, P[r][v] = bf16(exp(z[r][v] - m)) over this
// CTA's slice of [0, Vp) (zero in the pad [V, Vp)). CTA (0, r) also writes
// m, 1/l, argmax and conf = 1/l of row r.
__global__ void __launch_bounds__(256)
finalize_chunks_kernel(const float *__restrict__ z, const float *__restrict__ pm, const int *__restrict__ pa,
                       const float *__restrict__ pl, int chunks, float *__restrict__ m_out,
                       float *__restrict__ inv_l, int32_t *__restrict__ argmax, float *__restrict__ conf,
                       uint16_t *__restrict__ P, int V, int Vp, int slice, const float *__restrict__ z2,
                       long long ld2, int tail_v0) {
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x, r = blockIdx.y;
  __shared__ float s_m;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    float m = -INFINITY, l = 0.f;
    int a = 0x7fffffff;
    for (int k = lane; k < chunks; k += 32)
      merge_stats(m, l, a, pm[r * chunks + k], pl[r * chunks + k], pa[r * chunks + k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      merge_stats(m, l, a, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, l, o),
                  __shfl_xor_sync(0xffffffffu, a, o));
    if (lane == 0) {
      s_m = m;
      if (c == 0) {
        m_out[r] = m;
        inv_l[r] = 1.f / l;
        argmax[r] = a;
        conf[r] = 1.f / l;
      }
    }
  }
  if (!P) return;
  __syncthreads();
  const float mr = s_m;
  const int v0 = c * slice, v1 = min(Vp, v0 + slice);
  for (int v = v0 + threadIdx.x * 8; v < v1; v += blockDim.x * 8) {
    const float4 *src = reinterpret_cast<const float4 *>(z + static_cast<size_t>(r) * Vp + v);
    float4 x0 = src[0], x1 = src[1];
    if (v >= tail_v0) {   // split tail (tail_v0 is a multiple of 128): add the second K half
      const float4 *s2 = reinterpret_cast<const float4 *>(z2 + static_cast<size_t>(r) * ld2 + (v - tail_v0));
      const float4 y0 = s2[0], y1 = s2[1];
      x0 = make_float4(x0.x + y0.x, x0.y + y0.y, x0.z + y0.z, x0.w + y0.w);
      x1 = make_float4(x1.x + y1.x, x1.y + y1.y, x1.z + y1.z, x1.w + y1.w);
    }
    float f[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = (v + e < V) ? __expf(f[e] - mr) : 0.f;
    reinterpret_cast<uint4 *>(P + static_cast<size_t>(r) * Vp + v)[0] = pack8(f);
  }
}

// P[r][v] = bf16(exp(z[r][v] - m[r])) over this CTA's slice of [0, Vp)
// (zero in the pad [V, Vp)), from dz[r][v] = bf16(z[r][v] - q[r][v / 32])
// and the slice maxima q (the logits GEMM's statistics, `slices` per row).
__global__ void __launch_bounds__(256)
finalize_probs_kernel(const uint16_t *__restrict__ dz, const float *__restrict__ q, int slices,
                      const float *__restrict__ m_row, uint16_t *__restrict__ P, int V, int Vp, int slice) {
  pdl_trigger();
  pdl_wait();
  const int c = blockIdx.x, r = blockIdx.y;
  const float mr = m_row[r];
  const int v0 = c * slice, v1 = min(Vp, v0 + slice);
  for (int v = v0 + threadIdx.x * 8; v < v1; v += blockDim.x * 8) {
    const uint4 raw = reinterpret_cast<const uint4 *>(dz + static_cast<size_t>(r) * Vp + v)[0];
    const float off = v < V ? q[static_cast<size_t>(r) * slices + v / 32] - mr : 0.f;
    float f[8];
    unpack8(raw, f);
#pragma unroll
    for (int e = 0; e < 8; ++e) f[e] = (v + e < V) ? __expf(f[e] + off) : 0.f;
    reinterpret_cast<uint4 *>(P + static_cast<size_t>(r) * Vp + v)[0] = pack8(f);
  }
}

// Sum of the P.E vocabulary splits. A CTA covers 32 float4 outputs with 8
// groups of 32 threads; group g adds the splits g, g + 8, ... (independent
// loads in flight), then the 8 group sums are added in shared memory in a
// fixed order.
constexpr int kCombineGroups = 8;

__global__ void __launch_bounds__(256)
pe_combine_kernel(const float *__restrict__ part, float *__restrict__ pe, size_t n4, int splits) {
  pdl_trigger();
  pdl_wait();
  __shared__ float4 acc[kCombineGroups][32];
  const float4 *p4 = reinterpret_cast<const float4 *>(part);
  const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
  const size_t idx = static_cast<size_t>(blockIdx.x) * 32 + lane;
  float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
  if (idx < n4) {
#pragma unroll 4
    for (int s = g; s < splits; s += kCombineGroups) {
      const float4 x = p4[static_cast<size_t>(s) * n4 + idx];
      t.x += x.x; t.y += x.y; t.z += x.z; t.w += x.w;
    }
  }
  acc[g][lane] = t;
  __syncthreads();
  if (g == 0 && idx < n4) {
#pragma unroll
    for (int k = 1; k < kCombineGroups; ++k) {
      const float4 x = acc[k][lane];
      t.x += x.x; t.y += x.y; t.z += x.z; t.w += x.w;
    }
    reinterpret_cast<float4 *>(pe)[idx] = t;
  }
}

// N tile of the head GEMMs: the smallest that holds the rows (narrower tiles
// re-stream W / E per row block; BN = 16 at R = 32 measured 0.50 vs 0.36 ms).
int pick_bn(int R) {
  if (R <= 16) return 16;
  if (R <= 32) return 32;
  if (R <= 64) return 64;
  if (R <= 128) return 128;
  return 256;
}

// Vocabulary splits of the P.E GEMM (units = d tiles x row blocks x splits
// over the SMs): the split count that minimises
//   waves x (K steps per unit) x t_k + splits x (R x d fp32 partials written
//   and read back by pe_combine) / HBM bandwidth,
// t_k ~ 0.37 us being one K step of a unit (its 16 KB slice of E at an SM's
// share of HBM, about the tensor time of a 128 x 256 x 64 step too). Whole
// waves matter: 640 units on 152 SMs run as 5 waves, 448 as 3.
constexpr int kMaxPeSplits = 32;

int pe_splits(int m_tiles, int n_blocks, int k_steps, int R, int d) {
  const long long base = static_cast<long long>(m_tiles) * n_blocks;
  const int sms = sm_budget();
  const int cap = k_steps / 8 > 0 ? (k_steps / 8 < kMaxPeSplits ? k_steps / 8 : kMaxPeSplits) : 1;
  const double t_k = 0.37e-6, per_split = static_cast<double>(R) * d * 8.0 / 6.8e12;
  int best = 1;
  double best_cost = -1.0;
  for (int s = 1; s <= cap; ++s) {
    const int per = (k_steps + s - 1) / s;
    const int s_eff = (k_steps + per - 1) / per;
    const long long waves = (base * s_eff + sms - 1) / sms;
    const double cost = static_cast<double>(waves) * per * t_k + (s_eff > 1 ? s_eff * per_split : 0.0);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = s_eff;
    }
  }
  return best;
}

struct HeadWs {
  size_t z, z2, pm, pa, pl, m, inv_l, P, part, total;
  int Vp, splits, k_per_split;
  long long z2_cols;   // few rows: columns of the split tail's second halves (0: none)
};

// Split-tail columns: at most 128 tiles (a tail is at most half a round of
// CTAs), whatever the GPU.
constexpr int kTailCols = 128 * 128;

HeadWs head_ws_layout(int R, int d, int V, int with_pe, int splits) {
  HeadWs w{};
  w.Vp = (V + 63) / 64 * 64;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  // statistics per row: one per 32-wide vocab slice (many rows) or one per
  // chunk (few rows), whichever layout is larger
  size_t tiles = 4 * ((static_cast<size_t>(V) + 127) / 128);
  if (tiles < static_cast<size_t>(kStatChunks)) tiles = kStatChunks;
  w.z = take(static_cast<size_t>(R) * w.Vp * 4);
  w.z2_cols = R < kFusedStatsRows ? (w.Vp < kTailCols ? w.Vp : kTailCols) : 0;
  w.z2 = take(static_cast<size_t>(R) * w.z2_cols * 4);
  w.pm = take(static_cast<size_t>(R) * tiles * 4);
  w.pa = take(static_cast<size_t>(R) * tiles * 4);
  w.pl = take(static_cast<size_t>(R) * tiles * 4);
  w.m = take(static_cast<size_t>(R) * 4);
  w.inv_l = take(static_cast<size_t>(R) * 4);
  w.splits = splits;
  if (with_pe) {
    w.P = take(static_cast<size_t>(R) * w.Vp * 2);
    w.part = take(static_cast<size_t>(splits) * R * d * 4);
  }
  w.total = off;
  return w;
}

// Upper bound of the P.E split count, independent of the device (workspace
// sizing must not depend on which GPU is current).
int max_pe_splits(int d, int R, int V) {
  (void)d;
  (void)R;
  const int k_steps = (V + 63) / 64;
  return k_steps / 8 > 0 ? (k_steps / 8 < kMaxPeSplits ? k_steps / 8 : kMaxPeSplits) : 1;
}

// Per (row, 32-wide vocab slice) softmax statistics written by the logits GEMM.
struct TileStats {
  float *m, *l;
  int *a;
};

// Few rows: the logits GEMM may split its last round of vocabulary tiles
// into K halves (second halves to z2); v0 is then the first logit column
// with two halves, else INT_MAX.
struct SplitTail {
  float *z2;
  long long cols;
  int v0;
};

template <int BN>
bool launch_head_gemms(const uint16_t *hidden, const uint16_t *w_head, const uint16_t *emb, int R, int d, int V,
                       float *z, int Vp, const uint16_t *P, const float *inv_l, float *part, int splits,
                       bool logits, const TileStats &st, cudaStream_t s, SplitTail *tail) {
  CUtensorMap ta, tb;
  UmmaArgs a{};
  a.status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void **>(&a.status), g_status_head) != cudaSuccess) return false;
  if (logits) {
    if (!make_tmap_bf16_sw128(&ta, w_head, V, d, d, 128)) return false;
    if (!make_tmap_bf16_sw128(&tb, hidden, R, d, d, BN)) return false;
    a.m_tiles = (V + 127) / 128;
    a.n_blocks = (R + BN - 1) / BN;
    a.k_splits = 1;
    a.k_steps = d / 64;
    a.k_per_split = a.k_steps;
    a.M = V;
    a.N = R;
    a.out = z;
    a.ld = Vp;
    a.col_scale = nullptr;
    if (!st.m) {
      // whole rounds of tiles, then the rest split into K halves when that
      // takes at most half a round: every CTA ends after the same work
      const int G = a.m_tiles < sm_budget() ? a.m_tiles : sm_budget();
      const int full = (a.m_tiles / G) * G, t = a.m_tiles - full;
      if (tail && tail->z2 && a.n_blocks == 1 && full > 0 && t > 0 && 2 * t <= G && a.k_steps >= 2 &&
          static_cast<long long>(t) * 128 <= tail->cols) {
        a.out2 = tail->z2;
        a.ld2 = tail->cols;
        a.tail_m0 = full;
        a.full_units = full;
        tail->v0 = full * 128;
      }
      return launch_umma_gemm<BN, false, kEpiStoreT>(ta, tb, a, s);
    }
    a.st_m = st.m;
    a.st_l = st.l;
    a.st_a = st.a;
    a.st_ld = 4 * a.m_tiles;
    if constexpr (BN >= 128) {
      // many rows: the rows (tokens) on M in 256-row pairs, the vocabulary on
      // N in tiles of 256, so that each epilogue thread holds one row and
      // reduces its own 32-column chunks; the logits stored as bf16 relative
      // to their chunk's maximum (z as bf16 [R][Vp])
      constexpr int kVn = 256;
      if (!make_tmap_bf16_sw128(&ta, hidden, R, d, d, 128) || !make_tmap_bf16_sw128(&tb, w_head, V, d, d, kVn / 2))
        return false;
      a.m_tiles = (R + 255) / 256;
      a.n_blocks = (V + kVn - 1) / kVn;
      a.M = R;
      a.N = V;
      a.outb = reinterpret_cast<uint16_t *>(z);
      return launch_umma_pair<kVn, false, kEpiRowStats>(ta, tb, a, s);
    } else {
      return false;   // statistics are fused only at many rows
    }
  }
  if (!make_tmap_bf16_sw128(&ta, emb, V, d, d, 64)) return false;
  if (!make_tmap_bf16_sw128(&tb, P, R, Vp, Vp, BN)) return false;
  a.m_tiles = (d + 127) / 128;
  a.n_blocks = (R + BN - 1) / BN;
  a.k_steps = Vp / 64;
  a.k_per_split = (a.k_steps + splits - 1) / splits;
  a.k_splits = (a.k_steps + a.k_per_split - 1) / a.k_per_split;
  a.M = d;
  a.N = R;
  a.out = part;
  a.ld = d;
  a.col_scale = inv_l;
  if constexpr (BN >= 128) {
    // many rows: 256-wide d tile pairs on CTA pairs
    if (!make_tmap_bf16_sw128(&tb, P, R, Vp, Vp, BN / 2)) return false;
    a.m_tiles = (a.m_tiles + 1) / 2;
    return launch_umma_pair<BN, true, kEpiScaleT>(ta, tb, a, s);
  } else {
    return launch_umma_gemm<BN, true, kEpiScaleT>(ta, tb, a, s);
  }
}

bool head_gemm(int BN, const uint16_t *hidden, const uint16_t *w_head, const uint16_t *emb, int R, int d, int V,
               float *z, int Vp, const uint16_t *P, const float *inv_l, float *part, int splits, bool logits,
               const TileStats &st, cudaStream_t s, SplitTail *tail = nullptr) {
  switch (BN) {
    case 16:
      return launch_head_gemms<16>(hidden, w_head, emb, R, d, V, z, Vp, P, inv_l, part, splits, logits, st, s, tail);
    case 32:
      return launch_head_gemms<32>(hidden, w_head, emb, R, d, V, z, Vp, P, inv_l, part, splits, logits, st, s, tail);
    case 64:
      return launch_head_gemms<64>(hidden, w_head, emb, R, d, V, z, Vp, P, inv_l, part, splits, logits, st, s, tail);
    case 128:
      return launch_head_gemms<128>(hidden, w_head, emb, R, d, V, z, Vp, P, inv_l, part, splits, logits, st, s, tail);
    default:
      return launch_head_gemms<256>(hidden, w_head, emb, R, d, V, z, Vp, P, inv_l, part, splits, logits, st, s, tail);
  }
}

}  // namespace
}  // namespace dllm

using namespace dllm;

extern "C" size_t dllm_head_workspace(int R, int d, int V, int with_pe) {
  if (R < 0 || d < 0 || V < 0) return 0;
  return head_ws_layout(R, d, V, with_pe, max_pe_splits(d, R, V)).total;
}

extern "C" dllm_status dllm_head_confidence(const dllm_bf16 *hidden, const dllm_bf16 *w_head,
                                            const dllm_bf16 *emb, int R, int d, int V, int32_t *argmax,
                                            float *conf, float *pe, void *ws, size_t ws_bytes,
                                            dllm_stream stream) {
  if (R < 0 || d < 1 || V < 1) return DLLM_ERR_INVALID_ARG;
  if (d % 64 != 0 || d > 16384 || R > 4096) return DLLM_ERR_UNSUPPORTED;
  if (R == 0) return DLLM_OK;
  if (!hidden || !w_head || !argmax || !conf) return DLLM_ERR_INVALID_ARG;
  if (pe && !emb) return DLLM_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(w_head) || (emb && !aligned16(emb)) || (pe && !aligned16(pe)))
    return DLLM_ERR_INVALID_ARG;
  const int with_pe = pe != nullptr;
  const HeadWs L0 = head_ws_layout(R, d, V, with_pe, max_pe_splits(d, R, V));
  if (!ws || ws_bytes < L0.total || (reinterpret_cast<uintptr_t>(ws) & 255)) return DLLM_ERR_WORKSPACE;
  const int BN = pick_bn(R);
  const int n_blocks = (R + BN - 1) / BN;
  const int Vp = L0.Vp;
  int splits = pe_splits((d + 127) / 128, n_blocks, Vp / 64, R, d);
  if (splits > L0.splits) splits = L0.splits;
  const HeadWs L = head_ws_layout(R, d, V, with_pe, splits);

  char *base = static_cast<char *>(ws);
  float *z = reinterpret_cast<float *>(base + L.z);
  float *pm = reinterpret_cast<float *>(base + L.pm);
  int *pa = reinterpret_cast<int *>(base + L.pa);
  float *pl = reinterpret_cast<float *>(base + L.pl);
  float *m = reinterpret_cast<float *>(base + L.m);
  float *inv_l = reinterpret_cast<float *>(base + L.inv_l);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  uint16_t *P = with_pe ? reinterpret_cast<uint16_t *>(base + L.P) : nullptr;
  const int slice = ((Vp / kStatChunks + 7) / 8) * 8;   // P pass: multiple of 8 elements per CTA
  const dim3 p_grid((Vp + slice - 1) / slice, R);
  unsigned launches = (R >= kFusedStatsRows && !with_pe) ? 2 : 3;
  if (R >= kFusedStatsRows) {
    // logits + softmax statistics per 32-wide slice of every row,
    // their per-row merge, then P
    const TileStats st{pm, pl, pa};
    if (!head_gemm(BN, hidden, w_head, emb, R, d, V, z, Vp, nullptr, nullptr, nullptr, 1, true, st, s))
      return DLLM_ERR_CUDA;
    if (launch_pdl(stats_combine_kernel, dim3(R), dim3(256), 0, s, static_cast<const float *>(pm),
                   static_cast<const float *>(pl), static_cast<const int *>(pa), 4 * ((V + 127) / 128), m, inv_l,
                   argmax, conf) != cudaSuccess)
      return DLLM_ERR_CUDA;
    if (with_pe && launch_pdl(finalize_probs_kernel, p_grid, dim3(256), 0, s, reinterpret_cast<const uint16_t *>(z),
                              static_cast<const float *>(pm), 4 * ((V + 127) / 128), static_cast<const float *>(m),
                              P, V, Vp, slice) != cudaSuccess)
      return DLLM_ERR_CUDA;
  } else {
    // logits, per-chunk statistics, then their merge (+ P) per row
    SplitTail tail{reinterpret_cast<float *>(base + L.z2), L.z2_cols, 0x7fffffff};
    if (!head_gemm(BN, hidden, w_head, emb, R, d, V, z, Vp, nullptr, nullptr, nullptr, 1, true, TileStats{}, s,
                   &tail))
      return DLLM_ERR_CUDA;
    const float *z2 = tail.z2;
    const int chunk = (V + kStatChunks - 1) / kStatChunks;
    if (launch_pdl(stats_partial_kernel, dim3(kStatChunks, R), dim3(256), 0, s, static_cast<const float *>(z),
                   static_cast<long long>(Vp), V, chunk, pm, pa, pl, z2, tail.cols, tail.v0) != cudaSuccess)
      return DLLM_ERR_CUDA;
    if (launch_pdl(finalize_chunks_kernel, with_pe ? p_grid : dim3(1, R), dim3(with_pe ? 256 : 32), 0, s,
                   static_cast<const float *>(z), static_cast<const float *>(pm), static_cast<const int *>(pa),
                   static_cast<const float *>(pl), static_cast<int>(kStatChunks), m, inv_l, argmax, conf, P, V,
                   Vp, slice, z2, tail.cols, tail.v0) != cudaSuccess)
      return DLLM_ERR_CUDA;
  }
  if (with_pe) {
    float *part = reinterpret_cast<float *>(base + L.part);
    if (!head_gemm(BN, hidden, w_head, emb, R, d, V, z, Vp, P, inv_l, part, splits, false, TileStats{}, s))
      return DLLM_ERR_CUDA;
    const size_t n4 = static_cast<size_t>(R) * d / 4;
    const int g2 = static_cast<int>((n4 + 31) / 32);
    if (launch_pdl(pe_combine_kernel, dim3(g2), dim3(256), 0, s, static_cast<const float *>(part), pe, n4,
                   splits) != cudaSuccess)
      return DLLM_ERR_CUDA;
    launches += 2;
  }
  return launch_status(launches);
}
