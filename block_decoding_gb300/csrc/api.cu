// C-ABI glue: status strings, the device status word, and the composed
// denoise step (attention, head -> commit, no host sync).
#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "common.cuh"
#include "umma.cuh"

namespace dllm {
static std::atomic<uint64_t> g_launches{0};
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

void prefer_max_shared(const void *kern) {
  static std::mutex mu;
  static std::set<std::pair<int, const void *>> done;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  std::lock_guard<std::mutex> lock(mu);
  if (done.insert({dev, kern}).second)
    cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
}
}  // namespace dllm

using namespace dllm;

namespace {

struct StepWs {
  size_t attn, head, total;
};

StepWs step_ws_layout(const dllm_step_args *a) {
  StepWs w{};
  const size_t sa = a->attn_out ? dllm_block_attn_workspace(a->B, a->H, a->dh, a->max_q, a->max_kv) : 0;
  const size_t sh = dllm_head_workspace(a->R, a->d, a->V, a->pe != nullptr);
  w.attn = 0;
  w.head = align256(sa);
  w.total = w.head + align256(sh);
  return w;
}

// A second stream per (host thread, device) for the attention of a step,
// which no later stage of the step reads: it runs beside the head on the
// SMs the head leaves free. Created outside stream capture only.
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
  bool ok = false;
  ~SideStream() {   // host thread exit (errors ignored: the context may be gone)
    if (join) cudaEventDestroy(join);
    if (fork) cudaEventDestroy(fork);
    if (s) cudaStreamDestroy(s);
  }
};

SideStream *side_stream(bool may_create) {
  thread_local SideStream per[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream &x = per[dev];
  if (!x.ok && may_create) {
    if (!x.s && cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking) != cudaSuccess) x.s = nullptr;
    if (!x.fork && cudaEventCreateWithFlags(&x.fork, cudaEventDisableTiming) != cudaSuccess) x.fork = nullptr;
    if (!x.join && cudaEventCreateWithFlags(&x.join, cudaEventDisableTiming) != cudaSuccess) x.join = nullptr;
    x.ok = x.s && x.fork && x.join;
  }
  return x.ok ? &x : nullptr;
}

}  // namespace

extern "C" const char *dllm_status_string(dllm_status s) {
  switch (s) {
    case DLLM_OK: return "ok";
    case DLLM_ERR_INVALID_ARG: return "invalid argument";
    case DLLM_ERR_UNSUPPORTED: return "unsupported shape";
    case DLLM_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    case DLLM_ERR_CUDA: return "CUDA error";
    case DLLM_ERR_DEVICE_STATUS: return "device status word is set";
  }
  return "unknown status";
}

namespace dllm {
namespace {
thread_local cudaError_t t_last_cuda_error = cudaSuccess;
}  // namespace

dllm_status cuda_error(cudaError_t e) {
  t_last_cuda_error = e;
  return DLLM_ERR_CUDA;
}
}  // namespace dllm

extern "C" const char *dllm_last_cuda_error(void) {
  const cudaError_t e = t_last_cuda_error;
  t_last_cuda_error = cudaSuccess;
  return e == cudaSuccess ? nullptr : cudaGetErrorName(e);
}

extern "C" int dllm_version(void) { return 1; }

extern "C" uint64_t dllm_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

extern "C" dllm_status dllm_get_device_status(int32_t *host_out, int clear) {
  if (!host_out) return DLLM_ERR_INVALID_ARG;
  const bool c = clear != 0;
  const uint32_t v = status_attn(c) | status_head(c) | status_commit(c) | status_model(c) | status_moe(c);
  *host_out = static_cast<int32_t>(v);
  if (v & 0x80000000u) return DLLM_ERR_CUDA;
  return v ? DLLM_ERR_DEVICE_STATUS : DLLM_OK;
}

extern "C" size_t dllm_denoise_step_workspace(const dllm_step_args *a) {
  if (!a) return 0;
  return step_ws_layout(a).total;
}

extern "C" size_t dllm_workspace_bytes(int which, int B, int H, int dh, int max_q, int max_kv, int R, int d,
                                       int V) {
  switch (which) {
    case DLLM_WS_ATTN: return dllm_block_attn_workspace(B, H, dh, max_q, max_kv);
    case DLLM_WS_HEAD: return dllm_head_workspace(R, d, V, 0);
    case DLLM_WS_HEAD_PE: return dllm_head_workspace(R, d, V, 1);
    case DLLM_WS_STEP: {
      dllm_step_args a{};
      a.attn_out = reinterpret_cast<void *>(1);   // shape only: never dereferenced
      a.pe = reinterpret_cast<float *>(1);
      a.B = B;
      a.H = H;
      a.dh = dh;
      a.max_q = max_q;
      a.max_kv = max_kv;
      a.R = R;
      a.d = d;
      a.V = V;
      return step_ws_layout(&a).total;
    }
    default: return 0;
  }
}

extern "C" dllm_status dllm_denoise_step(const dllm_step_args *a, void *ws, size_t ws_bytes,
                                         dllm_stream stream) {
  if (!a) return DLLM_ERR_INVALID_ARG;
  const StepWs L = step_ws_layout(a);
  if (L.total > 0 && (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)))
    return DLLM_ERR_WORKSPACE;
  char *base = static_cast<char *>(ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  auto attention = [&](cudaStream_t on) {
    return dllm_block_attn(a->q, a->k, a->v, a->attn_out, a->attn_out_fp32, a->q_off, a->kv_off, a->B, a->H,
                           a->dh, a->max_q, a->max_kv, a->q_rows, a->kv_rows, a->scale,
                           base ? base + L.attn : nullptr, L.head - L.attn, on);
  };
  auto head_commit = [&]() {
    dllm_status st = dllm_head_confidence(a->hidden, a->w_head, a->emb, a->R, a->d, a->V, a->argmax, a->conf,
                                          a->pe, base ? base + L.head : nullptr, L.total - L.head, stream);
    if (st != DLLM_OK) return st;
    return dllm_commit(a->argmax, a->conf, a->pe, a->row_req, a->row_pos, a->R, a->B, a->blk, a->mask, a->tokens,
                       a->credit, a->prev_argmax, a->emb, a->V, a->d, a->next_emb, a->n_commit, &a->params, stream);
  };
  // The attention output feeds no later stage of the step. When one CTA per
  // (request, head, query tile) needs at most a quarter of the SMs, the
  // attention runs on a second stream beside the head, planned for exactly
  // those SMs (no key splits to merge), while the head's persistent GEMMs
  // leave them free. (The head needs about three quarters of the SMs to keep
  // HBM saturated: with 88 of 152 it measured 25 % slower.)
  const int sms = num_sms();
  const int attn_ctas = a->attn_out ? attn_base_ctas(a->B, a->H, a->dh, a->max_q) : 0;
  SideStream *side = nullptr;
  if (attn_ctas > 0 && attn_ctas * 4 <= sms) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) == cudaSuccess) side = side_stream(cap == cudaStreamCaptureStatusNone);
  }
  if (!side) {
    if (a->attn_out) {
      const dllm_status st = attention(s);
      if (st != DLLM_OK) return st;
    }
    return head_commit();
  }
  if (cudaEventRecord(side->fork, s) != cudaSuccess || cudaStreamWaitEvent(side->s, side->fork, 0) != cudaSuccess)
    return DLLM_ERR_CUDA;
  dllm_status sa;
  {
    SmBudget budget(attn_ctas);
    sa = attention(side->s);
  }
  // join even after a failed launch, so that a stream capture stays well formed
  const bool rec = cudaEventRecord(side->join, side->s) == cudaSuccess;
  dllm_status sh;
  {
    SmBudget budget(sms - attn_ctas);
    sh = head_commit();
  }
  const bool joined = rec && cudaStreamWaitEvent(s, side->join, 0) == cudaSuccess;
  if (sa != DLLM_OK) return sa;
  if (sh != DLLM_OK) return sh;
  return joined ? DLLM_OK : DLLM_ERR_CUDA;
}
