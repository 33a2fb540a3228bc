// C-ABI glue: status strings, the device status word, and the composed
// denoise step (attention -> head -> commit on one stream, no host sync).
#include <atomic>

#include "common.cuh"

namespace dllm {
static std::atomic<uint64_t> g_launches{0};
void count_launches(unsigned n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
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

extern "C" dllm_status dllm_denoise_step(const dllm_step_args *a, void *ws, size_t ws_bytes,
                                         dllm_stream stream) {
  if (!a) return DLLM_ERR_INVALID_ARG;
  const StepWs L = step_ws_layout(a);
  if (L.total > 0 && (!ws || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(ws) & 255)))
    return DLLM_ERR_WORKSPACE;
  char *base = static_cast<char *>(ws);
  dllm_status st;
  if (a->attn_out) {
    st = dllm_block_attn(a->q, a->k, a->v, a->attn_out, a->attn_out_fp32, a->q_off, a->kv_off,
                         a->B, a->H, a->dh, a->max_q, a->max_kv, a->q_rows, a->kv_rows, a->scale,
                         base ? base + L.attn : nullptr, L.head - L.attn, stream);
    if (st != DLLM_OK) return st;
  }
  st = dllm_head_confidence(a->hidden, a->w_head, a->emb, a->R, a->d, a->V, a->argmax, a->conf,
                            a->pe, base ? base + L.head : nullptr, L.total - L.head, stream);
  if (st != DLLM_OK) return st;
  return dllm_commit(a->argmax, a->conf, a->pe, a->row_req, a->row_pos, a->R, a->B, a->blk,
                     a->mask, a->tokens, a->credit, a->prev_argmax, a->emb, a->V, a->d,
                     a->next_emb, a->n_commit, &a->params, stream);
}
