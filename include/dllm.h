/*
 * dllm.h -- C ABI of the GB300 (sm_103a) block-decoding denoise step.
 *
 * One denoising iteration of block-cached masked-diffusion LLM decoding:
 *   (a) non-causal attention of the current window (left vicinity + block +
 *       right vicinity) over the cached prefix K/V plus the window's fresh
 *       K/V  [dInfer article, "vicinity KV refresh"; Sangam abstract:
 *       bidirectional attention, approximate KV caching];
 *   (b) the LM head fused with an online vocabulary softmax: argmax token,
 *       largest probability (confidence) and the expected embedding
 *       P.E = sum_v p_v E[v]  [dInfer article, decoding problem 3 and
 *       "iteration smoothing"];
 *   (c) the parallel-decode commit: threshold tau, credit accumulation,
 *       hierarchical centre-first selection, next-step input embeddings
 *       [dInfer article, "hierarchical decoding", "credit decoding",
 *       "iteration smoothing"].
 *
 * Conventions shared by every entry point
 *   - Every pointer argument is a DEVICE pointer owned by the caller unless
 *     its comment says "host". The library never allocates or frees device
 *     memory in these calls; scratch space is the caller's workspace `ws`
 *     of at least the size the matching *_workspace_bytes() returns
 *     (256-byte aligned).
 *   - bf16 data is passed as `dllm_bf16` (the 16-bit bfloat16 pattern).
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Every
 *     call only enqueues work: DLLM_OK means "enqueued". Nothing is
 *     synchronised, so every call may be captured into a CUDA graph.
 *   - Argument errors are detected on the host before anything is
 *     launched (DLLM_ERR_INVALID_ARG / DLLM_ERR_UNSUPPORTED /
 *     DLLM_ERR_WORKSPACE). Data errors only visible on the device (a bad
 *     row map, an out-of-range token id, a bounded wait that ran out) set
 *     bits of a per-device status word instead of trapping; read it with
 *     dllm_get_device_status() after synchronising.
 *   - No C++ exception crosses this boundary. Calls are thread-safe.
 */
#ifndef DLLM_H_
#define DLLM_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t dllm_bf16;   /* IEEE bfloat16 bit pattern */
typedef void *dllm_stream;    /* cudaStream_t */

typedef enum {
  DLLM_OK = 0,
  DLLM_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad offsets ... */
  DLLM_ERR_UNSUPPORTED = 2,   /* a shape outside the supported set           */
  DLLM_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned  */
  DLLM_ERR_CUDA = 4,          /* a CUDA runtime/driver call failed           */
  DLLM_ERR_DEVICE_STATUS = 5  /* the device status word is non-zero          */
} dllm_status;

/* Device status bits (dllm_get_device_status). */
#define DLLM_DEV_ROW_MISSING   0x1   /* a masked position had no head row       */
#define DLLM_DEV_ROW_DUPLICATE 0x2   /* two head rows named one position        */
#define DLLM_DEV_ID_RANGE      0x4   /* a token / argmax id outside [0, V)      */
#define DLLM_DEV_WAIT_TIMEOUT  0x8   /* a bounded device wait gave up           */
#define DLLM_DEV_ROW_RANGE     0x10  /* a row map entry outside [0,B) x [0,blk) */
#define DLLM_DEV_OFFSETS       0x20  /* q_off / kv_off beyond the given buffers  */

/* Decoding-strategy parameters (host struct, passed by pointer).
 *  tau          confidence threshold: commit when p >= tau
 *  lambda_      credit decay: credit <- lambda_*credit + p while the argmax
 *               is unchanged; on a change (or no history, prev = -1)
 *               credit <- p
 *  kappa        credit threshold: commit when credit >= kappa (may be +inf)
 *  hierarchical 1 = centre-first recursive bisection of each masked span,
 *               0 = commit every candidate
 *  hier_levels  recursion depth of the bisection (>= 1); levels >= blk
 *               selects every candidate
 *  smoothing    1 = still-masked positions get E[mask_id] + alpha*P.E as
 *               next input, 0 = E[mask_id]
 *  alpha        smoothing weight
 *  mask_id      token id of the mask token, in [0, V)                         */
typedef struct {
  float tau;
  float lambda_;
  float kappa;
  int hierarchical;
  int hier_levels;
  int smoothing;
  float alpha;
  int mask_id;
} dllm_params;

/* ---------------------------------------------------------------------
 * dllm_block_attn -- non-causal attention of window queries over
 * cached prefix + fresh window keys (dInfer article, "vicinity KV
 * refresh"; Sangam abstract, bidirectional attention).
 *
 *   For request i, head h, query row t in [q_off[i], q_off[i+1]):
 *     O[t,h,:] = sum_u softmax_u(scale * <q[t,h,:], k[u,h,:]>) v[u,h,:]
 *   over every key row u in [kv_off[i], kv_off[i+1]) -- no mask. By
 *   convention the first P_i of those rows are the cached prefix and the
 *   last W_i = q_off[i+1]-q_off[i] are the freshly computed window.
 *
 *   q      bf16 [sum W][H][dh], row stride H*dh (token-major)
 *   k, v   bf16 [sum L][H][dh], same layout
 *   out    [sum W][H][dh]: bf16 (out_fp32 = 0) or float (out_fp32 = 1)
 *   q_off, kv_off  int32 [B+1] on the device, non-decreasing, q_off[0] =
 *          kv_off[0] = 0; rows of a request are contiguous
 *   max_q, max_kv  host upper bounds of W_i and L_i (grid and split
 *          sizing); the part of a request beyond its bound is not processed
 *   q_rows, kv_rows  rows allocated in q/out and in k/v; rows named by the
 *          offsets beyond them are clipped (DLLM_DEV_OFFSETS), never read
 *   scale  softmax scale (normally 1/sqrt(dh))
 *   A request with queries but no keys gets zeros.
 *   Supported: dh in {64, 128}; H >= 1; B <= 4096.
 *   dllm_block_attn_workspace(B, H, dh, max_q, max_kv) bytes serve every
 *   call with these B, H, dh and any max_q' <= max_q, max_kv' <= max_kv, on
 *   any GPU (at most 256 x 128 partial rows: a few MB).
 * ------------------------------------------------------------------- */
size_t dllm_block_attn_workspace(int B, int H, int dh, int max_q, int max_kv);
dllm_status dllm_block_attn(const dllm_bf16 *q, const dllm_bf16 *k,
                            const dllm_bf16 *v, void *out, int out_fp32,
                            const int32_t *q_off, const int32_t *kv_off,
                            int B, int H, int dh, int max_q, int max_kv,
                            int q_rows, int kv_rows, float scale, void *ws,
                            size_t ws_bytes, dllm_stream stream);

/* ---------------------------------------------------------------------
 * dllm_head_confidence -- LM head with the online vocabulary softmax and
 * the expected embedding for iteration smoothing (dInfer article,
 * decoding problem 3 and "iteration smoothing").
 *
 *   z[r,v]   = <hidden[r,:], w_head[v,:]>        (fp32 accumulation)
 *   argmax[r]= lowest v with z[r,v] = max_v z[r,v]
 *   conf[r]  = 1 / sum_v exp(z[r,v] - max z[r,:])   (largest probability)
 *   pe[r,:]  = sum_v softmax(z[r,:])_v * emb[v,:]   (only if pe != NULL)
 *
 *   hidden bf16 [R][d]; w_head, emb bf16 [V][d] (row = vocabulary entry)
 *   argmax int32 [R]; conf float [R]; pe float [R][d] or NULL (then emb
 *   may be NULL). Supported: d % 64 == 0, 64 <= d <= 16384, 1 <= V,
 *   1 <= R <= 4096.
 * ------------------------------------------------------------------- */
size_t dllm_head_workspace(int R, int d, int V, int with_pe);
dllm_status dllm_head_confidence(const dllm_bf16 *hidden,
                                 const dllm_bf16 *w_head,
                                 const dllm_bf16 *emb, int R, int d, int V,
                                 int32_t *argmax, float *conf, float *pe,
                                 void *ws, size_t ws_bytes,
                                 dllm_stream stream);

/* ---------------------------------------------------------------------
 * dllm_head_confidence_noalloc -- the same head, for callers that cannot
 * allocate device memory. No passage of the pages has a counterpart: this
 * is an interface for callers such as a plugin whose host framework owns
 * all device memory and gives it no allocator, or a thread that must not
 * block (cudaMalloc can synchronise the device), which can neither call
 * cudaMalloc nor hold a workspace of their own.
 *
 *   Arguments, layouts and results are those of dllm_head_confidence
 *   without ws / ws_bytes. The scratch is a fixed device array of
 *   DLLM_HEAD_NOALLOC_SCRATCH_BYTES inside the library, reserved on every
 *   GPU that loads the library until the process exits; the call never
 *   calls cudaMalloc / cudaFree or any allocating routine.
 *   - Sizes whose workspace (dllm_head_workspace) exceeds the array are
 *     rejected with DLLM_ERR_UNSUPPORTED before anything is launched
 *     (R = 32 rows at d = 4096, V = 126464 with P.E fit).
 *   - The first call on each device looks the array's device address up
 *     (cudaGetSymbolAddress); make that first call before any stream
 *     capture on that device. The look-up is repeated when the device's
 *     context has changed (e.g. after cudaDeviceReset, which reloads the
 *     library's module); make the first call after such a reset outside
 *     stream capture too.
 *   - All calls share the array and it keeps the last call's contents;
 *     nothing in it has to start at zero. Calls whose GPU work overlaps
 *     (several streams or host threads) race on it: serialise them.
 * ------------------------------------------------------------------- */
#define DLLM_HEAD_NOALLOC_SCRATCH_BYTES (48u << 20)
dllm_status dllm_head_confidence_noalloc(const dllm_bf16 *hidden,
                                         const dllm_bf16 *w_head,
                                         const dllm_bf16 *emb, int R, int d,
                                         int V, int32_t *argmax, float *conf,
                                         float *pe, dllm_stream stream);

/* ---------------------------------------------------------------------
 * dllm_commit -- the parallel-decode commit of one step (dInfer article,
 * "credit decoding", "hierarchical decoding", "iteration smoothing").
 *
 *   Head row r in [0, R) belongs to request row_req[r], block position
 *   row_pos[r]. Rows at positions that are not masked are ignored. Every
 *   masked position needs exactly one row (else DLLM_DEV_ROW_MISSING /
 *   DLLM_DEV_ROW_DUPLICATE and that request is left unchanged).
 *   Per request i, over its masked positions j (mask[i][j] = 1):
 *     1. credit: if prev[i][j] == argmax: credit <- lambda_*credit + p
 *        (float32 product, then float32 sum), else credit <- p; then
 *        prev <- argmax                         (p = conf of the row)
 *     2. candidates: p >= tau or credit >= kappa
 *     3. selection: all candidates (hierarchical = 0), or per maximal run
 *        [l, r) of masked positions HS(l, r, hier_levels): the candidate
 *        nearest c = l + (r-l-1)/2 (ties: higher p, then lower position),
 *        plus HS on both sides with one level less
 *     4. if nothing is selected, the masked position with the highest p
 *        (lowest position on ties) is
 *     5. selected: tokens <- argmax, mask <- 0, credit <- 0, prev <- -1
 *   next_emb[i][j][:] (bf16) = emb[tokens] for committed positions, and
 *   emb[mask_id] + alpha*pe[row] (smoothing) or emb[mask_id] for the
 *   positions still masked. n_commit[i] = number committed now.
 *
 *   mask uint8 [B][blk]; tokens, prev_argmax int32 [B][blk]; credit float
 *   [B][blk] -- all updated in place. argmax int32 [R], conf float [R],
 *   pe float [R][d] (may be NULL when smoothing = 0), emb bf16 [V][d],
 *   next_emb bf16 [B][blk][d], n_commit int32 [B]. params: host pointer.
 *   Supported: 1 <= blk <= 64, B <= 4096, d % 8 == 0.
 *   One launch of blk x B CTAs; the state is written by each request's last
 *   CTA, found with an arrival count in library memory. Each call takes the
 *   next of 32 count slots, so up to 32 calls may run at once on a device
 *   (on any streams); a call captured in a CUDA graph keeps its slot at
 *   every replay, so graphs whose commits were captured a multiple of 32
 *   calls apart must not run at the same time.
 * ------------------------------------------------------------------- */
dllm_status dllm_commit(const int32_t *argmax, const float *conf,
                        const float *pe, const int32_t *row_req,
                        const int32_t *row_pos, int R, int B, int blk,
                        uint8_t *mask, int32_t *tokens, float *credit,
                        int32_t *prev_argmax, const dllm_bf16 *emb, int V,
                        int d, dllm_bf16 *next_emb, int32_t *n_commit,
                        const dllm_params *params, dllm_stream stream);

/* ---------------------------------------------------------------------
 * dllm_denoise_step -- attention, head and commit of one step enqueued
 * back to back on one stream with no host synchronisation (the serving
 * study's finding that host dispatch dominates a single request's wall
 * time is why the three run as one enqueue and capture as one graph).
 * Field meanings are those of the three calls above; `attn_out` may be
 * NULL to skip the attention (then q, k, v, offsets are unused).
 * ------------------------------------------------------------------- */
typedef struct {
  /* attention */
  const dllm_bf16 *q, *k, *v;
  void *attn_out;
  int attn_out_fp32;
  const int32_t *q_off, *kv_off;
  int H, dh, max_q, max_kv, q_rows, kv_rows;
  float scale;
  /* head */
  const dllm_bf16 *hidden, *w_head, *emb;
  int R, d, V;
  int32_t *argmax;
  float *conf, *pe;
  /* commit */
  const int32_t *row_req, *row_pos;
  int B, blk;
  uint8_t *mask;
  int32_t *tokens;
  float *credit;
  int32_t *prev_argmax;
  dllm_bf16 *next_emb;
  int32_t *n_commit;
  dllm_params params;
} dllm_step_args;

size_t dllm_denoise_step_workspace(const dllm_step_args *args /* host */);
dllm_status dllm_denoise_step(const dllm_step_args *args /* host */,
                              void *ws, size_t ws_bytes, dllm_stream stream);

/* Workspace bytes by shape alone (the same sizes as the per-call functions
 * above), which = DLLM_WS_ATTN: dllm_block_attn(B, H, dh, max_q, max_kv);
 * DLLM_WS_HEAD / DLLM_WS_HEAD_PE: dllm_head_confidence(R, d, V) without /
 * with P.E; DLLM_WS_STEP: dllm_denoise_step with attention and P.E. Unused
 * arguments are ignored; 0 for an unknown `which` or an unsupported shape. */
enum { DLLM_WS_ATTN = 0, DLLM_WS_HEAD = 1, DLLM_WS_HEAD_PE = 2, DLLM_WS_STEP = 3 };
size_t dllm_workspace_bytes(int which, int B, int H, int dh, int max_q,
                            int max_kv, int R, int d, int V);

/* ---------------------------------------------------------------------
 * dllm_gemm_bf16 -- C[M][N] = A[M][K] . W[N][K]^T on tcgen05 (bf16 in,
 * fp32 accumulate, bf16 out), the projection GEMM of the end-to-end model.
 *   epilogue 0: C = A W^T
 *   epilogue 1: C = A W^T + aux          (aux [M][N], may alias C)
 *   epilogue 2: C = silu(A Wg^T) * (A Wu^T), W = [2N][K] with the gate rows
 *               first, then the up rows (SwiGLU)
 *   All row-major. Supported: K % 64 == 0, N % 16 == 0 (N % 64 == 0 for
 *   SwiGLU), M <= 65536. No workspace.
 * ------------------------------------------------------------------- */
dllm_status dllm_gemm_bf16(const dllm_bf16 *A, const dllm_bf16 *W, dllm_bf16 *C,
                           int M, int N, int K, int epilogue,
                           const dllm_bf16 *aux, dllm_stream stream);

/* ---------------------------------------------------------------------
 * End-to-end block decoding with a small bidirectional transformer
 * (Sangam abstract: block-sized decodes, approximate K/V caching with
 * recurring prefills; dInfer article, "vicinity KV refresh").
 *
 * Layer (pre-norm): h = RMSNorm(x) (weight 1, eps rms_eps); q,k,v = h Wqkv^T
 * (Wqkv [3d][d]: q rows, k rows, v rows); RoPE on q and k (pairs (i, i+dh/2),
 * angle pos * rope_base^(-2i/dh), pos = absolute position); non-causal
 * attention over the cache rows [0, L); x += o Wo^T; x += SwiGLU FFN
 * (Wgu [2 ffn][d] gate rows then up rows, Wdown [d][ffn]); final RMSNorm.
 * Activations are bf16 between kernels.
 * ------------------------------------------------------------------- */
typedef struct {
  int layers, d, H, dh, ffn, V;
  int max_seq;                   /* rows of every K/V cache buffer          */
  float rms_eps, rope_base;
  const dllm_bf16 *emb;          /* [V][d] input embeddings                 */
  const dllm_bf16 *w_head;       /* [V][d] LM head (untied)                 */
  /* host arrays of `layers` device pointers */
  const dllm_bf16 *const *wqkv;  /* [3d][d]   */
  const dllm_bf16 *const *wo;    /* [d][d]    */
  const dllm_bf16 *const *wgu;   /* [2ffn][d] */
  const dllm_bf16 *const *wdown; /* [d][ffn]  */
} dllm_model;

/* dllm_model_forward: all layers over n input rows x_in [n][d] at positions
 * pos0 .. pos0+n-1. Each layer writes its K/V of these rows into rows
 * pos0.. of k_cache[l] / v_cache[l] ([max_seq][H][dh], host arrays of
 * device pointers) and attends over cache rows [0, pos0 + n): the cached
 * prefix plus these rows. hidden_out [n][d] = final-normed rows. */
size_t dllm_model_forward_workspace(const dllm_model *m, int n);
dllm_status dllm_model_forward(const dllm_model *m, const dllm_bf16 *x_in,
                               int n, int pos0, dllm_bf16 *const *k_cache,
                               dllm_bf16 *const *v_cache,
                               dllm_bf16 *hidden_out, void *ws,
                               size_t ws_bytes, dllm_stream stream);

/* State of the block decode loop of one request (all device buffers except
 * the host arrays k_cache / v_cache). Sequence: T = prompt_len + response
 * positions; block b covers [prompt_len + b*blk, +blk). */
typedef struct {
  int T, prompt_len, blk, vic;
  int32_t *tokens;               /* [T] token ids (mask_id where masked)    */
  uint8_t *masked;               /* [T] 1 = masked                          */
  dllm_bf16 *const *k_cache;     /* per layer [max_seq][H][dh]              */
  dllm_bf16 *const *v_cache;
  uint8_t *bmask;                /* [blk] block state, as in dllm_commit    */
  int32_t *btokens, *bprev;      /* [blk]                                   */
  float *bcredit;                /* [blk]                                   */
  dllm_bf16 *bnext_emb;          /* [blk][d] next-step input of the block   */
  int32_t *n_commit;             /* [1]                                     */
  int32_t *argmax;               /* [blk] head outputs of the last step     */
  float *conf;                   /* [blk]                                   */
  float *pe;                     /* [blk][d], needed when smoothing         */
  dllm_bf16 *hidden;             /* [blk][d] final-normed block rows, or NULL */
  dllm_params params;
  int eos_id;                    /* token ending the response, or -1: the
                                    decode graph skips the blocks after a
                                    block that committed it               */
  int dual_cache;                /* 0: window steps attend over the cached
                                    prefix + the window; 1: also over the
                                    cached rows right of the window (kept
                                    from the block's refresh), i.e. over
                                    cache rows [0, T)                      */
} dllm_decode_state;

/* dllm_decode_step: one denoise step of block `block`.
 *   refresh = 1: input rows for every position (committed tokens -> E[t],
 *     masked -> E[mask_id]) run through all layers, refreshing the whole
 *     K/V cache (the per-block recurring prefill); the block rows feed the
 *     head and the commit -- the block's first step. Call it at the start
 *     of a block, with the block state reset (all masked, credit 0,
 *     prev -1).
 *   refresh = 0: only the window [b0 - vic, b0 + blk + vic) (clipped to
 *     [0, T)) runs, its input rows being E[token] / bnext_emb (block) /
 *     E[mask_id]; keys = cache rows [0, window end), or [0, T) with
 *     dual_cache (prefix and suffix caches: the rows right of the window
 *     keep the K/V of the block's refresh; only the window's rows are
 *     rewritten). Masked-diffusion caching reuses K/V on both sides of the
 *     block between refreshes (dInfer article, vicinity KV refresh).
 *   Then head (argmax, conf, P.E), commit (dllm_commit semantics on the
 *   block state) and the write-back of the block's tokens / mask into the
 *   sequence. Host reads nothing; *n_commit tells the caller the progress. */
size_t dllm_decode_step_workspace(const dllm_model *m,
                                  const dllm_decode_state *st);
dllm_status dllm_decode_step(const dllm_model *m, const dllm_decode_state *st,
                             int block, int refresh, void *ws,
                             size_t ws_bytes, dllm_stream stream);

/* ---------------------------------------------------------------------
 * dllm_decode_graph_* -- the whole block decode loop of one request as one
 * CUDA graph, launched with no host round trip between steps (dInfer
 * article, system optimisations: loop unrolling removes the bubbles between
 * iterations; early stop after the end-of-sequence token). Per block b:
 * an IF node, taken while no committed response position before the block
 * holds eos_id, containing the block-state reset, the refresh step, and a
 * WHILE node of window steps whose condition a kernel sets after every
 * step to "a position of the block is still masked" (at most blk steps).
 *   create: records the pointers and sizes in m, st and ws (keep them valid
 *           and unchanged while the graph exists) and instantiates the
 *           graph -- a set-up call that creates CUDA objects; not for
 *           stream capture. launch: enqueues one whole decode on `stream`
 *           (tokens/masked must hold the prompt / masked response first).
 * ------------------------------------------------------------------- */
typedef struct dllm_decode_graph_s *dllm_decode_graph;
dllm_status dllm_decode_graph_create(const dllm_model *m,
                                     const dllm_decode_state *st, void *ws,
                                     size_t ws_bytes, dllm_decode_graph *out);
dllm_status dllm_decode_graph_launch(dllm_decode_graph g, dllm_stream stream);
dllm_status dllm_decode_graph_destroy(dllm_decode_graph g);

/* ---------------------------------------------------------------------
 * dllm_moe_ffn -- the mixture-of-experts FFN of a LLaDA-MoE-like block
 * (dInfer abstract: LLaDA-MoE; TIDE abstract: MoE dLLMs and their expert
 * activations), with top-k routing:
 *   z[t][e]   = h[t] . w_router[e]                      (fp32 accumulate)
 *   chosen    = the topk experts of largest z[t] (ties: lower index),
 *               highest first -> topk_ids[t][0..topk)
 *   weight    = exp(z - z_max) / sum over the chosen    -> topk_w[t][..]
 *               (the softmax probabilities renormalised over the chosen)
 *   expert e  = (silu(h W1_e^T) * (h W3_e^T)) W2_e^T
 *   out[t]    = sum_j weight[t][j] * expert_{chosen j}(h[t])
 *
 *   h        bf16 [n][d] (the normed rows entering the FFN)
 *   w_router bf16 [E][d]
 *   w13      bf16 [E][2F][d]: per expert its F gate rows (W1), then its F
 *            up rows (W3)
 *   w2       bf16 [E][d][F]
 *   out      [n][d] float (out_fp32 = 1) or bf16
 *   topk_ids int32 [n][topk], topk_w float [n][topk]: written (may be NULL
 *            -- then kept in the workspace)
 * The expert activations between the two expert GEMMs are rounded to bf16;
 * the expert outputs and the weighted sum are fp32. The host reads nothing
 * back: the expert-sorted order is built on the device. The order of a
 * token's rows inside its expert's segment may change from call to call;
 * the outputs do not (bitwise repeatable for the same inputs and GPU).
 * Supported: d, F multiples of 128, d <= 8192; 1 <= E <= 256;
 * 1 <= topk <= min(E, 16); n * topk <= 65536; pointers 16-byte aligned.
 * ------------------------------------------------------------------- */
size_t dllm_moe_ffn_workspace(int n, int d, int E, int F, int topk);
dllm_status dllm_moe_ffn(const dllm_bf16 *h, const dllm_bf16 *w_router,
                         const dllm_bf16 *w13, const dllm_bf16 *w2, int n,
                         int d, int E, int F, int topk, void *out,
                         int out_fp32, int32_t *topk_ids, float *topk_w,
                         void *ws, size_t ws_bytes, dllm_stream stream);

/* ---------------------------------------------------------------------
 * Status helpers.
 * ------------------------------------------------------------------- */
const char *dllm_status_string(dllm_status s);
/* Reads (and with clear != 0 also clears) the status word of the current
 * device. Synchronous: call after the work in question has finished. */
dllm_status dllm_get_device_status(int32_t *host_out, int clear);
/* Name of the CUDA runtime error behind the last DLLM_ERR_CUDA that this
 * host thread got from the library (e.g. "cudaErrorInvalidValue"), or NULL
 * when none was recorded (a failed tensor-map encoding records none).
 * Reading it clears it. */
const char *dllm_last_cuda_error(void);
/* Library version, for a loaded-library check. */
int dllm_version(void);
/* Number of kernels this library has enqueued since it was loaded (all
 * devices, all threads): a host-side counter, for launch accounting. */
uint64_t dllm_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* DLLM_H_ */
