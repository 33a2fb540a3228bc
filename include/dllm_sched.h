/* dllm_sched.h -- step-level scheduler of cached block decoding (host code).
 *
 * Cached masked-diffusion decoding repeats a prefill/decode structure per
 * request: every block starts with a refresh of the whole sequence's K/V
 * (an indivisible prefill: bidirectional attention rules out chunking it)
 * and is then decoded, one denoising step at a time, over a window around
 * the block (Sangam abstract; dInfer article, "vicinity KV refresh"). The
 * serving study asks for scheduling at the granularity of one denoising
 * step, with admission and eviction between steps (serving study, design
 * principles). This scheduler decides, before every step, which resident
 * requests decode and which prefills are admitted, under a deficit token
 * budget: in-flight decodes first, whole prefills only when the
 * accumulated budget allows, unused budget carried into the next step
 * (Sangam abstract).
 *
 * Rules (one step = one scheduling cycle):
 *   budget      deficit policy: D <- min(budget_cap, D + quantum);
 *               no_carry: D <- quantum; prefill_first: no budget.
 *   decodes     every resident request whose block is in progress runs,
 *               in slot order, and is charged its query rows: the window
 *               [b0 - vic, b0 + blk + vic) clipped to [0, T). D may go
 *               negative (the decodes are protected; prefills wait).
 *   prefills    one FIFO queue (new requests in submission order; a
 *               resident request joins it when its block is done and
 *               another remains). Scanned in order: a new request that
 *               needs a slot when none is free is passed over; the first
 *               one whose cost (T rows) exceeds D, or the step's row cap,
 *               ends the scan. Admitted prefills are charged T.
 *   conserving  a step that would run nothing admits the first
 *               slot-feasible prefill regardless of the budget.
 *   eviction    a request leaves (its slot is freed) when its last block
 *               is done, or when a block holding its end token is done.
 * The prefill step of block b is the block's first denoising step (the
 * refresh's block rows feed the head and the commit), so an admitted
 * request decodes from the next step on.
 *
 * All functions are host-only and thread-compatible (one thread per
 * scheduler object); none touches the GPU.
 */
#ifndef DLLM_SCHED_H
#define DLLM_SCHED_H

#include <stdint.h>

#include "dllm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dllm_sched dllm_sched; /* opaque */

enum {
  DLLM_SCHED_DEFICIT = 0,       /* carried deficit budget (Sangam)          */
  DLLM_SCHED_PREFILL_FIRST = 1, /* every ready prefill that fits the cap    */
  DLLM_SCHED_NO_CARRY = 2       /* budget reset to quantum every step       */
};

typedef struct {
  int slots;         /* resident requests at most (block-state / cache slots) */
  int blk, vic;      /* block size and vicinity of the window               */
  int quantum;       /* query rows of budget added per step, >= 0            */
  int budget_cap;    /* ceiling of the carried budget, >= quantum            */
  int max_step_rows; /* query rows one step may run, >= slots*(blk+2*vic)
                        and >= max_seq                                      */
  int max_seq;       /* longest request (prompt + response)                 */
  int policy;        /* DLLM_SCHED_*                                         */
  int dual_cache;    /* decodes attend over the whole sequence              */
} dllm_sched_config;

/* One request's part of a step. kind 0 = decode of block `block`: query
 * rows [q_pos0, q_pos0 + q_rows) of the sequence, keys [0, kv_rows).
 * kind 1 = prefill of block `block`: every position (q_pos0 = 0,
 * q_rows = kv_rows = T). b0 = first sequence position of the block. */
typedef struct {
  int slot, req, block, kind, q_pos0, q_rows, kv_rows, b0;
} dllm_sched_entry;

/* Validates cfg (DLLM_ERR_INVALID_ARG) and returns a new scheduler. */
dllm_status dllm_sched_create(const dllm_sched_config *cfg, dllm_sched **out);
void dllm_sched_destroy(dllm_sched *s);

/* Queues request `req` (unique id >= 0). DLLM_ERR_INVALID_ARG if the id is
 * taken, resp_len is not a positive multiple of blk, prompt_len < 0 or
 * prompt_len + resp_len > max_seq. */
dllm_status dllm_sched_submit(dllm_sched *s, int req, int prompt_len,
                              int resp_len);

/* Plans the next step into out[0 .. n) (decodes in slot order, then the
 * admitted prefills in queue order) and returns n (0 when idle), or a
 * negative dllm_status. cap >= slots. Each plan must be followed by one
 * dllm_sched_complete before the next plan (else DLLM_ERR_INVALID_ARG). */
int dllm_sched_plan(dllm_sched *s, dllm_sched_entry *out, int cap);

/* Reports the planned step's outcome: remaining[slot] = masked positions
 * left in the slot's block, eos[slot] != 0 = the block holds a committed end
 * token (may be NULL). Host arrays of `slots` entries; only the slots of
 * the last plan are read. */
dllm_status dllm_sched_complete(dllm_sched *s, const int32_t *remaining,
                                const uint8_t *eos);

/* Current carried budget D (after the last plan's charges). */
long long dllm_sched_budget(const dllm_sched *s);
/* Requests waiting for a prefill (new or resident). */
int dllm_sched_queued(const dllm_sched *s);
/* Moves up to cap finished request ids (in finishing order) into req_out
 * and returns how many were moved. */
int dllm_sched_finished(dllm_sched *s, int32_t *req_out, int cap);

/* The packed layout of a planned step for dllm_denoise_step with B = slots
 * (batch index = slot; slots not in the plan get no rows, and their block
 * state, all committed, is left unchanged by the commit):
 *   q_off, kv_off [slots + 1]: query / key rows of the entries in slot
 *     order (prefix sums of q_rows / kv_rows; 0 rows for absent slots);
 *   row_req, row_pos [n * blk]: head row r = (slot, block position), the
 *     entries' blocks in slot order.
 * Returns the number of head rows (n * blk) or a negative dllm_status. */
int dllm_sched_pack(const dllm_sched_entry *entries, int n, int slots,
                    int blk, int32_t *q_off, int32_t *kv_off,
                    int32_t *row_req, int32_t *row_pos);

#ifdef __cplusplus
}
#endif

#endif /* DLLM_SCHED_H */
