/*
 * pop_moe.h — C-ABI of an MoE layer of gated-MLP experts, each pruned with POP.
 *
 * Source: [POP] "POP: Online Structural Pruning Enables Efficient Inference of Large Foundation
 * Models" (papernotes.org notes), "Loss / training strategy": the method is applied to MoE models
 * with dynamic routing, the partition being taken at the first (prefill) forward. The pages give
 * no routing rule; this library takes these readings (identical in the CPU oracle):
 *   - routing: each token goes to the two experts with the largest router logits (ties to the
 *     lower expert index), weighted by the softmax over those two logits:
 *     w0 = 1 / (1 + exp(l1 - l0)), w1 = exp(l1 - l0) / (1 + exp(l1 - l0)), l0 >= l1;
 *   - each expert is one pop_ffn layer (pop_ffn.h) whose partition comes from the prompt tokens
 *     routed to it, in ascending token order; an expert with no routed prompt token has s = 0,
 *     so I = 0 and the index tie rule alone decides its R/C/P split;
 *   - every decode step advances every expert's step counter and memory; an expert that gets no
 *     token in a step scores every candidate 0 and contributes nothing;
 *   - y_t = w0 * expert_{e0}(x_t) + w1 * expert_{e1}(x_t), added in that order in fp32.
 *
 * Conventions are those of pop_ffn.h (device pointers 16-byte aligned, stream-ordered calls,
 * status returns, messages from pop_moe_last_error, device failures from pop_moe_check).
 */
#ifndef POP_MOE_H_
#define POP_MOE_H_

#include "pop_ffn.h"

#ifdef __cplusplus
extern "C" {
#endif

#define POP_MOE_MAX_EXPERTS 256 /* 2 <= n_experts <= POP_MOE_MAX_EXPERTS */

typedef struct pop_moe* pop_moe_t;

/* Creates an MoE layer of n_experts experts with the shared configuration cfg.
 *   Wg, W1, W2: host arrays of n_experts device pointers; expert e has Wg[e], W1[e] bf16
 *   [D_FF, D] and W2[e] bf16 [D, D_FF], as in pop_ffn_create (each expert copies its weights).
 *   cfg->max_batch bounds B of pop_moe_decode_step; cfg->out_f32 is the dtype of the layer's
 *   outputs (the experts compute in fp32 internally).
 * Allocates the experts and the decode scratch: per expert a [max_batch, D] bf16 input and a
 * [max_batch, D] fp32 output. Errors as pop_ffn_create; INVALID_ARG if n_experts is outside
 * [2, POP_MOE_MAX_EXPERTS] or a pointer array is NULL. On error *out is set to NULL. */
pop_status pop_moe_create(const pop_config* cfg, int n_experts, const void* const* Wg, const void* const* W1,
                          const void* const* W2, void* stream, pop_moe_t* out);

/* Frees everything the handle owns (syncs the device first). NULL is ignored. */
void pop_moe_destroy(pop_moe_t m);

/* Prefill of M prompt tokens: routes every token (logits: device fp32 [M, n_experts]), runs
 * each expert's pop_prefill_partition on its routed tokens (X: device bf16 [M, D]), and, if Y is
 * not NULL, writes the combined dense output Y (device [M, D], dtype per out_f32).
 * Syncs `stream` once (to size each expert's GEMMs by its token count) and allocates its grouped
 * buffers (2M rows of bf16 inputs and fp32 outputs) stream-ordered for the call.
 * Resets every expert's step counter and memory. INVALID_ARG: NULL X or logits, M < 1. */
pop_status pop_moe_prefill_partition(pop_moe_t m, const void* X, const float* logits, int M, void* Y,
                                     void* stream);

/* One decode step of B tokens: x device bf16 [B, D], logits device fp32 [B, n_experts],
 * y device [B, D] (dtype per out_f32), 1 <= B <= max_batch. Every expert runs pop_decode_step on
 * a [B, D] input holding its routed tokens in ascending token order followed by zero rows (a zero
 * row has z = 0, so it changes neither the batch-max scores nor the routed tokens' outputs).
 * No allocation and no host synchronization: 2 + 2 * n_experts kernels (the skip variant's
 * update steps add, per expert at B > 1, the rebuild of its slab's selected tiles). The routing
 * and the combine run on `stream`; the experts' kernels run as pop_moe_set_concurrent sets, and
 * the call is stream-ordered on `stream` either way (CUDA-graph capture included).
 * STATE if no partition has been set. */
pop_status pop_moe_decode_step(pop_moe_t m, const void* x, const float* logits, int B, void* y, void* stream);

/* How the experts' decode kernels are scheduled. on != 0 (the default): each expert runs on a
 * stream of its own that the handle owns, forked from the caller's stream after the routing (an
 * event) and joined back before the combine, so that one expert's kernels overlap another's;
 * the experts share no data, so y does not change. on = 0: the experts run one after another on
 * the caller's stream, so that per-kernel timing (pop_profile_enable on the experts) times each
 * kernel alone. INVALID_ARG for a NULL handle. */
pop_status pop_moe_set_concurrent(pop_moe_t m, int on);

/* Routing of the last prefill or decode call: host int experts[T][2] and float weights[T][2]
 * (either may be NULL); *T receives the number of tokens of that call. Syncs. STATE before the
 * first call. */
pop_status pop_moe_get_routing(pop_moe_t m, int* T, int* experts, float* weights);

/* Token count of each expert in the last call: host int counts[n_experts]. Syncs. */
pop_status pop_moe_get_counts(pop_moe_t m, int* counts);

/* Expert e's layer handle (borrowed: owned by m, valid until pop_moe_destroy), for the queries of
 * pop_ffn.h (partition, selection, importance, set_partition). NULL if e is out of range. */
pop_ffn_t pop_moe_expert(pop_moe_t m, int e);

/* Number of experts, or -1 for a NULL handle. */
int pop_moe_num_experts(pop_moe_t m);

/* Syncs; returns the first failure among the routing kernels and the experts' device error
 * words (as pop_check). */
pop_status pop_moe_check(pop_moe_t m);

/* Message of the last failed call on m (m = NULL: the last failed create). */
const char* pop_moe_last_error(pop_moe_t m);

#ifdef __cplusplus
}
#endif

#endif /* POP_MOE_H_ */
