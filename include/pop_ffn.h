/*
 * pop_ffn.h — C-ABI of the GB300 (sm_103a) library for partition-guided online
 * structured pruning (POP) of one gated-MLP FFN layer.
 *
 * The method (sources cited by page title and section):
 *   [BWAP] "Batch-wise adaptive pruning" (bittide page), Section 3.1 eq. (1):
 *          z = SiLU(Wg x) (.) (W1 x),  y = W2 z,  Wg, W1 in R^{D_FF x D}, W2 in R^{D x D_FF}.
 *   [POP]  "POP: Online Structural Pruning Enables Efficient Inference of Large
 *          Foundation Models" (papernotes.org notes):
 *          Key design 1 — prefill importance I_i = ||W2[:,i]||_2 * ||Z[:,:,i]||_2 over all
 *          prompt tokens, quantile cut-offs q_{r-delta}, q_{r+delta} splitting the channels into
 *          Retained R, Candidate C and Pruned P;
 *          Key design 2 — each decode step computes gate/up only over R u C, scores C only,
 *          sorts the candidates and fills |R| + k = (1 - r) * D_FF survivors;
 *          Loss / training strategy — gamma = 0.1 (about 20% candidates), Wanda metric,
 *          partition taken at the first (prefill) forward.
 *   [BWAP] abstract and Fig. 2(a) — a batch shares one mask (element-wise max over the batch);
 *          periodic top-k with an activation memory summed between updates.
 *
 * Readings where the pages are silent (fixed here, identical in the CPU oracle):
 *   delta = gamma; counts rounded half-to-even:
 *     n_P = round(max(0, r - gamma) * D_FF), n_R = D_FF - round(min(1, r + gamma) * D_FF),
 *     keep = D_FF - round(r * D_FF), k = keep - n_R, n_C = D_FF - n_P - n_R;
 *   ties at every cut-off go to the lower channel index;
 *   candidate score a_i = max_b |z_{b,i}| * ||W2[:,i]||_2;
 *   periodic memory: M += a every step; when step % period == 0 the selection is redone from M
 *   and M is cleared (period 1 = per-step POP).
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device pointers on the handle's device; "host" pointers
 *     are ordinary host memory. bf16 is IEEE bfloat16 stored as uint16; matrices are row-major.
 *     Device buffers must be 16-byte aligned.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls taking a stream are
 *     asynchronous and stream-ordered unless their comment says "syncs".
 *   - Every call returns a pop_status and never throws or aborts. Argument and state errors
 *     are found on the host before anything is enqueued. pop_last_error() gives the message.
 *   - Device-side failures (a bounded wait that ran out, an index out of range) are recorded
 *     in a device error word and returned by pop_check().
 *   - A handle may be used from one host thread at a time, and its calls must not overlap on the
 *     GPU (use one stream per handle, or order the streams).
 */
#ifndef POP_FFN_H
#define POP_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pop_ffn* pop_ffn_t;

typedef enum {
  POP_OK = 0,
  POP_ERR_INVALID_ARG = 1,   /* bad pointer, size or configuration */
  POP_ERR_STATE = 2,         /* e.g. decode before any partition exists */
  POP_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
  POP_ERR_OOM = 4,           /* device allocation failed */
  POP_ERR_TIMEOUT = 5,       /* a device-side bounded wait ran out (see pop_check) */
  POP_ERR_UNSUPPORTED = 6,   /* the device is not sm_103 (GB300) */
  POP_ERR_DEVICE = 7         /* a device-side consistency check failed (see pop_check) */
} pop_status;

/* Limits of this build. */
#define POP_MAX_D 16384        /* D must be a multiple of 8 and <= POP_MAX_D */
#define POP_MAX_D_FF 49152     /* D_FF <= POP_MAX_D_FF (the partition runs in one CTA) */
#define POP_MAX_BATCH 64       /* max_batch <= POP_MAX_BATCH */
#define POP_STATIC_MAX_D_FF 49152  /* largest D_FF of pop_ffn_dense_token_noalloc (its static scratch) */

typedef struct {
  int D;                  /* model width: length of x and y. Multiple of 8, 8..POP_MAX_D. */
  int D_FF;               /* intermediate channels N, 1..POP_MAX_D_FF. */
  double r;               /* FFN prune rate in [0, 1]: (1 - r) * D_FF channels survive each step. */
  double gamma;           /* partition half-width (delta = gamma), >= 0. */
  int period;             /* selection period P >= 1; 1 = per-step POP. */
  int max_batch;          /* largest B accepted by pop_decode_step, 1..POP_MAX_BATCH. */
  int max_prefill_tokens; /* prefill chunk: longer prompts run in chunks of this many tokens. >= 1. */
  int out_f32;            /* dtype of y / Y: 1 = float32, 0 = bf16. */
  int skip;               /* periodic skip variant (0 or 1; takes effect with period > 1): between
                             updates gate/up runs only over R and the held selection, and the memory
                             gains the scores of the held selection only. 0 = off. */
} pop_config;

typedef struct {
  int n_P, n_R, n_C;      /* region sizes ([POP] Key design 1) */
  int keep;               /* survivors per step = |R| + k ([POP] Key design 2) */
  int k;                  /* candidates selected per step */
} pop_counts;

/* Region sizes for (N, r, gamma) by the counting rule above. Host only, no handle needed.
 * POP_ERR_INVALID_ARG if r is outside [0,1], gamma < 0, N < 0 or out == NULL. */
pop_status pop_region_counts(int N, double r, double gamma, pop_counts* out);

/* Creates a handle on the current CUDA device and packs the weights ([BWAP] Section 3.1).
 *   Wg, W1: device bf16 [D_FF, D]; W2: device bf16 [D, D_FF] (row-major, as in eq. (1)).
 * The handle copies them into its own channel-major layout (gate row, up row and down column of
 * each channel contiguous) and computes ||W2[:,i]||_2 in fp32; the caller may free the inputs
 * once `stream` has passed this call. Allocates all device scratch the later calls need.
 * Errors: INVALID_ARG (NULL pointer, bad config, k outside [0, n_C]), UNSUPPORTED (device not
 * sm_103), OOM, CUDA. On error *out is set to NULL. */
pop_status pop_ffn_create(const pop_config* cfg, const void* Wg, const void* W1, const void* W2,
                          void* stream, pop_ffn_t* out);

/* Frees the handle and its device memory (synchronizes the device first). NULL is a no-op. */
void pop_ffn_destroy(pop_ffn_t h);

/* The region sizes of this handle. */
pop_status pop_ffn_counts(pop_ffn_t h, pop_counts* out);

/* Prefill ([POP] Key design 1; "Loss / training strategy": prefill runs dense and fixes the
 * partition). X: device bf16 [M, D] prompt tokens (all B*L of them), M >= 1. Runs the dense FFN
 * on the tensor cores, reduces sum_t z_{t,i}^2 per channel from un-rounded fp32 z, forms
 * I_i = ||W2[:,i]|| * sqrt(sum), and writes the R, C, P index lists on the device. Resets the
 * decode step counter and the activation memory.
 * Y: device [M, D] (float32 if out_f32 else bf16) receives the dense FFN output, or NULL to skip
 * the down GEMM. Prompts longer than max_prefill_tokens run in chunks; the sums carry over. */
pop_status pop_prefill_partition(pop_ffn_t h, const void* X, int M, void* Y, void* stream);

/* Sets the partition from a caller-given importance (device fp32 [D_FF]) instead of a prompt:
 * same cut-off and tie rule as pop_prefill_partition. Resets step counter and memory. */
pop_status pop_partition_from_importance(pop_ffn_t h, const float* importance, void* stream);

/* Sets the partition from host index lists (ascending, disjoint, covering [0, D_FF), sizes
 * n_R, n_C, n_P of pop_ffn_counts). Used to replay or restore a session. Resets step counter
 * and memory. Syncs `stream`. INVALID_ARG if the lists are not such a partition. */
pop_status pop_set_partition(pop_ffn_t h, const int* R, const int* C, const int* P, void* stream);

/* One decode step ([POP] Key design 2; [BWAP] batch max and periodic memory).
 * x: device bf16 [B, D], 1 <= B <= max_batch; y: device [B, D] (float32 if out_f32 else bf16).
 * Computes z over R u C, candidate scores a_i = max_b |z_{b,i}| * ||W2[:,i]||, updates the memory,
 * selects the k best candidates when step % period == 0 (ties to the lower index), and writes
 * y = sum over R u S of z_i * W2[:,i]. No allocation and no host synchronization. The step is two
 * kernels launched with programmatic dependent launch (gate/up, then the down projection; the
 * selection runs inside the gate/up kernel at B = 1 and inside the down kernel at B > 1, and at
 * B = 1 with |C| > 8192 as a third kernel between them). The next kernel's weight loads overlap
 * the previous kernel's tail; each kernel waits for its predecessor before it touches data a
 * previous call may still use. Steps can be captured in a CUDA graph. With cfg.skip and
 * period > 1 the steps between updates run over R and the held selection only; which steps those
 * are is decided on the host (a counter reset by every partition call), so a captured graph
 * replays the update/skip pattern it captured. At B > 1 an update step of the skip variant adds
 * a third kernel that rebuilds the selected rows' tiles of the skip steps' slab.
 * STATE if no partition has been set. */
pop_status pop_decode_step(pop_ffn_t h, const void* x, int B, void* y, void* stream);

/* Dense FFN y = W2 (SiLU(Wg x) (.) W1 x) for every row of X (device bf16 [M, D]) into Y (device
 * [M, D], dtype per out_f32). Does not touch the partition or decode state. */
pop_status pop_ffn_dense_ref(pop_ffn_t h, const void* X, int M, void* Y, void* stream);

/* Copies the partition to host arrays (any may be NULL) of sizes n_R, n_C, n_P. Syncs. */
pop_status pop_get_partition(pop_ffn_t h, int* R, int* C, int* P);

/* Copies the last prefill's importance I and channel sums sum_t z^2 (host float [D_FF], either
 * may be NULL). Syncs. */
pop_status pop_get_importance(pop_ffn_t h, float* importance, float* sumsq);

/* Copies the selected candidates of the last selection as ascending channel indices (host int
 * [k]); *k_out receives k. Syncs. STATE before the first decode step. */
pop_status pop_get_selected(pop_ffn_t h, int* k_out, int* channels);

/* Copies the last step's candidate scores and the activation memory (host float [n_C], in the
 * ascending channel order of C; either may be NULL). Syncs. */
pop_status pop_get_scores(pop_ffn_t h, float* scores, float* memory);

/* Number of decode steps since the partition was set (device counter). Syncs. */
pop_status pop_get_step(pop_ffn_t h, int* step);

/* Limit, in nanoseconds, for every device-side wait of this handle's kernels (default 2 s).
 * A wait that runs out sets POP_ERR_TIMEOUT in the device error word and the kernel returns. */
pop_status pop_set_wait_limit(pop_ffn_t h, uint64_t ns);

/* Per-kernel timing of decode steps (off by default). enable = n >= 1: one pop_decode_step in
 * every n records CUDA events on its stream between its kernel slots (gate/up, selection, down,
 * reduction; a slot a path does not launch reads near zero), for up to 256 timed steps between
 * reads. Each event adds a little GPU time, which sampling keeps out of most steps.
 * enable = 0 turns timing off. Enabling creates the events; disabling destroys them. */
pop_status pop_profile_enable(pop_ffn_t h, int enable);

/* Sums of the recorded kernel durations in milliseconds since the last read: ms[0] gate/up,
 * ms[1] selection, ms[2] down projection, ms[3] reduction; *steps receives the number of decode
 * steps recorded. Clears the record. Syncs. */
pop_status pop_profile_read(pop_ffn_t h, double* ms, int* steps);

/* Synchronizes the device and returns the first recorded device-side failure (TIMEOUT or
 * DEVICE) or POP_OK; clears the error word. CUDA if a CUDA call fails. */
pop_status pop_check(pop_ffn_t h);

/* Message of the last failed call on h (h == NULL: last failure of pop_ffn_create or of a call
 * given a NULL handle). Valid until the next call on the same handle. Never NULL. */
const char* pop_last_error(pop_ffn_t h);

/* Dense FFN of one token without any device allocation, for callers that cannot allocate GPU
 * memory when they run: processes whose device memory is reserved up front by their own memory
 * manager, and latency-critical loops that must not enter the CUDA allocator (it can block and
 * synchronise the device). The POP notes and the other pages have no counterpart to this call;
 * it is a deployment convenience of this library.
 *   Wg, W1: device bf16 [D_FF, D]; W2: device bf16 [D, D_FF] (row-major, as for pop_ffn_create);
 *   x: device bf16 [D]; y: device [D], float32 if out_f32 else bf16. No handle is involved.
 *   D: multiple of 8 in [8, POP_MAX_D]; D_FF: multiple of 8, at most POP_STATIC_MAX_D_FF.
 * Computes y = W2 (SiLU(Wg x) (.) W1 x), asynchronously on `stream`. The intermediate z lives in
 * one static device array of POP_STATIC_MAX_D_FF floats (192 KB), held by every GPU that loads
 * the library until the process exits. All calls on a device share it and it keeps the last
 * call's contents; every call rewrites all of z before reading it, but calls that overlap on the
 * GPU (other streams, other host threads) race on it and must be serialised by the caller.
 * The first call on each device, with that device current, looks up the array's device address
 * (cudaGetSymbolAddress); make that first call before any stream capture.
 * Errors: INVALID_ARG (NULL or misaligned pointer, D or D_FF outside the limits above, with the
 * message in pop_last_error(NULL)), UNSUPPORTED (not sm_103, or a device ordinal of 64 or more),
 * CUDA (also when a CUDA error from the caller's earlier work is still pending on the thread:
 * nothing is launched and that error is left in place). Calls no cudaMalloc/cudaFree. */
pop_status pop_ffn_dense_token_noalloc(const void* Wg, const void* W1, const void* W2, int D, int D_FF,
                                       const void* x, void* y, int out_f32, void* stream);

/* Name of a status code. Never NULL. */
const char* pop_status_string(pop_status s);

#ifdef __cplusplus
}
#endif

#endif /* POP_FFN_H */
