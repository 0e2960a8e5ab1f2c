// Internal launch interface between the C-ABI layer (pop_ffn.cu) and the kernel files.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pop {

// Bits of the device error word.
enum : unsigned {
  DEVERR_TIMEOUT_GATEUP = 1u << 0,  // prefill gate/up GEMM: a wait ran out
  DEVERR_TIMEOUT_DOWN = 1u << 1,    // prefill down GEMM: a wait ran out
  DEVERR_PARTITION = 1u << 2,       // partition: region sizes did not match the counts
  DEVERR_TOPK = 1u << 3,            // top-k: selected count did not match k
  DEVERR_INDEX = 1u << 4,           // an index list entry was out of range
  DEVERR_TIMEOUT_DECODE = 1u << 5,  // B = 1 decode: the selector's wait for the candidate scores ran out
  DEVERR_TIMEOUT_DECODE_TC = 1u << 6,  // B > 1 decode (tensor-core kernels): a wait ran out
  DEVERR_TIMEOUT_ANY =
      DEVERR_TIMEOUT_GATEUP | DEVERR_TIMEOUT_DOWN | DEVERR_TIMEOUT_DECODE | DEVERR_TIMEOUT_DECODE_TC,
};

// Packed weights: row i of Wp holds [Wg[i, 0:D] | W1[i, 0:D] | W2[0:D, i]] (3*D bf16); n2[i] is
// ||W2[:, i]||_2 in fp32.

// ---- pack (pop_pack.cu)
cudaError_t launch_pack(const uint16_t* Wg, const uint16_t* W1, const uint16_t* W2, uint16_t* Wp, float* n2,
                        int D, int N, cudaStream_t st);

// ---- decode step for B > 1 (pop_decode_tc.cu): stream-K skinny GEMMs on tcgen05
// The B operand of a decode GEMM: `rows` token rows of `inner` bf16, `ld` elements apart, box
// {64, NP} (rows NP > `rows` read as zero).
bool encode_tokens_map(CUtensorMap* m, const void* base, int inner, int rows, int ld, int NP);
struct DecodeTcArgs {
  const uint16_t* Wp;    // packed weights
  int D;
  int B, NP;             // tokens, and tokens padded to a multiple of 16 (the MMA's N)
  int rows;              // M extent: positions |R u C| (gate/up) or D (down)
  int K;                 // reduction extent: D (gate/up) or the kept items |R| + k (down)
  int N;                 // channel count, for the index guards
  const int* rc;         // gate/up: position -> channel ([C | R])
  const int* ch_r;       // down: channels of the items j < nR_items (R)
  const int* ch_s;       // down: channels of the items j >= nR_items (the selected candidates)
  int nR_items;
  int nC;                // gate/up: positions below nC are candidates
  const float* n2;       // ||W2[:, c]||
  float* z;              // gate/up out: fp32 [B][ldz]
  int ldz;
  uint16_t* zk;          // gate/up out: z of R positions at [b][p - nC], bf16 hi part
  uint16_t* zk_lo;       // ... and bf16 lo part z - hi
  int ldk;
  float* scores;         // gate/up out: [nC]
  void* y;               // down out: [B][D], fp32 or bf16
  int out_f32;
  int split;             // CTAs per tile along K (a cluster); set by the launcher
  unsigned* err;
  uint64_t wait_ns;
};
cudaError_t launch_gateup_tc(const CUtensorMap& x_map, const DecodeTcArgs& args, int num_sms, cudaStream_t st);
// zk_map / zk_lo_map: the hi and lo bf16 planes of z over the kept items
cudaError_t launch_down_tc(const CUtensorMap& zk_map, const CUtensorMap& zk_lo_map, const DecodeTcArgs& args,
                           int num_sms, cudaStream_t st);

// ---- decode step for B = 1 (pop_decode1.cu): gate/up with in-kernel top-k, tiled down
struct DecodeB1Args {
  const uint16_t* Wp;
  const float* n2;
  int D, N;
  const uint16_t* x;   // [D] bf16
  const int* rc;       // [C | R] channel indices (or all channels for the dense path)
  int nC, nR;
  int do_select;       // 1: CTA 0 of the gate/up grid runs the memory update and the top-k
  int k;               // candidates to select
  int kd;              // selected candidates the down projection adds (k, or 0 for the dense path)
  int period;
  float* z;            // [nC + nR]
  float* scores;       // [nC]
  float* memory;       // [nC]
  int* S;              // [k] positions into C
  int* step;
  float* ypart;        // [chunks][D]
  void* y;
  int out_f32;
  unsigned* sync;      // 1 counter: candidates scored so far (0 between launches)
  unsigned* tile_cnt;  // per 512-wide tile of y: chunk CTAs done (0 between launches)
  unsigned* err;
  uint64_t wait_ns;
};
int down_tiled_chunks(int D, int nitems, int num_sms);
cudaError_t launch_gateup_sel_b1(const DecodeB1Args& a, int grid, cudaStream_t st);
cudaError_t launch_down_tiled_b1(const DecodeB1Args& a, int num_sms, cudaStream_t st);

// largest |C| whose top-k runs inside the B = 1 gate/up kernel (its keys sit in shared memory)
constexpr int FZ_MAX_C = 8192;

// ---- selection (pop_select.cu)
// Importance from channel sums (if sumsq != NULL: I = n2 * sqrt(sumsq), written to I), then the
// R/C/P split by the counting rule; writes rc = [C ascending | R ascending], P ascending, resets
// step and memory.
cudaError_t launch_partition(const float* sumsq, const float* n2, float* I, int N, int n_P, int n_R, int* rc,
                             int* P, int* step, float* memory, unsigned* err, cudaStream_t st);
// Candidate selection for one decode step (periodic memory, top-k, step counter).
cudaError_t launch_select(const float* scores, float* memory, int nC, int k, int period, int* step, int* S,
                          unsigned* err, cudaStream_t st);
// The same for B > 1 (the top-k only), launched with programmatic dependent launch.
cudaError_t launch_select_bn(const float* scores, float* memory, int nC, int k, int period, int* step, int* S,
                             unsigned* err, cudaStream_t st);
// The selected candidates' side of the B > 1 down projection: ch_s[j] = rc[S[j]] and the hi / lo
// bf16 parts of z[b][S[j]] at zk[b][nR + j] / zk_lo[b][nR + j], for j < k, b < B. Many CTAs,
// launched with programmatic dependent launch.
cudaError_t launch_pack_selected(const int* S, int k, int nC, const int* rc, int N, int* ch_s, const float* z,
                                 int ldz, int B, uint16_t* zk, uint16_t* zk_lo, int ldk, int nR, unsigned* err,
                                 cudaStream_t st);
// sumsq[i] (+)= sum over rows p < rows of part[p * ld + i], p ascending.
cudaError_t launch_fold_sumsq(const float* part, int rows, int ld, int N, float* sumsq, int accumulate,
                              cudaStream_t st);

// ---- prefill GEMMs on tcgen05 (pop_prefill.cu)
struct PrefillMaps {
  CUtensorMap wg;  // over Wp: dims {D, N}, row stride 3D*2 bytes, box {64, 128}
  CUtensorMap w1;  // over Wp + D
  CUtensorMap w2;  // over Wp + 2D: dims {D, N}, box {64, 64} (d inner)
};
bool encode_weight_maps(PrefillMaps* m, const uint16_t* Wp, int D, int N);
bool encode_x_map(CUtensorMap* m, const uint16_t* X, int M, int D);
bool encode_z_map(CUtensorMap* m, const uint16_t* Z, int M, int N, int ldZ);
// Z[m][n] = bf16(SiLU(X Wg^T) * (X W1^T)); part[(m/32)][n] = sum over 32 rows of z^2 (fp32, un-rounded z).
cudaError_t launch_prefill_gateup(const CUtensorMap& x_map, const PrefillMaps& maps, int M, int N, int D,
                                  uint16_t* Z, int ldZ, float* part, int ldPart, unsigned* err, uint64_t wait_ns,
                                  int num_sms, cudaStream_t st);
// Y = Z W2^T, Y fp32 or bf16 [M, D].
cudaError_t launch_prefill_down(const CUtensorMap& z_map, const PrefillMaps& maps, int M, int N, int D, void* Y,
                                int out_f32, unsigned* err, uint64_t wait_ns, int num_sms, cudaStream_t st);
size_t prefill_smem_bytes();

// Sets the message that pop_last_error(NULL) returns on this thread.
void set_unbound_error(const char* msg);

}  // namespace pop
