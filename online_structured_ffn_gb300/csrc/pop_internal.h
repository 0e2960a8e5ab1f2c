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
  DEVERR_TIMEOUT_ANY = DEVERR_TIMEOUT_GATEUP | DEVERR_TIMEOUT_DOWN | DEVERR_TIMEOUT_DECODE,
};

// Packed weights: row i of Wp holds [Wg[i, 0:D] | W1[i, 0:D] | W2[0:D, i]] (3*D bf16).
struct PackedWeights {
  const uint16_t* Wp;
  const float* n2;  // ||W2[:, i]||_2, fp32
  int D;
  int N;
};

// ---- pack (pop_pack.cu)
cudaError_t launch_pack(const uint16_t* Wg, const uint16_t* W1, const uint16_t* W2, uint16_t* Wp, float* n2,
                        int D, int N, cudaStream_t st);

// ---- decode (pop_decode.cu)
// z[b * ldz + p] = z of item p (channel rc[p]) for token b; scores[p] = max_b |z| * n2 for p < nC.
cudaError_t launch_gateup_decode(const PackedWeights& w, const uint16_t* x, int B, const int* rc, int nRC, int nC,
                                 float* z, int ldz, float* scores, unsigned* err, int num_sms, cudaStream_t st);
// Down projection over the items R (rc positions nC .. nC+nR-1) and the selected candidates
// (rc positions S[0..k)); partial sums go to ypart [G][B][D]; returns G through *G_out.
cudaError_t launch_down_decode(const PackedWeights& w, const int* rc, int nC, int nR, const int* S, int k,
                               const float* z, int ldz, int B, float* ypart, int max_parts, int* G_out,
                               unsigned* err, int num_sms, cudaStream_t st);
int down_decode_parts(int D, int B, int nitems, int num_sms);
// y[b][d] = sum_g ypart[g][b][d] (g ascending); y is fp32 or bf16.
cudaError_t launch_reduce_y(const float* ypart, int G, int B, int D, void* y, int out_f32, cudaStream_t st);

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
