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

// ---- decode step for B > 1 (pop_decode_tc.cu): two skinny GEMMs on tcgen05
// The B operand of a decode GEMM: `rows` token rows of `inner` bf16, `ld` elements apart, box
// {64, NP} (rows NP > `rows` read as zero).
bool encode_tokens_map(CUtensorMap* m, const void* base, int inner, int rows, int ld, int NP);
// The z rows of the list as the down GEMM's B operand: `rows` rows of 2 NP bf16 (hi then lo parts),
// box {64, 64} (columns past 2 NP and rows past `rows` read as zero).
bool encode_zrows_map(CUtensorMap* m, const uint16_t* zcp, int rows, int NP);
struct GateUpTcArgs {
  const uint16_t* Wp;    // packed weights
  int D, N;
  int B, NP;             // tokens, and tokens padded to a multiple of 16 (the MMA's N)
  const int* rc;         // position -> channel: [C | R]
  int nC, nR;
  const float* n2;       // ||W2[:, c]||
  uint16_t* zcp;         // out: z of every position p as row p of 2 NP bf16 (hi parts of the tokens,
                         // then lo parts z - hi), [nC + nR][2 NP]
  float* scores;         // out: [nC]
  // work split (set by the launcher)
  int units, rows_cap, ks, stages;
  unsigned* err;
  uint64_t wait_ns;
};
struct DownTcArgs {
  const uint16_t* Wp;
  int D, N;
  int B, NP;
  int nR;                // R items: k-blocks [0, kbr) of the z planes' columns [0, nR)
  int kbr;               // ceil(nR / 64); the selected items start at column 64 * kbr
  int k;                 // selected candidates
  const int* ch_r;       // channels of R (ascending)
  int* ch_s;             // channels of the selected candidates (written by the selecting CTA)
  int r_pos0;            // list position of R item 0: its z row is zcp row r_pos0 + item
  void* y;               // out: [B][D], fp32 or bf16
  int out_f32;
  const uint16_t* dslab; // down slab of R (units are then the 128-output slices of the slab), or NULL
  // selection by the first cluster (sel = 1, decode with candidates)
  int sel;
  const float* scores;   // [nC] this step's candidate scores
  const uint16_t* zcp;   // [positions][2 NP] z rows (hi, lo) from the gate/up
  const int* rc;         // position -> channel, C first
  int nC, period;
  float* memory;
  int* S;
  int* step;
  int count_step;        // 1: advance the step counter (decode)
  unsigned* flag;        // selection of step `epoch` complete when *flag == epoch
  unsigned epoch;
  int skip;              // a skip-variant step between updates: the selecting CTA adds the scores of
                         // positions [0, k) to the memory at S_hold and selects nothing; S is [0, k)
  const int* S_hold;
  int* rcs;              // skip variant, update steps: rcs[j] = channel of selected j (or NULL)
  // work split (set by the launcher)
  int split, units;
  unsigned* err;
  uint64_t wait_ns;
};
// gate/up over R u C: z of the candidates, their scores, and the z planes of R
cudaError_t launch_gateup_tc(const CUtensorMap& x_map, GateUpTcArgs args, int num_sms, cudaStream_t st);

// ---- decode slabs for B > 1 (pop_decode_tc.cu): the weights a partition keeps, repacked once per
// partition into tiles that are byte for byte the shared-memory operand images of the decode GEMMs,
// so that decode streams them with one bulk copy per stage instead of gathering rows.
// Gate/up slab: positions [0, P) of rc in T tiles of RT positions; tile t, k-block kb is an A tile of
// `arows` rows x 128 bytes (128-byte swizzle) at ((t * KB + kb) * arows) * 64 elements. With RT <= 64
// ("paired") gate and up of position j share one MMA: row 32 (j / 16) + 16 g + j % 16; otherwise the
// gate rows fill rows [0, RT) and the up rows start at row round8(RT).
struct GuSlabGeom {
  int P, T, RT, KB, arows, paired;
  int Ts, P1;  // two regions: tiles [0, Ts) hold positions [0, P1), the rest [P1, P) (Ts = 0: one)
};
// List position held by row slot j of tile t, or -1 for an empty slot.
__host__ __device__ inline int gu_slab_pos(const GuSlabGeom& g, int t, int j) {
  if (j >= g.RT) return -1;
  if (t < g.Ts) {
    const int p = t * g.RT + j;
    return p < g.P1 ? p : -1;
  }
  const int p = g.P1 + (t - g.Ts) * g.RT + j;
  return p < g.P ? p : -1;
}
GuSlabGeom gu_slab_geom(int P, int D, int num_sms);
// The same tiles for a list in two regions, [0, P1) and [P1, P), kept in separate tiles so that
// the first region's tiles can be rebuilt alone.
GuSlabGeom gu_slab_geom_split(int P1, int P, int D, int num_sms);
// Builds tiles [t_lo, t_hi) of a gate/up slab from the packed weights and the list rc.
cudaError_t launch_build_gu_tiles(const uint16_t* Wp, const int* rc, int D, int N, const GuSlabGeom& g, int t_lo,
                                  int t_hi, uint16_t* gu_slab, unsigned* err, cudaStream_t st);
size_t gu_slab_elems(const GuSlabGeom& g);
// Down slab: the down columns of R in tiles of 64 items x 128 outputs (MN-major image: two halves of
// 64 outputs, 64 items x 128 bytes each, 128-byte swizzle) at ((o * kbr + b) * 8192) elements for
// output slice o (of ceil(D / 128)) and item block b (of kbr = ceil(nR / 64)).
size_t dn_slab_elems(int D, int nR);
cudaError_t launch_build_slabs(const uint16_t* Wp, const int* rc, int nC, int nR, int D, int N, const GuSlabGeom& g,
                               uint16_t* gu_slab, uint16_t* dn_slab, unsigned* err, cudaStream_t st);
struct GateUpSlabArgs {
  const uint16_t* slab;
  GuSlabGeom geom;
  int D, N;
  int B, NP;
  const int* rc;         // for the candidates' down-column norms
  int nC, nR;
  const float* n2;
  uint16_t* zcp;         // out: every position's z row, [nC + nR][2 NP] bf16 (hi parts of the NP
                         // tokens, then their lo parts), the down GEMM's MN-major operand
  float* scores;
  int ks, stages;        // set by the launcher
  unsigned* err;
  uint64_t wait_ns;
};
cudaError_t launch_gateup_slab(const CUtensorMap& x_map, GateUpSlabArgs args, int num_sms, cudaStream_t st);
// the selection (when args.sel), then y = sum over R and the selected items of z W2[:, channel]
// z_map: the z rows as a bf16 [r_pos0 + nR][2 NP] tensor, box {64, 64}, 128-byte swizzle
// (encode_zrows_map); the decode's R stages load their z rows through it.
cudaError_t launch_down_tc(const CUtensorMap& z_map, DownTcArgs args, int num_sms, cudaStream_t st);

// ---- decode step for B = 1 (pop_decode1.cu): gate/up with in-kernel top-k, tiled down
struct DecodeB1Args {
  const uint16_t* Wp;
  const float* n2;
  int D, N;
  const uint16_t* x;   // [D] bf16
  const int* rc;       // [C | R] channel indices (or all channels for the dense path)
  int nC, nR;
  int do_select;       // 1: CTA 0 of the gate/up grid runs the memory update and the top-k
  int skip;            // 1: a step between updates of the skip variant: rc lists [C[S] | R], nC = k,
                       //    CTA 0 adds the scores to the memory at the held positions S_hold
  const int* S_hold;   // the held selection (positions into C) on skip steps
  int* rcs;            // skip variant, update steps: CTA 0 writes rcs[j] = rc[S[j]] (or NULL)
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
  unsigned* tile_cnt;  // per output tile of y: chunk CTAs done (0 between launches)
  unsigned* err;
  uint64_t wait_ns;
};
int down_tiled_chunks(int D, int nitems, int num_sms);
// B = 1 down: outputs per tile of y; the handle keeps one inter-CTA counter per tile
constexpr int B1_DOWN_TILE = 256;
constexpr int b1_down_tiles(int D) { return (D + B1_DOWN_TILE - 1) / B1_DOWN_TILE; }
cudaError_t launch_gateup_sel_b1(const DecodeB1Args& a, int grid, cudaStream_t st);
cudaError_t launch_down_tiled_b1(const DecodeB1Args& a, int num_sms, cudaStream_t st);

// Raises a kernel's dynamic shared-memory limit to `bytes` on the current device, once per kernel,
// device and size (the attribute is per device; thread-safe). Call before every launch that needs
// more than the 48 KB default, counting the kernel's static shared memory in.
cudaError_t ensure_dyn_smem(const void* kernel, size_t bytes);

// largest |C| whose top-k runs inside the B = 1 gate/up kernel (its keys sit in shared memory).
// Larger candidate sets are selected by a kernel of their own: when (nearly) every channel is a
// candidate the in-kernel top-k cannot overlap the R stream, and measured slower than the
// separate kernel (full re-evaluation at D_FF = 11008: step 66 us against 58 us).
constexpr int FZ_MAX_C = 8192;

// ---- selection (pop_select.cu)
// Importance from channel sums (if sumsq != NULL: I = n2 * sqrt(sumsq), written to I), then the
// R/C/P split by the counting rule; writes rc = [C ascending | R ascending], P ascending, resets
// step and memory.
cudaError_t launch_partition(const float* sumsq, const float* n2, float* I, int N, int n_P, int n_R, int* rc,
                             int* P, int* step, float* memory, unsigned* err, cudaStream_t st);
// Candidate selection for one decode step (periodic memory, top-k, step counter).
// rcs (skip variant, or NULL): on update steps rcs[j] = rc[S[j]] for the selected j < k
cudaError_t launch_select(const float* scores, float* memory, int nC, int k, int period, int* step, int* S,
                          const int* rc, int* rcs, unsigned* err, cudaStream_t st);
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
// z = SiLU(X Wg^T) * (X W1^T) as two bf16 planes: Z[m][n] = bf16(z), Zlo[m][n] = bf16(z - Z[m][n]);
// part[(m/32)][n] = sum over 32 rows of z^2 (fp32, un-rounded z).
cudaError_t launch_prefill_gateup(const CUtensorMap& x_map, const PrefillMaps& maps, int M, int N, int D,
                                  uint16_t* Z, uint16_t* Zlo, int ldZ, float* part, int ldPart, unsigned* err,
                                  uint64_t wait_ns, int num_sms, cudaStream_t st);
// Y = (Z + Zlo) W2^T, Y fp32 or bf16 [M, D] (z_map, zlo_map: the two planes, encode_z_map).
cudaError_t launch_prefill_down(const CUtensorMap& z_map, const CUtensorMap& zlo_map, const PrefillMaps& maps,
                                int M, int N, int D, void* Y, int out_f32, unsigned* err, uint64_t wait_ns,
                                int num_sms, cudaStream_t st);
size_t prefill_smem_bytes();

// Sets the message that pop_last_error(NULL) returns on this thread.
void set_unbound_error(const char* msg);

}  // namespace pop
