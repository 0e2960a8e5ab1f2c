// C-ABI of the POP FFN library (declared in include/pop_ffn.h): handle, argument checks, device
// scratch, and the launch sequences of prefill, decode and the dense path.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "pop_ffn.h"
#include "pop_internal.h"

using namespace pop;

struct pop_ffn {
  pop_config cfg{};
  pop_counts cnt{};
  int D = 0, N = 0;
  int device = 0, num_sms = 0;
  // packed weights and norms
  uint16_t* Wp = nullptr;
  float* n2 = nullptr;
  // prefill scratch: z of one chunk as two bf16 planes, hi at Z, lo at Z + Mcap * ldZ
  uint16_t* Z = nullptr;
  int ldZ = 0, Mcap = 0;
  float* part = nullptr;
  int ldPart = 0;
  float* sumsq = nullptr;
  float* I = nullptr;
  PrefillMaps maps{};
  // partition: rc = [C ascending | R ascending], P ascending; idx_all = 0..N-1
  int* rc = nullptr;
  int* P = nullptr;
  int* idx_all = nullptr;
  // decode scratch
  float* z = nullptr;  // [max_batch][N]
  float* scores = nullptr;
  float* memory = nullptr;
  int* S = nullptr;
  float* ypart = nullptr;  // B = 1 down: partial tiles [chunks][D]
  int ypart_parts = 0;     // capacity in units of D floats
  // B > 1 decode (tensor-core kernels)
  int* ch_s = nullptr;     // channels of the selected candidates, in S order
  uint16_t* zcp = nullptr; // [N][2 * round_up(max_batch, 16)]: every list position's z row (hi, lo), B > 1
  int* rcs = nullptr;      // skip variant: [C[S] | R], the list of the steps between updates
  long long host_step = 0; // decode steps since the last partition (the device step counter's mirror)
  // B > 1 decode slabs (rebuilt at every partition): gate/up rows of R u C and down columns of R
  GuSlabGeom gu_geom{};
  uint16_t* gu_slab = nullptr;
  GuSlabGeom gu_geom_skip{};          // skip variant: the gate/up slab of [C[S] | R], rebuilt at each
  uint16_t* gu_slab_skip = nullptr;   // update step (B > 1)
  uint16_t* dn_slab = nullptr;
  int* step = nullptr;
  unsigned* err = nullptr;
  unsigned* fsync = nullptr;  // inter-CTA counters of the decode kernels
  unsigned epoch = 0;  // B > 1 decode calls so far: the selection flag of call e reads e
  bool partitioned = false;
  bool selected = false;
  uint64_t wait_ns = 2000000000ull;
  // optional per-kernel timing of decode steps: kProfEvents events per step
  std::vector<cudaEvent_t> prof_events;
  int prof_steps = 0;
  int prof_stride = 1;    // time one decode step in every prof_stride
  long long prof_calls = 0;
  bool prof_now = false;  // the current decode step is being timed
  std::string msg;
};

static constexpr int kProfEvents = 5;
// device counters: [4] candidates scored by the B = 1 gate/up, [5] the B > 1 selection flag, [8..]
// tiles of y done by the B = 1 down chunks (one per tile, up to the widest D)
static constexpr int kSyncWords = 8 + pop::b1_down_tiles(POP_MAX_D);
static constexpr int kProfMaxSteps = 256;

namespace {
thread_local std::string g_msg;

pop_status fail(pop_ffn* h, pop_status s, const std::string& m) {
  (h ? h->msg : g_msg) = m;
  return s;
}

pop_status cuda_fail(pop_ffn* h, cudaError_t e, const char* where) {
  return fail(h, e == cudaErrorMemoryAllocation ? POP_ERR_OOM : POP_ERR_CUDA,
              std::string(where) + ": " + cudaGetErrorString(e));
}

#define POP_CUDA(h, call)                                  \
  do {                                                     \
    cudaError_t e_ = (call);                               \
    if (e_ != cudaSuccess) return cuda_fail(h, e_, #call); \
  } while (0)

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int round_up(int v, int m) { return (v + m - 1) / m * m; }

long long round_half_even(double v) { return static_cast<long long>(std::nearbyint(v)); }

template <class T>
cudaError_t dalloc(T** p, size_t count) {
  if (count == 0) count = 1;
  return cudaMalloc(reinterpret_cast<void**>(p), count * sizeof(T));
}

void destroy_events(pop_ffn* h) {
  for (cudaEvent_t e : h->prof_events) cudaEventDestroy(e);
  h->prof_events.clear();
  h->prof_steps = 0;
  h->prof_calls = 0;
}

// Records profiling event `i` of the current decode step when timing is on and there is room.
void prof_begin(pop_ffn* h) {
  h->prof_now = !h->prof_events.empty() && h->prof_steps < kProfMaxSteps && (h->prof_calls % h->prof_stride) == 0;
  ++h->prof_calls;
}

void prof_mark(pop_ffn* h, int i, cudaStream_t st) {
  if (h->prof_now) cudaEventRecord(h->prof_events[static_cast<size_t>(h->prof_steps) * kProfEvents + i], st);
}

void prof_end(pop_ffn* h) {
  if (h->prof_now) ++h->prof_steps;
  h->prof_now = false;
}

void free_all(pop_ffn* h) {
  void* ptrs[] = {h->Wp,    h->n2,   h->Z,     h->part,    h->sumsq, h->I,      h->rc,     h->P,
                  h->idx_all, h->z, h->scores, h->memory, h->S,     h->ypart,  h->ch_s,
                  h->step, h->err,     h->fsync, h->gu_slab, h->dn_slab, h->zcp, h->rcs, h->gu_slab_skip};
  for (void* p : ptrs)
    if (p) cudaFree(p);
}

DecodeB1Args b1_args(pop_ffn* h, const uint16_t* x, void* y, const int* rc, int nC, int nR) {
  DecodeB1Args a{};
  a.Wp = h->Wp;
  a.n2 = h->n2;
  a.D = h->D;
  a.N = h->N;
  a.x = x;
  a.rc = rc;
  a.nC = nC;
  a.nR = nR;
  a.period = h->cfg.period;
  a.z = h->z;
  a.scores = h->scores;
  a.memory = h->memory;
  a.S = h->S;
  a.step = h->step;
  a.ypart = h->ypart;
  a.y = y;
  a.out_f32 = h->cfg.out_f32;
  a.sync = h->fsync + 4;
  a.tile_cnt = h->fsync + 8;
  a.err = h->err;
  a.wait_ns = h->wait_ns;
  return a;
}

// Zeroes every inter-CTA counter of the decode kernels (they are left at zero by each launch that
// completes, so this only matters after a partition change or a reported device error).
cudaError_t reset_counters(pop_ffn* h, cudaStream_t st) {
  return cudaMemsetAsync(h->fsync, 0, kSyncWords * sizeof(unsigned), st);
}

// The skip variant's list [C[S] | R]: R after the k selected slots (stream-ordered after the
// partition); the slots are written at each update step. Resets the host's step mirror.
cudaError_t skip_list_tail(pop_ffn* h, cudaStream_t st) {
  h->host_step = 0;
  if (h->cnt.n_R == 0) return cudaSuccess;
  cudaError_t e = cudaMemcpyAsync(h->rcs + h->cnt.k, h->rc + h->cnt.n_C, sizeof(int) * h->cnt.n_R,
                                  cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess || !h->gu_slab_skip) return e;
  // the skip slab's R tiles (its selected tiles are rebuilt at every update step)
  const GuSlabGeom& g = h->gu_geom_skip;
  return launch_build_gu_tiles(h->Wp, h->rcs, h->D, h->N, g, g.Ts, g.T, h->gu_slab_skip, h->err, st);
}

// Rebuilds the B > 1 decode slabs from the current partition (stream-ordered after it).
cudaError_t build_slabs(pop_ffn* h, cudaStream_t st) {
  if (!h->gu_slab) return cudaSuccess;
  return launch_build_slabs(h->Wp, h->rc, h->cnt.n_C, h->cnt.n_R, h->D, h->N, h->gu_geom, h->gu_slab, h->dn_slab,
                            h->err, st);
}

// gate/up over the positions of rc = [C (nC) | R (nR)] for B tokens: z of the candidates (zc),
// their scores, and the z planes of R.
// The same from the gate/up slab of the current partition.
pop_status gateup_slab(pop_ffn* h, const uint16_t* x, int B, cudaStream_t st, bool skip = false) {
  GateUpSlabArgs a{};
  a.slab = skip ? h->gu_slab_skip : h->gu_slab;
  a.geom = skip ? h->gu_geom_skip : h->gu_geom;
  a.D = h->D;
  a.N = h->N;
  a.B = B;
  a.NP = round_up(B, 16);
  a.rc = skip ? h->rcs : h->rc;
  a.nC = skip ? h->cnt.k : h->cnt.n_C;
  a.nR = h->cnt.n_R;
  a.n2 = h->n2;
  a.zcp = h->zcp;
  a.scores = h->scores;
  a.err = h->err;
  a.wait_ns = h->wait_ns;
  CUtensorMap xm;
  if (!encode_tokens_map(&xm, x, h->D, B, h->D, a.NP))
    return fail(h, POP_ERR_CUDA, "decode: cuTensorMapEncodeTiled failed for x");
  POP_CUDA(h, launch_gateup_slab(xm, a, h->num_sms, st));
  return POP_OK;
}

pop_status gateup_tc(pop_ffn* h, const uint16_t* x, int B, const int* rc, int nC, int nR, cudaStream_t st) {
  GateUpTcArgs a{};
  a.Wp = h->Wp;
  a.D = h->D;
  a.N = h->N;
  a.B = B;
  a.NP = round_up(B, 16);
  a.rc = rc;
  a.nC = nC;
  a.nR = nR;
  a.n2 = h->n2;
  a.zcp = h->zcp;
  a.scores = h->scores;
  a.err = h->err;
  a.wait_ns = h->wait_ns;
  CUtensorMap xm;
  if (!encode_tokens_map(&xm, x, h->D, B, h->D, a.NP))
    return fail(h, POP_ERR_CUDA, "decode: cuTensorMapEncodeTiled failed for x");
  POP_CUDA(h, launch_gateup_tc(xm, a, h->num_sms, st));
  return POP_OK;
}

// The selection of this decode step (decode: when there are candidates) and y[b] = sum over the
// kept items of z[b][item] W2[:, channel]: the nR items with channels ch_r[], then the k selected
// candidates. decode = false: the dense path (no selection, no step count).
pop_status down_tc(pop_ffn* h, int B, const int* ch_r, int nR, int k, bool decode, void* y, cudaStream_t st,
                   bool skip = false) {
  if (nR + k <= 0) {
    const size_t bytes = static_cast<size_t>(B) * h->D * (h->cfg.out_f32 ? 4 : 2);
    POP_CUDA(h, cudaMemsetAsync(y, 0, bytes, st));
  }
  DownTcArgs a{};
  a.Wp = h->Wp;
  a.D = h->D;
  a.N = h->N;
  a.B = B;
  a.NP = round_up(B, 16);
  a.nR = nR;
  a.kbr = (nR + 63) / 64;
  a.k = k;
  a.ch_r = ch_r;
  a.ch_s = h->ch_s;
  // R's z rows follow the list's candidates: |C| of the partition, the held selection's k on a skip
  // step, none in the dense path (every channel is an R item there)
  a.r_pos0 = decode ? (skip ? k : h->cnt.n_C) : 0;
  a.y = y;
  a.out_f32 = h->cfg.out_f32;
  a.dslab = decode ? h->dn_slab : nullptr;
  a.sel = decode && h->cnt.n_C > 0 ? 1 : 0;
  a.scores = h->scores;
  a.zcp = h->zcp;
  a.rc = h->rc;
  a.nC = skip ? k : h->cnt.n_C;  // a skip step's candidates are the held selection
  a.period = h->cfg.period;
  a.memory = h->memory;
  a.S = h->S;
  a.step = h->step;
  a.count_step = decode ? 1 : 0;
  a.flag = h->fsync + 5;
  a.epoch = decode ? ++h->epoch : 0;
  a.skip = skip ? 1 : 0;
  a.S_hold = h->S;
  a.rcs = h->cfg.skip && h->cfg.period > 1 ? h->rcs : nullptr;
  if (skip) {
    a.S = h->idx_all;  // the selected items are positions [0, k) of the skip list,
    a.ch_s = h->rcs;   // and their channels its head (written by whichever path ran the update)
  }
  a.err = h->err;
  a.wait_ns = h->wait_ns;
  CUtensorMap zm;
  if (!encode_zrows_map(&zm, h->zcp, a.r_pos0 + nR, a.NP))
    return fail(h, POP_ERR_CUDA, "decode: cuTensorMapEncodeTiled failed for the z rows");
  POP_CUDA(h, launch_down_tc(zm, a, h->num_sms, st));
  return POP_OK;
}

__global__ void k_iota(int* a, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) a[i] = i;
}
}  // namespace

void pop::set_unbound_error(const char* msg) { g_msg = msg; }

cudaError_t pop::ensure_dyn_smem(const void* kernel, size_t bytes) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, size_t> configured;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = configured[{kernel, dev}];
  if (bytes <= have) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
  if (e == cudaSuccess) have = bytes;
  return e;
}

extern "C" {

const char* pop_status_string(pop_status s) {
  switch (s) {
    case POP_OK: return "POP_OK";
    case POP_ERR_INVALID_ARG: return "POP_ERR_INVALID_ARG";
    case POP_ERR_STATE: return "POP_ERR_STATE";
    case POP_ERR_CUDA: return "POP_ERR_CUDA";
    case POP_ERR_OOM: return "POP_ERR_OOM";
    case POP_ERR_TIMEOUT: return "POP_ERR_TIMEOUT";
    case POP_ERR_UNSUPPORTED: return "POP_ERR_UNSUPPORTED";
    case POP_ERR_DEVICE: return "POP_ERR_DEVICE";
  }
  return "POP_ERR_UNKNOWN";
}

const char* pop_last_error(pop_ffn_t h) { return h ? h->msg.c_str() : g_msg.c_str(); }

pop_status pop_region_counts(int N, double r, double gamma, pop_counts* out) {
  if (!out) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_region_counts: out is NULL");
  if (!(r >= 0.0 && r <= 1.0) || !(gamma >= 0.0) || N < 0)
    return fail(nullptr, POP_ERR_INVALID_ARG, "pop_region_counts: need 0 <= r <= 1, gamma >= 0, N >= 0");
  double lo = r - gamma;
  if (lo < 0.0) lo = 0.0;
  double hi = r + gamma;
  if (hi > 1.0) hi = 1.0;
  pop_counts c;
  c.n_P = static_cast<int>(round_half_even(lo * N));
  c.n_R = N - static_cast<int>(round_half_even(hi * N));
  c.keep = N - static_cast<int>(round_half_even(r * N));
  c.k = c.keep - c.n_R;
  c.n_C = N - c.n_P - c.n_R;
  if (c.k < 0 || c.k > c.n_C)
    return fail(nullptr, POP_ERR_INVALID_ARG, "pop_region_counts: fill count outside [0, |C|]");
  *out = c;
  return POP_OK;
}

pop_status pop_ffn_create(const pop_config* cfg, const void* Wg, const void* W1, const void* W2, void* stream,
                          pop_ffn_t* out) {
  if (!out) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_create: out is NULL");
  *out = nullptr;
  if (!cfg || !Wg || !W1 || !W2) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_create: NULL argument");
  if (cfg->D < 8 || cfg->D > POP_MAX_D || cfg->D % 8 != 0)
    return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_create: D must be a multiple of 8 in [8, POP_MAX_D]");
  if (cfg->D_FF < 1 || cfg->D_FF > POP_MAX_D_FF)
    return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_create: D_FF must be in [1, POP_MAX_D_FF]");
  if (cfg->period < 1) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_create: period must be >= 1");
  if (cfg->max_batch < 1 || cfg->max_batch > POP_MAX_BATCH)
    return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_create: max_batch must be in [1, POP_MAX_BATCH]");
  if (cfg->max_prefill_tokens < 1)
    return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_create: max_prefill_tokens must be >= 1");
  if (cfg->skip != 0 && cfg->skip != 1) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_create: skip must be 0 or 1");
  if (!aligned16(Wg) || !aligned16(W1) || !aligned16(W2))
    return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_create: weights must be 16-byte aligned");
  pop_counts cnt;
  pop_status s = pop_region_counts(cfg->D_FF, cfg->r, cfg->gamma, &cnt);
  if (s != POP_OK) return s;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDevice");
  cudaDeviceProp prop;
  e = cudaGetDeviceProperties(&prop, dev);
  if (e != cudaSuccess) return cuda_fail(nullptr, e, "cudaGetDeviceProperties");
  if (!(prop.major == 10 && prop.minor == 3))
    return fail(nullptr, POP_ERR_UNSUPPORTED, "pop_ffn_create: this build targets sm_103a (GB300) only");

  pop_ffn* h = new pop_ffn();
  h->cfg = *cfg;
  h->cnt = cnt;
  h->D = cfg->D;
  h->N = cfg->D_FF;
  h->device = dev;
  h->num_sms = prop.multiProcessorCount;
  const int D = h->D, N = h->N;
  h->Mcap = round_up(cfg->max_prefill_tokens, 128);
  h->ldZ = round_up(N, 128);
  h->ldPart = h->ldZ;
  h->ypart_parts = 2 * h->num_sms;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  auto bail = [&](cudaError_t err, const char* where) {
    free_all(h);
    delete h;
    return cuda_fail(nullptr, err, where);
  };
#define POP_ALLOC(ptr, count)                                   \
  do {                                                          \
    cudaError_t e_ = dalloc(&(ptr), (count));                   \
    if (e_ != cudaSuccess) return bail(e_, "cudaMalloc " #ptr); \
  } while (0)
  POP_ALLOC(h->Wp, static_cast<size_t>(N) * 3 * D);
  POP_ALLOC(h->n2, N);
  POP_ALLOC(h->Z, 2 * static_cast<size_t>(h->Mcap) * h->ldZ);
  POP_ALLOC(h->part, static_cast<size_t>(h->Mcap / 32) * h->ldPart);
  POP_ALLOC(h->sumsq, N);
  POP_ALLOC(h->I, N);
  POP_ALLOC(h->rc, N);
  POP_ALLOC(h->P, N);
  POP_ALLOC(h->idx_all, N);
  POP_ALLOC(h->z, static_cast<size_t>(round_up(cfg->max_batch, 4)) * N);
  POP_ALLOC(h->scores, N);
  POP_ALLOC(h->memory, N);
  POP_ALLOC(h->S, N);
  POP_ALLOC(h->rcs, N);
  POP_ALLOC(h->ypart, static_cast<size_t>(h->ypart_parts) * D);
  if (cfg->max_batch > 1) {
    POP_ALLOC(h->ch_s, N);
    POP_ALLOC(h->zcp, static_cast<size_t>(N) * 2 * round_up(cfg->max_batch, 16));
    h->gu_geom = gu_slab_geom(cnt.n_C + cnt.n_R, D, h->num_sms);
    POP_ALLOC(h->gu_slab, gu_slab_elems(h->gu_geom));
    if (cfg->skip && cfg->period > 1 && cnt.n_C > 0) {
      h->gu_geom_skip = gu_slab_geom_split(cnt.k, cnt.k + cnt.n_R, D, h->num_sms);
      POP_ALLOC(h->gu_slab_skip, gu_slab_elems(h->gu_geom_skip));
    }
    POP_ALLOC(h->dn_slab, dn_slab_elems(D, cnt.n_R));
  }
  POP_ALLOC(h->step, 1);
  POP_ALLOC(h->err, 1);
  POP_ALLOC(h->fsync, kSyncWords);
#undef POP_ALLOC
  if ((e = cudaMemsetAsync(h->fsync, 0, kSyncWords * sizeof(unsigned), st)) != cudaSuccess)
    return bail(e, "cudaMemsetAsync");
  if ((e = cudaMemsetAsync(h->err, 0, sizeof(unsigned), st)) != cudaSuccess) return bail(e, "cudaMemsetAsync");
  if (h->ch_s && (e = cudaMemsetAsync(h->ch_s, 0, sizeof(int) * N, st)) != cudaSuccess)
    return bail(e, "cudaMemsetAsync");
  if ((e = cudaMemsetAsync(h->step, 0, sizeof(int), st)) != cudaSuccess) return bail(e, "cudaMemsetAsync");
  // index lists always hold valid positions, even before the first partition or selection
  if ((e = cudaMemsetAsync(h->S, 0, sizeof(int) * N, st)) != cudaSuccess) return bail(e, "cudaMemsetAsync");
  if ((e = cudaMemsetAsync(h->rc, 0, sizeof(int) * N, st)) != cudaSuccess) return bail(e, "cudaMemsetAsync");
  if ((e = cudaMemsetAsync(h->rcs, 0, sizeof(int) * N, st)) != cudaSuccess) return bail(e, "cudaMemsetAsync");
  k_iota<<<(N + 255) / 256, 256, 0, st>>>(h->idx_all, N);
  if ((e = cudaGetLastError()) != cudaSuccess) return bail(e, "k_iota");
  if ((e = launch_pack(static_cast<const uint16_t*>(Wg), static_cast<const uint16_t*>(W1),
                       static_cast<const uint16_t*>(W2), h->Wp, h->n2, D, N, st)) != cudaSuccess)
    return bail(e, "launch_pack");
  if (!encode_weight_maps(&h->maps, h->Wp, D, N)) {
    free_all(h);
    delete h;
    return fail(nullptr, POP_ERR_CUDA, "pop_ffn_create: cuTensorMapEncodeTiled failed");
  }
  *out = h;
  return POP_OK;
}

void pop_ffn_destroy(pop_ffn_t h) {
  if (!h) return;
  cudaDeviceSynchronize();
  destroy_events(h);
  free_all(h);
  delete h;
}

pop_status pop_ffn_counts(pop_ffn_t h, pop_counts* out) {
  if (!h || !out) return fail(h, POP_ERR_INVALID_ARG, "pop_ffn_counts: NULL argument");
  *out = h->cnt;
  return POP_OK;
}

pop_status pop_set_wait_limit(pop_ffn_t h, uint64_t ns) {
  if (!h || ns == 0) return fail(h, POP_ERR_INVALID_ARG, "pop_set_wait_limit: NULL handle or zero limit");
  h->wait_ns = ns;
  return POP_OK;
}

// Dense gate/up + down over M tokens through the tensor-core GEMMs (chunks of Mcap tokens).
// When `fold` is set, the channel sums of z^2 are accumulated into h->sumsq.
static pop_status prefill_gemms(pop_ffn* h, const uint16_t* X, int M, void* Y, bool fold, cudaStream_t st) {
  const size_t esz = h->cfg.out_f32 ? 4 : 2;
  for (int c0 = 0; c0 < M; c0 += h->Mcap) {
    const int Mc = std::min(h->Mcap, M - c0);
    uint16_t* Zlo = h->Z + static_cast<size_t>(h->Mcap) * h->ldZ;
    CUtensorMap xm, zm, zlm;
    if (!encode_x_map(&xm, X + static_cast<size_t>(c0) * h->D, Mc, h->D) ||
        !encode_z_map(&zm, h->Z, Mc, h->N, h->ldZ) || !encode_z_map(&zlm, Zlo, Mc, h->N, h->ldZ))
      return fail(h, POP_ERR_CUDA, "cuTensorMapEncodeTiled failed");
    POP_CUDA(h, launch_prefill_gateup(xm, h->maps, Mc, h->N, h->D, h->Z, Zlo, h->ldZ, h->part, h->ldPart, h->err,
                                      h->wait_ns, h->num_sms, st));
    if (fold)
      POP_CUDA(h, launch_fold_sumsq(h->part, 4 * ((Mc + 127) / 128), h->ldPart, h->N, h->sumsq, c0 > 0 ? 1 : 0, st));
    if (Y)
      POP_CUDA(h, launch_prefill_down(zm, zlm, h->maps, Mc, h->N, h->D,
                                      static_cast<uint8_t*>(Y) + static_cast<size_t>(c0) * h->D * esz,
                                      h->cfg.out_f32, h->err, h->wait_ns, h->num_sms, st));
  }
  return POP_OK;
}

pop_status pop_prefill_partition(pop_ffn_t h, const void* X, int M, void* Y, void* stream) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_prefill_partition: NULL handle");
  if (!X || M < 1) return fail(h, POP_ERR_INVALID_ARG, "pop_prefill_partition: X is NULL or M < 1");
  if (!aligned16(X) || (Y && !aligned16(Y)))
    return fail(h, POP_ERR_INVALID_ARG, "pop_prefill_partition: X and Y must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  pop_status s = prefill_gemms(h, static_cast<const uint16_t*>(X), M, Y, true, st);
  if (s != POP_OK) return s;
  POP_CUDA(h, launch_partition(h->sumsq, h->n2, h->I, h->N, h->cnt.n_P, h->cnt.n_R, h->rc, h->P, h->step,
                               h->memory, h->err, st));
  POP_CUDA(h, reset_counters(h, st));
  POP_CUDA(h, build_slabs(h, st));
  POP_CUDA(h, skip_list_tail(h, st));
  h->partitioned = true;
  h->selected = false;
  return POP_OK;
}

pop_status pop_partition_from_importance(pop_ffn_t h, const float* importance, void* stream) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_partition_from_importance: NULL handle");
  if (!importance) return fail(h, POP_ERR_INVALID_ARG, "pop_partition_from_importance: NULL importance");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  POP_CUDA(h, cudaMemcpyAsync(h->I, importance, sizeof(float) * h->N, cudaMemcpyDeviceToDevice, st));
  POP_CUDA(h, launch_partition(nullptr, h->n2, h->I, h->N, h->cnt.n_P, h->cnt.n_R, h->rc, h->P, h->step, h->memory,
                               h->err, st));
  POP_CUDA(h, reset_counters(h, st));
  POP_CUDA(h, build_slabs(h, st));
  POP_CUDA(h, skip_list_tail(h, st));
  h->partitioned = true;
  h->selected = false;
  return POP_OK;
}

pop_status pop_set_partition(pop_ffn_t h, const int* R, const int* C, const int* P, void* stream) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_set_partition: NULL handle");
  const int N = h->N, nR = h->cnt.n_R, nC = h->cnt.n_C, nP = h->cnt.n_P;
  if ((nR && !R) || (nC && !C) || (nP && !P)) return fail(h, POP_ERR_INVALID_ARG, "pop_set_partition: NULL list");
  std::vector<char> seen(N, 0);
  auto check = [&](const int* a, int n) {
    for (int i = 0; i < n; ++i) {
      if (a[i] < 0 || a[i] >= N || seen[a[i]] || (i > 0 && a[i] <= a[i - 1])) return false;
      seen[a[i]] = 1;
    }
    return true;
  };
  if (!check(R, nR) || !check(C, nC) || !check(P, nP))
    return fail(h, POP_ERR_INVALID_ARG, "pop_set_partition: lists must be ascending, disjoint and in [0, D_FF)");
  std::vector<int> rc(static_cast<size_t>(nC) + nR);
  if (nC) std::memcpy(rc.data(), C, sizeof(int) * nC);
  if (nR) std::memcpy(rc.data() + nC, R, sizeof(int) * nR);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!rc.empty())
    POP_CUDA(h, cudaMemcpyAsync(h->rc, rc.data(), sizeof(int) * rc.size(), cudaMemcpyHostToDevice, st));
  if (nP) POP_CUDA(h, cudaMemcpyAsync(h->P, P, sizeof(int) * nP, cudaMemcpyHostToDevice, st));
  POP_CUDA(h, cudaMemsetAsync(h->step, 0, sizeof(int), st));
  POP_CUDA(h, cudaMemsetAsync(h->memory, 0, sizeof(float) * (nC > 0 ? nC : 1), st));
  POP_CUDA(h, reset_counters(h, st));
  POP_CUDA(h, build_slabs(h, st));
  POP_CUDA(h, skip_list_tail(h, st));
  POP_CUDA(h, cudaStreamSynchronize(st));
  h->partitioned = true;
  h->selected = false;
  return POP_OK;
}

pop_status pop_decode_step(pop_ffn_t h, const void* x, int B, void* y, void* stream) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_decode_step: NULL handle");
  if (!x || !y) return fail(h, POP_ERR_INVALID_ARG, "pop_decode_step: NULL x or y");
  if (B < 1 || B > h->cfg.max_batch)
    return fail(h, POP_ERR_INVALID_ARG, "pop_decode_step: B outside [1, max_batch]");
  if (!aligned16(x) || !aligned16(y))
    return fail(h, POP_ERR_INVALID_ARG, "pop_decode_step: x, y must be 16-byte aligned");
  if (!h->partitioned) return fail(h, POP_ERR_STATE, "pop_decode_step: no partition (run a prefill first)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int nC = h->cnt.n_C, nR = h->cnt.n_R, k = h->cnt.k;
  // skip variant: steps between updates run over R and the held selection only (the device step
  // counter advances with every step, so the host's mirror tells the update steps apart)
  const bool skip_mode = h->cfg.skip && h->cfg.period > 1 && nC > 0;
  const bool skip = skip_mode && (h->host_step % h->cfg.period) != 0;
  int* rcs = skip_mode ? h->rcs : nullptr;
  prof_begin(h);
  if (B == 1) {
    const int grid = h->num_sms * 4;
    DecodeB1Args a = skip ? b1_args(h, static_cast<const uint16_t*>(x), y, h->rcs, k, nR)
                          : b1_args(h, static_cast<const uint16_t*>(x), y, h->rc, nC, nR);
    a.do_select = skip || nC <= FZ_MAX_C ? 1 : 0;
    a.skip = skip ? 1 : 0;
    a.S_hold = h->S;
    a.rcs = rcs;
    a.k = k;
    a.kd = k;
    if (skip) a.S = h->idx_all;  // the down projection's selected items: positions [0, k) of the list
    prof_mark(h, 0, st);
    POP_CUDA(h, launch_gateup_sel_b1(a, grid, st));
    prof_mark(h, 1, st);
    if (!a.do_select)
      POP_CUDA(h, launch_select(h->scores, h->memory, nC, k, h->cfg.period, h->step, h->S, h->rc, rcs, h->err, st));
    prof_mark(h, 2, st);
    POP_CUDA(h, launch_down_tiled_b1(a, h->num_sms, st));
    prof_mark(h, 3, st);
    // skip variant, update step: a later B > 1 skip step streams the slab of this selection's list
    if (skip_mode && !skip && h->gu_slab_skip)
      POP_CUDA(h, launch_build_gu_tiles(h->Wp, h->rcs, h->D, h->N, h->gu_geom_skip, 0, h->gu_geom_skip.Ts,
                                        h->gu_slab_skip, h->err, st));
    prof_mark(h, 4, st);
  } else {
    // gate/up, then the down GEMM over R and the selected items with the selection inside; a skip
    // step gathers the rows of R and of the held selection instead of streaming the slab
    prof_mark(h, 0, st);
    pop_status s = gateup_slab(h, static_cast<const uint16_t*>(x), B, st, skip);
    if (s != POP_OK) return s;
    prof_mark(h, 1, st);
    prof_mark(h, 2, st);
    s = down_tc(h, B, h->rc + nC, nR, k, true, y, st, skip);
    if (s != POP_OK) return s;
    prof_mark(h, 3, st);
    // skip variant, update step: the slab of [C[S] | R] for the steps until the next update (an
    // ordinary launch: it starts once the selection's list is complete)
    if (skip_mode && !skip && h->gu_slab_skip)
      POP_CUDA(h, launch_build_gu_tiles(h->Wp, h->rcs, h->D, h->N, h->gu_geom_skip, 0, h->gu_geom_skip.Ts,
                                        h->gu_slab_skip, h->err, st));
    prof_mark(h, 4, st);
  }
  prof_end(h);
  ++h->host_step;
  h->selected = true;
  return POP_OK;
}

pop_status pop_ffn_dense_ref(pop_ffn_t h, const void* X, int M, void* Y, void* stream) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_ffn_dense_ref: NULL handle");
  if (!X || !Y || M < 1) return fail(h, POP_ERR_INVALID_ARG, "pop_ffn_dense_ref: NULL X/Y or M < 1");
  if (!aligned16(X) || !aligned16(Y))
    return fail(h, POP_ERR_INVALID_ARG, "pop_ffn_dense_ref: X, Y must be 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (M > h->cfg.max_batch) return prefill_gemms(h, static_cast<const uint16_t*>(X), M, Y, false, st);
  if (M == 1) {
    DecodeB1Args a = b1_args(h, static_cast<const uint16_t*>(X), Y, h->idx_all, 0, h->N);
    POP_CUDA(h, launch_gateup_sel_b1(a, h->num_sms * 4, st));
    POP_CUDA(h, launch_down_tiled_b1(a, h->num_sms, st));
    return POP_OK;
  }
  // 2 <= M <= max_batch: the decode kernels over every channel (all positions count as retained)
  pop_status s = gateup_tc(h, static_cast<const uint16_t*>(X), M, h->idx_all, 0, h->N, st);
  if (s != POP_OK) return s;
  return down_tc(h, M, h->idx_all, h->N, 0, false, Y, st);
}

pop_status pop_get_partition(pop_ffn_t h, int* R, int* C, int* P) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_get_partition: NULL handle");
  if (!h->partitioned) return fail(h, POP_ERR_STATE, "pop_get_partition: no partition yet");
  POP_CUDA(h, cudaDeviceSynchronize());
  const int nC = h->cnt.n_C, nR = h->cnt.n_R, nP = h->cnt.n_P;
  if (C && nC) POP_CUDA(h, cudaMemcpy(C, h->rc, sizeof(int) * nC, cudaMemcpyDeviceToHost));
  if (R && nR) POP_CUDA(h, cudaMemcpy(R, h->rc + nC, sizeof(int) * nR, cudaMemcpyDeviceToHost));
  if (P && nP) POP_CUDA(h, cudaMemcpy(P, h->P, sizeof(int) * nP, cudaMemcpyDeviceToHost));
  return POP_OK;
}

pop_status pop_get_importance(pop_ffn_t h, float* importance, float* sumsq) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_get_importance: NULL handle");
  POP_CUDA(h, cudaDeviceSynchronize());
  if (importance) POP_CUDA(h, cudaMemcpy(importance, h->I, sizeof(float) * h->N, cudaMemcpyDeviceToHost));
  if (sumsq) POP_CUDA(h, cudaMemcpy(sumsq, h->sumsq, sizeof(float) * h->N, cudaMemcpyDeviceToHost));
  return POP_OK;
}

pop_status pop_get_selected(pop_ffn_t h, int* k_out, int* channels) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_get_selected: NULL handle");
  if (!h->selected) return fail(h, POP_ERR_STATE, "pop_get_selected: no decode step since the partition was set");
  if (k_out) *k_out = h->cnt.k;
  if (!channels || h->cnt.k == 0) return POP_OK;
  POP_CUDA(h, cudaDeviceSynchronize());
  std::vector<int> S(h->cnt.k), C(h->cnt.n_C);
  POP_CUDA(h, cudaMemcpy(S.data(), h->S, sizeof(int) * S.size(), cudaMemcpyDeviceToHost));
  POP_CUDA(h, cudaMemcpy(C.data(), h->rc, sizeof(int) * C.size(), cudaMemcpyDeviceToHost));
  for (int j = 0; j < h->cnt.k; ++j) {
    if (S[j] < 0 || S[j] >= h->cnt.n_C) return fail(h, POP_ERR_DEVICE, "pop_get_selected: position out of range");
    channels[j] = C[S[j]];
  }
  return POP_OK;
}

pop_status pop_get_scores(pop_ffn_t h, float* scores, float* memory) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_get_scores: NULL handle");
  POP_CUDA(h, cudaDeviceSynchronize());
  const int nC = h->cnt.n_C;
  if (scores && nC) POP_CUDA(h, cudaMemcpy(scores, h->scores, sizeof(float) * nC, cudaMemcpyDeviceToHost));
  if (memory && nC) POP_CUDA(h, cudaMemcpy(memory, h->memory, sizeof(float) * nC, cudaMemcpyDeviceToHost));
  return POP_OK;
}

pop_status pop_get_step(pop_ffn_t h, int* step) {
  if (!h || !step) return fail(h, POP_ERR_INVALID_ARG, "pop_get_step: NULL argument");
  POP_CUDA(h, cudaDeviceSynchronize());
  POP_CUDA(h, cudaMemcpy(step, h->step, sizeof(int), cudaMemcpyDeviceToHost));
  return POP_OK;
}

pop_status pop_profile_enable(pop_ffn_t h, int enable) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_profile_enable: NULL handle");
  POP_CUDA(h, cudaDeviceSynchronize());
  destroy_events(h);
  if (enable <= 0) return POP_OK;
  h->prof_stride = enable;
  h->prof_events.resize(static_cast<size_t>(kProfEvents) * kProfMaxSteps);
  for (auto& e : h->prof_events) {
    cudaError_t r = cudaEventCreate(&e);
    if (r != cudaSuccess) {
      e = nullptr;
      h->prof_events.erase(std::remove(h->prof_events.begin(), h->prof_events.end(), nullptr), h->prof_events.end());
      destroy_events(h);
      return cuda_fail(h, r, "cudaEventCreate");
    }
  }
  return POP_OK;
}

pop_status pop_profile_read(pop_ffn_t h, double* ms, int* steps) {
  if (!h || !ms || !steps) return fail(h, POP_ERR_INVALID_ARG, "pop_profile_read: NULL argument");
  for (int i = 0; i < kProfEvents - 1; ++i) ms[i] = 0.0;
  *steps = h->prof_steps;
  if (h->prof_events.empty()) return fail(h, POP_ERR_STATE, "pop_profile_read: profiling is not enabled");
  POP_CUDA(h, cudaDeviceSynchronize());
  for (int s = 0; s < h->prof_steps; ++s) {
    for (int i = 0; i < kProfEvents - 1; ++i) {
      float t = 0.f;
      POP_CUDA(h, cudaEventElapsedTime(&t, h->prof_events[static_cast<size_t>(s) * kProfEvents + i],
                                       h->prof_events[static_cast<size_t>(s) * kProfEvents + i + 1]));
      ms[i] += t;
    }
  }
  h->prof_steps = 0;
  return POP_OK;
}

pop_status pop_check(pop_ffn_t h) {
  if (!h) return fail(nullptr, POP_ERR_INVALID_ARG, "pop_check: NULL handle");
  POP_CUDA(h, cudaDeviceSynchronize());
  unsigned e = 0;
  POP_CUDA(h, cudaMemcpy(&e, h->err, sizeof(unsigned), cudaMemcpyDeviceToHost));
  if (e == 0) return POP_OK;
  POP_CUDA(h, cudaMemset(h->err, 0, sizeof(unsigned)));
  POP_CUDA(h, reset_counters(h, nullptr));
  POP_CUDA(h, cudaDeviceSynchronize());
  // a step that gave up may not have counted itself: the host's mirror follows the device counter
  int dstep = 0;
  POP_CUDA(h, cudaMemcpy(&dstep, h->step, sizeof(int), cudaMemcpyDeviceToHost));
  h->host_step = dstep;
  char buf[240];
  std::snprintf(buf, sizeof buf,
                "device error word 0x%x (1/2/32/64: prefill gate-up / prefill down / decode selector / decode "
                "tensor-core wait ran out; 4: partition; 8: top-k; 16: index)", e);
  return fail(h, (e & DEVERR_TIMEOUT_ANY) ? POP_ERR_TIMEOUT : POP_ERR_DEVICE, buf);
}

}  // extern "C"
