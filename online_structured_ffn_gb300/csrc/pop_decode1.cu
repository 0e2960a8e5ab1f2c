// Decode step of the POP FFN for one token (B = 1): two launches, no waits between CTAs.
//
// ("POP: Online Structural Pruning..." notes, Key design 2: H_t = f(X_t; R u C), score only C,
// fill |R| + k survivors; "Batch-wise adaptive pruning", abstract: periodic top-k with an
// activation memory.)
//
// Launch 1, k_gateup_sel_b1: gate/up over R u C, one warp per channel streaming the channel's two
// contiguous rows with 16-byte loads. Every worker warp scores its share of the candidates before
// it streams its share of R, so all candidate scores exist a few microseconds into the kernel.
// CTA 0 streams nothing: it waits (bounded) until the candidate count is complete, then runs the
// periodic memory update and the top-k while the workers are still streaming R, so the selection
// costs no time on the critical path. Progress is guaranteed: the workers wait on nobody, so CTA 0
// never holds up a CTA it waits for, even when the grid does not fit on the GPU at once.
//
// Launch 2, k_down_tiled_b1: y = sum over R u S of z_i W2[:, i]. CTA (t, c) owns the 256-wide
// tile t of y and the c-th chunk of the kept channels; 16 groups of 32 threads each read one
// channel's 512-byte slice of the contiguous down column with 16-byte loads. The last chunk CTA to
// finish a tile (atomic counter) adds the chunks' partial tiles in a fixed order: no extra
// launch, and the result does not depend on timing. (512-wide tiles, twice the chunks per tile,
// were 0.2 us slower per step at the LLaMA-2-7B FFN shape; 1024-wide ones 4.3 us.)
//
// Both kernels are launched with programmatic dependent launch when the caller's stream allows it.
// Before waiting for the previous kernel (griddepcontrol.wait) they touch constant data only: in
// the gate/up kernel an L2 prefetch of each warp's first load group, in the down kernel the
// channel ids of R, which only a partition changes; a partition is written by ordinary launches
// that have completed before the gate/up grid passes its wait, and the gate/up grid lets the down
// grid start only after that wait. x, z and S are read and z, S, y written only after the wait,
// so the overlap with the previous kernel's tail never races on data.
//
// The prefetch is kept small on purpose. CTAs that become resident during the previous kernel's
// tail share the memory system with it: a whole 16 KB channel per warp (80 MB over the grid) held
// back the previous grid's completion, and with it this grid's wait, by about 3 us, and an L2
// prefetch of all of R's down slices in the down kernel slowed the gate/up tail it overlapped by
// more than it saved. B = 1 decode step at the LLaMA-2-7B FFN shape: 42.2 us with both, 38.5 us
// with 2 KB + 2 KB per warp and no down prefetch, 37.4 us with 32 KB of down slices per down CTA
// added (1 + 1 KB per gate/up warp: 39.2 us; 4 + 4 KB: 39.0 us; 64 KB: 37.6 us).
#include "pop_device.cuh"
#include "pop_internal.h"
#include "pop_radix.cuh"

namespace pop {

namespace {
constexpr int GS_THREADS = 256;
constexpr int GS_WARPS = GS_THREADS / 32;
constexpr int DT_THREADS = 512;
constexpr int DT_TILE = B1_DOWN_TILE;  // outputs per tile: 32 threads x 8
static_assert(DT_TILE == 256, "the thread layout below assumes 256-wide tiles");
constexpr int DT_GROUPS = DT_THREADS / (DT_TILE / 8);
constexpr int DT_BATCH = 512;  // kept channels staged in shared memory at a time
constexpr int DT_UNROLL = 8;
constexpr int DT_PREFETCH = 64;  // retained items per down CTA whose slices are prefetched before the wait

struct BlockSync256 {
  __device__ void operator()() const { __syncthreads(); }
};

__device__ __forceinline__ int guard_idx(int v, int n, unsigned* err) {
  if (static_cast<unsigned>(v) >= static_cast<unsigned>(n)) {
    atomicOr(err, DEVERR_INDEX);
    return 0;
  }
  return v;
}

__device__ __forceinline__ float silu_1(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}
// One atomic that publishes this CTA's earlier writes (ordered before it by a CTA barrier) and,
// for the caller that sees the final count, makes the other CTAs' published writes visible.
__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}
__device__ __forceinline__ void red_add_release(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
}  // namespace

template <int NCHL>
__global__ void __launch_bounds__(GS_THREADS, 4) k_gateup_sel_b1(const __grid_constant__ DecodeB1Args a) {
  extern __shared__ float xs[];  // D floats of x (workers) or nC keys (selector)
  __shared__ RadixScratch<GS_THREADS> sc;
  __shared__ int s_ok;
  const int D = a.D;
  const int G = gridDim.x, cta = blockIdx.x;

  if (cta == 0) {
    // ---------------------------------------------------------------- selector
    pdl_wait();     // S, memory and step may still be read by the previous step's kernels
    pdl_trigger();  // the next kernel may take free SM slots; it waits for this grid before using S
    if (a.do_select) {
      if (threadIdx.x == 0) {
        bool ok = true;
        if (a.nC > 0) {
          const uint64_t t0 = globaltimer_ns();
          while (ld_acquire_u32(a.sync) < static_cast<unsigned>(a.nC)) {
            __nanosleep(200);
            if (globaltimer_ns() - t0 > a.wait_ns) {
              ok = false;
              break;
            }
          }
        }
        if (ok) atomicExch(a.sync, 0u);  // every candidate has been counted: ready for the next step
        else atomicOr(a.err, DEVERR_TIMEOUT_DECODE);
        __threadfence();
        s_ok = ok;
      }
      __syncthreads();
      if (s_ok && a.skip) {
        // skip variant between updates: the candidates scored are the held selection (position j
        // of this step's list is S_hold[j]); their scores join the memory, nothing is selected
        const int t = *a.step;
        for (int j = threadIdx.x; j < a.nC; j += GS_THREADS) {
          int ps = __ldg(a.S_hold + j);
          if (static_cast<unsigned>(ps) >= static_cast<unsigned>(a.N)) {
            atomicOr(a.err, DEVERR_INDEX);
            ps = 0;
          }
          a.memory[ps] += __ldcg(a.scores + j);
        }
        __syncthreads();
        if (threadIdx.x == 0) *a.step = t + 1;
      } else if (s_ok) {
        uint32_t* keys = reinterpret_cast<uint32_t*>(xs);
        const int t = *a.step;
        const bool update = (t % a.period) == 0;
        const bool sel = select_step<GS_THREADS>(
            threadIdx.x, [&](int i) { return __ldcg(a.scores + i); }, a.memory, a.nC, a.k, a.period, update, keys,
            a.S, sc, BlockSync256());
        __syncthreads();
        if (a.rcs && update)  // skip variant: the next steps' list starts with the selected channels
          for (int j = threadIdx.x; j < a.k; j += GS_THREADS) {
            int ps = a.S[j];
            if (static_cast<unsigned>(ps) >= static_cast<unsigned>(a.nC)) {
              atomicOr(a.err, DEVERR_INDEX);
              ps = 0;
            }
            a.rcs[j] = a.rc[ps];
          }
        if (threadIdx.x == 0) {
          if (!sel) atomicOr(a.err, DEVERR_TOPK);
          *a.step = t + 1;
        }
      }
    }
    return;
  }

  // ------------------------------------------------------------------ workers
  const int W = G - 1, j = cta - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // 32-bit splits (the launcher checks that the products fit): 64-bit division is slow here
  const unsigned uW = static_cast<unsigned>(W), uj = static_cast<unsigned>(j);
  const int cb0 = static_cast<int>(uj * static_cast<unsigned>(a.nC) / uW);
  const int cb1 = static_cast<int>((uj + 1u) * static_cast<unsigned>(a.nC) / uW);
  const int rb0 = a.nC + static_cast<int>(uj * static_cast<unsigned>(a.nR) / uW);
  const int rb1 = a.nC + static_cast<int>((uj + 1u) * static_cast<unsigned>(a.nR) / uW);
  const int c0 = cb0 + warp * (cb1 - cb0) / GS_WARPS, c1 = cb0 + (warp + 1) * (cb1 - cb0) / GS_WARPS;
  const int r0 = rb0 + warp * (rb1 - rb0) / GS_WARPS, r1 = rb0 + (warp + 1) * (rb1 - rb0) / GS_WARPS;
  const int nch = D >> 3;
  const size_t row3 = 3 * static_cast<size_t>(D);
  constexpr int GRP = NCHL < 4 ? NCHL : 4;  // 16-byte loads per lane and row in flight at once
  // constant data only before the wait: warm L2 with the first load group of this warp's first
  // channel, GRP x 512 bytes of its gate row and of its up row, one 128-byte line per lane (on a
  // skip step the list's head, the held selection, may be written by the kernel before: R only)
  {
    const int p = c0 < c1 && !a.skip ? c0 : (r0 < r1 ? r0 : -1);
    if (p >= 0 && lane < 4 * GRP && 64 * lane < D) {
      const int ch = __ldcg(a.rc + p);
      if (static_cast<unsigned>(ch) < static_cast<unsigned>(a.N)) {
        const uint16_t* rg = a.Wp + static_cast<size_t>(ch) * row3 + 64 * lane;
        prefetch_l2(rg);
        prefetch_l2(rg + D);
      }
    }
  }
  pdl_wait();
  pdl_trigger();  // after the wait: the partition this grid reads is then complete for the next grid too
  for (int c = threadIdx.x; c < nch; c += GS_THREADS) {
    const uint4 v = *reinterpret_cast<const uint4*>(a.x + 8 * c);
    reinterpret_cast<float4*>(xs + 8 * c)[0] = make_float4(bf16lo(v.x), bf16hi(v.x), bf16lo(v.y), bf16hi(v.y));
    reinterpret_cast<float4*>(xs + 8 * c)[1] = make_float4(bf16lo(v.z), bf16hi(v.z), bf16lo(v.w), bf16hi(v.w));
  }
  __syncthreads();

  auto item = [&](int p) {
    const int ch = guard_idx(__ldcg(a.rc + p), a.N, a.err);
    const uint16_t* rg = a.Wp + static_cast<size_t>(ch) * row3;
    const uint16_t* ru = rg + D;
    float ag0 = 0.f, ag1 = 0.f, au0 = 0.f, au1 = 0.f;
#pragma unroll 1
    for (int j0 = 0; j0 < NCHL; j0 += GRP) {
      uint4 vg[GRP], vu[GRP];
#pragma unroll
      for (int q = 0; q < GRP; ++q) {
        const int c = lane + 32 * (j0 + q);
        if (c < nch) {
          vg[q] = ldg_stream(rg + 8 * c);
          vu[q] = ldg_stream(ru + 8 * c);
        } else {
          vg[q] = make_uint4(0u, 0u, 0u, 0u);
          vu[q] = vg[q];
        }
      }
#pragma unroll
      for (int q = 0; q < GRP; ++q) {
        const int c = lane + 32 * (j0 + q);
        if (c < nch) {
          const float4 xa = *reinterpret_cast<const float4*>(xs + 8 * c);
          const float4 xb = *reinterpret_cast<const float4*>(xs + 8 * c + 4);
          ag0 = fmaf(bf16lo(vg[q].x), xa.x, ag0);
          ag1 = fmaf(bf16hi(vg[q].x), xa.y, ag1);
          ag0 = fmaf(bf16lo(vg[q].y), xa.z, ag0);
          ag1 = fmaf(bf16hi(vg[q].y), xa.w, ag1);
          ag0 = fmaf(bf16lo(vg[q].z), xb.x, ag0);
          ag1 = fmaf(bf16hi(vg[q].z), xb.y, ag1);
          ag0 = fmaf(bf16lo(vg[q].w), xb.z, ag0);
          ag1 = fmaf(bf16hi(vg[q].w), xb.w, ag1);
          au0 = fmaf(bf16lo(vu[q].x), xa.x, au0);
          au1 = fmaf(bf16hi(vu[q].x), xa.y, au1);
          au0 = fmaf(bf16lo(vu[q].y), xa.z, au0);
          au1 = fmaf(bf16hi(vu[q].y), xa.w, au1);
          au0 = fmaf(bf16lo(vu[q].z), xb.x, au0);
          au1 = fmaf(bf16hi(vu[q].z), xb.y, au1);
          au0 = fmaf(bf16lo(vu[q].w), xb.z, au0);
          au1 = fmaf(bf16hi(vu[q].w), xb.w, au1);
        }
      }
    }
    float ag = ag0 + ag1, au = au0 + au1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ag += __shfl_xor_sync(0xffffffffu, ag, o);
      au += __shfl_xor_sync(0xffffffffu, au, o);
    }
    if (lane == 0) {
      const float zz = silu_1(ag) * au;
      a.z[p] = zz;
      if (p < a.nC) a.scores[p] = fabsf(zz) * a.n2[ch];
    }
  };

  for (int p = c0; p < c1; ++p) item(p);
  if (a.do_select && c1 > c0 && lane == 0) red_add_release(a.sync, static_cast<unsigned>(c1 - c0));
  for (int p = r0; p < r1; ++p) item(p);
}

__global__ void __launch_bounds__(DT_THREADS, 2) k_down_tiled_b1(const __grid_constant__ DecodeB1Args a) {
  __shared__ int s_ch[DT_BATCH];
  __shared__ float s_z[DT_BATCH];
  __shared__ __align__(16) float red[DT_GROUPS][DT_TILE];
  __shared__ int s_last;
  const int D = a.D;
  const int tile = blockIdx.x, chunk = blockIdx.y, NCK = gridDim.y;
  const int grp = threadIdx.x / (DT_TILE / 8), tt = threadIdx.x % (DT_TILE / 8);
  const int d = tile * DT_TILE + 8 * tt;
  const bool dok = d < D;
  // chunk c takes the c-th share of R and the c-th share of S, so every CTA streams the same
  // number of columns
  const unsigned uc = static_cast<unsigned>(chunk), un = static_cast<unsigned>(NCK);
  const int r_lo = static_cast<int>(uc * static_cast<unsigned>(a.nR) / un);
  const int nr = static_cast<int>((uc + 1u) * static_cast<unsigned>(a.nR) / un) - r_lo;
  const int s_lo = static_cast<int>(uc * static_cast<unsigned>(a.kd) / un);
  const int ns = static_cast<int>((uc + 1u) * static_cast<unsigned>(a.kd) / un) - s_lo;
  const int n_items = nr + ns;  // item e < nr is R item r_lo + e, else S item s_lo + e - nr
  const size_t row3 = 3 * static_cast<size_t>(D);
  const uint16_t* W2 = a.Wp + 2 * static_cast<size_t>(D);  // down part of packed row 0
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  // Constant data only before the wait: the channel ids of the first batch's retained items (R
  // never changes between partitions, and a partition is written by an ordinary launch that has
  // finished before this grid's primary started), and an L2 prefetch of the down slices of the
  // first DT_PREFETCH of them, one 128-byte line per thread.
  const int nr0 = min(DT_BATCH, nr);
  for (int e = threadIdx.x; e < nr0; e += DT_THREADS) s_ch[e] = guard_idx(__ldcg(a.rc + a.nC + r_lo + e), a.N, a.err);
  __syncthreads();
  {
    constexpr int LPS = DT_TILE * 2 / 128;  // 128-byte lines per tile slice
    static_assert(DT_PREFETCH * LPS <= DT_THREADS, "one prefetch per thread");
    const int q = threadIdx.x;
    const int dd = tile * DT_TILE + (q % LPS) * 64;
    if (q < min(nr0, DT_PREFETCH) * LPS && dd < D) prefetch_l2(W2 + static_cast<size_t>(s_ch[q / LPS]) * row3 + dd);
  }
  pdl_trigger();
  pdl_wait();

  for (int base = 0; base < n_items; base += DT_BATCH) {
    const int cnt = min(DT_BATCH, n_items - base);
    const bool first = base == 0;
    if (!first) __syncthreads();
    for (int e = threadIdx.x; e < cnt; e += DT_THREADS) {
      const int it = base + e;
      if (it < nr) {
        if (!first) s_ch[e] = guard_idx(__ldcg(a.rc + a.nC + r_lo + it), a.N, a.err);
        s_z[e] = a.z[a.nC + r_lo + it];
      } else {
        const int pos = guard_idx(a.S[s_lo + it - nr], a.nC, a.err);
        s_ch[e] = guard_idx(__ldcg(a.rc + pos), a.N, a.err);
        s_z[e] = a.z[pos];
      }
    }
    __syncthreads();
    for (int ii = grp; ii < cnt; ii += DT_GROUPS * DT_UNROLL) {
      uint4 v[DT_UNROLL];
      float zz[DT_UNROLL];
#pragma unroll
      for (int u = 0; u < DT_UNROLL; ++u) {
        const int idx = ii + DT_GROUPS * u;
        const bool ok = idx < cnt && dok;
        v[u] = ok ? ldg_stream(W2 + static_cast<size_t>(s_ch[idx]) * row3 + d) : make_uint4(0u, 0u, 0u, 0u);
        zz[u] = idx < cnt ? s_z[idx] : 0.f;
      }
#pragma unroll
      for (int u = 0; u < DT_UNROLL; ++u) {
        acc[0] = fmaf(bf16lo(v[u].x), zz[u], acc[0]);
        acc[1] = fmaf(bf16hi(v[u].x), zz[u], acc[1]);
        acc[2] = fmaf(bf16lo(v[u].y), zz[u], acc[2]);
        acc[3] = fmaf(bf16hi(v[u].y), zz[u], acc[3]);
        acc[4] = fmaf(bf16lo(v[u].z), zz[u], acc[4]);
        acc[5] = fmaf(bf16hi(v[u].z), zz[u], acc[5]);
        acc[6] = fmaf(bf16lo(v[u].w), zz[u], acc[6]);
        acc[7] = fmaf(bf16hi(v[u].w), zz[u], acc[7]);
      }
    }
  }
  reinterpret_cast<float4*>(&red[grp][8 * tt])[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  reinterpret_cast<float4*>(&red[grp][8 * tt])[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  const int e = tile * DT_TILE + threadIdx.x;
  if (threadIdx.x < DT_TILE && e < D) {
    float s = 0.f;
#pragma unroll
    for (int g = 0; g < DT_GROUPS; ++g) s += red[g][threadIdx.x];
    a.ypart[static_cast<size_t>(chunk) * D + e] = s;
  }
  // release this chunk's partial tile; the last chunk CTA of the tile adds all of them
  __syncthreads();
  if (threadIdx.x == 0) s_last = atom_add_acq_rel(a.tile_cnt + tile, 1u) == static_cast<unsigned>(NCK) - 1u;
  __syncthreads();
  if (!s_last) return;
  // DT_THREADS / (DT_TILE / 4) subsets of the chunks, each summed in chunk order over float4
  // columns, then the subsets in order: a fixed order, so y does not depend on timing.
  constexpr int QPT = DT_TILE / 4;             // float4 columns of the tile
  constexpr int NSUB = DT_THREADS / QPT;       // chunk subsets
  static_assert(NSUB * QPT == DT_THREADS && NSUB <= DT_GROUPS, "tile reduction layout");
  const int qc = threadIdx.x % QPT, sub = threadIdx.x / QPT;
  const int e4 = tile * DT_TILE + 4 * qc;
  float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
  if (e4 < D) {
    // D is a multiple of 8, so a float4 column inside y lies wholly inside it. The chunks are
    // loaded 12 at a time (a 7B-sized tile has 19 chunks: one round of loads per thread) and
    // added in chunk order.
    constexpr int RL = 12;
    for (int c0 = sub; c0 < NCK; c0 += RL * NSUB) {
      float4 v[RL];
#pragma unroll
      for (int u = 0; u < RL; ++u) {
        const int c = c0 + u * NSUB;
        v[u] = c < NCK ? __ldcg(reinterpret_cast<const float4*>(a.ypart + static_cast<size_t>(c) * D + e4))
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < RL; ++u) {
        if (c0 + u * NSUB < NCK) {
          t4.x += v[u].x;
          t4.y += v[u].y;
          t4.z += v[u].z;
          t4.w += v[u].w;
        }
      }
    }
  }
  reinterpret_cast<float4*>(&red[sub][0])[qc] = t4;
  __syncthreads();
  if (threadIdx.x < DT_TILE && e < D) {
    float t = 0.f;
#pragma unroll
    for (int g = 0; g < NSUB; ++g) t += red[g][threadIdx.x];
    if (a.out_f32)
      static_cast<float*>(a.y)[e] = t;
    else
      static_cast<__nv_bfloat16*>(a.y)[e] = __float2bfloat16_rn(t);
  }
  if (threadIdx.x == 0) atomicExch(a.tile_cnt + tile, 0u);
}

// ------------------------------------------------------------------ launchers
static int pow2_ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

template <class K>
static cudaError_t launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const DecodeB1Args& a) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

// the kernels split work with 32-bit products (part index x item count)
static bool split_fits(long long parts, long long items) { return parts * items < (1LL << 32); }

cudaError_t launch_gateup_sel_b1(const DecodeB1Args& a, int grid, cudaStream_t st) {
  if (!split_fits(grid, a.nC > a.nR ? a.nC : a.nR)) return cudaErrorInvalidValue;
  const int nchl = pow2_ceil((a.D / 8 + 31) / 32);
  const size_t keys = a.do_select && !a.skip ? static_cast<size_t>(a.nC > 0 ? a.nC : 1) * sizeof(uint32_t) : 0;
  const size_t xsz = static_cast<size_t>(a.D) * sizeof(float);
  const size_t smem = keys > xsz ? keys : xsz;
#define POP_GS(NC)                                                                                              \
  case NC: {                                                                                                    \
    {                                                                                                           \
      cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(k_gateup_sel_b1<NC>), smem);                \
      if (e != cudaSuccess) return e;                                                                           \
    }                                                                                                           \
    { cudaError_t e = launch_pdl(k_gateup_sel_b1<NC>, dim3(grid), dim3(GS_THREADS), smem, st, a);             \
      if (e != cudaSuccess) return e; }                                                                         \
    break;                                                                                                      \
  }
  switch (nchl) {
    POP_GS(1) POP_GS(2) POP_GS(4) POP_GS(8) POP_GS(16) POP_GS(32) POP_GS(64)
    default: return cudaErrorInvalidValue;
  }
#undef POP_GS
  return cudaGetLastError();
}

int down_tiled_chunks(int D, int nitems, int num_sms) {
  const int tiles = (D + DT_TILE - 1) / DT_TILE;
  int nck = (2 * num_sms + tiles - 1) / tiles;
  if (nck > nitems) nck = nitems;
  return nck < 1 ? 1 : nck;
}

cudaError_t launch_down_tiled_b1(const DecodeB1Args& a, int num_sms, cudaStream_t st) {
  const int tiles = (a.D + DT_TILE - 1) / DT_TILE;
  const int nck = down_tiled_chunks(a.D, a.nR + a.kd, num_sms);
  if (!split_fits(nck, a.nR > a.kd ? a.nR : a.kd)) return cudaErrorInvalidValue;
  return launch_pdl(k_down_tiled_b1, dim3(tiles, nck), dim3(DT_THREADS), 0, st, a);
}

}  // namespace pop
