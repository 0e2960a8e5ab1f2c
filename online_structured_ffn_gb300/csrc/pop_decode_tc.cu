// Decode step of the POP FFN for B > 1 sequences on the 5th-generation tensor cores: two launches.
//
// What it computes ("POP: Online Structural Pruning..." notes, Key design 2; "Batch-wise adaptive
// pruning", Fig. 2(a) for the batch max and the abstract for the periodic memory):
//   gate/up: for every position p of rc = [C | R] and token b, z[b][p] = SiLU(Wg[c] x_b) * (W1[c] x_b)
//            with c = rc[p]; score[p] = max_b |z[b][p]| * ||W2[:, c]|| for the candidates p < |C|;
//   down:    the memory update and the top-k over C (every `period` steps), then
//            y[b][d] = sum over the kept items j (R, then the selected S) of z[b][j] * W2[d, channel of j].
//
// The MMA inputs are bf16. x and the weights are bf16 already; z is not, and rounding it to bf16
// would cost about 3 significant digits of y. So the down GEMM takes z as two bf16 parts, hi =
// bf16(z) and lo = bf16(z - hi), stacked as 2 x 16..64 token columns of one MMA; the epilogue adds
// the two halves, which leaves z's own fp32 rounding well below the output tolerance. The gate/up
// writes each position's z as one row of 2 NP bf16 (the hi parts of the tokens, then the lo parts),
// 16-byte stores of one contiguous row per thread; the down GEMM reads those rows as its MN-major
// B operand, for R (consecutive positions) and for the selected candidates alike.
//
// Both are skinny GEMMs with the tokens as the MMA's N (16..64, zero-padded to a multiple of 16)
// and 128 rows as M. The partition is fixed for a whole decode session, so each partition gets two
// slabs, built once per prefill (k_build_gu_slab, k_build_dn_slab): the gate/up rows of R u C and
// the down columns of R, copied from the packed weights into the exact shared-memory images the
// MMAs read (pre-tiled and pre-swizzled). A decode stage is then one contiguous bulk copy of 16-72
// KB, which streams at 6.7-7.2 TB/s, where gathering 128-512-byte row pieces with cp.async reached
// 4.7-6.2 TB/s. The selected candidates change every step, so their down columns are still
// gathered from the packed weights. Measured on this part: an MMA of M = 128, K = 16 costs ~44
// cycles for N <= 32 whatever its rows hold, so each MMA should carry as many real rows as it can.
// In the gathers a copy's landing arrives on its stage's barrier by itself
// (cp.async.mbarrier.arrive), so a producer only ever waits for a free slot; the MMA thread fences
// the landed copies for the tensor cores after its barrier wait.
//
// Gate/up by gathering (k_gateup_tc, used by the dense reference path at B > 1, where every
// channel is kept and no slab exists): one CTA per SM; each CTA streams "units" of at most 64
// positions over all of K. The unit ranges are ragged (P / units each) so that the number of units matches the number
// of CTAs. One MMA covers gate and up of a unit together: TMEM lane quarter q holds gate rows
// 16q..16q+15 in lanes 0-15 and the up rows of the same positions in lanes 16-31, so an epilogue
// warp pairs them with one shuffle. Rows past a unit's end are never written and the accumulator
// rows they produce are never read: row m of an MMA result depends on row m of A only. A stage
// holds 4 (or 2) consecutive k-blocks, so each gathered row is read in 512 (256) contiguous bytes.
// Weight rows and the partition are constant between partitions, so a CTA starts filling its ring
// before griddepcontrol.wait; only the x boxes and the stores of this step's data wait for the
// previous kernel.
//
// Down (k_down_tc): each unit (at most 128 outputs) is split along K over a cluster of `split`
// CTAs; every CTA streams its share of the R items first, then gathers its share of the selected
// items. In the decode one thread brings an R stage: a bulk copy of its slab tile and TMA boxes of
// its z rows (contiguous rows of the list); the eight producer warps gather the selected stages
// (and, in the dense reference path, every stage). A stage that all eight warps had to issue, each
// with its own barrier and copy instructions, took about 0.5 us of issue time whatever its size,
// which capped the R stream at about 40 KB per microsecond per CTA.
// The first cluster does the selection meanwhile: its CTA 0 updates the memory, takes the top-k,
// writes the selected positions and channels, and releases a flag. The other CTAs wait (bounded)
// for the flag when they reach their first selected item. Every item's z comes as the MMA's
// MN-major B operand: the producers gather the z rows like the down columns. The partial accumulators
// of a split unit are added through distributed shared memory in rank order (a fixed order:
// results do not depend on timing). No workspace, no atomics on data.
//
// Roles (416 threads): warps 0-7 gather, warp 8 lane 0 issues the MMAs and owns TMEM (two
// accumulator buffers, so the epilogue of one unit overlaps the MMAs of the next), warps 9-12 are
// the epilogue (TMEM lane quarter = warp % 4). Every wait is bounded; on a time-out the CTA records
// DEVERR_TIMEOUT_DECODE_TC, stops issuing, drains its own copies and MMAs (bounded), frees TMEM and
// returns. The warps of a role take every decision that guards a named barrier together, and every
// thread reaches the cluster barriers, so a time-out cannot leave a barrier waiting.
#include <algorithm>
#include <mutex>

#include "pop_device.cuh"
#include "pop_internal.h"
#include "pop_radix.cuh"

namespace pop {

namespace {
constexpr int TC_PW = 8;             // producer warps 0..7
constexpr int TC_MMA_WARP = TC_PW;   // warp 8
constexpr int TC_EPI0 = TC_PW + 1;   // warps 9..12
constexpr int TC_THREADS = 32 * (TC_PW + 5);
constexpr int TC_PROD_THREADS = 32 * TC_PW;
constexpr int TC_BM = 128;
constexpr int TC_BK = 64;
constexpr int TC_MAX_STAGES = 16;
constexpr uint64_t TC_DRAIN_NS = 1000000000ull;
constexpr uint32_t TC_TMEM_COLS = 256;  // two accumulator buffers of <= 128 fp32 columns
constexpr uint32_t TC_HALF = TC_TMEM_COLS / 2;
constexpr uint32_t TC_RING = 192 * 1024;
constexpr int GU_MAX_ROWS = 64;  // positions per unit (gate + up = 128 MMA rows)
// down: per producer warp, the channels of its 8 items of each of DN_WIN k-blocks
constexpr int DN_WIN = 32;
constexpr int DN_WIN_WORDS = 8 * DN_WIN * 8;
constexpr int GU_PRE = 2;         // stages of weights issued before waiting for the previous kernel

// Down stage: one k-block; A = 64 items x 128 outputs (two 64-wide halves, MN-major). B = z of the
// 64 items for 2 NP columns (the hi and lo parts of NP tokens), MN-major: one 128-byte row per item
// holding up to 64 columns, atoms of 64 columns 8 KB apart, gathered from the gate/up's z rows.
template <int NP>
struct DnCfg {
  static constexpr uint32_t A_BYTES = TC_BM * TC_BK * 2;
  static constexpr int ZATOMS = (2 * NP + 63) / 64;  // 64-column atoms of the z rows
  static constexpr uint32_t B_BYTES = TC_BK * 128 * ZATOMS;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = TC_RING / STAGE_BYTES < 12 ? TC_RING / STAGE_BYTES : 12;
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep the 1024-byte swizzle alignment");
  static_assert(static_cast<uint32_t>(TC_BM * NP * 4) <= STAGES * STAGE_BYTES, "partials reuse the ring");
};

struct TcCtl {
  uint64_t full[TC_MAX_STAGES];
  uint64_t empty[TC_MAX_STAGES];
  uint64_t afull[TC_MAX_STAGES];  // down: the stage's slab tile (bulk copy) has landed
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int seg_ok[2];  // by unit parity: a warp may still read one while the next is written
  unsigned sel_seen;  // down: the selection epoch warp 0 has seen complete
};

template <int NP>
constexpr size_t dn_smem_bytes() {
  return 1024 + DnCfg<NP>::STAGES * DnCfg<NP>::STAGE_BYTES;
}

// SiLU with the fast exponential and division: the epilogue of a decode tile runs exposed after its
// last MMA, and the accurate forms' dependent chains made it several microseconds longer at NP = 64
// (relative error ~1e-6, far inside the outputs' tolerance and the selection's flagged band).
__device__ __forceinline__ float silu_t(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

__device__ __forceinline__ int guard_ch(int v, int n, unsigned* err) {
  if (static_cast<unsigned>(v) >= static_cast<unsigned>(n)) {
    atomicOr(err, DEVERR_INDEX);
    return 0;
  }
  return v;
}

__device__ __forceinline__ void split_bf16(float v, uint16_t& hi, uint16_t& lo) {
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  const __nv_bfloat16 l = __float2bfloat16_rn(v - __bfloat162float(h));
  hi = *reinterpret_cast<const uint16_t*>(&h);
  lo = *reinterpret_cast<const uint16_t*>(&l);
}

// n (a multiple of 8) values as bf16 hi parts at hi[0..n) and lo parts at lo[0..n): 16-byte stores
template <int n>
__device__ __forceinline__ void store_hilo(uint16_t* hi, uint16_t* lo, const float* v) {
#pragma unroll
  for (int c = 0; c < n; c += 8) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint16_t h0, l0, h1, l1;
      split_bf16(v[c + 2 * i], h0, l0);
      split_bf16(v[c + 2 * i + 1], h1, l1);
      h[i] = h0 | (static_cast<uint32_t>(h1) << 16);
      l[i] = l0 | (static_cast<uint32_t>(l1) << 16);
    }
    *reinterpret_cast<uint4*>(hi + c) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4*>(lo + c) = make_uint4(l[0], l[1], l[2], l[3]);
  }
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros (nothing is read). No
// compiler memory barrier: the source is read-only for this kernel and the destination is touched
// by nothing else of this thread.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes));
}
// Waits until every cp.async this thread has issued has landed.
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Arrives on `bar` once every cp.async this thread has issued so far has landed (the arrival
// counts toward the barrier's initial count). The thread itself does not wait.
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Orders shared-memory writes of the generic proxy (landed cp.async copies, made visible to this
// thread by a barrier wait) before this thread's later tensor-core reads of them (async proxy).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void prod_bar() { asm volatile("bar.sync 2, %0;" ::"n"(TC_PROD_THREADS) : "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// All threads of all CTAs of the cluster; orders shared-memory writes before the barrier with
// (distributed) shared-memory reads after it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// The address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_peer4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// barrier over the eight producer warps (the selecting CTA uses the same warps)
struct ProdSync {
  __device__ void operator()() const { prod_bar(); }
};

// ------------------------------------------------------------------ selection (down, first cluster)
// Updates the periodic memory and selects the k best candidates when the step is an update step
// (select_step, warps 0-7), writes the selected positions (update steps) and their channels,
// advances the step counter and releases the flag. The GEMM CTAs then gather the selected items'
// z straight from the gate/up's candidate rows (an MN-major operand), so nothing is packed here.
__device__ void down_select(const DownTcArgs& a, uint8_t* smem, RadixScratch<TC_PROD_THREADS>& rsc) {
  if (a.skip) {
    // skip variant between updates: positions [0, k) of this step's list are the held selection
    // S_hold; their scores join the memory, the selection and its channels stay as they are
    for (int j = threadIdx.x; j < a.k; j += TC_THREADS) {
      int ps = __ldg(a.S_hold + j);
      if (static_cast<unsigned>(ps) >= static_cast<unsigned>(a.N)) {
        atomicOr(a.err, DEVERR_INDEX);
        ps = 0;
      }
      a.memory[ps] += __ldcg(a.scores + j);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      if (a.count_step) *a.step += 1;
      __threadfence();
      st_release_u32(a.flag, a.epoch);
    }
    return;
  }
  // While the GEMM CTAs stream, every global access of this CTA waits behind their requests
  // (microseconds), so all inputs are fetched in one round at the start, into shared memory:
  //   [keys: nC u32 | scores: nC f32 | channels of C: nC i32 | S: k i32 | memory: nC f32 (period > 1)]
  const int tid = threadIdx.x;
  const int nC = a.nC, k = a.k;
  uint32_t dyn = 0;
  asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
  const size_t avail = dyn > 1024 ? dyn - 1024 : 0;
  auto al16 = [](size_t v) { return (v + 15) & ~size_t(15); };
  const size_t o_keys = 0, o_sc = al16(static_cast<size_t>(nC) * 4), o_rc = o_sc + al16(static_cast<size_t>(nC) * 4);
  const size_t o_S = o_rc + al16(static_cast<size_t>(nC) * 4), o_m = o_S + al16(static_cast<size_t>(k) * 4);
  const bool periodic = a.period > 1;
  const bool small = o_m + (periodic ? al16(static_cast<size_t>(nC) * 4) : 0) <= avail;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + o_keys);
  float* s_sc = reinterpret_cast<float*>(smem + o_sc);
  int* s_rc = reinterpret_cast<int*>(smem + o_rc);
  int* sS = small ? reinterpret_cast<int*>(smem + o_S) : a.S;
  float* mem = small && periodic ? reinterpret_cast<float*>(smem + o_m) : a.memory;
  const int t = *a.step;
  const bool update = (t % a.period) == 0;
  if (small) {
    const uint32_t sb = smem_u32(smem);
    for (int i = tid; i < (nC + 3) / 4; i += TC_THREADS) {
      const uint32_t n = 4u * static_cast<uint32_t>(min(4, nC - 4 * i));
      cp_async16(sb + static_cast<uint32_t>(o_sc) + 16u * i, a.scores + 4 * i, n);
      cp_async16(sb + static_cast<uint32_t>(o_rc) + 16u * i, a.rc + 4 * i, n);
      if (periodic) cp_async16(sb + static_cast<uint32_t>(o_m) + 16u * i, a.memory + 4 * i, n);
    }
    if (!update)  // the held selection of the last update step
      for (int i = tid; i < (k + 3) / 4; i += TC_THREADS)
        cp_async16(sb + static_cast<uint32_t>(o_S) + 16u * i, a.S + 4 * i, 4u * min(4, k - 4 * i));
    cp_async_wait_all();
  }
  __syncthreads();
  __shared__ int s_sel;
  if (tid < TC_PROD_THREADS) {
    bool sel = true;
    if (nC > 0)
      sel = select_step<TC_PROD_THREADS>(
          tid, [&](int i) { return small ? s_sc[i] : __ldcg(a.scores + i); }, mem, nC, k, a.period, update, keys,
          sS, rsc, ProdSync());
    if (tid == 0) s_sel = sel ? 1 : 0;
  }
  __syncthreads();
  if (small && periodic)  // the memory as select_step left it (summed, or cleared on an update)
    for (int i = tid; i < nC; i += TC_THREADS) a.memory[i] = mem[i];
  if (update && small)
    for (int j = tid; j < k; j += TC_THREADS) a.S[j] = sS[j];
  // channels of the selected candidates
  for (int j = tid; j < k; j += TC_THREADS) {
    int ps = sS[j];
    if (static_cast<unsigned>(ps) >= static_cast<unsigned>(nC)) {
      atomicOr(a.err, DEVERR_INDEX);
      ps = 0;
      sS[j] = 0;
      if (update && small) a.S[j] = 0;
    }
    const int ch = guard_ch(small ? s_rc[ps] : __ldg(a.rc + ps), a.N, a.err);
    a.ch_s[j] = ch;
    if (a.rcs && update) a.rcs[j] = ch;  // skip variant: the list of the steps until the next update
  }
  __syncthreads();
  if (tid == 0) {
    if (!s_sel) atomicOr(a.err, DEVERR_TOPK);
    if (a.count_step) *a.step = t + 1;
    __threadfence();
    st_release_u32(a.flag, a.epoch);
  }
}
}  // namespace

// ------------------------------------------------------------------ gate/up over R u C
// NP: tokens padded to a multiple of 16 (16..64), a template parameter so that every per-token
// loop of the epilogue has a fixed trip count.
template <int NP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k_gateup_tc(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ GateUpTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ TcCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int W = static_cast<int>(gridDim.x), w = static_cast<int>(blockIdx.x);
  const int U = a.units;
  const int P = a.nC + a.nR;
  const int RC = a.rows_cap;  // multiple of 16, <= 64
  const int KS = a.ks;        // k-blocks per stage
  const uint32_t AROWS = 2 * RC;
  const uint32_t SUB = (AROWS + NP) * 128u;  // one k-block: A rows (gate and up interleaved) | x rows
  const uint32_t STAGE = KS * SUB;
  const int STAGES = a.stages;
  const int KB = (a.D + TC_BK - 1) / TC_BK;
  const int KBS = (KB + KS - 1) / KS;  // stages per unit
  const uint32_t tx_bytes = KS * NP * TC_BK * 2;
  auto unit_lo = [&](int u) { return static_cast<int>(static_cast<long long>(u) * P / U); };
  volatile int* abort_flag = &ctl.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl.full[s], TC_PROD_THREADS + 1);  // producer lanes + the x box's arrival with its bytes
      mbar_init(&ctl.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl.tfull[b], 1);
      mbar_init(&ctl.tempty[b], 4);
    }
    mbar_init(&ctl.drain, 1);
    ctl.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mapX);
  }
  if (warp == TC_MMA_WARP) {
    tmem_alloc(&ctl.tmem_base, TC_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  pdl_trigger();  // the down kernel only starts where this grid's CTAs have left an SM

  auto fail = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      atomicOr(a.err, DEVERR_TIMEOUT_DECODE_TC);
    }
  };

  if (warp < TC_PW) {
    // ------------------------------------------------------------ producers (eight warps)
    // A stage is KS consecutive k-blocks of the unit's rows. Lane group `grp` (8 lanes) copies the
    // rows (position j, gate/up g) numbered r = 2 j + g = grp, grp + 32, ... (at most 4 of them), each
    // lane 16-byte chunk cq of every k-block of the stage, so one warp instruction reads 128-byte
    // runs of four different rows (measured ~45% faster than one 512-byte run of one row per
    // instruction) and a lane walks KS x 128 contiguous bytes of its row. The rows a lane copies are
    // the same in every stage of a unit: their offsets and shared-memory places are computed once.
    // Warp 0 lane 0 adds the x boxes: for the first GU_PRE stages after griddepcontrol.wait (the
    // weights of those stages are already streaming by then), afterwards with each stage.
    const int cq = lane & 7, grp = (warp * 32 + lane) >> 3;
    const uint32_t row3 = 3u * static_cast<uint32_t>(a.D);  // 3 * D * D_FF < 2^32 under the size limits
    const bool tma_lane = warp == 0 && lane == 0;
    uint32_t issued = 0, x_done = 0;  // x boxes issued for stages [0, x_done)
    bool ok = true, waited = false;
    auto issue_x = [&](uint32_t i) {
      const int s = static_cast<int>(i % static_cast<uint32_t>(STAGES));
      const int sbk = static_cast<int>(i % static_cast<uint32_t>(KBS));
      mbar_arrive_expect_tx(&ctl.full[s], tx_bytes);
      for (int u = 0; u < KS; ++u)
        tma_load_2d(smem + s * STAGE + u * SUB + AROWS * 128, &mapX, &ctl.full[s], (sbk * KS + u) * TC_BK, 0);
    };
    for (int u = w; u < U && ok; u += W) {
      const int lo = unit_lo(u), nrows = unit_lo(u + 1) - lo;
      uint32_t rowbase[4], dst[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int rr = grp + 32 * t;  // row 2 j + g of the unit
        rowbase[t] = 0xffffffffu;
        dst[t] = 0u;
        if (rr < 2 * nrows) {
          const int g = rr & 1, j = rr >> 1;
          const int ch = guard_ch(__ldg(a.rc + lo + j), a.N, a.err);
          const int arow = 32 * (j >> 4) + 16 * g + (j & 15);
          rowbase[t] = static_cast<uint32_t>(ch) * row3 + static_cast<uint32_t>(g) * a.D + 8 * cq;
          dst[t] = arow * 128 + ((cq ^ (arow & 7)) << 4);
        }
      }
      for (int sbk = 0; sbk < KBS; ++sbk) {
        const int s = static_cast<int>(issued % static_cast<uint32_t>(STAGES));
        const uint32_t ph = (issued / static_cast<uint32_t>(STAGES)) & 1u;
        bool got = true;
        if (lane == 0) {
          got = mbar_wait_bounded(&ctl.empty[s], ph ^ 1u, a.wait_ns, abort_flag);
          if (!got) fail();
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(smem + s * STAGE);
        const uint32_t kbase = static_cast<uint32_t>(sbk * KS * TC_BK);
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          if (rowbase[t] != 0xffffffffu) {
#pragma unroll
            for (int u2 = 0; u2 < 4; ++u2) {
              if (u2 >= KS) break;
              const uint32_t k0 = kbase + u2 * TC_BK;  // the lane's chunk lies at k0 + 8 cq
              const uint32_t nbytes = k0 + 8 * cq < static_cast<uint32_t>(a.D) ? 16u : 0u;  // D: multiple of 8
              cp_async16(sa + u2 * SUB + dst[t], a.Wp + rowbase[t] + (nbytes ? k0 : 0u) - (nbytes ? 0u : 8u * cq),
                         nbytes);
            }
          }
        }
        cp_async_arrive(&ctl.full[s]);
        if (tma_lane) {
          if (waited) {
            issue_x(issued);
            x_done = issued + 1;
          } else if (issued + 1 >= static_cast<uint32_t>(STAGES < GU_PRE ? STAGES : GU_PRE)) {
            pdl_wait();  // x of this step is complete once the previous kernel is
            waited = true;
            for (uint32_t i = x_done; i <= issued; ++i) issue_x(i);
            x_done = issued + 1;
          }
        }
        ++issued;
      }
    }
    // x boxes still owed (a CTA with fewer stages than the ring); every copy this warp started
    // must land before the CTA can exit
    if (tma_lane && ok) {
      if (!waited) {
        pdl_wait();
        waited = true;
      }
      for (uint32_t i = x_done; i < issued; ++i) issue_x(i);
      x_done = issued;
    }
    cp_async_wait_all();
    if (tma_lane) {
      const uint32_t lo = x_done > static_cast<uint32_t>(STAGES) ? x_done - STAGES : 0;
      for (uint32_t i = lo; i < x_done; ++i) {
        volatile int never = 0;
        if (!mbar_wait_bounded(&ctl.full[i % STAGES], (i / STAGES) & 1u, TC_DRAIN_NS, &never)) fail();
      }
    }
    __syncwarp();
  } else if (warp == TC_MMA_WARP) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer (one thread)
      const uint32_t idesc = idesc_bf16_f32(TC_BM, NP, false, false);
      uint32_t consumed = 0;
      int it = 0;
      bool ok = true;
      for (int u = w; u < U && ok; u += W, ++it) {
        const int buf = it & 1;
        if (!mbar_wait_bounded(&ctl.tempty[buf], ((it >> 1) & 1) ^ 1, a.wait_ns, abort_flag)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * TC_HALF;
        for (int sbk = 0; sbk < KBS; ++sbk) {
          const int s = static_cast<int>(consumed % static_cast<uint32_t>(STAGES));
          const uint32_t ph = (consumed / static_cast<uint32_t>(STAGES)) & 1u;
          if (!mbar_wait_bounded(&ctl.full[s], ph, a.wait_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          fence_proxy_async();
          tc_fence_after();
          for (int u2 = 0; u2 < KS; ++u2) {
            const uint32_t sg = smem_u32(smem + s * STAGE) + u2 * SUB;
            const uint32_t sx = sg + AROWS * 128;
#pragma unroll
            for (int k = 0; k < TC_BK / 16; ++k) {
              const uint32_t acc = (sbk > 0 || u2 > 0 || k > 0) ? 1u : 0u;
              umma_f16(d_tmem, smem_desc_sw128(sg + 32u * k, 16u, 1024u), smem_desc_sw128(sx + 32u * k, 16u, 1024u),
                       idesc, acc);
            }
          }
          umma_commit(&ctl.empty[s]);
          ++consumed;
        }
        if (!ok) break;
        umma_commit(&ctl.tfull[buf]);
      }
      // all MMAs issued by this thread must finish before TMEM is freed
      umma_commit(&ctl.drain);
      volatile int never = 0;
      if (!mbar_wait_bounded(&ctl.drain, 0, TC_DRAIN_NS, &never)) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 9..12)
    pdl_wait();  // z rows and scores may still be read by the previous step's kernels
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int half = lane >> 4;
    const int j = 16 * q + (lane & 15);  // position within the unit; lanes 0-15 gate, 16-31 up
    const int et = threadIdx.x - 32 * TC_EPI0;  // 0..127
    constexpr int NH = NP / 2;                  // tokens per lane after the pairing
    const int b0 = half * NH;
    int it = 0;
    for (int u = w; u < U; u += W, ++it) {
      const int buf = it & 1;
      const int lo = unit_lo(u), hi = unit_lo(u + 1);
      const int p = lo + j;
      const bool valid = p < hi;
      const bool cand = valid && p < a.nC;
      // the candidates' down-column norms, fetched while the accumulators are still being built
      float n2v = 0.f;
      if (cand && half == 0) n2v = __ldg(a.n2 + guard_ch(__ldcg(a.rc + p), a.N, a.err));
      if (et == 0)
        ctl.seg_ok[buf] = mbar_wait_bounded(&ctl.tfull[buf], (it >> 1) & 1, a.wait_ns, abort_flag) ? 1 : 0;
      epi_bar();
      if (!ctl.seg_ok[buf]) {
        if (et == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf) * TC_HALF;
      float acc[NP];
#pragma unroll
      for (int c = 0; c < NP; c += 16) {
        uint32_t t16[16];
        tmem_ld16(taddr + c, t16);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[c + i] = __uint_as_float(t16[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.tempty[buf]);
      // pair gate (lanes 0-15) with up (lanes 16-31) of the same position: lane l < 16 takes
      // tokens [0, NP/2), lane l + 16 tokens [NP/2, NP)
      float zz[NH];
#pragma unroll
      for (int i = 0; i < NH; ++i) {
        const float mine = half ? acc[i] : acc[NH + i];
        const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
        const float g = half ? other : acc[i];
        const float uu = half ? acc[NH + i] : other;
        zz[i] = silu_t(g) * uu;
      }
      float m = 0.f;
#pragma unroll
      for (int i = 0; i < NH; ++i)
        if (b0 + i < a.B) m = fmaxf(m, fabsf(zz[i]));
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
      if (valid) {
        // the position's z row for the down GEMM: hi parts of the NP tokens, then lo parts
        uint16_t* row = a.zcp + static_cast<size_t>(p) * (2 * NP);
        store_hilo<NH>(row + b0, row + NP + b0, zz);
        if (cand && half == 0) a.scores[p] = m * n2v;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == TC_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TC_TMEM_COLS);
  }
}

// ------------------------------------------------------------------ decode slabs (built per partition)
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// One 16-byte chunk per thread (grid-stride): chunk e of the gate/up slab is position pos = e % 8 of
// A row ar of k-block kb of tile t; it holds data chunk c = pos ^ (ar % 8) (the 128-byte swizzle).
// IDX is the index type: 32-bit when the chunk count allows it (64-bit division is slow here).
template <class IDX>
__global__ void k_build_gu_slab(const uint16_t* __restrict__ Wp, const int* __restrict__ rc, int D, int N,
                                GuSlabGeom g, int t_lo, int t_hi, uint16_t* __restrict__ slab,
                                unsigned* __restrict__ err) {
  // chunks of tiles [t_lo, t_hi); chunk e of this range is chunk e0 + e of the slab
  const IDX e0 = static_cast<IDX>(t_lo) * g.KB * g.arows * 8;
  const IDX total = static_cast<IDX>(t_hi - t_lo) * g.KB * g.arows * 8;
  const int grows = (g.RT + 7) / 8 * 8;
  const IDX arows = static_cast<IDX>(g.arows), KB = static_cast<IDX>(g.KB);
  for (IDX e = static_cast<IDX>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<IDX>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(e & 7);
    IDX rest = e >> 3;
    const int ar = static_cast<int>(rest % arows);
    rest /= arows;
    const int kb = static_cast<int>(rest % KB);
    const int t = t_lo + static_cast<int>(rest / KB);
    const int c = pos ^ (ar & 7);
    int j, gu;
    if (g.paired) {
      const int rem = ar & 31;
      gu = rem >> 4;
      j = 16 * (ar >> 5) + (rem & 15);
    } else {
      gu = ar >= grows ? 1 : 0;
      j = gu ? ar - grows : ar;
    }
    const int p = gu_slab_pos(g, t, j);
    const int d = kb * TC_BK + 8 * c;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (p >= 0 && d < D) {
      int ch = __ldcg(rc + p);
      if (static_cast<unsigned>(ch) >= static_cast<unsigned>(N)) {
        atomicOr(err, DEVERR_INDEX);
        ch = 0;
      }
      v = ldg_stream(Wp + static_cast<size_t>(ch) * 3 * D + static_cast<size_t>(gu) * D + d);
    }
    *reinterpret_cast<uint4*>(slab + static_cast<size_t>(e0 + e) * 8) = v;
  }
}

// Chunk e of the down slab: position pos = e % 8 of item i of output half h of item block b of
// output slice o; it holds the 8 outputs 128 o + 64 h + 8 c, c = pos ^ (i % 8), of R item 64 b + i.
__global__ void k_build_dn_slab(const uint16_t* __restrict__ Wp, const int* __restrict__ rc, int nC, int nR, int D,
                                int N, int kbr, uint16_t* __restrict__ slab, unsigned* __restrict__ err) {
  const int O = (D + TC_BM - 1) / TC_BM;
  const size_t total = static_cast<size_t>(O) * kbr * 2 * TC_BK * 8;
  for (size_t e = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
       e += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const int pos = static_cast<int>(e & 7);
    size_t rest = e >> 3;
    const int i = static_cast<int>(rest & 63);
    rest >>= 6;
    const int h = static_cast<int>(rest & 1);
    rest >>= 1;
    const int b = static_cast<int>(rest % kbr);
    const int o = static_cast<int>(rest / kbr);
    const int c = pos ^ (i & 7);
    const int item = b * TC_BK + i;
    const int d = o * TC_BM + 64 * h + 8 * c;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (item < nR && d < D) {
      int ch = rc[nC + item];
      if (static_cast<unsigned>(ch) >= static_cast<unsigned>(N)) {
        atomicOr(err, DEVERR_INDEX);
        ch = 0;
      }
      v = *reinterpret_cast<const uint4*>(Wp + static_cast<size_t>(ch) * 3 * D + 2 * static_cast<size_t>(D) + d);
    }
    *reinterpret_cast<uint4*>(slab + e * 8) = v;
  }
}

// ------------------------------------------------------------------ gate/up over R u C from the slab
// One CTA per SM; CTA w streams tiles w, w + grid, ... Warp 0 lane 0 issues, per stage of KS
// k-blocks, one bulk copy of the tile's KS contiguous A images and KS TMA boxes of x; warp 1 lane 0
// issues the MMAs (one per K = 16 when gate and up share the tile's rows, two otherwise) and owns
// TMEM; warps 2-5 are the epilogue (TMEM lane quarter = warp % 4). The slab is constant between
// partitions, so the first GU_PRE stages' copies go out before griddepcontrol.wait; their x boxes
// after it.
constexpr int GS_THREADS = 192;
template <int NP, bool PAIRED>
__global__ void __launch_bounds__(GS_THREADS, 1)
    k_gateup_slab(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ GateUpSlabArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ TcCtl ctl;
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const GuSlabGeom g = a.geom;
  const int W = static_cast<int>(gridDim.x), w = static_cast<int>(blockIdx.x);
  const int KS = a.ks, STAGES = a.stages;
  const uint32_t ABYTES = static_cast<uint32_t>(g.arows) * 128u;
  const uint32_t XBYTES = NP * 128u;
  const uint32_t STAGE = KS * (ABYTES + XBYTES);
  const int KBS = (g.KB + KS - 1) / KS;  // stages per tile
  const uint32_t UP_OFF = static_cast<uint32_t>((g.RT + 7) / 8 * 8) * 128u;  // up rows (unpaired tiles)
  // Each CTA walks the k-blocks from its own starting stage: all CTAs read the same x tiles, and
  // moving in step they would all ask L2 for the same lines at once.
  const uint32_t rot = static_cast<uint32_t>(w) * 5u;
  volatile int* abort_flag = &ctl.abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl.tfull[b], 1);
      mbar_init(&ctl.tempty[b], 4);
    }
    mbar_init(&ctl.drain, 1);
    ctl.abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&mapX);
  }
  if (warp == 1) {
    tmem_alloc(&ctl.tmem_base, TC_TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  pdl_trigger();

  auto fail = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      atomicOr(a.err, DEVERR_TIMEOUT_DECODE_TC);
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer (one thread)
      uint32_t issued = 0, x_done = 0;
      bool ok = true, waited = false;
      auto stage_kb = [&](uint32_t i, int& kb0, int& nk) {
        kb0 = static_cast<int>((i + rot) % static_cast<uint32_t>(KBS)) * KS;
        nk = min(KS, g.KB - kb0);
      };
      auto issue_x = [&](uint32_t i) {
        int kb0, nk;
        stage_kb(i, kb0, nk);
        uint8_t* sx = smem + (i % static_cast<uint32_t>(STAGES)) * STAGE + KS * ABYTES;
        for (int u = 0; u < nk; ++u)
          tma_load_2d(sx + u * XBYTES, &mapX, &ctl.full[i % STAGES], (kb0 + u) * TC_BK, 0);
      };
      for (int t = w; t < g.T && ok; t += W) {
        for (int sbk = 0; sbk < KBS; ++sbk) {
          const int s = static_cast<int>(issued % static_cast<uint32_t>(STAGES));
          const uint32_t ph = (issued / static_cast<uint32_t>(STAGES)) & 1u;
          if (!mbar_wait_bounded(&ctl.empty[s], ph ^ 1u, a.wait_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          int kb0, nk;
          stage_kb(issued, kb0, nk);
          mbar_arrive_expect_tx(&ctl.full[s], static_cast<uint32_t>(nk) * (ABYTES + XBYTES));
          bulk_g2s(smem + s * STAGE, a.slab + (static_cast<size_t>(t) * g.KB + kb0) * g.arows * 64,
                   static_cast<uint32_t>(nk) * ABYTES, &ctl.full[s]);
          if (waited) {
            issue_x(issued);
            x_done = issued + 1;
          } else if (issued + 1 >= static_cast<uint32_t>(STAGES < GU_PRE ? STAGES : GU_PRE)) {
            pdl_wait();  // x of this step is complete once the previous kernel is
            waited = true;
            for (uint32_t i = x_done; i <= issued; ++i) issue_x(i);
            x_done = issued + 1;
          }
          ++issued;
        }
      }
      // x boxes still owed (fewer stages than GU_PRE, or an abort before the wait): issued in any case,
      // so that every issued stage's barrier completes once its bytes have landed
      if (!waited) {
        pdl_wait();
        waited = true;
        for (uint32_t i = x_done; i < issued; ++i) issue_x(i);
        x_done = issued;
      }
      // no copy of this CTA may be in flight when it exits
      const uint32_t lo = x_done > static_cast<uint32_t>(STAGES) ? x_done - STAGES : 0;
      for (uint32_t i = lo; i < x_done; ++i) {
        volatile int never = 0;
        if (!mbar_wait_bounded(&ctl.full[i % STAGES], (i / STAGES) & 1u, TC_DRAIN_NS, &never)) fail();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer (one thread)
      const uint32_t idesc = idesc_bf16_f32(TC_BM, NP, false, false);
      uint32_t consumed = 0;
      int it = 0;
      bool ok = true;
      for (int t = w; t < g.T && ok; t += W, ++it) {
        const int buf = it & 1;
        if (!mbar_wait_bounded(&ctl.tempty[buf], ((it >> 1) & 1) ^ 1, a.wait_ns, abort_flag)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * TC_HALF;
        for (int sbk = 0; sbk < KBS; ++sbk) {
          const int s = static_cast<int>(consumed % static_cast<uint32_t>(STAGES));
          const uint32_t ph = (consumed / static_cast<uint32_t>(STAGES)) & 1u;
          if (!mbar_wait_bounded(&ctl.full[s], ph, a.wait_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const int nk = min(KS, g.KB - static_cast<int>((static_cast<uint32_t>(sbk) + rot) % KBS) * KS);
          const uint32_t sa = smem_u32(smem + s * STAGE);
          // descriptors once per stage; a K step of 16 moves the start address by 32 bytes (+2)
          uint64_t ad = smem_desc_sw128(sa, 16u, 1024u);
          uint64_t bd = smem_desc_sw128(sa + KS * ABYTES, 16u, 1024u);
          const uint64_t up = UP_OFF >> 4;
          for (int u = 0; u < nk; ++u) {
            const uint32_t first = (sbk == 0 && u == 0) ? 0u : 1u;
            if (PAIRED) {
              umma_f16(d_tmem, ad, bd, idesc, first);
              umma_f16(d_tmem, ad + 2, bd + 2, idesc, 1u);
              umma_f16(d_tmem, ad + 4, bd + 4, idesc, 1u);
              umma_f16(d_tmem, ad + 6, bd + 6, idesc, 1u);
            } else {
              const uint32_t du = d_tmem + static_cast<uint32_t>(NP);
              umma_f16(d_tmem, ad, bd, idesc, first);
              umma_f16(du, ad + up, bd, idesc, first);
              umma_f16(d_tmem, ad + 2, bd + 2, idesc, 1u);
              umma_f16(du, ad + up + 2, bd + 2, idesc, 1u);
              umma_f16(d_tmem, ad + 4, bd + 4, idesc, 1u);
              umma_f16(du, ad + up + 4, bd + 4, idesc, 1u);
              umma_f16(d_tmem, ad + 6, bd + 6, idesc, 1u);
              umma_f16(du, ad + up + 6, bd + 6, idesc, 1u);
            }
            ad += ABYTES >> 4;
            bd += XBYTES >> 4;
          }
          umma_commit(&ctl.empty[s]);
          ++consumed;
        }
        if (!ok) break;
        umma_commit(&ctl.tfull[buf]);
      }
      umma_commit(&ctl.drain);
      volatile int never = 0;
      if (!mbar_wait_bounded(&ctl.drain, 0, TC_DRAIN_NS, &never)) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    pdl_wait();  // z rows and scores may still be read by the previous step's kernels
    const int q = warp & 3;
    const int et = threadIdx.x - 64;  // 0..127
    constexpr int NH = NP / 2;
    int it = 0;
    for (int t = w; t < g.T; t += W, ++it) {
      const int buf = it & 1;
      // paired: lane l < 16 holds gate, l + 16 up, of position 16 q + l % 16 (tokens split in two
      // halves between them); unpaired: lane l holds gate (columns [0, NP)) and up ([NP, 2 NP)) of
      // position 32 q + l
      const int j = PAIRED ? 16 * q + (lane & 15) : 32 * q + lane;
      const int p = gu_slab_pos(g, t, j);
      const bool valid = p >= 0;
      const bool cand = valid && p < a.nC;
      const int half = PAIRED ? (lane >> 4) : 0;
      float n2v = 0.f;
      if (cand && half == 0) n2v = __ldg(a.n2 + guard_ch(__ldcg(a.rc + p), a.N, a.err));
      if (et == 0)
        ctl.seg_ok[buf] = mbar_wait_bounded(&ctl.tfull[buf], (it >> 1) & 1, a.wait_ns, abort_flag) ? 1 : 0;
      epi_bar();
      if (!ctl.seg_ok[buf]) {
        if (et == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf) * TC_HALF;
      if (PAIRED) {
        float acc[NP];
#pragma unroll
        for (int c = 0; c < NP; c += 16) {
          uint32_t t16[16];
          tmem_ld16(taddr + c, t16);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) acc[c + i] = __uint_as_float(t16[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.tempty[buf]);
        const int b0 = half * NH;
        float zz[NH];
#pragma unroll
        for (int i = 0; i < NH; ++i) {
          const float mine = half ? acc[i] : acc[NH + i];
          const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
          const float gg = half ? other : acc[i];
          const float uu = half ? acc[NH + i] : other;
          zz[i] = silu_t(gg) * uu;
        }
        float m = 0.f;
#pragma unroll
        for (int i = 0; i < NH; ++i)
          if (b0 + i < a.B) m = fmaxf(m, fabsf(zz[i]));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if (valid) {
          // the position's z row for the down GEMM (its MN-major operand): hi parts of tokens
          // [0, NP), then lo parts
          uint16_t* row = a.zcp + static_cast<size_t>(p) * (2 * NP);
          store_hilo<NH>(row + b0, row + NP + b0, zz);
          if (cand && half == 0) a.scores[p] = m * n2v;
        }
      } else {
        float gv[NP], uv[NP];
#pragma unroll
        for (int c = 0; c < NP; c += 16) {
          uint32_t t16[16];
          tmem_ld16(taddr + c, t16);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) gv[c + i] = __uint_as_float(t16[i]);
          tmem_ld16(taddr + NP + c, t16);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) uv[c + i] = __uint_as_float(t16[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl.tempty[buf]);
        if (valid) {
          float zz[NP];
          float m = 0.f;
#pragma unroll
          for (int b = 0; b < NP; ++b) {
            zz[b] = silu_t(gv[b]) * uv[b];
            if (b < a.B) m = fmaxf(m, fabsf(zz[b]));
          }
          uint16_t* row = a.zcp + static_cast<size_t>(p) * (2 * NP);
          store_hilo<NP>(row, row + NP, zz);
          if (cand) a.scores[p] = m * n2v;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TC_TMEM_COLS);
  }
}

// The epilogue threads' part of a split unit's reduction. The partials sit token-major in each
// CTA's shared memory (pb[t * 128 + row]), so four consecutive rows of one token are one 16-byte
// word. CTA `rank` finishes rows [rank * 128 / SK, (rank + 1) * 128 / SK) of the unit; an item is
// (token t, group of 4 rows): its SK partial words are read from every CTA of the cluster (all loads
// before the first add), added in rank order and stored to y as 4 consecutive outputs. Consecutive
// threads take consecutive row groups of one token, so a warp stores whole runs of y.
template <int NP, int SK>
__device__ __forceinline__ void cluster_finish(const DownTcArgs& a, uint32_t pb, uint32_t rank, int et, int d_lo,
                                               int d_hi) {
  constexpr int ROWS = TC_BM / SK, RG = ROWS / 4, ITEMS = RG * NP;
  static_assert(ROWS % 4 == 0, "row groups of 4");
#pragma unroll 1
  for (int it = et; it < ITEMS; it += 128) {
    const int t = it / RG, rg = it % RG;
    const int row = static_cast<int>(rank) * ROWS + 4 * rg;
    const uint32_t off = pb + static_cast<uint32_t>(t * TC_BM + row) * 4u;
    float4 v[SK];
#pragma unroll
    for (int pr = 0; pr < SK; ++pr) v[pr] = ld_peer4(map_peer(off, static_cast<uint32_t>(pr)));
    float4 g = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int pr = 0; pr < SK; ++pr) {
      g.x += v[pr].x;
      g.y += v[pr].y;
      g.z += v[pr].z;
      g.w += v[pr].w;
    }
    const int d = d_lo + row;  // units hold whole groups of 8 outputs: d < d_hi implies d + 3 < d_hi
    if (t < a.B && d < d_hi) {
      const size_t o = static_cast<size_t>(t) * a.D + d;
      if (a.out_f32) {
        *reinterpret_cast<float4*>(static_cast<float*>(a.y) + o) = g;
      } else {
        *reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.y) + o) = make_uint2(pack_bf16x2(g.x, g.y), pack_bf16x2(g.z, g.w));
      }
    }
  }
}

// ------------------------------------------------------------------ selection + down over R u S
template <int NP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k_down_tc(const __grid_constant__ CUtensorMap mapZ, const __grid_constant__ DownTcArgs a) {
  using Cfg = DnCfg<NP>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr uint32_t STAGE_BYTES = Cfg::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ TcCtl ctl;
  __shared__ RadixScratch<TC_PROD_THREADS> rsc;
  __shared__ int dwin[DN_WIN_WORDS];   // per producer warp: channels of its items of DN_WIN stages
  __shared__ int dwinp[DN_WIN_WORDS];  // the same items' positions in C (selected stages)
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int SK = a.split;
  const uint32_t rank = SK > 1 ? cluster_rank() : 0u;
  const int ci = static_cast<int>(blockIdx.x) / SK;  // cluster index

  if (a.sel && ci == 0) {
    // ------------------------------------------------------------ the selecting cluster
    if (rank == 0) {
      pdl_wait();  // this step's scores and z rows; S, memory and step of the previous step
      pdl_trigger();
      down_select(a, smem, rsc);
    }
    return;
  }

  volatile int* abort_flag = &ctl.abort_flag;
  volatile unsigned* sel_seen = &ctl.sel_seen;
  const int unit0 = ci - a.sel, nunits = static_cast<int>(gridDim.x) / SK - a.sel;
  const int U = a.units;
  const int G = a.D / 8;  // output groups of 8 (16 bytes); a unit is a range of whole groups
  const bool slab = a.dslab != nullptr;  // R tiles from the slab; units are its 128-output slices
  auto unit_lo = [&](int u) {
    return slab ? min(a.D, TC_BM * u) : 8 * static_cast<int>(static_cast<long long>(u) * G / U);
  };
  // this CTA's k-blocks: R blocks [r0, r1), then selected blocks [s0, s1) (block kbr + t holds
  // selected items 64 t ..)
  const int kbs = (a.k + TC_BK - 1) / TC_BK;
  const int r0 = static_cast<int>(rank) * a.kbr / SK, r1 = (static_cast<int>(rank) + 1) * a.kbr / SK;
  const int s0 = static_cast<int>(rank) * kbs / SK, s1 = (static_cast<int>(rank) + 1) * kbs / SK;
  const int nblk = (r1 - r0) + (s1 - s0);  // stages per unit

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl.full[s], TC_PROD_THREADS);
      mbar_init(&ctl.empty[s], 1);
      mbar_init(&ctl.afull[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl.tfull[b], 1);
      mbar_init(&ctl.tempty[b], 4);
    }
    mbar_init(&ctl.drain, 1);
    ctl.abort_flag = 0;
    ctl.sel_seen = a.epoch - 1u;
    fence_mbar_init();
  }
  if (warp == TC_MMA_WARP) {
    tmem_alloc(&ctl.tmem_base, TC_TMEM_COLS);
    tmem_relinquish();
  }
  if (threadIdx.x == 0 && slab) prefetch_tmap(&mapZ);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  pdl_trigger();
  // Only the producers touch this step's data before the epilogue (which follows their copies
  // through the barriers); they wait for the previous kernel before the z rows (see below).

  auto fail = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      atomicOr(a.err, DEVERR_TIMEOUT_DECODE_TC);
    }
  };

  if (warp < TC_PW) {
    // ------------------------------------------------------------ producers (eight warps)
    // Per stage: the A pieces (item i, output half h) p = 2 i + h are copied by lane group
    // grp = p % 32 (16 contiguous bytes per lane, 8 lanes per 128-byte piece), so a warp reads two
    // items' 256 contiguous bytes; the z-plane chunks (NP / 16 per lane) follow. Items past the end
    // of R or of S are zero-filled, as are token rows past B. Each warp keeps the channels of its
    // items for DN_WIN stages in shared memory, fetched together (one round of loads per window).
    const int cq = lane & 7, grp = (warp * 32 + lane) >> 3;
    const uint16_t* W2 = a.Wp + 2 * static_cast<size_t>(a.D);
    const size_t row3 = 3 * static_cast<size_t>(a.D);
    const int h = grp & 1, ip = (grp & 3) >> 1;  // output half; item parity within the warp's pair
    const int nrs = r1 - r0;                     // R stages of each unit
    int* mywin = dwin + warp * (DN_WIN * 8);
    int* mywinp = dwinp + warp * (DN_WIN * 8);
    int wlo = 0, whi = 0;                        // stages [wlo, whi) are in the window
    auto fill = [&](int bi0) {
      const int seg_end = bi0 < nrs ? nrs : nblk;
      wlo = bi0;
      whi = min(seg_end, bi0 + DN_WIN);
      int c[8], ps[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        const int x = lane + 32 * v;
        const int bj = wlo + (x >> 3), e = x & 7;
        const int i = 2 * warp + (e & 1) + 16 * (e >> 1);  // item within its k-block
        c[v] = -1;
        ps[v] = -1;
        if (bj < whi) {
          if (bj < nrs) {
            const int item = (r0 + bj) * TC_BK + i;
            if (item < a.nR) c[v] = __ldg(a.ch_r + item);
          } else {
            const int item = (s0 + bj - nrs) * TC_BK + i;
            if (item < a.k) {
              c[v] = __ldcg(a.ch_s + item);
              ps[v] = __ldcg(a.S + item);
            }
          }
        }
      }
      __syncwarp();
#pragma unroll
      for (int v = 0; v < 8; ++v) {
        mywin[lane + 32 * v] = c[v];
        mywinp[lane + 32 * v] = ps[v];
      }
      __syncwarp();
    };
    auto issue_a = [&](int bi, uint32_t sa, int d0, bool dok) {
      if (!dok) return;  // outputs past the unit's end are left unwritten (their rows are never read)
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int i = (grp >> 1) + 16 * t;
        int ch = mywin[(bi - wlo) * 8 + ip + 2 * t];
        const uint32_t nb = ch >= 0 ? 16u : 0u;
        if (ch >= 0) ch = guard_ch(ch, a.N, a.err);
        cp_async16(sa + h * (TC_BK * 128) + i * 128 + ((cq ^ (i & 7)) << 4),
                   W2 + (nb ? static_cast<size_t>(ch) * row3 + d0 : 0), nb);
      }
    };
    auto issue_bs = [&](int bi, uint32_t sa) {
      // selected stage: item e of this warp's eight takes its candidate row (2 NP bf16, the hi then
      // lo parts) as CPI 16-byte chunks; chunk c goes to column atom c / 8 (8 KB apart), 16-byte
      // column group c % 8 of the item's 128-byte row, swizzled by the item's row within its 8
      constexpr int CPI = NP / 4;
#pragma unroll
      for (int v = 0; v < CPI / 4; ++v) {
        const int qd = lane + 32 * v;
        const int e = qd / CPI, c = qd % CPI;
        const int i = 2 * warp + (e & 1) + 16 * (e >> 1);
        int p = mywinp[(bi - wlo) * 8 + e];
        const uint32_t nb = p >= 0 ? 16u : 0u;
        if (p >= 0 && static_cast<unsigned>(p) >= static_cast<unsigned>(a.nC)) {
          atomicOr(a.err, DEVERR_INDEX);
          p = 0;
        }
        cp_async16(sa + Cfg::A_BYTES + (c >> 3) * (TC_BK * 128) + i * 128 + (((c & 7) ^ (i & 7)) << 4),
                   nb ? a.zcp + static_cast<size_t>(p) * (2 * NP) + 8 * c : a.zcp, nb);
      }
    };
    auto issue_b = [&](int bi, uint32_t sa) {
      if (bi >= nrs) {
        issue_bs(bi, sa);
        return;
      }
      // R stage: the z rows of R items 64 kb .. 64 kb + 63 (list positions r_pos0 + item, contiguous),
      // in the same MN-major layout as the selected items'; items past the end of R read as zero
      constexpr int CPI = NP / 4;
      const int kb = r0 + bi;
#pragma unroll
      for (int v = 0; v < CPI / 4; ++v) {
        const int qd = lane + 32 * v;
        const int e = qd / CPI, c = qd % CPI;
        const int i = 2 * warp + (e & 1) + 16 * (e >> 1);
        const int item = kb * TC_BK + i;
        const uint32_t nb = item < a.nR ? 16u : 0u;
        cp_async16(sa + Cfg::A_BYTES + (c >> 3) * (TC_BK * 128) + i * 128 + (((c & 7) ^ (i & 7)) << 4),
                   nb ? a.zcp + static_cast<size_t>(a.r_pos0 + item) * (2 * NP) + 8 * c : a.zcp, nb);
      }
    };
    // Nothing goes out before the wait for the previous kernel: slab copies issued early held the
    // CTAs' wait back by about 2 us, longer than they saved (LLaMA-2-7B FFN shape, B = 16: step
    // 40.2 us with two stages issued early, 38.6 us with none).
    pdl_wait();
    uint32_t issued = 0;
    bool ok = true;
    for (int unit = unit0; unit < U && ok; unit += nunits) {
      const int lo = unit_lo(unit), hi = unit_lo(unit + 1);
      const int d0 = lo + 64 * h + 8 * cq;
      const bool dok = d0 < hi;
      for (int bi = 0; bi < nblk; ++bi) {
        if (bi == nrs && bi < nblk) {
          // first selected block: the selection of this step must be complete. Warp 0 polls the
          // flag in global memory and posts what it saw in shared memory; the other warps watch
          // that (every wait bounded; no barrier across warps that a warp which gave up earlier
          // would miss).
          int good = 1;
          if (lane == 0) {
            const uint64_t t0 = globaltimer_ns();
            if (warp == 0) {
              while (static_cast<int>(ld_acquire_u32(a.flag) - a.epoch) < 0) {
                if (*abort_flag || globaltimer_ns() - t0 > a.wait_ns) {
                  good = 0;
                  break;
                }
                __nanosleep(256);
              }
              if (good) {
                __threadfence_block();
                *sel_seen = a.epoch;
              }
            } else {
              while (static_cast<int>(*sel_seen - a.epoch) < 0) {
                if (*abort_flag || globaltimer_ns() - t0 > a.wait_ns) {
                  good = 0;
                  break;
                }
                __nanosleep(64);
              }
              if (good) (void)ld_acquire_u32(a.flag);  // acquire for this warp's own reads
            }
            if (!good) fail();
          }
          good = __shfl_sync(0xffffffffu, good, 0);
          __syncwarp();  // orders lane 0's acquire before the other lanes' reads of the selection
          if (!good) {
            ok = false;
            break;
          }
        }
        const bool from_slab = slab && bi < nrs;
        // R blocks from the slab go in an order rotated per unit (the units of a rank read the same z
        // columns; in step they would ask L2 for the same lines at once)
        const int rb = from_slab ? (bi + 7 * unit) % nrs : bi;
        const int s = issued % STAGES;
        const uint32_t ph = (issued / STAGES) & 1u;
        if (from_slab) {
          // R stage: warp 0 lane 0 alone; its barrier counts the slab tile and the z boxes (rows of
          // items past the end of R lie outside the map and read as zero)
          if (warp == 0) {
            int good = 1;
            if (lane == 0) {
              if (!mbar_wait_bounded(&ctl.empty[s], ph ^ 1u, a.wait_ns, abort_flag)) {
                fail();
                good = 0;
              } else {
                uint8_t* st = smem + s * STAGE_BYTES;
                mbar_arrive_expect_tx(&ctl.afull[s], Cfg::A_BYTES + Cfg::B_BYTES);
                bulk_g2s(st, a.dslab + (static_cast<size_t>(unit) * a.kbr + r0 + rb) * (Cfg::A_BYTES / 2),
                         Cfg::A_BYTES, &ctl.afull[s]);
                for (int at = 0; at < Cfg::ZATOMS; ++at)
                  tma_load_2d(st + Cfg::A_BYTES + at * (TC_BK * 128), &mapZ, &ctl.afull[s], 64 * at,
                              a.r_pos0 + (r0 + rb) * TC_BK);
              }
            }
            if (!__shfl_sync(0xffffffffu, good, 0)) {
              ok = false;
              break;
            }
          }
          ++issued;
          continue;
        }
        if (bi < wlo || bi >= whi) fill(bi);
        bool got = true;
        if (lane == 0) {
          got = mbar_wait_bounded(&ctl.empty[s], ph ^ 1u, a.wait_ns, abort_flag);
          if (!got) fail();
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        // gathered stage (the selected items; every stage of the dense path): all eight warps, one
        // arrival per thread once its copies have landed
        const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
        if (warp == 0 && lane == 0) mbar_arrive(&ctl.afull[s]);
        issue_a(bi, sa, d0, dok);
        issue_b(rb, sa);
        cp_async_arrive(&ctl.full[s]);
        ++issued;
      }
    }
    if (!a.sel && a.count_step && blockIdx.x == 0 && threadIdx.x == 0) *a.step += 1;
    // every copy this warp started must land before the CTA can exit (the slab tiles: through their
    // barriers, for the last STAGES stages issued; earlier ones were consumed by the MMAs)
    cp_async_wait_all();
    if (warp == 0 && lane == 0) {
      const uint32_t lo = issued > static_cast<uint32_t>(STAGES) ? issued - STAGES : 0;
      for (uint32_t i = lo; i < issued; ++i) {
        volatile int never = 0;
        if (!mbar_wait_bounded(&ctl.afull[i % STAGES], (i / STAGES) & 1u, TC_DRAIN_NS, &never)) fail();
      }
    }
    __syncwarp();
  } else if (warp == TC_MMA_WARP) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer (one thread)
      const uint32_t idesc_s = idesc_bf16_f32(TC_BM, 2 * NP, true, true);  // A and B MN-major
      const int nrs = r1 - r0;
      uint32_t consumed = 0;
      uint32_t fph = 0;  // per slot: parity of the next phase of full[], which only gathered stages use
      int it = 0;
      bool ok = true;
      for (int unit = unit0; unit < U && ok; unit += nunits, ++it) {
        const int buf = it & 1;
        if (!mbar_wait_bounded(&ctl.tempty[buf], ((it >> 1) & 1) ^ 1, a.wait_ns, abort_flag)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * TC_HALF;
        for (int bi = 0; bi < nblk; ++bi) {
          const int s = consumed % STAGES;
          const uint32_t ph = (consumed / STAGES) & 1u;
          const bool gathered = !(slab && bi < nrs);
          if ((gathered && !mbar_wait_bounded(&ctl.full[s], (fph >> s) & 1u, a.wait_ns, abort_flag)) ||
              !mbar_wait_bounded(&ctl.afull[s], ph, a.wait_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          if (gathered) fph ^= 1u << s;
          fence_proxy_async();
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
          // descriptors once per stage: a K step of 16 items moves A and B (both MN-major) by 2048
          // bytes (+128)
          const uint64_t ad = smem_desc_sw128(sa, TC_BK * 128, 1024u);
          const uint64_t bd = smem_desc_sw128(sa + Cfg::A_BYTES, TC_BK * 128, 1024u);
          umma_f16(d_tmem, ad, bd, idesc_s, bi > 0 ? 1u : 0u);
          umma_f16(d_tmem, ad + 128, bd + 128, idesc_s, 1u);
          umma_f16(d_tmem, ad + 256, bd + 256, idesc_s, 1u);
          umma_f16(d_tmem, ad + 384, bd + 384, idesc_s, 1u);
          umma_commit(&ctl.empty[s]);
          ++consumed;
        }
        if (!ok) break;
        umma_commit(&ctl.tfull[buf]);
      }
      umma_commit(&ctl.drain);
      volatile int never = 0;
      if (!mbar_wait_bounded(&ctl.drain, 0, TC_DRAIN_NS, &never)) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 9..12)
    const int q = warp & 3;
    const int r = 32 * q + lane;
    const int et = threadIdx.x - 32 * TC_EPI0;
    int it = 0;
    for (int unit = unit0; unit < U; unit += nunits, ++it) {
      const int buf = it & 1;
      if (et == 0)
        ctl.seg_ok[buf] = mbar_wait_bounded(&ctl.tfull[buf], (it >> 1) & 1, a.wait_ns, abort_flag) ? 1 : 0;
      epi_bar();
      if (!ctl.seg_ok[buf]) {
        if (et == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf) * TC_HALF;
      // tokens 0..NP-1 of the z hi and lo halves of the accumulator
      float yv[NP];
#pragma unroll
      for (int c = 0; c < NP; c += 16) {
        uint32_t t16[16], l16[16];
        tmem_ld16(taddr + c, t16);
        tmem_ld16(taddr + NP + c, l16);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) yv[c + i] = __uint_as_float(t16[i]) + __uint_as_float(l16[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl.tempty[buf]);
      if (SK > 1) {
        // partial of a split unit: to this CTA's shared memory (the stage ring, idle by now: all
        // copies landed and all MMAs finished), token-major: pb[t * 128 + row]
        float* pb = reinterpret_cast<float*>(smem) + r;
#pragma unroll
        for (int c = 0; c < NP; ++c) pb[c * TC_BM] = yv[c];
        continue;
      }
      const int d = unit_lo(unit) + r;
      if (d < unit_lo(unit + 1)) {
#pragma unroll
        for (int b = 0; b < NP; ++b) {
          if (b < a.B) {
            if (a.out_f32)
              static_cast<float*>(a.y)[static_cast<size_t>(b) * a.D + d] = yv[b];
            else
              static_cast<__nv_bfloat16*>(a.y)[static_cast<size_t>(b) * a.D + d] = __float2bfloat16_rn(yv[b]);
          }
        }
      }
    }
  }

  if (SK > 1) {
    // ------------------------------------------------------------ cluster reduction of the split unit
    // Every thread of the cluster passes both barriers. Between them the epilogue threads of rank
    // `rank` finish its share of the unit's rows (cluster_finish), adding the SK partials in rank order.
    cluster_sync_all();
    if (warp >= TC_EPI0 && unit0 < U && !*abort_flag) {
      const int et = threadIdx.x - 32 * TC_EPI0;
      const uint32_t pb = smem_u32(smem);
      const int d_lo = unit_lo(unit0), d_hi = unit_lo(unit0 + 1);
      switch (SK) {
        case 2: cluster_finish<NP, 2>(a, pb, rank, et, d_lo, d_hi); break;
        case 4: cluster_finish<NP, 4>(a, pb, rank, et, d_lo, d_hi); break;
        default: cluster_finish<NP, 8>(a, pb, rank, et, d_lo, d_hi); break;
      }
    }
    cluster_sync_all();  // no CTA leaves while a peer may still read its partials
  }

  tc_fence_before();
  __syncthreads();
  if (warp == TC_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TC_TMEM_COLS);
  }
}

// ------------------------------------------------------------------ launchers
namespace {
// The gate/up work split: one CTA per SM, `units` ragged row ranges of at most 64 positions,
// rows_cap = their largest size rounded up to 16. A stage holds KS k-blocks, the most (up to 4) that
// leave three stages: longer runs per gathered row were measured to matter more than ring depth.
// Past the ring lies room for the MMA's reads of the unwritten rows of the last sub-stage (128
// rows of 128 bytes from its A tile, less what the sub-stage itself holds).
struct GuSplit {
  int grid, units, rows_cap, ks, stages;
  size_t smem;
};
GuSplit gateup_split(int P, int NP, int num_sms) {
  GuSplit g{};
  const int W = num_sms > 0 ? num_sms : 1;
  const long long m =
      P > 0 ? (P + static_cast<long long>(GU_MAX_ROWS) * W - 1) / (static_cast<long long>(GU_MAX_ROWS) * W) : 1;
  g.units = static_cast<int>(m * W);
  g.grid = W;
  const long long rows = P > 0 ? (P + g.units - 1) / g.units : 1;
  g.rows_cap = static_cast<int>((rows + 15) / 16 * 16);
  const uint32_t sub = static_cast<uint32_t>(2 * g.rows_cap + NP) * 128u;
  const uint32_t slack = sub >= TC_BM * 128u ? 0u : TC_BM * 128u - sub;
  const uint32_t budget = 227u * 1024u - 1024u - static_cast<uint32_t>(sizeof(TcCtl)) - 64u - slack;
  // KS = the most k-blocks per stage (at most 4) that still leaves three stages
  g.ks = 1;
  for (int ks = 4; ks >= 1; --ks) {
    if (budget / (ks * sub) >= 3) {
      g.ks = ks;
      break;
    }
  }
  const int st = static_cast<int>(budget / (g.ks * sub));
  g.stages = st > TC_MAX_STAGES ? TC_MAX_STAGES : (st < 2 ? 2 : st);
  g.smem = 1024 + static_cast<size_t>(g.stages) * g.ks * sub + slack;
  return g;
}

template <int NP>
cudaError_t launch_gateup_np(const CUtensorMap& xm, GateUpTcArgs a, int num_sms, cudaStream_t st) {
  const int P = a.nC + a.nR;
  if (P <= 0) return cudaSuccess;
  const GuSplit g = gateup_split(P, NP, num_sms);
  {
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(k_gateup_tc<NP>), g.smem);
    if (e != cudaSuccess) return e;
  }
  a.units = g.units;
  a.rows_cap = g.rows_cap;
  a.ks = g.ks;
  a.stages = g.stages;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(g.grid);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = g.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_gateup_tc<NP>, xm, a);
}

// The down work split: a cluster of `split` CTAs per unit of at most 128 outputs (whole groups of
// 8), plus the selecting cluster first. Among splits 1, 2, 4, 8 (each at most the k-blocks of the
// shorter of R and S, or of R alone) take the one whose busiest CTA streams the fewest
// rows x k-blocks, with units of at least 64 outputs where possible (shorter runs per gathered
// column cost DRAM efficiency); ties go to the smaller split.
template <int NP>
cudaError_t launch_down_np(const CUtensorMap& zm, DownTcArgs a, int num_sms, cudaStream_t st) {
  // the ring, or the selecting CTA's keys (|C| of them) if those need more
  size_t smem = dn_smem_bytes<NP>();
  constexpr size_t kStatic = sizeof(TcCtl) + sizeof(RadixScratch<TC_PROD_THREADS>) + 2 * sizeof(int) * DN_WIN_WORDS + 64;
  constexpr size_t kMaxDyn = 227 * 1024 - kStatic;
  const size_t c16 = (static_cast<size_t>(a.nC) * 4 + 15) & ~size_t(15);
  const size_t keys_bytes = 1024 + c16;
  // the selecting CTA: keys, scores, channels of C, S and (periodic) the memory in shared memory
  const size_t small_bytes = keys_bytes + 2 * c16 + ((static_cast<size_t>(a.k) * 4 + 15) & ~size_t(15)) +
                             (a.period > 1 ? c16 : 0);
  if (a.sel) {
    if (keys_bytes > kMaxDyn) return cudaErrorInvalidValue;  // |C| beyond what one CTA's keys can hold
    const size_t want = small_bytes <= kMaxDyn ? small_bytes : keys_bytes;
    if (want > smem) smem = want;
  }
  {
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(k_down_tc<NP>), smem);
    if (e != cudaSuccess) return e;
  }
  const int G = a.D / 8;
  const int tiles = (a.D + TC_BM - 1) / TC_BM;
  const int kbs = (a.k + TC_BK - 1) / TC_BK;
  const int KBT = a.kbr + kbs;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  cfg.attrs = attr;
  const int sel = a.sel ? 1 : 0;
  if (KBT <= 0 || G <= 0) {
    // nothing to stream: the selection (or the step count) only
    if (!sel && !a.count_step) return cudaSuccess;
    a.split = 1;
    a.units = 0;
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(1);
    return cudaLaunchKernelEx(&cfg, k_down_tc<NP>, zm, a);
  }
  // The split depends only on these sizes and the device: computed once per shape (the occupancy
  // queries cost host time on every step otherwise).
  struct Key {
    int D, kbr, kbs, sel, sms, dev, slab;
  };
  struct Entry {
    Key key;
    int sk, u;
  };
  static Entry cache[8];
  static int cache_n = 0;
  static std::mutex cache_mu;
  std::lock_guard<std::mutex> lock(cache_mu);
  int dev = 0;
  (void)cudaGetDevice(&dev);
  const int slab = a.dslab != nullptr ? 1 : 0;
  const Key key{a.D, a.kbr, kbs, sel, num_sms, dev, slab};
  int best_sk = 1, best_u = tiles;
  bool hit = false;
  for (int i = 0; i < cache_n; ++i) {
    const Key& c = cache[i].key;
    if (c.D == key.D && c.kbr == key.kbr && c.kbs == key.kbs && c.sel == key.sel && c.sms == key.sms &&
        c.dev == key.dev && c.slab == key.slab) {
      best_sk = cache[i].sk;
      best_u = cache[i].u;
      hit = true;
      break;
    }
  }
  const int minblk = a.kbr > 0 && kbs > 0 ? (a.kbr < kbs ? a.kbr : kbs) : KBT;
  const int u64 = G / 8 > 0 ? G / 8 : 1;  // units of >= 64 outputs
  long long best_cost = -1;
  for (int sk = 1; sk <= 8 && !hit; sk *= 2) {
    if (sk > 1 && sk > minblk) break;
    int ncl = num_sms;
    if (sk > 1) {
      attr[1].val.clusterDim.x = sk;
      attr[1].val.clusterDim.y = 1;
      attr[1].val.clusterDim.z = 1;
      cfg.numAttrs = 2;
      cfg.gridDim = dim3(sk * (num_sms / sk));
      ncl = 0;
      if (cudaOccupancyMaxActiveClusters(&ncl, k_down_tc<NP>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        continue;
      }
      ncl -= sel;
      if (ncl < tiles) continue;  // a split unit must have its own cluster, all resident at once
    } else {
      ncl -= sel;
    }
    if (ncl < 1) continue;
    int U = ncl < u64 ? ncl : u64;
    if (U < tiles || slab) U = tiles;  // with the slab, units are its 128-output slices
    const long long rows = 8LL * ((G + U - 1) / U);
    const long long rounds = (U + ncl - 1) / ncl;
    const long long blk = (a.kbr + sk - 1) / sk + (kbs + sk - 1) / sk;
    const long long cost = rounds * rows * blk;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_sk = sk;
      best_u = U;
    }
  }
  if (!hit) {
    cache[cache_n < 8 ? cache_n++ : 7] = Entry{key, best_sk, best_u};
  }
  a.split = best_sk;
  a.units = best_u;
  if (best_sk > 1) {
    attr[1].val.clusterDim.x = best_sk;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3((best_u + sel) * best_sk);
  } else {
    cfg.numAttrs = 1;
    const int ctas = best_u < num_sms - sel ? best_u : num_sms - sel;
    cfg.gridDim = dim3((ctas > 0 ? ctas : 1) + sel);
  }
  return cudaLaunchKernelEx(&cfg, k_down_tc<NP>, zm, a);
}
}  // namespace

cudaError_t launch_build_gu_tiles(const uint16_t* Wp, const int* rc, int D, int N, const GuSlabGeom& g, int t_lo,
                                  int t_hi, uint16_t* gu_slab, unsigned* err, cudaStream_t st) {
  if (!gu_slab || g.P <= 0 || t_hi <= t_lo) return cudaSuccess;
  const size_t chunks = static_cast<size_t>(t_hi - t_lo) * g.KB * g.arows * 8;
  const int grid = static_cast<int>(std::min<size_t>((chunks + 255) / 256, 152 * 16));
  if (gu_slab_elems(g) / 8 < (size_t(1) << 31))
    k_build_gu_slab<uint32_t><<<grid, 256, 0, st>>>(Wp, rc, D, N, g, t_lo, t_hi, gu_slab, err);
  else
    k_build_gu_slab<size_t><<<grid, 256, 0, st>>>(Wp, rc, D, N, g, t_lo, t_hi, gu_slab, err);
  return cudaGetLastError();
}

GuSlabGeom gu_slab_geom_split(int P1, int P, int D, int num_sms) {
  GuSlabGeom g = gu_slab_geom(P, D, num_sms);
  if (P1 <= 0 || P1 >= P) return g;
  const int W = num_sms > 0 ? num_sms : 1;
  // the same tile size, each region rounded up to whole tiles; grow the tiles while the two
  // regions need more tiles than there are SMs
  for (;;) {
    g.Ts = (P1 + g.RT - 1) / g.RT;
    g.T = g.Ts + (P - P1 + g.RT - 1) / g.RT;
    if (g.T <= W) break;
    g.RT += g.RT < GU_MAX_ROWS ? 16 : 8;
  }
  g.P1 = P1;
  g.paired = g.RT <= GU_MAX_ROWS ? 1 : 0;
  if (g.paired) {
    const int jm = g.RT - 1;
    g.arows = ((32 * (jm >> 4) + 16 + (jm & 15) + 1) + 7) / 8 * 8;
  } else {
    g.arows = 2 * ((g.RT + 7) / 8 * 8);
  }
  return g;
}

GuSlabGeom gu_slab_geom(int P, int D, int num_sms) {
  GuSlabGeom g{};
  g.P = P;
  g.KB = (D + TC_BK - 1) / TC_BK;
  const int W = num_sms > 0 ? num_sms : 1;
  // tiles of at most 128 positions, one per SM where the positions allow it
  int T = P > 0 ? (P + 127) / 128 : 1;
  if (T < W) T = P > 0 ? (W < (P + 15) / 16 ? W : (P + 15) / 16) : 1;
  g.T = T > 0 ? T : 1;
  g.RT = P > 0 ? (P + g.T - 1) / g.T : 1;
  // whole row groups: a paired tile stores gate and up of 16 positions per 32 rows, an unpaired
  // one 8-row blocks, so other tile sizes leave rows that are streamed but hold nothing (44
  // positions in 96 rows, 10% of the bytes); fewer, fuller tiles stream fewer bytes in all
  g.RT = g.RT <= GU_MAX_ROWS ? (g.RT + 15) / 16 * 16 : (g.RT + 7) / 8 * 8;
  g.T = P > 0 ? (P + g.RT - 1) / g.RT : 1;
  g.paired = g.RT <= GU_MAX_ROWS ? 1 : 0;
  if (g.paired) {
    const int jm = g.RT - 1;
    g.arows = ((32 * (jm >> 4) + 16 + (jm & 15) + 1) + 7) / 8 * 8;
  } else {
    g.arows = 2 * ((g.RT + 7) / 8 * 8);
  }
  return g;
}

size_t gu_slab_elems(const GuSlabGeom& g) { return static_cast<size_t>(g.T) * g.KB * g.arows * 64; }

size_t dn_slab_elems(int D, int nR) {
  const size_t O = (D + TC_BM - 1) / TC_BM, kbr = (nR + TC_BK - 1) / TC_BK;
  return O * kbr * TC_BK * TC_BM;
}

cudaError_t launch_build_slabs(const uint16_t* Wp, const int* rc, int nC, int nR, int D, int N, const GuSlabGeom& g,
                               uint16_t* gu_slab, uint16_t* dn_slab, unsigned* err, cudaStream_t st) {
  if (gu_slab && g.P > 0) {
    cudaError_t e = launch_build_gu_tiles(Wp, rc, D, N, g, 0, g.T, gu_slab, err, st);
    if (e != cudaSuccess) return e;
  }
  if (dn_slab && nR > 0) {
    k_build_dn_slab<<<1184, 256, 0, st>>>(Wp, rc, nC, nR, D, N, (nR + TC_BK - 1) / TC_BK, dn_slab, err);
    return cudaGetLastError();
  }
  return cudaSuccess;
}

namespace {
// The slab gate/up stage: KS k-blocks (the most, up to 4, that leave three stages); past the ring,
// room for the MMA's reads of 128 rows from the last A image's gate (and up) base.
template <int NP>
cudaError_t launch_gateup_slab_np(const CUtensorMap& xm, GateUpSlabArgs a, int num_sms, cudaStream_t st) {
  const GuSlabGeom& g = a.geom;
  if (g.P <= 0) return cudaSuccess;
  const uint32_t ab = static_cast<uint32_t>(g.arows) * 128u, xb = NP * 128u;
  const uint32_t up = g.paired ? 0u : static_cast<uint32_t>((g.RT + 7) / 8 * 8) * 128u;
  const uint32_t budget = 227u * 1024u - 1024u - static_cast<uint32_t>(sizeof(TcCtl)) - 64u;
  int ks = 1;
  uint32_t slack = 0;
  for (int k = 4; k >= 1; --k) {
    const uint32_t stage = k * (ab + xb);
    const uint32_t reach = (k - 1) * ab + up + TC_BM * 128u;  // end of the last MMA read from the stage base
    const uint32_t sl = reach > stage ? reach - stage : 0u;
    if (budget > sl && (budget - sl) / stage >= 3) {
      ks = k;
      slack = sl;
      break;
    }
    if (k == 1) {
      slack = sl;
    }
  }
  const uint32_t stage = ks * (ab + xb);
  int stages = static_cast<int>((budget - slack) / stage);
  stages = stages > TC_MAX_STAGES ? TC_MAX_STAGES : stages;
  if (stages < 2) return cudaErrorInvalidValue;
  const size_t smem = 1024 + static_cast<size_t>(stages) * stage + slack;
  {
    cudaError_t e = g.paired ? ensure_dyn_smem(reinterpret_cast<const void*>(k_gateup_slab<NP, true>), smem)
                             : ensure_dyn_smem(reinterpret_cast<const void*>(k_gateup_slab<NP, false>), smem);
    if (e != cudaSuccess) return e;
  }
  a.ks = ks;
  a.stages = stages;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(g.T < num_sms ? g.T : num_sms);
  cfg.blockDim = dim3(GS_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return g.paired ? cudaLaunchKernelEx(&cfg, k_gateup_slab<NP, true>, xm, a)
                  : cudaLaunchKernelEx(&cfg, k_gateup_slab<NP, false>, xm, a);
}
}  // namespace

cudaError_t launch_gateup_slab(const CUtensorMap& x_map, GateUpSlabArgs args, int num_sms, cudaStream_t st) {
  switch (args.NP) {
    case 16: return launch_gateup_slab_np<16>(x_map, args, num_sms, st);
    case 32: return launch_gateup_slab_np<32>(x_map, args, num_sms, st);
    case 48: return launch_gateup_slab_np<48>(x_map, args, num_sms, st);
    case 64: return launch_gateup_slab_np<64>(x_map, args, num_sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gateup_tc(const CUtensorMap& x_map, GateUpTcArgs args, int num_sms, cudaStream_t st) {
  switch (args.NP) {
    case 16: return launch_gateup_np<16>(x_map, args, num_sms, st);
    case 32: return launch_gateup_np<32>(x_map, args, num_sms, st);
    case 48: return launch_gateup_np<48>(x_map, args, num_sms, st);
    case 64: return launch_gateup_np<64>(x_map, args, num_sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_down_tc(const CUtensorMap& z_map, DownTcArgs args, int num_sms, cudaStream_t st) {
  switch (args.NP) {
    case 16: return launch_down_np<16>(z_map, args, num_sms, st);
    case 32: return launch_down_np<32>(z_map, args, num_sms, st);
    case 48: return launch_down_np<48>(z_map, args, num_sms, st);
    case 64: return launch_down_np<64>(z_map, args, num_sms, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pop
