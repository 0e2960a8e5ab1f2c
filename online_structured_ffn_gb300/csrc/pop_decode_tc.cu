// Decode step of the POP FFN for B > 1 sequences on the 5th-generation tensor cores.
//
// What it computes ("POP: Online Structural Pruning..." notes, Key design 2; "Batch-wise adaptive
// pruning", Fig. 2(a) for the batch max):
//   gate/up: for every position p of rc = [C | R] and token b, z[b][p] = SiLU(Wg[c] x_b) * (W1[c] x_b)
//            with c = rc[p]; score[p] = max_b |z[b][p]| * ||W2[:, c]|| for the candidates p < |C|;
//   down:    y[b][d] = sum over the kept items j (R, then S) of z[b][j] * W2[d, channel of j].
//
// The MMA inputs are bf16. x and the weights are bf16 already; z is not, and rounding it to bf16
// would cost about 3 significant digits of y. So the down GEMM takes z as two bf16 planes, hi =
// bf16(z) and lo = bf16(z - hi), stacked as 2 x 16..64 token columns of one MMA; the epilogue adds
// the two halves, which leaves z's own fp32 rounding well below the output tolerance.
//
// Both are skinny GEMMs with the tokens as the MMA's N (16..64, zero-padded to a multiple of 16)
// and 128 rows as M: 128 positions (gate/up; the A tiles are gathered rows of the packed weights,
// K-major) or 128 outputs d (down; A is gathered down columns, MN-major since d is contiguous in a
// packed row). The producer warps gather the rows straight from the packed weights with 16-byte
// cp.async copies into the 128-byte swizzle layout (no copy of the pruned weights is ever made;
// TMA's four-row gather moved too few bytes per operation to keep up with HBM here). The x (or z)
// tile is an ordinary TMA box.
//
// Work split. With few tiles (the usual decode shapes: |R u C| / 128 or D / 128 is well below the
// SM count) every tile is split along K over a cluster of `split` CTAs (1 CTA per SM, 2 / 4 / 8 per
// cluster); each CTA streams 1/split of the tile's k-blocks, then the partial accumulators are
// added through distributed shared memory in rank order (a fixed order: results do not depend on
// timing), each CTA finishing 128 / split of the rows. No workspace, no atomics. With many tiles
// (split = 1), CTAs take whole tiles round-robin and finish them straight from TMEM.
//
// Roles (224 threads): warps 0-1 issue the copies, warp 2 lane 0 issues the MMAs and owns TMEM
// (two accumulator buffers, so the epilogue of one tile overlaps the MMAs of the next), warps 3-6
// are the epilogue (one TMEM lane quarter each). Every wait is bounded; on a time-out the CTA
// records DEVERR_TIMEOUT_DECODE_TC, stops issuing, drains its own copies and MMAs (bounded), frees
// TMEM and returns. The epilogue warps take every decision that guards a named barrier together,
// and every thread reaches the cluster barriers, so a time-out cannot leave a barrier waiting.
//
// Programmatic dependent launch: the set-up (barriers, TMEM, tensor-map prefetch) runs before
// griddepcontrol.wait; every global read or write of this step's data comes after it.
#include "pop_device.cuh"
#include "pop_internal.h"

namespace pop {

namespace {
constexpr int TC_THREADS = 224;
constexpr int TC_PRODUCERS = 2;  // warps 0-1 gather rows, warp 2 issues MMAs, warps 3-6 are the epilogue
constexpr int TC_MMA_WARP = TC_PRODUCERS;
constexpr int TC_BM = 128;
constexpr int TC_BK = 64;
constexpr uint64_t TC_DRAIN_NS = 1000000000ull;
// shared memory for the stage ring (the down kernel also keeps its row-offset windows)
constexpr uint32_t TC_RING_BUDGET[2] = {212 * 1024, 192 * 1024};
// down: row offsets of the items of up to TC_WIN k-blocks, per producer warp (its 32 rows of each)
constexpr int TC_WIN = 64;

// A stage holds KS = 2 consecutive 64-wide k-blocks ("sub-stages"): gate/up rows are then read in
// 256 contiguous bytes (measured faster than 128), and the down GEMM's per-stage overhead is halved
// (4 k-blocks per stage measured slower: fewer, larger stages). Sub-stage layout: A (weight rows) then B (token tile).
// Gate/up: A = 128 gate rows + 128 up rows of 128 bytes, B = NP rows of x. Down: A = 64 items x
// 128 outputs (two 64-wide halves), B = the hi and lo planes of z, NP rows each. As many stages as
// fit the budget (at most 8).
template <int MODE, int NP>
struct TcCfg {
  static constexpr int KS = 2;
  static constexpr uint32_t A_BYTES = MODE == 0 ? 2 * TC_BM * TC_BK * 2 : TC_BM * TC_BK * 2;
  static constexpr uint32_t B_BYTES = (MODE == 0 ? NP : 2 * NP) * TC_BK * 2;
  static constexpr uint32_t SUB_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t STAGE_BYTES = KS * SUB_BYTES;
  static constexpr int STAGES = TC_RING_BUDGET[MODE] / STAGE_BYTES < 8 ? TC_RING_BUDGET[MODE] / STAGE_BYTES : 8;
  static constexpr uint32_t TMEM_COLS = 256;  // two accumulator buffers of 2 x NP <= 128 columns
  // partial accumulators exchanged in a cluster, fp32 per row: [g | u] (gate/up) or hi + lo (down)
  static constexpr int PCOLS = MODE == 0 ? 2 * NP : NP;
  static_assert(SUB_BYTES % 1024 == 0, "sub-stages must keep the 1024-byte swizzle alignment");
  static_assert(static_cast<uint32_t>(TC_BM * PCOLS * 4) <= STAGES * STAGE_BYTES, "partials reuse the ring");
};

struct TcCtl {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int seg_ok[2];  // by tile parity: a warp may still read one while the next is written
  float n2s[TC_BM];                 // gate/up, split tiles: norms of the rows each epilogue thread finishes
};

template <int MODE, int NP>
constexpr size_t tc_smem_bytes() {
  return 1024 + TcCfg<MODE, NP>::STAGES * TcCfg<MODE, NP>::STAGE_BYTES + sizeof(TcCtl) +
         (MODE == 1 ? TC_PRODUCERS * TC_WIN * 32 * sizeof(uint32_t) : 0);
}

__device__ __forceinline__ float silu_t(float g) { return g / (1.0f + expf(-g)); }

__device__ __forceinline__ int guard_ch(int v, int n, unsigned* err) {
  if (static_cast<unsigned>(v) >= static_cast<unsigned>(n)) {
    atomicOr(err, DEVERR_INDEX);
    return 0;
  }
  return v;
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros (nothing is read). No
// compiler memory barrier: the source is read-only and the destination is touched by nothing else
// of this thread before the commit / wait below, which do carry one; so the address arithmetic
// of consecutive copies can overlap.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
// Makes this thread's shared-memory writes (its landed cp.async copies) visible to the tensor cores.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

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
__device__ __forceinline__ float2 ld_peer2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
}  // namespace

// NP: tokens padded to a multiple of 16 (16..64), a template parameter so that every per-token
// loop of the epilogue has a fixed trip count (no per-column branches between its loads).
template <int MODE, int NP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k_decode_tc(const __grid_constant__ CUtensorMap mapB, const __grid_constant__ CUtensorMap mapB2,
                const __grid_constant__ DecodeTcArgs a) {
  using Cfg = TcCfg<MODE, NP>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr uint32_t STAGE_BYTES = Cfg::STAGE_BYTES;
  constexpr uint32_t HALF_COLS = Cfg::TMEM_COLS / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcCtl* ctl = reinterpret_cast<TcCtl*>(smem + STAGES * STAGE_BYTES);
  volatile int* abort_flag = &ctl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = (a.rows + TC_BM - 1) / TC_BM;
  const int KB = (a.K + TC_BK - 1) / TC_BK;
  constexpr int KSUB = Cfg::KS;
  const int KBS = (KB + KSUB - 1) / KSUB;  // stages per tile
  // this CTA's work: tiles unit, unit + nunits, ...; stages [sb_lo, sb_hi) of each
  const int SK = a.split;
  const uint32_t rank = SK > 1 ? cluster_rank() : 0u;
  const int unit = static_cast<int>(blockIdx.x) / SK, nunits = static_cast<int>(gridDim.x) / SK;
  const int sb_lo = static_cast<int>(rank) * KBS / SK, sb_hi = (static_cast<int>(rank) + 1) * KBS / SK;
  const int kb_end = min(KB, sb_hi * KSUB);  // this CTA's k-blocks: [sb_lo * KSUB, kb_end)
  // bytes the TMA boxes bring per stage (the weight rows come by cp.async): NP token rows of x
  // (gate/up) or 2 x NP (the hi and lo planes of z, down)
  const uint32_t tx_bytes = KSUB * static_cast<uint32_t>(MODE == 0 ? NP : 2 * NP) * TC_BK * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 32 * TC_PRODUCERS + 1);  // producer lanes + the TMA transaction count
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->tfull[b], 1);
      mbar_init(&ctl->tempty[b], 4);
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
    if (MODE == 1) prefetch_tmap(&mapB2);
    prefetch_tmap(&mapB);
  }
  if (warp == TC_MMA_WARP) {
    tmem_alloc(&ctl->tmem_base, Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  auto fail = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      atomicOr(a.err, DEVERR_TIMEOUT_DECODE_TC);
    }
  };

  if (warp < TC_PRODUCERS) {
    // ------------------------------------------------------------ producers (two whole warps)
    // The weight rows of a stage are gathered with 16-byte cp.async copies (lane l of producer warp
    // w copies chunk l % 8 of rows rg, rg + 8, ... with rg = l / 8 + 4 w), each written to its place
    // in the 128-byte swizzle pattern; the token tile (x, or the two z planes) is a TMA box issued
    // by warp 0. One commit group per stage: once a lane's group for stage i has landed (checked LAG
    // stages later, so LAG + 1 stages of copies stay in flight) the lane fences its writes for the
    // async proxy and arrives on the stage's barrier; warp 0 lane 0 also arrives with the TMA byte
    // count when it issues the box.
    const int cq = lane & 7, rg = (lane >> 3) + 4 * warp;
    constexpr int LAG = STAGES - 1;
    const uint16_t* Wbase = a.Wp + (MODE == 0 ? 0 : 2 * static_cast<size_t>(a.D));
    const size_t row3 = 3 * static_cast<size_t>(a.D);
    uint32_t issued = 0;
    bool ok = true;
    // Down: the row offsets of the items this warp copies (rows rg + 8m of each k-block), for a
    // window of up to TC_WIN k-blocks at a time, in shared memory. Lane l of warp w fetches item
    // (4w + l % 4) + 8 (l / 4) of each k-block of the window (one load per k-block, all in flight at
    // once); the lane that copies rows rg + 8m reads entry (rg - 4w) + 4m. Each warp fills and reads
    // only its own table, so the warps never wait on each other.
    uint32_t* win = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(ctl) + sizeof(TcCtl)) +
                    warp * TC_WIN * 32;
    int win_lo = -1, win_hi = -1;  // k-blocks [win_lo, win_hi) are in the window
    auto fill_window = [&](int kb0w) {
      win_lo = kb0w;
      win_hi = min(kb_end, kb0w + TC_WIN);
      const int item_in_kb = 4 * warp + (lane & 3) + 8 * (lane >> 2);
      __syncwarp();
      for (int c0 = win_lo; c0 < win_hi; c0 += 16) {
        int v[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int item = (c0 + u) * TC_BK + item_in_kb;
          v[u] = 0;
          if (c0 + u < win_hi && item < a.K) v[u] = item < a.nR_items ? a.ch_r[item] : a.ch_s[item - a.nR_items];
        }
#pragma unroll
        for (int u = 0; u < 16; ++u)
          if (c0 + u < win_hi) win[(c0 + u - win_lo) * 32 + lane] = static_cast<uint32_t>(guard_ch(v[u], a.N, a.err)) * row3;
      }
      __syncwarp();
    };
    for (int tile = unit; tile < tiles && ok; tile += nunits) {
      // MODE 0: the tile's 128 rows are positions 128 * tile + r; this lane copies rows rg + 8m.
      // MODE 1: the k-block's 64 rows are items 64 * kb + r; this lane copies items rg + 8m.
      // Row offsets (elements) stay in registers.
      constexpr int NROW = MODE == 0 ? TC_BM / 8 : TC_BK / 8;
      uint32_t rowoff[NROW];
      auto set_rows = [&](const int (&ids)[NROW]) {
#pragma unroll
        for (int m = 0; m < NROW; ++m) rowoff[m] = static_cast<uint32_t>(guard_ch(ids[m], a.N, a.err)) * row3;
      };
      if (MODE == 0) {
        int ids[NROW];
#pragma unroll
        for (int m = 0; m < NROW; ++m) {
          const int p = tile * TC_BM + rg + 8 * m;
          ids[m] = p < a.rows ? a.rc[p] : 0;
        }
        set_rows(ids);
      }
      for (int sbk = sb_lo; sbk < sb_hi; ++sbk) {
        uint32_t rowsub[KSUB][MODE == 1 ? NROW : 1];  // down: row offsets of each sub-stage's items
        if (MODE == 1) {
#pragma unroll
          for (int u = 0; u < KSUB; ++u) {
            const int kb = sbk * KSUB + u;
            if (kb < kb_end) {
              if (kb < win_lo || kb >= win_hi) fill_window(kb);
              const uint32_t* wrow = win + (kb - win_lo) * 32 + (rg - 4 * warp);
#pragma unroll
              for (int m = 0; m < NROW; ++m) rowsub[u][m % (MODE == 1 ? NROW : 1)] = wrow[4 * m];
            } else {
#pragma unroll
              for (int m = 0; m < NROW; ++m) rowsub[u][m % (MODE == 1 ? NROW : 1)] = 0u;  // past K: zeros
            }
          }
        }
        const int s = issued % STAGES;
        const uint32_t ph = (issued / STAGES) & 1u;
        bool got = true;
        if (lane == 0) {
          got = mbar_wait_bounded(&ctl->empty[s], ph ^ 1u, a.wait_ns, abort_flag);
          if (!got) fail();
          else if (warp == 0) mbar_arrive_expect_tx(&ctl->full[s], tx_bytes);
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
        if (MODE == 0) {
          // row by row, both k-blocks: KSUB x 128 contiguous bytes of each row back to back
#pragma unroll
          for (int m = 0; m < NROW; ++m) {
            const int r = rg + 8 * m;
#pragma unroll
            for (int u = 0; u < KSUB; ++u) {
              const int d0 = (sbk * KSUB + u) * TC_BK + 8 * cq;
              const uint32_t nbytes = d0 < a.D ? 16u : 0u;  // D is a multiple of 8: chunks all in or out
              const uint16_t* src = Wbase + rowoff[m] + (nbytes ? d0 : 0);
              const uint32_t dst = sa + u * Cfg::SUB_BYTES + r * 128 + ((cq ^ (r & 7)) << 4);
              cp_async16(dst, src, nbytes);
              cp_async16(dst + TC_BM * 128, src + a.D, nbytes);
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < KSUB; ++u) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int d0 = tile * TC_BM + 64 * h + 8 * cq;
              const uint32_t nbytes = d0 < a.D ? 16u : 0u;
              const uint16_t* base = Wbase + (nbytes ? d0 : 0);
#pragma unroll
              for (int m = 0; m < NROW; ++m) {
                const int r = rg + 8 * m;
                cp_async16(sa + u * Cfg::SUB_BYTES + h * (TC_BK * 128) + r * 128 + ((cq ^ (r & 7)) << 4),
                           base + rowsub[u][m % (MODE == 1 ? NROW : 1)], nbytes);
              }
            }
          }
        }
        cp_async_commit();
        if (issued >= static_cast<uint32_t>(LAG)) {
          cp_async_wait<LAG>();
          fence_proxy_async();
          mbar_arrive(&ctl->full[(issued - LAG) % STAGES]);
        }
        if (warp == 0 && lane == 0) {
#pragma unroll
          for (int u = 0; u < KSUB; ++u) {
            uint8_t* sb = smem + s * STAGE_BYTES + u * Cfg::SUB_BYTES + Cfg::A_BYTES;
            const int kx = (sbk * KSUB + u) * TC_BK;  // may lie past K: the box then reads zeros
            tma_load_2d(sb, &mapB, &ctl->full[s], kx, 0);
            if (MODE == 1) tma_load_2d(sb + NP * 128, &mapB2, &ctl->full[s], kx, 0);  // z lo plane
          }
        }
        ++issued;
      }
    }
    // the last stages' arrivals, and every copy this warp started must land before the CTA can exit
    cp_async_wait<0>();
    fence_proxy_async();
    if (ok)
      for (uint32_t u = issued > static_cast<uint32_t>(LAG) ? issued - LAG : 0; u < issued; ++u)
        mbar_arrive(&ctl->full[u % STAGES]);
    if (warp == 0 && lane == 0) {
      const uint32_t lo = issued > static_cast<uint32_t>(STAGES) ? issued - STAGES : 0;
      for (uint32_t u = lo; u < issued; ++u) {
        volatile int never = 0;
        if (!mbar_wait_bounded(&ctl->full[u % STAGES], (u / STAGES) & 1u, TC_DRAIN_NS, &never)) fail();
      }
    }
    __syncwarp();
  } else if (warp == TC_MMA_WARP) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer (one thread)
      const uint32_t idesc = idesc_bf16_f32(TC_BM, MODE == 0 ? NP : 2 * NP, false, MODE == 1);
      uint32_t consumed = 0;
      int it = 0;
      bool ok = true;
      for (int tile = unit; tile < tiles && ok; tile += nunits, ++it) {
        const int buf = it & 1;
        if (!mbar_wait_bounded(&ctl->tempty[buf], ((it >> 1) & 1) ^ 1, a.wait_ns, abort_flag)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * HALF_COLS;
        for (int sbk = sb_lo; sbk < sb_hi; ++sbk) {
          const int s = consumed % STAGES;
          const uint32_t ph = (consumed / STAGES) & 1u;
          if (!mbar_wait_bounded(&ctl->full[s], ph, a.wait_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int u = 0; u < KSUB; ++u) {
            const uint32_t sa = smem_u32(smem + s * STAGE_BYTES) + u * Cfg::SUB_BYTES;
            const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
            for (int k = 0; k < TC_BK / 16; ++k) {
              const uint32_t acc = (sbk > sb_lo || u > 0 || k > 0) ? 1u : 0u;
              const uint64_t bdesc = smem_desc_sw128(sb + 32u * k, 16u, 1024u);
              if (MODE == 0) {
                umma_f16(d_tmem, smem_desc_sw128(sa + 32u * k, 16u, 1024u), bdesc, idesc, acc);
                umma_f16(d_tmem + static_cast<uint32_t>(NP),
                         smem_desc_sw128(sa + TC_BM * 128 + 32u * k, 16u, 1024u), bdesc, idesc, acc);
              } else {
                umma_f16(d_tmem, smem_desc_sw128(sa + 2048u * k, TC_BK * 128, 1024u), bdesc, idesc, acc);
              }
            }
          }
          umma_commit(&ctl->empty[s]);
          ++consumed;
        }
        if (!ok) break;
        umma_commit(&ctl->tfull[buf]);
      }
      // all MMAs issued by this thread must finish before TMEM is freed
      umma_commit(&ctl->drain);
      volatile int never = 0;
      if (!mbar_wait_bounded(&ctl->drain, 0, TC_DRAIN_NS, &never)) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 3..6)
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int r = 32 * q + lane;
    const int et = threadIdx.x - 32 * (TC_MMA_WARP + 1);  // 0..127
    // split tiles: the norm of the candidate row this thread finishes after the cluster exchange,
    // fetched now while the tile streams
    if (MODE == 0 && SK > 1 && unit < tiles) {
      const int p = unit * TC_BM + static_cast<int>(rank) * (TC_BM / SK) + et / SK;
      if (p < a.nC) ctl->n2s[et] = a.n2[guard_ch(a.rc[p], a.N, a.err)];
    }
    int it = 0;
    for (int tile = unit; tile < tiles; tile += nunits, ++it) {
      const int buf = it & 1;
      // the candidates' down-column norms, fetched while the accumulators are still being built
      float n2v = 0.f;
      if (MODE == 0 && SK == 1) {
        const int p = tile * TC_BM + r;
        if (p < a.nC) n2v = a.n2[guard_ch(a.rc[p], a.N, a.err)];
      }
      if (et == 0)
        ctl->seg_ok[it & 1] = mbar_wait_bounded(&ctl->tfull[buf], (it >> 1) & 1, a.wait_ns, abort_flag) ? 1 : 0;
      epi_bar();
      if (!ctl->seg_ok[it & 1]) {
        if (et == 0) fail();
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf) * HALF_COLS;
      // tokens 0..NP-1 of the accumulator halves: gate and up (gate/up), or the z hi and lo parts (down)
      float gv[NP], uv[NP];
#pragma unroll
      for (int c = 0; c < NP; c += 16) {
        uint32_t t16[16];
        tmem_ld16(taddr + c, t16);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) gv[c + j] = __uint_as_float(t16[j]);
        tmem_ld16(taddr + NP + c, t16);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 16; ++j) uv[c + j] = __uint_as_float(t16[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->tempty[buf]);

      if (SK > 1) {
        // partial of a split tile: to this CTA's shared memory (the stage ring, idle by now: all
        // copies landed and all MMAs finished), rows of PCOLS floats
        float* pb = reinterpret_cast<float*>(smem) + r * Cfg::PCOLS;
#pragma unroll
        for (int c = 0; c < NP; ++c) {
          if (MODE == 0) {
            pb[c] = gv[c];
            pb[NP + c] = uv[c];
          } else {
            pb[c] = gv[c] + uv[c];
          }
        }
        continue;
      }
      if (MODE == 0) {
        const int p = tile * TC_BM + r;
        if (p < a.rows) {
          float m = 0.f;
#pragma unroll
          for (int b = 0; b < NP; ++b) {
            if (b < a.B) {
              const float zz = silu_t(gv[b]) * uv[b];
              a.z[static_cast<size_t>(b) * a.ldz + p] = zz;
              if (p >= a.nC) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(zz);
                const __nv_bfloat16 lo = __float2bfloat16_rn(zz - __bfloat162float(hi));
                const size_t o = static_cast<size_t>(b) * a.ldk + (p - a.nC);
                a.zk[o] = *reinterpret_cast<const uint16_t*>(&hi);
                a.zk_lo[o] = *reinterpret_cast<const uint16_t*>(&lo);
              }
              m = fmaxf(m, fabsf(zz));
            }
          }
          if (p < a.nC) a.scores[p] = m * n2v;
        }
      } else {
        const int d = tile * TC_BM + r;
        if (d < a.rows) {
#pragma unroll
          for (int b = 0; b < NP; ++b) {
            if (b < a.B) {
              const float yv = gv[b] + uv[b];
              if (a.out_f32)
                static_cast<float*>(a.y)[static_cast<size_t>(b) * a.rows + d] = yv;
              else
                static_cast<__nv_bfloat16*>(a.y)[static_cast<size_t>(b) * a.rows + d] = __float2bfloat16_rn(yv);
            }
          }
        }
      }
    }
  }

  if (SK > 1) {
    // ------------------------------------------------------------ cluster reduction of the split tile
    // Every thread of the cluster passes both barriers. Between them, epilogue thread et of rank
    // `rank` finishes row rank * 128 / SK + et / SK for tokens [part * NP / SK, (part + 1) * NP / SK),
    // part = et % SK, adding the SK partials in rank order.
    cluster_sync_all();
    if (warp > TC_MMA_WARP && unit < tiles && !*abort_flag) {
      const int et = threadIdx.x - 32 * (TC_MMA_WARP + 1);
      const int rows_per = TC_BM / SK, tpt = NP / SK;
      const int rl = et / SK, part = et % SK;
      const int row = static_cast<int>(rank) * rows_per + rl;
      const int b0 = part * tpt;
      const uint32_t pbase = smem_u32(smem) + static_cast<uint32_t>(row * Cfg::PCOLS) * 4u;
      float m = 0.f;
      const int p = unit * TC_BM + row;
      const float n2v = MODE == 0 && p < a.nC ? ctl->n2s[et] : 0.f;
      uint32_t peer[8];
#pragma unroll
      for (int pr = 0; pr < 8; ++pr) peer[pr] = pr < SK ? map_peer(pbase, static_cast<uint32_t>(pr)) : 0u;
      // tokens two at a time (tpt = NP / SK is even): SK peers x 8-byte loads, added in rank order
#pragma unroll 2
      for (int j = 0; j < tpt; j += 2) {
        const int b = b0 + j;
        float2 g2 = make_float2(0.f, 0.f), u2 = make_float2(0.f, 0.f);
        float2 lg[8], lu[8];
#pragma unroll
        for (int pr = 0; pr < 8; ++pr) {
          if (pr < SK) {
            lg[pr] = ld_peer2(peer[pr] + 4u * b);
            if (MODE == 0) lu[pr] = ld_peer2(peer[pr] + 4u * (NP + b));
          }
        }
#pragma unroll
        for (int pr = 0; pr < 8; ++pr) {
          if (pr < SK) {
            g2.x += lg[pr].x;
            g2.y += lg[pr].y;
            if (MODE == 0) {
              u2.x += lu[pr].x;
              u2.y += lu[pr].y;
            }
          }
        }
        for (int h = 0; h < 2; ++h) {
        const int b = b0 + j + h;
        const float g = h ? g2.y : g2.x, u = h ? u2.y : u2.x;
        if (b >= a.B) continue;
        if (MODE == 0) {
          if (p < a.rows) {
            const float zz = silu_t(g) * u;
            a.z[static_cast<size_t>(b) * a.ldz + p] = zz;
            if (p >= a.nC) {
              const __nv_bfloat16 hi = __float2bfloat16_rn(zz);
              const __nv_bfloat16 lo = __float2bfloat16_rn(zz - __bfloat162float(hi));
              const size_t o = static_cast<size_t>(b) * a.ldk + (p - a.nC);
              a.zk[o] = *reinterpret_cast<const uint16_t*>(&hi);
              a.zk_lo[o] = *reinterpret_cast<const uint16_t*>(&lo);
            }
            m = fmaxf(m, fabsf(zz));
          }
        } else {
          const int d = unit * TC_BM + row;
          if (d < a.rows) {
            if (a.out_f32)
              static_cast<float*>(a.y)[static_cast<size_t>(b) * a.rows + d] = g;
            else
              static_cast<__nv_bfloat16*>(a.y)[static_cast<size_t>(b) * a.rows + d] = __float2bfloat16_rn(g);
          }
        }
        }
      }
      if (MODE == 0) {
        // the row's SK threads are adjacent lanes: combine their maxima
        for (int o = SK / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (part == 0 && p < a.nC) a.scores[p] = m * n2v;
      }
    }
    cluster_sync_all();  // no CTA leaves while a peer may still read its partials
  }

  tc_fence_before();
  __syncthreads();
  if (warp == TC_MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ launchers
template <int MODE, int NP>
static cudaError_t launch_tc_np(const CUtensorMap& b, const CUtensorMap& b2, DecodeTcArgs args, int num_sms,
                                cudaStream_t st) {
  constexpr size_t smem = tc_smem_bytes<MODE, NP>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_decode_tc<MODE, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int tiles = (args.rows + TC_BM - 1) / TC_BM;
  const int KB = (args.K + TC_BK - 1) / TC_BK;
  constexpr int KSUB = TcCfg<MODE, NP>::KS;
  const int KBS = (KB + KSUB - 1) / KSUB;
  if (tiles <= 0 || KB <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg{};
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  cfg.attrs = attr;
  // split: the largest power of two <= 8 such that tiles x split CTAs fit the SMs at once (one CTA
  // per SM) with at least one k-block per CTA, confirmed by the cluster occupancy query
  int split = 1;
  while (split < 8 && tiles * split * 2 <= num_sms && split * 2 <= KBS) split *= 2;
  for (; split > 1; split /= 2) {
    attr[1].val.clusterDim.x = split;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
    cfg.gridDim = dim3(tiles * split);
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, k_decode_tc<MODE, NP>, &cfg) == cudaSuccess && clusters >= tiles)
      break;
    (void)cudaGetLastError();
  }
  args.split = split;
  if (split == 1) {
    cfg.numAttrs = 1;
    cfg.gridDim = dim3(tiles < num_sms ? tiles : num_sms);
  }
  return cudaLaunchKernelEx(&cfg, k_decode_tc<MODE, NP>, b, b2, args);
}

template <int MODE>
static cudaError_t launch_tc(const CUtensorMap& b, const CUtensorMap& b2, const DecodeTcArgs& args, int num_sms,
                             cudaStream_t st) {
  switch (args.NP) {
    case 16: return launch_tc_np<MODE, 16>(b, b2, args, num_sms, st);
    case 32: return launch_tc_np<MODE, 32>(b, b2, args, num_sms, st);
    case 48: return launch_tc_np<MODE, 48>(b, b2, args, num_sms, st);
    case 64: return launch_tc_np<MODE, 64>(b, b2, args, num_sms, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gateup_tc(const CUtensorMap& x_map, const DecodeTcArgs& args, int num_sms, cudaStream_t st) {
  return launch_tc<0>(x_map, x_map, args, num_sms, st);
}

cudaError_t launch_down_tc(const CUtensorMap& zk_map, const CUtensorMap& zk_lo_map, const DecodeTcArgs& args,
                           int num_sms, cudaStream_t st) {
  return launch_tc<1>(zk_map, zk_lo_map, args, num_sms, st);
}

}  // namespace pop
