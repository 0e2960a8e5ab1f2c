// Decode step of the POP FFN for B > 1 sequences on the 5th-generation tensor cores.
//
// What it computes ("POP: Online Structural Pruning..." notes, Key design 2; "Batch-wise adaptive
// pruning", Fig. 2(a) for the batch max):
//   gate/up: for every position p of rc = [C | R] and token b, z[b][p] = SiLU(Wg[c] x_b) * (W1[c] x_b)
//            with c = rc[p]; score[p] = max_b |z[b][p]| * ||W2[:, c]|| for the candidates p < |C|;
//   down:    y[b][d] = sum over the kept items j of z[b][j] * W2[d, ch_list[j]] (items: R, then S).
//
// The MMA inputs are bf16. x and the weights are bf16 already; z is not, and rounding it to bf16
// would cost about 3 significant digits of y. So the down GEMM takes z as two bf16 planes, hi =
// bf16(z) and lo = bf16(z - hi), stacked as 2 x 16..64 token columns of one MMA; the epilogue adds
// the two halves, which leaves z's own fp32 rounding well below the output tolerance.
//
// Both are skinny GEMMs with the tokens as the MMA's N (16..64, zero-padded to a multiple of 16)
// and 128 rows as M: 128 positions (gate/up; the A tiles are gathered rows of the packed weights,
// K-major) or 128 outputs d (down; A is gathered down columns, MN-major since d is contiguous in a
// packed row). The producer warp gathers the rows straight from the packed weights with 16-byte
// cp.async copies into the 128-byte swizzle layout (no copy of the pruned weights is ever made;
// TMA's four-row gather moved too few bytes per operation to keep up with HBM here). The x (or z)
// tile is an ordinary TMA box.
//
// Work split: stream-K over the (tile, 64-wide k-block) iterations, one CTA per SM, so every SM
// streams the same number of weight bytes (+-1 k-block) whatever the tile count. A CTA's range is a
// run of segments; a segment that covers a whole tile is finished in place, the others write
// partial accumulators to a workspace and the last of a tile's contributors (atomic counter) adds
// them in CTA order (a fixed order: results do not depend on timing) and finishes the tile.
//
// Roles (192 threads): warp 0 issues the copies, warp 1 lane 0
// issues the MMAs and owns TMEM (two accumulator buffers, so the epilogue of one segment overlaps
// the MMAs of the next), warps 2..5 are the epilogue (one TMEM lane quarter each). Every wait is
// bounded; on a time-out the CTA records DEVERR_TIMEOUT_DECODE_TC, stops issuing, drains its own
// copies and MMAs (bounded), frees TMEM and returns. The epilogue warps take every decision that
// guards a named barrier together, so a time-out cannot leave one of them waiting at a barrier.
//
// Programmatic dependent launch: the set-up (barriers, TMEM, tensor-map prefetch) runs before
// griddepcontrol.wait; every global read or write of this step's data comes after it.
#include "pop_device.cuh"
#include "pop_internal.h"

namespace pop {

namespace {
constexpr int TC_THREADS = 192;
constexpr int TC_BM = 128;
constexpr int TC_BK = 64;
constexpr uint64_t TC_DRAIN_NS = 1000000000ull;
constexpr int TC_WS_COLS = 128;  // workspace columns per slot (2 x 64 tokens for gate/up)

template <int MODE>
struct TcCfg;
template <>
struct TcCfg<0> {  // gate/up: A = 128 gate rows + 128 up rows, B = x
  static constexpr int STAGES = 5;
  static constexpr uint32_t A_BYTES = 2 * TC_BM * TC_BK * 2;  // 32 KB
  static constexpr uint32_t B_BYTES = 64 * TC_BK * 2;         // room for 64 tokens
  static constexpr uint32_t TMEM_COLS = 256;                  // two buffers of [g | u] x 64 tokens
};
template <>
struct TcCfg<1> {  // down: A = 64 items x 128 outputs (two 64-wide halves), B = z hi and lo planes
  static constexpr int STAGES = 6;
  static constexpr uint32_t A_BYTES = TC_BM * TC_BK * 2;  // 16 KB
  static constexpr uint32_t B_BYTES = 2 * 64 * TC_BK * 2;  // room for 2 x 64 token rows
  static constexpr uint32_t TMEM_COLS = 256;               // two buffers of [hi | lo] x 64 tokens
};

struct TcCtl {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int seg_ok[2];  // by segment parity: a warp may still read one while the next is written
  int last;
};

template <int MODE>
constexpr size_t tc_smem_bytes() {
  return 1024 + TcCfg<MODE>::STAGES * (TcCfg<MODE>::A_BYTES + TcCfg<MODE>::B_BYTES) + sizeof(TcCtl);
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

__device__ __forceinline__ unsigned atom_add_acq_rel_tc(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Stream-K partition of T iterations over G CTAs: CTA c owns [start(c), start(c + 1)).
__device__ __forceinline__ long long sk_start(int c, long long T, int G) { return static_cast<long long>(c) * T / G; }
// The CTA that owns iteration i.
__device__ __forceinline__ int sk_owner(long long i, long long T, int G) {
  return static_cast<int>(((i + 1) * G - 1) / T);
}
}  // namespace

// NP: tokens padded to a multiple of 16 (16..64), a template parameter so that every per-token
// loop of the epilogue has a fixed trip count (no per-column branches between its loads).
template <int MODE, int NP>
__global__ void __launch_bounds__(TC_THREADS, 1)
    k_decode_tc(const __grid_constant__ CUtensorMap mapB, const __grid_constant__ CUtensorMap mapB2,
                const __grid_constant__ DecodeTcArgs a) {
  using Cfg = TcCfg<MODE>;
  constexpr int STAGES = Cfg::STAGES;
  constexpr uint32_t STAGE_BYTES = Cfg::A_BYTES + Cfg::B_BYTES;
  constexpr uint32_t HALF_COLS = Cfg::TMEM_COLS / 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  TcCtl* ctl = reinterpret_cast<TcCtl*>(smem + STAGES * STAGE_BYTES);
  volatile int* abort_flag = &ctl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tiles = (a.rows + TC_BM - 1) / TC_BM;
  const int KB = (a.K + TC_BK - 1) / TC_BK;
  const long long T = static_cast<long long>(tiles) * KB;
  const int G = gridDim.x;
  const long long s_begin = sk_start(blockIdx.x, T, G), s_end = sk_start(blockIdx.x + 1, T, G);
  // bytes the TMA boxes bring per stage (the weight rows come by cp.async): NP token rows of x
  // (gate/up) or 2 x NP (the hi and lo planes of z, down)
  const uint32_t tx_bytes = static_cast<uint32_t>(MODE == 0 ? NP : 2 * NP) * TC_BK * 2;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 33);  // the producer's 32 lanes + lane 0's TMA transaction count
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
  if (warp == 1) {
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer (whole warp)
    // The weight rows of a stage are gathered with 16-byte cp.async copies (lane l copies chunk
    // l % 8 of rows l / 8, l / 8 + 4, ...), each written to its place in the 128-byte swizzle
    // pattern; the token tile (x, or the two z planes) is a TMA box. One commit group per stage:
    // once a lane's group for stage i has landed (checked LAG stages later, so LAG + 1 stages of
    // copies stay in flight) the lane fences its writes for the async proxy and arrives on the
    // stage's barrier; lane 0 also arrives with the TMA byte count when it issues the box.
    const int cq = lane & 7, rg = lane >> 3;
    constexpr int LAG = STAGES - 2;
    const uint16_t* Wbase = a.Wp + (MODE == 0 ? 0 : 2 * static_cast<size_t>(a.D));
    const size_t row3 = 3 * static_cast<size_t>(a.D);
    uint32_t issued = 0;
    bool ok = true;
    for (long long i = s_begin; i < s_end && ok;) {
      const int tile = static_cast<int>(i / KB);
      const int kb0 = static_cast<int>(i - static_cast<long long>(tile) * KB);
      const long long e = min(s_end, static_cast<long long>(tile + 1) * KB);
      const int kb1 = kb0 + static_cast<int>(e - i);
      // MODE 0: the tile's 128 rows are positions 128 * tile + r (fixed over the segment); this lane
      // copies rows rg + 4m. MODE 1: the k-block's 64 rows are items 64 * kb + r; this lane copies
      // items rg + 4m, and the next k-block's ids are loaded before this one's wait so that their
      // latency hides behind it. Row offsets (elements) stay in registers.
      constexpr int NROW = MODE == 0 ? TC_BM / 4 : TC_BK / 4;
      uint32_t rowoff[NROW];
      int ids_nxt[NROW];
      auto load_ids = [&](int kb, int (&o)[NROW]) {
#pragma unroll
        for (int m = 0; m < NROW; ++m) {
          const int item = kb * TC_BK + rg + 4 * m;
          o[m] = item < a.K ? a.ch_list[item] : 0;
        }
      };
      auto set_rows = [&](const int (&ids)[NROW]) {
#pragma unroll
        for (int m = 0; m < NROW; ++m) rowoff[m] = static_cast<uint32_t>(guard_ch(ids[m], a.N, a.err)) * row3;
      };
      if (MODE == 0) {
        int ids[NROW];
#pragma unroll
        for (int m = 0; m < NROW; ++m) {
          const int p = tile * TC_BM + rg + 4 * m;
          ids[m] = p < a.rows ? a.rc[p] : 0;
        }
        set_rows(ids);
      } else {
        load_ids(kb0, ids_nxt);
      }
      for (int kb = kb0; kb < kb1; ++kb) {
        if (MODE == 1) {
          set_rows(ids_nxt);
          if (kb + 1 < kb1) load_ids(kb + 1, ids_nxt);
        }
        const int s = issued % STAGES;
        const uint32_t ph = (issued / STAGES) & 1u;
        bool got = true;
        if (lane == 0) {
          got = mbar_wait_bounded(&ctl->empty[s], ph ^ 1u, a.wait_ns, abort_flag);
          if (!got) fail();
          else mbar_arrive_expect_tx(&ctl->full[s], tx_bytes);
        }
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
        uint8_t* sb = smem + s * STAGE_BYTES + Cfg::A_BYTES;
        if (MODE == 0) {
          const int d0 = kb * TC_BK + 8 * cq;
          const uint32_t nbytes = d0 < a.D ? 16u : 0u;  // D is a multiple of 8: chunks are all in or all out
          const uint16_t* base = Wbase + (nbytes ? d0 : 0);
#pragma unroll
          for (int m = 0; m < NROW; ++m) {
            const int r = rg + 4 * m;
            const uint32_t dst = sa + r * 128 + ((cq ^ (r & 7)) << 4);
            cp_async16(dst, base + rowoff[m], nbytes);
            cp_async16(dst + TC_BM * 128, base + rowoff[m] + a.D, nbytes);
          }
        } else {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int d0 = tile * TC_BM + 64 * h + 8 * cq;
            const uint32_t nbytes = d0 < a.D ? 16u : 0u;
            const uint16_t* base = Wbase + (nbytes ? d0 : 0);
#pragma unroll
            for (int m = 0; m < NROW; ++m) {
              const int r = rg + 4 * m;
              cp_async16(sa + h * (TC_BK * 128) + r * 128 + ((cq ^ (r & 7)) << 4), base + rowoff[m], nbytes);
            }
          }
        }
        cp_async_commit();
        if (issued >= static_cast<uint32_t>(LAG)) {
          cp_async_wait<LAG>();
          fence_proxy_async();
          mbar_arrive(&ctl->full[(issued - LAG) % STAGES]);
        }
        if (lane == 0) {
          tma_load_2d(sb, &mapB, &ctl->full[s], kb * TC_BK, 0);
          if (MODE == 1) tma_load_2d(sb + NP * 128, &mapB2, &ctl->full[s], kb * TC_BK, 0);  // z lo plane
        }
        ++issued;
      }
      i = e;
    }
    // the last stages' arrivals, and every copy this warp started must land before the CTA can exit
    cp_async_wait<0>();
    fence_proxy_async();
    if (ok)
      for (uint32_t u = issued > static_cast<uint32_t>(LAG) ? issued - LAG : 0; u < issued; ++u)
        mbar_arrive(&ctl->full[u % STAGES]);
    if (lane == 0) {
      const uint32_t lo = issued > static_cast<uint32_t>(STAGES) ? issued - STAGES : 0;
      for (uint32_t u = lo; u < issued; ++u) {
        volatile int never = 0;
        if (!mbar_wait_bounded(&ctl->full[u % STAGES], (u / STAGES) & 1u, TC_DRAIN_NS, &never)) fail();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer (one thread)
      const uint32_t idesc = idesc_bf16_f32(TC_BM, MODE == 0 ? NP : 2 * NP, false, MODE == 1);
      uint32_t consumed = 0;
      int it = 0;
      bool ok = true;
      for (long long i = s_begin; i < s_end && ok; ++it) {
        const int tile = static_cast<int>(i / KB);
        const int kb0 = static_cast<int>(i - static_cast<long long>(tile) * KB);
        const long long e = min(s_end, static_cast<long long>(tile + 1) * KB);
        const int kb1 = kb0 + static_cast<int>(e - i);
        const int buf = it & 1;
        if (!mbar_wait_bounded(&ctl->tempty[buf], ((it >> 1) & 1) ^ 1, a.wait_ns, abort_flag)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf) * HALF_COLS;
        for (int kb = kb0; kb < kb1; ++kb) {
          const int s = consumed % STAGES;
          const uint32_t ph = (consumed / STAGES) & 1u;
          if (!mbar_wait_bounded(&ctl->full[s], ph, a.wait_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
          for (int k = 0; k < TC_BK / 16; ++k) {
            const uint32_t acc = (kb > kb0 || k > 0) ? 1u : 0u;
            const uint64_t bdesc = smem_desc_sw128(sb + 32u * k, 16u, 1024u);
            if (MODE == 0) {
              umma_f16(d_tmem, smem_desc_sw128(sa + 32u * k, 16u, 1024u), bdesc, idesc, acc);
              umma_f16(d_tmem + static_cast<uint32_t>(NP), smem_desc_sw128(sa + TC_BM * 128 + 32u * k, 16u, 1024u),
                       bdesc, idesc, acc);
            } else {
              umma_f16(d_tmem, smem_desc_sw128(sa + 2048u * k, TC_BK * 128, 1024u), bdesc, idesc, acc);
            }
          }
          umma_commit(&ctl->empty[s]);
          ++consumed;
        }
        if (!ok) break;
        umma_commit(&ctl->tfull[buf]);
        i = e;
      }
      // all MMAs issued by this thread must finish before TMEM is freed
      umma_commit(&ctl->drain);
      volatile int never = 0;
      if (!mbar_wait_bounded(&ctl->drain, 0, TC_DRAIN_NS, &never)) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter of this warp
    const int r = 32 * q + lane;
    const int et = threadIdx.x - 64;  // 0..127
    int it = 0, seg = 0;
    for (long long i = s_begin; i < s_end; ++it, ++seg) {
      const int tile = static_cast<int>(i / KB);
      const int kb0 = static_cast<int>(i - static_cast<long long>(tile) * KB);
      const long long e = min(s_end, static_cast<long long>(tile + 1) * KB);
      const int kb1 = kb0 + static_cast<int>(e - i);
      const int buf = it & 1;
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

      bool finish = kb0 == 0 && kb1 == KB;
      if (!finish) {
        // partial tile: publish, then the last contributor adds all partials in CTA order
        const int slot = 2 * blockIdx.x + (seg == 0 ? 0 : 1);
        float* w = a.ws + static_cast<size_t>(slot) * TC_WS_COLS * TC_BM;
#pragma unroll
        for (int c = 0; c < NP; ++c) {
          w[c * TC_BM + r] = gv[c];
          w[(NP + c) * TC_BM + r] = uv[c];
        }
        epi_bar();
        if (et == 0) {
          const long long t0 = static_cast<long long>(tile) * KB;
          const int c_lo = sk_owner(t0, T, G), c_hi = sk_owner(t0 + KB - 1, T, G);
          unsigned* cnt = a.tile_cnt + tile;
          const unsigned old = atom_add_acq_rel_tc(cnt, 1u);
          const int last = old + 1 == static_cast<unsigned>(c_hi - c_lo + 1);
          if (last) atomicExch(cnt, 0u);  // every contributor has arrived: ready for the next launch
          ctl->last = last;
        }
        epi_bar();
        finish = ctl->last != 0;
        if (finish) {
          const long long t0 = static_cast<long long>(tile) * KB;
          const int c_lo = sk_owner(t0, T, G), c_hi = sk_owner(t0 + KB - 1, T, G);
#pragma unroll
          for (int c = 0; c < NP; ++c) {
            gv[c] = 0.f;
            uv[c] = 0.f;
          }
          for (int cc = c_lo; cc <= c_hi; ++cc) {
            const int sl = 2 * cc + (sk_start(cc, T, G) >= t0 ? 0 : 1);
            const float* wp = a.ws + static_cast<size_t>(sl) * TC_WS_COLS * TC_BM + r;
            float lg[NP], lu[NP];
#pragma unroll
            for (int c = 0; c < NP; ++c) {
              lg[c] = __ldcg(wp + c * TC_BM);
              lu[c] = __ldcg(wp + (NP + c) * TC_BM);
            }
#pragma unroll
            for (int c = 0; c < NP; ++c) {
              gv[c] += lg[c];
              uv[c] += lu[c];
            }
          }
        }
      }
      if (finish) {
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
            if (p < a.nC) a.scores[p] = m * a.n2[guard_ch(a.rc[p], a.N, a.err)];
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
      i = e;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ launchers
template <int MODE, int NP>
static cudaError_t launch_tc_np(const CUtensorMap& b, const CUtensorMap& b2, const DecodeTcArgs& args, int grid,
                                cudaStream_t st) {
  constexpr size_t smem = tc_smem_bytes<MODE>();
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(k_decode_tc<MODE, NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(TC_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_decode_tc<MODE, NP>, b, b2, args);
}

template <int MODE>
static cudaError_t launch_tc(const CUtensorMap& b, const CUtensorMap& b2, const DecodeTcArgs& args, int num_sms,
                             cudaStream_t st) {
  const long long T = static_cast<long long>((args.rows + TC_BM - 1) / TC_BM) * ((args.K + TC_BK - 1) / TC_BK);
  if (T <= 0) return cudaSuccess;
  const int grid = static_cast<int>(T < num_sms ? T : num_sms);
  switch (args.NP) {
    case 16: return launch_tc_np<MODE, 16>(b, b2, args, grid, st);
    case 32: return launch_tc_np<MODE, 32>(b, b2, args, grid, st);
    case 48: return launch_tc_np<MODE, 48>(b, b2, args, grid, st);
    case 64: return launch_tc_np<MODE, 64>(b, b2, args, grid, st);
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

size_t decode_tc_workspace_floats(int num_sms) { return static_cast<size_t>(2) * num_sms * TC_WS_COLS * TC_BM; }

}  // namespace pop
