// One decode step of the POP FFN for B = 1 in a single persistent kernel.
//
// What it computes ("POP: Online Structural Pruning..." notes, Key design 2; "Batch-wise adaptive
// pruning", abstract for the periodic memory):
//   z_i = SiLU(Wg[i,:] x) * (W1[i,:] x) for i in R u C,
//   a_i = |z_i| * ||W2[:,i]|| for i in C, S = the k largest (ties to the lower index),
//   y   = sum over i in R u S of z_i W2[:,i].
//
// How: one CTA per SM, all co-resident (cooperative launch). A producer warp streams each
// channel's packed row (gate | up | down, contiguous) from HBM into a shared-memory ring with
// bulk asynchronous copies (cp.async.bulk + mbarrier transaction counts); 8 consumer warps
// compute from the ring. Every CTA first scores its share of C (16 KB per channel: gate + up),
// then streams its share of R with the down projection fused (24 KB per channel: z is used as
// soon as it is known, since R is always kept). CTA 0, which gets fewer R channels, runs the
// top-k once every CTA has published its candidate scores; that overlaps the other CTAs' R
// stream. Then every CTA projects its share of S (8 KB per channel), writes its partial y, and
// after a grid barrier reduces one slice of y over all partials in a fixed order
// (deterministic).
//
// Inter-CTA waits use counters in global memory (C-phase arrivals, selection generation, grid
// barrier) that are left ready for the next launch. Every wait is bounded; a wait that runs out
// sets DEVERR_TIMEOUT_DECODE. Consumer threads never skip a named barrier, whatever a wait
// returned, so a time-out cannot turn into a hang.
#include "pop_device.cuh"
#include "pop_internal.h"
#include "pop_radix.cuh"

namespace pop {

namespace {
constexpr int FZ_CONS = 256;  // consumer threads (8 warps)
constexpr int FZ_WARPS = FZ_CONS / 32;
constexpr int FZ_THREADS = 32 + FZ_CONS;
constexpr int FZ_MAX_STAGES = 8;
constexpr int FZ_MIN_STAGES = 2;
constexpr size_t FZ_SMEM_CAP = 232448;  // opt-in shared memory per block on sm_103
constexpr uint64_t FZ_DRAIN_NS = 1000000000ull;

struct FusedCtl {
  uint64_t full[FZ_MAX_STAGES];
  uint64_t empty[FZ_MAX_STAGES];
  float red[2][FZ_WARPS][2];
  float yred[FZ_CONS];
  unsigned sel_gen0;
  unsigned bar_gen0;
  int abort_flag;
  int bcast_ok;
  RadixScratch<FZ_CONS> sc;
};

struct ConsumerSync {
  __device__ void operator()() const { asm volatile("bar.sync 1, 256;" ::: "memory"); }
};

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Spins until pred() holds or `limit_ns` passes. Returns pred's last value.
template <class Pred>
__device__ bool spin_bounded(Pred pred, uint64_t limit_ns) {
  if (pred()) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    __nanosleep(64);
    if (pred()) return true;
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
}

__device__ __forceinline__ float silu_fz(float g) { return g / (1.0f + expf(-g)); }

__host__ __device__ size_t ctl_offset(int D, int nC, int stages) {
  const size_t ring = static_cast<size_t>(stages) * 6 * D;
  const size_t keys = (static_cast<size_t>(nC > 0 ? nC : 1) * 4 + 127) / 128 * 128;
  return ring + keys;
}
}  // namespace

int decode_fused_stages(int D, int nC) {
  if (nC > FZ_MAX_C) return 0;
  const size_t fixed = (static_cast<size_t>(nC > 0 ? nC : 1) * 4 + 127) / 128 * 128 + sizeof(FusedCtl) + 128;
  if (fixed >= FZ_SMEM_CAP) return 0;
  int st = static_cast<int>((FZ_SMEM_CAP - fixed) / (6ull * D));
  if (st > FZ_MAX_STAGES) st = FZ_MAX_STAGES;
  return st >= FZ_MIN_STAGES ? st : 0;
}

template <int CPT>
__global__ void __launch_bounds__(FZ_THREADS, 1) k_decode_fused_b1(const __grid_constant__ FusedDecodeArgs a) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int D = a.D, nC = a.nC, nR = a.nR, k = a.k;
  const int stages = a.stages;
  const uint32_t stage_bytes = 6u * static_cast<uint32_t>(D);
  uint8_t* ring = smem;
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem + static_cast<size_t>(stages) * stage_bytes);
  FusedCtl* ctl = reinterpret_cast<FusedCtl*>(smem + ctl_offset(D, nC, stages));
  const int G = gridDim.x, cta = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t row3 = 3 * static_cast<size_t>(D);

  // balanced item ranges; CTA 0 takes r_skew fewer R channels (it also runs the top-k)
  const int c0 = static_cast<int>(static_cast<long long>(cta) * nC / G);
  const int c1 = static_cast<int>(static_cast<long long>(cta + 1) * nC / G);
  int share0 = G > 1 ? nR / G - a.r_skew : nR;
  if (share0 < 0) share0 = 0;
  auto r_lo = [&](int j) {
    if (j <= 0) return 0;
    if (j >= G) return nR;
    return share0 + static_cast<int>(static_cast<long long>(j - 1) * (nR - share0) / (G - 1));
  };
  const int r0 = r_lo(cta), r1 = r_lo(cta + 1);
  const int s0 = static_cast<int>(static_cast<long long>(cta) * k / G);
  const int s1 = static_cast<int>(static_cast<long long>(cta + 1) * k / G);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], FZ_WARPS);
    }
    ctl->sel_gen0 = ld_acquire(a.sync + 1);
    ctl->bar_gen0 = ld_acquire(a.sync + 3);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  volatile int* abort_flag = &ctl->abort_flag;
  auto fail = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      atomicOr(a.err, DEVERR_TIMEOUT_DECODE);
    }
  };

  if (warp == 0) {
    // ================================================================ producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      auto issue = [&](const uint16_t* src, uint32_t bytes) {
        const int s = it % stages;
        const uint32_t ph = (it / stages) & 1u;
        if (!mbar_wait_bounded(&ctl->empty[s], ph ^ 1u, a.wait_ns, abort_flag)) return false;
        mbar_arrive_expect_tx(&ctl->full[s], bytes);
        bulk_load(ring + static_cast<size_t>(s) * stage_bytes, src, bytes, &ctl->full[s]);
        ++it;
        return true;
      };
      for (int p = c0; p < c1 && ok; ++p) {
        const int ch = a.rc[p];
        ok = issue(a.Wp + static_cast<size_t>(static_cast<unsigned>(ch) < static_cast<unsigned>(a.N) ? ch : 0) * row3,
                   4u * D);
      }
      for (int p = r0; p < r1 && ok; ++p) {
        const int ch = a.rc[nC + p];
        ok = issue(a.Wp + static_cast<size_t>(static_cast<unsigned>(ch) < static_cast<unsigned>(a.N) ? ch : 0) * row3,
                   6u * D);
      }
      if (ok && s1 > s0) {
        const unsigned g0 = ctl->sel_gen0;
        ok = spin_bounded([&]() { return ld_acquire(a.sync + 1) != g0 || *abort_flag; }, a.wait_ns) && !*abort_flag;
        for (int j = s0; j < s1 && ok; ++j) {
          int pos = __ldcg(a.S + j);
          if (static_cast<unsigned>(pos) >= static_cast<unsigned>(nC)) pos = 0;
          int ch = a.rc[pos];
          if (static_cast<unsigned>(ch) >= static_cast<unsigned>(a.N)) ch = 0;
          ok = issue(a.Wp + static_cast<size_t>(ch) * row3 + 2 * static_cast<size_t>(D), 2u * D);
        }
      }
      if (!ok) fail();
      // every copy started here must land before the CTA may exit
      const uint32_t lo = it > static_cast<uint32_t>(stages) ? it - stages : 0;
      for (uint32_t u = lo; u < it; ++u) {
        volatile int never = 0;
        if (!mbar_wait_bounded(&ctl->full[u % stages], (u / stages) & 1u, FZ_DRAIN_NS, &never)) fail();
      }
    }
    return;
  }

  // ================================================================== consumers
  const int ct = threadIdx.x - 32;
  const int cw = ct >> 5;
  const ConsumerSync csync;
  const int nch = D >> 3;
  float xr[CPT][8], yacc[CPT][8];
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = ct + FZ_CONS * j;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (c < nch) v = *reinterpret_cast<const uint4*>(a.x + 8 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      xr[j][2 * q] = bf16lo(w[q]);
      xr[j][2 * q + 1] = bf16hi(w[q]);
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) yacc[j][e] = 0.f;
  }

  uint32_t it = 0;
  int par = 0;
  bool ok = true;
  auto wait_full = [&]() {
    const int s = it % stages;
    if (!mbar_wait_bounded(&ctl->full[s], (it / stages) & 1u, a.wait_ns, abort_flag)) {
      fail();
      ok = false;
    }
    return ring + static_cast<size_t>(s) * stage_bytes;
  };
  auto release = [&]() {
    __syncwarp();
    if (lane == 0) mbar_arrive(&ctl->empty[it % stages]);
    ++it;
  };
  // gate/up dot products of the staged row with x; every consumer thread returns the same z
  auto gateup = [&](const uint8_t* st) {
    float g0 = 0.f, g1 = 0.f, u0 = 0.f, u1 = 0.f;
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = ct + FZ_CONS * j;
      if (c < nch) {
        const uint4 wg = *reinterpret_cast<const uint4*>(st + 16 * c);
        const uint4 wu = *reinterpret_cast<const uint4*>(st + 2 * D + 16 * c);
        const uint32_t gw[4] = {wg.x, wg.y, wg.z, wg.w}, uw[4] = {wu.x, wu.y, wu.z, wu.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          g0 = fmaf(bf16lo(gw[q]), xr[j][2 * q], g0);
          g1 = fmaf(bf16hi(gw[q]), xr[j][2 * q + 1], g1);
          u0 = fmaf(bf16lo(uw[q]), xr[j][2 * q], u0);
          u1 = fmaf(bf16hi(uw[q]), xr[j][2 * q + 1], u1);
        }
      }
    }
    float g = g0 + g1, u = u0 + u1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      u += __shfl_xor_sync(0xffffffffu, u, o);
    }
    if (lane == 0) {
      ctl->red[par][cw][0] = g;
      ctl->red[par][cw][1] = u;
    }
    csync();
    float gs = 0.f, us = 0.f;
#pragma unroll
    for (int w = 0; w < FZ_WARPS; ++w) {
      gs += ctl->red[par][w][0];
      us += ctl->red[par][w][1];
    }
    par ^= 1;
    return silu_fz(gs) * us;
  };
  auto down = [&](const uint8_t* col, float z) {
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = ct + FZ_CONS * j;
      if (c < nch) {
        const uint4 w = *reinterpret_cast<const uint4*>(col + 16 * c);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          yacc[j][2 * q] = fmaf(bf16lo(ww[q]), z, yacc[j][2 * q]);
          yacc[j][2 * q + 1] = fmaf(bf16hi(ww[q]), z, yacc[j][2 * q + 1]);
        }
      }
    }
  };
  // a wait on another CTA done by one thread, its result shared with all consumers
  auto shared_wait = [&](auto pred) {
    if (ct == 0) {
      ctl->bcast_ok = spin_bounded(pred, a.wait_ns) ? 1 : 0;
      __threadfence();
    }
    csync();
    const bool r = ctl->bcast_ok != 0;
    csync();
    return r;
  };

  // ---- phase 1: candidates (gate/up, score)
  for (int p = c0; p < c1; ++p) {
    const uint8_t* st = wait_full();
    const float z = gateup(st);
    if (ct == 0) {
      int ch = a.rc[p];
      if (static_cast<unsigned>(ch) >= static_cast<unsigned>(a.N)) ch = 0;
      a.zC[p] = z;
      a.scores[p] = fabsf(z) * a.n2[ch];
    }
    release();
  }
  if (ct == 0) {
    __threadfence();
    atomicAdd(a.sync + 0, 1u);
  }

  // ---- CTA 0: periodic memory and top-k over all candidates
  if (cta == 0) {
    const bool all_in = shared_wait([&]() { return ld_acquire(a.sync + 0) >= static_cast<unsigned>(G); });
    if (!all_in) {
      if (ct == 0) fail();
      ok = false;
    } else {
      if (ct == 0) atomicExch(a.sync + 0, 0u);  // every CTA has arrived: ready for the next launch
      const int t = *a.step;
      const bool sel_ok = select_step<FZ_CONS>(
          ct, [&](int i) { return __ldcg(a.scores + i); }, a.memory, nC, k, a.period, (t % a.period) == 0, keys,
          a.S, ctl->sc, csync);
      csync();
      if (ct == 0) {
        if (!sel_ok) atomicOr(a.err, DEVERR_TOPK);
        *a.step = t + 1;
        __threadfence();
        atomicAdd(a.sync + 1, 1u);
      }
    }
  }

  // ---- phase 2: retained channels (gate/up and down together)
  for (int p = r0; p < r1; ++p) {
    const uint8_t* st = wait_full();
    const float z = gateup(st);
    down(st + 4 * D, z);
    release();
  }

  // ---- phase 3: selected candidates (down only)
  if (s1 > s0) {
    const unsigned g0 = ctl->sel_gen0;
    if (!shared_wait([&]() { return ld_acquire(a.sync + 1) != g0; })) {
      if (ct == 0) fail();
      ok = false;
    }
    __threadfence();
    for (int j = s0; j < s1; ++j) {
      const uint8_t* st = wait_full();
      int pos = __ldcg(a.S + j);
      if (static_cast<unsigned>(pos) >= static_cast<unsigned>(nC)) pos = 0;
      down(st, __ldcg(a.zC + pos));
      release();
    }
  }

  // ---- partial y, grid barrier, ordered reduction of one slice of y
  float* part = a.ypart + static_cast<size_t>(cta) * D;
#pragma unroll
  for (int j = 0; j < CPT; ++j) {
    const int c = ct + FZ_CONS * j;
    if (c < nch) {
      reinterpret_cast<float4*>(part + 8 * c)[0] = make_float4(yacc[j][0], yacc[j][1], yacc[j][2], yacc[j][3]);
      reinterpret_cast<float4*>(part + 8 * c)[1] = make_float4(yacc[j][4], yacc[j][5], yacc[j][6], yacc[j][7]);
    }
  }
  csync();
  if (ct == 0) {
    const unsigned bg0 = ctl->bar_gen0;
    __threadfence();
    const unsigned old = atomicAdd(a.sync + 2, 1u);
    bool passed = true;
    if (old == static_cast<unsigned>(G) - 1u) {
      atomicExch(a.sync + 2, 0u);  // ready for the next launch
      __threadfence();
      atomicAdd(a.sync + 3, 1u);
    } else {
      passed = spin_bounded([&]() { return ld_acquire(a.sync + 3) != bg0; }, a.wait_ns);
    }
    __threadfence();
    ctl->bcast_ok = passed ? 1 : 0;
    if (!passed) fail();
  }
  csync();
  const int d0 = static_cast<int>(static_cast<long long>(cta) * D / G);
  const int d1 = static_cast<int>(static_cast<long long>(cta + 1) * D / G);
  for (int base = d0; base < d1; base += FZ_CONS) {
    const int L = min(FZ_CONS, d1 - base);
    int gg = FZ_CONS / L;
    if (gg > G) gg = G;
    const int e = ct % L, grp = ct / L;
    if (grp < gg) {
      const int g0 = static_cast<int>(static_cast<long long>(grp) * G / gg);
      const int g1 = static_cast<int>(static_cast<long long>(grp + 1) * G / gg);
      float sum = 0.f;
      for (int g = g0; g < g1; ++g) sum += __ldcg(a.ypart + static_cast<size_t>(g) * D + base + e);
      ctl->yred[grp * L + e] = sum;
    }
    csync();
    if (ct < L) {
      float t = 0.f;
      for (int q = 0; q < gg; ++q) t += ctl->yred[q * L + ct];
      if (a.out_f32)
        static_cast<float*>(a.y)[base + ct] = t;
      else
        static_cast<__nv_bfloat16*>(a.y)[base + ct] = __float2bfloat16_rn(t);
    }
    csync();
  }
  (void)ok;
}

// ------------------------------------------------------------------ launcher
template <int CPT>
static cudaError_t launch_fused_cpt(const FusedDecodeArgs& a, int grid, size_t smem, cudaStream_t st) {
  static int configured = 0;  // largest dynamic smem set so far for this instance
  if (static_cast<int>(smem) > configured) {
    cudaError_t e = cudaFuncSetAttribute(k_decode_fused_b1<CPT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = static_cast<int>(smem);
  }
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_decode_fused_b1<CPT>, FZ_THREADS, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  void* args[] = {const_cast<FusedDecodeArgs*>(&a)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(k_decode_fused_b1<CPT>), dim3(grid), dim3(FZ_THREADS),
                                     args, smem, st);
}

size_t decode_fused_smem(int D, int nC, int stages) { return ctl_offset(D, nC, stages) + sizeof(FusedCtl); }

cudaError_t launch_decode_fused_b1(const FusedDecodeArgs& a, int num_sms, cudaStream_t st) {
  const size_t smem = decode_fused_smem(a.D, a.nC, a.stages);
  const int cpt = (a.D / 8 + FZ_CONS - 1) / FZ_CONS;
  if (cpt <= 1) return launch_fused_cpt<1>(a, num_sms, smem, st);
  if (cpt <= 2) return launch_fused_cpt<2>(a, num_sms, smem, st);
  if (cpt <= 4) return launch_fused_cpt<4>(a, num_sms, smem, st);
  return launch_fused_cpt<8>(a, num_sms, smem, st);
}

}  // namespace pop
