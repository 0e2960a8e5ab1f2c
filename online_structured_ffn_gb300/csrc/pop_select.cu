// Selection kernels of the POP FFN: the prefill R/C/P split and the per-step candidate top-k.
//
// "POP: Online Structural Pruning..." (papernotes.org notes), Key design 1: channels at or above
// q_{r+delta} form R, at or below q_{r-delta} form P, the rest C. Key design 2: candidates are
// sorted by their step score and the top ones fill |R| + k = (1 - r) * D_FF survivors.
// "Batch-wise adaptive pruning" (bittide page), abstract: top-k every update period from an
// activation memory that accumulates importance between updates.
//
// Both selections order elements by (score ascending, index descending), so that among equal
// scores the lower index counts as the more important. With that total order every cut-off is
// one order statistic, found by a block-wide radix select (8-bit digits, warp-aggregated
// shared-memory histograms); a block-wide ordered compaction then writes ascending index lists.
#include "pop_device.cuh"
#include "pop_internal.h"

namespace pop {

constexpr int SEL_THREADS = 1024;
constexpr int SEL_WARPS = SEL_THREADS / 32;

struct SelScratch {
  uint32_t hist[256];
  uint32_t bcast[4];
  uint32_t warp_tot[SEL_WARPS][3];
};

// Ascending rank `t` among the participating elements of [0, n), looking only at the bits from
// `top_shift + 7` down to 0 (top_shift = 24 for 32-bit keys, 8 for 16-bit keys).
// `value(i)` gives element i's key, `part(i)` whether element i takes part.
// Returns the selected value, the number of participants below it and the number equal to it.
template <class Val, class Part>
__device__ void radix_select(int n, uint32_t t, int top_shift, Val value, Part part, SelScratch& sc,
                             uint32_t& v_out, uint32_t& lt_out, uint32_t& eq_out) {
  const int lane = threadIdx.x & 31;
  uint32_t prefix = 0, pmask = 0, rank = t, lt = 0, eq = 0;
  for (int shift = top_shift; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += SEL_THREADS) sc.hist[i] = 0;
    if (threadIdx.x == 0) {
      sc.bcast[0] = 0;
      sc.bcast[1] = 0;
      sc.bcast[2] = 0;
    }
    __syncthreads();
    for (int base = threadIdx.x - lane; base < n; base += SEL_THREADS) {
      const int i = base + lane;
      uint32_t kv = 0;
      bool p = false;
      if (i < n && part(i)) {
        kv = value(i);
        p = (kv & pmask) == prefix;
      }
      const unsigned m = __ballot_sync(0xffffffffu, p);
      if (p) {
        const uint32_t digit = (kv >> shift) & 0xffu;
        const unsigned peers = __match_any_sync(m, digit);
        if (lane == __ffs(peers) - 1) atomicAdd(&sc.hist[digit], static_cast<uint32_t>(__popc(peers)));
      }
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      uint32_t c[8], s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = sc.hist[lane * 8 + j];
        s += c[j];
      }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - s;
      if (rank >= excl && rank < incl) {
        uint32_t acc = excl;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (rank >= acc && rank < acc + c[j]) {
            sc.bcast[0] = static_cast<uint32_t>(lane * 8 + j);
            sc.bcast[1] = acc;
            sc.bcast[2] = c[j];
          }
          acc += c[j];
        }
      }
    }
    __syncthreads();
    const uint32_t digit = sc.bcast[0];
    prefix |= digit << shift;
    pmask |= 0xffu << shift;
    rank -= sc.bcast[1];
    lt += sc.bcast[1];
    eq = sc.bcast[2];
    __syncthreads();
  }
  v_out = prefix;
  lt_out = lt;
  eq_out = eq;
}

// The element at ascending position t of the order (key ascending, index descending):
// returns its key v and index j.
__device__ void order_statistic(const uint32_t* keys, int n, uint32_t t, SelScratch& sc, uint32_t& v, int& j) {
  uint32_t lt, eq;
  radix_select(
      n, t, 24, [&](int i) { return keys[i]; }, [](int) { return true; }, sc, v, lt, eq);
  // among the eq elements equal to v (in descending index order) take offset t - lt, which is the
  // ascending-index rank eq - 1 - (t - lt).
  const uint32_t want = eq - 1u - (t - lt);
  const uint32_t vv = v;
  const int top = n > 65536 ? 24 : (n > 256 ? 8 : 0);
  uint32_t jv, jlt, jeq;
  radix_select(
      n, want, top, [](int i) { return static_cast<uint32_t>(i); }, [&](int i) { return keys[i] == vv; }, sc, jv,
      jlt, jeq);
  j = static_cast<int>(jv);
}

// Block-wide exclusive scan of three counters per thread (thread order). Returns the totals.
__device__ void block_scan3(const uint32_t (&c)[3], uint32_t (&excl)[3], uint32_t (&tot)[3], SelScratch& sc) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl[3];
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    incl[a] = c[a];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, incl[a], o);
      if (lane >= o) incl[a] += y;
    }
  }
  if (lane == 31)
#pragma unroll
    for (int a = 0; a < 3; ++a) sc.warp_tot[warp][a] = incl[a];
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      const uint32_t s = sc.warp_tot[lane][a];
      uint32_t in2 = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, in2, o);
        if (lane >= o) in2 += y;
      }
      sc.warp_tot[lane][a] = in2 - s;  // exclusive warp offsets
      if (lane == 31) sc.bcast[a] = in2;
    }
  }
  __syncthreads();
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    excl[a] = sc.warp_tot[warp][a] + incl[a] - c[a];
    tot[a] = sc.bcast[a];
  }
  __syncthreads();
}

// ------------------------------------------------------------------ prefill partition
__global__ void __launch_bounds__(SEL_THREADS, 1)
    k_partition(const float* __restrict__ sumsq, const float* __restrict__ n2, float* __restrict__ I, int N,
                int n_P, int n_R, int* __restrict__ rc, int* __restrict__ Plist, int* __restrict__ step,
                float* __restrict__ memory, unsigned* __restrict__ err) {
  extern __shared__ uint32_t keys[];
  __shared__ SelScratch sc;
  for (int i = threadIdx.x; i < N; i += SEL_THREADS) {
    float v;
    if (sumsq != nullptr) {
      v = n2[i] * sqrtf(sumsq[i]);
      I[i] = v;
    } else {
      v = I[i];
    }
    keys[i] = float_key(v);
  }
  __syncthreads();
  uint32_t vP = 0, vR = 0;
  int jP = -1, jR = N;
  if (n_P > 0) order_statistic(keys, N, static_cast<uint32_t>(n_P - 1), sc, vP, jP);
  if (n_R > 0) order_statistic(keys, N, static_cast<uint32_t>(N - n_R), sc, vR, jR);

  // class: 0 = P, 1 = C, 2 = R; thread t covers the contiguous index range [t*per, (t+1)*per)
  const int per = (N + SEL_THREADS - 1) / SEL_THREADS;
  const int i0 = min(N, static_cast<int>(threadIdx.x) * per);
  const int i1 = min(N, i0 + per);
  auto cls = [&](int i) {
    const uint32_t kv = keys[i];
    if (n_P > 0 && (kv < vP || (kv == vP && i >= jP))) return 0;
    if (n_R > 0 && (kv > vR || (kv == vR && i <= jR))) return 2;
    return 1;
  };
  uint32_t c[3] = {0, 0, 0};
  for (int i = i0; i < i1; ++i) c[cls(i)]++;
  uint32_t off[3], tot[3];
  block_scan3(c, off, tot, sc);
  const int nC = N - n_P - n_R;
  const bool ok = tot[0] == static_cast<uint32_t>(n_P) && tot[2] == static_cast<uint32_t>(n_R) &&
                  tot[1] == static_cast<uint32_t>(nC);
  if (!ok) {
    if (threadIdx.x == 0) atomicOr(err, DEVERR_PARTITION);
    return;
  }
  for (int i = i0; i < i1; ++i) {
    const int k = cls(i);
    if (k == 0)
      Plist[off[0]++] = i;
    else if (k == 1)
      rc[off[1]++] = i;
    else
      rc[nC + off[2]++] = i;
  }
  for (int i = threadIdx.x; i < nC; i += SEL_THREADS) memory[i] = 0.f;
  if (threadIdx.x == 0) *step = 0;
}

// ------------------------------------------------------------------ per-step candidate selection
__global__ void __launch_bounds__(SEL_THREADS, 1)
    k_select(const float* __restrict__ scores, float* __restrict__ memory, int nC, int k, int period,
             int* __restrict__ step, int* __restrict__ S, unsigned* __restrict__ err) {
  extern __shared__ uint32_t keys[];
  __shared__ SelScratch sc;
  const int t = *step;
  const bool update = (t % period) == 0;
  for (int i = threadIdx.x; i < nC; i += SEL_THREADS) {
    float v = scores[i];
    if (period > 1) {
      v += memory[i];
      memory[i] = update ? 0.f : v;
    }
    keys[i] = float_key(v);
  }
  __syncthreads();
  if (update && k > 0) {
    uint32_t vS = 0;
    int jS = nC;
    if (k < nC) order_statistic(keys, nC, static_cast<uint32_t>(nC - k), sc, vS, jS);
    const int per = (nC + SEL_THREADS - 1) / SEL_THREADS;
    const int i0 = min(nC, static_cast<int>(threadIdx.x) * per);
    const int i1 = min(nC, i0 + per);
    auto sel = [&](int i) {
      if (k >= nC) return true;
      const uint32_t kv = keys[i];
      return kv > vS || (kv == vS && i <= jS);
    };
    uint32_t c[3] = {0, 0, 0};
    for (int i = i0; i < i1; ++i) c[0] += sel(i) ? 1u : 0u;
    uint32_t off[3], tot[3];
    block_scan3(c, off, tot, sc);
    if (tot[0] != static_cast<uint32_t>(k)) {
      if (threadIdx.x == 0) atomicOr(err, DEVERR_TOPK);
    } else {
      for (int i = i0; i < i1; ++i)
        if (sel(i)) S[off[0]++] = i;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) *step = t + 1;
}

// ------------------------------------------------------------------ channel sums of squares
__global__ void k_fold_sumsq(const float* __restrict__ part, int rows, int ld, int N, float* __restrict__ sumsq,
                             int accumulate) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= N) return;
  float s = accumulate ? sumsq[i] : 0.f;
  for (int p = 0; p < rows; ++p) s += part[static_cast<size_t>(p) * ld + i];
  sumsq[i] = s;
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_partition(const float* sumsq, const float* n2, float* I, int N, int n_P, int n_R, int* rc,
                             int* P, int* step, float* memory, unsigned* err, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(N) * sizeof(uint32_t);
  cudaError_t e = cudaFuncSetAttribute(k_partition, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  k_partition<<<1, SEL_THREADS, smem, st>>>(sumsq, n2, I, N, n_P, n_R, rc, P, step, memory, err);
  return cudaGetLastError();
}

cudaError_t launch_select(const float* scores, float* memory, int nC, int k, int period, int* step, int* S,
                          unsigned* err, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(nC > 0 ? nC : 1) * sizeof(uint32_t);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(k_select, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  k_select<<<1, SEL_THREADS, smem, st>>>(scores, memory, nC, k, period, step, S, err);
  return cudaGetLastError();
}

cudaError_t launch_fold_sumsq(const float* part, int rows, int ld, int N, float* sumsq, int accumulate,
                              cudaStream_t st) {
  k_fold_sumsq<<<(N + 255) / 256, 256, 0, st>>>(part, rows, ld, N, sumsq, accumulate);
  return cudaGetLastError();
}

}  // namespace pop
