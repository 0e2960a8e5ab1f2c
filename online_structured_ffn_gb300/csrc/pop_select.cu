// Selection kernels of the POP FFN: the prefill R/C/P split and the per-step candidate top-k.
//
// "POP: Online Structural Pruning..." (papernotes.org notes), Key design 1: channels at or above
// q_{r+delta} form R, at or below q_{r-delta} form P, the rest C. Key design 2: candidates are
// sorted by their step score and the top ones fill |R| + k = (1 - r) * D_FF survivors.
// "Batch-wise adaptive pruning" (bittide page), abstract: top-k every update period from an
// activation memory that accumulates importance between updates.
//
// Both use the block-wide selection primitives of pop_radix.cuh with all 1024 threads.
#include "pop_device.cuh"
#include "pop_internal.h"
#include "pop_radix.cuh"

namespace pop {

constexpr int SEL_THREADS = 1024;

struct BlockSync {
  __device__ void operator()() const { __syncthreads(); }
};

// ------------------------------------------------------------------ prefill partition
__global__ void __launch_bounds__(SEL_THREADS, 1)
    k_partition(const float* __restrict__ sumsq, const float* __restrict__ n2, float* __restrict__ I, int N,
                int n_P, int n_R, int* __restrict__ rc, int* __restrict__ Plist, int* __restrict__ step,
                float* __restrict__ memory, unsigned* __restrict__ err) {
  extern __shared__ uint32_t keys[];
  __shared__ RadixScratch<SEL_THREADS> sc;
  const int tid = threadIdx.x;
  const BlockSync sync;
  for (int i = tid; i < N; i += SEL_THREADS) {
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
  if (n_P > 0) order_statistic<SEL_THREADS>(tid, keys, N, static_cast<uint32_t>(n_P - 1), sc, sync, vP, jP);
  if (n_R > 0) order_statistic<SEL_THREADS>(tid, keys, N, static_cast<uint32_t>(N - n_R), sc, sync, vR, jR);

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
  block_scan3<SEL_THREADS>(tid, c, off, tot, sc, sync);
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
             int* __restrict__ step, int* __restrict__ S, const int* __restrict__ rc, int* __restrict__ rcs,
             unsigned* __restrict__ err) {
  extern __shared__ uint32_t keys[];
  __shared__ RadixScratch<SEL_THREADS> sc;
  const int t = *step;
  const bool update = (t % period) == 0;
  const bool ok = select_step<SEL_THREADS>(
      threadIdx.x, [&](int i) { return scores[i]; }, memory, nC, k, period, update, keys, S, sc, BlockSync());
  if (!ok && threadIdx.x == 0) atomicOr(err, DEVERR_TOPK);
  __syncthreads();
  if (rcs && update)  // skip variant: the selected channels head the list of the steps until the next update
    for (int j = threadIdx.x; j < k; j += SEL_THREADS) {
      int ps = S[j];
      if (static_cast<unsigned>(ps) >= static_cast<unsigned>(nC)) {
        atomicOr(err, DEVERR_INDEX);
        ps = 0;
      }
      rcs[j] = rc[ps];
    }
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
                          const int* rc, int* rcs, unsigned* err, cudaStream_t st) {
  const size_t smem = static_cast<size_t>(nC > 0 ? nC : 1) * sizeof(uint32_t);
  // the keys plus the kernel's static scratch can pass the 48 KB default even below 48 KB of keys
  {
    cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(k_select), smem);
    if (e != cudaSuccess) return e;
  }
  k_select<<<1, SEL_THREADS, smem, st>>>(scores, memory, nC, k, period, step, S, rc, rcs, err);
  return cudaGetLastError();
}

cudaError_t launch_fold_sumsq(const float* part, int rows, int ld, int N, float* sumsq, int accumulate,
                              cudaStream_t st) {
  k_fold_sumsq<<<(N + 255) / 256, 256, 0, st>>>(part, rows, ld, N, sumsq, accumulate);
  return cudaGetLastError();
}

}  // namespace pop
