// Weight packing for the POP FFN: one contiguous row per intermediate channel,
//   Wp[i] = [ Wg[i, 0:D] | W1[i, 0:D] | W2[0:D, i] ]   (3*D bf16),
// and the down-column norms n2[i] = ||W2[:, i]||_2 (fp32), the weight factor of the Wanda-form
// importance ("POP: Online Structural Pruning..." notes, Key design 1 and "Loss / training
// strategy"). With this layout a decode step that gathers channel i reads one 16 KB gate/up run
// and one 8 KB down run (D = 4096) instead of 3 scattered rows/columns.
#include "pop_device.cuh"
#include "pop_internal.h"

namespace pop {

// Wg, W1 rows -> Wp[:, 0:2D]; 16-byte copies.
__global__ void k_pack_rows(const uint4* __restrict__ Wg, const uint4* __restrict__ W1, uint16_t* __restrict__ Wp,
                            int D, int N) {
  const int cpr = D / 8;  // 16-byte chunks per row
  const long long per = static_cast<long long>(N) * cpr;
  const long long total = 2 * per;
  for (long long e = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; e < total;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int which = static_cast<int>(e / per);
    const long long r = e % per;
    const int i = static_cast<int>(r / cpr), c = static_cast<int>(r % cpr);
    const uint4 v = which == 0 ? Wg[r] : W1[r];
    reinterpret_cast<uint4*>(Wp + static_cast<size_t>(i) * 3 * D + static_cast<size_t>(which) * D)[c] = v;
  }
}

// W2 [D, N] -> Wp[i, 2D + d] = W2[d, i]: 32x32 tiles through shared memory.
__global__ void k_pack_w2(const uint16_t* __restrict__ W2, uint16_t* __restrict__ Wp, int D, int N) {
  __shared__ uint16_t tile[32][33];
  const int i0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
  const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
  for (int yy = ty; yy < 32; yy += 8) {
    const int d = d0 + yy, i = i0 + tx;
    tile[yy][tx] = (d < D && i < N) ? W2[static_cast<size_t>(d) * N + i] : 0;
  }
  __syncthreads();
  for (int yy = ty; yy < 32; yy += 8) {
    const int i = i0 + yy, d = d0 + tx;
    if (i < N && d < D) Wp[static_cast<size_t>(i) * 3 * D + 2 * static_cast<size_t>(D) + d] = tile[tx][yy];
  }
}

// n2[i] = sqrt(sum_d W2[d, i]^2) from the packed down column; one warp per channel, fixed order.
__global__ void k_colnorm(const uint16_t* __restrict__ Wp, float* __restrict__ n2, int D, int N) {
  const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
  if (warp >= N) return;
  const uint16_t* col = Wp + static_cast<size_t>(warp) * 3 * D + 2 * static_cast<size_t>(D);
  float s = 0.f;
  for (int c = lane; c < D / 8; c += 32) {
    const uint4 v = *reinterpret_cast<const uint4*>(col + 8 * c);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = bf16lo(w[k]), b = bf16hi(w[k]);
      s = fmaf(a, a, s);
      s = fmaf(b, b, s);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) n2[warp] = sqrtf(s);
}

cudaError_t launch_pack(const uint16_t* Wg, const uint16_t* W1, const uint16_t* W2, uint16_t* Wp, float* n2,
                        int D, int N, cudaStream_t st) {
  k_pack_rows<<<1024, 256, 0, st>>>(reinterpret_cast<const uint4*>(Wg), reinterpret_cast<const uint4*>(W1), Wp, D,
                                    N);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_pack_w2<<<dim3((N + 31) / 32, (D + 31) / 32), dim3(32, 8), 0, st>>>(W2, Wp, D, N);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_colnorm<<<(N * 32 + 255) / 256, 256, 0, st>>>(Wp, n2, D, N);
  return cudaGetLastError();
}

}  // namespace pop
