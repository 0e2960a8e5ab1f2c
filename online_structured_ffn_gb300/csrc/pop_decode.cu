// Decode-step kernels of the POP FFN (one decode token per sequence, B sequences sharing a mask).
//
// Gate/up over R u C ("POP: Online Structural Pruning...", Key design 2: H_t = f(X_t; R u C)),
// the candidate score a_i = max_b |z_{b,i}| * ||W2[:,i]|| ("Batch-wise adaptive pruning",
// Fig. 2(a): element-wise max over the batch), and the down projection over R plus the selected
// candidates (POP notes, flowchart: combine R and the chosen candidates for the final FFN).
//
// Weights are read from the packed channel-major layout: row i = [Wg[i,:] | W1[i,:] | W2[:,i]],
// so every channel's gate/up rows (16 KB at D = 4096) and down column (8 KB) are contiguous and
// the gathers stream whole rows with 16-byte loads.
#include "pop_device.cuh"
#include "pop_internal.h"

namespace pop {

__device__ __forceinline__ float silu_f(float g) { return g / (1.0f + expf(-g)); }

// Index lists come from this library's own kernels or from host-validated uploads; a value out of
// range is still caught here, recorded in the error word, and replaced by 0 so that no access
// leaves the buffers.
__device__ __forceinline__ int guard_index(int v, int n, unsigned* err) {
  if (static_cast<unsigned>(v) >= static_cast<unsigned>(n)) {
    atomicOr(err, DEVERR_INDEX);
    return 0;
  }
  return v;
}

// ======================================================================= gate/up, B = 1
// One warp per channel; lanes stride over 16-byte chunks of the two contiguous rows; x (fp32)
// sits in shared memory. Channels are split into balanced contiguous ranges, one per warp.
constexpr int GU1_THREADS = 256;
constexpr int GU1_WARPS = GU1_THREADS / 32;

template <int NCHL>
__global__ void __launch_bounds__(GU1_THREADS, 4)
    k_gateup_b1(const uint16_t* __restrict__ Wp, const float* __restrict__ n2, const uint16_t* __restrict__ x,
                int D, int N, const int* __restrict__ rc, int nRC, int nC, float* __restrict__ z,
                float* __restrict__ scores, unsigned* __restrict__ err) {
  extern __shared__ float xs[];
  for (int d = threadIdx.x; d < D; d += GU1_THREADS) xs[d] = __uint_as_float(static_cast<uint32_t>(x[d]) << 16);
  __syncthreads();

  const int lane = threadIdx.x & 31;
  const long long W = static_cast<long long>(gridDim.x) * GU1_WARPS;
  const long long w = static_cast<long long>(blockIdx.x) * GU1_WARPS + (threadIdx.x >> 5);
  const int p0 = static_cast<int>(w * nRC / W);
  const int p1 = static_cast<int>((w + 1) * nRC / W);
  const int nch = D >> 3;
  const size_t row3 = 3 * static_cast<size_t>(D);
  constexpr int G = NCHL < 4 ? NCHL : 4;

  for (int p = p0; p < p1; ++p) {
    const int ch = guard_index(rc[p], N, err);
    const uint16_t* rg = Wp + static_cast<size_t>(ch) * row3;
    const uint16_t* ru = rg + D;
    float ag0 = 0.f, ag1 = 0.f, au0 = 0.f, au1 = 0.f;
#pragma unroll 1
    for (int j0 = 0; j0 < NCHL; j0 += G) {
      uint4 vg[G], vu[G];
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const int c = lane + 32 * (j0 + j);
        if (c < nch) {
          vg[j] = ldg_stream(rg + 8 * c);
          vu[j] = ldg_stream(ru + 8 * c);
        } else {
          vg[j] = make_uint4(0u, 0u, 0u, 0u);
          vu[j] = vg[j];
        }
      }
#pragma unroll
      for (int j = 0; j < G; ++j) {
        const int c = lane + 32 * (j0 + j);
        if (c < nch) {
          const float4 xa = *reinterpret_cast<const float4*>(xs + 8 * c);
          const float4 xb = *reinterpret_cast<const float4*>(xs + 8 * c + 4);
          ag0 = fmaf(bf16lo(vg[j].x), xa.x, ag0);
          ag1 = fmaf(bf16hi(vg[j].x), xa.y, ag1);
          ag0 = fmaf(bf16lo(vg[j].y), xa.z, ag0);
          ag1 = fmaf(bf16hi(vg[j].y), xa.w, ag1);
          ag0 = fmaf(bf16lo(vg[j].z), xb.x, ag0);
          ag1 = fmaf(bf16hi(vg[j].z), xb.y, ag1);
          ag0 = fmaf(bf16lo(vg[j].w), xb.z, ag0);
          ag1 = fmaf(bf16hi(vg[j].w), xb.w, ag1);
          au0 = fmaf(bf16lo(vu[j].x), xa.x, au0);
          au1 = fmaf(bf16hi(vu[j].x), xa.y, au1);
          au0 = fmaf(bf16lo(vu[j].y), xa.z, au0);
          au1 = fmaf(bf16hi(vu[j].y), xa.w, au1);
          au0 = fmaf(bf16lo(vu[j].z), xb.x, au0);
          au1 = fmaf(bf16hi(vu[j].z), xb.y, au1);
          au0 = fmaf(bf16lo(vu[j].w), xb.z, au0);
          au1 = fmaf(bf16hi(vu[j].w), xb.w, au1);
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
      const float zz = silu_f(ag) * au;
      z[p] = zz;
      if (p < nC) scores[p] = fabsf(zz) * n2[ch];
    }
  }
}

// ======================================================================= gate/up, B > 1
// Tensor cores (mma.sync m16n8k16, bf16 -> fp32) with channels as M = 16 and tokens as N = 8
// per tile. Each CTA owns 16 channels; its 4 warps split D in 64-wide blocks and are summed in
// shared memory. Each lane loads 32 contiguous bytes of a row per block, so the K order inside
// an MMA is permuted; x is loaded with the same permutation, which leaves the dot product as is:
// in k-step j (0..3) of block kb, lane (g, q) supplies d = 64kb + 16q + 4j + {0,1} for the
// fragment slots k = 2q + {0,1} and d = 64kb + 16q + 4j + {2,3} for k = 2q + 8 + {0,1}.
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const uint4& lo, const uint4& hi, int w) {
  switch (w) {
    case 0: return lo.x;
    case 1: return lo.y;
    case 2: return lo.z;
    case 3: return lo.w;
    case 4: return hi.x;
    case 5: return hi.y;
    case 6: return hi.z;
    default: return hi.w;
  }
}

template <int NT>
__global__ void __launch_bounds__(128)
    k_gateup_mma(const uint16_t* __restrict__ Wp, const float* __restrict__ n2, const uint16_t* __restrict__ x,
                 int B, int D, int N, const int* __restrict__ rc, int nRC, int nC, float* __restrict__ z,
                 int ldz, float* __restrict__ scores, unsigned* __restrict__ err) {
  __shared__ float red[4][2][16][NT * 8];
  __shared__ float smax[16][NT * 8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  const int pbase = blockIdx.x * 16;
  const int plo = pbase + g, phi = pbase + g + 8;
  const bool vlo = plo < nRC, vhi = phi < nRC;
  const size_t row3 = 3 * static_cast<size_t>(D);
  const int chlo = vlo ? guard_index(rc[plo], N, err) : 0;
  const int chhi = vhi ? guard_index(rc[phi], N, err) : 0;
  const uint16_t* glo = Wp + static_cast<size_t>(chlo) * row3;
  const uint16_t* ghi = Wp + static_cast<size_t>(chhi) * row3;
  const uint16_t* ulo = glo + D;
  const uint16_t* uhi = ghi + D;

  float accg[NT][4], accu[NT][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
#pragma unroll
    for (int e = 0; e < 4; ++e) accg[t][e] = accu[t][e] = 0.f;

  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  const int nkb = (D + 63) >> 6;
  for (int kb = warp; kb < nkb; kb += 4) {
    const int d0 = kb * 64 + 16 * q;
    const bool ok0 = d0 + 8 <= D, ok1 = d0 + 16 <= D;
    const uint4 gl0 = (vlo && ok0) ? ldg_stream(glo + d0) : zero4;
    const uint4 gl1 = (vlo && ok1) ? ldg_stream(glo + d0 + 8) : zero4;
    const uint4 gh0 = (vhi && ok0) ? ldg_stream(ghi + d0) : zero4;
    const uint4 gh1 = (vhi && ok1) ? ldg_stream(ghi + d0 + 8) : zero4;
    const uint4 ul0 = (vlo && ok0) ? ldg_stream(ulo + d0) : zero4;
    const uint4 ul1 = (vlo && ok1) ? ldg_stream(ulo + d0 + 8) : zero4;
    const uint4 uh0 = (vhi && ok0) ? ldg_stream(uhi + d0) : zero4;
    const uint4 uh1 = (vhi && ok1) ? ldg_stream(uhi + d0 + 8) : zero4;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int n = t * 8 + g;
      const uint16_t* xr = x + static_cast<size_t>(n) * D + d0;
      const uint4 x0 = (n < B && ok0) ? *reinterpret_cast<const uint4*>(xr) : zero4;
      const uint4 x1 = (n < B && ok1) ? *reinterpret_cast<const uint4*>(xr + 8) : zero4;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t b0 = word_of(x0, x1, 2 * j), b1 = word_of(x0, x1, 2 * j + 1);
        mma_bf16_16816(accg[t], word_of(gl0, gl1, 2 * j), word_of(gh0, gh1, 2 * j), word_of(gl0, gl1, 2 * j + 1),
                       word_of(gh0, gh1, 2 * j + 1), b0, b1);
        mma_bf16_16816(accu[t], word_of(ul0, ul1, 2 * j), word_of(uh0, uh1, 2 * j), word_of(ul0, ul1, 2 * j + 1),
                       word_of(uh0, uh1, 2 * j + 1), b0, b1);
      }
    }
  }
  // accumulator (row g, cols 2q, 2q+1) and (row g+8, same cols) of each n-tile
#pragma unroll
  for (int t = 0; t < NT; ++t) {
    const int c = t * 8 + 2 * q;
    red[warp][0][g][c] = accg[t][0];
    red[warp][0][g][c + 1] = accg[t][1];
    red[warp][0][g + 8][c] = accg[t][2];
    red[warp][0][g + 8][c + 1] = accg[t][3];
    red[warp][1][g][c] = accu[t][0];
    red[warp][1][g][c + 1] = accu[t][1];
    red[warp][1][g + 8][c] = accu[t][2];
    red[warp][1][g + 8][c + 1] = accu[t][3];
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < NT; ++i) {
    const int idx = threadIdx.x + 128 * i;
    const int row = idx & 15, col = idx >> 4;
    const float gs = ((red[0][0][row][col] + red[1][0][row][col]) + red[2][0][row][col]) + red[3][0][row][col];
    const float us = ((red[0][1][row][col] + red[1][1][row][col]) + red[2][1][row][col]) + red[3][1][row][col];
    const float zz = silu_f(gs) * us;
    const int p = pbase + row;
    smax[row][col] = (col < B) ? fabsf(zz) : 0.f;
    if (col < B && p < nRC) z[static_cast<size_t>(col) * ldz + p] = zz;
  }
  __syncthreads();
  if (threadIdx.x < 16) {
    const int p = pbase + threadIdx.x;
    if (p < nC) {
      float m = 0.f;
      for (int col = 0; col < B; ++col) m = fmaxf(m, smax[threadIdx.x][col]);
      scores[p] = m * n2[guard_index(rc[p], N, err)];
    }
  }
}

// ======================================================================= down, B = 1
// Items: R (rc positions nC .. nC+nR-1) followed by the selected candidates (rc positions S[]).
// CTA j owns a balanced contiguous range of items and a full partial y in registers: thread t
// owns the 8-element chunks t, t+512, ... of the down column.
constexpr int DN1_THREADS = 512;
constexpr int DN1_BATCH = 256;

template <int NCK>
__global__ void __launch_bounds__(DN1_THREADS)
    k_down_b1(const uint16_t* __restrict__ Wp, int D, int N, const int* __restrict__ rc, int nC, int nR,
              const int* __restrict__ S, int k, const float* __restrict__ z, float* __restrict__ ypart,
              unsigned* __restrict__ err) {
  __shared__ int s_ch[DN1_BATCH];
  __shared__ float s_z[DN1_BATCH];
  const long long n = static_cast<long long>(nR) + k;
  const int i0 = static_cast<int>(blockIdx.x * n / gridDim.x);
  const int i1 = static_cast<int>((blockIdx.x + 1) * n / gridDim.x);
  const int nch = D >> 3;
  const size_t row3 = 3 * static_cast<size_t>(D);
  float acc[NCK][8];
#pragma unroll
  for (int c = 0; c < NCK; ++c)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[c][e] = 0.f;

  for (int base = i0; base < i1; base += DN1_BATCH) {
    const int cnt = min(DN1_BATCH, i1 - base);
    __syncthreads();
    if (threadIdx.x < cnt) {
      const int it = base + threadIdx.x;
      const int pos = it < nR ? nC + it : guard_index(S[it - nR], nC, err);
      s_ch[threadIdx.x] = guard_index(rc[pos], N, err);
      s_z[threadIdx.x] = z[pos];
    }
    __syncthreads();
    constexpr int U = 8;
    for (int ii = 0; ii < cnt; ii += U) {
      uint4 v[U][NCK];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const bool ok = ii + u < cnt;
        const uint16_t* col = Wp + static_cast<size_t>(ok ? s_ch[ii + u] : 0) * row3 + 2 * static_cast<size_t>(D);
#pragma unroll
        for (int c = 0; c < NCK; ++c) {
          const int ck = threadIdx.x + DN1_THREADS * c;
          v[u][c] = (ok && ck < nch) ? ldg_stream(col + 8 * ck) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float zz = (ii + u < cnt) ? s_z[ii + u] : 0.f;
#pragma unroll
        for (int c = 0; c < NCK; ++c) {
          acc[c][0] = fmaf(bf16lo(v[u][c].x), zz, acc[c][0]);
          acc[c][1] = fmaf(bf16hi(v[u][c].x), zz, acc[c][1]);
          acc[c][2] = fmaf(bf16lo(v[u][c].y), zz, acc[c][2]);
          acc[c][3] = fmaf(bf16hi(v[u][c].y), zz, acc[c][3]);
          acc[c][4] = fmaf(bf16lo(v[u][c].z), zz, acc[c][4]);
          acc[c][5] = fmaf(bf16hi(v[u][c].z), zz, acc[c][5]);
          acc[c][6] = fmaf(bf16lo(v[u][c].w), zz, acc[c][6]);
          acc[c][7] = fmaf(bf16hi(v[u][c].w), zz, acc[c][7]);
        }
      }
    }
  }
  float* out = ypart + static_cast<size_t>(blockIdx.x) * D;
#pragma unroll
  for (int c = 0; c < NCK; ++c) {
    const int ck = threadIdx.x + DN1_THREADS * c;
    if (ck < nch) {
      float4* o = reinterpret_cast<float4*>(out + 8 * ck);
      o[0] = make_float4(acc[c][0], acc[c][1], acc[c][2], acc[c][3]);
      o[1] = make_float4(acc[c][4], acc[c][5], acc[c][6], acc[c][7]);
    }
  }
}

// ======================================================================= down, B > 1
// CUDA cores: CTA (d-tile of 512, item range); each thread owns 2 consecutive d and all tokens.
constexpr int DNB_THREADS = 256;
constexpr int DNB_ITEMS = 64;

template <int NBG>
__global__ void __launch_bounds__(DNB_THREADS)
    k_down_bn(const uint16_t* __restrict__ Wp, int D, int N, const int* __restrict__ rc, int nC, int nR,
              const int* __restrict__ S, int k, const float* __restrict__ z, int ldz, int B,
              float* __restrict__ ypart, unsigned* __restrict__ err) {
  constexpr int TB = NBG * 16;
  __shared__ int s_ch[DNB_ITEMS];
  __shared__ __align__(16) float s_z[DNB_ITEMS][TB];
  const long long n = static_cast<long long>(nR) + k;
  const int i0 = static_cast<int>(blockIdx.y * n / gridDim.y);
  const int i1 = static_cast<int>((blockIdx.y + 1) * n / gridDim.y);
  const int d0 = blockIdx.x * (2 * DNB_THREADS) + 2 * threadIdx.x;
  const bool dok = d0 < D;
  const size_t row3 = 3 * static_cast<size_t>(D);
  float acc[TB][2];
#pragma unroll
  for (int b = 0; b < TB; ++b) acc[b][0] = acc[b][1] = 0.f;

  for (int base = i0; base < i1; base += DNB_ITEMS) {
    const int cnt = min(DNB_ITEMS, i1 - base);
    __syncthreads();
    for (int e = threadIdx.x; e < cnt * TB; e += DNB_THREADS) {
      const int ii = e / TB, b = e % TB;
      const int it = base + ii;
      const int pos = it < nR ? nC + it : guard_index(S[it - nR], nC, err);
      if (b == 0) s_ch[ii] = guard_index(rc[pos], N, err);
      s_z[ii][b] = b < B ? z[static_cast<size_t>(b) * ldz + pos] : 0.f;
    }
    __syncthreads();
    for (int ii = 0; ii < cnt; ++ii) {
      const uint16_t* col = Wp + static_cast<size_t>(s_ch[ii]) * row3 + 2 * static_cast<size_t>(D);
      const uint32_t wv = dok ? *reinterpret_cast<const uint32_t*>(col + d0) : 0u;
      const float f0 = bf16lo(wv), f1 = bf16hi(wv);
#pragma unroll
      for (int b4 = 0; b4 < TB; b4 += 4) {
        const float4 zz = *reinterpret_cast<const float4*>(&s_z[ii][b4]);
        acc[b4][0] = fmaf(zz.x, f0, acc[b4][0]);
        acc[b4][1] = fmaf(zz.x, f1, acc[b4][1]);
        acc[b4 + 1][0] = fmaf(zz.y, f0, acc[b4 + 1][0]);
        acc[b4 + 1][1] = fmaf(zz.y, f1, acc[b4 + 1][1]);
        acc[b4 + 2][0] = fmaf(zz.z, f0, acc[b4 + 2][0]);
        acc[b4 + 2][1] = fmaf(zz.z, f1, acc[b4 + 2][1]);
        acc[b4 + 3][0] = fmaf(zz.w, f0, acc[b4 + 3][0]);
        acc[b4 + 3][1] = fmaf(zz.w, f1, acc[b4 + 3][1]);
      }
    }
  }
  if (dok) {
    float* out = ypart + static_cast<size_t>(blockIdx.y) * B * D;
#pragma unroll
    for (int b = 0; b < TB; ++b)
      if (b < B) *reinterpret_cast<float2*>(out + static_cast<size_t>(b) * D + d0) = make_float2(acc[b][0], acc[b][1]);
  }
}

// ======================================================================= reduction of partials
// y[e] = sum_g ypart[g][e], g ascending in 8 fixed groups, then the 8 group sums in order.
__global__ void __launch_bounds__(256)
    k_reduce_y(const float* __restrict__ ypart, int G, long long BD, void* __restrict__ y, int out_f32) {
  __shared__ float sh[8][32];
  const int lane = threadIdx.x & 31, grp = threadIdx.x >> 5;
  const long long e = static_cast<long long>(blockIdx.x) * 32 + lane;
  const int g0 = grp * G / 8, g1 = (grp + 1) * G / 8;
  float s = 0.f;
  if (e < BD) {
#pragma unroll 4
    for (int g = g0; g < g1; ++g) s += ypart[static_cast<size_t>(g) * BD + e];
  }
  sh[grp][lane] = s;
  __syncthreads();
  if (grp == 0 && e < BD) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) t += sh[i][lane];
    if (out_f32)
      static_cast<float*>(y)[e] = t;
    else
      static_cast<__nv_bfloat16*>(y)[e] = __float2bfloat16_rn(t);
  }
}

// ======================================================================= launchers
static int pow2_at_least(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}

cudaError_t launch_gateup_decode(const PackedWeights& w, const uint16_t* x, int B, const int* rc, int nRC, int nC,
                                 float* z, int ldz, float* scores, unsigned* err, int num_sms, cudaStream_t st) {
  if (nRC <= 0) return cudaSuccess;
  if (B == 1) {
    const int nchl = pow2_at_least((w.D / 8 + 31) / 32);
    const size_t smem = static_cast<size_t>(w.D) * sizeof(float);
    const int grid = num_sms * 4;
#define POP_GU1(NC)                                                                                  \
  case NC: {                                                                                         \
    if (smem > 48 * 1024)                                                                            \
      cudaFuncSetAttribute(k_gateup_b1<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    k_gateup_b1<NC><<<grid, GU1_THREADS, smem, st>>>(w.Wp, w.n2, x, w.D, w.N, rc, nRC, nC, z, scores, err); \
    break;                                                                                           \
  }
    switch (nchl) {
      POP_GU1(1) POP_GU1(2) POP_GU1(4) POP_GU1(8) POP_GU1(16) POP_GU1(32) POP_GU1(64)
      default: return cudaErrorInvalidValue;
    }
#undef POP_GU1
    return cudaGetLastError();
  }
  const int nt = (B + 7) / 8;
  const int grid = (nRC + 15) / 16;
#define POP_GUM(NTV)                                                                                    \
  case NTV:                                                                                             \
    k_gateup_mma<NTV><<<grid, 128, 0, st>>>(w.Wp, w.n2, x, B, w.D, w.N, rc, nRC, nC, z, ldz, scores, err); \
    break;
  switch (nt) {
    POP_GUM(1) POP_GUM(2) POP_GUM(3) POP_GUM(4) POP_GUM(5) POP_GUM(6) POP_GUM(7) POP_GUM(8)
    default: return cudaErrorInvalidValue;
  }
#undef POP_GUM
  return cudaGetLastError();
}

int down_decode_parts(int D, int B, int nitems, int num_sms) {
  if (nitems <= 0) return 1;
  if (B == 1) return nitems < num_sms ? nitems : num_sms;
  const int dt = (D + 2 * DNB_THREADS - 1) / (2 * DNB_THREADS);
  int gk = (2 * num_sms + dt - 1) / dt;
  if (gk > nitems) gk = nitems;
  return gk < 1 ? 1 : gk;
}

cudaError_t launch_down_decode(const PackedWeights& w, const int* rc, int nC, int nR, const int* S, int k,
                               const float* z, int ldz, int B, float* ypart, int max_parts, int* G_out,
                               unsigned* err, int num_sms, cudaStream_t st) {
  const int n = nR + k;
  int G = down_decode_parts(w.D, B, n, num_sms);
  if (G > max_parts) G = max_parts;
  *G_out = G;
  if (n == 0) {
    // nothing is kept: the output is zero
    *G_out = 1;
    return cudaMemsetAsync(ypart, 0, sizeof(float) * static_cast<size_t>(B) * w.D, st);
  }
  if (B == 1) {
    const int nck = pow2_at_least((w.D / 8 + DN1_THREADS - 1) / DN1_THREADS);
    switch (nck) {
      case 1: k_down_b1<1><<<G, DN1_THREADS, 0, st>>>(w.Wp, w.D, w.N, rc, nC, nR, S, k, z, ypart, err); break;
      case 2: k_down_b1<2><<<G, DN1_THREADS, 0, st>>>(w.Wp, w.D, w.N, rc, nC, nR, S, k, z, ypart, err); break;
      case 4: k_down_b1<4><<<G, DN1_THREADS, 0, st>>>(w.Wp, w.D, w.N, rc, nC, nR, S, k, z, ypart, err); break;
      default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
  }
  const dim3 grid((w.D + 2 * DNB_THREADS - 1) / (2 * DNB_THREADS), G);
  switch ((B + 15) / 16) {
    case 1: k_down_bn<1><<<grid, DNB_THREADS, 0, st>>>(w.Wp, w.D, w.N, rc, nC, nR, S, k, z, ldz, B, ypart, err); break;
    case 2: k_down_bn<2><<<grid, DNB_THREADS, 0, st>>>(w.Wp, w.D, w.N, rc, nC, nR, S, k, z, ldz, B, ypart, err); break;
    case 3: k_down_bn<3><<<grid, DNB_THREADS, 0, st>>>(w.Wp, w.D, w.N, rc, nC, nR, S, k, z, ldz, B, ypart, err); break;
    case 4: k_down_bn<4><<<grid, DNB_THREADS, 0, st>>>(w.Wp, w.D, w.N, rc, nC, nR, S, k, z, ldz, B, ypart, err); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_reduce_y(const float* ypart, int G, int B, int D, void* y, int out_f32, cudaStream_t st) {
  const long long BD = static_cast<long long>(B) * D;
  const unsigned grid = static_cast<unsigned>((BD + 31) / 32);
  k_reduce_y<<<grid, 256, 0, st>>>(ypart, G, BD, y, out_f32);
  return cudaGetLastError();
}

}  // namespace pop
