// Dense single-token FFN that allocates no device memory.
//
// For callers that cannot allocate GPU memory when they run: processes whose device memory is
// fully reserved at start-up by their own memory manager (an allocation at call time would fail
// or break its accounting), and latency-critical loops that must not enter the CUDA allocator,
// which can block and synchronise the device. They cannot create a pop_ffn handle, so this entry
// point takes the weights in their original row-major layout and keeps its one piece of scratch,
// the activation vector z, in a file-scope device array instead of memory it would allocate.
//
// The array holds POP_STATIC_MAX_D_FF floats (192 KB) on every device that loads the library,
// until the process exits. Every call on a device uses the same array; each call overwrites all
// of z[0, D_FF) before reading it, so nothing has to start at zero, but calls that overlap on the
// GPU (two streams, or two host threads) race on it.
#include <mutex>

#include "pop_device.cuh"
#include "pop_ffn.h"
#include "pop_internal.h"

namespace {

static __device__ __align__(256) float g_static_z[POP_STATIC_MAX_D_FF];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
float* g_z_addr[kMaxDevices] = {};  // device address of g_static_z, per device ordinal
pop_status static_fail(pop_status s, const char* m) {
  pop::set_unbound_error(m);  // readable through pop_last_error(NULL)
  return s;
}

__device__ __forceinline__ float silu_s(float g) { return g / (1.0f + expf(-g)); }

// z[i] = SiLU(Wg[i,:] . x) * (W1[i,:] . x); one warp per channel, rows of length D.
__global__ void __launch_bounds__(256)
    k_static_gateup(const uint16_t* __restrict__ Wg, const uint16_t* __restrict__ W1, const uint16_t* __restrict__ x,
                    int D, int N, float* __restrict__ z) {
  extern __shared__ float xs[];
  for (int d = threadIdx.x; d < D; d += blockDim.x) xs[d] = __uint_as_float(static_cast<uint32_t>(x[d]) << 16);
  __syncthreads();
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int nch = D >> 3;
  for (int i = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); i < N; i += warps) {
    const uint16_t* rg = Wg + static_cast<size_t>(i) * D;
    const uint16_t* ru = W1 + static_cast<size_t>(i) * D;
    float ag = 0.f, au = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const uint4 vg = pop::ldg_stream(rg + 8 * c);
      const uint4 vu = pop::ldg_stream(ru + 8 * c);
      const float* xv = xs + 8 * c;
      const uint32_t wg[4] = {vg.x, vg.y, vg.z, vg.w}, wu[4] = {vu.x, vu.y, vu.z, vu.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        ag = fmaf(pop::bf16lo(wg[k]), xv[2 * k], ag);
        ag = fmaf(pop::bf16hi(wg[k]), xv[2 * k + 1], ag);
        au = fmaf(pop::bf16lo(wu[k]), xv[2 * k], au);
        au = fmaf(pop::bf16hi(wu[k]), xv[2 * k + 1], au);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ag += __shfl_xor_sync(0xffffffffu, ag, o);
      au += __shfl_xor_sync(0xffffffffu, au, o);
    }
    if (lane == 0) z[i] = silu_s(ag) * au;
  }
}

// y[d] = W2[d,:] . z; one warp per output row, rows of length N (a multiple of 8).
__global__ void __launch_bounds__(256)
    k_static_down(const uint16_t* __restrict__ W2, const float* __restrict__ z, int D, int N, void* __restrict__ y,
                  int out_f32) {
  const int lane = threadIdx.x & 31;
  const int warps = gridDim.x * (blockDim.x >> 5);
  const int nch = N >> 3;
  for (int d = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); d < D; d += warps) {
    const uint16_t* row = W2 + static_cast<size_t>(d) * N;
    float acc = 0.f;
    for (int c = lane; c < nch; c += 32) {
      const uint4 v = pop::ldg_stream(row + 8 * c);
      const float4 za = *reinterpret_cast<const float4*>(z + 8 * c);
      const float4 zb = *reinterpret_cast<const float4*>(z + 8 * c + 4);
      acc = fmaf(pop::bf16lo(v.x), za.x, acc);
      acc = fmaf(pop::bf16hi(v.x), za.y, acc);
      acc = fmaf(pop::bf16lo(v.y), za.z, acc);
      acc = fmaf(pop::bf16hi(v.y), za.w, acc);
      acc = fmaf(pop::bf16lo(v.z), zb.x, acc);
      acc = fmaf(pop::bf16hi(v.z), zb.y, acc);
      acc = fmaf(pop::bf16lo(v.w), zb.z, acc);
      acc = fmaf(pop::bf16hi(v.w), zb.w, acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) {
      if (out_f32)
        static_cast<float*>(y)[d] = acc;
      else
        static_cast<__nv_bfloat16*>(y)[d] = __float2bfloat16_rn(acc);
    }
  }
}

bool aligned16s(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" {

pop_status pop_ffn_dense_token_noalloc(const void* Wg, const void* W1, const void* W2, int D, int D_FF,
                                       const void* x, void* y, int out_f32, void* stream) {
  if (!Wg || !W1 || !W2 || !x || !y) return static_fail(POP_ERR_INVALID_ARG, "dense_token_noalloc: NULL pointer");
  if (D < 8 || D > POP_MAX_D || D % 8 != 0)
    return static_fail(POP_ERR_INVALID_ARG, "dense_token_noalloc: D must be a multiple of 8 in [8, POP_MAX_D]");
  if (D_FF < 8 || D_FF % 8 != 0)
    return static_fail(POP_ERR_INVALID_ARG, "dense_token_noalloc: D_FF must be a positive multiple of 8");
  if (D_FF > POP_STATIC_MAX_D_FF)
    return static_fail(POP_ERR_INVALID_ARG,
                       "dense_token_noalloc: D_FF exceeds POP_STATIC_MAX_D_FF, the size of the static scratch");
  if (!aligned16s(Wg) || !aligned16s(W1) || !aligned16s(W2) || !aligned16s(x) || !aligned16s(y))
    return static_fail(POP_ERR_INVALID_ARG, "dense_token_noalloc: pointers must be 16-byte aligned");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return static_fail(POP_ERR_CUDA, "dense_token_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return static_fail(POP_ERR_UNSUPPORTED, "dense_token_noalloc: device ordinal beyond the 64 this entry point tracks");
  // an error left by the caller's own earlier work is reported as such, not as this call's launch
  // failure (and is left in place for the caller)
  if (cudaPeekAtLastError() != cudaSuccess)
    return static_fail(POP_ERR_CUDA, "dense_token_noalloc: a CUDA error from earlier work is pending on this thread");
  float* z = nullptr;
  {
    // first call on this device: look up the device address of the static array (host code only
    // sees a host-side stand-in under its name)
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_z_addr[dev]) {
      cudaDeviceProp prop;
      if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess)
        return static_fail(POP_ERR_CUDA, "dense_token_noalloc: cudaGetDeviceProperties failed");
      if (!(prop.major == 10 && prop.minor == 3))
        return static_fail(POP_ERR_UNSUPPORTED, "dense_token_noalloc: this build targets sm_103a (GB300) only");
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_static_z);
      if (e != cudaSuccess || !p) return static_fail(POP_ERR_CUDA, "dense_token_noalloc: cudaGetSymbolAddress failed");
      g_z_addr[dev] = static_cast<float*>(p);
    }
    z = g_z_addr[dev];
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t smem = static_cast<size_t>(D) * sizeof(float);
  if (pop::ensure_dyn_smem(reinterpret_cast<const void*>(k_static_gateup), smem) != cudaSuccess)
    return static_fail(POP_ERR_CUDA, "dense_token_noalloc: cudaFuncSetAttribute failed");
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (sms <= 0) sms = 1;
  k_static_gateup<<<sms * 4, 256, smem, st>>>(static_cast<const uint16_t*>(Wg), static_cast<const uint16_t*>(W1),
                                                static_cast<const uint16_t*>(x), D, D_FF, z);
  if (cudaGetLastError() != cudaSuccess) return static_fail(POP_ERR_CUDA, "dense_token_noalloc: gate/up launch failed");
  k_static_down<<<sms * 4, 256, 0, st>>>(static_cast<const uint16_t*>(W2), z, D, D_FF, y, out_f32);
  if (cudaGetLastError() != cudaSuccess) return static_fail(POP_ERR_CUDA, "dense_token_noalloc: down launch failed");
  return POP_OK;
}

}  // extern "C"
