// MoE layer of POP-pruned gated-MLP experts: routing, grouping and combining kernels, and the
// C ABI of include/pop_moe.h.
//
// [POP] "POP: Online Structural Pruning Enables Efficient Inference of Large Foundation Models",
// "Loss / training strategy": the method carries over to MoE models with dynamic routing, each
// expert's partition taken at the first forward. The routing rule (top-2 by router logit, ties to
// the lower expert, softmax over the two chosen logits) is this library's reading, stated in
// pop_moe.h. Each expert is a pop_ffn handle driven through its public C ABI; the kernels here only
// route tokens, gather them per expert and add the weighted expert outputs.
#include <cuda_runtime.h>

#include <cstdint>
#include <string>
#include <vector>

#include "pop_moe.h"

struct pop_moe {
  pop_config cfg{};
  int E = 0, D = 0, N = 0;
  std::vector<pop_ffn_t> ex;
  uint16_t* xe = nullptr;  // [E][max_batch][D] bf16: each expert's decode input
  float* ye = nullptr;     // [E][max_batch][D] fp32: each expert's decode output
  int* r_ex = nullptr;     // [cap][2] routed experts of the last call
  float* r_w = nullptr;    // [cap][2] their weights
  int* r_slot = nullptr;   // [cap][2] row of the token within each chosen expert's group
  int route_cap = 0;
  int* counts = nullptr;   // [E] tokens per expert, last call
  int* offsets = nullptr;  // [E + 1] first grouped row of each expert (prefill)
  float* zeros = nullptr;  // [N] importance of an expert without prompt tokens
  unsigned* err = nullptr; // device error word of the routing kernels
  // decode: each expert's two kernels run on a stream of their own, forked from the caller's stream
  // after the routing and joined before the combine (the experts share no data)
  std::vector<cudaStream_t> xs;
  std::vector<cudaEvent_t> xev;  // [E] each expert's step done
  cudaEvent_t fork = nullptr;    // the routing of this step done
  bool concurrent = true;        // pop_moe_set_concurrent
  int last_T = 0;
  bool partitioned = false;
  std::string msg;
};

namespace {

thread_local std::string g_moe_msg;
constexpr unsigned MOE_ERR_INDEX = 1u;
constexpr int MOE_THREADS = 256;

pop_status moe_fail(pop_moe* m, pop_status s, const std::string& msg) {
  (m ? m->msg : g_moe_msg) = msg;
  return s;
}

pop_status moe_cuda_fail(pop_moe* m, cudaError_t e, const char* where) {
  return moe_fail(m, e == cudaErrorMemoryAllocation ? POP_ERR_OOM : POP_ERR_CUDA,
                  std::string(where) + ": " + cudaGetErrorString(e));
}

pop_status moe_expert_fail(pop_moe* m, pop_status s, int e) {
  return moe_fail(m, s, "expert " + std::to_string(e) + ": " + pop_last_error(m->ex[e]));
}

#define MOE_CUDA(m, call)                                      \
  do {                                                         \
    cudaError_t e_ = (call);                                   \
    if (e_ != cudaSuccess) return moe_cuda_fail(m, e_, #call); \
  } while (0)

bool moe_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__device__ __forceinline__ void moe_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void moe_pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// The two largest logits of one token. A later expert replaces an earlier one only when its logit
// is strictly larger, so among equal logits the lower expert index ranks first. Any input, NaN
// included, yields two distinct experts in [0, E).
__device__ __forceinline__ void top2(const float* l, int E, int& e0, int& e1, float& w0, float& w1) {
  int b0 = 0, b1 = -1;
  float v0 = l[0], v1 = 0.f;
  for (int e = 1; e < E; ++e) {
    const float v = l[e];
    if (v > v0) {
      b1 = b0;
      v1 = v0;
      b0 = e;
      v0 = v;
    } else if (b1 < 0 || v > v1) {
      b1 = e;
      v1 = v;
    }
  }
  // softmax over the two chosen logits: w0 = 1 / (1 + exp(l1 - l0)), l1 <= l0
  const float t = expf(v1 - v0);
  w0 = 1.f / (1.f + t);
  w1 = t / (1.f + t);
  e0 = b0;
  e1 = b1;
}

// ---------------------------------------------------------------------------------- prefill

// One thread per token: its two experts and weights.
__global__ void k_moe_topk(const float* __restrict__ logits, int T, int E, int* __restrict__ r_ex,
                           float* __restrict__ r_w) {
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= T) return;
  int e0, e1;
  float w0, w1;
  top2(logits + static_cast<size_t>(t) * E, E, e0, e1, w0, w1);
  r_ex[2 * t] = e0;
  r_ex[2 * t + 1] = e1;
  r_w[2 * t] = w0;
  r_w[2 * t + 1] = w1;
}

// One CTA; warp w numbers the tokens of experts w, w + 32, ... in ascending token order (a ballot
// per 32 tokens), so each expert's group lists its tokens in order. Then the group offsets.
__global__ void __launch_bounds__(1024) k_moe_slots(const int* __restrict__ r_ex, int T, int E,
                                                    int* __restrict__ r_slot, int* __restrict__ counts,
                                                    int* __restrict__ offsets) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt = (1u << lane) - 1u;
  for (int e = warp; e < E; e += blockDim.x >> 5) {
    int base = 0;
    for (int c = 0; c < T; c += 128) {
      int j[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {  // four ballots' loads in flight
        const int t = c + 32 * u + lane;
        j[u] = -1;
        if (t < T) {
          const int2 p = *reinterpret_cast<const int2*>(r_ex + 2 * t);
          j[u] = p.x == e ? 0 : (p.y == e ? 1 : -1);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const unsigned msk = __ballot_sync(0xffffffffu, j[u] >= 0);
        if (j[u] >= 0) r_slot[2 * (c + 32 * u + lane) + j[u]] = base + __popc(msk & lt);
        base += __popc(msk);
      }
    }
    if (lane == 0) counts[e] = base;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int s = 0;
    for (int e = 0; e < E; ++e) {
      offsets[e] = s;
      s += counts[e];
    }
    offsets[E] = s;
  }
}

// One CTA per (token, choice): copies the token's row to its place in the chosen expert's group.
__global__ void __launch_bounds__(MOE_THREADS) k_moe_gather(const uint16_t* __restrict__ X, int T, int D,
                                                            const int* __restrict__ r_ex,
                                                            const int* __restrict__ r_slot,
                                                            const int* __restrict__ offsets,
                                                            uint16_t* __restrict__ Xg, unsigned* err) {
  const int p = blockIdx.x, t = p >> 1;
  const int row = offsets[r_ex[p]] + r_slot[p];
  if (row < 0 || row >= 2 * T) {
    if (threadIdx.x == 0) atomicOr(err, MOE_ERR_INDEX);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(X + static_cast<size_t>(t) * D);
  uint4* dst = reinterpret_cast<uint4*>(Xg + static_cast<size_t>(row) * D);
  for (int i = threadIdx.x; i < D / 8; i += MOE_THREADS) dst[i] = __ldg(src + i);
}

// ---------------------------------------------------------------------------------- decode

// CTA (s, e): every CTA routes the B tokens (B <= 64) in shared memory, finds the token that holds
// row s of expert e's input (the s-th routed token in ascending order) and copies it there, or
// writes a zero row. CTA (0, e) records expert e's count; CTAs (s, 0) record token s's routing.
__global__ void __launch_bounds__(MOE_THREADS) k_moe_route_scatter(const uint16_t* __restrict__ x,
                                                                   const float* __restrict__ logits, int B, int E,
                                                                   int D, uint16_t* __restrict__ xe,
                                                                   int* __restrict__ r_ex, float* __restrict__ r_w,
                                                                   int* __restrict__ r_slot,
                                                                   int* __restrict__ counts) {
  __shared__ int s_e0[64], s_e1[64];
  __shared__ float s_w0[64], s_w1[64];
  __shared__ int s_tok;
  moe_pdl_trigger();
  moe_pdl_wait();  // x, logits and the previous step's use of xe
  const int s = blockIdx.x, e = blockIdx.y;
  if (threadIdx.x < B) {
    int e0, e1;
    float w0, w1;
    top2(logits + static_cast<size_t>(threadIdx.x) * E, E, e0, e1, w0, w1);
    s_e0[threadIdx.x] = e0;
    s_e1[threadIdx.x] = e1;
    s_w0[threadIdx.x] = w0;
    s_w1[threadIdx.x] = w1;
  }
  __syncthreads();
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int found = -1, base = 0;
    for (int c = 0; c < B; c += 32) {
      const int t = c + lane;
      const bool hit = t < B && (s_e0[t] == e || s_e1[t] == e);
      const unsigned msk = __ballot_sync(0xffffffffu, hit);
      if (hit && base + __popc(msk & ((1u << lane) - 1u)) == s) found = t;
      base += __popc(msk);
    }
    found = __reduce_max_sync(0xffffffffu, found);
    if (lane == 0) {
      s_tok = found;
      if (s == 0) counts[e] = base;
    }
  } else if (e == 0 && threadIdx.x == 32) {
    // token s: both choices, their weights and its row in each chosen expert's input
    const int c0 = s_e0[s], c1 = s_e1[s];
    int n0 = 0, n1 = 0;
    for (int t = 0; t < s; ++t) {
      n0 += (s_e0[t] == c0 || s_e1[t] == c0) ? 1 : 0;
      n1 += (s_e0[t] == c1 || s_e1[t] == c1) ? 1 : 0;
    }
    r_ex[2 * s] = c0;
    r_ex[2 * s + 1] = c1;
    r_w[2 * s] = s_w0[s];
    r_w[2 * s + 1] = s_w1[s];
    r_slot[2 * s] = n0;
    r_slot[2 * s + 1] = n1;
  }
  __syncthreads();
  const int tok = s_tok;
  uint4* dst = reinterpret_cast<uint4*>(xe + (static_cast<size_t>(e) * B + s) * D);
  if (tok >= 0) {
    const uint4* src = reinterpret_cast<const uint4*>(x + static_cast<size_t>(tok) * D);
    for (int i = threadIdx.x; i < D / 8; i += MOE_THREADS) dst[i] = __ldg(src + i);
  } else {
    for (int i = threadIdx.x; i < D / 8; i += MOE_THREADS) dst[i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// ---------------------------------------------------------------------------------- combine

__device__ __forceinline__ uint16_t f32_to_bf16_rne(float f) {
  uint32_t u = __float_as_uint(f);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x40u);  // NaN stays NaN
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// y_t = w0 * out[row(e0, slot0)] + w1 * out[row(e1, slot1)], in that order, fp32. The expert
// output rows are grouped: row(e, s) = offsets[e] + s (prefill) or e * per_expert + s (decode).
// Grid (T, ceil(D / (4 * threads))); four outputs per thread.
__global__ void __launch_bounds__(MOE_THREADS) k_moe_combine(const int* __restrict__ r_ex,
                                                             const float* __restrict__ r_w,
                                                             const int* __restrict__ r_slot,
                                                             const int* __restrict__ offsets, int per_expert,
                                                             int E, int rows, const float* __restrict__ yg, int D,
                                                             void* __restrict__ y, int out_f32, unsigned* err) {
  moe_pdl_trigger();
  moe_pdl_wait();  // the experts' outputs
  const int t = blockIdx.x;
  const int d = 4 * (blockIdx.y * MOE_THREADS + threadIdx.x);
  if (d >= D) return;
  const int e0 = r_ex[2 * t], e1 = r_ex[2 * t + 1];
  if (e0 < 0 || e0 >= E || e1 < 0 || e1 >= E) {
    if (d == 0) atomicOr(err, MOE_ERR_INDEX);
    return;
  }
  const int row0 = (offsets ? offsets[e0] : e0 * per_expert) + r_slot[2 * t];
  const int row1 = (offsets ? offsets[e1] : e1 * per_expert) + r_slot[2 * t + 1];
  if (row0 < 0 || row0 >= rows || row1 < 0 || row1 >= rows) {
    if (d == 0) atomicOr(err, MOE_ERR_INDEX);
    return;
  }
  const float w0 = r_w[2 * t], w1 = r_w[2 * t + 1];
  const float4 a = *reinterpret_cast<const float4*>(yg + static_cast<size_t>(row0) * D + d);
  const float4 b = *reinterpret_cast<const float4*>(yg + static_cast<size_t>(row1) * D + d);
  float4 o;
  o.x = __fadd_rn(__fmul_rn(w0, a.x), __fmul_rn(w1, b.x));
  o.y = __fadd_rn(__fmul_rn(w0, a.y), __fmul_rn(w1, b.y));
  o.z = __fadd_rn(__fmul_rn(w0, a.z), __fmul_rn(w1, b.z));
  o.w = __fadd_rn(__fmul_rn(w0, a.w), __fmul_rn(w1, b.w));
  const size_t off = static_cast<size_t>(t) * D + d;
  if (out_f32) {
    *reinterpret_cast<float4*>(static_cast<float*>(y) + off) = o;
  } else {
    uint2 v;
    v.x = f32_to_bf16_rne(o.x) | (static_cast<uint32_t>(f32_to_bf16_rne(o.y)) << 16);
    v.y = f32_to_bf16_rne(o.z) | (static_cast<uint32_t>(f32_to_bf16_rne(o.w)) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(y) + off) = v;
  }
}

template <class K, class... Args>
cudaError_t launch_moe_pdl(K kernel, dim3 grid, dim3 block, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

void free_moe(pop_moe* m) {
  for (pop_ffn_t h : m->ex)
    if (h) pop_ffn_destroy(h);
  m->ex.clear();
  for (cudaStream_t q : m->xs) cudaStreamDestroy(q);
  m->xs.clear();
  for (cudaEvent_t v : m->xev) cudaEventDestroy(v);
  m->xev.clear();
  if (m->fork) cudaEventDestroy(m->fork);
  m->fork = nullptr;
  cudaFree(m->xe);
  cudaFree(m->ye);
  cudaFree(m->r_ex);
  cudaFree(m->r_w);
  cudaFree(m->r_slot);
  cudaFree(m->counts);
  cudaFree(m->offsets);
  cudaFree(m->zeros);
  cudaFree(m->err);
}

cudaError_t alloc_routes(pop_moe* m, int cap) {
  cudaFree(m->r_ex);
  cudaFree(m->r_w);
  cudaFree(m->r_slot);
  m->r_ex = nullptr;
  m->r_w = nullptr;
  m->r_slot = nullptr;
  m->route_cap = 0;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&m->r_ex), sizeof(int) * 2 * static_cast<size_t>(cap));
  if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&m->r_w), sizeof(float) * 2 * static_cast<size_t>(cap));
  if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&m->r_slot), sizeof(int) * 2 * static_cast<size_t>(cap));
  if (e == cudaSuccess) e = cudaMemset(m->r_ex, 0, sizeof(int) * 2 * static_cast<size_t>(cap));
  if (e == cudaSuccess) e = cudaMemset(m->r_slot, 0, sizeof(int) * 2 * static_cast<size_t>(cap));
  if (e == cudaSuccess) m->route_cap = cap;
  return e;
}

}  // namespace

extern "C" {

const char* pop_moe_last_error(pop_moe_t m) { return m ? m->msg.c_str() : g_moe_msg.c_str(); }

pop_status pop_moe_create(const pop_config* cfg, int n_experts, const void* const* Wg, const void* const* W1,
                          const void* const* W2, void* stream, pop_moe_t* out) {
  if (!out) return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_create: out is NULL");
  *out = nullptr;
  if (!cfg || !Wg || !W1 || !W2) return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_create: NULL argument");
  if (n_experts < 2 || n_experts > POP_MOE_MAX_EXPERTS)
    return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_create: n_experts must be in [2, POP_MOE_MAX_EXPERTS]");
  for (int e = 0; e < n_experts; ++e)
    if (!Wg[e] || !W1[e] || !W2[e]) return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_create: NULL weights");
  pop_moe* m = new pop_moe();
  m->cfg = *cfg;
  m->E = n_experts;
  m->D = cfg->D;
  m->N = cfg->D_FF;
  pop_config ecfg = *cfg;
  ecfg.out_f32 = 1;  // the combine adds fp32 expert outputs
  for (int e = 0; e < n_experts; ++e) {
    pop_ffn_t h = nullptr;
    const pop_status s = pop_ffn_create(&ecfg, Wg[e], W1[e], W2[e], stream, &h);
    if (s != POP_OK) {
      const std::string why = std::string("pop_moe_create: expert ") + std::to_string(e) + ": " + pop_last_error(nullptr);
      free_moe(m);
      delete m;
      return moe_fail(nullptr, s, why);
    }
    m->ex.push_back(h);
  }
  const size_t per = static_cast<size_t>(cfg->max_batch) * cfg->D;
  cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&m->xe), sizeof(uint16_t) * per * n_experts);
  if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&m->ye), sizeof(float) * per * n_experts);
  if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&m->counts), sizeof(int) * n_experts);
  if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&m->offsets), sizeof(int) * (n_experts + 1));
  if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&m->zeros), sizeof(float) * (m->N > 0 ? m->N : 1));
  if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void**>(&m->err), sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(m->zeros, 0, sizeof(float) * (m->N > 0 ? m->N : 1));
  if (e == cudaSuccess) e = cudaMemset(m->err, 0, sizeof(unsigned));
  if (e == cudaSuccess) e = cudaMemset(m->counts, 0, sizeof(int) * n_experts);
  if (e == cudaSuccess) e = alloc_routes(m, cfg->max_batch);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&m->fork, cudaEventDisableTiming);
  for (int x = 0; x < n_experts && e == cudaSuccess; ++x) {
    cudaStream_t q = nullptr;
    cudaEvent_t v = nullptr;
    e = cudaStreamCreateWithFlags(&q, cudaStreamNonBlocking);
    if (e == cudaSuccess) m->xs.push_back(q);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&v, cudaEventDisableTiming);
    if (e == cudaSuccess) m->xev.push_back(v);
  }
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) {
    free_moe(m);
    delete m;
    return moe_cuda_fail(nullptr, e, "pop_moe_create");
  }
  *out = m;
  return POP_OK;
}

void pop_moe_destroy(pop_moe_t m) {
  if (!m) return;
  cudaDeviceSynchronize();
  free_moe(m);
  delete m;
}

int pop_moe_num_experts(pop_moe_t m) { return m ? m->E : -1; }

pop_ffn_t pop_moe_expert(pop_moe_t m, int e) {
  if (!m || e < 0 || e >= m->E) return nullptr;
  return m->ex[e];
}

pop_status pop_moe_prefill_partition(pop_moe_t m, const void* X, const float* logits, int M, void* Y,
                                     void* stream) {
  if (!m) return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_prefill_partition: NULL handle");
  if (!X || !logits || M < 1)
    return moe_fail(m, POP_ERR_INVALID_ARG, "pop_moe_prefill_partition: X or logits is NULL, or M < 1");
  if (!moe_aligned16(X) || (Y && !moe_aligned16(Y)))
    return moe_fail(m, POP_ERR_INVALID_ARG, "pop_moe_prefill_partition: X and Y must be 16-byte aligned");
  if (M > (1 << 29)) return moe_fail(m, POP_ERR_INVALID_ARG, "pop_moe_prefill_partition: M too large");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int E = m->E, D = m->D;
  if (M > m->route_cap) {
    MOE_CUDA(m, cudaStreamSynchronize(st));
    MOE_CUDA(m, alloc_routes(m, M));
  }
  k_moe_topk<<<(M + 127) / 128, 128, 0, st>>>(logits, M, E, m->r_ex, m->r_w);
  MOE_CUDA(m, cudaGetLastError());
  k_moe_slots<<<1, 1024, 0, st>>>(m->r_ex, M, E, m->r_slot, m->counts, m->offsets);
  MOE_CUDA(m, cudaGetLastError());
  std::vector<int> off(E + 1);
  MOE_CUDA(m, cudaMemcpyAsync(off.data(), m->offsets, sizeof(int) * (E + 1), cudaMemcpyDeviceToHost, st));
  MOE_CUDA(m, cudaStreamSynchronize(st));
  if (off[E] != 2 * M) return moe_fail(m, POP_ERR_DEVICE, "pop_moe_prefill_partition: routing lost tokens");
  uint16_t* Xg = nullptr;
  float* Yg = nullptr;
  MOE_CUDA(m, cudaMallocAsync(reinterpret_cast<void**>(&Xg), sizeof(uint16_t) * 2 * static_cast<size_t>(M) * D, st));
  if (Y) {
    const cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&Yg), sizeof(float) * 2 * static_cast<size_t>(M) * D, st);
    if (e != cudaSuccess) {
      cudaFreeAsync(Xg, st);
      return moe_cuda_fail(m, e, "cudaMallocAsync");
    }
  }
  pop_status status = POP_OK;
  k_moe_gather<<<2 * M, MOE_THREADS, 0, st>>>(static_cast<const uint16_t*>(X), M, D, m->r_ex, m->r_slot, m->offsets,
                                              Xg, m->err);
  cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) status = moe_cuda_fail(m, ce, "k_moe_gather");
  for (int e = 0; e < E && status == POP_OK; ++e) {
    const int cnt = off[e + 1] - off[e];
    pop_status s;
    if (cnt > 0)
      s = pop_prefill_partition(m->ex[e], Xg + static_cast<size_t>(off[e]) * D, cnt,
                                Yg ? Yg + static_cast<size_t>(off[e]) * D : nullptr, st);
    else
      s = pop_partition_from_importance(m->ex[e], m->zeros, st);
    if (s != POP_OK) status = moe_expert_fail(m, s, e);
  }
  if (status == POP_OK && Y) {
    dim3 grid(M, (D / 4 + MOE_THREADS - 1) / MOE_THREADS);
    ce = launch_moe_pdl(k_moe_combine, grid, dim3(MOE_THREADS), st, static_cast<const int*>(m->r_ex),
                        static_cast<const float*>(m->r_w), static_cast<const int*>(m->r_slot),
                        static_cast<const int*>(m->offsets), 0, E, 2 * M, static_cast<const float*>(Yg), D, Y,
                        m->cfg.out_f32, m->err);
    if (ce != cudaSuccess) status = moe_cuda_fail(m, ce, "k_moe_combine");
  }
  cudaFreeAsync(Xg, st);
  if (Yg) cudaFreeAsync(Yg, st);
  if (status != POP_OK) return status;
  m->last_T = M;
  m->partitioned = true;
  return POP_OK;
}

pop_status pop_moe_decode_step(pop_moe_t m, const void* x, const float* logits, int B, void* y, void* stream) {
  if (!m) return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_decode_step: NULL handle");
  if (!x || !logits || !y) return moe_fail(m, POP_ERR_INVALID_ARG, "pop_moe_decode_step: NULL x, logits or y");
  if (B < 1 || B > m->cfg.max_batch)
    return moe_fail(m, POP_ERR_INVALID_ARG, "pop_moe_decode_step: B outside [1, max_batch]");
  if (!moe_aligned16(x) || !moe_aligned16(y))
    return moe_fail(m, POP_ERR_INVALID_ARG, "pop_moe_decode_step: x and y must be 16-byte aligned");
  if (!m->partitioned) return moe_fail(m, POP_ERR_STATE, "pop_moe_decode_step: no partition (run a prefill first)");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int E = m->E, D = m->D;
  MOE_CUDA(m, launch_moe_pdl(k_moe_route_scatter, dim3(B, E), dim3(MOE_THREADS), st, static_cast<const uint16_t*>(x),
                             logits, B, E, D, m->xe, m->r_ex, m->r_w, m->r_slot, m->counts));
  const size_t per = static_cast<size_t>(B) * D;
  if (m->concurrent) MOE_CUDA(m, cudaEventRecord(m->fork, st));
  for (int e = 0; e < E; ++e) {
    cudaStream_t es = st;
    if (m->concurrent) {
      es = m->xs[e];
      MOE_CUDA(m, cudaStreamWaitEvent(es, m->fork, 0));
    }
    const pop_status s = pop_decode_step(m->ex[e], m->xe + e * per, B, m->ye + e * per, es);
    if (s != POP_OK) return moe_expert_fail(m, s, e);
    if (m->concurrent) MOE_CUDA(m, cudaEventRecord(m->xev[e], es));
  }
  if (m->concurrent)
    for (int e = 0; e < E; ++e) MOE_CUDA(m, cudaStreamWaitEvent(st, m->xev[e], 0));
  dim3 grid(B, (D / 4 + MOE_THREADS - 1) / MOE_THREADS);
  MOE_CUDA(m, launch_moe_pdl(k_moe_combine, grid, dim3(MOE_THREADS), st, static_cast<const int*>(m->r_ex),
                             static_cast<const float*>(m->r_w), static_cast<const int*>(m->r_slot),
                             static_cast<const int*>(nullptr), B, E, E * B, static_cast<const float*>(m->ye), D, y,
                             m->cfg.out_f32, m->err));
  m->last_T = B;
  return POP_OK;
}

pop_status pop_moe_set_concurrent(pop_moe_t m, int on) {
  if (!m) return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_set_concurrent: NULL handle");
  m->concurrent = on != 0;
  return POP_OK;
}

pop_status pop_moe_get_routing(pop_moe_t m, int* T, int* experts, float* weights) {
  if (!m) return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_get_routing: NULL handle");
  if (!T) return moe_fail(m, POP_ERR_INVALID_ARG, "pop_moe_get_routing: T is NULL");
  if (m->last_T == 0) return moe_fail(m, POP_ERR_STATE, "pop_moe_get_routing: no call yet");
  MOE_CUDA(m, cudaDeviceSynchronize());
  *T = m->last_T;
  const size_t n = 2 * static_cast<size_t>(m->last_T);
  if (experts) MOE_CUDA(m, cudaMemcpy(experts, m->r_ex, sizeof(int) * n, cudaMemcpyDeviceToHost));
  if (weights) MOE_CUDA(m, cudaMemcpy(weights, m->r_w, sizeof(float) * n, cudaMemcpyDeviceToHost));
  return POP_OK;
}

pop_status pop_moe_get_counts(pop_moe_t m, int* counts) {
  if (!m) return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_get_counts: NULL handle");
  if (!counts) return moe_fail(m, POP_ERR_INVALID_ARG, "pop_moe_get_counts: counts is NULL");
  MOE_CUDA(m, cudaDeviceSynchronize());
  MOE_CUDA(m, cudaMemcpy(counts, m->counts, sizeof(int) * m->E, cudaMemcpyDeviceToHost));
  return POP_OK;
}

pop_status pop_moe_check(pop_moe_t m) {
  if (!m) return moe_fail(nullptr, POP_ERR_INVALID_ARG, "pop_moe_check: NULL handle");
  MOE_CUDA(m, cudaDeviceSynchronize());
  unsigned w = 0;
  MOE_CUDA(m, cudaMemcpy(&w, m->err, sizeof(unsigned), cudaMemcpyDeviceToHost));
  if (w) {
    MOE_CUDA(m, cudaMemset(m->err, 0, sizeof(unsigned)));
    return moe_fail(m, POP_ERR_DEVICE, "pop_moe_check: a routing kernel saw an index out of range");
  }
  for (int e = 0; e < m->E; ++e) {
    const pop_status s = pop_check(m->ex[e]);
    if (s != POP_OK) return moe_expert_fail(m, s, e);
  }
  return POP_OK;
}

}  // extern "C"
