// Prefill GEMMs of the POP FFN on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Prefill runs the FFN dense over all prompt tokens ("POP: Online Structural Pruning..." notes,
// "Loss / training strategy": the partition is taken at the first forward) and reduces the
// per-channel activation energy sum_t z_{t,i}^2 that the importance I_i = ||W2[:,i]|| * s_i needs
// (Key design 1). The gated MLP itself is eq. (1) of "Batch-wise adaptive pruning", Section 3.1.
//
// Kernel 1 (gate/up): for a tile of 128 tokens x 128 channels one UMMA of shape M=128, N=256
// computes gate (columns 0..127) and up (128..255) together: the B tile stacks 128 Wg rows on
// 128 W1 rows. The epilogue forms z = SiLU(g) * u in fp32 and stores it for the down GEMM as two
// bf16 planes, hi = bf16(z) and lo = bf16(z - hi) (together about 16 significant bits, so y keeps
// z's fp32 precision); it reduces z^2 (from the un-rounded fp32 z) over each warp's 32 rows with a
// butterfly reduce-scatter, writing one partial row per 32 tokens (deterministic; folded later).
// Kernel 2 (down): Y = Z W2^T = Z_hi W2^T + Z_lo W2^T with M=128 tokens, N=256 outputs; a stage
// holds the hi and lo tiles of one k-block and one W2 tile that both MMAs read. The W2 operand
// comes straight from the channel-major packed rows, so it is MN-major (d contiguous) in shared
// memory.
//
// Both kernels are persistent (at most one CTA per SM), warp-specialised (warp 0 TMA producer,
// warp 1 MMA issuer and TMEM owner, warps 2..5 epilogue), with a TMA ring of 192 KB (4 stages of
// 48 KB for gate/up, 3 of 64 KB for down) and two 256-column TMEM accumulators so that the
// epilogue of tile i overlaps the MMAs of tile i+1. Every mbarrier wait is bounded; on a time-out
// the CTA records DEVERR_TIMEOUT_*, stops issuing, waits (bounded) for its TMA copies and MMAs in
// flight, frees TMEM and returns.
#include "pop_device.cuh"
#include "pop_internal.h"

namespace pop {

namespace {
constexpr int BM = 128;
constexpr int BK = 64;  // one 128-byte swizzle row of bf16
constexpr int MAX_STAGES = 4;
constexpr int THREADS = 192;
constexpr uint32_t A_BYTES = BM * BK * 2;   // 16 KB
constexpr uint32_t B_BYTES = 256 * BK * 2;  // 32 KB
// gate/up: [A | B] x 4 stages; down: [A hi | A lo | B] x 3 stages (192 KB either way)
template <int MODE>
struct Ring {
  static constexpr int stages = MODE == 0 ? 4 : 3;
  static constexpr uint32_t a_planes = MODE == 0 ? 1u : 2u;
  static constexpr uint32_t stage_bytes = a_planes * A_BYTES + B_BYTES;
};
constexpr uint32_t RING_BYTES = 4 * (A_BYTES + B_BYTES);
static_assert(Ring<1>::stages * Ring<1>::stage_bytes == RING_BYTES, "both modes use the same ring");
constexpr uint32_t TMEM_COLS = 512;  // two accumulators of 256 fp32 columns
constexpr int GU_BN = 128;           // channels per gate/up tile
constexpr int DN_BN = 256;           // outputs per down tile
// Limit for the waits that drain a CTA's own copies and MMAs before it frees TMEM and exits;
// independent of the caller's wait limit so that a short limit never lets a CTA exit with work
// of its own in flight.
constexpr uint64_t DRAIN_NS = 1000000000ull;

struct Ctl {
  uint64_t full[MAX_STAGES];
  uint64_t empty[MAX_STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
constexpr size_t SMEM_BYTES = 1024 + RING_BYTES + sizeof(Ctl);
}  // namespace

size_t prefill_smem_bytes() { return SMEM_BYTES; }

__device__ __forceinline__ float silu_p(float g) { return g / (1.0f + expf(-g)); }

// MODE 0 (gate/up): mapA = X, mapB0 = Wg, mapB1 = W1; writes Z (hi plane) and Zlo, and part.
// MODE 1 (down): mapA = Z hi plane, mapA2 = Z lo plane, mapB0 = W2; writes Y.
template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    k_prefill_gemm(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapA2,
                   const __grid_constant__ CUtensorMap mapB0, const __grid_constant__ CUtensorMap mapB1, int M,
                   int Nout, int K, uint16_t* __restrict__ Z, uint16_t* __restrict__ Zlo, int ldZ,
                   float* __restrict__ part, int ldPart, void* __restrict__ Y, int out_f32,
                   unsigned* __restrict__ err, uint64_t wait_ns) {
  constexpr int STAGES = Ring<MODE>::stages;
  constexpr uint32_t STAGE_BYTES = Ring<MODE>::stage_bytes;
  constexpr uint32_t B_OFF = Ring<MODE>::a_planes * A_BYTES;  // B tile within a stage
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + RING_BYTES);
  volatile int* abort_flag = &ctl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  constexpr int BN = MODE == 0 ? GU_BN : DN_BN;
  const int num_m = (M + BM - 1) / BM;
  const int num_n = (Nout + BN - 1) / BN;
  const int num_tiles = num_m * num_n;
  const int nkb = (K + BK - 1) / BK;
  const unsigned my_err = MODE == 0 ? DEVERR_TIMEOUT_GATEUP : DEVERR_TIMEOUT_DOWN;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&ctl->full[s], 1);
      mbar_init(&ctl->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->tfull[b], 1);
      mbar_init(&ctl->tempty[b], 4);
    }
    mbar_init(&ctl->drain, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;

  auto fail = [&]() {
    if (!*abort_flag) {
      *abort_flag = 1;
      atomicOr(err, my_err);
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- TMA producer
      prefetch_tmap(&mapA);
      prefetch_tmap(&mapB0);
      if (MODE == 0) prefetch_tmap(&mapB1);
      if (MODE == 1) prefetch_tmap(&mapA2);
      uint32_t issued = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int m0 = (tile % num_m) * BM;
        const int n0 = (tile / num_m) * BN;
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = issued % STAGES;
          const uint32_t ph = (issued / STAGES) & 1u;
          if (!mbar_wait_bounded(&ctl->empty[s], ph ^ 1u, wait_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          uint8_t* sa = smem + s * STAGE_BYTES;
          uint8_t* sb = sa + B_OFF;
          mbar_arrive_expect_tx(&ctl->full[s], STAGE_BYTES);
          tma_load_2d(sa, &mapA, &ctl->full[s], kb * BK, m0);
          if (MODE == 1) tma_load_2d(sa + A_BYTES, &mapA2, &ctl->full[s], kb * BK, m0);
          if (MODE == 0) {
            tma_load_2d(sb, &mapB0, &ctl->full[s], kb * BK, n0);
            tma_load_2d(sb + B_BYTES / 2, &mapB1, &ctl->full[s], kb * BK, n0);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(sb + j * (B_BYTES / 4), &mapB0, &ctl->full[s], n0 + 64 * j, kb * BK);
          }
          ++issued;
        }
      }
      // every copy this thread started must land before the CTA can exit
      const uint32_t lo = issued > STAGES ? issued - STAGES : 0;
      for (uint32_t u = lo; u < issued; ++u) {
        volatile int never = 0;
        if (!mbar_wait_bounded(&ctl->full[u % STAGES], (u / STAGES) & 1u, DRAIN_NS, &never)) fail();
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer (one thread)
      constexpr uint32_t IDESC = idesc_bf16_f32(BM, 256, MODE == 1);
      uint32_t consumed = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++it) {
        const int buf = it & 1;
        if (!mbar_wait_bounded(&ctl->tempty[buf], ((it >> 1) & 1) ^ 1, wait_ns, abort_flag)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(buf * 256);
        for (int kb = 0; kb < nkb; ++kb) {
          const int s = consumed % STAGES;
          const uint32_t ph = (consumed / STAGES) & 1u;
          if (!mbar_wait_bounded(&ctl->full[s], ph, wait_ns, abort_flag)) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + s * STAGE_BYTES);
          const uint32_t sb = sa + B_OFF;
#pragma unroll
          for (int k = 0; k < BK / 16; ++k) {
            const uint64_t adesc = smem_desc_sw128(sa + 32u * k, 16u, 1024u);
            const uint64_t bdesc = MODE == 0 ? smem_desc_sw128(sb + 32u * k, 16u, 1024u)
                                             : smem_desc_sw128(sb + 2048u * k, B_BYTES / 4, 1024u);
            umma_f16(d_tmem, adesc, bdesc, IDESC, (kb > 0 || k > 0) ? 1u : 0u);
            if (MODE == 1)  // the lo plane against the same W2 tile
              umma_f16(d_tmem, smem_desc_sw128(sa + A_BYTES + 32u * k, 16u, 1024u), bdesc, IDESC, 1u);
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
      if (!mbar_wait_bounded(&ctl->drain, 0, DRAIN_NS, &never)) fail();
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int it = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
      const int buf = it & 1;
      bool ready = false;
      if (lane == 0) ready = mbar_wait_bounded(&ctl->tfull[buf], (it >> 1) & 1, wait_ns, abort_flag);
      ready = __shfl_sync(0xffffffffu, ready, 0);
      if (!ready) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after();
      const int m0 = (tile % num_m) * BM;
      const int n0 = (tile / num_m) * BN;
      const int row = m0 + 32 * q + lane;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(buf * 256);
      if (MODE == 0) {
#pragma unroll 1
        for (int c = 0; c < GU_BN; c += 32) {
          uint32_t gr[32], ur[32];
          tmem_ld32(taddr + c, gr);
          tmem_ld32(taddr + GU_BN + c, ur);
          tmem_ld_wait();
          float zv[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) zv[j] = silu_p(__uint_as_float(gr[j])) * __uint_as_float(ur[j]);
          const size_t zoff = static_cast<size_t>(row) * ldZ + n0 + c;
          uint4* zp = reinterpret_cast<uint4*>(Z + zoff);
          uint4* zlp = reinterpret_cast<uint4*>(Zlo + zoff);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float a = zv[8 * v + 2 * j], b = zv[8 * v + 2 * j + 1];
              hw[j] = pack_bf16x2(a, b);
              // z - hi is exact in fp32; its bf16 rounding leaves at most 2^-9 of it
              lw[j] = pack_bf16x2(a - bf16lo(hw[j]), b - bf16hi(hw[j]));
            }
            zp[v] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            zlp[v] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) zv[j] *= zv[j];
          // butterfly reduce-scatter over the 32 rows: lane l ends with column l's sum
#pragma unroll
          for (int w = 16; w >= 1; w >>= 1) {
            const bool upper = (lane & w) != 0;
#pragma unroll
            for (int j = 0; j < w; ++j) {
              const float send = upper ? zv[j] : zv[j + w];
              const float keep = upper ? zv[j + w] : zv[j];
              zv[j] = keep + __shfl_xor_sync(0xffffffffu, send, w);
            }
          }
          part[static_cast<size_t>((m0 >> 5) + q) * ldPart + n0 + c + lane] = zv[0];
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < DN_BN; c += 32) {
          uint32_t yr[32];
          tmem_ld32(taddr + c, yr);
          tmem_ld_wait();
          if (row < M) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const int d = n0 + c + 8 * v;
              if (d < Nout) {
                if (out_f32) {
                  float4* yp = reinterpret_cast<float4*>(static_cast<float*>(Y) + static_cast<size_t>(row) * Nout + d);
                  yp[0] = make_float4(__uint_as_float(yr[8 * v]), __uint_as_float(yr[8 * v + 1]),
                                      __uint_as_float(yr[8 * v + 2]), __uint_as_float(yr[8 * v + 3]));
                  yp[1] = make_float4(__uint_as_float(yr[8 * v + 4]), __uint_as_float(yr[8 * v + 5]),
                                      __uint_as_float(yr[8 * v + 6]), __uint_as_float(yr[8 * v + 7]));
                } else {
                  uint4* yp =
                      reinterpret_cast<uint4*>(static_cast<uint16_t*>(Y) + static_cast<size_t>(row) * Nout + d);
                  *yp = make_uint4(pack_bf16x2(__uint_as_float(yr[8 * v]), __uint_as_float(yr[8 * v + 1])),
                                   pack_bf16x2(__uint_as_float(yr[8 * v + 2]), __uint_as_float(yr[8 * v + 3])),
                                   pack_bf16x2(__uint_as_float(yr[8 * v + 4]), __uint_as_float(yr[8 * v + 5])),
                                   pack_bf16x2(__uint_as_float(yr[8 * v + 6]), __uint_as_float(yr[8 * v + 7])));
                }
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ------------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 2-D map: `inner` contiguous elements, `outer` rows `row_bytes` apart, box {box_in, box_out},
// 128-byte swizzle, out-of-range elements read as zero.
static bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                      uint32_t box_in, uint32_t box_out) {
  EncodeTiledFn fn = get_encode();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_in, box_out};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_weight_maps(PrefillMaps* m, const uint16_t* Wp, int D, int N) {
  const uint64_t rb = 3ull * D * 2;
  return encode_2d(&m->wg, Wp, D, N, rb, BK, GU_BN) && encode_2d(&m->w1, Wp + D, D, N, rb, BK, GU_BN) &&
         encode_2d(&m->w2, Wp + 2 * static_cast<size_t>(D), D, N, rb, 64, BK);
}

bool encode_x_map(CUtensorMap* m, const uint16_t* X, int M, int D) {
  return encode_2d(m, X, D, M, static_cast<uint64_t>(D) * 2, BK, BM);
}

bool encode_z_map(CUtensorMap* m, const uint16_t* Z, int M, int N, int ldZ) {
  return encode_2d(m, Z, N, M, static_cast<uint64_t>(ldZ) * 2, BK, BM);
}

bool encode_zrows_map(CUtensorMap* m, const uint16_t* zcp, int rows, int NP) {
  return encode_2d(m, zcp, static_cast<uint64_t>(2 * NP), static_cast<uint64_t>(rows > 0 ? rows : 1),
                   static_cast<uint64_t>(4 * NP), 64, 64);
}

bool encode_tokens_map(CUtensorMap* m, const void* base, int inner, int rows, int ld, int NP) {
  return encode_2d(m, base, static_cast<uint64_t>(inner), static_cast<uint64_t>(rows), static_cast<uint64_t>(ld) * 2,
                   64, static_cast<uint32_t>(NP));
}

// ------------------------------------------------------------------ launchers
cudaError_t launch_prefill_gateup(const CUtensorMap& x_map, const PrefillMaps& maps, int M, int N, int D,
                                  uint16_t* Z, uint16_t* Zlo, int ldZ, float* part, int ldPart, unsigned* err,
                                  uint64_t wait_ns, int num_sms, cudaStream_t st) {
  cudaError_t e =
      cudaFuncSetAttribute(k_prefill_gemm<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int tiles = ((M + BM - 1) / BM) * ((N + GU_BN - 1) / GU_BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  k_prefill_gemm<0><<<grid, THREADS, SMEM_BYTES, st>>>(x_map, x_map, maps.wg, maps.w1, M, N, D, Z, Zlo, ldZ, part,
                                                       ldPart, nullptr, 0, err, wait_ns);
  return cudaGetLastError();
}

cudaError_t launch_prefill_down(const CUtensorMap& z_map, const CUtensorMap& zlo_map, const PrefillMaps& maps,
                                int M, int N, int D, void* Y, int out_f32, unsigned* err, uint64_t wait_ns,
                                int num_sms, cudaStream_t st) {
  cudaError_t e =
      cudaFuncSetAttribute(k_prefill_gemm<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int tiles = ((M + BM - 1) / BM) * ((D + DN_BN - 1) / DN_BN);
  const int grid = tiles < num_sms ? tiles : num_sms;
  k_prefill_gemm<1><<<grid, THREADS, SMEM_BYTES, st>>>(z_map, zlo_map, maps.w2, maps.w2, M, D, N, nullptr, nullptr, 0,
                                                       nullptr, 0, Y, out_f32, err, wait_ns);
  return cudaGetLastError();
}

}  // namespace pop
