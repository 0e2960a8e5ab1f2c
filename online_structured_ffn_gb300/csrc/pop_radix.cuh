// Block-level selection primitives shared by the partition, the top-k and the decode kernels.
//
// Elements are ordered by (key ascending, index descending): among equal keys the lower index is
// the larger, i.e. the more important one ("POP: Online Structural Pruning..." notes, Key design 1
// and 2 cut-offs, ties given to the lower channel index). Every cut-off is then one order
// statistic. It is found by a radix select over the keys' offsets from their minimum, 11 bits at
// a time from the top of the occupied range (so the first pass already spreads the keys), with a
// shared-memory histogram and a block scan per pass. The index among equal keys needs no extra
// pass unless the cut-off value itself is repeated.
//
// NTH is the number of participating threads (whole warps, NTH/32 <= 32); `tid` is the thread's
// index in that group and `sync()` a barrier over exactly that group.
#pragma once
#include <stdint.h>

#include "pop_device.cuh"

namespace pop {

constexpr int RADIX_BITS = 11;
constexpr int RADIX_BINS = 1 << RADIX_BITS;

template <int NTH>
struct RadixScratch {
  uint32_t hist[RADIX_BINS];
  uint32_t wsum[NTH / 32];
  uint32_t bcast[4];
  uint32_t warp_tot[NTH / 32][3];
};

// Block-wide exclusive scan of one value per thread (thread order); returns the total.
template <int NTH, class Sync>
__device__ uint32_t block_excl_scan(int tid, uint32_t v, uint32_t& total, RadixScratch<NTH>& sc, Sync sync) {
  constexpr int NW = NTH / 32;
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sc.wsum[warp] = incl;
  sync();
  if (warp == 0) {
    const uint32_t s = lane < NW ? sc.wsum[lane] : 0u;
    uint32_t in2 = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, in2, o);
      if (lane >= o) in2 += y;
    }
    if (lane < NW) sc.wsum[lane] = in2 - s;
    if (lane == 31) sc.bcast[3] = in2;
  }
  sync();
  const uint32_t r = sc.wsum[warp] + incl - v;
  total = sc.bcast[3];
  sync();
  return r;
}

// Ascending rank `t` among the participating elements of [0, n), by their value(i).
// Returns the value, and how many participants are below / equal to it.
template <int NTH, class Sync, class Val, class Part>
__device__ void radix_select(int tid, int n, uint32_t t, Val value, Part part, RadixScratch<NTH>& sc, Sync sync,
                             uint32_t& v_out, uint32_t& lt_out, uint32_t& eq_out) {
  // occupied range of the participating values
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int i = tid; i < n; i += NTH)
    if (part(i)) {
      const uint32_t kv = value(i);
      lo = min(lo, kv);
      hi = max(hi, kv);
    }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
    hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
  }
  const int lane = tid & 31, warp = tid >> 5;
  if (lane == 0) {
    sc.warp_tot[warp][0] = lo;
    sc.warp_tot[warp][1] = hi;
  }
  sync();
  lo = 0xffffffffu;
  hi = 0u;
  for (int w = 0; w < NTH / 32; ++w) {
    lo = min(lo, sc.warp_tot[w][0]);
    hi = max(hi, sc.warp_tot[w][1]);
  }
  sync();
  const uint32_t range = hi >= lo ? hi - lo : 0u;
  int shift = range ? (32 - __clz(range)) : 0;  // number of occupied bits
  uint32_t prefix = 0, pmask = 0, rank = t, lt = 0, eq = 0;
  if (shift == 0) {
    // every participant has the same value
    uint32_t cnt = 0;
    for (int i = tid; i < n; i += NTH) cnt += part(i) ? 1u : 0u;
    uint32_t tot;
    block_excl_scan<NTH>(tid, cnt, tot, sc, sync);
    v_out = lo;
    lt_out = 0;
    eq_out = tot;
    return;
  }
  while (shift > 0) {
    const int w = shift >= RADIX_BITS ? RADIX_BITS : shift;
    shift -= w;
    const uint32_t dmask = (1u << w) - 1u;
    for (int i = tid; i < RADIX_BINS; i += NTH) sc.hist[i] = 0;
    sync();
    for (int i = tid; i < n; i += NTH) {
      if (!part(i)) continue;
      const uint32_t off = value(i) - lo;
      if ((off & pmask) == prefix) atomicAdd(&sc.hist[(off >> shift) & dmask], 1u);
    }
    sync();
    // each thread owns a contiguous run of bins; scan the run sums over the block
    constexpr int PER = RADIX_BINS / NTH;
    const int nb = 1 << w;
    uint32_t run = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      const int b = tid * PER + j;
      run += b < nb ? sc.hist[b] : 0u;
    }
    uint32_t tot;
    const uint32_t before = block_excl_scan<NTH>(tid, run, tot, sc, sync);
    if (rank >= before && rank < before + run) {
      uint32_t acc = before;
#pragma unroll
      for (int j = 0; j < PER; ++j) {
        const int b = tid * PER + j;
        const uint32_t c = b < nb ? sc.hist[b] : 0u;
        if (rank >= acc && rank < acc + c) {
          sc.bcast[0] = static_cast<uint32_t>(b);
          sc.bcast[1] = acc;
          sc.bcast[2] = c;
        }
        acc += c;
      }
    }
    sync();
    prefix |= sc.bcast[0] << shift;
    pmask |= dmask << shift;
    rank -= sc.bcast[1];
    lt += sc.bcast[1];
    eq = sc.bcast[2];
    sync();
  }
  v_out = lo + prefix;
  lt_out = lt;
  eq_out = eq;
}

// Element at ascending position t of the order (key ascending, index descending) over keys[0, n):
// returns its key v and its index j.
template <int NTH, class Sync>
__device__ void order_statistic(int tid, const uint32_t* keys, int n, uint32_t t, RadixScratch<NTH>& sc, Sync sync,
                                uint32_t& v, int& j) {
  uint32_t lt, eq;
  radix_select<NTH>(
      tid, n, t, [&](int i) { return keys[i]; }, [](int) { return true; }, sc, sync, v, lt, eq);
  const uint32_t vv = v;
  if (eq == 1) {
    for (int i = tid; i < n; i += NTH)
      if (keys[i] == vv) sc.bcast[0] = static_cast<uint32_t>(i);
    sync();
    j = static_cast<int>(sc.bcast[0]);
    sync();
    return;
  }
  // among the eq elements equal to v, in descending index order take offset t - lt, i.e. the
  // ascending-index rank eq - 1 - (t - lt)
  const uint32_t want = eq - 1u - (t - lt);
  uint32_t jv, jlt, jeq;
  radix_select<NTH>(
      tid, n, want, [](int i) { return static_cast<uint32_t>(i); }, [&](int i) { return keys[i] == vv; }, sc, sync,
      jv, jlt, jeq);
  j = static_cast<int>(jv);
}

// Exclusive scan of three counters per thread (in thread order) over the group; returns totals.
template <int NTH, class Sync>
__device__ void block_scan3(int tid, const uint32_t (&c)[3], uint32_t (&excl)[3], uint32_t (&tot)[3],
                            RadixScratch<NTH>& sc, Sync sync) {
  constexpr int NW = NTH / 32;
  const int lane = tid & 31, warp = tid >> 5;
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
  sync();
  if (warp == 0) {
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      const uint32_t s = lane < NW ? sc.warp_tot[lane][a] : 0u;
      uint32_t in2 = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, in2, o);
        if (lane >= o) in2 += y;
      }
      if (lane < NW) sc.warp_tot[lane][a] = in2 - s;
      if (lane == 31) sc.bcast[a] = in2;
    }
  }
  sync();
#pragma unroll
  for (int a = 0; a < 3; ++a) {
    excl[a] = sc.warp_tot[warp][a] + incl[a] - c[a];
    tot[a] = sc.bcast[a];
  }
  sync();
}

// Top-k of one decode step over n candidate keys (optionally accumulating the periodic memory):
// writes the k selected positions, ascending, to S. Returns false if the count came out wrong.
// keys must hold n entries. score(i) is the candidate's score for this step.
template <int NTH, class Sync, class Score>
__device__ bool select_step(int tid, Score score, float* memory, int n, int k, int period, bool update,
                            uint32_t* keys, int* S, RadixScratch<NTH>& sc, Sync sync) {
  for (int i = tid; i < n; i += NTH) {
    float v = score(i);
    if (period > 1) {
      v += memory[i];
      memory[i] = update ? 0.f : v;
    }
    keys[i] = float_key(v);
  }
  sync();
  if (!update || k <= 0) return true;
  uint32_t vS = 0;
  int jS = n;
  if (k < n) order_statistic<NTH>(tid, keys, n, static_cast<uint32_t>(n - k), sc, sync, vS, jS);
  const int per = (n + NTH - 1) / NTH;
  const int i0 = min(n, tid * per);
  const int i1 = min(n, i0 + per);
  auto sel = [&](int i) {
    if (k >= n) return true;
    const uint32_t kv = keys[i];
    return kv > vS || (kv == vS && i <= jS);
  };
  uint32_t c[3] = {0, 0, 0};
  for (int i = i0; i < i1; ++i) c[0] += sel(i) ? 1u : 0u;
  uint32_t off[3], tot[3];
  block_scan3<NTH>(tid, c, off, tot, sc, sync);
  if (tot[0] != static_cast<uint32_t>(k)) return false;
  for (int i = i0; i < i1; ++i)
    if (sel(i)) S[off[0]++] = i;
  return true;
}

}  // namespace pop
