// Block-level selection primitives shared by the partition, the top-k and the fused decode step.
//
// Elements are ordered by (key ascending, index descending): among equal keys the lower index is
// the larger, i.e. the more important one ("POP: Online Structural Pruning..." notes, Key design 1
// and 2 cut-offs, with ties given to the lower channel index). Every cut-off is then one order
// statistic, found by an LSD-free radix select on 8-bit digits with warp-aggregated shared-memory
// histograms, followed by a radix select over the indices of the keys equal to it.
//
// NTH is the number of participating threads (whole warps, NTH/32 <= 32); `tid` is the thread's
// index in that group and `sync()` a barrier over exactly that group.
#pragma once
#include <stdint.h>

#include "pop_device.cuh"

namespace pop {

template <int NTH>
struct RadixScratch {
  uint32_t hist[256];
  uint32_t bcast[4];
  uint32_t warp_tot[NTH / 32][3];
};

// Ascending rank `t` among the participating elements of [0, n), reading bits top_shift+7 .. 0
// of value(i). Returns the value, and how many participants are below / equal to it.
template <int NTH, class Sync, class Val, class Part>
__device__ void radix_select(int tid, int n, uint32_t t, int top_shift, Val value, Part part, RadixScratch<NTH>& sc,
                             Sync sync, uint32_t& v_out, uint32_t& lt_out, uint32_t& eq_out) {
  const int lane = tid & 31;
  uint32_t prefix = 0, pmask = 0, rank = t, lt = 0, eq = 0;
  for (int shift = top_shift; shift >= 0; shift -= 8) {
    for (int i = tid; i < 256; i += NTH) sc.hist[i] = 0;
    if (tid == 0) sc.bcast[0] = sc.bcast[1] = sc.bcast[2] = 0;
    sync();
    for (int base = tid - lane; base < n; base += NTH) {
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
    sync();
    if (tid < 32) {
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
    sync();
    prefix |= sc.bcast[0] << shift;
    pmask |= 0xffu << shift;
    rank -= sc.bcast[1];
    lt += sc.bcast[1];
    eq = sc.bcast[2];
    sync();
  }
  v_out = prefix;
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
      tid, n, t, 24, [&](int i) { return keys[i]; }, [](int) { return true; }, sc, sync, v, lt, eq);
  // among the `eq` elements equal to v, in descending index order take offset t - lt, which is
  // the ascending-index rank eq - 1 - (t - lt)
  const uint32_t want = eq - 1u - (t - lt);
  const uint32_t vv = v;
  const int top = n > 65536 ? 24 : (n > 256 ? 8 : 0);
  uint32_t jv, jlt, jeq;
  radix_select<NTH>(
      tid, n, want, top, [](int i) { return static_cast<uint32_t>(i); }, [&](int i) { return keys[i] == vv; }, sc,
      sync, jv, jlt, jeq);
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
// keys_smem must hold n entries. score(i) is the candidate's score for this step.
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
