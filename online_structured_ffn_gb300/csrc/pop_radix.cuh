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

// keys of the cut-off bin that the top-k ranks directly
constexpr int SEL_GATHER = 256;

template <int NTH>
struct RadixScratch {
  static_assert(NTH >= 64 && RADIX_BINS % NTH == 0, "whole warps, bins split evenly");
  uint32_t hist[RADIX_BINS];
  uint32_t wsum[NTH / 32];
  uint32_t bcast[4];
  uint32_t warp_tot[NTH / 32][3];
  uint32_t wmin[NTH / 32], wmax[NTH / 32], wcnt[NTH / 32];
  uint32_t gcnt;
  int gsel;
  uint32_t gkey[SEL_GATHER];
  int gidx[SEL_GATHER];
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
//
// The cut-off is found in one histogram pass: the top RADIX_BITS occupied bits of the key offsets
// split the keys into bins, a scan finds the bin holding the cut-off position, and, when that bin
// holds at most SEL_GATHER keys (the usual case: a few), its keys are gathered and ranked directly
// under the (key ascending, index descending) order. A fuller bin takes the general order statistic.
// The selected positions are written in ascending order by a warp-ballot compaction. Seven
// barriers in all on the usual path.
template <int NTH, class Sync, class Score>
__device__ bool select_step(int tid, Score score, float* memory, int n, int k, int period, bool update,
                            uint32_t* keys, int* S, RadixScratch<NTH>& sc, Sync sync) {
  constexpr int NW = NTH / 32;
  constexpr int U = 8;
  const int lane = tid & 31, warp = tid >> 5;
  const bool topk = update && k > 0;
  // fill the keys (and the memory); the whole-range bounds and the cleared histogram come with them
  uint32_t lo = 0xffffffffu, hi = 0u;
  for (int base = tid; base < n; base += NTH * U) {
    float v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * NTH;
      v[u] = i < n ? score(i) : 0.f;
    }
    if (period > 1) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = base + u * NTH;
        if (i < n) {
          v[u] += memory[i];
          memory[i] = update ? 0.f : v[u];
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = base + u * NTH;
      if (i < n) {
        const uint32_t kv = float_key(v[u]);
        keys[i] = kv;
        lo = min(lo, kv);
        hi = max(hi, kv);
      }
    }
  }
  if (topk && k < n) {
    for (int b = tid; b < RADIX_BINS; b += NTH) sc.hist[b] = 0u;
    if (tid == 0) sc.gcnt = 0u;
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
      sc.wmin[warp] = lo;
      sc.wmax[warp] = hi;
    }
  }
  sync();  // barrier 1
  if (!topk) return true;
  uint32_t vS = 0;
  int jS = n;
  if (k < n) {
    lo = 0xffffffffu;
    hi = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      lo = min(lo, sc.wmin[w]);
      hi = max(hi, sc.wmax[w]);
    }
    const uint32_t t = static_cast<uint32_t>(n - k);  // ascending position of the cut-off
    if (hi == lo) {
      // one key value: ascending order is descending index, position t is index n - 1 - t
      vS = lo;
      jS = k - 1;
    } else {
      const int bits = 32 - __clz(hi - lo);
      const int shift = bits > RADIX_BITS ? bits - RADIX_BITS : 0;
      for (int i = tid; i < n; i += NTH) atomicAdd(&sc.hist[(keys[i] - lo) >> shift], 1u);
      sync();  // barrier 2
      constexpr int PER = RADIX_BINS / NTH;
      uint32_t run = 0;
#pragma unroll
      for (int j = 0; j < PER; ++j) run += sc.hist[tid * PER + j];
      uint32_t incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (lane == 31) sc.wsum[warp] = incl;
      sync();  // barrier 3
      uint32_t before = incl - run;
#pragma unroll
      for (int w = 0; w < NW; ++w) before += w < warp ? sc.wsum[w] : 0u;
      if (t >= before && t < before + run) {
        uint32_t acc = before;
#pragma unroll
        for (int j = 0; j < PER; ++j) {
          const uint32_t c = sc.hist[tid * PER + j];
          if (t >= acc && t < acc + c) {
            sc.bcast[0] = static_cast<uint32_t>(tid * PER + j);
            sc.bcast[1] = acc;
            sc.bcast[2] = c;
          }
          acc += c;
        }
      }
      sync();  // barrier 4
      const uint32_t bin = sc.bcast[0], below = sc.bcast[1], cnt = sc.bcast[2];
      if (cnt <= static_cast<uint32_t>(SEL_GATHER)) {
        for (int i = tid; i < n; i += NTH) {
          const uint32_t kv = keys[i];
          if (((kv - lo) >> shift) == bin) {
            const uint32_t slot = atomicAdd(&sc.gcnt, 1u);
            if (slot < static_cast<uint32_t>(SEL_GATHER)) {
              sc.gkey[slot] = kv;
              sc.gidx[slot] = i;
            }
          }
        }
        sync();  // barrier 5
        const uint32_t want = t - below;
        for (uint32_t s = tid; s < cnt; s += NTH) {
          const uint32_t kv = sc.gkey[s];
          const int iv = sc.gidx[s];
          uint32_t rank = 0;
          for (uint32_t m = 0; m < cnt; ++m) {
            const uint32_t km = sc.gkey[m];
            rank += (km < kv || (km == kv && sc.gidx[m] > iv)) ? 1u : 0u;
          }
          if (rank == want) {
            sc.bcast[3] = kv;
            sc.gsel = iv;
          }
        }
        sync();  // barrier 6
        vS = sc.bcast[3];
        jS = sc.gsel;
      } else {
        uint32_t v;
        order_statistic<NTH>(tid, keys, n, t, sc, sync, v, jS);
        vS = v;
      }
    }
  }
  // ascending compaction: warp w owns a contiguous run of whole 32-key groups
  const int groups = (n + 31) / 32;
  const int g0 = warp * groups / NW, g1 = (warp + 1) * groups / NW;
  auto sel = [&](int i) {
    if (i >= n) return false;
    if (k >= n) return true;
    const uint32_t kv = keys[i];
    return kv > vS || (kv == vS && i <= jS);
  };
  uint32_t mine = 0;
  for (int g = g0; g < g1; ++g) mine += __popc(__ballot_sync(0xffffffffu, sel(32 * g + lane)));
  if (lane == 0) sc.wcnt[warp] = mine;
  sync();  // barrier 7
  uint32_t off = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) {
    const uint32_t c = sc.wcnt[w];
    off += w < warp ? c : 0u;
    tot += c;
  }
  if (tot != static_cast<uint32_t>(k)) return false;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int g = g0; g < g1; ++g) {
    const int i = 32 * g + lane;
    const bool b = sel(i);
    const uint32_t m = __ballot_sync(0xffffffffu, b);
    if (b) S[off + __popc(m & lt_mask)] = i;
    off += __popc(m);
  }
  return true;
}

}  // namespace pop
