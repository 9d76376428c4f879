// Top-k selection over indexer scores: the step that produces the top-k lists the decode reads
// ("Inside the Decode Performance Investigation", The Setup: index_topk = 512 positions per query,
// with the indexer launches in the per-step kernel inventory).  Per query b: among positions
// 0 .. len_b - 1 keep the k of largest score, ranked by IEEE totalOrder with ties to the lower
// position, and write them in increasing position order; when len_b <= k keep every position and
// pad with -1.
//
// One thread-block cluster per query row.  The row is cut into csize contiguous chunks, one per CTA
// of the cluster, loaded once from HBM (16-byte streaming loads) into shared memory as 32-bit order
// keys.  Selection is a radix select in two stages; every decision is taken identically by every CTA
// of the cluster from sums that each CTA pushes into all the others' shared memory (remote reductions)
// before a cluster barrier, so after the barrier each CTA reads only its own shared memory, no CTA
// leads and nothing waits on a flag:
//   1. a coarse 8-bit bin that is monotone in the key (sign, exponent within a 32-octave window, two
//      mantissa bits), histogrammed while the chunk loads (per-warp histograms): bins above the one
//      holding the k-th key are kept whole, bins below are dropped;
//   2. the entries of that bin (the candidates, listed per warp) are refined digit by digit, starting
//      below the leading bits all candidates share (from the cluster's smallest and largest
//      candidate); the select stops as soon as a digit's bin is kept whole.
// The outcome is one threshold key; an order-preserving compaction (per-warp ballots, per-warp and
// per-CTA bases) writes the kept positions in position order.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkBins = 256;
constexpr int kTkRefinePasses = 4;   // at most 32 bits in 8-bit digits
constexpr int kTkLoadUnroll = 4;     // 16-byte loads in flight per thread
constexpr int kTkWarpCands = 512;    // candidate indexes listed per warp (16-bit, in the histogram space)
constexpr int kTkWindowLo = 111;     // biased exponent of the coarse window's lowest octave (2^-16)

struct TkShared {
  union {
    uint32_t whist[kTkWarps][kTkBins];       // per-warp coarse histograms while the chunk loads
    uint16_t cand[kTkWarps][kTkWarpCands];   // then: chunk indexes of each warp's candidates
  } u;
  // cluster-wide sums, accumulated by remote reductions from every CTA of the cluster
  uint32_t hist_c[kTkBins];                  // coarse histogram
  uint32_t hist[kTkRefinePasses][kTkBins];   // refinement histograms
  // this CTA's own refinement histograms (pushed into the sums above)
  uint32_t hloc[kTkRefinePasses][kTkBins];
  uint32_t cmin, cmax;                       // smallest and largest candidate key
  uint32_t peer_cnt[kTopkMaxCluster][2];     // per CTA: kept-for-sure entries, tie-class entries
  // this CTA only
  uint32_t wcand[kTkWarps];                  // candidates per warp
  uint32_t wcnt[2][kTkWarps];                // per warp: kept-for-sure entries, tie-class entries
  uint32_t wbase[2][kTkWarps];               // per warp: output base, tie-rank base
  uint32_t scan[kTkWarps];
  uint32_t overflow;                         // a warp listed more candidates than it holds
  uint32_t bc, need, done;
};

// IEEE totalOrder as unsigned integer order: a negative pattern has all its bits flipped, a positive
// one its sign bit set.
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

// Coarse bin of a key, monotone (non-decreasing) in the key: 128 + idx for a positive value, 127 - idx
// for a negative one, idx = 4 (exponent - 111) + top two mantissa bits clamped to [0, 127] (magnitudes
// below 2^-16 share idx 0, those from 2^16 up, with the infinities and NaNs, share idx 127).
__device__ __forceinline__ uint32_t coarse_bin(uint32_t key) {
  const bool pos = (key >> 31) != 0;
  const uint32_t mag = (pos ? key : ~key) & 0x7FFFFFFFu;
  int idx = (int)(mag >> 21) - 4 * kTkWindowLo;
  idx = idx < 0 ? 0 : idx > 127 ? 127 : idx;
  return pos ? 128u + (uint32_t)idx : 127u - (uint32_t)idx;
}

// Smallest key whose coarse bin is bc (coarse_bin is monotone, so bin bc is the key interval
// [coarse_lo(bc), coarse_lo(bc + 1) - 1]).
__device__ __forceinline__ uint32_t coarse_lo(uint32_t bc) {
  if (bc >= 128u) {  // positive values: the smallest magnitude of index bc - 128
    const uint32_t idx = bc - 128u;
    return idx == 0 ? 0x80000000u : (0x80000000u | ((idx + 4u * kTkWindowLo) << 21));
  }
  const uint32_t idx = 127u - bc;  // negative values: the largest magnitude of index 127 - bc
  if (idx == 127u) return 0u;
  const uint32_t mag = ((idx + 4u * kTkWindowLo + 1u) << 21) - 1u;
  return ~(0x80000000u | mag);
}

__device__ __forceinline__ uint32_t coarse_hi(uint32_t bc) { return bc == 255u ? 0xFFFFFFFFu : coarse_lo(bc + 1u) - 1u; }

// Remote reductions into the shared memory of CTA `rank` of the cluster (any CTA, this one included).
__device__ __forceinline__ void red_add_cluster(uint32_t saddr, uint32_t rank, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(mapa(saddr, rank)), "r"(v) : "memory");
}
__device__ __forceinline__ void red_min_cluster(uint32_t saddr, uint32_t rank, uint32_t v) {
  asm volatile("red.shared::cluster.min.u32 [%0], %1;" ::"r"(mapa(saddr, rank)), "r"(v) : "memory");
}
__device__ __forceinline__ void red_max_cluster(uint32_t saddr, uint32_t rank, uint32_t v) {
  asm volatile("red.shared::cluster.max.u32 [%0], %1;" ::"r"(mapa(saddr, rank)), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t saddr, uint32_t rank, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(mapa(saddr, rank)), "r"(v) : "memory");
}


// Adds the active lanes' bins to histogram h (this CTA's shared memory); the lanes sharing the first
// active lane's bin add with one atomic (a tie-heavy row puts whole warps in one bin).  Every lane of
// the warp calls it.
__device__ __forceinline__ void hist_add(uint32_t* h, bool active, uint32_t bin) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!act) return;
  const int leader = __ffs(act) - 1;
  const uint32_t lb = __shfl_sync(0xffffffffu, bin, leader);
  const unsigned same = __ballot_sync(0xffffffffu, active && bin == lb);
  if ((int)(threadIdx.x & 31) == leader) atomicAdd(h + lb, (uint32_t)__popc(same));
  else if (active && bin != lb) atomicAdd(h + bin, 1u);
}

// Every thread of the row's CTAs (the cluster), or of this CTA when the row has one.
__device__ __forceinline__ void row_barrier(int csize) {
  if (csize > 1) cluster_sync_all();
  else __syncthreads();
}

// Adds this CTA's 256-bin histogram `local` into the cluster-wide sum `sum` of every CTA of the
// cluster (thread t < 256 pushes bin t).
__device__ __forceinline__ void push_hist(const uint32_t* local, uint32_t* sum, int csize) {
  const int t = threadIdx.x;
  if (t < kTkBins) {
    const uint32_t v = local[t];
    if (csize == 1) {
      sum[t] += v;
    } else if (v != 0) {
      const uint32_t a = smem_u32(sum + t);
      for (int r = 0; r < csize; ++r) red_add_cluster(a, (uint32_t)r, v);
    }
  }
}

// Kept entries of the tie class among `e` entries, given `before` such entries at lower positions.
__device__ __forceinline__ uint32_t kept_ties(uint32_t before, uint32_t e, uint32_t need) {
  if (before >= need) return 0;
  return min(need - before, e);
}

// Finds in the cluster-wide histogram h the bin holding the need-th largest entry.  Threads 0..255
// take bins 255..0, so an inclusive scan in thread order sums the bins from the top.  The one thread
// whose bin it is writes s.bc (the bin), s.need (the rank within it) and s.done (the bin is kept
// whole).  All threads call it; it ends with a block barrier.
__device__ __forceinline__ void pick_bin(TkShared& s, const uint32_t* h, uint32_t need) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t g = 0, incl = 0;
  if (tid < kTkBins) {
    g = h[kTkBins - 1 - tid];
    incl = g;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s.scan[warp] = incl;
  }
  __syncthreads();
  if (tid < kTkBins) {
    for (int w = 0; w < warp; ++w) incl += s.scan[w];
    const uint32_t excl = incl - g;
    if (excl < need && need <= incl) {
      s.bc = (uint32_t)(kTkBins - 1 - tid);
      s.need = need - excl;
      s.done = (g == need - excl) ? 1u : 0u;
    }
  }
  __syncthreads();
}

// The final rule: an entry is kept for sure when all_kept or key > t, and is in the tie class (kept in
// position order while fewer than `need` of the class precede it) when ties && key == t.
struct TkRule {
  uint32_t t;
  bool all_kept, ties;
  __device__ __forceinline__ bool gt(uint32_t key) const { return all_kept || key > t; }
  __device__ __forceinline__ bool eq(uint32_t key) const { return ties && key == t; }
};

__global__ void __launch_bounds__(kTkThreads, 2) topk_kernel(TopkParams p) {
  extern __shared__ __align__(16) uint32_t keys[];
  TkShared& s = *reinterpret_cast<TkShared*>(keys + p.chunk);
  const int csize = p.csize;
  const int rank = csize > 1 ? (int)cluster_ctarank() : 0;
  const int b = blockIdx.x / csize;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  int len = __ldg(p.seq_lens + b);
  if (len < 0 || len > p.num_cols) {
    if (rank == 0 && tid == 0 && p.err) atomicOr(p.err, SMLA_DEVERR_LEN_RANGE);
    len = len < 0 ? 0 : p.num_cols;
  }
  const int c0 = rank * p.chunk;
  const int n = max(0, min(len - c0, p.chunk));
  int32_t* out = p.out + (size_t)b * p.k;

  // a short row keeps every position (the same branch in every CTA of the cluster)
  if (len <= p.k) {
    for (int i = tid; i < n; i += kTkThreads) out[c0 + i] = c0 + i;
    if (rank == 0)
      for (int i = len + tid; i < p.k; i += kTkThreads) out[i] = -1;
    return;
  }

  for (int i = tid; i < kTkWarps * kTkBins; i += kTkThreads) (&s.u.whist[0][0])[i] = 0;
  for (int i = tid; i < kTkBins; i += kTkThreads) s.hist_c[i] = 0;
  for (int i = tid; i < kTkRefinePasses * kTkBins; i += kTkThreads) {
    (&s.hist[0][0])[i] = 0;
    (&s.hloc[0][0])[i] = 0;
  }
  if (tid < 2 * kTopkMaxCluster) (&s.peer_cnt[0][0])[tid] = 0;
  if (tid == 0) {
    s.cmin = 0xFFFFFFFFu;
    s.cmax = 0;
    s.overflow = 0;
  }
  // the cluster's sums are zero everywhere before any CTA pushes into them; the barrier completes
  // while the chunk loads
  if (csize > 1) cluster_arrive_release();
  __syncthreads();

  // load the chunk as order keys, with the coarse histogram
  uint32_t* wh = s.u.whist[warp];
  const float* row = p.scores + (size_t)b * p.stride + c0;
  if (p.vec4) {
    const int n4 = n >> 2;
    for (int base = 0; base < n4; base += kTkThreads * kTkLoadUnroll) {
      uint4 v[kTkLoadUnroll];
#pragma unroll
      for (int u = 0; u < kTkLoadUnroll; ++u) {
        const int j = base + u * kTkThreads + tid;
        if (j < n4) v[u] = ldg_stream(row + 4 * j);
      }
#pragma unroll
      for (int u = 0; u < kTkLoadUnroll; ++u) {
        const int j = base + u * kTkThreads + tid;
        if (j < n4) {
          const uint4 kk = make_uint4(order_key(v[u].x), order_key(v[u].y), order_key(v[u].z), order_key(v[u].w));
          reinterpret_cast<uint4*>(keys)[j] = kk;
          atomicAdd(wh + coarse_bin(kk.x), 1u);
          atomicAdd(wh + coarse_bin(kk.y), 1u);
          atomicAdd(wh + coarse_bin(kk.z), 1u);
          atomicAdd(wh + coarse_bin(kk.w), 1u);
        }
      }
    }
    const int i = (n4 << 2) + tid;  // at most three scalar tail entries
    if (tid < (n & 3)) {
      const uint32_t kk = order_key(__float_as_uint(__ldg(row + i)));
      keys[i] = kk;
      atomicAdd(wh + coarse_bin(kk), 1u);
    }
  } else {
    for (int base = 0; base < n; base += kTkThreads * kTkLoadUnroll) {
      uint32_t v[kTkLoadUnroll];
#pragma unroll
      for (int u = 0; u < kTkLoadUnroll; ++u) {
        const int i = base + u * kTkThreads + tid;
        if (i < n) v[u] = __float_as_uint(__ldg(row + i));
      }
#pragma unroll
      for (int u = 0; u < kTkLoadUnroll; ++u) {
        const int i = base + u * kTkThreads + tid;
        if (i < n) {
          const uint32_t kk = order_key(v[u]);
          keys[i] = kk;
          atomicAdd(wh + coarse_bin(kk), 1u);
        }
      }
    }
  }
  __syncthreads();
  if (tid < kTkBins) {
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < kTkWarps; ++w) t += s.u.whist[w][tid];
    s.u.whist[0][tid] = t;  // this CTA's coarse histogram
  }
  if (csize > 1) cluster_wait();  // every CTA's sums are zeroed
  push_hist(s.u.whist[0], s.hist_c, csize);
  row_barrier(csize);  // the coarse sums are complete

  pick_bin(s, s.hist_c, (uint32_t)p.k);
  const uint32_t bc = s.bc;
  const uint32_t clo = coarse_lo(bc), chi = coarse_hi(bc);
  uint32_t need = s.need, prefix = 0;
  bool done = s.done != 0;

  if (!done) {
    // each warp lists its candidates (coarse bin bc: keys in [clo, chi]) from its contiguous segment;
    // the per-warp histograms are dead (summed above), so their space holds the lists
    const int seg = p.chunk / kTkWarps;
    const int s0 = warp * seg;
    const int s_end = min(seg, n - s0);  // warp-uniform; may be <= 0
    uint16_t* my = s.u.cand[warp];
    uint32_t cnt = 0, lo = 0xFFFFFFFFu, hi = 0;
    const unsigned below = (1u << lane) - 1u;
    for (int j0 = 0; j0 < s_end; j0 += 128) {  // warp-uniform; entries j0 + 32 q + lane, q = 0..3
      uint32_t kq[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = j0 + 32 * q + lane;
        kq[q] = j < s_end ? keys[s0 + j] : 0u;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = j0 + 32 * q + lane;
        const bool c = j < s_end && kq[q] >= clo && kq[q] <= chi;
        const unsigned cb = __ballot_sync(0xffffffffu, c);
        if (c) {
          const uint32_t at = cnt + (uint32_t)__popc(cb & below);
          if (at < (uint32_t)kTkWarpCands) my[at] = (uint16_t)(s0 + j);
          lo = min(lo, kq[q]);
          hi = max(hi, kq[q]);
        }
        cnt += (uint32_t)__popc(cb);
      }
    }
    lo = __reduce_min_sync(0xffffffffu, lo);
    hi = __reduce_max_sync(0xffffffffu, hi);
    if (lane == 0) {
      s.wcand[warp] = cnt;
      if (cnt > (uint32_t)kTkWarpCands) s.overflow = 1;
      if (cnt) {
        if (csize == 1) {
          atomicMin(&s.cmin, lo);
          atomicMax(&s.cmax, hi);
        } else {
          for (int r = 0; r < csize; ++r) {
            red_min_cluster(smem_u32(&s.cmin), (uint32_t)r, lo);
            red_max_cluster(smem_u32(&s.cmax), (uint32_t)r, hi);
          }
        }
      }
    }
    row_barrier(csize);  // the candidate key range is complete

    // every candidate shares the leading bits common to the smallest and largest one
    const uint32_t gmin = s.cmin, gmax = s.cmax;
    const int common = __clz(gmin ^ gmax);  // 32 when they are equal
    uint32_t mask = common == 0 ? 0u : common == 32 ? 0xFFFFFFFFu : (0xFFFFFFFFu << (32 - common));
    prefix = gmin & mask;
    const bool listed = s.overflow == 0;
    const uint32_t my_cnt = s.wcand[warp];
    int rest = 32 - common;
    for (int pass = 0; rest > 0 && !done; ++pass) {
      const int w = rest < 8 ? rest : 8;
      const int shift = rest - w;
      const uint32_t dmask = (1u << w) - 1u;
      uint32_t* hloc = s.hloc[pass];
      if (listed) {
        for (uint32_t c = lane; c < ((my_cnt + 31u) & ~31u); c += 32) {  // warp-uniform trip count
          const bool ok = c < my_cnt;
          const uint32_t kk = ok ? keys[my[c]] : 0u;
          hist_add(hloc, ok && (kk & mask) == prefix, (kk >> shift) & dmask);
        }
      } else {  // a warp's list overflowed: every warp scans its segment for candidates
        for (int j0 = 0; j0 < s_end; j0 += 32) {
          const int j = j0 + lane;
          const uint32_t kk = j < s_end ? keys[s0 + j] : 0u;
          hist_add(hloc, j < s_end && kk >= clo && kk <= chi && (kk & mask) == prefix, (kk >> shift) & dmask);
        }
      }
      __syncthreads();  // this CTA's digit histogram is complete
      push_hist(hloc, s.hist[pass], csize);
      row_barrier(csize);  // the digit sums are complete
      pick_bin(s, s.hist[pass], need);
      prefix |= s.bc << shift;
      mask |= dmask << shift;
      need = s.need;
      done = s.done != 0;
      rest -= w;
    }
  }

  // done: the kept entries are exactly the keys >= max(prefix, clo) (the bins above bc whole, and the
  // candidates from the prefix up); otherwise every bit is decided and prefix is the k-th key itself
  TkRule rule;
  if (done) {
    const uint32_t lo = prefix > clo ? prefix : clo;
    rule.all_kept = lo == 0;
    rule.t = lo - 1u;
    rule.ties = false;
  } else {
    rule.all_kept = false;
    rule.t = prefix;
    rule.ties = true;
  }

  // counts per warp segment (contiguous, a multiple of 32 entries): kept for sure, tie class
  const int seg = p.chunk / kTkWarps;
  const int s0 = warp * seg;
  const int s_end = min(seg, n - s0);  // warp-uniform; may be <= 0
  uint32_t c_gt = 0, c_eq = 0;
  for (int j0 = 0; j0 < s_end; j0 += 128) {
    uint32_t kq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + 32 * q + lane;
      kq[q] = j < s_end ? keys[s0 + j] : 0u;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bool ok = j0 + 32 * q + lane < s_end;
      c_gt += ok && rule.gt(kq[q]);
      c_eq += ok && rule.eq(kq[q]);
    }
  }
  c_gt = __reduce_add_sync(0xffffffffu, c_gt);
  c_eq = __reduce_add_sync(0xffffffffu, c_eq);
  if (lane == 0) {
    s.wcnt[0][warp] = c_gt;
    s.wcnt[1][warp] = c_eq;
  }
  __syncthreads();
  if (tid == 0) {
    uint32_t a = 0, e = 0;
    for (int w = 0; w < kTkWarps; ++w) {
      a += s.wcnt[0][w];
      e += s.wcnt[1][w];
    }
    // CTAs of higher rank (later positions) need this CTA's counts
    for (int r = rank + 1; r < csize; ++r) {
      st_cluster_u32(smem_u32(&s.peer_cnt[rank][0]), (uint32_t)r, a);
      st_cluster_u32(smem_u32(&s.peer_cnt[rank][1]), (uint32_t)r, e);
    }
  }
  if (csize > 1) cluster_sync_all();  // the counts of every lower-rank CTA are here (the last cluster-wide step)
  if (tid == 0) {
    uint32_t sel = 0, eq = 0;  // kept entries and tie entries at lower positions
    for (int r = 0; r < rank; ++r) {
      const uint32_t gt_r = s.peer_cnt[r][0], eq_r = s.peer_cnt[r][1];
      sel += gt_r + (rule.ties ? kept_ties(eq, eq_r, need) : 0u);
      eq += eq_r;
    }
    for (int w = 0; w < kTkWarps; ++w) {
      s.wbase[0][w] = sel;
      s.wbase[1][w] = eq;
      sel += s.wcnt[0][w] + (rule.ties ? kept_ties(eq, s.wcnt[1][w], need) : 0u);
      eq += s.wcnt[1][w];
    }
  }
  __syncthreads();

  // order-preserving write of this warp's kept positions
  uint32_t sel_base = s.wbase[0][warp], eq_base = s.wbase[1][warp];
  const unsigned below = (1u << lane) - 1u;
  for (int j0 = 0; j0 < s_end; j0 += 128) {  // warp-uniform; entries j0 + 32 q + lane, in position order
    uint32_t kq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + 32 * q + lane;
      kq[q] = j < s_end ? keys[s0 + j] : 0u;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = j0 + 32 * q + lane;
      const bool ok = j < s_end;
      const bool gt = ok && rule.gt(kq[q]), eq = ok && rule.eq(kq[q]);
      const unsigned eqb = __ballot_sync(0xffffffffu, eq);
      const bool keep = gt || (eq && eq_base + (uint32_t)__popc(eqb & below) < need);
      const unsigned keepb = __ballot_sync(0xffffffffu, keep);
      if (keep) {
        const uint32_t pos = sel_base + (uint32_t)__popc(keepb & below);
        if (pos < (uint32_t)p.k) out[pos] = c0 + s0 + j;
      }
      sel_base += (uint32_t)__popc(keepb);
      eq_base += (uint32_t)__popc(eqb);
    }
  }
}

}  // namespace

size_t topk_smem_bytes(int chunk) { return (size_t)chunk * 4 + sizeof(TkShared); }

// Cluster size and chunk for rows of num_cols positions: every candidate size 1 .. 8 whose chunk fits
// (9 .. 16 only for rows longer than 8 full chunks), scored by waves x per-CTA time, the latter fitted
// to measured sweeps on GB300 (about 4 us fixed, 0.5 ns per position of the chunk for its four passes,
// 3.5 us for the cluster-wide exchanges of a cluster of more than one CTA); ties keep the smaller
// cluster.  When some size keeps every CTA on an SM of its own, only such sizes are considered: the
// kernel is issue-bound, so two CTAs sharing an SM run at about half speed (B = 32 x 32768: 4-CTA
// clusters 12.4 us, 8-CTA clusters 13.1 us).
bool topk_plan(int batch, int num_cols, int sm_count, int forced_csize, int* csize, int* chunk) {
  double best_t = 0;
  int best_c = 0, best_chunk = 0;
  const bool long_rows = num_cols > kTopkPortableCluster * kTopkMaxChunk;
  bool one_per_sm = false;  // some admissible size puts at most one CTA on each SM
  for (int c = 1; c <= kTopkPortableCluster && forced_csize == 0 && !long_rows; ++c) {
    const int ch = ((num_cols + c - 1) / c + 511) / 512 * 512;
    if (ch <= kTopkMaxChunk && (long long)batch * c <= sm_count) one_per_sm = true;
  }
  for (int c = 1; c <= kTopkMaxCluster; ++c) {
    if (forced_csize > 0 && c != forced_csize) continue;
    if (forced_csize == 0 && c > kTopkPortableCluster && !long_rows) continue;
    if (one_per_sm && (long long)batch * c > sm_count) continue;
    const int ch = ((num_cols + c - 1) / c + 511) / 512 * 512;
    if (ch > kTopkMaxChunk) continue;
    if (forced_csize == 0 && c > 1 && (size_t)(c - 1) * ch >= (size_t)num_cols) continue;  // no empty CTA
    const size_t smem = topk_smem_bytes(ch) + 1024;
    int cps = (int)((228u * 1024u) / smem);
    cps = cps < 1 ? 1 : cps > 2 ? 2 : cps;  // two CTAs of 512 threads at most (launch bounds)
    const double waves = ceil((double)batch * c / ((double)sm_count * cps));
    const double t = waves * (4.0 + 0.5e-3 * ch + (c > 1 ? 3.5 : 0.0));
    if (best_c == 0 || t < best_t - 1e-9) {
      best_t = t;
      best_c = c;
      best_chunk = ch;
    }
  }
  if (best_c == 0) return false;
  *csize = best_c;
  *chunk = best_chunk;
  return true;
}

constexpr int kMaxDevices = 64;

// Kernel attributes of topk_kernel on the current device: set once per device (a per-device flag, read
// without a lock once set; the first call on a device configures it under the lock).
cudaError_t configure_topk(int dev) {
  static std::atomic<bool> configured[kMaxDevices];
  static std::mutex mu;
  if (dev >= 0 && dev < kMaxDevices && configured[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lock(mu);
  if (dev >= 0 && dev < kMaxDevices && configured[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)topk_smem_bytes(kTopkMaxChunk));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) configured[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

cudaError_t launch_topk(const TopkParams& p, int batch, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure_topk(dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(batch * p.csize));
  cfg.blockDim = dim3(kTkThreads);
  cfg.dynamicSmemBytes = topk_smem_bytes(p.chunk);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, topk_kernel, p);
}

}  // namespace smla
