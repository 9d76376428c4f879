// Top-k selection over indexer scores: the step that produces the top-k lists the decode reads
// ("Inside the Decode Performance Investigation", The Setup: index_topk = 512 positions per query,
// with the indexer launches in the per-step kernel inventory).  Per query b: among positions
// 0 .. len_b - 1 keep the k of largest score, ranked by IEEE totalOrder with ties to the lower
// position, and write them in increasing position order; when len_b <= k keep every position and
// pad with -1.
//
// A row is cut into chunks of `chunk` positions, one per CTA; the CTAs of a row sit in one
// thread-block cluster.  With a power-of-two cluster size the rows are packed: a row of u chunks takes
// an aligned group of u' CTAs (u' = u rounded up to a power of two), the groups ordered by size, so a
// cluster holds one long row or several short ones and a ragged batch does not give every row a whole
// cluster.  Each warp streams its contiguous segment of the chunk from HBM once (16-byte streaming
// loads) as 32-bit order keys; shared memory keeps at most one byte per position (the key's top byte,
// when two CTAs still fit on an SM with it), so long chunks cost no occupancy.  Selection is a radix
// select in 11-, 11- and 10-bit digits: every decision is taken identically by every CTA of the row
// from digit histograms that each CTA adds into all the row's CTAs' shared memory (remote reductions)
// before a cluster barrier, so after the barrier each CTA reads only its own shared memory, no CTA
// leads and nothing waits on a flag:
//   1. the top digit (sign, exponent, two mantissa bits), histogrammed on the first pass: digits above
//      the one holding the k-th key are kept whole, digits below dropped;
//   2. each warp lists, in position order, the entries at or above that digit (the kept-for-sure
//      entries and the candidates) with their keys: from the key bytes, only the positions whose top
//      byte can reach the digit are read again (from L2); without them the whole segment is;
//   3. the candidates are refined digit by digit from the lists; the select stops as soon as a
//      digit's bin is kept whole.
// The outcome is one threshold key; per-warp counts over the lists, the counts of the row's lower CTAs
// (one more exchange) and ballots over the lists write the kept positions in position order.  A warp
// whose entries overflow its list reads its segment again from global memory at each of those steps.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstddef>
#include <mutex>

#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

constexpr int kTkThreads = 512;
constexpr int kTkWarps = kTkThreads / 32;
constexpr int kTkBins = 2048;          // 11-bit digits: key bits 31..21, then 20..10
constexpr int kTkLastBins = 1024;      // the last digit: key bits 9..0
constexpr int kTkLoadUnroll = 4;       // 16-byte (or 4-byte) loads in flight per thread
constexpr int kTkWarpList = 384;       // entries listed per warp (sized so that long chunks keep their key bytes)
constexpr int kTkMaxClass = 4;         // packed row groups of 1, 2, 4, 8 or 16 CTAs
constexpr int kTkRowsCached = 4;       // row lengths a thread keeps while the rows are packed
static_assert(kTkRowsCached * kTkThreads >= kTopkPackMaxRows, "every packed row's length fits the registers");
// launch-shape model of topk_plan (round numbers, checked against sweeps): us per wave, per chunk
// position (per CTA sharing the SM), per cluster
constexpr double kTkFixedUs = 4.0, kTkPosUs = 0.25e-3, kTkClusterUs = 3.0;

struct alignas(16) TkShared {
  // row-wide digit histograms, accumulated by remote reductions from every CTA of the row: the top
  // digit in [0], the second in [1], the last in [0] again (cleared once the top digit is picked)
  uint32_t hsum[2][kTkBins];
  union {
    uint32_t hloc[kTkBins];                  // this CTA's top-digit histogram while the chunk loads
    struct {                                 // then per warp, in position order:
      uint32_t key[kTkWarps][kTkWarpList];   //   the full order keys of the listed entries
      uint16_t idx[kTkWarps][kTkWarpList];   //   and their chunk indexes
    } l;
  } u;
  uint32_t wgt[kTkWarps], weq[kTkWarps];     // per warp: kept-for-sure entries, tie-class entries
  uint32_t wbase[2][kTkWarps];               // per warp: output base, tie-rank base
  uint32_t scan[kTkWarps];
  uint32_t peer_cnt[kTopkMaxCluster][2];     // per lower CTA of the row: kept-for-sure, tie-class entries
  uint32_t ncls[kTkMaxClass + 1];            // rows per packed group size
  int row_found, row_len;
  uint32_t bc, need, done;
};

// IEEE totalOrder as unsigned integer order: a negative pattern has all its bits flipped, a positive
// one its sign bit set.
__device__ __forceinline__ uint32_t order_key(uint32_t bits) {
  return (bits & 0x80000000u) ? ~bits : (bits | 0x80000000u);
}

// Remote reductions and stores into the shared memory of CTA `rank` of the cluster (this one included).
__device__ __forceinline__ void red_add_cluster(uint32_t saddr, uint32_t rank, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(mapa(saddr, rank)), "r"(v) : "memory");
}
__device__ __forceinline__ void st_cluster_u32(uint32_t saddr, uint32_t rank, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(mapa(saddr, rank)), "r"(v) : "memory");
}

// Every thread of the cluster, or of this CTA when the launch has no cluster.
__device__ __forceinline__ void row_sync(int csize) {
  if (csize > 1) cluster_sync_all();
  else __syncthreads();
}

// The row group a CTA works in: `gsz` CTAs of cluster ranks g0 .. g0 + gsz - 1, this CTA the sub-th.
struct TkGroup {
  int g0, gsz;
  // Adds v to bin `bin` of the histogram h in every CTA of the group.
  __device__ __forceinline__ void add(uint32_t* h, uint32_t bin, uint32_t v) const {
    if (gsz == 1) {
      atomicAdd(h + bin, v);
    } else {
      const uint32_t a = smem_u32(h + bin);
      for (int r = 0; r < gsz; ++r) red_add_cluster(a, (uint32_t)(g0 + r), v);
    }
  }
};

// Adds the active lanes' bins to histogram h of every CTA of the group; the lanes sharing the first
// active lane's bin add with one reduction (a tie-heavy row puts whole warps in one bin).  Every lane
// of the warp calls it.
__device__ __forceinline__ void hist_add(const TkGroup& grp, uint32_t* h, bool active, uint32_t bin) {
  const unsigned act = __ballot_sync(0xffffffffu, active);
  if (!act) return;
  const int leader = __ffs(act) - 1;
  const uint32_t lb = __shfl_sync(0xffffffffu, bin, leader);
  const unsigned same = __ballot_sync(0xffffffffu, active && bin == lb);
  if ((int)(threadIdx.x & 31) == leader) grp.add(h, lb, (uint32_t)__popc(same));
  else if (active && bin != lb) grp.add(h, bin, 1u);
}

// Kept entries of the tie class among `e` entries, given `before` such entries at lower positions.
__device__ __forceinline__ uint32_t kept_ties(uint32_t before, uint32_t e, uint32_t need) {
  if (before >= need) return 0;
  return min(need - before, e);
}

// Finds in the row-wide histogram h (NB bins) the bin holding the need-th largest entry.  Thread t
// takes bins NB - 1 - BPT t - i (i < BPT), so an inclusive scan in thread order sums the bins from the
// top.  The one thread whose bin it is writes s.bc (the bin), s.need (the rank within it) and s.done
// (the bin is kept whole).  All threads of the CTA call it; it ends with a block barrier.
template <int NB>
__device__ __forceinline__ void pick_bin(TkShared& s, const uint32_t* h, uint32_t need) {
  constexpr int BPT = NB / kTkThreads;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint32_t g[BPT], sum = 0;
#pragma unroll
  for (int i = 0; i < BPT; ++i) {
    g[i] = h[NB - 1 - BPT * tid - i];
    sum += g[i];
  }
  uint32_t incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s.scan[warp] = incl;
  __syncthreads();
  for (int w = 0; w < warp; ++w) incl += s.scan[w];
  uint32_t run = incl - sum;
  if (run < need && need <= incl) {
#pragma unroll
    for (int i = 0; i < BPT; ++i) {
      if (run < need && need <= run + g[i]) {
        s.bc = (uint32_t)(NB - 1 - BPT * tid - i);
        s.need = need - run;
        s.done = (g[i] == need - run) ? 1u : 0u;
      }
      run += g[i];
    }
  }
  __syncthreads();
}

// Adds this CTA's histogram `local` into the row-wide sum `sum` of every CTA of the group.
__device__ __forceinline__ void push_hist(const TkGroup& grp, const uint32_t* local, uint32_t* sum) {
  for (int bin = threadIdx.x; bin < kTkBins; bin += kTkThreads) {
    const uint32_t v = local[bin];
    if (grp.gsz == 1) sum[bin] = v;
    else if (v != 0) grp.add(sum, (uint32_t)bin, v);
  }
}

// The final rule: an entry is kept for sure when all_kept or key > t, and is in the tie class (kept in
// position order while fewer than `need` of the class precede it) when ties && key == t.
struct TkRule {
  uint32_t t;
  bool all_kept, ties;
  __device__ __forceinline__ bool gt(uint32_t key) const { return all_kept || key > t; }
  __device__ __forceinline__ bool eq(uint32_t key) const { return ties && key == t; }
};

// Length of row b clamped to [0, num_cols], and its packed group size class: log2 of the chunks it
// spans rounded up to a power of two (a row of at most one chunk, or none, has class 0).
__device__ __forceinline__ int clamp_len(const TopkParams& p, int len) {
  return len < 0 ? 0 : len > p.num_cols ? p.num_cols : len;
}
__device__ __forceinline__ int len_class(const TopkParams& p, int len) {
  const int u = (clamp_len(p, len) + p.chunk - 1) / p.chunk;
  return u <= 1 ? 0 : 32 - __clz(u - 1);
}

// Order key of score i of a row (a reread: L2 holds the rows just loaded).
__device__ __forceinline__ uint32_t key_at(const float* row, int i) {
  return order_key(__ldg(reinterpret_cast<const unsigned int*>(row) + i));
}

__global__ void __launch_bounds__(kTkThreads, 2) topk_kernel(TopkParams p) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  TkShared& s = *reinterpret_cast<TkShared*>(smem_raw);
  // with p.pre8: the top 8 bits of every position's key, after TkShared
  uint8_t* const pre8 = smem_raw + sizeof(TkShared);
  const int cs = p.csize;
  const int rank = cs > 1 ? (int)cluster_ctarank() : 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const unsigned below = (1u << lane) - 1u;

  // ---- the row of this CTA, its place in the row, and the row's CTAs (its group)
  int row = -1, sub = 0, raw_len = 0;
  TkGroup grp{rank, 1};
  if (!p.pack) {
    row = (int)blockIdx.x / cs;
    sub = rank;
    grp = TkGroup{0, cs};
    raw_len = __ldg(p.seq_lens + row);
  } else {
    // groups in decreasing size, rows in index order within a size: group starts are multiples of
    // their size, so no group crosses a cluster.  Every CTA reads all lengths once into registers
    // (packing is used for at most kTkRowsCached * kTkThreads rows).
    const int top = 31 - __clz(cs);
    if (tid <= kTkMaxClass) s.ncls[tid] = 0;
    if (tid == 0) s.row_found = -1;
    int lens_c[kTkRowsCached];
#pragma unroll
    for (int i = 0; i < kTkRowsCached; ++i) {
      const int b = i * kTkThreads + tid;
      lens_c[i] = b < p.batch ? __ldg(p.seq_lens + b) : 0;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kTkRowsCached; ++i) {
      if (i * kTkThreads >= p.batch) break;  // block-uniform
      const int b = i * kTkThreads + tid;
      const int len_b = lens_c[i];
      const int c = b < p.batch ? len_class(p, len_b) : -1;
      for (int j = 0; j <= top; ++j) {
        const unsigned m = __ballot_sync(0xffffffffu, c == j);
        if (lane == 0 && m) atomicAdd(&s.ncls[j], (uint32_t)__popc(m));
      }
    }
    __syncthreads();
    const uint32_t g = blockIdx.x;
    uint32_t off = 0, my_off = 0;
    int my_cls = -1;
    for (int j = top; j >= 0; --j) {
      const uint32_t span = s.ncls[j] << j;
      if (my_cls < 0 && g < off + span) {
        my_cls = j;
        my_off = off;
      }
      off += span;
    }
    if (g - (uint32_t)rank >= off) return;  // the whole cluster lies past the packed rows
    if (my_cls >= 0) {
      grp.gsz = 1 << my_cls;
      sub = (int)((g - my_off) & (uint32_t)(grp.gsz - 1));
      grp.g0 = rank - sub;
      const uint32_t q = (g - my_off) >> my_cls;  // rank of the row among the rows of its class
      uint32_t seen = 0;
#pragma unroll
      for (int i = 0; i < kTkRowsCached; ++i) {
        if (i * kTkThreads >= p.batch) break;  // block-uniform
        const int b = i * kTkThreads + tid;
        const int len_b = lens_c[i];
        const bool is = b < p.batch && len_class(p, len_b) == my_cls;
        const unsigned m = __ballot_sync(0xffffffffu, is);
        if (lane == 0) s.scan[warp] = (uint32_t)__popc(m);
        __syncthreads();
        uint32_t before = seen;
        for (int w = 0; w < kTkWarps; ++w) {
          if (w < warp) before += s.scan[w];
          seen += s.scan[w];
        }
        if (is && before + (uint32_t)__popc(m & below) == q) {
          s.row_found = b;
          s.row_len = len_b;
        }
        __syncthreads();
        if (s.row_found >= 0) break;
      }
      row = s.row_found;
      raw_len = s.row_len;
    }
  }

  int len = 0;
  if (row >= 0) {
    len = clamp_len(p, raw_len);
    if (len != raw_len && sub == 0 && tid == 0 && p.err) atomicOr(p.err, SMLA_DEVERR_LEN_RANGE);
  }
  const int c0 = sub * p.chunk;
  const int n = row >= 0 ? max(0, min(len - c0, p.chunk)) : 0;
  int32_t* out = p.out + (size_t)(row >= 0 ? row : 0) * p.k;
  const float* row_src = p.scores + (size_t)(row >= 0 ? row : 0) * p.stride;
  const bool active = row >= 0 && len > p.k;

  // a short row keeps every position
  if (row >= 0 && !active) {
    for (int i = tid; i < n; i += kTkThreads) out[c0 + i] = c0 + i;
    if (sub == 0)
      for (int i = len + tid; i < p.k; i += kTkThreads) out[i] = -1;
  }
  // a cluster holding one row takes every decision below uniformly; one that holds several rows (or
  // idle CTAs) runs every exchange, each row skipping the work it does not need
  const bool uniform = grp.gsz == cs && row >= 0;
  if (uniform && !active) return;

  // the row-wide sums are zero everywhere before any CTA pushes into them; the barrier completes while
  // the chunk loads
  if (active) {
    uint4* z = reinterpret_cast<uint4*>(&s.hsum[0][0]);
    constexpr int kZero = (2 * kTkBins + kTkBins) / 4;  // hsum and hloc
    static_assert(offsetof(TkShared, u) == offsetof(TkShared, hsum) + sizeof(uint32_t) * 2 * kTkBins,
                  "hloc follows hsum");
    for (int i = tid; i < kZero; i += kTkThreads) z[i] = make_uint4(0, 0, 0, 0);
  }
  if (cs > 1) cluster_arrive_release();
  __syncthreads();

  // ---- first pass over the warp's segment of the chunk (HBM): the top-digit histogram
  // the CTA's n positions in 16 contiguous segments of whole 128-entry steps (a short chunk spreads
  // over every warp, so that no warp lists more than its share)
  const int seg = ((n + kTkWarps - 1) / kTkWarps + 127) & ~127;
  const int s0 = warp * seg;
  const int s_len = max(0, min(seg, n - s0));  // warp-uniform
  const float* src = row_src + c0 + s0;         // this warp's segment
  if (active) {
    uint32_t* h = s.u.hloc;
    if (p.vec4) {
      const int n4 = s_len >> 2;
      for (int base = 0; base < n4; base += 32 * kTkLoadUnroll) {
        uint4 v[kTkLoadUnroll];
#pragma unroll
        for (int u = 0; u < kTkLoadUnroll; ++u) {
          const int j = base + 32 * u + lane;
          if (j < n4) v[u] = ldg_stream(src + 4 * j);
        }
#pragma unroll
        for (int u = 0; u < kTkLoadUnroll; ++u) {
          const int j = base + 32 * u + lane;
          if (j < n4) {
            const uint32_t k0 = order_key(v[u].x), k1 = order_key(v[u].y), k2 = order_key(v[u].z),
                           k3 = order_key(v[u].w);
            atomicAdd(h + (k0 >> 21), 1u);
            atomicAdd(h + (k1 >> 21), 1u);
            atomicAdd(h + (k2 >> 21), 1u);
            atomicAdd(h + (k3 >> 21), 1u);
            if (p.pre8)  // the four top bytes, in position order
              *reinterpret_cast<uint32_t*>(pre8 + s0 + 4 * j) =
                  __byte_perm(__byte_perm(k0, k1, 0x0073), __byte_perm(k2, k3, 0x0073), 0x5410);
          }
        }
      }
      if (lane < (s_len & 3)) {  // scalar tail
        const uint32_t kk = key_at(src, (n4 << 2) + lane);
        atomicAdd(h + (kk >> 21), 1u);
        if (p.pre8) pre8[s0 + (n4 << 2) + lane] = (uint8_t)(kk >> 24);
      }
    } else {
      for (int base = 0; base < s_len; base += 32 * kTkLoadUnroll) {
        uint32_t v[kTkLoadUnroll];
#pragma unroll
        for (int u = 0; u < kTkLoadUnroll; ++u) {
          const int i = base + 32 * u + lane;
          if (i < s_len) v[u] = __ldg(reinterpret_cast<const unsigned int*>(src) + i);
        }
#pragma unroll
        for (int u = 0; u < kTkLoadUnroll; ++u)
          if (base + 32 * u + lane < s_len) {
            const uint32_t kk = order_key(v[u]);
            atomicAdd(h + (kk >> 21), 1u);
            if (p.pre8) pre8[s0 + base + 32 * u + lane] = (uint8_t)(kk >> 24);
          }
      }
    }
  }
  __syncthreads();
  if (cs > 1) cluster_wait();  // every CTA's sums are zeroed
  if (active) push_hist(grp, s.u.hloc, s.hsum[0]);
  row_sync(cs);  // the row's top-digit sums are complete (and hloc is read: the lists take its space)

  uint32_t need = (uint32_t)p.k, prefix = 0, mask = 0;
  bool done = false;
  if (active) {
    pick_bin<kTkBins>(s, s.hsum[0], need);
    prefix = s.bc << 21;
    mask = 0xFFE00000u;
    need = s.need;
    done = s.done != 0;
    // clear the top-digit sums for the last digit (before the next cluster barrier)
    for (int i = tid; i < kTkBins / 4; i += kTkThreads)
      reinterpret_cast<uint4*>(s.hsum[0])[i] = make_uint4(0, 0, 0, 0);
  }

  // ---- second pass (L2): list this warp's entries >= prefix in position order, with their keys
  uint32_t my_cnt = 0;  // entries of this warp at or above prefix (the list holds the first kTkWarpList)
  uint32_t* lk = s.u.l.key[warp];
  uint16_t* li = s.u.l.idx[warp];
  // appends this lane's entries e0 + i (raw score bits x[i]) whose hit[i] is set, after those of the
  // lower lanes (a run of consecutive positions, four a lane, lane-major); every lane calls it
  auto append4 = [&](const uint32_t (&x)[4], const bool (&hit)[4], int e0) {
    if (!__any_sync(0xffffffffu, hit[0] || hit[1] || hit[2] || hit[3])) return;
    unsigned m[4];
    uint32_t at = my_cnt, total = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m[i] = __ballot_sync(0xffffffffu, hit[i]);
      at += (uint32_t)__popc(m[i] & below);
      total += (uint32_t)__popc(m[i]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (hit[i]) {
        if (at < (uint32_t)kTkWarpList) {
          lk[at] = order_key(x[i]);
          li[at] = (uint16_t)(e0 + i);
        }
        ++at;
      }
    my_cnt += total;
  };
  // order_key(x) >= prefix as one compare on the raw bits x: with prefix in the positive half, x read
  // as a signed integer reaches prefix's magnitude bits; otherwise x (unsigned) is at most ~prefix
  const bool pos_lo = (prefix >> 31) != 0;
  const int lo_s = (int)(prefix & 0x7FFFFFFFu);
  const uint32_t lo_u = ~prefix;
  auto reach = [&](uint32_t x) { return pos_lo ? (int)x >= lo_s : x <= lo_u; };
  bool streamed = !p.pre8;  // the listing reads the whole segment again (no key bytes, or too many candidates)
  if (active && p.pre8) {
    // candidates: positions whose top key byte reaches prefix's (a superset of the entries >= prefix),
    // listed in position order; lane l takes 16 consecutive positions per step
    // byte b >= t (t = prefix's top byte) four bytes at a time: (b & 0x7F) + 0x80 - (t & 0x7F) sets the
    // byte's top bit exactly when b & 0x7F >= t & 0x7F (no carry leaves the byte); combined with b's own
    // top bit by AND when t >= 0x80 (b must be at least 0x80 too) and by OR otherwise
    const uint32_t t8 = prefix >> 24;
    const uint32_t add = (0x80u - (t8 & 0x7Fu)) * 0x01010101u;
    const bool t_hi = t8 >= 0x80u;
    auto reach4 = [&](uint32_t w) {
      const uint32_t y = (w & 0x7F7F7F7Fu) + add;
      return (t_hi ? (y & w) : (y | w)) & 0x80808080u;
    };
    // the four flags of a word (bits 7, 15, 23, 31) as a nibble
    auto nibble = [](uint32_t y) { return (((y >> 7) * 0x00204081u) >> 21) & 0xFu; };
    uint32_t ncand = 0;
    for (int j0 = 0; j0 < s_len; j0 += 512) {  // warp-uniform
      const int j = j0 + 16 * lane;
      uint32_t y[4] = {0u, 0u, 0u, 0u};
      if (j < s_len) {
        const uint4 b = *reinterpret_cast<const uint4*>(pre8 + s0 + j);
        y[0] = reach4(b.x);
        y[1] = reach4(b.y);
        y[2] = reach4(b.z);
        y[3] = reach4(b.w);
      }
      if (!__any_sync(0xffffffffu, (y[0] | y[1] | y[2] | y[3]) != 0u)) continue;
      uint32_t m = nibble(y[0]) | (nibble(y[1]) << 4) | (nibble(y[2]) << 8) | (nibble(y[3]) << 12);
      const int lim = s_len - j;  // bit i: position j + i is a candidate (positions below s_len only)
      if (lim < 16) m &= lim > 0 ? (1u << lim) - 1u : 0u;
      const uint32_t c = (uint32_t)__popc(m);
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
      uint32_t at = ncand + incl - c;
      while (m) {
        const int i = __ffs(m) - 1;
        m &= m - 1;
        if (at < (uint32_t)kTkWarpList) li[at] = (uint16_t)(s0 + j + i);
        ++at;
      }
      ncand += total;
    }
    __syncwarp();
    if (ncand <= (uint32_t)kTkWarpList) {
      // resolve the candidates (their scores from L2, 128 in flight per warp), keeping the entries >=
      // prefix, compacted in place in position order
      for (uint32_t b0 = 0; b0 < ncand; b0 += 128) {  // warp-uniform
        uint32_t x[4], ix[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t c = b0 + 32 * q + lane;
          ix[q] = c < ncand ? li[c] : 0u;
          x[q] = c < ncand ? __ldg(reinterpret_cast<const unsigned int*>(row_src + c0) + ix[q]) : 0u;
        }
        __syncwarp();  // every candidate of this step is read before the compacted writes
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const bool hit = b0 + 32 * q + lane < ncand && reach(x[q]);
          const unsigned hm = __ballot_sync(0xffffffffu, hit);
          if (hit) {
            const uint32_t at = my_cnt + (uint32_t)__popc(hm & below);
            lk[at] = order_key(x[q]);
            li[at] = (uint16_t)ix[q];
          }
          my_cnt += (uint32_t)__popc(hm);
        }
        __syncwarp();
      }
    } else {
      streamed = true;
    }
  }
  if (active && streamed) {
    if (p.vec4) {
      const int n4 = s_len >> 2;
      for (int base = 0; base < n4; base += 32 * kTkLoadUnroll) {  // warp-uniform
        uint4 v[kTkLoadUnroll];
        bool ok[kTkLoadUnroll];
#pragma unroll
        for (int u = 0; u < kTkLoadUnroll; ++u) {
          const int j = base + 32 * u + lane;
          ok[u] = j < n4;
          if (ok[u]) v[u] = ldg_stream(src + 4 * j);
        }
#pragma unroll
        for (int u = 0; u < kTkLoadUnroll; ++u) {
          const int j = base + 32 * u + lane;
          const uint32_t x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          const bool hit[4] = {ok[u] && reach(x[0]), ok[u] && reach(x[1]), ok[u] && reach(x[2]),
                               ok[u] && reach(x[3])};
          append4(x, hit, s0 + 4 * j);
        }
      }
      // scalar tail: at most three entries, one a lane, after every quad
      const int i = (n4 << 2) + lane;
      const bool ok = lane < (s_len & 3);
      const uint32_t xt = ok ? __ldg(reinterpret_cast<const unsigned int*>(src) + i) : 0u;
      const uint32_t x[4] = {xt, 0u, 0u, 0u};
      const bool hit[4] = {ok && reach(xt), false, false, false};
      append4(x, hit, s0 + i);
    } else {
      for (int base = 0; base < s_len; base += 32 * kTkLoadUnroll) {  // warp-uniform
        uint32_t v[kTkLoadUnroll];
        bool okv[kTkLoadUnroll];
#pragma unroll
        for (int u = 0; u < kTkLoadUnroll; ++u) {
          const int i = base + 32 * u + lane;
          okv[u] = i < s_len;
          if (okv[u]) v[u] = __ldg(reinterpret_cast<const unsigned int*>(src) + i);
        }
#pragma unroll
        for (int u = 0; u < kTkLoadUnroll; ++u) {
          const int i = base + 32 * u + lane;
          const uint32_t x[4] = {v[u], 0u, 0u, 0u};
          const bool hit[4] = {okv[u] && reach(v[u]), false, false, false};
          append4(x, hit, s0 + i);
        }
      }
    }
    __syncwarp();
  }
  const bool listed = my_cnt <= (uint32_t)kTkWarpList;
  const uint32_t* lkey = lk;
  const uint16_t* lidx = li;

  // ---- refine the candidates: digit 2 (key bits 20..10) into hsum[1], digit 3 (bits 9..0) into hsum[0]
#pragma unroll 1
  for (int step = 0; step < 2; ++step) {
    if (uniform && done) break;  // cluster-uniform (a single row decides identically everywhere)
    const int shift = step == 0 ? 10 : 0;
    const uint32_t dmask = step == 0 ? 0x7FFu : 0x3FFu;
    uint32_t* h = s.hsum[step == 0 ? 1 : 0];
    if (active && !done) {
      if (listed) {
        for (uint32_t c = lane; c < ((my_cnt + 31u) & ~31u); c += 32) {  // warp-uniform trip count
          const bool ok = c < my_cnt;
          const uint32_t kk = ok ? lkey[c] : 0u;
          hist_add(grp, h, ok && (kk & mask) == prefix, (kk >> shift) & dmask);
        }
      } else {  // the list overflowed: read the segment again
        for (int j0 = 0; j0 < s_len; j0 += 128) {
          uint32_t kq[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int j = j0 + 32 * q + lane;
            kq[q] = j < s_len ? key_at(src, j) : 0u;
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            hist_add(grp, h, j0 + 32 * q + lane < s_len && (kq[q] & mask) == prefix, (kq[q] >> shift) & dmask);
        }
      }
    }
    row_sync(cs);  // the digit sums are complete
    if (active && !done) {
      if (step == 0) pick_bin<kTkBins>(s, h, need);
      else pick_bin<kTkLastBins>(s, h, need);
      prefix |= s.bc << shift;
      mask |= dmask << shift;
      need = s.need;
      done = s.done != 0;
    }
  }

  // done: the kept entries are exactly the keys >= prefix (the bins above each chosen digit whole,
  // and the last chosen bin whole); otherwise every bit is decided and prefix is the k-th key itself
  TkRule rule;
  if (done) {
    rule.all_kept = prefix == 0;
    rule.t = prefix - 1u;
    rule.ties = false;
  } else {
    rule.all_kept = false;
    rule.t = prefix;
    rule.ties = true;
  }

  // ---- per-warp counts: kept for sure, tie class
  if (active) {
    uint32_t c_gt = 0, c_eq = 0;
    if (listed) {
      for (uint32_t c = lane; c < my_cnt; c += 32) {
        const uint32_t kk = lkey[c];
        c_gt += rule.gt(kk);
        c_eq += rule.eq(kk);
      }
    } else {
      for (int j = lane; j < s_len; j += 32) {
        const uint32_t kk = key_at(src, j);
        c_gt += rule.gt(kk);
        c_eq += rule.eq(kk);
      }
    }
    c_gt = __reduce_add_sync(0xffffffffu, c_gt);
    c_eq = __reduce_add_sync(0xffffffffu, c_eq);
    if (lane == 0) {
      s.wgt[warp] = c_gt;
      s.weq[warp] = c_eq;
    }
  }
  __syncthreads();
  if (active && tid == 0 && grp.gsz > 1) {
    uint32_t a = 0, e = 0;
    for (int w = 0; w < kTkWarps; ++w) {
      a += s.wgt[w];
      e += s.weq[w];
    }
    // the row's CTAs at later positions need this CTA's counts
    for (int r = sub + 1; r < grp.gsz; ++r) {
      st_cluster_u32(smem_u32(&s.peer_cnt[sub][0]), (uint32_t)(grp.g0 + r), a);
      st_cluster_u32(smem_u32(&s.peer_cnt[sub][1]), (uint32_t)(grp.g0 + r), e);
    }
  }
  if (cs > 1) cluster_sync_all();  // the counts of every lower CTA of the row are here (the last exchange)
  if (!active) return;
  if (tid == 0) {
    uint32_t sel = 0, eq = 0;  // kept entries and tie entries at lower positions
    for (int r = 0; r < sub; ++r) {
      const uint32_t gt_r = s.peer_cnt[r][0], eq_r = s.peer_cnt[r][1];
      sel += gt_r + (rule.ties ? kept_ties(eq, eq_r, need) : 0u);
      eq += eq_r;
    }
    for (int w = 0; w < kTkWarps; ++w) {
      s.wbase[0][w] = sel;
      s.wbase[1][w] = eq;
      sel += s.wgt[w] + (rule.ties ? kept_ties(eq, s.weq[w], need) : 0u);
      eq += s.weq[w];
    }
  }
  __syncthreads();

  // ---- order-preserving write of this warp's kept positions
  uint32_t sel_base = s.wbase[0][warp], eq_base = s.wbase[1][warp];
  const uint32_t trips = listed ? my_cnt : (uint32_t)s_len;
  for (uint32_t c0w = 0; c0w < trips; c0w += 128) {  // warp-uniform; entries in position order
    uint32_t kq[4], iq[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t c = c0w + 32 * q + lane;
      const bool ok = c < trips;
      iq[q] = ok ? (listed ? (uint32_t)lidx[c] : (uint32_t)s0 + c) : 0u;
      kq[q] = ok ? (listed ? lkey[c] : key_at(row_src + c0, (int)iq[q])) : 0u;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const bool ok = c0w + 32 * q + lane < trips;
      const bool gt = ok && rule.gt(kq[q]), eq = ok && rule.eq(kq[q]);
      const unsigned eqb = __ballot_sync(0xffffffffu, eq);
      const bool keep = gt || (eq && eq_base + (uint32_t)__popc(eqb & below) < need);
      const unsigned keepb = __ballot_sync(0xffffffffu, keep);
      if (keep) {
        const uint32_t pos = sel_base + (uint32_t)__popc(keepb & below);
        if (pos < (uint32_t)p.k) out[pos] = c0 + (int)iq[q];
      }
      sel_base += (uint32_t)__popc(keepb);
      eq_base += (uint32_t)__popc(eqb);
    }
  }
}

}  // namespace

// One byte per position (the top 8 bits of its key) joins the shared memory when two CTAs still fit on
// an SM with it.
bool topk_key_bytes(int chunk) { return 2 * (sizeof(TkShared) + (size_t)chunk + 1024) <= 228u * 1024u; }

size_t topk_smem_bytes(int chunk) { return sizeof(TkShared) + (topk_key_bytes(chunk) ? (size_t)chunk : 0); }


// Clusters of c CTAs (c = 1 .. 16) resident at once on a 152-SM GB300 with one or two 512-thread CTAs
// per SM (cudaOccupancyMaxActiveClusters; a cluster's CTAs share one GPC).
constexpr int kClustersPerWave[2][kTopkMaxCluster] = {
    {152, 76, 46, 36, 28, 23, 15, 15, 15, 13, 8, 8, 7, 7, 7, 7},
    {304, 152, 97, 74, 58, 46, 38, 36, 30, 28, 23, 23, 19, 14, 14, 14}};

// Cluster size and chunk for rows of num_cols positions: every candidate size 1 .. 8 whose chunk fits
// (16 for rows longer than 8 full chunks), scored as full rows (one row per cluster) by waves x
// per-wave time: a fixed part, a part per position of the chunk times the CTAs sharing an SM, and the
// cluster-wide exchanges of a cluster of more than one CTA (round constants, checked against measured
// sweeps of every cluster size on GB300: the model's pick is the fastest measured size on each of the
// decode workloads' shapes); ties keep the smaller cluster.  Chunks are multiples of kTopkChunkAlign positions (every warp a segment
// of whole 128-entry steps).
bool topk_plan(int batch, int num_cols, int sm_count, int forced_csize, int* csize, int* chunk) {
  double best_t = 0;
  int best_c = 0, best_chunk = 0;
  const bool long_rows = num_cols > kTopkPortableCluster * kTopkMaxChunk;
  auto chunk_for = [&](int c) { return ((num_cols + c - 1) / c + kTopkChunkAlign - 1) / kTopkChunkAlign * kTopkChunkAlign; };
  for (int c = 1; c <= kTopkMaxCluster; ++c) {
    if (forced_csize > 0 && c != forced_csize) continue;
    if (forced_csize == 0 && c > kTopkPortableCluster && (!long_rows || c != kTopkMaxCluster)) continue;
    const int ch = chunk_for(c);
    if (ch > kTopkMaxChunk) continue;
    if (forced_csize == 0 && c > 1 && (size_t)(c - 1) * ch >= (size_t)num_cols) continue;  // no empty CTA
    const size_t smem = topk_smem_bytes(ch) + 1024;
    const int cps = smem * 2 <= 228u * 1024u ? 2 : 1;  // two CTAs of 512 threads at most (launch bounds)
    const int per_wave = std::max(1, kClustersPerWave[cps - 1][c - 1] * sm_count / 152);
    const int waves = (batch + per_wave - 1) / per_wave;
    const int resident = batch < per_wave ? batch : per_wave;          // clusters in a full wave
    const int sharing = (long long)resident * c > sm_count ? 2 : 1;    // CTAs per SM in that wave
    const double t = waves * (kTkFixedUs + kTkPosUs * ch * sharing + (c > 1 ? kTkClusterUs : 0.0));
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
  size_t most = 0;  // the largest shared memory any chunk takes
  for (int ch = kTopkChunkAlign; ch <= kTopkMaxChunk; ch += kTopkChunkAlign) most = std::max(most, topk_smem_bytes(ch));
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)most);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDevices) configured[dev].store(true, std::memory_order_release);
  return cudaSuccess;
}

cudaError_t launch_topk(const TopkParams& p_in, int batch, cudaStream_t stream) {
  if (batch == 0) return cudaSuccess;
  if (p_in.chunk <= 0 || p_in.chunk % kTopkChunkAlign != 0 || p_in.chunk > kTopkMaxChunk || p_in.csize < 1 ||
      p_in.csize > kTopkMaxCluster)
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = configure_topk(dev);
  if (e != cudaSuccess) return e;
  TopkParams p = p_in;
  p.batch = batch;
  // rows are packed by a pass over every length in every CTA: kept for batches whose lengths fit the
  // CTA's registers (larger batches take one row per cluster)
  p.pack = p.csize > 1 && (p.csize & (p.csize - 1)) == 0 && batch <= kTopkPackMaxRows;
  p.pre8 = topk_key_bytes(p.chunk);
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
