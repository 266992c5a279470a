// topk.cu -- exact per-query top-k over the indexer scores.
//
// "Why DeepSeek V4 Stands Apart", section "Core Architectural Innovations":
// CSA keeps the top-1024 (Pro) / top-512 (Flash) compressed entries per
// query.  Selection rule: the min(k, n) largest scores among the n visible
// entries, ties to the smaller entry index; the output order is unspecified.
//
// Scores are ranked as order-preserving uint32 keys, most significant digit
// first (11, 11 and 10 bits).  Two paths:
//
//   row path (rows that fit one CTA's shared memory, or many rows): one CTA
//   per row holds the row's keys in shared memory, builds the top digit's
//   histogram while loading, lists the keys of the threshold bin, and ranks
//   only that list in the later passes.
//
//   cluster path (few long rows, e.g. decode at 1M context: 8 rows of
//   262,144): a cluster of 8 or 16 CTAs per row, one kernel.  The row's
//   top-digit histogram comes from the indexer (which counts its scores as
//   it writes them: the sum of its CTAs' partials) or, without it, from the
//   cluster's own slices summed in the leader CTA's shared memory.  Every
//   CTA finds the bin of the k-th largest key and sweeps its slice: keys
//   above that bin are selected at once, keys in it (the candidates) go to
//   the leader's shared memory with their second-digit counts.  After one
//   cluster barrier the leader ranks the candidates -- the third digit, then,
//   only if more ties sit at the threshold than places are left, the tie
//   indices from the smallest -- and writes the rest.
//   The only scratch is for candidates past the leader's shared memory.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kBins = kSelBins;
// Row path: keys of the first pass's threshold bin up to which the compact
// path is taken; keys above that bin number fewer than k <= 2048.  Slice
// positions fit 16 bits (a row holds at most 49,152 keys).
constexpr int kMaxCand = 2048;
constexpr int kMaxAbove = 2048;
constexpr int kRowMaxKeys = 49152;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int64_t visible_count(int32_t t, int m, int64_t cap) {
  int64_t n = t < 0 ? 0 : (static_cast<int64_t>(t) + 1) / m;
  return n < cap ? n : cap;
}

struct ScanShared {
  uint32_t warp_tot[32];
  uint32_t digit;
  uint32_t above;
};

// Exclusive prefix of v over the threads of the block, in thread order.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, ScanShared* sh, int tid,
                                                         int nthr) {
  const int lane = tid & 31, warp = tid >> 5;
  uint32_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += x;
  }
  if (lane == 31) sh->warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = nthr >> 5;
    const uint32_t w = lane < nw ? sh->warp_tot[lane] : 0;
    uint32_t t = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += x;
    }
    if (lane < nw) sh->warp_tot[lane] = t - w;
  }
  __syncthreads();
  const uint32_t r = sh->warp_tot[warp] + inc - v;
  __syncthreads();  // warp_tot is reused by the next scan
  return r;
}

// Exclusive prefixes of two per-thread counts over the threads of the block,
// in thread order, and their totals (*tot_a, *tot_b).  One pass: the pair
// travels as one 64-bit value.
__device__ __forceinline__ void block_exclusive_scan2(uint32_t a, uint32_t b, uint32_t* pa,
                                                      uint32_t* pb, uint32_t* tot_a,
                                                      uint32_t* tot_b, uint64_t* warp_tot,
                                                      int tid, int nthr) {
  const int lane = tid & 31, warp = tid >> 5;
  const uint64_t v = (static_cast<uint64_t>(a) << 32) | b;
  uint64_t inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t x = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += x;
  }
  if (lane == 31) warp_tot[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int nw = nthr >> 5;
    const uint64_t w = lane < nw ? warp_tot[lane] : 0;
    uint64_t t = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t x = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += x;
    }
    if (lane < nw) warp_tot[lane] = t - w;
    if (lane == nw - 1) warp_tot[32] = t;
  }
  __syncthreads();
  const uint64_t r = warp_tot[warp] + inc - v;
  *pa = static_cast<uint32_t>(r >> 32);
  *pb = static_cast<uint32_t>(r);
  *tot_a = static_cast<uint32_t>(warp_tot[32] >> 32);
  *tot_b = static_cast<uint32_t>(warp_tot[32]);
  __syncthreads();  // warp_tot is reused by the next scan
}

// find_digit_desc by one warp (nb = 1024 or 2048 bins, nb / 32 per lane,
// lane 0 the top ones), which leaves the other warps free and takes one
// block barrier instead of four.  Every thread of the block calls it.
__device__ __noinline__ void find_digit_desc_warp(const uint32_t* h, int nb, uint32_t need,
                                                  ScanShared* sh, int tid) {
  if (tid < 32) {
    const int lane = tid;
    const int per = nb >> 5;
    const int hi = nb - per * lane;  // this lane's bins: [hi - per, hi)
    uint32_t tot = 0;
    const uint4* h4 = reinterpret_cast<const uint4*>(h + hi - per);
    for (int i = 0; i < per / 4; ++i) {
      const uint4 v = h4[i];
      tot += v.x + v.y + v.z + v.w;
    }
    uint32_t inc = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t x = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += x;
    }
    const uint32_t before = inc - tot;
    const unsigned who = __ballot_sync(0xffffffffu, before < need && inc >= need);
    if (who == 0) {
      if (lane == 0) {  // (need beyond the total: no bin)
        sh->digit = 0;
        sh->above = 0;
      }
    } else {
      // the found lane's per bins, per / 32 to a lane (top first), scanned
      // again across the warp
      const int f = __ffs(who) - 1;
      const uint32_t base_before = __shfl_sync(0xffffffffu, before, f);
      const int fhi = nb - per * f;
      const int sub = per >> 5;  // 1 or 2
      const int my_hi = fhi - sub * lane;
      uint32_t t2 = h[my_hi - 1];
      if (sub == 2) t2 += h[my_hi - 2];
      uint32_t inc2 = t2;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, inc2, o);
        if (lane >= o) inc2 += x;
      }
      const uint32_t b2 = base_before + inc2 - t2;
      if (b2 < need && b2 + t2 >= need) {
        const uint32_t c0 = h[my_hi - 1];
        const bool first = b2 + c0 >= need || sub == 1;
        sh->digit = static_cast<uint32_t>(first ? my_hi - 1 : my_hi - 2);
        sh->above = first ? b2 : b2 + c0;
      }
    }
  }
  __syncthreads();
}

// The bin holding the need-th largest key (1 <= need <= total): bins are
// visited from the top; sh->digit = that bin, sh->above = keys in the bins
// above it.  nb >= nthr, both powers of two.
__device__ __noinline__ void find_digit_desc(const uint32_t* h, int nb, uint32_t need,
                                                ScanShared* sh, int tid, int nthr) {
  if (tid == 0) {  // ordered before the finder's write by the scan's barriers
    sh->digit = 0;
    sh->above = 0;
  }
  const int bpt = nb / nthr;
  const int hi = nb - bpt * tid;  // this thread's bins: [hi - bpt, hi)
  uint32_t tot = 0;
  for (int i = 0; i < bpt; ++i) tot += h[hi - 1 - i];
  const uint32_t before = block_exclusive_scan(tot, sh, tid, nthr);
  if (before < need && before + tot >= need) {
    uint32_t run = before;
    for (int i = 0; i < bpt; ++i) {
      const uint32_t c = h[hi - 1 - i];
      if (run + c >= need) {
        sh->digit = static_cast<uint32_t>(hi - 1 - i);
        sh->above = run;
        break;
      }
      run += c;
    }
  }
  __syncthreads();
}

// The bin holding the need-th smallest value: bins visited from the bottom;
// sh->digit = that bin, sh->above = values in the bins below it.
__device__ __noinline__ void find_digit_asc(const uint32_t* h, int nb, uint32_t need,
                                               ScanShared* sh, int tid, int nthr) {
  if (tid == 0) {
    sh->digit = 0;
    sh->above = 0;
  }
  const int bpt = nb / nthr;
  const int lo = bpt * tid;
  uint32_t tot = 0;
  for (int i = 0; i < bpt; ++i) tot += h[lo + i];
  const uint32_t before = block_exclusive_scan(tot, sh, tid, nthr);
  if (before < need && before + tot >= need) {
    uint32_t run = before;
    for (int i = 0; i < bpt; ++i) {
      const uint32_t c = h[lo + i];
      if (run + c >= need) {
        sh->digit = static_cast<uint32_t>(lo + i);
        sh->above = run;
        break;
      }
      run += c;
    }
  }
  __syncthreads();
}

// Appends `take` (per thread) to a global counter with one atomic per warp;
// returns this thread's slot (valid where take).
__device__ __forceinline__ int warp_append(int* ctr, bool take) {
  const unsigned mask = __ballot_sync(0xffffffffu, take);
  if (!mask) return -1;
  const int lane = threadIdx.x & 31;
  const int leader = __ffs(mask) - 1;
  int base = 0;
  if (lane == leader) base = atomicAdd(ctr, __popc(mask));
  base = __shfl_sync(0xffffffffu, base, leader);
  return base + __popc(mask & ((1u << lane) - 1u));
}

// ============================================================ row path
struct RowShared {
  ScanShared scan;
  uint32_t hist[kBins];
  int counts[2];
  int ctr, ctr_eq;
  int n_cand, n_above;
  uint16_t cand[kMaxCand];
  uint16_t above_idx[kMaxAbove];
};

__global__ void __launch_bounds__(1024) topk_row_kernel(const TopkArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  RowShared* sh = reinterpret_cast<RowShared*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + sizeof(RowShared));
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int64_t row = static_cast<int64_t>(blockIdx.y) + static_cast<int64_t>(gridDim.y) * blockIdx.z;

  pdl_trigger();
  pdl_wait();  // the scores (and a dependent launch's predecessor) are complete
  if (row >= a.rows) return;
  const int len = static_cast<int>(visible_count(a.pos[row], a.m, a.N_cap));
  int32_t* out = a.idx + row * a.k;

  if (len <= a.k) {  // every visible entry is selected
    for (int e = tid; e < a.k; e += nthr) out[e] = e < len ? e : -1;
    return;
  }

  const float* src = a.scores + row * a.N_cap;
  for (int i = tid; i < kBins; i += nthr) sh->hist[i] = 0;
  __syncthreads();
  // the keys, and the first pass's histogram of their top 11 bits, in one sweep
  for (int e = tid; e < len; e += nthr) {
    const uint32_t key = order_key(src[e]);
    keys[e] = key;
    atomicAdd(&sh->hist[key >> 21], 1u);
  }
  __syncthreads();

  uint32_t prefix = 0;
  uint32_t need = static_cast<uint32_t>(a.k);
  // one radix pass: the digit of the need-th largest key among those left;
  // returns the keys in that digit's bin, and clears the histogram
  auto radix_pass = [&](int width) -> uint32_t {
    const int nb = 1 << width;
    find_digit_desc(sh->hist, nb, need, &sh->scan, tid, nthr);
    const uint32_t in_bin = sh->hist[sh->scan.digit];
    prefix = (prefix << width) | sh->scan.digit;
    need -= sh->scan.above;
    __syncthreads();  // every thread has read the bin
    for (int i = tid; i < kBins; i += nthr) sh->hist[i] = 0;
    __syncthreads();
    return in_bin;
  };
  // The keys left to rank are those in the bin of the k-th largest (about
  // 0.5% of normal scores).  When few enough, one sweep lists them (and the
  // keys above the bin, which are selected), and the remaining passes, the
  // counts and the writes visit only the lists.
  const bool compact = radix_pass(11) <= static_cast<uint32_t>(kMaxCand);
  const uint32_t d0 = prefix;
  if (tid == 0) {
    sh->n_cand = 0;
    sh->n_above = 0;
  }
  __syncthreads();
  int n_cand = 0, n_above = 0;
  if (compact) {
    for (int e = tid; e < len; e += nthr) {
      const uint32_t key = keys[e];
      const uint32_t d = key >> 21;
      if (d == d0) {
        sh->cand[atomicAdd(&sh->n_cand, 1)] = static_cast<uint16_t>(e);
        atomicAdd(&sh->hist[(key >> 10) & 2047u], 1u);
      } else if (d > d0) {
        sh->above_idx[atomicAdd(&sh->n_above, 1)] = static_cast<uint16_t>(e);
      }
    }
    __syncthreads();
    n_cand = sh->n_cand;
    n_above = sh->n_above;
    radix_pass(11);
    for (int c = tid; c < n_cand; c += nthr) {
      const uint32_t key = keys[sh->cand[c]];
      if ((key >> 10) == prefix) atomicAdd(&sh->hist[key & 1023u], 1u);
    }
    __syncthreads();
    radix_pass(10);
  } else {
    for (int e = tid; e < len; e += nthr) {
      const uint32_t key = keys[e];
      if ((key >> 21) == prefix) atomicAdd(&sh->hist[(key >> 10) & 2047u], 1u);
    }
    __syncthreads();
    radix_pass(11);
    for (int e = tid; e < len; e += nthr) {
      const uint32_t key = keys[e];
      if ((key >> 10) == prefix) atomicAdd(&sh->hist[key & 1023u], 1u);
    }
    __syncthreads();
    radix_pass(10);
  }
  const uint32_t thr = prefix;  // the k-th largest key; take `need` of its ties

  if (tid == 0) {
    sh->counts[1] = 0;
    sh->ctr = 0;
    sh->ctr_eq = 0;
  }
  __syncthreads();
  int eq = 0;
  if (compact) {
    for (int c = tid; c < n_cand; c += nthr) eq += keys[sh->cand[c]] == thr;
  } else {
    for (int e = tid; e < len; e += nthr) eq += keys[e] == thr;
  }
  if (eq) atomicAdd(&sh->counts[1], eq);
  __syncthreads();
  const int base = a.k - static_cast<int>(need);  // ties go to [base, k)
  const bool all_ties = sh->counts[1] == static_cast<int>(need);
  if (compact) {
    for (int c = tid; c < n_above; c += nthr) out[atomicAdd(&sh->ctr, 1)] = sh->above_idx[c];
    for (int c = tid; c < n_cand; c += nthr) {
      const int e = sh->cand[c];
      const uint32_t key = keys[e];
      if (key > thr) out[atomicAdd(&sh->ctr, 1)] = e;
      else if (key == thr && all_ties) out[base + atomicAdd(&sh->ctr_eq, 1)] = e;
    }
  } else {
    for (int e = tid; e < len; e += nthr) {
      const uint32_t key = keys[e];
      if (key > thr) out[atomicAdd(&sh->ctr, 1)] = e;
      else if (key == thr && all_ties) out[base + atomicAdd(&sh->ctr_eq, 1)] = e;
    }
  }
  if (!all_ties) {
    // more ties than places: the ties with the smaller indices win, so each
    // thread owns a contiguous run and ranks its ties by a block scan; the
    // count visits the run in a per-lane rotated order (no bank conflicts)
    const int per_t = (len + nthr - 1) / nthr;
    const int e0 = tid * per_t;
    const int n_run = max(0, min(len, e0 + per_t) - e0);
    const int r0 = n_run > 0 ? (tid & 31) % n_run : 0;
    uint32_t c = 0;
    for (int j = 0; j < n_run; ++j) {
      int jj = j + r0;
      if (jj >= n_run) jj -= n_run;
      c += keys[e0 + jj] == thr;
    }
    uint32_t rnk = block_exclusive_scan(c, &sh->scan, tid, nthr);
    for (int j = 0; j < n_run && c > 0 && rnk < need; ++j) {
      if (keys[e0 + j] == thr) {
        out[base + rnk] = e0 + j;
        ++rnk;
        --c;
      }
    }
  }
}

// ============================================================ cluster path
constexpr int kClusterSize = 8;          // CTAs per row (the portable cluster size)
constexpr int kClusterThreads = 1024;
constexpr int kSumBatch = 24;            // partial histograms whose loads a thread issues at once
constexpr int kSliceChunk = 8192;        // entries per bulk copy of the slice (32 KB)
constexpr int kSliceChunks = 4;
constexpr int kMaxSlice = kSliceChunk * kSliceChunks;  // entries a CTA stages in shared memory
constexpr int kCandCap = 6144;           // candidates the leader holds in shared memory
constexpr int kBinCap = 2048;            // the leader's list of one second-digit bin
static_assert(kBins == 2 * kClusterThreads, "one bin pair per thread");

struct ClusterShared {
  // (16-byte aligned arrays: hist and rowhist move as 16-byte vectors)
  alignas(16) uint32_t hist[kBins];     // the row's top-digit histogram; the leader's third-digit counts
  alignas(16) uint32_t rowhist[kBins];  // leader, no folded pass: the slices' top-digit histograms summed
  alignas(16) uint32_t hist2[kBins];    // leader: the row's candidates' second-digit histogram
  alignas(16) uint32_t lhist2[kBins];   // this CTA's candidates' second-digit histogram
  alignas(16) int32_t binlist[kBinCap];  // leader: the candidates in one second-digit bin
  uint64_t chunk_full[kSliceChunks];     // the slice's bulk copies have landed
  uint64_t wtot[33];                     // block_exclusive_scan2's warp totals
  ScanShared scan;
  int n_up, n_cand;         // leader: the row's list fills
  int base_up, base_cand;   // this CTA's ranges in the row's lists
  int n_gt, n_eq, n_bin;
};
static_assert(sizeof(ClusterShared) % 16 == 0, "the candidate arrays follow, 16-byte aligned");
// dynamic shared memory: the staged slice, ClusterShared, then the leader's
// candidate keys and entry indices (kCandCap each)
constexpr size_t kSliceBytes = static_cast<size_t>(kMaxSlice) * 4;
constexpr size_t kClusterSmem = kSliceBytes + sizeof(ClusterShared) + static_cast<size_t>(kCandCap) * 8;
static_assert(kClusterSmem <= 227 * 1024, "one CTA's shared memory");

// The indexer CTA whose slots contain slot x (its slots are
// [total * c / grid, total * (c + 1) / grid)).
__device__ __forceinline__ int64_t part_owner(int64_t x, int64_t total, int64_t grid) {
  return ((x + 1) * grid + total - 1) / total - 1;
}

// Candidates c and `need` places left (need < C), all in the top-digit bin
// d0; h2 holds the candidates' second-digit histogram.  Writes `need`
// entries to rest[]: those above the need-th largest key, then its ties
// with the smallest entry indices.  (The general ranking; the leader takes
// it when the second digit's bin holds more candidates than one warp ranks.)
template <class IdxOf, class KeyOf>
__device__ __noinline__ void rank_candidates(int C, uint32_t need, uint32_t d0, const uint32_t* h2,
                                             int32_t* rest, ClusterShared& sh, IdxOf idx_of,
                                             KeyOf key_of) {
  const int tid = threadIdx.x;
  const int room = static_cast<int>(need);
  // second digit from the gathered histogram, third by one pass
  find_digit_desc_warp(h2, kBins, need, &sh.scan, tid);
  uint32_t prefix = (d0 << 11) | sh.scan.digit;
  need -= sh.scan.above;
  for (int i = tid; i < kBins; i += kClusterThreads) sh.hist[i] = 0;
  __syncthreads();
  for (int c = tid; c < C; c += kClusterThreads) {
    const uint32_t key = key_of(c);
    if ((key >> 10) == prefix) atomicAdd(&sh.hist[key & 1023u], 1u);
  }
  __syncthreads();
  find_digit_desc_warp(sh.hist, 1024, need, &sh.scan, tid);
  const uint32_t thr = (prefix << 10) | sh.scan.digit;  // the k-th largest key
  need -= sh.scan.above;                                // its ties still to take
  // candidates above the threshold, and the count of ties at it (the loop
  // runs the same trip count in every thread: warp_append is warp-collective)
  if (tid == 0) {
    sh.n_gt = 0;
    sh.n_eq = 0;
  }
  __syncthreads();
  int eq = 0;
  for (int c0 = 0; c0 < C; c0 += kClusterThreads) {
    const int c = c0 + tid;
    const uint32_t key = c < C ? key_of(c) : 0u;
    const bool gt = c < C && key > thr;
    const int p = warp_append(&sh.n_gt, gt);  // shared-memory counter
    if (gt && p < room) rest[p] = idx_of(c);
    eq += c < C && key == thr;
  }
  if (eq) atomicAdd(&sh.n_eq, eq);
  __syncthreads();
  const int n_gt = sh.n_gt;
  const uint32_t n_eq = static_cast<uint32_t>(sh.n_eq);
  // ties at the threshold: the need smallest entry indices among them (every
  // tie when they are exactly the places left).  Radix select on the index
  // value, smallest first, finds the need-th smallest tie index ti.
  uint32_t ti = 0xffffffffu;
  if (n_eq != need) {
    uint32_t ip = 0, left = need;
    for (int pass = 0; pass < 3; ++pass) {
      const int width = pass == 2 ? 10 : 11;
      const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
      const int nb = 1 << width;
      for (int i = tid; i < kBins; i += kClusterThreads) sh.hist[i] = 0;
      __syncthreads();
      for (int c = tid; c < C; c += kClusterThreads) {
        if (key_of(c) != thr) continue;
        const uint32_t j = static_cast<uint32_t>(idx_of(c));
        if (pass > 0 && (j >> (shift + width)) != ip) continue;
        atomicAdd(&sh.hist[(j >> shift) & (nb - 1)], 1u);
      }
      __syncthreads();
      find_digit_asc(sh.hist, nb, left, &sh.scan, tid, kClusterThreads);
      ip = (ip << width) | sh.scan.digit;
      left -= sh.scan.above;
    }
    ti = ip;  // indices are distinct: the ties with index <= ti are exactly `need`
  }
  if (tid == 0) sh.n_gt = 0;
  __syncthreads();
  int32_t* ties_out = rest + n_gt;
  for (int c0 = 0; c0 < C; c0 += kClusterThreads) {
    const int c = c0 + tid;
    bool take = false;
    int32_t j = 0;
    if (c < C && key_of(c) == thr) {
      j = idx_of(c);
      take = static_cast<uint32_t>(j) <= ti;
    }
    const int p = warp_append(&sh.n_gt, take);
    if (take && n_gt + p < room) ties_out[p] = j;
  }
}

// One cluster of kClusterSize CTAs per row; CTA r of the cluster sweeps
// entries [r * slice, (r + 1) * slice) of the row.
__global__ void __launch_bounds__(kClusterThreads, 1) topk_cluster_kernel(const TopkArgs a) {
  extern __shared__ __align__(16) uint8_t csm[];
  float* sslice = reinterpret_cast<float*>(csm);
  ClusterShared& sh = *reinterpret_cast<ClusterShared*>(csm + kSliceBytes);
  uint32_t* ckey = reinterpret_cast<uint32_t*>(csm + kSliceBytes + sizeof(ClusterShared));
  int32_t* cidx = reinterpret_cast<int32_t*>(csm + kSliceBytes + sizeof(ClusterShared) + kCandCap * 4);
  const int tid = threadIdx.x;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int64_t row = static_cast<int64_t>(blockIdx.y) + static_cast<int64_t>(gridDim.y) * blockIdx.z;
  const int64_t lo = static_cast<int64_t>(rank) * a.slice;
  // this CTA's part of the row staged in shared memory by bulk copies
  // (rows 16-byte aligned, N_cap a multiple of 4): entries [lo, lo + staged)
  const int64_t room = a.N_cap - lo;
  const int staged = !a.vec4 || row >= a.rows || room <= 0
                         ? 0
                         : static_cast<int>(min(min(a.slice, static_cast<int64_t>(kMaxSlice)), room));
  if (tid == 0) {
    for (int c = 0; c < kSliceChunks; ++c) mbar_init(smem_u32(&sh.chunk_full[c]), 1);
    fence_barrier_init();
  }
  // the visible count: pos is an input of the step, read before the wait
  // (as the score kernel does)
  const int64_t n = row < a.rows ? visible_count(a.pos[row], a.m, a.N_cap) : 0;
  __syncthreads();
  pdl_trigger();
  pdl_wait();  // the scores (and the folded histograms) are complete
  const float* src = a.scores + row * a.N_cap;
  if (tid == 0) {
    for (int c = 0; c < kSliceChunks; ++c) {
      const int c0 = c * kSliceChunk;
      if (c0 >= staged) break;
      const uint32_t bytes = static_cast<uint32_t>(min(kSliceChunk, staged - c0)) * 4u;
      const uint32_t bar = smem_u32(&sh.chunk_full[c]);
      mbar_arrive_expect_tx(bar, bytes);
      bulk_copy_g2s(smem_u32(sslice + c0), src + lo + c0, bytes, bar);
    }
  }
  // every condition that ends a CTA early holds for its whole cluster (one row)
  bool ok = true;
  auto drain = [&]() {
    // the slice's copies land before the CTA's shared memory is released
    for (int c = 0; c * kSliceChunk < staged; ++c)
      mbar_wait(smem_u32(&sh.chunk_full[c]), 0, nullptr, a.status, kWaitLimitNs, 41);
  };
  if (row >= a.rows) return;  // (nothing staged)
  int32_t* out = a.idx + row * a.k;
  const int64_t hi = lo + a.slice < n ? lo + a.slice : n;
  if (n <= a.k) {
    // every visible entry is selected; the leader pads
    for (int64_t e = lo + tid; e < hi; e += kClusterThreads) out[e] = static_cast<int32_t>(e);
    if (leader)
      for (int64_t e = n + tid; e < a.k; e += kClusterThreads) out[e] = -1;
    drain();
    return;
  }
  const bool folded = a.hist_part != nullptr;
  for (int i = tid; i < kBins; i += kClusterThreads) {
    sh.lhist2[i] = 0;
    if (leader) {
      sh.hist2[i] = 0;
      sh.rowhist[i] = 0;
    }
    if (!folded) sh.hist[i] = 0;
  }
  if (tid == 0) {
    sh.n_up = 0;
    sh.n_cand = 0;
  }
  __syncthreads();
  cluster_arrive();  // (A) the leader's counters and histograms are cleared
  // the staged entries this CTA sweeps: [lo, lo + n_st), the rest of its
  // slice [lo + n_st, hi) from global memory
  const int n_st = static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(staged), hi - lo)));
  auto chunk_wait = [&](int c) {
    ok = mbar_wait(smem_u32(&sh.chunk_full[c]), 0, nullptr, a.status, kWaitLimitNs, 41) && ok;
  };
  if (folded) {
    // the row's histogram: the sum of the indexer CTAs' partials for it.
    // Thread t sums the bin pair t (one 32-bit word holds two 16-bit bins),
    // kSumBatch partials' loads in flight at once.  (Partial j = 1 of an
    // indexer CTA is its second row: only the first CTA of the row can hold
    // the row there, when its slots begin in the row before.)
    const int64_t first = row * a.part_nblk;
    const int64_t c_lo = part_owner(first, a.part_total, a.part_grid);
    const int64_t c_hi = part_owner(first + a.part_nblk - 1, a.part_total, a.part_grid);
    const int np = static_cast<int>(c_hi - c_lo + 1);
    const bool lo_second = a.part_total * c_lo / a.part_grid < first;
    const uint32_t* base = reinterpret_cast<const uint32_t*>(a.hist_part + c_lo * 2 * kBins) + tid;
    uint32_t c2[2] = {0u, 0u};
    for (int q0 = 0; q0 < np; q0 += kSumBatch) {
      uint32_t v[kSumBatch];
#pragma unroll
      for (int u = 0; u < kSumBatch; ++u) {
        const int q = q0 + u;
        // partial (c_lo + q, j) starts (2 q + j) * kBins / 2 words from base
        v[u] = q < np ? __ldcg(base + (2 * q + (q == 0 && lo_second ? 1 : 0)) * (kBins / 2)) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kSumBatch; ++u) {
        c2[0] += v[u] & 0xffffu;
        c2[1] += v[u] >> 16;
      }
    }
    sh.hist[2 * tid] = c2[0];
    sh.hist[2 * tid + 1] = c2[1];
    cluster_wait();  // (A)
  } else {
    // this slice's histogram, added into the leader's, which every CTA reads
    // back once all slices are in
    for (int c = 0; c * kSliceChunk < n_st; ++c) {
      chunk_wait(c);
      const int e1 = min(n_st, (c + 1) * kSliceChunk);
      for (int e = c * kSliceChunk + tid; e < e1; e += kClusterThreads)
        atomicAdd(&sh.hist[order_key(sslice[e]) >> 21], 1u);
    }
    for (int64_t e = lo + n_st + tid; e < hi; e += kClusterThreads)
      atomicAdd(&sh.hist[order_key(__ldcg(src + e)) >> 21], 1u);
    __syncthreads();
    cluster_wait();  // (A)
    for (int i = tid; i < kBins; i += kClusterThreads)
      if (sh.hist[i]) red_add_cluster(mapa_shared(smem_u32(&sh.rowhist[i]), 0), sh.hist[i]);
    cluster_arrive();
    cluster_wait();  // (B) every slice is in the leader's histogram
    const uint32_t rh = mapa_shared(smem_u32(sh.rowhist), 0);
    for (int i = tid; i < kBins / 4; i += kClusterThreads)
      reinterpret_cast<uint4*>(sh.hist)[i] = ld_cluster_v4(rh + 16u * i);
  }
  __syncthreads();
  find_digit_desc_warp(sh.hist, kBins, static_cast<uint32_t>(a.k), &sh.scan, tid);
  const uint32_t d0 = sh.scan.digit;
  const uint32_t n_above = sh.scan.above;  // keys in bins above d0: all selected
  int32_t* cand_g = a.cand + row * a.N_cap;  // candidates past the leader's capacity
  const uint32_t r_up = mapa_shared(smem_u32(&sh.n_up), 0);
  const uint32_t r_cand = mapa_shared(smem_u32(&sh.n_cand), 0);
  const uint32_t r_ckey = mapa_shared(smem_u32(ckey), 0);
  const uint32_t r_cidx = mapa_shared(smem_u32(cidx), 0);
  const uint32_t r_hist2 = mapa_shared(smem_u32(sh.hist2), 0);
  // Sweep the slice twice, each thread over the same entries: count the
  // entries above the threshold bin (selected) and in it (candidates), scan
  // the counts over the block and reserve the CTA's ranges in the row's
  // lists at the leader, then write each entry to its place.  No atomics on
  // a shared counter, and the common entry costs a compare.
  // The smallest score of bin d0, as a float (order_key is monotone): a
  // score x is at or above the bin iff !(x < T), one float compare instead
  // of a key (integer operations run at half the float rate).  NaN scores
  // fail every compare and take the exact key test, as do all scores when
  // the bin holds infinities or NaN keys (d0 outside [4, 2044]).
  float T = -INFINITY;
  if (d0 >= 4 && d0 <= 2044) {
    const uint32_t kl = d0 << 21;
    T = __uint_as_float((kl & 0x80000000u) ? (kl & 0x7fffffffu) : ~kl);
  }
  const float4* s4 = reinterpret_cast<const float4*>(sslice);
  auto visit = [&](auto&& fn) {
    for (int c = 0; c * kSliceChunk < n_st; ++c) {
      const int e1 = min(n_st, (c + 1) * kSliceChunk);
      for (int q = (c * kSliceChunk >> 2) + tid; 4 * q < e1; q += kClusterThreads) {
        const float4 v = s4[q];
        if (v.x < T && v.y < T && v.z < T && v.w < T) continue;
        const uint32_t k0 = order_key(v.x), k1 = order_key(v.y);
        const uint32_t k2 = order_key(v.z), k3 = order_key(v.w);
        const int64_t e = lo + 4 * q;
        // (entries past the visible count are not visited)
        if (4 * q < e1) fn(e, k0);
        if (4 * q + 1 < e1) fn(e + 1, k1);
        if (4 * q + 2 < e1) fn(e + 2, k2);
        if (4 * q + 3 < e1) fn(e + 3, k3);
      }
    }
    for (int64_t e = lo + n_st + tid; e < hi; e += kClusterThreads) fn(e, order_key(__ldcg(src + e)));
  };
  if (folded)
    for (int c = 0; c * kSliceChunk < n_st; ++c) chunk_wait(c);
  uint32_t cu = 0, cc = 0;
  visit([&](int64_t, uint32_t key) {
    cu += (key >> 21) > d0;
    cc += (key >> 21) == d0;
  });
  uint32_t ou, oc, tu, tc;
  block_exclusive_scan2(cu, cc, &ou, &oc, &tu, &tc, sh.wtot, tid, kClusterThreads);
  if (tid == 0) {
    sh.base_up = tu ? static_cast<int>(atom_add_cluster(r_up, tu)) : 0;
    sh.base_cand = tc ? static_cast<int>(atom_add_cluster(r_cand, tc)) : 0;
  }
  __syncthreads();
  uint32_t pu = static_cast<uint32_t>(sh.base_up) + ou;
  uint32_t pc = static_cast<uint32_t>(sh.base_cand) + oc;
  visit([&](int64_t e, uint32_t key) {
    const uint32_t d = key >> 21;
    if (d > d0) {
      if (pu < static_cast<uint32_t>(a.k)) out[pu] = static_cast<int32_t>(e);
      ++pu;
    } else if (d == d0) {
      if (pc < static_cast<uint32_t>(kCandCap)) {
        st_cluster_u32(r_ckey + 4u * pc, key);
        st_cluster_u32(r_cidx + 4u * pc, static_cast<uint32_t>(e));
      } else if (static_cast<int64_t>(pc) - kCandCap < a.N_cap) {
        cand_g[pc - kCandCap] = static_cast<int32_t>(e);
      }
      ++pc;
      atomicAdd(&sh.lhist2[(key >> 10) & 2047u], 1u);
    }
  });
  // the staged chunks past the visible entries were never waited for
  for (int c = 0; c * kSliceChunk < staged; ++c)
    if (c * kSliceChunk >= n_st) chunk_wait(c);
  __syncthreads();
  for (int i = tid; i < kBins; i += kClusterThreads)
    if (sh.lhist2[i]) red_add_cluster(r_hist2 + 4u * i, sh.lhist2[i]);
  // (C) the row's candidates are with the leader (and in the overflow
  // list); the other CTAs are done and their shared memory is not read
  cluster_arrive();
  cluster_wait();
  if (!leader || !ok) return;
  const int C = min(sh.n_cand, static_cast<int>(min(a.N_cap, static_cast<int64_t>(INT32_MAX))));
  const uint32_t need = static_cast<uint32_t>(a.k) - n_above;  // 1 <= need <= C
  int32_t* rest = out + n_above;
  auto idx_of = [&](int c) -> int32_t {
    return c < kCandCap ? cidx[c] : __ldcg(cand_g + (c - kCandCap));
  };
  auto key_of = [&](int c) -> uint32_t {
    return c < kCandCap ? ckey[c] : order_key(__ldcg(src + __ldcg(cand_g + (c - kCandCap))));
  };
  if (static_cast<int>(need) >= C) {
    for (int c = tid; c < C; c += kClusterThreads) rest[c] = idx_of(c);
    return;
  }
  // The second digit's bin from the gathered histogram, then one pass: the
  // candidates above that bin are selected, those in it listed.  The list
  // is a few entries for spread-out scores; one warp ranks up to 32 of them
  // (key descending, then entry index ascending), else the general ranking
  // runs.
  find_digit_desc_warp(sh.hist2, kBins, need, &sh.scan, tid);
  const uint32_t p1 = (d0 << 11) | sh.scan.digit;
  const uint32_t above1 = sh.scan.above;
  const uint32_t need1 = need - above1;  // >= 1
  if (tid == 0) {
    sh.n_gt = 0;
    sh.n_bin = 0;
  }
  __syncthreads();
  for (int c0 = 0; c0 < C; c0 += kClusterThreads) {
    const int c = c0 + tid;
    const uint32_t p = c < C ? key_of(c) >> 10 : 0u;
    const bool gt = c < C && p > p1;
    const bool in = c < C && p == p1;
    const int g = warp_append(&sh.n_gt, gt);
    if (gt && g < static_cast<int>(above1)) rest[g] = idx_of(c);
    const int b = warp_append(&sh.n_bin, in);
    if (in && b < kBinCap) sh.binlist[b] = c;
  }
  __syncthreads();
  const int nb = sh.n_bin;
  if (nb <= 32) {
    if (tid < 32) {
      // bitonic sort of the bin's (key, index) pairs over one warp, best first
      const int lane = tid;
      uint32_t key = 0u;
      int32_t j = INT32_MAX;
      if (lane < nb) {
        key = key_of(sh.binlist[lane]);
        j = idx_of(sh.binlist[lane]);
      }
      for (int kk = 2; kk <= 32; kk <<= 1) {
        for (int jj = kk >> 1; jj > 0; jj >>= 1) {
          const uint32_t ok2 = __shfl_xor_sync(0xffffffffu, key, jj);
          const int32_t oj = __shfl_xor_sync(0xffffffffu, j, jj);
          const bool mine_first = key > ok2 || (key == ok2 && j < oj);
          const bool lower = (lane & jj) == 0;
          const bool best_first = (lane & kk) == 0;
          if ((lower == best_first) != mine_first) {
            key = ok2;
            j = oj;
          }
        }
      }
      if (lane < static_cast<int>(need1)) rest[above1 + lane] = j;
    }
  } else {
    rank_candidates(C, need, d0, sh.hist2, rest, sh, idx_of, key_of);
  }
}

}  // namespace

static_assert(sizeof(RowShared) + kRowMaxKeys * 4 <= 227 * 1024,
              "a 49,152-key row and the shared state fit one CTA's shared memory");

bool plan_topk(int64_t rows, int64_t N_cap, int k, int num_sms, TopkPlan* p) {
  if (rows <= 0 || N_cap < 1 || k < 1) return false;
  *p = TopkPlan{};
  // Few long rows spread over a cluster of CTAs each (cluster path);
  // otherwise one CTA per row with the keys in shared memory (row path).
  const bool row_fits = N_cap <= kRowMaxKeys;
  const bool few_rows = rows * 2 < num_sms;
  if (row_fits && (!few_rows || N_cap <= 8192)) {
    p->slice_path = false;
    p->S = 1;
    p->threads = N_cap >= 8192 ? 1024 : (N_cap >= 2048 ? 512 : 256);
    p->smem_bytes = sizeof(RowShared) + static_cast<size_t>(N_cap) * 4;
  } else {
    p->slice_path = true;
    // 8 CTAs per row (the portable cluster size: any GPC holds one, so the
    // rows' clusters start together); a slice is a multiple of 64 entries
    p->S = kClusterSize;
    p->slice = ((N_cap + p->S - 1) / p->S + 63) / 64 * 64;
    p->threads = kClusterThreads;
    p->smem_bytes = kClusterSmem;
  }
  p->ws_bytes = topk_scratch_bytes(*p, rows, N_cap);
  return true;
}

size_t topk_scratch_bytes(const TopkPlan& p, int64_t rows, int64_t N_cap) {
  if (!p.slice_path) return 0;
  // the candidates past the leader's shared memory (a row of near-equal scores)
  return static_cast<size_t>(rows) * N_cap * sizeof(int32_t);
}

void topk_scratch_carve(const TopkPlan& p, int64_t rows, void* ws, TopkArgs* a) {
  (void)p;
  (void)rows;
  a->cand = static_cast<int32_t*>(ws);
}

cudaError_t launch_topk(const TopkArgs& a, const TopkPlan& p, bool dependent,
                        cudaStream_t stream) {
  // rows fold over grid y and z (y <= 65535)
  const int64_t gy = a.rows < 65535 ? a.rows : 65535;
  const int64_t gz = (a.rows + gy - 1) / gy;
  if (gz > 65535) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(p.threads, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  cfg.attrs = at;
  TopkArgs args = a;
  cudaError_t e;
  if (!p.slice_path) {
    args.S = 1;
    args.vec4 = 0;
    cfg.numAttrs = add_dependent_attr(at, 0, dependent);
    e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(p.smem_bytes));
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(1, static_cast<unsigned>(gy), static_cast<unsigned>(gz));
    cfg.dynamicSmemBytes = p.smem_bytes;
    e = cudaLaunchKernelEx(&cfg, topk_row_kernel, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  args.S = p.S;
  args.slice = p.slice;
  args.vec4 = (a.N_cap % 4 == 0) && (reinterpret_cast<uintptr_t>(a.scores) % 16 == 0) &&
              (p.slice % 4 == 0);
  e = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(kClusterSmem));
  if (e != cudaSuccess) return e;
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = static_cast<unsigned>(p.S);
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.numAttrs = add_dependent_attr(at, 1, dependent);
  cfg.gridDim = dim3(p.S, static_cast<unsigned>(gy), static_cast<unsigned>(gz));
  cfg.dynamicSmemBytes = kClusterSmem;
  e = cudaLaunchKernelEx(&cfg, topk_cluster_kernel, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hattn
