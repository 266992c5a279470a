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
//   slice path (few long rows, e.g. decode at 1M context: 8 rows of 262,144):
//   S CTAs per row, two kernels and no inter-CTA waiting.
//     topk_hist_kernel: each CTA histograms the top digit of its slice into
//       its own 2,048 16-bit bins of the scratch (no atomics, nothing to
//       clear), and CTA 0 of the row clears the row's counters.
//     topk_pick_kernel: each CTA sums the row's S histograms, finds the bin
//       of the k-th largest key, and sweeps its slice again: keys above that
//       bin are selected at once (appended to the output), keys in it are
//       appended to the row's candidate list.  The last CTA of the row to
//       finish (a ticket counter) ranks the candidates -- the remaining two
//       digits, then, only if more ties sit at the threshold than places
//       are left, the tie indices from the smallest -- and writes the rest.
//   The scratch is caller-owned (hattn_topk_workspace_bytes).
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kBins = 2048;
// Row path: keys of the first pass's threshold bin up to which the compact
// path is taken; keys above that bin number fewer than k <= 2048.  Slice
// positions fit 16 bits (a row holds at most 49,152 keys).
constexpr int kMaxCand = 2048;
constexpr int kMaxAbove = 2048;
constexpr int kRowMaxKeys = 49152;
constexpr int kPickThreads = 512;

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

// The bin holding the need-th largest key (1 <= need <= total): bins are
// visited from the top; sh->digit = that bin, sh->above = keys in the bins
// above it.  nb >= nthr, both powers of two.
__device__ __forceinline__ void find_digit_desc(const uint32_t* h, int nb, uint32_t need,
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
__device__ __forceinline__ void find_digit_asc(const uint32_t* h, int nb, uint32_t need,
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

// ============================================================ slice path
constexpr int kListCap = 2048;   // per-CTA shared-memory lists of the pick sweep
constexpr int kLoadBatch = 8;    // float4 loads a thread issues before using them
constexpr int kSumBatch = 24;    // slices whose histogram loads a thread issues at once
constexpr int kCandSmem = 8192;  // candidates the last CTA ranks in shared memory

struct SliceShared {
  ScanShared scan;
  uint32_t hist[kBins];
  int n_up, n_in;        // fills of the two lists
  int base_up, base_in;  // their ranges in the row's output and candidate list
  int last;
  int n_gt, n_eq;
  int32_t up[kListCap];  // entries above the threshold bin (selected)
  int32_t in[kListCap];  // entries in the threshold bin (candidates)
};

// Histogram of the top 11 key bits of this CTA's slice, into its own bins.
__global__ void __launch_bounds__(kPickThreads) topk_hist_kernel(const TopkArgs a) {
  __shared__ uint32_t hist[kBins];
  const int tid = threadIdx.x;
  const int s = blockIdx.x;
  const int64_t row = static_cast<int64_t>(blockIdx.y) + static_cast<int64_t>(gridDim.y) * blockIdx.z;
  pdl_trigger();
  pdl_wait();  // the scores are complete
  if (row >= a.rows) return;
  if (s == 0 && tid < 4) a.ctr[row * 4 + tid] = 0;  // read by topk_pick_kernel
  const int64_t n = visible_count(a.pos[row], a.m, a.N_cap);
  if (n <= a.k) return;  // every visible entry is selected (the pick kernel writes them)
  for (int i = tid; i < kBins; i += kPickThreads) hist[i] = 0;
  __syncthreads();
  const int64_t lo = static_cast<int64_t>(s) * a.slice;
  const int64_t hi = lo + a.slice < n ? lo + a.slice : n;
  const float* src = a.scores + row * a.N_cap;
  if (hi <= lo) {
    // nothing visible in this slice
  } else if (a.vec4) {
    // slices start at multiples of 4 and rows are 16-byte aligned; each
    // thread issues up to kLoadBatch float4 loads before using any of them
    const int64_t q_hi = hi >> 2;
    for (int64_t q0 = (lo >> 2) + tid; q0 < q_hi; q0 += kLoadBatch * kPickThreads) {
      float4 v[kLoadBatch];
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int64_t q = q0 + static_cast<int64_t>(u) * kPickThreads;
        v[u] = q < q_hi ? __ldcg(reinterpret_cast<const float4*>(src) + q)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        if (q0 + static_cast<int64_t>(u) * kPickThreads >= q_hi) break;
        atomicAdd(&hist[order_key(v[u].x) >> 21], 1u);
        atomicAdd(&hist[order_key(v[u].y) >> 21], 1u);
        atomicAdd(&hist[order_key(v[u].z) >> 21], 1u);
        atomicAdd(&hist[order_key(v[u].w) >> 21], 1u);
      }
    }
    for (int64_t e = (q_hi << 2) + tid; e < hi; e += kPickThreads)
      atomicAdd(&hist[order_key(__ldcg(src + e)) >> 21], 1u);
  } else {
    for (int64_t e = lo + tid; e < hi; e += kPickThreads)
      atomicAdd(&hist[order_key(__ldcg(src + e)) >> 21], 1u);
  }
  __syncthreads();
  uint16_t* dst = a.hist + (row * a.S + s) * kBins;
  for (int i = tid; i < kBins; i += kPickThreads) dst[i] = static_cast<uint16_t>(hist[i]);
}

// The ranking of the row's candidates by its last CTA: `need` more entries
// are taken from the C candidates (all in the threshold bin d0), written to
// rest[0 .. need).  idx_of(c) / key_of(c) give candidate c's entry index and
// order-preserving key.
template <class IdxOf, class KeyOf>
__device__ __forceinline__ void rank_candidates(int C, uint32_t need, uint32_t d0, int32_t* rest,
                                                SliceShared& sh, IdxOf idx_of, KeyOf key_of) {
  const int tid = threadIdx.x;
  const int room = static_cast<int>(need);
  // the two remaining digits of the need-th largest candidate key
  uint32_t prefix = d0;
  for (int pass = 0; pass < 2; ++pass) {
    const int width = pass == 0 ? 11 : 10;
    const int shift = pass == 0 ? 10 : 0;
    const int nb = 1 << width;
    for (int i = tid; i < kBins; i += kPickThreads) sh.hist[i] = 0;
    __syncthreads();
    for (int c = tid; c < C; c += kPickThreads) {
      const uint32_t key = key_of(c);
      if ((key >> (shift + width)) == prefix) atomicAdd(&sh.hist[(key >> shift) & (nb - 1)], 1u);
    }
    __syncthreads();
    find_digit_desc(sh.hist, nb, need, &sh.scan, tid, kPickThreads);
    prefix = (prefix << width) | sh.scan.digit;
    need -= sh.scan.above;
  }
  const uint32_t thr = prefix;  // the k-th largest key; `need` of its ties are taken
  // candidates above the threshold, and the count of ties at it (the loop
  // runs the same trip count in every thread: warp_append is warp-collective)
  if (tid == 0) {
    sh.n_gt = 0;
    sh.n_eq = 0;
  }
  __syncthreads();
  int eq = 0;
  for (int c0 = 0; c0 < C; c0 += kPickThreads) {
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
      for (int i = tid; i < kBins; i += kPickThreads) sh.hist[i] = 0;
      __syncthreads();
      for (int c = tid; c < C; c += kPickThreads) {
        if (key_of(c) != thr) continue;
        const uint32_t j = static_cast<uint32_t>(idx_of(c));
        if (pass > 0 && (j >> (shift + width)) != ip) continue;
        atomicAdd(&sh.hist[(j >> shift) & (nb - 1)], 1u);
      }
      __syncthreads();
      find_digit_asc(sh.hist, nb, left, &sh.scan, tid, kPickThreads);
      ip = (ip << width) | sh.scan.digit;
      left -= sh.scan.above;
    }
    ti = ip;  // indices are distinct: the ties with index <= ti are exactly `need`
  }
  if (tid == 0) sh.n_gt = 0;
  __syncthreads();
  int32_t* ties_out = rest + n_gt;
  for (int c0 = 0; c0 < C; c0 += kPickThreads) {
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

__global__ void __launch_bounds__(kPickThreads) topk_pick_kernel(const TopkArgs a) {
  __shared__ SliceShared sh;
  extern __shared__ __align__(16) uint8_t pick_dyn[];  // the last CTA's candidates
  const int tid = threadIdx.x;
  const int s = blockIdx.x;
  const int64_t row = static_cast<int64_t>(blockIdx.y) + static_cast<int64_t>(gridDim.y) * blockIdx.z;
  pdl_trigger();
  pdl_wait();  // the histograms (and the scores before them) are complete
  if (row >= a.rows) return;
  const int64_t n = visible_count(a.pos[row], a.m, a.N_cap);
  int32_t* out = a.idx + row * a.k;
  const int64_t lo = static_cast<int64_t>(s) * a.slice;
  const int64_t hi = lo + a.slice < n ? lo + a.slice : n;
  if (n <= a.k) {
    // every visible entry is selected; CTA 0 pads
    for (int64_t e = lo + tid; e < hi; e += kPickThreads) out[e] = static_cast<int32_t>(e);
    if (s == 0)
      for (int64_t e = n + tid; e < a.k; e += kPickThreads) out[e] = -1;
    return;
  }
  // the row's histogram: the sum of its S slices' bins.  Thread t sums bin
  // pairs t and t + 512 (one 32-bit load holds two 16-bit bins) with up to
  // kSumBatch slices' loads in flight at once, so a row of up to kSumBatch
  // slices costs one round of memory latency.
  static_assert(kBins == 4 * kPickThreads, "two bin pairs per thread");
  {
    const uint32_t* rh = reinterpret_cast<const uint32_t*>(a.hist + row * a.S * kBins);
    uint32_t c[4] = {0u, 0u, 0u, 0u};
    for (int q0 = 0; q0 < a.S; q0 += kSumBatch) {
      uint32_t v0[kSumBatch], v1[kSumBatch];
#pragma unroll
      for (int u = 0; u < kSumBatch; ++u) {
        const bool in = q0 + u < a.S;
        const uint32_t* p = rh + (q0 + u) * (kBins / 2) + tid;
        v0[u] = in ? __ldcg(p) : 0u;
        v1[u] = in ? __ldcg(p + kPickThreads) : 0u;
      }
#pragma unroll
      for (int u = 0; u < kSumBatch; ++u) {
        c[0] += v0[u] & 0xffffu;
        c[1] += v0[u] >> 16;
        c[2] += v1[u] & 0xffffu;
        c[3] += v1[u] >> 16;
      }
    }
    sh.hist[2 * tid] = c[0];
    sh.hist[2 * tid + 1] = c[1];
    sh.hist[2 * (tid + kPickThreads)] = c[2];
    sh.hist[2 * (tid + kPickThreads) + 1] = c[3];
  }
  if (tid == 0) {
    sh.n_up = 0;
    sh.n_in = 0;
  }
  __syncthreads();
  find_digit_desc(sh.hist, kBins, static_cast<uint32_t>(a.k), &sh.scan, tid, kPickThreads);
  const uint32_t d0 = sh.scan.digit;
  const uint32_t n_above = sh.scan.above;  // keys in bins above d0: all selected
  int* ctr = a.ctr + row * 4;              // [0] above appended, [1] candidates, [2] tickets
  int32_t* cand = a.cand + row * a.N_cap;
  const float* src = a.scores + row * a.N_cap;
  // Sweep the slice: above the bin -> the output, in the bin -> the
  // candidates.  Both go to shared-memory lists first (a slice holds few of
  // either), then one global reservation per list; entries beyond a list's
  // capacity (a slice of near-equal scores) are appended one by one.
  auto place = [&](int64_t e, float v) {
    const uint32_t d = order_key(v) >> 21;
    if (d > d0) {
      const int p = atomicAdd(&sh.n_up, 1);
      if (p < kListCap) {
        sh.up[p] = static_cast<int32_t>(e);
      } else {
        const int q = atomicAdd(&ctr[0], 1);
        if (q < a.k) out[q] = static_cast<int32_t>(e);
      }
    } else if (d == d0) {
      const int p = atomicAdd(&sh.n_in, 1);
      if (p < kListCap) {
        sh.in[p] = static_cast<int32_t>(e);
      } else {
        const int q = atomicAdd(&ctr[1], 1);
        if (q < a.N_cap) cand[q] = static_cast<int32_t>(e);
      }
    }
  };
  if (hi <= lo) {
    // nothing visible in this slice
  } else if (a.vec4) {
    const int64_t q_hi = hi >> 2;
    for (int64_t q0 = (lo >> 2) + tid; q0 < q_hi; q0 += kLoadBatch * kPickThreads) {
      float4 v[kLoadBatch];
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int64_t q = q0 + static_cast<int64_t>(u) * kPickThreads;
        v[u] = q < q_hi ? __ldcg(reinterpret_cast<const float4*>(src) + q)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int64_t q = q0 + static_cast<int64_t>(u) * kPickThreads;
        if (q >= q_hi) break;
        place(4 * q, v[u].x);
        place(4 * q + 1, v[u].y);
        place(4 * q + 2, v[u].z);
        place(4 * q + 3, v[u].w);
      }
    }
    for (int64_t e = (q_hi << 2) + tid; e < hi; e += kPickThreads) place(e, __ldcg(src + e));
  } else {
    for (int64_t e = lo + tid; e < hi; e += kPickThreads) place(e, __ldcg(src + e));
  }
  __syncthreads();
  const int nu = min(sh.n_up, kListCap), ni = min(sh.n_in, kListCap);
  if (tid == 0) {
    sh.base_up = nu ? atomicAdd(&ctr[0], nu) : 0;
    sh.base_in = ni ? atomicAdd(&ctr[1], ni) : 0;
  }
  __syncthreads();
  for (int i = tid; i < nu; i += kPickThreads)
    if (sh.base_up + i < a.k) out[sh.base_up + i] = sh.up[i];
  for (int i = tid; i < ni; i += kPickThreads)
    if (sh.base_in + i < a.N_cap) cand[sh.base_in + i] = sh.in[i];
  // the last CTA of the row to get here ranks the candidates
  __threadfence();
  __syncthreads();
  if (tid == 0) sh.last = atomicAdd(&ctr[2], 1) == a.S - 1;
  __syncthreads();
  if (!sh.last) return;
  __threadfence();
  const int C = min(__ldcg(&ctr[1]), static_cast<int>(a.N_cap));
  const uint32_t need = static_cast<uint32_t>(a.k) - n_above;  // 1 <= need <= C
  int32_t* rest = out + n_above;
  if (static_cast<int>(need) >= C) {
    for (int c = tid; c < C; c += kPickThreads) rest[c] = __ldcg(cand + c);
    return;
  }
  if (C <= kCandSmem) {
    // the candidates and their keys into shared memory, in one gather
    int32_t* cj = reinterpret_cast<int32_t*>(pick_dyn);
    uint32_t* ck = reinterpret_cast<uint32_t*>(pick_dyn + kCandSmem * 4);
    for (int c0 = tid; c0 < C; c0 += kLoadBatch * kPickThreads) {
      int32_t j[kLoadBatch];
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int c = c0 + u * kPickThreads;
        j[u] = c < C ? __ldcg(cand + c) : 0;
      }
      float v[kLoadBatch];
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) v[u] = __ldcg(src + j[u]);
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int c = c0 + u * kPickThreads;
        if (c < C) {
          cj[c] = j[u];
          ck[c] = order_key(v[u]);
        }
      }
    }
    __syncthreads();
    rank_candidates(C, need, d0, rest, sh, [&](int c) { return cj[c]; },
                    [&](int c) { return ck[c]; });
  } else {
    rank_candidates(C, need, d0, rest, sh, [&](int c) { return __ldcg(cand + c); },
                    [&](int c) { return order_key(__ldcg(src + __ldcg(cand + c))); });
  }
}

}  // namespace

static_assert(sizeof(RowShared) + kRowMaxKeys * 4 <= 227 * 1024,
              "a 49,152-key row and the shared state fit one CTA's shared memory");

bool plan_topk(int64_t rows, int64_t N_cap, int k, int num_sms, TopkPlan* p) {
  if (rows <= 0 || N_cap < 1 || k < 1) return false;
  *p = TopkPlan{};
  // Few long rows spread over many CTAs (slice path); otherwise one CTA per
  // row with the keys in shared memory (row path).
  const bool row_fits = N_cap <= kRowMaxKeys;
  const bool few_rows = rows * 2 < num_sms;
  if (row_fits && (!few_rows || N_cap <= 8192)) {
    p->slice_path = false;
    p->S = 1;
    p->threads = N_cap >= 8192 ? 1024 : (N_cap >= 2048 ? 512 : 256);
    p->smem_bytes = sizeof(RowShared) + static_cast<size_t>(N_cap) * 4;
  } else {
    p->slice_path = true;
    // about one CTA per SM over all rows; a slice is a multiple of 64
    // entries and holds at most 65,535 (the bins are 16-bit)
    int64_t S = num_sms / rows;
    if (S < 1) S = 1;
    int64_t slice = ((N_cap + S - 1) / S + 63) / 64 * 64;
    if (slice > 65472) slice = 65472;
    S = (N_cap + slice - 1) / slice;
    if (S > 65535) return false;
    p->S = static_cast<int>(S);
    p->slice = slice;
    p->threads = kPickThreads;
    p->smem_bytes = 0;
  }
  p->ws_bytes = topk_scratch_bytes(*p, rows, N_cap);
  return true;
}

size_t topk_scratch_bytes(const TopkPlan& p, int64_t rows, int64_t N_cap) {
  if (!p.slice_path) return 0;
  const size_t hist = static_cast<size_t>(rows) * p.S * kBins * sizeof(uint16_t);
  const size_t ctr = static_cast<size_t>(rows) * 4 * sizeof(int32_t);
  const size_t cand = static_cast<size_t>(rows) * N_cap * sizeof(int32_t);
  return (hist + 255) / 256 * 256 + (ctr + 255) / 256 * 256 + cand;
}

void topk_scratch_carve(const TopkPlan& p, int64_t rows, void* ws, TopkArgs* a) {
  uint8_t* b = static_cast<uint8_t*>(ws);
  const size_t hist = static_cast<size_t>(rows) * p.S * kBins * sizeof(uint16_t);
  const size_t ctr = static_cast<size_t>(rows) * 4 * sizeof(int32_t);
  a->hist = reinterpret_cast<uint16_t*>(b);
  b += (hist + 255) / 256 * 256;
  a->ctr = reinterpret_cast<int32_t*>(b);
  b += (ctr + 255) / 256 * 256;
  a->cand = reinterpret_cast<int32_t*>(b);
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
  cudaLaunchAttribute at[1];
  cfg.attrs = at;
  cfg.numAttrs = add_dependent_attr(at, 0, dependent);
  TopkArgs args = a;
  args.S = p.S;
  args.slice = p.slice;
  args.vec4 = (a.N_cap % 4 == 0) && (reinterpret_cast<uintptr_t>(a.scores) % 16 == 0) &&
              (p.slice % 4 == 0);
  cudaError_t e;
  if (!p.slice_path) {
    e = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(p.smem_bytes));
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(1, static_cast<unsigned>(gy), static_cast<unsigned>(gz));
    cfg.dynamicSmemBytes = p.smem_bytes;
    e = cudaLaunchKernelEx(&cfg, topk_row_kernel, args);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  cfg.gridDim = dim3(p.S, static_cast<unsigned>(gy), static_cast<unsigned>(gz));
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, topk_hist_kernel, args);
  if (e != cudaSuccess) return e;
  // the pick kernel reads what the histogram kernel wrote: always a
  // dependent of it (it waits before its first read)
  cfg.numAttrs = add_dependent_attr(at, 0, true);
  cfg.dynamicSmemBytes = kCandSmem * 8;
  e = cudaFuncSetAttribute(topk_pick_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kCandSmem * 8);
  if (e != cudaSuccess) return e;
  e = cudaLaunchKernelEx(&cfg, topk_pick_kernel, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hattn
