// topk.cu -- exact per-query top-k over the indexer scores.
//
// "Why DeepSeek V4 Stands Apart", section "Core Architectural Innovations":
// CSA keeps the top-1024 (Pro) / top-512 (Flash) compressed entries per
// query.  Selection rule: the min(k, n) largest scores among the n visible
// entries, ties to the smaller entry index; the output order is unspecified.
//
// One thread-block cluster of C CTAs handles one query row: CTA `rank` holds
// entries [rank*slice, (rank+1)*slice) as order-preserving uint32 keys in
// shared memory (one read of the fp32 scores).  Three radix passes (11, 11,
// 10 bits, most significant first) find the k-th largest key: every CTA
// builds a shared-memory histogram of the digit among the keys that still
// match the prefix and adds its nonzero bins into every CTA's copy of the
// cluster histogram with remote shared-memory atomics (double-buffered, so
// one cluster barrier per pass); every CTA then finds the digit with a
// block-wide suffix scan.  The final pass writes every key above the
// threshold, then the threshold ties in global index order until k are
// written.  No global atomics, no inter-kernel passes; the result is
// deterministic.
#include <cooperative_groups.h>

#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace cg = cooperative_groups;

namespace hattn {

namespace {

constexpr int kBins = 2048;
// Keys in the first pass's threshold bin, whole cluster, up to which the
// compact path is taken; keys above that bin number fewer than k <= 2048.
// Slice positions fit 16 bits (a slice holds at most 49,152 keys).
constexpr int kMaxCand = 2048;
constexpr int kMaxAbove = 2048;

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct TopkShared {
  uint32_t hist[kBins];
  uint32_t ghist[2][kBins];
  uint32_t warp_tot[32];
  int counts[2];       // keys above the threshold, keys equal to it (this CTA)
  int offs[2];         // the same counts summed over the lower-ranked CTAs
  int ctr, ctr_eq;
  int eq_total;        // keys equal to the threshold in the whole cluster
  int n_cand, n_above;
  uint16_t cand[kMaxCand];        // slice positions of the keys in the bin of the k-th largest
  uint16_t above_idx[kMaxAbove];  // slice positions of the keys above that bin
  uint32_t digit;
  uint32_t above;
};

// Inclusive scan over the threads of the block, in thread order; uses
// sh->warp_tot.  Returns this thread's exclusive prefix.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, TopkShared* sh, int tid,
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

// The bin holding the need-th largest key: bins are visited from the top;
// sh->digit = that bin, sh->above = the keys in the bins above it.
__device__ __forceinline__ void find_digit(const uint32_t* gh, int nb, uint32_t need,
                                           TopkShared* sh, int tid, int nthr) {
  const int bpt = nb / nthr;            // bins per thread (nb >= nthr)
  const int hi = nb - bpt * tid;        // this thread's bins: [hi - bpt, hi)
  uint32_t tot = 0;
  for (int i = 0; i < bpt; ++i) tot += gh[hi - 1 - i];
  const uint32_t before = block_exclusive_scan(tot, sh, tid, nthr);
  if (before < need && before + tot >= need) {
    uint32_t run = before;
    for (int i = 0; i < bpt; ++i) {
      const uint32_t c = gh[hi - 1 - i];
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

__global__ void topk_kernel(const TopkArgs a) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  TopkShared* sh = reinterpret_cast<TopkShared*>(smem_raw);
  uint32_t* keys = reinterpret_cast<uint32_t*>(smem_raw + sizeof(TopkShared));

  cg::cluster_group cluster = cg::this_cluster();
  const int C = a.cluster;
  const int rank = static_cast<int>(cluster.block_rank());
  const int row = blockIdx.y;
  const int tid = threadIdx.x;
  const int nthr = blockDim.x;

  pdl_trigger();
  pdl_wait();  // the scores (and a dependent launch's predecessor) are complete
  const int32_t t = a.pos[row];
  int64_t n = t < 0 ? 0 : (static_cast<int64_t>(t) + 1) / a.m;
  if (n > a.N_cap) n = a.N_cap;
  const int64_t start = static_cast<int64_t>(rank) * a.slice;
  int len = 0;
  if (n > start) len = static_cast<int>((n - start) < a.slice ? (n - start) : a.slice);
  int32_t* out = a.idx + static_cast<int64_t>(row) * a.k;

  if (n <= a.k) {  // every visible entry is selected (same branch for the whole cluster)
    for (int e = tid; e < len; e += nthr) out[start + e] = static_cast<int32_t>(start + e);
    if (rank == 0)
      for (int64_t p = n + tid; p < a.k; p += nthr) out[p] = -1;
    return;
  }

  const float* src = a.scores + static_cast<int64_t>(row) * a.N_cap + start;
  for (int i = tid; i < kBins; i += nthr) {
    sh->hist[i] = 0;
    sh->ghist[0][i] = 0;
    sh->ghist[1][i] = 0;
  }
  __syncthreads();
  // the keys, and the first pass's histogram of their top 11 bits, in one sweep
  for (int e = tid; e < len; e += nthr) {
    const uint32_t key = order_key(src[e]);
    keys[e] = key;
    atomicAdd(&sh->hist[key >> 21], 1u);
  }
  cluster.sync();  // every copy of the cluster histogram is zero before any add

  uint32_t prefix = 0;
  uint32_t need = static_cast<uint32_t>(a.k);
  // One radix pass over the histogram in sh->hist: add this CTA's nonzero
  // bins into every CTA's copy of the cluster histogram (buffer pass & 1),
  // reset the local bins and the other buffer (last scanned by this CTA in
  // the previous pass; the next adds into it come after the barrier), then
  // find the digit of the need-th largest key.
  auto radix_pass = [&](int pass, int width) {
    const int nb = 1 << width;
    const int buf = pass & 1;
    __syncthreads();
    for (int bin = tid; bin < nb; bin += nthr) {
      const uint32_t v = sh->hist[bin];
      if (v) {
        for (int q = 0; q < C; ++q) atomicAdd(cluster.map_shared_rank(&sh->ghist[buf][bin], q), v);
        sh->hist[bin] = 0;
      }
    }
    if (pass < 2)
      for (int i = tid; i < kBins; i += nthr) sh->ghist[buf ^ 1][i] = 0;
    cluster.sync();
    find_digit(sh->ghist[buf], nb, need, sh, tid, nthr);
    prefix = (prefix << width) | sh->digit;
    need -= sh->above;
  };
  radix_pass(0, 11);  // its histogram was built while loading
  // The keys left to rank are those in the bin of the k-th largest (about
  // 0.5% of normal scores).  When the whole cluster holds few enough, one
  // sweep lists them (and the keys above the bin, which are selected), and
  // the remaining passes, the counts and the writes visit only the lists.
  // The decision uses the cluster histogram, so every CTA takes the same path.
  const bool compact = sh->ghist[0][prefix] <= static_cast<uint32_t>(kMaxCand);
  int n_cand = 0, n_above = 0;
  if (compact) {
    if (tid == 0) {
      sh->n_cand = 0;
      sh->n_above = 0;
    }
    __syncthreads();
    // few keys qualify, so each takes its place with its own atomic
    for (int e = tid; e < len; e += nthr) {
      const uint32_t key = keys[e];
      const uint32_t d = key >> 21;
      if (d == prefix) {
        sh->cand[atomicAdd(&sh->n_cand, 1)] = static_cast<uint16_t>(e);
        atomicAdd(&sh->hist[(key >> 10) & 2047u], 1u);
      } else if (d > prefix) {
        sh->above_idx[atomicAdd(&sh->n_above, 1)] = static_cast<uint16_t>(e);
      }
    }
    __syncthreads();
    n_cand = sh->n_cand;
    n_above = sh->n_above;
    radix_pass(1, 11);
    for (int c = tid; c < n_cand; c += nthr) {
      const uint32_t key = keys[sh->cand[c]];
      if ((key >> 10) == prefix) atomicAdd(&sh->hist[key & 1023u], 1u);
    }
    radix_pass(2, 10);
  } else {
    for (int e = tid; e < len; e += nthr) {
      const uint32_t key = keys[e];
      if ((key >> 21) == prefix) atomicAdd(&sh->hist[(key >> 10) & 2047u], 1u);
    }
    radix_pass(1, 11);
    for (int e = tid; e < len; e += nthr) {
      const uint32_t key = keys[e];
      if ((key >> 10) == prefix) atomicAdd(&sh->hist[key & 1023u], 1u);
    }
    radix_pass(2, 10);
  }
  const uint32_t thr = prefix;  // the k-th largest key; take `need` of its ties

  if (tid == 0) {
    sh->counts[0] = 0;
    sh->counts[1] = 0;
    sh->ctr = 0;
    sh->ctr_eq = 0;
  }
  __syncthreads();
  int gt = 0, eq = 0;
  if (compact) {
    if (tid == 0) gt = n_above;
    for (int c = tid; c < n_cand; c += nthr) {
      const uint32_t key = keys[sh->cand[c]];
      gt += key > thr;
      eq += key == thr;
    }
  } else {
    for (int e = tid; e < len; e += nthr) {
      gt += keys[e] > thr;
      eq += keys[e] == thr;
    }
  }
  if (gt) atomicAdd(&sh->counts[0], gt);
  if (eq) atomicAdd(&sh->counts[1], eq);
  cluster.sync();
  if (tid < 32) {
    // counts of the lower-ranked CTAs, and the cluster's tie total, summed by
    // one warp (C <= 32)
    int g = 0, e = 0, et = 0;
    if (tid < C) {
      const int* rc = cluster.map_shared_rank(sh->counts, tid);
      et = rc[1];
      if (tid < rank) {
        g = rc[0];
        e = et;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      g += __shfl_xor_sync(0xffffffffu, g, o);
      e += __shfl_xor_sync(0xffffffffu, e, o);
      et += __shfl_xor_sync(0xffffffffu, et, o);
    }
    if (tid == 0) {
      sh->offs[0] = g;
      sh->offs[1] = e;
      sh->eq_total = et;
    }
  }
  __syncthreads();
  const int off_gt = sh->offs[0];
  const int off_eq = sh->offs[1];
  const int base = a.k - static_cast<int>(need);  // ties go to [base, k)
  const bool all_ties = sh->eq_total == static_cast<int>(need);
  if (compact) {
    // keys above the threshold bin, then the candidates above or (when every
    // tie is selected) at the threshold: any order
    for (int c = tid; c < n_above; c += nthr) {
      const int p = atomicAdd(&sh->ctr, 1);
      out[off_gt + p] = static_cast<int32_t>(start + sh->above_idx[c]);
    }
    for (int c = tid; c < n_cand; c += nthr) {
      const int e = sh->cand[c];
      const uint32_t key = keys[e];
      if (key > thr) {
        const int p = atomicAdd(&sh->ctr, 1);
        out[off_gt + p] = static_cast<int32_t>(start + e);
      } else if (key == thr && all_ties) {
        const int p = atomicAdd(&sh->ctr_eq, 1);
        out[base + off_eq + p] = static_cast<int32_t>(start + e);
      }
    }
  } else if (all_ties) {
    // every tie is selected (the usual case: one key holds the k-th score),
    // so no order is needed: keys above and at the threshold are appended
    for (int e = tid; e < len; e += nthr) {
      const uint32_t key = keys[e];
      if (key > thr) {
        const int p = atomicAdd(&sh->ctr, 1);
        out[off_gt + p] = static_cast<int32_t>(start + e);
      } else if (key == thr) {
        const int p = atomicAdd(&sh->ctr_eq, 1);
        out[base + off_eq + p] = static_cast<int32_t>(start + e);
      }
    }
  } else {
    // keys above the threshold: any order
    for (int e = tid; e < len; e += nthr) {
      if (keys[e] > thr) {
        const int p = atomicAdd(&sh->ctr, 1);
        out[off_gt + p] = static_cast<int32_t>(start + e);
      }
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
    uint32_t rnk = static_cast<uint32_t>(off_eq) + block_exclusive_scan(c, sh, tid, nthr);
    for (int j = 0; j < n_run && c > 0 && rnk < need; ++j) {
      if (keys[e0 + j] == thr) {
        out[base + rnk] = static_cast<int32_t>(start + e0 + j);
        ++rnk;
        --c;
      }
    }
  }
  cluster.sync();  // keep this CTA's shared memory alive for the others' reads
}

// Clusters of C CTAs (threads, smem per CTA) that the device can hold at
// once; queried once per (device, shape) and remembered.
struct OccKey {
  int dev, C, threads;
  size_t smem;
  int n;
};
OccKey g_occ[64];
int g_nocc = 0;
std::mutex g_occ_mu;

int query_active_clusters(int C, int threads, size_t smem);

int max_active_clusters(int C, int threads, size_t smem) {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lk(g_occ_mu);
  for (int i = 0; i < g_nocc; ++i)
    if (g_occ[i].dev == dev && g_occ[i].C == C && g_occ[i].threads == threads &&
        g_occ[i].smem == smem)
      return g_occ[i].n;
  const int n = query_active_clusters(C, threads, smem);
  if (g_nocc < 64) g_occ[g_nocc++] = OccKey{dev, C, threads, smem, n};
  return n;
}

int query_active_clusters(int C, int threads, size_t smem) {
  if (C > 8) cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem)) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = C;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, topk_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

void fill_plan(int C, int64_t N_cap, TopkPlan* p) {
  int slice = static_cast<int>((N_cap + C - 1) / C);
  if (slice < 1) slice = 1;
  p->cluster = C;
  p->slice = slice;
  p->threads = slice >= 8192 ? 1024 : (slice >= 2048 ? 512 : 256);
  p->smem_bytes = sizeof(TopkShared) + static_cast<size_t>(slice) * 4;
}

}  // namespace

static_assert(sizeof(TopkShared) + 49152 * 4 <= 227 * 1024,
              "a 49,152-key slice and the shared state fit one CTA's shared memory");

bool plan_topk(int rows, int64_t N_cap, int num_sms, TopkPlan* p) {
  if (rows <= 0 || N_cap < 0) return false;
  const int64_t max_slice = 49152;  // keys per CTA held in shared memory
  int C = 1;
  // spread small batches over more SMs, keep slices large enough to be worth it
  while (C < 16 && (int64_t)rows * C < num_sms && (N_cap + 2 * C - 1) / (2 * C) >= 2048) C *= 2;
  while (C < 16 && (N_cap + C - 1) / C > max_slice) C *= 2;
  if ((N_cap + C - 1) / C > max_slice) return false;
  // Clusters that do not all fit on the device at once run in waves, and a
  // second wave repeats every fixed cost (the barriers and scans of each
  // pass, about as much as 16K keys of work).  Take the cluster size with the
  // least (waves x (keys per CTA + 16K)), the larger size on ties.
  int64_t best_cost = -1;
  TopkPlan best = {};
  for (int c = C; c >= 1; c >>= 1) {
    if ((N_cap + c - 1) / c > max_slice) break;
    TopkPlan q;
    fill_plan(c, N_cap, &q);
    const int n = max_active_clusters(c, q.threads, q.smem_bytes);
    if (n < 1) continue;
    const int64_t waves = (rows + n - 1) / n;
    const int64_t cost = waves * (q.slice + 16384);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = q;
    }
  }
  if (best_cost < 0) return false;
  *p = best;
  return true;
}

cudaError_t launch_topk(const TopkArgs& a, const TopkPlan& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(p.smem_bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.cluster, a.rows, 1);
  cfg.blockDim = dim3(p.threads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = p.cluster;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = add_dependent_attr(at, 1);
  TopkArgs args = a;
  args.cluster = p.cluster;
  args.slice = p.slice;
  e = cudaLaunchKernelEx(&cfg, topk_kernel, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hattn
