// indexer.cu -- lightning-indexer scores on the tcgen05 tensor cores.
//
// "DeepSeek-V4" atlas, section "Design overview": CSA applies the V3.2
// lightning-indexer sparse attention over the compressed entries.  The score
// of compressed entry j for query t is
//     I(t, j) = sum_h w[t,h] * max(0, qI[t,h] . kI[j]).
//
// As a contraction: one 128-entry block of indexer keys (A, M=128 rows, K=dI)
// times the indexer queries of a group of G queries (B, N = G*HI rows padded
// to a multiple of 16, K=dI) gives a 128 x N fp32 tile in tensor memory; the
// epilogue applies ReLU, the per-head weights and the per-query head sum.
//
// Work = (query group, 128-entry block) slots, flattened and split evenly
// over a grid of one CTA per SM.  Roles: warp 0 issues TMA loads of key
// blocks (128B-swizzled, a ring of `stages` buffers) and of the group's
// queries; warp 1 issues the MMAs (M=128, N=NQ, K=16 steps) into one of two
// tensor-memory accumulators; warps 2-5 drain an accumulator (tcgen05.ld),
// reduce it and write fp32 scores with coalesced stores.  HBM traffic is the
// key blocks once plus the scores.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kIdxThreads = 224;  // producer, MMA (even slots), 4 epilogue warps, MMA (odd slots)
constexpr int kBlockRows = 128;
constexpr int kMaxStages = 8;

struct IdxSmem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t qfull;
  uint64_t qempty;
  uint64_t mma_done[2];
  uint32_t tmem_base;
  int abort;
  // per epilogue warp (no cross-warp barrier): visible entries per query of
  // the current group, and the head weight of every accumulator column
  int nt[4][256];
  alignas(16) float wcol[4][256];
};

__device__ __forceinline__ int64_t visible_entries(int32_t t, int m, int64_t cap) {
  int64_t n = t < 0 ? 0 : (static_cast<int64_t>(t) + 1) / m;
  return n < cap ? n : cap;
}

// Walks this CTA's slots in order.  Every role runs the same cursor, so all
// of them skip the same blocks; the 64-bit divisions happen only when the
// query group changes, never per slot.
struct SlotCursor {
  int64_t slot, end;
  int64_t group;   // b * groups_per_seq + query group within the sequence
  int blk;         // 128-entry block within the sequence
  int b, t0, gv;
  int64_t nmax;    // largest visible-entry count among the group's queries

  __device__ __forceinline__ void load_group(const IndexerArgs& a) {
    b = static_cast<int>(group / a.groups_per_seq);
    t0 = static_cast<int>(group - static_cast<int64_t>(b) * a.groups_per_seq) * a.G;
    gv = min(a.G, a.T - t0);
    nmax = 0;
    for (int g = 0; g < gv; ++g) {
      const int64_t v = visible_entries(a.pos[(int64_t)b * a.T + t0 + g], a.m, a.N_cap);
      nmax = v > nmax ? v : nmax;
    }
  }
  __device__ __forceinline__ void init(const IndexerArgs& a, int64_t s0, int64_t s1) {
    slot = s0;
    end = s1;
    group = s0 / a.nblk;
    blk = static_cast<int>(s0 - group * a.nblk);
    if (slot < end) load_group(a);
  }
  __device__ __forceinline__ bool live() const {
    return static_cast<int64_t>(blk) * kBlockRows < nmax;
  }
  // next slot; a dead block ends its group (the later blocks are dead too)
  __device__ __forceinline__ void advance(const IndexerArgs& a) {
    if (!live()) {
      slot += a.nblk - 1 - blk;
      blk = a.nblk - 1;
    }
    ++slot;
    if (++blk == a.nblk) {
      blk = 0;
      ++group;
      if (slot < end) load_group(a);
    }
  }
};

__global__ void __launch_bounds__(kIdxThreads, 1)
    indexer_score_kernel(const __grid_constant__ CUtensorMap tm_ik,
                         const __grid_constant__ CUtensorMap tm_iq, const IndexerArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128B-swizzled operand buffers
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t q_bytes = static_cast<uint32_t>(a.KC) * a.NQ * 128u;
  const uint32_t stage_bytes = static_cast<uint32_t>(a.KC) * 16384u;
  uint8_t* sQ = base;
  uint8_t* sA = base + q_bytes;
  IdxSmem* sm = reinterpret_cast<IdxSmem*>(sA + a.stages * stage_bytes);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();  // top-k may begin launching as SMs free up

  const int64_t s0 = a.total_slots * blockIdx.x / gridDim.x;
  const int64_t s1 = a.total_slots * (blockIdx.x + 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(smem_u32(&sm->full[i]), 1);
      mbar_init(smem_u32(&sm->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm->tfull[i]), 1);
      mbar_init(smem_u32(&sm->tempty[i]), 128);
    }
    mbar_init(smem_u32(&sm->qfull), 1);
    mbar_init(smem_u32(&sm->qempty), 2);  // both MMA issuers leave the query block
    mbar_init(smem_u32(&sm->mma_done[0]), 1);
    mbar_init(smem_u32(&sm->mma_done[1]), 1);
    sm->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_ik);
    tma_prefetch_desc(&tm_iq);
  }
  const uint32_t tmem_cols = (2 * a.NQ <= 32) ? 32 : (2 * a.NQ <= 64 ? 64 : (2 * a.NQ <= 128 ? 128 : (2 * a.NQ <= 256 ? 256 : 512)));
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort = &sm->abort;

  // Ring positions are tracked as (stage, phase) pairs advanced by one per
  // use, so the loops below divide nothing per slot.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      SlotCursor cur;
      int st = 0;
      uint32_t ph = 0;
      int64_t it = 0, qloads = 0, loaded = -1;
      bool keys_ready = false;  // the compressed keys of the previous kernel are visible
      for (cur.init(a, s0, s1); cur.slot < cur.end && !*abort; cur.advance(a)) {
        if (!cur.live()) continue;
        if (cur.group != loaded) {
          if (qloads > 0 &&
              !mbar_wait(smem_u32(&sm->qempty), (qloads - 1) & 1, abort, a.status, kWaitLimitNs, 10))
            break;
          const uint32_t qb = smem_u32(&sm->qfull);
          mbar_arrive_expect_tx(qb, q_bytes);
          const int row0 = ((cur.b * a.T) + cur.t0) * a.HI;
          for (int kc = 0; kc < a.KC; ++kc)
            tma_load_2d(smem_u32(sQ + kc * a.NQ * 128), &tm_iq, kc * 64, row0, qb);
          ++qloads;
          loaded = cur.group;
        }
        // stage st was last filled `stages` uses ago, in phase ph ^ 1
        if (it >= a.stages &&
            !mbar_wait(smem_u32(&sm->empty[st]), ph ^ 1u, abort, a.status, kWaitLimitNs, 11))
          break;
        if (!keys_ready &&
            (a.fresh_from < 0 || static_cast<int64_t>(cur.blk + 1) * kBlockRows > a.fresh_from)) {
          // a dependent launch waits here, before the first block that holds
          // entries its predecessor may have written (the other blocks stream
          // while that kernel still runs)
          pdl_wait();
          keys_ready = true;
        }
        const uint32_t fb = smem_u32(&sm->full[st]);
        mbar_arrive_expect_tx(fb, stage_bytes);
        for (int kc = 0; kc < a.KC; ++kc)
          tma_load_3d(smem_u32(sA + st * stage_bytes + kc * 16384), &tm_ik, kc * 64,
                      cur.blk * kBlockRows, cur.b, fb);
        ++it;
        if (++st == a.stages) { st = 0; ph ^= 1u; }
      }
      if (*abort) {
        // let the copies already issued land before the CTA exits
        const int64_t first = it > a.stages ? it - a.stages : 0;
        for (int64_t x = first; x < it; ++x)
          mbar_wait(smem_u32(&sm->full[x % a.stages]), (x / a.stages) & 1, nullptr, nullptr,
                    10000000ull, 12);
      }
    }
  } else if (warp == 1 || warp == 6) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues the products of the even live slots (accumulator 0) and
    // warp 6 those of the odd ones (accumulator 1): a single thread issues a
    // chained tcgen05.mma only every ~64 ns, close to a slot's share of the
    // key stream, so two issuers keep the tensor core ahead of it.
    const int par = warp == 1 ? 0 : 1;
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(128, a.NQ, 0, 0);
      SlotCursor cur;
      int st = 0;
      uint32_t ph = 0;
      int64_t it = 0, qn = 0, loaded = -1;
      for (cur.init(a, s0, s1); cur.slot < cur.end && !*abort; cur.advance(a)) {
        if (!cur.live()) continue;
        if (cur.group != loaded) {
          if (qn > 0) mma_commit(smem_u32(&sm->qempty));  // previous group's reads of sQ done
          if (!mbar_wait(smem_u32(&sm->qfull), qn & 1, abort, a.status, kWaitLimitNs, 13)) break;
          ++qn;
          loaded = cur.group;
        }
        const int acc = static_cast<int>(it & 1);
        if (acc == par) {
          if (it >= 2 &&
              !mbar_wait(smem_u32(&sm->tempty[acc]), ((it >> 1) + 1) & 1, abort, a.status,
                         kWaitLimitNs, 14))
            break;
          if (!mbar_wait(smem_u32(&sm->full[st]), ph, abort, a.status, kWaitLimitNs, 15)) break;
          tc_fence_after();
          const uint32_t d_tmem = tmem + acc * a.NQ;
          for (int kc = 0; kc < a.KC; ++kc) {
            const uint32_t a_addr = smem_u32(sA + st * stage_bytes + kc * 16384);
            const uint32_t b_addr = smem_u32(sQ + kc * a.NQ * 128);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t ad = smem_desc(a_addr + ks * 32, 16, 1024, kSwizzle128B);
              const uint64_t bd = smem_desc(b_addr + ks * 32, 16, 1024, kSwizzle128B);
              mma_bf16_ss(d_tmem, ad, bd, idesc, (kc | ks) != 0);
            }
          }
          mma_commit(smem_u32(&sm->empty[st]));
          mma_commit(smem_u32(&sm->tfull[acc]));
        }
        ++it;
        if (++st == a.stages) { st = 0; ph ^= 1u; }
      }
      // all issued MMAs complete before the accumulators are released
      mma_commit(smem_u32(&sm->mma_done[par]));
      mbar_wait(smem_u32(&sm->mma_done[par]), 0, nullptr, a.status, kWaitLimitNs, 16);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    float* wcol = sm->wcol[quad];
    int* ntv = sm->nt[quad];
    // heads a multiple of 32: every 32-column accumulator chunk belongs to
    // one query, so a query's score is a straight sum over its chunks
    const bool whole = (a.HI & 31) == 0;
    const int cpq = a.HI >> 5;
    SlotCursor cur;
    int64_t it = 0, wgroup = -1;
    for (cur.init(a, s0, s1); cur.slot < cur.end && !*abort; cur.advance(a)) {
      if (!cur.live()) continue;
      if (cur.group != wgroup) {
        __syncwarp();
        for (int c = lane; c < a.NQ; c += 32) {
          const int g = c / a.HI, h = c % a.HI;
          wcol[c] = (g < cur.gv) ? a.w[((int64_t)cur.b * a.T + cur.t0 + g) * a.HI + h] : 0.f;
        }
        for (int g = lane; g < a.G; g += 32)
          ntv[g] = g < cur.gv ? static_cast<int>(visible_entries(
                                    a.pos[(int64_t)cur.b * a.T + cur.t0 + g], a.m, a.N_cap))
                              : 0;
        __syncwarp();
        wgroup = cur.group;
      }
      const int acc = static_cast<int>(it & 1);
      const bool got = mbar_wait(smem_u32(&sm->tfull[acc]), (it >> 1) & 1, abort, a.status,
                                 kWaitLimitNs, 17);
      if (!__all_sync(0xffffffffu, got)) break;  // warp-uniform: tcgen05.ld follows
      tc_fence_after();
      const int64_t j = static_cast<int64_t>(cur.blk) * kBlockRows + row;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * a.NQ;
      float* srow = a.scores + ((int64_t)cur.b * a.T + cur.t0) * a.N_cap + j;
      if (whole) {
        for (int g = 0; g < cur.gv; ++g) {
          float sum = 0.f;
          for (int c = 0; c < cpq; c += 2) {
            const int col = (g * cpq + c) * 32;
            float x0[32], x1[32];
            tmem_ld32(taddr + col, x0);
            if (c + 1 < cpq) tmem_ld32(taddr + col + 32, x1);
            tmem_wait_ld();
            const float4* w0 = reinterpret_cast<const float4*>(wcol + col);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 wv = w0[i];
              sum = fmaf(wv.x, fmaxf(x0[4 * i], 0.f), sum);
              sum = fmaf(wv.y, fmaxf(x0[4 * i + 1], 0.f), sum);
              sum = fmaf(wv.z, fmaxf(x0[4 * i + 2], 0.f), sum);
              sum = fmaf(wv.w, fmaxf(x0[4 * i + 3], 0.f), sum);
            }
            if (c + 1 < cpq) {
              const float4* w1 = reinterpret_cast<const float4*>(wcol + col + 32);
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 wv = w1[i];
                sum = fmaf(wv.x, fmaxf(x1[4 * i], 0.f), sum);
                sum = fmaf(wv.y, fmaxf(x1[4 * i + 1], 0.f), sum);
                sum = fmaf(wv.z, fmaxf(x1[4 * i + 2], 0.f), sum);
                sum = fmaf(wv.w, fmaxf(x1[4 * i + 3], 0.f), sum);
              }
            }
          }
          if (j < ntv[g]) srow[(int64_t)g * a.N_cap] = sum;
        }
      } else {
        float sum = 0.f;
        int g = 0, h = 0;
        for (int cc = 0; cc < a.NQ; cc += 32) {
          float x[32];
          tmem_ld32(taddr + cc, x);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            sum = fmaf(wcol[cc + i], fmaxf(x[i], 0.f), sum);
            if (++h == a.HI) {
              if (g < cur.gv && j < ntv[g]) srow[(int64_t)g * a.N_cap] = sum;
              sum = 0.f;
              h = 0;
              ++g;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->tempty[acc]));
      ++it;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, tmem_cols);
}

}  // namespace

bool plan_indexer(int T, int HI, int dI, IndexerPlan* p) {
  if (HI <= 0 || HI > 256 || dI <= 0 || dI > 128) return false;
  int G = 256 / HI;
  if (G > T) G = T;
  if (G < 1) G = 1;
  int NQ = ((G * HI + 31) / 32) * 32;
  if (NQ > 256) return false;
  p->G = G;
  p->NQ = NQ;
  p->KC = (dI + 63) / 64;
  const size_t q_bytes = (size_t)p->KC * NQ * 128;
  const size_t stage_bytes = (size_t)p->KC * 16384;
  const size_t budget = 227 * 1024 - 1024 - sizeof(IdxSmem) - q_bytes;
  int stages = static_cast<int>(budget / stage_bytes);
  if (stages > kMaxStages) stages = kMaxStages;
  if (stages < 2) return false;
  p->stages = stages;
  p->tmem_cols = 2 * NQ;
  p->smem_bytes = 1024 + q_bytes + stages * stage_bytes + sizeof(IdxSmem);
  return true;
}

cudaError_t launch_indexer_score(const CUtensorMap& tm_ik, const CUtensorMap& tm_iq,
                                 const IndexerArgs& a, const IndexerPlan& p, int grid,
                                 cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(indexer_score_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(p.smem_bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kIdxThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  cfg.attrs = at;
  cfg.numAttrs = add_dependent_attr(at, 0);
  e = cudaLaunchKernelEx(&cfg, indexer_score_kernel, tm_ik, tm_iq, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hattn
