// hidden.cu -- compressed entries straight from hidden states.
//
// "Why DeepSeek V4 Stands Apart", section "Core Architectural Innovations":
// the compressor turns per-token KV rows into compressed entries; the
// per-token rows are themselves a projection x_u . W of the hidden states.
// Gate-softmax pooling is a weighted sum of token rows, so pooling the
// hidden states first and projecting once per entry gives the same entry:
//     sum_u a_u (x_u . W) = (sum_u a_u x_u) . W.
// The cache build then reads each hidden state once per window it belongs
// to, never writes per-token KV rows, and runs the projection on one row per
// entry: a quarter of the tokens for CSA, 1/128 for HCA.
//
// Two kernels per chunk of entries:
//   1. pool_hidden_kernel: the gate softmax of each window and the pooled row
//      x_bar in fp32, stored as a pair of bf16 rows hi + lo (hi = bf16(x_bar),
//      lo = bf16(x_bar - hi)) that together keep ~16 significant bits;
//   2. project_entries_kernel: Y = hi . W + lo . W on the tensor cores
//      (tcgen05, fp32 accumulation in tensor memory), then in its epilogue the
//      RMSNorm of Y's KV columns, RoPE at the entry's last token and the bf16
//      KV entry, or the indexer-key columns in bf16.  Y never leaves the SM.

#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kPoolThreads = 256;
constexpr int kPoolMaxW = 512;
constexpr int kPoolSlice = kPoolThreads * 8;  // columns of one pass of a block's threads

// Eight pooled fp32 values as the bf16 parts hi = bf16(v), lo = bf16(v - hi).
__device__ __forceinline__ void store_parts(const float (&acc)[8], __nv_bfloat16* xh,
                                            __nv_bfloat16* xl) {
  float hi[8], lo[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    hi[k] = bf16_round(acc[k]);
    lo[k] = acc[k] - hi[k];
  }
  *reinterpret_cast<uint4*>(xh) = make_uint4(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]),
                                             pack_bf16x2(hi[4], hi[5]), pack_bf16x2(hi[6], hi[7]));
  *reinterpret_cast<uint4*>(xl) = make_uint4(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]),
                                             pack_bf16x2(lo[4], lo[5]), pack_bf16x2(lo[6], lo[7]));
}

// The pooled row of entry j of sequence b (gate softmax over the window's
// tokens that exist, then the weighted sum of their hidden states, kept as
// bf16 parts hi + lo); every thread of the block calls it.
__device__ __forceinline__ void pool_entry(const HiddenArgs& a, int b, int64_t j,
                                           __nv_bfloat16* __restrict__ xh_row,
                                           __nv_bfloat16* __restrict__ xl_row, float* alpha,
                                           int c_begin, int c_end) {
  const int tid = threadIdx.x;
  const int64_t u0 = static_cast<int64_t>(a.m) * (j + 1) - a.w;
  // gate softmax over the window's tokens that exist (warp 0)
  if (tid < 32) {
    float gmax = -INFINITY;
    for (int s = tid; s < a.w; s += 32) {
      const int64_t u = u0 + s;
      if (u >= 0) gmax = fmaxf(gmax, __bfloat162float(a.gate[(int64_t)b * a.L_cap + u]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
    float z = 0.f;
    for (int s = tid; s < a.w; s += 32) {
      const int64_t u = u0 + s;
      const float ex =
          u >= 0 ? __expf(__bfloat162float(a.gate[(int64_t)b * a.L_cap + u]) - gmax) : 0.f;
      alpha[s] = ex;
      z += ex;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const float iz = 1.f / z;
    __syncwarp();
    for (int s = tid; s < a.w; s += 32) alpha[s] *= iz;
  }
  __syncthreads();
  // pooled row, 8 columns per thread per pass
  const int s_lo = u0 < 0 ? static_cast<int>(-u0) : 0;
  for (int c = c_begin + tid * 8; c < c_end; c += kPoolThreads * 8) {
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
    const __nv_bfloat16* src = a.x + ((int64_t)b * a.L_cap + u0) * a.dm + c;
    // eight token rows requested at once, then accumulated in order
    for (int s0 = s_lo; s0 < a.w; s0 += 8) {
      uint4 v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4* row = reinterpret_cast<const uint4*>(src + (int64_t)(s0 + q) * a.dm);
        v[q] = s0 + q < a.w ? __ldg(row) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float al = s0 + q < a.w ? alpha[s0 + q] : 0.f;
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[q]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(h[k]);
          acc[2 * k] = fmaf(al, f.x, acc[2 * k]);
          acc[2 * k + 1] = fmaf(al, f.y, acc[2 * k + 1]);
        }
      }
    }
    float hi[8], lo[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      hi[k] = bf16_round(acc[k]);
      lo[k] = acc[k] - hi[k];
    }
    uint4 uh, ul;
    uh.x = pack_bf16x2(hi[0], hi[1]);
    uh.y = pack_bf16x2(hi[2], hi[3]);
    uh.z = pack_bf16x2(hi[4], hi[5]);
    uh.w = pack_bf16x2(hi[6], hi[7]);
    ul.x = pack_bf16x2(lo[0], lo[1]);
    ul.y = pack_bf16x2(lo[2], lo[3]);
    ul.z = pack_bf16x2(lo[4], lo[5]);
    ul.w = pack_bf16x2(lo[6], lo[7]);
    *reinterpret_cast<uint4*>(xh_row + c) = uh;
    *reinterpret_cast<uint4*>(xl_row + c) = ul;
  }
  __syncthreads();  // alpha is rewritten for the next entry
}

__global__ void __launch_bounds__(kPoolThreads)
    pool_hidden_kernel(const __grid_constant__ HiddenArgs a, int64_t e0, int64_t ne,
                       __nv_bfloat16* __restrict__ xh, __nv_bfloat16* __restrict__ xl) {
  __shared__ float alpha[kPoolMaxW];
  const int64_t nj = a.j_end - a.j_begin;
  for (int64_t e = blockIdx.x; e < ne; e += gridDim.x) {
    const int64_t flat = e0 + e;  // (sequence, entry) over the whole call
    const int b = static_cast<int>(flat / nj);
    const int64_t j = a.j_begin + flat % nj;
    pool_entry(a, b, j, xh + e * a.dm, xl + e * a.dm, alpha, 0, a.dm);
  }
}

// Both caches in one read of the hidden states: block g of 128 tokens of a
// sequence holds the CSA entries 32h .. 32h + 31 (C(4, 8): their windows
// reach 4 tokens into the block before) and the HCA entry h (C(128, 128):
// the block itself), h = g's block within its sequence.  A CTA takes one
// column slice of kPoolSlice columns (grid y) of its blocks; its threads
// hold 8 columns each.  The gate softmaxes of the block's 32 CSA windows
// (8 lanes per window) and of its HCA window come first; then the block's
// tokens stream in 8 groups of 20 rows (16 new rows and the 4 that the
// group's first window shares with the group before), every group serving 4
// CSA entries and the HCA entry at once.  Chunk-relative rows: CSA entry
// (b, j) at b * nc + j - fc0, HCA entry (b, h) at b * nh + h - fh0.
__global__ void __launch_bounds__(kPoolThreads)
    pool_pair_kernel(const __grid_constant__ HiddenArgs ac, const __grid_constant__ HiddenArgs ah,
                     int64_t g0, int64_t ng, int64_t nbs, int64_t fc0, int64_t fh0,
                     __nv_bfloat16* __restrict__ xhc, __nv_bfloat16* __restrict__ xlc,
                     __nv_bfloat16* __restrict__ xhh, __nv_bfloat16* __restrict__ xlh) {
  __shared__ float alc[32][8];   // CSA window weights
  __shared__ float alh[128];     // HCA window weights
  __shared__ float red[8];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nc = ac.j_end, nh = ah.j_end;  // entries per sequence (from 0)
  const int c = blockIdx.y * kPoolSlice + tid * 8;  // this thread's first column
  const bool col_ok = c < ac.dm;
  for (int64_t q = blockIdx.x; q < ng; q += gridDim.x) {
    const int64_t g = g0 + q;
    const int b = static_cast<int>(g / nbs);
    const int64_t h = g - static_cast<int64_t>(b) * nbs;
    const int64_t t0 = 128 * h;  // the block's first token
    const __nv_bfloat16* gc = ac.gate + (int64_t)b * ac.L_cap;
    const __nv_bfloat16* gh = ah.gate + (int64_t)b * ah.L_cap;
    {
      // CSA: thread (entry e = tid / 8, window slot s = tid % 8), token
      // 4 (32 h + e) - 4 + s = t0 + 4 e - 4 + s, softmax over the 8 lanes
      const int e = tid >> 3, s8 = tid & 7;
      const int64_t u = t0 + 4 * e - 4 + s8;
      const bool in = u >= 0 && 32 * h + e < nc;
      const float gv = in ? __bfloat162float(gc[u]) : -INFINITY;
      float mx = gv;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o, 8));
      const float ex = in ? __expf(gv - mx) : 0.f;
      float z = ex;
#pragma unroll
      for (int o = 4; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o, 8);
      alc[e][s8] = z > 0.f ? ex / z : 0.f;
    }
    // HCA: the 128 gates of the block (threads 0..127), a block max and sum
    const bool hin = h < nh;
    float hg = -INFINITY;
    if (tid < 128 && hin) hg = __bfloat162float(gh[t0 + tid]);
    float hm = hg;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, o));
    if (lane == 0) red[warp] = hm;
    __syncthreads();
    hm = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    const float hx = (tid < 128 && hin) ? __expf(hg - hm) : 0.f;
    float hz = hx;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) hz += __shfl_xor_sync(0xffffffffu, hz, o);
    __syncthreads();  // every thread has read red[] as maxima
    if (lane == 0) red[warp] = hz;
    __syncthreads();
    hz = red[0] + red[1] + red[2] + red[3];
    if (tid < 128) alh[tid] = hin ? hx / hz : 0.f;
    __syncthreads();
    // the block's rows, 8 groups of 20
    float hacc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) hacc[k] = 0.f;
    for (int gq = 0; gq < 8; ++gq) {
      const int64_t u0 = t0 + 16 * gq - 4;  // the group's first row
      uint4 v[20];
#pragma unroll
      for (int r = 0; r < 20; ++r) {
        const int64_t u = u0 + r;
        v[r] = (col_ok && u >= 0 && u < ac.L_cap)
                   ? __ldg(reinterpret_cast<const uint4*>(ac.x + ((int64_t)b * ac.L_cap + u) * ac.dm + c))
                   : make_uint4(0, 0, 0, 0);
      }
      // entries 4 gq .. 4 gq + 3: entry e4 takes rows 4 e4 .. 4 e4 + 7
#pragma unroll
      for (int e4 = 0; e4 < 4; ++e4) {
        const int e = 4 * gq + e4;
        float acc[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] = 0.f;
#pragma unroll
        for (int s8 = 0; s8 < 8; ++s8) {
          const float al = alc[e][s8];
          const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&v[4 * e4 + s8]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(hv[k]);
            acc[2 * k] = fmaf(al, f.x, acc[2 * k]);
            acc[2 * k + 1] = fmaf(al, f.y, acc[2 * k + 1]);
          }
        }
        const int64_t j = 32 * h + e;
        if (col_ok && j < nc) {
          const int64_t row = static_cast<int64_t>(b) * nc + j - fc0;
          store_parts(acc, xhc + row * ac.dm + c, xlc + row * ac.dm + c);
        }
      }
      // the HCA window: the group's 16 new rows
#pragma unroll
      for (int r = 4; r < 20; ++r) {
        const float al = alh[16 * gq + r - 4];
        const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&v[r]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float2 f = __bfloat1622float2(hv[k]);
          hacc[2 * k] = fmaf(al, f.x, hacc[2 * k]);
          hacc[2 * k + 1] = fmaf(al, f.y, hacc[2 * k + 1]);
        }
      }
    }
    if (col_ok && hin) {
      const int64_t row = static_cast<int64_t>(b) * nh + h - fh0;
      store_parts(hacc, xhh + row * ah.dm + c, xlh + row * ah.dm + c);
    }
    __syncthreads();  // the weights are rewritten for the next block
  }
}

// ---------------------------------------------------------------- projection
// Y = hi . W + lo . W for a tile of 128 pooled entries, on the tensor cores,
// with the entry epilogue fused: one CTA per (128-entry tile, column group),
// column group 0 the D KV columns (RMSNorm, RoPE at the entry's last token,
// bf16 KV entry), group 1 the dI indexer-key columns (bf16).  K = dm runs in
// blocks of 64: per block the A tiles hi and lo (128 rows x 128 B each, TMA,
// 128-byte swizzle, K-major) and the W rows (64 x N, TMA boxes of 64 columns,
// MN-major), and per 16-wide K step one tcgen05.mma per A tile and 256-column
// piece of N, all into one fp32 accumulator in tensor memory.
// Warps: 0 loads, 1 issues the MMAs, 2..5 run the epilogue (one row each).
constexpr int kProjThreads = 192;
constexpr int kProjMaxStages = 4;

struct ProjSmem {
  uint64_t full[kProjMaxStages];
  uint64_t empty[kProjMaxStages];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
};

struct ProjPlan {
  int n;       // accumulator columns of the tile (a multiple of 64)
  int stages;
  uint32_t stage_bytes, tmem_cols;
  size_t smem_bytes;
};

__host__ __device__ inline ProjPlan proj_plan(int n) {
  ProjPlan p;
  p.n = n;
  p.stage_bytes = 2u * 16384u + static_cast<uint32_t>(n) * 128u;
  const size_t room = 227 * 1024 - 1024 - (sizeof(ProjSmem) + 15) / 16 * 16;
  p.stages = static_cast<int>(room / p.stage_bytes);
  if (p.stages > kProjMaxStages) p.stages = kProjMaxStages;
  p.tmem_cols = n <= 64 ? 64 : (n <= 128 ? 128 : (n <= 256 ? 256 : 512));
  p.smem_bytes = 1024 + static_cast<size_t>(p.stages) * p.stage_bytes + (sizeof(ProjSmem) + 15) / 16 * 16;
  return p;
}

__global__ void __launch_bounds__(kProjThreads, 1)
    project_entries_kernel(const __grid_constant__ CUtensorMap tm_ah,
                           const __grid_constant__ CUtensorMap tm_al,
                           const __grid_constant__ CUtensorMap tm_w,
                           const __grid_constant__ HiddenArgs a, int64_t e0, int64_t ne,
                           int n_kv, int n_ik, int* status) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const bool kv_tile = blockIdx.y == 0;
  const int n = kv_tile ? n_kv : n_ik;  // accumulator columns
  const ProjPlan pl = proj_plan(n);
  ProjSmem* sm = reinterpret_cast<ProjSmem*>(base + pl.stages * pl.stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t m0 = static_cast<int64_t>(blockIdx.x) * 128;  // first entry of the tile (chunk-relative)
  const int col0 = kv_tile ? 0 : a.D;                          // first W column of the group
  const int nkb = (a.dm + 63) / 64;
  if (threadIdx.x == 0) {
    for (int s = 0; s < pl.stages; ++s) {
      mbar_init(smem_u32(&sm->full[s]), 1);
      mbar_init(smem_u32(&sm->empty[s]), 1);
    }
    mbar_init(smem_u32(&sm->done), 1);
    sm->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_ah);
    tma_prefetch_desc(&tm_al);
    tma_prefetch_desc(&tm_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm->tmem_base), pl.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort = &sm->abort;
  if (warp == 0) {
    // ------------------------------------------------------------ loads
    if (lane == 0) {
      int64_t issued = 0;
      for (int kb = 0; kb < nkb && !*abort; ++kb) {
        const int st = kb % pl.stages;
        const uint32_t ph = static_cast<uint32_t>(kb / pl.stages) & 1u;
        // the stage's previous use (block kb - stages) has been read by its MMAs
        if (kb >= pl.stages &&
            !mbar_wait(smem_u32(&sm->empty[st]), ph ^ 1u, abort, status, kWaitLimitNs, 50))
          break;
        uint8_t* sb = base + st * pl.stage_bytes;
        const uint32_t fb = smem_u32(&sm->full[st]);
        mbar_arrive_expect_tx(fb, pl.stage_bytes);
        tma_load_2d(smem_u32(sb), &tm_ah, kb * 64, static_cast<int32_t>(m0), fb);
        tma_load_2d(smem_u32(sb + 16384), &tm_al, kb * 64, static_cast<int32_t>(m0), fb);
        for (int c = 0; c < n / 64; ++c)
          tma_load_2d(smem_u32(sb + 32768 + c * 8192), &tm_w, col0 + c * 64, kb * 64, fb);
        ++issued;
      }
      if (*abort) {
        // the copies already issued land before the CTA exits
        for (int64_t x = issued > pl.stages ? issued - pl.stages : 0; x < issued; ++x)
          mbar_wait(smem_u32(&sm->full[x % pl.stages]), static_cast<uint32_t>(x / pl.stages) & 1u,
                    nullptr, nullptr, 10000000ull, 51);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMAs
    if (lane == 0) {
      bool ok = true;
      for (int kb = 0; kb < nkb && ok; ++kb) {
        const int st = kb % pl.stages;
        ok = mbar_wait(smem_u32(&sm->full[st]), static_cast<uint32_t>(kb / pl.stages) & 1u, abort,
                       status, kWaitLimitNs, 52);
        if (!ok) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(base + st * pl.stage_bytes);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ah = smem_desc(sa + ks * 32, 16, 1024, kSwizzle128B);
          const uint64_t al = smem_desc(sa + 16384 + ks * 32, 16, 1024, kSwizzle128B);
          for (int c0 = 0; c0 < n; c0 += 256) {
            const int nn = n - c0 < 256 ? n - c0 : 256;
            const uint32_t idesc = idesc_bf16(128, nn, 0, 1);
            // W rows of this K step, columns c0 .. c0 + nn: MN-major, one
            // 64-column chunk (64 K rows x 128 B) after another
            const uint64_t bd =
                smem_desc(sa + 32768 + (c0 / 64) * 8192 + ks * 2048, 8192, 1024, kSwizzle128B);
            mma_bf16_ss(tmem + c0, ah, bd, idesc, (kb | ks) != 0 ? 1u : 0u);
            mma_bf16_ss(tmem + c0, al, bd, idesc, 1u);
          }
        }
        mma_commit(smem_u32(&sm->empty[st]));
      }
      // every MMA issued above completes before `done` (also on an abort)
      mma_commit(smem_u32(&sm->done));
      if (!ok) mbar_wait(smem_u32(&sm->done), 0, nullptr, nullptr, 10000000ull, 53);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;
    const int row = quad * 32 + lane;  // tensor-memory lane = tile row
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = mbar_wait(smem_u32(&sm->done), 0, abort, status, kWaitLimitNs, 54);
    ok = __all_sync(0xffffffffu, ok);
    if (ok) {
      tc_fence_after();
      const int64_t e = m0 + row;  // chunk-relative entry
      const bool valid = e < ne;
      const int ncols = kv_tile ? a.D : a.dI;
      // the stage buffers are free once every MMA has completed: each row
      // is staged as bf16 there, then leaves by one bulk copy
      const int rstride = ncols * 2 + 16;
      uint8_t* srow = base + row * rstride;
      float inv = 1.f;
      if (kv_tile) {
        float ss = 0.f;
        for (int c = 0; c < a.D; c += 32) {
          float y[32];
          tmem_ld32(tmem + lane_base + c, y);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) ss = fmaf(y[i], y[i], ss);
        }
        inv = rsqrtf(ss / static_cast<float>(a.D) + a.eps);
      }
      const int64_t nj = a.j_end - a.j_begin;
      const int64_t flat = e0 + (valid ? e : 0);
      const int bb = static_cast<int>(flat / nj);
      const int64_t j = a.j_begin + flat % nj;
      const int64_t p = static_cast<int64_t>(a.m) * (j + 1) - 1;  // the entry's last token
      const int d0 = a.D - a.r;
      for (int c = 0; c < ncols; c += 32) {
        float y[32];
        tmem_ld32(tmem + lane_base + c, y);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float x0 = y[i], x1 = y[i + 1];
          if (kv_tile) {
            const int d = c + i;
            x0 *= inv * (a.gamma ? a.gamma[d] : 1.f);
            x1 *= inv * (a.gamma ? a.gamma[d + 1] : 1.f);
            if (d >= d0) {
              float sn, cs;
              rope_cs(a.rope.c, (d - d0) >> 1, p, &sn, &cs);
              const float t0 = x0 * cs - x1 * sn;
              x1 = x0 * sn + x1 * cs;
              x0 = t0;
            }
          }
          pk[i >> 1] = pack_bf16x2(x0, x1);
        }
        // (ncols is a multiple of 8: whole 16-byte pieces)
        const int nq = (ncols - c) < 32 ? (ncols - c) / 8 : 4;
        for (int q = 0; q < nq; ++q)
          reinterpret_cast<uint4*>(srow + c * 2)[q] =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      fence_proxy_async_smem();
      if (valid) {
        __nv_bfloat16* dst = kv_tile ? a.kv_out + ((int64_t)bb * a.N_cap + j) * a.D
                                     : a.ik_out + ((int64_t)bb * a.N_cap + j) * a.dI;
        bulk_copy_s2g(dst, smem_u32(srow), static_cast<uint32_t>(ncols) * 2u);
        bulk_commit();
        bulk_wait_read();
      }
    } else {
      // no MMA may still write the accumulator when it is released
      mbar_wait(smem_u32(&sm->done), 0, nullptr, nullptr, 10000000ull, 55);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, pl.tmem_cols);
}
}  // namespace

size_t hidden_part_bytes(size_t ce, int dm) { return (ce * dm * 2 + 255) / 256 * 256; }

size_t hidden_chunk_entries(int64_t total) { return total < kHiddenChunk ? total : kHiddenChunk; }

size_t hidden_workspace_bytes(int64_t total, int dm, int P) {
  (void)P;
  const size_t ce = hidden_chunk_entries(total);
  return 2 * hidden_part_bytes(ce, dm);
}

int hidden_ik_cols(int dI) { return dI <= 0 ? 0 : (dI + 63) / 64 * 64; }

cudaError_t launch_compress_hidden(const HiddenArgs& a, void* ws, int num_sms,
                                   const CUtensorMap& tm_ah, const CUtensorMap& tm_al,
                                   const CUtensorMap& tm_w, int* status, cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(a.B) * (a.j_end - a.j_begin);
  if (total <= 0) return cudaSuccess;
  const int64_t ce = static_cast<int64_t>(hidden_chunk_entries(total));
  uint8_t* p = static_cast<uint8_t*>(ws);
  __nv_bfloat16* xh = reinterpret_cast<__nv_bfloat16*>(p);
  __nv_bfloat16* xl = reinterpret_cast<__nv_bfloat16*>(p + hidden_part_bytes(ce, a.dm));
  const int n_kv = a.D, n_ik = hidden_ik_cols(a.dI);
  // each column group's plan fits one CTA; the launch gives the larger
  const size_t s_kv = proj_plan(n_kv).smem_bytes;
  const size_t s_ik = n_ik > 0 ? proj_plan(n_ik).smem_bytes : 0;
  const size_t smem = s_kv > s_ik ? s_kv : s_ik;
  cudaError_t e = cudaFuncSetAttribute(project_entries_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  for (int64_t e0 = 0; e0 < total; e0 += ce) {
    const int64_t ne = (total - e0) < ce ? (total - e0) : ce;
    const int64_t grid = ne < (int64_t)num_sms * 8 ? ne : (int64_t)num_sms * 8;
    pool_hidden_kernel<<<static_cast<unsigned>(grid), kPoolThreads, 0, stream>>>(a, e0, ne, xh,
                                                                               xl);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    // one CTA per (128-entry tile, column group); the shared memory of the
    // larger group serves both
    const dim3 g(static_cast<unsigned>((ne + 127) / 128), n_ik > 0 ? 2u : 1u, 1u);
    project_entries_kernel<<<g, kProjThreads, smem, stream>>>(tm_ah, tm_al, tm_w, a, e0, ne, n_kv,
                                                              n_ik, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

constexpr int64_t kPairBlocks = kHiddenChunk / 32;  // 128-token blocks per pass

size_t hidden_pair_workspace_bytes(int B, int64_t nc, int64_t nh, int dm) {
  const int64_t rows_c = (int64_t)B * nc < kHiddenChunk ? (int64_t)B * nc : kHiddenChunk;
  return 2 * hidden_part_bytes(rows_c, dm) + 2 * hidden_part_bytes((int64_t)B * nh, dm);
}

cudaError_t launch_compress_hidden_pair(const HiddenArgs& ac, const HiddenArgs& ah, void* ws,
                                        int num_sms, const CUtensorMap& tm_ch,
                                        const CUtensorMap& tm_cl, const CUtensorMap& tm_wc,
                                        const CUtensorMap& tm_hh, const CUtensorMap& tm_hl,
                                        const CUtensorMap& tm_wh, int* status,
                                        cudaStream_t stream) {
  const int B = ac.B;
  const int64_t nc = ac.j_end, nh = ah.j_end;
  if (nc <= 0) return cudaSuccess;
  const int64_t nbs = (nc + 31) / 32;  // blocks per sequence
  const int64_t rows_c = (int64_t)B * nc < kHiddenChunk ? (int64_t)B * nc : kHiddenChunk;
  uint8_t* p = static_cast<uint8_t*>(ws);
  __nv_bfloat16* xhc = reinterpret_cast<__nv_bfloat16*>(p);
  p += hidden_part_bytes(rows_c, ac.dm);
  __nv_bfloat16* xlc = reinterpret_cast<__nv_bfloat16*>(p);
  p += hidden_part_bytes(rows_c, ac.dm);
  __nv_bfloat16* xhh = reinterpret_cast<__nv_bfloat16*>(p);
  p += hidden_part_bytes((int64_t)B * nh, ac.dm);
  __nv_bfloat16* xlh = reinterpret_cast<__nv_bfloat16*>(p);
  const int n_kv = ac.D, n_ik = hidden_ik_cols(ac.dI);
  const size_t s_kv = proj_plan(n_kv).smem_bytes;
  const size_t s_ik = n_ik > 0 ? proj_plan(n_ik).smem_bytes : 0;
  const size_t smem = s_kv > s_ik ? s_kv : s_ik;
  cudaError_t e = cudaFuncSetAttribute(project_entries_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // the flat CSA index of block g's first entry
  auto flatc = [&](int64_t g) {
    const int64_t b = g / nbs, h = g % nbs;
    return b * nc + (32 * h < nc ? 32 * h : nc);
  };
  const int64_t total_g = (int64_t)B * nbs;
  for (int64_t g0 = 0; g0 < total_g; g0 += kPairBlocks) {
    const int64_t ng = total_g - g0 < kPairBlocks ? total_g - g0 : kPairBlocks;
    const int64_t fc0 = flatc(g0), fc1 = flatc(g0 + ng);
    const int slices = (ac.dm + kPoolSlice - 1) / kPoolSlice;
    const int64_t grid = ng < (int64_t)num_sms * 8 ? ng : (int64_t)num_sms * 8;
    pool_pair_kernel<<<dim3(static_cast<unsigned>(grid), static_cast<unsigned>(slices), 1),
                       kPoolThreads, 0, stream>>>(ac, ah, g0, ng, nbs, fc0, 0, xhc, xlc, xhh,
                                                  xlh);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int64_t ne = fc1 - fc0;
    if (ne > 0) {
      const dim3 g(static_cast<unsigned>((ne + 127) / 128), n_ik > 0 ? 2u : 1u, 1u);
      project_entries_kernel<<<g, kProjThreads, smem, stream>>>(tm_ch, tm_cl, tm_wc, ac, fc0, ne,
                                                                n_kv, n_ik, status);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  // the HCA entries of every sequence, in one projection
  if (nh > 0) {
    const int64_t ne = (int64_t)B * nh;
    const dim3 g(static_cast<unsigned>((ne + 127) / 128), 1u, 1u);
    project_entries_kernel<<<g, kProjThreads, smem, stream>>>(tm_hh, tm_hl, tm_wh, ah, 0, ne,
                                                              ah.D, 0, status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace hattn
