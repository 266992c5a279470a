// attention.cu -- the three attention branches of the hybrid layer on the
// tcgen05 tensor cores, with split-KV partials.
//
// "Why DeepSeek V4 Stands Apart", section "Core Architectural Innovations":
// SWA attends to the most recent 128 tokens; CSA attends to the top-k
// selected compressed entries; HCA attends densely to the 128:1 compressed
// entries.  "DeepSeek-V4" atlas: RMSNorm on queries (section "Design
// overview"), partial RoPE on the last 64 dims (provenance 16), shared-KV MQA
// (section "Inference efficiency"): one D-dim latent per key serves as key
// and value for every head.
//
// One CTA owns a row block (G queries x H heads <= 128 rows, the MMA M
// dimension), a key range (one split of the visible keys) and one half of
// the output columns (nds = 2 for D = 512: the fp32 accumulator of 128 rows
// x 512 columns would fill the whole tensor memory, so each CTA of a pair
// keeps 256 of them).  Per 64-key tile:
//   S = Q K^T   (M=128, N=64, K=D)      -> tensor memory, two buffers
//   softmax     (one thread per row, online max with lazy rescaling)
//   O += P V    (M=128, N=64 per 64-column chunk, K=64 keys)
// Key rows reach shared memory as 64x64 bf16 chunks (8 KB, 128-byte
// swizzle) in a ring of `nslot` slots: HCA by TMA tiles, CSA by a 16-byte
// cp.async gather through the top-k indices, SWA by normalising and roping
// the raw tokens on load.  Warps 0-3 produce chunks, warp 4 issues the MMAs,
// warps 5-8 run the softmax and the epilogue.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kThreads = 288;
constexpr int kTile = 64;
constexpr int kMaxSlots = 16;
constexpr int kProdThreads = 128;

struct AttnShared {
  uint64_t full[kMaxSlots];
  uint64_t empty[kMaxSlots];
  uint64_t s_full[2];
  uint64_t p_full;
  uint64_t o_full;
  uint32_t tmem_base;
  int abort;
  float inv_rms[kTile];  // SWA: per-row norm of the tile being produced
  double theta[64];      // RoPE frequencies, r <= 128
};

__device__ __forceinline__ int64_t vis(int32_t t, int m) {
  return t < 0 ? 0 : (static_cast<int64_t>(t) + 1) / m;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void load8f(const __nv_bfloat16* p, float (&x)[8]) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float (&y)[8]) {
  uint4 u;
  u.x = pack_bf16x2(y[0], y[1]);
  u.y = pack_bf16x2(y[2], y[3]);
  u.z = pack_bf16x2(y[4], y[5]);
  u.w = pack_bf16x2(y[6], y[7]);
  return u;
}

// RoPE on the pairs of an 8-element piece starting at dim d_first.
__device__ __forceinline__ void rope8(float (&y)[8], int d_first, int D, int r, int64_t p,
                                      const double* theta) {
  const int d0 = D - r;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const int d = d_first + e;
    if (d >= d0) {
      float sn, cs;
      rope_sincos(theta[(d - d0) >> 1], p, &sn, &cs);
      const float x0 = y[e], x1 = y[e + 1];
      y[e] = x0 * cs - x1 * sn;
      y[e + 1] = x0 * sn + x1 * cs;
    }
  }
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_kv, const AttnArgs a, const int nslot,
                const int pd) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int ndc = a.D / 64;                // 64-wide d chunks
  const int n_own = ndc / a.nds;           // chunks of this CTA's output columns
  const int n_other = ndc - n_own;
  uint8_t* sQ = base;                      // ndc x [128 rows x 128 B]
  uint8_t* sP = sQ + ndc * 16384;          // [128 rows x 64 keys] bf16
  uint8_t* sRing = sP + 16384;             // nslot x [64 keys x 128 B]
  AttnShared* sm = reinterpret_cast<AttnShared*>(sRing + nslot * 8192);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int dh = blockIdx.x % a.nds;
  const int split = blockIdx.x / a.nds;
  const int rb = blockIdx.y;
  const int b = blockIdx.z;
  const int t0 = rb * a.G;
  const int gv = min(a.G, a.T - t0);
  const int nrows = gv * a.H;

  // ---------------------------------------------------------------- key range
  int64_t total = 0, u_lo = 0;
  if (KIND == kSparse) {
    total = a.k;
  } else if (KIND == kHca) {
    for (int g = 0; g < gv; ++g) {
      int64_t v = vis(a.pos[(int64_t)b * a.T + t0 + g], a.m);
      total = v > total ? v : total;
    }
    if (total > a.N_rows) total = a.N_rows;
  } else {
    int64_t lo = INT64_MAX, hi = -1;
    for (int g = 0; g < gv; ++g) {
      int64_t t = a.pos[(int64_t)b * a.T + t0 + g];
      int64_t l = t - a.W + 1;
      if (l < 0) l = 0;
      lo = l < lo ? l : lo;
      hi = t > hi ? t : hi;
    }
    if (hi > a.N_rows - 1) hi = a.N_rows - 1;
    u_lo = lo;
    total = hi >= lo ? hi - lo + 1 : 0;
  }
  const int64_t kbeg = static_cast<int64_t>(split) * a.keys_per_split;
  int64_t kend = kbeg + a.keys_per_split;
  if (kend > total) kend = total;
  const int nk = kend > kbeg ? static_cast<int>(kend - kbeg) : 0;
  const int nt = (nk + kTile - 1) / kTile;
  const int ocols = n_own * 64;

  if (nt == 0) {
    // empty split: o = 0, lse = -inf
    for (int rI = threadIdx.x; rI < nrows; rI += kThreads) {
      const int g = rI / a.H, h = rI % a.H;
      const int64_t row = ((int64_t)b * a.T + t0 + g) * a.H + h;
      if (a.nsplit == 1) {
        for (int c = 0; c < ocols; ++c) a.o[row * a.D + dh * ocols + c] = __float2bfloat16(0.f);
        if (dh == 0) a.lse[row] = -INFINITY;
      } else {
        float* po = a.part_o + (row * a.nsplit + split) * a.D + dh * ocols;
        for (int c = 0; c < ocols; ++c) po[c] = 0.f;
        if (dh == 0) a.part_lse[row * a.nsplit + split] = -INFINITY;
      }
    }
    return;
  }

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    const uint32_t full_count = (KIND == kHca) ? 1 : kProdThreads;
    for (int i = 0; i < nslot; ++i) {
      mbar_init(smem_u32(&sm->full[i]), full_count);
      mbar_init(smem_u32(&sm->empty[i]), 1);
    }
    mbar_init(smem_u32(&sm->s_full[0]), 1);
    mbar_init(smem_u32(&sm->s_full[1]), 1);
    mbar_init(smem_u32(&sm->p_full), 128);
    mbar_init(smem_u32(&sm->o_full), 1);
    sm->abort = 0;
    fence_barrier_init();
    if (KIND == kHca) tma_prefetch_desc(&tm_kv);
  }
  for (int i = threadIdx.x; i < a.r / 2; i += kThreads)
    sm->theta[i] = pow(static_cast<double>(a.rope_base), -2.0 * i / static_cast<double>(a.r));
  if (warp == 4) {
    tmem_alloc(smem_u32(&sm->tmem_base), 512);
    tmem_relinquish();
  }
  __syncthreads();  // theta ready

  // ---------------------------------------------------------------- Q prologue
  // q~ = RoPE_t(RMSNorm(q; gamma_q, eps)) per row, bf16, 128B-swizzled chunks
  {
    const int npieces = a.D / 8;
    for (int rI = warp; rI < 128; rI += kThreads / 32) {
      const bool valid = rI < nrows;
      const int g = valid ? rI / a.H : 0, h = valid ? rI % a.H : 0;
      const __nv_bfloat16* qrow = a.q + (((int64_t)b * a.T + t0 + g) * a.H + h) * a.D;
      const int64_t tpos = valid ? a.pos[(int64_t)b * a.T + t0 + g] : 0;
      float x[2][8];
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int pc = lane + 32 * i;
        if (valid && pc < npieces) {
          load8f(qrow + pc * 8, x[i]);
#pragma unroll
          for (int e = 0; e < 8; ++e) ss = fmaf(x[i][e], x[i][e], ss);
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) x[i][e] = 0.f;
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      const float inv = rsqrtf(ss / static_cast<float>(a.D) + a.eps);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int pc = lane + 32 * i;
        if (pc < npieces) {
          float y[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float gm = a.gamma_q ? a.gamma_q[pc * 8 + e] : 1.f;
            y[e] = valid ? x[i][e] * inv * gm : 0.f;
          }
          if (valid) rope8(y, pc * 8, a.D, a.r, tpos, sm->theta);
          *reinterpret_cast<uint4*>(sQ + (pc >> 3) * 16384 + swz128(rI, pc & 7)) = pack8(y);
        }
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort = &sm->abort;
  const uint32_t tS = tmem;          // columns [0, 128): two 64-column S buffers
  const uint32_t tO = tmem + 128;    // columns [128, 128 + ocols)

  // chunk order within a tile: the other half's d chunks first, then ours
  auto chunk_dc = [&](int p) -> int {
    if (p < n_other) {
      const int oth = (dh == 0) ? 1 : 0;
      return oth * n_own + p;
    }
    return dh * n_own + (p - n_other);
  };

  if (warp < 4) {
    // ============================================================ producers
    const int pt = threadIdx.x;  // 0..127
    int64_t ctr = 0;
    if (KIND == kHca) {
      if (pt == 0) {
        for (int i = 0; i < nt && !*abort; ++i) {
          for (int p = 0; p < ndc; ++p, ++ctr) {
            const int slot = static_cast<int>(ctr % nslot);
            if (ctr >= nslot &&
                !mbar_wait(smem_u32(&sm->empty[slot]), ((ctr / nslot) + 1) & 1, abort, a.status, kWaitLimitNs, 18))
              break;
            const uint32_t fb = smem_u32(&sm->full[slot]);
            mbar_arrive_expect_tx(fb, 8192);
            tma_load_2d(smem_u32(sRing + slot * 8192), &tm_kv, chunk_dc(p) * 64,
                        static_cast<int32_t>((int64_t)b * a.N_rows + kbeg + (int64_t)i * kTile),
                        fb);
          }
        }
        if (*abort) {
          const int64_t first = ctr > nslot ? ctr - nslot : 0;
          for (int64_t x = first; x < ctr; ++x)
            mbar_wait(smem_u32(&sm->full[x % nslot]), (x / nslot) & 1, nullptr, nullptr,
                      10000000ull, 19);
        }
      }
    } else if (KIND == kSparse) {
      // 512 16-byte pieces per chunk: this thread copies pieces pt + 128 q
      const int32_t* idx_row = a.idx + ((int64_t)b * a.T + t0) * a.k;
      int64_t pending_from = 0;  // oldest counter not yet signalled
      for (int i = 0; i < nt && !*abort; ++i) {
        const __nv_bfloat16* src[4];
        int bytes[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int rI = (pt + 128 * q) >> 3;
          const int64_t kk = kbeg + (int64_t)i * kTile + rI;
          int32_t j = -1;
          if (kk < kend) j = idx_row[kk];
          if (j >= a.N_rows) {
            if ((pt & 7) == 0) record_status(a.status, kStatusBadIndex);
            j = -1;
          }
          bytes[q] = j >= 0 ? 16 : 0;
          src[q] = a.kv + ((int64_t)b * a.N_rows + (j >= 0 ? j : 0)) * a.D + ((pt + 128 * q) & 7) * 8;
        }
        for (int p = 0; p < ndc; ++p, ++ctr) {
          const int slot = static_cast<int>(ctr % nslot);
          if (ctr >= nslot &&
              !mbar_wait(smem_u32(&sm->empty[slot]), ((ctr / nslot) + 1) & 1, abort, a.status, kWaitLimitNs, 20))
            break;
          const int dcol = chunk_dc(p) * 64;
          const uint32_t dst = smem_u32(sRing + slot * 8192);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int pc = pt + 128 * q;
            cp_async16(dst + swz128(pc >> 3, pc & 7), src[q] + dcol, bytes[q]);
          }
          cp_async_commit();
          // signal the chunk `pd` counters back once its copies have landed
          if (ctr - pending_from >= pd) {
            if (pd == 0) cp_async_wait<0>();
            else if (pd == 1) cp_async_wait<1>();
            else cp_async_wait<2>();
            fence_proxy_async_smem();
            mbar_arrive(smem_u32(&sm->full[pending_from % nslot]));
            ++pending_from;
          }
        }
      }
      cp_async_wait<0>();
      fence_proxy_async_smem();
      for (; pending_from < ctr; ++pending_from)
        mbar_arrive(smem_u32(&sm->full[pending_from % nslot]));
    } else {
      // SWA: keys are RMSNorm'd and RoPE'd raw tokens at their own positions.
      // Warp w owns key rows [16w, 16w+16) of every chunk, so the per-row norms
      // it needs are its own and only warp-level synchronisation is used.
      for (int i = 0; i < nt && !*abort; ++i) {
        for (int rr = 0; rr < 16; ++rr) {
          const int rI = warp * 16 + rr;
          const int64_t kk = kbeg + (int64_t)i * kTile + rI;
          float ss = 0.f;
          if (kk < kend) {
            const __nv_bfloat16* row = a.kv + ((int64_t)b * a.N_rows + u_lo + kk) * a.D;
            for (int pc = lane; pc < a.D / 8; pc += 32) {
              float x[8];
              load8f(row + pc * 8, x);
#pragma unroll
              for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
            }
          }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
          if (lane == 0) sm->inv_rms[rI] = rsqrtf(ss / static_cast<float>(a.D) + a.eps);
        }
        __syncwarp();
        for (int p = 0; p < ndc; ++p, ++ctr) {
          const int slot = static_cast<int>(ctr % nslot);
          const bool got = ctr < nslot ||
                           mbar_wait(smem_u32(&sm->empty[slot]), ((ctr / nslot) + 1) & 1, abort,
                                     a.status, kWaitLimitNs, 21);
          if (!__all_sync(0xffffffffu, got)) break;  // warp-uniform (shuffles follow)
          const int dcol = chunk_dc(p) * 64;
          uint8_t* dst = sRing + slot * 8192;
          const int piece = lane & 7;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int rI = warp * 16 + (lane >> 3) + 4 * q;
            const int64_t kk = kbeg + (int64_t)i * kTile + rI;
            float y[8];
            if (kk < kend) {
              const int64_t u = u_lo + kk;
              load8f(a.kv + ((int64_t)b * a.N_rows + u) * a.D + dcol + piece * 8, y);
              const float inv = sm->inv_rms[rI];
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const float gm = a.gamma_kv ? a.gamma_kv[dcol + piece * 8 + e] : 1.f;
                y[e] = y[e] * inv * gm;
              }
              rope8(y, dcol + piece * 8, a.D, a.r, u, sm->theta);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) y[e] = 0.f;
            }
            *reinterpret_cast<uint4*>(dst + swz128(rI, piece)) = pack8(y);
          }
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&sm->full[slot]));
        }
        __syncwarp();  // inv_rms of this warp's rows is rewritten by the next tile
      }
    }
  } else if (warp == 4) {
    // ============================================================ MMA issuer
    const uint32_t idesc_qk = idesc_bf16(128, 64, 0, 0);
    const uint32_t idesc_pv = idesc_bf16(128, 64, 0, 1);
    const uint32_t sQa = smem_u32(sQ), sPa = smem_u32(sP), sRa = smem_u32(sRing);
    int64_t ctr = 0;
    bool ok = true;
    // wait for a chunk; for an HCA tail tile, zero its invalid key rows first
    auto wait_chunk = [&](int64_t c, int nvalid) -> bool {
      const int slot = static_cast<int>(c % nslot);
      const bool got = mbar_wait(smem_u32(&sm->full[slot]), (c / nslot) & 1, abort, a.status,
                                 kWaitLimitNs, 22);
      if (!__all_sync(0xffffffffu, got)) return false;  // warp-uniform
      if (KIND == kHca && nvalid < kTile) {
        uint8_t* dst = sRing + slot * 8192;
        for (int pc = nvalid * 8 + lane; pc < kTile * 8; pc += 32)
          *reinterpret_cast<uint4*>(dst + swz128(pc >> 3, pc & 7)) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      return true;
    };
    auto issue_qk = [&](int sb, int64_t c, bool first) {
      const int slot = static_cast<int>(c % nslot);
      const int dc = chunk_dc(static_cast<int>(c % ndc));
      if (lane == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = smem_desc(sQa + dc * 16384 + ks * 32, 16, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(sRa + slot * 8192 + ks * 32, 16, 1024, kSwizzle128B);
          mma_bf16_ss(tS + sb * 64, ad, bd, idesc_qk, (first && ks == 0) ? 0u : 1u);
        }
      }
      __syncwarp();
    };
    auto issue_pv = [&](int j) -> bool {
      const bool got = mbar_wait(smem_u32(&sm->p_full), j & 1, abort, a.status, kWaitLimitNs, 23);
      if (!__all_sync(0xffffffffu, got)) return false;  // warp-uniform
      if (lane == 0) {
        tc_fence_after();
        for (int e = 0; e < n_own; ++e) {
          const int64_t c = (int64_t)j * ndc + n_other + e;
          const int slot = static_cast<int>(c % nslot);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ad = smem_desc(sPa + ks * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(sRa + slot * 8192 + ks * 2048, 16, 1024, kSwizzle128B);
            mma_bf16_ss(tO + e * 64, ad, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&sm->empty[slot]));
        }
      }
      __syncwarp();
      return true;
    };
    for (int i = 0; i < nt && ok; ++i) {
      const int nvalid = static_cast<int>((kend - (kbeg + (int64_t)i * kTile)) < kTile ? (kend - (kbeg + (int64_t)i * kTile)) : kTile);
      const int sb = i & 1;
      // S(i) over the other half's chunks
      for (int p = 0; p < n_other && ok; ++p) {
        ok = wait_chunk(ctr + p, nvalid);
        if (ok) issue_qk(sb, ctr + p, p == 0);
      }
      if (!ok) break;
      if (lane == 0)
        for (int p = 0; p < n_other; ++p)
          mma_commit(smem_u32(&sm->empty[(ctr + p) % nslot]));
      __syncwarp();
      // O += P(i-1) V(i-1)
      if (i > 0 && !(ok = issue_pv(i - 1))) break;
      // S(i) over our chunks
      for (int p = n_other; p < ndc && ok; ++p) {
        ok = wait_chunk(ctr + p, nvalid);
        if (ok) issue_qk(sb, ctr + p, p == 0);
      }
      if (!ok) break;
      if (lane == 0) mma_commit(smem_u32(&sm->s_full[sb]));
      __syncwarp();
      ctr += ndc;
    }
    if (ok) ok = issue_pv(nt - 1);
    if (lane == 0) mma_commit(smem_u32(&sm->o_full));
    __syncwarp();
    if (!ok) {
      // wait (bounded) for the MMAs already issued before the memory is released
      mbar_wait(smem_u32(&sm->o_full), 0, nullptr, nullptr, 10000000ull, 24);
    }
  } else {
    // ============================================================ softmax
    const int quad = warp & 3;
    const int rI = quad * 32 + lane;
    const bool row_valid = rI < nrows;
    const int g = row_valid ? rI / a.H : 0;
    const int h = row_valid ? rI % a.H : 0;
    const int32_t tq = row_valid ? a.pos[(int64_t)b * a.T + t0 + g] : 0;
    // per-row key limits (absolute key coordinates of the branch)
    int64_t row_hi = 0, row_lo = 0;  // HCA: keys < row_hi; SWA: row_lo <= u <= row_hi
    if (KIND == kHca) {
      row_hi = vis(tq, a.m);
      if (row_hi > a.N_rows) row_hi = a.N_rows;
    } else if (KIND == kSwa) {
      row_lo = tq - a.W + 1;
      if (row_lo < 0) row_lo = 0;
      row_hi = tq;
    }
    const float sl2 = a.scale * 1.4426950408889634f;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    const int32_t* idx_row = a.idx + ((int64_t)b * a.T + t0) * a.k;
    float m_used = -INFINITY, l = 0.f;
    bool ok = true;
    for (int i = 0; i < nt; ++i) {
      const int64_t kt = kbeg + (int64_t)i * kTile;
      uint64_t colmask = 0;  // keys of this tile that exist for every row
      if (KIND == kSparse) {
        const int64_t k0 = kt + lane, k1 = kt + 32 + lane;
        const int32_t j0 = k0 < kend ? idx_row[k0] : -1;
        const int32_t j1 = k1 < kend ? idx_row[k1] : -1;
        const unsigned b0 = __ballot_sync(0xffffffffu, j0 >= 0 && j0 < a.N_rows);
        const unsigned b1 = __ballot_sync(0xffffffffu, j1 >= 0 && j1 < a.N_rows);
        colmask = static_cast<uint64_t>(b0) | (static_cast<uint64_t>(b1) << 32);
      } else {
        const int nv = static_cast<int>((kend - kt) < kTile ? (kend - kt) : kTile);
        colmask = nv >= 64 ? ~0ull : ((1ull << nv) - 1);
      }
      const int sb = i & 1;
      const bool got = mbar_wait(smem_u32(&sm->s_full[sb]), (i >> 1) & 1, abort, a.status,
                                 kWaitLimitNs, 25);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }  // warp-uniform exit
      tc_fence_after();
      float s[64];
      {
        float* s0 = s;
        float* s1 = s + 32;
        tmem_ld32(tS + lane_base + sb * 64, *reinterpret_cast<float(*)[32]>(s0));
        tmem_ld32(tS + lane_base + sb * 64 + 32, *reinterpret_cast<float(*)[32]>(s1));
        tmem_wait_ld();
      }
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        bool v = row_valid && ((colmask >> c) & 1ull);
        if (KIND == kHca) v = v && (kt + c < row_hi);
        if (KIND == kSwa) {
          const int64_t u = u_lo + kt + c;
          v = v && u >= row_lo && u <= row_hi;
        }
        s[c] = v ? s[c] * sl2 : -INFINITY;
        mx = fmaxf(mx, s[c]);
      }
      // Lazy rescale: only when the running max grows by more than 2^8.  The
      // tensor-memory loads/stores are warp-collective, so the decision is
      // taken per warp; lanes that need no rescale multiply by 1.
      const bool grow = mx > m_used + 8.f;
      const bool need_rescale = grow && m_used != -INFINITY && i > 0;
      if (__any_sync(0xffffffffu, need_rescale)) {
        const float f = need_rescale ? exp2f(m_used - mx) : 1.f;
        for (int cc = 0; cc < ocols; cc += 32) {
          float o[32];
          tmem_ld32(tO + lane_base + cc, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] *= f;
          tmem_st32(tO + lane_base + cc, o);
        }
        tmem_wait_st();
        l *= f;
      }
      if (grow) m_used = mx;
      uint8_t* prow = sP;
#pragma unroll
      for (int pc = 0; pc < 8; ++pc) {
        float y[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x = s[pc * 8 + e];
          const float p = (x == -INFINITY) ? 0.f : exp2f(x - m_used);
          y[e] = bf16_round(p);
          l += y[e];
        }
        *reinterpret_cast<uint4*>(prow + swz128(rI, pc)) = pack8(y);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->p_full));
    }
    // ------------------------------------------------------------ epilogue
    // The tensor-memory loads are warp-collective: every lane of the warp runs
    // them; only rows that exist store.
    bool done = ok && mbar_wait(smem_u32(&sm->o_full), 0, abort, a.status, kWaitLimitNs, 40);
    done = __all_sync(0xffffffffu, done);
    if (done) {
      tc_fence_after();
      const int64_t row = ((int64_t)b * a.T + t0 + g) * a.H + h;
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const float lse = l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
      for (int cc = 0; cc < ocols; cc += 32) {
        float o[32];
        tmem_ld32(tO + lane_base + cc, o);
        tmem_wait_ld();
        if (!row_valid) continue;
        if (a.nsplit == 1) {
          __nv_bfloat16* dst = a.o + row * a.D + dh * ocols + cc;
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            float y[8];
#pragma unroll
            for (int z = 0; z < 8; ++z) y[z] = o[e + z] * inv_l;
            *reinterpret_cast<uint4*>(dst + e) = pack8(y);
          }
        } else {
          float* dst = a.part_o + (row * a.nsplit + split) * a.D + dh * ocols + cc;
#pragma unroll
          for (int e = 0; e < 32; e += 4)
            *reinterpret_cast<float4*>(dst + e) =
                make_float4(o[e] * inv_l, o[e + 1] * inv_l, o[e + 2] * inv_l, o[e + 3] * inv_l);
        }
      }
      if (row_valid && dh == 0) {
        if (a.nsplit == 1) a.lse[row] = lse;
        else a.part_lse[row * a.nsplit + split] = lse;
      }
    } else {
      // drain: make sure no MMA is still writing the accumulators
      mbar_wait(smem_u32(&sm->o_full), 0, nullptr, nullptr, 10000000ull, 41);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 4) tmem_dealloc(tmem, 512);
}

}  // namespace

bool plan_attention(int kind, int B, int T, int H, int D, int64_t n_keys, int num_sms,
                    AttnPlan* p) {
  if (H < 1 || H > 128 || D < 64 || D > 512 || (D % 64) || B < 1 || T < 1) return false;
  const int G = (kind == kSparse) ? 1 : (128 / H);
  const int n_rb = (T + G - 1) / G;
  const int nds = D > 256 ? 2 : 1;
  const int64_t max_keys = kind == kSwa ? (n_keys + G - 1) : n_keys;
  const int64_t tiles = (max_keys + kTile - 1) / kTile;
  const int64_t pairs = (int64_t)B * n_rb;
  int64_t nsplit = num_sms / (nds * pairs);
  if (nsplit < 1) nsplit = 1;
  if (nsplit > tiles) nsplit = tiles > 0 ? tiles : 1;
  int64_t tps = (tiles + nsplit - 1) / nsplit;
  if (tps < 1) tps = 1;
  nsplit = (tiles + tps - 1) / tps;
  if (nsplit < 1) nsplit = 1;
  if (nsplit > 65535) return false;
  p->G = G;
  p->n_rb = n_rb;
  p->nds = nds;
  p->nsplit = static_cast<int>(nsplit);
  p->keys_per_split = static_cast<int>(tps * kTile);
  const int ndc = D / 64;
  const size_t fixed = 1024 + (size_t)ndc * 16384 + 16384 + sizeof(AttnShared);
  int nslot = static_cast<int>((227 * 1024 - fixed) / 8192);
  if (nslot > kMaxSlots) nslot = kMaxSlots;
  if (nslot < ndc + 2) return false;
  p->nslot = nslot;
  p->smem_bytes = fixed + (size_t)nslot * 8192;
  p->ws_bytes = p->nsplit > 1 ? (size_t)B * T * H * p->nsplit * (D + 1) * sizeof(float) : 0;
  return true;
}

cudaError_t launch_attention(const CUtensorMap& tm_kv, const AttnArgs& a, const AttnPlan& p,
                             cudaStream_t stream) {
  const int ndc = a.D / 64;
  const int n_own = ndc / p.nds;
  // the producer may run `pd` chunks ahead of its completion signals without
  // waiting on a slot that only frees after one of those signals
  int pd = p.nslot - ndc;
  (void)n_own;
  if (pd > 2) pd = 2;
  if (pd < 0) pd = 0;
  dim3 grid(p.nds * p.nsplit, p.n_rb, a.B);
  cudaError_t e = cudaSuccess;
  switch (a.kind) {
    case kSparse:
      e = cudaFuncSetAttribute(attn_kernel<kSparse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(p.smem_bytes));
      if (e == cudaSuccess)
        attn_kernel<kSparse><<<grid, kThreads, p.smem_bytes, stream>>>(tm_kv, a, p.nslot, pd);
      break;
    case kHca:
      e = cudaFuncSetAttribute(attn_kernel<kHca>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(p.smem_bytes));
      if (e == cudaSuccess)
        attn_kernel<kHca><<<grid, kThreads, p.smem_bytes, stream>>>(tm_kv, a, p.nslot, pd);
      break;
    default:
      e = cudaFuncSetAttribute(attn_kernel<kSwa>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(p.smem_bytes));
      if (e == cudaSuccess)
        attn_kernel<kSwa><<<grid, kThreads, p.smem_bytes, stream>>>(tm_kv, a, p.nslot, pd);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hattn
