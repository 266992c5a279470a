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
// dimension), a key range (one split of the visible keys) and a share of
// the head dim.  For D > 256 the fp32 accumulator of 128 rows x D columns
// does not fit the tensor memory next to S, so two CTAs of a cluster split
// D in halves (nds = 2): each holds its half of Q, reads only its half of
// every key row, computes a partial S over its half and accumulates its half
// of O.  The two fp32 partials of S are swapped through distributed shared
// memory every tile and summed identically on both sides (fp32 addition is
// commutative), so both CTAs run the same softmax.  Per 64-key tile:
//   S_half = Q_half K_half^T    (M=128, N=64, K=D/nds)   -> tensor memory
//   S = S_half + S_peer;  online softmax (one thread per row, lazy rescale)
//   O_half += P V_half          (M=128, N=64 per 64-column chunk, K=64 keys)
// Key rows reach shared memory as 64x64 bf16 chunks (8 KB, 128-byte
// swizzle) in a ring of `nslot` slots: HCA by TMA tiles, CSA by a 16-byte
// cp.async gather through the top-k indices, SWA by TMA tiles normalised and
// roped in place.  Warps 0-3 produce chunks (from kernel entry), warp 4
// loads Q by TMA and issues the MMAs, warps 5-8 normalise Q, then run the
// softmax, the S exchange and the epilogue.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kThreads = 288;
constexpr int kTile = 64;
constexpr int kMaxSlots = 16;
constexpr int kProdThreads = 128;
constexpr int kXBytes = 2 * 128 * kTile * 4;  // S exchange buffers, 2 x 32 KB

struct AttnShared {
  uint64_t full[kMaxSlots];
  uint64_t raw[kMaxSlots];  // SWA: the TMA copy of a raw chunk has landed
  uint64_t empty[kMaxSlots];
  uint64_t s_full[2];
  uint64_t x_full[2];       // the peer's S partial of this tile is here
  uint64_t x_empty[2];      // the peer has read what this CTA sent it
  uint64_t p_full;
  uint64_t pv_done;
  uint64_t o_full;
  uint64_t q_full;
  uint32_t tmem_base;
  int abort;
  float inv_rms[2][kTile];  // SWA: per-row norms, double-buffered by tile
  float rc[4][kMaxRopePairs];  // RoPE coefficients (see RopeCoef)
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

__device__ __forceinline__ void unpack8(const uint4& u, float (&x)[8]) {
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

__device__ __forceinline__ float sumsq8(const uint4& u) {
  float x[8];
  unpack8(u, x);
  float s = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) s = fmaf(x[e], x[e], s);
  return s;
}

// RoPE on the pairs of an 8-element piece starting at dim d_first, at
// position p (angles computed here).
__device__ __forceinline__ void rope8(float (&y)[8], int d_first, int D, int r, int64_t p,
                                      const float (*rc)[kMaxRopePairs]) {
  const int d0 = D - r;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const int d = d_first + e;
    if (d >= d0) {
      float sn, cs;
      rope_cs(rc, (d - d0) >> 1, p, &sn, &cs);
      const float x0 = y[e], x1 = y[e + 1];
      y[e] = x0 * cs - x1 * sn;
      y[e + 1] = x0 * sn + x1 * cs;
    }
  }
}

// The same with the (cos, sin) of every pair of the position precomputed.
__device__ __forceinline__ void rope8_tab(float (&y)[8], int d_first, int D, int r,
                                          const float2* cs_row) {
  const int d0 = D - r;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const int d = d_first + e;
    if (d >= d0) {
      const float2 t = cs_row[(d - d0) >> 1];
      const float x0 = y[e], x1 = y[e + 1];
      y[e] = x0 * t.x - x1 * t.y;
      y[e + 1] = x0 * t.y + x1 * t.x;
    }
  }
}

// Byte offset of float4 number c (0..15) of row r in an S exchange buffer
// (256 B per row; the swizzle spreads the 32 rows of a warp over the banks).
__device__ __forceinline__ uint32_t xoff(int r, int c) {
  return static_cast<uint32_t>(r) * 256u + (static_cast<uint32_t>(c ^ (r & 15)) << 4);
}

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_q,
                const __grid_constant__ AttnArgs a, const int nslot, const int pd) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int nds = a.nds;
  const int ndc = a.D / 64;                // 64-wide d chunks of a full row
  const int n_own = ndc / nds;             // chunks of this CTA's share of D
  uint8_t* sQ = base;                      // n_own x [128 rows x 128 B]
  uint8_t* sX = sQ + n_own * 16384;        // nds == 2: S exchange, 2 x [128 x 64] fp32
  uint8_t* sP = sX + (nds == 2 ? kXBytes : 0);  // [128 rows x 64 keys] bf16
  uint8_t* sRing = sP + 16384;             // nslot x [64 keys x 128 B]
  AttnShared* sm = reinterpret_cast<AttnShared*>(sRing + nslot * 8192);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int dh = blockIdx.x % nds;         // = rank in the cluster of a pair
  const int split = blockIdx.x / nds;
  const int rb = blockIdx.y;
  const int b = blockIdx.z;
  const int t0 = rb * a.G;
  const int gv = min(a.G, a.T - t0);
  const int nrows = gv * a.H;
  const uint32_t peer = static_cast<uint32_t>(dh ^ 1);

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
    // empty split (the same for both CTAs of a pair): o = 0, lse = -inf
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
      mbar_init(smem_u32(&sm->raw[i]), 1);
      mbar_init(smem_u32(&sm->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm->s_full[i]), 1);
      mbar_init(smem_u32(&sm->x_full[i]), 128);
      mbar_init(smem_u32(&sm->x_empty[i]), 128);
    }
    mbar_init(smem_u32(&sm->p_full), 128);
    mbar_init(smem_u32(&sm->pv_done), 1);
    mbar_init(smem_u32(&sm->o_full), 1);
    mbar_init(smem_u32(&sm->q_full), 1);
    sm->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    if (KIND != kSparse) tma_prefetch_desc(&tm_kv);
  }
  const int npair = a.r / 2;
  for (int i = threadIdx.x; i < npair; i += kThreads) {
#pragma unroll
    for (int c = 0; c < 4; ++c) sm->rc[c][i] = a.rope.c[c][i];
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(&sm->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // the peer's barriers are initialised before anything of it is touched
  if (nds == 2) cluster_sync_all();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort = &sm->abort;
  const uint32_t tS = tmem;          // columns [0, 128): two 64-column S buffers
  const uint32_t tO = tmem + 128;    // columns [128, 128 + ocols)

  if (warp < 4) {
    // ============================================================ producers
    const int pt = threadIdx.x;  // 0..127
    int64_t ctr = 0;
    int slot = 0;
    uint32_t ph = 0;  // ring position (slot, phase) of counter ctr
    auto advance = [&]() {
      ++ctr;
      if (++slot == nslot) { slot = 0; ph ^= 1u; }
    };
    if (KIND == kHca) {
      if (pt == 0) {
        for (int i = 0; i < nt && !*abort; ++i) {
          for (int e = 0; e < n_own; ++e, advance()) {
            if (ctr >= nslot &&
                !mbar_wait(smem_u32(&sm->empty[slot]), ph ^ 1u, abort, a.status, kWaitLimitNs, 18))
              break;
            const uint32_t fb = smem_u32(&sm->full[slot]);
            mbar_arrive_expect_tx(fb, 8192);
            tma_load_2d(smem_u32(sRing + slot * 8192), &tm_kv, (dh * n_own + e) * 64,
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
          src[q] = a.kv + ((int64_t)b * a.N_rows + (j >= 0 ? j : 0)) * a.D +
                   ((pt + 128 * q) & 7) * 8;
        }
        for (int e = 0; e < n_own; ++e, advance()) {
          if (ctr >= nslot &&
              !mbar_wait(smem_u32(&sm->empty[slot]), ph ^ 1u, abort, a.status, kWaitLimitNs, 20))
            break;
          const int dcol = (dh * n_own + e) * 64;
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
      // Row norms come first, from the full rows in global memory (two
      // threads per row, eight 16-byte loads in flight each); then each
      // chunk of this CTA's half is copied by TMA and normalised in place.
      const int nr = pt >> 1, hf = pt & 1;
      const int half_pieces = a.D / 16;  // 16-byte pieces per half row
      bool ok = true;
      for (int i = 0; i < nt; ++i) {
        const int64_t kt = kbeg + (int64_t)i * kTile;
        const int nvalid = static_cast<int>((kend - kt) < kTile ? (kend - kt) : kTile);
        float ss = 0.f;
        if (nr < nvalid) {
          const uint4* row = reinterpret_cast<const uint4*>(
              a.kv + ((int64_t)b * a.N_rows + u_lo + kt + nr) * a.D) + hf * half_pieces;
          for (int p0 = 0; p0 < half_pieces; p0 += 8) {
            uint4 v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = p0 + e < half_pieces ? __ldg(row + p0 + e)
                                                                    : make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int e = 0; e < 8; ++e) ss += sumsq8(v[e]);
          }
        }
        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
        if (hf == 0) sm->inv_rms[i & 1][nr] = rsqrtf(ss / static_cast<float>(a.D) + a.eps);
        // the loop contains this barrier: all 128 threads leave it together
        if (!named_bar_and(3, kProdThreads, ok && !*abort)) break;
        const float* inv_rms = sm->inv_rms[i & 1];
        for (int e = 0; e < n_own; ++e, advance()) {
          if (pt == 0 && ok) {
            ok = ctr < nslot ||
                 mbar_wait(smem_u32(&sm->empty[slot]), ph ^ 1u, abort, a.status, kWaitLimitNs, 21);
            if (ok) {
              const uint32_t rb_ = smem_u32(&sm->raw[slot]);
              mbar_arrive_expect_tx(rb_, 8192);
              tma_load_2d(smem_u32(sRing + slot * 8192), &tm_kv, (dh * n_own + e) * 64,
                          static_cast<int32_t>((int64_t)b * a.N_rows + u_lo + kt), rb_);
            }
          }
          if (ok) ok = mbar_wait(smem_u32(&sm->raw[slot]), ph, abort, a.status, kWaitLimitNs, 26);
          if (!ok) continue;  // no copy to wait for; the next barrier ends the loop
          const int dcol = (dh * n_own + e) * 64;
          uint8_t* dst = sRing + slot * 8192;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int pc = pt + 128 * q;
            const int rI = pc >> 3, piece = pc & 7;
            uint4* cell = reinterpret_cast<uint4*>(dst + swz128(rI, piece));
            float y[8];
            if (rI < nvalid) {
              unpack8(*cell, y);
              const float inv = inv_rms[rI];
#pragma unroll
              for (int z = 0; z < 8; ++z) {
                const float gm = a.gamma_kv ? a.gamma_kv[dcol + piece * 8 + z] : 1.f;
                y[z] = y[z] * inv * gm;
              }
              rope8(y, dcol + piece * 8, a.D, a.r, u_lo + kt + rI, sm->rc);
            } else {
#pragma unroll
              for (int z = 0; z < 8; ++z) y[z] = 0.f;
            }
            *cell = pack8(y);
          }
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&sm->full[slot]));
        }
      }
      if (!ok && pt == 0) {
        // copies issued whose completion nobody waited for land before exit
        const int64_t first = ctr > nslot ? ctr - nslot : 0;
        for (int64_t x = first; x < ctr; ++x)
          mbar_wait(smem_u32(&sm->raw[x % nslot]), (x / nslot) & 1, nullptr, nullptr,
                    10000000ull, 27);
      }
    }
  } else if (warp == 4) {
    // ============================================================ Q load + MMA issuer
    const int64_t qrow0 = ((int64_t)b * a.T + t0) * a.H;
    if (lane == 0) {
      const uint32_t qb = smem_u32(&sm->q_full);
      mbar_arrive_expect_tx(qb, static_cast<uint32_t>(ndc) * 16384u);
      for (int dc = 0; dc < ndc; ++dc) {
        uint8_t* dst = (dc / n_own == dh ? sQ : sX) + (dc % n_own) * 16384;
        tma_load_2d(smem_u32(dst), &tm_q, dc * 64, static_cast<int32_t>(qrow0), qb);
      }
    }
    named_bar_sync(2, 160);  // Q normalised (warps 4-8)
    const uint32_t idesc_qk = idesc_bf16(128, 64, 0, 0);
    const uint32_t idesc_pv = idesc_bf16(128, 64, 0, 1);
    const uint32_t sQa = smem_u32(sQ), sPa = smem_u32(sP), sRa = smem_u32(sRing);
    bool ok = true;
    // wait for a chunk; for an HCA tail tile, zero its invalid key rows first
    auto wait_chunk = [&](int s, uint32_t phase, int nvalid) -> bool {
      const bool got = mbar_wait(smem_u32(&sm->full[s]), phase, abort, a.status, kWaitLimitNs, 22);
      if (!__all_sync(0xffffffffu, got)) return false;  // warp-uniform
      if (KIND == kHca && nvalid < kTile) {
        uint8_t* dst = sRing + s * 8192;
        for (int pc = nvalid * 8 + lane; pc < kTile * 8; pc += 32)
          *reinterpret_cast<uint4*>(dst + swz128(pc >> 3, pc & 7)) = make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      __syncwarp();
      return true;
    };
    // PV of tile j, whose chunks start at ring position (s0, ...)
    auto issue_pv = [&](int j, int s0) -> bool {
      const bool got = mbar_wait(smem_u32(&sm->p_full), j & 1, abort, a.status, kWaitLimitNs, 23);
      if (!__all_sync(0xffffffffu, got)) return false;  // warp-uniform
      if (lane == 0) {
        tc_fence_after();
        int s = s0;
        for (int e = 0; e < n_own; ++e) {
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ad = smem_desc(sPa + ks * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(sRa + s * 8192 + ks * 2048, 16, 1024, kSwizzle128B);
            mma_bf16_ss(tO + e * 64, ad, bd, idesc_pv, (j > 0 || ks > 0) ? 1u : 0u);
          }
          mma_commit(smem_u32(&sm->empty[s]));
          if (++s == nslot) s = 0;
        }
        mma_commit(smem_u32(&sm->pv_done));
      }
      __syncwarp();
      return true;
    };
    int slot = 0, prev_slot = 0;
    uint32_t ph = 0;
    for (int i = 0; i < nt && ok; ++i) {
      const int64_t kt = kbeg + (int64_t)i * kTile;
      const int nvalid = static_cast<int>((kend - kt) < kTile ? (kend - kt) : kTile);
      const int sb = i & 1;
      const int tile_slot = slot;
      // S(i) = Q_half K_half(i)^T
      for (int e = 0; e < n_own && ok; ++e) {
        ok = wait_chunk(slot, ph, nvalid);
        if (ok && lane == 0) {
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t ad = smem_desc(sQa + e * 16384 + ks * 32, 16, 1024, kSwizzle128B);
            const uint64_t bd = smem_desc(sRa + slot * 8192 + ks * 32, 16, 1024, kSwizzle128B);
            mma_bf16_ss(tS + sb * 64, ad, bd, idesc_qk, (e == 0 && ks == 0) ? 0u : 1u);
          }
        }
        __syncwarp();
        if (++slot == nslot) { slot = 0; ph ^= 1u; }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(smem_u32(&sm->s_full[sb]));
      __syncwarp();
      // O += P(i-1) V(i-1), while the softmax works on S(i)
      if (i > 0 && !(ok = issue_pv(i - 1, prev_slot))) break;
      prev_slot = tile_slot;
    }
    if (ok) ok = issue_pv(nt - 1, prev_slot);
    if (lane == 0) mma_commit(smem_u32(&sm->o_full));
    __syncwarp();
    if (!ok) {
      // wait (bounded) for the MMAs already issued before the memory is released
      mbar_wait(smem_u32(&sm->o_full), 0, nullptr, nullptr, 10000000ull, 24);
    }
  } else {
    // ============================================================ softmax
    const int quad = warp & 3;             // tensor-memory lane quarter of this warp
    const int rI = quad * 32 + lane;
    const int st = threadIdx.x - 160;      // 0..127 within warps 5-8
    const bool row_valid = rI < nrows;
    const int g = row_valid ? rI / a.H : 0;
    const int h = row_valid ? rI % a.H : 0;
    const int32_t tq = row_valid ? a.pos[(int64_t)b * a.T + t0 + g] : 0;

    // ---------------------------------------------------------- Q prologue
    // q~ = RoPE_t(RMSNorm(q; gamma_q, eps)) of every row, in place in sQ; the
    // other half of the row (nds = 2), staged in sX, only enters the norm.
    float2* qcs = reinterpret_cast<float2*>(sP);  // free until the first softmax
    const bool qtab = gv * npair <= 16384 / static_cast<int>(sizeof(float2));
    if (qtab)
      for (int e = st; e < gv * npair; e += 128) {
        const int gg = e / npair, i = e % npair;
        float sn, cs;
        rope_cs(sm->rc, i, a.pos[(int64_t)b * a.T + t0 + gg], &sn, &cs);
        qcs[e] = make_float2(cs, sn);
      }
    named_bar_sync(1, 128);
    bool qok = mbar_wait(smem_u32(&sm->q_full), 0, abort, a.status, kWaitLimitNs, 29);
    {
      float ss = 0.f;
      if (row_valid && qok) {
        for (int dc = 0; dc < ndc; ++dc) {
          const uint8_t* src = (dc / n_own == dh ? sQ : sX) + (dc % n_own) * 16384;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            ss += sumsq8(*reinterpret_cast<const uint4*>(src + swz128(rI, q)));
        }
      }
      const float inv = rsqrtf(ss / static_cast<float>(a.D) + a.eps);
      for (int e = 0; e < n_own; ++e) {
        const int dc = dh * n_own + e;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4* cell = reinterpret_cast<uint4*>(sQ + e * 16384 + swz128(rI, q));
          float y[8];
          if (row_valid && qok) {
            unpack8(*cell, y);
#pragma unroll
            for (int z = 0; z < 8; ++z) {
              const float gm = a.gamma_q ? a.gamma_q[dc * 64 + q * 8 + z] : 1.f;
              y[z] = y[z] * inv * gm;
            }
            if (qtab) rope8_tab(y, dc * 64 + q * 8, a.D, a.r, qcs + g * npair);
            else rope8(y, dc * 64 + q * 8, a.D, a.r, tq, sm->rc);
          } else {
#pragma unroll
            for (int z = 0; z < 8; ++z) y[z] = 0.f;
          }
          *cell = pack8(y);
        }
      }
    }
    fence_proxy_async_smem();
    // the staging in sX is consumed: the peer may now write its S partials
    uint32_t peer_x_full[2] = {0, 0}, peer_x_empty[2] = {0, 0}, peer_xbuf = 0;
    if (nds == 2) {
      for (int i = 0; i < 2; ++i) {
        peer_x_full[i] = mapa_shared(smem_u32(&sm->x_full[i]), peer);
        peer_x_empty[i] = mapa_shared(smem_u32(&sm->x_empty[i]), peer);
        mbar_arrive_remote(peer_x_empty[i]);
      }
      peer_xbuf = mapa_shared(smem_u32(sX), peer);
    }
    named_bar_sync(1, 128);  // every row of the P area's RoPE table is used
    named_bar_sync(2, 160);  // Q ready for the MMA warp

    // ---------------------------------------------------------- softmax
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
    bool ok = __all_sync(0xffffffffu, qok);
    for (int i = 0; i < nt && ok; ++i) {
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
      const uint32_t xph = (i >> 1) & 1;
      bool got = mbar_wait(smem_u32(&sm->s_full[sb]), xph, abort, a.status, kWaitLimitNs, 25);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }  // warp-uniform exit
      tc_fence_after();
      float s[64];
      tmem_ld32(tS + lane_base + sb * 64, *reinterpret_cast<float(*)[32]>(s));
      tmem_ld32(tS + lane_base + sb * 64 + 32, *reinterpret_cast<float(*)[32]>(s + 32));
      tmem_wait_ld();
      if (nds == 2) {
        // swap the fp32 partials of this row with the peer and sum them
        got = mbar_wait_cluster(smem_u32(&sm->x_empty[sb]), xph, abort, a.status, kWaitLimitNs,
                                30);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const uint32_t dst = peer_xbuf + sb * (kXBytes / 2);
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_cluster_v4(dst + xoff(rI, c),
                        make_float4(s[4 * c], s[4 * c + 1], s[4 * c + 2], s[4 * c + 3]));
        mbar_arrive_remote(peer_x_full[sb]);
        got = mbar_wait_cluster(smem_u32(&sm->x_full[sb]), xph, abort, a.status, kWaitLimitNs, 31);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        const uint8_t* xb = sX + sb * (kXBytes / 2);
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 v = *reinterpret_cast<const float4*>(xb + xoff(rI, c));
          s[4 * c] += v.x;
          s[4 * c + 1] += v.y;
          s[4 * c + 2] += v.z;
          s[4 * c + 3] += v.w;
        }
        mbar_arrive_remote(peer_x_empty[sb]);
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
      // O may be rescaled below only once PV(i-1) has finished writing it
      if (i > 0) {
        got = mbar_wait(smem_u32(&sm->pv_done), (i - 1) & 1, abort, a.status, kWaitLimitNs, 32);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
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
        *reinterpret_cast<uint4*>(sP + swz128(rI, pc)) = pack8(y);
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
  // keep this CTA's shared memory alive until the peer is done with it
  if (nds == 2) cluster_sync_all();
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
  if (nsplit * nds > 65535 || n_rb > 65535) return false;
  p->G = G;
  p->n_rb = n_rb;
  p->nds = nds;
  p->nsplit = static_cast<int>(nsplit);
  p->keys_per_split = static_cast<int>(tps * kTile);
  const int ndc = D / 64;
  if (ndc % nds) return false;  // the halves of a split row are whole chunks
  const int n_own = ndc / nds;
  const size_t fixed = 1024 + (size_t)n_own * 16384 + (nds == 2 ? kXBytes : 0) + 16384 +
                       sizeof(AttnShared);
  int nslot = static_cast<int>((227 * 1024 - fixed) / 8192);
  if (nslot > kMaxSlots) nslot = kMaxSlots;
  // QK of the next tile is issued before PV of the current one: two tiles of
  // this CTA's chunks must fit the ring at once
  if (nslot < 2 * n_own + 1) return false;
  if (nds == 2 && n_own * 16384 > kXBytes) return false;  // Q staging fits sX
  p->nslot = nslot;
  p->smem_bytes = fixed + (size_t)nslot * 8192;
  p->ws_bytes = p->nsplit > 1 ? (size_t)B * T * H * p->nsplit * (D + 1) * sizeof(float) : 0;
  return true;
}

cudaError_t launch_attention(const CUtensorMap& tm_kv, const CUtensorMap& tm_q, const AttnArgs& a,
                             const AttnPlan& p, cudaStream_t stream) {
  const int ndc = a.D / 64;
  const int n_own = ndc / p.nds;
  // the sparse producer may run `pd` chunks ahead of its completion signals
  // without waiting on a slot that only frees after one of those signals
  int pd = p.nslot - 2 * n_own;
  if (pd > 2) pd = 2;
  if (pd < 0) pd = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nds * p.nsplit, p.n_rb, a.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = p.nds;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.attrs = at;
  cfg.numAttrs = p.nds > 1 ? 1 : 0;  // the two CTAs of a split row form a cluster
  cudaError_t e = cudaSuccess;
  switch (a.kind) {
    case kSparse:
      e = cudaFuncSetAttribute(attn_kernel<kSparse>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(p.smem_bytes));
      if (e == cudaSuccess)
        e = cudaLaunchKernelEx(&cfg, attn_kernel<kSparse>, tm_kv, tm_q, a, p.nslot, pd);
      break;
    case kHca:
      e = cudaFuncSetAttribute(attn_kernel<kHca>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(p.smem_bytes));
      if (e == cudaSuccess)
        e = cudaLaunchKernelEx(&cfg, attn_kernel<kHca>, tm_kv, tm_q, a, p.nslot, pd);
      break;
    default:
      e = cudaFuncSetAttribute(attn_kernel<kSwa>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(p.smem_bytes));
      if (e == cudaSuccess)
        e = cudaLaunchKernelEx(&cfg, attn_kernel<kSwa>, tm_kv, tm_q, a, p.nslot, pd);
      break;
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hattn
