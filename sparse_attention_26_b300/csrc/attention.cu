// attention.cu -- the three attention branches of the hybrid layer on the
// tcgen05 tensor cores, with split-KV partials.
//
// "Why DeepSeek V4 Stands Apart", section "Core Architectural Innovations":
// SWA attends to the most recent 128 tokens; CSA attends to the top-k
// selected compressed entries; HCA attends densely to the 128:1 compressed
// entries.  "DeepSeek-V4" atlas, section "Inference efficiency": shared-KV
// MQA, one D-dim latent per key serves as key and value for every head.
//
// The kernel reads prepared queries q~ = RoPE(RMSNorm(q)) (qprep.cu).  One
// CTA owns a row block (G queries x H heads <= 128 rows, the MMA M
// dimension), a key range (one split of the visible keys) and a share of the
// output columns.  For D > 256 the fp32 accumulator of 128 rows x D columns
// would fill the tensor memory, so two CTAs (nds = 2) each keep half of O
// and both compute the full S; each keeps its own half of Q in shared memory
// and the other half in the tensor memory left over (S 128 + O 256 + Q 128
// columns), which leaves room for a ring deep enough to prefetch whole tiles.
// Per 64-key tile:
//   S = Q K^T   (M=128, N=64, K=D; A from shared or tensor memory)
//   softmax     (one thread per row, online max with lazy rescaling); the
//               bf16 P overwrites the consumed S columns in tensor memory
//   O += P V    (A = P from tensor memory; M=128, N=64 per 64-column chunk)
// Key rows reach shared memory as 64x64 bf16 chunks (8 KB, 128-byte
// swizzle) in a ring of `nslot` slots: HCA by TMA tiles, CSA by a 16-byte
// cp.async gather through the top-k indices, SWA by TMA tiles normalised and
// roped in place.  Warps 0-3 produce chunks from kernel entry; warps 4 and 9
// issue the QK products of even and odd tiles (one S buffer each; a single
// thread issues a tcgen05.mma only every ~50 ns, so two issuers keep the
// tensor core busier), warp 10 issues the PV products (one N = D/nds MMA
// per 16 keys), warps 5-8 run the softmax and the epilogue, which writes
// whole fp32 rows through shared memory so every store instruction is
// contiguous.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kThreads = 352;
constexpr int kTile = 64;
constexpr int kNSB = 3;  // S/P buffers in tensor memory (64 columns each)
constexpr int kMaxSlots = 20;
constexpr int kProdThreads = 128;

struct AttnShared {
  uint64_t full[kMaxSlots];
  uint64_t raw[kMaxSlots];  // SWA: the TMA copy of a raw chunk has landed
  uint64_t empty[kMaxSlots];
  uint64_t s_full[kNSB];
  uint64_t s_free[kNSB];    // PV of the tile that last used this S/P buffer is done
  uint64_t p_full[kNSB];    // P of the tile using this S/P buffer is in tensor memory
  uint64_t o_full;
  uint64_t q_full;
  uint64_t q_tmem;          // the other half of Q is in tensor memory
  uint64_t q_ready;         // Q complete (both MMA warps may start)
  uint64_t drain[2];        // the QK warps' own MMAs have completed
  uint32_t tmem_base;
  int abort;
  float inv_rms[2][kTile];  // SWA: per-row norms, double-buffered by tile
};

__device__ __forceinline__ int64_t vis(int32_t t, int m) {
  return t < 0 ? 0 : (static_cast<int64_t>(t) + 1) / m;
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}
// Arrive (once) on the mbarrier when every cp.async this thread issued so
// far has landed; the arrival counts against the barrier's expected count.
__device__ __forceinline__ void cp_async_mbar_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// 2^x on the special-function unit (relative error ~2^-22; 2^-inf = +0).
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

__device__ __forceinline__ uint4 pack8_f16(const float (&y)[8]) {
  uint4 u;
  u.x = pack_f16x2(y[0], y[1]);
  u.y = pack_f16x2(y[2], y[3]);
  u.z = pack_f16x2(y[4], y[5]);
  u.w = pack_f16x2(y[6], y[7]);
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
// position p.
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

// Fused kind: one query's keys are three segments of 64-key tiles -- 0: the
// top-k CSA entries (gathered), 1: the visible HCA entries, 2: the query's W
// SWA keys (both by TMA).  Split s of nsplit takes tiles
// [s*n/nsplit, (s+1)*n/nsplit) of each segment, so every split gets its share
// of the gathered and the streamed tiles.
struct SegTiles {
  int first[3], count[3];
  int64_t nkeys[3];
  __device__ __forceinline__ void init(int64_t n0, int64_t n1, int64_t n2, int split,
                                       int nsplit) {
    nkeys[0] = n0;
    nkeys[1] = n1;
    nkeys[2] = n2;
#pragma unroll
    for (int g = 0; g < 3; ++g) {
      const int64_t t = (nkeys[g] + kTile - 1) / kTile;
      const int64_t lo = t * split / nsplit, hi = t * (split + 1) / nsplit;
      first[g] = static_cast<int>(lo);
      count[g] = static_cast<int>(hi - lo);
    }
  }
  __device__ __forceinline__ int total() const { return count[0] + count[1] + count[2]; }
  // tile i of this split: its segment, first key (within the segment) and
  // number of keys
  __device__ __forceinline__ void map(int i, int& seg, int64_t& kt, int& nvalid) const {
    seg = 0;
    if (i >= count[0]) {
      i -= count[0];
      seg = 1;
      if (i >= count[1]) {
        i -= count[1];
        seg = 2;
      }
    }
    kt = static_cast<int64_t>(first[seg] + i) * kTile;
    const int64_t rem = nkeys[seg] - kt;
    nvalid = static_cast<int>(rem < kTile ? rem : kTile);
  }
};

template <int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ CUtensorMap tm_kv,
                const __grid_constant__ CUtensorMap tm_kv2,
                const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ AttnArgs a,
                const int nslot) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int ndc = a.D / 64;                // 64-wide d chunks of a row
  const int n_own = ndc / a.nds;           // chunks of this CTA's output columns
  const int n_other = ndc - n_own;
  const int n_tq = a.n_tq;                 // chunks of the other half held in tensor memory
  const int n_sq = n_own + n_other - n_tq; // chunks of Q held in shared memory
  uint8_t* sQ = base;                      // n_sq x [128 rows x 128 B]: own chunks, then
                                           // the other half's shared-memory chunks
  uint8_t* sRing = sQ + n_sq * 16384;      // nslot x [64 keys x 128 B]
  AttnShared* sm = reinterpret_cast<AttnShared*>(sRing + nslot * 8192);
  // the other half's tensor-memory chunks of Q are staged in the last ring
  // slots until they have been copied into tensor memory
  const int stage_slot = nslot - 2 * n_tq;
  uint8_t* sQstage = sRing + stage_slot * 8192;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The SWA branch normalises and ropes its keys in this kernel, so their
  // products run in fp16 (11 significant bits): Q is converted once, the
  // normalised keys and P are rounded to fp16 rather than bf16.  Every other
  // kind reads bf16 caches and runs in bf16.
  constexpr bool kF16 = KIND == kSwa;
  pdl_trigger();  // the merge may begin launching as SMs free up
  const int dh = blockIdx.x % a.nds;
  const int split = blockIdx.x / a.nds;
  const int rb = blockIdx.y;
  const int b = blockIdx.z;
  const int t0 = rb * a.G;
  const int gv = min(a.G, a.T - t0);
  const int nrows = gv * a.H;

  // ---------------------------------------------------------------- key range
  int64_t total = 0, u_lo = 0;
  SegTiles st;
  if (KIND == kFused) {
    // one query per row block (G = 1)
    int64_t nh = 0;
    if (a.segments & 2) {
      nh = vis(a.pos[(int64_t)b * a.T + t0], a.m);
      if (nh > a.N_h) nh = a.N_h;
    }
    st.init((a.segments & 1) ? a.k : 0, (a.segments & 2) ? nh : 0, (a.segments & 4) ? a.W : 0,
            split, a.nsplit);
  } else if (KIND == kSparse) {
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
  const int nt = KIND == kFused ? st.total() : (nk + kTile - 1) / kTile;
  const int ocols = n_own * 64;
  // tile i: segment (the kind's own, or the fused list's), first key and keys
  auto tile_of = [&](int i, int& seg, int64_t& kt, int& nvalid) {
    if (KIND == kFused) {
      st.map(i, seg, kt, nvalid);
    } else {
      seg = KIND == kSparse ? 0 : (KIND == kHca ? 1 : 2);
      kt = kbeg + static_cast<int64_t>(i) * kTile;
      nvalid = static_cast<int>((kend - kt) < kTile ? (kend - kt) : kTile);
    }
  };

  if (nt == 0) {
    pdl_wait();
    // empty split: o = 0, lse = -inf (a finalised output: 0, and the
    // sink alone in lse_out)
    for (int rI = threadIdx.x; rI < nrows; rI += kThreads) {
      const int g = rI / a.H, h = rI % a.H;
      const int64_t row = ((int64_t)b * a.T + t0 + g) * a.H + h;
      if (a.out) {
        for (int c = 0; c < ocols; ++c) a.out[row * a.D + dh * ocols + c] = __float2bfloat16(0.f);
        if (dh == 0 && a.lse_out) a.lse_out[row] = a.sink ? a.sink[h] : -INFINITY;
      } else if (a.nsplit == 1 && !a.partials) {
        for (int c = 0; c < ocols; ++c) a.o[row * a.D + dh * ocols + c] = 0.f;
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
    for (int i = 0; i < kNSB; ++i) {
      mbar_init(smem_u32(&sm->s_full[i]), 1);
      mbar_init(smem_u32(&sm->s_free[i]), 1);
    }
    mbar_init(smem_u32(&sm->drain[0]), 1);
    mbar_init(smem_u32(&sm->drain[1]), 1);
    for (int i = 0; i < kNSB; ++i) mbar_init(smem_u32(&sm->p_full[i]), 128);
    mbar_init(smem_u32(&sm->o_full), 1);
    mbar_init(smem_u32(&sm->q_full), 1);
    mbar_init(smem_u32(&sm->q_tmem), 128);
    mbar_init(smem_u32(&sm->q_ready), 1);
    sm->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_q);
    // (the fused call's maps exist only for the segments it covers)
    if (KIND == kHca || KIND == kSwa || (KIND == kFused && (a.segments & 2)))
      tma_prefetch_desc(&tm_kv);
    if (KIND == kFused && (a.segments & 4)) tma_prefetch_desc(&tm_kv2);
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(&sm->tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // a dependent launch has overlapped the setup above with its predecessor;
  // everything below may read what the predecessor wrote
  pdl_wait();
  const uint32_t tmem = sm->tmem_base;
  volatile int* abort = &sm->abort;
  const uint32_t tS = tmem;                  // columns [0, 64 kNSB): the S/P buffers
  const uint32_t tO = tmem + 64 * kNSB;      // ocols columns
  const uint32_t tQ = tO + ocols;            // n_tq chunks of the other half of Q, 32 columns each

  // The ring holds groups of gsz = n_own consecutive 8 KB chunk slots.  A
  // tile is the group of the other half's d chunks (nds = 2: keys only, free
  // once QK has read them), then the group of this CTA's own chunks (keys
  // and values: PV reads the group as one operand).  A streamed group is one
  // 3-D TMA copy {64 dims, 64 keys, gsz chunks}.
  const int gsz = n_own;
  const int ng = nslot / gsz;   // groups in the ring
  const int ngt = ndc / gsz;    // groups per tile: 1 or 2
  // the tensor-memory chunks of Q are staged in the last groups of the ring
  // until they have been copied into tensor memory
  const int64_t stage_group = n_tq > 0 ? (nslot - 2 * n_tq) / gsz : -1;
  // first d chunk of group q of a tile
  auto group_dc = [&](int q) -> int {
    if (q < ngt - 1) return (dh == 0 ? 1 : 0) * n_own;  // the other half
    return dh * n_own;
  };

  if (warp < 4) {
    // ============================================================ producers
    const int pt = threadIdx.x;  // 0..127
    int64_t gc = 0;              // groups requested so far
    int gs = 0;
    uint32_t ph = 0;             // ring position (group slot, phase) of gc
    auto advance = [&]() {
      ++gc;
      if (++gs == ng) { gs = 0; ph ^= 1u; }
    };
    // the group slot of gc may be refilled: its last reader is done, and the
    // staging groups of Q have been copied into tensor memory
    auto group_free = [&](int site) -> bool {
      if (gc == stage_group &&
          !mbar_wait(smem_u32(&sm->q_tmem), 0, abort, a.status, kWaitLimitNs, 33))
        return false;
      return gc < ng ||
             mbar_wait(smem_u32(&sm->empty[gs]), ph ^ 1u, abort, a.status, kWaitLimitNs, site);
    };
    // copies issued whose completion nobody waited for land before exit
    auto drain = [&](const uint64_t* bars, int64_t issued) {
      const int64_t first = issued > ng ? issued - ng : 0;
      for (int64_t x = first; x < issued; ++x)
        mbar_wait(smem_u32(&bars[x % ng]), (x / ng) & 1, nullptr, nullptr, 10000000ull, 19);
    };
    const uint32_t gbytes = static_cast<uint32_t>(gsz) * 8192u;
    if (KIND == kHca) {
      if (pt == 0) {
        bool ok = true;
        for (int i = 0; i < nt && ok && !*abort; ++i) {
          const int32_t row0 =
              static_cast<int32_t>((int64_t)b * a.N_rows + kbeg + (int64_t)i * kTile);
          for (int q = 0; q < ngt; ++q, advance()) {
            if (!(ok = group_free(18))) break;
            const uint32_t fb = smem_u32(&sm->full[gs]);
            mbar_arrive_expect_tx(fb, gbytes);
            tma_load_3d(smem_u32(sRing + gs * gbytes), &tm_kv, 0, row0, group_dc(q), fb);
          }
        }
        if (!ok || *abort) drain(sm->full, gc);
      }
    } else if (KIND == kSparse || KIND == kFused) {
      // Gathered tiles: 512 16-byte pieces per chunk, this thread copies
      // pieces pt + 128 j of every chunk of the group; its arrival on the
      // group's barrier fires when its copies have landed, so it never waits
      // for them itself.  Streamed tiles (fused): thread 0 arms the barrier
      // and issues the copy, the others just arrive (128 arrivals either way).
      const int32_t* idx_row = a.idx + ((int64_t)b * a.T + t0) * a.k;
      bool ok = true;
      int64_t tma_issued = 0;  // groups up to the last one thread 0 copied by TMA
      for (int i = 0; i < nt && ok && !*abort; ++i) {
        int seg, nvalid;
        int64_t kt;
        tile_of(i, seg, kt, nvalid);
        const __nv_bfloat16* src[4];
        int bytes[4];
        if (seg == 0) {
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const int rI = (pt + 128 * j4) >> 3;
            int32_t j = -1;
            if (rI < nvalid) j = idx_row[kt + rI];
            if (j >= a.N_rows) {
              if ((pt & 7) == 0) record_status(a.status, kStatusBadIndex);
              j = -1;
            }
            bytes[j4] = j >= 0 ? 16 : 0;
            src[j4] = a.kv + ((int64_t)b * a.N_rows + (j >= 0 ? j : 0)) * a.D +
                      ((pt + 128 * j4) & 7) * 8;
          }
        }
        int32_t row0 = 0;
        if (KIND == kFused && seg != 0)
          row0 = seg == 1 ? static_cast<int32_t>((int64_t)b * a.N_h + kt)
                          : static_cast<int32_t>(((int64_t)b * a.T + t0) * a.W + kt);
        for (int q = 0; q < ngt; ++q, advance()) {
          if (!(ok = group_free(20))) break;
          const uint32_t dst = smem_u32(sRing + gs * gbytes);
          const uint32_t fb = smem_u32(&sm->full[gs]);
          if (seg == 0) {
            const int dc0 = group_dc(q);
            for (int e = 0; e < gsz; ++e) {
              const int dcol = (dc0 + e) * 64;
#pragma unroll
              for (int j4 = 0; j4 < 4; ++j4) {
                const int pc = pt + 128 * j4;
                cp_async16(dst + e * 8192 + swz128(pc >> 3, pc & 7), src[j4] + dcol, bytes[j4]);
              }
            }
            cp_async_mbar_arrive(fb);
          } else if (pt == 0) {
            mbar_arrive_expect_tx(fb, gbytes);
            tma_load_3d(dst, seg == 1 ? &tm_kv : &tm_kv2, 0, row0, group_dc(q), fb);
            tma_issued = gc + 1;
          } else {
            mbar_arrive(fb);
          }
        }
      }
      cp_async_wait_all();  // no copy outlives the CTA
      if ((!ok || *abort) && pt == 0 && tma_issued > 0) drain(sm->full, tma_issued);
    } else {
      // SWA: keys are RMSNorm'd and RoPE'd raw tokens at their own positions.
      // Row norms come first, from the rows in global memory (two threads per
      // row, eight 16-byte loads in flight each); then the tile's groups are
      // requested by TMA, and each is normalised in place as it lands.
      const int nr = pt >> 1, hf = pt & 1;
      const int half_pieces = a.D / 16;  // 16-byte pieces per half row
      bool ok = true;
      int64_t issued = 0;  // groups thread 0 has requested
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
        if (pt == 0) {
          // request the tile's groups (thread 0 walks ahead of the others'
          // ring position by up to one tile)
          int64_t c = gc;
          int s = gs;
          uint32_t phs = ph;
          for (int q = 0; q < ngt && ok; ++q) {
            ok = (c != stage_group ||
                  mbar_wait(smem_u32(&sm->q_tmem), 0, abort, a.status, kWaitLimitNs, 33)) &&
                 (c < ng ||
                  mbar_wait(smem_u32(&sm->empty[s]), phs ^ 1u, abort, a.status, kWaitLimitNs, 21));
            if (ok) {
              const uint32_t rbar = smem_u32(&sm->raw[s]);
              mbar_arrive_expect_tx(rbar, gbytes);
              tma_load_3d(smem_u32(sRing + s * gbytes), &tm_kv, 0,
                          static_cast<int32_t>((int64_t)b * a.N_rows + u_lo + kt), group_dc(q),
                          rbar);
              issued = c + 1;
            }
            ++c;
            if (++s == ng) { s = 0; phs ^= 1u; }
          }
        }
        for (int q = 0; q < ngt; ++q, advance()) {
          if (ok) ok = mbar_wait(smem_u32(&sm->raw[gs]), ph, abort, a.status, kWaitLimitNs, 26);
          if (!ok) continue;  // nothing more to wait for; the next barrier ends the loop
          const int dc0 = group_dc(q);
          for (int e = 0; e < gsz; ++e) {
            const int dcol = (dc0 + e) * 64;
            uint8_t* dst = sRing + gs * gbytes + e * 8192;
#pragma unroll
            for (int j4 = 0; j4 < 4; ++j4) {
              const int pc = pt + 128 * j4;
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
                rope8(y, dcol + piece * 8, a.D, a.r, u_lo + kt + rI, a.rope.c);
              } else {
#pragma unroll
                for (int z = 0; z < 8; ++z) y[z] = 0.f;
              }
              *cell = kF16 ? pack8_f16(y) : pack8(y);
            }
          }
          fence_proxy_async_smem();
          mbar_arrive(smem_u32(&sm->full[gs]));
        }
      }
      if (!ok && pt == 0) drain(sm->raw, issued);
    }
  } else if (warp == 4 || warp == 9) {
    // ============================================================ QK issuers
    // warp 4 loads Q and issues QK for even tiles, warp 9 for odd tiles
    const int par = warp == 4 ? 0 : 1;
    bool ok = true;
    if (warp == 4) {
      if (lane == 0) {
        const uint32_t qb = smem_u32(&sm->q_full);
        mbar_arrive_expect_tx(qb, static_cast<uint32_t>(ndc) * 16384u);
        const int32_t qrow0 = static_cast<int32_t>(((int64_t)b * a.T + t0) * a.H);
        for (int dc = 0; dc < ndc; ++dc) {
          const int e = dc - dh * n_own;  // own chunk index, or outside [0, n_own)
          const int oc = dc - (dh == 0 ? n_own : 0);  // else: chunk of the other half
          uint8_t* dst = (e >= 0 && e < n_own) ? sQ + e * 16384
                         : (oc < n_tq ? sQstage + oc * 16384 : sQ + (n_own + oc - n_tq) * 16384);
          tma_load_2d(smem_u32(dst), &tm_q, dc * 64, qrow0, qb);
        }
      }
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm->q_full), 0, abort, a.status,
                                             kWaitLimitNs, 29));
      // on an abort the query copies issued above land before the CTA exits
      if (!ok && lane == 0)
        mbar_wait(smem_u32(&sm->q_full), 0, nullptr, nullptr, 10000000ull, 42);
      // the query rows of other queries (or past the tensor) in the box are
      // zeroed, so they contribute nothing to S
      if (ok && nrows < 128) {
        for (int e = 0; e < n_sq; ++e)
          for (int pc = nrows * 8 + lane; pc < 128 * 8; pc += 32)
            *reinterpret_cast<uint4*>(sQ + e * 16384 + swz128(pc >> 3, pc & 7)) =
                make_uint4(0, 0, 0, 0);
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (ok && (n_tq > 0 || kF16))
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm->q_tmem), 0, abort, a.status,
                                               kWaitLimitNs, 34));
      if (lane == 0) mbar_arrive(smem_u32(&sm->q_ready));  // also on failure: abort is set
    } else {
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm->q_ready), 0, abort, a.status,
                                             kWaitLimitNs, 36));
    }
    ok = ok && !*abort;
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    const uint32_t idesc_qk = kF16 ? idesc_f16(128, 64, 0, 0) : idesc_bf16(128, 64, 0, 0);
    const uint32_t sQa = smem_u32(sQ), sRa = smem_u32(sRing);
    for (int i = par; i < nt && ok; i += 2) {
      int seg, nvalid;
      int64_t kt;
      tile_of(i, seg, kt, nvalid);
      const int sb = i % kNSB;
      // the S/P buffer is reused once PV of tile i - kNSB has read its P.
      // (Buffers alternate between the two issuers, but each wait is still
      // exact: this issuer's previous tile, i - 2, waited for PV(i - 2 - kNSB),
      // so the phase before the one waited for here has completed.)
      if (i >= kNSB) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm->s_free[sb]), ((i / kNSB) - 1) & 1,
                                               abort, a.status, kWaitLimitNs, 37));
        if (!ok) break;
        tc_fence_after();
      }
      // S(i) = Q K(i)^T over all ndc chunks, group by group; the other
      // half's group holds only keys and is released once this product has
      // read it
      for (int q = 0; q < ngt && ok; ++q) {
        const int64_t g = (int64_t)i * ngt + q;
        const int gsl = static_cast<int>(g % ng);
        const bool got = mbar_wait(smem_u32(&sm->full[gsl]), static_cast<uint32_t>((g / ng) & 1),
                                   abort, a.status, kWaitLimitNs, 22);
        ok = __all_sync(0xffffffffu, got);  // warp-uniform
        if (!ok) break;
        // gathered rows were written by cp.async (generic proxy); the MMA
        // reads through the async proxy.  (The invalid key rows of a streamed
        // tail tile may hold anything: their S columns are masked, and the
        // PV issuer zeroes them as values.)
        if (KIND == kSparse || KIND == kFused) fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          for (int e = 0; e < gsz; ++e) {
            const int p = q * gsz + e;  // chunk of the tile: the other half first
            const uint32_t slot_a = sRa + static_cast<uint32_t>(gsl * gsz + e) * 8192u;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t bd = smem_desc(slot_a + ks * 32, 16, 1024, kSwizzle128B);
              const uint32_t acc = (p == 0 && ks == 0) ? 0u : 1u;
              if (p < n_tq) {
                mma_bf16_ts(tS + sb * 64, tQ + p * 32 + ks * 8, bd, idesc_qk, acc);
              } else {
                // the other half's shared-memory chunks follow the own ones
                const int qc = p < n_other ? n_own + p - n_tq : p - n_other;
                const uint64_t ad =
                    smem_desc(sQa + qc * 16384 + ks * 32, 16, 1024, kSwizzle128B);
                mma_bf16_ss(tS + sb * 64, ad, bd, idesc_qk, acc);
              }
            }
          }
          if (q < ngt - 1) mma_commit(smem_u32(&sm->empty[gsl]));
        }
        __syncwarp();
      }
      if (!ok) break;
      if (lane == 0) mma_commit(smem_u32(&sm->s_full[sb]));
      __syncwarp();
    }
    // this thread's MMAs complete before the tensor memory is released
    if (lane == 0) {
      mma_commit(smem_u32(&sm->drain[par]));
      mbar_wait(smem_u32(&sm->drain[par]), 0, nullptr, nullptr, 10000000ull, 24);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ============================================================ PV issuer
    // O += P(i) V(i): P from tensor memory (S/P buffer i & 1), V = the n_own
    // chunks of tile i, consecutive ring slots (the ring holds a whole number
    // of such groups), read as one MN-major operand of N = ocols
    const uint32_t idesc_pv = kF16 ? idesc_f16(128, ocols, 0, 1) : idesc_bf16(128, ocols, 0, 1);
    const uint32_t sRa = smem_u32(sRing);
    bool ok = true;
    for (int i = 0; i < nt && ok; ++i) {
      // one barrier per S/P buffer: the softmax of tile i + kNSB needs
      // S(i + kNSB), whose QK waited for PV(i), so no phase is skipped
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm->p_full[i % kNSB]), (i / kNSB) & 1,
                                             abort, a.status,
                                             kWaitLimitNs, 23));
      if (!ok) break;
      const int64_t g = (int64_t)i * ngt + (ngt - 1);  // the tile's own group
      const int gsl = static_cast<int>(g % ng);
      int seg, nvalid;
      int64_t kt;
      tile_of(i, seg, kt, nvalid);
      // a streamed tail tile: its invalid key rows may hold anything (even
      // NaN, and P = 0 times NaN is NaN), so this warp zeroes them as values
      // before its product reads the group
      const bool zero_tail = (KIND == kHca || (KIND == kFused && seg != 0)) && nvalid < kTile;
      if (KIND == kSparse || KIND == kFused || zero_tail) {
        // this warp's view of the copied rows (the copy landed before QK(i)
        // read them), for the zeroing and for the async proxy
        ok = __all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&sm->full[gsl]), static_cast<uint32_t>((g / ng) & 1),
                                  abort, a.status, kWaitLimitNs, 38));
        if (!ok) break;
        if (zero_tail) {
          uint8_t* dst = sRing + gsl * gsz * 8192;
          for (int pc = nvalid * 8 + lane; pc < kTile * 8; pc += 32)
            for (int e = 0; e < gsz; ++e)
              *reinterpret_cast<uint4*>(dst + e * 8192 + swz128(pc >> 3, pc & 7)) =
                  make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      if (lane == 0) {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bd =
              smem_desc(sRa + static_cast<uint32_t>(gsl * gsz) * 8192u + ks * 2048, 8192, 1024,
                        kSwizzle128B);
          mma_bf16_ts(tO, tS + (i % kNSB) * 64 + ks * 8, bd, idesc_pv,
                      (i > 0 || ks > 0) ? 1u : 0u);
        }
        mma_commit(smem_u32(&sm->empty[gsl]));
        mma_commit(smem_u32(&sm->s_free[i % kNSB]));
      }
      __syncwarp();
    }
    if (lane == 0) mma_commit(smem_u32(&sm->o_full));
    __syncwarp();
    if (!ok) {
      // wait (bounded) for the MMAs already issued before the memory is released
      mbar_wait(smem_u32(&sm->o_full), 0, nullptr, nullptr, 10000000ull, 39);
    }
  } else {
    // ============================================================ softmax
    const int quad = warp & 3;             // tensor-memory lane quarter of this warp
    const int rI = quad * 32 + lane;
    const bool row_valid = rI < nrows;
    const int g = row_valid ? rI / a.H : 0;
    const int h = row_valid ? rI % a.H : 0;
    const int32_t tq = row_valid ? a.pos[(int64_t)b * a.T + t0 + g] : 0;
    const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
    bool ok = true;
    if (n_tq > 0 || kF16) {
      // the other half of this row's q~ into tensor memory (zeros for rows
      // that are not this block's); with fp16 products, this row of the own
      // half is converted in shared memory too (the QK issuer zeroes the
      // rows past the block's, these threads convert the others)
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&sm->q_full), 0, abort, a.status,
                                             kWaitLimitNs, 35));
      if (kF16 && row_valid && ok) {
        for (int e = 0; e < n_sq; ++e)
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            uint4* cell = reinterpret_cast<uint4*>(sQ + e * 16384 + swz128(rI, q));
            *cell = bf16x8_to_f16x8(*cell);
          }
        fence_proxy_async_smem();  // the tensor core reads these rows
      }
      for (int e = 0; e < n_tq; ++e) {
        float w[32];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 u = make_uint4(0, 0, 0, 0);
          if (row_valid && ok)
            u = *reinterpret_cast<const uint4*>(sQstage + e * 16384 + swz128(rI, q));
          if (kF16) u = bf16x8_to_f16x8(u);
          w[4 * q] = __uint_as_float(u.x);
          w[4 * q + 1] = __uint_as_float(u.y);
          w[4 * q + 2] = __uint_as_float(u.z);
          w[4 * q + 3] = __uint_as_float(u.w);
        }
        tmem_st32(tQ + lane_base + e * 32, w);
      }
      if (n_tq > 0) tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->q_tmem));
    }
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
    const float sl2 = a.scale * 1.4426950408889634f;  // logits in base 2
    const int32_t* idx_row = a.idx + ((int64_t)b * a.T + t0) * a.k;
    float m_used = -INFINITY, l = 0.f;
    for (int i = 0; i < nt && ok; ++i) {
      int seg, nv;
      int64_t kt;
      tile_of(i, seg, kt, nv);
      uint64_t colmask = 0;  // keys of this tile that exist for every row
      if (seg == 0) {
        const int64_t k0 = kt + lane, k1 = kt + 32 + lane;
        const int32_t j0 = lane < nv ? idx_row[k0] : -1;
        const int32_t j1 = 32 + lane < nv ? idx_row[k1] : -1;
        const unsigned b0 = __ballot_sync(0xffffffffu, j0 >= 0 && j0 < a.N_rows);
        const unsigned b1 = __ballot_sync(0xffffffffu, j1 >= 0 && j1 < a.N_rows);
        colmask = static_cast<uint64_t>(b0) | (static_cast<uint64_t>(b1) << 32);
      } else {
        colmask = nv >= 64 ? ~0ull : ((1ull << nv) - 1);
      }
      // the row's own limits as tile columns: valid c in [c_lo, c_hi)
      int c_lo = 0, c_hi = row_valid ? 64 : 0;
      if (KIND == kHca) {
        const int64_t hi = row_hi - kt;
        c_hi = row_valid ? static_cast<int>(hi < 0 ? 0 : (hi > 64 ? 64 : hi)) : 0;
      } else if (KIND == kSwa) {
        const int64_t lo = row_lo - (u_lo + kt), hi = row_hi + 1 - (u_lo + kt);
        c_lo = static_cast<int>(lo < 0 ? 0 : (lo > 64 ? 64 : lo));
        c_hi = row_valid ? static_cast<int>(hi < 0 ? 0 : (hi > 64 ? 64 : hi)) : 0;
      } else if (KIND == kFused && seg == 2) {
        // window key j is the raw token tq - W + 1 + j; tokens before 0 do not exist
        const int64_t lo = (int64_t)a.W - 1 - tq - kt;
        c_lo = static_cast<int>(lo < 0 ? 0 : (lo > 64 ? 64 : lo));
      }
      const bool full_tile =
          __all_sync(0xffffffffu, colmask == ~0ull && c_lo == 0 && c_hi == 64);
      const int sb = i % kNSB;
      bool got = mbar_wait(smem_u32(&sm->s_full[sb]), (i / kNSB) & 1, abort, a.status,
                           kWaitLimitNs, 25);
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }  // warp-uniform exit
      tc_fence_after();
      float s[64];
      tmem_ld32(tS + lane_base + sb * 64, *reinterpret_cast<float(*)[32]>(s));
      tmem_ld32(tS + lane_base + sb * 64 + 32, *reinterpret_cast<float(*)[32]>(s + 32));
      tmem_wait_ld();
      if (!full_tile) {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const bool v = ((colmask >> c) & 1ull) && c >= c_lo && c < c_hi;
          s[c] = v ? s[c] : -INFINITY;
        }
      }
      // row max of the raw logits, as a tree
      float t8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float m0 = fmaxf(fmaxf(s[j], s[j + 8]), fmaxf(s[j + 16], s[j + 24]));
        const float m1 = fmaxf(fmaxf(s[j + 32], s[j + 40]), fmaxf(s[j + 48], s[j + 56]));
        t8[j] = fmaxf(m0, m1);
      }
      const float mraw = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])),
                               fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
      const float mx = mraw * sl2;  // sl2 > 0: the max of the scaled logits
      // Lazy rescale: only when the running max grows by more than 2^8.  The
      // tensor-memory loads/stores are warp-collective, so the decision is
      // taken per warp; lanes that need no rescale multiply by 1.  O is
      // touched only then, after PV(i-1) has finished writing it.
      const bool grow = mx > m_used + 8.f;
      const bool need_rescale = grow && m_used != -INFINITY && i > 0;
      if (__any_sync(0xffffffffu, need_rescale)) {
        // PV(i-1) has completed once it frees its S buffer; the phase before
        // (PV(i-1-kNSB)) completed before QK(i-1) was issued, and PV(i)
        // needs this thread's P, so the parity names PV(i-1) alone
        got = mbar_wait(smem_u32(&sm->s_free[(i - 1) % kNSB]), ((i - 1) / kNSB) & 1, abort,
                        a.status, kWaitLimitNs, 32);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        const float f = need_rescale ? ex2_fast(m_used - mx) : 1.f;
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
      // P = 2^(s * sl2 - m) rounded to bf16, two per 32-bit column, into the
      // first 32 columns of this S buffer (the PV product reads it there); l
      // sums the rounded values, so the normalisation matches what the
      // tensor cores multiply.  A row with no key so far has m = -inf: its
      // logits are all -inf and so are its P (2^-inf = 0).
      const float moff = (m_used == -INFINITY) ? 0.f : -m_used;
      float pk[32];
      float l4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < 64; c += 2) {
        const float p0 = ex2_fast(fmaf(s[c], sl2, moff));
        const float p1 = ex2_fast(fmaf(s[c + 1], sl2, moff));
        if (kF16) {
          const uint32_t u = pack_f16x2(p0, p1);
          const float2 f = unpack_f16x2(u);
          l4[(c >> 1) & 3] += f.x + f.y;
          pk[c >> 1] = __uint_as_float(u);
        } else {
          const uint32_t u = pack_bf16x2(p0, p1);
          l4[(c >> 1) & 3] += __uint_as_float(u << 16) + __uint_as_float(u & 0xffff0000u);
          pk[c >> 1] = __uint_as_float(u);
        }
      }
      l += (l4[0] + l4[1]) + (l4[2] + l4[3]);
      tmem_st32(tS + lane_base + sb * 64, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->p_full[sb]));
    }
    // ------------------------------------------------------------ epilogue
    // O rows go through shared memory (the Q area and the ring, free once
    // every MMA has completed) so that each store instruction writes one
    // contiguous row.
    bool done = ok && mbar_wait(smem_u32(&sm->o_full), 0, abort, a.status, kWaitLimitNs, 40);
    done = __all_sync(0xffffffffu, done);
    if (done) {
      tc_fence_after();
      // Finalised output (a.out): the sink-augmented merge of this single
      // split, Z = sum_j e^l_j + e^sink, y = sum_j e^l_j v_j / Z, taken in
      // base 2 around the larger of the two terms; else the split's own
      // normalisation and log-sum-exp.
      const bool fin = a.out != nullptr;
      float inv_l, lse;
      if (fin) {
        const float s2 = a.sink ? __ldg(a.sink + h) * 1.4426950408889634f : -INFINITY;
        const float lb = l > 0.f ? m_used + log2f(l) : -INFINITY;  // log2 sum_j 2^(l_j log2 e)
        const float mx = fmaxf(lb, s2);
        if (mx == -INFINITY) {
          inv_l = 0.f;
          lse = -INFINITY;
        } else {
          const float lz = mx + log2f(exp2f(lb - mx) + exp2f(s2 - mx));
          inv_l = l > 0.f ? exp2f(m_used - lz) : 0.f;  // 2^m / Z: o is the unnormalised sum
          lse = lz * 0.6931471805599453f;
        }
      } else {
        inv_l = l > 0.f ? 1.f / l : 0.f;
        lse = l > 0.f ? (m_used + log2f(l)) * 0.6931471805599453f : -INFINITY;
      }
      // this warp's 32 rows, fp32, row stride ocols + 4 floats (bank spread)
      float* stage = reinterpret_cast<float*>(sQ) + quad * 32 * (ocols + 4);
      for (int cc = 0; cc < ocols; cc += 32) {
        float o[32];
        tmem_ld32(tO + lane_base + cc, o);
        tmem_wait_ld();
        float* dstrow = stage + lane * (ocols + 4) + cc;
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(dstrow + e) =
              make_float4(o[e] * inv_l, o[e + 1] * inv_l, o[e + 2] * inv_l, o[e + 3] * inv_l);
      }
      if (fin && row_valid) {
        // the last r dims rotated back by the query position, then the row
        // as bf16 over the start of its own staging row (each 4-byte pair
        // is read before the 2 bytes written at or below it)
        float* srow = stage + lane * (ocols + 4);
        const int d0 = a.D - a.r;
        for (int c = 0; c < ocols; c += 2) {
          const int d = dh * ocols + c;
          float x0 = srow[c], x1 = srow[c + 1];
          if (d >= d0) {
            float sn, cs;
            rope_cs(a.rope.c, (d - d0) >> 1, -static_cast<int64_t>(tq), &sn, &cs);
            const float y0 = x0 * cs - x1 * sn;
            x1 = x0 * sn + x1 * cs;
            x0 = y0;
          }
          reinterpret_cast<uint32_t*>(srow)[c >> 1] = pack_bf16x2(x0, x1);
        }
      }
      // the staged row of this thread goes out as one bulk copy by the copy
      // engine (all 128 rows stream in parallel)
      const bool direct = a.nsplit == 1 && !a.partials;
      fence_proxy_async_smem();
      if (fin && row_valid) {
        const int64_t row = ((int64_t)b * a.T + t0 + g) * a.H + h;
        bulk_copy_s2g(a.out + row * a.D + dh * ocols, smem_u32(stage + lane * (ocols + 4)),
                      static_cast<uint32_t>(ocols) * 2u);
        bulk_commit();
        if (dh == 0 && a.lse_out) a.lse_out[row] = lse;
        bulk_wait_read();
      } else if (row_valid) {
        const int64_t row = ((int64_t)b * a.T + t0 + g) * a.H + h;
        float* dst = direct ? a.o + row * a.D + dh * ocols
                            : a.part_o + (row * a.nsplit + split) * a.D + dh * ocols;
        bulk_copy_s2g(dst, smem_u32(stage + lane * (ocols + 4)),
                      static_cast<uint32_t>(ocols) * 4u);
        bulk_commit();
        if (dh == 0) {
          if (direct) a.lse[row] = lse;
          else a.part_lse[row * a.nsplit + split] = lse;
        }
        bulk_wait_read();
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
  const int G = (kind == kSparse || kind == kFused) ? 1 : (128 / H);
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
  if (nsplit > kMaxMergeParts) {  // the merges weigh at most this many partials per row
    tps = (tiles + kMaxMergeParts - 1) / kMaxMergeParts;
    nsplit = (tiles + tps - 1) / tps;
  }
  if (nsplit * nds > 65535 || n_rb > 65535) return false;
  const int ndc = D / 64;
  if (ndc % nds) return false;  // the halves of the output are whole chunks
  const int n_own = ndc / nds;
  const int n_other = ndc - n_own;
  // tensor memory: the S/P buffers, O (own columns), then as many chunks of
  // the other half of Q as fit (32 columns each); the rest of Q stays in
  // shared memory
  const int tq_fit = (512 - kNSB * 64 - n_own * 64) / 32;
  if (tq_fit < 0) return false;
  const int n_tq = n_other < tq_fit ? n_other : tq_fit;
  const int n_sq = ndc - n_tq;
  p->G = G;
  p->n_rb = n_rb;
  p->nds = nds;
  p->n_tq = n_tq;
  p->nsplit = static_cast<int>(nsplit);
  p->keys_per_split = static_cast<int>(tps * kTile);
  const size_t fixed = 1024 + (size_t)n_sq * 16384 + sizeof(AttnShared);
  int nslot = static_cast<int>((227 * 1024 - fixed) / 8192);
  if (nslot > kMaxSlots) nslot = kMaxSlots;
  // the own chunks of a tile are consecutive slots: a tile's own group
  // starts at a multiple of n_own and the ring holds whole groups
  nslot -= nslot % n_own;
  // QK of the next tile (all ndc chunks) is issued before PV of the current
  // one (our n_own chunks): both must fit the ring at once, and the staging
  // of the tensor-memory chunks of Q (two slots per chunk) fits at its end
  if (nslot < ndc + n_own || nslot < 2 * n_tq) return false;
  // epilogue staging of 128 rows x (own columns + 4) fp32 over the Q area
  // and the ring, both free once every MMA has completed
  if ((size_t)128 * (n_own * 64 + 4) * 4 > (size_t)n_sq * 16384 + (size_t)nslot * 8192)
    return false;
  p->nslot = nslot;
  p->smem_bytes = fixed + (size_t)nslot * 8192;
  p->ws_bytes = p->nsplit > 1 ? (size_t)B * T * H * p->nsplit * (D + 1) * sizeof(float) : 0;
  return true;
}

template <int KIND>
cudaError_t launch_kind(const CUtensorMap& tm_kv, const CUtensorMap& tm_kv2,
                        const CUtensorMap& tm_q, const AttnArgs& a, const AttnPlan& p,
                        cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<KIND>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(p.smem_bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nds * p.nsplit, p.n_rb, a.B);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  cfg.attrs = at;
  cfg.numAttrs = add_dependent_attr(at, 0, a.dependent != 0);
  e = cudaLaunchKernelEx(&cfg, attn_kernel<KIND>, tm_kv, tm_kv2, tm_q, a, p.nslot);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_attention(const CUtensorMap& tm_kv, const CUtensorMap& tm_kv2,
                             const CUtensorMap& tm_q, const AttnArgs& a, const AttnPlan& p,
                             cudaStream_t stream) {
  switch (a.kind) {
    case kSparse:
      return launch_kind<kSparse>(tm_kv, tm_kv2, tm_q, a, p, stream);
    case kHca:
      return launch_kind<kHca>(tm_kv, tm_kv2, tm_q, a, p, stream);
    case kSwa:
      return launch_kind<kSwa>(tm_kv, tm_kv2, tm_q, a, p, stream);
    default:
      return launch_kind<kFused>(tm_kv, tm_kv2, tm_q, a, p, stream);
  }
}

}  // namespace hattn
