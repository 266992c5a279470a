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
// over a grid of one CTA per SM.  Roles: two producer threads (warp 0 and
// the last warp) issue the TMA loads of the key blocks of even and odd slots
// into a ring of `stages` buffers (and warp 0 the group's queries); warps 1
// and 2 issue the MMAs (M=128, N=NQ) of alternate slots into a ring of
// `nacc` tensor-memory accumulators; three groups of four warps (two when
// nacc is not a multiple of 3) drain the accumulators in turn (tcgen05.ld),
// reduce them and write fp32 scores with coalesced stores.  HBM traffic is
// the key blocks once plus the scores.
//
// FP8 keys ("DeepSeek-V4" atlas spec sheet, "Inference efficiency": the
// indexer QK path runs in low precision): each key is 128 E4M3 codes (one
// 128-byte swizzle row) with an fp32 row scale s_j.  The epilogue warps
// quantise the group's bf16 query rows the same way in shared memory
// (codes plus a scale s_h per row), the MMAs run kind::f8f6f4 (K = 32 per
// call, 4 calls per block), and since both scales are positive,
//     I(t, j) = s_j * sum_h (w[t,h] * s_h) * max(0, q8_h . k8_j),
// so the scales cost one multiply per column weight and one per score.
// A key costs 128 + 4 bytes instead of 256.
//
// MXFP4 keys (the same spec sheet names MXFP4 for that path): 64 bytes of
// E2M1 codes and 4 E8M0 block scales per key.  The epilogue warps quantise
// the query rows to E2M1 codes and block scales; the MMAs run
// kind::mxf4 with block scaling (K = 64 per call, 2 calls per block), the
// scales of both operands copied into tensor memory, so the product is the
// score's dot product over the decoded values.  A key costs 68 bytes.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

// warps: 0 producer (even slots), 1 and 2 MMA issuers (even / odd slots),
// then kEpiGroups x 4 epilogue warps (any 4 consecutive warps cover the four
// 32-lane quarters of tensor memory), then the producer of the odd slots
constexpr int kEpiGroups = 3;
constexpr int kEpiWarps = 4 * kEpiGroups;
constexpr int kFirstEpiWarp = 3;
constexpr int kProducer2 = kFirstEpiWarp + kEpiWarps;  // the second producer, last warp
constexpr int kIdxThreads = 32 * (kProducer2 + 1);
constexpr int kBlockRows = 128;
constexpr int kMaxStages = 12;
constexpr int kMaxStagesBf16 = 8;
constexpr int kMaxAcc = 8;  // accumulators in flight (TMEM columns permitting)
// key formats of the score kernel
constexpr int kKeyBf16 = kIdxKeysBf16, kKeyE4m3 = kIdxKeysE4m3, kKeyMx4 = kIdxKeysMx4;
// MXFP4 keys (dI = 128): a block of 128 keys is 128 x 64 code bytes, then
// its 128 x 4 E8M0 scale bytes
constexpr uint32_t kMxStageBytes = 128 * 64 + 128 * 4;
constexpr int kHistWords = kSelBins / 2;  // a row's 16-bit bins, two per word

struct IdxSmem {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t sempty[kMaxStages];  // FP8: the epilogue has read the stage's key scales
  uint64_t tfull[kMaxAcc];
  uint64_t tempty[kMaxAcc];
  uint64_t qfull;
  uint64_t qempty;
  uint64_t q8full;  // FP8 keys: the group's query codes and scales are in place
  uint64_t mma_done[2];
  uint32_t tmem_base;
  int abort;
};

// The rest of the epilogue's shared state follows IdxSmem, sized by the
// plan: per epilogue warp (no cross-warp barrier) the head weight of every
// accumulator column and the visible entries of each query of the current
// group; the query row scales (FP8 keys); and, when the call folds the
// selection's first pass in, two 2,048-bin histograms of 16-bit counts
// (packed in pairs) for the first and second row of this CTA's slots.
struct EpiLayout {
  uint32_t wcol, qscale, nt, hist, bytes;
};
// The bytes before the bf16 query rows: E4M3 query rows (FP8 keys), or the
// E2M1 query rows and their 512-byte scale atom (MXFP4 keys), a multiple of
// 1024 so the bf16 rows keep their 128-byte swizzle atoms aligned.
__host__ __device__ __forceinline__ uint32_t indexer_q8_bytes(int kf, int NQ) {
  if (kf == kIdxKeysE4m3) return static_cast<uint32_t>(NQ) * 128u;
  if (kf == kIdxKeysMx4) return (static_cast<uint32_t>(NQ) * 64u + 512u + 1023u) / 1024u * 1024u;
  return 0u;
}

__host__ __device__ __forceinline__ EpiLayout epi_layout(int NQ, int G, bool hist) {
  EpiLayout l;
  uint32_t o = 0;
  l.wcol = o;
  o += kEpiWarps * NQ * 4;
  l.qscale = o;
  o += (NQ * 4 + 15) / 16 * 16;
  l.nt = o;
  o += (kEpiWarps * G * 4 + 15) / 16 * 16;
  l.hist = o;
  o += hist ? 2 * kHistWords * 4 : 0;
  l.bytes = o;
  return l;
}

// order-preserving key of a score (the selection ranks these)
__device__ __forceinline__ uint32_t score_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);  // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int64_t visible_entries(int32_t t, int m, int64_t cap) {
  int64_t n = t < 0 ? 0 : (static_cast<int64_t>(t) + 1) / m;
  return n < cap ? n : cap;
}

// Walks this CTA's live slots in order.  Every role runs the same cursor, so
// all of them visit the same blocks: the blocks of a group that hold an entry
// some query of the group sees (the later blocks of the group are dead).  A
// step is one 32-bit compare; the 64-bit divisions and the visibility reads
// happen only when the query group changes, which `fresh` flags.
struct SlotCursor {
  int64_t group;   // b * groups_per_seq + query group within the sequence
  int64_t last;    // the last group the CTA's slots reach
  int blk;         // 128-entry block within the sequence
  int blk_end;     // one past the group's last live block within the CTA's slots
  int last_end;    // one past the CTA's last block within group `last`
  int b, t0, gv;
  bool fresh;      // first live slot of its group
  bool done;

  __device__ __forceinline__ void load_group(const IndexerArgs& a) {
    b = static_cast<int>(group / a.groups_per_seq);
    t0 = static_cast<int>(group - static_cast<int64_t>(b) * a.groups_per_seq) * a.G;
    gv = min(a.G, a.T - t0);
    int64_t nmax = 0;  // largest visible-entry count among the group's queries
    for (int g = 0; g < gv; ++g) {
      const int64_t v = visible_entries(a.pos[(int64_t)b * a.T + t0 + g], a.m, a.N_cap);
      nmax = v > nmax ? v : nmax;
    }
    const int cap = group == last ? last_end : a.nblk;
    const int64_t live = (nmax + kBlockRows - 1) / kBlockRows;
    blk_end = live < cap ? static_cast<int>(live) : cap;
    fresh = true;
  }
  // the first live block of a later group, or done
  __device__ __forceinline__ void next_group(const IndexerArgs& a) {
    do {
      if (group >= last) {
        done = true;
        return;
      }
      ++group;
      blk = 0;
      load_group(a);
    } while (blk_end <= 0);
  }
  __device__ __forceinline__ void init(const IndexerArgs& a, int64_t s0, int64_t s1) {
    done = s0 >= s1;
    if (done) return;
    group = s0 / a.nblk;
    blk = static_cast<int>(s0 - group * a.nblk);
    last = (s1 - 1) / a.nblk;
    last_end = static_cast<int>(s1 - last * a.nblk);
    load_group(a);
    if (blk >= blk_end) next_group(a);
  }
  __device__ __forceinline__ void advance(const IndexerArgs& a) {
    fresh = false;
    if (++blk >= blk_end) next_group(a);
  }
};

// A role's walk over the CTA's live slots together with the rings they
// index: slot it uses stage it % stages (phase bit ph) and accumulator
// it % nacc (phase bit aph).
struct SlotWalk {
  SlotCursor cur;
  int64_t it;
  int st, acc;
  uint32_t ph, aph;
  __device__ __forceinline__ void init(const IndexerArgs& a, int64_t s0, int64_t s1) {
    cur.init(a, s0, s1);
    it = 0;
    st = acc = 0;
    ph = aph = 0;
  }
  // one slot on (the cursor may enter a new query group: cur.fresh)
  __device__ __forceinline__ void step(const IndexerArgs& a) {
    cur.advance(a);
    ++it;
    if (++st == a.stages) { st = 0; ph ^= 1u; }
    if (++acc == a.nacc) { acc = 0; aph ^= 1u; }
  }
  // n slots on by plain arithmetic when they stay in the current group
  // (n <= stages and n <= nacc: each ring wraps at most once); else false
  __device__ __forceinline__ bool leap(const IndexerArgs& a, int n) {
    if (cur.blk + n >= cur.blk_end) return false;
    cur.blk += n;
    it += n;
    st += n;
    if (st >= a.stages) { st -= a.stages; ph ^= 1u; }
    acc += n;
    if (acc >= a.nacc) { acc -= a.nacc; aph ^= 1u; }
    return true;
  }
};

// ------------------------------------------------------------ MXFP4
// MXFP4 operands of the block-scaled products.  The codes of a row (128
// elements, 64 bytes) sit in 64-byte-swizzled rows: 16-byte piece c of row r
// at r * 64 + ((c ^ ((r >> 1) & 3)) << 4), eight rows to a 512-byte atom (the
// layout TMA writes for a 64-byte box row under 64-byte swizzle).  The block
// scales of 128 rows sit in a 512-byte scale atom: byte r * 16 + j * 4 + k
// holds block k of row 32 j + r, the layout tensor memory takes them in (one
// 32-bit word per row, four rows per lane) by tcgen05.cp.32x128b.warpx4.
__device__ __forceinline__ uint32_t swz64(uint32_t row, uint32_t piece) {
  return row * 64u + ((piece ^ ((row >> 1) & 3u)) << 4);
}
__device__ __forceinline__ uint32_t scale_atom_byte(uint32_t row, uint32_t block) {
  return (row & 31u) * 16u + (row >> 5) * 4u + block;
}

// E2M1 codes of two floats (nearest, ties to even, saturating at 6): lo in
// the low nibble.
__device__ __forceinline__ uint32_t e2m1x2_code(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// MXFP4 quantisation of the group's bf16 query rows (sQ, 128B-swizzled
// 64-dim chunks) into E2M1 codes (sQ4, 64-byte-swizzled rows) and block
// scales (the scale atom sfb): blocks of 32 dims share the scale
// 2^(floor(log2 amax) - 2) (exponent at least -127), elements round to E2M1
// (nearest, ties to even, saturating at 6).  Epilogue warp e takes rows e,
// e + kEpiWarps, ...; lane l holds dims 4l .. 4l+3, so lanes 8g .. 8g+7 hold
// block g.
__device__ __forceinline__ void mx_query_codes(const uint8_t* sQ, uint8_t* sQ4, uint8_t* sfb,
                                               int NQ, int ew, int lane) {
  const int d = 4 * lane;
  const uint32_t off = static_cast<uint32_t>(d >> 6) * NQ * 128u;
  const uint32_t piece = (d & 63) >> 3, within = (d & 7) * 2;
  for (int r = ew; r < NQ; r += kEpiWarps) {
    const uint2 u = *reinterpret_cast<const uint2*>(sQ + off + swz128(r, piece) + within);
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    float amax = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int se = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127 - 2;
    se = se < -127 ? -127 : se;
    const float inv = __uint_as_float(static_cast<uint32_t>(127 - se) << 23);  // 2^-se
    const uint32_t c0 = e2m1x2_code(__fmul_rn(f0.x, inv), __fmul_rn(f0.y, inv));
    const uint32_t c1 = e2m1x2_code(__fmul_rn(f1.x, inv), __fmul_rn(f1.y, inv));
    // dims 4l .. 4l+3 are code bytes 2l, 2l+1: piece l / 8, byte 2 (l % 8)
    *reinterpret_cast<uint16_t*>(sQ4 + swz64(r, lane >> 3) + 2 * (lane & 7)) =
        static_cast<uint16_t>(c0 | (c1 << 8));
    if ((lane & 7) == 0) sfb[scale_atom_byte(r, lane >> 3)] = static_cast<uint8_t>(se + 127);
  }
}

// Quantises the group's bf16 query rows (sQ, 128B-swizzled 64-dim chunks)
// to E4M3 codes in sQ8 (one 128-byte swizzled row each) and their scales;
// epilogue warp e takes rows e, e + kEpiWarps, ...  Lane l holds dims
// 4l .. 4l+3 of a row.
__device__ __forceinline__ void quantize_query_rows(const uint8_t* sQ, uint8_t* sQ8,
                                                    float* qscale, int NQ, int ew, int lane) {
  const int d = 4 * lane;
  const uint32_t src_off = static_cast<uint32_t>(d >> 6) * NQ * 128u;
  const uint32_t piece = (d & 63) >> 3, within = (d & 7) * 2;
  for (int r = ew; r < NQ; r += kEpiWarps) {
    const uint2 u = *reinterpret_cast<const uint2*>(sQ + src_off + swz128(r, piece) + within);
    const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
    const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    const float v[4] = {f0.x, f0.y, f1.x, f1.y};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const E4m3Row q = e4m3_row(amax);
    *reinterpret_cast<uint32_t*>(sQ8 + swz128(r, lane >> 2) + 4 * (lane & 3)) = e4m3x4(v, q.inv);
    if (lane == 0) qscale[r] = q.scale;
  }
}

template <int KF>
__global__ void __launch_bounds__(kIdxThreads, 1)
    indexer_score_kernel(const __grid_constant__ CUtensorMap tm_ik,
                         const __grid_constant__ CUtensorMap tm_iq,
                         const __grid_constant__ CUtensorMap tm_ks, const IndexerArgs a) {
  constexpr bool F8 = KF == kKeyE4m3;  // E4M3 keys: kind::f8f6f4 products
  constexpr bool MX = KF == kKeyMx4;   // MXFP4 keys: kind::mxf4 block-scaled products
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the 128B-swizzled operand buffers
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  // [E4M3 query rows (FP8 keys) | E2M1 query rows and their scale atom
  // (MXFP4 keys)] [bf16 query rows] [key stages] [key scales of each stage
  // (FP8 keys) | a scale atom per accumulator (MXFP4 keys)] [IdxSmem]
  const uint32_t q8_bytes = indexer_q8_bytes(KF, a.NQ);
  const uint32_t q_bytes = static_cast<uint32_t>(a.KC) * a.NQ * 128u;
  const uint32_t stage_bytes =
      F8 ? 16384u : (MX ? kMxStageBytes : static_cast<uint32_t>(a.KC) * 16384u);
  uint8_t* sQ8 = base;  // FP8: E4M3 rows; MXFP4: E2M1 rows, then their scale atom
  uint8_t* sQ4 = base;
  uint8_t* sfb_atom = base + static_cast<uint32_t>(a.NQ) * 64u;
  uint8_t* sQ = base + q8_bytes;
  uint8_t* sA = sQ + q_bytes;
  float* sScale = reinterpret_cast<float*>(sA + a.stages * stage_bytes);
  uint8_t* sfa_atoms = sA + a.stages * stage_bytes;  // MXFP4: 512 bytes per accumulator
  IdxSmem* sm = reinterpret_cast<IdxSmem*>(
      sA + a.stages * stage_bytes +
      (F8 ? a.stages * kBlockRows * 4 : (MX ? a.nacc * 512 : 0)));
  const EpiLayout el = epi_layout(a.NQ, a.G, a.hist_part != nullptr);
  uint8_t* epi = reinterpret_cast<uint8_t*>(sm) + (sizeof(IdxSmem) + 15) / 16 * 16;
  float* qscale = reinterpret_cast<float*>(epi + el.qscale);
  uint32_t* hist = reinterpret_cast<uint32_t*>(epi + el.hist);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  pdl_trigger();  // top-k may begin launching as SMs free up

  const int64_t s0 = a.total_slots * blockIdx.x / gridDim.x;
  const int64_t s1 = a.total_slots * (blockIdx.x + 1) / gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.stages; ++i) {
      mbar_init(smem_u32(&sm->full[i]), 1);
      mbar_init(smem_u32(&sm->empty[i]), 1);
      // FP8: the four warps of the slot's epilogue group read its scales
      mbar_init(smem_u32(&sm->sempty[i]), 4);
    }
    for (int i = 0; i < a.nacc; ++i) {
      mbar_init(smem_u32(&sm->tfull[i]), 1);
      mbar_init(smem_u32(&sm->tempty[i]), 128);  // the four warps of one epilogue group
    }
    mbar_init(smem_u32(&sm->qfull), 1);
    mbar_init(smem_u32(&sm->qempty), 2);  // both MMA issuers leave the query block
    mbar_init(smem_u32(&sm->q8full), kEpiWarps);  // each epilogue warp quantised its rows
  }
  if (MX) {
    // the query scale atom's rows past NQ (never written per group): 2^0
    for (int i = threadIdx.x; i < 512; i += kIdxThreads) sfb_atom[i] = 127;
    fence_proxy_async_smem();  // read by tcgen05.cp
  }
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm->mma_done[0]), 1);
    mbar_init(smem_u32(&sm->mma_done[1]), 1);
    sm->abort = 0;
    fence_barrier_init();
    tma_prefetch_desc(&tm_ik);
    tma_prefetch_desc(&tm_iq);
    if (F8 || MX) tma_prefetch_desc(&tm_ks);
  }
  const int acc_cols = a.nacc * a.NQ + (MX ? 4 * a.nacc + 8 : 0);  // MXFP4: scale columns too
  const uint32_t tmem_cols = acc_cols <= 32 ? 32 : (acc_cols <= 64 ? 64 : (acc_cols <= 128 ? 128 : (acc_cols <= 256 ? 256 : 512)));
  // Slot it accumulates into accumulator it % nacc, its (it / nacc)-th use;
  // every role tracks (acc, parity of the use) as a counter pair.  With six
  // accumulators three epilogue groups drain them (slot it to group it % 3,
  // so each accumulator belongs to one group), else two.
  const int egroups = a.nacc % 3 == 0 ? 3 : 2;
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
  if (warp == 0 || warp == kProducer2) {
    // ------------------------------------------------------------ producers
    // Two producer threads (warp 0 and the last warp) issue the copies of
    // the even and the odd live slots: a single thread issues a slot's
    // copies only every ~0.45 us, less than the key stream needs.  The ring
    // is even, so each stage belongs to one of them.  Producer 0 also loads
    // each group's query rows.
    if (lane == 0) {
      const int ppar = warp == 0 ? 0 : 1;
      SlotCursor cur;
      int st = 0;
      uint32_t ph = 0;
      int64_t it = 0, qloads = 0, hi = 0;  // hi: one past the last slot this thread issued
      bool keys_ready = false;  // the compressed keys of the previous kernel are visible
      const uint64_t once = l2_policy_evict_first();
      const int nst = a.stages;
      // a new query group: producer 0 loads its query rows once the MMA
      // issuers have left the previous group's
      auto enter_group = [&]() -> bool {
        if (ppar != 0) return true;
        if (qloads > 0 &&
            !mbar_wait(smem_u32(&sm->qempty), (qloads - 1) & 1, abort, a.status, kWaitLimitNs, 10))
          return false;
        const uint32_t qb = smem_u32(&sm->qfull);
        mbar_arrive_expect_tx(qb, q_bytes);
        const int row0 = ((cur.b * a.T) + cur.t0) * a.HI;
        for (int kc = 0; kc < a.KC; ++kc)
          tma_load_2d(smem_u32(sQ + kc * a.NQ * 128), &tm_iq, kc * 64, row0, qb);
        ++qloads;
        return true;
      };
      auto step = [&]() -> bool {
        cur.advance(a);
        ++it;
        if (++st == nst) { st = 0; ph ^= 1u; }
        return !cur.done && (!cur.fresh || enter_group());
      };
      cur.init(a, s0, s1);
      bool more = !cur.done && enter_group();
      if (more && static_cast<int>(it & 1) != ppar) more = step();
      while (more && !*abort) {
        // stage st was last filled `stages` uses ago, in phase ph ^ 1; with
        // FP8 keys its scales are also read by the epilogue, which lags the
        // MMAs (MXFP4: the slot's MMA warp reads the scales before its
        // products, which release the stage)
        if (it >= a.stages &&
            !mbar_wait(smem_u32(&sm->empty[st]), ph ^ 1u, abort, a.status, kWaitLimitNs, 11))
          break;
        if (F8 && it >= nst &&
            !mbar_wait(smem_u32(&sm->sempty[st]), ph ^ 1u, abort, a.status, kWaitLimitNs, 20))
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
        mbar_arrive_expect_tx(fb, stage_bytes + (F8 ? kBlockRows * 4 : 0));
        // the keys are read once: first out of L2 (the scores written
        // meanwhile, and whatever the attention reads again, stay)
        if (MX) {
          // 128 rows of 64 code bytes (64-byte swizzle); their scales, 4 keys
          // per 16-byte row
          uint8_t* rs = sA + st * stage_bytes;
          tma_load_3d_hint(smem_u32(rs), &tm_ik, 0, cur.blk * kBlockRows, cur.b, fb, once);
          tma_load_3d_hint(smem_u32(rs + 8192), &tm_ks, 0, cur.blk * (kBlockRows / 4), cur.b, fb,
                           once);
        } else if (F8) {
          tma_load_3d_hint(smem_u32(sA + st * stage_bytes), &tm_ik, 0, cur.blk * kBlockRows,
                           cur.b, fb, once);
          tma_load_2d_hint(smem_u32(sScale + st * kBlockRows), &tm_ks, cur.blk * kBlockRows,
                           cur.b, fb, once);
        } else
          for (int kc = 0; kc < a.KC; ++kc)
            tma_load_3d_hint(smem_u32(sA + st * stage_bytes + kc * 16384), &tm_ik, kc * 64,
                             cur.blk * kBlockRows, cur.b, fb, once);
        hi = it + 1;
        // this thread's next slot, two on: plain arithmetic within the group
        if (cur.blk + 2 < cur.blk_end) {
          cur.blk += 2;
          it += 2;
          st += 2;
          if (st >= nst) { st -= nst; ph ^= 1u; }
        } else {
          more = step() && step();
        }
      }
      if (*abort) {
        // let the copies already issued land before the CTA exits: the last
        // query block (its predecessor's phase completed before it was
        // issued: the issuers had released it), then this thread's key
        // stages among the last `stages` slots
        if (qloads > 0)
          mbar_wait(smem_u32(&sm->qfull), (qloads - 1) & 1, nullptr, nullptr, 10000000ull, 13);
        for (int64_t x = hi > nst ? hi - nst : 0; x < hi; ++x)
          if (static_cast<int>(x & 1) == ppar)
            mbar_wait(smem_u32(&sm->full[x % nst]), (x / nst) & 1, nullptr, nullptr, 10000000ull,
                      12);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Warp 1 issues the products of the even live slots and warp 2 those of
    // the odd ones, so that one issuer's waits and per-slot bookkeeping
    // overlap the other's products.  Slot `it` accumulates into accumulator
    // it % nacc, its (it / nacc)-th use.
    const int par = warp == 1 ? 0 : 1;
    if (MX) {
      // MXFP4 keys: block-scaled products (kind::mxf4, K = 64 per call, two
      // per slot) of the key codes, as the copy lands them, and the group's
      // E2M1 query rows.  The scales reach tensor memory by tcgen05.cp from
      // 512-byte scale atoms: the query atom (the epilogue warps write it) at
      // each group change into this warp's own four columns, and per slot
      // the keys' scales, which travel with the stage key by key and which
      // the warp lays out as the atom of the slot's accumulator (lane r:
      // keys r, r + 32, r + 64, r + 96), into that accumulator's columns.
      const uint32_t sfa_col = tmem + static_cast<uint32_t>(a.nacc * a.NQ);
      const uint32_t sfb_col = sfa_col + 4u * a.nacc + 4u * par;
      const uint32_t qbar = smem_u32(&sm->q8full);  // the group's E2M1 rows and scales
      SlotWalk w;
      int64_t qn = 0;
      // a new query group: the previous group's rows are released, this
      // group's are ready, and their scales go to this warp's columns
      auto enter_group = [&]() -> bool {
        if (lane == 0 && qn > 0) mma_commit(smem_u32(&sm->qempty));
        if (!__all_sync(0xffffffffu, mbar_wait(qbar, qn & 1, abort, a.status, kWaitLimitNs, 13)))
          return false;
        ++qn;
        if (lane == 0) {
          tc_fence_after();
          tmem_cp_32x128b_x4(sfb_col, smem_desc(smem_u32(sfb_atom), 128, 128, kSwizzleNone));
        }
        return true;
      };
      auto step = [&]() -> bool {
        w.step(a);
        return !w.cur.done && (!w.cur.fresh || enter_group());
      };
      w.init(a, s0, s1);
      bool more = !w.cur.done && enter_group();
      if (more && static_cast<int>(w.it & 1) != par) more = step();
      while (more && !*abort) {
        const int st = w.st, acc = w.acc;
        bool got = true;
        // the accumulator's previous use has been drained by the epilogue
        // (its products and the copy of its scale atom are complete)
        if (w.it >= a.nacc)
          got = mbar_wait(smem_u32(&sm->tempty[acc]), w.aph ^ 1u, abort, a.status, kWaitLimitNs,
                          14);
        // the copy has landed
        got = got && mbar_wait(smem_u32(&sm->full[st]), w.ph, abort, a.status, kWaitLimitNs, 15);
        if (!__all_sync(0xffffffffu, got)) break;
        const uint8_t* stage = sA + st * stage_bytes;
        const uint32_t* ks = reinterpret_cast<const uint32_t*>(stage + 8192);
        uint8_t* atom = sfa_atoms + acc * 512;
        *reinterpret_cast<uint4*>(atom + lane * 16) =
            make_uint4(ks[lane], ks[32 + lane], ks[64 + lane], ks[96 + lane]);
        fence_proxy_async_smem();  // read by tcgen05.cp
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sfa = sfa_col + 4u * acc;
          tmem_cp_32x128b_x4(sfa, smem_desc(smem_u32(atom), 128, 128, kSwizzleNone));
          const uint32_t d_tmem = tmem + acc * a.NQ;
          const uint32_t a_addr = smem_u32(stage), b_addr = smem_u32(sQ4);
#pragma unroll
          for (int kh = 0; kh < 2; ++kh) {  // elements 64 kh .. 64 kh + 63: 32 bytes a row
            const uint64_t ad = smem_desc(a_addr + kh * 32, 16, 512, kSwizzle64B);
            const uint64_t bd = smem_desc(b_addr + kh * 32, 16, 512, kSwizzle64B);
            mma_mxf4_ss(d_tmem, ad, bd, idesc_mxf4(128, a.NQ, 2u * kh, 2u * kh), sfa, sfb_col,
                        kh);
          }
          mma_commit(smem_u32(&sm->empty[st]));
          mma_commit(smem_u32(&sm->tfull[acc]));
        }
        __syncwarp();
        // this warp's next slot, two on
        if (!w.leap(a, 2)) more = step() && step();
      }
      // all issued MMAs complete before the accumulators are released
      if (lane == 0) {
        mma_commit(smem_u32(&sm->mma_done[par]));
        mbar_wait(smem_u32(&sm->mma_done[par]), 0, nullptr, a.status, kWaitLimitNs, 16);
      }
      __syncwarp();
    } else {
      // bf16 or E4M3 keys.  The whole warp walks the slots and computes the
      // operand descriptors (warp-uniform values, so they stay in uniform
      // registers); lane 0 issues the products.
      const uint32_t idesc = F8 ? idesc_e4m3(128, a.NQ) : idesc_bf16(128, a.NQ, 0, 0);
      // the operand rows the products read: E4M3 codes, or the bf16 rows
      const uint32_t qbar = smem_u32(F8 ? &sm->q8full : &sm->qfull);
      // descriptors: 128-byte swizzle, 8-row atoms 1024 bytes apart; a K
      // step of 32 bytes adds 2 to the start address field, a 64-dim chunk
      // (16 KB of keys, NQ x 128 bytes of queries) adds its size / 16
      const uint64_t q_desc = smem_desc(smem_u32(F8 ? sQ8 : sQ), 16, 1024, kSwizzle128B);
      const uint64_t k_desc0 = smem_desc(smem_u32(sA), 16, 1024, kSwizzle128B);
      SlotWalk w;
      int64_t qn = 0;
      // a new query group: the previous group's reads of the query rows are
      // released and this group's are ready
      auto enter_group = [&]() -> bool {
        if (lane == 0 && qn > 0) mma_commit(smem_u32(&sm->qempty));
        if (!__all_sync(0xffffffffu, mbar_wait(qbar, qn & 1, abort, a.status, kWaitLimitNs, 13)))
          return false;
        ++qn;
        return true;
      };
      auto step = [&]() -> bool {
        w.step(a);
        return !w.cur.done && (!w.cur.fresh || enter_group());
      };
      w.init(a, s0, s1);
      bool more = !w.cur.done && enter_group();
      if (more && static_cast<int>(w.it & 1) != par) more = step();
      while (more && !*abort) {
        const int st = w.st, acc = w.acc;
        bool got = true;
        // the accumulator's previous use has been drained by the epilogue
        if (w.it >= a.nacc)
          got = mbar_wait(smem_u32(&sm->tempty[acc]), w.aph ^ 1u, abort, a.status, kWaitLimitNs,
                          14);
        got = got && mbar_wait(smem_u32(&sm->full[st]), w.ph, abort, a.status, kWaitLimitNs, 15);
        if (!__all_sync(0xffffffffu, got)) break;
        const uint32_t d_tmem = tmem + acc * a.NQ;
        const uint64_t k_desc = k_desc0 + static_cast<uint64_t>(st * (stage_bytes >> 4));
        if (lane == 0) {
          tc_fence_after();
          if (F8) {
            // one 128-byte row per key and per query: 4 steps of K = 32
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_f8_ss(d_tmem, k_desc + 2 * ks, q_desc + 2 * ks, idesc, ks != 0);
          } else {
            for (int kc = 0; kc < a.KC; ++kc) {
              const uint64_t kd = k_desc + kc * (16384 >> 4);
              const uint64_t qd = q_desc + static_cast<uint64_t>(kc * a.NQ * (128 >> 4));
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_bf16_ss(d_tmem, kd + 2 * ks, qd + 2 * ks, idesc, (kc | ks) != 0);
            }
          }
          mma_commit(smem_u32(&sm->empty[st]));
          mma_commit(smem_u32(&sm->tfull[acc]));
        }
        __syncwarp();
        // this warp's next slot, two on
        if (!w.leap(a, 2)) more = step() && step();
      }
      // all issued MMAs complete before the accumulators are released
      if (lane == 0) {
        mma_commit(smem_u32(&sm->mma_done[par]));
        mbar_wait(smem_u32(&sm->mma_done[par]), 0, nullptr, a.status, kWaitLimitNs, 16);
      }
      __syncwarp();
    }
  } else if (warp >= kFirstEpiWarp && warp < kFirstEpiWarp + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    // Group eg drains the slots it with it % egroups == eg (a group past
    // egroups drains none but still quantises its share of each group's
    // query rows); its warp for tensor-memory lanes quad*32 .. quad*32+31
    // handles those 32 entries.
    const int ew = warp - kFirstEpiWarp;
    const int eg = ew >> 2;
    const int quad = warp & 3;
    const int row = quad * 32 + lane;
    float* wcol = reinterpret_cast<float*>(epi + el.wcol) + ew * a.NQ;
    const uint32_t wcol_s = smem_u32(wcol);
    int* ntv = reinterpret_cast<int*>(epi + el.nt) + ew * a.G;
    // Folded first selection pass (one query per group): the top 11 bits of
    // each visible score's key are counted per row, for the first and the
    // second row this CTA's slots touch (its slots span at most two rows).
    const bool fold = a.hist_part != nullptr;
    const int64_t row0 = s0 / a.nblk;
    // the scores are read again by the selection right after this kernel
    const uint64_t keep = l2_policy_evict_last();
    if (fold) {
      for (int i = threadIdx.x - kFirstEpiWarp * 32; i < 2 * kHistWords; i += kEpiWarps * 32)
        hist[i] = 0u;
      named_bar_sync(1, kEpiWarps * 32);
    }
    // heads a multiple of 32: every 32-column accumulator chunk belongs to
    // one query, so a query's score is a straight sum over its chunks
    const bool whole = (a.HI & 31) == 0;
    const int cpq = a.HI >> 5;
    SlotCursor cur;
    int64_t it = 0, qn = 0;
    int st = 0;  // the slot's key stage (FP8: its scales are read from there)
    uint32_t ph = 0;
    float* sbase = nullptr;  // the group's first score row, at this thread's entry of block 0
    int hoff = 0;            // the group's histogram (first or second row of the CTA)
    int rot = 0;             // it % egroups: the epilogue group of slot it
    int acc = 0;             // it % nacc
    uint32_t aph = 0;        // parity of (it / nacc)
    // A new query group: its weights and visible counts, and (FP8, MXFP4)
    // this warp's share of the query rows' quantisation.  Every epilogue warp
    // enters every group, in order.  False when a wait gave up.
    auto enter_group = [&]() -> bool {
      sbase = a.scores + ((int64_t)cur.b * a.T + cur.t0) * a.N_cap + row;
      hoff = cur.group == row0 ? 0 : kHistWords;
      if (F8 || MX) {
        // the group's bf16 query rows have landed: quantise this warp's
        // share, publish it to the MMA issuers, then wait for the others'
        // row scales (MXFP4: the rows' E2M1 codes and their scale atom)
        bool got = mbar_wait(smem_u32(&sm->qfull), qn & 1, abort, a.status, kWaitLimitNs, 18);
        if (!__all_sync(0xffffffffu, got)) return false;
        if (MX) mx_query_codes(sQ, sQ4, sfb_atom, a.NQ, ew, lane);
        else quantize_query_rows(sQ, sQ8, qscale, a.NQ, ew, lane);
        fence_proxy_async_smem();  // visible to the tensor core's reads
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->q8full));
        got = mbar_wait(smem_u32(&sm->q8full), qn & 1, abort, a.status, kWaitLimitNs, 19);
        if (!__all_sync(0xffffffffu, got)) return false;
        ++qn;
      }
      __syncwarp();
      for (int c = lane; c < a.NQ; c += 32) {
        const int g = c / a.HI, h = c % a.HI;
        const float wv = (g < cur.gv) ? a.w[((int64_t)cur.b * a.T + cur.t0 + g) * a.HI + h] : 0.f;
        wcol[c] = F8 ? wv * qscale[c] : wv;
      }
      for (int g = lane; g < a.G; g += 32)
        ntv[g] = g < cur.gv ? static_cast<int>(visible_entries(
                                  a.pos[(int64_t)cur.b * a.T + cur.t0 + g], a.m, a.N_cap))
                            : 0;
      __syncwarp();
      return true;
    };
    // on to the next live slot (entering its group); false at the end
    auto step = [&]() -> bool {
      cur.advance(a);
      ++it;
      if (++rot == egroups) rot = 0;
      if (++acc == a.nacc) { acc = 0; aph ^= 1u; }
      if (++st == a.stages) { st = 0; ph ^= 1u; }
      return !cur.done && (!cur.fresh || enter_group());
    };
    // this group's next slot, egroups slots on: plain arithmetic while they
    // stay in the current query group (the common case), else slot by slot
    // (every warp enters every group)
    const bool leap = a.stages >= egroups;  // a leap wraps each ring at most once
    auto next_own = [&]() -> bool {
      if (leap && cur.blk + egroups < cur.blk_end) {
        cur.blk += egroups;
        it += egroups;
        acc += egroups;
        if (acc >= a.nacc) { acc -= a.nacc; aph ^= 1u; }
        st += egroups;
        if (st >= a.stages) { st -= a.stages; ph ^= 1u; }
        return true;
      }
      bool m = true;
      for (int k = 0; k < egroups && m; ++k) m = step();
      return m;
    };
    cur.init(a, s0, s1);
    bool more = !cur.done && enter_group();  // a first slot always opens its group
    while (more && rot != eg) more = step();
    // one pass per slot of this group: the slots of the other groups are
    // stepped over between passes
    while (more) {
      const int sst = st;
      const uint32_t sph = ph;
      const int j = cur.blk * kBlockRows + row;
      const bool got =
          mbar_wait(smem_u32(&sm->tfull[acc]), aph, abort, a.status, kWaitLimitNs, 17);
      if (!__all_sync(0xffffffffu, got)) break;  // warp-uniform: tcgen05.ld follows
      tc_fence_after();
      float ks = 1.f;
      if (F8) {
        // the stage's copy completed before its MMAs ran; this wait returns
        // at once and makes the scales the copy wrote visible here
        const bool sg = mbar_wait(smem_u32(&sm->full[sst]), sph, abort, a.status, kWaitLimitNs, 21);
        if (!__all_sync(0xffffffffu, sg)) break;
        ks = sScale[sst * kBlockRows + row];
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sm->sempty[sst]));
      }
      const uint32_t taddr = tmem + (static_cast<uint32_t>(quad * 32) << 16) + acc * a.NQ;
      float* srow = sbase + cur.blk * kBlockRows;
      if (whole) {
        for (int g = 0; g < cur.gv; ++g) {
          // four independent partial sums (one per column of a float4), so
          // the FMAs do not wait on one another; scalar FMAs, which take the
          // maxima from any register (a packed FMA wants them as a pair)
          float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
          for (int c = 0; c < cpq; c += 2) {
            const int col = (g * cpq + c) * 32;
            float x0[32], x1[32];
            tmem_ld32(taddr + col, x0);
            if (c + 1 < cpq) tmem_ld32(taddr + col + 32, x1);
            tmem_wait_ld();
            const uint32_t w0 = wcol_s + col * 4;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 wv = lds_f4(w0 + 16 * i);
              p0 = fmaf(wv.x, fmaxf(x0[4 * i], 0.f), p0);
              p1 = fmaf(wv.y, fmaxf(x0[4 * i + 1], 0.f), p1);
              p2 = fmaf(wv.z, fmaxf(x0[4 * i + 2], 0.f), p2);
              p3 = fmaf(wv.w, fmaxf(x0[4 * i + 3], 0.f), p3);
            }
            if (c + 1 < cpq) {
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float4 wv = lds_f4(w0 + 128 + 16 * i);
                p0 = fmaf(wv.x, fmaxf(x1[4 * i], 0.f), p0);
                p1 = fmaf(wv.y, fmaxf(x1[4 * i + 1], 0.f), p1);
                p2 = fmaf(wv.z, fmaxf(x1[4 * i + 2], 0.f), p2);
                p3 = fmaf(wv.w, fmaxf(x1[4 * i + 3], 0.f), p3);
              }
            }
          }
          const float sum = (p0 + p1) + (p2 + p3);
          if (j < ntv[g]) {
            const float sc = F8 ? sum * ks : sum;
            st_global_hint(srow + (int64_t)g * a.N_cap, sc, keep);
            if (fold) {
              const uint32_t bin = score_key(sc) >> 21;
              atomicAdd(&hist[hoff + (bin >> 1)],
                        1u << ((bin & 1u) * 16u));
            }
          }
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
              if (g < cur.gv && j < ntv[g]) {
                const float sc = F8 ? sum * ks : sum;
                st_global_hint(srow + (int64_t)g * a.N_cap, sc, keep);
                if (fold) {
                  const uint32_t bin = score_key(sc) >> 21;
                  atomicAdd(&hist[hoff + (bin >> 1)],
                            1u << ((bin & 1u) * 16u));
                }
              }
              sum = 0.f;
              h = 0;
              ++g;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&sm->tempty[acc]));
      more = next_own();
    }
    if (fold) {
      // this CTA's partial histograms, part[cta][0] for its first row and
      // part[cta][1] for the second (when its slots reach one)
      named_bar_sync(1, kEpiWarps * 32);
      const int64_t row1 = (s1 - 1) / a.nblk;
      const int nv = (row1 != row0 ? 2 : 1) * kHistWords / 4;
      uint4* dst = reinterpret_cast<uint4*>(a.hist_part + static_cast<int64_t>(blockIdx.x) * 2 * kSelBins);
      const uint4* src = reinterpret_cast<const uint4*>(hist);
      for (int i = threadIdx.x - kFirstEpiWarp * 32; i < nv; i += kEpiWarps * 32) dst[i] = src[i];
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, tmem_cols);
}

}  // namespace

bool plan_indexer(int T, int HI, int dI, int kf, bool fold, IndexerPlan* p) {
  if (HI <= 0 || HI > 256 || dI <= 0 || dI > 128) return false;
  const bool f8 = kf == kKeyE4m3, mx = kf == kKeyMx4;
  if ((f8 || mx) && dI != 128) return false;
  // MXFP4: at most 128 query rows a group, so that two accumulators and the
  // scale columns fit in tensor memory
  const int max_nq = mx ? 128 : 256;
  int G = max_nq / HI;
  if (G > T) G = T;
  if (G < 1) G = 1;
  int NQ = ((G * HI + 31) / 32) * 32;
  if (NQ > max_nq) return false;
  p->G = G;
  p->NQ = NQ;
  p->KC = (dI + 63) / 64;
  const size_t q_bytes = (size_t)p->KC * NQ * 128 + indexer_q8_bytes(kf, NQ);
  // FP8: 16 KB of codes plus the block's 128 fp32 scales per stage; MXFP4:
  // 8 KB of codes plus 512 bytes of scales
  const size_t stage_bytes =
      f8 ? 16384 + kBlockRows * 4 : (mx ? kMxStageBytes : (size_t)p->KC * 16384);
  if (fold && G != 1) return false;  // the folded pass counts one query per group
  // Accumulators: six when tensor memory holds them (three epilogue groups
  // drain them, slot s to group s % 3), else as many as it holds up to
  // kMaxAcc, a power of 2 (two epilogue groups).  MXFP4 also keeps four
  // scale columns per accumulator and four per MMA issuer.
  auto cols = [&](int n) { return n * NQ + (mx ? 4 * n + 8 : 0); };
  int nacc = 2;
  while (nacc * 2 <= kMaxAcc && cols(nacc * 2) <= 512) nacc *= 2;
  if (cols(6) <= 512) nacc = 6;
  if (cols(nacc) > 512) return false;
  const int egroups = nacc % 3 == 0 ? 3 : 2;
  const size_t fixed = (sizeof(IdxSmem) + 15) / 16 * 16 + epi_layout(NQ, G, fold).bytes +
                       (mx ? (size_t)nacc * 512 : 0);
  const size_t budget = 227 * 1024 - 1024 - fixed - q_bytes;
  int stages = static_cast<int>(budget / stage_bytes);
  const int cap = (f8 || mx) ? kMaxStages : kMaxStagesBf16;
  if (stages > cap) stages = cap;
  // Slot s uses stage s % stages and accumulator s % nacc, is issued by MMA
  // warp s % 2 and drained by epilogue group s % egroups.  A ring whose
  // length is a multiple of the roles sharing it gives each stage (each
  // accumulator) to one issuer and one group, so each waits on a barrier's
  // phases in order.  Otherwise a stage alternates between, say, the
  // issuers, and an issuer that runs a lap ahead of the other would wait on
  // the parity of a phase whose predecessor is still pending -- a parity
  // wait that passes at once.  The stages of bf16 and MXFP4 keys are the
  // issuers' alone; the epilogue reads the FP8 key scales from its slot's
  // stage.
  const int ring = f8 ? 2 * egroups : 2;
  stages -= stages % ring;
  if (stages < ring) return false;
  p->stages = stages;
  p->nacc = nacc;
  p->tmem_cols = cols(nacc);
  p->smem_bytes = 1024 + q_bytes + stages * stage_bytes + fixed;
  return true;
}

cudaError_t launch_indexer_score(const CUtensorMap& tm_ik, const CUtensorMap& tm_iq,
                                 const CUtensorMap& tm_ks, const IndexerArgs& a,
                                 const IndexerPlan& p, int kf, int grid, cudaStream_t stream) {
  auto kernel = kf == kKeyE4m3 ? indexer_score_kernel<kKeyE4m3>
                               : (kf == kKeyMx4 ? indexer_score_kernel<kKeyMx4>
                                                : indexer_score_kernel<kKeyBf16>);
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(p.smem_bytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kIdxThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  cfg.attrs = at;
  cfg.numAttrs = add_dependent_attr(at, 0, a.dependent != 0);
  e = cudaLaunchKernelEx(&cfg, kernel, tm_ik, tm_iq, tm_ks, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace hattn
