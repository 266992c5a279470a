// compress.cu -- the KV compressor C(m, w) used by CSA (m=4, w=8, with the
// indexer key) and HCA (m=w=128, KV only).
//
// "Why DeepSeek V4 Stands Apart", section "Core Architectural Innovations":
// CSA compresses KV 4x (m=4), HCA 128:1.  "DeepSeek-V4" atlas, section
// "Design overview": every 4 tokens are compressed into two overlapping
// streams, and the compressed KV entries are RMSNorm'd.  Provenance 16: RoPE
// on the last 64 dims.
//
// Entry j pools tokens u in [m(j+1)-w, m(j+1)-1] (u >= 0) with weights
// softmax(gate_u); the pooled KV is RMSNorm'd and RoPE'd at position m(j+1)-1;
// the pooled indexer key uses the same weights, no norm, no RoPE.
//
// One CTA processes one (sequence, entry) at a time in a grid-stride loop.
// Threads are laid out as NC column pieces (16 bytes = 8 bf16 of the
// concatenated [KV | indexer-key] row) x S token slices; every token row of
// the window is read once, with 16-byte coalesced loads, and every output
// row is written once.  Accumulation is fp32; the entry is rounded to bf16
// once at the end.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kCompressThreads = 512;
constexpr int kMaxW = 512;

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
  uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    x[2 * i] = f.x;
    x[2 * i + 1] = f.y;
  }
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float (&y)[8]) {
  uint4 u;
  u.x = pack_bf16x2(y[0], y[1]);
  u.y = pack_bf16x2(y[2], y[3]);
  u.z = pack_bf16x2(y[4], y[5]);
  u.w = pack_bf16x2(y[6], y[7]);
  *reinterpret_cast<uint4*>(p) = u;
}

// Row of token u in the raw buffers: u itself, or u mod ring when they are a
// ring of the last `ring` tokens (a power of two).
__device__ __forceinline__ int64_t token_row(const CompressArgs& a, int64_t u) {
  return a.ring > 0 ? (u & (a.ring - 1)) : u;
}

// Largest magnitude of the bf16-rounded values of one 8-wide piece.
__device__ __forceinline__ float amax8_bf16(const float (&y)[8]) {
  float m = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(bf16_round(y[e])));
  return m;
}

// E4M3 codes of the bf16-rounded values of one 8-wide piece (the values the
// bf16 indexer key holds), scaled by the row's inv.
__device__ __forceinline__ void store8_e4m3(uint8_t* p, const float (&y)[8], float inv) {
  float r[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) r[e] = bf16_round(y[e]);
  uint2 u;
  u.x = e4m3x4(r, inv);
  u.y = e4m3x4(r + 4, inv);
  *reinterpret_cast<uint2*>(p) = u;
}

// MXFP4 codes and block scale of the bf16-rounded values of an 8-wide piece
// of the indexer key (the values the bf16 key holds), as the row quantiser
// writes them: a block of 32 elements is the pieces of 4 consecutive lanes
// (piece p on a lane with lane % 4 == p % 4), its scale 2^se with se =
// floor(log2 amax) - 2 (at least -127), elements x * 2^-se rounded to E2M1
// (nearest, ties to even, saturating), the low nibble the even element, a
// zero stored as +0.  Every lane of the warp calls it (the block's amax is
// reduced by shuffles); `valid` marks the lanes that hold a piece.
__device__ __forceinline__ void store8_mxfp4(bool valid, const float (&y)[8], uint8_t* codes,
                                             uint8_t* scales, int piece) {
  float r[8];
  float am = 0.f;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    r[e] = bf16_round(y[e]);
    am = fmaxf(am, fabsf(r[e]));
  }
  if (!valid) am = 0.f;
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
  if (!valid) return;
  int se = static_cast<int>((__float_as_uint(am) >> 23) & 0xffu) - 127 - 2;
  se = se < -127 ? -127 : se;
  const float inv = __uint_as_float(static_cast<uint32_t>(127 - se) << 23);  // 2^-se
  uint32_t w = 0;
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    uint32_t c;
    asm("{\n\t.reg .b8 t;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
        "cvt.u32.u8 %0, t;\n\t}"
        : "=r"(c)
        : "f"(__fmul_rn(r[e + 1], inv)), "f"(__fmul_rn(r[e], inv)));
    w |= c << (4 * e);
  }
  const uint32_t mag = w & 0x77777777u;
  w = mag | (w & ((mag + 0x77777777u) & 0x88888888u));  // drop the sign of zero nibbles
  *reinterpret_cast<uint32_t*>(codes + piece * 4) = w;
  if ((piece & 3) == 0) scales[piece >> 2] = static_cast<uint8_t>(se + 127);
}

__global__ void __launch_bounds__(kCompressThreads)
    compress_kernel(const __grid_constant__ CompressArgs a) {
  __shared__ float alpha[kMaxW];
  __shared__ float partial[4096];  // S x (D + dI) floats, S * NC <= 512 -> <= 4096
  __shared__ float rc[4][kMaxRopePairs];
  __shared__ float red[kCompressThreads / 32];
  __shared__ float red_am[kCompressThreads / 32];
  __shared__ float inv_rms_s, amax_s;

  pdl_trigger();  // a dependent launch after this kernel may begin
  const int tid = threadIdx.x;
  const int NCk = a.D / 8;                 // KV pieces
  const int NCi = a.ik_raw ? a.dI / 8 : 0; // indexer-key pieces
  const int NC = NCk + NCi;
  const int S = kCompressThreads / NC;     // token slices
  const int width = NC * 8;

  for (int i = tid; i < a.r / 2; i += kCompressThreads) {
#pragma unroll
    for (int c = 0; c < 4; ++c) rc[c][i] = a.rope.c[c][i];
  }

  const int64_t nj = a.j_end - a.j_begin;
  const int64_t items = nj * a.B;
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int b = static_cast<int>(item / nj);
    const int64_t j = a.j_begin + item % nj;
    const int64_t u0 = static_cast<int64_t>(a.m) * (j + 1) - a.w;

    // A window that one pass of the token loop covers (CSA: 8 tokens) has
    // its token rows requested before the gate softmax, so the two global
    // round trips overlap.
    const bool one_pass = a.w <= 8 * S;
    const int c_pre = tid % NC, s_pre = tid / NC;
    uint4 pre[8];
    if (one_pass && tid < S * NC) {
      const __nv_bfloat16* src = c_pre < NCk
          ? a.kv_raw + (int64_t)b * a.L_cap * a.D + c_pre * 8
          : a.ik_raw + (int64_t)b * a.L_cap * a.dI + (c_pre - NCk) * 8;
      const int64_t stride = c_pre < NCk ? a.D : a.dI;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = s_pre + q * S;
        const int64_t u = u0 + i;
        pre[q] = (i < a.w && u >= 0) ? __ldg(reinterpret_cast<const uint4*>(src + token_row(a, u) * stride))
                                     : make_uint4(0, 0, 0, 0);
      }
    }

    // gate softmax over the tokens that exist (warp 0)
    if (tid < 32) {
      float gmax = -INFINITY;
      for (int s = tid; s < a.w; s += 32) {
        int64_t u = u0 + s;
        if (u >= 0) gmax = fmaxf(gmax, __bfloat162float(a.gate[(int64_t)b * a.L_cap + token_row(a, u)]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
      float z = 0.f;
      for (int s = tid; s < a.w; s += 32) {
        int64_t u = u0 + s;
        float e = 0.f;
        if (u >= 0) e = __expf(__bfloat162float(a.gate[(int64_t)b * a.L_cap + token_row(a, u)]) - gmax);
        alpha[s] = e;
        z += e;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      const float iz = 1.f / z;
      __syncwarp();
      for (int s = tid; s < a.w; s += 32) alpha[s] *= iz;
    }
    __syncthreads();

    // weighted sums: thread (c, s) covers piece c over tokens s, s+S, ...,
    // eight token rows in flight at a time
    if (tid < S * NC) {
      const int c = tid % NC;
      const int s = tid / NC;
      const __nv_bfloat16* src = c < NCk ? a.kv_raw + (int64_t)b * a.L_cap * a.D + c * 8
                                         : a.ik_raw + (int64_t)b * a.L_cap * a.dI + (c - NCk) * 8;
      const int64_t stride = c < NCk ? a.D : a.dI;
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.f;
      for (int i0 = s; i0 < a.w; i0 += 8 * S) {
        uint4 v[8];
        float al[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const int i = i0 + q * S;
          const int64_t u = u0 + i;
          const bool live = i < a.w && u >= 0;
          if (one_pass)
            v[q] = pre[q];  // requested before the softmax (zero where not live)
          else
            v[q] = live ? __ldg(reinterpret_cast<const uint4*>(src + token_row(a, u) * stride))
                        : make_uint4(0, 0, 0, 0);
          al[q] = live ? alpha[i] : 0.f;
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float x[8];
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[q]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            x[2 * e] = f.x;
            x[2 * e + 1] = f.y;
          }
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = fmaf(al[q], x[e], acc[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) partial[s * width + c * 8 + e] = acc[e];
    }
    __syncthreads();

    // reduce the slices (fixed order), RMS over the KV part, largest
    // magnitude of the indexer key (for its E4M3 codes)
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = 0.f;
    float ss = 0.f, am = 0.f;
    if (tid < NC) {
      for (int s = 0; s < S; ++s)
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] += partial[s * width + tid * 8 + e];
      if (tid < NCk) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[e], v[e], ss);
      } else if (a.ik8_out) {
        am = amax8_bf16(v);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, o);
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    }
    if ((tid & 31) == 0) {
      red[tid >> 5] = ss;
      red_am[tid >> 5] = am;
    }
    __syncthreads();
    if (tid == 0) {
      float t = 0.f, mx = 0.f;
      for (int i = 0; i < kCompressThreads / 32; ++i) {
        t += red[i];
        mx = fmaxf(mx, red_am[i]);
      }
      inv_rms_s = rsqrtf(t / static_cast<float>(a.D) + a.eps);
      amax_s = mx;
    }
    __syncthreads();

    if (tid < NCk) {
      const float inv = inv_rms_s;
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float g = a.gamma ? a.gamma[tid * 8 + e] : 1.f;
        y[e] = v[e] * inv * g;
      }
      const int d0 = a.D - a.r;
      const int64_t p = static_cast<int64_t>(a.m) * (j + 1) - 1;
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const int d = tid * 8 + e;
        if (d >= d0) {
          float sn, cs;
          rope_cs(rc, (d - d0) / 2, p, &sn, &cs);
          const float x0 = y[e], x1 = y[e + 1];
          y[e] = x0 * cs - x1 * sn;
          y[e + 1] = x0 * sn + x1 * cs;
        }
      }
      store8(a.kv_out + ((int64_t)b * a.N_cap + j) * a.D + tid * 8, y);
    } else if (tid < NC) {
      const int64_t row = (int64_t)b * a.N_cap + j;
      if (a.ik_out) store8(a.ik_out + row * a.dI + (tid - NCk) * 8, v);
      if (a.ik8_out) {
        const E4m3Row q = e4m3_row(amax_s);
        store8_e4m3(a.ik8_out + row * a.dI + (tid - NCk) * 8, v, q.inv);
        if (tid == NCk) a.ik_scale_out[row] = q.scale;
      }
    }
    if (a.ik4_out) {
      const int64_t row = (int64_t)b * a.N_cap + j;
      store8_mxfp4(tid >= NCk && tid < NC, v, a.ik4_out + row * (a.dI / 2),
                   a.ik4_scale_out + row * (a.dI / 32), tid - NCk);
    }
    __syncthreads();
  }
}

// A few entries with short windows (CSA at decode: one entry per sequence,
// 8 tokens): 128 threads and ~1 KB of shared memory, so a CTA fits beside a
// CTA of the persistent indexer on the same SM instead of delaying it.
// Thread c owns 16-byte piece c of the [KV | indexer-key] row and has every
// token of the window in flight at once.
constexpr int kSmallThreads = 128;
constexpr int kSmallMaxW = 16;

__global__ void __launch_bounds__(kSmallThreads)
    compress_small_kernel(const __grid_constant__ CompressArgs a) {
  __shared__ float alpha[kSmallMaxW];
  __shared__ float rc[4][kMaxRopePairs];
  __shared__ float red[kSmallThreads / 32];
  __shared__ float red_am[kSmallThreads / 32];
  pdl_trigger();  // a dependent launch after this kernel may begin
  const int tid = threadIdx.x;
  const int NCk = a.D / 8;
  const int NC = NCk + (a.ik_raw ? a.dI / 8 : 0);
  for (int i = tid; i < a.r / 2; i += kSmallThreads) {
#pragma unroll
    for (int c = 0; c < 4; ++c) rc[c][i] = a.rope.c[c][i];
  }
  const int64_t nj = a.j_end - a.j_begin;
  const int64_t items = nj * a.B;
  for (int64_t item = blockIdx.x; item < items; item += gridDim.x) {
    const int b = static_cast<int>(item / nj);
    const int64_t j = a.j_begin + item % nj;
    const int64_t u0 = static_cast<int64_t>(a.m) * (j + 1) - a.w;
    // the window's rows of this thread's piece, all requested at once
    uint4 v[kSmallMaxW];
    if (tid < NC) {
      const __nv_bfloat16* src = tid < NCk
          ? a.kv_raw + (int64_t)b * a.L_cap * a.D + tid * 8
          : a.ik_raw + (int64_t)b * a.L_cap * a.dI + (tid - NCk) * 8;
      const int64_t stride = tid < NCk ? a.D : a.dI;
#pragma unroll
      for (int q = 0; q < kSmallMaxW; ++q) {
        const int64_t u = u0 + q;
        v[q] = (q < a.w && u >= 0) ? __ldg(reinterpret_cast<const uint4*>(src + token_row(a, u) * stride))
                                   : make_uint4(0, 0, 0, 0);
      }
    }
    // gate softmax over the tokens that exist (warp 0, one token per lane)
    if (tid < 32) {
      const int64_t u = u0 + tid;
      const bool live = tid < a.w && u >= 0;
      const float g = live ? __bfloat162float(a.gate[(int64_t)b * a.L_cap + token_row(a, u)]) : -INFINITY;
      float gmax = g;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
      const float e = live ? __expf(g - gmax) : 0.f;
      float z = e;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      if (tid < kSmallMaxW) alpha[tid] = e / z;
    }
    __syncthreads();
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    float ss = 0.f, am = 0.f;
    if (tid < NC) {
#pragma unroll
      for (int q = 0; q < kSmallMaxW; ++q) {
        const float al = alpha[q];  // zero for tokens that do not exist or lie past w
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[q]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(h[e]);
          acc[2 * e] = fmaf(al, f.x, acc[2 * e]);
          acc[2 * e + 1] = fmaf(al, f.y, acc[2 * e + 1]);
        }
      }
      if (tid < NCk) {
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(acc[e], acc[e], ss);
      } else if (a.ik8_out) {
        am = amax8_bf16(acc);
      }
    }
    // RMS over the KV part, largest magnitude of the indexer key
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      ss += __shfl_xor_sync(0xffffffffu, ss, o);
      am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    }
    if ((tid & 31) == 0) {
      red[tid >> 5] = ss;
      red_am[tid >> 5] = am;
    }
    __syncthreads();
    float tot = 0.f, amax = 0.f;
#pragma unroll
    for (int i = 0; i < kSmallThreads / 32; ++i) {
      tot += red[i];
      amax = fmaxf(amax, red_am[i]);
    }
    const float inv = rsqrtf(tot / static_cast<float>(a.D) + a.eps);
    if (tid < NCk) {
      float y[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float g = a.gamma ? a.gamma[tid * 8 + e] : 1.f;
        y[e] = acc[e] * inv * g;
      }
      const int d0 = a.D - a.r;
      const int64_t p = static_cast<int64_t>(a.m) * (j + 1) - 1;
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        const int d = tid * 8 + e;
        if (d >= d0) {
          float sn, cs;
          rope_cs(rc, (d - d0) / 2, p, &sn, &cs);
          const float x0 = y[e], x1 = y[e + 1];
          y[e] = x0 * cs - x1 * sn;
          y[e + 1] = x0 * sn + x1 * cs;
        }
      }
      store8(a.kv_out + ((int64_t)b * a.N_cap + j) * a.D + tid * 8, y);
    } else if (tid < NC) {
      const int64_t row = (int64_t)b * a.N_cap + j;
      if (a.ik_out) store8(a.ik_out + row * a.dI + (tid - NCk) * 8, acc);
      if (a.ik8_out) {
        const E4m3Row q = e4m3_row(amax);
        store8_e4m3(a.ik8_out + row * a.dI + (tid - NCk) * 8, acc, q.inv);
        if (tid == NCk) a.ik_scale_out[row] = q.scale;
      }
    }
    if (a.ik4_out) {
      const int64_t row = (int64_t)b * a.N_cap + j;
      store8_mxfp4(tid >= NCk && tid < NC, acc, a.ik4_out + row * (a.dI / 2),
                   a.ik4_scale_out + row * (a.dI / 32), tid - NCk);
    }
    __syncthreads();  // alpha and red are rewritten by the next entry
  }
}

}  // namespace

cudaError_t launch_compress(const CompressArgs& a, int num_sms, cudaStream_t stream) {
  const int64_t items = (a.j_end - a.j_begin) * a.B;
  if (items <= 0) return cudaSuccess;
  const int NC = a.D / 8 + (a.ik_raw ? a.dI / 8 : 0);
  if (a.w <= kSmallMaxW && NC <= kSmallThreads && items <= 4 * (int64_t)num_sms) {
    compress_small_kernel<<<static_cast<unsigned>(items), kSmallThreads, 0, stream>>>(a);
    return cudaGetLastError();
  }
  const int64_t grid = items < (int64_t)num_sms * 8 ? items : (int64_t)num_sms * 8;
  compress_kernel<<<static_cast<unsigned>(grid), kCompressThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace hattn
