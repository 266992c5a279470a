// quant.cu -- E4M3 and MXFP4 rows of the low-precision indexer path.
//
// "DeepSeek-V4" atlas spec sheet, section "Inference efficiency": the
// indexer's QK path runs in low precision.  Here the keys are stored as FP8
// E4M3 codes with one fp32 scale per row: code_i = e4m3(x_i * 448 / amax),
// decoded as code_i * amax / 448.  The E4M3 kernel quantises whole bf16 rows
// (cache builds); the compressor quantises each new entry as it writes it and
// the indexer quantises its query rows in shared memory, all through the
// same row scaling (e4m3_row).  The pages' own format, MXFP4, has a kernel
// for whole rows below (keys and queries in that format for the scoring
// kernel to read).
//
// E4M3: one warp per row; lane l covers elements 4l, 4l+1, 4l+2, 4l+3 of each
// 128-element span, so a row is read twice from L1/L2-resident lines (once
// for the largest magnitude, once for the codes) and written once.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kQuantThreads = 256;

__global__ void __launch_bounds__(kQuantThreads)
    quantize_e4m3_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int n,
                         uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (kQuantThreads / 32);
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * (kQuantThreads / 32) + (threadIdx.x >> 5);
       row < rows; row += warps) {
    const __nv_bfloat16* xr = x + row * n;
    float amax = 0.f;
    for (int i = lane * 4; i < n; i += 128) {
      const uint2 u = *reinterpret_cast<const uint2*>(xr + i);
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      amax = fmaxf(amax, fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const E4m3Row s = e4m3_row(amax);
    for (int i = lane * 4; i < n; i += 128) {
      const uint2 u = *reinterpret_cast<const uint2*>(xr + i);
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      const float v[4] = {f0.x, f0.y, f1.x, f1.y};
      *reinterpret_cast<uint32_t*>(codes + row * n + i) = e4m3x4(v, s.inv);
    }
    if (lane == 0) scales[row] = s.scale;
  }
}

// MXFP4 rows (OCP Microscaling: E2M1 elements, one E8M0 scale per 32
// consecutive elements).  The block scale is X = 2^(floor(log2 amax) - 2),
// the largest E2M1 exponent being 2, so amax / X lies in [4, 8); its
// exponent is read off amax's fp32 exponent field and clamped to [-127, 125]
// (the lower end also covers zero and subnormal blocks).  x / X is exact in
// fp32, and the hardware conversion rounds it to the nearest E2M1 value
// (ties to even) saturating at +-6.  Element 2i goes to the low nibble of
// byte i; a zero result is stored as +0.
//
// A warp takes kMxRows rows at a time and issues all their loads before it
// reduces any of them, so an SM keeps enough bytes in flight to cover HBM
// latency; lane l holds elements 4l..4l+3 of each 128-element span, so lanes
// 8g..8g+7 hold block g of the span and reduce its amax among themselves.
// n is a multiple of 32, so a span's blocks are whole.
constexpr int kMxRows = 8;

__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\t"
      "cvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// kN > 0: rows of exactly kN elements (row offsets become immediates); kN = 0:
// any n, a multiple of 32.
// kMapped: row r of the call is row (r / nj) * ncap + j0 + r % nj of x,
// codes and scales (an entry range [j0, j0 + nj) of every sequence of a
// [B][ncap][n] cache); else row r is row r (the offsets of a group's rows
// are then immediates).
template <int kN, bool kMapped>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_mxfp4_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int n_arg,
                          uint8_t* __restrict__ codes, uint8_t* __restrict__ scales, int64_t nj,
                          int64_t j0, int64_t ncap) {
  const int n = kN > 0 ? kN : n_arg;
  const int lane = threadIdx.x & 31;
  const int64_t warp = static_cast<int64_t>(blockIdx.x) * (kQuantThreads / 32) + (threadIdx.x >> 5);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kQuantThreads / 32) * kMxRows;
  for (int64_t row0 = warp * kMxRows; row0 < rows; row0 += stride) {
    // rows of this group that exist (warp-uniform); row k sits k * n
    // elements past the group's first
    const int nk = rows - row0 < kMxRows ? static_cast<int>(rows - row0) : kMxRows;
    int64_t rk[kMxRows];  // the rows' places: one division per group when mapped
    if (kMapped) {
      int64_t q = row0 / nj, rem = row0 - q * nj;
#pragma unroll
      for (int k = 0; k < kMxRows; ++k) {
        rk[k] = q * ncap + j0 + rem;
        if (++rem == nj) {
          rem = 0;
          ++q;
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < kMxRows; ++k) rk[k] = row0 + k;
    }
    for (int base = 0; base < n; base += 128) {
      const int i = base + lane * 4;
      const bool in = i < n;
      uint2 u[kMxRows];
#pragma unroll
      for (int k = 0; k < kMxRows; ++k) {
        u[k] = make_uint2(0u, 0u);
        if (in && k < nk) u[k] = *reinterpret_cast<const uint2*>(x + rk[k] * n + i);
      }
#pragma unroll
      for (int k = 0; k < kMxRows; ++k) {
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[k].x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[k].y));
        float amax = fmaxf(fmaxf(fabsf(f0.x), fabsf(f0.y)), fmaxf(fabsf(f1.x), fabsf(f1.y)));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        int se = static_cast<int>((__float_as_uint(amax) >> 23) & 0xffu) - 127 - 2;
        se = se < -127 ? -127 : se;
        const float inv = __uint_as_float(static_cast<uint32_t>(127 - se) << 23);  // 2^-se
        if (in && k < nk) {
          uint32_t w = e2m1x2(__fmul_rn(f0.x, inv), __fmul_rn(f0.y, inv)) |
                       (e2m1x2(__fmul_rn(f1.x, inv), __fmul_rn(f1.y, inv)) << 8);
          const uint32_t mag = w & 0x7777u;
          w = mag | (w & ((mag + 0x7777u) & 0x8888u));  // drop the sign of zero nibbles
          *reinterpret_cast<uint16_t*>(codes + rk[k] * (n / 2) + i / 2) = static_cast<uint16_t>(w);
          if ((lane & 7) == 0) scales[rk[k] * (n / 32) + i / 32] = static_cast<uint8_t>(se + 127);
        }
      }
    }
  }
}

// E4M3 rows of exactly 128 (indexer keys): one warp-wide span per row, and a
// warp takes kMxRows rows at a time with all their loads issued first, as
// the MXFP4 kernel does.
__global__ void __launch_bounds__(kQuantThreads)
    quantize_e4m3_rows128_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                 uint8_t* __restrict__ codes, float* __restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = static_cast<int64_t>(blockIdx.x) * (kQuantThreads / 32) + (threadIdx.x >> 5);
  const int64_t stride = static_cast<int64_t>(gridDim.x) * (kQuantThreads / 32) * kMxRows;
  for (int64_t row0 = warp * kMxRows; row0 < rows; row0 += stride) {
    const int nk = rows - row0 < kMxRows ? static_cast<int>(rows - row0) : kMxRows;
    const __nv_bfloat16* xg = x + row0 * 128 + lane * 4;
    uint8_t* cg = codes + row0 * 128 + lane * 4;
    uint2 u[kMxRows];
#pragma unroll
    for (int k = 0; k < kMxRows; ++k) {
      u[k] = make_uint2(0u, 0u);
      if (k < nk) u[k] = *reinterpret_cast<const uint2*>(xg + k * 128);
    }
#pragma unroll
    for (int k = 0; k < kMxRows; ++k) {
      const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[k].x));
      const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[k].y));
      const float v[4] = {f0.x, f0.y, f1.x, f1.y};
      float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      const E4m3Row sc = e4m3_row(amax);
      if (k < nk) {
        *reinterpret_cast<uint32_t*>(cg + k * 128) = e4m3x4(v, sc.inv);
        if (lane == 0) scales[row0 + k] = sc.scale;
      }
    }
  }
}

}  // namespace

cudaError_t launch_quantize_mxfp4(const __nv_bfloat16* x, int64_t rows, int n, uint8_t* codes,
                                  uint8_t* scales, int num_sms, cudaStream_t stream, int64_t nj,
                                  int64_t j0, int64_t ncap) {
  if (rows <= 0) return cudaSuccess;
  // one wave of resident CTAs, each striding over groups of rows
  const bool mapped = nj > 0;
  auto kernel = n == 128 ? (mapped ? quantize_mxfp4_kernel<128, true>
                                   : quantize_mxfp4_kernel<128, false>)
                         : (mapped ? quantize_mxfp4_kernel<0, true> : quantize_mxfp4_kernel<0, false>);
  int resident = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, kernel, kQuantThreads, 0);
  if (e != cudaSuccess) return e;
  const int64_t per_cta = (kQuantThreads / 32) * kMxRows;
  const int64_t want = (rows + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(num_sms) * (resident > 0 ? resident : 1);
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  if (!mapped) {  // plain rows
    nj = rows;
    j0 = 0;
    ncap = rows;
  }
  kernel<<<grid, kQuantThreads, 0, stream>>>(x, rows, n, codes, scales, nj, j0, ncap);
  return cudaGetLastError();
}

cudaError_t launch_quantize_e4m3(const __nv_bfloat16* x, int64_t rows, int n, uint8_t* codes,
                                 float* scales, int num_sms, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  if (n == 128) {  // one wave of resident CTAs, each striding over groups of rows
    int resident = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
        &resident, quantize_e4m3_rows128_kernel, kQuantThreads, 0);
    if (e != cudaSuccess) return e;
    const int64_t per_cta = (kQuantThreads / 32) * kMxRows;
    const int64_t want = (rows + per_cta - 1) / per_cta;
    const int64_t cap = static_cast<int64_t>(num_sms) * (resident > 0 ? resident : 1);
    const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
    quantize_e4m3_rows128_kernel<<<grid, kQuantThreads, 0, stream>>>(x, rows, codes, scales);
    return cudaGetLastError();
  }
  const int64_t per_cta = kQuantThreads / 32;
  const int64_t want = (rows + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  quantize_e4m3_kernel<<<grid, kQuantThreads, 0, stream>>>(x, rows, n, codes, scales);
  return cudaGetLastError();
}

}  // namespace hattn
