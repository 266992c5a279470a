// quant.cu -- E4M3 rows of the low-precision indexer path.
//
// "DeepSeek-V4" atlas spec sheet, section "Inference efficiency": the
// indexer's QK path runs in low precision.  Here the keys are stored as FP8
// E4M3 codes with one fp32 scale per row: code_i = e4m3(x_i * 448 / amax),
// decoded as code_i * amax / 448.  This kernel quantises whole bf16 rows
// (cache builds); the compressor quantises each new entry as it writes it and
// the indexer quantises its query rows in shared memory, all through the
// same row scaling (e4m3_row).
//
// One warp per row; lane l covers elements 4l, 4l+1, 4l+2, 4l+3 of each
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

}  // namespace

cudaError_t launch_quantize_e4m3(const __nv_bfloat16* x, int64_t rows, int n, uint8_t* codes,
                                 float* scales, int num_sms, cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int64_t per_cta = kQuantThreads / 32;
  const int64_t want = (rows + per_cta - 1) / per_cta;
  const int64_t cap = static_cast<int64_t>(num_sms) * 8;
  const unsigned grid = static_cast<unsigned>(want < cap ? want : cap);
  quantize_e4m3_kernel<<<grid, kQuantThreads, 0, stream>>>(x, rows, n, codes, scales);
  return cudaGetLastError();
}

}  // namespace hattn
