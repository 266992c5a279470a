// merge.cu -- log-sum-exp merges.
//
// combine: the split-KV partials of one branch (each normalised by its own
// softmax sum, with its log-sum-exp) merged in a fixed split order into the
// branch output o (bf16) and lse (fp32).
//
// merge: the sink-augmented merge of the branch outputs ("DeepSeek-V4" atlas,
// section "Spec sheet / Core block": attention sinks; provenance 16: inverse
// RoPE on the outputs):
//     Z = sum_i exp(lse_i) + exp(sink_h),  y = sum_i exp(lse_i) o_i / Z,
//     out = y with its last r dims rotated back by the query position.
// Both are HBM-bound elementwise passes: one warp per (query, head) row,
// 16-byte vector loads and stores.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kRowsPerBlock = 8;

__global__ void __launch_bounds__(256) combine_kernel(const CombineArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + warp;
  if (row >= a.rows) return;
  const float* pl = a.part_lse + row * a.nsplit;
  float mx = -INFINITY;
  for (int s = 0; s < a.nsplit; ++s) mx = fmaxf(mx, pl[s]);
  __nv_bfloat16* o = a.o + row * a.D;
  if (mx == -INFINITY) {
    for (int d = lane * 8; d < a.D; d += 256) *reinterpret_cast<uint4*>(o + d) = make_uint4(0, 0, 0, 0);
    if (lane == 0) a.lse[row] = -INFINITY;
    return;
  }
  float z = 0.f;
  for (int s = 0; s < a.nsplit; ++s) z += __expf(pl[s] - mx);
  const float iz = 1.f / z;
  for (int d = lane * 8; d < a.D; d += 256) {
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int s = 0; s < a.nsplit; ++s) {
      const float c = __expf(pl[s] - mx) * iz;
      if (c == 0.f) continue;
      const float4* src = reinterpret_cast<const float4*>(a.part_o + (row * a.nsplit + s) * a.D + d);
      const float4 v0 = src[0], v1 = src[1];
      acc[0] = fmaf(c, v0.x, acc[0]);
      acc[1] = fmaf(c, v0.y, acc[1]);
      acc[2] = fmaf(c, v0.z, acc[2]);
      acc[3] = fmaf(c, v0.w, acc[3]);
      acc[4] = fmaf(c, v1.x, acc[4]);
      acc[5] = fmaf(c, v1.y, acc[5]);
      acc[6] = fmaf(c, v1.z, acc[6]);
      acc[7] = fmaf(c, v1.w, acc[7]);
    }
    uint4 u;
    u.x = pack_bf16x2(acc[0], acc[1]);
    u.y = pack_bf16x2(acc[2], acc[3]);
    u.z = pack_bf16x2(acc[4], acc[5]);
    u.w = pack_bf16x2(acc[6], acc[7]);
    *reinterpret_cast<uint4*>(o + d) = u;
  }
  if (lane == 0) a.lse[row] = mx + __logf(z);
}

__global__ void __launch_bounds__(256) merge_kernel(const MergeArgs a) {
  __shared__ double theta[256];
  for (int i = threadIdx.x; i < a.r / 2; i += blockDim.x)
    theta[i] = pow(static_cast<double>(a.rope_base), -2.0 * i / static_cast<double>(a.r));
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + warp;
  if (row >= rows) return;
  const int h = static_cast<int>(row % a.H);
  const int64_t bt = row / a.H;
  float lse_b[4];
  float mx = a.sink ? a.sink[h] : -INFINITY;
  for (int i = 0; i < a.nb; ++i) {
    lse_b[i] = a.lse[i][row];
    mx = fmaxf(mx, lse_b[i]);
  }
  __nv_bfloat16* out = a.out + row * a.D;
  if (mx == -INFINITY) {
    for (int d = lane * 8; d < a.D; d += 256) *reinterpret_cast<uint4*>(out + d) = make_uint4(0, 0, 0, 0);
    if (lane == 0 && a.lse_out) a.lse_out[row] = -INFINITY;
    return;
  }
  float z = a.sink ? __expf(a.sink[h] - mx) : 0.f;
  for (int i = 0; i < a.nb; ++i) z += __expf(lse_b[i] - mx);
  const float lz = mx + __logf(z);
  float coef[4];
  for (int i = 0; i < a.nb; ++i) coef[i] = __expf(lse_b[i] - lz);
  const int64_t p = a.pos[bt];
  const int d0 = a.D - a.r;
  for (int d = lane * 8; d < a.D; d += 256) {
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = 0.f;
    for (int i = 0; i < a.nb; ++i) {
      if (coef[i] == 0.f) continue;
      const uint4 u = *reinterpret_cast<const uint4*>(a.o[i] + row * a.D + d);
      const __nv_bfloat162* hv = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(hv[e]);
        y[2 * e] = fmaf(coef[i], f.x, y[2 * e]);
        y[2 * e + 1] = fmaf(coef[i], f.y, y[2 * e + 1]);
      }
    }
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const int dd = d + e;
      if (dd >= d0) {
        float sn, cs;
        rope_sincos(theta[(dd - d0) >> 1], -p, &sn, &cs);
        const float x0 = y[e], x1 = y[e + 1];
        y[e] = x0 * cs - x1 * sn;
        y[e + 1] = x0 * sn + x1 * cs;
      }
    }
    uint4 u;
    u.x = pack_bf16x2(y[0], y[1]);
    u.y = pack_bf16x2(y[2], y[3]);
    u.z = pack_bf16x2(y[4], y[5]);
    u.w = pack_bf16x2(y[6], y[7]);
    *reinterpret_cast<uint4*>(out + d) = u;
  }
  if (lane == 0 && a.lse_out) a.lse_out[row] = lz;
}

// One thread waits on an mbarrier that nothing arrives on; the bounded wait
// gives up after `timeout_ns` and records the timeout in the status word.
__global__ void wait_selftest_kernel(uint64_t timeout_ns, int* status) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
    mbar_wait(smem_u32(&bar), 0, nullptr, status, timeout_ns, 28);
  }
}

}  // namespace

cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream) {
  if (a.rows <= 0) return cudaSuccess;
  const int64_t blocks = (a.rows + kRowsPerBlock - 1) / kRowsPerBlock;
  combine_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  merge_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, int* status, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
  return cudaGetLastError();
}

}  // namespace hattn
