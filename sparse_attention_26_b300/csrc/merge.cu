// merge.cu -- log-sum-exp merges.
//
// combine: the split-KV partials of one branch (each normalised by its own
// softmax sum, with its log-sum-exp) merged in a fixed split order into the
// branch output o and lse (fp32).
//
// merge: the sink-augmented merge of the branch outputs ("DeepSeek-V4" atlas,
// section "Spec sheet / Core block": attention sinks; provenance 16: inverse
// RoPE on the outputs):
//     Z = sum_i exp(lse_i) + exp(sink_h),  y = sum_i exp(lse_i) o_i / Z,
//     out = y with its last r dims rotated back by the query position.
// Both are HBM-bound elementwise passes: one thread per 8 columns of a
// (query, head) row, 16-byte vector loads and stores.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kMergeThreads = 256;

// One thread per (row, 8-column group): every load of a row's partials is
// independent, so a launch keeps thousands of 16-byte loads in flight.
__global__ void __launch_bounds__(kMergeThreads) combine_kernel(const CombineArgs a) {
  const int groups = a.D / 8;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x;
  const int64_t row = gid / groups;
  const int c8 = static_cast<int>(gid - row * groups);
  if (row >= a.rows) return;
  const float* pl = a.part_lse + row * a.nsplit;
  float mx = -INFINITY;
  for (int s = 0; s < a.nsplit; ++s) mx = fmaxf(mx, pl[s]);
  float* o = a.o + row * a.D + c8 * 8;
  if (mx == -INFINITY) {
    reinterpret_cast<float4*>(o)[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    reinterpret_cast<float4*>(o)[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (c8 == 0) a.lse[row] = -INFINITY;
    return;
  }
  float z = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  const float* po = a.part_o + row * a.nsplit * a.D + c8 * 8;
#pragma unroll 4
  for (int s = 0; s < a.nsplit; ++s) {
    const float c = __expf(pl[s] - mx);
    z += c;
    const float4 v0 = *reinterpret_cast<const float4*>(po + (int64_t)s * a.D);
    const float4 v1 = *reinterpret_cast<const float4*>(po + (int64_t)s * a.D + 4);
    // an empty split has weight 0 and zero partials
    acc[0] = fmaf(c, v0.x, acc[0]);
    acc[1] = fmaf(c, v0.y, acc[1]);
    acc[2] = fmaf(c, v0.z, acc[2]);
    acc[3] = fmaf(c, v0.w, acc[3]);
    acc[4] = fmaf(c, v1.x, acc[4]);
    acc[5] = fmaf(c, v1.y, acc[5]);
    acc[6] = fmaf(c, v1.z, acc[6]);
    acc[7] = fmaf(c, v1.w, acc[7]);
  }
  const float iz = 1.f / z;
  reinterpret_cast<float4*>(o)[0] = make_float4(acc[0] * iz, acc[1] * iz, acc[2] * iz, acc[3] * iz);
  reinterpret_cast<float4*>(o)[1] = make_float4(acc[4] * iz, acc[5] * iz, acc[6] * iz, acc[7] * iz);
  if (c8 == 0) a.lse[row] = mx + __logf(z);
}

// One thread per (row, 8-column group), as above.
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ MergeArgs a) {
  __shared__ float rc[4][kMaxRopePairs];
  for (int i = threadIdx.x; i < a.r / 2; i += kMergeThreads) {
#pragma unroll
    for (int c = 0; c < 4; ++c) rc[c][i] = a.rope.c[c][i];
  }
  __syncthreads();
  const int groups = a.D / 8;
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * kMergeThreads + threadIdx.x;
  const int64_t row = gid / groups;
  const int c8 = static_cast<int>(gid - row * groups);
  if (row >= rows) return;
  const int h = static_cast<int>(row % a.H);
  const int64_t bt = row / a.H;
  float lse_b[4];
  float mx = a.sink ? a.sink[h] : -INFINITY;
  for (int i = 0; i < a.nb; ++i) {
    lse_b[i] = a.lse[i][row];
    mx = fmaxf(mx, lse_b[i]);
  }
  const int d = c8 * 8;
  __nv_bfloat16* out = a.out + row * a.D + d;
  if (mx == -INFINITY) {
    *reinterpret_cast<uint4*>(out) = make_uint4(0, 0, 0, 0);
    if (c8 == 0 && a.lse_out) a.lse_out[row] = -INFINITY;
    return;
  }
  float z = a.sink ? __expf(a.sink[h] - mx) : 0.f;
  for (int i = 0; i < a.nb; ++i) z += __expf(lse_b[i] - mx);
  const float lz = mx + __logf(z);
  float y[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) y[e] = 0.f;
  for (int i = 0; i < a.nb; ++i) {
    const float coef = __expf(lse_b[i] - lz);
    if (coef == 0.f) continue;  // an empty branch (its o is not read)
    const float4 v0 = *reinterpret_cast<const float4*>(a.o[i] + row * a.D + d);
    const float4 v1 = *reinterpret_cast<const float4*>(a.o[i] + row * a.D + d + 4);
    y[0] = fmaf(coef, v0.x, y[0]);
    y[1] = fmaf(coef, v0.y, y[1]);
    y[2] = fmaf(coef, v0.z, y[2]);
    y[3] = fmaf(coef, v0.w, y[3]);
    y[4] = fmaf(coef, v1.x, y[4]);
    y[5] = fmaf(coef, v1.y, y[5]);
    y[6] = fmaf(coef, v1.z, y[6]);
    y[7] = fmaf(coef, v1.w, y[7]);
  }
  const int d0 = a.D - a.r;
  const int64_t p = a.pos[bt];
#pragma unroll
  for (int e = 0; e < 8; e += 2) {
    const int dd = d + e;
    if (dd >= d0) {
      float sn, cs;
      rope_cs(rc, (dd - d0) >> 1, -p, &sn, &cs);
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
  *reinterpret_cast<uint4*>(out) = u;
  if (c8 == 0 && a.lse_out) a.lse_out[row] = lz;
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
  const int64_t blocks = (a.rows * (a.D / 8) + kMergeThreads - 1) / kMergeThreads;
  combine_kernel<<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows * (a.D / 8) + kMergeThreads - 1) / kMergeThreads;
  merge_kernel<<<static_cast<unsigned>(blocks), kMergeThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, int* status, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
  return cudaGetLastError();
}

}  // namespace hattn
