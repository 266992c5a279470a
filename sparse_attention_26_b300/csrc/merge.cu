// merge.cu -- log-sum-exp merges.
//
// combine: the split-KV partials of one branch (each normalised by its own
// softmax sum, with its log-sum-exp) merged in a fixed split order into the
// branch output o and lse (fp32).
//
// merge: the sink-augmented merge of the branches ("DeepSeek-V4" atlas,
// section "Spec sheet / Core block": attention sinks; provenance 16: inverse
// RoPE on the outputs), over every split partial of every branch at once:
//     Z = sum_(b,s) exp(lse_bs) + exp(sink_h),  y = sum_(b,s) exp(lse_bs) o_bs / Z,
//     out = y with its last r dims rotated back by the query position.
// A branch's own normalisation cancels: merging its partials directly equals
// merging its combined output.
//
// A block of 256 threads merges two (query, head) rows, 128 threads each:
// the first warp of a row loads the row's log-sum-exps (one per lane),
// reduces them with shuffles and leaves the weights in shared memory; then
// every thread accumulates 4 columns over all partials (16-byte loads,
// independent across partials).
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kRowThreads = 128;  // threads per row
constexpr int kMergeBlock = 256;  // two rows per block

struct Part {
  const float* o;
  const float* lse;
  int nsplit;
};

// Weights exp(lse_k - log Z) of the row's partials into coef[], with Z the sum
// over the partials (and the sink); run by one warp.  Returns log Z (or -inf
// when the row has no key and no sink).
__device__ __forceinline__ float row_weights(const Part* parts, int nb, int total, int64_t row,
                                             float sink, bool has_sink, float* coef, int lane) {
  float mx = has_sink ? sink : -INFINITY;
  for (int k = lane; k < total; k += 32) {
    int i = 0, s = k;
    while (s >= parts[i].nsplit) s -= parts[i++].nsplit;
    const float v = parts[i].lse[row * parts[i].nsplit + s];
    coef[k] = v;
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (mx == -INFINITY) {
    for (int k = lane; k < total; k += 32) coef[k] = 0.f;
    return -INFINITY;
  }
  float z = (lane == 0 && has_sink) ? __expf(sink - mx) : 0.f;
  for (int k = lane; k < total; k += 32) z += __expf(coef[k] - mx);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
  const float lz = mx + __logf(z);
  for (int k = lane; k < total; k += 32) coef[k] = __expf(coef[k] - lz);
  return lz;
}

// Columns 4*c4 .. 4*c4+3 of the row: sum over the partials of weight x value.
__device__ __forceinline__ float4 row_columns(const Part* parts, int nb, int64_t row, int D,
                                              int c4, const float* coef) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int k = 0;
  for (int i = 0; i < nb; ++i) {
    const float* base = parts[i].o + row * parts[i].nsplit * D + 4 * c4;
#pragma unroll 4
    for (int s = 0; s < parts[i].nsplit; ++s, ++k) {
      const float c = coef[k];
      const float4 v = *reinterpret_cast<const float4*>(base + (int64_t)s * D);
      // an empty split has weight 0 and zero partials
      acc.x = fmaf(c, v.x, acc.x);
      acc.y = fmaf(c, v.y, acc.y);
      acc.z = fmaf(c, v.z, acc.z);
      acc.w = fmaf(c, v.w, acc.w);
    }
  }
  return acc;
}

__global__ void __launch_bounds__(kMergeBlock) combine_kernel(const CombineArgs a) {
  __shared__ float coef[kMergeBlock / kRowThreads][kMaxMergeParts];
  __shared__ float lz_s[kMergeBlock / kRowThreads];
  pdl_trigger();
  pdl_wait();  // the partials of the attention call are complete
  const int half = threadIdx.x / kRowThreads, t = threadIdx.x % kRowThreads;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kMergeBlock / kRowThreads) + half;
  const bool live = row < a.rows;
  Part p{a.part_o, a.part_lse, a.nsplit};
  if (live && t < 32) lz_s[half] = row_weights(&p, 1, a.nsplit, row, 0.f, false, coef[half], t);
  __syncthreads();
  if (!live) return;
  for (int c4 = t; c4 < a.D / 4; c4 += kRowThreads)
    *reinterpret_cast<float4*>(a.o + row * a.D + 4 * c4) = row_columns(&p, 1, row, a.D, c4, coef[half]);
  if (t == 0) a.lse[row] = lz_s[half];
}

__global__ void __launch_bounds__(kMergeBlock) merge_kernel(const __grid_constant__ MergeArgs a) {
  pdl_trigger();
  pdl_wait();  // the branch outputs / partials are complete
  __shared__ float coef[kMergeBlock / kRowThreads][kMaxMergeParts];
  __shared__ float lz_s[kMergeBlock / kRowThreads];
  __shared__ float rc[4][kMaxRopePairs];
  for (int i = threadIdx.x; i < a.r / 2; i += kMergeBlock) {
#pragma unroll
    for (int c = 0; c < 4; ++c) rc[c][i] = a.rope.c[c][i];
  }
  const int half = threadIdx.x / kRowThreads, t = threadIdx.x % kRowThreads;
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kMergeBlock / kRowThreads) + half;
  const bool live = row < rows;
  Part parts[4];
  int total = 0;
  for (int i = 0; i < a.nb; ++i) {
    parts[i] = Part{a.o[i], a.lse[i], a.nsplit[i]};
    total += a.nsplit[i];
  }
  const int h = live ? static_cast<int>(row % a.H) : 0;
  if (live && t < 32)
    lz_s[half] = row_weights(parts, a.nb, total, row, a.sink ? a.sink[h] : 0.f,
                             a.sink != nullptr, coef[half], t);
  __syncthreads();
  if (!live) return;
  const int64_t pos = a.pos[row / a.H];
  const int d0 = a.D - a.r;
  for (int c4 = t; c4 < a.D / 4; c4 += kRowThreads) {
    const float4 acc = row_columns(parts, a.nb, row, a.D, c4, coef[half]);
    float y[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int e = 0; e < 4; e += 2) {
      const int d = 4 * c4 + e;
      if (d >= d0) {
        float sn, cs;
        rope_cs(rc, (d - d0) >> 1, -pos, &sn, &cs);
        const float x0 = y[e], x1 = y[e + 1];
        y[e] = x0 * cs - x1 * sn;
        y[e + 1] = x0 * sn + x1 * cs;
      }
    }
    *reinterpret_cast<uint2*>(a.out + row * a.D + 4 * c4) =
        make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
  }
  if (t == 0 && a.lse_out) a.lse_out[row] = lz_s[half];
}

// The same merge when the row has at most kFastParts partials and a row's
// float4 columns divide the block: every thread issues the loads of all the
// row's partials for its four columns at once (one round of memory latency),
// then weighs them itself from the row's log-sum-exps (read by every thread
// of the row from the same addresses) -- no shared memory, no block barrier.
constexpr int kFastParts = 16;
__global__ void __launch_bounds__(kMergeBlock)
    merge_fast_kernel(const __grid_constant__ MergeArgs a, const int tpr) {
  pdl_trigger();
  pdl_wait();  // the branch outputs / partials are complete
  const int rpb = kMergeBlock / tpr;
  const int t = threadIdx.x % tpr;
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * rpb + threadIdx.x / tpr;
  if (row >= rows) return;
  const int total = a.cum[a.nb];
  float4 v[kFastParts];
  float l[kFastParts];
#pragma unroll
  for (int k = 0; k < kFastParts; ++k) {
    v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    l[k] = -INFINITY;
    if (k < total) {
      const int i = (k >= a.cum[1]) + (k >= a.cum[2]) + (k >= a.cum[3]);
      const int ns = a.nsplit[i];
      const int64_t part = row * ns + (k - a.cum[i]);
      v[k] = __ldcg(reinterpret_cast<const float4*>(a.o[i] + part * a.D) + t);
      l[k] = __ldcg(a.lse[i] + part);
    }
  }
  const int h = static_cast<int>(row % a.H);
  const bool has_sink = a.sink != nullptr;
  const float sink = has_sink ? __ldg(a.sink + h) : -INFINITY;
  float mx = sink;
#pragma unroll
  for (int k = 0; k < kFastParts; ++k) mx = fmaxf(mx, l[k]);
  float y[4] = {0.f, 0.f, 0.f, 0.f};
  float lz = -INFINITY;
  if (mx != -INFINITY) {
    float z = has_sink ? __expf(sink - mx) : 0.f;
#pragma unroll
    for (int k = 0; k < kFastParts; ++k) {
      const float e = __expf(l[k] - mx);  // an empty split: exp(-inf) = 0
      z += e;
      y[0] = fmaf(e, v[k].x, y[0]);
      y[1] = fmaf(e, v[k].y, y[1]);
      y[2] = fmaf(e, v[k].z, y[2]);
      y[3] = fmaf(e, v[k].w, y[3]);
    }
    const float inv = 1.f / z;
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] *= inv;
    lz = mx + __logf(z);
  }
  const int64_t pos = a.pos[row / a.H];
  const int d0 = a.D - a.r;
#pragma unroll
  for (int e = 0; e < 4; e += 2) {
    const int d = 4 * t + e;
    if (d >= d0) {
      float sn, cs;
      rope_cs(a.rope.c, (d - d0) >> 1, -pos, &sn, &cs);
      const float x0 = y[e], x1 = y[e + 1];
      y[e] = x0 * cs - x1 * sn;
      y[e + 1] = x0 * sn + x1 * cs;
    }
  }
  *reinterpret_cast<uint2*>(a.out + row * a.D + 4 * t) =
      make_uint2(pack_bf16x2(y[0], y[1]), pack_bf16x2(y[2], y[3]));
  if (t == 0 && a.lse_out) a.lse_out[row] = lz;
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
  const int per = kMergeBlock / kRowThreads;
  const int64_t blocks = (a.rows + per - 1) / per;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kMergeBlock, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  cfg.attrs = at;
  cfg.numAttrs = add_dependent_attr(at, 0, a.dependent != 0);
  cudaError_t e = cudaLaunchKernelEx(&cfg, combine_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  if (rows <= 0) return cudaSuccess;
  // fast path: few partials per row, and a row's float4 columns divide the block
  const int tpr = a.D / 4;
  const bool fast = a.cum[a.nb] <= kFastParts && a.D % 4 == 0 && tpr <= kMergeBlock &&
                    kMergeBlock % tpr == 0;
  const int per = fast ? kMergeBlock / tpr : kMergeBlock / kRowThreads;
  const int64_t blocks = (rows + per - 1) / per;
  if (blocks > 0x7fffffffll) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kMergeBlock, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute at[1];
  cfg.attrs = at;
  cfg.numAttrs = add_dependent_attr(at, 0, a.dependent != 0);
  cudaError_t e = fast ? cudaLaunchKernelEx(&cfg, merge_fast_kernel, a, tpr)
                       : cudaLaunchKernelEx(&cfg, merge_kernel, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(uint64_t timeout_ns, int* status, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
  return cudaGetLastError();
}

}  // namespace hattn
