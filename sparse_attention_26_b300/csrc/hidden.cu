// hidden.cu -- compressed entries straight from hidden states.
//
// "Why DeepSeek V4 Stands Apart", section "Core Architectural Innovations":
// the compressor turns per-token KV rows into compressed entries; the
// per-token rows are themselves a projection x_u . W of the hidden states.
// Gate-softmax pooling is a weighted sum of token rows, so pooling the
// hidden states first and projecting once per entry gives the same entry:
//     sum_u a_u (x_u . W) = (sum_u a_u x_u) . W.
// The cache build then reads each hidden state once per window it belongs
// to, never writes per-token KV rows, and runs the projection on one row per
// entry: a quarter of the tokens for CSA, 1/128 for HCA.
//
// Three steps per chunk of entries:
//   1. pool_hidden_kernel: the gate softmax of each window and the pooled row
//      x_bar in fp32, stored as a pair of bf16 rows hi + lo (hi = bf16(x_bar),
//      lo = bf16(x_bar - hi)) that together keep ~16 significant bits;
//   2. two bf16 GEMMs (cuBLASLt, fp32 accumulation and output):
//      Y = hi . W + lo . W;
//   3. entry_norm_rope_kernel: RMSNorm of Y's KV columns, RoPE at the
//      entry's last token, bf16 KV entry; the indexer-key columns in bf16.
#include <cublasLt.h>

#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kPoolThreads = 256;
constexpr int kPoolMaxW = 512;

__global__ void __launch_bounds__(kPoolThreads)
    pool_hidden_kernel(const __grid_constant__ HiddenArgs a, int64_t e0, int64_t ne,
                       __nv_bfloat16* __restrict__ xh, __nv_bfloat16* __restrict__ xl) {
  __shared__ float alpha[kPoolMaxW];
  const int tid = threadIdx.x;
  const int64_t nj = a.j_end - a.j_begin;
  for (int64_t e = blockIdx.x; e < ne; e += gridDim.x) {
    const int64_t flat = e0 + e;  // (sequence, entry) over the whole call
    const int b = static_cast<int>(flat / nj);
    const int64_t j = a.j_begin + flat % nj;
    const int64_t u0 = static_cast<int64_t>(a.m) * (j + 1) - a.w;
    // gate softmax over the window's tokens that exist (warp 0)
    if (tid < 32) {
      float gmax = -INFINITY;
      for (int s = tid; s < a.w; s += 32) {
        const int64_t u = u0 + s;
        if (u >= 0) gmax = fmaxf(gmax, __bfloat162float(a.gate[(int64_t)b * a.L_cap + u]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gmax = fmaxf(gmax, __shfl_xor_sync(0xffffffffu, gmax, o));
      float z = 0.f;
      for (int s = tid; s < a.w; s += 32) {
        const int64_t u = u0 + s;
        const float ex =
            u >= 0 ? __expf(__bfloat162float(a.gate[(int64_t)b * a.L_cap + u]) - gmax) : 0.f;
        alpha[s] = ex;
        z += ex;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
      const float iz = 1.f / z;
      __syncwarp();
      for (int s = tid; s < a.w; s += 32) alpha[s] *= iz;
    }
    __syncthreads();
    // pooled row, 8 columns per thread per pass
    const int s_lo = u0 < 0 ? static_cast<int>(-u0) : 0;
    for (int c = tid * 8; c < a.dm; c += kPoolThreads * 8) {
      float acc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = 0.f;
      const __nv_bfloat16* src = a.x + ((int64_t)b * a.L_cap + u0) * a.dm + c;
      // eight token rows requested at once, then accumulated in order
      for (int s0 = s_lo; s0 < a.w; s0 += 8) {
        uint4 v[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint4* row = reinterpret_cast<const uint4*>(src + (int64_t)(s0 + q) * a.dm);
          v[q] = s0 + q < a.w ? __ldg(row) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float al = s0 + q < a.w ? alpha[s0 + q] : 0.f;
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[q]);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float2 f = __bfloat1622float2(h[k]);
            acc[2 * k] = fmaf(al, f.x, acc[2 * k]);
            acc[2 * k + 1] = fmaf(al, f.y, acc[2 * k + 1]);
          }
        }
      }
      float hi[8], lo[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        hi[k] = bf16_round(acc[k]);
        lo[k] = acc[k] - hi[k];
      }
      uint4 uh, ul;
      uh.x = pack_bf16x2(hi[0], hi[1]);
      uh.y = pack_bf16x2(hi[2], hi[3]);
      uh.z = pack_bf16x2(hi[4], hi[5]);
      uh.w = pack_bf16x2(hi[6], hi[7]);
      ul.x = pack_bf16x2(lo[0], lo[1]);
      ul.y = pack_bf16x2(lo[2], lo[3]);
      ul.z = pack_bf16x2(lo[4], lo[5]);
      ul.w = pack_bf16x2(lo[6], lo[7]);
      *reinterpret_cast<uint4*>(xh + e * a.dm + c) = uh;
      *reinterpret_cast<uint4*>(xl + e * a.dm + c) = ul;
    }
    __syncthreads();  // alpha is rewritten for the next entry
  }
}

// One warp per entry: RMSNorm + RoPE of the KV columns, the indexer key.
__global__ void __launch_bounds__(256)
    entry_norm_rope_kernel(const __grid_constant__ HiddenArgs a, int64_t e0, int64_t ne,
                           const float* __restrict__ Y) {
  __shared__ float rc[4][kMaxRopePairs];
  load_rope_coef(rc, a.rope, a.r);
  const int lane = threadIdx.x & 31;
  const int64_t e = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (e >= ne) return;
  const int64_t nj = a.j_end - a.j_begin;
  const int64_t flat = e0 + e;
  const int b = static_cast<int>(flat / nj);
  const int64_t j = a.j_begin + flat % nj;
  const int P = a.D + a.dI;
  const float* y = Y + e * P;
  float ss = 0.f;
  for (int d = lane; d < a.D; d += 32) ss = fmaf(y[d], y[d], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / static_cast<float>(a.D) + a.eps);
  const int64_t p = static_cast<int64_t>(a.m) * (j + 1) - 1;
  const int d0 = a.D - a.r;
  __nv_bfloat16* kv = a.kv_out + ((int64_t)b * a.N_cap + j) * a.D;
  // lanes take consecutive pairs so that each rotation stays in one lane
  for (int d = 2 * lane; d < a.D; d += 64) {
    float x0 = y[d] * inv * (a.gamma ? a.gamma[d] : 1.f);
    float x1 = y[d + 1] * inv * (a.gamma ? a.gamma[d + 1] : 1.f);
    if (d >= d0) {
      float sn, cs;
      rope_cs(rc, (d - d0) / 2, p, &sn, &cs);
      const float t0 = x0 * cs - x1 * sn;
      x1 = x0 * sn + x1 * cs;
      x0 = t0;
    }
    *reinterpret_cast<uint32_t*>(kv + d) = pack_bf16x2(x0, x1);
  }
  if (a.ik_out) {
    __nv_bfloat16* ik = a.ik_out + ((int64_t)b * a.N_cap + j) * a.dI;
    for (int d = 2 * lane; d < a.dI; d += 64)
      *reinterpret_cast<uint32_t*>(ik + d) = pack_bf16x2(y[a.D + d], y[a.D + d + 1]);
  }
}

// One cuBLASLt handle per host thread (created on first use).
thread_local cublasLtHandle_t t_lt = nullptr;

// Y [ne][P] fp32 (row-major) = X [ne][dm] bf16 . W [dm][P] bf16, added to Y
// when accumulate is set.  In cuBLASLt's column-major terms this is
// Y^T (P x ne) = W^T (P x dm) . X^T (dm x ne), no transposes.
cudaError_t project(const __nv_bfloat16* X, const __nv_bfloat16* W, float* Y, int64_t ne, int dm,
                    int P, bool accumulate, void* lt_ws, size_t lt_ws_bytes, cudaStream_t stream) {
  if (!t_lt && cublasLtCreate(&t_lt) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  cudaError_t err = cudaErrorUnknown;
  const float one = 1.f, beta = accumulate ? 1.f : 0.f;
  cublasLtMatmulHeuristicResult_t heur = {};
  int found = 0;
  if (cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS)
    goto done;
  if (cublasLtMatrixLayoutCreate(&la, CUDA_R_16BF, P, dm, P) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&lb, CUDA_R_16BF, dm, ne, dm) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&lc, CUDA_R_32F, P, ne, P) != CUBLAS_STATUS_SUCCESS)
    goto done;
  if (cublasLtMatmulPreferenceCreate(&pref) != CUBLAS_STATUS_SUCCESS) goto done;
  cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES,
                                       &lt_ws_bytes, sizeof lt_ws_bytes);
  if (cublasLtMatmulAlgoGetHeuristic(t_lt, op, la, lb, lc, lc, pref, 1, &heur, &found) !=
          CUBLAS_STATUS_SUCCESS ||
      found < 1)
    goto done;
  if (cublasLtMatmul(t_lt, op, &one, W, la, X, lb, &beta, Y, lc, Y, lc, &heur.algo, lt_ws,
                     lt_ws_bytes, stream) == CUBLAS_STATUS_SUCCESS)
    err = cudaSuccess;
done:
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (lc) cublasLtMatrixLayoutDestroy(lc);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  return err;
}

}  // namespace

size_t hidden_chunk_entries(int64_t total) { return total < kHiddenChunk ? total : kHiddenChunk; }

size_t hidden_workspace_bytes(int64_t total, int dm, int P) {
  const size_t ce = hidden_chunk_entries(total);
  auto up = [](size_t n) { return (n + 255) / 256 * 256; };
  return 2 * up(ce * dm * 2) + up(ce * P * 4) + kHiddenLtWorkspace;
}

cudaError_t launch_compress_hidden(const HiddenArgs& a, void* ws, int num_sms,
                                   cudaStream_t stream) {
  const int64_t total = static_cast<int64_t>(a.B) * (a.j_end - a.j_begin);
  if (total <= 0) return cudaSuccess;
  const int64_t ce = static_cast<int64_t>(hidden_chunk_entries(total));
  auto up = [](size_t n) { return (n + 255) / 256 * 256; };
  uint8_t* p = static_cast<uint8_t*>(ws);
  __nv_bfloat16* xh = reinterpret_cast<__nv_bfloat16*>(p);
  p += up((size_t)ce * a.dm * 2);
  __nv_bfloat16* xl = reinterpret_cast<__nv_bfloat16*>(p);
  p += up((size_t)ce * a.dm * 2);
  float* Y = reinterpret_cast<float*>(p);
  p += up((size_t)ce * (a.D + a.dI) * 4);
  void* lt_ws = p;
  for (int64_t e0 = 0; e0 < total; e0 += ce) {
    const int64_t ne = (total - e0) < ce ? (total - e0) : ce;
    const int64_t grid = ne < (int64_t)num_sms * 8 ? ne : (int64_t)num_sms * 8;
    pool_hidden_kernel<<<static_cast<unsigned>(grid), kPoolThreads, 0, stream>>>(a, e0, ne, xh,
                                                                               xl);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    e = project(xh, a.W, Y, ne, a.dm, a.D + a.dI, false, lt_ws, kHiddenLtWorkspace, stream);
    if (e != cudaSuccess) return e;
    e = project(xl, a.W, Y, ne, a.dm, a.D + a.dI, true, lt_ws, kHiddenLtWorkspace, stream);
    if (e != cudaSuccess) return e;
    entry_norm_rope_kernel<<<static_cast<unsigned>((ne + 7) / 8), 256, 0, stream>>>(a, e0, ne, Y);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace hattn
