// qprep.cu -- query preparation shared by the three attention branches.
//
// "DeepSeek-V4" atlas, section "Design overview": RMSNorm on the queries
// (replacing QK-Clip); provenance 16: RoPE on the last 64 dims.  Every head
// of every query becomes q~ = RoPE_pos(RMSNorm(q; gamma_q, eps)), stored in
// bf16 once, so the attention kernels start from a plain TMA copy.
//
// One warp per (query, head) row: each lane loads its 16-byte pieces (all
// loads of a row in flight at once), the sum of squares is reduced with
// shuffles, and the normalised, rotated pieces are stored back in place of
// the loaded ones.
#include "common.cuh"
#include "kernels.h"

namespace hattn {

namespace {

constexpr int kQpThreads = 256;
constexpr int kMaxPiecesPerLane = 2;  // D <= 512: 64 pieces of 8 over 32 lanes

__global__ void __launch_bounds__(kQpThreads) qprep_kernel(const __grid_constant__ QPrepArgs a) {
  __shared__ float rc[4][kMaxRopePairs];
  for (int i = threadIdx.x; i < a.r / 2; i += kQpThreads) {
#pragma unroll
    for (int c = 0; c < 4; ++c) rc[c][i] = a.rope.c[c][i];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kQpThreads / 32) + warp;
  if (row >= rows) return;
  const int np = a.D / 8;
  const uint4* src = reinterpret_cast<const uint4*>(a.q + row * a.D);
  uint4 v[kMaxPiecesPerLane];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxPiecesPerLane; ++i) {
    const int pc = lane + 32 * i;
    v[i] = pc < np ? __ldg(src + pc) : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      ss = fmaf(f.x, f.x, ss);
      ss = fmaf(f.y, f.y, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = rsqrtf(ss / static_cast<float>(a.D) + a.eps);
  const int64_t p = a.pos[row / a.H];
  const int d0 = a.D - a.r;
  uint4* dst = reinterpret_cast<uint4*>(a.q_out + row * a.D);
#pragma unroll
  for (int i = 0; i < kMaxPiecesPerLane; ++i) {
    const int pc = lane + 32 * i;
    if (pc >= np) continue;
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
    float y[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      y[2 * e] = f.x * inv * (a.gamma ? a.gamma[pc * 8 + 2 * e] : 1.f);
      y[2 * e + 1] = f.y * inv * (a.gamma ? a.gamma[pc * 8 + 2 * e + 1] : 1.f);
    }
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const int d = pc * 8 + e;
      if (d >= d0) {
        float sn, cs;
        rope_cs(rc, (d - d0) >> 1, p, &sn, &cs);
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
    dst[pc] = u;
  }
}

}  // namespace

cudaError_t launch_qprep(const QPrepArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + kQpThreads / 32 - 1) / (kQpThreads / 32);
  qprep_kernel<<<static_cast<unsigned>(blocks), kQpThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace hattn
