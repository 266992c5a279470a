// qprep.cu -- query preparation shared by the three attention branches, and
// the normalised, roped SWA keys of the fused attention.
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

// One row of D bf16 values: RMSNorm (gamma, eps), RoPE of the last r dims at
// position p, one bf16 rounding; src == nullptr writes a zero row.  Called
// by a whole warp, each lane holding up to two 16-byte pieces.
__device__ __forceinline__ void norm_rope_row(const __nv_bfloat16* src, __nv_bfloat16* dst_row,
                                              int D, int r, int64_t p, const float* gamma,
                                              float eps, const float (*rc)[kMaxRopePairs],
                                              int lane) {
  const int np = D / 8;
  uint4* dst = reinterpret_cast<uint4*>(dst_row);
  if (!src) {
    for (int pc = lane; pc < np; pc += 32) dst[pc] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  uint4 v[kMaxPiecesPerLane];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxPiecesPerLane; ++i) {
    const int pc = lane + 32 * i;
    v[i] = pc < np ? __ldg(s4 + pc) : make_uint4(0, 0, 0, 0);
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
  const float inv = rsqrtf(ss / static_cast<float>(D) + eps);
  const int d0 = D - r;
#pragma unroll
  for (int i = 0; i < kMaxPiecesPerLane; ++i) {
    const int pc = lane + 32 * i;
    if (pc >= np) continue;
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v[i]);
    float y[8];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      y[2 * e] = f.x * inv * (gamma ? gamma[pc * 8 + 2 * e] : 1.f);
      y[2 * e + 1] = f.y * inv * (gamma ? gamma[pc * 8 + 2 * e + 1] : 1.f);
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

__global__ void __launch_bounds__(kQpThreads) qprep_kernel(const __grid_constant__ QPrepArgs a) {
  __shared__ float rc[4][kMaxRopePairs];
  pdl_trigger();
  load_rope_coef(rc, a.rope, a.r);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kQpThreads / 32) + warp;
  if (row >= rows) return;
  norm_rope_row(a.q + row * a.D, a.q_out + row * a.D, a.D, a.r, a.pos[row / a.H], a.gamma, a.eps,
                rc, lane);
}

// "Why DeepSeek V4 Stands Apart", section "Core Architectural Innovations":
// SWA attends to the most recent 128 tokens, read here as raw tokens in the
// same normalised, roped space as the compressed entries.  Row (b, t, j) of
// the key buffer is raw token u = pos[b][t] - W + 1 + j, RMSNorm'd with
// gamma_kv and roped at u; tokens outside [0, L_cap) give zero rows.
__global__ void __launch_bounds__(kQpThreads)
    swa_keys_kernel(const __grid_constant__ SwaKeysArgs a) {
  __shared__ float rc[4][kMaxRopePairs];
  pdl_trigger();
  load_rope_coef(rc, a.rope, a.r);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.W;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (kQpThreads / 32) + warp;
  if (row >= rows) return;
  const int64_t bt = row / a.W;
  const int j = static_cast<int>(row - bt * a.W);
  const int64_t b = bt / a.T;
  const int64_t u = static_cast<int64_t>(a.pos[bt]) - a.W + 1 + j;
  // in a ring of the last `ring` tokens (a power of two), token u is row u mod ring
  const bool exists = u >= 0 && (a.ring > 0 || u < a.L_cap);
  const int64_t ru = a.ring > 0 ? (u & (a.ring - 1)) : u;
  norm_rope_row(exists ? a.kv_raw + (b * a.L_cap + ru) * a.D : nullptr, a.kv_w + row * a.D, a.D,
                a.r, u, a.gamma, a.eps, rc, lane);
}

}  // namespace

cudaError_t launch_qprep(const QPrepArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.H;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + kQpThreads / 32 - 1) / (kQpThreads / 32);
  qprep_kernel<<<static_cast<unsigned>(blocks), kQpThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_swa_keys(const SwaKeysArgs& a, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(a.B) * a.T * a.W;
  if (rows <= 0) return cudaSuccess;
  const int64_t blocks = (rows + kQpThreads / 32 - 1) / (kQpThreads / 32);
  swa_keys_kernel<<<static_cast<unsigned>(blocks), kQpThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace hattn
