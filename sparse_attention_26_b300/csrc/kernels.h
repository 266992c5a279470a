// kernels.h -- internal launch interface between the C ABI layer (abi.cu)
// and the kernels.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace hattn {

// Appends the programmatic-serialization attribute to attrs[n] when
// `dependent` (the call's HATTN_LAUNCH_DEPENDENT flag) is set: the kernel
// may then start while the previous kernel in its stream still runs, and
// waits (griddepcontrol.wait) before reading what that kernel writes.
// Returns the new attribute count.
int add_dependent_attr(cudaLaunchAttribute* attrs, int n, bool dependent);

// ------------------------------------------------------------ compressor
struct CompressArgs {
  const __nv_bfloat16* kv_raw;  // [B][L_cap][D]
  const __nv_bfloat16* ik_raw;  // [B][L_cap][dI] or null (no indexer key)
  const __nv_bfloat16* gate;    // [B][L_cap]
  const float* gamma;           // [D] or null
  __nv_bfloat16* kv_out;        // [B][N_cap][D]
  __nv_bfloat16* ik_out;        // [B][N_cap][dI] or null
  uint8_t* ik8_out;             // [B][N_cap][dI] E4M3 codes of the indexer key, or null
  float* ik_scale_out;          // [B][N_cap] their row scales (with ik8_out)
  uint8_t* ik4_out;             // [B][N_cap][dI/2] MXFP4 codes of the indexer key, or null
  uint8_t* ik4_scale_out;       // [B][N_cap][dI/32] their E8M0 block scales (with ik4_out)
  int B, D, dI, m, w, r;
  int64_t L_cap, N_cap, j_begin, j_end;
  int64_t ring;                 // 0: token u in row u; else row u mod ring (L_cap == ring)
  float eps;
  RopeCoef rope;
};
cudaError_t launch_compress(const CompressArgs& a, int num_sms, cudaStream_t stream);

// ------------------------------------------------------------ indexer score
// Bins of the selection's first radix pass: the top 11 bits of a score's
// order-preserving key.
constexpr int kSelBins = 2048;

struct IndexerArgs {
  const float* w;        // [B][T][HI]
  const int32_t* pos;    // [B][T]
  float* scores;         // [B][T][N_cap]
  int* status;
  int B, T, HI, dI, m;
  int G;                 // queries per group (B operand rows = G*HI, padded to NQ)
  int NQ;                // MMA N
  int KC;                // 64-wide K chunks of the bf16 operands
  int stages;
  int nacc;              // tensor-memory accumulators in flight (2, 4 or 8)
  int groups_per_seq;    // ceil(T / G)
  int nblk;              // ceil(N_cap / 128)
  int64_t fresh_from;    // entries >= this may be written by the previous kernel (-1: any)
  int64_t N_cap;
  int64_t total_slots;   // B * groups_per_seq * nblk
  int dependent;         // launched as a programmatic dependent
  // Folded first pass of the selection (one query per group, each CTA's
  // slots within two rows): CTA c writes the 2,048-bin histogram of the top
  // 11 key bits of its visible scores, 16-bit counts, to
  // hist_part[c][0][.] for the row of its first slot and hist_part[c][1][.]
  // for the row of its last slot when that differs.  nullptr: no histograms.
  uint16_t* hist_part;
};
struct IndexerPlan {
  int G, NQ, KC, stages, nacc, tmem_cols;
  size_t smem_bytes;
};
// Key formats: bf16 keys and queries; E4M3 keys (dI = 128, one 128-byte row
// each) with the queries quantised in the kernel; MXFP4 keys (dI = 128: 64
// code bytes and 4 E8M0 scale bytes each) decoded to bf16 in shared memory,
// with the queries taken through the same round trip in the kernel.
enum IndexerKeys { kIdxKeysBf16 = 0, kIdxKeysE4m3 = 1, kIdxKeysMx4 = 2 };
bool plan_indexer(int T, int HI, int dI, int keys, bool fold, IndexerPlan* p);
// tm_ks: the FP8 keys' row scales [B][N_cap] fp32, boxes of 128 (FP8); the
// MXFP4 keys' scales as [B][N_cap / 4][16] bytes, boxes {16, 32} (MXFP4).
cudaError_t launch_indexer_score(const CUtensorMap& tm_ik, const CUtensorMap& tm_iq,
                                 const CUtensorMap& tm_ks, const IndexerArgs& a,
                                 const IndexerPlan& p, int keys, int grid, cudaStream_t stream);

// ------------------------------------------------------------ entries from hidden states
struct HiddenArgs {
  const __nv_bfloat16* x;       // [B][L_cap][dm] hidden states
  const __nv_bfloat16* W;       // [dm][D + dI]: KV columns, then indexer-key columns
  const __nv_bfloat16* gate;    // [B][L_cap]
  const float* gamma;           // [D] or null
  __nv_bfloat16* kv_out;        // [B][N_cap][D]
  __nv_bfloat16* ik_out;        // [B][N_cap][dI] or null (dI == 0)
  int B, dm, D, dI, m, w, r;
  int64_t L_cap, N_cap, j_begin, j_end;
  float eps;
  RopeCoef rope;
};
constexpr int64_t kHiddenChunk = 16384;          // entries pooled and projected per pass
size_t hidden_chunk_entries(int64_t total);
size_t hidden_part_bytes(size_t ce, int dm);      // one pooled part (hi or lo) of a chunk
size_t hidden_workspace_bytes(int64_t total, int dm, int P);
int hidden_ik_cols(int dI);                       // accumulator columns of the indexer-key group
// tm_ah / tm_al: the pooled parts [chunk entries][dm] bf16 in the workspace
// (boxes {64, 128}); tm_w: W [dm][D + dI] (boxes {64 columns, 64 rows});
// all 128-byte swizzled.
cudaError_t launch_compress_hidden(const HiddenArgs& a, void* ws, int num_sms,
                                   const CUtensorMap& tm_ah, const CUtensorMap& tm_al,
                                   const CUtensorMap& tm_w, int* status, cudaStream_t stream);
// Both caches in one read of the hidden states: ac the CSA pass (C(4, 8),
// entries [0, ac.j_end) per sequence, dI > 0 allowed), ah the HCA pass
// (C(128, 128), entries [0, ah.j_end), dI = 0), sharing x, dm and D.
// Workspace (hidden_pair_workspace_bytes): the CSA parts of one pass, then
// the HCA parts of every entry; tm_ch/tm_cl and tm_hh/tm_hl map them,
// tm_wc / tm_wh the two projections.
size_t hidden_pair_workspace_bytes(int B, int64_t nc, int64_t nh, int dm);
cudaError_t launch_compress_hidden_pair(const HiddenArgs& ac, const HiddenArgs& ah, void* ws,
                                        int num_sms, const CUtensorMap& tm_ch,
                                        const CUtensorMap& tm_cl, const CUtensorMap& tm_wc,
                                        const CUtensorMap& tm_hh, const CUtensorMap& tm_hl,
                                        const CUtensorMap& tm_wh, int* status,
                                        cudaStream_t stream);

// ------------------------------------------------------------ E4M3 rows
// rows x n bf16 -> E4M3 codes [rows][n] and row scales [rows]; n % 4 == 0.
cudaError_t launch_quantize_e4m3(const __nv_bfloat16* x, int64_t rows, int n, uint8_t* codes,
                                 float* scales, int num_sms, cudaStream_t stream);

// ------------------------------------------------------------ MXFP4 rows
// rows x n bf16 -> E2M1 codes [rows][n/2] (element 2i in the low nibble of
// byte i) and E8M0 block scales [rows][n/32]; n % 32 == 0.
cudaError_t launch_quantize_mxfp4(const __nv_bfloat16* x, int64_t rows, int n, uint8_t* codes,
                                  uint8_t* scales, int num_sms, cudaStream_t stream, int64_t nj = 0,
                                  int64_t j0 = 0, int64_t ncap = 0);

// ------------------------------------------------------------ top-k select
struct TopkArgs {
  const float* scores;   // [rows][N_cap]
  const int32_t* pos;    // [rows]
  int32_t* idx;          // [rows][k]
  // cluster path: the folded first pass (the indexer's partial histograms,
  // IndexerArgs::hist_part, one query per row) or nullptr (the kernel
  // histograms the scores itself), and the indexer's slot split it follows
  const uint16_t* hist_part;
  int64_t part_total;    // indexer slots
  int64_t part_grid;     // indexer CTAs
  int64_t part_nblk;     // indexer slots per row
  int32_t* cand;         // [rows][N_cap] candidates past the leader's shared memory (scratch)
  int* status;           // device status word (a wait that gave up)
  int64_t rows;
  int k, m;
  int S;                 // CTAs per row: the cluster size (cluster path)
  int vec4;              // rows are 16-byte aligned and slices start at multiples of 4
  int64_t N_cap;
  int64_t slice;         // entries per CTA (cluster path)
};
struct TopkPlan {
  bool slice_path;
  int S, threads;
  int64_t slice;
  size_t smem_bytes, ws_bytes;
};
bool plan_topk(int64_t rows, int64_t N_cap, int k, int num_sms, TopkPlan* p);
size_t topk_scratch_bytes(const TopkPlan& p, int64_t rows, int64_t N_cap);
// Points a->cand into a scratch of topk_scratch_bytes().
void topk_scratch_carve(const TopkPlan& p, int64_t rows, void* ws, TopkArgs* a);
cudaError_t launch_topk(const TopkArgs& a, const TopkPlan& p, bool dependent,
                        cudaStream_t stream);

// ------------------------------------------------------------ attention
// kFused: one query's CSA (top-k), HCA and SWA keys as one key list, so a
// single softmax (and one set of split partials) covers all three branches.
enum AttnKind { kSparse = 0, kHca = 1, kSwa = 2, kFused = 3 };

// ------------------------------------------------------------ query prep
struct QPrepArgs {
  const __nv_bfloat16* q;       // [B][T][H][D]
  const float* gamma;           // [D] or null
  const int32_t* pos;           // [B][T]
  __nv_bfloat16* q_out;         // [B][T][H][D]
  int B, T, H, D, r;
  float eps;
  RopeCoef rope;
};
cudaError_t launch_qprep(const QPrepArgs& a, cudaStream_t stream);

struct AttnArgs {
  const __nv_bfloat16* q;       // prepared queries q~ [B][T][H][D]
  const __nv_bfloat16* kv;      // cache [B][N_cap][D] (sparse/HCA/fused CSA) or raw [B][L_cap][D] (SWA)
  const float* gamma_kv;        // SWA only
  const int32_t* idx;           // sparse only [B][T][k]
  const int32_t* pos;           // [B][T]
  float* o;                     // [B][T][H][D] fp32 (direct output when nsplit == 1)
  float* lse;                   // [B][T][H]
  float* part_o;                // [B*T*H][nsplit][D] partials (nsplit > 1 or partials)
  float* part_lse;              // [B*T*H][nsplit]
  int partials;                 // 1: always write partials, even for one split
  // Finalised output (one split, no partials): the sink-augmented merge and
  // the inverse RoPE of this call's single softmax, out [B][T][H][D] bf16
  // and lse_out [B][T][H] (or null); sink [H] or null.  out == null: o/lse
  // or partials as above.
  __nv_bfloat16* out;
  float* lse_out;
  const float* sink;
  int* status;
  int kind, B, T, H, D, r;
  int64_t N_rows;               // rows per sequence of kv (N_cap or L_cap)
  int64_t N_h;                  // fused: HCA entries per sequence (second tensor map)
  int segments;                 // fused: bit 0 CSA, bit 1 HCA, bit 2 SWA keys
  int k, m, W;                  // fused: W keys per query in the SWA key buffer [B][T][W][D]
  float eps, scale;             // eps: SWA key norm
  RopeCoef rope;                // SWA key RoPE
  int G;                        // queries per row block
  int n_rb;                     // row blocks per sequence = ceil(T / G)
  int nsplit;                   // key splits
  int keys_per_split;           // multiple of 64
  int nds;                      // D splits (1 or 2)
  int n_tq;                     // chunks of the other D half of Q kept in tensor memory
  int dependent;                // launched as a programmatic dependent
};
struct AttnPlan {
  int G, n_rb, nsplit, keys_per_split, nds, n_tq, nslot;
  size_t smem_bytes, ws_bytes;
};
bool plan_attention(int kind, int B, int T, int H, int D, int64_t n_keys, int num_sms,
                    AttnPlan* p);
// tm_kv: HCA entries / SWA raw tokens (fused: HCA entries); tm_kv2: fused only,
// the SWA key buffer.
cudaError_t launch_attention(const CUtensorMap& tm_kv, const CUtensorMap& tm_kv2,
                             const CUtensorMap& tm_q, const AttnArgs& a, const AttnPlan& p,
                             cudaStream_t stream);

// ------------------------------------------------------------ SWA keys
// kv_w[b][t][j] = RoPE_u(RMSNorm(kv_raw[b][u])), u = pos[b][t] - W + 1 + j
// (a zero row where u < 0 or u >= L_cap).
struct SwaKeysArgs {
  const __nv_bfloat16* kv_raw;  // [B][L_cap][D]
  const float* gamma;           // [D] or null
  const int32_t* pos;           // [B][T]
  __nv_bfloat16* kv_w;          // [B][T][W][D]
  int B, T, D, r, W;
  int64_t L_cap;
  int64_t ring;                 // 0: token u in row u; else row u mod ring (L_cap == ring)
  float eps;
  RopeCoef rope;
};
cudaError_t launch_swa_keys(const SwaKeysArgs& a, cudaStream_t stream);

// ------------------------------------------------------------ merges
struct CombineArgs {
  const float* part_o;
  const float* part_lse;
  float* o;
  float* lse;
  int64_t rows;   // B*T*H
  int nsplit, D;
  int dependent;  // launched as a programmatic dependent
};
cudaError_t launch_combine(const CombineArgs& a, cudaStream_t stream);

// Sink-augmented merge of nb branches, each given as nsplit[i] partials per
// row ([rows][nsplit][D] fp32 with [rows][nsplit] log-sum-exps; a branch
// output is the case nsplit = 1).
constexpr int kMaxMergeParts = 128;
struct MergeArgs {
  const float* o[4];            // fp32 partials of each branch
  const float* lse[4];
  int nsplit[4];
  int cum[5];                   // cum[i] = partials of branches before i (cum[nb] = total)
  int nb;
  const float* sink;    // [H] or null
  const int32_t* pos;   // [B][T]
  __nv_bfloat16* out;
  float* lse_out;       // or null
  int B, T, H, D, r;
  int dependent;        // launched as a programmatic dependent
  RopeCoef rope;
};
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);

// Host: RoPE coefficients of base^(-2i/r) for i < r/2 (r <= 2 * kMaxRopePairs).
void make_rope_coef(double base, int r, RopeCoef* rc);

cudaError_t launch_wait_selftest(uint64_t timeout_ns, int* status, cudaStream_t stream);

}  // namespace hattn
