/*
 * hattn.h -- C ABI of libhattn, a B300 (sm_103a) implementation of the
 * DeepSeek-V4 hybrid attention layer: CSA (compressed sparse attention),
 * HCA (heavily compressed attention), SWA (sliding-window attention) and the
 * sink-augmented log-sum-exp merge of their outputs.
 *
 * Sources (web pages on DeepSeek-V4, cited by title and section):
 *   [DD] "Why DeepSeek V4 Stands Apart: A Deep Dive into Its Architecture and
 *        Performance", section "Core Architectural Innovations".
 *   [AT] "DeepSeek-V4" (atlas spec sheet), sections "Design overview",
 *        "Spec sheet / Core block", "Inference efficiency", and
 *        "Provenance references" items 15-18.
 *
 * Conventions shared by every call
 *   - Tensors are dense, row-major, in DEVICE memory.  bf16 tensors are passed
 *     as `const void*` (16-bit storage).  Every tensor pointer must be 16-byte
 *     aligned (HATTN_ERR_MISALIGNED otherwise).
 *   - Shapes use: B sequences, T queries per sequence, H query heads, D head
 *     dim (= the shared KV latent dim, a multiple of 64, at most 512), r RoPE
 *     dims (the last r of each vector, even, r <= D, r <= 128), HI indexer
 *     heads, dI indexer dim (a multiple of 8, at most 128), W SWA window.
 *   - `pos` is an int32 device array [B][T] of absolute query positions.  A
 *     query at position t has its own token already in the raw cache.
 *   - RoPE rotates interleaved pairs (D-r+2i, D-r+2i+1) by the angle
 *     p * rope_base^(-2i/r); RMSNorm is x / sqrt(mean(x^2) + eps) * gamma
 *     (gamma fp32 [D], NULL means all ones).
 *   - The caller owns every buffer, including workspaces; the library never
 *     allocates device memory.  Every call only enqueues work on `stream`
 *     (a cudaStream_t, NULL = legacy default stream) and never synchronises.
 *   - Return value: HATTN_OK or an error code.  Argument errors are detected
 *     on the host before anything is enqueued; the thread-local message from
 *     hattn_last_error() says which argument.  Errors found on the device
 *     (an out-of-range index, a wait that gave up) never trap the GPU: the
 *     kernel records a code in a device status word and returns, and
 *     hattn_check_status() reports it.
 */
#ifndef HATTN_H
#define HATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define HATTN_API __attribute__((visibility("default")))
#else
#define HATTN_API
#endif

typedef void* hattn_stream_t; /* cudaStream_t */

/* Launch flags of the calls that take `flags` (a per-call argument; the
 * library keeps no launch mode between calls).
 *
 * HATTN_LAUNCH_DEPENDENT: launch the call's kernels as programmatic
 * dependents (CUDA programmatic dependent launch) of the previous kernel in
 * `stream`.  They may start -- allocate tensor memory, initialise barriers,
 * prefetch descriptors -- while that kernel finishes, and wait for it
 * (griddepcontrol.wait) before reading anything it may write.  Set it only
 * where the previous kernel in the stream is the one producing the call's
 * inputs: it relaxes only that one dependency.  Each call's comment says
 * which of its inputs it may read before that wait.  Every kernel of the
 * library lets its own dependents start early.
 *
 * HATTN_EVENT_EXTERNAL: a call that records an event of the caller's
 * (hattn_indexer_topk_ex's split_event) records it with
 * cudaEventRecordExternal, so that under stream capture it becomes an event
 * record node a graph replay can be timed by.  Without it a captured record
 * only marks a point other streams can wait for. */
#define HATTN_LAUNCH_DEPENDENT 1
#define HATTN_EVENT_EXTERNAL 2

enum {
  HATTN_OK = 0,
  HATTN_ERR_INVALID_ARG = 1, /* null pointer, size out of range, inconsistent sizes */
  HATTN_ERR_MISALIGNED = 2,  /* a tensor pointer is not 16-byte aligned */
  HATTN_ERR_UNSUPPORTED = 3, /* valid by the definitions, but no kernel for this shape */
  HATTN_ERR_CUDA = 4,        /* a CUDA runtime/driver call or launch failed */
  HATTN_ERR_TIMEOUT = 5,     /* a device-side wait gave up (reported by hattn_check_status) */
  HATTN_ERR_DEVICE_INDEX = 6 /* a device-side index was out of range (hattn_check_status) */
};

/* -------------------------------------------------------------------------
 * KV compression.  [DD]: CSA compresses KV 4x (m=4), HCA 128:1.  [AT] "Design
 * overview": CSA compresses every 4 tokens into two overlapping streams;
 * RMSNorm on the compressed KV entries.
 *
 * Entry j pools the tokens u in [m(j+1)-w, m(j+1)-1] that exist (u >= 0) with
 * weights softmax over those tokens of the bf16 gate logit gate[b][u]; the
 * pooled KV vector is RMSNorm'd (gamma_kv, eps) and RoPE'd at position
 * m(j+1)-1; the pooled indexer key uses the same weights, with no norm and
 * no RoPE.  CSA is m=4, w=8 (the 8 tokens [4j-4, 4j+4)).
 *
 *   kv_raw [B][L_cap][D] bf16, ik_raw [B][L_cap][dI] bf16, gate [B][L_cap] bf16
 *   entries j in [j_begin, j_end) are written to row j of
 *   kv_c [B][N_cap][D] bf16 and ik_c [B][N_cap][dI] bf16 (other rows untouched);
 *   requires j_end <= N_cap, m*j_end <= L_cap, w % m == 0, w >= m, w <= 512.
 *   j_begin == j_end is a no-op.  Fused single pass: each token row is read
 *   from HBM once per window it belongs to, each entry written once.
 * ---------------------------------------------------------------------- */
HATTN_API int hattn_csa_compress(const void* kv_raw, const void* ik_raw, const void* gate,
                       const float* gamma_kv, int B, int64_t L_cap, int D, int dI, int m, int w,
                       int r, float rope_base, float eps, int64_t j_begin, int64_t j_end,
                       void* kv_c, void* ik_c, int64_t N_cap, hattn_stream_t stream);

/* HCA compression: the same compressor with w = m (non-overlapping windows,
 * m = 128 on the pages) and no indexer key.  kv_h [B][N_cap][D] bf16. */
HATTN_API int hattn_hca_compress(const void* kv_raw, const void* gate, const float* gamma_kv, int B,
                       int64_t L_cap, int D, int m, int r, float rope_base, float eps,
                       int64_t j_begin, int64_t j_end, void* kv_h, int64_t N_cap,
                       hattn_stream_t stream);

/* Compressed entries straight from hidden states (cache build).  Each
 * token's KV and indexer-key row is the projection x_u . W of its hidden
 * state (W [dm][D + dI] bf16: the D KV columns, then the dI indexer-key
 * columns), and entry j is C(m, w) of those rows as in hattn_csa_compress:
 * gate-softmax pooling, RMSNorm and RoPE of the KV part.  Pooling is linear,
 * so the library pools the hidden states first and projects once per entry,
 * (sum_u a_u x_u) . W, which is the same entry up to rounding: the hidden
 * states are read once per window, no per-token KV row is written, and the
 * projection runs on one row per entry.  The pooled row is kept to ~16
 * significant bits (two bf16 parts) and projected by cuBLASLt with fp32
 * accumulation.
 *   x [B][L_cap][dm] bf16 (dm a multiple of 8), gate [B][L_cap] bf16;
 *   entries [j_begin, j_end) go to kv_out [B][N_cap][D] and, when dI > 0,
 *   ik_out [B][N_cap][dI] (NULL when dI == 0: HCA is m = w = 128, dI = 0);
 *   workspace of hattn_compress_hidden_workspace_bytes() bytes. */
HATTN_API size_t hattn_compress_hidden_workspace_bytes(int B, int64_t j_begin, int64_t j_end,
                                                       int dm, int D, int dI);
HATTN_API int hattn_compress_hidden(const void* x, const void* W, const void* gate,
                                    const float* gamma_kv, int B, int64_t L_cap, int dm, int D,
                                    int dI, int m, int w, int r, float rope_base, float eps,
                                    int64_t j_begin, int64_t j_end, void* kv_out, void* ik_out,
                                    int64_t N_cap, void* workspace, size_t ws_bytes,
                                    hattn_stream_t stream);

/* Both caches of a layer from hidden states in one read of them ([DD]
 * "Infrastructure and Deployment": fewer passes over the data): the CSA
 * entries C(4, 8) with their indexer keys (W_c [dm][D + dI], gate_c) and the
 * HCA entries C(128, 128) (W_h [dm][D], gate_h) of the first L tokens of each
 * sequence, as hattn_compress_hidden computes each (same pooling, projection,
 * RMSNorm with gamma_kv, RoPE at the entry's last token):
 *   kv_c [B][N_c][D], ik_c [B][N_c][dI] (NULL when dI == 0), entries
 *   j < min(N_c, L/4); kv_h [B][N_h][D], entries j < min(N_h, L/128), which
 *   need min(N_c, L/4) >= 32 * (HCA entries - 1) + 1 (full caches do).
 * Each 128-token block's hidden states come from HBM once: its CSA windows
 * read them, and its HCA window, pooled right after, finds them in L2.
 * Workspace: hattn_compress_hidden_pair_workspace_bytes() bytes (the pooled
 * rows of one pass of 16,384 CSA entries, then those of every HCA entry). */
HATTN_API size_t hattn_compress_hidden_pair_workspace_bytes(int B, int64_t L, int64_t N_c,
                                                            int64_t N_h, int dm);
HATTN_API int hattn_compress_hidden_pair(const void* x, const void* W_c, const void* gate_c,
                                         const void* W_h, const void* gate_h,
                                         const float* gamma_kv, int B, int64_t L_cap, int64_t L,
                                         int dm, int D, int dI, int r, float rope_base, float eps,
                                         void* kv_c, void* ik_c, int64_t N_c, void* kv_h,
                                         int64_t N_h, void* workspace, size_t ws_bytes,
                                         hattn_stream_t stream);

/* Ring-buffer raw caches.  A decode loop needs only the newest raw tokens:
 * the compressors read the window of the entry the newest token completes
 * (8 tokens for CSA, 128 for HCA) and the window keys the last W tokens.  In
 * these forms the raw buffers kv_ring [B][ring][D], ik_ring [B][ring][dI] and
 * gate_ring [B][ring] hold token u in row u mod ring (ring a power of two),
 * so a 256-row ring replaces a 1M-row cache.  Positions (pos, entry indices)
 * stay absolute.  The caller keeps every token a call reads in the ring:
 * for the compressors the m*(j_end-j_begin)+w-m tokens ending at
 * m*j_end-1, for the window keys the W+T-1 tokens ending at each
 * sequence's newest query position.  Otherwise as hattn_csa_compress,
 * hattn_hca_compress and hattn_swa_keys. */
HATTN_API int hattn_csa_compress_ring(const void* kv_ring, const void* ik_ring,
                                      const void* gate_ring, const float* gamma_kv, int B,
                                      int64_t ring, int D, int dI, int m, int w, int r,
                                      float rope_base, float eps, int64_t j_begin, int64_t j_end,
                                      void* kv_c, void* ik_c, int64_t N_cap,
                                      hattn_stream_t stream);
HATTN_API int hattn_hca_compress_ring(const void* kv_ring, const void* gate_ring,
                                      const float* gamma_kv, int B, int64_t ring, int D, int m,
                                      int r, float rope_base, float eps, int64_t j_begin,
                                      int64_t j_end, void* kv_h, int64_t N_cap,
                                      hattn_stream_t stream);

/* -------------------------------------------------------------------------
 * FP8 indexer keys.  [AT] "Inference efficiency": the indexer's QK path runs
 * in low precision.  The pages name no format; this library stores E4M3
 * codes (OCP FP8: bias 7, 3 mantissa bits, largest finite 448, saturating)
 * with one fp32 scale per row:
 *   amax = max_i |x_i|, inv = 448 / amax, code_i = e4m3_rne(x_i * inv),
 *   scale = amax / 448 (each step one correctly rounded fp32 operation);
 * the row decodes as code_i * scale.  A zero row has zero codes, scale 0.
 *
 * hattn_quantize_e4m3: rows x n bf16 -> codes [rows][n] (bytes) and
 *   scales [rows] fp32; n a multiple of 4.  Used to build an FP8 key cache
 *   from bf16 keys.  With rows = 0 the pointers are not checked.
 * hattn_csa_compress_fp8: hattn_csa_compress that also writes each entry's
 *   indexer key as E4M3 codes ik8 [B][N_cap][dI] and scale ik_scale
 *   [B][N_cap] fp32, quantised from the bf16-rounded key (the value ik_c
 *   holds); ik_c may be NULL (then only the FP8 key is written).
 * ---------------------------------------------------------------------- */
HATTN_API int hattn_quantize_e4m3(const void* x, int64_t rows, int n, void* codes, float* scales,
                                  hattn_stream_t stream);

/* -------------------------------------------------------------------------
 * MXFP4 indexer rows.  [AT] "Inference efficiency" names the indexer QK
 * path's format: FP4 (MXFP4); [DD] "Core Architectural Innovations" (FP4
 * quantization-aware training) names the FP4 element type, E2M1.  MXFP4 is
 * the OCP Microscaling format: blocks of 32 consecutive elements share one
 * power-of-two scale, stored as an E8M0 code c (value 2^(c-127)).
 *   amax_b = max |x_i| over block b, X_b = 2^(floor(log2 amax_b) - 2)
 *     (exponent clamped to [-127, 125]; an all-zero block takes c = 0),
 *   code_i = e2m1_rne_satfinite(x_i / X_b)   (magnitudes 0, 0.5, 1, 1.5,
 *     2, 3, 4, 6; ties to the even code; beyond 6 clamps to 6; a zero
 *     result is stored as +0),
 * and element i decodes as e2m1(code_i) * X_b.  Inputs must be finite.
 *
 * hattn_quantize_mxfp4: rows x n bf16 (n a multiple of 32) -> codes
 *   [rows][n/2] bytes, element 2i in the low nibble and 2i+1 in the high
 *   nibble of byte i, and scales [rows][n/32] E8M0 bytes.  For a 128-dim
 *   indexer row: 64 code bytes and 4 scale bytes (68 B, against 256 B of
 *   bf16).  All three pointers device memory, 16-byte aligned, caller-owned
 *   (any value when rows = 0: nothing is touched); the call is asynchronous
 *   on `stream`.
 * ---------------------------------------------------------------------- */
HATTN_API int hattn_quantize_mxfp4(const void* x, int64_t rows, int n, void* codes, void* scales,
                                   hattn_stream_t stream);

/* hattn_quantize_mxfp4 over the entries [j_begin, j_end) of every sequence
 * of a cache x [B][N_cap][n] bf16, into codes [B][N_cap][n/2] and scales
 * [B][N_cap][n/32] (other entries untouched): keeps an MXFP4 key cache in
 * step with the entries a decode step compresses. */
HATTN_API int hattn_quantize_mxfp4_entries(const void* x, int B, int64_t N_cap, int n,
                                           int64_t j_begin, int64_t j_end, void* codes,
                                           void* scales, hattn_stream_t stream);

/* hattn_csa_compress that also writes each entry's indexer key as MXFP4:
 * codes ik4 [B][N_cap][dI/2] and E8M0 scales ik4_scale [B][N_cap][dI/32],
 * quantised from the bf16-rounded key (the value ik_c holds) exactly as
 * hattn_quantize_mxfp4 does; dI a multiple of 32.  One launch instead of the
 * compression and a quantisation of its entries. */
HATTN_API int hattn_csa_compress_mxfp4(const void* kv_raw, const void* ik_raw, const void* gate,
                                       const float* gamma_kv, int B, int64_t L_cap, int D, int dI,
                                       int m, int w, int r, float rope_base, float eps,
                                       int64_t j_begin, int64_t j_end, void* kv_c, void* ik_c,
                                       void* ik4, void* ik4_scale, int64_t N_cap,
                                       hattn_stream_t stream);

/* Indexer scores over MXFP4 keys ([AT] "Inference efficiency": the indexer's
 * QK path in FP4): ik4 [B][N_cap][64] code bytes and ik4_scale [B][N_cap][4]
 * E8M0 bytes as hattn_quantize_mxfp4 writes them (dI must be 128; N_cap a
 * multiple of 4, so that a block's scales are whole 16-byte rows).  Each bf16
 * query row iq[b][t][h] takes the same MXFP4 round trip inside the kernel,
 * and the score is the plain definition over the decoded values,
 *   I[j] = sum_h w[b][t][h] * max(0, q~[b][t][h] . k~[b][j]),
 * with fp32 accumulation.  A key costs 68 bytes of HBM (against 256 for
 * bf16).  The products run on the block-scaled FP4 tensor-core path
 * (kind::mxf4): the E2M1 codes of keys and queries are the operands and
 * their E8M0 scales the block scales, so no key is decoded.  The other
 * arguments, limits and flags are hattn_indexer_scores_ex's; queries go in
 * groups of at most 128 rows (G * HI <= 128). */
HATTN_API int hattn_indexer_scores_mxfp4(const void* iq, const float* w, const void* ik4,
                                         const void* ik4_scale, const int32_t* pos, int B, int T,
                                         int HI, int dI, int64_t N_cap, int m, int n_sms,
                                         int64_t fresh_from, float* score_out, int flags,
                                         hattn_stream_t stream);
/* hattn_indexer_topk_ex over MXFP4 keys (scores as hattn_indexer_scores_mxfp4;
 * the workspace is hattn_indexer_topk_workspace_bytes()). */
HATTN_API int hattn_indexer_topk_mxfp4(const void* iq, const float* w, const void* ik4,
                                       const void* ik4_scale, const int32_t* pos, int B, int T,
                                       int HI, int dI, int64_t N_cap, int k, int m, int n_sms,
                                       int64_t fresh_from, int32_t* idx_out, float* score_out,
                                       void* workspace, size_t ws_bytes, int flags,
                                       void* split_event, hattn_stream_t stream);

HATTN_API int hattn_csa_compress_fp8(const void* kv_raw, const void* ik_raw, const void* gate,
                                     const float* gamma_kv, int B, int64_t L_cap, int D, int dI,
                                     int m, int w, int r, float rope_base, float eps,
                                     int64_t j_begin, int64_t j_end, void* kv_c, void* ik_c,
                                     void* ik8, float* ik_scale, int64_t N_cap,
                                     hattn_stream_t stream);

/* -------------------------------------------------------------------------
 * Lightning indexer + per-query top-k.  [DD]: CSA keeps the top-1024 (Pro) /
 * top-512 (Flash) compressed entries per query.  [AT] "Design overview": the
 * V3.2 lightning-indexer sparse attention.
 *
 * For each query (b, t) with n = min(floor((pos+1)/m), N_cap) visible entries:
 *   I[j] = sum_h w[b][t][h] * max(0, iq[b][t][h] . ik_c[b][j])   for j < n
 *   idx_out[b][t][0..k) = the min(k, n) entries with the largest I (ties to the
 *   smaller j), in unspecified order, then -1 padding.
 *
 *   iq [B][T][HI][dI] bf16, w [B][T][HI] fp32, ik_c [B][N_cap][dI] bf16,
 *   idx_out [B][T][k] int32, score_out [B][T][N_cap] fp32 or NULL (when given,
 *   receives I for j < n; entries j >= n are left untouched).
 *   workspace: device buffer of at least hattn_indexer_topk_workspace_bytes()
 *   bytes (may be NULL when that is 0): the scores (unless score_out is
 *   given), the score kernel's per-CTA histograms (when the selection runs
 *   in clusters, see hattn_topk_select), then the selection's scratch;
 *   contents need no initialisation.  Calls sharing one workspace must not
 *   overlap on the GPU.
 *   With one query per indexer group (T == 1 or HI > 128) and few long rows,
 *   the score kernel also counts the top 11 bits of each score's
 *   order-preserving key per row as it writes the scores, so the selection
 *   starts from the row's histogram instead of a pass over the scores.
 *   Limits: 1 <= k <= 2048, HI * min(T, 256 / HI) <= 256, N_cap < 2^31.
 * ---------------------------------------------------------------------- */
HATTN_API int hattn_indexer_topk(const void* iq, const float* w, const void* ik_c, const int32_t* pos,
                       int B, int T, int HI, int dI, int64_t N_cap, int k, int m,
                       int32_t* idx_out, float* score_out, void* workspace, size_t ws_bytes,
                       hattn_stream_t stream);
HATTN_API size_t hattn_indexer_topk_workspace_bytes(int B, int T, int64_t N_cap, int k,
                                          int score_out_given);
/* hattn_indexer_topk with the options of hattn_indexer_scores_ex and FP8 keys:
 *   ik_scale: NULL for bf16 keys ik_c [B][N_cap][dI]; else ik_c holds E4M3
 *   codes [B][N_cap][128] with these row scales [B][N_cap] fp32 (see
 *   hattn_indexer_scores_fp8 for the limits and the arithmetic).
 *   n_sms, fresh_from, flags: as hattn_indexer_scores_ex, for the score
 *   kernel; the selection kernel is always launched as a programmatic
 *   dependent of it and reads only pos before its wait.
 *   workspace: hattn_indexer_topk_workspace_bytes() bytes, as above.
 *   split_event: a cudaEvent_t (cast to void*) recorded on `stream` between
 *   the score and the selection kernel, or NULL: other streams may wait for
 *   the scores alone on it, and with HATTN_EVENT_EXTERNAL in flags it times
 *   the two kernels apart (an external record keeps the selection from
 *   starting early). */
HATTN_API int hattn_indexer_topk_ex(const void* iq, const float* w, const void* ik_c,
                                    const float* ik_scale, const int32_t* pos, int B, int T,
                                    int HI, int dI, int64_t N_cap, int k, int m, int n_sms,
                                    int64_t fresh_from, int32_t* idx_out, float* score_out,
                                    void* workspace, size_t ws_bytes, int flags,
                                    void* split_event, hattn_stream_t stream);

/* hattn_indexer_topk for callers that cannot allocate device memory: code
 * that runs where cudaMalloc is not allowed or not wanted, such as an engine
 * that owns a fixed memory pool, a plugin host that forbids device
 * allocations, or a stream-ordered path that must not synchronise on the
 * allocator.  The same selection as hattn_indexer_topk, but the fp32 scores
 * and the selection's scratch live in an array compiled into this library
 * (34 MiB: 4,194,304 scores, then up to 18 MiB of histograms and selection scratch, held
 * on every device that loads the library until the process exits), so the
 * call allocates nothing; the caller still passes inputs and idx_out.  The
 * pages have no counterpart of this call.
 *   - B * T * N_cap must not exceed 4,194,304 (HATTN_ERR_INVALID_ARG).
 *   - The first call on a device looks the scratch address up (cudaGetSymbolAddress)
 *     with that device current; make that first call before any stream capture.
 *   - Every call on a device shares the one scratch array: calls whose work
 *     overlaps on the GPU (other streams, other host threads) race.  No
 *     contents need clearing between calls: every score, histogram and
 *     counter the selection reads is written earlier in the same call. */
HATTN_API int hattn_indexer_topk_noalloc(const void* iq, const float* w, const void* ik_c,
                                         const int32_t* pos, int B, int T, int HI, int dI,
                                         int64_t N_cap, int k, int m, int32_t* idx_out,
                                         hattn_stream_t stream);

/* The two stages of hattn_indexer_topk as separate calls.
 * hattn_indexer_scores writes I[j] for j < n into score_out [B][T][N_cap] fp32
 * (entries j >= n untouched).  hattn_topk_select reads those scores and writes
 * idx_out [B][T][k] with the selection rule above (same limits). */
HATTN_API int hattn_indexer_scores(const void* iq, const float* w, const void* ik_c,
                                   const int32_t* pos, int B, int T, int HI, int dI,
                                   int64_t N_cap, int m, float* score_out, hattn_stream_t stream);
/* hattn_indexer_scores with scheduling options.
 *   n_sms: run the persistent score kernel on at most that many SMs (0 = all;
 *   one CTA per SM used), leaving the others to work on another stream.
 *   flags: HATTN_LAUNCH_DEPENDENT or 0.  A dependent launch reads iq, w and
 *   pos before its wait, so those must not be written by the previous
 *   kernel in the stream; of ik_c it reads before the wait only the blocks
 *   of entries below fresh_from.
 *   fresh_from: with HATTN_LAUNCH_DEPENDENT, the entries of ik_c at index >=
 *   fresh_from are the only ones the previous kernel in the stream may write
 *   (say, the compressor of the newest entry); blocks of entries below it
 *   are read without waiting for that kernel.  -1: any entry may be written
 *   (wait before the first key read).  Ignored without the flag. */
HATTN_API int hattn_indexer_scores_ex(const void* iq, const float* w, const void* ik_c,
                                      const int32_t* pos, int B, int T, int HI, int dI,
                                      int64_t N_cap, int m, int n_sms, int64_t fresh_from,
                                      float* score_out, int flags, hattn_stream_t stream);
/* hattn_topk_select: scores [B][T][N_cap] fp32 (entries j < n as written by
 * the score calls) -> idx_out [B][T][k] int32.  Few long rows (say 8 rows of
 * 262,144) are each spread over a thread-block cluster of 8 or 16 CTAs,
 * which needs a caller-owned scratch of hattn_topk_workspace_bytes(B, T,
 * N_cap, k) bytes (B * T * N_cap int32: the candidates of a row whose
 * threshold bin holds more than 12,288 entries, say a row of near-equal
 * scores); it is 0 when the rows fit one CTA each, and workspace may then be
 * NULL.  The scratch needs no initialisation; calls sharing one scratch must
 * not overlap on the GPU.
 * flags: HATTN_LAUNCH_DEPENDENT or 0 (with the flag, the cluster path reads
 * pos before the wait, so the previous kernel must not write pos; the
 * scores are read after it). */
HATTN_API size_t hattn_topk_workspace_bytes(int B, int T, int64_t N_cap, int k);
HATTN_API int hattn_topk_select(const float* scores, const int32_t* pos, int B, int T,
                                int64_t N_cap, int k, int m, int32_t* idx_out, void* workspace,
                                size_t ws_bytes, int flags, hattn_stream_t stream);

/* hattn_indexer_scores_ex over FP8 keys: ik8 [B][N_cap][128] E4M3 codes and
 * ik_scale [B][N_cap] fp32 (see hattn_quantize_e4m3; dI must be 128 and
 * N_cap a multiple of 4, so that a block's scales are whole 16-byte rows).  Each
 * bf16 query row iq[b][t][h] is quantised the same way inside the kernel,
 * and the score is the plain definition over the decoded values,
 *   I[j] = sum_h w[b][t][h] * max(0, q^[b][t][h] . k^[b][j]),
 * computed as ik_scale[j] * sum_h (w * q_scale_h) * max(0, q8_h . k8_j) with
 * the code products on the tensor cores (fp32 accumulation).  Scores go to
 * score_out as for hattn_indexer_scores; n_sms, fresh_from and flags as for
 * hattn_indexer_scores_ex (a dependent launch reads ik_scale like ik8).  The
 * key stream is 132 bytes per entry instead of 256. */
HATTN_API int hattn_indexer_scores_fp8(const void* iq, const float* w, const void* ik8,
                                       const float* ik_scale, const int32_t* pos, int B, int T,
                                       int HI, int dI, int64_t N_cap, int m, int n_sms,
                                       int64_t fresh_from, float* score_out, int flags,
                                       hattn_stream_t stream);

/* -------------------------------------------------------------------------
 * Query preparation.  [AT] "Design overview": RMSNorm on the queries;
 * provenance 16: RoPE on the last r dims.  For every (b, t, h):
 *   q_out = RoPE_pos[b][t](RMSNorm(q; gamma_q, eps))   (bf16)
 * q, q_out [B][T][H][D] bf16 (may not overlap); gamma_q fp32 [D] or NULL.
 * The three attention calls accept q_out with q_prepped = 1, so one
 * preparation serves every branch of a layer.
 * ---------------------------------------------------------------------- */
HATTN_API int hattn_query_prep(const void* q, const float* gamma_q, const int32_t* pos, int B,
                               int T, int H, int D, int r, float rope_base, float eps,
                               void* q_out, hattn_stream_t stream);

/* -------------------------------------------------------------------------
 * Attention branches.  Shared-KV MQA latent ([AT] "Inference efficiency"):
 * keys and values are the same D-dim vectors K~ for all heads.  Each query
 * head is prepared as q~ = RoPE_pos(RMSNorm(q; gamma_q, eps)); logits are
 * scale * q~ . K~_j; the branch output is o = sum_j softmax_j K~_j (fp32) and
 * lse = log sum_j exp(logit_j) (fp32, natural log).  An empty key set gives
 * o = 0, lse = -inf.  Branch outputs stay fp32 so the merge rounds to bf16
 * once.
 *
 *   q [B][T][H][D] bf16: raw queries (q_prepped = 0; the call prepares them
 *   into its workspace with gamma_q and eps), or the output of
 *   hattn_query_prep (q_prepped = 1; gamma_q and eps are then not used for
 *   the queries).  o [B][T][H][D] fp32, lse [B][T][H] fp32.
 *   workspace: at least hattn_attn_workspace_bytes(kind, ..., q_prepped)
 *   bytes (prepared queries, then split-KV partials); contents need no
 *   initialisation.  H <= 128; D a multiple of 64 up to 512 (a multiple of
 *   128 above 256).
 * ---------------------------------------------------------------------- */

/* CSA branch ([DD]: sparse attention over the selected compressed entries):
 * keys are kv_c[b][idx[b][t][i]] for every i with idx >= 0 (-1 is padding).
 * kv_c [B][N_cap][D] bf16 (normalised + roped entries), idx [B][T][k] int32.
 * An idx >= N_cap is skipped and reported as HATTN_ERR_DEVICE_INDEX. */
HATTN_API int hattn_sparse_attn(const void* q, const float* gamma_q, int q_prepped,
                      const void* kv_c, const int32_t* idx,
                      const int32_t* pos, int B, int T, int H, int D, int64_t N_cap, int k, int r,
                      float rope_base, float eps, float scale, void* o, float* lse,
                      void* workspace, size_t ws_bytes, hattn_stream_t stream);

/* HCA branch ([DD]: dense global attention over the 128:1 compressed KV):
 * keys are kv_h[b][j] for j < min(floor((pos+1)/m), N_cap).  kv_h [B][N_cap][D]. */
HATTN_API int hattn_hca_attn(const void* q, const float* gamma_q, int q_prepped, const void* kv_h,
                   const int32_t* pos,
                   int B, int T, int H, int D, int64_t N_cap, int m, int r, float rope_base,
                   float eps, float scale, void* o, float* lse, void* workspace,
                   size_t ws_bytes, hattn_stream_t stream);

/* SWA branch ([DD]: the most recent 128 tokens): keys are the raw tokens
 * u in [max(0, pos-W+1), pos], each RMSNorm'd (gamma_kv, eps) and RoPE'd at
 * position u on load.  kv_raw [B][L_cap][D] bf16. */
HATTN_API int hattn_swa_attn(const void* q, const float* gamma_q, int q_prepped, const void* kv_raw,
                   const float* gamma_kv, const int32_t* pos, int B, int T, int H, int D,
                   int64_t L_cap, int W, int r, float rope_base, float eps, float scale, void* o,
                   float* lse, void* workspace, size_t ws_bytes, hattn_stream_t stream);

/* SWA keys for hattn_hybrid_attn ([DD]: the most recent W tokens, each in the
 * normalised, roped space of the compressed entries):
 *   kv_w[b][t][j] = RoPE_u(RMSNorm(kv_raw[b][u]; gamma_kv, eps)),
 *   u = pos[b][t] - W + 1 + j   (j < W; a zero row where u < 0 or u >= L_cap)
 * kv_raw [B][L_cap][D] bf16, kv_w [B][T][W][D] bf16 (caller-owned). */
HATTN_API int hattn_swa_keys(const void* kv_raw, const float* gamma_kv, const int32_t* pos, int B,
                             int T, int64_t L_cap, int D, int W, int r, float rope_base,
                             float eps, void* kv_w, hattn_stream_t stream);
/* hattn_swa_keys over a ring-buffer raw cache kv_ring [B][ring][D] (token u
 * in row u mod ring; ring a power of two, at least W + T - 1). */
HATTN_API int hattn_swa_keys_ring(const void* kv_ring, const float* gamma_kv, const int32_t* pos,
                                  int B, int T, int64_t ring, int D, int W, int r,
                                  float rope_base, float eps, void* kv_w, hattn_stream_t stream);

/* The three branches as one attention ([DD] CSA + HCA + SWA, merged by
 * log-sum-exp): for each query the keys are the selected CSA entries
 * kv_c[b][idx[b][t][i]] (idx >= 0), the visible HCA entries kv_h[b][j],
 * j < min(floor((pos+1)/m), N_h), and the existing window tokens
 * kv_w[b][t][j] (from hattn_swa_keys, j >= W-1-pos), all under one softmax.
 * Because each branch's own normalisation cancels in the sink merge, merging
 * this result (or its partials) with hattn_lse_merge(_splits) gives the
 * layer output of the three branch calls merged together.
 *   segments: bit 0 CSA, bit 1 HCA, bit 2 SWA -- the key sets this call
 *   covers (7 = all); the pointers of the others may be NULL.  Calls over
 *   disjoint segment sets leave partials that one hattn_lse_merge_splits
 *   combines, so the part that does not need the top-k result can run
 *   concurrently with the indexer.
 *   n_sms: the number of SMs the split plan assumes (0 = all of them); a
 *   call meant to share the GPU with concurrent work plans for its share.
 * The output conventions (o/lse, partials with o == lse == NULL, q_prepped,
 * workspace) are those of the branch calls; the workspace size and split
 * count come from the two functions below, given the same segments and
 * n_sms.  One query per row block: the MMA rows are the H heads of one
 * query (H <= 128).  flags: HATTN_LAUNCH_DEPENDENT or 0 (a dependent launch
 * reads pos before its wait, everything else after it). */
HATTN_API int hattn_hybrid_attn(const void* q, const float* gamma_q, int q_prepped,
                                const void* kv_c, const int32_t* idx, int64_t N_c, int k,
                                const void* kv_h, int64_t N_h, int m, const void* kv_w, int W,
                                const int32_t* pos, int B, int T, int H, int D, int r,
                                float rope_base, float eps, float scale, int segments, int n_sms,
                                void* o, float* lse, void* workspace, size_t ws_bytes,
                                int flags, hattn_stream_t stream);
/* hattn_hybrid_attn straight to the layer output: the sink merge and the
 * inverse RoPE ([AT] "Spec sheet / Core block": attention sinks, inverse RoPE
 * on the outputs) applied to the call's single softmax,
 *   Z = sum_j e^(l_j) + e^(sink[h]),  y = sum_j e^(l_j) v_j / Z,
 *   out = y with its last r dims rotated back by the query position,
 *   lse_out = log Z,
 * which equals hattn_hybrid_attn's partials merged by hattn_lse_merge_splits
 * when the call covers every key set of the layer.  When each query's keys
 * take one split (prefill: many row blocks) the attention kernel writes out
 * and lse_out itself, with no partials; otherwise it leaves partials in the
 * workspace and a merge kernel follows (launched as its dependent).
 *   sink [H] fp32 or NULL; out [B][T][H][D] bf16; lse_out [B][T][H] fp32 or
 *   NULL.  The other arguments, the limits and flags are hattn_hybrid_attn's;
 *   workspace: hattn_hybrid_attn_out_workspace_bytes() bytes (0 when the
 *   queries come prepared and the keys take one split). */
HATTN_API int hattn_hybrid_attn_out(const void* q, const float* gamma_q, int q_prepped,
                                    const void* kv_c, const int32_t* idx, int64_t N_c, int k,
                                    const void* kv_h, int64_t N_h, int m, const void* kv_w,
                                    int W, const int32_t* pos, int B, int T, int H, int D, int r,
                                    float rope_base, float eps, float scale, int segments,
                                    int n_sms, const float* sink, void* out, float* lse_out,
                                    void* workspace, size_t ws_bytes, int flags,
                                    hattn_stream_t stream);
HATTN_API size_t hattn_hybrid_attn_out_workspace_bytes(int B, int T, int H, int D, int k,
                                                       int64_t N_h, int W, int segments,
                                                       int n_sms, int q_prepped);
HATTN_API size_t hattn_hybrid_attn_workspace_bytes(int B, int T, int H, int D, int k,
                                                   int64_t N_h, int W, int segments, int n_sms,
                                                   int q_prepped, int partials);
HATTN_API int hattn_hybrid_attn_splits(int B, int T, int H, int D, int k, int64_t N_h, int W,
                                       int segments, int n_sms);

/* Split partials instead of a branch output: with o == NULL and lse == NULL
 * an attention call leaves the softmax of each key split in its workspace,
 * right after the prepared queries (if any):
 *   part_o   [B*T*H][nsplit][D] fp32 (each split normalised by its own sum)
 *   part_lse [B*T*H][nsplit]    fp32 (that split's log-sum-exp)
 * with nsplit = hattn_attn_splits(...).  hattn_lse_merge_splits merges such
 * partials of several branches in one pass (no per-branch combine).
 *
 * kind: 0 = CSA sparse (n_keys = k), 1 = HCA (n_keys = N_cap), 2 = SWA (n_keys = W).
 * partials: 1 when the call is made in the partials form above.  0 means no
 * workspace is needed (or no kernel exists for the shape). */
HATTN_API size_t hattn_attn_workspace_bytes(int kind, int B, int T, int H, int D, int64_t n_keys,
                                            int q_prepped, int partials);
/* Key splits (partials per row) an attention call of this shape uses; 0 if
 * no kernel exists for it. */
HATTN_API int hattn_attn_splits(int kind, int B, int T, int H, int D, int64_t n_keys);

/* -------------------------------------------------------------------------
 * Merge.  [AT] "Spec sheet / Core block": attention sinks; provenance 16:
 * "-i RoPE on outputs".  For every (b, t, h):
 *   Z = sum_i exp(lse_i) + exp(sink[h]);  y = sum_i exp(lse_i) o_i / Z
 *   out = y with its last r dims rotated by -pos (inverse RoPE); lse_out = log Z.
 * o_list / lse_list: HOST arrays of nb (1..4) DEVICE pointers to fp32
 * [B][T][H][D] / fp32 [B][T][H] branch outputs (16-byte aligned).  sink fp32 [H] device or NULL
 * (no sink term).  out [B][T][H][D] bf16, lse_out [B][T][H] fp32 or NULL.
 * ---------------------------------------------------------------------- */
HATTN_API int hattn_lse_merge(const void* const* o_list, const float* const* lse_list, int nb,
                    const float* sink, const int32_t* pos, int B, int T, int H, int D, int r,
                    float rope_base, void* out, float* lse_out, hattn_stream_t stream);

/* The same merge over split partials: branch i is given by nsplit[i] (host
 * array) partials per row, part_o_list[i] fp32 [B*T*H][nsplit[i]][D] and
 * part_lse_list[i] fp32 [B*T*H][nsplit[i]] (as left by an attention call with
 * o == lse == NULL).  The result equals combining each branch's splits and
 * then merging (a branch's own normalisation cancels).  At most 128 partials
 * per row in total.  flags: HATTN_LAUNCH_DEPENDENT or 0 (every input is read
 * after the wait). */
HATTN_API int hattn_lse_merge_splits(const void* const* part_o_list,
                                     const float* const* part_lse_list, const int* nsplit, int nb,
                                     const float* sink, const int32_t* pos, int B, int T, int H,
                                     int D, int r, float rope_base, void* out, float* lse_out,
                                     int flags, hattn_stream_t stream);

/* -------------------------------------------------------------------------
 * Status and diagnostics.
 * ---------------------------------------------------------------------- */
HATTN_API const char* hattn_status_string(int code);
/* Thread-local description of the last error returned on this thread. */
HATTN_API const char* hattn_last_error(void);
/* Synchronises `stream`, then returns and clears the device status word of
 * the current device (HATTN_OK, HATTN_ERR_TIMEOUT or HATTN_ERR_DEVICE_INDEX),
 * or HATTN_ERR_CUDA if the synchronisation itself failed. */
HATTN_API int hattn_check_status(hattn_stream_t stream);
/* Test hook for the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier nothing arrives on, giving up after timeout_ns nanoseconds; the
 * kernel then records HATTN_ERR_TIMEOUT and returns (no fault, no hang). */
HATTN_API int hattn_selftest_wait_timeout(uint64_t timeout_ns, hattn_stream_t stream);
/* Library version string. */
HATTN_API const char* hattn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HATTN_H */
