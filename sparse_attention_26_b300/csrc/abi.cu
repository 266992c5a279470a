// abi.cu -- the extern "C" entry points of libhattn (declared in
// include/hattn.h): argument validation, launch planning, TMA descriptor
// encoding, kernel launches, and the device status word.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "../../include/hattn.h"
#include "common.cuh"
#include "kernels.h"

using namespace hattn;

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return code;
}

int ok() {
  g_last_error[0] = '\0';
  return HATTN_OK;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(HATTN_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// Device status word: one int per device, read and cleared by hattn_check_status.
__device__ int g_device_status[4];  // code, wait site, block, thread

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int* g_status_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};

bool device_info(int* dev_out, int** status, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess) return false;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    g_status_ptr[dev] = static_cast<int*>(p);
    g_num_sms[dev] = n;
  }
  if (dev_out) *dev_out = dev;
  if (status) *status = g_status_ptr[dev];
  if (sms) *sms = g_num_sms[dev];
  return true;
}

int num_sms_or_default() {
  int sms = 0;
  if (!device_info(nullptr, nullptr, &sms)) {
    cudaGetLastError();
    return 148;
  }
  return sms;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// bf16 tensor map, 128-byte swizzle.  dims/strides innermost first; strides
// in bytes for dims 1..rank-1.
int make_tmap(CUtensorMap* tm, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box, const char* what,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(HATTN_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides[i];
  CUresult r = fn(tm, dtype, rank, const_cast<void*>(base), gd, gs, bx,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(HATTN_ERR_CUDA, "tensor map for %s: CUresult %d", what, (int)r);
  return HATTN_OK;
}

#define REQUIRE(cond, ...)                                  \
  do {                                                      \
    if (!(cond)) return fail(HATTN_ERR_INVALID_ARG, __VA_ARGS__); \
  } while (0)
#define REQUIRE_PTR(p)                                                         \
  do {                                                                         \
    if (!(p)) return fail(HATTN_ERR_INVALID_ARG, "%s must not be NULL", #p);   \
    if (!aligned16(p)) return fail(HATTN_ERR_MISALIGNED, "%s is not 16-byte aligned", #p); \
  } while (0)
#define REQUIRE_F32(p)                                                         \
  do {                                                                         \
    if ((p) && !aligned4(p)) return fail(HATTN_ERR_MISALIGNED, "%s is not 4-byte aligned", #p); \
  } while (0)

int check_flags(int flags) {
  REQUIRE((flags & ~(HATTN_LAUNCH_DEPENDENT | HATTN_EVENT_EXTERNAL)) == 0,
          "flags=%d: unknown bits", flags);
  return HATTN_OK;
}

int check_rope(int D, int r, float rope_base, float eps) {
  REQUIRE(r >= 0 && r % 2 == 0 && r <= D && r <= 2 * kMaxRopePairs,
          "r=%d must be even, <= D and <= %d", r, 2 * kMaxRopePairs);
  REQUIRE(rope_base > 0.f, "rope_base must be positive");
  REQUIRE(eps >= 0.f, "eps must be >= 0");
  return HATTN_OK;
}

int compress_common(const void* kv_raw, const void* ik_raw, const void* gate,
                    const float* gamma_kv, int B, int64_t L_cap, int D, int dI, int m, int w,
                    int r, float rope_base, float eps, int64_t j_begin, int64_t j_end, void* kv_c,
                    void* ik_c, int64_t N_cap, hattn_stream_t stream, void* ik8 = nullptr,
                    float* ik_scale = nullptr, int64_t ring = 0, void* ik4 = nullptr,
                    void* ik4_scale = nullptr) {
  REQUIRE_PTR(kv_raw);
  REQUIRE_PTR(gate);
  REQUIRE_PTR(kv_c);
  REQUIRE_F32(gamma_kv);
  REQUIRE((ik8 == nullptr) == (ik_scale == nullptr), "ik8 and ik_scale must both be given or both NULL");
  REQUIRE((ik4 == nullptr) == (ik4_scale == nullptr),
          "ik4 and ik4_scale must both be given or both NULL");
  REQUIRE((ik_raw == nullptr) == (ik_c == nullptr && ik8 == nullptr),
          "ik_raw needs an indexer-key output (ik_c or ik8), and an output needs ik_raw");
  if (ik_raw) {
    REQUIRE_PTR(ik_raw);
    if (ik_c) REQUIRE_PTR(ik_c);
    if (ik8) {
      REQUIRE_PTR(ik8);
      REQUIRE_PTR(ik_scale);
    }
    if (ik4) {
      REQUIRE_PTR(ik4);
      REQUIRE_PTR(ik4_scale);
      REQUIRE(dI % 32 == 0, "MXFP4 indexer keys need dI a multiple of 32, got %d", dI);
    }
    REQUIRE(dI >= 8 && dI <= 128 && dI % 8 == 0, "dI=%d must be a multiple of 8 in [8, 128]", dI);
  }
  REQUIRE(B >= 1 && L_cap >= 1 && N_cap >= 1, "B, L_cap and N_cap must be >= 1");
  REQUIRE(D >= 64 && D <= 512 && D % 64 == 0, "D=%d must be a multiple of 64 in [64, 512]", D);
  REQUIRE(m >= 1 && w >= m && w % m == 0 && w <= 512, "need 1 <= m <= w <= 512, w %% m == 0 (m=%d w=%d)", m, w);
  int rc = check_rope(D, r, rope_base, eps);
  if (rc) return rc;
  REQUIRE(j_begin >= 0 && j_end >= j_begin && j_end <= N_cap, "entry range [%lld, %lld) outside [0, N_cap=%lld)",
          (long long)j_begin, (long long)j_end, (long long)N_cap);
  if (ring > 0) {
    // the raw buffers hold the last `ring` tokens: the window of every entry
    // compressed in this call must still be in it
    REQUIRE((ring & (ring - 1)) == 0 && ring == L_cap, "ring=%lld must be a power of two equal to L_cap",
            (long long)ring);
    REQUIRE((int64_t)m * (j_end - j_begin) + w - m <= ring,
            "entries [%lld, %lld) span more tokens than the ring of %lld holds", (long long)j_begin,
            (long long)j_end, (long long)ring);
  } else {
    REQUIRE((int64_t)m * j_end <= L_cap, "entry %lld needs tokens beyond L_cap=%lld", (long long)(j_end - 1),
            (long long)L_cap);
  }
  if (j_end == j_begin) return ok();
  CompressArgs a;
  a.kv_raw = static_cast<const __nv_bfloat16*>(kv_raw);
  a.ik_raw = static_cast<const __nv_bfloat16*>(ik_raw);
  a.gate = static_cast<const __nv_bfloat16*>(gate);
  a.gamma = gamma_kv;
  a.kv_out = static_cast<__nv_bfloat16*>(kv_c);
  a.ik_out = static_cast<__nv_bfloat16*>(ik_c);
  a.ik8_out = static_cast<uint8_t*>(ik8);
  a.ik_scale_out = ik_scale;
  a.ik4_out = static_cast<uint8_t*>(ik4);
  a.ik4_scale_out = static_cast<uint8_t*>(ik4_scale);
  a.B = B;
  a.D = D;
  a.dI = ik_raw ? dI : 0;
  a.m = m;
  a.w = w;
  a.r = r;
  a.L_cap = L_cap;
  a.N_cap = N_cap;
  a.j_begin = j_begin;
  a.j_end = j_end;
  a.ring = ring;
  a.eps = eps;
  make_rope_coef(rope_base, r, &a.rope);
  cudaError_t e = launch_compress(a, num_sms_or_default(), static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "compress launch");
  return ok();
}

// Bytes of the split partials of an attention call: [B*T*H][nsplit][D] fp32
// outputs, then [B*T*H][nsplit] fp32 log-sum-exps.
size_t partial_bytes(int B, int T, int H, int D, int nsplit) {
  return (size_t)B * T * H * nsplit * (D + 1) * sizeof(float);
}

// Bytes of the prepared-query copy at the start of an attention workspace
// (none when the caller passes prepared queries).
size_t qprep_bytes(int B, int T, int H, int D, int q_prepped) {
  return q_prepped ? 0 : (size_t)B * T * H * D * 2;
}

int query_prep_impl(const void* q, const float* gamma_q, const int32_t* pos, int B, int T, int H,
                    int D, int r, float rope_base, float eps, void* q_out,
                    hattn_stream_t stream) {
  REQUIRE_PTR(q);
  REQUIRE_PTR(pos);
  REQUIRE_PTR(q_out);
  REQUIRE_F32(gamma_q);
  REQUIRE(B >= 1 && T >= 1 && H >= 1, "B, T and H must be >= 1");
  REQUIRE(D >= 64 && D <= 512 && D % 64 == 0, "D=%d must be a multiple of 64 in [64, 512]", D);
  int rc = check_rope(D, r, rope_base, eps);
  if (rc) return rc;
  QPrepArgs a;
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.gamma = gamma_q;
  a.pos = pos;
  a.q_out = static_cast<__nv_bfloat16*>(q_out);
  a.B = B;
  a.T = T;
  a.H = H;
  a.D = D;
  a.r = r;
  a.eps = eps;
  make_rope_coef(rope_base, r, &a.rope);
  cudaError_t e = launch_qprep(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "query prep launch");
  return HATTN_OK;
}

// The fused call's second and third key sources.
// The layer output of a fused call: the sink merge and the inverse RoPE
// applied to its single softmax (hattn_hybrid_attn_out).
struct FinalOut {
  void* out;          // [B][T][H][D] bf16
  float* lse_out;     // [B][T][H] or null
  const float* sink;  // [H] or null
};

int merge_impl(const void* const* o_list, const float* const* lse_list, const int* nsplit, int nb,
               const float* sink, const int32_t* pos, int B, int T, int H, int D, int r,
               float rope_base, void* out, float* lse_out, hattn_stream_t stream, int flags);

struct FusedSources {
  const void* kv_h;   // [B][N_h][D] HCA entries
  int64_t N_h;
  const void* kv_w;   // [B][T][W][D] SWA keys (hattn_swa_keys)
  int segments;       // bit 0: CSA, bit 1: HCA, bit 2: SWA
  int n_sms;          // SMs the split plan may assume (0: all)
};

// Keys the fused call plans for: each segment it covers rounded up to whole
// tiles.
int64_t fused_keys(int k, int64_t N_h, int W, int segments) {
  auto up = [](int64_t n) { return (n + 63) / 64 * 64; };
  return ((segments & 1) ? up(k) : 0) + ((segments & 2) ? up(N_h) : 0) +
         ((segments & 4) ? up(W) : 0);
}

int fused_sms(int n_sms) {
  const int all = num_sms_or_default();
  return n_sms > 0 && n_sms < all ? n_sms : all;
}

int attn_common(int kind, const void* q, const float* gamma_q, int q_prepped, const void* kv,
                const float* gamma_kv, const int32_t* idx, const int32_t* pos, int B, int T, int H,
                int D, int64_t N_rows, int k, int m, int W, int r, float rope_base, float eps,
                float scale, void* o, float* lse, void* workspace, size_t ws_bytes,
                hattn_stream_t stream, const FusedSources* fs = nullptr, int flags = 0,
                const FinalOut* fo = nullptr) {
  if (int rcf = check_flags(flags)) return rcf;
  const bool dependent = (flags & HATTN_LAUNCH_DEPENDENT) != 0;
  REQUIRE_PTR(q);
  if (kind != kFused || (fs && (fs->segments & 1))) REQUIRE_PTR(kv);
  REQUIRE_PTR(pos);
  if (fo) {
    REQUIRE_PTR(fo->out);
    REQUIRE_F32(fo->lse_out);
    REQUIRE_F32(fo->sink);
  }
  // o == lse == NULL: leave the split partials in the workspace for
  // hattn_lse_merge_splits instead of combining them (or, with a final
  // output, for this call's own merge when the keys take several splits)
  const bool partials = o == nullptr && lse == nullptr;
  if (!partials) {
    REQUIRE_PTR(o);
    REQUIRE(lse != nullptr, "lse must not be NULL when o is given");
    REQUIRE_F32(lse);
  }
  REQUIRE_F32(gamma_q);
  REQUIRE_F32(gamma_kv);
  if (kind == kSparse) REQUIRE_PTR(idx);
  if (kind == kFused) {
    REQUIRE(fs != nullptr, "fused sources missing");
    REQUIRE(fs->segments >= 1 && fs->segments <= 7, "segments=%d must be a mask in [1, 7]",
            fs->segments);
    REQUIRE(fs->n_sms >= 0, "n_sms=%d must be >= 0", fs->n_sms);
    if (fs->segments & 1) REQUIRE_PTR(idx);
    if (fs->segments & 2) {
      REQUIRE_PTR(fs->kv_h);
      REQUIRE(fs->N_h >= 1, "the HCA cache needs at least one row");
      REQUIRE((int64_t)B * fs->N_h < (1ll << 31), "B * N_h must be < 2^31");
    }
    if (fs->segments & 4) {
      REQUIRE_PTR(fs->kv_w);
      REQUIRE((int64_t)B * T * W < (1ll << 31), "B * T * W must be < 2^31");
    }
  }
  REQUIRE(B >= 1 && T >= 1, "B and T must be >= 1");
  REQUIRE(H >= 1 && H <= 128, "H=%d must be in [1, 128]", H);
  REQUIRE(D >= 64 && D <= 512 && D % 64 == 0, "D=%d must be a multiple of 64 in [64, 512]", D);
  REQUIRE(N_rows >= 1, "the key cache needs at least one row");
  REQUIRE((int64_t)B * N_rows < (1ll << 31), "B * rows of the cache must be < 2^31");
  const int segs = kind == kFused ? fs->segments : 0;
  if (kind == kSparse || (segs & 1)) REQUIRE(k >= 1 && k <= 65536, "k=%d out of range", k);
  if (kind == kHca || (segs & 2)) REQUIRE(m >= 1, "m must be >= 1");
  if (kind == kSwa || (segs & 4)) REQUIRE(W >= 1 && W <= 65536, "W=%d out of range", W);
  REQUIRE(scale > 0.f, "scale must be positive");
  int rc = check_rope(D, r, rope_base, eps);
  if (rc) return rc;
  const int64_t n_keys = kind == kFused ? fused_keys(k, fs->N_h, W, fs->segments)
                                         : (kind == kSparse ? k : (kind == kHca ? N_rows : W));
  AttnPlan p;
  if (!plan_attention(kind, B, T, H, D, n_keys,
                      kind == kFused ? fused_sms(fs->n_sms) : num_sms_or_default(), &p))
    return fail(HATTN_ERR_UNSUPPORTED, "no attention kernel for H=%d D=%d", H, D);
  const size_t qbytes = qprep_bytes(B, T, H, D, q_prepped);
  // a final output in one split needs no partials
  const bool final_direct = fo && p.nsplit == 1;
  const size_t pbytes = final_direct ? 0
                        : (partials ? partial_bytes(B, T, H, D, p.nsplit) : p.ws_bytes);
  const size_t need = qbytes + pbytes;
  if (need > 0) {
    REQUIRE_PTR(workspace);
    REQUIRE(ws_bytes >= need, "workspace of %zu bytes, need %zu", ws_bytes, need);
  }
  int* status = nullptr;
  if (!device_info(nullptr, &status, nullptr)) return fail(HATTN_ERR_CUDA, "no CUDA device");
  CUtensorMap tm, tm2, tm_q;
  memset(&tm, 0, sizeof tm);
  memset(&tm2, 0, sizeof tm2);
  // Streamed keys arrive as groups of gsz 64-dim chunks (one CTA's share of
  // a row's dims): a 3-D view {64 dims, rows, D/64 chunks} of the row-major
  // cache, copied as boxes of {64, 64 keys, gsz} (8 KB per chunk, 128-byte
  // swizzle, chunk after chunk in shared memory).
  const int gsz = D / 64 / p.nds;
  auto key_map = [&](CUtensorMap* m, const void* base, uint64_t rows, const char* what) {
    const uint64_t dims[3] = {64, rows, (uint64_t)D / 64};
    const uint64_t strides[2] = {(uint64_t)D * 2, 128};
    const uint32_t box[3] = {64, 64, (uint32_t)gsz};
    return make_tmap(m, base, 3, dims, strides, box, what);
  };
  if (kind == kHca || kind == kSwa) {
    rc = key_map(&tm, kv, (uint64_t)B * (uint64_t)N_rows, kind == kHca ? "kv_h" : "kv_raw");
    if (rc) return rc;
  } else if (kind == kFused) {
    if (fs->segments & 2) {
      rc = key_map(&tm, fs->kv_h, (uint64_t)B * (uint64_t)fs->N_h, "kv_h");
      if (rc) return rc;
    }
    if (fs->segments & 4) {
      rc = key_map(&tm2, fs->kv_w, (uint64_t)B * (uint64_t)T * (uint64_t)W, "kv_w");
      if (rc) return rc;
    }
  }
  // prepared queries: the caller's, or this call's into the workspace
  const void* qt = q_prepped ? q : workspace;
  {
    // query rows of a row block: 128 rows x 64 dims per copy
    const uint64_t dims[2] = {(uint64_t)D, (uint64_t)B * (uint64_t)T * (uint64_t)H};
    const uint64_t strides[1] = {(uint64_t)D * 2};
    const uint32_t box[2] = {64, 128};
    rc = make_tmap(&tm_q, qt, 2, dims, strides, box, "q");
    if (rc) return rc;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (!q_prepped) {
    rc = query_prep_impl(q, gamma_q, pos, B, T, H, D, r, rope_base, eps, workspace, stream);
    if (rc) return rc;
  }
  AttnArgs a;
  a.q = static_cast<const __nv_bfloat16*>(qt);
  a.kv = static_cast<const __nv_bfloat16*>(kv);
  a.gamma_kv = gamma_kv;
  a.idx = idx;
  a.pos = pos;
  a.o = static_cast<float*>(o);
  a.lse = lse;
  float* ws = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + qbytes);
  const int64_t rows = (int64_t)B * T * H;
  const bool split_out = !final_direct && (partials || p.nsplit > 1);
  a.part_o = split_out ? ws : nullptr;
  a.part_lse = split_out ? ws + rows * p.nsplit * D : nullptr;
  a.partials = partials && !final_direct ? 1 : 0;
  a.out = final_direct ? static_cast<__nv_bfloat16*>(fo->out) : nullptr;
  a.lse_out = final_direct ? fo->lse_out : nullptr;
  a.sink = final_direct ? fo->sink : nullptr;
  a.status = status;
  a.kind = kind;
  a.B = B;
  a.T = T;
  a.H = H;
  a.D = D;
  a.r = r;
  a.N_rows = N_rows;
  a.N_h = fs ? fs->N_h : 0;
  a.segments = fs ? fs->segments : 0;
  a.k = k;
  a.m = m;
  a.W = W;
  a.eps = eps;
  a.scale = scale;
  make_rope_coef(rope_base, r, &a.rope);
  a.G = p.G;
  a.n_rb = p.n_rb;
  a.nsplit = p.nsplit;
  a.keys_per_split = p.keys_per_split;
  a.nds = p.nds;
  a.n_tq = p.n_tq;
  // the attention kernel is a dependent of the query preparation it follows
  a.dependent = (dependent || !q_prepped) ? 1 : 0;
  cudaError_t e = launch_attention(tm, tm2, tm_q, a, p, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  if (fo && !final_direct) {
    // several key splits: the merge of this call's partials with the sink
    const void* ol[1] = {a.part_o};
    const float* ll[1] = {a.part_lse};
    const int ns[1] = {p.nsplit};
    return merge_impl(ol, ll, ns, 1, fo->sink, pos, B, T, H, D, r, rope_base, fo->out,
                      fo->lse_out, stream, HATTN_LAUNCH_DEPENDENT);
  }
  if (p.nsplit > 1 && !partials) {
    CombineArgs c;
    c.part_o = a.part_o;
    c.part_lse = a.part_lse;
    c.o = a.o;
    c.lse = lse;
    c.rows = rows;
    c.nsplit = p.nsplit;
    c.D = D;
    c.dependent = 1;  // follows the attention kernel it combines
    e = launch_combine(c, st);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
  }
  return ok();
}

}  // namespace

namespace hattn {

int add_dependent_attr(cudaLaunchAttribute* attrs, int n, bool dependent) {
  if (!dependent) return n;
  attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[n].val.programmaticStreamSerializationAllowed = 1;
  return n + 1;
}

void make_rope_coef(double base, int r, RopeCoef* rc) {
  memset(rc, 0, sizeof *rc);
  const double two_pi = 6.283185307179586476925286766559;
  for (int i = 0; i < r / 2 && i < kMaxRopePairs; ++i) {
    const double theta = pow(base, -2.0 * i / static_cast<double>(r));
    const double f = theta / two_pi;           // turns per position
    const double g = fmod(4096.0 * f, 1.0);    // turns per 4096 positions, reduced
    rc->c[0][i] = static_cast<float>(f);
    rc->c[1][i] = static_cast<float>(f - static_cast<double>(rc->c[0][i]));
    rc->c[2][i] = static_cast<float>(g);
    rc->c[3][i] = static_cast<float>(g - static_cast<double>(rc->c[2][i]));
  }
}

}  // namespace hattn

extern "C" {

int hattn_csa_compress(const void* kv_raw, const void* ik_raw, const void* gate,
                       const float* gamma_kv, int B, int64_t L_cap, int D, int dI, int m, int w,
                       int r, float rope_base, float eps, int64_t j_begin, int64_t j_end,
                       void* kv_c, void* ik_c, int64_t N_cap, hattn_stream_t stream) {
  return compress_common(kv_raw, ik_raw, gate, gamma_kv, B, L_cap, D, dI, m, w, r, rope_base, eps,
                         j_begin, j_end, kv_c, ik_c, N_cap, stream);
}

int hattn_csa_compress_fp8(const void* kv_raw, const void* ik_raw, const void* gate,
                           const float* gamma_kv, int B, int64_t L_cap, int D, int dI, int m,
                           int w, int r, float rope_base, float eps, int64_t j_begin,
                           int64_t j_end, void* kv_c, void* ik_c, void* ik8, float* ik_scale,
                           int64_t N_cap, hattn_stream_t stream) {
  REQUIRE_PTR(ik_raw);
  REQUIRE_PTR(ik8);
  REQUIRE_PTR(ik_scale);
  return compress_common(kv_raw, ik_raw, gate, gamma_kv, B, L_cap, D, dI, m, w, r, rope_base, eps,
                         j_begin, j_end, kv_c, ik_c, N_cap, stream, ik8, ik_scale);
}

int hattn_csa_compress_mxfp4(const void* kv_raw, const void* ik_raw, const void* gate,
                             const float* gamma_kv, int B, int64_t L_cap, int D, int dI, int m,
                             int w, int r, float rope_base, float eps, int64_t j_begin,
                             int64_t j_end, void* kv_c, void* ik_c, void* ik4, void* ik4_scale,
                             int64_t N_cap, hattn_stream_t stream) {
  REQUIRE_PTR(ik_raw);
  REQUIRE_PTR(ik_c);
  REQUIRE_PTR(ik4);
  REQUIRE_PTR(ik4_scale);
  return compress_common(kv_raw, ik_raw, gate, gamma_kv, B, L_cap, D, dI, m, w, r, rope_base, eps,
                         j_begin, j_end, kv_c, ik_c, N_cap, stream, nullptr, nullptr, 0, ik4,
                         ik4_scale);
}

int hattn_csa_compress_ring(const void* kv_ring, const void* ik_ring, const void* gate_ring,
                            const float* gamma_kv, int B, int64_t ring, int D, int dI, int m,
                            int w, int r, float rope_base, float eps, int64_t j_begin,
                            int64_t j_end, void* kv_c, void* ik_c, int64_t N_cap,
                            hattn_stream_t stream) {
  REQUIRE(ring >= 1, "ring=%lld must be >= 1", (long long)ring);
  return compress_common(kv_ring, ik_ring, gate_ring, gamma_kv, B, ring, D, dI, m, w, r, rope_base,
                         eps, j_begin, j_end, kv_c, ik_c, N_cap, stream, nullptr, nullptr, ring);
}

int hattn_hca_compress_ring(const void* kv_ring, const void* gate_ring, const float* gamma_kv,
                            int B, int64_t ring, int D, int m, int r, float rope_base, float eps,
                            int64_t j_begin, int64_t j_end, void* kv_h, int64_t N_cap,
                            hattn_stream_t stream) {
  REQUIRE(ring >= 1, "ring=%lld must be >= 1", (long long)ring);
  return compress_common(kv_ring, nullptr, gate_ring, gamma_kv, B, ring, D, 0, m, m, r, rope_base,
                         eps, j_begin, j_end, kv_h, nullptr, N_cap, stream, nullptr, nullptr, ring);
}

size_t hattn_compress_hidden_workspace_bytes(int B, int64_t j_begin, int64_t j_end, int dm, int D,
                                             int dI) {
  if (B < 1 || j_end <= j_begin || dm < 1 || D < 1 || dI < 0) return 0;
  return hidden_workspace_bytes((int64_t)B * (j_end - j_begin), dm, D + dI);
}

int hattn_compress_hidden(const void* x, const void* W, const void* gate, const float* gamma_kv,
                          int B, int64_t L_cap, int dm, int D, int dI, int m, int w, int r,
                          float rope_base, float eps, int64_t j_begin, int64_t j_end, void* kv_out,
                          void* ik_out, int64_t N_cap, void* workspace, size_t ws_bytes,
                          hattn_stream_t stream) {
  REQUIRE_PTR(x);
  REQUIRE_PTR(W);
  REQUIRE_PTR(gate);
  REQUIRE_PTR(kv_out);
  REQUIRE_F32(gamma_kv);
  REQUIRE((ik_out == nullptr) == (dI == 0), "ik_out must be given exactly when dI > 0");
  if (ik_out) REQUIRE_PTR(ik_out);
  REQUIRE(B >= 1 && L_cap >= 1 && N_cap >= 1, "B, L_cap and N_cap must be >= 1");
  REQUIRE(dm >= 8 && dm % 8 == 0, "dm=%d must be a positive multiple of 8", dm);
  REQUIRE(D >= 64 && D <= 512 && D % 64 == 0, "D=%d must be a multiple of 64 in [64, 512]", D);
  REQUIRE(dI == 0 || (dI >= 8 && dI <= 128 && dI % 8 == 0),
          "dI=%d must be 0 or a multiple of 8 in [8, 128]", dI);
  REQUIRE(m >= 1 && w >= m && w % m == 0 && w <= 512,
          "need 1 <= m <= w <= 512, w %% m == 0 (m=%d w=%d)", m, w);
  int rc = check_rope(D, r, rope_base, eps);
  if (rc) return rc;
  REQUIRE(j_begin >= 0 && j_end >= j_begin && j_end <= N_cap,
          "entry range [%lld, %lld) outside [0, N_cap=%lld)", (long long)j_begin,
          (long long)j_end, (long long)N_cap);
  REQUIRE((int64_t)m * j_end <= L_cap, "entry %lld needs tokens beyond L_cap=%lld",
          (long long)(j_end - 1), (long long)L_cap);
  if (j_end == j_begin) return ok();
  const size_t need = hattn_compress_hidden_workspace_bytes(B, j_begin, j_end, dm, D, dI);
  REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= need, "workspace of %zu bytes, need %zu", ws_bytes, need);
  HiddenArgs a;
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.W = static_cast<const __nv_bfloat16*>(W);
  a.gate = static_cast<const __nv_bfloat16*>(gate);
  a.gamma = gamma_kv;
  a.kv_out = static_cast<__nv_bfloat16*>(kv_out);
  a.ik_out = static_cast<__nv_bfloat16*>(ik_out);
  a.B = B;
  a.dm = dm;
  a.D = D;
  a.dI = dI;
  a.m = m;
  a.w = w;
  a.r = r;
  a.L_cap = L_cap;
  a.N_cap = N_cap;
  a.j_begin = j_begin;
  a.j_end = j_end;
  a.eps = eps;
  make_rope_coef(rope_base, r, &a.rope);
  int sms = 0;
  int* status = nullptr;
  if (!device_info(nullptr, &status, &sms)) return fail(HATTN_ERR_CUDA, "no CUDA device");
  // the projection's operands: the pooled parts of a chunk (rows past the
  // chunk's entries read zeros or the previous chunk's rows, and their
  // outputs are not written) and W, all in 128-byte swizzled boxes
  const size_t ce = hidden_chunk_entries((int64_t)B * (j_end - j_begin));
  CUtensorMap tm_ah, tm_al, tm_w;
  {
    const uint64_t dims[2] = {(uint64_t)dm, (uint64_t)ce};
    const uint64_t strides[1] = {(uint64_t)dm * 2};
    const uint32_t box[2] = {64, 128};
    rc = make_tmap(&tm_ah, workspace, 2, dims, strides, box, "pooled hi");
    if (rc) return rc;
    rc = make_tmap(&tm_al, static_cast<uint8_t*>(workspace) + hidden_part_bytes(ce, dm), 2, dims,
                   strides, box, "pooled lo");
    if (rc) return rc;
  }
  {
    const uint64_t dims[2] = {(uint64_t)(D + dI), (uint64_t)dm};
    const uint64_t strides[1] = {(uint64_t)(D + dI) * 2};
    const uint32_t box[2] = {64, 64};
    rc = make_tmap(&tm_w, W, 2, dims, strides, box, "W");
    if (rc) return rc;
  }
  cudaError_t e = launch_compress_hidden(a, workspace, sms, tm_ah, tm_al, tm_w, status,
                                         static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "compress from hidden states");
  return ok();
}

size_t hattn_compress_hidden_pair_workspace_bytes(int B, int64_t L, int64_t N_c, int64_t N_h,
                                                  int dm) {
  if (B < 1 || L < 1 || dm < 8) return 0;
  const int64_t nc = N_c < L / 4 ? N_c : L / 4, nh = N_h < L / 128 ? N_h : L / 128;
  if (nc <= 0) return 0;
  return hidden_pair_workspace_bytes(B, nc, nh, dm);
}

int hattn_compress_hidden_pair(const void* x, const void* W_c, const void* gate_c,
                               const void* W_h, const void* gate_h, const float* gamma_kv, int B,
                               int64_t L_cap, int64_t L, int dm, int D, int dI, int r,
                               float rope_base, float eps, void* kv_c, void* ik_c, int64_t N_c,
                               void* kv_h, int64_t N_h, void* workspace, size_t ws_bytes,
                               hattn_stream_t stream) {
  REQUIRE_PTR(x);
  REQUIRE_PTR(W_c);
  REQUIRE_PTR(gate_c);
  REQUIRE_PTR(W_h);
  REQUIRE_PTR(gate_h);
  REQUIRE_PTR(kv_c);
  REQUIRE_PTR(kv_h);
  REQUIRE_F32(gamma_kv);
  REQUIRE((ik_c == nullptr) == (dI == 0), "ik_c must be given exactly when dI > 0");
  if (ik_c) REQUIRE_PTR(ik_c);
  REQUIRE(B >= 1 && L_cap >= 1 && N_c >= 1 && N_h >= 1, "B, L_cap, N_c and N_h must be >= 1");
  REQUIRE(L >= 0 && L <= L_cap, "L=%lld must be in [0, L_cap=%lld]", (long long)L,
          (long long)L_cap);
  REQUIRE(dm >= 8 && dm % 8 == 0, "dm=%d must be a positive multiple of 8", dm);
  REQUIRE(D >= 64 && D <= 512 && D % 64 == 0, "D=%d must be a multiple of 64 in [64, 512]", D);
  REQUIRE(dI == 0 || (dI >= 8 && dI <= 128 && dI % 8 == 0),
          "dI=%d must be 0 or a multiple of 8 in [8, 128]", dI);
  int rc = check_rope(D, r, rope_base, eps);
  if (rc) return rc;
  const int64_t nc = N_c < L / 4 ? N_c : L / 4, nh = N_h < L / 128 ? N_h : L / 128;
  // the HCA entries ride on the CSA pass's 128-token blocks
  REQUIRE(nh <= (nc + 31) / 32, "N_c=%lld holds too few CSA entries for the %lld HCA entries",
          (long long)N_c, (long long)nh);
  if (nc == 0) return ok();
  const size_t need = hidden_pair_workspace_bytes(B, nc, nh, dm);
  REQUIRE_PTR(workspace);
  REQUIRE(ws_bytes >= need, "workspace of %zu bytes, need %zu", ws_bytes, need);
  HiddenArgs ac;
  ac.x = static_cast<const __nv_bfloat16*>(x);
  ac.W = static_cast<const __nv_bfloat16*>(W_c);
  ac.gate = static_cast<const __nv_bfloat16*>(gate_c);
  ac.gamma = gamma_kv;
  ac.kv_out = static_cast<__nv_bfloat16*>(kv_c);
  ac.ik_out = static_cast<__nv_bfloat16*>(ik_c);
  ac.B = B;
  ac.dm = dm;
  ac.D = D;
  ac.dI = dI;
  ac.m = 4;
  ac.w = 8;
  ac.r = r;
  ac.L_cap = L_cap;
  ac.N_cap = N_c;
  ac.j_begin = 0;
  ac.j_end = nc;
  ac.eps = eps;
  make_rope_coef(rope_base, r, &ac.rope);
  HiddenArgs ah = ac;
  ah.W = static_cast<const __nv_bfloat16*>(W_h);
  ah.gate = static_cast<const __nv_bfloat16*>(gate_h);
  ah.kv_out = static_cast<__nv_bfloat16*>(kv_h);
  ah.ik_out = nullptr;
  ah.dI = 0;
  ah.m = 128;
  ah.w = 128;
  ah.N_cap = N_h;
  ah.j_end = nh;
  int sms = 0;
  int* status = nullptr;
  if (!device_info(nullptr, &status, &sms)) return fail(HATTN_ERR_CUDA, "no CUDA device");
  const int64_t rows_c = (int64_t)B * nc < kHiddenChunk ? (int64_t)B * nc : kHiddenChunk;
  const int64_t rows_h = (int64_t)B * nh;
  uint8_t* wsb = static_cast<uint8_t*>(workspace);
  CUtensorMap tm_ch, tm_cl, tm_wc, tm_hh, tm_hl, tm_wh;
  auto part_map = [&](CUtensorMap* m, const void* base, int64_t rows, const char* what) {
    const uint64_t dims[2] = {(uint64_t)dm, (uint64_t)(rows > 0 ? rows : 1)};
    const uint64_t strides[1] = {(uint64_t)dm * 2};
    const uint32_t box[2] = {64, 128};
    return make_tmap(m, base, 2, dims, strides, box, what);
  };
  auto w_map = [&](CUtensorMap* m, const void* base, int P, const char* what) {
    const uint64_t dims[2] = {(uint64_t)P, (uint64_t)dm};
    const uint64_t strides[1] = {(uint64_t)P * 2};
    const uint32_t box[2] = {64, 64};
    return make_tmap(m, base, 2, dims, strides, box, what);
  };
  const size_t pc = hidden_part_bytes(rows_c, dm), ph = hidden_part_bytes(rows_h, dm);
  if ((rc = part_map(&tm_ch, wsb, rows_c, "CSA pooled hi")) ||
      (rc = part_map(&tm_cl, wsb + pc, rows_c, "CSA pooled lo")) ||
      (rc = part_map(&tm_hh, wsb + 2 * pc, rows_h, "HCA pooled hi")) ||
      (rc = part_map(&tm_hl, wsb + 2 * pc + ph, rows_h, "HCA pooled lo")) ||
      (rc = w_map(&tm_wc, W_c, D + dI, "W_c")) || (rc = w_map(&tm_wh, W_h, D, "W_h")))
    return rc;
  cudaError_t e = launch_compress_hidden_pair(ac, ah, workspace, sms, tm_ch, tm_cl, tm_wc, tm_hh,
                                              tm_hl, tm_wh, status,
                                              static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "compress pair from hidden states");
  return ok();
}

int hattn_quantize_e4m3(const void* x, int64_t rows, int n, void* codes, float* scales,
                        hattn_stream_t stream) {
  REQUIRE(rows >= 0, "rows must be >= 0");
  REQUIRE(n >= 4 && n % 4 == 0 && n <= (1 << 20), "n=%d must be a multiple of 4 in [4, 2^20]", n);
  if (rows == 0) return ok();  // nothing to read or write: any pointers
  REQUIRE_PTR(x);
  REQUIRE_PTR(codes);
  REQUIRE_PTR(scales);
  cudaError_t e = launch_quantize_e4m3(static_cast<const __nv_bfloat16*>(x), rows, n,
                                       static_cast<uint8_t*>(codes), scales, num_sms_or_default(),
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return ok();
}

int hattn_quantize_mxfp4(const void* x, int64_t rows, int n, void* codes, void* scales,
                         hattn_stream_t stream) {
  REQUIRE(rows >= 0, "rows must be >= 0");
  REQUIRE(n >= 32 && n % 32 == 0 && n <= (1 << 20), "n=%d must be a multiple of 32 in [32, 2^20]",
          n);
  if (rows == 0) return ok();  // nothing to read or write: any pointers
  REQUIRE_PTR(x);
  REQUIRE_PTR(codes);
  REQUIRE_PTR(scales);
  cudaError_t e = launch_quantize_mxfp4(static_cast<const __nv_bfloat16*>(x), rows, n,
                                        static_cast<uint8_t*>(codes),
                                        static_cast<uint8_t*>(scales), num_sms_or_default(),
                                        static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return ok();
}

int hattn_quantize_mxfp4_entries(const void* x, int B, int64_t N_cap, int n, int64_t j_begin,
                                 int64_t j_end, void* codes, void* scales, hattn_stream_t stream) {
  REQUIRE(B >= 1 && N_cap >= 1, "B and N_cap must be >= 1");
  REQUIRE(n >= 32 && n % 32 == 0 && n <= (1 << 20), "n=%d must be a multiple of 32 in [32, 2^20]",
          n);
  REQUIRE(j_begin >= 0 && j_end >= j_begin && j_end <= N_cap,
          "entry range [%lld, %lld) outside [0, N_cap=%lld)", (long long)j_begin,
          (long long)j_end, (long long)N_cap);
  if (j_end == j_begin) return ok();
  REQUIRE_PTR(x);
  REQUIRE_PTR(codes);
  REQUIRE_PTR(scales);
  cudaError_t e = launch_quantize_mxfp4(
      static_cast<const __nv_bfloat16*>(x), (int64_t)B * (j_end - j_begin), n,
      static_cast<uint8_t*>(codes), static_cast<uint8_t*>(scales), num_sms_or_default(),
      static_cast<cudaStream_t>(stream), j_end - j_begin, j_begin, N_cap);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return ok();
}

int hattn_hca_compress(const void* kv_raw, const void* gate, const float* gamma_kv, int B,
                       int64_t L_cap, int D, int m, int r, float rope_base, float eps,
                       int64_t j_begin, int64_t j_end, void* kv_h, int64_t N_cap,
                       hattn_stream_t stream) {
  return compress_common(kv_raw, nullptr, gate, gamma_kv, B, L_cap, D, 0, m, m, r, rope_base, eps,
                         j_begin, j_end, kv_h, nullptr, N_cap, stream);
}

}  // extern "C"

namespace {

// Scores of bf16 indexer keys (ik_c), or of E4M3 keys when k_scale is given
// (ik_c then holds the codes, [B][N_cap][128] bytes), or with mx of MXFP4
// keys (ik_c the codes [B][N_cap][64] bytes, k_scale the E8M0 scales
// [B][N_cap][4] bytes).
// hist_part: the folded first selection pass (IndexerArgs::hist_part; the
// caller has checked fold_plan), else nullptr.  grid_out: the CTAs launched.
int indexer_scores_impl(const void* iq, const float* w, const void* ik_c, const int32_t* pos,
                        int B, int T, int HI, int dI, int64_t N_cap, int m, float* scores,
                        hattn_stream_t stream, int n_sms = 0, int64_t fresh_from = -1,
                        const void* k_scale = nullptr, int flags = 0,
                        uint16_t* hist_part = nullptr, int64_t* grid_out = nullptr,
                        bool mx = false) {
  if (int rcf = check_flags(flags)) return rcf;
  REQUIRE_PTR(iq);
  REQUIRE_PTR(w);
  REQUIRE_PTR(ik_c);
  REQUIRE_PTR(pos);
  REQUIRE_PTR(scores);
  REQUIRE(B >= 1 && T >= 1 && N_cap >= 1, "B, T and N_cap must be >= 1");
  REQUIRE(HI >= 1 && HI <= 256, "HI=%d must be in [1, 256]", HI);
  REQUIRE(dI >= 8 && dI <= 128 && dI % 8 == 0, "dI=%d must be a multiple of 8 in [8, 128]", dI);
  REQUIRE(m >= 1, "m must be >= 1");
  REQUIRE((int64_t)B * T * HI < (1ll << 31), "too many query heads");
  REQUIRE(n_sms >= 0, "n_sms=%d must be >= 0", n_sms);
  const bool f8 = k_scale != nullptr && !mx;
  if (f8 || mx) {
    REQUIRE_PTR(k_scale);
    REQUIRE(dI == 128, "%s indexer keys need dI = 128, got %d", mx ? "MXFP4" : "FP8", dI);
    REQUIRE(N_cap % 4 == 0, "%s indexer keys need N_cap %% 4 == 0 (16-byte scale rows), got %lld",
            mx ? "MXFP4" : "FP8", (long long)N_cap);
  }
  const int keys = mx ? kIdxKeysMx4 : (f8 ? kIdxKeysE4m3 : kIdxKeysBf16);
  IndexerPlan ip;
  if (!plan_indexer(T, HI, dI, keys, hist_part != nullptr, &ip))
    return fail(HATTN_ERR_UNSUPPORTED, "no indexer kernel for HI=%d dI=%d", HI, dI);
  int sms = 0;
  int* status = nullptr;
  if (!device_info(nullptr, &status, &sms)) return fail(HATTN_ERR_CUDA, "no CUDA device");
  CUtensorMap tm_ik, tm_iq, tm_ks;
  if (mx) {
    // a key block: 128 rows of 64 code bytes, 64-byte swizzled (the layout
    // the block-scaled products read); its scales as 32 rows of 16 bytes
    // (4 keys each)
    const uint64_t dims[3] = {64, (uint64_t)N_cap, (uint64_t)B};
    const uint64_t strides[2] = {64, (uint64_t)N_cap * 64};
    const uint32_t box[3] = {64, 128, 1};
    int rc = make_tmap(&tm_ik, ik_c, 3, dims, strides, box, "ik4", CU_TENSOR_MAP_DATA_TYPE_UINT8,
                       CU_TENSOR_MAP_SWIZZLE_64B);
    if (rc) return rc;
    const uint64_t sdims[3] = {16, (uint64_t)N_cap / 4, (uint64_t)B};
    const uint64_t sstrides[2] = {16, (uint64_t)N_cap * 4};
    const uint32_t sbox[3] = {16, 32, 1};
    rc = make_tmap(&tm_ks, k_scale, 3, sdims, sstrides, sbox, "ik4_scale",
                   CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  } else if (f8) {
    const uint64_t dims[3] = {128, (uint64_t)N_cap, (uint64_t)B};
    const uint64_t strides[2] = {128, (uint64_t)N_cap * 128};
    const uint32_t box[3] = {128, 128, 1};
    int rc = make_tmap(&tm_ik, ik_c, 3, dims, strides, box, "ik8", CU_TENSOR_MAP_DATA_TYPE_UINT8);
    if (rc) return rc;
    // the 128 row scales of a key block, beside its codes
    const uint64_t sdims[2] = {(uint64_t)N_cap, (uint64_t)B};
    const uint64_t sstrides[1] = {(uint64_t)N_cap * 4};
    const uint32_t sbox[2] = {128, 1};
    rc = make_tmap(&tm_ks, k_scale, 2, sdims, sstrides, sbox, "ik_scale",
                   CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (rc) return rc;
  } else {
    const uint64_t dims[3] = {(uint64_t)dI, (uint64_t)N_cap, (uint64_t)B};
    const uint64_t strides[2] = {(uint64_t)dI * 2, (uint64_t)N_cap * dI * 2};
    const uint32_t box[3] = {64, 128, 1};
    int rc = make_tmap(&tm_ik, ik_c, 3, dims, strides, box, "ik_c");
    if (rc) return rc;
    tm_ks = tm_ik;  // unused without FP8 keys
  }
  {
    const uint64_t dims[2] = {(uint64_t)dI, (uint64_t)B * T * HI};
    const uint64_t strides[1] = {(uint64_t)dI * 2};
    const uint32_t box[2] = {64, (uint32_t)ip.NQ};
    int rc = make_tmap(&tm_iq, iq, 2, dims, strides, box, "iq");
    if (rc) return rc;
  }
  IndexerArgs a;
  a.w = w;
  a.pos = pos;
  a.scores = scores;
  a.status = status;
  a.B = B;
  a.T = T;
  a.HI = HI;
  a.dI = dI;
  a.m = m;
  a.G = ip.G;
  a.NQ = ip.NQ;
  a.KC = ip.KC;
  a.stages = ip.stages;
  a.nacc = ip.nacc;
  a.groups_per_seq = (T + ip.G - 1) / ip.G;
  a.nblk = static_cast<int>((N_cap + 127) / 128);
  a.fresh_from = fresh_from;
  a.dependent = (flags & HATTN_LAUNCH_DEPENDENT) ? 1 : 0;
  a.N_cap = N_cap;
  a.total_slots = (int64_t)B * a.groups_per_seq * a.nblk;
  // persistent: one CTA per SM it may use (n_sms of them when given, so
  // that concurrent work keeps the others)
  if (n_sms > 0 && n_sms < sms) sms = n_sms;
  const int grid = static_cast<int>(a.total_slots < sms ? a.total_slots : sms);
  a.hist_part = hist_part;
  if (grid_out) *grid_out = grid;
  cudaError_t e =
      launch_indexer_score(tm_ik, tm_iq, tm_ks, a, ip, keys, grid, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "indexer score launch");
  return ok();
}

// part_*: the folded first pass (TopkArgs::hist_part and the indexer's slot
// split), or part == nullptr.
int topk_impl(const float* scores, const int32_t* pos, int64_t rows, int64_t N_cap, int k, int m,
              int32_t* idx_out, void* workspace, size_t ws_bytes, int flags,
              hattn_stream_t stream, const uint16_t* part = nullptr, int64_t part_total = 0,
              int64_t part_grid = 0, int64_t part_nblk = 0) {
  if (int rcf = check_flags(flags)) return rcf;
  REQUIRE_PTR(scores);
  REQUIRE_PTR(pos);
  REQUIRE_PTR(idx_out);
  REQUIRE(rows >= 1 && N_cap >= 1, "rows and N_cap must be >= 1");
  REQUIRE(N_cap < (1ll << 31), "N_cap=%lld must be < 2^31", (long long)N_cap);
  REQUIRE(rows <= 65535ll * 65535ll, "rows=%lld: at most 65535^2 query rows", (long long)rows);
  REQUIRE(k >= 1 && k <= 2048, "k=%d must be in [1, 2048]", k);
  REQUIRE(m >= 1, "m must be >= 1");
  // the plan (and so the scratch it needs) is checked before any device call
  TopkPlan tp;
  if (!plan_topk(rows, N_cap, k, num_sms_or_default(), &tp))
    return fail(HATTN_ERR_UNSUPPORTED, "top-k over N_cap=%lld entries is not supported",
                (long long)N_cap);
  TopkArgs t = {};
  if (tp.ws_bytes > 0) {
    REQUIRE_PTR(workspace);
    REQUIRE(ws_bytes >= tp.ws_bytes, "top-k workspace of %zu bytes, need %zu", ws_bytes,
            tp.ws_bytes);
    topk_scratch_carve(tp, rows, workspace, &t);
  }
  t.scores = scores;
  t.pos = pos;
  t.idx = idx_out;
  t.rows = rows;
  t.k = k;
  t.m = m;
  t.N_cap = N_cap;
  if (tp.slice_path) {
    int sms = 0;
    if (!device_info(nullptr, &t.status, &sms)) return fail(HATTN_ERR_CUDA, "no CUDA device");
  }
  if (tp.slice_path && part) {
    t.hist_part = part;
    t.part_total = part_total;
    t.part_grid = part_grid;
    t.part_nblk = part_nblk;
  }
  cudaError_t e = launch_topk(t, tp, (flags & HATTN_LAUNCH_DEPENDENT) != 0,
                              static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
  return ok();
}

// Scratch bytes of the selection (0 when it runs in shared memory alone).
size_t topk_ws_bytes(int64_t rows, int64_t N_cap, int k) {
  TopkPlan tp;
  if (rows < 1 || N_cap < 1 || k < 1 || !plan_topk(rows, N_cap, k, num_sms_or_default(), &tp))
    return 0;
  return tp.ws_bytes;
}

// Scratch of hattn_indexer_topk_noalloc: a fixed device array that every GPU
// loading this library holds until the process exits, so that call needs no
// allocation.  It holds the fp32 scores, then the selection's scratch:
// 4,194,304 scores (16 MiB, enough for B * T * N_cap = 8 x 1 x 262,144, a
// 1M-token decode batch of 8, twice over), then the indexer's partial
// histograms (up to 2 MiB) and at most as many candidate indices (16 MiB).
constexpr int64_t kNoallocScores = int64_t(1) << 22;
constexpr size_t kNoallocTopkBytes = (size_t(1) << 22) * 4 + (size_t(2) << 20);
constexpr size_t kNoallocBytes = kNoallocScores * 4 + kNoallocTopkBytes;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocBytes];

// Device address of g_noalloc_scratch for each device, looked up once with
// that device current (in host code the array's name is only a host-side
// stand-in, not a device address).
uint8_t* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(HATTN_ERR_CUDA, "device %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
    g_noalloc_ptr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return HATTN_OK;
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// Bytes of the indexer's partial histograms for the folded first pass.
size_t part_bytes(int64_t grid) { return round256((size_t)grid * 2 * kSelBins * sizeof(uint16_t)); }

// Whether the indexer can count the selection's first pass as it writes the
// scores (one query per indexer group, each CTA's slots within two rows and
// at most 65,535 entries, and the cluster path of the selection), for an
// indexer grid of `grid` CTAs.
bool fold_plan(int T, int HI, int dI, int keys, int64_t rows, int64_t N_cap, int k,
               int64_t grid) {
  IndexerPlan ip;
  if (!plan_indexer(T, HI, dI, keys, true, &ip)) return false;
  TopkPlan tp;
  if (!plan_topk(rows, N_cap, k, num_sms_or_default(), &tp) || !tp.slice_path) return false;
  const int64_t nblk = (N_cap + 127) / 128;
  const int64_t total = rows * nblk;  // one query per group: a group is a row
  if (grid < 1 || grid > total) return false;
  const int64_t spc = (total + grid - 1) / grid;
  return spc <= nblk && spc * 128 <= 65535;
}

// The indexer's grid for a call (as indexer_scores_impl launches it).
int64_t indexer_grid(int64_t rows_times_nblk_groups, int n_sms, int sms) {
  if (n_sms > 0 && n_sms < sms) sms = n_sms;
  return rows_times_nblk_groups < sms ? rows_times_nblk_groups : sms;
}

// Scores, then selection (folded when fold_plan allows).  workspace layout:
// [scores, unless score_out] [partial histograms, on the cluster path]
// [selection scratch].
int indexer_topk_impl(const void* iq, const float* w, const void* ik_c, const void* ik_scale,
                      const int32_t* pos, int B, int T, int HI, int dI, int64_t N_cap, int k,
                      int m, int n_sms, int64_t fresh_from, int32_t* idx_out, float* score_out,
                      uint8_t* workspace, size_t ws_bytes, int flags, void* split_event,
                      hattn_stream_t stream, bool mx = false) {
  const int keys = mx ? kIdxKeysMx4 : (ik_scale ? kIdxKeysE4m3 : kIdxKeysBf16);
  const int64_t rows = (int64_t)B * T;
  float* scores = score_out;
  uint8_t* rest = workspace;
  if (!scores) {
    scores = reinterpret_cast<float*>(workspace);
    rest += round256((size_t)rows * N_cap * sizeof(float));
  }
  TopkPlan tp;
  const bool cluster = plan_topk(rows, N_cap, k, num_sms_or_default(), &tp) && tp.slice_path;
  uint16_t* part = nullptr;
  int64_t grid = 0;
  if (cluster) {
    int sms = 0;
    int* status = nullptr;
    if (!device_info(nullptr, &status, &sms)) return fail(HATTN_ERR_CUDA, "no CUDA device");
    grid = indexer_grid(rows * ((N_cap + 127) / 128), n_sms, sms);
    if (fold_plan(T, HI, dI, keys, rows, N_cap, k, grid) &&
        part_bytes(grid) <= part_bytes(num_sms_or_default()))
      part = reinterpret_cast<uint16_t*>(rest);
    rest += part_bytes(num_sms_or_default());
  }
  const size_t used = (size_t)(rest - workspace);
  const size_t left = ws_bytes > used ? ws_bytes - used : 0;
  int64_t launched = 0;
  int rc = indexer_scores_impl(iq, w, ik_c, pos, B, T, HI, dI, N_cap, m, scores, stream, n_sms,
                               fresh_from, ik_scale, flags, part, &launched, mx);
  if (rc) return rc;
  if (split_event) {
    // external: an event record node when the stream is being captured
    cudaError_t e = cudaEventRecordWithFlags(
        static_cast<cudaEvent_t>(split_event), static_cast<cudaStream_t>(stream),
        (flags & HATTN_EVENT_EXTERNAL) ? cudaEventRecordExternal : cudaEventRecordDefault);
    if (e != cudaSuccess) return cuda_fail(e, "split event record");
  }
  // the selection waits for the scores before its first read: always a
  // dependent launch of the score kernel
  return topk_impl(scores, pos, rows, N_cap, k, m, idx_out, rest, left, HATTN_LAUNCH_DEPENDENT,
                   stream, part, rows * ((N_cap + 127) / 128), launched, (N_cap + 127) / 128);
}

size_t indexer_topk_ws(int B, int T, int64_t N_cap, int k, bool score_out_given) {
  if (B < 1 || T < 1 || N_cap < 1) return 0;
  const int64_t rows = (int64_t)B * T;
  const size_t scores = score_out_given ? 0 : round256((size_t)rows * N_cap * sizeof(float));
  TopkPlan tp;
  const bool cluster = k >= 1 && plan_topk(rows, N_cap, k, num_sms_or_default(), &tp) &&
                       tp.slice_path;
  return scores + (cluster ? part_bytes(num_sms_or_default()) : 0) + topk_ws_bytes(rows, N_cap, k);
}

}  // namespace

extern "C" {

int hattn_indexer_scores(const void* iq, const float* w, const void* ik_c, const int32_t* pos,
                         int B, int T, int HI, int dI, int64_t N_cap, int m, float* score_out,
                         hattn_stream_t stream) {
  return indexer_scores_impl(iq, w, ik_c, pos, B, T, HI, dI, N_cap, m, score_out, stream);
}

int hattn_indexer_scores_ex(const void* iq, const float* w, const void* ik_c,
                            const int32_t* pos, int B, int T, int HI, int dI, int64_t N_cap,
                            int m, int n_sms, int64_t fresh_from, float* score_out, int flags,
                            hattn_stream_t stream) {
  return indexer_scores_impl(iq, w, ik_c, pos, B, T, HI, dI, N_cap, m, score_out, stream, n_sms,
                             fresh_from < 0 ? -1 : fresh_from, nullptr, flags);
}

int hattn_indexer_scores_fp8(const void* iq, const float* w, const void* ik8,
                             const float* ik_scale, const int32_t* pos, int B, int T, int HI,
                             int dI, int64_t N_cap, int m, int n_sms, int64_t fresh_from,
                             float* score_out, int flags, hattn_stream_t stream) {
  REQUIRE_PTR(ik_scale);
  return indexer_scores_impl(iq, w, ik8, pos, B, T, HI, dI, N_cap, m, score_out, stream, n_sms,
                             fresh_from < 0 ? -1 : fresh_from, ik_scale, flags);
}

int hattn_indexer_scores_mxfp4(const void* iq, const float* w, const void* ik4,
                               const void* ik4_scale, const int32_t* pos, int B, int T, int HI,
                               int dI, int64_t N_cap, int m, int n_sms, int64_t fresh_from,
                               float* score_out, int flags, hattn_stream_t stream) {
  REQUIRE_PTR(ik4_scale);
  return indexer_scores_impl(iq, w, ik4, pos, B, T, HI, dI, N_cap, m, score_out, stream, n_sms,
                             fresh_from < 0 ? -1 : fresh_from, ik4_scale, flags, nullptr, nullptr,
                             true);
}

size_t hattn_topk_workspace_bytes(int B, int T, int64_t N_cap, int k) {
  if (B < 1 || T < 1) return 0;
  return topk_ws_bytes((int64_t)B * T, N_cap, k);
}

int hattn_topk_select(const float* scores, const int32_t* pos, int B, int T, int64_t N_cap, int k,
                      int m, int32_t* idx_out, void* workspace, size_t ws_bytes, int flags,
                      hattn_stream_t stream) {
  REQUIRE(B >= 1 && T >= 1, "B and T must be >= 1");
  return topk_impl(scores, pos, (int64_t)B * T, N_cap, k, m, idx_out, workspace, ws_bytes, flags,
                   stream);
}

size_t hattn_indexer_topk_workspace_bytes(int B, int T, int64_t N_cap, int k,
                                          int score_out_given) {
  return indexer_topk_ws(B, T, N_cap, k, score_out_given != 0);
}

int hattn_indexer_topk(const void* iq, const float* w, const void* ik_c, const int32_t* pos,
                       int B, int T, int HI, int dI, int64_t N_cap, int k, int m,
                       int32_t* idx_out, float* score_out, void* workspace, size_t ws_bytes,
                       hattn_stream_t stream) {
  return hattn_indexer_topk_ex(iq, w, ik_c, nullptr, pos, B, T, HI, dI, N_cap, k, m, 0, -1,
                               idx_out, score_out, workspace, ws_bytes, 0, nullptr, stream);
}

int hattn_indexer_topk_ex(const void* iq, const float* w, const void* ik_c, const float* ik_scale,
                          const int32_t* pos, int B, int T, int HI, int dI, int64_t N_cap, int k,
                          int m, int n_sms, int64_t fresh_from, int32_t* idx_out,
                          float* score_out, void* workspace, size_t ws_bytes, int flags,
                          void* split_event, hattn_stream_t stream) {
  if (int rcf = check_flags(flags)) return rcf;
  REQUIRE_PTR(iq);
  REQUIRE_PTR(w);
  REQUIRE_PTR(ik_c);
  REQUIRE_PTR(pos);
  REQUIRE(k >= 1 && k <= 2048, "k=%d must be in [1, 2048]", k);
  REQUIRE_PTR(idx_out);
  REQUIRE(dI >= 8 && dI <= 128 && dI % 8 == 0, "dI=%d must be a multiple of 8 in [8, 128]", dI);
  REQUIRE(B >= 1 && T >= 1 && N_cap >= 1, "B, T and N_cap must be >= 1");
  REQUIRE(n_sms >= 0, "n_sms=%d must be >= 0", n_sms);
  const size_t need = indexer_topk_ws(B, T, N_cap, k, score_out != nullptr);
  if (need > 0) {
    REQUIRE_PTR(workspace);
    REQUIRE(ws_bytes >= need, "workspace of %zu bytes, need %zu", ws_bytes, need);
  }
  return indexer_topk_impl(iq, w, ik_c, ik_scale, pos, B, T, HI, dI, N_cap, k, m, n_sms,
                           fresh_from < 0 ? -1 : fresh_from, idx_out, score_out,
                           static_cast<uint8_t*>(workspace), ws_bytes, flags, split_event,
                           stream);
}

int hattn_indexer_topk_mxfp4(const void* iq, const float* w, const void* ik4,
                             const void* ik4_scale, const int32_t* pos, int B, int T, int HI,
                             int dI, int64_t N_cap, int k, int m, int n_sms, int64_t fresh_from,
                             int32_t* idx_out, float* score_out, void* workspace,
                             size_t ws_bytes, int flags, void* split_event,
                             hattn_stream_t stream) {
  if (int rcf = check_flags(flags)) return rcf;
  REQUIRE_PTR(iq);
  REQUIRE_PTR(w);
  REQUIRE_PTR(ik4);
  REQUIRE_PTR(ik4_scale);
  REQUIRE_PTR(pos);
  REQUIRE(k >= 1 && k <= 2048, "k=%d must be in [1, 2048]", k);
  REQUIRE_PTR(idx_out);
  REQUIRE(dI == 128, "MXFP4 indexer keys need dI = 128, got %d", dI);
  REQUIRE(B >= 1 && T >= 1 && N_cap >= 1, "B, T and N_cap must be >= 1");
  REQUIRE(n_sms >= 0, "n_sms=%d must be >= 0", n_sms);
  const size_t need = indexer_topk_ws(B, T, N_cap, k, score_out != nullptr);
  if (need > 0) {
    REQUIRE_PTR(workspace);
    REQUIRE(ws_bytes >= need, "workspace of %zu bytes, need %zu", ws_bytes, need);
  }
  return indexer_topk_impl(iq, w, ik4, ik4_scale, pos, B, T, HI, dI, N_cap, k, m, n_sms,
                           fresh_from < 0 ? -1 : fresh_from, idx_out, score_out,
                           static_cast<uint8_t*>(workspace), ws_bytes, flags, split_event,
                           stream, true);
}

int hattn_indexer_topk_noalloc(const void* iq, const float* w, const void* ik_c,
                               const int32_t* pos, int B, int T, int HI, int dI, int64_t N_cap,
                               int k, int m, int32_t* idx_out, hattn_stream_t stream) {
  REQUIRE_PTR(iq);
  REQUIRE_PTR(w);
  REQUIRE_PTR(ik_c);
  REQUIRE_PTR(pos);
  REQUIRE_PTR(idx_out);
  REQUIRE(k >= 1 && k <= 2048, "k=%d must be in [1, 2048]", k);
  REQUIRE(dI >= 8 && dI <= 128 && dI % 8 == 0, "dI=%d must be a multiple of 8 in [8, 128]", dI);
  REQUIRE(B >= 1 && T >= 1 && N_cap >= 1, "B, T and N_cap must be >= 1");
  REQUIRE((int64_t)B * T * N_cap <= kNoallocScores,
          "B * T * N_cap = %lld scores exceed the fixed scratch of %lld (use hattn_indexer_topk "
          "with a workspace)", (long long)((int64_t)B * T * N_cap), (long long)kNoallocScores);
  const size_t sel = indexer_topk_ws(B, T, N_cap, k, true);
  REQUIRE(sel <= kNoallocTopkBytes,
          "the selection needs %zu bytes of scratch, the fixed scratch holds %zu (use "
          "hattn_indexer_topk with a workspace)", sel, kNoallocTopkBytes);
  uint8_t* scratch = nullptr;
  int rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  // every score the selection reads (entries j < visible count) is written
  // by the score kernel first, and every histogram and counter it reads is
  // written in the same call, so nothing in the shared scratch needs
  // clearing between calls
  return indexer_topk_impl(iq, w, ik_c, nullptr, pos, B, T, HI, dI, N_cap, k, m, 0, -1, idx_out,
                           reinterpret_cast<float*>(scratch), scratch + kNoallocScores * 4,
                           kNoallocTopkBytes, 0, nullptr, stream);
}

size_t hattn_attn_workspace_bytes(int kind, int B, int T, int H, int D, int64_t n_keys,
                                  int q_prepped, int partials) {
  AttnPlan p;
  if (kind < 0 || kind > 2) return 0;
  if (!plan_attention(kind, B, T, H, D, n_keys, num_sms_or_default(), &p)) return 0;
  return qprep_bytes(B, T, H, D, q_prepped) +
         (partials ? partial_bytes(B, T, H, D, p.nsplit) : p.ws_bytes);
}

int hattn_attn_splits(int kind, int B, int T, int H, int D, int64_t n_keys) {
  AttnPlan p;
  if (kind < 0 || kind > 2) return 0;
  if (!plan_attention(kind, B, T, H, D, n_keys, num_sms_or_default(), &p)) return 0;
  return p.nsplit;
}

int hattn_query_prep(const void* q, const float* gamma_q, const int32_t* pos, int B, int T, int H,
                     int D, int r, float rope_base, float eps, void* q_out,
                     hattn_stream_t stream) {
  int rc = query_prep_impl(q, gamma_q, pos, B, T, H, D, r, rope_base, eps, q_out, stream);
  return rc ? rc : ok();
}

int hattn_sparse_attn(const void* q, const float* gamma_q, int q_prepped, const void* kv_c,
                      const int32_t* idx,
                      const int32_t* pos, int B, int T, int H, int D, int64_t N_cap, int k, int r,
                      float rope_base, float eps, float scale, void* o, float* lse,
                      void* workspace, size_t ws_bytes, hattn_stream_t stream) {
  return attn_common(kSparse, q, gamma_q, q_prepped, kv_c, nullptr, idx, pos, B, T, H, D, N_cap, k, 1, 1, r,
                     rope_base, eps, scale, o, lse, workspace, ws_bytes, stream);
}

int hattn_hca_attn(const void* q, const float* gamma_q, int q_prepped, const void* kv_h,
                   const int32_t* pos,
                   int B, int T, int H, int D, int64_t N_cap, int m, int r, float rope_base,
                   float eps, float scale, void* o, float* lse, void* workspace,
                   size_t ws_bytes, hattn_stream_t stream) {
  return attn_common(kHca, q, gamma_q, q_prepped, kv_h, nullptr, nullptr, pos, B, T, H, D, N_cap, 1, m, 1, r,
                     rope_base, eps, scale, o, lse, workspace, ws_bytes, stream);
}

int hattn_hybrid_attn(const void* q, const float* gamma_q, int q_prepped, const void* kv_c,
                      const int32_t* idx, int64_t N_c, int k, const void* kv_h, int64_t N_h,
                      int m, const void* kv_w, int W, const int32_t* pos, int B, int T, int H,
                      int D, int r, float rope_base, float eps, float scale, int segments,
                      int n_sms, void* o, float* lse, void* workspace, size_t ws_bytes,
                      int flags, hattn_stream_t stream) {
  const FusedSources fs{kv_h, N_h, kv_w, segments, n_sms};
  return attn_common(kFused, q, gamma_q, q_prepped, kv_c, nullptr, idx, pos, B, T, H, D, N_c, k,
                     m, W, r, rope_base, eps, scale, o, lse, workspace, ws_bytes, stream, &fs,
                     flags);
}

int hattn_hybrid_attn_out(const void* q, const float* gamma_q, int q_prepped, const void* kv_c,
                          const int32_t* idx, int64_t N_c, int k, const void* kv_h, int64_t N_h,
                          int m, const void* kv_w, int W, const int32_t* pos, int B, int T, int H,
                          int D, int r, float rope_base, float eps, float scale, int segments,
                          int n_sms, const float* sink, void* out, float* lse_out,
                          void* workspace, size_t ws_bytes, int flags, hattn_stream_t stream) {
  const FusedSources fs{kv_h, N_h, kv_w, segments, n_sms};
  const FinalOut fo{out, lse_out, sink};
  // one key set alone runs its own branch kernel (the same keys, without
  // the fused call's segment bookkeeping; the HCA kind also stacks several
  // queries' heads when H < 128)
  if (segments == 2 && n_sms == 0)
    return attn_common(kHca, q, gamma_q, q_prepped, kv_h, nullptr, nullptr, pos, B, T, H, D, N_h,
                       1, m, 1, r, rope_base, eps, scale, nullptr, nullptr, workspace, ws_bytes,
                       stream, nullptr, flags, &fo);
  if (segments == 1 && n_sms == 0)
    return attn_common(kSparse, q, gamma_q, q_prepped, kv_c, nullptr, idx, pos, B, T, H, D, N_c,
                       k, 1, 1, r, rope_base, eps, scale, nullptr, nullptr, workspace, ws_bytes,
                       stream, nullptr, flags, &fo);
  return attn_common(kFused, q, gamma_q, q_prepped, kv_c, nullptr, idx, pos, B, T, H, D, N_c, k,
                     m, W, r, rope_base, eps, scale, nullptr, nullptr, workspace, ws_bytes,
                     stream, &fs, flags, &fo);
}

size_t hattn_hybrid_attn_out_workspace_bytes(int B, int T, int H, int D, int k, int64_t N_h,
                                             int W, int segments, int n_sms, int q_prepped) {
  AttnPlan p;
  if (segments < 1 || segments > 7 || n_sms < 0) return 0;
  // (the kind hattn_hybrid_attn_out runs for this segment set)
  const bool hca = segments == 2 && n_sms == 0, csa = segments == 1 && n_sms == 0;
  const int kind = hca ? kHca : (csa ? kSparse : kFused);
  const int64_t nk = hca ? N_h : (csa ? k : fused_keys(k, N_h, W, segments));
  if (!plan_attention(kind, B, T, H, D, nk, kind == kFused ? fused_sms(n_sms) : num_sms_or_default(),
                      &p))
    return 0;
  return qprep_bytes(B, T, H, D, q_prepped) +
         (p.nsplit > 1 ? partial_bytes(B, T, H, D, p.nsplit) : 0);
}

size_t hattn_hybrid_attn_workspace_bytes(int B, int T, int H, int D, int k, int64_t N_h, int W,
                                         int segments, int n_sms, int q_prepped,
                                         int partials) {
  AttnPlan p;
  if (segments < 1 || segments > 7 || n_sms < 0) return 0;
  if (!plan_attention(kFused, B, T, H, D, fused_keys(k, N_h, W, segments), fused_sms(n_sms),
                      &p))
    return 0;
  return qprep_bytes(B, T, H, D, q_prepped) +
         (partials ? partial_bytes(B, T, H, D, p.nsplit) : p.ws_bytes);
}

int hattn_hybrid_attn_splits(int B, int T, int H, int D, int k, int64_t N_h, int W,
                             int segments, int n_sms) {
  AttnPlan p;
  if (segments < 1 || segments > 7 || n_sms < 0) return 0;
  if (!plan_attention(kFused, B, T, H, D, fused_keys(k, N_h, W, segments), fused_sms(n_sms),
                      &p))
    return 0;
  return p.nsplit;
}

static int swa_keys_common(const void* kv_raw, const float* gamma_kv, const int32_t* pos, int B, int T,
                    int64_t L_cap, int D, int W, int r, float rope_base, float eps, void* kv_w,
                    hattn_stream_t stream, int64_t ring) {
  REQUIRE_PTR(kv_raw);
  REQUIRE_PTR(pos);
  REQUIRE_PTR(kv_w);
  REQUIRE_F32(gamma_kv);
  REQUIRE(B >= 1 && T >= 1 && L_cap >= 1, "B, T and L_cap must be >= 1");
  REQUIRE(W >= 1 && W <= 65536, "W=%d out of range", W);
  REQUIRE(D >= 64 && D <= 512 && D % 64 == 0, "D=%d must be a multiple of 64 in [64, 512]", D);
  int rc = check_rope(D, r, rope_base, eps);
  if (rc) return rc;
  SwaKeysArgs a;
  a.kv_raw = static_cast<const __nv_bfloat16*>(kv_raw);
  a.gamma = gamma_kv;
  a.pos = pos;
  a.kv_w = static_cast<__nv_bfloat16*>(kv_w);
  a.B = B;
  a.T = T;
  a.D = D;
  a.r = r;
  a.W = W;
  a.L_cap = L_cap;
  a.ring = ring;
  a.eps = eps;
  make_rope_coef(rope_base, r, &a.rope);
  cudaError_t e = launch_swa_keys(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "SWA keys launch");
  return ok();
}

int hattn_swa_keys(const void* kv_raw, const float* gamma_kv, const int32_t* pos, int B, int T,
                   int64_t L_cap, int D, int W, int r, float rope_base, float eps, void* kv_w,
                   hattn_stream_t stream) {
  return swa_keys_common(kv_raw, gamma_kv, pos, B, T, L_cap, D, W, r, rope_base, eps, kv_w, stream,
                         0);
}

int hattn_swa_keys_ring(const void* kv_ring, const float* gamma_kv, const int32_t* pos, int B,
                        int T, int64_t ring, int D, int W, int r, float rope_base, float eps,
                        void* kv_w, hattn_stream_t stream) {
  // the T queries of a sequence together need the W + T - 1 newest tokens
  REQUIRE(ring >= 1 && (ring & (ring - 1)) == 0, "ring=%lld must be a power of two", (long long)ring);
  REQUIRE(ring >= (int64_t)W + T - 1, "ring=%lld holds fewer than W + T - 1 = %d tokens", (long long)ring,
          W + T - 1);
  return swa_keys_common(kv_ring, gamma_kv, pos, B, T, ring, D, W, r, rope_base, eps, kv_w, stream,
                         ring);
}

int hattn_swa_attn(const void* q, const float* gamma_q, int q_prepped, const void* kv_raw,
                   const float* gamma_kv, const int32_t* pos, int B, int T, int H, int D,
                   int64_t L_cap, int W, int r, float rope_base, float eps, float scale, void* o,
                   float* lse, void* workspace, size_t ws_bytes, hattn_stream_t stream) {
  return attn_common(kSwa, q, gamma_q, q_prepped, kv_raw, gamma_kv, nullptr, pos, B, T, H, D, L_cap, 1, 1, W,
                     r, rope_base, eps, scale, o, lse, workspace, ws_bytes, stream);
}

}  // extern "C"

namespace {

int merge_impl(const void* const* o_list, const float* const* lse_list, const int* nsplit, int nb,
               const float* sink, const int32_t* pos, int B, int T, int H, int D, int r,
               float rope_base, void* out, float* lse_out, hattn_stream_t stream, int flags) {
  if (int rcf = check_flags(flags)) return rcf;
  REQUIRE(o_list && lse_list, "o_list and lse_list must not be NULL");
  REQUIRE(nb >= 1 && nb <= 4, "nb=%d must be in [1, 4]", nb);
  MergeArgs a;
  int parts = 0;
  for (int i = 0; i < nb; ++i) {
    if (!o_list[i] || !lse_list[i]) return fail(HATTN_ERR_INVALID_ARG, "branch %d is NULL", i);
    if (!aligned16(o_list[i])) return fail(HATTN_ERR_MISALIGNED, "o_list[%d] is not 16-byte aligned", i);
    if (!aligned4(lse_list[i])) return fail(HATTN_ERR_MISALIGNED, "lse_list[%d] is not 4-byte aligned", i);
    const int ns = nsplit ? nsplit[i] : 1;
    REQUIRE(ns >= 1, "nsplit[%d]=%d must be >= 1", i, ns);
    parts += ns;
    a.o[i] = static_cast<const float*>(o_list[i]);
    a.lse[i] = lse_list[i];
    a.nsplit[i] = ns;
  }
  REQUIRE(parts <= kMaxMergeParts, "%d partials per row, at most %d", parts, kMaxMergeParts);
  a.cum[0] = 0;
  for (int i = 0; i < 4; ++i) a.cum[i + 1] = a.cum[i] + (i < nb ? a.nsplit[i] : 0);
  REQUIRE_PTR(pos);
  REQUIRE_PTR(out);
  REQUIRE_F32(sink);
  REQUIRE_F32(lse_out);
  REQUIRE(B >= 1 && T >= 1 && H >= 1, "B, T and H must be >= 1");
  REQUIRE(D >= 8 && D <= 4096 && D % 8 == 0, "D=%d must be a multiple of 8 in [8, 4096]", D);
  REQUIRE(r >= 0 && r % 2 == 0 && r <= D && r <= 2 * kMaxRopePairs,
          "r=%d must be even, <= D and <= %d", r, 2 * kMaxRopePairs);
  REQUIRE(rope_base > 0.f, "rope_base must be positive");
  a.nb = nb;
  a.sink = sink;
  a.pos = pos;
  a.out = static_cast<__nv_bfloat16*>(out);
  a.lse_out = lse_out;
  a.B = B;
  a.T = T;
  a.H = H;
  a.D = D;
  a.r = r;
  a.dependent = (flags & HATTN_LAUNCH_DEPENDENT) ? 1 : 0;
  make_rope_coef(rope_base, r, &a.rope);
  cudaError_t e = launch_merge(a, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "merge launch");
  return ok();
}

}  // namespace

extern "C" {

int hattn_lse_merge(const void* const* o_list, const float* const* lse_list, int nb,
                    const float* sink, const int32_t* pos, int B, int T, int H, int D, int r,
                    float rope_base, void* out, float* lse_out, hattn_stream_t stream) {
  return merge_impl(o_list, lse_list, nullptr, nb, sink, pos, B, T, H, D, r, rope_base, out,
                    lse_out, stream, 0);
}

int hattn_lse_merge_splits(const void* const* part_o_list, const float* const* part_lse_list,
                           const int* nsplit, int nb, const float* sink, const int32_t* pos, int B,
                           int T, int H, int D, int r, float rope_base, void* out, float* lse_out,
                           int flags, hattn_stream_t stream) {
  if (!nsplit) return fail(HATTN_ERR_INVALID_ARG, "nsplit must not be NULL");
  return merge_impl(part_o_list, part_lse_list, nsplit, nb, sink, pos, B, T, H, D, r, rope_base,
                    out, lse_out, stream, flags);
}

const char* hattn_status_string(int code) {
  switch (code) {
    case HATTN_OK: return "ok";
    case HATTN_ERR_INVALID_ARG: return "invalid argument";
    case HATTN_ERR_MISALIGNED: return "misaligned pointer";
    case HATTN_ERR_UNSUPPORTED: return "unsupported shape";
    case HATTN_ERR_CUDA: return "CUDA error";
    case HATTN_ERR_TIMEOUT: return "device wait timed out";
    case HATTN_ERR_DEVICE_INDEX: return "device index out of range";
    default: return "unknown status";
  }
}

const char* hattn_last_error(void) { return g_last_error; }

int hattn_check_status(hattn_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronise");
  int* status = nullptr;
  if (!device_info(nullptr, &status, nullptr)) return fail(HATTN_ERR_CUDA, "no CUDA device");
  int v[4] = {0, 0, 0, 0};
  e = cudaMemcpy(v, status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  const int zero[4] = {0, 0, 0, 0};
  e = cudaMemcpy(status, zero, sizeof zero, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_fail(e, "status clear");
  if (v[0] != 0)
    return fail(v[0], "device reported: %s (wait site %d, block %d, thread %d)",
                hattn_status_string(v[0]), v[1], v[2], v[3]);
  return ok();
}

int hattn_selftest_wait_timeout(uint64_t timeout_ns, hattn_stream_t stream) {
  int* status = nullptr;
  if (!device_info(nullptr, &status, nullptr)) return fail(HATTN_ERR_CUDA, "no CUDA device");
  cudaError_t e = launch_wait_selftest(timeout_ns, status, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "selftest launch");
  return ok();
}

const char* hattn_version(void) { return "hattn 0.2 sm_103a"; }

}  // extern "C"
