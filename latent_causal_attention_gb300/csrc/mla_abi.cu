// C ABI of the library (declared in include/mla.h): argument validation,
// choice of path, tensor-map construction and kernel launches on the caller's
// stream.  No allocation, no host synchronisation, no exceptions.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/mla.h"
#include "internal.h"

namespace mla {

// ---------------------------------------------------------------------------
// cuTensorMapEncodeTiled through the runtime's driver entry point (no -lcuda).
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
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

bool make_tmap_3d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2,
                  bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {s1, s2};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt =
      elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(map, dt, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The fused kernel's output tiles: out (rows, H, d) fp32 or bf16 as {d, H, rows},
// 128-byte swizzled boxes of 128 bytes x 1 head x 128 rows.
static bool make_out_tmap(CUtensorMap* map, void* out, bool bf16, int d, int H, uint64_t rows) {
  const int es = bf16 ? 2 : 4;
  return make_tmap_3d(map, out, es, (uint64_t)d, (uint64_t)H, rows, (uint64_t)d * es,
                      (uint64_t)H * d * es, 128u / es, 1, 128, true);
}

// The persistent pair kernel's output tiles: out (B, Tq, H, d) as {d, H, Tq, B},
// so that a tile store never crosses into the next batch entry.
static bool make_out_tmap_4d(CUtensorMap* map, void* out, bool bf16, int d, int H, int Tq,
                             int B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t es = bf16 ? 2 : 4;
  const cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)H, (cuuint64_t)Tq, (cuuint64_t)B};
  const cuuint64_t strides[3] = {d * es, (uint64_t)H * d * es, (uint64_t)Tq * H * d * es};
  const cuuint32_t box[4] = {(cuuint32_t)(128 / es), 1, 128, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                  4, out, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// Options
// ---------------------------------------------------------------------------
static int g_attn_path = 0;     // 0 auto, 1 warp, 2 tensor core
static int g_kv_splits = 0;     // 0 auto
static int g_prefill_fused = 1; // 1: one fused kernel per head for long prefill
static int g_num_sms = 0;       // > 0: SM count the planner assumes (0: the device's own)
static int g_persistent = 1;    // 1: persistent kernel for single-CTA prefill with d = 64
static void** g_stage_events = nullptr;
static int g_stage_events_n = 0;
static unsigned long long g_launches = 0;

// Records the "before" (edge 0) or "after" (edge 1) event of a stage.
static void stage_event(int stage, int edge, cudaStream_t stream) {
  const int i = 2 * stage + edge;
  if (g_stage_events && i < g_stage_events_n && g_stage_events[i])
    cudaEventRecord(static_cast<cudaEvent_t>(g_stage_events[i]), stream);
}

// Wraps one kernel launch: stage events around it and the launch counter.
template <typename F>
static cudaError_t staged(int stage, cudaStream_t stream, F&& launch) {
  stage_event(stage, 0, stream);
  cudaError_t e = launch();
  stage_event(stage, 1, stream);
  if (e == cudaSuccess) __atomic_add_fetch(&g_launches, 1ull, __ATOMIC_RELAXED);
  return e;
}

static inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

static int pick_bn(int N) {
  if (N % 256 == 0) return 256;
  if (N % 128 == 0) return 128;
  return 64;
}

// ---------------------------------------------------------------------------
// Attention path planning (shared by the workspace query and the call)
// ---------------------------------------------------------------------------
struct AttnPlan {
  bool tc;
  bool fused;             // per-head fused kernel (no workspace)
  int pair, RC, row_blocks, splits;
  int64_t rows;           // B*Tq*H
  size_t off_qp, off_olat, off_po, off_pml, total;
};

constexpr int kMaxDevices = 64;
static std::atomic<int> g_sm_count[kMaxDevices];

// SM count of the current device, asked once per device and cached; the
// option MLA_OPT_NUM_SMS overrides it, and a host without a usable device
// plans for kDefaultNumSMs.
static int planner_sm_count() {
  if (g_num_sms > 0) return g_num_sms;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    cudaGetLastError();              // leave no error behind for a later launch check
    return kDefaultNumSMs;
  }
  int n = g_sm_count[dev].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return kDefaultNumSMs;
  }
  g_sm_count[dev].store(n, std::memory_order_relaxed);
  return n;
}

static bool tc_shape_ok(int d, int R) {
  if (d % 64 != 0 || d > 256) return false;
  if (R % 64 != 0 || R > 512) return false;
  if (R > 256 && (R % 128 != 0)) return false;
  return true;
}

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static AttnPlan plan_attention(int B, int Tq, int Tkv, int H, int d, int R, int in_dtype,
                               int causal) {
  AttnPlan p = {};
  const bool shape_tc = in_dtype == MLA_BF16 && tc_shape_ok(d, R);
  p.tc = (g_attn_path == 2) ? shape_tc : (g_attn_path == 1 ? false : shape_tc);
  if (!p.tc) return p;
  p.pair = R > 256 ? 1 : 0;
  p.RC = p.pair ? R / 2 : R;
  p.rows = (int64_t)B * Tq * H;
  // Long prefill: rows are 128 query positions of one head, so the kernel can
  // absorb w_up_k and apply w_up_v itself; needs d <= 128 for its staging.
  p.fused = g_prefill_fused && g_kv_splits == 0 && Tq >= 64 && d <= 128;
  if (p.fused) {
    p.row_blocks = (Tq + 127) / 128;
    p.splits = 1;
    p.total = 0;
    return p;
  }
  p.row_blocks = (int)(((int64_t)Tq * H + 127) / 128);
  const int csize = p.pair ? 2 : 1;
  const int64_t ctas = (int64_t)p.row_blocks * B * csize;
  const int kv_tiles = (Tkv + 63) / 64;
  int splits = 1;
  if (g_kv_splits > 0) {
    splits = g_kv_splits;
  } else {
    const int sms = planner_sm_count();
    if (ctas < sms / 2) splits = (int)((sms + ctas - 1) / ctas);
  }
  if (splits > kv_tiles) splits = kv_tiles;
  if (splits < 1) splits = 1;
  (void)causal;
  p.splits = splits;
  size_t off = 0;
  p.off_qp = off;   off = align256(off + (size_t)p.rows * R * 2);
  p.off_olat = off; off = align256(off + (size_t)p.rows * R * 2);
  if (splits > 1) {
    p.off_po = off;  off = align256(off + (size_t)splits * p.rows * R * 4);
    p.off_pml = off; off = align256(off + (size_t)splits * p.rows * 2 * 4);
  }
  p.total = off;
  return p;
}

// The tensor-core path reads and writes through TMA and 16-byte vectors.
static bool tc_pointers_ok(const void* q, const void* lat, const void* wk, const void* wv,
                           const void* out) {
  return aligned16(q) && aligned16(lat) && aligned16(wk) && aligned16(wv) && aligned16(out);
}

static mla_status_t cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

}  // namespace mla

using namespace mla;

extern "C" {

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_NULL: return "null pointer";
    case MLA_ERR_SHAPE: return "invalid shape";
    case MLA_ERR_DTYPE: return "unsupported dtype";
    case MLA_ERR_ALIGN: return "misaligned pointer";
    case MLA_ERR_WORKSPACE: return "workspace missing or too small";
    case MLA_ERR_CUDA: return "CUDA error";
    case MLA_ERR_TIMEOUT: return "device-side wait timed out";
    case MLA_ERR_UNSUPPORTED: return "unsupported by this library";
    default: return "unknown status";
  }
}

mla_status_t mla_set_option(int option, int64_t value) {
  switch (option) {
    case MLA_OPT_ATTN_PATH:
      if (value < 0 || value > 2) return MLA_ERR_SHAPE;
      g_attn_path = (int)value;
      return MLA_OK;
    case MLA_OPT_KV_SPLITS:
      if (value < 0 || value > 4096) return MLA_ERR_SHAPE;
      g_kv_splits = (int)value;
      return MLA_OK;
    case MLA_OPT_PREFILL_FUSED:
      if (value < 0 || value > 1) return MLA_ERR_SHAPE;
      g_prefill_fused = (int)value;
      return MLA_OK;
    case MLA_OPT_NUM_SMS:
      if (value < 0 || value > 4096) return MLA_ERR_SHAPE;
      g_num_sms = (int)value;
      return MLA_OK;
    case MLA_OPT_PERSISTENT:
      if (value < 0 || value > 1) return MLA_ERR_SHAPE;
      g_persistent = (int)value;
      return MLA_OK;
    default:
      return MLA_ERR_UNSUPPORTED;
  }
}

mla_status_t mla_set_stage_events(void** events, int n) {
  if (events != nullptr && n <= 0) return MLA_ERR_SHAPE;
  g_stage_events = events;
  g_stage_events_n = events ? n : 0;
  return MLA_OK;
}

mla_status_t mla_check_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 10u * 1000u * 1000u) return MLA_ERR_SHAPE;
  return cuda_status(launch_wait_timeout_probe((unsigned long long)limit_us * 1000ull,
                                               static_cast<cudaStream_t>(stream)));
}

uint64_t mla_launch_count(void) { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

mla_status_t mla_get_device_error(unsigned int* code, int clear) {
  if (!code) return MLA_ERR_NULL;
  unsigned int a = 0, b = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  if (gemm_read_device_error(&a, clear) != cudaSuccess) return MLA_ERR_CUDA;
  if (flash_read_device_error(&b, clear) != cudaSuccess) return MLA_ERR_CUDA;
  *code = a ? a : b;
  return MLA_OK;
}

// ---------------------------------------------------------------------------
mla_status_t mla_kv_latent_project(const void* hidden, const void* w_down, const void* w_up_k,
                                   const void* w_up_v, void* latent, void* k, void* v,
                                   int64_t M, int model_dim, int rank, int kv_dim, int in_dtype,
                                   int out_dtype, void* stream_) {
  if (!hidden || !w_down || !latent) return MLA_ERR_NULL;
  if ((k && !w_up_k) || (v && !w_up_v)) return MLA_ERR_NULL;
  if (M <= 0 || model_dim <= 0 || rank <= 0) return MLA_ERR_SHAPE;
  if ((k || v) && kv_dim <= 0) return MLA_ERR_SHAPE;
  if (M > kMaxIndex) return MLA_ERR_SHAPE;
  if (in_dtype != MLA_F32 && in_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (out_dtype != MLA_F32 && out_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (in_dtype == MLA_F32 && out_dtype != MLA_F32) return MLA_ERR_DTYPE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const bool want_kv = (k != nullptr) || (v != nullptr);

  const bool tc = in_dtype == MLA_BF16 && model_dim % 64 == 0 && rank % 64 == 0 && rank <= 512 &&
                  (!want_kv || (kv_dim % 64 == 0 && out_dtype == MLA_BF16)) &&
                  aligned16(hidden) && aligned16(w_down) && aligned16(latent) &&
                  (!k || (aligned16(k) && aligned16(w_up_k))) &&
                  (!v || (aligned16(v) && aligned16(w_up_v)));
  if (!tc) {
    if (rank > 512) return MLA_ERR_UNSUPPORTED;
    return cuda_status(staged(4, stream, [&] {
      return launch_projection_cuda_core(hidden, w_down, w_up_k, w_up_v, latent, k, v, M,
                                         model_dim, rank, want_kv ? kv_dim : 0,
                                         in_dtype == MLA_BF16, out_dtype == MLA_BF16, stream);
    }));
  }
  // Stage 1: latent = hidden @ w_down  (A K-major, B = w_down MN-major).
  CUtensorMap mA, mB;
  if (!make_tmap_3d(&mA, hidden, 2, model_dim, 1, M, (uint64_t)model_dim * 2,
                    (uint64_t)model_dim * 2, 64, 1, 128, true))
    return MLA_ERR_CUDA;
  if (!make_tmap_3d(&mB, w_down, 2, rank, 1, model_dim, (uint64_t)rank * 2, (uint64_t)rank * 2, 64,
                    1, 64, true))
    return MLA_ERR_CUDA;
  GemmArgs g = {};
  g.M = (int)M; g.N = rank; g.K = model_dim; g.G = 1; g.BN = pick_bn(rank); g.alpha = 1.f;
  g.C = latent; g.c_bf16 = out_dtype == MLA_BF16; g.c_rs = rank; g.c_gs = 0;
  cudaError_t e = staged(4, stream, [&] { return launch_gemm_tc(mA, mB, true, g, stream); });
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  if (!want_kv) return MLA_OK;
  // Stage 2: k / v = latent(bf16) @ w_up_k / w_up_v.
  CUtensorMap mL;
  if (!make_tmap_3d(&mL, latent, 2, rank, 1, M, (uint64_t)rank * 2, (uint64_t)rank * 2, 64, 1,
                    128, true))
    return MLA_ERR_CUDA;
  const void* ws[2] = {w_up_k, w_up_v};
  void* outs[2] = {k, v};
  for (int i = 0; i < 2; ++i) {
    if (!outs[i]) continue;
    CUtensorMap mW;
    if (!make_tmap_3d(&mW, ws[i], 2, kv_dim, 1, rank, (uint64_t)kv_dim * 2, (uint64_t)kv_dim * 2,
                      64, 1, 64, true))
      return MLA_ERR_CUDA;
    GemmArgs g2 = {};
    g2.M = (int)M; g2.N = kv_dim; g2.K = rank; g2.G = 1; g2.BN = pick_bn(kv_dim); g2.alpha = 1.f;
    g2.C = outs[i]; g2.c_bf16 = 1; g2.c_rs = kv_dim; g2.c_gs = 0;
    e = staged(5, stream, [&] { return launch_gemm_tc(mL, mW, true, g2, stream); });
    if (e != cudaSuccess) return MLA_ERR_CUDA;
  }
  return MLA_OK;
}

// ---------------------------------------------------------------------------
size_t mla_latent_attention_workspace_size(int B, int Tq, int Tkv, int H, int d, int rank,
                                           int in_dtype, int causal) {
  if (B <= 0 || Tq <= 0 || Tkv <= 0 || H <= 0 || d <= 0 || rank <= 0 || Tq > Tkv) return 0;
  AttnPlan p = plan_attention(B, Tq, Tkv, H, d, rank, in_dtype, causal);
  return p.tc ? p.total : 0;
}

int mla_latent_attention_kv_splits(int B, int Tq, int Tkv, int H, int d, int rank, int in_dtype,
                                   int causal) {
  if (B <= 0 || Tq <= 0 || Tkv <= 0 || H <= 0 || d <= 0 || rank <= 0 || Tq > Tkv) return 0;
  AttnPlan p = plan_attention(B, Tq, Tkv, H, d, rank, in_dtype, causal);
  return p.tc ? p.splits : 0;
}

mla_status_t mla_latent_attention(const void* q, const void* kv_latent, const void* w_up_k,
                                  const void* w_up_v, void* out, int B, int Tq, int Tkv, int H,
                                  int d, int rank, float scale, int causal, int in_dtype,
                                  int out_dtype, void* workspace, size_t workspace_bytes,
                                  void* stream_) {
  if (!q || !kv_latent || !w_up_k || !w_up_v || !out) return MLA_ERR_NULL;
  if (B <= 0 || Tq <= 0 || Tkv <= 0 || H <= 0 || d <= 0 || rank <= 0 || Tq > Tkv)
    return MLA_ERR_SHAPE;
  if ((int64_t)B * Tq * H > kMaxIndex || (int64_t)B * Tkv > kMaxIndex) return MLA_ERR_SHAPE;
  if (in_dtype != MLA_F32 && in_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (out_dtype != MLA_F32 && out_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (in_dtype == MLA_F32 && out_dtype != MLA_F32) return MLA_ERR_DTYPE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);

  AttnPlan p = plan_attention(B, Tq, Tkv, H, d, rank, in_dtype, causal);
  if (p.tc && !tc_pointers_ok(q, kv_latent, w_up_k, w_up_v, out)) {
    if (g_attn_path == 2) return MLA_ERR_ALIGN;
    p.tc = false;
  }
  if (!p.tc) {
    if (g_attn_path == 2) return MLA_ERR_UNSUPPORTED;
    if (rank > 1024 || d > 256) return MLA_ERR_UNSUPPORTED;
    return cuda_status(staged(1, stream, [&] {
      return launch_warp_attention(q, kv_latent, w_up_k, w_up_v, out, B, Tq, Tkv, H, d, rank,
                                   scale, causal, in_dtype == MLA_BF16, out_dtype == MLA_BF16,
                                   stream);
    }));
  }
  const int R = rank;
  const int64_t BT = (int64_t)B * Tq;
  if (p.fused) {
    // one kernel: q . w_up_k -> flash loop over the latent -> . w_up_v -> out
    CUtensorMap mQ, mL, mWk, mWv, mO;
    if (!make_tmap_3d(&mQ, q, 2, d, H, BT, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, 128,
                      true) ||
        !make_tmap_3d(&mL, kv_latent, 2, R, Tkv, B, (uint64_t)R * 2, (uint64_t)Tkv * R * 2, 64, 64,
                      1, true) ||
        !make_tmap_3d(&mWk, w_up_k, 2, d, H, R, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1,
                      p.RC, true) ||
        !make_tmap_3d(&mWv, w_up_v, 2, d, H, R, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, 64,
                      true) ||
        !make_out_tmap(&mO, out, out_dtype == MLA_BF16, d, H, (uint64_t)BT))
      return MLA_ERR_CUDA;
    FlashArgs fa = {};
    fa.B = B; fa.Tq = Tq; fa.Tkv = Tkv; fa.H = H; fa.R = R; fa.RC = p.RC; fa.pair = p.pair;
    fa.row_blocks = p.row_blocks; fa.splits = 1; fa.causal = causal ? 1 : 0;
    fa.d = d; fa.qscale = scale * 1.4426950408889634f; fa.out = out;
    fa.out_bf16 = out_dtype == MLA_BF16;
    const int64_t items = (int64_t)p.row_blocks * B * H;
    CUtensorMap mO4;
    const bool have_o4 = make_out_tmap_4d(&mO4, out, out_dtype == MLA_BF16, d, H, Tq, B);
    if (g_persistent && !p.pair && d == 64 && have_o4) {
      // one resident CTA per SM works through the (b, head, row block) items
      const int ctas = (int)(items < planner_sm_count() ? items : planner_sm_count());
      if (staged(1, stream, [&] {
            return launch_flash_persistent(mQ, mL, mWk, mWv, mO4, fa, ctas, stream);
          }) != cudaSuccess)
        return MLA_ERR_CUDA;
      return MLA_OK;
    }
    if (g_persistent && p.pair) {
      // one resident CTA pair per two SMs (as many as fit at once)
      int64_t pairs = flash_pair_slots(p.RC, d);
      if (pairs > planner_sm_count() / 2) pairs = planner_sm_count() / 2;
      if (pairs > items) pairs = items;
      if (pairs > 0 && have_o4) {
        if (staged(1, stream, [&] {
              return launch_flash_persistent_pair(mQ, mL, mWk, mWv, mO4, fa, (int)pairs, stream);
            }) != cudaSuccess)
          return MLA_ERR_CUDA;
        return MLA_OK;
      }
    }
    if (staged(1, stream,
               [&] { return launch_flash_fused(mQ, mL, mWk, mWv, mO, fa, stream); }) !=
        cudaSuccess)
      return MLA_ERR_CUDA;
    return MLA_OK;
  }
  if (!workspace) return MLA_ERR_WORKSPACE;
  if (workspace_bytes < p.total) return MLA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return MLA_ERR_ALIGN;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  void* qp = ws + p.off_qp;
  void* olat = ws + p.off_olat;

  // 1. absorption: q'[(b,i), h, :] = scale*log2(e) * w_up_k[:, h, :] q[(b,i), h, :]
  CUtensorMap mA, mB;
  if (!make_tmap_3d(&mA, q, 2, d, H, BT, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, 128, true))
    return MLA_ERR_CUDA;
  const int bn_abs = pick_bn(R);
  if (!make_tmap_3d(&mB, w_up_k, 2, d, H, R, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, bn_abs,
                    true))
    return MLA_ERR_CUDA;
  GemmArgs g = {};
  g.M = (int)BT; g.N = R; g.K = d; g.G = H; g.BN = bn_abs;
  // one query row block per head (decode): the whole rank in one CTA, so the
  // heads' tiles run in one wave
  if (R == 512 && BT <= 128) g.BN = 512;
  g.alpha = scale * 1.4426950408889634f;
  g.C = qp; g.c_bf16 = 1; g.c_rs = (int64_t)H * R; g.c_gs = R;
  if (staged(0, stream, [&] { return launch_gemm_tc(mA, mB, false, g, stream); }) != cudaSuccess)
    return MLA_ERR_CUDA;

  // 2. flash loop over the latent
  CUtensorMap mQ, mL;
  if (!make_tmap_3d(&mQ, qp, 2, R, (uint64_t)Tq * H, B, (uint64_t)R * 2,
                    (uint64_t)Tq * H * R * 2, 64, 128, 1, true))
    return MLA_ERR_CUDA;
  if (!make_tmap_3d(&mL, kv_latent, 2, R, Tkv, B, (uint64_t)R * 2, (uint64_t)Tkv * R * 2, 64, 64, 1,
                    true))
    return MLA_ERR_CUDA;
  FlashArgs fa = {};
  fa.B = B; fa.Tq = Tq; fa.Tkv = Tkv; fa.H = H; fa.R = R; fa.RC = p.RC; fa.pair = p.pair;
  fa.row_blocks = p.row_blocks; fa.splits = p.splits; fa.causal = causal ? 1 : 0;
  fa.olat = olat;
  fa.part_o = p.splits > 1 ? reinterpret_cast<float*>(ws + p.off_po) : nullptr;
  fa.part_ml = p.splits > 1 ? reinterpret_cast<float*>(ws + p.off_pml) : nullptr;
  if (staged(1, stream, [&] { return launch_flash_packed(mQ, mL, fa, stream); }) != cudaSuccess)
    return MLA_ERR_CUDA;

  // 3. merge the key-range partitions
  if (p.splits > 1) {
    if (staged(2, stream, [&] {
          return launch_merge_partials(fa.part_ml, 2, nullptr, fa.part_o, olat, p.splits,
                                       (int)p.rows, R, 1, stream);
        }) != cudaSuccess)
      return MLA_ERR_CUDA;
  }

  // 4. value up-projection: out[(b,i), h, :] = o_lat[(b,i), h, :] @ w_up_v[:, h, :]
  CUtensorMap mO, mV;
  if (!make_tmap_3d(&mO, olat, 2, R, H, BT, (uint64_t)R * 2, (uint64_t)H * R * 2, 64, 1, 128,
                    true))
    return MLA_ERR_CUDA;
  if (!make_tmap_3d(&mV, w_up_v, 2, d, H, R, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, 64, true))
    return MLA_ERR_CUDA;
  GemmArgs g2 = {};
  g2.M = (int)BT; g2.N = d; g2.K = R; g2.G = H; g2.BN = pick_bn(d); g2.alpha = 1.f;
  g2.C = out; g2.c_bf16 = out_dtype == MLA_BF16; g2.c_rs = (int64_t)H * d; g2.c_gs = d;
  if (staged(3, stream, [&] { return launch_gemm_tc(mO, mV, true, g2, stream); }) != cudaSuccess)
    return MLA_ERR_CUDA;
  return MLA_OK;
}

mla_status_t mla_latent_attention_varlen(const void* q, const void* kv_latent, const void* w_up_k,
                                         const void* w_up_v, void* out, const int* cu_seqlens_q,
                                         const int* cu_seqlens_kv, int B, int max_seqlen_q,
                                         int total_q, int total_kv, int H, int d, int rank,
                                         float scale, int causal, int in_dtype, int out_dtype,
                                         void* stream_) {
  if (!q || !kv_latent || !w_up_k || !w_up_v || !out || !cu_seqlens_q || !cu_seqlens_kv)
    return MLA_ERR_NULL;
  if (B <= 0 || max_seqlen_q <= 0 || total_q <= 0 || total_kv <= 0 || H <= 0 ||
      max_seqlen_q > total_q)
    return MLA_ERR_SHAPE;
  if ((int64_t)total_q * H > kMaxIndex) return MLA_ERR_SHAPE;
  if (d % 64 != 0 || d > 128 || !tc_shape_ok(d, rank)) return MLA_ERR_SHAPE;
  if (in_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (out_dtype != MLA_F32 && out_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (!(aligned16(q) && aligned16(kv_latent) && aligned16(w_up_k) && aligned16(w_up_v) &&
        aligned16(out)) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3) != 0 ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_kv) & 3) != 0)
    return MLA_ERR_ALIGN;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const int R = rank;
  const int pair = R > 256 ? 1 : 0;
  const int RC = pair ? R / 2 : R;
  CUtensorMap mQ, mL, mWk, mWv, mO;
  if (!make_tmap_3d(&mQ, q, 2, d, H, (uint64_t)total_q, (uint64_t)d * 2, (uint64_t)H * d * 2, 64,
                    1, 128, true) ||
      !make_tmap_3d(&mL, kv_latent, 2, R, (uint64_t)total_kv, 1, (uint64_t)R * 2,
                    (uint64_t)total_kv * R * 2, 64, 64, 1, true) ||
      !make_tmap_3d(&mWk, w_up_k, 2, d, H, R, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, RC,
                    true) ||
      !make_tmap_3d(&mWv, w_up_v, 2, d, H, R, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, 64,
                    true) ||
      !make_out_tmap(&mO, out, out_dtype == MLA_BF16, d, H, (uint64_t)total_q))
    return MLA_ERR_CUDA;
  FlashArgs fa = {};
  fa.B = B; fa.Tq = max_seqlen_q; fa.Tkv = 0; fa.H = H; fa.R = R; fa.RC = RC; fa.pair = pair;
  fa.row_blocks = (max_seqlen_q + 127) / 128; fa.splits = 1; fa.causal = causal ? 1 : 0;
  fa.d = d; fa.qscale = scale * 1.4426950408889634f; fa.out = out;
  fa.out_bf16 = out_dtype == MLA_BF16;
  fa.cu_q = cu_seqlens_q; fa.cu_kv = cu_seqlens_kv;
  fa.total_q = total_q; fa.total_kv = total_kv;
  return cuda_status(
      staged(1, stream, [&] { return launch_flash_fused(mQ, mL, mWk, mWv, mO, fa, stream); }));
}

mla_status_t mla_explicit_attention(const void* q, const void* k, const void* v, void* out, int B,
                                    int Tq, int Tkv, int H, int d, float scale, int causal,
                                    int in_dtype, int out_dtype, void* stream_) {
  if (!q || !k || !v || !out) return MLA_ERR_NULL;
  if (B <= 0 || Tq <= 0 || Tkv <= 0 || H <= 0 || Tq > Tkv) return MLA_ERR_SHAPE;
  if (d != 64 && d != 128) return MLA_ERR_SHAPE;
  if ((int64_t)B * Tq * H > kMaxIndex || (int64_t)B * Tkv * H > kMaxIndex) return MLA_ERR_SHAPE;
  if (in_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (out_dtype != MLA_F32 && out_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (!(aligned16(q) && aligned16(k) && aligned16(v) && aligned16(out))) return MLA_ERR_ALIGN;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const uint64_t BT = (uint64_t)B * Tq, BS = (uint64_t)B * Tkv;
  CUtensorMap mQ, mK, mV;
  if (!make_tmap_3d(&mQ, q, 2, d, H, BT, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, 128, true) ||
      !make_tmap_3d(&mK, k, 2, d, H, BS, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, 64, true) ||
      !make_tmap_3d(&mV, v, 2, d, H, BS, (uint64_t)d * 2, (uint64_t)H * d * 2, 64, 1, 64, true))
    return MLA_ERR_CUDA;
  FlashArgs fa = {};
  fa.B = B; fa.Tq = Tq; fa.Tkv = Tkv; fa.H = H; fa.R = d; fa.RC = d; fa.pair = 0;
  fa.row_blocks = (Tq + 127) / 128; fa.splits = 1; fa.causal = causal ? 1 : 0;
  fa.d = d; fa.qscale = scale * 1.4426950408889634f; fa.out = out;
  fa.out_bf16 = out_dtype == MLA_BF16;
  return cuda_status(
      staged(1, stream, [&] { return launch_flash_explicit(mQ, mK, mV, fa, stream); }));
}

mla_status_t mla_merge_partials(const float* m, const float* l, const float* o, void* out,
                                int parts, int rows, int width, int out_dtype, void* stream_) {
  if (!m || !l || !o || !out) return MLA_ERR_NULL;
  if (parts <= 0 || rows <= 0 || width <= 0 || width % 4 != 0) return MLA_ERR_SHAPE;
  if (out_dtype != MLA_F32 && out_dtype != MLA_BF16) return MLA_ERR_DTYPE;
  if (!aligned16(o) || !aligned16(out)) return MLA_ERR_ALIGN;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  return cuda_status(staged(2, stream, [&] {
    return launch_merge_partials(m, 1, l, o, out, parts, rows, width, out_dtype == MLA_BF16,
                                 stream);
  }));
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free attention: the scratch is this file's device array.
// ---------------------------------------------------------------------------
namespace mla {

// Device scratch of mla_latent_attention_noalloc, one copy per GPU that loads
// the library.  In host code this name is only a stand-in for the symbol: its
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[MLA_NOALLOC_SCRATCH_BYTES];

static std::mutex g_noalloc_mu;
static void* g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device.
static cudaError_t noalloc_scratch(void** addr) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_noalloc_addr[dev] = p;
  }
  *addr = g_noalloc_addr[dev];
  return cudaSuccess;
}

}  // namespace mla

extern "C" mla_status_t mla_latent_attention_noalloc(const void* q, const void* kv_latent,
                                                     const void* w_up_k, const void* w_up_v,
                                                     void* out, int B, int Tq, int Tkv, int H,
                                                     int d, int rank, float scale, int causal,
                                                     int in_dtype, int out_dtype, void* stream) {
  // The scratch the regular call would use: none when it falls back to the
  // warp path for pointers the tensor-core path cannot address.
  size_t need = mla_latent_attention_workspace_size(B, Tq, Tkv, H, d, rank, in_dtype, causal);
  if (need > 0 && mla::g_attn_path != 2 &&
      !mla::tc_pointers_ok(q, kv_latent, w_up_k, w_up_v, out))
    need = 0;
  if (need > (size_t)MLA_NOALLOC_SCRATCH_BYTES) return MLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0 && mla::noalloc_scratch(&scratch) != cudaSuccess) return MLA_ERR_CUDA;
  return mla_latent_attention(q, kv_latent, w_up_k, w_up_v, out, B, Tq, Tkv, H, d, rank, scale,
                              causal, in_dtype, out_dtype, scratch,
                              need > 0 ? (size_t)MLA_NOALLOC_SCRATCH_BYTES : 0, stream);
}
