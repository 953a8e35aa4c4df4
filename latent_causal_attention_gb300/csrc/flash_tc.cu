// Causal latent attention flash loop for sm_103a (tcgen05 + TMA + TMEM).
//
// Definition (page "FW-GLM-5-1 l2_p31", fused MLA-style attention from
// compressed KV latents, "The algorithm"): for each row (b, t, h),
//   logit_s = scale * q[b,t,h] . (latent[b,s] @ w_up_k[:,h])   for s <= t,
//   out = sum_s softmax(logit)_s * (latent[b,s] @ w_up_v[:,h]).
// The key weights are absorbed into the query beforehand, q' = w_up_k[:,h] q
// (length rank, pre-multiplied by scale * log2 e), so every head attends the
// SAME matrix, the latent rows themselves:
//   S = q' L^T (contraction over rank),  O_lat = softmax(S) L,
// and w_up_v is applied to O_lat afterwards, once per output row.  The
// softmax is the online (running max / running sum / rescaled accumulator)
// form of page "Kimi-K2.6 l2_p29" (online softmax derivation), evaluated in
// base 2, with its -inf rules: an entry at -inf contributes 0 and a row with
// no visible key yet keeps m = -inf without producing NaN.
//
// Tile: 128 rows (query position, head) x 64 keys.  The latent tile in shared
// memory (128-byte swizzle, rank-contiguous rows) is the B operand of both
// MMAs: K-major for S = q' L^T and MN-major for O += P L.  q' (bf16) sits in
// tensor memory as the A operand of S, so S reads only the latent tile from
// shared memory.  Tensor memory (512 columns x 128 lanes of 32 bits):
//   [0, RC)      O_lat, fp32         [256, 384)  two 64-column S buffers
//   [384, 512)   q', bf16 pairs (RC/2 columns)
// A 512-wide rank cannot keep O_lat next to S, so for rank > 256 two CTAs of a
// cluster split the rank: each holds q', the latent tiles and O_lat for its
// half and computes a partial S over its half; dedicated exchange warps send
// each partial S tile to the peer through distributed shared memory one step
// ahead of the softmax (four receive buffers).  The partial S travels as fp16;
// each CTA adds the peer's fp16 partial to its own fp32 partial, runs the
// softmax over the 128 x 64 tile and accumulates its half of O_lat with its own
// running max and sum (the two CTAs' logits differ only by the fp16 rounding of
// the partial each receives).
//
// Warp roles (512 threads): warp 0 lane 0 = TMA producer (q' once, then a
// 4-stage ring of latent tiles); warp 1 = TMEM owner, lane 0 issues the S MMAs;
// warp 15 lane 0 issues the O MMAs; warps 2-5 = partial-S
// exchange (CTA pair only); warps 6-13 = softmax and epilogue, two warps per
// row quadrant (each takes 32 of a tile's 64 keys and half of O_lat's
// columns); warp 14 forwards receive-buffer releases to the peer (CTA pair
// only).  Warp w reads TMEM lanes 32*(w%4)..+31.
#include <atomic>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kRows = 128;           // rows per CTA tile (MMA M)
constexpr int kKeys = 64;            // keys per tile (S MMA N, O MMA K)
constexpr int kStages = 4;           // latent tile ring
constexpr int kXBuf = 4;             // receive buffers of partial S (CTA pair)
constexpr int kMaxRC = 256;          // rank columns per CTA
constexpr int kThreads = 512;          // 16 warps
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O when the max grows by > 2^8

constexpr int kLStage = kKeys * kMaxRC * 2;       // 32 KB
constexpr int kPBytes = kRows * kKeys * 2;        // 16 KB
constexpr int kXBytes = kRows * kKeys * 2;        // 16 KB per receive buffer (fp16 partial S)
constexpr int kOffL = 0;
constexpr int kOffP = kOffL + kStages * kLStage;  // P, then receive buffers (prologue staging)
constexpr int kOffX = kOffP + 2 * kPBytes;
constexpr int kOffRed = kOffX + kXBuf * kXBytes;  // 2 x 128 floats: softmax warp-pair exchange
constexpr int kOffBar = kOffRed + 1024;
constexpr int kBarBytes = 512;
constexpr int kSmemBytes = kOffBar + kBarBytes + 1024;   // + barriers + alignment slack
static_assert(kSmemBytes <= 232448, "dynamic shared memory limit");

// Fused prefill staging (d <= 128, RC <= 256).  Prologue: the q tile (d/64 x
// 16 KB) in the P buffers and this CTA's w_up_k rows (d/64 x RC*128 B) in the
// receive buffers, both free until q' is in TMEM, so the latent ring starts at
// once.  Epilogue: w_up_v rows (d/64 x RC*128 B) in the ring stages that tiles
// nt and nt+1 would take (free as soon as P.L of tiles nt-4 and nt-3 has
// completed, so the load overlaps the end of the loop); the normalised O_lat
// goes to TMEM as bf16 (q''s columns) and the output tile, once computed, is
// staged for its tile store at the start of the ring.
static_assert(2 * kRows * 128 <= 2 * kPBytes, "q tile staging");
static_assert(2 * kMaxRC * 128 <= kXBuf * kXBytes, "w_up_k staging");
static_assert(kMaxRC * 128 <= kLStage, "w_up_v staging");

// CTA pair, fused epilogue: each CTA sends the peer the half of its partial
// output that the peer stores, as fp16 rows (128-byte-swizzled, dh/8 16-byte
// chunks per 128-byte row) multiplied by a power of two that puts the row's
// largest magnitude in [2^14, 2^15), followed by the inverse factors (one
// 16-byte slot per row).  The rounding is 2^-11 of the row's largest entry,
// below the bf16 rounding the normalised O_lat already takes before the output
// MMA; the scaling keeps any magnitude clear of fp16's range.
constexpr uint32_t kEpiScaleOff = kRows * 128;
__device__ __forceinline__ uint32_t epi_x_bytes(int dh) {
  return (uint32_t)(kRows * (dh * 2 + 16));
}

struct EpiStages {
  uint32_t wv_lo;    // stage of w_up_v chunk 0 (d columns 0..63)
  uint32_t wv_lbo;   // byte distance to chunk 1 (d columns 64..127)
};

__device__ __forceinline__ EpiStages epi_stages(int nt, int dch) {
  const uint32_t s0 = (uint32_t)(nt % kStages), s1 = (uint32_t)((nt + 1) % kStages);
  EpiStages e;
  e.wv_lo = dch > 1 ? min(s0, s1) : s0;
  e.wv_lbo = dch > 1 ? (max(s0, s1) - min(s0, s1)) * (uint32_t)kLStage : (uint32_t)kLStage;
  return e;
}

constexpr uint32_t kTmemO = 0;       // columns [0, RC)
constexpr uint32_t kTmemS = 256;     // two 64-column S buffers at 256, 320
constexpr uint32_t kTmemQ = 384;     // q' as bf16 pairs, RC/2 columns

struct Bars {
  uint64_t q_full;             // q' staged in shared memory (TMA)
  uint64_t q_ready;            // q' copied into tensor memory (softmax threads)
  uint64_t l_full[kStages];
  uint64_t l_empty[kStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];         // softmax threads (+ exchange threads in a pair)
  uint64_t p_full[2];
  uint64_t p_empty[2];
  uint64_t o_last;
  uint64_t x_full[kXBuf];      // my receive buffer b was filled by the peer
  uint64_t x_empty[kXBuf];     // the peer's receive buffer b may be written again
  uint64_t x_consumed[kXBuf];  // my softmax warps are done with my receive buffer b
  uint64_t pro_full;           // fused prefill: q tile and w_up_k staged (TMA)
  uint64_t pro_done;           // fused prefill: q . w_up_k^T computed into TMEM
  uint64_t epi_a;              // fused prefill: normalised O_lat (bf16) written to TMEM
  uint64_t epi_w;              // fused prefill: w_up_v staged (TMA)
  uint64_t epi_done;           // fused prefill: O_lat . w_up_v computed into TMEM
  uint64_t epi_x;              // fused prefill, CTA pair: the peer's partial output arrived
  uint32_t tmem_slot;
  int abort_flag;
};

static_assert(sizeof(Bars) <= kBarBytes, "barrier block");

// The barriers are initialised one per lane of warp 0: their index in the
// block above and the arrival count each expects.
constexpr int kNumBars = 37;
static_assert(offsetof(Bars, q_ready) == 1 * 8 && offsetof(Bars, s_empty) == 12 * 8 &&
                  offsetof(Bars, p_full) == 14 * 8 && offsetof(Bars, o_last) == 18 * 8 &&
                  offsetof(Bars, x_consumed) == 27 * 8 && offsetof(Bars, epi_a) == 33 * 8 &&
                  offsetof(Bars, epi_x) == (kNumBars - 1) * 8,
              "barrier indices");

__device__ __forceinline__ uint32_t bar_arrivals(int i, bool pair) {
  if (i == 1 || i == 14 || i == 15 || i == 33) return 256;   // q_ready, p_full, epi_a
  if (i == 12 || i == 13) return pair ? 384 : 256;           // s_empty (+ exchange warps)
  if (i == 18) return pair ? 2 : 3;                          // o_last: one per MMA issuer
  if (i >= 27 && i <= 30) return 8;                          // x_consumed: softmax warps
  return 1;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Every lane waits, then the warp agrees: a lane that timed out makes the whole
// warp give up, so warp-collective tcgen05 instructions never see a split warp.
template <bool kCluster = false>
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, int site,
                                          volatile int* abort) {
  const bool ok = mbar_wait<kCluster>(bar, parity, site, abort);
  return __all_sync(0xffffffffu, ok);
}

// Byte offset of 16-byte chunk ch of row r in rows of `row_bytes` (a multiple
// of 128): the low three chunk bits are XOR-ed with the row (bank spread).
__device__ __forceinline__ uint32_t xrow_offset(uint32_t r, uint32_t ch, uint32_t row_bytes) {
  return r * row_bytes + (((ch & ~7u) | ((ch ^ r) & 7u)) << 4);
}

// Two bf16 values (low half first) times s, rounded back to bf16 (bf16 -> fp32
// is exact: the bf16 bits are the high half of the fp32 word).
__device__ __forceinline__ uint32_t scale_bf16x2(uint32_t u, float s) {
  return pack_bf16x2(__uint_as_float(u << 16) * s, __uint_as_float(u & 0xffff0000u) * s);
}

// max(a, b, c) in one instruction (three-input max.f32, sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Tree max / sum of 32 values: log-depth dependency chains; three-input max
// and paired (float2) adds halve the instruction count.
__device__ __forceinline__ float tree_max32(const float (&v)[32]) {
  float a[11];
#pragma unroll
  for (int c = 0; c < 10; ++c) a[c] = fmax3(v[3 * c], v[3 * c + 1], v[3 * c + 2]);
  a[10] = fmaxf(v[30], v[31]);
  const float b0 = fmax3(a[0], a[1], a[2]), b1 = fmax3(a[3], a[4], a[5]);
  const float b2 = fmax3(a[6], a[7], a[8]), b3 = fmaxf(a[9], a[10]);
  return fmaxf(fmax3(b0, b1, b2), b3);
}

__device__ __forceinline__ float tree_sum32(const float (&v)[32]) {
  float2 a[8];
#pragma unroll
  for (int c = 0; c < 8; ++c)
    a[c] = __fadd2_rn(make_float2(v[2 * c], v[2 * c + 1]),
                      make_float2(v[2 * c + 16], v[2 * c + 17]));
#pragma unroll
  for (int c = 0; c < 4; ++c) a[c] = __fadd2_rn(a[c], a[c + 4]);
  a[0] = __fadd2_rn(a[0], a[2]);
  a[1] = __fadd2_rn(a[1], a[3]);
  a[0] = __fadd2_rn(a[0], a[1]);
  return a[0].x + a[0].y;
}

// This thread's row of fp32 TMEM columns [src, src+n) times s, as bf16 pairs at
// columns [dst, dst+n/2) (n a multiple of 32; two 32-column loads per wait).
__device__ __forceinline__ void tmem_rows_to_bf16(uint32_t src, uint32_t dst, int n, float s) {
  int c = 0;
  for (; c + 64 <= n; c += 64) {
    float v[2][32];
    tmem_ld32(src + c, v[0]);
    tmem_ld32(src + c + 32, v[1]);
    tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        const float2 t = __fmul2_rn(make_float2(v[h][2 * e], v[h][2 * e + 1]), make_float2(s, s));
        pk[e] = __uint_as_float(pack_bf16x2(t.x, t.y));
      }
      tmem_st16(dst + (c + 32 * h) / 2, pk);
    }
  }
  if (c < n) {
    float v[32];
    tmem_ld32(src + c, v);
    tmem_wait_ld();
    float pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e)
      pk[e] = __uint_as_float(pack_bf16x2(v[2 * e] * s, v[2 * e + 1] * s));
    tmem_st16(dst + c / 2, pk);
  }
}

// Kernel modes: head-packed rows with q' from the workspace; the fused per-head
// prefill (absorption and w_up_v inside); explicit K/V (per-head rows, K and V
// tiles in place of the latent, no up-projections).
constexpr int kModePacked = 0, kModeFused = 1, kModeExplicit = 2;

template <int kRC, int kMode>
__global__ void __launch_bounds__(kThreads, 1)
    flash_packed_kernel(const __grid_constant__ CUtensorMap mapQ,
                        const __grid_constant__ CUtensorMap mapL,
                        const __grid_constant__ CUtensorMap mapWk,
                        const __grid_constant__ CUtensorMap mapWv,
                        const __grid_constant__ CUtensorMap mapO, FlashArgs a) {
  extern __shared__ uint8_t flash_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(flash_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sL = smem + kOffL;
  uint8_t* sP = smem + kOffP;
  uint8_t* sX = smem + kOffX;
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort_flag = &bars->abort_flag;

  constexpr bool kFused = kMode == kModeFused;
  constexpr bool kExplicit = kMode == kModeExplicit;
  constexpr bool kPerHead = kMode != kModePacked;     // rows = query positions of one head
  static_assert(!kExplicit || kRC <= 128, "K and V tiles share one 32 KB stage");
  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int csize = a.pair ? 2 : 1;
  const uint32_t crank = a.pair ? cluster_ctarank() : 0u;
  const uint32_t peer = crank ^ 1u;

  // ---- work item: heavy row blocks first ----
  // Head-packed rows: row = i*H + h of one batch entry (q' from the workspace).
  // Fused prefill rows: row = query position i of one (batch entry, head).
  const int work = blockIdx.x / csize;
  const int per_rb = kPerHead ? a.B * a.H : a.B * a.splits;
  const int rb = a.row_blocks - 1 - work / per_rb;
  const int b = kPerHead ? (work % per_rb) / a.H : (work / a.splits) % a.B;
  const int head = kPerHead ? work % a.H : 0;
  const int sp = kPerHead ? 0 : work % a.splits;
  // batch entry b's query rows start at q0 and its keys at kv0 (of the packed
  // tensors of a variable-length batch, or b*Tq and b*Tkv otherwise)
  int q0 = b * a.Tq, kv0 = b * a.Tkv, Tq_b = a.Tq, Tkv_b = a.Tkv;
  const bool varlen = kPerHead && a.cu_q != nullptr;
  if (varlen) {
    grid_dep_wait();                       // the offsets may come from the previous kernel
    q0 = a.cu_q[b];
    Tq_b = a.cu_q[b + 1] - q0;
    kv0 = a.cu_kv[b];
    Tkv_b = a.cu_kv[b + 1] - kv0;
    if (q0 < 0 || Tq_b < 0 || q0 + Tq_b > a.total_q || kv0 < 0 || Tkv_b < Tq_b ||
        kv0 + Tkv_b > a.total_kv) {
      if (threadIdx.x == 0 && head == 0 && rb == a.row_blocks - 1 && crank == 0)
        report_error(kErrBadLengths | (unsigned)(b & 0xff));
      Tq_b = 0;                            // no rows: nothing read, nothing written
      Tkv_b = 0;
    }
  }
  const int rows_b = kPerHead ? Tq_b : a.Tq * a.H;
  const int row0 = rb * kRows;
  const int last_row = min(row0 + kRows, rows_b) - 1;
  const int t_max = Tkv_b - Tq_b + (kPerHead ? last_row : last_row / a.H);
  // (a row block past the end of its sequence, possible in a variable-length
  // batch, has no work)
  const int kv_len = row0 >= rows_b ? 0 : a.causal ? min(t_max + 1, Tkv_b) : Tkv_b;
  const int n_tiles_all = (kv_len + kKeys - 1) / kKeys;
  const int per_split = (n_tiles_all + a.splits - 1) / a.splits;
  const int tile0 = sp * per_split;
  const int nt = max(0, min(n_tiles_all, tile0 + per_split) - tile0);
  constexpr int RC = kRC;                  // rank columns per CTA
  const int c0 = (int)crank * RC;          // first rank column of this CTA
  constexpr int nchunk = RC / 64;
  constexpr uint32_t kVOff = kKeys * kRC * 2;   // explicit mode: V tile after the K tile

  if (warp == 0) {
    uint64_t* const bar0 = &bars->q_full;
    for (int i = lane; i < kNumBars; i += 32) mbar_init(bar0 + i, bar_arrivals(i, a.pair != 0));
    if (lane == 0) bars->abort_flag = 0;
    fence_mbarrier_init_cluster();   // every lane: its own inits
  }
  if (warp == 1) tmem_alloc(&bars->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  // CTA pair: every thread announces that this CTA's barriers exist; only the
  // warps that touch the peer's shared memory (exchange, release forwarding)
  // wait for the peer's announcement before their loops, the others just
  // before the exit barrier, so the round trip is off the prologue's path.
  const bool touches_peer = (warp >= 2 && warp < 6) || warp == 14;
  if (a.pair) cluster_arrive();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  grid_dep_wait();        // set-up above overlaps the previous kernel's tail

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0 && nt > 0) {
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapL);
      if constexpr (kFused) {
        // q tile (128 positions x d of one head) into the P buffers and this
        // CTA's rows of w_up_k into the receive buffers; the latent ring
        // starts at once
        const int dch = a.d / 64;
        mbar_arrive_expect_tx(&bars->pro_full, (uint32_t)(kRows * a.d * 2 + RC * a.d * 2));
        for (int kc = 0; kc < dch; ++kc) {
          tma_load_3d(sP + kc * (kRows * 128), &mapQ, &bars->pro_full, 64 * kc, head,
                      q0 + row0);
          tma_load_3d(sX + kc * (RC * 128), &mapWk, &bars->pro_full, 64 * kc, head, c0);
        }
      } else if constexpr (kExplicit) {
        // q tile (128 positions x d of one head) into the staging area
        mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(kRows * RC * 2));
        for (int kc = 0; kc < nchunk; ++kc)
          tma_load_3d(sP + kc * (kRows * 128), &mapQ, &bars->q_full, 64 * kc, head,
                      q0 + row0);
      } else {
        mbar_arrive_expect_tx(&bars->q_full, (uint32_t)(kRows * RC * 2));
        for (int kc = 0; kc < nchunk; ++kc)
          tma_load_3d(sP + kc * (kRows * 128), &mapQ, &bars->q_full, c0 + 64 * kc, row0, b);
      }
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int st = j % kStages;
        if (!mbar_wait(&bars->l_empty[st], ((j / kStages) & 1) ^ 1, 10, abort_flag)) break;
        uint8_t* dst = sL + st * kLStage;
        if constexpr (kExplicit) {
          // K and V tiles (64 keys x d of one head); keys past this sequence's end
          // belong to the next one (or are zero-filled) and are masked
          mbar_arrive_expect_tx(&bars->l_full[st], (uint32_t)(2 * kKeys * RC * 2));
          const int key = kv0 + (tile0 + j) * kKeys;
          for (int kc = 0; kc < nchunk; ++kc) {
            tma_load_3d(dst + kc * (kKeys * 128), &mapL, &bars->l_full[st], 64 * kc, head, key);
            tma_load_3d(dst + kVOff + kc * (kKeys * 128), &mapWk, &bars->l_full[st], 64 * kc,
                        head, key);
          }
        } else {
          mbar_arrive_expect_tx(&bars->l_full[st], (uint32_t)(kKeys * RC * 2));
          for (int kc = 0; kc < nchunk; ++kc)
            tma_load_3d(dst + kc * (kKeys * 128), &mapL, &bars->l_full[st], c0 + 64 * kc,
                        (varlen ? kv0 : 0) + (tile0 + j) * kKeys, varlen ? 0 : b);
        }
        ++issued;
      }
      // Do not leave copies in flight: wait for the last loads of each stage.
      for (int j = max(0, issued - kStages); j < issued; ++j)
        mbar_wait(&bars->l_full[j % kStages], (j / kStages) & 1, 11, nullptr);
      if constexpr (kFused) {
        // w_up_v rows of this CTA (MN-major B of the output MMA) into the ring
        // stages that tiles nt and nt+1 would take, as soon as they are free
        const int dch = a.d / 64;
        const EpiStages es = epi_stages(nt, dch);
        mbar_wait(&bars->pro_full, 0, 13, nullptr);     // the prologue copies have landed
        bool okw = issued == nt;
        for (int nc = 0; nc < dch && okw; ++nc)
          okw = mbar_wait(&bars->l_empty[(nt + nc) % kStages],
                          (((nt + nc) / kStages) & 1) ^ 1, 14, abort_flag);
        if (okw) {
          mbar_arrive_expect_tx(&bars->epi_w, (uint32_t)(RC * a.d * 2));
          for (int nc = 0; nc < dch; ++nc)
            for (int kb = 0; kb < RC / 64; ++kb)
              tma_load_3d(sL + es.wv_lo * kLStage + nc * es.wv_lbo + kb * (64 * 128), &mapWv,
                          &bars->epi_w, 64 * nc, head, c0 + 64 * kb);
          mbar_wait(&bars->epi_w, 0, 15, nullptr);
        }
      } else {
        mbar_wait(&bars->q_full, 0, 12, nullptr);
      }
    }
  } else if (warp == 1 || warp == 15 || (warp == 2 && !a.pair)) {
    // ======================= MMA issuers =======================
    // Issuing threads (lane 0) on different SM sub-partitions.  Lane 0 of warp
    // 1 issues the S(j) = q' L(j)^T MMAs (16 narrow N = 64 K-steps per tile;
    // it also issues the fused kernel's prologue and epilogue MMAs); one other
    // thread issues every O(j) += P(j) L(j) (four long N = RC K-steps).  A
    // thread that has just issued MMAs waits for the tensor core to take them
    // before its next barrier test completes, and a single thread issues N = 64
    // MMAs more slowly than the tensor core runs them; so in a single CTA the
    // S tiles are split between warp 1 (even j) and warp 15 (odd j) and warp 2,
    // which has no exchange to do there, issues the O MMAs; in a CTA pair warp
    // 15 issues the O MMAs.  The O MMAs come from one thread in tile order, so
    // the P.L products accumulate in tile order whatever the interleaving.
    // O_lat was zeroed by the softmax warps, so every P.L accumulates.
    const bool s_role = warp == 1 || (warp == 15 && !a.pair);
    const int s_first = (warp == 15) ? 1 : 0, s_step = a.pair ? 1 : 2;
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(kRows, kKeys, false, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(kRows, kRC, false, true);
      constexpr int kSSteps = kRC / 16;            // K-steps of one S tile
      const uint32_t l0 = smem_u32(sL), p0 = smem_u32(sP);
      const uint32_t tq = tmem + kTmemQ;
      bool ok = true;
      if constexpr (kFused) {
        if (warp == 1) {
          // q' (fp32, this CTA's rank columns) = q . w_up_k[:, h, c0:c0+RC]^T into O's columns
          ok = mbar_wait(&bars->pro_full, 0, 24, abort_flag);
          tc_fence_after();
          if (ok) {
            constexpr uint32_t idesc_q = make_idesc_bf16(kRows, kRC, false, false);
            const uint64_t aq = make_sdesc_sw128(p0, 16, 1024);
            const uint64_t bw = make_sdesc_sw128(smem_u32(sX), 16, 1024);
            for (int k = 0; k < a.d / 16; ++k)
              umma_bf16(tmem + kTmemO,
                        aq + (uint64_t)(((k >> 2) * (kRows * 128) + (k & 3) * 32) >> 4),
                        bw + (uint64_t)(((k >> 2) * (kRC * 128) + (k & 3) * 32) >> 4), idesc_q,
                        k > 0 ? 1u : 0u);
          }
          umma_commit(&bars->pro_done);
        }
      }
      ok = ok && mbar_wait(&bars->q_ready, 0, 20, abort_flag);
      tc_fence_after();
      // S K-step k of a tile: A = q' columns [8k, 8k+8) of TMEM, B = latent K-chunk k/4
#define MLA_S_STEP(sbuf, bd, k)                                                          \
  umma_bf16_ta((sbuf), tq + (k) * 8,                                                     \
               (bd) + (uint64_t)((((k) >> 2) * (kKeys * 128) + ((k) & 3) * 32) >> 4), idesc_s, \
               (k) > 0 ? 1u : 0u)
      if (s_role) {
        // S(j) as soon as latent tile j has landed and the readers of S(j-2)
        // have let its buffer go
        for (int js = s_first; ok && js < nt; js += s_step) {
          const int sb = js & 1;
          ok = mbar_wait(&bars->l_full[js % kStages], (js / kStages) & 1, 22, abort_flag) &&
               mbar_wait(&bars->s_empty[sb], ((js >> 1) & 1) ^ 1, 23, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t bds = make_sdesc_sw128(l0 + (js % kStages) * kLStage, 16, 1024);
          const uint32_t sbuf = tmem + kTmemS + sb * kKeys;
#pragma unroll
          for (int k = 0; k < kSSteps; ++k) MLA_S_STEP(sbuf, bds, k);
          umma_commit(&bars->s_full[sb]);
        }
      } else {
        // O(j) as soon as P(j) is written; its completion frees P buffer j%2
        // and latent stage j%kStages
        for (int jo = 0; ok && jo < nt; ++jo) {
          const int pb = jo & 1;
          ok = mbar_wait(&bars->p_full[pb], (jo >> 1) & 1, 21, abort_flag);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ad = make_sdesc_sw128(p0 + pb * kPBytes, 16, 1024);
          const uint64_t bdo = make_sdesc_sw128(
              l0 + (jo % kStages) * kLStage + (kExplicit ? kVOff : 0u), kKeys * 128, 1024);
#pragma unroll
          for (int kk = 0; kk < kKeys / 16; ++kk)
            umma_bf16(tmem + kTmemO, ad + (uint64_t)((kk * 32) >> 4),
                      bdo + (uint64_t)((kk * 2048) >> 4), idesc_o, 1u);
          umma_commit(&bars->p_empty[pb]);
          umma_commit(&bars->l_empty[jo % kStages]);
        }
      }
#undef MLA_S_STEP
      umma_commit(&bars->o_last);
      if constexpr (kFused) {
        if (warp == 1) {
          // out_partial = O_lat(bf16, smem) . w_up_v[c0:c0+RC, h, :] into S's columns
          if (ok && mbar_wait(&bars->epi_a, 0, 25, abort_flag) &&
              mbar_wait(&bars->epi_w, 0, 26, abort_flag)) {
            tc_fence_after();
            const uint32_t idesc_v = make_idesc_bf16(kRows, a.d, false, true);
            const EpiStages es = epi_stages(nt, a.d / 64);
            const uint64_t bv = make_sdesc_sw128(l0 + es.wv_lo * kLStage, es.wv_lbo, 1024);
#pragma unroll
            for (int k = 0; k < kRC / 16; ++k)
              umma_bf16_ta(tmem + kTmemS, tq + k * 8, bv + (uint64_t)((k * 2048) >> 4), idesc_v,
                           k > 0 ? 1u : 0u);
          }
          umma_commit(&bars->epi_done);
        }
      }
    }
  } else if (warp < 6) {
    // ======================= partial-S exchange (CTA pair) =======================
    if (a.pair) cluster_wait();
    if (a.pair && nt > 0) {
      const int qd = warp & 3;
      const uint32_t r = (uint32_t)(qd * 32 + lane);
      const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
      const uint32_t x_peer0 = mapa_shared(smem_u32(sX), peer);
      const uint32_t xfull_peer0 = mapa_shared(smem_u32(&bars->x_full[0]), peer);
      for (int j = 0; j < nt; ++j) {
        const int bi = j & 1, k = j >> 1;                 // S buffer and its use count
        const int xb = j % kXBuf, xk = j / kXBuf;         // receive buffer and its use count
        // the peer's receive buffer first (normally free long before S is ready),
        // so that the partial leaves as soon as S(j) is complete
        if (!warp_wait<true>(&bars->x_empty[xb], xk & 1, 41, abort_flag)) break;
        if (!warp_wait(&bars->s_full[bi], k & 1, 40, abort_flag)) break;
        tc_fence_after();
        const uint32_t dst = x_peer0 + xb * kXBytes;
        const uint32_t bar = xfull_peer0 + xb * 8;
        float v[2][32];                           // my row, both 32-column halves in flight
        tmem_ld32(tmem + lane_base + kTmemS + bi * kKeys, v[0]);
        tmem_ld32(tmem + lane_base + kTmemS + bi * kKeys + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_empty[bi]);          // S(j) is in registers
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)            // sent as fp16
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_async_v4u(dst + sw128_offset(r, hh * 4 + c),
                         pack_half2(v[hh][8 * c], v[hh][8 * c + 1]),
                         pack_half2(v[hh][8 * c + 2], v[hh][8 * c + 3]),
                         pack_half2(v[hh][8 * c + 4], v[hh][8 * c + 5]),
                         pack_half2(v[hh][8 * c + 6], v[hh][8 * c + 7]), bar);
      }
      if constexpr (kFused) {
        // send the peer the half of this CTA's partial output that the peer stores,
        // once the peer's receive buffers are free (their last release)
        const int dh = a.d / 2;
        const int send0 = (int)peer * dh;
        bool okx = warp_wait(&bars->epi_done, 0, 42, abort_flag);
        for (int xb = 0; xb < kXBuf; ++xb)          // last release of each receive buffer
          okx = okx && warp_wait<true>(&bars->x_empty[xb], ((nt - xb + kXBuf - 1) / kXBuf) & 1,
                                       43, abort_flag);
        if (okx) {
          tc_fence_after();
          const uint32_t epx_peer = mapa_shared(smem_u32(&bars->epi_x), peer);
          float v[4][16];                               // dh <= 64 columns of my row
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
            if (c4 * 16 < dh) tmem_ld16(tmem + lane_base + kTmemS + send0 + c4 * 16, v[c4]);
          tmem_wait_ld();
          float mx = 0.f;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (c4 * 16 < dh) mx = fmaxf(mx, fabsf(v[c4][e]));
          // 2^(14 - exponent of mx), as a biased exponent kept inside [1, 253]
          const int ex = (int)((__float_as_uint(mx) >> 23) & 0xffu);
          const uint32_t sb = (uint32_t)min(max(268 - ex, 1), 253);
          const float sc = __uint_as_float(sb << 23);
          const float inv_sc = __uint_as_float((254u - sb) << 23);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (c4 * 16 < dh) {
                const float* w = &v[c4][8 * h];
                st_async_v4u(x_peer0 + xrow_offset(r, (uint32_t)(2 * c4 + h), 128u),
                             pack_half2(w[0] * sc, w[1] * sc), pack_half2(w[2] * sc, w[3] * sc),
                             pack_half2(w[4] * sc, w[5] * sc), pack_half2(w[6] * sc, w[7] * sc),
                             epx_peer);
              }
          st_async_v4u(x_peer0 + kEpiScaleOff + r * 16, __float_as_uint(inv_sc), 0u, 0u, 0u,
                       epx_peer);
        }
      }
    }
  } else if (warp == 14) {
    // ======================= release forwarding (CTA pair) =======================
    // Passes "my receive buffer b is free" from the local softmax warps to the
    // peer's x_empty[b]: the initial release of every buffer, then one per tile.
    // The cluster-scope arrival is a round trip; keeping it on this warp keeps
    // it off the softmax warps' path.
    if (a.pair) cluster_wait();
    if (a.pair && nt > 0 && lane == 0) {
      const uint32_t xe_peer0 = mapa_shared(smem_u32(&bars->x_empty[0]), peer);
      for (int n = 0; n < nt + kXBuf; ++n) {
        // n < kXBuf: the initial release of buffer n; then tile j = n - kXBuf
        const int xb = n < kXBuf ? n : (n - kXBuf) % kXBuf;
        const int ph = n < kXBuf ? 0 : (n - kXBuf) / kXBuf + 1;   // completion index
        if (!mbar_wait(&bars->x_consumed[xb], ph & 1, 45, abort_flag)) break;
        mbar_arrive_remote(xe_peer0 + xb * 8);
      }
    }
  } else {
    // ======================= softmax / epilogue =======================
    // Two warps per TMEM lane quadrant: the same 32 rows, keys split in halves
    // of 32 (and O's columns split in halves for rescaling and the epilogue).
    const int qd = warp & 3;                      // TMEM lane quadrant
    const int half = (warp - 6) >> 2;             // 0: keys 0..31, 1: keys 32..63
    const int r = qd * 32 + lane;                 // row within the tile
    const int grow = row0 + r;                    // row within batch entry b
    const bool row_valid = grow < rows_b;
    const int t_row = Tkv_b - Tq_b + (row_valid ? (kPerHead ? grow : grow / a.H) : 0);
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t x_local = smem_u32(sX);
    float* red = reinterpret_cast<float*>(smem + kOffRed);   // [2][128] partner exchange
    const uint32_t bar_id = 1u + (uint32_t)qd;               // named barrier of the warp pair
    const int oc0 = half * (RC / 2);                          // O columns handled by this warp

    float m_run = -INFINITY, l_half = 0.f;
    bool ok = nt > 0;
    if (ok) {
      if constexpr (kFused) {
        // q' (fp32 in O's columns) -> scaled by scale*log2(e) -> bf16 pairs in TMEM
        ok = warp_wait(&bars->pro_done, 0, 28, abort_flag);
        if (ok) {
          tc_fence_after();
          tmem_rows_to_bf16(tmem + lane_base + kTmemO + oc0, tmem + lane_base + kTmemQ + oc0 / 2,
                            RC / 2, a.qscale);
          if (a.pair && warp == 6 && lane == 0)
            mbar_arrive_expect_tx(&bars->epi_x, epi_x_bytes(a.d / 2));
        }
      } else {
      // q' (staged by TMA in the receive buffers, 128-byte swizzled rows) -> TMEM
      ok = warp_wait(&bars->q_full, 0, 29, abort_flag);
      if (ok) {
        const uint32_t qs = smem_u32(sP);
        for (int kc = half; kc < nchunk; kc += 2) {
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t u0, u1, u2, u3;
            const uint32_t addr = qs + kc * (kRows * 128) + sw128_offset((uint32_t)r, (uint32_t)c);
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(u0), "=r"(u1), "=r"(u2), "=r"(u3)
                         : "r"(addr)
                         : "memory");
            if constexpr (kExplicit) {     // raw q: fold in scale * log2(e)
              u0 = scale_bf16x2(u0, a.qscale); u1 = scale_bf16x2(u1, a.qscale);
              u2 = scale_bf16x2(u2, a.qscale); u3 = scale_bf16x2(u3, a.qscale);
            }
            asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(
                             tmem + lane_base + kTmemQ + kc * 32 + c * 4),
                         "r"(u0), "r"(u1), "r"(u2), "r"(u3)
                         : "memory");
          }
        }
      }
      }
      if (ok) {
        // O_lat starts at zero (every P.L accumulates): my quadrant, my half of the columns
        float z[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) z[e] = 0.f;
        for (int c = oc0; c < oc0 + RC / 2; c += 32) tmem_st32(tmem + lane_base + kTmemO + c, z);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->q_ready);
        if (a.pair) {                 // my receive buffers may now be written by the peer
          if (warp == 6 && lane == 0)     // arm the receive barriers of the first tiles
            for (int xb = 0; xb < kXBuf && xb < nt; ++xb)
              mbar_arrive_expect_tx(&bars->x_full[xb], (uint32_t)kXBytes);
          // every lane's reads are consumed before __syncwarp; the forwarding
          // warp passes the release on to the peer
          __syncwarp();
          if (lane == 0)
            for (int xb = 0; xb < kXBuf; ++xb) mbar_arrive(&bars->x_consumed[xb]);
        }
      }
    }
    for (int j = 0; j < nt && ok; ++j) {
      const int bi = j & 1, k = j >> 1;
      float s[32];
      if (!warp_wait(&bars->s_full[bi], k & 1, 30, abort_flag)) { ok = false; break; }
      tc_fence_after();
      tmem_ld32(tmem + lane_base + kTmemS + bi * kKeys + half * 32, s);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(&bars->s_empty[bi]);      // S(j) is in registers: the buffer may be refilled

      if (a.pair) {
        // the peer's partial S over its half of the rank (my 32 keys)
        const int xb = j % kXBuf, xk = j / kXBuf;
        if (!warp_wait<true>(&bars->x_full[xb], xk & 1, 32, abort_flag)) { ok = false; break; }
        const uint32_t src = x_local + xb * kXBytes;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t u0, u1, u2, u3;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(u0), "=r"(u1), "=r"(u2), "=r"(u3)
                       : "r"(src + sw128_offset((uint32_t)r, (uint32_t)(half * 4 + c)))
                       : "memory");
          const float2 f[4] = {unpack_half2(u0), unpack_half2(u1), unpack_half2(u2),
                               unpack_half2(u3)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 t = __fadd2_rn(make_float2(s[8 * c + 2 * e], s[8 * c + 2 * e + 1]), f[e]);
            s[8 * c + 2 * e] = t.x;
            s[8 * c + 2 * e + 1] = t.y;
          }
        }
      }

      // mask: key s_idx visible iff s_idx < Tkv and (not causal or s_idx <= t)
      const int key0 = (tile0 + j) * kKeys + half * 32;
      const int lim = a.causal ? min(t_row + 1, Tkv_b) : Tkv_b;   // visible keys < lim
      if (!row_valid || key0 + 32 > lim) {
#pragma unroll
        for (int c = 0; c < 32; ++c)
          if (!row_valid || key0 + c >= lim) s[c] = -INFINITY;
      }
      const float mx_half = tree_max32(s);
      // row max over both halves through shared memory
      red[half * 128 + r] = mx_half;
      named_bar_sync(bar_id, 64);
      const float mx = fmaxf(mx_half, red[(half ^ 1) * 128 + r]);
      named_bar_sync(bar_id, 64);
      const float m_new = fmaxf(m_run, mx);
      const bool grow_max = m_new > m_run + kRescaleThreshold;   // false while both -inf
      const float m_ref = grow_max ? m_new : m_run;
      const float alpha = grow_max ? ex2(m_run - m_new) : 1.f;   // m_run = -inf -> 0
      const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float2 t = __fadd2_rn(make_float2(s[2 * c], s[2 * c + 1]), make_float2(-m_use, -m_use));
        s[2 * c] = ex2(t.x);
        s[2 * c + 1] = ex2(t.y);
      }
      l_half = l_half * alpha + tree_sum32(s);
      m_run = m_ref;

      // P(j-2).L(j-2) has finished reading P buffer bi
      if (!warp_wait(&bars->p_empty[bi], (k & 1) ^ 1, 34, abort_flag)) { ok = false; break; }
      // rescale my half of O_lat's columns once every earlier P.L has landed:
      // O(j-1) and O(j-2) complete (each issuer's commit covers its earlier MMAs)
      if (__any_sync(0xffffffffu, grow_max && j > 0)) {
        if (!warp_wait(&bars->p_empty[(j - 1) & 1], ((j - 1) >> 1) & 1, 33, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int c = oc0; c < oc0 + RC / 2; c += 16) {
          float o[16];
          tmem_ld16(tmem + lane_base + kTmemO + c, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float2 t = __fmul2_rn(make_float2(o[2 * e], o[2 * e + 1]), make_float2(alpha, alpha));
            o[2 * e] = t.x;
            o[2 * e + 1] = t.y;
          }
          tmem_st16(tmem + lane_base + kTmemO + c, o);
        }
        tmem_wait_st();
      }

      // P (bf16) into the K-major swizzled P buffer: my 4 of the row's 8 chunks
      const uint32_t pb = smem_u32(sP + bi * kPBytes);
#pragma unroll
      for (int c = 0; c < 4; ++c)
        st_shared_v4(pb + sw128_offset(r, half * 4 + c), pack_bf16x2(s[8 * c], s[8 * c + 1]),
                     pack_bf16x2(s[8 * c + 2], s[8 * c + 3]),
                     pack_bf16x2(s[8 * c + 4], s[8 * c + 5]),
                     pack_bf16x2(s[8 * c + 6], s[8 * c + 7]));
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&bars->p_full[bi]);
      if (a.pair) {
        // the receive buffer is released off the softmax chain (the peer writes it
        // again only four tiles later): re-arm its barrier for tile j+kXBuf (its
        // phase for tile j is complete), then pass the release on
        const int xb = j % kXBuf;
        if (warp == 6 && lane == 0 && j + kXBuf < nt)
          mbar_arrive_expect_tx(&bars->x_full[xb], (uint32_t)kXBytes);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->x_consumed[xb]);
      }
    }

    // ---------------- epilogue ----------------
    // the row sum is the two halves' sums (added in the same order in both warps)
    red[half * 128 + r] = l_half;
    named_bar_sync(bar_id, 64);
    const float l_run = red[r] + red[128 + r];
    const int64_t gr = (int64_t)b * rows_b + grow;     // row in (B*Tq*H)
    const int64_t nrows = (int64_t)a.B * rows_b;
    bool have_o = false;
    if (ok && nt > 0) {
      have_o = warp_wait(&bars->o_last, 0, 35, abort_flag);
      tc_fence_after();
    }
    if constexpr (kFused) {
      // normalised O_lat as bf16 pairs in q''s columns (free once the last S
      // has been computed): the A operand of the output MMA, from TMEM
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      if (have_o) {
        tmem_rows_to_bf16(tmem + lane_base + kTmemO + oc0, tmem + lane_base + kTmemQ + oc0 / 2,
                          RC / 2, inv);
      } else {
        float z[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) z[e] = 0.f;
        for (int c = oc0; c < oc0 + RC / 2; c += 32)
          tmem_st16(tmem + lane_base + kTmemQ + c / 2, z);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->epi_a);
      // out[b, i, h, :] = O_lat . w_up_v[:, h, :]; a CTA pair adds the peer's
      // partial product for the half of the columns this CTA stores
      bool have_out = have_o && warp_wait(&bars->epi_done, 0, 36, abort_flag);
      tc_fence_after();
      const int dh = a.pair ? a.d / 2 : a.d;                 // columns stored by this CTA
      const int cfirst = (a.pair ? (int)crank * dh : 0) + half * (dh / 2);
      bool have_peer = true;
      if (a.pair) have_peer = have_out && warp_wait<true>(&bars->epi_x, 0, 37, abort_flag);
      const int64_t orow = (((int64_t)q0 + grow) * a.H + head) * a.d;
      // A full 128-row block leaves as tile stores of 128 x 128-byte boxes,
      // staged (128-byte swizzle) in the latent ring, which the output MMA no
      // longer reads; the rows of a partial block, or a column range narrower
      // than one box, are written one by one.
      const int box_cols = a.out_bf16 ? 64 : 32;
      const bool tile_store = row0 + kRows <= rows_b && dh % box_cols == 0;
      const int cbase = a.pair ? (int)crank * dh : 0;        // first column stored here
      const uint32_t stage0 = smem_u32(sL);
      for (int c = cfirst; c < cfirst + dh / 2; c += 16) {
        float v[16];
        if (have_out) {
          tmem_ld16(tmem + lane_base + kTmemS + c, v);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 16; ++e) v[e] = 0.f;
        }
        if (a.pair && have_peer) {
          const int cc = c - (int)crank * dh;          // column within the received half
          float inv_sc, y0, y1, y2;
          ld_shared_v4f(x_local + kEpiScaleOff + (uint32_t)r * 16, inv_sc, y0, y1, y2);
#pragma unroll
          for (int q = 0; q < 2; ++q) {               // 16 columns = 2 chunks of 8 fp16
            float x[4];
            ld_shared_v4f(x_local + xrow_offset((uint32_t)r, (uint32_t)((cc >> 3) + q), 128u),
                          x[0], x[1], x[2], x[3]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = unpack_half2(__float_as_uint(x[e]));
              v[8 * q + 2 * e] += f.x * inv_sc;
              v[8 * q + 2 * e + 1] += f.y * inv_sc;
            }
          }
        }
        if (tile_store) {
          const int cr = c - cbase;
          const uint32_t box = stage0 + (uint32_t)(cr / box_cols) * (kRows * 128);
          if (a.out_bf16) {
            const uint32_t ch = (uint32_t)((cr % 64) >> 3);      // 16 columns = 2 chunks
            st_shared_v4(box + sw128_offset((uint32_t)r, ch), pack_bf16x2(v[0], v[1]),
                         pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                         pack_bf16x2(v[6], v[7]));
            st_shared_v4(box + sw128_offset((uint32_t)r, ch + 1), pack_bf16x2(v[8], v[9]),
                         pack_bf16x2(v[10], v[11]), pack_bf16x2(v[12], v[13]),
                         pack_bf16x2(v[14], v[15]));
          } else {
            const uint32_t ch = (uint32_t)((cr % 32) >> 2);      // 16 columns = 4 chunks
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(box + sw128_offset((uint32_t)r, ch + (uint32_t)q),
                           __float_as_uint(v[4 * q]), __float_as_uint(v[4 * q + 1]),
                           __float_as_uint(v[4 * q + 2]), __float_as_uint(v[4 * q + 3]));
          }
        } else if (row_valid && have_peer) {
          if (a.out_bf16) {
            uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow + c);
            d4[0] = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                               pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
            d4[1] = make_uint4(pack_bf16x2(v[8], v[9]), pack_bf16x2(v[10], v[11]),
                               pack_bf16x2(v[12], v[13]), pack_bf16x2(v[14], v[15]));
          } else {
            float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow + c);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
          }
        }
      }
      if (tile_store) {
        // all eight softmax warps have staged their columns: one thread stores
        fence_proxy_async_smem();
        named_bar_sync(5, 256);
        if (warp == 6 && lane == 0 && have_peer) {
          for (int bx = 0; bx < dh / box_cols; ++bx)
            tma_store_3d(&mapO, stage0 + (uint32_t)bx * (kRows * 128), cbase + bx * box_cols,
                         head, q0 + row0);
          bulk_commit_group();
          bulk_wait_read_all();     // the staging must outlive the reads, not the writes
        }
      }
    } else if constexpr (kExplicit) {
      // out[b, i, h, :] = O / l, fp32 or bf16; my half of the d columns
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      const int64_t orow = (((int64_t)q0 + grow) * a.H + head) * a.d;
      for (int c = oc0; c < oc0 + RC / 2; c += 32) {
        float o[32];
        if (have_o) {
          tmem_ld32(tmem + lane_base + kTmemO + c, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = 0.f;
        }
        if (!row_valid) continue;
        if (a.out_bf16) {
          uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow + c);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            d4[q] = make_uint4(pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv),
                               pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                               pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                               pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
        } else {
          float4* d4 = reinterpret_cast<float4*>(static_cast<float*>(a.out) + orow + c);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            d4[q] = make_float4(o[4 * q] * inv, o[4 * q + 1] * inv, o[4 * q + 2] * inv,
                                o[4 * q + 3] * inv);
        }
      }
    } else {
      if (a.splits == 1) {
        const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.olat) + gr * a.R + c0;
        for (int c = oc0; c < oc0 + RC / 2; c += 32) {
          float o[32];
          if (have_o) {
            tmem_ld32(tmem + lane_base + kTmemO + c, o);
            tmem_wait_ld();
          } else {
  #pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0.f;
          }
          if (row_valid) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c);
  #pragma unroll
            for (int q = 0; q < 4; ++q)
              d4[q] = make_uint4(pack_bf16x2(o[8 * q] * inv, o[8 * q + 1] * inv),
                                 pack_bf16x2(o[8 * q + 2] * inv, o[8 * q + 3] * inv),
                                 pack_bf16x2(o[8 * q + 4] * inv, o[8 * q + 5] * inv),
                                 pack_bf16x2(o[8 * q + 6] * inv, o[8 * q + 7] * inv));
          }
        }
      } else {
        float* dst = a.part_o + ((int64_t)sp * nrows + gr) * a.R + c0;
        for (int c = oc0; c < oc0 + RC / 2; c += 32) {
          float o[32];
          if (have_o) {
            tmem_ld32(tmem + lane_base + kTmemO + c, o);
            tmem_wait_ld();
          } else {
  #pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = 0.f;
          }
          if (row_valid) {
            float4* d4 = reinterpret_cast<float4*>(dst + c);
  #pragma unroll
            for (int q = 0; q < 8; ++q)
              d4[q] = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
          }
        }
        if (row_valid && crank == 0 && half == 0) {
          float* ml = a.part_ml + ((int64_t)sp * nrows + gr) * 2;
          ml[0] = have_o ? m_run : -INFINITY;
          ml[1] = have_o ? l_run : 0.f;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (a.pair) {
    if (!touches_peer) cluster_wait();
    cluster_sync();     // neither CTA leaves while the other may still address it
  }
}

// ---------------------------------------------------------------------------
// Persistent single-CTA prefill (rank <= 256, d = 64): one resident CTA per
// SM works through a list of (batch entry, head, 128-row block) items, so
// that an item's set-up runs under the previous item's loop and epilogue.
// The arithmetic of each item is the fused kernel's (same MMA sequences, same
// softmax), so results are bit for bit those of flash_packed_kernel<RC, fused>.
//
//   shared memory: latent ring (4 x 32 KB), P (2 x 16 KB), staging (64 KB: the
//     next item's q tile at +0 and w_up_k rows at +16 KB), row-max exchange;
//   tensor memory: as the fused kernel (O_lat, two S buffers, q').
//
// Roles: warp 0 lane 0 TMA producer (q / w_up_k of each item as soon as the
// previous item's absorption has read the staging, latent tiles into the
// ring, w_up_v into the ring slot after the item's last tile); warp 1 lane 0
// the absorption MMA, the S MMAs of even tiles and the output MMA; warp 15
// lane 0 the S MMAs of odd tiles; warp 2 lane 0 the O MMAs; warps 6-13
// softmax, normalisation and q' conversion; warps 3, 4, 5 and 14 (one per
// TMEM lane quadrant) the output.  Item boundary: the softmax warps normalise
// O_lat into q''s columns (epi_a), warp 1 issues the output MMA and then the
// next item's absorption into O's columns; the output warps read the output
// from S's columns, stage it in the P buffers and write it with tile stores
// (stg_free once read out); the softmax warps turn the next q' into bf16 and
// zero O (q_ready, with the output warps' read) and write their next P only
// after stg_free.
//
// Items are dealt in rounds of gridDim.x, heavy row blocks first, alternating
// direction every round (CTA c takes items c, 2G-1-c, 2G+c, ...), which
// balances the causal work between CTAs without a shared counter.  Ring slots
// and S / P buffers are counted across items (a ring slot per latent tile and
// one for the item's w_up_v); each per-item barrier completes once per item.
// ---------------------------------------------------------------------------
struct PBars {
  uint64_t l_full[kStages];    // ring slot landed (latent tile; w_up_v slots: plain arrive)
  uint64_t l_empty[kStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];         // softmax threads have read S
  uint64_t p_full[2];          // softmax threads have written P
  uint64_t p_empty[2];
  uint64_t pro_full;           // the item's q tile and w_up_k rows staged (TMA)
  uint64_t pro_done;           // absorption MMA done: staging free, q' (fp32) in O's columns
  uint64_t q_ready;            // q' (bf16) in TMEM and O zeroed (softmax threads)
  uint64_t o_last;             // every MMA of the item's loop has completed (three issuers)
  uint64_t epi_a;              // normalised O_lat (bf16) in q''s columns (softmax threads)
  uint64_t epi_done;           // output MMA done
  uint64_t epi_w[2];           // w_up_v of item r staged (TMA), by item parity: the
                               // producer may stage item r+1's before item r's is used
  uint64_t stg_free;           // the item's output staging (P buffers) has been read out
  uint32_t tmem_slot;
  int abort_flag;
};
constexpr int kPNumBars = 25;
static_assert(offsetof(PBars, s_empty) == 10 * 8 && offsetof(PBars, p_full) == 12 * 8 &&
                  offsetof(PBars, q_ready) == 18 * 8 && offsetof(PBars, o_last) == 19 * 8 &&
                  offsetof(PBars, epi_a) == 20 * 8 && offsetof(PBars, epi_w) == 22 * 8 &&
                  offsetof(PBars, stg_free) == 24 * 8,
              "persistent barrier indices");
static_assert(sizeof(PBars) <= kBarBytes, "persistent barrier block");

__device__ __forceinline__ uint32_t pbar_arrivals(int i) {
  if (i == 18) return 384;                         // q_ready: softmax + output warps
  if (i == 10 || i == 11 || i == 12 || i == 13 || i == 20) return 256;
  if (i == 19) return 3;
  return 1;
}

struct PItem {
  int b, head, row0, nt;
};

// Item of round r for worker c of G (a CTA, or a CTA pair); false when the
// list is exhausted.
__device__ __forceinline__ bool persist_item(const FlashArgs& a, int r, int G, int c, PItem& it) {
  const int w = r * G + ((r & 1) ? G - 1 - c : c);
  const int per_rb = a.B * a.H;
  if (w >= a.row_blocks * per_rb) return false;
  const int rb = a.row_blocks - 1 - w / per_rb;
  it.b = (w % per_rb) / a.H;
  it.head = w % a.H;
  it.row0 = rb * kRows;
  const int last_row = min(it.row0 + kRows, a.Tq) - 1;
  const int t_max = a.Tkv - a.Tq + last_row;
  const int kv_len = a.causal ? min(t_max + 1, a.Tkv) : a.Tkv;
  it.nt = (kv_len + kKeys - 1) / kKeys;
  return true;
}

template <int kRC>
__global__ void __launch_bounds__(kThreads, 1)
    flash_persistent_kernel(const __grid_constant__ CUtensorMap mapQ,
                            const __grid_constant__ CUtensorMap mapL,
                            const __grid_constant__ CUtensorMap mapWk,
                            const __grid_constant__ CUtensorMap mapWv,
                            const __grid_constant__ CUtensorMap mapO, FlashArgs a) {
  extern __shared__ uint8_t flash_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(flash_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sL = smem + kOffL;
  uint8_t* sP = smem + kOffP;
  uint8_t* sX = smem + kOffX;                 // staging: q tile at +0, w_up_k at +16 KB
  PBars* bars = reinterpret_cast<PBars*>(smem + kOffBar);
  volatile int* abort_flag = &bars->abort_flag;
  constexpr int RC = kRC;
  constexpr uint32_t kWkOff = kRows * 128;    // 16 KB: after the q tile (d = 64)
  static_assert(kWkOff + RC * 128 <= kXBuf * kXBytes, "persistent staging");
  static_assert(RC * 128 <= kLStage, "w_up_v slot");

  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) {
    uint64_t* const bar0 = &bars->l_full[0];
    for (int i = lane; i < kPNumBars; i += 32) mbar_init(bar0 + i, pbar_arrivals(i));
    if (lane == 0) bars->abort_flag = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 1) tmem_alloc(&bars->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  grid_dep_wait();        // set-up above overlaps the previous kernel's tail

  if (warp == 0) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapL);
      int R = 0, hi = 0, armed = -1, armed_w = -1;   // next ring slot, slots armed, last items staged
      bool ok = true;
      PItem it;
      for (int r = 0; ok && persist_item(a, r, (int)gridDim.x, (int)blockIdx.x, it); ++r) {
        // the staging is free once the previous item's absorption has read it
        if (r > 0 && !(ok = mbar_wait(&bars->pro_done, (r - 1) & 1, 60, abort_flag))) break;
        mbar_arrive_expect_tx(&bars->pro_full, (uint32_t)(kRows * 128 + RC * 128));
        tma_load_3d(sX, &mapQ, &bars->pro_full, 0, it.head, it.b * a.Tq + it.row0);
        tma_load_3d(sX + kWkOff, &mapWk, &bars->pro_full, 0, it.head, 0);
        armed = r;
        for (int j = 0; j < it.nt; ++j) {
          const int slot = R + j, st = slot % kStages;
          if (!(ok = mbar_wait(&bars->l_empty[st], ((slot / kStages) & 1) ^ 1, 61, abort_flag)))
            break;
          mbar_arrive_expect_tx(&bars->l_full[st], (uint32_t)(kKeys * RC * 2));
          for (int kc = 0; kc < RC / 64; ++kc)
            tma_load_3d(sL + st * kLStage + kc * (kKeys * 128), &mapL, &bars->l_full[st], 64 * kc,
                        j * kKeys, it.b);
          hi = slot + 1;
        }
        if (!ok) break;
        // w_up_v rows of the head (MN-major B of the output MMA) into the next slot
        const int slot = R + it.nt, st = slot % kStages;
        if (!(ok = mbar_wait(&bars->l_empty[st], ((slot / kStages) & 1) ^ 1, 62, abort_flag)))
          break;
        mbar_arrive(&bars->l_full[st]);              // the slot's phase, nothing to wait for
        uint64_t* ew = &bars->epi_w[r & 1];
        mbar_arrive_expect_tx(ew, (uint32_t)(RC * 128));
        for (int kb = 0; kb < RC / 64; ++kb)
          tma_load_3d(sL + st * kLStage + kb * (64 * 128), &mapWv, ew, 0, it.head, 64 * kb);
        hi = slot + 1;
        armed_w = r;
        R += it.nt + 1;
      }
      if (!ok) {
        // leave no copy in flight: the last slot of every stage and the last
        // item's staging (bounded waits)
        for (int slot = max(0, hi - kStages); slot < hi; ++slot)
          mbar_wait(&bars->l_full[slot % kStages], (slot / kStages) & 1, 63, nullptr);
        if (armed >= 0) mbar_wait(&bars->pro_full, armed & 1, 63, nullptr);
        if (armed_w >= 0) mbar_wait(&bars->epi_w[armed_w & 1], (armed_w >> 1) & 1, 63, nullptr);
      }
    }
  } else if (warp == 1 || warp == 15 || warp == 2) {
    // ======================= MMA issuers =======================
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(kRows, kKeys, false, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(kRows, kRC, false, true);
      constexpr uint32_t idesc_q = make_idesc_bf16(kRows, kRC, false, false);
      constexpr uint32_t idesc_v = make_idesc_bf16(kRows, 64, false, true);
      constexpr int kSSteps = kRC / 16;
      const uint32_t l0 = smem_u32(sL), p0 = smem_u32(sP), x0 = smem_u32(sX);
      const uint32_t tq = tmem + kTmemQ;
      // output MMA of an item: out = O_lat(bf16, q''s columns) . w_up_v into S's columns
      auto output_mma = [&](int r, int wslot) -> bool {
        if (!mbar_wait(&bars->epi_a, r & 1, 64, abort_flag) ||
            !mbar_wait(&bars->epi_w[r & 1], (r >> 1) & 1, 65, abort_flag)) {
          umma_commit(&bars->epi_done);
          return false;
        }
        tc_fence_after();
        const uint64_t bv = make_sdesc_sw128(l0 + (wslot % kStages) * kLStage, kLStage, 1024);
#pragma unroll
        for (int k = 0; k < kRC / 16; ++k)
          umma_bf16_ta(tmem + kTmemS, tq + k * 8, bv + (uint64_t)((k * 2048) >> 4), idesc_v,
                       k > 0 ? 1u : 0u);
        umma_commit(&bars->epi_done);
        umma_commit(&bars->l_empty[wslot % kStages]);
        return true;
      };
      int T = 0, R = 0, prev_wslot = -1;
      bool ok = true;
      PItem it;
      int r = 0;
      for (; ok && persist_item(a, r, (int)gridDim.x, (int)blockIdx.x, it); ++r) {
        if (warp == 1) {
          if (r > 0) ok = output_mma(r - 1, prev_wslot);
          // this item's q' (fp32) = q . w_up_k[:, h, :]^T into O's columns, which the
          // previous item's normalisation has read (epi_a, waited just above)
          ok = ok && mbar_wait(&bars->pro_full, r & 1, 66, abort_flag);
          if (ok) {
            tc_fence_after();
            const uint64_t aq = make_sdesc_sw128(x0, 16, 1024);
            const uint64_t bw = make_sdesc_sw128(x0 + kWkOff, 16, 1024);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              umma_bf16(tmem + kTmemO, aq + (uint64_t)((k * 32) >> 4),
                        bw + (uint64_t)((k * 32) >> 4), idesc_q, k > 0 ? 1u : 0u);
          }
          umma_commit(&bars->pro_done);
        }
        ok = ok && mbar_wait(&bars->q_ready, r & 1, 67, abort_flag);
        tc_fence_after();
        if (warp != 2) {
          // S(j) = q' L(j)^T for this thread's tiles (global tile count even / odd)
          const int par = warp == 1 ? 0 : 1;
          for (int j = 0; ok && j < it.nt; ++j) {
            const int g = T + j;
            if ((g & 1) != par) continue;
            const int slot = R + j, st = slot % kStages;
            ok = mbar_wait(&bars->l_full[st], (slot / kStages) & 1, 68, abort_flag) &&
                 mbar_wait(&bars->s_empty[g & 1], ((g >> 1) & 1) ^ 1, 69, abort_flag);
            if (!ok) break;
            tc_fence_after();
            const uint64_t bds = make_sdesc_sw128(l0 + st * kLStage, 16, 1024);
            const uint32_t sbuf = tmem + kTmemS + (g & 1) * kKeys;
#pragma unroll
            for (int k = 0; k < kSSteps; ++k)
              umma_bf16_ta(sbuf, tq + k * 8,
                           bds + (uint64_t)((((k) >> 2) * (kKeys * 128) + ((k) & 3) * 32) >> 4),
                           idesc_s, k > 0 ? 1u : 0u);
            umma_commit(&bars->s_full[g & 1]);
          }
        } else {
          // O(j) += P(j) L(j), in tile order from this one thread
          for (int j = 0; ok && j < it.nt; ++j) {
            const int g = T + j, pb = g & 1;
            const int st = (R + j) % kStages;
            if (!(ok = mbar_wait(&bars->p_full[pb], (g >> 1) & 1, 70, abort_flag))) break;
            tc_fence_after();
            const uint64_t ad = make_sdesc_sw128(p0 + pb * kPBytes, 16, 1024);
            const uint64_t bdo = make_sdesc_sw128(l0 + st * kLStage, kKeys * 128, 1024);
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)
              umma_bf16(tmem + kTmemO, ad + (uint64_t)((kk * 32) >> 4),
                        bdo + (uint64_t)((kk * 2048) >> 4), idesc_o, 1u);
            umma_commit(&bars->p_empty[pb]);
            umma_commit(&bars->l_empty[st]);
          }
        }
        umma_commit(&bars->o_last);
        prev_wslot = R + it.nt;
        T += it.nt;
        R += it.nt + 1;
      }
      if (warp == 1 && ok && r > 0) output_mma(r - 1, prev_wslot);
    }
  } else if (warp >= 6 && warp < 14) {
    // ======================= softmax / epilogue =======================
    const int qd = warp & 3;
    const int half = (warp - 6) >> 2;
    const int r_ = qd * 32 + lane;                // row within the tile
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    float* red = reinterpret_cast<float*>(smem + kOffRed);
    const uint32_t bar_id = 1u + (uint32_t)qd;
    const int oc0 = half * (RC / 2);
    int T = 0;
    bool ok = true;
    PItem it;
    for (int r = 0; ok && persist_item(a, r, (int)gridDim.x, (int)blockIdx.x, it); ++r) {
      const int grow = it.row0 + r_;
      const bool row_valid = grow < a.Tq;
      const int t_row = a.Tkv - a.Tq + (row_valid ? grow : 0);
      // q' (fp32 in O's columns) -> scaled by scale*log2(e) -> bf16 pairs in TMEM;
      // q''s columns are free once the previous item's output MMA has read them
      if (!(ok = warp_wait(&bars->pro_done, r & 1, 71, abort_flag))) break;
      tc_fence_after();
      tmem_rows_to_bf16(tmem + lane_base + kTmemO + oc0, tmem + lane_base + kTmemQ + oc0 / 2,
                        RC / 2, a.qscale);
      {
        float z[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) z[e] = 0.f;
        for (int c = oc0; c < oc0 + RC / 2; c += 32) tmem_st32(tmem + lane_base + kTmemO + c, z);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->q_ready);

      float m_run = -INFINITY, l_half = 0.f;
      for (int j = 0; j < it.nt; ++j) {
        const int g = T + j, bi = g & 1, k = g >> 1;
        float s[32];
        if (!(ok = warp_wait(&bars->s_full[bi], k & 1, 72, abort_flag))) break;
        tc_fence_after();
        tmem_ld32(tmem + lane_base + kTmemS + bi * kKeys + half * 32, s);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_empty[bi]);
        const int key0 = j * kKeys + half * 32;
        const int lim = a.causal ? min(t_row + 1, a.Tkv) : a.Tkv;
        if (!row_valid || key0 + 32 > lim) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (!row_valid || key0 + c >= lim) s[c] = -INFINITY;
        }
        const float mx_half = tree_max32(s);
        red[half * 128 + r_] = mx_half;
        named_bar_sync(bar_id, 64);
        const float mx = fmaxf(mx_half, red[(half ^ 1) * 128 + r_]);
        named_bar_sync(bar_id, 64);
        const float m_new = fmaxf(m_run, mx);
        const bool grow_max = m_new > m_run + kRescaleThreshold;
        const float m_ref = grow_max ? m_new : m_run;
        const float alpha = grow_max ? ex2(m_run - m_new) : 1.f;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float2 t = __fadd2_rn(make_float2(s[2 * c], s[2 * c + 1]),
                                      make_float2(-m_use, -m_use));
          s[2 * c] = ex2(t.x);
          s[2 * c + 1] = ex2(t.y);
        }
        l_half = l_half * alpha + tree_sum32(s);
        m_run = m_ref;
        if (!(ok = warp_wait(&bars->p_empty[bi], (k & 1) ^ 1, 73, abort_flag))) break;
        if (__any_sync(0xffffffffu, grow_max && j > 0)) {
          if (!(ok = warp_wait(&bars->p_empty[(g - 1) & 1], ((g - 1) >> 1) & 1, 74, abort_flag)))
            break;
          tc_fence_after();
          for (int c = oc0; c < oc0 + RC / 2; c += 16) {
            float o[16];
            tmem_ld16(tmem + lane_base + kTmemO + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float2 t = __fmul2_rn(make_float2(o[2 * e], o[2 * e + 1]),
                                          make_float2(alpha, alpha));
              o[2 * e] = t.x;
              o[2 * e + 1] = t.y;
            }
            tmem_st16(tmem + lane_base + kTmemO + c, o);
          }
          tmem_wait_st();
        }
        // the previous item's output staging has been read out of the P buffers
        if (j == 0 && r > 0 && !(ok = warp_wait(&bars->stg_free, (r - 1) & 1, 78, abort_flag)))
          break;
        const uint32_t pb = smem_u32(sP + bi * kPBytes);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_shared_v4(pb + sw128_offset(r_, half * 4 + c), pack_bf16x2(s[8 * c], s[8 * c + 1]),
                       pack_bf16x2(s[8 * c + 2], s[8 * c + 3]),
                       pack_bf16x2(s[8 * c + 4], s[8 * c + 5]),
                       pack_bf16x2(s[8 * c + 6], s[8 * c + 7]));
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[bi]);
      }
      if (!ok) break;

      // ---------------- epilogue of the item ----------------
      red[half * 128 + r_] = l_half;
      named_bar_sync(bar_id, 64);
      const float l_run = red[r_] + red[128 + r_];
      named_bar_sync(bar_id, 64);              // red[] is reused by the next item
      if (!(ok = warp_wait(&bars->o_last, r & 1, 75, abort_flag))) break;
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      tmem_rows_to_bf16(tmem + lane_base + kTmemO + oc0, tmem + lane_base + kTmemQ + oc0 / 2,
                        RC / 2, inv);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->epi_a);
      T += it.nt;
    }
  } else if ((warp >= 3 && warp <= 5) || warp == 14) {
    // ======================= item outputs =======================
    // out[b, i, h, 0..64) of the previous item by tile stores of 128 x 128-byte
    // boxes staged (128-byte swizzle) in the P buffers, free between the item's
    // last O MMA and the next item's first P; the map is per batch entry, so the
    // rows of a partial block past the sequence's end are not written
    const int qd = warp & 3;                       // lane quadrant of this warp
    const uint32_t rr = (uint32_t)(qd * 32 + lane);
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t row = smem_u32(sP) + rr * 128, sw = rr & 7;
    bool ok = true;
    PItem it;
    for (int r = 0; ok; ++r) {
      const bool have = persist_item(a, r, (int)gridDim.x, (int)blockIdx.x, it);
      if (r > 0) {
        if (!(ok = warp_wait(&bars->epi_done, (r - 1) & 1, 76, abort_flag))) break;
        tc_fence_after();
        float v[2][32];
        tmem_ld32(tmem + lane_base + kTmemS, v[0]);
        tmem_ld32(tmem + lane_base + kTmemS + 32, v[1]);
        tmem_wait_ld();
        tc_fence_before();
        if (have) mbar_arrive(&bars->q_ready);   // item r's S may overwrite the output
        PItem prev;
        persist_item(a, r - 1, (int)gridDim.x, (int)blockIdx.x, prev);
        if (a.out_bf16) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float* w = &v[q >> 2][8 * (q & 3)];
            st_shared_v4(row + ((((uint32_t)q) ^ sw) << 4), pack_bf16x2(w[0], w[1]),
                         pack_bf16x2(w[2], w[3]), pack_bf16x2(w[4], w[5]),
                         pack_bf16x2(w[6], w[7]));
          }
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float* w = &v[q >> 3][4 * (q & 7)];
            st_shared_v4(row + (uint32_t)(q >> 3) * (kRows * 128) + ((((uint32_t)q & 7u) ^ sw) << 4),
                         __float_as_uint(w[0]), __float_as_uint(w[1]), __float_as_uint(w[2]),
                         __float_as_uint(w[3]));
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(6, 128);                    // all four warps have staged their rows
        if (warp == 3 && lane == 0) {
          const int nbox = a.out_bf16 ? 1 : 2;
          for (int bx = 0; bx < nbox; ++bx)
            tma_store_4d(&mapO, smem_u32(sP) + (uint32_t)bx * (kRows * 128), bx * (64 / nbox),
                         prev.head, prev.row0, prev.b);
          bulk_commit_group();
          bulk_wait_read_all();                    // the staging must outlive the reads
          mbar_arrive(&bars->stg_free);
        }
      } else if (have) {
        mbar_arrive(&bars->q_ready);
      }
      if (!have) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
// Persistent CTA-pair prefill (rank 384 or 512: each CTA of a cluster of two
// holds RC = rank / 2 rank columns; d = 64 or 128): one resident pair per two
// SMs works through the (batch entry, head, 128-row block) items in the order
// of the single-CTA kernel, and both CTAs of a pair take the same items.  The
// arithmetic of an item is the fused kernel's (same MMA sequences, softmax,
// partial-S and partial-output exchange), so the results are bit for bit those
// of flash_packed_kernel<RC, fused> with a CTA pair.
//
// What changes is the item boundary.  The fused kernel ends an item with the
// normalisation, the output MMA, the exchange of the partial outputs and the
// stores, and the next CTA then starts with its set-up, the q / w_up_k loads
// and the absorption.  Here the output MMA of item r and the absorption of
// item r+1 are issued back to back, and the exchange and stores of item r's
// output run while item r+1's first score tile is computed and exchanged.
//
// Shared memory per item:
//   ring slots (32 KB each, counted across items): w_up_k of the head (one
//     slot per 64 d columns, the absorption's B), the latent tiles, w_up_v
//     (one slot per 64 d columns, the output MMA's B);
//   receive buffers: with T the global index of the item's first tile, the
//     q tile of the item sits in buffers T%4 and (T+1)%4 (one per 64 d
//     columns) and the peer's partial output of the previous item in buffers
//     (T+2)%4 (fp16 rows) and (T+3)%4 (row factors); these are the buffers of
//     the previous item's last four tiles, so they are free before the item
//     boundary.  Tile g uses buffer g%4, as in the fused kernel.
//
// Receive-buffer releases: the peer writes a buffer (a partial S tile or a
// partial output) only after the release of its previous write, forwarded by
// warp 14 from the local consumers (x_consumed -> the peer's x_empty), so the
// n-th write into a buffer waits for the n-th release; both sides keep the
// parity of each buffer's next release in a 4-bit mask.  A buffer that is to
// take the next item's q tile is not released after its last use: its release
// waits until the absorption has read the q tile.
//
// Roles: warp 0 lane 0 ring producer; warp 1 lane 0 absorption, S MMAs and
// output MMA; warp 15 lane 0 O MMAs; warps 2-5 partial-S exchange and, at an
// item boundary, the output: the peer's half sent, this CTA's half added to
// the peer's partial and stored (tile stores staged in the P buffers, which
// the softmax threads write again only after stg_free); warp 14 lane 0
// release forwarding and the q-tile loads (it sees every consumption of the
// receive buffers in order); warps 6-13 softmax, normalisation and the q'
// conversion.
// ---------------------------------------------------------------------------
struct QBars {
  uint64_t l_full[kStages];    // ring slot landed (latent tile, w_up_k or w_up_v rows)
  uint64_t l_empty[kStages];
  uint64_t s_full[2];
  uint64_t s_empty[2];         // softmax and exchange threads have read S
  uint64_t p_full[2];
  uint64_t p_empty[2];
  uint64_t pro_full;           // the item's q tile staged in the receive buffers (TMA)
  uint64_t pro_done;           // absorption MMA done
  uint64_t q_ready;            // q' in TMEM, O zeroed, the previous output read (softmax + exchange)
  uint64_t o_last;             // the item's S and O MMAs have completed (two issuers)
  uint64_t epi_a;              // normalised O_lat (bf16) in q''s columns, the item's last S read
  uint64_t epi_done;           // output MMA done
  uint64_t x_full[kXBuf];      // my receive buffer b holds the peer's partial S of a tile
  uint64_t x_empty[kXBuf];     // the peer's receive buffer b may be used again
  uint64_t x_consumed[kXBuf];  // my softmax threads are done with my receive buffer b
  uint64_t epi_x;              // the peer's partial output of the item has arrived
  uint64_t stg_free;           // the item's output staging (P buffers) has been read out
  uint32_t tmem_slot;
  int abort_flag;
};
constexpr int kQNumBars = 36;
static_assert(offsetof(QBars, s_empty) == 10 * 8 && offsetof(QBars, p_full) == 12 * 8 &&
                  offsetof(QBars, q_ready) == 18 * 8 && offsetof(QBars, o_last) == 19 * 8 &&
                  offsetof(QBars, epi_a) == 20 * 8 && offsetof(QBars, x_consumed) == 30 * 8 &&
                  offsetof(QBars, epi_x) == 34 * 8 && offsetof(QBars, stg_free) == 35 * 8,
              "pair persistent barrier indices");
static_assert(sizeof(QBars) <= kBarBytes, "pair persistent barrier block");

__device__ __forceinline__ uint32_t qbar_arrivals(int i) {
  if (i == 10 || i == 11 || i == 18 || i == 20) return 384;   // s_empty, q_ready, epi_a
  if (i == 12 || i == 13) return 256;                         // p_full
  if (i == 19) return 2;                             // o_last
  if (i >= 30 && i <= 33) return 8;                  // x_consumed
  return 1;
}

// The w_up_v slots of an item, s and s+1 (d = 128) or s alone: d chunk nc lives
// at stage lo + nc * lbo / 32 KB (the lower stage first, whatever the slot order).
__device__ __forceinline__ EpiStages wv_stages(int s, int dch) {
  const uint32_t s0 = (uint32_t)(s % kStages), s1 = (uint32_t)((s + 1) % kStages);
  EpiStages e;
  e.wv_lo = dch > 1 ? min(s0, s1) : s0;
  e.wv_lbo = dch > 1 ? (max(s0, s1) - min(s0, s1)) * (uint32_t)kLStage : (uint32_t)kLStage;
  return e;
}

// The pair kernel's item of round r: the pair index and count are re-read from
// the special registers at each call (cheap) instead of being kept live.
__device__ __forceinline__ bool pair_item(const FlashArgs& a, int r, PItem& it) {
  uint32_t cta, ncta;
  asm volatile("mov.u32 %0, %%ctaid.x;" : "=r"(cta));
  asm volatile("mov.u32 %0, %%nctaid.x;" : "=r"(ncta));
  return persist_item(a, r, (int)(ncta >> 1), (int)(cta >> 1), it);
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

template <int kRC, int kD>
__global__ void __launch_bounds__(kThreads, 1)
    flash_persistent_pair_kernel(const __grid_constant__ CUtensorMap mapQ,
                                 const __grid_constant__ CUtensorMap mapL,
                                 const __grid_constant__ CUtensorMap mapWk,
                                 const __grid_constant__ CUtensorMap mapWv,
                                 const __grid_constant__ CUtensorMap mapO, FlashArgs a) {
  extern __shared__ uint8_t flash_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(flash_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sL = smem + kOffL;
  uint8_t* sX = smem + kOffX;
  QBars* bars = reinterpret_cast<QBars*>(smem + kOffBar);
  volatile int* abort_flag = &bars->abort_flag;
  constexpr int RC = kRC;
  static_assert(RC * 128 <= kLStage, "weight slot");

  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_ctarank();
  const uint32_t peer = crank ^ 1u;
  const int c0 = (int)crank * RC;                               // first rank column here
  constexpr int dch = kD / 64;                                 // 64-column chunks of d
  constexpr int dh = kD / 2;                                   // output columns stored here

  if (warp == 0) {
    uint64_t* const bar0 = &bars->l_full[0];
    for (int i = lane; i < kQNumBars; i += 32) mbar_init(bar0 + i, qbar_arrivals(i));
    if (lane == 0) bars->abort_flag = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 1) tmem_alloc(&bars->tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  const bool touches_peer = (warp >= 2 && warp < 6) || warp == 14;
  cluster_arrive();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_slot;
  grid_dep_wait();

  if (warp == 0) {
    // ======================= ring producer =======================
    if (lane == 0) {
      prefetch_tensormap(&mapL);
      prefetch_tensormap(&mapWk);
      prefetch_tensormap(&mapWv);
      int S = 0, hi = 0;                   // next ring slot, slots issued
      bool ok = true;
      PItem it;
      for (int r = 0; ok && pair_item(a, r, it); ++r) {
        // w_up_k rows of this CTA's rank columns, one slot per 64 d columns; every
        // chunk completes on the first slot's barrier (the others just arrive)
        for (int kc = 0; ok && kc < dch; ++kc) {
          const int slot = S + kc;
          ok = mbar_wait(&bars->l_empty[slot % kStages], ((slot / kStages) & 1) ^ 1, 80,
                         abort_flag);
        }
        if (!ok) break;
        {
          uint64_t* bar = &bars->l_full[S % kStages];
          mbar_arrive_expect_tx(bar, (uint32_t)(dch * RC * 128));
          for (int kc = 1; kc < dch; ++kc) mbar_arrive(&bars->l_full[(S + kc) % kStages]);
          for (int kc = 0; kc < dch; ++kc)
            tma_load_3d(sL + ((S + kc) % kStages) * kLStage, &mapWk, bar, 64 * kc, it.head, c0);
          hi = S + dch;
        }
        S += dch;
        for (int j = 0; ok && j < it.nt; ++j) {
          const int slot = S + j, st = slot % kStages;
          if (!(ok = mbar_wait(&bars->l_empty[st], ((slot / kStages) & 1) ^ 1, 81, abort_flag)))
            break;
          mbar_arrive_expect_tx(&bars->l_full[st], (uint32_t)(kKeys * RC * 2));
          for (int kc = 0; kc < RC / 64; ++kc)
            tma_load_3d(sL + st * kLStage + kc * (kKeys * 128), &mapL, &bars->l_full[st],
                        c0 + 64 * kc, j * kKeys, it.b);
          hi = slot + 1;
        }
        S += it.nt;
        // w_up_v rows (MN-major B of the output MMA): both slots free first
        for (int nc = 0; ok && nc < dch; ++nc) {
          const int slot = S + nc;
          ok = mbar_wait(&bars->l_empty[slot % kStages], ((slot / kStages) & 1) ^ 1, 82,
                         abort_flag);
        }
        if (!ok) break;
        const EpiStages ws = wv_stages(S, dch);
        {
          uint64_t* bar = &bars->l_full[S % kStages];     // all chunks on the first slot's
          mbar_arrive_expect_tx(bar, (uint32_t)(dch * RC * 128));
          for (int nc = 1; nc < dch; ++nc) mbar_arrive(&bars->l_full[(S + nc) % kStages]);
          for (int nc = 0; nc < dch; ++nc)
            for (int kb = 0; kb < RC / 64; ++kb)
              tma_load_3d(sL + ws.wv_lo * kLStage + nc * ws.wv_lbo + kb * (64 * 128), &mapWv, bar,
                          64 * nc, it.head, c0 + 64 * kb);
        }
        hi = S + dch;
        S += dch;
      }
      if (!ok) {
        // leave no copy in flight: the last slot of every stage (bounded waits)
        for (int slot = max(0, hi - kStages); slot < hi; ++slot)
          mbar_wait(&bars->l_full[slot % kStages], (slot / kStages) & 1, 83, nullptr);
      }
    }
  } else if (warp == 1 || warp == 15) {
    // ======================= MMA issuers =======================
    if (lane == 0) {
      constexpr uint32_t idesc_s = make_idesc_bf16(kRows, kKeys, false, false);
      constexpr uint32_t idesc_o = make_idesc_bf16(kRows, kRC, false, true);
      constexpr uint32_t idesc_q = make_idesc_bf16(kRows, kRC, false, false);
      constexpr uint32_t idesc_v = make_idesc_bf16(kRows, kD, false, true);
      constexpr int kSSteps = kRC / 16;
      const uint32_t l0 = smem_u32(sL), p0 = smem_u32(smem + kOffP), x0 = smem_u32(sX);
      const uint32_t tq = tmem + kTmemQ;
      // output MMA of an item: out_partial = O_lat(bf16, q''s columns) . w_up_v into
      // S's columns, once the normalisation is done and the item's last S tiles have
      // been read (epi_a) and w_up_v has landed (the first slot's barrier)
      auto output_mma = [&](int r, int wv_slot) -> bool {
        const bool good =
            mbar_wait(&bars->epi_a, r & 1, 84, abort_flag) &&
            mbar_wait(&bars->l_full[wv_slot % kStages], (wv_slot / kStages) & 1, 86, abort_flag);
        if (!good) {
          umma_commit(&bars->epi_done);
          return false;
        }
        tc_fence_after();
        const EpiStages ws = wv_stages(wv_slot, dch);
        const uint64_t bv = make_sdesc_sw128(l0 + ws.wv_lo * kLStage, ws.wv_lbo, 1024);
#pragma unroll
        for (int k = 0; k < kRC / 16; ++k)
          umma_bf16_ta(tmem + kTmemS, tq + k * 8, bv + (uint64_t)((k * 2048) >> 4), idesc_v,
                       k > 0 ? 1u : 0u);
        umma_commit(&bars->epi_done);
        for (int nc = 0; nc < dch; ++nc) umma_commit(&bars->l_empty[(wv_slot + nc) % kStages]);
        return true;
      };
      int T = 0, S = 0, r = 0, prev_wv = 0;
      bool ok = true;
      PItem it;
      for (; ok && pair_item(a, r, it); ++r) {
        const int wk_slot = S, l_slot = S + dch;
        if (warp == 1) {
          if (r > 0) ok = output_mma(r - 1, prev_wv);
          // q' (fp32, this CTA's rank columns) = q . w_up_k^T into O's columns; A = the
          // q tile in receive buffers T%4 and (T+1)%4, B = the w_up_k slots
          ok = ok && mbar_wait(&bars->pro_full, r & 1, 87, abort_flag) &&
               mbar_wait(&bars->l_full[wk_slot % kStages], (wk_slot / kStages) & 1, 88, abort_flag);
          if (ok) {
            tc_fence_after();
            for (int kc = 0; kc < dch; ++kc) {
              const uint64_t aq = make_sdesc_sw128(x0 + (uint32_t)((T + kc) & 3) * kXBytes, 16, 1024);
              const uint64_t bw =
                  make_sdesc_sw128(l0 + (uint32_t)((wk_slot + kc) % kStages) * kLStage, 16, 1024);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                umma_bf16(tmem + kTmemO, aq + (uint64_t)((k * 32) >> 4),
                          bw + (uint64_t)((k * 32) >> 4), idesc_q, (kc | k) ? 1u : 0u);
            }
          }
          umma_commit(&bars->pro_done);
          if (ok)
            for (int kc = 0; kc < dch; ++kc) umma_commit(&bars->l_empty[(wk_slot + kc) % kStages]);
        }
        ok = ok && mbar_wait(&bars->q_ready, r & 1, 89, abort_flag);
        tc_fence_after();
        if (warp == 1) {
          // S(g) = q' L(g)^T as soon as the tile has landed and S(g-2) has been read
          for (int j = 0; ok && j < it.nt; ++j) {
            const int g = T + j, slot = l_slot + j, st = slot % kStages;
            ok = mbar_wait(&bars->l_full[st], (slot / kStages) & 1, 90, abort_flag) &&
                 mbar_wait(&bars->s_empty[g & 1], ((g >> 1) & 1) ^ 1, 91, abort_flag);
            if (!ok) break;
            tc_fence_after();
            const uint64_t bds = make_sdesc_sw128(l0 + st * kLStage, 16, 1024);
            const uint32_t sbuf = tmem + kTmemS + (g & 1) * kKeys;
#pragma unroll
            for (int k = 0; k < kSSteps; ++k)
              umma_bf16_ta(sbuf, tq + k * 8,
                           bds + (uint64_t)((((k) >> 2) * (kKeys * 128) + ((k) & 3) * 32) >> 4),
                           idesc_s, k > 0 ? 1u : 0u);
            umma_commit(&bars->s_full[g & 1]);
          }
        } else {
          // O(g) += P(g) L(g), in tile order from this one thread
          for (int j = 0; ok && j < it.nt; ++j) {
            const int g = T + j, pb = g & 1, st = (l_slot + j) % kStages;
            if (!(ok = mbar_wait(&bars->p_full[pb], (g >> 1) & 1, 92, abort_flag))) break;
            tc_fence_after();
            const uint64_t ad = make_sdesc_sw128(p0 + pb * kPBytes, 16, 1024);
            const uint64_t bdo = make_sdesc_sw128(l0 + st * kLStage, kKeys * 128, 1024);
#pragma unroll
            for (int kk = 0; kk < kKeys / 16; ++kk)   // the item's first product starts O
              umma_bf16(tmem + kTmemO, ad + (uint64_t)((kk * 32) >> 4),
                        bdo + (uint64_t)((kk * 2048) >> 4), idesc_o, (j | kk) ? 1u : 0u);
            umma_commit(&bars->p_empty[pb]);
            umma_commit(&bars->l_empty[st]);
          }
        }
        umma_commit(&bars->o_last);
        prev_wv = l_slot + it.nt;
        T += it.nt;
        S = l_slot + it.nt + dch;
      }
      if (warp == 1 && ok && r > 0) output_mma(r - 1, prev_wv);
    }
  } else if (warp < 6) {
    // ======================= exchange with the peer =======================
    cluster_wait();
    const int qd = warp & 3;
    const uint32_t rr = (uint32_t)(qd * 32 + lane);
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t x_peer0 = mapa_shared(smem_u32(sX), peer);
    const uint32_t xfull_peer0 = mapa_shared(smem_u32(&bars->x_full[0]), peer);
    const uint32_t epx_peer = mapa_shared(smem_u32(&bars->epi_x), peer);
    const int send0 = (int)peer * dh;      // output columns the peer stores
    const uint32_t x_local = smem_u32(sX);
    int T = 0;
    uint32_t xpar = 0;                       // parity of each peer buffer's next release
    bool ok = true;
    PItem it;
    if (warp == 2 && lane == 0)            // item 0's partial output from the peer
      mbar_arrive_expect_tx(&bars->epi_x, epi_x_bytes(dh));
    for (int r = 0; ok; ++r) {
      const bool have = pair_item(a, r, it);
      // ---- boundary before item r: the previous item's output ----
      if (r > 0) {
        float v[4][16];                    // dh <= 64 columns of my row
        if (!(ok = warp_wait(&bars->epi_done, (r - 1) & 1, 93, abort_flag))) break;
        tc_fence_after();
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          if (c4 * 16 < dh) tmem_ld16(tmem + lane_base + kTmemS + send0 + c4 * 16, v[c4]);
        tmem_wait_ld();
        // the peer's half: fp16 rows scaled by a power of two (the row's largest
        // magnitude in [2^14, 2^15)) into the peer's buffer (T+2)%4, the inverse
        // factors into (T+3)%4
        const int xa = (T + 2) & 3, xf = (T + 3) & 3;
        if (!(ok = warp_wait<true>(&bars->x_empty[xa], (xpar >> xa) & 1u, 94, abort_flag) &&
                   warp_wait<true>(&bars->x_empty[xf], (xpar >> xf) & 1u, 94, abort_flag)))
          break;
        xpar ^= (1u << xa) | (1u << xf);
        {
          const uint32_t xo = x_peer0 + (uint32_t)xa * kXBytes;
          const uint32_t xs = x_peer0 + (uint32_t)xf * kXBytes;
          float mx = 0.f;
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
            for (int e = 0; e < 16; ++e)
              if (c4 * 16 < dh) mx = fmaxf(mx, fabsf(v[c4][e]));
          const int ex = (int)((__float_as_uint(mx) >> 23) & 0xffu);
          const uint32_t sb = (uint32_t)min(max(268 - ex, 1), 253);
          const float sc = __uint_as_float(sb << 23);
          const float inv_sc = __uint_as_float((254u - sb) << 23);
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4)
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (c4 * 16 < dh) {
                const float* w = &v[c4][8 * h];
                st_async_v4u(xo + xrow_offset(rr, (uint32_t)(2 * c4 + h), 128u),
                             pack_half2(w[0] * sc, w[1] * sc), pack_half2(w[2] * sc, w[3] * sc),
                             pack_half2(w[4] * sc, w[5] * sc), pack_half2(w[6] * sc, w[7] * sc),
                             epx_peer);
              }
          st_async_v4u(xs + rr * 16, __float_as_uint(inv_sc), 0u, 0u, 0u, epx_peer);
        }
        // my half, then item r's S may overwrite the output columns
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          if (c4 * 16 < dh)
            tmem_ld16(tmem + lane_base + kTmemS + (int)crank * dh + c4 * 16, v[c4]);
        tmem_wait_ld();
        tc_fence_before();
        if (have) mbar_arrive(&bars->q_ready);
        // plus the peer's partial product for my half (fp16 rows times 2^k)
        if (!(ok = warp_wait<true>(&bars->epi_x, (r - 1) & 1, 101, abort_flag))) break;
        {
          const uint32_t xo = x_local + (uint32_t)((T + 2) & 3) * kXBytes;
          const uint32_t xs = x_local + (uint32_t)((T + 3) & 3) * kXBytes;
          float inv_sc, y0, y1, y2;
          ld_shared_v4f(xs + rr * 16, inv_sc, y0, y1, y2);
#pragma unroll
          for (int q = 0; q < 8; ++q) {          // 8 fp16 per 16-byte chunk
            if (q * 8 < dh) {
              float x[4];
              ld_shared_v4f(xo + xrow_offset(rr, (uint32_t)q, 128u), x[0], x[1], x[2], x[3]);
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float2 f = unpack_half2(__float_as_uint(x[e]));
                v[q >> 1][8 * (q & 1) + 2 * e] += f.x * inv_sc;
                v[q >> 1][8 * (q & 1) + 2 * e + 1] += f.y * inv_sc;
              }
            }
            if (q == 3) asm volatile("" ::: "memory");   // two halves: fewer loads in flight
          }
        }
        if (have && warp == 2 && lane == 0)  // item r's partial output comes next
          mbar_arrive_expect_tx(&bars->epi_x, epi_x_bytes(dh));
        __syncwarp();
        if (have && lane < 2) {              // the partial-output buffers are free
          mbar_arrive(&bars->x_consumed[(T + 2) & 3]);
          mbar_arrive(&bars->x_consumed[(T + 3) & 3]);
        }
        // out[b, i, h, crank*dh ..+dh) by tile stores of 128 x 128-byte boxes staged
        // (128-byte swizzle) in the P buffers, free between the item's last O MMA and
        // the next item's first P; the map is per batch entry, so the rows of a
        // partial block past the sequence's end are not written.  (bf16 with d = 64
        // stores 64 bytes per row: row by row.)
        PItem prev;
        pair_item(a, r - 1, prev);
        constexpr bool kBoxesFit = dh % 64 == 0;   // both dtypes' boxes tile the columns
        if (kBoxesFit || !a.out_bf16) {
          const uint32_t stg = smem_u32(smem + kOffP);
          const uint32_t row = stg + rr * 128, sw = rr & 7;
          if (a.out_bf16) {
#pragma unroll
            for (int q = 0; q < dh / 8; ++q) {
              const float* w = &v[q >> 1][8 * (q & 1)];
              st_shared_v4(row + (uint32_t)(q >> 3) * (kRows * 128) + ((((uint32_t)q & 7u) ^ sw) << 4),
                           pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]),
                           pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7]));
            }
          } else {
#pragma unroll
            for (int q = 0; q < dh / 4; ++q) {
              const float* w = &v[q >> 2][4 * (q & 3)];
              st_shared_v4(row + (uint32_t)(q >> 3) * (kRows * 128) + ((((uint32_t)q & 7u) ^ sw) << 4),
                           __float_as_uint(w[0]), __float_as_uint(w[1]), __float_as_uint(w[2]),
                           __float_as_uint(w[3]));
            }
          }
          fence_proxy_async_smem();
          named_bar_sync(6, 128);                  // all four warps have staged their rows
          if (warp == 2 && lane == 0) {
            const int box_cols = a.out_bf16 ? 64 : 32;
            for (int bx = 0; bx < dh / box_cols; ++bx)
              tma_store_4d(&mapO, stg + (uint32_t)bx * (kRows * 128),
                           (int)crank * dh + bx * box_cols, prev.head, prev.row0, prev.b);
            bulk_commit_group();
            bulk_wait_read_all();                  // the staging must outlive the reads
          }
        } else if (prev.row0 + (int)rr < a.Tq) {
          const int64_t orow =
              (((int64_t)prev.b * a.Tq + prev.row0 + (int)rr) * a.H + prev.head) * kD +
              (int)crank * dh;
          uint4* d4 = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + orow);
#pragma unroll
          for (int q = 0; q < dh / 8; ++q) {
            const float* w = &v[q >> 1][8 * (q & 1)];
            d4[q] = make_uint4(pack_bf16x2(w[0], w[1]), pack_bf16x2(w[2], w[3]),
                               pack_bf16x2(w[4], w[5]), pack_bf16x2(w[6], w[7]));
          }
        }
        if (warp == 2 && lane == 0) mbar_arrive(&bars->stg_free);
      } else {
        tc_fence_before();
        mbar_arrive(&bars->q_ready);
      }
      if (!have) break;
      // ---- the item's tiles: my partial S (fp16) into the peer's buffer g%4 ----
      for (int j = 0; j < it.nt; ++j) {
        const int g = T + j, bi = g & 1, k = g >> 1, xb = g & 3;
        if (!warp_wait<true>(&bars->x_empty[xb], (xpar >> xb) & 1u, 95, abort_flag) ||
            !warp_wait(&bars->s_full[bi], k & 1, 96, abort_flag)) {
          ok = false;
          break;
        }
        xpar ^= 1u << xb;
        tc_fence_after();
        const uint32_t dst = x_peer0 + xb * kXBytes;
        const uint32_t bar = xfull_peer0 + xb * 8;
        float s2[2][32];
        tmem_ld32(tmem + lane_base + kTmemS + bi * kKeys, s2[0]);
        tmem_ld32(tmem + lane_base + kTmemS + bi * kKeys + 32, s2[1]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_empty[bi]);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_async_v4u(dst + sw128_offset(rr, hh * 4 + c),
                         pack_half2(s2[hh][8 * c], s2[hh][8 * c + 1]),
                         pack_half2(s2[hh][8 * c + 2], s2[hh][8 * c + 3]),
                         pack_half2(s2[hh][8 * c + 4], s2[hh][8 * c + 5]),
                         pack_half2(s2[hh][8 * c + 6], s2[hh][8 * c + 7]), bar);
      }
      if (ok) mbar_arrive(&bars->epi_a);     // the item's S columns may be overwritten
      T += it.nt;
    }
  } else if (warp == 14) {
    // ======================= releases and q tiles =======================
    // Consumption events of item r, in order, at positions p = -4..nt-1 of
    // buffer (T+p)%4: p = -4, -3 the absorption has read the item's q tile;
    // p = -2, -1 the previous item's partial output has been stored (item 0:
    // the initial release); p >= 0 tile T+p.  Each is forwarded to the peer,
    // except the last uses of the next item's q buffers (p = nt-4, nt-3).
    cluster_wait();
    if (lane == 0) {
      prefetch_tensormap(&mapQ);
      const uint32_t xe_peer0 = mapa_shared(smem_u32(&bars->x_empty[0]), peer);
      // the q tile of an item starting at global tile t0 into buffers t0%4, (t0+1)%4
      auto load_q = [&](const PItem& q_it, int t0) {
        mbar_arrive_expect_tx(&bars->pro_full, (uint32_t)(kRows * kD * 2));
        for (int kc = 0; kc < dch; ++kc)
          tma_load_3d(sX + ((t0 + kc) & 3) * kXBytes, &mapQ, &bars->pro_full, 64 * kc, q_it.head,
                      q_it.b * a.Tq + q_it.row0);
      };
      bool ok = true;
      uint32_t cpar = 0;                   // parity of each buffer's next consumption
      PItem it, nx;
      int T = 0, armed = -1;
      if (pair_item(a, 0, it)) {
        load_q(it, 0);
        armed = 0;
      }
      for (int r = 0; ok && pair_item(a, r, it); ++r) {
        const bool have_next = pair_item(a, r + 1, nx);
        for (int p = -4; p < it.nt; ++p) {
          const int xb = (T + p) & 3;
          if (!(ok = mbar_wait(&bars->x_consumed[xb], (cpar >> xb) & 1u, 97, abort_flag))) break;
          cpar ^= 1u << xb;
          if (!(have_next && (p == it.nt - 4 || p == it.nt - 3)))
            mbar_arrive_remote(xe_peer0 + (uint32_t)xb * 8);
          if (have_next && p == it.nt - 3) {   // both of the next q buffers are free
            load_q(nx, T + it.nt);
            armed = r + 1;
          }
        }
        T += it.nt;
      }
      if (!ok && armed >= 0) mbar_wait(&bars->pro_full, armed & 1, 98, nullptr);
    }
  } else if (warp >= 6) {
    // ======================= softmax, normalisation, q' conversion =======================
    const int qd = warp & 3;
    const int half = (warp - 6) >> 2;
    const int r_ = qd * 32 + lane;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t x_local = smem_u32(sX);
    const uint32_t red_mine = smem_u32(smem + kOffRed) + (uint32_t)(half * 128 + r_) * 4;
    const uint32_t red_other = red_mine ^ (128u * 4u);      // the partner warp's slot
    const uint32_t bar_id = 1u + (uint32_t)qd;
    const int oc0 = half * (RC / 2);
    if (warp == 6 && lane == 0)            // receive barriers of the first four tiles
      for (int xb = 0; xb < kXBuf; ++xb)
        mbar_arrive_expect_tx(&bars->x_full[xb], (uint32_t)kXBytes);
    __syncwarp();
    if (lane == 0) {                       // initial release of buffers 2 and 3 (0 and 1
      mbar_arrive(&bars->x_consumed[2]);   // hold item 0's q tile)
      mbar_arrive(&bars->x_consumed[3]);
    }
    int T = 0;
    bool ok = true;
    PItem it;
    for (int r = 0; ok && pair_item(a, r, it); ++r) {
      // ---- item r's q' (fp32 in O's columns, scaled by scale*log2 e) -> bf16 in TMEM ----
      if (!(ok = warp_wait(&bars->pro_done, r & 1, 99, abort_flag))) break;
      tc_fence_after();
      tmem_rows_to_bf16(tmem + lane_base + kTmemO + oc0, tmem + lane_base + kTmemQ + oc0 / 2,
                        RC / 2, a.qscale);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->q_ready);
      __syncwarp();
      if (lane == 0) {                       // the absorption has read the q buffers
        mbar_arrive(&bars->x_consumed[T & 3]);
        mbar_arrive(&bars->x_consumed[(T + 1) & 3]);
      }
      // ---- the item's tiles ----
      // keys visible to my row: key < lim (none for a row past the end)
      const int grow = it.row0 + r_;
      const int lim = grow >= a.Tq ? 0 : a.causal ? min(a.Tkv - a.Tq + grow + 1, a.Tkv) : a.Tkv;
      const int key_base = half * 32 - T * kKeys;     // key0 of tile g = g * 64 + key_base
      const int g_end = T + it.nt;
      float m_run = -INFINITY, l_half = 0.f;
      for (int g = T; g < g_end; ++g) {
        const int bi = g & 1, k = g >> 1, xb = g & 3;
        float s[32];
        if (!(ok = warp_wait(&bars->s_full[bi], k & 1, 102, abort_flag))) break;
        tc_fence_after();
        tmem_ld32(tmem + lane_base + kTmemS + bi * kKeys + half * 32, s);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(&bars->s_empty[bi]);
        // the peer's partial S over its half of the rank (my 32 keys)
        if (!(ok = warp_wait<true>(&bars->x_full[xb], (g >> 2) & 1, 103, abort_flag))) break;
        const uint32_t src = x_local + xb * kXBytes;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t u0, u1, u2, u3;
          asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                       : "=r"(u0), "=r"(u1), "=r"(u2), "=r"(u3)
                       : "r"(src + sw128_offset((uint32_t)r_, (uint32_t)(half * 4 + c)))
                       : "memory");
          const float2 f[4] = {unpack_half2(u0), unpack_half2(u1), unpack_half2(u2),
                               unpack_half2(u3)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 t = __fadd2_rn(make_float2(s[8 * c + 2 * e], s[8 * c + 2 * e + 1]), f[e]);
            s[8 * c + 2 * e] = t.x;
            s[8 * c + 2 * e + 1] = t.y;
          }
        }

        const int key0 = g * kKeys + key_base;
        if (key0 + 32 > lim) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (key0 + c >= lim) s[c] = -INFINITY;
        }
        const float mx_half = tree_max32(s);
        st_shared_f32(red_mine, mx_half);
        named_bar_sync(bar_id, 64);
        const float mx = fmaxf(mx_half, ld_shared_f32(red_other));
        named_bar_sync(bar_id, 64);
        const float m_new = fmaxf(m_run, mx);
        const bool grow_max = m_new > m_run + kRescaleThreshold;
        const float m_ref = grow_max ? m_new : m_run;
        const float alpha = grow_max ? ex2(m_run - m_new) : 1.f;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float2 t = __fadd2_rn(make_float2(s[2 * c], s[2 * c + 1]),
                                      make_float2(-m_use, -m_use));
          s[2 * c] = ex2(t.x);
          s[2 * c + 1] = ex2(t.y);
        }
        l_half = l_half * alpha + tree_sum32(s);
        m_run = m_ref;
        if (!(ok = warp_wait(&bars->p_empty[bi], (k & 1) ^ 1, 104, abort_flag))) break;
        if (__any_sync(0xffffffffu, grow_max && g > T)) {
          if (!(ok = warp_wait(&bars->p_empty[(g - 1) & 1], ((g - 1) >> 1) & 1, 105, abort_flag)))
            break;
          tc_fence_after();
          for (int c = oc0; c < oc0 + RC / 2; c += 16) {
            float o[16];
            tmem_ld16(tmem + lane_base + kTmemO + c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float2 t = __fmul2_rn(make_float2(o[2 * e], o[2 * e + 1]),
                                          make_float2(alpha, alpha));
              o[2 * e] = t.x;
              o[2 * e + 1] = t.y;
            }
            tmem_st16(tmem + lane_base + kTmemO + c, o);
          }
          tmem_wait_st();
        }
        // the previous item's output staging has been read out of the P buffers
        if (g == T && r > 0 &&
            !(ok = warp_wait(&bars->stg_free, (r - 1) & 1, 107, abort_flag)))
          break;
        const uint32_t pb = smem_u32(smem + kOffP + bi * kPBytes);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          st_shared_v4(pb + sw128_offset(r_, half * 4 + c), pack_bf16x2(s[8 * c], s[8 * c + 1]),
                       pack_bf16x2(s[8 * c + 2], s[8 * c + 3]),
                       pack_bf16x2(s[8 * c + 4], s[8 * c + 5]),
                       pack_bf16x2(s[8 * c + 6], s[8 * c + 7]));
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full[bi]);
        // the receive buffer is released off the softmax chain: the peer writes it
        // again only four tiles later
        if (warp == 6 && lane == 0)          // this buffer's next tile
          mbar_arrive_expect_tx(&bars->x_full[xb], (uint32_t)kXBytes);
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->x_consumed[xb]);
      }
      if (!ok) break;

      // ---- end of the item: normalised O_lat (bf16) into q''s columns ----
      // the row sum is the two halves' sums, added in the same order in both warps
      st_shared_f32(red_mine, l_half);
      named_bar_sync(bar_id, 64);
      const float l_lo = ld_shared_f32(half ? red_other : red_mine);
      const float l_hi = ld_shared_f32(half ? red_mine : red_other);
      const float l_run = l_lo + l_hi;
      named_bar_sync(bar_id, 64);
      if (!(ok = warp_wait(&bars->o_last, r & 1, 106, abort_flag))) break;
      tc_fence_after();
      const float inv = (l_run > 0.f) ? 1.f / l_run : 0.f;
      tmem_rows_to_bf16(tmem + lane_base + kTmemO + oc0, tmem + lane_base + kTmemQ + oc0 / 2,
                        RC / 2, inv);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->epi_a);
      T += it.nt;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, 512);
  if (!touches_peer) cluster_wait();
  cluster_sync();     // neither CTA leaves while the other may still address it
}

// ---------------------------------------------------------------------------
// Split-KV merge: out[r,:] = sum_p 2^(m_p - M) o_p[r,:] / sum_p 2^(m_p - M) l_p
// (page "Kimi-K2.6 l2_p29", online softmax, applied to whole partitions).
// One block of width/4 threads per row, float4 per thread.
// ---------------------------------------------------------------------------
__global__ void merge_partials_kernel(const float* __restrict__ ml, int ml_stride,
                                      const float* __restrict__ lsep,
                                      const float* __restrict__ o, void* __restrict__ out,
                                      int parts, int rows, int width, int out_bf16) {
  const int row = blockIdx.x;
  if (row >= rows) return;
  // m of part p at ml[(p*rows + row)*ml_stride]; l at +1 (or lsep[p*rows+row]).
  float M = -INFINITY;
  for (int p = 0; p < parts; ++p) M = fmaxf(M, ml[((int64_t)p * rows + row) * ml_stride]);
  float lsum = 0.f;
  for (int p = 0; p < parts; ++p) {
    const float mp = ml[((int64_t)p * rows + row) * ml_stride];
    const float lp = lsep ? lsep[(int64_t)p * rows + row]
                          : ml[((int64_t)p * rows + row) * ml_stride + 1];
    if (mp != -INFINITY) lsum += ex2(mp - M) * lp;
  }
  const float inv = (lsum > 0.f) ? 1.f / lsum : 0.f;
  for (int c = threadIdx.x * 4; c < width; c += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p = 0; p < parts; ++p) {
      const float mp = ml[((int64_t)p * rows + row) * ml_stride];
      if (mp == -INFINITY) continue;
      const float w = ex2(mp - M);
      const float4 v = *reinterpret_cast<const float4*>(o + ((int64_t)p * rows + row) * width + c);
      acc.x = fmaf(w, v.x, acc.x);
      acc.y = fmaf(w, v.y, acc.y);
      acc.z = fmaf(w, v.z, acc.z);
      acc.w = fmaf(w, v.w, acc.w);
    }
    if (out_bf16) {
      uint2 pk = make_uint2(pack_bf16x2(acc.x * inv, acc.y * inv),
                            pack_bf16x2(acc.z * inv, acc.w * inv));
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(out) + (int64_t)row * width + c) = pk;
    } else {
      *reinterpret_cast<float4*>(static_cast<float*>(out) + (int64_t)row * width + c) =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    }
  }
}

// Bounded-wait check: one thread waits on an mbarrier that nothing arrives on,
// with a caller-chosen limit, records kErrWaitTimeout | 0x7f and returns -- the
// same path every wait in the kernels above takes when it runs out of time.
__global__ void wait_timeout_probe_kernel(unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_mbarrier_init_cluster();
  const uint32_t a = smem_u32(&bar);
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(a, 0)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      report_error(kErrWaitTimeout | 0x7fu);
      return;
    }
  }
}

}  // namespace

cudaError_t launch_wait_timeout_probe(unsigned long long limit_ns, cudaStream_t stream) {
  wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

template <int kRC, int kMode>
static cudaError_t launch_flash_rc(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                                  const CUtensorMap& mapWk, const CUtensorMap& mapWv,
                                  const CUtensorMap& mapO, const FlashArgs& args,
                                  cudaStream_t stream) {
  auto kern = flash_packed_kernel<kRC, kMode>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  const int csize = args.pair ? 2 : 1;
  const int per_rb = kMode != kModePacked ? args.B * args.H : args.B * args.splits;
  const unsigned blocks = (unsigned)(args.row_blocks * per_rb * csize);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = csize;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, mapQ, mapL, mapWk, mapWv, mapO, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_flash_packed(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                                const FlashArgs& args, cudaStream_t stream) {
  switch (args.RC) {
    case 64: return launch_flash_rc<64, kModePacked>(mapQ, mapL, mapQ, mapQ, mapQ, args, stream);
    case 128: return launch_flash_rc<128, kModePacked>(mapQ, mapL, mapQ, mapQ, mapQ, args, stream);
    case 192: return launch_flash_rc<192, kModePacked>(mapQ, mapL, mapQ, mapQ, mapQ, args, stream);
    case 256: return launch_flash_rc<256, kModePacked>(mapQ, mapL, mapQ, mapQ, mapQ, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_flash_fused(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                               const CUtensorMap& mapWk, const CUtensorMap& mapWv,
                               const CUtensorMap& mapO, const FlashArgs& args,
                               cudaStream_t stream) {
  switch (args.RC) {
    case 64:
      return launch_flash_rc<64, kModeFused>(mapQ, mapL, mapWk, mapWv, mapO, args, stream);
    case 128:
      return launch_flash_rc<128, kModeFused>(mapQ, mapL, mapWk, mapWv, mapO, args, stream);
    case 192:
      return launch_flash_rc<192, kModeFused>(mapQ, mapL, mapWk, mapWv, mapO, args, stream);
    case 256:
      return launch_flash_rc<256, kModeFused>(mapQ, mapL, mapWk, mapWv, mapO, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

template <int kRC>
static cudaError_t launch_persistent_rc(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                                        const CUtensorMap& mapWk, const CUtensorMap& mapWv,
                                        const CUtensorMap& mapO, const FlashArgs& args,
                                        int num_ctas, cudaStream_t stream) {
  auto kern = flash_persistent_kernel<kRC>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)num_ctas, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, mapQ, mapL, mapWk, mapWv, mapO, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_flash_persistent(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                                    const CUtensorMap& mapWk, const CUtensorMap& mapWv,
                                    const CUtensorMap& mapO, const FlashArgs& args, int num_ctas,
                                    cudaStream_t stream) {
  if (args.pair || args.d != 64 || args.cu_q != nullptr || num_ctas <= 0)
    return cudaErrorInvalidValue;
  switch (args.RC) {
    case 64: return launch_persistent_rc<64>(mapQ, mapL, mapWk, mapWv, mapO, args, num_ctas, stream);
    case 128: return launch_persistent_rc<128>(mapQ, mapL, mapWk, mapWv, mapO, args, num_ctas, stream);
    case 192: return launch_persistent_rc<192>(mapQ, mapL, mapWk, mapWv, mapO, args, num_ctas, stream);
    case 256: return launch_persistent_rc<256>(mapQ, mapL, mapWk, mapWv, mapO, args, num_ctas, stream);
    default: return cudaErrorInvalidValue;
  }
}

static cudaLaunchConfig_t pair_config(int pairs, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

// CTA pairs of the persistent pair kernel that fit on the current device at
// once (a cluster needs two free SMs of one GPC), 0 if the query fails.
template <int kRC, int kD>
static int pair_slots_rc() {
  auto kern = flash_persistent_pair_kernel<kRC, kD>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config(1, nullptr, attr);
  int clusters = 0;
  if (cudaOccupancyMaxActiveClusters(&clusters, kern, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return clusters;
}

int flash_pair_slots(int RC, int d) {
  constexpr int kDevices = 64;
  static std::atomic<int> cache[4][kDevices];   // 0: not yet queried, else slots + 1
  if ((RC != 192 && RC != 256) || (d != 64 && d != 128)) return 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevices) {
    cudaGetLastError();
    return 0;
  }
  const int k = (RC == 256 ? 2 : 0) + (d == 128 ? 1 : 0);
  std::atomic<int>& c = cache[k][dev];
  int v = c.load(std::memory_order_relaxed);
  if (v == 0) {
    switch (k) {
      case 0: v = pair_slots_rc<192, 64>(); break;
      case 1: v = pair_slots_rc<192, 128>(); break;
      case 2: v = pair_slots_rc<256, 64>(); break;
      default: v = pair_slots_rc<256, 128>(); break;
    }
    c.store(v + 1, std::memory_order_relaxed);
    return v;
  }
  return v - 1;
}

template <int kRC, int kD>
static cudaError_t launch_persistent_pair_rc(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                                             const CUtensorMap& mapWk, const CUtensorMap& mapWv,
                                             const CUtensorMap& mapO, const FlashArgs& args,
                                             int pairs, cudaStream_t stream) {
  auto kern = flash_persistent_pair_kernel<kRC, kD>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  const cudaLaunchConfig_t cfg = pair_config(pairs, stream, attr);
  e = cudaLaunchKernelEx(&cfg, kern, mapQ, mapL, mapWk, mapWv, mapO, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_flash_persistent_pair(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                                         const CUtensorMap& mapWk, const CUtensorMap& mapWv,
                                         const CUtensorMap& mapO, const FlashArgs& args,
                                         int pairs, cudaStream_t stream) {
  if (!args.pair || args.cu_q != nullptr || pairs <= 0) return cudaErrorInvalidValue;
  const int k = (args.RC == 256 ? 2 : args.RC == 192 ? 0 : -8) + (args.d == 128 ? 1 : args.d == 64 ? 0 : -8);
  switch (k) {
    case 0: return launch_persistent_pair_rc<192, 64>(mapQ, mapL, mapWk, mapWv, mapO, args, pairs, stream);
    case 1: return launch_persistent_pair_rc<192, 128>(mapQ, mapL, mapWk, mapWv, mapO, args, pairs, stream);
    case 2: return launch_persistent_pair_rc<256, 64>(mapQ, mapL, mapWk, mapWv, mapO, args, pairs, stream);
    case 3: return launch_persistent_pair_rc<256, 128>(mapQ, mapL, mapWk, mapWv, mapO, args, pairs, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_flash_explicit(const CUtensorMap& mapQ, const CUtensorMap& mapK,
                                  const CUtensorMap& mapV, const FlashArgs& args,
                                  cudaStream_t stream) {
  switch (args.RC) {
    case 64:
      return launch_flash_rc<64, kModeExplicit>(mapQ, mapK, mapV, mapV, mapQ, args, stream);
    case 128:
      return launch_flash_rc<128, kModeExplicit>(mapQ, mapK, mapV, mapV, mapQ, args, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t flash_read_device_error(unsigned int* code, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(unsigned int));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
  }
  return e;
}

cudaError_t launch_merge_partials(const float* ml, int ml_stride, const float* l, const float* o,
                                  void* out, int parts, int rows, int width, int out_bf16,
                                  cudaStream_t stream) {
  const int threads = min(256, max(32, ((width / 4 + 31) / 32) * 32));
  merge_partials_kernel<<<rows, threads, 0, stream>>>(ml, ml_stride, l, o, out, parts, rows,
                                                      width, out_bf16);
  return cudaGetLastError();
}

}  // namespace mla
