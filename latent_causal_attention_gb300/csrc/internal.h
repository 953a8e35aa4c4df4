// Internal launchers shared by the C-ABI layer (mla_abi.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

// SM count assumed when the device cannot be asked (no GPU visible to the
// host code that plans a call; a GB300 has 152).
constexpr int kDefaultNumSMs = 152;
// Largest row or position count the kernels index with 32-bit integers.
constexpr int64_t kMaxIndex = ((int64_t)1 << 31) - 1;

// ----- CUDA-core paths ------------------------------------------------------
cudaError_t launch_warp_attention(const void* q, const void* lat, const void* wk, const void* wv,
                                  void* out, int B, int Tq, int Tkv, int H, int d, int R,
                                  float scale, int causal, int in_bf16, int out_bf16,
                                  cudaStream_t stream);

cudaError_t launch_projection_cuda_core(const void* hidden, const void* w_down,
                                        const void* w_up_k, const void* w_up_v, void* latent,
                                        void* k, void* v, int64_t M, int Dm, int R, int C,
                                        int in_bf16, int out_bf16, cudaStream_t stream);

// ----- tensor-core GEMM -----------------------------------------------------
// C[g][m, n] = alpha * sum_k A[g][m, k] * B[g][k, n]   (bf16 in, fp32 accumulate)
//   A: 3-D tensor map {K, G, M}, box {64, 1, 128}, 128-byte swizzle (K-major).
//   B: K-major  -> tensor map {K, G, N}, box {64, 1, BN};
//      MN-major -> tensor map {N, G, K}, box {64, 1, 64}.
//   C: element (g, m, n) at C + g*c_gs + m*c_rs + n, fp32 or bf16.
struct GemmArgs {
  int M, N, K, G;
  int BN;            // 64, 128, 256 (divides N) or 512 (= N, K-major B, B box 256 rows)
  float alpha;
  void* C;
  int c_bf16;
  int64_t c_rs, c_gs;
};
cudaError_t launch_gemm_tc(const CUtensorMap& mapA, const CUtensorMap& mapB, bool b_mn_major,
                           const GemmArgs& args, cudaStream_t stream);

// ----- flash loop over latent tiles (head-packed rows) ----------------------
// Rows of one batch entry are (i, h) pairs, r = i*H + h, of the absorbed query
// q' (bf16, already multiplied by scale*log2 e).  Each CTA (or CTA pair,
// splitting the rank) runs 128 rows against a contiguous range of 64-key tiles.
struct FlashArgs {
  int B, Tq, Tkv, H, R;
  int RC;            // rank columns per CTA (R, or R/2 with a CTA pair)
  int pair;          // 1: cluster of two CTAs splitting the rank
  int row_blocks;    // ceil(Tq*H / 128)
  int splits;        // key-range partitions
  int causal;
  // fused prefill (rows = query positions of one head): q and the weights are
  // read directly, out (B,Tq,H,d) written; no workspace
  int d;
  float qscale;      // scale * log2(e), applied to q' before rounding to bf16
  void* out;
  int out_bf16;
  void* olat;        // splits == 1: normalised latent-space output, bf16 (B*Tq*H, R)
  float* part_o;     // splits > 1: (splits, B*Tq*H, R) unnormalised
  float* part_ml;    // splits > 1: (splits, B*Tq*H, 2) = (max in log2 units, sum)
  // variable-length batch (per-head modes only): batch entry b owns query rows
  // [cu_q[b], cu_q[b+1]) of total_q and latent rows [cu_kv[b], cu_kv[b+1]) of
  // total_kv (device int32, B+1 entries); Tq is then the longest query range.
  const int* cu_q;
  const int* cu_kv;
  int total_q, total_kv;
};
cudaError_t launch_flash_packed(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                                const FlashArgs& args, cudaStream_t stream);

// Fused prefill: q (3-D map {d, H, B*Tq}, box {64,1,128}), latent, w_up_k
// (K-major, {d, H, R}, box {64,1,RC}), w_up_v (MN-major, {d, H, R}, box {64,1,64}),
// out ({d, H, B*Tq} or {d, H, total_q}, 128-byte swizzle, box {128/elem bytes, 1,
// 128}; the tile store of full 128-row blocks).
// Explicit K/V attention: mapQ over q {d, H, B*Tq}, mapK / mapV over k, v
// {d, H, B*Tkv}; args.RC = args.d (64 or 128), no CTA pair.
cudaError_t launch_flash_explicit(const CUtensorMap& mapQ, const CUtensorMap& mapK,
                                  const CUtensorMap& mapV, const FlashArgs& args,
                                  cudaStream_t stream);
cudaError_t launch_flash_fused(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                               const CUtensorMap& mapWk, const CUtensorMap& mapWv,
                               const CUtensorMap& mapO, const FlashArgs& args,
                               cudaStream_t stream);

// Persistent single-CTA prefill (rank <= 256, d = 64, dense batch): num_ctas
// resident CTAs work through the (batch entry, head, 128-row block) items; same
// tensor maps as the fused prefill except the output map, which is 4-D
// ({d, H, Tq, B}, 128-byte swizzle, box {128 / element bytes, 1, 128, 1}) so
// that the tile stores of a partial row block stop at its sequence's end;
// results bitwise equal to launch_flash_fused's.
cudaError_t launch_flash_persistent(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                                    const CUtensorMap& mapWk, const CUtensorMap& mapWv,
                                    const CUtensorMap& mapO, const FlashArgs& args, int num_ctas,
                                    cudaStream_t stream);

// Persistent CTA-pair prefill (rank 384 or 512, d = 64 or 128, dense batch):
// `pairs` resident clusters of two CTAs (at most flash_pair_slots(RC, d)) work
// through the items; maps as launch_flash_fused except the output map, which is
// 4-D ({d, H, Tq, B}, 128-byte swizzle, box {128 / element bytes, 1, 128, 1}) so
// that the tile stores of a partial row block stop at its sequence's end;
// results bitwise equal to launch_flash_fused's.  flash_pair_slots returns how
// many such pairs fit on the current device at once (cached per device), 0
// when unknown.
int flash_pair_slots(int RC, int d);
cudaError_t launch_flash_persistent_pair(const CUtensorMap& mapQ, const CUtensorMap& mapL,
                                         const CUtensorMap& mapWk, const CUtensorMap& mapWv,
                                         const CUtensorMap& mapO, const FlashArgs& args,
                                         int pairs, cudaStream_t stream);

cudaError_t launch_merge_partials(const float* m_l, int ml_stride, const float* l, const float* o,
                                  void* out, int parts, int rows, int width, int out_bf16,
                                  cudaStream_t stream);

// Launches a kernel whose only wait can never complete, bounded by limit_ns.
cudaError_t launch_wait_timeout_probe(unsigned long long limit_ns, cudaStream_t stream);

// Device-side error words (one per translation unit with bounded waits).
cudaError_t gemm_read_device_error(unsigned int* code, int clear);
cudaError_t flash_read_device_error(unsigned int* code, int clear);

// ----- helpers ---------------------------------------------------------------
// 3-D bf16/fp32 tensor map, dims innermost first, strides in bytes for dims 1, 2.
bool make_tmap_3d(CUtensorMap* map, const void* base, int elem_bytes, uint64_t d0, uint64_t d1,
                  uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2,
                  bool swizzle128);

}  // namespace mla
