// Tensor-core GEMM for sm_103a: TMA-staged 128-byte-swizzled tiles, tcgen05.mma
// (kind::f16, bf16 inputs, fp32 accumulate) into tensor memory, tcgen05.ld
// epilogue.  One CTA computes one 128 x BN tile of one group.
//
// It serves three steps of the path, all plain contractions:
//   - the down-projection latent = hidden @ w_down (page "FW-GLM-5-1 l2_p1",
//     problem statement) and the optional k / v up-projections;
//   - the query absorption q'[., h, :] = w_up_k[:, h, :] q[., h, :] (one group
//     per head);
//   - the value up-projection out[., h, :] = o_lat[., h, :] @ w_up_v[:, h, :].
//
// Warp roles (128 threads): warp 0 lane 0 issues TMA loads into a 4-stage
// ring, warp 1 owns the tensor memory and its lane 0 issues the MMAs; all four
// warps then drain the accumulator (warp w reads TMEM lanes 32w..32w+31).
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "ptx.cuh"

namespace mla {

namespace {

constexpr int kBM = 128, kBK = 64, kThreads = 128;
constexpr int kAStage = kBM * kBK * 2;      // 16 KB

// Tile shapes: BN <= 256 with a 4-stage ring, or BN = 512 (two N = 256 MMAs per
// K-step into all 512 TMEM columns) with 2 stages, for narrow-M contractions
// whose whole N fits one CTA (one wave of CTAs instead of two).
template <bool kWide>
struct GemmShape {
  static constexpr int kStages = kWide ? 2 : 4;
  static constexpr int kBNMax = kWide ? 512 : 256;
  static constexpr int kBStage = kBNMax * kBK * 2;   // 64 or 32 KB
  static constexpr int kTmemCols = kWide ? 512 : 256;
  static constexpr int kSmemBytes = kStages * (kAStage + kBStage) + 256 + 1024;
};

template <bool kBMN, bool kWide>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                   const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapC, int c_tile_store, GemmArgs g) {
  constexpr int kStages = GemmShape<kWide>::kStages;
  constexpr int kBStage = GemmShape<kWide>::kBStage;
  constexpr int kTmemCols = GemmShape<kWide>::kTmemCols;
  static_assert(!(kWide && kBMN), "BN = 512 is for K-major B");
  extern __shared__ uint8_t gemm_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kAStage;
  uint64_t* full = reinterpret_cast<uint64_t*>(sB + kStages * kBStage);
  uint64_t* empty = full + kStages;
  uint64_t* accum = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  grid_dep_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int BN = g.BN;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * kBM, grp = blockIdx.z;
  const int kblocks = g.K / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    *abort_flag = 0;
    fence_mbarrier_init_cluster();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  grid_dep_wait();        // set-up above overlaps the previous kernel's tail

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer ----------------
    prefetch_tensormap(&mapA);
    prefetch_tensormap(&mapB);
    const uint32_t bytes = (uint32_t)(kAStage + BN * kBK * 2);
    int issued = 0;
    for (int kb = 0; kb < kblocks; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait(&empty[s], ((kb / kStages) & 1) ^ 1, 1, abort_flag)) break;
      ++issued;
      mbar_arrive_expect_tx(&full[s], bytes);
      tma_load_3d(sA + s * kAStage, &mapA, &full[s], kb * kBK, grp, m0);
      if (kWide) {                       // two boxes of 256 rows of B
        tma_load_3d(sB + s * kBStage, &mapB, &full[s], kb * kBK, grp, n0);
        tma_load_3d(sB + s * kBStage + 256 * 128, &mapB, &full[s], kb * kBK, grp, n0 + 256);
      } else if (!kBMN) {
        tma_load_3d(sB + s * kBStage, &mapB, &full[s], kb * kBK, grp, n0);
      } else {
        for (int c = 0; c < BN / 64; ++c)
          tma_load_3d(sB + s * kBStage + c * (kBK * 128), &mapB, &full[s], n0 + 64 * c, grp,
                      kb * kBK);
      }
    }
    // Do not leave copies in flight: wait for the last load of each stage.
    for (int kb = (issued > kStages ? issued - kStages : 0); kb < issued; ++kb)
      mbar_wait(&full[kb % kStages], (kb / kStages) & 1, 4, nullptr);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc = make_idesc_bf16(kBM, kWide ? 256 : BN, false, kBMN);
    bool ok = true;
    for (int kb = 0; kb < kblocks && ok; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait(&full[s], (kb / kStages) & 1, 2, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const uint32_t a0 = smem_u32(sA + s * kAStage);
      const uint32_t b0 = smem_u32(sB + s * kBStage);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t ad = make_sdesc_sw128(a0 + kk * 32, 16, 1024);
        const uint64_t bd = kBMN ? make_sdesc_sw128(b0 + kk * 2048, kBK * 128, 1024)
                                 : make_sdesc_sw128(b0 + kk * 32, 16, 1024);
        umma_bf16(tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
        if (kWide)                       // columns 256..511: B rows 256..511
          umma_bf16(tmem + 256, ad, bd + (uint64_t)((256 * 128) >> 4), idesc,
                    (kb | kk) != 0 ? 1u : 0u);
      }
      umma_commit(&empty[s]);
    }
    umma_commit(accum);
  }
  __syncwarp();

  // ---------------- epilogue: TMEM -> registers -> global ----------------
  // With c_tile_store the 128 x BN tile is staged in the (now idle) operand
  // stages as 128-byte-swizzled boxes of 128 rows x 128 bytes and leaves by TMA
  // tile stores (rows past M are clipped by the map); otherwise each thread
  // writes its own row.
  const bool ok = mbar_wait(accum, 0, 3, abort_flag);
  __syncwarp();
  tc_fence_after();
  const uint32_t stage0 = smem_u32(smem);
  if (ok) {
    const int r = warp * 32 + lane;
    const int row = m0 + r;
    const bool valid = row < g.M;
    const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16);
    // two 32-column loads in flight per wait (BN is a multiple of 64)
    for (int c2 = 0; c2 < BN / 32; c2 += 2) {
      float vv[2][32];
      tmem_ld32(tbase + c2 * 32, vv[0]);
      tmem_ld32(tbase + c2 * 32 + 32, vv[1]);
      tmem_wait_ld();
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int c = c2 + h2;
        const float (&v)[32] = vv[h2];
        if (c_tile_store) {
          if (g.c_bf16) {           // 32 columns = half a box row
            const uint32_t box = stage0 + (uint32_t)(c >> 1) * (kBM * 128);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              st_shared_v4(box + sw128_offset((uint32_t)r, (uint32_t)((c & 1) * 4 + q)),
                           pack_bf16x2(v[8 * q] * g.alpha, v[8 * q + 1] * g.alpha),
                           pack_bf16x2(v[8 * q + 2] * g.alpha, v[8 * q + 3] * g.alpha),
                           pack_bf16x2(v[8 * q + 4] * g.alpha, v[8 * q + 5] * g.alpha),
                           pack_bf16x2(v[8 * q + 6] * g.alpha, v[8 * q + 7] * g.alpha));
          } else {                  // 32 columns = one box row
            const uint32_t box = stage0 + (uint32_t)c * (kBM * 128);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_shared_v4(box + sw128_offset((uint32_t)r, (uint32_t)q),
                           __float_as_uint(v[4 * q] * g.alpha),
                           __float_as_uint(v[4 * q + 1] * g.alpha),
                           __float_as_uint(v[4 * q + 2] * g.alpha),
                           __float_as_uint(v[4 * q + 3] * g.alpha));
          }
        } else if (valid) {
          const int64_t off = (int64_t)grp * g.c_gs + (int64_t)row * g.c_rs + n0 + c * 32;
          if (g.c_bf16) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(g.C) + off);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              dst[q] = make_uint4(pack_bf16x2(v[8 * q] * g.alpha, v[8 * q + 1] * g.alpha),
                                  pack_bf16x2(v[8 * q + 2] * g.alpha, v[8 * q + 3] * g.alpha),
                                  pack_bf16x2(v[8 * q + 4] * g.alpha, v[8 * q + 5] * g.alpha),
                                  pack_bf16x2(v[8 * q + 6] * g.alpha, v[8 * q + 7] * g.alpha));
          } else {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(g.C) + off);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(v[4 * q] * g.alpha, v[4 * q + 1] * g.alpha,
                                   v[4 * q + 2] * g.alpha, v[4 * q + 3] * g.alpha);
          }
        }
      }
    }
  }
  if (c_tile_store) {
    fence_proxy_async_smem();
    __syncthreads();
    if (ok && threadIdx.x == 0) {
      const int box_cols = g.c_bf16 ? 64 : 32;
      for (int bx = 0; bx < BN / box_cols; ++bx)
        tma_store_3d(&mapC, stage0 + (uint32_t)bx * (kBM * 128), n0 + bx * box_cols, m0, grp);
      bulk_commit_group();
      bulk_wait_read_all();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t gemm_read_device_error(unsigned int* code, int clear) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(unsigned int));
  if (e == cudaSuccess && clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
  }
  return e;
}

template <bool kBMN, bool kWide>
static cudaError_t launch_shape(const CUtensorMap& mapA, const CUtensorMap& mapB,
                                const GemmArgs& args, cudaStream_t stream) {
  dim3 grid(args.N / args.BN, (args.M + kBM - 1) / kBM, args.G);
  auto k = gemm_tc_kernel<kBMN, kWide>;
  constexpr int smem = GemmShape<kWide>::kSmemBytes;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  // The output tile store: C as {N, M, G} with 128-byte boxes of 128 rows,
  // when the tile fits the operand stages and C's layout suits TMA; else the
  // kernel writes row by row.
  const int es = args.c_bf16 ? 2 : 4;
  const int64_t gs = args.G > 1 ? args.c_gs : (int64_t)args.M * args.c_rs;
  CUtensorMap mapC;
  constexpr int64_t kStageBytes =
      (int64_t)GemmShape<kWide>::kStages * (kAStage + GemmShape<kWide>::kBStage);
  int tile_store =
      (int64_t)kBM * args.BN * es <= kStageBytes &&
      (reinterpret_cast<uintptr_t>(args.C) & 15) == 0 && (args.c_rs * es) % 16 == 0 &&
      (gs * es) % 16 == 0 && (args.BN * es) % 128 == 0 && (args.N * es) % 16 == 0;
  if (tile_store)
    tile_store = make_tmap_3d(&mapC, args.C, es, (uint64_t)args.N, (uint64_t)args.M,
                              (uint64_t)args.G, (uint64_t)args.c_rs * es, (uint64_t)gs * es,
                              128u / es, kBM, 1, true)
                     ? 1
                     : 0;
  if (!tile_store) mapC = mapA;                 // not read
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, k, mapA, mapB, mapC, tile_store, args);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gemm_tc(const CUtensorMap& mapA, const CUtensorMap& mapB, bool b_mn_major,
                           const GemmArgs& args, cudaStream_t stream) {
  if (args.BN == 512) {
    if (b_mn_major) return cudaErrorInvalidValue;
    return launch_shape<false, true>(mapA, mapB, args, stream);
  }
  if (args.BN > 256) return cudaErrorInvalidValue;
  return b_mn_major ? launch_shape<true, false>(mapA, mapB, args, stream)
                    : launch_shape<false, false>(mapA, mapB, args, stream);
}

}  // namespace mla
