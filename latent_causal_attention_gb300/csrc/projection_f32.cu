// Fused two-stage latent projection on CUDA cores (fp32 arithmetic):
//   latent = hidden @ w_down            (stage 1, latent tile kept in smem)
//   k = latent @ w_up_k, v = latent @ w_up_v   (stage 2, read from that tile)
//
// Page "FW-GLM-5-1 l2_p1" (fused latent projection): the problem statement
// fixes the three products; its second design ("compute the latent
// cooperatively per row into shared memory, then k and v from it") is the
// structure kept here.  Its 96 KB all-weights-in-smem kernel failed to
// launch for want of the dynamic shared memory opt-in; this kernel stages
// only a K-chunk of w_down at a time and opts in explicitly.
//
// Block = 256 threads, kRows rows of hidden.  hidden is read with 128-bit
// loads when its row length allows it.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"

namespace mla {

namespace {

constexpr int kRows = 16;
constexpr int kChunk = 32;        // model_dim chunk staged per step
constexpr int kThreads = 256;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ void st_f(T* p, float v);
template <>
__device__ __forceinline__ void st_f<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

// MAXR: compile-time bound on rank (accumulators per thread = kRows*MAXR/kThreads).
template <typename TI, typename TO, int MAXR>
__global__ void __launch_bounds__(kThreads)
    projection_kernel(const TI* __restrict__ hidden, const TI* __restrict__ w_down,
                      const TI* __restrict__ w_up_k, const TI* __restrict__ w_up_v,
                      TO* __restrict__ latent, TO* __restrict__ k, TO* __restrict__ v, int64_t M,
                      int Dm, int R, int C, int vec4) {
  extern __shared__ float psmem[];
  float* s_lat = psmem;                          // kRows * R   (the latent tile)
  float* s_h = s_lat + kRows * R;                // kRows * kChunk
  float* s_w = s_h + kRows * kChunk;             // kChunk * R
  const int tid = threadIdx.x;
  const int64_t m0 = (int64_t)blockIdx.x * kRows;
  constexpr int kAcc = (kRows * MAXR + kThreads - 1) / kThreads;

  // ---- stage 1: latent tile = hidden[m0:m0+kRows] @ w_down ----
  float acc[kAcc];
#pragma unroll
  for (int a = 0; a < kAcc; ++a) acc[a] = 0.f;
  for (int j0 = 0; j0 < Dm; j0 += kChunk) {
    const int jn = min(kChunk, Dm - j0);
    // hidden chunk (kRows x jn)
    if (vec4 && jn == kChunk) {
      for (int idx = tid; idx < kRows * (kChunk / 4); idx += kThreads) {
        const int rr = idx / (kChunk / 4), c4 = idx % (kChunk / 4);
        float4 val = make_float4(0.f, 0.f, 0.f, 0.f);
        if (m0 + rr < M)
          val = __ldg(reinterpret_cast<const float4*>(
              reinterpret_cast<const float*>(hidden) + (m0 + rr) * Dm + j0) + c4);
        reinterpret_cast<float4*>(s_h + rr * kChunk)[c4] = val;
      }
    } else {
      for (int idx = tid; idx < kRows * kChunk; idx += kThreads) {
        const int rr = idx / kChunk, c = idx % kChunk;
        float val = 0.f;
        if (m0 + rr < M && c < jn) val = to_f(hidden[(m0 + rr) * Dm + j0 + c]);
        s_h[idx] = val;
      }
    }
    // w_down chunk (jn x R)
    for (int idx = tid; idx < kChunk * R; idx += kThreads) {
      const int jj = idx / R, r = idx % R;
      s_w[idx] = (jj < jn) ? to_f(w_down[(int64_t)(j0 + jj) * R + r]) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int a = 0; a < kAcc; ++a) {
      const int o = tid + a * kThreads;
      if (o < kRows * R) {
        const int rr = o / R, r = o % R;
        float sum = acc[a];
#pragma unroll 8
        for (int jj = 0; jj < kChunk; ++jj) sum = fmaf(s_h[rr * kChunk + jj], s_w[jj * R + r], sum);
        acc[a] = sum;
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int a = 0; a < kAcc; ++a) {
    const int o = tid + a * kThreads;
    if (o < kRows * R) {
      const int rr = o / R, r = o % R;
      s_lat[o] = acc[a];
      if (m0 + rr < M) st_f(latent + (m0 + rr) * R + r, acc[a]);
    }
  }
  __syncthreads();
  if (k == nullptr && v == nullptr) return;

  // ---- stage 2: k, v = latent tile @ w_up_k / w_up_v (fp32 latent) ----
  for (int c = tid; c < C; c += kThreads) {
    float ak[kRows], av[kRows];
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) { ak[rr] = 0.f; av[rr] = 0.f; }
    for (int r = 0; r < R; ++r) {
      const float wkv = k ? to_f(w_up_k[(int64_t)r * C + c]) : 0.f;
      const float wvv = v ? to_f(w_up_v[(int64_t)r * C + c]) : 0.f;
#pragma unroll
      for (int rr = 0; rr < kRows; ++rr) {
        const float lv = s_lat[rr * R + r];
        ak[rr] = fmaf(lv, wkv, ak[rr]);
        av[rr] = fmaf(lv, wvv, av[rr]);
      }
    }
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) {
      if (m0 + rr < M) {
        if (k) st_f(k + (m0 + rr) * C + c, ak[rr]);
        if (v) st_f(v + (m0 + rr) * C + c, av[rr]);
      }
    }
  }
}

template <typename TI, typename TO, int MAXR>
cudaError_t launch_typed(const void* hidden, const void* w_down, const void* w_up_k,
                         const void* w_up_v, void* latent, void* k, void* v, int64_t M, int Dm,
                         int R, int C, cudaStream_t stream) {
  const size_t smem = sizeof(float) * ((size_t)kRows * R + kRows * kChunk + (size_t)kChunk * R);
  auto kern = projection_kernel<TI, TO, MAXR>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int vec4 = (sizeof(TI) == 4) && (Dm % 4 == 0) &&
                   ((reinterpret_cast<uintptr_t>(hidden) & 15) == 0);
  const int64_t blocks = (M + kRows - 1) / kRows;
  kern<<<(unsigned)blocks, kThreads, smem, stream>>>(
      static_cast<const TI*>(hidden), static_cast<const TI*>(w_down),
      static_cast<const TI*>(w_up_k), static_cast<const TI*>(w_up_v), static_cast<TO*>(latent),
      static_cast<TO*>(k), static_cast<TO*>(v), M, Dm, R, C, vec4);
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_r(const void* hidden, const void* w_down, const void* w_up_k,
                     const void* w_up_v, void* latent, void* k, void* v, int64_t M, int Dm, int R,
                     int C, cudaStream_t stream) {
  if (R <= 64)
    return launch_typed<TI, TO, 64>(hidden, w_down, w_up_k, w_up_v, latent, k, v, M, Dm, R, C,
                                    stream);
  if (R <= 256)
    return launch_typed<TI, TO, 256>(hidden, w_down, w_up_k, w_up_v, latent, k, v, M, Dm, R, C,
                                     stream);
  return launch_typed<TI, TO, 512>(hidden, w_down, w_up_k, w_up_v, latent, k, v, M, Dm, R, C,
                                   stream);
}

}  // namespace

cudaError_t launch_projection_cuda_core(const void* hidden, const void* w_down,
                                        const void* w_up_k, const void* w_up_v, void* latent,
                                        void* k, void* v, int64_t M, int Dm, int R, int C,
                                        int in_bf16, int out_bf16, cudaStream_t stream) {
  if (!in_bf16)
    return launch_r<float, float>(hidden, w_down, w_up_k, w_up_v, latent, k, v, M, Dm, R, C,
                                  stream);
  if (out_bf16)
    return launch_r<__nv_bfloat16, __nv_bfloat16>(hidden, w_down, w_up_k, w_up_v, latent, k, v,
                                                  M, Dm, R, C, stream);
  return launch_r<__nv_bfloat16, float>(hidden, w_down, w_up_k, w_up_v, latent, k, v, M, Dm, R,
                                        C, stream);
}

}  // namespace mla
