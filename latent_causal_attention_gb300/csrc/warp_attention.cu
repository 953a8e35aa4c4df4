// Warp-per-query latent attention on CUDA cores (fp32 arithmetic).
//
// One warp computes one output row (b, i, h).  It works in the latent space:
// the query is first multiplied into the key weights (q'[r] = sum_e
// w_up_k[r,h,e] q[e], the identity (latent W_k).q = latent.(W_k q)), the
// flash-style online softmax then runs over the latent rows s <= t with
// lanes splitting the rank dimension and shuffles reducing the dot products,
// and w_up_v is applied once to the normalised latent-space sum at the end.
//
// Definition: page "FW-GLM-5-1 l2_p31" (fused MLA-style attention from
// compressed KV latents), "The algorithm"; the one-thread-per-query layout
// and the block-wide weight reuse discussed there are replaced by a warp per
// query so that 32 lanes share the rank-length dot products.  Online softmax
// with a running max: page "Kimi-K2.6 l2_p29", online softmax derivation.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"

namespace mla {

namespace {

template <typename T>
__device__ __forceinline__ float ld_f(const T* p);
template <>
__device__ __forceinline__ float ld_f<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_f<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void st_f(T* p, float v);
template <>
__device__ __forceinline__ void st_f<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_f<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr int kWarpsPerBlock = 4;

// RPL = rank elements per lane (rank <= 32 * RPL).
template <typename TI, typename TO, int RPL>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
    warp_attention_kernel(const TI* __restrict__ q, const TI* __restrict__ lat,
                          const TI* __restrict__ wk, const TI* __restrict__ wv,
                          TO* __restrict__ out, int B, int Tq, int Tkv, int H, int d, int R,
                          float scale_log2, int causal) {
  extern __shared__ float warp_smem[];                // kWarpsPerBlock * R floats
  const int lane = threadIdx.x & 31;
  const int wid = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * kWarpsPerBlock + wid;   // (b, i, h) flattened
  const int64_t rows = (int64_t)B * Tq * H;
  if (row >= rows) return;
  const int h = (int)(row % H);
  const int i = (int)((row / H) % Tq);
  const int b = (int)(row / ((int64_t)H * Tq));
  const int t = Tkv - Tq + i;
  const int n_keys = causal ? t + 1 : Tkv;
  float* olat = warp_smem + wid * R;

  // q'[r] = (scale * log2 e) * sum_e w_up_k[r,h,e] * q[b,i,h,e]
  const TI* qrow = q + row * d;
  float qa[RPL];
#pragma unroll
  for (int k = 0; k < RPL; ++k) {
    const int r = lane + 32 * k;
    float acc = 0.f;
    if (r < R) {
      const TI* w = wk + ((int64_t)r * H + h) * d;
      for (int e = 0; e < d; ++e) acc = fmaf(ld_f(w + e), ld_f(qrow + e), acc);
    }
    qa[k] = acc * scale_log2;
  }

  // Online softmax over the latent rows, in log2 units.
  float m = -INFINITY, l = 0.f;
  float o[RPL];
#pragma unroll
  for (int k = 0; k < RPL; ++k) o[k] = 0.f;
  const TI* lb = lat + (int64_t)b * Tkv * R;
  for (int s = 0; s < n_keys; ++s) {
    const TI* ls = lb + (int64_t)s * R;
    float lv[RPL];
    float part = 0.f;
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const int r = lane + 32 * k;
      lv[k] = (r < R) ? ld_f(ls + r) : 0.f;
      part = fmaf(qa[k], lv[k], part);
    }
    const float x = warp_sum(part);
    const float m_new = fmaxf(m, x);
    const float alpha = fast_exp2(m - m_new);        // m = -inf on the first key -> 0
    const float p = fast_exp2(x - m_new);
    l = l * alpha + p;
#pragma unroll
    for (int k = 0; k < RPL; ++k) o[k] = fmaf(o[k], alpha, p * lv[k]);
    m = m_new;
  }

  const float inv_l = 1.f / l;
#pragma unroll
  for (int k = 0; k < RPL; ++k) {
    const int r = lane + 32 * k;
    if (r < R) olat[r] = o[k] * inv_l;
  }
  __syncwarp();

  // out[e] = sum_r olat[r] * w_up_v[r,h,e]
  TO* orow = out + row * d;
  for (int e = lane; e < d; e += 32) {
    float acc = 0.f;
    const TI* w = wv + (int64_t)h * d + e;
    const int64_t step = (int64_t)H * d;
    for (int r = 0; r < R; ++r) acc = fmaf(olat[r], ld_f(w + r * step), acc);
    st_f(orow + e, acc);
  }
}

template <typename TI, typename TO, int RPL>
cudaError_t launch_rpl(const void* q, const void* lat, const void* wk, const void* wv, void* out,
                       int B, int Tq, int Tkv, int H, int d, int R, float scale, int causal,
                       cudaStream_t stream) {
  const int64_t rows = (int64_t)B * Tq * H;
  const int64_t blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
  const size_t smem = sizeof(float) * kWarpsPerBlock * R;
  auto kern = warp_attention_kernel<TI, TO, RPL>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  const float scale_log2 = scale * 1.4426950408889634f;
  kern<<<(unsigned)blocks, kWarpsPerBlock * 32, smem, stream>>>(
      static_cast<const TI*>(q), static_cast<const TI*>(lat), static_cast<const TI*>(wk),
      static_cast<const TI*>(wv), static_cast<TO*>(out), B, Tq, Tkv, H, d, R, scale_log2,
      causal);
  return cudaGetLastError();
}

template <typename TI, typename TO>
cudaError_t launch_typed(const void* q, const void* lat, const void* wk, const void* wv,
                         void* out, int B, int Tq, int Tkv, int H, int d, int R, float scale,
                         int causal, cudaStream_t stream) {
  if (R <= 64)
    return launch_rpl<TI, TO, 2>(q, lat, wk, wv, out, B, Tq, Tkv, H, d, R, scale, causal, stream);
  if (R <= 256)
    return launch_rpl<TI, TO, 8>(q, lat, wk, wv, out, B, Tq, Tkv, H, d, R, scale, causal, stream);
  return launch_rpl<TI, TO, 32>(q, lat, wk, wv, out, B, Tq, Tkv, H, d, R, scale, causal, stream);
}

}  // namespace

cudaError_t launch_warp_attention(const void* q, const void* lat, const void* wk, const void* wv,
                                  void* out, int B, int Tq, int Tkv, int H, int d, int R,
                                  float scale, int causal, int in_bf16, int out_bf16,
                                  cudaStream_t stream) {
  if (!in_bf16)
    return launch_typed<float, float>(q, lat, wk, wv, out, B, Tq, Tkv, H, d, R, scale, causal,
                                      stream);
  if (out_bf16)
    return launch_typed<__nv_bfloat16, __nv_bfloat16>(q, lat, wk, wv, out, B, Tq, Tkv, H, d, R,
                                                      scale, causal, stream);
  return launch_typed<__nv_bfloat16, float>(q, lat, wk, wv, out, B, Tq, Tkv, H, d, R, scale,
                                            causal, stream);
}

}  // namespace mla
