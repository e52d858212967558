// tfx_combine.cu -- routing-weighted sum of a row's k expert outputs ("combine output" of
// the equality probe in TensorFold PR #2983, "Kernel contract"): for each row r and output
// m, y = fma chain over the slots j = 0..k-1 in slot order from +0 of w[r][j] * d[r][j][m],
// then rounded to bf16 (nearest even). Each thread owns four consecutive outputs of one row,
// read as float4 per slot.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tfx_common.cuh"

namespace tfx {

// K8 > 0: k is known (<= 8) and every slot's loads are issued before the fma chain.
template <int K8>
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ d, const float* __restrict__ w, int R,
                                                      int k, int H, uint16_t* __restrict__ y, float* y32) {
  const int q4 = H / 4;
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (long long)R * q4) return;
  const int r = (int)(i / q4), m4 = (int)(i - (long long)r * q4);
  const float* dr = d + (size_t)r * k * H + 4 * m4;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if constexpr (K8 > 0) {
    float4 v[K8];
    float wj[K8];
#pragma unroll
    for (int j = 0; j < K8; ++j) {
      v[j] = *reinterpret_cast<const float4*>(dr + (size_t)j * H);
      wj[j] = w[(size_t)r * K8 + j];
    }
#pragma unroll
    for (int j = 0; j < K8; ++j) {
      acc.x = __fmaf_rn(wj[j], v[j].x, acc.x);
      acc.y = __fmaf_rn(wj[j], v[j].y, acc.y);
      acc.z = __fmaf_rn(wj[j], v[j].z, acc.z);
      acc.w = __fmaf_rn(wj[j], v[j].w, acc.w);
    }
  } else {
    for (int j = 0; j < k; ++j) {
      const float wj = w[(size_t)r * k + j];
      const float4 v = *reinterpret_cast<const float4*>(dr + (size_t)j * H);
      acc.x = __fmaf_rn(wj, v.x, acc.x);
      acc.y = __fmaf_rn(wj, v.y, acc.y);
      acc.z = __fmaf_rn(wj, v.z, acc.z);
      acc.w = __fmaf_rn(wj, v.w, acc.w);
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 pk;
  pk.x = *reinterpret_cast<uint32_t*>(&lo);
  pk.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(y + (size_t)r * H + 4 * m4) = pk;
  if (y32) *reinterpret_cast<float4*>(y32 + (size_t)r * H + 4 * m4) = acc;
}

}  // namespace tfx

using namespace tfx;

extern "C" int tfx_xp_combine(tfx_dims d, int32_t rows, const float* out, const float* topk_w, uint16_t* y,
                              float* y_f32_dbg, void* stream) {
  if (d.hidden <= 0 || d.hidden % 64 != 0 || d.top_k < 1 || d.top_k > 32 || rows < 0) return TFX_EINVAL;
  if (rows == 0) return TFX_OK;
  auto al = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
  if (!out || !topk_w || !y || !al(out, 16) || !al(y, 8) || (y_f32_dbg && !al(y_f32_dbg, 16))) return TFX_EINVAL;
  const long long n = (long long)rows * (d.hidden / 4);
  const int blocks = (int)((n + 255) / 256);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (d.top_k) {
#define TFX_CK(K) case K: combine_kernel<K><<<blocks, 256, 0, st>>>(out, topk_w, rows, d.top_k, d.hidden, y, y_f32_dbg); break;
    TFX_CK(1) TFX_CK(2) TFX_CK(4) TFX_CK(6) TFX_CK(8)
#undef TFX_CK
    default: combine_kernel<0><<<blocks, 256, 0, st>>>(out, topk_w, rows, d.top_k, d.hidden, y, y_f32_dbg);
  }
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}
