// tfx_router.cu -- routing ids and weights from router logits (top-k per row), optionally
// with a shared expert appended to every row.
//
// The pages take the routing as given (the rows kernels of TensorFold PR #2983 start from the
// routed ids); this entry produces it with the conventions the library's inputs use: the k
// largest logits of a row are selected, ties going to the lower expert id, in descending
// order; the weights are a softmax over the selected logits (or normalised sigmoid scores).
//
// One warp per row. Lane l holds logits l, l + 32, ... in registers; each of the k rounds
// takes every lane's best remaining candidate, the warp's largest order key (redux.sync max)
// and the lowest id holding it (redux.sync min); the winner lane retires it. Order keys rank
// NaN below every number and -0 with +0, so that equal values go to the lower id.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tfx_common.cuh"

namespace tfx {

constexpr int RO_WARPS = 8;

// Monotone unsigned key of a float value: NaN -> 0, otherwise larger value -> larger key,
// with -0 and +0 equal.
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v != v) return 0u;
  uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

template <int NI>
__global__ void __launch_bounds__(RO_WARPS * 32) router_kernel(const float* __restrict__ logits, int R, int E, int k,
                                                                int mode, int shared, int32_t* __restrict__ ids,
                                                                float* __restrict__ w) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * RO_WARPS + (threadIdx.x >> 5);
  if (row >= R) return;  // whole warps only
  const float* lrow = logits + (size_t)row * E;
  uint32_t key[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    key[i] = e < E ? order_key(__ldg(lrow + e)) : 0u;
  }
  uint32_t live = 0u;  // candidates this lane still holds
#pragma unroll
  for (int i = 0; i < NI; ++i)
    if (lane + 32 * i < E) live |= 1u << i;
  int my_id = -1;  // lane j < k: the id selected in round j
  for (int j = 0; j < k; ++j) {
    // best candidate of this lane: largest key, then lowest id (lower i)
    uint32_t bk = 0u;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (((live >> i) & 1u) && (bi < 0 || key[i] > bk)) {
        bk = key[i];
        bi = i;
      }
    // the warp's largest key, then the lowest id holding it
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bi >= 0 ? bk : 0u);
    const uint32_t cand = (bi >= 0 && bk == kmax) ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu;
    const int win = (int)__reduce_min_sync(0xffffffffu, cand);
    if (bi >= 0 && lane + 32 * bi == win) live &= ~(1u << bi);
    if (lane == j) my_id = win;
  }
  // weights over the selected logits, in slot order
  float lv = 0.0f;
  if (lane < k) lv = __ldg(lrow + my_id);
  float t = 0.0f;
  if (mode == TFX_ROUTER_SOFTMAX) {
    const float mx = __shfl_sync(0xffffffffu, lv, 0);
    t = lane < k ? expf(lv - mx) : 0.0f;
  } else {
    t = lane < k ? __fdiv_rn(1.0f, 1.0f + expf(-lv)) : 0.0f;
  }
  float s = 0.0f;
  for (int j = 0; j < k; ++j) s = __fadd_rn(s, __shfl_sync(0xffffffffu, t, j));
  const int stride = k + (shared >= 0 ? 1 : 0);
  if (lane < k) {
    ids[(size_t)row * stride + lane] = my_id;
    w[(size_t)row * stride + lane] = __fdiv_rn(t, s);
  }
  if (shared >= 0 && lane == 0) {
    ids[(size_t)row * stride + k] = shared;
    w[(size_t)row * stride + k] = 1.0f;
  }
}

}  // namespace tfx

using namespace tfx;

extern "C" int tfx_xp_router(int32_t rows, int32_t n_logits, int32_t top_k, const float* logits, int32_t mode,
                             int32_t shared_expert, int32_t* ids, float* topk_w, void* stream) {
  if (rows < 0 || n_logits < 1 || n_logits > 1024 || top_k < 1 || top_k > 32 || top_k > n_logits) return TFX_EINVAL;
  if (mode != TFX_ROUTER_SOFTMAX && mode != TFX_ROUTER_SIGMOID) return TFX_EINVAL;
  if (shared_expert < -1) return TFX_EINVAL;
  if (rows == 0) return TFX_OK;
  if (!logits || !ids || !topk_w) return TFX_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = (rows + RO_WARPS - 1) / RO_WARPS;
  if (n_logits <= 256)
    router_kernel<8><<<grid, RO_WARPS * 32, 0, st>>>(logits, rows, n_logits, top_k, mode, shared_expert, ids, topk_w);
  else
    router_kernel<32><<<grid, RO_WARPS * 32, 0, st>>>(logits, rows, n_logits, top_k, mode, shared_expert, ids, topk_w);
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}
