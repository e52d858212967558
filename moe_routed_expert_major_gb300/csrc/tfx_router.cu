// tfx_router.cu -- routing ids and weights from router logits (top-k per row), optionally
// with a shared expert appended to every row.
//
// The pages take the routing as given (the rows kernels of TensorFold PR #2983 start from the
// routed ids); this entry produces it with the conventions the library's inputs use: the k
// largest logits of a row are selected, ties going to the lower expert id, in descending
// order; the weights are a softmax over the selected logits (or normalised sigmoid scores).
//
// One warp per row. Lane l holds logits l, l + 32, ... in registers and the k rounds of
// topk_rounds pick the ids. Order keys rank NaN below every number and -0 with +0, so that
// equal values go to the lower id.
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

// k rounds over the candidates this lane holds (bit i of live: candidate lane + 32 i, order
// key key[i]); each round takes every lane's best remaining candidate (largest key, then
// lower id), the warp's largest key (redux.sync max) and the lowest id holding it (redux.sync
// min), and the winner lane retires it. Returns, in lane j < k, the id taken in round j.
template <int NI>
__device__ __forceinline__ int topk_rounds(const uint32_t (&key)[NI], uint32_t live, int k, int lane) {
  int my_id = -1;
  for (int j = 0; j < k; ++j) {
    uint32_t bk = 0u;
    int bi = -1;
#pragma unroll
    for (int i = 0; i < NI; ++i)
      if (((live >> i) & 1u) && (bi < 0 || key[i] > bk)) {
        bk = key[i];
        bi = i;
      }
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, bi >= 0 ? bk : 0u);
    const uint32_t cand = (bi >= 0 && bk == kmax) ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu;
    const int win = (int)__reduce_min_sync(0xffffffffu, cand);
    if (bi >= 0 && lane + 32 * bi == win) live &= ~(1u << bi);
    if (lane == j) my_id = win;
  }
  return my_id;
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
  const int my_id = topk_rounds<NI>(key, live, k, lane);  // lane j < k: the id selected in round j
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

// ---------------------------------------------------------------- group-limited routing
// The sigmoid of the grouped router, every step one IEEE fp32 operation rounded to nearest
// (no contraction), so that its value is fixed by the definition: t = exp(y) for
// y = max(-|l|, -86) by Cody-Waite reduction (n = rint(y / ln 2), r = (y - n*ln2_hi) -
// n*ln2_lo, with a 16-bit ln2_hi so that n*ln2_hi is exact) and the degree-7 Taylor
// polynomial of exp(r) in Horner form, times 2^n; then 1 / (1 + t) for l >= 0, t / (1 + t)
// below. NaN stays NaN; logits below -86 are taken as -86 (their sigmoid is below 5e-38).
__device__ __forceinline__ float sigmoid32(float l) {
  if (l != l) return l;
  const float y = fmaxf(-fabsf(l), -86.0f);
  const float n = rintf(__fmul_rn(y, __uint_as_float(0x3FB8AA3Bu)));                 // 1/ln 2
  const float r = __fsub_rn(__fsub_rn(y, __fmul_rn(n, __uint_as_float(0x3F317200u))),  // ln2_hi
                            __fmul_rn(n, __uint_as_float(0x35BFBE8Eu)));              // ln2_lo
  // 1/j! for j = 7 .. 0
  constexpr uint32_t kInvFact[8] = {0x39500D01u, 0x3AB60B61u, 0x3C088889u, 0x3D2AAAABu,
                                    0x3E2AAAABu, 0x3F000000u, 0x3F800000u, 0x3F800000u};
  float p = __uint_as_float(kInvFact[0]);
#pragma unroll
  for (int j = 1; j < 8; ++j) p = __fadd_rn(__fmul_rn(p, r), __uint_as_float(kInvFact[j]));
  const float t = __fmul_rn(p, __int_as_float(((int)n + 127) << 23));
  const float d = __fadd_rn(1.0f, t);
  return l >= 0.0f ? __fdiv_rn(1.0f, d) : __fdiv_rn(t, d);
}

constexpr int RG_WARPS = 4;

// One warp per row. Choice scores c = sigmoid32(l) + bias go to a shared-memory row; lane g <
// n_group scans group g for its two best scores (order key, then lower id) and sums them; the
// topk_group best groups are taken in redux.sync rounds (equal sums: lower group), and the
// top_k rounds of router_kernel then run over the experts of the kept groups only.
template <int NI>
__global__ void __launch_bounds__(RG_WARPS * 32)
    router_grouped_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int R, int E, int k,
                          int ng, int kg, float scale, int shared, int32_t* __restrict__ ids,
                          float* __restrict__ w) {
  __shared__ float cbuf[RG_WARPS][32 * NI];
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * RG_WARPS + (threadIdx.x >> 5);
  if (row >= R) return;  // whole warps only
  float* cb = cbuf[threadIdx.x >> 5];
  const float* lrow = logits + (size_t)row * E;
  uint32_t key[NI];
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    key[i] = 0u;
    if (e < E) {
      const float s = sigmoid32(__ldg(lrow + e));
      const float c = bias ? __fadd_rn(s, __ldg(bias + e)) : s;
      cb[e] = c;
      key[i] = order_key(c);
    }
  }
  __syncwarp();
  // group scores: the sum of each group's two best choice scores, best first
  const int gs = E / ng;
  uint32_t gkey = 0u;
  bool glive = false;
  if (lane < ng) {
    uint32_t k1 = 0u, k2 = 0u;
    float c1 = 0.0f, c2 = 0.0f;
    int n1 = -1, n2 = -1;
    for (int t = 0; t < gs; ++t) {
      const float c = cb[lane * gs + t];
      const uint32_t kk = order_key(c);
      if (n1 < 0 || kk > k1) {
        k2 = k1; c2 = c1; n2 = n1;
        k1 = kk; c1 = c; n1 = t;
      } else if (n2 < 0 || kk > k2) {
        k2 = kk; c2 = c; n2 = t;
      }
    }
    gkey = order_key(__fadd_rn(c1, c2));
    glive = true;
  }
  uint32_t gsel = 0u;
  for (int j = 0; j < kg; ++j) {
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, glive ? gkey : 0u);
    const uint32_t cand = (glive && gkey == kmax) ? (uint32_t)lane : 0xFFFFFFFFu;
    const int win = (int)__reduce_min_sync(0xffffffffu, cand);
    if (lane == win) glive = false;
    gsel |= 1u << win;
  }
  uint32_t live = 0u;
#pragma unroll
  for (int i = 0; i < NI; ++i) {
    const int e = lane + 32 * i;
    if (e < E && ((gsel >> (e / gs)) & 1u)) live |= 1u << i;
  }
  const int my_id = topk_rounds<NI>(key, live, k, lane);
  // weights: the selected experts' sigmoid (no bias), normalised in slot order, then scaled
  const float sv = lane < k ? sigmoid32(__ldg(lrow + my_id)) : 0.0f;
  float ssum = 0.0f;
  for (int j = 0; j < k; ++j) ssum = __fadd_rn(ssum, __shfl_sync(0xffffffffu, sv, j));
  const int stride = k + (shared >= 0 ? 1 : 0);
  if (lane < k) {
    ids[(size_t)row * stride + lane] = my_id;
    w[(size_t)row * stride + lane] = __fmul_rn(__fdiv_rn(sv, ssum), scale);
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

extern "C" int tfx_xp_router_grouped(int32_t rows, int32_t n_logits, int32_t top_k, const float* logits,
                                     const float* bias, int32_t n_group, int32_t topk_group, float scale,
                                     int32_t shared_expert, int32_t* ids, float* topk_w, void* stream) {
  if (rows < 0 || n_logits < 1 || n_logits > 1024 || top_k < 1 || top_k > 32) return TFX_EINVAL;
  if (n_group < 1 || n_group > 32 || n_logits % n_group != 0 || n_logits / n_group < 2) return TFX_EINVAL;
  if (topk_group < 1 || topk_group > n_group || top_k > topk_group * (n_logits / n_group)) return TFX_EINVAL;
  if (shared_expert < -1 || !(scale == scale)) return TFX_EINVAL;
  if (rows == 0) return TFX_OK;
  if (!logits || !ids || !topk_w) return TFX_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int grid = (rows + RG_WARPS - 1) / RG_WARPS;
  if (n_logits <= 256)
    router_grouped_kernel<8><<<grid, RG_WARPS * 32, 0, st>>>(logits, bias, rows, n_logits, top_k, n_group, topk_group,
                                                             scale, shared_expert, ids, topk_w);
  else
    router_grouped_kernel<32><<<grid, RG_WARPS * 32, 0, st>>>(logits, bias, rows, n_logits, top_k, n_group,
                                                              topk_group, scale, shared_expert, ids, topk_w);
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}
