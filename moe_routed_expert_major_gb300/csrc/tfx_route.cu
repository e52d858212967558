// tfx_route.cu -- expert-major row lists ("every expert's rows", commit message of the rows
// kernels in TensorFold PR #2983): a stable counting sort of the (row, slot) pairs by expert
// id, by CTAs of 1024 threads.
//
// CTA c of G scatters the c-th contiguous block of pairs; every CTA counts all pairs, those
// before its block separately (pre[e]), so that no CTA needs another's results (no scratch,
// no grid-wide wait). Its block is split into 32 contiguous chunks, one per warp. Phase 1:
// each warp counts its chunk per expert (shared-memory histogram [32][E]); the other pairs go
// to pre[e] (before the block) and tot[e] (all). Phase 2: per expert, exclusive sums over the
// warps, and over the experts of the totals, give each (warp, expert) its first position,
// the offsets and the active list. Phase 3: each warp walks its chunk in rounds of 32 pairs;
// a pair's position is offs[e] + pre[e] + its (warp, expert) base + its rank among the
// round's pairs of the same expert (__match_any_sync), so every expert's pairs come out in
// ascending (row, slot) order whatever the thread timing. When the ids fit, each CTA first
// copies them into shared memory (coalesced) and records each pair's validity there, so that
// neither the duplicate checks nor the scatter go back to global memory. One CTA serves up to
// 2,048 pairs; larger launches use one CTA per 1,024 pairs, up to one per SM.
#include <cuda_runtime.h>
#include <stdint.h>

#include "tfx_common.cuh"

namespace tfx {

constexpr int RT_THREADS = 1024;
constexpr int RT_WARPS = RT_THREADS / 32;

// A pair is valid if its id is in range and no earlier slot of its row has the same id.
__device__ __forceinline__ int pair_expert(const int32_t* ids, int q, int k, int E, int* bad) {
  const int e = ids[q];
  if (e < 0 || e >= E) { *bad |= TFX_ST_RANGE; return -1; }
  const int r0 = q - q % k;
  for (int jj = r0; jj < q; ++jj)
    if (ids[jj] == e) { *bad |= TFX_ST_DUP; return -1; }
  return e;
}

template <bool STAGED>
__global__ void __launch_bounds__(RT_THREADS) route_kernel(const int32_t* __restrict__ ids_g, int P, int k, int E,
                                                           int32_t* offs, int32_t* pair_row, int32_t* pair_slot,
                                                           int32_t* active, int32_t* n_active, int32_t* status) {
  extern __shared__ int hist[];  // [RT_WARPS][E], scan scratch [E], pre [E], tot [E]; staged: ids [P], valid [P] bytes
  int* eoff = hist + RT_WARPS * E;
  int* pre = eoff + E;
  int* tot = pre + E;
  int* s_ids = tot + E;
  uint8_t* s_valid = reinterpret_cast<uint8_t*>(s_ids + (STAGED ? P : 0));
  __shared__ int s_bad;
  __shared__ int s_nact;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < (RT_WARPS + 3) * E; i += RT_THREADS) hist[i] = 0;
  if (STAGED)
    for (int i = tid; i < P; i += RT_THREADS) s_ids[i] = ids_g[i];
  if (tid == 0) { s_bad = 0; s_nact = 0; }
  __syncthreads();
  const int32_t* ids = STAGED ? s_ids : ids_g;

  // this CTA's block of pairs [b0, b1), and this warp's chunk [c0, c1) of it
  const int bsz = (P + (int)gridDim.x - 1) / (int)gridDim.x;
  const int b0 = min(P, (int)blockIdx.x * bsz), b1 = min(P, b0 + bsz);
  const int chunk = (b1 - b0 + RT_WARPS - 1) / RT_WARPS;
  const int c0 = min(b1, b0 + warp * chunk), c1 = min(b1, c0 + chunk);
  int bad = 0;
  // phase 1: per-warp histogram of the block; counts of the pairs outside it
  for (int q = c0 + lane; q < c1; q += 32) {
    const int e = pair_expert(ids, q, k, E, &bad);
    if (STAGED) s_valid[q] = e >= 0 ? 1 : 0;
    if (e >= 0) {
      atomicAdd(&hist[warp * E + e], 1);
      atomicAdd(&tot[e], 1);
    }
  }
  // the other pairs, a row a thread (one index division per row, not two per pair)
  for (int r = tid; r < P / k; r += RT_THREADS) {
    const int q0 = r * k;
    if (q0 >= b0 && q0 + k <= b1) continue;  // the whole row is in the block
    for (int q = q0; q < q0 + k; ++q) {
      if (q >= b0 && q < b1) continue;
      const int e = ids[q];
      if (e < 0 || e >= E) { bad |= TFX_ST_RANGE; continue; }
      bool dup = false;
      for (int jj = q0; jj < q; ++jj)
        if (ids[jj] == e) { dup = true; break; }
      if (dup) { bad |= TFX_ST_DUP; continue; }
      atomicAdd(&tot[e], 1);
      if (q < b0) atomicAdd(&pre[e], 1);
    }
  }
  if (bad) atomicOr(&s_bad, bad);
  __syncthreads();

  // phase 2: per expert, exclusive sum over warps; then over experts (serial per block of 32
  // experts a warp, then a scan of the block totals by warp 0)
  for (int e = tid; e < E; e += RT_THREADS) {
    int run = 0;
    for (int w = 0; w < RT_WARPS; ++w) {
      const int c = hist[w * E + e];
      hist[w * E + e] = run;
      run += c;
    }
    eoff[e] = tot[e];  // total of expert e for now
  }
  __syncthreads();
  if (warp == 0) {
    int base = 0, abase = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + lane;
      const int c = e < E ? eoff[e] : 0;
      int inc = c, act = (c > 0) ? 1 : 0;
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        const int a = __shfl_up_sync(0xffffffffu, act, o);
        if (lane >= o) { inc += v; act += a; }
      }
      if (e < E) {
        const int start = base + inc - c;
        eoff[e] = start + pre[e];  // this block's first position of expert e
        if (blockIdx.x == 0) {
          offs[e] = start;
          if (c > 0) active[abase + act - 1] = e;
        }
      }
      base += __shfl_sync(0xffffffffu, inc, 31);
      abase += __shfl_sync(0xffffffffu, act, 31);
    }
    if (lane == 0 && blockIdx.x == 0) {
      offs[E] = base;
      s_nact = abase;
    }
  }
  __syncthreads();
  if (tid == 0 && blockIdx.x == 0) {  // every CTA checks every pair: the first reports
    *n_active = s_nact;
    if (s_bad && status) atomicOr(status, s_bad);
  }

  // phase 3: stable scatter
  for (int q0 = c0; q0 < c1; q0 += 32) {
    const int q = q0 + lane;
    int dummy = 0;
    int e = -1;
    if (q < c1) e = STAGED ? (s_valid[q] ? ids[q] : -1) : pair_expert(ids, q, k, E, &dummy);
    const unsigned peers = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(peers & ((1u << lane) - 1u));
    const int leader = __ffs(peers) - 1;
    if (e >= 0) {
      const int pos = eoff[e] + hist[warp * E + e] + rank;
      pair_row[pos] = q / k;
      pair_slot[pos] = q % k;
    }
    __syncwarp();
    if (e >= 0 && lane == leader) hist[warp * E + e] += __popc(peers);
    __syncwarp();
  }
}

}  // namespace tfx

using namespace tfx;

extern "C" int tfx_xp_route(tfx_dims d, int32_t rows, const int32_t* ids, int32_t* offs, int32_t* pair_row,
                            int32_t* pair_slot, int32_t* active, int32_t* n_active, int32_t* status, void* stream) {
  if (d.n_experts < 1 || d.n_experts > 1024 || d.top_k < 1 || d.top_k > 32 || rows < 0) return TFX_EINVAL;
  if ((int64_t)rows * d.top_k > (1ll << 30)) return TFX_EINVAL;
  if (!offs || !active || !n_active || !status) return TFX_EINVAL;
  if (rows > 0 && (!ids || !pair_row || !pair_slot)) return TFX_EINVAL;
  const int E = d.n_experts;
  const int P = rows * d.top_k;
  // ids staged in shared memory (4 bytes + 1 validity byte per pair) when they fit
  const size_t base = (size_t)(RT_WARPS + 3) * E * sizeof(int);
  const size_t staged = base + (size_t)P * 5 + 16;
  const bool stage = P > 0 && staged <= 200 * 1024;
  const size_t smem = stage ? staged : base;
  auto kern = stage ? route_kernel<true> : route_kernel<false>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TFX_ELAUNCH;
  int grid = 1;
  if (P > 2048) {
    int dev = 0, sms = 1;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return TFX_ECUDA;
    grid = min(max(sms, 1), (P + 1023) / 1024);
  }
  kern<<<grid, RT_THREADS, smem, static_cast<cudaStream_t>(stream)>>>(ids, P, d.top_k, E, offs, pair_row, pair_slot,
                                                                    active, n_active, status);
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}
