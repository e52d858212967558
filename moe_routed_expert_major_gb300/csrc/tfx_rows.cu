// tfx_rows.cu -- expert-major "rows" kernels for launches of few rows per expert (decode):
// gate/up (+ SwiGLU + activation quantiser), down, and the whole layer fused in one launch.
//
// Method: "dsv41 metal: decode experts decode an expert's weights once for all of its rows"
// (TensorFold PR #2983). A work item is (active expert, block of outputs). Its weights are
// streamed once per pass; every 32-group is decoded once and applied to every row of the pass
// (pass sized by the rows left; padding rows repeat the last real row, are computed and never
// written). Each row's accumulators follow the fixed order of "What this changes": per group
// a sequential fma chain of the 32 unscaled products from +0 in k order, one scaled fma into
// accumulator (group mod 8), then the eight-way tree.
//
// GB300 mapping:
//   * one producer warp streams 17,408-byte stages (64 weight rows x 512 k of codes, then their
//     scales: contiguous in the packed layout) into a ring of shared-memory slots with
//     cp.async.bulk + mbarrier (every wait bounded);
//   * eight consumer warps; lane (t & 7) of an octet owns accumulator lane j = group mod 8 of
//     two output columns, so the eight-way tree is three xor-shuffles. A lane handles groups j
//     and j + 8 of each stage and both columns as four independent chains, interleaved;
//   * E2M1 codes decode with cvt.rn.f16x2.e2m1x2; activations sit in shared memory as f16
//     (exact for E4M3; bf16 rows are shifted per 32-group by a power of two so that they are
//     exact in f16, with an exact fp32 fallback for groups that do not fit); the chain runs on
//     fma.rn.f32.f16 (fp32 accumulate, one rounding per step).
//   * The fused layer launch (cooperative: all CTAs resident) computes the row lists in shared
//     memory in every CTA, runs all gate/up items, then the down items (each waits, bounded,
//     for its expert's gate/up items), and combines each (row, 64-output block) in the CTA
//     whose down item completes the row's last slot. Completion counters live in caller
//     scratch, which the last CTA to finish returns to zero.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "tfx_common.cuh"

namespace tfx {

constexpr int KC = 512;                          // k per stage
constexpr int GPS = KC / 32;                     // groups per stage
constexpr int TROWS = 64;                        // weight rows per stage
constexpr int CODE_B = KC / 2;                   // code bytes per row per stage
constexpr int STAGE_B = TROWS * (CODE_B + GPS);  // 17,408
constexpr int NCW = 8;                           // consumer warps
constexpr int NCONS = NCW * kWarp;               // 256
constexpr int NTHREADS = NCONS + kWarp;          // + one producer warp
constexpr int MAX_NSTAGE = 8;
constexpr int FUSED_MAX_PAIRS = 256;

enum { PH_UPC = 1, PH_DOWN = 2, PH_FUSED = 3 };

struct Proj {
  int K, S, G, GB, units;  // reduction length, stages, groups, group blocks of 8 (= 2S), items/expert
  size_t unit_bytes, expert_bytes;
  const uint8_t* w;
};

struct RowsParams {
  int H, I, E, k, R;
  Proj pu, pd;
  int nstage;
  int gbmax;            // group blocks allotted per activation row in shared memory
  int route_ints;       // shared-memory ints of the in-kernel route (fused)
  const void* x;        // token activations [R][H]
  const uint8_t* xs;    // E8M0 scales [R][H/32] (E4M3)
  const int32_t* ids;   // fused: top-k ids [R][k]
  const float* topk_w;  // fused: routing weights [R][k]
  int32_t *offs, *pair_row, *pair_slot, *active, *n_active;
  void* h;              // [P][I] E4M3 codes or bf16
  uint8_t* hs;          // [P][I/32]
  float* gu_dbg;        // [P][2][I]
  float* h_dbg;         // [P][I]
  float* out;           // [R][k][H]
  uint16_t* y;          // fused: [R][H] bf16
  float* y32;           // fused: [R][H] or null
  int32_t* scratch;     // fused: [0] exit count, [1..E] gate/up items done per active expert,
                        //        then [R][H/64] slots written per (row, block)
  int32_t* status;
  int tier_mode;
  uint64_t timeout_ns;
};

// ---------------------------------------------------------------- shared-memory layout
struct Layout {
  int bars, ctrl, pass, epi, route, ring, xs, xm, total;
};
__host__ __device__ inline Layout layout_of(const RowsParams& p, int maxr) {
  Layout L;
  L.bars = 0;      // full[8], empty[8]
  L.ctrl = 128;    // abort flag
  L.pass = 256;    // prow[8], ppair[8]
  L.epi = 512;     // float [8][64]
  L.route = 2560;  // fused: ints
  L.ring = (L.route + 4 * p.route_ints + 127) & ~127;
  L.xs = L.ring + p.nstage * STAGE_B;
  L.xm = L.xs + maxr * p.gbmax * 512;
  L.total = L.xm + maxr * p.gbmax * 8 * 4;
  return L;
}

template <bool DOWN>
__device__ __forceinline__ int tier_of(int left, int maxr, int mode) {
  if (mode == 1) return maxr;
  int t;
  if (!DOWN) t = left >= 7 ? 8 : left >= 5 ? 6 : left >= 3 ? 4 : left >= 2 ? 2 : 1;
  else t = left >= 3 ? 4 : left >= 2 ? 2 : 1;
  return t > maxr ? maxr : t;
}

// Byte offset in the permuted activation layout of row r, group g, 8-element chunk tc:
// chunk ((r*GB + g/8)*4 + tc)*8 + g%8 of 16 bytes, so the eight lanes that read one chunk
// index of eight consecutive groups touch 128 consecutive bytes.
__device__ __forceinline__ int xoff(int r, int g, int tc, int GB) {
  return ((((r * GB + (g >> 3)) * 4 + tc) * 8 + (g & 7)) << 4);
}

// Exact fp32 chain for a bf16 group whose values do not fit f16 after the shift: the
// group's codes are decoded again, and each product of an E2M1 value with the bf16 value read
// back from memory (at L2) is accumulated in k order from +0.
__device__ __noinline__ float chain_bf16_exact(uint4 codes, const uint16_t* xrow, int g) {
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
  float p = 0.0f;
  for (int q = 0; q < 4; ++q) {
    uint32_t hq[4];
    e2m1x8_to_f16x2(cw[q], hq[0], hq[1], hq[2], hq[3]);
    for (int i = 0; i < 4; ++i) {
      const __half2 hw = *reinterpret_cast<const __half2*>(&hq[i]);
      const int k = 32 * g + 8 * q + 2 * i;
      const uint32_t two = __ldcg(reinterpret_cast<const unsigned int*>(xrow + k));
      p = __fmaf_rn(__low2float(hw), __uint_as_float(two << 16), p);
      p = __fmaf_rn(__high2float(hw), __uint_as_float(two & 0xFFFF0000u), p);
    }
  }
  return p;
}

// Stage the activation rows of one pass into shared memory (consumer threads only). Groups
// from G up to the stage boundary are zero with multiplier 1, so that lanes past the end of
// the reduction add +0 to their accumulators.
template <int KIND>
__device__ void stage_rows(const uint8_t* __restrict__ X8, const uint8_t* __restrict__ XS, int K, int G, int GB,
                           uint8_t* xs_s, float* xm_s, const int* prow, int real, int tid) {
  const int nch = K / 8;          // chunks of 8 elements with data
  const int nall = GB * 8 * 4;    // chunks up to the stage boundary
  if (KIND == TFX_ACT_E4M3) {
    for (int i = tid; i < real * nall; i += NCONS) {
      const int r = i / nall, c = i - r * nall;
      uint4 o = make_uint4(0u, 0u, 0u, 0u);
      if (c < nch) {
        const uint2 v = __ldcg(reinterpret_cast<const uint2*>(X8 + (size_t)prow[r] * K + 8 * c));
        o.x = e4m3x2_to_f16x2(v.x);
        o.y = e4m3x2_to_f16x2(v.x >> 16);
        o.z = e4m3x2_to_f16x2(v.y);
        o.w = e4m3x2_to_f16x2(v.y >> 16);
      }
      *reinterpret_cast<uint4*>(xs_s + xoff(r, c >> 2, c & 3, GB)) = o;
    }
    for (int i = tid; i < real * GB * 8; i += NCONS) {
      const int r = i / (GB * 8), g = i - r * (GB * 8);
      xm_s[r * GB * 8 + g] = g < G ? e8m0_to_f32(__ldcg(XS + (size_t)prow[r] * G + g)) : 1.0f;
    }
  } else {
    // bf16: a half-warp converts one 32-group (two values a lane) with a power-of-two shift
    // 2^sigma that maps the group's largest magnitude into [2^15, 2^16). The group is exact in
    // f16 and its chain equals the unshifted fp32 chain times 2^sigma when every finite nonzero
    // value has exponent in [e_max - 32, e_max], e_max <= 119 and e_min >= -141 (products and
    // partial sums then stay in fp32's normal range, or on its subnormal grid, on both sides).
    // Otherwise the multiplier is 0 and the exact fallback runs for that group.
    const uint16_t* X = reinterpret_cast<const uint16_t*>(X8);
    const int wp = tid >> 5, half = (tid >> 4) & 1, lane16 = tid & 15;
    const int gall = GB * 8;
    const int total = real * gall;
    for (int i0 = 2 * wp; i0 < total; i0 += 2 * NCW) {  // uniform trip count per warp
      const int i = i0 + half;
      const bool act = i < total;
      int r = 0, g = 0;
      uint32_t two = 0;
      if (act) {
        r = i / gall;
        g = i - r * gall;
        if (g < G) two = __ldcg(reinterpret_cast<const unsigned int*>(X + (size_t)prow[r] * K + 32 * g + 2 * lane16));
      }
      int emax = -1000, emin = 1000;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const uint32_t b = (two >> (16 * hh)) & 0xFFFFu;
        const uint32_t ef = (b >> 7) & 0xFFu, m = b & 0x7Fu;
        if (ef == 255u || (ef == 0u && m == 0u)) continue;  // NaN/Inf or zero
        const int e = ef ? (int)ef - 127 : (31 - __clz((int)m)) - 133;
        emax = max(emax, e);
        emin = min(emin, e);
      }
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) {
        emax = max(emax, __shfl_xor_sync(0xffffffffu, emax, o));
        emin = min(emin, __shfl_xor_sync(0xffffffffu, emin, o));
      }
      if (!act) continue;
      int sigma = 0;
      bool safe = true;
      if (emax > -1000) {
        sigma = 15 - emax;
        safe = (emax <= 119) && (emin >= -141) && (emax - emin <= 32);
      }
      float lo = __uint_as_float(two << 16), hi = __uint_as_float(two & 0xFFFF0000u);
      if (safe) {
        const int s1 = min(max(sigma, -126), 127), s2 = sigma - s1;  // 2^sigma as two exact factors
        const float f1 = __uint_as_float((uint32_t)(127 + s1) << 23);
        const float f2 = __uint_as_float((uint32_t)(127 + s2) << 23);
        lo = __fmul_rn(__fmul_rn(lo, f1), f2);
        hi = __fmul_rn(__fmul_rn(hi, f1), f2);
      }
      const __half2 h2 = __floats2half2_rn(lo, hi);
      const int t = 2 * lane16;
      *reinterpret_cast<__half2*>(xs_s + xoff(r, g, t >> 3, GB) + ((t & 7) << 1)) = h2;
      if (lane16 == 0) {
        float m = 0.0f;  // 0 marks the exact fallback
        if (g >= G) m = 1.0f;
        else if (safe) {
          const int ns = -sigma;  // 2^-sigma, possibly subnormal (exact)
          m = ns >= -126 ? __uint_as_float((uint32_t)(127 + ns) << 23) : __uint_as_float(0x00400000u >> (-127 - ns));
        }
        xm_s[r * GB * 8 + g] = m;
      }
    }
  }
}

// Row lists of a small launch, computed in shared memory (fused layer): per-pair expert (or -1
// if left out), per-expert counts -> offsets, active experts, stable positions, per-row slot
// counts. All NTHREADS threads take part. Ints used: 3E + 2 + 3P + R.
struct SRoute {
  int *offs, *prow, *pslot, *act, *rowcnt, *ev, *cnt, *nact;
};
__device__ void route_smem(const RowsParams& p, int* base, SRoute& rt, int tid) {
  const int E = p.E, k = p.k, P = p.R * p.k;
  rt.offs = base;               // E + 1
  rt.cnt = rt.offs + E + 1;     // E
  rt.act = rt.cnt + E;          // E
  rt.nact = rt.act + E;         // 1
  rt.ev = rt.nact + 1;          // P
  rt.prow = rt.ev + P;          // P
  rt.pslot = rt.prow + P;       // P
  rt.rowcnt = rt.pslot + P;     // R
  for (int i = tid; i < E; i += NTHREADS) rt.cnt[i] = 0;
  for (int i = tid; i < p.R; i += NTHREADS) rt.rowcnt[i] = 0;
  __syncthreads();
  int bad = 0;
  for (int q = tid; q < P; q += NTHREADS) {
    const int e = p.ids[q];
    int v = e;
    if (e < 0 || e >= E) { v = -1; bad |= TFX_ST_RANGE; }
    else {
      for (int jj = q - q % k; jj < q; ++jj)
        if (p.ids[jj] == e) { v = -1; bad |= TFX_ST_DUP; break; }
    }
    rt.ev[q] = v;
    if (v >= 0) {
      atomicAdd(&rt.cnt[v], 1);
      atomicAdd(&rt.rowcnt[q / k], 1);
    }
  }
  if (bad && blockIdx.x == 0) report(p.status, bad);
  __syncthreads();
  if (tid < 32) {  // one warp: exclusive scan of counts and the active list
    int base_off = 0, base_act = 0;
    for (int e0 = 0; e0 < E; e0 += 32) {
      const int e = e0 + tid;
      const int c = e < E ? rt.cnt[e] : 0;
      int inc = c, a = c > 0 ? 1 : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o), w = __shfl_up_sync(0xffffffffu, a, o);
        if (tid >= o) { inc += v; a += w; }
      }
      if (e < E) {
        rt.offs[e] = base_off + inc - c;
        if (c > 0) rt.act[base_act + a - 1] = e;
      }
      base_off += __shfl_sync(0xffffffffu, inc, 31);
      base_act += __shfl_sync(0xffffffffu, a, 31);
    }
    if (tid == 0) {
      rt.offs[E] = base_off;
      *rt.nact = base_act;
    }
  }
  __syncthreads();
  for (int q = tid; q < P; q += NTHREADS) {
    const int e = rt.ev[q];
    if (e < 0) continue;
    int rank = 0;
    for (int qq = 0; qq < q; ++qq) rank += rt.ev[qq] == e;
    const int pos = rt.offs[e] + rank;
    rt.prow[pos] = q / k;
    rt.pslot[pos] = q % k;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- one pass of T rows
// Consumes the pass's S stages from the ring and leaves the eight-way-tree results of both
// columns of every real row in epi[r][0..63] (column o at o, column 32 + o at 32 + o).
template <int KIND, int T>
__device__ __forceinline__ void run_pass(const RowsParams& P, const Proj& pj, uint8_t* ring, uint64_t* full,
                                         uint64_t* empty, volatile int* abort_flag, const uint8_t* xs_s,
                                         const float* xm_s, const int* prow, const uint16_t* xraw, int real,
                                         uint32_t& it, bool& dead, float* epi) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = lane & 7, o = (warp << 2) | (lane >> 3);
  const int NST = P.nstage, GB = pj.GB;
  float acc0[T], acc1[T];
  int xr[T];
#pragma unroll
  for (int r = 0; r < T; ++r) {
    acc0[r] = 0.0f;
    acc1[r] = 0.0f;
    xr[r] = min(r, real - 1);
  }
  for (int s = 0; s < pj.S; ++s, ++it) {
    const int slot = it % NST;
    const uint32_t ph = (it / NST) & 1u;
    if (!dead) {
      // warp-uniform outcome, so the full-warp shuffles and reductions after it stay legal
      bool ok = (*abort_flag == 0) && mbar_wait(&full[slot], ph, P.timeout_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        dead = true;
        if (lane == 0) {
          report(P.status, TFX_ST_TIMEOUT);
          *abort_flag = 1;
        }
      }
    }
    if (!dead) {
      const uint8_t* tile = ring + (size_t)slot * STAGE_B;
      const uint8_t* sc = tile + TROWS * CODE_B;
      const uint4 cA0 = *reinterpret_cast<const uint4*>(tile + o * CODE_B + 16 * j);
      const uint4 cA1 = *reinterpret_cast<const uint4*>(tile + (32 + o) * CODE_B + 16 * j);
      const uint4 cB0 = *reinterpret_cast<const uint4*>(tile + o * CODE_B + 128 + 16 * j);
      const uint4 cB1 = *reinterpret_cast<const uint4*>(tile + (32 + o) * CODE_B + 128 + 16 * j);
      const float sA0 = e8m0_to_f32(sc[o * GPS + j]), sA1 = e8m0_to_f32(sc[(32 + o) * GPS + j]);
      const float sB0 = e8m0_to_f32(sc[o * GPS + 8 + j]), sB1 = e8m0_to_f32(sc[(32 + o) * GPS + 8 + j]);
      const int gA = s * GPS + j, gB = gA + 8;
      float pA0[T], pA1[T], pB0[T], pB1[T];
#pragma unroll
      for (int r = 0; r < T; ++r) { pA0[r] = 0.0f; pA1[r] = 0.0f; pB0[r] = 0.0f; pB1[r] = 0.0f; }
      const uint32_t* wA0 = reinterpret_cast<const uint32_t*>(&cA0);
      const uint32_t* wA1 = reinterpret_cast<const uint32_t*>(&cA1);
      const uint32_t* wB0 = reinterpret_cast<const uint32_t*>(&cB0);
      const uint32_t* wB1 = reinterpret_cast<const uint32_t*>(&cB1);
#pragma unroll
      for (int tc = 0; tc < 4; ++tc) {
        uint32_t a0[4], a1[4], b0[4], b1[4];
        e2m1x8_to_f16x2(wA0[tc], a0[0], a0[1], a0[2], a0[3]);
        e2m1x8_to_f16x2(wA1[tc], a1[0], a1[1], a1[2], a1[3]);
        e2m1x8_to_f16x2(wB0[tc], b0[0], b0[1], b0[2], b0[3]);
        e2m1x8_to_f16x2(wB1[tc], b1[0], b1[1], b1[2], b1[3]);
#pragma unroll
        for (int r = 0; r < T; ++r) {
          const uint4 xa = *reinterpret_cast<const uint4*>(xs_s + xoff(xr[r], gA, tc, GB));
          const uint4 xb = *reinterpret_cast<const uint4*>(xs_s + xoff(xr[r], gB, tc, GB));
          const uint32_t* va = reinterpret_cast<const uint32_t*>(&xa);
          const uint32_t* vb = reinterpret_cast<const uint32_t*>(&xb);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            pA0[r] = fma2_f16(a0[i], va[i], pA0[r]);
            pA1[r] = fma2_f16(a1[i], va[i], pA1[r]);
            pB0[r] = fma2_f16(b0[i], vb[i], pB0[r]);
            pB1[r] = fma2_f16(b1[i], vb[i], pB1[r]);
          }
        }
      }
#pragma unroll
      for (int r = 0; r < T; ++r) {
        const float mA = xm_s[xr[r] * GB * 8 + gA], mB = xm_s[xr[r] * GB * 8 + gB];
        if (KIND == TFX_ACT_E4M3) {
          acc0[r] = __fmaf_rn(pA0[r], __fmul_rn(sA0, mA), acc0[r]);
          acc1[r] = __fmaf_rn(pA1[r], __fmul_rn(sA1, mA), acc1[r]);
          acc0[r] = __fmaf_rn(pB0[r], __fmul_rn(sB0, mB), acc0[r]);
          acc1[r] = __fmaf_rn(pB1[r], __fmul_rn(sB1, mB), acc1[r]);
        } else {
          float qA0 = pA0[r], qA1 = pA1[r], qB0 = pB0[r], qB1 = pB1[r];
          const uint16_t* xrow = xraw + (size_t)prow[xr[r]] * pj.K;
          if (mA == 0.0f) {
            qA0 = chain_bf16_exact(cA0, xrow, gA);
            qA1 = chain_bf16_exact(cA1, xrow, gA);
          } else {
            qA0 = __fmul_rn(qA0, mA);
            qA1 = __fmul_rn(qA1, mA);
          }
          if (mB == 0.0f) {
            qB0 = chain_bf16_exact(cB0, xrow, gB);
            qB1 = chain_bf16_exact(cB1, xrow, gB);
          } else {
            qB0 = __fmul_rn(qB0, mB);
            qB1 = __fmul_rn(qB1, mB);
          }
          acc0[r] = __fmaf_rn(qA0, sA0, acc0[r]);
          acc1[r] = __fmaf_rn(qA1, sA1, acc1[r]);
          acc0[r] = __fmaf_rn(qB0, sB0, acc0[r]);
          acc1[r] = __fmaf_rn(qB1, sB1, acc1[r]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
  // eight-way tree: ((a0+a4)+(a2+a6)) + ((a1+a5)+(a3+a7)) across the octet
#pragma unroll
  for (int r = 0; r < T; ++r) {
    float v0 = acc0[r], v1 = acc1[r];
    v0 = v0 + __shfl_xor_sync(0xffffffffu, v0, 4);
    v1 = v1 + __shfl_xor_sync(0xffffffffu, v1, 4);
    v0 = v0 + __shfl_xor_sync(0xffffffffu, v0, 2);
    v1 = v1 + __shfl_xor_sync(0xffffffffu, v1, 2);
    v0 = v0 + __shfl_xor_sync(0xffffffffu, v0, 1);
    v1 = v1 + __shfl_xor_sync(0xffffffffu, v1, 1);
    if (j == 0 && r < real) {
      epi[r * 64 + o] = v0;
      epi[r * 64 + 32 + o] = v1;
    }
  }
}

template <int KIND, int MAXR, bool DOWN>
__device__ __forceinline__ void dispatch_pass(int t, const RowsParams& P, const Proj& pj, uint8_t* ring,
                                              uint64_t* full, uint64_t* empty, volatile int* abort_flag,
                                              const uint8_t* xs_s, const float* xm_s, const int* prow,
                                              const uint16_t* xraw, int real, uint32_t& it, bool& dead, float* epi) {
#define TFX_PASS(TT) run_pass<KIND, TT>(P, pj, ring, full, empty, abort_flag, xs_s, xm_s, prow, xraw, real, it, dead, epi)
  switch (t) {
    case 1: TFX_PASS(1); break;
    case 2: if constexpr (MAXR >= 2) TFX_PASS(2); break;
    case 4: if constexpr (MAXR >= 4) TFX_PASS(4); break;
    case 6: if constexpr (!DOWN && MAXR >= 8) TFX_PASS(6); break;
    case 8: if constexpr (!DOWN && MAXR >= 8) TFX_PASS(8); break;
    default: break;
  }
#undef TFX_PASS
}

// ---------------------------------------------------------------- the kernel
template <int KIND, int MAXR_U, int MAXR_D, int PH>
__global__ void __launch_bounds__(NTHREADS, ((PH & PH_UPC) ? MAXR_U : MAXR_D) <= 2 ? 2 : 1)
    rows_kernel(const RowsParams P) {
  constexpr int MAXR = ((PH & PH_UPC) && MAXR_U > MAXR_D) || !(PH & PH_DOWN) ? MAXR_U : MAXR_D;
  extern __shared__ __align__(128) uint8_t smem[];
  const Layout Ly = layout_of(P, MAXR);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Ly.bars);
  uint64_t* empty = full + MAX_NSTAGE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly.ctrl);
  int* prow = reinterpret_cast<int*>(smem + Ly.pass);
  int* ppair = prow + 8;
  float* epi = reinterpret_cast<float*>(smem + Ly.epi);
  uint8_t* ring = smem + Ly.ring;
  uint8_t* xs_s = smem + Ly.xs;
  float* xm_s = reinterpret_cast<float*>(smem + Ly.xm);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NST = P.nstage;
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_fence_init();
    *abort_flag = 0;
  }

  // row lists: computed here (fused) or read from a previous route launch
  const int *r_offs, *r_prow, *r_pslot, *r_act, *r_rowcnt = nullptr;
  int n_act;
  if (PH == PH_FUSED) {
    SRoute rt;
    route_smem(P, reinterpret_cast<int*>(smem + Ly.route), rt, tid);  // synchronises the block
    n_act = *rt.nact;
    r_offs = rt.offs;
    r_prow = rt.prow;
    r_pslot = rt.pslot;
    r_act = rt.act;
    r_rowcnt = rt.rowcnt;
    if (blockIdx.x == 0) {  // publish the row lists
      const int Pn = P.R * P.k;
      for (int i = tid; i <= P.E; i += NTHREADS) P.offs[i] = rt.offs[i];
      for (int i = tid; i < Pn; i += NTHREADS) {
        P.pair_row[i] = i < rt.offs[P.E] ? rt.prow[i] : 0;
        P.pair_slot[i] = i < rt.offs[P.E] ? rt.pslot[i] : 0;
      }
      for (int i = tid; i < n_act; i += NTHREADS) P.active[i] = rt.act[i];
      if (tid == 0) *P.n_active = n_act;
    }
  } else {
    __syncthreads();
    n_act = *P.n_active;
    r_offs = P.offs;
    r_prow = P.pair_row;
    r_pslot = P.pair_slot;
    r_act = P.active;
  }
  const int n_upc = (PH & PH_UPC) ? n_act * P.pu.units : 0;
  const int n_down = (PH & PH_DOWN) ? n_act * P.pd.units : 0;
  const int total = n_upc + n_down;
  int32_t* done_upc = PH == PH_FUSED ? P.scratch + 1 : nullptr;
  int32_t* slots_done = PH == PH_FUSED ? P.scratch + 1 + P.E : nullptr;

  if (warp == NCW) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      for (int item = blockIdx.x; item < total && !stop; item += gridDim.x) {
        const bool dn = item >= n_upc;
        const Proj& pj = dn ? P.pd : P.pu;
        const int li = dn ? item - n_upc : item;
        const int a = li / pj.units, u = li - a * pj.units;
        const int e = r_act[a];
        if (e < 0 || e >= P.E) continue;
        const int p0 = r_offs[e], n = r_offs[e + 1] - p0;
        if (n <= 0 || p0 < 0 || p0 + n > P.R * P.k) continue;
        const uint8_t* src = pj.w + (size_t)e * pj.expert_bytes + (size_t)u * pj.unit_bytes;
        for (int left = n; left > 0 && !stop;) {
          const int t = dn ? tier_of<true>(left, MAXR_D, P.tier_mode) : tier_of<false>(left, MAXR_U, P.tier_mode);
          left -= min(t, left);
          for (int s = 0; s < pj.S; ++s, ++it) {
            const int slot = it % NST;
            const uint32_t ph = (it / NST) & 1u;
            if (*abort_flag) { stop = true; break; }
            if (it >= (uint32_t)NST && !mbar_wait(&empty[slot], ph ^ 1u, P.timeout_ns)) {
              report(P.status, TFX_ST_TIMEOUT);
              *abort_flag = 1;
              stop = true;
              break;
            }
            if (*abort_flag) { stop = true; break; }
            mbar_arrive_expect_tx(&full[slot], STAGE_B);
            bulk_g2s(ring + (size_t)slot * STAGE_B, src + (size_t)s * STAGE_B, STAGE_B, &full[slot]);
          }
        }
      }
      // Drain: every issued stage must have landed before the block may exit.
      const uint32_t first = it > (uint32_t)NST ? it - NST : 0u;
      for (uint32_t q = first; q < it; ++q) {
        if (!mbar_wait(&full[q % NST], (q / NST) & 1u, P.timeout_ns)) {
          report(P.status, TFX_ST_TIMEOUT);
          break;
        }
      }
    }
  } else {
    // ---------------------------------------------------------------- consumers
    uint32_t it = 0;
    bool dead = false;
    for (int item = blockIdx.x; item < total; item += gridDim.x) {
      const bool dn = item >= n_upc;
      const Proj& pj = dn ? P.pd : P.pu;
      const int li = dn ? item - n_upc : item;
      const int a = li / pj.units, u = li - a * pj.units;
      const int e = r_act[a];
      if (e < 0 || e >= P.E) { if (tid == 0) report(P.status, TFX_ST_SHAPE); continue; }
      const int p0 = r_offs[e], n = r_offs[e + 1] - p0;
      if (n <= 0 || p0 < 0 || p0 + n > P.R * P.k) { if (tid == 0 && n != 0) report(P.status, TFX_ST_SHAPE); continue; }
      if (PH == PH_FUSED && dn) {
        // the expert's h must be complete: wait (bounded) for all of its gate/up items
        if (tid == 0 && !dead) {
          const uint64_t t0 = global_ns();
          while (true) {
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(done_upc + a) : "memory");
            if (v >= P.pu.units) break;
            if (*abort_flag || global_ns() - t0 > P.timeout_ns) {
              report(P.status, TFX_ST_TIMEOUT);
              *abort_flag = 1;
              break;
            }
            __nanosleep(64);
          }
        }
        named_sync(1, NCONS);
        if (*abort_flag) dead = true;
      }
      const uint8_t* X8 = dn ? static_cast<const uint8_t*>(P.h) : static_cast<const uint8_t*>(P.x);
      const uint8_t* XS = dn ? P.hs : P.xs;
      int pos = p0;
      for (int left = n; left > 0;) {
        const int t = dn ? tier_of<true>(left, MAXR_D, P.tier_mode) : tier_of<false>(left, MAXR_U, P.tier_mode);
        const int real = min(t, left);
        named_sync(1, NCONS);
        if (tid < 8) {  // pass rows: real rows, then padding rows that repeat the last real row
          const int src = pos + min(tid, real - 1);
          int row = src;
          if (!dn) {
            row = r_prow[src];
            if (row < 0 || row >= P.R) { report(P.status, TFX_ST_SHAPE); row = 0; }
          }
          prow[tid] = row;
          ppair[tid] = src;
        }
        named_sync(1, NCONS);
        stage_rows<KIND>(X8, XS, pj.K, pj.G, pj.GB, xs_s, xm_s, prow, real, tid);
        named_sync(1, NCONS);
        if (dn) dispatch_pass<KIND, MAXR_D, true>(t, P, pj, ring, full, empty, abort_flag, xs_s, xm_s, prow,
                                                  reinterpret_cast<const uint16_t*>(X8), real, it, dead, epi);
        else dispatch_pass<KIND, MAXR_U, false>(t, P, pj, ring, full, empty, abort_flag, xs_s, xm_s, prow,
                                                reinterpret_cast<const uint16_t*>(X8), real, it, dead, epi);
        named_sync(1, NCONS);

        // ------------------------------------------------------------ epilogue
        if (warp < real && !dead) {
          const int r = warp;
          const int p = ppair[r];
          if (!dn) {
            const int I = P.I;
            const int nn = 32 * u + lane;
            const float g = epi[r * 64 + lane], uu = epi[r * 64 + 32 + lane];
            const float den = __fadd_rn(1.0f, expf(-g));
            const float hv = __fmul_rn(__fdiv_rn(g, den), uu);
            if (P.gu_dbg) {
              P.gu_dbg[(size_t)p * 2 * I + nn] = g;
              P.gu_dbg[(size_t)p * 2 * I + I + nn] = uu;
            }
            if (P.h_dbg) P.h_dbg[(size_t)p * I + nn] = hv;
            if (KIND == TFX_ACT_E4M3) {
              const bool bad = __any_sync(0xffffffffu, isnan(hv) || isinf(hv));
              const uint32_t amax_b = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv)));
              uint32_t sc;
              if (bad) sc = 255u;
              else if (amax_b == 0u) sc = 127u;
              else {
                const int e2 = amax_b >= 0x00800000u ? (int)(amax_b >> 23) - 127 : (31 - __clz((int)amax_b)) - 149;
                sc = (uint32_t)min(max(e2 - 8 + 127, 0), 254);
              }
              const uint32_t code = bad ? 0x7Fu : f32_to_e4m3(__fmul_rn(hv, e8m0_recip_f32(sc)));
              static_cast<uint8_t*>(P.h)[(size_t)p * I + nn] = (uint8_t)code;
              if (lane == 0) P.hs[(size_t)p * (I / 32) + u] = (uint8_t)sc;
            } else {
              static_cast<__nv_bfloat16*>(P.h)[(size_t)p * I + nn] = __float2bfloat16_rn(hv);
            }
          } else {
            const int row = r_prow[p], slot = r_pslot[p];
            if (row >= 0 && row < P.R && slot >= 0 && slot < P.k) {
              float* dst = P.out + ((size_t)row * P.k + slot) * P.H + 64 * u;
              dst[lane] = epi[r * 64 + lane];
              dst[32 + lane] = epi[r * 64 + 32 + lane];
              if (PH == PH_FUSED) {
                // combine (row, block u) in the CTA that writes its row's last slot
                __threadfence();
                int last = 0;
                if (lane == 0) last = atomicAdd(&slots_done[(size_t)row * P.pd.units + u], 1) == r_rowcnt[row] - 1;
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                  __threadfence();
#pragma unroll
                  for (int hh = 0; hh < 2; ++hh) {
                    const int m = 64 * u + 32 * hh + lane;
                    float yv = 0.0f;
                    for (int jj = 0; jj < P.k; ++jj)
                      yv = __fmaf_rn(P.topk_w[(size_t)row * P.k + jj], __ldcg(P.out + ((size_t)row * P.k + jj) * P.H + m), yv);
                    P.y[(size_t)row * P.H + m] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
                    if (P.y32) P.y32[(size_t)row * P.H + m] = yv;
                  }
                }
              }
            } else if (lane == 0) {
              report(P.status, TFX_ST_SHAPE);
            }
          }
        }
        pos += real;
        left -= real;
      }
      if (PH == PH_FUSED && !dn) {  // publish this gate/up item
        __threadfence();
        named_sync(1, NCONS);
        if (tid == 0) atomicAdd(done_upc + a, 1);
      }
    }
  }
  if (PH == PH_FUSED) {
    // the last CTA to finish returns the counters to zero for the next launch
    __syncthreads();
    if (tid == 0) {
      __threadfence();
      const int prev = atomicAdd(P.scratch, 1);
      if (prev == (int)gridDim.x - 1) {
        __threadfence();
        for (int i = 1; i <= P.E; ++i) P.scratch[i] = 0;
        const int nc = P.R * P.pd.units;
        for (int i = 0; i < nc; ++i) slots_done[i] = 0;
        __threadfence();
        P.scratch[0] = 0;
      }
    }
  }
}

// ------------------------------------------------------------------------------ host side

static std::mutex g_mu;

static int dev_sms(int* sms, size_t* optin) {
  int dev;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TFX_ECUDA;
  static int c_sms[64];
  static size_t c_opt[64];
  std::lock_guard<std::mutex> lk(g_mu);
  if (!c_sms[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TFX_ECUDA;
    c_sms[dev] = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return TFX_ECUDA;
    c_opt[dev] = (size_t)v;
  }
  *sms = c_sms[dev];
  *optin = c_opt[dev];
  return TFX_OK;
}

// Ring depth and blocks per SM: the depth (2..6 stages) that keeps the most stage bytes in
// flight per SM, fewer stages breaking ties towards more resident blocks. Chosen once per
// (device, kernel instance, shared-memory shape) and cached, so steady-state launches (and
// launches under stream capture) issue only the kernel.
template <int KIND, int MAXR_U, int MAXR_D, int PH>
static int launch_rows(RowsParams P, int max_items, cudaStream_t st) {
  constexpr int MAXR = ((PH & PH_UPC) && MAXR_U > MAXR_D) || !(PH & PH_DOWN) ? MAXR_U : MAXR_D;
  int sms;
  size_t optin;
  int rc = dev_sms(&sms, &optin);
  if (rc) return rc;
  auto kern = rows_kernel<KIND, MAXR_U, MAXR_D, PH>;
  struct Entry { int key_gb, key_route, nst, nb; size_t smem; };
  static Entry cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TFX_ECUDA;
  Entry ent;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    ent = cache[dev];
    if (ent.nb == 0 || ent.key_gb != P.gbmax || ent.key_route != P.route_ints) {
      RowsParams q = P;
      q.nstage = 6;
      const size_t smax = (size_t)layout_of(q, MAXR).total;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)min(smax, optin)) != cudaSuccess)
        return TFX_ELAUNCH;
      int best = -1, best_nst = 0, best_nb = 0;
      size_t best_smem = 0;
      for (int nst = 2; nst <= 6; ++nst) {
        q.nstage = nst;
        const size_t sm = (size_t)layout_of(q, MAXR).total;
        if (sm > optin) break;
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, NTHREADS, sm) != cudaSuccess) return TFX_ELAUNCH;
        if (nb < 1) break;
        const int score = nb * nst;
        if (score > best || (score == best && nb > best_nb)) {
          best = score;
          best_nst = nst;
          best_nb = nb;
          best_smem = sm;
        }
      }
      if (best_nst == 0) return TFX_EUNSUPPORTED;
      ent = Entry{P.gbmax, P.route_ints, best_nst, best_nb, best_smem};
      cache[dev] = ent;
    }
  }
  P.nstage = ent.nst;
  const int grid = min(max_items, ent.nb * sms);
  if (grid < 1) return TFX_OK;
  if (PH == PH_FUSED) {
    // CTAs of the fused launch wait on one another: launch cooperatively, so that the runtime
    // guarantees every CTA is resident at once (or refuses the launch).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NTHREADS);
    cfg.dynamicSmemBytes = ent.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, P) != cudaSuccess) {
      (void)cudaGetLastError();
      return TFX_ELAUNCH;
    }
    return TFX_OK;
  }
  kern<<<grid, NTHREADS, ent.smem, st>>>(P);
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool dims_ok(const tfx_dims& d) {
  return d.hidden > 0 && d.hidden % 64 == 0 && d.inter > 0 && d.inter % 32 == 0 && d.n_experts >= 1 &&
         d.n_experts <= 1024 && d.top_k >= 1 && d.top_k <= 32 && d.top_k <= d.n_experts &&
         (int64_t)d.hidden * d.inter < (1ll << 31);
}

static Proj proj_of(const tfx_dims& d, bool down, const uint8_t* w) {
  Proj p;
  p.K = down ? d.inter : d.hidden;
  p.S = (p.K + KC - 1) / KC;
  p.G = p.K / 32;
  p.GB = 2 * p.S;
  p.units = down ? d.hidden / 64 : d.inter / 32;
  p.unit_bytes = (size_t)p.S * STAGE_B;
  p.expert_bytes = (size_t)p.units * p.unit_bytes;
  p.w = w;
  return p;
}

size_t packed_gu_bytes(const tfx_dims& d) {
  return (size_t)d.n_experts * (d.inter / 32) * ((d.hidden + KC - 1) / KC) * STAGE_B;
}
size_t packed_d_bytes(const tfx_dims& d) {
  return (size_t)d.n_experts * (d.hidden / 64) * ((d.inter + KC - 1) / KC) * STAGE_B;
}

static int pass_of(const tfx_rows_opts* opts, bool down, int R) {
  int m = opts ? opts->max_pass : 0;
  if (m == 0) {
    if (!down) m = R >= 5 ? 8 : R >= 3 ? 4 : R >= 2 ? 2 : 1;
    else m = R >= 3 ? 4 : R >= 2 ? 2 : 1;
  }
  return m;
}

static int common_args(tfx_dims d, int32_t rows, int32_t kind, const uint8_t* packed, const void* x,
                       const uint8_t* xs, int32_t* status, const tfx_rows_opts* opts, RowsParams& P) {
  if (!dims_ok(d) || rows < 0 || !packed || !status) return TFX_EINVAL;
  if ((int64_t)rows * d.top_k > (1ll << 30)) return TFX_EINVAL;
  if (kind != TFX_ACT_E4M3 && kind != TFX_ACT_BF16) return TFX_EINVAL;
  if (rows > 0 && (!x || !aligned16(x) || !aligned16(packed))) return TFX_EINVAL;
  if (kind == TFX_ACT_E4M3 && rows > 0 && !xs) return TFX_EINVAL;
  if (opts && (opts->tier_mode < 0 || opts->tier_mode > 1 || opts->timeout_ns < 0)) return TFX_EINVAL;
  P = RowsParams{};
  P.H = d.hidden;
  P.I = d.inter;
  P.E = d.n_experts;
  P.k = d.top_k;
  P.R = rows;
  P.pu = proj_of(d, false, packed);
  P.pd = proj_of(d, true, packed + packed_gu_bytes(d));
  P.x = x;
  P.xs = xs;
  P.status = status;
  P.tier_mode = opts ? opts->tier_mode : 0;
  P.timeout_ns = (opts && opts->timeout_ns > 0) ? (uint64_t)opts->timeout_ns : kDefaultTimeoutNs;
  return TFX_OK;
}

template <int KIND, int PH>
static int dispatch(const RowsParams& P, int mu, int md, int max_items, cudaStream_t st) {
  if (PH == PH_UPC) {
    switch (mu) {
      case 1: return launch_rows<KIND, 1, 1, PH_UPC>(P, max_items, st);
      case 2: return launch_rows<KIND, 2, 1, PH_UPC>(P, max_items, st);
      case 4: return launch_rows<KIND, 4, 1, PH_UPC>(P, max_items, st);
      case 8: return launch_rows<KIND, 8, 1, PH_UPC>(P, max_items, st);
    }
  } else if (PH == PH_DOWN) {
    switch (md) {
      case 1: return launch_rows<KIND, 1, 1, PH_DOWN>(P, max_items, st);
      case 2: return launch_rows<KIND, 1, 2, PH_DOWN>(P, max_items, st);
      case 4: return launch_rows<KIND, 1, 4, PH_DOWN>(P, max_items, st);
    }
  } else {
    if (mu == 1 && md == 1) return launch_rows<KIND, 1, 1, PH_FUSED>(P, max_items, st);
    if (mu == 2 && md == 2) return launch_rows<KIND, 2, 2, PH_FUSED>(P, max_items, st);
    if (mu == 4 && md == 4) return launch_rows<KIND, 4, 4, PH_FUSED>(P, max_items, st);
    if (mu == 8 && md == 4) return launch_rows<KIND, 8, 4, PH_FUSED>(P, max_items, st);
  }
  return TFX_EINVAL;
}

}  // namespace tfx

using namespace tfx;

extern "C" int tfx_xp_upc_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                               const uint8_t* x_scale, const tfx_route* rt, void* h, uint8_t* h_scale,
                               float* gu_dbg, float* h_dbg, int32_t* status, const tfx_rows_opts* opts,
                               void* stream) {
  RowsParams P;
  int rc = common_args(d, rows, act_kind, packed, x, x_scale, status, opts, P);
  if (rc) return rc;
  if (!rt || !rt->offs || !rt->pair_row || !rt->pair_slot || !rt->active || !rt->n_active) return TFX_EINVAL;
  const int mu = pass_of(opts, false, rows);
  if (!(mu == 1 || mu == 2 || mu == 4 || mu == 8)) return TFX_EINVAL;
  if (rows == 0) return TFX_OK;
  if (!h || (act_kind == TFX_ACT_E4M3 && !h_scale)) return TFX_EINVAL;
  P.offs = const_cast<int32_t*>(rt->offs);
  P.pair_row = const_cast<int32_t*>(rt->pair_row);
  P.pair_slot = const_cast<int32_t*>(rt->pair_slot);
  P.active = const_cast<int32_t*>(rt->active);
  P.n_active = const_cast<int32_t*>(rt->n_active);
  P.h = h;
  P.hs = h_scale;
  P.gu_dbg = gu_dbg;
  P.h_dbg = h_dbg;
  P.gbmax = P.pu.GB;
  const int max_items = min(rows * d.top_k, d.n_experts) * P.pu.units;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch<TFX_ACT_E4M3, PH_UPC>(P, mu, 1, max_items, st);
  return dispatch<TFX_ACT_BF16, PH_UPC>(P, mu, 1, max_items, st);
}

extern "C" int tfx_xp_down_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* h,
                                const uint8_t* h_scale, const tfx_route* rt, float* out, int32_t* status,
                                const tfx_rows_opts* opts, void* stream) {
  RowsParams P;
  int rc = common_args(d, rows, act_kind, packed, h, h_scale, status, opts, P);
  if (rc) return rc;
  if (!rt || !rt->offs || !rt->pair_row || !rt->pair_slot || !rt->active || !rt->n_active) return TFX_EINVAL;
  const int md = pass_of(opts, true, rows);
  if (!(md == 1 || md == 2 || md == 4)) return TFX_EINVAL;
  if (rows == 0) return TFX_OK;
  if (!out) return TFX_EINVAL;
  P.offs = const_cast<int32_t*>(rt->offs);
  P.pair_row = const_cast<int32_t*>(rt->pair_row);
  P.pair_slot = const_cast<int32_t*>(rt->pair_slot);
  P.active = const_cast<int32_t*>(rt->active);
  P.n_active = const_cast<int32_t*>(rt->n_active);
  P.h = const_cast<void*>(h);
  P.hs = const_cast<uint8_t*>(h_scale);
  P.out = out;
  P.gbmax = P.pd.GB;
  const int max_items = min(rows * d.top_k, d.n_experts) * P.pd.units;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch<TFX_ACT_E4M3, PH_DOWN>(P, 1, md, max_items, st);
  return dispatch<TFX_ACT_BF16, PH_DOWN>(P, 1, md, max_items, st);
}

extern "C" size_t tfx_xp_moe_rows_scratch_bytes(tfx_dims d, int32_t rows) {
  if (!dims_ok(d) || rows < 0) return 0;
  return sizeof(int32_t) * ((size_t)2 + d.n_experts + (size_t)rows * (d.hidden / 64));
}

extern "C" int tfx_xp_moe_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                               const uint8_t* x_scale, const int32_t* ids, const float* topk_w, int32_t* offs,
                               int32_t* pair_row, int32_t* pair_slot, int32_t* active, int32_t* n_active, void* h,
                               uint8_t* h_scale, float* out, uint16_t* y, float* y_f32_dbg, int32_t* scratch,
                               int32_t* status, const tfx_rows_opts* opts, void* stream) {
  RowsParams P;
  int rc = common_args(d, rows, act_kind, packed, x, x_scale, status, opts, P);
  if (rc) return rc;
  if ((int64_t)rows * d.top_k > FUSED_MAX_PAIRS) return TFX_EUNSUPPORTED;
  const int mu = pass_of(opts, false, rows);
  const int md = min(pass_of(opts, true, rows), 4);  // the down pass stops at 4 rows
  if (!((mu == 1 && md == 1) || (mu == 2 && md == 2) || (mu == 4 && md == 4) || (mu == 8 && md == 4)))
    return TFX_EINVAL;
  if (!offs || !active || !n_active || !scratch || (reinterpret_cast<uintptr_t>(scratch) & 3u)) return TFX_EINVAL;
  if (rows == 0) return TFX_OK;
  if (!ids || !topk_w || !pair_row || !pair_slot || !h || !out || !y || (act_kind == TFX_ACT_E4M3 && !h_scale))
    return TFX_EINVAL;
  P.ids = ids;
  P.topk_w = topk_w;
  P.offs = offs;
  P.pair_row = pair_row;
  P.pair_slot = pair_slot;
  P.active = active;
  P.n_active = n_active;
  P.h = h;
  P.hs = h_scale;
  P.out = out;
  P.y = y;
  P.y32 = y_f32_dbg;
  P.scratch = scratch;
  P.gbmax = max(P.pu.GB, P.pd.GB);
  P.route_ints = 3 * d.n_experts + 2 + 3 * rows * d.top_k + rows;
  const int max_items = min(rows * d.top_k, d.n_experts) * (P.pu.units + P.pd.units);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch<TFX_ACT_E4M3, PH_FUSED>(P, mu, md, max_items, st);
  return dispatch<TFX_ACT_BF16, PH_FUSED>(P, mu, md, max_items, st);
}

// ------------------------------------------------------------------------------ no-alloc variant
// The one-launch layer for callers that cannot allocate device memory themselves: its
// completion counters live in a buffer compiled into the library instead of caller scratch.
namespace tfx {

// Capacity of the built-in counter buffer, in int32 words (64 KiB on every device that
// loads the library, held until the process exits).
constexpr int NOALLOC_SCRATCH_INTS = 16384;
static __device__ __align__(256) int32_t g_noalloc_scratch[NOALLOC_SCRATCH_INTS];

// Device address of g_noalloc_scratch per device, looked up once with that device current.
// (In host code the array's name is only a host-side stand-in, never a device address.)
static int32_t* g_noalloc_ptr[64];

static int noalloc_scratch(int32_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TFX_ECUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_noalloc_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      return TFX_ECUDA;
    }
    g_noalloc_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_noalloc_ptr[dev];
  return TFX_OK;
}

}  // namespace tfx

extern "C" int tfx_xp_moe_rows_noalloc(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed,
                                       const void* x, const uint8_t* x_scale, const int32_t* ids,
                                       const float* topk_w, int32_t* offs, int32_t* pair_row, int32_t* pair_slot,
                                       int32_t* active, int32_t* n_active, void* h, uint8_t* h_scale, float* out,
                                       uint16_t* y, float* y_f32_dbg, int32_t* status, const tfx_rows_opts* opts,
                                       void* stream) {
  const size_t need = tfx_xp_moe_rows_scratch_bytes(d, rows) / sizeof(int32_t);
  if (need > (size_t)NOALLOC_SCRATCH_INTS) return TFX_EUNSUPPORTED;  // beyond the built-in buffer
  int32_t* scratch = nullptr;
  if (need > 0 && rows > 0) {
    const int rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    // the counters must start at zero; a previous call on this device may have stopped early
    if (cudaMemsetAsync(scratch, 0, need * sizeof(int32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess) {
      (void)cudaGetLastError();
      return TFX_ELAUNCH;
    }
  } else {
    scratch = reinterpret_cast<int32_t*>(16);  // never touched: zero rows or arguments rejected below
  }
  return tfx_xp_moe_rows(d, rows, act_kind, packed, x, x_scale, ids, topk_w, offs, pair_row, pair_slot, active,
                         n_active, h, h_scale, out, y, y_f32_dbg, scratch, status, opts, stream);
}
