// tfx_rows.cuh -- the expert-major "rows" engine for launches of few rows per expert (decode):
// gate/up (+ SwiGLU + activation quantiser), down, and the whole layer fused in one launch.
// Included by the translation units that instantiate it (one per activation format and
// phase, so that they compile in parallel) and by tfx_rows.cu, which holds the C entry points.
//
// Method: "dsv41 metal: decode experts decode an expert's weights once for all of its rows"
// (TensorFold PR #2983). A work item is (active expert, block of outputs). Its weights are
// streamed once per pass; every 32-group is decoded once and applied to every row of the pass
// (pass sized by the rows left; padding rows, when a caller asks for padded passes, repeat the
// last real row, are computed and never written). Each row's accumulators follow the fixed
// order of "What this changes": per group a sequential fma chain of the 32 unscaled products
// from +0 in k order, one scaled fma into accumulator (group mod 8), then the eight-way tree.
//
// GB300 mapping:
//   * one producer warp streams 17,408-byte stages (64 weight rows x 512 k of codes, then their
//     scales: contiguous in the packed layout) into a ring of shared-memory slots with
//     cp.async.bulk + mbarrier (every wait bounded);
//   * consumer warps: lane (t & 7) of an octet owns accumulator lane j = group mod 8 of its
//     output columns, so the eight-way tree is three xor-shuffles. A lane handles groups j and
//     j + 8 of each stage. Kernels whose passes hold at most 2 rows run 8 consumer warps (two
//     columns a lane, two CTAs an SM); kernels with longer passes run 16 consumer warps (one
//     column a lane, one CTA an SM), so that the fma-bound passes of many rows have four
//     consumer warps per scheduler and at most 104 registers a thread;
//   * E2M1 codes decode with cvt.rn.f16x2.e2m1x2; activations sit in shared memory as f16
//     (exact for E4M3; bf16 rows are shifted per 32-group by a power of two so that they are
//     exact in f16, with an exact fp32 fallback for groups that do not fit); the chain runs on
//     fma.rn.f32.f16 (fp32 accumulate, one rounding per step).
//   * The fused layer launch (cooperative: all CTAs resident) computes the row lists in shared
//     memory in every CTA and hands out work units of one pass each, pass-major: first every
//     expert's first gate/up pass, then the second passes, ..., then the down passes in the
//     same order (each waits, bounded, for its expert's gate/up units). A CTA's consecutive
//     units then mostly share their rows, whose staged activations it keeps. Each (row,
//     64-output block) is combined in the CTA whose down unit completes the row's last slot.
//     Completion counters live in caller scratch; each counter's last user returns it to zero.
#pragma once
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
constexpr int MAX_NSTAGE = 8;
constexpr int FUSED_MAX_PAIRS = 256;
constexpr int MAX_PASS_U = 8;                    // longest gate/up pass
constexpr int MAX_PASS_D = 4;                    // longest down pass
constexpr int QD = 4;                            // claimed-item queue depth (fused)

enum { PH_UPC = 1, PH_DOWN = 2, PH_FUSED = 3 };

// Shape of a kernel instance whose passes hold at most MAXR rows.
template <int MAXR>
struct Cfg {
  static constexpr int NCW = MAXR <= 2 ? 8 : 16;     // consumer warps
  static constexpr int COLS = 64 / (NCW * 4);        // output columns per consumer lane
  static constexpr int NT = NCW * kWarp + 3 * kWarp;  // + producer, stager and epilogue warps
  static constexpr int MINB = MAXR <= 2 ? 2 : 1;     // resident CTAs per SM
  // registers a thread may take with MINB CTAs of NT threads resident: each of the SM's four
  // schedulers holds a quarter of the 65,536 registers and up to ceil(warps / 4) warps of a
  // CTA (whole 8-register steps)
  static constexpr int MAXREG = (16384 / (MINB * ((NT / kWarp + 3) / 4) * kWarp)) / 8 * 8;
  static constexpr int W_PROD = NCW, W_HELP = NCW + 1, W_EPI = NCW + 2;
};

struct Proj {
  int K, S, G, GB, units;  // reduction length, stages, groups, group blocks of 8 (= 2S), items/expert
  size_t unit_bytes, expert_bytes;
  const uint8_t* w;
};

struct RowsParams {
  int H, I, E, k, R;
  Proj pu, pd;
  int cap_u, cap_d;     // longest pass of gate/up and of down (rows)
  int nstage;
  int nxb;              // activation buffers in shared memory (2: the next pass stages while this one runs)
  int use_raw;          // 1: activation rows arrive by bulk copy into a shared-memory raw buffer
  int raw_row, raw_sc;  // raw buffer bytes per row (128-aligned) and per row of scales (16-aligned)
  int sc_tma_u, sc_tma_d;  // scales of gate/up (x) / down (h) rows come by bulk copy too
  int gbmax;            // group blocks allotted per activation row in shared memory
  int route_ints;       // shared-memory ints of the in-kernel route and pass lists (fused)
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
  int32_t* scratch;     // fused: [0] unused, [1] work counter, [2..E+1] gate/up units done per
                        //        active expert, [E+2..2E+1] down units past their wait per active
                        //        expert, then [R][H/64] slots written per (row, block)
  int32_t* status;
  int tier_mode;        // 0: passes of min(rows left, cap); 1: every pass at cap; 2: the pages' tiers
  uint64_t timeout_ns;
};

// Shared-memory ints of the fused launch's row lists and pass lists (nw: warps of the CTA).
__host__ __device__ inline int fused_route_ints(int E, int R, int k, int nw) {
  const int P = R * k;
  return 3 * E + 2 + 3 * P + R + 2 * nw + 3 * P + 2;
}

// ---------------------------------------------------------------- shared-memory layout
struct Layout {
  int bars, ctrl, pdesc, epi, route, ring, xs, xm, xs_stride, xm_stride, raw, total;
};
__host__ __device__ inline Layout layout_of(const RowsParams& p, int maxr) {
  Layout L;
  L.bars = 0;      // full[8], empty[8], xfull[2], xempty[2], efull[2], eempty[2], rawfull, qfull[4], qempty[4]
  L.ctrl = 384;    // abort flag, then the claimed-item queue ids
  L.pdesc = 448;   // two pass descriptors: prow[8], ppair[8]
  L.epi = 640;     // two float [8][64] result buffers
  L.route = 4736;  // fused: ints
  L.ring = (L.route + 4 * p.route_ints + 127) & ~127;
  L.xs = L.ring + p.nstage * STAGE_B;
  L.xs_stride = maxr * p.gbmax * 512;
  L.xm = L.xs + p.nxb * L.xs_stride;
  L.xm_stride = maxr * p.gbmax * 8 * 4;
  L.raw = (L.xm + p.nxb * L.xm_stride + 127) & ~127;
  L.total = L.raw + (p.use_raw ? maxr * (p.raw_row + p.raw_sc) : 0);
  return L;
}

// Rows of the pass that starts with `left` rows of an item left, for a pass cap and tier mode:
// 0 -> min(left, cap); 1 -> cap (padded); 2 -> the pages' tiers (gate/up 8 if >= 7 rows left, 6
// if >= 5, 4 if >= 3, else 2 or 1; down 4 if >= 3, else 2 or 1), capped.
__device__ __forceinline__ int tier_of(int left, int cap, int mode, bool down) {
  int t;
  if (mode == 1) t = cap;
  else if (mode == 2) {
    if (!down) t = left >= 7 ? 8 : left >= 5 ? 6 : left >= 3 ? 4 : left >= 2 ? 2 : 1;
    else t = left >= 3 ? 4 : left >= 2 ? 2 : 1;
  } else t = left;
  return t > cap ? cap : t;
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
static __device__ __noinline__ float chain_bf16_exact(uint4 codes, const uint16_t* xrow, int g) {
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

// Stage the activation rows of one pass into the f16 activation buffer (the NT threads of the
// calling role). Row r is read at X8 + row(r) * xstride and its scales at XS + row(r) * sstride,
// where row(r) = prow[r] for rows in global memory, or r for rows already bulk-copied into
// shared memory (FROM_SMEM). Global loads go through L2 (the rows may have been written by
// other CTAs of the same launch) and are issued in batches so that many are in flight. Groups
// from G up to the stage boundary are zero with multiplier 1, so that lanes past the end of the
// reduction add +0 to their accumulators.
// X32 (bf16 only): the rows are kept as fp32 values, unshifted (multiplier 1), in chunks of
// 8 values at twice the f16 offsets; no group needs the exact fallback then.
template <int KIND, bool FROM_SMEM, bool SC_SMEM, bool X32 = false>
__device__ void stage_rows(const uint8_t* __restrict__ X8, size_t xstride, const uint8_t* __restrict__ XS,
                           size_t sstride, int K, int G, int GB, uint8_t* xs_s, float* xm_s, const int* prow,
                           int real, int tid, int NT) {
  const int nch = K / 8;          // chunks of 8 elements with data
  const int nall = GB * 8 * 4;    // chunks up to the stage boundary
  constexpr int BATCH = 8;
  if (KIND == TFX_ACT_E4M3) {
    const int gall = GB * 8;
    for (int r = 0; r < real; ++r) {
      const uint8_t* xrow = X8 + (size_t)(FROM_SMEM ? r : prow[r]) * xstride;
      for (int c0 = tid; c0 < nall; c0 += BATCH * NT) {
        uint2 v[BATCH];
#pragma unroll
        for (int q = 0; q < BATCH; ++q) {
          const int c = c0 + q * NT;
          v[q] = make_uint2(0u, 0u);
          if (c < nch)
            v[q] = FROM_SMEM ? *reinterpret_cast<const uint2*>(xrow + 8 * c)
                             : __ldcg(reinterpret_cast<const uint2*>(xrow + 8 * c));
        }
#pragma unroll
        for (int q = 0; q < BATCH; ++q) {
          const int c = c0 + q * NT;
          if (c >= nall) break;
          uint4 o;
          o.x = e4m3x2_to_f16x2(v[q].x);
          o.y = e4m3x2_to_f16x2(v[q].x >> 16);
          o.z = e4m3x2_to_f16x2(v[q].y);
          o.w = e4m3x2_to_f16x2(v[q].y >> 16);
          *reinterpret_cast<uint4*>(xs_s + xoff(r, c >> 2, c & 3, GB)) = o;
        }
      }
      const uint8_t* srow = XS + (size_t)(SC_SMEM ? r : prow[r]) * sstride;
      for (int g0 = tid; g0 < gall; g0 += BATCH * NT) {
        uint32_t sv[BATCH];
#pragma unroll
        for (int q = 0; q < BATCH; ++q) {
          const int g = g0 + q * NT;
          sv[q] = 127u;
          if (g < G) sv[q] = SC_SMEM ? srow[g] : __ldcg(srow + g);
        }
#pragma unroll
        for (int q = 0; q < BATCH; ++q) {
          const int g = g0 + q * NT;
          if (g >= gall) break;
          xm_s[r * gall + g] = g < G ? e8m0_to_f32(sv[q]) : 1.0f;
        }
      }
    }
  } else {
    // bf16: one thread converts one 32-group with a power-of-two shift 2^sigma that maps the
    // group's largest magnitude into [2^15, 2^16). The group is exact in f16 and its chain
    // equals the unshifted fp32 chain times 2^sigma when every finite nonzero value has
    // exponent in [e_max - 32, e_max], e_max <= 119 and e_min >= -141 (products and partial
    // sums then stay in fp32's normal range, or on its subnormal grid, on both sides).
    // Otherwise the multiplier is 0 and the exact fallback runs for that group.
    const int gall = GB * 8;
    const int total = real * gall;
    for (int i = tid; i < total; i += NT) {
      const int r = i / gall, g = i - r * gall;
      uint4 v[4];  // the group's 32 bf16 values, element 2j in the low half of word j
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = make_uint4(0u, 0u, 0u, 0u);
      if (g < G) {
        const uint8_t* src = X8 + (size_t)(FROM_SMEM ? r : prow[r]) * xstride + 64 * g;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          v[q] = FROM_SMEM ? *reinterpret_cast<const uint4*>(src + 16 * q)
                           : __ldcg(reinterpret_cast<const uint4*>(src + 16 * q));
      }
      const uint32_t* wv = reinterpret_cast<const uint32_t*>(v);
      if (X32) {
#pragma unroll
        for (int tc = 0; tc < 4; ++tc) {
          uint4 o0, o1;
          o0.x = wv[4 * tc] << 16;
          o0.y = wv[4 * tc] & 0xFFFF0000u;
          o0.z = wv[4 * tc + 1] << 16;
          o0.w = wv[4 * tc + 1] & 0xFFFF0000u;
          o1.x = wv[4 * tc + 2] << 16;
          o1.y = wv[4 * tc + 2] & 0xFFFF0000u;
          o1.z = wv[4 * tc + 3] << 16;
          o1.w = wv[4 * tc + 3] & 0xFFFF0000u;
          uint4* dst = reinterpret_cast<uint4*>(xs_s + 2 * xoff(r, g, tc, GB));
          dst[0] = o0;
          dst[1] = o1;
        }
        xm_s[r * gall + g] = 1.0f;
        continue;
      }
      // the exponents of the largest and of the smallest nonzero finite magnitude (magnitude bits
      // order like the values); NaN, Inf and zeros take no part
      uint32_t mxb = 0u, mnb = 0xFFFFu;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const uint32_t mag = (wv[j >> 1] >> (16 * (j & 1))) & 0x7FFFu;
        const bool fin = mag - 1u < 0x7F7Fu;  // nonzero, exponent field below 255
        mxb = max(mxb, fin ? mag : 0u);
        mnb = min(mnb, fin ? mag : 0xFFFFu);
      }
      int emax = -1000, emin = 1000;
      if (mxb) {
        const uint32_t ex = mxb >> 7, en = mnb >> 7;
        emax = ex ? (int)ex - 127 : (31 - __clz((int)(mxb & 0x7Fu))) - 133;
        emin = en ? (int)en - 127 : (31 - __clz((int)(mnb & 0x7Fu))) - 133;
      }
      int sigma = 0;
      bool safe = true;
      if (emax > -1000) {
        sigma = 15 - emax;
        safe = (emax <= 119) && (emin >= -141) && (emax - emin <= 32);
      }
      const int s1 = min(max(sigma, -126), 127), s2 = sigma - s1;  // 2^sigma as two exact factors
      const float f1 = __uint_as_float((uint32_t)(127 + s1) << 23);
      const float f2 = __uint_as_float((uint32_t)(127 + s2) << 23);
#pragma unroll
      for (int tc = 0; tc < 4; ++tc) {
        uint32_t o[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t two = wv[4 * tc + q];
          float lo = __uint_as_float(two << 16), hi = __uint_as_float(two & 0xFFFF0000u);
          if (safe) {
            lo = __fmul_rn(__fmul_rn(lo, f1), f2);
            hi = __fmul_rn(__fmul_rn(hi, f1), f2);
          }
          const __half2 h2 = __floats2half2_rn(lo, hi);
          o[q] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(xs_s + xoff(r, g, tc, GB)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      float m = 0.0f;  // 0 marks the exact fallback
      if (g >= G) m = 1.0f;
      else if (safe) {
        const int ns = -sigma;  // 2^-sigma, possibly subnormal (exact)
        m = ns >= -126 ? __uint_as_float((uint32_t)(127 + ns) << 23) : __uint_as_float(0x00400000u >> (-127 - ns));
      }
      xm_s[r * gall + g] = m;
    }
  }
}

// Row lists of a small launch, computed in shared memory (fused layer): per-pair expert (or -1
// if left out), per-expert counts -> offsets, active experts, stable positions, per-row slot
// counts; then the pass lists of both projections (pass-major: every expert's first pass, then
// every second pass, ...). All NT threads take part. Ints used: fused_route_ints(E, R, k).
struct SRoute {
  int *offs, *prow, *pslot, *act, *rowcnt, *ev, *cnt, *nact;
  int *plist_u, *plist_d;  // pass lists: a | start << 10 | real << 18 | t << 22
  uint16_t *np_u, *np_d;   // passes per active expert
  int *nlist;              // [0] gate/up passes, [1] down passes
};
__device__ __forceinline__ int pack_pass(int a, int start, int real, int t) {
  return a | (start << 10) | (real << 18) | (t << 22);
}

// Passes of an expert with n rows and the rows of its b-th pass.
__device__ __forceinline__ int passes_of(int n, int cap, int mode, bool down) {
  if (mode != 2) return (n + cap - 1) / cap;
  int np = 0;
  for (int left = n; left > 0; ++np) left -= min(tier_of(left, cap, mode, down), left);
  return np;
}
__device__ __forceinline__ void pass_rows(int n, int b, int cap, int mode, bool down, int& start, int& real, int& t) {
  if (mode != 2) {
    start = b * cap;
    real = min(cap, n - start);
    t = mode == 1 ? cap : real;
    return;
  }
  int left = n;
  start = 0;
  for (int i = 0; i < b; ++i) {
    const int r = min(tier_of(left, cap, mode, down), left);
    start += r;
    left -= r;
  }
  t = tier_of(left, cap, mode, down);
  real = min(t, left);
}

template <int NT>
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
  constexpr int NW = NT / 32;
  int* wsum = rt.rowcnt + p.R;                               // 2 * NW
  rt.plist_u = wsum + 2 * NW;                                // P
  rt.plist_d = rt.plist_u + P;                               // P
  rt.np_u = reinterpret_cast<uint16_t*>(rt.plist_d + P);     // P halves (>= active experts)
  rt.np_d = rt.np_u + P;                                     // P halves
  rt.nlist = rt.plist_d + 2 * P;                             // 2
  for (int i = tid; i < E; i += NT) rt.cnt[i] = 0;
  for (int i = tid; i < p.R; i += NT) rt.rowcnt[i] = 0;
  for (int q = tid; q < P; q += NT) rt.prow[q] = p.ids[q];  // ids, staged (prow is free until the scatter)
  __syncthreads();
  int bad = 0;
  for (int q = tid; q < P; q += NT) {
    const int e = rt.prow[q];
    int v = e;
    if (e < 0 || e >= E) { v = -1; bad |= TFX_ST_RANGE; }
    else {
      for (int jj = q - q % k; jj < q; ++jj)
        if (rt.prow[jj] == e) { v = -1; bad |= TFX_ST_DUP; break; }
    }
    rt.ev[q] = v;
    if (v >= 0) {
      atomicAdd(&rt.cnt[v], 1);
      atomicAdd(&rt.rowcnt[q / k], 1);
    }
  }
  if (bad && blockIdx.x == 0) report(p.status, bad);
  __syncthreads();
  // Exclusive scan of the counts and of the active flags over the whole block: every thread
  // takes a contiguous run of experts, the warps scan the run totals, warp 0 scans the warp
  // totals.
  const int lane = tid & 31, warp = tid >> 5;
  const int per = (E + NT - 1) / NT;
  const int e0 = min(E, tid * per), e1 = min(E, e0 + per);
  int c_run = 0, a_run = 0;
  for (int e = e0; e < e1; ++e) {
    const int c = rt.cnt[e];
    c_run += c;
    a_run += c > 0;
  }
  int ci = c_run, ai = a_run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, ci, o), w = __shfl_up_sync(0xffffffffu, ai, o);
    if (lane >= o) { ci += v; ai += w; }
  }
  if (lane == 31) {
    wsum[warp] = ci;
    wsum[NW + warp] = ai;
  }
  __syncthreads();
  if (warp == 0) {
    const int c = lane < NW ? wsum[lane] : 0, a = lane < NW ? wsum[NW + lane] : 0;
    int cs = c, as = a;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, cs, o), w = __shfl_up_sync(0xffffffffu, as, o);
      if (lane >= o) { cs += v; as += w; }
    }
    __syncwarp();
    if (lane < NW) {
      wsum[lane] = cs - c;
      wsum[NW + lane] = as - a;
    }
    if (lane == 31) {
      rt.offs[E] = cs;
      *rt.nact = as;
    }
  }
  __syncthreads();
  {
    int off = wsum[warp] + ci - c_run, na = wsum[NW + warp] + ai - a_run;
    for (int e = e0; e < e1; ++e) {
      const int c = rt.cnt[e];
      rt.offs[e] = off;
      rt.cnt[e] = off;  // from here on: the expert's next free position
      off += c;
      if (c > 0) rt.act[na++] = e;
    }
  }
  __syncthreads();
  if (warp == 0) {
    // Stable scatter, 32 pairs at a time: a pair's position is its expert's cursor plus the
    // number of earlier lanes of the chunk with the same expert.
    for (int q0 = 0; q0 < P; q0 += 32) {
      const int q = q0 + lane;
      const int e = q < P ? rt.ev[q] : -2;
      const unsigned m = __match_any_sync(0xffffffffu, e);
      if (e >= 0) {
        const int pos = rt.cnt[e] + __popc(m & ((1u << lane) - 1u));
        rt.prow[pos] = q / k;
        rt.pslot[pos] = q - (q / k) * k;
      }
      __syncwarp();
      if (e >= 0 && lane == __ffs(m) - 1) rt.cnt[e] += __popc(m);
      __syncwarp();
    }
  } else if (warp == 1 || warp == 2) {
    // Pass lists (warp 1: gate/up, warp 2: down), pass-major.
    const bool down = warp == 2;
    const int cap = down ? p.cap_d : p.cap_u;
    int* list = down ? rt.plist_d : rt.plist_u;
    uint16_t* np = down ? rt.np_d : rt.np_u;
    const int na = *rt.nact;
    int maxp = 0;
    for (int a = lane; a < na; a += 32) {
      const int e = rt.act[a];
      const int v = passes_of(rt.offs[e + 1] - rt.offs[e], cap, p.tier_mode, down);
      np[a] = (uint16_t)v;
      maxp = max(maxp, v);
    }
    maxp = __reduce_max_sync(0xffffffffu, maxp);
    __syncwarp();
    int count = 0;
    for (int b = 0; b < maxp; ++b) {
      for (int a0 = 0; a0 < na; a0 += 32) {
        const int a = a0 + lane;
        const bool has = a < na && np[a] > b;
        const unsigned m = __ballot_sync(0xffffffffu, has);
        if (has) {
          const int e = rt.act[a];
          int start, real, t;
          pass_rows(rt.offs[e + 1] - rt.offs[e], b, cap, p.tier_mode, down, start, real, t);
          list[count + __popc(m & ((1u << lane) - 1u))] = pack_pass(a, start, real, t);
        }
        count += __popc(m);
      }
    }
    if (lane == 0) rt.nlist[down ? 1 : 0] = count;
  }
  __syncthreads();
}

// Loads from shared memory by 32-bit shared-window address (keeps per-row addresses in one
// register each).
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float4 lds128f(uint32_t a) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ float lds32f(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
  return v;
}

// ---------------------------------------------------------------- one pass of T rows
// Barriers of the shared-memory handoffs between the roles.
struct Bars {
  uint64_t *full, *empty;   // weight ring: producer -> consumers, consumers -> producer
  uint64_t *xfull, *xempty; // activation buffers: helper -> consumers, consumers -> helper
  uint64_t *efull, *eempty; // result buffers: consumers -> helper, helper -> consumers
};

// Bounded wait whose outcome is uniform across the calling warp; on failure the block is
// marked aborted (the caller then skips its remaining work and waits).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const RowsParams& P,
                                          volatile int* abort_flag, bool& dead) {
  if (dead) return false;
  // a completed phase needs neither the abort flag nor the bounded loop
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  bool ok = (*abort_flag == 0) && mbar_wait(bar, parity, P.timeout_ns);
  ok = __all_sync(0xffffffffu, ok);
  if (!ok) {
    dead = true;
    if ((threadIdx.x & 31) == 0) {
      if (*abort_flag == 0) report(P.status, TFX_ST_TIMEOUT);
      *abort_flag = 1;
    }
  }
  return ok;
}

// E8M0 code -> fp32 bits (those of e8m0_to_f32), a table read through L1 by the consumers.
struct E8m0Table {
  uint32_t v[256];
  constexpr E8m0Table() : v() {
    for (int c = 0; c < 256; ++c) v[c] = c == 0 ? 0x00400000u : c == 255 ? 0x7FC00000u : (uint32_t)c << 23;
  }
};
static __device__ const E8m0Table e8m0_table = E8m0Table();
__device__ __forceinline__ float e8m0_lookup(uint32_t code) { return __uint_as_float(__ldg(e8m0_table.v + code)); }

// Consumers: consume the pass's S weight stages against activation buffer xs_s/xm_s, release
// the buffer, then hand the eight-way-tree results of every real row to the epilogue warp in
// epi[r][0..63] (column c of the stage's 64 weight rows at c). A lane owns COLS columns: o and,
// with two columns, 32 + o, where o = 4 * warp + lane / 8.
template <int KIND, int T, int COLS, bool X32 = false>
__device__ __forceinline__ void run_pass(const RowsParams& P, const Proj& pj, uint8_t* ring, const Bars& B,
                                         int bx, int be, uint32_t eph, bool ewait, volatile int* abort_flag,
                                         const uint8_t* xs_s, const float* xm_s, const int* prow,
                                         const uint16_t* xraw, int real, uint32_t& it, bool& dead, float* epi) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = lane & 7, o = (warp << 2) | (lane >> 3);
  int col[COLS];
#pragma unroll
  for (int c = 0; c < COLS; ++c) col[c] = o + 32 * c;
  const int NST = P.nstage, GB = pj.GB;
  float acc[COLS][T];
  // shared-window addresses of each row's activations (lane's chunk j) and group multipliers:
  // the buffer holds all T rows of the pass (padding rows staged as copies of the last real
  // row), so row r sits at a fixed offset from row 0
  const uint32_t xs_a = smem_addr(xs_s) + (X32 ? 2 : 1) * j * 16, xm_a = smem_addr(xm_s) + 4 * j;
  const uint32_t xrs = (X32 ? 2 : 1) * GB * 512, xms = 4 * GB * 8;  // bytes per row
#pragma unroll
  for (int r = 0; r < T; ++r)
#pragma unroll
    for (int c = 0; c < COLS; ++c) acc[c][r] = 0.0f;
  // ring position, advanced incrementally (no division per stage)
  int slot = (int)(it % (uint32_t)NST);
  uint32_t ph = (it / (uint32_t)NST) & 1u;
  for (int s = 0; s < pj.S; ++s, ++it, slot = slot + 1 == NST ? 0 : slot + 1, ph ^= slot == 0 ? 1u : 0u) {
    if (warp_wait(&B.full[slot], ph, P, abort_flag, dead)) {
      const uint8_t* tile = ring + (size_t)slot * STAGE_B;
      const uint8_t* sc = tile + TROWS * CODE_B;
      uint4 cA[COLS], cB[COLS];
      float sA[COLS], sB[COLS];
#pragma unroll
      for (int c = 0; c < COLS; ++c) {
        cA[c] = *reinterpret_cast<const uint4*>(tile + col[c] * CODE_B + 16 * j);
        cB[c] = *reinterpret_cast<const uint4*>(tile + col[c] * CODE_B + 128 + 16 * j);
        sA[c] = e8m0_lookup(sc[col[c] * GPS + j]);
        sB[c] = e8m0_lookup(sc[col[c] * GPS + 8 + j]);
      }
      const int gA = s * GPS + j, gB = gA + 8;
      float pA[COLS][T], pB[COLS][T];
#pragma unroll
      for (int r = 0; r < T; ++r)
#pragma unroll
        for (int c = 0; c < COLS; ++c) { pA[c][r] = 0.0f; pB[c][r] = 0.0f; }
#pragma unroll
      for (int tc = 0; tc < 4; ++tc) {
        uint32_t a[COLS][4], b[COLS][4];
#pragma unroll
        for (int c = 0; c < COLS; ++c) {
          e2m1x8_to_f16x2(reinterpret_cast<const uint32_t*>(&cA[c])[tc], a[c][0], a[c][1], a[c][2], a[c][3]);
          e2m1x8_to_f16x2(reinterpret_cast<const uint32_t*>(&cB[c])[tc], b[c][0], b[c][1], b[c][2], b[c][3]);
        }
#pragma unroll
        for (int r = 0; r < T; ++r) {
          if (X32) {
            // fp32 rows: the same chunks at twice the offsets, plain fp32 fma (exact products)
            const uint32_t xp = xs_a + r * xrs + 2 * (s * 1024 + tc * 128);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {  // four values of each group at a time
              const float4 xa = lds128f(xp + 16 * hf);
              const float4 xb = lds128f(xp + 1024 + 16 * hf);
#pragma unroll
              for (int ii = 0; ii < 2; ++ii) {
                const int i = 2 * hf + ii;
                const float xa_lo = ii ? xa.z : xa.x, xa_hi = ii ? xa.w : xa.y;
                const float xb_lo = ii ? xb.z : xb.x, xb_hi = ii ? xb.w : xb.y;
#pragma unroll
                for (int c = 0; c < COLS; ++c) {
                  const __half2 wa = *reinterpret_cast<const __half2*>(&a[c][i]);
                  const __half2 wb = *reinterpret_cast<const __half2*>(&b[c][i]);
                  pA[c][r] = __fmaf_rn(__low2float(wa), xa_lo, pA[c][r]);
                  pA[c][r] = __fmaf_rn(__high2float(wa), xa_hi, pA[c][r]);
                  pB[c][r] = __fmaf_rn(__low2float(wb), xb_lo, pB[c][r]);
                  pB[c][r] = __fmaf_rn(__high2float(wb), xb_hi, pB[c][r]);
                }
              }
            }
            continue;
          }
          // xoff(row, 16s + j (+ 8), tc) = row*GB*512 + s*1024 (+ 512) + tc*128 + j*16
          const uint32_t xp = xs_a + r * xrs + s * 1024 + tc * 128;
          const uint4 xa = lds128(xp);
          const uint4 xb = lds128(xp + 512);
          const uint32_t* va = reinterpret_cast<const uint32_t*>(&xa);
          const uint32_t* vb = reinterpret_cast<const uint32_t*>(&xb);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int c = 0; c < COLS; ++c) {
              pA[c][r] = fma2_f16(a[c][i], va[i], pA[c][r]);
              pB[c][r] = fma2_f16(b[c][i], vb[i], pB[c][r]);
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < T; ++r) {
        const float mA = lds32f(xm_a + r * xms + 4 * s * GPS), mB = lds32f(xm_a + r * xms + 4 * (s * GPS + 8));
#pragma unroll
        for (int c = 0; c < COLS; ++c) {
          if (KIND == TFX_ACT_E4M3) {
            acc[c][r] = __fmaf_rn(pA[c][r], __fmul_rn(sA[c], mA), acc[c][r]);
            acc[c][r] = __fmaf_rn(pB[c][r], __fmul_rn(sB[c], mB), acc[c][r]);
          } else {
            float qA = pA[c][r], qB = pB[c][r];
            const uint16_t* xrow = xraw + (size_t)prow[r] * pj.K;
            if (!X32 && mA == 0.0f) qA = chain_bf16_exact(cA[c], xrow, gA);
            else qA = __fmul_rn(qA, mA);
            if (!X32 && mB == 0.0f) qB = chain_bf16_exact(cB[c], xrow, gB);
            else qB = __fmul_rn(qB, mB);
            acc[c][r] = __fmaf_rn(qA, sA[c], acc[c][r]);
            acc[c][r] = __fmaf_rn(qB, sB[c], acc[c][r]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.empty[slot]);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&B.xempty[bx]);  // this warp is done with the activation buffer
  // eight-way tree: ((a0+a4)+(a2+a6)) + ((a1+a5)+(a3+a7)) across the octet
  float v[COLS][T];
#pragma unroll
  for (int r = 0; r < T; ++r)
#pragma unroll
    for (int c = 0; c < COLS; ++c) {
      float t = acc[c][r];
      t = t + __shfl_xor_sync(0xffffffffu, t, 4);
      t = t + __shfl_xor_sync(0xffffffffu, t, 2);
      t = t + __shfl_xor_sync(0xffffffffu, t, 1);
      v[c][r] = t;
    }
  if (ewait) warp_wait(&B.eempty[be], eph, P, abort_flag, dead);
  if (!dead && j == 0) {
#pragma unroll
    for (int r = 0; r < T; ++r)
      if (r < real) {
#pragma unroll
        for (int c = 0; c < COLS; ++c) epi[r * 64 + col[c]] = v[c][r];
      }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&B.efull[be]);
}

template <int KIND, int MAXR, bool DOWN, int COLS>
__device__ __forceinline__ void dispatch_pass(int t, const RowsParams& P, const Proj& pj, uint8_t* ring,
                                              const Bars& B, int bx, int be, uint32_t eph, bool ewait,
                                              volatile int* abort_flag, const uint8_t* xs_s, const float* xm_s,
                                              const int* prow, const uint16_t* xraw, int real, uint32_t& it,
                                              bool& dead, float* epi) {
  constexpr int LIM = DOWN ? (MAXR < MAX_PASS_D ? MAXR : MAX_PASS_D) : MAXR;
#define TFX_PASS(TT)                                                                                          \
  if constexpr (TT <= LIM)                                                                                    \
    run_pass<KIND, TT, COLS, DOWN && KIND == TFX_ACT_BF16>(P, pj, ring, B, bx, be, eph, ewait, abort_flag, xs_s, \
                                                           xm_s, prow, xraw, real, it, dead, epi)
  switch (t) {
    case 1: TFX_PASS(1); break;
    case 2: TFX_PASS(2); break;
    case 3: TFX_PASS(3); break;
    case 4: TFX_PASS(4); break;
    case 5: TFX_PASS(5); break;
    case 6: TFX_PASS(6); break;
    case 7: TFX_PASS(7); break;
    case 8: TFX_PASS(8); break;
    default: break;
  }
#undef TFX_PASS
}

// One pass as the helper sees it (all fields warp-uniform).
struct HPass {
  bool dn, last;
  int a, u, real, pidx;
  int pair[8];
};

// Epilogue warp: the epilogue of one pass, from result buffer epi. Gate/up: SwiGLU, the
// activation quantiser and h (+ debug copies); fused launches publish a finished gate/up unit.
// Down: the expert outputs d; fused launches combine each (row, block) whose last slot this
// writes.
template <int KIND, int PH>
__device__ void helper_epilogue(const RowsParams& P, const HPass& q, const Bars& B, const float* epi,
                                const int* r_prow, const int* r_pslot, const int* r_rowcnt, int32_t* done_upc,
                                int32_t* slots_done, volatile int* abort_flag, bool& dead) {
  const int lane = threadIdx.x & 31;
  const int be = q.pidx & 1;
  warp_wait(&B.efull[be], (q.pidx >> 1) & 1, P, abort_flag, dead);
  if (!dead) {
    for (int r = 0; r < q.real; ++r) {
      const int p = q.pair[r];
      if (!q.dn) {
        const int I = P.I;
        const int nn = 32 * q.u + lane;
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
          if (lane == 0) P.hs[(size_t)p * (I / 32) + q.u] = (uint8_t)sc;
        } else {
          static_cast<__nv_bfloat16*>(P.h)[(size_t)p * I + nn] = __float2bfloat16_rn(hv);
        }
      } else {
        const int row = r_prow[p], slot = r_pslot[p];
        if (row >= 0 && row < P.R && slot >= 0 && slot < P.k) {
          float* dst = P.out + ((size_t)row * P.k + slot) * P.H + 64 * q.u;
          dst[lane] = epi[r * 64 + lane];
          dst[32 + lane] = epi[r * 64 + 32 + lane];
          if (PH == PH_FUSED) {
            // combine (row, block u) in the CTA that writes the row's last slot
            __threadfence();
            int last = 0;
            if (lane == 0) last = atomicAdd(&slots_done[(size_t)row * P.pd.units + q.u], 1) == r_rowcnt[row] - 1;
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
              if (lane == 0) slots_done[(size_t)row * P.pd.units + q.u] = 0;  // last user of the counter
              __threadfence();
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int m = 64 * q.u + 32 * hh + lane;
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
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&B.eempty[be]);
  if (PH == PH_FUSED && !q.dn && q.last) {  // publish a finished gate/up unit
    __threadfence();
    __syncwarp();
    if (lane == 0 && !dead) atomicAdd(done_upc + q.a, 1);
  }
}

// ---------------------------------------------------------------- the sequence of passes
// Every role walks the same sequence of passes. Separate launches: this CTA's items
// (blockIdx.x + i * gridDim.x; an item is (active expert, output block), its passes sized by
// the rows left). Fused launch: the claimed work units, each one pass: unit i < n_upc is
// gate/up pass list entry i / units, output block i % units; the down units follow.
struct PassDesc {
  bool dn, first, last;
  int a, u, e, p0, pos, real, t, pidx;
};
struct PassGen {
  int item, left, pos, pidx;
  bool open, done;
  bool dn;
  int a, u, e, p0;
};
struct SeqCtx {
  int total, n_upc;
  const int *act, *offs;
  const int *plist_u, *plist_d;  // fused: pass lists
};
// next_item() yields this CTA's next item (or unit) index, or -1 when there is none.
template <int PH, typename NextItem>
__device__ __forceinline__ bool gen_next(PassGen& g, PassDesc& d, const RowsParams& P, const SeqCtx& c,
                                         NextItem&& next_item) {
  if constexpr (PH == PH_FUSED) {
    while (true) {
      if (g.done) return false;
      const int i = next_item();
      if (i < 0 || i >= c.total) {
        g.done = true;
        return false;
      }
      const bool dn = i >= c.n_upc;
      const Proj& pj = dn ? P.pd : P.pu;
      const int li = dn ? i - c.n_upc : i;
      const int q = li / pj.units, u = li - q * pj.units;
      const int ent = (dn ? c.plist_d : c.plist_u)[q];
      const int a = ent & 1023, start = (ent >> 10) & 255, real = (ent >> 18) & 15, t = (ent >> 22) & 15;
      const int e = c.act[a];
      const int p0 = (e >= 0 && e < P.E) ? c.offs[e] : 0;
      const int n = (e >= 0 && e < P.E) ? c.offs[e + 1] - p0 : 0;
      if (e < 0 || e >= P.E || real < 1 || t < real || t > MAX_PASS_U || start + real > n || p0 < 0 ||
          p0 + n > P.R * P.k) {
        if (threadIdx.x == 0) report(P.status, TFX_ST_SHAPE);
        continue;
      }
      d.dn = dn;
      d.first = true;
      d.last = true;
      d.a = a;
      d.u = u;
      d.e = e;
      d.p0 = p0;
      d.pos = p0 + start;
      d.real = real;
      d.t = t;
      d.pidx = g.pidx++;
      return true;
    }
  } else {
  while (true) {
    if (!g.open) {
      if (g.done) return false;
      g.item = next_item();
      if (g.item < 0 || g.item >= c.total) {
        g.done = true;
        return false;
      }
      const bool dn = g.item >= c.n_upc;
      const Proj& pj = dn ? P.pd : P.pu;
      const int li = dn ? g.item - c.n_upc : g.item;
      const int a = li / pj.units, u = li - a * pj.units;
      const int e = c.act[a];
      const int p0 = (e >= 0 && e < P.E) ? c.offs[e] : 0;
      const int n = (e >= 0 && e < P.E) ? c.offs[e + 1] - p0 : 0;
      if (e < 0 || e >= P.E || n <= 0 || p0 < 0 || p0 + n > P.R * P.k) {
        if (n != 0 && threadIdx.x == 0) report(P.status, TFX_ST_SHAPE);
        continue;
      }
      g.open = true;
      g.dn = dn;
      g.a = a;
      g.u = u;
      g.e = e;
      g.p0 = p0;
      g.pos = p0;
      g.left = n;
    }
    const int t = tier_of(g.left, g.dn ? P.cap_d : P.cap_u, P.tier_mode, g.dn);
    const int real = min(t, g.left);
    d.dn = g.dn;
    d.first = g.pos == g.p0;
    d.last = g.left == real;
    d.a = g.a;
    d.u = g.u;
    d.e = g.e;
    d.p0 = g.p0;
    d.pos = g.pos;
    d.real = real;
    d.t = t;
    d.pidx = g.pidx++;
    g.pos += real;
    g.left -= real;
    if (g.left == 0) g.open = false;
    return true;
  }
  }
}

// ---------------------------------------------------------------- the kernel
// Roles: the consumer warps compute; the next warp produces (weight stages); the next stages:
// it brings each pass's activation rows in by bulk copy one pass ahead and converts them into
// the f16 buffer; the last runs each pass's epilogue (SwiGLU and quantisation of h, or the d
// rows and, in the fused launch, the combine) while the consumers go on with the next pass.
template <int KIND, int MAXR_U, int MAXR_D, int PH>
struct RowsShape {
  static constexpr int MAXR = ((PH & PH_UPC) && MAXR_U > MAXR_D) || !(PH & PH_DOWN) ? MAXR_U : MAXR_D;
  using C = Cfg<MAXR>;
};

template <int KIND, int MAXR_U, int MAXR_D, int PH>
__global__ void __launch_bounds__(RowsShape<KIND, MAXR_U, MAXR_D, PH>::C::NT)
    __maxnreg__((RowsShape<KIND, MAXR_U, MAXR_D, PH>::C::MAXREG)) rows_kernel(const RowsParams P) {
  using Sh = RowsShape<KIND, MAXR_U, MAXR_D, PH>;
  using C = typename Sh::C;
  constexpr int MAXR = Sh::MAXR;
  constexpr int NCW = C::NCW, NT = C::NT;
  constexpr int AB = KIND == TFX_ACT_E4M3 ? 1 : 2;  // activation bytes per element
  extern __shared__ __align__(128) uint8_t smem[];
  const Layout Ly = layout_of(P, MAXR);
  Bars B;
  B.full = reinterpret_cast<uint64_t*>(smem + Ly.bars);
  B.empty = B.full + MAX_NSTAGE;
  B.xfull = B.empty + MAX_NSTAGE;
  B.xempty = B.xfull + 2;
  B.efull = B.xempty + 2;
  B.eempty = B.efull + 2;
  uint64_t* rawfull = B.eempty + 2;
  uint64_t* qfull = rawfull + 1;  // fused: claimed-item queue, producer -> helper and consumers
  uint64_t* qempty = qfull + QD;  //        and back
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly.ctrl);
  int* pdesc = reinterpret_cast<int*>(smem + Ly.pdesc);  // [2][16]: prow[8], ppair[8]
  float* epi = reinterpret_cast<float*>(smem + Ly.epi);    // [2][8][64]
  uint8_t* ring = smem + Ly.ring;
  uint8_t* raw = smem + Ly.raw;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NST = P.nstage, NXB = P.nxb;
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&B.full[s], 1);
      mbar_init(&B.empty[s], NCW);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B.xfull[b], 1);
      mbar_init(&B.xempty[b], NCW);
      mbar_init(&B.efull[b], NCW);
      mbar_init(&B.eempty[b], 1);
    }
    mbar_init(rawfull, 1);
    for (int b = 0; b < QD; ++b) {
      mbar_init(&qfull[b], 1);
      mbar_init(&qempty[b], NCW + 2);
    }
    mbar_fence_init();
    *abort_flag = 0;
  }

  // row lists: computed here (fused) or read from a previous route launch
  const int *r_offs, *r_prow, *r_pslot, *r_act, *r_rowcnt = nullptr;
  const uint16_t *np_u = nullptr, *np_d = nullptr;  // fused: passes per active expert
  int n_act;
  SeqCtx sc;
  if (PH == PH_FUSED) {
    SRoute rt;
    route_smem<NT>(P, reinterpret_cast<int*>(smem + Ly.route), rt, tid);  // synchronises the block
    n_act = *rt.nact;
    np_u = rt.np_u;
    np_d = rt.np_d;
    r_offs = rt.offs;
    r_prow = rt.prow;
    r_pslot = rt.pslot;
    r_act = rt.act;
    r_rowcnt = rt.rowcnt;
    sc.plist_u = rt.plist_u;
    sc.plist_d = rt.plist_d;
    sc.n_upc = rt.nlist[0] * P.pu.units;
    sc.total = sc.n_upc + rt.nlist[1] * P.pd.units;
    if (blockIdx.x == 0) {  // publish the row lists
      const int Pn = P.R * P.k;
      for (int i = tid; i <= P.E; i += NT) P.offs[i] = rt.offs[i];
      for (int i = tid; i < Pn; i += NT) {
        P.pair_row[i] = i < rt.offs[P.E] ? rt.prow[i] : 0;
        P.pair_slot[i] = i < rt.offs[P.E] ? rt.pslot[i] : 0;
      }
      for (int i = tid; i < n_act; i += NT) P.active[i] = rt.act[i];
      if (tid == 0) *P.n_active = n_act;
    }
  } else {
    __syncthreads();
    n_act = *P.n_active;
    r_offs = P.offs;
    r_prow = P.pair_row;
    r_pslot = P.pair_slot;
    r_act = P.active;
    sc.plist_u = sc.plist_d = nullptr;
    sc.n_upc = (PH & PH_UPC) ? n_act * P.pu.units : 0;
    sc.total = sc.n_upc + ((PH & PH_DOWN) ? n_act * P.pd.units : 0);
  }
  sc.act = r_act;
  sc.offs = r_offs;
  int32_t* work_ctr = PH == PH_FUSED ? P.scratch + 1 : nullptr;
  int32_t* done_upc = PH == PH_FUSED ? P.scratch + 2 : nullptr;
  int32_t* down_seen = PH == PH_FUSED ? P.scratch + 2 + P.E : nullptr;
  int32_t* slots_done = PH == PH_FUSED ? P.scratch + 2 + 2 * P.E : nullptr;
  int* qid = reinterpret_cast<int*>(smem + Ly.ctrl + 16);  // [QD] claimed item ids
  PassGen gen = {};
  PassDesc d;
  // Separate launches stride over the items; the fused launch hands units out dynamically: the
  // producer claims them from a global counter, in order (gate/up units pass-major, then down
  // units), and passes them to the helper and the consumers through a small queue.
  int static_next = blockIdx.x - (int)gridDim.x;
  uint32_t qpos = 0;
  auto next_static = [&]() { static_next += gridDim.x; return static_next; };
  auto next_popped = [&]() {  // helper and consumers (warp-wide)
    const int slot = qpos % QD;
    bool dq = false;
    warp_wait(&qfull[slot], (qpos / QD) & 1, P, abort_flag, dq);
    int v = dq ? -1 : qid[slot];
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(&qempty[slot]);
    ++qpos;
    return v;
  };

  if (warp == C::W_PROD) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      uint32_t claims = 0;
      auto claim = [&]() {  // producer lane: claim a unit and publish it to the queue
        const int slot = claims % QD;
        int v = -1;
        if (claims >= (uint32_t)QD && !mbar_wait(&qempty[slot], ((claims / QD) & 1) ^ 1, P.timeout_ns)) {
          if (*abort_flag == 0) report(P.status, TFX_ST_TIMEOUT);
          *abort_flag = 1;
        } else if (!*abort_flag) {
          // A CTA's first unit is its own index; the counter hands out the rest. Every CTA
          // with a first unit claims once more than it gets, so the launch makes exactly
          // max(0, total - grid) + min(total, grid) counter claims; the last one returns the
          // counter to zero for the next launch.
          if (claims == 0) {
            v = (int)blockIdx.x;
          } else {
            const int raw = atomicAdd(work_ctr, 1);
            const int g = (int)gridDim.x;
            if (raw == max(0, sc.total - g) + min(sc.total, g) - 1) *work_ctr = 0;
            v = raw + g;
          }
          if (v >= sc.total) v = -1;
        }
        qid[slot] = v;
        mbar_arrive(&qfull[slot]);
        ++claims;
        return v;
      };
      // The queue runs one unit ahead of the producer, so the stager learns of the next unit
      // (and can stage its activations) while the current one streams. The claim of that next
      // unit is made once the current unit's first stages are on their way.
      int ahead = -2;
      bool pending = false;
      auto claim_pending = [&]() {
        if (pending) {
          ahead = claim();
          pending = false;
        }
      };
      auto next_claimed = [&]() {
        if (ahead == -2) ahead = claim();
        claim_pending();
        const int v = ahead;
        if (v >= 0) pending = true;
        else ahead = -1;
        return v;
      };
      auto next_prod = [&]() { return PH == PH_FUSED ? next_claimed() : next_static(); };
      while (!stop && gen_next<PH>(gen, d, P, sc, next_prod)) {
        const Proj& pj = d.dn ? P.pd : P.pu;
        const uint8_t* src = pj.w + (size_t)d.e * pj.expert_bytes + (size_t)d.u * pj.unit_bytes;
        for (int s = 0; s < pj.S; ++s, ++it) {
          const int slot = it % NST;
          const uint32_t ph = (it / NST) & 1u;
          if (*abort_flag) { stop = true; break; }
          if (it >= (uint32_t)NST && !mbar_wait(&B.empty[slot], ph ^ 1u, P.timeout_ns)) {
            if (*abort_flag == 0) report(P.status, TFX_ST_TIMEOUT);
            *abort_flag = 1;
            stop = true;
            break;
          }
          if (*abort_flag) { stop = true; break; }
          mbar_arrive_expect_tx(&B.full[slot], STAGE_B);
          bulk_g2s(ring + (size_t)slot * STAGE_B, src + (size_t)s * STAGE_B, STAGE_B, &B.full[slot]);
          if (PH == PH_FUSED && (it + 1 >= (uint32_t)NST || s == pj.S - 1)) claim_pending();
        }
      }
      if (PH == PH_FUSED) claim_pending();
      if (PH == PH_FUSED && !gen.done) {
        // stopped early (abort): tell the helper and the consumers there is nothing more
        *abort_flag = 1;
        for (int q = 0; q < 2 * QD && !gen.done; ++q) {
          const int slot = claims % QD;
          mbar_wait(&qempty[slot], ((claims / QD) & 1) ^ 1, 1000000ull);
          qid[slot] = -1;
          mbar_arrive(&qfull[slot]);
          ++claims;
        }
      }
      // Drain: every issued stage must have landed before the block may exit.
      const uint32_t first = it > (uint32_t)NST ? it - NST : 0u;
      for (uint32_t q = first; q < it; ++q) {
        if (!mbar_wait(&B.full[q % NST], (q / NST) & 1u, P.timeout_ns)) {
          report(P.status, TFX_ST_TIMEOUT);
          break;
        }
      }
    }
  } else if (warp == C::W_HELP) {
    // ---------------------------------------------------------------- helper
    bool dead = false;
    uint32_t raw_issued = 0, raw_waited = 0;

    // rows of a pass: token rows (gate/up) or pair rows (down); padding repeats the last
    auto row_of = [&](const PassDesc& q, int r) {
      const int src = q.pos + min(r, q.real - 1);
      if (q.dn) return src;
      const int row = r_prow[src];
      return (row < 0 || row >= P.R) ? 0 : row;
    };
    // fused down: wait (bounded) until every gate/up unit of the expert has published its h
    auto wait_dependency = [&](const PassDesc& q) {
      if (!(PH == PH_FUSED && q.dn && q.first) || dead) return;
      int okw = 1;
      if (lane == 0) {
        const int need = np_u[q.a] * P.pu.units;
        const uint64_t t0 = global_ns();
        while (true) {
          int v;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(done_upc + q.a) : "memory");
          if (v >= need) break;
          if (*abort_flag || global_ns() - t0 > P.timeout_ns) {
            if (*abort_flag == 0) report(P.status, TFX_ST_TIMEOUT);
            *abort_flag = 1;
            okw = 0;
            break;
          }
          __nanosleep(64);
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");  // h is read next by the async proxy
        // the expert's last down unit past this point returns both counters to zero
        if (okw && atomicAdd(down_seen + q.a, 1) == np_d[q.a] * P.pd.units - 1) {
          done_upc[q.a] = 0;
          down_seen[q.a] = 0;
        }
      }
      if (!__shfl_sync(0xffffffffu, okw, 0)) dead = true;
    };
    // bulk copies of the pass's activation rows (and scales) into the raw buffer
    // Rows of the pass last staged into each activation buffer (lane r < 8 holds row r): a pass
    // whose buffer already holds its rows (every gate/up pass of a one-row launch, for one) is
    // not staged again.
    int krow0 = -1, krow1 = -1, kdn0 = -1, kdn1 = -1, kreal0 = 0, kreal1 = 0;
    bool pend_skip = false, pend_copy = false;
    // other: compare with the buffer the pass does not use (two buffers)
    auto same_rows = [&](const PassDesc& q, bool other = false) {
      const bool b1 = NXB == 2 && (((q.pidx & 1) != 0) != other);
      const int mine = lane < 8 ? row_of(q, lane) : 0;
      const bool eq = lane >= 8 || (b1 ? krow1 : krow0) == mine;
      return (b1 ? kdn1 : kdn0) == (int)q.dn && (b1 ? kreal1 : kreal0) == q.t && __all_sync(0xffffffffu, eq);
    };
    auto issue_raw = [&](const PassDesc& q) {
      pend_skip = same_rows(q);
      pend_copy = !pend_skip && NXB == 2 && same_rows(q, true);  // the other buffer has them: copy it
      if (pend_skip || pend_copy || !P.use_raw || dead) return;
      const Proj& pj = q.dn ? P.pd : P.pu;
      const int rowb = pj.K * AB;
      const bool tsc = KIND == TFX_ACT_E4M3 && (q.dn ? P.sc_tma_d : P.sc_tma_u);
      const uint8_t* X8 = q.dn ? static_cast<const uint8_t*>(P.h) : static_cast<const uint8_t*>(P.x);
      const uint8_t* XS = q.dn ? P.hs : P.xs;
      int rows[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) rows[r] = row_of(q, r);
      __syncwarp();  // the previous conversion's reads of the raw buffer are done
      if (lane == 0) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(rawfull, (uint32_t)(q.t * (rowb + (tsc ? pj.G : 0))));
        for (int r = 0; r < q.t; ++r) {
          bulk_g2s(raw + r * P.raw_row, X8 + (size_t)rows[r] * rowb, rowb, rawfull);
          if (tsc) bulk_g2s(raw + MAXR * P.raw_row + r * P.raw_sc, XS + (size_t)rows[r] * pj.G, pj.G, rawfull);
        }
      }
      ++raw_issued;
    };
    // wait for the pass's activation buffer, fill it, hand it to the consumers
    auto finish_stage = [&](const PassDesc& q) {
      const Proj& pj = q.dn ? P.pd : P.pu;
      const int bx = NXB == 2 ? (q.pidx & 1) : 0;
      if (q.pidx >= NXB) warp_wait(&B.xempty[bx], ((q.pidx / NXB) & 1) ^ 1, P, abort_flag, dead);
      int* pd = pdesc + 16 * bx;
      if (lane < 8) {
        pd[lane] = row_of(q, lane);
        pd[8 + lane] = q.pos + min(lane, q.real - 1);
      }
      __syncwarp();
      uint8_t* xs_s = smem + Ly.xs + bx * Ly.xs_stride;
      float* xm_s = reinterpret_cast<float*>(smem + Ly.xm + bx * Ly.xm_stride);
      const uint8_t* X8 = q.dn ? static_cast<const uint8_t*>(P.h) : static_cast<const uint8_t*>(P.x);
      const uint8_t* XS = q.dn ? P.hs : P.xs;
      if (pend_skip) {
        // the buffer holds these rows already
      } else if (pend_copy) {
        if (!dead) {  // the other buffer holds these rows, staged the same way: copy its rows and multipliers
          const int xb = (KIND == TFX_ACT_BF16 && q.dn ? 2 : 1) * q.t * pj.GB * 512;
          const uint4* s4 = reinterpret_cast<const uint4*>(smem + Ly.xs + (bx ^ 1) * Ly.xs_stride);
          uint4* d4 = reinterpret_cast<uint4*>(xs_s);
          for (int i = lane; i < xb / 16; i += kWarp) d4[i] = s4[i];
          const float* sm = reinterpret_cast<const float*>(smem + Ly.xm + (bx ^ 1) * Ly.xm_stride);
          for (int i = lane; i < q.t * pj.GB * 8; i += kWarp) xm_s[i] = sm[i];
        }
      } else if (P.use_raw) {
        if (raw_waited < raw_issued) {
          warp_wait(rawfull, raw_waited & 1u, P, abort_flag, dead);
          ++raw_waited;
        }
        const bool tsc = KIND == TFX_ACT_E4M3 && (q.dn ? P.sc_tma_d : P.sc_tma_u);
        if (!dead) {
          if (tsc)
            stage_rows<KIND, true, true>(raw, P.raw_row, raw + MAXR * P.raw_row, P.raw_sc, pj.K, pj.G, pj.GB, xs_s,
                                         xm_s, pd, q.t, lane, 32);
          else if (KIND == TFX_ACT_BF16 && q.dn)
            stage_rows<KIND, true, false, true>(raw, P.raw_row, XS, pj.G, pj.K, pj.G, pj.GB, xs_s, xm_s, pd, q.t,
                                                lane, 32);
          else
            stage_rows<KIND, true, false>(raw, P.raw_row, XS, pj.G, pj.K, pj.G, pj.GB, xs_s, xm_s, pd, q.t,
                                          lane, 32);
        }
      } else if (!dead) {
        if (KIND == TFX_ACT_BF16 && q.dn)
          stage_rows<KIND, false, false, true>(X8, (size_t)pj.K * AB, XS, pj.G, pj.K, pj.G, pj.GB, xs_s, xm_s, pd,
                                               q.t, lane, 32);
        else
          stage_rows<KIND, false, false>(X8, (size_t)pj.K * AB, XS, pj.G, pj.K, pj.G, pj.GB, xs_s, xm_s, pd, q.t,
                                         lane, 32);
      }
      if (!pend_skip && !dead) {
        const int mine = lane < 8 ? row_of(q, lane) : 0;
        if (bx) { krow1 = mine; kdn1 = q.dn; kreal1 = q.t; }
        else { krow0 = mine; kdn0 = q.dn; kreal0 = q.t; }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.xfull[bx]);
    };
    PassDesc cur, nxt;
    auto next_hc = [&]() { return PH == PH_FUSED ? next_popped() : next_static(); };
    bool hc = gen_next<PH>(gen, cur, P, sc, next_hc);
    if (hc) {
      wait_dependency(cur);
      issue_raw(cur);
    }
    while (hc) {
      finish_stage(cur);
      if (!gen_next<PH>(gen, nxt, P, sc, next_hc)) break;
      wait_dependency(nxt);
      issue_raw(nxt);
      cur = nxt;
    }
    // a bulk copy issued before an abort must land before the block may exit
    if (lane == 0 && raw_waited < raw_issued && !mbar_wait(rawfull, raw_waited & 1u, P.timeout_ns))
      report(P.status, TFX_ST_TIMEOUT);
  } else if (warp == C::W_EPI) {
    // ---------------------------------------------------------------- epilogue
    bool dead = false;
    auto epilogue = [&](const PassDesc& q) {
      HPass hp;
      hp.dn = q.dn;
      hp.last = q.last;
      hp.a = q.a;
      hp.u = q.u;
      hp.real = q.real;
      hp.pidx = q.pidx;
#pragma unroll
      for (int r = 0; r < 8; ++r) hp.pair[r] = q.pos + min(r, q.real - 1);
      helper_epilogue<KIND, PH>(P, hp, B, epi + (q.pidx & 1) * 512, r_prow, r_pslot, r_rowcnt, done_upc, slots_done,
                                abort_flag, dead);
    };

    auto next_e = [&]() { return PH == PH_FUSED ? next_popped() : next_static(); };
    PassDesc q;
    while (gen_next<PH>(gen, q, P, sc, next_e)) epilogue(q);
  } else {
    // ---------------------------------------------------------------- consumers
    uint32_t it = 0;
    bool dead = false;
    auto next_c = [&]() { return PH == PH_FUSED ? next_popped() : next_static(); };
    while (gen_next<PH>(gen, d, P, sc, next_c)) {
      const Proj& pj = d.dn ? P.pd : P.pu;
      const int bx = NXB == 2 ? (d.pidx & 1) : 0;
      const int be = d.pidx & 1;
      warp_wait(&B.xfull[bx], (d.pidx / NXB) & 1, P, abort_flag, dead);
      const uint8_t* xs_s = smem + Ly.xs + bx * Ly.xs_stride;
      const float* xm_s = reinterpret_cast<const float*>(smem + Ly.xm + bx * Ly.xm_stride);
      const uint16_t* xraw = reinterpret_cast<const uint16_t*>(d.dn ? P.h : P.x);
      const int* prow = pdesc + 16 * bx;
      float* ep = epi + be * 512;
      const uint32_t eph = ((d.pidx >> 1) & 1) ^ 1;
      if (d.dn) dispatch_pass<KIND, MAXR_D, true, C::COLS>(d.t, P, pj, ring, B, bx, be, eph, d.pidx >= 2, abort_flag,
                                                           xs_s, xm_s, prow, xraw, d.real, it, dead, ep);
      else dispatch_pass<KIND, MAXR_U, false, C::COLS>(d.t, P, pj, ring, B, bx, be, eph, d.pidx >= 2, abort_flag,
                                                       xs_s, xm_s, prow, xraw, d.real, it, dead, ep);
    }
  }
}

// ------------------------------------------------------------------------------ host side

std::mutex& rows_mutex();
int dev_sms(int* sms, size_t* optin);

// Shared-memory shape and blocks per SM, chosen once per (device, kernel instance, shape) and
// cached, so that steady-state launches (and launches under stream capture) issue only the
// kernel. Candidates: activation rows by bulk copy or by global loads, one or two activation
// buffers (two let the next pass stage while this one runs), ring depth 2..6. The pick keeps
// the most weight bytes in flight per SM (resident blocks x ring stages, up to 6 a block),
// then prefers two buffers, then bulk-copied rows, then more resident blocks.
template <int KIND, int MAXR_U, int MAXR_D, int PH>
int launch_rows(RowsParams P, int max_items, cudaStream_t st) {
  using Sh = RowsShape<KIND, MAXR_U, MAXR_D, PH>;
  constexpr int MAXR = Sh::MAXR;
  constexpr int NT = Sh::C::NT;
  int sms;
  size_t optin;
  int rc = dev_sms(&sms, &optin);
  if (rc) return rc;
  auto kern = rows_kernel<KIND, MAXR_U, MAXR_D, PH>;
  struct Entry { int key_gb, key_route, key_raw, nst, nxb, use_raw, nb; size_t smem; };
  static Entry cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TFX_ECUDA;
  Entry ent;
  {
    std::lock_guard<std::mutex> lk(rows_mutex());
    ent = cache[dev];
    if (ent.nb == 0 || ent.key_gb != P.gbmax || ent.key_route != P.route_ints || ent.key_raw != P.raw_row) {
      RowsParams q = P;
      q.nstage = 6;
      q.nxb = 2;
      q.use_raw = 1;
      const size_t smax = (size_t)layout_of(q, MAXR).total;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)min(smax, optin)) != cudaSuccess)
        return TFX_ELAUNCH;
      Entry best = {};
      long best_score = -1;
      for (int raw = 0; raw <= 1; ++raw)
        for (int nxb = 1; nxb <= 2; ++nxb)
          for (int nst = 2; nst <= 6; ++nst) {
            q.nstage = nst;
            q.use_raw = raw;
            q.nxb = nxb;
            const size_t sm = (size_t)layout_of(q, MAXR).total;
            if (sm > optin) continue;
            int nb = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, NT, sm) != cudaSuccess) return TFX_ELAUNCH;
            if (nb < 1) continue;
            const long score = (long)min(nb * nst, 8) * 1000 + (nxb == 2 ? 100 : 0) + raw * 10 + nb;
            if (score > best_score) {
              best_score = score;
              best = Entry{P.gbmax, P.route_ints, P.raw_row, nst, nxb, raw, nb, sm};
            }
          }
      if (best_score < 0) return TFX_EUNSUPPORTED;
      ent = best;
      cache[dev] = ent;
    }
  }
  P.use_raw = ent.use_raw;
  P.nxb = ent.nxb;
  P.nstage = ent.nst;
  const int grid = min(max_items, ent.nb * sms);
  if (grid < 1) return TFX_OK;
  if (PH == PH_FUSED) {
    // CTAs of the fused launch wait on one another: launch cooperatively, so that the runtime
    // guarantees every CTA is resident at once (or refuses the launch).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(NT);
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
  kern<<<grid, NT, ent.smem, st>>>(P);
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}

// The kernel instance for the pass caps: the smallest of 1, 2, 4, 8 rows at or above the cap.
__host__ __device__ constexpr int instance_rows(int cap) { return cap <= 1 ? 1 : cap <= 2 ? 2 : cap <= 4 ? 4 : 8; }
// Warps of the fused instance for a gate/up pass cap.
inline int instance_warps(int cap) {
  switch (instance_rows(cap)) {
    case 1: return Cfg<1>::NT / kWarp;
    case 2: return Cfg<2>::NT / kWarp;
    case 4: return Cfg<4>::NT / kWarp;
    default: return Cfg<8>::NT / kWarp;
  }
}

template <int KIND, int PH>
int dispatch(const RowsParams& P, int max_items, cudaStream_t st) {
  if (PH == PH_UPC) {
    switch (instance_rows(P.cap_u)) {
      case 1: return launch_rows<KIND, 1, 1, PH_UPC>(P, max_items, st);
      case 2: return launch_rows<KIND, 2, 1, PH_UPC>(P, max_items, st);
      case 4: return launch_rows<KIND, 4, 1, PH_UPC>(P, max_items, st);
      default: return launch_rows<KIND, 8, 1, PH_UPC>(P, max_items, st);
    }
  } else if (PH == PH_DOWN) {
    switch (instance_rows(P.cap_d)) {
      case 1: return launch_rows<KIND, 1, 1, PH_DOWN>(P, max_items, st);
      case 2: return launch_rows<KIND, 1, 2, PH_DOWN>(P, max_items, st);
      default: return launch_rows<KIND, 1, 4, PH_DOWN>(P, max_items, st);
    }
  } else {
    switch (instance_rows(P.cap_u)) {
      case 1: return launch_rows<KIND, 1, 1, PH_FUSED>(P, max_items, st);
      case 2: return launch_rows<KIND, 2, 2, PH_FUSED>(P, max_items, st);
      case 4: return launch_rows<KIND, 4, 4, PH_FUSED>(P, max_items, st);
      default: return launch_rows<KIND, 8, 4, PH_FUSED>(P, max_items, st);
    }
  }
}

}  // namespace tfx
