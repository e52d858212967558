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
//     scratch; each counter's last user returns it to zero (no end-of-launch barrier).
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
constexpr int NTHREADS = NCONS + 3 * kWarp;      // + producer, stager and epilogue warps
constexpr int W_PROD = NCW;                      // producer warp index (weight stages)
constexpr int W_HELP = NCW + 1;                  // stager warp index (activation buffers)
constexpr int W_EPI = NCW + 2;                   // epilogue warp index (results out)
constexpr int MAX_NSTAGE = 8;
constexpr int FUSED_MAX_PAIRS = 256;
constexpr int QD = 4;                            // claimed-item queue depth (fused)

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
  int nxb;              // activation buffers in shared memory (2: the next pass stages while this one runs)
  int use_raw;          // 1: activation rows arrive by bulk copy into a shared-memory raw buffer
  int raw_row, raw_sc;  // raw buffer bytes per row (128-aligned) and per row of scales (16-aligned)
  int sc_tma_u, sc_tma_d;  // scales of gate/up (x) / down (h) rows come by bulk copy too
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
  int32_t* scratch;     // fused: [0] unused, [1] work counter, [2..E+1] gate/up items done per
                        //        active expert, [E+2..2E+1] down items past their wait per active
                        //        expert, then [R][H/64] slots written per (row, block)
  int32_t* status;
  int tier_mode;
  uint64_t timeout_ns;
};

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
// counts. All NTHREADS threads take part. Ints used: 3E + 2 + 3P + R + 2 * (NTHREADS / 32).
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
  for (int q = tid; q < P; q += NTHREADS) rt.prow[q] = p.ids[q];  // ids, staged (prow is free until the scatter)
  __syncthreads();
  int bad = 0;
  for (int q = tid; q < P; q += NTHREADS) {
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
  constexpr int NW = NTHREADS / 32;
  int* wsum = rt.rowcnt + p.R;  // 2 * NW
  const int lane = tid & 31, warp = tid >> 5;
  const int per = (E + NTHREADS - 1) / NTHREADS;
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
  // Stable scatter, one warp, 32 pairs at a time: a pair's position is its expert's cursor plus
  // the number of earlier lanes of the chunk with the same expert.
  if (warp == 0) {
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
  }
  __syncthreads();
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
__device__ const E8m0Table e8m0_table = E8m0Table();
__device__ __forceinline__ float e8m0_lookup(uint32_t code) { return __uint_as_float(__ldg(e8m0_table.v + code)); }

// Consumers: consume the pass's S weight stages against activation buffer xs_s/xm_s, release
// the buffer, then hand the eight-way-tree results of both columns of every real row to the
// helper in epi[r][0..63] (column o at o, column 32 + o at 32 + o).
template <int KIND, int T, bool X32 = false>
__device__ __forceinline__ void run_pass(const RowsParams& P, const Proj& pj, uint8_t* ring, const Bars& B,
                                         int bx, int be, uint32_t eph, bool ewait, volatile int* abort_flag,
                                         const uint8_t* xs_s, const float* xm_s, const int* prow,
                                         const uint16_t* xraw, int real, uint32_t& it, bool& dead, float* epi) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = lane & 7, o = (warp << 2) | (lane >> 3);
  const int NST = P.nstage, GB = pj.GB;
  float acc0[T], acc1[T];
  int xr[T];
  const uint8_t* xrow_s[T];
  const float* xmrow_s[T];
#pragma unroll
  for (int r = 0; r < T; ++r) {
    acc0[r] = 0.0f;
    acc1[r] = 0.0f;
    xr[r] = min(r, real - 1);
    xrow_s[r] = xs_s + (X32 ? 2 : 1) * (xr[r] * GB * 512 + j * 16);
    xmrow_s[r] = xm_s + xr[r] * GB * 8 + j;
  }
  // ring position, advanced incrementally (no division per stage)
  int slot = (int)(it % (uint32_t)NST);
  uint32_t ph = (it / (uint32_t)NST) & 1u;
  for (int s = 0; s < pj.S; ++s, ++it, slot = slot + 1 == NST ? 0 : slot + 1, ph ^= slot == 0 ? 1u : 0u) {
    if (warp_wait(&B.full[slot], ph, P, abort_flag, dead)) {
      const uint8_t* tile = ring + (size_t)slot * STAGE_B;
      const uint8_t* sc = tile + TROWS * CODE_B;
      const uint4 cA0 = *reinterpret_cast<const uint4*>(tile + o * CODE_B + 16 * j);
      const uint4 cA1 = *reinterpret_cast<const uint4*>(tile + (32 + o) * CODE_B + 16 * j);
      const uint4 cB0 = *reinterpret_cast<const uint4*>(tile + o * CODE_B + 128 + 16 * j);
      const uint4 cB1 = *reinterpret_cast<const uint4*>(tile + (32 + o) * CODE_B + 128 + 16 * j);
      const float sA0 = e8m0_lookup(sc[o * GPS + j]), sA1 = e8m0_lookup(sc[(32 + o) * GPS + j]);
      const float sB0 = e8m0_lookup(sc[o * GPS + 8 + j]), sB1 = e8m0_lookup(sc[(32 + o) * GPS + 8 + j]);
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
          if (X32) {
            // fp32 rows: the same chunks at twice the offsets, plain fp32 fma (exact products)
            const uint8_t* xp = xrow_s[r] + 2 * (s * 1024 + tc * 128);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {  // four values of each group at a time
              const float4 xa = *reinterpret_cast<const float4*>(xp + 16 * hf);
              const float4 xb = *reinterpret_cast<const float4*>(xp + 1024 + 16 * hf);
#pragma unroll
              for (int ii = 0; ii < 2; ++ii) {
                const int i = 2 * hf + ii;
                const float xa_lo = ii ? xa.z : xa.x, xa_hi = ii ? xa.w : xa.y;
                const float xb_lo = ii ? xb.z : xb.x, xb_hi = ii ? xb.w : xb.y;
                const __half2 wa0 = *reinterpret_cast<const __half2*>(&a0[i]);
                const __half2 wa1 = *reinterpret_cast<const __half2*>(&a1[i]);
                const __half2 wb0 = *reinterpret_cast<const __half2*>(&b0[i]);
                const __half2 wb1 = *reinterpret_cast<const __half2*>(&b1[i]);
                pA0[r] = __fmaf_rn(__low2float(wa0), xa_lo, pA0[r]);
                pA0[r] = __fmaf_rn(__high2float(wa0), xa_hi, pA0[r]);
                pA1[r] = __fmaf_rn(__low2float(wa1), xa_lo, pA1[r]);
                pA1[r] = __fmaf_rn(__high2float(wa1), xa_hi, pA1[r]);
                pB0[r] = __fmaf_rn(__low2float(wb0), xb_lo, pB0[r]);
                pB0[r] = __fmaf_rn(__high2float(wb0), xb_hi, pB0[r]);
                pB1[r] = __fmaf_rn(__low2float(wb1), xb_lo, pB1[r]);
                pB1[r] = __fmaf_rn(__high2float(wb1), xb_hi, pB1[r]);
              }
            }
            continue;
          }
          // xoff(row, 16s + j (+ 8), tc) = row*GB*512 + s*1024 (+ 512) + tc*128 + j*16
          const uint8_t* xp = xrow_s[r] + s * 1024 + tc * 128;
          const uint4 xa = *reinterpret_cast<const uint4*>(xp);
          const uint4 xb = *reinterpret_cast<const uint4*>(xp + 512);
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
        const float mA = xmrow_s[r][s * GPS], mB = xmrow_s[r][s * GPS + 8];
        if (KIND == TFX_ACT_E4M3) {
          acc0[r] = __fmaf_rn(pA0[r], __fmul_rn(sA0, mA), acc0[r]);
          acc1[r] = __fmaf_rn(pA1[r], __fmul_rn(sA1, mA), acc1[r]);
          acc0[r] = __fmaf_rn(pB0[r], __fmul_rn(sB0, mB), acc0[r]);
          acc1[r] = __fmaf_rn(pB1[r], __fmul_rn(sB1, mB), acc1[r]);
        } else {
          float qA0 = pA0[r], qA1 = pA1[r], qB0 = pB0[r], qB1 = pB1[r];
          const uint16_t* xrow = xraw + (size_t)prow[xr[r]] * pj.K;
          if (!X32 && mA == 0.0f) {
            qA0 = chain_bf16_exact(cA0, xrow, gA);
            qA1 = chain_bf16_exact(cA1, xrow, gA);
          } else {
            qA0 = __fmul_rn(qA0, mA);
            qA1 = __fmul_rn(qA1, mA);
          }
          if (!X32 && mB == 0.0f) {
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
    if (lane == 0) mbar_arrive(&B.empty[slot]);
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&B.xempty[bx]);  // this warp is done with the activation buffer
  // eight-way tree: ((a0+a4)+(a2+a6)) + ((a1+a5)+(a3+a7)) across the octet
  float v0r[T], v1r[T];
#pragma unroll
  for (int r = 0; r < T; ++r) {
    float v0 = acc0[r], v1 = acc1[r];
    v0 = v0 + __shfl_xor_sync(0xffffffffu, v0, 4);
    v1 = v1 + __shfl_xor_sync(0xffffffffu, v1, 4);
    v0 = v0 + __shfl_xor_sync(0xffffffffu, v0, 2);
    v1 = v1 + __shfl_xor_sync(0xffffffffu, v1, 2);
    v0 = v0 + __shfl_xor_sync(0xffffffffu, v0, 1);
    v1 = v1 + __shfl_xor_sync(0xffffffffu, v1, 1);
    v0r[r] = v0;
    v1r[r] = v1;
  }
  if (ewait) warp_wait(&B.eempty[be], eph, P, abort_flag, dead);
  if (!dead && j == 0) {
#pragma unroll
    for (int r = 0; r < T; ++r)
      if (r < real) {
        epi[r * 64 + o] = v0r[r];
        epi[r * 64 + 32 + o] = v1r[r];
      }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&B.efull[be]);
}

template <int KIND, int MAXR, bool DOWN>
__device__ __forceinline__ void dispatch_pass(int t, const RowsParams& P, const Proj& pj, uint8_t* ring,
                                              const Bars& B, int bx, int be, uint32_t eph, bool ewait,
                                              volatile int* abort_flag, const uint8_t* xs_s, const float* xm_s,
                                              const int* prow, const uint16_t* xraw, int real, uint32_t& it,
                                              bool& dead, float* epi) {
#define TFX_PASS(TT)                                                                                  \
  run_pass<KIND, TT, DOWN && KIND == TFX_ACT_BF16>(P, pj, ring, B, bx, be, eph, ewait, abort_flag, xs_s, xm_s, prow, \
                                                   xraw, real, it, dead, epi)
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

// One pass as the helper sees it (all fields warp-uniform).
struct HPass {
  bool dn, last;
  int a, u, real, pidx;
  int pair[8];
};

// Helper: the epilogue of one pass, from result buffer epi. Gate/up: SwiGLU, the activation
// quantiser and h (+ debug copies); fused launches publish a finished gate/up item. Down: the
// expert outputs d; fused launches combine each (row, block) whose last slot this writes.
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
  if (PH == PH_FUSED && !q.dn && q.last) {  // publish a finished gate/up item
    __threadfence();
    __syncwarp();
    if (lane == 0 && !dead) atomicAdd(done_upc + q.a, 1);
  }
}

// ---------------------------------------------------------------- the sequence of passes
// Every role walks the same sequence: this CTA's items (blockIdx.x + i * gridDim.x; gate/up
// items before down items), and within an item its passes sized by the rows left.
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
};
// next_item() yields this CTA's next item index, or -1 when there is none.
template <int MAXR_U, int MAXR_D, typename NextItem>
__device__ __forceinline__ bool gen_next(PassGen& g, PassDesc& d, const RowsParams& P, const SeqCtx& c,
                                         NextItem&& next_item) {
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
    const int t = g.dn ? tier_of<true>(g.left, MAXR_D, P.tier_mode) : tier_of<false>(g.left, MAXR_U, P.tier_mode);
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

// ---------------------------------------------------------------- the kernel
// Roles: warps 0..7 consume (compute); warp 8 produces (weight stages); warp 9 stages: it
// brings each pass's activation rows in by bulk copy one pass ahead and converts them into
// the f16 buffer; warp 10 runs each pass's epilogue (SwiGLU and quantisation of h, or the d
// rows and, in the fused launch, the combine) while the consumers go on with the next pass.
template <int KIND, int MAXR_U, int MAXR_D, int PH>
__global__ void __launch_bounds__(NTHREADS, ((PH & PH_UPC) ? MAXR_U : MAXR_D) <= 2 ? 2 : 1)
    rows_kernel(const RowsParams P) {
  constexpr int MAXR = ((PH & PH_UPC) && MAXR_U > MAXR_D) || !(PH & PH_DOWN) ? MAXR_U : MAXR_D;
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
  SeqCtx sc;
  sc.n_upc = (PH & PH_UPC) ? n_act * P.pu.units : 0;
  sc.total = sc.n_upc + ((PH & PH_DOWN) ? n_act * P.pd.units : 0);
  sc.act = r_act;
  sc.offs = r_offs;
  int32_t* work_ctr = PH == PH_FUSED ? P.scratch + 1 : nullptr;
  int32_t* done_upc = PH == PH_FUSED ? P.scratch + 2 : nullptr;
  int32_t* down_seen = PH == PH_FUSED ? P.scratch + 2 + P.E : nullptr;
  int32_t* slots_done = PH == PH_FUSED ? P.scratch + 2 + 2 * P.E : nullptr;
  int* qid = reinterpret_cast<int*>(smem + Ly.ctrl + 16);  // [QD] claimed item ids
  PassGen gen = {};
  PassDesc d;
  // Separate launches stride over the items; the fused launch hands items out dynamically: the
  // producer claims them from a global counter, in order (gate/up items expert by expert, then
  // down items), and passes them to the helper and the consumers through a small queue.
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

  if (warp == W_PROD) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      uint32_t claims = 0;
      auto claim = [&]() {  // producer lane: claim an item and publish it to the queue
        const int slot = claims % QD;
        int v = -1;
        if (claims >= (uint32_t)QD && !mbar_wait(&qempty[slot], ((claims / QD) & 1) ^ 1, P.timeout_ns)) {
          if (*abort_flag == 0) report(P.status, TFX_ST_TIMEOUT);
          *abort_flag = 1;
        } else if (!*abort_flag) {
          // A CTA's first item is its own index; the counter hands out the rest. Every CTA
          // with a first item claims once more than it gets, so the launch makes exactly
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
      // The queue runs one item ahead of the producer, so the stager learns of the next item
      // (and can stage its activations) while the current one streams. The claim of that next
      // item is made once the current item's first stages are on their way.
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
      while (!stop && gen_next<MAXR_U, MAXR_D>(gen, d, P, sc, next_prod)) {
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
  } else if (warp == W_HELP) {
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
    // fused down: wait (bounded) until every gate/up item of the expert has published its h
    auto wait_dependency = [&](const PassDesc& q) {
      if (!(PH == PH_FUSED && q.dn && q.first) || dead) return;
      int okw = 1;
      if (lane == 0) {
        const uint64_t t0 = global_ns();
        while (true) {
          int v;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(done_upc + q.a) : "memory");
          if (v >= P.pu.units) break;
          if (*abort_flag || global_ns() - t0 > P.timeout_ns) {
            if (*abort_flag == 0) report(P.status, TFX_ST_TIMEOUT);
            *abort_flag = 1;
            okw = 0;
            break;
          }
          __nanosleep(64);
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");  // h is read next by the async proxy
        // the expert's last down item past this point returns both counters to zero
        if (okw && atomicAdd(down_seen + q.a, 1) == P.pd.units - 1) {
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
      return (b1 ? kdn1 : kdn0) == (int)q.dn && (b1 ? kreal1 : kreal0) == q.real && __all_sync(0xffffffffu, eq);
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
        mbar_arrive_expect_tx(rawfull, (uint32_t)(q.real * (rowb + (tsc ? pj.G : 0))));
        for (int r = 0; r < q.real; ++r) {
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
          const int xb = (KIND == TFX_ACT_BF16 && q.dn ? 2 : 1) * q.real * pj.GB * 512;
          const uint4* s4 = reinterpret_cast<const uint4*>(smem + Ly.xs + (bx ^ 1) * Ly.xs_stride);
          uint4* d4 = reinterpret_cast<uint4*>(xs_s);
          for (int i = lane; i < xb / 16; i += kWarp) d4[i] = s4[i];
          const float* sm = reinterpret_cast<const float*>(smem + Ly.xm + (bx ^ 1) * Ly.xm_stride);
          for (int i = lane; i < q.real * pj.GB * 8; i += kWarp) xm_s[i] = sm[i];
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
                                         xm_s, pd, q.real, lane, 32);
          else if (KIND == TFX_ACT_BF16 && q.dn)
            stage_rows<KIND, true, false, true>(raw, P.raw_row, XS, pj.G, pj.K, pj.G, pj.GB, xs_s, xm_s, pd, q.real,
                                                lane, 32);
          else
            stage_rows<KIND, true, false>(raw, P.raw_row, XS, pj.G, pj.K, pj.G, pj.GB, xs_s, xm_s, pd, q.real,
                                          lane, 32);
        }
      } else if (!dead) {
        if (KIND == TFX_ACT_BF16 && q.dn)
          stage_rows<KIND, false, false, true>(X8, (size_t)pj.K * AB, XS, pj.G, pj.K, pj.G, pj.GB, xs_s, xm_s, pd,
                                               q.real, lane, 32);
        else
          stage_rows<KIND, false, false>(X8, (size_t)pj.K * AB, XS, pj.G, pj.K, pj.G, pj.GB, xs_s, xm_s, pd, q.real,
                                         lane, 32);
      }
      if (!pend_skip && !dead) {
        const int mine = lane < 8 ? row_of(q, lane) : 0;
        if (bx) { krow1 = mine; kdn1 = q.dn; kreal1 = q.real; }
        else { krow0 = mine; kdn0 = q.dn; kreal0 = q.real; }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.xfull[bx]);
    };
    PassDesc cur, nxt;
    auto next_hc = [&]() { return PH == PH_FUSED ? next_popped() : next_static(); };
    bool hc = gen_next<MAXR_U, MAXR_D>(gen, cur, P, sc, next_hc);
    if (hc) {
      wait_dependency(cur);
      issue_raw(cur);
    }
    while (hc) {
      finish_stage(cur);
      if (!gen_next<MAXR_U, MAXR_D>(gen, nxt, P, sc, next_hc)) break;
      wait_dependency(nxt);
      issue_raw(nxt);
      cur = nxt;
    }
    // a bulk copy issued before an abort must land before the block may exit
    if (lane == 0 && raw_waited < raw_issued && !mbar_wait(rawfull, raw_waited & 1u, P.timeout_ns))
      report(P.status, TFX_ST_TIMEOUT);
  } else if (warp == W_EPI) {
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
    while (gen_next<MAXR_U, MAXR_D>(gen, q, P, sc, next_e)) epilogue(q);
  } else {
    // ---------------------------------------------------------------- consumers
    uint32_t it = 0;
    bool dead = false;
    auto next_c = [&]() { return PH == PH_FUSED ? next_popped() : next_static(); };
    while (gen_next<MAXR_U, MAXR_D>(gen, d, P, sc, next_c)) {
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
      if (d.dn) dispatch_pass<KIND, MAXR_D, true>(d.t, P, pj, ring, B, bx, be, eph, d.pidx >= 2, abort_flag, xs_s,
                                                  xm_s, prow, xraw, d.real, it, dead, ep);
      else dispatch_pass<KIND, MAXR_U, false>(d.t, P, pj, ring, B, bx, be, eph, d.pidx >= 2, abort_flag, xs_s,
                                              xm_s, prow, xraw, d.real, it, dead, ep);
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

// Shared-memory shape and blocks per SM. Preference: activation rows by bulk copy with two
// activation buffers (the next pass stages while this one runs), then two buffers fed by
// global loads, then one buffer. Within a shape, the ring depth (2..6 stages) that keeps the
// most stage bytes in flight per SM (counting at most 4 stages a block), ties going to more
// resident blocks. Chosen once per (device, kernel instance, shape) and cached, so that
// steady-state launches (and launches under stream capture) issue only the kernel.
template <int KIND, int MAXR_U, int MAXR_D, int PH>
static int launch_rows(RowsParams P, int max_items, cudaStream_t st) {
  constexpr int MAXR = ((PH & PH_UPC) && MAXR_U > MAXR_D) || !(PH & PH_DOWN) ? MAXR_U : MAXR_D;
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
    std::lock_guard<std::mutex> lk(g_mu);
    ent = cache[dev];
    if (ent.nb == 0 || ent.key_gb != P.gbmax || ent.key_route != P.route_ints || ent.key_raw != P.raw_row) {
      RowsParams q = P;
      q.nstage = 6;
      q.nxb = 2;
      q.use_raw = 1;
      const size_t smax = (size_t)layout_of(q, MAXR).total;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)min(smax, optin)) != cudaSuccess)
        return TFX_ELAUNCH;
      const int shapes[4][2] = {{1, 2}, {0, 2}, {1, 1}, {0, 1}};  // (raw, buffers) in order of preference
      Entry best = {};
      int best_score = -1;
      for (int sh = 0; sh < 4 && best_score < 0; ++sh) {
        for (int nst = 2; nst <= 6; ++nst) {
          q.nstage = nst;
          q.use_raw = shapes[sh][0];
          q.nxb = shapes[sh][1];
          const size_t sm = (size_t)layout_of(q, MAXR).total;
          if (sm > optin) break;
          int nb = 0;
          if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, NTHREADS, sm) != cudaSuccess) return TFX_ELAUNCH;
          if (nb < 1) break;
          const int score = nb * min(nst, 4);
          if (score > best_score || (score == best_score && nb > best.nb)) {
            best_score = score;
            best = Entry{P.gbmax, P.route_ints, P.raw_row, nst, q.nxb, q.use_raw, nb, sm};
          }
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

// Raw-buffer geometry for activation rows of width kmax (bulk copies need 16-byte multiples;
// scales come by bulk copy only when a row of them is a 16-byte multiple and 16-byte aligned).
static void set_raw(RowsParams& P, int kind, int kmax, int gmax) {
  const int ab = kind == TFX_ACT_E4M3 ? 1 : 2;
  P.raw_row = (kmax * ab + 127) & ~127;
  P.raw_sc = kind == TFX_ACT_E4M3 ? ((gmax + 15) & ~15) : 0;
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
  set_raw(P, act_kind, P.pu.K, P.pu.G);
  P.sc_tma_u = act_kind == TFX_ACT_E4M3 && P.pu.G % 16 == 0 && aligned16(x_scale);
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
  P.gbmax = (act_kind == TFX_ACT_BF16 ? 2 : 1) * P.pd.GB;  // bf16 h is staged as fp32
  set_raw(P, act_kind, P.pd.K, P.pd.G);
  P.sc_tma_d = act_kind == TFX_ACT_E4M3 && P.pd.G % 16 == 0 && aligned16(h_scale);
  const int max_items = min(rows * d.top_k, d.n_experts) * P.pd.units;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch<TFX_ACT_E4M3, PH_DOWN>(P, 1, md, max_items, st);
  return dispatch<TFX_ACT_BF16, PH_DOWN>(P, 1, md, max_items, st);
}

extern "C" size_t tfx_xp_moe_rows_scratch_bytes(tfx_dims d, int32_t rows) {
  if (!dims_ok(d) || rows < 0) return 0;
  return sizeof(int32_t) * ((size_t)2 + 2 * (size_t)d.n_experts + (size_t)rows * (d.hidden / 64));  // see RowsParams
}

namespace tfx {

// Argument checks and parameters of the one-launch layer, without launching anything (shared
// by tfx_xp_moe_rows and tfx_xp_moe_rows_noalloc, which checks every argument before it
// touches its built-in counter buffer). `scratch` may be null here when check_scratch is 0.
static int moe_rows_prepare(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                            const uint8_t* x_scale, const int32_t* ids, const float* topk_w, int32_t* offs,
                            int32_t* pair_row, int32_t* pair_slot, int32_t* active, int32_t* n_active, void* h,
                            uint8_t* h_scale, float* out, uint16_t* y, float* y_f32_dbg, int32_t* scratch,
                            bool check_scratch, int32_t* status, const tfx_rows_opts* opts, RowsParams& P, int& mu,
                            int& md, int& max_items) {
  int rc = common_args(d, rows, act_kind, packed, x, x_scale, status, opts, P);
  if (rc) return rc;
  if ((int64_t)rows * d.top_k > FUSED_MAX_PAIRS) return TFX_EUNSUPPORTED;
  mu = pass_of(opts, false, rows);
  md = min(pass_of(opts, true, rows), 4);  // the down pass stops at 4 rows
  if (!((mu == 1 && md == 1) || (mu == 2 && md == 2) || (mu == 4 && md == 4) || (mu == 8 && md == 4)))
    return TFX_EINVAL;
  if (!offs || !active || !n_active) return TFX_EINVAL;
  if (check_scratch && (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 3u))) return TFX_EINVAL;
  if (rows == 0) return TFX_OK;
  if (!ids || !topk_w || !pair_row || !pair_slot || !h || !aligned16(h) || !out || !y ||
      (act_kind == TFX_ACT_E4M3 && !h_scale))
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
  P.gbmax = max(P.pu.GB, (act_kind == TFX_ACT_BF16 ? 2 : 1) * P.pd.GB);  // bf16 h is staged as fp32
  P.route_ints = 3 * d.n_experts + 2 + 3 * rows * d.top_k + rows + 2 * (NTHREADS / 32);
  set_raw(P, act_kind, max(P.pu.K, P.pd.K), max(P.pu.G, P.pd.G));
  P.sc_tma_u = act_kind == TFX_ACT_E4M3 && P.pu.G % 16 == 0 && aligned16(x_scale);
  P.sc_tma_d = act_kind == TFX_ACT_E4M3 && P.pd.G % 16 == 0 && aligned16(h_scale);
  max_items = min(rows * d.top_k, d.n_experts) * (P.pu.units + P.pd.units);
  return TFX_OK;
}

static int moe_rows_launch(const RowsParams& P, int32_t act_kind, int mu, int md, int max_items, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch<TFX_ACT_E4M3, PH_FUSED>(P, mu, md, max_items, st);
  return dispatch<TFX_ACT_BF16, PH_FUSED>(P, mu, md, max_items, st);
}

}  // namespace tfx

extern "C" int tfx_xp_moe_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                               const uint8_t* x_scale, const int32_t* ids, const float* topk_w, int32_t* offs,
                               int32_t* pair_row, int32_t* pair_slot, int32_t* active, int32_t* n_active, void* h,
                               uint8_t* h_scale, float* out, uint16_t* y, float* y_f32_dbg, int32_t* scratch,
                               int32_t* status, const tfx_rows_opts* opts, void* stream) {
  RowsParams P;
  int mu = 0, md = 0, max_items = 0;
  const int rc = moe_rows_prepare(d, rows, act_kind, packed, x, x_scale, ids, topk_w, offs, pair_row, pair_slot,
                                  active, n_active, h, h_scale, out, y, y_f32_dbg, scratch, true, status, opts, P,
                                  mu, md, max_items);
  if (rc || rows == 0) return rc;
  return moe_rows_launch(P, act_kind, mu, md, max_items, stream);
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
  // every other argument is checked before the built-in buffer is touched
  RowsParams P;
  int mu = 0, md = 0, max_items = 0;
  int rc = moe_rows_prepare(d, rows, act_kind, packed, x, x_scale, ids, topk_w, offs, pair_row, pair_slot, active,
                            n_active, h, h_scale, out, y, y_f32_dbg, nullptr, false, status, opts, P, mu, md,
                            max_items);
  if (rc || rows == 0) return rc;
  int32_t* scratch = nullptr;
  rc = noalloc_scratch(&scratch);
  if (rc) return rc;
  // the counters must start at zero; a previous call on this device may have stopped early
  if (cudaMemsetAsync(scratch, 0, need * sizeof(int32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    (void)cudaGetLastError();
    return TFX_ELAUNCH;
  }
  P.scratch = scratch;
  return moe_rows_launch(P, act_kind, mu, md, max_items, stream);
}
