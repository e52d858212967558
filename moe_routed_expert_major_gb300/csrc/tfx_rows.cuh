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
//   * a ring of shared-memory slots, one per stage of 512 k: the producer warp bulk-copies the
//     stage's weights (64 rows x 512 k of codes, then their scales: 17,408 contiguous bytes of
//     the packed layout, per packed unit of the item) and the pass's activation rows for the
//     same 512 k (cp.async.bulk + mbarrier, every wait bounded);
//   * the stager warp converts each slot's activation chunk into f16 (E4M3: exact; bf16 rows
//     shifted per 32-group by a power of two so that they are exact in f16, with an exact fp32
//     fallback for groups that do not fit; bf16 h of the down passes as fp32) and completes the
//     slot. Shared memory thus holds a few stages, whatever the pass's rows and K;
//   * consumer warps: lane (t & 7) of an octet owns accumulator lane j = group mod 8 of two
//     output columns (the gate and up rows of one output, or two down rows), so the eight-way
//     tree is three xor-shuffles, and every activation value read from shared memory feeds two
//     columns. A lane handles groups j and j + 8 of each stage. E2M1 codes decode with
//     cvt.rn.f16x2.e2m1x2; the chain runs on fma.rn.f32.f16 (fp32 accumulate, one rounding per
//     step). One-row kernels run 8 consumer warps on one packed unit per item, two CTAs an SM;
//     kernels with longer passes run 16 consumer warps on two packed units per item, one CTA an
//     SM, so that the fma-bound passes of many rows have four consumer warps per scheduler;
//   * the epilogue warp takes each pass's results (SwiGLU and the activation quantiser, or the
//     expert outputs and, in the fused launch, the combine) while the consumers go on;
//   * the fused layer launch (cooperative: all CTAs resident) computes the row lists in shared
//     memory in every CTA and hands out work units of one pass each, expert-major: every
//     gate/up pass of the first active expert, then of the second, ..., then the down passes in
//     the same order (each waits, bounded, for its expert's gate/up units), so that the down
//     units claimed first are those of the experts whose gate/up units were handed out first. Each (row, 64-output
//     block) is combined in the CTA whose down unit completes the row's last slot. Completion
//     counters live in caller scratch; each counter's last user returns it to zero.
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
constexpr int TROWS = 64;                        // weight rows per packed unit and stage
constexpr int CODE_B = KC / 2;                   // code bytes per row per stage
constexpr int STAGE_B = TROWS * (CODE_B + GPS);  // 17,408
constexpr int MAX_NSTAGE = 8;
constexpr int FUSED_MAX_PAIRS = 256;
constexpr int MAX_PASS_U = 8;                    // longest gate/up pass
constexpr int MAX_PASS_D = 4;                    // longest down pass
constexpr int QD = 4;                            // claimed-item queue depth (fused)
constexpr int UNITS_IN_FLIGHT = 6;               // weight stages (of one packed unit) in flight per SM
constexpr int GU_SPLIT = 8;                      // gate/up passes of this many (row, unit) items or more:
                                                 // epilogue run by the consumer warps

enum { PH_UPC = 1, PH_DOWN = 2, PH_FUSED = 3 };

// Shape of a kernel instance whose passes hold at most MAXR rows.
template <int MAXR>
struct Cfg {
  static constexpr int NCW = MAXR <= 1 ? 8 : 16;     // consumer warps
  static constexpr int UPI = NCW / 8;                // packed units (64 weight rows each) per item
  static constexpr int NSTG = 2;                     // stager warps (alternate stages)
  static constexpr int NT = NCW * kWarp + (2 + NSTG) * kWarp;  // + producer, stagers and epilogue warps
  static constexpr int MINB = MAXR <= 1 ? 2 : 1;     // resident CTAs per SM
  static constexpr int W_PROD = NCW, W_HELP = NCW + 1, W_EPI = NCW + 1 + NSTG;
};

// Bytes per activation row of a stage in a slot, converted (f16, or fp32 for the bf16 down
// passes, the bf16 kind reserving the larger), and of its group multipliers.
template <int KIND>
struct SlotRow {
  static constexpr int ACT = KIND == TFX_ACT_E4M3 ? 2 * KC : 4 * KC;
  static constexpr int XM = 4 * GPS;
};

struct Proj {
  int K, S, G, units;  // reduction length, stages, groups, packed units per expert
  size_t unit_bytes, expert_bytes;
  const uint8_t* w;
};

struct RowsParams {
  int H, I, E, k, R;
  Proj pu, pd;
  int cap_u, cap_d;     // longest pass of gate/up and of down (rows)
  int nstage;           // ring slots
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
                        //        active expert, [E+2..2E+1] stager passes of down units past their
                        //        wait per active expert, then [R][H/64] slots written per (row, block)
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
// bars: full[8], empty[8], efull[2], eempty[2], qfull[4], qempty[4], hdone[2]; ctrl: abort flag and the
// claimed-item queue; epi: two result buffers [maxr][64 upi] fp32; route: the fused launch's
// lists; then the ring of slots: [upi weight stages | maxr converted activation rows | maxr x 16
// group multipliers].
struct Layout {
  int bars, ctrl, epi, route, ring, slot, w, act, xm, total;
};
__host__ __device__ inline Layout layout_of(const RowsParams& p, int maxr, int upi, int act_row) {
  Layout L;
  L.bars = 0;
  L.ctrl = 384;
  L.epi = 512;
  L.route = L.epi + 2 * maxr * 64 * upi * 4;
  L.ring = (L.route + 4 * p.route_ints + 127) & ~127;
  L.w = 0;
  L.act = upi * STAGE_B;
  L.xm = L.act + maxr * act_row;
  L.slot = (L.xm + maxr * 4 * GPS + 127) & ~127;
  L.total = L.ring + p.nstage * L.slot;
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

// Byte offset, in a converted activation row of one stage, of local group g (0..15) and
// 8-element chunk tc: chunk ((g/8)*4 + tc)*8 + g%8 of 16 bytes, so the eight lanes that read
// one chunk index of eight consecutive groups touch 128 consecutive bytes. fp32 rows split each
// chunk into halves hf of four values: 16-byte piece (((g/8)*4 + tc)*2 + hf)*8 + g%8, so that
// each 16-byte read of eight lanes is again 128 consecutive bytes.
__device__ __forceinline__ int xoff(int g, int tc) { return ((((g >> 3) * 4 + tc) * 8 + (g & 7)) << 4); }
__device__ __forceinline__ int xoff32(int g, int tc, int hf) {
  return (((((g >> 3) * 4 + tc) * 2 + hf) * 8 + (g & 7)) << 4);
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

// Convert one stage (512 k from k0 = 512 s) of t activation rows, read from global memory, into
// a slot's converted rows and group multipliers (the calling warp). Row r is X8 row rw[r]
// (K elements) with scales XS row rw[r] (G = K/32); every load of the stage is issued before
// its conversions, so that a stage costs one memory latency. The stage covers local groups g < gv =
// min(16, G - 16 s) with data; later groups are zero with multiplier 1, so that lanes past the
// end of the reduction add +0 to their accumulators. COH: the rows were written in this launch
// (h of the fused down passes) and are read at L2; else (x) they may stay in L1.
//   MODE 0 (E4M3): codes -> f16 (exact); multipliers from the E8M0 scales.
//   MODE 1 (bf16): one lane per 32-group shifts it by 2^sigma, mapping its largest magnitude
//     into [2^15, 2^16): the group is exact in f16 and its chain equals the unshifted fp32
//     chain times 2^sigma when every finite nonzero value has exponent in [e_max - 32, e_max],
//     e_max <= 119 and e_min >= -141 (products and partial sums then stay in fp32's normal
//     range, or on its subnormal grid, on both sides); the multiplier is 2^-sigma then, else 0,
//     which sends the group to the exact fallback.
//   MODE 2 (bf16 as fp32): values unshifted in 32-byte chunks, multiplier 1.
template <bool COH, typename V>
__device__ __forceinline__ V ld_act(const void* p) {
  return COH ? __ldcg(reinterpret_cast<const V*>(p)) : __ldg(reinterpret_cast<const V*>(p));
}
// Row rr of MR row indices held in registers (rr uniform per call site, so no local memory).
template <int MR>
__device__ __forceinline__ int pick_row(const int (&rw)[MR], int rr) {
  int v = rw[0];
#pragma unroll
  for (int r = 1; r < MR; ++r) v = rr == r ? rw[r] : v;
  return v;
}
// A stage's activation data in registers, between its loads and its conversion.
template <int KIND, int MODE, int MR>
struct StageRegs {
  static constexpr int NQ = (MR + 1) / 2;           // items of (row, group) a lane holds (MODE 1)
  uint2 v0[MODE == 0 ? MR : 1][2];                  // MODE 0: codes
  uint32_t sv[MODE == 0 ? NQ : 1];                  // MODE 0: scale codes
  // MODE 1 (bf16 rows shifted into f16) keeps nothing here: its loads run in the store phase,
  // two (row, group) items at a time, to bound the registers
  uint4 v2[MODE == 2 ? MR : 1][2];                  // MODE 2: bf16 chunks
};

template <int KIND, int MODE, bool COH, int MR>
__device__ __forceinline__ void stage_load(StageRegs<KIND, MODE, MR>& R_, const uint8_t* X8, const uint8_t* XS,
                                           int t, int s, int K, int G, const int (&rw)[MR], int lane) {
  constexpr int AB = KIND == TFX_ACT_E4M3 ? 1 : 2;
  const int gv = min(GPS, G - GPS * s);
  const size_t koff = (size_t)KC * s * AB;
  if (MODE == 0) {
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      const uint8_t* rr = X8 + (size_t)rw[r] * K + koff;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
        R_.v0[r][h] = make_uint2(0u, 0u);
        if (r < t && (c >> 2) < gv) R_.v0[r][h] = ld_act<COH, uint2>(rr + 8 * c);
      }
    }
#pragma unroll
    for (int q = 0; q < StageRegs<KIND, MODE, MR>::NQ; ++q) {
      const int r = 2 * q + (lane >> 4), g = lane & 15;
      R_.sv[q] = 127u;
      if (r < t && g < gv) R_.sv[q] = ld_act<COH, uint8_t>(XS + (size_t)pick_row(rw, r) * G + GPS * s + g);
    }
  } else if (MODE == 1) {
    // loaded in stage_store
  } else {
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      const uint8_t* rr = X8 + (size_t)rw[r] * K * AB + koff;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h;
        R_.v2[r][h] = make_uint4(0u, 0u, 0u, 0u);
        if (r < t && (c >> 2) < gv) R_.v2[r][h] = ld_act<COH, uint4>(rr + 16 * c);
      }
    }
  }
}

template <int KIND, int MODE, bool COH, int MR>
__device__ __forceinline__ void stage_store(const StageRegs<KIND, MODE, MR>& R_, uint8_t* act, int act_stride,
                                            float* xm, int xm_stride, int t, int s, int K, int G, const uint8_t* X8,
                                            const int (&rw)[MR], int lane) {
  constexpr int AB = KIND == TFX_ACT_E4M3 ? 1 : 2;
  const int gv = min(GPS, G - GPS * s);
  const size_t koff = (size_t)KC * s * AB;
  if (MODE == 0) {
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      if (r >= t) break;
      uint8_t* ar = act + r * act_stride;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h, g = c >> 2, tc = c & 3;
        uint4 o;
        o.x = e4m3x2_to_f16x2(R_.v0[r][h].x);
        o.y = e4m3x2_to_f16x2(R_.v0[r][h].x >> 16);
        o.z = e4m3x2_to_f16x2(R_.v0[r][h].y);
        o.w = e4m3x2_to_f16x2(R_.v0[r][h].y >> 16);
        *reinterpret_cast<uint4*>(ar + xoff(g, tc)) = o;
      }
    }
#pragma unroll
    for (int q = 0; q < StageRegs<KIND, MODE, MR>::NQ; ++q) {
      const int r = 2 * q + (lane >> 4), g = lane & 15;
      if (r < t) xm[r * xm_stride + g] = g < gv ? e8m0_to_f32(R_.sv[q]) : 1.0f;
    }
  } else if (MODE == 1) {
    constexpr int NQ = StageRegs<KIND, MODE, MR>::NQ;
#pragma unroll
    for (int q0 = 0; q0 < NQ; q0 += 2) {
     uint4 v[2][4];
#pragma unroll
     for (int u = 0; u < 2; ++u) {
      const int r = 2 * (q0 + u) + (lane >> 4), g = lane & 15;
#pragma unroll
      for (int k = 0; k < 4; ++k) v[u][k] = make_uint4(0u, 0u, 0u, 0u);
      if (q0 + u < NQ && r < t && g < gv) {
        const uint8_t* src = X8 + (size_t)pick_row(rw, r) * K * AB + koff + 64 * g;
#pragma unroll
        for (int k = 0; k < 4; ++k) v[u][k] = ld_act<COH, uint4>(src + 16 * k);
      }
     }
#pragma unroll
     for (int u = 0; u < 2; ++u) {
      const int r = 2 * (q0 + u) + (lane >> 4), g = lane & 15;
      if (q0 + u >= NQ || r >= t) continue;
      const uint32_t* wv = reinterpret_cast<const uint32_t*>(v[u]);
      // the exponents of the largest and of the smallest nonzero finite magnitude (magnitude
      // bits order like the values); NaN, Inf and zeros take no part
      uint32_t mxb = 0u, mnb = 0xFFFFu;
#pragma unroll
      for (int jj = 0; jj < 32; ++jj) {
        const uint32_t mag = (wv[jj >> 1] >> (16 * (jj & 1))) & 0x7FFFu;
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
      uint8_t* ar = act + r * act_stride;
#pragma unroll
      for (int tc = 0; tc < 4; ++tc) {
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint32_t two = wv[4 * tc + k];
          float lo = __uint_as_float(two << 16), hi = __uint_as_float(two & 0xFFFF0000u);
          if (safe) {
            lo = __fmul_rn(__fmul_rn(lo, f1), f2);
            hi = __fmul_rn(__fmul_rn(hi, f1), f2);
          }
          const __half2 h2 = __floats2half2_rn(lo, hi);
          o[k] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        *reinterpret_cast<uint4*>(ar + xoff(g, tc)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
      float m = 0.0f;  // 0 marks the exact fallback
      if (g >= gv) m = 1.0f;
      else if (safe) {
        const int ns = -sigma;  // 2^-sigma, possibly subnormal (exact)
        m = ns >= -126 ? __uint_as_float((uint32_t)(127 + ns) << 23) : __uint_as_float(0x00400000u >> (-127 - ns));
      }
      xm[r * xm_stride + g] = m;
     }
    }
  } else {
#pragma unroll
    for (int r = 0; r < MR; ++r) {
      if (r >= t) break;
      uint8_t* ar = act + r * act_stride;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int c = lane + 32 * h, g = c >> 2, tc = c & 3;
        const uint4 v = R_.v2[r][h];
        uint4 o0, o1;
        o0.x = v.x << 16;
        o0.y = v.x & 0xFFFF0000u;
        o0.z = v.y << 16;
        o0.w = v.y & 0xFFFF0000u;
        o1.x = v.z << 16;
        o1.y = v.z & 0xFFFF0000u;
        o1.z = v.w << 16;
        o1.w = v.w & 0xFFFF0000u;
        *reinterpret_cast<uint4*>(ar + xoff32(g, tc, 0)) = o0;
        *reinterpret_cast<uint4*>(ar + xoff32(g, tc, 1)) = o1;
      }
      if (lane < GPS) xm[r * xm_stride + lane] = 1.0f;
    }
  }
}

// Row lists of a small launch, computed in shared memory (fused layer): per-pair expert (or -1
// if left out), per-expert counts -> offsets, active experts, stable positions, per-row slot
// counts; then the pass lists of both projections (expert-major: the first active expert's
// passes, then the second's, ...). All NT threads take part. Ints used: fused_route_ints(E, R, k).
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
    // Pass lists (warp 1: gate/up, warp 2: down), expert-major: a warp scan of the pass counts
    // places each expert's passes.
    const bool down = warp == 2;
    const int cap = down ? p.cap_d : p.cap_u;
    int* list = down ? rt.plist_d : rt.plist_u;
    uint16_t* np = down ? rt.np_d : rt.np_u;
    const int na = *rt.nact;
    for (int a = lane; a < na; a += 32) {
      const int e = rt.act[a];
      np[a] = (uint16_t)passes_of(rt.offs[e + 1] - rt.offs[e], cap, p.tier_mode, down);
    }
    __syncwarp();
    int count = 0;
    for (int a0 = 0; a0 < na; a0 += 32) {
      const int a = a0 + lane;
      const int v = a < na ? (int)np[a] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (a < na) {
        const int e = rt.act[a];
        for (int b = 0; b < v; ++b) {
          int start, real, t;
          pass_rows(rt.offs[e + 1] - rt.offs[e], b, cap, p.tier_mode, down, start, real, t);
          list[count + incl - v + b] = pack_pass(a, start, real, t);
        }
      }
      count += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) rt.nlist[down ? 1 : 0] = count;
  }
  __syncthreads();
}

// ---------------------------------------------------------------- one pass of T rows
// Barriers of the shared-memory handoffs between the roles.
struct Bars {
  uint64_t *full, *empty;   // ring slots: producer (weights landed) and stager (activations
                            // converted) -> consumers; consumers -> producer and stager
  uint64_t *efull, *eempty; // result buffers: consumers -> epilogue, epilogue -> consumers
  uint64_t* hdone;           // gate/up: the consumers' h stores of a pass are out -> epilogue
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

// L2 policy for data read once: evicted before anything else, so that the kernel's code and
// the data it reuses stay resident while the weight stream passes through.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// One-dimensional bulk copy global -> shared with an L2 cache policy (as bulk_g2s).
__device__ __forceinline__ void bulk_g2s_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(pol)
      : "memory");
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

// Consumers: consume the pass's S stages, then hand the eight-way-tree results of every real
// row to the epilogue warp in epi[r][0..64 upi): lane (o = 4 warp + lane / 8, j = lane % 8)
// owns rows rr = o % 32 and 32 + rr of packed unit o / 32 of the item (the gate and up rows of
// one output, or two down rows), results at 64 (o / 32) + rr and + 32. SEQ: the two groups of
// a stage run one after the other (fewer live registers for long passes); else interleaved.
template <int KIND, int T, int UPI, bool X32, bool SEQ>
__device__ __forceinline__ void run_pass(const RowsParams& P, const Proj& pj, const uint8_t* smem, const Layout& Ly,
                                         const Bars& B, int be, uint32_t eph, bool ewait, volatile int* abort_flag,
                                         const int* r_prow, int pos, int real, bool dn, uint32_t& it, bool& dead,
                                         float* epi) {
  using SR = SlotRow<KIND>;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int j = lane & 7, o = (warp << 2) | (lane >> 3);
  const int uu = o >> 5, rr = o & 31;
  constexpr int XB = X32 ? 2 : 1;  // converted bytes per f16 position
  float acc0[T], acc1[T];
#pragma unroll
  for (int r = 0; r < T; ++r) {
    acc0[r] = 0.0f;
    acc1[r] = 0.0f;
  }
  constexpr int xrs = SlotRow<KIND>::ACT;  // bytes per activation row of a slot
  constexpr int xms = GPS;                  // multipliers per row
  const uint8_t* ring = smem + Ly.ring;
  // group multiplier m of row r and local group g, and the fallback's exact chain for bf16
  auto fold = [&](int r, int g, float p0, float p1, float s0, float s1, uint4 c0, uint4 c1, const float* xm,
                  int gglob) {
    const float m = xm[r * xms + g];
    if (KIND == TFX_ACT_E4M3) {
      acc0[r] = __fmaf_rn(p0, __fmul_rn(s0, m), acc0[r]);
      acc1[r] = __fmaf_rn(p1, __fmul_rn(s1, m), acc1[r]);
    } else {
      float q0, q1;
      if (!X32 && m == 0.0f) {
        const int src = pos + min(r, real - 1);
        const uint16_t* xrow = reinterpret_cast<const uint16_t*>(dn ? P.h : P.x) + (size_t)(dn ? src : r_prow[src]) * pj.K;
        q0 = chain_bf16_exact(c0, xrow, gglob);
        q1 = chain_bf16_exact(c1, xrow, gglob);
      } else {
        q0 = __fmul_rn(p0, m);
        q1 = __fmul_rn(p1, m);
      }
      acc0[r] = __fmaf_rn(q0, s0, acc0[r]);
      acc1[r] = __fmaf_rn(q1, s1, acc1[r]);
    }
  };
  // one group's chains of both columns for every row: p += w * x over the group's 32 k in order
  auto chains = [&](const uint32_t* w0, const uint32_t* w1, const uint8_t* xg, float (&p0)[T], float (&p1)[T]) {
#pragma unroll
    for (int tc = 0; tc < 4; ++tc) {
      uint32_t a0[4], a1[4];
      e2m1x8_to_f16x2(w0[tc], a0[0], a0[1], a0[2], a0[3]);
      e2m1x8_to_f16x2(w1[tc], a1[0], a1[1], a1[2], a1[3]);
#pragma unroll
      for (int r = 0; r < T; ++r) {
        const uint8_t* xp = xg + r * xrs + XB * tc * 128;
        if (X32) {
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const float4 xa = *reinterpret_cast<const float4*>(xp + 128 * hf);
#pragma unroll
            for (int ii = 0; ii < 2; ++ii) {
              const int i = 2 * hf + ii;
              const float lo = ii ? xa.z : xa.x, hi = ii ? xa.w : xa.y;
              const __half2 h0 = *reinterpret_cast<const __half2*>(&a0[i]);
              const __half2 h1 = *reinterpret_cast<const __half2*>(&a1[i]);
              p0[r] = __fmaf_rn(__low2float(h0), lo, p0[r]);
              p0[r] = __fmaf_rn(__high2float(h0), hi, p0[r]);
              p1[r] = __fmaf_rn(__low2float(h1), lo, p1[r]);
              p1[r] = __fmaf_rn(__high2float(h1), hi, p1[r]);
            }
          }
        } else {
          const uint4 xa = *reinterpret_cast<const uint4*>(xp);
          const uint32_t* va = reinterpret_cast<const uint32_t*>(&xa);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            p0[r] = fma2_f16(a0[i], va[i], p0[r]);
            p1[r] = fma2_f16(a1[i], va[i], p1[r]);
          }
        }
      }
    }
  };
  // ring position, advanced incrementally (no division per stage)
  const int NST = P.nstage;
  int slot = (int)(it % (uint32_t)NST);
  uint32_t ph = (it / (uint32_t)NST) & 1u;
  for (int s = 0; s < pj.S; ++s, ++it, slot = slot + 1 == NST ? 0 : slot + 1, ph ^= slot == 0 ? 1u : 0u) {
    if (warp_wait(&B.full[slot], ph, P, abort_flag, dead)) {
      const uint8_t* sb = ring + (size_t)slot * Ly.slot;
      const uint8_t* tile = sb + uu * STAGE_B;
      const uint8_t* sc = tile + TROWS * CODE_B;
      const uint8_t* xa_base = sb + Ly.act + 16 * j;  // f16 chunks: xoff; fp32 halves: xoff32
      const float* xm = reinterpret_cast<const float*>(sb + Ly.xm);
      const uint4 cA0 = *reinterpret_cast<const uint4*>(tile + rr * CODE_B + 16 * j);
      const uint4 cA1 = *reinterpret_cast<const uint4*>(tile + (32 + rr) * CODE_B + 16 * j);
      const float sA0 = e8m0_lookup(sc[rr * GPS + j]), sA1 = e8m0_lookup(sc[(32 + rr) * GPS + j]);
      if (SEQ) {
        float p0[T], p1[T];
#pragma unroll
        for (int r = 0; r < T; ++r) { p0[r] = 0.0f; p1[r] = 0.0f; }
        chains(reinterpret_cast<const uint32_t*>(&cA0), reinterpret_cast<const uint32_t*>(&cA1), xa_base, p0, p1);
#pragma unroll
        for (int r = 0; r < T; ++r) fold(r, j, p0[r], p1[r], sA0, sA1, cA0, cA1, xm, s * GPS + j);
        const uint4 cB0 = *reinterpret_cast<const uint4*>(tile + rr * CODE_B + 128 + 16 * j);
        const uint4 cB1 = *reinterpret_cast<const uint4*>(tile + (32 + rr) * CODE_B + 128 + 16 * j);
        const float sB0 = e8m0_lookup(sc[rr * GPS + 8 + j]), sB1 = e8m0_lookup(sc[(32 + rr) * GPS + 8 + j]);
#pragma unroll
        for (int r = 0; r < T; ++r) { p0[r] = 0.0f; p1[r] = 0.0f; }
        chains(reinterpret_cast<const uint32_t*>(&cB0), reinterpret_cast<const uint32_t*>(&cB1), xa_base + XB * 512,
               p0, p1);
#pragma unroll
        for (int r = 0; r < T; ++r) fold(r, j + 8, p0[r], p1[r], sB0, sB1, cB0, cB1, xm, s * GPS + 8 + j);
      } else {
        const uint4 cB0 = *reinterpret_cast<const uint4*>(tile + rr * CODE_B + 128 + 16 * j);
        const uint4 cB1 = *reinterpret_cast<const uint4*>(tile + (32 + rr) * CODE_B + 128 + 16 * j);
        const float sB0 = e8m0_lookup(sc[rr * GPS + 8 + j]), sB1 = e8m0_lookup(sc[(32 + rr) * GPS + 8 + j]);
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
            const uint8_t* xp = xa_base + r * xrs + XB * tc * 128;
            if (X32) {
#pragma unroll
              for (int hf = 0; hf < 2; ++hf) {  // four values of each group at a time
                const float4 xa = *reinterpret_cast<const float4*>(xp + 128 * hf);
                const float4 xb = *reinterpret_cast<const float4*>(xp + 1024 + 128 * hf);
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
          fold(r, j, pA0[r], pA1[r], sA0, sA1, cA0, cA1, xm, s * GPS + j);
          fold(r, j + 8, pB0[r], pB1[r], sB0, sB1, cB0, cB1, xm, s * GPS + 8 + j);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.empty[slot]);
  }
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
        epi[r * 64 * UPI + 64 * uu + rr] = v0r[r];
        epi[r * 64 * UPI + 64 * uu + 32 + rr] = v1r[r];
      }
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&B.efull[be]);
}

template <int KIND, int MAXR, bool DOWN, int UPI>
__device__ __forceinline__ void dispatch_pass(int t, const RowsParams& P, const Proj& pj, const uint8_t* smem,
                                              const Layout& Ly, const Bars& B, int be, uint32_t eph, bool ewait,
                                              volatile int* abort_flag, const int* r_prow, int pos, int real,
                                              uint32_t& it, bool& dead, float* epi) {
  constexpr int LIM = DOWN ? (MAXR < MAX_PASS_D ? MAXR : MAX_PASS_D) : MAXR;
  constexpr bool X32 = DOWN && KIND == TFX_ACT_BF16;
#define TFX_PASS(TT)                                                                                         \
  if constexpr (TT <= LIM)                                                                                   \
    run_pass<KIND, TT, UPI, X32, (TT > 4)>(P, pj, smem, Ly, B, be, eph, ewait, abort_flag, r_prow, pos, real, \
                                           DOWN, it, dead, epi)
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

// One pass as the epilogue warp sees it (all fields warp-uniform).
struct HPass {
  bool dn, last;
  int a, ub, nu, real, pidx;  // ub: first packed unit of the item, nu: its units
  int pair[8];
};

// The gate/up epilogue of items i0, i0 + DI, ... of a pass (item i: row i / nu, unit i % nu),
// by the calling warp, four items at a time so that their latency chains overlap: SwiGLU, the
// activation quantiser and h (+ debug copies), from result buffer epi.
template <int KIND, int UPI, int DI>
__device__ __forceinline__ void gu_items(const RowsParams& P, const HPass& q, const float* epi, int i0) {
  const int lane = threadIdx.x & 31;
  const int n_items = q.real * q.nu;
  const int I = P.I;
  for (int ib = i0; ib < n_items; ib += 4 * DI) {
    float g[4], u[4], hv[4];
    int pp[4], nn[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int i = ib + c * DI;
      if (i >= n_items) break;
      const int r = i / q.nu, uu = i - r * q.nu;
      const float* er = epi + r * 64 * UPI + 64 * uu;
      pp[c] = q.pair[r];
      nn[c] = 32 * (q.ub + uu) + lane;
      g[c] = er[lane];
      u[c] = er[32 + lane];
      const float den = __fadd_rn(1.0f, expf(-g[c]));
      hv[c] = __fmul_rn(__fdiv_rn(g[c], den), u[c]);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      if (ib + c * DI >= n_items) break;
      const size_t p = (size_t)pp[c];
      if (P.gu_dbg) {
        P.gu_dbg[p * 2 * I + nn[c]] = g[c];
        P.gu_dbg[p * 2 * I + I + nn[c]] = u[c];
      }
      if (P.h_dbg) P.h_dbg[p * I + nn[c]] = hv[c];
      if (KIND == TFX_ACT_E4M3) {
        const bool bad = __any_sync(0xffffffffu, isnan(hv[c]) || isinf(hv[c]));
        const uint32_t amax_b = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv[c])));
        uint32_t sc;
        if (bad) sc = 255u;
        else if (amax_b == 0u) sc = 127u;
        else {
          const int e2 = amax_b >= 0x00800000u ? (int)(amax_b >> 23) - 127 : (31 - __clz((int)amax_b)) - 149;
          sc = (uint32_t)min(max(e2 - 8 + 127, 0), 254);
        }
        const uint32_t code = bad ? 0x7Fu : f32_to_e4m3(__fmul_rn(hv[c], e8m0_recip_f32(sc)));
        static_cast<uint8_t*>(P.h)[p * I + nn[c]] = (uint8_t)code;
        if (lane == 0) P.hs[p * (I / 32) + (nn[c] >> 5)] = (uint8_t)sc;
      } else {
        static_cast<__nv_bfloat16*>(P.h)[p * I + nn[c]] = __float2bfloat16_rn(hv[c]);
      }
    }
  }
}

// Epilogue warp: the epilogue of one pass. Gate/up: in instances whose passes can reach GU_SPLIT
// items (CSPLIT), such passes were run by the consumer warps themselves and this warp waits on
// hdone until they are through (their h stores out); other passes it runs here, from result
// buffer epi. It then frees the buffer and, in fused launches, publishes a finished gate/up unit
// (a release fence, then the expert's counter). Down: from result buffer epi, the expert outputs d; fused launches then count each
// (row, 64-output block) written, with one fence for the whole pass, and combine the blocks
// whose last slot this pass wrote.
template <int KIND, int PH, int UPI, bool CSPLIT>
__device__ void helper_epilogue(const RowsParams& P, const HPass& q, const Bars& B, const float* epi,
                                const int* r_prow, const int* r_pslot, const int* r_rowcnt, int32_t* done_upc,
                                int32_t* slots_done, volatile int* abort_flag, bool& dead) {
  const int lane = threadIdx.x & 31;
  const int be = q.pidx & 1;
  warp_wait(q.dn || !CSPLIT ? &B.efull[be] : &B.hdone[be], (q.pidx >> 1) & 1, P, abort_flag, dead);
  const int n_items = q.real * q.nu;  // item i: row i / nu, unit i % nu
  if (!q.dn) {
    if (!dead && (!CSPLIT || n_items < GU_SPLIT)) gu_items<KIND, UPI, 1>(P, q, epi, 0);
  } else if (!dead) {
    bool bad = false;
    for (int i = 0; i < n_items; ++i) {
      const int r = i / q.nu, uu = i - r * q.nu;
      const int p = q.pair[r], row = r_prow[p], slot = r_pslot[p];
      if (row >= 0 && row < P.R && slot >= 0 && slot < P.k) {
        const float* er = epi + r * 64 * UPI + 64 * uu;
        float* dst = P.out + ((size_t)row * P.k + slot) * P.H + 64 * (q.ub + uu);
        dst[lane] = er[lane];
        dst[32 + lane] = er[32 + lane];
      } else {
        bad = true;
      }
    }
    if (bad && lane == 0) report(P.status, TFX_ST_SHAPE);
    if (PH == PH_FUSED) {
      // combine (row, block) in the CTA that writes the row's last slot
      __threadfence();
      __syncwarp();
      int last = 0, ctr = -1, row = -1, blk = 0;
      if (lane < n_items) {
        const int r = lane / q.nu, uu = lane - r * q.nu;
        const int p = q.pair[r];
        row = r_prow[p];
        const int slot = r_pslot[p];
        blk = q.ub + uu;
        if (row >= 0 && row < P.R && slot >= 0 && slot < P.k) {
          ctr = row * P.pd.units + blk;
          last = atomicAdd(&slots_done[ctr], 1) == r_rowcnt[row] - 1;
          if (last) slots_done[ctr] = 0;  // last user of the counter
        }
      }
      unsigned lm = __ballot_sync(0xffffffffu, last);
      if (lm) {
        __threadfence();
        while (lm) {
          const int src = __ffs(lm) - 1;
          lm &= lm - 1;
          const int rw = __shfl_sync(0xffffffffu, row, src), bk = __shfl_sync(0xffffffffu, blk, src);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int m = 64 * bk + 32 * hh + lane;
            float yv = 0.0f;
            for (int jj = 0; jj < P.k; ++jj)
              yv = __fmaf_rn(P.topk_w[(size_t)rw * P.k + jj], __ldcg(P.out + ((size_t)rw * P.k + jj) * P.H + m), yv);
            P.y[(size_t)rw * P.H + m] = __bfloat16_as_ushort(__float2bfloat16_rn(yv));
            if (P.y32) P.y32[(size_t)rw * P.H + m] = yv;
          }
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
// (blockIdx.x + i * gridDim.x; an item is (active expert, UPI packed units of outputs), its
// passes sized by the rows left). Fused launch: the claimed work units, each one pass: unit
// i < n_upc is gate/up pass list entry i / items, item i % items (items = units of an expert
// in groups of UPI); the down units follow.
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
template <int PH, int UPI, typename NextItem>
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
      const int items = (pj.units + UPI - 1) / UPI;
      const int q = li / items, u = li - q * items;
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
      const int items = (pj.units + UPI - 1) / UPI;
      const int a = li / items, u = li - a * items;
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
// Roles: the consumer warps compute; the next warp produces (weight stages and the pass's
// activation rows of each stage, by bulk copy); the next converts each stage's activations in
// its slot and completes the slot; the last runs each pass's epilogue (SwiGLU and quantisation
// of h, or the d rows and, in the fused launch, the combine) while the consumers go on.
template <int KIND, int MAXR_U, int MAXR_D, int PH>
struct RowsShape {
  static constexpr int MAXR = ((PH & PH_UPC) && MAXR_U > MAXR_D) || !(PH & PH_DOWN) ? MAXR_U : MAXR_D;
  using C = Cfg<MAXR>;
};

template <int KIND, int MAXR_U, int MAXR_D, int PH>
__global__ void __launch_bounds__(RowsShape<KIND, MAXR_U, MAXR_D, PH>::C::NT,
                                  RowsShape<KIND, MAXR_U, MAXR_D, PH>::C::MINB)
    rows_kernel(const RowsParams P) {
  using Sh = RowsShape<KIND, MAXR_U, MAXR_D, PH>;
  using C = typename Sh::C;
  using SR = SlotRow<KIND>;
  constexpr int MAXR = Sh::MAXR;
  constexpr int NCW = C::NCW, NT = C::NT, UPI = C::UPI;
  constexpr int AB = KIND == TFX_ACT_E4M3 ? 1 : 2;  // activation bytes per element
  // the 8-row instance (gate/up passes of up to 8 rows x 2 units): the consumers run the epilogues
  // of passes of GU_SPLIT items or more (hdone handshake); measured slower at fewer rows
  constexpr bool CSPLIT = (PH & PH_UPC) && MAXR_U >= 8 && MAXR_U * UPI >= GU_SPLIT;
  extern __shared__ __align__(128) uint8_t smem[];
  const Layout Ly = layout_of(P, MAXR, UPI, SR::ACT);
  Bars B;
  B.full = reinterpret_cast<uint64_t*>(smem + Ly.bars);
  B.empty = B.full + MAX_NSTAGE;
  B.efull = B.empty + MAX_NSTAGE;
  B.eempty = B.efull + 2;
  uint64_t* qfull = B.eempty + 2;  // fused: claimed-item queue, producer -> stager, epilogue, consumers
  uint64_t* qempty = qfull + QD;   //        and back
  B.hdone = qempty + QD;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Ly.ctrl);
  int* qid = reinterpret_cast<int*>(smem + Ly.ctrl + 16);    // [QD] claimed item ids
  float* epi = reinterpret_cast<float*>(smem + Ly.epi);      // [2][maxr][64 upi]
  uint8_t* ring = smem + Ly.ring;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NST = P.nstage;
  // the consumers' weight-scale table (1 KB) is brought into L1 while the row lists are built
  if (tid < (int)sizeof(E8m0Table) / 128) asm volatile("prefetch.global.L1 [%0];" ::"l"(e8m0_table.v + 32 * tid));
  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&B.full[s], 2);  // the producer's weights (with their bytes) and the stager
      mbar_init(&B.empty[s], NCW);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&B.efull[b], NCW);
      mbar_init(&B.eempty[b], 1);
    }
    for (int b = 0; b < QD; ++b) {
      mbar_init(&qfull[b], 1);
      mbar_init(&qempty[b], NCW + 1 + C::NSTG);
    }
    for (int b = 0; b < 2; ++b) mbar_init(&B.hdone[b], NCW);
    mbar_fence_init();
    *abort_flag = 0;
  }

  // row lists: computed here (fused) or read from a previous route launch
  const int *r_offs, *r_prow, *r_pslot, *r_act, *r_rowcnt = nullptr;
  const uint16_t *np_u = nullptr, *np_d = nullptr;  // fused: passes per active expert
  int n_act;
  SeqCtx sc;
  const int items_u = (P.pu.units + UPI - 1) / UPI, items_d = (P.pd.units + UPI - 1) / UPI;
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
    sc.n_upc = rt.nlist[0] * items_u;
    sc.total = sc.n_upc + rt.nlist[1] * items_d;
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
    sc.n_upc = (PH & PH_UPC) ? n_act * items_u : 0;
    sc.total = sc.n_upc + ((PH & PH_DOWN) ? n_act * items_d : 0);
  }
  sc.act = r_act;
  sc.offs = r_offs;
  int32_t* work_ctr = PH == PH_FUSED ? P.scratch + 1 : nullptr;
  int32_t* done_upc = PH == PH_FUSED ? P.scratch + 2 : nullptr;
  int32_t* down_seen = PH == PH_FUSED ? P.scratch + 2 + P.E : nullptr;
  int32_t* slots_done = PH == PH_FUSED ? P.scratch + 2 + 2 * P.E : nullptr;
  PassGen gen = {};
  PassDesc d;
  // the epilogue's view of a pass
  auto hpass_of = [&](const PassDesc& q) {
    HPass hp;
    hp.dn = q.dn;
    hp.last = q.last;
    hp.a = q.a;
    const Proj& pj = q.dn ? P.pd : P.pu;
    hp.ub = UPI * q.u;
    hp.nu = min(UPI, pj.units - hp.ub);
    hp.real = q.real;
    hp.pidx = q.pidx;
#pragma unroll
    for (int r = 0; r < 8; ++r) hp.pair[r] = q.pos + min(r, q.real - 1);
    return hp;
  };
  // rows of a pass: token rows (gate/up) or pair rows (down); padding repeats the last
  auto row_of = [&](const PassDesc& q, int r) {
    const int src = q.pos + min(r, q.real - 1);
    if (q.dn) return src;
    const int row = r_prow[src];
    return (row < 0 || row >= P.R) ? 0 : row;
  };
  // Separate launches stride over the items; the fused launch hands units out dynamically: the
  // producer claims them from a global counter, in order (gate/up units expert-major, then down
  // units), and passes them to the other roles through a small queue.
  int static_next = blockIdx.x - (int)gridDim.x;
  uint32_t qpos = 0;
  auto next_static = [&]() { static_next += gridDim.x; return static_next; };
  auto next_popped = [&]() {  // stager, epilogue and consumers (warp-wide)
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
      // every weight byte is read once a launch: evict it first, so that the code, the
      // activations, h, d and the counters stay in L2 while 23 MB an expert stream through
      // (measured: 0.4 us on the one-row layer, 2-4% on shared and apart layers)
      const uint64_t wpol = l2_evict_first_policy();
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
      // The queue runs one unit ahead of the producer, so the other roles learn of the next
      // unit while the current one streams. The next unit is claimed when the current unit's
      // last stage is issued: the ring still holds that unit's queued stages while the claim
      // returns, and the units left are handed to the CTAs that are closest to done. (Claimed
      // at a unit's first stage, the one-row layer's second gate/up wave went at start-up to
      // CTAs that finished their first unit up to 8 us apart: 4-5% slower.)
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
      while (!stop && gen_next<PH, UPI>(gen, d, P, sc, next_prod)) {
        const Proj& pj = d.dn ? P.pd : P.pu;
        const int ub = UPI * d.u, nu = min(UPI, pj.units - ub);
        const uint8_t* src = pj.w + (size_t)d.e * pj.expert_bytes + (size_t)ub * pj.unit_bytes;
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
          uint8_t* sb = ring + (size_t)slot * Ly.slot;
          mbar_arrive_expect_tx(&B.full[slot], (uint32_t)(nu * STAGE_B));
          for (int v = 0; v < nu; ++v)
            bulk_g2s_hint(sb + v * STAGE_B, src + (size_t)v * pj.unit_bytes + (size_t)s * STAGE_B, STAGE_B, &B.full[slot],
                          wpol);
          if (PH == PH_FUSED && s == pj.S - 1) claim_pending();
        }
      }
      if (PH == PH_FUSED) claim_pending();
      if (PH == PH_FUSED && !gen.done) {
        // stopped early (abort): tell the other roles there is nothing more
        *abort_flag = 1;
        for (int q = 0; q < 2 * QD && !gen.done; ++q) {
          const int slot = claims % QD;
          mbar_wait(&qempty[slot], ((claims / QD) & 1) ^ 1, 1000000ull);
          qid[slot] = -1;
          mbar_arrive(&qfull[slot]);
          ++claims;
        }
      }
      // Drain: every issued stage must have landed before the block may exit (the slot's phase
      // also needs the stager, which completes it unless the block aborted).
      const uint32_t first = it > (uint32_t)NST ? it - NST : 0u;
      for (uint32_t q = first; q < it; ++q) {
        if (!mbar_wait(&B.full[q % NST], (q / NST) & 1u, P.timeout_ns)) {
          report(P.status, TFX_ST_TIMEOUT);
          break;
        }
      }
    }
  } else if (warp >= C::W_HELP && warp < C::W_HELP + C::NSTG) {
    // ---------------------------------------------------------------- stagers
    // Stager sid converts the stages whose running index is sid modulo NSTG, so that one
    // stage's loads are in flight while another converts.
    const int sid = warp - C::W_HELP;
    bool dead = false;

    uint32_t it = 0;
    auto next_h = [&]() { return PH == PH_FUSED ? next_popped() : next_static(); };
    while (gen_next<PH, UPI>(gen, d, P, sc, next_h)) {
      const Proj& pj = d.dn ? P.pd : P.pu;
      const uint8_t* X8 = d.dn ? static_cast<const uint8_t*>(P.h) : static_cast<const uint8_t*>(P.x);
      const uint8_t* XS = d.dn ? P.hs : P.xs;
      int rw[MAXR];  // the pass's rows (padding rows repeat the last real row)
#pragma unroll
      for (int r = 0; r < MAXR; ++r) rw[r] = row_of(d, min(r, d.t - 1));
      if (PH == PH_FUSED && d.dn && d.first && !dead) {
        // fused down: wait (bounded) until every gate/up unit of the expert has published its h
        int okw = 1;
        if (lane == 0) {
          const int need = np_u[d.a] * items_u;
          const uint64_t t0 = global_ns();
          while (true) {
            int v;
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(done_upc + d.a) : "memory");
            if (v >= need) break;
            if (*abort_flag || global_ns() - t0 > P.timeout_ns) {
              if (*abort_flag == 0) report(P.status, TFX_ST_TIMEOUT);
              *abort_flag = 1;
              okw = 0;
              break;
            }
            __nanosleep(64);
          }
          // every stager of every down unit of the expert counts itself past this wait; the last
          // one returns both counters to zero (no waiter can still be reading them then)
          if (okw && atomicAdd(down_seen + d.a, 1) == C::NSTG * np_d[d.a] * items_d - 1) {
            done_upc[d.a] = 0;
            down_seen[d.a] = 0;
          }
        }
        if (!__shfl_sync(0xffffffffu, okw, 0)) dead = true;
      }
      __syncwarp();
      for (int s = 0; s < pj.S; ++s, ++it) {
        if ((int)(it % C::NSTG) != sid) continue;
        const int slot = it % NST;
        const uint32_t ph = (it / NST) & 1u;
        // the stage's loads are issued first; the slot is free once the consumers have released
        // its previous use, and only then is it written
        auto run_stage = [&](auto mode_tag, auto coh_tag, const auto& rows) {
          constexpr int MODE = decltype(mode_tag)::value;
          constexpr bool COH = decltype(coh_tag)::value;
          constexpr int MR = sizeof(rows) / sizeof(int);
          StageRegs<KIND, MODE, MR> sr;
          if (!dead) stage_load<KIND, MODE, COH, MR>(sr, X8, XS, d.t, s, pj.K, pj.G, rows, lane);
          if ((it < (uint32_t)NST || warp_wait(&B.empty[slot], ph ^ 1u, P, abort_flag, dead)) && !dead) {
            uint8_t* sb = ring + (size_t)slot * Ly.slot;
            stage_store<KIND, MODE, COH, MR>(sr, sb + Ly.act, SR::ACT, reinterpret_cast<float*>(sb + Ly.xm), GPS, d.t, s,
                                             pj.K, pj.G, X8, rows, lane);
          }
        };
        if (KIND == TFX_ACT_E4M3) {
          if constexpr (MAXR_U >= 8) {
            // the 8-row instance stages x as it stages h (through L2): one copy of the staging
            // code instead of two (measured: 3-4% faster shared 5-16 rows, 17% apart 16 rows;
            // the smaller instances keep x in L1, one row 2% faster that way)
            run_stage(std::integral_constant<int, 0>(), std::true_type(), rw);
          } else if (d.dn) {
            run_stage(std::integral_constant<int, 0>(), std::true_type(), rw);
          } else {
            run_stage(std::integral_constant<int, 0>(), std::false_type(), rw);
          }
        } else if (d.dn) {
          int rwd[MAXR_D];
#pragma unroll
          for (int r = 0; r < MAXR_D; ++r) rwd[r] = rw[r];
          run_stage(std::integral_constant<int, 2>(), std::true_type(), rwd);
        } else {
          run_stage(std::integral_constant<int, 1>(), std::false_type(), rw);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.full[slot]);
      }
      __syncwarp();
    }
  } else if (warp == C::W_EPI) {
    // ---------------------------------------------------------------- epilogue
    bool dead = false;
    auto epilogue = [&](const PassDesc& q) {
      helper_epilogue<KIND, PH, UPI, CSPLIT>(P, hpass_of(q), B, epi + (q.pidx & 1) * (MAXR * 64 * UPI), r_prow, r_pslot,
                                     r_rowcnt, done_upc, slots_done, abort_flag, dead);
    };
    auto next_e = [&]() { return PH == PH_FUSED ? next_popped() : next_static(); };
    PassDesc q;
    while (gen_next<PH, UPI>(gen, q, P, sc, next_e)) epilogue(q);
  } else {
    // ---------------------------------------------------------------- consumers
    uint32_t it = 0;
    bool dead = false;
    auto next_c = [&]() { return PH == PH_FUSED ? next_popped() : next_static(); };
    while (gen_next<PH, UPI>(gen, d, P, sc, next_c)) {
      const Proj& pj = d.dn ? P.pd : P.pu;
      const int be = d.pidx & 1;
      float* ep = epi + be * (MAXR * 64 * UPI);
      const uint32_t eph = ((d.pidx >> 1) & 1) ^ 1;
      if constexpr (KIND == TFX_ACT_E4M3 && MAXR_D <= MAXR_U) {
        // E4M3 gate/up and down passes of up to MAXR_U rows are the same code (the down flag only
        // matters to bf16): one inlined copy of it, for the instruction cache (measured: 0.3-3%
        // faster layers)
        dispatch_pass<KIND, MAXR_U, false, UPI>(d.t, P, pj, smem, Ly, B, be, eph, d.pidx >= 2, abort_flag, r_prow,
                                                d.pos, d.real, it, dead, ep);
      } else if (d.dn) {
        dispatch_pass<KIND, MAXR_D, true, UPI>(d.t, P, pj, smem, Ly, B, be, eph, d.pidx >= 2, abort_flag, r_prow, d.pos,
                                               d.real, it, dead, ep);
      } else {
        dispatch_pass<KIND, MAXR_U, false, UPI>(d.t, P, pj, smem, Ly, B, be, eph, d.pidx >= 2, abort_flag, r_prow,
                                                d.pos, d.real, it, dead, ep);
      }
      // gate/up passes of GU_SPLIT or more (row, unit) items: once every consumer warp's results
      // are in the buffer, the consumers run the epilogue items themselves (a lone epilogue warp
      // gets few issue slots beside them); smaller passes leave them to the epilogue warp
      if constexpr (CSPLIT) {
        if (!d.dn && d.real * min(UPI, pj.units - UPI * d.u) >= GU_SPLIT &&
            warp_wait(&B.efull[be], (d.pidx >> 1) & 1, P, abort_flag, dead))
          gu_items<KIND, UPI, NCW>(P, hpass_of(d), ep, warp);
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.hdone[be]);
      }
    }
  }
}

// ------------------------------------------------------------------------------ host side

std::mutex& rows_mutex();
int dev_sms(int* sms, size_t* optin);

// Ring depth and blocks per SM, chosen once per (device, kernel instance, route size) and
// cached, so that steady-state launches (and launches under stream capture) issue only the
// kernel: about UNITS_IN_FLIGHT packed-unit stages in flight per SM (resident CTAs x slots x
// units per slot), then more resident CTAs.
template <int KIND, int MAXR_U, int MAXR_D, int PH>
int launch_rows(RowsParams P, int max_items, cudaStream_t st) {
  using Sh = RowsShape<KIND, MAXR_U, MAXR_D, PH>;
  using SR = SlotRow<KIND>;
  constexpr int MAXR = Sh::MAXR;
  constexpr int NT = Sh::C::NT, UPI = Sh::C::UPI;
  int sms;
  size_t optin;
  int rc = dev_sms(&sms, &optin);
  if (rc) return rc;
  auto kern = rows_kernel<KIND, MAXR_U, MAXR_D, PH>;
  struct Entry { int key_route, nst, nb; size_t smem; };
  static Entry cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TFX_ECUDA;
  Entry ent;
  {
    std::lock_guard<std::mutex> lk(rows_mutex());
    ent = cache[dev];
    if (ent.nb == 0 || ent.key_route != P.route_ints) {
      RowsParams q = P;
      q.nstage = MAX_NSTAGE;
      const size_t smax = (size_t)layout_of(q, MAXR, UPI, SR::ACT).total;
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)min(smax, optin)) != cudaSuccess)
        return TFX_ELAUNCH;
      Entry best = {};
      long best_score = -1;
      for (int nst = 2; nst <= MAX_NSTAGE; ++nst) {
        q.nstage = nst;
        const size_t sm = (size_t)layout_of(q, MAXR, UPI, SR::ACT).total;
        if (sm > optin) break;
        int nb = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, NT, sm) != cudaSuccess) return TFX_ELAUNCH;
        if (nb < 1) break;
        // about 6 packed units in flight per SM keep HBM busy; more only lengthen the queues
        // that the gate/up -> down dependency waits in (measured against 8: level on the
        // one-row layer, 1-6% faster on shared-row layers of 2-16 rows and 0.4-2% on bf16
        // layers of 4-16 rows apart, 3% slower on 2 rows apart)
        const int units = nb * nst * UPI;
        const long score = (units <= UNITS_IN_FLIGHT ? units * 100 : UNITS_IN_FLIGHT * 100 - (units - UNITS_IN_FLIGHT) * 10) + nb;
        if (score > best_score) {
          best_score = score;
          best = Entry{P.route_ints, nst, nb, sm};
        }
      }
      if (best_score < 0) return TFX_EUNSUPPORTED;
      ent = best;
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
