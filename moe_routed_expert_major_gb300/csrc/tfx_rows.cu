// tfx_rows.cu -- expert-major "rows" kernels: gate/up (+ SwiGLU + activation quantiser) and
// down, for launches of few rows per expert (decode).
//
// Method: "dsv41 metal: decode experts decode an expert's weights once for all of its rows"
// (TensorFold PR #2983). Each work item is (active expert, block of outputs). Its weights are
// streamed once per pass; every 32-group is decoded once and applied to every row of the pass
// (pass sized by the rows left, padding rows repeat the last real row, are computed and never
// written). Each row's accumulators follow the fixed order of "What this changes": per group
// a sequential fma chain of the 32 unscaled products from +0 in k order, one scaled fma into
// accumulator (group mod 8), then the eight-way tree.
//
// GB300 mapping:
//   * one producer warp streams 17,408-byte stages (64 weight rows x 512 k of codes + scales,
//     contiguous in the packed layout) into a ring of shared-memory slots with
//     cp.async.bulk + mbarrier (bounded waits);
//   * eight consumer warps; lane (t & 7) of an octet owns accumulator lane j = group mod 8 of
//     one output column pair, so the eight-way tree is three xor-shuffles;
//   * E2M1 codes are decoded with cvt.rn.f16x2.e2m1x2, activations are held in shared memory
//     as f16 (exact for E4M3; bf16 rows are shifted per 32-group by a power of two so that
//     they are exact in f16, with an exact fp32 fallback for groups that do not fit), and the
//     chain runs on fma.rn.f32.f16 (fp32 accumulate, one rounding per step).
#include <cuda_runtime.h>
#include <stdint.h>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <mutex>
#include <type_traits>

#include "tfx_common.cuh"

namespace tfx {

constexpr int KC = 512;                 // k per stage
constexpr int GPS = KC / 32;            // groups per stage
constexpr int TROWS = 64;               // weight rows per stage
constexpr int CODE_B = KC / 2;          // code bytes per row per stage
constexpr int STAGE_B = TROWS * (CODE_B + GPS);  // 17,408
constexpr int NCW = 8;                  // consumer warps
constexpr int NCONS = NCW * kWarp;      // 256
constexpr int NTHREADS = NCONS + kWarp; // + one producer warp
constexpr int MAX_NSTAGE = 8;

enum { MODE_UPC = 0, MODE_DOWN = 1 };

struct RowsParams {
  int H, I, E, k, R;
  int K, S, G, GB;     // reduction length, stages, groups, group-blocks of 8
  int units;           // output blocks per expert
  int nstage;
  size_t unit_bytes, expert_bytes;
  const uint8_t* w;    // packed weights of this projection
  const void* x;       // activations: upc -> token rows [R][H]; down -> pair rows [P][I]
  const uint8_t* xs;   // E8M0 scales of x (E4M3 launches)
  const int32_t *offs, *pair_row, *pair_slot, *active, *n_active;
  void* h;             // upc out: [P][I] (E4M3 codes or bf16)
  uint8_t* hs;         // upc out: [P][I/32]
  float* gu_dbg;       // upc debug [P][2][I]
  float* h_dbg;        // upc debug [P][I]
  float* out;          // down out: [R][k][H]
  int32_t* status;
  int max_pass, tier_mode;
  uint64_t timeout_ns;
};

// Shared-memory layout (dynamic), offsets in bytes.
struct Smem {
  static constexpr int BARS = 0;                       // full[8], empty[8]
  static constexpr int CTRL = 128;                     // abort flag, pass info
  static constexpr int PASS_ROW = 256;                 // int32 [8]: activation row of each pass row
  static constexpr int PASS_PAIR = 288;                // int32 [8]: pair index of each pass row
  static constexpr int EPI = 512;                      // float [8][64]
  static constexpr int RING = 2560;                    // 16-byte aligned
};

__host__ __device__ inline size_t smem_bytes(const RowsParams& p, int maxr) {
  size_t xs = (size_t)maxr * p.GB * 512;               // f16 activations, permuted
  size_t xm = (size_t)maxr * p.GB * 8 * 4;             // fp32 per-group multipliers
  return Smem::RING + (size_t)p.nstage * STAGE_B + xs + xm;
}

template <int MODE>
__device__ __forceinline__ int tier_of(int left, int maxr, int mode) {
  if (mode == 1) return maxr;
  int t;
  if (MODE == MODE_UPC) t = left >= 7 ? 8 : left >= 5 ? 6 : left >= 3 ? 4 : left >= 2 ? 2 : 1;
  else t = left >= 3 ? 4 : left >= 2 ? 2 : 1;
  return t > maxr ? maxr : t;
}

// Byte offset in the permuted activation layout of element k of pass row r: chunk
// ((r*GB + g/8)*4 + t/8)*8 + g%8 of 16 bytes, element t%8 inside it (g = k/32, t = k%32),
// so the eight lanes that read one chunk index for eight consecutive groups touch 128
// consecutive bytes.
__device__ __forceinline__ int xoff(int r, int g, int tc, int GB) {
  return ((((r * GB + (g >> 3)) * 4 + tc) * 8 + (g & 7)) << 4);
}

// Exact fp32 chain for a bf16 group whose values do not fit f16 after the shift: the
// group's 32 codes are decoded again, and each product of an E2M1 value (exact in fp32) with
// the bf16 value read back from global memory is accumulated in k order from +0.
__device__ __noinline__ float chain_bf16_exact(uint4 codes, const uint16_t* xrow, int g) {
  const uint32_t cw[4] = {codes.x, codes.y, codes.z, codes.w};
  float p = 0.0f;
  for (int q = 0; q < 4; ++q) {
    uint32_t h[4];
    e2m1x8_to_f16x2(cw[q], h[0], h[1], h[2], h[3]);
    for (int i = 0; i < 4; ++i) {
      const __half2 hw = *reinterpret_cast<const __half2*>(&h[i]);
      const int k = 32 * g + 8 * q + 2 * i;
      p = __fmaf_rn(__low2float(hw), __uint_as_float((uint32_t)xrow[k] << 16), p);
      p = __fmaf_rn(__high2float(hw), __uint_as_float((uint32_t)xrow[k + 1] << 16), p);
    }
  }
  return p;
}

// Stage the activation rows of one pass into shared memory (consumer threads only).
template <int KIND>
__device__ void stage_rows(const RowsParams& P, uint8_t* xs_s, float* xm_s, const int* prow, int real, int tid) {
  const int K = P.K, G = P.G, GB = P.GB;
  if (KIND == TFX_ACT_E4M3) {
    const uint8_t* X = static_cast<const uint8_t*>(P.x);
    const int nch = K / 8;
    for (int i = tid; i < real * nch; i += NCONS) {
      int r = i / nch, c = i - r * nch;
      const uint2 v = *reinterpret_cast<const uint2*>(X + (size_t)prow[r] * K + 8 * c);
      uint4 o;
      o.x = e4m3x2_to_f16x2(v.x);
      o.y = e4m3x2_to_f16x2(v.x >> 16);
      o.z = e4m3x2_to_f16x2(v.y);
      o.w = e4m3x2_to_f16x2(v.y >> 16);
      int g = c >> 2, tc = c & 3;
      *reinterpret_cast<uint4*>(xs_s + xoff(r, g, tc, GB)) = o;
    }
    for (int i = tid; i < real * G; i += NCONS) {
      int r = i / G, g = i - r * G;
      xm_s[r * GB * 8 + g] = e8m0_to_f32(P.xs[(size_t)prow[r] * G + g]);
    }
  } else {
    // bf16: a half-warp converts one 32-group (two values a lane), choosing a power-of-two
    // shift 2^sigma that maps the group's largest magnitude into [2^15, 2^16). The group is
    // exact in f16 and its chain equals the unshifted fp32 chain times 2^sigma when every
    // finite nonzero value has exponent in [e_max - 32, e_max], e_max <= 119 and e_min >=
    // -141 (products and partial sums then stay in fp32's normal range or on its subnormal
    // grid on both sides). Otherwise the multiplier is 0 and the exact fallback runs.
    const uint16_t* X = static_cast<const uint16_t*>(P.x);
    const int wp = tid >> 5, half = (tid >> 4) & 1, lane16 = tid & 15;
    const int total = real * G;
    for (int i0 = 2 * wp; i0 < total; i0 += 2 * NCW) {  // uniform trip count per warp
      const int i = i0 + half;
      const bool act = i < total;
      int r = 0, g = 0;
      uint32_t two = 0;
      if (act) {
        r = i / G;
        g = i - r * G;
        two = *reinterpret_cast<const uint32_t*>(X + (size_t)prow[r] * K + 32 * g + 2 * lane16);
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
        // 2^sigma, sigma in [-104, 148], as two exact factors
        const int s1 = min(max(sigma, -126), 127), s2 = sigma - s1;
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
        if (safe) {
          const int ns = -sigma;  // 2^-sigma, possibly subnormal (exact)
          m = ns >= -126 ? __uint_as_float((uint32_t)(127 + ns) << 23) : __uint_as_float(0x00400000u >> (-127 - ns));
        }
        xm_s[r * GB * 8 + g] = m;
      }
    }
  }
}

template <int MODE, int KIND, int MAXR>
__global__ void __launch_bounds__(NTHREADS, (MAXR <= 2 ? 2 : 1)) rows_kernel(const RowsParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + Smem::BARS);
  uint64_t* empty = full + MAX_NSTAGE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Smem::CTRL);
  int* prow = reinterpret_cast<int*>(smem + Smem::PASS_ROW);
  int* ppair = reinterpret_cast<int*>(smem + Smem::PASS_PAIR);
  float* epi = reinterpret_cast<float*>(smem + Smem::EPI);
  uint8_t* ring = smem + Smem::RING;
  uint8_t* xs_s = ring + (size_t)P.nstage * STAGE_B;
  float* xm_s = reinterpret_cast<float*>(xs_s + (size_t)MAXR * P.GB * 512);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int NST = P.nstage;

  if (tid == 0) {
    for (int s = 0; s < NST; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NCW);
    }
    mbar_fence_init();
    *abort_flag = 0;
  }
  __syncthreads();

  const int n_act = *P.n_active;
  const int total = n_act * P.units;

  if (warp == NCW) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t it = 0;
      bool stop = false;
      for (int item = blockIdx.x; item < total && !stop; item += gridDim.x) {
        const int a = item / P.units, u = item - a * P.units;
        const int e = P.active[a];
        if (e < 0 || e >= P.E) continue;
        const int p0 = P.offs[e], n = P.offs[e + 1] - p0;
        if (n <= 0 || p0 < 0 || p0 + n > P.R * P.k) continue;
        const uint8_t* src = P.w + (size_t)e * P.expert_bytes + (size_t)u * P.unit_bytes;
        for (int left = n; left > 0 && !stop;) {
          const int t = tier_of<MODE>(left, MAXR, P.tier_mode);
          left -= min(t, left);
          for (int s = 0; s < P.S; ++s, ++it) {
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
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int j = lane & 7;                   // accumulator lane = group mod 8
  const int o = (warp << 2) | (lane >> 3);  // octet index 0..31
  uint32_t it = 0;
  bool dead = false;

  for (int item = blockIdx.x; item < total; item += gridDim.x) {
    const int a = item / P.units, u = item - a * P.units;
    const int e = P.active[a];
    if (e < 0 || e >= P.E) { if (tid == 0) report(P.status, TFX_ST_SHAPE); continue; }
    const int p0 = P.offs[e], n = P.offs[e + 1] - p0;
    if (n <= 0 || p0 < 0 || p0 + n > P.R * P.k) { if (tid == 0 && n != 0) report(P.status, TFX_ST_SHAPE); continue; }
    int pos = p0;
    for (int left = n; left > 0;) {
      const int t = tier_of<MODE>(left, MAXR, P.tier_mode);
      const int real = min(t, left);
      // pass rows: real rows, then padding rows that repeat the last real row
      named_sync(1, NCONS);
      if (tid < 8) {
        const int src = pos + min(tid, real - 1);
        int row = src;
        if (MODE == MODE_UPC) {
          row = P.pair_row[src];
          if (row < 0 || row >= P.R) { report(P.status, TFX_ST_SHAPE); row = 0; }
        }
        prow[tid] = row;
        ppair[tid] = src;
      }
      named_sync(1, NCONS);
      stage_rows<KIND>(P, xs_s, xm_s, prow, real, tid);
      named_sync(1, NCONS);

      auto run = [&](auto TT) {
        constexpr int T = decltype(TT)::value;
        float acc0[T], acc1[T];
#pragma unroll
        for (int r = 0; r < T; ++r) { acc0[r] = 0.0f; acc1[r] = 0.0f; }
        int xr[T];
#pragma unroll
        for (int r = 0; r < T; ++r) xr[r] = min(r, real - 1);

        for (int s = 0; s < P.S; ++s, ++it) {
          const int slot = it % NST;
          const uint32_t ph = (it / NST) & 1u;
          if (!dead) {
            // warp-uniform outcome, so later full-warp shuffles and reductions stay legal
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
#pragma unroll
            for (int q = 0; q < 2; ++q) {
              const int g = s * GPS + 8 * q + j;
              if (g < P.G) {
                const uint4 c0 = *reinterpret_cast<const uint4*>(tile + o * CODE_B + 128 * q + 16 * j);
                const uint4 c1 = *reinterpret_cast<const uint4*>(tile + (32 + o) * CODE_B + 128 * q + 16 * j);
                const float sw0 = e8m0_to_f32(sc[o * GPS + 8 * q + j]);
                const float sw1 = e8m0_to_f32(sc[(32 + o) * GPS + 8 * q + j]);
                uint32_t w0[16], w1[16];
                e2m1x8_to_f16x2(c0.x, w0[0], w0[1], w0[2], w0[3]);
                e2m1x8_to_f16x2(c0.y, w0[4], w0[5], w0[6], w0[7]);
                e2m1x8_to_f16x2(c0.z, w0[8], w0[9], w0[10], w0[11]);
                e2m1x8_to_f16x2(c0.w, w0[12], w0[13], w0[14], w0[15]);
                e2m1x8_to_f16x2(c1.x, w1[0], w1[1], w1[2], w1[3]);
                e2m1x8_to_f16x2(c1.y, w1[4], w1[5], w1[6], w1[7]);
                e2m1x8_to_f16x2(c1.z, w1[8], w1[9], w1[10], w1[11]);
                e2m1x8_to_f16x2(c1.w, w1[12], w1[13], w1[14], w1[15]);
                float pg[T], pu[T];
#pragma unroll
                for (int r = 0; r < T; ++r) { pg[r] = 0.0f; pu[r] = 0.0f; }
#pragma unroll
                for (int tc = 0; tc < 4; ++tc) {
#pragma unroll
                  for (int r = 0; r < T; ++r) {
                    const uint4 xv = *reinterpret_cast<const uint4*>(xs_s + xoff(xr[r], g, tc, P.GB));
                    pg[r] = fma2_f16(w0[4 * tc + 0], xv.x, pg[r]);
                    pu[r] = fma2_f16(w1[4 * tc + 0], xv.x, pu[r]);
                    pg[r] = fma2_f16(w0[4 * tc + 1], xv.y, pg[r]);
                    pu[r] = fma2_f16(w1[4 * tc + 1], xv.y, pu[r]);
                    pg[r] = fma2_f16(w0[4 * tc + 2], xv.z, pg[r]);
                    pu[r] = fma2_f16(w1[4 * tc + 2], xv.z, pu[r]);
                    pg[r] = fma2_f16(w0[4 * tc + 3], xv.w, pg[r]);
                    pu[r] = fma2_f16(w1[4 * tc + 3], xv.w, pu[r]);
                  }
                }
#pragma unroll
                for (int r = 0; r < T; ++r) {
                  const float m = xm_s[xr[r] * P.GB * 8 + g];
                  if (KIND == TFX_ACT_E4M3) {
                    acc0[r] = __fmaf_rn(pg[r], __fmul_rn(sw0, m), acc0[r]);
                    acc1[r] = __fmaf_rn(pu[r], __fmul_rn(sw1, m), acc1[r]);
                  } else {
                    float a0 = pg[r], a1 = pu[r];
                    if (m == 0.0f) {
                      const uint16_t* xrow = static_cast<const uint16_t*>(P.x) + (size_t)prow[xr[r]] * P.K;
                      a0 = chain_bf16_exact(c0, xrow, g);
                      a1 = chain_bf16_exact(c1, xrow, g);
                    } else {
                      a0 = __fmul_rn(a0, m);
                      a1 = __fmul_rn(a1, m);
                    }
                    acc0[r] = __fmaf_rn(a0, sw0, acc0[r]);
                    acc1[r] = __fmaf_rn(a1, sw1, acc1[r]);
                  }
                }
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
      };

      switch (t) {
        case 1: run(std::integral_constant<int, 1>{}); break;
        case 2: if constexpr (MAXR >= 2) run(std::integral_constant<int, 2>{}); break;
        case 4: if constexpr (MAXR >= 4) run(std::integral_constant<int, 4>{}); break;
        case 6: if constexpr (MODE == MODE_UPC && MAXR >= 8) run(std::integral_constant<int, 6>{}); break;
        case 8: if constexpr (MODE == MODE_UPC && MAXR >= 8) run(std::integral_constant<int, 8>{}); break;
        default: break;
      }
      named_sync(1, NCONS);

      // ---------------------------------------------------------------- epilogue
      if (warp < real && !dead) {
        const int r = warp;
        const int p = ppair[r];
        if (MODE == MODE_UPC) {
          const int I = P.I;
          const int nn = 32 * u + lane;
          const float g = epi[r * 64 + lane], uu = epi[r * 64 + 32 + lane];
          const float den = __fadd_rn(1.0f, expf(-g));
          const float h = __fmul_rn(__fdiv_rn(g, den), uu);
          if (P.gu_dbg) {
            P.gu_dbg[(size_t)p * 2 * I + nn] = g;
            P.gu_dbg[(size_t)p * 2 * I + I + nn] = uu;
          }
          if (P.h_dbg) P.h_dbg[(size_t)p * I + nn] = h;
          if (KIND == TFX_ACT_E4M3) {
            const bool bad = __any_sync(0xffffffffu, isnan(h) || isinf(h));
            const uint32_t amax_b = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(h)));
            uint32_t sc;
            if (bad) sc = 255u;
            else if (amax_b == 0u) sc = 127u;
            else {
              const int e2 = amax_b >= 0x00800000u ? (int)(amax_b >> 23) - 127 : (31 - __clz((int)amax_b)) - 149;
              sc = (uint32_t)min(max(e2 - 8 + 127, 0), 254);
            }
            const uint32_t code = bad ? 0x7Fu : f32_to_e4m3(__fmul_rn(h, e8m0_recip_f32(sc)));
            static_cast<uint8_t*>(P.h)[(size_t)p * I + nn] = (uint8_t)code;
            if (lane == 0) P.hs[(size_t)p * (I / 32) + u] = (uint8_t)sc;
          } else {
            const __nv_bfloat16 b = __float2bfloat16_rn(h);
            static_cast<__nv_bfloat16*>(P.h)[(size_t)p * I + nn] = b;
          }
        } else {
          const int row = P.pair_row[p], slot = P.pair_slot[p];
          if (row >= 0 && row < P.R && slot >= 0 && slot < P.k) {
            float* dst = P.out + ((size_t)row * P.k + slot) * P.H + 64 * u;
            dst[lane] = epi[r * 64 + lane];
            dst[32 + lane] = epi[r * 64 + 32 + lane];
          } else if (lane == 0) {
            report(P.status, TFX_ST_SHAPE);
          }
        }
      }
      pos += real;
      left -= real;
    }
  }
}

// ------------------------------------------------------------------------------ host side

static std::mutex g_mu;

struct DevInfo {
  int sms = 0;
  size_t smem_optin = 0;
};

static int dev_info(DevInfo* out) {
  int dev;
  if (cudaGetDevice(&dev) != cudaSuccess) return TFX_ECUDA;
  static DevInfo cache[64];
  static bool have[64];
  std::lock_guard<std::mutex> lk(g_mu);
  if (dev < 0 || dev >= 64) return TFX_ECUDA;
  if (!have[dev]) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TFX_ECUDA;
    cache[dev].sms = v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return TFX_ECUDA;
    cache[dev].smem_optin = (size_t)v;
    have[dev] = true;
  }
  *out = cache[dev];
  return TFX_OK;
}

template <int MODE, int KIND, int MAXR>
static int launch_rows(const RowsParams& P, int max_items, cudaStream_t st) {
  DevInfo di;
  int rc = dev_info(&di);
  if (rc) return rc;
  const size_t smem = smem_bytes(P, MAXR);
  if (smem > di.smem_optin) return TFX_EUNSUPPORTED;
  auto kern = rows_kernel<MODE, KIND, MAXR>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return TFX_ELAUNCH;
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, NTHREADS, smem) != cudaSuccess || nb < 1)
    return TFX_ELAUNCH;
  int grid = min(max_items, nb * di.sms);
  if (grid < 1) return TFX_OK;
  kern<<<grid, NTHREADS, smem, st>>>(P);
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}

template <int MODE, int KIND>
static int dispatch_maxr(const RowsParams& P, int maxr, int max_items, cudaStream_t st) {
  switch (maxr) {
    case 1: return launch_rows<MODE, KIND, 1>(P, max_items, st);
    case 2: return launch_rows<MODE, KIND, 2>(P, max_items, st);
    case 4: return launch_rows<MODE, KIND, 4>(P, max_items, st);
    case 8:
      if constexpr (MODE == MODE_UPC) return launch_rows<MODE, KIND, 8>(P, max_items, st);
      return TFX_EUNSUPPORTED;
    default: return TFX_EUNSUPPORTED;
  }
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool dims_ok(const tfx_dims& d) {
  return d.hidden > 0 && d.hidden % 64 == 0 && d.inter > 0 && d.inter % 32 == 0 && d.n_experts >= 1 &&
         d.n_experts <= 1024 && d.top_k >= 1 && d.top_k <= 32 && d.top_k <= d.n_experts &&
         (int64_t)d.hidden * d.inter < (1ll << 31);
}

static int route_ok(const tfx_route* rt) {
  return rt && rt->offs && rt->pair_row && rt->pair_slot && rt->active && rt->n_active;
}

static void geometry(RowsParams& P, int mode) {
  P.K = mode == MODE_UPC ? P.H : P.I;
  P.S = (P.K + KC - 1) / KC;
  P.G = P.K / 32;
  P.GB = (P.G + 7) / 8;
  P.units = mode == MODE_UPC ? P.I / 32 : P.H / 64;
  P.unit_bytes = (size_t)P.S * STAGE_B;
  P.expert_bytes = (size_t)P.units * P.unit_bytes;
}

size_t packed_gu_bytes(const tfx_dims& d) {
  return (size_t)d.n_experts * (d.inter / 32) * ((d.hidden + KC - 1) / KC) * STAGE_B;
}
size_t packed_d_bytes(const tfx_dims& d) {
  return (size_t)d.n_experts * (d.hidden / 64) * ((d.inter + KC - 1) / KC) * STAGE_B;
}

static int opts_maxr(const tfx_rows_opts* opts, int mode, int R) {
  int m = opts ? opts->max_pass : 0;
  if (m == 0) {
    if (mode == MODE_UPC) m = R >= 5 ? 8 : R >= 3 ? 4 : R >= 2 ? 2 : 1;
    else m = R >= 3 ? 4 : R >= 2 ? 2 : 1;
  }
  return m;
}

static int rows_common(int mode, tfx_dims d, int32_t rows, int32_t kind, const uint8_t* packed, const void* x,
                       const uint8_t* xs, const tfx_route* rt, int32_t* status, const tfx_rows_opts* opts,
                       RowsParams& P, int& maxr) {
  if (!dims_ok(d) || rows < 0 || !packed || !route_ok(rt) || !status) return TFX_EINVAL;
  if ((int64_t)rows * d.top_k > (1ll << 30)) return TFX_EINVAL;
  if (kind != TFX_ACT_E4M3 && kind != TFX_ACT_BF16) return TFX_EINVAL;
  if (rows > 0 && (!x || !aligned16(x) || !aligned16(packed))) return TFX_EINVAL;
  if (kind == TFX_ACT_E4M3 && rows > 0 && !xs) return TFX_EINVAL;
  maxr = opts_maxr(opts, mode, rows);
  if (!(maxr == 1 || maxr == 2 || maxr == 4 || (maxr == 8 && mode == MODE_UPC))) return TFX_EINVAL;
  if (opts && (opts->tier_mode < 0 || opts->tier_mode > 1 || opts->timeout_ns < 0)) return TFX_EINVAL;
  P = RowsParams{};
  P.H = d.hidden;
  P.I = d.inter;
  P.E = d.n_experts;
  P.k = d.top_k;
  P.R = rows;
  geometry(P, mode);
  P.nstage = 4;
  P.x = x;
  P.xs = xs;
  P.offs = rt->offs;
  P.pair_row = rt->pair_row;
  P.pair_slot = rt->pair_slot;
  P.active = rt->active;
  P.n_active = rt->n_active;
  P.status = status;
  P.max_pass = maxr;
  P.tier_mode = opts ? opts->tier_mode : 0;
  P.timeout_ns = (opts && opts->timeout_ns > 0) ? (uint64_t)opts->timeout_ns : kDefaultTimeoutNs;
  P.w = mode == MODE_UPC ? packed : packed + packed_gu_bytes(d);
  return TFX_OK;
}

}  // namespace tfx

using namespace tfx;

extern "C" int tfx_xp_upc_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                               const uint8_t* x_scale, const tfx_route* rt, void* h, uint8_t* h_scale,
                               float* gu_dbg, float* h_dbg, int32_t* status, const tfx_rows_opts* opts,
                               void* stream) {
  RowsParams P;
  int maxr;
  int rc = rows_common(MODE_UPC, d, rows, act_kind, packed, x, x_scale, rt, status, opts, P, maxr);
  if (rc) return rc;
  if (rows == 0) return TFX_OK;
  if (!h || (act_kind == TFX_ACT_E4M3 && !h_scale)) return TFX_EINVAL;
  P.h = h;
  P.hs = h_scale;
  P.gu_dbg = gu_dbg;
  P.h_dbg = h_dbg;
  const int max_items = min(rows * d.top_k, d.n_experts) * P.units;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch_maxr<MODE_UPC, TFX_ACT_E4M3>(P, maxr, max_items, st);
  return dispatch_maxr<MODE_UPC, TFX_ACT_BF16>(P, maxr, max_items, st);
}

extern "C" int tfx_xp_down_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* h,
                                const uint8_t* h_scale, const tfx_route* rt, float* out, int32_t* status,
                                const tfx_rows_opts* opts, void* stream) {
  RowsParams P;
  int maxr;
  int rc = rows_common(MODE_DOWN, d, rows, act_kind, packed, h, h_scale, rt, status, opts, P, maxr);
  if (rc) return rc;
  if (rows == 0) return TFX_OK;
  if (!out) return TFX_EINVAL;
  P.out = out;
  const int max_items = min(rows * d.top_k, d.n_experts) * P.units;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch_maxr<MODE_DOWN, TFX_ACT_E4M3>(P, maxr, max_items, st);
  return dispatch_maxr<MODE_DOWN, TFX_ACT_BF16>(P, maxr, max_items, st);
}
