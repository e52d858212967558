// tfx_chunk.cu -- the many-rows-per-expert (prompt chunk) path. Gate/up and down of every
// routed pair run as a dense block-scaled contraction on the fifth-generation tensor cores:
// tcgen05.mma kind::mxf8f6f4 with E4M3 activations (operand A, one routed pair per row) and
// E2M1 weights (operand B, one weight row per column), one E8M0 scale per 32 k on each side,
// fp32 accumulators in tensor memory. The same maths as the rows kernels, reached through
// the tensor cores' own summation order instead of the fixed fma chain: results are within
// the float64 tolerance, and every pair's bits are independent of which other pairs share
// its launch (the instruction shape, the k order and the pair's operands are the same
// whatever the chunk; only its lane changes).
//
// Source: "dsv41 metal: decode experts decode an expert's weights once for all of its rows"
// (TensorFold PR #2983), which keeps prompt chunks on their own chunk-invariant kernels. A
// 4,096-row chunk routes about 128 rows to each expert, so gate/up and down there are dense
// contractions close to the HBM/tensor ridge.
//
// CTA roles (448 threads, one CTA per SM, persistent over tiles):
//   warps 0-3, 10-13  epilogue: tensor memory -> registers -> SwiGLU + quantiser (gate/up) or
//              d rows (down). A warp reads the lanes of its quadrant (warp % 4: pairs
//              32 (warp % 4) .. + 31 of the tile); warps 0-3 take accumulator columns 0-127,
//              warps 10-13 columns 128-255.
//   warps 4-7  scale movers: each thread owns one pair row of the tile; once a stage has
//              landed it writes both scale sets of the stage into tensor memory
//   warp 8     allocates tensor memory and issues the MMAs (one lane)
//   warp 9     TMA (one lane): the weight tile (E2M1 expanded into 16-byte slots by the
//              tensor map's 16U4_ALIGN16B type), the weight scales (bulk copies), the tile's
//              activation rows and their scales. Activations are read in pair order (h for
//              down; for gate/up a copy of x gathered into pair order first), so a tile's 128
//              rows are one box. The operands land 128B-swizzled.
// A tile is 128 routed pairs of one expert x 256 weight rows (four packed units); each
// pipeline stage carries 128 k (four MMAs of K = 32).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tfx_common.cuh"

namespace tfx {

size_t packed_gu_bytes(const tfx_dims& d);

namespace {

constexpr int CK_M = 128;        // routed pairs per tile (MMA M: tensor-memory lanes)
constexpr int CK_N = 256;        // weight rows per tile (MMA N: accumulator columns)
constexpr int CK_KT = 128;       // k per pipeline stage
constexpr int CK_NS = 4;         // pipeline stages
constexpr int CK_THREADS = 448;  // 8 epilogue + 4 scale-mover warps + MMA warp + TMA warp
constexpr int CK_EPI_WARPS = 8;
// Shared memory: a ring of CK_NS stages (weights, then activations; both 128B-swizzled,
// 1024-byte aligned), then two buffers of scales. Scales come once per packed stage (512 k,
// four ring stages): every buffer holds all 16 groups of the packed stage, for the weight
// rows ([4 units][64 rows][16]) and for the tile's pairs ([128][16]).
constexpr int CK_B_OFF = 0;          // 32,768: E2M1 weights, 8 code bytes per 16-byte slot
constexpr int CK_A_OFF = 32768;      // 16,384: E4M3 activations
constexpr int CK_STAGE = 49152;      // 48 x 1024
constexpr int CK_SB_BYTES = 4096;    // weight scales of one packed stage
constexpr int CK_SA_BYTES = 2048;    // pair scales of one packed stage
constexpr int CK_SC_BUF = CK_SB_BYTES + CK_SA_BYTES;
constexpr uint32_t CK_TX = 16384 + 16384;                // bytes of every stage's copies
constexpr uint32_t CK_TX_SC = CK_SB_BYTES + 128 * 16;    // plus, at a packed stage's first stage, its scales
constexpr int CK_TMEM_COLS = 512;
constexpr int CK_SF_COL = 256;   // scale columns of stage s: 256 + 12 s (A: 4, B: 8)
// packed weight layout (tfx_pack.cu): stages of 64 rows x 256 code bytes, then 64 x 16 scales
constexpr int PK_STAGE_BYTES = 64 * (256 + 16), PK_CODE_BYTES = 64 * 256;

struct ChunkParams {
  int K, G;          // contraction width (H for gate/up, I for down) and its 32-groups
  int ntn;           // weight-row tiles of 256 (2I/256 or H/256)
  int E, k, R, P, I, H;
  int down;
  const uint8_t* w;  // packed projection
  size_t unit_bytes, expert_bytes;
  const uint8_t* x;  // activation rows: x [R][H] (gate/up, by pair_row) or h [P][I] (down, by pair)
  const uint8_t* xs; // their E8M0 scales [rows][K/32]
  const int32_t *offs, *pair_row, *pair_slot, *active, *n_active;
  uint8_t* h;
  uint8_t* hs;
  float* gu_dbg;
  float* h_dbg;
  float* out;
  int32_t* status;
  uint64_t timeout_ns;
};

struct Tile {
  int e, p0, mreal, u0;  // expert, first pair, pairs (<= 128), first packed unit of the weight rows
};

// ------------------------------------------------------------------ tcgen05 / cp.async wrappers
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand in the 128-byte swizzle layout: rows
// of 128 bytes, eight-row atoms of 1024 bytes (stride between atoms), 1024-byte aligned tile.
__device__ __forceinline__ uint64_t smem_desc_sw128(const void* p) {
  const uint32_t a = smem_addr(p);
  return (uint64_t)((a >> 4) & 0x3FFFu) | (uint64_t)1 << 16 | (uint64_t)(1024 >> 4) << 32 | (uint64_t)1 << 46 |
         (uint64_t)2 << 61;
}
__device__ __forceinline__ void tma_4d(void* dst, const CUtensorMap* tm, int c0, int c1, int c2, int c3,
                                       uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(smem_addr(dst)),
      "l"(tm), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_addr(bar))
      : "memory");
}
__device__ __forceinline__ void tma_2d(void* dst, const CUtensorMap* tm, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_addr(dst)),
      "l"(tm), "r"(c0), "r"(c1), "r"(smem_addr(bar))
      : "memory");
}
// Instruction descriptor of kind::mxf8f6f4 with block scaling: A E4M3 (0), B E2M1 (5), both
// K-major, E8M0 scales, M = 128, N = 256; sf_id picks the byte of the scale words.
__device__ __forceinline__ uint32_t mma_idesc(uint32_t sf_id) {
  return (sf_id & 3u) << 4 | 0u << 7 | 5u << 10 | (uint32_t)(CK_N >> 3) << 17 | 1u << 23 |
         (uint32_t)(CK_M >> 4) << 24 | (sf_id & 3u) << 29;
}
__device__ __forceinline__ void mma_issue(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                          uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%5], [%6], p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(sfa), "r"(sfb)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait that also gives up once another role has aborted the CTA.
__device__ __forceinline__ bool ck_wait(uint64_t* bar, uint32_t parity, const ChunkParams& P, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
#pragma unroll 1
  while (!mbar_try_wait(bar, parity)) {
    if (*abort) return false;
    if (global_ns() - t0 > P.timeout_ns) {
      if (*abort == 0) report(P.status, TFX_ST_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
  return true;
}

// Tile t of this launch: tiles are numbered expert by expert (active order), then by
// weight-row tile, then by 128-pair block, so concurrent CTAs share experts in L2.
__device__ __forceinline__ bool tile_of(const ChunkParams& P, const int* tpre, int n_act, int t, int& a,
                                        Tile& T) {
  while (a < n_act && tpre[a + 1] <= t) ++a;
  if (a >= n_act) return false;
  const int e = P.active[a];
  if (e < 0 || e >= P.E) return false;
  const int p0 = P.offs[e], ne = P.offs[e + 1] - p0;
  if (ne <= 0 || p0 < 0 || p0 + ne > P.P) return false;
  const int mtn = (ne + CK_M - 1) / CK_M;
  const int local = t - tpre[a];
  const int nt = local / mtn, mt = local - nt * mtn;
  T.e = e;
  T.p0 = p0 + CK_M * mt;
  T.mreal = min(CK_M, ne - CK_M * mt);
  T.u0 = nt * (CK_N / 64);
  return true;
}

__global__ void __launch_bounds__(CK_THREADS, 1)
    chunk_kernel(const ChunkParams P, const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                 const __grid_constant__ CUtensorMap tm_xs) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);  // 1024-byte aligned ring
  uint8_t* scbuf = smem + CK_NS * CK_STAGE;  // [2][weight scales | pair scales]
  uint64_t* full_tma = reinterpret_cast<uint64_t*>(scbuf + 2 * CK_SC_BUF);
  uint64_t* full_sc = full_tma + CK_NS;
  uint64_t* empty = full_sc + CK_NS;
  uint64_t* acc_full = empty + CK_NS;
  uint64_t* acc_empty = acc_full + 1;
  uint64_t* drain = acc_empty + 1;
  volatile int* ctrl = reinterpret_cast<volatile int*>(drain + 1);  // [0] tensor-memory base, [1] abort
  int* tpre = const_cast<int*>(ctrl) + 4;                           // tile prefix over active experts
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(const_cast<int*>(ctrl))),
                 "n"(CK_TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    for (int s = 0; s < CK_NS; ++s) {
      mbar_init(&full_tma[s], 1);
      mbar_init(&full_sc[s], 4);
      mbar_init(&empty[s], 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, CK_EPI_WARPS);
    mbar_init(drain, 1);
    mbar_fence_init();
    ctrl[1] = 0;
  }
  int n_act = *P.n_active;
  n_act = n_act < 0 ? 0 : (n_act > P.E ? P.E : n_act);
  if (warp == 0) {  // tiles per active expert, exclusive prefix
    int carry = 0;
    for (int a0 = 0; a0 < n_act; a0 += 32) {
      const int a = a0 + lane;
      int t = 0;
      if (a < n_act) {
        const int e = P.active[a];
        if (e >= 0 && e < P.E) {
          const int ne = P.offs[e + 1] - P.offs[e];
          if (ne > 0) t = P.ntn * ((ne + CK_M - 1) / CK_M);
        }
      }
      int inc = t;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += v;
      }
      if (a < n_act) tpre[a] = carry + inc - t;
      carry += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) tpre[n_act] = carry;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = (uint32_t)ctrl[0];
  volatile int* abort = ctrl + 1;
  const int total = tpre[n_act];
  const int nks = P.K / CK_KT;

  if (warp == 9) {
    // ---------------------------------------------------------------- TMA
    uint32_t it = 0;
    int slot = 0;
    uint32_t ph = 0;
    int a_hint = 0;
    bool dead = false;
    for (int t = blockIdx.x; t < total && !dead; t += gridDim.x) {
      Tile T;
      if (!tile_of(P, tpre, n_act, t, a_hint, T)) continue;
      const int wunit = T.e * (P.ntn * (CK_N / 64)) + T.u0;  // packed unit index (expert-major)
      const uint8_t* wexp = P.w + (size_t)T.e * P.expert_bytes;
      for (int ks = 0; ks < nks; ++ks) {
        if (it >= (uint32_t)CK_NS &&
            !__all_sync(0xffffffffu, ck_wait(&empty[slot], ph ^ 1u, P, abort))) {
          dead = true;
          break;
        }
        uint8_t* st = smem + slot * CK_STAGE;
        const int k0 = ks * CK_KT, ps = k0 >> 9, kin = k0 & 511;
        const bool first = kin == 0;  // a packed stage starts: bring its scales too
        uint8_t* sc = scbuf + ((it >> 2) & 1u) * CK_SC_BUF;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full_tma[slot], CK_TX + (first ? CK_TX_SC : 0u));
          tma_4d(st + CK_B_OFF, &tm_w, kin, 0, ps, wunit, &full_tma[slot]);
          tma_2d(st + CK_A_OFF, &tm_x, k0, T.p0, &full_tma[slot]);  // rows past the pairs read as zero
          if (first) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              bulk_g2s(sc + 1024 * c,
                       wexp + (size_t)(T.u0 + c) * P.unit_bytes + (size_t)ps * PK_STAGE_BYTES + PK_CODE_BYTES, 1024,
                       &full_tma[slot]);
            tma_2d(sc + CK_SB_BYTES, &tm_xs, 16 * ps, T.p0, &full_tma[slot]);
          }
        }
        __syncwarp();
        ++it;
        if (++slot == CK_NS) {
          slot = 0;
          ph ^= 1u;
        }
      }
    }
    // copies still in flight (after an abort) land before the CTA may exit
    if (lane == 0)
      for (uint32_t j = it > (uint32_t)CK_NS ? it - CK_NS : 0u; j < it; ++j)
        if (!mbar_wait(&full_tma[j % CK_NS], (j / CK_NS) & 1u, P.timeout_ns)) report(P.status, TFX_ST_TIMEOUT);
    __syncwarp();
  } else if (warp >= 4 && warp < 8) {
    // ---------------------------------------------------------------- scale movers
    const int tp = tid - 128, q = warp - 4;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
    uint32_t it = 0;
    int slot = 0;
    uint32_t ph = 0;
    bool dead = false;
    int a_hint = 0;
    for (int t = blockIdx.x; t < total && !dead; t += gridDim.x) {
      Tile T;
      if (!tile_of(P, tpre, n_act, t, a_hint, T)) continue;
      for (int ks = 0; ks < nks; ++ks) {
        if (!__all_sync(0xffffffffu, ck_wait(&full_tma[slot], ph, P, abort))) {
          dead = true;
          break;
        }
        const uint8_t* sc = scbuf + ((it >> 2) & 1u) * CK_SC_BUF;
        const int g4 = ((ks * CK_KT) & 511) >> 5;  // first of the stage's 4 groups within the packed stage
        const uint32_t sa = *reinterpret_cast<const uint32_t*>(sc + CK_SB_BYTES + 16 * tp + g4);
        uint32_t sb[8];
#pragma unroll
        for (int c = 0; c < 8; ++c)  // weight row 32 c + lane: unit c/2, row 32 (c&1) + lane
          sb[c] = *reinterpret_cast<const uint32_t*>(sc + 1024 * (c >> 1) + (32 * (c & 1) + lane) * 16 + g4);
        const uint32_t col = CK_SF_COL + 12 * slot;
        asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tq + col + q), "r"(sa) : "memory");
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(tq + col + 4),
                     "r"(sb[0]), "r"(sb[1]), "r"(sb[2]), "r"(sb[3]), "r"(sb[4]), "r"(sb[5]), "r"(sb[6]), "r"(sb[7])
                     : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&full_sc[slot]);
        ++it;
        if (++slot == CK_NS) {
          slot = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------------- MMA issue
    if (lane == 0) {
      uint32_t it = 0, ntile = 0;
      int slot = 0;
      uint32_t ph = 0;
      int a_hint = 0;
      bool dead = false;
      for (int t = blockIdx.x; t < total && !dead; t += gridDim.x) {
        Tile T;
        if (!tile_of(P, tpre, n_act, t, a_hint, T)) continue;
        if (ntile > 0 && !ck_wait(acc_empty, (ntile - 1) & 1u, P, abort)) break;
        tc_fence_after();
        for (int ks = 0; ks < nks; ++ks) {
          if (!ck_wait(&full_sc[slot], ph, P, abort) || !ck_wait(&full_tma[slot], ph, P, abort)) {
            dead = true;
            break;
          }
          tc_fence_after();
          const uint8_t* st = smem + slot * CK_STAGE;
          const uint32_t sfa = tmem + CK_SF_COL + 12 * slot, sfb = sfa + 4;
#pragma unroll
          for (int u = 0; u < 4; ++u)
            mma_issue(tmem, smem_desc_sw128(st + CK_A_OFF + 32 * u), smem_desc_sw128(st + CK_B_OFF + 32 * u),
                      mma_idesc((uint32_t)u), sfa, sfb, (ks | u) != 0);
          mma_commit(&empty[slot]);
          ++it;
          if (++slot == CK_NS) {
            slot = 0;
            ph ^= 1u;
          }
        }
        if (dead) break;
        mma_commit(acc_full);
        ++ntile;
      }
      // every MMA this thread issued has completed before tensor memory is released
      mma_commit(drain);
      if (!mbar_wait(drain, 0, P.timeout_ns)) report(P.status, TFX_ST_TIMEOUT);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue (warps 0-3, 10-13)
    const int qd = warp & 3, half = warp >= 10 ? 1 : 0;
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16) + 128 * half;
    const int m = 32 * qd + lane;
    uint32_t ntile = 0;
    int a_hint = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      Tile T;
      if (!tile_of(P, tpre, n_act, t, a_hint, T)) continue;
      if (!__all_sync(0xffffffffu, ck_wait(acc_full, ntile & 1u, P, abort))) break;
      tc_fence_after();
      const bool valid = m < T.mreal;
      const int p = T.p0 + m;
      if (!P.down) {
        const int I = P.I;
#pragma unroll 1
        for (int jj = 0; jj < 2; ++jj) {  // packed unit u0 + j: 32 gate columns, then the 32 up columns
          const int j = 2 * half + jj;
          float g[32], u[32];
          tmem_ld16(tq + 64 * jj, *reinterpret_cast<float(*)[16]>(g));
          tmem_ld16(tq + 64 * jj + 16, *reinterpret_cast<float(*)[16]>(g + 16));
          tmem_ld16(tq + 64 * jj + 32, *reinterpret_cast<float(*)[16]>(u));
          tmem_ld16(tq + 64 * jj + 48, *reinterpret_cast<float(*)[16]>(u + 16));
          const int n0 = 32 * (T.u0 + j);
          float hv[32];
          bool bad = false;
          uint32_t amax_b = 0u;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            // silu(g) * u with the fast exponential and division: the chunk path is held to
            // the float64 bound, not to the rows path's bits
            hv[c] = __fdividef(g[c], 1.0f + __expf(-g[c])) * u[c];
            bad |= isnan(hv[c]) || isinf(hv[c]);
            amax_b = max(amax_b, __float_as_uint(fabsf(hv[c])));
          }
          if (valid) {
            if (P.gu_dbg) {
              float* gd = P.gu_dbg + (size_t)p * 2 * I + n0;
#pragma unroll
              for (int c = 0; c < 32; c += 4) {
                *reinterpret_cast<float4*>(gd + c) = make_float4(g[c], g[c + 1], g[c + 2], g[c + 3]);
                *reinterpret_cast<float4*>(gd + I + c) = make_float4(u[c], u[c + 1], u[c + 2], u[c + 3]);
              }
            }
            if (P.h_dbg) {
              float* hd = P.h_dbg + (size_t)p * I + n0;
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(hd + c) = make_float4(hv[c], hv[c + 1], hv[c + 2], hv[c + 3]);
            }
            uint32_t sc;
            if (bad) sc = 255u;
            else if (amax_b == 0u) sc = 127u;
            else {
              const int e2 =
                  amax_b >= 0x00800000u ? (int)(amax_b >> 23) - 127 : (31 - __clz((int)amax_b)) - 149;
              sc = (uint32_t)min(max(e2 - 8 + 127, 0), 254);
            }
            const float rs = e8m0_recip_f32(sc);
            uint32_t wv[8];
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
              uint32_t w = 0;
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const uint32_t code = bad ? 0x7Fu : f32_to_e4m3(__fmul_rn(hv[4 * c4 + b], rs));
                w |= code << (8 * b);
              }
              wv[c4] = w;
            }
            uint4* hp = reinterpret_cast<uint4*>(P.h + (size_t)p * I + n0);
            hp[0] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
            hp[1] = make_uint4(wv[4], wv[5], wv[6], wv[7]);
            P.hs[(size_t)p * (I / 32) + T.u0 + j] = (uint8_t)sc;
          }
        }
      } else {
        int row = -1, slot = -1;
        if (valid) {
          row = P.pair_row[p];
          slot = P.pair_slot[p];
          if (row < 0 || row >= P.R || slot < 0 || slot >= P.k) {
            report(P.status, TFX_ST_SHAPE);
            row = -1;
          }
        }
        float* dst = row >= 0 ? P.out + ((size_t)row * P.k + slot) * P.H + 64 * T.u0 + 128 * half : nullptr;
#pragma unroll 1
        for (int j = 0; j < CK_N / 32; ++j) {
          float v[16];
          tmem_ld16(tq + 16 * j, v);
          if (dst) {  // whole 32-byte sectors, not kept in L1 (the combine reads d much later)
#pragma unroll
            for (int c = 0; c < 16; c += 8)
              asm volatile("st.global.L1::no_allocate.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst + 16 * j + c),
                           "f"(v[c]), "f"(v[c + 1]), "f"(v[c + 2]), "f"(v[c + 3]), "f"(v[c + 4]), "f"(v[c + 5]),
                           "f"(v[c + 6]), "f"(v[c + 7])
                           : "memory");
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty);
      ++ntile;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 8)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(CK_TMEM_COLS) : "memory");
}

// Gate/up activations in pair order: xp[p] = x[pair_row[p]] and xsp[p] = xs[pair_row[p]] for
// the routed pairs p < offs[E] (one warp per pair, 16-byte copies), so that the chunk kernel
// loads a tile's 128 rows as one box.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint8_t* __restrict__ x, const uint8_t* __restrict__ xs,
                                                          const int32_t* __restrict__ pair_row,
                                                          const int32_t* __restrict__ offs, int E, int R, int H, int G,
                                                          int P, uint8_t* __restrict__ xp, uint8_t* __restrict__ xsp) {
  const int n = min(max(offs[E], 0), P);
  const int lane = threadIdx.x & 31;
  const int nw = (int)(gridDim.x * blockDim.x) >> 5;
  for (int p = (int)(blockIdx.x * blockDim.x + threadIdx.x) >> 5; p < n; p += nw) {
    int r = pair_row[p];
    if (r < 0 || r >= R) r = 0;
    const uint4* src = reinterpret_cast<const uint4*>(x + (size_t)r * H);
    uint4* dst = reinterpret_cast<uint4*>(xp + (size_t)p * H);
    for (int i = lane; i < H / 16; i += 32) dst[i] = __ldg(src + i);
    const uint4* ss = reinterpret_cast<const uint4*>(xs + (size_t)r * G);
    uint4* sd = reinterpret_cast<uint4*>(xsp + (size_t)p * G);
    for (int i = lane; i < G / 16; i += 32) sd[i] = __ldg(ss + i);
  }
}

size_t ws_part(size_t b) { return (b + 255) & ~(size_t)255; }

// alignment slack, ring, two scale buffers, 15 mbarriers (full_tma[4], full_sc[4], empty[4],
// acc_full, acc_empty, drain), control words, tile prefix
size_t chunk_smem_bytes(int E) {
  return 1024 + (size_t)CK_NS * CK_STAGE + 2 * CK_SC_BUF + 15 * 8 + 16 + 4 * (size_t)(E + 1);
}

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// Tensor maps of one launch: the packed projection's codes as a 4-D tensor of E2M1 values
// (512 k of a stage row, 64 rows, stages, experts x units), loaded as 128 k x 64 rows x 4
// units boxes into 16-byte slots; the activation rows in pair order [pairs][K] (bytes) as
// 128 k x 128 pair boxes (both 128-byte swizzled); their scales [pairs][K/32] as 16 x 128
// boxes.
int encode_maps(const ChunkParams& P, int nrows, CUtensorMap* tw, CUtensorMap* tx, CUtensorMap* txs) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return TFX_ECUDA;
  const int S = (P.K + 511) / 512;
  const cuuint64_t units = (cuuint64_t)P.E * (cuuint64_t)(P.ntn * (CK_N / 64));
  const cuuint64_t gdw[4] = {512, 64, (cuuint64_t)S, units};
  const cuuint64_t gsw[3] = {256, (cuuint64_t)PK_STAGE_BYTES, (cuuint64_t)P.unit_bytes};
  const cuuint32_t bw[4] = {128, 64, 1, 4}, es[4] = {1, 1, 1, 1};
  if (enc(tw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<uint8_t*>(P.w), gdw, gsw, bw, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TFX_EINVAL;
  const cuuint64_t gdx[2] = {(cuuint64_t)P.K, (cuuint64_t)nrows}, gsx[1] = {(cuuint64_t)P.K};
  const cuuint32_t bx[2] = {128, CK_M};
  if (enc(tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(P.x), gdx, gsx, bx, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TFX_EINVAL;
  const cuuint64_t gds[2] = {(cuuint64_t)P.G, (cuuint64_t)nrows}, gss[1] = {(cuuint64_t)P.G};
  const cuuint32_t bs[2] = {16, CK_M};
  if (enc(txs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(P.xs), gds, gss, bs, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TFX_EINVAL;
  return TFX_OK;
}

int chunk_launch(const ChunkParams& P, int nrows, cudaStream_t st) {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))
    return TFX_ECUDA;
  static int configured[64] = {0};
  const size_t smem = chunk_smem_bytes(P.E);
  if (dev < 0 || dev >= 64) return TFX_ECUDA;
  if (configured[dev] < (int)smem) {
    if (cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return TFX_ELAUNCH;
    configured[dev] = (int)smem;
  }
  alignas(64) CUtensorMap tw, tx, txs;
  const int rc = encode_maps(P, nrows, &tw, &tx, &txs);
  if (rc) return rc;
  chunk_kernel<<<sms, CK_THREADS, smem, st>>>(P, tw, tx, txs);
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}

int chunk_common(tfx_dims d, int32_t rows, int32_t kind, const uint8_t* packed, const tfx_route* rt,
                 int32_t* status, const tfx_rows_opts* opts, ChunkParams& P) {
  if (d.hidden <= 0 || d.hidden % 64 || d.inter <= 0 || d.inter % 32 || d.n_experts < 1 || d.n_experts > 1024 ||
      d.top_k < 1 || d.top_k > 32 || d.top_k > d.n_experts || (int64_t)d.hidden * d.inter >= (1ll << 31))
    return TFX_EINVAL;
  if (rows < 0 || (int64_t)rows * d.top_k > (1ll << 30) || !packed || !status || !al(packed, 32)) return TFX_EINVAL;
  if (kind != TFX_ACT_E4M3 && kind != TFX_ACT_BF16) return TFX_EINVAL;
  if (!rt || !rt->offs || !rt->pair_row || !rt->pair_slot || !rt->active || !rt->n_active) return TFX_EINVAL;
  if (opts && opts->timeout_ns < 0) return TFX_EINVAL;
  if (kind != TFX_ACT_E4M3 || d.hidden % 512 || d.inter % 512) return TFX_EUNSUPPORTED;
  P = ChunkParams{};
  P.E = d.n_experts;
  P.k = d.top_k;
  P.R = rows;
  P.P = rows * d.top_k;
  P.I = d.inter;
  P.H = d.hidden;
  P.offs = rt->offs;
  P.pair_row = rt->pair_row;
  P.pair_slot = rt->pair_slot;
  P.active = rt->active;
  P.n_active = rt->n_active;
  P.status = status;
  P.timeout_ns = (opts && opts->timeout_ns > 0) ? (uint64_t)opts->timeout_ns : kDefaultTimeoutNs;
  return TFX_OK;
}

void set_proj(const tfx_dims& d, bool down, const uint8_t* packed, ChunkParams& P) {
  P.down = down ? 1 : 0;
  P.K = down ? d.inter : d.hidden;
  P.G = P.K / 32;
  const int S = (P.K + 511) / 512;
  const int units = down ? d.hidden / 64 : d.inter / 32;
  P.unit_bytes = (size_t)S * PK_STAGE_BYTES;
  P.expert_bytes = (size_t)units * P.unit_bytes;
  P.w = down ? packed + packed_gu_bytes(d) : packed;
  P.ntn = (down ? d.hidden : 2 * d.inter) / CK_N;
}

}  // namespace
}  // namespace tfx

using namespace tfx;

extern "C" size_t tfx_xp_upc_chunk_ws_bytes(tfx_dims d, int32_t rows) {
  if (rows < 0 || d.hidden <= 0 || d.top_k <= 0) return 0;
  const size_t P = (size_t)rows * d.top_k;
  return ws_part(P * d.hidden) + ws_part(P * (d.hidden / 32));
}

extern "C" int tfx_xp_upc_chunk(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                                const uint8_t* x_scale, const tfx_route* rt, void* h, uint8_t* h_scale,
                                float* gu_dbg, float* h_dbg, void* ws, size_t ws_bytes, int32_t* status,
                                const tfx_rows_opts* opts, void* stream) {
  ChunkParams P;
  const int rc = chunk_common(d, rows, act_kind, packed, rt, status, opts, P);
  if (rc) return rc;
  if (rows == 0) return TFX_OK;
  if (!x || !x_scale || !h || !h_scale || !al(x, 16) || !al(x_scale, 16) || !al(h, 16) || !al(h_scale, 16) ||
      (gu_dbg && !al(gu_dbg, 16)) || (h_dbg && !al(h_dbg, 16)))
    return TFX_EINVAL;
  if (!ws || !al(ws, 256) || ws_bytes < tfx_xp_upc_chunk_ws_bytes(d, rows)) return TFX_EINVAL;
  set_proj(d, false, packed, P);
  uint8_t* xp = static_cast<uint8_t*>(ws);
  uint8_t* xsp = xp + ws_part((size_t)P.P * d.hidden);
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev))
    return TFX_ECUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  gather_rows_kernel<<<4 * sms, 256, 0, st>>>(static_cast<const uint8_t*>(x), x_scale, rt->pair_row, rt->offs, d.n_experts,
                                               rows, d.hidden, d.hidden / 32, P.P, xp, xsp);
  if (cudaGetLastError() != cudaSuccess) return TFX_ELAUNCH;
  P.x = xp;
  P.xs = xsp;
  P.h = static_cast<uint8_t*>(h);
  P.hs = h_scale;
  P.gu_dbg = gu_dbg;
  P.h_dbg = h_dbg;
  return chunk_launch(P, P.P, st);
}

extern "C" int tfx_xp_down_chunk(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* h,
                                 const uint8_t* h_scale, const tfx_route* rt, float* out, int32_t* status,
                                 const tfx_rows_opts* opts, void* stream) {
  ChunkParams P;
  const int rc = chunk_common(d, rows, act_kind, packed, rt, status, opts, P);
  if (rc) return rc;
  if (rows == 0) return TFX_OK;
  if (!h || !h_scale || !out || !al(h, 16) || !al(h_scale, 16) || !al(out, 32)) return TFX_EINVAL;
  set_proj(d, true, packed, P);
  P.x = static_cast<const uint8_t*>(h);
  P.xs = h_scale;
  P.out = out;
  return chunk_launch(P, rows * d.top_k, static_cast<cudaStream_t>(stream));
}
