// tfx_chunk.cu -- the many-rows-per-expert (prompt chunk) path. Gate/up and down of every
// routed pair run as dense block-scaled contractions on the fifth-generation tensor cores:
// tcgen05.mma kind::mxf8f6f4 with E2M1 weights (operand A: 128 weight rows, K-major) and E4M3
// activations (operand B: the expert's routed pairs, K-major), one E8M0 scale per 32 k on each
// side, fp32 accumulators in tensor memory. The same maths as the rows kernels, reached
// through the tensor cores' own summation order instead of the fixed fma chain: results are
// within the float64 tolerance, and every pair's bits are independent of which other pairs
// share its launch (the pair's operands and the k order are the same whatever the chunk; the
// pair only changes column).
//
// Source: "dsv41 metal: decode experts decode an expert's weights once for all of its rows"
// (TensorFold PR #2983), which keeps prompt chunks on their own chunk-invariant kernels. A
// 4,096-row chunk routes about 128 rows to each expert, so gate/up and down there are dense
// contractions close to the HBM/tensor ridge.
//
// Tiles. A tile is one expert's block of up to CK_NMAX routed pairs (the MMA's N, rounded up
// to 16, so an expert's pairs are not padded to a power of two) against 256 weight rows, as
// two accumulators of 128 lanes:
//   gate/up: accumulator 0 = the 128 gate rows of four packed units (n = 32 u0 .. 32 u0 + 127),
//            accumulator 1 = the 128 up rows of the same n: lane l of both holds the same n,
//            so SwiGLU is thread-local and a warp's 32 lanes are one quantisation group;
//   down:    accumulator 0 = m0 .. m0 + 127, accumulator 1 = m0 + 128 .. m0 + 255.
// Each pipeline stage carries 128 k: two MMAs (one per accumulator) for each K = 32 step.
//
// CTA roles (448 threads, one CTA per SM, persistent over tiles):
//   warps 0-3, 10-13  epilogue: tensor memory -> registers -> SwiGLU + quantiser (gate/up) or
//              d (down). A warp reads the lanes of its quadrant (warp % 4); warps 0-3 take the
//              even 16-column chunks of the tile's pairs, warps 10-13 the odd ones.
//   warps 4-7  scale movers: once a stage has landed, write its weight-row and pair scales
//              into tensor memory (tcgen05.st, each warp its own lane quadrant)
//   warp 8     allocates tensor memory and issues the MMAs (one lane)
//   warp 9     TMA (one lane): the weight rows (E2M1 expanded into 16-byte slots by the tensor
//              map's 16U4_ALIGN16B type) and their scales, and the pairs' activation rows and
//              scales in pair order (h for down; for gate/up a copy of x gathered into pair
//              order first), one box each. Operands land 128B-swizzled.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tfx_common.cuh"

namespace tfx {

size_t packed_gu_bytes(const tfx_dims& d);

namespace {

constexpr int CK_M = 128;        // weight rows per accumulator (MMA M: tensor-memory lanes)
constexpr int CK_NMAX = 160;     // routed pairs per tile at most (MMA N, a multiple of 16)
constexpr int CK_KT = 128;       // k per pipeline stage
constexpr int CK_NS = 4;         // pipeline stages
constexpr int CK_THREADS = 448;  // 8 epilogue + 4 scale-mover warps + MMA warp + TMA warp
constexpr int CK_EPI_WARPS = 8;
// A stage: the two weight-row operands, then the pair operand (all 128B-swizzled, 1024-byte
// aligned). Scales come once per packed stage (512 k = four ring stages) into one of two
// buffers: the four units' weight-row scales as packed ([4][64 rows][16 groups]) and the
// tile's pair scales ([pair][16 groups]).
constexpr int CK_A0_OFF = 0;         // 16,384: 128 weight rows, E2M1 in 16-byte slots
constexpr int CK_A1_OFF = 16384;     // 16,384
constexpr int CK_B_OFF = 32768;      // 20,480: up to 160 pairs x 128 bytes, E4M3
constexpr int CK_STAGE = 53248;      // 52 x 1024
constexpr int CK_SW_BYTES = 4096;    // weight-row scales of one packed stage
constexpr int CK_SP_BYTES = CK_NMAX * 16;  // pair scales of one packed stage
constexpr int CK_SC_BUF = CK_SW_BYTES + CK_SP_BYTES;
constexpr int CK_TMEM_COLS = 512;
constexpr int CK_D1_COL = CK_NMAX;   // accumulator 1 (accumulator 0 at column 0)
constexpr int CK_SF_COL = 2 * CK_NMAX;  // scale columns of stage s: 320 + 16 s (A0: 4, A1: 4, B: 8)
static_assert(CK_SF_COL + 16 * CK_NS <= CK_TMEM_COLS, "tensor memory");
static_assert(CK_NMAX % 32 == 0 && CK_NMAX <= 256, "pair boxes of 32");
// packed weight layout (tfx_pack.cu): stages of 64 rows x 256 code bytes, then 64 x 16 scales
constexpr int PK_STAGE_BYTES = 64 * (256 + 16), PK_CODE_BYTES = 64 * 256;

struct ChunkParams {
  int K, G;          // contraction width (H for gate/up, I for down) and its 32-groups
  int nwb;           // 256-row weight blocks of the projection (I/128 for gate/up, H/256 for down)
  int units;         // packed units per expert
  int E, k, R, P, I, H;
  int down;
  const uint8_t* w;  // packed projection
  size_t unit_bytes, expert_bytes;
  const uint8_t* xs; // activation scales in pair order [P][K/32] (for the tensor map)
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
  int e, p0, np, u0;  // expert, first pair, pairs (<= CK_NMAX), first packed unit of the weight block
};

// ------------------------------------------------------------------ tcgen05 / TMA wrappers
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
// Instruction descriptor of kind::mxf8f6f4 with block scaling: A E2M1 (5), B E4M3 (0), both
// K-major, E8M0 scales, M = 128, N = n; sf_id picks the byte of the scale words.
__device__ __forceinline__ uint32_t mma_idesc(uint32_t n, uint32_t sf_id) {
  return (sf_id & 3u) << 4 | 5u << 7 | 0u << 10 | (n >> 3) << 17 | 1u << 23 | (uint32_t)(CK_M >> 4) << 24 |
         (sf_id & 3u) << 29;
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
// Issues the load of 16 columns of this warp's 32 lanes; the registers are valid after tmem_wait().
__device__ __forceinline__ void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

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

// Pair blocks of an expert with ne pairs: as many blocks of at most CK_NMAX as needed, sizes
// as equal as possible.
__device__ __forceinline__ int pair_blocks(int ne) { return (ne + CK_NMAX - 1) / CK_NMAX; }

// Tile t of this launch: tiles are numbered expert by expert (active order), then by pair
// block, then by weight block, so that concurrent CTAs share an expert's pairs and weights in L2.
__device__ __forceinline__ bool tile_of(const ChunkParams& P, const int* tpre, int n_act, int t, int& a,
                                        Tile& T) {
  while (a < n_act && tpre[a + 1] <= t) ++a;
  if (a >= n_act) return false;
  const int e = P.active[a];
  if (e < 0 || e >= P.E) return false;
  const int p0 = P.offs[e], ne = P.offs[e + 1] - p0;
  if (ne <= 0 || p0 < 0 || p0 + ne > P.P) return false;
  const int nb = pair_blocks(ne);
  const int local = t - tpre[a];
  const int pb = local / P.nwb, wb = local - pb * P.nwb;
  const int base = ne / nb, rem = ne - base * nb;
  T.e = e;
  T.p0 = p0 + pb * base + min(pb, rem);
  T.np = base + (pb < rem ? 1 : 0);
  T.u0 = 4 * wb;
  return true;
}

__global__ void __launch_bounds__(CK_THREADS, 1)
    chunk_kernel(const ChunkParams P, const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_ws,
                 const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_xs) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);  // 1024-byte aligned ring
  uint8_t* scbuf = smem + CK_NS * CK_STAGE;  // [2][weight-row scales | pair scales]
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
          if (ne > 0) t = P.nwb * pair_blocks(ne);
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
      const int ub = T.e * P.units + T.u0;  // packed unit index of the block (expert-major)
      const uint32_t tx = 2u * 8192u + (uint32_t)CK_NMAX * 128u;  // weight halves (packed bytes) + pair box
      const uint32_t tx_sc = (uint32_t)(CK_SW_BYTES + CK_SP_BYTES);
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
          mbar_arrive_expect_tx(&full_tma[slot], tx + (first ? tx_sc : 0u));
          if (!P.down) {  // 32 gate rows of each of the four units, then their 32 up rows
            tma_4d(st + CK_A0_OFF, &tm_w, kin, 0, ps, ub, &full_tma[slot]);
            tma_4d(st + CK_A1_OFF, &tm_w, kin, 32, ps, ub, &full_tma[slot]);
          } else {        // units u0, u0+1 (m0 .. m0+127), then u0+2, u0+3
            tma_4d(st + CK_A0_OFF, &tm_w, kin, 0, ps, ub, &full_tma[slot]);
            tma_4d(st + CK_A1_OFF, &tm_w, kin, 0, ps, ub + 2, &full_tma[slot]);
          }
          // the tile's pairs (rows past them are read, as zero past the end, and not used)
          tma_2d(st + CK_B_OFF, &tm_x, k0, T.p0, &full_tma[slot]);
          if (first) {
            tma_4d(sc, &tm_ws, 0, 0, ps, T.e * P.units + T.u0, &full_tma[slot]);
            tma_2d(sc + CK_SW_BYTES, &tm_xs, 16 * ps, T.p0, &full_tma[slot]);
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
    const int q = warp - 4;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
    uint32_t it = 0;
    int slot = 0;
    uint32_t ph = 0;
    bool dead = false;
    int a_hint = 0;
    // weight row of lane (q, lane) in each accumulator: gate/up: unit u0+q, rows lane (gate)
    // and 32+lane (up); down: unit u0+q/2 (+2), row 32 (q&1) + lane
    const int w0 = P.down ? 1024 * (q >> 1) + (32 * (q & 1) + lane) * 16 : 1024 * q + lane * 16;
    const int w1 = P.down ? 1024 * (2 + (q >> 1)) + (32 * (q & 1) + lane) * 16 : 1024 * q + (32 + lane) * 16;
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
        const uint32_t sa0 = *reinterpret_cast<const uint32_t*>(sc + w0 + g4);
        const uint32_t sa1 = *reinterpret_cast<const uint32_t*>(sc + w1 + g4);
        uint32_t sb[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {  // pair column 32 c + lane (columns past CK_NMAX: scale 1)
          const int n = 32 * c + lane;
          sb[c] = n < CK_NMAX ? *reinterpret_cast<const uint32_t*>(sc + CK_SW_BYTES + 16 * n + g4) : 0x7F7F7F7Fu;
        }
        const uint32_t col = CK_SF_COL + 16 * slot;
        asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tq + col + q), "r"(sa0) : "memory");
        asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(tq + col + 4 + q), "r"(sa1)
                     : "memory");
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(tq + col + 8),
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
      uint32_t ntile = 0;
      int slot = 0;
      uint32_t ph = 0;
      int a_hint = 0;
      bool dead = false;
      for (int t = blockIdx.x; t < total && !dead; t += gridDim.x) {
        Tile T;
        if (!tile_of(P, tpre, n_act, t, a_hint, T)) continue;
        const uint32_t n16 = (uint32_t)((T.np + 15) & ~15);
        if (ntile > 0 && !ck_wait(acc_empty, (ntile - 1) & 1u, P, abort)) break;
        tc_fence_after();
        for (int ks = 0; ks < nks; ++ks) {
          if (!ck_wait(&full_sc[slot], ph, P, abort) || !ck_wait(&full_tma[slot], ph, P, abort)) {
            dead = true;
            break;
          }
          tc_fence_after();
          const uint8_t* st = smem + slot * CK_STAGE;
          const uint32_t sf = tmem + CK_SF_COL + 16 * slot;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint64_t bd = smem_desc_sw128(st + CK_B_OFF + 32 * u);
            const uint32_t id = mma_idesc(n16, (uint32_t)u);
            mma_issue(tmem, smem_desc_sw128(st + CK_A0_OFF + 32 * u), bd, id, sf, sf + 8, (ks | u) != 0);
            mma_issue(tmem + CK_D1_COL, smem_desc_sw128(st + CK_A1_OFF + 32 * u), bd, id, sf + 4, sf + 8,
                      (ks | u) != 0);
          }
          mma_commit(&empty[slot]);
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
    const uint32_t tq = tmem + ((uint32_t)(32 * qd) << 16);
    uint32_t ntile = 0;
    int a_hint = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      Tile T;
      if (!tile_of(P, tpre, n_act, t, a_hint, T)) continue;
      if (!__all_sync(0xffffffffu, ck_wait(acc_full, ntile & 1u, P, abort))) break;
      tc_fence_after();
      // this warp's pair columns: chunks of 16, alternating between the two halves
      const int nch = (T.np + 15) >> 4;
      // down: (row, slot) of this warp's pairs, fetched at once (lane l < 16 of chunk slot ci
      // holds pair 16 (half + 2 ci) + l)
      int rsv[(CK_NMAX / 16 + 1) / 2];
      if (P.down) {
#pragma unroll
        for (int ci = 0; ci < (CK_NMAX / 16 + 1) / 2; ++ci) {
          const int j = 16 * (half + 2 * ci) + lane;
          rsv[ci] = -1;
          if (lane < 16 && j < T.np) {
            const int p = T.p0 + j;
            const int row = P.pair_row[p], sl = P.pair_slot[p];
            rsv[ci] = (row >= 0 && row < P.R && sl >= 0 && sl < P.k) ? row * P.k + sl : -2;
          }
        }
      }
      // one 16-column chunk of both accumulators, already in registers
      auto proc = [&](const uint32_t (&ra)[16], const uint32_t (&rb)[16], int ch) {
        const int c0 = 16 * ch;
        if (!P.down) {
          const int I = P.I;
          const int n = 32 * (T.u0 + qd) + lane;  // this lane's output n (gate in ra, up in rb)
          float hv[16];
          uint32_t amax[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            // silu(g) * u with the fast exponential and division: the chunk path is held to
            // the float64 bound, not to the rows path's bits
            const float g = __uint_as_float(ra[c]);
            hv[c] = __fdividef(g, 1.0f + __expf(-g)) * __uint_as_float(rb[c]);
            amax[c] = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv[c])));  // NaN/Inf: >= 0x7F800000
          }
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int j = c0 + c;
            const uint32_t amax_b = amax[c];
            const bool bad = amax_b >= 0x7F800000u;
            uint32_t sc;
            if (bad) sc = 255u;
            else if (amax_b == 0u) sc = 127u;
            else {
              const int e2 = amax_b >= 0x00800000u ? (int)(amax_b >> 23) - 127 : (31 - __clz((int)amax_b)) - 149;
              sc = (uint32_t)min(max(e2 - 8 + 127, 0), 254);
            }
            const uint32_t code = bad ? 0x7Fu : f32_to_e4m3(__fmul_rn(hv[c], e8m0_recip_f32(sc)));
            if (j < T.np) {
              const int p = T.p0 + j;
              P.h[(size_t)p * I + n] = (uint8_t)code;
              if (lane == 0) P.hs[(size_t)p * (I / 32) + T.u0 + qd] = (uint8_t)sc;
              if (P.gu_dbg) {
                P.gu_dbg[(size_t)p * 2 * I + n] = __uint_as_float(ra[c]);
                P.gu_dbg[(size_t)p * 2 * I + I + n] = __uint_as_float(rb[c]);
              }
              if (P.h_dbg) P.h_dbg[(size_t)p * I + n] = hv[c];
            }
          }
        } else {
          // lane holds m = m0 + 32 qd + lane (ra) and m + 128 (rb); d of pair j goes to out[row][slot]
          const int m = 64 * T.u0 + 32 * qd + lane;
          int rs = -1;
#pragma unroll
          for (int ci = 0; ci < (CK_NMAX / 16 + 1) / 2; ++ci)
            if (half + 2 * ci == ch) rs = rsv[ci];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int r = __shfl_sync(0xffffffffu, rs, c);
            if (r >= 0) {
              float* dst = P.out + (size_t)r * P.H + m;
              __stcs(dst, __uint_as_float(ra[c]));
              __stcs(dst + 128, __uint_as_float(rb[c]));
            } else if (r == -2 && lane == 0) {
              report(P.status, TFX_ST_SHAPE);
            }
          }
        }
      };
      // this warp's chunks are half, half + 2, ...: loads run one chunk ahead of the
      // processing, alternating between two register sets
      uint32_t xa[16], xb[16], ya[16], yb[16];
      if (half < nch) {
        tmem_ld16_issue(tq + 16 * half, xa);
        tmem_ld16_issue(tq + CK_D1_COL + 16 * half, xb);
      }
      tmem_wait();
      for (int ch = half; ch < nch; ch += 4) {
        if (ch + 2 < nch) {  // warp-uniform
          tmem_ld16_issue(tq + 16 * (ch + 2), ya);
          tmem_ld16_issue(tq + CK_D1_COL + 16 * (ch + 2), yb);
        }
        proc(xa, xb, ch);
        tmem_wait();
        if (ch + 2 < nch) {
          if (ch + 4 < nch) {
            tmem_ld16_issue(tq + 16 * (ch + 4), xa);
            tmem_ld16_issue(tq + CK_D1_COL + 16 * (ch + 4), xb);
          }
          proc(ya, yb, ch + 2);
          tmem_wait();
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
// loads a tile's pairs as 32-row boxes.
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
// (512 k of a stage row, 64 rows, stages, experts x units), loaded as 128 k boxes of 32 rows x
// 4 units (gate/up: the gate or the up halves) or 64 rows x 2 units (down), expanded into
// 16-byte slots; the same rows' scales (16 groups x 64 rows x 4 units per box); the
// activation rows in pair order [pairs][K] (bytes) as 128 k x CK_NMAX pair boxes (these and
// the weights 128-byte swizzled); their scales [pairs][K/32] as 16 x CK_NMAX boxes.
int encode_maps(const ChunkParams& P, const void* x, int nrows, CUtensorMap* tw, CUtensorMap* tws, CUtensorMap* tx,
                CUtensorMap* txs) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
  if (!enc) return TFX_ECUDA;
  const int S = (P.K + 511) / 512;
  const cuuint64_t gdw[4] = {512, 64, (cuuint64_t)S, (cuuint64_t)P.E * (cuuint64_t)P.units};
  const cuuint64_t gsw[3] = {256, (cuuint64_t)PK_STAGE_BYTES, (cuuint64_t)P.unit_bytes};
  const cuuint32_t bw_gu[4] = {128, 32, 1, 4}, bw_d[4] = {128, 64, 1, 2}, es[4] = {1, 1, 1, 1};
  if (enc(tw, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 4, const_cast<uint8_t*>(P.w), gdw, gsw, P.down ? bw_d : bw_gu, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TFX_EINVAL;
  // the weight rows' scales: 16 groups of a stage row, 64 rows, stages, experts x units
  const cuuint64_t gdws[4] = {16, 64, (cuuint64_t)S, (cuuint64_t)P.E * (cuuint64_t)P.units};
  const cuuint64_t gsws[3] = {16, (cuuint64_t)PK_STAGE_BYTES, (cuuint64_t)P.unit_bytes};
  const cuuint32_t bws[4] = {16, 64, 1, 4};
  if (enc(tws, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<uint8_t*>(P.w) + PK_CODE_BYTES, gdws, gsws, bws, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TFX_EINVAL;
  const cuuint64_t gdx[2] = {(cuuint64_t)P.K, (cuuint64_t)nrows}, gsx[1] = {(cuuint64_t)P.K};
  const cuuint32_t bx[2] = {128, CK_NMAX};
  if (enc(tx, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(x), gdx, gsx, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
      CUDA_SUCCESS)
    return TFX_EINVAL;
  const cuuint64_t gds[2] = {(cuuint64_t)P.G, (cuuint64_t)nrows}, gss[1] = {(cuuint64_t)P.G};
  const cuuint32_t bs[2] = {16, CK_NMAX};
  if (enc(txs, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(P.xs), gds, gss, bs, es,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_64B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return TFX_EINVAL;
  return TFX_OK;
}

int chunk_launch(const ChunkParams& P, const void* x, int nrows, cudaStream_t st) {
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
  alignas(64) CUtensorMap tw, tws, tx, txs;
  const int rc = encode_maps(P, x, nrows, &tw, &tws, &tx, &txs);
  if (rc) return rc;
  chunk_kernel<<<sms, CK_THREADS, smem, st>>>(P, tw, tws, tx, txs);
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
  P.units = down ? d.hidden / 64 : d.inter / 32;
  P.unit_bytes = (size_t)S * PK_STAGE_BYTES;
  P.expert_bytes = (size_t)P.units * P.unit_bytes;
  P.w = down ? packed + packed_gu_bytes(d) : packed;
  P.nwb = P.units / 4;
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
  P.xs = xsp;
  P.h = static_cast<uint8_t*>(h);
  P.hs = h_scale;
  P.gu_dbg = gu_dbg;
  P.h_dbg = h_dbg;
  return chunk_launch(P, xp, P.P, st);
}

extern "C" int tfx_xp_down_chunk(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* h,
                                 const uint8_t* h_scale, const tfx_route* rt, float* out, int32_t* status,
                                 const tfx_rows_opts* opts, void* stream) {
  ChunkParams P;
  const int rc = chunk_common(d, rows, act_kind, packed, rt, status, opts, P);
  if (rc) return rc;
  if (rows == 0) return TFX_OK;
  if (!h || !h_scale || !out || !al(h, 16) || !al(h_scale, 16) || !al(out, 16)) return TFX_EINVAL;
  set_proj(d, true, packed, P);
  P.xs = h_scale;
  P.out = out;
  return chunk_launch(P, h, P.P, static_cast<cudaStream_t>(stream));
}
