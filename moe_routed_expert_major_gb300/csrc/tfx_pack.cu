// tfx_pack.cu -- one-time conversion of canonical MXFP4 expert weights into the packed
// stage layout read by the rows kernels (one contiguous 17,408-byte block per stage: 64 rows
// x 256 code bytes, then the 64 rows' 16 scale bytes).
#include <cuda_runtime.h>
#include <stdint.h>

#include "tfx_common.cuh"

namespace tfx {

constexpr int PK_KC = 512, PK_STAGE = 64 * (256 + 16), PK_CODES = 64 * 256;
size_t packed_gu_bytes(const tfx_dims& d);
size_t packed_d_bytes(const tfx_dims& d);

// rows_of(rho, u) -> (matrix, row) of one packed stage row; codes [E][N][K/2], scales [E][N][K/32]
__global__ void pack_kernel(int H, int I, int E, const uint8_t* __restrict__ wg, const uint8_t* __restrict__ sg,
                            const uint8_t* __restrict__ wu, const uint8_t* __restrict__ su,
                            const uint8_t* __restrict__ wd, const uint8_t* __restrict__ sd, uint8_t* __restrict__ out,
                            size_t gu_words, size_t total_words) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  const int Sgu = (H + PK_KC - 1) / PK_KC, Sd = (I + PK_KC - 1) / PK_KC;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_words; i += stride) {
    const bool down = i >= gu_words;
    const size_t li = down ? i - gu_words : i;
    const size_t blk = li / (PK_STAGE / 4);
    const int off = (int)(li - blk * (PK_STAGE / 4)) * 4;
    const int S = down ? Sd : Sgu;
    const int units = down ? H / 64 : I / 32;
    const int s = (int)(blk % S);
    const int u = (int)((blk / S) % units);
    const int e = (int)(blk / ((size_t)S * units));
    const int K = down ? I : H;
    const int G = K / 32;
    const uint8_t *wc, *ws;
    int row;
    if (down) {
      row = 64 * u + (off < PK_CODES ? off / 256 : (off - PK_CODES) / 16);
      wc = wd;
      ws = sd;
      row += 0;
    } else {
      const int rho = off < PK_CODES ? off / 256 : (off - PK_CODES) / 16;
      row = 32 * u + (rho & 31);
      wc = rho < 32 ? wg : wu;
      ws = rho < 32 ? sg : su;
    }
    const int N = down ? H : I;
    uint32_t v = 0;
    if (off < PK_CODES) {
      const int kb = 256 * s + (off & 255);
      if (kb < K / 2) v = *reinterpret_cast<const uint32_t*>(wc + ((size_t)e * N + row) * (K / 2) + kb);
    } else {
      const int q0 = (off - PK_CODES) & 15;
      for (int b = 0; b < 4; ++b) {
        const int g = 16 * s + q0 + b;
        if (g < G) v |= (uint32_t)ws[((size_t)e * N + row) * G + g] << (8 * b);
      }
    }
    reinterpret_cast<uint32_t*>(out)[i] = v;
  }
}

}  // namespace tfx

using namespace tfx;

extern "C" size_t tfx_xp_packed_bytes(tfx_dims d) {
  if (d.hidden <= 0 || d.hidden % 64 || d.inter <= 0 || d.inter % 32 || d.n_experts < 1) return 0;
  return packed_gu_bytes(d) + packed_d_bytes(d);
}

extern "C" int tfx_xp_pack(tfx_dims d, const uint8_t* wg, const uint8_t* sg, const uint8_t* wu, const uint8_t* su,
                           const uint8_t* wd, const uint8_t* sd, uint8_t* packed, void* stream) {
  const size_t bytes = tfx_xp_packed_bytes(d);
  if (!bytes || !wg || !sg || !wu || !su || !wd || !sd || !packed) return TFX_EINVAL;
  if (((uintptr_t)packed | (uintptr_t)wg | (uintptr_t)wu | (uintptr_t)wd) & 15u) return TFX_EINVAL;
  const size_t words = bytes / 4, gu_words = packed_gu_bytes(d) / 4;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return TFX_ECUDA;
  pack_kernel<<<sms * 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(d.hidden, d.inter, d.n_experts, wg, sg, wu, su,
                                                                      wd, sd, packed, gu_words, words);
  return cudaGetLastError() == cudaSuccess ? TFX_OK : TFX_ELAUNCH;
}
