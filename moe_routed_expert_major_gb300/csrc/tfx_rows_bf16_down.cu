// tfx_rows_bf16_down.cu -- the rows engine's kernel instances for bf16 activations, down rows (tfx_rows.cuh);
// one translation unit per activation format and phase so that they compile in parallel.
#include "tfx_rows.cuh"

namespace tfx {
template int dispatch<TFX_ACT_BF16, PH_DOWN>(const RowsParams&, int, cudaStream_t);
}  // namespace tfx
