// tfx_rows_e4m3_upc.cu -- the rows engine's kernel instances for e4m3 activations, upc rows (tfx_rows.cuh);
// one translation unit per activation format and phase so that they compile in parallel.
#include "tfx_rows.cuh"

namespace tfx {
template int dispatch<TFX_ACT_E4M3, PH_UPC>(const RowsParams&, int, cudaStream_t);
}  // namespace tfx
