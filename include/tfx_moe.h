/*
 * tfx_moe.h -- C ABI of the GB300 routed-expert MoE library (libtfx_moe.so, sm_103a).
 *
 * The library computes the routed-expert part of a DeepSeek-style MoE layer over
 * block-scaled FP4 weights for a launch of R token rows:
 *   route:    top-k expert ids [R][k] -> expert-major row lists (each expert's rows)
 *   upc_rows: per routed (row, slot) pair, g = x.Wg_e, u = x.Wu_e, h = silu(g) * u,
 *             h quantised to the launch's activation format
 *   down_rows: d[row][slot] = h . Wd_e
 *   combine:  y[row] = sum over slots (in slot order) of w[row][slot] * d[row][slot], bf16
 * Source of the method: "dsv41 metal: decode experts decode an expert's weights once for all
 * of its rows" (TensorFold PR #2983): "What this changes" and the commit message of the
 * rows kernels (tf_dsv41_xp_upc_rows / tf_dsv41_xp_down_rows, passes sized by the rows
 * left, padding rows computed and never written, the combine output checked per row).
 *
 * Numbers and formats
 *   Weights: MXFP4 (OCP MX v1.0): E2M1 codes, two per byte, the lower k in the low nibble,
 *   one E8M0 scale (2^(s-127), 0xFF = NaN) per 32 consecutive k of one output row.
 *   Activations: E4M3 (OCP OFP8, no infinities, 0x7F/0xFF NaN) with one E8M0 scale per 32
 *   consecutive k (TFX_ACT_E4M3), or bf16 (TFX_ACT_BF16).
 *   Accumulators (g, u, d) follow one fixed fp32 order for every row, whatever else is in
 *   the launch ("What this changes": each row's 32 products run as a sequential fma chain
 *   from zero in k order, then the scaled fma, then the eight-way tree):
 *     for each 32-group G:  p = fma chain of the 32 unscaled products, from +0, k ascending
 *                           acc[G mod 8] = fma(p, 2^(sw-127) * 2^(sx-127), acc[G mod 8])
 *     result = ((acc0+acc4) + (acc2+acc6)) + ((acc1+acc5) + (acc3+acc7))
 *   so every row's g, u and d are bit-identical alone or with any other rows and routing.
 *   Epilogue: h = (g / (1 + exp(-g))) * u in fp32. E4M3 launches quantise h per 32
 *   consecutive outputs with the OCP MX rule (shared exponent floor(log2 amax) - 8, nearest
 *   even, saturating at 448; amax 0 -> scale code 127; NaN/Inf in the block -> scale 0xFF
 *   and NaN codes). bf16 launches round h to bf16 (nearest even).
 *   Combine: y = fma chain over the k slots in slot order from +0, then bf16 (nearest even).
 *
 * Conventions
 *   Every pointer is a DEVICE pointer owned by the caller unless stated. The library never
 *   allocates, frees, synchronises or keeps a pointer after a call returns; every call is
 *   asynchronous on `stream` (a cudaStream_t; NULL is the legacy default stream).
 *   Return value: TFX_OK, or a negative TFX_E* found before anything was launched.
 *   Faults found on the device are OR-ed into the caller's `status` word (int32, device
 *   memory; TFX_ST_* bits), which the caller reads after its own synchronisation; the
 *   library never clears it. A pair whose expert id is out of range or repeats an earlier
 *   slot's id in the same row is left out of every list and its outputs are not written.
 *   Waits inside the kernels are bounded: a wait that runs out sets TFX_ST_TIMEOUT and the
 *   kernel returns early (outputs then incomplete).
 *   R = 0 is a no-op returning TFX_OK.
 */
#ifndef TFX_MOE_H
#define TFX_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- codes */
#define TFX_OK 0
#define TFX_EINVAL (-1)       /* null/misaligned pointer, negative or inconsistent sizes */
#define TFX_EUNSUPPORTED (-2) /* shape the kernels do not cover (see each entry point) */
#define TFX_ELAUNCH (-3)      /* the CUDA launch itself failed */
#define TFX_ECUDA (-4)        /* a CUDA query (device, attributes) failed */

#define TFX_ST_RANGE 1   /* an expert id was outside [0, E) */
#define TFX_ST_DUP 2     /* an expert id repeated an earlier slot of the same row */
#define TFX_ST_TIMEOUT 4 /* a bounded wait ran out; the kernel stopped early */
#define TFX_ST_SHAPE 8   /* route data inconsistent with the launch (corrupt lists) */

#define TFX_ACT_E4M3 0 /* E4M3 codes [rows][K] + E8M0 scales [rows][K/32] */
#define TFX_ACT_BF16 1 /* bf16 [rows][K] */

typedef struct {
  int32_t hidden;    /* H: model width; multiple of 64 */
  int32_t inter;     /* I: expert intermediate width; multiple of 32 */
  int32_t n_experts; /* E: routed experts; 1..1024 */
  int32_t top_k;     /* k: experts per row; 1..32 and <= E */
} tfx_dims;

/* Expert-major row lists written by tfx_xp_route (all device pointers).
 *   offs      [E+1]  pairs of expert e are offs[e] .. offs[e+1]-1
 *   pair_row  [R*k]  token row of each pair, ascending (row, slot) within an expert
 *   pair_slot [R*k]  slot (0..k-1) of each pair
 *   active    [min(R*k, E)]  experts with at least one pair, ascending id
 *   n_active  [1]    number of entries in active */
typedef struct {
  const int32_t* offs;
  const int32_t* pair_row;
  const int32_t* pair_slot;
  const int32_t* active;
  const int32_t* n_active;
} tfx_route;

/* Optional knobs of the rows kernels (pass NULL for the defaults). None changes a bit of
 * any output; they exist for tuning and for the tests that prove it.
 *   max_pass  largest pass (rows decoded against one read of the weights): 0 = min(R, 8)
 *             for gate/up and min(R, 4) for down; else 1..8 (gate/up) and 1..4 (down).
 *   tier_mode 0 = every pass takes min(rows left, max_pass) rows (sized by the rows left,
 *             no padding);
 *             1 = every pass at max_pass (padding rows repeat the last real row, are
 *             computed and never written);
 *             2 = the pages' tiers, capped at max_pass (gate/up 8 if >= 7 rows left, 6 if
 *             >= 5, 4 if >= 3, else 2 or 1; down 4 if >= 3, else 2 or 1), padded likewise.
 *   timeout_ns bound of every wait; 0 = 2 s. */
typedef struct {
  int32_t max_pass;
  int32_t tier_mode;
  int64_t timeout_ns;
} tfx_rows_opts;

/* ---------------------------------------------------------------- weights
 * The rows kernels read the experts' weights in a packed device layout that puts each
 * CTA's stage of codes and scales in one contiguous block, so that one bulk copy fetches
 * it. tfx_xp_pack converts the canonical layout once (at load time):
 *   wg, wu: codes [E][I][H/2], sg, su: scales [E][I][H/32]   (gate and up projections)
 *   wd: codes [E][H][I/2], sd: scales [E][H][I/32]           (down projection)
 * into `packed` (tfx_xp_packed_bytes(d) bytes, 16-byte aligned). Packed layout: for each
 * expert, for each block of 32 outputs n of I, for each stage of 512 k: 64 rows (32 gate
 * rows, then the 32 up rows of the same n) of 256 code bytes, then those 64 rows' 16
 * scale bytes; after all experts' gate/up, the same for the down projection with blocks of
 * 64 outputs m of H. k beyond H (or I) in the last stage is zero-filled.
 * Returns TFX_EINVAL for null pointers or bad dims. */
size_t tfx_xp_packed_bytes(tfx_dims d);
int tfx_xp_pack(tfx_dims d, const uint8_t* wg, const uint8_t* sg, const uint8_t* wu, const uint8_t* su,
                const uint8_t* wd, const uint8_t* sd, uint8_t* packed, void* stream);

/* ---------------------------------------------------------------- route
 * Builds the expert-major row lists ("every expert's rows", #2983 commit message) from
 * ids [R][k] (int32, row-major). Pairs of one expert are in ascending (row, slot) order;
 * active experts in ascending id. Invalid ids set TFX_ST_RANGE / TFX_ST_DUP in *status and
 * are left out. Output buffers: offs [E+1], pair_row and pair_slot [R*k],
 * active [min(R*k, E)], n_active [1]. E must be <= 1024. No scratch: launches of more than
 * 2,048 pairs run one CTA per 1,024 pairs (at most one per SM), each of which counts every
 * pair itself. Returns TFX_EINVAL for bad sizes or null pointers, TFX_ECUDA if the device
 * query fails, TFX_ELAUNCH if the launch fails; asynchronous on `stream`. */
int tfx_xp_route(tfx_dims d, int32_t rows, const int32_t* ids, int32_t* offs, int32_t* pair_row,
                 int32_t* pair_slot, int32_t* active, int32_t* n_active, int32_t* status, void* stream);

/* ---------------------------------------------------------------- gate/up rows
 * For every routed pair p (expert-major order of `rt`), with row r = pair_row[p]:
 *   g = x[r] . Wg_e, u = x[r] . Wu_e (fp32 chains above), h = silu(g) * u,
 * written as h[p][0..I) in the launch's activation format:
 *   TFX_ACT_E4M3: x = E4M3 codes [R][H] + x_scale E8M0 [R][H/32]; h = E4M3 codes [R*k][I]
 *                 + h_scale [R*k][I/32]
 *   TFX_ACT_BF16: x = bf16 [R][H] (x_scale NULL); h = bf16 [R*k][I] (h_scale NULL)
 * Each expert's weights are read once per pass for all of the pass's rows ("decode each
 * 32-group of an expert's MXFP4 weights once per pass and apply it to every row in it").
 * Optional debug outputs (NULL to skip): gu_dbg fp32 [R*k][2][I] (g then u), h_dbg fp32
 * [R*k][I] (h before quantisation). x, h and packed must be 16-byte aligned. */
int tfx_xp_upc_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                    const uint8_t* x_scale, const tfx_route* rt, void* h, uint8_t* h_scale, float* gu_dbg,
                    float* h_dbg, int32_t* status, const tfx_rows_opts* opts, void* stream);

/* ---------------------------------------------------------------- down rows
 * The down projection of the same page: the commit message of the rows kernels names
 * tf_dsv41_xp_down_rows beside the gate/up kernel (passes sized by the rows left, padding
 * rows computed and never written), and "What this changes" gives its products as fp4 by
 * E4M3 (or bf16) in the same fp32 chain.
 * For every routed pair p: out[pair_row[p]][pair_slot[p]][0..H) = h[p] . Wd_e (fp32 chain).
 * h and h_scale as written by tfx_xp_upc_rows; out is fp32 [R][k][H]. Entries of pairs
 * that were left out (invalid ids) are not written. The expert's weights are read once per
 * pass for all of the pass's pairs, as for gate/up. Returns TFX_EINVAL for bad sizes, kinds,
 * null or misaligned pointers (h, packed 16-byte aligned) or a bad max_pass (1, 2 or 4). */
int tfx_xp_down_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* h,
                     const uint8_t* h_scale, const tfx_route* rt, float* out, int32_t* status,
                     const tfx_rows_opts* opts, void* stream);

/* ---------------------------------------------------------------- chunk path (tensor cores)
 * The same two operations as tfx_xp_upc_rows and tfx_xp_down_rows, for launches with many
 * rows per expert (a prompt chunk: 4,096 rows route about 128 rows to each of 256 experts).
 * The page keeps prompt chunks on their own, chunk-invariant kernels. Here each expert's
 * gate/up and down are dense block-scaled contractions on the tensor cores: tcgen05.mma
 * kind::mxf8f6f4, with E4M3 activations x E2M1 weights, one E8M0 scale per 32 k on each
 * side, and fp32 accumulation in tensor memory. A tile is 128 pairs of one expert x 256
 * weight rows, streamed 128 k at a time.
 *
 * Numerics. The accumulation order is the tensor cores' own, not the fixed fp32 chain of
 * the _rows entries, so the two paths are separate invariance domains: the caller picks one,
 * and nothing switches between them implicitly.
 *   - Every pair's results are independent of the other pairs in the launch. They are
 *     bit-identical whether the row runs alone or in any chunk.
 *   - g, u, h (before quantisation) and d are within 1e-3 * sum|terms| + 1e-6 of float64.
 *   - SwiGLU runs in fp32 with the fast exponential and division (g / (1 + e^-g) * u); the
 *     E4M3 quantiser of h is that of tfx_xp_upc_rows.
 *
 * Arguments, layouts and outputs are those of the _rows entries, plus a workspace for gate/up.
 *   - ws: tfx_xp_upc_chunk_ws_bytes(d, R) bytes of device memory, 256-byte aligned, owned by
 *     the caller; the call first copies the activation rows (and scales) into pair order
 *     there, so that each tile's rows are one TMA box. Its contents are scratch.
 *   - TFX_EUNSUPPORTED: bf16 activations; H or I not a multiple of 512.
 *   - Alignment: packed and out 32-byte aligned; x, h, x_scale and h_scale 16-byte aligned;
 *     gu_dbg and h_dbg (when given) 16-byte aligned.
 *   - opts: only timeout_ns is read.
 *
 * Resources. One CTA per SM runs persistently over the tiles. Each CTA holds about 214 KB of
 * shared memory and all 512 columns of its SM's tensor memory for the duration of the launch.
 * Operands arrive by TMA (the packed weights through a tensor map that expands E2M1 into the
 * tensor cores' 16-byte slots, the activation rows and their scales by four-row gathers). The first call
 * looks up cuTensorMapEncodeTiled through the runtime (cudaGetDriverEntryPointByVersion);
 * TFX_ECUDA if the driver does not provide it.
 * Waits are bounded (TFX_ST_TIMEOUT). */
size_t tfx_xp_upc_chunk_ws_bytes(tfx_dims d, int32_t rows);
int tfx_xp_upc_chunk(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                     const uint8_t* x_scale, const tfx_route* rt, void* h, uint8_t* h_scale, float* gu_dbg,
                     float* h_dbg, void* ws, size_t ws_bytes, int32_t* status, const tfx_rows_opts* opts,
                     void* stream);
int tfx_xp_down_chunk(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* h,
                      const uint8_t* h_scale, const tfx_route* rt, float* out, int32_t* status,
                      const tfx_rows_opts* opts, void* stream);

/* ---------------------------------------------------------------- router
 * Routing ids and weights from router logits (no counterpart on the pages, which take the
 * routing as given; this entry produces ids [R][k] and topk_w [R][k] in the form the entries
 * above consume). For each row r of logits [rows][n_logits] (fp32, row-major, device):
 *   selection: the top_k largest logits, ties going to the lower expert id; slot order is
 *     descending logit (equal logits: lower id first). NaN ranks below every number and is
 *     taken only when a row has fewer than top_k numbers; -0 and +0 are equal.
 *   TFX_ROUTER_SOFTMAX: t_j = expf(l_j - l_0) (l_0 the largest selected logit),
 *     s = t_0 + t_1 + ... + t_{k-1} summed in slot order in fp32, w_j = t_j / s.
 *   TFX_ROUTER_SIGMOID: t_j = 1 / (1 + expf(-l_j)), then the same normalisation.
 * shared_expert >= 0 appends a shared (always-routed) expert to every row: the rows of ids and
 * topk_w then hold top_k + 1 slots, the last one shared_expert with weight 1. The layer is
 * then called with top_k + 1 slots; shared_expert must index the packed weights and lie
 * outside the routed ids (for example n_logits itself), or the route flags a duplicate.
 * Limits: n_logits <= 1024, 1 <= top_k <= min(32, n_logits). rows = 0 is a no-op.
 * Returns TFX_EINVAL for bad sizes, a bad mode or null pointers (rows > 0); TFX_ELAUNCH if
 * the launch fails. One warp per row; asynchronous on `stream`. */
#define TFX_ROUTER_SOFTMAX 0
#define TFX_ROUTER_SIGMOID 1
int tfx_xp_router(int32_t rows, int32_t n_logits, int32_t top_k, const float* logits, int32_t mode,
                  int32_t shared_expert, int32_t* ids, float* topk_w, void* stream);

/* Group-limited sigmoid routing (DeepSeek-V3 style; no counterpart on the pages either), in
 * fp32 throughout, every step one IEEE operation rounded to nearest, so that ids and weights
 * are fixed bit for bit by this definition. For each row of logits [rows][n_logits]:
 *   s_e = sigmoid32(l_e): t = exp(max(-|l|, -86)) by Cody-Waite reduction (n = rint(y / ln 2),
 *     r = (y - n*ln2_hi) - n*ln2_lo, ln2_hi with 16 significant bits) and the degree-7 Taylor
 *     polynomial of exp(r) in Horner form, times 2^n; s = 1/(1+t) for l >= 0, t/(1+t) below.
 *   c_e = s_e + bias[e] (bias [n_logits] fp32 on the device, or NULL: c_e = s_e).
 *   The experts form n_group contiguous groups of n_logits / n_group; a group's score is the
 *     fp32 sum of its two best c (best first). The topk_group best groups are kept (equal
 *     scores: lower group first), and the top_k best experts of the kept groups by c are the
 *     ids, best first (equal c: lower id first; NaN ranks below every number; -0 equals +0).
 *   w_j = (s_j / S) * scale, S = s_0 + ... + s_{top_k-1} summed in slot order from +0. The
 *     bias steers the choice only.
 * shared_expert >= 0 appends a shared expert with weight 1, as for tfx_xp_router.
 * Limits: n_logits <= 1024; 1 <= n_group <= 32 dividing n_logits into groups of at least 2;
 * 1 <= topk_group <= n_group; 1 <= top_k <= min(32, topk_group * n_logits / n_group); scale not
 * NaN. rows = 0 is a no-op. Returns TFX_EINVAL for bad sizes or null logits/ids/topk_w
 * (rows > 0), TFX_ELAUNCH if the launch fails. One warp per row; asynchronous on `stream`. */
int tfx_xp_router_grouped(int32_t rows, int32_t n_logits, int32_t top_k, const float* logits, const float* bias,
                          int32_t n_group, int32_t topk_group, float scale, int32_t shared_expert, int32_t* ids,
                          float* topk_w, void* stream);

/* ---------------------------------------------------------------- whole layer, one launch
 * Route, gate/up, down and combine of a small launch (R*k <= 256 routed pairs: decode) in a
 * single kernel launch, with the same results, bit for bit, as tfx_xp_route followed by
 * tfx_xp_upc_rows, tfx_xp_down_rows and tfx_xp_combine. Every CTA builds the row lists in
 * shared memory (the first also writes them to offs .. n_active, sized as for tfx_xp_route);
 * down items wait (bounded) for their expert's gate/up items; each (row, 64-output block) is
 * combined by the CTA whose down item writes the row's last valid slot. As with
 * tfx_xp_combine, a row with a left-out slot (invalid id, flagged in status) combines that
 * slot's unwritten (stale) entries of out.
 * ids int32 [R][k], topk_w fp32 [R][k]; h / h_scale / out as for the separate entries; y bf16
 * [R][H]; y_f32_dbg fp32 [R][H], gu_dbg fp32 [R*k][2][I] and h_dbg fp32 [R*k][I] (as for
 * tfx_xp_upc_rows) are debug copies, NULL to skip.
 * scratch: tfx_xp_moe_rows_scratch_bytes(d, R) bytes of device memory, 4-byte aligned, zero
 * before its first use; every call that completes returns it to zero (each counter's last
 * user clears it; a call that stopped early on TFX_ST_TIMEOUT may leave counters set, and the
 * caller then zeroes the buffer before the next call), so calls sharing one scratch buffer
 * must not overlap on the device. The CTAs of one launch wait on one another, so the launch
 * is cooperative (all CTAs resident at once; the runtime refuses it otherwise: TFX_ELAUNCH);
 * a wait that runs out sets TFX_ST_TIMEOUT.
 * Work is handed out one (pass, packed units) item at a time, expert-major (every gate/up pass
 * of the first active expert, then of the second, ..., then the down passes in the same order),
 * so that the down items claimed first are those whose gate/up items were handed out first, and
 * consecutive items on one CTA mostly share their activation rows.
 * Returns TFX_EUNSUPPORTED for R*k > 256. opts->max_pass applies to gate/up (1..8); the down
 * pass is the same capped at 4. */
size_t tfx_xp_moe_rows_scratch_bytes(tfx_dims d, int32_t rows);
int tfx_xp_moe_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                    const uint8_t* x_scale, const int32_t* ids, const float* topk_w, int32_t* offs,
                    int32_t* pair_row, int32_t* pair_slot, int32_t* active, int32_t* n_active, void* h,
                    uint8_t* h_scale, float* out, uint16_t* y, float* y_f32_dbg, float* gu_dbg, float* h_dbg,
                    int32_t* scratch, int32_t* status, const tfx_rows_opts* opts, void* stream);

/* The one-launch layer without caller scratch (no counterpart on the pages: it is an
 * interface for callers that cannot allocate). Some callers cannot call cudaMalloc: code
 * running inside a host runtime that owns every device allocation through its own pool, or
 * a plugin on a path where an allocation would synchronise the device or fail. This entry
 * point allocates nothing and calls no allocating routine: the completion counters live in a
 * 64 KiB buffer compiled into the library (a file-scope __device__ array, held by every GPU
 * that loads the library until the process exits), cleared on `stream` at the start of each
 * call. Arguments and results are those of tfx_xp_moe_rows without `scratch`; the caller
 * still passes every input and output buffer.
 * Limit: tfx_xp_moe_rows_scratch_bytes(d, R) <= 65536 bytes (16,384 counters), else
 * TFX_EUNSUPPORTED. That size check comes first; then every other argument is checked as by
 * tfx_xp_moe_rows, and only a call that passes them all clears the buffer and launches.
 * The first call on a device looks up the buffer's device address (cudaGetSymbolAddress).
 * With CUDA's default lazy module loading, that first use (or the first launch) also loads
 * the library's module on the device, which allocates device memory (the buffer among it)
 * and may synchronise: make one call at start-up, outside any stream capture and outside any
 * region where allocation is not allowed, before relying on the no-allocation property.
 * Every call on a device shares the one buffer: calls that overlap on the GPU (other streams,
 * other threads) race and give wrong results; serialise them. */
int tfx_xp_moe_rows_noalloc(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                            const uint8_t* x_scale, const int32_t* ids, const float* topk_w, int32_t* offs,
                            int32_t* pair_row, int32_t* pair_slot, int32_t* active, int32_t* n_active, void* h,
                            uint8_t* h_scale, float* out, uint16_t* y, float* y_f32_dbg, int32_t* status,
                            const tfx_rows_opts* opts, void* stream);

/* The one-launch layer from host buffers (no counterpart on the pages: an interface for
 * callers whose activations and routing sit in host memory, and the call that the end-to-end
 * measurement makes). One call queues on `stream`, in order:
 *   - the inputs' way to the device (x, x_scale, ids and topk_w, laid out as for
 *     tfx_xp_moe_rows; x_scale is ignored for bf16 activations). When all of them are pinned
 *     host memory that the device can address, and x is 16-byte aligned, the layer reads them
 *     in place and nothing is copied. Otherwise they are copied into ws (see below);
 *   - the layer, exactly as tfx_xp_moe_rows (same results, bit for bit);
 *   - y (bf16 [R][H]) into y_host, and, if status_host is not NULL, a copy of the status word
 *     to status_host. When y_host is pinned host memory that the device can address
 *     (cudaPointerGetAttributes reports host memory with a device pointer), the layer's combine
 *     stores y there itself; otherwise y is copied there after the layer.
 * It returns once they are queued. The host buffers must stay valid, the inputs unchanged and
 * y_host and status_host unread, until the stream has passed the layer and its copies. With
 * pinned (page-locked) host memory nothing waits on the host; with pageable memory the runtime
 * waits for each copy on the host.
 * When the inputs are copied, one copy moves all four if they lie back to back in one host
 * block: x_scale_host, ids_host and topk_w_host at the byte offsets from x_host that
 * tfx_xp_moe_rows_host_layout gives (offsets[0..3], 16-byte aligned; in_bytes is the block's
 * size). Otherwise each input is copied on its own.
 * ws: tfx_xp_moe_rows_host_ws_bytes(d, R, act_kind) bytes of device memory, 256-byte aligned,
 *   owned by the caller. It holds the scratch counters (zero before the first call, as for
 *   tfx_xp_moe_rows) and the device copies of the inputs, row lists, h, out and y. Calls
 *   sharing one ws must not overlap on the device.
 * status: an int32 on the device that the layer ORs its flags into, as for tfx_xp_moe_rows.
 * packed: the device copy of the packed weights (tfx_xp_pack).
 * Returns TFX_EUNSUPPORTED for R*k > 256; TFX_EINVAL for bad sizes or kind, a ws that is NULL,
 * misaligned or too small, a NULL host pointer (rows > 0) or any argument that tfx_xp_moe_rows
 * refuses; all checks come before anything is queued. Returns TFX_ELAUNCH if a copy or the
 * launch cannot be queued. rows = 0 queues nothing.
 * tfx_xp_moe_rows_host_ws_bytes returns 0 for bad sizes or kind, or for R*k > 256;
 * tfx_xp_moe_rows_host_layout returns TFX_EINVAL for those or NULL outputs. */
size_t tfx_xp_moe_rows_host_ws_bytes(tfx_dims d, int32_t rows, int32_t act_kind);
int tfx_xp_moe_rows_host_layout(tfx_dims d, int32_t rows, int32_t act_kind, size_t* offsets, size_t* in_bytes);
int tfx_xp_moe_rows_host(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x_host,
                         const uint8_t* x_scale_host, const int32_t* ids_host, const float* topk_w_host,
                         uint16_t* y_host, int32_t* status, int32_t* status_host, void* ws, size_t ws_bytes,
                         const tfx_rows_opts* opts, void* stream);

/* ---------------------------------------------------------------- combine
 * The routing-weighted sum of a row's expert outputs, whose bf16 result "Receipt > Kernel
 * contract" of the same page checks per row (the combine output, bit-equal alone or with
 * other rows).
 * y[r][m] = fma chain over j = 0..k-1 of topk_w[r][j] * out[r][j][m] from +0, rounded to
 * bf16 (nearest even). out fp32 [R][k][H], topk_w fp32 [R][k], y bf16 bits [R][H],
 * y_f32_dbg fp32 [R][H] or NULL. Returns TFX_EINVAL for bad dims, rows < 0 or null pointers
 * (rows > 0). */
int tfx_xp_combine(tfx_dims d, int32_t rows, const float* out, const float* topk_w, uint16_t* y,
                   float* y_f32_dbg, void* stream);

/* ---------------------------------------------------------------- misc */
const char* tfx_strerror(int code);
int tfx_version(void);

/* Self-test of the bounded wait: launches one block that waits on a barrier nothing will
 * complete, with the given limit in nanoseconds; the wait runs out, TFX_ST_TIMEOUT is OR-ed
 * into *status and the kernel returns. */
int tfx_selftest_wait_timeout(int32_t* status, int64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif
#endif
