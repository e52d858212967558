// tfx_rows.cu -- C entry points of the rows engine (tfx_rows.cuh): gate/up rows, down rows
// and the one-launch layer, with their argument checks. The kernel instances themselves are
// compiled in tfx_rows_<format>_<phase>.cu.
//
// Method: "dsv41 metal: decode experts decode an expert's weights once for all of its rows"
// (TensorFold PR #2983): "What this changes" and the commit message of the rows kernels.
#include "tfx_rows.cuh"

namespace tfx {

extern template int dispatch<TFX_ACT_E4M3, PH_UPC>(const RowsParams&, int, cudaStream_t);
extern template int dispatch<TFX_ACT_E4M3, PH_DOWN>(const RowsParams&, int, cudaStream_t);
extern template int dispatch<TFX_ACT_E4M3, PH_FUSED>(const RowsParams&, int, cudaStream_t);
extern template int dispatch<TFX_ACT_BF16, PH_UPC>(const RowsParams&, int, cudaStream_t);
extern template int dispatch<TFX_ACT_BF16, PH_DOWN>(const RowsParams&, int, cudaStream_t);
extern template int dispatch<TFX_ACT_BF16, PH_FUSED>(const RowsParams&, int, cudaStream_t);

std::mutex& rows_mutex() {
  static std::mutex mu;
  return mu;
}

int dev_sms(int* sms, size_t* optin) {
  int dev;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return TFX_ECUDA;
  static int c_sms[64];
  static size_t c_opt[64];
  std::lock_guard<std::mutex> lk(rows_mutex());
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
  p.units = down ? d.hidden / 64 : d.inter / 32;
  p.unit_bytes = (size_t)p.S * STAGE_B;
  p.expert_bytes = (size_t)p.units * p.unit_bytes;
  p.w = w;
  return p;
}

size_t packed_gu_bytes(const tfx_dims& d) {
  return (size_t)d.n_experts * (d.inter / 32) * ((d.hidden + KC - 1) / KC) * STAGE_B;
}
size_t packed_d_bytes(const tfx_dims& d) {
  return (size_t)d.n_experts * (d.hidden / 64) * ((d.inter + KC - 1) / KC) * STAGE_B;
}

// Longest pass in rows: opts->max_pass (1..8 for gate/up, 1..4 for down), or by default every
// row of an expert in one pass up to 8 (gate/up) or 4 (down) rows. 0 = not a valid cap.
static int pass_cap(const tfx_rows_opts* opts, bool down, int R) {
  const int lim = down ? MAX_PASS_D : MAX_PASS_U;
  const int m = opts ? opts->max_pass : 0;
  if (m == 0) return max(1, min(R, lim));
  return (m >= 1 && m <= lim) ? m : 0;
}

static int common_args(tfx_dims d, int32_t rows, int32_t kind, const uint8_t* packed, const void* x,
                       const uint8_t* xs, int32_t* status, const tfx_rows_opts* opts, RowsParams& P) {
  if (!dims_ok(d) || rows < 0 || !packed || !status) return TFX_EINVAL;
  if ((int64_t)rows * d.top_k > (1ll << 30)) return TFX_EINVAL;
  if (kind != TFX_ACT_E4M3 && kind != TFX_ACT_BF16) return TFX_EINVAL;
  if (rows > 0 && (!x || !aligned16(x) || !aligned16(packed))) return TFX_EINVAL;
  if (kind == TFX_ACT_E4M3 && rows > 0 && !xs) return TFX_EINVAL;
  if (opts && (opts->tier_mode < 0 || opts->tier_mode > 2 || opts->timeout_ns < 0)) return TFX_EINVAL;
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
  P.cap_u = pass_cap(opts, false, rows);
  P.cap_d = 1;
  if (!P.cap_u) return TFX_EINVAL;
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
  const int max_items = min(rows * d.top_k, d.n_experts) * P.pu.units;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch<TFX_ACT_E4M3, PH_UPC>(P, max_items, st);
  return dispatch<TFX_ACT_BF16, PH_UPC>(P, max_items, st);
}

extern "C" int tfx_xp_down_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* h,
                                const uint8_t* h_scale, const tfx_route* rt, float* out, int32_t* status,
                                const tfx_rows_opts* opts, void* stream) {
  RowsParams P;
  int rc = common_args(d, rows, act_kind, packed, h, h_scale, status, opts, P);
  if (rc) return rc;
  if (!rt || !rt->offs || !rt->pair_row || !rt->pair_slot || !rt->active || !rt->n_active) return TFX_EINVAL;
  P.cap_u = 1;
  P.cap_d = pass_cap(opts, true, rows);
  if (!P.cap_d) return TFX_EINVAL;
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
  const int max_items = min(rows * d.top_k, d.n_experts) * P.pd.units;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch<TFX_ACT_E4M3, PH_DOWN>(P, max_items, st);
  return dispatch<TFX_ACT_BF16, PH_DOWN>(P, max_items, st);
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
                            uint8_t* h_scale, float* out, uint16_t* y, float* y_f32_dbg, float* gu_dbg,
                            float* h_dbg, int32_t* scratch, bool check_scratch, int32_t* status, const tfx_rows_opts* opts, RowsParams& P,
                            int& max_items) {
  int rc = common_args(d, rows, act_kind, packed, x, x_scale, status, opts, P);
  if (rc) return rc;
  if ((int64_t)rows * d.top_k > FUSED_MAX_PAIRS) return TFX_EUNSUPPORTED;
  P.cap_u = pass_cap(opts, false, rows);
  if (!P.cap_u) return TFX_EINVAL;
  P.cap_d = min(P.cap_u, MAX_PASS_D);  // the down pass stops at 4 rows
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
  P.gu_dbg = gu_dbg;
  P.h_dbg = h_dbg;
  P.scratch = scratch;
  P.route_ints = fused_route_ints(d.n_experts, rows, d.top_k, instance_warps(P.cap_u));
  max_items = min(rows * d.top_k, d.n_experts) * (P.pu.units + P.pd.units);
  return TFX_OK;
}

static int moe_rows_launch(const RowsParams& P, int32_t act_kind, int max_items, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (act_kind == TFX_ACT_E4M3) return dispatch<TFX_ACT_E4M3, PH_FUSED>(P, max_items, st);
  return dispatch<TFX_ACT_BF16, PH_FUSED>(P, max_items, st);
}

}  // namespace tfx

extern "C" int tfx_xp_moe_rows(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed, const void* x,
                               const uint8_t* x_scale, const int32_t* ids, const float* topk_w, int32_t* offs,
                               int32_t* pair_row, int32_t* pair_slot, int32_t* active, int32_t* n_active, void* h,
                               uint8_t* h_scale, float* out, uint16_t* y, float* y_f32_dbg, float* gu_dbg,
                               float* h_dbg, int32_t* scratch, int32_t* status, const tfx_rows_opts* opts,
                               void* stream) {
  RowsParams P;
  int max_items = 0;
  const int rc = moe_rows_prepare(d, rows, act_kind, packed, x, x_scale, ids, topk_w, offs, pair_row, pair_slot,
                                  active, n_active, h, h_scale, out, y, y_f32_dbg, gu_dbg, h_dbg, scratch, true,
                                  status, opts, P,
                                  max_items);
  if (rc || rows == 0) return rc;
  return moe_rows_launch(P, act_kind, max_items, stream);
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
  std::lock_guard<std::mutex> lk(rows_mutex());
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
  int max_items = 0;
  int rc = moe_rows_prepare(d, rows, act_kind, packed, x, x_scale, ids, topk_w, offs, pair_row, pair_slot, active,
                            n_active, h, h_scale, out, y, y_f32_dbg, nullptr, nullptr, nullptr, false, status,
                            opts, P,
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
  return moe_rows_launch(P, act_kind, max_items, stream);
}

// ------------------------------------------------------------------------------ host-buffer entry
// The one-launch layer from host buffers: the inputs' copy to the device, the layer and the
// copy of y back, queued on one stream by one call, with every device buffer carved from one
// workspace.
namespace tfx {

struct HostLayout {
  size_t in[4], in_bytes;  // x, x_scale, ids, topk_w within one input block (16-byte aligned)
  size_t scratch, inputs, offs, prow, pslot, act, nact, h, hs, out, y, total;  // within ws
};

static size_t up16(size_t v) { return (v + 15) & ~(size_t)15; }
static size_t up256(size_t v) { return (v + 255) & ~(size_t)255; }

static bool host_layout(tfx_dims d, int32_t rows, int32_t kind, HostLayout& L) {
  if (!dims_ok(d) || rows < 0 || (kind != TFX_ACT_E4M3 && kind != TFX_ACT_BF16)) return false;
  if ((int64_t)rows * d.top_k > FUSED_MAX_PAIRS) return false;
  const size_t R = (size_t)rows, H = (size_t)d.hidden, I = (size_t)d.inter, E = (size_t)d.n_experts;
  const size_t Pn = R * (size_t)d.top_k;
  const bool e4 = kind == TFX_ACT_E4M3;
  L.in[0] = 0;
  L.in[1] = up16(R * H * (e4 ? 1 : 2));
  L.in[2] = up16(L.in[1] + (e4 ? R * H / 32 : 0));
  L.in[3] = up16(L.in[2] + Pn * sizeof(int32_t));
  L.in_bytes = L.in[3] + Pn * sizeof(float);
  size_t o = 0;
  auto put = [&](size_t bytes) {
    const size_t at = o;
    o = up256(o + bytes);
    return at;
  };
  L.scratch = put(tfx_xp_moe_rows_scratch_bytes(d, rows));
  L.inputs = put(L.in_bytes);
  L.offs = put((E + 1) * sizeof(int32_t));
  L.prow = put(Pn * sizeof(int32_t));
  L.pslot = put(Pn * sizeof(int32_t));
  L.act = put(E * sizeof(int32_t));
  L.nact = put(sizeof(int32_t));
  L.h = put(Pn * I * (e4 ? 1 : 2));
  L.hs = put(e4 ? Pn * I / 32 : 0);
  L.out = put(Pn * H * sizeof(float));
  L.y = put(R * H * sizeof(uint16_t));
  L.total = o;
  return true;
}

}  // namespace tfx

extern "C" size_t tfx_xp_moe_rows_host_ws_bytes(tfx_dims d, int32_t rows, int32_t act_kind) {
  HostLayout L;
  return host_layout(d, rows, act_kind, L) ? L.total : 0;
}

extern "C" int tfx_xp_moe_rows_host_layout(tfx_dims d, int32_t rows, int32_t act_kind, size_t* offsets,
                                           size_t* in_bytes) {
  HostLayout L;
  if (!offsets || !in_bytes || !host_layout(d, rows, act_kind, L)) return TFX_EINVAL;
  for (int i = 0; i < 4; ++i) offsets[i] = L.in[i];
  *in_bytes = L.in_bytes;
  return TFX_OK;
}

extern "C" int tfx_xp_moe_rows_host(tfx_dims d, int32_t rows, int32_t act_kind, const uint8_t* packed,
                                    const void* x_host, const uint8_t* x_scale_host, const int32_t* ids_host,
                                    const float* topk_w_host, uint16_t* y_host, int32_t* status,
                                    int32_t* status_host, void* ws, size_t ws_bytes, const tfx_rows_opts* opts,
                                    void* stream) {
  HostLayout L;
  if (dims_ok(d) && (int64_t)rows * d.top_k > FUSED_MAX_PAIRS) return TFX_EUNSUPPORTED;  // as tfx_xp_moe_rows
  if (!host_layout(d, rows, act_kind, L)) return TFX_EINVAL;
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) || ws_bytes < L.total) return TFX_EINVAL;
  const bool e4 = act_kind == TFX_ACT_E4M3;
  if (rows > 0 && (!x_host || (e4 && !x_scale_host) || !ids_host || !topk_w_host || !y_host)) return TFX_EINVAL;
  uint8_t* w8 = static_cast<uint8_t*>(ws);
  uint8_t* din = w8 + L.inputs;
  // y goes straight to y_host when the device can address it (pinned host memory, mapped into
  // the device's address space): the combine's stores then replace the copy back
  auto device_view = [](const void* p) -> void* {  // p's device address, if it has one
    cudaPointerAttributes a;
    if (p && cudaPointerGetAttributes(&a, p) == cudaSuccess && a.type == cudaMemoryTypeHost && a.devicePointer)
      return a.devicePointer;
    (void)cudaGetLastError();
    return nullptr;
  };
  uint16_t* y_dev = reinterpret_cast<uint16_t*>(w8 + L.y);
  bool y_direct = false, in_place = false;
  const void* xd = din + L.in[0];
  const void* xsd = e4 ? din + L.in[1] : nullptr;
  const void* idd = din + L.in[2];
  const void* wd = din + L.in[3];
  if (rows > 0) {
    if (void* v = device_view(y_host)) {
      y_dev = static_cast<uint16_t*>(v);
      y_direct = true;
    }
    void* vx = device_view(x_host);
    void* vxs = e4 ? device_view(x_scale_host) : nullptr;
    void* vid = device_view(ids_host);
    void* vw = device_view(topk_w_host);
    if (vx && aligned16(vx) && (!e4 || vxs) && vid && vw) {
      xd = vx;
      xsd = vxs;
      idd = vid;
      wd = vw;
      in_place = true;
    }
  }
  RowsParams P;
  int max_items = 0;
  int rc = moe_rows_prepare(d, rows, act_kind, packed, xd, static_cast<const uint8_t*>(xsd),
                            static_cast<const int32_t*>(idd), static_cast<const float*>(wd),
                            reinterpret_cast<int32_t*>(w8 + L.offs),
                            reinterpret_cast<int32_t*>(w8 + L.prow), reinterpret_cast<int32_t*>(w8 + L.pslot),
                            reinterpret_cast<int32_t*>(w8 + L.act), reinterpret_cast<int32_t*>(w8 + L.nact),
                            w8 + L.h, e4 ? w8 + L.hs : nullptr, reinterpret_cast<float*>(w8 + L.out),
                            y_dev, nullptr, nullptr, nullptr,
                            reinterpret_cast<int32_t*>(w8 + L.scratch), true, status, opts, P, max_items);
  if (rc || rows == 0) return rc;  // every argument checked before anything is queued
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t R = (size_t)rows, H = (size_t)d.hidden, Pn = R * (size_t)d.top_k;
  const uint8_t* xb = static_cast<const uint8_t*>(x_host);
  auto h2d = [&](size_t off, const void* src, size_t n) {
    return cudaMemcpyAsync(din + off, src, n, cudaMemcpyHostToDevice, st) == cudaSuccess;
  };
  // inputs laid out back to back as tfx_xp_moe_rows_host_layout gives: one copy moves them all
  const bool one_block = (!e4 || x_scale_host == xb + L.in[1]) &&
                         reinterpret_cast<const uint8_t*>(ids_host) == xb + L.in[2] &&
                         reinterpret_cast<const uint8_t*>(topk_w_host) == xb + L.in[3];
  bool ok = true;
  if (in_place) {
    // the layer reads the inputs where they are
  } else if (one_block) {
    ok = h2d(0, xb, L.in_bytes);
  } else {
    ok = h2d(L.in[0], xb, R * H * (e4 ? 1 : 2)) && (!e4 || h2d(L.in[1], x_scale_host, R * H / 32)) &&
         h2d(L.in[2], ids_host, Pn * sizeof(int32_t)) && h2d(L.in[3], topk_w_host, Pn * sizeof(float));
  }
  if (!ok) {
    (void)cudaGetLastError();
    return TFX_ELAUNCH;
  }
  rc = moe_rows_launch(P, act_kind, max_items, stream);
  if (rc) return rc;
  if ((!y_direct &&
       cudaMemcpyAsync(y_host, w8 + L.y, R * H * sizeof(uint16_t), cudaMemcpyDeviceToHost, st) != cudaSuccess) ||
      (status_host && cudaMemcpyAsync(status_host, status, sizeof(int32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess)) {
    (void)cudaGetLastError();
    return TFX_ELAUNCH;
  }
  return TFX_OK;
}
