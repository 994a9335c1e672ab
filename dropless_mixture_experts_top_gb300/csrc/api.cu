// api.cu -- the C ABI (include/moe.h): argument validation, workspace
// carving, and the launch sequence of each call.  Everything after validation
// is enqueued on the caller's stream; nothing is allocated or synchronised
// here except in moe_get_device_status.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/moe.h"
#include "internal.h"

namespace moe {

void *tensor_map_encoder() {
  static void *fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = p;
  });
  return fn;
}

namespace {

constexpr size_t kHeader = 256;  // status word at offset 0

inline size_t align256(size_t n) { return (n + 255) & ~static_cast<size_t>(255); }

struct Layout {
  // route scratch (r_zero: bytes from the start that each call zeroes: header and tickets)
  size_t r_tickets, r_lrank, r_hist, r_gpref, r_zero, r_total;
  // saved
  size_t s_xperm, s_G, s_U, s_A, s_Y, s_Aw, s_total;
  // forward scratch (f_pad: fp8_bwd's padded expert offsets)
  size_t f_pad, f_total;
  // backward scratch
  size_t b_dyp, b_dG, b_dU, b_dX, b_maps, b_gpart, b_total;
  // fp8_bwd and mxfp8: quantised operands inside the backward scratch (zero otherwise)
  moe_fp8_layout q;
  // mxfp8: quantised operands of the forward GEMMs inside the forward scratch
  moe_mxfp8_fwd_layout fq;
};

bool shape_ok(const moe_config *c) {
  if (!c) return false;
  if (c->T < 0 || c->H < 64 || c->I < 64 || c->H % 64 || c->I % 64) return false;
  if (c->E < 1 || c->E > kMaxExperts || c->k < 1 || c->k > kMaxTopK || c->k > c->E) return false;
  if (static_cast<int64_t>(c->T) * c->k >= (int64_t{1} << 31)) return false;
  if (c->precision != MOE_PREC_BF16 && c->precision != MOE_PREC_FP8_BWD &&
      c->precision != MOE_PREC_MXFP8)
    return false;
  // MXFP8 GEMMs stage K in 128-byte blocks and keep scale atoms of 128 rows
  if (c->precision != MOE_PREC_BF16 && (c->H % 128 || c->I % 128)) return false;
  return true;
}

// Padded token capacity of the fp8_bwd operands: every expert's rows rounded
// up to a multiple of 128 fit in M + 127 E, itself rounded up to 128.
inline size_t fp8_mpad(size_t M, size_t E) { return ((M + 127 * E + 127) / 128) * 128; }

// Partials per row of the router weight's gradient that the bf16 dA GEMM
// writes: one per column half of each 256-column tile.
inline int router_grad_parts(int I) { return 2 * ((I + 255) / 256); }

// Scale-atom row grouping: A operands in plain 128-row blocks; B operands (the
// GEMMs' N side) in 192-row groups restarting at every `seg` rows (an expert's
// rows of a weight, or the whole transposed operand).
inline SfLayout sf_a(size_t rows) { return SfLayout{static_cast<int>(rows), 128}; }
inline SfLayout sf_b(size_t seg) { return SfLayout{static_cast<int>(seg), kMxBN}; }

Layout layout_of(const moe_config *c) {
  Layout L{};
  const size_t T = c->T, H = c->H, I = c->I, E = c->E, k = c->k, M = T * k;
  const size_t nblk = static_cast<size_t>(route_num_blocks(c->T));
  const size_t ngroups = static_cast<size_t>(route_scan_groups(c->T));
  size_t o = kHeader;
  L.r_tickets = o;
  o += align256((1 + ngroups) * 4);
  L.r_zero = o;
  L.r_lrank = o;
  o += align256(M);
  L.r_hist = o;
  o += align256(nblk * E * 4);
  L.r_gpref = o;
  o += align256(ngroups * E * 4);
  L.r_total = o;
  o = 0;
  L.s_xperm = o;
  o += align256(M * H * 2);
  L.s_G = o;
  o += align256(M * I * 2);
  L.s_U = o;
  o += align256(M * I * 2);
  L.s_A = o;
  o += align256(M * I * 2);
  L.s_Y = o;
  o += align256(M * H * 2);
  L.s_Aw = o;
  o += align256(M * I * 2);
  if (c->precision != MOE_PREC_BF16) {
    // an MXFP8 backward's dW_down operand, w * A along tokens, written by the
    // forward's gate/up epilogue (instead of the bf16 A_w)
    const size_t Mp = fp8_mpad(M, E);
    L.q.m_pad = Mp;
    L.q.aw_t = o;
    o += align256(I * Mp);
    L.q.aw_t_sf = o;
    o += align256(I * Mp / 32);
  }
  if (c->precision != MOE_PREC_BF16) {
    // the backward's weight operands, written by the forward: in fp8_bwd by the
    // bf16 GEMMs as the weights pass through them, in mxfp8 by its weight passes
    moe_fp8_layout &q = L.q;
    auto take = [&o](size_t bytes) {
      const size_t at = o;
      o += align256(bytes);
      return at;
    };
    q.wd_q = take(E * I * H);
    q.wd_sf = take(sf_layout_bytes(E * I, H, sf_b(I)));
    q.wg_q = take(E * H * I);
    q.wg_sf = take(sf_layout_bytes(E * H, I, sf_b(H)));
    q.wu_q = take(E * H * I);
    q.wu_sf = take(sf_layout_bytes(E * H, I, sf_b(H)));
    // x along tokens (dW_gate/up's A operand), gathered from x by the forward
    q.x_t = take(H * L.q.m_pad);
    q.x_t_sf = take(H * L.q.m_pad / 32);
    if (c->precision == MOE_PREC_MXFP8) {
      moe_mxfp8_fwd_layout &f = L.fq;
      f.bwd_wd_q = q.wd_q;
      f.bwd_wd_sf = q.wd_sf;
      f.bwd_wg_q = q.wg_q;
      f.bwd_wg_sf = q.wg_sf;
      f.bwd_wu_q = q.wu_q;
      f.bwd_wu_sf = q.wu_sf;
    }
  }
  L.s_total = o > 0 ? o : 256;
  o = kHeader;
  if (c->precision == MOE_PREC_FP8_BWD) {
    L.f_pad = o;
    o += align256((E + 1) * 4);
  }
  if (c->precision == MOE_PREC_MXFP8) {
    const size_t Mp = fp8_mpad(M, E);
    moe_mxfp8_fwd_layout &f = L.fq;
    auto take = [&o](size_t bytes) {
      const size_t at = o;
      o += align256(bytes);
      return at;
    };
    f.m_pad = Mp;
    f.pad_offsets = take((E + 1) * 4);
    f.x_q = take(Mp * H);
    f.x_sf = take(Mp * H / 32);
    f.a_q = take(Mp * I);
    f.a_sf = take(Mp * I / 32);
    f.wgu_q = take(E * 2 * I * H);
    f.wgu_sf = take(sf_layout_bytes(E * 2 * I, H, sf_b(2 * I)));
    f.wdt_q = take(E * H * I);
    f.wdt_sf = take(sf_layout_bytes(E * H, I, sf_b(H)));
  }
  L.f_total = o;
  o = kHeader;
  if (c->precision == MOE_PREC_BF16) {  // the fp8 modes quantise dy straight from dy (no bf16 copy)
    L.b_dyp = o;
    o += align256(M * H * 2);
  }
  if (c->precision == MOE_PREC_BF16) {  // fp8_bwd: dG and dU exist only quantised
    L.b_dG = o;
    o += align256(M * I * 2);
    L.b_dU = o;
    o += align256(M * I * 2);
  }
  L.b_dX = o;
  o += align256(M * H * 2);
  L.b_maps = o;
  o += align256(E * kExpertMapBytes);
  // the router weight's gradient in partial sums per row: from the bf16 dA GEMM's
  // epilogue, or from the fp8 modes' pass over dy
  L.b_gpart = o;
  o += align256(M * (c->precision == MOE_PREC_BF16 ? router_grad_parts(c->I) : dy_quant_col_blocks(c->H)) * 4);
  if (c->precision != MOE_PREC_BF16) {
    const size_t Mp = fp8_mpad(M, E);
    moe_fp8_layout &q = L.q;
    q.m_pad = Mp;
    auto take = [&o](size_t bytes) {
      const size_t at = o;
      o += align256(bytes);
      return at;
    };
    q.pad_offsets = take((E + 1) * 4);
    q.dy_q = take(Mp * H);
    q.dy_sf = take(Mp * H / 32);
    q.dg_q = take(Mp * I);
    q.dg_sf = take(Mp * I / 32);
    q.du_q = take(Mp * I);
    q.du_sf = take(Mp * I / 32);
    q.dy_t = take(H * Mp);
    q.dy_t_sf = take(sf_layout_bytes(H, Mp, sf_b(H)));
    q.dg_t = take(I * Mp);
    q.dg_t_sf = take(sf_layout_bytes(I, Mp, sf_b(I)));
    q.du_t = take(I * Mp);
    q.du_t_sf = take(sf_layout_bytes(I, Mp, sf_b(I)));
  }
  L.b_total = o;
  return L;
}

inline bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DevInfo {
  int sms = 0;
  bool ok = false;
};

moe_status device_info(DevInfo *out) {
  static DevInfo cache[kMaxDevices];
  static std::once_flag flags[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
  std::call_once(flags[dev], [dev] {
    int maj = 0, min = 0, sms = 0;
    cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    cache[dev].sms = sms;
    cache[dev].ok = (maj == 10 && min == 3);
  });
  if (!cache[dev].ok) return MOE_ERR_UNSUPPORTED;
  *out = cache[dev];
  return MOE_OK;
}

// ---- optional per-kernel timing
std::atomic<void *const *> g_events{nullptr};
std::atomic<int> g_cap{0};
std::atomic<int> g_count{0};
const char *g_labels[4096];

template <class F>
moe_status timed(const char *label, cudaStream_t s, F &&launch) {
  void *const *ev = g_events.load();
  int slot = -1;
  if (ev) {
    slot = g_count.fetch_add(1);
    if (slot >= g_cap.load() || slot >= 4096) slot = -1;
  }
  if (slot >= 0) {
    g_labels[slot] = label;
    if (cudaEventRecord(static_cast<cudaEvent_t>(ev[2 * slot]), s) != cudaSuccess) {
      cudaGetLastError();  // the failed record, not a launch error
      return MOE_ERR_CUDA;
    }
  }
  cudaError_t e = launch();
  if (slot >= 0 && e == cudaSuccess &&
      cudaEventRecord(static_cast<cudaEvent_t>(ev[2 * slot + 1]), s) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

#define MOE_TRY(x)                      \
  do {                                  \
    moe_status _st = (x);               \
    if (_st != MOE_OK) return _st;      \
  } while (0)

// Token-sized arrays may be null when there are no tokens.
moe_status check_routing(const moe_routing *r, int T) {
  if (!r || !r->counts || !r->offsets) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!r->topk_idx || !r->topk_w || !r->row_of_slot || !r->slot_of_row || !r->w_row))
    return MOE_ERR_INVALID_ARG;
  if (!al16(r->topk_idx) || !al16(r->topk_w) || !al16(r->counts) || !al16(r->offsets) ||
      !al16(r->row_of_slot) || !al16(r->slot_of_row) || !al16(r->w_row))
    return MOE_ERR_ALIGNMENT;
  return MOE_OK;
}

GemmArgs gemm_base(const moe_config *c, const moe_routing *r, int sms, int32_t *status) {
  GemmArgs g{};
  g.M_rows = c->T * c->k;
  g.H = c->H;
  g.I = c->I;
  g.E = c->E;
  g.offsets = r->offsets;
  g.status = status;
  g.num_sms = sms;
  return g;
}

// The fp8_bwd backward after the router backward: each grouped GEMM's operands
// are quantised to MXFP8 along that GEMM's K (weights along rows; activations
// along features into a per-expert padded row space; token-axis operands
// transposed, blocks of 32 tokens from each expert's first row), then the
// block-scaled GEMMs run with the bf16 epilogues.
struct Fp8Bwd {
  const moe_config *cfg;
  const moe_routing *r;
  const moe_fp8_layout *q;
  uint8_t *sc;
  int sms;
  int32_t *status;
  const uint16_t *x, *G, *U, *Y, *dy;
  const uint8_t *aw_t, *aw_t_sf;  // w * A along tokens, from the forward (in `saved`)
  const uint8_t *x_t, *x_t_sf;    // x along tokens, from the forward (in `saved`)
  uint16_t *dX, *dx, *dW_gate, *dW_up, *dW_down;
  float *g_part, *d_logits, *d_topk_w;
  // the weights' codes for the three GEMMs that read them, written by the
  // forward (in `saved`)
  const uint8_t *wd_q, *wd_sf, *wg_q, *wg_sf, *wu_q, *wu_sf;
};

moe_status backward_fp8(const Fp8Bwd &f, cudaStream_t s) {
  const int T = f.cfg->T, H = f.cfg->H, I = f.cfg->I, E = f.cfg->E, k = f.cfg->k;
  const int Mp = static_cast<int>(f.q->m_pad);
  const moe_fp8_layout &q = *f.q;
  uint8_t *sc = f.sc;
  int32_t *pad_off = reinterpret_cast<int32_t *>(sc + q.pad_offsets);
  const int32_t *off = f.r->offsets;
  MOE_TRY(timed("mx_pad_offsets", s, [&] { return launch_pad_offsets(off, E, pad_off, s); }));
  MxGemmArgs m{};
  m.H = H;
  m.I = I;
  m.E = E;
  m.Mpad = Mp;
  m.M = T * k;
  m.offsets = off;
  m.pad_off = pad_off;
  m.G = f.G;
  m.U = f.U;
  m.w_row = f.r->w_row;
  m.status = f.status;
  m.num_sms = f.sms;
  // One pass over dy, read through each permuted row's token: quantised along H
  // (dA's A operand) and along tokens (dW_down's B operand), and g_tj = <dy_t,
  // Y_tj> from the saved Y in partial sums (the MXFP8 dA's accumulator carries
  // dy's and W_down's quantisation error, so the router gradient is not taken
  // from it); the router gradients follow from g.
  const int gcb = dy_quant_col_blocks(H);
  MOE_TRY(timed("mx_dy_quant_gdot", s, [&] {
    return launch_dy_quant(f.dy, f.Y, f.r->slot_of_row, k, H, Mp, off, pad_off, E, sc + q.dy_t, sc + q.dy_t_sf,
                           sf_b(H), RowCodes{sc + q.dy_q, sc + q.dy_sf, sf_a(Mp)}, f.g_part, gcb, s);
  }));
  MOE_TRY(timed("router_grad", s, [&] {
    return launch_router_grad(f.r->row_of_slot, f.r->topk_idx, f.r->topk_w, f.g_part, gcb, f.d_logits,
                              f.d_topk_w, T, E, k, s);
  }));
  // dA = w (Q(dy) . Q(W_down)^T), K = H; dSwiGLU epilogue -> Q(dG), Q(dU) on both axes.
  m.a0 = sc + q.dy_q;
  m.sfa0 = sc + q.dy_sf;
  m.b0 = f.wd_q;
  m.sfb0 = f.wd_sf;
  // dA's epilogue writes dG and dU quantised along I (for dX) and along tokens
  // (for dW_gate/up); they are never stored in bf16
  m.o0 = m.o1 = nullptr;
  m.dg_q = sc + q.dg_q;
  m.dg_sf = sc + q.dg_sf;
  m.du_q = sc + q.du_q;
  m.du_sf = sc + q.du_sf;
  m.dg_t = sc + q.dg_t;
  m.dg_t_sf = sc + q.dg_t_sf;
  m.du_t = sc + q.du_t;
  m.du_t_sf = sc + q.du_t_sf;
  MOE_TRY(timed("mx_gemm_dA_dswiglu", s, [&] { return launch_mx_gemm(kMxGemmDA, m, s); }));
  // dX = Q(dG) . Q(W_gate)^T + Q(dU) . Q(W_up)^T, K = I
  m.a0 = sc + q.dg_q;
  m.sfa0 = sc + q.dg_sf;
  m.a1 = sc + q.du_q;
  m.sfa1 = sc + q.du_sf;
  m.b0 = f.wg_q;
  m.sfb0 = f.wg_sf;
  m.b1 = f.wu_q;
  m.sfb1 = f.wu_sf;
  m.o0 = f.dX;
  m.o1 = nullptr;
  MOE_TRY(timed("mx_gemm_dX", s, [&] { return launch_mx_gemm(kMxGemmDX, m, s); }));
  MOE_TRY(timed("unpermute_sum", s, [&] {
    return launch_gather_sum(f.dX, f.r->row_of_slot, nullptr, f.dx, T, H, k, s);
  }));
  // dW_down = Q(w a)^T . Q(dy), K = the expert's tokens; Q(w a) along tokens comes
  // from the forward's gate/up epilogue
  m.a0 = f.aw_t;
  m.sfa0 = f.aw_t_sf;
  m.b0 = sc + q.dy_t;
  m.sfb0 = sc + q.dy_t_sf;
  m.a1 = m.b1 = m.sfa1 = m.sfb1 = nullptr;
  m.o0 = f.dW_down;
  MOE_TRY(timed("mx_gemm_dW_down", s, [&] { return launch_mx_gemm(kMxGemmDWDown, m, s); }));
  // dW_gate = Q(x)^T . Q(dG), dW_up = Q(x)^T . Q(dU), K = the expert's tokens;
  // Q(x) along tokens comes from the forward
  m.a0 = f.x_t;
  m.sfa0 = f.x_t_sf;
  m.b0 = sc + q.dg_t;
  m.sfb0 = sc + q.dg_t_sf;
  m.b1 = sc + q.du_t;
  m.sfb1 = sc + q.du_t_sf;
  m.o0 = f.dW_gate;
  m.o1 = f.dW_up;
  MOE_TRY(timed("mx_gemm_dW_gateup", s, [&] { return launch_mx_gemm(kMxGemmDWGateUp, m, s); }));
  return MOE_OK;
}

// The mxfp8 forward: both grouped GEMMs in MXFP8.  The permute also quantises
// x along H into the padded row space; the weights along their middle axis,
// transposed (W_gate | W_up interleaved by 32 columns, so one 192-row B tile
// holds 96 gate and the same 96 up columns); GEMM1's epilogue writes the bf16
// activations and A quantised along I; GEMM2 writes Y.
struct Mx8Fwd {
  const moe_config *cfg;
  const moe_routing *r;
  const moe_mxfp8_fwd_layout *q;
  uint8_t *sc;
  int sms;
  int32_t *status;
  const uint16_t *x, *W_gate, *W_up, *W_down;
  uint16_t *x_perm, *A, *G, *U, *A_w, *Y;
  uint8_t *saved;  // the backward's weight codes go here
  uint8_t *aw_t, *aw_t_sf;  // and w * A along tokens
  uint8_t *x_t, *x_t_sf;    // and x along tokens
  bool keep;       // write what the backward reads (the bf16 activations, the weight codes)
};

moe_status forward_mx(const Mx8Fwd &f, cudaStream_t s) {
  const int T = f.cfg->T, H = f.cfg->H, I = f.cfg->I, E = f.cfg->E, k = f.cfg->k;
  const int Mp = static_cast<int>(f.q->m_pad);
  const moe_mxfp8_fwd_layout &q = *f.q;
  uint8_t *sc = f.sc;
  int32_t *pad_off = reinterpret_cast<int32_t *>(sc + q.pad_offsets);
  const int32_t *off = f.r->offsets;
  MOE_TRY(timed("mx_pad_offsets_fwd", s, [&] { return launch_pad_offsets(off, E, pad_off, s); }));
  MOE_TRY(timed("permute_quant_x", s, [&] {
    return launch_permute_quant(f.x, f.r->row_of_slot, f.r->topk_idx, off, pad_off, nullptr, sc + q.x_q,
                                sc + q.x_sf, sf_a(Mp), T, H, k, s);
  }));
  MOE_TRY(timed("mx_zero_pad_rows", s, [&] {
    return launch_zero_pad_rows(off, pad_off, E, H, sc + q.x_q, sc + q.x_sf, sf_a(Mp), s);
  }));
  if (f.keep)  // the backward's dW_gate/up operand: x along tokens, gathered from x by token
    MOE_TRY(timed("mx_quantT_x", s, [&] {
      return launch_quant_cols(f.x, H, Mp, off, pad_off, E, f.x_t, f.x_t_sf, sf_a(H), s,
                               f.r->slot_of_row, k);
    }));
  // each weight read once: along H for GEMM1 (transposed, interleaved) and
  // along I for the backward's dX (row by row, into `saved`)
  MOE_TRY(timed("mx_quant_W_gateup_fwd", s, [&] {
    const RowCodes wg = f.keep ? RowCodes{f.saved + q.bwd_wg_q, f.saved + q.bwd_wg_sf, sf_b(H)} : RowCodes{};
    const RowCodes wu = f.keep ? RowCodes{f.saved + q.bwd_wu_q, f.saved + q.bwd_wu_sf, sf_b(H)} : RowCodes{};
    const cudaError_t e = launch_quant_wT(f.W_gate, E, H, I, 1, 0, sc + q.wgu_q, sc + q.wgu_sf, sf_b(2 * I), wg, s);
    if (e != cudaSuccess) return e;
    return launch_quant_wT(f.W_up, E, H, I, 1, 1, sc + q.wgu_q, sc + q.wgu_sf, sf_b(2 * I), wu, s);
  }));
  MxGemmArgs m{};
  m.H = H;
  m.I = I;
  m.E = E;
  m.Mpad = Mp;
  m.M = T * k;
  m.offsets = off;
  m.pad_off = pad_off;
  m.w_row = f.r->w_row;
  m.status = f.status;
  m.num_sms = f.sms;
  m.a0 = sc + q.x_q;
  m.sfa0 = sc + q.x_sf;
  m.b0 = sc + q.wgu_q;
  m.sfb0 = sc + q.wgu_sf;
  m.o0 = f.keep ? f.A : nullptr;
  m.o1 = f.keep ? f.G : nullptr;
  m.o2 = f.keep ? f.U : nullptr;
  m.o3 = nullptr;  // the backward reads w * A quantised along tokens, not in bf16
  m.aq = sc + q.a_q;
  m.aq_sf = sc + q.a_sf;
  m.aw_t = f.keep ? f.aw_t : nullptr;
  m.aw_t_sf = f.keep ? f.aw_t_sf : nullptr;
  MOE_TRY(timed("mx_gemm_gateup_swiglu", s, [&] { return launch_mx_gemm(kMxGemmGateUp, m, s); }));
  MOE_TRY(timed("mx_quant_W_down_fwd", s, [&] {
    // along I for GEMM2 (transposed) and along H for the backward's dA (row by row, into `saved`)
    return launch_quant_wT(f.W_down, E, I, H, 0, 0, sc + q.wdt_q, sc + q.wdt_sf, sf_b(H),
                           f.keep ? RowCodes{f.saved + q.bwd_wd_q, f.saved + q.bwd_wd_sf, sf_b(I)} : RowCodes{}, s);
  }));
  m.a0 = sc + q.a_q;
  m.sfa0 = sc + q.a_sf;
  m.b0 = sc + q.wdt_q;
  m.sfb0 = sc + q.wdt_sf;
  m.o0 = f.Y;
  m.o1 = m.o2 = m.o3 = nullptr;
  m.aq = m.aq_sf = m.aw_t = m.aw_t_sf = nullptr;
  MOE_TRY(timed("mx_gemm_down", s, [&] { return launch_mx_gemm(kMxGemmDown, m, s); }));
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

namespace moe {
namespace {

// What a forward call leaves behind.  Full: out and everything the backward
// reads (in `saved`).  NoSave: out only (`saved` is used as scratch; a
// checkpointed layer's first pass).  Recompute: what the backward reads, not
// out (a checkpointed layer's second pass, just before the backward).
enum FwdKind { kFwdFull, kFwdNoSave, kFwdRecompute };

moe_status forward_impl(FwdKind kind, const moe_config *cfg, const void *x, const moe_routing *r,
                        const void *W_gate, const void *W_up, const void *W_down, void *out,
                        void *saved, size_t saved_bytes, void *scratch, size_t scratch_bytes,
                        void *stream) {
  const bool need_out = kind != kFwdRecompute;
  if (!shape_ok(cfg)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_routing(r, cfg->T));
  if (!W_gate || !W_up || !W_down || !saved || !scratch || (cfg->T > 0 && (!x || (need_out && !out))))
    return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(W_gate) || !al16(W_up) || !al16(W_down) || (need_out && !al16(out)) ||
      !al16(saved) || !al16(scratch))
    return MOE_ERR_ALIGNMENT;
  const Layout L = layout_of(cfg);
  if (saved_bytes < L.s_total || scratch_bytes < L.f_total) return MOE_ERR_WORKSPACE;
  DevInfo di;
  MOE_TRY(device_info(&di));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *sc = static_cast<uint8_t *>(scratch);
  uint8_t *sv = static_cast<uint8_t *>(saved);
  if (cudaMemsetAsync(sc, 0, kHeader, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cfg->T == 0) return MOE_OK;
  const int T = cfg->T, H = cfg->H, k = cfg->k;
  int32_t *status = reinterpret_cast<int32_t *>(sc);
  uint16_t *x_perm = reinterpret_cast<uint16_t *>(sv + L.s_xperm);
  uint16_t *G = reinterpret_cast<uint16_t *>(sv + L.s_G);
  uint16_t *U = reinterpret_cast<uint16_t *>(sv + L.s_U);
  uint16_t *A = reinterpret_cast<uint16_t *>(sv + L.s_A);
  uint16_t *Y = reinterpret_cast<uint16_t *>(sv + L.s_Y);
  uint16_t *A_w = reinterpret_cast<uint16_t *>(sv + L.s_Aw);

  if (cfg->precision == MOE_PREC_MXFP8) {
    Mx8Fwd f;
    f.cfg = cfg;
    f.r = r;
    f.q = &L.fq;
    f.sc = sc;
    f.sms = di.sms;
    f.status = status;
    f.x = static_cast<const uint16_t *>(x);
    f.x_perm = x_perm;
    f.W_gate = static_cast<const uint16_t *>(W_gate);
    f.W_up = static_cast<const uint16_t *>(W_up);
    f.W_down = static_cast<const uint16_t *>(W_down);
    f.A = A;
    f.G = G;
    f.U = U;
    f.aw_t = sv + L.q.aw_t;
    f.aw_t_sf = sv + L.q.aw_t_sf;
    f.Y = Y;
    f.saved = sv;
    f.aw_t = sv + L.q.aw_t;
    f.aw_t_sf = sv + L.q.aw_t_sf;
    f.x_t = sv + L.q.x_t;
    f.x_t_sf = sv + L.q.x_t_sf;
    f.keep = kind != kFwdNoSave;
    MOE_TRY(forward_mx(f, s));
  } else {
    const bool keep = kind != kFwdNoSave;  // G, U and w * A are only the backward's
    const bool fp8b = cfg->precision == MOE_PREC_FP8_BWD;  // its dW_down reads w * A quantised along tokens
    if (keep && fp8b) {
      // the permute in destination order, fused with x quantised along tokens
      // (dW_gate/up's A operand in the MXFP8 backward) into the padded token axis
      int32_t *pad_off = reinterpret_cast<int32_t *>(sc + L.f_pad);
      MOE_TRY(timed("mx_pad_offsets_fwd", s, [&] { return launch_pad_offsets(r->offsets, cfg->E, pad_off, s); }));
      MOE_TRY(timed("permute_rows_quantT_x", s, [&] {
        return launch_quant_cols(static_cast<const uint16_t *>(x), H, static_cast<int>(L.q.m_pad), r->offsets,
                                 pad_off, cfg->E, sv + L.q.x_t, sv + L.q.x_t_sf, sf_a(H), s,
                                 r->slot_of_row, k, x_perm);
      }));
    } else {
      MOE_TRY(timed("permute_rows", s, [&] {
        return launch_permute_rows(static_cast<const uint16_t *>(x), r->row_of_slot, x_perm, T, H, k, s);
      }));
    }
    GemmArgs g = gemm_base(cfg, r, di.sms, status);
    g.x_perm = x_perm;
    g.W_gate = static_cast<const uint16_t *>(W_gate);
    g.W_up = static_cast<const uint16_t *>(W_up);
    g.W_down = static_cast<const uint16_t *>(W_down);
    g.w_row = r->w_row;
    g.o0 = A;
    g.o1 = keep ? G : nullptr;
    g.o2 = keep ? U : nullptr;
    g.o3 = keep && !fp8b ? A_w : nullptr;
    g.aw_t = keep && fp8b ? sv + L.q.aw_t : nullptr;
    g.aw_t_sf = keep && fp8b ? sv + L.q.aw_t_sf : nullptr;
    g.Mpad = static_cast<int>(L.q.m_pad);
    if (keep && fp8b) {  // the backward's W_gate and W_up codes, quantised as they pass through GEMM1
      g.wq[0] = sv + L.q.wg_q;
      g.wq_sf[0] = sv + L.q.wg_sf;
      g.wq[1] = sv + L.q.wu_q;
      g.wq_sf[1] = sv + L.q.wu_sf;
    }
    MOE_TRY(timed(gemm_mode_name(kFwdGateUp), s, [&] { return launch_grouped_gemm(kFwdGateUp, g, s); }));
    // the bf16 backward never reads Y (its router gradient comes from the dA GEMM),
    // so a recompute for it stops after GEMM1; the fp8 modes' backward reads Y
    if (kind == kFwdRecompute && cfg->precision == MOE_PREC_BF16) return MOE_OK;
    g.act = A;
    g.o0 = Y;
    g.o1 = g.o2 = g.o3 = nullptr;
    g.aw_t = g.aw_t_sf = nullptr;
    g.wq[0] = keep && fp8b ? sv + L.q.wd_q : nullptr;  // and W_down's, through GEMM2
    g.wq_sf[0] = keep && fp8b ? sv + L.q.wd_sf : nullptr;
    g.wq[1] = g.wq_sf[1] = nullptr;
    MOE_TRY(timed(gemm_mode_name(kFwdDown), s, [&] { return launch_grouped_gemm(kFwdDown, g, s); }));
  }
  if (kind == kFwdRecompute) return MOE_OK;
  MOE_TRY(timed("combine", s, [&] {
    return launch_gather_sum(Y, r->row_of_slot, r->topk_w, static_cast<uint16_t *>(out), T, H, k,
                             s);
  }));
  return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" {

moe_status moe_query_workspace(const moe_config *cfg, size_t *route_scratch, size_t *saved,
                               size_t *fwd_scratch, size_t *bwd_scratch) {
  if (!shape_ok(cfg)) return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(cfg);
  if (route_scratch) *route_scratch = L.r_total;
  if (saved) *saved = L.s_total;
  if (fwd_scratch) *fwd_scratch = L.f_total;
  if (bwd_scratch) *bwd_scratch = L.b_total;
  return MOE_OK;
}

moe_status moe_saved_offsets(const moe_config *cfg, moe_saved_layout *out) {
  if (!shape_ok(cfg) || !out) return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(cfg);
  out->x_perm = L.s_xperm;
  out->G = L.s_G;
  out->U = L.s_U;
  out->A = L.s_A;
  out->Y = L.s_Y;
  out->A_w = L.s_Aw;
  return MOE_OK;
}

moe_status moe_mxfp8_forward_offsets(const moe_config *cfg, moe_mxfp8_fwd_layout *out) {
  if (!shape_ok(cfg) || !out || cfg->precision != MOE_PREC_MXFP8) return MOE_ERR_INVALID_ARG;
  *out = layout_of(cfg).fq;
  return MOE_OK;
}

moe_status moe_fp8_scratch_offsets(const moe_config *cfg, moe_fp8_layout *out) {
  if (!shape_ok(cfg) || !out || cfg->precision == MOE_PREC_BF16) return MOE_ERR_INVALID_ARG;
  *out = layout_of(cfg).q;
  return MOE_OK;
}

moe_status moe_route(const moe_config *cfg, const float *logits, const moe_routing *r,
                     void *scratch, size_t scratch_bytes, void *stream) {
  if (!shape_ok(cfg)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_routing(r, cfg->T));
  if (!scratch || (cfg->T > 0 && !logits)) return MOE_ERR_INVALID_ARG;
  if (!al16(scratch) || !al16(logits)) return MOE_ERR_ALIGNMENT;
  const Layout L = layout_of(cfg);
  if (scratch_bytes < L.r_total) return MOE_ERR_WORKSPACE;
  DevInfo di;
  MOE_TRY(device_info(&di));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *sc = static_cast<uint8_t *>(scratch);
  if (cudaMemsetAsync(sc, 0, L.r_zero, s) != cudaSuccess) return MOE_ERR_CUDA;  // status and scan tickets
  if (cfg->T == 0) {  // no tokens: empty groups
    if (cudaMemsetAsync(r->counts, 0, sizeof(int32_t) * cfg->E, s) != cudaSuccess ||
        cudaMemsetAsync(r->offsets, 0, sizeof(int32_t) * (cfg->E + 1), s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  RouteArgs a{};
  a.logits = logits;
  a.T = cfg->T;
  a.E = cfg->E;
  a.k = cfg->k;
  a.topk_idx = r->topk_idx;
  a.topk_w = r->topk_w;
  a.counts = r->counts;
  a.offsets = r->offsets;
  a.row_of_slot = r->row_of_slot;
  a.slot_of_row = r->slot_of_row;
  a.w_row = r->w_row;
  a.lrank = sc + L.r_lrank;
  a.hist = reinterpret_cast<int32_t *>(sc + L.r_hist);
  a.gpref = reinterpret_cast<int32_t *>(sc + L.r_gpref);
  a.tickets = reinterpret_cast<int32_t *>(sc + L.r_tickets);
  a.status = reinterpret_cast<int32_t *>(sc);
  MOE_TRY(timed("route_topk", s, [&] { return launch_route_topk(a, s); }));
  MOE_TRY(timed("route_index", s, [&] { return launch_route_index(a, s); }));
  return MOE_OK;
}

moe_status moe_forward(const moe_config *cfg, const void *x, const moe_routing *r,
                       const void *W_gate, const void *W_up, const void *W_down, void *out,
                       void *saved, size_t saved_bytes, void *scratch, size_t scratch_bytes,
                       void *stream) {
  return moe::forward_impl(moe::kFwdFull, cfg, x, r, W_gate, W_up, W_down, out, saved, saved_bytes, scratch,
                           scratch_bytes, stream);
}

moe_status moe_forward_nosave(const moe_config *cfg, const void *x, const moe_routing *r,
                              const void *W_gate, const void *W_up, const void *W_down, void *out,
                              void *saved, size_t saved_bytes, void *scratch, size_t scratch_bytes,
                              void *stream) {
  return moe::forward_impl(moe::kFwdNoSave, cfg, x, r, W_gate, W_up, W_down, out, saved, saved_bytes, scratch,
                           scratch_bytes, stream);
}

moe_status moe_forward_recompute(const moe_config *cfg, const void *x, const moe_routing *r,
                                 const void *W_gate, const void *W_up, const void *W_down, void *saved,
                                 size_t saved_bytes, void *scratch, size_t scratch_bytes, void *stream) {
  return moe::forward_impl(moe::kFwdRecompute, cfg, x, r, W_gate, W_up, W_down, nullptr, saved, saved_bytes,
                           scratch, scratch_bytes, stream);
}

moe_status moe_backward(const moe_config *cfg, const void *dy, const void *x,
                        const moe_routing *r, const void *W_gate, const void *W_up,
                        const void *W_down, const void *saved, size_t saved_bytes, void *dx,
                        void *dW_gate, void *dW_up, void *dW_down, float *d_logits,
                        float *d_topk_w, void *scratch, size_t scratch_bytes, void *stream) {
  if (!shape_ok(cfg)) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_routing(r, cfg->T));
  if (!W_gate || !W_up || !W_down || !saved || !dW_gate || !dW_up || !dW_down || !scratch ||
      (cfg->T > 0 && (!dy || !x || !dx || !d_logits)))
    return MOE_ERR_INVALID_ARG;
  if (!al16(dy) || !al16(x) || !al16(W_gate) || !al16(W_up) || !al16(W_down) || !al16(saved) ||
      !al16(dx) || !al16(dW_gate) || !al16(dW_up) || !al16(dW_down) || !al16(d_logits) ||
      !al16(scratch) || (d_topk_w && !al16(d_topk_w)))
    return MOE_ERR_ALIGNMENT;
  const Layout L = layout_of(cfg);
  if (saved_bytes < L.s_total || scratch_bytes < L.b_total) return MOE_ERR_WORKSPACE;
  DevInfo di;
  MOE_TRY(device_info(&di));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *sc = static_cast<uint8_t *>(scratch);
  const uint8_t *sv = static_cast<const uint8_t *>(saved);
  if (cudaMemsetAsync(sc, 0, kHeader, s) != cudaSuccess) return MOE_ERR_CUDA;
  const int T = cfg->T, H = cfg->H, I = cfg->I, E = cfg->E, k = cfg->k;
  if (T == 0) {  // every expert is empty: weight gradients are zero
    const size_t wbytes = static_cast<size_t>(E) * H * I * 2;
    if (cudaMemsetAsync(dW_gate, 0, wbytes, s) != cudaSuccess ||
        cudaMemsetAsync(dW_up, 0, wbytes, s) != cudaSuccess ||
        cudaMemsetAsync(dW_down, 0, wbytes, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  int32_t *status = reinterpret_cast<int32_t *>(sc);
  const uint16_t *x_perm = reinterpret_cast<const uint16_t *>(sv + L.s_xperm);
  const uint16_t *G = reinterpret_cast<const uint16_t *>(sv + L.s_G);
  const uint16_t *U = reinterpret_cast<const uint16_t *>(sv + L.s_U);
  const uint16_t *A = reinterpret_cast<const uint16_t *>(sv + L.s_A);
  const uint16_t *Y = reinterpret_cast<const uint16_t *>(sv + L.s_Y);
  const uint16_t *A_w = reinterpret_cast<const uint16_t *>(sv + L.s_Aw);
  uint16_t *dy_perm = reinterpret_cast<uint16_t *>(sc + L.b_dyp);  // bf16 only
  float *g_part = reinterpret_cast<float *>(sc + L.b_gpart);
  uint16_t *dG = reinterpret_cast<uint16_t *>(sc + L.b_dG);
  uint16_t *dU = reinterpret_cast<uint16_t *>(sc + L.b_dU);
  uint16_t *dX = reinterpret_cast<uint16_t *>(sc + L.b_dX);

  if (cfg->precision != MOE_PREC_BF16) {
    Fp8Bwd f;
    f.cfg = cfg;
    f.r = r;
    f.q = &L.q;
    f.sc = sc;
    f.sms = di.sms;
    f.status = status;
    f.x = static_cast<const uint16_t *>(x);
    f.G = G;
    f.U = U;
    f.aw_t = sv + L.q.aw_t;
    f.aw_t_sf = sv + L.q.aw_t_sf;
    f.x_t = sv + L.q.x_t;
    f.x_t_sf = sv + L.q.x_t_sf;
    f.Y = Y;
    f.dy = static_cast<const uint16_t *>(dy);
    f.g_part = g_part;
    f.d_logits = d_logits;
    f.d_topk_w = d_topk_w;
    f.dX = dX;
    f.dx = static_cast<uint16_t *>(dx);
    f.dW_gate = static_cast<uint16_t *>(dW_gate);
    f.dW_up = static_cast<uint16_t *>(dW_up);
    f.dW_down = static_cast<uint16_t *>(dW_down);
    f.wd_q = sv + L.q.wd_q;
    f.wd_sf = sv + L.q.wd_sf;
    f.wg_q = sv + L.q.wg_q;
    f.wg_sf = sv + L.q.wg_sf;
    f.wu_q = sv + L.q.wu_q;
    f.wu_sf = sv + L.q.wu_sf;
    return backward_fp8(f, s);
  }
  // bf16: dy is permuted; the router weight's gradient g_tj = <dy_t . W_down^T,
  // A_r> comes from the dA GEMM's epilogue (Y is not read again)
  MOE_TRY(timed("permute_dy", s, [&] {
    return launch_permute_rows(static_cast<const uint16_t *>(dy), r->row_of_slot, dy_perm, T, H, k, s);
  }));
  (void)Y;
  GemmArgs g = gemm_base(cfg, r, di.sms, status);
  g.x_perm = x_perm;
  g.W_gate = static_cast<const uint16_t *>(W_gate);
  g.W_up = static_cast<const uint16_t *>(W_up);
  g.W_down = static_cast<const uint16_t *>(W_down);
  g.act = A;
  g.g_part = g_part;
  g.G = G;
  g.U = U;
  g.dy_perm = dy_perm;
  g.map_scratch = sc + L.b_maps;
  g.act_w = A_w;
  g.w_row = r->w_row;
  g.dG = dG;
  g.dU = dU;
  g.o0 = dG;
  g.o1 = dU;
  MOE_TRY(timed(gemm_mode_name(kBwdDA), s, [&] { return launch_grouped_gemm(kBwdDA, g, s); }));
  g.g_part = nullptr;
  MOE_TRY(timed("router_grad", s, [&] {
    return launch_router_grad(r->row_of_slot, r->topk_idx, r->topk_w, g_part, router_grad_parts(I), d_logits,
                              d_topk_w, T, E, k, s);
  }));
  g.o0 = dX;
  g.o1 = nullptr;
  MOE_TRY(timed(gemm_mode_name(kBwdDX), s, [&] { return launch_grouped_gemm(kBwdDX, g, s); }));
  MOE_TRY(timed("unpermute_sum", s, [&] {
    return launch_gather_sum(dX, r->row_of_slot, nullptr, static_cast<uint16_t *>(dx), T, H, k, s);
  }));
  g.o0 = static_cast<uint16_t *>(dW_down);
  MOE_TRY(timed(gemm_mode_name(kBwdDWDown), s, [&] { return launch_grouped_gemm(kBwdDWDown, g, s); }));
  g.o0 = static_cast<uint16_t *>(dW_gate);
  g.o1 = static_cast<uint16_t *>(dW_up);
  MOE_TRY(timed(gemm_mode_name(kBwdDWGateUp), s,
                [&] { return launch_grouped_gemm(kBwdDWGateUp, g, s); }));
  (void)I;
  return MOE_OK;
}

// ---- router projection (logits = x . W_r and its backward)

namespace {
bool router_shape_ok(const moe_config *c) {
  if (!c) return false;
  if (c->T < 0 || c->H < 64 || c->H % 64) return false;
  if (c->E < 8 || c->E > kMaxExperts || c->E % 8) return false;  // 16-byte rows for the TMA
  return true;
}
constexpr size_t kRouterSplit = kHeader;          // int32 [S + 1]: the weight gradient's token segments
constexpr size_t kRouterMaps = kHeader + 256;     // 3 tensor maps per segment for the weight gradient
// Backward scratch after the maps: fp32 partials [S][H][E] of the weight
// gradient when it is split (S > 1), then bf16 d_logits [T,E].
struct RouterBwdLayout {
  int S;
  size_t parts, dlog, total;
};
RouterBwdLayout router_bwd_layout(const moe_config *c) {
  RouterBwdLayout L{};
  L.S = router_dw_segments(c->T, c->H, c->E);
  L.parts = kRouterMaps + align256(static_cast<size_t>(L.S) * kExpertMapBytes);
  L.dlog = L.parts + (L.S > 1 ? align256(static_cast<size_t>(L.S) * c->H * c->E * 4) : 0);
  L.total = L.dlog + align256(static_cast<size_t>(c->T) * c->E * 2);
  return L;
}
}  // namespace

moe_status moe_router_workspace(const moe_config *cfg, size_t *fwd_scratch, size_t *bwd_scratch) {
  if (!router_shape_ok(cfg)) return MOE_ERR_INVALID_ARG;
  if (fwd_scratch) *fwd_scratch = kRouterMaps;
  if (bwd_scratch) *bwd_scratch = router_bwd_layout(cfg).total;
  return MOE_OK;
}

moe_status moe_router_forward(const moe_config *cfg, const void *x, const void *W_r, float *logits,
                              void *scratch, size_t scratch_bytes, void *stream) {
  if (!router_shape_ok(cfg)) return MOE_ERR_INVALID_ARG;
  if (!W_r || !scratch || (cfg->T > 0 && (!x || !logits))) return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(W_r) || !al16(logits) || !al16(scratch)) return MOE_ERR_ALIGNMENT;
  if (scratch_bytes < kRouterMaps) return MOE_ERR_WORKSPACE;
  DevInfo di;
  MOE_TRY(device_info(&di));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *sc = static_cast<uint8_t *>(scratch);
  if (cudaMemsetAsync(sc, 0, kHeader, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cfg->T == 0) return MOE_OK;
  GemmArgs g{};  // no offsets: one segment of T rows
  g.M_rows = cfg->T;
  g.H = cfg->H;
  g.E = cfg->E;
  g.r_x = static_cast<const uint16_t *>(x);
  g.r_w = static_cast<const uint16_t *>(W_r);
  g.r_out = logits;
  g.status = reinterpret_cast<int32_t *>(sc);
  g.num_sms = di.sms;
  MOE_TRY(timed(gemm_mode_name(kRouterFwd), s, [&] { return launch_grouped_gemm(kRouterFwd, g, s); }));
  return MOE_OK;
}

moe_status moe_router_backward(const moe_config *cfg, const void *x, const void *W_r,
                               const float *d_logits, void *dx, float *dW_r, void *scratch,
                               size_t scratch_bytes, void *stream) {
  if (!router_shape_ok(cfg)) return MOE_ERR_INVALID_ARG;
  if (!W_r || !dW_r || !scratch || (cfg->T > 0 && (!x || !d_logits || !dx)))
    return MOE_ERR_INVALID_ARG;
  if (!al16(x) || !al16(W_r) || !al16(d_logits) || !al16(dx) || !al16(dW_r) || !al16(scratch))
    return MOE_ERR_ALIGNMENT;
  size_t need = 0;
  moe_router_workspace(cfg, nullptr, &need);
  if (scratch_bytes < need) return MOE_ERR_WORKSPACE;
  DevInfo di;
  MOE_TRY(device_info(&di));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *sc = static_cast<uint8_t *>(scratch);
  if (cudaMemsetAsync(sc, 0, kHeader, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cfg->T == 0) {  // no tokens: dW_r = 0, dx untouched
    if (cudaMemsetAsync(dW_r, 0, sizeof(float) * cfg->H * cfg->E, s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  const RouterBwdLayout RL = router_bwd_layout(cfg);
  int32_t *split = reinterpret_cast<int32_t *>(sc + kRouterSplit);
  uint16_t *dlog = reinterpret_cast<uint16_t *>(sc + RL.dlog);
  float *parts = reinterpret_cast<float *>(sc + RL.parts);
  MOE_TRY(timed("router_dlogits_bf16", s, [&] {
    return launch_router_dlogits(d_logits, dlog, static_cast<int64_t>(cfg->T) * cfg->E, split, cfg->T, RL.S, s);
  }));
  GemmArgs g{};  // dx: no offsets, one segment of T rows
  g.M_rows = cfg->T;
  g.H = cfg->H;
  g.E = cfg->E;
  g.r_x = static_cast<const uint16_t *>(x);
  g.r_w = static_cast<const uint16_t *>(W_r);
  g.r_dlog = dlog;
  g.o0 = static_cast<uint16_t *>(dx);
  g.r_out = dW_r;
  g.map_scratch = sc + kRouterMaps;
  g.status = reinterpret_cast<int32_t *>(sc);
  g.num_sms = di.sms;
  MOE_TRY(timed(gemm_mode_name(kRouterDX), s, [&] { return launch_grouped_gemm(kRouterDX, g, s); }));
  // the weight gradient reduces over all T tokens into only ceil(H/256) x ceil(E/256)
  // tiles: split the tokens into S segments (partials), then add them in order
  g.offsets = split;
  g.r_segments = RL.S;
  g.r_out = RL.S > 1 ? parts : dW_r;
  MOE_TRY(timed(gemm_mode_name(kRouterDW), s, [&] { return launch_grouped_gemm(kRouterDW, g, s); }));
  if (RL.S > 1)
    MOE_TRY(timed("router_dW_sum", s, [&] {
      return launch_sum_segments(parts, RL.S, static_cast<int64_t>(cfg->H) * cfg->E, dW_r, s);
    }));
  return MOE_OK;
}

moe_status moe_get_device_status(const void *scratch, void *stream, int32_t *host_code) {
  if (!scratch || !host_code) return MOE_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return MOE_ERR_CUDA;
  int32_t v = 0;
  if (cudaMemcpy(&v, scratch, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  *host_code = v;
  return v == 0 ? MOE_OK : MOE_ERR_DEVICE;
}

const char *moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null pointer, shape or precision)";
    case MOE_ERR_ALIGNMENT: return "pointer not 16-byte aligned";
    case MOE_ERR_WORKSPACE: return "workspace smaller than moe_query_workspace requires";
    case MOE_ERR_UNSUPPORTED: return "unsupported device or precision";
    case MOE_ERR_CUDA: return "CUDA call failed";
    case MOE_ERR_DEVICE: return "device reported an anomaly (see status flags)";
  }
  return "unknown status";
}

moe_status moe_timing_attach(void *const *events, int32_t capacity) {
  if (events && capacity <= 0) return MOE_ERR_INVALID_ARG;
  g_events.store(nullptr);
  g_count.store(0);
  g_cap.store(events ? capacity : 0);
  g_events.store(events);
  return MOE_OK;
}

int32_t moe_timing_count(void) {
  const int n = g_count.load(), c = g_cap.load();
  return n < c ? n : c;
}

const char *moe_timing_label(int32_t i) {
  if (i < 0 || i >= moe_timing_count() || i >= 4096) return nullptr;
  return g_labels[i];
}

}  // extern "C"
