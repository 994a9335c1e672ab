// internal.h -- host-side declarations shared by the library's translation
// units (kernel launchers called by the C-ABI in api.cu).  Not installed.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>
#include <utility>

namespace moe {

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 16;

// Per-device one-time setup of a launcher (a kernel's shared-memory opt-in, an
// occupancy query): setup(&value) runs once per device under std::call_once,
// so concurrent first calls from several host threads are safe, and its
// result and value are returned on every later call for that device.
constexpr int kMaxDevices = 64;
struct DeviceOnce {
  std::once_flag flag[kMaxDevices];
  cudaError_t err[kMaxDevices] = {};
  int value[kMaxDevices] = {};
  template <class Setup>
  cudaError_t get(Setup &&setup, int *out = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::call_once(flag[dev], [&] { err[dev] = setup(&value[dev]); });
    if (out) *out = value[dev];
    return err[dev];
  }
};

// Launches `kernel` on stream s allowed to start before the kernel ahead of it
// in the stream has finished (programmatic dependent launch); the kernel waits
// for that one's completion (griddepcontrol.wait) before it reads its outputs.
// Optionally as clusters of `cluster` CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster,
                       Args &&...args) {
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  return e != cudaSuccess ? e : cudaGetLastError();
}

// Status flags written by kernels into the scratch status word.
constexpr int32_t kDevNonfiniteLogit = 0x1;
constexpr int32_t kDevWaitTimeout = 0x2;

// ---- routing (route.cu)
constexpr int kRouteTokensPerBlock = 64;  // tokens per route block (one histogram row)
constexpr int kRouteThreads = 256;        // four per token; at least kMaxExperts

struct RouteArgs {
  const float *logits;  // [T,E]
  int T, E, k;
  int32_t *topk_idx;    // [T,k]
  float *topk_w;        // [T,k]
  int32_t *counts;      // [E]
  int32_t *offsets;     // [E+1]
  int32_t *row_of_slot; // [T*k]
  int32_t *slot_of_row; // [T*k]
  float *w_row;         // [T*k]
  uint8_t *lrank;       // [T*k] scratch: rank of a slot among its block's slots of the same expert
  int32_t *hist;        // [nblk,E] scratch: per-block expert histogram, then its prefix inside its scan group
  int32_t *gpref;       // [ngroups,E] scratch: group totals, then their exclusive prefix over groups
  int32_t *tickets;     // [1 + ngroups] scratch, zero on entry: arrival counters of the scan
  int32_t *status;      // scratch status word
};
int route_num_blocks(int T);
int route_scan_groups(int T);
cudaError_t launch_route_topk(const RouteArgs &a, cudaStream_t s);
cudaError_t launch_route_index(const RouteArgs &a, cudaStream_t s);

// ---- row movement (gather.cu)
// x_perm[row_of_slot[t,j]] = x[t]
cudaError_t launch_permute_rows(const uint16_t *x, const int32_t *row_of_slot, uint16_t *x_perm,
                                int T, int H, int k, cudaStream_t s);
// out[t] = sum_j w[t,j] * rows[row_of_slot[t,j]]   (w == nullptr: plain sum)
cudaError_t launch_gather_sum(const uint16_t *rows, const int32_t *row_of_slot, const float *w,
                              uint16_t *out, int T, int H, int k, cudaStream_t s);
// router projection: fp32 -> bf16 (nearest even), n % 4 == 0; offsets {0, T}
// the router's d_logits [T,E] fp32 -> bf16 (n = T * E), and split = the S + 1
// offsets of S equal token segments for the weight gradient (S <= 63)
cudaError_t launch_router_dlogits(const float *d_logits, uint16_t *out, int64_t n, int32_t *split, int T, int S,
                                  cudaStream_t s);
// out [n] = sum over s of parts [S][n], in order of s (n a multiple of 8)
cudaError_t launch_sum_segments(const float *parts, int S, int64_t n, float *out, cudaStream_t s);
// d_logits and d_topk_w from g computed in the bf16 dA epilogue: g[r] = the sum
// of the np partials g_part[r * np + p]
cudaError_t launch_router_grad(const int32_t *row_of_slot, const int32_t *topk_idx, const float *topk_w,
                               const float *g_part, int np, float *d_logits, float *d_topk_w, int T, int E, int k,
                               cudaStream_t s);
// ---- grouped GEMMs (gemm.cu)
enum GemmMode : int {
  kFwdGateUp = 0,   // [x_perm] . [W_gate | W_up]  -> SwiGLU epilogue: A, G, U, A_w  (ragged M)
  kFwdDown = 1,     // A . W_down                 -> Y                              (ragged M)
  kBwdDA = 2,       // dy_perm . W_down^T, times w -> dSwiGLU epilogue: dG, dU      (ragged M)
  kBwdDX = 3,       // [dG | dU] . [W_gate | W_up]^T -> dX_perm                     (ragged M)
  kBwdDWDown = 4,   // A_w^T . dy_perm            -> dW_down                        (ragged K)
  kBwdDWGateUp = 5, // x_perm^T . [dG | dU]       -> dW_gate, dW_up                 (ragged K)
  // router projection: one "expert" spanning all T tokens
  kRouterFwd = 6,   // x . W_r                    -> logits fp32                    (ragged M)
  kRouterDX = 7,    // bf16(d_logits) . W_r^T     -> dx += (bf16, in place)         (ragged M)
  kRouterDW = 8     // x^T . bf16(d_logits)       -> dW_r fp32                      (ragged K)
};

struct GemmArgs {
  int M_rows;  // permuted rows M = T*k
  int H, I, E;
  const int32_t *offsets;  // [E+1] expert row offsets (device)
  // operands (device, bf16)
  const uint16_t *x_perm, *W_gate, *W_up, *W_down;
  const uint16_t *act;    // A [M,I]
  const uint16_t *act_w;  // A_w = w * A [M,I]
  const uint16_t *G, *U;
  const uint16_t *dy_perm;  // dy rows in permuted order [M,H]
  const uint16_t *dG, *dU;
  const float *w_row;       // [M] router weight per permuted row
  float *g_part;            // dA: the router weight's gradient, 2 partials per 256-column tile [M][np]
  // outputs (device, bf16)
  uint16_t *o0, *o1, *o2, *o3;
  // gate/up for an MXFP8 backward: w * A quantised along tokens into the padded
  // token axis (codes [I, Mpad], scales in 128-row atoms over K = Mpad), or null
  uint8_t *aw_t, *aw_t_sf;
  int Mpad;
  // forward GEMMs for an MXFP8 backward: the weights quantised along their last
  // axis as they pass through the GEMM (gate/up: W_gate [0] and W_up [1] as
  // [E*H, I]; down: W_down [0] as [E*I, H]; codes and scale atoms), or null
  uint8_t *wq[2], *wq_sf[2];
  // router projection: x [T,H], W_r [H,E], d_logits as bf16 [T,E]; fp32 output, its columns
  const uint16_t *r_x, *r_w, *r_dlog;
  float *r_out;
  int r_segments;  // dW_r: token segments reduced separately (offsets[0..S]), partials [S][H][E] in r_out
  int32_t *status;
  void *map_scratch;  // ragged K: device scratch for E * 3 tensor maps (128 B each, 128-B aligned)
  int num_sms;
};
constexpr size_t kExpertMapBytes = 3 * 128;  // per expert
cudaError_t launch_grouped_gemm(GemmMode mode, const GemmArgs &a, cudaStream_t s);
// dW_r = x^T . d_logits split over the tokens: how many segments keep every CTA
// pair of the part (152 SMs) busy, at least 1024 tokens each; 1 = no split.
int router_dw_segments(int T, int H, int E);
const char *gemm_mode_name(GemmMode mode);

// ---- MXFP8 backward (mxfp8.cu, gemm_mx.cu)
// Row grouping of a scale-atom buffer: segments of `seg` rows, each cut into
// groups of `group` rows (128, or kMxBN for B operands), each group spanning
// ceil(group/128) 128-row atoms.
constexpr int kMxBN = 192;  // N extent of an MXFP8 GEMM tile
struct SfLayout {
  int seg, group;
};
inline size_t sf_layout_bytes(size_t rows, size_t K, SfLayout L) {
  const size_t nseg = (rows + L.seg - 1) / L.seg, gps = (L.seg + L.group - 1) / L.group;
  const size_t apg = (L.group + 127) / 128;
  return nseg * gps * apg * (K / 128) * 512;
}
// pad_off[e] = sum over e' < e of ceil(count/128)*128
cudaError_t launch_pad_offsets(const int32_t *offsets, int E, int32_t *pad_off, cudaStream_t s);
// Codes and scales of an operand quantised row by row (along its columns).
struct RowCodes {
  uint8_t *codes, *sf;
  SfLayout L;
};
// along tokens: [M, C] permuted rows -> codes [C, Mpad] (padded token axis;
// scales in one segment, groups of 128: L.seg >= C, L.group == 128; or none,
// codes == nullptr).  With slot_of_row set, src is token-major ([T, C]) and
// permuted row r reads token slot_of_row[r] / k; with xp set, the permuted
// rows are also written in bf16 to xp [M, C] (a permute fused with the
// quantisation).  Other layouts: cudaErrorInvalidValue.
cudaError_t launch_quant_cols(const uint16_t *src, int C, int Mpad, const int32_t *offsets,
                              const int32_t *pad_off, int E, uint8_t *codes, uint8_t *sf, SfLayout L,
                              cudaStream_t s, const int32_t *slot_of_row = nullptr, int k = 1,
                              uint16_t *xp = nullptr);

// The MXFP8 backward's one pass over dy: dy rows gathered by token for every
// permuted row, quantised along H into the padded row space (rows) and along
// tokens (codes_t [H, Mpad]), and g = <dy_t, Y_r> in col_blocks partial sums per
// row (g_part [M][col_blocks], added in order by launch_router_grad).  Both
// scale layouts are one segment: Lt grouped by kMxBN, rows.L by 128; other
// layouts: cudaErrorInvalidValue.
cudaError_t launch_dy_quant(const uint16_t *dy, const uint16_t *Y, const int32_t *slot_of_row, int k, int H,
                            int Mpad, const int32_t *offsets, const int32_t *pad_off, int E, uint8_t *codes_t,
                            uint8_t *sf_t, SfLayout Lt, RowCodes rows, float *g_part, int col_blocks,
                            cudaStream_t s);
int dy_quant_col_blocks(int H);  // column blocks of that pass (its partials per row)

// mxfp8 forward: the permute with x quantised along H fused (codes and scales
// to the padded row of every permuted row; H % 128 == 0; scales of the padded
// rows in one segment of L.seg rows, groups of 128, else cudaErrorInvalidValue),
// and zero codes and scales for the padded rows past each expert's count
cudaError_t launch_permute_quant(const uint16_t *x, const int32_t *row_of_slot, const int32_t *topk_idx,
                                 const int32_t *offsets, const int32_t *pad_off, uint16_t *x_perm,
                                 uint8_t *codes, uint8_t *sf, SfLayout L, int T, int H, int k, cudaStream_t s);
cudaError_t launch_zero_pad_rows(const int32_t *offsets, const int32_t *pad_off, int E, int K, uint8_t *codes,
                                 uint8_t *sf, SfLayout L, cudaStream_t s);

// Weights [E, R, C] quantised along R (R % 128 == 0, C % 64 == 0), transposed:
// codes [E * C, R] (interleave 0) or the gate|up interleave of the mxfp8 GEMM1
// (interleave 1, codes [E * 2C, R]: row e*2C + (c/32)*64 + half*32 + c%32);
// with rows.codes set, also along C row by row: codes [E * R, C].  Scales
// grouped by kMxBN in per-expert segments (L.seg = 2C or C, rows.L.seg = R);
// other layouts: cudaErrorInvalidValue.
cudaError_t launch_quant_wT(const uint16_t *W, int E, int R, int C, int interleave, int half,
                            uint8_t *codes, uint8_t *sf, SfLayout L, RowCodes rows, cudaStream_t s);

// MXFP8 grouped GEMMs: the fp8_bwd backward's four, and the mxfp8 forward's two
enum MxGemmMode : int {
  kMxGemmDA = 0,
  kMxGemmDX = 1,
  kMxGemmDWDown = 2,
  kMxGemmDWGateUp = 3,
  kMxGemmGateUp = 4,  // Q(x) . Q(W_gate | W_up)^T (interleaved B rows) -> SwiGLU: A, G, U, A_w, Q(A)
  kMxGemmDown = 5     // Q(A) . Q(W_down)^T -> Y
};
struct MxGemmArgs {
  int H, I, E, Mpad;
  int M;  // permuted rows T*k (rows of G and U)
  const int32_t *offsets, *pad_off;
  const uint8_t *a0, *a1, *b0, *b1;          // E4M3 codes
  const uint8_t *sfa0, *sfa1, *sfb0, *sfb1;  // scale atoms
  const uint16_t *G, *U;
  const float *w_row;
  uint16_t *o0, *o1, *o2, *o3;
  // mxfp8 GEMM1: A quantised along I for the down GEMM (codes [Mpad, I], 128-row atoms),
  // and (or null) w * A along tokens for the backward's dW_down (codes [I, Mpad])
  uint8_t *aq, *aq_sf, *aw_t, *aw_t_sf;
  // dA: its epilogue quantises dG and dU for the next two GEMMs -- along I
  // (codes [Mpad, I], 128-row scale atoms: dX's A operand) and along tokens
  // (codes [I, Mpad], 192-row scale groups: dW_gate/up's B operand)
  uint8_t *dg_q, *du_q, *dg_sf, *du_sf, *dg_t, *du_t, *dg_t_sf, *du_t_sf;
  int32_t *status;
  int num_sms;
};
cudaError_t launch_mx_gemm(int mode, const MxGemmArgs &a, cudaStream_t s);

// driver entry point for tensor-map encoding (api.cu)
void *tensor_map_encoder();

}  // namespace moe
