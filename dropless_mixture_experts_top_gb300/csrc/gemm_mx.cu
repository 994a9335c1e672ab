// gemm_mx.cu -- MXFP8 grouped GEMMs of the fp8_bwd backward on the 5th-generation
// tensor core: tcgen05.mma kind::mxf8f6f4 with block scaling (E4M3 operands,
// one UE8M0 scale per 32 elements of K, fp32 accumulation in TMEM).
//
// The four backward GEMMs (dA, dX, dW_down, dW_gate/up) read operands written
// by the quantisers in mxfp8.cu: K-major E4M3 codes, scale factors in 512-byte
// atoms, ragged operands in a per-expert row space padded to 128 rows (so tiles
// and 32-element blocks along tokens never straddle two experts, and the padded
// rows are zeros).  dX and the weight gradients write bf16 through the same
// epilogues as the bf16 engine.  dA's epilogue computes dSwiGLU and quantises
// its dG and dU itself, in the form the two GEMMs that read them load: along
// I (a lane's 32 consecutive columns are one block of its row) and along
// tokens (a warp's 32 rows are one 32-token block of the padded row space,
// transposed through the warp's staging tile), from the bf16-rounded values a
// bf16 tensor would hold; dG and dU never exist in bf16.
//
// The mxfp8 mode adds the two forward GEMMs: gate|up (its B rows interleave
// 32 columns of W_gate and the same 32 of W_up, so a 192-row tile yields 96
// output columns and the epilogue computes SwiGLU, writes the bf16 A, G, U,
// A_w and quantises A along I for the down GEMM), and down (plain bf16 Y).
//
// One CTA per SM, persistent, static round-robin over 128 x 192 tiles:
//   warp 0      producer: TMA boxes of codes (128-byte swizzle) and bulk copies
//               of the scale atoms into a 5-stage ring (4 for dA)
//   warp 1      MMA issuer: per stage, tcgen05.cp of the scale atoms into a
//               tensor-memory slot (32x128b.warpx4: row r's four block scales
//               land in lane r%32, column r/32), then four K=32 MMAs selecting
//               the block's scale byte with the descriptor's scale-factor ids
//   warps 2..   epilogue: tcgen05.ld of the accumulator, bf16 stores; 4 warps
//               (one per TMEM lane quarter), 8 for dA (one per column half)
// TMEM holds two 192-column accumulators (the epilogue of one tile overlaps
// the MMAs of the next) and a ring of scale slots.  B-operand scales are
// grouped per 192 rows (two atoms, the second half used) so every tile's
// scales start on an atom.  Every wait is bounded; on a timeout the kernel
// flags the status word and returns after draining its copies and MMAs.
#include <cuda.h>

#include "common.cuh"
#include "epilogue.cuh"
#include "mxfp8.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = kMxBN;  // 128 x 192 tiles
constexpr int BKB = 128;             // K per stage in elements (= bytes): one 128-byte swizzle row
// 5-stage ring; 3 for dA, whose shared memory also holds 8 staging tiles and a
// 4-slot G/U ring (two slots per column half, so a half's next chunk lands
// while it works on the current one)
__host__ __device__ constexpr int stages_of(int mode) { return mode == 0 ? 3 : mode == 4 ? 4 : 5; }
constexpr int kMxGuSlots = 4;
constexpr int kABytes = BM * BKB;    // 16 KB
constexpr int kBBytes = BN * BKB;    // 24 KB
constexpr int kSfBytes = 512 * 3;    // A atom + two B atoms
constexpr int kStageBytes = kABytes + kBBytes;  // 40 KB: keeps every stage 1024-byte aligned
// Warps: producer, MMA issuer, then 4 epilogue warps (one per TMEM lane
// quarter), or 8 (two per quarter) for the epilogue-heavy dA (dSwiGLU, and a
// loader warp that streams G and U into a shared-memory ring ahead of them)
// and gate|up (SwiGLU, four bf16 outputs and A's quantisation; 4 stages).
__host__ __device__ constexpr int epi_warps(int mode) { return (mode == 0 || mode == 4) ? 8 : 4; }
__host__ __device__ constexpr int gu_warps(int mode) { return mode == 0 ? 1 : 0; }
__host__ __device__ constexpr int threads_of(int mode) {
  return 64 + 32 * (epi_warps(mode) + gu_warps(mode));
}
constexpr uint32_t kTmemCols = 512;  // accumulators at 0 and BN, scale slots from 2*BN
constexpr uint32_t kSfCol = 2 * BN, kSfSlotCols = 16;
// Shared memory: code stages | scale atoms | barriers (256) | three [E+1]
// tables | epilogue staging tiles | dA: the G/U ring (1024-aligned), from a
// 1024-aligned base.
__host__ __device__ constexpr int epi_off(int mode) {
  return (stages_of(mode) * (kStageBytes + kSfBytes) + 256 + 3 * (kMaxExperts + 1) * 4 + 15) / 16 * 16;
}
__host__ __device__ constexpr int gu_off(int mode) {
  return (epi_off(mode) + epi_warps(mode) * kEpiTileBytes + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int smem_bytes(int mode) {
  return gu_off(mode) + gu_warps(mode) * kMxGuSlots * kGuChunkBytes + 1024;
}
static_assert(smem_bytes(0) <= 227 * 1024 && smem_bytes(1) <= 227 * 1024 && smem_bytes(4) <= 227 * 1024,
              "shared memory budget");
static_assert(kSfCol + 5 * kSfSlotCols <= kTmemCols, "TMEM budget");

enum MxMode : int { kMxDA = 0, kMxDX = 1, kMxDWDown = 2, kMxDWGateUp = 3, kMxGateUp = 4, kMxDown = 5 };
static_assert(kMxDA == 0 && kMxGateUp == 4, "stages_of, epi_warps");

struct MxParams {
  int H, I, E;
  int Mpad;                 // padded token count the token-axis operands were written with
  const int32_t *offsets;   // [E+1] expert row offsets (unpadded)
  const int32_t *pad_off;   // [E+1] padded offsets (multiples of 128)
  const uint8_t *sfa0, *sfa1, *sfb0, *sfb1;  // scale atoms of the operands
  const uint16_t *G, *U;
  const float *w_row;
  uint16_t *o0, *o1, *o2, *o3;
  uint8_t *aq, *aq_sf;  // gate|up: A quantised along I
  uint8_t *aw_t, *aw_t_sf;  // gate|up: w * A along tokens for the backward (or null)
  uint8_t *dg_q, *du_q, *dg_sf, *du_sf, *dg_t, *du_t, *dg_t_sf, *du_t_sf;  // dA's quantised outputs
  int32_t *status;
  int n_tiles, m_tiles;
  int b_gps;  // B scales: 192-row groups per segment
};

// What the shared epilogue reads: the layer's sizes and buffers, or for the
// weight gradients of W_gate / W_up a [H rows, I columns] view of one of them.
struct EpiView {
  int H, I;
  const uint16_t *G, *U;
  const float *w_row;
  uint16_t *o0, *o1, *o2, *o3;
};

template <int MODE>
struct MxTraits {
  static constexpr bool kRaggedK = (MODE == kMxDWDown || MODE == kMxDWGateUp);
  // dW_gate and dW_up tiles use the dW_down epilogue on a transposed view
  // (dA and gate|up have their own epilogues; down stores Y like dX stores dX)
  static constexpr int kEpi = (MODE == kMxDX || MODE == kMxDown) ? kBwdDX : kBwdDWDown;
  // ragged M: the reduction length and the B rows of one expert
  __host__ __device__ static int kdim(const MxParams &p) {
    return MODE == kMxDX ? 2 * p.I : MODE == kMxDown ? p.I : p.H;
  }
  __host__ __device__ static int brows(const MxParams &p) {
    return MODE == kMxDA ? p.I : MODE == kMxGateUp ? 2 * p.I : p.H;
  }
};

// Block-scaled instruction descriptor: E4M3 x E4M3, fp32 D, UE8M0 scales,
// scale-factor ids select the byte (K block within the 4-block word).
__device__ __forceinline__ uint32_t idesc_mx(int sf_id) {
  return (static_cast<uint32_t>(sf_id) << 4)       // B scale-factor id
         | (static_cast<uint32_t>(BN >> 3) << 17)  // N / 8
         | (1u << 23)                              // scale format: UE8M0
         | (static_cast<uint32_t>(BM >> 4) << 24)  // M / 16
         | (static_cast<uint32_t>(sf_id) << 29);   // A scale-factor id
}

__device__ __forceinline__ void tc_mma_mx(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t sfa_tmem, uint32_t sfb_tmem,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

// 32 rows x 16 bytes of scale atom (contiguous, no swizzle) into 4 TMEM columns,
// replicated to all four lane quarters.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, const void *smem_atom) {
  uint64_t d = static_cast<uint64_t>((smem_addr(smem_atom) >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(1) << 16;    // leading byte offset (unused here) 16 B
  d |= static_cast<uint64_t>(8) << 32;    // stride byte offset: 128 B per 8 rows
  d |= 1ull << 46;                        // descriptor version
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}

__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

struct MxTile {
  Tile t;       // output placement (unpadded rows) for the shared epilogue
  int arow;     // first row of A in its (padded) operand
  int kb0;      // first 128-wide K block in the padded token axis (ragged K)
  int mat;      // dW_gate/up: 0 = gate, 1 = up
  size_t bsf;   // row block of the first of the tile's two B scale atoms
};

template <int MODE>
__device__ __forceinline__ MxTile decode_mx(int tile, const MxParams &p, const int *s_off,
                                            const int *s_pad, const int *s_ord) {
  MxTile x;
  Tile &t = x.t;
  x.mat = 0;
  if constexpr (!MxTraits<MODE>::kRaggedK) {
    const int mt_lin = tile / p.n_tiles, nt = tile % p.n_tiles;
    const int prow = mt_lin * BM;  // padded row of the tile
    int lo = 0, hi = p.E - 1;      // expert whose padded segment holds prow
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_pad[mid] <= prow)
        lo = mid;
      else
        hi = mid - 1;
    }
    t.e = lo;
    t.m0 = s_off[lo] + (prow - s_pad[lo]);
    t.row_end = s_off[lo + 1];
    t.n0 = nt * BN;
    t.nkb = MxTraits<MODE>::kdim(p) / BKB;
    t.krow0 = 0;
    t.kcount = 0;
    x.arow = prow;
    x.kb0 = 0;
    x.bsf = (static_cast<size_t>(lo) * p.b_gps + nt) * 2;  // B rows of expert lo, group nt
  } else {
    if (MODE == kMxDWGateUp) {  // gate and up tiles of the same (e, m, n) are adjacent
      x.mat = tile & 1;
      tile >>= 1;
    }
    const int per = p.m_tiles * p.n_tiles;
    t.e = s_ord[tile / per];  // experts in decreasing order of rows
    const int rem = tile % per;
    const int nt = rem % p.n_tiles;
    t.m0 = (rem / p.n_tiles) * BM;
    t.n0 = nt * BN;
    t.krow0 = s_pad[t.e];
    t.kcount = s_pad[t.e + 1] - s_pad[t.e];
    t.nkb = t.kcount / BKB;  // padded: whole blocks, the rows past the expert's count are zero
    t.row_end = 0;
    x.arow = t.m0;
    x.kb0 = t.krow0 / BKB;
    x.bsf = static_cast<size_t>(nt) * 2;  // one segment: the whole transposed operand
  }
  return x;
}

// dA's epilogue in the fp8_bwd backward: ring, dSwiGLU and the weighting as
// in the bf16 engine's dA, then dG and dU rounded to bf16 (zero in the padded
// rows past the expert's count) and quantised along I and along tokens.
template <int NCH>
__device__ __forceinline__ bool epilogue_da_mx(const MxTile &x, uint32_t tb, int rit, const MxParams &p,
                                               int part, uint8_t *tile, const uint8_t *ring,
                                               uint64_t *gu_full, uint64_t *gu_empty, int &gbase,
                                               volatile int *abort_flag) {
  const Tile &t = x.t;
  const int lane = threadIdx.x & 31;
  const int row = t.m0 + rit;  // unpadded row
  const bool valid = row < t.row_end;
  const int prow = x.arow + rit, prow0 = prow - lane;  // padded rows; prow0 starts a 32-token block
  const float w = valid ? __ldg(p.w_row + row) : 0.f;  // dA = w * (dy . W_down^T)
  const int nch = min(NCH, (p.I - t.n0) / 32);
  // Scale bytes (atom_byte without its divisions).  Along I: 128-row atoms of
  // the padded rows, K = I; this lane's row prow, K block col/32.  Along
  // tokens: rows = columns of dG, grouped per 192 (the tile's n index is the
  // group, as tiles are 192 wide), K = Mpad; this lane's column n0 + 32c + lane,
  // K block prow0/32.
  const int wi = prow & 127;
  const size_t sfi_base = static_cast<size_t>(prow >> 7) * (p.I >> 7) * 512 + (wi & 31) * 16 + (wi >> 5) * 4;
  const int kbt = prow0 >> 5, nt = t.n0 / kMxBN;
  const size_t kblocks_t = static_cast<size_t>(p.Mpad >> 7);
  uint32_t r0[32];
  float v1[32], v2[32];
  bool ok = true;
  for (int c = part; c < nch; c += 2) {
    const int g = gbase + c, slot = g % kMxGuSlots;
    if (!wait_lane0(&gu_full[slot], static_cast<uint32_t>(g / kMxGuSlots) & 1u, abort_flag)) {
      ok = false;
      break;
    }
    __syncwarp();  // the other lanes read the chunk after lane 0 saw it land
    const uint8_t *gs = ring + slot * kGuChunkBytes, *us = gs + kGuHalfBytes;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 xg = *reinterpret_cast<const uint4 *>(gs + epi_swz(rit, q));
      const uint4 xu = *reinterpret_cast<const uint4 *>(us + epi_swz(rit, q));
      const uint32_t wg[4] = {xg.x, xg.y, xg.z, xg.w}, wu[4] = {xu.x, xu.y, xu.z, xu.w};
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        v1[8 * q + 2 * h] = bf16_lo(wg[h]);
        v1[8 * q + 2 * h + 1] = bf16_hi(wg[h]);
        v2[8 * q + 2 * h] = bf16_lo(wu[h]);
        v2[8 * q + 2 * h + 1] = bf16_hi(wu[h]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&gu_empty[slot]);
    const int col = t.n0 + 32 * c;
    tmem_ld32(tb + 32 * c, r0);
    tmem_ld_wait();
    const F2 w2 = f2(w, w), one = f2(1.f, 1.f);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {  // in place: v1 G -> dU, v2 U -> dG; two columns at a time
      const F2 da = f2_mul(w2, f2(__uint_as_float(r0[i]), __uint_as_float(r0[i + 1])));
      const F2 gg = f2(v1[i], v1[i + 1]), u = f2(v2[i], v2[i + 1]);
      const F2 sg = f2(sigmoidf_(v1[i]), sigmoidf_(v1[i + 1]));
      // dG = dA u sg (1 + g (1 - sg)), dU = dA g sg (dA * silu(G))
      const float2 dg = f2_get(f2_mul(f2_mul(f2_mul(da, u), sg), f2_fma(gg, f2_sub(one, sg), one)));
      const float2 du = f2_get(f2_mul(f2_mul(da, gg), sg));
      v2[i] = valid ? round_bf16(dg.x) : 0.f;
      v2[i + 1] = valid ? round_bf16(dg.y) : 0.f;
      v1[i] = valid ? round_bf16(du.x) : 0.f;
      v1[i + 1] = valid ? round_bf16(du.y) : 0.f;
    }
    // along I (dX's A operand): this lane's 32 values are one block of its row
    const int kbi = col >> 5;
    const size_t sfi = sfi_base + (kbi >> 2) * 512 + (kbi & 3);
    p.dg_sf[sfi] = quant32(v2, reinterpret_cast<uint4 *>(p.dg_q + static_cast<size_t>(prow) * p.I + col));
    p.du_sf[sfi] = quant32(v1, reinterpret_cast<uint4 *>(p.du_q + static_cast<size_t>(prow) * p.I + col));
    // along tokens (dW_gate/up's B operand): the warp's 32 rows are one block
    const int rr = 32 * c + lane, wt = rr & 127;
    const size_t sft = ((2 * nt + (rr >> 7)) * kblocks_t + (kbt >> 2)) * 512 + (wt & 31) * 16 +
                       (wt >> 5) * 4 + (kbt & 3);
    quant_down_rows32(tile, v2, p.dg_t, static_cast<size_t>(p.Mpad), col, prow0, p.dg_t_sf + sft);
    quant_down_rows32(tile, v1, p.du_t, static_cast<size_t>(p.Mpad), col, prow0, p.du_t_sf + sft);
  }
  gbase += nch;
  return ok;
}

// The mxfp8 gate|up epilogue: accumulator columns [gate 32 | up 32] x 3 are
// the output columns n0/2 + 32 j (pair j); SwiGLU as in the bf16 engine (A, G
// and U in bf16, rows past the expert's count not stored), A quantised along I
// into the padded row space for the down GEMM, from the bf16 value A holds
// (zero in the padded rows past the count), and w * A quantised along tokens
// for the backward's dW_down (its bf16 value; zero past the count).
template <int NCH>
__device__ __forceinline__ void epilogue_gateup_mx(const MxTile &x, uint32_t tb, int rit, const MxParams &p,
                                                   int part, uint8_t *tile) {
  const Tile &t = x.t;
  const int lane = threadIdx.x & 31;
  const int row = t.m0 + rit, row0 = row - lane;
  const bool valid = row < t.row_end;
  const int nvalid = clamp_rows(t.row_end - row0);
  const int prow = x.arow + rit;
  const float w = valid ? __ldg(p.w_row + row) : 0.f;
  const int ocol0 = t.n0 / 2;
  const int npair = min(NCH / 2, (p.I - ocol0) / 32);
  const int wi = prow & 127;  // A's scale byte (along I: 128-row atoms of the padded rows, K = I)
  const size_t sfi_base = static_cast<size_t>(prow >> 7) * (p.I >> 7) * 512 + (wi & 31) * 16 + (wi >> 5) * 4;
  uint32_t r0[32], r1[32];
  float v0[32], v1[32], v2[32];
  for (int j = part; j < npair; j += 2) {
    tmem_ld32(tb + 64 * j, r0);
    tmem_ld32(tb + 64 * j + 32, r1);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float g = __uint_as_float(r0[i]), u = __uint_as_float(r1[i]);
      v0[i] = g * sigmoidf_(g) * u;  // SwiGLU
      v1[i] = g;
      v2[i] = u;
    }
    const int col = ocol0 + 32 * j;
    const size_t off = static_cast<size_t>(row0) * p.I + col;
    const bool keep = p.o0 != nullptr;  // the bf16 A, G, U, A_w are the backward's only
    if (keep) {
      store_rows32(tile, p.o0 + off, p.I, nvalid, v0);
      store_rows32(tile, p.o1 + off, p.I, nvalid, v1);
      store_rows32(tile, p.o2 + off, p.I, nvalid, v2);
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) v1[i] = valid ? round_bf16(v0[i]) : 0.f;
    const int kb = col >> 5;
    p.aq_sf[sfi_base + (kb >> 2) * 512 + (kb & 3)] =
        quant32(v1, reinterpret_cast<uint4 *>(p.aq + static_cast<size_t>(prow) * p.I + col));
    if (p.o3 || p.aw_t) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v0[i] *= w;  // A_w = w * A, the dW_down operand
      if (p.o3) store_rows32(tile, p.o3 + off, p.I, nvalid, v0);
      if (p.aw_t) {  // along tokens from its bf16 value: the warp's 32 rows are one block (+0 past the count)
#pragma unroll
        for (int i = 0; i < 32; ++i) v1[i] = valid ? round_bf16(v0[i]) : 0.f;
        const int prow0 = prow - lane;
        const size_t sfb = atom_row_sg<128>(0, col + lane, p.Mpad, p.I) + atom_kblock(prow0 >> 5);  // one segment
        quant_down_rows32(tile, v1, p.aw_t, static_cast<size_t>(p.Mpad), col, prow0, p.aw_t_sf + sfb);
      }
    }
  }
}

// One stage: A codes (128 rows), B codes (192 rows), the A scale atom and the
// two B scale atoms of K block kb.
template <int MODE>
__device__ __forceinline__ void produce_mx(const MxTile &x, int kb, uint8_t *st, uint8_t *sf,
                                           uint64_t *bar, const MxParams &p,
                                           const CUtensorMap *a0, const CUtensorMap *a1,
                                           const CUtensorMap *b0, const CUtensorMap *b1) {
  const Tile &t = x.t;
  uint8_t *sa = st, *sb = st + kABytes;
  const uint8_t *sfa, *sfb;
  int K, k;
  if constexpr (MODE == kMxDA || MODE == kMxGateUp || MODE == kMxDown) {
    // dA: A = dy (padded rows, K = H), B = W_down rows e*I + n;  gate|up: A = x
    // (K = H), B = interleaved gate|up rows e*2I + n;  down: A = A (K = I), B =
    // W_down^T rows e*H + n
    K = MxTraits<MODE>::kdim(p);
    k = kb;
    tma_load_2d(sa, a0, bar, k * BKB, x.arow);
    tma_load_2d(sb, b0, bar, k * BKB, t.e * MxTraits<MODE>::brows(p) + t.n0);
    sfa = p.sfa0;
    sfb = p.sfb0;
  } else if constexpr (MODE == kMxDX) {  // A = [dG | dU] (padded rows, K = I each); B = W_gate | W_up
    K = p.I;
    const int kbi = p.I / BKB;
    const bool first = kb < kbi;
    k = first ? kb : kb - kbi;
    tma_load_2d(sa, first ? a0 : a1, bar, k * BKB, x.arow);
    tma_load_2d(sb, first ? b0 : b1, bar, k * BKB, t.e * p.H + t.n0);
    sfa = first ? p.sfa0 : p.sfa1;
    sfb = first ? p.sfb0 : p.sfb1;
  } else {  // ragged K: operands transposed, K = padded tokens
    K = p.Mpad;
    k = x.kb0 + kb;
    tma_load_2d(sa, a0, bar, k * BKB, x.arow);
    const bool up = MODE == kMxDWGateUp && x.mat;
    tma_load_2d(sb, up ? b1 : b0, bar, k * BKB, t.n0);  // dy^T (dW_down) or dG^T / dU^T rows
    sfa = p.sfa0;
    sfb = up ? p.sfb1 : p.sfb0;
  }
  const size_t kblocks = static_cast<size_t>(K / 128);
  bulk_load(sf, sfa + (static_cast<size_t>(x.arow / BM) * kblocks + k) * 512, 512, bar);
  bulk_load(sf + 512, sfb + (x.bsf * kblocks + k) * 512, 512, bar);
  bulk_load(sf + 1024, sfb + ((x.bsf + 1) * kblocks + k) * 512, 512, bar);
}

template <int MODE>
__global__ void __launch_bounds__(threads_of(MODE), 1)
    grouped_gemm_mx_kernel(const __grid_constant__ CUtensorMap tmA0,
                           const __grid_constant__ CUtensorMap tmA1,
                           const __grid_constant__ CUtensorMap tmB0,
                           const __grid_constant__ CUtensorMap tmB1, const MxParams p) {
  constexpr int STAGES = stages_of(MODE);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *stages = smem;                                  // [STAGES] A | B codes
  uint8_t *sfs = smem + STAGES * kStageBytes;              // [STAGES] scale atoms
  uint64_t *bars = reinterpret_cast<uint64_t *>(sfs + STAGES * kSfBytes);
  uint64_t *full = bars, *empty = bars + STAGES;
  uint64_t *tfull = bars + 2 * STAGES;  // [2] accumulator ready
  uint64_t *tempty = tfull + 2;         // [2] accumulator drained by the epilogue
  uint64_t *drain = tempty + 2;
  uint64_t *gu_full = drain + 1;            // [kMxGuSlots] dA: a G/U chunk landed
  uint64_t *gu_empty = gu_full + kMxGuSlots;  // [kMxGuSlots] dA: its 4 epilogue warps read it
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(gu_empty + kMxGuSlots);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_off = reinterpret_cast<int *>(sfs + STAGES * kSfBytes + 256);
  int *s_pad = s_off + (kMaxExperts + 1);
  int *s_ord = s_pad + (kMaxExperts + 1);  // ragged K: experts by decreasing row count
  uint8_t *epi_tiles = smem + epi_off(MODE);  // [epilogue warp] 32 x 32 bf16 staging tiles
  uint8_t *gu_ring = smem + gu_off(MODE);     // dA: [kMxGuSlots] G chunk | U chunk
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 32 * epi_warps(MODE));  // every epilogue thread
    }
    mbar_init(drain, 1);
    for (int s = 0; s < kMxGuSlots; ++s) {
      mbar_init(&gu_full[s], 1);
      mbar_init(&gu_empty[s], 4);  // the four warps (lane quarters) of one column half
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA0);
    tma_prefetch_desc(&tmA1);
    tma_prefetch_desc(&tmB0);
    tma_prefetch_desc(&tmB1);
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  griddep_wait();  // the set-up above overlaps the previous kernel's end; its outputs are read below
  for (int e = threadIdx.x; e <= E; e += threads_of(MODE)) {
    s_off[e] = __ldg(p.offsets + e);
    s_pad[e] = __ldg(p.pad_off + e);
  }
  __syncthreads();
  if (MxTraits<MODE>::kRaggedK) {
    // Skewed routing (an expert with more than twice the mean rows): longest
    // reductions first, so the static round-robin hands out the experts' tiles
    // in decreasing order of work.  Balanced routing keeps the natural order.
    int cmax = 0;
    for (int f = 0; f < E; ++f) cmax = max(cmax, s_pad[f + 1] - s_pad[f]);
    const bool skewed = static_cast<int64_t>(cmax) * E > 2 * static_cast<int64_t>(s_pad[E]);
    for (int e = threadIdx.x; e < E; e += threads_of(MODE)) {
      const int c = s_pad[e + 1] - s_pad[e];
      int r = 0;
      for (int f = 0; f < E; ++f) {
        const int cf = s_pad[f + 1] - s_pad[f];
        r += (cf > c || (cf == c && f < e)) ? 1 : 0;
      }
      s_ord[skewed ? r : e] = e;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = MODE == kMxDWGateUp ? 2 * E * p.m_tiles * p.n_tiles
                    : MODE == kMxDWDown ? E * p.m_tiles * p.n_tiles
                                        : (s_pad[E] / BM) * p.n_tiles;
  constexpr uint32_t kTx = kABytes + kBBytes + kSfBytes;

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    // Lane 0 runs the loop alone: no warp collective per stage.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, arm_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const MxTile x = decode_mx<MODE>(tile, p, s_off, s_pad, s_ord);
        for (int kb = 0; kb < x.t.nkb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], kTx);
          produce_mx<MODE>(x, kb, stages + stage * kStageBytes, sfs + stage * kSfBytes, &full[stage],
                           p, &tmA0, &tmA1, &tmB0, &tmB1);
          armed |= 1u << stage;
          arm_par = (arm_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      griddep_launch_dependents();  // all loads issued: the next kernel may be launched
      if (*abort_flag) {  // let the copies in flight land before the CTA exits
        for (int s = 0; s < STAGES; ++s) {
          if (!((armed >> s) & 1u)) continue;
          for (int i = 0; i < (1 << 22) && !mbar_try_wait(&full[s], (arm_par >> s) & 1u); ++i) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // Lane 0 runs the loop alone: no warp collective per stage.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x, ++it) {
        const MxTile x = decode_mx<MODE>(tile, p, s_off, s_pad, s_ord);
        const int buf = it & 1;
        const uint32_t use = (it >> 1) & 1;
        if (!mbar_wait(&tempty[buf], use ^ 1, abort_flag)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + buf * BN;
        if (x.t.nkb == 0) {  // empty expert: the epilogue writes zeros
          mbar_arrive(&tfull[buf]);
          continue;
        }
        for (int kb = 0; kb < x.t.nkb; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t *st = stages + stage * kStageBytes;
          uint8_t *sf = sfs + stage * kSfBytes;
          const uint32_t slot = tmem_base + kSfCol + kSfSlotCols * stage;
          tc_cp_sf(slot, sf);             // A scales: columns slot .. slot+3
          tc_cp_sf(slot + 4, sf + 512);   // B rows 0..127: slot+4 .. slot+7
          tc_cp_sf(slot + 8, sf + 1024);  // B rows 128..191: slot+8, slot+9
          const uint32_t a_base = smem_addr(st), b_base = smem_addr(st + kABytes);
#pragma unroll
          for (int k32 = 0; k32 < BKB / 32; ++k32) {
            const uint64_t adesc = smem_desc_sw128(a_base + k32 * 32, 16, 1024);
            const uint64_t bdesc = smem_desc_sw128(b_base + k32 * 32, 16, 1024);
            tc_mma_mx(d_tmem, adesc, bdesc, idesc_mx(k32), slot, slot + 4, (kb | k32) != 0 ? 1u : 0u);
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[buf]);
      }
      if (*abort_flag) {  // wait for issued MMAs before TMEM is freed
        tc_commit(drain);
        for (int i = 0; i < (1 << 22) && !mbar_try_wait(drain, 0); ++i) {
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + epi_warps(MODE)) {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // column range: warps 2..5 the first, 6..9 the second (a constant 0 with 4 warps)
    const int part = epi_warps(MODE) == 8 ? (warp - 2) >> 2 : 0;
    const int rit = q * 32 + lane;
    int it = 0, gbase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++it) {
      const MxTile x = decode_mx<MODE>(tile, p, s_off, s_pad, s_ord);
      const int buf = it & 1;
      const uint32_t use = (it >> 1) & 1;
      if (!wait_lane0(&tfull[buf], use, abort_flag)) break;
      __syncwarp();  // every lane reads the accumulator after lane 0 saw it complete
      tc_fence_after();
      EpiView v{p.H, p.I, p.G, p.U, p.w_row, p.o0, p.o1, nullptr, nullptr};
      if (MODE == kMxDWGateUp) {  // [H rows, I columns] of dW_gate or dW_up
        v.H = p.I;
        v.I = p.H;
        v.o0 = x.mat ? p.o1 : p.o0;
        v.o1 = nullptr;
      }
      const uint32_t tb = tmem_base + buf * BN + (static_cast<uint32_t>(q * 32) << 16);
      uint8_t *stile = epi_tiles + (warp - 2) * kEpiTileBytes;
      if constexpr (MODE == kMxDA) {
        if (!epilogue_da_mx<BN / 32>(x, tb, rit, p, part, stile, gu_ring, gu_full, gu_empty, gbase,
                                     abort_flag))
          break;
      } else if constexpr (MODE == kMxGateUp) {
        epilogue_gateup_mx<BN / 32>(x, tb, rit, p, part, stile);
      } else {
        epilogue_tile<MxTraits<MODE>::kEpi, EpiView, BN / 32>(x.t, tb, rit, v, part,
                                                              epi_warps(MODE) / 4, stile);
      }
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
    }
  } else {
    // ---------------------------------------------------------------- dA: G/U loader
    // Walks the tiles in the epilogue's order and loads each tile's G and U
    // (128 rows from the tile's first unpadded row) in 32-column chunks
    // (lane 0 alone).
    if (lane == 0) {
      int g = 0;
      uint32_t armed = 0, arm_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
        const MxTile x = decode_mx<MODE>(tile, p, s_off, s_pad, s_ord);
        const int nch = min(BN / 32, (p.I - x.t.n0) / 32);
        for (int c = 0; c < nch; ++c, ++g) {
          const int slot = g % kMxGuSlots;
          const uint32_t ph = static_cast<uint32_t>(g / kMxGuSlots) & 1u;
          if (!mbar_wait(&gu_empty[slot], ph ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          uint8_t *dst = gu_ring + slot * kGuChunkBytes;
          mbar_arrive_expect_tx(&gu_full[slot], kGuChunkBytes);
          tma_load_2d(dst, &tmA1, &gu_full[slot], x.t.n0 + 32 * c, x.t.m0);                 // G
          tma_load_2d(dst + kGuHalfBytes, &tmB1, &gu_full[slot], x.t.n0 + 32 * c, x.t.m0);  // U
          armed |= 1u << slot;
          arm_par = (arm_par & ~(1u << slot)) | (ph << slot);
        }
      }
      if (*abort_flag) {  // let the copies in flight land before exit
        for (int sl = 0; sl < kMxGuSlots; ++sl) {
          if (!((armed >> sl) & 1u)) continue;
          for (int i = 0; i < (1 << 22) && !mbar_try_wait(&gu_full[sl], (arm_par >> sl) & 1u); ++i) {
          }
        }
      }
    }
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag) flag_status(p.status, kDevWaitTimeout);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// 2-D byte tensor map over row-major [rows, inner] codes, box {128, box_rows}.
bool make_map_u8(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows, uint32_t box_rows) {
  auto fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 map over G or U [rows, I]: box {32, 128} (64-byte rows), 64-byte
// swizzle, zero fill out of bounds.
bool make_map_gu_bf16(CUtensorMap *m, const void *ptr, uint64_t inner, uint64_t rows) {
  auto fn = reinterpret_cast<EncodeTiledFn>(tensor_map_encoder());
  if (!fn) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {32, static_cast<cuuint32_t>(BM)};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline int cdiv(int a, int b) { return (a + b - 1) / b; }

template <int MODE>
cudaError_t launch_mx_mode(const MxGemmArgs &a, cudaStream_t s) {
  CUtensorMap mA0, mA1, mB0, mB1;
  MxParams p{};
  p.H = a.H;
  p.I = a.I;
  p.E = a.E;
  p.Mpad = a.Mpad;
  p.offsets = a.offsets;
  p.pad_off = a.pad_off;
  p.G = a.G;
  p.U = a.U;
  p.w_row = a.w_row;
  p.o0 = a.o0;
  p.o1 = a.o1;
  p.o2 = a.o2;
  p.o3 = a.o3;
  p.aq = a.aq;
  p.aq_sf = a.aq_sf;
  p.aw_t = a.aw_t;
  p.aw_t_sf = a.aw_t_sf;
  p.dg_q = a.dg_q;
  p.du_q = a.du_q;
  p.dg_sf = a.dg_sf;
  p.du_sf = a.du_sf;
  p.dg_t = a.dg_t;
  p.du_t = a.du_t;
  p.dg_t_sf = a.dg_t_sf;
  p.du_t_sf = a.du_t_sf;
  p.status = a.status;
  p.sfa0 = a.sfa0;
  p.sfa1 = a.sfa1;
  p.sfb0 = a.sfb0;
  p.sfb1 = a.sfb1;
  const uint64_t H = a.H, I = a.I, E = a.E, Mp = a.Mpad;
  bool ok = true;
  switch (MODE) {
    case kMxDA:  // [Mp, H] x [E*I, H]^T; A1, B1: G and U [M, I] for the epilogue's ring
      ok = make_map_u8(&mA0, a.a0, H, Mp, BM) && make_map_u8(&mB0, a.b0, H, E * I, BN) &&
           make_map_gu_bf16(&mA1, a.G, I, a.M) && make_map_gu_bf16(&mB1, a.U, I, a.M);
      p.n_tiles = p.b_gps = cdiv(a.I, BN);
      break;
    case kMxDX:  // [Mp, I] x [E*H, I]^T, twice
      ok = make_map_u8(&mA0, a.a0, I, Mp, BM) && make_map_u8(&mA1, a.a1, I, Mp, BM) &&
           make_map_u8(&mB0, a.b0, I, E * H, BN) && make_map_u8(&mB1, a.b1, I, E * H, BN);
      p.n_tiles = p.b_gps = cdiv(a.H, BN);
      break;
    case kMxDWDown:  // per expert: [I, tokens] x [H, tokens]^T
      ok = make_map_u8(&mA0, a.a0, Mp, I, BM) && make_map_u8(&mB0, a.b0, Mp, H, BN);
      mA1 = mA0;
      mB1 = mB0;
      p.m_tiles = a.I / BM;
      p.n_tiles = p.b_gps = cdiv(a.H, BN);
      break;
    case kMxGateUp:  // [Mp, H] x [E*2I, H]^T (gate|up rows interleaved by 32)
      ok = make_map_u8(&mA0, a.a0, H, Mp, BM) && make_map_u8(&mB0, a.b0, H, E * 2 * I, BN);
      mA1 = mA0;
      mB1 = mB0;
      p.n_tiles = p.b_gps = cdiv(2 * a.I, BN);
      break;
    case kMxDown:  // [Mp, I] x [E*H, I]^T
      ok = make_map_u8(&mA0, a.a0, I, Mp, BM) && make_map_u8(&mB0, a.b0, I, E * H, BN);
      mA1 = mA0;
      mB1 = mB0;
      p.n_tiles = p.b_gps = cdiv(a.H, BN);
      break;
    default:  // kMxDWGateUp, per expert: [H, tokens] x [I, tokens]^T for dG and for dU
      ok = make_map_u8(&mA0, a.a0, Mp, H, BM) && make_map_u8(&mB0, a.b0, Mp, I, BN) &&
           make_map_u8(&mB1, a.b1, Mp, I, BN);
      mA1 = mA0;
      p.m_tiles = a.H / BM;
      p.n_tiles = p.b_gps = cdiv(a.I, BN);
      break;
  }
  if (!ok) return cudaErrorInvalidValue;
  static DeviceOnce once;  // the shared-memory opt-in, once per device
  const cudaError_t e = once.get([](int *) {
    return cudaFuncSetAttribute(grouped_gemm_mx_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_bytes(MODE));
  });
  if (e != cudaSuccess) return e;
  return launch_pdl(grouped_gemm_mx_kernel<MODE>, dim3(a.num_sms), dim3(threads_of(MODE)), smem_bytes(MODE), s, 1,
                    mA0, mA1, mB0, mB1, p);
}

}  // namespace

cudaError_t launch_mx_gemm(int mode, const MxGemmArgs &a, cudaStream_t s) {
  switch (mode) {
    case kMxGemmDA: return launch_mx_mode<kMxDA>(a, s);
    case kMxGemmDX: return launch_mx_mode<kMxDX>(a, s);
    case kMxGemmDWDown: return launch_mx_mode<kMxDWDown>(a, s);
    case kMxGemmDWGateUp: return launch_mx_mode<kMxDWGateUp>(a, s);
    case kMxGemmGateUp: return launch_mx_mode<kMxGateUp>(a, s);
    case kMxGemmDown: return launch_mx_mode<kMxDown>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace moe
